"""Inputs at the edges of the integer dot product's input format.

Every GEMV stages its input as 24-bit fixed point with one power-of-two
exponent per group of 64 values, so an input far below its group's largest
value keeps fewer bits. These cases put that to the test against the fp64
oracle, element-wise, at the usual tolerance:
  * one value 2^10 times the rest in every group, random weights;
  * the same outliers on "dead" input channels (their weights exactly zero),
    so the output depends only on the small values beside them;
  * rows whose two halves cancel exactly (output 0) next to ordinary rows;
  * SwiGLU outputs with outliers feeding the down projection, through the
    grouped expert kernels and through the batch-1 layer kernel.
"""

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from oracle import bgq_oracle as O
from tests.helpers import TC_OWN_TOL, ExpertSource, assert_bf16_output, bits16, f64, rel_l2

pytestmark = pytest.mark.gpu

MID = {2: 2, 4: 8, 8: 128}  # code with weight (q - MID) * s when bias = -MID * s


def set_codes(q, bits, rows, col, code):
    """Write `code` into column `col` of the given rows of packed words q (int32 [rows][words])."""
    per = 32 // bits
    w, sh = col // per, bits * (col % per)
    mask = ((1 << bits) - 1) << sh
    v = q[rows, w].to(torch.int64) & 0xFFFFFFFF
    v = (v & ~mask) | (code << sh)
    q[rows, w] = (v - ((v >> 31) << 32)).to(torch.int32)


def outlier_input(seed, batch, cols, dev, ratio=1024.0, every=64, offset=5):
    x = synth.activations(seed, 77, batch, cols, device=dev).float()
    x[:, offset::every] = ratio * 1.5 * torch.sign(x[:, offset::every] + 1e-3)
    return x.to(torch.bfloat16)


def gemv_fn(bits):
    return {4: lib.q4_gemv, 2: lib.q2_gemv, 8: lib.q8_gemv}[bits]


@pytest.mark.parametrize("bits", [4, 2, 8])
@pytest.mark.parametrize("dead", [False, True])
def test_gemv_outliers(cuda_device, bits, dead):
    rows, cols, B = 1024, 4096, 3
    q, sb = synth.qmatrix(61, rows, cols, bits, device=cuda_device)
    x = outlier_input(61, B, cols, cuda_device)
    if dead:  # the outlier columns carry weight exactly 0: code MID, bias -MID*scale
        allr = torch.arange(rows, device=cuda_device)
        for col in range(5, cols, 64):
            set_codes(q, bits, allr, col, MID[bits])
        sb[:, :, 1] = (sb[:, :, 0].float() * -MID[bits]).to(torch.bfloat16)  # exact: a power-of-two multiple
    y = gemv_fn(bits)(lib.QMatrix(q, sb, rows, cols, bits), x)
    torch.cuda.synchronize()
    W = O.dequant(q.cpu().numpy(), bits16(sb), bits)
    if dead:
        assert np.all(W[:, 5::64] == 0.0)
    ref = f64(x) @ W.T
    for t in range(B):
        assert_bf16_output(f64(y)[t], ref[t], (bits, dead, t))


@pytest.mark.parametrize("bits", [4, 2])
def test_gemv_rows_that_cancel(cuda_device, bits):
    """Rows 0, 2, 4, ... have second-half codes 2*MID-1-q and biases that make
    W[n, k + cols/2] = -W[n, k]; with x = [v, v] those rows are exactly 0 (in
    the oracle), the odd rows are ordinary. The cancelling rows' outputs must
    be 0 within 1e-3 of the largest output."""
    rows, cols = 512, 4096
    half = cols // 2
    q, sb = synth.qmatrix(62, rows, cols, bits, device=cuda_device)
    qmax = (1 << bits) - 1
    codes = O.unpack_codes(q.cpu().numpy(), bits)
    even = np.arange(0, rows, 2)
    codes[even, half:] = qmax - codes[even, :half]
    per = 32 // bits
    words = np.zeros((rows, cols // per), dtype=np.int64)
    for j in range(per):
        words |= codes[:, j::per].astype(np.int64) << (bits * j)
    q = torch.from_numpy(((words + 2 ** 31) % 2 ** 32 - 2 ** 31).astype(np.int32)).to(cuda_device)
    s = 2.0 ** -7
    sbn = sb.float().cpu().numpy()
    sbn[even, :, 0] = s
    sbn[even, : half // 64, 1] = -MID[bits] * s
    sbn[even, half // 64:, 1] = (MID[bits] - qmax) * s  # -b - qmax*s: exact in bf16
    sb = torch.from_numpy(sbn).to(torch.bfloat16).to(cuda_device)
    xv = outlier_input(62, 2, half, cuda_device, ratio=64.0)
    x = torch.cat([xv, xv], dim=1).contiguous()
    y = gemv_fn(bits)(lib.QMatrix(q, sb, rows, cols, bits), x)
    torch.cuda.synchronize()
    ref = O.gemv(q.cpu().numpy(), bits16(sb), bits, f64(x))
    assert np.all(ref[:, even] == 0.0)
    for t in range(2):
        assert_bf16_output(f64(y)[t], ref[t], t)


def expert_with_h_outliers(seed, d, f, bits, dev, dead):
    """An expert whose up rows 3, 67, 131, ... have 256x larger scales (so h
    has outliers 2^8 x its other values); with dead=True the down matrix's
    columns at those h positions carry weight exactly 0."""
    shape = synth.PoolShape(d, f, 1, bits)
    q, sb = synth.expert_pool_range(seed, 0, shape, 0, 1, device=dev)
    mats = synth.expert_matrices(q[0], sb[0], shape)
    hot = torch.arange(3, f, 64, device=dev)
    up_sb = mats[1][1]
    up_sb[hot, :, 0] = (up_sb[hot, :, 0].float() * 256).to(torch.bfloat16)
    up_sb[hot, :, 1] = (up_sb[hot, :, 1].float() * 256).to(torch.bfloat16)
    if dead:
        dq, dsb = mats[2]
        for col in hot.tolist():
            set_codes(dq, bits, torch.arange(d, device=dev), col, MID[bits])
        dsb[:, :, 1] = (dsb[:, :, 0].float() * -MID[bits]).to(torch.bfloat16)
    dims = [(f, d), (f, d), (d, f)]
    ex = lib.Expert(*[lib.QMatrix(m[0], m[1], r, c, bits) for m, (r, c) in zip(mats, dims)])
    return ex, [(m[0].cpu().numpy(), bits16(m[1])) for m in mats]


@pytest.mark.parametrize("bits", [4, 2])
@pytest.mark.parametrize("dead", [False, True])
@pytest.mark.parametrize("B", [1, 5])
def test_expert_swiglu_outputs_with_outliers(cuda_device, bits, dead, B):
    d, f = 4096, 1024
    ex, mats = expert_with_h_outliers(63, d, f, bits, cuda_device, dead)
    x = synth.activations(63, 5, B, d, device=cuda_device)  # the outliers are in h, not in x
    y, yf = lib.moe_expert_swiglu(ex, x, want_f32=True)
    torch.cuda.synchronize()
    g = O.gemv(*mats[0], bits, f64(x))
    u = O.gemv(*mats[1], bits, f64(x))
    h = O.silu(g) * u
    hot = np.median(np.abs(h[:, 3::64])) / np.median(np.abs(h))
    assert hot > 30  # the outliers are real
    for t in range(B):
        ref = O.expert_swiglu(*mats, bits, f64(x)[t])
        assert_bf16_output(f64(y)[t], ref, (t, dead))
        assert rel_l2(f64(yf)[t], ref) <= 2e-4


@pytest.mark.parametrize("B", [1, 3])
@pytest.mark.parametrize("bits", [4, 2])
def test_layer_with_outlier_inputs(cuda_device, B, bits):
    """A whole layer (batch 1: the persistent kernel; 3: the grouped kernels)
    on inputs with 2^10 outliers in every group."""
    E, d, f, K = 16, 1024, 256, 4
    shape = synth.PoolShape(d, f, E, bits)
    t = synth.layer_tensors(64, 0, shape, device=cuda_device)
    t["router"].copy_((t["router"].float() * 0.25).to(torch.bfloat16))
    L = lib.MoELayer(d, f, E, K, bits, t["router"], t["shared_gate"], t["pool_q"][:E], t["pool_sb"][:E],
                     t["pool_q"][E], t["pool_sb"][E])
    x = outlier_input(64, B, d, cuda_device)
    out, _, idx, _, _ = lib.moe_layer_forward(L, x, want_route=True)
    torch.cuda.synchronize()
    src = ExpertSource(64, 0, shape)
    Rb, Gb = bits16(t["router"]), bits16(t["shared_gate"])
    for tok in range(B):
        xt = f64(x)[tok]
        logits = O.route(Rb, xt, K, Gb)[0]
        s = np.sort(logits)[::-1]
        assert s[K - 1] - s[K] > 1e-3  # no near tie in this case
        ref, oi, _, _ = O.moe_layer(Rb, Gb, src, src(E), bits, xt, K)
        assert idx[tok].cpu().tolist() == oi.tolist()
        assert_bf16_output(f64(out)[tok], ref, tok)


@pytest.mark.parametrize("B", [16, 40])
def test_tensorcore_operands_beyond_fp16_range(cuda_device, B):
    """The tensor-core path multiplies fp16 operands; each token's inputs are
    scaled by a power of two before the conversion and scaled back after, so
    inputs beyond fp16's range (|x| ~ 1e5 > 65504), tiny inputs (~1e-7) and
    SwiGLU outputs far beyond 65504 keep the usual tolerance."""
    d, f, bits = 4096, 1024, 4
    ex, mats = expert_with_h_outliers(65, d, f, bits, cuda_device, dead=False)
    x = synth.activations(65, 9, B, d, device=cuda_device).float()
    x[0] *= 4.0e4   # |x| beyond 65504
    x[1] *= 1.0e-7  # tiny
    x[2, ::64] *= 1.0e4  # outliers beyond fp16's range in every group
    x = x.to(torch.bfloat16)
    assert float(x.float().abs().max()) > 65504
    y, yf = lib.moe_expert_swiglu(ex, x, want_f32=True)
    torch.cuda.synchronize()
    xd = f64(x)
    h0 = O.silu(O.gemv(*mats[0], bits, xd[0])) * O.gemv(*mats[1], bits, xd[0])
    assert np.abs(h0).max() > 65504  # the SwiGLU outputs overflow fp16 unscaled
    for t in sorted({0, 1, 2, 3, B - 1}):
        ref = O.expert_swiglu(*mats, bits, xd[t])
        assert np.all(np.isfinite(f64(yf)[t]))
        assert_bf16_output(f64(y)[t], ref, t, own_tol=TC_OWN_TOL)
