"""GPU parity of the standalone GEMV and the router against the fp64 oracle.

Tolerances: outputs within max relative L2 error 2e-3 (bf16 out, fp32
accumulate); expert indices exact wherever the K-th and (K+1)-th oracle
logits differ by more than 1e-3, a valid top-K otherwise.
"""

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from oracle import bgq_oracle as O
from tests.helpers import TIE_GAP, assert_bf16_output, bits16, check_topk_valid, f64, topk_gap

pytestmark = pytest.mark.gpu


def make_matrix(seed, rows, cols, bits, dev):
    q, sb = synth.qmatrix(seed, rows, cols, bits, device=dev)
    return lib.QMatrix(q, sb, rows, cols, bits), q, sb


GEMV_CASES = [
    # (rows, cols, bits, batch)
    (1024, 4096, 4, 1),  # the single-GEMV workload
    (1000, 4096, 4, 3),  # ragged rows (not a multiple of a CTA's rows)
    (4096, 1024, 4, 1),  # down-projection shape
    (37, 1024, 4, 8),
    (96, 3072, 4, 2),
    (256, 64, 4, 5),  # 2 parts per row: 16 rows per warp pass
    (130, 128, 4, 13),  # batch above 8 splits into launches
    (1024, 4096, 2, 1),
    (515, 2048, 2, 4),
    (4096, 1024, 2, 1),  # 16 lanes per row at 2 bits
    (64, 64, 2, 1),  # 1 part per row
    (4096, 4096, 4, 1),  # a square 4-bit projection (attention-like)
    (4096, 4096, 4, 9),  # ... at a batch that takes two launches
    (4096, 8192, 4, 8),  # wide rows: the staged inputs fill most of shared memory
    (256, 16384, 2, 3),  # wider still: fewer inputs per launch
]


@pytest.mark.parametrize("rows,cols,bits,batch", GEMV_CASES)
def test_gemv_matches_oracle(cuda_device, rows, cols, bits, batch):
    W, q, sb = make_matrix(100 + rows + cols, rows, cols, bits, cuda_device)
    x = synth.activations(7, rows, batch, cols, device=cuda_device)
    fn = lib.q4_gemv if bits == 4 else lib.q2_gemv
    y = fn(W, x)
    torch.cuda.synchronize()
    ref = O.gemv(q.cpu().numpy(), bits16(sb), bits, f64(x))
    got = f64(y)
    for t in range(batch):
        assert_bf16_output(got[t], ref[t], t)


@pytest.mark.parametrize("variant", [lib.DQ_STANDARD, lib.DQ_REORDERED, lib.DQ_HOISTED])
@pytest.mark.parametrize("bits", [4, 2])
def test_gemv_variants_match_oracle(cuda_device, variant, bits):
    rows, cols = 300, 4096
    W, q, sb = make_matrix(5, rows, cols, bits, cuda_device)
    x = synth.activations(8, 0, 2, cols, device=cuda_device)
    y = lib.qgemv_variant(W, x, variant)
    torch.cuda.synchronize()
    ref = O.gemv(q.cpu().numpy(), bits16(sb), bits, f64(x))
    for t in range(2):
        assert_bf16_output(f64(y)[t], ref[t], t)


def test_gemv_deterministic(cuda_device):
    W, q, sb = make_matrix(3, 1024, 4096, 4, cuda_device)
    x = synth.activations(3, 0, 4, 4096, device=cuda_device)
    a = lib.q4_gemv(W, x).clone()
    b = lib.q4_gemv(W, x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_gemv_batch_equals_single(cuda_device):
    """Each token's result does not depend on the others in the batch (bitwise)."""
    W, q, sb = make_matrix(4, 512, 4096, 4, cuda_device)
    x = synth.activations(4, 0, 6, 4096, device=cuda_device)
    yb = lib.q4_gemv(W, x)
    for t in range(6):
        y1 = lib.q4_gemv(W, x[t:t + 1].contiguous())
        assert torch.equal(yb[t].view(torch.int16), y1[0].view(torch.int16))


def test_gemv_column_probe(cuda_device):
    """x = e_k returns column k of the dequantised matrix, rounded to bf16 (exactly)."""
    rows, cols = 256, 1024
    W, q, sb = make_matrix(9, rows, cols, 4, cuda_device)
    ks = [0, 1, 7, 8, 63, 64, 511, 1023]
    x = torch.zeros((len(ks), cols), dtype=torch.bfloat16, device=cuda_device)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = lib.q4_gemv(W, x)
    Wd = O.dequant(q.cpu().numpy(), bits16(sb), 4)
    for i, k in enumerate(ks):
        assert np.array_equal(bits16(y[i]), O.f64_to_bf16_bits(Wd[:, k])), k


# ------------------------------------------------------------------ router
def route_case(dev, seed, B, E=512, d=4096, K=4, with_gate=True):
    R = synth.router(seed, 0, E, d, device=dev)
    G = synth.shared_gate(seed, 0, d, device=dev) if with_gate else None
    x = synth.activations(seed, 1, B, d, device=dev)
    return R, G, x


@pytest.mark.parametrize("B", [1, 5, 64, 200])
def test_route_matches_oracle(cuda_device, B):
    K = 4
    R, G, x = route_case(cuda_device, 20 + B, B)
    idx, w, gamma, logits = lib.moe_route_topk(R, G, x, K, want_logits=True)
    torch.cuda.synchronize()
    Rb, Gb, xd = bits16(R), bits16(G), f64(x)
    for t in range(B):
        l, p, oi, ow, og = O.route(Rb, xd[t], K, Gb)
        gl = logits[t].cpu().double().numpy()
        assert np.max(np.abs(gl - l)) <= 1e-5 * max(1.0, np.abs(l).max())
        gi = idx[t].cpu().numpy()
        if topk_gap(l, K) > TIE_GAP:
            assert gi.tolist() == oi.tolist()
            assert np.allclose(w[t].cpu().numpy(), ow, rtol=1e-5, atol=1e-6)
        else:
            check_topk_valid(gi, l, K)
            pw = p[gi] / p[gi].sum()
            assert np.allclose(w[t].cpu().numpy(), pw, rtol=1e-5, atol=1e-6)
        assert abs(float(gamma[t]) - og) <= 1e-6
        assert abs(float(w[t].sum()) - 1.0) <= 1e-6


def test_route_planted_ties_pick_lowest_index(cuda_device):
    """Duplicate router rows give bit-identical logits; the lower index must win.

    Rows 3 and 9 are the same strongly aligned row, rows 7, 40 and 50 the same
    less aligned row, so the top-4 is [3, 9, 7, 40] with two exact ties."""
    E, d, K = 64, 1024, 4
    R, _, x = route_case(cuda_device, 31, 1, E=E, d=d)
    R = R.clone()
    sgn = x[0].float().sign()
    big = (0.05 * sgn).to(torch.bfloat16)
    mid = (0.04 * sgn).to(torch.bfloat16)
    for e in (3, 9):
        R[e] = big
    for e in (7, 40, 50):
        R[e] = mid
    idx, w, gamma, logits = lib.moe_route_topk(R, None, x, K, want_logits=True)
    torch.cuda.synchronize()
    assert logits[0, 3] == logits[0, 9] and logits[0, 7] == logits[0, 40] == logits[0, 50]
    assert idx[0].cpu().tolist() == [3, 9, 7, 40]
    l = O.route(bits16(R), f64(x)[0], K)[0]
    assert O.topk_stable(l, K).tolist() == [3, 9, 7, 40]
    assert float(gamma[0]) == 1.0


def test_route_no_gate_and_other_k(cuda_device):
    for K, E, d in [(1, 8, 256), (8, 1024, 2048), (2, 100, 768)]:
        R, _, x = route_case(cuda_device, 40 + K, 3, E=E, d=d)
        idx, w, gamma, _ = lib.moe_route_topk(R, None, x, K)
        torch.cuda.synchronize()
        for t in range(3):
            l, p, oi, ow, og = O.route(bits16(R), f64(x)[t], K)
            if topk_gap(l, K) > TIE_GAP:
                assert idx[t].cpu().tolist() == oi.tolist()
                assert np.allclose(w[t].cpu().numpy(), ow, rtol=1e-5, atol=1e-6)
            assert float(gamma[t]) == 1.0


@pytest.mark.parametrize("B,d", [(1, 4096), (3, 4096), (16, 1024), (257, 256)])
def test_rmsnorm_matches_oracle(cuda_device, B, d):
    """bgq_rmsnorm: a[b] = bf16(h[b] / sqrt(mean(h[b]^2) + eps) * rho), per row."""
    h = synth.activations(9, d + B, B, d, device=cuda_device).float() * 3.0 - 0.5
    rho = synth.rho(9, 0, d, device=cuda_device)
    a = lib.bgq_rmsnorm(h, rho, 1e-6)
    a1 = lib.bgq_rmsnorm(h, None, 1e-6)
    torch.cuda.synchronize()
    for b in range(B):
        ref = O.rmsnorm(f64(h)[b], bits16(rho), 1e-6)
        assert_bf16_output(f64(a)[b], ref, b)
        assert_bf16_output(f64(a1)[b], O.rmsnorm(f64(h)[b], None, 1e-6), b)


@pytest.mark.parametrize("n", [1, 4096, 3 * 4096 + 7])
def test_residual_add(cuda_device, n):
    """bgq_residual_add: h += delta elementwise in fp32 (exact: one rounding each)."""
    h = torch.randn(n, generator=torch.Generator().manual_seed(n)).to(cuda_device)
    delta = torch.randn(n, generator=torch.Generator().manual_seed(n + 1)).to(cuda_device)
    ref = h.cpu() + delta.cpu()
    lib.bgq_residual_add(h, delta)
    torch.cuda.synchronize()
    assert torch.equal(h.cpu(), ref)
