"""GPU parity of the 8-bit GEMV (q8_gemv: int8 MLP / QKV weights with a
(scale, bias) pair per group of 64, and the per-row FC2 format) against the
fp64 oracle.

Tolerances: the same as every GEMV (bf16 out, fp32 accumulate): rel-L2 <= 2e-3
against the unrounded oracle for outputs of >= 512 elements, the kernel's own
error <= 1e-3 against the oracle rounded to bf16, each element within one bf16
spacing. Column probes are bit-exact (s*q + b is exact in fp32 for these
values, so the single bf16 rounding matches the oracle's).
"""

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from oracle import bgq_oracle as O
from tests.helpers import assert_bf16_output, bits16, f64

pytestmark = pytest.mark.gpu


def make_matrix8(seed, rows, cols, group, dev):
    q, sb = synth.qmatrix(seed, rows, cols, 8, device=dev, group=group)
    return lib.QMatrix(q, sb, rows, cols, 8, group), q, sb


Q8_CASES = [
    # (rows, cols, group, batch)
    (1024, 4096, 64, 1),  # the same shape as the 4-bit single-GEMV workload
    (4096, 4096, 64, 1),  # a square projection (QKV-like), 16.8 MB of codes
    (1000, 4096, 64, 3),  # ragged rows
    (4096, 1024, 64, 2),  # FC2-like shape: 2 parts per lane
    (333, 512, 64, 8),  # one part per lane
    (200, 256, 64, 5),  # 16 lanes per row
    (64, 64, 64, 2),  # 4 lanes per row, 8 rows per warp pass
    (96, 12288, 64, 9),  # 12 parts per lane (two register batches); 7 + 2 inputs per launch
    (256, 4096, 64, 64),  # largest batch: 8 launches of 8
    (1024, 4096, 4096, 1),  # per-row scale/bias (FC2 format)
    (777, 1024, 1024, 6),  # per-row, ragged
    (128, 128, 128, 1),  # per-row, 8 lanes per row
    (300, 1536, 64, 3),  # 3 parts per lane: one row per item
    (50, 2560, 2560, 3),  # 5 parts per lane, per row
    (5000, 1024, 64, 3),  # streaming kernel: several rows per warp, four rows packed per item
    (20000, 256, 256, 4),  # streaming kernel: 16 lanes per row, eight row pairs per item; per row
    (16384, 4096, 64, 2),  # one-shot kernel over several waves
]


@pytest.mark.parametrize("rows,cols,group,batch", Q8_CASES)
def test_q8_gemv_matches_oracle(cuda_device, rows, cols, group, batch):
    W, q, sb = make_matrix8(300 + rows + cols + group, rows, cols, group, cuda_device)
    x = synth.activations(9, rows + batch, batch, cols, device=cuda_device)
    y = lib.q8_gemv(W, x)
    torch.cuda.synchronize()
    ref = O.gemv(q.cpu().numpy(), bits16(sb), 8, f64(x), group=group)
    got = f64(y)
    for t in range(batch):
        assert_bf16_output(got[t], ref[t], t)


@pytest.mark.parametrize("group", [64, 2048])
def test_q8_gemv_column_probe(cuda_device, group):
    """x = e_k returns column k of the dequantised W, rounded once to bf16, bit for bit."""
    rows, cols = 512, 2048
    W, q, sb = make_matrix8(41, rows, cols, group, cuda_device)
    ks = [0, 1, 3, 4, 63, 64, 1000, 2047]
    x = torch.zeros(len(ks), cols, dtype=torch.bfloat16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = lib.q8_gemv(W, x.to(cuda_device))
    torch.cuda.synchronize()
    Wd = O.dequant(q.cpu().numpy(), bits16(sb), 8, group)
    expect = O.f64_to_bf16_bits(Wd[:, ks].T)
    assert np.array_equal(bits16(y), expect)


def test_q8_gemv_signed_int8(cuda_device):
    """Symmetric signed int8 weights (w = c*s) in their affine storage q = c + 128, b = -128*s."""
    rows, cols = 768, 4096
    g = torch.Generator().manual_seed(12)
    c = torch.randint(-128, 128, (rows, cols), generator=g)
    s = (torch.rand(rows, cols // 64, generator=g) * 0.018 + 0.002).to(torch.bfloat16)
    sb = torch.stack([s, (s.float() * -128.0).to(torch.bfloat16)], dim=-1)
    qb = (c + 128).to(torch.int64).reshape(rows, cols // 4, 4)
    words = qb[..., 0] | (qb[..., 1] << 8) | (qb[..., 2] << 16) | (qb[..., 3] << 24)
    q = torch.where(words >= 2 ** 31, words - 2 ** 32, words).to(torch.int32)
    x = synth.activations(13, 0, 2, cols)
    W = lib.QMatrix(q.to(cuda_device), sb.to(cuda_device), rows, cols, 8)
    y = lib.q8_gemv(W, x.to(cuda_device))
    torch.cuda.synchronize()
    ref = (c.double() * s.double().repeat_interleave(64, dim=1)) @ torch.from_numpy(f64(x)).T
    ref = ref.T.numpy()
    assert np.allclose(O.gemv(q.numpy(), bits16(sb), 8, f64(x)), ref, rtol=1e-12, atol=1e-12)
    for t in range(2):
        assert_bf16_output(f64(y)[t], ref[t], t)


def test_q8_gemv_deterministic_and_batch_invariant(cuda_device):
    rows, cols = 2048, 4096
    W, q, sb = make_matrix8(5, rows, cols, 64, cuda_device)
    x = synth.activations(14, 0, 11, cols, device=cuda_device)
    a = lib.q8_gemv(W, x).clone()
    b = lib.q8_gemv(W, x)
    one = [lib.q8_gemv(W, x[t:t + 1]).clone() for t in (0, 5, 10)]
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    for i, t in enumerate((0, 5, 10)):
        assert torch.equal(a[t:t + 1], one[i])


def test_q8_gemv_zero_input_and_zero_codes(cuda_device):
    rows, cols = 300, 1024
    W, q, sb = make_matrix8(6, rows, cols, 64, cuda_device)
    y = lib.q8_gemv(W, torch.zeros(1, cols, dtype=torch.bfloat16, device=cuda_device))
    torch.cuda.synchronize()
    assert torch.count_nonzero(y.float()) == 0
    # all codes zero: y_n = sum_g b_ng * sum_{k in g} x_k
    zq = torch.zeros_like(q)
    x = synth.activations(15, 0, 1, cols, device=cuda_device)
    Wz = lib.QMatrix(zq, sb, rows, cols, 8)
    yz = lib.q8_gemv(Wz, x)
    torch.cuda.synchronize()
    ref = O.gemv(zq.cpu().numpy(), bits16(sb), 8, f64(x))
    assert_bf16_output(f64(yz)[0], ref[0], "zero codes")
