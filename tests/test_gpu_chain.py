"""GPU parity of bgq_gemv_chain: the decoder's projections around the MoE
block as a chain of dependent group-quantized GEMVs (dependent launches).

Against the fp64 oracle (oracle.gemv_chain, which rounds the inner vectors to
bf16 as the chain does): bf16 outputs within the workload tolerance
(assert_bf16_output, own error 1.5e-3 as the inner roundings may fall on
either side of a bf16 boundary), fp32 outputs within rel-L2 5e-4. Against the
separate calls (bgq_rmsnorm, then q4_gemv / q2_gemv per step): the same bits.
"""

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from oracle import bgq_oracle as O
from tests.helpers import assert_bf16_output, bits16, f64, rel_l2

pytestmark = pytest.mark.gpu

EPS = 1e-6


def chain_mats(seed, dims, bits, dev):
    """W_i: dims[i+1] x dims[i]; returns the library matrices and the oracle's (q, sb) pairs."""
    mats, pairs = [], []
    for i in range(len(dims) - 1):
        rows, cols = dims[i + 1], dims[i]
        q, sb = synth.qmatrix(seed + 31 * i, rows, cols, bits, device=dev)
        mats.append(lib.QMatrix(q, sb, rows, cols, bits))
        pairs.append((q.cpu().numpy(), bits16(sb)))
    return mats, pairs


CHAIN_CASES = [
    # (dims, bits, batch, norm, residual); W_i is dims[i+1] x dims[i]
    ([4096, 4096, 4096], 4, 1, True, True),  # an attention-sized projection, then o_proj + residual
    ([4096, 4096, 4096], 4, 3, True, True),
    ([4096, 4096, 4096], 4, 8, True, True),
    ([4096, 12288, 4096], 4, 2, True, True),  # stacked q/k/v rows feeding a 12288-column step
    ([2048, 1024, 3072, 1000], 4, 5, False, False),  # three steps, ragged last rows
    ([4096, 4096, 4096], 2, 2, True, True),
    ([1024, 4096, 1024], 2, 8, True, False),
    ([4096, 4096], 4, 4, False, True),  # one step with the residual
]


@pytest.mark.parametrize("dims,bits,batch,norm,residual", CHAIN_CASES)
def test_chain_matches_oracle(cuda_device, dims, bits, batch, norm, residual):
    seed = 500 + sum(dims) + batch
    mats, pairs = chain_mats(seed, dims, bits, cuda_device)
    x = synth.activations(seed, 1, batch, dims[0], device=cuda_device)
    rho = synth.rho(seed, 0, dims[0], device=cuda_device) if norm else None
    out, out_f32 = lib.gemv_chain(mats, x, norm=norm, rho=rho, eps=EPS, residual=residual, want_f32=True)
    torch.cuda.synchronize()
    ref = O.gemv_chain(pairs, bits, bits16(x), norm=norm, rho_bits=None if rho is None else bits16(rho),
                       eps=EPS, residual=residual)
    got, gotf = f64(out), f64(out_f32)
    for t in range(batch):
        assert_bf16_output(got[t], ref[t], t, own_tol=1.5e-3)
        assert rel_l2(gotf[t], ref[t]) <= 5e-4, (t, rel_l2(gotf[t], ref[t]))


@pytest.mark.parametrize("bits", [4, 2])
def test_chain_has_the_bits_of_the_separate_calls(cuda_device, bits):
    """rmsnorm (bgq_rmsnorm on the widened x), then one GEMV per step: the
    chain's output bits; with the residual, the fp32 sum of x and the last
    step's fp32 output."""
    dims, B = [4096, 4096, 2048, 4096], 3
    mats, _ = chain_mats(77 + bits, dims, bits, cuda_device)
    x = synth.activations(78, 1, B, dims[0], device=cuda_device)
    rho = synth.rho(79, 0, dims[0], device=cuda_device)
    gemv = lib.q4_gemv if bits == 4 else lib.q2_gemv
    v = lib.bgq_rmsnorm(x.float(), rho, EPS)
    for W in mats:
        v = gemv(W, v)
    out, out_f32 = lib.gemv_chain(mats, x, norm=True, rho=rho, eps=EPS, want_f32=True)
    res, res_f32 = lib.gemv_chain(mats, x, norm=True, rho=rho, eps=EPS, residual=True, want_f32=True)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), v.view(torch.int16))
    assert torch.equal(out.view(torch.int16), out_f32.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(res_f32, x.float() + out_f32)
    assert torch.equal(res.view(torch.int16), res_f32.to(torch.bfloat16).view(torch.int16))


def test_chain_of_one_step_is_the_gemv(cuda_device):
    mats, _ = chain_mats(90, [4096, 1000], 4, cuda_device)
    x = synth.activations(91, 1, 8, 4096, device=cuda_device)
    out, _ = lib.gemv_chain(mats, x)
    y = lib.q4_gemv(mats[0], x)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), y.view(torch.int16))


def test_chain_reuses_its_workspace(cuda_device):
    """Each call clears the step counter: calls on one workspace give the
    bits of fresh workspaces, and the status word stays ok."""
    dims = [4096, 4096, 4096]
    mats, _ = chain_mats(93, dims, 4, cuda_device)
    ws = lib.workspace(lib.gemv_chain_workspace_bytes(mats, 4), cuda_device)
    rho = synth.rho(94, 0, 4096, device=cuda_device)
    for call in range(3):
        x = synth.activations(95, call, 4, 4096, device=cuda_device)
        a, _ = lib.gemv_chain(mats, x, norm=True, rho=rho, residual=True, ws=ws)
        a = a.clone()
        b, _ = lib.gemv_chain(mats, x, norm=True, rho=rho, residual=True)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), call
    assert lib.read_device_status(ws) == lib.OK
