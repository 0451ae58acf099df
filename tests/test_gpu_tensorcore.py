"""GPU parity of the tensor-core (tcgen05) grouped GEMM: experts that receive
16 or more tokens are computed as dense GEMMs with weights dequantised to
fp16. Tolerances as in the other parity tests."""

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from oracle import bgq_oracle as O
from tests.helpers import TC_OWN_TOL, ExpertSource, assert_bf16_output, bits16, f64, rel_l2
from tests.test_gpu_layer import build_layer, expert_binding

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,f,bits,B", [(4096, 1024, 4, 16), (4096, 1024, 4, 64), (1024, 512, 4, 37),
                                        (2048, 1024, 2, 24), (512, 256, 4, 130),
                                        # 256 tokens: four 64-column epilogue passes, each between cluster barriers
                                        (1024, 512, 4, 256), (1024, 512, 2, 200),
                                        # 3072 x 512: six gate/up K steps per CTA (a copy stage of four,
                                        # then one of two), two down steps per CTA
                                        (3072, 512, 4, 48)])
def test_expert_tensorcore_matches_oracle(cuda_device, d, f, bits, B):
    shape = synth.PoolShape(d, f, 1, bits)
    q, sb = synth.expert_pool_range(91, 0, shape, 0, 1, device=cuda_device)
    ex = expert_binding(q[0], sb[0], shape)
    x = synth.activations(91, d + B, B, d, device=cuda_device)
    y, yf = lib.moe_expert_swiglu(ex, x, want_f32=True)
    torch.cuda.synchronize()
    mats = [(m[0].cpu().numpy(), bits16(m[1])) for m in synth.expert_matrices(q[0], sb[0], shape)]
    xd = f64(x)
    for t in sorted({0, 1, B // 2, B - 1}):
        ref = O.expert_swiglu(*mats, bits, xd[t])
        assert_bf16_output(f64(y)[t], ref, t, own_tol=TC_OWN_TOL)
        assert rel_l2(f64(yf)[t], ref) <= 1e-3, t


def test_expert_tensorcore_deterministic(cuda_device):
    shape = synth.PoolShape(4096, 1024, 1, 4)
    q, sb = synth.expert_pool_range(92, 0, shape, 0, 1, device=cuda_device)
    ex = expert_binding(q[0], sb[0], shape)
    x = synth.activations(92, 0, 32, 4096, device=cuda_device)
    a = lib.moe_expert_swiglu(ex, x)[0].clone()
    b = lib.moe_expert_swiglu(ex, x)[0]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("bits,B", [(4, 80), (2, 64)])
def test_skewed_routing_sends_every_token_to_four_experts(cuda_device, bits, B):
    """Router rows 0..3 aligned with a component shared by all tokens: every
    token selects experts 0, 1, 2, 3, so the four routed experts (and the
    shared one) get >= 64 tokens each and run on the tensor-core path."""
    E, d, f, K = 64, 1024, 512, 4
    shape = synth.PoolShape(d, f, E, bits)
    L, t = build_layer(17, 0, shape, K, cuda_device)
    base = synth.activations(17, 1, 1, d, device=cuda_device)[0].float()
    noise = synth.activations(17, 2, B, d, device=cuda_device).float()
    x = (base[None, :] + 0.1 * noise).to(torch.bfloat16)
    for e, c in enumerate([1.0, 0.9, 0.8, 0.7]):
        t["router"][e] = (0.05 * c * base.sign()).to(torch.bfloat16)
    out, out_f32, idx, w, gamma = lib.moe_layer_forward(L, x, want_f32=True, want_route=True)
    torch.cuda.synchronize()
    assert torch.all(idx.cpu() == torch.tensor([0, 1, 2, 3], dtype=torch.int32))
    src = ExpertSource(17, 0, shape)
    Rb, Gb, xd = bits16(t["router"]), bits16(t["shared_gate"]), f64(x)
    for tok in sorted({0, B // 3, B - 1}):
        ref, oi, ow, og = O.moe_layer(Rb, Gb, src, src(E), bits, xd[tok], K)
        assert oi.tolist() == [0, 1, 2, 3]
        assert_bf16_output(f64(out)[tok], ref, tok, own_tol=TC_OWN_TOL)
        assert rel_l2(f64(out_f32)[tok], ref) <= 1e-3, tok
    # the same tokens one by one (grouped-GEMV path) agree within tolerance
    for tok in (0, B - 1):
        o1 = lib.moe_layer_forward(L, x[tok:tok + 1].contiguous(), want_f32=True)[1]
        assert rel_l2(f64(o1)[0], f64(out_f32)[tok]) <= 1e-3
