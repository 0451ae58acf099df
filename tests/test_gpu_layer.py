"""GPU parity of the SwiGLU expert, the MoE layer and the decode stack
against the fp64 oracle (same tolerances as the GEMV tests)."""

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from oracle import bgq_oracle as O
from tests.helpers import (REL_L2_TOL, TIE_GAP, ExpertSource, assert_bf16_output, bits16, check_topk_valid, f64,
                           own_tol_for, rel_l2, topk_gap)

pytestmark = pytest.mark.gpu


def expert_binding(q_row, sb_row, shape):
    mats = synth.expert_matrices(q_row, sb_row, shape)
    dims = [(shape.f, shape.d), (shape.f, shape.d), (shape.d, shape.f)]
    return lib.Expert(*[lib.QMatrix(m[0], m[1], r, c, shape.bits) for m, (r, c) in zip(mats, dims)])


@pytest.mark.parametrize("d,f,bits,B", [(4096, 1024, 4, 1), (4096, 1024, 4, 11), (4096, 1024, 2, 3),
                                        (512, 256, 4, 17), (1024, 2048, 2, 1)])
def test_expert_matches_oracle(cuda_device, d, f, bits, B):
    shape = synth.PoolShape(d, f, 1, bits)
    q, sb = synth.expert_pool_range(77, 0, shape, 0, 1, device=cuda_device)
    ex = expert_binding(q[0], sb[0], shape)
    x = synth.activations(77, d, B, d, device=cuda_device)
    y, yf = lib.moe_expert_swiglu(ex, x, want_f32=True)
    torch.cuda.synchronize()
    mats = [(m[0].cpu().numpy(), bits16(m[1])) for m in synth.expert_matrices(q[0], sb[0], shape)]
    xd = f64(x)
    for t in range(B):
        ref = O.expert_swiglu(*mats, bits, xd[t])
        assert_bf16_output(f64(y)[t], ref, t, own_tol=own_tol_for(B))
        assert rel_l2(f64(yf)[t], ref) <= (2e-4 if B < 16 else 1e-3)  # unrounded fp32 output
    assert torch.equal(y, yf.to(torch.bfloat16))


def build_layer(seed, layer, shape, K, dev, with_gate=True):
    t = synth.layer_tensors(seed, layer, shape, device=dev, with_gate=with_gate)
    E = shape.E
    L = lib.MoELayer(shape.d, shape.f, E, K, shape.bits, t["router"], t["shared_gate"], t["pool_q"][:E],
                     t["pool_sb"][:E], t["pool_q"][E], t["pool_sb"][E])
    return L, t


def oracle_layer_token(t, src, shape, K, x_tok, gpu_idx=None):
    """Oracle layer output for one token; near-tie tokens use the GPU's expert set."""
    Rb = bits16(t["router"])
    Gb = None if t["shared_gate"] is None else bits16(t["shared_gate"])
    logits = O.route(Rb, x_tok, K, Gb)[0]
    force = None
    if gpu_idx is not None and topk_gap(logits, K) <= TIE_GAP:
        check_topk_valid(gpu_idx, logits, K)
        force = gpu_idx
    out, idx, w, gamma = O.moe_layer(Rb, Gb, src, src(shape.E), shape.bits, x_tok, K, force_idx=force)
    return out, idx, w, gamma, logits


@pytest.mark.parametrize("E,d,f,K,bits,B", [
    (16, 256, 128, 4, 4, 1),
    (16, 256, 128, 4, 4, 40),  # several 8-token tasks per expert
    (8, 512, 256, 2, 2, 13),
    (64, 1024, 512, 4, 4, 64),
    (32, 2048, 1024, 8, 4, 5),
    # batch 1 at shapes the persistent kernel takes (rows of d read by all 32 lanes)
    (16, 1024, 256, 4, 4, 1),
    (8, 2048, 512, 2, 2, 1),
    (64, 1024, 512, 8, 4, 1),
    # limits and degenerate cases: 1024 experts with top-8 (the largest the
    # kernels take), every expert selected (E == K), a single expert (K == 1)
    (1024, 256, 128, 8, 4, 3),
    (1024, 1024, 256, 8, 4, 1),
    (4, 256, 128, 4, 4, 2),
    (4, 1024, 256, 4, 4, 1),
    (16, 512, 256, 1, 4, 9),
    (16, 1024, 256, 1, 4, 1),
    # down rows of 2048 columns at 4 bits: the per-task down kernel, then a
    # separate combine launch
    (8, 512, 2048, 2, 4, 3),
])
def test_small_layer_matches_oracle(cuda_device, E, d, f, K, bits, B):
    shape = synth.PoolShape(d, f, E, bits)
    L, t = build_layer(5, 0, shape, K, cuda_device)
    # spread the tiny router's logits like the 4096-wide one
    t["router"].copy_((t["router"].float() * np.sqrt(4096 / d)).to(torch.bfloat16))
    x = synth.activations(5, 2, B, d, device=cuda_device)
    out, out_f32, idx, w, gamma = lib.moe_layer_forward(L, x, want_f32=True, want_route=True)
    torch.cuda.synchronize()
    src = ExpertSource(5, 0, shape)
    xd = f64(x)
    for tok in range(B):
        gi = idx[tok].cpu().numpy()
        ref, oi, ow, og, logits = oracle_layer_token(t, src, shape, K, xd[tok], gi)
        if topk_gap(logits, K) > TIE_GAP:
            assert gi.tolist() == oi.tolist()
        assert_bf16_output(f64(out)[tok], ref, tok, own_tol=own_tol_for(B))
        assert rel_l2(f64(out_f32)[tok], ref) <= (5e-4 if B < 16 else 1e-3), tok
        assert abs(float(gamma[tok]) - og) <= 1e-6


@pytest.fixture(scope="module")
def full_layer(cuda_device):
    shape = synth.PoolShape(4096, 1024, 512, 4)
    L, t = build_layer(0, 0, shape, 4, cuda_device)
    return shape, L, t


@pytest.mark.parametrize("B,sample", [(1, [0]), (4, [0, 3]), (16, [0, 9, 15]), (64, [0, 31, 63]),
                                      (256, [0, 130, 255])])  # the largest batch: the shared expert's 256 tokens on tensor cores
def test_full_layer_matches_oracle_on_sampled_tokens(cuda_device, full_layer, B, sample):
    shape, L, t = full_layer
    x = synth.activations(0, 100 + B, B, shape.d, device=cuda_device)
    out, _, idx, w, gamma = lib.moe_layer_forward(L, x, want_route=True)
    torch.cuda.synchronize()
    src = ExpertSource(0, 0, shape)
    xd = f64(x)
    for tok in sample:
        gi = idx[tok].cpu().numpy()
        ref, oi, ow, og, logits = oracle_layer_token(t, src, shape, 4, xd[tok], gi)
        if topk_gap(logits, 4) > TIE_GAP:
            assert gi.tolist() == oi.tolist()
            assert np.allclose(w[tok].cpu().numpy(), ow, rtol=1e-5, atol=1e-6)
        assert_bf16_output(f64(out)[tok], ref, tok, own_tol=own_tol_for(B))
    # every token: valid routing, weights sum to 1
    assert torch.all((idx >= 0) & (idx < 512))
    assert torch.allclose(w.sum(dim=1), torch.ones(B, device=cuda_device), atol=1e-6)


def test_layer_batch_equals_single_bitwise(cuda_device, full_layer):
    """Grouping tokens by expert does not change any token's result."""
    shape, L, t = full_layer
    x = synth.activations(0, 900, 12, shape.d, device=cuda_device)
    ob = lib.moe_layer_forward(L, x)[0]
    for tok in range(12):
        o1 = lib.moe_layer_forward(L, x[tok:tok + 1].contiguous())[0]
        assert torch.equal(ob[tok].view(torch.int16), o1[0].view(torch.int16)), tok


def test_layer_workspace_reused_across_batches(cuda_device, full_layer):
    """One workspace sized for the largest batch serves calls of several batch
    sizes (every region a call reads is written earlier in the same call or
    left at zero by the previous one, whatever its layout) and gives the bits
    of a fresh one."""
    shape, L, t = full_layer
    ws = lib.workspace(lib.moe_layer_workspace_bytes(L, 100), cuda_device)
    for B in (100, 64, 1, 100, 64):
        x = synth.activations(0, 700 + B, B, shape.d, device=cuda_device)
        a = lib.moe_layer_forward(L, x, ws=ws)[0].clone()
        b = lib.moe_layer_forward(L, x)[0]
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), B
    assert lib.read_device_status(ws) == lib.OK


def test_batch1_calls_in_a_row_share_a_workspace(cuda_device, full_layer):
    """The batch-1 kernel exchanges the routing logits as words tagged with the
    layer; the last CTA of every launch clears them, so consecutive calls on
    one workspace (different inputs, same tags) give the bits of fresh
    workspaces and never read the previous call's logits."""
    shape, L, t = full_layer
    ws = lib.workspace(lib.moe_layer_workspace_bytes(L, 1), cuda_device)
    for call in range(4):
        x = synth.activations(0, 950 + call, 1, shape.d, device=cuda_device)
        a, _, ia, _, _ = lib.moe_layer_forward(L, x, ws=ws, want_route=True)
        a, ia = a.clone(), ia.clone()
        b, _, ib, _, _ = lib.moe_layer_forward(L, x, want_route=True)
        torch.cuda.synchronize()
        assert torch.equal(ia, ib), call
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), call
    assert lib.read_device_status(ws) == lib.OK


def test_layer_deterministic(cuda_device, full_layer):
    shape, L, t = full_layer
    x = synth.activations(0, 901, 16, shape.d, device=cuda_device)
    ws = lib.workspace(lib.moe_layer_workspace_bytes(L, 16), cuda_device)
    a = lib.moe_layer_forward(L, x, ws=ws)[0].clone()
    b = lib.moe_layer_forward(L, x, ws=ws)[0]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert lib.read_device_status(ws) == lib.OK


def test_layer_expert_permutation(cuda_device):
    """Permuting the router rows together with the expert pool leaves the output unchanged."""
    shape = synth.PoolShape(512, 256, 16, 4)
    L, t = build_layer(8, 0, shape, 4, cuda_device)
    x = synth.activations(8, 0, 6, shape.d, device=cuda_device)
    out, _, idx, _, _ = lib.moe_layer_forward(L, x, want_route=True)
    perm = torch.randperm(16, generator=torch.Generator().manual_seed(0)).to(cuda_device)
    R2 = t["router"][perm].contiguous()
    q2 = t["pool_q"][:16][perm].contiguous()
    sb2 = t["pool_sb"][:16][perm].contiguous()
    L2 = lib.MoELayer(shape.d, shape.f, 16, 4, 4, R2, t["shared_gate"], q2, sb2, t["pool_q"][16], t["pool_sb"][16])
    out2, _, idx2, _, _ = lib.moe_layer_forward(L2, x, want_route=True)
    torch.cuda.synchronize()
    assert torch.equal(perm[idx2.long()], idx.long())
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("B", [1, 4])
def test_layer_all_equal_logits_pick_lowest_indices(cuda_device, B):
    """A zero router makes all 512 logits equal: the top-4 are experts 0..3
    (ties to the lower index, the oracle's stable top-K), each weighted 1/4.
    Every logit is then a candidate of the block top-K (its path for more
    than 32 candidates): batch 1 runs the persistent kernel, batch 4 the
    cooperative router."""
    shape = synth.PoolShape(1024, 256, 512, 4)
    L, t = build_layer(41, 0, shape, 4, cuda_device)
    t["router"].zero_()
    x = synth.activations(41, 1, B, shape.d, device=cuda_device)
    out, _, idx, w, _ = lib.moe_layer_forward(L, x, want_route=True)
    torch.cuda.synchronize()
    assert idx.cpu().tolist() == [[0, 1, 2, 3]] * B
    assert torch.all(w == 0.25)
    src = ExpertSource(41, 0, shape)
    xd = f64(x)
    for tok in range(B):
        ref, oi, _, _, _ = oracle_layer_token(t, src, shape, 4, xd[tok])
        assert oi.tolist() == [0, 1, 2, 3]
        assert_bf16_output(f64(out)[tok], ref, tok, own_tol=own_tol_for(B))


# ------------------------------------------------------------------ stack
def stack_case(dev, seed, n_layers, shape, K):
    built = [build_layer(seed, l, shape, K, dev) for l in range(n_layers)]
    rhos = [synth.rho(seed, l, shape.d, device=dev) for l in range(n_layers)]
    return built, rhos


def oracle_stack(seed, built, rhos, shape, K, x_bits, gpu_idx):
    layers = []
    for l, (L, t) in enumerate(built):
        layers.append(dict(router=bits16(t["router"]), shared_gate=bits16(t["shared_gate"]), rho=bits16(rhos[l]),
                           get_expert=ExpertSource(seed, l, shape), shared=None))
        layers[-1]["shared"] = layers[-1]["get_expert"](shape.E)
    # near ties: evaluate with the GPU's expert set (checked valid inside)
    h = O.bf16_to_f64(x_bits)
    force = []
    for l, L in enumerate(layers):
        a = O.round_bf16(O.rmsnorm(h, L["rho"]))
        logits = O.route(L["router"], a, K, L["shared_gate"])[0]
        if topk_gap(logits, K) <= TIE_GAP:
            check_topk_valid(gpu_idx[l], logits, K)
            force.append(np.asarray(gpu_idx[l]))
        else:
            force.append(None)
        out, _, _, _ = O.moe_layer(L["router"], L["shared_gate"], L["get_expert"], L["shared"], shape.bits, a, K,
                                   force_idx=force[-1])
        h = h + out
    return O.stack_token(layers, x_bits, shape.bits, K, force_idx=force)


@pytest.mark.parametrize("n_layers,d,f,E,bits", [(6, 512, 256, 16, 4), (6, 1024, 256, 16, 4),
                                                 (4, 4096, 1024, 512, 4), (3, 4096, 1024, 512, 2)])
def test_stack_matches_oracle(cuda_device, n_layers, d, f, E, bits):
    K = 4
    shape = synth.PoolShape(d, f, E, bits)
    built, rhos = stack_case(cuda_device, 3, n_layers, shape, K)
    if d != 4096:
        for L, t in built:
            t["router"].copy_((t["router"].float() * np.sqrt(4096 / d)).to(torch.bfloat16))
    st = lib.Stack([b[0] for b in built], rhos)
    x = synth.activations(3, 5, 1, d, device=cuda_device)[0]
    x_next = lib.alloc(x.shape, x.dtype, x.device)
    h = lib.alloc((d,), torch.float32, cuda_device)
    idx = lib.alloc((n_layers, K), torch.int32, cuda_device)
    lib.moe_stack_decode(st, x, 1e-6, x_next=x_next, h_out=h, idx_out=idx)
    torch.cuda.synchronize()
    xo, ho, oidx = oracle_stack(3, built, rhos, shape, K, bits16(x), idx.cpu().numpy())
    assert rel_l2(f64(h), ho) <= REL_L2_TOL
    # x_next against the oracle's unrounded normalised residual. Every layer
    # rounds its normalised input to bf16 on both sides, from slightly
    # different values, so the stack's own error may exceed one layer's.
    assert_bf16_output(O.bf16_to_f64(bits16(x_next)), O.rmsnorm(ho, None), "x_next", own_tol=REL_L2_TOL)
    assert rel_l2(O.bf16_to_f64(bits16(x_next)), O.bf16_to_f64(xo)) <= REL_L2_TOL


def test_stack_tokens_in_a_row_share_a_workspace(cuda_device):
    """Decode steps on one workspace (the next token's input is the previous
    token's output) give the bits of steps on fresh workspaces."""
    K = 4
    shape = synth.PoolShape(1024, 256, 16, 4)
    built, rhos = stack_case(cuda_device, 4, 3, shape, K)
    st = lib.Stack([b[0] for b in built], rhos)
    ws = lib.workspace(st.ws_bytes, cuda_device)
    x = synth.activations(4, 6, 1, shape.d, device=cuda_device)[0].clone()
    for step in range(3):
        xa = lib.alloc(x.shape, x.dtype, x.device)
        xb = lib.alloc(x.shape, x.dtype, x.device)
        lib.moe_stack_decode(st, x, 1e-6, ws=ws, x_next=xa)
        lib.moe_stack_decode(st, x, 1e-6, x_next=xb)
        torch.cuda.synchronize()
        assert torch.equal(xa.view(torch.int16), xb.view(torch.int16)), step
        x = xa
    assert lib.read_device_status(ws) == lib.OK


def test_bounded_wait_times_out_cleanly(cuda_device):
    """A grid-wide wait on a counter nothing sets gives up after its limit and
    reports BGQ_ERR_TIMEOUT through the status word; the context stays usable."""
    ws = lib.workspace(4096, cuda_device)
    lib.wait_selftest(ws, 2_000_000)  # 2 ms
    assert lib.read_device_status(ws) == lib.ERR_TIMEOUT
    assert lib.read_device_status(ws) == lib.OK  # reading clears it
    x = torch.ones(16, device=cuda_device)
    assert float((x * 2).sum()) == 32.0
