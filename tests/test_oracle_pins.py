"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Hand-computed brute-force cases (tests/golden), closed forms, special inputs,
library special cases (torch float64 routines), invariants of the method,
and size figures printed on the Flash-MoE page. The last block plants
plausible mistakes in the oracle and checks that some pin catches each one.
"""

import os
import re

import numpy as np
import pytest
import torch

from oracle import bgq_oracle as O
from bit_group_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers
def pack_rows(code_rows, bits):
    """Pack per-row code lists into uint32 words, column 0 in the lowest bits."""
    per = 32 // bits
    out = []
    for codes in code_rows:
        words = []
        for i in range(0, len(codes), per):
            w = 0
            for j, c in enumerate(codes[i:i + per]):
                w |= int(c) << (bits * j)
            words.append(w)
        out.append(words)
    return np.array(out, dtype=np.uint64).astype(np.uint32)


def bf16_bits(values):
    return O.f64_to_bf16_bits(np.asarray(values, dtype=np.float64))


def load_hand_cases():
    text = open(os.path.join(GOLDEN, "hand_gemv_2x64.txt"), encoding="utf-8").read()
    cases = []
    for block in re.split(r"\n(?=case )", text):
        lines = [l for l in block.splitlines() if l and not l.startswith("#")]
        if not lines or not lines[0].startswith("case "):
            continue
        head = lines[0].split()
        c = {"name": head[1], "bits": int(head[2].split("=")[1]), "cols": int(head[3].split("=")[1])}
        for l in lines[1:]:
            key, val = l.split(" ", 1)
            c[key] = val.strip()
        cases.append(c)
    return cases


def hand_case_arrays(c):
    bits, cols = c["bits"], c["cols"]
    rows = [[int(ch, 16) for ch in c["q0"]], [int(ch, 16) for ch in c["q1"]]]
    assert all(len(r) == cols for r in rows)
    q = pack_rows(rows, bits)
    sb = []
    for key in ("sb0", "sb1"):
        groups = [tuple(float(v) for v in g.split(",")) for g in c[key].split(";")]
        assert len(groups) == cols // 64
        sb.append([v for g in groups for v in g])
    sb = bf16_bits(sb).reshape(2, cols // 64, 2)
    spec = c["x"].split()
    x = np.zeros(cols)
    if spec[0] == "all":
        x[:] = float(spec[1])
    else:
        x[int(spec[1])] = 1.0
    y = np.array([float(v) for v in c["y"].split()])
    return q, sb, x, y


HAND = load_hand_cases()


# --------------------------------------------------------- A. hand cases
def check_hand_cases():
    assert len(HAND) >= 7
    for c in HAND:
        q, sb, x, y = hand_case_arrays(c)
        got = O.gemv(q, sb, c["bits"], x)
        assert np.array_equal(got, y), (c["name"], got, y)


def test_hand_cases():
    check_hand_cases()


# ------------------------------------------- A'. 8-bit hand cases (int8 MLP / QKV / FC2 format)
def load_hand_cases8():
    text = open(os.path.join(GOLDEN, "hand_gemv8.txt"), encoding="utf-8").read()
    cases = []
    for block in re.split(r"\n(?=case )", text):
        lines = [l for l in block.splitlines() if l and not l.startswith("#")]
        if not lines or not lines[0].startswith("case "):
            continue
        head = lines[0].split()
        c = {"name": head[1]}
        for kv in head[2:]:
            k, v = kv.split("=")
            c[k] = int(v)
        for l in lines[1:]:
            key, val = l.split(" ", 1)
            c[key] = val.strip()
        cases.append(c)
    return cases


def hand_case8_arrays(c):
    cols, group = c["cols"], c["group"]
    rows = [[int(c[k][2 * i:2 * i + 2], 16) for i in range(cols)] for k in ("q0", "q1")]
    q = pack_rows(rows, 8)
    sb = []
    for key in ("sb0", "sb1"):
        groups = [tuple(float(v) for v in g.split(",")) for g in c[key].split(";")]
        assert len(groups) == cols // group
        sb.append([v for g in groups for v in g])
    sb = bf16_bits(sb).reshape(2, cols // group, 2)
    spec = c["x"].split()
    x = np.zeros(cols)
    if spec[0] == "all":
        x[:] = float(spec[1])
    else:
        x[int(spec[1])] = 1.0
    y = np.array([float(v) for v in c["y"].split()])
    return q, sb, x, y


HAND8 = load_hand_cases8()


def check_hand_cases8():
    assert len(HAND8) >= 8
    for c in HAND8:
        q, sb, x, y = hand_case8_arrays(c)
        got = O.gemv(q, sb, 8, x, group=c["group"])
        assert np.array_equal(got, y), (c["name"], got, y)


def test_hand_cases_8bit():
    check_hand_cases8()


def test_eight_bit_equals_four_bit_repack():
    """4-bit codes (0..15) repacked one per byte give the same oracle result at 8 bits."""
    q4, sb = synth.qmatrix(23, 6, 256, 4)
    codes = codes_by_string(q4.numpy(), 4)
    q8 = pack_rows(codes.tolist(), 8)
    x = O.round_bf16(np.random.default_rng(4).standard_normal(256))
    assert np.array_equal(O.gemv(q4.numpy(), sb, 4, x), O.gemv(q8, sb, 8, x))


def test_per_row_equals_uniform_groups():
    """One (scale, bias) per row equals the per-group format with that pair in every group."""
    q, sb_row = synth.qmatrix(24, 5, 512, 8, group=512)
    sb_groups = sb_row.repeat(1, 512 // 64, 1)  # [5][8][2], every group the row's pair
    x = O.round_bf16(np.random.default_rng(5).standard_normal(512))
    assert np.array_equal(O.gemv(q.numpy(), sb_row, 8, x, group=512), O.gemv(q.numpy(), sb_groups, 8, x))


def test_signed_int8_closed_form():
    """Symmetric int8 c (w = c*s) stored as q = c + 128 with bias -128*s dequantises to c*s exactly."""
    rng = np.random.default_rng(6)
    c = rng.integers(-128, 128, size=(3, 128))
    s = O.round_bf16(rng.uniform(0.001, 0.05, size=(3, 2)))
    sb = np.stack([s, -128.0 * s], axis=-1)  # -128*s is exact in bf16
    sbb = bf16_bits(sb)
    assert np.array_equal(O.bf16_to_f64(sbb), sb)
    q = pack_rows((c + 128).tolist(), 8)
    w = O.dequant(q, sbb, 8)
    assert np.array_equal(w, c * np.repeat(s, 64, axis=1))


# --------------------------------------------------------- bf16 rounding
def check_bf16_rounding():
    cases = {
        1.0: 0x3F80,
        -2.0: 0xC000,
        1.0 + 2 ** -8: 0x3F80,  # exact tie, even stays
        1.0 + 3 * 2 ** -8: 0x3F82,  # tie, rounds up to even
        1.0 + 2 ** -8 + 2 ** -30: 0x3F81,  # just above the tie
        0.1: 0x3DCD,
        3.0e38: 0x7F62,
    }
    for v, bits in cases.items():
        assert int(O.f64_to_bf16_bits(np.array([v]))[0]) == bits, (v, hex(bits))
    assert O.bf16_to_f64(np.array([0x3F80, 0xBFC0], dtype=np.uint16)).tolist() == [1.0, -1.5]
    # agreement with torch's float32 -> bf16 (RNE) for values exact in float32
    v = torch.randn(4096, generator=torch.Generator().manual_seed(1), dtype=torch.float32)
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(O.f64_to_bf16_bits(v.double().numpy()), ref)


def test_bf16_rounding():
    check_bf16_rounding()


# --------------------------------------------------- F. closed forms, packing
def codes_by_string(q_words, bits):
    """Codes read from a binary string of each word (independent of the oracle's shifts)."""
    w = np.asarray(q_words).astype(np.int64) & 0xFFFFFFFF
    per = 32 // bits
    out = np.zeros((w.shape[0], w.shape[1] * per), dtype=np.int64)
    for n in range(w.shape[0]):
        for i in range(w.shape[1]):
            s = format(int(w[n, i]), "032b")  # most significant bit first
            for j in range(per):
                lo = 32 - bits * (j + 1)
                out[n, i * per + j] = int(s[lo:lo + bits], 2)
    return out


def check_column_extraction(bits):
    q, sb = synth.qmatrix(11, 8, 256, bits)
    qn = q.numpy()
    sbv = O.bf16_to_f64(sb.view(torch.int16).numpy()).reshape(8, 4, 2)
    codes = codes_by_string(qn, bits)
    for k in (0, 1, 7, 8, 63, 64, 130, 255):
        x = np.zeros(256)
        x[k] = 1.0
        expect = codes[:, k] * sbv[:, k // 64, 0] + sbv[:, k // 64, 1]
        assert np.array_equal(O.gemv(qn, sb, bits, x), expect), k


@pytest.mark.parametrize("bits", [4, 2, 8])
def test_column_extraction(bits):
    check_column_extraction(bits)


def check_zero_codes_and_zero_scale():
    rng = np.random.default_rng(3)
    rows, cols = 4, 192
    x = O.round_bf16(rng.standard_normal(cols))
    sb = synth.qmatrix(5, rows, cols, 4)[1]
    sbv = O.bf16_to_f64(sb.view(torch.int16).numpy()).reshape(rows, 3, 2)
    xg = x.reshape(3, 64).sum(axis=1)
    # all codes zero: y_n = sum_g b_ng * sum_{k in g} x_k
    zq = np.zeros((rows, cols // 8), dtype=np.uint32)
    assert np.allclose(O.gemv(zq, sb, 4, x), sbv[:, :, 1] @ xg, rtol=1e-14, atol=1e-14)
    # scale zero: the codes do not matter
    sb0 = sb.clone()
    sb0[..., 0] = 0
    sbv0 = O.bf16_to_f64(sb0.view(torch.int16).numpy()).reshape(rows, 3, 2)
    q = synth.qmatrix(6, rows, cols, 4)[0].numpy()
    assert np.allclose(O.gemv(q, sb0, 4, x), sbv0[:, :, 1] @ xg, rtol=1e-14, atol=1e-14)


def test_zero_codes_and_zero_scale():
    check_zero_codes_and_zero_scale()


def test_two_bit_equals_four_bit_repack():
    q2, sb = synth.qmatrix(21, 6, 128, 2)
    codes = codes_by_string(q2.numpy(), 2)  # values 0..3
    q4 = pack_rows(codes.tolist(), 4)
    x = O.round_bf16(np.random.default_rng(0).standard_normal(128))
    assert np.array_equal(O.gemv(q2.numpy(), sb, 2, x), O.gemv(q4, sb, 4, x))


def test_gemv_matches_torch_float64():
    q, sb = synth.qmatrix(2, 64, 512, 4)
    x = synth.activations(2, 0, 1, 512)[0]
    xd = O.bf16_to_f64(x.view(torch.int16).numpy())
    # independent dequantisation with torch integer ops
    w = q.to(torch.int64) & 0xFFFFFFFF
    codes = torch.stack([(w >> (4 * j)) & 15 for j in range(8)], dim=-1).reshape(64, 512)
    s = sb[..., 0].double().repeat_interleave(64, dim=1)
    b = sb[..., 1].double().repeat_interleave(64, dim=1)
    y = ((codes.double() * s + b) @ torch.from_numpy(xd)).numpy()
    assert np.allclose(O.gemv(q, sb, 4, xd), y, rtol=1e-13, atol=1e-13)


# ------------------------------------------------ B. reordering identity
def test_fma_reordering_identity():
    """(q*s + b)*x == fma(q, s*x, b*x): exact in float64 for bf16 s, b, x.

    [Flash-MoE page, "FMA Dequant"] calls the reordering mathematically
    equivalent. In float32 the two differ by at most a few rounding units of
    the terms; checked here with torch float32 arithmetic.
    """
    rng = np.random.default_rng(7)
    n = 100000
    q = rng.integers(0, 16, n).astype(np.float64)
    s = O.round_bf16(rng.uniform(0.002, 0.02, n))
    b = O.round_bf16(-8 * s + 1e-4 * rng.standard_normal(n))
    x = O.round_bf16(rng.standard_normal(n))
    std = O.dot_terms_standard(q, s, b, x)
    reo = O.dot_terms_reordered(q, s, b, x)
    assert np.array_equal(std, reo)
    # float32: one fused multiply-add against the unfused standard form
    t = lambda a: torch.from_numpy(a).float()
    f_std = (t(q) * t(s) + t(b)) * t(x)
    f_reo = torch.addcmul(t(b) * t(x), t(q), t(s) * t(x))
    bound = 4 * 2.0 ** -24 * (np.abs(q * s * x) + np.abs(b * x))
    assert np.all(np.abs(f_std.double().numpy() - std) <= bound)
    assert np.all(np.abs(f_reo.double().numpy() - std) <= bound)


# ------------------------------------------------- C. routing invariants
def check_route_invariants():
    rng = np.random.default_rng(11)
    E, d = 64, 128
    R = bf16_bits(0.02 * rng.standard_normal((E, d)) * 8)
    G = bf16_bits(0.02 * rng.standard_normal(d))
    for t in range(20):
        x = O.round_bf16(rng.standard_normal(d))
        logits, p, idx, w, gamma = O.route(R, x, 4, G)
        chosen = logits[idx]
        others = np.delete(logits, idx)
        assert chosen.min() >= others.max()
        assert np.all(np.diff(chosen) <= 0)  # descending
        assert abs(w.sum() - 1.0) < 1e-12
        # closed form: renormalised top-K softmax == softmax of the chosen logits alone
        e = np.exp(chosen - chosen.max())
        assert np.allclose(w, e / e.sum(), rtol=1e-12, atol=0)
        assert np.isclose(p.sum(), 1.0)
        z = O.bf16_to_f64(G) @ x
        assert np.isclose(gamma, 1 / (1 + np.exp(-z)), rtol=1e-14)
    # planted exact ties: the lower index wins and comes first
    l = np.zeros(16)
    l[[3, 9, 12]] = 2.0
    l[[5, 14]] = 1.0
    assert O.topk_stable(l, 4).tolist() == [3, 9, 12, 5]


def test_route_invariants():
    check_route_invariants()


def test_route_matches_torch():
    rng = np.random.default_rng(12)
    R = bf16_bits(0.02 * rng.standard_normal((512, 256)) * 4)
    for t in range(10):
        x = O.round_bf16(rng.standard_normal(256))
        logits, p, idx, w, _ = O.route(R, x, 4)
        tl = torch.from_numpy(O.bf16_to_f64(R)) @ torch.from_numpy(x)
        tp = torch.softmax(tl, dim=0)
        order = torch.sort(tl, descending=True, stable=True).indices[:4]
        assert order.tolist() == idx.tolist()
        tw = tp[order] / tp[order].sum()
        assert np.allclose(tw.numpy(), w, rtol=1e-13)
        assert np.allclose(tp.numpy(), p, rtol=1e-13, atol=1e-300)


def check_silu():
    z = np.linspace(-30, 30, 2001)
    ref = torch.nn.functional.silu(torch.from_numpy(z)).numpy()
    assert np.allclose(O.silu(z), ref, rtol=1e-14, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0


def test_silu():
    check_silu()


def test_rmsnorm_closed_forms():
    h = np.full(64, 3.0)
    assert np.allclose(O.rmsnorm(h, None, 0.0), np.ones(64))
    h = np.array([3.0, 4.0] * 8)  # mean square 12.5
    got = O.rmsnorm(h, None, 1e-6)
    assert np.allclose(got, h / np.sqrt(12.5 + 1e-6), rtol=1e-15)
    rho = bf16_bits(np.linspace(0.5, 2.0, 16))
    assert np.allclose(O.rmsnorm(h, rho, 0.0), h / np.sqrt(12.5) * O.bf16_to_f64(rho), rtol=1e-15)


# ----------------------------------------- D. expert-permutation invariance
def tiny_layer(seed, E=8, d=128, f=64, bits=4):
    shape = synth.PoolShape(d, f, E, bits)
    q, sb = synth.expert_pool(seed, 0, shape)
    mats = [synth.expert_matrices(q[e], sb[e], shape) for e in range(E + 1)]
    R = synth.router(seed, 0, E, d)
    R = (R.float() * 16).to(torch.bfloat16)  # spread the logits of a tiny layer
    G = synth.shared_gate(seed, 0, d)
    return shape, mats, R, G


def test_expert_permutation_invariance():
    shape, mats, R, G = tiny_layer(31)
    E = shape.E
    perm = np.random.default_rng(0).permutation(E)
    Rn = R.view(torch.int16).numpy()
    Rp = Rn[perm]  # new expert j is old expert perm[j]
    for t in range(6):
        x = O.bf16_to_f64(synth.activations(31, t, 1, shape.d).view(torch.int16).numpy()[0])
        out, idx, w, g = O.moe_layer(Rn, G, lambda e: mats[e], mats[E], 4, x, 2)
        outp, idxp, wp, gp = O.moe_layer(Rp, G, lambda e: mats[perm[e]], mats[E], 4, x, 2)
        assert perm[idxp].tolist() == idx.tolist()
        assert np.allclose(out, outp, rtol=1e-12, atol=1e-12)
        assert np.allclose(w, wp, rtol=1e-12)


def test_layer_combine_definition():
    """out = sum_k w_k * expert_k(x) + gamma * shared(x), with expert() the SwiGLU definition."""
    shape, mats, R, G = tiny_layer(32)
    x = O.bf16_to_f64(synth.activations(32, 0, 1, shape.d).view(torch.int16).numpy()[0])
    out, idx, w, gamma = O.moe_layer(R, G, lambda e: mats[e], mats[shape.E], 4, x, 2)

    def dense(m):
        return torch.from_numpy(O.dequant(m[0].numpy(), m[1], 4))

    xt = torch.from_numpy(x)
    ref = torch.zeros(shape.d, dtype=torch.float64)
    for k, e in enumerate(idx.tolist() + [shape.E]):
        g, u, dn = (dense(m) for m in mats[e])
        y = dn @ (torch.nn.functional.silu(g @ xt) * (u @ xt))
        ref += (w[k] if k < 2 else gamma) * y
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_stack_with_zero_experts():
    """All expert weights zero: every layer adds 0, so x1 = bf16(rmsnorm(x0))."""
    shape, mats, R, G = tiny_layer(33)
    zero = [(m[0] * 0, m[1] * 0) for m in mats[0]]
    layers = [dict(router=R, shared_gate=G, rho=synth.rho(33, l, shape.d),
                   get_expert=lambda e: zero, shared=zero) for l in range(3)]
    x0 = synth.activations(33, 0, 1, shape.d)[0].view(torch.int16).numpy()
    x1, h, idx = O.stack_token(layers, x0, 4, 2)
    x0d = O.bf16_to_f64(x0)
    assert np.array_equal(h, x0d)
    assert np.array_equal(x1, O.f64_to_bf16_bits(x0d / np.sqrt(np.mean(x0d ** 2) + 1e-6)))


# ------------------------------------- the stack's layer input, non-zero experts
def torch_dense_layer(R, G, mats_of, shared, x, K, force=None):
    """One layer from torch float64 library routines on the dequantised weights:
    softmax, a stable descending sort for the top-K, SiLU, dense matmuls."""
    xt = torch.as_tensor(x, dtype=torch.float64)
    Rt = torch.from_numpy(O.bf16_to_f64(np.asarray(R.view(torch.int16) if torch.is_tensor(R) else R)))
    logits = Rt @ xt
    p = torch.softmax(logits, dim=0)
    idx = torch.sort(logits, descending=True, stable=True).indices[:K] if force is None else \
        torch.as_tensor(force, dtype=torch.int64)
    w = p[idx] / p[idx].sum()
    Gt = torch.from_numpy(O.bf16_to_f64(np.asarray(G.view(torch.int16) if torch.is_tensor(G) else G)))
    gamma = torch.sigmoid(Gt @ xt)

    def expert(m):
        g, u, dn = (torch.from_numpy(O.dequant(mm[0], mm[1], 4)) for mm in m)
        return dn @ (torch.nn.functional.silu(g @ xt) * (u @ xt))

    out = torch.zeros(Rt.shape[1], dtype=torch.float64)
    for k in range(K):
        out += w[k] * expert(mats_of(int(idx[k])))
    out += gamma * expert(shared)
    return out, idx.numpy(), w.numpy()


def torch_stack_token(layers, x0_bits, K, eps=1e-6):
    """The decode step from torch routines: a = bf16(rms_norm(h) * rho) before
    each layer, h += layer(a), next input bf16(rms_norm(h))."""
    h = torch.from_numpy(O.bf16_to_f64(x0_bits))
    idxs = []
    for L in layers:
        rho = torch.from_numpy(O.bf16_to_f64(L["rho"]))
        a = torch.nn.functional.rms_norm(h, (h.shape[0],), weight=rho, eps=eps)
        a = a.to(torch.bfloat16).to(torch.float64)
        out, idx, _ = torch_dense_layer(L["router"], L["shared_gate"], L["get_expert"], L["shared"], a, K)
        h = h + out
        idxs.append(idx)
    xn = torch.nn.functional.rms_norm(h, (h.shape[0],), eps=eps).to(torch.bfloat16)
    return xn.view(torch.int16).numpy().astype(np.uint16), h.numpy(), idxs


def nonzero_stack(seed, n_layers=3):
    shape, mats, R, G = tiny_layer(seed)
    layers = []
    for l in range(n_layers):
        Rl = synth.router(seed, l, shape.E, shape.d)
        Rl = (Rl.float() * 16).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
        Gl = synth.shared_gate(seed, l, shape.d).view(torch.int16).numpy().astype(np.uint16)
        q, sb = synth.expert_pool(seed, l, shape)
        ml = [[(m[0].numpy(), m[1].view(torch.int16).numpy().astype(np.uint16))
               for m in synth.expert_matrices(q[e], sb[e], shape)] for e in range(shape.E + 1)]
        layers.append(dict(router=Rl, shared_gate=Gl,
                           rho=synth.rho(seed, l, shape.d).view(torch.int16).numpy().astype(np.uint16),
                           get_expert=(lambda ml: (lambda e: ml[e]))(ml), shared=ml[shape.E]))
    x0 = synth.activations(seed, 0, 1, shape.d)[0].view(torch.int16).numpy().astype(np.uint16)
    return layers, x0


def check_stack_token_input(seed=34):
    layers, x0 = nonzero_stack(seed)
    xo, ho, io = O.stack_token(layers, x0, 4, 2)
    xt, ht, it = torch_stack_token(layers, x0, 2)
    assert np.abs(ho).max() > 0.1 and not np.array_equal(ho, O.bf16_to_f64(x0))  # the layers add something
    assert [list(a) for a in io] == [list(b) for b in it]
    assert np.allclose(ho, ht, rtol=1e-12, atol=1e-12)
    assert np.array_equal(xo, xt)


def test_stack_token_layer_input():
    """The stack feeds each layer bf16(rmsnorm(h) * rho), adds the layer's
    unrounded output to h, and emits bf16(rmsnorm(h)): checked against torch's
    rms_norm, bf16 cast, softmax, stable sort and SiLU on a 3-layer stack whose
    experts are not zero (so every layer's input shows in its output)."""
    check_stack_token_input()


def test_planted_layer_fed_residual_is_caught(monkeypatch):
    good = O.rmsnorm
    monkeypatch.setattr(O, "rmsnorm", lambda h, rho, eps=1e-6: np.asarray(h, float) if rho is not None
                        else good(h, rho, eps))
    _raises(check_stack_token_input)


def test_planted_dropped_rho_is_caught(monkeypatch):
    good = O.rmsnorm
    monkeypatch.setattr(O, "rmsnorm", lambda h, rho, eps=1e-6: good(h, None, eps))
    _raises(check_stack_token_input)


def test_planted_unrounded_layer_input_is_caught(monkeypatch):
    monkeypatch.setattr(O, "round_bf16", lambda v: np.asarray(v, dtype=np.float64))
    _raises(check_stack_token_input)


# ------------------------------------------------ the layer on a forced expert set
def check_forced_set(seed=35):
    shape, mats, R, G = tiny_layer(seed)
    x = O.bf16_to_f64(synth.activations(seed, 1, 1, shape.d).view(torch.int16).numpy()[0])
    Rn = R.view(torch.int16).numpy().astype(np.uint16)
    Gn = G.view(torch.int16).numpy().astype(np.uint16)
    natural = O.route(Rn, x, 2, Gn)[2]
    for force in ([int(natural[1]), int(natural[0])],                    # the same set, other order
                  [int(O.topk_stable(O.route(Rn, x, 2, Gn)[0], 4)[2]), int(natural[0])],  # 3rd-ranked in
                  [7, 5]):                                               # any set
        out, idx, w, gamma = O.moe_layer(Rn, Gn, lambda e: mats[e], mats[shape.E], 4, x, 2, force_idx=force)
        ref, ridx, rw = torch_dense_layer(Rn, Gn, lambda e: mats[e], mats[shape.E], x, 2, force=force)
        assert list(idx) == list(force) == list(ridx)
        assert np.allclose(w, rw, rtol=1e-12) and abs(w.sum() - 1) < 1e-12
        assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layer_on_a_forced_expert_set():
    """moe_layer(force_idx=S) weights expert S_k by softmax(l)[S_k] renormalised
    over S alone (torch softmax over all logits, then divided by the sum over S),
    in the order S gives, plus the gated shared expert."""
    check_forced_set()


def test_planted_forced_set_renormalised_over_natural_top_k_is_caught(monkeypatch):
    good = O.route

    def route(R, x, K, G=None):
        logits, p, idx, w, gamma = good(R, x, K, G)
        return logits, np.where(np.isin(np.arange(len(p)), idx), p, 0.0), idx, w, gamma

    monkeypatch.setattr(O, "route", route)  # probabilities outside the natural top-K lost
    _raises(check_forced_set)


# ------------------------------------------------------- G. size figures
def test_expert_size_matches_page():
    """[Flash-MoE page, "架构设计"]: each expert is about 6.75 MB at 4-bit.

    gate+up+down of 1024x4096 at 4 bits plus one bf16 (scale, bias) pair per
    64 weights is exactly 6.75 MiB, which pins group 64 with 32 bits of
    scale/bias per group for this shape. [Flash-MoE page, "2-bit vs 4-bit"]:
    the model shrinks to about 120 GB at 2 bits; 60 layers x 512 experts x
    the 2-bit expert size is 120.8 GB.
    """
    s4 = synth.PoolShape(4096, 1024, 512, 4)
    assert s4.expert_bytes == 7_077_888 == int(6.75 * 2 ** 20)
    s2 = synth.PoolShape(4096, 1024, 512, 2)
    assert s2.expert_bytes == 3_932_160
    total2 = 60 * 512 * s2.expert_bytes
    assert abs(total2 / 1e9 - 120) / 120 < 0.01
    total4 = 60 * 512 * s4.expert_bytes
    assert abs(total4 / 1e9 - 209) / 209 < 0.05  # within 5% of the page's 209 GB


# ------------------------------------------- planted mistakes are caught
def _raises(fn):
    with pytest.raises(AssertionError):
        fn()


def test_planted_msb_first_unpack_is_caught(monkeypatch):
    good = O.unpack_codes

    def msb_first(qw, bits):
        q = good(qw, bits)
        per = 32 // bits
        return q.reshape(q.shape[0], -1, per)[:, :, ::-1].reshape(q.shape)

    monkeypatch.setattr(O, "unpack_codes", msb_first)
    _raises(lambda: check_column_extraction(4))
    _raises(check_hand_cases)


def test_planted_msb_first_byte_order_is_caught(monkeypatch):
    good = O.unpack_codes

    def msb_first(qw, bits):
        q = good(qw, bits)
        per = 32 // bits
        return q.reshape(q.shape[0], -1, per)[:, :, ::-1].reshape(q.shape)

    monkeypatch.setattr(O, "unpack_codes", msb_first)
    _raises(check_hand_cases8)


def test_planted_per_row_as_first_group_is_caught(monkeypatch):
    good = O.dequant

    def dequant_group64(qw, sb, bits, group=64):
        # a plausible slip: the per-row pair applied only to the first 64 columns
        w = good(qw, sb, bits, group)
        if group != 64:
            q = O.unpack_codes(qw, bits).astype(np.float64)
            w[:, 64:] = q[:, 64:]
        return w

    monkeypatch.setattr(O, "dequant", dequant_group64)
    _raises(check_hand_cases8)


def test_planted_swapped_scale_bias_is_caught(monkeypatch):
    good = O.bf16_to_f64

    def dequant_swapped(qw, sb, bits, group=64):
        q = O.unpack_codes(qw, bits).astype(np.float64)
        sbv = good(sb).reshape(q.shape[0], q.shape[1] // 64, 2)
        s = np.repeat(sbv[:, :, 1], 64, axis=1)
        b = np.repeat(sbv[:, :, 0], 64, axis=1)
        return q * s + b

    monkeypatch.setattr(O, "dequant", dequant_swapped)
    _raises(check_hand_cases)


def test_planted_dropped_bias_is_caught(monkeypatch):
    def dequant_nobias(qw, sb, bits, group=64):
        q = O.unpack_codes(qw, bits).astype(np.float64)
        sbv = O.bf16_to_f64(sb).reshape(q.shape[0], q.shape[1] // 64, 2)
        return q * np.repeat(sbv[:, :, 0], 64, axis=1)

    monkeypatch.setattr(O, "dequant", dequant_nobias)
    _raises(check_hand_cases)
    _raises(check_zero_codes_and_zero_scale)


def test_planted_wrong_group_index_is_caught(monkeypatch):
    def dequant_modgroup(qw, sb, bits, group=64):
        q = O.unpack_codes(qw, bits).astype(np.float64)
        sbv = O.bf16_to_f64(sb).reshape(q.shape[0], q.shape[1] // 64, 2)
        g = np.arange(q.shape[1]) % sbv.shape[1]
        return q * sbv[:, g, 0] + sbv[:, g, 1]

    monkeypatch.setattr(O, "dequant", dequant_modgroup)
    _raises(check_hand_cases)


def test_planted_tie_to_highest_index_is_caught(monkeypatch):
    monkeypatch.setattr(O, "topk_stable",
                        lambda v, k: (len(v) - 1 - np.argsort(-np.asarray(v)[::-1], kind="stable"))[:k])
    _raises(check_route_invariants)


def test_planted_missing_renormalisation_is_caught(monkeypatch):
    good = O.route

    def route_no_renorm(R, x, k, G=None):
        logits, p, idx, w, gamma = good(R, x, k, G)
        return logits, p, idx, p[idx], gamma

    monkeypatch.setattr(O, "route", route_no_renorm)
    _raises(check_route_invariants)


def test_planted_silu_as_sigmoid_is_caught(monkeypatch):
    monkeypatch.setattr(O, "silu", lambda z: 1 / (1 + np.exp(-np.asarray(z, dtype=np.float64))))
    _raises(check_silu)


def test_planted_bf16_truncation_is_caught(monkeypatch):
    def trunc(v):
        f = np.asarray(v, dtype=np.float64).astype(np.float32)
        return (f.view(np.uint32) >> 16).astype(np.uint16)

    monkeypatch.setattr(O, "f64_to_bf16_bits", trunc)
    _raises(check_bf16_rounding)


# ------------------------------------------------ the projection chain
def uniform_matrix(rows, cols, code, scale, bias, bits=4):
    """Every code `code`; group g's (scale, bias) = (scale[g], bias[g]) (scalars broadcast)."""
    q = pack_rows([[code] * cols for _ in range(rows)], bits)
    ng = cols // 64
    s = np.broadcast_to(np.asarray(scale, dtype=np.float64), (ng,))
    b = np.broadcast_to(np.asarray(bias, dtype=np.float64), (ng,))
    sb = np.stack([bf16_bits(s), bf16_bits(b)], axis=-1)  # [ng][2]
    return q, np.broadcast_to(sb, (rows, ng, 2)).copy()


def check_chain_closed_forms():
    rng = np.random.default_rng(5)
    # one step, no norm, no residual: the GEMV itself
    q = pack_rows(rng.integers(0, 16, size=(24, 128)), 4)
    sb = bf16_bits(rng.normal(0, 0.05, size=(24, 2, 2)))
    xb = bf16_bits(rng.normal(0, 1, size=(3, 128)))
    assert np.array_equal(O.gemv_chain([(q, sb)], 4, xb), O.gemv(q, sb, 4, O.bf16_to_f64(xb)))
    # the inner vector is rounded to bf16: step 1 gives 64/64 + 64 * 2^-16 = 1 + 2^-10 per row,
    # whose bf16 is 1, so the all-ones step 2 sums 64 ones (64.0625 unrounded)
    W1 = uniform_matrix(64, 128, 0, 0.0, [1.0 / 64, 2.0 ** -16])
    W2 = uniform_matrix(8, 64, 1, 1.0, 0.0)
    ones = bf16_bits(np.ones(128))
    assert np.array_equal(O.gemv_chain([W1], 4, ones), np.full(64, 1 + 2.0 ** -10))
    assert np.array_equal(O.gemv_chain([W1, W2], 4, ones), np.full(8, 64.0))
    # the norm: a constant 3 normalises to bf16(3 / sqrt(9 + eps)) = 1 (0.5 with rho = 0.5)
    threes = bf16_bits(np.full((2, 64), 3.0))
    Wsum = uniform_matrix(64, 64, 1, 1.0, 0.0)
    assert np.array_equal(O.gemv_chain([Wsum], 4, threes, norm=True), np.full((2, 64), 64.0))
    half = bf16_bits(np.full(64, 0.5))
    assert np.array_equal(O.gemv_chain([Wsum], 4, threes, norm=True, rho_bits=half), np.full((2, 64), 32.0))
    # the residual adds x itself (not the normalised input)
    assert np.array_equal(O.gemv_chain([Wsum], 4, threes, norm=True, residual=True), np.full((2, 64), 67.0))
    # zero weights: the residual chain returns x
    Wz = uniform_matrix(64, 64, 5, 0.0, 0.0)
    xr = bf16_bits(rng.normal(0, 1, size=(2, 64)))
    assert np.array_equal(O.gemv_chain([Wz, Wz], 4, xr, residual=True), O.bf16_to_f64(xr))
    # 2-bit codes: all code 3 with scale 1 over 128 ones sums to 384
    W2b = uniform_matrix(4, 128, 3, 1.0, 0.0, bits=2)
    assert np.array_equal(O.gemv_chain([W2b], 2, ones), np.full(4, 384.0))


def test_chain_closed_forms():
    check_chain_closed_forms()


def test_planted_unrounded_chain_vector_is_caught(monkeypatch):
    monkeypatch.setattr(O, "round_bf16", lambda v: np.asarray(v, dtype=np.float64))
    _raises(check_chain_closed_forms)


def test_planted_chain_norm_without_rho_is_caught(monkeypatch):
    good = O.rmsnorm
    monkeypatch.setattr(O, "rmsnorm", lambda h, rho, eps=1e-6: good(h, None, eps))
    _raises(check_chain_closed_forms)
