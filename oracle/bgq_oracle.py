"""fp64 CPU oracle for the group-quantized MoE decode path.

TEST INFRASTRUCTURE ONLY. This module is the correctness reference that the
CUDA library is compared against. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the library and its
Python binding never do, and nothing here is shared with them (the only
common code is the seeded input generator, which holds none of this
arithmetic).

Every function is the plain definition of one step, written with numpy in
float64, with no blocking, fusion or reordering beyond what the definition
states. Matrix-vector products use ``numpy.matmul`` (a library primitive).
Inputs are the packed words and bf16 bit patterns exactly as stored; bf16
values are widened to float64 exactly.

Sources (web pages; the method is described on the first):
  [FM]   "397B参数的模型跑在48GB笔记本上：Flash-MoE用纯C打爆Python推理框架"
         (blog.js-css.com/topics/2026/03/23/519). Sections cited by heading:
         "先搞清楚为什么这件事很难" (layer shape: 512 experts, top-4 + 1 shared),
         "架构设计：SSD当显存用" (per-token pipeline: routing, softmax + topK,
         expert forward + combine + norm), "FMA Dequant：一条指令省12%"
         (w = nibble*scale + bias and its fma reordering), "2-bit vs 4-bit".
  [H3]   "Redis 之父下场手写推理引擎：antirez 用约 24000 行原生代码驯服视频生成模型"
         (text-matrix.pages.dev/posts/tech/antirez-h3-metal/): the paragraph
         on --use-int8-row-fc2 (int8 MLP weights with a scale per group; FC2
         with one scale per row).
Where the page is silent the workload definition fixes the value (group 64,
bf16 scale and bias, LSB-first packing, renormalised top-K weights, lowest
index wins ties, a sigmoid-gated shared expert, RMSNorm before each layer).
Readings of silent points are marked READING.

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
(hand-computed cases, closed forms, library special cases, invariants);
``gemv_chain`` composes pinned steps and is pinned on its own there too.
"""

from __future__ import annotations

import numpy as np

GROUP = 64


# ------------------------------------------------------------------ bf16 bits
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16 / int16 arrays or torch tensors)."""
    a = np.asarray(_np(bits)).astype(np.uint16).astype(np.uint32) << 16
    return a.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v) -> np.ndarray:
    """Round float64 values to bf16, round-to-nearest-even, in one step.

    bf16 keeps 8 significant bits; the rounding is done on the float64 bit
    pattern (45 dropped mantissa bits), so there is no double rounding
    through float32. Finite values in the normal bf16 range only.
    """
    v = np.asarray(v, dtype=np.float64)
    u = v.view(np.uint64)
    drop = np.uint64(45)
    half = np.uint64(1) << np.uint64(44)
    lsb = (u >> drop) & np.uint64(1)
    r = (u + half - np.uint64(1) + lsb) & ~((np.uint64(1) << drop) - np.uint64(1))
    f32 = r.view(np.float64).astype(np.float32)  # exact: 8 significant bits
    return (f32.view(np.uint32) >> 16).astype(np.uint16)


def round_bf16(v) -> np.ndarray:
    return bf16_to_f64(f64_to_bf16_bits(v))


def _np(t):
    if hasattr(t, "detach"):  # torch tensor
        t = t.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            import torch

            t = t.view(torch.int16)
        return t.numpy()
    return np.asarray(t)


# ------------------------------------------------------------- packed format
def unpack_codes(q_words, bits: int) -> np.ndarray:
    """Codes q[n, k] from packed words [n][cols*bits/32].

    READING (the page says only that weights are 4-bit nibbles): the codes
    are stored least-significant-first, element k of a row in word
    k // (32/bits) at bit offset bits * (k % (32/bits)). bits is 2, 4 or 8
    (8: four bytes per word, byte 0 first).
    """
    w = np.asarray(_np(q_words)).astype(np.int64) & 0xFFFFFFFF
    per = 32 // bits
    mask = (1 << bits) - 1
    fields = [(w >> (bits * j)) & mask for j in range(per)]
    q = np.stack(fields, axis=-1)  # [n, words, per]
    return q.reshape(w.shape[0], w.shape[1] * per)


def dequant(q_words, sb, bits: int, group: int = GROUP) -> np.ndarray:
    """w[n, k] = q[n, k] * s[n, g] + b[n, g], g = k // group.

    [FM] "FMA Dequant": each weight is ``nibble * scale + bias``. scale and
    bias are bf16, one pair per group of 64 consecutive columns of a row.
    [H3] (the --use-int8-row-fc2 paragraph): int8 weights with one scale per
    group, or, for FC2, a single scale per row. READING: the same affine form
    at 8 bits (codes 0..255); the per-row format is ``group`` = row length.
    """
    q = unpack_codes(q_words, bits).astype(np.float64)
    sbv = bf16_to_f64(sb).reshape(q.shape[0], q.shape[1] // group, 2)
    s = np.repeat(sbv[:, :, 0], group, axis=1)
    b = np.repeat(sbv[:, :, 1], group, axis=1)
    return q * s + b


def gemv(q_words, sb, bits: int, x, group: int = GROUP) -> np.ndarray:
    """y = W x with W dequantised in float64 (x: [cols] or [batch][cols])."""
    W = dequant(q_words, sb, bits, group)
    x = np.asarray(x, dtype=np.float64)
    return x @ W.T if x.ndim == 2 else W @ x


def dot_terms_standard(q, s, b, x):
    """The per-weight product as first written on [FM] "FMA Dequant": (q*s + b) * x."""
    return (q * s + b) * x


def dot_terms_reordered(q, s, b, x):
    """The page's reordering of the same product: fma(q, s*x, b*x).

    numpy has no fused multiply-add; in float64 every partial result here is
    exact for bf16 s, b, x and integer q <= 15 (at most 8+8+4 significant
    bits per product), so the unfused expression equals the fused one.
    """
    return q * (s * x) + (b * x)


# ------------------------------------------------------------------- routing
def softmax(logits) -> np.ndarray:
    """softmax over the last axis, exp(l - max) / sum."""
    l = np.asarray(logits, dtype=np.float64)
    e = np.exp(l - l.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def topk_stable(values, k: int) -> np.ndarray:
    """Indices of the k largest values, largest first; equal values keep index order."""
    v = np.asarray(values, dtype=np.float64)
    return np.argsort(-v, kind="stable")[:k]


def route(router_bits, x, top_k: int, shared_gate_bits=None):
    """Router of one token.

    [FM] "架构设计": routing logits are computed on the GPU, then softmax and
    top-K are taken (K = 4 of 512 per "先搞清楚为什么这件事很难").
    l = R x; p = softmax(l); the K experts with the largest p are selected
    (selection is done on l, which orders them identically and cannot
    create ties that p's rounding might; equal logits -> lower index first);
    w_k = p_k / sum_{j in top-K} p_j (renormalised);
    gamma = sigmoid(G . x) for the shared expert (1 if there is no gate).
    Returns (logits, probs, idx, w, gamma).
    """
    R = bf16_to_f64(router_bits)
    x = np.asarray(x, dtype=np.float64)
    logits = R @ x
    p = softmax(logits)
    idx = topk_stable(logits, top_k)
    w = p[idx] / p[idx].sum()
    if shared_gate_bits is None:
        gamma = 1.0
    else:
        z = float(bf16_to_f64(shared_gate_bits) @ x)
        gamma = 1.0 / (1.0 + np.exp(-z))
    return logits, p, idx, w, gamma


# ------------------------------------------------------------------- experts
def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def expert_swiglu(gate, up, down, bits: int, x) -> np.ndarray:
    """SwiGLU expert: down( silu(gate x) * (up x) ), each matrix group-quantized.

    gate, up, down are (q_words, sb) pairs. [FM] "架构设计": CMD3 runs the
    selected experts' forward pass on packed weights.
    """
    g = gemv(*gate, bits, x)
    u = gemv(*up, bits, x)
    h = silu(g) * u
    return gemv(*down, bits, h)


def moe_layer(router_bits, shared_gate_bits, get_expert, shared_expert, bits: int, x,
              top_k: int, force_idx=None):
    """One MoE layer for one token.

    out = sum_k w_k * expert_{idx_k}(x) + gamma * shared(x), in float64, summed
    in the order k = 0..K-1 then the shared expert ([FM] "架构设计": expert
    forward + combine; each token uses 4 routed experts plus 1 shared expert).
    ``get_expert(e)`` returns (gate, up, down) of routed expert e.
    ``force_idx`` evaluates the layer with a given expert set (used where the
    top-K is a near tie and another valid set was chosen); the weights are
    then the renormalised softmax of those experts.
    Returns (out, idx, w, gamma).
    """
    logits, p, idx, w, gamma = route(router_bits, x, top_k, shared_gate_bits)
    if force_idx is not None:
        idx = np.asarray(force_idx, dtype=np.int64)
        w = p[idx] / p[idx].sum()
    out = np.zeros(_expert_out_dim(shared_expert), dtype=np.float64)
    for k in range(top_k):
        out = out + w[k] * expert_swiglu(*get_expert(int(idx[k])), bits, x)
    out = out + gamma * expert_swiglu(*shared_expert, bits, x)
    return out, idx, w, gamma


def _expert_out_dim(expert) -> int:
    down_q = np.asarray(_np(expert[2][0]))
    return down_q.shape[0]


# --------------------------------------------------------------------- stack
def rmsnorm(h, rho_bits, eps: float = 1e-6) -> np.ndarray:
    """h / sqrt(mean(h^2) + eps) * rho.

    [FM] "架构设计" lists a norm before routing and after the combine; the
    workload fixes RMSNorm with a bf16 weight before each layer.
    READING: eps = 1e-6.
    """
    h = np.asarray(h, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(h * h) + eps)
    rho = 1.0 if rho_bits is None else bf16_to_f64(rho_bits)
    return h * r * rho


def stack_token(layers, x0_bits, bits: int, top_k: int, eps: float = 1e-6, force_idx=None):
    """One decode token through a stack of layers.

    h = x0; per layer l: a = bf16(rmsnorm(h, rho_l)); h = h + layer_l(a).
    The token's output (the next token's input) is bf16(rmsnorm(h, none)).
    READING: the workload says only that tokens run sequentially from a
    seeded start vector; the normalised final residual, rounded to bf16, is
    fed back so that every token's input has unit RMS like x ~ N(0, 1).
    ``layers[l]`` is a dict with router, shared_gate, rho, get_expert, shared.
    Returns (x_next_bits, h_final, per-layer idx).
    """
    h = bf16_to_f64(x0_bits)
    all_idx = []
    for l, L in enumerate(layers):
        a = round_bf16(rmsnorm(h, L["rho"], eps))
        fi = None if force_idx is None else force_idx[l]
        out, idx, _, _ = moe_layer(L["router"], L["shared_gate"], L["get_expert"], L["shared"],
                                   bits, a, top_k, force_idx=fi)
        h = h + out
        all_idx.append(idx)
    x_next = f64_to_bf16_bits(rmsnorm(h, None, eps))
    return x_next, h, all_idx


# --------------------------------------------------------- projection chain
def gemv_chain(mats, bits: int, x_bits, norm: bool = False, rho_bits=None, eps: float = 1e-6,
               residual: bool = False) -> np.ndarray:
    """The decoder's projections around the MoE block as a chain of GEMVs.

    [FM] "架构设计：SSD当显存用": each layer runs the attention input
    projections (CMD1) and o_proj + norm (CMD2) on the GPU. READING: the
    attention mixing between them is not part of this workload, so the chain
    feeds each projection's output to the next one:
        v_0 = bf16(rmsnorm(x) * rho) if norm else x
        v_i = bf16(W_i v_{i-1}),  i = 1..n-1
        out = W_n v_{n-1} (+ x if residual)      (float64, before rounding)
    The bf16 roundings of the inner vectors follow the standalone GEMV, whose
    output is bf16. mats: [(q_words, sb)], x_bits: bf16 [cols] or [batch][cols].
    """
    x = bf16_to_f64(np.asarray(_np(x_bits)))
    v = x
    if norm:
        v = np.stack([round_bf16(rmsnorm(row, rho_bits, eps)) for row in np.atleast_2d(x)])
        v = v.reshape(x.shape)
    n = len(mats)
    for i, (q, sb) in enumerate(mats):
        y = gemv(np.asarray(_np(q)), np.asarray(_np(sb)), bits, v)
        v = y if i == n - 1 else round_bf16(y)
    return x + v if residual else v
