"""Seeded synthetic inputs for the group-quantized MoE decode path.

This module draws random numbers and shapes them into the workload's value
distributions. It holds none of the method's arithmetic: no unpacking,
dequantisation, dot products, softmax, top-K, SwiGLU or normalisation. Both
sides of every parity check (the CUDA library and the fp64 oracle) take their
inputs from here, and nothing else is shared between them.

Generator
---------
A counter-based stream. The i-th 32-bit draw of a stream with keys (k1, k2) is

    v(i) = H(H(i XOR k1) XOR k2)

where H is the ``lowbias32`` integer hash published by C. Wellons
(hash-prospector, 2018)::

    x ^= x >> 16; x *= 0x7feb352d; x ^= x >> 15; x *= 0x846ca68b; x ^= x >> 16

(multiplications modulo 2**32). Every operation runs on int64 torch tensors
with explicit masking, so the same counters give bit-identical words on the
CPU and on a GPU; this is what lets a test regenerate, on the host, exactly
the expert that a GPU run selected.

Derived values (each step is a single correctly-rounded fp32 operation, so
CPU and GPU agree bit for bit):

* uniform u in [0, 1):  (v >> 8) * 2**-24
* approximately normal n:  Irwin-Hall sum of twelve 16-bit uniforms minus 6
  (twelve halves of six draws), range [-6, 6], unit variance.
* packed code words: the raw 32-bit draw. Every 8-, 4- or 2-bit field of a
  uniform 32-bit word is itself uniform on 0..255 (0..15, 0..3).

Value distributions (the workload's recipe; the second parameter of N(.,.)
is read as a standard deviation, the usual convention for weight inits):

* scale  s = bf16(0.002 + 0.018 u)                    (U[0.002, 0.02])
* bias   b = bf16(-m * s + 1e-4 n),  m = 2**(bits-1)   (m = 8 at 4-bit)
* x      = bf16(n)                                     (N(0, 1))
* router = bf16(0.02 n)                                (N(0, 0.02))
* shared-expert gate vector = bf16(0.02 n)
* RMSNorm weight rho = bf16(1 + 0.01 n)

Packed layout produced here (the library's documented storage format): a
matrix of ``rows x cols`` codes is ``q`` uint32 ``[rows][cols*bits/32]``
(stored as int32 bit patterns) and ``sb`` bf16 ``[rows][cols/64][2]`` holding
(scale, bias) per group of 64 consecutive columns. An expert is gate
``[f][d]``, up ``[f][d]``, down ``[d][f]`` concatenated in that order, in a
``q`` pool row and an ``sb`` pool row.
"""

from __future__ import annotations

import torch

MASK32 = 0xFFFFFFFF
GROUP = 64

# Stream tags: one independent stream per kind of tensor.
TAG_EXPERT_Q = 1
TAG_EXPERT_SCALE = 2
TAG_EXPERT_BIASNOISE = 3
TAG_ROUTER = 4
TAG_SHARED_GATE = 5
TAG_RHO = 6
TAG_X = 7
TAG_MATRIX_Q = 8
TAG_MATRIX_SCALE = 9
TAG_MATRIX_BIASNOISE = 10


# ---------------------------------------------------------------- scalar hash
def _h32(x: int) -> int:
    x &= MASK32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & MASK32
    x ^= x >> 15
    x = (x * 0x846CA68B) & MASK32
    x ^= x >> 16
    return x


def stream_keys(seed: int, *tags: int) -> tuple[int, int]:
    """Two 32-bit keys for the stream named by (seed, tags...)."""
    k = _h32(seed ^ 0x2545F491)
    for t in tags:
        k = _h32((k + (t & MASK32) + 0x9E3779B9) & MASK32)
    return k, _h32(k ^ 0x5BD1E995)


# ---------------------------------------------------------------- tensor hash
def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    # (x * c) mod 2**32 for x in [0, 2**32) without int64 overflow.
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + ((x * hi) & 0xFFFF) * 65536) & MASK32


def _h32_t(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def draws_at(keys: tuple[int, int], counters: torch.Tensor) -> torch.Tensor:
    """32-bit draws (int64 in [0, 2**32)) at the given int64 counters."""
    k1, k2 = keys
    return _h32_t(_h32_t(counters ^ k1) ^ k2)


def draws(keys, start: int, count: int, device) -> torch.Tensor:
    c = torch.arange(start, start + count, dtype=torch.int64, device=device)
    return draws_at(keys, c)


def _as_int32_bits(v: torch.Tensor) -> torch.Tensor:
    # Reinterpret [0, 2**32) as a two's-complement int32 bit pattern.
    return (v - ((v >> 31) << 32)).to(torch.int32)


def uniform_at(keys, counters: torch.Tensor) -> torch.Tensor:
    v = draws_at(keys, counters)
    return (v >> 8).to(torch.float32) * (2.0 ** -24)


def normal_at(keys, index: torch.Tensor) -> torch.Tensor:
    """Approximate N(0,1) draw number ``index`` (uses counters 6i..6i+5)."""
    base = index * 6
    total = torch.zeros_like(index)
    for j in range(6):
        v = draws_at(keys, base + j)
        total = total + (v & 0xFFFF) + (v >> 16)
    # sum of twelve (u16 + 0.5)/65536 minus 6, as one exact fp32 value
    return (total + 6 - 6 * 65536).to(torch.float32) * (2.0 ** -16)


def _arange(start, count, device):
    return torch.arange(start, start + count, dtype=torch.int64, device=device)


# ---------------------------------------------------------------- packed rows
def _scale_bias(keys_s, keys_n, gstart: int, ngroups: int, bits: int, device):
    """(scale, bias) bf16 pairs for groups [gstart, gstart+ngroups)."""
    g = _arange(gstart, ngroups, device)
    u = uniform_at(keys_s, g)
    s = ((u * 0.018) + 0.002).to(torch.bfloat16)
    n = normal_at(keys_n, g)
    mid = float(1 << (bits - 1))
    b = ((s.to(torch.float32) * (-mid)) + (n * 1e-4)).to(torch.bfloat16)
    return torch.stack([s, b], dim=-1)  # [ngroups, 2]


def words_per_row(cols: int, bits: int) -> int:
    return cols * bits // 32


def qmatrix(seed: int, rows: int, cols: int, bits: int = 4, device="cpu", tag: int = 0, group: int = GROUP):
    """A standalone packed matrix: (q int32 [rows][cols*bits/32], sb bf16 [rows][cols/group][2]).

    bits 2, 4 or 8; group 64, or cols for one (scale, bias) pair per row (the
    per-row 8-bit format). At 8 bits the bias is -128*s + noise, the affine
    form of symmetric signed int8.
    """
    assert cols % GROUP == 0 and bits in (2, 4, 8) and group in (GROUP, cols)
    wpr = words_per_row(cols, bits)
    kq = stream_keys(seed, TAG_MATRIX_Q, tag)
    q = _as_int32_bits(draws(kq, 0, rows * wpr, device)).view(rows, wpr)
    ks = stream_keys(seed, TAG_MATRIX_SCALE, tag)
    kn = stream_keys(seed, TAG_MATRIX_BIASNOISE, tag)
    sb = _scale_bias(ks, kn, 0, rows * (cols // group), bits, device)
    return q, sb.view(rows, cols // group, 2)


# ---------------------------------------------------------------- expert pools
class PoolShape:
    """Sizes of one layer's expert pool (routed experts + 1 shared expert)."""

    def __init__(self, d_model: int, d_ff: int, n_experts: int, bits: int = 4):
        assert d_model % GROUP == 0 and d_ff % GROUP == 0 and bits in (2, 4)
        self.d, self.f, self.E, self.bits = d_model, d_ff, n_experts, bits
        self.n_total = n_experts + 1  # index n_experts is the shared expert
        self.mat_words = d_model * d_ff * bits // 32  # words per matrix
        self.mat_groups = d_model * d_ff // GROUP  # groups per matrix
        self.q_stride = 3 * self.mat_words  # words per expert
        self.sb_stride = 3 * self.mat_groups * 2  # bf16 elements per expert

    @property
    def expert_bytes(self) -> int:
        return self.q_stride * 4 + self.sb_stride * 2


def expert_pool_range(seed: int, layer: int, shape: PoolShape, e0: int, ne: int, device="cpu"):
    """Experts [e0, e0+ne) of a layer's pool as (q int32 [ne][q_stride], sb bf16 [ne][sb_stride])."""
    kq = stream_keys(seed, TAG_EXPERT_Q, layer)
    ks = stream_keys(seed, TAG_EXPERT_SCALE, layer)
    kn = stream_keys(seed, TAG_EXPERT_BIASNOISE, layer)
    q = _as_int32_bits(draws(kq, e0 * shape.q_stride, ne * shape.q_stride, device))
    ng = 3 * shape.mat_groups
    sb = _scale_bias(ks, kn, e0 * ng, ne * ng, shape.bits, device)
    return q.view(ne, shape.q_stride), sb.reshape(ne, shape.sb_stride)


def expert_pool(seed: int, layer: int, shape: PoolShape, device="cpu", chunk_experts: int = 32,
                out_q: torch.Tensor | None = None, out_sb: torch.Tensor | None = None):
    """The whole pool of a layer, generated in chunks (fits large pools on a GPU)."""
    n = shape.n_total
    if out_q is None:
        out_q = torch.empty((n, shape.q_stride), dtype=torch.int32, device=device)
    if out_sb is None:
        out_sb = torch.empty((n, shape.sb_stride), dtype=torch.bfloat16, device=device)
    for e0 in range(0, n, chunk_experts):
        ne = min(chunk_experts, n - e0)
        q, sb = expert_pool_range(seed, layer, shape, e0, ne, device)
        out_q[e0:e0 + ne].copy_(q)
        out_sb[e0:e0 + ne].copy_(sb)
    return out_q, out_sb


def expert_matrices(q_row: torch.Tensor, sb_row: torch.Tensor, shape: PoolShape):
    """Split one expert's pool rows into ((q, sb) gate, up, down) views."""
    d, f, mw, mg = shape.d, shape.f, shape.mat_words, shape.mat_groups
    out = []
    for i, (r, c) in enumerate(((f, d), (f, d), (d, f))):
        q = q_row[i * mw:(i + 1) * mw].view(r, c * shape.bits // 32)
        sb = sb_row[i * mg * 2:(i + 1) * mg * 2].view(r, c // GROUP, 2)
        out.append((q, sb))
    return out


def router(seed: int, layer: int, n_experts: int, d_model: int, device="cpu"):
    k = stream_keys(seed, TAG_ROUTER, layer)
    n = normal_at(k, _arange(0, n_experts * d_model, device))
    return (n * 0.02).to(torch.bfloat16).view(n_experts, d_model)


def shared_gate(seed: int, layer: int, d_model: int, device="cpu"):
    k = stream_keys(seed, TAG_SHARED_GATE, layer)
    return (normal_at(k, _arange(0, d_model, device)) * 0.02).to(torch.bfloat16)


def rho(seed: int, layer: int, d_model: int, device="cpu"):
    k = stream_keys(seed, TAG_RHO, layer)
    return ((normal_at(k, _arange(0, d_model, device)) * 0.01) + 1.0).to(torch.bfloat16)


def activations(seed: int, stream: int, batch: int, d_model: int, device="cpu"):
    k = stream_keys(seed, TAG_X, stream)
    return normal_at(k, _arange(0, batch * d_model, device)).to(torch.bfloat16).view(batch, d_model)


def layer_tensors(seed: int, layer: int, shape: PoolShape, device="cpu", with_gate: bool = True):
    """All tensors of one synthetic MoE layer.

    Returns a dict: router bf16 [E][d], shared_gate bf16 [d] (or None),
    pool_q int32 [E+1][q_stride], pool_sb bf16 [E+1][sb_stride] (routed experts
    0..E-1, the shared expert at index E).
    """
    pool_q, pool_sb = expert_pool(seed, layer, shape, device)
    return dict(router=router(seed, layer, shape.E, shape.d, device),
                shared_gate=shared_gate(seed, layer, shape.d, device) if with_gate else None,
                pool_q=pool_q, pool_sb=pool_sb)
