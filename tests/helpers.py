"""Shared test helpers: oracle input marshalling and error metrics."""

import numpy as np
import torch

from bit_group_quantized_gb300 import synth
from oracle import bgq_oracle as O

REL_L2_TOL = 2e-3  # max relative L2 error of an output vector (bf16 out, fp32 accumulate)
TIE_GAP = 1e-3  # K-th vs (K+1)-th logit gap below which several expert sets are correct
BIG_TOK = 16  # experts with at least this many tokens run on the tensor-core (fp16 operand) path
# The tensor-core path rounds three operands to fp16 (11 significant bits):
# the dequantised weights, the inputs and the SwiGLU outputs. Each adds about
# 2^-11/sqrt(3) ~ 2.8e-4 relative L2, so the kernel's own error (against the
# oracle rounded to bf16, which also counts bf16 rounding flips) is bounded at
# 1.5e-3 there instead of 1e-3; the workload tolerance (2e-3 against the
# unrounded oracle) is the same for every path.
TC_OWN_TOL = 1.5e-3


def own_tol_for(batch: int) -> float:
    """Kernel-own-error bound for a call on `batch` tokens (the shared expert
    takes every token, so batch >= 16 puts it on the tensor-core path)."""
    return TC_OWN_TOL if batch >= BIG_TOK else 1e-3


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return O.bf16_to_f64(bits16(t))
    return t.detach().cpu().double().numpy()


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


class ExpertSource:
    """Regenerates single experts of a synthetic layer on the host, with a cache."""

    def __init__(self, seed, layer, shape: synth.PoolShape):
        self.seed, self.layer, self.shape = seed, layer, shape
        self.cache = {}

    def __call__(self, e: int):
        if e not in self.cache:
            q, sb = synth.expert_pool_range(self.seed, self.layer, self.shape, e, 1, "cpu")
            mats = synth.expert_matrices(q[0], sb[0], self.shape)
            self.cache[e] = [(m[0].numpy(), bits16(m[1])) for m in mats]
        return self.cache[e]


def topk_gap(logits: np.ndarray, k: int) -> float:
    s = np.sort(logits)[::-1]
    return float(s[k - 1] - s[k]) if len(s) > k else np.inf


def check_topk_valid(gpu_idx, oracle_logits, k, gap=TIE_GAP):
    """gpu_idx is a correct top-k within `gap`: every chosen logit >= every
    unchosen logit - gap, all distinct."""
    gi = [int(i) for i in gpu_idx]
    assert len(set(gi)) == k
    chosen = oracle_logits[gi]
    others = np.delete(oracle_logits, gi)
    assert chosen.min() >= others.max() - gap


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def assert_bf16_output(got_bf16, ref_f64, what="", own_tol=1e-3):
    """A bf16 output vector against its float64 oracle value.

    * rel-L2 <= 2e-3 against the unrounded oracle (the workload tolerance),
      asserted for vectors of at least 512 elements: the output rounding
      alone costs about 1.5e-3 on average and varies more on short vectors;
    * rel-L2 <= own_tol (1e-3) against the oracle rounded to bf16 (the
      kernel's own error, beyond the output rounding), for every length;
    * every element within one bf16 spacing of the oracle value (plus 1e-3
      of the vector's largest magnitude for elements near zero).
    """
    got = np.asarray(got_bf16, dtype=np.float64)
    ref = np.asarray(ref_f64, dtype=np.float64)
    if got.size >= 512:
        assert rel_l2(got, ref) <= REL_L2_TOL, (what, rel_l2(got, ref))
    assert rel_l2(got, O.round_bf16(ref)) <= own_tol, (what, rel_l2(got, O.round_bf16(ref)))
    tol = bf16_ulp(ref) + 1e-3 * np.abs(ref).max()
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (what, np.flatnonzero(bad)[:10], got[bad][:5], ref[bad][:5])


def oracle_stack_token(seed, bits, n_layers, x_bits, gpu_idx, d=4096, f=1024, E=512, K=4, eps=1e-6,
                       torch_threads=2):
    """One decode token of the synthetic stack (seed, layers 0..n_layers-1)
    through the fp64 oracle, teacher-forced on the input bits x_bits.

    Regenerates every weight it needs on the host from the seeded generator,
    so it can run in a worker process with no GPU. Where a layer's K-th and
    (K+1)-th oracle logits are within TIE_GAP, the layer is evaluated with the
    GPU's expert set gpu_idx[l] (after checking that set is a valid top-K).
    Returns (x_next bits, h, per-layer oracle top-K, per-layer gap, per-layer
    'forced' flags)."""
    torch.set_num_threads(torch_threads)
    shape = synth.PoolShape(d, f, E, bits)
    layers, gaps, nat, forced = [], [], [], []
    h = O.bf16_to_f64(np.asarray(x_bits, dtype=np.uint16))
    force = []
    for l in range(n_layers):
        R = bits16(synth.router(seed, l, E, d))
        G = bits16(synth.shared_gate(seed, l, d))
        rho = bits16(synth.rho(seed, l, d))
        src = ExpertSource(seed, l, shape)
        L = dict(router=R, shared_gate=G, rho=rho, get_expert=src, shared=src(E))
        a = O.round_bf16(O.rmsnorm(h, rho, eps))
        logits = O.route(R, a, K, G)[0]
        gap = topk_gap(logits, K)
        fi = None
        if gap <= TIE_GAP:
            check_topk_valid(gpu_idx[l], logits, K)
            fi = np.asarray(gpu_idx[l], dtype=np.int64)
        out, idx, _, _ = O.moe_layer(R, G, src, L["shared"], bits, a, K, force_idx=fi)
        h = h + out
        gaps.append(gap)
        nat.append([int(i) for i in O.topk_stable(logits, K)])
        forced.append(fi is not None)
        force.append(fi)
        L["shared"] = None  # keep the worker's memory small: one layer's experts at a time
        src.cache.clear()
    x_next = O.f64_to_bf16_bits(O.rmsnorm(h, None, eps))
    return x_next, h, nat, gaps, forced


# ------------------------------------------------------------------ guard canaries
GUARD_BYTES = 4096  # a multiple of 256: the guarded buffer keeps torch's alignment
GUARD_FILL = 0xA5


class GuardedAllocator:
    """Buffers with guard regions in front of and behind them, filled with a
    known byte, for the outputs and workspaces the binding creates
    (lib.set_allocator) and for the ones tests create with `empty`. check()
    finds any byte of any guard that a kernel overwrote: the bounds check used
    in place of a sanitizer."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype, device, zero=False):
        return self.empty(shape, dtype, device, zero)

    def empty(self, shape, dtype, device, zero=False):
        n = 1
        for s in shape:
            n *= int(s)
        esize = torch.empty((), dtype=dtype).element_size()
        nbytes = max(n * esize, 1)
        body = (nbytes + 255) // 256 * 256
        raw = torch.full((2 * GUARD_BYTES + body,), GUARD_FILL, dtype=torch.uint8, device=device)
        inner = raw[GUARD_BYTES:GUARD_BYTES + n * esize]
        if zero:
            inner.zero_()
        self.bufs.append((raw, GUARD_BYTES + n * esize))
        return inner.view(dtype).view(tuple(int(s) for s in shape))

    def check(self):
        for raw, end in self.bufs:
            front = raw[:GUARD_BYTES]
            back = raw[end:]
            bad_f = int((front != GUARD_FILL).sum())
            bad_b = int((back != GUARD_FILL).sum())
            assert bad_f == 0 and bad_b == 0, f"guard bytes overwritten: {bad_f} in front, {bad_b} behind"
        return len(self.bufs)
