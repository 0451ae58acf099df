"""moe_layer_forward_noalloc: the layer forward for callers that cannot
allocate device memory at call time (it uses the library's fixed 4 MiB scratch
array instead of a workspace). Its results must match moe_layer_forward's on
the same inputs, call after call, since both run the same kernels.

This file is collected last so that a failure here stops a `-x` run only after
every other test has run; it also passes on its own in a fresh process.
"""

import ctypes as C

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from tests.helpers import assert_bf16_output, f64

pytestmark = pytest.mark.gpu


def layer(dev, E, d, f, K, seed):
    shape = synth.PoolShape(d, f, E, 4)
    t = synth.layer_tensors(seed, 0, shape, device=dev)
    return lib.MoELayer(d, f, E, K, 4, t["router"], t["shared_gate"], t["pool_q"][:E], t["pool_sb"][:E],
                        t["pool_q"][E], t["pool_sb"][E])


@pytest.mark.parametrize("E,d,f,B", [(512, 4096, 1024, 1), (512, 4096, 1024, 16), (64, 1024, 512, 7)])
def test_noalloc_matches_workspace_entry_point(cuda_device, E, d, f, B):
    K = 4
    L = layer(cuda_device, E, d, f, K, seed=11)
    for call in range(2):  # two calls in a row share the fixed scratch array
        x = synth.activations(11, 50 + call, B, d, device=cuda_device)
        ref, ref_f32, ref_idx, ref_w, ref_g = lib.moe_layer_forward(L, x, want_f32=True, want_route=True)
        out = lib.alloc((B, d), torch.bfloat16, cuda_device)
        out_f32 = lib.alloc((B, d), torch.float32, cuda_device)
        idx = lib.alloc((B, K), torch.int32, cuda_device)
        w = lib.alloc((B, K), torch.float32, cuda_device)
        g = lib.alloc((B,), torch.float32, cuda_device)
        lib.moe_layer_forward_noalloc(L, x, out=out, out_f32=out_f32, idx=idx, w=w, gamma=g)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        assert torch.allclose(w, ref_w, rtol=1e-6, atol=0) and torch.allclose(g, ref_g, rtol=1e-6, atol=0)
        for t in range(B):
            # within the tests' bf16 output tolerance of the workspace entry point's fp32 result
            assert_bf16_output(f64(out)[t], f64(ref_f32)[t], (call, t))
            assert np.allclose(f64(out_f32)[t], f64(ref_f32)[t], rtol=1e-6, atol=1e-6)


def test_noalloc_rejects_batches_beyond_the_fixed_scratch(cuda_device):
    L = layer(cuda_device, 64, 1024, 512, 4, seed=12)
    s = L.struct()
    too_big = next(b for b in range(1, 257) if lib.load().moe_layer_workspace_bytes(C.byref(s), b) > (4 << 20))
    x = synth.activations(12, 0, too_big, 1024, device=cuda_device)
    out = lib.alloc((too_big, 1024), torch.bfloat16, cuda_device)
    with pytest.raises(lib.BGQError) as ei:
        lib.moe_layer_forward_noalloc(L, x, out=out)
    assert ei.value.status == lib.ERR_WORKSPACE


def test_noalloc_alternating_shapes_reach_the_tensor_core_path(cuda_device):
    """The fixed array is shared by calls of every layer shape. The regions
    that must start at zero (control block, tagged logits) have
    shape-dependent sizes, and every other region sits at a shape-dependent
    place, so one shape's leftovers land in another shape's scratch. Alternate
    shapes, including batch-64 calls whose shared expert runs on the tensor
    cores with split K, and compare every call with moe_layer_forward on a
    fresh zeroed workspace."""
    K = 4
    full = layer(cuda_device, 512, 4096, 1024, K, seed=13)   # 4 MiB-class call, batch 31
    tiny = layer(cuda_device, 8, 256, 128, K, seed=14)       # its logits overlap tc's scratch
    tc = layer(cuda_device, 16, 512, 256, K, seed=15)        # batch 64: the tensor-core path
    seq = [(full, 4096, 31), (tiny, 256, 20), (tc, 512, 64), (tc, 512, 1), (full, 4096, 1), (tc, 512, 64),
           (tiny, 256, 3), (tc, 512, 100)]
    for i, (L, d, B) in enumerate(seq):
        x = synth.activations(13, 200 + i, B, d, device=cuda_device)
        ref = lib.moe_layer_forward(L, x, want_out=False, want_f32=True)[1]
        out_f32 = lib.alloc((B, d), torch.float32, cuda_device)
        lib.moe_layer_forward_noalloc(L, x, out_f32=out_f32)
        torch.cuda.synchronize()
        # same kernels, same inputs: the same bits as a fresh workspace
        assert torch.equal(out_f32, ref), (i, d, B, float((out_f32 - ref).abs().max()))
