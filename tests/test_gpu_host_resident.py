"""Experts kept in pinned host memory (read over the CPU-GPU link by the
grouped kernels) give the same layer outputs as experts in device memory,
and match the fp64 oracle."""

import numpy as np
import pytest
import torch

from bit_group_quantized_gb300 import lib, synth
from tests.helpers import ExpertSource, TIE_GAP, assert_bf16_output, f64, own_tol_for, topk_gap
from tests.test_gpu_layer import build_layer, oracle_layer_token

pytestmark = pytest.mark.gpu


def host_copy(L, t, shape, K, move_router=False):
    """The same layer with the routed-expert pool (and optionally router,
    shared gate and shared expert) copied to pinned host memory."""
    E = shape.E
    keep = {"pool_q": t["pool_q"][:E].cpu().pin_memory(), "pool_sb": t["pool_sb"][:E].cpu().pin_memory()}
    if move_router:
        keep["router"] = t["router"].cpu().pin_memory()
        keep["gate"] = t["shared_gate"].cpu().pin_memory()
        keep["sq"] = t["pool_q"][E].cpu().pin_memory()
        keep["ssb"] = t["pool_sb"][E].cpu().pin_memory()
    else:
        keep["router"], keep["gate"] = t["router"], t["shared_gate"]
        keep["sq"], keep["ssb"] = t["pool_q"][E], t["pool_sb"][E]
    H = lib.MoELayer(shape.d, shape.f, E, K, shape.bits, keep["router"], keep["gate"], keep["pool_q"],
                     keep["pool_sb"], keep["sq"], keep["ssb"])
    return H, keep


@pytest.mark.parametrize("E,d,f,bits,B,move_router", [
    (16, 1024, 256, 4, 1, False),   # batch 1: the device copy runs the persistent kernel
    (16, 1024, 256, 4, 5, True),
    (8, 512, 256, 2, 3, False),
])
def test_host_resident_layer_equals_device_layer(cuda_device, E, d, f, bits, B, move_router):
    shape = synth.PoolShape(d, f, E, bits)
    L, t = build_layer(21, 0, shape, 4, cuda_device)
    t["router"].copy_((t["router"].float() * np.sqrt(4096 / d)).to(torch.bfloat16))
    Hl, keep = host_copy(L, t, shape, 4, move_router)
    x = synth.activations(21, 1, B, d, device=cuda_device)
    a = lib.moe_layer_forward(L, x, want_f32=True, want_route=True)
    b = lib.moe_layer_forward(Hl, x, want_f32=True, want_route=True)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2])  # same experts
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))  # same bits (batches < 16)
    assert torch.equal(a[1], b[1])


def test_host_resident_layer_matches_oracle_at_batch_20(cuda_device):
    """Batch 20: on the device the shared expert's 20 tokens run on tensor
    cores; with host-resident weights everything runs on the grouped GEMVs."""
    shape = synth.PoolShape(1024, 512, 16, 4)
    L, t = build_layer(22, 0, shape, 4, cuda_device)
    t["router"].copy_((t["router"].float() * np.sqrt(4096 / 1024)).to(torch.bfloat16))
    Hl, keep = host_copy(L, t, shape, 4, move_router=True)
    B = 20
    x = synth.activations(22, 1, B, shape.d, device=cuda_device)
    out, _, idx, _, _ = lib.moe_layer_forward(Hl, x, want_route=True)
    torch.cuda.synchronize()
    src = ExpertSource(22, 0, shape)
    xd = f64(x)
    for tok in (0, 7, 19):
        gi = idx[tok].cpu().numpy()
        ref, oi, _, _, logits = oracle_layer_token(t, src, shape, 4, xd[tok], gi)
        if topk_gap(logits, 4) > TIE_GAP:
            assert gi.tolist() == oi.tolist()
        assert_bf16_output(f64(out)[tok], ref, tok, own_tol=own_tol_for(1))


def test_pageable_host_weights_are_rejected(cuda_device):
    shape = synth.PoolShape(512, 256, 8, 4)
    L, t = build_layer(23, 0, shape, 2, cuda_device)
    pageable = t["pool_q"][:8].cpu()  # not pinned: the runtime does not know it
    bad = lib.MoELayer(shape.d, shape.f, 8, 2, 4, t["router"], t["shared_gate"], pageable, t["pool_sb"][:8],
                       t["pool_q"][8], t["pool_sb"][8])
    x = synth.activations(23, 1, 2, shape.d, device=cuda_device)
    with pytest.raises(lib.BGQError) as ei:
        lib.moe_layer_forward(bad, x)
    assert ei.value.status == lib.ERR_INVALID_ARG


@pytest.mark.parametrize("E,d,f,bits,B,move_router", [
    (16, 1024, 256, 4, 1, False),
    (16, 1024, 256, 4, 5, True),
    (8, 512, 256, 2, 3, False),
    (512, 4096, 1024, 4, 4, False),  # the benchmark layer
])
def test_streamed_layer_equals_device_layer(cuda_device, E, d, f, bits, B, move_router):
    """Experts copied into device slots before computing give the same bits as
    the device-resident layer, and the slot header lists exactly the distinct
    selected experts, ascending."""
    shape = synth.PoolShape(d, f, E, bits)
    L, t = build_layer(24, 0, shape, 4, cuda_device)
    t["router"].copy_((t["router"].float() * np.sqrt(4096 / d)).to(torch.bfloat16))
    Hl, keep = host_copy(L, t, shape, 4, move_router)
    x = synth.activations(24, 1, B, d, device=cuda_device)
    slots = lib.alloc((lib.moe_stream_slots_bytes(Hl, B),), torch.uint8, cuda_device)
    a = lib.moe_layer_forward(L, x, want_f32=True, want_route=True)
    b = lib.moe_layer_forward_streamed(Hl, x, slots=slots, want_f32=True, want_route=True)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2])
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1])
    hdr = slots[:256].view(torch.int32).cpu()
    distinct = sorted(set(b[2].cpu().flatten().tolist()))
    assert int(hdr[0]) == len(distinct)
    assert hdr[1:1 + len(distinct)].tolist() == distinct


def test_streamed_layer_matches_oracle_at_batch_20(cuda_device):
    shape = synth.PoolShape(1024, 512, 16, 4)
    L, t = build_layer(25, 0, shape, 4, cuda_device)
    t["router"].copy_((t["router"].float() * np.sqrt(4096 / 1024)).to(torch.bfloat16))
    Hl, keep = host_copy(L, t, shape, 4, move_router=True)
    B = 20
    x = synth.activations(25, 1, B, shape.d, device=cuda_device)
    out, _, idx, _, _ = lib.moe_layer_forward_streamed(Hl, x, want_route=True)
    torch.cuda.synchronize()
    src = ExpertSource(25, 0, shape)
    xd = f64(x)
    for tok in (0, 9, 19):
        gi = idx[tok].cpu().numpy()
        ref, oi, _, _, logits = oracle_layer_token(t, src, shape, 4, xd[tok], gi)
        if topk_gap(logits, 4) > TIE_GAP:
            assert gi.tolist() == oi.tolist()
        assert_bf16_output(f64(out)[tok], ref, tok, own_tol=own_tol_for(1))
