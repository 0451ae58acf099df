"""C ABI checks that need no GPU: the library builds, loads and exports every
entry point declared in include/bgq.h, and argument validation rejects bad
calls before anything is launched (no CUDA call is reached on these paths)."""

import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bgq.h")


@pytest.fixture(scope="module")
def lib():
    from bit_group_quantized_gb300 import build, lib as L

    build.build()
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int32_t|size_t|char\s*\*|const char\s*\*)\s*\*?\s*(\w+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["q4_gemv", "q2_gemv", "moe_route_topk", "moe_expert_swiglu", "moe_layer_forward",
              "moe_layer_workspace_bytes", "moe_stack_decode", "bgq_status_string", "bgq_read_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    L = lib.load()
    for n in names:
        assert hasattr(L, n)
    assert set(lib._SIGS) >= set(names)


def test_q8_gemv_validation(lib):
    L = lib.load()
    W = qmat(lib, bits=8)
    assert L.q8_gemv(None, FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(W), None, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(W), FAKE + 2, FAKE, 1, None) == lib.ERR_INVALID_ARG  # misaligned x
    assert L.q8_gemv(C.byref(W), FAKE, FAKE + 8, 1, None) == lib.ERR_INVALID_ARG  # misaligned y
    assert L.q8_gemv(C.byref(W), FAKE, FAKE, 0, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(W), FAKE, FAKE, 65, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(qmat(lib, bits=4)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG  # wrong bits
    assert L.q4_gemv(C.byref(W), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG  # 8-bit only through q8_gemv
    assert L.bgq_qgemv_variant(C.byref(W), FAKE, FAKE, 1, 1, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(qmat(lib, bits=8, group=128)), FAKE, FAKE, 1, None) == lib.ERR_UNSUPPORTED
    assert L.q8_gemv(C.byref(qmat(lib, bits=8, cols=100)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(qmat(lib, bits=8, cols=768)), FAKE, FAKE, 1, None) == lib.ERR_UNSUPPORTED
    assert L.q8_gemv(C.byref(qmat(lib, bits=8, cols=65536 + 512)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(qmat(lib, bits=8, q=FAKE + 4)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(qmat(lib, bits=8, sb=FAKE + 2)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q8_gemv(C.byref(qmat(lib, bits=8, rows=0)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG


def test_status_strings(lib):
    assert lib.status_string(0) == "ok"
    assert "workspace" in lib.status_string(5)
    assert lib.load().bgq_abi_version() == 103


FAKE = 0x10000000  # 256-byte aligned, never dereferenced: validation fails first


def qmat(lib, rows=1024, cols=4096, bits=4, q=FAKE, sb=FAKE, group=64):
    return lib.bgq_qmatrix(q, sb, rows, cols, bits, group)


def test_gemv_validation(lib):
    L = lib.load()
    W = qmat(lib)
    assert L.q4_gemv(None, FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q4_gemv(C.byref(W), None, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q4_gemv(C.byref(W), FAKE + 2, FAKE, 1, None) == lib.ERR_INVALID_ARG  # misaligned x
    assert L.q4_gemv(C.byref(W), FAKE, FAKE, 0, None) == lib.ERR_INVALID_ARG  # batch 0
    assert L.q4_gemv(C.byref(W), FAKE, FAKE, 65, None) == lib.ERR_INVALID_ARG
    W2 = qmat(lib, bits=2)
    assert L.q4_gemv(C.byref(W2), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG  # wrong bits for q4
    assert L.q2_gemv(C.byref(W), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q4_gemv(C.byref(qmat(lib, group=128)), FAKE, FAKE, 1, None) == lib.ERR_UNSUPPORTED
    assert L.q4_gemv(C.byref(qmat(lib, cols=100)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q4_gemv(C.byref(qmat(lib, cols=192)), FAKE, FAKE, 1, None) == lib.ERR_UNSUPPORTED
    assert L.q4_gemv(C.byref(qmat(lib, bits=3)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q4_gemv(C.byref(qmat(lib, q=FAKE + 4)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.q4_gemv(C.byref(qmat(lib, rows=0)), FAKE, FAKE, 1, None) == lib.ERR_INVALID_ARG
    assert L.bgq_qgemv_variant(C.byref(W), FAKE, FAKE, 1, 7, None) == lib.ERR_INVALID_ARG


def layer_struct(lib, **kw):
    d, f, E, K, bits = kw.get("d", 4096), kw.get("f", 1024), kw.get("E", 512), kw.get("K", 4), kw.get("bits", 4)
    mw = d * f * bits // 32
    mg = d * f // 64 * 2
    return lib.bgq_moe_layer(d, f, E, K, bits, kw.get("group", 64), FAKE, FAKE, FAKE, FAKE,
                             kw.get("qs", 3 * mw), kw.get("sbs", 3 * mg), FAKE, FAKE)


def test_layer_validation_and_workspace(lib):
    L = lib.load()
    Ls = layer_struct(lib)
    need = L.moe_layer_workspace_bytes(C.byref(Ls), 1)
    assert need > 0 and need % 256 == 0
    assert L.moe_layer_workspace_bytes(C.byref(Ls), 64) > need
    args = lambda ws, n: (C.byref(Ls), FAKE, 1, FAKE, None, None, None, None, ws, n, None)
    assert L.moe_layer_forward(*args(None, need)) == lib.ERR_WORKSPACE
    assert L.moe_layer_forward(*args(FAKE, need - 256)) == lib.ERR_WORKSPACE
    assert L.moe_layer_forward(*args(FAKE + 16, need)) == lib.ERR_WORKSPACE  # misaligned ws
    for bad in (dict(K=9), dict(E=2000), dict(K=600, E=512), dict(group=32), dict(d=4000)):
        Lb = layer_struct(lib, **bad)
        r = L.moe_layer_forward(C.byref(Lb), FAKE, 1, FAKE, None, None, None, None, FAKE, 1 << 30, None)
        assert r in (lib.ERR_UNSUPPORTED, lib.ERR_INVALID_ARG), bad
    Lb = layer_struct(lib, qs=100)  # expert stride shorter than one expert
    assert L.moe_layer_forward(C.byref(Lb), FAKE, 1, FAKE, None, None, None, None, FAKE, 1 << 30, None) == \
        lib.ERR_INVALID_ARG
    assert L.moe_layer_forward(C.byref(Ls), FAKE, 0, FAKE, None, None, None, None, FAKE, 1 << 30, None) == \
        lib.ERR_INVALID_ARG
    assert L.moe_layer_forward(C.byref(Ls), FAKE, 257, FAKE, None, None, None, None, FAKE, 1 << 30, None) == \
        lib.ERR_INVALID_ARG
    assert L.moe_layer_forward(C.byref(Ls), FAKE, 1, None, None, None, None, None, FAKE, 1 << 30, None) == \
        lib.ERR_INVALID_ARG  # no output at all


def test_route_and_expert_validation(lib):
    L = lib.load()
    need = L.moe_route_workspace_bytes(1, 512)
    assert need > 0
    r = L.moe_route_topk(FAKE, None, FAKE, 1, 4096, 512, 4, FAKE, FAKE, None, None, FAKE, need - 1, None)
    assert r == lib.ERR_WORKSPACE
    r = L.moe_route_topk(FAKE, None, FAKE, 1, 4096, 512, 9, FAKE, FAKE, None, None, FAKE, need, None)
    assert r == lib.ERR_UNSUPPORTED
    r = L.moe_route_topk(FAKE, None, FAKE, 1, 4000, 512, 4, FAKE, FAKE, None, None, FAKE, need, None)
    assert r == lib.ERR_UNSUPPORTED
    e = lib.bgq_expert(qmat(lib, 1024, 4096), qmat(lib, 1024, 4096), qmat(lib, 4096, 1024))
    need = L.moe_expert_workspace_bytes(C.byref(e), 1)
    assert L.moe_expert_swiglu(C.byref(e), FAKE, 1, FAKE, None, FAKE, need - 256, None) == lib.ERR_WORKSPACE
    bad = lib.bgq_expert(qmat(lib, 1024, 4096), qmat(lib, 1024, 4096), qmat(lib, 4096, 2048))
    assert L.moe_expert_swiglu(C.byref(bad), FAKE, 1, FAKE, None, FAKE, 1 << 30, None) == lib.ERR_INVALID_ARG


def test_stack_validation(lib):
    L = lib.load()
    layers = (lib.bgq_moe_layer * 2)(layer_struct(lib), layer_struct(lib, f=2048))
    rho = (C.c_void_p * 2)(FAKE, FAKE)
    r = L.moe_stack_decode(layers, rho, 2, 1e-6, FAKE, FAKE, None, None, FAKE, 1 << 30, None)
    assert r == lib.ERR_INVALID_ARG  # mixed shapes
    layers = (lib.bgq_moe_layer * 1)(layer_struct(lib))
    assert L.moe_stack_decode(layers, rho, 0, 1e-6, FAKE, FAKE, None, None, FAKE, 1 << 30, None) == \
        lib.ERR_INVALID_ARG
    need = L.moe_stack_workspace_bytes(layers, 1)
    assert L.moe_stack_decode(layers, rho, 1, 1e-6, FAKE, FAKE, None, None, FAKE, need - 256, None) == \
        lib.ERR_WORKSPACE
    assert L.bgq_rmsnorm(FAKE, None, 1, 100, 1e-6, FAKE, None) == lib.ERR_INVALID_ARG
    assert L.bgq_read_device_status(None, None) == lib.ERR_INVALID_ARG


def test_streamed_slot_bytes_and_validation(lib):
    """moe_stream_slots_bytes: a 256-byte-aligned header (count + one int per
    slot), then min(batch*K, E) slots of one expert's gate/up/down codes and
    scale/bias rows; the streamed forward rejects missing, short or misaligned
    slot buffers before touching anything."""
    L = lib.load()
    Ls = layer_struct(lib)
    q = 3 * 4096 * 1024 * 4 // 8           # codes of gate, up, down (4-bit)
    sb = 3 * (4096 * 1024 // 64) * 2 * 2    # one bf16 (scale, bias) pair per group of 64
    assert L.moe_stream_slots_bytes(C.byref(Ls), 1) == 256 + 4 * (q + sb)
    assert L.moe_stream_slots_bytes(C.byref(Ls), 3) == 256 + 12 * (q + sb)
    assert L.moe_stream_slots_bytes(C.byref(Ls), 200) == 2304 + 512 * (q + sb)  # capped at E slots
    L2 = layer_struct(lib, bits=2)
    assert L.moe_stream_slots_bytes(C.byref(L2), 1) == 256 + 4 * (q // 2 + sb)
    need = L.moe_layer_workspace_bytes(C.byref(Ls), 1)
    slots = L.moe_stream_slots_bytes(C.byref(Ls), 1)
    call = lambda sl, n: L.moe_layer_forward_streamed(C.byref(Ls), FAKE, 1, FAKE, None, None, None, None, sl, n,
                                                      FAKE, need, None)
    assert call(None, slots) == lib.ERR_WORKSPACE
    assert call(FAKE, slots - 256) == lib.ERR_WORKSPACE
    assert call(FAKE + 16, slots) == lib.ERR_WORKSPACE


def test_noalloc_rejects_what_the_workspace_entry_point_rejects(lib):
    """moe_layer_forward_noalloc runs moe_layer_forward's argument checks, in
    the same order, before it clears its scratch array: a bad call returns the
    same status from both entry points and nothing is enqueued (no CUDA call
    is reached on these paths, so this runs without a GPU)."""
    L = lib.load()
    Ls = layer_struct(lib)
    big = 1 << 30

    def both(layer, x=FAKE, batch=1, out=FAKE, out_f32=None):
        a = L.moe_layer_forward(C.byref(layer) if layer is not None else None, x, batch, out, out_f32, None, None,
                                None, FAKE, big, None)
        b = L.moe_layer_forward_noalloc(C.byref(layer) if layer is not None else None, x, batch, out, out_f32, None,
                                        None, None, None)
        return a, b

    cases = [
        dict(layer=None),
        dict(layer=Ls, x=None),
        dict(layer=Ls, x=FAKE + 2),       # misaligned input
        dict(layer=Ls, out=None),         # no output at all
        dict(layer=Ls, out=FAKE + 8),     # misaligned output
        dict(layer=Ls, out_f32=FAKE + 4),
        dict(layer=Ls, batch=0),
        dict(layer=Ls, batch=257),
        dict(layer=layer_struct(lib, E=2000)),        # beyond the expert limit: unsupported, not "workspace"
        dict(layer=layer_struct(lib, K=9)),
        dict(layer=layer_struct(lib, group=32)),
        dict(layer=layer_struct(lib, bits=3)),
        dict(layer=layer_struct(lib, d=4000)),
        dict(layer=layer_struct(lib, qs=100)),
    ]
    for c in cases:
        a, b = both(**c)
        assert a == b and a in (lib.ERR_INVALID_ARG, lib.ERR_UNSUPPORTED), (c, a, b)
    assert both(layer_struct(lib, E=2000))[1] == lib.ERR_UNSUPPORTED
    # a valid call too large for the 4 MiB array (batch 36 at the full shape)
    assert L.moe_layer_workspace_bytes(C.byref(Ls), 36) > (4 << 20)
    assert L.moe_layer_forward_noalloc(C.byref(Ls), FAKE, 36, FAKE, None, None, None, None, None) == \
        lib.ERR_WORKSPACE


def test_gemv_chain_validation(lib):
    L = lib.load()

    def chain(*mats):
        arr = (lib.bgq_qmatrix * len(mats))()
        for i, m in enumerate(mats):
            arr[i] = m
        return arr

    good = chain(qmat(lib, rows=4096, cols=4096), qmat(lib, rows=4096, cols=4096))
    ws_bytes = L.bgq_gemv_chain_workspace_bytes(good, 2, 1)
    assert ws_bytes >= 512 + 2 * 4096 * 2

    def call(W, n, x=FAKE, batch=1, norm=1, eps=1e-6, residual=1, out=FAKE, out_f32=None, ws=FAKE, nbytes=ws_bytes):
        return L.bgq_gemv_chain(W, n, x, batch, norm, None, eps, residual, out, out_f32, ws, nbytes, None)

    assert call(None, 2) == lib.ERR_INVALID_ARG
    assert call(good, 0) == lib.ERR_INVALID_ARG
    assert call(good, 9) == lib.ERR_INVALID_ARG
    assert call(good, 2, x=None) == lib.ERR_INVALID_ARG
    assert call(good, 2, x=FAKE + 2) == lib.ERR_INVALID_ARG  # misaligned x
    assert call(good, 2, out=None) == lib.ERR_INVALID_ARG  # no output at all
    assert call(good, 2, batch=0) == lib.ERR_INVALID_ARG
    assert call(good, 2, batch=9) == lib.ERR_INVALID_ARG
    assert call(good, 2, eps=0.0) == lib.ERR_INVALID_ARG  # norm needs eps > 0
    assert call(good, 2, ws=None) == lib.ERR_WORKSPACE
    assert call(good, 2, nbytes=ws_bytes - 1) == lib.ERR_WORKSPACE
    # each step's columns are the previous step's rows
    bad = chain(qmat(lib, rows=4096, cols=4096), qmat(lib, rows=4096, cols=2048))
    assert call(bad, 2) == lib.ERR_INVALID_ARG
    assert L.bgq_gemv_chain_workspace_bytes(bad, 2, 1) == 0
    # mixed bits
    assert call(chain(qmat(lib, rows=4096, cols=4096), qmat(lib, rows=4096, cols=4096, bits=2)), 2) == \
        lib.ERR_INVALID_ARG
    # residual needs the last step back at d rows
    wide = chain(qmat(lib, rows=2048, cols=4096))
    assert call(wide, 1, nbytes=L.bgq_gemv_chain_workspace_bytes(wide, 1, 1)) == lib.ERR_INVALID_ARG
    # each step's GEMV stages as many inputs per launch as fit in shared
    # memory, so 12288 columns are taken at any batch; a row so wide that not
    # even one staged input fits is not
    qkv = chain(qmat(lib, rows=12288, cols=4096), qmat(lib, rows=4096, cols=12288))
    assert L.bgq_gemv_chain_workspace_bytes(qkv, 2, 8) > 0
    huge = chain(qmat(lib, rows=4096, cols=81920))
    assert call(huge, 1, batch=1, nbytes=1 << 30) == lib.ERR_UNSUPPORTED
    assert L.bgq_gemv_chain_workspace_bytes(huge, 1, 1) == 0
