"""Host-side check of the 8-bit GEMV's work split (no GPU needed).

The index arithmetic of gemv8.cu, restated: the input staging (one thread per
8 values, two 16-byte slots per 16-code part), the one-shot kernel (one row
group per warp) and the persistent streaming kernel (row groups strided over
the grid's warps, rows packed several to an item when a row has fewer than 8
parts per lane, or split into chunks when it has more). For every shape the
entry point accepts: each staged slot and part-info entry is written exactly
once and inside its buffer, every (row, part) of the matrix is read exactly
once and every output row is written exactly once, with all loads inside the
code and scale/bias arrays.
"""

import pytest

NIT_REGS = 8  # parts per lane held in registers (kG8Nit)
THREADS = 256
MAX_SMEM = 227 * 1024


def row_geo(cols):
    P = cols * 8 // 128
    LPR = 32 if P >= 32 else P
    return P, LPR, 32 // LPR, P // LPR


def cols_supported(cols):
    if cols <= 0 or cols % 64:
        return False
    P = cols // 16
    return P % 32 == 0 or 32 % P == 0


def max_tokens(cols):
    T = 8
    while T > 0 and T * cols * 3 + T * (cols // 16) * 8 > MAX_SMEM:
        T -= 1
    return T


def check_staging(T, cols):
    P, LPR, RPP, NIT = row_geo(cols)
    nslots, npi = T * cols * 2 // 16, T * P
    hpr, total = cols // 8, T * cols // 8
    slots, pis = set(), set()
    for i in range(total):
        t, h = divmod(i, hpr)
        p, j = divmod(h, 2)
        it, lp = divmod(p, LPR)
        s = ((t * NIT + it) * 2 + j) * LPR + lp
        assert 0 <= s < nslots and s not in slots
        slots.add(s)
        if j == 0:
            assert t * P + p not in pis
            pis.add(t * P + p)
    assert len(slots) == nslots and len(pis) == npi
    # a group of 64 values is 8 consecutive threads of one warp (shuffle max)
    assert hpr % 8 == 0 and THREADS % 8 == 0


def check_one_shot(rows, cols, gpr):
    P, LPR, RPP, NIT = row_geo(cols)
    wpr = cols // 4
    grid = -(-rows // (8 * RPP))
    seen, out = set(), set()
    for b in range(grid):
        for warp in range(8):
            for lane in range(32):
                rs, lp = divmod(lane, LPR)
                row = (b * 8 + warp) * RPP + rs
                if row >= rows:
                    continue
                for it in range(NIT):
                    p = it * LPR + lp
                    assert row * wpr + 4 * p + 3 < rows * wpr
                    g = 0 if gpr == 1 else p >> 2
                    assert g < gpr and row * gpr + g < rows * gpr
                    assert (row, p) not in seen
                    seen.add((row, p))
                if lp == 0:
                    assert row not in out
                    out.add(row)
    assert len(seen) == rows * P and len(out) == rows


def check_stream(rows, cols, gpr, nsm=152):
    P, LPR, RPP, NIT = row_geo(cols)
    wpr = cols // 4
    nrg = -(-rows // RPP)
    grid = min(-(-nrg // 8), 2 * nsm)
    W = grid * 8
    pack = NIT < NIT_REGS and NIT_REGS % NIT == 0
    RI = NIT_REGS // NIT if pack else 1
    nchunk = 1 if pack else -(-NIT // NIT_REGS)
    seen, out = set(), set()
    for gw in range(W):
        nmine = (nrg - 1 - gw) // W + 1 if gw < nrg else 0
        nitems = -(-nmine // RI) if pack else nmine * nchunk
        for item in range(nitems):
            for lane in range(32):
                rs, lp = divmod(lane, LPR)
                for i in range(NIT_REGS):
                    if RI == 1:
                        j = item // nchunk
                        it = (item - j * nchunk) * NIT_REGS + i
                    else:
                        r = i // NIT
                        j, it = item * RI + r, i - r * NIT
                    if not (j < nmine and it < NIT):
                        continue
                    row = (gw + j * W) * RPP + rs
                    if row >= rows:
                        continue
                    p = it * LPR + lp
                    assert row * wpr + 4 * p + 3 < rows * wpr
                    g = 0 if gpr == 1 else p >> 2
                    assert g < gpr
                    assert (row, p) not in seen
                    seen.add((row, p))
                    if it == NIT - 1 and lp == 0:
                        assert row not in out
                        out.add(row)
    assert len(seen) == rows * P and len(out) == rows


SHAPES = [(1024, 4096, 64), (1000, 4096, 64), (4096, 1024, 64), (333, 512, 64), (200, 256, 64), (64, 64, 64),
          (96, 12288, 64), (1024, 4096, 4096), (777, 1024, 1024), (128, 128, 128), (300, 1536, 64),
          (50, 2560, 2560), (5000, 1024, 64), (20000, 256, 256)]


@pytest.mark.parametrize("rows,cols,group", SHAPES)
def test_q8_work_split_covers_the_matrix_once(rows, cols, group):
    assert cols_supported(cols)
    gpr = 1 if group == cols else cols // 64
    check_one_shot(rows, cols, gpr)
    check_stream(rows, cols, gpr)


@pytest.mark.parametrize("cols", [64, 128, 256, 512, 1024, 1536, 4096, 8192, 8704, 11264, 11776, 65536])
def test_q8_staging_slots_written_once(cols):
    T = max_tokens(cols)
    assert T >= 1
    check_staging(T, cols)
    if cols <= 8192:
        assert T == 8
    assert T * cols * 3 + T * (cols // 16) * 8 <= MAX_SMEM


def test_q8_token_index_by_reciprocal_is_exact():
    """Streaming staging finds t = floor(i / hpr) as int((i + 0.5) * fl(1 / hpr)) in fp32."""
    np = pytest.importorskip("numpy")
    for cols in [c for c in range(512, 65537, 512)] + [64, 128, 256]:
        T = max_tokens(cols)
        hpr = cols // 8
        i = np.arange(T * hpr, dtype=np.int64)
        inv = np.float32(1.0) / np.float32(hpr)
        t = ((i.astype(np.float32) + np.float32(0.5)) * inv).astype(np.int64)
        assert np.array_equal(t, i // hpr), cols
