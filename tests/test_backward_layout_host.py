"""Bounds of the backward scan's shared-memory staging, checked on the CPU for every supported
shape (dk, dv in {64, 128}, 0 <= R <= 15, float32 or bfloat16 io, ragged T).

The scan kernel copies each chunk's per-token inputs into one of two shared-memory buffers with
16- and 4-byte cp.async and reads them back per lane.  This file restates the buffer layout and
the copy and read index arithmetic of prism_backward.cu (the constants are read from the source)
and checks that every copy and read stays inside its region and its tensor, with the alignment
the copy size needs, and that both buffers fit the shared memory the kernel is given.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "ssm_sequence_layer_gb300", "csrc", "prism_backward.cu")).read()


def const(name):
    m = re.search(r"constexpr int %s = ([0-9 *]+);" % name, SRC)
    assert m, name
    return eval(m.group(1))  # a product of integer literals


LPR, SCAN_WARPS, SCAN_SMEM, NT = const("LPR"), const("SCAN_WARPS"), const("kScanSmem"), const("NT")
ROWS = SCAN_WARPS * 32 // LPR
RMAX = const("RMAX")


def align16(n):
    return (n + 15) & ~15


def layout(ct, dk, R, io):
    q = 0
    k = q + align16(ct * dk * io)
    u = k + align16(ct * dk * io)
    row = u + align16(ct * R * dk * io)
    x = row + ct * ROWS * 4
    gate = x + ct * R * ROWS * 4
    return dict(q=q, k=k, u=u, row=row, x=x, gate=gate, bytes=gate + align16(2 * ct * 4))


def scan_chunk(dk, R, io):
    ct = 32
    while ct > 1 and 2 * layout(ct, dk, R, io)["bytes"] > SCAN_SMEM:
        ct >>= 1
    return ct


def test_layout_matches_the_source():
    # the regions and their order, as the kernel lays them out
    for part in ("s.q = 0", "s.k = s.q + align16(ct * dk * io_bytes)", "s.u = s.k + align16(ct * dk * io_bytes)",
                 "s.row = s.u + align16(ct * R * dk * io_bytes)", "s.x = s.row + ct * ROWS * 4",
                 "s.gate = s.x + ct * R * ROWS * 4", "s.bytes = s.gate + align16(2 * ct * 4)"):
        assert part in SRC, part


SHAPES = [(dk, dv, R, io) for dk in (64, 128) for dv in (64, 128) for R in range(RMAX + 1) for io in (2, 4)]


@pytest.mark.parametrize("dk,dv,R,io", SHAPES)
def test_staging_copies_and_reads_stay_in_bounds(dk, dv, R, io):
    ct = scan_chunk(dk, R, io)
    L = layout(ct, dk, R, io)
    assert ct >= 1 and 2 * L["bytes"] <= SCAN_SMEM <= 227 * 1024
    assert all(L[p] % 16 == 0 for p in ("k", "u", "row", "x", "gate", "bytes"))
    assert dv % ROWS == 0 and dk % LPR == 0
    npl = dk // LPR
    per16 = 16 // io
    for T in (1, 3, ct, ct + 5, 3 * ct - 1):
        for t0 in range(0, T, ct):
            n = min(ct, T - t0)
            for i0 in range(0, dv, ROWS):
                # k and q: n * dk elements from token t0, 16-byte pieces
                nk = n * dk // per16
                assert (n * dk) % per16 == 0
                assert L["k"] + nk * 16 <= L["u"] and L["q"] + nk * 16 <= L["k"]
                assert (t0 * dk + nk * per16) <= T * dk and (dk * io) % 16 == 0
                # u: n * R * dk elements
                nu = n * R * dk // per16
                assert L["u"] + nu * 16 <= L["row"] and t0 * R * dk + nu * per16 <= T * R * dk
                # the rows' v (io) or dout (fp32) entries: 16-byte pieces of one token's ROWS values
                for row_bytes, elem in ((ROWS * io, io), (ROWS * 4, 4)):
                    pieces = row_bytes // 16
                    assert row_bytes % 16 == 0 and pieces * 16 <= ROWS * 4
                    last = (t0 + n - 1) * dv + i0 + (pieces - 1) * (16 // elem) + 16 // elem
                    assert last <= T * dv
                    assert ((i0 * elem) % 16 == 0) and ((dv * elem) % 16 == 0)
                assert L["row"] + n * ROWS * 4 <= L["x"]
                # x: (token, level) pairs, ROWS floats each in 16-byte pieces
                assert L["x"] + n * R * ROWS * 4 <= L["gate"]
                assert ((t0 + n - 1) * R + (R - 1)) * dv + i0 + ROWS <= max(T * R * dv, 0) or R == 0
                # gates: alpha then beta, n floats each, 4-byte pieces
                assert L["gate"] + 2 * n * 4 <= L["bytes"]
            # per-lane reads: columns [col, col + npl) of a token's row, 16-byte vectors
            for lane in range(32):
                col = (lane % LPR) * npl
                assert col + npl <= dk and (col * io) % 16 == 0 and (npl * io) % 16 == 0
                rw = lane // LPR
                assert rw < 32 // LPR


@pytest.mark.parametrize("dk", [64, 128])
@pytest.mark.parametrize("dv", [64, 128])
def test_token_grad_shared_memory_fits_its_attribute(dk, dv):
    def floats(dk_, dv_, R):
        return (dv_ * dk_ + dk_ + 4 * dv_ + R * dv_ + (NT // dk_) * (3 + R) * dk_ + (NT // 32) * (4 + R) + NT // 32
                + 4 + R)
    assert "return (size_t)dv * dk + dk + 4 * (size_t)dv + (size_t)R * dv + (size_t)(NT / dk) * (3 + R) * dk +" in SRC
    most = floats(dk, 128, RMAX) * 4  # what the attribute is set to
    for R in range(RMAX + 1):
        assert floats(dk, dv, R) * 4 <= most <= 227 * 1024
