"""Pins of the oracle's bf16 and E4M3 encoders (CPU).

The cache-write bytes must be bit-exact, so the oracle's own encoders are
checked exhaustively against library routines (torch's bf16 and float8_e4m3fn
casts, both round-to-nearest-even) and against the OCP E4M3 definition
(mainarch: "FP8 here is OCP e4m3fn"; Loom Kernels, "Evidence" table, row
"Static FP8 KV-cache write": exact E4M3 cache bytes)."""
import math
import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from tests import _exhaustive


def _pool():
    return ProcessPoolExecutor(max_workers=min(8, os.cpu_count() or 1), mp_context=mp.get_context("spawn"))


def _ranges(lo, hi, parts):
    step = (hi - lo + parts - 1) // parts
    return [(a, min(hi, a + step)) for a in range(lo, hi, step)]


def test_bf16_exhaustive_against_torch():
    """Every one of the 2^32 float32 patterns rounds to torch's bf16 (NaN
    inputs only need to give a NaN)."""
    rs = _ranges(0, 1 << 32, 64)
    with _pool() as ex:
        bad = sum(ex.map(_exhaustive.bf16_range, [r[0] for r in rs], [r[1] for r in rs]))
    assert bad == 0


def test_bf16_worked_values():
    """Hand-worked ties and carries (bf16 keeps 7 mantissa bits)."""
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),                 # tie, 1.0 is even -> down
        (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie, odd 0x3F81 -> up to 0x3F82
        (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),    # above the tie -> up
        (-2.0, 0xC000),
        (65280.0 + 128.0, 0x4780),                 # 65408 = 0x477F8000: tie, 0x477F odd -> 0x4780
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (float(np.float32(3.4e38)), 0x7F80),       # above max finite bf16 + half ulp -> inf
        (2.0 ** -133, 0x0001),                     # smallest bf16 subnormal, exact
        (2.0 ** -134, 0x0000),                     # half of it: tie, 0 is even -> 0
        (1.5 * 2.0 ** -134, 0x0001),               # above the tie -> smallest subnormal
    ]
    x = np.array([c[0] for c in cases], np.float32)
    got = oracle.bf16_rne(x)
    assert [int(g) for g in got] == [c[1] for c in cases]


def test_e4m3_table_matches_ocp_definition():
    """Decode table from the OCP E4M3 (e4m3fn) definition, spot values and
    structure: bias 7, 3 mantissa bits, subnormals m * 2^-9, max 448, NaN
    only at S.1111.111, no infinities."""
    t = oracle.e4m3_table()
    assert t[0x00] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0 and t[0x80] == 0.0
    assert t[0x01] == 2.0 ** -9
    assert t[0x07] == 7 * 2.0 ** -9
    assert t[0x08] == 2.0 ** -6
    assert t[0x38] == 1.0
    assert t[0x7E] == 448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.count_nonzero(np.isnan(t)) == 2
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(t[0x80:0xFF], -t[:0x7F])


def test_e4m3_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    t = oracle.e4m3_table()
    same = (t == ref) | (np.isnan(t) & np.isnan(ref))
    assert same.all()


def test_e4m3_exhaustive_in_range_against_torch():
    """Every float32 with |x| <= 464 (both signs) encodes like torch's
    float8_e4m3fn cast. (Beyond 464 torch gives NaN; saturation is pinned
    separately.)"""
    hi = int(np.array([464.0], np.float32).view(np.uint32)[0]) + 1
    rs = _ranges(0, hi, 64)
    with _pool() as ex:
        bad = sum(ex.map(_exhaustive.e4m3_range, [r[0] for r in rs], [r[1] for r in rs]))
    assert bad == 0


def test_e4m3_saturation_and_specials():
    x = np.array([448.0, 449.0, 464.0, 465.0, 1e6, np.inf, -np.inf, -1e30, np.nan, -np.nan,
                  2.0 ** -10, -2.0 ** -11, 3 * 2.0 ** -11], np.float32)
    got = oracle.e4m3_sat_rne(x)
    exp = [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0xFF, 0x00, 0x80, 0x01]
    assert [int(g) for g in got] == exp


def test_e4m3_worked_ties():
    """Ties between neighbours go to the even code: 1 + 1/16 lies halfway
    between 1.0 (0x38) and 1.125 (0x39) -> 0x38; 1 + 3/16 between 0x39 and
    0x3A -> 0x3A; 2^-10 (halfway between 0 and 2^-9) -> 0x00; 3*2^-10
    (halfway between 0x01 and 0x02) -> 0x02."""
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10], np.float32)
    assert [int(g) for g in oracle.e4m3_sat_rne(x)] == [0x38, 0x3A, 0x00, 0x02]
