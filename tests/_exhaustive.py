"""Workers for the exhaustive encoder pins (run in spawned processes).

Each worker compares the oracle's encoder with torch's cast over one range
of float32 bit patterns and returns the number of mismatches."""
import numpy as np


def bf16_range(lo: int, hi: int) -> int:
    import torch
    import oracle
    bad = 0
    step = 1 << 22
    for a in range(lo, hi, step):
        b = min(hi, a + step)
        u = np.arange(a, b, dtype=np.uint64).astype(np.uint32)
        x = u.view(np.float32)
        mine = oracle.bf16_rne(x)
        ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan_in = np.isnan(x)
        # NaN payloads are not compared: both sides must give some NaN.
        mine_nan = ((mine & 0x7F80) == 0x7F80) & ((mine & 0x7F) != 0)
        bad += int(np.count_nonzero((mine != ref) & ~nan_in))
        bad += int(np.count_nonzero(nan_in & ~mine_nan))
    return bad


def e4m3_range(lo: int, hi: int) -> int:
    """Patterns in [lo, hi) of non-negative float32 magnitudes, both signs."""
    import torch
    import oracle
    bad = 0
    step = 1 << 22
    for a in range(lo, hi, step):
        b = min(hi, a + step)
        u = np.arange(a, b, dtype=np.uint64).astype(np.uint32)
        for sign in (0, 0x80000000):
            x = (u | np.uint32(sign)).view(np.float32)
            mine = oracle.e4m3_sat_rne(x)
            ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            bad += int(np.count_nonzero(mine != ref))
    return bad
