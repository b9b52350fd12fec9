"""Comparison rules of the GPU path against the float64 oracle.

Cache bytes and rotated q are unique results: compared bit for bit.
Attention outputs (bf16 out, float32 partials) must satisfy
|gpu - oracle| <= 2e-3 + 1e-2 * |oracle| element by element, and LSE values
|gpu - oracle| <= 1e-3 (an oracle -inf, for an empty split or sequence,
must be -inf on the GPU too)."""
import numpy as np

ATOL = 2e-3
RTOL = 1e-2
LSE_ATOL = 1e-3


def bf16_u16_to_f64(a: np.ndarray) -> np.ndarray:
    return (np.asarray(a, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def assert_close_out(got: np.ndarray, ref: np.ndarray, what: str = "out") -> None:
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu {got[i]!r} oracle {ref[i]!r}")


def assert_close_lse(got: np.ndarray, ref: np.ndarray, what: str = "lse") -> None:
    got = np.asarray(got, np.float64)
    ninf = ref == -np.inf
    if not np.array_equal(got == -np.inf, ninf):
        raise AssertionError(f"{what}: -inf pattern differs ({int((got == -np.inf).sum())} vs {int(ninf.sum())})")
    with np.errstate(invalid="ignore"):
        err = np.abs(np.where(ninf, 0.0, got - ref))
    if not (err <= LSE_ATOL).all():
        i = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"{what}: max |err| {err[i]} at {i}: gpu {got[i]} oracle {ref[i]}")
