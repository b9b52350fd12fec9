"""The FP8 operand forms of the MLA decode, checked over every input value
(CPU; torch's float8 casts round to nearest even, like the kernel's cvt).

* q_lat: two E4M3 terms under a per-head power of two 2^k chosen so that
  2^k max|q| is in (224, 448]. Exact wherever 2^k|q| >= 2^-2, i.e. for every
  value within 2^9 of the head's largest; below, the error is <= 2^-10 (in
  the scaled units).
* softmax weights: x = 2^7 P in f16, split into three E5M2 terms each
  rounded to nearest; they sum exactly to x for x >= 2^-6 and to within
  2^-17 below, and no term saturates for x <= 2^15."""
import numpy as np
import torch

F8E4 = torch.float8_e4m3fn
F8E5 = torch.float8_e5m2


def _all_bf16_positive():
    v = torch.arange(1, 0x7F80, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double()
    return v[torch.isfinite(v)]


def _scale_exponent(mx: float) -> int:
    """The kernel's choice of k for a head whose largest magnitude is mx."""
    if mx <= 0.0:
        return 0
    e = int(np.frexp(mx)[1]) - 1                 # mx in [2^e, 2^(e+1))
    k = min(max(8 - e, -126), 126)
    if mx * 2.0 ** k > 448.0:
        k -= 1
    return k


def test_scale_puts_the_largest_magnitude_in_224_448():
    for mx in _all_bf16_positive()[::7].tolist():
        k = _scale_exponent(mx)
        if -126 < k < 126:
            assert 224.0 < mx * 2.0 ** k <= 448.0, (mx, k)


def test_two_e4m3_terms_exact_above_a_quarter():
    x = _all_bf16_positive()
    x = x[x <= 448.0]                            # scaled values (the scale is a power of two)
    t1 = x.float().to(F8E4).double()
    t2 = (x - t1).float().to(F8E4).double()
    err = (x - t1 - t2).abs()
    assert torch.all(err[x >= 0.25] == 0)
    assert err.max().item() <= 2.0 ** -10
    assert err[x < 0.25].max().item() > 0        # the threshold is tight


def test_three_e5m2_terms_reproduce_the_f16_weight():
    h = torch.arange(1, 0x7C00, dtype=torch.int32).to(torch.int16).view(torch.float16).double()
    x = h[h <= 2.0 ** 15]
    e1 = x.float().to(F8E5).double()
    y = x - e1
    assert torch.equal(y.half().double(), y)     # the remainders are f16 values: the subtractions are exact
    e2 = y.float().to(F8E5).double()
    z = y - e2
    assert torch.equal(z.half().double(), z)
    e3 = z.float().to(F8E5).double()
    err = (x - e1 - e2 - e3).abs()
    assert torch.all(err[x >= 2.0 ** -6] == 0)
    assert err.max().item() <= 2.0 ** -17
    assert torch.isfinite(e1).all() and e1.max().item() <= 57344.0
