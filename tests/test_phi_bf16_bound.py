"""The packed-bf16 feature map of the tensor-core kernels against e^x, by emulation.

The tensor-core kernels apply phi(x) = elu(x) + 1 ("Why Replace Attention?",
section 5.3, the boxed map) to bf16 tiles in shared memory:
    n = max(-x, 0), p = max(x, 0)       (packed bf16 fma with relu, exact)
    t = fp32(n) * fp32(-log2 e)         (one fp32 product: min(x, 0) log2 e)
    e = ex2.approx.ftz.f32(t)           (fp32 hardware 2^t; results below 2^-126 -> 0)
    e = bf16_rn(e)                      (cvt.rn.bf16x2.f32)
    phi = bf16_rn(p + e)                (packed bf16 add)
This file runs those steps in float64 over every finite bf16 input. The fp32
ex2 is modelled as 2^t within a relative error of 2^-21 in either direction
(bf16 rounding is monotone, so both ends of that interval bound the result),
and the test asserts the bound the kernel source states: relative error at
most 2^-8 + 1e-5 for x >= -87.3, and 0 below (where e^x < 1.2e-38).

It also runs the earlier design (t rounded to bf16 before a bf16 ex2) to
show that this check separates the two: that design already exceeds the bound
in [-2, 0) (0.9 %), and its error grows with |x| to about 13 % in [-40, -20).
"""
import numpy as np

LOG2E_F32 = np.float32(1.4426950408889634)
EX2_REL = 2.0 ** -21          # modelled error of the fp32 hardware ex2
BOUND = 2.0 ** -8 + 1e-5      # stated in the kernel source
FTZ_X = -87.3                 # below: ex2 result under 2^-126, flushed to zero


def all_bf16():
    """Every finite bf16 value, as float64 (and as the float32 it widens to)."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    f32 = (bits << 16).view(np.float32)
    keep = np.isfinite(f32)
    return f32[keep].astype(np.float64), f32[keep]


def bf16_rn(y):
    """Round float64 values to bf16 (8 significant bits), ties to even; zeros stay zero."""
    y = np.asarray(y, np.float64)
    m, e = np.frexp(y)                       # y = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def phi_exact(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def ex2_model(t, ex2_scale):
    """fp32 hardware 2^t (result scaled by ex2_scale), flushed to 0 below 2^-126, then bf16."""
    e = np.exp2(t) * ex2_scale
    e = np.where(np.exp2(t) < 2.0 ** -126, 0.0, e)
    return bf16_rn(e)


def phi_kernel(x64, x32, ex2_scale):
    """The kernel's steps with the fp32 ex2 result scaled by ex2_scale."""
    n32 = np.maximum(-x32, np.float32(0.0))         # relu(-x), exact in bf16
    with np.errstate(over="ignore"):                # huge -x: t = -inf, e = 0
        t = (n32 * -LOG2E_F32).astype(np.float64)   # fp32 product, rounded once
    e = ex2_model(t, ex2_scale)
    p = np.maximum(x64, 0.0)
    return bf16_rn(p + e)


def phi_min_max_form(x64, x32, ex2_scale):
    """The same map as max(x, 0) + min(e^x, 1), e^x of the whole input."""
    with np.errstate(over="ignore"):                # huge x: t = inf, min(e, 1) = 1
        t = (x32 * LOG2E_F32).astype(np.float64)
    t = np.minimum(t, 1.0)                          # t > 0 only feeds min(e, 1) = 1
    m = np.minimum(ex2_model(t, ex2_scale), 1.0)
    return bf16_rn(np.maximum(x64, 0.0) + m)


def phi_old_design(x64):
    """Earlier design: t = bf16(x * bf16(log2 e)), 2^t by a bf16 ex2 (modelled exactly)."""
    log2e_bf16 = bf16_rn(np.log2(np.e))
    t = np.minimum(bf16_rn(x64 * log2e_bf16), 1.0)   # t > 0 only feeds min(e, 1) = 1
    e = bf16_rn(np.exp2(t))
    return bf16_rn(np.maximum(x64, 0.0) + np.minimum(e, 1.0))


def rel_err(got, x):
    ref = phi_exact(x)
    return np.abs(got - ref) / ref


def test_bf16_rounding_helper():
    # Exact bf16 values are fixed points; halfway cases go to the even neighbour.
    x64, _ = all_bf16()
    np.testing.assert_array_equal(bf16_rn(x64), x64)
    assert bf16_rn(1.0 + 2.0 ** -8) == 1.0                 # tie -> even (1.0)
    assert bf16_rn(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6   # tie -> even (odd neighbour up)
    assert bf16_rn(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7


def test_phi_within_stated_bound_over_every_bf16_input():
    x64, x32 = all_bf16()
    live = x64 >= FTZ_X
    worst = 0.0
    for scale in (1.0 - EX2_REL, 1.0, 1.0 + EX2_REL):
        got = phi_kernel(x64, x32, scale)
        err = rel_err(got[live], x64[live])
        worst = max(worst, float(err.max()))
        # Below the flush limit the kernel gives 0 and e^x is below 1.2e-38.
        assert np.all(got[~live] == 0.0)
        assert np.all(phi_exact(x64[~live]) < 1.2e-38)
    assert worst <= BOUND, worst
    # The bound is the bf16 rounding of phi itself: nothing tighter holds.
    assert worst > 2.0 ** -8 * 0.99


def test_relu_form_equals_min_max_form_on_every_bf16_input():
    # exp of min(x, 0) against min(exp(x), 1): the same bits for every finite input,
    # at both ends of the modelled ex2 error as well.
    x64, x32 = all_bf16()
    for scale in (1.0 - EX2_REL, 1.0, 1.0 + EX2_REL):
        np.testing.assert_array_equal(phi_kernel(x64, x32, scale),
                                      phi_min_max_form(x64, x32, scale))


def test_phi_special_values():
    x = np.array([0.0, -0.0, 1.0, -1.0, 2.0 ** -100, -(2.0 ** -100)])
    got = phi_kernel(x, x.astype(np.float32), 1.0)
    np.testing.assert_array_equal(got, [1.0, 1.0, 2.0, bf16_rn(np.exp(-1.0)), 1.0, 1.0])


def test_earlier_design_fails_the_bound_where_it_was_untested():
    x64, _ = all_bf16()
    x64 = x64[x64 >= FTZ_X]
    got = phi_old_design(x64)
    err = rel_err(got, x64)
    band = (x64 >= -40.0) & (x64 < -20.0)
    assert err[band].max() > 0.10          # ~13 % in this band
    assert err[(x64 >= -8.0) & (x64 < -4.0)].max() > 0.03
    assert BOUND < err[(x64 >= -2.0) & (x64 <= 0.0)].max() <= 0.01
