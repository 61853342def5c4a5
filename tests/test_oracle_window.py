"""Pins of the oracle's statistics and window choice (ZipCCL digest, 3.1).

* s1 and s2 are compared bit for bit with Python's exact rational sums
  (``fractions.Fraction``; ``float()`` of a Fraction rounds correctly).
* var is compared with numpy's float64 ``var(ddof=1)`` (torch.std's Bessel
  correction) and with the exact rational variance.
* E0 is compared with the integer nearest the argmax of the window mass
  P_win(x) = erf(2^(x+7)/(sigma sqrt 2)) - erf(2^x/(sigma sqrt 2)) (Eq. 1),
  found numerically with math.erf -- independent of the closed form.
* The closed-form constants (u ~ 0.0172, x_opt = log2 sigma - 5.35) and
  the Figure-2 worked example (sigma = 1: per-binade shares, 97.5% window,
  2.5% escapes) are checked against tests/golden/zipccl_fig2_binades.txt.
* Exact ties round up; the fallbacks and the clamp behave as stated.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def bf16_to_f64(x):
    # NaN patterns stay NaN (numpy flags the cast of a signalling NaN)
    with np.errstate(invalid="ignore"):
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def exact_sums(x):
    v = bf16_to_f64(x)
    fin = np.isfinite(v)
    s1 = sum((Fraction(float(a)) for a in v[fin]), Fraction(0))
    s2 = sum((Fraction(float(a)) ** 2 for a in v[fin]), Fraction(0))
    return s1, s2, int(fin.sum())


def rand_bf16(rng, n, kind):
    if kind == "gauss":
        v = rng.normal(0, 0.02, n)
    elif kind == "wide":
        v = rng.normal(0, 1, n) * np.exp2(rng.integers(-130, 120, n))
    elif kind == "mean":
        v = 1.0 + rng.normal(0, 0.01, n)
    elif kind == "sub":
        return rng.integers(0, 256, n).astype(np.uint16) | (rng.integers(0, 2, n).astype(np.uint16) << 15)
    else:
        return rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16)
    f = v.astype(np.float32)  # test-side quantisation only needs some BF16 values
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("kind", ["gauss", "wide", "mean", "sub", "bits"])
@pytest.mark.parametrize("n", [1, 2, 3, 17, 1000])
def test_sums_are_exact_then_rounded(orc, kind, n):
    rng = np.random.default_rng(hash((kind, n)) % 2**32)
    x = rand_bf16(rng, n, kind)
    st = orc.stats(x)
    s1, s2, nf = exact_sums(x)
    assert st["n"] == n and st["n_finite"] == nf
    assert st["s1"] == float(s1)
    assert st["s2"] == float(s2)
    hist = np.bincount(((x.astype(np.uint32) >> 7) & 0xFF), minlength=256)
    assert np.array_equal(st["hist"], hist.astype(np.uint64))
    if nf >= 2:
        exact_var = (s2 - s1 * s1 / nf) / (nf - 1)
        if exact_var > 0 and kind != "mean":
            assert st["var"] == pytest.approx(float(exact_var), rel=1e-12)
            v = bf16_to_f64(x)
            v = v[np.isfinite(v)]
            if np.all(np.abs(v) < 1e150):
                assert st["var"] == pytest.approx(np.var(v, ddof=1), rel=1e-9)
        if kind == "mean" and exact_var > 0:
            # cancellation: s2 and s1^2/N agree to ~1e-4 relative
            assert st["var"] == pytest.approx(float(exact_var), rel=1e-8)


def test_window_K_and_closed_form_constants(orc):
    K = orc.window_K()
    assert K == 16383.0 / (14.0 * math.log(2.0))
    # (128^2 - 1) u^2 = ln 128  ->  u ~ 0.0172  (digest 3.1)
    u = math.sqrt(math.log(128.0) / (128 ** 2 - 1))
    assert round(u, 4) == 0.0172
    # x_opt - log2 sigma = log2(sqrt(2) u) = 1/2 log2(14 ln2 / 16383) ~ -5.35
    c = math.log2(math.sqrt(2.0) * u)
    assert c == pytest.approx(0.5 * math.log2(14 * math.log(2) / 16383), abs=1e-12)
    assert round(c, 2) in (-5.36, -5.35)
    # the threshold form: var >= K 2^(2k-1)  <=>  x_opt + 1/2 >= k
    assert 0.5 * math.log2(1.0 / K) == pytest.approx(c, abs=1e-12)


def p_win(x, sigma):
    a = math.erf(2.0 ** (x + 7) / (sigma * math.sqrt(2)))
    b = math.erf(2.0 ** x / (sigma * math.sqrt(2)))
    return a - b


def argmax_pwin(sigma):
    """Golden-section search of Eq. 1's window mass over real x."""
    lo = math.log2(sigma) - 12
    hi = math.log2(sigma) + 2
    g = (math.sqrt(5) - 1) / 2
    a, b = lo, hi
    for _ in range(200):
        c = b - g * (b - a)
        d = a + g * (b - a)
        if p_win(c, sigma) > p_win(d, sigma):
            b = d
        else:
            a = c
    return 0.5 * (a + b)


def test_window_is_nearest_integer_to_eq1_argmax(orc):
    rng = np.random.default_rng(7)
    checked = 0
    for log2s in list(np.linspace(-14, 6, 81)) + list(rng.uniform(-20, 10, 60)):
        sigma = 2.0 ** log2s
        xs = argmax_pwin(sigma)
        if abs((xs - math.floor(xs)) - 0.5) < 1e-6:
            continue  # too close to a tie for the numerical search
        x0 = math.floor(xs + 0.5)
        assert orc.window_from_var(sigma * sigma) == x0 + 127, (sigma, xs)
        checked += 1
    assert checked > 120


def load_fig2():
    shares, extra = {}, {}
    with open(os.path.join(HERE, "golden", "zipccl_fig2_binades.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            k, v = line.split()
            if k in ("window", "escape"):
                extra[k] = float(v)
            else:
                shares[int(k)] = float(v)
    return shares, extra


def test_figure2_worked_example(orc):
    shares, extra = load_fig2()
    # the printed bars are erf differences per binade at sigma = 1
    for x, pct in shares.items():
        p = math.erf(2.0 ** (x + 1) / math.sqrt(2)) - math.erf(2.0 ** x / math.sqrt(2))
        assert round(100 * p, 1) == pytest.approx(pct, abs=0.051), x
    assert sum(shares.values()) == pytest.approx(extra["window"], abs=0.15)
    # sigma = 1: window from binade -5 (E0 = 122) covering -5..+1
    assert orc.window_from_var(1.0) == 122
    assert sorted(shares) == list(range(-5, 2))
    # on a seeded N(0,1) sample the oracle's histogram reproduces the bars
    # and the escape share, within binomial tolerance
    import synth
    n = 1 << 20
    x = synth.gaussian_bf16(n, 1.0, synth.key_of(11, 0)).numpy().view(np.uint16)
    st = orc.stats(x)
    assert st["E0"] == 122 and st["rule"] == 0
    for xb, pct in shares.items():
        frac = st["hist"][127 + xb] / n
        p = pct / 100
        assert abs(frac - p) < 5 * math.sqrt(p * (1 - p) / n) + 0.0006, xb
    esc = st["n_escape"] / n
    assert esc == pytest.approx(extra["escape"] / 100, abs=0.002)


def test_exact_tie_rounds_up(orc):
    K = orc.window_K()
    for k in (-20, -11, -6, 0, 3):
        t = math.ldexp(K, 2 * k - 1)
        assert orc.window_from_var(t) == 127 + k
        assert orc.window_from_var(math.nextafter(t, 0)) == 127 + k - 1
        assert orc.window_from_var(math.nextafter(t, math.inf)) == 127 + k


def test_sums_round_ties_to_even(orc):
    """Exact sums halfway between two doubles (and a hair above) round to
    nearest, ties to even, at several scales: the stated value of each
    constructed case, and float() of the exact Fraction."""
    import synth
    cases = synth.rounding_tie_cases()
    assert len(cases) == 66
    for name, x in cases:
        st = orc.stats(x)
        s1, s2, _ = exact_sums(x)
        assert st["s1"] == float(s1), name
        assert st["s2"] == float(s2), name
    by = dict(cases)
    assert orc.stats(by["s1 tie even k=0+"])["s1"] == 1.0
    assert orc.stats(by["s1 tie odd k=0+"])["s1"] == 1.0 + 2.0 ** -51
    assert orc.stats(by["s1 above tie k=0+"])["s1"] == 1.0 + 2.0 ** -52
    assert orc.stats(by["s1 tie odd k=16-"])["s1"] == -(2.0 ** 16) * (1.0 + 2.0 ** -51)
    assert orc.stats(by["s2 tie even k=0"])["s2"] == 1.0
    assert orc.stats(by["s2 tie odd k=0"])["s2"] == 1.0 + 2.0 ** -51
    assert orc.stats(by["s2 above tie k=0"])["s2"] == 1.0 + 2.0 ** -52


def _norm_weights(n, seed):
    """LayerNorm-like weights: 1.0 + N(0, 0.01), rounded to BF16."""
    rng = np.random.default_rng(seed)
    v = (1.0 + rng.normal(0, 0.01, n)).astype(np.float32)
    b = v.view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_histogram_window_is_the_fewest_escapes(orc):
    """Window mode 1 takes the base with the fewest values outside its 7
    bins (brute force over every base on an independent histogram), ties to
    the lowest base, and leaves the moments as they are."""
    rng = np.random.default_rng(11)
    cases = [_norm_weights(5000, 1), rand_bf16(rng, 4000, "gauss"), rand_bf16(rng, 4000, "wide"),
             rand_bf16(rng, 3000, "bits"), rand_bf16(rng, 2000, "sub"),
             np.full(100, 0x3F80, np.uint16), np.zeros(0, np.uint16),
             np.concatenate([np.full(5, 10 << 7), np.full(5, 100 << 7)]).astype(np.uint16)]
    for x in cases:
        h = np.bincount((x.astype(np.uint32) >> 7) & 0xFF, minlength=256)
        esc = [x.size - int(h[b:b + 7].sum()) for b in range(250)]
        best = int(np.argmin(esc))              # first minimum: the lowest base
        s0, s1 = orc.stats(x, 0), orc.stats(x, 1)
        assert s1["E0"] == best and s1["n_escape"] == esc[best] and s1["rule"] == 1
        assert s1["n_escape"] <= s0["n_escape"]
        for k in ("s1", "s2", "var", "sigma", "n_finite"):
            assert s1[k] == s0[k] or (math.isnan(s1[k]) and math.isnan(s0[k])), k


def test_sigma_window_misses_norm_weights(orc):
    """The sigma-only window's weak case: weights near 1.0 with a small
    spread put the window ~12 binades below 1.0, so every value escapes; the
    histogram window codes all of them."""
    x = _norm_weights(20000, 2)
    s0, s1 = orc.stats(x, 0), orc.stats(x, 1)
    assert s0["rule"] == 0 and s0["n_escape"] == x.size
    assert s1["n_escape"] == 0 and s1["E0"] <= 126 <= s1["E0"] + 6


def test_clamp(orc):
    assert orc.window_from_var(1e-300) == 0
    assert orc.window_from_var(1e300) == 249


def test_fallbacks(orc):
    # all-equal tensor: var == 0 exactly -> histogram fallback
    x = np.full(1000, 0x3F80, np.uint16)           # 1.0, E = 127
    st = orc.stats(x)
    assert st["var"] == 0.0 and st["rule"] == 1
    assert st["E0"] == 121 and st["n_escape"] == 0  # smallest base covering 127
    # fewer than two finite values
    x = np.array([0x7F80, 0xFF80, 0x4000], np.uint16)  # +inf, -inf, 2.0
    st = orc.stats(x)
    assert st["n_finite"] == 1 and st["rule"] == 1
    assert st["hist"][255] == 2
    # the densest 7-bin run wins, ties to the smallest base
    x = np.concatenate([np.full(5, 10 << 7), np.full(5, 100 << 7)]).astype(np.uint16)
    x = np.concatenate([x, np.full(1, 0x7FC0, np.uint16)])   # one NaN, N finite = 10
    st = orc.stats(x)
    assert st["rule"] == 0    # var > 0 here: the sigma rule applies
    st = orc.stats(np.array([10 << 7], np.uint16))
    assert st["rule"] == 1 and st["E0"] == 4


def test_nonfinite_values_stay_out_of_sigma(orc):
    rng = np.random.default_rng(3)
    x = rand_bf16(rng, 500, "gauss")
    y = np.concatenate([x, np.array([0x7F80, 0xFFC1, 0x7FFF], np.uint16)])
    a, b = orc.stats(x), orc.stats(y)
    assert (a["s1"], a["s2"], a["var"], a["E0"]) == (b["s1"], b["s2"], b["var"], b["E0"])
    assert b["hist"][255] == 3 and b["n_finite"] == 500


def test_config2_like_expectations(orc):
    """Gaussian N(0, 0.02): E0 = 116 and ~2.1% escapes; ratio ~1.43
    (digest 3.1: 11 + 8*escape bits per value, 16/11.2 ~ 1.43x)."""
    import synth
    n = 1 << 22
    x = synth.gaussian_bf16(n, 0.02, synth.key_of(12, 0)).numpy().view(np.uint16)
    st = orc.stats(x)
    assert st["E0"] == 116
    esc = st["n_escape"] / n
    # escape share from the erf model with BF16 rounding edges: a value lands
    # in binade x when |v| in [2^x (1 - 2^-9), 2^(x+1) (1 - 2^-9))
    s = 0.02
    e = 1 - 2.0 ** -9
    lo = 2.0 ** (116 - 127) * e
    hi = 2.0 ** (116 - 127 + 7) * e
    p_in = math.erf(hi / (s * math.sqrt(2))) - math.erf(lo / (s * math.sqrt(2)))
    p = 1 - p_in
    assert abs(esc - p) < 5 * math.sqrt(p * (1 - p) / n)
    bits = 11 + 8 * esc
    assert 16 / bits == pytest.approx(1.43, abs=0.01)
