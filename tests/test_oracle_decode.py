"""Pins for the oracle's number decoders against library decoders.

binary16 against numpy's float16, OCP E4M3 against torch's float8_e4m3fn,
over every code, so a wrong bias, a wrong subnormal rule or a wrong NaN
rule fails here."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_half_every_code_matches_numpy():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.half_to_double(codes)
    want = codes.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zero and infinities keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_half_landmarks():
    # smallest subnormal, largest subnormal, smallest normal, one, max finite
    assert oracle.half_to_double(np.array([0x0001], np.uint16))[0] == 2.0 ** -24
    assert oracle.half_to_double(np.array([0x03FF], np.uint16))[0] == 1023 * 2.0 ** -24
    assert oracle.half_to_double(np.array([0x0400], np.uint16))[0] == 2.0 ** -14
    assert oracle.half_to_double(np.array([0x3C00], np.uint16))[0] == 1.0
    assert oracle.half_to_double(np.array([0x7BFF], np.uint16))[0] == 65504.0
    assert oracle.half_to_double(np.array([0xC000], np.uint16))[0] == -2.0


def test_e4m3_every_code_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = oracle.e4m3_to_double(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert nan.sum() == 2  # S.1111.111 for both signs
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_e4m3_landmarks():
    dec = lambda b: oracle.e4m3_to_double(np.array([b], np.uint8))[0]
    assert dec(0x01) == 2.0 ** -9          # smallest subnormal
    assert dec(0x08) == 2.0 ** -6          # smallest normal
    assert dec(0x38) == 1.0
    assert dec(0x7E) == 448.0              # largest finite
    assert dec(0xFE) == -448.0
    assert np.isnan(dec(0x7F))


# ---------------------------------------------------------------- E4M3 encoding (FP8 output)

def _finite_codes():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    vals = oracle.e4m3_to_double(codes)
    keep = ~np.isnan(vals)
    return codes[keep], vals[keep]


def test_e4m3_encode_round_trips_every_finite_code():
    codes, vals = _finite_codes()
    got = oracle.e4m3_from_double(vals)
    # +0 and -0 both decode to 0; every other code must come back unchanged
    same = (got == codes) | ((vals == 0) & ((got & 0x7F) == 0))
    assert same.all()


def _nearest_code_violations(x, got):
    """Entries of got (E4M3 codes for the doubles x) that are not the nearest
    finite code, ties to the even mantissa, saturated at 448, sign kept."""
    codes, vals = _finite_codes()
    pos = np.unique(vals[vals >= 0])                     # 0 .. 448, ascending
    a = np.minimum(np.abs(x), 448.0)
    dist = np.abs(pos[None, :] - a[:, None])
    best = dist.min(axis=1)
    even = {v: (int(c) & 1) == 0 for c, v in zip(codes, vals) if v >= 0 and (int(c) & 0x80) == 0}
    want_mag = np.empty(a.size)
    for i in range(a.size):
        cand = pos[np.nonzero(dist[i] == best[i])[0]]
        want_mag[i] = cand[0] if cand.size == 1 else [v for v in cand if even[v]][0]
    got_val = oracle.e4m3_to_double(got)
    bad = np.abs(got_val) != want_mag
    nz = want_mag != 0
    bad[nz] |= np.signbit(got_val[nz]) != np.signbit(x[nz])
    return np.nonzero(bad)[0]


def _encode_probe_values():
    codes, vals = _finite_codes()
    pos = np.unique(vals[vals >= 0])
    rng = np.random.default_rng(5)
    x = np.concatenate([
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(600.0), 4000)),
        (pos[1:] + pos[:-1]) / 2,                        # exact midpoints (ties)
        pos,                                             # representable values
        [500.0, 456.0, 464.0, 1e6],                      # beyond the largest finite value
    ])
    return np.concatenate([x, -x])


def test_e4m3_encode_is_nearest_code_ties_to_even():
    """Brute force over the 254 finite codes."""
    x = _encode_probe_values()
    assert _nearest_code_violations(x, oracle.e4m3_from_double(x)).size == 0


def test_e4m3_encode_matches_library_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-8, 5, 20000))
    x = x[np.abs(x) <= 448.0]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = oracle.e4m3_from_double(x)
    assert np.array_equal(oracle.e4m3_to_double(lib), oracle.e4m3_to_double(ours))


def test_e4m3_encode_pin_catches_planted_mistakes():
    """Mistakes planted in the oracle's codes (on the CPU) must fail the pin:
    rounding toward zero, a wrong tie rule, a lost sign, no saturation."""
    x = _encode_probe_values()
    good = oracle.e4m3_from_double(x)
    vals = oracle.e4m3_to_double(good)
    mag = np.abs(vals)
    up = mag > np.abs(x)                                 # rounded away from zero
    toward_zero = good.copy()
    toward_zero[up & (mag > 0)] -= 1                     # the code just below in magnitude
    ties = good.copy()
    codes, fin = _finite_codes()
    pos = np.unique(fin[fin >= 0])
    mids = np.isin(np.abs(x), (pos[1:] + pos[:-1]) / 2)
    ties[mids & up] -= 1                                 # ties to the lower code instead of even
    sign = good ^ 0x80
    nosat = good.copy()
    nosat[np.abs(x) > 448.0] = 0x00                      # overflow to zero
    for planted in (toward_zero, ties, sign, nosat):
        assert _nearest_code_violations(x, planted).size > 0
