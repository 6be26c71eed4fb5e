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
