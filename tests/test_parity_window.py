"""The GPU parity checks can see one lost or doubled scatter point.

The stated tolerance for fp16 inputs (1e-2 * max|ref| + 1e-3) is global: on
the canonical workload it is several times one point's contribution, so a
kernel that dropped or doubled a point at an owner-share boundary would pass
it.  The per-element FP32 window of tests/gpu_common.py must not.  These CPU
tests build the output a correct kernel gives (the oracle's FP64 value
rounded once to fp16) and outputs with one planted mistake, and check that
the window accepts the first and rejects the others while the global
tolerance accepts all three."""
import numpy as np
import pytest

from gpu_common import (assert_forward_close, half_ulp_fp16, longest_interval, oracle_values, tolerance,
                        window_violations)


def _point_contribution(wl, p):
    """depth[p] * feat[row(p), :] in FP64 for frustum point p (fp16 workloads)."""
    hw = wl.H * wl.W
    nc, rem = divmod(p, wl.D * hw)
    row = nc * hw + rem % hw
    d = float(wl.depth.reshape(-1)[p])
    return d * wl.feat.reshape(wl.n_feat_rows, wl.C)[row].astype(np.float64)


@pytest.fixture(scope="module")
def case(wl_cache):
    wl = wl_cache("canonical")
    ref = oracle_values(wl)
    s_abs = oracle_values(wl, absolute=True)
    kept = np.flatnonzero(wl.cell_ids >= 0)
    size = np.array([np.abs(_point_contribution(wl, p)).max() for p in kept[::50]])
    # a typical point: the median contribution size of a sample of kept points
    p = int(kept[::50][np.argsort(size)[len(size) // 2]])
    return wl, ref, s_abs, p


def _rounded(x):
    return x.astype(np.float16).astype(np.float64)


def test_correct_output_passes_both(case):
    wl, ref, s_abs, _ = case
    got = _rounded(ref)
    assert not window_violations(got, ref, s_abs, longest_interval(wl.cell_ids)).any()
    assert_forward_close(wl, got, ref)


@pytest.mark.parametrize("mistake", ["dropped", "doubled"])
def test_one_planted_point_fails_the_window_only(case, mistake):
    wl, ref, s_abs, p = case
    cell = int(wl.cell_ids[p])
    v = _point_contribution(wl, p)
    bad = ref.copy()
    bad[cell] += -v if mistake == "dropped" else v
    got = _rounded(bad)
    err = np.abs(got - ref).max()
    assert err <= tolerance(wl, ref), "the planted point should hide under the global tolerance"
    viol = window_violations(got, ref, s_abs, longest_interval(wl.cell_ids))
    assert viol.any(), f"window missed a {mistake} point of size {np.abs(v).max():.3g}"
    assert set(np.argwhere(viol)[:, 0]) == {cell}
    with pytest.raises(AssertionError, match="FP32 window"):
        assert_forward_close(wl, got, ref)


def test_half_ulp_matches_fp16_rounding():
    """Rounding any value to fp16 moves it by at most the half spacing used."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 1, 10000) * 10.0 ** rng.integers(-8, 4, 10000), [0.0, 2.0 ** -24, 65504.0]])
    r = x.astype(np.float16).astype(np.float64)
    assert np.all(np.abs(r - x) <= half_ulp_fp16(r, x))
