"""GPU parity on the shapes of the pages' Table 1 (small / large / very large
at C = 80, wide C = 128 and 256; FP16 and E4M3 inputs), at full size: the
scatter map bit-exact, the forward within the fp16 / E4M3 tolerances."""
import numpy as np
import pytest

from gpu_common import MAP_KEYS, assert_forward_close, gpu_forward, oracle_forward, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from depth_weighted_scatter_gb300 import workloads  # noqa: E402

NAMES = list(workloads.TABLE1) + [n + "_fp8" for n in workloads.TABLE1]


@pytest.fixture(scope="module")
def bp():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


@pytest.mark.parametrize("name", NAMES)
def test_table1_shape_parity(bp, name, wl_cache):
    import oracle

    wl = wl_cache(name)
    cells, depth, feat = upload(wl)
    m = bp.build_map(cells, *wl.dims(), wl.n_cells)
    ref_map = oracle.build_map(wl.cell_ids, *wl.dims(), wl.n_cells)
    got = m.host()
    for k in MAP_KEYS:
        assert np.array_equal(got[k], ref_map[k]), f"{name}: {k} differs"
    out = torch.full((wl.n_cells, wl.C), float("nan"), dtype=torch.float16, device="cuda")
    gpu_forward(wl, m, depth, feat, out=out)
    torch.cuda.synchronize()
    assert_forward_close(wl, out, oracle_forward(wl))
