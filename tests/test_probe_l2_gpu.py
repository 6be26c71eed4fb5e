"""The L2 streaming probe (bevpool_probe_l2) reads every byte of its buffer
exactly `passes` times, writes the documented pattern and copies the
documented values, on ragged sizes (not a multiple of the grid's stride) and
on a size of the order bench.py times."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

SALT = 0x9E3779B9


@pytest.fixture(scope="module")
def bp():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from depth_weighted_scatter_gb300 import bevpool

    return bevpool


@pytest.mark.parametrize("n_vec,passes", [(1, 1), (257, 2), (100_003, 3), (3 * 1024 * 1024, 2)])
def test_read_probe_reads_every_word_passes_times(bp, n_vec, passes):
    import torch

    rng = np.random.default_rng(n_vec)
    words = rng.integers(0, 2**32, size=4 * n_vec, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    bp.probe_l2(buf, passes, sink=sink)
    got = int(sink.cpu().numpy().view(np.uint32)[0])
    want = (passes * int(words.astype(np.uint64).sum())) % 2**32
    assert got == want


@pytest.mark.parametrize("n_vec,passes", [(1, 1), (257, 3), (100_003, 2), (3 * 1024 * 1024, 2)])
def test_write_probe_leaves_the_last_pass_pattern(bp, n_vec, passes):
    import torch

    buf = torch.zeros(4 * n_vec, dtype=torch.int32, device="cuda")
    bp.probe_l2(buf, passes, mode=bp.PROBE_WRITE)
    got = buf.cpu().numpy().view(np.uint32)
    salt = ((passes - 1) * SALT) % 2**32
    want = (np.arange(4 * n_vec, dtype=np.uint64) % 2**32).astype(np.uint32) ^ np.uint32(salt)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n_vec,passes", [(1, 1), (257, 3), (100_003, 2), (3 * 1024 * 1024, 2)])
def test_copy_probe_copies_the_first_half(bp, n_vec, passes):
    import torch

    rng = np.random.default_rng(7 + n_vec)
    src = rng.integers(0, 2**32, size=4 * n_vec, dtype=np.uint64).astype(np.uint32)
    host = np.concatenate([src, np.zeros_like(src)])
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    bp.probe_l2(buf, passes, mode=bp.PROBE_COPY)
    got = buf.cpu().numpy().view(np.uint32)
    salt = np.uint32(((passes - 1) * SALT) % 2**32)
    assert np.array_equal(got[:4 * n_vec], src)
    assert np.array_equal(got[4 * n_vec:], src ^ salt)


def test_probe_counts_one_launch(bp):
    import torch

    buf = torch.zeros(4096, dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = bp.bevpool_kernel_launches()
    bp.probe_l2(buf, 1, sink=sink)
    torch.cuda.synchronize()
    assert bp.bevpool_kernel_launches() == before + 1


@pytest.mark.parametrize("row_bytes,n_rows,n_points,ctas", [(16, 5, 1, 1), (160, 16_896, 7, 3), (160, 16_896, 100_003, 3),
                                                            (256, 1_000, 20_000, 8), (512, 333, 4_097, 2),
                                                            (96, 50, 0, 3)])
def test_gather_probe_reads_every_listed_row(bp, row_bytes, n_rows, n_points, ctas):
    """The gather probe adds the word sum of every listed row (once per listing,
    rows out of range skipped) to the sink."""
    import torch

    rng = np.random.default_rng(row_bytes * 7 + n_points)
    words = rng.integers(0, 2**32, size=n_rows * row_bytes // 4, dtype=np.uint64).astype(np.uint32)
    rows = rng.integers(-2, n_rows + 2, size=max(n_points, 1)).astype(np.int32)[:n_points]
    feat = torch.from_numpy(words.view(np.int32)).cuda()
    rows_d = torch.from_numpy(rows).cuda() if n_points else torch.zeros(1, dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = bp.bevpool_probe_gather(feat.data_ptr(), n_rows, row_bytes, rows_d.data_ptr(), n_points, ctas,
                                 sink.data_ptr(), 0)
    assert st == bp.BEVPOOL_OK
    got = int(sink.cpu().numpy().view(np.uint32)[0])
    row_sums = words.reshape(n_rows, row_bytes // 4).astype(np.uint64).sum(axis=1)
    valid = rows[(rows >= 0) & (rows < n_rows)]
    assert got == int(row_sums[valid].sum()) % 2**32


def test_gather_probe_rejects_bad_arguments(bp):
    import torch

    feat = torch.zeros(1024, dtype=torch.int32, device="cuda")
    rows = torch.zeros(4, dtype=torch.int32, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    ok = lambda **kw: bp.bevpool_probe_gather(*[kw.get(k, v) for k, v in dict(
        feat=feat.data_ptr(), n_rows=16, row_bytes=256, rows=rows.data_ptr(), n=4, ctas=3, sink=sink.data_ptr(),
        stream=0).items()])
    assert ok() == bp.BEVPOOL_OK
    assert ok(row_bytes=24) == bp.BEVPOOL_ERR_INVALID_ARG
    assert ok(row_bytes=528) == bp.BEVPOOL_ERR_INVALID_ARG
    assert ok(ctas=9) == bp.BEVPOOL_ERR_INVALID_ARG
    assert ok(sink=0) == bp.BEVPOOL_OK                    # the timing mode
    assert ok(feat=feat.data_ptr() + 4) == bp.BEVPOOL_ERR_INVALID_ARG
