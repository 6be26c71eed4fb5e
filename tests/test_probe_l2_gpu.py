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
