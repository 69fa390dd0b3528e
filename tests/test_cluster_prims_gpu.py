"""GPU unit tests of the DSMEM collectives (ClusterReduce all-reduce and
reduce-scatter forms, ClusterGather) through the test exports of libcf.so.

Inputs are small integers stored as floats, so every sum is exact and the
results are compared bit for bit with host-computed values.
"""
import pytest
import torch

from attention_block_gb300 import binding

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 4, 8, 16]


@pytest.fixture(scope="module", autouse=True)
def _need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    binding.lib()


def _ints(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-1000, 1000, shape, generator=g).float().cuda()


@pytest.mark.parametrize("N", SIZES)
@pytest.mark.parametrize("n", [4, 132, 1024])
def test_allreduce_sum_and_max(N, n):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = _ints((N, n), N * 1000 + n)
    for op, ref in ((0, x.sum(0)), (1, x.max(0).values)):
        out = torch.full_like(x, float("nan"))
        assert binding.cf_test_cluster_allreduce(N, op, n, x, out, err) == binding.CF_OK
        torch.cuda.synchronize()
        for r in range(N):
            assert torch.equal(out[r], ref), (N, n, op, r)
    assert int(err.item()) == 0


@pytest.mark.parametrize("N", [2, 4, 8])
def test_allreduce_with_threads_that_push_nothing_repeated(N):
    """n = 512 floats: only half of the threads push a chunk, all of them
    combine, so the combine must wait until every chunk has been read for the
    push.  Many launches back to back vary the timing."""
    n, reps = 512, 200
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = _ints((N, n), 7 * N)
    ref = x.sum(0)
    outs = [torch.full_like(x, float("nan")) for _ in range(reps)]
    for out in outs:
        assert binding.cf_test_cluster_allreduce(N, 0, n, x, out, err) == binding.CF_OK
    torch.cuda.synchronize()
    for i, out in enumerate(outs):
        for r in range(N):
            assert torch.equal(out[r], ref), (N, i, r)
    assert int(err.item()) == 0


def test_allreduce_max_with_ties_and_negative_infinity():
    N, n = 8, 8
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.full((N, n), float("-inf"), device="cuda")
    x[3, :4] = 5.0
    x[6, :4] = 5.0
    out = torch.empty_like(x)
    assert binding.cf_test_cluster_allreduce(N, 1, n, x, out, err) == binding.CF_OK
    torch.cuda.synchronize()
    ref = x.max(0).values
    for r in range(N):
        assert torch.equal(out[r], ref)


@pytest.mark.parametrize("N", SIZES)
@pytest.mark.parametrize("n", [4, 96])
def test_reduce_scatter(N, n):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = _ints((N, N * n), 7 * N + n)
    out = torch.full((N, n), float("nan"), device="cuda")
    assert binding.cf_test_cluster_reduce_scatter(N, n, x, out, err) == binding.CF_OK
    torch.cuda.synchronize()
    total = x.sum(0).view(N, n)
    assert torch.equal(out, total)
    assert int(err.item()) == 0


@pytest.mark.parametrize("N", SIZES)
@pytest.mark.parametrize("n", [4, 48, 400])
def test_gather(N, n):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = _ints((N, n), 11 * N + n)
    out = torch.full((N, N * n), float("nan"), device="cuda")
    assert binding.cf_test_cluster_gather(N, n, x, out, err) == binding.CF_OK
    torch.cuda.synchronize()
    for r in range(N):
        assert torch.equal(out[r], x.reshape(-1))
    assert int(err.item()) == 0


def test_bad_arguments_rejected_without_launch():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.zeros(64, device="cuda")
    assert binding.cf_test_cluster_allreduce(3, 0, 4, x, x, err) == binding.CF_ERR_INVALID_ARG
    assert binding.cf_test_cluster_allreduce(2, 0, 6, x, x, err) == binding.CF_ERR_INVALID_ARG
    assert binding.cf_test_cluster_gather(2, 4, None, x, err) == binding.CF_ERR_INVALID_ARG


# SM cycles after which the lost-transfer test's wait gives up (~50 us at
# 2 GHz; the decode kernels wait about one second).
SHORT_LIMIT = 100_000
TIMEOUT_BIT = 2  # the device bit the host reports as CF_ERR_DEVICE_TIMEOUT


@pytest.mark.parametrize("drop", [1, 0])
def test_lost_transfer_times_out_reports_and_leaves_the_context_usable(drop):
    """A block whose partner never sends: the bounded wait gives up after the
    short limit, the launch finishes by itself with the timeout bit set, the
    partner's side of the exchange is intact, and ordinary launches work
    afterwards (no fault, trap or hang is involved)."""
    n = 256
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = _ints((2, n), 99 + drop)
    out = torch.full_like(x, float("nan"))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    assert binding.cf_test_lost_transfer(n, drop, SHORT_LIMIT, x, out, err) == binding.CF_OK
    t1.record()
    torch.cuda.synchronize()
    assert int(err.item()) & TIMEOUT_BIT
    keep = 1 - drop  # did not receive: its row is its own input
    assert torch.equal(out[keep], x[keep])
    assert torch.equal(out[drop], x.sum(0))  # received its partner's row
    assert t0.elapsed_time(t1) < 1000.0  # ms: ended by the short limit, not the default
    # the same exchange with nothing dropped, then a plain collective
    err.zero_()
    out.fill_(float("nan"))
    assert binding.cf_test_lost_transfer(n, -1, SHORT_LIMIT, x, out, err) == binding.CF_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out[0], x.sum(0)) and torch.equal(out[1], x.sum(0))
    y = _ints((4, 64), 5)
    out4 = torch.empty_like(y)
    assert binding.cf_test_cluster_allreduce(4, 0, 64, y, out4, err) == binding.CF_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for r in range(4):
        assert torch.equal(out4[r], y.sum(0))


def test_lost_transfer_bad_arguments_rejected_without_launch():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.zeros(2, 64, device="cuda")
    f = binding.cf_test_lost_transfer
    assert f(6, 1, SHORT_LIMIT, x, x, err) == binding.CF_ERR_INVALID_ARG
    assert f(64, 2, SHORT_LIMIT, x, x, err) == binding.CF_ERR_INVALID_ARG
    assert f(64, 1, 0, x, x, err) == binding.CF_ERR_INVALID_ARG
    assert f(64, 1, SHORT_LIMIT, x, x, None) == binding.CF_ERR_INVALID_ARG
