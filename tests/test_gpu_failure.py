"""Failure handling on the GPU without a fault: a bounded in-kernel wait that
runs out reports PA_FLAG_TIMEOUT and the kernel returns.

The library's kernels wait on mbarriers only through one bounded wait; the
self-check kernel waits, with a short limit, on a barrier nothing completes
(one thread's wait, and a whole warp's wait decided by vote) with no copy in
flight, and on a barrier that has completed.  The context stays usable: the
next work on the stream runs normally.
"""
import pytest
import torch

import paged_kv_cache_240_gb300 as pa
from gpu_util import new_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit", [200_000, 2_000_000])
def test_bounded_wait_gives_up_and_reports(limit):
    result = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    err = new_err()
    pa.pa_selftest_bounded_wait(limit, result, err)
    torch.cuda.synchronize()
    r = result.cpu().tolist()
    assert r[0] == 1 and r[1] == 1          # both waits on the silent barrier gave up
    assert r[2] == 1                        # the completed barrier's wait returned
    assert r[3] >= limit                    # not before its limit
    assert int(err[0]) == pa.PA_FLAG_TIMEOUT
    # the context is intact: ordinary work on the same stream still runs
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2


def test_bounded_wait_rejects_bad_limits():
    result = torch.zeros(4, dtype=torch.int64, device="cuda")
    for bad in (0, -5, 5_000_000_000):
        with pytest.raises(pa.PaError) as e:
            pa.pa_selftest_bounded_wait(bad, result, new_err())
        assert e.value.status == pa.PA_ERR_INVALID_ARG
