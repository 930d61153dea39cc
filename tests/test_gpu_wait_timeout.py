"""Failure detection without a GPU fault: a bounded pipeline wait is made to run
out on purpose, on an mbarrier that nothing arrives at, with the library's own
wait code (mbar_wait with the CTA's abort state).  The kernel must return with
FI_DEV_WAIT_TIMEOUT in the status word, the other waiting warps must give up
through the abort flag long before their own limit, the copy that was in
flight must be drained, and the context must then run the regular path
correctly (append bytes bit-exact, attention within the tolerances)."""
import numpy as np
import pytest
import torch

from gpu_util import (assert_within_tolerance, cache_to_host, compare_attention, device_inputs,
                      fi, oracle_attention, oracle_cache, run_path)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def diag():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_paged_kv_slot_b300.diag as d
    return d


@pytest.mark.parametrize("timeout_ms", [1, 5])
def test_bounded_wait_runs_out_and_the_context_stays_usable(diag, timeout_ms):
    m = fi()
    src = torch.randint(0, 256, (4096,), dtype=torch.uint8, device="cuda")
    copy_out = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    report = torch.zeros(4, dtype=torch.int64, device="cuda")
    diag.wait_timeout(timeout_ms * 1_000_000, src, copy_out, status, report)
    torch.cuda.synchronize()
    rep = report.cpu().tolist()
    assert int(status.item()) == m.FI_DEV_WAIT_TIMEOUT
    # warp 0 waited its own limit (and not much longer: it checks the clock
    # after every poll); warp 1 gave up through the abort flag, well before
    # its own 2 s limit
    assert timeout_ms * 1e6 <= rep[0] < timeout_ms * 1e6 + 50e6, rep
    assert rep[1] < 100e6, rep
    assert rep[2] == 66, rep          # 1 + 1 + 64 waits gave up
    assert rep[3] == 1, rep           # the copy in flight was drained
    assert torch.equal(copy_out, src)

    # the context is usable afterwards: the regular path, against the oracle
    d = device_inputs("ragged_small")
    out, lse, cache, st, _ = run_path(d)
    assert st == 0
    host = oracle_cache(d)
    g = cache_to_host(cache)
    for name in ("k_data", "v_data", "k_sf", "v_sf"):
        assert np.array_equal(g[name], host[name]), name
    ref_out, ref_lse = oracle_attention(d, host)
    assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))
