"""The bench's end-to-end step: pinned host inputs copied in and O and LSE
copied out, with two device buffer sets alternating between steps on two copy
streams.  Its host results must be the bytes of the same step run on
device-resident inputs, and it must declare the bytes it copies."""
import pytest
import torch

from gpu_util import fi

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", ["ragged_small", "uniform_small", "decode_small"])
def test_double_buffered_e2e_matches_the_device_step(name):
    import bench
    runner = bench.PathRunner(fi(), name, torch.device("cuda"))
    stream = torch.cuda.Stream()
    runner.step(stream)
    torch.cuda.synchronize()
    ref_out, ref_lse = runner.out.cpu(), runner.lse.cpu()
    inputs = (runner.k, runner.v, runner.q, runner.slots, runner.page_table)
    own = inputs + (runner.out, runner.lse)
    # warm-up step + 3 timed steps: both buffer sets are used twice
    _, h2d, d2h, (ho, hl) = bench.time_e2e(runner, stream, 3, 1)
    assert torch.equal(ho, ref_out)
    assert torch.equal(hl, ref_lse)
    assert h2d == sum(t.numel() * t.element_size() for t in inputs)
    assert d2h == ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    # the runner is left on its own buffers
    assert all(a is b for a, b in zip(own, (runner.k, runner.v, runner.q, runner.slots,
                                            runner.page_table, runner.out, runner.lse)))
    assert runner.status() == 0
    runner.close()
