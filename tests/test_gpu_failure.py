"""Device-side failure path without a GPU fault: a bounded wait that runs out
records PA_DEVERR_TIMEOUT, the host reads it, and the context stays usable
for the next (correct) launch."""
import pytest
import torch

from gpu_util import compare, device_inputs, oracle_decode
from paged_kv_cache_192_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_192_gb300 import build
    build.build()


def test_wait_that_runs_out_is_reported_and_context_survives():
    from paged_kv_cache_192_gb300 import _lib, ops
    assert ops.device_error() == 0
    ops.check_wait_timeout()
    torch.cuda.synchronize()  # completes: the wait is bounded
    assert ops.device_error(clear=True) == _lib.PA_DEVERR_TIMEOUT
    assert ops.device_error() == 0  # cleared
    # the context is still good: a decode right after matches the oracle
    w = synth.decode_workload("8b", seed=21, lens=[1, 100, 700])
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    out = ops.decode(w.q.to(DEV), k_cache, v_cache, table, lens)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    compare(out.double().cpu().numpy(), oracle_decode(w), torch.bfloat16, "after timeout")
