"""pa_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (a plug-in whose host program owns every device allocation, or
a loop where cudaMalloc is not allowed).  It takes its split-KV workspace from
a fixed array inside the library instead of a caller buffer.

Called through the C ABI; its output must match pa_decode with a caller
workspace, within the bf16 tolerance of the other tests, on two calls in a
row (the second call reuses the array the first one left behind), and both
must match the fp64 oracle.  This file
is collected last so a failure here cannot hide the others; it also passes
when run alone in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from gpu_util import TOL, compare, device_inputs, oracle_decode_all
from paged_kv_cache_192_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_192_gb300 import build
    build.build()
    from paged_kv_cache_192_gb300 import _lib
    return _lib.lib()


def _decode_noalloc(L, w, out, q, k_cache, v_cache, table, lens, partition):
    from paged_kv_cache_192_gb300._lib import PA_BF16
    return L.pa_decode_noalloc(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(),
                               v_cache.data_ptr(), table.data_ptr(), table.shape[1],
                               lens.data_ptr(), w.B, w.Hq, w.Hkv, w.d, w.bs, w.num_blocks,
                               1.0 / math.sqrt(w.d), partition, PA_BF16,
                               torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_decode_twice(lib):
    from paged_kv_cache_192_gb300 import ops
    # two batches that both split into several partitions (the scratch is used)
    batches = [synth.decode_workload("8b", seed=21, B=24),
               synth.decode_workload("8b", seed=22, B=40)]
    atol, rtol = TOL[torch.bfloat16]
    for w in batches:
        k_cache, v_cache, table, lens = device_inputs(w, DEV)
        q = w.q.to(DEV)
        ref = ops.decode(q, k_cache, v_cache, table, lens, partition_tokens=256)
        out = torch.full_like(q, float("nan"))
        rc = _decode_noalloc(lib, w, out, q, k_cache, v_cache, table, lens, 256)
        assert rc == 0, lib.pa_last_error_string()
        torch.cuda.synchronize()
        got, exp = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.isfinite(got).all()
        assert np.all(np.abs(got - exp) <= atol + rtol * np.abs(exp))
        oracle_out = oracle_decode_all(w)
        compare(got, oracle_out, torch.bfloat16, "noalloc vs oracle")
        compare(exp, oracle_out, torch.bfloat16, "decode vs oracle")


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    cap = lib.pa_decode_noalloc_capacity()
    assert cap == 16 << 20
    need = ctypes.c_size_t()
    # 70B-shaped long-context batch: 32 x 64 heads x 64 partitions of 512
    assert lib.pa_decode_workspace_size(32, 64, 128, 1024, 32, 512, ctypes.byref(need)) == 0
    assert need.value > cap
    x = torch.zeros(16, device=DEV)
    rc = lib.pa_decode_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                               x.data_ptr(), 1024, x.data_ptr(), 32, 64, 8, 128, 32, 1000, 0.08,
                               512, 0, None)
    assert rc == 1 and b"scratch" in lib.pa_last_error_string()


def test_noalloc_through_the_python_binding(lib):
    """ops.decode_noalloc (same call through the binding) matches ops.decode
    bit for bit: both run the same kernel on the same inputs, only the
    workspace differs."""
    from paged_kv_cache_192_gb300 import ops
    assert ops.decode_noalloc_capacity() == 16 << 20
    w = synth.decode_workload("8b", seed=23, B=16)
    k_cache, v_cache, table, lens = device_inputs(w, DEV)
    q = w.q.to(DEV)
    ref = ops.decode(q, k_cache, v_cache, table, lens, partition_tokens=256)
    out = ops.decode_noalloc(q, k_cache, v_cache, table, lens, partition_tokens=256)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    assert torch.equal(out, ref)
