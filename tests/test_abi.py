"""The C ABI library builds, loads without a GPU, exports every symbol
include/pa.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_192_gb300 import build
    build.build()
    from paged_kv_cache_192_gb300 import _lib
    return _lib.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_hot_path_calls():
    names = declared_functions()
    for n in ("pa_reshape_and_cache", "pa_decode", "pa_prefill_chunk", "pa_copy_blocks",
              "pa_decode_workspace_size", "pa_bm_create", "pa_bm_append", "pa_bm_fork"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from paged_kv_cache_192_gb300._lib import SIGNATURES
    names = declared_functions()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in pa.h but not exported"
    assert set(names) == set(SIGNATURES), "binding signatures must mirror pa.h"


def test_version(lib):
    assert lib.pa_version() == 1


def _count_bytes(rows):
    return -(-rows * 4 // 256) * 256


def test_workspace_size_host_only(lib):
    from paged_kv_cache_192_gb300 import ops
    # 8B-shaped: 64 seqs, 32 heads, d 128, 256 blocks of 16 -> 8 partitions of
    # 512 + 1 segment slots per (sequence, head), after a 4-byte partial count per
    # (sequence, head) padded to a multiple of 256 bytes
    assert ops.decode_workspace_size(64, 32, 128, 256, 16, 512) == (
        _count_bytes(64 * 32) + 64 * 32 * 9 * 130 * 4)
    assert ops.decode_workspace_size(4, 4, 64, 4, 16, 0) == _count_bytes(16) + 16 * 2 * 66 * 4
    assert ops.decode_workspace_size(0, 4, 64, 4, 16, 0) == 0
    # odd B x Hq: the fp32 partials still start 256 bytes into the buffer
    assert ops.decode_workspace_size(5, 3, 128, 8, 16, 64) == 256 + 15 * 3 * 130 * 4


def test_workspace_size_overflow_is_rejected(lib):
    """Sizes whose workspace does not fit in size_t are refused, not wrapped
    into a small number that a caller (or the fixed no-alloc scratch) would
    accept."""
    out = ctypes.c_size_t(0)
    big = 2 ** 31 - 1
    rc = lib.pa_decode_workspace_size(big, big, 128, 2 ** 26, 16, 32, ctypes.byref(out))
    assert rc == 1 and b"size_t" in lib.pa_last_error_string()
    # the largest table capacity (2^30 tokens) at the largest batch pa_decode
    # takes still fits
    assert lib.pa_decode_workspace_size(65535, 8, 128, 2 ** 26, 16, 32, ctypes.byref(out)) == 0
    assert out.value > 2 ** 40


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), 1),               # bad dtype
    (dict(head_dim=96), 4),           # unsupported head_dim
    (dict(Hq=12, Hkv=8), 1),          # Hq not a multiple of Hkv
    (dict(Hq=32, Hkv=2), 4),          # group of 16 unsupported
    (dict(block_size=24), 4),         # not a power of two
    (dict(partition_tokens=48), 1),   # not a multiple of 32
    (dict(scale=-1.0), 1),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    args = dict(out=None, q=None, k=None, v=None, bt=None, MB=4, lens=None, B=1, Hq=4, Hkv=4,
                head_dim=64, block_size=16, NB=8, scale=0.125, partition_tokens=0, ws=None,
                ws_bytes=0, dtype=1, stream=None)
    args.update(kw)
    rc = lib.pa_decode(args["out"], args["q"], args["k"], args["v"], args["bt"], args["MB"],
                       args["lens"], args["B"], args["Hq"], args["Hkv"], args["head_dim"],
                       args["block_size"], args["NB"], args["scale"], args["partition_tokens"],
                       args["ws"], args["ws_bytes"], args["dtype"], args["stream"])
    assert rc == code
    assert lib.pa_last_error_string()


@pytest.mark.parametrize("args", [
    (-1, 8, 256, 16, 0),    # negative batch
    (4, 0, 256, 16, 0),     # no KV heads
    (4, 8, 0, 16, 0),       # empty table
    (4, 8, 256, 24, 0),     # block size not a power of two
    (4, 8, 256, 16, 48),    # partition not a multiple of 32
])
def test_decode_kernel_for_rejects_bad_sizes(lib, args):
    k = ctypes.c_int(0)
    assert lib.pa_decode_kernel_for(*args, ctypes.byref(k)) == 1
    assert lib.pa_last_error_string()
    assert lib.pa_decode_kernel_for(4, 8, 256, 16, 0, None) == 1


def test_decode_kernel_for_needs_a_device(lib):
    """Valid sizes: the choice depends on the device's SM count, so without a
    CUDA device the call fails cleanly (PA_ERR_CUDA) instead of guessing."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    k = ctypes.c_int(-1)
    assert lib.pa_decode_kernel_for(64, 8, 256, 16, 0, ctypes.byref(k)) == 3
    assert k.value == -1 and lib.pa_last_error_string()


def test_null_pointers_rejected(lib):
    rc = lib.pa_decode(None, None, None, None, None, 4, None, 2, 4, 4, 64, 16, 8, 0.125, 0, None,
                       0, 1, None)
    assert rc == 1 and b"NULL" in lib.pa_last_error_string()
    rc = lib.pa_reshape_and_cache(None, None, None, None, None, 3, 8, 4, 16, 64, 0, None)
    assert rc == 1


def test_empty_calls_are_noops(lib):
    assert lib.pa_reshape_and_cache(None, None, None, None, None, 0, 8, 4, 16, 64, 0, None) == 0
    assert lib.pa_copy_blocks(None, None, None, 0, 8, 4, 16, 64, 0, None) == 0
    assert lib.pa_decode(None, None, None, None, None, 4, None, 0, 4, 4, 64, 16, 8, 0.125, 0,
                         None, 0, 1, None) == 0


def test_prefill_rejects_fp32(lib):
    rc = lib.pa_prefill_chunk(None, None, None, None, None, 4, None, None, 1, 8, 4, 4, 64, 16, 8,
                              0.125, 1, None)
    assert rc == 4


def test_misaligned_pool_rejected(lib):
    rc = lib.pa_reshape_and_cache(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(8),
                                  ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 8, 4, 16, 64, 0,
                                  None)
    assert rc == 1 and b"aligned" in lib.pa_last_error_string()


def test_decode_tile_for_host_only(lib):
    """The tensor-core tile serves bf16 groups of 4 and 8 heads; fp32, groups
    of 1 and 2, and pools too large for 32-bit tensor-copy coordinates use the
    CUDA-core tile (a host rule, no device needed)."""
    from paged_kv_cache_192_gb300 import ops
    assert ops.decode_tile_for(32, 8, 128, 16, 10358) == "tensor_core"   # 8B shape
    assert ops.decode_tile_for(64, 8, 128, 32, 30000) == "tensor_core"   # 70B shape
    assert ops.decode_tile_for(16, 2, 64, 8, 100) == "tensor_core"
    assert ops.decode_tile_for(32, 8, 128, 16, 10358, torch.float32) == "cuda_core"
    assert ops.decode_tile_for(8, 4, 128, 16, 100) == "cuda_core"
    assert ops.decode_tile_for(4, 4, 128, 16, 100) == "cuda_core"
    assert ops.decode_tile_for(32, 8, 128, 16, 2 ** 24) == "cuda_core"  # 2^31 pool rows
    out = ctypes.c_int(0)
    assert lib.pa_decode_tile_for(12, 8, 128, 16, 100, 0, ctypes.byref(out)) == 1
    assert lib.pa_decode_tile_for(32, 8, 96, 16, 100, 0, ctypes.byref(out)) == 1


def test_prefill_kernel_for_host_only(lib):
    """Prefill kernel choice from sizes alone (no device): the persistent grid
    for batches of at most 256 (request, 256-row) pairs and 512 work items,
    one CTA per item past that, the 128-thread kernel for 128-token blocks
    and block tables longer than 1024 entries."""
    from paged_kv_cache_192_gb300 import ops
    # mixed batch: 4 chunks of 512 tokens, 32/8 heads -> 32 pairs, 256 items
    assert ops.prefill_kernel_for(4, 512, 32, 8, 128, 16, 100000, 512) == "persistent"
    # 64 items per KV head at 8 KV heads: exactly 512 items
    assert ops.prefill_kernel_for(64, 64, 32, 8, 128, 16, 100000, 512) == "persistent"
    assert ops.prefill_kernel_for(65, 64, 32, 8, 128, 16, 100000, 512) == "item_grid"
    # 280 pairs of 2 KV heads (560 items): past both limits
    assert ops.prefill_kernel_for(70, 200, 8, 2, 128, 16, 100000, 64) == "item_grid"
    # groups of 8 heads: 32-token query tiles
    assert ops.prefill_kernel_for(2, 1024, 64, 8, 128, 16, 100000, 512) == "persistent"
    assert ops.prefill_kernel_for(4, 512, 32, 8, 128, 128, 100000, 64) == "simple"
    assert ops.prefill_kernel_for(2, 64, 8, 2, 128, 8, 100000, 1038) == "simple"
    out = ctypes.c_int(0)
    assert lib.pa_prefill_kernel_for(4, 512, 32, 8, 96, 16, 100000, 512, ctypes.byref(out)) == 4
    assert lib.pa_prefill_kernel_for(4, 512, 32, 8, 128, 24, 100000, 512, ctypes.byref(out)) == 4
    assert lib.pa_prefill_kernel_for(-1, 512, 32, 8, 128, 16, 100000, 512, ctypes.byref(out)) == 1
    assert lib.pa_prefill_kernel_for(4, 512, 32, 8, 128, 16, 100000, 512, None) == 1


def test_contiguous_and_shared_workspace_sizes_host_only(lib):
    """Workspace sizes of the contiguous control and of the shared-prefix
    decode: the paged size for the same capacity, plus one prefix slot per
    256 shared tokens for the latter; bad reservations are refused."""
    from paged_kv_cache_192_gb300 import ops
    assert ops.decode_contiguous_workspace_size(64, 32, 128, 4096, 512) == \
        ops.decode_workspace_size(64, 32, 128, 256, 16, 512)
    assert ops.decode_shared_workspace_size(320, 32, 128, 96, 16, 512, 1024) == (
        _count_bytes(320 * 32) + 320 * 32 * (3 + 1 + 4) * 130 * 4)
    out = ctypes.c_size_t(0)
    assert lib.pa_decode_contiguous_workspace_size(4, 4, 128, 40, 0, ctypes.byref(out)) == 1
