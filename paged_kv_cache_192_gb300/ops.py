"""Torch-facing binding of the paged-attention ops (argument marshalling only).

Every function passes device pointers, sizes and the current CUDA stream to
the C ABI of include/pa.h; all work runs in the library's sm_103a kernels.
Tensors must be contiguous CUDA tensors.  Outputs and workspaces that the
caller does not pass are allocated here with torch (the library itself never
allocates).
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import PA_BF16, PA_F32, check, lib

_DTYPES = {torch.bfloat16: PA_BF16, torch.float32: PA_F32}


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DTYPES[t.dtype]


def _cuda(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _require(cond: bool, msg: str):
    """Shape check of a call's tensors (raised, not asserted: the kernels size
    their reads and writes from these shapes)."""
    if not cond:
        raise ValueError(msg)


def _pairs_ok(pairs) -> bool:
    return pairs.numel() == 0 or (pairs.dim() == 2 and pairs.shape[1] == 2)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def set_validate(on: bool):
    check(lib().pa_set_validate(int(bool(on))))


def device_error(clear: bool = True, stream=None) -> int:
    """Device error bits (PA_DEVERR_*) recorded by kernels; 0 if none."""
    bits = ctypes.c_int(0)
    rc = lib().pa_device_error(ctypes.byref(bits), int(clear), _stream(stream))
    if rc not in (_lib.PA_OK, _lib.PA_ERR_DEVICE):
        check(rc)
    return bits.value


def check_wait_timeout(stream=None):
    """Launch the bounded-wait diagnostic (about 2 s on the GPU); its
    outcome is read with device_error()."""
    check(lib().pa_check_wait_timeout(_stream(stream)))


def reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping, stream=None):
    """Store new K/V rows into their slots of the pools (pa_reshape_and_cache).

    k_new, v_new: [T][Hkv][d], the pools' dtype.  k_cache, v_cache:
    [NB][Hkv][bs][d], written in place.  slot_mapping: int64 [T], slot =
    physical block * bs + offset; a negative slot is padding and is skipped.
    Bit exact.  Duplicate slots in one call are a caller error."""
    _require(k_cache.dim() == 4 and k_new.dim() == 3,
             "pools must be [NB][Hkv][bs][d] and k_new [T][Hkv][d]")
    NB, Hkv, bs, d = k_cache.shape
    T = k_new.shape[0]
    _require(k_new.shape == (T, Hkv, d) and v_new.shape == k_new.shape,
             f"k_new/v_new must be [T][Hkv][d] = [{T}][{Hkv}][{d}]")
    _require(v_cache.shape == k_cache.shape, "k_cache and v_cache must have the same shape")
    _require(slot_mapping.shape == (T,), f"slot_mapping must be [{T}]")
    check(lib().pa_reshape_and_cache(
        _cuda(k_new, "k_new", k_cache.dtype), _cuda(v_new, "v_new", k_cache.dtype),
        _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache", k_cache.dtype),
        _cuda(slot_mapping, "slot_mapping", torch.int64), T, NB, Hkv, bs, d, _dt(k_cache),
        _stream(stream)))


def copy_blocks(k_cache, v_cache, pairs, stream=None):
    """Copy-on-write copies (pa_copy_blocks): for each row (src, dst) of the
    int64 [n][2] device tensor `pairs`, block dst of both pools becomes a byte
    copy of block src.  No dst may equal a src or another dst of the call."""
    _require(k_cache.dim() == 4, "pools must be [NB][Hkv][bs][d]")
    NB, Hkv, bs, d = k_cache.shape
    _require(v_cache.shape == k_cache.shape, "k_cache and v_cache must have the same shape")
    _require(_pairs_ok(pairs), "pairs must be [n][2]")
    n = pairs.shape[0] if pairs.numel() else 0
    check(lib().pa_copy_blocks(
        _cuda(k_cache, "k_cache"), _cuda(v_cache, "v_cache", k_cache.dtype),
        _cuda(pairs, "pairs", torch.int64) if n else None, n, NB, Hkv, bs, d, _dt(k_cache),
        _stream(stream)))


def swap_blocks(dst_k, dst_v, src_k, src_v, pairs, stream=None):
    """Copy blocks pairs[i][0] of the source pools into blocks pairs[i][1] of
    the destination pools; either side may be pinned host memory."""
    _require(src_k.dim() == 4 and dst_k.dim() == 4, "pools must be [NB][Hkv][bs][d]")
    NBs, Hkv, bs, d = src_k.shape
    NBd = dst_k.shape[0]
    _require(dst_k.shape[1:] == src_k.shape[1:] and dst_v.shape == dst_k.shape,
             "destination pools must be [NB'][Hkv][bs][d] like the source pools")
    _require(src_v.shape == src_k.shape, "src_k and src_v must have the same shape")
    _require(src_k.dtype == dst_k.dtype == src_v.dtype == dst_v.dtype, "pools must share a dtype")
    _require(_pairs_ok(pairs), "pairs must be [n][2]")
    n = pairs.shape[0] if pairs.numel() else 0
    for name, t in (("dst_k", dst_k), ("dst_v", dst_v), ("src_k", src_k), ("src_v", src_v),
                    ("pairs", pairs)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if pairs.dtype != torch.int64:
        raise TypeError("pairs must be int64")
    check(lib().pa_swap_blocks(dst_k.data_ptr(), dst_v.data_ptr(), src_k.data_ptr(),
                               src_v.data_ptr(), pairs.data_ptr() if n else None, n, NBs, NBd,
                               Hkv, bs, d, _dt(src_k), _stream(stream)))


def decode_workspace_size(B, Hq, head_dim, max_blocks_per_seq, block_size, partition_tokens=0):
    out = ctypes.c_size_t(0)
    check(lib().pa_decode_workspace_size(B, Hq, head_dim, max_blocks_per_seq, block_size,
                                         partition_tokens, ctypes.byref(out)))
    return out.value


def decode_kernel_for(B, Hkv, max_blocks_per_seq, block_size, partition_tokens=0) -> str:
    """Kernel pa_decode runs for these sizes on the current device:
    "persistent" or "grid"."""
    out = ctypes.c_int(0)
    check(lib().pa_decode_kernel_for(B, Hkv, max_blocks_per_seq, block_size, partition_tokens,
                                     ctypes.byref(out)))
    return {_lib.PA_DECODE_PERSISTENT: "persistent", _lib.PA_DECODE_GRID: "grid"}[out.value]


def prefill_kernel_for(R, max_query_len, Hq, Hkv, head_dim, block_size, num_blocks,
                       max_blocks_per_seq) -> str:
    """Kernel pa_prefill_chunk runs for these sizes: "persistent" (one CTA per
    SM running a list of work items), "item_grid" (one CTA per item) or
    "simple" (128-thread CTAs; other block sizes and longer tables)."""
    out = ctypes.c_int(0)
    check(lib().pa_prefill_kernel_for(R, max_query_len, Hq, Hkv, head_dim, block_size,
                                      num_blocks, max_blocks_per_seq, ctypes.byref(out)))
    return {_lib.PA_PREFILL_PERSISTENT_GRID: "persistent", _lib.PA_PREFILL_ITEM_GRID: "item_grid",
            _lib.PA_PREFILL_SIMPLE: "simple"}[out.value]


def decode_tile_for(Hq, Hkv, head_dim, block_size, num_blocks, dtype=torch.bfloat16) -> str:
    """Tile the persistent decode kernel uses for these shapes: "tensor_core"
    (bf16, groups of 4 or 8 heads) or "cuda_core"."""
    out = ctypes.c_int(0)
    check(lib().pa_decode_tile_for(Hq, Hkv, head_dim, block_size, num_blocks,
                                   _DTYPES[dtype], ctypes.byref(out)))
    return {_lib.PA_DECODE_TILE_CUDA_CORE: "cuda_core",
            _lib.PA_DECODE_TILE_TENSOR_CORE: "tensor_core"}[out.value]


def _check_decode_shapes(q, k_cache, v_cache, block_table, context_lens, out):
    _require(q.dim() == 3 and k_cache.dim() == 4, "q must be [B][Hq][d], pools [NB][Hkv][bs][d]")
    B, Hq, d = q.shape
    _require(k_cache.shape[3] == d, f"pools must have head_dim {d} like q")
    _require(v_cache.shape == k_cache.shape, "k_cache and v_cache must have the same shape")
    _require(block_table.dim() == 2 and block_table.shape[0] == B,
             f"block_table must be [{B}][max_blocks_per_seq]")
    _require(context_lens.shape == (B,), f"context_lens must be [{B}]")
    _require(out is None or out.shape == q.shape, "out must have the shape of q")


def decode(q, k_cache, v_cache, block_table, context_lens, scale=None, partition_tokens=0,
           workspace=None, out=None, stream=None):
    """Paged decode attention (pa_decode): one query token per sequence.

    q: [B][Hq][d]; k_cache, v_cache: [NB][Hkv][bs][d] (same dtype, bf16 or
    fp32); block_table: int32 [B][max_blocks_per_seq]; context_lens: int32
    [B], each in [1, max_blocks_per_seq * bs] and counting the newest token.
    Query head h attends over KV head h // (Hq // Hkv).  scale defaults to
    1/sqrt(d); partition_tokens (0 = 512) sets the split-KV partitions.
    workspace (fp32 tensor of at least decode_workspace_size bytes) and out
    ([B][Hq][d]) are allocated when not given.  Returns out.  Asynchronous on
    `stream` (default: the current stream)."""
    _check_decode_shapes(q, k_cache, v_cache, block_table, context_lens, out)
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    MB = block_table.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = decode_workspace_size(B, Hq, d, MB, bs, partition_tokens)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().pa_decode(
        _cuda(out, "out", q.dtype), _cuda(q, "q", k_cache.dtype), _cuda(k_cache, "k_cache"),
        _cuda(v_cache, "v_cache", k_cache.dtype), _cuda(block_table, "block_table", torch.int32),
        MB, _cuda(context_lens, "context_lens", torch.int32), B, Hq, Hkv, d, bs, NB, scale,
        partition_tokens, ws_ptr, ws_len, _dt(q), _stream(stream)))
    return out


def decode_contiguous_workspace_size(B, Hq, head_dim, max_len, partition_tokens=0):
    out = ctypes.c_size_t(0)
    check(lib().pa_decode_contiguous_workspace_size(B, Hq, head_dim, max_len, partition_tokens,
                                                    ctypes.byref(out)))
    return out.value


def decode_contiguous(q, k, v, context_lens, scale=None, partition_tokens=0, workspace=None,
                      out=None, stream=None):
    """Decode over plain contiguous caches (pa_decode_contiguous): k, v
    [B][Hkv][max_len][d], max_len a multiple of 32; no block table.  The
    paging-overhead control of decode."""
    _require(q.dim() == 3 and k.dim() == 4 and v.shape == k.shape,
             "q must be [B][Hq][d], k and v [B][Hkv][max_len][d]")
    B, Hq, d = q.shape
    _require(k.shape[0] == B and k.shape[3] == d, f"k must be [{B}][Hkv][max_len][{d}]")
    _require(context_lens.shape == (B,), f"context_lens must be [{B}]")
    _require(out is None or out.shape == q.shape, "out must have the shape of q")
    Hkv, max_len = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = decode_contiguous_workspace_size(B, Hq, d, max_len, partition_tokens)
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().pa_decode_contiguous(
        _cuda(out, "out", q.dtype), _cuda(q, "q", k.dtype), _cuda(k, "k"), _cuda(v, "v", k.dtype),
        _cuda(context_lens, "context_lens", torch.int32), B, Hq, Hkv, d, max_len, scale,
        partition_tokens, ws_ptr, ws_len, _dt(q), _stream(stream)))
    return out


def decode_shared_workspace_size(B, Hq, head_dim, max_blocks_per_seq, block_size,
                                 partition_tokens=0, max_shared_len=0):
    out = ctypes.c_size_t(0)
    check(lib().pa_decode_shared_workspace_size(B, Hq, head_dim, max_blocks_per_seq, block_size,
                                                partition_tokens, max_shared_len,
                                                ctypes.byref(out)))
    return out.value


def decode_shared(q, k_cache, v_cache, block_table, context_lens, shared_len, group_start,
                  group_seqs, max_group_size, max_shared_len, scale=None, partition_tokens=0,
                  workspace=None, out=None, stream=None):
    """Paged decode of a batch whose groups share prefix blocks (pa_decode_shared).

    As decode, plus: shared_len int32 [B] (tokens each sequence takes from its
    group's shared blocks, 0 outside any group), group_start int32 [G+1] and
    group_seqs int32 [members] (CSR member lists of the groups), and host
    bounds max_group_size and max_shared_len.  The shared blocks of each group
    are read once per KV head for all members; the result equals decode's
    within the error bound."""
    _check_decode_shapes(q, k_cache, v_cache, block_table, context_lens, out)
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    MB = block_table.shape[1]
    _require(shared_len.shape == (B,), f"shared_len must be [{B}]")
    _require(group_start.dim() == 1 and group_start.numel() >= 1, "group_start must be [G+1]")
    G = group_start.numel() - 1
    M = group_seqs.numel()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = decode_shared_workspace_size(B, Hq, d, MB, bs, partition_tokens, max_shared_len)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().pa_decode_shared(
        _cuda(out, "out", q.dtype), _cuda(q, "q", k_cache.dtype), _cuda(k_cache, "k_cache"),
        _cuda(v_cache, "v_cache", k_cache.dtype), _cuda(block_table, "block_table", torch.int32),
        MB, _cuda(context_lens, "context_lens", torch.int32), B, Hq, Hkv, d, bs, NB, scale,
        partition_tokens, _cuda(shared_len, "shared_len", torch.int32),
        _cuda(group_start, "group_start", torch.int32),
        _cuda(group_seqs, "group_seqs", torch.int32) if M else None, G, M, int(max_group_size),
        int(max_shared_len), ws_ptr, ws_len, _dt(q), _stream(stream)))
    return out


def decode_shared_forks_workspace_size(B, Hq, head_dim, max_blocks_per_seq, block_size,
                                       partition_tokens=0, max_shared_len=0):
    out = ctypes.c_size_t(0)
    check(lib().pa_decode_shared_forks_workspace_size(B, Hq, head_dim, max_blocks_per_seq,
                                                      block_size, partition_tokens,
                                                      max_shared_len, ctypes.byref(out)))
    return out.value


def decode_shared_forks(q, k_cache, v_cache, block_table, context_lens, shared_len,
                        group_start, group_seqs, max_group_size, max_shared_len, fork_parent,
                        fork_len, scale=None, partition_tokens=0, workspace=None, out=None,
                        stream=None):
    """pa_decode_shared_forks: decode_shared for a batch that also holds forked
    children.  fork_parent int32 [B] (a child's parent row, else -1) and
    fork_len int32 [B] (tokens whose blocks a child shares with its parent):
    the blocks a child shares with its parent are read once for both."""
    _check_decode_shapes(q, k_cache, v_cache, block_table, context_lens, out)
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    MB = block_table.shape[1]
    _require(shared_len.shape == (B,), f"shared_len must be [{B}]")
    _require(fork_parent.shape == (B,) and fork_len.shape == (B,),
             f"fork_parent and fork_len must be [{B}]")
    _require(group_start.dim() == 1 and group_start.numel() >= 1, "group_start must be [G+1]")
    G = group_start.numel() - 1
    M = group_seqs.numel()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = decode_shared_forks_workspace_size(B, Hq, d, MB, bs, partition_tokens,
                                                  max_shared_len)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().pa_decode_shared_forks(
        _cuda(out, "out", q.dtype), _cuda(q, "q", k_cache.dtype), _cuda(k_cache, "k_cache"),
        _cuda(v_cache, "v_cache", k_cache.dtype), _cuda(block_table, "block_table", torch.int32),
        MB, _cuda(context_lens, "context_lens", torch.int32), B, Hq, Hkv, d, bs, NB, scale,
        partition_tokens, _cuda(shared_len, "shared_len", torch.int32),
        _cuda(group_start, "group_start", torch.int32),
        _cuda(group_seqs, "group_seqs", torch.int32) if M else None, G, M, int(max_group_size),
        int(max_shared_len), _cuda(fork_parent, "fork_parent", torch.int32),
        _cuda(fork_len, "fork_len", torch.int32), ws_ptr, ws_len, _dt(q), _stream(stream)))
    return out


def decode_noalloc_capacity() -> int:
    """Bytes of the library's fixed decode scratch (pa_decode_noalloc)."""
    return int(lib().pa_decode_noalloc_capacity())


def decode_noalloc(q, k_cache, v_cache, block_table, context_lens, scale=None,
                   partition_tokens=0, out=None, stream=None):
    """pa_decode_noalloc: as decode, with the split-KV workspace taken from the
    library's fixed device array (nothing is allocated when `out` is given);
    calls that overlap on the GPU race on that array."""
    _check_decode_shapes(q, k_cache, v_cache, block_table, context_lens, out)
    B, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    check(lib().pa_decode_noalloc(
        _cuda(out, "out", q.dtype), _cuda(q, "q", k_cache.dtype), _cuda(k_cache, "k_cache"),
        _cuda(v_cache, "v_cache", k_cache.dtype), _cuda(block_table, "block_table", torch.int32),
        block_table.shape[1], _cuda(context_lens, "context_lens", torch.int32), B, Hq, Hkv, d,
        bs, NB, scale, partition_tokens, _dt(q), _stream(stream)))
    return out


def prefill_chunk(q, k_cache, v_cache, block_table, query_start, context_lens, max_query_len,
                  scale=None, out=None, stream=None):
    """Causal chunked prefill over paged context (pa_prefill_chunk), bf16.

    R requests; request r owns query rows query_start[r] .. query_start[r+1]
    of q [sum n][Hq][d], the chunk's newest tokens, whose K/V are already in
    the pools.  context_lens: int32 [R], prior + new tokens; the query at
    position P_r + i attends to positions 0 .. P_r + i.  block_table: int32
    [R][max_blocks_per_seq]; max_query_len bounds the chunks' lengths.
    Returns out [sum n][Hq][d]."""
    _require(q.dim() == 3 and k_cache.dim() == 4 and context_lens.dim() == 1,
             "q must be [tokens][Hq][d], pools [NB][Hkv][bs][d], context_lens [R]")
    Tq, Hq, d = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    R = context_lens.shape[0]
    _require(k_cache.shape[3] == d, f"pools must have head_dim {d} like q")
    _require(v_cache.shape == k_cache.shape, "k_cache and v_cache must have the same shape")
    _require(query_start.shape == (R + 1,), f"query_start must be [{R + 1}]")
    _require(block_table.dim() == 2 and block_table.shape[0] == R,
             f"block_table must be [{R}][max_blocks_per_seq]")
    _require(out is None or out.shape == q.shape, "out must have the shape of q")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    check(lib().pa_prefill_chunk(
        _cuda(out, "out", q.dtype), _cuda(q, "q", k_cache.dtype), _cuda(k_cache, "k_cache"),
        _cuda(v_cache, "v_cache", k_cache.dtype), _cuda(block_table, "block_table", torch.int32),
        block_table.shape[1], _cuda(query_start, "query_start", torch.int32),
        _cuda(context_lens, "context_lens", torch.int32), R, int(max_query_len), Hq, Hkv, d, bs,
        NB, scale, _dt(q), _stream(stream)))
    return out
