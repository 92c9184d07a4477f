"""fp64 CPU oracle for paged attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or executes anything here, and this
package imports nothing from the product.

Contents
--------
* ``pa_oracle.c``  plain C, fp64 loops: causal attention over each sequence's
  logical K/V, the block-table slot rule, the byte-level reshape_and_cache
  scatter and copy_blocks copy.  Built with gcc by :func:`build`.
* ``bm_model.py``  a pure-Python reference model of the block manager (free
  list, refcounts, fork, append with copy-on-write).

Every function states the passage of the pages it follows; see the header of
``pa_oracle.c``.  All attention inputs are float64 arrays holding the exact
values the GPU sees (bf16 values are upcast exactly).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lib = None


def _lib_path(src: str = _SRC) -> str:
    with open(src, "rb") as f:
        h = hashlib.sha1(f.read()).hexdigest()[:12]
    return os.path.join(_BUILD, f"liboracle_{h}.so")


def compile_source(src: str, out: str) -> str:
    """Compile one C source file of the oracle into a shared object."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """Compile pa_oracle.c (if needed) and return the shared object path."""
    path = _lib_path()
    if not os.path.exists(path):
        compile_source(_SRC, path)
    return path


def _declare(lib):
    i64p = ctypes.POINTER(ctypes.c_int64)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention.argtypes = [dp, dp, dp, dp, i64p, i64p, i64p, i64p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_double, ctypes.c_int]
    lib.oracle_slot_mapping.restype = None
    lib.oracle_slot_mapping.argtypes = [ctypes.POINTER(ctypes.c_int32), ctypes.c_int64,
                                        ctypes.c_int, i64p]
    lib.oracle_reshape_and_cache.restype = ctypes.c_int
    lib.oracle_reshape_and_cache.argtypes = [ctypes.c_void_p] * 4 + [i64p, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int]
    lib.oracle_copy_blocks.restype = ctypes.c_int
    lib.oracle_copy_blocks.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i64p, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int]
    return lib


def load(path: str | None = None):
    """Load the oracle library (the default build, or another compiled copy)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _p(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def attention(q, k, v, q_counts, q_pos0, kv_lens, scale, nthreads=None, lib=None):
    """Causal attention of each sequence's query rows over its logical K/V.

    q        float64 [sum(q_counts)][Hq][d]
    k, v     float64 [sum(kv_lens)][Hkv][d]   (sequences stacked in order)
    q_counts query rows per sequence
    q_pos0   absolute position of each sequence's first query row
    kv_lens  K/V rows per sequence
    Returns float64 [sum(q_counts)][Hq][d].
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    S = len(q_counts)
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    q_start = np.zeros(S + 1, dtype=np.int64)
    q_start[1:] = np.cumsum(np.asarray(q_counts, dtype=np.int64))
    kv_len = np.ascontiguousarray(kv_lens, dtype=np.int64)
    kv_start = np.zeros(S, dtype=np.int64)
    if S > 1:
        kv_start[1:] = np.cumsum(kv_len)[:-1]
    pos0 = np.ascontiguousarray(q_pos0, dtype=np.int64)
    assert q.shape[0] == q_start[-1] and k.shape[0] == kv_len.sum() and v.shape == k.shape
    out = np.empty_like(q)
    rc = lib.oracle_attention(_p(q, ctypes.c_double), _p(k, ctypes.c_double),
                              _p(v, ctypes.c_double), _p(out, ctypes.c_double),
                              _p(q_start, ctypes.c_int64), _p(pos0, ctypes.c_int64),
                              _p(kv_start, ctypes.c_int64), _p(kv_len, ctypes.c_int64),
                              S, Hq, Hkv, d, float(scale),
                              int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_attention failed with status {rc}")
    return out


def decode(q, k, v, kv_lens, scale, nthreads=None, lib=None):
    """Decode: one query per sequence at position L-1 (the newest token).

    q [B][Hq][d]; k, v stacked logical histories [sum L][Hkv][d].
    """
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    return attention(q, k, v, np.ones(len(kv_lens), np.int64), kv_lens - 1, kv_lens,
                     scale, nthreads, lib)


def prefill_chunk(q, k, v, n_new, prior, scale, nthreads=None, lib=None):
    """Chunked prefill: request r has prior[r] cached tokens and n_new[r] new
    query tokens at positions prior[r] .. prior[r]+n_new[r]-1; its logical
    K/V history holds prior[r]+n_new[r] rows."""
    n_new = np.asarray(n_new, dtype=np.int64)
    prior = np.asarray(prior, dtype=np.int64)
    return attention(q, k, v, n_new, prior, prior + n_new, scale, nthreads, lib)


def slot_mapping(table_row, n, bs, lib=None):
    """Slots of logical tokens 0..n-1 of one sequence with this block-table row."""
    lib = lib or load()
    t = np.ascontiguousarray(table_row, dtype=np.int32)
    out = np.empty(int(n), dtype=np.int64)
    lib.oracle_slot_mapping(_p(t, ctypes.c_int32), int(n), int(bs), _p(out, ctypes.c_int64))
    return out


def reshape_and_cache(k_new, v_new, k_cache, v_cache, slots, bs, lib=None):
    """In-place byte scatter of new K/V rows into the pools.

    k_new, v_new  [T][Hkv][d] numpy arrays (any element type)
    k_cache, v_cache  [NB][Hkv][bs][d] numpy arrays, modified in place
    """
    lib = lib or load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    s = np.ascontiguousarray(slots, dtype=np.int64)
    NB, Hkv, _, d = k_cache.shape
    rc = lib.oracle_reshape_and_cache(k_new.ctypes.data, v_new.ctypes.data,
                                      k_cache.ctypes.data, v_cache.ctypes.data,
                                      _p(s, ctypes.c_int64), len(s), NB, Hkv, int(bs), d,
                                      k_cache.itemsize)
    if rc != 0:
        raise ValueError("slot outside the pool")


def copy_blocks(k_cache, v_cache, pairs, lib=None):
    """In-place block copies (src -> dst) of both pools."""
    lib = lib or load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    p = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    NB, Hkv, bs, d = k_cache.shape
    rc = lib.oracle_copy_blocks(k_cache.ctypes.data, v_cache.ctypes.data,
                                _p(p, ctypes.c_int64), p.shape[0], NB, Hkv, bs, d,
                                k_cache.itemsize)
    if rc != 0:
        raise ValueError("block index outside the pool")
