"""Shared helpers of the GPU parity tests (not a test module)."""
import numpy as np
import torch

import oracle

# Pass rule per element: |gpu - oracle| <= ATOL + RTOL * |oracle|.
# bf16 K/V: max abs 2e-3, max rel 1e-2; fp32 K/V: 1e-5.
TOL = {torch.bfloat16: (2e-3, 1e-2), torch.float32: (1e-5, 1e-5)}


def compare(got, ref, dtype, what=""):
    """Assert the pass rule; return (max abs err, max rel err over |ref| >= atol/rtol)."""
    atol, rtol = TOL[dtype]
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    big = np.abs(ref) >= atol / rtol
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance, "
                           f"max abs {err.max():.3e}, max rel {max_rel:.3e}")
    return float(err.max()), max_rel


def device_inputs(w, dev="cuda", poison=True):
    """Pools filled from the workload's logical K/V through pa_reshape_and_cache."""
    from paged_kv_cache_192_gb300 import layout
    k_cache, v_cache = layout.alloc_pools(w.num_blocks, w.Hkv, w.bs, w.d, w.dtype, dev, poison)
    layout.fill_pools(k_cache, v_cache, w.k, w.v, w.table, w.lens, w.bs)
    table = torch.from_numpy(np.ascontiguousarray(w.table)).to(dev)
    lens = torch.from_numpy(w.lens.astype(np.int32)).to(dev)
    return k_cache, v_cache, table, lens


def oracle_decode(w, seqs=None, nthreads=None):
    """fp64 oracle for the decode of the selected sequences (all by default)."""
    offs = w.kv_offsets
    seqs = np.arange(w.B) if seqs is None else np.asarray(seqs)
    ks = [w.k[offs[s]:offs[s] + w.lens[s]] for s in seqs]
    vs = [w.v[offs[s]:offs[s] + w.lens[s]] for s in seqs]
    k = torch.cat(ks).double().numpy()
    v = torch.cat(vs).double().numpy()
    q = w.q[torch.from_numpy(seqs)].double().numpy()
    return oracle.decode(q, k, v, w.lens[seqs], 1.0 / np.sqrt(w.d), nthreads)


def oracle_decode_all(w, chunk=8, nthreads=None):
    """fp64 oracle for every sequence of the batch, a few sequences at a time
    (bounds the host memory of the float64 copies of long histories)."""
    parts = [oracle_decode(w, np.arange(i, min(i + chunk, w.B)), nthreads)
             for i in range(0, w.B, chunk)]
    return np.concatenate(parts)
