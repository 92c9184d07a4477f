"""Benchmark of the paged-attention hot path on GB300.

One step = one pass of the decode hot path over one batch of the
Llama-3-8B-shaped workload (64 sequences, L ~ U[128,4096], 32 query / 8 KV
heads, head_dim 128, bf16, 16-token blocks in a shuffled pool 1.2x the need):
pa_reshape_and_cache of the 64 new tokens, then pa_decode (split-KV partials
+ log-sum-exp merge).  Inputs are resident in HBM and larger than L2; three
independent pools are rotated between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle on a bounded sample of the same workload instead.

Multi-GPU: sequences are independent, so every rank runs its own replica of
the batch (weak scaling, no collective on the data path); ranks meet only at
the barriers around the timed region and in the max-over-ranks reduction of
the elapsed time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_192_gb300 import synth  # noqa: E402

METRIC = "paged decode attn: KV GB/s (% of GB300 HBM peak) and tokens/s at 1 GPU"
WORKLOAD = "llama3-8b-gqa-decode"
N_POOLS = 3
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas only)
# ----------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(value, world, device="cpu"):
    """Max of a float over ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, world, device="cpu"):
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------
# workload accounting
# ----------------------------------------------------------------------------

def decode_bytes(w):
    """Algorithmic HBM bytes of one pa_decode: every cached token's K and V
    row once per KV head, q and out once, the block-table entries read, the
    context lengths.  Split-KV partials are overhead, not counted."""
    es = 2 if w.dtype == torch.bfloat16 else 4
    kv = int(w.lens.sum()) * 2 * w.Hkv * w.d * es
    qo = 2 * w.B * w.Hq * w.d * es
    tables = int(sum(-(-int(L) // w.bs) for L in w.lens)) * 4 + w.B * 4
    return kv + qo + tables


def reshape_bytes(w):
    es = 2 if w.dtype == torch.bfloat16 else 4
    return w.B * (2 * 2 * w.Hkv * w.d * es + 8)  # read + write K and V rows, slot


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_traffic():
    """ncu DRAM bytes per decode launch, if recorded for the current kernel
    source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        j = json.load(f)
    if j.get("source_sha1") != source_sha1():
        return None
    return j.get("bytes_per_launch")


def source_sha1():
    h = hashlib.sha1()
    for name in ("pa_decode.cu", "pa_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_192_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.t0 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args, world, rank, local):
    from paged_kv_cache_192_gb300 import build
    build.build()
    from paged_kv_cache_192_gb300 import layout, ops
    from paged_kv_cache_192_gb300._lib import PA_BF16, check, lib

    assert torch.cuda.is_available(), "the GPU arm needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    w = synth.decode_workload("8b", seed=args.seed)
    B, Hq, Hkv, d, bs = w.B, w.Hq, w.Hkv, w.d, w.bs
    MB = w.max_blocks
    PT = args.partition
    scale = 1.0 / math.sqrt(d)

    # resident inputs: N_POOLS independent pools (each 1.2x the batch's blocks)
    pools = []
    for _ in range(args.pools):
        kc, vc = layout.alloc_pools(w.num_blocks, Hkv, bs, d, w.dtype, dev, poison=False)
        layout.fill_pools(kc, vc, w.k, w.v, w.table, w.lens, bs)
        pools.append((kc, vc))
    table = torch.from_numpy(w.table).to(dev)
    lens = torch.from_numpy(w.lens.astype(np.int32)).to(dev)
    q = w.q.to(dev)
    offs = w.kv_offsets
    last = torch.from_numpy(offs + w.lens - 1)
    k_new = w.k[last].contiguous().to(dev)
    v_new = w.v[last].contiguous().to(dev)
    slots = torch.from_numpy(np.array(
        [layout.slots_for(w.table[s], [w.lens[s] - 1], bs)[0] for s in range(B)],
        dtype=np.int64)).to(dev)
    ws_bytes = ops.decode_workspace_size(B, Hq, d, MB, bs, PT)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device=dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    L = lib()
    launches_per_step = 2  # reshape_and_cache + the persistent decode kernel (B <= 1024)

    def step(i, t_dec=None):
        kc, vc = pools[i % len(pools)]
        check(L.pa_reshape_and_cache(k_new.data_ptr(), v_new.data_ptr(), kc.data_ptr(),
                                     vc.data_ptr(), slots.data_ptr(), B, w.num_blocks, Hkv, bs, d,
                                     PA_BF16, sp))
        if t_dec is not None:
            t_dec[0].record(stream)
        check(L.pa_decode(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                          table.data_ptr(), MB, lens.data_ptr(), B, Hq, Hkv, d, bs, w.num_blocks,
                          scale, PT, ws.data_ptr(), ws_bytes, PA_BF16, sp))
        if t_dec is not None:
            t_dec[1].record(stream)

    # warm-up: W steps, then keep the GPU busy >= 1 s so clocks settle
    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    t_end = time.time() + (0.0 if args.quick else 1.0)
    i = 0
    while time.time() < t_end:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize()

    # timed region: exactly K steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        step(i, ev[i])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    # keep the sampler running a little under load for the clock record
    t_end = time.time() + (0.0 if args.quick else 0.5)
    while time.time() < t_end:
        for _ in range(50):
            step(i)
        torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed_ms = e0.elapsed_time(e1)
    dec_ms = [a.elapsed_time(b) for a, b in ev]
    elapsed_ms = reduce_max(elapsed_ms, world, dev)
    ms_per_step = elapsed_ms / args.steps

    step_bytes = decode_bytes(w) + reshape_bytes(w)
    units = reduce_sum(step_bytes * args.steps, world, dev)
    value = units / (elapsed_ms / 1e3) / 1e9  # GB/s, whole job
    tokens = reduce_sum(B * args.steps, world, dev)
    tok_s = tokens / (elapsed_ms / 1e3)

    # end to end: host buffers through the C ABI, copies inside the timed region
    h_q = q.cpu().pin_memory()
    h_kn, h_vn = k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
    h_slots = slots.cpu().pin_memory()
    h_table = table.cpu().pin_memory()
    h_lens = lens.cpu().pin_memory()
    h_out = torch.empty_like(q, device="cpu").pin_memory()
    d_q, d_kn, d_vn = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new)
    d_slots, d_table, d_lens = torch.empty_like(slots), torch.empty_like(table), torch.empty_like(
        lens)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_kn, h_vn, h_slots, h_table, h_lens))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step(i):
        kc, vc = pools[i % len(pools)]
        for dst, src in ((d_q, h_q), (d_kn, h_kn), (d_vn, h_vn), (d_slots, h_slots),
                         (d_table, h_table), (d_lens, h_lens)):
            dst.copy_(src, non_blocking=True)
        check(L.pa_reshape_and_cache(d_kn.data_ptr(), d_vn.data_ptr(), kc.data_ptr(),
                                     vc.data_ptr(), d_slots.data_ptr(), B, w.num_blocks, Hkv, bs,
                                     d, PA_BF16, sp))
        check(L.pa_decode(out.data_ptr(), d_q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                          d_table.data_ptr(), MB, d_lens.data_ptr(), B, Hq, Hkv, d, bs,
                          w.num_blocks, scale, PT, ws.data_ptr(), ws_bytes, PA_BF16, sp))
        h_out.copy_(out, non_blocking=True)

    if args.quick:
        print(json.dumps({"quick": True, "ms_per_step": ms_per_step, "value": value}))
        return
    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(f0.elapsed_time(f1), world, dev)
    e2e_value = reduce_sum(step_bytes * args.steps, world, dev) / (e2e_ms / 1e3) / 1e9

    # roofline of the dominant op (pa_decode: partial kernel + merge), timed live
    peak, peak_kind = peaks()
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    achieved = decode_bytes(w) / (dec_avg_ms / 1e3) / 1e9
    traffic = kernel_traffic()
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 K/V/q; shuffled block placement)",
        "config": {"workload": WORKLOAD, "B": B, "Hq": Hq, "Hkv": Hkv, "head_dim": d,
                   "block_size": bs, "context_len": "U[128,4096] seed %d" % args.seed,
                   "total_context_tokens": int(w.lens.sum()), "pool_blocks": w.num_blocks,
                   "partition_tokens": PT, "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2 ({decode_bytes(w) / 1e6:.0f} MB per step) "
                         f"and {len(pools)} pools rotated"},
        "tokens_per_s": round(tok_s, 1),
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "pa_decode (decode_persistent_kernel, split-KV merge inside)",
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "avg_launch_us": round(dec_avg_ms * 1e3, 2),
                     "algorithmic_bytes": decode_bytes(w)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 5)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ----------------------------------------------------------------------------

def oracle_sample(w, n_seq, seed):
    seqs = synth.sample_indices(w.B, n_seq, seed=seed)
    offs = w.kv_offsets
    k = torch.cat([w.k[offs[s]:offs[s] + w.lens[s]] for s in seqs]).double().numpy()
    v = torch.cat([w.v[offs[s]:offs[s] + w.lens[s]] for s in seqs]).double().numpy()
    q = w.q[torch.from_numpy(seqs)].double().numpy()
    lens = w.lens[seqs]
    es = 2 if w.dtype == torch.bfloat16 else 4
    nbytes = int(lens.sum()) * 2 * w.Hkv * w.d * es + 2 * len(seqs) * w.Hq * w.d * es
    return q, k, v, lens, nbytes, seqs


def time_oracle(w, n_seq, seed, threads):
    import oracle
    q, k, v, lens, nbytes, seqs = oracle_sample(w, n_seq, seed)
    t0 = time.perf_counter()
    oracle.decode(q, k, v, lens, 1.0 / math.sqrt(w.d), nthreads=threads)
    dt = time.perf_counter() - t0
    return dt, nbytes, len(seqs)


def cpu_baseline(w, args, budget_s=10.0):
    """The oracle as it stands on the host cores: the whole batch's decode,
    repeated until about budget_s seconds of CPU time have passed."""
    import oracle
    threads = os.cpu_count() or 1
    q, k, v, lens, nbytes, seqs = oracle_sample(w, w.B, args.seed)
    reps, total = 0, 0.0
    while reps == 0 or total < budget_s:
        t0 = time.perf_counter()
        oracle.decode(q, k, v, lens, 1.0 / math.sqrt(w.d), nthreads=threads)
        total += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps * nbytes / total / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"whole batch ({w.B} sequences) decoded {reps}x by the fp64 C oracle on "
                      f"{threads} threads, {total:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = synth.decode_workload("8b", seed=args.seed)
    threads = os.cpu_count() or 1
    n_seq = args.cpu_sample_seqs
    for _ in range(args.warmup):
        time_oracle(w, max(1, n_seq // 8), args.seed, threads)
    total_t, total_b = 0.0, 0
    for i in range(args.steps):
        dt, nbytes, n = time_oracle(w, n_seq, args.seed + i, threads)
        total_t += dt
        total_b += nbytes
    value = total_b / total_t / 1e9
    res = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d,
                   "block_size": w.bs, "context_len": "U[128,4096] seed %d" % args.seed,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{n_seq} of {w.B} sequences per step (seeded), fp64 C "
                                   f"oracle, {threads} threads"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--partition", type=int, default=512)
    ap.add_argument("--cpu-sample-seqs", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pools", type=int, default=N_POOLS, help="pools rotated between steps")
    ap.add_argument("--quick", action="store_true",
                    help="profiling case: no clock warm loop, no e2e, no CPU baseline")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)


if __name__ == "__main__":
    main()
