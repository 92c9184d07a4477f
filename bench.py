"""Benchmark of the paged-attention hot path on GB300.

A step is one pass of the hot path over one batch, every call through the C
ABI of include/pa.h, inputs resident in HBM:

* 8b (default, the headline): Llama-3-8B-shaped decode batch (64 sequences,
  L ~ U[128,4096], 32 query / 8 KV heads, head_dim 128, bf16, 16-token blocks
  shuffled over a pool 1.2x the need): pa_reshape_and_cache of the 64 new
  tokens, then pa_decode (persistent kernel, split-KV merged inside).
* 70b: Llama-3-70B-shaped long-context decode (32 sequences, L ~ U[16k,32k],
  64/8 heads, 32-token blocks, 512-token split-KV partitions).
* prefix: 256 sequences sharing a 1024-token system prompt plus 64
  parallel-sampling forks set up through the native block manager; the step
  runs the fork's copy-on-write block copies, stores the 320 new tokens and
  decodes all 320 sequences.
* mixed: continuous batch of 128 decodes (L ~ U[256,8192]) and 4 chunked-prefill
  requests of 512 tokens over 0..3584 prior tokens in one pool; the step stores
  all 2176 new tokens, decodes and runs the prefill chunks.

Inputs are larger than L2 and three independent pools are rotated between
steps.  Prints ONE JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
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
import re
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
WORKLOADS = {"8b": "llama3-8b-gqa-decode", "70b": "llama3-70b-long-decode",
             "prefix": "shared-prefix-decode-with-forks", "mixed": "mixed-decode-prefill-batch"}
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

def _es(dtype):
    return 2 if dtype == torch.bfloat16 else 4


def decode_bytes(lens, B, Hq, Hkv, d, bs, dtype):
    """Algorithmic HBM bytes of one pa_decode: every cached token's K and V row
    once per KV head, q and out once, the block-table entries read and the
    context lengths.  Split-KV partials are overhead, not counted."""
    es = _es(dtype)
    kv = int(np.sum(lens)) * 2 * Hkv * d * es
    return kv + 2 * B * Hq * d * es + int(sum(-(-int(L) // bs) for L in lens)) * 4 + B * 4


def store_bytes(T, Hkv, d, dtype):
    """pa_reshape_and_cache: read and write of T rows of K and V, slots."""
    return T * (2 * 2 * Hkv * d * _es(dtype) + 8)


def prefill_flops(priors, n_new, Hq, d):
    """QK^T and PV of causal chunks: 4*Hq*d*(n*P + n(n+1)/2) per request."""
    return int(sum(4 * Hq * d * (n * P + n * (n + 1) // 2) for P, n in zip(priors, n_new)))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops_sustained"]), "measured"
    return 6800.0, 1700.0, "fallback"


def source_sha1(*names):
    """sha1 of the kernel sources with comments removed and whitespace
    collapsed: a counter record stays valid across comment and layout edits
    and no longer across code edits."""
    h = hashlib.sha1()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_192_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


# kernel sources each traffic record is keyed to (the decode call of a
# workload; the prefill chunk of the mixed batch)
DECODE_SOURCES = ("pa_decode.cu", "pa_device.cuh")
PREFIX_SOURCES = DECODE_SOURCES + ("pa_prefill.cu", "pa_prefill.cuh", "pa_tcgen05.cuh")
PREFILL_SOURCES = ("pa_prefill_persist.cu", "pa_prefill.cuh", "pa_tcgen05.cuh", "pa_device.cuh")


def traffic_sources(workload):
    return PREFIX_SOURCES if workload == "prefix" else DECODE_SOURCES


def kernel_traffic(record, *sources):
    """ncu DRAM bytes per launch of a kernel, if recorded for its current
    source (else None)."""
    path = os.path.join(ROOT, "profiles", record)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        j = json.load(f)
    if j.get("source_sha1") != source_sha1(*sources):
        return None
    return j.get("bytes_per_launch")


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

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
# step plans
# ----------------------------------------------------------------------------

class Plan:
    """Device-resident inputs of one workload and the calls of one step."""

    def __init__(self, name):
        self.name = name
        self.pools = []        # [(k_cache, v_cache)]
        self.inputs = {}       # name -> device tensor re-sent each e2e step
        self.outputs = {}      # name -> device tensor read back each e2e step
        self.config = {}
        self.extra = {}
        self.step_bytes = 0    # algorithmic bytes of one step (the metric's unit)
        self.tokens = 0        # query tokens produced per step
        self.decode_bytes = 0
        self.roofline_bytes = None   # HBM roofline numerator if not decode_bytes
        self.roofline_basis = "algorithmic bytes"
        self.prefill_flops = 0
        self.launches = 0
        self.decode_kernel = None
        self.oracle_sample = None  # callable(n_seq, seed, threads) -> (seconds, bytes, n)

    def run(self, i, L, sp, ev=None, src=None, dst=None):
        raise NotImplementedError


def unique_kv_bytes(table, lens, bs, Hkv, d, es):
    """K and V bytes of the distinct physical blocks that a decode batch reads
    (each whole (block, KV head) piece once, however many sequences share it)."""
    used = set()
    for r, L in enumerate(lens):
        used.update(np.asarray(table[r][:-(-int(L) // bs)]).tolist())
    return len(used) * Hkv * bs * d * es * 2


def decode_kernel_info(B, Hq, Hkv, d, MB, bs, NB, PT):
    """(name of the decode kernel for the roofline line, launches of one
    pa_decode) for a bf16 batch of these sizes."""
    from paged_kv_cache_192_gb300 import ops
    if ops.decode_kernel_for(B, Hkv, MB, bs, PT) == "persistent":
        tile = ops.decode_tile_for(Hq, Hkv, d, bs, NB).replace("_", "-")
        return (f"pa_decode (decode_persistent_kernel, {tile} tile, then "
                "partial_merge_kernel merging split items)", 2)
    return "pa_decode (decode_kernel, then merge_kernel)", 2


def _slots_last(table, lens, bs):
    from paged_kv_cache_192_gb300 import layout
    return np.array([layout.slots_for(table[s], [lens[s] - 1], bs)[0] for s in range(len(lens))],
                    dtype=np.int64)


class DecodePlan(Plan):
    """Store each sequence's newest token, then decode the batch."""

    def __init__(self, name, dev, args):
        super().__init__(name)
        from paged_kv_cache_192_gb300 import layout, ops
        gen_dev = "cuda" if name == "70b" else "cpu"
        w = synth.decode_workload(name, seed=args.seed, gen_device=gen_dev,
                                  bs=args.block_size or None, B=args.batch or None)
        if args.placement == "identity":
            # paging-overhead control: every sequence's blocks consecutive
            table = np.zeros_like(w.table)
            pos = 0
            for s_, L_ in enumerate(w.lens):
                nb_ = -(-int(L_) // w.bs)
                table[s_, :nb_] = np.arange(pos, pos + nb_)
                pos += nb_
            w.table = table
        self.w = w
        self.contig = args.layout == "contiguous"
        # contiguous control: every sequence reserves the config's maximum length
        self.max_len = -(-synth.CONFIGS[name]["len_range"][1] // 32) * 32
        for _ in range(args.pools):
            if self.contig:
                kc = torch.zeros(w.B, w.Hkv, self.max_len, w.d, dtype=w.dtype, device=dev)
                vc = torch.zeros_like(kc)
                offs = w.kv_offsets
                for b_ in range(w.B):
                    L_ = int(w.lens[b_])
                    kc[b_, :, :L_] = w.k[offs[b_]:offs[b_] + L_].to(dev).transpose(0, 1)
                    vc[b_, :, :L_] = w.v[offs[b_]:offs[b_] + L_].to(dev).transpose(0, 1)
            else:
                kc, vc = layout.alloc_pools(w.num_blocks, w.Hkv, w.bs, w.d, w.dtype, dev,
                                            poison=False)
                layout.fill_pools(kc, vc, w.k, w.v, w.table, w.lens, w.bs)
            self.pools.append((kc, vc))
        if w.k.is_cuda:  # keep only the pools on the device
            w.k, w.v, w.q = w.k.cpu(), w.v.cpu(), w.q.cpu()
        last = torch.from_numpy(w.kv_offsets + w.lens - 1)
        self.inputs = {
            "q": w.q.to(dev), "k_new": w.k[last].contiguous().to(dev),
            "v_new": w.v[last].contiguous().to(dev),
            "slots": torch.from_numpy(_slots_last(w.table, w.lens, w.bs)).to(dev),
            "table": torch.from_numpy(w.table).to(dev),
            "lens": torch.from_numpy(w.lens.astype(np.int32)).to(dev)}
        self.outputs = {"out": torch.empty_like(self.inputs["q"])}
        self.PT = args.partition
        self.ws_bytes = ops.decode_workspace_size(w.B, w.Hq, w.d, w.max_blocks, w.bs, self.PT)
        self.decode_kernel, n_dec = decode_kernel_info(w.B, w.Hq, w.Hkv, w.d, w.max_blocks, w.bs,
                                                        w.num_blocks, self.PT)
        self.decode_bytes = decode_bytes(w.lens, w.B, w.Hq, w.Hkv, w.d, w.bs, w.dtype)
        self.step_bytes = self.decode_bytes + store_bytes(w.B, w.Hkv, w.d, w.dtype)
        self.launches = 1 + n_dec
        if self.contig:
            # the same decode over contiguous reservations: no table, no store
            self.ws_bytes = ops.decode_contiguous_workspace_size(w.B, w.Hq, w.d, self.max_len,
                                                                 self.PT)
            self.decode_kernel = ("pa_decode_contiguous (decode_persistent_kernel over "
                                  f"[B][Hkv][{self.max_len}][d] reservations, then "
                                  "partial_merge_kernel)")
            self.decode_bytes -= int(sum(-(-int(L) // w.bs) for L in w.lens)) * 4
            self.step_bytes = self.decode_bytes
            self.launches = 2
            self.inputs = {k_: self.inputs[k_] for k_ in ("q", "lens")}
        self.ws = torch.zeros(max(self.ws_bytes // 4, 1), dtype=torch.float32, device=dev)
        self.tokens = w.B
        lo, hi = synth.CONFIGS[name]["len_range"]
        self.config = {"B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d, "block_size": w.bs,
                       "context_len": f"U[{lo},{hi}] seed {args.seed}",
                       "total_context_tokens": int(w.lens.sum()), "pool_blocks": w.num_blocks,
                       "partition_tokens": self.PT, "placement": args.placement}
        if self.contig:
            self.config.update(layout=f"contiguous [B][Hkv][{self.max_len}][d] reservations "
                                      "(paging-overhead control; step = decode only)",
                               placement=None, pool_blocks=None)
        paged, contig = layout.kv_utilization(w.lens, w.bs, hi)
        self.extra = {"kv_utilization_paged": round(paged, 4),
                      f"kv_utilization_contiguous_reserve_{hi}": round(contig, 4),
                      "block_table_bytes": int(sum(-(-int(L) // w.bs) for L in w.lens)) * 4}
        self.oracle_sample = lambda n, seed, threads=None: time_oracle_decode(w, n, seed, threads)

    def run(self, i, L, sp, ev=None, src=None, dst=None):
        from paged_kv_cache_192_gb300._lib import PA_BF16, check
        w, x = self.w, (src or self.inputs)
        kc, vc = self.pools[i % len(self.pools)]
        if self.contig:
            if ev:
                ev["decode"][0].record()
            check(L.pa_decode_contiguous((dst or self.outputs)["out"].data_ptr(),
                                         x["q"].data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                         x["lens"].data_ptr(), w.B, w.Hq, w.Hkv, w.d,
                                         self.max_len, 1.0 / math.sqrt(w.d), self.PT,
                                         self.ws.data_ptr(), self.ws_bytes, PA_BF16, sp))
            if ev:
                ev["decode"][1].record()
            return
        check(L.pa_reshape_and_cache(x["k_new"].data_ptr(), x["v_new"].data_ptr(), kc.data_ptr(),
                                     vc.data_ptr(), x["slots"].data_ptr(), w.B, w.num_blocks,
                                     w.Hkv, w.bs, w.d, PA_BF16, sp))
        if ev:
            ev["decode"][0].record()
        check(L.pa_decode((dst or self.outputs)["out"].data_ptr(), x["q"].data_ptr(), kc.data_ptr(),
                          vc.data_ptr(), x["table"].data_ptr(), w.max_blocks,
                          x["lens"].data_ptr(), w.B, w.Hq, w.Hkv, w.d, w.bs, w.num_blocks,
                          1.0 / math.sqrt(w.d), self.PT, self.ws.data_ptr(), self.ws_bytes,
                          PA_BF16, sp))
        if ev:
            ev["decode"][1].record()


class PrefixPlan(Plan):
    """Shared system prompt + private suffixes + 64 forks, through the native
    block manager; step = CoW block copies, store 320 new tokens, decode 320."""

    def __init__(self, dev, args):
        super().__init__("prefix")
        from paged_kv_cache_192_gb300 import layout, ops
        cfg = synth.CONFIGS["prefix"]
        pf = synth.prefix_fork_workload(seed=args.seed)
        w = pf.base
        P = w.extra["prefix"]
        Hkv, d, bs, Hq = w.Hkv, w.d, w.bs, w.Hq
        B, nf = w.B, cfg["forks"]
        st = layout.place_prefix_forks(pf, bm_seed=args.seed + 5)
        NB, table, lens, pairs = st["num_blocks"], st["table"], st["lens"], st["pairs"]
        MB = table.shape[1]
        order = list(range(B + nf))
        for _ in range(args.pools):
            kc = torch.zeros(NB, Hkv, bs, d, dtype=w.dtype, device=dev)
            vc = torch.zeros_like(kc)
            # prompt once, then each sequence's private history (all but its newest token)
            ops.reshape_and_cache(w.k[:P].to(dev), w.v[:P].to(dev), kc, vc,
                                  torch.from_numpy(st["prompt_slots"]).to(dev))
            rows = torch.from_numpy(st["hist_rows"])
            ops.reshape_and_cache(w.k[rows].to(dev), w.v[rows].to(dev), kc, vc,
                                  torch.from_numpy(st["hist_slots"]).to(dev))
            self.pools.append((kc, vc))
        new_slots = st["new_slots"]
        k_new, v_new = st["k_new"], st["v_new"]
        q_children = pf.q_child
        # decode order: each child right after its parent, so that the child's
        # reads of the parent's private blocks find them in L2
        child_of = {int(par): B + i for i, par in enumerate(pf.parents)}
        dec_order = []
        for s_ in range(B):
            dec_order.append(s_)
            if s_ in child_of:
                dec_order.append(child_of[s_])
        dec_order = np.asarray(dec_order)
        table, lens = table[dec_order], lens[dec_order]
        q_all = torch.cat([w.q, q_children])[torch.from_numpy(dec_order)]
        self.NB, self.MB, self.Bd = NB, MB, len(order)
        self.Hq, self.Hkv, self.d, self.bs, self.dtype = Hq, Hkv, d, bs, w.dtype
        self.npairs = len(pairs)
        self.inputs = {
            "q": q_all.to(dev), "k_new": k_new.to(dev),
            "v_new": v_new.to(dev),
            "slots": torch.tensor(new_slots, dtype=torch.int64, device=dev),
            "table": torch.from_numpy(np.ascontiguousarray(table)).to(dev),
            "lens": torch.from_numpy(lens.astype(np.int32)).to(dev),
            "pairs": torch.tensor(pairs if pairs else [[0, 0]], dtype=torch.int64, device=dev)}
        self.outputs = {"out": torch.empty_like(self.inputs["q"])}
        self.PT = args.partition
        # every sequence takes the 1024-token system prompt from one group's
        # shared blocks (default); with forks each child also takes the blocks
        # before its fork point from its parent's reads (measured slower here:
        # the fork kernel's wider slot rows and extra per-tile work cost more
        # than the 38 MB of reads it saves)
        self.path = args.prefix_path
        self.shared = self.path in ("shared", "forks")
        Bd = B + nf
        pos = {int(o): k for k, o in enumerate(dec_order)}
        fork_parent = np.full(Bd, -1, dtype=np.int32)
        fork_len = np.zeros(Bd, dtype=np.int32)
        for i, par in enumerate(pf.parents):
            # the parent's blocks at the fork, but its last, partly filled one
            # (copied on write by whichever writes first)
            fork_parent[pos[B + i]] = pos[int(par)]
            fork_len[pos[B + i]] = (int(w.lens[par]) - 1) // bs * bs
        self.inputs.update({
            "shared_len": torch.full((Bd,), P, dtype=torch.int32, device=dev),
            "group_start": torch.tensor([0, Bd], dtype=torch.int32, device=dev),
            "group_seqs": torch.arange(Bd, dtype=torch.int32, device=dev),
            "fork_parent": torch.from_numpy(fork_parent).to(dev),
            "fork_len": torch.from_numpy(fork_len).to(dev)})
        self.P = P
        if self.shared:
            wsf = (ops.decode_shared_forks_workspace_size if self.path == "forks"
                   else ops.decode_shared_workspace_size)
            self.ws_bytes = wsf(Bd, Hq, d, MB, bs, self.PT, P)
            name, n_dec = decode_kernel_info(Bd, Hq, Hkv, d, MB, bs, NB, self.PT)
            self.decode_kernel = (
                ("pa_decode_shared_forks" if self.path == "forks" else "pa_decode_shared") +
                " (" + name + "; then the shared prompt once per KV head for all members on "
                "tensor cores" + ("; each child's query heads ride with its parent's reads "
                                  "over the blocks before its fork" if self.path == "forks"
                                  else "") + ")")
            n_dec += 1
        else:
            self.ws_bytes = ops.decode_workspace_size(Bd, Hq, d, MB, bs, self.PT)
            self.decode_kernel, n_dec = decode_kernel_info(Bd, Hq, Hkv, d, MB, bs, NB, self.PT)
        self.ws = torch.zeros(max(self.ws_bytes // 4, 1), dtype=torch.float32, device=dev)
        es = _es(w.dtype)
        self.decode_bytes = decode_bytes(lens, self.Bd, Hq, Hkv, d, bs, w.dtype)
        unique = unique_kv_bytes(table, lens, bs, Hkv, d, es)
        # roofline on unique bytes: the shared prompt is read from HBM once and
        # then served from L2 to every sequence that shares it
        logical_kv = int(np.sum(lens)) * 2 * Hkv * d * es
        self.roofline_bytes = unique + (self.decode_bytes - logical_kv)
        self.roofline_basis = "unique bytes (each physical block once) + q, out, tables"
        self.step_bytes = (self.decode_bytes + store_bytes(self.Bd, Hkv, d, w.dtype) +
                           self.npairs * 2 * 2 * Hkv * bs * d * es)
        self.tokens = self.Bd
        self.launches = (2 if self.npairs else 1) + n_dec
        self.extra = {"unique_kv_bytes": unique, "logical_kv_bytes": self.decode_bytes,
                      "cow_pairs": self.npairs}
        self.config = {"B": self.Bd, "sequences": f"{B} sharing a {P}-token prompt + {nf} forks "
                                                  "(each child decoded right after its parent)",
                       "suffix_len": "U[1,512]", "Hq": Hq, "Hkv": Hkv, "head_dim": d,
                       "block_size": bs, "pool_blocks": NB, "partition_tokens": self.PT,
                       "cow_pairs": self.npairs,
                       "decode": {"forks": "pa_decode_shared_forks, one group of all "
                                           f"sequences over the {P}-token prompt and the "
                                           f"{nf} forks",
                                  "shared": "pa_decode_shared, one group of all sequences "
                                            f"over the {P}-token prompt",
                                  "plain": "pa_decode"}[self.path]}
        self.oracle_sample = lambda n, seed, threads=None: time_oracle_decode(w, n, seed, threads)

    def run(self, i, L, sp, ev=None, src=None, dst=None):
        from paged_kv_cache_192_gb300._lib import PA_BF16, check
        x = src or self.inputs
        kc, vc = self.pools[i % len(self.pools)]
        if self.npairs:
            check(L.pa_copy_blocks(kc.data_ptr(), vc.data_ptr(), x["pairs"].data_ptr(),
                                   self.npairs, self.NB, self.Hkv, self.bs, self.d, PA_BF16, sp))
        check(L.pa_reshape_and_cache(x["k_new"].data_ptr(), x["v_new"].data_ptr(), kc.data_ptr(),
                                     vc.data_ptr(), x["slots"].data_ptr(), self.Bd, self.NB,
                                     self.Hkv, self.bs, self.d, PA_BF16, sp))
        if ev:
            ev["decode"][0].record()
        if self.path == "forks":
            check(L.pa_decode_shared_forks(
                (dst or self.outputs)["out"].data_ptr(), x["q"].data_ptr(), kc.data_ptr(),
                vc.data_ptr(), x["table"].data_ptr(), self.MB, x["lens"].data_ptr(), self.Bd,
                self.Hq, self.Hkv, self.d, self.bs, self.NB, 1.0 / math.sqrt(self.d), self.PT,
                x["shared_len"].data_ptr(), x["group_start"].data_ptr(),
                x["group_seqs"].data_ptr(), 1, self.Bd, self.Bd, self.P,
                x["fork_parent"].data_ptr(), x["fork_len"].data_ptr(), self.ws.data_ptr(),
                self.ws_bytes, PA_BF16, sp))
        elif self.shared:
            check(L.pa_decode_shared(
                (dst or self.outputs)["out"].data_ptr(), x["q"].data_ptr(), kc.data_ptr(),
                vc.data_ptr(), x["table"].data_ptr(), self.MB, x["lens"].data_ptr(), self.Bd,
                self.Hq, self.Hkv, self.d, self.bs, self.NB, 1.0 / math.sqrt(self.d), self.PT,
                x["shared_len"].data_ptr(), x["group_start"].data_ptr(),
                x["group_seqs"].data_ptr(), 1, self.Bd, self.Bd, self.P, self.ws.data_ptr(),
                self.ws_bytes, PA_BF16, sp))
        else:
            check(L.pa_decode((dst or self.outputs)["out"].data_ptr(), x["q"].data_ptr(),
                              kc.data_ptr(), vc.data_ptr(), x["table"].data_ptr(), self.MB,
                              x["lens"].data_ptr(), self.Bd, self.Hq, self.Hkv, self.d, self.bs,
                              self.NB, 1.0 / math.sqrt(self.d), self.PT, self.ws.data_ptr(),
                              self.ws_bytes, PA_BF16, sp))
        if ev:
            ev["decode"][1].record()


class MixedPlan(Plan):
    """128 decodes + 4 chunked-prefill requests sharing one pool."""

    def __init__(self, dev, args):
        super().__init__("mixed")
        from paged_kv_cache_192_gb300 import layout, ops
        dec, pre = synth.mixed_workload(seed=args.seed)
        self.dec, self.pre = dec, pre
        n, R = pre.extra["chunk"], pre.B
        priors = pre.extra["prior"]
        doffs, poffs = dec.kv_offsets, pre.kv_offsets
        # history = every decode token but the newest and every prior prefill token
        hist_rows_d = np.concatenate([np.arange(doffs[s], doffs[s] + dec.lens[s] - 1)
                                      for s in range(dec.B)])
        hist_slots_d = np.concatenate([layout.slots_for(dec.table[s], np.arange(dec.lens[s] - 1),
                                                        dec.bs) for s in range(dec.B)])
        hist_rows_p = np.concatenate([np.arange(poffs[r], poffs[r] + priors[r]) for r in range(R)])
        hist_slots_p = np.concatenate([layout.slots_for(pre.table[r], np.arange(priors[r]),
                                                        pre.bs) for r in range(R)])
        new_rows_p = np.concatenate([np.arange(poffs[r] + priors[r], poffs[r] + pre.lens[r])
                                     for r in range(R)])
        new_slots_p = np.concatenate([layout.slots_for(pre.table[r],
                                                       np.arange(priors[r], pre.lens[r]), pre.bs)
                                      for r in range(R)])
        for _ in range(args.pools):
            kc, vc = layout.alloc_pools(dec.num_blocks, dec.Hkv, dec.bs, dec.d, dec.dtype, dev,
                                        poison=False)
            ops.reshape_and_cache(dec.k[hist_rows_d].to(dev), dec.v[hist_rows_d].to(dev), kc, vc,
                                  torch.from_numpy(hist_slots_d).to(dev))
            if len(hist_rows_p):
                ops.reshape_and_cache(pre.k[hist_rows_p].to(dev), pre.v[hist_rows_p].to(dev), kc,
                                      vc, torch.from_numpy(hist_slots_p).to(dev))
            self.pools.append((kc, vc))
        last = torch.from_numpy(doffs + dec.lens - 1)
        k_new = torch.cat([dec.k[last], pre.k[new_rows_p]])
        v_new = torch.cat([dec.v[last], pre.v[new_rows_p]])
        slots = np.concatenate([_slots_last(dec.table, dec.lens, dec.bs), new_slots_p])
        self.inputs = {
            "q": dec.q.to(dev), "qp": pre.q.to(dev), "k_new": k_new.to(dev),
            "v_new": v_new.to(dev), "slots": torch.from_numpy(slots).to(dev),
            "table": torch.from_numpy(np.ascontiguousarray(dec.table)).to(dev),
            "lens": torch.from_numpy(dec.lens.astype(np.int32)).to(dev),
            "ptable": torch.from_numpy(np.ascontiguousarray(pre.table)).to(dev),
            "plens": torch.from_numpy(pre.lens.astype(np.int32)).to(dev),
            "qstart": torch.arange(0, (R + 1) * n, n, dtype=torch.int32, device=dev)}
        self.outputs = {"out": torch.empty_like(self.inputs["q"]),
                        "outp": torch.empty_like(self.inputs["qp"])}
        self.T = len(slots)
        self.n, self.R = n, R
        self.PT = args.partition
        self.ws_bytes = ops.decode_workspace_size(dec.B, dec.Hq, dec.d, dec.max_blocks, dec.bs,
                                                  self.PT)
        self.decode_kernel, n_dec = decode_kernel_info(dec.B, dec.Hq, dec.Hkv, dec.d,
                                                       dec.max_blocks, dec.bs, dec.num_blocks,
                                                       self.PT)
        self.ws = torch.zeros(max(self.ws_bytes // 4, 1), dtype=torch.float32, device=dev)
        self.decode_bytes = decode_bytes(dec.lens, dec.B, dec.Hq, dec.Hkv, dec.d, dec.bs,
                                         dec.dtype)
        es = _es(dec.dtype)
        prefill_kv = (int(pre.lens.sum()) * 2 * pre.Hkv * pre.d * es +
                      2 * R * n * pre.Hq * pre.d * es)
        self.step_bytes = (self.decode_bytes + prefill_kv +
                           store_bytes(self.T, dec.Hkv, dec.d, dec.dtype))
        self.prefill_flops = prefill_flops(priors, [n] * R, pre.Hq, pre.d)
        self.prefill_kernel = {
            "persistent": f"prefill_persist_kernel<{pre.d},{pre.Hq // pre.Hkv}>",
            "item_grid": f"prefill_tc2_kernel<{pre.d},{pre.Hq // pre.Hkv}>",
            "simple": f"prefill_tc_kernel<{pre.d},{pre.Hq // pre.Hkv}>"}[
            ops.prefill_kernel_for(R, n, pre.Hq, pre.Hkv, pre.d, pre.bs, dec.num_blocks,
                                   pre.max_blocks)]
        self.tokens = dec.B + R * n
        self.launches = 2 + n_dec
        self.extra = {"prefill_flops": self.prefill_flops, "priors": [int(x) for x in priors]}
        self.config = {"B_decode": dec.B, "decode_len": "U[256,8192]", "prefill_requests": R,
                       "chunk": n, "priors": [int(x) for x in priors], "Hq": dec.Hq,
                       "Hkv": dec.Hkv, "head_dim": dec.d, "block_size": dec.bs,
                       "pool_blocks": dec.num_blocks, "partition_tokens": self.PT}
        self.oracle_sample = lambda k, seed, threads=None: time_oracle_decode(dec, k, seed, threads)

    def run(self, i, L, sp, ev=None, src=None, dst=None):
        from paged_kv_cache_192_gb300._lib import PA_BF16, check
        dec, pre, x = self.dec, self.pre, (src or self.inputs)
        kc, vc = self.pools[i % len(self.pools)]
        check(L.pa_reshape_and_cache(x["k_new"].data_ptr(), x["v_new"].data_ptr(), kc.data_ptr(),
                                     vc.data_ptr(), x["slots"].data_ptr(), self.T, dec.num_blocks,
                                     dec.Hkv, dec.bs, dec.d, PA_BF16, sp))
        if ev:
            ev["decode"][0].record()
        check(L.pa_decode((dst or self.outputs)["out"].data_ptr(), x["q"].data_ptr(), kc.data_ptr(),
                          vc.data_ptr(), x["table"].data_ptr(), dec.max_blocks,
                          x["lens"].data_ptr(), dec.B, dec.Hq, dec.Hkv, dec.d, dec.bs,
                          dec.num_blocks, 1.0 / math.sqrt(dec.d), self.PT, self.ws.data_ptr(),
                          self.ws_bytes, PA_BF16, sp))
        if ev:
            ev["decode"][1].record()
            ev["prefill"][0].record()
        check(L.pa_prefill_chunk((dst or self.outputs)["outp"].data_ptr(), x["qp"].data_ptr(),
                                 kc.data_ptr(), vc.data_ptr(), x["ptable"].data_ptr(),
                                 pre.max_blocks, x["qstart"].data_ptr(), x["plens"].data_ptr(),
                                 self.R, self.n, pre.Hq, pre.Hkv, pre.d, pre.bs, dec.num_blocks,
                                 1.0 / math.sqrt(pre.d), PA_BF16, sp))
        if ev:
            ev["prefill"][1].record()


def make_plan(name, dev, args):
    if name in ("8b", "70b"):
        return DecodePlan(name, dev, args)
    if name == "prefix":
        return PrefixPlan(dev, args)
    return MixedPlan(dev, args)


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def _events(n, keys):
    return [{k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for k in keys} for _ in range(n)]


def run_gpu(args, world, rank, local):
    from paged_kv_cache_192_gb300 import build
    build.build()
    from paged_kv_cache_192_gb300._lib import lib

    assert torch.cuda.is_available(), "the GPU arm needs a CUDA device"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    plan = make_plan(args.workload, dev, args)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    L = lib()
    keys = ["decode"] + (["prefill"] if plan.prefill_flops else [])

    # warm-up: W steps, then keep the GPU busy >= 1 s so clocks settle
    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        plan.run(i, L, sp)
    torch.cuda.synchronize()
    t_end = time.time() + (0.0 if args.quick else 1.0)
    i = 0
    while time.time() < t_end:
        for _ in range(20):
            plan.run(i, L, sp)
            i += 1
        torch.cuda.synchronize()

    # timed region: exactly K steps, nothing else on the stream between the
    # calls (an event recorded between two of the library's launches would
    # serialize their programmatic-dependent launch)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        plan.run(i, L, sp)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    # kernel pass: the same K steps again with CUDA events on the stream
    # around each dominant call, for the roofline's average launch duration
    ev = _events(args.steps, keys)
    torch.cuda.synchronize()
    for i in range(args.steps):
        plan.run(i, L, sp, ev[i])
    torch.cuda.synchronize()
    t_end = time.time() + (0.0 if args.quick else 0.5)
    while time.time() < t_end:
        for _ in range(20):
            plan.run(i, L, sp)
        torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed_ms = reduce_max(e0.elapsed_time(e1), world, dev)
    ms_per_step = elapsed_ms / args.steps
    value = reduce_sum(plan.step_bytes * args.steps, world, dev) / (elapsed_ms / 1e3) / 1e9
    tok_s = reduce_sum(plan.tokens * args.steps, world, dev) / (elapsed_ms / 1e3)
    if args.quick:
        print(json.dumps({"quick": True, "workload": args.workload, "ms_per_step": ms_per_step,
                          "value": value}))
        return

    # end to end: host buffers through the C ABI, every step's copies inside the
    # timed region.  Three streams pipeline the steps: the inputs of step i+1
    # go up (h2d stream) while step i computes, and step i's result comes back
    # (d2h stream) while step i+1 computes; device buffers alternate between
    # two sets, ordered by events.
    h_in = {k: t.cpu().pin_memory() for k, t in plan.inputs.items()}
    d_in = [{k: torch.empty_like(t) for k, t in plan.inputs.items()} for _ in range(2)]
    d_out = [{k: torch.empty_like(t) for k, t in plan.outputs.items()} for _ in range(2)]
    h_out = {k: torch.empty_like(t, device="cpu").pin_memory() for k, t in plan.outputs.items()}
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of a buffer set landed
    ev_run = [torch.cuda.Event() for _ in range(2)]   # a set's step computed
    ev_out = [torch.cuda.Event() for _ in range(2)]   # a set's result read back

    def upload(i):
        b = i % 2
        with torch.cuda.stream(up):
            up.wait_event(ev_run[b])          # step i-2 is done with these inputs
            for k in h_in:
                d_in[b][k].copy_(h_in[k], non_blocking=True)
            ev_in[b].record(up)

    def e2e_steps(n, first):
        upload(first)
        for i in range(first, first + n):
            b = i % 2
            if i + 1 < first + n:
                upload(i + 1)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])      # step i-2's result has been read back
            plan.run(i, L, sp, src=d_in[b], dst=d_out[b])
            ev_run[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_run[b])
                for k in h_out:
                    h_out[k].copy_(d_out[b][k], non_blocking=True)
                ev_out[b].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    e2e_steps(args.warmup, 0)
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    up.wait_event(f0)
    down.wait_event(f0)
    e2e_steps(args.steps, args.warmup)
    f1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(f0.elapsed_time(f1), world, dev)
    e2e_value = reduce_sum(plan.step_bytes * args.steps, world, dev) / (e2e_ms / 1e3) / 1e9

    # roofline of the dominant kernel(s), timed live with events on the stream
    hbm, bf16_sus, peak_kind = peaks()
    dec_ms = sum(e["decode"][0].elapsed_time(e["decode"][1]) for e in ev) / len(ev)
    rbytes = plan.roofline_bytes or plan.decode_bytes
    achieved = rbytes / (dec_ms / 1e3) / 1e9
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 K/V/q; shuffled block placement)",
        "config": dict({"workload": WORKLOADS[args.workload]}, **plan.config,
                       parallelism=f"replicas{world}",
                       l2="inputs larger than L2 and %d pools rotated" % len(plan.pools)),
        "tokens_per_s": round(tok_s, 1),
        "pct_of_hbm_peak": round(100 * value / hbm, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     # the prefix record was taken on the default (shared) path
                     "traffic": (kernel_traffic(f"decode_traffic_{args.workload}.json",
                                                *traffic_sources(args.workload))
                                 if getattr(plan, "path", "shared") == "shared" else None),
                     "kernel": plan.decode_kernel,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "avg_launch_us": round(dec_ms * 1e3, 2),
                     "timing": "CUDA events on the launching stream around each pa_decode "
                               "call, in a pass of the same K steps right after the timed "
                               "region",
                     "algorithmic_bytes": rbytes, "bytes_basis": plan.roofline_basis},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 5)},
        "gpu_launches": plan.launches * args.steps,
        "clocks": clk,
    }
    if plan.prefill_flops:
        pre_ms = sum(e["prefill"][0].elapsed_time(e["prefill"][1]) for e in ev) / len(ev)
        tf = plan.prefill_flops / (pre_ms / 1e3) / 1e12
        result["roofline_prefill"] = {
            "bound": "tensor", "achieved": round(tf, 2), "peak": bf16_sus, "unit": "TFLOP/s",
            "frac": round(tf / bf16_sus, 4),
            "traffic": kernel_traffic("prefill_traffic_mixed.json", *PREFILL_SOURCES),
            "kernel": plan.prefill_kernel,
            "peak_source": f"{peak_kind} bf16_tflops_sustained",
            "avg_launch_us": round(pre_ms * 1e3, 2), "algorithmic_flops": plan.prefill_flops}
    if plan.extra:
        result["workload_detail"] = plan.extra
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(plan, args)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ----------------------------------------------------------------------------

def time_oracle_decode(w, n_seq, seed, threads=None):
    """Time the fp64 oracle's decode of n_seq seeded sequences of workload w."""
    import oracle
    seqs = synth.sample_indices(w.B, n_seq, seed=seed)
    offs = w.kv_offsets
    k = torch.cat([w.k[offs[s]:offs[s] + w.lens[s]] for s in seqs]).double().cpu().numpy()
    v = torch.cat([w.v[offs[s]:offs[s] + w.lens[s]] for s in seqs]).double().cpu().numpy()
    q = w.q[torch.from_numpy(seqs).to(w.q.device)].double().cpu().numpy()
    lens = w.lens[seqs]
    es = _es(w.dtype)
    nbytes = int(lens.sum()) * 2 * w.Hkv * w.d * es + 2 * len(seqs) * w.Hq * w.d * es
    t0 = time.perf_counter()
    oracle.decode(q, k, v, lens, 1.0 / math.sqrt(w.d), nthreads=threads or os.cpu_count() or 1)
    return time.perf_counter() - t0, nbytes, len(seqs)


def cpu_baseline(plan, args, budget_s=10.0):
    """The oracle as it stands on the host cores, on a bounded seeded sample of
    the workload's decode, repeated until about budget_s seconds have passed."""
    threads = os.cpu_count() or 1
    n = args.cpu_sample_seqs
    reps, total, nb, k = 0, 0.0, 0, 0
    while reps == 0 or total < budget_s:
        dt, nbytes, k = plan.oracle_sample(n, args.seed + reps)
        total += dt
        nb += nbytes
        reps += 1
    # the same oracle on one thread, on a smaller sample (about 1 s)
    dt1, nb1, k1, r1 = 0.0, 0, 0, 0
    while r1 == 0 or dt1 < 1.0:
        dt, nbytes, k1 = plan.oracle_sample(2, args.seed + r1, 1)
        dt1 += dt
        nb1 += nbytes
        r1 += 1
    return {"value": round(nb / total / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{reps} x {k} seeded sequences of the workload's decode, fp64 C oracle on "
                      f"{threads} threads, {total:.1f} s",
            "one_thread": {"value": round(nb1 / dt1 / 1e9, 4), "unit": "GB/s",
                           "sample": f"{r1} x {k1} seeded sequences, 1 thread, {dt1:.1f} s"}}


def reference_workload(args):
    """The host-side synthetic workload whose decode the oracle times: the
    same seeded inputs as the GPU arm's workload (its cpu_baseline samples
    the same decode).  Returns (workload, context-length description)."""
    name = args.workload
    if name in ("8b", "70b"):
        w = synth.decode_workload(name, seed=args.seed, bs=args.block_size or None,
                                  B=args.batch or None)
        lo, hi = synth.CONFIGS[name]["len_range"]
        return w, f"U[{lo},{hi}] seed {args.seed}"
    if name == "prefix":
        pf = synth.prefix_fork_workload(seed=args.seed)
        return pf.base, (f"{pf.base.extra['prefix']}-token shared prompt + U[1,512] private "
                         f"suffix, seed {args.seed} (the sequences before the forks)")
    dec, _ = synth.mixed_workload(seed=args.seed)
    return dec, f"the mixed batch's decodes, seed {args.seed} (its prefill chunks not timed)"


def run_reference(args, world, rank):
    if rank != 0:
        return
    w, ctx = reference_workload(args)
    threads = os.cpu_count() or 1
    n_seq = args.cpu_sample_seqs
    for _ in range(args.warmup):
        time_oracle_decode(w, max(1, n_seq // 8), args.seed, threads)
    total_t, total_b = 0.0, 0
    for i in range(args.steps):
        dt, nbytes, n = time_oracle_decode(w, n_seq, args.seed + i, threads)
        total_t += dt
        total_b += nbytes
    value = total_b / total_t / 1e9
    res = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total_t / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS[args.workload], "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "head_dim": w.d, "block_size": w.bs, "context_len": ctx,
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
    ap.add_argument("--workload", choices=list(WORKLOADS), default="8b")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--partition", type=int, default=512)
    ap.add_argument("--block-size", type=int, default=0,
                    help="override the decode workload's block size (block-size sweep)")
    ap.add_argument("--placement", choices=["shuffled", "identity"], default="shuffled",
                    help="physical placement of each sequence's blocks (decode workloads)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the decode workload's batch size (small profiling cases "
                         "of the same shape)")
    ap.add_argument("--layout", choices=["paged", "contiguous"], default="paged",
                    help="decode workloads: paged pools, or the contiguous-reservation control "
                         "(pa_decode_contiguous, no block table)")
    ap.add_argument("--prefix-path", choices=["shared", "forks", "plain"], default="shared",
                    help="prefix workload: decode with the prompt group (pa_decode_shared), "
                         "the prompt group and the forks (pa_decode_shared_forks) or every "
                         "sequence whole (pa_decode)")
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
