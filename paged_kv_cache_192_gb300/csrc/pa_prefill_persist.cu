// Chunked prefill over a paged KV cache on a persistent grid (bf16, tcgen05).
//
// Same result as prefill_tc2_kernel ("Melihat Lebih Dalam vLLM v0.7", section
// "Blueprint Arsitektur 3: Chunked Prefill": new token i of request r sits at
// position P_r + i and attends causally to positions 0..P_r+i of its request,
// read through the block table), with the work dealt out differently.  A work
// item is still (request, 256 query rows, KV head), but one CTA per SM runs a
// list of items: barriers and TMEM are set up once per SM, and the next
// item's block-table slice, query tile and first K/V tiles load while the
// current item's last products and its epilogue run.
//
// Assignment: items are ranked by their number of 64-token K/V tiles (longest
// first) and dealt by longest-processing-time list scheduling: each item in
// turn to the CTA with the least load so far (cost = its tiles plus a fixed
// per-item charge).  Every CTA computes the same assignment; CTA c starts on
// item c at once (the first gridDim.x items go to CTAs 0, 1, ... in order)
// while a spare warp computes the rest.  No global counter and no workspace,
// so launches on different streams never interfere.
//
// Warps: 0-3 and 4-7 softmax of the item's two 128-row query tiles A and B;
// 8 and 11 issue the tcgen05.mma of tile A and of tile B (one lane each, so
// one tile's products never wait behind the other tile's P); 9 loads K/V
// tiles with TMA through a 4-stage ring (a stage is free once both tiles' PV
// are done); 10 schedules and then loads each item's query tiles (3D tensor
// copies: one 16 KB box per full tile and 64 columns).
// TMEM (512 columns): O_A [0,128), O_B [128,256), then per query tile 64
// columns of S and 64 of P (hi, lo): S_A [256,320), P_A [320,384), S_B
// [384,448), P_B [448,512).  A softmax group frees S as soon as it has
// loaded it, so S of the next tile is computed while it works on this one;
// P of the next tile overwrites P only after this tile's PV is done (the
// group waits for that PV before it may rescale O anyway).  Every barrier
// phase follows a CTA-wide tile or item counter, so the pipelines run across
// item boundaries; every wait is bounded.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "pa_prefill.cuh"

namespace {

using namespace pa::pf;

#ifndef PA_PERSIST_NST
#define PA_PERSIST_NST 4  // K/V ring stages
#endif
#ifndef PA_PERSIST_PDL
#define PA_PERSIST_PDL 1  // 0: ordinary stream-ordered launch (A/B of the dependent launch)
#endif
constexpr int kPPairsMax = 256;   // (request, query tile) pairs ranked in-kernel
constexpr int kPItemsMax = 512;   // work items (pair, KV head) per launch
constexpr int kPCharge = 16;      // fixed cost of an item, in 1/8 tiles (~2.5 us)
constexpr int kPCostCap = 4000;   // tiles: 512 items' loads stay below 2^24
constexpr int kPCtasMax = 255;    // the CTA index sits in the low 8 bits of a load

template <int D>
struct PLayout {
    static constexpr int NST = PA_PERSIST_NST;
    static constexpr int THREADS = 12 * 32;
    static constexpr int MMA_WARP = 8, LOAD_WARP = 9, Q_WARP = 10, MMA_WARP_B = 11;
    static constexpr int TMEM_COLS = 512;
    static constexpr int Q_BYTES = 2 * 128 * D * 2;  // two query tiles
    static constexpr int T_BYTES = kT2KT * D * 2;    // one K or V tile
    static constexpr int OFF_KV = Q_BYTES;           // [stage][K|V]
    static constexpr int OFF_BAR = OFF_KV + NST * 2 * T_BYTES;
    // kv_full, kv_empty [NST]; s_full, s_free [2]; p_full, o_done, o_free [2];
    // q_full, q_empty, sched, drain
    static constexpr int N_BAR = 2 * NST + 4 + 6 + 4;
    static constexpr int OFF_MISC = OFF_BAR + 8 * N_BAR;  // TMEM slot, fail flag, list length
    static constexpr int OFF_BT = OFF_MISC + 16;
    static constexpr int BT_MAX = 1024;
    static constexpr int OFF_PAIR = OFF_BT + 4 * BT_MAX;            // 5 int arrays per pair
    static constexpr int OFF_LIST = OFF_PAIR + 5 * 4 * kPPairsMax;  // this CTA's items (u16)
    static constexpr int SMEM = OFF_LIST + 2 * kPItemsMax + 1024;
};

// One work item: query rows t0 .. t0 + 256/GQ - 1 of request r (tokens qs..
// of q, n new tokens, P prior ones), KV head hk, keys [0, kv_end).
struct Item {
    int r, qs, n, P, t0, hk, kv_end, ntiles;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(pa::smem_u32(bar))
        : "memory");
}

// Expect `bytes` more transaction bytes on `bar` in its current phase
// (without arriving).
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(
                     pa::smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

template <int D, int GQ>
__global__ void __launch_bounds__(PLayout<D>::THREADS, 1)
    prefill_persist_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap,
                           const __grid_constant__ CUtensorMap qmap_tile,
                           const __grid_constant__ CUtensorMap qmap_row8) {
    using Lay = PLayout<D>;
    constexpr int NST = Lay::NST;
    constexpr int CH = D * 2 / 16;   // 16-byte chunks per row
    constexpr int QTOK = 256 / GQ;   // query tokens per item
    constexpr int TILE_TX = 2 * kT2KT * D * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sq = pa::smem_u32(smem);
    const uint32_t skv = sq + Lay::OFF_KV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BAR);
    uint64_t *kv_full = bars, *kv_empty = bars + NST;
    uint64_t *s_full = bars + 2 * NST, *s_free = s_full + 2;  // [group]
    uint64_t *p_full = s_full + 4, *o_done = p_full + 2, *o_free = o_done + 2;
    uint64_t *q_full = o_free + 2, *q_empty = q_full + 1, *sched = q_empty + 1, *drain = sched + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + Lay::OFF_MISC);
    volatile int *fail = reinterpret_cast<volatile int *>(smem + Lay::OFF_MISC + 4);
    int *nmine = reinterpret_cast<int *>(smem + Lay::OFF_MISC + 8);
    int32_t *bt_s = reinterpret_cast<int32_t *>(smem + Lay::OFF_BT);
    int *pr_qs = reinterpret_cast<int *>(smem + Lay::OFF_PAIR);
    int *pr_n = pr_qs + kPPairsMax, *pr_P = pr_n + kPPairsMax;
    int *pr_tiles = pr_P + kPPairsMax;  // K/V tiles of the pair; -1: no work
    int *order = pr_tiles + kPPairsMax;  // pairs by decreasing tiles, ties by index
    uint16_t *mine = reinterpret_cast<uint16_t *>(smem + Lay::OFF_LIST);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap_tile)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap_row8)) : "memory");
    }
    // ---- set-up: barriers, TMEM ------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < NST; ++i) {
            pa::mbar_init(&kv_full[i], 1);
            pa::mbar_init(&kv_empty[i], 2);  // both query tiles' PV
        }
        for (int i = 0; i < 2; ++i) {
            pa::mbar_init(&s_full[i], 1);
            pa::mbar_init(&s_free[i], 4);  // one arrival per softmax warp
            pa::mbar_init(&p_full[i], 4);  // one arrival per softmax warp
            pa::mbar_init(&o_done[i], 1);
            pa::mbar_init(&o_free[i], 4);
        }
        pa::mbar_init(q_full, 1);
        pa::mbar_init(q_empty, 2);  // both query tiles' last S
        pa::mbar_init(sched, 1);
        pa::mbar_init(drain, 2);  // both MMA warps
        *fail = 0;
        *nmine = 1;
        mine[0] = static_cast<uint16_t>(blockIdx.x);
        pa::fence_barrier_init();
    }
    if (warp == Lay::MMA_WARP) pa::tc::alloc(tslot, Lay::TMEM_COLS);
    pa::tc::fence_before();
    __syncthreads();
    pa::tc::fence_after();
    const uint32_t tmem = *tslot;
    // launched as a programmatic dependent: everything above may overlap the
    // previous kernel's tail; its results are visible past this point
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- the work items, identical in every CTA ---------------------------------
    const int nqt = (p.max_query_len + QTOK - 1) / QTOK;
    const int npairs = p.R * nqt;  // <= kPPairsMax (host check)
    bool has_work = false;
    if (tid < npairs) {
        const int r = tid / nqt, t0 = (tid % nqt) * QTOK;
        const int qs = p.query_start[r], n = p.query_start[r + 1] - qs, L = p.context_lens[r];
        int tiles = -1;
        if (t0 < n) {
            if (L > (p.MB << p.bs_log2) || L < n) {
                pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            } else {
                tiles = (min(L, L - n + t0 + QTOK) + kT2KT - 1) / kT2KT;
                has_work = true;
            }
        }
        pr_qs[tid] = qs;
        pr_n[tid] = n;
        pr_P[tid] = L - n;
        pr_tiles[tid] = tiles;
    }
    const int nvalid = __syncthreads_count(has_work);
    if (has_work) {
        const int ci = pr_tiles[tid];
        int rank = 0;
        for (int j = 0; j < npairs; ++j) {
            const int cj = pr_tiles[j];
            rank += (cj > ci || (cj == ci && j < tid)) ? 1 : 0;
        }
        order[rank] = tid;
    }
    __syncthreads();
    const int nitems = nvalid * p.Hkv;
    const bool idle = static_cast<int>(blockIdx.x) >= nitems;  // whole CTA: nothing to do

    auto item_of = [&](int k) {
        Item it;
        const int pr = order[k / p.Hkv];
        it.hk = k % p.Hkv;
        it.r = pr / nqt;
        it.t0 = (pr % nqt) * QTOK;
        it.qs = pr_qs[pr];
        it.n = pr_n[pr];
        it.P = pr_P[pr];
        it.kv_end = min(it.P + it.n, it.P + it.t0 + QTOK);
        it.ntiles = pr_tiles[pr];
        return it;
    };
    // item number `it` of this CTA's list into *k; false past the end (or when
    // the wait for the schedule ran out, which sets the fail flag)
    auto next_item = [&](int it, int *k) -> bool {
        if (it == 0) {
            *k = blockIdx.x;
            return true;
        }
        if (!pa::mbar_wait(sched, 0)) {
            *fail = 1;
            return false;
        }
        if (it >= *reinterpret_cast<volatile int *>(nmine)) return false;
        *k = reinterpret_cast<volatile uint16_t *>(mine)[it];
        return true;
    };

    int loads_issued = 0;  // loader lane 0: K/V tiles issued (for the drain after a failure)

    if (idle) {
        // no item: straight to the tear-down
    } else if (warp == Lay::Q_WARP) {
        // ---------------- query tiles and the schedule ----------------
        // Rows m = 128 * tile + i: query token t0 + m / GQ, head hk * GQ + m % GQ.
        // A query tile whose 128 / GQ tokens all lie inside the request comes
        // in as one 3D tensor copy per 64 columns (16 KB); in a tile that the
        // request ends in, groups of 8 / GQ tokens (8 rows) inside it come as
        // 1 KB copies and a last, partial group row by row (cp.async).  Rows
        // past the request's new tokens are not loaded: they keep earlier
        // contents, and as every row's scores, probabilities and output depend
        // on that row alone and such rows are never stored, they affect nothing.
        constexpr int TPB = 8 / GQ;     // tokens per 8-row box
        constexpr int TPT = 128 / GQ;   // tokens per query tile
        auto load_q = [&](const Item &I) {
            const int vtok = min(QTOK, I.n - I.t0);  // new tokens of the item
            const int qt_part = vtok / TPT;          // the tile the request ends in (2: none)
            const int in_part = vtok - qt_part * TPT;  // its tokens inside the request
            const int nsmall = in_part / TPB;          // whole 8-row groups there
            if (in_part % TPB) {
                const int m_part = qt_part * 128 + nsmall * 8;  // first row of the partial group
                for (int idx = lane; idx < 8 * CH; idx += 32) {
                    const int m = m_part + idx / CH, c = idx % CH;
                    const int t = I.t0 + m / GQ;
                    const bool valid = t < I.n;
                    const __nv_bfloat16 *src =
                        p.q + (static_cast<size_t>(I.qs + (valid ? t : 0)) * p.Hq + I.hk * GQ + m % GQ) *
                                  D +
                        c * 8;
                    cp_async16(sq + (m >> 7) * (128 * D * 2) + pa::tc::sw128(m & 127, c * 8, 128),
                               src, valid);
                }
            }
            if (lane == 0) {
                const int nbig = min(qt_part, 2);
                mbar_expect_tx(q_full, static_cast<uint32_t>(nbig * 16 + (qt_part < 2 ? nsmall : 0)) *
                                           (D / 64) * 1024u);
                for (int qt = 0; qt < nbig; ++qt)
#pragma unroll
                    for (int h = 0; h < D / 64; ++h)
                        tma_load_3d(sq + qt * (128 * D * 2) + h * (128 * 128), &qmap_tile, h * 64,
                                    I.hk * GQ, I.qs + I.t0 + qt * TPT, q_full);
                if (qt_part < 2) {
                    for (int b = 0; b < nsmall; ++b)
#pragma unroll
                        for (int h = 0; h < D / 64; ++h)
                            tma_load_3d(sq + qt_part * (128 * D * 2) + h * (128 * 128) + b * 1024,
                                        &qmap_row8, h * 64, I.hk * GQ,
                                        I.qs + I.t0 + qt_part * TPT + b * TPB, q_full);
                }
            }
            cp_async_commit();
            cp_async_wait<0>();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        };
        load_q(item_of(blockIdx.x));

        // Longest-processing-time assignment of items gridDim.x .. nitems-1.
        // Lane l keeps the loads of CTAs l, l + 32, ..., each packed as
        // (load << 8 | CTA) so that one 32-bit minimum picks the least-loaded
        // CTA, the lowest index among equals; lmin is the lane's own minimum.
        // The Hkv items of a (request, query tile) pair are consecutive in
        // rank order and cost the same.
        const int G = gridDim.x;
        auto pair_cost = [&](int rank) -> uint32_t {
            return static_cast<uint32_t>(min(pr_tiles[order[rank]], kPCostCap)) * 8u + kPCharge;
        };
        uint32_t ld[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int c = lane + 32 * s;
            ld[s] = c < G ? ((c < nitems ? pair_cost(c / p.Hkv) : 0u) << 8) | static_cast<uint32_t>(c)
                          : 0xffffffffu;
        }
        auto own_min = [&]() {
            return min(min(min(ld[0], ld[1]), min(ld[2], ld[3])),
                       min(min(ld[4], ld[5]), min(ld[6], ld[7])));
        };
        uint32_t lmin = own_min();
        int cnt = 1;
        for (int k = G; k < nitems;) {
            const int rank = k / p.Hkv;
            const uint32_t add = pair_cost(rank) << 8;
            const int kend = min(nitems, (rank + 1) * p.Hkv);
            for (; k < kend; ++k) {
                const uint32_t mn = __reduce_min_sync(pa::kFull, lmin);
                const int c = static_cast<int>(mn & 0xffu);
                if ((c & 31) == lane) {
#pragma unroll
                    for (int s = 0; s < 8; ++s) ld[s] += s == (c >> 5) ? add : 0u;
                    lmin = own_min();
                }
                if (c == static_cast<int>(blockIdx.x) && lane == 0)
                    mine[cnt++] = static_cast<uint16_t>(k);
            }
        }
        if (lane == 0) {
            *reinterpret_cast<volatile int *>(nmine) = cnt;
            mbar_arrive(sched);
        }
        cnt = __shfl_sync(pa::kFull, cnt, 0);
        for (int it = 1; it < cnt && !*fail; ++it) {
            // the query tiles of item it-1 are free once its last QK^T is done
            if (!__all_sync(pa::kFull, pa::mbar_wait(q_empty, (it - 1) & 1))) {
                *fail = 1;
                break;
            }
            load_q(item_of(mine[it]));
        }
    } else if (warp == Lay::LOAD_WARP) {
        // ---------------- K/V loader ----------------
        const int rows_total = static_cast<int>(p.num_blocks * p.Hkv) << p.bs_log2;
        int g = 0;  // CTA-wide K/V tile counter
        int k;
        for (int it = 0; !*fail && next_item(it, &k); ++it) {
            const Item I = item_of(k);
            // block-table slice of the item (the previous item's tiles are all
            // issued: their row coordinates were taken when they were issued)
            const int nblk = (I.kv_end + p.bs - 1) >> p.bs_log2;
            const int32_t *bt_g = p.block_table + static_cast<size_t>(I.r) * p.MB;
            for (int base = 0; base < nblk; base += 8 * 32) {  // 8 independent loads per lane
                int v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = base + u * 32 + lane;
                    v[u] = i < nblk ? bt_g[i] : 0;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = base + u * 32 + lane;
                    if (i >= nblk) break;
                    if (v[u] < 0 || v[u] >= p.num_blocks) {
                        pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
                        v[u] = 0;
                    }
                    bt_s[i] = v[u];
                }
            }
            __syncwarp();
            if (lane == 0) {
                for (int j = 0; j < I.ntiles; ++j, ++g) {
                    const int st = g % NST;
                    if (g >= NST && !pa::mbar_wait(&kv_empty[st], ((g / NST) - 1) & 1)) {
                        *fail = 1;
                        break;
                    }
                    pa::mbar_arrive_expect_tx(&kv_full[st], TILE_TX);
                    ++loads_issued;
                    const uint32_t kst = skv + st * 2 * Lay::T_BYTES, vst = kst + Lay::T_BYTES;
                    for (int b = 0; b < kT2KT; b += p.bs) {  // bs >= 8: boxes land 1024-aligned
                        const int tok = j * kT2KT + b;
                        const int y = tok < I.kv_end
                                          ? ((bt_s[tok >> p.bs_log2] * p.Hkv + I.hk) << p.bs_log2)
                                          : rows_total;  // out of bounds: zero-filled
#pragma unroll
                        for (int h = 0; h < D / 64; ++h) {
                            const uint32_t off = h * kT2KT * 128 + b * 128;
                            tma_load_2d(kst + off, &kmap, h * 64, y, &kv_full[st]);
                            tma_load_2d(vst + off, &vmap, h * 64, y, &kv_full[st]);
                        }
                    }
                }
            }
            g = __shfl_sync(pa::kFull, g, 0);
            __syncwarp();
        }
    } else if (warp == Lay::MMA_WARP || warp == Lay::MMA_WARP_B) {
        // ---------------- MMA issuers, one per query tile ----------------
        const int wg = warp == Lay::MMA_WARP ? 0 : 1;
        constexpr uint32_t kIdS = pa::tc::idesc_bf16(128, kT2KT, 0, 0);
        constexpr uint32_t kIdO = pa::tc::idesc_bf16(128, D, 0, 1);
        constexpr uint32_t kStage = (2 * Lay::T_BYTES) >> 4;
        const uint64_t dq = pa::tc::sdesc(sq, 16, 1024) +
                            static_cast<uint32_t>(wg * ((128 * D * 2) >> 4));
        const uint64_t dk = pa::tc::sdesc(skv, 16, 1024);
        const uint64_t dv = pa::tc::sdesc(skv + Lay::T_BYTES, kT2KT * 128, 1024);
        const uint32_t sc = tmem + 256 + wg * 128, ph = sc + 64, pl = ph + 32;
        const uint32_t od = tmem + wg * 128;
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(pa::kFull, pa::mbar_wait(bar, parity));
        };
        // S of CTA tile g: TMEM columns 256 + 128 wg, once the group has
        // loaded S of tile g - 1 from them
        auto issue_s = [&](int g) {
            if (g > 0 && !wait_all(&s_free[wg], (g - 1) & 1)) return false;
            pa::tc::fence_after();
            const uint64_t b0 = dk + static_cast<uint32_t>((g % NST) * kStage);
            if (pa::tc::elect_one()) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    pa::tc::mma_ss(sc, dq + (((ks >> 2) * 128 * 128 + (ks & 3) * 32) >> 4),
                                   b0 + (((ks >> 2) * kT2KT * 128 + (ks & 3) * 32) >> 4), kIdS,
                                   ks > 0);
                pa::tc::commit(&s_full[wg]);
            }
            __syncwarp();
            return true;
        };
        // O (+)= P_hi V + P_lo V; P sits in the 64 columns after the group's
        // S.  The K/V stage is free once both query tiles' PV are done.
        auto issue_pv = [&](int g, int acc0) {
            const uint64_t b0 = dv + static_cast<uint32_t>((g % NST) * kStage);
            if (pa::tc::elect_one()) {
#pragma unroll
                for (int ks = 0; ks < kT2KT / 16; ++ks) {
                    const uint64_t b = b0 + ((ks * 16 * 128) >> 4);
                    pa::tc::mma_ts(od, ph + ks * 8, b, kIdO, ks == 0 ? acc0 : 1);
                    pa::tc::mma_ts(od, pl + ks * 8, b, kIdO, 1);
                }
                pa::tc::commit(&o_done[wg]);
                pa::tc::commit(&kv_empty[g % NST]);
            }
            __syncwarp();
        };
        // Per item: S(0) once its query tiles are in; then per tile S(g+1)
        // and PV(g).  After the item's last S this query tile is released;
        // the item's first PV waits until the group has read the previous
        // item's O out of TMEM.
        bool ok = true;
        int g = 0, k;
        for (int it = 0; ok && next_item(it, &k); ++it) {
            const int nt = item_of(k).ntiles;
            ok = wait_all(q_full, it & 1) && wait_all(&kv_full[g % NST], (g / NST) & 1);
            if (!ok) break;
            pa::tc::fence_after();
            ok = issue_s(g);
            for (int j = 0; j < nt && ok; ++j, ++g) {
                if (j + 1 < nt) {
                    ok = wait_all(&kv_full[(g + 1) % NST], ((g + 1) / NST) & 1);
                    if (!ok) break;
                    pa::tc::fence_after();
                    ok = issue_s(g + 1);
                    if (!ok) break;
                } else {
                    if (pa::tc::elect_one()) pa::tc::commit(q_empty);
                    __syncwarp();
                }
                if (j == 0 && it > 0) ok = wait_all(&o_free[wg], (it - 1) & 1);
                if (ok) ok = wait_all(&p_full[wg], g & 1);
                if (!ok) break;
                pa::tc::fence_after();
                issue_pv(g, j > 0);
            }
        }
        if (!ok) *fail = 1;
    } else {
        // ---------------- softmax warp groups ----------------
        const int wg = warp >> 2;   // query tile A or B
        const int row = tid & 127;  // TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t o_col = wg * 128;
        const int m = wg * 128 + row;
        const float qs2 = p.qscale;  // softmax scale in log2 units
        // PV of CTA tile gg of this group done (one phase per tile; the next
        // phase needs this group's P of a later tile)
        auto pv_done = [&](int gg) { return pa::mbar_wait(&o_done[wg], gg & 1); };
        bool ok = true;
        int g = 0, k;
        for (int it = 0; ok && next_item(it, &k); ++it) {
            const Item I = item_of(k);
            const int pos = I.P + min(I.t0 + m / GQ, I.n - 1);  // last key this row sees
            float m_used = -INFINITY, lsum = 0.f;
            for (int j = 0; j < I.ntiles; ++j, ++g) {
                const uint32_t s_col = 256 + wg * 128, p_col = s_col + 64;
                ok = pa::mbar_wait(&s_full[wg], g & 1);
                if (!ok) break;
                pa::tc::fence_after();
                uint32_t sr[2][32];
                pa::tc::ld32(lane_base + s_col, sr[0]);
                pa::tc::ld32(lane_base + s_col + 32, sr[1]);
                pa::tc::wait_ld();
                // S may now be overwritten by the next tile's
                pa::tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[wg]);
                const int j0 = j * kT2KT;
                float s[64];
#pragma unroll
                for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
                if (j0 + kT2KT - 1 > pos) {  // tile on or past the diagonal: mask
#pragma unroll
                    for (int c = 0; c < 64; ++c)
                        if (j0 + c > pos) s[c] = -INFINITY;
                }
                float mx[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float m3 = max3f(s[e], s[8 + e], s[16 + e]);
                    m3 = max3f(m3, s[24 + e], s[32 + e]);
                    m3 = max3f(m3, s[40 + e], s[48 + e]);
                    mx[e] = fmaxf(m3, s[56 + e]);
                }
                const float tmax = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                                         fmaxf(mx[6], mx[7])) *
                                   qs2;
                float alpha = 1.f;
                if (tmax > m_used + kTcTau) {
                    alpha = (m_used == -INFINITY) ? 0.f : exp2f(m_used - tmax);
                    m_used = tmax;
                }
                uint32_t ph[32], pl[32];
                float2 rs2[4] = {};
                const float2 q2 = make_float2(qs2, qs2), nm2 = make_float2(-m_used, -m_used);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float2 x = pa::ffma2(make_float2(s[2 * c], s[2 * c + 1]), q2, nm2);
                    const float p0 = fast_exp2(x.x);
                    const float p1 = fast_exp2(x.y);
                    rs2[c & 3] = __fadd2_rn(rs2[c & 3], make_float2(p0, p1));
                    ph[c] = pack_bf16(p0, p1);
                    const float2 lo = pa::ffma2(pa::bf16x2_to_float2(ph[c]),
                                                make_float2(-1.f, -1.f), make_float2(p0, p1));
                    pl[c] = pack_bf16(lo.x, lo.y);
                }
                const float rs = ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y)) +
                                 ((rs2[2].x + rs2[2].y) + (rs2[3].x + rs2[3].y));
                lsum = lsum * alpha + rs;
                if (j > 0) {  // PV of the previous tile must be done before O is rescaled
                    ok = pv_done(g - 1);
                    if (!ok) break;
                    pa::tc::fence_after();
                    if (__any_sync(pa::kFull, alpha != 1.f)) {
#pragma unroll
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t o[32];
                            pa::tc::ld32(lane_base + o_col + c0, o);
                            pa::tc::wait_ld();
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                            pa::tc::st32(lane_base + o_col + c0, o);
                        }
                    }
                }
                if (j == I.ntiles - 1) {
                    // rows past the context in the last tile may hold anything
                    // (unwritten slots); P is 0 there but 0 * NaN is NaN: zero
                    // them.  Each group does so before its own P arrival (its
                    // PV may run before the other group's); both write zeros.
                    const int first = I.kv_end - j0;
                    const uint32_t vst = skv + (g % NST) * 2 * Lay::T_BYTES + Lay::T_BYTES;
                    for (int idx = row; idx < (kT2KT - first) * CH; idx += 128) {
                        const int rr = first + idx / CH, c = idx % CH;
                        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                                         vst + pa::tc::sw128(rr, c * 8, kT2KT)),
                                     "r"(0u)
                                     : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                pa::tc::st32(lane_base + p_col, ph);
                pa::tc::st32(lane_base + p_col + 32, pl);
                pa::tc::wait_st();
                pa::tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[wg]);
            }
            if (!ok) break;
            ok = pv_done(g - 1);  // PV of the item's last tile
            if (!ok) break;
            pa::tc::fence_after();
            const int t = I.t0 + m / GQ;
            const float inv = 1.f / lsum;
            __nv_bfloat16 *dst =
                p.out + (static_cast<size_t>(I.qs + min(t, I.n - 1)) * p.Hq + I.hk * GQ + m % GQ) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 64) {  // two TMEM loads per wait
                uint32_t o[2][32];
                pa::tc::ld32(lane_base + o_col + c0, o[0]);
                pa::tc::ld32(lane_base + o_col + c0 + 32, o[1]);
                pa::tc::wait_ld();
                if (t < I.n) {
#pragma unroll
                    for (int c = 0; c < 64; c += 8) {
                        const uint32_t *oc = &o[c >> 5][c & 31];
                        uint4 w4;
                        w4.x = pack_bf16(__uint_as_float(oc[0]) * inv, __uint_as_float(oc[1]) * inv);
                        w4.y = pack_bf16(__uint_as_float(oc[2]) * inv, __uint_as_float(oc[3]) * inv);
                        w4.z = pack_bf16(__uint_as_float(oc[4]) * inv, __uint_as_float(oc[5]) * inv);
                        w4.w = pack_bf16(__uint_as_float(oc[6]) * inv, __uint_as_float(oc[7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + c0 + c) = w4;
                    }
                }
            }
            // O of this group may be overwritten once every warp has read it
            pa::tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[wg]);
        }
        if (!ok) *fail = 1;
    }

    // ---- tear-down ----------------------------------------------------------------
    pa::tc::fence_before();
    __syncthreads();
    if (*fail) {
        // a wait ran out: record it, then let the MMAs and the K/V copies in
        // flight land (bounded) before TMEM and shared memory go away
        if (tid == 0) pa::record_error(p.err, PA_DEVERR_TIMEOUT);
        if (warp == Lay::MMA_WARP || warp == Lay::MMA_WARP_B) {
            if (pa::tc::elect_one()) pa::tc::commit(drain);
            __syncwarp();
            (void)pa::mbar_wait(drain, 0);
        }
        if (warp == Lay::LOAD_WARP && lane == 0) {
            // the last tile issued into each stage
            for (int st = 0; st < NST && st < loads_issued; ++st) {
                const int g_last = st + NST * ((loads_issued - 1 - st) / NST);
                (void)pa::mbar_wait(&kv_full[st], (g_last / NST) & 1);
            }
        }
        pa::tc::fence_before();
        __syncthreads();
    }
    if (warp == Lay::MMA_WARP) {
        pa::tc::fence_after();
        pa::tc::dealloc(tmem, Lay::TMEM_COLS);
    }
}

int sm_count_cached() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

template <int D, int GQ>
int launch_persist_t(const PrefillParams &p, cudaStream_t stream) {
    const int64_t rows = (p.num_blocks * p.Hkv) << p.bs_log2;
    CUtensorMap kmap, vmap, qmap_tile, qmap_row8;
    if (int rc = pa::pool_tensor_map(&kmap, p.k_cache, rows, D, p.bs)) return rc;
    if (int rc = pa::pool_tensor_map(&vmap, p.v_cache, rows, D, p.bs)) return rc;
    // R * max_query_len bounds the number of query tokens; the kernel copies
    // only boxes that lie inside a request's new tokens
    const int64_t qtokens = int64_t(p.R) * p.max_query_len;
    if (int rc = pa::q_tensor_map(&qmap_tile, p.q, qtokens, p.Hq, D, GQ, 128 / GQ)) return rc;
    if (int rc = pa::q_tensor_map(&qmap_row8, p.q, qtokens, p.Hq, D, GQ, 8 / GQ)) return rc;
    using Lay = PLayout<D>;
    auto kern = prefill_persist_kernel<D, GQ>;
    static std::atomic<uint64_t> attr_done{0};
    if (int rc = set_smem_once(kern, Lay::SMEM, &attr_done)) return rc;
    constexpr int qtok = 256 / GQ;
    const int items = (p.max_query_len + qtok - 1) / qtok * p.R * p.Hkv;
    const int sms = sm_count_cached();
    if (sms <= 0) return pa::fail(PA_ERR_CUDA, "prefill: SM count");
    const int grid = std::min(std::min(sms, items), kPCtasMax);
    (void)cudaGetLastError();
    // a programmatic dependent of the previous kernel in the stream: the
    // set-up above griddepcontrol.wait overlaps that kernel's tail
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Lay::THREADS);
    cfg.dynamicSmemBytes = Lay::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PA_PERSIST_PDL ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p, kmap, vmap, qmap_tile, qmap_row8);
    if (e != cudaSuccess) return pa::cuda_fail(e, "prefill launch");
    return pa::check_launch("prefill launch");
}

}  // namespace

namespace pa {
namespace pf {

bool persist_ok(int R, int max_query_len, int Hq, int Hkv) {
    const int qtok = 256 / (Hq / Hkv);
    const int64_t pairs = int64_t(R) * ((max_query_len + qtok - 1) / qtok);
    return pairs <= kPPairsMax && pairs * Hkv <= kPItemsMax;
}

int launch_persist(const PrefillParams &p, int D, int gq, cudaStream_t stream) {
    auto pick = [&](auto d) -> int {
        constexpr int DD = decltype(d)::value;
        switch (gq) {
            case 1: return launch_persist_t<DD, 1>(p, stream);
            case 2: return launch_persist_t<DD, 2>(p, stream);
            case 4: return launch_persist_t<DD, 4>(p, stream);
            case 8: return launch_persist_t<DD, 8>(p, stream);
            default: return pa::fail(PA_ERR_UNSUPPORTED, "prefill: Hq/Hkv=%d unsupported", gq);
        }
    };
    if (D == 128) return pick(std::integral_constant<int, 128>{});
    if (D == 64) return pick(std::integral_constant<int, 64>{});
    return pa::fail(PA_ERR_UNSUPPORTED, "prefill: head_dim %d unsupported", D);
}

}  // namespace pf
}  // namespace pa
