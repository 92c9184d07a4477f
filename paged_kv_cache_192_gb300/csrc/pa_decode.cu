// Paged decode attention for sm_103a.
//
// What it computes: for each sequence b and query head h, attention of the
// one new query over the L_b cached tokens, which are reached through the
// block table (logical block i -> physical block) before K and V are loaded
// ("PagedAttention: memetakan blok KV logis ke memori fisik tidak kontigu",
// section "Kernel attention harus mengikuti block table"); the attention
// equation is the ordinary one (same page, opening section).
//
// How (decode is HBM-bound: "Melihat Lebih Dalam vLLM v0.7", section
// "Blueprint Arsitektur 3", the decode phase is memory-bandwidth intensive):
//  * One CTA of kWarps warps per work item (sequence b, KV head, partition of
//    PT tokens).  Partitions are merged by log-sum-exp in a second kernel
//    when a sequence spans more than one (split-KV).
//  * Each warp takes every kWarps-th tile of TT tokens of the partition and
//    streams it through its own ring of NST shared-memory stages.  One lane
//    issues a bulk copy (cp.async.bulk, non-tensor TMA) per contiguous
//    (block, KV head) piece of K and of V, completing on an mbarrier.
//  * All GQ query heads of a KV head share one K/V load.  A token row is split
//    over G lanes in 16-byte chunks (conflict-free shared loads); QK partial
//    dots of the S steps x GQ heads are reduced across the G lanes by a
//    transpose-reduce (each round halves the values a lane carries), which
//    leaves every (token, head) score in exactly one lane.
//  * Online softmax in the log2 domain (q pre-scaled by scale*log2(e)) with a
//    lazy rescale: the running max only moves when a score exceeds it by more
//    than kTau; the result is exact whatever max is used.
//  * PV accumulates in fp32 with packed fp32 FMAs; the partial sums of the
//    token groups, then of the warps, are combined in a fixed order, so the
//    result depends only on the logical token order, never on the physical
//    placement of blocks.
#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

constexpr int kWarps = 4;              // warps per CTA
constexpr int kRingBytes = 16 * 1024;  // per-warp K+V staging ring
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.0f;           // lazy-rescale headroom (log2 units)
constexpr int kDefaultPartition = 512;
constexpr int kMaxPartition = 8192;

template <typename T, int D, int GQ>
struct Cfg {
    static constexpr int ES = sizeof(T);
    static constexpr int ROW = D * ES;       // bytes of one token row of one KV head
    static constexpr int CHUNKS = ROW / 16;  // 16-byte chunks per row
    static constexpr int G0 = GQ >= 8 ? 16 : 8;
    static constexpr int G = G0 < CHUNKS ? G0 : CHUNKS;  // lanes per token
    static constexpr int CPL = CHUNKS / G;               // chunks per lane
    static constexpr int EPC = 16 / ES;                  // elements per chunk
    static constexpr int E = CPL * EPC;                  // elements per lane
    static constexpr int P = E / 2;                      // float2 pairs per lane
    static constexpr int TPS = 32 / G;                   // tokens per step
    static constexpr int SMIN = (G + GQ - 1) / GQ;
    static constexpr int S = SMIN > 4 ? SMIN : 4;        // steps per tile
    static constexpr int TT = S * TPS;                   // tokens per tile
    static constexpr int V = S * GQ;                     // partial dots per lane
    static constexpr int VPL = V / G;                    // scores per lane after reduction
    static constexpr int TILE = TT * ROW;                // bytes per tile per cache
    static constexpr int STAGE = 2 * TILE;               // K then V
    // stages per warp: as many as fit the ring, at least 2 when 2 fit in
    // 160 KB per CTA, else 1 (the warp then refills a stage after using it)
    static constexpr int NST = kRingBytes / STAGE >= 2 ? kRingBytes / STAGE
                               : (kWarps * 2 * STAGE <= 160 * 1024 ? 2 : 1);
    static constexpr int WARP_SMEM = NST * STAGE;
    static constexpr int OFF_P = kWarps * WARP_SMEM;                  // p and score buffers
    static constexpr int OFF_BAR = OFF_P + kWarps * 2 * TT * GQ * 4;  // mbarriers
    static constexpr int OFF_FLAG = OFF_BAR + kWarps * NST * 8;       // failure flag
    static constexpr int OFF_BT = OFF_FLAG + 16;                      // block-table slice
    static_assert(G * CPL == CHUNKS, "row must split evenly over the lanes of a token");
    static_assert(V % G == 0 && VPL <= GQ && GQ % VPL == 0, "bad reduction shape");
    static_assert(E % 2 == 0 && TT <= 32, "bad tile");
    static_assert(GQ * D * 4 + 2 * GQ * 4 <= WARP_SMEM, "merge buffer must fit the ring");
};

struct DecodeParams {
    void *out;
    const void *q;
    const uint8_t *k_cache;
    const uint8_t *v_cache;
    const int32_t *block_table;
    const int32_t *context_lens;
    float *ws_acc;  // [B][Hq][max_parts][D]
    float *ws_ml;   // [B][Hq][max_parts][2] (max, sum)
    int *err;
    int64_t num_blocks;
    int B, Hq, Hkv, bs, bs_log2, MB, PT, max_parts;
    float qscale;  // scale * log2(e)
};

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Reduce V per-lane partial sums across the G lanes of a token group so that
// lane gl ends with the totals of indices [gl*V/G, (gl+1)*V/G) in v[0..V/G).
template <int V, int G>
__device__ __forceinline__ void transpose_reduce(float (&v)[V], int lane) {
#pragma unroll
    for (int m = G / 2; m >= 1; m /= 2) {
        const int half = V * m / G;
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = upper ? v[k] : v[k + half];
            const float keep = upper ? v[k + half] : v[k];
            v[k] = keep + __shfl_xor_sync(pa::kFull, send, m);
        }
    }
}

template <typename T, int D, int GQ>
__global__ void __launch_bounds__(kWarps * 32, 3) decode_kernel(const DecodeParams p) {
    using C = Cfg<T, D, GQ>;
    extern __shared__ __align__(128) uint8_t smem[];

    const int part = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int cap = p.MB << p.bs_log2;
    int L = p.context_lens[b];
    if (L > cap || L < 0) {
        if (threadIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
        L = L < 0 ? 0 : cap;
    }
    const int nparts = (L + p.PT - 1) / p.PT;
    if (part >= nparts) return;  // uniform over the CTA
    const int tok0 = part * p.PT;
    const int ntok = min(L - tok0, p.PT);
    const int ntiles = (ntok + C::TT - 1) / C::TT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gl = lane % C::G, grp = lane / C::G;

    uint8_t *ring = smem + warp * C::WARP_SMEM;
    float *pbuf = reinterpret_cast<float *>(smem + C::OFF_P) + warp * 2 * C::TT * GQ;
    float *sbuf = pbuf + C::TT * GQ;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR) + warp * C::NST;
    volatile int *fail_flag = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
    int32_t *btab = reinterpret_cast<int32_t *>(smem + C::OFF_BT);

    // Block-table slice of this partition -> shared memory (bad ids recorded
    // and replaced by block 0 so that no load leaves the pool).
    const int blk0 = tok0 >> p.bs_log2;
    const int nblk = (ntok + p.bs - 1) >> p.bs_log2;
    const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.MB + blk0;
    for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
        int v = bt_row[i];
        if (v < 0 || v >= p.num_blocks) {
            pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            v = 0;
        }
        btab[i] = v;
    }
    if (threadIdx.x == 0) *fail_flag = 0;
    if (lane == 0) {
        for (int s = 0; s < C::NST; ++s) pa::mbar_init(&bars[s], 1);
        pa::fence_barrier_init();
    }
    __syncthreads();

    const int my_ntiles = ntiles > warp ? (ntiles - 1 - warp) / kWarps + 1 : 0;

    // Producer (lane 0): bulk-copy the K and V rows of this warp's i-th tile.
    auto issue = [&](int i) {
        const int rel = (warp + i * kWarps) * C::TT;  // first token, relative to tok0
        uint8_t *dk = ring + (i % C::NST) * C::STAGE;
        uint8_t *dv = dk + C::TILE;
        uint64_t *bar = &bars[i % C::NST];
        if (C::TT <= p.bs) {
            const int bi = rel >> p.bs_log2;
            const int r0 = rel & (p.bs - 1);
            const size_t off =
                ((static_cast<size_t>(btab[bi]) * p.Hkv + hk) * p.bs + r0) * C::ROW;
            pa::mbar_arrive_expect_tx(bar, 2 * C::TILE);
            pa::bulk_g2s(dk, p.k_cache + off, C::TILE, bar);
            pa::bulk_g2s(dv, p.v_cache + off, C::TILE, bar);
        } else {
            const int per = C::TT >> p.bs_log2;  // blocks per tile
            const uint32_t bytes = static_cast<uint32_t>(p.bs) * C::ROW;
            int avail = 0;
            for (int j = 0; j < per; ++j) avail += (rel + j * p.bs < ntok) ? 1 : 0;
            pa::mbar_arrive_expect_tx(bar, 2u * avail * bytes);
            for (int j = 0; j < avail; ++j) {
                const int bi = (rel >> p.bs_log2) + j;
                const size_t off = (static_cast<size_t>(btab[bi]) * p.Hkv + hk) * p.bs * C::ROW;
                pa::bulk_g2s(dk + j * bytes, p.k_cache + off, bytes, bar);
                pa::bulk_g2s(dv + j * bytes, p.v_cache + off, bytes, bar);
            }
        }
    };

    // q of the GQ heads of this KV head, this lane's elements, pre-scaled.
    float2 q2[GQ][C::P];
    {
        const T *qb = static_cast<const T *>(p.q) + (static_cast<size_t>(b) * p.Hq + hk * GQ) * D;
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(
                    qb + h * D + (c * C::G + gl) * C::EPC);
                float2 f[C::EPC / 2];
                pa::Elem<T>::unpack(raw, f);
#pragma unroll
                for (int i = 0; i < C::EPC / 2; ++i)
                    q2[h][c * C::EPC / 2 + i] =
                        make_float2(f[i].x * p.qscale, f[i].y * p.qscale);
            }
    }

    if (lane == 0)
        for (int i = 0; i < min(C::NST, my_ntiles); ++i) issue(i);

    float m_run[GQ];
    float2 acc[GQ][C::P];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        m_run[h] = -INFINITY;
#pragma unroll
        for (int j = 0; j < C::P; ++j) acc[h][j] = make_float2(0.f, 0.f);
    }
    // After the transpose-reduce this lane holds the scores of step s_mine,
    // heads h0 .. h0+VPL-1, i.e. token row row_mine of the tile.
    const int h0 = (gl * C::VPL) % GQ;
    const int row_mine = ((gl * C::VPL) / GQ) * C::TPS + grp;
    float lsum[C::VPL], mh[C::VPL];
#pragma unroll
    for (int k = 0; k < C::VPL; ++k) {
        lsum[k] = 0.f;
        mh[k] = -INFINITY;
    }

    int failed_at = -1;
    for (int i = 0; i < my_ntiles; ++i) {
        const int st = i % C::NST;
        const bool ok = __all_sync(pa::kFull, pa::mbar_wait(&bars[st], (i / C::NST) & 1));
        if (!ok) {
            failed_at = i;
            break;
        }
        const int nvalid = min(C::TT, ntok - (warp + i * kWarps) * C::TT);
        const uint32_t kaddr = pa::smem_u32(ring + st * C::STAGE);
        const uint32_t vaddr = kaddr + C::TILE;
        const bool masked = nvalid < C::TT;

        // ---- QK: partial dots of S token rows x GQ heads -----------------
        float part_[C::V];
#pragma unroll
        for (int s = 0; s < C::S; ++s) {
            const int row = s * C::TPS + grp;
            float2 kf[C::P];
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
                const uint4 raw = pa::lds128(kaddr + row * C::ROW + (c * C::G + gl) * 16);
                float2 f[C::EPC / 2];
                pa::Elem<T>::unpack(raw, f);
#pragma unroll
                for (int j = 0; j < C::EPC / 2; ++j) kf[c * C::EPC / 2 + j] = f[j];
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                float2 a = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < C::P; ++j) a = pa::ffma2(q2[h][j], kf[j], a);
                part_[s * GQ + h] = a.x + a.y;
            }
        }
        transpose_reduce<C::V, C::G>(part_, lane);

        float sc[C::VPL];
        const bool row_valid = row_mine < nvalid;
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) sc[k] = row_valid ? part_[k] : -INFINITY;

        // ---- online softmax with lazy rescale -------------------------------
        bool need = false;
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) need |= sc[k] > mh[k] + kTau;
        if (__any_sync(pa::kFull, need)) {
#pragma unroll
            for (int k = 0; k < C::VPL; ++k) sbuf[row_mine * GQ + h0 + k] = sc[k];
            __syncwarp();
            const int hh = lane % GQ;
            float tmax = -INFINITY;
            for (int r = 0; r < C::TT; ++r) tmax = fmaxf(tmax, sbuf[r * GQ + hh]);
            float mold = m_run[0];
#pragma unroll
            for (int h = 1; h < GQ; ++h) mold = (hh == h) ? m_run[h] : mold;
            const float mnew_l = fmaxf(mold, tmax);
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float mnew = __shfl_sync(pa::kFull, mnew_l, h);
                const float alpha = (m_run[h] == -INFINITY) ? 0.f : exp2f(m_run[h] - mnew);
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int j = 0; j < C::P; ++j) acc[h][j] = __fmul2_rn(acc[h][j], a2);
#pragma unroll
                for (int k = 0; k < C::VPL; ++k)
                    if (h == h0 + k) lsum[k] *= alpha;
                m_run[h] = mnew;
            }
#pragma unroll
            for (int k = 0; k < C::VPL; ++k) {
                float m = m_run[0];
#pragma unroll
                for (int h = 1; h < GQ; ++h) m = (h == h0 + k) ? m_run[h] : m;
                mh[k] = m;
            }
            __syncwarp();
        }
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) {
            const float pk = fast_exp2(sc[k] - mh[k]);
            lsum[k] += pk;
            pbuf[row_mine * GQ + h0 + k] = pk;
        }
        __syncwarp();

        // ---- PV ---------------------------------------------------------------
#pragma unroll
        for (int s = 0; s < C::S; ++s) {
            const int row = s * C::TPS + grp;
            float prow[GQ];
            if constexpr (GQ % 4 == 0) {
#pragma unroll
                for (int h = 0; h < GQ; h += 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(pbuf + row * GQ + h);
                    prow[h] = t4.x;
                    prow[h + 1] = t4.y;
                    prow[h + 2] = t4.z;
                    prow[h + 3] = t4.w;
                }
            } else {
#pragma unroll
                for (int h = 0; h < GQ; ++h) prow[h] = pbuf[row * GQ + h];
            }
            float2 vf[C::P];
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
                const uint4 raw = pa::lds128(vaddr + row * C::ROW + (c * C::G + gl) * 16);
                float2 f[C::EPC / 2];
                pa::Elem<T>::unpack(raw, f);
#pragma unroll
                for (int j = 0; j < C::EPC / 2; ++j) vf[c * C::EPC / 2 + j] = f[j];
            }
            if (masked && row >= nvalid) {
                // p is 0 there, but the stale row may hold NaN: 0 * NaN = NaN
#pragma unroll
                for (int j = 0; j < C::P; ++j) vf[j] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float2 pp = make_float2(prow[h], prow[h]);
#pragma unroll
                for (int j = 0; j < C::P; ++j) acc[h][j] = pa::ffma2(pp, vf[j], acc[h][j]);
            }
        }
        __syncwarp();
        if (lane == 0 && i + C::NST < my_ntiles) {
            pa::fence_proxy_async();
            issue(i + C::NST);
        }
    }

    if (failed_at >= 0) {
        // A copy never completed: record it, wait (bounded) for this warp's
        // other copies in flight so none lands after the CTA exits, and
        // write nothing.
        if (lane == 0) {
            pa::record_error(p.err, PA_DEVERR_TIMEOUT);
            *fail_flag = 1;
            const int last = min(failed_at + C::NST, my_ntiles);
            for (int i = failed_at + 1; i < last; ++i)
                (void)pa::mbar_wait(&bars[i % C::NST], (i / C::NST) & 1);
        }
        __syncwarp();
    }

    // ---- warp epilogue: sum over token groups, l per head ---------------------
#pragma unroll
    for (int off = C::G; off < 32; off <<= 1)
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int j = 0; j < C::P; ++j) {
                acc[h][j].x += __shfl_xor_sync(pa::kFull, acc[h][j].x, off);
                acc[h][j].y += __shfl_xor_sync(pa::kFull, acc[h][j].y, off);
            }
    float lh[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) t += (h == h0 + k) ? lsum[k] : 0.f;
        lh[h] = t;
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
#pragma unroll
        for (int h = 0; h < GQ; ++h) lh[h] += __shfl_xor_sync(pa::kFull, lh[h], off);

    // ---- CTA merge of the warps' (max, sum, acc) ----------------------------
    __syncthreads();  // every ring is drained: reuse it as the merge buffer
    float *wacc = reinterpret_cast<float *>(ring);  // [GQ][D]
    float *wml = wacc + GQ * D;                     // max[GQ], sum[GQ]
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int c = 0; c < C::CPL; ++c)
#pragma unroll
                for (int j = 0; j < C::EPC / 2; ++j) {
                    const int dim = (c * C::G + gl) * C::EPC + 2 * j;
                    *reinterpret_cast<float2 *>(wacc + h * D + dim) = acc[h][c * C::EPC / 2 + j];
                }
    }
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            wml[h] = m_run[h];
            wml[GQ + h] = lh[h];
        }
    __syncthreads();
    if (*fail_flag) return;

    T *out = static_cast<T *>(p.out);
    for (int idx = threadIdx.x; idx < GQ * D; idx += blockDim.x) {
        const int h = idx / D, dim = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *ml = reinterpret_cast<const float *>(smem + w * C::WARP_SMEM) + GQ * D;
            M = fmaxf(M, ml[h]);
        }
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *wa = reinterpret_cast<const float *>(smem + w * C::WARP_SMEM);
            const float mw = wa[GQ * D + h];
            if (mw == -INFINITY) continue;
            const float f = exp2f(mw - M);
            num += f * wa[h * D + dim];
            den += f * wa[GQ * D + GQ + h];
        }
        const int hq = hk * GQ + h;
        if (nparts == 1) {
            pa::Elem<T>::store(out + (static_cast<size_t>(b) * p.Hq + hq) * D + dim, num / den);
        } else {
            const size_t slot = (static_cast<size_t>(b) * p.Hq + hq) * p.max_parts + part;
            p.ws_acc[slot * D + dim] = num;
            if (dim == 0) {
                p.ws_ml[2 * slot] = M;
                p.ws_ml[2 * slot + 1] = den;
            }
        }
    }
}

// Log-sum-exp merge of the partitions of one (sequence, query head).
template <typename T, int D>
__global__ void __launch_bounds__(D) merge_kernel(const DecodeParams p) {
    const int hq = blockIdx.x, b = blockIdx.y;
    const int cap = p.MB << p.bs_log2;
    int L = p.context_lens[b];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int nparts = (L + p.PT - 1) / p.PT;
    if (nparts <= 1) return;
    const size_t base = (static_cast<size_t>(b) * p.Hq + hq) * p.max_parts;
    float M = -INFINITY;
    for (int i = 0; i < nparts; ++i) M = fmaxf(M, p.ws_ml[2 * (base + i)]);
    const int dim = threadIdx.x;
    float num = 0.f, den = 0.f;
    for (int i = 0; i < nparts; ++i) {
        const float f = exp2f(p.ws_ml[2 * (base + i)] - M);
        num += f * p.ws_acc[(base + i) * D + dim];
        den += f * p.ws_ml[2 * (base + i) + 1];
    }
    pa::Elem<T>::store(static_cast<T *>(p.out) + (static_cast<size_t>(b) * p.Hq + hq) * D + dim,
                       num / den);
}

int log2_int(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

int resolve_partition(int partition_tokens) {
    return partition_tokens == 0 ? kDefaultPartition : partition_tokens;
}

bool partition_ok(int pt, int bs) {
    return pt > 0 && pt <= kMaxPartition && pt % 32 == 0 && pt % bs == 0;
}

template <typename T, int D, int GQ>
int launch(const DecodeParams &p, cudaStream_t stream) {
    using C = Cfg<T, D, GQ>;
    const size_t smem = C::OFF_BT + sizeof(int32_t) * (p.PT / p.bs + 1);
    auto kern = decode_kernel<T, D, GQ>;
    (void)cudaGetLastError();  // drop a stale error that is not ours
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode: shared memory attribute");
    dim3 grid(p.max_parts, p.Hkv, p.B);
    kern<<<grid, kWarps * 32, smem, stream>>>(p);
    if (int rc = pa::check_launch("decode launch")) return rc;
    if (p.max_parts > 1) {
        merge_kernel<T, D><<<dim3(p.Hq, p.B), D, 0, stream>>>(p);
        if (int rc = pa::check_launch("decode merge launch")) return rc;
    }
    return PA_OK;
}

template <typename T, int D>
int dispatch_gq(int gq, const DecodeParams &p, cudaStream_t s) {
    switch (gq) {
        case 1: return launch<T, D, 1>(p, s);
        case 2: return launch<T, D, 2>(p, s);
        case 4: return launch<T, D, 4>(p, s);
        case 8: return launch<T, D, 8>(p, s);
        default: return pa::fail(PA_ERR_UNSUPPORTED, "decode: Hq/Hkv=%d unsupported", gq);
    }
}

size_t workspace_bytes_for(int B, int Hq, int D, int max_parts) {
    if (max_parts <= 1) return 0;
    return static_cast<size_t>(B) * Hq * max_parts * (D + 2) * sizeof(float);
}

}  // namespace

extern "C" {

int pa_decode_workspace_size(int B, int Hq, int head_dim, int max_blocks_per_seq, int block_size,
                             int partition_tokens, size_t *bytes) {
    pa::clear_error();
    if (!bytes) return pa::fail(PA_ERR_INVALID, "workspace_size: bytes is NULL");
    if (B < 0 || Hq <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 ||
        !pa::pow2_in(block_size, 8, 128))
        return pa::fail(PA_ERR_INVALID, "workspace_size: bad sizes");
    const int pt = resolve_partition(partition_tokens);
    if (!partition_ok(pt, block_size))
        return pa::fail(PA_ERR_INVALID, "workspace_size: bad partition_tokens %d", pt);
    const int64_t cap = int64_t(max_blocks_per_seq) * block_size;
    const int max_parts = static_cast<int>((cap + pt - 1) / pt);
    *bytes = workspace_bytes_for(B, Hq, head_dim, max_parts);
    return PA_OK;
}

int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, int max_blocks_per_seq, const int32_t *context_lens,
              int B, int Hq, int Hkv, int head_dim, int block_size, int64_t num_blocks,
              float scale, int partition_tokens, void *workspace, size_t workspace_bytes,
              int dtype, pa_stream_t stream) {
    pa::clear_error();
    if (dtype != PA_BF16 && dtype != PA_F32) return pa::fail(PA_ERR_INVALID, "decode: bad dtype");
    if (B < 0 || B > 65535 || Hq <= 0 || Hkv <= 0 || Hkv > 65535 || Hq % Hkv || num_blocks <= 0 ||
        max_blocks_per_seq <= 0)
        return pa::fail(PA_ERR_INVALID, "decode: bad sizes");
    if (head_dim != 64 && head_dim != 128)
        return pa::fail(PA_ERR_UNSUPPORTED, "decode: head_dim %d unsupported", head_dim);
    if (Hq / Hkv != 1 && Hq / Hkv != 2 && Hq / Hkv != 4 && Hq / Hkv != 8)
        return pa::fail(PA_ERR_UNSUPPORTED, "decode: Hq/Hkv=%d unsupported", Hq / Hkv);
    if (!pa::pow2_in(block_size, 8, 128))
        return pa::fail(PA_ERR_UNSUPPORTED, "decode: block_size %d unsupported", block_size);
    if (int64_t(max_blocks_per_seq) * block_size > (int64_t(1) << 30))
        return pa::fail(PA_ERR_INVALID, "decode: table capacity too large");
    const int pt = resolve_partition(partition_tokens);
    if (!partition_ok(pt, block_size))
        return pa::fail(PA_ERR_INVALID,
                        "decode: partition_tokens %d must be a multiple of 32 and of block_size "
                        "and at most %d",
                        pt, kMaxPartition);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return pa::fail(PA_ERR_INVALID, "decode: scale must be positive and finite");
    if (B == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !context_lens)
        return pa::fail(PA_ERR_INVALID, "decode: NULL pointer");
    if (!pa::aligned16(q) || !pa::aligned16(k_cache) || !pa::aligned16(v_cache))
        return pa::fail(PA_ERR_INVALID, "decode: q and pools must be 16-byte aligned");
    const int64_t cap = int64_t(max_blocks_per_seq) * block_size;
    const int max_parts = static_cast<int>((cap + pt - 1) / pt);
    const size_t need = workspace_bytes_for(B, Hq, head_dim, max_parts);
    if (need > workspace_bytes || (need && !workspace))
        return pa::fail(PA_ERR_INVALID, "decode: workspace needs %zu bytes, got %zu", need,
                        workspace_bytes);
    if (need && !pa::aligned16(workspace))
        return pa::fail(PA_ERR_INVALID, "decode: workspace must be 16-byte aligned");
    if (pa::validate_on()) {
        std::vector<int32_t> lens(B), table(size_t(B) * max_blocks_per_seq);
        if (int rc = pa::fetch(lens.data(), context_lens, B * sizeof(int32_t), stream)) return rc;
        if (int rc = pa::fetch(table.data(), block_table, table.size() * sizeof(int32_t), stream))
            return rc;
        for (int b = 0; b < B; ++b) {
            if (lens[b] < 1 || lens[b] > cap)
                return pa::fail(PA_ERR_INVALID, "validate: context_lens[%d]=%d outside [1,%lld]", b,
                                lens[b], (long long)cap);
            const int nb = (lens[b] + block_size - 1) / block_size;
            for (int i = 0; i < nb; ++i) {
                const int32_t v = table[size_t(b) * max_blocks_per_seq + i];
                if (v < 0 || v >= num_blocks)
                    return pa::fail(PA_ERR_INVALID, "validate: block_table[%d][%d]=%d outside pool",
                                    b, i, v);
            }
        }
    }
    DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_cache = static_cast<const uint8_t *>(k_cache);
    p.v_cache = static_cast<const uint8_t *>(v_cache);
    p.block_table = block_table;
    p.context_lens = context_lens;
    p.ws_acc = static_cast<float *>(workspace);
    p.ws_ml = need ? p.ws_acc + size_t(B) * Hq * max_parts * head_dim : nullptr;
    p.err = pa::device_error_word();
    p.num_blocks = num_blocks;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.bs = block_size;
    p.bs_log2 = log2_int(block_size);
    p.MB = max_blocks_per_seq;
    p.PT = pt;
    p.max_parts = max_parts;
    p.qscale = scale * kLog2e;
    const int gq = Hq / Hkv;
    if (dtype == PA_BF16)
        return head_dim == 128 ? dispatch_gq<__nv_bfloat16, 128>(gq, p, stream)
                               : dispatch_gq<__nv_bfloat16, 64>(gq, p, stream);
    return head_dim == 128 ? dispatch_gq<float, 128>(gq, p, stream)
                           : dispatch_gq<float, 64>(gq, p, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of pa_decode.
//
// Some callers cannot allocate device memory: a plug-in whose host program
// owns every device allocation through its own pool, or a latency-critical
// loop where cudaMalloc (which can synchronize the device) is not allowed.
// pa_decode_noalloc takes the split-KV workspace from a fixed array that the
// library itself holds in device memory, so such a caller passes only inputs
// and outputs.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes; every
// GPU that loads the library keeps it until the process exits.  Host code may
// not use the array's name as a device address, so the first call on each
// device (with that device current) looks up its address with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls on a device share the array and it keeps the contents
// of the last call; nothing in it needs to start at zero (every partial is
// written before it is read in the same call).  Calls that overlap on the GPU
// (different streams, or host threads racing) race on the array: serialize
// them.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};
std::mutex g_noalloc_mu;

// Device address of this device's scratch array (looked up once per device).
int noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return pa::fail(PA_ERR_UNSUPPORTED, "decode_noalloc: device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return pa::cuda_fail(e, "decode_noalloc: cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" {

size_t pa_decode_noalloc_capacity(void) { return kNoAllocScratchBytes; }

int pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_table, int max_blocks_per_seq,
                      const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                      int block_size, int64_t num_blocks, float scale, int partition_tokens,
                      int dtype, pa_stream_t stream) {
    pa::clear_error();
    size_t need = 0;
    if (int rc = pa_decode_workspace_size(B, Hq, head_dim, max_blocks_per_seq, block_size,
                                          partition_tokens, &need))
        return rc;
    if (need > kNoAllocScratchBytes)
        return pa::fail(PA_ERR_INVALID,
                        "decode_noalloc: this batch needs %zu bytes of split-KV workspace, more "
                        "than the library's fixed %zu-byte scratch; use pa_decode with a caller "
                        "workspace, fewer sequences or longer partitions",
                        need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if (need) {
        if (int rc = noalloc_scratch(&scratch)) return rc;
    }
    return pa_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, B,
                     Hq, Hkv, head_dim, block_size, num_blocks, scale, partition_tokens, scratch,
                     need ? kNoAllocScratchBytes : 0, dtype, stream);
}

}  // extern "C"
