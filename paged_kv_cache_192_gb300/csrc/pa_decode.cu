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
//  * Work unit: one tile of TT tokens of one (sequence, KV head) item.  All
//    GQ query heads of a KV head share one K/V load.
//  * Default kernel (decode_persistent_kernel): a persistent grid of 2 CTAs
//    of 4 warps per SM; every warp owns an equal, contiguous range of units across all
//    items (perfect balance) and streams its tiles through its own ring of NST
//    shared-memory stages.  One lane issues the copies of a tile, completing
//    on an mbarrier: a bulk copy (cp.async.bulk, non-tensor TMA) per
//    contiguous (block, KV head) piece, or 2D tensor copies with the 128-byte
//    swizzle for the tensor-core tile; the block-table entry of the next tile
//    is loaded one tile ahead.  When a warp's range ends inside an item, the
//    item's ranges (segments) write partial (max, sum, acc) to the workspace
//    and partial_merge_kernel, a programmatic dependent launch, merges them
//    by log-sum-exp (with the shared-prefix partials of pa_decode_shared).
//  * Grid kernel for very large batches and for batches of little work
//    (decode_kernel): one CTA per (sequence, KV head, partition), merged by
//    merge_kernel, a programmatic dependent launch.
//  * Per tile, tensor-core tile (bf16, groups of 4 or 8 heads): see MmaAttn.
//  * Per tile, CUDA-core tile: a token row is split over G lanes in 16-byte chunks
//    (conflict-free shared loads); QK partial dots of S steps x GQ heads are
//    reduced across the G lanes by a transpose-reduce (each round halves the
//    values a lane carries), leaving each (token, head) score in one lane;
//    online softmax in the log2 domain (q pre-scaled by scale*log2(e)) with a
//    lazy rescale (the running max moves only when a score exceeds it by more
//    than kTau; exact whatever max is used); PV with packed fp32 FMAs.
//  * Every sum runs in an order fixed by logical token positions and the
//    batch's lengths, never by where blocks sit in the pool.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

// Tuning knobs (compile-time): CTAs per SM the register budget targets, the
// per-warp staging ring, and lanes per token row for groups of <= 4 heads.
#ifndef PA_DECODE_MIN_CTAS
#define PA_DECODE_MIN_CTAS 2
#endif
#ifndef PA_DECODE_RING_KB
#define PA_DECODE_RING_KB 16
#endif
#ifndef PA_DECODE_LANES_SMALL_GROUP
#define PA_DECODE_LANES_SMALL_GROUP 8
#endif
#ifndef PA_DECODE_MIN_STEPS
#define PA_DECODE_MIN_STEPS 4  // token-row steps per tile (tile = steps x 32/G tokens)
#endif
#ifndef PA_DECODE_LOADER
#define PA_DECODE_LOADER 0  // 0: one bulk (TMA) copy per block piece; 1: per-lane cp.async
#endif
#ifndef PA_DECODE_Q_SMEM
#define PA_DECODE_Q_SMEM 0  // 1: keep the scaled q in shared memory, not registers
#endif
#ifndef PA_DECODE_MMA_MIN_GQ
#define PA_DECODE_MMA_MIN_GQ 4  // bf16 groups of at least this many heads use the tensor-core tile
#endif
#ifndef PA_DECODE_MMA_CTAS
#define PA_DECODE_MMA_CTAS 2    // CTAs per SM of the tensor-core persistent grid
#endif
constexpr int kWarps = 4;              // warps per CTA
constexpr int kMinCtas = PA_DECODE_MIN_CTAS;
constexpr int kRingBytes = PA_DECODE_RING_KB * 1024;  // per-warp K+V staging ring
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTau = 8.0f;           // lazy-rescale headroom (log2 units)
constexpr int kDefaultPartition = 512;
constexpr int kMaxPartition = 8192;
// the persistent kernel keeps [B] tables in shared memory: (3 B + 1) ints,
// two CTAs per SM up to about 3,200 sequences, one beyond (the occupancy
// query at launch decides)
constexpr int kPersistentMaxB = 4096;

template <typename T, int D, int GQ>
struct Cfg {
    static constexpr int ES = sizeof(T);
    static constexpr int ROW = D * ES;       // bytes of one token row of one KV head
    static constexpr int CHUNKS = ROW / 16;  // 16-byte chunks per row
    static constexpr int G0 = GQ >= 8 ? 16 : PA_DECODE_LANES_SMALL_GROUP;
    static constexpr int G = G0 < CHUNKS ? G0 : CHUNKS;  // lanes per token
    static constexpr int CPL = CHUNKS / G;               // chunks per lane
    static constexpr int EPC = 16 / ES;                  // elements per chunk
    static constexpr int E = CPL * EPC;                  // elements per lane
    static constexpr int P = E / 2;                      // float2 pairs per lane
    static constexpr int TPS = 32 / G;                   // tokens per step
    static constexpr int SMIN = (G + GQ - 1) / GQ;
    static constexpr int S = SMIN > PA_DECODE_MIN_STEPS ? SMIN : PA_DECODE_MIN_STEPS;
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
    // CTAs per SM the register budget targets (groups of 8 heads need ~220
    // registers per thread, so they run at 2)
    static constexpr int MINB = GQ >= 8 ? 2 : kMinCtas;
    static constexpr int OFF_P = kWarps * WARP_SMEM;                  // p and score buffers
    static constexpr bool QS = PA_DECODE_Q_SMEM != 0;
    static constexpr int OFF_Q = OFF_P + kWarps * 2 * TT * GQ * 4;    // scaled q (QS)
    static constexpr int OFF_BAR = OFF_Q + (QS ? kWarps * GQ * D * 4 : 0);  // mbarriers
    static constexpr int OFF_FLAG = OFF_BAR + kWarps * NST * 8;       // flag / scan scratch
    static constexpr int OFF_BT = OFF_FLAG + 16;                      // per-batch tables
    static_assert(G * CPL == CHUNKS, "row must split evenly over the lanes of a token");
    static_assert(V % G == 0 && VPL <= GQ && GQ % VPL == 0, "bad reduction shape");
    static_assert(E % 2 == 0 && TT <= 32, "bad tile");
    static_assert(GQ * D * 4 + 2 * GQ * 4 <= WARP_SMEM, "merge buffer must fit the ring");
    static_assert(kWarps * 4 <= 16, "scan scratch");
};

struct DecodeParams {
    void *out;
    const void *q;
    const uint8_t *k_cache;
    const uint8_t *v_cache;
    const int32_t *block_table;
    const int32_t *context_lens;
    float *ws_acc;               // [B][Hq][rowslots][D]
    float *ws_ml;                // [B][Hq][rowslots][2] (max, sum)
    unsigned *meta;              // [B][Hkv] partials per item (persistent kernel)
    int *err;
    const int32_t *shared_len;   // [B] tokens covered by a shared-prefix partial, or NULL
    int64_t num_blocks;
    int B, Hq, Hkv, bs, bs_log2, MB, PT, max_parts, maxseg;
    int rowslots;                // partial slots per (sequence, query head)
    int pslot0, npfx;            // shared-prefix partials: slots pslot0 .. pslot0+npfx-1
    // forked children (pa_decode_shared_forks): fork_parent[b] >= 0 names the
    // row whose blocks [0, fork_len[b]) row b shares; the parent's items then
    // serve b's heads over [shared_len, fork_len) too (NULL: none)
    const int32_t *fork_parent, *fork_len;
    int contig_len;              // > 0: contiguous caches [B][Hkv][contig_len][D], no table
    int early_dependents;        // persistent kernel: release the next kernel at the start
    float qscale;                // scale * log2(e)
};

// Wait until the kernels this grid was launched behind (as a programmatic
// dependent) have completed and their writes are visible; a no-op for a grid
// launched without that attribute.  Every decode grid runs this before it
// reads any input.
__device__ __forceinline__ void wait_prior_grids() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

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

// One warp's attention state for one (sequence, KV head) item: q of the GQ
// heads (this lane's elements), running max, per-lane partial sums, and the
// PV accumulators of this lane's elements.
template <typename T, int D, int GQ>
struct WarpAttn {
    using C = Cfg<T, D, GQ>;
    int lane, gl, grp, h0, row_mine;
    float *qs;  // per-warp scaled q [GQ][D] in shared memory (QS)
    float2 q2[C::QS ? 1 : GQ][C::QS ? 1 : C::P];
    float m_run[GQ];
    float2 acc[GQ][C::P];
    float lsum[C::VPL], mh[C::VPL];
    float mhh;  // running max of head lane % GQ

    __device__ __forceinline__ void init(int lane_) {
        lane = lane_;
        gl = lane % C::G;
        grp = lane / C::G;
        // after the transpose-reduce this lane holds the scores of heads
        // h0 .. h0+VPL-1 of token row row_mine of the tile
        h0 = (gl * C::VPL) % GQ;
        row_mine = ((gl * C::VPL) / GQ) * C::TPS + grp;
    }

    // element index of pair j of chunk c of this lane
    __device__ __forceinline__ int dim_of(int c, int j) const {
        return (c * C::G + gl) * C::EPC + 2 * j;
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            m_run[h] = -INFINITY;
#pragma unroll
            for (int j = 0; j < C::P; ++j) acc[h][j] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < C::VPL; ++k) {
            lsum[k] = 0.f;
            mh[k] = -INFINITY;
        }
        mhh = -INFINITY;
    }

    // qb points at q[b][first head of the group][0]
    __device__ __forceinline__ void load_q(const T *qb, float qscale) {
        if constexpr (C::QS) __syncwarp();  // the previous item's reads are done
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int c = 0; c < C::CPL; ++c) {
                const uint4 raw =
                    *reinterpret_cast<const uint4 *>(qb + h * D + (c * C::G + gl) * C::EPC);
                float2 f[C::EPC / 2];
                pa::Elem<T>::unpack(raw, f);
#pragma unroll
                for (int i = 0; i < C::EPC / 2; ++i) {
                    const float2 v = make_float2(f[i].x * qscale, f[i].y * qscale);
                    if constexpr (C::QS) {
                        if (grp == 0)
                            *reinterpret_cast<float2 *>(qs + h * D + (c * C::G + gl) * C::EPC +
                                                        2 * i) = v;
                    } else {
                        q2[h][c * C::EPC / 2 + i] = v;
                    }
                }
            }
        if constexpr (C::QS) __syncwarp();
    }

    __device__ __forceinline__ float2 qpair(int h, int j) const {
        if constexpr (C::QS) {
            const int c = j / (C::EPC / 2), i = j % (C::EPC / 2);
            return *reinterpret_cast<const float2 *>(qs + h * D + (c * C::G + gl) * C::EPC + 2 * i);
        } else {
            return q2[h][j];
        }
    }

    // One staged tile: K rows at kaddr, V rows at vaddr (shared), nvalid rows valid.
    __device__ __forceinline__ void tile(uint32_t kaddr, uint32_t vaddr, int nvalid, float *pbuf,
                                         float *sbuf) {
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
                for (int j = 0; j < C::P; ++j) a = pa::ffma2(qpair(h, j), kf[j], a);
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
            // Lane l computes head (l % GQ)'s new max and rescale factor;
            // every other value travels by shuffle (no per-lane indexing of
            // the per-head arrays, which would push them to local memory).
            const int hh = lane % GQ;
            float tmax = -INFINITY;
            for (int r = 0; r < C::TT; ++r) tmax = fmaxf(tmax, sbuf[r * GQ + hh]);
            const float mnew_l = fmaxf(mhh, tmax);
            const float alpha_l = (mhh == -INFINITY) ? 0.f : exp2f(mhh - mnew_l);
            mhh = mnew_l;
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float alpha = __shfl_sync(pa::kFull, alpha_l, h);
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int j = 0; j < C::P; ++j) acc[h][j] = __fmul2_rn(acc[h][j], a2);
                m_run[h] = __shfl_sync(pa::kFull, mnew_l, h);
            }
#pragma unroll
            for (int k = 0; k < C::VPL; ++k) {
                lsum[k] *= __shfl_sync(pa::kFull, alpha_l, h0 + k);
                mh[k] = __shfl_sync(pa::kFull, mnew_l, h0 + k);
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
    }

    // Sum acc over the token groups (every lane ends with the totals of its
    // elements) and the per-head softmax denominators over all lanes.
    __device__ __forceinline__ void reduce(float (&lh)[GQ]) {
#pragma unroll
        for (int off = C::G; off < 32; off <<= 1)
#pragma unroll
            for (int h = 0; h < GQ; ++h)
#pragma unroll
                for (int j = 0; j < C::P; ++j) {
                    acc[h][j].x += __shfl_xor_sync(pa::kFull, acc[h][j].x, off);
                    acc[h][j].y += __shfl_xor_sync(pa::kFull, acc[h][j].y, off);
                }
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
    }

    // The whole item ended in this warp: out[h][:] = acc / lh[h] for its GQ
    // heads (outh points at the first head's row; lh from reduce()).
    __device__ __forceinline__ void store_out(T *outh, const float (&lh)[GQ]);

    // Partial of this segment: acc (unnormalised) at acc_dst + h * head_stride,
    // (max, sum) at ml_dst + h * ml_stride for each head h.
    __device__ __forceinline__ void store_partial(float *acc_dst, size_t head_stride,
                                                  float *ml_dst, size_t ml_stride,
                                                  const float (&lh)[GQ]) {
        if (grp == 0) {
#pragma unroll
            for (int h = 0; h < GQ; ++h)
#pragma unroll
                for (int cc = 0; cc < C::CPL; ++cc)
#pragma unroll
                    for (int j = 0; j < C::EPC / 2; ++j)
                        *reinterpret_cast<float2 *>(acc_dst + h * head_stride + dim_of(cc, j)) =
                            acc[h][cc * C::EPC / 2 + j];
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < GQ; ++h)
                *reinterpret_cast<float2 *>(ml_dst + h * ml_stride) = make_float2(m_run[h], lh[h]);
        }
    }
};

template <typename T>
__device__ __forceinline__ void store_pair(T *dst, float a, float b);
template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(__nv_bfloat16 *dst, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(a, b);
}
template <>
__device__ __forceinline__ void store_pair<float>(float *dst, float a, float b) {
    *reinterpret_cast<float2 *>(dst) = make_float2(a, b);
}

template <typename T, int D, int GQ>
__device__ __forceinline__ void WarpAttn<T, D, GQ>::store_out(T *outh, const float (&lh)[GQ]) {
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            const float inv = 1.f / lh[h];
#pragma unroll
            for (int cc = 0; cc < C::CPL; ++cc)
#pragma unroll
                for (int j = 0; j < C::EPC / 2; ++j) {
                    const float2 a = acc[h][cc * C::EPC / 2 + j];
                    store_pair<T>(outh + h * D + dim_of(cc, j), a.x * inv, a.y * inv);
                }
        }
    }
}

// ---------------------------------------------------------------------------
// Tensor-core tile (bf16, groups of 8 heads): per 16-token tile of one
// (sequence, KV head) item, one warp computes
//   S^T[token][head] = K[token][:] . q[head][:]      (m16n8k16, M = tokens)
//   O^T[d][head]    += V^T[d][token] . P^T[token][head]   (M = head dims)
// with warp-level bf16 MMAs (fp32 accumulate).  The 8 heads of a group are
// the N = 8 columns, so no row of either product is padding.  K and V
// arrive by 2D tensor copies with the 128-byte swizzle (bank-conflict-free
// ldmatrix); q stays in registers as the B fragments of the first product,
// unscaled (S is scaled in fp32).  Lane (g, t) = (lane / 4, lane % 4) holds
// S^T for tokens g, g+8 of heads 2t, 2t+1, and O^T for dims 16m+g, 16m+g+8 of
// the same two heads, so the online softmax (max, rescale, exp, sum) needs
// no shuffle other than the per-head max over the 8 lanes of a column.  P
// enters the second product as two bf16 terms (hi + lo: p to ~2^-16
// relative), transposed into B fragments by movmatrix.  Tokens past the
// context get score -inf and their V rows are zeroed in shared memory (a
// stale row may hold NaN; 0 * NaN = NaN).
// ---------------------------------------------------------------------------
// QH: query rows carried in a stage with an item's first tile (GQ, or 2 GQ
// when an item also serves a forked child's heads in the spare columns).
template <int D, int GQ, int QH = GQ>
struct MmaCfg {
    static constexpr int TT = 16;               // tokens per tile (the M of the first product)
    static constexpr int HALVES = D / 64;       // 128-byte column blocks of a row (64 bf16)
    static constexpr int HALF = TT * 128;       // bytes of one column block of one cache's tile
    static constexpr int TILE = HALVES * HALF;  // one cache's tile
    static constexpr int QB = QH * D * 2;       // the q rows (first tile of an item)
    // K, V, then q; stages stay 1024-byte aligned for the swizzle
    static constexpr int STAGE = (2 * TILE + QB + 1023) / 1024 * 1024;
    static constexpr int NST = kRingBytes / STAGE >= 2 ? kRingBytes / STAGE : 2;
    static constexpr int WARP_SMEM = NST * STAGE;
    static constexpr int MINB = PA_DECODE_MMA_CTAS;
    static constexpr bool QS = false;
    static constexpr int OFF_P = kWarps * WARP_SMEM;  // no p / score buffers
    static constexpr int OFF_Q = OFF_P;
    static constexpr int OFF_BAR = OFF_Q;
    static constexpr int OFF_FLAG = OFF_BAR + kWarps * NST * 8;
    static constexpr int OFF_BT = OFF_FLAG + 16;
    static constexpr int KS = D / 16;           // k-steps of QK^T = m-tiles of PV
    static_assert(D % 64 == 0 && GQ <= 8 && 8 % GQ == 0 && QH <= 8, "tensor-core tile shape");
    static_assert(HALF % 1024 == 0 && STAGE % 1024 == 0, "swizzle atoms must stay aligned");
};

template <int D, int GQ, int QH = GQ>
struct MmaAttn {
    using C = MmaCfg<D, GQ, QH>;
    static constexpr int KS = C::KS;
    int lane, g, t, grp;
    float *qs;  // unused (interface of WarpAttn)
    float qscale;
    uint32_t qf[KS][2];   // B fragments of q^T: head g, dims 16k + 2t (+1) and 16k + 2t + 8 (+9)
    float acc[KS][4];     // O^T fragments: dims 16m + g (+8) x heads 2t, 2t+1
    float m_run[2], lsum[2];
    uint32_t koff[4], voff[4];  // per-lane ldmatrix row offsets (swizzled), by k-step % 4

    __device__ __forceinline__ void init(int lane_) {
        lane = lane_;
        g = lane >> 2;
        t = lane & 3;
        grp = 0;
        const int x7 = lane & 7;
        const int tk = (lane & 7) + ((lane >> 3) & 1) * 8, hk_ = lane >> 4;  // K: matrices (tok, chunk)
        const int tv = (lane & 7) + ((lane >> 4) & 1) * 8, hv = (lane >> 3) & 1;  // V^T
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            koff[j] = tk * 128 + (((2 * j + hk_) ^ x7) << 4);
            voff[j] = tv * 128 + (((2 * j + hv) ^ x7) << 4);
        }
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int m = 0; m < KS; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[m][i] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        lsum[0] = lsum[1] = 0.f;
    }

    __device__ __forceinline__ void load_q(const __nv_bfloat16 *qb, float qscale_) {
        qscale = qscale_;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            uint32_t b0 = 0u, b1 = 0u;
            if (g < GQ) {
                const uint32_t *row = reinterpret_cast<const uint32_t *>(qb + g * D + 16 * k);
                b0 = __ldg(row + t);
                b1 = __ldg(row + t + 4);
            }
            qf[k][0] = b0;
            qf[k][1] = b1;
        }
    }

    // q of the item from the stage (the producer copied the group's GQ rows
    // there with the item's first tile): lane (g, t) takes head g's dims
    // 16k + 2t (+1) and 16k + 2t + 8 (+9) as its B fragments.
    __device__ __forceinline__ void load_q_smem(uint32_t qaddr, float qscale_, int ncols = GQ) {
        qscale = qscale_;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            uint32_t b0 = 0u, b1 = 0u;
            if (g < ncols) {
                const uint32_t a = qaddr + g * D * 2 + (16 * k + 2 * t) * 2;
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b0) : "r"(a));
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b1) : "r"(a + 16));
            }
            qf[k][0] = b0;
            qf[k][1] = b1;
        }
    }

    // Column g of the products reads q row `row` (NULL: a zero column).
    __device__ __forceinline__ void load_q_row(const __nv_bfloat16 *row, float qscale_) {
        qscale = qscale_;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            uint32_t b0 = 0u, b1 = 0u;
            if (row) {
                const uint32_t *r = reinterpret_cast<const uint32_t *>(row + 16 * k);
                b0 = __ldg(r + t);
                b1 = __ldg(r + t + 4);
            }
            qf[k][0] = b0;
            qf[k][1] = b1;
        }
    }

    // nvalid: tokens of the tile inside the context; with QH > GQ, the
    // columns from GQ on (a forked child's heads) see only the first
    // nvalid_hi of them.
    __device__ __forceinline__ void tile(uint32_t kaddr, uint32_t vaddr, int nvalid, float *,
                                         float *, int nvalid_hi = 0) {
        // ---- S^T = K q^T (two accumulators: shorter dependency chains) ----
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            uint32_t a[4];
            pa::ldsm_x4(a, kaddr + (k >> 2) * C::HALF + koff[k & 3]);
            if (k & 1) pa::mma_bf16_16816(s2, a, qf[k][0], qf[k][1]);
            else pa::mma_bf16_16816(s, a, qf[k][0], qf[k][1]);
        }
        if (nvalid < C::TT) {
            // zero the V rows past the context (both column blocks)
            const int n = (C::TT - nvalid) * C::HALVES * 8;
            for (int i = lane; i < n; i += 32) {
                const int r = nvalid + i / (C::HALVES * 8), w = i % (C::HALVES * 8);
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                                 vaddr + (w >> 3) * C::HALF + r * 128 + (w & 7) * 16),
                             "r"(0u)
                             : "memory");
            }
            __syncwarp();
        }
        const int nv = (QH > GQ && 2 * t >= GQ) ? nvalid_hi : nvalid;
        const bool v0 = g < nv, v1 = g + 8 < nv;
        const float x0 = v0 ? (s[0] + s2[0]) * qscale : -INFINITY;  // token g, head 2t
        const float x1 = v0 ? (s[1] + s2[1]) * qscale : -INFINITY;  // token g, head 2t+1
        const float x2 = v1 ? (s[2] + s2[2]) * qscale : -INFINITY;  // token g+8, head 2t
        const float x3 = v1 ? (s[3] + s2[3]) * qscale : -INFINITY;  // token g+8, head 2t+1
        // ---- online softmax (log2 domain, lazy rescale) ----------------------
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(pa::kFull, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(pa::kFull, mx1, o));
        }
        const bool n0 = mx0 > m_run[0] + kTau, n1 = mx1 > m_run[1] + kTau;
        if (__any_sync(pa::kFull, n0 || n1)) {
            const float m0 = n0 ? fmaxf(m_run[0], mx0) : m_run[0];
            const float m1 = n1 ? fmaxf(m_run[1], mx1) : m_run[1];
            const float a0 = m_run[0] == -INFINITY ? 0.f : exp2f(m_run[0] - m0);
            const float a1 = m_run[1] == -INFINITY ? 0.f : exp2f(m_run[1] - m1);
#pragma unroll
            for (int m = 0; m < KS; ++m) {
                acc[m][0] *= a0;
                acc[m][1] *= a1;
                acc[m][2] *= a0;
                acc[m][3] *= a1;
            }
            lsum[0] *= a0;
            lsum[1] *= a1;
            m_run[0] = m0;
            m_run[1] = m1;
        }
        // a column that has seen no token yet (m = -inf) takes p = 0, not
        // exp2(-inf + inf): the forked child's columns past its fork point
        const float mr0 = (QH > GQ && m_run[0] == -INFINITY) ? 0.f : m_run[0];
        const float mr1 = (QH > GQ && m_run[1] == -INFINITY) ? 0.f : m_run[1];
        const float p0 = fast_exp2(x0 - mr0), p1 = fast_exp2(x1 - mr1);
        const float p2 = fast_exp2(x2 - mr0), p3 = fast_exp2(x3 - mr1);
        lsum[0] += p0 + p2;
        lsum[1] += p1 + p3;
        // ---- P^T as bf16 hi + lo B fragments --------------------------------
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(p0, p1);
        const __nv_bfloat162 h23 = __floats2bfloat162_rn(p2, p3);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        const __nv_bfloat162 l01 = __floats2bfloat162_rn(p0 - f01.x, p1 - f01.y);
        const __nv_bfloat162 l23 = __floats2bfloat162_rn(p2 - f23.x, p3 - f23.y);
        const uint32_t bh0 = pa::movmatrix_trans(*reinterpret_cast<const uint32_t *>(&h01));
        const uint32_t bh1 = pa::movmatrix_trans(*reinterpret_cast<const uint32_t *>(&h23));
        const uint32_t bl0 = pa::movmatrix_trans(*reinterpret_cast<const uint32_t *>(&l01));
        const uint32_t bl1 = pa::movmatrix_trans(*reinterpret_cast<const uint32_t *>(&l23));
        // ---- O^T += V^T P^T ---------------------------------------------------
#pragma unroll
        for (int m = 0; m < KS; ++m) {
            uint32_t a[4];
            pa::ldsm_x4_trans(a, vaddr + (m >> 2) * C::HALF + voff[m & 3]);
            pa::mma_bf16_16816(acc[m], a, bh0, bh1);
            pa::mma_bf16_16816(acc[m], a, bl0, bl1);
        }
    }

    // Softmax sums of this lane's heads 2t, 2t+1 (reduced over the 8 lanes
    // of each column) into lh[0], lh[1].
    template <int N>
    __device__ __forceinline__ void reduce(float (&lh)[N]) const {
        static_assert(N >= 2, "two columns per lane");
        float l0 = lsum[0], l1 = lsum[1];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(pa::kFull, l0, o);
            l1 += __shfl_xor_sync(pa::kFull, l1, o);
        }
        lh[0] = l0;
        lh[1] = l1;
    }

    __device__ __forceinline__ void store_out(__nv_bfloat16 *outh, const float (&lh)[GQ]) {
        static_assert(GQ % 2 == 0, "a lane's two columns are heads of one sequence");
        const float2 l = make_float2(lh[0], lh[1]);
        if (2 * t >= GQ) return;
        const float i0 = 1.f / l.x, i1 = 1.f / l.y;
        __nv_bfloat16 *o0 = outh + (2 * t) * D + g, *o1 = o0 + D;
#pragma unroll
        for (int m = 0; m < KS; ++m) {
            o0[16 * m] = __float2bfloat16_rn(acc[m][0] * i0);
            o1[16 * m] = __float2bfloat16_rn(acc[m][1] * i1);
            o0[16 * m + 8] = __float2bfloat16_rn(acc[m][2] * i0);
            o1[16 * m + 8] = __float2bfloat16_rn(acc[m][3] * i1);
        }
    }

    __device__ __forceinline__ void store_partial(float *acc_dst, size_t head_stride,
                                                  float *ml_dst, size_t ml_stride,
                                                  const float (&lh)[GQ]) {
        static_assert(GQ % 2 == 0, "a lane's two columns are heads of one sequence");
        const float2 l = make_float2(lh[0], lh[1]);
        if (2 * t >= GQ) return;
        float *a0 = acc_dst + (2 * t) * head_stride + g, *a1 = a0 + head_stride;
#pragma unroll
        for (int m = 0; m < KS; ++m) {
            a0[16 * m] = acc[m][0];
            a1[16 * m] = acc[m][1];
            a0[16 * m + 8] = acc[m][2];
            a1[16 * m + 8] = acc[m][3];
        }
        if (g == 0) {
            *reinterpret_cast<float2 *>(ml_dst + (2 * t) * ml_stride) = make_float2(m_run[0], l.x);
            *reinterpret_cast<float2 *>(ml_dst + (2 * t + 1) * ml_stride) =
                make_float2(m_run[1], l.y);
        }
    }

    // The partial of columns GQ .. 2 GQ - 1 (a forked child's heads) into the
    // child's rows: acc_dst / ml_dst address its head 0.
    __device__ __forceinline__ void store_partial_hi(float *acc_dst, size_t head_stride,
                                                     float *ml_dst, size_t ml_stride,
                                                     const float (&lh)[GQ]) {
        static_assert(QH == 2 * GQ && GQ % 2 == 0, "the child's heads fill columns GQ ..");
        const float2 l = make_float2(lh[0], lh[1]);
        const int c0 = 2 * t - GQ;
        if (c0 < 0 || c0 >= GQ) return;
        float *a0 = acc_dst + c0 * head_stride + g, *a1 = a0 + head_stride;
#pragma unroll
        for (int m = 0; m < KS; ++m) {
            a0[16 * m] = acc[m][0];
            a1[16 * m] = acc[m][1];
            a0[16 * m + 8] = acc[m][2];
            a1[16 * m + 8] = acc[m][3];
        }
        if (g == 0) {
            *reinterpret_cast<float2 *>(ml_dst + c0 * ml_stride) = make_float2(m_run[0], l.x);
            *reinterpret_cast<float2 *>(ml_dst + (c0 + 1) * ml_stride) = make_float2(m_run[1], l.y);
        }
    }
};

// ---------------------------------------------------------------------------
// Persistent kernel (default)
// ---------------------------------------------------------------------------
struct Cursor {
    int b, hk, t, nt, L;  // item (b, hk), tile t of nt tiles, context length L
    int s0;               // first token the item's tiles cover (shared prefix excluded)
};

__device__ __forceinline__ int first_token(const Cursor &c, int TT) { return c.s0 + c.t * TT; }

// Tables of the persistent kernel in shared memory: tile prefix over the
// sequences ([B+1]), clamped context lengths ([B]) and first tokens ([B]).
struct BatchTables {
    const int32_t *pre;
    const int32_t *lens;
    const int32_t *starts;
};

// Cursor at unit u: the largest b with Hkv*pre[b] <= u, then (hk, t).
__device__ __forceinline__ Cursor locate_unit(int64_t u, const BatchTables &bt, int B, int Hkv) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (int64_t(Hkv) * bt.pre[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    Cursor c;
    c.b = lo;
    c.nt = bt.pre[lo + 1] - bt.pre[lo];
    c.L = bt.lens[lo];
    c.s0 = bt.starts[lo];
    const int64_t rem = u - int64_t(Hkv) * bt.pre[lo];
    c.hk = static_cast<int>(rem / c.nt);
    c.t = static_cast<int>(rem - int64_t(c.hk) * c.nt);
    return c;
}

// Next unit: next tile, else next KV head, else next sequence with tiles.
__device__ __forceinline__ Cursor next_unit(Cursor c, const BatchTables &bt, int B, int Hkv) {
    if (++c.t == c.nt) {
        c.t = 0;
        if (++c.hk == Hkv) {
            c.hk = 0;
            do {
                ++c.b;
            } while (c.b < B && bt.pre[c.b + 1] == bt.pre[c.b]);
            if (c.b < B) {
                c.nt = bt.pre[c.b + 1] - bt.pre[c.b];
                c.L = bt.lens[c.b];
                c.s0 = bt.starts[c.b];
            }
        }
    }
    return c;
}

template <int TT>
__device__ __forceinline__ int block_entry(const DecodeParams &p, const Cursor &c, int j) {
    if (p.contig_len) return 0;  // contiguous caches: no block table
    return __ldg(p.block_table + static_cast<size_t>(c.b) * p.MB +
                 (first_token(c, TT) >> p.bs_log2) + j);
}

// Contiguous caches: first row of tile c, as a row index of [B][Hkv][len][D].
__device__ __forceinline__ int64_t contig_row(const DecodeParams &p, const Cursor &c, int tok) {
    return (static_cast<int64_t>(c.b) * p.Hkv + c.hk) * p.contig_len + tok;
}

__device__ __forceinline__ int checked_block(const DecodeParams &p, int v) {
    if (v < 0 || v >= p.num_blocks) {
        pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
        v = 0;
    }
    return v;
}

// Producer (one lane): bulk-copy the K and V rows of tile c into the stage.
template <typename T, int D, int GQ>
__device__ __forceinline__ void produce_tile(const DecodeParams &p, const Cursor &c, int blk,
                                             uint8_t *stage, uint64_t *bar) {
    using C = Cfg<T, D, GQ>;
    uint8_t *dk = stage;
    uint8_t *dv = stage + C::TILE;
    const int tok = first_token(c, C::TT);
    if (p.contig_len) {  // one copy of TT whole rows per cache (contig_len % 32 == 0)
        const size_t off = static_cast<size_t>(contig_row(p, c, tok)) * C::ROW;
        pa::mbar_arrive_expect_tx(bar, 2 * C::TILE);
        pa::bulk_g2s(dk, p.k_cache + off, C::TILE, bar);
        pa::bulk_g2s(dv, p.v_cache + off, C::TILE, bar);
    } else if (C::TT <= p.bs) {
        const int r0 = tok & (p.bs - 1);
        const size_t off = ((static_cast<size_t>(blk) * p.Hkv + c.hk) * p.bs + r0) * C::ROW;
        pa::mbar_arrive_expect_tx(bar, 2 * C::TILE);
        pa::bulk_g2s(dk, p.k_cache + off, C::TILE, bar);
        pa::bulk_g2s(dv, p.v_cache + off, C::TILE, bar);
    } else {
        const int nb = C::TT >> p.bs_log2;  // blocks per tile
        const uint32_t bytes = static_cast<uint32_t>(p.bs) * C::ROW;
        int avail = 0;
        for (int j = 0; j < nb; ++j) avail += (tok + j * p.bs < c.L) ? 1 : 0;
        pa::mbar_arrive_expect_tx(bar, 2u * avail * bytes);
        for (int j = 0; j < avail; ++j) {
            const int id = j == 0 ? blk : checked_block(p, block_entry<C::TT>(p, c, j));
            const size_t off = (static_cast<size_t>(id) * p.Hkv + c.hk) * p.bs * C::ROW;
            pa::bulk_g2s(dk + j * bytes, p.k_cache + off, bytes, bar);
            pa::bulk_g2s(dv + j * bytes, p.v_cache + off, bytes, bar);
        }
    }
}

// Producer (one lane) of the tensor-core tile: 2D tensor copies of the K and
// V rows of tile c (boxes of min(TT, bs) rows x 64 columns, 128-byte swizzle)
// into the stage: [K block 0 | K block 1 | V block 0 | V block 1] by 64-column
// block.  Tiles longer than a block take one box per block; blocks past the
// context are not copied (their rows are masked).
template <int D, int GQ, int QH = GQ>
__device__ __forceinline__ void produce_tile_tma(const DecodeParams &p, const Cursor &c, int blk,
                                                 uint8_t *stage, uint64_t *bar,
                                                 const CUtensorMap *kmap,
                                                 const CUtensorMap *vmap, bool with_q = false,
                                                 int child_row = -1) {
    using C = MmaCfg<D, GQ, QH>;
    constexpr uint32_t QG = GQ * D * 2;  // one sequence's group of q rows
    const uint32_t sk = pa::smem_u32(stage), sv = sk + C::TILE;
    const int tok = first_token(c, C::TT);
    const bool with_child = QH > GQ && with_q && child_row >= 0;
    const uint32_t qbytes = with_q ? QG * (with_child ? 2u : 1u) : 0u;
    if (with_q)  // the group's q rows, contiguous in q [B][Hq][D]
        pa::bulk_g2s(stage + 2 * C::TILE,
                     static_cast<const __nv_bfloat16 *>(p.q) +
                         (static_cast<size_t>(c.b) * p.Hq + c.hk * GQ) * D,
                     QG, bar);
    if (with_child)  // then the forked child's, for the spare columns
        pa::bulk_g2s(stage + 2 * C::TILE + QG,
                     static_cast<const __nv_bfloat16 *>(p.q) +
                         (static_cast<size_t>(child_row) * p.Hq + c.hk * GQ) * D,
                     QG, bar);
    if (p.contig_len || C::TT <= p.bs) {
        const int y = p.contig_len ? static_cast<int>(contig_row(p, c, tok))
                                   : (blk * p.Hkv + c.hk) * p.bs + (tok & (p.bs - 1));
        pa::mbar_arrive_expect_tx(bar, 2 * C::TILE + qbytes);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
            pa::tma_2d_g2s(sk + h * C::HALF, kmap, 64 * h, y, bar);
            pa::tma_2d_g2s(sv + h * C::HALF, vmap, 64 * h, y, bar);
        }
    } else {
        const int nb = C::TT >> p.bs_log2;  // blocks per tile
        int avail = 0;
        for (int j = 0; j < nb; ++j) avail += (tok + j * p.bs < c.L) ? 1 : 0;
        pa::mbar_arrive_expect_tx(bar, 2u * avail * C::HALVES * p.bs * 128 + qbytes);
        for (int j = 0; j < avail; ++j) {
            const int id = j == 0 ? blk : checked_block(p, block_entry<C::TT>(p, c, j));
            const int y = (id * p.Hkv + c.hk) * p.bs;
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h) {
                pa::tma_2d_g2s(sk + h * C::HALF + j * p.bs * 128, kmap, 64 * h, y, bar);
                pa::tma_2d_g2s(sv + h * C::HALF + j * p.bs * 128, vmap, 64 * h, y, bar);
            }
        }
    }
}

// Producer (whole warp): 16-byte cp.async copies of tile c's K and V rows,
// lane l taking chunks l, l+32, ...; each lane's completions arrive on the
// stage's mbarrier (initialised with one arrival per lane).
template <typename T, int D, int GQ>
__device__ __forceinline__ void produce_tile_lanes(const DecodeParams &p, const Cursor &c, int blk,
                                                   uint8_t *stage, uint64_t *bar, int lane) {
    using C = Cfg<T, D, GQ>;
    const int tok = first_token(c, C::TT);
    const uint32_t sk = pa::smem_u32(stage);
#pragma unroll
    for (int k = 0; k < C::TILE / 16 / 32; ++k) {
        const int ch = lane + 32 * k;
        const int row = ch / C::CHUNKS, within = ch % C::CHUNKS;
        const int t = tok + row;
        if (t >= c.L) continue;  // rows past the end stay stale and are masked
        int id = blk;
        if (!p.contig_len && C::TT > p.bs && (t >> p.bs_log2) != (tok >> p.bs_log2))
            id = checked_block(p, __ldg(p.block_table + static_cast<size_t>(c.b) * p.MB +
                                        (t >> p.bs_log2)));
        const size_t off =
            (p.contig_len ? static_cast<size_t>(contig_row(p, c, t))
                          : (static_cast<size_t>(id) * p.Hkv + c.hk) * p.bs + (t & (p.bs - 1))) *
                C::ROW +
            within * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sk + ch * 16),
                     "l"(p.k_cache + off)
                     : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sk + C::TILE + ch * 16),
                     "l"(p.v_cache + off)
                     : "memory");
    }
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(pa::smem_u32(bar))
                 : "memory");
}

// Bring an item's q into L1 ahead of its first tile (lanes < q lines).
template <typename T, int D, int GQ>
__device__ __forceinline__ void prefetch_q(const DecodeParams &p, const Cursor &c, int lane) {
    constexpr int kLines = GQ * D * int(sizeof(T)) / 128;
    const char *qa = reinterpret_cast<const char *>(
        static_cast<const T *>(p.q) + (static_cast<size_t>(c.b) * p.Hq + c.hk * GQ) * D);
    if (lane < kLines) asm volatile("prefetch.global.L1 [%0];" ::"l"(qa + lane * 128));
}

// Merge of an item spread over more than 32 warps (a few very long
// sequences): the weights are recomputed from loads instead of travelling
// by shuffle.  Kept out of line so the common path's code is unaffected.
// Slot of the i-th partial of an item with nseg segments: its segments,
// then the shared-prefix partials.
__device__ __forceinline__ int slot_of(const DecodeParams &p, int i, int nseg) {
    return i < nseg ? i : p.pslot0 + (i - nseg);
}

// End of this warp's segment of item c.  An item that lies whole in this
// warp's range (and has no shared-prefix partials) is written out directly;
// otherwise the segment writes its partial (max, sum, unnormalised weighted
// values) to its slot and partial_merge_kernel, launched behind this grid,
// merges the item's partials.  The item's first segment records how many
// there are.  No segment waits for, or signals, any other.
// Fork tables of the persistent kernel (pa_decode_shared_forks), in shared
// memory: each row's validated shared_len, the child its items also serve
// (-1: none) and the parent whose items serve its fork range (-1: none).
struct ForkTables {
    const int32_t *slen, *child, *parent;
};

template <typename T, int D, int GQ, bool FORK = false, typename St>
__device__ __forceinline__ void finish_segment(St &st, const DecodeParams &p,
                                               const BatchTables &bt, const Cursor &c,
                                               int64_t per, int64_t w, int lane,
                                               const ForkTables &ft = ForkTables{}) {
    float lh[GQ];
    st.reduce(lh);
    const int64_t ia = int64_t(p.Hkv) * bt.pre[c.b] + int64_t(c.hk) * c.nt;
    const int64_t wa = ia / per, wb = (ia + c.nt - 1) / per;
    const int nseg = static_cast<int>(wb - wa + 1), seg = static_cast<int>(w - wa);
    const size_t hq0 = static_cast<size_t>(c.b) * p.Hq + c.hk * GQ;
    // an item that starts after a shared prefix also merges the prefix partials
    int npre = c.s0 > 0 ? p.npfx : 0;
    int npair = 0;  // a forked child's partials from its parent's item segments
    if constexpr (FORK) {
        npre = ft.slen[c.b] > 0 ? p.npfx : 0;
        const int par = ft.parent[c.b];
        if (par >= 0) {
            const int ntp = bt.pre[par + 1] - bt.pre[par];
            const int64_t iap = int64_t(p.Hkv) * bt.pre[par] + int64_t(c.hk) * ntp;
            npair = static_cast<int>((iap + ntp - 1) / per - iap / per + 1);
        }
        const int cr = ft.child[c.b];
        if (cr >= 0) {  // this segment's partial for the child's heads, after its prefix slots
            const size_t hqc = static_cast<size_t>(cr) * p.Hq + c.hk * GQ;
            const size_t slot =
                hqc * p.rowslots + p.pslot0 + (ft.slen[cr] > 0 ? p.npfx : 0) + seg;
            st.store_partial_hi(p.ws_acc + slot * D, size_t(p.rowslots) * D, p.ws_ml + 2 * slot,
                                size_t(p.rowslots) * 2, lh);
        }
    }
    const bool whole = nseg == 1 && npre == 0 && npair == 0;
    if (seg == 0 && lane == 0)
        p.meta[static_cast<size_t>(c.b) * p.Hkv + c.hk] =
            whole ? 0u : static_cast<unsigned>(nseg) | (static_cast<unsigned>(npre + npair) << 16);
    if (whole) {
        st.store_out(static_cast<T *>(p.out) + hq0 * D, lh);
        return;
    }
    if (seg < 0 || seg >= p.maxseg) {  // cannot happen with maxseg from the host
        if (lane == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
        return;
    }
    st.store_partial(p.ws_acc + (hq0 * p.rowslots + seg) * D, size_t(p.rowslots) * D,
                     p.ws_ml + 2 * (hq0 * p.rowslots + seg), size_t(p.rowslots) * 2, lh);
}

// ---------------------------------------------------------------------------
// Shared-prefix partials (bf16, tensor core).  Members of a group share the
// physical blocks of their first S tokens ("PagedAttention: memetakan blok KV
// logis ke memori fisik tidak kontigu", section "Sharing blok dapat
// menghindari duplikasi state KV": one physical copy serves every sequence
// that references it), so those blocks are read once per (group, KV head,
// token chunk, CTA of members) instead of once per member.  One CTA: a
// loader warp streams 16-token K/V tiles of the chunk (2D tensor copies,
// through the first member's block table) into a ring shared by
// kPfxWarps consumer warps; each consumer runs the tensor-core tile with its
// 8 columns = 8 / GQ members x GQ heads, and writes the chunk's partial
// (max, sum, unnormalised weighted values) of every (member, head) to its
// prefix slot.  The decode then covers only tokens S .. L-1 of each member
// and merges these partials with its own by log-sum-exp.
// ---------------------------------------------------------------------------
#ifndef PA_PFX_WARPS
#define PA_PFX_WARPS 8
#endif
#ifndef PA_PFX_STAGES
#define PA_PFX_STAGES 4
#endif
constexpr int kPfxWarps = PA_PFX_WARPS;  // consumer warps per CTA (plus one loader warp)
constexpr int kPfxNST = PA_PFX_STAGES;   // K/V ring stages shared by the CTA

struct PrefixParams {
    const int32_t *group_start;  // [G+1] member ranges into group_seqs
    const int32_t *group_seqs;   // [num_members] batch rows of the members
    int G, nc, num_members;      // groups, token chunks per group, group_seqs length
};

template <int D>
constexpr size_t prefix_smem_bytes() {
    return kPfxNST * MmaCfg<D, 8>::STAGE + 2 * kPfxNST * 8 + 16 + 1024;
}

template <int D, int GQ>
__global__ void __launch_bounds__((kPfxWarps + 1) * 32)
    prefix_kernel(const DecodeParams p, const PrefixParams pp,
                  const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    using C = MmaCfg<D, GQ>;
    constexpr int MPW = 8 / GQ;              // members per consumer warp
    constexpr int MPC = kPfxWarps * MPW;     // members per CTA
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kPfxNST * C::STAGE);
    uint64_t *empty = full + kPfxNST;
    volatile int *fail = reinterpret_cast<volatile int *>(empty + kPfxNST);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hk = blockIdx.y, g = blockIdx.z / pp.nc, chunk = blockIdx.z % pp.nc;
    wait_prior_grids();

    int mbeg = pp.group_start[g], mend = pp.group_start[g + 1];
    if (mbeg < 0 || mend > pp.num_members || mbeg > mend) {
        if (threadIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
        return;
    }
    const int m0 = mbeg + blockIdx.x * MPC;
    if (m0 >= mend) return;  // uniform over the CTA
    // the first member's block-table row holds the shared blocks
    const int b0 = pp.group_seqs[mbeg];
    int S = 0;
    if (b0 >= 0 && b0 < p.B) {
        S = p.shared_len[b0];
        const int L0 = p.context_lens[b0];
        if (S < 0 || S >= L0 || (S & (p.bs - 1)) || S > (p.MB << p.bs_log2)) S = 0;
    }
    if (S == 0 && threadIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
    const int ch = ((S + 15) / 16 + pp.nc - 1) / pp.nc * 16;  // tokens per chunk
    const int t_lo = min(S, chunk * ch), t_hi = min(S, t_lo + ch);
    const int ntiles = (t_hi - t_lo + 15) / 16;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPfxNST; ++i) {
            pa::mbar_init(&full[i], 1);
            pa::mbar_init(&empty[i], kPfxWarps);
        }
        *fail = 0;
        pa::fence_barrier_init();
    }
    __syncthreads();

    if (warp == kPfxWarps) {
        // ---- loader ------------------------------------------------------
        if (lane == 0 && ntiles > 0) {
            Cursor c{b0, hk, 0, ntiles, t_hi, t_lo};
            int issued = 0;
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % kPfxNST;
                if (i >= kPfxNST && !pa::mbar_wait(&empty[st], ((i / kPfxNST) - 1) & 1)) {
                    pa::record_error(p.err, PA_DEVERR_TIMEOUT);
                    *fail = 1;
                    break;
                }
                c.t = i;
                produce_tile_tma<D, GQ>(p, c, checked_block(p, block_entry<16>(p, c, 0)),
                                        smem + st * C::STAGE, &full[st], &kmap, &vmap);
                issued = i + 1;
            }
            // every copy must have landed before the CTA may exit
            for (int i = max(0, issued - kPfxNST); i < issued; ++i)
                (void)pa::mbar_wait(&full[i % kPfxNST], (i / kPfxNST) & 1);
        }
        return;
    }

    // ---- consumers ---------------------------------------------------------
    MmaAttn<D, GQ> st;
    st.init(lane);
    st.reset();
    // this lane's column g: member m0 + warp * MPW + g / GQ, head g % GQ
    auto col_row = [&](int col) -> int64_t {
        const int m = m0 + warp * MPW + col / GQ;
        if (m >= mend) return -1;
        const int b = pp.group_seqs[m];
        if (b < 0 || b >= p.B || p.shared_len[b] != S || S == 0) {
            pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);  // not a consistent member
            return -1;
        }
        return static_cast<int64_t>(b) * p.Hq + hk * GQ + col % GQ;
    };
    const int64_t qrow = col_row(st.g);
    st.load_q_row(qrow >= 0 ? static_cast<const __nv_bfloat16 *>(p.q) + qrow * D : nullptr,
                  p.qscale);
    for (int i = 0; i < ntiles; ++i) {
        const int sti = i % kPfxNST;
        const bool ok = __all_sync(pa::kFull, pa::mbar_wait(&full[sti], (i / kPfxNST) & 1));
        if (!ok || *fail) {
            if (lane == 0) pa::record_error(p.err, PA_DEVERR_TIMEOUT);
            break;
        }
        const uint32_t kaddr = pa::smem_u32(smem + sti * C::STAGE);
        st.tile(kaddr, kaddr + C::TILE, min(16, t_hi - (t_lo + 16 * i)), nullptr, nullptr);
        __syncwarp();
        if (lane == 0) {
            pa::fence_proxy_async();
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(pa::smem_u32(&empty[sti]))
                         : "memory");
        }
    }
    // ---- partials of this lane's columns 2t, 2t+1 -----------------------------
    float lh[2];
    st.reduce(lh);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int64_t row = col_row(2 * st.t + j);
        if (row < 0) continue;
        const size_t slot = static_cast<size_t>(row) * p.rowslots + p.pslot0 + chunk;
        float *a = p.ws_acc + slot * D + st.g;
#pragma unroll
        for (int m = 0; m < C::KS; ++m) {
            a[16 * m] = st.acc[m][j];
            a[16 * m + 8] = st.acc[m][2 + j];
        }
        if (st.g == 0)
            *reinterpret_cast<float2 *>(p.ws_ml + 2 * slot) = make_float2(st.m_run[j], lh[j]);
    }
}

template <typename T, int D, int GQ, bool MMA>
struct AttnOf {
    using type = WarpAttn<T, D, GQ>;
};
template <int D, int GQ>
struct AttnOf<__nv_bfloat16, D, GQ, true> {
    using type = MmaAttn<D, GQ>;
};
// with forked children: the tile's spare columns carry a child's heads
template <typename T, int D, int GQ, bool MMA, bool FORK>
struct KernelAttn {
    using type = typename AttnOf<T, D, GQ, MMA>::type;
};
template <int D, int GQ>
struct KernelAttn<__nv_bfloat16, D, GQ, true, true> {
    using type = MmaAttn<D, GQ, 2 * GQ>;
};

// MMA: the tensor-core tile (K/V by 2D tensor copies through kmap / vmap);
// otherwise the CUDA-core tile (bulk copies; the maps are not read).
// FORK (tensor-core tile, groups of at most 4 heads): a forked child's heads
// ride in the spare columns of its parent's items over the blocks they share
// (pa_decode_shared_forks); the child's own items start at its fork point.
template <typename T, int D, int GQ, bool MMA, bool FORK = false>
__global__ void __launch_bounds__(kWarps * 32, (AttnOf<T, D, GQ, MMA>::type::C::MINB))
    decode_persistent_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap) {
    static_assert(!FORK || (MMA && 2 * GQ <= 8), "forks ride in the tensor-core tile's columns");
    using St = typename KernelAttn<T, D, GQ, MMA, FORK>::type;
    using C = typename St::C;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // swizzled tensor copies need 1024-byte aligned stages
    uint8_t *smem = MMA ? reinterpret_cast<uint8_t *>(
                              (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))
                        : smem_raw;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *ring = smem + warp * C::WARP_SMEM;
    float *pbuf = reinterpret_cast<float *>(smem + C::OFF_P) + warp * 2 * C::TT * GQ;
    float *sbuf = pbuf + C::TT * GQ;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR) + warp * C::NST;
    int *scan = reinterpret_cast<int *>(smem + C::OFF_FLAG);
    int32_t *pre = reinterpret_cast<int32_t *>(smem + C::OFF_BT);  // [B+1] tile prefix
    int32_t *lens = pre + p.B + 1;                                  // [B]
    int32_t *starts = lens + p.B;                                   // [B]
    int32_t *slen = starts + p.B;     // FORK: [B] validated shared_len
    int32_t *child = slen + p.B;      // FORK: [B] child served by the row's items
    int32_t *parent = child + p.B;    // FORK: [B] parent serving the row's fork range
    wait_prior_grids();  // inputs are ready past this point
    // With the shared-prefix kernel behind this grid: that kernel launches
    // once every CTA of this grid has passed this point, so its CTAs take the
    // SMs this grid leaves as it drains (it reads none of this grid's results
    // and waits for it before it exits).  The merge otherwise launches at
    // this grid's end (launched early, its waiting CTAs slowed the 8B step).
    if (p.early_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr bool kLanes = PA_DECODE_LOADER != 0 && !MMA;

    // ---- tiles per sequence and their prefix sums (whole CTA) ---------------
    const int cap = p.MB << p.bs_log2;
    int carry = 0;
    // Every sequence's context length and shared length into the tables first,
    // eight independent loads per thread at a time: one memory latency per
    // 8 x blockDim sequences (not one per blockDim behind two CTA barriers).
    for (int b0 = threadIdx.x; b0 < p.B; b0 += 8 * blockDim.x) {
        int Lv[8], Sv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int b = b0 + u * blockDim.x;
            Lv[u] = b < p.B ? p.context_lens[b] : 1;
            Sv[u] = b < p.B && p.shared_len ? p.shared_len[b] : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int b = b0 + u * blockDim.x;
            if (b >= p.B) break;
            int L = Lv[u];
            if (L < 1 || L > cap) {
                if (blockIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
                L = L < 1 ? 0 : cap;
            }
            // tokens before S are covered by the sequence's shared-prefix
            // partials (a multiple of the block size, below L; else none)
            int S = Sv[u];
            if (S < 0 || S >= L || (S & (p.bs - 1))) {
                if (S != 0 && blockIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
                S = 0;
            }
            lens[b] = L;
            starts[b] = S;
        }
    }
    __syncthreads();
    if constexpr (FORK) {
        for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
            slen[b] = starts[b];
            child[b] = 0x7fffffff;
            parent[b] = -1;
        }
        __syncthreads();
        // A child takes its parent when both have the same shared length, its
        // fork length is a multiple of the block size in [S, both lengths),
        // and the parent is no child itself; of several children of one
        // parent the lowest row (same choice in every CTA).  Others decode
        // their fork range themselves.
        auto fork_ok = [&](int c) {
            const int par = p.fork_parent[c];
            if (par < 0) return false;
            const int F = p.fork_len[c];
            const bool ok = par < p.B && par != c && p.fork_parent[par] < 0 && F > 0 &&
                            !(F & (p.bs - 1)) && F >= slen[c] && F < lens[c] && F < lens[par] &&
                            slen[par] == slen[c];
            if (!ok && blockIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            return ok;
        };
        for (int c = threadIdx.x; c < p.B; c += blockDim.x)
            if (fork_ok(c)) atomicMin(&child[p.fork_parent[c]], c);
        __syncthreads();
        for (int c = threadIdx.x; c < p.B; c += blockDim.x) {
            const int par = p.fork_parent[c];
            if (par < 0) continue;
            if (par < p.B && par != c && child[par] == c) {
                parent[c] = par;
                starts[c] = p.fork_len[c];
            } else if (blockIdx.x == 0) {  // an invalid fork, or a parent's second child
                pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            }
        }
        __syncthreads();
        for (int b = threadIdx.x; b < p.B; b += blockDim.x)
            if (child[b] == 0x7fffffff) child[b] = -1;
        __syncthreads();
    }
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int nt = b < p.B ? (lens[b] - starts[b] + C::TT - 1) / C::TT : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(pa::kFull, nt, o);
            if (lane >= o) nt += y;
        }
        if (lane == 31) scan[warp] = nt;
        __syncthreads();
        int off = carry, total = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) {
            off += w2 < warp ? scan[w2] : 0;
            total += scan[w2];
        }
        if (b < p.B) pre[b + 1] = off + nt;
        carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) pre[0] = 0;
    if (lane == 0) {
        for (int s = 0; s < C::NST; ++s) pa::mbar_init(&bars[s], kLanes ? 32 : 1);
        pa::fence_barrier_init();
    }
    __syncthreads();
    const BatchTables bt{pre, lens, starts};
    const ForkTables ft{slen, child, parent};
    constexpr int QH = FORK ? 2 * GQ : GQ;
    auto child_of = [&](const Cursor &c) { return FORK ? child[c.b] : -1; };

    // ---- this warp's range of units ------------------------------------------
    const int64_t U = int64_t(p.Hkv) * pre[p.B];
    const int64_t W = int64_t(gridDim.x) * kWarps;
    int64_t per = (U + W - 1) / W;
    const int64_t pmin = p.PT / C::TT;
    if (per < pmin) per = pmin;
    const int64_t w = int64_t(blockIdx.x) * kWarps + warp;
    const int64_t u0 = w * per;
    if (u0 >= U) return;  // warp-uniform; no CTA barrier follows
    const int my_n = static_cast<int>(min(per, U - u0));

    St st;
    st.init(lane);
    st.qs = reinterpret_cast<float *>(smem + C::OFF_Q) + warp * GQ * D;
    const T *qbase = static_cast<const T *>(p.q);

    // ---- pipeline prologue ----------------------------------------------------
    Cursor pc = locate_unit(u0, bt, p.B, p.Hkv);  // next tile to produce
    Cursor cc = pc;                               // next tile to consume
    int pend = 0;  // raw block-table entry of pc's tile (lane 0, or every lane)
    if (kLanes || lane == 0) pend = block_entry<C::TT>(p, pc, 0);
    const int npro = min(C::NST, my_n);
    for (int i = 0; i < npro; ++i) {
        if constexpr (MMA) {
            if (lane == 0)
                produce_tile_tma<D, GQ, QH>(p, pc, checked_block(p, pend), ring + i * C::STAGE,
                                            &bars[i], &kmap, &vmap, i == 0 || pc.t == 0,
                                            child_of(pc));
        } else if (kLanes) {
            produce_tile_lanes<T, D, GQ>(p, pc, checked_block(p, pend), ring + i * C::STAGE,
                                         &bars[i], lane);
        } else if (lane == 0) {
            produce_tile<T, D, GQ>(p, pc, checked_block(p, pend), ring + i * C::STAGE, &bars[i]);
        }
        if (!MMA && i > 0 && pc.t == 0) prefetch_q<T, D, GQ>(p, pc, lane);
        pc = next_unit(pc, bt, p.B, p.Hkv);
        if ((kLanes || lane == 0) && i + 1 < my_n) pend = block_entry<C::TT>(p, pc, 0);
    }

    int failed_at = -1;
    for (int i = 0; i < my_n; ++i) {
        const int s = i % C::NST;
        const bool ok = __all_sync(pa::kFull, pa::mbar_wait(&bars[s], (i / C::NST) & 1));
        if (!ok) {
            failed_at = i;
            break;
        }
        const uint32_t kaddr = pa::smem_u32(ring + s * C::STAGE);
        if (i == 0 || cc.t == 0) {
            st.reset();
            if constexpr (MMA)  // q came with this tile (and the child's, if any)
                st.load_q_smem(kaddr + 2 * C::TILE, p.qscale, child_of(cc) >= 0 ? QH : GQ);
            else
                st.load_q(qbase + (static_cast<size_t>(cc.b) * p.Hq + cc.hk * GQ) * D, p.qscale);
        }
        const int tok0 = first_token(cc, C::TT);
        if constexpr (FORK) {
            // the child's heads see the tile's tokens below its fork point
            const int cr = child[cc.b];
            const int nhi = cr >= 0 ? max(0, min(C::TT, starts[cr] - tok0)) : 0;
            st.tile(kaddr, kaddr + C::TILE, min(C::TT, cc.L - tok0), pbuf, sbuf, nhi);
        } else {
            st.tile(kaddr, kaddr + C::TILE, min(C::TT, cc.L - tok0), pbuf, sbuf);
        }
        __syncwarp();
        if (i + C::NST < my_n) {
            if constexpr (MMA) {
                if (lane == 0) {
                    pa::fence_proxy_async();
                    produce_tile_tma<D, GQ, QH>(p, pc, checked_block(p, pend), ring + s * C::STAGE,
                                                &bars[s], &kmap, &vmap, pc.t == 0, child_of(pc));
                }
            } else if (kLanes) {
                produce_tile_lanes<T, D, GQ>(p, pc, checked_block(p, pend), ring + s * C::STAGE,
                                             &bars[s], lane);
            } else if (lane == 0) {
                pa::fence_proxy_async();
                produce_tile<T, D, GQ>(p, pc, checked_block(p, pend), ring + s * C::STAGE,
                                       &bars[s]);
            }
            if (!MMA && pc.t == 0) prefetch_q<T, D, GQ>(p, pc, lane);
            pc = next_unit(pc, bt, p.B, p.Hkv);
            if ((kLanes || lane == 0) && i + C::NST + 1 < my_n)
                pend = block_entry<C::TT>(p, pc, 0);
        }
        if (cc.t == cc.nt - 1 || i == my_n - 1)
            finish_segment<T, D, GQ, FORK>(st, p, bt, cc, per, w, lane, ft);
        cc = next_unit(cc, bt, p.B, p.Hkv);
    }
    if (failed_at >= 0) {
        // A copy never completed: record it and wait (bounded) for this warp's
        // other copies in flight so none lands after the CTA exits.
        if (lane == 0) {
            pa::record_error(p.err, PA_DEVERR_TIMEOUT);
            const int last = min(failed_at + C::NST, my_n);
            for (int i = failed_at + 1; i < last; ++i)
                (void)pa::mbar_wait(&bars[i % C::NST], (i / C::NST) & 1);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// Grid kernel for batches too large for the persistent kernel's tables:
// one CTA of kWarps warps per (sequence, KV head, partition of PT tokens).
// ---------------------------------------------------------------------------
template <typename T, int D, int GQ>
__global__ void __launch_bounds__(kWarps * 32, (Cfg<T, D, GQ>::MINB)) decode_kernel(const DecodeParams p) {
    using C = Cfg<T, D, GQ>;
    extern __shared__ __align__(128) uint8_t smem[];

    const int part = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int cap = p.MB << p.bs_log2;
    wait_prior_grids();
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

    WarpAttn<T, D, GQ> st;
    st.init(lane);
    st.qs = reinterpret_cast<float *>(smem + C::OFF_Q) + warp * GQ * D;
    st.reset();
    st.load_q(static_cast<const T *>(p.q) + (static_cast<size_t>(b) * p.Hq + hk * GQ) * D,
              p.qscale);

    if (lane == 0)
        for (int i = 0; i < min(C::NST, my_ntiles); ++i) issue(i);

    int failed_at = -1;
    for (int i = 0; i < my_ntiles; ++i) {
        const int s = i % C::NST;
        const bool ok = __all_sync(pa::kFull, pa::mbar_wait(&bars[s], (i / C::NST) & 1));
        if (!ok) {
            failed_at = i;
            break;
        }
        const int nvalid = min(C::TT, ntok - (warp + i * kWarps) * C::TT);
        const uint32_t kaddr = pa::smem_u32(ring + s * C::STAGE);
        st.tile(kaddr, kaddr + C::TILE, nvalid, pbuf, sbuf);
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

    // the merge kernel may start launching once every CTA is past its stream
    // (programmatic dependent launch; it waits for this grid's results)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    float lh[GQ];
    st.reduce(lh);

    // ---- CTA merge of the warps' (max, sum, acc) ----------------------------
    __syncthreads();  // every ring is drained: reuse it as the merge buffer
    float *wacc = reinterpret_cast<float *>(ring);  // [GQ][D]
    float *wml = wacc + GQ * D;                     // max[GQ], sum[GQ]
    if (st.grp == 0) {
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int c = 0; c < C::CPL; ++c)
#pragma unroll
                for (int j = 0; j < C::EPC / 2; ++j)
                    *reinterpret_cast<float2 *>(wacc + h * D + st.dim_of(c, j)) =
                        st.acc[h][c * C::EPC / 2 + j];
    }
    if (lane == 0)
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            wml[h] = st.m_run[h];
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
    // launched as a programmatic dependent of decode_kernel: wait until that
    // grid has completed and its partials are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
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

// Merge of the persistent kernel's partials: one warp per (sequence,
// query head) of item blockIdx.x = b * Hkv + hk merges the item's segment
// partials and its shared-prefix partials by log-sum-exp.  Launched as a
// programmatic dependent of the decode grid; waits for it before reading.
template <typename T, int D, int GQ>
__global__ void __launch_bounds__(GQ * 32) partial_merge_kernel(const DecodeParams p) {
    constexpr int EL = D / 32;
    constexpr int kSpec = 8;  // segment slots loaded before the item's count is known
    constexpr int kSpecP = 4; // shared-prefix slots loaded likewise (p.npfx of them)
    const int item = blockIdx.x, h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    wait_prior_grids();
    // a kernel launched behind this one as a programmatic dependent (the
    // persistent prefill) may start its set-up while the merge drains; it
    // waits for this grid before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const size_t row = static_cast<size_t>(item / p.Hkv) * p.Hq + (item % p.Hkv) * GQ + h;
    const size_t sb = row * p.rowslots;
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml) + sb;
    const float *src = p.ws_acc + sb * D + EL * lane;
    // One round trip for the common case (at most kSpec segments and at most
    // kSpecP shared-prefix partials): the count, the (max, sum) of segment
    // slots 0..kSpec-1 and of the prefix slots, and this lane's values of
    // them are all requested at once.  Lane / index i < kSpec stands for
    // segment slot i, kSpec + k for prefix slot pslot0 + k.
    // batches with shared-prefix partials have short private parts (one or
    // two segments per item): fewer speculative segment slots there
    const int spec = min(p.npfx > 0 ? 2 : kSpec, p.pslot0);
    const int specp = p.npfx <= kSpecP ? p.npfx : 0;
    auto spec_slot = [&](int i) { return i < kSpec ? i : p.pslot0 + (i - kSpec); };
    auto spec_on = [&](int i) { return i < kSpec ? i < spec : i - kSpec < specp; };
    const unsigned meta = __ldcg(p.meta + item);
    float2 v = make_float2(-INFINITY, 0.f);
    if (lane < kSpec + kSpecP && spec_on(lane)) v = __ldcg(&ml[spec_slot(lane)]);
    float pre[kSpec + kSpecP][EL];
#pragma unroll
    for (int i = 0; i < kSpec + kSpecP; ++i) {
        if (spec_on(i)) {
            if constexpr (EL == 4) {
                const float4 a = __ldcg(reinterpret_cast<const float4 *>(src + spec_slot(i) * D));
                pre[i][0] = a.x;
                pre[i][1] = a.y;
                pre[i][2] = a.z;
                pre[i][3] = a.w;
            } else {
                const float2 a = __ldcg(reinterpret_cast<const float2 *>(src + spec_slot(i) * D));
                pre[i][0] = a.x;
                pre[i][1] = a.y;
            }
        }
    }
    const int nseg = static_cast<int>(meta & 0xffffu), ns = nseg + static_cast<int>(meta >> 16);
    if (ns == 0) return;  // written out by the decode
    float acc[EL];
#pragma unroll
    for (int e = 0; e < EL; ++e) acc[e] = 0.f;
    float den = 0.f, M = -INFINITY;
    const int npre = ns - nseg;
    if (nseg <= spec && (npre == 0 || npre == specp)) {
        // lanes in use: segments 0..nseg-1 and the npre prefix slots
        const bool used = lane < kSpec ? lane < nseg : (lane < kSpec + kSpecP && lane - kSpec < npre);
        if (!used) v = make_float2(-INFINITY, 0.f);
        M = v.x;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(pa::kFull, M, o));
        const float wl = used && v.x != -INFINITY ? exp2f(v.x - M) : 0.f;
        den = wl * v.y;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(pa::kFull, den, o);
#pragma unroll
        for (int i = 0; i < kSpec + kSpecP; ++i) {
            const float f = __shfl_sync(pa::kFull, wl, i);
            if (i < kSpec ? i < nseg : i - kSpec < npre)
#pragma unroll
                for (int e = 0; e < EL; ++e) acc[e] += f * pre[i][e];
        }
    } else {
        // 32 partials at a time: lane s holds partial s's (max, sum); the
        // weights travel by shuffle and every value load is independent
        for (int base = 0; base < ns; base += 32) {
            const int k = min(32, ns - base);
            float2 w2 = make_float2(-INFINITY, 0.f);
            if (lane < k) w2 = __ldcg(&ml[slot_of(p, base + lane, nseg)]);
            float Mc = w2.x;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(pa::kFull, Mc, o));
            const float Mn = fmaxf(M, Mc);
            const float rescale = M == -INFINITY ? 0.f : exp2f(M - Mn);
            M = Mn;
            const float wl = lane < k ? exp2f(w2.x - M) : 0.f;
            float d = wl * w2.y;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(pa::kFull, d, o);
            den = den * rescale + d;
#pragma unroll
            for (int e = 0; e < EL; ++e) acc[e] *= rescale;
#pragma unroll 8
            for (int i = 0; i < k; ++i) {
                const float f = __shfl_sync(pa::kFull, wl, i);
                const float *sp = src + static_cast<size_t>(slot_of(p, base + i, nseg)) * D;
                if constexpr (EL == 4) {
                    const float4 a = __ldcg(reinterpret_cast<const float4 *>(sp));
                    acc[0] += f * a.x;
                    acc[1] += f * a.y;
                    acc[2] += f * a.z;
                    acc[3] += f * a.w;
                } else {
                    const float2 a = __ldcg(reinterpret_cast<const float2 *>(sp));
                    acc[0] += f * a.x;
                    acc[1] += f * a.y;
                }
            }
        }
    }
    const float inv = 1.f / den;
    T *out = static_cast<T *>(p.out) + row * D + EL * lane;
#pragma unroll
    for (int e = 0; e < EL; e += 2) store_pair<T>(out + e, acc[e] * inv, acc[e + 1] * inv);
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

// Launch `kern` as a programmatic dependent of the previous kernel in the
// stream: its CTAs may start while that kernel drains and wait for it with
// griddepcontrol.wait.
#ifndef PA_DECODE_PDL
#define PA_DECODE_PDL 1  // 0: ordinary stream-ordered launches (A/B of the dependent launch)
#endif
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PA_DECODE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

struct SharedPlan;
int launch_prefix_any(const DecodeParams &p, const SharedPlan &sp, int D, bool after_decode,
                      cudaStream_t stream);

template <typename T, int D, int GQ, bool MMA, bool FORK = false>
int launch_persistent(const DecodeParams &p, cudaStream_t stream,
                      const SharedPlan *prefix_after = nullptr) {
    using C = typename KernelAttn<T, D, GQ, MMA, FORK>::type::C;
    const size_t smem =
        C::OFF_BT + sizeof(int32_t) * ((FORK ? 6 : 3) * p.B + 1) + (MMA ? 1024 : 0);
    auto kern = decode_persistent_kernel<T, D, GQ, MMA, FORK>;
    CUtensorMap kmap{}, vmap{};
    if constexpr (MMA) {
        const int64_t rows = p.num_blocks * p.Hkv * p.bs;
        const int box = std::min(MmaCfg<D, GQ>::TT, p.bs);
        if (int rc = pa::pool_tensor_map(&kmap, p.k_cache, rows, D, box)) return rc;
        if (int rc = pa::pool_tensor_map(&vmap, p.v_cache, rows, D, box)) return rc;
    }
    (void)cudaGetLastError();  // drop a stale error that is not ours
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode: shared memory attribute");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode: occupancy");
    // the split of the work (and the register budget) is designed for MINB
    // CTAs per SM; more would only add split items (measured slower)
    per_sm = std::min(per_sm, C::MINB);
#ifdef PA_DECODE_FORCE_PER_SM
    per_sm = PA_DECODE_FORCE_PER_SM;
#endif
    const int sms = sm_count();
    if (sms <= 0) return pa::fail(PA_ERR_CUDA, "decode: no SM count");
    const int grid = sms * std::max(per_sm, 1);
    DecodeParams pk = p;
    pk.early_dependents = prefix_after ? 1 : 0;
    e = launch_dependent(kern, dim3(grid), dim3(kWarps * 32), smem, stream, pk, kmap, vmap);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode launch");
    if (int rc = pa::check_launch("decode launch")) return rc;
    // shared-prefix partials on the tcgen05 kernel go behind the decode grid:
    // they read none of its results, so their CTAs take the SMs its CTAs
    // leave; the merge behind them then finds both complete
    if (prefix_after)
        if (int rc = launch_prefix_any(p, *prefix_after, D, true, stream)) return rc;
    const int64_t items = int64_t(p.B) * p.Hkv;
    e = launch_dependent(partial_merge_kernel<T, D, GQ>, dim3(static_cast<unsigned>(items)),
                         dim3(GQ * 32), 0, stream, p);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode merge launch");
    return pa::check_launch("decode merge launch");
}

// The tensor-core tile serves bf16 groups of 4 or 8 heads whose pool rows
// are addressable by 32-bit tensor-copy coordinates.  Measured on the 8B
// batch (groups of 4): 98.9 us per step against 104.0 with the CUDA-core
// tile; on the 70B batch (groups of 8): 495 against 928 us.
bool tile_is_mma(int gq, int dtype, int64_t num_blocks, int Hkv, int bs) {
    return dtype == PA_BF16 && gq >= PA_DECODE_MMA_MIN_GQ && gq <= 8 && gq % 2 == 0 &&
           num_blocks * Hkv * bs <= int64_t(INT32_MAX);
}

template <typename T, int GQ>
bool use_mma(const DecodeParams &p) {
    return tile_is_mma(GQ, std::is_same<T, __nv_bfloat16>::value ? PA_BF16 : PA_F32,
                       p.num_blocks, p.Hkv, p.bs);
}

template <typename T, int D, int GQ>
int launch_grid(const DecodeParams &p, cudaStream_t stream) {
    using C = Cfg<T, D, GQ>;
    const size_t smem = C::OFF_BT + sizeof(int32_t) * (p.PT / p.bs + 1);
    auto kern = decode_kernel<T, D, GQ>;
    (void)cudaGetLastError();  // drop a stale error that is not ours
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode: shared memory attribute");
    // both launches are programmatic dependents: the decode grid's launch
    // overlaps the previous kernel's tail, the merge kernel's the decode's
    e = launch_dependent(kern, dim3(p.max_parts, p.Hkv, p.B), dim3(kWarps * 32), smem, stream, p);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode launch");
    if (int rc = pa::check_launch("decode launch")) return rc;
    if (p.max_parts > 1) {
        e = launch_dependent(merge_kernel<T, D>, dim3(p.Hq, p.B), dim3(D), 0, stream, p);
        if (e != cudaSuccess) return pa::cuda_fail(e, "decode merge launch");
        if (int rc = pa::check_launch("decode merge launch")) return rc;
    }
    return PA_OK;
}

// Which kernel a batch runs on; sizes only, so the host decides without
// reading device data.  The persistent kernel needs the batch's tile counts in
// shared memory and 32-bit tile prefix sums.  A batch with little work runs on
// the grid kernel: there every (sequence, KV head, partition) gets a CTA of
// four warps, while the persistent split leaves a partition to one warp (its
// tiles streamed one after another) and an item's segments to one merging
// warp.  Measured with 512-token partitions, 32 query / 8 KV heads, d 128,
// 16-token blocks and 4096-token tables: grid against persistent kernel 20.3
// against 53.2 us at 1 sequence, 25.6 against 53.2 at 8, 69.3 against 69.6 at
// 32, 76.6 at 38 against 71.1 at 39; 64 query heads, 32-token blocks and
// 32k-token tables: 63.6 against 155.7 us at 1, 151.1 against 190.5 at 4,
// 233 against 231 at 8 (with the merge as an ordinary second launch; as a
// programmatic dependent launch it takes another 2.5-3.4 us off the grid
// side).  Rule: the grid kernel while its CTA count, bounded by the table
// capacity, is at most 1.75 times the persistent grid's warps.
int kernel_for(int B, int Hkv, int MB, int bs_log2, int partitions, int sms) {
    if (B > kPersistentMaxB || int64_t(B) * (int64_t(MB) << bs_log2) / 8 >= (1ll << 31))
        return PA_DECODE_GRID;
    const int64_t grid_ctas = int64_t(B) * Hkv * partitions;
    return 4 * grid_ctas <= 7ll * sms * kMinCtas * kWarps ? PA_DECODE_GRID : PA_DECODE_PERSISTENT;
}

template <int D, int GQ>
int launch_prefix(const DecodeParams &p, const PrefixParams &pp, int max_group_size,
                  cudaStream_t stream) {
    constexpr int MPC = kPfxWarps * (8 / GQ);
    CUtensorMap kmap{}, vmap{};
    const int64_t rows = p.num_blocks * p.Hkv * p.bs;
    const int box = std::min(MmaCfg<D, GQ>::TT, p.bs);
    if (int rc = pa::pool_tensor_map(&kmap, p.k_cache, rows, D, box)) return rc;
    if (int rc = pa::pool_tensor_map(&vmap, p.v_cache, rows, D, box)) return rc;
    const size_t smem = prefix_smem_bytes<D>();
    auto kern = prefix_kernel<D, GQ>;
    (void)cudaGetLastError();
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode_shared: shared memory attribute");
    const dim3 grid((max_group_size + MPC - 1) / MPC, p.Hkv, pp.G * pp.nc);
    e = launch_dependent(kern, grid, dim3((kPfxWarps + 1) * 32), smem, stream, p, pp, kmap, vmap);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode_shared: prefix launch");
    return pa::check_launch("decode_shared: prefix launch");
}

// Shared-prefix work of a call (pa_decode_shared), or none.
struct SharedPlan {
    PrefixParams pp;
    int max_group_size;
    bool tc;  // tcgen05 prefill kernel in prefix mode, else prefix_kernel
};

int launch_prefix_any(const DecodeParams &p, const SharedPlan &sp, int D, bool after_decode,
                      cudaStream_t stream) {
    pa::PrefixTcArgs a{};
    a.after_decode = after_decode;
    a.q = p.q;
    a.k_cache = p.k_cache;
    a.v_cache = p.v_cache;
    a.block_table = p.block_table;
    a.context_lens = p.context_lens;
    a.group_start = sp.pp.group_start;
    a.group_seqs = sp.pp.group_seqs;
    a.shared_len = p.shared_len;
    a.acc = p.ws_acc;
    a.ml = p.ws_ml;
    a.err = p.err;
    a.num_blocks = p.num_blocks;
    a.B = p.B;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.D = D;
    a.bs = p.bs;
    a.MB = p.MB;
    a.G = sp.pp.G;
    a.nc = sp.pp.nc;
    a.max_group_size = sp.max_group_size;
    a.num_members = sp.pp.num_members;
    a.rowslots = p.rowslots;
    a.pslot0 = p.pslot0;
    a.qscale = p.qscale;
    return pa::launch_prefix_tc(a, stream);
}

template <typename T, int D, int GQ>
int launch(const DecodeParams &p, const SharedPlan *sp, cudaStream_t stream) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        if (sp) {  // the host checked: bf16, persistent kernel, 32-bit pool rows
            // the tcgen05 prefix kernel runs behind the decode grid, the
            // warp-level one before it
            const SharedPlan *after = sp->tc ? sp : nullptr;
            if (!sp->tc)
                if (int rc = launch_prefix<D, GQ>(p, sp->pp, sp->max_group_size, stream)) return rc;
            if constexpr (GQ % 2 == 0 && GQ >= PA_DECODE_MMA_MIN_GQ)
                if (use_mma<T, GQ>(p)) {
                    if constexpr (2 * GQ <= 8)
                        if (p.fork_parent)
                            return launch_persistent<T, D, GQ, true, true>(p, stream, after);
                    return launch_persistent<T, D, GQ, true>(p, stream, after);
                }
            return launch_persistent<T, D, GQ, false>(p, stream, after);
        }
        // forked children without shared-prefix groups (the host checked:
        // persistent kernel, tensor-core tile, groups of at most 4 heads)
        if constexpr (GQ % 2 == 0 && GQ >= PA_DECODE_MMA_MIN_GQ && 2 * GQ <= 8)
            if (p.fork_parent) return launch_persistent<T, D, GQ, true, true>(p, stream);
    }
    const int sms = sm_count();
    if (sms <= 0) return pa::fail(PA_ERR_CUDA, "decode: no SM count");
    if (!p.contig_len &&
        kernel_for(p.B, p.Hkv, p.MB, p.bs_log2, p.max_parts - 1, sms) != PA_DECODE_PERSISTENT)
        return launch_grid<T, D, GQ>(p, stream);
    if constexpr (std::is_same<T, __nv_bfloat16>::value && GQ % 2 == 0 &&
                  GQ >= PA_DECODE_MMA_MIN_GQ)
        if (use_mma<T, GQ>(p)) return launch_persistent<T, D, GQ, true>(p, stream);
    return launch_persistent<T, D, GQ, false>(p, stream);
}

template <typename T, int D>
int dispatch_gq(int gq, const DecodeParams &p, const SharedPlan *sp, cudaStream_t s) {
    switch (gq) {
        case 1: return launch<T, D, 1>(p, sp, s);
        case 2: return launch<T, D, 2>(p, sp, s);
        case 4: return launch<T, D, 4>(p, sp, s);
        case 8: return launch<T, D, 8>(p, sp, s);
        default: return pa::fail(PA_ERR_UNSUPPORTED, "decode: Hq/Hkv=%d unsupported", gq);
    }
}

// Workspace layout: per-item partial counts u32 [B][Hq] (the persistent
// kernel uses [B][Hkv] of them) padded to a multiple of 256 bytes, then acc fp32
// [B][Hq][maxseg][D], then (max, sum) fp32 [B][Hq][maxseg][2]; maxseg =
// partitions per sequence + 1 bounds the segments of one item in the
// persistent kernel and the partitions of the grid kernel.  The padding keeps
// the fp32 regions 256-byte aligned whatever B*Hq is (the merge reads them as
// float4).  Every product is checked: false when the size does not fit size_t.
constexpr size_t kWsAlign = 256;
struct WsLayout {
    size_t meta_bytes, acc_bytes, ml_bytes, total;
};

bool workspace_layout(int64_t B, int64_t Hq, int64_t D, int64_t maxseg, WsLayout *l) {
    *l = WsLayout{0, 0, 0, 0};
    if (B <= 0) return true;
    size_t rows, tick, acc, ml, t;
    if (__builtin_mul_overflow(static_cast<size_t>(B), static_cast<size_t>(Hq), &rows) ||
        __builtin_mul_overflow(rows, sizeof(unsigned), &tick) ||
        __builtin_add_overflow(tick, kWsAlign - 1, &tick))
        return false;
    tick -= tick % kWsAlign;
    if (__builtin_mul_overflow(rows, static_cast<size_t>(maxseg), &rows) ||
        __builtin_mul_overflow(rows, static_cast<size_t>(D) * sizeof(float), &acc) ||
        __builtin_mul_overflow(rows, 2 * sizeof(float), &ml) ||
        __builtin_add_overflow(tick, acc, &t) || __builtin_add_overflow(t, ml, &t))
        return false;
    *l = WsLayout{tick, acc, ml, t};
    return true;
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
    const int64_t maxseg = (cap + pt - 1) / pt + 1;
    WsLayout l;
    if (!workspace_layout(B, Hq, head_dim, maxseg, &l))
        return pa::fail(PA_ERR_INVALID, "workspace_size: size does not fit in size_t");
    *bytes = l.total;
    return PA_OK;
}

int pa_decode_kernel_for(int B, int Hkv, int max_blocks_per_seq, int block_size,
                         int partition_tokens, int *kernel) {
    pa::clear_error();
    if (!kernel) return pa::fail(PA_ERR_INVALID, "decode_kernel_for: kernel is NULL");
    if (B < 0 || Hkv <= 0 || max_blocks_per_seq <= 0 || !pa::pow2_in(block_size, 8, 128))
        return pa::fail(PA_ERR_INVALID, "decode_kernel_for: bad sizes");
    const int pt = resolve_partition(partition_tokens);
    if (!partition_ok(pt, block_size))
        return pa::fail(PA_ERR_INVALID, "decode_kernel_for: bad partition_tokens %d", pt);
    const int sms = sm_count();
    if (sms <= 0) return pa::fail(PA_ERR_CUDA, "decode_kernel_for: no SM count");
    const int64_t cap = int64_t(max_blocks_per_seq) * block_size;
    *kernel = kernel_for(B, Hkv, max_blocks_per_seq, log2_int(block_size),
                         static_cast<int>((cap + pt - 1) / pt), sms);
    return PA_OK;
}

int pa_decode_tile_for(int Hq, int Hkv, int head_dim, int block_size, int64_t num_blocks,
                       int dtype, int *tile) {
    pa::clear_error();
    if (!tile) return pa::fail(PA_ERR_INVALID, "decode_tile_for: tile is NULL");
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || (head_dim != 64 && head_dim != 128) ||
        !pa::pow2_in(block_size, 8, 128) || num_blocks <= 0 ||
        (dtype != PA_BF16 && dtype != PA_F32))
        return pa::fail(PA_ERR_INVALID, "decode_tile_for: bad sizes");
    *tile = tile_is_mma(Hq / Hkv, dtype, num_blocks, Hkv, block_size) ? PA_DECODE_TILE_TENSOR_CORE
                                                                      : PA_DECODE_TILE_CUDA_CORE;
    return PA_OK;
}

}  // extern "C"

namespace {

// Groups of a pa_decode_shared call (NULL for pa_decode).
struct SharedArgs {
    const int32_t *shared_len, *group_start, *group_seqs;
    int G, num_members, max_group_size, max_shared_len;
    const int32_t *fork_parent = nullptr, *fork_len = nullptr;  // pa_decode_shared_forks
};

constexpr int kPfxChunkMin = 256;  // tokens: the prefix slots bound is max_shared_len / this

int prefix_slots_for(int max_shared_len) {
    return max_shared_len > 0 ? (max_shared_len + kPfxChunkMin - 1) / kPfxChunkMin : 0;
}

int validate_groups(const SharedArgs &sh, const int32_t *context_lens, const int32_t *block_table,
                    int B, int MB, int bs, cudaStream_t stream) {
    std::vector<int32_t> lens(B), S(B), gs(sh.G + 1), mem(sh.num_members),
        table(size_t(B) * MB);
    if (int rc = pa::fetch(lens.data(), context_lens, B * sizeof(int32_t), stream)) return rc;
    if (int rc = pa::fetch(S.data(), sh.shared_len, B * sizeof(int32_t), stream)) return rc;
    if (int rc = pa::fetch(gs.data(), sh.group_start, gs.size() * sizeof(int32_t), stream))
        return rc;
    if (sh.num_members > 0)
        if (int rc = pa::fetch(mem.data(), sh.group_seqs, mem.size() * sizeof(int32_t), stream))
            return rc;
    if (int rc = pa::fetch(table.data(), block_table, table.size() * sizeof(int32_t), stream))
        return rc;
    std::vector<int> group_of(B, -1);
    for (int g = 0; g < sh.G; ++g) {
        if (gs[g] < 0 || gs[g + 1] < gs[g] || gs[g + 1] > sh.num_members)
            return pa::fail(PA_ERR_INVALID, "validate: group_start[%d..%d] out of range", g, g + 1);
        if (gs[g + 1] - gs[g] > sh.max_group_size)
            return pa::fail(PA_ERR_INVALID, "validate: group %d larger than max_group_size", g);
        for (int m = gs[g]; m < gs[g + 1]; ++m) {
            const int b = mem[m];
            if (b < 0 || b >= B) return pa::fail(PA_ERR_INVALID, "validate: member %d not in batch", b);
            if (group_of[b] >= 0)
                return pa::fail(PA_ERR_INVALID, "validate: sequence %d in two groups", b);
            group_of[b] = g;
            const int b0 = mem[gs[g]];
            if (S[b] != S[b0] || S[b] <= 0 || S[b] % bs || S[b] >= lens[b] ||
                S[b] > sh.max_shared_len)
                return pa::fail(PA_ERR_INVALID,
                                "validate: shared_len[%d]=%d (group %d: positive, a multiple of "
                                "block_size, below the context length, equal in the group)",
                                b, S[b], g);
            for (int i = 0; i < S[b] / bs; ++i)
                if (table[size_t(b) * MB + i] != table[size_t(b0) * MB + i])
                    return pa::fail(PA_ERR_INVALID,
                                    "validate: sequence %d does not share block %d of group %d", b,
                                    i, g);
        }
    }
    for (int b = 0; b < B; ++b)
        if (group_of[b] < 0 && S[b] != 0)
            return pa::fail(PA_ERR_INVALID, "validate: shared_len[%d] != 0 outside any group", b);
    return PA_OK;
}

// Validate mode: a child names a parent row (no child itself) with the same
// shared_len, its fork length is a multiple of the block size in
// [shared_len, both lengths), the two table rows agree on the blocks before
// it, and no parent is named twice.
int validate_forks(const SharedArgs &sh, const int32_t *context_lens, const int32_t *block_table,
                   int B, int MB, int bs, cudaStream_t stream) {
    std::vector<int32_t> lens(B), S(B, 0), fp(B), fl(B), table(size_t(B) * MB);
    if (int rc = pa::fetch(lens.data(), context_lens, B * sizeof(int32_t), stream)) return rc;
    if (sh.shared_len)
        if (int rc = pa::fetch(S.data(), sh.shared_len, B * sizeof(int32_t), stream)) return rc;
    if (int rc = pa::fetch(fp.data(), sh.fork_parent, B * sizeof(int32_t), stream)) return rc;
    if (int rc = pa::fetch(fl.data(), sh.fork_len, B * sizeof(int32_t), stream)) return rc;
    if (int rc = pa::fetch(table.data(), block_table, table.size() * sizeof(int32_t), stream))
        return rc;
    std::vector<char> named(B, 0);
    for (int c = 0; c < B; ++c) {
        const int par = fp[c];
        if (par < 0) continue;
        if (par >= B || par == c || fp[par] >= 0)
            return pa::fail(PA_ERR_INVALID, "validate: fork_parent[%d]=%d", c, par);
        if (named[par]++)
            return pa::fail(PA_ERR_INVALID, "validate: row %d is the fork parent of two rows", par);
        const int F = fl[c];
        if (S[par] != S[c] || F <= 0 || F % bs || F < S[c] || F >= lens[c] || F >= lens[par])
            return pa::fail(PA_ERR_INVALID, "validate: fork_len[%d]=%d", c, F);
        for (int i = 0; i < F / bs; ++i)
            if (table[size_t(c) * MB + i] != table[size_t(par) * MB + i])
                return pa::fail(PA_ERR_INVALID,
                                "validate: rows %d and %d differ in block %d before the fork", c,
                                par, i);
    }
    return PA_OK;
}

int decode_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                const int32_t *block_table, int max_blocks_per_seq, const int32_t *context_lens,
                int B, int Hq, int Hkv, int head_dim, int block_size, int64_t num_blocks,
                float scale, int partition_tokens, const SharedArgs *sh, void *workspace,
                size_t workspace_bytes, int dtype, cudaStream_t stream, int contig_len = 0) {
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
    if (!out || !q || !k_cache || !v_cache || (!block_table && !contig_len) || !context_lens)
        return pa::fail(PA_ERR_INVALID, "decode: NULL pointer");
    if (!pa::aligned16(q) || !pa::aligned16(out) || !pa::aligned16(k_cache) ||
        !pa::aligned16(v_cache))
        return pa::fail(PA_ERR_INVALID, "decode: q, out and pools must be 16-byte aligned");
    const int64_t cap = int64_t(max_blocks_per_seq) * block_size;
    const int max_parts = static_cast<int>((cap + pt - 1) / pt);
    const int npslot = sh ? prefix_slots_for(sh->max_shared_len) : 0;
    // with fork arrays: a child's partials from its parent's item segments
    const int nfslot = (sh && sh->fork_parent) ? max_parts + 1 : 0;
    WsLayout wl;
    if (!workspace_layout(B, Hq, head_dim, int64_t(max_parts) + 1 + npslot + nfslot, &wl))
        return pa::fail(PA_ERR_INVALID, "decode: workspace size does not fit in size_t");
    const size_t need = wl.total;
    if (need > workspace_bytes || !workspace)
        return pa::fail(PA_ERR_INVALID, "decode: workspace needs %zu bytes, got %zu", need,
                        workspace_bytes);
    if (!pa::aligned16(workspace))
        return pa::fail(PA_ERR_INVALID, "decode: workspace must be 16-byte aligned");
    if (pa::validate_on()) {
        std::vector<int32_t> lens(B), table(contig_len ? 0 : size_t(B) * max_blocks_per_seq);
        if (int rc = pa::fetch(lens.data(), context_lens, B * sizeof(int32_t), stream)) return rc;
        if (!contig_len)
            if (int rc = pa::fetch(table.data(), block_table, table.size() * sizeof(int32_t),
                                   stream))
                return rc;
        for (int b = 0; b < B; ++b) {
            if (lens[b] < 1 || lens[b] > cap)
                return pa::fail(PA_ERR_INVALID, "validate: context_lens[%d]=%d outside [1,%lld]", b,
                                lens[b], (long long)cap);
            const int nb = contig_len ? 0 : (lens[b] + block_size - 1) / block_size;
            for (int i = 0; i < nb; ++i) {
                const int32_t v = table[size_t(b) * max_blocks_per_seq + i];
                if (v < 0 || v >= num_blocks)
                    return pa::fail(PA_ERR_INVALID, "validate: block_table[%d][%d]=%d outside pool",
                                    b, i, v);
            }
        }
        if (sh)
            if (int rc = validate_groups(*sh, context_lens, block_table, B, max_blocks_per_seq,
                                         block_size, stream))
                return rc;
        if (sh && sh->fork_parent)
            if (int rc = validate_forks(*sh, context_lens, block_table, B, max_blocks_per_seq,
                                        block_size, stream))
                return rc;
    }
    DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_cache = static_cast<const uint8_t *>(k_cache);
    p.v_cache = static_cast<const uint8_t *>(v_cache);
    p.block_table = block_table;
    p.context_lens = context_lens;
    p.meta = static_cast<unsigned *>(workspace);
    p.ws_acc = reinterpret_cast<float *>(static_cast<char *>(workspace) + wl.meta_bytes);
    p.ws_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) + wl.meta_bytes +
                                        wl.acc_bytes);
    p.err = pa::device_error_word();
    p.num_blocks = num_blocks;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.bs = block_size;
    p.bs_log2 = log2_int(block_size);
    p.MB = max_blocks_per_seq;
    p.PT = pt;
    p.max_parts = max_parts + 1;  // slot stride of the grid kernel
    p.maxseg = max_parts + 1;
    p.rowslots = max_parts + 1 + npslot + nfslot;  // slot stride of the persistent kernel
    p.shared_len = nullptr;
    p.pslot0 = max_parts + 1;
    p.npfx = 0;
    p.contig_len = contig_len;
    p.qscale = scale * kLog2e;
    const int gq = Hq / Hkv;
    // Shared-prefix path: bf16 batches that run on the persistent kernel and
    // whose pool rows fit 32-bit tensor-copy coordinates; other calls decode
    // every sequence whole (the same result: the groups only save reads).
    SharedPlan plan{};
    const SharedPlan *sp = nullptr;
    if (sh && sh->G > 0 && npslot > 0 && dtype == PA_BF16 &&
        num_blocks * Hkv * block_size <= int64_t(INT32_MAX)) {
        const int sms = sm_count();
        if (sms <= 0) return pa::fail(PA_ERR_CUDA, "decode_shared: no SM count");
        if (kernel_for(B, Hkv, max_blocks_per_seq, p.bs_log2, max_parts, sms) ==
            PA_DECODE_PERSISTENT) {
            // prefix work on the tcgen05 prefill kernel (one CTA of 256 (member,
            // head) rows per SM; token chunks until about one wave), else on
            // the warp-level prefix_kernel (two waves of smaller CTAs)
            // (a chunk of the prefill kernel spans at most 512 * block_size + 64
            // tokens: within its 1024-entry block-table slice)
            const int nc_min = (sh->max_shared_len + 512 * block_size - 1) / (512 * block_size);
            plan.tc = nc_min <= npslot && pa::prefix_tc_ok(block_size, num_blocks, Hkv,
                                                           512 * block_size + 64);
            const int mpc = plan.tc ? pa::prefix_tc_members(gq) : kPfxWarps * (8 / gq);
            const int64_t ctas = int64_t((sh->max_group_size + mpc - 1) / mpc) * Hkv * sh->G;
            int64_t want = plan.tc ? int64_t(sms) / std::max<int64_t>(ctas, 1)
                                   : (2 * int64_t(sms) + ctas - 1) / std::max<int64_t>(ctas, 1);
            if (plan.tc) want = std::max<int64_t>(want, nc_min);
#ifdef PA_PFX_NC
            want = std::max(PA_PFX_NC, nc_min);
#endif
            plan.pp.group_start = sh->group_start;
            plan.pp.group_seqs = sh->group_seqs;
            plan.pp.G = sh->G;
            plan.pp.num_members = sh->num_members;
            plan.pp.nc = static_cast<int>(std::min<int64_t>(std::max<int64_t>(want, 1), npslot));
            plan.max_group_size = sh->max_group_size;
            if (int64_t(plan.pp.G) * plan.pp.nc > 65535)
                return pa::fail(PA_ERR_UNSUPPORTED, "decode_shared: too many groups");
            p.shared_len = sh->shared_len;
            p.npfx = plan.pp.nc;
            sp = &plan;
        }
    }
    // Forked children: bf16 groups of 4 heads on the persistent kernel's
    // tensor-core tile (the child's heads take the tile's 4 spare columns);
    // elsewhere every sequence reads its whole range itself.
    if (sh && sh->fork_parent && dtype == PA_BF16 && gq * 2 <= 8 && gq >= PA_DECODE_MMA_MIN_GQ &&
        tile_is_mma(gq, dtype, num_blocks, Hkv, block_size) && !contig_len) {
        const int sms = sm_count();
        if (sms <= 0) return pa::fail(PA_ERR_CUDA, "decode_shared: no SM count");
        if (kernel_for(B, Hkv, max_blocks_per_seq, p.bs_log2, max_parts, sms) ==
            PA_DECODE_PERSISTENT) {
            p.fork_parent = sh->fork_parent;
            p.fork_len = sh->fork_len;
            // without the prefix plan p.shared_len stays NULL: every row starts
            // at token 0 (or its fork point)
        }
    }
    if (dtype == PA_BF16)
        return head_dim == 128 ? dispatch_gq<__nv_bfloat16, 128>(gq, p, sp, stream)
                               : dispatch_gq<__nv_bfloat16, 64>(gq, p, sp, stream);
    return head_dim == 128 ? dispatch_gq<float, 128>(gq, p, nullptr, stream)
                           : dispatch_gq<float, 64>(gq, p, nullptr, stream);
}

}  // namespace

extern "C" {

int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, int max_blocks_per_seq, const int32_t *context_lens,
              int B, int Hq, int Hkv, int head_dim, int block_size, int64_t num_blocks,
              float scale, int partition_tokens, void *workspace, size_t workspace_bytes,
              int dtype, pa_stream_t stream) {
    pa::clear_error();
    return decode_impl(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, B,
                       Hq, Hkv, head_dim, block_size, num_blocks, scale, partition_tokens, nullptr,
                       workspace, workspace_bytes, dtype, stream);
}

int pa_decode_contiguous_workspace_size(int B, int Hq, int head_dim, int max_len,
                                        int partition_tokens, size_t *bytes) {
    pa::clear_error();
    if (max_len <= 0 || max_len % 32)
        return pa::fail(PA_ERR_INVALID, "contiguous_workspace_size: max_len must be a positive "
                                        "multiple of 32");
    return pa_decode_workspace_size(B, Hq, head_dim, max_len / 16, 16, partition_tokens, bytes);
}

int pa_decode_contiguous(void *out, const void *q, const void *k, const void *v,
                         const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                         int max_len, float scale, int partition_tokens, void *workspace,
                         size_t workspace_bytes, int dtype, pa_stream_t stream) {
    pa::clear_error();
    if (max_len <= 0 || max_len % 32 || max_len > (1 << 30))
        return pa::fail(PA_ERR_INVALID, "decode_contiguous: max_len must be a positive "
                                        "multiple of 32");
    if (B > kPersistentMaxB)
        return pa::fail(PA_ERR_UNSUPPORTED, "decode_contiguous: at most %d sequences",
                        kPersistentMaxB);
    if (B > 0 && int64_t(B) * max_len / 8 >= (int64_t(1) << 31))
        return pa::fail(PA_ERR_UNSUPPORTED, "decode_contiguous: B * max_len too large");
    // the caches viewed as B * max_len / 16 blocks of 16 rows (no table is read)
    return decode_impl(out, q, k, v, nullptr, max_len / 16, context_lens, B, Hq, Hkv, head_dim,
                       16, std::max<int64_t>(int64_t(B) * max_len / 16, 1), scale,
                       partition_tokens, nullptr, workspace, workspace_bytes, dtype, stream,
                       max_len);
}

int pa_decode_shared_workspace_size(int B, int Hq, int head_dim, int max_blocks_per_seq,
                                    int block_size, int partition_tokens, int max_shared_len,
                                    size_t *bytes) {
    pa::clear_error();
    if (!bytes) return pa::fail(PA_ERR_INVALID, "shared_workspace_size: bytes is NULL");
    if (B < 0 || Hq <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || max_shared_len < 0 ||
        !pa::pow2_in(block_size, 8, 128))
        return pa::fail(PA_ERR_INVALID, "shared_workspace_size: bad sizes");
    const int pt = resolve_partition(partition_tokens);
    if (!partition_ok(pt, block_size))
        return pa::fail(PA_ERR_INVALID, "shared_workspace_size: bad partition_tokens %d", pt);
    const int64_t cap = int64_t(max_blocks_per_seq) * block_size;
    const int64_t slots = (cap + pt - 1) / pt + 1 + prefix_slots_for(max_shared_len);
    WsLayout l;
    if (!workspace_layout(B, Hq, head_dim, slots, &l))
        return pa::fail(PA_ERR_INVALID, "shared_workspace_size: size does not fit in size_t");
    *bytes = l.total;
    return PA_OK;
}

int pa_decode_shared(void *out, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, int max_blocks_per_seq,
                     const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                     int block_size, int64_t num_blocks, float scale, int partition_tokens,
                     const int32_t *shared_len, const int32_t *group_start,
                     const int32_t *group_seqs, int G, int num_members, int max_group_size,
                     int max_shared_len, void *workspace, size_t workspace_bytes, int dtype,
                     pa_stream_t stream) {
    pa::clear_error();
    if (G < 0 || num_members < 0 || max_group_size < 0 || max_shared_len < 0)
        return pa::fail(PA_ERR_INVALID, "decode_shared: bad group sizes");
    if (G > 0 && (!shared_len || !group_start || (num_members > 0 && !group_seqs)))
        return pa::fail(PA_ERR_INVALID, "decode_shared: NULL group array");
    if (max_shared_len > (int64_t(max_blocks_per_seq) * block_size))
        return pa::fail(PA_ERR_INVALID, "decode_shared: max_shared_len beyond the table");
    const SharedArgs sh{shared_len, group_start, group_seqs, G,
                        num_members, max_group_size, max_shared_len};
    return decode_impl(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, B,
                       Hq, Hkv, head_dim, block_size, num_blocks, scale, partition_tokens, &sh,
                       workspace, workspace_bytes, dtype, stream);
}

int pa_decode_shared_forks_workspace_size(int B, int Hq, int head_dim, int max_blocks_per_seq,
                                          int block_size, int partition_tokens,
                                          int max_shared_len, size_t *bytes) {
    pa::clear_error();
    if (!bytes) return pa::fail(PA_ERR_INVALID, "shared_forks_workspace_size: bytes is NULL");
    if (B < 0 || Hq <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0 || max_shared_len < 0 ||
        !pa::pow2_in(block_size, 8, 128))
        return pa::fail(PA_ERR_INVALID, "shared_forks_workspace_size: bad sizes");
    const int pt = resolve_partition(partition_tokens);
    if (!partition_ok(pt, block_size))
        return pa::fail(PA_ERR_INVALID, "shared_forks_workspace_size: bad partition_tokens %d",
                        pt);
    const int64_t cap = int64_t(max_blocks_per_seq) * block_size;
    const int64_t parts = (cap + pt - 1) / pt + 1;
    const int64_t slots = 2 * parts + prefix_slots_for(max_shared_len);
    WsLayout l;
    if (!workspace_layout(B, Hq, head_dim, slots, &l))
        return pa::fail(PA_ERR_INVALID, "shared_forks_workspace_size: size does not fit in size_t");
    *bytes = l.total;
    return PA_OK;
}

int pa_decode_shared_forks(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                           int block_size, int64_t num_blocks, float scale, int partition_tokens,
                           const int32_t *shared_len, const int32_t *group_start,
                           const int32_t *group_seqs, int G, int num_members, int max_group_size,
                           int max_shared_len, const int32_t *fork_parent,
                           const int32_t *fork_len, void *workspace, size_t workspace_bytes,
                           int dtype, pa_stream_t stream) {
    pa::clear_error();
    if (G < 0 || num_members < 0 || max_group_size < 0 || max_shared_len < 0)
        return pa::fail(PA_ERR_INVALID, "decode_shared_forks: bad group sizes");
    if (G > 0 && (!shared_len || !group_start || (num_members > 0 && !group_seqs)))
        return pa::fail(PA_ERR_INVALID, "decode_shared_forks: NULL group array");
    if (B > 0 && (!fork_parent || !fork_len))
        return pa::fail(PA_ERR_INVALID, "decode_shared_forks: NULL fork array");
    if (max_shared_len > (int64_t(max_blocks_per_seq) * block_size))
        return pa::fail(PA_ERR_INVALID, "decode_shared_forks: max_shared_len beyond the table");
    SharedArgs sh{shared_len, group_start, group_seqs, G,
                  num_members, max_group_size, max_shared_len};
    sh.fork_parent = fork_parent;
    sh.fork_len = fork_len;
    return decode_impl(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens, B,
                       Hq, Hkv, head_dim, block_size, num_blocks, scale, partition_tokens, &sh,
                       workspace, workspace_bytes, dtype, stream);
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
// of the last call; nothing in it needs to start at zero (every partial
// and per-item count is written before it is read in the same call).  Calls
// that overlap on the GPU
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
