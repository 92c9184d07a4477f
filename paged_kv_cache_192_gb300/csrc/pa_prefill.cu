// Chunked prefill over a paged KV cache (bf16), tensor-core tiles.
//
// What it computes ("Melihat Lebih Dalam vLLM v0.7", section "Blueprint
// Arsitektur 3: Chunked Prefill"): a prompt is cut into chunks (e.g. 512
// tokens) that run in the same step as decodes.  New token i of request r sits
// at absolute position P_r + i and attends causally to positions 0..P_r+i of
// its request, the prior context and the chunk itself, all read through the
// block table (nalar.dev, section "Kernel attention harus mengikuti block
// table").  Prefill is the compute-bound phase (same page), so QK^T and PV run
// as dense bf16 tiles on the tensor cores with fp32 accumulation.
//
// A row is one (query token, query head) pair, so the GQ heads that share a
// KV head share every K/V tile (GQA packed into the M dimension); K/V tiles
// of 64 tokens; online softmax in the log2 domain with a lazy rescale.
// Kernels (pa_prefill_kernel_for picks one from the sizes):
//   prefill_persist_kernel (pa_prefill_persist.cu; batches of at most 512
//                       work items) one CTA per SM running a list of work
//                       items with the warp specialisation below;
//   prefill_tc2_kernel  (larger batches) warp-specialised tcgen05, one CTA per
//                       work item: TMA loader warp, MMA warp, two softmax
//                       warp groups over 2 x 128 rows;
//   prefill_tc_kernel   (block sizes outside 8..64, block tables longer than
//                       1024 entries) 128 threads per 128 rows, tcgen05,
//                       cp.async K/V;
//   prefill_kernel      (compile-time alternative, PA_PREFILL_TCGEN05=0)
//                       warp-level mma.sync, kept for comparison.
#include <cuda.h>

#include <atomic>
#include <type_traits>
#include <cmath>
#include <vector>

#include "pa_prefill.cuh"

namespace {

using namespace pa::pf;

constexpr int kRows = 64;   // query rows (token, head) per CTA
constexpr int kKT = 64;     // KV tokens per tile
constexpr int kThreads = 128;

// Swizzled address of 16-byte chunk `c` of row `r` in a tile of rows of
// `CH` chunks: chunk positions are XORed with the row's low 3 bits so that
// ldmatrix reads of 8 consecutive rows hit 8 different bank groups.
template <int CH>
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c) {
    return base + r * (CH * 16) + ((c ^ (r & 7)) * 16);
}


__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                          uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


template <int D, int GQ>
__global__ void __launch_bounds__(kThreads, 2) prefill_kernel(const PrefillParams p) {
    constexpr int CH = D * 2 / 16;  // 16-byte chunks per row
    constexpr int KS = D / 16;      // k-steps over head_dim
    constexpr int NT = kKT / 8;     // score n-tiles per KV tile
    constexpr int OT = D / 8;       // output n-tiles
    constexpr int QTOK = kRows / GQ;
    constexpr int TILE_BYTES = kKT * D * 2;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sq = pa::smem_u32(smem);
    const uint32_t sk = sq + kRows * D * 2;       // [2][kKT][D]
    const uint32_t sv = sk + 2 * TILE_BYTES;      // [2][kKT][D]

    const int qt = blockIdx.x, hk = blockIdx.y, r = blockIdx.z;
    const int qs = p.query_start[r];
    const int n = p.query_start[r + 1] - qs;
    const int t0 = qt * QTOK;
    if (t0 >= n) return;
    const int cap = p.MB << p.bs_log2;
    int L = p.context_lens[r];
    if (L > cap || L < n) {
        if (threadIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
        return;
    }
    const int P = L - n;
    const int kv_end = min(L, P + t0 + QTOK);  // last position of this tile + 1
    const int ntiles = (kv_end + kKT - 1) / kKT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- Q tile: row m = token (m / GQ), head (m % GQ) ----------------------
    for (int idx = tid; idx < kRows * CH; idx += kThreads) {
        const int m = idx / CH, c = idx % CH;
        const int t = t0 + m / GQ;
        const bool valid = t < n;
        const __nv_bfloat16 *src =
            p.q + (static_cast<size_t>(qs + (valid ? t : 0)) * p.Hq + hk * GQ + m % GQ) * D + c * 8;
        cp_async16(swz<CH>(sq, m, c), src, valid);
    }
    const int32_t *bt = p.block_table + static_cast<size_t>(r) * p.MB;
    auto load_tile = [&](int it, int buf) {
        const int j0 = it * kKT;
        for (int idx = tid; idx < kKT * CH; idx += kThreads) {
            const int row = idx / CH, c = idx % CH;
            const int j = j0 + row;
            const bool valid = j < kv_end;
            size_t off = 0;
            if (valid) {
                int blk = bt[j >> p.bs_log2];
                if (blk < 0 || blk >= p.num_blocks) {
                    pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
                    blk = 0;
                }
                off = ((static_cast<size_t>(blk) * p.Hkv + hk) * p.bs + (j & (p.bs - 1))) * D * 2 +
                      c * 16;
            }
            cp_async16(swz<CH>(sk + buf * TILE_BYTES, row, c), p.k_cache + off, valid);
            cp_async16(swz<CH>(sv + buf * TILE_BYTES, row, c), p.v_cache + off, valid);
        }
    };
    load_tile(0, 0);
    cp_async_commit();

    // This thread's two rows of the warp's 16: g and g+8.
    const int g = lane >> 2, cq = lane & 3;
    int pos[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int m = warp * 16 + g + 8 * i;
        const int t = min(t0 + m / GQ, n - 1);  // rows past the chunk reuse the last row
        pos[i] = P + t;
    }

    uint32_t qf[KS][4];
    float o[OT][4];
#pragma unroll
    for (int j = 0; j < OT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

    for (int it = 0; it < ntiles; ++it) {
        const int buf = it & 1;
        if (it + 1 < ntiles) load_tile(it + 1, buf ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (it == 0) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int row = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int c = ks * 2 + (lane >> 4);
                ldsm_x4(swz<CH>(sq, row, c), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
            }
        }
        const uint32_t kb = sk + buf * TILE_BYTES, vb = sv + buf * TILE_BYTES;
        // ---- S = Q K^T (16 x 64 per warp) ----------------------------------------
        float s[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
            for (int j = 0; j < NT; j += 2) {
                const int row = j * 8 + (lane & 7) + 8 * (lane >> 4);
                const int c = ks * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(swz<CH>(kb, row, c), b0, b1, b2, b3);
                mma_bf16(s[j], qf[ks], b0, b1);
                mma_bf16(s[j + 1], qf[ks], b2, b3);
            }
        }
        // ---- scale, causal mask, online softmax ---------------------------------
        const int j0 = it * kKT;
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = j0 + j * 8 + cq * 2 + (e & 1);
                const int ri = e >> 1;
                float v = s[j][e] * p.qscale;
                v = col <= pos[ri] ? v : -INFINITY;
                s[j][e] = v;
                tmax[ri] = fmaxf(tmax[ri], v);
            }
        float alpha[2];
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            tmax[ri] = fmaxf(tmax[ri], __shfl_xor_sync(pa::kFull, tmax[ri], 1));
            tmax[ri] = fmaxf(tmax[ri], __shfl_xor_sync(pa::kFull, tmax[ri], 2));
            const float mnew = fmaxf(mrow[ri], tmax[ri]);
            alpha[ri] = mrow[ri] == -INFINITY ? 0.f : fast_exp2(mrow[ri] - mnew);
            mrow[ri] = mnew;
        }
        // P enters the tensor cores as bf16; a single bf16 rounding of the
        // softmax weights (2^-9 relative) is too coarse for short contexts,
        // so P = hi + lo with both parts bf16 (2^-17 relative) and PV runs
        // twice into the same fp32 accumulators.
        float rsum[2] = {0.f, 0.f};
        uint32_t pf[NT / 2][4], pl[NT / 2][4];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float p0 = fast_exp2(s[j][0] - mrow[0]);
            const float p1 = fast_exp2(s[j][1] - mrow[0]);
            const float p2 = fast_exp2(s[j][2] - mrow[1]);
            const float p3 = fast_exp2(s[j][3] - mrow[1]);
            rsum[0] += p0 + p1;
            rsum[1] += p2 + p3;
            const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
            const float2 r01 = pa::bf16x2_to_float2(h01), r23 = pa::bf16x2_to_float2(h23);
            pf[j / 2][(j & 1) * 2 + 0] = h01;
            pf[j / 2][(j & 1) * 2 + 1] = h23;
            pl[j / 2][(j & 1) * 2 + 0] = pack_bf16(p0 - r01.x, p1 - r01.y);
            pl[j / 2][(j & 1) * 2 + 1] = pack_bf16(p2 - r23.x, p3 - r23.y);
        }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) lrow[ri] = lrow[ri] * alpha[ri] + rsum[ri];
#pragma unroll
        for (int j = 0; j < OT; ++j) {
            o[j][0] *= alpha[0];
            o[j][1] *= alpha[0];
            o[j][2] *= alpha[1];
            o[j][3] *= alpha[1];
        }
        // ---- O += P V --------------------------------------------------------------
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk) {
#pragma unroll
            for (int j = 0; j < OT; j += 2) {
                const int row = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int c = j + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(swz<CH>(vb, row, c), b0, b1, b2, b3);
                mma_bf16(o[j], pf[kk], b0, b1);
                mma_bf16(o[j + 1], pf[kk], b2, b3);
                mma_bf16(o[j], pl[kk], b0, b1);
                mma_bf16(o[j + 1], pl[kk], b2, b3);
            }
        }
        __syncthreads();  // buffer `buf` is refilled two iterations on
    }
    cp_async_wait<0>();

    // ---- normalise and store ------------------------------------------------------
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
        lrow[ri] += __shfl_xor_sync(pa::kFull, lrow[ri], 1);
        lrow[ri] += __shfl_xor_sync(pa::kFull, lrow[ri], 2);
    }
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
        const int m = warp * 16 + g + 8 * ri;
        const int t = t0 + m / GQ;
        if (t >= n) continue;
        const float inv = 1.f / lrow[ri];
        __nv_bfloat16 *dst = p.out + (static_cast<size_t>(qs + t) * p.Hq + hk * GQ + m % GQ) * D;
#pragma unroll
        for (int j = 0; j < OT; ++j) {
            const uint32_t v = pack_bf16(o[j][2 * ri] * inv, o[j][2 * ri + 1] * inv);
            *reinterpret_cast<uint32_t *>(dst + j * 8 + cq * 2) = v;
        }
    }
}

// ---------------------------------------------------------------------------
// tcgen05 prefill kernel (default).
//
// One CTA of 128 threads per (request, KV head, tile of 128/GQ query tokens);
// thread r owns query row r = (token r / GQ, head r % GQ), which is also TMEM
// lane r, so every row's softmax is thread-local.  Per 64-token K/V tile:
//   S = Q K^T   tcgen05.mma, Q and K from 128-byte-swizzled shared memory,
//               S (fp32) in TMEM
//   softmax     tcgen05.ld of the row, scale, causal mask, running max with a
//               lazy rescale of O, p = exp2(s - m), row sum in fp32;
//               P = hi + lo (both bf16) written back to TMEM
//   O += P V    tcgen05.mma with A = P from TMEM and B = V (MN-major) from
//               shared memory, twice (hi, lo), O (fp32) stays in TMEM
// K/V tiles are gathered block by block through the block table with cp.async
// into two buffers (tile j+1 loads while tile j computes).  TMEM columns:
// O [0, D), S [128, 192), P hi [192, 224), P lo [224, 256).
// ---------------------------------------------------------------------------
constexpr int kTcKT = 64;        // KV tokens per tile
constexpr int kTcCols = 256;     // TMEM columns per CTA
constexpr int kTcS = 128, kTcPH = 192, kTcPL = 224;

template <int D>
struct TcLayout {
    static constexpr int Q_BYTES = 128 * D * 2;
    static constexpr int T_BYTES = kTcKT * D * 2;  // one K or V tile
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int OFF_V = OFF_K + 2 * T_BYTES;
    static constexpr int OFF_BAR = OFF_V + 2 * T_BYTES;
    static constexpr int OFF_BT = OFF_BAR + 64;        // block-table slice
    static constexpr int BT_MAX = 1024;                // entries kept in smem
    static constexpr int SMEM = OFF_BT + 4 * BT_MAX + 1024;  // + alignment slack
};

__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity) {
    return pa::mbar_wait(bar, parity);
}

template <int D, int GQ>
__global__ void __launch_bounds__(128, 2) prefill_tc_kernel(const PrefillParams p) {
    using Lay = TcLayout<D>;
    constexpr int CH = D * 2 / 16;  // 16-byte chunks per row
    constexpr int QTOK = 128 / GQ;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sq = pa::smem_u32(smem);
    const uint32_t sk = sq + Lay::OFF_K, sv = sq + Lay::OFF_V;
    uint64_t *bar_s = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BAR);
    uint64_t *bar_o = bar_s + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar_s + 2);

    // later query tiles see more context: start them first
    const int qt = gridDim.x - 1 - blockIdx.x, hk = blockIdx.y, r = blockIdx.z;
    const int qs = p.query_start[r];
    const int n = p.query_start[r + 1] - qs;
    const int t0 = qt * QTOK;
    if (t0 >= n) return;
    const int cap = p.MB << p.bs_log2;
    const int L = p.context_lens[r];
    if (L > cap || L < n) {
        if (threadIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
        return;
    }
    const int P = L - n;
    const int kv_end = min(L, P + t0 + QTOK);
    const int ntiles = (kv_end + kTcKT - 1) / kTcKT;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int32_t *bt_g = p.block_table + static_cast<size_t>(r) * p.MB;
    // this CTA's block-table entries, checked, in shared memory when they fit
    int32_t *bt_s = reinterpret_cast<int32_t *>(smem + Lay::OFF_BT);
    const int nblk = (kv_end + p.bs - 1) >> p.bs_log2;
    const bool bt_in_smem = nblk <= Lay::BT_MAX;
    auto checked = [&](int blk) {
        if (blk < 0 || blk >= p.num_blocks) {
            pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            blk = 0;
        }
        return blk;
    };
    if (bt_in_smem) {
        for (int i = tid; i < nblk; i += 128) bt_s[i] = checked(bt_g[i]);
        __syncthreads();
    }

    // ---- loads (cp.async, swizzled) ----------------------------------------------
    for (int idx = tid; idx < 128 * CH; idx += 128) {
        const int m = idx / CH, c = idx % CH;
        const int t = t0 + m / GQ;
        const bool valid = t < n;
        const __nv_bfloat16 *src =
            p.q + (static_cast<size_t>(qs + (valid ? t : 0)) * p.Hq + hk * GQ + m % GQ) * D + c * 8;
        cp_async16(sq + pa::tc::sw128(m, c * 8, 128), src, valid);
    }
    auto load_tile = [&](int it, int buf) {
        const int j0 = it * kTcKT;
        const uint32_t dk = sk + buf * Lay::T_BYTES, dv = sv + buf * Lay::T_BYTES;
        for (int idx = tid; idx < kTcKT * CH; idx += 128) {
            const int row = idx / CH, c = idx % CH;
            const int j = j0 + row;
            const bool valid = j < kv_end;
            size_t off = 0;
            if (valid) {
                const int blk =
                    bt_in_smem ? bt_s[j >> p.bs_log2] : checked(bt_g[j >> p.bs_log2]);
                off = ((static_cast<size_t>(blk) * p.Hkv + hk) * p.bs + (j & (p.bs - 1))) * D * 2 +
                      c * 16;
            }
            const uint32_t o = pa::tc::sw128(row, c * 8, kTcKT);
            cp_async16(dk + o, p.k_cache + off, valid);
            cp_async16(dv + o, p.v_cache + off, valid);
        }
    };
    load_tile(0, 0);
    cp_async_commit();
    if (ntiles > 1) {
        load_tile(1, 1);
        cp_async_commit();
    }

    if (tid == 0) {
        pa::mbar_init(bar_s, 1);
        pa::mbar_init(bar_o, 1);
        pa::fence_barrier_init();
    }
    if (warp == 0) pa::tc::alloc(tslot, kTcCols);
    pa::tc::fence_before();
    __syncthreads();
    pa::tc::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);

    const int g = tid / GQ;
    const int pos = P + min(t0 + g, n - 1);  // rows past the chunk reuse the last row
    float m_used = -INFINITY, lsum = 0.f;
    bool failed = false;
    constexpr uint32_t kIdS = pa::tc::idesc_bf16(128, kTcKT, 0, 0);
    constexpr uint32_t kIdO = pa::tc::idesc_bf16(128, D, 0, 1);

    for (int it = 0; it < ntiles; ++it) {
        const int buf = it & 1;
        if (it == 0 && ntiles > 1) cp_async_wait<1>();
        else cp_async_wait<0>();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        pa::tc::fence_before();
        __syncthreads();
        pa::tc::fence_after();
        // ---- S = Q K^T -------------------------------------------------------------
        if (tid == 0) {
            const uint32_t kb = sk + buf * Lay::T_BYTES;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t a = pa::tc::sdesc(sq + (ks >> 2) * 128 * 128 + (ks & 3) * 32, 16, 1024);
                const uint64_t b =
                    pa::tc::sdesc(kb + (ks >> 2) * kTcKT * 128 + (ks & 3) * 32, 16, 1024);
                pa::tc::mma_ss(tmem + kTcS, a, b, kIdS, ks > 0);
            }
            pa::tc::commit(bar_s);
        }
        // PV of the previous tile done: its buffers take tile it+1 now, while
        // this tile's S and softmax run
        if (it > 0) {
            failed = __syncthreads_or(!tc_wait(bar_o, (it - 1) & 1));
            if (failed) break;
            if (it + 1 < ntiles) {
                load_tile(it + 1, (it + 1) & 1);
                cp_async_commit();
            }
        }
        failed = __syncthreads_or(!tc_wait(bar_s, it & 1));
        if (failed) break;
        pa::tc::fence_after();
        // ---- softmax of this row --------------------------------------------------------
        uint32_t sr[2][32];
        pa::tc::ld32(lane_base + kTcS, sr[0]);
        pa::tc::ld32(lane_base + kTcS + 32, sr[1]);
        pa::tc::wait_ld();
        const int j0 = it * kTcKT;
        float s[64];
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const float v = __uint_as_float(sr[c >> 5][c & 31]) * p.qscale;
            s[c] = (j0 + c <= pos) ? v : -INFINITY;
            tmax = fmaxf(tmax, s[c]);
        }
        float alpha = 1.f;
        if (tmax > m_used + kTcTau) {  // also true on the first tile (m_used = -inf)
            alpha = (m_used == -INFINITY) ? 0.f : exp2f(m_used - tmax);
            m_used = tmax;
        }
        uint32_t ph[32], pl[32];
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const float p0 = fast_exp2(s[2 * c] - m_used);
            const float p1 = fast_exp2(s[2 * c + 1] - m_used);
            rs += p0 + p1;
            ph[c] = pack_bf16(p0, p1);
            const float2 hv = pa::bf16x2_to_float2(ph[c]);
            pl[c] = pack_bf16(p0 - hv.x, p1 - hv.y);
        }
        lsum = lsum * alpha + rs;
        // ---- rescale O (the previous PV is complete) ---------------------------------
        if (it > 0) {
            if (__any_sync(pa::kFull, alpha != 1.f)) {
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    pa::tc::ld32(lane_base + c0, o);
                    pa::tc::wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    pa::tc::st32(lane_base + c0, o);
                }
            }
        }
        pa::tc::st32(lane_base + kTcPH, ph);
        pa::tc::st32(lane_base + kTcPL, pl);
        pa::tc::wait_st();
        pa::tc::fence_before();
        __syncthreads();
        pa::tc::fence_after();
        // ---- O += P V (hi, then lo) ---------------------------------------------------
        if (tid == 0) {
            const uint32_t vb = sv + buf * Lay::T_BYTES;
#pragma unroll
            for (int ks = 0; ks < kTcKT / 16; ++ks) {
                const uint64_t b = pa::tc::sdesc(vb + ks * 16 * 128, kTcKT * 128, 1024);
                pa::tc::mma_ts(tmem, tmem + kTcPH + ks * 8, b, kIdO, (it > 0 || ks > 0) ? 1 : 0);
                pa::tc::mma_ts(tmem, tmem + kTcPL + ks * 8, b, kIdO, 1);
            }
            pa::tc::commit(bar_o);
        }
    }
    // ---- normalise and store ----------------------------------------------------------
    if (!failed) failed = __syncthreads_or(!tc_wait(bar_o, (ntiles - 1) & 1));
    if (!failed) {
        pa::tc::fence_after();
        const int t = t0 + g;
        const float inv = 1.f / lsum;
        __nv_bfloat16 *dst =
            p.out + (static_cast<size_t>(qs + min(t, n - 1)) * p.Hq + hk * GQ + tid % GQ) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            pa::tc::ld32(lane_base + c0, o);
            pa::tc::wait_ld();
            if (t < n) {
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv);
                    w.y = pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
                    w.z = pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
                    w.w = pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
                    *reinterpret_cast<uint4 *>(dst + c0 + c) = w;
                }
            }
        }
    } else {
        // a wait ran out: record it, wait (bounded) for this CTA's MMAs and
        // copies, free TMEM, write nothing
        if (tid == 0) {
            pa::record_error(p.err, PA_DEVERR_TIMEOUT);
            // give MMAs still in flight one more bounded chance to finish
            // before their TMEM is released
            (void)pa::mbar_wait(bar_s, 0);
            (void)pa::mbar_wait(bar_o, 0);
        }
        cp_async_wait<0>();
    }
    pa::tc::fence_before();
    __syncthreads();
    if (warp == 0) pa::tc::dealloc(tmem, kTcCols);
}

// ---------------------------------------------------------------------------
// tcgen05 prefill kernel, warp-specialised (default).
//
// One CTA of 320 threads per (request, KV head, 2 x 128 query rows):
//   warps 0-3  softmax of query tile A (rows 0..127, TMEM lanes 0..127)
//   warps 4-7  softmax of query tile B (rows 128..255, same lanes)
//   warp 8     issues every tcgen05.mma (one lane)
//   warp 9     loads K/V tiles with TMA (2D tensor copies, 128-byte swizzle)
// S is double-buffered per query tile and computed one K/V tile ahead: the
// MMA warp issues QK^T of tile j+1 before PV of tile j, so a softmax warp
// group finds its next S ready when it finishes the current one, and the
// tensor core works on the other group's products meanwhile.  P (bf16 hi and
// lo halves) overwrites the S buffer it was computed from.  64-token K/V
// tiles go through a 3-stage ring; a (block, 64 columns) box per copy,
// gathered through the block table; boxes for blocks past the context are
// read out of bounds and arrive zero-filled.  TMEM (512 columns):
// O_A [0,128), O_B [128,256), S_A[0..1] [256,384), S_B[0..1] [384,512).
// All hand-offs are mbarriers; every wait is bounded.
// ---------------------------------------------------------------------------
#ifndef PA_PREFILL_NST
#define PA_PREFILL_NST 4  // K/V ring stages of the two-query-tile kernel (3: 105.7 us, 4: 102.2 us on the mixed batch)
#endif
constexpr int kT2RankMax = 256;  // (request, query tile) pairs ranked in-kernel

// NQ query tiles of 128 rows per CTA: NQ = 2 (320 threads, 512 TMEM columns,
// 3-stage K/V ring, one CTA per SM) or NQ = 1 (192 threads, 256 columns,
// 2-stage ring, two CTAs per SM).
template <int D, int NQ = 2>
struct Tc2Layout {
    static constexpr int ROWS = 128 * NQ;
    static constexpr int NST = NQ == 2 ? PA_PREFILL_NST : 2;  // K/V ring stages
    static constexpr int THREADS = (4 * NQ + 2) * 32;  // softmax groups, MMA warp, loader warp
    static constexpr int MMA_WARP = 4 * NQ, LOAD_WARP = 4 * NQ + 1;
    static constexpr int TMEM_COLS = 256 * NQ;       // O per group, then S (2 x 64) per group
    static constexpr int Q_BYTES = NQ * 128 * D * 2;  // the query tiles
    static constexpr int T_BYTES = kT2KT * D * 2;    // one K or V tile
    static constexpr int OFF_KV = Q_BYTES;           // [stage][K|V]
    static constexpr int OFF_BAR = OFF_KV + NST * 2 * T_BYTES;
    static constexpr int N_BAR = 2 * NST + 4 * NQ;   // kv_full, kv_empty, s x 2NQ, (p, o) x NQ
    static constexpr int OFF_SLOT = OFF_BAR + 8 * N_BAR;
    static constexpr int OFF_BT = OFF_SLOT + 16;
    static constexpr int BT_MAX = 1024;
    static constexpr int OFF_ROWS = OFF_BT + 4 * BT_MAX;  // prefix mode: row of each row
    static constexpr int SMEM = OFF_ROWS + 8 * ROWS + 1024;
};


template <int D, int GQ, bool PFX, int NQ>
__global__ void __launch_bounds__(Tc2Layout<D, NQ>::THREADS, 3 - NQ)
    prefill_tc2_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
    using Lay = Tc2Layout<D, NQ>;
    constexpr int kT2NST = Lay::NST;
    constexpr int kT2Threads = Lay::THREADS;
    constexpr int ROWS = Lay::ROWS;
    constexpr int CH = D * 2 / 16;
    constexpr int QTOK = ROWS / GQ;  // query tokens per CTA
    constexpr int TILE_TX = 2 * kT2KT * D * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sq = pa::smem_u32(smem);
    const uint32_t skv = sq + Lay::OFF_KV;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BAR);
    uint64_t *kv_full = bars, *kv_empty = bars + kT2NST;
    // s_full[2 * group + buffer]; p_full / o_done per query-tile group
    uint64_t *s_full = bars + 2 * kT2NST, *p_full = s_full + 2 * NQ, *o_done = p_full + NQ;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + Lay::OFF_SLOT);
    volatile int *fail = reinterpret_cast<volatile int *>(smem + Lay::OFF_SLOT + 4);
    int32_t *bt_s = reinterpret_cast<int32_t *>(smem + Lay::OFF_BT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // launched as a programmatic dependent in prefix mode: inputs are ready
    // past this point (a no-op otherwise).  Behind the decode grid
    // (pfx_wait_end) the inputs were complete before that grid started this
    // one, and the wait moves to every exit instead.
    const bool wait_end = PFX && p.pfx_wait_end;
    if (!wait_end) asm volatile("griddepcontrol.wait;" ::: "memory");
    // behind the decode grid the merge comes next: it may launch now (its
    // CTAs wait for this grid, which itself waits for the decode at exit)
    if (wait_end) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    auto exit_wait = [&]() {
        if (wait_end) asm volatile("griddepcontrol.wait;" ::: "memory");
    };
    int hk, kv_end, ntiles, nblk;
    const int32_t *bt_g;
    int qs = 0, n = 0, t0 = 0, P = 0;            // chunked-prefill work item
    int pm0 = 0, pmend = 0, pS = 0, pchunk = 0;  // prefix-mode work item
    if constexpr (PFX) {
        // blockIdx.x = ((group * member tiles + member tile) * chunks + chunk)
        //              * Hkv + KV head
        hk = blockIdx.x % p.Hkv;
        int rest = blockIdx.x / p.Hkv;
        pchunk = rest % p.pfx_nc;
        rest /= p.pfx_nc;
        const int mt = rest % p.pfx_nmt, g = rest / p.pfx_nmt;
        const int mbeg = p.pfx_group_start[g], mend = p.pfx_group_start[g + 1];
        if (mbeg < 0 || mend > p.pfx_members || mbeg > mend) {
            if (tid == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            exit_wait();
            return;
        }
        pm0 = mbeg + mt * QTOK;
        pmend = mend;
        if (pm0 >= mend) {
            exit_wait();
            return;
        }
        const int b0 = p.pfx_group_seqs[mbeg];  // its table row holds the shared blocks
        if (b0 >= 0 && b0 < p.pfx_B) {
            pS = p.pfx_shared_len[b0];
            const int L0 = p.context_lens[b0];
            if (pS < 0 || pS >= L0 || (pS & (p.bs - 1)) || pS > (p.MB << p.bs_log2)) pS = 0;
        }
        if (pS == 0) {
            if (tid == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            exit_wait();
            return;
        }
        const int ch = ((pS + kT2KT - 1) / kT2KT + p.pfx_nc - 1) / p.pfx_nc * kT2KT;
        const int t_lo = min(pS, pchunk * ch), t_hi = min(pS, t_lo + ch);
        kv_end = t_hi - t_lo;  // token indices below are relative to t_lo
        ntiles = (kv_end + kT2KT - 1) / kT2KT;
        nblk = (kv_end + p.bs - 1) >> p.bs_log2;
        bt_g = p.block_table + static_cast<size_t>(b0) * p.MB + (t_lo >> p.bs_log2);
    } else {
        // Work item: the (request, query tile) pair of rank blockIdx.x / Hkv when
        // all pairs are ordered by decreasing number of K/V tiles (longest
        // first, so the biggest items do not form the tail), KV head
        // blockIdx.x % Hkv.  Pairs that do not exist (t0 >= n) cost -1.
        const int nqt = (p.max_query_len + QTOK - 1) / QTOK;
        const int npairs = p.R * nqt;
        int *pick = reinterpret_cast<int *>(smem + Lay::OFF_SLOT + 8);
        auto cost = [&](int pair) {
            const int rr = pair / nqt, tq = (pair % nqt) * QTOK;
            const int nr = p.query_start[rr + 1] - p.query_start[rr];
            if (tq >= nr) return -1;
            const int Pr = p.context_lens[rr] - nr;
            return (Pr + tq + QTOK + kT2KT - 1) / kT2KT;
        };
        const int want = blockIdx.x / p.Hkv;
        hk = blockIdx.x % p.Hkv;
        int pair = want;  // natural order when there are too many pairs to rank
        if (npairs <= kT2RankMax) {
            int *costs = reinterpret_cast<int *>(smem + Lay::OFF_BT);  // reused below
            for (int i = tid; i < npairs; i += kT2Threads) costs[i] = cost(i);
            if (tid == 0) *pick = -1;
            __syncthreads();
            for (int i = tid; i < npairs; i += kT2Threads) {
                const int ci = costs[i];
                int rank = 0;
                for (int j = 0; j < npairs; ++j) {
                    const int cj = costs[j];
                    rank += (cj > ci || (cj == ci && j < i)) ? 1 : 0;
                }
                if (rank == want) *pick = i;
            }
            __syncthreads();
            pair = *pick;
        }
        if (pair < 0) return;
        const int r = pair / nqt, qt = pair % nqt;
        qs = p.query_start[r];
        n = p.query_start[r + 1] - qs;
        t0 = qt * QTOK;
        if (t0 >= n) return;
        const int cap = p.MB << p.bs_log2;
        const int L = p.context_lens[r];
        if (L > cap || L < n) {
            if (threadIdx.x == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            return;
        }
        P = L - n;
        kv_end = min(L, P + t0 + QTOK);
        ntiles = (kv_end + kT2KT - 1) / kT2KT;
        nblk = (kv_end + p.bs - 1) >> p.bs_log2;
        bt_g = p.block_table + static_cast<size_t>(r) * p.MB;
    }
    if (nblk > Lay::BT_MAX) {  // the host routes such requests elsewhere
        if (tid == 0) pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
        exit_wait();
        return;
    }
    // prefix mode: the decode-workspace row of CTA row m (-1: no member)
    auto pfx_row = [&](int m) -> int64_t {
        const int mem = pm0 + m / GQ;
        if (mem >= pmend) return -1;
        const int b = p.pfx_group_seqs[mem];
        if (b < 0 || b >= p.pfx_B || p.pfx_shared_len[b] != pS) return -1;
        return static_cast<int64_t>(b) * p.Hq + hk * GQ + m % GQ;
    };
    if constexpr (PFX) {
        if (ntiles == 0) {
            // a chunk past this group's prefix: neutral partials (weight 0)
            for (int m = tid; m < ROWS; m += kT2Threads) {
                const int64_t row = pfx_row(m);
                if (row < 0) continue;
                const size_t slot = static_cast<size_t>(row) * p.pfx_rowslots + p.pfx_pslot0 + pchunk;
                *reinterpret_cast<float2 *>(p.pfx_ml + 2 * slot) = make_float2(-INFINITY, 0.f);
                for (int c = 0; c < D; c += 4)
                    *reinterpret_cast<float4 *>(p.pfx_acc + slot * D + c) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
            }
            exit_wait();
            return;
        }
    }

    // ---- set-up: block-table slice, barriers, TMEM; then the loader starts
    // while warps 0-8 bring in the Q tiles (cp.async) ------------------------------
    for (int i = tid; i < nblk; i += kT2Threads) {
        int b = bt_g[i];
        if (b < 0 || b >= p.num_blocks) {
            pa::record_error(p.err, PA_DEVERR_BAD_BLOCK);
            b = 0;
        }
        bt_s[i] = b;
    }
    int64_t *rows_s = reinterpret_cast<int64_t *>(smem + Lay::OFF_ROWS);
    if constexpr (PFX) {
        for (int m = tid; m < ROWS; m += kT2Threads) rows_s[m] = pfx_row(m);
    }
    if (tid == 0) {
        for (int i = 0; i < kT2NST; ++i) {
            pa::mbar_init(&kv_full[i], 1);
            pa::mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2 * NQ; ++i) pa::mbar_init(&s_full[i], 1);
        for (int i = 0; i < NQ; ++i) {
            pa::mbar_init(&p_full[i], 4);  // one arrival per softmax warp
            pa::mbar_init(&o_done[i], 1);
        }
        *fail = 0;
        pa::fence_barrier_init();
    }
    if (warp == Lay::MMA_WARP) pa::tc::alloc(tslot, Lay::TMEM_COLS);
    pa::tc::fence_before();
    __syncthreads();
    pa::tc::fence_after();
    const uint32_t tmem = *tslot;
    if (warp != Lay::LOAD_WARP) {
        // Q tiles: only the MMA warp's QK^T reads them; every warp but the
        // loader loads them and they meet on named barrier 1 before it
        constexpr int kQThreads = kT2Threads - 32;
        for (int idx = tid; idx < ROWS * CH; idx += kQThreads) {
            const int m = idx / CH, c = idx % CH;  // row m of the CTA's 256
            bool valid;
            const __nv_bfloat16 *src;
            if constexpr (PFX) {
                const int64_t row = rows_s[m];
                valid = row >= 0;
                src = p.q + (valid ? row : 0) * D + c * 8;
            } else {
                const int t = t0 + m / GQ;
                valid = t < n;
                src = p.q + (static_cast<size_t>(qs + (valid ? t : 0)) * p.Hq + hk * GQ + m % GQ) * D +
                      c * 8;
            }
            const uint32_t tile = sq + (m >> 7) * (128 * D * 2);
            cp_async16(tile + pa::tc::sw128(m & 127, c * 8, 128), src, valid);
        }
        cp_async_commit();
        cp_async_wait<0>();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("bar.sync 1, %0;" ::"n"(kQThreads) : "memory");
    }

    if (warp == Lay::LOAD_WARP) {
        // ---------------- loader ----------------
        if (lane == 0) {
            const int rows_total = static_cast<int>(p.num_blocks * p.Hkv) << p.bs_log2;
            for (int j = 0; j < ntiles && !*fail; ++j) {
                const int st = j % kT2NST;
                if (j >= kT2NST && !pa::mbar_wait(&kv_empty[st], ((j / kT2NST) - 1) & 1)) {
                    *fail = 1;
                    break;
                }
                pa::mbar_arrive_expect_tx(&kv_full[st], TILE_TX);
                const uint32_t kst = skv + st * 2 * Lay::T_BYTES, vst = kst + Lay::T_BYTES;
                for (int b = 0; b < kT2KT; b += p.bs) {  // bs >= 8: boxes land 1024-aligned
                    const int tok = j * kT2KT + b;
                    const int y = tok < kv_end
                                      ? ((bt_s[tok >> p.bs_log2] * p.Hkv + hk) << p.bs_log2)
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
    } else if (warp == Lay::MMA_WARP) {
        // ---------------- MMA issuer ----------------
        // The whole warp follows the schedule (barrier waits, descriptor
        // arithmetic on warp-uniform values); one elected lane issues each
        // tcgen05 operation.  Shared-memory descriptors are built once and
        // advanced by constant offsets (16-byte units in the start-address
        // field; every operand lies below 227 KB, so the field cannot carry).
        constexpr uint32_t kIdS = pa::tc::idesc_bf16(128, kT2KT, 0, 0);
        constexpr uint32_t kIdO = pa::tc::idesc_bf16(128, D, 0, 1);
        constexpr uint32_t kStage = (2 * Lay::T_BYTES) >> 4;
        const uint64_t dq = pa::tc::sdesc(sq, 16, 1024);
        const uint64_t dk = pa::tc::sdesc(skv, 16, 1024);
        const uint64_t dv = pa::tc::sdesc(skv + Lay::T_BYTES, kT2KT * 128, 1024);
        // S of tile j for group wg goes to TMEM columns 256 + 128 wg + 64 (j % 2)
        auto issue_s = [&](int wg, int j) {
            const uint64_t a0 = dq + static_cast<uint32_t>(wg * ((128 * D * 2) >> 4));
            const uint64_t b0 = dk + static_cast<uint32_t>((j % kT2NST) * kStage);
            const uint32_t sc = tmem + 128 * NQ + wg * 128 + (j & 1) * 64;
            if (pa::tc::elect_one()) {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    pa::tc::mma_ss(sc, a0 + (((ks >> 2) * 128 * 128 + (ks & 3) * 32) >> 4),
                                   b0 + (((ks >> 2) * kT2KT * 128 + (ks & 3) * 32) >> 4), kIdS,
                                   ks > 0);
                pa::tc::commit(&s_full[2 * wg + (j & 1)]);
            }
            __syncwarp();
        };
        // O_wg += P_hi V + P_lo V; P of tile j sits in the S buffer it came from
        auto issue_pv = [&](int wg, int j) {
            const uint64_t b0 = dv + static_cast<uint32_t>((j % kT2NST) * kStage);
            const uint32_t ph = tmem + 128 * NQ + wg * 128 + (j & 1) * 64, pl = ph + 32;
            const uint32_t od = tmem + wg * 128;
            const int acc0 = j > 0;
            if (pa::tc::elect_one()) {
#pragma unroll
                for (int ks = 0; ks < kT2KT / 16; ++ks) {
                    const uint64_t b = b0 + ((ks * 16 * 128) >> 4);
                    pa::tc::mma_ts(od, ph + ks * 8, b, kIdO, ks == 0 ? acc0 : 1);
                    pa::tc::mma_ts(od, pl + ks * 8, b, kIdO, 1);
                }
                pa::tc::commit(&o_done[wg]);
            }
            __syncwarp();
        };
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(pa::kFull, pa::mbar_wait(bar, parity));
        };
        // Issue order: S(0) of both groups; then per tile j: S(j+1) of both
        // groups (its buffer last held P(j-1), whose PV was issued before),
        // PV(j) of group 0, PV(j) of group 1, release of the K/V stage.
        // Group 1's PV of the last tile thus follows group 0's arrival, which
        // comes after group 0 cleared the stale V rows of that tile.
        bool ok = wait_all(&kv_full[0], 0);
        if (ok) {
            pa::tc::fence_after();
            for (int wg = 0; wg < NQ; ++wg) issue_s(wg, 0);
        }
        for (int j = 0; j < ntiles && ok; ++j) {
            if (j + 1 < ntiles) {
                ok = wait_all(&kv_full[(j + 1) % kT2NST], ((j + 1) / kT2NST) & 1);
                if (!ok) break;
                pa::tc::fence_after();
                for (int wg = 0; wg < NQ; ++wg) issue_s(wg, j + 1);
            }
            for (int wg = 0; wg < NQ && ok; ++wg) {
                ok = wait_all(&p_full[wg], j & 1);
                if (!ok) break;
                pa::tc::fence_after();
                issue_pv(wg, j);
            }
            if (ok && pa::tc::elect_one()) pa::tc::commit(&kv_empty[j % kT2NST]);
            __syncwarp();
        }
        if (!ok) *fail = 1;
    } else {
        // ---------------- softmax warp groups ----------------
        const int wg = warp >> 2;                 // query tile A or B
        const int row = tid & 127;                // TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t o_col = wg * 128;
        const int m = wg * 128 + row;
        // last key position this row sees (prefix mode: every key of the chunk)
        const int pos = PFX ? kv_end - 1 : P + min(t0 + m / GQ, n - 1);
        const float qs2 = p.qscale;  // softmax scale in log2 units
        float m_used = -INFINITY, lsum = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const uint32_t s_col = 128 * NQ + wg * 128 + (j & 1) * 64;
            ok = pa::mbar_wait(&s_full[2 * wg + (j & 1)], (j >> 1) & 1);
            if (!ok) break;
            pa::tc::fence_after();
            uint32_t sr[2][32];
            pa::tc::ld32(lane_base + s_col, sr[0]);
            pa::tc::ld32(lane_base + s_col + 32, sr[1]);
            pa::tc::wait_ld();
            const int j0 = j * kT2KT;
            float s[64];
#pragma unroll
            for (int c = 0; c < 64; ++c) s[c] = __uint_as_float(sr[c >> 5][c & 31]);
            if (j0 + kT2KT - 1 > pos) {  // tile on or past the diagonal: mask
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (j0 + c > pos) s[c] = -INFINITY;
            }
            // row maximum: 8 independent chains of three-input maxima
            float mx[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float m3 = max3f(s[e], s[8 + e], s[16 + e]);
                m3 = max3f(m3, s[24 + e], s[32 + e]);
                m3 = max3f(m3, s[40 + e], s[48 + e]);
                mx[e] = fmaxf(m3, s[56 + e]);
            }
            const float tmax =
                max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) *
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
                const float2 lo = pa::ffma2(pa::bf16x2_to_float2(ph[c]), make_float2(-1.f, -1.f),
                                            make_float2(p0, p1));
                pl[c] = pack_bf16(lo.x, lo.y);
            }
            const float rs = ((rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y)) +
                             ((rs2[2].x + rs2[2].y) + (rs2[3].x + rs2[3].y));
            lsum = lsum * alpha + rs;
            if (j > 0) {  // PV(j-1) must be done before O is rescaled
                ok = pa::mbar_wait(&o_done[wg], (j - 1) & 1);
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
            if (j == ntiles - 1 && wg == 0) {
                // rows past the context in the last tile may hold anything
                // (unwritten slots); P is 0 there but 0 * NaN is NaN: zero them.
                // Group 1's PV of this tile is issued after group 0's arrival.
                const int first = kv_end - j0;
                const uint32_t vst = skv + (j % kT2NST) * 2 * Lay::T_BYTES + Lay::T_BYTES;
                for (int idx = row; idx < (kT2KT - first) * CH; idx += 128) {
                    const int rr = first + idx / CH, c = idx % CH;
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                                     vst + pa::tc::sw128(rr, c * 8, kT2KT)),
                                 "r"(0u)
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            pa::tc::st32(lane_base + s_col, ph);
            pa::tc::st32(lane_base + s_col + 32, pl);
            pa::tc::wait_st();
            pa::tc::fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[wg]);
        }
        if (ok) ok = pa::mbar_wait(&o_done[wg], (ntiles - 1) & 1);
        if (ok && PFX) {
            // partial of this (member, head) row over the chunk: unnormalised
            // O, running max and sum, into its prefix slot
            pa::tc::fence_after();
            const int64_t prow = rows_s[m];
            const size_t slot =
                static_cast<size_t>(prow < 0 ? 0 : prow) * p.pfx_rowslots + p.pfx_pslot0 + pchunk;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                pa::tc::ld32(lane_base + o_col + c0, o);
                pa::tc::wait_ld();
                if (prow >= 0) {
                    float *dst = p.pfx_acc + slot * D + c0;
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4 *>(dst + c) =
                            make_float4(__uint_as_float(o[c]), __uint_as_float(o[c + 1]),
                                        __uint_as_float(o[c + 2]), __uint_as_float(o[c + 3]));
                }
            }
            if (prow >= 0)
                *reinterpret_cast<float2 *>(p.pfx_ml + 2 * slot) = make_float2(m_used, lsum);
        } else if (ok) {
            pa::tc::fence_after();
            const int t = t0 + m / GQ;
            const float inv = 1.f / lsum;
            __nv_bfloat16 *dst =
                p.out + (static_cast<size_t>(qs + min(t, n - 1)) * p.Hq + hk * GQ + m % GQ) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                pa::tc::ld32(lane_base + o_col + c0, o);
                pa::tc::wait_ld();
                if (t < n) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w4;
                        w4.x = pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv);
                        w4.y = pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
                        w4.z = pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
                        w4.w = pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + c0 + c) = w4;
                    }
                }
            }
        } else {
            *fail = 1;
        }
    }
    // ---- tear-down ----------------------------------------------------------------
    pa::tc::fence_before();
    __syncthreads();
    if (*fail) {
        // a wait ran out: record it and give the MMAs and copies in flight a
        // bounded chance to land before the TMEM and shared memory go away
        if (tid == 0) {
            pa::record_error(p.err, PA_DEVERR_TIMEOUT);
            for (int i = 0; i < NQ; ++i) (void)pa::mbar_wait(&o_done[i], 0);
            for (int i = 0; i < kT2NST; ++i) (void)pa::mbar_wait(&kv_full[i], 0);
        }
        __syncthreads();
    }
    if (warp == Lay::MMA_WARP) pa::tc::dealloc(tmem, Lay::TMEM_COLS);
    exit_wait();
}


#ifndef PA_PREFILL_TCGEN05
#define PA_PREFILL_TCGEN05 1  // 1: tcgen05 kernel; 0: warp-level mma.sync kernel
#endif
#ifndef PA_PREFILL_NQ
#define PA_PREFILL_NQ 2  // query tiles of 128 rows per CTA of the warp-specialised kernel
#endif

template <int D, int GQ>
int launch_tc(const PrefillParams &p, int max_query_len, cudaStream_t stream) {
    const size_t smem = TcLayout<D>::SMEM;
    auto kern = prefill_tc_kernel<D, GQ>;
    (void)cudaGetLastError();
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "prefill: shared memory attribute");
    constexpr int qtok = 128 / GQ;
    dim3 grid((max_query_len + qtok - 1) / qtok, p.Hkv, p.R);
    kern<<<grid, 128, smem, stream>>>(p);
    return pa::check_launch("prefill launch");
}


// The warp-specialised kernel needs blocks of 8..64 tokens, a block-table
// slice of at most BT_MAX entries and 32-bit pool row coordinates.
template <int D>
bool tc2_ok(const PrefillParams &p) {
    const int64_t rows = (p.num_blocks * p.Hkv) << p.bs_log2;
    return p.bs >= 8 && p.bs <= 64 && p.MB <= Tc2Layout<D, 2>::BT_MAX && rows < (int64_t(1) << 31);
}

template <int D, int GQ>
int launch_tc2(const PrefillParams &p, int max_query_len, cudaStream_t stream) {
    const int64_t rows = (p.num_blocks * p.Hkv) << p.bs_log2;
    CUtensorMap kmap, vmap;
    if (int rc = pa::pool_tensor_map(&kmap, p.k_cache, rows, D, p.bs)) return rc;
    if (int rc = pa::pool_tensor_map(&vmap, p.v_cache, rows, D, p.bs)) return rc;
    using Lay = Tc2Layout<D, PA_PREFILL_NQ>;
    const size_t smem = Lay::SMEM;
    auto kern = prefill_tc2_kernel<D, GQ, false, PA_PREFILL_NQ>;
    static std::atomic<uint64_t> attr_done{0};
    if (int rc = set_smem_once(kern, smem, &attr_done)) return rc;
    (void)cudaGetLastError();
    constexpr int qtok = Lay::ROWS / GQ;
    const int64_t ctas = int64_t((max_query_len + qtok - 1) / qtok) * p.R * p.Hkv;
    if (ctas > 0x7fffffff) return pa::fail(PA_ERR_INVALID, "prefill: grid too large");
    kern<<<static_cast<unsigned>(ctas), Lay::THREADS, smem, stream>>>(p, kmap, vmap);
    return pa::check_launch("prefill launch");
}

#ifndef PA_PREFILL_WARP_SPECIALIZED
#define PA_PREFILL_WARP_SPECIALIZED 1
#endif

#ifndef PA_PREFILL_PERSISTENT
#define PA_PREFILL_PERSISTENT 1  // 1: persistent kernel for batches of at most 512 items
#endif

template <int D, int GQ>
int launch(const PrefillParams &p, int max_query_len, cudaStream_t stream) {
    if (PA_PREFILL_TCGEN05 && PA_PREFILL_WARP_SPECIALIZED && tc2_ok<D>(p)) {
        if (PA_PREFILL_PERSISTENT && persist_ok(p.R, max_query_len, p.Hq, p.Hkv))
            return launch_persist(p, D, GQ, stream);
        return launch_tc2<D, GQ>(p, max_query_len, stream);
    }
    if (PA_PREFILL_TCGEN05) return launch_tc<D, GQ>(p, max_query_len, stream);
    const size_t smem = kRows * D * 2 + 4 * kKT * D * 2;
    auto kern = prefill_kernel<D, GQ>;
    (void)cudaGetLastError();
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "prefill: shared memory attribute");
    constexpr int qtok = kRows / GQ;
    dim3 grid((max_query_len + qtok - 1) / qtok, p.Hkv, p.R);
    kern<<<grid, kThreads, smem, stream>>>(p);
    return pa::check_launch("prefill launch");
}

template <int D>
int dispatch_gq(int gq, const PrefillParams &p, int mq, cudaStream_t s) {
    switch (gq) {
        case 1: return launch<D, 1>(p, mq, s);
        case 2: return launch<D, 2>(p, mq, s);
        case 4: return launch<D, 4>(p, mq, s);
        case 8: return launch<D, 8>(p, mq, s);
        default: return pa::fail(PA_ERR_UNSUPPORTED, "prefill: Hq/Hkv=%d unsupported", gq);
    }
}

template <int D, int GQ>
int launch_prefix_tc_t(const pa::PrefixTcArgs &a, cudaStream_t stream) {
    PrefillParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.k_cache = static_cast<const uint8_t *>(a.k_cache);
    p.v_cache = static_cast<const uint8_t *>(a.v_cache);
    p.block_table = a.block_table;
    p.context_lens = a.context_lens;
    p.err = a.err;
    p.num_blocks = a.num_blocks;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.bs = a.bs;
    p.bs_log2 = log2_int(a.bs);
    p.MB = a.MB;
    p.qscale = a.qscale;
    p.pfx_group_start = a.group_start;
    p.pfx_group_seqs = a.group_seqs;
    p.pfx_shared_len = a.shared_len;
    p.pfx_acc = a.acc;
    p.pfx_ml = a.ml;
    p.pfx_G = a.G;
    p.pfx_nc = a.nc;
    constexpr int qtok = 256 / GQ;
    p.pfx_nmt = (a.max_group_size + qtok - 1) / qtok;
    p.pfx_members = a.num_members;
    p.pfx_rowslots = a.rowslots;
    p.pfx_pslot0 = a.pslot0;
    p.pfx_B = a.B;
    p.pfx_wait_end = a.after_decode ? 1 : 0;
    const int64_t rows = (a.num_blocks * a.Hkv) << p.bs_log2;
    CUtensorMap kmap, vmap;
    if (int rc = pa::pool_tensor_map(&kmap, a.k_cache, rows, D, a.bs)) return rc;
    if (int rc = pa::pool_tensor_map(&vmap, a.v_cache, rows, D, a.bs)) return rc;
    using Lay = Tc2Layout<D, 2>;
    const size_t smem = Lay::SMEM;
    auto kern = prefill_tc2_kernel<D, GQ, true, 2>;
    static std::atomic<uint64_t> attr_done{0};
    if (int rc = set_smem_once(kern, smem, &attr_done)) return rc;
    const int64_t ctas = int64_t(p.pfx_nmt) * a.G * a.nc * a.Hkv;
    if (ctas > 0x7fffffff) return pa::fail(PA_ERR_INVALID, "decode_shared: prefix grid too large");
    if (ctas == 0) return PA_OK;
    (void)cudaGetLastError();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(Lay::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p, kmap, vmap);
    if (e != cudaSuccess) return pa::cuda_fail(e, "decode_shared: prefix launch");
    return pa::check_launch("decode_shared: prefix launch");
}

}  // namespace

namespace pa {

bool prefix_tc_ok(int bs, int64_t num_blocks, int Hkv, int max_chunk_tokens) {
    return bs >= 8 && bs <= 64 && (num_blocks * Hkv * bs) < (int64_t(1) << 31) &&
           (max_chunk_tokens + bs - 1) / bs <= Tc2Layout<128>::BT_MAX;
}

int launch_prefix_tc(const PrefixTcArgs &a, cudaStream_t stream) {
    const int gq = a.Hq / a.Hkv;
    auto pick = [&](auto d) -> int {
        constexpr int D = decltype(d)::value;
        switch (gq) {
            case 1: return launch_prefix_tc_t<D, 1>(a, stream);
            case 2: return launch_prefix_tc_t<D, 2>(a, stream);
            case 4: return launch_prefix_tc_t<D, 4>(a, stream);
            case 8: return launch_prefix_tc_t<D, 8>(a, stream);
            default: return pa::fail(PA_ERR_UNSUPPORTED, "decode_shared: Hq/Hkv=%d", gq);
        }
    };
    if (a.D == 128) return pick(std::integral_constant<int, 128>{});
    if (a.D == 64) return pick(std::integral_constant<int, 64>{});
    return pa::fail(PA_ERR_UNSUPPORTED, "decode_shared: head_dim %d", a.D);
}

}  // namespace pa

namespace {

int check_sizes(int R, int max_query_len, int Hq, int Hkv, int head_dim, int block_size,
                int64_t num_blocks, int max_blocks_per_seq) {
    if (R < 0 || R > 65535 || Hq <= 0 || Hkv <= 0 || Hkv > 65535 || Hq % Hkv ||
        max_query_len < 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return pa::fail(PA_ERR_INVALID, "prefill: bad sizes");
    if (head_dim != 64 && head_dim != 128)
        return pa::fail(PA_ERR_UNSUPPORTED, "prefill: head_dim %d unsupported", head_dim);
    if (Hq / Hkv != 1 && Hq / Hkv != 2 && Hq / Hkv != 4 && Hq / Hkv != 8)
        return pa::fail(PA_ERR_UNSUPPORTED, "prefill: Hq/Hkv=%d unsupported", Hq / Hkv);
    if (!pa::pow2_in(block_size, 8, 128))
        return pa::fail(PA_ERR_UNSUPPORTED, "prefill: block_size %d unsupported", block_size);
    if (int64_t(max_blocks_per_seq) * block_size > (int64_t(1) << 30))
        return pa::fail(PA_ERR_INVALID, "prefill: table capacity too large");
    return PA_OK;
}

}  // namespace

extern "C" int pa_prefill_kernel_for(int R, int max_query_len, int Hq, int Hkv, int head_dim,
                                     int block_size, int64_t num_blocks, int max_blocks_per_seq,
                                     int *kernel) {
    pa::clear_error();
    if (!kernel) return pa::fail(PA_ERR_INVALID, "prefill_kernel_for: NULL kernel");
    if (int rc = check_sizes(R, max_query_len, Hq, Hkv, head_dim, block_size, num_blocks,
                             max_blocks_per_seq))
        return rc;
    PrefillParams p{};
    p.num_blocks = num_blocks;
    p.Hkv = Hkv;
    p.bs = block_size;
    p.bs_log2 = log2_int(block_size);
    p.MB = max_blocks_per_seq;
    if (!(PA_PREFILL_TCGEN05 && PA_PREFILL_WARP_SPECIALIZED && tc2_ok<128>(p)))
        *kernel = PA_PREFILL_SIMPLE;
    else if (PA_PREFILL_PERSISTENT && persist_ok(R, max_query_len, Hq, Hkv))
        *kernel = PA_PREFILL_PERSISTENT_GRID;
    else
        *kernel = PA_PREFILL_ITEM_GRID;
    return PA_OK;
}

extern "C" int pa_prefill_chunk(void *out, const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_table, int max_blocks_per_seq,
                                const int32_t *query_start, const int32_t *context_lens, int R,
                                int max_query_len, int Hq, int Hkv, int head_dim, int block_size,
                                int64_t num_blocks, float scale, int dtype, pa_stream_t stream) {
    pa::clear_error();
    if (dtype != PA_BF16)
        return pa::fail(PA_ERR_UNSUPPORTED, "prefill: only bf16 is supported (dtype %d)", dtype);
    if (int rc = check_sizes(R, max_query_len, Hq, Hkv, head_dim, block_size, num_blocks,
                             max_blocks_per_seq))
        return rc;
    if (!(scale > 0.f) || !std::isfinite(scale))
        return pa::fail(PA_ERR_INVALID, "prefill: scale must be positive and finite");
    if (R == 0 || max_query_len == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !query_start || !context_lens)
        return pa::fail(PA_ERR_INVALID, "prefill: NULL pointer");
    if (!pa::aligned16(q) || !pa::aligned16(out) || !pa::aligned16(k_cache) ||
        !pa::aligned16(v_cache))
        return pa::fail(PA_ERR_INVALID, "prefill: tensors must be 16-byte aligned");
    if (pa::validate_on()) {
        std::vector<int32_t> qsv(R + 1), lens(R), table(size_t(R) * max_blocks_per_seq);
        if (int rc = pa::fetch(qsv.data(), query_start, (R + 1) * sizeof(int32_t), stream))
            return rc;
        if (int rc = pa::fetch(lens.data(), context_lens, R * sizeof(int32_t), stream)) return rc;
        if (int rc = pa::fetch(table.data(), block_table, table.size() * sizeof(int32_t), stream))
            return rc;
        const int64_t cap = int64_t(max_blocks_per_seq) * block_size;
        for (int r = 0; r < R; ++r) {
            const int nr = qsv[r + 1] - qsv[r];
            if (nr < 0 || nr > max_query_len)
                return pa::fail(PA_ERR_INVALID, "validate: request %d has %d new tokens", r, nr);
            if (lens[r] < nr || lens[r] > cap)
                return pa::fail(PA_ERR_INVALID, "validate: context_lens[%d]=%d", r, lens[r]);
            const int nb = (lens[r] + block_size - 1) / block_size;
            for (int i = 0; i < nb; ++i) {
                const int32_t v = table[size_t(r) * max_blocks_per_seq + i];
                if (v < 0 || v >= num_blocks)
                    return pa::fail(PA_ERR_INVALID, "validate: block_table[%d][%d]=%d", r, i, v);
            }
        }
    }
    PrefillParams p{};
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_cache = static_cast<const uint8_t *>(k_cache);
    p.v_cache = static_cast<const uint8_t *>(v_cache);
    p.block_table = block_table;
    p.query_start = query_start;
    p.context_lens = context_lens;
    p.err = pa::device_error_word();
    p.num_blocks = num_blocks;
    p.R = R;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.bs = block_size;
    p.bs_log2 = log2_int(block_size);
    p.MB = max_blocks_per_seq;
    p.max_query_len = max_query_len;
    p.qscale = scale * kLog2e;
    const int gq = Hq / Hkv;
    return head_dim == 128 ? dispatch_gq<128>(gq, p, max_query_len, stream)
                           : dispatch_gq<64>(gq, p, max_query_len, stream);
}
