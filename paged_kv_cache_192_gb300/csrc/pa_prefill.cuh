// Pieces shared by the prefill translation units: the launch parameters and
// small device helpers (cp.async, bf16 packing, TMA tensor copies, mbarrier
// arrival) and the host helpers that set a kernel's shared-memory limit.
#pragma once

#include <cuda.h>

#include <atomic>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace pf {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kT2KT = 64;  // KV tokens per tile of the tcgen05 kernels
#ifndef PA_PREFILL_TAU
#define PA_PREFILL_TAU 8.0f
#endif
constexpr float kTcTau = PA_PREFILL_TAU;  // lazy-rescale headroom (log2 units)

struct PrefillParams {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const uint8_t *k_cache;
    const uint8_t *v_cache;
    const int32_t *block_table;
    const int32_t *query_start;
    const int32_t *context_lens;
    int *err;
    int64_t num_blocks;
    int R, Hq, Hkv, bs, bs_log2, MB, max_query_len;
    float qscale;
    // shared-prefix mode of prefill_tc2_kernel (pa::launch_prefix_tc): rows are
    // (group member, query head) pairs of a decode batch, all attending to
    // the group's shared tokens [t_lo, t_hi) of one token chunk; the result is
    // a log-sum-exp partial in the decode workspace
    const int32_t *pfx_group_start, *pfx_group_seqs, *pfx_shared_len;
    float *pfx_acc, *pfx_ml;
    int pfx_G, pfx_nc, pfx_nmt, pfx_members, pfx_rowslots, pfx_pslot0, pfx_B;
    // prefix mode launched behind the decode grid, whose outputs it does not
    // read: no wait before the work, a wait for that grid before exiting (so
    // that a kernel waiting for this one also finds the decode complete)
    int pfx_wait_end;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;  // 0: zero-fill without reading
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(pa::smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(pa::smem_u32(bar)) : "memory");
}

inline int log2_int(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

// cudaFuncSetAttribute for the dynamic shared memory of `kern`, once per
// device (bit d of *done).
template <typename K>
inline int set_smem_once(K kern, size_t smem, std::atomic<uint64_t> *done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return pa::cuda_fail(cudaGetLastError(), "prefill: device");
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (done->load(std::memory_order_acquire) & bit)) return PA_OK;
    (void)cudaGetLastError();
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return pa::cuda_fail(e, "prefill: shared memory attribute");
    if (bit) done->fetch_or(bit, std::memory_order_acq_rel);
    return PA_OK;
}

// Persistent tcgen05 prefill (pa_prefill_persist.cu): one CTA per SM runs a
// list of (request, 256 query rows, KV head) items.  Usable when the batch
// has at most 256 (request, query tile) pairs and 512 items, with the block
// sizes, table lengths and pool sizes of the warp-specialised kernel.
bool persist_ok(int R, int max_query_len, int Hq, int Hkv);
int launch_persist(const PrefillParams &p, int D, int gq, cudaStream_t stream);

}  // namespace pf
}  // namespace pa
