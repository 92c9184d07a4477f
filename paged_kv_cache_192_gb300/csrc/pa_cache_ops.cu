// reshape_and_cache and copy_blocks: the bit-exact data movement of the
// paged KV cache.  Both are HBM-bound copies done in 16-byte vectors.
#include <algorithm>
#include <unordered_set>
#include <vector>

#include "pa_device.cuh"
#include "pa_internal.h"

#ifndef PA_STORE_PDL
#define PA_STORE_PDL 1  // 0: ordinary stream-ordered launch (A/B of the dependent launch)
#endif

namespace {

// One thread per 16-byte chunk of one (token, KV head) row.  Source rows are
// contiguous ([T][Hkv][row]); the destination of row (t, h) is
// [slot / bs][h][slot % bs] in the pool.  Negative slots are padding.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, const int64_t *__restrict__ slots, int64_t total, int Hkv,
    int bs_log2, int chunks, int64_t num_blocks, int *err) {
    // Launched as a programmatic dependent: wait for the kernels before it
    // (they may still read the pool), then let the next kernel in the stream
    // (typically the decode that reads these rows) start launching; that
    // kernel waits for this grid to complete before it reads anything.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += stride) {
        const int64_t row = i / chunks;
        const int c = static_cast<int>(i - row * chunks);
        const int64_t t = row / Hkv;
        const int h = static_cast<int>(row - t * Hkv);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        const int64_t blk = slot >> bs_log2;
        const int64_t off = slot & ((1ll << bs_log2) - 1);
        if (blk >= num_blocks) {
            pa::record_error(err, PA_DEVERR_BAD_BLOCK);
            continue;
        }
        const int64_t dst = (((blk * Hkv + h) << bs_log2) + off) * chunks + c;
        k_cache[dst] = __ldg(k_new + i);
        v_cache[dst] = __ldg(v_new + i);
    }
}

// blockIdx.x = pair, blockIdx.y = cache (0: K, 1: V).  Each CTA copies one
// whole physical block of one cache.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *__restrict__ k_cache,
                                                          uint4 *__restrict__ v_cache,
                                                          const int64_t *__restrict__ pairs,
                                                          int64_t chunks_per_block,
                                                          int64_t num_blocks, int *err) {
    const int64_t p = blockIdx.x;
    const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
        if (threadIdx.x == 0) pa::record_error(err, PA_DEVERR_BAD_BLOCK);
        return;
    }
    uint4 *base = blockIdx.y ? v_cache : k_cache;
    const uint4 *s = base + src * chunks_per_block;
    uint4 *d = base + dst * chunks_per_block;
    for (int64_t i = threadIdx.x; i < chunks_per_block; i += blockDim.x) d[i] = s[i];
}

// blockIdx.x = pair, blockIdx.y = cache (0: K, 1: V): block dst of the
// destination pool becomes a copy of block src of the source pool (either
// pool may be pinned host memory reached through its device alias).
__global__ void __launch_bounds__(256) swap_blocks_kernel(uint4 *__restrict__ dst_k,
                                                          uint4 *__restrict__ dst_v,
                                                          const uint4 *__restrict__ src_k,
                                                          const uint4 *__restrict__ src_v,
                                                          const int64_t *__restrict__ pairs,
                                                          int64_t chunks_per_block,
                                                          int64_t src_blocks, int64_t dst_blocks,
                                                          int *err) {
    const int64_t p = blockIdx.x;
    const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || dst < 0 || src >= src_blocks || dst >= dst_blocks) {
        if (threadIdx.x == 0) pa::record_error(err, PA_DEVERR_BAD_BLOCK);
        return;
    }
    const uint4 *s = (blockIdx.y ? src_v : src_k) + src * chunks_per_block;
    uint4 *d = (blockIdx.y ? dst_v : dst_k) + dst * chunks_per_block;
    for (int64_t i = threadIdx.x; i < chunks_per_block; i += blockDim.x) d[i] = s[i];
}

// Device address of a pool: device memory as is, pinned host memory through
// its mapped device alias; anything else is rejected.
int device_view(const void *ptr, void **dev, const char *what) {
    cudaPointerAttributes a{};
    cudaError_t e = cudaPointerGetAttributes(&a, ptr);
    if (e != cudaSuccess) return pa::cuda_fail(e, what);
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
        *dev = const_cast<void *>(ptr);
        return PA_OK;
    }
    if (a.type == cudaMemoryTypeHost) {
        if (a.devicePointer) {
            *dev = a.devicePointer;
            return PA_OK;
        }
        e = cudaHostGetDevicePointer(dev, const_cast<void *>(ptr), 0);
        return e == cudaSuccess ? PA_OK : pa::cuda_fail(e, what);
    }
    return pa::fail(PA_ERR_INVALID, "%s: pool must be device or pinned host memory", what);
}

int log2_int(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

int grid_for(int64_t work, int threads) {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (work + threads - 1) / threads;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(sms) * 16)));
}

}  // namespace

extern "C" {

int pa_reshape_and_cache(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t T, int64_t num_blocks, int Hkv,
                         int block_size, int head_dim, int dtype, pa_stream_t stream) {
    pa::clear_error();
    const size_t es = pa::dtype_size(dtype);
    if (!es) return pa::fail(PA_ERR_INVALID, "reshape_and_cache: bad dtype %d", dtype);
    if (T < 0 || num_blocks <= 0 || Hkv <= 0 || head_dim <= 0)
        return pa::fail(PA_ERR_INVALID, "reshape_and_cache: bad sizes");
    if (!pa::pow2_in(block_size, 1, 1024))
        return pa::fail(PA_ERR_INVALID, "reshape_and_cache: block_size must be a power of two");
    if ((head_dim * es) % 16)
        return pa::fail(PA_ERR_INVALID, "reshape_and_cache: row bytes must be a multiple of 16");
    if (T == 0) return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
        return pa::fail(PA_ERR_INVALID, "reshape_and_cache: NULL pointer");
    if (!pa::aligned16(k_new) || !pa::aligned16(v_new) || !pa::aligned16(k_cache) ||
        !pa::aligned16(v_cache))
        return pa::fail(PA_ERR_INVALID, "reshape_and_cache: pointers must be 16-byte aligned");
    if (pa::validate_on()) {
        std::vector<int64_t> s(T);
        if (int rc = pa::fetch(s.data(), slot_mapping, T * sizeof(int64_t), stream)) return rc;
        std::unordered_set<int64_t> seen;
        for (int64_t t = 0; t < T; ++t) {
            if (s[t] < 0) continue;
            if (s[t] >= num_blocks * block_size)
                return pa::fail(PA_ERR_INVALID, "validate: slot %lld of token %lld out of pool",
                                (long long)s[t], (long long)t);
            if (!seen.insert(s[t]).second)
                return pa::fail(PA_ERR_INVALID, "validate: duplicate slot %lld", (long long)s[t]);
        }
    }
    const int chunks = static_cast<int>(head_dim * es / 16);
    const int64_t total = T * Hkv * chunks;
    (void)cudaGetLastError();  // drop a stale error that is not ours
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_for(total, 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PA_STORE_PDL ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, reshape_and_cache_kernel, static_cast<const uint4 *>(k_new),
        static_cast<const uint4 *>(v_new), static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), slot_mapping, total, Hkv, log2_int(block_size), chunks,
        num_blocks, pa::device_error_word());
    if (e != cudaSuccess) return pa::cuda_fail(e, "reshape_and_cache launch");
    return pa::check_launch("reshape_and_cache launch");
}

int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int64_t n,
                   int64_t num_blocks, int Hkv, int block_size, int head_dim, int dtype,
                   pa_stream_t stream) {
    pa::clear_error();
    const size_t es = pa::dtype_size(dtype);
    if (!es) return pa::fail(PA_ERR_INVALID, "copy_blocks: bad dtype %d", dtype);
    if (n < 0 || num_blocks <= 0 || Hkv <= 0 || block_size <= 0 || head_dim <= 0)
        return pa::fail(PA_ERR_INVALID, "copy_blocks: bad sizes");
    const size_t block_bytes = size_t(Hkv) * block_size * head_dim * es;
    if (block_bytes % 16) return pa::fail(PA_ERR_INVALID, "copy_blocks: block bytes % 16 != 0");
    if (n == 0) return PA_OK;
    if (!k_cache || !v_cache || !pairs) return pa::fail(PA_ERR_INVALID, "copy_blocks: NULL");
    if (!pa::aligned16(k_cache) || !pa::aligned16(v_cache))
        return pa::fail(PA_ERR_INVALID, "copy_blocks: pools must be 16-byte aligned");
    if (n > 0x7fffffff) return pa::fail(PA_ERR_INVALID, "copy_blocks: too many pairs");
    if (pa::validate_on()) {
        std::vector<int64_t> p(2 * n);
        if (int rc = pa::fetch(p.data(), pairs, 2 * n * sizeof(int64_t), stream)) return rc;
        std::unordered_set<int64_t> srcs, dsts;
        for (int64_t i = 0; i < n; ++i) {
            for (int j = 0; j < 2; ++j)
                if (p[2 * i + j] < 0 || p[2 * i + j] >= num_blocks)
                    return pa::fail(PA_ERR_INVALID, "validate: pair %lld outside the pool",
                                    (long long)i);
            srcs.insert(p[2 * i]);
            if (!dsts.insert(p[2 * i + 1]).second)
                return pa::fail(PA_ERR_INVALID, "validate: duplicate destination block");
        }
        for (int64_t d : dsts)
            if (srcs.count(d)) return pa::fail(PA_ERR_INVALID, "validate: dst is also a src");
    }
    dim3 grid(static_cast<unsigned>(n), 2);
    (void)cudaGetLastError();
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), pairs,
        static_cast<int64_t>(block_bytes / 16), num_blocks, pa::device_error_word());
    return pa::check_launch("copy_blocks launch");
}

int pa_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                   const int64_t *pairs, int64_t n, int64_t src_num_blocks,
                   int64_t dst_num_blocks, int Hkv, int block_size, int head_dim, int dtype,
                   pa_stream_t stream) {
    pa::clear_error();
    const size_t es = pa::dtype_size(dtype);
    if (!es) return pa::fail(PA_ERR_INVALID, "swap_blocks: bad dtype %d", dtype);
    if (n < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || Hkv <= 0 || block_size <= 0 ||
        head_dim <= 0)
        return pa::fail(PA_ERR_INVALID, "swap_blocks: bad sizes");
    const size_t block_bytes = size_t(Hkv) * block_size * head_dim * es;
    if (block_bytes % 16) return pa::fail(PA_ERR_INVALID, "swap_blocks: block bytes % 16 != 0");
    if (n == 0) return PA_OK;
    if (!dst_k || !dst_v || !src_k || !src_v || !pairs)
        return pa::fail(PA_ERR_INVALID, "swap_blocks: NULL pointer");
    if (!pa::aligned16(dst_k) || !pa::aligned16(dst_v) || !pa::aligned16(src_k) ||
        !pa::aligned16(src_v))
        return pa::fail(PA_ERR_INVALID, "swap_blocks: pools must be 16-byte aligned");
    if (n > 0x7fffffff) return pa::fail(PA_ERR_INVALID, "swap_blocks: too many pairs");
    void *dk, *dv, *sk2, *sv2, *pp;
    if (int rc = device_view(dst_k, &dk, "swap_blocks dst_k")) return rc;
    if (int rc = device_view(dst_v, &dv, "swap_blocks dst_v")) return rc;
    if (int rc = device_view(src_k, &sk2, "swap_blocks src_k")) return rc;
    if (int rc = device_view(src_v, &sv2, "swap_blocks src_v")) return rc;
    if (int rc = device_view(pairs, &pp, "swap_blocks pairs")) return rc;
    if (pa::validate_on()) {
        std::vector<int64_t> p(2 * n);
        if (int rc = pa::fetch(p.data(), pairs, 2 * n * sizeof(int64_t), stream)) return rc;
        std::unordered_set<int64_t> dsts;
        for (int64_t i = 0; i < n; ++i) {
            if (p[2 * i] < 0 || p[2 * i] >= src_num_blocks || p[2 * i + 1] < 0 ||
                p[2 * i + 1] >= dst_num_blocks)
                return pa::fail(PA_ERR_INVALID, "validate: swap pair %lld outside its pool",
                                (long long)i);
            if (!dsts.insert(p[2 * i + 1]).second)
                return pa::fail(PA_ERR_INVALID, "validate: duplicate destination block");
        }
    }
    dim3 grid(static_cast<unsigned>(n), 2);
    (void)cudaGetLastError();
    swap_blocks_kernel<<<grid, 256, 0, stream>>>(
        static_cast<uint4 *>(dk), static_cast<uint4 *>(dv), static_cast<const uint4 *>(sk2),
        static_cast<const uint4 *>(sv2), static_cast<const int64_t *>(pp),
        static_cast<int64_t>(block_bytes / 16), src_num_blocks, dst_num_blocks,
        pa::device_error_word());
    return pa::check_launch("swap_blocks launch");
}

}  // extern "C"
