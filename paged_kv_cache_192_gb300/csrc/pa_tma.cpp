// Tensor maps (TMA descriptors) over the paged K/V pools, shared by the
// prefill and decode kernels that load pool rows with 2D tensor copies.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// libcuda link dependency), looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        (void)cudaGetLastError();
    });
    return fn;
}

int encode_pool_map(CUtensorMap *map, const void *pool, int64_t rows, int D, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(PA_ERR_UNSUPPORTED, "no cuTensorMapEncodeTiled");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : fail(PA_ERR_CUDA, "tensor map encode failed (%d)", (int)r);
}

int encode_q_map(CUtensorMap *map, const void *q, int64_t tokens, int Hq, int D, int gq,
                 int box_tokens) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(PA_ERR_UNSUPPORTED, "no cuTensorMapEncodeTiled");
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                                static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(Hq) * D * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(gq), static_cast<cuuint32_t>(box_tokens)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : fail(PA_ERR_CUDA, "tensor map encode failed (%d)", (int)r);
}

}  // namespace

// Query rows [tokens][Hq][D] (bf16) viewed as a 3D tensor, read in boxes of
// 64 columns x gq heads x box_tokens tokens (rows of 128 bytes, the 128-byte
// swizzle).  Cached by value like the pool maps.
int q_tensor_map(CUtensorMap *map, const void *q, int64_t tokens, int Hq, int D, int gq,
                 int box_tokens) {
    struct Entry {
        const void *q;
        int64_t tokens;
        int Hq, D, gq, box_tokens;
        CUtensorMap map;
    };
    constexpr int kSlots = 8;
    static std::mutex mu;
    static Entry cache[kSlots];
    static int used = 0, next = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].q == q && cache[i].tokens == tokens && cache[i].Hq == Hq &&
                cache[i].D == D && cache[i].gq == gq && cache[i].box_tokens == box_tokens) {
                *map = cache[i].map;
                return PA_OK;
            }
    }
    if (int rc = encode_q_map(map, q, tokens, Hq, D, gq, box_tokens)) return rc;
    std::lock_guard<std::mutex> lk(mu);
    cache[next] = Entry{q, tokens, Hq, D, gq, box_tokens, *map};
    next = (next + 1) % kSlots;
    if (used < kSlots) ++used;
    return PA_OK;
}

// A bf16 pool viewed as a 2D tensor of rows (block, KV head, slot) x D,
// read in boxes of 64 columns x box_rows rows with the 128-byte swizzle.
// A map is a pure function of its arguments, so the last few encoded maps
// are kept and reused by value: a serving loop calls with the same pools
// every step and the encode (host work of a few microseconds per map) is
// then paid once.
int pool_tensor_map(CUtensorMap *map, const void *pool, int64_t rows, int D, int box_rows) {
    struct Entry {
        const void *pool;
        int64_t rows;
        int D, box_rows;
        CUtensorMap map;
    };
    constexpr int kSlots = 8;
    static std::mutex mu;
    static Entry cache[kSlots];
    static int used = 0, next = 0;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].pool == pool && cache[i].rows == rows && cache[i].D == D &&
                cache[i].box_rows == box_rows) {
                *map = cache[i].map;
                return PA_OK;
            }
    }
    if (int rc = encode_pool_map(map, pool, rows, D, box_rows)) return rc;
    std::lock_guard<std::mutex> lk(mu);
    cache[next] = Entry{pool, rows, D, box_rows, *map};
    next = (next + 1) % kSlots;
    if (used < kSlots) ++used;
    return PA_OK;
}

}  // namespace pa
