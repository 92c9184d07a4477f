// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdint>
#include <string>

#include "pa.h"

namespace pa {

// Record a message for pa_last_error_string() and return `code`.
int fail(int code, const char *fmt, ...);
// Clear the message (called at the start of every API entry).
void clear_error();
// Validate mode switch (pa_set_validate).
bool validate_on();
// Device address of the device error word of the current device.
int *device_error_word();

inline int cuda_fail(cudaError_t e, const char *what) {
    (void)cudaGetLastError();  // do not leave the error for the next call to find
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline int check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, what);
}

// 2D tensor map (128-byte swizzle, boxes of 64 columns x box_rows rows) over
// a bf16 pool of `rows` rows of D elements; cached by value (pa_tma.cpp).
int pool_tensor_map(CUtensorMap *map, const void *pool, int64_t rows, int D, int box_rows);
// 3D tensor map over query rows [tokens][Hq][D] (bf16): boxes of 64 columns x
// gq heads x box_tokens tokens, 128-byte swizzle; gq * box_tokens rows of
// 128 bytes per box (a multiple of 8, at most 256 tokens).
int q_tensor_map(CUtensorMap *map, const void *q, int64_t tokens, int Hq, int D, int gq,
                 int box_tokens);

inline size_t dtype_size(int dtype) { return dtype == PA_BF16 ? 2 : (dtype == PA_F32 ? 4 : 0); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

// Shared-prefix partials on the tcgen05 prefill kernel (pa_decode_shared):
// for every group, member tile of prefix_tc_members(Hq / Hkv) members, KV
// head and token chunk, one CTA computes the (max, sum, unnormalised O)
// partial of each (member, query head) over the chunk of the group's shared
// tokens and writes it to slot pslot0 + chunk of the member's decode
// workspace row.  Launched as a programmatic dependent of the previous kernel.
struct PrefixTcArgs {
    const void *q, *k_cache, *v_cache;
    const int32_t *block_table, *context_lens, *group_start, *group_seqs, *shared_len;
    float *acc, *ml;
    int *err;
    int64_t num_blocks;
    int B, Hq, Hkv, D, bs, MB, G, nc, max_group_size, num_members, rowslots, pslot0;
    float qscale;  // softmax scale * log2(e)
    // launched behind the decode grid (whose trigger follows its own wait for
    // the inputs) instead of before it: the kernel waits for that grid only
    // before exiting, so its CTAs fill the SMs the decode grid leaves
    bool after_decode;
};
inline int prefix_tc_members(int gq) { return 256 / gq; }
// Block sizes 8..64, 32-bit pool rows and chunks of at most 1024 blocks.
bool prefix_tc_ok(int bs, int64_t num_blocks, int Hkv, int max_chunk_tokens);
int launch_prefix_tc(const PrefixTcArgs &a, cudaStream_t stream);

// Copy `bytes` of device memory to a host buffer, synchronizing `stream`
// (validate mode only).
int fetch(void *host, const void *dev, size_t bytes, cudaStream_t stream);

}  // namespace pa
