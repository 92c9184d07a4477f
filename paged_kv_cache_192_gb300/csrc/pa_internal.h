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

inline size_t dtype_size(int dtype) { return dtype == PA_BF16 ? 2 : (dtype == PA_F32 ? 4 : 0); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

// Copy `bytes` of device memory to a host buffer, synchronizing `stream`
// (validate mode only).
int fetch(void *host, const void *dev, size_t bytes, cudaStream_t stream);

}  // namespace pa
