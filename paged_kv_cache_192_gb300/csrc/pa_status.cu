// Error reporting, validate mode and the device error word.
#include <cstdio>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {
thread_local std::string g_msg;
bool g_validate = false;
constexpr int kMaxDevices = 64;
int *g_word_ptr[kMaxDevices] = {};
std::mutex g_word_mu;
}  // namespace

// One error word per device; kernels OR PA_DEVERR_* bits into it.
__device__ int g_pa_device_error = 0;

namespace {

// One warp waits, with the library's bounded pipeline wait, on an mbarrier
// that nothing arrives on.  When the wait runs out it records
// PA_DEVERR_TIMEOUT and returns, as a decode or prefill kernel does when a
// copy never lands.
__global__ void wait_timeout_kernel(int *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        pa::mbar_init(&bar, 1);
        pa::fence_barrier_init();
    }
    __syncwarp();
    const bool ok = __all_sync(pa::kFull, pa::mbar_wait(&bar, 0));
    if (!ok && threadIdx.x == 0) pa::record_error(err, PA_DEVERR_TIMEOUT);
}

}  // namespace

namespace pa {

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_msg = buf;
    return code;
}

void clear_error() { g_msg.clear(); }

bool validate_on() { return g_validate; }

int *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_word_mu);
    if (!g_word_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_device_error) != cudaSuccess) return nullptr;
        g_word_ptr[dev] = static_cast<int *>(p);
    }
    return g_word_ptr[dev];
}

int fetch(void *host, const void *dev, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return PA_OK;
    cudaError_t e = cudaMemcpyAsync(host, dev, bytes, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "validate: device-to-host copy");
}

}  // namespace pa

extern "C" {

const char *pa_last_error_string(void) { return g_msg.c_str(); }

int pa_version(void) { return 1; }

int pa_set_validate(int on) {
    g_validate = on != 0;
    return PA_OK;
}

int pa_device_error(int *bits, int clear, pa_stream_t stream) {
    pa::clear_error();
    if (!bits) return pa::fail(PA_ERR_INVALID, "pa_device_error: bits is NULL");
    int *word = pa::device_error_word();
    if (!word) return pa::fail(PA_ERR_CUDA, "pa_device_error: no device error word");
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, word, sizeof v, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(word, 0, sizeof v, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return pa::cuda_fail(e, "pa_device_error");
    *bits = v;
    return v ? pa::fail(PA_ERR_DEVICE, "device error bits 0x%x", v) : PA_OK;
}

int pa_check_wait_timeout(pa_stream_t stream) {
    pa::clear_error();
    int *word = pa::device_error_word();
    if (!word) return pa::fail(PA_ERR_CUDA, "pa_check_wait_timeout: no device error word");
    (void)cudaGetLastError();
    wait_timeout_kernel<<<1, 32, 0, stream>>>(word);
    return pa::check_launch("wait-timeout check launch");
}

}  // extern "C"
