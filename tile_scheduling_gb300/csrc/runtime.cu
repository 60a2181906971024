// Library runtime: error reporting, device properties, the device status word.
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "common.h"

namespace ts {

__device__ unsigned long long g_status_word[kStatusWords];

namespace {
thread_local std::string t_detail;
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int g_smem_optin[kMaxDevices];
unsigned long long *g_status_ptr[kMaxDevices];
std::mutex g_mu;

const char *wait_name(int where) {
    switch (where) {
        case WAIT_PRODUCER_EMPTY: return "producer waiting for an empty ring stage";
        case WAIT_MMA_FULL: return "MMA waiting for a full ring stage";
        case WAIT_MMA_TMEM_EMPTY: return "MMA waiting for a free TMEM accumulator";
        case WAIT_EPI_TMEM_FULL: return "epilogue waiting for a finished accumulator";
        case WAIT_SCHED_CLC_EMPTY: return "CLC scheduler waiting for a free response slot";
        case WAIT_CLC_FULL: return "waiting for a CLC response";
        case WAIT_DRAIN: return "waiting for in-flight copies at exit";
        case WAIT_ROWS_CLC: return "row copy waiting for a CLC response";
        case WAIT_SCHED_PRODUCER: return "CLC scheduler waiting for the producer to begin its unit";
        default: return "unknown wait";
    }
}
}  // namespace

ts_status fail(ts_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_detail = buf;
    return s;
}

ts_status cuda_fail(cudaError_t e, const char *what) {
    return fail(TS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return 0;
    return d;
}

int device_sms(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return -1;
    std::lock_guard<std::mutex> g(g_mu);
    if (g_sms[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        g_sms[dev] = v;
    }
    return g_sms[dev];
}

int device_smem_optin(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return -1;
    std::lock_guard<std::mutex> g(g_mu);
    if (g_smem_optin[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return -1;
        g_smem_optin[dev] = v;
    }
    return g_smem_optin[dev];
}

unsigned long long *device_status_word(ts_status *err) {
    const int dev = current_device();
    if (dev < 0 || dev >= kMaxDevices) {
        *err = fail(TS_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) {
            *err = cuda_fail(e, "cudaGetSymbolAddress(status word)");
            return nullptr;
        }
        g_status_ptr[dev] = static_cast<unsigned long long *>(p);
    }
    *err = TS_OK;
    return g_status_ptr[dev];
}

}  // namespace ts

extern "C" {

const char *ts_status_string(ts_status s) {
    switch (s) {
        case TS_OK: return "TS_OK";
        case TS_ERR_INVALID_ARG: return "TS_ERR_INVALID_ARG";
        case TS_ERR_UNSUPPORTED: return "TS_ERR_UNSUPPORTED";
        case TS_ERR_CUDA: return "TS_ERR_CUDA";
        case TS_ERR_TIMEOUT: return "TS_ERR_TIMEOUT";
    }
    return "TS_ERR_UNKNOWN";
}

const char *ts_last_error_detail(void) { return ts::t_detail.c_str(); }

int32_t ts_num_sms(void) { return ts::device_sms(ts::current_device()); }

ts_status ts_sync_and_check(void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return ts::cuda_fail(e, "cudaStreamSynchronize");
    ts_status st;
    unsigned long long *dev = ts::device_status_word(&st);
    if (!dev) return st;
    unsigned long long h[ts::kStatusWords] = {0, 0, 0, 0};
    e = cudaMemcpy(h, dev, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return ts::cuda_fail(e, "reading the status word");
    if (h[0] == 0) return TS_OK;
    const unsigned long long zero[ts::kStatusWords] = {0, 0, 0, 0};
    e = cudaMemcpy(dev, zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return ts::cuda_fail(e, "clearing the status word");
    if (h[0] == 2)
        return ts::fail(TS_ERR_INVALID_ARG,
                        "row %llu of the jagged copy has bounds outside [0, n] or decreasing; %llu rows not copied",
                        h[1], h[2]);
    if (h[0] == 3)
        return ts::fail(TS_ERR_INVALID_ARG,
                        "row %llu of the chunked copy has pieces past the launch's work tiles (overlapping rows "
                        "need a larger tiles); %llu rows not fully copied",
                        h[1], h[2]);
    const int where = static_cast<int>(h[1] >> 32);
    const unsigned block = static_cast<unsigned>(h[1] & 0xffffffffu);
    return ts::fail(TS_ERR_TIMEOUT, "barrier wait timed out (%s) in block %u; %llu errors recorded",
                    ts::wait_name(where), block, h[2]);
}

}  // extern "C"
