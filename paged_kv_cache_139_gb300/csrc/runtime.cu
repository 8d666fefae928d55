// Library runtime: the per-device status word, error reporting, launch
// counting and device properties.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "pkv_host.cuh"

namespace pkv {

// One status word per device that loads the library.
__device__ DeviceStatus g_status;

namespace {

thread_local char t_msg[512] = "no error";
std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceStatus *g_status_addr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
// Device-wait timeouts pkv_check has reported and cleared, per device.
std::atomic<unsigned int> g_timeout_epoch[kMaxDevices];

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return d;
}

// One CTA waits on a barrier that never completes; the bounded wait must
// give up and latch the timeout.
__global__ void wait_timeout_selftest_kernel(long long limit, DeviceStatus *st) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit)) latch(st, kFlagTimeout, limit);
}

}  // namespace

pkv_status fail(pkv_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_msg, sizeof t_msg, fmt, ap);
    va_end(ap);
    return st;
}

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

DeviceStatus *status_ptr() {
    int d = current_device();
    if (d < 0 || d >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_addr[d]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
        g_status_addr[d] = static_cast<DeviceStatus *>(p);
    }
    return g_status_addr[d];
}

unsigned int timeout_epoch() {
    int d = current_device();
    if (d < 0 || d >= kMaxDevices) return 0;
    return g_timeout_epoch[d].load(std::memory_order_acquire);
}

int sm_count() {
    int d = current_device();
    if (d < 0 || d >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
        g_sms[d] = n;
    }
    return g_sms[d];
}

}  // namespace pkv

extern "C" {

const char *pkv_last_error_string(void) { return pkv::t_msg; }

uint64_t pkv_launch_count(void) { return pkv::g_launches.load(std::memory_order_relaxed); }

int pkv_version(void) { return 114; }

pkv_status pkv_check(struct CUstream_st *stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return pkv::fail(PKV_ECUDA, "pkv_check: %s", cudaGetErrorString(e));
    pkv::DeviceStatus h;
    e = cudaMemcpyFromSymbol(&h, pkv::g_status, sizeof h);
    if (e != cudaSuccess) return pkv::fail(PKV_ECUDA, "pkv_check: reading status: %s", cudaGetErrorString(e));
    if (h.flags == 0) return PKV_OK;
    if (h.flags & pkv::kFlagTimeout) {
        // a kernel that gave up may have left work-ticket counters mid-count
        const int d = pkv::current_device();
        if (d >= 0 && d < pkv::kMaxDevices) pkv::g_timeout_epoch[d].fetch_add(1u, std::memory_order_acq_rel);
    }
    pkv::DeviceStatus zero;
    std::memset(&zero, 0, sizeof zero);
    e = cudaMemcpyToSymbol(pkv::g_status, &zero, sizeof zero);
    if (e != cudaSuccess) return pkv::fail(PKV_ECUDA, "pkv_check: clearing status: %s", cudaGetErrorString(e));
    if (h.flags & pkv::kFlagBadWorkspace)
        return pkv::fail(PKV_EINVAL, "device error flags 0x%x: attention workspace not initialised "
                                     "(paged_attention_workspace_init)", h.flags);
    const char *what = (h.first_flag & pkv::kFlagBadSlot)      ? "slot outside the pool"
                       : (h.first_flag & pkv::kFlagBadBlock)   ? "block-table entry outside the pool"
                       : (h.first_flag & pkv::kFlagBadPair)    ? "copy pair outside the pool"
                       : (h.first_flag & pkv::kFlagBadContext) ? "context length outside the table"
                       : (h.first_flag & pkv::kFlagSlotNotLast)
                           ? "decode slot is not position context_len - 1 of its sequence's block table"
                       : (h.first_flag & pkv::kFlagTimeout)    ? "device wait timed out"
                                                               : "unknown";
    pkv_status st = (h.flags & ~pkv::kFlagTimeout) ? PKV_EINDEX : PKV_ETIMEOUT;
    return pkv::fail(st, "device error flags 0x%x; first: %s (value %lld)", h.flags, what, h.first_bad);
}

pkv_status pkv_selftest_wait_timeout(long long limit_cycles, struct CUstream_st *stream) {
    if (limit_cycles <= 0 || limit_cycles > (1ll << 32))
        return pkv::fail(PKV_EINVAL, "pkv_selftest_wait_timeout: limit %lld cycles out of range", limit_cycles);
    pkv::DeviceStatus *st = pkv::status_ptr();
    if (!st) return pkv::fail(PKV_ECUDA, "pkv_selftest_wait_timeout: no device status word");
    cudaError_t e = pkv::launch(pkv::wait_timeout_selftest_kernel, dim3(1), dim3(32), 0, stream, limit_cycles, st);
    if (e != cudaSuccess) return pkv::fail(PKV_ECUDA, "pkv_selftest_wait_timeout: launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

pkv_status pkv_validate_copy_pairs(const int32_t *pairs, int n, int num_blocks) {
    if (n < 0 || num_blocks < 0 || (n > 0 && !pairs))
        return pkv::fail(PKV_EINVAL, "pkv_validate_copy_pairs: bad argument");
    // mark[b]: bit 0 = b is a source, bit 1 = b is a destination
    std::vector<unsigned char> mark((size_t)num_blocks, 0);
    for (int i = 0; i < n; i++) {
        int32_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks)
            return pkv::fail(PKV_EINVAL, "copy pair %d (%d -> %d) outside a pool of %d blocks", i, s, d, num_blocks);
        mark[s] |= 1;
    }
    for (int i = 0; i < n; i++) {
        int32_t d = pairs[2 * i + 1];
        if (mark[d] & 2) return pkv::fail(PKV_EINVAL, "copy pairs: destination %d appears twice", d);
        if (mark[d] & 1) return pkv::fail(PKV_EINVAL, "copy pairs: destination %d is also a source", d);
        mark[d] |= 2;
    }
    return PKV_OK;
}

}  // extern "C"
