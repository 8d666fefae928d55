// paged_attention_decode for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at the point where they run the
// attention: a plugin invoked by a host framework while that framework is
// capturing a CUDA graph or running a latency-critical execution callback
// (an allocation there synchronises the device or is refused outright), or a
// service that fixes its whole device-memory budget at start-up and may not
// grow it later.  This entry point needs no workspace from them: the
// partition partials live in a fixed-size array in the library's own device
// memory, reserved on every GPU that loads the library until the process
// exits.
//
// The kernels are the ones paged_attention_decode launches; only the origin
// of the scratch differs.
#include <climits>
#include <mutex>

#include "pkv_host.cuh"

namespace {

// Upper bound on the partials one call may need (m, l and o for every
// sequence, head and partition).  16 MiB covers, for example, 8 sequences x
// 32 heads x 64 partitions of 512 tokens at head_dim 128 (8.5 MB).
constexpr size_t kScratchBytes = 16u << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Prepared {
    void *addr;            // device address of g_scratch (null until the first call)
    unsigned int epoch;    // pkv::timeout_epoch() when the counters were last prepared
};
Prepared g_prepared[kMaxDevices] = {};

// Device address of g_scratch on the current device, with its counters
// ready.  In host code the name g_scratch is only a host-side stand-in for
// the symbol, never a device address, so the address is looked up once per
// device and cached.  The counters are prepared on the first call and again
// after pkv_check has reported a device-wait timeout (a kernel that gave up
// may have left them mid-count): one zeroing kernel on `stream`, waited for
// before the address is handed out, so that a later call on any stream finds
// the array ready.  That preparation cannot be recorded into a CUDA graph, so
// it is refused while `stream` is capturing.
void *scratch_address(cudaStream_t stream, pkv_status *st) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *st = pkv::fail(PKV_ECUDA, "paged_attention_decode_noalloc: no current device (%s)",
                        cudaGetErrorString(e));
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    Prepared &pr = g_prepared[dev];
    const unsigned int epoch = pkv::timeout_epoch();
    if (pr.addr && pr.epoch == epoch) return pr.addr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) {
        *st = pkv::fail(PKV_ECUDA, "paged_attention_decode_noalloc: stream capture status: %s", cudaGetErrorString(e));
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone) {
        *st = pkv::fail(PKV_EINVAL,
                        "paged_attention_decode_noalloc: the built-in scratch of device %d must be prepared outside "
                        "stream capture (make the first call on a device, and the first after pkv_check reported "
                        "PKV_ETIMEOUT, before capturing)",
                        dev);
        return nullptr;
    }
    void *p = pr.addr;
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p) {
            *st = pkv::fail(PKV_ECUDA, "paged_attention_decode_noalloc: scratch address on device %d: %s", dev,
                            cudaGetErrorString(e));
            return nullptr;
        }
    }
    const pkv_status ist = paged_attention_workspace_init(p, kScratchBytes, stream);
    if (ist != PKV_OK) {
        *st = ist;
        return nullptr;
    }
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) {
        *st = pkv::fail(PKV_ECUDA, "paged_attention_decode_noalloc: preparing the scratch: %s", cudaGetErrorString(e));
        return nullptr;
    }
    pr.addr = p;
    pr.epoch = epoch;
    return p;
}

}  // namespace

extern "C" pkv_status paged_attention_decode_noalloc(
    void *out, const void *query, const void *key_cache, const void *value_cache, const int32_t *block_tables,
    const int32_t *context_lens, int num_seqs, int max_blocks_per_seq, int max_context_len, int block_size,
    int num_blocks, int num_heads, int num_kv_heads, int head_dim, float scale, int partition_size,
    pkv_dtype dtype, struct CUstream_st *stream) {
    // The same context bound paged_attention_decode uses, to size the partials.
    long long bound = max_context_len > 0 ? (long long)max_context_len
                                          : (long long)max_blocks_per_seq * (long long)block_size;
    if (bound > INT_MAX) bound = INT_MAX;
    const size_t need = paged_attention_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, (int)bound,
                                                       partition_size < 0 ? 0 : partition_size);
    if (need > kScratchBytes)
        return pkv::fail(PKV_EINVAL,
                         "paged_attention_decode_noalloc: these sizes need %zu bytes of partition scratch; the "
                         "built-in scratch holds %zu (use paged_attention_decode with a caller workspace)",
                         need, kScratchBytes);
    pkv_status st = PKV_OK;
    void *ws = scratch_address(stream, &st);
    if (!ws) return st;
    return paged_attention_decode(out, query, key_cache, value_cache, block_tables, context_lens, num_seqs,
                                  max_blocks_per_seq, max_context_len, block_size, num_blocks, num_heads,
                                  num_kv_heads, head_dim, scale, partition_size, ws, kScratchBytes, dtype, stream);
}
