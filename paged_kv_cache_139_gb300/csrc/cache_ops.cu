// The slot-mapped KV write and the copy-on-write block copy.
//
// "vLLM & PagedAttention: Efficient Memory Management for LLM Serving", §X:
//   fused reshape + block write -- new keys/values are split into blocks,
//   put in the cache layout and written at their block-table positions in
//   one launch; fused block copy -- the copy-on-write copies of scattered
//   blocks are batched into one launch instead of many small copies.
//
// Both kernels are bandwidth-bound copies of 16-byte vectors.
#include "pkv_host.cuh"

namespace pkv {
namespace {

// One thread per 16-byte chunk of a (token, kv head) row of K (and V).
// key/value: [T][Hkv][d], cache: [NB][Hkv][B][d]; chunks = d / 8.
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *__restrict__ key_cache,
    uint4 *__restrict__ value_cache, const int64_t *__restrict__ slots, int num_tokens, int num_kv_heads,
    int chunks, int log2_block, int64_t num_slots, DeviceStatus *st) {
    pdl_trigger();
    pdl_wait();
    const int64_t per_token = (int64_t)num_kv_heads * chunks;
    const int64_t total = (int64_t)num_tokens * per_token;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t t = i / per_token;
        const int64_t r = i - t * per_token;
        const int64_t h = r / chunks;
        const int64_t c = r - h * chunks;
        const int64_t s = slots[t];
        if (s < 0) continue;                           // padding token
        if (s >= num_slots) {
            if (r == 0) latch(st, kFlagBadSlot, s);
            continue;
        }
        const int64_t blk = s >> log2_block;
        const int64_t off = s & ((1ll << log2_block) - 1);
        const int64_t dst = (((blk * num_kv_heads + h) << log2_block) + off) * chunks + c;
        const uint4 k = key[i];
        const uint4 v = value[i];
        key_cache[dst] = k;
        value_cache[dst] = v;
    }
}

// Grid (chunks of a block, pairs).  Each CTA copies a contiguous stretch of
// one block with four 16-byte loads in flight per thread.
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    uint4 *__restrict__ cache, const int32_t *__restrict__ pairs, int64_t vecs_per_block,
    int64_t vecs_per_cta, int num_blocks, DeviceStatus *st) {
    pdl_trigger();
    pdl_wait();
    const int p = blockIdx.y;
    const int32_t src = pairs[2 * p];
    const int32_t dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            latch(st, kFlagBadPair, (src < 0 || src >= num_blocks) ? src : dst);
        return;
    }
    const uint4 *s = cache + (int64_t)src * vecs_per_block;
    uint4 *d = cache + (int64_t)dst * vecs_per_block;
    const int64_t begin = (int64_t)blockIdx.x * vecs_per_cta;
    const int64_t end = min(begin + vecs_per_cta, vecs_per_block);
    for (int64_t i = begin + threadIdx.x; i < end; i += (int64_t)kCopyThreads * kCopyUnroll) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const int64_t j = i + (int64_t)u * kCopyThreads;
            if (j < end) v[u] = s[j];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; u++) {
            const int64_t j = i + (int64_t)u * kCopyThreads;
            if (j < end) d[j] = v[u];
        }
    }
}

// Block copies between two pools (swapping): pair p copies block pairs[p][0]
// of src to block pairs[p][1] of dst.  Either pool (and the pairs) may be in
// host memory the GPU can address (pinned), reached over the CPU-GPU link: one
// launch moves every block, however small.  CTAs (x: a share of a block, y: a
// pair, looping over pairs past gridDim.y).
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(
    uint4 *__restrict__ dst, const uint4 *__restrict__ src, const int32_t *__restrict__ pairs, int num_pairs,
    int64_t vecs_per_block, int64_t vecs_per_cta, int src_blocks, int dst_blocks, DeviceStatus *st) {
    pdl_trigger();
    pdl_wait();
    for (int p = blockIdx.y; p < num_pairs; p += gridDim.y) {
        const int32_t sb = pairs[2 * p];
        const int32_t db = pairs[2 * p + 1];
        if (sb < 0 || sb >= src_blocks || db < 0 || db >= dst_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) latch(st, kFlagBadPair, (sb < 0 || sb >= src_blocks) ? sb : db);
            continue;
        }
        const uint4 *s = src + (int64_t)sb * vecs_per_block;
        uint4 *d = dst + (int64_t)db * vecs_per_block;
        const int64_t begin = (int64_t)blockIdx.x * vecs_per_cta;
        const int64_t end = min(begin + vecs_per_cta, vecs_per_block);
        for (int64_t i = begin + threadIdx.x; i < end; i += (int64_t)kCopyThreads * kCopyUnroll) {
            uint4 v[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; u++) {
                const int64_t j = i + (int64_t)u * kCopyThreads;
                if (j < end) v[u] = s[j];
            }
#pragma unroll
            for (int u = 0; u < kCopyUnroll; u++) {
                const int64_t j = i + (int64_t)u * kCopyThreads;
                if (j < end) d[j] = v[u];
            }
        }
    }
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status kv_reshape_and_cache(const void *key, const void *value, void *key_cache, void *value_cache,
                                const int64_t *slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, pkv_dtype dtype, struct CUstream_st *stream) {
    using namespace pkv;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_EINVAL, "kv_reshape_and_cache: bad dtype %d", (int)dtype);
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || head_dim % 8 || !is_pow2(block_size) ||
        num_blocks < 0)
        return fail(PKV_EINVAL,
                    "kv_reshape_and_cache: bad sizes (tokens %d, kv heads %d, head_dim %d, block %d, blocks %d)",
                    num_tokens, num_kv_heads, head_dim, block_size, num_blocks);
    if (num_tokens == 0) return PKV_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping)
        return fail(PKV_EINVAL, "kv_reshape_and_cache: NULL pointer");
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
        return fail(PKV_EINVAL, "kv_reshape_and_cache: pointers must be 16-byte aligned");
    DeviceStatus *st = status_ptr();
    if (!st) return fail(PKV_ECUDA, "kv_reshape_and_cache: no device status word");
    const int chunks = head_dim / 8;
    const int64_t total = (int64_t)num_tokens * num_kv_heads * chunks;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    cudaError_t e = launch(reshape_and_cache_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                           (const uint4 *)key, (const uint4 *)value, (uint4 *)key_cache, (uint4 *)value_cache,
                           slot_mapping, num_tokens, num_kv_heads, chunks, ilog2(block_size),
                           (int64_t)num_blocks * block_size, st);
    if (e != cudaSuccess) return fail(PKV_ECUDA, "kv_reshape_and_cache: launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

pkv_status copy_blocks(void *cache, const int32_t *pairs, int num_pairs, int64_t block_bytes, int num_blocks,
                       struct CUstream_st *stream) {
    using namespace pkv;
    if (num_pairs < 0 || block_bytes <= 0 || block_bytes % 16 || num_blocks < 0 || num_pairs > 65535)
        return fail(PKV_EINVAL, "copy_blocks: bad sizes (pairs %d, block bytes %lld, blocks %d)", num_pairs,
                    (long long)block_bytes, num_blocks);
    if (num_pairs == 0) return PKV_OK;
    if (!cache || !pairs) return fail(PKV_EINVAL, "copy_blocks: NULL pointer");
    if (!aligned16(cache)) return fail(PKV_EINVAL, "copy_blocks: cache must be 16-byte aligned");
    DeviceStatus *st = status_ptr();
    if (!st) return fail(PKV_ECUDA, "copy_blocks: no device status word");
    const int64_t vecs = block_bytes / 16;
    // Enough CTAs per pair that the whole copy spans several waves of the GPU.
    const int64_t per_iter = (int64_t)kCopyThreads * kCopyUnroll;
    int64_t ctas_per_pair = (vecs + per_iter - 1) / per_iter;
    const int64_t want = (int64_t)sm_count() * 8;
    if (ctas_per_pair * num_pairs > want) {
        ctas_per_pair = (want + num_pairs - 1) / num_pairs;
        if (ctas_per_pair < 1) ctas_per_pair = 1;
    }
    const int64_t vecs_per_cta = (vecs + ctas_per_pair - 1) / ctas_per_pair;
    ctas_per_pair = (vecs + vecs_per_cta - 1) / vecs_per_cta;
    cudaError_t e = launch(copy_blocks_kernel, dim3((unsigned)ctas_per_pair, (unsigned)num_pairs), dim3(kCopyThreads),
                           0, stream, (uint4 *)cache, pairs, vecs, vecs_per_cta, num_blocks, st);
    if (e != cudaSuccess) return fail(PKV_ECUDA, "copy_blocks: launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

pkv_status swap_blocks(void *dst_pool, const void *src_pool, const int32_t *pairs, int num_pairs,
                       int64_t block_bytes, int src_blocks, int dst_blocks, struct CUstream_st *stream) {
    using namespace pkv;
    if (num_pairs < 0 || block_bytes <= 0 || block_bytes % 16 || src_blocks < 0 || dst_blocks < 0)
        return fail(PKV_EINVAL, "swap_blocks: bad sizes (pairs %d, block bytes %lld, blocks %d / %d)", num_pairs,
                    (long long)block_bytes, src_blocks, dst_blocks);
    if (num_pairs == 0) return PKV_OK;
    if (!dst_pool || !src_pool || !pairs) return fail(PKV_EINVAL, "swap_blocks: NULL pointer");
    if (dst_pool == src_pool) return fail(PKV_EINVAL, "swap_blocks: source and destination pool are the same (copy_blocks)");
    if (!aligned16(dst_pool) || !aligned16(src_pool)) return fail(PKV_EINVAL, "swap_blocks: pools must be 16-byte aligned");
    DeviceStatus *st = status_ptr();
    if (!st) return fail(PKV_ECUDA, "swap_blocks: no device status word");
    const int64_t vecs = block_bytes / 16;
    const int64_t per_iter = (int64_t)kCopyThreads * kCopyUnroll;
    // enough CTAs that every SM has several in flight; small blocks take one CTA each
    int64_t ctas_per_pair = (vecs + per_iter - 1) / per_iter;
    const int64_t want = (int64_t)sm_count() * 8;
    if (ctas_per_pair * num_pairs > want) {
        ctas_per_pair = (want + num_pairs - 1) / num_pairs;
        if (ctas_per_pair < 1) ctas_per_pair = 1;
    }
    const int64_t vecs_per_cta = (vecs + ctas_per_pair - 1) / ctas_per_pair;
    ctas_per_pair = (vecs + vecs_per_cta - 1) / vecs_per_cta;
    const unsigned gy = (unsigned)(num_pairs < 65535 ? num_pairs : 65535);
    cudaError_t e = launch(swap_blocks_kernel, dim3((unsigned)ctas_per_pair, gy), dim3(kCopyThreads), 0, stream,
                           (uint4 *)dst_pool, (const uint4 *)src_pool, pairs, num_pairs, vecs, vecs_per_cta, src_blocks,
                           dst_blocks, st);
    if (e != cudaSuccess) return fail(PKV_ECUDA, "swap_blocks: launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}

}  // extern "C"
