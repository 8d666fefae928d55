// Prompt-phase (prefill) paged attention on the fifth-generation tensor cores.
//
// What it computes ("vLLM & PagedAttention: Efficient Memory Management for
// LLM Serving", §I attention equation with its causal sum over t <= i, §II and
// §V for the prompt phase, §VII for a shared prefix whose blocks are already
// cached): sequence s has n_s new tokens, the last n_s of its context_lens[s]
// tokens, whose keys and values are already in the paged cache.  New token j
// (position p = context_lens[s] - n_s + j) and query head h give
//     out = sum_{t <= p} softmax_t(scale * q . k_t) v_t,
// key t of sequence s read from physical block block_tables[s][t / B] at
// offset t % B, kv head h / (H / Hkv).  With n_s = context_lens[s] this is a
// plain prompt; with fewer new tokens the first tokens are a cached prefix.
//
// How (sm_103a):
//   * One CTA per (128 new tokens, query head, sequence): the tokens' queries
//     are the 128 rows (M) of both products.  The grid walks a sequence's
//     tiles from the last (the most keys) to the first.
//   * A producer warp loads the query tile (tiled TMA over the query tensor)
//     and then, for each 128-key tile, the tile's K and V blocks (tiled TMA
//     over the cache, one box of B tokens x 64 elements per block and
//     64-element panel of d) into a two-stage ring.  Boxes land 128-byte
//     swizzled, the layout the MMA descriptors describe.
//   * One thread of the MMA warp issues tcgen05.mma: S = Q K^T (M 128, N 128,
//     fp32 in TMEM) one tile ahead, then O += P V (N 64 per panel of d, V
//     read MN-major straight from the cache layout), each group committed to
//     an mbarrier.
//   * Four softmax warps (one thread per row) read S from TMEM, mask keys
//     after the row's position, keep a running max and sum in fp32 (log2
//     domain; the reference max moves only when it grows by more than 8, so
//     probabilities stay below 2^8), write P as 16-bit to shared memory (for
//     bf16 as a rounded part and its remainder) and rescale O in TMEM when a
//     row's reference moved.  At the end they divide
//     by the sum and store the rows.
//   * All waits are bounded; a wait that gives up latches a timeout, the CTA
//     drains its copies and MMAs and frees its TMEM.
#include <cfloat>
#include <climits>
#include <cstring>
#include <type_traits>

#include "pkv_host.cuh"
#include "pkv_tcgen05.cuh"
#include "pkv_tmap.h"

namespace pkv {
namespace {

constexpr int kRows = 128;               // query rows per CTA
constexpr int kKeys = 128;               // keys per KV tile
constexpr int kStages = 2;               // K/V ring depth
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kPanelBytes = 128 * 128;   // 128 rows x 64 16-bit elements
constexpr uint32_t kTmemCols = 256;           // S: 128 columns, O: up to 128
constexpr float kRescaleLog2 = 8.f;           // reference max moves past this growth

struct PrefillArgs {
    void *out;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start;
    DeviceStatus *status;
    int num_seqs, num_tokens, max_blocks, log2_block, num_blocks;
    int num_heads, group;
    float scale_log2;                    // scale * log2(e)
};

// bf16 probabilities carry 8 significant bits: a row over a handful of keys
// would see their rounding in its output.  For bf16 the kernel therefore
// writes P = P_hi + P_lo (both bf16, P_lo the rounding remainder, together 16
// significant bits) and accumulates both products; fp16 (11 bits) needs one.
template <int D, bool SPLIT> struct PfLayout {
    static constexpr int NP = D / 64;                              // panels of d
    static constexpr int NPP = SPLIT ? 2 : 1;                       // P parts
    static constexpr uint32_t q = 0;                                // NP panels
    static constexpr uint32_t p = q + NP * kPanelBytes;             // NPP x 2 panels of keys
    static constexpr uint32_t k = p + NPP * 2 * kPanelBytes;        // kStages x NP panels
    static constexpr uint32_t v = k + kStages * NP * kPanelBytes;
    static constexpr uint32_t bars = v + kStages * NP * kPanelBytes;
    static constexpr uint32_t bytes = bars + 256;
    static constexpr size_t alloc = bytes + 1024;                   // room to align the base
};

// barrier slots
enum : int { bQFull = 0, bKFull = 1, bVFull = 3, bKEmpty = 5, bVEmpty = 7, bSFull = 9, bSFree = 10,
             bPFull = 11, bODone = 12, bDrain = 13, kNumBars = 14 };

__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, long long limit) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit));
}

template <typename T> __device__ __forceinline__ uint32_t pack16(float x, float y);
template <> __device__ __forceinline__ uint32_t pack16<__half>(float x, float y) {
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack16<__nv_bfloat16>(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tmq,
                         const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    using L = PfLayout<D, kBf16>;
    constexpr int NP = L::NP;
    extern __shared__ uint8_t smem_pf[];
    uint8_t *sm = smem_pf + ((1024u - (smem_u32(smem_pf) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = (int)gridDim.x - 1 - (int)blockIdx.x;
    const int h = blockIdx.y, s = blockIdx.z;

    pdl_wait();
    DeviceStatus *st = a.status;
    if (timed_out(st)) return;
    const int q_begin = a.query_start[s], q_end = a.query_start[s + 1], ctx = a.context_lens[s];
    const int n = q_end - q_begin;
    const int B = 1 << a.log2_block;
    const int t0 = tile * kRows;
    if (n < 0 || q_begin < 0 || q_end > a.num_tokens || n > ctx || ctx > a.max_blocks * B) {
        if (tid == 0 && tile == 0 && h == 0) latch(st, kFlagBadContext, s);
        return;
    }
    if (t0 >= n) return;                       // this sequence has fewer tiles
    const int rows = min(kRows, n - t0);
    const int pos0 = ctx - n + t0;             // position of row 0
    const int pos_last = pos0 + rows - 1;
    const int nkv = pos_last / kKeys + 1;      // key tiles this CTA reads
    const int g = h / a.group;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    if (tid == 0) {
        mbar_init(&bars[bQFull], 1);
        for (int i = 0; i < kStages; i++) {
            mbar_init(&bars[bKFull + i], 1);
            mbar_init(&bars[bVFull + i], 1);
            mbar_init(&bars[bKEmpty + i], 1);
            mbar_init(&bars[bVEmpty + i], 1);
        }
        mbar_init(&bars[bSFull], 1);
        mbar_init(&bars[bSFree], kSoftmaxWarps * 32);
        mbar_init(&bars[bPFull], kSoftmaxWarps * 32);
        mbar_init(&bars[bODone], 1);
        mbar_init(&bars[bDrain], 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(tslot, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem, tO = tmem + kKeys;

    if (warp == kProducerWarp) {
        // ---------------- producer: Q once, then K and V per key tile ----------------
        const uint64_t pol_q = policy_evict_first();
        const uint64_t pol_kv = policy_evict_last();   // read again by the sequence's other tiles and heads
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[bQFull], NP * kPanelBytes);
            for (int p = 0; p < NP; p++)
                tma_load_3d(sm + L::q + p * kPanelBytes, &tmq, 64 * p, h, q_begin + t0, &bars[bQFull], pol_q);
        }
        const int32_t *row = a.block_tables + (size_t)s * a.max_blocks;
        const int nblk_used = (ctx + B - 1) >> a.log2_block;
        const int bpt = kKeys >> a.log2_block;          // blocks per key tile (B <= 128)
        int j = 0;
        for (; j < nkv; j++) {
            const int stg = j & 1;
            const int nb = min(bpt, nblk_used - j * bpt);
            const uint32_t bytes = (uint32_t)nb * (uint32_t)B * 128u * NP;
            for (int which = 0; which < 2; which++) {       // K, then V
                if (j >= kStages) {
                    ok = wait_warp(&bars[(which ? bVEmpty : bKEmpty) + stg], ((j >> 1) - 1) & 1, kWaitLimitCycles);
                    if (!ok) break;
                }
                uint64_t *full = &bars[(which ? bVFull : bKFull) + stg];
                if (lane == 0) mbar_arrive_expect_tx(full, bytes);
                __syncwarp();
                uint8_t *dst = sm + (which ? L::v : L::k) + (uint32_t)stg * NP * kPanelBytes;
                for (int b = lane; b < nb; b += 32) {
                    int phys = row[j * bpt + b];
                    if (phys < 0 || phys >= a.num_blocks) {
                        latch(st, kFlagBadBlock, phys);
                        phys = 0;                           // keep the byte count; the output is flagged
                    }
                    for (int p = 0; p < NP; p++)
                        tma_load_4d(dst + p * kPanelBytes + (uint32_t)b * B * 128u, which ? &tmv : &tmk, 64 * p, 0, g,
                                    phys, full, pol_kv);
                }
            }
            if (!ok) break;
        }
        if (!ok) {
            if (lane == 0) latch(st, kFlagTimeout, j);
            // copies already issued must land before the CTA's memory is reused
            for (int jj = max(0, j - kStages); jj <= min(j, nkv - 1); jj++) {
                mbar_wait(&bars[bKFull + (jj & 1)], (jj >> 1) & 1, kDrainLimitCycles);
                mbar_wait(&bars[bVFull + (jj & 1)], (jj >> 1) & 1, kDrainLimitCycles);
            }
            mbar_wait(&bars[bQFull], 0, kDrainLimitCycles);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            const uint32_t id_s = tc::idesc_f16(kRows, kKeys, kBf16, false);
            const uint32_t id_o = tc::idesc_f16(kRows, 64, kBf16, true);
            const uint32_t q_base = smem_u32(sm + L::q), p_base = smem_u32(sm + L::p);
            auto issue_s = [&](int stg) {
                const uint32_t k_base = smem_u32(sm + L::k) + (uint32_t)stg * NP * kPanelBytes;
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    const uint32_t off = (k / 4) * kPanelBytes + (k % 4) * 32;
                    tc::mma_f16_ss(tS, tc::smem_desc_sw128(q_base + off, 1024, 1024),
                                   tc::smem_desc_sw128(k_base + off, 1024, 1024), id_s, k > 0);
                }
            };
            auto issue_o = [&](int stg, bool acc) {
                const uint32_t v_base = smem_u32(sm + L::v) + (uint32_t)stg * NP * kPanelBytes;
#pragma unroll
                for (int part = 0; part < L::NPP; part++)
#pragma unroll
                    for (int k = 0; k < kKeys / 16; k++) {
                        const uint32_t aoff = part * 2 * kPanelBytes + (k / 4) * kPanelBytes + (k % 4) * 32;
#pragma unroll
                        for (int p = 0; p < NP; p++)
                            tc::mma_f16_ss(tO + 64 * p, tc::smem_desc_sw128(p_base + aoff, 1024, 1024),
                                           tc::smem_desc_sw128(v_base + p * kPanelBytes + k * 2048, 1024, 1024),
                                           id_o, (acc || part > 0 || k > 0) ? 1u : 0u);
                    }
            };
            bool ok = mbar_wait(&bars[bQFull], 0, kWaitLimitCycles) && mbar_wait(&bars[bKFull], 0, kWaitLimitCycles);
            int j = 0;
            if (ok) {
                tc::fence_after();
                issue_s(0);
                tc::mma_commit(&bars[bKEmpty]);
                tc::mma_commit(&bars[bSFull]);
                for (; j < nkv; j++) {
                    if (j + 1 < nkv) {
                        const int s1 = (j + 1) & 1;
                        ok = mbar_wait(&bars[bKFull + s1], ((j + 1) >> 1) & 1, kWaitLimitCycles) &&
                             mbar_wait(&bars[bSFree], j & 1, kWaitLimitCycles);
                        if (!ok) break;
                        tc::fence_after();
                        issue_s(s1);
                        tc::mma_commit(&bars[bKEmpty + s1]);
                        tc::mma_commit(&bars[bSFull]);
                    }
                    ok = mbar_wait(&bars[bVFull + (j & 1)], (j >> 1) & 1, kWaitLimitCycles) &&
                         mbar_wait(&bars[bPFull], j & 1, kWaitLimitCycles);
                    if (!ok) break;
                    tc::fence_after();
                    issue_o(j & 1, j > 0);
                    tc::mma_commit(&bars[bVEmpty + (j & 1)]);
                    tc::mma_commit(&bars[bODone]);
                }
            }
            if (!ok) {
                latch(st, kFlagTimeout, 1000000 + j);
                // every MMA issued so far completes before TMEM is freed
                tc::mma_commit(&bars[bDrain]);
                mbar_wait(&bars[bDrain], 0, kDrainLimitCycles);
            }
        }
        __syncwarp();
    } else {
        // ---------------- softmax: one thread per query row ----------------
        const int r = tid;                                   // 0..127, TMEM lane r
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        const int my_pos = r < rows ? pos0 + r : pos_last;   // last key this row may see
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        int j = 0;
        for (; j < nkv; j++) {
            ok = wait_warp(&bars[bSFull], j & 1, kWaitLimitCycles);
            if (!ok) break;
            tc::fence_after();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; c++) tc::tmem_ld32(tS + lane_off + 32 * c, sr[c]);
#pragma unroll
            for (int c = 0; c < 4; c++) tc::tmem_wait_ld(sr[c]);
            tc::fence_before();
            mbar_arrive(&bars[bSFree]);                      // S may be overwritten by the next tile

            const int lim = my_pos - j * kKeys;              // keys 0..lim of this tile are visible
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; c++)
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    float x = __uint_as_float(sr[c][i]) * a.scale_log2;
                    x = (32 * c + i <= lim) ? x : -INFINITY;
                    sr[c][i] = __float_as_uint(x);
                    mx = fmaxf(mx, x);
                }
            const bool moved = mx > m_run + kRescaleLog2;
            const float m_new = moved ? mx : m_run;
            const float alpha = exp2f(m_run - m_new);        // 0 on the first tile, 1 when not moved
            m_run = m_new;
            float lsum = 0.f;
#pragma unroll
            for (int c = 0; c < 4; c++)
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const float pv = exp2f(__uint_as_float(sr[c][i]) - m_run);
                    lsum += pv;
                    sr[c][i] = __float_as_uint(pv);              // the score register now holds p
                }
            l_run = l_run * alpha + lsum;

            if (j > 0) {                                     // PV of the previous tile: O stable, P free
                ok = wait_warp(&bars[bODone], (j - 1) & 1, kWaitLimitCycles);
                if (!ok) break;
                tc::fence_after();
                if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                    for (int c = 0; c < D / 32; c++) {
                        uint32_t o[32];
                        tc::tmem_ld32(tO + lane_off + 32 * c, o);
                        tc::tmem_wait_ld(o);
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc::tmem_st32(tO + lane_off + 32 * c, o);
                    }
                    tc::tmem_wait_st();
                }
            }
            const int kbase = j * kKeys;
            if (j == nkv - 1 && kbase + kKeys > ctx) {
                // rows past the end of the context hold other data: P is 0 there, but 0 x NaN is not
                ok = wait_warp(&bars[bVFull + (j & 1)], (j >> 1) & 1, kWaitLimitCycles);
                if (!ok) break;
                const int first = ctx - kbase;
                uint8_t *vs = sm + L::v + (uint32_t)(j & 1) * NP * kPanelBytes;
                const int nvec = (kKeys - first) * 8;        // 16-byte vectors per panel
                for (int i = tid; i < nvec * NP; i += kSoftmaxWarps * 32) {
                    const int p = i / nvec, rem = i % nvec;
                    *reinterpret_cast<uint4 *>(vs + p * kPanelBytes + (first + rem / 8) * 128 + (rem % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            uint8_t *ps = sm + L::p;
#pragma unroll
            for (int q = 0; q < 16; q++) {
                const int panel = q >> 3, c = q & 7;
                const uint32_t *pv = &sr[q / 4][8 * (q % 4)];
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const float p0 = __uint_as_float(pv[2 * e]), p1 = __uint_as_float(pv[2 * e + 1]);
                    hi[e] = pack16<T>(p0, p1);
                    if (kBf16)   // remainder after rounding (bf16 widens exactly by a shift)
                        lo[e] = pack16<T>(p0 - __uint_as_float(hi[e] << 16), p1 - __uint_as_float(hi[e] & 0xffff0000u));
                }
                const uint32_t off = panel * kPanelBytes + r * 128 + ((c ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(ps + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                if (kBf16)
                    *reinterpret_cast<uint4 *>(ps + 2 * kPanelBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();                        // generic writes -> tensor-core reads
            tc::fence_before();
            mbar_arrive(&bars[bPFull]);
        }
        if (ok) ok = wait_warp(&bars[bODone], (nkv - 1) & 1, kWaitLimitCycles);
        if (ok) {
            tc::fence_after();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            T *orow = reinterpret_cast<T *>(a.out) + ((size_t)(q_begin + t0 + r) * a.num_heads + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; c++) {
                uint32_t o[32];
                tc::tmem_ld32(tO + lane_off + 32 * c, o);
                tc::tmem_wait_ld(o);
                if (r < rows) {
#pragma unroll
                    for (int v = 0; v < 4; v++) {
                        uint4 w;
                        w.x = pack16<T>(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                        w.y = pack16<T>(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                        w.z = pack16<T>(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                        w.w = pack16<T>(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + 32 * c + 8 * v) = w;
                    }
                }
            }
        } else if (lane == 0) {
            latch(st, kFlagTimeout, 2000000 + j);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after();
        tc::tmem_free(tmem, kTmemCols);
    }
}

template <int D, typename T>
cudaError_t launch_prefill(const PrefillArgs &a, const void *query, const void *kc, const void *vc, int Hkv,
                           int max_query_len, cudaStream_t stream) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    using L = PfLayout<D, kBf16>;
    auto kern = paged_prefill_kernel<D, T>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int B = 1 << a.log2_block;
    CUtensorMap tmq, tmk, tmv;
    std::memset(&tmq, 0, sizeof tmq);
    std::memset(&tmk, 0, sizeof tmk);
    std::memset(&tmv, 0, sizeof tmv);
    // query [T][H][D]: box of 64 elements x 1 head x 128 tokens
    const cuuint64_t qdims[3] = {(cuuint64_t)D, (cuuint64_t)a.num_heads, (cuuint64_t)a.num_tokens};
    const cuuint64_t qstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_heads * D * 2};
    const cuuint32_t qbox[3] = {64u, 1u, (cuuint32_t)kRows};
    // cache [NB][Hkv][B][D]: box of 64 elements x B tokens of one (block, kv head)
    const cuuint64_t cdims[4] = {(cuuint64_t)D, (cuuint64_t)B, (cuuint64_t)Hkv, (cuuint64_t)a.num_blocks};
    const cuuint64_t cstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)B * D * 2, (cuuint64_t)Hkv * B * D * 2};
    const cuuint32_t cbox[4] = {64u, (cuuint32_t)B, 1u, 1u};
    if (!encode_tiled16(&tmq, query, 3, qdims, qstr, qbox, kBf16) || !encode_tiled16(&tmk, kc, 4, cdims, cstr, cbox, kBf16) ||
        !encode_tiled16(&tmv, vc, 4, cdims, cstr, cbox, kBf16))
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((max_query_len + kRows - 1) / kRows), (unsigned)a.num_heads, (unsigned)a.num_seqs);
    return launch(kern, grid, dim3(kThreads), L::alloc, stream, a, tmq, tmk, tmv);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_attention_prefill(void *out, const void *query, const void *key_cache,
                                              const void *value_cache, const int32_t *block_tables,
                                              const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                                              int num_tokens, int max_query_len, int max_blocks_per_seq,
                                              int block_size, int num_blocks, int num_heads, int num_kv_heads,
                                              int head_dim, float scale, pkv_dtype dtype, struct CUstream_st *stream) {
    if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0)
        return fail(PKV_EINVAL, "paged_attention_prefill: negative size (num_seqs %d, num_tokens %d, max_query_len %d)",
                    num_seqs, num_tokens, max_query_len);
    if (num_seqs > 65535)
        return fail(PKV_EINVAL, "paged_attention_prefill: num_seqs %d above 65535", num_seqs);
    if (head_dim != 64 && head_dim != 128)
        return fail(PKV_EINVAL, "paged_attention_prefill: head_dim %d not 64 or 128", head_dim);
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
        return fail(PKV_EINVAL, "paged_attention_prefill: num_heads %d not a multiple of num_kv_heads %d", num_heads,
                    num_kv_heads);
    if (!is_pow2(block_size) || block_size < 4 || block_size > 128)
        return fail(PKV_EINVAL, "paged_attention_prefill: block_size %d not a power of two in [4, 128]", block_size);
    if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_EINVAL, "paged_attention_prefill: bad dtype %d", (int)dtype);
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
        return fail(PKV_EINVAL, "paged_attention_prefill: scale not finite");
    if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
    if (max_query_len == 0 || max_query_len > num_tokens) max_query_len = num_tokens;
    if (num_blocks <= 0 || max_blocks_per_seq <= 0)
        return fail(PKV_EINVAL, "paged_attention_prefill: num_blocks %d / max_blocks_per_seq %d not positive",
                    num_blocks, max_blocks_per_seq);
    if ((long long)max_blocks_per_seq * block_size > INT_MAX)
        return fail(PKV_EINVAL, "paged_attention_prefill: table capacity above 2^31 tokens");
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens || !query_start)
        return fail(PKV_EINVAL, "paged_attention_prefill: null pointer");
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
        return fail(PKV_EINVAL, "paged_attention_prefill: out, query and caches must be 16-byte aligned");
    DeviceStatus *st = status_ptr();
    if (!st) return fail(PKV_ECUDA, "paged_attention_prefill: no device status word");
    PrefillArgs a;
    a.out = out;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.status = st;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.max_blocks = max_blocks_per_seq;
    a.log2_block = ilog2(block_size);
    a.num_blocks = num_blocks;
    a.num_heads = num_heads;
    a.group = num_heads / num_kv_heads;
    a.scale_log2 = (float)((double)scale * 1.4426950408889634);
    const bool bf16 = dtype == PKV_BF16;
    cudaError_t e;
    if (head_dim == 128)
        e = bf16 ? launch_prefill<128, __nv_bfloat16>(a, query, key_cache, value_cache, num_kv_heads, max_query_len, stream)
                 : launch_prefill<128, __half>(a, query, key_cache, value_cache, num_kv_heads, max_query_len, stream);
    else
        e = bf16 ? launch_prefill<64, __nv_bfloat16>(a, query, key_cache, value_cache, num_kv_heads, max_query_len, stream)
                 : launch_prefill<64, __half>(a, query, key_cache, value_cache, num_kv_heads, max_query_len, stream);
    if (e != cudaSuccess) return fail(PKV_ECUDA, "paged_attention_prefill: launch: %s", cudaGetErrorString(e));
    return PKV_OK;
}
