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
//   * One CTA per (256 new tokens, query head, sequence): two query tiles of
//     128 rows (M of both products) that take turns on the tensor core.  The
//     grid walks a sequence's tiles from the last (the most keys) to the first.
//   * A producer warp loads the query tiles (tiled TMA over the query tensor)
//     and then, for each 128-key tile, the tile's K and V blocks (tiled TMA
//     over the cache, one box of B tokens x 64 elements per block and
//     64-element panel of d) into a two-stage ring.  Boxes land 128-byte
//     swizzled, the layout the MMA descriptors describe.
//   * One thread of the MMA warp issues tcgen05.mma: S = Q K^T (M 128, N 128,
//     fp32 in TMEM), then O += P V with P read from TMEM and V read MN-major
//     straight from the cache layout (N = d: one product per 16 keys).  While one tile's
//     softmax runs, the tensor core computes the other tile's products.
//   * Four softmax warps per tile (one thread per row) read S from TMEM, mask
//     keys after the row's position, keep a running max and sum in fp32 (log2
//     domain; the reference max moves only when it grows by more than 8, so
//     probabilities stay below 2^8), write P as 16-bit over the scores in
//     TMEM (for bf16 as a rounded part and its remainder) and rescale O in
//     TMEM when a row's reference moved.  At the end they divide by the sum
//     and store the rows.
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

constexpr int kRows = 128;               // query rows per tile (M of both products)
constexpr int kTiles = 2;                // query tiles per CTA, alternating on the tensor core
constexpr int kKeys = 128;               // keys per KV tile
constexpr int kStages = 2;               // K/V ring depth
constexpr int kSoftmaxWarps = 4;         // per query tile
constexpr int kProducerWarp = kTiles * kSoftmaxWarps;
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr uint32_t kPanelBytes = 128 * 128;   // 128 rows x 64 16-bit elements
constexpr uint32_t kTmemCols = 512;           // per tile: S/P 128 columns, O 128
constexpr uint32_t kTileCols = 256;
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

// Shared memory: the two query tiles and the K/V ring.  P stays in TMEM,
// over the tile's S columns.  The allocation is padded to keep one CTA per
// SM (each CTA takes all 512 TMEM columns).
template <int D> struct PfLayout {
    static constexpr int NP = D / 64;                              // panels of d
    static constexpr uint32_t q = 0;                                // kTiles x NP panels
    static constexpr uint32_t k = q + kTiles * NP * kPanelBytes;    // kStages x NP panels
    static constexpr uint32_t v = k + kStages * NP * kPanelBytes;
    static constexpr uint32_t bars = v + kStages * NP * kPanelBytes;
    static constexpr uint32_t bytes = bars + 256;
    static constexpr size_t alloc = (bytes + 1024 > 120u * 1024u) ? bytes + 1024 : 120u * 1024u;
};

// barrier slots
enum : int { bQFull = 0, bKFull = 1, bVFull = 3, bKEmpty = 5, bVEmpty = 7, bSFull = 9, bPFull = 11, bODone = 13,
             bDrain = 15, kNumBars = 16 };

// 2^x by the hardware approximation (MUFU); 2^-inf = 0.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max(a, b, c) in one instruction (three-input form, sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float m;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
    return m;
}

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

// Probabilities in TMEM.  Chunk c (keys 32c .. 32c+31) of the row is written
// over its own score columns: 16 columns of packed 16-bit p (two keys per
// column, the even key in the lower half) at 32c, and for bf16 16 columns of
// the rounding remainder at 32c + 16.  The product's A operand for keys
// 16t .. 16t+15 is then 8 columns at 32 (t / 2) + 8 (t % 2) (+ 16 for the
// remainder).
//
// bf16 probabilities carry 8 significant bits: a row over a handful of keys
// would see their rounding in its output, so for bf16 P = P_hi + P_lo (both
// bf16, together 16 significant bits) and both products are accumulated;
// fp16 (11 bits) needs one.
__device__ __forceinline__ uint32_t p_col(int t, bool lo) { return 32 * (t >> 1) + 8 * (t & 1) + (lo ? 16 : 0); }

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    paged_prefill_kernel(const PrefillArgs a, const __grid_constant__ CUtensorMap tmq,
                         const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    using L = PfLayout<D>;
    constexpr int NP = L::NP;
    extern __shared__ uint8_t smem_pf[];
    uint8_t *sm = smem_pf + ((1024u - (smem_u32(smem_pf) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pair = (int)gridDim.x - 1 - (int)blockIdx.x;
    const int h = blockIdx.y, s = blockIdx.z;

    pdl_wait();
    DeviceStatus *st = a.status;
    if (timed_out(st)) return;
    const int q_begin = a.query_start[s], q_end = a.query_start[s + 1], ctx = a.context_lens[s];
    const int n = q_end - q_begin;
    const int B = 1 << a.log2_block;
    const int t0 = pair * kTiles * kRows;
    if (n < 0 || q_begin < 0 || q_end > a.num_tokens || n > ctx || ctx > a.max_blocks * B) {
        if (tid == 0 && pair == 0 && h == 0) latch(st, kFlagBadContext, s);
        return;
    }
    if (t0 >= n) return;                       // this sequence has fewer tiles
    // per tile x: valid rows, position of row 0, key tiles read (tile 1 sees at least tile 0's keys)
    const int rows0 = min(kRows, n - t0), rows1 = max(0, min(kRows, n - t0 - kRows));
    const int pos00 = ctx - n + t0, pos01 = pos00 + kRows;
    const int nkv0 = (pos00 + rows0 - 1) / kKeys + 1;
    const int nkv1 = rows1 ? (pos01 + rows1 - 1) / kKeys + 1 : 0;
    const int ntiles = rows1 ? 2 : 1;
    const int nkv = max(nkv0, nkv1);
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
        for (int x = 0; x < kTiles; x++) {
            mbar_init(&bars[bSFull + x], 1);
            mbar_init(&bars[bPFull + x], kSoftmaxWarps * 32);
            mbar_init(&bars[bODone + x], 1);
        }
        mbar_init(&bars[bDrain], 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(tslot, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kProducerWarp) {
        // ---------------- producer: Q tiles once, then K and V per key tile ----------------
        const uint64_t pol_q = policy_evict_first();
        const uint64_t pol_kv = policy_evict_last();   // read again by the sequence's other tiles and heads
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(&bars[bQFull], ntiles * NP * kPanelBytes);
            for (int x = 0; x < ntiles; x++)
                for (int p = 0; p < NP; p++)
                    tma_load_3d(sm + L::q + (x * NP + p) * kPanelBytes, &tmq, 64 * p, h, q_begin + t0 + x * kRows,
                                &bars[bQFull], pol_q);
        }
        const int32_t *row = a.block_tables + (size_t)s * a.max_blocks;
        const int nblk_used = (ctx + B - 1) >> a.log2_block;
        const int bpt = kKeys >> a.log2_block;          // blocks per key tile: 1..32, one per lane
        auto blocks_in = [&](int jj) { return min(bpt, nblk_used - jj * bpt); };
        int cur = lane < blocks_in(0) ? row[lane] : 0;  // this lane's block of the current tile
        int j = 0;
        for (; j < nkv; j++) {
            const int stg = j & 1;
            const int nb = blocks_in(j);
            // the next tile's block id, read ahead of the waits
            const int nxt = (j + 1 < nkv && lane < blocks_in(j + 1)) ? row[(j + 1) * bpt + lane] : 0;
            int phys = cur;
            if (lane < nb && (phys < 0 || phys >= a.num_blocks)) {
                latch(st, kFlagBadBlock, phys);
                phys = 0;                                   // keep the byte count; the output is flagged
            }
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
                if (lane < nb)
                    for (int p = 0; p < NP; p++)
                        tma_load_4d(dst + p * kPanelBytes + (uint32_t)lane * B * 128u, which ? &tmv : &tmk, 64 * p, 0,
                                    g, phys, full, pol_kv);
            }
            if (!ok) break;
            cur = nxt;
        }
        if (!ok) {
            if (lane == 0) latch(st, kFlagTimeout, j);
            // copies already issued must land before the CTA's memory is reused
            for (int jj = max(0, j - kStages); jj < j; jj++) {
                mbar_wait(&bars[bKFull + (jj & 1)], (jj >> 1) & 1, kDrainLimitCycles);
                mbar_wait(&bars[bVFull + (jj & 1)], (jj >> 1) & 1, kDrainLimitCycles);
            }
            mbar_wait(&bars[bQFull], 0, kDrainLimitCycles);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue (one thread) ----------------
        // Order: S_0(0) S_1(0), then per key tile j: O_0 += P_0 V_j, S_0(j+1), O_1 += P_1 V_j,
        // S_1(j+1): while one tile's softmax runs, the tensor core works on the other's products.
        // The products of one thread run in issue order, so S(j+1) overwrites P(j) only after
        // O += P(j) V_j has read it.
        if (lane == 0) {
            const uint32_t id_s = tc::idesc_f16(kRows, kKeys, kBf16, false);
            // O += P V: one product of N = D per 16 keys (for D = 128 the two 64-wide panels of V
            // are 16 KB apart, the descriptor's leading byte offset)
            const uint32_t id_o = tc::idesc_f16(kRows, D, kBf16, true);
            const uint32_t q_base = smem_u32(sm + L::q);
            auto issue_s = [&](int x, int stg) {
                const uint32_t k_base = smem_u32(sm + L::k) + (uint32_t)stg * NP * kPanelBytes;
                const uint32_t qx = q_base + (uint32_t)x * NP * kPanelBytes;
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    const uint32_t off = (k / 4) * kPanelBytes + (k % 4) * 32;
                    tc::mma_f16_ss(tmem + x * kTileCols, tc::smem_desc_sw128(qx + off, 1024, 1024),
                                   tc::smem_desc_sw128(k_base + off, 1024, 1024), id_s, k > 0);
                }
                tc::mma_commit(&bars[bSFull + x]);
            };
            auto issue_o = [&](int x, int stg, bool acc) {
                const uint32_t v_base = smem_u32(sm + L::v) + (uint32_t)stg * NP * kPanelBytes;
                const uint32_t tp = tmem + x * kTileCols, to = tp + kKeys;
#pragma unroll
                for (int part = 0; part < (kBf16 ? 2 : 1); part++)
#pragma unroll
                    for (int t = 0; t < kKeys / 16; t++)
                        tc::mma_f16_ts(to, tp + p_col(t, part == 1),
                                       tc::smem_desc_sw128(v_base + t * 2048, kPanelBytes, 1024), id_o,
                                       (acc || part > 0 || t > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(&bars[bQFull], 0, kWaitLimitCycles) && mbar_wait(&bars[bKFull], 0, kWaitLimitCycles);
            int j = 0;
            if (ok) {
                tc::fence_after();
                for (int x = 0; x < ntiles; x++) issue_s(x, 0);
                tc::mma_commit(&bars[bKEmpty]);
                for (; j < nkv && ok; j++) {
                    const int stg = j & 1;
                    ok = mbar_wait(&bars[bVFull + stg], (j >> 1) & 1, kWaitLimitCycles);
                    for (int x = 0; x < ntiles && ok; x++) {
                        const int nkv_x = x ? nkv1 : nkv0;
                        if (j >= nkv_x) continue;
                        ok = mbar_wait(&bars[bPFull + x], j & 1, kWaitLimitCycles);
                        if (!ok) break;
                        tc::fence_after();
                        issue_o(x, stg, j > 0);
                        if (j + 1 == nkv_x) {
                            tc::mma_commit(&bars[bODone + x]);
                        } else {
                            ok = mbar_wait(&bars[bKFull + ((j + 1) & 1)], ((j + 1) >> 1) & 1, kWaitLimitCycles);
                            if (!ok) break;
                            tc::fence_after();
                            issue_s(x, (j + 1) & 1);
                        }
                    }
                    if (ok) {
                        tc::mma_commit(&bars[bVEmpty + stg]);               // V_j read by every tile
                        if (j + 1 < nkv) tc::mma_commit(&bars[bKEmpty + ((j + 1) & 1)]);   // K_{j+1} too
                    }
                }
            }
            if (!ok) latch(st, kFlagTimeout, 1000000 + j);
            // every MMA issued so far, and every arrive it makes, completes before the CTA
            // frees its TMEM and shared memory
            tc::mma_commit(&bars[bDrain]);
            mbar_wait(&bars[bDrain], 0, ok ? kWaitLimitCycles : kDrainLimitCycles);
        }
        __syncwarp();
    } else {
        // ---------------- softmax: one thread per query row of its tile ----------------
        const int x = warp / kSoftmaxWarps;                  // query tile
        const int r = tid % (kSoftmaxWarps * 32);            // row, TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp % 4)) << 16;
        const uint32_t tS = tmem + x * kTileCols + lane_off, tO = tS + kKeys;
        bool ok = true;
        const int rows_x = x ? rows1 : rows0, pos0_x = x ? pos01 : pos00, nkv_x = x ? nkv1 : nkv0;
        if (rows_x > 0) {
            const int my_pos = r < rows_x ? pos0_x + r : pos0_x + rows_x - 1;   // last key this row sees
            float m_run = -INFINITY, l_run = 0.f;
            // the tile that zeroes V rows past the context (before its product reads them)
            const bool zero_duty = (x == 0) == (nkv0 == nkv);
            int j = 0;
            for (; j < nkv_x; j++) {
                ok = wait_warp(&bars[bSFull + x], j & 1, kWaitLimitCycles);
                if (!ok) break;
                tc::fence_after();
                const int lim = my_pos - j * kKeys;          // keys 0..lim of this tile are visible
                // Tiles below the diagonal are visible to every row of the warp: no mask, and the
                // scale folds into the exponent (the scale is positive, so the raw maximum is the
                // scaled one's).
                const bool full = __all_sync(0xffffffffu, lim >= kKeys - 1);
                const float c2 = a.scale_log2;
                // pass 1, the row maximum: the row's 128 scores in four loads, one wait
                float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                {
                    uint32_t sr[4][32];
#pragma unroll
                    for (int c = 0; c < 4; c++) tc::tmem_ld32(tS + 32 * c, sr[c]);
#pragma unroll
                    for (int c = 0; c < 4; c++) tc::tmem_wait_ld(sr[c]);
                    if (full) {
#pragma unroll
                        for (int c = 0; c < 4; c++)
#pragma unroll
                            for (int i = 0; i < 32; i += 2)
                                mxs[(i >> 1) & 3] = max3(mxs[(i >> 1) & 3], __uint_as_float(sr[c][i]),
                                                         __uint_as_float(sr[c][i + 1]));
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; c++)
#pragma unroll
                            for (int i = 0; i < 32; i++)
                                if (32 * c + i <= lim) mxs[i & 3] = fmaxf(mxs[i & 3], __uint_as_float(sr[c][i]));
                    }
                }
                // pass 2 reads the scores again chunk by chunk, each load in flight while the
                // previous chunk is computed; the first one already now
                uint32_t sb[2][32];
                tc::tmem_ld32(tS, sb[0]);
                const float mraw = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3]));
                const float mx = mraw * c2;                   // -inf when no key of the tile is visible
                const bool moved = mx > m_run + kRescaleLog2;
                const float m_new = moved ? mx : m_run;
                const float alpha = fast_exp2(m_run - m_new);  // 0 on the first tile, 1 when not moved
                m_run = m_new;
                // O of the previous tiles is complete (its products were issued before this S)
                if (j > 0 && __any_sync(0xffffffffu, moved)) {
#pragma unroll
                    for (int c = 0; c < D / 32; c++) {
                        uint32_t o[32];
                        tc::tmem_ld32(tO + 32 * c, o);
                        tc::tmem_wait_ld(o);
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tc::tmem_st32(tO + 32 * c, o);
                    }
                }
                const int kbase = j * kKeys;
                if (zero_duty && j == nkv - 1 && kbase + kKeys > ctx) {
                    // rows past the end of the context hold other data: P is 0 there, but 0 x NaN is not
                    ok = wait_warp(&bars[bVFull + (j & 1)], (j >> 1) & 1, kWaitLimitCycles);
                    if (!ok) break;
                    const int first = ctx - kbase;
                    uint8_t *vs = sm + L::v + (uint32_t)(j & 1) * NP * kPanelBytes;
                    const int nvec = (kKeys - first) * 8;    // 16-byte vectors per panel
                    for (int i = r; i < nvec * NP; i += kSoftmaxWarps * 32) {
                        const int p = i / nvec, rem = i % nvec;
                        *reinterpret_cast<uint4 *>(vs + p * kPanelBytes + (first + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();                // generic writes -> tensor-core reads
                }
                // pass 2, probabilities written over the scores
                const float neg_m = -m_run;
                float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t (&sc)[32] = sb[c & 1];
                    tc::tmem_wait_ld(sc);
                    if (c < 3) tc::tmem_ld32(tS + 32 * (c + 1), sb[(c + 1) & 1]);
                    const int kc = 32 * c;
                    uint32_t pk[kBf16 ? 32 : 16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        float p0 = fast_exp2(fmaf(__uint_as_float(sc[i]), c2, neg_m));
                        float p1 = fast_exp2(fmaf(__uint_as_float(sc[i + 1]), c2, neg_m));
                        if (!full) {
                            p0 = kc + i <= lim ? p0 : 0.f;
                            p1 = kc + i + 1 <= lim ? p1 : 0.f;
                        }
                        ls[(i >> 1) & 3] += p0 + p1;
                        const uint32_t hi = pack16<T>(p0, p1);
                        pk[i / 2] = hi;
                        // remainder after rounding (bf16 widens exactly by a shift)
                        if constexpr (kBf16)
                            pk[16 + i / 2] = pack16<T>(p0 - __uint_as_float(hi << 16),
                                                       p1 - __uint_as_float(hi & 0xffff0000u));
                    }
                    if constexpr (kBf16) tc::tmem_st32(tS + kc, pk);
                    else tc::tmem_st16(tS + kc, pk);
                }
                l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));
                tc::tmem_wait_st();
                tc::fence_before();
                mbar_arrive(&bars[bPFull + x]);
            }
            if (ok) ok = wait_warp(&bars[bODone + x], 0, kWaitLimitCycles);
            if (ok) {
                tc::fence_after();
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                T *orow = reinterpret_cast<T *>(a.out) +
                          ((size_t)(q_begin + t0 + x * kRows + r) * a.num_heads + h) * D;
#pragma unroll
                for (int c = 0; c < D / 32; c++) {
                    uint32_t o[32];
                    tc::tmem_ld32(tO + 32 * c, o);
                    tc::tmem_wait_ld(o);
                    if (r < rows_x) {
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
    using L = PfLayout<D>;
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
    const int rows_per_cta = kTiles * kRows;
    const dim3 grid((unsigned)((max_query_len + rows_per_cta - 1) / rows_per_cta), (unsigned)a.num_heads,
                    (unsigned)a.num_seqs);
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
    if (!(scale > 0.f) || scale == INFINITY)
        return fail(PKV_EINVAL, "paged_attention_prefill: scale must be positive and finite");
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
