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
//   * Work items: (sequence, query head, 256 new tokens) = two query tiles of
//     128 rows (M of both products) that take turns on the tensor core.  One
//     persistent CTA per SM takes items from a ticket counter in the caller's
//     workspace (without one, every gridDim-th ticket), the pairs of tiles
//     with the most keys first.
//   * A producer warp claims and looks up the next item while the current one
//     streams and hands it to the other warps through a two-slot item ring; it
//     loads each item's query tiles (tiled TMA over the query tensor) and then,
//     for each 128-key tile, the tile's K blocks (tiled TMA over the cache, one
//     box of B tokens x 64 elements per block and 64-element panel of d) into
//     a two-stage ring that runs on across items; a value warp does the same
//     for the V blocks in a ring of its own, so that neither waits behind the
//     other's copy issue.  Boxes land 128-byte swizzled, the layout the MMA
//     descriptors describe.
//   * The MMA warp (converged; one elected lane issues) runs tcgen05.mma:
//     S = Q K^T (M 128, N 128, fp32 in TMEM), then O += P V with P read from
//     TMEM and V read MN-major straight from the cache layout (N = d: one
//     product per 16 keys).  While one tile's softmax runs, the tensor core
//     computes the other tile's products.  An item with a single query tile
//     gives its key tiles alternately to both tiles' TMEM and softmax warps
//     (each pair of key tiles then overlaps as the two tiles of a pair do),
//     and the two partial outputs are merged at the end.
//   * Four softmax warps per tile (one thread per row) read S from TMEM (on a
//     tile that crosses the diagonal they first overwrite the scores of keys
//     after the row's position with -inf, so that every tile runs the same
//     unmasked code), keep a running max and sum in fp32 (log2
//     domain; the reference max moves only when it grows by more than 8, so
//     probabilities stay below 2^8), write P as 16-bit over the scores in
//     TMEM (for bf16 as a rounded part and its remainder) and rescale O in
//     TMEM when a row's reference moved.  At the end they divide by the sum
//     and write the rows through a per-warp shared-memory buffer, so that
//     each store covers whole 128-byte row segments.
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
constexpr int kProducerWarp = kTiles * kSoftmaxWarps;   // items, queries, keys
constexpr int kMmaWarp = kProducerWarp + 1;
constexpr int kValueWarp = kMmaWarp + 1;                // values
constexpr int kThreads = (kValueWarp + 1) * 32;
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
    WsHeader *hdr;                       // ticket counters; null: static round robin
    int num_seqs, num_tokens, max_blocks, log2_block, num_blocks;
    int num_heads, group;
    int head_pairs;                      // 1: an item's two tiles are the same rows of two query heads
                                         // of one kv head (group even); 0: two row tiles of one head
    int num_pairs;                       // row tiles (head_pairs) or pairs of them per sequence (of the longest)
    int num_items;                       // num_pairs x (query heads, or head pairs) x num_seqs tickets
    float scale_log2;                    // scale * log2(e)
};

// A work item as the producer publishes it to the other warps: (sequence s,
// query head h, the two 128-row tiles from new token t0), or (sequence s,
// query heads h and h1 of one kv head, the 128-row tile from t0 of each).
struct PfItem {
    int s, h, t0, q_begin, ctx, pos00;   // pos00: position of the item's first new token
    int rows0, rows1;                    // valid rows of the two tiles (rows1 = 0: one tile)
    int nkv0, nkv1;                      // key tiles each tile reads
    int stop;                            // no further items
    int split;                           // one query tile, its key tiles alternating between both slots
    int h1;                              // query head of tile 1
    int rstep;                           // rows between the tiles' first tokens: 128, or 0 (two heads)
    int pad[2];
};

// Shared memory: the two query tiles, the K/V ring, two item slots and a
// 4 KB buffer per softmax warp through which its output rows go to global
// memory as whole lines.  P stays in TMEM, over the tile's S columns.  The allocation keeps one CTA per
// SM (each CTA takes all 512 TMEM columns).
template <int D> struct PfLayout {
    static constexpr int NP = D / 64;                              // panels of d
    static constexpr uint32_t q = 0;                                // kTiles x NP panels
    static constexpr uint32_t k = q + kTiles * NP * kPanelBytes;    // kStages x NP panels
    static constexpr uint32_t v = k + kStages * NP * kPanelBytes;
    static constexpr uint32_t bars = v + kStages * NP * kPanelBytes;
    static constexpr uint32_t items = bars + 256;
    static constexpr uint32_t stage = items + 2 * sizeof(PfItem);   // kTiles x kSoftmaxWarps x 4 KB
    static constexpr uint32_t bytes = stage + kTiles * kSoftmaxWarps * 4096;
    static constexpr size_t alloc = (bytes + 1024 > 120u * 1024u) ? bytes + 1024 : 120u * 1024u;
};

// barrier slots
enum : int { bQFull = 0, bQEmpty = 1, bKFull = 2, bVFull = 4, bKEmpty = 6, bVEmpty = 8, bSFull = 10, bPFull = 12,
             bODone = 14, bItemFull = 16, bItemEmpty = 18, bDrain = 20, bMerge = 21, bMerged = 22, kNumBars = 23 };
// an item slot is released by every softmax warp, the MMA warp and the value warp
constexpr int kItemReaders = kTiles * kSoftmaxWarps + 2;

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
constexpr uint32_t p_col(int t, bool lo) { return 32 * (t >> 1) + 8 * (t & 1) + (lo ? 16 : 0); }
// (the product runs below write these columns as immediates)
static_assert(p_col(1, false) == 8 && p_col(2, false) == 32 && p_col(3, false) == 40 && p_col(7, false) == 104 &&
                  p_col(0, true) == 16 && p_col(5, true) == 88 && p_col(7, true) == 120,
              "P column layout");

// A tile's products as one run of one elected lane (one election, the operands'
// descriptors stepped by immediates).  The offsets follow the shared-memory and
// TMEM layouts above: S = Q K^T steps 32 bytes along a 64-element panel (2 in
// descriptor units) and a panel (kPanelBytes >> 4 = 1024) after four steps;
// O += P V steps the P columns as p_col and V by 16 keys (2048 bytes, 128 units).
static_assert((kPanelBytes >> 4) == 1024 && (32 >> 4) == 2 && ((16 * 128) >> 4) == 128 && kKeys == 128,
              "descriptor steps written as immediates in the product runs");
#define PKV_SS(o, acc) "add.s64 qa, %1, " #o ";\n\tadd.s64 kb, %2, " #o ";\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], qa, kb, %3, " acc ";\n\t"
#define PKV_TS(ao, bo, acc) "add.u32 ta, %1, " #ao ";\n\tadd.s64 vb, %2, " #bo ";\n\t" \
    "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], vb, %3, " acc ";\n\t"
#define PKV_RUN_HEAD "{\n\t.reg .pred e, t, f, pa;\n\t.reg .b64 qa, kb, vb;\n\t.reg .b32 ta;\n\t" \
    "setp.ne.b32 f, %4, %4;\n\tsetp.eq.b32 t, %4, %4;\n\tsetp.ne.b32 pa, %5, 0;\n\t" \
    "elect.sync _|e, 0xffffffff;\n\t"

// S = Q K^T over the head dimension (the first product overwrites).
template <int D> __device__ __forceinline__ void mma_s_run(uint32_t d, uint64_t qd, uint64_t kd, uint32_t idesc) {
    if constexpr (D == 128) {
        asm volatile(PKV_RUN_HEAD PKV_SS(0, "f") PKV_SS(2, "t") PKV_SS(4, "t") PKV_SS(6, "t")
                     PKV_SS(1024, "t") PKV_SS(1026, "t") PKV_SS(1028, "t") PKV_SS(1030, "t") "}"
                     ::"r"(d), "l"(qd), "l"(kd), "r"(idesc), "r"(0u), "r"(0u) : "memory");
    } else {
        asm volatile(PKV_RUN_HEAD PKV_SS(0, "f") PKV_SS(2, "t") PKV_SS(4, "t") PKV_SS(6, "t") "}"
                     ::"r"(d), "l"(qd), "l"(kd), "r"(idesc), "r"(0u), "r"(0u) : "memory");
    }
}

// O (+)= P V over the tile's 128 keys, P from TMEM (a = its first column), the first product
// accumulating when `acc`; for bf16 also the remainder part (columns + 16).
template <bool kLo> __device__ __forceinline__ void mma_o_run(uint32_t d, uint32_t a, uint64_t vd, uint32_t idesc,
                                                            uint32_t acc) {
    if constexpr (!kLo) {
        asm volatile(PKV_RUN_HEAD PKV_TS(0, 0, "pa") PKV_TS(8, 128, "t") PKV_TS(32, 256, "t") PKV_TS(40, 384, "t")
                     PKV_TS(64, 512, "t") PKV_TS(72, 640, "t") PKV_TS(96, 768, "t") PKV_TS(104, 896, "t") "}"
                     ::"r"(d), "r"(a), "l"(vd), "r"(idesc), "r"(0u), "r"(acc) : "memory");
    } else {
        asm volatile(PKV_RUN_HEAD PKV_TS(0, 0, "pa") PKV_TS(8, 128, "t") PKV_TS(32, 256, "t") PKV_TS(40, 384, "t")
                     PKV_TS(64, 512, "t") PKV_TS(72, 640, "t") PKV_TS(96, 768, "t") PKV_TS(104, 896, "t")
                     PKV_TS(16, 0, "t") PKV_TS(24, 128, "t") PKV_TS(48, 256, "t") PKV_TS(56, 384, "t")
                     PKV_TS(80, 512, "t") PKV_TS(88, 640, "t") PKV_TS(112, 768, "t") PKV_TS(120, 896, "t") "}"
                     ::"r"(d), "r"(a), "l"(vd), "r"(idesc), "r"(0u), "r"(acc) : "memory");
    }
}
#undef PKV_SS
#undef PKV_TS
#undef PKV_RUN_HEAD

// Ticket t in [0, num_items): the tiles with the most keys first (row-tile or
// pair index descending), then sequence, then head (or head pair: h is its
// first head).
__device__ __forceinline__ void ticket_item(const PrefillArgs &a, int t, int &s, int &h, int &pair) {
    const int nh = a.head_pairs ? a.num_heads / 2 : a.num_heads;
    const int hs = nh * a.num_seqs;
    pair = a.num_pairs - 1 - t / hs;
    const int rem = t % hs;
    s = rem / nh;
    h = (rem % nh) * (a.head_pairs ? 2 : 1);
}

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
    const int G = (int)gridDim.x;

    pdl_wait();
    DeviceStatus *st = a.status;
    WsHeader *hdr = a.hdr;
    if (hdr && hdr->magic != kWsMagic) {
        if (blockIdx.x == 0 && tid == 0) latch(st, kFlagBadWorkspace, (long long)hdr->magic);
        return;
    }
    if (timed_out(st)) {
        // this CTA claims no ticket, but it still counts towards the counters' reset
        if (hdr && tid == 0) {
            __threadfence();
            if (atomicAdd(&hdr->done, 1u) == (unsigned)G - 1) {
                hdr->next = 0;
                hdr->done = 0;
                __threadfence();
            }
        }
        return;
    }
    const int B = 1 << a.log2_block;

    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::bars);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    PfItem *items = reinterpret_cast<PfItem *>(sm + L::items);
    if (tid == 0) {
        mbar_init(&bars[bQFull], 1);
        mbar_init(&bars[bQEmpty], 1);
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
        for (int i = 0; i < 2; i++) {
            mbar_init(&bars[bItemFull + i], 1);
            mbar_init(&bars[bItemEmpty + i], kItemReaders);
        }
        mbar_init(&bars[bDrain], 1);
        mbar_init(&bars[bMerge], kSoftmaxWarps * 32);
        mbar_init(&bars[bMerged], kSoftmaxWarps * 32);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(tslot, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tslot;

    if (warp == kProducerWarp) {
        // ---------------- producer: items, then per item its queries and K/V tiles ----------------
        const uint64_t pol_q = policy_evict_first();
        const uint64_t pol_kv = policy_evict_last();   // read again by the sequence's other tiles and heads
        // the ticket after `prev` (dynamic: a new claim)
        auto next_ticket = [&](int prev) -> int {
            if (!hdr) return prev + G;
            unsigned t = 0;
            if (lane == 0) t = (unsigned)G + atomicAdd(&hdr->next, 1u);
            t = __shfl_sync(0xffffffffu, t, 0);
            return t > (unsigned)a.num_items ? a.num_items : (int)t;
        };
        // the first item with work at or after ticket t (following the claims); stop when none
        auto resolve = [&](int t, PfItem &o) -> int {
            while (t < a.num_items) {
                int s, h, pair;
                ticket_item(a, t, s, h, pair);
                const int qb = a.query_start[s], qe = a.query_start[s + 1], ctx = a.context_lens[s];
                const int n = qe - qb, t0 = pair * (a.head_pairs ? kRows : kTiles * kRows);
                if (n < 0 || qb < 0 || qe > a.num_tokens || n > ctx || ctx > a.max_blocks * B) {
                    if (lane == 0 && pair == 0 && h == 0) latch(st, kFlagBadContext, s);
                } else if (t0 < n) {
                    o.s = s;
                    o.h = h;
                    o.t0 = t0;
                    o.q_begin = qb;
                    o.ctx = ctx;
                    o.pos00 = ctx - n + t0;
                    o.rows0 = min(kRows, n - t0);
                    o.nkv0 = (o.pos00 + o.rows0 - 1) / kKeys + 1;
                    if (a.head_pairs) {                        // the same rows of the next head
                        o.rows1 = o.rows0;
                        o.nkv1 = o.nkv0;
                        o.h1 = h + 1;
                        o.rstep = 0;
                    } else {
                        o.rows1 = max(0, min(kRows, n - t0 - kRows));
                        o.nkv1 = o.rows1 ? (o.pos00 + kRows + o.rows1 - 1) / kKeys + 1 : 0;
                        o.h1 = h;
                        o.rstep = kRows;
                    }
                    o.stop = 0;
                    o.split = (o.rows1 == 0 && o.nkv0 >= 2) ? 1 : 0;
                    return t;
                }
                t = next_ticket(t);
            }
            o.stop = 1;
            return t;
        };
        bool ok = true;
        int k = 0;       // items published
        int gj = 0;      // key tiles loaded: ring position
        int j = 0;
        PfItem cur;
        int cur_t = resolve((int)blockIdx.x, cur);
        for (;; k++) {
            const int slot = k & 1;
            if (k >= 2) {
                ok = wait_warp(&bars[bItemEmpty + slot], ((k >> 1) - 1) & 1, kWaitLimitCycles);
                if (!ok) break;
            }
            if (lane == 0) items[slot] = cur;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[bItemFull + slot]);
            if (cur.stop) break;
            // the previous item's products must have read its queries
            if (k >= 1) {
                ok = wait_warp(&bars[bQEmpty], (k - 1) & 1, kWaitLimitCycles);
                if (!ok) break;
            }
            const int ntiles = cur.rows1 ? 2 : 1, nkv = max(cur.nkv0, cur.nkv1);
            const int g = cur.h / a.group;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[bQFull], ntiles * NP * kPanelBytes);
                for (int x = 0; x < ntiles; x++)
                    for (int p = 0; p < NP; p++)
                        tma_load_3d(sm + L::q + (x * NP + p) * kPanelBytes, &tmq, 64 * p, x ? cur.h1 : cur.h,
                                    cur.q_begin + cur.t0 + x * cur.rstep, &bars[bQFull], pol_q);
            }
            const int32_t *row = a.block_tables + (size_t)cur.s * a.max_blocks;
            const int nblk_used = (cur.ctx + B - 1) >> a.log2_block;
            const int bpt = kKeys >> a.log2_block;          // blocks per key tile: 1..32, one per lane
            auto blocks_in = [&](int jj) { return min(bpt, nblk_used - jj * bpt); };
            int cb = lane < blocks_in(0) ? row[lane] : 0;  // this lane's block of the current tile
            PfItem nxt_item;
            int nxt_t = 0;
            for (j = 0; j < nkv; j++, gj++) {
                const int stg = gj & 1;
                const int nb = blocks_in(j);
                // the next tile's block id, read ahead of the waits
                const int nxt = (j + 1 < nkv && lane < blocks_in(j + 1)) ? row[(j + 1) * bpt + lane] : 0;
                int phys = cb;
                if (lane < nb && (phys < 0 || phys >= a.num_blocks)) {
                    latch(st, kFlagBadBlock, phys);
                    phys = 0;                                   // keep the byte count; the output is flagged
                }
                const uint32_t bytes = (uint32_t)nb * (uint32_t)B * 128u * NP;
                for (int which = 0; which < 1; which++) {       // K (the value warp loads V)
                    if (gj >= kStages) {
                        ok = wait_warp(&bars[(which ? bVEmpty : bKEmpty) + stg], ((gj >> 1) - 1) & 1,
                                       kWaitLimitCycles);
                        if (!ok) break;
                    }
                    uint64_t *full = &bars[(which ? bVFull : bKFull) + stg];
                    if (lane == 0) mbar_arrive_expect_tx(full, bytes);
                    __syncwarp();
                    uint8_t *dst = sm + (which ? L::v : L::k) + (uint32_t)stg * NP * kPanelBytes;
                    if (lane < nb)
                        for (int p = 0; p < NP; p++)
                            tma_load_4d(dst + p * kPanelBytes + (uint32_t)lane * B * 128u, which ? &tmv : &tmk,
                                        64 * p, 0, g, phys, full, pol_kv);
                }
                if (!ok) break;
                cb = nxt;
                // claim and look up the next item while this one's tiles stream in
                if (j == 0) nxt_t = resolve(next_ticket(cur_t), nxt_item);
            }
            if (!ok) break;
            cur = nxt_item;
            cur_t = nxt_t;
        }
        if (!ok) {
            if (lane == 0) latch(st, kFlagTimeout, gj);
            // copies already issued must land before the CTA's memory is reused
            for (int jj = max(0, gj - kStages); jj <= gj; jj++)
                mbar_wait(&bars[bKFull + (jj & 1)], (jj >> 1) & 1, kDrainLimitCycles);
            mbar_wait(&bars[bQFull], k & 1, kDrainLimitCycles);
        }
        // the last CTA to finish leaves the counters at zero for the next call
        if (hdr && lane == 0) {
            __threadfence();
            if (atomicAdd(&hdr->done, 1u) == (unsigned)G - 1) {
                hdr->next = 0;
                hdr->done = 0;
                __threadfence();
            }
        }
    } else if (warp == kValueWarp) {
        // ---------------- values: per item, its V tiles into their own two-stage ring ----------------
        // A warp of its own, so that the values' copies are issued beside the keys', not
        // behind them (each tile takes its issuing warp about half a microsecond at B = 16).
        const uint64_t pol_kv = policy_evict_last();
        bool ok = true;
        int gj = 0, k = 0;
        for (;; k++) {
            const int slot = k & 1;
            ok = wait_warp(&bars[bItemFull + slot], (k >> 1) & 1, kWaitLimitCycles);
            if (!ok) break;
            const PfItem it = items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[bItemEmpty + slot]);
            if (it.stop) break;
            const int nkv = max(it.nkv0, it.nkv1);
            const int g = it.h / a.group;
            const int32_t *row = a.block_tables + (size_t)it.s * a.max_blocks;
            const int nblk_used = (it.ctx + B - 1) >> a.log2_block;
            const int bpt = kKeys >> a.log2_block;
            auto blocks_in = [&](int jj) { return min(bpt, nblk_used - jj * bpt); };
            int cb = lane < blocks_in(0) ? row[lane] : 0;
            for (int j = 0; j < nkv; j++, gj++) {
                const int stg = gj & 1;
                const int nb = blocks_in(j);
                const int nxt = (j + 1 < nkv && lane < blocks_in(j + 1)) ? row[(j + 1) * bpt + lane] : 0;
                int phys = cb;
                if (lane < nb && (phys < 0 || phys >= a.num_blocks)) {
                    latch(st, kFlagBadBlock, phys);
                    phys = 0;
                }
                if (gj >= kStages) {
                    ok = wait_warp(&bars[bVEmpty + stg], ((gj >> 1) - 1) & 1, kWaitLimitCycles);
                    if (!ok) break;
                }
                uint64_t *full = &bars[bVFull + stg];
                if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)nb * (uint32_t)B * 128u * NP);
                __syncwarp();
                uint8_t *dst = sm + L::v + (uint32_t)stg * NP * kPanelBytes;
                if (lane < nb)
                    for (int p = 0; p < NP; p++)
                        tma_load_4d(dst + p * kPanelBytes + (uint32_t)lane * B * 128u, &tmv, 64 * p, 0, g, phys, full,
                                    pol_kv);
                cb = nxt;
            }
            if (!ok) break;
        }
        if (!ok) {
            if (lane == 0) latch(st, kFlagTimeout, 3000000 + gj);
            for (int jj = max(0, gj - kStages); jj <= gj; jj++)
                mbar_wait(&bars[bVFull + (jj & 1)], (jj >> 1) & 1, kDrainLimitCycles);
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issue ----------------
        // Per item: S_0(0) S_1(0), then per key tile j: O_0 += P_0 V_j, S_0(j+1), O_1 += P_1 V_j,
        // S_1(j+1): while one tile's softmax runs, the tensor core works on the other's products.
        // The products run in issue order, so S(j+1) overwrites P(j) only after O += P(j) V_j has
        // read it, and the next item's first S only after this item's last product.  The next
        // item's first O product (which overwrites O) waits for that tile's first P, which its
        // softmax threads write only after they have read this item's O.
        // The whole warp runs the loop (its waits and descriptors are warp-uniform values); one
        // elected lane issues each tile's run of products (one election per run) and each commit.
        // A tile of 64 rows or fewer takes M = 64 products (half the tensor work); their rows
        // sit in TMEM lanes 0-15 of each 32-lane quarter (row r in lane 32 (r / 16) + r % 16).
        const uint32_t id_s128 = tc::idesc_f16(kRows, kKeys, kBf16, false), id_s64 = tc::idesc_f16(64, kKeys, kBf16, false);
        // O += P V: one product of N = D per 16 keys (for D = 128 the two 64-wide panels of V
        // are 16 KB apart, the descriptor's leading byte offset)
        const uint32_t id_o128 = tc::idesc_f16(kRows, D, kBf16, true), id_o64 = tc::idesc_f16(64, D, kBf16, true);
        int m64m = 0;                                    // bit x: slot x of the current item has M = 64
        // descriptors of the first query tile and of ring stage 0; the start-address field
        // (address >> 4, 14 bits) takes byte offsets >> 4 without carrying out
        const uint64_t q_desc = tc::smem_desc_sw128(smem_u32(sm + L::q), 1024, 1024);
        const uint64_t k_desc = tc::smem_desc_sw128(smem_u32(sm + L::k), 1024, 1024);
        const uint64_t v_desc = tc::smem_desc_sw128(smem_u32(sm + L::v), kPanelBytes, 1024);
        constexpr uint32_t kStageStep = NP * kPanelBytes >> 4;
        // S of slot x (its TMEM columns) from query buffer qx
        auto issue_s = [&](int x, int stg, int qx) {
            const uint64_t kd = k_desc + (uint64_t)(stg * kStageStep);
            const uint64_t qd = q_desc + (uint64_t)(qx * kStageStep);
            mma_s_run<D>(tmem + x * kTileCols, qd, kd, (m64m >> x) & 1 ? id_s64 : id_s128);
            tc::mma_commit_warp(&bars[bSFull + x]);
        };
        auto issue_o = [&](int x, int stg, bool acc) {
            const uint64_t vd = v_desc + (uint64_t)(stg * kStageStep);
            const uint32_t tp = tmem + x * kTileCols, to = tp + kKeys;
            mma_o_run<kBf16>(to, tp, vd, (m64m >> x) & 1 ? id_o64 : id_o128, acc ? 1u : 0u);
        };
        bool ok = true;
        int gj = 0, pc[kTiles] = {0, 0};
        int k = 0;
        for (;; k++) {
            const int slot = k & 1;
            ok = wait_warp(&bars[bItemFull + slot], (k >> 1) & 1, kWaitLimitCycles);
            if (!ok) break;
            const PfItem it = items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[bItemEmpty + slot]);
            if (it.stop) break;
            const int ntiles = it.rows1 ? 2 : 1, nkv = max(it.nkv0, it.nkv1);
            m64m = it.split ? (it.rows0 <= 64 ? 3 : 0) : (it.rows0 <= 64 ? 1 : 0) | (it.rows1 > 0 && it.rows1 <= 64 ? 2 : 0);
            ok = wait_warp(&bars[bQFull], k & 1, kWaitLimitCycles) &&
                 wait_warp(&bars[bKFull + (gj & 1)], (gj >> 1) & 1, kWaitLimitCycles);
            if (!ok) break;
            tc::fence_after();
            if (it.split) {
                // One query tile; key tile j goes to slot j % 2, each slot with its own S, P and O:
                // S_0(0) S_1(1), then per key tile j: O_x += P_x V_j, S_x(j + 2).  The slots'
                // softmax chains overlap as the two tiles' do in a pair.
                issue_s(0, gj & 1, 0);
                tc::mma_commit_warp(&bars[bKEmpty + (gj & 1)]);
                ok = wait_warp(&bars[bKFull + ((gj + 1) & 1)], ((gj + 1) >> 1) & 1, kWaitLimitCycles);
                if (!ok) break;
                tc::fence_after();
                issue_s(1, (gj + 1) & 1, 0);
                tc::mma_commit_warp(&bars[bKEmpty + ((gj + 1) & 1)]);
                if (nkv == 2) tc::mma_commit_warp(&bars[bQEmpty]);
                for (int j = 0; j < nkv && ok; j++) {
                    const int g = gj + j, stg = g & 1, x = j & 1;
                    const int pcx = x ? pc[1] : pc[0];          // (no dynamic index: pc stays in registers)
                    ok = wait_warp(&bars[bVFull + stg], (g >> 1) & 1, kWaitLimitCycles) &&
                         wait_warp(&bars[bPFull + x], pcx & 1, kWaitLimitCycles);
                    if (x) pc[1]++;
                    else pc[0]++;
                    if (!ok) break;
                    tc::fence_after();
                    issue_o(x, stg, j >= 2);
                    if (j + 2 < nkv) {
                        ok = wait_warp(&bars[bKFull + ((g + 2) & 1)], ((g + 2) >> 1) & 1, kWaitLimitCycles);
                        if (!ok) break;
                        tc::fence_after();
                        issue_s(x, (g + 2) & 1, 0);
                        tc::mma_commit_warp(&bars[bKEmpty + ((g + 2) & 1)]);      // K_{j+2} read
                        if (j + 3 == nkv) tc::mma_commit_warp(&bars[bQEmpty]);  // the item's last S
                    } else {
                        tc::mma_commit_warp(&bars[bODone + x]);
                    }
                    tc::mma_commit_warp(&bars[bVEmpty + stg]);                    // V_j read
                }
                if (!ok) break;
                gj += nkv;
                continue;
            }
            for (int x = 0; x < ntiles; x++) issue_s(x, gj & 1, x);
            tc::mma_commit_warp(&bars[bKEmpty + (gj & 1)]);
            if (nkv == 1) tc::mma_commit_warp(&bars[bQEmpty]);   // the item's last S has been issued
            for (int j = 0; j < nkv && ok; j++) {
                const int g = gj + j, stg = g & 1;
                ok = wait_warp(&bars[bVFull + stg], (g >> 1) & 1, kWaitLimitCycles);
                for (int x = 0; x < ntiles && ok; x++) {
                    const int nkv_x = x ? it.nkv1 : it.nkv0;
                    if (j >= nkv_x) continue;
                    ok = wait_warp(&bars[bPFull + x], pc[x] & 1, kWaitLimitCycles);
                    pc[x]++;
                    if (!ok) break;
                    tc::fence_after();
                    issue_o(x, stg, j > 0);
                    if (j + 1 == nkv_x) {
                        tc::mma_commit_warp(&bars[bODone + x]);
                    } else {
                        ok = wait_warp(&bars[bKFull + ((g + 1) & 1)], ((g + 1) >> 1) & 1, kWaitLimitCycles);
                        if (!ok) break;
                        tc::fence_after();
                        issue_s(x, (g + 1) & 1, x);
                    }
                }
                if (ok) {
                    tc::mma_commit_warp(&bars[bVEmpty + stg]);                        // V_j read by every tile
                    if (j + 1 < nkv) tc::mma_commit_warp(&bars[bKEmpty + ((g + 1) & 1)]);   // K_{j+1} too
                    if (j + 2 == nkv) tc::mma_commit_warp(&bars[bQEmpty]);            // and the last S issued
                }
            }
            if (!ok) break;
            gj += nkv;
        }
        if (!ok && lane == 0) latch(st, kFlagTimeout, 1000000 + k);
        // every MMA issued so far, and every arrive it makes, completes before the CTA
        // frees its TMEM and shared memory
        tc::mma_commit_warp(&bars[bDrain]);
        wait_warp(&bars[bDrain], 0, ok ? kWaitLimitCycles : kDrainLimitCycles);
        __syncwarp();
    } else {
        // ---------------- softmax: one thread per query row of its tile ----------------
        const int x = warp / kSoftmaxWarps;                  // query tile
        const int r = tid % (kSoftmaxWarps * 32);            // row, TMEM lane
        const uint32_t lane_off = (uint32_t)(32 * (warp % 4)) << 16;
        const uint32_t tS = tmem + x * kTileCols + lane_off, tO = tS + kKeys;
        bool ok = true;
        int gj = 0, sc = 0, u = 0, k = 0, j = 0, um = 0;
        // split items: the other slot's O and the buffer for its (max, sum)
        const uint32_t tO1 = tmem + kTileCols + lane_off + kKeys;
        float *xch = reinterpret_cast<float *>(sm + L::stage + (uint32_t)(kSoftmaxWarps + warp % 4) * 4096u);
        for (;; k++) {
            const int slot = k & 1;
            ok = wait_warp(&bars[bItemFull + slot], (k >> 1) & 1, kWaitLimitCycles);
            if (!ok) break;
            const PfItem it = items[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[bItemEmpty + slot]);
            if (it.stop) break;
            const int nkv = max(it.nkv0, it.nkv1);
            const int gbase = gj;
            gj += nkv;
            const bool split = it.split != 0;
            // split: both slots serve tile 0's rows, slot x its key tiles x, x + 2, ...
            const int rows_x = split ? it.rows0 : (x ? it.rows1 : it.rows0);
            if (rows_x <= 0) continue;
            const int pos0_x = split ? it.pos00 : it.pos00 + x * it.rstep;
            const int nkv_x = split ? (nkv - x + 1) / 2 : (x ? it.nkv1 : it.nkv0);
            const int kstep = split ? 2 : 1, kfirst = split ? x : 0;
            // the tile row this thread holds: lane 32 q + i holds row 32 q + i (M = 128) or, for a
            // tile of 64 rows or fewer (M = 64 products), row 16 q + i for i < 16 and none above
            const bool m64 = rows_x <= 64;
            const int rr = m64 ? (lane < 16 ? 16 * (warp % 4) + lane : kRows) : r;
            const int my_pos = rr < rows_x ? pos0_x + rr : pos0_x + rows_x - 1;   // last key this row sees
            float m_run = -INFINITY, l_run = 0.f;
            // the slot that zeroes V rows past the context (before its product reads them)
            const bool zero_duty = split ? x == ((nkv - 1) & 1) : (x == 0) == (it.nkv0 == nkv);
            for (int i = 0; i < nkv_x; i++) {
                j = kfirst + kstep * i;                      // the key tile
                ok = wait_warp(&bars[bSFull + x], sc & 1, kWaitLimitCycles);
                sc++;
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
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        // keys 0..t of this chunk are visible to this row
                        const int t = lim - 32 * c;
                        if (!full && __any_sync(0xffffffffu, t < 31)) {
                            // keys after the row's position: the score becomes -inf, in the registers
                            // for the maximum and in TMEM for pass 2 (whose exponent then gives 0),
                            // so that both passes run the same unmasked code on every tile
#pragma unroll
                            for (int i = 0; i < 32; i++) sr[c][i] = i <= t ? sr[c][i] : 0xff800000u;
                            tc::tmem_st32(tS + 32 * c, sr[c]);
                        }
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            mxs[(i >> 1) & 3] = max3(mxs[(i >> 1) & 3], __uint_as_float(sr[c][i]),
                                                     __uint_as_float(sr[c][i + 1]));
                    }
                    if (!full) tc::tmem_wait_st();
                }
                // pass 2 reads the scores again chunk by chunk, each load in flight while the
                // previous chunk is computed; the first one already now
                uint32_t sb[2][32];
                tc::tmem_ld32(tS, sb[0]);
                const float mraw = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3]));
                const float mx = mraw * c2;                   // -inf when no key of the tile is visible
                const bool moved = mx > m_run + kRescaleLog2;
                const float m_new = moved ? mx : m_run;
                // 0 on the first visible tile, 1 when not moved (and while no key was visible)
                const float alpha = m_new == -INFINITY ? 1.f : fast_exp2(m_run - m_new);
                m_run = m_new;
                // O of the previous tiles is complete (its products were issued before this S)
                if (i > 0 && __any_sync(0xffffffffu, moved)) {
                    // (rare after a row's first tiles: a loop, not unrolled, keeps the code small)
#pragma unroll 1
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
                if (zero_duty && j == nkv - 1 && kbase + kKeys > it.ctx) {
                    // rows past the end of the context hold other data: P is 0 there, but 0 x NaN is not
                    const int g = gbase + j;
                    ok = wait_warp(&bars[bVFull + (g & 1)], (g >> 1) & 1, kWaitLimitCycles);
                    if (!ok) break;
                    const int first = it.ctx - kbase;
                    uint8_t *vs = sm + L::v + (uint32_t)(g & 1) * NP * kPanelBytes;
                    const int nvec = (kKeys - first) * 8;    // 16-byte vectors per panel
                    for (int i = r; i < nvec * NP; i += kSoftmaxWarps * 32) {
                        const int p = i / nvec, rem = i % nvec;
                        *reinterpret_cast<uint4 *>(vs + p * kPanelBytes + (first + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();                // generic writes -> tensor-core reads
                }
                // pass 2, probabilities written over the scores
                // exponents and row sums two lanes at a time (packed fp32 pairs)
                // (a row that sees no key yet has m_run = -inf and only -inf scores: its
                // exponents are taken against 0, so that they give 0 and not NaN)
                const float mref = m_run == -INFINITY ? 0.f : m_run;
                const unsigned long long c2x2 = pack2(c2, c2), negm2 = pack2(-mref, -mref);
                unsigned long long ls2[2] = {0ull, 0ull};
                // (for bf16, whose probabilities take twice the instructions, a loop over pairs of
                // chunks, not unrolled: the kernel's code stays small)
                constexpr int kPairUnroll = kBf16 ? 1 : 2;
#pragma unroll kPairUnroll
                for (int cc = 0; cc < 4; cc += 2)
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int c = cc + h;
                    uint32_t (&sc)[32] = sb[h];
                    tc::tmem_wait_ld(sc);
                    if (c < 3) tc::tmem_ld32(tS + 32 * (c + 1), sb[h ^ 1]);
                    const int kc = 32 * c;
                    uint32_t pk[kBf16 ? 32 : 16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const unsigned long long xx =
                            fma2(pack2(__uint_as_float(sc[i]), __uint_as_float(sc[i + 1])), c2x2, negm2);
                        const float p0 = fast_exp2(lo2(xx));
                        const float p1 = fast_exp2(hi2(xx));
                        ls2[(i >> 1) & 1] = add2(ls2[(i >> 1) & 1], pack2(p0, p1));
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
                l_run = l_run * alpha + ((lo2(ls2[0]) + hi2(ls2[0])) + (lo2(ls2[1]) + hi2(ls2[1])));
                tc::tmem_wait_st();
                tc::fence_before();
                mbar_arrive(&bars[bPFull + x]);
            }
            if (!ok) break;
            ok = wait_warp(&bars[bODone + x], u & 1, kWaitLimitCycles);
            u++;
            if (!ok) break;
            tc::fence_after();
            float a0 = 1.f, a1 = 0.f;                        // weights of this slot's O and the other's
            if (split) {
                if (x == 1) {
                    // hand (max, sum) to slot 0, which merges; wait until it has read this O
                    xch[2 * lane] = m_run;
                    xch[2 * lane + 1] = l_run;
                    tc::fence_before();
                    mbar_arrive(&bars[bMerge]);
                    ok = wait_warp(&bars[bMerged], um & 1, kWaitLimitCycles);
                    um++;
                    if (!ok) break;
                    continue;
                }
                ok = wait_warp(&bars[bMerge], um & 1, kWaitLimitCycles);
                if (!ok) break;
                tc::fence_after();
                const float m1 = xch[2 * lane], l1 = xch[2 * lane + 1];
                const float M = fmaxf(m_run, m1);
                a0 = fast_exp2(m_run - M);
                a1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
                l_run = l_run * a0 + l1 * a1;
            }
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            // 32 columns of this row's output (over both slots of a split item), unscaled
            auto load_out = [&](int col, uint32_t (&o)[32]) {
                tc::tmem_ld32(tO + col, o);
                if (split) {
                    uint32_t o1[32];
                    tc::tmem_ld32(tO1 + col, o1);
                    tc::tmem_wait_ld(o);
                    tc::tmem_wait_ld(o1);
#pragma unroll
                    for (int i = 0; i < 32; i++)
                        o[i] = __float_as_uint(fmaf(__uint_as_float(o[i]), a0, __uint_as_float(o1[i]) * a1));
                } else {
                    tc::tmem_wait_ld(o);
                }
            };
            // Each 64-column panel of the warp's 32 rows goes through the warp's buffer: every
            // thread writes its row (16-byte units swizzled by row, free of bank conflicts), then
            // each store instruction writes 4 whole 128-byte row segments.
            uint8_t *wb = sm + L::stage + (uint32_t)warp * 4096u;
            const int wrow0 = 32 * (warp % 4);              // the warp's first tile row
            T *obase = reinterpret_cast<T *>(a.out) +
                       ((size_t)(it.q_begin + it.t0 + x * it.rstep) * a.num_heads + (x ? it.h1 : it.h)) * D;
            const size_t rstride = (size_t)a.num_heads * D;
            // 32 output columns (unscaled) into the warp's buffer as 16-byte units
            auto stage_chunk = [&](int c, const uint32_t (&o)[32]) {
#pragma unroll
                for (int v = 0; v < 4; v++) {
                    uint4 w;
                    w.x = pack16<T>(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                    w.y = pack16<T>(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                    w.z = pack16<T>(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                    w.w = pack16<T>(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                    const int unit = 4 * c + v;
                    *reinterpret_cast<uint4 *>(wb + lane * 128 + ((unit ^ (lane & 7)) << 4)) = w;
                }
            };
            // the buffer's 32 rows of panel p to global memory, 4 whole 128-byte row segments per store
            auto store_panel = [&](int p) {
                __syncwarp();
#pragma unroll
                for (int qq = 0; qq < 8; qq++) {
                    const int lr = 4 * qq + (lane >> 3), unit = lane & 7;
                    const uint4 w = *reinterpret_cast<const uint4 *>(wb + lr * 128 + ((unit ^ (lr & 7)) << 4));
                    const int trow = m64 ? (lr < 16 ? 16 * (warp % 4) + lr : kRows) : wrow0 + lr;
                    if (trow < rows_x) *reinterpret_cast<uint4 *>(obase + (size_t)trow * rstride + 64 * p + 8 * unit) = w;
                }
                __syncwarp();
            };
            if (!split) {
                // each chunk's TMEM load is in flight while the previous chunk is staged and stored
                uint32_t ob[2][32];
                tc::tmem_ld32(tO, ob[0]);
#pragma unroll
                for (int q = 0; q < D / 32; q++) {
                    tc::tmem_wait_ld(ob[q & 1]);
                    if (q + 1 < D / 32) tc::tmem_ld32(tO + 32 * (q + 1), ob[(q + 1) & 1]);
                    stage_chunk(q & 1, ob[q & 1]);
                    if (q & 1) store_panel(q >> 1);
                }
            } else {
#pragma unroll 1
                for (int p = 0; p < NP; p++) {
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        uint32_t o[32];
                        load_out(64 * p + 32 * c, o);
                        stage_chunk(c, o);
                    }
                    store_panel(p);
                }
            }
            if (split) {
                // the other slot's O has been read: its softmax threads may go on
                tc::fence_before();
                mbar_arrive(&bars[bMerged]);
                um++;
            }
        }
        if (!ok && lane == 0) latch(st, kFlagTimeout, 2000000 + 1000 * k + j);
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
    // persistent CTAs, one per SM (each holds all of its SM's TMEM), at most one per item
    const int sms = sm_count();
    const int ctas = a.num_items < sms ? a.num_items : sms;
    return launch(kern, dim3((unsigned)(ctas > 0 ? ctas : 1)), dim3(kThreads), L::alloc, stream, a, tmq, tmk, tmv);
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status paged_attention_prefill(void *out, const void *query, const void *key_cache,
                                              const void *value_cache, const int32_t *block_tables,
                                              const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                                              int num_tokens, int max_query_len, int max_blocks_per_seq,
                                              int block_size, int num_blocks, int num_heads, int num_kv_heads,
                                              int head_dim, float scale, void *workspace, size_t workspace_bytes,
                                              pkv_dtype dtype, struct CUstream_st *stream) {
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
    if (workspace && (!aligned16(workspace) || workspace_bytes < kWsHeaderBytes))
        return fail(PKV_EINVAL, "paged_attention_prefill: workspace must be 16-byte aligned and at least %zu bytes",
                    kWsHeaderBytes);
    // grouped query heads share their kv head's tiles: pair the heads, not the rows
    const int group = num_heads / num_kv_heads;
    const bool head_pairs = group % 2 == 0;
    const int rows_per_item = head_pairs ? kRows : kTiles * kRows;
    const long long num_pairs = ((long long)max_query_len + rows_per_item - 1) / rows_per_item;
    const long long num_items = num_pairs * (head_pairs ? num_heads / 2 : num_heads) * num_seqs;
    if (num_items > INT_MAX / 2)
        return fail(PKV_EINVAL, "paged_attention_prefill: %lld work items (query tile pairs x heads x sequences) "
                                "above 2^30", num_items);
    DeviceStatus *st = status_ptr();
    if (!st) return fail(PKV_ECUDA, "paged_attention_prefill: no device status word");
    PrefillArgs a;
    a.out = out;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.status = st;
    a.hdr = reinterpret_cast<WsHeader *>(workspace);
    a.num_pairs = (int)num_pairs;
    a.head_pairs = head_pairs ? 1 : 0;
    a.num_items = (int)num_items;
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
