// Paged decode attention: block-table gather, QK scores, online softmax, PV,
// split into context partitions with a log-sum-exp merge.
//
// What it computes ("vLLM & PagedAttention: Efficient Memory Management for
// LLM Serving", §I attention equation and §III blockwise equation;
// "PagedAttention and vLLM, annotated" §4.1): for each sequence s and query
// head h, out = sum_t softmax_t(scale * q . k_t) v_t over the sequence's
// context, where token t lives in physical block block_tables[s][t / B] at
// offset t % B.  The result equals attention over a contiguous array.
//
// How (sm_103a):
//   * One CTA per (kv head x query-head tile, sequence, context partition).
//     A partition is P tokens (a multiple of 32); a sequence with one
//     partition writes its output directly, otherwise the CTA writes its
//     partition's (max, sum of exponentials, un-normalised PV) and a second
//     kernel merges the partitions.
//   * A producer warp walks the block table (32 entries per coalesced load)
//     and streams each 32-token stage of K and V -- whole blocks, or a
//     32-token slice of a larger block, contiguous in the cache layout
//     [NB][Hkv][B][d] -- into a shared-memory ring with 1-D bulk TMA copies
//     completing on mbarriers.
//   * Four consumer warps take stages round-robin.  In a stage each lane
//     holds a 16-byte chunk of a row (d/8 lanes per row); QK partial dots are
//     combined by a butterfly reduce-scatter so that each lane ends with the
//     score of one token; the online softmax keeps a running max and sum per
//     head in fp32 (log2 domain); PV accumulates fp32 per lane.  At the end
//     the four warps' states are merged through shared memory.
//   * All mbarrier waits are bounded; a wait that gives up latches a timeout
//     in the status word and the kernel drains its copies and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <array>
#include <cstring>
#include <map>
#include <mutex>
#include <type_traits>

#include "pkv_host.cuh"
#include "pkv_tmap.h"

namespace pkv {
namespace {

// Tuning knobs (compile-time): ring slots per consumer warp for head_dim 128
// and 64, and resident CTAs per SM of the persistent kernel.
#ifndef PKV_SLOTS_PER_WARP_D128
#define PKV_SLOTS_PER_WARP_D128 1
#endif
#ifndef PKV_SLOTS_PER_WARP_D64
#define PKV_SLOTS_PER_WARP_D64 2
#endif
#ifndef PKV_PERSISTENT_CTAS_PER_SM
#define PKV_PERSISTENT_CTAS_PER_SM 3
#endif
// tensor-core (query-head group) variant: consumer warps per CTA, ring slots
// per consumer warp, resident CTAs per SM
#ifndef PKV_MMA_CONSUMER_WARPS
#define PKV_MMA_CONSUMER_WARPS 1
#endif
#ifndef PKV_MMA_SLOTS_PER_WARP
#define PKV_MMA_SLOTS_PER_WARP 4
#endif
#ifndef PKV_MMA_CTAS_PER_SM
#define PKV_MMA_CTAS_PER_SM 3
#endif

// consumer warps per CTA of the CUDA-core variants
#ifndef PKV_SIMT_CONSUMER_WARPS
#define PKV_SIMT_CONSUMER_WARPS 4
#endif

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageRows = 32;              // tokens per ring stage
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

template <int D> struct Geometry {
    static constexpr int LPR = D / 8;       // lanes per row (16 bytes each)
    static constexpr int RPI = 32 / LPR;    // rows covered by one warp-wide load
    static constexpr int NI = kStageRows / RPI;   // loads per stage (== LPR)
    // Stage k goes to consumer warp k % W and ring slot k % NSTAGE.  NSTAGE is
    // a multiple of W, so every slot belongs to one warp, which waits for its
    // phases in order: a parity wait can never see a phase two ahead.
    static constexpr int SLOTS_PER_WARP = D >= 128 ? PKV_SLOTS_PER_WARP_D128 : PKV_SLOTS_PER_WARP_D64;
    static constexpr int NSTAGE = kConsumerWarps * SLOTS_PER_WARP;
    static constexpr int STAGE_ELEMS = kStageRows * D;   // per tensor
    static_assert(NSTAGE % kConsumerWarps == 0, "ring slots must divide among the consumer warps");
};

// CTAs per SM the register budget is sized for (shared memory allows 3).
template <int G> constexpr int min_ctas() { return G >= 4 ? 2 : 3; }
// Resident CTAs per SM of the persistent kernel (four query heads need the
// registers of two).
template <int G> constexpr int persistent_ctas() { return G >= 4 ? 2 : PKV_PERSISTENT_CTAS_PER_SM; }

template <int D, typename T> constexpr size_t smem_bytes() {
    using Gm = Geometry<D>;
    return (size_t)Gm::NSTAGE * 2 * Gm::STAGE_ELEMS * sizeof(T) + Gm::NSTAGE * 2 * sizeof(uint64_t) +
           Gm::NSTAGE * sizeof(int);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// v[0..N-1] held by each of N consecutive lanes (lane index c within the
// group).  Returns, on lane c, the sum over the group of v[c].
template <int N> __device__ __forceinline__ float reduce_scatter(float (&v)[N], int c) {
#pragma unroll
    for (int m = N / 2; m >= 1; m >>= 1) {
        const bool upper = (c & m) != 0;
#pragma unroll
        for (int j = 0; j < m; j++) {
            const float send = upper ? v[j] : v[j + m];
            const float keep = upper ? v[j + m] : v[j];
            v[j] = keep + __shfl_xor_sync(kFull, send, m);
        }
    }
    return v[0];
}

// One 32-token stage for G query heads.  Ks/Vs: [32][D] in shared memory.
template <int D, int G, typename T, bool FULL_STAGE>
__device__ __forceinline__ void consume_stage(const T *Ks, const T *Vs, int nvalid, int r, int c,
                                              const float (&qf)[G][8], float (&m)[G], float (&lsum)[G],
                                              float (&acc)[G][8]) {
    using Gm = Geometry<D>;
    constexpr int NI = Gm::NI, RPI = Gm::RPI, LPR = Gm::LPR;
    float part[G][NI];
#pragma unroll
    for (int i = 0; i < NI; i++) {
        const int row = i * RPI + r;
        const uint4 raw = *reinterpret_cast<const uint4 *>(Ks + row * D + c * 8);
        float kf[8];
        F16Traits<T>::to_f32(raw, kf);
#pragma unroll
        for (int h = 0; h < G; h++) {
            float a = qf[h][0] * kf[0];
#pragma unroll
            for (int e = 1; e < 8; e++) a = fmaf(qf[h][e], kf[e], a);
            part[h][i] = a;
        }
    }
    // lane (r, c) now owns token c * RPI + r of the stage
    const int myrow = c * RPI + r;
    float p[G];
#pragma unroll
    for (int h = 0; h < G; h++) {
        float sc = reduce_scatter<NI>(part[h], c);
        if (!FULL_STAGE && myrow >= nvalid) sc = -INFINITY;
        const float mnew = fmaxf(m[h], warp_max(sc));
        const float alpha = exp2f(m[h] - mnew);
        p[h] = exp2f(sc - mnew);
        lsum[h] = lsum[h] * alpha + p[h];
#pragma unroll
        for (int e = 0; e < 8; e++) acc[h][e] *= alpha;
        m[h] = mnew;
    }
#pragma unroll
    for (int i = 0; i < NI; i++) {
        const int row = i * RPI + r;
        const uint4 raw = *reinterpret_cast<const uint4 *>(Vs + row * D + c * 8);
        float vf[8];
        F16Traits<T>::to_f32(raw, vf);
        if (!FULL_STAGE && row >= nvalid) {
#pragma unroll
            for (int e = 0; e < 8; e++) vf[e] = 0.f;      // rows past the context may hold anything
        }
#pragma unroll
        for (int h = 0; h < G; h++) {
            const float w = __shfl_sync(kFull, p[h], r * LPR + i);
#pragma unroll
            for (int e = 0; e < 8; e++) acc[h][e] = fmaf(w, vf[e], acc[h][e]);
        }
    }
}

// The persistent kernel's CUDA-core stage: as consume_stage, but QK^T runs as
// fp32-accumulating FMAs straight on the 16-bit q and k values (no
// conversions; the score is scaled afterwards) and PV on pairs of fp32 lanes.
// qw[h][j] holds the two 16-bit query values j of the lane's chunk.
template <int D, int G, typename T, bool FULL_STAGE>
__device__ __forceinline__ void consume_stage_v2(const T *Ks, const T *Vs, int nvalid, int r, int c,
                                                 const uint32_t (&qw)[G][4], float scale_log2, float (&m)[G],
                                                 float (&lsum)[G], unsigned long long (&acc)[G][4]) {
    using Gm = Geometry<D>;
    constexpr int NI = Gm::NI, RPI = Gm::RPI, LPR = Gm::LPR;
    float part[G][NI];
#pragma unroll
    for (int i = 0; i < NI; i++) {
        const int row = i * RPI + r;
        const uint4 raw = *reinterpret_cast<const uint4 *>(Ks + row * D + c * 8);
        const uint32_t kw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int h = 0; h < G; h++) {
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < 4; j++) {
                a = fma_mixed<T>((unsigned short)(qw[h][j] & 0xffffu), (unsigned short)(kw[j] & 0xffffu), a);
                a = fma_mixed<T>((unsigned short)(qw[h][j] >> 16), (unsigned short)(kw[j] >> 16), a);
            }
            part[h][i] = a;
        }
    }
    const int myrow = c * RPI + r;
    float p[G];
#pragma unroll
    for (int h = 0; h < G; h++) {
        float sc = reduce_scatter<NI>(part[h], c) * scale_log2;
        if (!FULL_STAGE && myrow >= nvalid) sc = -INFINITY;
        const float mnew = fmaxf(m[h], warp_max(sc));
        const float alpha = exp2f(m[h] - mnew);
        p[h] = exp2f(sc - mnew);
        lsum[h] = lsum[h] * alpha + p[h];
        const unsigned long long a2 = pack2(alpha, alpha);
#pragma unroll
        for (int j = 0; j < 4; j++) acc[h][j] = mul2(acc[h][j], a2);
        m[h] = mnew;
    }
#pragma unroll
    for (int i = 0; i < NI; i++) {
        const int row = i * RPI + r;
        const uint4 raw = *reinterpret_cast<const uint4 *>(Vs + row * D + c * 8);
        float vf[8];
        F16Traits<T>::to_f32(raw, vf);
        if (!FULL_STAGE && row >= nvalid) {
#pragma unroll
            for (int e = 0; e < 8; e++) vf[e] = 0.f;      // rows past the context may hold anything
        }
        unsigned long long v2[4];
#pragma unroll
        for (int j = 0; j < 4; j++) v2[j] = pack2(vf[2 * j], vf[2 * j + 1]);
#pragma unroll
        for (int h = 0; h < G; h++) {
            const float w = __shfl_sync(kFull, p[h], r * LPR + i);
            const unsigned long long w2 = pack2(w, w);
#pragma unroll
            for (int j = 0; j < 4; j++) acc[h][j] = fma2(w2, v2[j], acc[h][j]);
        }
    }
}

// ---------------------------------------------------------------------------
// Tensor-core stage for query-head groups (GQA): the G heads of one kv head
// form the rows of a 16 x d query tile, so QK^T and PV become m16n8k16 MMAs
// (fp32 accumulation).  The K and V tiles come from tiled TMA copies with the
// 128-byte swizzle: a tile is [d/64 halves][32 tokens][64 elements], and the
// 16-byte chunk c of row r sits at chunk c ^ (r % 8), which keeps ldmatrix
// free of bank conflicts.
// ---------------------------------------------------------------------------

// Element offset of 16-byte chunk `chunk` (0 .. d/8-1) of token row `row`.
__device__ __forceinline__ int swz(int row, int chunk) {
    return (chunk >> 3) * (kStageRows * 64) + row * 64 + (((chunk & 7) ^ (row & 7)) << 3);
}

template <int D> struct MmaState {
    static constexpr int NT = D / 8;   // 8-wide column tiles of the output
    float o[NT][4];                    // rows lane/4 (c0, c1) and lane/4 + 8 (c2, c3, unused)
    float m;                           // running max of row lane/4 (log2 domain)
    float l;                           // this lane's share of the row's sum of exponentials
};

template <int D> __device__ __forceinline__ void mma_reset(MmaState<D> &st) {
#pragma unroll
    for (int n = 0; n < MmaState<D>::NT; n++)
#pragma unroll
        for (int e = 0; e < 4; e++) st.o[n][e] = 0.f;
    st.m = -INFINITY;
    st.l = 0.f;
}

// qa[ks] = (a0, a2) of k-step ks: query row lane/4 (zero past G heads);
// rows 8-15 of the tile (a1, a3) are zero.
template <int D, int G, typename T>
__device__ __forceinline__ void mma_load_q(uint32_t (&qa)[D / 16][2], const T *q, int lane) {
    const int row = lane >> 2, cq = lane & 3;
#pragma unroll
    for (int ks = 0; ks < D / 16; ks++) {
        if (row < G) {
            qa[ks][0] = *reinterpret_cast<const uint32_t *>(q + row * D + ks * 16 + cq * 2);
            qa[ks][1] = *reinterpret_cast<const uint32_t *>(q + row * D + ks * 16 + 8 + cq * 2);
        } else {
            qa[ks][0] = qa[ks][1] = 0u;
        }
    }
}

template <int D, typename T, bool FULL_STAGE>
__device__ __forceinline__ void consume_stage_mma(const T *Ks, T *Vs, int nvalid, int lane,
                                                  const uint32_t (&qa)[D / 16][2], MmaState<D> &st,
                                                  float scale_log2) {
    constexpr int NT = D / 8;
    const int cq = lane & 3;
    if (!FULL_STAGE) {
        // rows past the context may hold anything: zero them in V (0 * NaN would poison PV)
        for (int r = nvalid; r < kStageRows; r++)
            for (int e = lane * 8; e < D; e += 32 * 8)
                *reinterpret_cast<uint4 *>(Vs + (e >> 6) * (kStageRows * 64) + r * 64 + (e & 63)) =
                    make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
    }
    // S = Q K^T: 4 column tiles of 8 tokens
    // two accumulator sets (even and odd k-steps) halve the dependent MMA chain
    float s[4][4], s2[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) s[nt][e] = s2[nt][e] = 0.f;
#pragma unroll
    for (int kp = 0; kp < D / 32; kp++) {
#pragma unroll
        for (int nt = 0; nt < 4; nt++) {
            uint32_t b[4];
            ldmatrix_x4(b, Ks + swz(nt * 8 + (lane & 7), kp * 4 + (lane >> 3)));
            const uint32_t a0[4] = {qa[2 * kp][0], 0u, qa[2 * kp][1], 0u};
            const uint32_t a1[4] = {qa[2 * kp + 1][0], 0u, qa[2 * kp + 1][1], 0u};
            Mma<T>::run(s[nt], a0, b[0], b[1]);
            Mma<T>::run(s2[nt], a1, b[2], b[3]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < 4; nt++)
#pragma unroll
        for (int e = 0; e < 4; e++) s[nt][e] += s2[nt][e];
    // online softmax over the row's 8 tokens on this lane (a quad holds the row)
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
        x[j] = s[j >> 1][j & 1] * scale_log2;
        if (!FULL_STAGE && (j >> 1) * 8 + cq * 2 + (j & 1) >= nvalid) x[j] = -INFINITY;
    }
    float mx = x[0];
#pragma unroll
    for (int j = 1; j < 8; j++) mx = fmaxf(mx, x[j]);
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    const float mnew = fmaxf(st.m, mx);
    const float alpha = exp2f(st.m - mnew);
    float p[8], psum = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        p[j] = exp2f(x[j] - mnew);
        psum += p[j];
    }
    st.l = st.l * alpha + psum;
    st.m = mnew;
#pragma unroll
    for (int n = 0; n < NT; n++) {
        st.o[n][0] *= alpha;
        st.o[n][1] *= alpha;
    }
    // O += P V: the S accumulators of two column tiles are the A fragment of one k-step
#pragma unroll
    for (int kt = 0; kt < 2; kt++) {
        const uint32_t pa[4] = {Mma<T>::pack(p[4 * kt], p[4 * kt + 1]), 0u, Mma<T>::pack(p[4 * kt + 2], p[4 * kt + 3]),
                                0u};
        const int mi = lane >> 3;
        const int tok = kt * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int np = 0; np < NT / 2; np++) {
            uint32_t b[4];
            ldmatrix_x4_trans(b, Vs + swz(tok, 2 * np + (mi >> 1)));
            Mma<T>::run(st.o[2 * np], pa, b[0], b[1]);
            Mma<T>::run(st.o[2 * np + 1], pa, b[2], b[3]);
        }
    }
}

struct AttnArgs {
    void *out;                   // [S][H][D] T
    float *ws_m;                 // [S][H][MP]
    float *ws_l;                 // [S][H][MP]
    float *ws_o;                 // [S][H][MP][D]
    const void *q;               // [S][H][D]
    const void *k_cache;         // [NB][Hkv][B][D]
    const void *v_cache;
    const int32_t *tables;       // [S][max_blocks]
    const int32_t *ctx_lens;     // [S]
    DeviceStatus *st;
    WsHeader *hdr;               // work-ticket counters at the head of the workspace
    int num_seqs;
    int max_blocks;
    int max_ctx;
    int log2_block;
    int num_blocks;
    int num_heads;
    int num_kv_heads;
    int head_tiles;              // (H / Hkv) / G
    int partition;               // P
    int max_parts;               // MP
    float scale_log2;            // scale * log2(e)
    unsigned int *cnt;           // [S][H] partitions finished (fused merge); zero between calls
    int fused_merge;             // 1: the last partition of a (sequence, head tile) merges them all
    // the step's new tokens, written into the cache by the kernel (null: already written)
    const void *new_k;           // [S][Hkv][D]
    const void *new_v;
    const int64_t *slots;        // [S]
};

// Splits of up to this many partitions merge inside the attention kernel:
// the CTA that completes the last partition of a (sequence, query-head tile)
// -- found by an atomic counter -- merges them.  Longer splits go to
// partition_reduce_kernel.
#ifndef PKV_FUSED_MAX_PARTS
#define PKV_FUSED_MAX_PARTS 16
#endif
constexpr int kFusedMaxParts = PKV_FUSED_MAX_PARTS;
static_assert(kFusedMaxParts <= 32, "the in-kernel merge keeps one partition per lane");

// Log-sum-exp merge, by one warp, of the np partitions of query heads
// h0 .. h0 + G - 1 of sequence s (np <= 32, one per lane):
// M = max m_p, L = sum l_p 2^(m_p - M), out = sum o_p 2^(m_p - M) / L.
// Lane L owns D/32 consecutive elements of a row.  The partials were written
// by other CTAs: they are read past L1.  A head's m, l and first 8 rows are
// loaded together, so a head costs one round trip per 8 partitions.
template <int D, int G, typename T>
__device__ __forceinline__ void merge_partitions_warp(const AttnArgs &a, int s, int h0, int np, int lane) {
    constexpr int EPL = D / 32;
#pragma unroll 1
    for (int h = 0; h < G; h++) {
        const size_t base = ((size_t)s * a.num_heads + h0 + h) * a.max_parts;
        const float mp = lane < np ? __ldcg(a.ws_m + base + lane) : -INFINITY;
        const float lp = lane < np ? __ldcg(a.ws_l + base + lane) : 0.f;
        float acc[EPL];
#pragma unroll
        for (int k = 0; k < EPL; k++) acc[k] = 0.f;
        float wp = 0.f;
#pragma unroll 1
        for (int p0 = 0; p0 < np; p0 += 8) {
            float ov[8][EPL];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float *src = a.ws_o + (base + p0 + j) * D + lane * EPL;
                if (p0 + j < np) {
                    if constexpr (EPL == 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
                        ov[j][0] = v.x; ov[j][1] = v.y; ov[j][2] = v.z; ov[j][3] = v.w;
                    } else {
                        const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
                        ov[j][0] = v.x; ov[j][1] = v.y;
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < EPL; k++) ov[j][k] = 0.f;
                }
            }
            if (p0 == 0) {                       // uniform: the weights, while the first rows load
                const float M = warp_max(mp);
                wp = lane < np ? exp2f(mp - M) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const float w = __shfl_sync(kFull, wp, (p0 + j) & 31);
#pragma unroll
                for (int k = 0; k < EPL; k++) acc[k] = fmaf(w, ov[j][k], acc[k]);
            }
        }
        const float L = warp_sum(lp * wp);
        T *dst = static_cast<T *>(a.out) + ((size_t)s * a.num_heads + h0 + h) * D + lane * EPL;
#pragma unroll
        for (int k = 0; k < EPL; k++) dst[k] = F16Traits<T>::from_f32(L > 0.f ? acc[k] / L : 0.f);
    }
}

template <int D, int G, typename T>
__global__ void __launch_bounds__(kThreads, min_ctas<G>()) paged_attention_kernel(const AttnArgs a) {
    using Gm = Geometry<D>;
    constexpr int NSTAGE = Gm::NSTAGE, SE = Gm::STAGE_ELEMS, LPR = Gm::LPR;
    extern __shared__ __align__(128) unsigned char smem[];
    T *ring = reinterpret_cast<T *>(smem);                         // [NSTAGE][2][32][D]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NSTAGE * 2 * SE * sizeof(T));
    uint64_t *empty = full + NSTAGE;
    int *nvalid_s = reinterpret_cast<int *>(empty + NSTAGE);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.y, part = blockIdx.z;
    const int g = blockIdx.x / a.head_tiles;
    const int h0 = g * (a.head_tiles * G) + (blockIdx.x % a.head_tiles) * G;
    const int B = 1 << a.log2_block;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_mbar_init();
    }
    __shared__ int abort_cta;
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) abort_cta = timed_out(a.st);
    __syncthreads();
    if (abort_cta) return;                                       // an earlier wait gave up

    int ctx = a.ctx_lens[s];
    if (ctx < 0 || ctx > a.max_ctx) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && part == 0) latch(a.st, kFlagBadContext, ctx);
        ctx = ctx < 0 ? 0 : a.max_ctx;
    }
    const int nparts = (ctx + a.partition - 1) / a.partition;
    if (part >= (nparts > 1 ? nparts : 1)) return;                // uniform over the CTA
    const int tok0 = part * a.partition;
    const int ntok = ctx - tok0 < a.partition ? ctx - tok0 : a.partition;
    const int nstages = ntok > 0 ? (ntok + kStageRows - 1) / kStageRows : 0;

    if (warp == kConsumerWarps) {
        // ---------------- producer: block table -> bulk copies ----------------
        const T *kc = static_cast<const T *>(a.k_cache);
        const T *vc = static_cast<const T *>(a.v_cache);
        const int32_t *trow = a.tables + (size_t)s * a.max_blocks;
        const int nblk = (ctx + B - 1) >> a.log2_block;
        const int cps = B >= kStageRows ? 1 : kStageRows >> a.log2_block;   // copies per stage
        const int rows_per_copy = B >= kStageRows ? kStageRows : B;
        const uint32_t copy_bytes = (uint32_t)(rows_per_copy * D * sizeof(T));
        const uint64_t policy = policy_evict_first();
        int win = -(1 << 30), ent = -1;
        bool dead = false;
        for (int k = 0; k < nstages; k++) {
            const int t_first = tok0 + k * kStageRows;
            const int lb0 = t_first >> a.log2_block;
            const int off0 = t_first & (B - 1);                      // non-zero only when B > 32
            if (lb0 < win || lb0 + cps > win + 32) {
                win = lb0;
                const int j = win + lane;
                ent = j < nblk ? __ldg(trow + j) : -1;
            }
            int e[8];
#pragma unroll
            for (int j = 0; j < 8; j++) e[j] = __shfl_sync(kFull, ent, (lb0 + j - win) & 31);
            if (lane == 0) {
                const int slot = k % NSTAGE;
                if (k >= NSTAGE && !dead &&
                    !mbar_wait(&empty[slot], ((k / NSTAGE) - 1) & 1, kWaitLimitCycles)) {
                    latch(a.st, kFlagTimeout, k);
                    dead = true;
                }
                int nv = ntok - k * kStageRows < kStageRows ? ntok - k * kStageRows : kStageRows;
                int ncopies = 0;
                if (dead) {
                    nv = 0;
                } else {
                    for (int j = 0; j < cps && j < 8; j++) {
                        if (j * rows_per_copy >= nv) break;
                        const int p = e[j];
                        if (p < 0 || p >= a.num_blocks) {
                            latch(a.st, kFlagBadBlock, p);
                            nv = j * rows_per_copy;                  // stop the stage at the bad block
                            break;
                        }
                        ncopies = j + 1;
                    }
                }
                nvalid_s[slot] = nv;
                mbar_arrive_expect_tx(&full[slot], 2u * copy_bytes * (uint32_t)ncopies);
                for (int j = 0; j < ncopies; j++) {
                    const size_t goff = (((size_t)e[j] * a.num_kv_heads + g) * B + off0) * D;
                    T *dk = ring + (size_t)(slot * 2) * SE + (size_t)j * rows_per_copy * D;
                    bulk_g2s_hint(dk, kc + goff, copy_bytes, &full[slot], policy);
                    bulk_g2s_hint(dk + SE, vc + goff, copy_bytes, &full[slot], policy);
                }
            }
            __syncwarp();
        }
        return;
    }

    // ---------------- consumers ----------------
    const int r = lane / LPR, c = lane % LPR;
    float qf[G][8];
    {
        const T *qp = static_cast<const T *>(a.q) + ((size_t)s * a.num_heads + h0) * D + c * 8;
#pragma unroll
        for (int h = 0; h < G; h++) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(qp + (size_t)h * D);
            F16Traits<T>::to_f32(raw, qf[h]);
#pragma unroll
            for (int e = 0; e < 8; e++) qf[h][e] *= a.scale_log2;
        }
    }
    float m[G], lsum[G], acc[G][8];
#pragma unroll
    for (int h = 0; h < G; h++) {
        m[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; e++) acc[h][e] = 0.f;
    }
    bool dead = false;
    for (int k = warp; k < nstages; k += kConsumerWarps) {
        const int slot = k % NSTAGE;
        // warp-uniform, so that a give-up never splits the warp
        const bool ok = __all_sync(kFull, mbar_wait(&full[slot], (k / NSTAGE) & 1,
                                                    dead ? kDrainLimitCycles : kWaitLimitCycles));
        if (!ok && !dead) {
            if (lane == 0) latch(a.st, kFlagTimeout, k);
            dead = true;
        }
        if (!dead) {
            const int nv = nvalid_s[slot];
            const T *Ks = ring + (size_t)(slot * 2) * SE;
            if (nv == kStageRows)
                consume_stage<D, G, T, true>(Ks, Ks + SE, nv, r, c, qf, m, lsum, acc);
            else if (nv > 0)
                consume_stage<D, G, T, false>(Ks, Ks + SE, nv, r, c, qf, m, lsum, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ---------------- merge the consumer warps ----------------
#pragma unroll
    for (int h = 0; h < G; h++) {
        lsum[h] = warp_sum(lsum[h]);
#pragma unroll
        for (int e = 0; e < 8; e++) {
#pragma unroll
            for (int o = LPR; o < 32; o <<= 1) acc[h][e] += __shfl_xor_sync(kFull, acc[h][e], o);
        }
    }
    named_bar_sync(1, kConsumerWarps * 32);        // every stage consumed: the ring is free
    float *mw = reinterpret_cast<float *>(smem);   // [W][G]
    float *lw = mw + kConsumerWarps * G;           // [W][G]
    float *ow = lw + kConsumerWarps * G;           // [W][G][D]
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; h++) {
            mw[warp * G + h] = m[h];
            lw[warp * G + h] = lsum[h];
        }
    }
    if (r == 0) {
#pragma unroll
        for (int h = 0; h < G; h++)
#pragma unroll
            for (int e = 0; e < 8; e++) ow[(warp * G + h) * D + c * 8 + e] = acc[h][e];
    }
    named_bar_sync(1, kConsumerWarps * 32);
    for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
        const int h = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) M = fmaxf(M, mw[w * G + h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; w++) {
            const float mwv = mw[w * G + h];
            const float wt = mwv == -INFINITY ? 0.f : exp2f(mwv - M);
            L = fmaf(lw[w * G + h], wt, L);
            O = fmaf(ow[(w * G + h) * D + e], wt, O);
        }
        const size_t sh = (size_t)s * a.num_heads + h0 + h;
        if (nparts <= 1) {
            static_cast<T *>(a.out)[sh * D + e] = F16Traits<T>::from_f32(L > 0.f ? O / L : 0.f);
        } else {
            const size_t sp = sh * a.max_parts + part;
            a.ws_o[sp * D + e] = O;
            if (e == 0) {
                a.ws_m[sp] = M;
                a.ws_l[sp] = L;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Persistent variant.  One or two CTAs per SM stay resident and claim work
// items -- (sequence, partition, query-head tile), in that order -- with
// tickets from a counter at the head of the workspace.  Each CTA first turns
// the context lengths into a prefix sum of partitions per sequence in shared
// memory, so a ticket maps to a real item with one binary search and no
// empty CTA is ever launched.  The ring keeps streaming across items; an
// item's stages are padded to a multiple of the consumer-warp count so that
// every warp takes part in every item's merge, which goes through shared
// memory and an mbarrier (bounded waits only, no named barriers).
// ---------------------------------------------------------------------------

constexpr int kMaxPersistentSeqs = 4096;      // sequence tables kept in shared memory
constexpr size_t kMaxSmemPerCta = 227 * 1024;

enum : int { kMetaFirst = 1, kMetaLast = 2, kMetaStop = 4 };

struct StageMeta {
    int s, h0, part, nparts;  // the work item
    int nvalid;               // tokens in the stage (0: padding)
    int flags;                // kMeta*
    int qbuf;                 // query buffer of the item
    int pad;
};

// Shape of the persistent kernel: W consumer warps with R ring slots each
// (NSTAGE = W * R, so every slot belongs to one warp), one producer warp,
// CTAS resident CTAs per SM.
template <int D, int G, bool MMA> struct PConf {
    static constexpr int W = MMA ? PKV_MMA_CONSUMER_WARPS : PKV_SIMT_CONSUMER_WARPS;
    static constexpr int R = MMA ? PKV_MMA_SLOTS_PER_WARP : Geometry<D>::SLOTS_PER_WARP * kConsumerWarps / W;
    static constexpr int NSTAGE = W * R;
    static constexpr int THREADS = (W + 1) * 32;
    static constexpr int CTAS = MMA ? PKV_MMA_CTAS_PER_SM : persistent_ctas<G>();
};

template <int D, int G, typename T, bool MMA> struct PLayout {
    using C = PConf<D, G, MMA>;
    static constexpr int NQ = C::R;                                   // query buffers (see the producer)
    static constexpr size_t ring = 0;
    static constexpr size_t qs = ring + (size_t)C::NSTAGE * 2 * Geometry<D>::STAGE_ELEMS * sizeof(T);
    static constexpr size_t merge = qs + (size_t)NQ * C::W * G * D * sizeof(T);
    static constexpr size_t bars = merge + (size_t)2 * C::W * G * (D + 2) * sizeof(float);
    static constexpr size_t meta = bars + (size_t)(2 * C::NSTAGE + 2) * sizeof(uint64_t);
    static constexpr size_t misc = meta + (size_t)C::NSTAGE * sizeof(StageMeta);   // flags + scan scratch
    static constexpr size_t seqs = misc + 64 * sizeof(int);
    static size_t bytes(int S) { return seqs + (size_t)(2 * S + 1) * sizeof(int); }
};

// In place: v[1..n] := inclusive prefix sums of v[1..n]; v[0] := 0.
// warp_tot: shared scratch of one int per warp.
__device__ __forceinline__ void block_prefix_sum(int *v, int n, int *warp_tot) {
    const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int chunk = (n + nt - 1) / nt;
    const int b0 = tid * chunk < n ? tid * chunk : n;
    const int b1 = b0 + chunk < n ? b0 + chunk : n;
    int sum = 0;
    for (int i = b0; i < b1; i++) sum += v[i + 1];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    int off = 0;
    for (int w = 0; w < wid; w++) off += warp_tot[w];
    int run = off + incl - sum;
    for (int i = b0; i < b1; i++) {
        run += v[i + 1];
        v[i + 1] = run;
    }
    if (tid == 0) v[0] = 0;
    __syncthreads();
}

// A work item as the producer sees it.  ent holds, on lane j, block-table
// entry win + j of the item's sequence (-1 past its blocks).
struct Item {
    int s, part, nparts, g, h0, tok0, ntok, nst, npad, nblk, win, ent;
};

// Ticket t -> item: t / tiles indexes the partitions of all sequences in
// order (pref holds their prefix sums), t % tiles the query-head tile.
template <int G, int W>
__device__ __forceinline__ void decode_item(const AttnArgs &a, const int *pref, const int *ctxs, int S, int tiles,
                                            unsigned int t, int lane, Item &it) {
    const int pidx = (int)(t / (unsigned int)tiles);
    const int tile = (int)(t % (unsigned int)tiles);
    int lo = 0, hi = S;                                            // pref[lo] <= pidx < pref[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pref[mid] <= pidx) lo = mid; else hi = mid;
    }
    it.s = lo;
    it.part = pidx - pref[lo];
    it.nparts = pref[lo + 1] - pref[lo];
    it.g = tile / a.head_tiles;
    it.h0 = it.g * (a.head_tiles * G) + (tile % a.head_tiles) * G;
    const int ctx = ctxs[lo];
    it.tok0 = it.part * a.partition;
    int ntok = ctx - it.tok0 < a.partition ? ctx - it.tok0 : a.partition;
    it.ntok = ntok < 0 ? 0 : ntok;
    it.nst = (it.ntok + kStageRows - 1) / kStageRows;
    it.npad = ((it.nst > 0 ? it.nst : 1) + W - 1) / W * W;
    it.nblk = (ctx + (1 << a.log2_block) - 1) >> a.log2_block;
    it.win = it.tok0 >> a.log2_block;
    const int j = it.win + lane;
    it.ent = j < it.nblk ? __ldg(a.tables + (size_t)lo * a.max_blocks + j) : -1;
}

// MMA selects the tensor-core stage (query-head groups of 4 or 8) fed by
// tiled TMA copies through tmk / tmv; otherwise the CUDA-core stage fed by
// 1-D bulk copies (tmk / tmv unused).
template <int D, int G, typename T, bool MMA>
__global__ void __launch_bounds__(PConf<D, G, MMA>::THREADS, PConf<D, G, MMA>::CTAS)
    paged_attention_persistent_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                                      const __grid_constant__ CUtensorMap tmv) {
    using Gm = Geometry<D>;
    using L = PLayout<D, G, T, MMA>;
    using Cf = PConf<D, G, MMA>;
    constexpr int NSTAGE = Cf::NSTAGE, SE = Gm::STAGE_ELEMS, LPR = Gm::LPR, W = Cf::W;
    constexpr int NQ = L::NQ;
    // the 128-byte swizzle repeats every 1024 bytes: the ring starts on such a boundary
    extern __shared__ __align__(1024) unsigned char smem_p[];
    unsigned char *smem = smem_p;
    T *ring = reinterpret_cast<T *>(smem + L::ring);                 // [NSTAGE][2][32][D]
    T *qs = reinterpret_cast<T *>(smem + L::qs);                     // [NQ][W][G][D]
    float *mg = reinterpret_cast<float *>(smem + L::merge);          // [2][W][G][D + 2]: o, m, l
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bars);
    uint64_t *empty = full + NSTAGE;
    uint64_t *mbar = empty + NSTAGE;                                 // [2] item merges
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + L::meta);
    const int S = a.num_seqs;
    int *pref = reinterpret_cast<int *>(smem + L::seqs);             // [S + 1] partitions before s
    int *ctxs = pref + S + 1;                                        // [S]
    int &cta_flags = *reinterpret_cast<int *>(smem + L::misc);
    int *scan_tmp = reinterpret_cast<int *>(smem + L::misc) + 32;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = a.num_kv_heads * a.head_tiles;
    WsHeader *hdr = a.hdr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGE; i++) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&mbar[0], W * 32);
        mbar_init(&mbar[1], W * 32);
        fence_mbar_init();
    }
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0)
        cta_flags = (timed_out(a.st) ? 1 : 0) | (hdr->magic != kWsMagic ? 2 : 0) | ((smem_u32(smem) & 1023u) ? 4 : 0);
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
        int c = a.ctx_lens[i];
        if (c < 0 || c > a.max_ctx) {
            if (blockIdx.x == 0) latch(a.st, kFlagBadContext, c);
            c = c < 0 ? 0 : a.max_ctx;
        }
        ctxs[i] = c;
        pref[i + 1] = c > 0 ? (c + a.partition - 1) / a.partition : 1;
    }
    __syncthreads();
    if (cta_flags) {                                   // uniform over the CTA
        if ((cta_flags & 2) && blockIdx.x == 0 && threadIdx.x == 0) latch(a.st, kFlagBadWorkspace, hdr->magic);
        if ((cta_flags & 4) && blockIdx.x == 0 && threadIdx.x == 0) latch(a.st, kFlagTimeout, -2);
        return;
    }
    block_prefix_sum(pref, S, scan_tmp);
    const unsigned int N = (unsigned int)pref[S] * (unsigned int)tiles;
    const int B = 1 << a.log2_block;

    if (warp == W) {
        // ---------------- producer: tickets -> items -> bulk copies ----------------
        const T *kc = static_cast<const T *>(a.k_cache);
        const T *vc = static_cast<const T *>(a.v_cache);
        const T *qg = static_cast<const T *>(a.q);
        const int cps = B >= kStageRows ? 1 : kStageRows >> a.log2_block;
        const int rows_per_copy = B >= kStageRows ? kStageRows : B;
        const uint32_t copy_bytes = (uint32_t)(rows_per_copy * D * sizeof(T));
        const uint32_t q_bytes = (uint32_t)(G * D * sizeof(T));
        const uint64_t policy = policy_evict_first();
        // Tickets: the first item of CTA c is item c; later ones come from the
        // counter, offset by the grid size.  The next ticket is claimed two
        // stages before the current item's last stage, and decoded (its first
        // 32 block-table entries loaded) one stage later: late enough that a
        // CTA never holds a whole unstarted item when the pool runs dry, early
        // enough to hide the atomic and the block-table load.
        unsigned int cur_t = blockIdx.x;
        Item cur, nx;
        if (cur_t < N) decode_item<G, W>(a, pref, ctxs, S, tiles, cur_t, lane, cur);
        int kk = 0, items = 0;
        bool dead = false;
        while (cur_t < N && !dead) {
            unsigned int nxt_raw = 0, nxt_t = 0xffffffffu;
            bool claimed = false, decoded = false;
            const int s = cur.s, part = cur.part, nparts = cur.nparts, g = cur.g, h0 = cur.h0;
            const int tok0 = cur.tok0, ntok = cur.ntok, nst = cur.nst, npad = cur.npad, nblk = cur.nblk;
            const int32_t *trow = a.tables + (size_t)s * a.max_blocks;
            // Query buffer: written with the item's first W stages; with NQ =
            // NSTAGE / W buffers and every item at least W stages long, a
            // buffer is rewritten only after its previous item's first stages
            // have been consumed.
            const int qb = items % NQ;
            int win = cur.win, ent = cur.ent;
            if (a.new_k && part == nparts - 1) {
                // The step's new token of sequence s (position ctx - 1, in this partition): the
                // producer writes its key and value rows for kv head g into the cache, then makes
                // the writes visible to the copies below (every item that reads the slot writes it
                // first; items of other kv heads or partitions never read it).  That holds only for
                // the slot of position ctx - 1 in the sequence's own table, so any other slot is
                // latched and not written (it could race the copies of another item).
                constexpr int VEC = D * (int)sizeof(T) / 16;       // 16-byte vectors per row
                const long long slot = a.slots[s];
                if (slot >= 0) {                                    // uniform over the warp
                    const long long blk = slot >> a.log2_block;
                    const int pos = tok0 + ntok - 1;                // -1 for an empty context
                    const int lbl = pos >> a.log2_block;
                    int own = -1;                                   // the table's block of position pos
                    if (pos >= 0) {
                        const int ew = __shfl_sync(kFull, ent, (lbl - win) & 31);
                        own = lbl - win < 32 ? ew : __ldg(trow + lbl);
                    }
                    if (blk >= a.num_blocks) {
                        if (lane == 0) latch(a.st, kFlagBadSlot, slot);
                    } else if (pos < 0 || blk != (long long)own || (int)(slot & (B - 1)) != (pos & (B - 1))) {
                        if (lane == 0) latch(a.st, kFlagSlotNotLast, slot);
                    } else if (lane < 2 * VEC) {
                        const int off = (int)(slot & (B - 1));
                        const int v = lane % VEC;
                        const bool isv = lane >= VEC;
                        const uint4 *src = reinterpret_cast<const uint4 *>(isv ? a.new_v : a.new_k) +
                                           ((size_t)s * a.num_kv_heads + g) * VEC + v;
                        uint4 *dst = reinterpret_cast<uint4 *>(const_cast<void *>(isv ? a.v_cache : a.k_cache)) +
                                     (((size_t)blk * a.num_kv_heads + g) * B + off) * VEC + v;
                        *dst = __ldg(src);
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    }
                }
                __syncwarp();
            }
            const int i_claim = npad > 2 ? npad - 2 : 0, i_decode = npad > 1 ? npad - 1 : 0;
            for (int i = 0; i < npad; i++, kk++) {
                if (i == i_claim) {
                    if (lane == 0) nxt_raw = gridDim.x + atomicAdd(&hdr->next, 1u);
                    claimed = true;
                }
                if (i == i_decode) {
                    nxt_t = __shfl_sync(kFull, nxt_raw, 0);
                    if (nxt_t < N) decode_item<G, W>(a, pref, ctxs, S, tiles, nxt_t, lane, nx);
                    decoded = true;
                }
                const int slot = kk % NSTAGE;
                const bool withq = i < W && i < nst;               // warp i's first stage of the item
                // the stage's tokens, blocks and copies (the same on every lane)
                int nv = 0, nb = 0, off0 = 0, pj = -1;
                if (i < nst) {                                     // uniform over the warp
                    const int t_first = tok0 + i * kStageRows;
                    const int lb0 = t_first >> a.log2_block;
                    off0 = t_first & (B - 1);
                    nv = ntok - i * kStageRows < kStageRows ? ntok - i * kStageRows : kStageRows;
                    nb = (nv + rows_per_copy - 1) / rows_per_copy;
                    if (lb0 < win || lb0 + cps > win + 32) {
                        win = lb0;
                        const int j = win + lane;
                        ent = j < nblk ? __ldg(trow + j) : -1;
                    }
                    // this lane's block: lane >> 1 (bulk copies) or lane / (2 * halves) (tiled)
                    const int jl = MMA ? lane / (2 * (D / 64)) : lane >> 1;
                    pj = __shfl_sync(kFull, ent, (lb0 + jl - win) & 31);
                    const bool bad = jl < nb && (pj < 0 || pj >= a.num_blocks);
                    const unsigned badm = __ballot_sync(kFull, bad);
                    if (badm) {                                    // stop the stage at the first bad block
                        const int jb = MMA ? (__ffs(badm) - 1) / (2 * (D / 64)) : (__ffs(badm) - 1) >> 1;
                        if (lane == __ffs(badm) - 1) latch(a.st, kFlagBadBlock, pj);
                        nb = jb;
                        nv = jb * rows_per_copy;
                    }
                }
                if (kk >= NSTAGE &&
                    !__all_sync(kFull, mbar_wait(&empty[slot], ((kk / NSTAGE) - 1) & 1, kWaitLimitCycles))) {
                    if (lane == 0) latch(a.st, kFlagTimeout, kk);
                    dead = true;
                    break;
                }
                if (lane == 0) {
                    int4 *mv = reinterpret_cast<int4 *>(&meta[slot]);
                    mv[0] = make_int4(s, h0, part, nparts);
                    mv[1] = make_int4(nv, (i < W ? kMetaFirst : 0) | (i >= npad - W ? kMetaLast : 0), qb, 0);
                    mbar_arrive_expect_tx(&full[slot], 2u * copy_bytes * (uint32_t)nb + (withq ? q_bytes : 0u));
                }
                __syncwarp();
                if (MMA) {
                    // one tiled copy per lane: lane (2j + h) * 2 + t moves half h (64 elements of d)
                    // of block j's K (t = 0) or V (t = 1) tile; lane 0 also moves the query heads
                    constexpr int HALVES = D / 64;
                    if (lane < nb * HALVES * 2) {
                        const int t = lane & 1, h = (lane >> 1) % HALVES, j = (lane >> 1) / HALVES;
                        T *dst = ring + (size_t)(slot * 2 + t) * SE + h * (kStageRows * 64) + j * rows_per_copy * 64;
                        tma_load_4d(dst, t ? (const void *)&tmv : (const void *)&tmk, h * 64, off0, g, pj, &full[slot],
                                    policy);
                    }
                    if (withq && lane == 0)
                        bulk_g2s(qs + (size_t)(qb * W + i) * G * D, qg + ((size_t)s * a.num_heads + h0) * D, q_bytes,
                                 &full[slot]);
                } else {
                    // one bulk copy per lane: lane 2j moves block j's K tile, lane 2j+1 its V tile,
                    // lane 2 * nb the item's query heads
                    if (lane < 2 * nb) {
                        const int j = lane >> 1;
                        const size_t goff = (((size_t)pj * a.num_kv_heads + g) * B + off0) * D;
                        T *dst = ring + (size_t)(slot * 2 + (lane & 1)) * SE + (size_t)j * rows_per_copy * D;
                        bulk_g2s_hint(dst, ((lane & 1) ? vc : kc) + goff, copy_bytes, &full[slot], policy);
                    } else if (withq && lane == 2 * nb) {
                        bulk_g2s(qs + (size_t)(qb * W + i) * G * D, qg + ((size_t)s * a.num_heads + h0) * D, q_bytes,
                                 &full[slot]);
                    }
                }
            }
            if (dead) break;
            if (!claimed && lane == 0) nxt_raw = gridDim.x + atomicAdd(&hdr->next, 1u);
            if (!decoded) {
                nxt_t = __shfl_sync(kFull, nxt_raw, 0);
                if (nxt_t < N) decode_item<G, W>(a, pref, ctxs, S, tiles, nxt_t, lane, nx);
            }
            items++;
            cur_t = nxt_t;
            cur = nx;
        }
        if (lane == 0) {
            // one stop mark per consumer warp
            for (int w = 0; w < W && !dead; w++, kk++) {
                const int slot = kk % NSTAGE;
                if (kk >= NSTAGE && !mbar_wait(&empty[slot], ((kk / NSTAGE) - 1) & 1, kWaitLimitCycles)) {
                    latch(a.st, kFlagTimeout, kk);
                    dead = true;
                    break;
                }
                meta[slot].flags = kMetaStop;
                mbar_arrive_expect_tx(&full[slot], 0u);
            }
            // the last CTA to finish leaves the counters at zero for the next call
            __threadfence();
            if (atomicAdd(&hdr->done, 1u) == gridDim.x - 1) {
                hdr->next = 0;
                hdr->done = 0;
                __threadfence();
            }
        }
        return;
    }

    // ---------------- consumers ----------------
    const int r = lane / LPR, c = lane % LPR;
    uint32_t qw[G][4];                                 // CUDA-core stage state
    float m[G], lsum[G];
    unsigned long long acc[G][4];
    uint32_t qa[D / 16][2];                            // tensor-core stage state
    MmaState<D> ms;
    auto reset = [&]() {
        if constexpr (MMA) {
            mma_reset(ms);
        } else {
#pragma unroll
            for (int h = 0; h < G; h++) {
                m[h] = -INFINITY;
                lsum[h] = 0.f;
#pragma unroll
                for (int j = 0; j < 4; j++) acc[h][j] = 0ull;
            }
        }
    };
    reset();
    int jitem = 0;
    for (int k = warp;; k += W) {
        const int slot = k % NSTAGE;
        const bool ok = __all_sync(kFull, mbar_wait(&full[slot], (k / NSTAGE) & 1, kWaitLimitCycles));
        if (!ok) {
            if (lane == 0) latch(a.st, kFlagTimeout, k);
            break;
        }
        const StageMeta md = meta[slot];
        if (md.flags & kMetaStop) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            break;
        }
        const T *qp = qs + (size_t)(md.qbuf * W + warp) * G * D;
        T *Ks = ring + (size_t)(slot * 2) * SE;
        if constexpr (MMA) {
            if ((md.flags & kMetaFirst) && md.nvalid > 0) mma_load_q<D, G, T>(qa, qp, lane);
            if (md.nvalid == kStageRows) {
                consume_stage_mma<D, T, true>(Ks, Ks + SE, md.nvalid, lane, qa, ms, a.scale_log2);
            } else if (md.nvalid > 0) {
                consume_stage_mma<D, T, false>(Ks, Ks + SE, md.nvalid, lane, qa, ms, a.scale_log2);
                fence_proxy_async_smem();        // the zeroed rows, before TMA refills the slot
            }
        } else {
            if ((md.flags & kMetaFirst) && md.nvalid > 0) {
#pragma unroll
                for (int h = 0; h < G; h++) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(qp + h * D + c * 8);
                    qw[h][0] = raw.x;
                    qw[h][1] = raw.y;
                    qw[h][2] = raw.z;
                    qw[h][3] = raw.w;
                }
            }
            if (md.nvalid == kStageRows)
                consume_stage_v2<D, G, T, true>(Ks, Ks + SE, md.nvalid, r, c, qw, a.scale_log2, m, lsum, acc);
            else if (md.nvalid > 0)
                consume_stage_v2<D, G, T, false>(Ks, Ks + SE, md.nvalid, r, c, qw, a.scale_log2, m, lsum, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (!(md.flags & kMetaLast)) continue;

        // ---- the item's merge: this warp's state into buffer b, then W-way combine ----
        const int b = jitem & 1;
        float *mw = mg + (size_t)(b * W + warp) * G * (D + 2);
        if constexpr (MMA) {
            ms.l += __shfl_xor_sync(kFull, ms.l, 1);
            ms.l += __shfl_xor_sync(kFull, ms.l, 2);
            const int row = lane >> 2, cq = lane & 3;
            if (row < G) {
                float *mr = mw + row * (D + 2);
#pragma unroll
                for (int n = 0; n < D / 8; n++) {
                    mr[n * 8 + cq * 2] = ms.o[n][0];
                    mr[n * 8 + cq * 2 + 1] = ms.o[n][1];
                }
                if (cq == 0) {
                    mr[D] = ms.m;
                    mr[D + 1] = ms.l;
                }
            }
        } else {
            float accf[G][8];
#pragma unroll
            for (int h = 0; h < G; h++) {
                lsum[h] = warp_sum(lsum[h]);
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    accf[h][2 * j] = lo2(acc[h][j]);
                    accf[h][2 * j + 1] = hi2(acc[h][j]);
                }
#pragma unroll
                for (int e = 0; e < 8; e++) {
#pragma unroll
                    for (int o = LPR; o < 32; o <<= 1) accf[h][e] += __shfl_xor_sync(kFull, accf[h][e], o);
                }
            }
            if (r == 0) {
#pragma unroll
                for (int h = 0; h < G; h++)
#pragma unroll
                    for (int e = 0; e < 8; e++) mw[h * (D + 2) + c * 8 + e] = accf[h][e];
            }
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < G; h++) {
                    mw[h * (D + 2) + D] = m[h];
                    mw[h * (D + 2) + D + 1] = lsum[h];
                }
            }
        }
        mbar_arrive(&mbar[b]);                                   // every lane, after its own writes
        if (!__all_sync(kFull, mbar_wait(&mbar[b], (jitem >> 1) & 1, kWaitLimitCycles))) {
            if (lane == 0) latch(a.st, kFlagTimeout, -1 - jitem);
            break;
        }
        const float *mb = mg + (size_t)b * W * G * (D + 2);
        // one warp combines the item (round robin); the others go on.  Buffer b
        // is written again two items later, after the next item's barrier,
        // which this warp reaches only when the combine is done.
        if (warp == jitem % W) {
        for (int idx = lane; idx < G * D; idx += 32) {
            const int h = idx / D, e = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; w++) M = fmaxf(M, mb[(w * G + h) * (D + 2) + D]);
            float Lsum = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < W; w++) {
                const float *x = mb + (w * G + h) * (D + 2);
                const float wt = x[D] == -INFINITY ? 0.f : exp2f(x[D] - M);
                Lsum = fmaf(x[D + 1], wt, Lsum);
                O = fmaf(x[e], wt, O);
            }
            const size_t sh = (size_t)md.s * a.num_heads + md.h0 + h;
            if (md.nparts <= 1) {
                static_cast<T *>(a.out)[sh * D + e] = F16Traits<T>::from_f32(Lsum > 0.f ? O / Lsum : 0.f);
            } else {
                const size_t sp = sh * a.max_parts + md.part;
                a.ws_o[sp * D + e] = O;
                if (e == 0) {
                    a.ws_m[sp] = M;
                    a.ws_l[sp] = Lsum;
                }
            }
        }
        if (a.fused_merge && md.nparts > 1) {
            // count this partition in; the one that completes the set merges it
            __threadfence();
            __syncwarp();
            unsigned int done = 0;
            unsigned int *cnt = a.cnt + (size_t)md.s * a.num_heads + md.h0;
            if (lane == 0) done = atomicAdd(cnt, 1u);
            done = __shfl_sync(kFull, done, 0);
            if (done == (unsigned int)md.nparts - 1) {
                __threadfence();
                merge_partitions_warp<D, G, T>(a, md.s, md.h0, md.nparts, lane);
                if (lane == 0) *cnt = 0u;
            }
        }
        }
        jitem++;
        reset();
    }
}

// Merge the partitions of each (sequence, head) with more than one:
// M = max_p m_p, L = sum_p l_p 2^(m_p - M), out = sum_p o_p 2^(m_p - M) / L.
// One CTA per (head, sequence).  Thread t owns the 16-byte column t % CPR of
// the partial rows t / CPR, t / CPR + RG, ... of a chunk of RG * kReduceRows
// partitions: a chunk's rows are all requested at once, before the weights
// they need are known, so a split of up to one chunk (64 partitions at
// head_dim 128) costs about two round trips to L2.
constexpr int kReduceThreads = 256;
constexpr int kReduceRows = 8;                      // partial rows per thread per chunk

template <int D, typename T>
__global__ void __launch_bounds__(kReduceThreads) partition_reduce_kernel(const AttnArgs a) {
    constexpr int CPR = D / 4;                      // float4 columns per row
    constexpr int RG = kReduceThreads / CPR;        // row groups
    constexpr int CH = RG * kReduceRows;            // partitions per chunk
    static_assert(CH <= kReduceThreads, "one weight per thread and chunk");
    __shared__ float wsh[CH];
    __shared__ float red[2][kReduceThreads / 32];
    __shared__ float4 opart[RG][CPR];
    pdl_trigger();
    pdl_wait();
    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int ctx = a.ctx_lens[s];
    ctx = ctx < 0 ? 0 : (ctx > a.max_ctx ? a.max_ctx : ctx);
    const int np = (ctx + a.partition - 1) / a.partition;
    if (np <= 1) return;                            // uniform over the CTA
    const size_t base = ((size_t)s * a.num_heads + h) * a.max_parts;
    const float *m = a.ws_m + base;
    const float *l = a.ws_l + base;
    const float4 *o = reinterpret_cast<const float4 *>(a.ws_o + base * D);
    const int c = tid % CPR, rg = tid / CPR;
    float4 ov[kReduceRows];
    auto load_chunk = [&](int p0) {
#pragma unroll
        for (int k = 0; k < kReduceRows; k++) {
            const int p = p0 + rg + RG * k;
            ov[k] = p < np ? __ldcg(o + (size_t)p * CPR + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    // the first chunk's rows and the first kReduceThreads (m, l) are requested together
    load_chunk(0);
    const float m0 = tid < np ? __ldcg(m + tid) : -INFINITY;
    const float l0 = tid < np ? __ldcg(l + tid) : 0.f;
    float mx = m0;
    for (int p = tid + kReduceThreads; p < np; p += kReduceThreads) mx = fmaxf(mx, __ldcg(m + p));
    mx = warp_max(mx);
    if (lane == 0) red[0][wid] = mx;
    __syncthreads();
    float M = red[0][0];
#pragma unroll
    for (int w = 1; w < kReduceThreads / 32; w++) M = fmaxf(M, red[0][w]);
    const float w0 = tid < np ? exp2f(m0 - M) : 0.f;
    float lp = l0 * w0;
    for (int p = tid + kReduceThreads; p < np; p += kReduceThreads)
        lp = fmaf(__ldcg(l + p), exp2f(__ldcg(m + p) - M), lp);
    lp = warp_sum(lp);
    if (lane == 0) red[1][wid] = lp;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < np; p0 += CH) {
        if (p0 > 0) load_chunk(p0);
        if (tid < CH) wsh[tid] = p0 == 0 ? w0 : (p0 + tid < np ? exp2f(__ldcg(m + p0 + tid) - M) : 0.f);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kReduceRows; k++) {
            const float w = wsh[rg + RG * k];
            acc.x = fmaf(w, ov[k].x, acc.x);
            acc.y = fmaf(w, ov[k].y, acc.y);
            acc.z = fmaf(w, ov[k].z, acc.z);
            acc.w = fmaf(w, ov[k].w, acc.w);
        }
        __syncthreads();
    }
    opart[rg][c] = acc;
    __syncthreads();
    if (rg == 0) {
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kReduceThreads / 32; w++) L += red[1][w];
#pragma unroll
        for (int g = 1; g < RG; g++) {
            const float4 x = opart[g][c];
            acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
        }
        T *dst = static_cast<T *>(a.out) + ((size_t)s * a.num_heads + h) * D + c * 4;
        dst[0] = F16Traits<T>::from_f32(L > 0.f ? acc.x / L : 0.f);
        dst[1] = F16Traits<T>::from_f32(L > 0.f ? acc.y / L : 0.f);
        dst[2] = F16Traits<T>::from_f32(L > 0.f ? acc.z / L : 0.f);
        dst[3] = F16Traits<T>::from_f32(L > 0.f ? acc.w / L : 0.f);
    }
}

constexpr int kDefaultPartition = 512;

int parts_for(int max_ctx, int P) { return max_ctx > 0 ? (max_ctx + P - 1) / P : 1; }

// The default partition: 512 tokens at head_dim 128.  A head_dim-64 token is
// half the bytes, so 2048 tokens keep the bytes per work item up (measured on
// the 256-sequence Llama-2-7B-layer batch: +4 % at block size 16, +7 % at 64;
// flat at head_dim 128), halved down to 512 while that would leave fewer than
// 2048 work items (sequences x kv heads x partitions) for the persistent CTAs.
int choose_partition(int partition_size, int num_seqs, int num_kv_heads, int head_dim, int max_ctx) {
    if (partition_size > 0) return partition_size;
    int P = head_dim <= 64 ? 4 * kDefaultPartition : kDefaultPartition;
    while (P > kDefaultPartition && (long long)num_seqs * num_kv_heads * parts_for(max_ctx, P) < 2048) P /= 2;
    return P;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct WsLayout {
    size_t m_off, l_off, o_off, cnt_off, bytes;
};

// Workspace: the ticket header, then (when contexts may span partitions)
// m, l [S][H][MP], o [S][H][MP][D] and the merge counters [S][H], each
// region 256-byte aligned.
WsLayout ws_layout(int S, int H, int D, int MP) {
    WsLayout w{};
    w.bytes = kWsHeaderBytes;
    if (MP <= 1) return w;
    const size_t n = (size_t)S * H * MP;
    w.m_off = kWsHeaderBytes;
    w.l_off = w.m_off + align256(n * sizeof(float));
    w.o_off = w.l_off + align256(n * sizeof(float));
    w.cnt_off = w.o_off + align256(n * D * sizeof(float));
    w.bytes = w.cnt_off + align256((size_t)S * H * sizeof(unsigned int));
    return w;
}

// Zero the whole workspace, then mark the header initialised.
__global__ void workspace_init_kernel(uint4 *ws, size_t n16) {
    pdl_trigger();
    pdl_wait();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
        ws[i] = make_uint4(0u, 0u, 0u, 0u);
}

// The merge counters of a call sit after its partials, at offsets that
// depend on the call's sizes, so a region that one call used for partials may
// be another call's counters.  Every completed call leaves its own counters at
// zero; the library remembers, per workspace, the layout of the last call
// (a freshly initialised workspace is all zero) and zeroes the counter
// regions before a call whose layout differs.
using WsSig = std::array<int, 6>;                 // S, H, Hkv, D, MP, fused merge
const WsSig kWsClean = {0, 0, 0, 0, 0, 0};
std::mutex g_ws_mu;
std::map<std::pair<int, uintptr_t>, WsSig> g_ws_last;

int current_dev() {
    int d = -1;
    return cudaGetDevice(&d) == cudaSuccess ? d : -1;
}

// Workspaces remembered at most; past that the record starts afresh, and a
// workspace it has forgotten gets its counters zeroed once more (never wrong).
constexpr size_t kMaxRememberedWorkspaces = 4096;

void ws_remember(const void *ws, const WsSig &sig) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (g_ws_last.size() >= kMaxRememberedWorkspaces) g_ws_last.clear();
    g_ws_last[{current_dev(), reinterpret_cast<uintptr_t>(ws)}] = sig;
}

// True unless the workspace is known to hold zero counters for this layout.
bool ws_counters_stale(const void *ws, const WsSig &sig) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto it = g_ws_last.find({current_dev(), reinterpret_cast<uintptr_t>(ws)});
    return it == g_ws_last.end() || (it->second != sig && it->second != kWsClean);
}

__global__ void workspace_magic_kernel(WsHeader *h) {
    pdl_trigger();
    pdl_wait();
    h->magic = kWsMagic;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
// The cache [NB][Hkv][B][D] as a 4-D tensor (innermost first); a box is 64
// elements of d by min(B, 32) tokens of one (block, kv head), 128-byte swizzle.
bool encode_cache_map(CUtensorMap *map, const void *base, int num_blocks, int Hkv, int B, int D, bool bf16) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)B, (cuuint64_t)Hkv, (cuuint64_t)(num_blocks > 0 ? num_blocks : 1)};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)B * D * 2, (cuuint64_t)Hkv * B * D * 2};
    const cuuint32_t box[4] = {64u, (cuuint32_t)(B < kStageRows ? B : kStageRows), 1u, 1u};
    return encode_tiled16(map, base, 4, dims, strides, box, bf16);
}

template <int D, int G, typename T, bool MMA>
cudaError_t launch_persistent(const AttnArgs &a, dim3 grid, cudaStream_t st) {
    using Cf = PConf<D, G, MMA>;
    const size_t psmem = PLayout<D, G, T, MMA>::bytes(a.num_seqs);
    static size_t configured_p = 0;          // largest size set so far for this instance
    auto kern = paged_attention_persistent_kernel<D, G, T, MMA>;
    if (psmem > configured_p) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
        if (e != cudaSuccess) return e;
        configured_p = psmem;
    }
    CUtensorMap tmk, tmv;
    std::memset(&tmk, 0, sizeof tmk);
    std::memset(&tmv, 0, sizeof tmv);
    if (MMA) {
        const bool bf16 = sizeof(T) == 2 && std::is_same<T, __nv_bfloat16>::value;
        if (!encode_cache_map(&tmk, a.k_cache, a.num_blocks, a.num_kv_heads, 1 << a.log2_block, D, bf16) ||
            !encode_cache_map(&tmv, a.v_cache, a.num_blocks, a.num_kv_heads, 1 << a.log2_block, D, bf16))
            return cudaErrorInvalidValue;
    }
    // enough CTAs to fill the GPU, never more than there can be items
    const long long items = (long long)grid.x * grid.y * grid.z;
    long long ctas = (long long)sm_count() * Cf::CTAS;
    if (ctas > items) ctas = items;
    return launch(kern, dim3((unsigned)ctas), dim3(Cf::THREADS), psmem, st, a, tmk, tmv);
}

template <int D, int G, typename T> cudaError_t launch_attention(const AttnArgs &a, dim3 grid, cudaStream_t st) {
    if (a.num_seqs <= kMaxPersistentSeqs && PLayout<D, G, T, false>::bytes(a.num_seqs) <= kMaxSmemPerCta)
        return launch_persistent<D, G, T, false>(a, grid, st);
    static bool configured = false;
    auto kern = paged_attention_kernel<D, G, T>;
    const size_t smem = smem_bytes<D, T>();
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch(kern, grid, dim3(kThreads), smem, st, a);
}

// Query-head tile per CTA item for a group of `group` query heads per kv head:
// 8 or 4 heads go to the tensor-core stage, 2 or 1 to the CUDA-core stage
// (the grid kernel, used for very large batches, has the CUDA-core stage
// only and tiles at most 4 heads).
int head_tile(int group, bool persistent) {
    if (persistent && group % 8 == 0) return 8;
    if (group % 4 == 0) return 4;
    if (group % 2 == 0) return 2;
    return 1;
}

bool use_persistent(int num_seqs, int D, int G, int esize) {
    (void)esize;
    if (num_seqs > kMaxPersistentSeqs) return false;
    size_t need = 0;
    if (D == 64)
        need = G == 8   ? PLayout<64, 8, __half, true>::bytes(num_seqs)
               : G == 4 ? PLayout<64, 4, __half, true>::bytes(num_seqs)
                        : PLayout<64, 2, __half, false>::bytes(num_seqs);
    else
        need = G == 8   ? PLayout<128, 8, __half, true>::bytes(num_seqs)
               : G == 4 ? PLayout<128, 4, __half, true>::bytes(num_seqs)
                        : PLayout<128, 2, __half, false>::bytes(num_seqs);
    return need <= kMaxSmemPerCta;
}

template <int D, typename T> cudaError_t dispatch_g(int G, const AttnArgs &a, dim3 grid, cudaStream_t st) {
    const bool persistent = use_persistent(a.num_seqs, D, G, 2);
    if (persistent && G == 8) return launch_persistent<D, 8, T, true>(a, grid, st);
    if (persistent && G == 4) return launch_persistent<D, 4, T, true>(a, grid, st);
    switch (G) {
    case 4: return launch_attention<D, 4, T>(a, grid, st);
    case 2: return launch_attention<D, 2, T>(a, grid, st);
    default: return launch_attention<D, 1, T>(a, grid, st);
    }
}

template <typename T> cudaError_t dispatch_d(int D, int G, const AttnArgs &a, dim3 grid, cudaStream_t st) {
    return D == 64 ? dispatch_g<64, T>(G, a, grid, st) : dispatch_g<128, T>(G, a, grid, st);
}

template <typename T> cudaError_t launch_reduce(int D, const AttnArgs &a, dim3 grid, cudaStream_t st) {
    if (D == 64) return launch(partition_reduce_kernel<64, T>, grid, dim3(kReduceThreads), 0, st, a);
    return launch(partition_reduce_kernel<128, T>, grid, dim3(kReduceThreads), 0, st, a);
}

}  // namespace
}  // namespace pkv

extern "C" {

int paged_attention_partition_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                   int max_context_len, int partition_size) {
    (void)num_heads;
    return pkv::choose_partition(partition_size, num_seqs, num_kv_heads, head_dim, max_context_len);
}

pkv_status paged_attention_workspace_init(void *workspace, size_t workspace_bytes, struct CUstream_st *stream) {
    using namespace pkv;
    if (!workspace || workspace_bytes < kWsHeaderBytes || !aligned16(workspace))
        return fail(PKV_EINVAL, "paged_attention_workspace_init: need a 16-byte aligned workspace of at least %zu bytes",
                    kWsHeaderBytes);
    const size_t n16 = workspace_bytes / 16;
    long long blocks = (long long)((n16 + 255) / 256);
    const long long cap = (long long)sm_count() * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch(workspace_init_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                           static_cast<uint4 *>(workspace), n16);
    if (e == cudaSuccess)
        e = launch(workspace_magic_kernel, dim3(1), dim3(1), 0, stream, static_cast<WsHeader *>(workspace));
    if (e != cudaSuccess) return fail(PKV_ECUDA, "paged_attention_workspace_init: launch: %s", cudaGetErrorString(e));
    ws_remember(workspace, kWsClean);
    return PKV_OK;
}

size_t paged_attention_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                      int max_context_len, int partition_size) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0 || partition_size < 0)
        return 0;
    if (max_context_len == 0) return pkv::kWsHeaderBytes;
    const int P = paged_attention_partition_size(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len,
                                                 partition_size);
    return pkv::ws_layout(num_seqs, num_heads, head_dim, pkv::parts_for(max_context_len, P)).bytes;
}

}  // extern "C"

namespace pkv {
namespace {

pkv_status decode_impl(void *out, const void *query, const void *key_cache, const void *value_cache,
                       const int32_t *block_tables, const int32_t *context_lens, int num_seqs, int max_blocks_per_seq,
                       int max_context_len, int block_size, int num_blocks, int num_heads, int num_kv_heads,
                       int head_dim, float scale, int partition_size, void *workspace, size_t workspace_bytes,
                       pkv_dtype dtype, struct CUstream_st *stream, const void *new_k, const void *new_v,
                       const int64_t *slots) {
    if (dtype != PKV_F16 && dtype != PKV_BF16) return fail(PKV_EINVAL, "paged_attention_decode: bad dtype %d", (int)dtype);
    if (num_seqs < 0 || num_seqs > 65535 || max_blocks_per_seq < 0 || num_blocks < 0)
        return fail(PKV_EINVAL, "paged_attention_decode: bad sizes (seqs %d, table width %d, blocks %d)", num_seqs,
                    max_blocks_per_seq, num_blocks);
    if (head_dim != 64 && head_dim != 128)
        return fail(PKV_EINVAL, "paged_attention_decode: head_dim %d not supported (64 or 128)", head_dim);
    if (!is_pow2(block_size) || block_size < 4 || block_size > 128)
        return fail(PKV_EINVAL, "paged_attention_decode: block_size %d not a power of two in [4, 128]", block_size);
    if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads)
        return fail(PKV_EINVAL, "paged_attention_decode: %d query heads do not group over %d kv heads", num_heads,
                    num_kv_heads);
    if (partition_size < 0 || partition_size % kStageRows)
        return fail(PKV_EINVAL, "paged_attention_decode: partition_size %d not a multiple of %d", partition_size,
                    kStageRows);
    const int64_t table_cap = (int64_t)max_blocks_per_seq * block_size;
    if (max_context_len < 0 || max_context_len > table_cap)
        return fail(PKV_EINVAL, "paged_attention_decode: max_context_len %d beyond the table (%lld tokens)",
                    max_context_len, (long long)table_cap);
    if (num_seqs == 0) return PKV_OK;
    const int max_ctx = max_context_len > 0 ? max_context_len : (int)(table_cap > INT32_MAX ? INT32_MAX : table_cap);
    if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens)
        return fail(PKV_EINVAL, "paged_attention_decode: NULL pointer");
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
        return fail(PKV_EINVAL, "paged_attention_decode: pointers must be 16-byte aligned");
    const int P = choose_partition(partition_size, num_seqs, num_kv_heads, head_dim, max_ctx);
    const int MP = parts_for(max_ctx, P);
    if (MP > 65535) return fail(PKV_EINVAL, "paged_attention_decode: %d partitions per sequence", MP);
    const WsLayout wl = ws_layout(num_seqs, num_heads, head_dim, MP);
    if (!workspace || workspace_bytes < wl.bytes || !aligned16(workspace))
        return fail(PKV_EINVAL, "paged_attention_decode: workspace of %zu bytes needed, %zu given", wl.bytes,
                    workspace ? workspace_bytes : (size_t)0);
    DeviceStatus *st = status_ptr();
    if (!st) return fail(PKV_ECUDA, "paged_attention_decode: no device status word");

    const int group = num_heads / num_kv_heads;
    int G = head_tile(group, true);
    const bool persistent = use_persistent(num_seqs, head_dim, G, 2);
    if (!persistent) G = head_tile(group, false);
    if (new_k && !persistent) {
        // the grid kernel has no fused write: write first, then attend
        const pkv_status ws_ = kv_reshape_and_cache(new_k, new_v, const_cast<void *>(key_cache),
                                                    const_cast<void *>(value_cache), slots, num_seqs, num_kv_heads,
                                                    head_dim, block_size, num_blocks, dtype, stream);
        if (ws_ != PKV_OK) return ws_;
        new_k = new_v = nullptr;
        slots = nullptr;
    }
    AttnArgs a;
    a.new_k = new_k;
    a.new_v = new_v;
    a.slots = slots;
    a.out = out;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    a.hdr = reinterpret_cast<WsHeader *>(ws);
    a.ws_m = MP > 1 ? reinterpret_cast<float *>(ws + wl.m_off) : nullptr;
    a.ws_l = MP > 1 ? reinterpret_cast<float *>(ws + wl.l_off) : nullptr;
    a.ws_o = MP > 1 ? reinterpret_cast<float *>(ws + wl.o_off) : nullptr;
    a.cnt = MP > 1 ? reinterpret_cast<unsigned int *>(ws + wl.cnt_off) : nullptr;
    a.num_seqs = num_seqs;
    a.q = query;
    a.k_cache = key_cache;
    a.v_cache = value_cache;
    a.tables = block_tables;
    a.ctx_lens = context_lens;
    a.st = st;
    a.max_blocks = max_blocks_per_seq;
    a.max_ctx = max_ctx;
    a.log2_block = ilog2(block_size);
    a.num_blocks = num_blocks;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_tiles = group / G;
    a.partition = P;
    a.max_parts = MP;
    a.scale_log2 = scale * kLog2e;
    a.fused_merge = persistent && MP > 1 && MP <= kFusedMaxParts;

    const dim3 grid((unsigned)(num_kv_heads * a.head_tiles), (unsigned)num_seqs, (unsigned)MP);
    const WsSig sig = {num_seqs, num_heads, num_kv_heads, head_dim, MP, a.fused_merge};
    cudaError_t e = cudaSuccess;
    if (a.fused_merge && ws_counters_stale(workspace, sig)) {
        // the counter regions (16-byte multiples: every region is 256-byte aligned)
        const size_t n16 = (wl.bytes - wl.cnt_off) / 16;
        long long blocks = (long long)((n16 + 255) / 256);
        if (blocks > sm_count()) blocks = sm_count() > 0 ? sm_count() : 1;
        e = launch(workspace_init_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                   reinterpret_cast<uint4 *>(ws + wl.cnt_off), n16);
        if (e != cudaSuccess) return fail(PKV_ECUDA, "paged_attention_decode: counter reset: %s", cudaGetErrorString(e));
    }
    e = dtype == PKV_F16 ? dispatch_d<__half>(head_dim, G, a, grid, stream)
                         : dispatch_d<__nv_bfloat16>(head_dim, G, a, grid, stream);
    if (e != cudaSuccess) return fail(PKV_ECUDA, "paged_attention_decode: launch: %s", cudaGetErrorString(e));
    ws_remember(workspace, sig);
    if (MP > 1 && !a.fused_merge) {
        const dim3 rgrid((unsigned)num_heads, (unsigned)num_seqs);
        e = dtype == PKV_F16 ? launch_reduce<__half>(head_dim, a, rgrid, stream)
                             : launch_reduce<__nv_bfloat16>(head_dim, a, rgrid, stream);
        if (e != cudaSuccess) return fail(PKV_ECUDA, "paged_attention_decode: reduce launch: %s", cudaGetErrorString(e));
    }
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" {

pkv_status paged_attention_decode(void *out, const void *query, const void *key_cache, const void *value_cache,
                                  const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                                  int max_blocks_per_seq, int max_context_len, int block_size, int num_blocks,
                                  int num_heads, int num_kv_heads, int head_dim, float scale, int partition_size,
                                  void *workspace, size_t workspace_bytes, pkv_dtype dtype,
                                  struct CUstream_st *stream) {
    return pkv::decode_impl(out, query, key_cache, value_cache, block_tables, context_lens, num_seqs,
                            max_blocks_per_seq, max_context_len, block_size, num_blocks, num_heads, num_kv_heads,
                            head_dim, scale, partition_size, workspace, workspace_bytes, dtype, stream, nullptr,
                            nullptr, nullptr);
}

pkv_status paged_attention_decode_write(void *out, const void *query, const void *key, const void *value,
                                        void *key_cache, void *value_cache, const int64_t *slot_mapping,
                                        const int32_t *block_tables, const int32_t *context_lens, int num_seqs,
                                        int max_blocks_per_seq, int max_context_len, int block_size, int num_blocks,
                                        int num_heads, int num_kv_heads, int head_dim, float scale,
                                        int partition_size, void *workspace, size_t workspace_bytes, pkv_dtype dtype,
                                        struct CUstream_st *stream) {
    using namespace pkv;
    if (num_seqs > 0 && (!key || !value || !slot_mapping))
        return fail(PKV_EINVAL, "paged_attention_decode_write: NULL key, value or slot_mapping");
    if (num_seqs > 0 && (!aligned16(key) || !aligned16(value)))
        return fail(PKV_EINVAL, "paged_attention_decode_write: key and value must be 16-byte aligned");
    return decode_impl(out, query, key_cache, value_cache, block_tables, context_lens, num_seqs, max_blocks_per_seq,
                       max_context_len, block_size, num_blocks, num_heads, num_kv_heads, head_dim, scale,
                       partition_size, workspace, workspace_bytes, dtype, stream, key, value, slot_mapping);
}

}  // extern "C"
