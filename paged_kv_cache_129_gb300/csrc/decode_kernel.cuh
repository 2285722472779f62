// Paged decode attention kernel (one CTA per (sequence, kv head, head chunk,
// partition)) and the split-KV merge kernel.
//
// The method (MiniPaged-Qwen, sections 5.1-5.2 and 6.2): for every logical
// position pos of the context, pb = block_table[pos / bs] and the key/value
// rows are key_cache[pb, kvh, pos % bs, :]; scores s = scale * q.k are
// normalised over the whole context with a running maximum m, a running
// denominator l and an unnormalised output o~ (online softmax):
//     m' = max(m, max s),  l' = l * 2^(m - m') + sum 2^(s - m'),
//     o~' = o~ * 2^(m - m') + sum 2^(s - m') v,    o = o~ / l.
// (Scores are kept in the log2 domain: s is pre-multiplied by log2(e), so
// 2^(s - m) equals the page's e^(s - m).)  GQA: kv head kvh serves the query
// heads kvh*g .. kvh*g + g - 1 (section 9.1), so one CTA reads every K/V page
// once for all of them.  Long contexts are cut into partitions of
// `partition_pages` pages (the "partitioned reduction" of section 10.2); each
// partition emits (m, l, o~) and the merge kernel combines them with the same
// rescaling rule.
//
// CTA layout: warps 0..NW-1 consume pages, warp NW produces them.  The
// producer reads the block-table entries of its partition (one 32-entry chunk
// ahead, through registers) and issues TMA tile loads of each page's K and V
// slices ([pb, kvh, :, :] is bs * d contiguous elements) into a shared-memory
// ring of NSLOT page slots; every page's arrival is tracked by an mbarrier
// with transaction bytes.  Page i lands in slot i % NSLOT and is consumed by
// warp i % NW, which then releases the slot.  Tiles are 128-byte-swizzled so
// that the consumers' shared-memory reads are free of bank conflicts.
//
// Consumers:
//  * tensor-core path (f16/bf16): per 16-token sub-tile,
//      S[16 heads x 8 tok]  = Q[16 x d] . K^T   (m16n8k16, heads padded to 16)
//      O^T[16 d x 8 heads] += V^T[16 x 16 tok] . P^T[16 tok x 8 heads]
//    The fp32 score fragment of QK^T is exactly the B fragment PV needs, so
//    P never goes through shared memory.
//  * CUDA-core path (all dtypes): one or two lanes per token for QK^T (q in
//    shared memory as fp32), one lane per d-slice for PV.
#pragma once

#include <atomic>

#include <cfloat>
#include <type_traits>

#include <cuda_fp8.h>

#include "decode_launch.h"
#include "pa_common.cuh"

// Lean-kernel tuning knobs (compile time): resident CTAs per SM the register
// allocation must allow, and the page ring per CTA in KB.
#ifndef PA_LEAN_MIN_BLOCKS
#define PA_LEAN_MIN_BLOCKS 3
#endif
#ifndef PA_LEAN_RING_KB
#define PA_LEAN_RING_KB 64
#endif
// Resident lean CTAs per SM the FP8 kernel's register allocation aims for.
#ifndef PA_LEAN_F8_MIN_BLOCKS
#define PA_LEAN_F8_MIN_BLOCKS 3
#endif
// Prefetch the context lengths and block tables into L2 before the lean kernel's dependency wait.
#ifndef PA_LEAN_L2_PREFETCH
#define PA_LEAN_L2_PREFETCH 1
#endif
// Idle nap of the lean producer lane between polls of its warps' slots (ns): every poll takes
// issue slots from the consumers that share its SM sub-partition.
#ifndef PA_PRODUCER_NAP_NS
#define PA_PRODUCER_NAP_NS 20
#endif

namespace pa {

constexpr int kConsumerWarps = 4;

template <typename T, int D, int BS, bool MMA, int GMAX>
struct DecodeCfg {
    static constexpr int kEB = sizeof(T);
    static constexpr int kNW = kConsumerWarps;
    static constexpr int kThreads = (kNW + 1) * 32;
    static constexpr int kBoxElems = 128 / kEB;           // one 128-byte swizzle row of d
    static constexpr int kNBox = D / kBoxElems;           // boxes per page
    static constexpr int kBoxBytes = BS * 128;            // BS rows of 128 bytes
    static constexpr int kPageBytes = kNBox * kBoxBytes;  // = BS * D * sizeof(T)
    static constexpr int kSlotBytes = 2 * kPageBytes;     // K page + V page
    static constexpr int kRingTarget = 64 * 1024;
    static constexpr int kNSlotRaw = (kRingTarget / kSlotBytes) / kNW * kNW;
    static constexpr int kNSlot = kNSlotRaw < kNW ? kNW : kNSlotRaw;
    static constexpr int kRingBytes = kNSlot * kSlotBytes;
    static constexpr int kHeads = MMA ? 8 : GMAX;          // query heads per CTA
    static constexpr int kOStride = D + 4;                 // padded fp32 row of the combine buffer
    static constexpr int kCombineFloats = kNW * kHeads * kOStride + 2 * kNW * kHeads;
    static constexpr int a16(int x) { return (x + 15) & ~15; }
    static constexpr int kBarOffset = kRingBytes;
    static constexpr int kIssuedOffset = a16(kBarOffset + 2 * kNSlot * 8);
    static constexpr int kQsOffset = a16(kIssuedOffset + kNSlot * 4);
    static constexpr int kQsBytes = MMA ? 0 : GMAX * D * 4;
    static constexpr int kPsOffset = a16(kQsOffset + kQsBytes);
    static constexpr int kPsBytes = MMA ? 0 : kNW * GMAX * BS * 4;
    static constexpr int kStatOffset = a16(kPsOffset + kPsBytes);  // per head: M, W, then per-warp weights
    static constexpr int kStatBytes = kHeads * (2 + kNW) * 4;
    static constexpr int kFlagOffset = a16(kStatOffset + kStatBytes);
    static constexpr int kSmemBytes = kFlagOffset + 16 + 1024;  // + slack to align the base to 1024
    // Resident CTAs per SM the register allocation must allow (0: no bound).  Registers are
    // split between the SM's four sub-partitions, so three CTAs of five warps need <= 128 per
    // thread.  The 16-token page kernels stay under that unbounded (an explicit bound of 1 makes
    // the compiler take ~137); the 32-token ones (two sub-tiles per page) would take ~135 and
    // lose a CTA per SM; head_dim 256 needs ~200 (two CTAs per SM).
    static constexpr int kMinBlocks = (D <= 128 && BS == 32) ? 3 : 0;

    static_assert(D % kBoxElems == 0, "head_dim must be a multiple of 128 bytes");
    static_assert(BS <= 256 && BS >= 8, "TMA box height");
    static_assert(!MMA || BS % 16 == 0, "the tensor-core path needs 16-token sub-tiles");
    static_assert(!MMA || D % 16 == 0, "k-steps of 16");
    static_assert(MMA || (32 % BS == 0 || BS == 32), "CUDA-core path: 32 must be a multiple of BS");
    static_assert(kCombineFloats * 4 <= kRingBytes, "combine buffer must fit in the ring");
    static_assert(kQsOffset % 16 == 0 && kPsOffset % 16 == 0, "float4 access to q_s");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

// Byte offset of (row, element) in a 128-byte-swizzled page of kNBox boxes.
template <typename T, int BS>
__device__ __forceinline__ uint32_t swz_offset(int row, int elem) {
    constexpr int kBoxElems = 128 / sizeof(T);
    const int box = elem / kBoxElems;
    const int byte = (elem % kBoxElems) * (int)sizeof(T);
    const int chunk = byte >> 4;
    return (uint32_t)(box * BS * 128 + row * 128 + (((chunk ^ (row & 7)) << 4) | (byte & 15)));
}

// ------------------------------------------------------------------------------------------
// Query and output rows of a unit.  A kv head serves rows = q_len * group query rows; row
// v = t * group + h is query token t (position L - q_len + t) of head kvh * group + h, and
// query / out are [B, q_len, H_q, D] (q_len = 1: [B, H_q, D]).  Row r of a unit is row
// v0 + r of its kv head.
struct UnitRows {
    int b, kvh, v0, q_len, group, num_heads;
    __device__ __forceinline__ size_t row(int r) const {
        const int v = v0 + r;
        const int t = v / group;
        return ((size_t)b * q_len + t) * num_heads + kvh * group + (v - t * group);
    }
    // The last position row r attends (causal bound), for a context of L positions.
    __device__ __forceinline__ int last_pos(int r, int L) const { return L - q_len + (v0 + r) / group; }
};

// Weight of a state whose running max is m against a common max mm: 0 for an empty state
// (m = -inf), also when every state is empty (mm = -inf).
__device__ __forceinline__ float rescale(float m, float mm) { return m == -INFINITY ? 0.f : exp2f(m - mm); }

// ------------------------------------------------------------------------------------------
// The step's new token in append mode.  Its K and V rows (D elements each) are held by
// one warp as 16-byte chunks: chunks 0..kChunks-1 of K, then those of V, lane-strided.
// The warp that consumes the page holding position L - 1 overwrites that row of its
// staged K and V tiles (so the page need not be re-read after the cache write) and, for
// one head chunk of the kv head, stores the rows into the cache: the same bytes
// pa_write_kv would store, with the slot the block table gives position L - 1.
template <typename T, int D, int BS>
struct NewToken {
    static constexpr int kChunks = D * (int)sizeof(T) / 16;      // 16-byte chunks per row
    static constexpr int kPerLane = (2 * kChunks + 31) / 32;
    uint4 c[kPerLane];

    // key_row, value_row: new_key[b, kvh, :], new_value[b, kvh, :] (16-byte aligned).
    __device__ __forceinline__ void load(const T* key_row, const T* value_row, int lane) {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int idx = lane + 32 * i;
            if (idx < kChunks)
                c[i] = __ldg(reinterpret_cast<const uint4*>(key_row) + idx);
            else if (idx < 2 * kChunks)
                c[i] = __ldg(reinterpret_cast<const uint4*>(value_row) + idx - kChunks);
        }
    }

    // Overwrite row r of the 128-byte-swizzled K and V tiles; then order these generic
    // writes before the async-proxy (TMA) writes that will later refill the slot.
    __device__ __forceinline__ void patch(uint8_t* kpage, uint8_t* vpage, int r, int lane) const {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int idx = lane + 32 * i;
            if (idx < 2 * kChunks) {
                const int ch = idx < kChunks ? idx : idx - kChunks;
                uint8_t* tile = idx < kChunks ? kpage : vpage;
                const int box = ch >> 3, cc = ch & 7;
                *reinterpret_cast<uint4*>(tile + box * BS * 128 + r * 128 + ((cc ^ (r & 7)) << 4)) = c[i];
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
    }

    // Store the rows at cache row `row` = (pb * Hkv + kvh) * BS + r of both caches.
    __device__ __forceinline__ void store(void* key_cache, void* value_cache, int row, int lane) const {
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int idx = lane + 32 * i;
            if (idx < kChunks)
                reinterpret_cast<uint4*>(static_cast<T*>(key_cache) + (size_t)row * D)[idx] = c[i];
            else if (idx < 2 * kChunks)
                reinterpret_cast<uint4*>(static_cast<T*>(value_cache) + (size_t)row * D)[idx - kChunks] = c[i];
        }
    }
};

// Partitioned-grid kernel: fetch the new token of (b, kvh) and put it into the staged page
// `lb` (the page holding position L - 1; nvalid of its rows are in the context), and, for
// head chunk 0, into the cache at the slot the block table gives.
template <typename T, int D, int BS>
__device__ __noinline__ void append_token(const DecodeArgs& a, int b, int kvh, int hc, int lb, uint8_t* kpage,
                                          uint8_t* vpage, int nvalid, int lane) {
    NewToken<T, D, BS> tok;
    const size_t nt = ((size_t)b * a.num_kv_heads + kvh) * D;
    tok.load(static_cast<const T*>(a.new_key) + nt, static_cast<const T*>(a.new_value) + nt, lane);
    tok.patch(kpage, vpage, nvalid - 1, lane);
    if (hc != 0) return;
    const int pb = __ldg(a.block_tables + (size_t)b * a.max_blocks + lb);
    if ((unsigned)pb < (unsigned)a.num_blocks) tok.store(a.key_cache, a.value_cache, (pb * a.num_kv_heads + kvh) * BS + nvalid - 1, lane);
}

// ------------------------------------------------------------------------------------------
// Tensor-core consumer (f16 / bf16).
// CAUSAL: rows carry their own causal bound (multi-query decode); without it every row
// attends the whole context and the bound checks compile away.
//
// Both products keep the page's tokens or head dimensions on the M side of m16n8k16 and the
// (up to) 8 query rows on the N side, so no half of an operand is padding:
//  * S^T = K Q^T: A = 16 tokens x 16 dims of K (ldmatrix), B = Q^T (lane g holds query row g);
//    the accumulator gives lane (g, t) tokens g, g + 8 of query rows 2t, 2t + 1.
//  * O^T += V^T P^T: A = 16 dims x 16 tokens of V (ldmatrix.trans), B = P^T, which is the
//    scores' accumulator layout transposed per 8 x 8 block (movmatrix); the accumulator gives
//    lane (g, t) dims g, g + 8 of every 16 for query rows 2t, 2t + 1, so the rescale factors of
//    a lane's output columns are its own rows' and need no shuffle.
// The running max of rows 2t, 2t + 1 is uniform over the 8 lanes of a column (t); each lane
// keeps its part of the denominators (its two tokens of every sub-tile) until finish().
template <typename T, int D, int BS, bool CAUSAL>
struct MmaConsumer {
    static constexpr int KS = D / 16;  // k-steps of K Q^T, m-tiles of V^T P^T
    uint32_t qb[KS][2];                // Q^T B fragment: row g, dims 16kk + 2t, +1 and 16kk + 8 + 2t, +1
    float o[KS][4];                    // O^T fragments: rows d, columns query rows 2t, 2t + 1
    float m_lo, m_hi;                  // running max (log2 domain) of rows 2t, 2t + 1
    float l_lo, l_hi;                  // this lane's part of their denominators
    int lim_lo, lim_hi;                // the last positions rows 2t, 2t + 1 attend

    // q_row: query row lane / 4 of the unit, read only when live; last_lo / last_hi: the causal
    // bounds of rows 2 (lane % 4) and 2 (lane % 4) + 1.
    __device__ __forceinline__ void init(const T* q_row, bool live, int last_lo, int last_hi, int lane) {
        const int t = lane & 3;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(q_row);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qb[kk][0] = live ? __ldg(row + (kk * 16 + 2 * t) / 2) : 0u;
            qb[kk][1] = live ? __ldg(row + (kk * 16 + 8 + 2 * t) / 2) : 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) o[kk][e] = 0.f;
        }
        m_lo = m_hi = -INFINITY;
        l_lo = l_hi = 0.f;
        lim_lo = last_lo;
        lim_hi = last_hi;
    }

    // 8 x 8 b16 transpose across the warp: lane (g, t) gives elements (g, 2t), (g, 2t + 1) and
    // gets (2t, g), (2t + 1, g).
    static __device__ __forceinline__ uint32_t transpose8(uint32_t x) {
        uint32_t y;
        asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
        return y;
    }

    // Max over the 8 lanes of a column (lanes t, t + 4, ..., t + 28).
    static __device__ __forceinline__ float column_max(float v) {
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
        return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
    }

    // S^T of N 16-token sub-tiles (rows row0[i] .. row0[i] + 15 of staged K page kbase[i]), each
    // accumulated over the dims in two chains (even and odd k-steps); all 2N chains run side by side.
    template <int N>
    __device__ __forceinline__ void scores(float (&s)[N][4], const uint32_t (&kbase)[N], const int (&row0)[N],
                                           int lane) const {
        const int j = lane >> 3, r8 = lane & 7;
        const int acol = (j >> 1) * 8;  // ldmatrix order: A0 rows 0-7, A1 rows 8-15, A2/A3 dims 8-15
        float e[N][4], f[N][4];
#pragma unroll
        for (int i = 0; i < N; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) e[i][c] = f[i][c] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
            for (int i = 0; i < N; ++i) {
                uint32_t af[4];
                ldmatrix_x4(af, kbase[i] + swz_offset<T, BS>(row0[i] + (j & 1) * 8 + r8, kk * 16 + acol));
                Mma<T>::run((kk & 1) ? f[i] : e[i], af[0], af[1], af[2], af[3], qb[kk][0], qb[kk][1]);
            }
        }
#pragma unroll
        for (int i = 0; i < N; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[i][c] = e[i][c] + f[i][c];
    }

    // Scaled scores of a sub-tile with the tokens a row does not attend set to -inf: tokens g,
    // g + 8 of the sub-tile starting at position base, nv of its tokens in the context.
    __device__ __forceinline__ void mask(float (&x)[4], const float (&s)[4], int nv, int base, float scale_log2,
                                         int lane) const {
        const int g = lane >> 2;
        const int n_lo = CAUSAL ? min(nv, lim_lo - base + 1) : nv;
        const int n_hi = CAUSAL ? min(nv, lim_hi - base + 1) : nv;
        x[0] = g < n_lo ? s[0] * scale_log2 : -INFINITY;
        x[1] = g < n_hi ? s[1] * scale_log2 : -INFINITY;
        x[2] = g + 8 < n_lo ? s[2] * scale_log2 : -INFINITY;
        x[3] = g + 8 < n_hi ? s[3] * scale_log2 : -INFINITY;
    }

    // Zero V rows nv .. 15 of a sub-tile (rows past the context may hold anything, NaN included:
    // p = 0 times them must stay 0 in the MMA).
    __device__ __forceinline__ static void zero_tail(uint8_t* vpage, int row0, int nv, int lane) {
        if (nv >= 16) return;
        constexpr int kChunksPerRow = (D * (int)sizeof(T)) / 16;
        for (int idx = lane; idx < (16 - nv) * kChunksPerRow; idx += 32) {
            const int r = row0 + nv + idx / kChunksPerRow;
            const int c = idx % kChunksPerRow;
            *reinterpret_cast<uint4*>(vpage + (c / 8) * BS * 128 + r * 128 + (c % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
    }

    // Online-softmax step over the masked scores of n sub-tiles (x[4 * i ..] for sub-tile i):
    // returns the P^T B fragments (two per sub-tile) and leaves the rescale factors of rows 2t,
    // 2t + 1 in alpha_lo / alpha_hi.
    template <int N>
    __device__ __forceinline__ void softmax(const float (&x)[4 * N], uint32_t (&pb)[2 * N], float& alpha_lo,
                                            float& alpha_hi) {
        float mx_lo = x[0], mx_hi = x[1];
#pragma unroll
        for (int i = 0; i < 2 * N; ++i) {
            mx_lo = fmaxf(mx_lo, x[2 * i]);
            mx_hi = fmaxf(mx_hi, x[2 * i + 1]);
        }
        mx_lo = column_max(mx_lo);
        mx_hi = column_max(mx_hi);
        // -inf only while a row has attended nothing yet (a causal bound before these tokens):
        // then alpha and p are 0, not NaN.  Without causal bounds token 0 is always attended.
        const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
        const float ref_lo = (CAUSAL && mn_lo == -INFINITY) ? 0.f : mn_lo;
        const float ref_hi = (CAUSAL && mn_hi == -INFINITY) ? 0.f : mn_hi;
        alpha_lo = exp2f(m_lo - ref_lo);
        alpha_hi = exp2f(m_hi - ref_hi);
        float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
        for (int i = 0; i < 2 * N; ++i) {
            float r0, r1;
            pb[i] = transpose8(Mma<T>::pack(exp2f(x[2 * i] - ref_lo), exp2f(x[2 * i + 1] - ref_hi), r0, r1));
            sum_lo += r0;
            sum_hi += r1;
        }
        l_lo = l_lo * alpha_lo + sum_lo;
        l_hi = l_hi * alpha_hi + sum_hi;
        m_lo = mn_lo;
        m_hi = mn_hi;
    }

    // O^T = alpha O^T + V^T P^T over n sub-tiles (vrow0[i]: the first V row of sub-tile i).
    template <int N>
    __device__ __forceinline__ void accumulate(const uint32_t (&vbase)[N], const int (&vrow0)[N],
                                               const uint32_t (&pb)[2 * N], float alpha_lo, float alpha_hi,
                                               int lane) {
        const int j = lane >> 3, r8 = lane & 7;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            o[mt][0] *= alpha_lo;
            o[mt][1] *= alpha_hi;
            o[mt][2] *= alpha_lo;
            o[mt][3] *= alpha_hi;
#pragma unroll
            for (int i = 0; i < N; ++i) {
                uint32_t af[4];
                ldmatrix_x4_trans(af, vbase[i] + swz_offset<T, BS>(vrow0[i] + (j >> 1) * 8 + r8, mt * 16 + (j & 1) * 8));
                Mma<T>::run(o[mt], af[0], af[1], af[2], af[3], pb[2 * i], pb[2 * i + 1]);
            }
        }
    }

    // One page (BS tokens from position pos0, nvalid of them inside the context; a row
    // attends only the tokens up to its own bound).
    __device__ __forceinline__ void page(uint8_t* kpage, uint8_t* vpage, int nvalid, int pos0, float scale_log2,
                                         int lane) {
        const uint32_t kbase = smem_addr(kpage);
        const uint32_t vbase[1] = {smem_addr(vpage)};
#pragma unroll
        for (int sub = 0; sub < BS / 16; ++sub) {
            const int nv = nvalid - sub * 16;
            if (nv <= 0) break;
            zero_tail(vpage, sub * 16, nv, lane);
            float s[1][4], x[4];
            const uint32_t kb[1] = {kbase};
            const int row0[1] = {sub * 16};
            scores<1>(s, kb, row0, lane);
            mask(x, s[0], nv, pos0 + sub * 16, scale_log2, lane);
            uint32_t pb[2];
            float alpha_lo, alpha_hi;
            softmax<1>(x, pb, alpha_lo, alpha_hi);
            const int vrow0[1] = {sub * 16};
            accumulate<1>(vbase, vrow0, pb, alpha_lo, alpha_hi, lane);
        }
    }

    // Two 16-token pages (each with at least one token in the context, starting at positions
    // pos0 and pos1) in one online-softmax step: their score chains run side by side and the
    // running max and the rescale are taken once for the 32 tokens.
    __device__ __forceinline__ void page_pair(uint8_t* kp0, uint8_t* vp0, int nv0, int pos0, uint8_t* kp1,
                                              uint8_t* vp1, int nv1, int pos1, float scale_log2, int lane) {
        static_assert(BS == 16, "pairs of one-sub-tile pages");
        zero_tail(vp0, 0, nv0, lane);
        zero_tail(vp1, 0, nv1, lane);
        float sc[2][4], x[8];
        const uint32_t kb[2] = {smem_addr(kp0), smem_addr(kp1)};
        const int row0[2] = {0, 0};
        scores<2>(sc, kb, row0, lane);
        float x0[4], x1[4];
        mask(x0, sc[0], nv0, pos0, scale_log2, lane);
        mask(x1, sc[1], nv1, pos1, scale_log2, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = x0[i];
            x[4 + i] = x1[i];
        }
        uint32_t pb[4];
        float alpha_lo, alpha_hi;
        softmax<2>(x, pb, alpha_lo, alpha_hi);
        const uint32_t vbase[2] = {smem_addr(vp0), smem_addr(vp1)};
        accumulate<2>(vbase, row0, pb, alpha_lo, alpha_hi, lane);
    }

    // Complete the denominators (sum over the column's 8 lanes); call once after a unit's last page.
    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int w = 4; w < 32; w <<= 1) {
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, w);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, w);
        }
    }

    // Forget the unit (init() sets everything again): keeps its registers free meanwhile.
    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qb[kk][0] = qb[kk][1] = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) o[kk][e] = 0.f;
        }
        m_lo = m_hi = -INFINITY;
        l_lo = l_hi = 0.f;
    }

    // out[row(r) * D + d] = o~ / l for the gc rows (after finish()); a row that attended
    // nothing (l = 0) gets zeros.
    __device__ __forceinline__ void write_out(T* out, const UnitRows& rows, int gc, int lane) const {
        const int g = lane >> 2, t = lane & 3;
        const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
        const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
        T* lo = out + rows.row(min(2 * t, gc - 1)) * D;
        T* hi = out + rows.row(min(2 * t + 1, gc - 1)) * D;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            if (2 * t < gc) {
                lo[mt * 16 + g] = from_float<T>(o[mt][0] * inv_lo);
                lo[mt * 16 + 8 + g] = from_float<T>(o[mt][2] * inv_lo);
            }
            if (2 * t + 1 < gc) {
                hi[mt * 16 + g] = from_float<T>(o[mt][1] * inv_hi);
                hi[mt * 16 + 8 + g] = from_float<T>(o[mt][3] * inv_hi);
            }
        }
    }

    // Store m, l of rows 2t, 2t + 1 (lanes of g = 0) at m_at[r], l_at[r] (after finish()).
    __device__ __forceinline__ void write_stats(float* m_at, float* l_at, size_t stride, int gc, int lane) const {
        const int g = lane >> 2, t = lane & 3;
        if (g == 0) {
            if (2 * t < gc) {
                m_at[(size_t)(2 * t) * stride] = m_lo;
                l_at[(size_t)(2 * t) * stride] = l_lo;
            }
            if (2 * t + 1 < gc) {
                m_at[(size_t)(2 * t + 1) * stride] = m_hi;
                l_at[(size_t)(2 * t + 1) * stride] = l_hi;
            }
        }
    }

    // o~ of rows 2t, 2t + 1 at lo[d], hi[d].
    __device__ __forceinline__ void write_o(float* lo, float* hi, int gc, int lane) const {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            if (2 * t < gc) {
                lo[mt * 16 + g] = o[mt][0];
                lo[mt * 16 + 8 + g] = o[mt][2];
            }
            if (2 * t + 1 < gc) {
                hi[mt * 16 + g] = o[mt][1];
                hi[mt * 16 + 8 + g] = o[mt][3];
            }
        }
    }

    // Partial record of kHeads = 8 heads: m[8], l[8], o~[8][D] (after finish()).
    __device__ __forceinline__ void write_partial(float* rec, int gc, int lane) const {
        const int t = lane & 3;
        write_stats(rec, rec + 8, 1, gc, lane);
        write_o(rec + 16 + (size_t)(2 * t) * D, rec + 16 + (size_t)(2 * t + 1) * D, gc, lane);
    }

    // Split-KV partials of the gc rows straight into the workspace (after finish()):
    // ws_m / ws_l [row][part], ws_o [row][part][D], rows row0 .. row0 + gc - 1.
    __device__ __forceinline__ void write_split(float* ws_m, float* ws_l, float* ws_o, size_t row0, int max_parts,
                                                int part, int gc, int lane) const {
        const int t = lane & 3;
        write_stats(ws_m + row0 * max_parts + part, ws_l + row0 * max_parts + part, (size_t)max_parts, gc, lane);
        write_o(ws_o + ((row0 + 2 * t) * max_parts + part) * D, ws_o + ((row0 + 2 * t + 1) * max_parts + part) * D,
                gc, lane);
    }

    // Write this warp's state (all 8 rows) into the CTA combine buffer.
    __device__ __forceinline__ void store(float* co, float* cm, float* cl, int warp, int lane, int ostride) {
        const int t = lane & 3;
        finish();
        write_stats(cm + warp * 8, cl + warp * 8, 1, 8, lane);
        write_o(co + (size_t)(warp * 8 + 2 * t) * ostride, co + (size_t)(warp * 8 + 2 * t + 1) * ostride, 8, lane);
    }
};

// ------------------------------------------------------------------------------------------
// Tensor-core consumer for an FP8 (E4M3) cache with a float32 scale per (physical block,
// kv head) for K and for V.  The codes are widened to f16 exactly (e4m3x2 -> f16x2) and
// multiplied on the f16 tensor path with fp32 accumulation; the page's K scale multiplies
// its scores, its V scale enters through the running output's rescale factor (the output
// is kept in units of the current page's V scale).  The query row is brought to f16 exactly
// by a power of two (its largest magnitude lands in [2^14, 2^15)), undone in the score
// factor, so bf16 and f16 queries of any range stay exact.
//
// Fragment layouts (m16n8k16 f16, g = lane / 4, c = lane % 4):
//  * S = Q K^T: the k index of a k-step is a permutation of d shared by both operands:
//    lane c owns d in [32c, 32c + 32) and k-step kk takes its bytes 4kk .. 4kk + 3
//    (k = 2c, 2c+1 -> 32c + 4kk + {0, 1};  k = 2c+8, 2c+9 -> 32c + 4kk + {2, 3}), so a
//    token's K row is two 16-byte shared-memory loads per lane.
//  * O^T += V^T P^T: m-tile i maps row g to d = 16g + 2i and row g+8 to d = 16g + 2i + 1,
//    so lane g reads bytes 16g .. 16g+15 of four V rows (one 16-byte load each) and the
//    token pairs of the A fragment come from byte permutes; the lane ends up holding
//    d = 16g .. 16g+15 of its two output rows.
// Both patterns are free of bank conflicts under the 128-byte swizzle.
// Four E4M3 codes (bytes 0..3 of w) -> two f16x2: lo = (byte 0, byte 1), hi = (byte 2, byte 3), the
// lower byte in the lower half (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// The step's new token for an FP8 cache (append mode of pa_decode_fp8_append): the new K and V rows
// (D elements of T each, one 16-byte chunk per lane: lanes 0..15 K, 16..31 V) are quantised with the
// scale of the block that receives them, exactly as pa_write_kv_fp8 does (float32 division, E4M3 with
// round-to-nearest-even and saturation), patched into the staged page and stored into the cache.
template <typename T, int D, int BS>
struct NewTokenF8 {
    static_assert(D * (int)sizeof(T) == 256, "one 16-byte chunk of K or V per lane at head_dim 128");
    uint8_t* stage;  // this warp's 512-byte staging area in shared memory
    uint2 code;      // this lane's E4M3 codes (after patch())

    // Start the copy of this lane's 8 source elements into the staging area (no registers held
    // while the pages before the token's page are consumed).
    __device__ __forceinline__ void load(const T* key_row, const T* value_row, int lane) {
        cp_async_16(stage + 16 * lane, reinterpret_cast<const uint4*>(lane < 16 ? key_row : value_row) + (lane & 15));
        cp_async_commit();
    }

    // Quantise with the block's K / V scale and overwrite row r of the staged K and V tiles.
    __device__ __forceinline__ void patch(uint8_t* kpage, uint8_t* vpage, int r, float ks, float vs, int lane) {
        cp_async_wait_all();  // this lane's own 16 bytes
        float x[8];
        unpack16<T>(*reinterpret_cast<const uint4*>(stage + 16 * lane), x);
        const float sc = lane < 16 ? ks : vs;
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * h] / sc, x[4 * h + 1] / sc), __NV_SATFINITE,
                                                         __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * h + 2] / sc, x[4 * h + 3] / sc),
                                                         __NV_SATFINITE, __NV_E4M3);
            w[h] = lo | (hi << 16);
        }
        code = make_uint2(w[0], w[1]);
        const int ch = lane & 15;  // bytes 8ch .. 8ch + 7 of the 128-byte row
        uint8_t* tile = lane < 16 ? kpage : vpage;
        *reinterpret_cast<uint2*>(tile + r * 128 + ((((ch >> 1) ^ (r & 7))) << 4) + (ch & 1) * 8) = code;
        fence_proxy_async_smem();
        __syncwarp();
    }

    // Store the codes at row `off` of record row `rec_row` = (pb * Hkv + kvh) * BS of the caches.
    __device__ __forceinline__ void store(void* key_cache, void* value_cache, int rec_row, int off, bool interleaved,
                                          int lane) const {
        const int ch = lane & 15;
        size_t at;
        uint8_t* base;
        if (interleaved) {  // [N, H_kv, 2, BS, D] in key_cache
            at = ((size_t)2 * rec_row + (lane < 16 ? 0 : BS) + off) * D;
            base = static_cast<uint8_t*>(key_cache);
        } else {
            at = ((size_t)rec_row + off) * D;
            base = static_cast<uint8_t*>(lane < 16 ? key_cache : value_cache);
        }
        *reinterpret_cast<uint2*>(base + at + ch * 8) = code;
    }
};

template <typename T, int D, int BS>
struct MmaConsumerF8 {
    static_assert(D == 128, "the FP8 consumer's lane layout is for head_dim 128");
    static_assert(BS % 16 == 0, "16-token sub-tiles");
    static constexpr int KS = D / 16;  // k-steps of QK^T, m-tiles of PV
    uint32_t qa[KS][2];                // f16 Q^T B fragments of query row lane / 4
    float o[KS][4];                    // O^T fragments (columns: query rows 2c, 2c + 1), in units of vs_cur
    float m_lo, m_hi;                  // running max of rows 2c, 2c + 1 (uniform over the column's lanes)
    float l_lo, l_hi;                  // this lane's part of their denominators
    float qf_lo, qf_hi;                // their score factors: 2^-e * scale * log2(e)
    float vs_cur;                      // V scale o is expressed in (0 before the first page)

    // q_row: this lane's query row (row lane / 4 of the unit), read only when live.
    __device__ __forceinline__ void init(const T* q_row, bool live, float scale_log2, int lane) {
        const int c = lane & 3;
        float x[32];
        const uint4* src = reinterpret_cast<const uint4*>(q_row + c * (D / 4));
#pragma unroll
        for (int i = 0; i < 4; ++i) unpack16<T>(live ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u), x + 8 * i);
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int e = 0;
        if (amax > 0.f) {
            int ex;
            frexpf(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1)
            e = min(max(15 - ex, -126), 127);
        }
        const float p2 = __int_as_float((e + 127) << 23);  // 2^e, exact
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const __half2 lo = __floats2half2_rn(x[4 * kk] * p2, x[4 * kk + 1] * p2);
            const __half2 hi = __floats2half2_rn(x[4 * kk + 2] * p2, x[4 * kk + 3] * p2);
            qa[kk][0] = *reinterpret_cast<const uint32_t*>(&lo);
            qa[kk][1] = *reinterpret_cast<const uint32_t*>(&hi);
#pragma unroll
            for (int r = 0; r < 4; ++r) o[kk][r] = 0.f;
        }
        const float qf = scale_log2 * __int_as_float((127 - e) << 23);  // row lane / 4's factor, 2^-e
        qf_lo = __shfl_sync(0xffffffffu, qf, (2 * c) * 4);
        qf_hi = __shfl_sync(0xffffffffu, qf, (2 * c + 1) * 4);
        m_lo = m_hi = -INFINITY;
        l_lo = l_hi = 0.f;
        vs_cur = 0.f;
    }

    // One page (BS tokens, nvalid of them inside the context) with its K and V scales.
    __device__ __forceinline__ void page(const uint8_t* kpage, uint8_t* vpage, int nvalid, float ks, float vs,
                                         int lane) {
        const int g = lane >> 2, c = lane & 3;
        float vr = vs_cur == 0.f ? 1.f : vs_cur / vs;  // o into units of this page's V scale
        vs_cur = vs;
        const float sf_lo = qf_lo * ks, sf_hi = qf_hi * ks;
#pragma unroll
        for (int sub = 0; sub < BS / 16; ++sub) {
            const int nv = nvalid - sub * 16;
            if (nv <= 0) break;
            if (nv < 16) {
                // V rows past the context may hold anything (NaN codes included): zero them.
                for (int idx = lane; idx < (16 - nv) * 8; idx += 32)
                    *reinterpret_cast<uint4*>(vpage + (sub * 16 + nv + idx / 8) * 128 + (idx % 8) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- S^T = K Q^T: the sub-tile's 16 tokens on the MMA's rows (tokens g and g + 8 here), the
            // query rows on its columns; summed in two chains (even and odd k-steps) ----
            const int tok = sub * 16 + g;
            const uint8_t* rk0 = kpage + tok * 128;
            const uint8_t* rk1 = rk0 + 8 * 128;  // token g + 8: the same swizzle phase
            const int sw = tok & 7;
            const uint4 k00 = *reinterpret_cast<const uint4*>(rk0 + (((2 * c) ^ sw) << 4));
            const uint4 k01 = *reinterpret_cast<const uint4*>(rk0 + (((2 * c + 1) ^ sw) << 4));
            const uint4 k10 = *reinterpret_cast<const uint4*>(rk1 + (((2 * c) ^ sw) << 4));
            const uint4 k11 = *reinterpret_cast<const uint4*>(rk1 + (((2 * c + 1) ^ sw) << 4));
            const uint32_t kw0[8] = {k00.x, k00.y, k00.z, k00.w, k01.x, k01.y, k01.z, k01.w};
            const uint32_t kw1[8] = {k10.x, k10.y, k10.z, k10.w, k11.x, k11.y, k11.z, k11.w};
            float se[4] = {0.f, 0.f, 0.f, 0.f};
            float so[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(kw0[kk], a0, a2);  // token g: k = 2c, 2c + 1 | 2c + 8, 2c + 9
                e4m3x4_to_f16x2x2(kw1[kk], a1, a3);  // token g + 8
                Mma<__half>::run((kk & 1) ? so : se, a0, a1, a2, a3, qa[kk][0], qa[kk][1]);
            }
            // ---- online softmax for rows 2c, 2c + 1 over tokens g, g + 8 (token 0 is attended: finite max) ----
            const float x0 = g < nv ? (se[0] + so[0]) * sf_lo : -INFINITY;
            const float x1 = g < nv ? (se[1] + so[1]) * sf_hi : -INFINITY;
            const float x2 = g + 8 < nv ? (se[2] + so[2]) * sf_lo : -INFINITY;
            const float x3 = g + 8 < nv ? (se[3] + so[3]) * sf_hi : -INFINITY;
            float mx_lo = fmaxf(x0, x2), mx_hi = fmaxf(x1, x3);
#pragma unroll
            for (int w = 4; w < 32; w <<= 1) {
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, w));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, w));
            }
            const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
            const float alpha_lo = exp2f(m_lo - mn_lo), alpha_hi = exp2f(m_hi - mn_hi);
            float r0, r1, r2, r3;
            const uint32_t pk0 = Mma<__half>::pack(exp2f(x0 - mn_lo), exp2f(x1 - mn_hi), r0, r1);
            const uint32_t pk1 = Mma<__half>::pack(exp2f(x2 - mn_lo), exp2f(x3 - mn_hi), r2, r3);
            l_lo = l_lo * alpha_lo + (r0 + r2);
            l_hi = l_hi * alpha_hi + (r1 + r3);
            m_lo = mn_lo;
            m_hi = mn_hi;
            // P^T B fragments (tokens 2c, 2c + 1 | 2c + 8, 2c + 9 of query row g): the 8 x 8 blocks transposed
            const uint32_t pb0 = transpose8(pk0);
            const uint32_t pb1 = transpose8(pk1);
            const float a_lo = alpha_lo * vr;
            const float a_hi = alpha_hi * vr;
            vr = 1.f;
            // ---- O^T += V^T P^T ----
            const int t0 = sub * 16 + 2 * c;
            const uint4 v0 = *reinterpret_cast<const uint4*>(vpage + t0 * 128 + ((g ^ (t0 & 7)) << 4));
            const uint4 v1 = *reinterpret_cast<const uint4*>(vpage + (t0 + 1) * 128 + ((g ^ ((t0 + 1) & 7)) << 4));
            const uint4 v2 = *reinterpret_cast<const uint4*>(vpage + (t0 + 8) * 128 + ((g ^ ((t0 + 8) & 7)) << 4));
            const uint4 v3 = *reinterpret_cast<const uint4*>(vpage + (t0 + 9) * 128 + ((g ^ ((t0 + 9) & 7)) << 4));
            const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
            const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w}, w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;  // bytes 2(i&1), 2(i&1)+1 of both words
                const uint32_t p01 = __byte_perm(w0[i >> 1], w1[i >> 1], sel);
                const uint32_t p23 = __byte_perm(w2[i >> 1], w3[i >> 1], sel);
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(p01, a0, a1);
                e4m3x4_to_f16x2x2(p23, a2, a3);
                o[i][0] *= a_lo;
                o[i][1] *= a_hi;
                o[i][2] *= a_lo;
                o[i][3] *= a_hi;
                Mma<__half>::run(o[i], a0, a1, a2, a3, pb0, pb1);
            }
        }
    }

    // 8 x 8 b16 transpose across the warp: lane (g, c) gives elements (g, 2c), (g, 2c + 1), gets (2c, g), (2c + 1, g).
    static __device__ __forceinline__ uint32_t transpose8(uint32_t x) {
        uint32_t y;
        asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
        return y;
    }

    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int w = 4; w < 32; w <<= 1) {
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, w);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, w);
        }
    }

    __device__ __forceinline__ void clear() {
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qa[kk][0] = qa[kk][1] = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) o[kk][e] = 0.f;
        }
        m_lo = m_hi = -INFINITY;
        l_lo = l_hi = 0.f;
        vs_cur = 0.f;
    }

    // out[row(r) * D + d] = o~ / l for the gc rows (after finish()); a row with l = 0 gets zeros.
    __device__ __forceinline__ void write_out(T* out, const UnitRows& rows, int gc, int lane) const {
        const int g = lane >> 2, c = lane & 3;
        const float f_lo = l_lo > 0.f ? vs_cur / l_lo : 0.f;
        const float f_hi = l_hi > 0.f ? vs_cur / l_hi : 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = 2 * c + half;
            if (r >= gc) continue;
            const float f = half ? f_hi : f_lo;
            T v[16];
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                v[2 * i] = from_float<T>(o[i][half] * f);
                v[2 * i + 1] = from_float<T>(o[i][2 + half] * f);
            }
            uint4* dst = reinterpret_cast<uint4*>(out + rows.row(r) * D + 16 * g);
            dst[0] = *reinterpret_cast<const uint4*>(v);
            dst[1] = *reinterpret_cast<const uint4*>(v + 8);
        }
    }

    // Partial record of 8 rows: m[8], l[8], o~[8][D] in true units (after finish()).
    __device__ __forceinline__ void write_partial(float* rec, int gc, int lane) const {
        const int g = lane >> 2, c = lane & 3;
        if (g == 0) {
            if (2 * c < gc) {
                rec[2 * c] = m_lo;
                rec[8 + 2 * c] = l_lo;
            }
            if (2 * c + 1 < gc) {
                rec[2 * c + 1] = m_hi;
                rec[9 + 2 * c] = l_hi;
            }
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = 2 * c + half;
            if (r >= gc) continue;
            float4* dst = reinterpret_cast<float4*>(rec + 16 + (size_t)r * D + 16 * g);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                dst[q4] = make_float4(o[2 * q4][half] * vs_cur, o[2 * q4][2 + half] * vs_cur,
                                      o[2 * q4 + 1][half] * vs_cur, o[2 * q4 + 1][2 + half] * vs_cur);
        }
    }
};

// ------------------------------------------------------------------------------------------
// CUDA-core consumer (all dtypes).
template <typename T, int D, int BS, int GMAX>
struct SimtConsumer {
    static constexpr int LPT = 32 / BS;          // lanes per token in QK^T
    static constexpr int E = 16 / sizeof(T);     // elements per 16-byte chunk
    static constexpr int NCHUNK = D / E;
    static constexpr int DPL = D / 32;           // output elements per lane in PV
    static constexpr int VBYTES = DPL * sizeof(T);
    static_assert(VBYTES == 4 || VBYTES == 8 || VBYTES == 16, "PV load width");
    float o[GMAX][DPL];
    float m[GMAX], l[GMAX];
    int lim0, v0, group;  // row h attends positions up to lim0 + (v0 + h) / group

    __device__ __forceinline__ void init(int lim_base = 0x7fffffff, int first_row = 0, int rows_per_token = 1) {
        lim0 = lim_base;
        v0 = first_row;
        group = rows_per_token;
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[h][e] = 0.f;
        }
    }

    __device__ __forceinline__ void load_v(const uint8_t* p, float* vf) {
        if constexpr (VBYTES == 16) {
            unpack16<T>(*reinterpret_cast<const uint4*>(p), vf);
        } else if constexpr (VBYTES == 8) {
            const uint2 raw = *reinterpret_cast<const uint2*>(p);
            const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
            for (int i = 0; i < DPL; ++i) vf[i] = to_float(e[i]);
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(p);
            const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
            for (int i = 0; i < DPL; ++i) vf[i] = to_float(e[i]);
        }
    }

    __device__ __forceinline__ void page(const uint8_t* kpage, const uint8_t* vpage, int nvalid, int pos0,
                                         float scale_log2, const float* q_s, float* p_s, int lane) {
        const int tok = lane % BS;
        const int part = lane / BS;
        float acc[GMAX];
#pragma unroll
        for (int h = 0; h < GMAX; ++h) acc[h] = 0.f;
        if (tok < nvalid) {
#pragma unroll 4
            for (int c = part; c < NCHUNK; c += LPT) {
                float kf[E];
                unpack16<T>(*reinterpret_cast<const uint4*>(kpage + swz_offset<T, BS>(tok, c * E)), kf);
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    const float4* qv = reinterpret_cast<const float4*>(q_s + h * D + c * E);
#pragma unroll
                    for (int e4 = 0; e4 < E / 4; ++e4) {
                        const float4 qq = qv[e4];
                        acc[h] = fmaf(qq.x, kf[4 * e4 + 0], acc[h]);
                        acc[h] = fmaf(qq.y, kf[4 * e4 + 1], acc[h]);
                        acc[h] = fmaf(qq.z, kf[4 * e4 + 2], acc[h]);
                        acc[h] = fmaf(qq.w, kf[4 * e4 + 3], acc[h]);
                    }
                }
            }
        }
#pragma unroll
        for (int off = BS; off < 32; off <<= 1)
#pragma unroll
            for (int h = 0; h < GMAX; ++h) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            const int nr = min(nvalid, lim0 == 0x7fffffff ? nvalid : lim0 + (v0 + h) / group - pos0 + 1);
            const float x = tok < nr ? acc[h] * scale_log2 : -INFINITY;
            float mx = x;
#pragma unroll
            for (int off = 1; off < BS; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            // -inf only while the row has attended nothing yet: then alpha and p are 0, not NaN
            const float m_new = fmaxf(m[h], mx);
            const float m_ref = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = exp2f(m[h] - m_ref);
            const float p = exp2f(x - m_ref);
            l[h] = l[h] * alpha + (part == 0 ? p : 0.f);
            m[h] = m_new;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[h][e] *= alpha;
            if (part == 0) p_s[h * BS + tok] = p;
        }
        __syncwarp();
        for (int tk = 0; tk < nvalid; ++tk) {
            float vf[DPL];
            load_v(vpage + swz_offset<T, BS>(tk, lane * DPL), vf);
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
                const float pp = p_s[h * BS + tk];
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[h][e] = fmaf(pp, vf[e], o[h][e]);
            }
        }
        __syncwarp();
    }

    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
    }

    __device__ __forceinline__ void clear() { init(lim0, v0, group); }

    // out[row(h) * D + d] = o~ / l for the gc rows; a row that attended nothing gets zeros.
    __device__ __forceinline__ void write_out(T* out, const UnitRows& rows, int gc, int lane) const {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            if (h >= gc) break;
            const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
            T* dst = out + rows.row(h) * D;
#pragma unroll
            for (int e = 0; e < DPL; ++e) dst[lane * DPL + e] = from_float<T>(o[h][e] * inv);
        }
    }

    // Partial record of GMAX heads: m[GMAX], l[GMAX], then o~[GMAX][D] at a 16-byte
    // aligned offset (after finish()).
    __device__ __forceinline__ void write_partial(float* rec, int gc, int lane) const {
        constexpr int kOOff = ((2 * GMAX + 3) / 4) * 4;
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            if (h >= gc) break;
            if (lane == 0) {
                rec[h] = m[h];
                rec[GMAX + h] = l[h];
            }
#pragma unroll
            for (int e = 0; e < DPL; ++e) rec[kOOff + (size_t)h * D + lane * DPL + e] = o[h][e];
        }
    }

    __device__ __forceinline__ void store(float* co, float* cm, float* cl, int warp, int lane, int ostride) {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
            float lh = l[h];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) lh += __shfl_xor_sync(0xffffffffu, lh, off);
            if (lane == 0) {
                cm[warp * GMAX + h] = m[h];
                cl[warp * GMAX + h] = lh;
            }
            float* row = co + (size_t)(warp * GMAX + h) * ostride + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) row[e] = o[h][e];
        }
    }
};

// ------------------------------------------------------------------------------------------
template <typename T, int D, int BS, bool MMA, int GMAX, bool CAUSAL>
__global__ void __launch_bounds__(DecodeCfg<T, D, BS, MMA, GMAX>::kThreads,
                                  ((MMA && CAUSAL && BS == 16 && D <= 128) ? 3
                                                                           : DecodeCfg<T, D, BS, MMA, GMAX>::kMinBlocks))
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                        const DecodeArgs a) {
    using C = DecodeCfg<T, D, BS, MMA, GMAX>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint64_t* empty = full + C::kNSlot;
    int* issued = reinterpret_cast<int*>(smem + C::kIssuedOffset);
    float* stat = reinterpret_cast<float*>(smem + C::kStatOffset);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + C::kFlagOffset);  // [0]: abort

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // Wait for the previous grid in the stream (programmatic dependent launch), then let
    // the next one (the merge, when there is one) get resident early; it waits for this
    // grid's completion before reading anything.
    griddep_wait();
    griddep_launch_dependents();

    // ---- which work unit ----
    const int units = a.num_seqs * a.num_kv_heads * a.head_chunks;
    const int p = blockIdx.x / units;
    const int unit = blockIdx.x - p * units;
    const int hc = unit % a.head_chunks;
    const int bk = unit / a.head_chunks;
    const int kvh = bk % a.num_kv_heads;
    const int b = bk / a.num_kv_heads;
    // Row split: every consumer warp takes one row chunk of the kv head and every page.
    const bool rs = CAUSAL && a.row_split;
    const int nchunks = rs ? (a.rows + C::kHeads - 1) / C::kHeads : 1;
    // the unit's query/output rows (built where used, so that no copy lives across the page loop)
#define PA_UNIT_ROWS UnitRows{b, kvh, hc * C::kHeads, a.q_len, a.group, a.num_heads}
    const int gc = min(C::kHeads, a.rows - hc * C::kHeads);

    int L = __ldg(a.context_lens + b);
    const int l_cap = min(a.max_blocks, a.max_parts * a.partition_pages) * BS;
    if (L < 0 || L > l_cap) {
        if (p == 0 && tid == 0) atomicOr(a.err, kErrBadContext);
        L = L < 0 ? 0 : l_cap;
    }
    const int nblk = (L + BS - 1) / BS;
    const int nparts = (nblk + a.partition_pages - 1) / a.partition_pages;
    T* out = static_cast<T*>(a.out);

    if (L == 0) {  // empty context: zero rows (partition 0 writes them)
        if (p == 0)
            for (int idx = tid; idx < (rs ? a.rows : gc) * D; idx += C::kThreads)
                out[PA_UNIT_ROWS.row(idx / D) * D + idx % D] = from_float<T>(0.f);
        return;
    }
    const int first = p * a.partition_pages;
    if (first >= nblk) return;
    const int npages = min(a.partition_pages, nblk - first);

    if (tid == 0) {
        for (int s = 0; s < C::kNSlot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nchunks);  // row split: every chunk's warp releases the slot
            issued[s] = 0;
        }
        flags[0] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == C::kNW) {
        // ================= producer warp =================
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        // Pages are read once per call: let them leave L2 first.
        const uint64_t stream_policy = l2_policy_evict_first();
        const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks + first;
        int next = lane < npages ? __ldg(bt + lane) : 0;
        bool ok = true;
        for (int c = 0; c < npages && ok; c += 32) {
            const int cur = next;
            if (c + 32 + lane < npages) next = __ldg(bt + c + 32 + lane);
            const int n = min(32, npages - c);
            for (int jj = 0; jj < n; ++jj) {
                const int pb = __shfl_sync(0xffffffffu, cur, jj);
                int good = 1;
                if (lane == 0) {
                    const int i = c + jj;
                    const int s = i % C::kNSlot;
                    if (i >= C::kNSlot)
                        good = mbar_wait_bounded(&empty[s], ((i / C::kNSlot) - 1) & 1, a.err, flags) ? 1 : 0;
                    if (good) {
                        issued[s] += 1;
                        if ((unsigned)pb < (unsigned)a.num_blocks) {
                            mbar_arrive_expect_tx(&full[s], C::kSlotBytes);
                            const int row = (pb * a.num_kv_heads + kvh) * BS;
                            uint8_t* kdst = ring + s * C::kSlotBytes;
                            uint8_t* vdst = kdst + C::kPageBytes;
#pragma unroll
                            for (int bx = 0; bx < C::kNBox; ++bx)
                                tma_load_2d_hint(kdst + bx * C::kBoxBytes, &tmap_k, bx * C::kBoxElems, row, &full[s],
                                                 stream_policy);
#pragma unroll
                            for (int bx = 0; bx < C::kNBox; ++bx)
                                tma_load_2d_hint(vdst + bx * C::kBoxBytes, &tmap_v, bx * C::kBoxElems, row, &full[s],
                                                 stream_policy);
                        } else {
                            atomicOr(a.err, kErrBadTable);  // skip the load; the slot keeps stale data
                            mbar_arrive(&full[s]);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                if (!ok) break;
            }
        }
    } else {
        // ================= consumer warps =================
        const T* q = static_cast<const T*>(a.q);
        // Append mode: the warp that consumes the page holding position L - 1 takes the
        // new token into its staged copy of the page, and (head chunk 0) into the cache.
        // The token is fetched when that page comes up (holding it in registers across the
        // page loop would cost this kernel its occupancy).
        const int i_tok = a.new_key != nullptr ? nblk - 1 - first : -1;  // that page's index here
        if constexpr (MMA) {
            MmaConsumer<T, D, BS, CAUSAL> cons;
            const int chunk = rs ? warp : hc;  // this warp's row chunk
            const int cgc = rs ? min(C::kHeads, a.rows - chunk * C::kHeads) : gc;
            if (cgc > 0) {
                const UnitRows rows{b, kvh, chunk * C::kHeads, a.q_len, a.group, a.num_heads};
                const int r = min(lane >> 2, cgc - 1);
                cons.init(q + rows.row(r) * D, (lane >> 2) < cgc, rows.last_pos(2 * (lane & 3), L),
                          rows.last_pos(2 * (lane & 3) + 1, L), lane);
            }
            // without row split the warps share the pages round-robin; with it a warp whose
            // chunk is empty (fewer than four chunks) takes no part
            int i0 = rs ? (cgc > 0 ? 0 : npages) : warp;
            if constexpr (CAUSAL && BS == 16) {
                // Row split: every warp consumes every page, two at a time (one softmax step
                // per 32 tokens); an odd last page goes through the loop below.
                if (rs) {
                    for (; i0 + 1 < npages; i0 += 2) {
                        const int s0 = i0 % C::kNSlot, s1 = (i0 + 1) % C::kNSlot;
                        const bool got = mbar_wait_bounded(&full[s0], (i0 / C::kNSlot) & 1, a.err, flags) &&
                                         mbar_wait_bounded(&full[s1], ((i0 + 1) / C::kNSlot) & 1, a.err, flags);
                        if (!__all_sync(0xffffffffu, got)) {
                            i0 = npages;
                            break;
                        }
                        const int nv0 = min(BS, L - (first + i0) * BS), nv1 = min(BS, L - (first + i0 + 1) * BS);
                        uint8_t* kp0 = ring + s0 * C::kSlotBytes;
                        uint8_t* kp1 = ring + s1 * C::kSlotBytes;
                        if (i0 == i_tok)
                            append_token<T, D, BS>(a, b, kvh, hc, nblk - 1, kp0, kp0 + C::kPageBytes, nv0, lane);
                        if (i0 + 1 == i_tok)
                            append_token<T, D, BS>(a, b, kvh, hc, nblk - 1, kp1, kp1 + C::kPageBytes, nv1, lane);
                        cons.page_pair(kp0, kp0 + C::kPageBytes, nv0, (first + i0) * BS, kp1, kp1 + C::kPageBytes,
                                       nv1, (first + i0 + 1) * BS, a.scale_log2, lane);
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(&empty[s0]);
                            mbar_arrive(&empty[s1]);
                        }
                    }
                }
            }
            for (int i = i0; i < npages; i += rs ? 1 : C::kNW) {
                const int s = i % C::kNSlot;
                const bool got = mbar_wait_bounded(&full[s], (i / C::kNSlot) & 1, a.err, flags);
                if (!__all_sync(0xffffffffu, got)) break;
                const int nvalid = min(BS, L - (first + i) * BS);
                uint8_t* kp = ring + s * C::kSlotBytes;
                if (i == i_tok) append_token<T, D, BS>(a, b, kvh, hc, nblk - 1, kp, kp + C::kPageBytes, nvalid, lane);
                cons.page(kp, kp + C::kPageBytes, nvalid, (first + i) * BS, a.scale_log2, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if (rs) {
                // each warp holds whole rows: no combine, its rows go straight out
                if (cgc > 0 && !flags[0]) {
                    cons.finish();
                    if (nparts == 1) {
                        cons.write_out(out, UnitRows{b, kvh, chunk * C::kHeads, a.q_len, a.group, a.num_heads}, cgc,
                                       lane);
                    } else {
                        cons.write_split(a.ws_m, a.ws_l, a.ws_o,
                                         ((size_t)b * a.num_kv_heads + kvh) * a.rows + chunk * C::kHeads, a.max_parts,
                                         p, cgc, lane);
                    }
                }
            } else {
                // All consumers are past their last page, so every TMA into the ring has
                // landed and been read: the ring can hold the combine buffer.
                asm volatile("bar.sync 1, %0;" ::"r"(C::kNW * 32) : "memory");
                if (!flags[0]) {
                    float* co = reinterpret_cast<float*>(ring);
                    float* cm = co + C::kNW * C::kHeads * C::kOStride;
                    float* cl = cm + C::kNW * C::kHeads;
                    cons.store(co, cm, cl, warp, lane, C::kOStride);
                }
            }
        } else {
            float* q_s = reinterpret_cast<float*>(smem + C::kQsOffset);
            float* p_s = reinterpret_cast<float*>(smem + C::kPsOffset) + warp * GMAX * BS;
            for (int idx = tid; idx < GMAX * D; idx += C::kNW * 32) {
                const int h = idx / D;
                q_s[idx] = h < gc ? to_float(q[PA_UNIT_ROWS.row(h) * D + idx % D]) : 0.f;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(C::kNW * 32) : "memory");
            SimtConsumer<T, D, BS, GMAX> cons;
            cons.init(L - a.q_len, hc * C::kHeads, a.group);
            for (int i = warp; i < npages; i += C::kNW) {
                const int s = i % C::kNSlot;
                const bool got = mbar_wait_bounded(&full[s], (i / C::kNSlot) & 1, a.err, flags);
                if (!__all_sync(0xffffffffu, got)) break;
                const int nvalid = min(BS, L - (first + i) * BS);
                uint8_t* kp = ring + s * C::kSlotBytes;
                if (i == i_tok) append_token<T, D, BS>(a, b, kvh, hc, nblk - 1, kp, kp + C::kPageBytes, nvalid, lane);
                cons.page(kp, kp + C::kPageBytes, nvalid, (first + i) * BS, a.scale_log2, q_s, p_s, lane);
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            asm volatile("bar.sync 1, %0;" ::"r"(C::kNW * 32) : "memory");
            if (!flags[0]) {
                float* co = reinterpret_cast<float*>(ring);
                float* cm = co + C::kNW * C::kHeads * C::kOStride;
                float* cl = cm + C::kNW * C::kHeads;
                cons.store(co, cm, cl, warp, lane, C::kOStride);
            }
        }
    }
    __syncthreads();  // pipeline finished (or abandoned); combine buffer written

    if (flags[0]) {
        // A wait gave up: let every issued copy land before the CTA's shared memory goes away.
        if (tid == 0)
            for (int s = 0; s < C::kNSlot; ++s)
                if (issued[s] > 0) {
                    const unsigned long long start = global_timer_ns();
                    while (!mbar_try_wait(&full[s], (issued[s] - 1) & 1) &&
                           global_timer_ns() - start < kWaitLimitNs) {
                    }
                }
        return;
    }
    if (rs) return;  // row split: the warps wrote their own rows

    // ---- combine the consumer warps' states ----
    const float* co = reinterpret_cast<const float*>(ring);
    const float* cm = co + C::kNW * C::kHeads * C::kOStride;
    const float* cl = cm + C::kNW * C::kHeads;
    float* stat_m = stat;
    float* stat_w = stat + C::kHeads;
    float* wgt = stat + 2 * C::kHeads;  // [kNW][kHeads]
    if (tid < gc) {
        float mm = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kNW; ++w) mm = fmaxf(mm, cm[w * C::kHeads + tid]);
        float ws = 0.f;
#pragma unroll
        for (int w = 0; w < C::kNW; ++w) {
            // 0 for a warp that saw no page, or a row whose bound lies before it
            const float f = rescale(cm[w * C::kHeads + tid], mm);
            wgt[w * C::kHeads + tid] = f;
            ws += f * cl[w * C::kHeads + tid];
        }
        stat_m[tid] = mm;
        stat_w[tid] = ws;
    }
    __syncthreads();
    const bool single = nparts == 1;
    // split-KV partials are indexed by the kv head's row: (b * H_kv + kvh) * rows + v
    const UnitRows rows = PA_UNIT_ROWS;
#undef PA_UNIT_ROWS
    const size_t row0 = ((size_t)b * a.num_kv_heads + kvh) * a.rows + rows.v0;
    for (int idx = tid; idx < gc * D; idx += C::kThreads) {
        const int h = idx / D;
        const int d = idx - h * D;
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < C::kNW; ++w) acc += wgt[w * C::kHeads + h] * co[(w * C::kHeads + h) * C::kOStride + d];
        if (single) {
            out[rows.row(h) * D + d] = from_float<T>(stat_w[h] > 0.f ? acc / stat_w[h] : 0.f);
        } else {
            a.ws_o[((row0 + h) * a.max_parts + p) * D + d] = acc;
        }
    }
    if (!single && tid < gc) {
        a.ws_m[(row0 + tid) * a.max_parts + p] = stat_m[tid];
        a.ws_l[(row0 + tid) * a.max_parts + p] = stat_w[tid];
    }
}

// ------------------------------------------------------------------------------------------
// Split-KV merge: one CTA per output row (b, qh); rows whose context fits one
// partition were finished by the decode kernel and are skipped.
//     M = max_p m_p,  W = sum_p 2^(m_p - M) l_p,  o = sum_p 2^(m_p - M) o~_p / W.
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxParts = 4096;

// One warp per output row: lane p holds partition p's m and l (32 partitions at a time), and
// lane i holds dims i * DPL .. i * DPL + DPL - 1 of the merged row.  The m, l and the first
// kMergePre partial outputs of a row are loaded together, so a row of up to kMergePre
// partitions costs one round trip to memory.
constexpr int kMergePre = 8;

template <int DPL>
__device__ __forceinline__ void load_dims(float (&v)[DPL], const float* src) {
    if constexpr (DPL % 4 == 0) {
#pragma unroll
        for (int e = 0; e < DPL; e += 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src + e));
            v[e] = x.x;
            v[e + 1] = x.y;
            v[e + 2] = x.z;
            v[e + 3] = x.w;
        }
    } else if constexpr (DPL == 2) {
        const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
        v[0] = x.x;
        v[1] = x.y;
    } else {
#pragma unroll
        for (int e = 0; e < DPL; ++e) v[e] = __ldcg(src + e);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) splitkv_merge_kernel(const MergeArgs a) {
    static_assert(D % 32 == 0, "whole dims per lane");
    static_assert(32 % kMergePre == 0, "partition batches inside a 32-partition chunk");
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);  // (b * H_kv + kvh) * rows + v

    // Wait for the decode kernel's partials (programmatic dependent launch); then the
    // next grid in the stream may start launching.
    griddep_wait();
    griddep_launch_dependents();
    if (row >= a.num_seqs * a.num_kv_heads * a.rows) return;
    const int b = row / (a.num_kv_heads * a.rows);

    int L = __ldg(a.context_lens + b);
    const int l_cap = min(a.max_blocks, a.max_parts * a.partition_pages) * a.block_size;
    L = L < 0 ? 0 : (L > l_cap ? l_cap : L);
    const int nblk = (L + a.block_size - 1) / a.block_size;
    const int n = (nblk + a.partition_pages - 1) / a.partition_pages;
    if (n <= 1) return;  // the decode kernel wrote the row itself

    const float* mrow = a.ws_m + (size_t)row * a.max_parts;
    const float* lrow = a.ws_l + (size_t)row * a.max_parts;
    const float* obase = a.ws_o + (size_t)row * a.max_parts * D + lane * DPL;
    const float m0 = lane < n ? __ldcg(mrow + lane) : -INFINITY;
    const float l0 = lane < n ? __ldcg(lrow + lane) : 0.f;
    float v[kMergePre][DPL];
#pragma unroll
    for (int i = 0; i < kMergePre; ++i) {
        if (i < n) {
            load_dims<DPL>(v[i], obase + (size_t)i * D);
        } else {
#pragma unroll
            for (int e = 0; e < DPL; ++e) v[i][e] = 0.f;
        }
    }
    // 1) the common max over the partitions
    float mm = m0;
    for (int c = 32; c < n; c += 32)
        if (c + lane < n) mm = fmaxf(mm, __ldcg(mrow + c + lane));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, off));
    // 2) weights (a partition a row's causal bound excludes weighs 0) and the merged
    //    denominator; 3) the weighted sum of the partial outputs
    float f = rescale(m0, mm);  // weight of partition c + lane of the current chunk
    float ws = f * l0;
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < kMergePre; ++i) {
        const float fi = __shfl_sync(0xffffffffu, f, i);
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] += fi * v[i][e];
    }
    for (int q0 = kMergePre; q0 < n; q0 += kMergePre) {
        if (q0 % 32 == 0) {
            const int q = q0 + lane;
            f = q < n ? rescale(__ldcg(mrow + q), mm) : 0.f;
            ws += q < n ? f * __ldcg(lrow + q) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kMergePre; ++i) {
            if (q0 + i < n) {
                load_dims<DPL>(v[i], obase + (size_t)(q0 + i) * D);
            } else {
#pragma unroll
                for (int e = 0; e < DPL; ++e) v[i][e] = 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kMergePre; ++i) {
            const float fi = __shfl_sync(0xffffffffu, f, (q0 + i) % 32);
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[e] += fi * v[i][e];
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);

    const int rest = row - b * a.num_kv_heads * a.rows;
    const int kvh = rest / a.rows;
    const UnitRows rows{b, kvh, rest - kvh * a.rows, a.q_len, a.group, a.num_heads};
    T* out = static_cast<T*>(a.out) + rows.row(0) * D + lane * DPL;
    const float inv = ws > 0.f ? 1.f / ws : 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) out[e] = from_float<T>(acc[e] * inv);
}


// ------------------------------------------------------------------------------------------
// Lean (stream-K) schedule.  A persistent grid of C CTAs (one wave); the pages
// of all (sequence, kv head, head chunk) units are laid end to end (sequence-
// major, then kv head, then head chunk, pages in logical order) and cut into
// C * NW equal contiguous ranges, one per consumer warp.  So every warp streams
// the same number of pages whatever the context lengths are.  A warp finishes
// every unit that lies wholly inside its range (o = o~ / l straight to out);
// for a unit cut by a range boundary it writes a partial (m, l, o~) record (two
// record slots per warp: its first and its last unit), which lean_merge_kernel
// combines with the same rescaling rule as the online softmax.
constexpr int kLeanMaxSeqs = 4096;

template <typename T, int D, int BS, bool MMA, int GMAX>
struct LeanCfg {
    using Base = DecodeCfg<T, D, BS, MMA, GMAX>;
    static constexpr int kNW = Base::kNW;
    static constexpr int kThreads = Base::kThreads;
    // Page slots per consumer warp: about PA_LEAN_RING_KB of ring per CTA, 1 to 6 slots a warp.
    static constexpr int kSPWRaw = (PA_LEAN_RING_KB * 1024) / (kNW * Base::kSlotBytes);
    static constexpr int kSPW = kSPWRaw < 1 ? 1 : (kSPWRaw > 6 ? 6 : kSPWRaw);
    static constexpr int kNSlot = kNW * kSPW;
    static constexpr int kSlotBytes = Base::kSlotBytes;
    static constexpr int kPageBytes = Base::kPageBytes;
    static constexpr int kRingBytes = kNSlot * kSlotBytes;
    static constexpr int kHeads = Base::kHeads;
    static constexpr int kOOff = ((2 * kHeads + 3) / 4) * 4;  // o~ offset in a partial record
    static constexpr int kRecFloats = kOOff + kHeads * D;      // one partial record
    static constexpr int kRowQueue = 64;  // published page rows per consumer warp (two chunks of 32)
    // Shared-memory regions after the ring, each 16-byte aligned.
    static constexpr int a16(int x) { return (x + 15) & ~15; }
    static constexpr int kBarOffset = kRingBytes;                                   // full[], empty[]
    static constexpr int kIssuedOffset = a16(kBarOffset + 2 * kNSlot * 8);          // int issued[kNSlot]
    static constexpr int kFlagOffset = a16(kIssuedOffset + kNSlot * 4);             // int flags[2]: abort, redo
    static constexpr int kScanOffset = a16(kFlagOffset + 8);                        // int warp sums[8]
    static constexpr int kRowsOffset = a16(kScanOffset + 8 * 4);                    // int rows[kNW][kRowQueue]
    static constexpr int kCountOffset = a16(kRowsOffset + kNW * kRowQueue * 4);     // int fill_cnt[kNW]
    static constexpr int kQsOffset = a16(kCountOffset + kNW * 4);                   // fp32 q per warp
    static constexpr int kQsBytes = MMA ? 0 : kNW * GMAX * D * 4;
    static constexpr int kPsOffset = a16(kQsOffset + kQsBytes);                     // fp32 p per warp
    static constexpr int kPsBytes = MMA ? 0 : kNW * GMAX * BS * 4;
    // FP8 append: the new token's 16-bit K and V source rows per warp, staged by cp.async
    static constexpr int kTokOffset = a16(kPsOffset + kPsBytes);
    static constexpr int kTokBytes = sizeof(T) == 1 ? kNW * 2 * D * 2 : 0;
    // (num_seqs + 1) ints of page prefix sums, then num_seqs clamped context lengths
    static constexpr int kPrefixOffset = a16(kTokOffset + kTokBytes);
    static constexpr int kFixedSmemBytes = kPrefixOffset + 1024;      // + slack to align the base
    static constexpr int kMaxSmemBytes = kFixedSmemBytes + (2 * kLeanMaxSeqs + 1) * 4;
    static int smem_bytes(int num_seqs) { return kFixedSmemBytes + (2 * num_seqs + 1) * 4; }
    // Resident CTAs per SM the register allocation aims for: PA_LEAN_MIN_BLOCKS, but no more
    // than shared memory allows (for short batches), and 2 for head_dim 256 (larger fragments).
    static constexpr int kSmemBlocks = (228 * 1024) / (kFixedSmemBytes + 1024);
    static constexpr int kMinBlocksRaw = PA_LEAN_MIN_BLOCKS < kSmemBlocks ? PA_LEAN_MIN_BLOCKS : kSmemBlocks;
    static constexpr int kMinBlocks = D > 128 ? (kMinBlocksRaw < 2 ? kMinBlocksRaw : 2)
                                              : (kMinBlocksRaw < 1 ? 1 : kMinBlocksRaw);
    static_assert(kMaxSmemBytes <= 227 * 1024, "shared memory per CTA");
    static_assert(kOOff % 4 == 0 && kRecFloats % 4 == 0, "16-byte aligned records");
    static_assert(kQsOffset % 16 == 0 && kPsOffset % 16 == 0, "alignment");
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// Exclusive prefix sum over the CTA's threads; *total receives the sum of all values.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int nwarps, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    int base = 0, tot = 0;
    for (int w = 0; w < nwarps; ++w) {
        const int ws = warp_sums[w];
        if (w < warp) base += ws;
        tot += ws;
    }
    *total = tot;
    return base + x - v;
}

// Global page g -> sequence b, unit within the sequence uu, page j within the unit, pages per unit nb.
// (The plan guarantees that all page indices, times units per sequence, fit in int.)
__device__ __forceinline__ void lean_locate(const int* pre, int num_seqs, int upb, int g, int& b, int& uu, int& j,
                                            int& nb) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] * upb <= g) lo = mid;
        else hi = mid - 1;
    }
    b = lo;
    nb = pre[b + 1] - pre[b];
    const int r = g - pre[b] * upb;
    uu = r / nb;
    j = r - uu * nb;
}


// F8: the caches hold E4M3 codes with a scale per (block, kv head) (MmaConsumerF8); T is then
// the query and output type.
// F8: E4M3 pages with per-(block, kv head) scales.  The append mode (the step's new token
// written inside the decode) is a runtime choice (new_key != nullptr) for the 16/32-bit caches
// and a separate instantiation (F8_APPEND) for FP8, whose consumer has no registers to spare
// for a path it does not take.
template <typename T, int D, int BS, bool MMA, int GMAX, bool CAUSAL, bool F8 = false, bool F8_APPEND = false>
__global__ void __launch_bounds__(DecodeCfg<T, D, BS, MMA, GMAX>::kThreads,
                                  (F8 ? PA_LEAN_F8_MIN_BLOCKS : LeanCfg<T, D, BS, MMA, GMAX>::kMinBlocks))
    paged_decode_lean_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                             const DecodeArgs a) {
    using C = LeanCfg<std::conditional_t<F8, uint8_t, T>, D, BS, MMA, GMAX>;
    static_assert(!F8 || (MMA && !CAUSAL), "the FP8 path is the single-query tensor-core consumer");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint64_t* empty = full + C::kNSlot;
    int* issued = reinterpret_cast<int*>(smem + C::kIssuedOffset);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + C::kFlagOffset);  // [0]: abort
    int* warp_sums = reinterpret_cast<int*>(smem + C::kScanOffset);
    int* pre = reinterpret_cast<int*>(smem + C::kPrefixOffset);
    int* lens_s = pre + (a.num_seqs + 1);  // the context lengths, clamped to the tables

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int B = a.num_seqs;
    const int l_cap = a.max_blocks * BS;
    T* out = static_cast<T*>(a.out);

    // ---- set-up, started before the dependency wait ----
    // The shared-memory pipeline state touches no global memory: initialise it first.
    if (tid == 0) {
        for (int s = 0; s < C::kNSlot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            issued[s] = 0;
        }
        flags[0] = 0;  // abort
        flags[1] = 0;  // the set-up guess was wrong
        fence_barrier_init();
    }
    int* row_queue = reinterpret_cast<int*>(smem + C::kRowsOffset);                   // [kNW][kRowQueue]
    volatile int* fill_cnt = reinterpret_cast<volatile int*>(smem + C::kCountOffset);  // [kNW]
    int* queue = row_queue + min(warp, C::kNW - 1) * C::kRowQueue;                     // this consumer warp's rows
    const int upb = a.num_kv_heads * a.head_chunks;  // units per sequence
    const int wg = (int)blockIdx.x * C::kNW + warp;   // a consumer warp's share index
    const int per = (B + C::kThreads - 1) / C::kThreads;
    const int b_lo = min(B, tid * per);
    const int b_hi = min(B, b_lo + per);
    int total = 0, q_per_warp = 0, lo = 0, hi = 0, n = 0;
    // consumer warps the pages are cut for (equal shares rounded up; the warps past them idle)
    const int share_warps = max(1, min(a.lean_share_warps, (int)gridDim.x * C::kNW));
    int my_len = 0;  // the (clamped) length of this thread's sequence when it has exactly one
    int first_pb = -1, first_kvh = 0;  // a consumer lane's page `lane` of its share: block id, kv head
    size_t first_at = 0;               // and its block-table index
    // Pages per sequence (context lengths clamped to the table), their prefix sums, this warp's
    // share and the tensor rows of its first 32 pages (published to the producer).  `guess`: run
    // before the wait, while the previous grid in the stream may still be writing the lengths or
    // the tables; every load goes through L2 only (no stale line may stay in L1), and whatever it
    // read is read again and compared after the wait.
    auto setup = [&](bool guess) {
        int mine = 0;
        for (int b = b_lo; b < b_hi; ++b) {
            int L = __ldcg(a.context_lens + b);
            if (L < 0 || L > l_cap) {
                if (!guess && blockIdx.x == 0) atomicOr(a.err, kErrBadContext);
                L = L < 0 ? 0 : l_cap;
            }
            lens_s[b] = L;
            my_len = L;
            pre[b] = (L + BS - 1) / BS;
            mine += pre[b];
        }
        int total_pages = 0;
        int acc = block_exclusive_scan(mine, warp_sums, C::kNW + 1, &total_pages);
        for (int b = b_lo; b < b_hi; ++b) {
            const int nb_ = pre[b];
            pre[b] = acc;
            acc += nb_;
        }
        if (tid == 0) {
            pre[B] = total_pages;
            for (int w = 0; w < C::kNW; ++w) fill_cnt[w] = 0;  // no page rows published yet
        }
        __syncthreads();
        total = total_pages * upb;
        q_per_warp = (total + share_warps - 1) / share_warps;
        lo = min(total, wg * q_per_warp);
        hi = min(total, lo + q_per_warp);
        n = warp < C::kNW ? hi - lo : 0;
        first_pb = -1;
        if (lane < n) {
            int sb, su, sj, sn;
            lean_locate(pre, B, upb, lo + lane, sb, su, sj, sn);
            first_kvh = su / a.head_chunks;
            first_at = (size_t)sb * a.max_blocks + sj;
            first_pb = __ldcg(a.block_tables + first_at);
            queue[lane] = (unsigned)first_pb < (unsigned)a.num_blocks ? (first_pb * a.num_kv_heads + first_kvh) * BS
                                                                      : -1;
        }
        __syncwarp();
        if (warp < C::kNW && lane == 0) {
            __threadfence_block();
            fill_cnt[warp] = min(n, 32);
        }
        __syncthreads();  // every warp's first rows are published before the producer's first pass
    };

    // The producer lane's state (lane 0 of warp kNW).  Each consumer warp publishes the TMA rows
    // of its own pages well ahead (row_queue / fill_cnt); the producer only polls the page slots
    // and issues the next published page of every warp that has a free slot.  It never waits on
    // global memory and never waits behind one particular warp.
    static_assert(C::kNW == 4, "the issue loop is unrolled for four consumer warps");
    int iss[C::kNW], n_w[C::kNW];
    const bool producer = warp == C::kNW && lane == 0;
    // Pages are read once per call: let them leave L2 first, so that the partial records the merge
    // reads stay resident.
    const uint64_t stream_policy = producer ? l2_policy_evict_first() : 0;
    auto producer_start = [&]() {
#pragma unroll
        for (int wi = 0; wi < C::kNW; ++wi) {
            iss[wi] = 0;
            const int lo_w = min(total, ((int)blockIdx.x * C::kNW + wi) * q_per_warp);
            n_w[wi] = min(total, lo_w + q_per_warp) - lo_w;
        }
    };
    // One pass over the consumer warps; returns whether every page of the CTA has been issued.
    auto issue_pass = [&](bool& progress, bool one_each = false) -> bool {
        bool done = true;
#pragma unroll
        for (int wi = 0; wi < C::kNW; ++wi) {
            const int avail = fill_cnt[wi];
            __threadfence_block();  // the rows below were written before fill_cnt
            // FP8 pages (4 KB, four slots a warp): at most one page per warp and pass, round robin
            // over the warps (measured: 13 % on long contexts, 9 % on the Qwen-shaped step);
            // 16-bit pages (two slots a warp): every free slot at once (one page per pass cost 2 %
            // there).
            for (int burst = 0; iss[wi] < avail && (!(F8 || one_each) || burst == 0); ++burst) {
                const int s = wi * C::kSPW + iss[wi] % C::kSPW;
                const int use = iss[wi] / C::kSPW;
                if (use >= 1 && !mbar_test_wait(&empty[s], (use - 1) & 1)) break;
                const int r = row_queue[wi * C::kRowQueue + iss[wi] % C::kRowQueue];
                issued[s] += 1;
                if (r >= 0) {
                    mbar_arrive_expect_tx(&full[s], C::kSlotBytes);
                    uint8_t* kdst = ring + s * C::kSlotBytes;
                    uint8_t* vdst = kdst + C::kPageBytes;
                    if (F8 && a.kv_interleaved) {
                        // K rows 2r .. 2r + BS - 1, then V: one box of 2 * BS rows (one 128-byte box
                        // a row at head_dim 128), landing as the K page followed by the V page
                        static_assert(!F8 || C::Base::kNBox == 1, "one box per FP8 row");
                        tma_load_2d_hint(kdst, &tmap_k, 0, 2 * r, &full[s], stream_policy);
                    } else {
#pragma unroll
                        for (int bx = 0; bx < C::Base::kNBox; ++bx)
                            tma_load_2d_hint(kdst + bx * C::Base::kBoxBytes, &tmap_k, bx * C::Base::kBoxElems, r,
                                             &full[s], stream_policy);
#pragma unroll
                        for (int bx = 0; bx < C::Base::kNBox; ++bx)
                            tma_load_2d_hint(vdst + bx * C::Base::kBoxBytes, &tmap_v, bx * C::Base::kBoxElems, r,
                                             &full[s], stream_policy);
                    }
                } else {
                    atomicOr(a.err, kErrBadTable);  // skip the load; the slot keeps stale data
                    mbar_arrive(&full[s]);
                }
                ++iss[wi];
                progress = true;
            }
            done = done && iss[wi] >= n_w[wi];
        }
        return done;
    };

    if (producer) {
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_v);
    }
#if PA_LEAN_L2_PREFETCH
    {   // warm L2 with this CTA's share of the block tables (prefetches return no data)
        const long long tab_bytes = (long long)B * a.max_blocks * 4;
        const long long share = (tab_bytes + gridDim.x - 1) / gridDim.x;
        const char* tab = reinterpret_cast<const char*>(a.block_tables) + share * blockIdx.x;
        for (long long off = tid * 128; off < share && share * blockIdx.x + off < tab_bytes; off += C::kThreads * 128)
            prefetch_l2(tab + off);
    }
#endif
    __syncthreads();  // barrier initialisation before any use
    setup(true);
    // Warm L2 with each consumer warp's first pages (one per ring slot) on the guess, before the wait:
    // the previous grid is then still finishing and HBM is otherwise idle.  A prefetch returns no data,
    // and a later write by the previous grid goes through L2, so a stale guess costs only bandwidth
    // (measured: the Qwen-shaped call 52.6 -> 51.8 us, long context 310.8 -> 307.2 us).
    if (warp < C::kNW && lane < min(n, C::kSPW)) {
        const int r = queue[lane];
        if (r >= 0) {
            if (F8 && a.kv_interleaved) {
                tma_prefetch_l2_2d(&tmap_k, 0, 2 * r);
            } else {
#pragma unroll
                for (int bx = 0; bx < C::Base::kNBox; ++bx) {
                    tma_prefetch_l2_2d(&tmap_k, bx * C::Base::kBoxElems, r);
                    tma_prefetch_l2_2d(&tmap_v, bx * C::Base::kBoxElems, r);
                }
            }
        }
    }
    // Wait for the previous grid in the stream, then let the merge kernel get scheduled as
    // early as possible; it reads nothing this kernel writes before its own wait.
    griddep_wait();
    griddep_launch_dependents();
    // ---- consumer state (consumer warps only) ----
    int unit_first = 0, unit_last = -1;
    int b = 0, uu = 0, nb = 0, L = 0, gc = 0, kvh = 0;
    UnitRows rows{0, 0, 0, a.q_len, a.group, a.num_heads};
    int wrote = 0;  // bit s: a partial record was written to slot s
    const bool append = F8 ? F8_APPEND : a.new_key != nullptr;
    std::conditional_t<F8, NewTokenF8<T, D, BS>, NewToken<T, D, BS>> tok;
    if constexpr (F8) tok.stage = smem + C::kTokOffset + min(warp, C::kNW - 1) * 4 * D;
    bool tok_ready = false, tok_writer = false;
    std::conditional_t<F8, MmaConsumerF8<T, D, BS>,
                       std::conditional_t<MMA, MmaConsumer<T, D, BS, CAUSAL>, SimtConsumer<T, D, BS, GMAX>>>
        cons;
    float* q_s = reinterpret_cast<float*>(smem + C::kQsOffset) + min(warp, C::kNW - 1) * GMAX * D;
    float* p_s = reinterpret_cast<float*>(smem + C::kPsOffset) + min(warp, C::kNW - 1) * GMAX * BS;
    // The unit holding global page g starts: its place, its length (from shared memory) and its
    // query rows (loaded here; a load on the consumer's critical path).
    auto start_unit = [&](int g) {
        int j0;
        lean_locate(pre, B, upb, g, b, uu, j0, nb);
        unit_first = g - j0;
        unit_last = unit_first + nb - 1;
        kvh = uu / a.head_chunks;
        const int hc = uu - kvh * a.head_chunks;
        tok_writer = hc == 0;
        rows = UnitRows{b, kvh, hc * C::kHeads, a.q_len, a.group, a.num_heads};
        gc = min(C::kHeads, a.rows - hc * C::kHeads);
        L = lens_s[b];
        const T* q = static_cast<const T*>(a.q);
        if constexpr (F8) {
            const int r = min(lane >> 2, gc - 1);
            cons.init(q + rows.row(r) * D, (lane >> 2) < gc, a.scale_log2, lane);
        } else if constexpr (MMA) {
            const int r = min(lane >> 2, gc - 1);
            cons.init(q + rows.row(r) * D, (lane >> 2) < gc, rows.last_pos(2 * (lane & 3), L),
                      rows.last_pos(2 * (lane & 3) + 1, L), lane);
        } else {
            __syncwarp();
            for (int idx = lane; idx < GMAX * D; idx += 32)
                q_s[idx] = idx / D < gc ? to_float(q[rows.row(idx / D) * D + idx % D]) : 0.f;
            __syncwarp();
            cons.init(L - a.q_len, rows.v0, a.group);
        }
    };

    // After the wait, in this order: the small loads (the re-reads that check the guess, every
    // consumer warp's first query rows), the producer's first page loads, then the check; the
    // consumers then go straight to their first page.  Between the first page loads and the
    // first page nothing here touches shared memory (the check compares registers and decides
    // with one barrier): while a burst of page copies is being issued, other memory
    // instructions of the SM wait behind it.
    int chk_len = 0, chk_pb = 0;
    for (int bb = b_lo; bb < b_hi; ++bb) chk_len = __ldcg(a.context_lens + bb);  // B <= threads: one each
    if (lane < n) chk_pb = __ldcg(a.block_tables + first_at);
    if (warp < C::kNW && n > 0) start_unit(lo);
    __syncthreads();
    if (producer) {  // the first pages go out at once, on the guess: one per warp (a smaller burst)
        producer_start();
        bool progress = false;
        issue_pass(progress, true);
    }
    bool bad = a.force_restart != 0;
    if (b_hi - b_lo == 1) {
        int Lc = chk_len;
        if (Lc < 0 || Lc > l_cap) {
            if (blockIdx.x == 0) atomicOr(a.err, kErrBadContext);
            Lc = Lc < 0 ? 0 : l_cap;
        }
        bad = bad || Lc != my_len;
    } else {
        for (int bb = b_lo; bb < b_hi; ++bb) {
            int Lc = __ldcg(a.context_lens + bb);
            if (Lc < 0 || Lc > l_cap) {
                if (blockIdx.x == 0) atomicOr(a.err, kErrBadContext);
                Lc = Lc < 0 ? 0 : l_cap;
            }
            bad = bad || Lc != lens_s[bb];
        }
    }
    if (lane < n && chk_pb != first_pb) bad = true;
    bool aborted = false;
    if (__syncthreads_or(bad)) {
        // The guess was wrong (rare: the previous grid changed the lengths or the tables).  Let the
        // copies issued from it land, discard them, and set up again from the values read now.
        bool drained = true;
        if (tid == 0) {
            for (int s = 0; s < C::kNSlot; ++s) {
                if (issued[s] == 0) continue;
                const unsigned long long start = global_timer_ns();
                while (!mbar_try_wait(&full[s], (issued[s] - 1) & 1)) {
                    if (global_timer_ns() - start > kWaitLimitNs) {
                        drained = false;
                        break;
                    }
                }
            }
            if (drained) {
                for (int s = 0; s < C::kNSlot; ++s) {
                    mbar_inval(&full[s]);
                    mbar_inval(&empty[s]);
                    mbar_init(&full[s], 1);
                    mbar_init(&empty[s], 1);
                    issued[s] = 0;
                }
                fence_barrier_init();
            } else {
                atomicOr(a.err, kErrTimeout);
                flags[0] = 1;  // the copies never landed: give up (the exit path drains again)
            }
        }
        aborted = __syncthreads_or(!drained) != 0;
        if (!aborted) {
            setup(false);
            if (producer) producer_start();
            if (warp < C::kNW && n > 0) start_unit(lo);
        }
    }
    if (total == 0 && !aborted) {
        // Nothing to stream: only the zero rows of empty contexts (spread over the CTAs).
        for (int bz = warp; bz < B; bz += C::kNW + 1)
            if ((bz % (int)gridDim.x) == (int)blockIdx.x)
                for (int idx = lane; idx < a.q_len * a.num_heads * D; idx += 32)
                    out[(size_t)bz * a.q_len * a.num_heads * D + idx] = from_float<T>(0.f);
        return;
    }

    if (warp == C::kNW) {
        // ================= producer warp =================
        if (producer && !aborted) {
            unsigned long long last_progress = global_timer_ns();
            while (true) {
                bool progress = false;
                if (issue_pass(progress)) break;
                if (progress) {
                    last_progress = global_timer_ns();
                } else {
                    if (flags[0]) break;
                    if (global_timer_ns() - last_progress > kWaitLimitNs) {
                        atomicOr(a.err, kErrTimeout);
                        flags[0] = 1;
                        break;
                    }
                    __nanosleep(PA_PRODUCER_NAP_NS);
                }
            }
        }
    } else if (!aborted) {
        // ================= consumer warps =================
        // FP8: lane i holds the K and V scales of page 32 * chunk + i of the current chunk
        // (cur_*) and of the next one (pend_*, loaded when that chunk is published).
        float cur_ks = 0.f, cur_vs = 0.f, pend_ks = 0.f, pend_vs = 0.f;
        if constexpr (F8) {
            const bool ok = lane < n && (unsigned)first_pb < (unsigned)a.num_blocks;
            cur_ks = ok ? __ldg(a.k_scale + first_pb * a.num_kv_heads + first_kvh) : 0.f;
            cur_vs = ok ? __ldg(a.v_scale + first_pb * a.num_kv_heads + first_kvh) : 0.f;
        }
        // Page rows for the producer, published in chunks of 32: chunk c + 1 when this warp
        // reaches page 32c + 16, with the block-table loads of chunk c + 2 then left in flight.
        int pend_pb = -1, pend_kvh = 0;
        if (32 + lane < n) {
            int sb, su, sj, sn;
            lean_locate(pre, B, upb, lo + 32 + lane, sb, su, sj, sn);
            pend_kvh = su / a.head_chunks;
            pend_pb = __ldg(a.block_tables + (size_t)sb * a.max_blocks + sj);
        }
        for (int off = 0; off < n; ++off) {
            if constexpr (F8) {
                if ((off & 31) == 0 && off > 0) {
                    cur_ks = pend_ks;
                    cur_vs = pend_vs;
                }
            }
            if ((off & 31) == 16) {
                const int c = (off >> 5) + 1;  // the chunk published now
                const int page = 32 * c + lane;
                if constexpr (F8) {
                    const bool ok = page < n && (unsigned)pend_pb < (unsigned)a.num_blocks;
                    pend_ks = ok ? __ldg(a.k_scale + pend_pb * a.num_kv_heads + pend_kvh) : 0.f;
                    pend_vs = ok ? __ldg(a.v_scale + pend_pb * a.num_kv_heads + pend_kvh) : 0.f;
                }
                if (page < n)
                    queue[page % C::kRowQueue] = (unsigned)pend_pb < (unsigned)a.num_blocks
                                                     ? (pend_pb * a.num_kv_heads + pend_kvh) * BS
                                                     : -1;
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    fill_cnt[warp] = min(n, 32 * (c + 1));
                }
                const int next = page + 32;
                pend_pb = -1;
                if (next < n) {
                    int sb, su, sj, sn;
                    lean_locate(pre, B, upb, lo + next, sb, su, sj, sn);
                    pend_kvh = su / a.head_chunks;
                    pend_pb = __ldg(a.block_tables + (size_t)sb * a.max_blocks + sj);
                }
            }
            const int g = lo + off;
            if (g > unit_last) start_unit(g);  // a new unit starts
            const int j = g - unit_first;
            // Append mode: fetch the new token one page ahead of the page holding L - 1.
            const bool tok_page = append && g == unit_last;
            if (append && (g + 1 == unit_last || (tok_page && !tok_ready))) {
                const size_t nt = ((size_t)b * a.num_kv_heads + kvh) * D;
                tok.load(static_cast<const T*>(a.new_key) + nt, static_cast<const T*>(a.new_value) + nt, lane);
                tok_ready = true;
            }
            const int s = warp * C::kSPW + off % C::kSPW;
            const bool got = mbar_wait_bounded(&full[s], (off / C::kSPW) & 1, a.err, flags);
            if (!__all_sync(0xffffffffu, got)) break;
            const int nvalid = min(BS, L - j * BS);
            uint8_t* kp = ring + s * C::kSlotBytes;
            float ks = 0.f, vs = 0.f;  // FP8: this page's K and V scales
            if constexpr (F8) {
                ks = __shfl_sync(0xffffffffu, cur_ks, off & 31);
                vs = __shfl_sync(0xffffffffu, cur_vs, off & 31);
            }
            if (tok_page) {
                const int row = queue[off % C::kRowQueue];  // (pb * Hkv + kvh) * BS, or -1
                if constexpr (F8) {
                    tok.patch(kp, kp + C::kPageBytes, nvalid - 1, ks, vs, lane);
                    if (tok_writer && row >= 0)
                        tok.store(a.key_cache, a.value_cache, row, nvalid - 1, a.kv_interleaved != 0, lane);
                } else {
                    tok.patch(kp, kp + C::kPageBytes, nvalid - 1, lane);
                    if (tok_writer && row >= 0) tok.store(a.key_cache, a.value_cache, row + nvalid - 1, lane);
                }
                tok_ready = false;
            }
            if constexpr (F8) {
                cons.page(kp, kp + C::kPageBytes, nvalid, ks, vs, lane);
                __syncwarp();
            } else if constexpr (MMA) {
                cons.page(kp, kp + C::kPageBytes, nvalid, j * BS, a.scale_log2, lane);
                __syncwarp();
            } else {
                cons.page(kp, kp + C::kPageBytes, nvalid, j * BS, a.scale_log2, q_s, p_s, lane);
            }
            if (lane == 0) mbar_arrive(&empty[s]);

            if (g == unit_last || off == n - 1) {  // this warp is done with the unit
                cons.finish();
                if (unit_first >= lo && unit_last < hi) {
                    cons.write_out(out, rows, gc, lane);
                    cons.clear();
                } else {
                    const int slot = unit_first <= lo ? 0 : 1;  // 0: the warp's first unit, 1: its last
                    float* rec = a.ws_part + ((size_t)wg * 2 + slot) * C::kRecFloats;
                    cons.write_partial(rec, gc, lane);
                    cons.clear();
                    wrote |= 1 << slot;
                }
            }
            if (off == n - 1 && wrote) {
                // Publish the records for the merge kernel, once, after the warp's last page
                // (a GPU-scope fence in the middle of the page stream would stall it).  The warp
                // barrier orders every lane's record stores before lane 0's release stores, and a
                // release is cumulative: a merge that acquires the flag sees the whole record (a
                // separate fence before them cost 0.5 us at the end of the Qwen-shaped step).
                __syncwarp();
                if (lane == 0) {
                    if (wrote & 1) st_release_gpu(a.ws_flag + (size_t)wg * 2, a.epoch);
                    if (wrote & 2) st_release_gpu(a.ws_flag + (size_t)wg * 2 + 1, a.epoch);
                }
            }
        }
        // A token copy may still be in flight when a wait gave up before its page.
        if constexpr (F8 && F8_APPEND) cp_async_wait_all();
        // Empty contexts produce zero rows (spread over the CTAs), written once the pages are done.
        for (int bz = warp; bz < B; bz += C::kNW)
            if (pre[bz] == pre[bz + 1] && (bz % (int)gridDim.x) == (int)blockIdx.x)
                for (int idx = lane; idx < a.q_len * a.num_heads * D; idx += 32)
                    out[(size_t)bz * a.q_len * a.num_heads * D + idx] = from_float<T>(0.f);
    }
    __syncthreads();
    if (flags[0]) {
        // A wait gave up: let every issued copy land before the CTA's shared memory goes away.
        if (tid == 0)
            for (int s = 0; s < C::kNSlot; ++s)
                if (issued[s] > 0) {
                    const unsigned long long start = global_timer_ns();
                    while (!mbar_try_wait(&full[s], (issued[s] - 1) & 1) &&
                           global_timer_ns() - start < kWaitLimitNs) {
                    }
                }
    }
}


#ifndef PA_LEAN_MERGE_THREADS
#define PA_LEAN_MERGE_THREADS 256
#endif
#ifndef PA_LEAN_MERGE_MINB
#define PA_LEAN_MERGE_MINB 2
#endif
constexpr int kLeanMergeThreads = PA_LEAN_MERGE_THREADS;
constexpr int kLeanMergeBatch = 8;  // records whose loads a thread keeps in flight together

// Lean merge: one CTA per (sequence, kv head, head chunk) unit.  A unit that the lean
// decode cut between consumer warps w_lo..w_hi left one partial record per warp
// (m, l, o~ per head); the merge combines them with the online-softmax rule,
//     M = max_p m_p,  W = sum_p 2^(m_p - M) l_p,  o = sum_p 2^(m_p - M) o~_p / W.
// Units that fit in one warp's range were finished by the decode kernel.
// Launched with programmatic stream serialisation, the merge runs while the decode
// drains: the unit's place in the page order is recomputed from the context lengths,
// then the CTA waits for the flags of its unit's records (each warp of the decode
// publishes its records once its pages are done) rather than for the whole decode
// grid, merges, and only then waits for the decode grid to complete, so that a grid
// after this one still sees the decode finished.  Reading the lengths early is safe:
// this grid starts only once every decode CTA has passed its own wait for the grids
// before it.  Every thread merges its own float4 columns of o~ over all records on its
// own: no barriers, all loads of a batch of records issued before any is used.
// Merge launch of a lean decode of `grid` CTAs: one CTA per unit, or, when units outnumber the
// decode's consumer warps, one per boundary between two warps' shares (a unit is cut only at
// such a boundary).  Sets the merge's fields of m; returns its grid size.
inline int lean_merge_setup(DecodeArgs& m, int grid) {
    const long long units = (long long)m.num_seqs * m.num_kv_heads * m.head_chunks;
    const long long warps = (long long)grid * m.lean_warps_per_cta;
    m.lean_grid = grid;
    m.lean_merge_by_boundary = units > warps ? 1 : 0;
    return (int)(m.lean_merge_by_boundary ? (warps > 1 ? warps - 1 : 1) : units);
}

template <typename T, int D, int H, int BS>
__global__ void __launch_bounds__(kLeanMergeThreads, PA_LEAN_MERGE_MINB) lean_merge_kernel(const DecodeArgs a) {
    constexpr int kOOff = ((2 * H + 3) / 4) * 4;
    constexpr int kRec = kOOff + H * D;
    __shared__ int warp_sums[kLeanMergeThreads / 32];
    __shared__ int seq_before[2];  // pages of the sequences before b, pages of b
    griddep_launch_dependents();  // the next grid waits for this one's completion itself
    const int tid = threadIdx.x;
    const int upb = a.num_kv_heads * a.head_chunks;
    const int B = a.num_seqs;
    const int l_cap = a.max_blocks * BS;
    const int warps = a.lean_grid * a.lean_warps_per_cta;
    const int share_warps = max(1, min(a.lean_share_warps, warps));  // as the decode cuts its shares
    auto pages_of = [&](int s) {  // pages of sequence s, its length clamped like the decode's
        int L = __ldg(a.context_lens + s);
        L = L < 0 ? 0 : (L > l_cap ? l_cap : L);
        return (L + BS - 1) / BS;
    };

    // This CTA's unit (b, uu): its sequence's page count nb, the pages of the sequences before
    // it (pre_b) and the total tot.  One CTA per unit, or, when units outnumber the decode's
    // warps, one per boundary w = blockIdx.x + 1 between the shares of warps w - 1 and w: the
    // CTA takes the unit holding the boundary's first page and merges it only if this is the
    // first boundary inside it (so every cut unit is merged once, with far fewer CTAs).
    int b, uu, nb, pre_b, tot, q;
    bool skip = false;
    if (!a.lean_merge_by_boundary) {
        b = blockIdx.x / upb;
        uu = blockIdx.x - b * upb;
        int before = 0, all = 0;
        for (int s = tid; s < B; s += kLeanMergeThreads) {
            const int n = pages_of(s);
            all += n;
            if (s < b) before += n;
            if (s == b) seq_before[1] = n;
        }
        block_exclusive_scan(all, warp_sums, kLeanMergeThreads / 32, &tot);
        __syncthreads();
        block_exclusive_scan(before, warp_sums, kLeanMergeThreads / 32, &pre_b);
        __syncthreads();
        nb = seq_before[1];
        q = (tot * upb + share_warps - 1) / share_warps;
    } else {
        // contiguous runs of sequences per thread, so that a thread's scan base is their prefix
        const int chunk = (B + kLeanMergeThreads - 1) / kLeanMergeThreads;
        const int s0 = min(B, tid * chunk), s1 = min(B, s0 + chunk);
        int mine = 0;
        for (int s = s0; s < s1; ++s) mine += pages_of(s);
        if (tid == 0) seq_before[0] = -1;
        int run = block_exclusive_scan(mine, warp_sums, kLeanMergeThreads / 32, &tot);
        __syncthreads();
        q = (tot * upb + share_warps - 1) / share_warps;
        const int P = (blockIdx.x + 1) * q;  // first page of warp blockIdx.x + 1
        for (int s = s0; s < s1; ++s) {
            const int n = pages_of(s);
            if (P >= run * upb && P < (run + n) * upb) {
                seq_before[0] = s;
                seq_before[1] = n;
                warp_sums[0] = run;  // (the scan is done with warp_sums)
            }
            run += n;
        }
        __syncthreads();
        b = seq_before[0];
        nb = seq_before[1];
        pre_b = warp_sums[0];
        skip = b < 0;
        if (!skip) {
            uu = (P - pre_b * upb) / nb;
            const int first = pre_b * upb + uu * nb;
            skip = first == P || first / q + 1 != (int)blockIdx.x + 1;
        }
    }
    const int first = skip ? 0 : pre_b * upb + uu * nb;
    const int w_lo = q > 0 ? first / q : 0, w_hi = q > 0 ? (first + nb - 1) / q : 0;
    if (skip || nb == 0 || q <= 0 || w_lo == w_hi) {
        // Nothing to merge (the decode kernel finished the unit).  Every CTA still waits
        // for the decode grid before it ends: a grid that follows this one waits only for
        // this grid, so this grid must not end before the decode has.
        griddep_wait();
        return;
    }
    const int n = w_hi - w_lo + 1;
    const int slot0 = first != w_lo * q ? 1 : 0;  // w_lo holds the unit in slot 1 unless its range starts here
    // The pieces' records are folded batch by batch, each batch as soon as the flags of its pieces
    // read this call's epoch (each warp of the decode publishes its records once its pages are
    // done), not after the whole decode grid nor after every piece: a batch whose pieces are
    // done is folded while the pieces of a later batch are still streaming.  Each wait is
    // bounded; one that gives up reports kErrTimeout and the CTA writes nothing.
    __shared__ volatile int gave_up;
    if (tid == 0) gave_up = 0;
    __syncthreads();
    const int kvh = uu / a.head_chunks, hc = uu - kvh * a.head_chunks;
    const UnitRows rows{b, kvh, hc * H, a.q_len, a.group, a.num_heads};
    const int gc = min(H, a.rows - hc * H);
    const float* base = a.ws_part + (size_t)w_lo * 2 * kRec;

    // thread = (float4 column of the gc live heads, slice of the records): each thread folds
    // its records (online), then slice 0 folds the slices' (max, denominator, o~) triples.
    __shared__ float red[6][kLeanMergeThreads];
    const int cols = gc * (D / 4);
    const int slices = kLeanMergeThreads >= cols ? kLeanMergeThreads / cols : 1;
    const int per_batch = kLeanMergeBatch * slices;  // records of one batch, over all slices
    for (int cbase = 0; cbase < cols; cbase += kLeanMergeThreads) {
    const int col = slices > 1 ? tid % cols : cbase + tid;
    const int slice = slices > 1 ? tid / cols : (col < cols ? 0 : 1);
    const int h = col / (D / 4);
    float mm = -INFINITY, ww = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int pb = 0; pb < n; pb += per_batch) {
        for (int p = pb + tid; p < min(n, pb + per_batch); p += kLeanMergeThreads) {
            const unsigned long long* f = a.ws_flag + (size_t)(w_lo + p) * 2 + (p == 0 ? slot0 : 0);
            if (ld_acquire_gpu(f) == a.epoch) continue;
            const unsigned long long start = global_timer_ns();
            while (ld_acquire_gpu(f) != a.epoch) {
                if (gave_up || global_timer_ns() - start > a.wait_ns) {
                    if (!gave_up) atomicOr(a.err, kErrTimeout);
                    gave_up = 1;
                    break;
                }
                __nanosleep(32);
            }
        }
        __syncthreads();
        if (gave_up) break;
        if (slice < slices) {
            const int p0 = pb + slice;
            float mv[kLeanMergeBatch], lv[kLeanMergeBatch];
            float4 ov[kLeanMergeBatch];
#pragma unroll
            for (int k = 0; k < kLeanMergeBatch; ++k) {
                const int p = p0 + k * slices;
                if (p < n) {
                    const float* r = base + ((size_t)p * 2 + (p == 0 ? slot0 : 0)) * kRec;
                    mv[k] = __ldcg(r + h);
                    lv[k] = __ldcg(r + H + h);
                    ov[k] = __ldcg(reinterpret_cast<const float4*>(r + kOOff) + col);
                }
            }
#pragma unroll
            for (int k = 0; k < kLeanMergeBatch; ++k) {
                if (p0 + k * slices < n) {
                    if (mv[k] == -INFINITY) continue;  // a piece the row's causal bound excludes
                    const float m_new = fmaxf(mm, mv[k]);
                    const float keep = exp2f(mm - m_new);  // 0 on the first record
                    const float f = exp2f(mv[k] - m_new);
                    ww = ww * keep + f * lv[k];
                    acc.x = acc.x * keep + f * ov[k].x;
                    acc.y = acc.y * keep + f * ov[k].y;
                    acc.z = acc.z * keep + f * ov[k].z;
                    acc.w = acc.w * keep + f * ov[k].w;
                    mm = m_new;
                }
            }
        }
    }
    if (gave_up) break;
    if (slices > 1) {
        red[0][tid] = mm;
        red[1][tid] = ww;
        red[2][tid] = acc.x;
        red[3][tid] = acc.y;
        red[4][tid] = acc.z;
        red[5][tid] = acc.w;
        __syncthreads();
        if (slice == 0) {
            for (int k = 1; k < slices; ++k) {
                const int t = k * cols + col;
                const float m2 = red[0][t];
                const float m_new = fmaxf(mm, m2);
                if (m_new == -INFINITY) continue;  // both slices empty
                const float k1 = rescale(mm, m_new), k2 = rescale(m2, m_new);
                ww = ww * k1 + red[1][t] * k2;
                acc.x = acc.x * k1 + red[2][t] * k2;
                acc.y = acc.y * k1 + red[3][t] * k2;
                acc.z = acc.z * k1 + red[4][t] * k2;
                acc.w = acc.w * k1 + red[5][t] * k2;
                mm = m_new;
            }
        }
    }
    if (slice == 0) {
        const float inv = ww > 0.f ? 1.f / ww : 0.f;  // 0: the row attends no position
        T* out = static_cast<T*>(a.out) + rows.row(h) * D + (col - h * (D / 4)) * 4;
        out[0] = from_float<T>(acc.x * inv);
        out[1] = from_float<T>(acc.y * inv);
        out[2] = from_float<T>(acc.z * inv);
        out[3] = from_float<T>(acc.w * inv);
    }
    }
    // Every flag is read by this CTA alone: clear the ones it consumed, so that the next call on
    // this workspace starts from zeros even if it reuses this call's epoch (a replayed capture).
    if (!gave_up)
        for (int p = tid; p < n; p += kLeanMergeThreads)
            a.ws_flag[(size_t)(w_lo + p) * 2 + (p == 0 ? slot0 : 0)] = 0ull;
    griddep_wait();  // this grid must not end before the decode grid has
}

// ------------------------------------------------------------------------------------------
// ------------------------------------------------------------------------------------------
// Persistent row-split schedule (multi-query decode: a kv head's rows in 2..4 chunks of 8).
// One wave of CTAs.  The pages of all (sequence, kv head) units, laid end to end (sequence-major,
// then kv head, pages in logical order), are cut into equal contiguous shares, one per CTA.  The
// producer warp streams its share's pages once through the ring and consumer warp w takes row
// chunk w of every page, so each page is read once for all of its kv head's rows and every CTA
// streams the same number of pages whatever the context lengths are.  A unit that lies wholly
// inside a share is written out by its CTA; a unit cut by a share boundary leaves one partial
// record per row chunk in each CTA it spans (slot 0: the share's first unit, slot 1: its last
// unit), and rs_lean_merge_kernel combines them.
template <typename T, int D, int BS>
struct RsLeanCfg {
    using C = DecodeCfg<T, D, BS, true, 8>;
    static constexpr int kMaxChunks = 4;
    static constexpr int kRecFloats = 16 + 8 * D;  // m[8], l[8], o~[8][D] (MmaConsumer::write_partial)
    // (num_seqs + 1) ints of page prefix sums, then num_seqs clamped context lengths
    static constexpr int kPrefixOffset = C::a16(C::kFlagOffset + 16);
    static int smem_bytes(int num_seqs) { return kPrefixOffset + (2 * num_seqs + 1) * 4 + 1024; }
    static constexpr int kMaxSmemBytes = kPrefixOffset + (2 * kLeanMaxSeqs + 1) * 4 + 1024;
    static_assert(C::kStatBytes >= (C::kNW + 1) * 4, "the scan's warp sums live in the stat area");
    static_assert(C::kNW >= kMaxChunks, "a consumer warp per row chunk");
};

// Pages per sequence (context lengths clamped to the tables: [0, max_blocks * BS]) and their
// exclusive prefix sums into pre[0 .. B]; lens[b] receives the clamped length.  Every thread of
// the CTA calls it.
template <int BS>
__device__ __forceinline__ void rs_page_prefix(const int32_t* context_lens, int B, int max_blocks, int* pre, int* lens,
                                               int* warp_sums, int nwarps, bool report, unsigned* err) {
    const int nthreads = nwarps * 32;
    const int l_cap = max_blocks * BS;
    const int per = (B + nthreads - 1) / nthreads;
    const int b_lo = min(B, (int)threadIdx.x * per);
    const int b_hi = min(B, b_lo + per);
    int mine = 0;
    for (int b = b_lo; b < b_hi; ++b) {
        int L = __ldcg(context_lens + b);
        if (L < 0 || L > l_cap) {
            if (report) atomicOr(err, kErrBadContext);
            L = L < 0 ? 0 : l_cap;
        }
        if (lens) lens[b] = L;
        pre[b] = (L + BS - 1) / BS;
        mine += pre[b];
    }
    int total = 0;
    int acc = block_exclusive_scan(mine, warp_sums, nwarps, &total);
    for (int b = b_lo; b < b_hi; ++b) {
        const int nb = pre[b];
        pre[b] = acc;
        acc += nb;
    }
    if (threadIdx.x == 0) pre[B] = total;
    __syncthreads();
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(DecodeCfg<T, D, BS, true, 8>::kThreads, D <= 128 ? 3 : 2)
    paged_decode_rs_lean_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                                const DecodeArgs a) {
    using R = RsLeanCfg<T, D, BS>;
    using C = typename R::C;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
    uint64_t* empty = full + C::kNSlot;
    int* issued = reinterpret_cast<int*>(smem + C::kIssuedOffset);
    int* warp_sums = reinterpret_cast<int*>(smem + C::kStatOffset);
    volatile int* flags = reinterpret_cast<volatile int*>(smem + C::kFlagOffset);  // [0]: abort
    int* pre = reinterpret_cast<int*>(smem + R::kPrefixOffset);
    int* lens_s = pre + (a.num_seqs + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int B = a.num_seqs;
    const int nchunks = (a.rows + C::kHeads - 1) / C::kHeads;  // 2..4 (the plan takes this schedule only then)

    if (tid == 0) {
        for (int s = 0; s < C::kNSlot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nchunks);  // every chunk's warp releases the slot
            issued[s] = 0;
        }
        flags[0] = 0;
        fence_barrier_init();
    }
    // Wait for the previous grid in the stream (it may write the lengths, the tables or the
    // queries); the merge grid may launch at once, it waits for this grid's completion itself.
    griddep_wait();
    griddep_launch_dependents();

    rs_page_prefix<BS>(a.context_lens, B, a.max_blocks, pre, lens_s, warp_sums, C::kNW + 1, blockIdx.x == 0, a.err);
    const int upb = a.num_kv_heads;  // units per sequence
    const int total = pre[B] * upb;
    const int share = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int g0 = min(total, (int)blockIdx.x * share);
    const int g1 = min(total, g0 + share);
    if (g0 >= g1) return;  // no pages for this CTA (fewer pages than CTAs)

    if (warp == C::kNW) {
        // ================= producer warp =================
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_v);
        }
        // Pages are read once per call: let them leave L2 first.
        const uint64_t stream_policy = l2_policy_evict_first();
        int i = 0;  // the page's index in the share; its ring slot is i % kNSlot
        bool ok = true;
        for (int g = g0; g < g1 && ok;) {
            int b, kvh, j, nb;
            lean_locate(pre, B, upb, g, b, kvh, j, nb);
            const int cnt = min(g1 - g, nb - j);  // this unit's pages in the share
            const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks + j;
            for (int c = 0; c < cnt && ok; c += 32) {
                const int pbl = c + lane < cnt ? __ldcg(bt + c + lane) : 0;
                const int m = min(32, cnt - c);
                for (int jj = 0; jj < m; ++jj) {
                    const int pb = __shfl_sync(0xffffffffu, pbl, jj);
                    int good = 1;
                    if (lane == 0) {
                        const int s = i % C::kNSlot;
                        if (i >= C::kNSlot)
                            good = mbar_wait_bounded(&empty[s], ((i / C::kNSlot) - 1) & 1, a.err, flags) ? 1 : 0;
                        if (good) {
                            issued[s] += 1;
                            if ((unsigned)pb < (unsigned)a.num_blocks) {
                                mbar_arrive_expect_tx(&full[s], C::kSlotBytes);
                                const int row = (pb * a.num_kv_heads + kvh) * BS;
                                uint8_t* kdst = ring + s * C::kSlotBytes;
                                uint8_t* vdst = kdst + C::kPageBytes;
#pragma unroll
                                for (int bx = 0; bx < C::kNBox; ++bx)
                                    tma_load_2d_hint(kdst + bx * C::kBoxBytes, &tmap_k, bx * C::kBoxElems, row,
                                                     &full[s], stream_policy);
#pragma unroll
                                for (int bx = 0; bx < C::kNBox; ++bx)
                                    tma_load_2d_hint(vdst + bx * C::kBoxBytes, &tmap_v, bx * C::kBoxElems, row,
                                                     &full[s], stream_policy);
                            } else {
                                atomicOr(a.err, kErrBadTable);  // skip the load; the slot keeps stale data
                                mbar_arrive(&full[s]);
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                    if (!ok) break;
                    ++i;
                }
            }
            g += cnt;
        }
    } else if (warp < nchunks) {
        // ================= consumer warps: warp w takes row chunk w =================
        const T* q = static_cast<const T*>(a.q);
        T* out = static_cast<T*>(a.out);
        MmaConsumer<T, D, BS, true> cons;
        const int cgc = min(C::kHeads, a.rows - warp * C::kHeads);  // this chunk's rows
        int i = 0;
        bool alive = true;
        for (int g = g0; g < g1 && alive;) {
            int j, nb, cnt, L;
            {
                int b, kvh;
                lean_locate(pre, B, upb, g, b, kvh, j, nb);
                cnt = min(g1 - g, nb - j);
                L = lens_s[b];
                const UnitRows rows{b, kvh, warp * C::kHeads, a.q_len, a.group, a.num_heads};
                const int r = min(lane >> 2, cgc - 1);
                cons.init(q + rows.row(r) * D, (lane >> 2) < cgc, rows.last_pos(2 * (lane & 3), L),
                          rows.last_pos(2 * (lane & 3) + 1, L), lane);
            }
            int k = 0;
            if constexpr (BS == 16) {
                // two pages at a time (one softmax step per 32 tokens); an odd last page below
                for (; k + 1 < cnt; k += 2) {
                    const int i0 = i + k;
                    const int s0 = i0 % C::kNSlot, s1 = (i0 + 1) % C::kNSlot;
                    const bool got = mbar_wait_bounded(&full[s0], (i0 / C::kNSlot) & 1, a.err, flags) &&
                                     mbar_wait_bounded(&full[s1], ((i0 + 1) / C::kNSlot) & 1, a.err, flags);
                    if (!__all_sync(0xffffffffu, got)) {
                        alive = false;
                        break;
                    }
                    const int p0 = j + k;  // the pair's first page in the unit
                    uint8_t* kp0 = ring + s0 * C::kSlotBytes;
                    uint8_t* kp1 = ring + s1 * C::kSlotBytes;
                    cons.page_pair(kp0, kp0 + C::kPageBytes, min(BS, L - p0 * BS), p0 * BS, kp1, kp1 + C::kPageBytes,
                                   min(BS, L - (p0 + 1) * BS), (p0 + 1) * BS, a.scale_log2, lane);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[s0]);
                        mbar_arrive(&empty[s1]);
                    }
                }
            }
            for (; alive && k < cnt; ++k) {
                const int i0 = i + k;
                const int s = i0 % C::kNSlot;
                const bool got = mbar_wait_bounded(&full[s], (i0 / C::kNSlot) & 1, a.err, flags);
                if (!__all_sync(0xffffffffu, got)) {
                    alive = false;
                    break;
                }
                const int p = j + k;
                uint8_t* kp = ring + s * C::kSlotBytes;
                cons.page(kp, kp + C::kPageBytes, min(BS, L - p * BS), p * BS, a.scale_log2, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if (!alive) break;
            i += cnt;
            cons.finish();
            if (cnt == nb) {
                // the whole unit lies in this share (its sequence and kv head found again: fewer
                // registers live across the page loop)
                int b, kvh, jj, nn;
                lean_locate(pre, B, upb, g, b, kvh, jj, nn);
                cons.write_out(out, UnitRows{b, kvh, warp * C::kHeads, a.q_len, a.group, a.num_heads}, cgc, lane);
            } else {
                const int slot = g == g0 ? 0 : 1;
                float* rec = a.ws_part + (((size_t)blockIdx.x * 2 + slot) * R::kMaxChunks + warp) * R::kRecFloats;
                cons.write_partial(rec, cgc, lane);
            }
            g += cnt;
        }
    }
    __syncthreads();  // pipeline finished (or abandoned)
    if (flags[0] && tid == 0) {
        // A wait gave up: let every issued copy land before the CTA's shared memory goes away.
        for (int s = 0; s < C::kNSlot; ++s)
            if (issued[s] > 0) {
                const unsigned long long start = global_timer_ns();
                while (!mbar_try_wait(&full[s], (issued[s] - 1) & 1) && global_timer_ns() - start < kWaitLimitNs) {
                }
            }
    }
}

// Combines the partial records of the units that the row-split schedule's shares cut: one warp
// per output row (b, kv head, row v of the kv head), with the page layout and share size
// recomputed from the lengths exactly as the decode grid computed them (a.lean_grid CTAs).  A
// sequence with an empty context gets zero rows here.
template <typename T, int D, int BS>
__global__ void __launch_bounds__(kMergeThreads) rs_lean_merge_kernel(const DecodeArgs a) {
    using R = RsLeanCfg<T, D, BS>;
    static_assert(D % 32 == 0, "whole dims per lane");
    constexpr int DPL = D / 32;
    constexpr int kWarps = kMergeThreads / 32;
    extern __shared__ int mpre[];  // [num_seqs + 1] page prefix sums
    __shared__ int msums[kWarps];
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);  // (b * H_kv + kvh) * rows + v

    griddep_wait();  // the decode grid's records and rows are complete
    griddep_launch_dependents();
    const int B = a.num_seqs;
    rs_page_prefix<BS>(a.context_lens, B, a.max_blocks, mpre, nullptr, msums, kWarps, false, a.err);
    if (row >= B * a.num_kv_heads * a.rows) return;
    const int b = row / (a.num_kv_heads * a.rows);
    const int rest = row - b * a.num_kv_heads * a.rows;
    const int kvh = rest / a.rows;
    const int v = rest - kvh * a.rows;
    const UnitRows rows{b, kvh, v, a.q_len, a.group, a.num_heads};
    T* out = static_cast<T*>(a.out) + rows.row(0) * D + lane * DPL;
    const int nb = mpre[b + 1] - mpre[b];
    if (nb == 0) {
#pragma unroll
        for (int e = 0; e < DPL; ++e) out[e] = from_float<T>(0.f);
        return;
    }
    const int total = mpre[B] * a.num_kv_heads;
    const int share = (total + a.lean_grid - 1) / a.lean_grid;
    const int start = mpre[b] * a.num_kv_heads + kvh * nb;
    const int c0 = start / share;
    const int n = (start + nb - 1) / share - c0 + 1;  // CTAs whose shares hold pages of the unit
    if (n <= 1) return;                               // the decode grid wrote the row itself
    const int chunk = v >> 3, r = v & 7;
    // CTA c0 holds the unit as its last unit unless the unit starts its share; later CTAs as their first
    const int slot0 = start == c0 * share ? 0 : 1;
    auto rec = [&](int p) {
        return a.ws_part + (((size_t)(c0 + p) * 2 + (p == 0 ? slot0 : 0)) * R::kMaxChunks + chunk) * R::kRecFloats;
    };
    const float m0 = lane < n ? __ldcg(rec(lane) + r) : -INFINITY;
    const float l0 = lane < n ? __ldcg(rec(lane) + 8 + r) : 0.f;
    float vals[kMergePre][DPL];
#pragma unroll
    for (int i = 0; i < kMergePre; ++i) {
        if (i < n) {
            load_dims<DPL>(vals[i], rec(i) + 16 + r * D + lane * DPL);
        } else {
#pragma unroll
            for (int e = 0; e < DPL; ++e) vals[i][e] = 0.f;
        }
    }
    float mm = m0;
    for (int c = 32; c < n; c += 32)
        if (c + lane < n) mm = fmaxf(mm, __ldcg(rec(c + lane) + r));
    mm = warp_max(mm);
    float f = rescale(m0, mm);
    float ws = f * l0;
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < kMergePre; ++i) {
        const float fi = __shfl_sync(0xffffffffu, f, i);
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] += fi * vals[i][e];
    }
    for (int q0 = kMergePre; q0 < n; q0 += kMergePre) {
        if (q0 % 32 == 0) {
            const int qq = q0 + lane;
            f = qq < n ? rescale(__ldcg(rec(qq) + r), mm) : 0.f;
            ws += qq < n ? f * __ldcg(rec(qq) + 8 + r) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kMergePre; ++i) {
            if (q0 + i < n) {
                load_dims<DPL>(vals[i], rec(q0 + i) + 16 + r * D + lane * DPL);
            } else {
#pragma unroll
                for (int e = 0; e < DPL; ++e) vals[i][e] = 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kMergePre; ++i) {
            const float fi = __shfl_sync(0xffffffffu, f, (q0 + i) % 32);
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[e] += fi * vals[i][e];
        }
    }
    ws = warp_sum(ws);
    const float inv = ws > 0.f ? 1.f / ws : 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) out[e] = from_float<T>(acc[e] * inv);
}

// Host-side helpers for the per-dtype translation units.
template <typename T, int D, int BS, bool MMA, int GMAX, bool CAUSAL>
struct DecodeKernel {
    using C = DecodeCfg<T, D, BS, MMA, GMAX>;
    using LC = LeanCfg<T, D, BS, MMA, GMAX>;
    // the persistent row-split schedule: tensor-core kernel with causal bounds, 16-bit types
    static constexpr bool kRowSplit = MMA && CAUSAL && sizeof(T) == 2;

    static bool configure(int device) {
        static unsigned long long done_mask = 0;  // one bit per device (< 64)
        const unsigned long long bit = 1ull << (device & 63);
        if (done_mask & bit) return true;
        if (cudaFuncSetAttribute(paged_decode_kernel<T, D, BS, MMA, GMAX, CAUSAL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
            return false;
        if (cudaFuncSetAttribute(paged_decode_lean_kernel<T, D, BS, MMA, GMAX, CAUSAL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, LC::kMaxSmemBytes) != cudaSuccess)
            return false;
        if constexpr (kRowSplit) {
            if (cudaFuncSetAttribute(paged_decode_rs_lean_kernel<T, D, BS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     RsLeanCfg<T, D, BS>::kMaxSmemBytes) != cudaSuccess)
                return false;
        }
        done_mask |= bit;
        return true;
    }

    // Resident lean CTAs per SM for a given dynamic shared-memory size (memoised per device and KB).
    static int lean_occupancy(int device, int smem) {
        static std::atomic<int> cache[64][232];
        const int kb = (smem + 1023) / 1024;
        std::atomic<int>& slot = cache[device & 63][kb < 232 ? kb : 231];
        int n = slot.load(std::memory_order_relaxed);
        if (n > 0) return n;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_lean_kernel<T, D, BS, MMA, GMAX, CAUSAL>,
                                                          LC::kThreads, kb * 1024) != cudaSuccess ||
            n <= 0)
            n = 1;
        slot.store(n, std::memory_order_relaxed);
        return n;
    }

    static bool info(int num_seqs, KernelInfo* info) {
        int device = 0;
        if (cudaGetDevice(&device) != cudaSuccess) return false;
        if (!configure(device)) return false;
        info->threads = C::kThreads;
        info->smem_bytes = C::kSmemBytes;
        info->heads_per_cta = C::kHeads;
        info->merge_parts_cap = kMergeMaxParts;
        // resident CTAs per SM of the partitioned-grid kernel, memoised per device (an occupancy
        // query per call would cost the host several microseconds)
        static std::atomic<int> grid_occ[64];
        int n = grid_occ[device & 63].load(std::memory_order_relaxed);
        if (n <= 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_decode_kernel<T, D, BS, MMA, GMAX, CAUSAL>,
                                                              C::kThreads, C::kSmemBytes) != cudaSuccess ||
                n <= 0)
                n = 1;
            grid_occ[device & 63].store(n, std::memory_order_relaxed);
        }
        info->ctas_per_sm = n;
        const int seqs = num_seqs < 1 ? 1 : (num_seqs > kLeanMaxSeqs ? kLeanMaxSeqs : num_seqs);
        info->lean_smem_bytes = LC::smem_bytes(seqs);
        info->lean_ctas_per_sm = lean_occupancy(device, info->lean_smem_bytes);
        info->lean_warps_per_cta = LC::kNW;
        info->lean_record_floats = LC::kRecFloats;
        info->lean_max_seqs = kLeanMaxSeqs;
        info->rs_ctas_per_sm = 0;
        info->rs_smem_bytes = 0;
        info->rs_record_floats = 0;
        if constexpr (kRowSplit) {
            using R = RsLeanCfg<T, D, BS>;
            info->rs_smem_bytes = R::smem_bytes(seqs);
            info->rs_record_floats = R::kRecFloats;
            static std::atomic<int> rs_occ[64][232];
            const int kb = (info->rs_smem_bytes + 1023) / 1024;
            std::atomic<int>& slot = rs_occ[device & 63][kb < 232 ? kb : 231];
            int r = slot.load(std::memory_order_relaxed);
            if (r <= 0) {
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, paged_decode_rs_lean_kernel<T, D, BS>,
                                                                  C::kThreads, kb * 1024) != cudaSuccess)
                    r = 0;
                slot.store(r > 0 ? r : -1, std::memory_order_relaxed);
            }
            info->rs_ctas_per_sm = r > 0 ? r : 0;
        }
        return true;
    }

    static cudaError_t launch(int schedule, const CUtensorMap& k, const CUtensorMap& v, const DecodeArgs& a, int grid,
                              int num_seqs, cudaStream_t stream) {
        int device = 0;
        cudaError_t e = cudaGetDevice(&device);
        if (e != cudaSuccess) return e;
        if (!configure(device)) return cudaGetLastError();
        if (schedule == kScheduleLean || schedule == kScheduleLeanMergeOnly) {
            DecodeArgs d = a;
            // 16-bit pages: cut the pages for 95 % of the consumer warps.  With every warp
            // streaming, the Qwen-shaped step took 53.3 us and the long-context one 324 us; with
            // 95 % (the last CTAs idle) 52.5 and 314 us; 90 %: 53.0 and 312 us, 85 %: 55.9 and 325 us.
            d.lean_share_warps = grid * LC::kNW * 95 / 100;
            if (schedule == kScheduleLean) {
                e = launch_pdl(paged_decode_lean_kernel<T, D, BS, MMA, GMAX, CAUSAL>, dim3(grid), dim3(LC::kThreads),
                               LC::smem_bytes(num_seqs), stream, k, v, d);
                if (e != cudaSuccess) return e;
            }
            DecodeArgs m = d;
            const int mgrid = lean_merge_setup(m, grid);
            return launch_pdl(lean_merge_kernel<T, D, LC::kHeads, BS>, dim3(mgrid), dim3(kLeanMergeThreads), 0,
                              stream, m);
        } else if (schedule == kScheduleRowSplit) {
            if constexpr (kRowSplit) {
                using R = RsLeanCfg<T, D, BS>;
                DecodeArgs d = a;
                d.lean_grid = grid;
                e = launch_pdl(paged_decode_rs_lean_kernel<T, D, BS>, dim3(grid), dim3(C::kThreads),
                               R::smem_bytes(num_seqs), stream, k, v, d);
                if (e != cudaSuccess) return e;
                const int rows = a.num_seqs * a.num_kv_heads * a.rows;
                constexpr int kRowsPerCta = kMergeThreads / 32;
                return launch_pdl(rs_lean_merge_kernel<T, D, BS>, dim3((rows + kRowsPerCta - 1) / kRowsPerCta),
                                  dim3(kMergeThreads), (num_seqs + 1) * (int)sizeof(int), stream, d);
            } else {
                return cudaErrorInvalidValue;
            }
        } else {
            return launch_pdl(paged_decode_kernel<T, D, BS, MMA, GMAX, CAUSAL>, dim3(grid), dim3(C::kThreads), C::kSmemBytes,
                              stream, k, v, a);
        }
    }
};

// FP8 caches: the lean decode with the FP8 consumer and the lean merge (no partitioned grid).
template <typename T, int D, int BS>
struct DecodeKernelF8 {
    using LC = LeanCfg<uint8_t, D, BS, true, 8>;
    using Fn = void (*)(const CUtensorMap, const CUtensorMap, const DecodeArgs);
    static Fn kernel(bool append) {
        return append ? paged_decode_lean_kernel<T, D, BS, true, 8, false, true, true>
                      : paged_decode_lean_kernel<T, D, BS, true, 8, false, true, false>;
    }

    static bool configure(int device) {
        static unsigned long long done_mask = 0;
        const unsigned long long bit = 1ull << (device & 63);
        if (done_mask & bit) return true;
        for (const bool append : {false, true})
            if (cudaFuncSetAttribute(kernel(append), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     LC::kMaxSmemBytes) != cudaSuccess)
                return false;
        done_mask |= bit;
        return true;
    }

    static bool info(int num_seqs, KernelInfo* info) {
        int device = 0;
        if (cudaGetDevice(&device) != cudaSuccess) return false;
        if (!configure(device)) return false;
        const int seqs = num_seqs < 1 ? 1 : (num_seqs > kLeanMaxSeqs ? kLeanMaxSeqs : num_seqs);
        const int smem = LC::smem_bytes(seqs);
        static std::atomic<int> cache[64][232];
        const int kb = (smem + 1023) / 1024;
        std::atomic<int>& slot = cache[device & 63][kb < 232 ? kb : 231];
        int n = slot.load(std::memory_order_relaxed);
        if (n <= 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel(false), LC::kThreads, kb * 1024) !=
                    cudaSuccess ||
                n <= 0)
                n = 1;
            slot.store(n, std::memory_order_relaxed);
        }
        info->threads = LC::kThreads;
        info->smem_bytes = 0;
        info->heads_per_cta = LC::kHeads;
        info->ctas_per_sm = 0;
        info->merge_parts_cap = 0;
        info->lean_smem_bytes = smem;
        info->lean_ctas_per_sm = n;
        info->lean_warps_per_cta = LC::kNW;
        info->lean_record_floats = LC::kRecFloats;
        info->lean_max_seqs = kLeanMaxSeqs;
        info->rs_ctas_per_sm = 0;
        info->rs_smem_bytes = 0;
        info->rs_record_floats = 0;
        return true;
    }

    static cudaError_t launch(const CUtensorMap& k, const CUtensorMap& v, const DecodeArgs& a, int grid, int num_seqs,
                              cudaStream_t stream) {
        int device = 0;
        cudaError_t e = cudaGetDevice(&device);
        if (e != cudaSuccess) return e;
        if (!configure(device)) return cudaGetLastError();
        DecodeArgs d = a;
        // FP8 pages: every consumer warp streams (fewer took longer: 43.9 us on the Qwen-shaped
        // step with all warps, 45.1 with 95 %, 46.3 with 90 %).
        d.lean_share_warps = grid * LC::kNW;
        e = launch_pdl(kernel(a.new_key != nullptr), dim3(grid), dim3(LC::kThreads), LC::smem_bytes(num_seqs), stream,
                       k, v, d);
        if (e != cudaSuccess) return e;
        DecodeArgs m = d;
        const int mgrid = lean_merge_setup(m, grid);
        return launch_pdl(lean_merge_kernel<T, D, LC::kHeads, BS>, dim3(mgrid), dim3(kLeanMergeThreads), 0, stream,
                          m);
    }
};

template <typename T, int D>
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
    constexpr int kRowsPerCta = kMergeThreads / 32;
    const int merge_rows = a.num_seqs * a.num_heads * a.q_len;
    return launch_pdl(splitkv_merge_kernel<T, D>, dim3((merge_rows + kRowsPerCta - 1) / kRowsPerCta), dim3(kMergeThreads), 0,
                      stream, a);
}

}  // namespace pa
