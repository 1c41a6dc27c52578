// Block-sparse attention backward for sm_103a (tcgen05 + TMA).
//
// The gradients of the forward in vsa_attn.cu (FastVideo kernel page,
// hao-ai-lab/FastVideo commit 8503617; the Attn-QAT SM100 commit names the
// backward pass and its dQ / dK-dV tiles): for a valid query row i with key
// list L and the forward's natural-log LSE,
//   p_ie = exp(scale * q_i.k_e - lse_i),  delta_i = sum_d dout_id * out_id,
//   ds_ie = p_ie * (dout_i.v_e - delta_i),
//   dq_i = scale * sum_e ds_ie k_e,  dk_e = scale * sum_i ds_ie q_i,
//   dv_e = sum_i p_ie dout_i.
//
// The kernels work on 128-row "kernel tiles" whatever the caller's tile T:
// with T = 128 a kernel tile is a caller tile; with T = 256 it is one half of
// one (tile_size clamps the valid count); with T = 64 it holds two caller
// tiles, rows 0-63 and 64-127.  A pair of kernel tiles carries a 4-bit mask of
// which (64-row sub-tile, 64-row sub-tile) blocks are selected, so 64-token
// selections need no other change; with T >= 128 every mask is full.
//
// Kernels:
//   delta_kernel   per row -delta = -rowsum(dout * out) in fp32 (one pass over
//                  both) and -lse in log2 units, the two per-row terms the
//                  elementwise step adds, stored with a row stride of whole
//                  kernel tiles.
//   pairs_kernel   per (batch, head, query kernel tile) the selected key kernel
//                  tiles, ascending, each with its block mask (one warp each).
//   k2q_kernel     per (batch, head) the transposed lists: for every key
//                  kernel tile, the query kernel tiles that select it, in
//                  ascending order (one CTA per (batch, head), deterministic).
//   bwd_kernel<D, true>   one CTA per (batch, head, key tile j): K_j and V_j
//                  stay in shared memory; the query tiles t that select j
//                  stream through two buffers (the next pair's copies overlap
//                  this pair's work).  A pair is done in two 64-column halves
//                  (64 of the query tile's rows), each in its own TMEM slot:
//                  S^T = K_j Q_t^T and dP^T = V_j dO_t^T of the half go to the
//                  slot; eight elementwise warps (two threads per key row)
//                  write P^T and dS^T as bf16 back over the columns they read;
//                  dV += P^T dO_t and dK += dS^T Q_t accumulate in TMEM with
//                  the A operand taken from the slot.  One thread issues the
//                  accumulations, a second the copies and S, a third dP (the
//                  N = 64 products each read 6 KB of shared-memory operands,
//                  48 cycles at 128 bytes a clock, and a thread issuing them
//                  also waits on its barriers; two issuers overlap that); S
//                  and dP go into a slot as soon as the previous pair's
//                  accumulations have read it: the next pair's products
//                  overlap this pair's elementwise step.
//   bwd_kernel<D, false>  one CTA per (batch, head, query tile t): Q_t and dO_t
//                  stay; for every selected key tile, S and dP again, dS back
//                  into TMEM, dQ += dS K_j.  Recomputing S and dP keeps dQ
//                  free of atomics and the result deterministic.
// Padding rows are kept out of every product: P and dS are set (not
// multiplied) to 0 in the partner's padding columns and in unselected blocks,
// and padding rows of an operand that is summed over (Q and dO in dk/dv, K in
// dq) are zeroed in shared memory first, so NaN/Inf padding never meets a zero
// weight.  Padding rows of the resident tile reach only their own rows of the
// accumulators, which the epilogue writes as 0.  Every wait is bounded; on
// expiry the CTA flags VSA_ERR_TIMEOUT and returns.
#include <cuda_bf16.h>

#include "vsa_internal.h"
#include "vsa_ptx.cuh"
#include "vsa_wait.cuh"

namespace vsa {
namespace {

using namespace ptx;

constexpr int kBT = 128;            // tile rows (queries or keys)
constexpr int kEwSplit = 2;                 // elementwise threads per row
constexpr int kEwThreads = kEwSplit * kBT;  // elementwise warps first
constexpr int kEwCols = 64 / kEwSplit;      // columns per thread in each 64-column half
constexpr int kCtlWarp = kEwThreads / 32;   // lane 0 issues the accumulation MMAs
constexpr int kSdpWarp = kCtlWarp + 1;      // lane 0 issues the TMA copies and the S MMAs
constexpr int kDpWarp = kCtlWarp + 2;       // lane 0 issues the dP MMAs
constexpr int kThreads = kEwThreads + 96;
constexpr uint32_t kChunkBytes = kBT * 128;  // one 64-column (128-byte) chunk of a 128-row tile

template <int D>
struct BwdCfg {
    static constexpr uint32_t kTile = kBT * D * 2;   // one Q/K/V/dO tile in shared memory
    static constexpr uint32_t kIdescHalf = idesc_bf16(128, 64, false);  // S-like products, N = 64
    static constexpr uint32_t kIdescAcc = idesc_bf16(128, D, true);    // accumulations, B MN-major
};

// Zeroes row `row` of a 128-row tile of D columns (a whole row, so the
// swizzle does not matter).
template <int D>
__device__ __forceinline__ void zero_row(uint8_t *tile, int row) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        uint4 *p = reinterpret_cast<uint4 *>(tile + c * kChunkBytes + row * 128);
#pragma unroll
        for (int g = 0; g < 8; ++g) p[g] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Issues the D/16 MMAs of a 128 x 64 product over D: the 128 resident rows
// times 64 rows of a partner tile (both operands K-major; b_saddr points at
// the first of the 64 rows inside the tile's first column chunk).
template <int D>
__device__ __forceinline__ void mma_half(uint32_t tdst, uint32_t a_saddr, uint32_t b_saddr) {
    const uint64_t a = sdesc_sw128(a_saddr, 16, 1024), b = sdesc_sw128(b_saddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tdst, a + (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2, b + (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2,
               BwdCfg<D>::kIdescHalf, kk > 0 ? 1u : 0u);
}

// ---------------------------------------------------------------- delta
// Caller row (bh, s), s < Sp, goes to vector entry bh * Spk + s.
__global__ void __launch_bounds__(256) delta_kernel(const uint4 *__restrict__ out, const uint4 *__restrict__ dout,
                                                   const float *__restrict__ lse, float *__restrict__ ndelta,
                                                   float *__restrict__ nlse2, int64_t rows, int Dv, int64_t Sp,
                                                   int64_t Spk) {
    // one 8-lane group per row (Dv <= 16 vectors of 8 bf16)
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t row = gid >> 3;
    const int sub = (int)(gid & 7);
    float acc = 0.f;
    if (row < rows) {
        for (int v = sub; v < Dv; v += 8) {
            const uint4 a = __ldg(out + row * Dv + v), b = __ldg(dout + row * Dv + v);
            const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(__uint_as_float(x[i] << 16), __uint_as_float(y[i] << 16), acc);
                acc = fmaf(__uint_as_float(x[i] & 0xffff0000u), __uint_as_float(y[i] & 0xffff0000u), acc);
            }
        }
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (row < rows && sub == 0) {
        const int64_t o = (row / Sp) * Spk + row % Sp;
        ndelta[o] = -acc;
        nlse2[o] = -__ldg(lse + row) * 1.4426950408889634f;
    }
}

// Kernel-tile geometry of a caller tiling: T caller tile rows, NTc caller tiles.
struct Geo {
    int32_t T, NTc, NTk;
};

// Valid rows of kernel tile z in its two 64-row halves: row r is valid iff
// r < 64 ? r < lo : r - 64 < hi.
struct Rows {
    int lo, hi;
    __device__ __forceinline__ bool valid(int r) const { return r < 64 ? r < lo : r - 64 < hi; }
};

__device__ __forceinline__ Rows ktile_rows(const int32_t *bs, const Geo &G, int z) {
    int n;
    if (G.T == 64) {
        const int a = 2 * z < G.NTc ? __ldg(bs + 2 * z) : 0, b = 2 * z + 1 < G.NTc ? __ldg(bs + 2 * z + 1) : 0;
        return Rows{a < 0 ? 0 : (a > 64 ? 64 : a), b < 0 ? 0 : (b > 64 ? 64 : b)};
    }
    if (G.T == 128) {
        n = __ldg(bs + z);
    } else {
        n = __ldg(bs + (z >> 1)) - 128 * (z & 1);
    }
    n = n < 0 ? 0 : (n > 128 ? 128 : n);
    return Rows{n < 64 ? n : 64, n > 64 ? n - 64 : 0};
}

// A partner list entry: partner kernel tile y (13 bits), its valid rows per
// half (7 bits each) and the block mask (4 bits).
__device__ __forceinline__ int32_t pack_entry(int y, Rows rw, int mask) {
    return (int32_t)(((uint32_t)y << 18) | ((uint32_t)rw.lo << 11) | ((uint32_t)rw.hi << 4) | (uint32_t)mask);
}
__device__ __forceinline__ int entry_y(int32_t e) { return (int)((uint32_t)e >> 18); }
__device__ __forceinline__ Rows entry_rows(int32_t e) { return Rows{(e >> 11) & 127, (e >> 4) & 127}; }

// One warp per (bh, query kernel tile X): the key kernel tiles Y its caller
// tiles select, ascending, as pack_entry(Y, rows of Y, mask) with mask bit
// 2a + b set when query half a selects key half b.  Key tiles without valid
// rows are left out.
// list [BH*NTk, maxlen], cnt [BH*NTk].  Entries out of range are skipped and
// flagged.
__global__ void __launch_bounds__(128)
    pairs_kernel(const int32_t *__restrict__ q2k_idx, const int32_t *__restrict__ q2k_num,
                 const int32_t *__restrict__ bs, Geo G, int max_kv, int maxlen, int64_t BH,
                 int32_t *__restrict__ list, int32_t *__restrict__ cnt, int32_t *status) {
    extern __shared__ uint32_t mw[];  // [4 warps][NTk / 4 + 1] words of 4 mask bytes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int words = G.NTk / 4 + 1;
    uint32_t *m = mw + warp * words;
    const int64_t gx = (int64_t)blockIdx.x * 4 + warp;  // bh * NTk + X
    if (gx >= BH * G.NTk) return;
    const int64_t bh = gx / G.NTk;
    const int X = (int)(gx - bh * G.NTk);
    for (int w = lane; w < words; w += 32) m[w] = 0u;
    __syncwarp();
    bool bad = false;
    // caller query tiles of X: (t, the mask bits of its rows' halves)
    const int nsrc = G.T == 64 ? 2 : 1;
    for (int a = 0; a < nsrc; ++a) {
        const int t = G.T == 64 ? 2 * X + a : (G.T == 128 ? X : X >> 1);
        if (t >= G.NTc) continue;
        int K = __ldg(q2k_num + bh * G.NTc + t);
        if (K < 0 || K > max_kv) {
            bad = true;
            K = K < 0 ? 0 : max_kv;
        }
        const int32_t *sel = q2k_idx + (bh * G.NTc + t) * (int64_t)max_kv;
        for (int i = lane; i < K; i += 32) {
            const int jc = __ldg(sel + i);
            if (jc < 0 || jc >= G.NTc) {
                bad = true;
                continue;
            }
            const int n = __ldg(bs + jc);
            if (G.T == 64) {
                if (n <= 0) continue;
                const int Y = jc >> 1;
                atomicOr(&m[Y >> 2], (1u << (2 * a + (jc & 1))) << ((Y & 3) * 8));
            } else if (G.T == 128) {
                if (n <= 0) continue;
                atomicOr(&m[jc >> 2], 0xFu << ((jc & 3) * 8));
            } else {
                for (int hb = 0; hb < 2; ++hb) {
                    if (n - 128 * hb <= 0) continue;
                    const int Y = 2 * jc + hb;
                    atomicOr(&m[Y >> 2], 0xFu << ((Y & 3) * 8));
                }
            }
        }
    }
    __syncwarp();
    int32_t *out = list + gx * maxlen;
    int c = 0;
    for (int base = 0; base < G.NTk; base += 32) {
        const int Y = base + lane;
        const uint32_t mk = Y < G.NTk ? (m[Y >> 2] >> ((Y & 3) * 8)) & 0xFu : 0u;
        const uint32_t bal = __ballot_sync(0xffffffffu, mk != 0u);
        const int pos = c + __popc(bal & ((1u << lane) - 1u));
        if (mk != 0u && pos < maxlen) out[pos] = pack_entry(Y, ktile_rows(bs, G, Y), (int)mk);
        c += __popc(bal);
    }
    if (lane == 0) cnt[gx] = c < maxlen ? c : maxlen;
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(status, kFlagIndex);
}

// Mask with the roles of the two sides swapped: bit 2a + b -> bit 2b + a.
__device__ __forceinline__ int swap_mask(int m) { return (m & 9) | ((m & 2) << 1) | ((m & 4) >> 1); }

// offs [B*H, NTk+1] and list [B*H, NTk*maxlen]: list[bh][offs[bh][Y] ...] are
// pack_entry(X, rows of X, mask) for the query kernel tiles X selecting key
// kernel tile Y, ascending in X, with mask bit 2a + b set when key half a
// meets query half b.
__global__ void __launch_bounds__(1024)
    k2q_kernel(const int32_t *__restrict__ pl, const int32_t *__restrict__ pc, const int32_t *__restrict__ bs,
               Geo G, int maxlen, int32_t *__restrict__ offs, int32_t *__restrict__ list) {
    const int NTk = G.NTk;
    extern __shared__ int32_t cur[];  // [NTk + 1]
    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    for (int j = tid; j <= NTk; j += blockDim.x) cur[j] = 0;
    __syncthreads();
    const int32_t *plb = pl + bh * (int64_t)NTk * maxlen;
    const int32_t *pcb = pc + bh * (int64_t)NTk;
    for (int64_t e = tid; e < (int64_t)NTk * maxlen; e += blockDim.x) {
        const int X = (int)(e / maxlen), i = (int)(e - (int64_t)X * maxlen);
        if (i < __ldg(pcb + X)) atomicAdd(&cur[entry_y(__ldg(plb + e)) + 1], 1);
    }
    __syncthreads();
    if (tid == 0) {  // exclusive scan (NTk <= 8192: a short serial pass)
        for (int j = 1; j <= NTk; ++j) cur[j] += cur[j - 1];
    }
    __syncthreads();
    for (int j = tid; j <= NTk; j += blockDim.x) offs[bh * (NTk + 1) + j] = cur[j];
    __syncthreads();
    // fill in ascending X: one list per round; a key tile appears at most once
    // per list, so its cursor advances in X order
    int32_t *lst = list + bh * (int64_t)NTk * maxlen;
    // the rounds are sequential, so each thread loads its first entry of the
    // next round (and the round's count) while this round runs
    int c = __ldg(pcb);
    int32_t e0 = (tid < c) ? __ldg(plb + tid) : 0;
    for (int X = 0; X < NTk; ++X) {
        const int c_next = (X + 1 < NTk) ? __ldg(pcb + X + 1) : 0;
        const int32_t e0_next = (tid < c_next) ? __ldg(plb + (int64_t)(X + 1) * maxlen + tid) : 0;
        if (c > 0) {
            const Rows rx = ktile_rows(bs, G, X);
            for (int i = tid; i < c; i += blockDim.x) {
                const int32_t e = (i == tid) ? e0 : __ldg(plb + (int64_t)X * maxlen + i);
                lst[atomicAdd(&cur[entry_y(e)], 1)] = pack_entry(X, rx, swap_mask(e & 15));
            }
        }
        c = c_next;
        e0 = e0_next;
        __syncthreads();
    }
}

// ---------------------------------------------------------------- shared memory
// Resident pair of tiles (K_j, V_j for dK/dV; Q_t, dO_t for dQ), two buffers of
// the per-pair tiles (so the next pair's copies overlap this pair's work), and
// per buffer the lse and delta rows of the query tile (dK/dV only).
template <int D>
struct BwdSmem {
    static constexpr uint32_t kRes0 = 0;
    static constexpr uint32_t kRes1 = kRes0 + BwdCfg<D>::kTile;
    static constexpr uint32_t kBuf = kRes1 + BwdCfg<D>::kTile;                  // [2][2 tiles]
    static constexpr uint32_t kVec = kBuf + 4 * BwdCfg<D>::kTile;               // [2][lse 128 | delta 128]
    static constexpr uint32_t kBars = kVec + 2 * 2 * kBT * 4;                   // mbarriers
    static constexpr uint32_t kSlot = kBars + 8 * 8;                            // TMEM address
    static constexpr uint32_t kFlag = kSlot + 4;                                // abort flag
    static constexpr uint32_t kTotal = kFlag + 4 + 1024;                        // + alignment slack
    static __device__ __forceinline__ uint32_t buf(int b, int which) {
        return kBuf + (uint32_t)(2 * b + which) * BwdCfg<D>::kTile;
    }
};

struct BwdArgs {
    const float *nlse2;         // [B*H*Spk] -lse * log2(e)
    const float *ndelta;        // [B*H*Spk] -rowsum(dout * out)
    const int32_t *block_sizes;
    const int32_t *pl, *pc;     // pairs_kernel lists and counts
    const int32_t *k2q_offs, *k2q_list;
    void *dq, *dk, *dv;         // bf16 [B*H*Sp, D]
    int32_t *status;
    Geo G;
    int32_t maxlen;
    int64_t Sp, Spk;            // caller rows per (b, h); NTk * 128
    float scale;
};

// mbarriers: resident tiles loaded, per-buffer tiles loaded (two), and per
// TMEM slot (one 64-column half of a pair): S and dP in the slot, P/dS written
// back to it, its accumulations done (the slot is free); the final drain.
enum { kBarRes = 0, kBarBuf0 = 1, kBarBuf1 = 2, kBarS0 = 3, kBarS1 = 4, kBarEw0 = 5, kBarEw1 = 6, kBarFree0 = 7,
       kBarFree1 = 8, kBarDrain = 9 };
constexpr int kNumBars = 10;
constexpr uint32_t kHalfBytes = 64 * 128;  // 64 rows of one 128-byte column chunk

// Where the bf16 pairs of S/dP columns [16kk, 16kk + 16) sit in TMEM: the
// thread that read the kEwCols columns [c0, c0 + kEwCols) writes their packed
// columns back over the first half of them, so no thread overwrites columns
// another thread may still be reading.
__device__ __forceinline__ uint32_t packed_col(int kk) {
    const int c0 = (16 * kk / kEwCols) * kEwCols;
    return (uint32_t)(c0 + (16 * kk - c0) / 2);
}

// TMEM loads of 32 or 16 columns (waited for) and stores of 16 or 8.
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&r)[N]) {
    static_assert(N == 32 || N == 16, "columns");
    if constexpr (N == 32) tmem_ld32(taddr, r);
    else tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
    static_assert(N == 16 || N == 8, "columns");
    if constexpr (N == 16) tmem_st16(taddr, v);
    else tmem_st8(taddr, v);
}

// P and dS of kEwCols columns [c0, c0 + kEwCols) of one row, as bf16 pairs:
//   p = 2^(scale log2(e) s - lse log2(e)),  ds = p (dp - delta),
// with the per-column terms from shared memory (KV: columns are queries) or
// this row's (dQ).  MASK sets p and ds (not multiplies them) to 0 in columns
// c >= n_y (the partner's padding, whose S and dP may be non-finite).
// Rows are not masked: a padding row's values reach only its own row of the
// accumulators, which the epilogue writes as 0.
template <bool KV, bool MASK>
__device__ __forceinline__ void ew_cols(const float (&sv)[kEwCols], const float (&dp)[kEwCols],
                                        uint32_t (&pw)[kEwCols / 2], uint32_t (&dw)[kEwCols / 2], int c0, int n_y,
                                        float c1, const float2 *s_nl2, const float2 *s_ndl, float nl2_r,
                                        float ndl_r) {
#pragma unroll
    for (int e = 0; e < kEwCols; e += 2) {
        const int c = c0 + e;  // column pair c, c+1: queries (KV) or keys
        float2 nl2, ndl;
        if (KV) {
            nl2 = s_nl2[c >> 1];
            ndl = s_ndl[c >> 1];
        } else {
            nl2 = make_float2(nl2_r, nl2_r);
            ndl = make_float2(ndl_r, ndl_r);
        }
        float x0, x1, t0, t1, d0, d1;
        fma2v(x0, x1, sv[e], sv[e + 1], c1, c1, nl2.x, nl2.y);  // scale*s*log2e - lse*log2e
        float p0 = ex2(x0), p1 = ex2(x1);
        fma2v(t0, t1, dp[e], dp[e + 1], 1.f, 1.f, ndl.x, ndl.y);  // dp - delta
        fma2v(d0, d1, p0, p1, t0, t1, 0.f, 0.f);                   // p * (dp - delta)
        if (MASK) {
            p0 = c < n_y ? p0 : 0.f;
            d0 = c < n_y ? d0 : 0.f;
            p1 = c + 1 < n_y ? p1 : 0.f;
            d1 = c + 1 < n_y ? d1 : 0.f;
        }
        pw[e >> 1] = pack_bf16x2(p0, p1);
        dw[e >> 1] = pack_bf16x2(d0, d1);
    }
}

// Issues the 4 MMAs of one half (64 of the 128 summed rows) of
// acc(128 x D) += A(128 x 128, bf16 pairs in TMEM) x tile(128 x D, MN-major in
// shared memory: the tile's rows are summed).  ta is the half's TMEM slot,
// which holds the bf16 pairs of its 64 columns.
// BM (64-token tiles): the accumulator's two 64-row halves belong to two
// caller tiles, and lanes of a half whose tile does not meet this summed half
// (mask bit 2a + half clear for accumulator half a) are left out of the
// product altogether; the accumulators then start at zero and every MMA
// accumulates.
template <int D, bool BM>
__device__ __forceinline__ void mma_acc_half(uint32_t tacc, uint32_t ta, uint32_t tile_saddr, int half,
                                             bool accumulate, int mk) {
    const uint64_t b = sdesc_sw128(tile_saddr, kChunkBytes, 1024);
    const uint32_t off_lo = ((mk >> half) & 1) ? 0u : ~0u, off_hi = ((mk >> (2 + half)) & 1) ? 0u : ~0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int kk = half * 4 + q;
        if constexpr (BM)
            mma_ts_lanes(tacc, ta + packed_col(q), b + kk * (2048 >> 4), BwdCfg<D>::kIdescAcc, 1u, off_lo, off_hi);
        else
            mma_ts(tacc, ta + packed_col(q), b + kk * (2048 >> 4), BwdCfg<D>::kIdescAcc,
                   (accumulate || kk > 0) ? 1u : 0u);
    }
}

// Common shape of both kernels: one resident tile pair, a list of partner
// tiles streamed through two buffers, per pair and 64-column half two
// 128 x 64 products into a TMEM slot (S-like and dP-like), an elementwise step
// by 256 threads that writes bf16 operands back into the slot, and one or two
// accumulations from it.
// BM: pairs carry block masks (64-token tiles); otherwise every mask is full.
template <int D, bool KV, bool BM>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdArgs A) {
    using C = BwdCfg<D>;
    using L = BwdSmem<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *g = smem_raw + (base - raw);
    const uint32_t bars = base + L::kBars;
    auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
    volatile int *abort_flag = reinterpret_cast<int *>(g + L::kFlag);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // the resident tile x and its list of partners: key tile j and the query
    // tiles selecting it (KV), or query tile t and its selected key tiles
    const int64_t bhx = blockIdx.x;
    const int NTk = A.G.NTk;
    const int x = (int)(bhx % NTk);
    const int64_t bh = bhx / NTk;
    const Rows rx = ktile_rows(A.block_sizes, A.G, x);
    const int32_t *lst;
    int n;
    if (KV) {
        const int32_t off0 = __ldg(A.k2q_offs + bh * (NTk + 1) + x), off1 = __ldg(A.k2q_offs + bh * (NTk + 1) + x + 1);
        lst = A.k2q_list + bh * (int64_t)NTk * A.maxlen + off0;
        n = off1 - off0;
    } else {
        lst = A.pl + bhx * A.maxlen;
        n = __ldg(A.pc + bhx);
    }
    // pair i: partner kernel tile, its valid rows and the block mask
    auto entry = [&](int i) -> int32_t { return __ldg(lst + i); };

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNumBars; ++b)
            // a slot's S and dP are committed by two threads; three issuers drain
            mbar_init(BAR(b), (b == kBarEw0 || b == kBarEw1) ? kEwThreads
                              : (b == kBarDrain ? 3 : ((b == kBarS0 || b == kBarS1) ? 2 : 1)));
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kCtlWarp) {
        tmem_alloc(base + L::kSlot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(g + L::kSlot);
    // TMEM: accumulators first (dV, dK) or (dQ), then two slots of 128
    // columns, one per 64-column half of a pair: S-like in the first 64, dP-like
    // in the other 64; the bf16 P / dS operands are written back over them
    const uint32_t tAcc0 = tmem, tAcc1 = tmem + D;
    const uint32_t tSlot0 = tmem + (KV ? 2 * D : D);
    auto slot = [&](int hv) -> uint32_t { return tSlot0 + 128u * (uint32_t)hv; };

    if (warp == kSdpWarp) {
        // ------------------------------------------------------------ copies, S and dP
        if (lane == 0) {
            bool ok = true;
            int issued[2] = {0, 0}, seen[2] = {0, 0};  // per-buffer loads issued / waited for
            const int32_t xrow = (int32_t)(bh * A.Sp + (int64_t)x * kBT);
            auto load_pair = [&](int i) {
                const int b = i & 1, y = entry_y(entry(i));
                const int64_t yrow = bh * A.Sp + (int64_t)y * kBT;
                const int64_t yvec = bh * A.Spk + (int64_t)y * kBT;
                const uint32_t bar = BAR(kBarBuf0 + b);
                mbar_arrive_expect_tx(bar, 2 * C::kTile + (KV ? 2 * kBT * 4 : 0));
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(base + L::buf(b, 0) + c * kChunkBytes, KV ? (const void *)&tm_q : (const void *)&tm_k,
                                c * 64, (int32_t)yrow, bar, l2_policy_evict_last());
                    tma_load_2d(base + L::buf(b, 1) + c * kChunkBytes, KV ? (const void *)&tm_do : (const void *)&tm_v,
                                c * 64, (int32_t)yrow, bar, l2_policy_evict_last());
                }
                if (KV) {
                    bulk_load(base + L::kVec + b * 2 * kBT * 4, A.nlse2 + yvec, kBT * 4, bar);
                    bulk_load(base + L::kVec + b * 2 * kBT * 4 + kBT * 4, A.ndelta + yvec, kBT * 4, bar);
                }
                ++issued[b];
            };
            // S of the half hv of pair i into slot hv (dP: warp kDpWarp).  S and
            // dP go to different columns of the slot and are issued by two
            // threads, so each thread's barrier waits overlap the other's
            // products.
            auto issue_sdp = [&](int i, int hv) {
                const int b = i & 1;
                // KV: S^T = K_j Q_t^T; else S = Q_t K_j^T
                mma_half<D>(slot(hv), base + L::kRes0, base + L::buf(b, 0) + hv * kHalfBytes);
                mma_commit(BAR(kBarS0 + hv));
            };
            if (n > 0) {
                mbar_arrive_expect_tx(BAR(kBarRes), 2 * C::kTile);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(base + L::kRes0 + c * kChunkBytes, KV ? (const void *)&tm_k : (const void *)&tm_q,
                                c * 64, xrow, BAR(kBarRes), l2_policy_evict_first());
                    tma_load_2d(base + L::kRes1 + c * kChunkBytes, KV ? (const void *)&tm_v : (const void *)&tm_do,
                                c * 64, xrow, BAR(kBarRes), l2_policy_evict_first());
                }
                load_pair(0);
                ok = wait_bar(BAR(kBarRes), 0u, abort_flag, A.status) &&
                     wait_bar(BAR(kBarBuf0), 0u, abort_flag, A.status);
                if (ok) {
                    ++seen[0];
                    tc_fence_after();
                    issue_sdp(0, 0);
                    issue_sdp(0, 1);
                    if (n > 1) load_pair(1);
                }
            }
            // S and dP of half hv of pair i + 1 go into slot hv once the
            // accumulations of half hv of pair i have read it, so the next
            // pair's products run while this pair's other half is in the
            // elementwise step.
            for (int i = 0; i + 1 < n && ok; ++i) {
                for (int hv = 0; hv < 2 && ok; ++hv) {
                    if (!(ok = wait_bar(BAR(kBarFree0 + hv), i & 1u, abort_flag, A.status))) break;
                    if (hv == 0) {
                        const int b1 = (i + 1) & 1;
                        if (!(ok = wait_bar(BAR(kBarBuf0 + b1), ((i + 1) >> 1) & 1u, abort_flag, A.status))) break;
                        ++seen[b1];
                    }
                    tc_fence_after();
                    issue_sdp(i + 1, hv);
                    // pair i's accumulations are done: its buffer takes pair i + 2
                    if (hv == 1 && i + 2 < n) load_pair(i + 2);
                }
            }
            if (!ok) {
                // copies in flight must land before the CTA leaves
                if (n > 0) drain_wait(BAR(kBarRes), 0u);
                for (int b = 0; b < 2; ++b)
                    if (issued[b] > seen[b]) drain_wait(BAR(kBarBuf0 + b), (issued[b] - 1) & 1u);
            }
            // every MMA of both issuers completes before TMEM is released
            mma_commit(BAR(kBarDrain));
            drain_wait(BAR(kBarDrain), 0u);
        }
        __syncwarp();
    } else if (warp == kDpWarp) {
        // ------------------------------------------------------------ dP
        // dP of the half hv of pair i into the second 64 columns of slot hv,
        // at the same points as S (the slot free, the pair's tiles landed).
        if (lane == 0) {
            bool ok = true;
            auto issue_dp = [&](int i, int hv) {
                const int b = i & 1;
                // KV: dP^T = V_j dO_t^T; else dP = dO_t V_j^T
                mma_half<D>(slot(hv) + 64, base + L::kRes1, base + L::buf(b, 1) + hv * kHalfBytes);
                mma_commit(BAR(kBarS0 + hv));
            };
            if (n > 0) {
                ok = wait_bar(BAR(kBarRes), 0u, abort_flag, A.status) &&
                     wait_bar(BAR(kBarBuf0), 0u, abort_flag, A.status);
                if (ok) {
                    tc_fence_after();
                    issue_dp(0, 0);
                    issue_dp(0, 1);
                }
            }
            for (int i = 0; i + 1 < n && ok; ++i) {
                for (int hv = 0; hv < 2 && ok; ++hv) {
                    if (!(ok = wait_bar(BAR(kBarFree0 + hv), i & 1u, abort_flag, A.status))) break;
                    if (hv == 0 &&
                        !(ok = wait_bar(BAR(kBarBuf0 + ((i + 1) & 1)), ((i + 1) >> 1) & 1u, abort_flag, A.status)))
                        break;
                    tc_fence_after();
                    issue_dp(i + 1, hv);
                }
            }
            mma_commit(BAR(kBarDrain));
            drain_wait(BAR(kBarDrain), 0u);
        }
        __syncwarp();
    } else if (warp == kCtlWarp) {
        // ------------------------------------------------------------ accumulations
        if (lane == 0) {
            bool ok = true;
            // the accumulations over the half hv of pair i, from slot hv, as soon
            // as the elementwise step has written it
            for (int i = 0; i < n && ok; ++i) {
                const int b = i & 1;
                // the pair's block mask, loaded before the waits so its latency
                // stays off the chain from the elementwise step to these MMAs
                const int mk = BM ? (entry(i) & 15) : 15;
                for (int hv = 0; hv < 2 && ok; ++hv) {
                    if (!(ok = wait_bar(BAR(kBarEw0 + hv), i & 1u, abort_flag, A.status))) break;
                    tc_fence_after();
                    if (KV) {
                        mma_acc_half<D, BM>(tAcc0, slot(hv), base + L::buf(b, 1), hv, i > 0, mk);       // dV += P^T dO_t
                        mma_acc_half<D, BM>(tAcc1, slot(hv) + 64, base + L::buf(b, 0), hv, i > 0, mk);  // dK += dS^T Q_t
                    } else {
                        mma_acc_half<D, BM>(tAcc0, slot(hv), base + L::buf(b, 0), hv, i > 0, mk);       // dQ += dS K_j
                    }
                    mma_commit(BAR(kBarFree0 + hv));
                }
            }
            mma_commit(BAR(kBarDrain));
            drain_wait(BAR(kBarDrain), 0u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ elementwise
        // threads r + 128h (h < kEwSplit) share TMEM lane r (a key row (KV) or
        // a query row); within each 64-column half thread r + 128h takes
        // columns [h kEwCols, (h + 1) kEwCols)
        const int r = threadIdx.x & (kBT - 1);
        const int h = threadIdx.x / kBT;
        const uint32_t tl = (uint32_t)((warp & 3) * 32) << 16;
        const float c1 = A.scale * 1.4426950408889634f;
        const int64_t xrow_r = bh * A.Sp + (int64_t)x * kBT + r;   // caller row
        const int64_t xvec_r = bh * A.Spk + (int64_t)x * kBT + r;  // per-row vectors
        const float nl2_r = KV ? 0.f : __ldg(A.nlse2 + xvec_r);
        const float ndl_r = KV ? 0.f : __ldg(A.ndelta + xvec_r);
        const int ra = r >> 6;  // this row's 64-row half of the resident tile (warp-uniform)
        bool ok = true;
        if (BM && n > 0) {
            // the accumulators start at zero (every masked accumulation adds);
            // these stores complete before the first arrival on the slot
            // barrier below (tmem_wait_st there)
            const uint32_t z[16] = {};
            const int ncols = KV ? 2 * D : D;  // dV and dK, or dQ
            for (int cb = h * (ncols / kEwSplit); cb < (h + 1) * (ncols / kEwSplit); cb += 16)
                tmem_st16(tAcc0 + tl + cb, z);
        }
        for (int i = 0; i < n; ++i) {
            const int b = i & 1;
            const int32_t e_i = entry(i);
            const int mk = e_i & 15;
            const Rows ry = entry_rows(e_i);
            const float2 *s_nl2 = reinterpret_cast<const float2 *>(g + L::kVec + b * 2 * kBT * 4);
            const float2 *s_ndl = s_nl2 + kBT / 2;
#pragma unroll 1
            for (int hv = 0; hv < 2; ++hv) {
                if (!(ok = wait_warp(BAR(kBarS0 + hv), i & 1u, abort_flag, A.status))) break;
                // the pair's copies are complete and visible here
                if (hv == 0 && !(ok = wait_warp(BAR(kBarBuf0 + b), (i >> 1) & 1u, abort_flag, A.status))) break;
                tc_fence_after();
                // padding rows of this half of the operands summed over their rows
                // (Q_t and dO_t for KV, K_j for dQ) are cleared before the half's
                // accumulations; the S/dP MMAs of the other half do not read them
                const int pr = hv * 64 + (threadIdx.x & 63), grp = threadIdx.x >> 6;
                const bool zr = !ry.valid(pr) && (grp == 0 || (KV && grp == 1));
                if (zr) zero_row<D>(g + L::buf(b, grp), pr);
                const uint32_t ts = slot(hv) + tl + h * kEwCols;  // this thread's S columns of the slot
                const int c0 = hv * 64 + h * kEwCols;              // the pair column of the first
                const int nyh = hv ? ry.hi : ry.lo;                // valid columns of this half
                uint32_t pw[kEwCols / 2], dw[kEwCols / 2];
                if (!BM || ((mk >> (2 * ra + hv)) & 1)) {  // warp-uniform
                    float sv[kEwCols], dp[kEwCols];
                    ld_cols(ts, sv);
                    ld_cols(ts + 64, dp);
                    // only a partner half with padding needs the column mask
                    if (nyh >= h * kEwCols + kEwCols)
                        ew_cols<KV, false>(sv, dp, pw, dw, c0, 0, c1, s_nl2, s_ndl, nl2_r, ndl_r);
                    else
                        ew_cols<KV, true>(sv, dp, pw, dw, c0, hv * 64 + nyh, c1, s_nl2, s_ndl, nl2_r, ndl_r);
                } else {
                    // a block the selection leaves out: P = dS = 0
#pragma unroll
                    for (int w = 0; w < kEwCols / 2; ++w) pw[w] = dw[w] = 0u;
                }
                // bf16 pairs back over the first half of the columns just read
                if (KV) st_cols(ts, pw);
                st_cols(KV ? ts + 64 : ts, dw);
                if (zr) fence_proxy_async_smem();  // this thread's zeroed row, for the MMAs
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(BAR(kBarEw0 + hv));
            }
            if (!ok) break;
        }
        // ------------------------------------------------------------ epilogue
        // the last accumulation (of the last pair's second half) is done
        if (ok && n > 0 && !wait_warp(BAR(kBarFree1), (n - 1) & 1u, abort_flag, A.status)) ok = false;
        if (ok) {
            tc_fence_after();
            const bool live = n > 0 && rx.valid(r);
            const bool exists = (int64_t)x * kBT + r < A.Sp;  // the last half of an odd 64-tile count is not
            {
                // KV: threads of even h write dV, odd h dK; dQ: every h a share of the columns
                const int which = KV ? (h & 1) : 0;
                void *dst_base = KV ? (which ? A.dk : A.dv) : A.dq;
                const float mul = (KV && which == 0) ? 1.f : A.scale;
                uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(dst_base) + xrow_r * D);
                const uint32_t tacc = which ? tAcc1 : tAcc0;
                const int cb0 = KV ? (h >> 1) : h, cstep = KV ? kEwSplit / 2 : kEwSplit;
#pragma unroll 1
                for (int cb = cb0; cb < D / 32; cb += cstep) {
                    float a[32] = {};
                    if (n > 0) tmem_ld32(tacc + tl + cb * 32, a);
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = live ? pack_bf16x2(a[2 * e] * mul, a[2 * e + 1] * mul) : 0u;
                    if (exists)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[cb * 4 + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kCtlWarp) tmem_dealloc(tmem, 512);
}

}  // namespace

size_t bwd_smem_bytes(int D) { return D == 128 ? BwdSmem<128>::kTotal : BwdSmem<64>::kTotal; }
int bwd_threads() { return kThreads; }

template <int D, bool KV, bool BM>
static cudaError_t bwd_attr() {
    return cudaFuncSetAttribute(bwd_kernel<D, KV, BM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)BwdSmem<D>::kTotal);
}

template <int D, bool BM>
static cudaError_t bwd_attr2() {
    cudaError_t e = bwd_attr<D, true, BM>();
    return e != cudaSuccess ? e : bwd_attr<D, false, BM>();
}

cudaError_t bwd_prepare() {
    cudaError_t e;
    if ((e = bwd_attr2<64, false>()) != cudaSuccess) return e;
    if ((e = bwd_attr2<64, true>()) != cudaSuccess) return e;
    if ((e = bwd_attr2<128, false>()) != cudaSuccess) return e;
    return bwd_attr2<128, true>();
}

// The dK/dV kernel, then the dQ kernel.
template <int D, bool BM>
static cudaError_t launch_pair(const BwdLaunch &L, const BwdArgs &A, unsigned grid, cudaStream_t stream) {
    bwd_kernel<D, true, BM><<<grid, kThreads, BwdSmem<D>::kTotal, stream>>>(*L.tm_q, *L.tm_k, *L.tm_v, *L.tm_do, A);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_kernel<D, false, BM><<<grid, kThreads, BwdSmem<D>::kTotal, stream>>>(*L.tm_q, *L.tm_k, *L.tm_v, *L.tm_do, A);
    return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdLaunch &L, cudaStream_t stream) {
    const int64_t rows = (int64_t)L.BH * L.Sp;
    const int Dv = L.D / 8;
    delta_kernel<<<(unsigned)((rows * 8 + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(L.out), reinterpret_cast<const uint4 *>(L.dout), L.lse, L.ndelta, L.nlse2,
        rows, Dv, L.Sp, L.Spk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const Geo G{L.T, L.NTc, L.NTk};
    const int64_t nx = (int64_t)L.BH * L.NTk;
    pairs_kernel<<<(unsigned)((nx + 3) / 4), 128, (size_t)4 * (L.NTk / 4 + 1) * 4, stream>>>(
        L.q2k_idx, L.q2k_num, L.block_sizes, G, L.max_kv, L.maxlen, (int64_t)L.BH, L.pl, L.pc, L.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k2q_kernel<<<(unsigned)L.BH, 1024, (size_t)(L.NTk + 1) * 4, stream>>>(L.pl, L.pc, L.block_sizes, G, L.maxlen,
                                                                          L.k2q_offs, L.k2q_list);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    BwdArgs A;
    A.nlse2 = L.nlse2;
    A.ndelta = L.ndelta;
    A.block_sizes = L.block_sizes;
    A.pl = L.pl;
    A.pc = L.pc;
    A.k2q_offs = L.k2q_offs;
    A.k2q_list = L.k2q_list;
    A.dq = L.dq;
    A.dk = L.dk;
    A.dv = L.dv;
    A.status = L.status;
    A.G = G;
    A.maxlen = L.maxlen;
    A.Sp = L.Sp;
    A.Spk = L.Spk;
    A.scale = L.scale;
    const unsigned grid = (unsigned)nx;
    const bool bm = L.T == 64;
    if (L.D == 128) return bm ? launch_pair<128, true>(L, A, grid, stream) : launch_pair<128, false>(L, A, grid, stream);
    return bm ? launch_pair<64, true>(L, A, grid, stream) : launch_pair<64, false>(L, A, grid, stream);
}

}  // namespace vsa
