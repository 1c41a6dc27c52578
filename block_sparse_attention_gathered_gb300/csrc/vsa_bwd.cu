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
// Kernels (128-token tiles):
//   delta_kernel   delta = rowsum(dout * out) in fp32, one pass over both.
//   k2q_kernel     per (batch, head) the transposed selection: for every key
//                  tile, the query tiles that select it, in ascending order
//                  (one CTA per (batch, head), deterministic).
//   dkdv_kernel    one CTA per (batch, head, key tile j): K_j and V_j stay in
//                  shared memory; for every query tile t that selects j,
//                  S^T = K_j Q_t^T and dP^T = V_j dO_t^T go to TMEM, four
//                  elementwise warps (one thread per key row) form P^T and
//                  dS^T in bf16 in shared memory, and dV += P^T dO_t,
//                  dK += dS^T Q_t accumulate in TMEM.
//   dq_kernel      one CTA per (batch, head, query tile t): Q_t and dO_t stay;
//                  for every selected key tile, S and dP again, dS in shared
//                  memory, dQ += dS K_j in TMEM.  Recomputing S and dP keeps
//                  dQ free of atomics and the result deterministic.
// Padding rows are kept out of every product: P and dS are set (not
// multiplied) to 0 outside the valid rows and columns, and padding rows of an
// operand that is summed over (Q and dO in dk/dv, K in dq) are zeroed in shared
// memory first, so NaN/Inf padding never meets a zero weight.  Every wait is
// bounded; on expiry the CTA flags VSA_ERR_TIMEOUT and returns.
#include <cuda_bf16.h>

#include "vsa_internal.h"
#include "vsa_ptx.cuh"
#include "vsa_wait.cuh"

namespace vsa {
namespace {

using namespace ptx;

constexpr int kBT = 128;            // tile rows (queries or keys)
constexpr int kEwThreads = 128;     // elementwise warps 0..3, one thread per row
constexpr int kCtlWarp = 4;         // TMA + MMA issue (lane 0)
constexpr uint32_t kChunkBytes = kBT * 128;  // one 64-column (128-byte) chunk of a 128-row tile

template <int D>
struct BwdCfg {
    static constexpr uint32_t kTile = kBT * D * 2;   // one Q/K/V/dO tile in shared memory
    static constexpr uint32_t kPanel = kBT * kBT * 2;  // P^T, dS^T or dS: 128 x 128 bf16
    static constexpr uint32_t kIdescSq = idesc_bf16(128, kBT, false);  // S-like products, N = 128
    static constexpr uint32_t kIdescAcc = idesc_bf16(128, D, true);    // accumulations, B MN-major
};

// Byte offset of element (row, col) of a 128-row bf16 panel stored as 64-column
// chunks with the 128-byte swizzle (16-byte granule g of row r sits at g ^ (r & 7)).
__device__ __forceinline__ uint32_t sw128(int row, int col) {
    const int chunk = col >> 6, g = (col >> 3) & 7;
    return (uint32_t)(chunk * kChunkBytes + row * 128 + ((g ^ (row & 7)) << 4) + (col & 7) * 2);
}

// Zeroes rows [from, 128) of a tile of D columns (whole rows, so the swizzle
// does not matter); thread `row` clears its own row.
template <int D>
__device__ __forceinline__ void zero_row_if(uint8_t *tile, int row, int from) {
    if (row < from) return;
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        uint4 *p = reinterpret_cast<uint4 *>(tile + c * kChunkBytes + row * 128);
#pragma unroll
        for (int g = 0; g < 8; ++g) p[g] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Issues the D/16 MMAs of a 128 x 128 product over D (both operands K-major).
template <int D>
__device__ __forceinline__ void mma_sq(uint32_t tdst, uint32_t a_saddr, uint32_t b_saddr) {
    const uint64_t a = sdesc_sw128(a_saddr, 16, 1024), b = sdesc_sw128(b_saddr, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        mma_ss(tdst, a + (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2, b + (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2,
               BwdCfg<D>::kIdescSq, kk > 0 ? 1u : 0u);
}

// Issues the 8 MMAs of acc(128 x D) += panel(128 x 128, K-major) x tile(128 x D,
// MN-major: the tile's rows are the summed dimension).
template <int D>
__device__ __forceinline__ void mma_acc(uint32_t tacc, uint32_t panel_saddr, uint32_t tile_saddr, bool accumulate) {
    const uint64_t a = sdesc_sw128(panel_saddr, 16, 1024), b = sdesc_sw128(tile_saddr, kChunkBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < kBT / 16; ++kk)
        mma_ss(tacc, a + (kk >> 2) * (kChunkBytes >> 4) + (kk & 3) * 2, b + kk * (2048 >> 4), BwdCfg<D>::kIdescAcc,
               (accumulate || kk > 0) ? 1u : 0u);
}

// ---------------------------------------------------------------- delta
__global__ void __launch_bounds__(256) delta_kernel(const uint4 *__restrict__ out, const uint4 *__restrict__ dout,
                                                   float *__restrict__ delta, int64_t rows, int Dv) {
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
    if (row < rows && sub == 0) delta[row] = acc;
}

// ---------------------------------------------------------------- k2q
// offs [B*H, NT+1] and list [B*H, NT*max_kv]: list[bh][offs[bh][j] ...] are the
// query tiles selecting key tile j, ascending.  Entries out of range are
// skipped and flagged.
__global__ void __launch_bounds__(1024)
    k2q_kernel(const int32_t *__restrict__ q2k_idx, const int32_t *__restrict__ q2k_num, int NT, int max_kv,
               int32_t *__restrict__ offs, int32_t *__restrict__ list, int32_t *status) {
    extern __shared__ int32_t cnt[];  // [NT + 1]
    const int64_t bh = blockIdx.x;
    const int tid = threadIdx.x;
    for (int j = tid; j <= NT; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    bool bad = false;
    for (int64_t e = tid; e < (int64_t)NT * max_kv; e += blockDim.x) {
        const int t = (int)(e / max_kv), i = (int)(e - (int64_t)t * max_kv);
        int K = __ldg(q2k_num + bh * NT + t);
        K = K < 0 ? 0 : (K > max_kv ? max_kv : K);
        if (i >= K) continue;
        const int j = __ldg(q2k_idx + (bh * NT + t) * max_kv + i);
        if (j < 0 || j >= NT) {
            bad = true;
            continue;
        }
        atomicAdd(&cnt[j + 1], 1);
    }
    __syncthreads();
    if (tid == 0) {  // exclusive scan (NT <= 8192: a short serial pass)
        for (int j = 1; j <= NT; ++j) cnt[j] += cnt[j - 1];
    }
    __syncthreads();
    for (int j = tid; j <= NT; j += blockDim.x) offs[bh * (NT + 1) + j] = cnt[j];
    __syncthreads();
    // fill in ascending t: one row t per round, each key tile appears at most
    // once per row (distinct selections), so its cursor advances in t order
    int32_t *lst = list + bh * (int64_t)NT * max_kv;
    for (int t = 0; t < NT; ++t) {
        int K = __ldg(q2k_num + bh * NT + t);
        K = K < 0 ? 0 : (K > max_kv ? max_kv : K);
        for (int i = tid; i < K; i += blockDim.x) {
            const int j = __ldg(q2k_idx + (bh * NT + t) * max_kv + i);
            if (j < 0 || j >= NT) continue;
            lst[atomicAdd(&cnt[j], 1)] = t;
        }
        __syncthreads();
    }
    if (bad) atomicOr(status, kFlagIndex);
}

// ---------------------------------------------------------------- shared memory
template <int D>
struct BwdSmem {
    static constexpr uint32_t kA = 0;                                   // K_j (dkdv) / Q_t (dq)
    static constexpr uint32_t kB = kA + BwdCfg<D>::kTile;               // V_j / dO_t
    static constexpr uint32_t kC = kB + BwdCfg<D>::kTile;               // Q_t / K_j
    static constexpr uint32_t kE = kC + BwdCfg<D>::kTile;               // dO_t / V_j
    static constexpr uint32_t kP = kE + BwdCfg<D>::kTile;               // P^T panel (dkdv)
    static constexpr uint32_t kS = kP + BwdCfg<D>::kPanel;              // dS^T / dS panel
    static constexpr uint32_t kVec = kS + BwdCfg<D>::kPanel;            // lse [128], delta [128] floats
    static constexpr uint32_t kBars = kVec + 2 * kBT * 4;               // 8 mbarriers
    static constexpr uint32_t kSlot = kBars + 8 * 8;                    // TMEM address
    static constexpr uint32_t kFlag = kSlot + 4;                        // abort flag
    static constexpr uint32_t kTotal = kFlag + 4 + 1024;                // + alignment slack
};

struct BwdArgs {
    const float *lse;           // [B*H*Sp] natural log
    const float *delta;         // [B*H*Sp]
    const int32_t *q2k_idx, *q2k_num, *block_sizes;
    const int32_t *k2q_offs, *k2q_list;
    void *dq, *dk, *dv;         // bf16 [B*H*Sp, D]
    int32_t *status;
    int32_t NT, max_kv;
    int64_t Sp;
    float scale;
};

// mbarriers: resident tiles loaded, per-pair tiles loaded, S and dP in TMEM,
// P/dS panels written, pair's accumulations done, and the issuer's final drain
enum { kBarLd0 = 0, kBarLd1 = 1, kBarS = 2, kBarEw = 3, kBarPair = 4, kBarDrain = 5 };

// ---------------------------------------------------------------- dK, dV
template <int D>
__global__ void __launch_bounds__(160, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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
    const float *s_lse = reinterpret_cast<const float *>(g + L::kVec);
    const float *s_dl = s_lse + kBT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int64_t bhj = blockIdx.x;
    const int NT = A.NT;
    const int j = (int)(bhj % NT);
    const int64_t bh = bhj / NT;
    const int n_j = __ldg(A.block_sizes + j);
    const int32_t off0 = __ldg(A.k2q_offs + bh * (NT + 1) + j), off1 = __ldg(A.k2q_offs + bh * (NT + 1) + j + 1);
    const int32_t *lst = A.k2q_list + bh * (int64_t)NT * A.max_kv + off0;
    const int n = off1 - off0;

    if (threadIdx.x == 0) {
        mbar_init(BAR(kBarLd0), 1);
        mbar_init(BAR(kBarLd1), 1);
        mbar_init(BAR(kBarS), 1);
        mbar_init(BAR(kBarEw), kEwThreads);
        mbar_init(BAR(kBarPair), 1);
        mbar_init(BAR(kBarDrain), 1);
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
    const uint32_t tS = tmem, tdP = tmem + kBT, tdV = tmem + 2 * kBT, tdK = tmem + 2 * kBT + D;

    if (warp == kCtlWarp) {
        if (lane == 0) {
            const int32_t krow = (int32_t)(bh * A.Sp + (int64_t)j * kBT);
            bool ok = true;
            int ld1 = 0, ld1_seen = 0;  // per-pair loads issued / waited for
            if (n > 0) {
                mbar_arrive_expect_tx(BAR(kBarLd0), 2 * C::kTile);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(base + L::kA + c * kChunkBytes, &tm_k, c * 64, krow, BAR(kBarLd0), l2_policy_evict_first());
                    tma_load_2d(base + L::kB + c * kChunkBytes, &tm_v, c * 64, krow, BAR(kBarLd0), l2_policy_evict_first());
                }
            }
            for (int i = 0; i < n && ok; ++i) {
                const int t = __ldg(lst + i);
                // the previous pair's products are done: Q, dO and both panels are free
                if (i > 0 && !(ok = wait_bar(BAR(kBarPair), (i - 1) & 1u, abort_flag, A.status))) break;
                const int64_t qrow = bh * A.Sp + (int64_t)t * kBT;
                mbar_arrive_expect_tx(BAR(kBarLd1), 2 * C::kTile + 2 * kBT * 4);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(base + L::kC + c * kChunkBytes, &tm_q, c * 64, (int32_t)qrow, BAR(kBarLd1), l2_policy_evict_last());
                    tma_load_2d(base + L::kE + c * kChunkBytes, &tm_do, c * 64, (int32_t)qrow, BAR(kBarLd1), l2_policy_evict_last());
                }
                bulk_load(base + L::kVec, A.lse + qrow, kBT * 4, BAR(kBarLd1));
                bulk_load(base + L::kVec + kBT * 4, A.delta + qrow, kBT * 4, BAR(kBarLd1));
                ++ld1;
                if (i == 0 && !(ok = wait_bar(BAR(kBarLd0), 0u, abort_flag, A.status))) break;
                if (!(ok = wait_bar(BAR(kBarLd1), i & 1u, abort_flag, A.status))) break;
                ++ld1_seen;
                tc_fence_after();
                mma_sq<D>(tS, base + L::kA, base + L::kC);   // S^T = K_j Q_t^T
                mma_sq<D>(tdP, base + L::kB, base + L::kE);  // dP^T = V_j dO_t^T
                mma_commit(BAR(kBarS));
                if (!(ok = wait_bar(BAR(kBarEw), i & 1u, abort_flag, A.status))) break;
                tc_fence_after();
                mma_acc<D>(tdV, base + L::kP, base + L::kE, i > 0);  // dV += P^T dO_t
                mma_acc<D>(tdK, base + L::kS, base + L::kC, i > 0);  // dK += dS^T Q_t
                mma_commit(BAR(kBarPair));
            }
            if (!ok) {
                // copies in flight must land before the CTA leaves
                if (n > 0) drain_wait(BAR(kBarLd0), 0u);
                if (ld1 > ld1_seen) drain_wait(BAR(kBarLd1), (ld1 - 1) & 1u);
            }
            // every MMA this thread issued completes before TMEM is released
            mma_commit(BAR(kBarDrain));
            drain_wait(BAR(kBarDrain), 0u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ elementwise
        const int r = threadIdx.x;  // key row (TMEM lane)
        const uint32_t tl = (uint32_t)(warp * 32) << 16;
        const float c1 = A.scale * 1.4426950408889634f;
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            const int t = __ldg(lst + i);
            const int n_t = __ldg(A.block_sizes + t);
            if (!(ok = wait_warp(BAR(kBarS), i & 1u, abort_flag, A.status))) break;
            // the pair's copies (Q_t, dO_t, lse, delta) are complete and visible here
            if (!(ok = wait_warp(BAR(kBarLd1), i & 1u, abort_flag, A.status))) break;
            tc_fence_after();
            // Q_t and dO_t are summed over their rows next: clear the padding rows
            zero_row_if<D>(g + L::kC, r, n_t);
            zero_row_if<D>(g + L::kE, r, n_t);
#pragma unroll 1
            for (int cb = 0; cb < kBT / 32; ++cb) {
                float s[32], dp[32];
                tmem_ld32(tS + tl + cb * 32, s);
                tmem_ld32(tdP + tl + cb * 32, dp);
                uint32_t pw[16], dw[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = cb * 32 + e + h;  // query column
                        const bool live = r < n_j && c < n_t;
                        const float p = live ? ex2(fmaf(c1, s[e + h], -s_lse[c] * 1.4426950408889634f)) : 0.f;
                        pv[h] = p;
                        dv[h] = live ? p * (dp[e + h] - s_dl[c]) : 0.f;
                    }
                    pw[e >> 1] = pack_bf16x2(pv[0], pv[1]);
                    dw[e >> 1] = pack_bf16x2(dv[0], dv[1]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // four 16-byte granules of 8 columns
                    const uint32_t o = sw128(r, cb * 32 + q * 8);
                    *reinterpret_cast<uint4 *>(g + L::kP + o) = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
                    *reinterpret_cast<uint4 *>(g + L::kS + o) = make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(BAR(kBarEw));
        }
        // ------------------------------------------------------------ epilogue
        if (ok && n > 0 && !wait_warp(BAR(kBarPair), (n - 1) & 1u, abort_flag, A.status)) ok = false;
        if (ok) {
            tc_fence_after();
            const int64_t orow = bh * A.Sp + (int64_t)j * kBT + r;
            uint4 *dk = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(A.dk) + orow * D);
            uint4 *dv = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(A.dv) + orow * D);
            const bool live = n > 0 && r < n_j;
#pragma unroll 1
            for (int cb = 0; cb < D / 32; ++cb) {
                float a[32] = {}, b[32] = {};
                if (n > 0) {
                    tmem_ld32(tdK + tl + cb * 32, a);
                    tmem_ld32(tdV + tl + cb * 32, b);
                }
                uint32_t wk[16], wv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    wk[e] = live ? pack_bf16x2(a[2 * e] * A.scale, a[2 * e + 1] * A.scale) : 0u;
                    wv[e] = live ? pack_bf16x2(b[2 * e], b[2 * e + 1]) : 0u;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    dk[cb * 4 + q] = make_uint4(wk[4 * q], wk[4 * q + 1], wk[4 * q + 2], wk[4 * q + 3]);
                    dv[cb * 4 + q] = make_uint4(wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kCtlWarp) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- dQ
template <int D>
__global__ void __launch_bounds__(160, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do, const BwdArgs A) {
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

    const int64_t bht = blockIdx.x;
    const int NT = A.NT;
    const int t = (int)(bht % NT);
    const int64_t bh = bht / NT;
    const int n_t = __ldg(A.block_sizes + t);
    int n = __ldg(A.q2k_num + bht);
    n = n < 0 ? 0 : (n > A.max_kv ? A.max_kv : n);
    const int32_t *sel = A.q2k_idx + bht * A.max_kv;

    if (threadIdx.x == 0) {
        mbar_init(BAR(kBarLd0), 1);
        mbar_init(BAR(kBarLd1), 1);
        mbar_init(BAR(kBarS), 1);
        mbar_init(BAR(kBarEw), kEwThreads);
        mbar_init(BAR(kBarPair), 1);
        mbar_init(BAR(kBarDrain), 1);
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
    const uint32_t tS = tmem, tdP = tmem + kBT, tdQ = tmem + 2 * kBT;

    if (warp == kCtlWarp) {
        if (lane == 0) {
            const int32_t qrow = (int32_t)(bh * A.Sp + (int64_t)t * kBT);
            bool ok = true;
            int ld1 = 0, ld1_seen = 0;
            if (n > 0) {
                mbar_arrive_expect_tx(BAR(kBarLd0), 2 * C::kTile);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(base + L::kA + c * kChunkBytes, &tm_q, c * 64, qrow, BAR(kBarLd0), l2_policy_evict_first());
                    tma_load_2d(base + L::kB + c * kChunkBytes, &tm_do, c * 64, qrow, BAR(kBarLd0), l2_policy_evict_first());
                }
            }
            for (int i = 0; i < n && ok; ++i) {
                int jj = __ldg(sel + i);
                jj = (jj < 0 || jj >= NT) ? 0 : jj;  // bad entries were flagged by k2q_kernel; read a valid tile
                if (i > 0 && !(ok = wait_bar(BAR(kBarPair), (i - 1) & 1u, abort_flag, A.status))) break;
                const int32_t krow = (int32_t)(bh * A.Sp + (int64_t)jj * kBT);
                mbar_arrive_expect_tx(BAR(kBarLd1), 2 * C::kTile);
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(base + L::kC + c * kChunkBytes, &tm_k, c * 64, krow, BAR(kBarLd1), l2_policy_evict_last());
                    tma_load_2d(base + L::kE + c * kChunkBytes, &tm_v, c * 64, krow, BAR(kBarLd1), l2_policy_evict_last());
                }
                ++ld1;
                if (i == 0 && !(ok = wait_bar(BAR(kBarLd0), 0u, abort_flag, A.status))) break;
                if (!(ok = wait_bar(BAR(kBarLd1), i & 1u, abort_flag, A.status))) break;
                ++ld1_seen;
                tc_fence_after();
                mma_sq<D>(tS, base + L::kA, base + L::kC);   // S = Q_t K_j^T
                mma_sq<D>(tdP, base + L::kB, base + L::kE);  // dP = dO_t V_j^T
                mma_commit(BAR(kBarS));
                if (!(ok = wait_bar(BAR(kBarEw), i & 1u, abort_flag, A.status))) break;
                tc_fence_after();
                mma_acc<D>(tdQ, base + L::kS, base + L::kC, i > 0);  // dQ += dS K_j
                mma_commit(BAR(kBarPair));
            }
            if (!ok) {
                if (n > 0) drain_wait(BAR(kBarLd0), 0u);
                if (ld1 > ld1_seen) drain_wait(BAR(kBarLd1), (ld1 - 1) & 1u);
            }
            mma_commit(BAR(kBarDrain));
            drain_wait(BAR(kBarDrain), 0u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ elementwise
        const int r = threadIdx.x;  // query row (TMEM lane)
        const uint32_t tl = (uint32_t)(warp * 32) << 16;
        const float c1 = A.scale * 1.4426950408889634f;
        const int64_t orow = bh * A.Sp + (int64_t)t * kBT + r;
        const float lse2 = __ldg(A.lse + orow) * 1.4426950408889634f;
        const float dl = __ldg(A.delta + orow);
        bool ok = true;
        for (int i = 0; i < n; ++i) {
            int jj = __ldg(sel + i);
            const int n_j = (jj < 0 || jj >= NT) ? 0 : __ldg(A.block_sizes + jj);
            if (!(ok = wait_warp(BAR(kBarS), i & 1u, abort_flag, A.status))) break;
            // the pair's copies (K_j, V_j) are complete and visible here
            if (!(ok = wait_warp(BAR(kBarLd1), i & 1u, abort_flag, A.status))) break;
            tc_fence_after();
            // K_j is summed over its rows next: clear the padding rows
            zero_row_if<D>(g + L::kC, r, n_j);
#pragma unroll 1
            for (int cb = 0; cb < kBT / 32; ++cb) {
                float s[32], dp[32];
                tmem_ld32(tS + tl + cb * 32, s);
                tmem_ld32(tdP + tl + cb * 32, dp);
                uint32_t dw[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float dv[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = cb * 32 + e + h;  // key column
                        const bool live = r < n_t && c < n_j;
                        const float p = live ? ex2(fmaf(c1, s[e + h], -lse2)) : 0.f;
                        dv[h] = live ? p * (dp[e + h] - dl) : 0.f;
                    }
                    dw[e >> 1] = pack_bf16x2(dv[0], dv[1]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t o = sw128(r, cb * 32 + q * 8);
                    *reinterpret_cast<uint4 *>(g + L::kS + o) = make_uint4(dw[4 * q], dw[4 * q + 1], dw[4 * q + 2], dw[4 * q + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(BAR(kBarEw));
        }
        if (ok && n > 0 && !wait_warp(BAR(kBarPair), (n - 1) & 1u, abort_flag, A.status)) ok = false;
        if (ok) {
            tc_fence_after();
            uint4 *dq = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(A.dq) + orow * D);
            const bool live = n > 0 && r < n_t;
#pragma unroll 1
            for (int cb = 0; cb < D / 32; ++cb) {
                float a[32] = {};
                if (n > 0) tmem_ld32(tdQ + tl + cb * 32, a);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = live ? pack_bf16x2(a[2 * e] * A.scale, a[2 * e + 1] * A.scale) : 0u;
#pragma unroll
                for (int q = 0; q < 4; ++q) dq[cb * 4 + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
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

cudaError_t bwd_prepare() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(dkdv_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdSmem<64>::kTotal)))
        return e;
    if ((e = cudaFuncSetAttribute(dkdv_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdSmem<128>::kTotal)))
        return e;
    if ((e = cudaFuncSetAttribute(dq_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdSmem<64>::kTotal)))
        return e;
    return cudaFuncSetAttribute(dq_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdSmem<128>::kTotal);
}

cudaError_t launch_bwd(const BwdLaunch &L, cudaStream_t stream) {
    const int64_t rows = (int64_t)L.BH * L.Sp;
    const int Dv = L.D / 8;
    delta_kernel<<<(unsigned)((rows * 8 + 255) / 256), 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(L.out), reinterpret_cast<const uint4 *>(L.dout), L.delta, rows, Dv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k2q_kernel<<<(unsigned)L.BH, 1024, (size_t)(L.NT + 1) * 4, stream>>>(L.q2k_idx, L.q2k_num, L.NT, L.max_kv,
                                                                         L.k2q_offs, L.k2q_list, L.status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    BwdArgs A;
    A.lse = L.lse;
    A.delta = L.delta;
    A.q2k_idx = L.q2k_idx;
    A.q2k_num = L.q2k_num;
    A.block_sizes = L.block_sizes;
    A.k2q_offs = L.k2q_offs;
    A.k2q_list = L.k2q_list;
    A.dq = L.dq;
    A.dk = L.dk;
    A.dv = L.dv;
    A.status = L.status;
    A.NT = L.NT;
    A.max_kv = L.max_kv;
    A.Sp = L.Sp;
    A.scale = L.scale;
    const unsigned grid = (unsigned)((int64_t)L.BH * L.NT);
    if (L.D == 128) {
        dkdv_kernel<128><<<grid, 160, BwdSmem<128>::kTotal, stream>>>(*L.tm_q, *L.tm_k, *L.tm_v, *L.tm_do, A);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        dq_kernel<128><<<grid, 160, BwdSmem<128>::kTotal, stream>>>(*L.tm_q, *L.tm_k, *L.tm_v, *L.tm_do, A);
    } else {
        dkdv_kernel<64><<<grid, 160, BwdSmem<64>::kTotal, stream>>>(*L.tm_q, *L.tm_k, *L.tm_v, *L.tm_do, A);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        dq_kernel<64><<<grid, 160, BwdSmem<64>::kTotal, stream>>>(*L.tm_q, *L.tm_k, *L.tm_v, *L.tm_do, A);
    }
    return cudaGetLastError();
}

}  // namespace vsa
