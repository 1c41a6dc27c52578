// Block-sparse attention forward for sm_103a: warp-specialised, TMA + tcgen05.
//
// What it computes (FastVideo commit 8503617, fastvideo-kernel/python: the
// commit adding the sm_121a tile-128 forward, and the sm_121a hardening
// commit): for every query tile t of every (batch, head), softmax(scale *
// Q_t K_L^T) V_L over the valid rows L of the key tiles listed in
// q2k_idx[0:q2k_num]; keys past a tile's valid count are masked, rows without
// keys are 0, a NaN softmax sum gives a NaN row, padding output rows are 0.
//
// Design (this file's own; the page's kernels target other hardware):
//   * One persistent CTA per SM takes 256-query-row work items (two 128-row
//     "units") from an on-device order list, longest first.  A unit is one
//     128-token query tile, or two consecutive 64-token tiles.
//   * The producer warp turns the selections of the item's tiles into
//     shared-memory bitmaps and streams the UNION of the selected key tiles,
//     in ascending order, through a ring of K/V stages with TMA, so a key
//     tile that both units select is fetched once ("gathered" fetch).
//   * The MMA warp issues S_u = Q_u K_j^T (tcgen05, smem x smem -> TMEM) for
//     the units that select j, and O_u += P_u V_j with P read from TMEM.
//   * Two softmax warpgroups, one per unit, run the online softmax with exp2
//     on their TMEM rows (one thread per query row), write P (bf16) into the
//     TMEM columns of S, rescale O only when the running maximum grows by more
//     than 2^8 (lazy rescale), and finish with O / l.  The two units
//     ping-pong: the tensor core works on one unit while the other's softmax
//     runs.
//   * Masks are applied only on tail key tiles (valid count < tile); the V
//     rows past the valid count of a tail tile are zeroed in shared memory
//     before P V, so NaN/Inf padding cannot reach the output (0 * NaN = NaN).
//   * Every wait is bounded (about 2 s); on expiry the CTA sets the timeout
//     flag, drains its outstanding copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>

#include "vsa_internal.h"
#include "vsa_ptx.cuh"

namespace vsa {
namespace {

using namespace ptx;

constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kProducerWarp = 9;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

// Instruction descriptor, tcgen05.mma kind::f16: bf16 A and B, fp32 D,
// A K-major, B K-major or MN-major, shape M x N.
constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle (rows of 128 bytes,
// 8-row / 1024-byte swizzle atoms; buffers are 1024-byte aligned).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

template <int T, int D>
struct Cfg {
    static_assert(T == 64 || T == 128, "tile");
    static_assert(D == 64 || D == 128, "head_dim");
    static constexpr int kChunks = D / 64;                    // 128-byte column chunks per row
    static constexpr uint32_t kQChunk = kUnitRows * 128;      // bytes of one Q column chunk
    static constexpr uint32_t kQBytes = kUnitRows * D * 2;    // one unit's Q
    static constexpr uint32_t kKVChunk = T * 128;             // bytes of one K/V column chunk
    static constexpr uint32_t kStageBytes = T * D * 2;        // one K or V tile
    static constexpr int kStages = kStageBytes >= 32768 ? 4 : 8;
    static constexpr uint32_t kTmemO0 = 0, kTmemO1 = D, kTmemS0 = 2 * D, kTmemS1 = 2 * D + T;
    static constexpr uint32_t kTmemCols = (2 * D + 2 * T <= 256) ? 256 : 512;
    static constexpr uint32_t kIdescQK = idesc_bf16(128, T, false);
    static constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
    // barrier indices
    static constexpr int kKvFull = 0, kKvEmpty = kStages, kQFull = 2 * kStages, kQEmpty = kQFull + 2,
                         kSFull = kQEmpty + 2, kPFull = kSFull + 2, kODone = kPFull + 2,
                         kBmFull = kODone + 2, kBmEmpty = kBmFull + 2, kDone = kBmEmpty + 2,
                         kNumBars = kDone + 1;
};

struct SmemPlan {
    uint32_t q, ring, bm, hdr, bars, tslot, flag, total;
};

template <int T, int D>
__host__ __device__ inline SmemPlan smem_plan(int bm_words) {
    using C = Cfg<T, D>;
    SmemPlan s;
    s.q = 0;
    s.ring = 2 * C::kQBytes;
    s.bm = s.ring + C::kStages * C::kStageBytes;
    s.hdr = s.bm + 2u * 4u * 4u * (uint32_t)bm_words;
    s.bars = s.hdr + 32;
    s.tslot = s.bars + 8u * C::kNumBars;
    s.flag = s.tslot + 4;
    s.total = ((s.flag + 4 + 15) & ~15u) + 1024;  // + slack to align the base to 1024
    return s;
}

// Bounded wait on an mbarrier phase.  Returns false when the CTA is aborting
// (another role gave up) or when this wait itself ran past the limit.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         int32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(status, kFlagTimeout);
                return false;
            }
        }
    }
}

// Warp-uniform form: every lane of the warp gets the same answer, so the
// .sync.aligned tcgen05 instructions that follow are never reached by part of
// a warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *status) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, status));
}

// Wait used only while draining after an abort: ignores the abort flag, gives
// up after the limit (the copies it waits for complete on their own).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

// Tile index held by bitmap slot s (unit = s/2, half = s%2) of item g.
template <int T>
__device__ __forceinline__ int tile_of_slot(int g, int s) {
    if (T == 128) return (s & 1) ? -1 : 2 * g + (s >> 1);
    return 4 * g + s;
}

template <int T, int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams P) {
    using C = Cfg<T, D>;
    constexpr int NS = C::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int W = P.bm_words;
    const SmemPlan L = smem_plan<T, D>(W);
    const uint32_t sQ = base + L.q;
    const uint32_t sRing = base + L.ring;
    uint32_t *bm = reinterpret_cast<uint32_t *>(gbase + L.bm);       // [2][4][W]
    volatile int32_t *hdr = reinterpret_cast<int32_t *>(gbase + L.hdr);  // [2][4]
    const uint32_t bars = base + L.bars;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(gbase + L.tslot);
    volatile int *abort_flag = reinterpret_cast<int *>(gbase + L.flag);
    auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(BAR(C::kKvFull + s), 1);
            mbar_init(BAR(C::kKvEmpty + s), 1);
        }
        for (int u = 0; u < 2; ++u) {
            mbar_init(BAR(C::kQFull + u), 1);
            mbar_init(BAR(C::kQEmpty + u), 1);
            mbar_init(BAR(C::kSFull + u), 1);
            mbar_init(BAR(C::kPFull + u), 128);
            mbar_init(BAR(C::kODone + u), 1);
            mbar_init(BAR(C::kBmFull + u), 32);
            mbar_init(BAR(C::kBmEmpty + u), 32 + 32 * kSoftmaxWarps);
        }
        mbar_init(BAR(C::kDone), 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tslot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    const int NT = P.NT;
    const int64_t Sp = P.Sp;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        const uint64_t pol_kv = l2_policy_evict_last();
        const uint64_t pol_q = l2_policy_evict_first();
        uint32_t fills = 0;
        uint32_t q_loads = 0;
        for (uint32_t it = 0;; ++it) {
            const int p = it & 1;
            if (!wait_warp(BAR(C::kBmEmpty + p), ((it >> 1) & 1u) ^ 1u, abort_flag, P.status)) break;
            int slot = 0;
            if (lane == 0) slot = atomicAdd(P.work_counter, 1);
            slot = __shfl_sync(0xffffffffu, slot, 0);
            const int item = (slot < P.n_items) ? __ldg(P.order + slot) : -1;
            uint32_t *bmp = bm + p * 4 * W;
            int bad = 0;
            if (item >= 0) {
                for (int i = lane; i < 4 * W; i += 32) bmp[i] = 0u;
                __syncwarp();
                const int bh = item / P.G, g = item - (item / P.G) * P.G;
                for (int s = 0; s < 4; ++s) {
                    const int t = tile_of_slot<T>(g, s);
                    if (t < 0 || t >= NT) continue;
                    const int64_t row = (int64_t)bh * NT + t;
                    int K = __ldg(P.q2k_num + row);
                    if (K < 0 || K > P.max_kv) {
                        bad = 1;
                        K = K < 0 ? 0 : P.max_kv;
                    }
                    const int32_t *sel = P.q2k_idx + row * P.max_kv;
                    for (int i = lane; i < K; i += 32) {
                        const int j = __ldg(sel + i);
                        if (j < 0 || j >= NT) {
                            bad = 1;
                            continue;
                        }
                        if (__ldg(P.block_sizes + j) <= 0) continue;
                        const uint32_t bit = 1u << (j & 31);
                        const uint32_t old = atomicOr(&bmp[s * W + (j >> 5)], bit);
                        if (old & bit) bad = 1;  // repeated index
                    }
                }
                if (lane == 0) hdr[p * 4] = item;
            } else if (lane == 0) {
                hdr[p * 4] = -1;
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(P.status, kFlagIndex);
            __syncwarp();
            mbar_arrive(BAR(C::kBmFull + p));
            if (item < 0) break;

            const int bh = item / P.G, g = item - (item / P.G) * P.G;
            const int64_t row0 = (int64_t)bh * Sp + (int64_t)g * kItemRows;
            bool ok = true;
            for (int u = 0; u < 2 && ok; ++u) {
                ok = wait_warp(BAR(C::kQEmpty + u), (it & 1u) ^ 1u, abort_flag, P.status);
                if (ok && lane == 0) {
                    mbar_arrive_expect_tx(BAR(C::kQFull + u), C::kQBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_2d(sQ + u * C::kQBytes + c * C::kQChunk, &tm_q, c * 64,
                                    (int32_t)(row0 + u * kUnitRows), BAR(C::kQFull + u), pol_q);
                }
            }
            if (!ok) break;
            ++q_loads;
            for (int w = 0; w < W && ok; ++w) {
                uint32_t bits = bmp[w] | bmp[W + w] | bmp[2 * W + w] | bmp[3 * W + w];
                while (bits && ok) {
                    const int j = w * 32 + __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int32_t krow = (int32_t)((int64_t)bh * Sp + (int64_t)j * T);
                    for (int kv = 0; kv < 2; ++kv) {
                        const int st = fills % NS;
                        ok = wait_warp(BAR(C::kKvEmpty + st), ((fills / NS) & 1u) ^ 1u, abort_flag, P.status);
                        if (!ok) break;
                        if (lane == 0) {
                            mbar_arrive_expect_tx(BAR(C::kKvFull + st), C::kStageBytes);
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_2d(sRing + st * C::kStageBytes + c * C::kKVChunk,
                                            kv ? (const void *)&tm_v : (const void *)&tm_k, c * 64, krow,
                                            BAR(C::kKvFull + st), pol_kv);
                        }
                        __syncwarp();
                        ++fills;
                    }
                }
            }
            if (!ok) break;
        }
        // Every copy issued must land before the CTA may exit.  In the normal
        // path the consumers already waited for all of them; after an abort
        // this drains whatever is still in flight.
        if (*abort_flag && lane == 0) {
            const uint32_t first = fills > (uint32_t)NS ? fills - NS : 0u;
            for (uint32_t f = first; f < fills; ++f) drain_wait(BAR(C::kKvFull + f % NS), (f / NS) & 1u);
            if (q_loads > 0)
                for (int u = 0; u < 2; ++u) drain_wait(BAR(C::kQFull + u), (q_loads - 1) & 1u);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        uint32_t fills = 0;
        uint32_t pcnt[2] = {0u, 0u};
        bool ok = true;
        for (uint32_t it = 0; ok; ++it) {
            const int p = it & 1;
            if (!(ok = wait_warp(BAR(C::kBmFull + p), (it >> 1) & 1u, abort_flag, P.status))) break;
            const int item = hdr[p * 4];
            if (item < 0) break;
            const uint32_t *bmp = bm + p * 4 * W;
            ok = wait_warp(BAR(C::kQFull + 0), it & 1u, abort_flag, P.status) &&
                 wait_warp(BAR(C::kQFull + 1), it & 1u, abort_flag, P.status);
            if (!ok) break;
            tc_fence_after();
            bool pending[2] = {false, false};
            bool first[2] = {true, true};
            uint32_t pend_v[2] = {0u, 0u};

            // O_u += P_u V (the V stage of u's previous member entry).
            auto flush = [&](int u) -> bool {
                if (!wait_warp(BAR(C::kPFull + u), pcnt[u] & 1u, abort_flag, P.status)) return false;
                ++pcnt[u];
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t d = tmem + (u ? C::kTmemO1 : C::kTmemO0);
                    const uint32_t a = tmem + (u ? C::kTmemS1 : C::kTmemS0);
                    const uint32_t vb = sRing + pend_v[u] * C::kStageBytes;
#pragma unroll
                    for (int kk = 0; kk < T / 16; ++kk) {
                        const uint64_t bdesc = sdesc_sw128(vb + kk * 16 * 128, C::kKVChunk, 1024);
                        mma_ts(d, a + kk * 8, bdesc, C::kIdescPV, (first[u] && kk == 0) ? 0u : 1u);
                    }
                    mma_commit(BAR(C::kODone + u));
                    const int o = 1 - u;
                    if (!(pending[o] && pend_v[o] == pend_v[u])) mma_commit(BAR(C::kKvEmpty + pend_v[u]));
                }
                __syncwarp();
                first[u] = false;
                pending[u] = false;
                return true;
            };

            for (int w = 0; w < W && ok; ++w) {
                const uint32_t m0w = bmp[w] | bmp[W + w];
                const uint32_t m1w = bmp[2 * W + w] | bmp[3 * W + w];
                uint32_t bits = m0w | m1w;
                while (bits && ok) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int j = w * 32 + b;
                    const bool mem[2] = {((m0w >> b) & 1u) != 0u, ((m1w >> b) & 1u) != 0u};
                    const uint32_t kst = fills % NS, kph = (fills / NS) & 1u;
                    ++fills;
                    const uint32_t vst = fills % NS, vph = (fills / NS) & 1u;
                    ++fills;
                    if (!(ok = wait_warp(BAR(C::kKvFull + kst), kph, abort_flag, P.status))) break;
                    tc_fence_after();
                    for (int u = 0; u < 2 && ok; ++u) {
                        if (!mem[u]) continue;
                        if (pending[u] && !(ok = flush(u))) break;
                        if (lane == 0) {
                            const uint32_t d = tmem + (u ? C::kTmemS1 : C::kTmemS0);
                            const uint32_t qb = sQ + u * C::kQBytes;
                            const uint32_t kb = sRing + kst * C::kStageBytes;
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off = (kk & 3) * 32u;  // K16 slice inside the 128-byte row
                                const uint64_t ad = sdesc_sw128(qb + (kk >> 2) * C::kQChunk + off, 16, 1024);
                                const uint64_t bd = sdesc_sw128(kb + (kk >> 2) * C::kKVChunk + off, 16, 1024);
                                mma_ss(d, ad, bd, C::kIdescQK, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(BAR(C::kSFull + u));
                        }
                        __syncwarp();
                    }
                    for (int u = 0; u < 2 && ok; ++u)
                        if (!mem[u] && pending[u]) ok = flush(u);
                    if (!ok) break;
                    if (lane == 0) mma_commit(BAR(C::kKvEmpty + kst));
                    __syncwarp();
                    if (!(ok = wait_warp(BAR(C::kKvFull + vst), vph, abort_flag, P.status))) break;
                    const int nj = __ldg(P.block_sizes + j);
                    if (nj < T) {
                        // Zero the V rows past the valid count so 0 * NaN never
                        // enters P V (rows of 128 bytes; the swizzle stays in-row).
                        uint4 *vs = reinterpret_cast<uint4 *>(gbase + L.ring + vst * C::kStageBytes);
                        const int n16 = (T - nj) * 8;
                        for (int c = 0; c < C::kChunks; ++c)
                            for (int i = lane; i < n16; i += 32)
                                vs[(c * C::kKVChunk + nj * 128) / 16 + i] = make_uint4(0u, 0u, 0u, 0u);
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    for (int u = 0; u < 2; ++u)
                        if (mem[u]) {
                            pending[u] = true;
                            pend_v[u] = vst;
                        }
                }
            }
            for (int u = 0; u < 2 && ok; ++u)
                if (pending[u]) ok = flush(u);
            if (!ok) break;
            if (lane == 0) {
                mma_commit(BAR(C::kQEmpty + 0));
                mma_commit(BAR(C::kQEmpty + 1));
            }
            __syncwarp();
            mbar_arrive(BAR(C::kBmEmpty + p));
        }
        // All MMAs of this CTA complete before TMEM is released.
        if (lane == 0) {
            mma_commit(BAR(C::kDone));
            drain_wait(BAR(C::kDone), 0u);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int u = warp >> 2;
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;  // query row within the unit
        const int half = (T == 64) ? (row >> 6) : 0;
        const uint32_t tl = (uint32_t)(q4 * 32) << 16;
        const uint32_t tS = tmem + tl + (u ? C::kTmemS1 : C::kTmemS0);
        const uint32_t tO = tmem + tl + (u ? C::kTmemO1 : C::kTmemO0);
        const float c = P.scale_log2;
        uint32_t cnt = 0;  // member entries of this unit seen so far (all items)
        for (uint32_t it = 0;; ++it) {
            const int p = it & 1;
            if (!wait_warp(BAR(C::kBmFull + p), (it >> 1) & 1u, abort_flag, P.status)) break;
            const int item = hdr[p * 4];
            if (item < 0) break;
            const uint32_t *bmp = bm + p * 4 * W;
            const int bh = item / P.G, g = item - (item / P.G) * P.G;
            const int t = (T == 128) ? 2 * g + u : 4 * g + 2 * u + half;
            const int r = (T == 128) ? row : (row & 63);
            const int n_t = (t < NT) ? __ldg(P.block_sizes + t) : 0;
            float m = -INFINITY, l = 0.f;
            uint32_t n_mine = 0;
            bool ok = true;
            const uint32_t *pa = bmp + (2 * u) * W, *pb = bmp + (2 * u + 1) * W;
            const uint32_t *pm = half ? pb : pa;
            for (int w = 0; w < W && ok; ++w) {
                uint32_t bits = pa[w] | pb[w];
                const uint32_t mine = pm[w];
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int j = w * 32 + b;
                    if (!(ok = wait_warp(BAR(C::kSFull + u), cnt & 1u, abort_flag, P.status))) break;
                    tc_fence_after();
                    if ((mine >> b) & 1u) {
                        const int nj = __ldg(P.block_sizes + j);
                        float s[T];
                        if constexpr (T == 128) tmem_ld128(tS, s);
                        else tmem_ld64(tS, s);
                        if (nj < T) {
#pragma unroll
                            for (int i = 0; i < T; ++i)
                                if (i >= nj) s[i] = -INFINITY;
                        }
                        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                        for (int i = 4; i < T; i += 4) {
                            mx0 = fmaxf(mx0, s[i]);
                            mx1 = fmaxf(mx1, s[i + 1]);
                            mx2 = fmaxf(mx2, s[i + 2]);
                            mx3 = fmaxf(mx3, s[i + 3]);
                        }
                        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
                        const float m_new = fmaxf(m, mx);
                        const bool fresh = (m == -INFINITY);
                        const bool resc = !fresh && (m_new > m + kRescaleThreshold);
                        if (__any_sync(0xffffffffu, resc)) {
                            // O of this unit holds the sum up to the previous
                            // entry once that PV completes.
                            if (!(ok = wait_warp(BAR(C::kODone + u), (cnt - 1u) & 1u, abort_flag, P.status)))
                                break;
                            tc_fence_after();
                            const float alpha = resc ? ex2(m - m_new) : 1.f;
#pragma unroll
                            for (int ch = 0; ch < D / 32; ++ch) {
                                float o[32];
                                tmem_ld32(tO + ch * 32, o);
#pragma unroll
                                for (int i = 0; i < 32; ++i) o[i] *= alpha;
                                tmem_st32(tO + ch * 32, o);
                            }
                            tmem_wait_st();
                            l *= alpha;
                        }
                        if (fresh || resc) m = m_new;
                        const float neg_m = -m;
                        float l0 = 0.f, l1 = 0.f;
#pragma unroll
                        for (int ch = 0; ch < T / 32; ++ch) {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float p0 = ex2(fmaf(s[ch * 32 + 2 * i], c, neg_m));
                                const float p1 = ex2(fmaf(s[ch * 32 + 2 * i + 1], c, neg_m));
                                pk[i] = pack_bf16x2(p0, p1);
                                // l sums the bf16 values P V actually uses, so the
                                // weights P / l stay exactly normalised.
                                l0 += __uint_as_float(pk[i] << 16);
                                l1 += __uint_as_float(pk[i] & 0xffff0000u);
                            }
                            tmem_st16(tS + ch * 16, pk);
                        }
                        l += l0 + l1;
                    } else {
                        // This half of the unit does not select tile j: its P
                        // rows are zero so O is left unchanged.
                        const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u,
                                                0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
                        for (int ch = 0; ch < T / 32; ++ch) tmem_st16(tS + ch * 16, z);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(BAR(C::kPFull + u));
                    ++cnt;
                    ++n_mine;
                }
            }
            if (!ok) break;
            // -------------------------------------------------------- epilogue
            if (n_mine > 0) {
                if (!wait_warp(BAR(C::kODone + u), (cnt - 1u) & 1u, abort_flag, P.status)) break;
                tc_fence_after();
            }
            const bool write_row = t < NT;
            const bool valid = r < n_t;
            const bool use_o = (n_mine > 0) && valid && (l != 0.f);  // NaN l keeps use_o: NaN row
            const float inv = use_o ? 1.f / l : 0.f;
            const int64_t orow = (int64_t)bh * Sp + (int64_t)t * T + r;
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(P.out) + orow * D);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                float o[32];
                if (n_mine > 0) {
                    tmem_ld32(tO + ch * 32, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;
                }
                if (write_row) {
                    uint32_t wv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        wv[i] = use_o ? pack_bf16x2(o[2 * i] * inv, o[2 * i + 1] * inv) : 0u;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[ch * 4 + i] = make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                }
            }
            if (P.lse && write_row) {
                float v = -INFINITY;
                if (use_o) v = (m + lg2(l)) * 0.69314718055994531f;
                P.lse[orow] = v;
            }
            tc_fence_before();
            mbar_arrive(BAR(C::kBmEmpty + p));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

template <int T, int D>
cudaError_t launch_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v, const AttnParams &p,
                     int grid, cudaStream_t stream) {
    const SmemPlan L = smem_plan<T, D>(p.bm_words);
    attn_fwd_kernel<T, D><<<grid, kAttnThreads, L.total, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

template <int T, int D>
AttnLaunchInfo info_t(int bm_words) {
    return AttnLaunchInfo{Cfg<T, D>::kStages, (int)smem_plan<T, D>(bm_words).total};
}

template <int T, int D>
cudaError_t prepare_t() {
    const SmemPlan L = smem_plan<T, D>((kMaxTiles + 31) / 32);
    return cudaFuncSetAttribute(attn_fwd_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)L.total);
}

}  // namespace

AttnLaunchInfo attn_launch_info(int tile, int head_dim, int bm_words) {
    if (tile == 128 && head_dim == 128) return info_t<128, 128>(bm_words);
    if (tile == 128 && head_dim == 64) return info_t<128, 64>(bm_words);
    if (tile == 64 && head_dim == 128) return info_t<64, 128>(bm_words);
    return info_t<64, 64>(bm_words);
}

cudaError_t attn_prepare(int tile, int head_dim, int) {
    if (tile == 128 && head_dim == 128) return prepare_t<128, 128>();
    if (tile == 128 && head_dim == 64) return prepare_t<128, 64>();
    if (tile == 64 && head_dim == 128) return prepare_t<64, 128>();
    return prepare_t<64, 64>();
}

cudaError_t launch_attn(int tile, int head_dim, const CUtensorMap &q, const CUtensorMap &k,
                        const CUtensorMap &v, const AttnParams &p, int grid, cudaStream_t stream) {
    if (tile == 128 && head_dim == 128) return launch_t<128, 128>(q, k, v, p, grid, stream);
    if (tile == 128 && head_dim == 64) return launch_t<128, 64>(q, k, v, p, grid, stream);
    if (tile == 64 && head_dim == 128) return launch_t<64, 128>(q, k, v, p, grid, stream);
    return launch_t<64, 64>(q, k, v, p, grid, stream);
}

}  // namespace vsa
