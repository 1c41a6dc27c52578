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
//     tile that both units select is fetched once ("gathered" fetch).  The
//     ring is as deep as shared memory allows.
//   * S_u = Q_u K_j^T (tcgen05, smem x smem -> TMEM) for the key tiles unit u
//     selects, and O_u += P_u V_j with P read from TMEM, are issued in one of
//     two forms (a template parameter; the host picks it from the selection
//     width).  One thread issues back-to-back MMAs at the pipe's rate
//     (measured: 64 cycles an M128 N128 K16 MMA; an M128 N64 K16 S product
//     takes 48, the time its 6 KB of shared-memory operands take at 128 bytes
//     a clock); the issue layouts differ in which waits sit between the MMAs
//     of one thread:
//       - dense form (rows that can hold every key tile): with 128-token
//         tiles one thread per unit issues both of its products, the next S
//         before the current P V, which keeps P V out of the way of the S
//         hand-off between the units ("paired" issue); with 64-token tiles a
//         ring entry holds a pair of key tiles, so S is 128 keys wide;
//       - sparse form (where a key tile mostly serves one unit): one thread
//         issues every S, and one thread per unit its P V as soon as P is
//         stored, so S and P V issue overlap ("split" issue), one key tile per
//         ring entry.
//   * TMEM holds O of both units, the S buffer (one per unit where it fits,
//     else ONE the units take turns on; a shared-memory counter tells an
//     issuer when every earlier S has been copied out), and P of each unit as
//     bf16 pairs.
//   * Eight softmax warps per unit, two threads per query row in the same
//     warp (the .16x32bx2 TMEM shape: thread t holds row t%16 of the warp's
//     16 lanes and one half of its columns).  The row maximum and the final
//     row sum combine the halves with one shuffle.  Online softmax with exp2;
//     O is rescaled only when the running maximum grows by more than 2^8
//     (lazy rescale); l accumulates the bf16-rounded P that P V uses; the
//     epilogue writes O / l and the natural-log LSE.
//   * Masks are applied only on tail key tiles (valid count < tile).  For a
//     tail tile P V runs only over the 16-key blocks that hold valid keys, and
//     one control warp zeroes the few padding rows inside the last block in
//     shared memory first, so NaN/Inf padding in V never meets a zero weight
//     (0 * NaN = NaN).
//   * With 64-token tiles a unit is two query tiles in one 128-lane
//     accumulator; a P V with a key tile only one of them selects disables
//     the other's 64 output lanes, so each tile's O holds its own key tiles
//     only (O is zeroed at the start of an item and every P V accumulates).
//     In the dense form each thread half of a row holds one key tile of the
//     entry's pair, masked whole when its query tile does not select it.
//   * The producer counts the (query tile, key tile) steps it hands out,
//     tail and full, into a device word the host reads for route checks.
//   * 20 warps: four softmax warpgroups, then a control warpgroup (three
//     MMA-issuing warps, one of which zeroes tail V rows, and the TMA
//     producer) that hands registers to the softmax warpgroups with
//     setmaxnreg.
//   * Every wait is bounded (about 2 s); on expiry the CTA sets the timeout
//     flag, drains its outstanding copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>

#include "vsa_internal.h"
#include "vsa_ptx.cuh"
#include "vsa_wait.cuh"

namespace vsa {
namespace {

using namespace ptx;

constexpr int kSoftmaxWarps = 16;
constexpr int kUnitWarps = 8;      // softmax warps per unit; each adds 1 to the S counter per S
// Control warps (roles per layout, see the kernel):
//   paired: 16 + u issues every MMA of unit u; 19 zeroes tail V rows.
//   split:  16 issues every S; 17 issues P V of unit 0 and zeroes tail V rows;
//           19 issues P V of unit 1.
constexpr int kSWarp = 16;         // also allocates TMEM
constexpr int kPvWarp0 = 17;
constexpr int kProducerWarp = 18;
constexpr int kPvWarp1 = 19;
constexpr int kIssuers = 3;        // split layout: a ring fill is released by three arrivals
constexpr int kPairedIssuers = 2;  // paired layout: by two, and the tail-V zeroing warp
constexpr int kMaxStages = 8;
// Register split (control warpgroup, four softmax warpgroups); the sum stays
// within the 640 x 96 registers the CTA is launched with.
template <int T> struct RegSplit {
    static constexpr uint32_t kControl = 64;
    static constexpr uint32_t kSoftmax = 104;
    static_assert(128 * kControl + 512 * kSoftmax <= kAttnThreads * 96, "register split");
};
constexpr uint32_t kSmemLimit = 232448;  // 227 KB opt-in per CTA
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

// Key rows of one ring entry: a tile, or for the dense form at 64-token tiles
// a pair of tiles.
template <int T, bool kDense>
__host__ __device__ constexpr int key_rows() {
    return (T == 64 && kDense) ? 128 : T;
}

template <int T, int D, int KEYROWS>
struct Cfg {
    static_assert(T == 64 || T == 128, "tile");
    static_assert(KEYROWS == T || (T == 64 && KEYROWS == 128), "key rows per ring entry");
    static_assert(D == 64 || D == 128, "head_dim");
    static constexpr int kChunks = D / 64;                    // 128-byte column chunks per row
    static constexpr uint32_t kQChunk = kUnitRows * 128;      // bytes of one Q column chunk
    static constexpr uint32_t kQBytes = kUnitRows * D * 2;    // one unit's Q
    // A ring entry holds KT key rows: one tile, or (the dense form at 64-token
    // tiles) the pair of tiles (2m, 2m+1), which sit back to back in the
    // tile-major layout.  S of a pair entry is N = 128 wide, which runs at the
    // tensor pipe's rate; an N = 64 S product is bound by its 6 KB of
    // shared-memory operands (48 cycles against 32 of math).  Pairs stream a
    // key tile no query tile selects whenever its partner is selected, so
    // they are taken only for dense selections.
    static constexpr int KT = KEYROWS;
    static constexpr uint32_t kKVChunk = KT * 128;            // bytes of one K/V column chunk
    static constexpr uint32_t kStageBytes = KT * D * 2;       // one entry's K or V
    // TMEM columns: O of each unit (fp32), S (fp32) and P of each unit (bf16
    // pairs).  With 128-token tiles the units take turns on one S buffer (a
    // second does not fit next to two O and two P); with 64-token tiles each
    // unit has its own, so one unit's S never waits for the other's to be
    // copied out.
    // one S buffer per unit whenever two O, two S and two P fit in TMEM
    static constexpr int kSBufs = (2 * D + 3 * KT <= 512) ? 2 : 1;
    static constexpr uint32_t kTmemO0 = 0, kTmemO1 = D, kTmemS0 = 2 * D, kTmemS1 = 2 * D + (kSBufs - 1) * KT,
                              kTmemP0 = 2 * D + kSBufs * KT, kTmemP1 = 2 * D + kSBufs * KT + KT / 2;
    static constexpr uint32_t kTmemCols = (2 * D + (kSBufs + 1) * KT <= 256) ? 256 : 512;
    static_assert(2 * D + (kSBufs + 1) * KT <= 512, "TMEM plan");
    static constexpr uint32_t kIdescQK = idesc_bf16(128, KT, false);
    static constexpr uint32_t kIdescPV = idesc_bf16(128, D, true);
};

// Barrier indices for a ring of NS stages.
struct Bars {
    int NS;
    __host__ __device__ int kv_full(int s) const { return s; }
    __host__ __device__ int kv_empty(int s) const { return NS + s; }
    __host__ __device__ int vz(int s) const { return 2 * NS + s; }  // tail V rows zeroed
    __host__ __device__ int q_full(int u) const { return 3 * NS + u; }
    __host__ __device__ int q_empty(int u) const { return 3 * NS + 2 + u; }
    __host__ __device__ int s_full(int u) const { return 3 * NS + 4 + u; }
    __host__ __device__ int p_full(int u) const { return 3 * NS + 6 + u; }
    __host__ __device__ int o_done(int u) const { return 3 * NS + 8 + u; }
    __host__ __device__ int bm_full(int p) const { return 3 * NS + 10 + p; }
    __host__ __device__ int bm_empty(int p) const { return 3 * NS + 12 + p; }
    __host__ __device__ int done(int i) const { return 3 * NS + 14 + i; }  // one per issuer
    __host__ __device__ int count() const { return 3 * NS + 14 + kIssuers; }
};

struct SmemPlan {
    uint32_t q, ring, bm, hdr, bars, tslot, flag, sfree, sprog, total;
};

template <int T, int D, int KT>
__host__ __device__ inline SmemPlan smem_plan(int bm_words, int NS) {
    using C = Cfg<T, D, KT>;
    SmemPlan s;
    s.q = 0;
    s.ring = 2 * C::kQBytes;
    s.bm = s.ring + (uint32_t)NS * C::kStageBytes;
    s.hdr = s.bm + 2u * (uint32_t)kItemBitmaps * 4u * (uint32_t)bm_words;
    s.bars = s.hdr + 32;
    s.tslot = s.bars + 8u * (uint32_t)Bars{NS}.count();
    s.flag = s.tslot + 4;
    s.sfree = s.flag + 4;
    s.sprog = s.sfree + 8;  // one S-release counter per S buffer
    s.total = ((s.sprog + 4 + 15) & ~15u) + 1024;  // + slack to align the base to 1024
    return s;
}

template <int T, int D, int KT>
inline int stages_for(int bm_words) {
    int ns = kMaxStages;
    while (ns > 2 && smem_plan<T, D, KT>(bm_words, ns).total > kSmemLimit) --ns;
    return ns;
}

// Ring position: stage index and the parity of its current fill.
struct Ring {
    uint32_t st = 0, ph = 0;
    __device__ __forceinline__ void next(uint32_t ns) {
        if (++st == ns) {
            st = 0;
            ph ^= 1u;
        }
    }
};

// Bounded wait until a monotonic shared-memory counter reaches `target`.  A
// counter, not an mbarrier: the waiter may be any number of S tiles ahead of
// the last release, which an mbarrier's phase parity cannot tell apart.
__device__ __forceinline__ bool wait_count(uint32_t addr, uint32_t target, volatile int *abort_flag,
                                           int32_t *status) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        // tight polling: the S hand-off is on the critical path (measured
        // 2.17 vs 2.22 ms dense against a 32 ns sleep between polls)
        if ((int32_t)(ld_acquire(addr) - target) >= 0) return true;
        if ((it & 63u) == 63u) {
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

// Ring entries of a 32-tile bitmap word x (the union of an item's slots): bit
// b marks an entry whose key rows start at kernel tile 32w + b.  When an entry
// is a pair of 64-token tiles (2m, 2m+1) it is marked at the even bit.
template <int T, int KT>
__device__ __forceinline__ uint32_t entry_bits(uint32_t x) {
    if (KT == T) return x;
    return (x | (x >> 1)) & 0x55555555u;
}

// Tile index held by bitmap slot s (unit = s/2, half = s%2) of item g.
template <int T>
__device__ __forceinline__ int tile_of_slot(int g, int s) {
    if (T == 128) return (s & 1) ? -1 : 2 * g + (s >> 1);
    return 4 * g + s;
}

// Valid tokens of kernel tile jj.  With 256-token tiles (sub == 2) the kernel
// works on 128-token halves: half jj of caller tile jj/2 holds the tile's
// tokens from 128*(jj%2) on.
__device__ __forceinline__ int tile_size(const int32_t *block_sizes, int jj, int sub) {
    if (sub == 1) return __ldg(block_sizes + jj);
    const int n = __ldg(block_sizes + (jj >> 1)) - 128 * (jj & 1);
    return n < 0 ? 0 : (n > 128 ? 128 : n);
}

// kPaired selects the dense form: with 128-token tiles the paired MMA-issue
// layout, with 64-token tiles ring entries of key-tile pairs (issued in the
// split layout).
template <int T, int D, bool kPaired, bool kGB>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams P) {
    using C = Cfg<T, D, key_rows<T, kPaired>()>;
    constexpr bool kIssuePaired = kPaired && T == 128;  // the paired MMA-issue layout
    const int NS = P.stages;
    const Bars BI{NS};
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const int W = P.bm_words;
    // the selection bitmaps: in shared memory, or (kGB: beyond
    // kSmemBitmapTiles kernel tiles) in this CTA's region of the workspace;
    // a compile-time choice, so the shared-memory form reads them with
    // shared-memory loads
    const SmemPlan L = smem_plan<T, D, C::KT>(kGB ? 0 : W, NS);
    const uint32_t sQ = base + L.q;
    // Count of S tiles the softmax warps have copied out of an S buffer (each
    // of the eight warps of a unit adds 1 per S): one shared count, or one per
    // unit when each unit has its own buffer (sFree + 4u).
    const uint32_t sFree = base + L.sfree;
    // Count of ring fills the S issuer has seen land.  The S issuer waits for
    // every fill in order; the P V issuers wait for V fills only, and a parity
    // wait on a stage refers to the fill meant only once the stage's previous
    // fill has landed, which this count tells them.
    const uint32_t sProg = base + L.sprog;
    const uint32_t sRing = base + L.ring;
    uint32_t *bm = kGB ? P.bm_global + (size_t)blockIdx.x * 2 * kItemBitmaps * W
                       : reinterpret_cast<uint32_t *>(gbase + L.bm);  // [2][kItemBitmaps][W]
    volatile int32_t *hdr = reinterpret_cast<int32_t *>(gbase + L.hdr);  // [2][4]
    const uint32_t bars = base + L.bars;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(gbase + L.tslot);
    volatile int *abort_flag = reinterpret_cast<int *>(gbase + L.flag);
    auto BAR = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(BAR(BI.kv_full(s)), 1);
            // releases per fill: paired, both issuers and the warp that zeroes
            // tail V rows; split, three by the issuers
            mbar_init(BAR(BI.kv_empty(s)), kIssuePaired ? kPairedIssuers + 1 : kIssuers);
            mbar_init(BAR(BI.vz(s)), 32);
        }
        #pragma unroll
        for (int u = 0; u < 2; ++u) {
            mbar_init(BAR(BI.q_full(u)), 1);
            mbar_init(BAR(BI.q_empty(u)), 1);
            mbar_init(BAR(BI.s_full(u)), 1);
            mbar_init(BAR(BI.p_full(u)), 32 * kUnitWarps);
            mbar_init(BAR(BI.o_done(u)), 1);
            mbar_init(BAR(BI.bm_full(u)), 32);
            // lane 0 of two issuing warps, all lanes of the warp that zeroes
            // tail V rows, the softmax warps (either layout)
            mbar_init(BAR(BI.bm_empty(u)), 2 + 32 + 32 * kSoftmaxWarps);
        }
        for (int i = 0; i < kIssuers; ++i) mbar_init(BAR(BI.done(i)), 1);
        *abort_flag = 0;
        reinterpret_cast<volatile uint32_t *>(gbase + L.sfree)[0] = 0u;
        reinterpret_cast<volatile uint32_t *>(gbase + L.sfree)[1] = 0u;
        *reinterpret_cast<volatile uint32_t *>(gbase + L.sprog) = 0u;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == kSWarp) {
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

    // Registers: launched at 96 per thread (640 threads); the control
    // warpgroup (MMA issuers, producer, tail V zeroing) drops to
    // RegSplit::kControl and the four softmax warpgroups rise to
    // RegSplit::kSoftmax.  Each re-split sits inside its own role branch so no
    // code of one role runs under the other's limit.
    if (warp >= kSoftmaxWarps) {
      regs_dec<RegSplit<T>::kControl>();
      // Role layout of the MMA issue (a template parameter; the host picks
      // it from the tile size, head dim and selection width):
      //   paired (dense selections: most key tiles serve both units): lane 0
      //     of warp 16 + u issues every MMA of unit u, S_u of the next key
      //     tile before O_u += P_u V of the current one; warp 19 zeroes tail
      //     V rows.  The S hand-off between the units through the shared S
      //     buffer is then the critical chain, and a P V queued behind the
      //     next S keeps out of its way.
      //   split (sparse selections, where a key tile mostly serves one unit):
      //     lane 0 of warp 16 issues every S; warp 17 + 2u issues O_u += P_u V
      //     as soon as P_u is stored; warp 17 zeroes tail V rows.  The S
      //     stream and the P V streams wait on different barriers, so with
      //     separate issuing threads neither waits behind the other.
      constexpr bool paired = kIssuePaired;
      if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        const uint64_t pol_kv = l2_policy_evict_last();
        const uint64_t pol_q = l2_policy_evict_first();
        Ring ring;
        uint32_t fills = 0;
        uint32_t q_loads = 0;
        for (uint32_t it = 0;; ++it) {
            const int p = it & 1;
            if (!wait_warp(BAR(BI.bm_empty(p)), ((it >> 1) & 1u) ^ 1u, abort_flag, P.status)) break;
            int slot = 0;
            if (lane == 0) slot = atomicAdd(P.work_counter, 1);
            slot = __shfl_sync(0xffffffffu, slot, 0);
            // order entries: work item << 5 | key part << 2 | which units run
            // (0 both, 1 or 2 one)
            const int entry = (slot < P.n_items) ? __ldg(P.order + slot) : -1;
            const int item = entry < 0 ? -1 : entry >> kEntryItemShift, mode = entry < 0 ? 0 : entry & 3;
            // a part of a split tail unit takes the key tiles [k_lo, k_hi) only
            // (even bounds: a 64-token key-tile pair stays in one part; the
            // host cuts units of 128-token kernel tiles only)
            int piece = -1, k_lo = 0, k_hi = NT;
            if (T == 128 && entry >= 0 && mode != 0 && P.n_parts > 1) {
                const int part = (entry >> 2) & 7;
                piece = slot - P.tail_start;
                k_lo = (part * NT / P.n_parts) & ~1;
                k_hi = (part + 1 == P.n_parts) ? NT : ((part + 1) * NT / P.n_parts) & ~1;
            }
            uint32_t *bmp = bm + p * kItemBitmaps * W;
            int bad = 0;
            uint32_t n_tail = 0, n_full = 0;  // this lane's (query tile, key tile) steps
            if (item >= 0) {
                for (int i = lane; i < kItemBitmaps * W; i += 32) bmp[i] = 0u;
                __syncwarp();
                const int bh = item / P.G, g = item - (item / P.G) * P.G;
                // selections are per caller tile: with 256-token tiles both units
                // (the two halves of tile g) share row g, and a selected tile j
                // stands for its two halves 2j and 2j+1
                const int sub = P.sub, NTc = NT / sub;
                for (int s = 0; s < 4; ++s) {
                    const int t = tile_of_slot<T>(g, s);
                    if (t < 0 || t >= NT) continue;
                    if (mode != 0 && mode != (s >> 1) + 1) continue;  // unit s/2 runs elsewhere
                    const int64_t row = (int64_t)bh * NTc + t / sub;
                    int K = __ldg(P.q2k_num + row);
                    if (K < 0 || K > P.max_kv) {
                        bad = 1;
                        K = K < 0 ? 0 : P.max_kv;
                    }
                    const int32_t *sel = P.q2k_idx + row * P.max_kv;
                    for (int i = lane; i < K; i += 32) {
                        const int j = __ldg(sel + i);
                        if (j < 0 || j >= NTc) {
                            bad = 1;
                            continue;
                        }
                        for (int h2 = 0; h2 < sub; ++h2) {
                            const int jj = j * sub + h2;
                            if (T == 128 && (jj < k_lo || jj >= k_hi)) continue;  // another part's key tile
                            const int nj = tile_size(P.block_sizes, jj, sub);
                            if (nj <= 0) continue;
                            const uint32_t bit = 1u << (jj & 31);
                            const uint32_t old = atomicOr(&bmp[s * W + (jj >> 5)], bit);
                            if (old & bit) {
                                bad = 1;  // repeated index
                            } else if (nj < T) {
                                ++n_tail;  // the softmax masks this step's columns past nj
                                atomicOr(&bmp[4 * W + (jj >> 5)], bit);  // partial tile
                            } else {
                                ++n_full;
                            }
                        }
                    }
                }
                if (lane == 0) {
                    hdr[p * 4] = item;
                    hdr[p * 4 + 1] = mode;
                    hdr[p * 4 + 2] = piece;
                }
            } else if (lane == 0) {
                hdr[p * 4] = -1;
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(P.status, kFlagIndex);
            n_tail = __reduce_add_sync(0xffffffffu, n_tail);
            n_full = __reduce_add_sync(0xffffffffu, n_full);
            if (lane == 0 && (n_tail | n_full)) {
                atomicAdd(P.steps, (unsigned long long)n_tail);
                atomicAdd(P.steps + 1, (unsigned long long)n_full);
            }
            __syncwarp();
            mbar_arrive(BAR(BI.bm_full(p)));
            if (item < 0) break;

            const int bh = item / P.G, g = item - (item / P.G) * P.G;
            const int64_t row0 = (int64_t)bh * Sp + (int64_t)g * kItemRows;
            bool ok = true;
            #pragma unroll
            for (int u = 0; u < 2 && ok; ++u) {
                ok = wait_warp(BAR(BI.q_empty(u)), (it & 1u) ^ 1u, abort_flag, P.status);
                if (ok && lane == 0) {
                    mbar_arrive_expect_tx(BAR(BI.q_full(u)), C::kQBytes);
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_2d(sQ + u * C::kQBytes + c * C::kQChunk, &tm_q, c * 64,
                                    (int32_t)(row0 + u * kUnitRows), BAR(BI.q_full(u)), pol_q);
                }
            }
            if (!ok) break;
            ++q_loads;
            for (int w = 0; w < W && ok; ++w) {
                uint32_t bits = entry_bits<T, C::KT>(bmp[w] | bmp[W + w] | bmp[2 * W + w] | bmp[3 * W + w]);
                while (bits && ok) {
                    const int j = w * 32 + __ffs(bits) - 1;  // first kernel tile of the entry
                    bits &= bits - 1;
                    // KT rows from tile j on (for a pair of 64-token tiles j and
                    // j + 1; past the last tile the box reads rows no product uses)
                    const int32_t krow = (int32_t)((int64_t)bh * Sp + (int64_t)j * T);
                    for (int kv = 0; kv < 2; ++kv) {
                        const uint32_t st = ring.st;
                        ok = wait_warp(BAR(BI.kv_empty(st)), ring.ph ^ 1u, abort_flag, P.status);
                        if (!ok) break;
                        if (lane == 0) {
                            mbar_arrive_expect_tx(BAR(BI.kv_full(st)), C::kStageBytes);
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_2d(sRing + st * C::kStageBytes + c * C::kKVChunk,
                                            kv ? (const void *)&tm_v : (const void *)&tm_k, c * 64, krow,
                                            BAR(BI.kv_full(st)), pol_kv);
                        }
                        __syncwarp();
                        ring.next(NS);
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
            for (uint32_t f = first; f < fills; ++f)
                drain_wait(BAR(BI.kv_full(f % NS)), (f / NS) & 1u);
            if (q_loads > 0)
                #pragma unroll
                for (int u = 0; u < 2; ++u) drain_wait(BAR(BI.q_full(u)), (q_loads - 1) & 1u);
        }
        __syncwarp();
      } else if (paired && warp == kPvWarp1) {  // (paired is a compile-time constant)
        // ============================================ paired layout
        // ------------------------------------------------------------ tail V zeroing (paired layout)
        // For a tail key tile (valid count not a multiple of 16) P V reads the
        // last 16-key block, whose padding rows may hold NaN/Inf: zero them
        // (rows of 128 bytes; the swizzle permutes 16-byte chunks within a row
        // only) once the tile has landed, then release the MMA issuers.
        Ring ring;
        for (uint32_t it = 0;; ++it) {
            const int p = it & 1;
            if (!wait_warp(BAR(BI.bm_full(p)), (it >> 1) & 1u, abort_flag, P.status)) break;
            if (hdr[p * 4] < 0) break;
            const uint32_t *bmp = bm + p * kItemBitmaps * W;
            bool ok = true;
            for (int w = 0; w < W && ok; ++w) {
                uint32_t bits = bmp[w] | bmp[W + w] | bmp[2 * W + w] | bmp[3 * W + w];
                const uint32_t part_w = bmp[4 * W + w];  // partial tiles
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    const int j = w * 32 + b;
                    bits &= bits - 1;
                    const uint32_t kst = ring.st, kph = ring.ph;
                    ring.next(NS);
                    const uint32_t vst = ring.st, vph = ring.ph;
                    ring.next(NS);
                    // Wait for every fill in order and give each its third
                    // release, so no stage is refilled before this warp has seen
                    // its current fill: every parity wait here refers to the fill
                    // meant.
                    if (!(ok = wait_warp(BAR(BI.kv_full(kst)), kph, abort_flag, P.status))) break;
                    if (lane == 0) mbar_arrive(BAR(BI.kv_empty(kst)));
                    if (!(ok = wait_warp(BAR(BI.kv_full(vst)), vph, abort_flag, P.status))) break;
                    const int nj = ((part_w >> b) & 1u) ? tile_size(P.block_sizes, j, P.sub) : T;
                    if ((nj & 15) != 0) {
                        uint4 *vs = reinterpret_cast<uint4 *>(gbase + L.ring + vst * C::kStageBytes);
                        const int n16 = (16 - (nj & 15)) * 8;
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c)
                            for (int i = lane; i < n16; i += 32)
                                vs[(c * C::kKVChunk + nj * 128) / 16 + i] = make_uint4(0u, 0u, 0u, 0u);
                        fence_proxy_async_smem();
                        __syncwarp();
                        mbar_arrive(BAR(BI.vz(vst)));
                    }
                    if (lane == 0) mbar_arrive(BAR(BI.kv_empty(vst)));
                }
            }
            if (!ok) break;
            __syncwarp();
            mbar_arrive(BAR(BI.bm_empty(p)));
        }
      } else if (paired) {
        // ------------------------------------------------------------ MMA issuers (paired layout)
        // Lane 0 of warp 16 + u issues every MMA of unit u: S_u = Q_u
        // K_j^T and O_u += P_u V_j.  tcgen05.mma issue runs only ~2
        // instructions ahead of execution and each barrier wait costs the
        // issuing thread ~100 cycles, so (a) two issuers let one unit's waits
        // overlap the other's issue, and (b) all waits of an entry come before
        // its MMAs, leaving nothing between a unit's P V and its next S.
        if (lane == 0) {
            const int u = warp - kSWarp;  // warps 16 and 17
            Ring ring;
            uint32_t pcnt = 0;    // P V issued (= p_full phases consumed)
            uint32_t gcnt = 0;    // S tiles of both units before this entry (union order, unit 0 first)
            uint32_t s_own = 0;   // S tiles of this unit issued so far
            uint32_t vz_par = 0;  // per stage: parity of its next tail-zeroing phase
            const uint64_t dq = sdesc_sw128(sQ + u * C::kQBytes, 16, 1024);  // Q_u, K-major
            const uint64_t dk = sdesc_sw128(sRing, 16, 1024);                // stage 0 as K-major B
            const uint64_t dv = sdesc_sw128(sRing, C::kKVChunk, 1024);       // stage 0 as MN-major B
            constexpr uint32_t kStage16 = C::kStageBytes >> 4;
            const uint32_t tS = tmem + (u ? C::kTmemS1 : C::kTmemS0);
            const uint32_t tP = tmem + (u ? C::kTmemP1 : C::kTmemP0);
            const uint32_t tO = tmem + (u ? C::kTmemO1 : C::kTmemO0);
            bool ok = true;
            for (uint32_t it = 0; ok; ++it) {
                const int p = it & 1;
                if (!(ok = wait_bar(BAR(BI.bm_full(p)), (it >> 1) & 1u, abort_flag, P.status))) break;
                if (hdr[p * 4] < 0) break;
                const uint32_t *bmp = bm + p * kItemBitmaps * W;
                const uint32_t *pa = bmp + (2 * u) * W, *pb = pa + W;
                // member entries of this unit, so Q can be released right after its last S
                uint32_t n_mine = 0;
                for (int w = 0; w < W; ++w) n_mine += __popc(pa[w] | pb[w]);
                if (!(ok = wait_bar(BAR(BI.q_full(u)), it & 1u, abort_flag, P.status))) break;
                tc_fence_after();
                bool pending = false, first = true;
                uint32_t pend_v = 0, pend_ph = 0;
                int pend_kb = 0;
                bool pend_tail = false;
                uint32_t seen = 0;

                // O_u += P_u V of the pending entry (P from TMEM), then this
                // issuer's release of that V stage.  (This issue layout runs
                // with 128-token tiles only.)
                auto pv = [&]() -> bool {
                    if (!wait_bar(BAR(pend_tail ? BI.vz(pend_v) : BI.kv_full(pend_v)), pend_ph, abort_flag, P.status))
                        return false;
                    if (!wait_bar_spin(BAR(BI.p_full(u)), pcnt & 1u, abort_flag, P.status)) return false;
                    ++pcnt;
                    tc_fence_after();
                    const uint64_t b = dv + pend_v * kStage16;
                    mma_ts(tO, tP, b, C::kIdescPV, first ? 0u : 1u);
#pragma unroll
                    for (int kk = 1; kk < T / 16; ++kk)
                        if (kk < pend_kb) mma_ts(tO, tP + kk * 8, b + kk * 128, C::kIdescPV, 1u);
                    mma_commit(BAR(BI.o_done(u)));
                    mma_commit(BAR(BI.kv_empty(pend_v)));
                    first = false;
                    pending = false;
                    return true;
                };

                for (int w = 0; w < W && ok; ++w) {
                    const uint32_t mw = pa[w] | pb[w];
                    const uint32_t part_w = bmp[4 * W + w];  // partial tiles
                    uint32_t bits = bmp[w] | bmp[W + w] | bmp[2 * W + w] | bmp[3 * W + w];
                    while (bits && ok) {
                        const int b = __ffs(bits) - 1;
                        bits &= bits - 1;
                        const int j = w * 32 + b;
                        const uint32_t kst = ring.st, kph = ring.ph;
                        ring.next(NS);
                        const uint32_t vst = ring.st, vph = ring.ph;
                        ring.next(NS);
                        const int nj = ((part_w >> b) & 1u) ? tile_size(P.block_sizes, j, P.sub) : T;
                        const bool tail = (nj & 15) != 0;
                        const uint32_t vzp = (vz_par >> vst) & 1u;
                        if (tail) vz_par ^= 1u << vst;
                        const uint32_t m0 = ((bmp[w] | bmp[W + w]) >> b) & 1u;
                        const uint32_t m1 = ((bmp[2 * W + w] | bmp[3 * W + w]) >> b) & 1u;
                        const uint32_t g = gcnt + (u ? m0 : 0u);  // this S in the shared-buffer order
                        gcnt += m0 + m1;
                        if ((mw >> b) & 1u) {
                            // S first: it needs only K and the softmax having loaded
                            // the previous S; then the pending P V.
                            if (!(ok = wait_bar_spin(BAR(BI.kv_full(kst)), kph, abort_flag, P.status))) break;
                            // every earlier S tile has left the S buffer (shared: both
                            // units' S in union order; per unit: this unit's)
                            if (C::kSBufs == 2) {
                                if (!(ok = wait_count(sFree + 4u * u, (uint32_t)kUnitWarps * s_own, abort_flag,
                                                      P.status)))
                                    break;
                            } else if (!(ok = wait_count(sFree, (uint32_t)kUnitWarps * g, abort_flag, P.status))) {
                                break;
                            }
                            ++s_own;
                            tc_fence_after();
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tS, dq + (kk >> 2) * (C::kQChunk >> 4) + (kk & 3) * 2,
                                       dk + kst * kStage16 + (kk >> 2) * (C::kKVChunk >> 4) + (kk & 3) * 2,
                                       C::kIdescQK, kk > 0 ? 1u : 0u);
                            mma_commit(BAR(BI.s_full(u)));
                            if (++seen == n_mine) mma_commit(BAR(BI.q_empty(u)));
                            mma_commit(BAR(BI.kv_empty(kst)));
                            if (pending && !(ok = pv())) break;
                            pending = true;
                            pend_v = vst;
                            pend_ph = tail ? vzp : vph;
                            pend_kb = (nj + 15) >> 4;
                            pend_tail = tail;
                        } else {
                            // not selected by this unit: issue the pending P V (it
                            // frees a V stage), then release both stages of the entry
                            if (pending && !(ok = pv())) break;
                            if (!(ok = wait_bar(BAR(BI.kv_full(kst)), kph, abort_flag, P.status))) break;
                            mbar_arrive(BAR(BI.kv_empty(kst)));
                            if (!(ok = wait_bar(BAR(BI.kv_full(vst)), vph, abort_flag, P.status))) break;
                            mbar_arrive(BAR(BI.kv_empty(vst)));
                        }
                    }
                }
                if (ok && pending) ok = pv();
                if (!ok) break;
                if (n_mine == 0) mma_commit(BAR(BI.q_empty(u)));  // no S issued: release Q
                mbar_arrive(BAR(BI.bm_empty(p)));
            }
            // All MMAs of this issuer complete before TMEM is released.
            mma_commit(BAR(BI.done(u)));
            drain_wait(BAR(BI.done(u)), 0u);
        }
        __syncwarp();
      } else if (warp == kSWarp) {
        // ============================================ split layout
        // ------------------------------------------------------------ S issuer
        // Lane 0 issues S_u = Q_u K_j^T for both units, in the order the
        // units take the shared S buffer (union order, unit 0 first), each
        // once the softmax warps have copied every earlier S out.
        if (lane == 0) {
            Ring ring;
            uint32_t g = 0;  // S tiles issued so far (both units, all items)
            uint64_t dq[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) dq[u] = sdesc_sw128(sQ + u * C::kQBytes, 16, 1024);  // Q_u, K-major
            const uint64_t dk = sdesc_sw128(sRing, 16, 1024);                              // stage 0 as K-major B
            constexpr uint32_t kStage16 = C::kStageBytes >> 4;
            uint32_t s_unit[2] = {0u, 0u};  // S tiles issued so far per unit (per-unit buffers)
            bool ok = true;
            for (uint32_t it = 0; ok; ++it) {
                const int p = it & 1;
                if (!(ok = wait_bar(BAR(BI.bm_full(p)), (it >> 1) & 1u, abort_flag, P.status))) break;
                if (hdr[p * 4] < 0) break;
                const uint32_t *bmp = bm + p * kItemBitmaps * W;
                // member entries per unit, so Q_u is released right after its last S
                uint32_t n_mine[2] = {0u, 0u}, seen[2] = {0u, 0u};
                for (int w = 0; w < W; ++w) {
                    n_mine[0] += __popc(entry_bits<T, C::KT>(bmp[w] | bmp[W + w]));
                    n_mine[1] += __popc(entry_bits<T, C::KT>(bmp[2 * W + w] | bmp[3 * W + w]));
                }
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    if (ok) ok = wait_bar(BAR(BI.q_full(u)), it & 1u, abort_flag, P.status);
                if (!ok) break;
                tc_fence_after();
                for (int w = 0; w < W && ok; ++w) {
                    // entries each unit takes part in
                    const uint32_t m0w = entry_bits<T, C::KT>(bmp[w] | bmp[W + w]);
                    const uint32_t m1w = entry_bits<T, C::KT>(bmp[2 * W + w] | bmp[3 * W + w]);
                    uint32_t bits = m0w | m1w;
                    while (bits && ok) {
                        const int b = __ffs(bits) - 1;
                        bits &= bits - 1;
                        const uint32_t kst = ring.st, kph = ring.ph;
                        ring.next(NS);
                        const uint32_t vst = ring.st, vph = ring.ph;
                        ring.next(NS);
                        if (!(ok = wait_bar_spin(BAR(BI.kv_full(kst)), kph, abort_flag, P.status))) break;
                        red_add_release(sProg, 1u);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            if (!ok || !((((u ? m1w : m0w) >> b) & 1u))) continue;
                            // every earlier S tile has left the S buffer (shared: both
                            // units' S in union order; per unit: this unit's)
                            if (C::kSBufs == 2) {
                                if (!(ok = wait_count(sFree + 4u * u, (uint32_t)kUnitWarps * s_unit[u], abort_flag,
                                                      P.status)))
                                    break;
                            } else if (!(ok = wait_count(sFree, (uint32_t)kUnitWarps * g, abort_flag, P.status))) {
                                break;
                            }
                            ++s_unit[u];
                            tc_fence_after();
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk)
                                mma_ss(tmem + (u ? C::kTmemS1 : C::kTmemS0), dq[u] + (kk >> 2) * (C::kQChunk >> 4) + (kk & 3) * 2,
                                       dk + kst * kStage16 + (kk >> 2) * (C::kKVChunk >> 4) + (kk & 3) * 2,
                                       C::kIdescQK, kk > 0 ? 1u : 0u);
                            mma_commit(BAR(BI.s_full(u)));
                            if (++seen[u] == n_mine[u]) mma_commit(BAR(BI.q_empty(u)));
                            ++g;
                        }
                        if (!ok) break;
                        // K fills are released by this thread alone (the P V
                        // issuers never read them): two arrivals now, the
                        // third when the S MMAs that read K have completed.
                        mbar_arrive(BAR(BI.kv_empty(kst)));
                        mbar_arrive(BAR(BI.kv_empty(kst)));
                        mma_commit(BAR(BI.kv_empty(kst)));
                        // V of the tile is not read here; its fill is still
                        // waited for (and released: one of its three
                        // arrivals) in order, so every parity wait of this
                        // thread refers to the fill it means.
                        if (!(ok = wait_bar(BAR(BI.kv_full(vst)), vph, abort_flag, P.status))) break;
                        red_add_release(sProg, 1u);
                        mbar_arrive(BAR(BI.kv_empty(vst)));
                    }
                }
                if (!ok) break;
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    if (n_mine[u] == 0) mma_commit(BAR(BI.q_empty(u)));  // no S of this unit: release Q_u
                mbar_arrive(BAR(BI.bm_empty(p)));
            }
            // All MMAs of this issuer complete before TMEM is released.
            mma_commit(BAR(BI.done(0)));
            drain_wait(BAR(BI.done(0)), 0u);
        }
        __syncwarp();
      } else {
        // ------------------------------------------------------------ P V issuers
        // Warp kPvWarp0 + 2u issues O_u += P_u V_j (lane 0) as soon as the
        // softmax has stored P_u.  Warp kPvWarp0 also zeroes the padding rows
        // of a tail key tile's V inside its last 16-key block (rows of 128
        // bytes; the swizzle permutes 16-byte chunks within a row only) once
        // the tile has landed, so NaN/Inf padding never meets a zero weight;
        // warp kPvWarp1 waits for that before its P V.
        const int u = (warp == kPvWarp0) ? 0 : 1;
        const bool fixer = (u == 0);
        Ring ring;
        uint32_t fills = 0;   // ring fills walked so far (K and V of every tile)
        uint32_t pcnt = 0;    // P V issued (= p_full phases consumed)
        uint32_t vz_par = 0;  // per stage: parity of its next tail-zeroing phase
        const uint64_t dv = sdesc_sw128(sRing, C::kKVChunk, 1024);  // stage 0 as MN-major B
        constexpr uint32_t kStage16 = C::kStageBytes >> 4;
        const uint32_t tP = tmem + (u ? C::kTmemP1 : C::kTmemP0);
        const uint32_t tO = tmem + (u ? C::kTmemO1 : C::kTmemO0);
        bool ok = true;
        for (uint32_t it = 0; ok; ++it) {
            const int p = it & 1;
            if (!(ok = wait_warp(BAR(BI.bm_full(p)), (it >> 1) & 1u, abort_flag, P.status))) break;
            if (hdr[p * 4] < 0) break;
            const uint32_t *bmp = bm + p * kItemBitmaps * W;
            bool first = true;
            for (int w = 0; w < W && ok; ++w) {
                const uint32_t sa_w = bmp[(2 * u) * W + w], sb_w = bmp[(2 * u + 1) * W + w];  // this unit's tiles
                const uint32_t all_w = bmp[w] | bmp[W + w] | bmp[2 * W + w] | bmp[3 * W + w];
                const uint32_t mw = entry_bits<T, C::KT>(sa_w | sb_w);  // entries this unit takes part in
                const uint32_t part_w = bmp[4 * W + w];          // partial tiles
                uint32_t bits = entry_bits<T, C::KT>(all_w);
                while (bits && ok) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int j = w * 32 + b;
                    ring.next(NS);  // K fill of entry j: the S issuer waits for it and releases it
                    const uint32_t vst = ring.st, vph = ring.ph;
                    ring.next(NS);
                    const uint32_t vfill = fills + 1;  // index of this V fill
                    fills += 2;
                    // the S issuer has seen the stage's previous fill (index
                    // vfill - NS) land, so the parity wait below means this fill
                    if (vfill >= (uint32_t)NS &&
                        !(ok = __all_sync(0xffffffffu, wait_count(sProg, vfill - (uint32_t)NS + 1u, abort_flag,
                                                                  P.status))))
                        break;
                    if (!(ok = __all_sync(0xffffffffu, wait_bar_spin(BAR(BI.kv_full(vst)), vph, abort_flag, P.status))))
                        break;
                    // valid keys of each tile of the entry (64-token tiles: the
                    // pair j, j + 1, rows 64h on); a tail is a tile some product
                    // reads whose valid keys end inside a 16-key block
                    constexpr int kHalves = C::KT / T;
                    int nj[kHalves];
                    bool tail = false;
#pragma unroll
                    for (int h = 0; h < kHalves; ++h) {
                        nj[h] = ((part_w >> (b + h)) & 1u) ? tile_size(P.block_sizes, j + h, P.sub) : T;
                        if (((all_w >> (b + h)) & 1u) && (nj[h] & 15) != 0) tail = true;
                    }
                    const uint32_t vzp = (vz_par >> vst) & 1u;
                    if (tail) {
                        vz_par ^= 1u << vst;
                        if (fixer) {
                            uint4 *vs = reinterpret_cast<uint4 *>(gbase + L.ring + vst * C::kStageBytes);
#pragma unroll
                            for (int h = 0; h < kHalves; ++h) {
                                if (!((all_w >> (b + h)) & 1u) || (nj[h] & 15) == 0) continue;
                                const int r0 = h * T + nj[h];  // first padding row of the tile
                                const int n16 = (16 - (nj[h] & 15)) * 8;
#pragma unroll
                                for (int c = 0; c < C::kChunks; ++c)
                                    for (int i = lane; i < n16; i += 32)
                                        vs[(c * C::kKVChunk + r0 * 128) / 16 + i] = make_uint4(0u, 0u, 0u, 0u);
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            mbar_arrive(BAR(BI.vz(vst)));
                        } else if (!(ok = wait_warp(BAR(BI.vz(vst)), vzp, abort_flag, P.status))) {
                            break;
                        }
                    }
                    if ((mw >> b) & 1u) {
                        if (!(ok = __all_sync(0xffffffffu,
                                              wait_bar_spin(BAR(BI.p_full(u)), pcnt & 1u, abort_flag, P.status))))
                            break;
                        ++pcnt;
                        if (lane == 0) {
                            tc_fence_after();
                            const uint64_t bd = dv + vst * kStage16;
                            if constexpr (T == 64) {
                                // two 64-row query tiles share the accumulator and two
                                // 64-key tiles the entry: the 16-key blocks of key tile
                                // j + h go only to the query tiles that select it (the
                                // other's 64 output lanes disabled), and only up to its
                                // valid keys
#pragma unroll
                                for (int h = 0; h < kHalves; ++h) {
                                    const uint32_t lo = (sa_w >> (b + h)) & 1u, hi = (sb_w >> (b + h)) & 1u;
                                    if (!(lo | hi)) continue;
                                    const uint32_t off_lo = lo ? 0u : ~0u, off_hi = hi ? 0u : ~0u;
                                    const int kb = (nj[h] + 15) >> 4;  // 16-key blocks holding valid keys
#pragma unroll
                                    for (int kk = 0; kk < T / 16; ++kk)
                                        if (kk < kb)
                                            mma_ts_lanes(tO, tP + (h * (T / 16) + kk) * 8, bd + (h * (T / 16) + kk) * 128,
                                                         C::kIdescPV, 1u, off_lo, off_hi);
                                }
                            } else {
                                const int kb = (nj[0] + 15) >> 4;  // 16-key blocks holding valid keys
                                mma_ts(tO, tP, bd, C::kIdescPV, first ? 0u : 1u);
#pragma unroll
                                for (int kk = 1; kk < T / 16; ++kk)
                                    if (kk < kb) mma_ts(tO, tP + kk * 8, bd + kk * 128, C::kIdescPV, 1u);
                            }
                            mma_commit(BAR(BI.o_done(u)));
                            mma_commit(BAR(BI.kv_empty(vst)));
                        }
                        first = false;
                    } else if (lane == 0) {
                        mbar_arrive(BAR(BI.kv_empty(vst)));  // not selected by this unit
                    }
                    __syncwarp();
                }
            }
            if (!ok) break;
            __syncwarp();
            if (fixer || lane == 0) mbar_arrive(BAR(BI.bm_empty(p)));
        }
        // All MMAs of this issuer complete before TMEM is released.
        if (lane == 0) {
            mma_commit(BAR(BI.done(1 + u)));
            drain_wait(BAR(BI.done(1 + u)), 0u);
        }
        __syncwarp();
      }
    } else {
        regs_inc<RegSplit<T>::kSoftmax>();
        // ------------------------------------------------------------ softmax
        // Eight warps per unit, two threads per query row in the same warp.
        // Warp 8u + 4sb + q4 takes TMEM lanes (rows) 32q4 + 16sb .. +15 with
        // the .16x32bx2 shape: thread t holds row t%16 and the columns of half
        // t/16 (S: 64 columns, O: D/2 columns, P: 32 packed columns).  With
        // 64-token tiles a half is exactly one key tile of the entry's pair.
        // The row maximum and the final row sum combine the halves with one
        // shuffle.
        constexpr int TH = C::KT / 2;  // S columns per thread
        // 128-token tiles: P goes to registers before the wait for the unit's
        // previous P V, so the exponentials overlap that product.  (64-token
        // tiles measured slower that way.)
        constexpr bool kEarlyP = T == 128;
        constexpr int DH = D / 2;   // O columns per thread
        const int u = warp >> 3;
        const int sb = (warp >> 2) & 1;
        const int q4 = warp & 3;
        const int hf = lane >> 4;                        // column half
        const int rb0 = q4 * 32 + sb * 16;               // first row of this warp's block
        const int row = rb0 + (lane & 15);               // query row within the unit
        const int tsub = (T == 64) ? (q4 >> 1) : 0;      // which 64-row tile of the unit (T == 64)
        const uint32_t tl = (uint32_t)rb0 << 16;
        const uint32_t tS = tmem + tl + (u ? C::kTmemS1 : C::kTmemS0);
        const uint32_t sFreeU = sFree + (C::kSBufs == 2 ? 4u * u : 0u);  // the count this unit adds to
        const uint32_t tP = tmem + tl + (u ? C::kTmemP1 : C::kTmemP0);
        const uint32_t tO = tmem + tl + (u ? C::kTmemO1 : C::kTmemO0);
        const float c = P.scale_log2;
        uint32_t cnt = 0;  // member entries of this unit seen so far (all items)
        for (uint32_t it = 0;; ++it) {
            const int p = it & 1;
            if (!wait_warp(BAR(BI.bm_full(p)), (it >> 1) & 1u, abort_flag, P.status)) break;
            const int item = hdr[p * 4];
            const int mode = hdr[p * 4 + 1];
            const int piece = (T == 128) ? hdr[p * 4 + 2] : -1;  // >= 0: one key range of a split tail unit
            if (item < 0) break;
            const uint32_t *bmp = bm + p * kItemBitmaps * W;
            const int bh = item / P.G, g = item - (item / P.G) * P.G;
            const int t = (T == 128) ? 2 * g + u : 4 * g + 2 * u + tsub;
            const int r = (T == 128) ? row : (row & 63);
            const int n_t = (t < NT) ? tile_size(P.block_sizes, t, P.sub) : 0;
            float m = -INFINITY, l0 = 0.f, l1 = 0.f;  // l: this thread's columns
            uint32_t n_mine = 0;
            bool ok = true;
            const uint32_t *pa = bmp + (2 * u) * W, *pb = bmp + (2 * u + 1) * W;
            const uint32_t *pm = tsub ? pb : pa;
            if constexpr (T == 64) {
                // Every P V accumulates (the rows of a tile that does not select
                // a key tile are masked out of its product, so no single MMA
                // may start O afresh): O starts at zero.  The stores complete
                // before this unit's first P is released (tmem_wait_st), and the
                // last item's P V finished before its epilogue read O.
                const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ch = 0; ch < DH / 8; ++ch) tmem_st2x_8f<DH>(tO + ch * 8, z);
            }
            for (int w = 0; w < W && ok; ++w) {
                uint32_t bits = entry_bits<T, C::KT>(pa[w] | pb[w]);
                const uint32_t mine = pm[w];
                const uint32_t part_w = bmp[4 * W + w];  // partial tiles
                while (bits) {
                    const int b = __ffs(bits) - 1;
                    bits &= bits - 1;
                    const int j = w * 32 + b;
                    // This thread's key tile (j, or j + hf of a 64-token pair) and
                    // its valid keys, loaded before the wait for S: in the split
                    // layout only for partial tiles; the paired form loads every
                    // tile's count (the load hides under the wait, and this form
                    // measured 2 % faster on dense selections than the bitmap test)
                    const int jt = (C::KT == T) ? j : j + hf;
                    const int nj =
                        (kIssuePaired || ((part_w >> (jt & 31)) & 1u)) ? tile_size(P.block_sizes, jt, P.sub) : T;
                    if (!(ok = wait_warp(BAR(BI.s_full(u)), cnt & 1u, abort_flag, P.status))) break;
                    tc_fence_after();
                    // warp-uniform: does this warp's query tile take part in the
                    // entry?  With 128-token tiles every entry of the unit is its
                    // own, stated at compile time (which also keeps the early P
                    // free of spills).
                    const bool member_row = (T == 128) || ((entry_bits<T, C::KT>(mine) >> b) & 1u) != 0u;
                    // per thread with 64-token tiles: does it select this half's tile?
                    const bool member_t = (C::KT == T) || ((mine >> (jt & 31)) & 1u) != 0u;
                    float s[TH];
                    if (member_row) {
                        if constexpr (TH == 64) tmem_ld2x_64<TH>(tS, s);
                        else tmem_ld2x_32<TH>(tS, s);
                    }
                    // S is in registers: the shared S buffer may take the next S.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) red_add_release(sFreeU, 1u);
                    float m_new = m;
                    bool fresh = false, resc = false;
                    if (member_row) {
                        // columns past the valid keys (and, with 64-token tiles, a
                        // whole half whose tile this row does not select) are -inf
                        const int lim = !member_t ? 0 : (C::KT == T ? nj - hf * TH : nj);
                        if (lim < TH) {
#pragma unroll
                            for (int i = 0; i < TH; ++i)
                                if (i >= lim) s[i] = -INFINITY;
                        }
                        float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
                        for (int i = 0; i < TH; i += 8) {
                            a0 = max3(a0, s[i], s[i + 1]);
                            a1 = max3(a1, s[i + 2], s[i + 3]);
                            a2 = max3(a2, s[i + 4], s[i + 5]);
                            a3 = max3(a3, s[i + 6], s[i + 7]);
                        }
                        float mx = max3(a0, a1, fmaxf(a2, a3));
                        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                        m_new = fmaxf(m, mx * c);
                        fresh = (m == -INFINITY);
                        resc = !fresh && (m_new > m + kRescaleThreshold);
                    }
                    // this tile's part of l in 4 independent sums
                    float lq[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (kEarlyP) {
                        // O's rescale factor, from the old maximum
                        const bool any_resc = __any_sync(0xffffffffu, resc);
                        const float alpha = resc ? ex2(m - m_new) : 1.f;
                        if (fresh || resc) m = m_new;
                        const float neg_m = -m;
                        // P of this tile into registers while the previous P V of the
                        // unit may still run
                        uint32_t pk[TH / 2];
#pragma unroll
                        for (int i = 0; i < TH / 2; ++i) {
                            if (member_row) {
                                float x0, x1;
                                fma2_scalar(x0, x1, s[2 * i], s[2 * i + 1], c, neg_m);
                                pk[i] = pack_bf16x2(ex2(x0), ex2(x1));
                                // l sums the bf16 values P V actually uses, so the
                                // weights P / l stay exactly normalised.
                                add_bf16x2_f32(lq[2 * (i & 1)], lq[2 * (i & 1) + 1], pk[i]);
                            } else {
                                pk[i] = 0u;  // this tile of the unit does not select tile j: zero P rows
                            }
                        }
                        // The previous P V of this unit must be done before P is
                        // overwritten and O rescaled.
                        if (n_mine > 0) {
                            if (!(ok = wait_warp(BAR(BI.o_done(u)), (cnt - 1u) & 1u, abort_flag, P.status))) break;
                            tc_fence_after();
                        }
                        if (any_resc) {
#pragma unroll
                            for (int ch = 0; ch < DH / 8; ++ch) {
                                float o[8];
                                tmem_ld2x_8<DH>(tO + ch * 8, o);
#pragma unroll
                                for (int i = 0; i < 8; ++i) o[i] *= alpha;
                                tmem_st2x_8f<DH>(tO + ch * 8, o);
                            }
                            l0 *= alpha;
                            l1 *= alpha;
                        }
#pragma unroll
                        for (int cc = 0; cc < TH / 16; ++cc) {
                            uint32_t pc[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) pc[i] = pk[cc * 8 + i];
                            tmem_st2x_8<TH / 2>(tP + cc * 8, pc);
                        }
                    } else {
                        // The previous P V of this unit must be done: it reads the P
                        // columns about to be overwritten and accumulates into O.
                        if (n_mine > 0) {
                            if (!(ok = wait_warp(BAR(BI.o_done(u)), (cnt - 1u) & 1u, abort_flag, P.status))) break;
                            tc_fence_after();
                        }
                        if (__any_sync(0xffffffffu, resc)) {
                            const float alpha = resc ? ex2(m - m_new) : 1.f;
                            // 8 columns at a time: S is still held in registers here
#pragma unroll
                            for (int ch = 0; ch < DH / 8; ++ch) {
                                float o[8];
                                tmem_ld2x_8<DH>(tO + ch * 8, o);
#pragma unroll
                                for (int i = 0; i < 8; ++i) o[i] *= alpha;
                                tmem_st2x_8f<DH>(tO + ch * 8, o);
                            }
                            l0 *= alpha;
                            l1 *= alpha;
                        }
                        if (fresh || resc) m = m_new;
                        const float neg_m = -m;
#pragma unroll
                        for (int cc = 0; cc < TH / 16; ++cc) {
                            uint32_t pk[8];
                            if (member_row) {
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    float x0, x1;
                                    fma2_scalar(x0, x1, s[cc * 16 + 2 * i], s[cc * 16 + 2 * i + 1], c, neg_m);
                                    pk[i] = pack_bf16x2(ex2(x0), ex2(x1));
                                    // l sums the bf16 values P V actually uses, so the
                                    // weights P / l stay exactly normalised.
                                    add_bf16x2_f32(lq[2 * (i & 1)], lq[2 * (i & 1) + 1], pk[i]);
                                }
                            } else {
                                // this tile of the unit does not select tile j: zero P rows
#pragma unroll
                                for (int i = 0; i < 8; ++i) pk[i] = 0u;
                            }
                            tmem_st2x_8<TH / 2>(tP + cc * 8, pk);
                        }
                    }
                    l0 += lq[0] + lq[2];
                    l1 += lq[1] + lq[3];
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(BAR(BI.p_full(u)));
                    ++cnt;
                    ++n_mine;
                }
            }
            if (!ok) break;
            // -------------------------------------------------------- epilogue
            if (n_mine > 0) {
                if (!wait_warp(BAR(BI.o_done(u)), (cnt - 1u) & 1u, abort_flag, P.status)) break;
                tc_fence_after();
            }
            float l = l0 + l1;
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            // a unit that another CTA runs (a split item) leaves its rows alone;
            // one key range of a split tail unit (128-token tiles; the host cuts
            // no others) leaves unnormalised O, the row maximum and the row sum
            // in the workspace instead, for tail_merge_kernel
            const bool piece_row = T == 128 && piece >= 0 && mode == u + 1;
            const bool write_row = t < NT && (mode == 0 || mode == u + 1) && piece < 0;
            const bool valid = r < n_t;
            const bool use_o = (n_mine > 0) && valid && (l != 0.f);  // NaN l keeps use_o: NaN row
            const float inv = use_o ? 1.f / l : 0.f;
            const int64_t orow = (int64_t)bh * Sp + (int64_t)t * T + r;
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(P.out) + orow * D + hf * DH);
            float4 *po = reinterpret_cast<float4 *>(P.tail_o + ((size_t)(piece_row ? piece : 0) * kUnitRows + row) * D +
                                                    hf * DH);
#pragma unroll
            for (int ch = 0; ch < DH / 16; ++ch) {
                float o[16];
                if (n_mine > 0) {
                    tmem_ld2x_16<DH>(tO + ch * 16, o);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] = 0.f;
                }
                if (piece_row) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        po[ch * 4 + i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                } else if (write_row) {
                    uint32_t wv[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) wv[i] = use_o ? pack_bf16x2(o[2 * i] * inv, o[2 * i + 1] * inv) : 0u;
                    dst[2 * ch] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    dst[2 * ch + 1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                }
            }
            if (piece_row && hf == 0)
                P.tail_ml[(size_t)piece * kUnitRows + row] =
                    make_float2(n_mine > 0 ? m : -INFINITY, n_mine > 0 ? l : 0.f);
            if (P.lse && write_row && hf == 0) {
                float v = -INFINITY;
                if (use_o) v = (m + lg2(l)) * 0.69314718055994531f;
                P.lse[orow] = v;
            }
            tc_fence_before();
            mbar_arrive(BAR(BI.bm_empty(p)));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kSWarp) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ split tail merge
// Merges the key ranges of each split tail unit (128-token kernel tiles) into
// the output: for a query row with ranges r = 0 .. np-1 (unnormalised O_r,
// row maximum m_r in log2 units, row sum l_r)
//   M = max m_r,  w_r = 2^(m_r - M),  L = sum w_r l_r,  O = sum w_r O_r / L,
//   LSE = (M + log2 L) ln 2,
// summed in range order, with the rules of the attention kernel's epilogue: a
// row past the valid rows or with L == 0 is +0 and its LSE -inf (no range
// selected a key tile: M = -inf, L = 0); a NaN L gives a NaN row.  One thread
// per (unit, row, 16 columns).
constexpr int kMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) tail_merge_kernel(TailMergeParams q) {
    constexpr int kChunks = D / 16;
    const int64_t gid = (int64_t)blockIdx.x * kMergeThreads + threadIdx.x;
    if (gid >= (int64_t)q.units * kUnitRows * kChunks) return;
    const int ch = (int)(gid % kChunks);
    const int row = (int)((gid / kChunks) % kUnitRows);
    const int unit = (int)(gid / ((int64_t)kChunks * kUnitRows));
    const int item = q.tail_items[unit >> 1];
    const int bh = item / q.G, g = item - (item / q.G) * q.G;
    const int t = 2 * g + (unit & 1);  // the unit's 128-row kernel tile
    if (t >= q.NT) return;
    const bool valid = row < tile_size(q.block_sizes, t, q.sub);
    const int np = q.n_parts;
    const size_t b0 = (size_t)unit * np * kUnitRows + row;  // range r's row: b0 + r * kUnitRows
    float mr[kMaxParts], wr[kMaxParts];
#pragma unroll
    for (int r = 0; r < kMaxParts; ++r) {
        mr[r] = -INFINITY;
        wr[r] = 0.f;
        if (r < np) {
            const float2 ml = __ldcg(q.tail_ml + b0 + (size_t)r * kUnitRows);
            mr[r] = ml.x;
            wr[r] = ml.y;
        }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxParts; ++r) M = fmaxf(M, mr[r]);
    float L = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxParts; ++r) {
        const float w = (M != -INFINITY && mr[r] != -INFINITY) ? ex2(mr[r] - M) : 0.f;
        L += w * wr[r];
        wr[r] = w;
    }
    const bool use = valid && (L != 0.f);  // NaN L keeps it: NaN row
    const float inv = use ? 1.f / L : 0.f;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxParts; ++r) {
        if (r >= np) break;
        const float4 *src = reinterpret_cast<const float4 *>(q.tail_o + (b0 + (size_t)r * kUnitRows) * D) + ch * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 x = __ldcg(src + i);
            acc[4 * i] += wr[r] * x.x;
            acc[4 * i + 1] += wr[r] * x.y;
            acc[4 * i + 2] += wr[r] * x.z;
            acc[4 * i + 3] += wr[r] * x.w;
        }
    }
    const int64_t orow = (int64_t)bh * q.Sp + (int64_t)t * kUnitRows + row;
    uint32_t wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) wv[i] = use ? pack_bf16x2(acc[2 * i] * inv, acc[2 * i + 1] * inv) : 0u;
    uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(q.out) + orow * D) + ch * 2;
    dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
    if (q.lse && ch == 0) q.lse[orow] = use ? (M + lg2(L)) * 0.69314718055994531f : -INFINITY;
}

// The dense form (kPaired) runs with the selection bitmaps in shared memory
// only; beyond kSmemBitmapTiles kernel tiles the split, per-tile form runs.
template <int T, int D>
cudaError_t launch_t(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v, AttnParams p, bool paired,
                     int grid, cudaStream_t stream) {
    const int smem_words = p.bm_global ? 0 : p.bm_words;  // bitmap words held in shared memory
    const bool dense = paired && !p.bm_global;
    if (dense) {
        constexpr int KT = key_rows<T, true>();
        p.stages = stages_for<T, D, KT>(smem_words);
        const SmemPlan L = smem_plan<T, D, KT>(smem_words, p.stages);
        attn_fwd_kernel<T, D, true, false><<<grid, kAttnThreads, L.total, stream>>>(q, k, v, p);
    } else {
        constexpr int KT = key_rows<T, false>();
        p.stages = stages_for<T, D, KT>(smem_words);
        const SmemPlan L = smem_plan<T, D, KT>(smem_words, p.stages);
        if (p.bm_global)
            attn_fwd_kernel<T, D, false, true><<<grid, kAttnThreads, L.total, stream>>>(q, k, v, p);
        else
            attn_fwd_kernel<T, D, false, false><<<grid, kAttnThreads, L.total, stream>>>(q, k, v, p);
    }
    return cudaGetLastError();
}

template <int T, int D>
AttnLaunchInfo info_t(int bm_words, bool dense) {
    if (dense) {
        constexpr int KT = key_rows<T, true>();
        const int ns = stages_for<T, D, KT>(bm_words);
        return AttnLaunchInfo{ns, (int)smem_plan<T, D, KT>(bm_words, ns).total};
    }
    constexpr int KT = key_rows<T, false>();
    const int ns = stages_for<T, D, KT>(bm_words);
    return AttnLaunchInfo{ns, (int)smem_plan<T, D, KT>(bm_words, ns).total};
}

template <int T, int D>
cudaError_t prepare_t() {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<T, D, true, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_fwd_kernel<T, D, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemLimit);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_fwd_kernel<T, D, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemLimit);
}

}  // namespace

AttnLaunchInfo attn_launch_info(int tile, int head_dim, int bm_words, bool dense) {
    if (tile == 128 && head_dim == 128) return info_t<128, 128>(bm_words, dense);
    if (tile == 128 && head_dim == 64) return info_t<128, 64>(bm_words, dense);
    if (tile == 64 && head_dim == 128) return info_t<64, 128>(bm_words, dense);
    return info_t<64, 64>(bm_words, dense);
}

cudaError_t attn_prepare(int tile, int head_dim, int) {
    if (tile == 128 && head_dim == 128) return prepare_t<128, 128>();
    if (tile == 128 && head_dim == 64) return prepare_t<128, 64>();
    if (tile == 64 && head_dim == 128) return prepare_t<64, 128>();
    return prepare_t<64, 64>();
}

cudaError_t launch_attn(int tile, int head_dim, bool paired, const CUtensorMap &q, const CUtensorMap &k,
                        const CUtensorMap &v, AttnParams p, int grid, cudaStream_t stream) {
    if (tile == 128 && head_dim == 128) return launch_t<128, 128>(q, k, v, p, paired, grid, stream);
    if (tile == 128 && head_dim == 64) return launch_t<128, 64>(q, k, v, p, paired, grid, stream);
    if (tile == 64 && head_dim == 128) return launch_t<64, 128>(q, k, v, p, paired, grid, stream);
    return launch_t<64, 64>(q, k, v, p, paired, grid, stream);
}

cudaError_t launch_tail_merge(int head_dim, const TailMergeParams &q, cudaStream_t stream) {
    const int64_t threads = (int64_t)q.units * kUnitRows * (head_dim / 16);
    const unsigned blocks = (unsigned)((threads + kMergeThreads - 1) / kMergeThreads);
    if (head_dim == 128) tail_merge_kernel<128><<<blocks, kMergeThreads, 0, stream>>>(q);
    else tail_merge_kernel<64><<<blocks, kMergeThreads, 0, stream>>>(q);
    return cudaGetLastError();
}

}  // namespace vsa
