// Coarse key-tile selection for video sparse attention on sm_103a: the step
// that produces q2k_idx / q2k_num for the block-sparse forward.
//
// The FastVideo kernel page (hao-ai-lab/FastVideo commit 8503617,
// fastvideo-kernel/python) names video sparse attention and its block-sparse
// fine stage (commit adding the sm_121a tile-128 forward; "Wan VSA inference"
// in the fused tile_to_bhsd commit) but not the coarse stage's arithmetic.
// This library reads it as: pool every non-empty tile to the mean of its valid
// rows, score query tile t against key tile j by the dot product of the two
// means, keep the topk best key tiles per query tile (ties to the smaller
// index; empty tiles and NaN scores are never kept), written in ascending order.
//
// The kept set is an integer result decided by floating point, so the
// arithmetic is fixed: fp32, each mean summed over rows in order and divided
// once, each score summed over d in order of fused multiply-adds (one
// rounding per term).  Any implementation that follows these rules gets the
// same bits, and so the same selection.
//
//   pool_kernel    one thread per 16-byte column vector of one tile of Q or K,
//                  walking the tile's valid rows in order with 16 rows of loads
//                  in flight.  HBM-bound (reads every valid row of Q and K once).
//   select_kernel  one warp per query tile: scores against all key tiles into
//                  shared memory (key means staged in 64-tile chunks, two key
//                  tiles per lane, 16-byte shared loads), then a
//                  4-pass 8-bit radix select of the topk-th largest score and
//                  an ascending emit with ballots.
#include "vsa_internal.h"

namespace vsa {
namespace {

constexpr int kSelectKeyChunk = 64;  // key tiles staged in shared memory at a time

constexpr int kPoolThreads = 256;
constexpr int kPoolBatch = 16;  // rows whose loads are in flight together

// Thread = one 16-byte column vector of one tile of Q or K; consecutive
// threads cover a row, so each warp reads whole 128- or 256-byte rows.
__global__ void __launch_bounds__(kPoolThreads)
    pool_kernel(const uint4 *__restrict__ q, const uint4 *__restrict__ k, const int32_t *__restrict__ block_sizes,
                float *__restrict__ qm, float *__restrict__ km, int32_t *status, int64_t n_tiles, int NT, int T,
                int Dv) {
    const int64_t gid = (int64_t)blockIdx.x * kPoolThreads + threadIdx.x;
    const int64_t slot = gid / Dv;  // (tile, tensor) pair: tile = slot >> 1
    const int vec = (int)(gid - slot * Dv);
    const int64_t bht = slot >> 1;  // (b*H + h)*NT + t
    const int which = (int)(slot & 1);  // 0: q, 1: k
    if (bht >= n_tiles) return;
    const int t = (int)(bht % NT);
    int n = __ldg(block_sizes + t);
    if (n < 0 || n > T) {  // never read outside the tile; report the bad size
        if (vec == 0 && which == 0 && bht < NT) atomicOr(status, kFlagIndex);
        n = n < 0 ? 0 : T;
    }
    const uint4 *src = (which ? k : q) + bht * (int64_t)T * Dv + vec;
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = 0.f;
    // rows in order (fixed summation order); the loads of 16 rows are issued
    // before their adds, so each thread keeps 256 bytes in flight
    int r = 0;
    for (; r + kPoolBatch <= n; r += kPoolBatch) {
        uint4 v[kPoolBatch];
#pragma unroll
        for (int u = 0; u < kPoolBatch; ++u) v[u] = __ldg(src + (int64_t)(r + u) * Dv);
#pragma unroll
        for (int u = 0; u < kPoolBatch; ++u) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s[2 * i] = __fadd_rn(s[2 * i], __uint_as_float(w[i] << 16));
                s[2 * i + 1] = __fadd_rn(s[2 * i + 1], __uint_as_float(w[i] & 0xffff0000u));
            }
        }
    }
    for (; r < n; ++r) {
        const uint4 v = __ldg(src + (int64_t)r * Dv);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s[2 * i] = __fadd_rn(s[2 * i], __uint_as_float(w[i] << 16));
            s[2 * i + 1] = __fadd_rn(s[2 * i + 1], __uint_as_float(w[i] & 0xffff0000u));
        }
    }
    float4 *dst = reinterpret_cast<float4 *>((which ? km : qm) + bht * (int64_t)Dv * 8 + vec * 8);
    const float fn = (float)n;
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = n > 0 ? __fdiv_rn(s[i], fn) : 0.f;
    dst[0] = make_float4(m[0], m[1], m[2], m[3]);
    dst[1] = make_float4(m[4], m[5], m[6], m[7]);
}

// Order-preserving map of a score to an unsigned key (larger score -> larger
// key); 0 marks a tile that may not be kept (empty, or a NaN score).
__device__ __forceinline__ uint32_t score_key(float s, bool candidate) {
    if (!candidate || s != s) return 0u;
    const uint32_t u = __float_as_uint(s + 0.f);  // -0 -> +0: equal scores get equal keys
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Dynamic shared memory: query means [W][D], key-mean chunk [64][D+4],
// keys [W][NT], histograms [W][256].
template <int D>
__global__ void select_kernel(const float *__restrict__ qm, const float *__restrict__ km,
                              const int32_t *__restrict__ block_sizes, int32_t *__restrict__ q2k_idx,
                              int32_t *__restrict__ q2k_num, int NT, int T, int topk) {
    constexpr int KS = D + 4;  // padded key-mean row: 16-byte aligned, no bank conflicts on 16-byte loads
    extern __shared__ __align__(16) float sm[];
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = blockIdx.y;
    const int t0 = blockIdx.x * nw;
    float *sq = sm;                                   // [nw][D]
    float *skc = sq + nw * D;                         // [64][KS]
    uint32_t *keys = reinterpret_cast<uint32_t *>(skc + kSelectKeyChunk * KS);  // [nw][NT]
    uint32_t *hist = keys + (size_t)nw * NT;          // [nw][256]
    const int t = t0 + warp;
    const bool live = t < NT;

    for (int i = threadIdx.x; i < nw * D; i += blockDim.x) {
        const int w = i / D, tt = t0 + w;
        sq[i] = tt < NT ? qm[(bh * NT + tt) * D + (i - w * D)] : 0.f;
    }
    uint32_t *mykeys = keys + (size_t)warp * NT;
    // ---- scores of query tile t against every key tile, as keys.  Each lane
    // scores two key tiles of a 64-tile chunk; every score is a sum over d in
    // order of fused multiply-adds.
    for (int j0 = 0; j0 < NT; j0 += kSelectKeyChunk) {
        __syncthreads();  // previous chunk consumed (and sq written, first time)
        const int nj = NT - j0 < kSelectKeyChunk ? NT - j0 : kSelectKeyChunk;
        for (int i = threadIdx.x; i < nj * (D / 4); i += blockDim.x) {
            const int jj = i / (D / 4), d4 = i - jj * (D / 4);
            reinterpret_cast<float4 *>(skc + jj * KS)[d4] =
                reinterpret_cast<const float4 *>(km + (bh * NT + j0 + jj) * D)[d4];
        }
        __syncthreads();
        if (live && lane < nj) {
            const float4 *a = reinterpret_cast<const float4 *>(sq + warp * D);
            const float4 *b0 = reinterpret_cast<const float4 *>(skc + lane * KS);
            const float4 *b1 = reinterpret_cast<const float4 *>(skc + (lane + 32) * KS);
            const bool two = lane + 32 < nj;
            float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
            for (int d4 = 0; d4 < D / 4; ++d4) {
                const float4 x = a[d4], y = b0[d4];
                s0 = __fmaf_rn(x.x, y.x, s0);
                s0 = __fmaf_rn(x.y, y.y, s0);
                s0 = __fmaf_rn(x.z, y.z, s0);
                s0 = __fmaf_rn(x.w, y.w, s0);
                if (two) {
                    const float4 z = b1[d4];
                    s1 = __fmaf_rn(x.x, z.x, s1);
                    s1 = __fmaf_rn(x.y, z.y, s1);
                    s1 = __fmaf_rn(x.z, z.z, s1);
                    s1 = __fmaf_rn(x.w, z.w, s1);
                }
            }
            const int j = j0 + lane;
            const int n0 = __ldg(block_sizes + j);
            mykeys[j] = score_key(s0, n0 > 0 && n0 <= T);
            if (two) {
                const int n1 = __ldg(block_sizes + j + 32);
                mykeys[j + 32] = score_key(s1, n1 > 0 && n1 <= T);
            }
        }
    }
    __syncwarp();
    if (!live) return;

    // ---- number kept: every candidate up to topk; none for an empty query tile
    int n_cand = 0;
    for (int j = lane; j < NT; j += 32) n_cand += mykeys[j] != 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n_cand += __shfl_xor_sync(0xffffffffu, n_cand, o);
    const int nt_tok = __ldg(block_sizes + t);
    const int kk = (nt_tok > 0 && nt_tok <= T) ? (topk < n_cand ? topk : n_cand) : 0;
    int32_t *out = q2k_idx + (bh * NT + t) * (int64_t)topk;
    if (lane == 0) q2k_num[bh * NT + t] = kk;
    if (kk == 0) {
        for (int i = lane; i < topk; i += 32) out[i] = -1;
        return;
    }

    // ---- radix select of the kk-th largest key, 8 bits per pass from the top
    uint32_t *h = hist + warp * 256;
    uint32_t prefix = 0u;  // digits decided so far
    int need = kk;         // keys still to take at or below the current prefix
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        __syncwarp();  // every lane has read the previous pass's bins
        for (int i = lane; i < 256; i += 32) h[i] = 0u;
        __syncwarp();
        const uint32_t hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
        // lanes with the same digit add their count once (scores of a row often
        // share their leading digits, which would serialise plain atomics)
        for (int j0 = 0; j0 < NT; j0 += 32) {
            const int j = j0 + lane;
            const uint32_t key = j < NT ? mykeys[j] : 0u;
            const bool act = key != 0u && (key & hi_mask) == prefix;
            const uint32_t dig = act ? ((key >> shift) & 255u) : 256u;
            const uint32_t peers = __match_any_sync(0xffffffffu, dig);
            if (act && lane == __ffs(peers) - 1) atomicAdd(&h[dig], (uint32_t)__popc(peers));
        }
        __syncwarp();
        // lane l owns digits 255-8l .. 248-8l (descending); find the digit where
        // the count of keys at or above it first reaches `need`
        uint32_t c[8];
        uint32_t own = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c[i] = h[255 - 8 * lane - i];
            own += c[i];
        }
        uint32_t incl = own;  // inclusive scan over lanes (higher digits first)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const uint32_t excl = incl - own;
        const bool here = excl < (uint32_t)need && incl >= (uint32_t)need;
        const uint32_t who = __ballot_sync(0xffffffffu, here);
        const int src = __ffs(who) - 1;
        uint32_t digit = 0, above = 0;
        if (lane == src) {
            uint32_t run = excl;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (run + c[i] >= (uint32_t)need) {
                    digit = 255u - 8u * lane - i;
                    above = run;
                    break;
                }
                run += c[i];
            }
        }
        digit = __shfl_sync(0xffffffffu, digit, src);
        above = __shfl_sync(0xffffffffu, above, src);
        prefix |= digit << shift;
        need -= (int)above;
    }
    // prefix is now the kk-th largest key; take every larger key and the first
    // `need` keys equal to it, in ascending tile order
    int base = 0, eq_seen = 0;
    const uint32_t lt = (1u << lane) - 1u;
    for (int j0 = 0; j0 < NT; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < NT ? mykeys[j] : 0u;
        const bool gt = key > prefix, eq = key == prefix && key != 0u;
        const uint32_t beq = __ballot_sync(0xffffffffu, eq);
        const bool sel = gt || (eq && eq_seen + __popc(beq & lt) < need);
        const uint32_t bsel = __ballot_sync(0xffffffffu, sel);
        if (sel) out[base + __popc(bsel & lt)] = j;
        base += __popc(bsel);
        eq_seen += __popc(beq);
    }
    for (int i = kk + lane; i < topk; i += 32) out[i] = -1;
}

}  // namespace

size_t select_smem_bytes(int NT, int D, int warps) {
    return sizeof(float) * ((size_t)warps * D + (size_t)kSelectKeyChunk * (D + 4)) +
           sizeof(uint32_t) * ((size_t)warps * NT + (size_t)warps * 256);
}

int select_warps(int NT, int D) {
    int w = 8;
    while (w > 1 && select_smem_bytes(NT, D, w) > kSelectSmemLimit) --w;
    return w;
}

cudaError_t select_prepare() {
    cudaError_t e = cudaFuncSetAttribute(select_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSelectSmemLimit);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(select_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSelectSmemLimit);
}

cudaError_t launch_select(const SelectParams &p, cudaStream_t stream) {
    const int64_t n_tiles = (int64_t)p.B * p.H * p.NT;
    const int Dv = p.D / 8;
    const int64_t threads = n_tiles * 2 * Dv;
    pool_kernel<<<(unsigned)((threads + kPoolThreads - 1) / kPoolThreads), kPoolThreads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(p.q), reinterpret_cast<const uint4 *>(p.k), p.block_sizes, p.qm, p.km,
        p.status, n_tiles, p.NT, p.T, Dv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int w = select_warps(p.NT, p.D);
    dim3 grid((unsigned)((p.NT + w - 1) / w), (unsigned)(p.B * p.H));
    const size_t smem = select_smem_bytes(p.NT, p.D, w);
    if (p.D == 128)
        select_kernel<128><<<grid, 32 * w, smem, stream>>>(p.qm, p.km, p.block_sizes, p.q2k_idx, p.q2k_num, p.NT,
                                                             p.T, p.topk);
    else
        select_kernel<64><<<grid, 32 * w, smem, stream>>>(p.qm, p.km, p.block_sizes, p.q2k_idx, p.q2k_num, p.NT,
                                                            p.T, p.topk);
    return cudaGetLastError();
}

}  // namespace vsa
