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
//   select_kernel  four query tiles per warp, two key tiles per lane: scores
//                  against all key tiles into shared memory (key means staged
//                  in 64-tile chunks, each 16-byte load serving four scores),
//                  then per query tile a bitwise search (per-lane counts, one
//                  warp reduction per bit) for the topk-th largest score and an
//                  ascending emit with ballots.
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

constexpr int kKeyRegs = 16;  // most keys per lane held in registers for the top-k search (NT <= 512)

// Writes the topk best of one row of keys (ascending tile order, -1 after)
// and returns how many were kept.  The kk-th largest key is found one bit at
// a time from the top: among keys that share the bits decided so far, those
// with bit b set are larger than those with it clear.  KR > 0 keeps the row's
// keys in KR registers per lane (NT <= 32 * KR) and counts in four
// independent partial sums; KR == 0 re-reads them from shared memory on every
// pass.
template <int KR>
__device__ __forceinline__ int row_topk(const uint32_t *rk, int NT, int topk, int nt_tok, int T, int32_t *out,
                                        int lane) {
    uint32_t kr[KR > 0 ? KR : 1];
    const int chunks = (NT + 31) / 32;
    unsigned n_cand = 0;
    if constexpr (KR > 0) {
#pragma unroll
        for (int c = 0; c < KR; ++c) {
            const int j = c * 32 + lane;
            kr[c] = j < NT ? rk[j] : 0u;
            n_cand += kr[c] != 0u;
        }
    } else {
        for (int c = 0; c < chunks; ++c) {
            const int j = c * 32 + lane;
            n_cand += j < NT && rk[j] != 0u;
        }
    }
    n_cand = __reduce_add_sync(0xffffffffu, n_cand);
    const int kk = (nt_tok > 0 && nt_tok <= T) ? (topk < (int)n_cand ? topk : (int)n_cand) : 0;
    if (kk == 0) {
        for (int i = lane; i < topk; i += 32) out[i] = -1;
        return 0;
    }
    uint32_t prefix = 0u;
    int need = kk;  // keys still to take at or below the current prefix
#pragma unroll 1
    for (int b = 31; b >= 0; --b) {
        const uint32_t m = 0xffffffffu << b, cand = prefix | (1u << b);
        // a key with the candidate prefix is non-zero, so no separate test for 0
        unsigned c4[4] = {0u, 0u, 0u, 0u};
        if constexpr (KR > 0) {
#pragma unroll
            for (int c = 0; c < KR; ++c) c4[c & 3] += (kr[c] & m) == cand;
        } else {
            for (int c = 0; c < chunks; ++c) {
                const int j = c * 32 + lane;
                c4[0] += j < NT && (rk[j] & m) == cand;
            }
        }
        const unsigned cnt = __reduce_add_sync(0xffffffffu, (c4[0] + c4[1]) + (c4[2] + c4[3]));
        if ((int)cnt >= need) prefix = cand;
        else need -= (int)cnt;
    }
    // every larger key and the first `need` keys equal to it, ascending
    const uint32_t lt = (1u << lane) - 1u;
    int base = 0, eq_seen = 0;
    for (int c = 0; c < chunks; ++c) {
        const int j = c * 32 + lane;
        const uint32_t key = j < NT ? rk[j] : 0u;
        const bool gt = key > prefix, eq = key == prefix && key != 0u;
        const uint32_t beq = __ballot_sync(0xffffffffu, eq);
        const bool sel = gt || (eq && eq_seen + __popc(beq & lt) < need);
        const uint32_t bsel = __ballot_sync(0xffffffffu, sel);
        if (sel) out[base + __popc(bsel & lt)] = j;
        base += __popc(bsel);
        eq_seen += __popc(beq);
    }
    for (int i = kk + lane; i < topk; i += 32) out[i] = -1;
    return kk;
}

// Dynamic shared memory: query means [WARPS*QPW][D], key-mean chunk
// [64][D+4], keys [WARPS*QPW][NT].
template <int D, int QPW, int WARPS>
__global__ void __launch_bounds__(WARPS * 32)
    select_kernel(const float *__restrict__ qm, const float *__restrict__ km, const int32_t *__restrict__ block_sizes,
                  int32_t *__restrict__ q2k_idx, int32_t *__restrict__ q2k_num, int NT, int T, int topk) {
    constexpr int KS = D + 4;  // padded key-mean row: 16-byte aligned, no bank conflicts on 16-byte loads
    constexpr int ROWS = WARPS * QPW;
    constexpr int LOADS = kSelectKeyChunk * (D / 4) / (WARPS * 32);  // float4 copies per thread per chunk
    extern __shared__ __align__(16) float sm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = blockIdx.y;
    const int t0 = blockIdx.x * ROWS;
    float *sq = sm;                                                              // [ROWS][D]
    float *skc = sq + ROWS * D;                                                  // [64][KS]
    uint32_t *keys = reinterpret_cast<uint32_t *>(skc + kSelectKeyChunk * KS);  // [ROWS][NT]

    for (int i = threadIdx.x; i < ROWS * D; i += WARPS * 32) {
        const int w = i / D, tt = t0 + w;
        sq[i] = tt < NT ? qm[(bh * NT + tt) * D + (i - w * D)] : 0.f;
    }
    // ---- scores: each warp takes QPW query tiles, each lane two key tiles of
    // a 64-tile chunk, so one 16-byte load of a key mean serves QPW scores.
    // Every score is a sum over d in order of fused multiply-adds.
    const int r0 = warp * QPW;  // first row (query tile) of this warp
    // key means of the next chunk travel in registers while the current chunk
    // is scored, so the global-load latency overlaps the arithmetic
    float4 tmp[LOADS];
    auto fetch = [&](int j0) {
        const int nj = NT - j0 < kSelectKeyChunk ? NT - j0 : kSelectKeyChunk;
#pragma unroll
        for (int u = 0; u < LOADS; ++u) {
            const int i = threadIdx.x + u * WARPS * 32;
            const int jj = i / (D / 4);
            tmp[u] = jj < nj ? reinterpret_cast<const float4 *>(km + (bh * NT + j0 + jj) * D)[i - jj * (D / 4)]
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    fetch(0);
    for (int j0 = 0; j0 < NT; j0 += kSelectKeyChunk) {
        __syncthreads();  // previous chunk consumed (and sq written, first time)
#pragma unroll
        for (int u = 0; u < LOADS; ++u) {
            const int i = threadIdx.x + u * WARPS * 32;
            const int jj = i / (D / 4);
            reinterpret_cast<float4 *>(skc + jj * KS)[i - jj * (D / 4)] = tmp[u];
        }
        __syncthreads();
        if (j0 + kSelectKeyChunk < NT) fetch(j0 + kSelectKeyChunk);
        const int nj = NT - j0 < kSelectKeyChunk ? NT - j0 : kSelectKeyChunk;
        float acc0[QPW], acc1[QPW];
#pragma unroll
        for (int q = 0; q < QPW; ++q) acc0[q] = acc1[q] = 0.f;
        const float4 *b0 = reinterpret_cast<const float4 *>(skc + lane * KS);
        const float4 *b1 = reinterpret_cast<const float4 *>(skc + (lane + 32) * KS);
#pragma unroll 4
        for (int d4 = 0; d4 < D / 4; ++d4) {
            const float4 y = b0[d4], z = b1[d4];
#pragma unroll
            for (int q = 0; q < QPW; ++q) {
                const float4 x = reinterpret_cast<const float4 *>(sq + (r0 + q) * D)[d4];
                acc0[q] = __fmaf_rn(x.x, y.x, acc0[q]);
                acc0[q] = __fmaf_rn(x.y, y.y, acc0[q]);
                acc0[q] = __fmaf_rn(x.z, y.z, acc0[q]);
                acc0[q] = __fmaf_rn(x.w, y.w, acc0[q]);
                acc1[q] = __fmaf_rn(x.x, z.x, acc1[q]);
                acc1[q] = __fmaf_rn(x.y, z.y, acc1[q]);
                acc1[q] = __fmaf_rn(x.z, z.z, acc1[q]);
                acc1[q] = __fmaf_rn(x.w, z.w, acc1[q]);
            }
        }
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int jj = lane + 32 * h2;
            if (jj < nj) {
                const int j = j0 + jj;
                const int n = __ldg(block_sizes + j);
                const bool cand = n > 0 && n <= T;
#pragma unroll
                for (int q = 0; q < QPW; ++q)
                    keys[(size_t)(r0 + q) * NT + j] = score_key(h2 ? acc1[q] : acc0[q], cand);
            }
        }
    }
    __syncwarp();

    // ---- top-k of each of this warp's rows
    for (int q = 0; q < QPW; ++q) {
        const int t = t0 + r0 + q;
        if (t >= NT) break;
        const uint32_t *rk = keys + (size_t)(r0 + q) * NT;
        int32_t *out = q2k_idx + (bh * NT + t) * (int64_t)topk;
        const int nt_tok = __ldg(block_sizes + t);
        int kk;
        if (NT <= 32 * 4) kk = row_topk<4>(rk, NT, topk, nt_tok, T, out, lane);
        else if (NT <= 32 * 8) kk = row_topk<8>(rk, NT, topk, nt_tok, T, out, lane);
        else if (NT <= 32 * 12) kk = row_topk<12>(rk, NT, topk, nt_tok, T, out, lane);
        else if (NT <= 32 * kKeyRegs) kk = row_topk<kKeyRegs>(rk, NT, topk, nt_tok, T, out, lane);
        else kk = row_topk<0>(rk, NT, topk, nt_tok, T, out, lane);
        if (lane == 0) q2k_num[bh * NT + t] = kk;
    }
}

}  // namespace

// Layouts of the select kernel: 4 warps x 4 query tiles per warp while their
// score rows fit in shared memory, else 4 warps x 1 query tile.
struct SelectShape {
    int warps, qpw;
};

SelectShape select_shape(int NT, int D) {
    if (select_smem_bytes(NT, D, 4 * 4) <= kSelectSmemLimit) return {4, 4};
    return {4, 1};
}

size_t select_smem_bytes(int NT, int D, int rows) {
    return sizeof(float) * ((size_t)rows * D + (size_t)kSelectKeyChunk * (D + 4)) + sizeof(uint32_t) * (size_t)rows * NT;
}

int select_warps(int NT, int D) { return select_shape(NT, D).warps; }

int select_rows(int NT, int D) {
    const SelectShape sh = select_shape(NT, D);
    return sh.warps * sh.qpw;
}

template <int D, int QPW, int WARPS>
cudaError_t select_attr() {
    return cudaFuncSetAttribute(select_kernel<D, QPW, WARPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSelectSmemLimit);
}

cudaError_t select_prepare() {
    cudaError_t e;
    if ((e = select_attr<64, 4, 4>()) != cudaSuccess) return e;
    if ((e = select_attr<128, 4, 4>()) != cudaSuccess) return e;
    if ((e = select_attr<64, 1, 4>()) != cudaSuccess) return e;
    return select_attr<128, 1, 4>();
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
    const SelectShape sh = select_shape(p.NT, p.D);
    const int rows = sh.warps * sh.qpw;
    dim3 grid((unsigned)((p.NT + rows - 1) / rows), (unsigned)(p.B * p.H));
    const size_t smem = select_smem_bytes(p.NT, p.D, rows);
    if (sh.qpw == 4) {
        if (p.D == 128)
            select_kernel<128, 4, 4><<<grid, 128, smem, stream>>>(p.qm, p.km, p.block_sizes, p.q2k_idx, p.q2k_num,
                                                                 p.NT, p.T, p.topk);
        else
            select_kernel<64, 4, 4><<<grid, 128, smem, stream>>>(p.qm, p.km, p.block_sizes, p.q2k_idx, p.q2k_num,
                                                                p.NT, p.T, p.topk);
    } else {
        if (p.D == 128)
            select_kernel<128, 1, 4><<<grid, 128, smem, stream>>>(p.qm, p.km, p.block_sizes, p.q2k_idx, p.q2k_num,
                                                                 p.NT, p.T, p.topk);
        else
            select_kernel<64, 1, 4><<<grid, 128, smem, stream>>>(p.qm, p.km, p.block_sizes, p.q2k_idx, p.q2k_num,
                                                                p.NT, p.T, p.topk);
    }
    return cudaGetLastError();
}

}  // namespace vsa
