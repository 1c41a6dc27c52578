// Fused tile layout and its inverse for sm_103a (fused tile_to_bhsd commit on the FastVideo
// kernel page, hao-ai-lab/FastVideo commit 8503617: one pass that moves
// token-major Q/K/V into tile-major BHSD instead of a scatter plus transposed
// copies).
//
// Formulated as a gather by destination row: every tile-major row is written
// exactly once, either from its source token or with +0 for a padding row, so
// padding is zeroed in the same pass.  Each thread owns one 16-byte column
// vector of one head and walks rows; the threads of a row slice read the
// token's H*D contiguous elements and write H runs of D*2 contiguous bytes.
// Up to three tensors move per pass.  HBM-bound: no shared memory, no
// tensor cores.
#include "vsa_internal.h"

namespace vsa {
namespace {

constexpr int kLayoutThreads = 256;
constexpr int kRowsInFlight = 2;   // layout: three tensors, so six loads in flight per thread
constexpr int kUntileRows = 4;     // un-tiling: two loads per row

__global__ void __launch_bounds__(kLayoutThreads)
    layout_kernel(const LayoutParams P, int rows_per_block, int hv_per_block) {
    const int HV = P.H * P.Dv;
    const int rl = threadIdx.x / hv_per_block;
    const int hv = blockIdx.y * hv_per_block + (threadIdx.x - rl * hv_per_block);
    if (rl >= rows_per_block || hv >= HV) return;
    const int h = hv / P.Dv;
    const int vec = hv - h * P.Dv;
    const int b = blockIdx.z;
    const int64_t Sp = P.Sp;
    const int64_t src_b = (int64_t)b * P.S * HV + hv;                     // + s*HV
    const int64_t dst_bh = (((int64_t)b * P.H + h) * Sp) * P.Dv + vec;   // + row*Dv
    const int64_t step = (int64_t)gridDim.x * rows_per_block;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    bool bad = false;

    for (int64_t row0 = (int64_t)blockIdx.x * rows_per_block + rl; row0 < Sp; row0 += step * kRowsInFlight) {
        int64_t rows[kRowsInFlight];
        int32_t tok[kRowsInFlight];
#pragma unroll
        for (int i = 0; i < kRowsInFlight; ++i) {
            rows[i] = row0 + i * step;
            tok[i] = rows[i] < Sp ? __ldg(P.row_to_token + rows[i]) : -1;
            if (tok[i] >= P.S || tok[i] < -1) {
                bad = true;
                tok[i] = -1;
            }
        }
        uint4 v[kRowsInFlight][3];
#pragma unroll
        for (int i = 0; i < kRowsInFlight; ++i)
#pragma unroll
            for (int x = 0; x < 3; ++x) {
                v[i][x] = zero;
                if (x < P.n_tensors && tok[i] >= 0)
                    v[i][x] = __ldcs(reinterpret_cast<const uint4 *>(P.src[x]) + src_b + (int64_t)tok[i] * HV);
            }
#pragma unroll
        for (int i = 0; i < kRowsInFlight; ++i) {
            if (rows[i] >= Sp) continue;
#pragma unroll
            for (int x = 0; x < 3; ++x)
                if (x < P.n_tensors) reinterpret_cast<uint4 *>(P.dst[x])[dst_bh + rows[i] * P.Dv] = v[i][x];
        }
    }
    if (bad) atomicOr(P.status, kFlagIndex);
}

// Output un-tiling, the inverse of layout_kernel: every tile-major row that
// holds a token goes back to token-major order, times the token's gate when
// one is given.  bf16 x bf16 is exact in fp32, so the product is rounded once
// (to nearest even) to bf16.  Padding rows are not read.
__global__ void __launch_bounds__(kLayoutThreads)
    untile_kernel(const UntileParams P, int rows_per_block, int hv_per_block) {
    const int HV = P.H * P.Dv;
    const int rl = threadIdx.x / hv_per_block;
    const int hv = blockIdx.y * hv_per_block + (threadIdx.x - rl * hv_per_block);
    if (rl >= rows_per_block || hv >= HV) return;
    const int h = hv / P.Dv;
    const int vec = hv - h * P.Dv;
    const int b = blockIdx.z;
    const int64_t Sp = P.Sp;
    const uint4 *src = reinterpret_cast<const uint4 *>(P.o_tile) + (((int64_t)b * P.H + h) * Sp) * P.Dv + vec;
    const int64_t tok_b = (int64_t)b * P.S * HV + hv;  // + s*HV
    const int64_t step = (int64_t)gridDim.x * rows_per_block;
    bool bad = false;
    for (int64_t row0 = (int64_t)blockIdx.x * rows_per_block + rl; row0 < Sp; row0 += step * kUntileRows) {
        int64_t rows[kUntileRows];
        int32_t tok[kUntileRows];
        uint4 o[kUntileRows], gt[kUntileRows];
#pragma unroll
        for (int i = 0; i < kUntileRows; ++i) {
            rows[i] = row0 + i * step;
            tok[i] = rows[i] < Sp ? __ldg(P.row_to_token + rows[i]) : -1;
            if (tok[i] >= P.S || tok[i] < -1) {
                bad = true;
                tok[i] = -1;
            }
            if (tok[i] >= 0) {
                o[i] = __ldcs(src + rows[i] * P.Dv);
                if (P.gate) gt[i] = __ldcs(reinterpret_cast<const uint4 *>(P.gate) + tok_b + (int64_t)tok[i] * HV);
            }
        }
#pragma unroll
        for (int i = 0; i < kUntileRows; ++i) {
            if (tok[i] < 0) continue;
            uint4 v = o[i];
            if (P.gate) {
                uint32_t a[4] = {o[i].x, o[i].y, o[i].z, o[i].w}, g[4] = {gt[i].x, gt[i].y, gt[i].z, gt[i].w};
                uint32_t r[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = __uint_as_float(a[k] << 16) * __uint_as_float(g[k] << 16);
                    const float hi = __uint_as_float(a[k] & 0xffff0000u) * __uint_as_float(g[k] & 0xffff0000u);
                    uint32_t w;
                    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
                    r[k] = w;
                }
                v = make_uint4(r[0], r[1], r[2], r[3]);
            }
            __stcs(reinterpret_cast<uint4 *>(P.out) + tok_b + (int64_t)tok[i] * HV, v);
        }
    }
    if (bad) atomicOr(P.status, kFlagIndex);
}

}  // namespace

static dim3 row_grid(int H, int Dv, int B, int64_t Sp, int num_sms, int *R_out, int *hvb_out) {
    const int HV = H * Dv;
    const int hvb = HV < kLayoutThreads ? HV : kLayoutThreads;
    const int R = kLayoutThreads / hvb;  // rows per block iteration
    const int gy = (HV + hvb - 1) / hvb;
    const int64_t row_blocks = (Sp + R - 1) / R;
    int64_t gx = ((int64_t)num_sms * (2048 / kLayoutThreads) + (int64_t)gy * B - 1) / ((int64_t)gy * B);
    gx = gx < 1 ? 1 : gx;
    gx = gx > row_blocks ? row_blocks : gx;
    *R_out = R;
    *hvb_out = hvb;
    return dim3((unsigned)gx, (unsigned)gy, (unsigned)B);
}

cudaError_t launch_untile(const UntileParams &p, int num_sms, cudaStream_t stream) {
    int R, hvb;
    const dim3 grid = row_grid(p.H, p.Dv, p.B, p.Sp, num_sms, &R, &hvb);
    untile_kernel<<<grid, R * hvb, 0, stream>>>(p, R, hvb);
    return cudaGetLastError();
}

cudaError_t launch_layout(const LayoutParams &p, int num_sms, cudaStream_t stream) {
    int R, hvb;
    const dim3 grid = row_grid(p.H, p.Dv, p.B, p.Sp, num_sms, &R, &hvb);
    layout_kernel<<<grid, R * hvb, 0, stream>>>(p, R, hvb);
    return cudaGetLastError();
}

}  // namespace vsa
