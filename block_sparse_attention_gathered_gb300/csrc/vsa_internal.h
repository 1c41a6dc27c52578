// Internal interface between the host API (vsa_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace vsa {

// Bits of the device status word.
enum : int32_t { kFlagIndex = 1, kFlagTimeout = 2 };

// Query rows of one work item: two 128-row units, each one MMA M=128.
constexpr int kUnitRows = 128;
constexpr int kItemRows = 256;
constexpr int kAttnThreads = 640;  // 16 softmax warps, 2 MMA issuers, 1 producer, 1 fix-up warp
constexpr int kSmemBitmapTiles = 8192;  // VSA_SMEM_BITMAP_TILES
// Bitmaps per work-item buffer of the attention kernel: the four selection
// bitmaps (one per query-tile slot) and one of the selected tiles that are
// partial (fewer valid keys than the tile), so the kernel reads block_sizes
// only for those.
constexpr int kItemBitmaps = 5;
constexpr int kMaxGridCtas = 1024;      // bound on the attention grid (one CTA per SM), for workspace sizing
// Split tail: the work items of a last wave that fills at most half of the
// CTAs run as one-unit entries, and each of those can be cut further into up
// to kMaxParts parts by key-tile range (at most kMaxSplit entries in all).
// Each part leaves its unit's unnormalised O with the row maximum and row sum
// in the workspace; tail_merge_kernel then merges them into the output.
constexpr int kMaxSplit = 256;
constexpr int kMaxParts = 8;
// Order-list entries: work item << 5 | key part << 2 | units (0 both, 1 or 2 one).
constexpr int kEntryItemShift = 5;

struct AttnParams {
    const int32_t *q2k_idx;      // [B*H*NT, max_kv]
    const int32_t *q2k_num;      // [B*H*NT]
    const int32_t *block_sizes;  // [NT]
    void *out;                   // bf16 [B*H*Sp, D]
    float *lse;                  // [B*H*Sp] or nullptr
    const int32_t *order;        // [n_items] work order (longest first)
    int32_t *work_counter;       // next slot of `order` to hand out
    int32_t *status;             // device status word
    unsigned long long *steps;   // (tail, full) key-tile steps, added to by the producer warps
    uint32_t *bm_global;         // per-CTA selection bitmaps in the workspace (more than
                                 // kSmemBitmapTiles kernel tiles), or nullptr: in shared memory
    int32_t NT;                  // kernel tiles (128-token halves when sub == 2)
    int32_t sub;                 // kernel tiles per caller tile: 1, or 2 for 256-token tiles
    int32_t max_kv;
    int32_t G;                   // work items per (b, h)
    int32_t bm_words;            // 32-bit words of one selection bitmap
    int32_t n_items;
    int32_t stages;              // K/V ring depth (set by launch_attn)
    int64_t Sp;                  // NT * tile
    float scale_log2;            // softmax scale * log2(e)
    // split tail cut by key range (n_parts > 1 only): order slots from
    // tail_start on are the parts, unit by unit (piece = slot - tail_start,
    // its unit piece / n_parts)
    int32_t n_parts;
    int32_t tail_start;
    float *tail_o;               // [kMaxSplit pieces][kUnitRows][D] unnormalised O
    float2 *tail_ml;             // [kMaxSplit pieces][kUnitRows] (row maximum in log2 units, row sum)
};

// The split tail's merge (after the attention kernel, same stream): unit
// 2 ti + uu is unit uu of work item tail_items[ti]; its ranges are pieces
// unit * n_parts .. + n_parts - 1 of tail_o / tail_ml.
struct TailMergeParams {
    const float *tail_o;
    const float2 *tail_ml;
    const int32_t *tail_items;   // [units / 2] work item of each split tail item
    const int32_t *block_sizes;
    void *out;                   // bf16 [B*H*Sp, D]
    float *lse;                  // or nullptr
    int32_t units, n_parts, G, NT, sub;
    int64_t Sp;
};

cudaError_t launch_tail_merge(int head_dim, const TailMergeParams &q, cudaStream_t stream);

struct AttnLaunchInfo {
    int stages;
    int smem_bytes;
};

// Ring depth and dynamic shared memory of the attention kernel variant: the
// deepest K/V ring that fits the 227 KB per-CTA limit next to the Q tiles and
// the selection bitmaps (bm_words: bitmap words kept in shared memory, 0 when
// they live in the workspace; dense: the dense form, see launch_attn).
AttnLaunchInfo attn_launch_info(int tile, int head_dim, int bm_words, bool dense);

// Enables the variant's shared-memory size on the current device (once).
cudaError_t attn_prepare(int tile, int head_dim, int device);

// Launches with p.stages taken from attn_launch_info (the caller's value is
// ignored).  `paired` picks the dense form (all forms are exact; they differ
// only in speed): with 128-token kernel tiles the paired MMA-issue layout,
// with 64-token tiles ring entries of key-tile pairs, whose K and V maps then
// have 128-row boxes.  With bitmaps in the workspace it is ignored.
cudaError_t launch_attn(int tile, int head_dim, bool paired, const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                        const CUtensorMap &tm_v, AttnParams p, int grid, cudaStream_t stream);

struct LayoutParams {
    const void *src[3];
    void *dst[3];
    const int32_t *row_to_token;
    int32_t *status;
    int32_t n_tensors;
    int32_t B, S, H, Dv;  // Dv = head_dim / 8 (16-byte vectors per row)
    int64_t Sp;
};

cudaError_t launch_layout(const LayoutParams &p, int num_sms, cudaStream_t stream);

struct UntileParams {
    const void *o_tile;         // bf16 [B, H, Sp, D] tile-major output
    const void *gate;           // bf16 [B, S, H, D] or nullptr
    void *out;                  // bf16 [B, S, H, D] token-major
    const int32_t *row_to_token;
    int32_t *status;
    int32_t B, S, H, Dv;        // Dv = head_dim / 8
    int64_t Sp;
};

cudaError_t launch_untile(const UntileParams &p, int num_sms, cudaStream_t stream);

// Backward pass (vsa_bwd.cu).  It works on 128-row kernel tiles: a caller
// tile of 128, one half of a caller tile of 256, or two caller tiles of 64.
struct BwdGeo {
    int32_t NTk;     // kernel tiles per (b, h)
    int32_t maxlen;  // longest partner list of a kernel tile
};

inline BwdGeo bwd_geo(int T, int NTc, int max_kv) {
    BwdGeo g;
    g.NTk = T == 64 ? (NTc + 1) / 2 : (T == 128 ? NTc : 2 * NTc);
    const int per = (T == 128) ? 1 : 2;  // kernel tiles one selection entry can reach
    const int64_t m = (int64_t)per * (max_kv > 0 ? max_kv : 1);
    g.maxlen = (int32_t)(m < g.NTk ? m : g.NTk);
    if (g.maxlen < 1) g.maxlen = 1;
    return g;
}

struct BwdLaunch {
    const CUtensorMap *tm_q, *tm_k, *tm_v, *tm_do;  // rows of D bf16, box {64, 128}
    const void *out, *dout;                           // bf16 [B*H*Sp, D]
    const float *lse;                                 // [B*H*Sp]
    float *ndelta, *nlse2;                            // workspace [B*H*Spk] each: -delta, -lse*log2(e)
    const int32_t *q2k_idx, *q2k_num, *block_sizes;
    int32_t *pl, *pc;                                 // workspace [B*H*NTk, maxlen], [B*H*NTk]
    int32_t *k2q_offs, *k2q_list;                     // workspace [B*H, NTk+1], [B*H, NTk*maxlen]
    void *dq, *dk, *dv;                               // bf16 [B*H*Sp, D]
    int32_t *status;
    int32_t BH, T, NTc, NTk, D, max_kv, maxlen;
    int64_t Sp, Spk;                                  // NTc * T; NTk * 128
    float scale;
};

size_t bwd_smem_bytes(int D);
int bwd_threads();
cudaError_t bwd_prepare();
cudaError_t launch_bwd(const BwdLaunch &L, cudaStream_t stream);

// Coarse key-tile selection (vsa_select.cu).
constexpr uint32_t kSelectSmemLimit = 232448;  // 227 KB opt-in per CTA

struct SelectParams {
    const void *q, *k;           // bf16 tile-major [B*H*NT*T, D]
    const int32_t *block_sizes;  // [NT]
    float *qm, *km;              // workspace: fp32 tile means [B*H*NT, D]
    int32_t *q2k_idx;            // [B*H*NT, topk]
    int32_t *q2k_num;            // [B*H*NT]
    int32_t *status;             // device status word
    int32_t B, H, NT, T, D, topk;
};

// Warps and query tiles (score rows) per select CTA, chosen so the score rows fit.
int select_warps(int NT, int D);
int select_rows(int NT, int D);
size_t select_smem_bytes(int NT, int D, int rows);
cudaError_t select_prepare();
cudaError_t launch_select(const SelectParams &p, cudaStream_t stream);

// 64-bit ID of the calling thread's current CUDA context (unique for the
// process's life, so a context made after cudaDeviceReset gets a new one), or
// 0 when there is none yet or the driver cannot say.  Per-device caches of
// device addresses and function attributes are keyed on it.
unsigned long long current_context_id();

// Bounded-wait probe (vsa_check.cu).
cudaError_t launch_wait_probe(int32_t arrive, uint64_t limit_ns, int32_t *status, cudaStream_t stream);

}  // namespace vsa
