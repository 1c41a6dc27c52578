// Host side of the C ABI declared in include/vsa.h: argument and limit checks,
// the per-device cache, TMA descriptor encoding, the on-device work ordering
// (host scheduler step), the opt-in selection check and the device status
// word.
//
// Limits and fail-closed behaviour follow the sm_121a hardening commit on the
// FastVideo kernel page (hao-ai-lab/FastVideo commit 8503617): batch*heads <=
// 65535 and rows < 2^31 are checked before any launch; a device the kernels
// were not built for is refused with an error instead of returning
// uninitialised output; the SM count and the shared-memory opt-in are cached
// per device in atomics.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {
namespace {

__device__ int32_t g_device_status;  // bits kFlag*; read and cleared by vsa_check_device_status
// (tail, full) key-tile steps of the last forward call: zeroed by the ordering
// kernel, counted by the attention kernel, read by vsa_last_step_counts
__device__ unsigned long long g_step_counts[2];

constexpr int kMaxDevices = 64;

struct DeviceCache {
    std::atomic<int> state{0};  // 0 unknown, 1 supported sm_103, -1 unsupported
    // the context the entries below were taken in: after cudaDeviceReset the
    // device gets a new context, a new address for the status word and no
    // function attributes, so the entry is rebuilt
    std::atomic<unsigned long long> ctx_id{0};
    std::atomic<int> sm_count{0};
    std::atomic<unsigned> attn_prepared{0};  // bit per (tile, head_dim) variant
    std::atomic<int32_t *> status_ptr{nullptr};
    std::atomic<unsigned long long *> steps_ptr{nullptr};
};
DeviceCache g_dev[kMaxDevices];

thread_local vsa_route t_route{};

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
std::once_flag g_ctx_once;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

}  // namespace

unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(a);
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(b);
        }
        cudaGetLastError();
    });
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr || g_ctx_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

namespace {

// Current device, checked to be an sm_103 part; fills its cache entry.
vsa_status current_device(int *dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return VSA_ERR_ARCH;
    DeviceCache &c = g_dev[dev];
    int st = c.state.load(std::memory_order_acquire);
    if (st == 1 && c.ctx_id.load(std::memory_order_acquire) != current_context_id()) {
        // a new context since the entry was made (cudaDeviceReset): take it afresh
        c.attn_prepared.store(0u, std::memory_order_release);
        st = 0;
    }
    if (st == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return VSA_ERR_CUDA;
        }
        st = (major == 10 && minor == 3) ? 1 : -1;
        if (st == 1) {
            int32_t *p = nullptr;
            if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_device_status) != cudaSuccess) {
                cudaGetLastError();
                return VSA_ERR_CUDA;
            }
            unsigned long long *steps = nullptr;
            if (cudaGetSymbolAddress(reinterpret_cast<void **>(&steps), g_step_counts) != cudaSuccess) {
                cudaGetLastError();
                return VSA_ERR_CUDA;
            }
            c.status_ptr.store(p, std::memory_order_release);
            c.steps_ptr.store(steps, std::memory_order_release);
            c.sm_count.store(sms, std::memory_order_release);
            c.ctx_id.store(current_context_id(), std::memory_order_release);  // the symbol lookup made it current
        }
        c.state.store(st, std::memory_order_release);
    }
    if (st != 1) return VSA_ERR_ARCH;
    *dev_out = dev;
    return VSA_OK;
}

int64_t kernel_tiles(const vsa_dims *d) { return (int64_t)d->num_tiles * (d->tile == 256 ? 2 : 1); }

vsa_status check_dims(const vsa_dims *d) {
    if (!d) return VSA_ERR_ARG;
    if (d->B <= 0 || d->H <= 0 || d->num_tiles <= 0 || d->max_kv < 0) return VSA_ERR_ARG;
    if (d->tile != 64 && d->tile != 128 && d->tile != 256) return VSA_ERR_ARG;
    if (d->head_dim != 64 && d->head_dim != 128) return VSA_ERR_ARG;
    if (!std::isfinite(d->scale)) return VSA_ERR_ARG;
    if ((int64_t)d->B * d->H > VSA_MAX_BATCH_HEADS) return VSA_ERR_LIMITS;
    // 256-token tiles run as two 128-token halves each
    if (kernel_tiles(d) > VSA_MAX_TILES) return VSA_ERR_LIMITS;
    const int64_t rows = (int64_t)d->B * d->H * d->num_tiles * d->tile;
    if (rows + kItemRows >= (int64_t(1) << VSA_MAX_ROWS_LOG2)) return VSA_ERR_LIMITS;
    if ((int64_t)d->B * d->H * d->num_tiles * (int64_t)d->max_kv >= (int64_t(1) << 31)) return VSA_ERR_LIMITS;
    return VSA_OK;
}

int64_t items_per_seq(const vsa_dims *d) { return ((int64_t)d->num_tiles * d->tile + kItemRows - 1) / kItemRows; }

constexpr size_t kWsHeader = 256;  // work counter, padded

// Work items of the last, partly filled wave may run as one-unit entries on
// several CTAs (at most kMaxSplit entries in all, kMaxSplit and kMaxParts in
// vsa_internal.h): the order list grows by at most kMaxSplit entries.
// Beyond kTailMinItems work items (where a last wave can be partly filled on
// this part, 148 SMs or more) the workspace also holds the split tail's
// partial results.
constexpr int64_t kTailMinItems = 128;

// Dims the backward and the coarse selection accept: check_dims plus their
// tighter tile limit.
vsa_status check_dims_small(const vsa_dims *d) {
    const vsa_status st = check_dims(d);
    if (st != VSA_OK) return st;
    return kernel_tiles(d) > VSA_MAX_TILES_BWD ? VSA_ERR_LIMITS : VSA_OK;
}

// Workspace of the forward: a 256 B header (work counter), the order list,
// and, beyond kSmemBitmapTiles kernel tiles, the selection bitmaps of every
// CTA (two buffers of kItemBitmaps bitmaps of ceil(kernel tiles / 32) words each),
// 256-byte aligned.
int bitmap_words(const vsa_dims *d) { return (int)((kernel_tiles(d) + 31) / 32); }
bool bitmaps_in_workspace(const vsa_dims *d) { return kernel_tiles(d) > kSmemBitmapTiles; }
size_t order_bytes_for(const vsa_dims *d) {
    const int64_t n_items = (int64_t)d->B * d->H * items_per_seq(d);
    return kWsHeader + (size_t)(n_items + kMaxSplit) * sizeof(int32_t);
}
size_t bitmap_offset_for(const vsa_dims *d) { return (order_bytes_for(d) + 255) & ~(size_t)255; }
size_t bitmap_bytes_per_cta(const vsa_dims *d) {
    return (size_t)2 * kItemBitmaps * bitmap_words(d) * sizeof(uint32_t);
}

// The least workspace the forward accepts: header, order list and (beyond
// kSmemBitmapTiles kernel tiles) the bitmaps.
size_t base_bytes_for(const vsa_dims *d) {
    if (!bitmaps_in_workspace(d)) return order_bytes_for(d);
    const int64_t n_items = (int64_t)d->B * d->H * items_per_seq(d);
    const int64_t ctas = n_items < kMaxGridCtas ? n_items : kMaxGridCtas;
    return bitmap_offset_for(d) + (size_t)ctas * bitmap_bytes_per_cta(d);
}
// Split-tail region, 256-byte aligned after the base: the work item of each
// split tail item (kMaxSplit slots), then kMaxSplit pieces of (row maximum,
// row sum) per unit row, then kMaxSplit pieces of unnormalised O rows (fp32).
size_t tail_offset_for(const vsa_dims *d) { return (base_bytes_for(d) + 255) & ~(size_t)255; }
constexpr size_t kTailCntBytes = (size_t)kMaxSplit * sizeof(int32_t);
constexpr size_t kTailMlBytes = (size_t)kMaxSplit * kUnitRows * 2 * sizeof(float);
size_t tail_bytes_for(const vsa_dims *d) {
    const int64_t n_items = (int64_t)d->B * d->H * items_per_seq(d);
    if (n_items <= kTailMinItems) return 0;
    return kTailCntBytes + kTailMlBytes + (size_t)kMaxSplit * kUnitRows * d->head_dim * sizeof(float);
}
size_t workspace_bytes_for(const vsa_dims *d) {
    const size_t tail = tail_bytes_for(d);
    return tail ? tail_offset_for(d) + tail : base_bytes_for(d);
}

vsa_status encode_rows_map(CUtensorMap *m, const void *ptr, int64_t rows, int D, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return VSA_ERR_CUDA;
    cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), gdim, gstride, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? VSA_OK : VSA_ERR_CUDA;
}

// ------------------------------------------------------------------ schedule
// Orders the 256-row work items by their total number of selected key tiles,
// largest first (a counting sort into `bins` buckets), and resets the work
// counter the attention kernel's CTAs draw from.  One CTA; equal keys land in
// any order, which does not change any output (items are independent, and a
// one-unit entry computes its unit exactly as the whole item does).  Items cut
// into key ranges (parts > 1) do round differently, so those are not taken
// from the sorted order but are always the last `split` items by index, which
// keeps every output bit-identical from call to call.
constexpr int kSchedThreads = 1024;

__global__ void __launch_bounds__(kSchedThreads)
    schedule_kernel(const int32_t *__restrict__ q2k_num, int NT, int T, int max_kv, int G, int n_items, int bins,
                    int split, int parts, int32_t *__restrict__ order, int32_t *__restrict__ counter,
                    int32_t *__restrict__ tail_items, unsigned long long *__restrict__ steps) {
    extern __shared__ int32_t sh[];
    int32_t *hist = sh;          // [bins], indexed by descending rank
    int32_t *cursor = sh + bins;  // [bins]
    __shared__ int32_t warp_tot[kSchedThreads / 32];
    const int tid = threadIdx.x;
    const int per_item = kItemRows / T;  // caller tiles per work item: 4, 2 or 1
    const int64_t wmax = (int64_t)per_item * (max_kv > 0 ? max_kv : 1);
    for (int i = tid; i < bins; i += kSchedThreads) hist[i] = 0;
    __syncthreads();
    auto rank_of = [&](int item) -> int {
        const int bh = item / G, g = item - (item / G) * G;
        int64_t w = 0;
        for (int k = 0; k < per_item; ++k) {
            const int t = g * per_item + k;
            if (t >= NT) break;
            int n = __ldg(q2k_num + (int64_t)bh * NT + t);
            n = n < 0 ? 0 : (n > max_kv ? max_kv : n);
            w += n;
        }
        const int bin = (int)(w * (bins - 1) / wmax);
        return bins - 1 - bin;  // larger weight -> smaller rank
    };
    const int whole = n_items - split;
    const int sorted = parts > 1 ? whole : n_items;  // items placed by the sort
    for (int i = tid; i < sorted; i += kSchedThreads) atomicAdd(&hist[rank_of(i)], 1);
    __syncthreads();
    // exclusive scan of hist over ranks: each thread owns a contiguous run
    const int per = (bins + kSchedThreads - 1) / kSchedThreads;
    const int lo = tid * per, hi = min(bins, lo + per);
    int32_t run = 0;
    for (int i = lo; i < hi; ++i) run += hist[i];
    int32_t incl = run;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int32_t x = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        warp_tot[lane] = x;  // inclusive over warps
    }
    __syncthreads();
    int32_t pos = incl - run + (wid > 0 ? warp_tot[wid - 1] : 0);
    for (int i = lo; i < hi; ++i) {
        cursor[i] = pos;
        pos += hist[i];
    }
    __syncthreads();
    // entries are item << 5 | key part << 2 | units: 0 both; the `split` tail
    // items (with parts == 1 the last sorted positions, the shortest items;
    // else the last items by index) become 2 x parts entries each, unit 0 only
    // (1) and unit 1 only (2), each in `parts` key-tile ranges, so the last
    // partial wave spreads over 2 x parts times the CTAs
    auto put_tail = [&](int ti, int i) {
        const int q = whole + 2 * parts * ti;
        for (int uu = 0; uu < 2; ++uu)
            for (int part = 0; part < parts; ++part)
                order[q + uu * parts + part] = (i << kEntryItemShift) | (part << 2) | (uu + 1);
        if (tail_items) tail_items[ti] = i;  // for the merge of its ranges
    };
    for (int i = tid; i < sorted; i += kSchedThreads) {
        const int pos = atomicAdd(&cursor[rank_of(i)], 1);
        if (pos < whole) order[pos] = i << kEntryItemShift;
        else put_tail(pos - whole, i);
    }
    if (parts > 1)
        for (int ti = tid; ti < split; ti += kSchedThreads) put_tail(ti, whole + ti);
    if (tid == 0) {
        *counter = 0;
        steps[0] = 0ull;
        steps[1] = 0ull;
    }
}

// ------------------------------------------------------------------ validate
__global__ void validate_kernel(const int32_t *__restrict__ q2k_idx, const int32_t *__restrict__ q2k_num,
                                const int32_t *__restrict__ block_sizes, int64_t n_rows, int NT, int T, int max_kv,
                                int32_t *dev_status) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    bool bad = false;
    if (i < NT) {
        const int n = block_sizes[i];
        bad |= (n < 0 || n > T);
    }
    if (i < n_rows) {
        const int K = q2k_num[i];
        if (K < 0 || K > max_kv) {
            bad = true;
        } else {
            const int32_t *sel = q2k_idx + i * max_kv;
            for (int a = 0; a < K && !bad; ++a) {
                const int j = sel[a];
                if (j < 0 || j >= NT) bad = true;
                for (int b = 0; b < a && !bad; ++b)
                    if (sel[b] == j) bad = true;
            }
        }
    }
    if (bad) atomicExch(dev_status, (int32_t)VSA_ERR_INDEX);
}

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" {

int32_t vsa_version(void) { return 1002; }

const char *vsa_status_string(vsa_status s) {
    switch (s) {
        case VSA_OK: return "ok";
        case VSA_ERR_ARG: return "invalid argument";
        case VSA_ERR_ALIGN: return "pointer not 16-byte aligned";
        case VSA_ERR_LIMITS: return "launch limit exceeded";
        case VSA_ERR_ARCH: return "device is not sm_103 (GB300)";
        case VSA_ERR_CUDA: return "CUDA runtime error";
        case VSA_ERR_TIMEOUT: return "device-side wait timed out";
        case VSA_ERR_INDEX: return "invalid selection index, count or row map";
        case VSA_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

size_t vsa_block_sparse_workspace_size(const vsa_dims *dims) {
    if (check_dims(dims) != VSA_OK) return 0;
    return workspace_bytes_for(dims);
}

size_t vsa_block_sparse_workspace_size_min(const vsa_dims *dims) {
    if (check_dims(dims) != VSA_OK) return 0;
    return base_bytes_for(dims);
}

vsa_status vsa_block_sparse_fwd(const void *q, const void *k, const void *v, const int32_t *q2k_idx,
                                const int32_t *q2k_num, const int32_t *block_sizes, void *out, float *lse,
                                const vsa_dims *dims, void *workspace, size_t workspace_bytes,
                                vsa_stream_t stream) {
    vsa_status st = check_dims(dims);
    if (st != VSA_OK) return st;
    if (!q || !k || !v || !q2k_num || !block_sizes || !out || (!q2k_idx && dims->max_kv > 0))
        return VSA_ERR_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(q2k_num, 4) ||
        !aligned(block_sizes, 4) || (q2k_idx && !aligned(q2k_idx, 4)) || (lse && !aligned(lse, 4)))
        return VSA_ERR_ALIGN;
    const size_t need = base_bytes_for(dims);
    if (!workspace || workspace_bytes < need) return VSA_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return VSA_ERR_ALIGN;
    // the split tail's partial results need the full size
    const size_t tail_bytes = tail_bytes_for(dims);
    const bool tail_room = tail_bytes > 0 && workspace_bytes >= tail_offset_for(dims) + tail_bytes;
    int dev = 0;
    if ((st = current_device(&dev)) != VSA_OK) return st;
    DeviceCache &dc = g_dev[dev];

    const int T = dims->tile, D = dims->head_dim, NT = dims->num_tiles;
    // 256-token tiles: the 128-token kernel on the two halves of every tile
    const int Tk = T == 256 ? 128 : T, sub = T / Tk;
    const unsigned variant_bit = 1u << ((Tk == 128 ? 2 : 0) + (D == 128 ? 1 : 0));
    if (!(dc.attn_prepared.load(std::memory_order_acquire) & variant_bit)) {
        if (attn_prepare(Tk, D, dev) != cudaSuccess) {
            cudaGetLastError();
            return VSA_ERR_CUDA;
        }
        dc.attn_prepared.fetch_or(variant_bit, std::memory_order_acq_rel);
    }

    // The dense form: when the rows of q2k_idx can hold every key tile (a
    // dense selection) or with 256-token tiles (both units are halves of one
    // query tile and share its selection).
    //  * 128-token kernel tiles, D = 128: the paired MMA-issue layout.  The
    //    split layout measured faster as soon as a few key tiles serve only
    //    one unit (95 % selections included), and at every density with
    //    D = 64, where a P V product is N = 64 wide.
    //  * 64-token tiles: ring entries of key-tile pairs, so S is N = 128 wide
    //    (dense T64 D128: 2.86 -> 2.50 ms).  Pairs measured 1.5-1.8 times
    //    slower on top-k and uniform sparse selections, which rarely take both
    //    tiles of a pair.
    // The host cannot see the selections without a sync, so the row length
    // stands in for the density.  Results do not depend on the form.  It runs
    // with the selection bitmaps in shared memory only.
    const bool dense_sel = sub == 2 || dims->max_kv >= NT;
    const bool paired = !bitmaps_in_workspace(dims) && dense_sel && ((Tk == 128 && D == 128) || Tk == 64);
    const int key_rows = (Tk == 64 && paired) ? 128 : Tk;

    const int64_t Sp = (int64_t)NT * T;
    const int64_t rows = (int64_t)dims->B * dims->H * Sp;
    CUtensorMap tm_q, tm_k, tm_v;
    if ((st = encode_rows_map(&tm_q, q, rows, D, kUnitRows)) != VSA_OK) return st;
    // K and V go by ring entries of key_rows rows (a tile, or a pair of
    // 64-token tiles)
    if ((st = encode_rows_map(&tm_k, k, rows, D, key_rows)) != VSA_OK) return st;
    if ((st = encode_rows_map(&tm_v, v, rows, D, key_rows)) != VSA_OK) return st;

    const int G = (int)items_per_seq(dims);
    const int n_items = (int)((int64_t)dims->B * dims->H * G);
    const int per_item = kItemRows / T;
    const int64_t wmax = (int64_t)per_item * (dims->max_kv > 0 ? dims->max_kv : 1);
    const int bins = (int)(wmax + 1 < 2048 ? wmax + 1 : 2048);
    int32_t *counter = reinterpret_cast<int32_t *>(workspace);
    int32_t *order = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(workspace) + kWsHeader);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // One persistent CTA per SM.  When the last wave would fill at most half
    // of them, its items are split into one-unit entries, and with 128-token
    // kernel tiles and room in the workspace each of those into `parts`
    // key-tile ranges, as many as keep the entries within the grid (a unit's
    // time then drops to about 1/parts).
    // (kMaxGridCtas bounds the grid for the workspace's per-CTA bitmap regions)
    const int sms = std::min(dc.sm_count.load(std::memory_order_acquire), kMaxGridCtas);
    const int grid = n_items < sms ? n_items : sms;
    const int rem = n_items > grid ? n_items % grid : 0;
    const int split = (rem > 0 && 2 * rem <= grid && 2 * rem <= kMaxSplit) ? rem : 0;
    int parts = 1;
    if (split > 0 && tail_room && Tk == 128) parts = std::max(1, std::min(kMaxParts, std::min(grid, kMaxSplit) / (2 * split)));
    char *tail = reinterpret_cast<char *>(workspace) + tail_offset_for(dims);
    int32_t *tail_items = parts > 1 ? reinterpret_cast<int32_t *>(tail) : nullptr;
    schedule_kernel<<<1, kSchedThreads, 2 * bins * sizeof(int32_t), s>>>(q2k_num, NT, T, dims->max_kv, G, n_items,
                                                                        bins, split, parts, order, counter, tail_items,
                                                                        dc.steps_ptr.load(std::memory_order_acquire));
    if (cudaGetLastError() != cudaSuccess) return VSA_ERR_CUDA;

    AttnParams p;
    p.q2k_idx = q2k_idx;
    p.q2k_num = q2k_num;
    p.block_sizes = block_sizes;
    p.out = out;
    p.lse = lse;
    p.order = order;
    p.work_counter = counter;
    p.status = dc.status_ptr.load(std::memory_order_acquire);
    p.steps = dc.steps_ptr.load(std::memory_order_acquire);
    p.bm_global = bitmaps_in_workspace(dims)
                      ? reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(workspace) + bitmap_offset_for(dims))
                      : nullptr;
    p.NT = NT * sub;
    p.sub = sub;
    p.max_kv = dims->max_kv;
    p.G = G;
    p.bm_words = (NT * sub + 31) / 32;
    p.n_items = n_items - split + 2 * split * parts;
    p.n_parts = parts;
    p.tail_start = n_items - split;
    p.tail_ml = parts > 1 ? reinterpret_cast<float2 *>(tail + kTailCntBytes) : nullptr;
    p.tail_o = parts > 1 ? reinterpret_cast<float *>(tail + kTailCntBytes + kTailMlBytes) : nullptr;
    p.Sp = Sp;
    const float scale = dims->scale > 0.f ? dims->scale : 1.0f / std::sqrt((float)D);
    p.scale_log2 = scale * 1.4426950408889634f;
    if (launch_attn(Tk, D, paired, tm_q, tm_k, tm_v, p, grid, s) != cudaSuccess) return VSA_ERR_CUDA;
    if (parts > 1) {
        TailMergeParams mq;
        mq.tail_o = p.tail_o;
        mq.tail_ml = p.tail_ml;
        mq.tail_items = tail_items;
        mq.block_sizes = block_sizes;
        mq.out = out;
        mq.lse = lse;
        mq.units = 2 * split;
        mq.n_parts = parts;
        mq.G = G;
        mq.NT = NT * sub;
        mq.sub = sub;
        mq.Sp = Sp;
        if (launch_tail_merge(D, mq, s) != cudaSuccess) return VSA_ERR_CUDA;
    }

    const AttnLaunchInfo info = attn_launch_info(Tk, D, p.bm_global ? 0 : p.bm_words, paired);
    t_route.kernel = VSA_KERNEL_ATTN_TCGEN05;
    t_route.tile = T;
    t_route.head_dim = D;
    t_route.grid = grid;
    t_route.block = kAttnThreads;
    t_route.stages = info.stages;
    t_route.work_items = n_items;
    t_route.sort_bins = bins;
    t_route.smem_bytes = info.smem_bytes;
    t_route.layout = paired ? VSA_LAYOUT_PAIRED : VSA_LAYOUT_SPLIT;
    t_route.tail_parts = split > 0 ? parts : 0;
    return VSA_OK;
}

vsa_status vsa_tile_layout(const void *q_tok, const void *k_tok, const void *v_tok, void *q_tile, void *k_tile,
                           void *v_tile, const int32_t *row_to_token, int32_t B, int32_t S, int32_t H, int32_t D,
                           int32_t num_tiles, int32_t tile, vsa_stream_t stream) {
    if (!row_to_token || B <= 0 || S < 0 || H <= 0 || D <= 0 || (D % 8) != 0 || num_tiles <= 0 || tile <= 0)
        return VSA_ERR_ARG;
    const void *src[3] = {q_tok, k_tok, v_tok};
    void *dst[3] = {q_tile, k_tile, v_tile};
    LayoutParams p;
    p.n_tensors = 0;
    for (int i = 0; i < 3; ++i) {
        if ((src[i] == nullptr) != (dst[i] == nullptr)) return VSA_ERR_ARG;
        if (!src[i]) continue;
        if (!aligned(src[i], 16) || !aligned(dst[i], 16)) return VSA_ERR_ALIGN;
        p.src[p.n_tensors] = src[i];
        p.dst[p.n_tensors] = dst[i];
        ++p.n_tensors;
    }
    for (int i = p.n_tensors; i < 3; ++i) {
        p.src[i] = nullptr;
        p.dst[i] = nullptr;
    }
    if (p.n_tensors == 0) return VSA_ERR_ARG;
    if (!aligned(row_to_token, 4)) return VSA_ERR_ALIGN;
    if (B > 65535) return VSA_ERR_LIMITS;
    if ((int64_t)B * H > VSA_MAX_BATCH_HEADS) return VSA_ERR_LIMITS;
    const int64_t Sp = (int64_t)num_tiles * tile;
    if ((int64_t)B * H * Sp >= (int64_t(1) << VSA_MAX_ROWS_LOG2) || (int64_t)B * S * H >= (int64_t(1) << 31))
        return VSA_ERR_LIMITS;
    int dev = 0;
    vsa_status st = current_device(&dev);
    if (st != VSA_OK) return st;
    DeviceCache &dc = g_dev[dev];
    p.row_to_token = row_to_token;
    p.status = dc.status_ptr.load(std::memory_order_acquire);
    p.B = B;
    p.S = S;
    p.H = H;
    p.Dv = D / 8;
    p.Sp = Sp;
    if (launch_layout(p, dc.sm_count.load(std::memory_order_acquire), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return VSA_ERR_CUDA;
    t_route = vsa_route{};
    t_route.kernel = VSA_KERNEL_LAYOUT;
    t_route.tile = tile;
    t_route.head_dim = D;
    return VSA_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the backward, per (b, h) over NTk kernel tiles of 128 rows:
// [header | -delta | -lse*log2(e) | partner counts | partner lists |
//  transposed offsets | transposed lists].
struct BwdWs {
    BwdGeo geo;
    size_t delta, lse2, pc, pl, offs, list, total;
};

static BwdWs bwd_ws(const vsa_dims *d) {
    BwdWs w;
    w.geo = bwd_geo(d->tile, d->num_tiles, d->max_kv);
    const size_t BH = (size_t)d->B * d->H, NTk = (size_t)w.geo.NTk, Spk = NTk * 128;
    const size_t lists = 4 * BH * NTk * (size_t)w.geo.maxlen;
    w.delta = kWsHeader;
    w.lse2 = w.delta + align256(4 * BH * Spk);
    w.pc = w.lse2 + align256(4 * BH * Spk);
    w.pl = w.pc + align256(4 * BH * NTk);
    w.offs = w.pl + align256(lists);
    w.list = w.offs + align256(4 * BH * (NTk + 1));
    w.total = w.list + align256(lists);
    return w;
}

size_t vsa_block_sparse_bwd_workspace_size(const vsa_dims *dims) {
    if (check_dims_small(dims) != VSA_OK) return 0;
    return bwd_ws(dims).total;
}

vsa_status vsa_block_sparse_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
                                const float *lse, const int32_t *q2k_idx, const int32_t *q2k_num,
                                const int32_t *block_sizes, void *dq, void *dk, void *dv, const vsa_dims *dims,
                                void *workspace, size_t workspace_bytes, vsa_stream_t stream) {
    vsa_status st = check_dims_small(dims);
    if (st != VSA_OK) return st;
    if (!q || !k || !v || !out || !dout || !lse || !q2k_num || !block_sizes || !dq || !dk || !dv ||
        (!q2k_idx && dims->max_kv > 0))
        return VSA_ERR_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(dout, 16) ||
        !aligned(lse, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(q2k_num, 4) ||
        !aligned(block_sizes, 4) || (q2k_idx && !aligned(q2k_idx, 4)))
        return VSA_ERR_ALIGN;
    const BwdWs w = bwd_ws(dims);
    if (!workspace || workspace_bytes < w.total) return VSA_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return VSA_ERR_ALIGN;
    int dev = 0;
    if ((st = current_device(&dev)) != VSA_OK) return st;
    DeviceCache &dc = g_dev[dev];
    constexpr unsigned kBwdBit = 1u << 5;
    if (!(dc.attn_prepared.load(std::memory_order_acquire) & kBwdBit)) {
        if (bwd_prepare() != cudaSuccess) {
            cudaGetLastError();
            return VSA_ERR_CUDA;
        }
        dc.attn_prepared.fetch_or(kBwdBit, std::memory_order_acq_rel);
    }
    const int D = dims->head_dim, NT = dims->num_tiles;
    const int64_t Sp = (int64_t)NT * dims->tile;
    const int64_t rows = (int64_t)dims->B * dims->H * Sp;
    CUtensorMap tm_q, tm_k, tm_v, tm_do;
    if ((st = encode_rows_map(&tm_q, q, rows, D, 128)) != VSA_OK) return st;
    if ((st = encode_rows_map(&tm_k, k, rows, D, 128)) != VSA_OK) return st;
    if ((st = encode_rows_map(&tm_v, v, rows, D, 128)) != VSA_OK) return st;
    if ((st = encode_rows_map(&tm_do, dout, rows, D, 128)) != VSA_OK) return st;
    char *ws = reinterpret_cast<char *>(workspace);
    BwdLaunch L;
    L.tm_q = &tm_q;
    L.tm_k = &tm_k;
    L.tm_v = &tm_v;
    L.tm_do = &tm_do;
    L.out = out;
    L.dout = dout;
    L.lse = lse;
    L.ndelta = reinterpret_cast<float *>(ws + w.delta);
    L.nlse2 = reinterpret_cast<float *>(ws + w.lse2);
    L.q2k_idx = q2k_idx;
    L.q2k_num = q2k_num;
    L.block_sizes = block_sizes;
    L.pc = reinterpret_cast<int32_t *>(ws + w.pc);
    L.pl = reinterpret_cast<int32_t *>(ws + w.pl);
    L.k2q_offs = reinterpret_cast<int32_t *>(ws + w.offs);
    L.k2q_list = reinterpret_cast<int32_t *>(ws + w.list);
    L.dq = dq;
    L.dk = dk;
    L.dv = dv;
    L.status = dc.status_ptr.load(std::memory_order_acquire);
    L.BH = dims->B * dims->H;
    L.T = dims->tile;
    L.NTc = NT;
    L.NTk = w.geo.NTk;
    L.D = D;
    L.max_kv = dims->max_kv;
    L.maxlen = w.geo.maxlen;
    L.Sp = Sp;
    L.Spk = (int64_t)w.geo.NTk * 128;
    L.scale = dims->scale > 0.f ? dims->scale : 1.0f / std::sqrt((float)D);
    if (launch_bwd(L, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    t_route = vsa_route{};
    t_route.kernel = VSA_KERNEL_BWD;
    t_route.tile = dims->tile;
    t_route.head_dim = D;
    t_route.grid = (int32_t)((int64_t)L.BH * L.NTk);
    t_route.block = bwd_threads();
    t_route.work_items = (int64_t)L.BH * L.NTk;
    t_route.smem_bytes = (int32_t)bwd_smem_bytes(D);
    return VSA_OK;
}

vsa_status vsa_untile(const void *o_tile, const void *gate_tok, void *out_tok, const int32_t *row_to_token,
                      int32_t B, int32_t S, int32_t H, int32_t D, int32_t num_tiles, int32_t tile,
                      vsa_stream_t stream) {
    if (!o_tile || !out_tok || !row_to_token || B <= 0 || S < 0 || H <= 0 || D <= 0 || (D % 8) != 0 ||
        num_tiles <= 0 || tile <= 0)
        return VSA_ERR_ARG;
    if (!aligned(o_tile, 16) || !aligned(out_tok, 16) || (gate_tok && !aligned(gate_tok, 16)) ||
        !aligned(row_to_token, 4))
        return VSA_ERR_ALIGN;
    if ((int64_t)B * H > VSA_MAX_BATCH_HEADS) return VSA_ERR_LIMITS;
    const int64_t Sp = (int64_t)num_tiles * tile;
    if ((int64_t)B * H * Sp >= (int64_t(1) << VSA_MAX_ROWS_LOG2) || (int64_t)B * S * H >= (int64_t(1) << 31))
        return VSA_ERR_LIMITS;
    int dev = 0;
    vsa_status st = current_device(&dev);
    if (st != VSA_OK) return st;
    DeviceCache &dc = g_dev[dev];
    UntileParams p;
    p.o_tile = o_tile;
    p.gate = gate_tok;
    p.out = out_tok;
    p.row_to_token = row_to_token;
    p.status = dc.status_ptr.load(std::memory_order_acquire);
    p.B = B;
    p.S = S;
    p.H = H;
    p.Dv = D / 8;
    p.Sp = Sp;
    if (launch_untile(p, dc.sm_count.load(std::memory_order_acquire), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return VSA_ERR_CUDA;
    t_route = vsa_route{};
    t_route.kernel = VSA_KERNEL_UNTILE;
    t_route.tile = tile;
    t_route.head_dim = D;
    return VSA_OK;
}

vsa_status vsa_validate_indices(const int32_t *q2k_idx, const int32_t *q2k_num, const int32_t *block_sizes,
                                const vsa_dims *dims, int32_t *dev_status, vsa_stream_t stream) {
    vsa_status st = check_dims(dims);
    if (st != VSA_OK) return st;
    if (!q2k_num || !block_sizes || !dev_status || (!q2k_idx && dims->max_kv > 0)) return VSA_ERR_ARG;
    if (!aligned(q2k_num, 4) || !aligned(block_sizes, 4) || !aligned(dev_status, 4) ||
        (q2k_idx && !aligned(q2k_idx, 4)))
        return VSA_ERR_ALIGN;
    int dev = 0;
    if ((st = current_device(&dev)) != VSA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess) return VSA_ERR_CUDA;
    const int64_t n_rows = (int64_t)dims->B * dims->H * dims->num_tiles;
    const int64_t n = n_rows > dims->num_tiles ? n_rows : dims->num_tiles;
    const int threads = 256;
    validate_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(
        q2k_idx, q2k_num, block_sizes, n_rows, dims->num_tiles, dims->tile, dims->max_kv, dev_status);
    if (cudaGetLastError() != cudaSuccess) return VSA_ERR_CUDA;
    t_route = vsa_route{};
    t_route.kernel = VSA_KERNEL_VALIDATE;
    return VSA_OK;
}

size_t vsa_coarse_select_workspace_size(const vsa_dims *dims) {
    if (check_dims_small(dims) != VSA_OK) return 0;
    return 2 * (size_t)dims->B * dims->H * dims->num_tiles * dims->head_dim * sizeof(float);
}

vsa_status vsa_coarse_select(const void *q, const void *k, const int32_t *block_sizes, int32_t topk,
                             int32_t *q2k_idx, int32_t *q2k_num, const vsa_dims *dims, void *workspace,
                             size_t workspace_bytes, vsa_stream_t stream) {
    vsa_status st = check_dims_small(dims);
    if (st != VSA_OK) return st;
    if (!q || !k || !block_sizes || !q2k_num || topk < 0 || (!q2k_idx && topk > 0)) return VSA_ERR_ARG;
    if (topk > VSA_MAX_TILES_BWD) return VSA_ERR_LIMITS;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(block_sizes, 4) || !aligned(q2k_num, 4) ||
        (q2k_idx && !aligned(q2k_idx, 4)))
        return VSA_ERR_ALIGN;
    const size_t need = vsa_coarse_select_workspace_size(dims);
    if (!workspace || workspace_bytes < need) return VSA_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return VSA_ERR_ALIGN;
    int dev = 0;
    if ((st = current_device(&dev)) != VSA_OK) return st;
    DeviceCache &dc = g_dev[dev];
    constexpr unsigned kSelectBit = 1u << 4;
    if (!(dc.attn_prepared.load(std::memory_order_acquire) & kSelectBit)) {
        if (select_prepare() != cudaSuccess) {
            cudaGetLastError();
            return VSA_ERR_CUDA;
        }
        dc.attn_prepared.fetch_or(kSelectBit, std::memory_order_acq_rel);
    }
    SelectParams p;
    p.q = q;
    p.k = k;
    p.block_sizes = block_sizes;
    const size_t means = (size_t)dims->B * dims->H * dims->num_tiles * dims->head_dim;
    p.qm = reinterpret_cast<float *>(workspace);
    p.km = p.qm + means;
    p.q2k_idx = q2k_idx;
    p.q2k_num = q2k_num;
    p.status = dc.status_ptr.load(std::memory_order_acquire);
    p.B = dims->B;
    p.H = dims->H;
    p.NT = dims->num_tiles;
    p.T = dims->tile;
    p.D = dims->head_dim;
    p.topk = topk;
    if (launch_select(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    const int rows = select_rows(p.NT, p.D);
    t_route = vsa_route{};
    t_route.kernel = VSA_KERNEL_SELECT;
    t_route.tile = p.T;
    t_route.head_dim = p.D;
    t_route.grid = (p.NT + rows - 1) / rows * p.B * p.H;
    t_route.block = 32 * select_warps(p.NT, p.D);
    t_route.work_items = (int64_t)p.B * p.H * p.NT;
    t_route.smem_bytes = (int32_t)select_smem_bytes(p.NT, p.D, rows);
    return VSA_OK;
}

vsa_status vsa_wait_probe(int32_t arrive, uint32_t limit_us, vsa_stream_t stream) {
    if (limit_us < 1 || limit_us > 2000000u) return VSA_ERR_ARG;
    int dev = 0;
    vsa_status st = current_device(&dev);
    if (st != VSA_OK) return st;
    if (launch_wait_probe(arrive, (uint64_t)limit_us * 1000ull, g_dev[dev].status_ptr.load(std::memory_order_acquire),
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    return VSA_OK;
}

vsa_status vsa_check_device_status(vsa_stream_t stream) {
    int dev = 0;
    vsa_status st = current_device(&dev);
    if (st != VSA_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    int32_t word = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof word) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    if (word & kFlagTimeout) return VSA_ERR_TIMEOUT;
    if (word & kFlagIndex) return VSA_ERR_INDEX;
    return VSA_OK;
}

vsa_status vsa_last_route(vsa_route *route) {
    if (!route) return VSA_ERR_ARG;
    *route = t_route;
    return VSA_OK;
}

vsa_status vsa_last_step_counts(int64_t *tail_steps, int64_t *full_steps) {
    if (!tail_steps || !full_steps) return VSA_ERR_ARG;
    int dev = 0;
    vsa_status st = current_device(&dev);
    if (st != VSA_OK) return st;
    unsigned long long c[2] = {0ull, 0ull};
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpyFromSymbol(c, g_step_counts, sizeof c) != cudaSuccess) {
        cudaGetLastError();
        return VSA_ERR_CUDA;
    }
    *tail_steps = (int64_t)c[0];
    *full_steps = (int64_t)c[1];
    return VSA_OK;
}

}  // extern "C"
