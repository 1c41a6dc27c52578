/*
 * vsa.h -- C ABI of the GB300 (sm_103a) block-sparse attention library.
 *
 * The operation is the block-sparse attention forward pass of video sparse
 * attention as described on the FastVideo kernel page (hao-ai-lab/FastVideo
 * commit 8503617, fastvideo-kernel/python):
 *   - commit adding the sm_121a tile-128 forward: inputs q, k, v, q2k_idx,
 *     q2k_num, variable_block_sizes; output out; tiles of 64 or 128 tokens;
 *     each query tile attends only to the key tiles its selection lists;
 *   - sm_121a hardening commit: keys past a tile's valid count are masked,
 *     NaN/Inf padding never reaches the output, a query row with no keys is 0,
 *     a NaN softmax sum gives a NaN row; launch limits batch*heads <= 65535,
 *     rows < 2^31, tiles < 2^22, checked before launch; a GPU the kernel was
 *     not built for gets an error, never uninitialised output;
 *   - fused tile_to_bhsd commit: one pass that scatters token-major Q/K/V into
 *     tile-major BHSD;
 *   - Attn-QAT SM100 commit: the forward pass also yields softmax statistics
 *     (here the natural-log log-sum-exp of each query row).
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference after the call returns and allocates no device
 *     memory.  Scratch memory is passed in by the caller (workspace).
 *   - bf16 tensors are contiguous, 16-byte aligned.  Tile-major layout is
 *     [B, H, num_tiles*tile, head_dim]: row t*tile + r holds token r of tile t;
 *     rows r >= block_sizes[t] are padding and their contents are never read.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Argument, limit and architecture errors are returned
 *     synchronously before anything is launched.  Errors detected on the
 *     device (bad indices, a wait that timed out) are recorded in a device
 *     status word and reported by vsa_check_device_status().
 *   - Only GPUs of compute capability 10.3 (sm_103) are supported; any other
 *     device returns VSA_ERR_ARCH.
 */
#ifndef VSA_H
#define VSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *vsa_stream_t; /* same type as cudaStream_t */

typedef enum {
    VSA_OK = 0,
    VSA_ERR_ARG = -1,       /* null pointer, bad size, unsupported tile or head_dim */
    VSA_ERR_ALIGN = -2,     /* a pointer is not 16-byte aligned */
    VSA_ERR_LIMITS = -3,    /* a launch limit below is exceeded */
    VSA_ERR_ARCH = -4,      /* the current device is not sm_103 */
    VSA_ERR_CUDA = -5,      /* a CUDA runtime call or launch failed */
    VSA_ERR_TIMEOUT = -6,   /* a device-side wait gave up (reported later) */
    VSA_ERR_INDEX = -7,     /* bad q2k_idx / q2k_num / row map seen on the device */
    VSA_ERR_WORKSPACE = -8  /* workspace missing or smaller than required */
} vsa_status;

/* Launch limits, checked before any launch: the sm_121a hardening commit's
 * MaxBatchHeads, MaxRows and MaxTiles (within_launch_limits).  The tile limit
 * counts kernel tiles: a 256-token tile is two of them. */
#define VSA_MAX_BATCH_HEADS 65535
#define VSA_MAX_ROWS_LOG2 31              /* B*H*num_tiles*tile < 2^31 */
#define VSA_MAX_TILES ((1 << 22) - 1)     /* forward: kernel tiles < 2^22 */
/* The forward keeps each work item's selection bitmaps in shared memory up
 * to this many kernel tiles, and in a per-CTA region of the workspace beyond
 * (vsa_block_sparse_workspace_size counts it). */
#define VSA_SMEM_BITMAP_TILES 8192
/* The backward and the coarse selection: num_tiles <= 8192 (4096 with
 * 256-token tiles); their partner lists pack a tile index in 13 bits. */
#define VSA_MAX_TILES_BWD 8192

typedef struct {
    int32_t B;          /* batch */
    int32_t H;          /* heads */
    int32_t num_tiles;  /* tiles per sequence (NT) */
    int32_t tile;       /* tokens per tile: 64, 128 or 256 (256: the fused-layout
                           commit's training tiles; run as two 128-token halves) */
    int32_t head_dim;   /* 64 or 128 */
    int32_t max_kv;     /* row length of q2k_idx (>= 0) */
    float scale;        /* softmax scale; <= 0 selects 1/sqrt(head_dim) */
} vsa_dims;

/* Identifies the kernel that ran, for tests (route assertion). */
typedef struct {
    int32_t kernel;       /* VSA_KERNEL_* */
    int32_t tile;
    int32_t head_dim;
    int32_t grid;         /* CTAs launched (persistent) */
    int32_t block;        /* threads per CTA */
    int32_t stages;       /* K/V ring depth in shared memory */
    int64_t work_items;   /* 256-query-row work items scheduled */
    int32_t sort_bins;    /* bins of the on-device work ordering */
    int32_t smem_bytes;   /* dynamic shared memory per CTA */
    int32_t layout;       /* VSA_LAYOUT_*: the attention kernel's form, sparse or dense
                             (results agree within the stated tolerance) */
    int32_t tail_parts;   /* 0: no split tail; else the key-tile ranges each one-unit
                             entry of the split last wave was cut into (1: not cut) */
} vsa_route;

/* Attention kernel forms (vsa_route.layout).  SPLIT, the sparse form: one
   thread issues every S = Q K^T, one thread per 128-row query unit its P V,
   and the K/V ring holds one key tile per entry.  PAIRED, the dense form:
   with 128-token kernel tiles and head_dim 128, one thread per unit issues
   both of its products (bit-identical to SPLIT); with 64-token tiles, a ring
   entry holds a pair of key tiles so S is 128 keys wide (within the stated
   tolerance of SPLIT: the running maximum advances per entry).  Chosen from
   vsa_dims: PAIRED when the selection bitmaps fit shared memory
   (VSA_SMEM_BITMAP_TILES) and either tile == 256 with head_dim == 128, or
   max_kv >= num_tiles with tile == 64, or with tile == 128 and
   head_dim == 128. */
#define VSA_LAYOUT_SPLIT 0
#define VSA_LAYOUT_PAIRED 1

#define VSA_KERNEL_NONE 0
#define VSA_KERNEL_ATTN_TCGEN05 1
#define VSA_KERNEL_LAYOUT 2
#define VSA_KERNEL_VALIDATE 3
#define VSA_KERNEL_SELECT 4
#define VSA_KERNEL_UNTILE 5
#define VSA_KERNEL_BWD 6

/* Bytes of workspace vsa_block_sparse_fwd should get for `dims`: the
 * on-device work order and its counter, the selection bitmaps beyond
 * VSA_SMEM_BITMAP_TILES kernel tiles, and, beyond 128 work items of 256 query
 * rows, room for the split tail's partial results (256 x 128 rows of fp32 O
 * plus row maximum and sum, about 17 MB at head_dim 128).  Returns 0 when
 * `dims` is invalid.
 *
 * Split tail: when the last wave of work items would fill at most half of the
 * SMs, each of its items runs as two one-unit (128-row) entries, and with
 * 128-token kernel tiles each of those is cut into up to 8 ranges of key
 * tiles on separate SMs; every range leaves its unnormalised O, row maximum
 * and row sum in the workspace, and a small merge kernel on the same stream
 * combines them in a fixed order, so results stay deterministic. */
size_t vsa_block_sparse_workspace_size(const vsa_dims *dims);

/* The least workspace vsa_block_sparse_fwd accepts for `dims` (no room for
 * the split tail's partial results: the last wave then runs its one-unit
 * entries whole).  Returns 0 when `dims` is invalid. */
size_t vsa_block_sparse_workspace_size_min(const vsa_dims *dims);

/*
 * Block-sparse attention forward (commit adding the sm_121a tile-128
 * forward; sm_121a hardening commit for the masking and NaN rules).
 *
 *   q, k, v      bf16 [B, H, NT*tile, D] tile-major, read only
 *   q2k_idx      int32 [B, H, NT, max_kv]; entries [0, q2k_num) of each row are
 *                the selected key tiles, distinct, in [0, NT); order is free
 *   q2k_num      int32 [B, H, NT], each in [0, max_kv]
 *   block_sizes  int32 [NT], each in [0, tile]: valid tokens of each tile
 *                (shared by queries and keys; Sq == Sk)
 *   out          bf16 [B, H, NT*tile, D]: for a valid query row r < n_t,
 *                softmax(scale * q_r . K_L^T) V_L over the valid rows L of the
 *                selected key tiles; +0 when L is empty; a NaN softmax sum
 *                gives a NaN row; padding rows r >= n_t are written as +0.
 *   lse          NULL, or fp32 [B, H, NT*tile]: natural-log log-sum-exp of the
 *                scaled scores per row; -inf for padding rows and empty rows.
 *   workspace    device scratch of vsa_block_sparse_workspace_size(dims) bytes
 *                (at least vsa_block_sparse_workspace_size_min(dims)),
 *                16-byte aligned; contents need not be initialised; must not
 *                be used by another call that runs concurrently.
 *
 * Out-of-range or repeated indices and out-of-range counts never fault: they
 * are skipped / clamped and flagged as VSA_ERR_INDEX in the device status
 * word.  Use vsa_validate_indices() to check a selection up front.
 * With tile == 64, two tiles share one 128-row MMA; a product with a key tile
 * that only one of them selects leaves the other's rows out entirely, so NaN
 * or Inf in a valid row reaches only the tiles that select it.
 */
vsa_status vsa_block_sparse_fwd(const void *q, const void *k, const void *v, const int32_t *q2k_idx,
                                const int32_t *q2k_num, const int32_t *block_sizes, void *out,
                                float *lse, const vsa_dims *dims, void *workspace,
                                size_t workspace_bytes, vsa_stream_t stream);

/*
 * Block-sparse attention forward for callers that cannot allocate device
 * memory.  The paper has no counterpart to this entry point; it exists for
 * this library's users.
 *
 * Same arguments, layouts and results as vsa_block_sparse_fwd, without the
 * workspace: the scratch it needs lives in a fixed array inside the library
 * (VSA_NOALLOC_SCRATCH_BYTES bytes of device memory, held by every GPU that
 * loads the library until the process exits).  Useful where cudaMalloc is not
 * available to the caller -- host callbacks, plug-ins whose device memory is
 * owned by a host framework, or code that must keep a fixed footprint.
 *
 *   - Problems needing more scratch than the array holds return
 *     VSA_ERR_LIMITS before anything is launched.  The scratch of a problem is
 *     vsa_block_sparse_workspace_size_min(): a 256-byte header plus 4 bytes
 *     per work item (256 query rows of one (batch, head)) and 4 bytes for each
 *     of up to 256 split entries, so at most
 *     (VSA_NOALLOC_SCRATCH_BYTES - 256) / 4 - 256 = 261,824 work items fit.
 *     The array has no room for the split tail's partial results, so a last
 *     wave runs its one-unit entries whole.
 *   - The first call on a device looks up the array's device address; make
 *     that first call before any stream capture on the device.  The address
 *     belongs to the device's current context: after cudaDeviceReset (a new
 *     context) the next call looks it up again, so that call too must come
 *     before any capture.
 *   - Calls allocate nothing (no cudaMalloc / cudaFree).  Every call on a
 *     device shares the one array: calls that may run concurrently on the GPU
 *     race on it and must be ordered by the caller (one stream, or events).
 *     Each call rewrites the array's contents before use, so results never
 *     depend on an earlier call.
 */
#define VSA_NOALLOC_SCRATCH_BYTES (1u << 20)

vsa_status vsa_block_sparse_fwd_noalloc(const void *q, const void *k, const void *v,
                                        const int32_t *q2k_idx, const int32_t *q2k_num,
                                        const int32_t *block_sizes, void *out, float *lse,
                                        const vsa_dims *dims, vsa_stream_t stream);

/*
 * Fused tile layout (fused tile_to_bhsd commit): one pass over up to three
 * tensors that gathers token-major rows into tile-major order.
 *
 *   x_tok        bf16 [B, S, H, D] token-major (q, k, v; a pair may be NULL/NULL)
 *   x_tile       bf16 [B, H, NT*tile, D] tile-major output
 *   row_to_token int32 [NT*tile]: source token of every tile-major row, or -1
 *                for a padding row, which is written as +0.  A value outside
 *                [-1, S) writes +0 and flags VSA_ERR_INDEX on the device.
 *   D            head_dim, a multiple of 8 (16-byte rows)
 */
vsa_status vsa_tile_layout(const void *q_tok, const void *k_tok, const void *v_tok, void *q_tile,
                           void *k_tile, void *v_tile, const int32_t *row_to_token, int32_t B,
                           int32_t S, int32_t H, int32_t D, int32_t num_tiles, int32_t tile,
                           vsa_stream_t stream);

/*
 * Block-sparse attention backward (the Attn-QAT SM100 commit names the
 * backward pass and its dQ / dK-dV tiles; the gradients are those of
 * vsa_block_sparse_fwd).  With p = exp(scale * q.k - lse) over the valid rows
 * of the selected key tiles and delta = rowsum(dout * out):
 *   dv_k = sum_i p_ik dout_i,   ds_ik = p_ik (dout_i.v_k - delta_i),
 *   dq_i = scale * sum_k ds_ik k_k,   dk_k = scale * sum_i ds_ik q_i.
 * Rows with no keys get dq = 0, keys no row selects get dk = dv = 0, padding
 * rows are +0; a NaN row of the forward gives NaN gradients on its keys.
 *
 *   q, k, v, out, dout  bf16 [B, H, NT*tile, D] tile-major (out and lse as
 *                       vsa_block_sparse_fwd wrote them; lse is required)
 *   q2k_idx, q2k_num, block_sizes  the forward's selection (distinct,
 *                       in-range tiles; out-of-range entries are skipped and
 *                       flagged, a repeated one counts once)
 *   dq, dk, dv          bf16 [B, H, NT*tile, D] outputs, written completely
 *   dims                tile 64, 128 or 256; head_dim 64 or 128
 *   workspace           vsa_block_sparse_bwd_workspace_size(dims) bytes
 *                       (0 for invalid dims)
 * The kernels work on 128-row tiles: a 256-token tile as two halves, two
 * 64-token tiles together with a mask of which 64 x 64 blocks are selected.
 * Accumulations over a 64 x 64 block the selection leaves out do not touch
 * the rows of that block at all, so, as in the forward, NaN or Inf in a valid
 * row reaches only the gradients the definition sends it to.
 * Deterministic: dQ is recomputed per query tile instead of accumulated with
 * atomics, and dK/dV sum their query tiles in ascending order.
 */
size_t vsa_block_sparse_bwd_workspace_size(const vsa_dims *dims);

vsa_status vsa_block_sparse_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
                                const float *lse, const int32_t *q2k_idx, const int32_t *q2k_num,
                                const int32_t *block_sizes, void *dq, void *dk, void *dv, const vsa_dims *dims,
                                void *workspace, size_t workspace_bytes, vsa_stream_t stream);

/*
 * Output un-tiling with the gate, the inverse of vsa_tile_layout (the fused
 * tile_to_bhsd commit describes the layer's tiled path: Q, K, V and the gate
 * go into a tile buffer; this is the step back).  For every tile-major row r
 * with a token s = row_to_token[r] >= 0:
 *   out_tok[b, s, h, :] = bf16( float(o_tile[b, h, r, :]) * float(gate[b, s, h, :]) )
 * or a plain copy of the row when gate_tok is NULL.  The product of two bf16
 * values is exact in fp32, so the result is rounded once, to nearest even.
 * Padding rows are not read; tokens that no row maps to are not written.
 *
 *   o_tile       bf16 [B, H, NT*tile, D] tile-major (the forward's output)
 *   gate_tok     NULL, or bf16 [B, S, H, D] token-major gate
 *   out_tok      bf16 [B, S, H, D] token-major output
 *   row_to_token int32 [NT*tile], the map vsa_tile_layout used; a value
 *                outside [-1, S) skips the row and flags VSA_ERR_INDEX
 *   D            head_dim, a multiple of 8 (16-byte rows)
 */
vsa_status vsa_untile(const void *o_tile, const void *gate_tok, void *out_tok, const int32_t *row_to_token,
                      int32_t B, int32_t S, int32_t H, int32_t D, int32_t num_tiles, int32_t tile,
                      vsa_stream_t stream);

/*
 * Opt-in selection check (sm_121a hardening commit, launch-limit and
 * fail-closed items).  Writes to *dev_status (a device int32): 0 when every
 * q2k_num is in [0, max_kv], every live index is in [0, NT) and distinct within
 * its row, and every block size is in [0, tile]; VSA_ERR_INDEX otherwise.
 * Asynchronous; never traps.
 */
vsa_status vsa_validate_indices(const int32_t *q2k_idx, const int32_t *q2k_num,
                                const int32_t *block_sizes, const vsa_dims *dims,
                                int32_t *dev_status, vsa_stream_t stream);

/*
 * Coarse key-tile selection: produces the q2k_idx / q2k_num that
 * vsa_block_sparse_fwd consumes.  The FastVideo kernel page names video
 * sparse attention and its block-sparse fine stage (commit adding the sm_121a
 * tile-128 forward; "Wan VSA inference" in the fused tile_to_bhsd commit) but
 * not the coarse stage's arithmetic; this is its plain reading:
 *   1. every non-empty tile t is pooled to the mean of its valid rows
 *      (rows r < block_sizes[t] of q and of k; padding rows are never read);
 *   2. query tile t scores key tile j by the dot product of the two means;
 *   3. query tile t keeps the topk key tiles with the largest scores (ties to
 *      the smaller index), never an empty key tile or a NaN score; fewer if
 *      fewer qualify; none for an empty query tile.
 * The kept set is decided in fp32 with a fixed arithmetic -- each mean summed
 * over rows in order then divided once, each score summed over d in order of
 * fused multiply-adds -- so it is reproducible bit for bit.
 *
 *   q, k         bf16 [B, H, NT*tile, D] tile-major (the attention inputs)
 *   block_sizes  int32 [NT], each in [0, tile]; a size outside that range
 *                is never read past the tile, makes the tile unselectable and
 *                flags VSA_ERR_INDEX in the device status word
 *   topk         kept tiles per query tile, 0 <= topk <= VSA_MAX_TILES_BWD
 *   q2k_idx      int32 [B, H, NT, topk] out: kept tiles in ascending order,
 *                -1 after the last one (may be NULL when topk == 0)
 *   q2k_num      int32 [B, H, NT] out: number kept
 *   dims         B, H, num_tiles, tile, head_dim as for the forward pass
 *                (max_kv and scale are not used)
 *   workspace    vsa_coarse_select_workspace_size(dims) bytes of device
 *                scratch (the fp32 tile means), 16-byte aligned
 * The outputs feed vsa_block_sparse_fwd directly with max_kv = topk.
 */
size_t vsa_coarse_select_workspace_size(const vsa_dims *dims);

vsa_status vsa_coarse_select(const void *q, const void *k, const int32_t *block_sizes, int32_t topk,
                             int32_t *q2k_idx, int32_t *q2k_num, const vsa_dims *dims, void *workspace,
                             size_t workspace_bytes, vsa_stream_t stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * word: VSA_OK, VSA_ERR_INDEX or VSA_ERR_TIMEOUT (the most severe seen since
 * the last check). */
vsa_status vsa_check_device_status(vsa_stream_t stream);

/*
 * Probe of the failure path behind VSA_ERR_TIMEOUT (sm_121a hardening commit:
 * failures are reported, never left as a hung GPU).  Launches one warp that
 * waits, with the same bounded wait every kernel uses, on a barrier phase
 * that completes only when `arrive` is nonzero.  With arrive == 0 nothing
 * completes it: after limit_us microseconds the wait gives up, sets
 * VSA_ERR_TIMEOUT in the device status word (read it with
 * vsa_check_device_status) and the kernel returns; the context stays usable.
 *   arrive     nonzero: the phase completes and the status word is untouched
 *   limit_us   1 .. 2000000 (the kernels' own limit is about 2 s)
 * Returns VSA_ERR_ARG for a limit outside that range; asynchronous otherwise.
 */
vsa_status vsa_wait_probe(int32_t arrive, uint32_t limit_us, vsa_stream_t stream);

/* Route of the last successful launch on the calling host thread. */
vsa_status vsa_last_route(vsa_route *route);

/*
 * Key-tile steps of the last vsa_block_sparse_fwd (or _noalloc) call on the
 * current device, for route assertions in tests (the sm_121a hardening commit:
 * tests assert which route ran; the Attn-QAT SM100 commit: full key tiles run
 * unmasked, the tail tile in a separate masked step).  A step is one query
 * tile of the kernel (64 or 128 tokens; a 128-token half of a 256-token tile)
 * against one selected key tile (likewise) with at least one valid key.
 *   tail_steps  steps whose key tile holds fewer valid keys than the tile:
 *               the softmax masks the columns past the valid count and P V
 *               reads only the 16-key blocks holding valid keys
 *   full_steps  steps with a full key tile: no mask at all
 * The counts are made on the device (zeroed by the call's ordering kernel,
 * added to by the attention kernel), so this call waits for the device to
 * finish (cudaDeviceSynchronize): not for use inside stream capture.  Calls
 * that overlap on the GPU add to the same counts.
 */
vsa_status vsa_last_step_counts(int64_t *tail_steps, int64_t *full_steps);

/* Static description of a status code. */
const char *vsa_status_string(vsa_status status);

/* Library ABI version (major*1000 + minor). */
int32_t vsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VSA_H */
