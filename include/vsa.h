/*
 * vsa.h -- C ABI of the GB300 (sm_103a) VSA library: the coarse-to-fine
 * block-sparse video attention of "VSA: Accelerating Video Diffusion Inference
 * with Sparse Attention on AMD GPUs" (ROCm blog; cited below as [AMD] with the
 * section name) and of "VSA: Faster Video Diffusion with Trainable Sparse
 * Attention" (Abstract; cited as [ABS]).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers are DEVICE pointers unless stated otherwise, owned by the
 *    caller.  The library never allocates or frees memory; scratch space is a
 *    caller-provided workspace whose size the *_workspace_bytes queries give.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call only enqueues work on that stream and returns; results are
 *    ready when the stream reaches that point.
 *  - Q, K, V (and gates, dO) are bf16, contiguous [B, heads, N, d] with
 *    N = T*H*W tokens in native (t, h, w) raster order, token n = (t*H+h)*W+w,
 *    unless a function says it takes the "cube order" (after vsa_permute).
 *  - Cubes are (Ct, Ch, Cw) = (4, 4, 4) = 64 tokens ([AMD] "Stage 1: Coarse
 *    Selection"): Nc = ceil(T/4) * ceil(H/4) * ceil(W/4) cubes.  A side that
 *    is not a multiple of 4 ends in partial cubes: the cube keeps its 64
 *    slots in cube order, and the slots whose token would fall outside the
 *    grid are padding -- zero in cube-order tensors, left out of the cube's
 *    mean (which divides by the cube's token count), masked out of the keys
 *    by vsa_forward, and never written back to native order.  Cube-order
 *    tensors are [BH, Np, d] with Np = 64 * Nc (= N when 4 divides T, H, W).
 *  - d (head dim) must be 64 or 128.
 *  - Cube order: the 3D space-filling-curve reordering of [AMD] "Two-Stage
 *    Architecture".  By default cube-raster order: cube c = ((t/4)*Hc +
 *    h/4)*Wc + w/4 with Hc = ceil(H/4), Wc = ceil(W/4), offset
 *    o = ((t%4)*4 + h%4)*4 + w%4, position 64c + o; vsa_cube_order gives the
 *    Hilbert order instead.
 *  - Block index list ("LUT", [AMD] "Block-Sparse Encoding" and "Using VSA
 *    with CK Tile"): kv_block_idx int32 [BH, Nc, max_kv_blocks] holds the key
 *    cubes each query cube attends to; valid_block_num int32 [BH, Nc] holds how
 *    many entries of each row are used (0 <= count <= max_kv_blocks).
 *    vsa_coarse_topk writes rows in descending coarse score, ties to the lower
 *    cube id; vsa_forward saves the same sets in ascending cube id (the fine
 *    kernels walk a row as a set, so its order changes no result).  Entries
 *    are used as given (a repeated cube counts twice).
 *  - Output dtype selectors take VSA_DTYPE_BF16 or VSA_DTYPE_F32.
 *  - Return value: VSA_OK, or a negative vsa_status_t.  Argument and shape
 *    errors are found on the host before anything is enqueued.  Errors found
 *    by a kernel while it runs (an index outside [0, Nc), a count above
 *    max_kv_blocks, a bounded wait that expired) are latched in a device-side
 *    flag: the offending entry is skipped, and vsa_device_status() reports
 *    and clears the flag.
 *  - Precision: the pooled vectors, coarse scores and Top-K are fp32; the
 *    fine-stage tensor-core products take 16-bit operands with fp32
 *    accumulation.  vsa_forward / vsa_backward / vsa_fine_bwd, and
 *    vsa_fine_fwd given a workspace, convert Q, K, V and dO_f = g_fine * dO
 *    to fp16 (exact for bf16 values of magnitude up to 65504; 8x finer
 *    rounding of the probabilities and of dS than bf16).  An operand beyond
 *    65504 is saturated and latches VSA_ERR_RANGE.  vsa_fine_fwd without a
 *    workspace multiplies Q K^T in bf16 and P V in fp16 (V converted on
 *    chip); vsa_forward_inference both in bf16 (P rounded to bf16: it feeds
 *    no backward).
 */
#ifndef VSA_H_
#define VSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    VSA_OK = 0,
    VSA_ERR_ARG = -1,         /* null pointer, bad enum, non-positive size */
    VSA_ERR_SHAPE = -2,       /* N not a multiple of 64 where cube order is taken */
    VSA_ERR_UNSUPPORTED = -3, /* d not in {64,128}, cube shape not (4,4,4) */
    VSA_ERR_CUDA = -4,        /* a CUDA runtime call failed */
    VSA_ERR_TIMEOUT = -5,     /* a kernel's bounded wait expired */
    VSA_ERR_LUT = -6,         /* index list entry or count out of range */
    VSA_ERR_WORKSPACE = -7,   /* workspace missing or too small */
    VSA_ERR_RANGE = -8        /* an operand exceeded the fp16 range (see below) */
} vsa_status_t;

typedef enum { VSA_DTYPE_BF16 = 0, VSA_DTYPE_F32 = 1 } vsa_dtype_t;

/* Latent video grid and cube shape.  ct = ch = cw = 4 only.
 * cube_order: NULL for cube-raster order, or a device table written by
 * vsa_cube_order for this grid (it must stay valid while calls that take the
 * grid run); it fixes which cube sits at which position of the sequence. */
typedef struct {
    int T, H, W;
    int ct, ch, cw;
    const int32_t* cube_order;
} vsa_grid_t;

/* Cube orders of vsa_cube_order. */
enum { VSA_CURVE_RASTER = 0, VSA_CURVE_HILBERT = 1 };

/*
 * vsa_cube_order -- the order of the cubes along the 3D space-filling curve.
 * [AMD] "Two-Stage Architecture", pre-stage: tokens are reordered along a 3D
 * space-filling curve so that each block of the sequence is a compact
 * spatio-temporal region; the page names the curve (Jenga's) but does not
 * print it.
 *   g       the grid (g.cube_order is ignored).
 *   curve   VSA_CURVE_RASTER: cube (ct, ch, cw) at position
 *           (ct * H/4 + ch) * W/4 + cw.
 *           VSA_CURVE_HILBERT: cubes in the order in which the 3-D Hilbert
 *           curve (J. Skilling, "Programming the Hilbert curve", 2004) of the
 *           smallest enclosing 2^b x 2^b x 2^b cube grid visits them, cells
 *           outside the grid skipped; the index bits interleave t, h, w with
 *           t the most significant.  Each side of the cube grid <= 1024.
 *   order   out int32 [2 * Nc], device: order[p] = raster id
 *           (ct * H/4 + ch) * W/4 + cw of the cube at position p, and
 *           order[Nc + r] = position of raster cube r.
 * Tokens inside a cube keep (t%4, h%4, w%4) raster order.  Pass the table as
 * g.cube_order to vsa_permute, vsa_forward, vsa_backward and
 * vsa_lut_add_neighbors; cube ids in index lists are then positions along the
 * curve (so Top-K ties go to the cube met first).  Asynchronous on stream.
 */
int vsa_cube_order(vsa_grid_t g, int curve, int32_t* order, void* stream);

/*
 * vsa_permute -- 3D space-filling-curve token reordering, with the cube
 * mean-pool fused.  [AMD] "Two-Stage Architecture" (pre-stage SFC reordering;
 * Stage 1 mean-pools each cube into one vector).
 *   x        bf16 native [BH, N, d] (inverse = 0) or cube order [BH, Np, d] (1).
 *   y        bf16 cube order [BH, Np, d], padding slots zero (inverse = 0), or
 *            native [BH, N, d] (inverse = 1).  Must not alias x.
 *   pooled   fp32 [BH, Nc, d] or NULL: with inverse = 0, the mean of the
 *            tokens of every cube.  Must be NULL when inverse = 1.
 */
int vsa_permute(const void* x, void* y, float* pooled, int BH, int d, vsa_grid_t g, int inverse, void* stream);

/*
 * vsa_coarse_topk -- coarse cube-to-cube attention and the per-query-cube
 * Top-K selection.  [AMD] "Stage 1: Coarse Selection" and "Generating Sparsity
 * Patterns" (scores of pooled Q against pooled K, torch.topk over the last
 * dimension); the coarse output of "Stage 2: Fine Computation" (global
 * context).  All arithmetic is fp32.
 *   qc, kc, vc  fp32 [BH, Nc, d] pooled Q, K, V (vc may be NULL when
 *               o_coarse is NULL).
 *   topk        1 <= topk <= Nc.
 *   scale       score scale (1/sqrt(d) for the SDPA one).
 *   o_coarse    fp32 [BH, Nc, d] or NULL: softmax(scale*Qc Kc^T) Vc.
 *   lse_coarse  fp32 [BH, Nc]: log-sum-exp of each score row; may be NULL
 *               only when o_coarse is NULL.
 *   kv_block_idx    int32 [BH, Nc, topk]: selected key cubes, highest first.
 *   valid_block_num int32 [BH, Nc] or NULL: set to topk.
 *   scores      fp32 [BH, Nc, Nc] or NULL: receives the scaled coarse scores
 *               too (for inspection; the computation does not need it).
 * No Nc x Nc matrix is needed: a CTA keeps the score rows of 16 query cubes
 * in shared memory while Kc streams through, takes each row's log-sum-exp
 * and Top-K there (one warp per row: radix selection, then the picks ranked),
 * and streams Vc through for O_c.  Limit (the rows must fit the 227 KB of
 * shared memory): Nc <= 2304 for d = 128, Nc <= 2944 for d = 64, else
 * VSA_ERR_UNSUPPORTED; vsa_forward has the same limit.
 */
int vsa_coarse_topk(const float* qc, const float* kc, const float* vc, int BH, int Nc, int d, int topk,
                    float scale, float* o_coarse, float* lse_coarse, int32_t* kv_block_idx,
                    int32_t* valid_block_num, float* scores, void* stream);

/*
 * vsa_fine_fwd -- fine token-level attention inside the listed cubes only,
 * online softmax.  [AMD] "Stage 2: Fine Computation", "Kernel Architecture"
 * (running max and sum), "Sparse Traversal" (the index-list loop).
 *   qp, kp, vp  bf16 [BH, N, d] in cube order.
 *   o_fine      [BH, N, d] in cube order, dtype o_dtype:
 *               O_f[i] = softmax_j(scale * q_i . k_j) v_j over the tokens j of
 *               the listed cubes of i's cube; rows of a query cube with count 0
 *               are 0.
 *   lse         fp32 [BH, N] or NULL: natural-log sum-exp of each row
 *               (-inf for count 0).
 *   ws          NULL, or a workspace of vsa_workspace_bytes(VSA_OP_FINE_FWD,
 *               ...) bytes (16-byte aligned).  With it the call copies Q, K, V
 *               to fp16 in one pass (as vsa_forward does: exact within
 *               +-65504, VSA_ERR_RANGE beyond) and pairs the query cubes of
 *               each 128-row tile by list overlap, then runs vsa_forward's
 *               fine kernel.  Without it the call allocates nothing: Q K^T
 *               takes the bf16 operands, V is converted on chip, and cubes
 *               2t, 2t + 1 share a tile (slower).
 */
int vsa_fine_fwd(const void* qp, const void* kp, const void* vp, const int32_t* kv_block_idx,
                 const int32_t* valid_block_num, int max_kv_blocks, int BH, int N, int d, float scale,
                 void* o_fine, int o_dtype, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * vsa_fine_bwd -- gradient of the fine stage.  [ABS] (VSA is trained end to
 * end as one differentiable operator); the index list is held constant.
 *   qp, kp, vp, kv_block_idx, valid_block_num, max_kv_blocks, scale: as in
 *               the forward call.
 *   o_fine      [BH, N, d] the forward output (dtype o_dtype), lse fp32 [BH, N].
 *   do_fine     bf16 [BH, N, d]: dL/dO_f in cube order.
 *   Every pointer 16-byte aligned (VSA_ERR_ARG otherwise).
 *   dq, dk, dv  fp32 [BH, N, d] in cube order (overwritten).
 *   ws          workspace of vsa_workspace_bytes(VSA_OP_FINE_BWD, ...) bytes:
 *               fp16 copies of Q, K, V, dO_f (one pass), the inverse lists,
 *               and the query-cube and key-cube pair plans (the tiles of the
 *               dQ and dK/dV kernels, paired by list overlap as in
 *               vsa_backward).
 * As in vsa_backward, the dK/dV kernel runs on the library's auxiliary
 * stream, forked from `stream` and joined back to it before the call's work
 * ends, beside the dQ kernel on `stream`.
 */
int vsa_fine_bwd(const void* qp, const void* kp, const void* vp, const void* o_fine, int o_dtype,
                 const float* lse, const void* do_fine, const int32_t* kv_block_idx,
                 const int32_t* valid_block_num, int max_kv_blocks, int BH, int N, int d, float scale,
                 float* dq, float* dk, float* dv, void* ws, size_t ws_bytes, void* stream);

/*
 * vsa_fine_bwd_noalloc -- vsa_fine_bwd without a caller workspace.  The
 * pages have no counterpart of this call; it exists for callers that cannot
 * give the library scratch memory: code inside a runtime or framework that
 * hands out device memory only through its own pool (or allows no new
 * allocations once running), and plain C callers that hold the inputs and
 * outputs but no allocator for a workspace.
 *   Arguments and results are those of vsa_fine_bwd, minus ws / ws_bytes.
 *   Scratch: a fixed device array of VSA_NOALLOC_SCRATCH_BYTES inside the
 *   library.  A device holds it from the first vsa_fine_bwd_noalloc call on
 *   that device until the process exits (from library load instead when
 *   CUDA_MODULE_LOADING=EAGER).  Problems whose vsa_fine_bwd workspace
 *   exceeds it are rejected with VSA_ERR_WORKSPACE before anything is
 *   enqueued: the limit is about BH * N <= 65000 query rows (for example 15
 *   heads of 4096 tokens at d = 128 and 16 listed cubes); use vsa_fine_bwd
 *   beyond it.
 *   The call allocates nothing.  Its first call on a device looks up the
 *   array's device address (cudaGetSymbolAddress) with that device current
 *   and keeps it for the life of the process; make that first call before
 *   any stream capture.  cudaDeviceReset destroys the array with the
 *   context, and the kept address then points at nothing: do not use this
 *   entry point on a device after resetting it.  All calls share the one
 *   array and leave their contents in it (the parts that must start at zero
 *   are cleared on the stream by each call): calls whose GPU work overlaps
 *   -- on different streams, or from different threads -- race with each
 *   other, so serialise them.
 */
#define VSA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int vsa_fine_bwd_noalloc(const void* qp, const void* kp, const void* vp, const void* o_fine, int o_dtype,
                         const float* lse, const void* do_fine, const int32_t* kv_block_idx,
                         const int32_t* valid_block_num, int max_kv_blocks, int BH, int N, int d, float scale,
                         float* dq, float* dk, float* dv, void* stream);

/*
 * vsa_forward -- the whole VSA forward pass: reorder + pool, coarse attention
 * + Top-K, fine block-sparse attention, gated combination, inverse reorder.
 * [AMD] "Two-Stage Architecture" end to end; the gated combination of the
 * coarse and fine outputs ("Stage 2: Fine Computation", "Algorithmic Design")
 * is read as out = g_coarse * O_c + g_fine * O_f elementwise, O_c broadcast to
 * the 64 tokens of its cube.
 *   q, k, v     bf16 [B, heads, N, d] native order.
 *   g_coarse, g_fine  bf16 [B, heads, N, d] native order, or NULL (= ones).
 *   topk        1 <= topk <= Nc: the Top-K of each coarse score row.
 *   radius      -1: the selection is the Top-K alone (rows in ascending
 *               cube id).  0..7: the Top-K united with every cube whose (t, h,
 *               w) cube coordinates each differ from the query cube's by at
 *               most radius (the query cube included) -- [AMD] "Comparison
 *               with Jenga", "Algorithmic Design": block selection as the union
 *               of an importance mask and an adjacency mask; the rows are then
 *               ascending with per-row counts, max_kv_blocks = min(Nc, topk +
 *               (2 radius + 1)^3) wide.  vsa_backward uses the same lists.
 *   scale       score scale for both stages (1/sqrt(d) for SDPA).
 *   out         [B, heads, N, d] native order, dtype out_dtype.
 *   ws          workspace of vsa_workspace_bytes(VSA_OP_FORWARD, ...) bytes.
 *               It holds everything vsa_backward needs (the saved state):
 *               keep it unchanged until the matching vsa_backward is done.
 */
int vsa_forward(const void* q, const void* k, const void* v, const void* g_coarse, const void* g_fine, int B,
                int heads, int d, vsa_grid_t g, int topk, int radius, float scale, void* out, int out_dtype, void* ws,
                size_t ws_bytes, void* stream);

/*
 * vsa_forward_inference -- the same output as vsa_forward, without the state
 * a backward pass needs.  The fine stage reads Q, K and V in their native
 * layout: each (4, 4, 4) cube is one 5-D TMA box of the [B*heads, T, H, W, d]
 * tensor (zeros where the box leaves the grid), so no reordered copy of Q, K,
 * V is written -- the permutation is folded into the TMA addressing; only the
 * cube means are computed in a separate pass.  Arguments as vsa_forward; ws is
 * vsa_workspace_bytes(VSA_OP_FORWARD_INFERENCE, ...) bytes of scratch.  The
 * fine products run in bf16 with the softmax weights rounded to bf16
 * (vsa_forward: fp16 copies and fp16 weights), so the two outputs agree to
 * that rounding, well within the parity tolerance.
 */
int vsa_forward_inference(const void* q, const void* k, const void* v, const void* g_coarse, const void* g_fine,
                          int B, int heads, int d, vsa_grid_t g, int topk, int radius, float scale, void* out,
                          int out_dtype, void* ws, size_t ws_bytes, void* stream);

/*
 * vsa_backward -- gradients of vsa_forward.  [ABS].
 *   fwd_ws      the workspace the forward call filled (read only).
 *   g_coarse, g_fine, B, heads, d, g, topk, radius, scale: the same as in the
 *               forward (the selection lists it saved are held constant).
 *   dout        bf16 [B, heads, N, d] native order: dL/dout.
 *   dq, dk, dv  [B, heads, N, d] native order, dtype grad_dtype.
 *   dg_coarse, dg_fine  [B, heads, N, d] native, dtype grad_dtype; may be NULL,
 *               and are ignored when the matching gate is NULL.
 *   ws          workspace of vsa_workspace_bytes(VSA_OP_BACKWARD, ...) bytes.
 * The fine backward kernels finish the gradients in their epilogues (the
 * backward of the mean pool and the inverse reorder), so dq, dk, dv are
 * written once, by them.  The dK/dV kernel runs on a library-owned stream of
 * the highest priority (one per device, created on first use), forked from
 * `stream` by an event at the start of the call and joined back into it at
 * the end; the dQ kernel runs on `stream` beside it.  To the caller this is ordinary stream-ordered work
 * (it also records into a CUDA graph).  Calls on one device that overlap in
 * time from several host threads take their turn at the fork.
 */
int vsa_backward(const void* fwd_ws, const void* g_coarse, const void* g_fine, const void* dout, int B,
                 int heads, int d, vsa_grid_t g, int topk, int radius, float scale, void* dq, void* dk, void* dv,
                 void* dg_coarse, void* dg_fine, int grad_dtype, void* ws, size_t ws_bytes, void* stream);

enum {
    VSA_OP_FORWARD = 0,
    VSA_OP_BACKWARD = 1,
    VSA_OP_FINE_BWD = 2,
    VSA_OP_FORWARD_INFERENCE = 3,
    VSA_OP_FINE_FWD = 4
};

/* Workspace bytes for an operation (0 on a bad argument); topk and radius as
 * in vsa_forward.  For VSA_OP_FINE_FWD and VSA_OP_FINE_BWD, B*heads is BH,
 * g gives N (its cube count times 64), topk is max_kv_blocks, and radius is
 * ignored. */
size_t vsa_workspace_bytes(int op, int B, int heads, int d, vsa_grid_t g, int topk, int radius);

/* Device pointers into a forward workspace (the saved state), for callers
 * that want the intermediate results. */
typedef struct {
    void* qp;          /* fp16 [BH, N, d] cube order */
    void* kp;
    void* vp;
    float* qc;         /* fp32 [BH, Nc, d] pooled */
    float* kc;
    float* vc;
    float* o_coarse;   /* fp32 [BH, Nc, d] */
    float* lse_coarse; /* fp32 [BH, Nc] */
    int32_t* kv_block_idx;    /* [BH, Nc, max_kv_blocks] the selection lists */
    int32_t* valid_block_num; /* [BH, Nc] */
    float* o_fine;     /* fp32 [BH, N, d] cube order */
    float* lse;        /* fp32 [BH, N] */
    int32_t* tile_pairs; /* [BH, (Nc + 1) / 2, 2] query cubes of each fine-kernel tile
                            (second -1: a lone cube); a scheduling choice, not a result */
    int max_kv_blocks;   /* width of the lists: topk, or min(Nc, topk + (2 radius + 1)^3) */
} vsa_saved_t;

int vsa_forward_saved(const void* fwd_ws, int B, int heads, int d, vsa_grid_t g, int topk, int radius,
                      vsa_saved_t* out);

/* Device pointer into a backward workspace after vsa_backward: the key-cube
 * pairs of the dK/dV kernel's tiles, int32 [BH, (Nc + 1) / 2, 2] (second -1:
 * a lone cube).  A scheduling choice, not a result: each tile computes dK and
 * dV of its two key cubes over the union of their inverse lists. */
int vsa_backward_tile_pairs(const void* bwd_ws, int B, int heads, int d, vsa_grid_t g, int topk, int radius,
                            int32_t** key_pairs);

/*
 * Kernel timing (instrumentation, off by default).  While enabled, every
 * launch of the kernels below is bracketed by a pair of CUDA events recorded
 * on the stream the kernel is launched on.  vsa_timing_read waits for the
 * recorded events of one kernel, returns the summed elapsed milliseconds and
 * the number of launches since the last read, and forgets them.
 */
enum {
    VSA_K_PERMUTE = 0,     /* reorder + pool (vsa_permute, vsa_forward) */
    VSA_K_COARSE = 1,      /* coarse attention + Top-K */
    VSA_K_FINE_FWD = 2,    /* tcgen05 fine forward */
    VSA_K_COMBINE = 3,     /* gated combine + inverse reorder */
    VSA_K_BWD_PREP = 4,    /* backward of the combine */
    VSA_K_COARSE_BWD = 5,  /* coarse backward (three kernels) */
    VSA_K_FINE_BWD = 6,    /* tcgen05 fine backward, dK/dV kernel */
    VSA_K_FINE_BWD_DQ = 7, /* tcgen05 fine backward, dQ kernel */
    VSA_K_COUNT = 8
};
int vsa_timing_enable(int on);
int vsa_timing_read(int kernel, double* total_ms, int* launches);

/* Waits for `stream`, then returns and clears the device-side error flag:
 * VSA_OK, VSA_ERR_LUT, VSA_ERR_TIMEOUT, VSA_ERR_RANGE, or VSA_ERR_ARG when a
 * coarse score was NaN (a non-finite input; the Top-K then ranks NaN above
 * every number) -- or VSA_ERR_CUDA. */
int vsa_device_status(void* stream);

/* Static description of a status code. */
const char* vsa_status_string(int status);

/*
 * vsa_mask_to_lut -- converts a block relation matrix into index lists.
 * [AMD] "Sparse Encoding in CK Tile": Jenga stores the full M x M one-hot
 * block matrix B, VSA the selected blocks of each query block plus a valid
 * count; this call turns the first form into the second, on the device.
 *   mask             uint8 [BH, Nc, Nc], row-major: nonzero = query cube i
 *                    attends to key cube j (i = row, j = column).
 *   max_kv_blocks    list length per row (>= 1).
 *   kv_block_idx     out int32 [BH, Nc, max_kv_blocks]: the kept key cubes of
 *                    each row in ascending id, then -1.
 *   valid_block_num  out int32 [BH, Nc]: the number kept (<= max_kv_blocks).
 * A row with more nonzero cells than max_kv_blocks keeps its lowest ids and
 * latches VSA_ERR_LUT (read with vsa_device_status).  Asynchronous on stream;
 * argument errors are returned before any launch.
 */
int vsa_mask_to_lut(const uint8_t* mask, int BH, int Nc, int max_kv_blocks, int32_t* kv_block_idx,
                    int32_t* valid_block_num, void* stream);

/*
 * vsa_lut_add_neighbors -- unites every row's list with its cube's spatial
 * neighbourhood.  [AMD] "Comparison with Jenga", "Algorithmic Design":
 * Jenga's block selection is the union of three masks, one of them spatial
 * adjacency; this adds that adjacency to a Top-K list.  Cube ids are
 * positions in the cube sequence of g (g.cube_order; with NULL the raster id
 * c = (t * Hc + h) * Wc + w on the cube grid (Tc, Hc, Wc) = (T/4, H/4, W/4));
 * neighbourhoods are taken on the grid coordinates.
 *   kv_block_idx_in, valid_block_num_in (may be NULL = max_kv_blocks_in),
 *   max_kv_blocks_in   the input lists [BH, Nc, max_kv_blocks_in].
 *   g                  the video grid (as in vsa_forward; 4 x 4 x 4 cubes).
 *   radius             0..7: cubes whose t, h and w cube coordinates each
 *                      differ from the query cube's by at most radius (the
 *                      query cube itself included) are added.
 *   max_kv_blocks_out  output list length; kv_block_idx_out int32
 *                      [BH, Nc, max_kv_blocks_out] ascending, then -1;
 *                      valid_block_num_out int32 [BH, Nc].
 * Overflow: as vsa_mask_to_lut.  Entries of the input outside [0, Nc) are
 * skipped and latch VSA_ERR_LUT.  Input and output must not overlap.
 */
int vsa_lut_add_neighbors(const int32_t* kv_block_idx_in, const int32_t* valid_block_num_in, int max_kv_blocks_in,
                          int BH, vsa_grid_t g, int radius, int max_kv_blocks_out, int32_t* kv_block_idx_out,
                          int32_t* valid_block_num_out, void* stream);

/*
 * vsa_selftest_wait_timeout -- exercises the failure path every kernel of
 * this library takes when a wait never completes (the pages have no
 * counterpart; this is the library's own failure detection).  Launches one
 * thread that waits, with the same bounded mbarrier wait the fine kernels
 * use, on a barrier nothing will complete; after `polls` polls it gives up,
 * latches the timeout bit and exits.  The GPU context stays usable:
 * vsa_device_status() then returns VSA_ERR_TIMEOUT (and clears it).
 *   polls  number of polls before giving up (1 .. 2^24; VSA_ERR_ARG otherwise).
 */
int vsa_selftest_wait_timeout(uint32_t polls, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VSA_H_ */
