/*
 * wsattn.h - C ABI of libwsattn: frame-aligned window-sparse attention for
 * NVIDIA GB300 (sm_103a).
 *
 * The method is the one the Google Developers Blog post "HeyGen x Google
 * Cloud: Bringing Avatar IV to TPUs" describes for the super-resolution
 * stage's sparse attention:
 *   - section "Deleting the mask" (Fig. 3): every frame's tokens attend a
 *     window of nearby frames plus one global reference frame; with block
 *     sizes that are multiples of 16 and divide the frame token span, every
 *     key block is either fully active or skipped, so the kernel needs no
 *     mask predicate, no padding and no second pass for the reference frame;
 *   - section "Breaking softmax's dependency chain" (Fig. 4): keys are
 *     mean-centered, each query row gets a Cauchy-Schwarz upper bound on its
 *     logits (its norm times the max key norm) that serves as a fixed softmax
 *     max, and heads whose bound is too loose fall back to the online-max
 *     path inside the same kernel.
 *
 * Conventions shared by every call
 *   - Token order: the R reference frames first, then video frames 0..F-1,
 *     each T tokens long; N = (R + F) * T.  Query token i attends key token j
 *     iff j lies in a reference frame, or i lies in a reference frame, or
 *     their video frames differ by at most `window`.
 *   - Tensors are row-major [batch, heads, N, head_dim], contiguous, in
 *     device memory owned by the caller, with 16-byte aligned base pointers.
 *     q, k, v are bf16 (passed as void*); out is fp32.
 *   - softmax scale = 1 / sqrt(head_dim).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); all device
 *     work is enqueued on it.  No call synchronises the host except the
 *     wsattn_get_* readers and wsattn_device_status, and the calls that grow
 *     a plan's workspace (the first call for a larger batch); each says so.
 *   - Every call returns a status code (WSATTN_OK = 0 or one of the errors
 *     below) and never throws or aborts.  Argument errors are reported before
 *     any work is enqueued.  Asynchronous device errors (CUDA faults, expired
 *     device-side waits) surface through wsattn_device_status or the next
 *     synchronising call.
 *   - A plan is not thread-safe; calls on one plan must be serialised by the
 *     caller.  Device buffers a plan owns live on the device that was current
 *     at its first device call.
 */
#ifndef WSATTN_H_
#define WSATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum wsattn_status {
  WSATTN_OK = 0,
  WSATTN_ERR_BAD_ARG = 1,        /* null/misaligned pointer, size out of range */
  WSATTN_ERR_BAD_BLOCK = 2,      /* block size not a multiple of 16 or not dividing T */
  WSATTN_ERR_UNSUPPORTED = 3,    /* head_dim or block_k outside what the kernels implement */
  WSATTN_ERR_NOT_PREPARED = 4,   /* wsattn_forward before any wsattn_prepare on the plan */
  WSATTN_ERR_BATCH_MISMATCH = 5, /* forward batch differs from the last prepare's */
  WSATTN_ERR_CUDA = 6,           /* a CUDA runtime call failed (launch, copy, alloc) */
  WSATTN_ERR_TIMEOUT = 7,        /* a device-side wait expired; results are invalid */
  WSATTN_ERR_NO_MEMORY = 8,      /* host allocation failed */
  WSATTN_ERR_BOUNDS = 9          /* debug build only: a device bounds check failed (the
                                    access was skipped); results are invalid */
};

typedef struct wsattn_plan_s* wsattn_plan_t;

/*
 * Builds the block map for one attention shape ("Deleting the mask", Fig. 3).
 * Host-only: allocates no device memory and needs no GPU.
 *   frames            F >= 1 video frames
 *   tokens_per_frame  T >= 16, a multiple of 16
 *   window            w >= 0; w >= F - 1 makes the mask dense
 *   ref_frames        R >= 0 global reference frames (prefix of the sequence)
 *   heads             H >= 1
 *   head_dim          D; the kernels implement 64 and 128
 *   block_q, block_k  block sizes of the map: multiples of 16 dividing T, or
 *                     0 to let the plan choose.  The forward kernel streams
 *                     keys in steps of floor(160 / block_k) consecutive
 *                     active blocks, so block_k must be <= 160 for
 *                     wsattn_forward; the automatic size is the valid size
 *                     (<= 160) whose step holds the most keys, the larger
 *                     size on ties.
 *   out               receives the plan handle (owned by the caller; release
 *                     with wsattn_plan_destroy).
 * Errors: BAD_ARG (sizes, null out), BAD_BLOCK, UNSUPPORTED (head_dim),
 *         NO_MEMORY.
 */
int wsattn_plan(int frames, int tokens_per_frame, int window, int ref_frames, int heads,
                int head_dim, int block_q, int block_k, wsattn_plan_t* out);

/* Variants of the mask family (or-ed into mask_flags; 0 = the mask described
 * at the top of this file).  Every variant keeps each frame's active key
 * blocks in at most two runs, so the same kernels run it unchanged. */
enum wsattn_mask_flags {
  WSATTN_MASK_CAUSAL = 1,     /* video frame f attends video frames f - w .. f only */
  WSATTN_MASK_REF_SUFFIX = 2, /* the R reference frames follow the F video frames */
  WSATTN_MASK_REF_LOCAL = 4   /* reference queries attend only reference keys */
};

/* wsattn_plan with a mask variant.  wsattn_plan(...) is
 * wsattn_plan_ex(..., 0, out).  With WSATTN_MASK_REF_SUFFIX the token order
 * is video frames 0..F-1, then the reference frames.
 * Errors: as wsattn_plan; BAD_ARG for unknown flag bits. */
int wsattn_plan_ex(int frames, int tokens_per_frame, int window, int ref_frames, int heads,
                   int head_dim, int block_q, int block_k, int mask_flags, wsattn_plan_t* out);

/* Releases the plan and every host and device buffer it owns.  The caller
 * must make sure no work that uses the plan is still running on the GPU.
 * NULL is accepted and ignored. */
int wsattn_plan_destroy(wsattn_plan_t plan);

/*
 * Fixed-max statistics ("Breaking softmax's dependency chain").  For every
 * (b, h), with scale = 1/sqrt(D):
 *   mu      = mean of the N keys (fp32, fixed reduction order);
 *   K_h     = max_j ||k_j - mu||, the max norm of the centered keys;
 *   b_i     = scale * ||q_i|| * K_h, row i's bound on its centered logits
 *             scale * q_i.(k_j - mu) (Cauchy-Schwarz);
 *   m_i     = b_i + scale * q_i.mu, the same bound on the logits of the keys
 *             as given: centering shifts every logit of row i by the same
 *             scale * q_i.mu, which the softmax does not see, so the forward
 *             multiplies the caller's keys unchanged and uses m_i as the
 *             row's fixed max;
 *   B_h     = max_i b_i;  eligible_h = (B_h <= tau) and (2 * B_h < 126 ln 2),
 *             tau = 40 unless overridden with wsattn_plan_set_debug.
 * q and k are read only.  The statistics live in a workspace the plan owns
 * (allocated on the first call, grown when batch grows; growing synchronises
 * `stream`).
 *   q  bf16 [batch, H, N, D]
 *   k  bf16 [batch, H, N, D]
 * Errors: BAD_ARG, CUDA.
 */
int wsattn_prepare(wsattn_plan_t plan, int batch, const void* q, const void* k, void* stream);

/*
 * Pre-attention producer with the statistics folded in (Google Developers
 * Blog post "HeyGen x Google Cloud: Bringing Avatar IV to TPUs", section
 * "Layout is ABI", Figure 5: normalisation, rotary embedding, projection and
 * head packing fused into one kernel that writes the attention's input
 * layout).  The pages name the ops only; this call takes, per token t of
 * every batch element:
 *   xh_t = x_t / sqrt(mean_c x_tc^2 + eps)   RMS normalisation, no gain (fold
 *                                           a gain into w_qkv's columns)
 *   y_t  = w_qkv xh_t                       projection, no bias; y_t holds
 *                                           the q features (head-major,
 *                                           dim-minor), then k, then v
 *   q, k: dims (2p, 2p+1) turn by the angle whose cosine and sine are
 *         rope_cos[t][p], rope_sin[t][p]: (a, b) -> (a c - b s, a s + b c);
 *         v is not turned
 *   q, k, v rounded to bf16 and written [batch, H, N, D]
 * and then computes the fixed-max statistics of wsattn_prepare for the q and
 * k it wrote (the key mean from column sums the projection kernel emits, so
 * k is not read back for it).  After it, wsattn_forward may run on q, k, v
 * with the same batch, as after wsattn_prepare.  The product W x_t runs on
 * the tensor cores in fp32; 1 / rms_t is applied to its fp32 result.
 *   x          bf16 [batch, N, model_dim]
 *   model_dim  C, a multiple of 64
 *   w_qkv      bf16 [3 * H * D, model_dim], row-major
 *   rope_cos   fp32 [N, D / 2] (the angle table: it encodes each token's
 *   rope_sin   fp32 [N, D / 2]  position; shared by the batch and the heads)
 *   eps        >= 0
 *   q, k, v    bf16 [batch, H, N, D] outputs, fully overwritten
 * Needs H * D to be a multiple of 128.  All pointers 16-byte aligned device
 * memory; x, w_qkv and the tables are read only.  The plan's workspace grows
 * as for wsattn_prepare.
 * Errors: BAD_ARG, UNSUPPORTED (H * D not a multiple of 128), CUDA.
 */
int wsattn_produce(wsattn_plan_t plan, int batch, const void* x, int model_dim,
                   const void* w_qkv, const float* rope_cos, const float* rope_sin, float eps,
                   void* q, void* k, void* v, void* stream);

/*
 * out = masked softmax(q k^T * scale) v, computed in one pass over the
 * plan's active key blocks by a persistent tcgen05 kernel: QK^T and PV on
 * the tensor cores (bf16 inputs, fp32 accumulation in tensor memory), the
 * row bound m_i as a fixed softmax max on eligible heads, the online max on
 * the others.  P is rounded to bf16 for the PV product ("Proving pixels
 * unchanged" moves the final attention matmul to bf16).
 *   q    bf16 [batch, H, N, D]
 *   k    bf16 [batch, H, N, D], the same keys wsattn_prepare saw
 *   v    bf16 [batch, H, N, D]
 *   out  fp32 [batch, H, N, D], fully overwritten
 * Requires a prior wsattn_prepare on this plan with the same batch.
 * Work items (a query tile of one head) are dealt out on the device, in
 * order of decreasing key-list length, to whichever CTA is free first, from
 * a counter the plan owns: two forwards of one plan must not run at the
 * same time on the device (on different streams without ordering).
 * Errors: BAD_ARG, NOT_PREPARED, BATCH_MISMATCH, UNSUPPORTED (block_k > 160),
 *         CUDA.
 */
int wsattn_forward(wsattn_plan_t plan, int batch, const void* q, const void* k, const void* v,
                   float* out, void* stream);

/*
 * No-allocation variant of wsattn_prepare.  The paper has no counterpart: it
 * exists for callers that must not let the library allocate device memory
 * (a host framework that owns all device memory through its own pool or a
 * fixed budget, or a latency-critical loop that cannot take cudaMalloc's
 * implicit synchronisation).  It computes, with no plan, into buffers the
 * caller owns, the statistics wsattn_prepare computes on a plan left at the
 * default global bound (WSATTN_BOUND_GLOBAL): window bounds and mask flags
 * do not apply.  It never calls cudaMalloc, cudaFree or any other
 * allocating routine.
 *   batch, heads, n_tokens, head_dim   shape of q and k ([batch, heads,
 *                     n_tokens, head_dim] bf16, 16-byte aligned); head_dim
 *                     64 or 128
 *   tau               eligibility threshold (> 0; the library default is 40)
 *   b_rows, m_rows    fp32 [batch*heads*n_tokens] outputs: b_i and m_i
 *   mu                fp32 [batch*heads*head_dim] output
 *   kmax, bmax        fp32 [batch*heads] outputs: K_h and B_h
 *   elig              uint8 [batch*heads] output
 * Its scratch is one fixed array in the library's device image: 2048 chunk
 * slots and 2048 per-head entries (1,081,344 bytes), held by every GPU that
 * loads the library until the process exits.  batch*heads above 2048 is
 * rejected with BAD_ARG before anything is enqueued (so is a row chunking
 * that would need more than the 2048 slots, which cannot happen on a GPU
 * with at most 512 SMs).  All calls share the array and it keeps the last
 * call's contents; the only part that must start at zero, the per-head
 * counters of finished chunks, is zero when the library loads and every
 * call leaves it at zero.  Calls whose kernels can overlap on the GPU race
 * on it and must be ordered by the caller.  The first call on a device looks up the array's device address
 * with that device current (so make it before any stream capture).
 * Errors: BAD_ARG, UNSUPPORTED (head_dim), CUDA.
 */
int wsattn_prepare_static(int batch, int heads, int n_tokens, int head_dim, float tau,
                          const void* q, const void* k, float* b_rows, float* m_rows, float* mu,
                          float* kmax, float* bmax, uint8_t* elig, void* stream);

/* ---------------------------------------------------------- introspection */

/* Plan geometry.  info[0..9] = N, block_q, block_k, q blocks, k blocks,
 * active blocks (CSR nnz), work tiles per (b, h) (128-row query tiles,
 * with consecutive frames' short tails merged; see wsattn_get_tiles),
 * head_dim, heads, active (query, key) element pairs per (b, h).  n is the
 * capacity of info; at most n entries are written. */
int wsattn_plan_info(wsattn_plan_t plan, int64_t* info, int n);

/* Copies the forward work list (in its execution order) into host memory:
 * 10 int32 per tile, {row0, nvalid, nblk, run0, len0, run1, nstep, kbeg,
 * gsz, gtab}, and the group table of the merged tail tiles, 4 int32 per
 * row group {run0, len0, run1, len1}.  Key runs are in units of block_k.
 * Rows are query tokens within a head.  A tile with gsz = 0 covers tokens
 * [row0, row0 + nvalid) of one frame, with that frame's key blocks: run0 ..
 * run0 + len0 - 1, then run1 .. run1 + nblk - len0 - 1.
 * Frames whose token span T is not a multiple of 128 end in a short tail
 * tile.  A tile with gsz > 0 merges consecutive frames' tails ("Deleting the
 * mask" of the Google Developers Blog post "HeyGen x Google Cloud: Bringing
 * Avatar IV to TPUs" streams only active key blocks; merging the tails keeps
 * a frame's short last tile from costing a whole tile's key steps):
 *   - its row group i holds tile rows [i*gsz, (i+1)*gsz), which are tokens
 *     row0 + i*T .. row0 + i*T + gsz - 1;
 *   - the tile walks the union of the groups' key blocks;
 *   - group i's own blocks are entry gtab + i of the group table.
 * n_tiles and n_groups are capacities in int32 (n_tiles >= 10 x work
 * tiles per (b, h) from wsattn_plan_info; n_groups >= 4 x row groups; both
 * pointers may be NULL when the count is zero).
 * Errors: BAD_ARG if a capacity is too small. */
int wsattn_get_tiles(wsattn_plan_t plan, int32_t* tiles, size_t n_tiles, int32_t* groups,
                     size_t n_groups);

/* Copies the block bitmap (row-major [N/block_q, N/block_k], 1 = active)
 * into host memory of n bytes.  Errors: BAD_ARG if n is too small. */
int wsattn_get_block_map(wsattn_plan_t plan, uint8_t* host, size_t n);

/* Copies the CSR of active blocks: row_ptr[N/block_q + 1], col[nnz] (key
 * block indices, increasing within a row), into host arrays of the given
 * capacities.  Errors: BAD_ARG if a capacity is too small. */
int wsattn_get_csr(wsattn_plan_t plan, int32_t* row_ptr, int32_t* col, size_t n_row_ptr,
                   size_t n_col);

/* Synchronises `stream`, then copies the statistics of the last prepare to
 * host memory: b_rows fp32 [batch*H*N] (b_i), m_rows fp32 [batch*H*N] (m_i),
 * mu fp32 [batch*H*D], kmax fp32 [batch*H] (K_h), bmax fp32 [batch*H] (B_h),
 * elig uint8 [batch*H].  Any pointer may be NULL to skip it.
 * Errors: NOT_PREPARED, CUDA. */
int wsattn_get_stats(wsattn_plan_t plan, float* b_rows, float* m_rows, float* mu, float* kmax,
                     float* bmax, uint8_t* elig, void* stream);

/* Test hook.  force_path: -1 = per-head eligibility (default), 0 = fixed max
 * on every head, 1 = online max on every head.  tau > 0 replaces the
 * eligibility threshold used by later prepares (40 by default). */
int wsattn_plan_set_debug(wsattn_plan_t plan, int force_path, float tau);

/* Key-norm maximum the row bounds use (see wsattn_plan_set_bound). */
enum wsattn_bound {
  WSATTN_BOUND_GLOBAL = 0, /* K_h = max over all N centered keys of the head (default) */
  WSATTN_BOUND_WINDOW = 1  /* K_h,a = max over the keys frame a attends */
};

/*
 * Selects the key-norm maximum of the row bounds for later prepares.  The
 * bound of the section "Breaking softmax's dependency chain" multiplies a
 * query's norm by the largest centered key norm; any key subset that
 * contains the row's active keys gives a valid bound, and the smallest one
 * is the row's own window:
 *   WSATTN_BOUND_GLOBAL  b_i = scale * ||q_i|| * max_j ||k_j - mu||  (all N keys)
 *   WSATTN_BOUND_WINDOW  b_i = scale * ||q_i|| * max_{j attended by i} ||k_j - mu||
 * Every query of a frame attends the same keys, so the window maximum is one
 * value per (b, h, query frame): the largest per-frame maximum over the
 * frames it attends.  m_i, B_h and eligibility follow from b_i as described
 * at wsattn_prepare; the window bound is never larger, so B_h can only fall
 * and heads can only become eligible.  Outputs are unchanged in exact
 * arithmetic.  In window mode wsattn_get_stats' kmax still reports the
 * global maximum of each head.  The plan must be prepared again before the
 * next forward.
 * Errors: BAD_ARG (unknown mode).
 */
int wsattn_plan_set_bound(wsattn_plan_t plan, int mode);

/* Synchronises `stream` and reports the plan's device status word: OK,
 * BOUNDS if a debug build's bounds check failed (see wsattn_build_flags), or
 * TIMEOUT if a device-side wait of a kernel launched with this plan expired
 * (the word is then cleared, and so are the plan's forward work counters,
 * which a forward that gave up may have left mid-count).  CUDA if the
 * synchronisation itself failed. */
int wsattn_device_status(wsattn_plan_t plan, void* stream);

/* Failure-path self test: launches a one-thread kernel that waits on a
 * barrier nothing completes, with a wait limit of about `limit_ms`
 * milliseconds, and reports the status the kernel wrote (TIMEOUT expected)
 * in *status.  Synchronises `stream`.  Returns CUDA if the launch failed. */
int wsattn_selftest_timeout(int limit_ms, int* status, void* stream);

/* Build flags of the loaded library: bit 0 (WSATTN_BUILD_DEBUG) is set in a
 * build compiled with WSATTN_DEBUG, whose kernels check every TMA
 * coordinate, tensor-memory column range, shared-memory layout, output row
 * and work-item index against its limit before the access; a failed check
 * skips the access and sets a status bit that wsattn_device_status reports
 * as BOUNDS (no trap, no assert).  The paper has no counterpart: it is a
 * test aid standing in for a memory checker.  Release builds return 0. */
enum { WSATTN_BUILD_DEBUG = 1 };
int wsattn_build_flags(void);

/* Static text for a status code. */
const char* wsattn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* WSATTN_H_ */
