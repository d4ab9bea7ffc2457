// Internal declarations shared by the translation units of libwsattn.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "wsattn.h"

namespace wsattn {

// Rows of one query tile: the M of every tcgen05.mma the forward issues.
constexpr int kTileM = 128;
// Largest key block, and the key step the plan aims for: floor(160 / bk)
// blocks (one block when bk > 160 is rejected by the forward).
constexpr int kMaxBlockK = 160;
constexpr int kStepKeys = 160;
// Tensor memory (512 columns) holds O (D columns), one S buffer (step
// columns), two P buffers (step/2 columns each) and Q (D/2 columns).
constexpr int kTmemColumns = 512;
inline bool forward_tmem_fits(int D, int step_keys) {
  return D + D / 2 + 2 * step_keys <= kTmemColumns;
}
// Default eligibility threshold, in scaled-logit units.
constexpr float kDefaultTau = 40.0f;

// One unit of forward work for one (b, h): a 128-row query tile inside one
// frame and that frame's active key blocks.  A frame's key blocks form at
// most two runs of consecutive blocks (the reference frames and the window),
// so the kernel walks them arithmetically: block j is run0 + j for j < len0,
// else run1 + (j - len0).
//
// When T is not a multiple of 128, each frame ends in a short tail tile of
// T mod 128 rows.  The tails of up to 128 / (T mod 128) consecutive frames
// are merged into one tile whose key list is the union of theirs (still at
// most two runs), when that takes fewer key steps than the separate tails.
// Row group i (tile rows [i*gsz, (i+1)*gsz)) is the tail of the first
// frame's successor i, i.e. tokens row0 + i*T onwards.  Its own key runs are
// in the group table, and the keys of the union that its frame does not
// attend get probability zero.
struct WorkTile {
  int32_t row0;    // first query token of the tile (within the head)
  int32_t nvalid;  // rows of the tile that belong to its frame(s) (<= 128)
  int32_t nblk;    // active key blocks of the tile (of the union for merged tails)
  int32_t run0;    // first key block of the first run (units of bk)
  int32_t len0;    // blocks in the first run
  int32_t run1;    // first key block of the second run
  int32_t nstep;   // key steps: ceil(nblk / G) (the runs walked as one sequence)
  int32_t kbeg;    // first of the (first) frame's blocks in kcol (kcol[kbeg + j])
  int32_t gsz;     // merged tails: rows per row group; 0 for a tile of one frame
  int32_t gtab;    // merged tails: first group's entry in the group table
};
// Group table entry of a merged tile's row group: its frame's key runs
// {run0, len0, run1, len1} (units of bk; len1 may be 0).
constexpr int kGroupInts = 4;

// Token (within the head) of row r of tile t, T tokens per frame.
__host__ __device__ inline int64_t tile_row_token(const WorkTile& t, int r, int T) {
  return t.gsz ? t.row0 + static_cast<int64_t>(r / t.gsz) * T + r % t.gsz : t.row0 + r;
}

// Host-side plan: geometry, block map, and the forward work list.
struct HostPlan {
  int F = 0, T = 0, w = 0, R = 0, H = 0, D = 0, bq = 0, bk = 0;
  int flags = 0;                   // wsattn_mask_flags
  int64_t N = 0, nqb = 0, nkb = 0;
  std::vector<uint8_t> bitmap;     // [nqb * nkb]
  std::vector<int32_t> row_ptr;    // [nqb + 1]
  std::vector<int32_t> col;        // [nnz]
  std::vector<WorkTile> tiles;     // longest first
  std::vector<int32_t> kcol;       // per frame, key block indices (units of bk)
  std::vector<int32_t> grp;        // group table of merged tail tiles (kGroupInts per group)
  int gsz = 0;                     // rows per row group of the merged tail tiles (0: none)
  // Tiles with equal key-list length form a class; class c covers tiles
  // [cls[c], cls[c + 1]).  The forward visits work items class by class
  // (longest first) and, inside a class, head by head, so CTAs running at
  // the same time stream the same head's keys and values.
  std::vector<int32_t> cls;
  int64_t active_pairs = 0;        // active (query, key) pairs per (b, h)
  int G = 1;                       // blocks per key step of the forward kernel
};

// Builds everything above; returns a WSATTN_* status.
int build_host_plan(int frames, int tokens_per_frame, int window, int ref_frames, int heads,
                    int head_dim, int block_q, int block_k, int mask_flags, HostPlan* out);

// Frame rule of the mask family: query frame a attends key frame c (frame
// indices in token order).  Host and device share it.
__host__ __device__ inline bool frames_interact(int a, int c, int F, int w, int R, int flags) {
  const bool suffix = (flags & WSATTN_MASK_REF_SUFFIX) != 0;
  const bool ref_a = suffix ? a >= F : a < R;
  const bool ref_c = suffix ? c >= F : c < R;
  if (ref_a) return (flags & WSATTN_MASK_REF_LOCAL) ? ref_c : true;
  if (ref_c) return true;
  const int d = a - c;  // video indices differ by the same amount as frame indices
  if (flags & WSATTN_MASK_CAUSAL) return d >= 0 && d <= w;
  return (d < 0 ? -d : d) <= w;
}

// Picks a block size for T: among the valid sizes (multiples of 16 dividing
// T, at most kStepKeys), the one whose forward key step
// floor(kStepKeys / bk) * bk is longest, the larger on ties.
int auto_block(int T);

// ------------------------------------------------------------ prepare
// What prepare leaves on the device: per row ||q_i|| and c_i = scale q_i.mu,
// per (b, h) and query frame the key-norm bound K (the head's K_h, or the
// window's), and per (b, h) K_h, B_h and eligibility.  The row bound and the
// fixed max follow as b_i = (scale ||q_i||) K and m_i = b_i + c_i (the
// forward forms m_i when it starts a tile; finalize_rows writes both out for
// readers).
struct PrepBuffers {
  float* qn_rows;       // [BH * N] ||q_i||
  float* c_rows;        // [BH * N] c_i = scale q_i.mu
  float* kq;            // [BH * nfq] key-norm bound of each query frame
  int nfq;              // query frames per head (1 when the head is one frame)
  int64_t tq;           // rows per query frame
  float* mu;            // [BH * D]
  float* kmax;          // [BH]
  float* bmax;          // [BH]
  uint8_t* elig;        // [BH]
  float* part_sum;      // [BH * nchunk * D]
  float* part_kmax;     // [BH * nchunk]
  float* part_qmax;     // [BH * nchunk]
  int* head_count;      // [BH] pass B chunks finished per head (0 between launches)
  int nchunk;
  int rows_per_chunk;
};

// Frame structure for window bounds: chunk c of a head is frame c (T rows),
// and query frame a attends key frame g as frames_interact says.
struct FrameWindow {
  int nf;  // R + F frames (= chunks per head)
  int F;
  int R;
  int w;
  int flags;  // wsattn_mask_flags
};

// Enqueues the prepare passes (A: key column sums; B: mean, norms, and in
// each head's last CTA the per-frame bounds, B_h and eligibility); returns a
// cudaError_t.  With `win` non-null the chunks must be the frames and the
// bounds are the per-window key-norm maxima (buf.nfq = frames).  With
// `key_sums` non-null ([BH, kKeySumRows, D]: each head's key column sums in
// kKeySumRows partial rows, from the producer) pass A is skipped.
cudaError_t launch_prepare(const void* q, const void* k, int BH, int64_t N, int D, float scale,
                           float tau, const PrepBuffers& buf, const FrameWindow* win,
                           const float* key_sums, cudaStream_t stream);

// b_i = (scale ||q_i||) K and m_i = b_i + c_i for every row, from what
// prepare left in `buf`, into b_out and m_out ([BH * N]; they may be
// buf.qn_rows and buf.c_rows themselves).  For readers of the statistics;
// the forward forms m_i itself.
cudaError_t launch_finalize_rows(const PrepBuffers& buf, int BH, int64_t N, float scale,
                                 float* b_out, float* m_out, cudaStream_t stream);

// The row bound and fixed max exactly as every kernel forms them (rounded
// products, no contraction), so readers see the values the forward uses.
__device__ __forceinline__ float row_bound(float scale, float qn, float k) {
  return __fmul_rn(__fmul_rn(scale, qn), k);
}

// Chunking of the N rows of one head across CTAs.
void prepare_chunking(int BH, int64_t N, int num_sms, int* nchunk, int* rows_per_chunk);

// ------------------------------------------------------------ forward
struct FwdParams {
  CUtensorMap tm_q;  // [BH*N, D] bf16, box {64, 128}, 128-byte swizzle
  CUtensorMap tm_qg; // [BH*N, D] bf16, box {64, gsz}: one row group of a merged tail tile
  CUtensorMap tm_k;  // [BH*N, D] bf16, box {64, G * bk}
  CUtensorMap tm_v;  // [BH*N, D] bf16, box {64, G * bk}
  CUtensorMap tm_k1; // [BH*N, D] bf16, box {64, bk}: one block of a step that spans both runs
  CUtensorMap tm_v1; // [BH*N, D] bf16, box {64, bk}
  CUtensorMap tm_o;  // [BH*N, D] fp32, box {16, 32}, no swizzle (epilogue stores)
  const WorkTile* tiles;
  const int32_t* grp;    // group table of the merged tail tiles
  const int32_t* cls;    // class boundaries into tiles, n_cls + 1 entries
  int* work;             // [2]: next work item, CTAs finished (both 0 between launches)
  int n_cls;
  const float* qn_rows;  // [BH*N] ||q_i||
  const float* c_rows;   // [BH*N] c_i = scale q_i.mu
  const float* kq;       // [BH * nfq] key-norm bound per query frame
  int nfq;               // query frames per head
  int tq;                // rows per query frame
  float scale;           // softmax scale
  const uint8_t* elig;   // [BH]
  float* out;            // [BH*N, D]
  int* status;           // device status word (bit set on an expired wait)
  int n_tiles;           // work tiles per (b, h)
  int bh;                // batch * heads
  int n;                 // tokens per head
  int bk;                // key block rows
  int G;                 // blocks per full key step (step keys <= kStepKeys)
  int stages_k, stages_v;
  int force_path;        // -1 auto, 0 fixed, 1 online
  float scale_log2;      // softmax scale * log2(e)
};

// Dynamic shared memory the forward kernel needs for (D, bk, stages).
size_t forward_smem_bytes(int D, int step_keys, int stages_k, int stages_v);
// Largest stage counts (<= 4 each) that fit the per-block shared memory.
void forward_stages(int D, int step_keys, size_t smem_optin, int* stages_k, int* stages_v);
// Launches the persistent forward kernel on `grid` CTAs.
cudaError_t launch_forward(const FwdParams& p, int D, int grid, size_t smem, cudaStream_t s);

// ------------------------------------------------------------ producer
// Pre-attention producer: y = (x W^T) / rms(x), rotary turn of q and k,
// bf16, head-packed [B, H, N, D] stores, and per-32-row key column sums.
constexpr int kProdTileM = 128;  // tokens per tile (one batch element)
constexpr int kProdTileK = 64;   // model-dim slice per pipeline stage
constexpr int kKeySumRows = 8;   // partial key-sum rows per head the producer hands to prepare
struct ProdParams {
  CUtensorMap tm_x;       // x [B, N, C] bf16, 3-D {C, N, B}, box {64, 128, 1}, 128-byte swizzle
  CUtensorMap tm_w;       // W [3HD, C] bf16, 2-D, box {64, BN}, 128-byte swizzle
  CUtensorMap tm_out[3];  // q, k, v [BH, N, D] bf16, 3-D {D, N, BH}, box {64, 32, 1}, swizzled
  const float* inv_rms;   // [B * N] 1 / sqrt(mean x^2 + eps)
  const float* rope_cos;  // [N, D / 2]
  const float* rope_sin;  // [N, D / 2]
  float* part_sum;        // [BH, nparts, D] key column sums of 32-row groups
  int* status;            // device status word (bit set on an expired wait)
  int batch, heads, n, c;
  int mtiles;             // ceil(N / 128)
  int ntiles;             // 3HD / BN
  int nparts;             // 4 * mtiles
};
// BN (feature columns per tile) for H * D, 0 if unsupported.
int produce_tile_n(int heads, int head_dim);
size_t produce_smem_bytes(int bn);
// RMS pre-pass, the producer GEMM (persistent, at most `grid` CTAs) and the reduction of the key column sums into [BH, D]; returns a
// cudaError_t.
cudaError_t launch_produce(const ProdParams& p, const uint16_t* x, float eps, int D, int bn,
                           int grid, float* inv_rms, float* key_sums, cudaStream_t stream);

// Self test of the bounded wait (see wsattn_selftest_timeout).
cudaError_t launch_timeout_selftest(long long limit_cycles, int* status, cudaStream_t s);

// Launches `kernel` with programmatic stream serialization: it may begin
// while the previous kernel in the stream is finishing, and each of its
// threads calls ptx::griddep_wait() before reading that kernel's results or
// writing anything an earlier kernel may still read.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Kernel launch attributes are set once per device (a process may drive
// several; cudaFuncSetAttribute acts on the current one).
constexpr int kMaxDevices = 64;
inline int current_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices ? d : -1;
}

// Device status bits.
constexpr int kStatusTimeoutProducer = 1;
constexpr int kStatusTimeoutMma = 2;
constexpr int kStatusTimeoutSoftmax = 4;
constexpr int kStatusTimeoutSelftest = 8;
constexpr int kStatusBounds = 16;  // a debug build's bounds check failed

// Bounds checks of the debug build (compiled with -DWSATTN_DEBUG): each
// TMA coordinate, tensor-memory column range, shared-memory layout, output
// row and work-item index the kernels use is checked against its limit
// before the access.  A failed check sets kStatusBounds in the status word
// and the access is skipped; nothing traps.  Release builds compile the
// checks out (the condition is not evaluated).
#ifdef WSATTN_DEBUG
constexpr bool kDebugBuild = true;
__device__ __forceinline__ bool bounds_ok(int* status, bool ok) {
  if (!ok && status) atomicOr(status, kStatusBounds);
  return ok;
}
#define WSATTN_BOUNDS(status, cond) (::wsattn::bounds_ok((status), (cond)))
#else
constexpr bool kDebugBuild = false;
#define WSATTN_BOUNDS(status, cond) (true)
#endif

}  // namespace wsattn
