// C ABI of libwsattn (declared in include/wsattn.h): plan lifecycle, device
// buffers, TMA tensor maps and kernel launches.  Nothing here computes on the
// host beyond argument checks and the block map (plan.cpp).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

using wsattn::FwdParams;
using wsattn::HostPlan;
using wsattn::PrepBuffers;
using wsattn::WorkTile;

struct wsattn_plan_s {
  HostPlan hp;
  int device = -1;
  int num_sms = 0;
  size_t smem_optin = 0;
  int clock_khz = 0;
  WorkTile* d_tiles = nullptr;
  int32_t* d_grp = nullptr;  // group table of the merged tail tiles (at least one entry)
  int32_t* d_cls = nullptr;
  int* d_status = nullptr;
  int* d_work = nullptr;  // the forward's work counters (zero between launches)
  // statistics workspace, sized for ws_batch
  int ws_batch = 0;
  void* ws = nullptr;
  PrepBuffers buf{};
  int prepared_batch = 0;
  int force_path = -1;
  float tau = wsattn::kDefaultTau;
  int bound_mode = WSATTN_BOUND_GLOBAL;
  // producer workspace (inverse RMS per token, key sums), sized for prod_batch
  int prod_batch = 0;
  void* prod_ws = nullptr;
  float* inv_rms = nullptr;    // [B * N]
  float* key_parts = nullptr;  // [BH, 4 * ceil(N / 128), D]
  float* key_sums = nullptr;   // [BH, kKeySumRows, D]
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D view [rows, D] of a bf16 tensor; box {64, box_rows}; 128-byte swizzle.
// fp32 [rows, D] output, box {16 columns, 32 rows}: one softmax warp's
// normalised rows of one 16-column group.
bool encode_out_map(CUtensorMap* m, void* ptr, int64_t rows, int D) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 4};
  const cuuint32_t box[2] = {16, 32};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int D, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// x [B, N, C] bf16 as a 3-D map {C, N, B}: 128 tokens x 64 features per
// box, 128-byte swizzle (K-major tcgen05 operand).  Tokens past N read as
// zero, so a batch element's last tile never sees the next one's rows.
bool encode_x_map(CUtensorMap* m, const void* ptr, int B, int64_t N, int C) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(C) * 2,
                                 static_cast<cuuint64_t>(N) * C * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q, k or v [BH, N, D] bf16 as a 3-D map {D, N, BH}: 32 tokens x 64
// dims per box (one epilogue warp's chunk); stores past N are dropped.
bool encode_head_map(CUtensorMap* m, void* ptr, int BH, int64_t N, int D) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(N) * D * 2};
  const cuuint32_t box[3] = {64, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// First device call: remember the device, upload the work list.
int ensure_device(wsattn_plan_s* p) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WSATTN_ERR_CUDA;
  if (p->device >= 0) return dev == p->device ? WSATTN_OK : WSATTN_ERR_BAD_ARG;
  int sms = 0, optin = 0, clk = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  const HostPlan& hp = p->hp;
  const size_t tiles_bytes = hp.tiles.size() * sizeof(WorkTile);
  const size_t cls_bytes = hp.cls.size() * sizeof(int32_t);
  const size_t grp_bytes =
      std::max<size_t>(hp.grp.size(), wsattn::kGroupInts) * sizeof(int32_t);
  if (cudaMalloc(&p->d_tiles, tiles_bytes) != cudaSuccess ||
      cudaMalloc(&p->d_grp, grp_bytes) != cudaSuccess ||
      cudaMalloc(&p->d_cls, cls_bytes) != cudaSuccess ||
      cudaMalloc(&p->d_status, sizeof(int)) != cudaSuccess ||
      cudaMalloc(&p->d_work, 2 * sizeof(int)) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  if (cudaMemcpy(p->d_tiles, hp.tiles.data(), tiles_bytes, cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemcpy(p->d_cls, hp.cls.data(), cls_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(p->d_grp, 0, grp_bytes) != cudaSuccess ||
      (!hp.grp.empty() && cudaMemcpy(p->d_grp, hp.grp.data(), hp.grp.size() * sizeof(int32_t),
                                     cudaMemcpyHostToDevice) != cudaSuccess) ||
      cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess ||
      cudaMemset(p->d_work, 0, 2 * sizeof(int)) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  p->device = dev;
  p->num_sms = sms;
  p->smem_optin = static_cast<size_t>(optin);
  p->clock_khz = clk;
  return WSATTN_OK;
}

// Statistics workspace for `batch`; growing it synchronises the stream.
int ensure_workspace(wsattn_plan_s* p, int batch, cudaStream_t stream) {
  if (batch <= p->ws_batch) return WSATTN_OK;
  const HostPlan& hp = p->hp;
  const int BH = batch * hp.H;
  int nchunk = 0, rpc = 0;
  wsattn::prepare_chunking(BH, hp.N, p->num_sms, &nchunk, &rpc);
  // Chunk slots: any batch <= this one needs at most BH * max(1, 4 SMs / BH)
  // <= 4 SMs + BH of them (prepare_chunking fills one wave).
  size_t slots = static_cast<size_t>(BH) * nchunk;
  const size_t bound = static_cast<size_t>(4) * p->num_sms + BH;
  if (slots < bound) slots = bound;
  // window bounds use one chunk per frame
  const size_t frame_slots = static_cast<size_t>(BH) * (hp.F + hp.R);
  if (slots < frame_slots) slots = frame_slots;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t n_b = up(sizeof(float) * BH * hp.N);  // qn_rows, and again for c_rows
  const size_t n_mu = up(sizeof(float) * BH * hp.D);
  const size_t n_h = up(sizeof(float) * BH);
  const size_t n_el = up(BH);
  const size_t n_ps = up(sizeof(float) * slots * hp.D);
  const size_t n_pm = up(sizeof(float) * slots);
  const size_t n_kq = up(sizeof(float) * BH * (hp.F + hp.R));
  const size_t n_cnt = up(sizeof(int) * BH);
  const size_t total = 2 * n_b + n_mu + 2 * n_h + n_el + n_ps + 2 * n_pm + n_kq + n_cnt;
  if (p->ws) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return WSATTN_ERR_CUDA;
    cudaFree(p->ws);
    p->ws = nullptr;
    p->ws_batch = 0;
  }
  if (cudaMalloc(&p->ws, total) != cudaSuccess) {
    p->ws = nullptr;
    return WSATTN_ERR_CUDA;
  }
  char* c = static_cast<char*>(p->ws);
  PrepBuffers& b = p->buf;
  b.qn_rows = reinterpret_cast<float*>(c); c += n_b;
  b.c_rows = reinterpret_cast<float*>(c); c += n_b;
  b.mu = reinterpret_cast<float*>(c); c += n_mu;
  b.kmax = reinterpret_cast<float*>(c); c += n_h;
  b.bmax = reinterpret_cast<float*>(c); c += n_h;
  b.elig = reinterpret_cast<uint8_t*>(c); c += n_el;
  b.part_sum = reinterpret_cast<float*>(c); c += n_ps;
  b.part_kmax = reinterpret_cast<float*>(c); c += n_pm;
  b.part_qmax = reinterpret_cast<float*>(c); c += n_pm;
  b.kq = reinterpret_cast<float*>(c); c += n_kq;
  b.head_count = reinterpret_cast<int*>(c);
  b.nfq = hp.F + hp.R;
  b.tq = hp.T;
  b.nchunk = nchunk;
  b.rows_per_chunk = rpc;
  // pass B's per-head counters start at zero (each launch leaves them so)
  if (cudaMemsetAsync(b.head_count, 0, n_cnt, stream) != cudaSuccess) return WSATTN_ERR_CUDA;
  p->ws_batch = batch;
  p->prepared_batch = 0;
  return WSATTN_OK;
}

// Producer workspace for `batch`; growing it synchronises the stream.
int ensure_prod_workspace(wsattn_plan_s* p, int batch, cudaStream_t stream) {
  if (batch <= p->prod_batch) return WSATTN_OK;
  const HostPlan& hp = p->hp;
  const size_t BH = static_cast<size_t>(batch) * hp.H;
  const size_t nparts = 4 * static_cast<size_t>((hp.N + wsattn::kProdTileM - 1) /
                                                wsattn::kProdTileM);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t n_inv = up(sizeof(float) * batch * hp.N);
  const size_t n_parts = up(sizeof(float) * BH * nparts * hp.D);
  const size_t n_sums = up(sizeof(float) * BH * wsattn::kKeySumRows * hp.D);
  if (p->prod_ws) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return WSATTN_ERR_CUDA;
    cudaFree(p->prod_ws);
    p->prod_ws = nullptr;
    p->prod_batch = 0;
  }
  if (cudaMalloc(&p->prod_ws, n_inv + n_parts + n_sums) != cudaSuccess) {
    p->prod_ws = nullptr;
    return WSATTN_ERR_CUDA;
  }
  char* c = static_cast<char*>(p->prod_ws);
  p->inv_rms = reinterpret_cast<float*>(c);
  p->key_parts = reinterpret_cast<float*>(c + n_inv);
  p->key_sums = reinterpret_cast<float*>(c + n_inv + n_parts);
  p->prod_batch = batch;
  return WSATTN_OK;
}

void free_device(wsattn_plan_s* p) {
  if (p->prod_ws) cudaFree(p->prod_ws);
  p->prod_ws = nullptr;
  if (p->d_tiles) cudaFree(p->d_tiles);
  if (p->d_grp) cudaFree(p->d_grp);
  if (p->d_cls) cudaFree(p->d_cls);
  if (p->d_status) cudaFree(p->d_status);
  if (p->d_work) cudaFree(p->d_work);
  if (p->ws) cudaFree(p->ws);
  p->d_tiles = nullptr;
  p->d_grp = nullptr;
  p->d_cls = nullptr;
  p->d_status = nullptr;
  p->d_work = nullptr;
  p->ws = nullptr;
}

// Enqueues the statistics passes for q, k (global or window bounds); with
// key_sums ([BH, kKeySumRows, D], from the producer) the key-sum pass is
// skipped.
int enqueue_prepare(wsattn_plan_s* plan, int batch, const void* q, const void* k,
                    const float* key_sums, cudaStream_t s) {
  const HostPlan& hp = plan->hp;
  const int BH = batch * hp.H;
  int nchunk = 0, rpc = 0;
  wsattn::FrameWindow win{hp.F + hp.R, hp.F, hp.R, hp.w, hp.flags};
  const bool window = plan->bound_mode == WSATTN_BOUND_WINDOW;
  if (window) {
    nchunk = win.nf;  // one chunk per frame: its maxima are the frame's
    rpc = hp.T;
  } else {
    wsattn::prepare_chunking(BH, hp.N, plan->num_sms, &nchunk, &rpc);
  }
  PrepBuffers b = plan->buf;
  b.nchunk = nchunk;
  b.rows_per_chunk = rpc;
  const float scale = 1.0f / std::sqrt(static_cast<float>(hp.D));
  if (wsattn::launch_prepare(q, k, BH, hp.N, hp.D, scale, plan->tau, b, window ? &win : nullptr,
                             key_sums, s) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  return WSATTN_OK;
}

}  // namespace

extern "C" {

int wsattn_plan(int frames, int tokens_per_frame, int window, int ref_frames, int heads,
                int head_dim, int block_q, int block_k, wsattn_plan_t* out) {
  return wsattn_plan_ex(frames, tokens_per_frame, window, ref_frames, heads, head_dim, block_q,
                        block_k, 0, out);
}

int wsattn_plan_ex(int frames, int tokens_per_frame, int window, int ref_frames, int heads,
                   int head_dim, int block_q, int block_k, int mask_flags, wsattn_plan_t* out) {
  if (!out) return WSATTN_ERR_BAD_ARG;
  *out = nullptr;
  wsattn_plan_s* p = new (std::nothrow) wsattn_plan_s();
  if (!p) return WSATTN_ERR_NO_MEMORY;
  const int rc = wsattn::build_host_plan(frames, tokens_per_frame, window, ref_frames, heads,
                                         head_dim, block_q, block_k, mask_flags, &p->hp);
  if (rc != WSATTN_OK) {
    delete p;
    return rc;
  }
  *out = p;
  return WSATTN_OK;
}

int wsattn_plan_destroy(wsattn_plan_t plan) {
  if (!plan) return WSATTN_OK;
  free_device(plan);
  delete plan;
  return WSATTN_OK;
}

int wsattn_prepare(wsattn_plan_t plan, int batch, const void* q, const void* k, void* stream) {
  if (!plan || batch < 1 || !q || !k || !aligned16(q) || !aligned16(k)) return WSATTN_ERR_BAD_ARG;
  const HostPlan& hp = plan->hp;
  if (static_cast<int64_t>(batch) * hp.H * hp.N >= (int64_t(1) << 31)) return WSATTN_ERR_BAD_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = ensure_device(plan);
  if (rc != WSATTN_OK) return rc;
  rc = ensure_workspace(plan, batch, s);
  if (rc != WSATTN_OK) return rc;
  rc = enqueue_prepare(plan, batch, q, k, nullptr, s);
  if (rc == WSATTN_OK) plan->prepared_batch = batch;
  return rc;
}

int wsattn_produce(wsattn_plan_t plan, int batch, const void* x, int model_dim,
                   const void* w_qkv, const float* rope_cos, const float* rope_sin, float eps,
                   void* q, void* k, void* v, void* stream) {
  if (!plan || batch < 1 || !x || !w_qkv || !rope_cos || !rope_sin || !q || !k || !v)
    return WSATTN_ERR_BAD_ARG;
  if (!aligned16(x) || !aligned16(w_qkv) || !aligned16(rope_cos) || !aligned16(rope_sin) ||
      !aligned16(q) || !aligned16(k) || !aligned16(v))
    return WSATTN_ERR_BAD_ARG;
  if (model_dim < wsattn::kProdTileK || model_dim % wsattn::kProdTileK != 0 || !(eps >= 0.f) ||
      !std::isfinite(eps))
    return WSATTN_ERR_BAD_ARG;
  const HostPlan& hp = plan->hp;
  if (static_cast<int64_t>(batch) * hp.H * hp.N >= (int64_t(1) << 31) ||
      static_cast<int64_t>(batch) * hp.N * model_dim >= (int64_t(1) << 40))
    return WSATTN_ERR_BAD_ARG;
  const int bn = wsattn::produce_tile_n(hp.H, hp.D);
  if (bn == 0) return WSATTN_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = ensure_device(plan);
  if (rc != WSATTN_OK) return rc;
  if (wsattn::produce_smem_bytes(bn) > plan->smem_optin) return WSATTN_ERR_UNSUPPORTED;
  rc = ensure_workspace(plan, batch, s);
  if (rc != WSATTN_OK) return rc;
  rc = ensure_prod_workspace(plan, batch, s);
  if (rc != WSATTN_OK) return rc;
  if (!get_encode()) return WSATTN_ERR_CUDA;
  const int BH = batch * hp.H;
  wsattn::ProdParams prm;
  std::memset(&prm, 0, sizeof(prm));
  void* outs[3] = {q, k, v};
  if (!encode_x_map(&prm.tm_x, x, batch, hp.N, model_dim) ||
      !encode_map(&prm.tm_w, w_qkv, 3LL * hp.H * hp.D, model_dim, bn))
    return WSATTN_ERR_CUDA;
  for (int i = 0; i < 3; ++i)
    if (!encode_head_map(&prm.tm_out[i], outs[i], BH, hp.N, hp.D)) return WSATTN_ERR_CUDA;
  prm.inv_rms = plan->inv_rms;
  prm.rope_cos = rope_cos;
  prm.rope_sin = rope_sin;
  prm.part_sum = plan->key_parts;
  prm.status = plan->d_status;
  prm.batch = batch;
  prm.heads = hp.H;
  prm.n = static_cast<int>(hp.N);
  prm.c = model_dim;
  prm.mtiles = static_cast<int>((hp.N + wsattn::kProdTileM - 1) / wsattn::kProdTileM);
  prm.ntiles = 3 * hp.H * hp.D / bn;
  prm.nparts = 4 * prm.mtiles;
  const int grid = plan->num_sms;  // one CTA per SM at most
  if (wsattn::launch_produce(prm, static_cast<const uint16_t*>(x), eps, hp.D, bn, grid,
                             plan->inv_rms, plan->key_sums, s) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  rc = enqueue_prepare(plan, batch, q, k, plan->key_sums, s);
  if (rc == WSATTN_OK) plan->prepared_batch = batch;
  return rc;
}

int wsattn_forward(wsattn_plan_t plan, int batch, const void* q, const void* k, const void* v,
                   float* out, void* stream) {
  if (!plan || batch < 1 || !q || !k || !v || !out) return WSATTN_ERR_BAD_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return WSATTN_ERR_BAD_ARG;
  const HostPlan& hp = plan->hp;
  if (plan->prepared_batch == 0) return WSATTN_ERR_NOT_PREPARED;
  if (batch != plan->prepared_batch) return WSATTN_ERR_BATCH_MISMATCH;
  if (hp.bk > wsattn::kMaxBlockK) return WSATTN_ERR_UNSUPPORTED;
  int rc = ensure_device(plan);
  if (rc != WSATTN_OK) return rc;
  if (!get_encode()) return WSATTN_ERR_CUDA;
  const int BH = batch * hp.H;
  const int64_t rows = static_cast<int64_t>(BH) * hp.N;
  FwdParams prm;
  std::memset(&prm, 0, sizeof(prm));
  // A key step is G consecutive blocks of one run, i.e. G * bk consecutive
  // rows: K and V are loaded one box of a whole step per 64-column slab.
  const int step_keys = hp.G * hp.bk;
  if (!encode_map(&prm.tm_q, q, rows, hp.D, wsattn::kTileM) ||
      (hp.gsz > 0 && !encode_map(&prm.tm_qg, q, rows, hp.D, hp.gsz)) ||
      !encode_map(&prm.tm_k, k, rows, hp.D, step_keys) ||
      !encode_map(&prm.tm_v, v, rows, hp.D, step_keys) ||
      !encode_map(&prm.tm_k1, k, rows, hp.D, hp.bk) ||
      !encode_map(&prm.tm_v1, v, rows, hp.D, hp.bk) ||
      !encode_out_map(&prm.tm_o, out, rows, hp.D))
    return WSATTN_ERR_CUDA;
  prm.tiles = plan->d_tiles;
  prm.grp = plan->d_grp;
  prm.cls = plan->d_cls;
  prm.n_cls = static_cast<int>(hp.cls.size()) - 1;
  prm.qn_rows = plan->buf.qn_rows;
  prm.c_rows = plan->buf.c_rows;
  prm.kq = plan->buf.kq;
  prm.nfq = plan->buf.nfq;
  prm.tq = static_cast<int>(plan->buf.tq);
  prm.scale = 1.0f / std::sqrt(static_cast<float>(hp.D));
  prm.elig = plan->buf.elig;
  prm.out = out;
  prm.status = plan->d_status;
  prm.n_tiles = static_cast<int>(hp.tiles.size());
  prm.bh = BH;
  prm.n = static_cast<int>(hp.N);
  prm.bk = hp.bk;
  prm.G = hp.G;
  if (!wsattn::forward_tmem_fits(hp.D, step_keys)) return WSATTN_ERR_UNSUPPORTED;
  wsattn::forward_stages(hp.D, step_keys, plan->smem_optin, &prm.stages_k, &prm.stages_v);
  prm.force_path = plan->force_path;
  prm.scale_log2 = (1.0f / std::sqrt(static_cast<float>(hp.D))) * 1.4426950408889634f;
  const size_t smem = wsattn::forward_smem_bytes(hp.D, step_keys, prm.stages_k, prm.stages_v);
  if (prm.stages_k < 2 || smem > plan->smem_optin) return WSATTN_ERR_UNSUPPORTED;
  const int64_t items = static_cast<int64_t>(prm.n_tiles) * BH;
  const int grid = static_cast<int>(items < plan->num_sms ? items : plan->num_sms);
  prm.work = plan->d_work;
  if (wsattn::launch_forward(prm, hp.D, grid, smem, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return WSATTN_ERR_CUDA;
  return WSATTN_OK;
}

int wsattn_plan_info(wsattn_plan_t plan, int64_t* info, int n) {
  if (!plan || !info || n < 0) return WSATTN_ERR_BAD_ARG;
  const HostPlan& hp = plan->hp;
  const int64_t v[10] = {hp.N,
                         hp.bq,
                         hp.bk,
                         hp.nqb,
                         hp.nkb,
                         static_cast<int64_t>(hp.col.size()),
                         static_cast<int64_t>(hp.tiles.size()),
                         hp.D,
                         hp.H,
                         hp.active_pairs};
  for (int i = 0; i < n && i < 10; ++i) info[i] = v[i];
  return WSATTN_OK;
}

int wsattn_get_tiles(wsattn_plan_t plan, int32_t* tiles, size_t n_tiles, int32_t* groups,
                     size_t n_groups) {
  if (!plan) return WSATTN_ERR_BAD_ARG;
  const HostPlan& hp = plan->hp;
  constexpr size_t kTileInts = sizeof(WorkTile) / sizeof(int32_t);
  if ((!tiles && !hp.tiles.empty()) || n_tiles < hp.tiles.size() * kTileInts ||
      (!groups && !hp.grp.empty()) || n_groups < hp.grp.size())
    return WSATTN_ERR_BAD_ARG;
  if (!hp.tiles.empty()) std::memcpy(tiles, hp.tiles.data(), hp.tiles.size() * sizeof(WorkTile));
  if (!hp.grp.empty()) std::memcpy(groups, hp.grp.data(), hp.grp.size() * sizeof(int32_t));
  return WSATTN_OK;
}

int wsattn_get_block_map(wsattn_plan_t plan, uint8_t* host, size_t n) {
  if (!plan || !host || n < plan->hp.bitmap.size()) return WSATTN_ERR_BAD_ARG;
  std::memcpy(host, plan->hp.bitmap.data(), plan->hp.bitmap.size());
  return WSATTN_OK;
}

int wsattn_get_csr(wsattn_plan_t plan, int32_t* row_ptr, int32_t* col, size_t n_row_ptr,
                   size_t n_col) {
  if (!plan || !row_ptr || (!col && !plan->hp.col.empty())) return WSATTN_ERR_BAD_ARG;
  if (n_row_ptr < plan->hp.row_ptr.size() || n_col < plan->hp.col.size())
    return WSATTN_ERR_BAD_ARG;
  std::memcpy(row_ptr, plan->hp.row_ptr.data(), plan->hp.row_ptr.size() * sizeof(int32_t));
  if (!plan->hp.col.empty())
    std::memcpy(col, plan->hp.col.data(), plan->hp.col.size() * sizeof(int32_t));
  return WSATTN_OK;
}

int wsattn_get_stats(wsattn_plan_t plan, float* b_rows, float* m_rows, float* mu, float* kmax,
                     float* bmax, uint8_t* elig, void* stream) {
  if (!plan) return WSATTN_ERR_BAD_ARG;
  if (plan->prepared_batch == 0) return WSATTN_ERR_NOT_PREPARED;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  const HostPlan& hp = plan->hp;
  const size_t BH = static_cast<size_t>(plan->prepared_batch) * hp.H;
  const PrepBuffers& b = plan->buf;
  if (b_rows || m_rows) {
    // b_i and m_i are formed from what prepare keeps (||q_i||, c_i, the
    // frame bounds) by a small kernel, into a temporary buffer
    const size_t rows = BH * hp.N;
    float* tmp = nullptr;
    if (cudaMalloc(&tmp, 2 * rows * sizeof(float)) != cudaSuccess) return WSATTN_ERR_CUDA;
    const float scale = 1.0f / std::sqrt(static_cast<float>(hp.D));
    bool ok = wsattn::launch_finalize_rows(b, static_cast<int>(BH), hp.N, scale, tmp, tmp + rows,
                                           nullptr) == cudaSuccess &&
              cudaDeviceSynchronize() == cudaSuccess;
    if (ok && b_rows)
      ok = cudaMemcpy(b_rows, tmp, rows * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess;
    if (ok && m_rows)
      ok = cudaMemcpy(m_rows, tmp + rows, rows * sizeof(float), cudaMemcpyDeviceToHost) ==
           cudaSuccess;
    cudaFree(tmp);
    if (!ok) return WSATTN_ERR_CUDA;
  }
  if (mu && cudaMemcpy(mu, b.mu, BH * hp.D * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  if (kmax && cudaMemcpy(kmax, b.kmax, BH * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  if (bmax && cudaMemcpy(bmax, b.bmax, BH * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  if (elig && cudaMemcpy(elig, b.elig, BH, cudaMemcpyDeviceToHost) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  return WSATTN_OK;
}

int wsattn_plan_set_debug(wsattn_plan_t plan, int force_path, float tau) {
  if (!plan || force_path < -1 || force_path > 1 || !(tau >= 0.0f)) return WSATTN_ERR_BAD_ARG;
  plan->force_path = force_path;
  if (tau > 0.0f) plan->tau = tau;
  return WSATTN_OK;
}

int wsattn_plan_set_bound(wsattn_plan_t plan, int mode) {
  if (!plan || (mode != WSATTN_BOUND_GLOBAL && mode != WSATTN_BOUND_WINDOW))
    return WSATTN_ERR_BAD_ARG;
  plan->bound_mode = mode;
  plan->prepared_batch = 0;  // the statistics depend on the mode
  return WSATTN_OK;
}

int wsattn_device_status(wsattn_plan_t plan, void* stream) {
  if (!plan) return WSATTN_ERR_BAD_ARG;
  if (plan->device < 0) return WSATTN_OK;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  int st = 0;
  if (cudaMemcpy(&st, plan->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  if (st == 0) return WSATTN_OK;
  const int code = (st & wsattn::kStatusBounds) ? WSATTN_ERR_BOUNDS : WSATTN_ERR_TIMEOUT;
  // A forward that gave up on a wait may leave its work counters non-zero
  // (the last CTA to finish resets them); the next forward would then skip
  // items.  Reset them with the status word.
  if (cudaMemset(plan->d_status, 0, sizeof(int)) != cudaSuccess ||
      (plan->d_work && cudaMemset(plan->d_work, 0, 2 * sizeof(int)) != cudaSuccess))
    return WSATTN_ERR_CUDA;
  return code;
}

int wsattn_selftest_timeout(int limit_ms, int* status, void* stream) {
  if (!status || limit_ms < 1 || limit_ms > 10000) return WSATTN_ERR_BAD_ARG;
  int dev = 0, clk = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  int* d = nullptr;
  if (cudaMalloc(&d, sizeof(int)) != cudaSuccess) return WSATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = WSATTN_OK;
  int st = -1;
  if (cudaMemsetAsync(d, 0xFF, sizeof(int), s) != cudaSuccess ||
      wsattn::launch_timeout_selftest(static_cast<long long>(limit_ms) * clk, d, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(&st, d, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    rc = WSATTN_ERR_CUDA;
  cudaFree(d);
  if (rc == WSATTN_OK) *status = st == wsattn::kStatusTimeoutSelftest ? WSATTN_ERR_TIMEOUT
                                 : st == 0                            ? WSATTN_OK
                                                                      : WSATTN_ERR_CUDA;
  return rc;
}

int wsattn_build_flags(void) { return wsattn::kDebugBuild ? WSATTN_BUILD_DEBUG : 0; }

const char* wsattn_status_string(int status) {
  switch (status) {
    case WSATTN_OK: return "ok";
    case WSATTN_ERR_BAD_ARG: return "bad argument";
    case WSATTN_ERR_BAD_BLOCK: return "block size must be a multiple of 16 dividing tokens_per_frame";
    case WSATTN_ERR_UNSUPPORTED: return "unsupported head_dim or block_k";
    case WSATTN_ERR_NOT_PREPARED: return "forward called before prepare";
    case WSATTN_ERR_BATCH_MISMATCH: return "batch differs from the last prepare";
    case WSATTN_ERR_CUDA: return "CUDA runtime error";
    case WSATTN_ERR_TIMEOUT: return "device-side wait expired";
    case WSATTN_ERR_NO_MEMORY: return "host allocation failed";
    case WSATTN_ERR_BOUNDS: return "device bounds check failed (debug build)";
    default: return "unknown status";
  }
}

}  // extern "C"
