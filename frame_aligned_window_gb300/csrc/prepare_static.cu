// wsattn_prepare_static: the prepare statistics without any device
// allocation.
//
// wsattn_prepare keeps its per-chunk partial sums in a workspace the plan
// allocates with cudaMalloc.  Some callers cannot let a library do that: a
// host framework that owns every byte of device memory through its own pool
// or a fixed budget, or a latency-critical loop that cannot afford
// cudaMalloc's implicit device synchronisation.  This entry point runs the
// same three prepare kernels, writes the statistics into buffers the caller
// passes in, and takes its scratch from a fixed array in the library's own
// device image instead of allocating it.  It takes no plan, so it always
// uses the global bound (the maximum key norm over all keys of the head):
// its results equal wsattn_prepare's on a plan left at the default bound;
// window bounds (wsattn_plan_set_bound) and mask flags do not apply.
//
// The scratch array, g_prepare_scratch below, holds kStaticSlots chunk slots
// (a partial key-column sum of up to 128 floats plus two partial maxima per
// slot) and, per (b, h), the head's key-norm bound and a counter of finished
// chunks: 2048 slots, 1,081,344 bytes.  Every GPU that loads the library
// holds that memory until the process exits.
//
// Sharing rules:
//   - every call uses the same array, and the array keeps whatever the last
//     call left in it.  Each pass writes every slot that a later pass of the
//     same call reads; the counters must start at zero, as they do when the
//     library is loaded, and every call leaves them at zero again;
//   - calls whose kernels can overlap on the GPU (for example calls on two
//     streams of one process with no event ordering them) race on the array
//     and corrupt each other's results; callers must order such calls.  Each
//     process has its own copy of the array;
//   - the first call on a device looks up the array's device address (with
//     that device current) and caches it; make that first call before any
//     stream capture begins.
#include <mutex>

#include "internal.h"

namespace wsattn {
namespace {

constexpr int kStaticSlots = 2048;
constexpr int kStaticMaxDim = 128;
// part_sum [slots][128], part_kmax [slots], part_qmax [slots], per-head
// bound [2048], per-head counter [2048] (as int)
constexpr size_t kStaticFloats =
    static_cast<size_t>(kStaticSlots) * kStaticMaxDim + 4 * static_cast<size_t>(kStaticSlots);

// Host code must not use this name as a device address: on the host it is a
// stand-in object.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) float g_prepare_scratch[kStaticFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Device address of the scratch array and SM count for the current device,
// looked up once per device.
int scratch_for_current_device(float** ptr, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WSATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return WSATTN_ERR_BAD_ARG;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prepare_scratch) != cudaSuccess || !p)
      return WSATTN_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return WSATTN_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<float*>(p);
    g_num_sms[dev] = sms;
  }
  *ptr = g_scratch_ptr[dev];
  *num_sms = g_num_sms[dev];
  return WSATTN_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace wsattn

extern "C" int wsattn_prepare_static(int batch, int heads, int n_tokens, int head_dim, float tau,
                                     const void* q, const void* k, float* b_rows, float* m_rows,
                                     float* mu, float* kmax, float* bmax, uint8_t* elig,
                                     void* stream) {
  using namespace wsattn;
  if (batch < 1 || heads < 1 || n_tokens < 1 || !(tau > 0.0f)) return WSATTN_ERR_BAD_ARG;
  if (head_dim != 64 && head_dim != 128) return WSATTN_ERR_UNSUPPORTED;
  if (!q || !k || !b_rows || !m_rows || !mu || !kmax || !bmax || !elig) return WSATTN_ERR_BAD_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(b_rows, 4) || !aligned(m_rows, 4) ||
      !aligned(mu, 4) || !aligned(kmax, 4) || !aligned(bmax, 4))
    return WSATTN_ERR_BAD_ARG;
  const int64_t bh64 = static_cast<int64_t>(batch) * heads;
  // The scratch holds one chunk slot per (b, h) at the very least.
  if (bh64 > kStaticSlots) return WSATTN_ERR_BAD_ARG;
  if (bh64 * n_tokens >= (int64_t(1) << 31)) return WSATTN_ERR_BAD_ARG;
  const int BH = static_cast<int>(bh64);
  const int64_t N = n_tokens;

  float* scratch = nullptr;
  int num_sms = 0;
  const int rc = scratch_for_current_device(&scratch, &num_sms);
  if (rc != WSATTN_OK) return rc;

  int nchunk = 0, rpc = 0;
  prepare_chunking(BH, N, num_sms, &nchunk, &rpc);
  // prepare_chunking gives at most max(BH, 4 * SMs) chunks in all, so this
  // holds on every GPU with at most 512 SMs; refuse rather than overrun the
  // scratch if the chunking ever asks for more.
  if (static_cast<int64_t>(nchunk) * BH > kStaticSlots) return WSATTN_ERR_BAD_ARG;

  // Pass B leaves ||q_i|| and c_i in the caller's b_rows and m_rows; the
  // finishing kernel turns them into b_i and m_i in place.
  PrepBuffers b;
  b.qn_rows = b_rows;
  b.c_rows = m_rows;
  b.mu = mu;
  b.kmax = kmax;
  b.bmax = bmax;
  b.elig = elig;
  b.part_sum = scratch;
  b.part_kmax = scratch + static_cast<size_t>(kStaticSlots) * kStaticMaxDim;
  b.part_qmax = b.part_kmax + kStaticSlots;
  b.kq = b.part_qmax + kStaticSlots;  // one bound per (b, h): the head is one frame
  b.nfq = 1;
  b.tq = N;
  b.head_count = reinterpret_cast<int*>(b.kq + kStaticSlots);
  b.nchunk = nchunk;
  b.rows_per_chunk = rpc;
  const float scale = 1.0f / sqrtf(static_cast<float>(head_dim));
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_prepare(q, k, BH, N, head_dim, scale, tau, b, nullptr, nullptr, st) != cudaSuccess ||
      launch_finalize_rows(b, BH, N, scale, b_rows, m_rows, st) != cudaSuccess)
    return WSATTN_ERR_CUDA;
  return WSATTN_OK;
}
