// Fixed-max statistics: key mean, Cauchy-Schwarz row bounds and per-head
// eligibility.
//
// Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
// TPUs", section "Breaking softmax's dependency chain": a query's largest
// logit is at most its norm times the largest key norm; centering the keys
// on their shared mean first tightens that bound and leaves the softmax
// unchanged; a head whose bound is too loose (its exponentials would
// underflow) takes the online path.  The small per-row arrays this produces
// are what the forward kernel reads at the start of each query tile.
//
// The centering is applied to the bound, not to the stored keys: with
//   s'_ij = scale q_i.(k_j - mu) = s_ij - c_i,   c_i = scale q_i.mu,
// the fixed-max probability exp(s'_ij - b_i) equals exp(s_ij - m_i) with
// m_i = b_i + c_i.  The forward kernel multiplies the caller's bf16 keys as
// they are (no second rounding of k - mu) and uses m_i as the row's fixed max.
//
// Three HBM-bound passes over [BH, N, D] bf16, each CTA owning one chunk of
// rows of one (b, h); every reduction runs in a fixed order (no atomics), so
// the results are bit-reproducible:
//   A  per-chunk key column sums                                (reads k)
//   B  mu = ordered sum of the chunk sums / N; key norms ||k_j - mu|| and
//      their per-chunk max; query norms ||q_i||, c_i, per-chunk max query
//      norm (row norms reduced with warp shuffles)        (reads k and q)
//   C  K_h = max of the chunk maxima (with window bounds, where the chunks
//      are the frames: the max over the frames the row's frame attends);
//      b_i = (scale ||q_i||) K_h;
//      m_i = b_i + c_i; B_h = (scale max ||q_i||) K_h, which equals max_i b_i
//      because the expression is monotone in ||q_i||;
//      eligible = B_h <= tau and 2 B_h < 126 ln 2.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace wsattn {
namespace {

constexpr int kPrepThreads = 256;
// Rows a thread group loads before it reduces any of them: the passes are
// bound by HBM only with several 16-byte loads in flight per thread.
constexpr int kUnroll = 4;

// Eight bf16 in a 16-byte word -> fp32 (exact: bf16 is the top half of fp32).
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int kLanes>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Max over the CTA; the result is valid in thread 0.  Contains __syncthreads.
__device__ __forceinline__ float block_max(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x / 32] = v;
  __syncthreads();
  float m = 0.f;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kPrepThreads / 32; ++w) m = fmaxf(m, scratch[w]);
  }
  return m;
}

// Max of v[0, n) (values >= 0) over the calling warp (every lane gets it):
// lane l takes v[l], v[l + 32], ...; max is exact in any order.
__device__ __forceinline__ float warp_max_of(const float* __restrict__ v, int n) {
  float m = 0.f;
  for (int i = threadIdx.x & 31; i < n; i += 32) m = fmaxf(m, v[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    prep_pass_a(const uint16_t* __restrict__ k, int64_t n, int rpc, int nchunk,
                float* __restrict__ part_sum) {
  constexpr int kLanes = D / 8;                 // threads sharing one row
  constexpr int kRows = kPrepThreads / kLanes;  // rows in flight per CTA
  __shared__ float red[kRows][D];
  ptx::griddep_wait();  // whatever ran before may still read part_sum or write k
  const int bh = blockIdx.y, c = blockIdx.x;
  const int lr = threadIdx.x % kLanes, rs = threadIdx.x / kLanes;
  const int64_t r0 = static_cast<int64_t>(c) * rpc;
  const int64_t r1 = min(n, r0 + rpc);
  const size_t base = static_cast<size_t>(bh) * n;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int64_t rb = r0; rb < r1; rb += kRows * kUnroll) {
    uint4 kv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t r = rb + u * kRows + rs;
      kv[u] = r < r1 ? __ldg(reinterpret_cast<const uint4*>(k + (base + r) * D) + lr)
                     : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float kf[8];
      unpack8(kv[u], kf);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += kf[i];
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[rs][lr * 8 + i] = acc[i];
  __syncthreads();
  if (threadIdx.x < D) {
    float s = 0.f;
    for (int g = 0; g < kRows; ++g) s += red[g][threadIdx.x];
    part_sum[(static_cast<size_t>(bh) * nchunk + c) * D + threadIdx.x] = s;
  }
}

template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    prep_pass_b(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k, int64_t n, int rpc,
                int nchunk, float scale, const float* __restrict__ part_sum, int nsum,
                float* __restrict__ mu_out, float* __restrict__ qn, float* __restrict__ crow,
                float* __restrict__ part_kmax, float* __restrict__ part_qmax) {
  constexpr int kLanes = D / 8;
  constexpr int kRows = kPrepThreads / kLanes;
  __shared__ float mu_s[D];
  __shared__ float wmax[kPrepThreads / 32];
  ptx::griddep_wait();  // the key sums come from the previous kernel
  const int bh = blockIdx.y, c = blockIdx.x;
  const int lr = threadIdx.x % kLanes, rs = threadIdx.x / kLanes;
  if (threadIdx.x < D) {
    // four interleaved partial sums keep four loads in flight; they combine
    // in a fixed order, so the mean stays reproducible
    const float* ps = part_sum + static_cast<size_t>(bh) * nsum * D + threadIdx.x;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int cc = 0;
    for (; cc + 3 < nsum; cc += 4) {
      a0 += ps[static_cast<size_t>(cc) * D];
      a1 += ps[static_cast<size_t>(cc + 1) * D];
      a2 += ps[static_cast<size_t>(cc + 2) * D];
      a3 += ps[static_cast<size_t>(cc + 3) * D];
    }
    for (; cc < nsum; ++cc) a0 += ps[static_cast<size_t>(cc) * D];
    const float s = (a0 + a1) + (a2 + a3);
    const float m = s / static_cast<float>(n);
    mu_s[threadIdx.x] = m;
    if (c == 0) mu_out[static_cast<size_t>(bh) * D + threadIdx.x] = m;
  }
  __syncthreads();
  float mloc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) mloc[i] = mu_s[lr * 8 + i];
  const int64_t r0 = static_cast<int64_t>(c) * rpc;
  const int64_t r1 = min(n, r0 + rpc);
  const size_t base = static_cast<size_t>(bh) * n;
  float km = 0.f, qm = 0.f;
  // Row groups in reverse order: pass A just streamed this chunk's keys in
  // forward order, so the most recently read ones (the likeliest still in
  // L2) come first.  q is read once here: evict-first, no L1 allocation.
  const uint64_t q_policy = ptx::policy_evict_first();
  constexpr int64_t kGroup = kRows * kUnroll;
  const int64_t n_groups = (r1 - r0 + kGroup - 1) / kGroup;
  for (int64_t g = n_groups - 1; g >= 0; --g) {  // uniform trip count per warp
    const int64_t rb = r0 + g * kGroup;
    uint4 kv[kUnroll], qv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t r = rb + u * kRows + rs;
      if (r < r1) {
        kv[u] = __ldg(reinterpret_cast<const uint4*>(k + (base + r) * D) + lr);
        qv[u] = ptx::ld_stream_v4(reinterpret_cast<const uint4*>(q + (base + r) * D) + lr,
                                  q_policy);
      } else {
        kv[u] = make_uint4(0u, 0u, 0u, 0u);
        qv[u] = kv[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t r = rb + u * kRows + rs;
      float kss = 0.f, qss = 0.f, qmu = 0.f;
      if (r < r1) {
        float kf[8], qf[8];
        unpack8(kv[u], kf);
        unpack8(qv[u], qf);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x = kf[i] - mloc[i];
          kss = fmaf(x, x, kss);
          qss = fmaf(qf[i], qf[i], qss);
          qmu = fmaf(qf[i], mloc[i], qmu);
        }
      }
      kss = group_sum<kLanes>(kss);
      qss = group_sum<kLanes>(qss);
      qmu = group_sum<kLanes>(qmu);
      const float qnorm = sqrtf(qss);
      if (r < r1 && lr == 0) {
        qn[base + r] = qnorm;
        crow[base + r] = scale * qmu;
      }
      if (r < r1) {
        km = fmaxf(km, sqrtf(kss));
        qm = fmaxf(qm, qnorm);
      }
    }
  }
  const float kmb = block_max(km, wmax);
  __syncthreads();  // wmax is reused
  const float qmb = block_max(qm, wmax);
  if (threadIdx.x == 0) {
    part_kmax[static_cast<size_t>(bh) * nchunk + c] = kmb;
    part_qmax[static_cast<size_t>(bh) * nchunk + c] = qmb;
  }
}

__global__ void __launch_bounds__(kPrepThreads)
    prep_pass_c(int64_t n, int rpc, int nchunk, float scale, float tau, float* __restrict__ b_rows,
                float* __restrict__ m_rows, const float* __restrict__ part_kmax,
                const float* __restrict__ part_qmax, float* __restrict__ kmax,
                float* __restrict__ bmax, uint8_t* __restrict__ elig) {
  __shared__ float k_s;
  ptx::griddep_wait();  // the chunk maxima and row values come from pass B
  const int bh = blockIdx.y, c = blockIdx.x;
  if (threadIdx.x < 32) {
    const float kh = warp_max_of(part_kmax + static_cast<size_t>(bh) * nchunk, nchunk);
    if (threadIdx.x == 0) k_s = kh;
  }
  __syncthreads();
  const float kh = k_s;
  const int64_t r0 = static_cast<int64_t>(c) * rpc;
  const int64_t r1 = min(n, r0 + rpc);
  const size_t base = static_cast<size_t>(bh) * n;
  for (int64_t r = r0 + threadIdx.x; r < r1; r += kPrepThreads) {
    const float b = (scale * b_rows[base + r]) * kh;  // b_rows holds ||q_i|| here
    b_rows[base + r] = b;
    m_rows[base + r] = b + m_rows[base + r];          // m_rows holds c_i here
  }
  if (c == 0 && threadIdx.x < 32) {
    const float qm = warp_max_of(part_qmax + static_cast<size_t>(bh) * nchunk, nchunk);
    if (threadIdx.x != 0) return;
    const float bm = (scale * qm) * kh;
    const float underflow_limit = 126.0f * 0.693147180559945309f;
    kmax[bh] = kh;
    bmax[bh] = bm;
    elig[bh] = static_cast<uint8_t>(bm <= tau && 2.0f * bm < underflow_limit);
  }
}

// Window bounds (one chunk per frame): K_a = largest per-frame key-norm
// maximum over the frames query frame a attends; b_i = (scale ||q_i||) K_a;
// B_h = max_a (scale max_{i in a} ||q_i||) K_a, which equals max_i b_i (the
// expression is monotone in ||q_i||).  kmax keeps the head's global maximum.
__global__ void __launch_bounds__(kPrepThreads)
    prep_pass_c_window(int64_t n, int rpc, int nchunk, int F, int R, int w, int flags,
                       float scale, float tau,
                       float* __restrict__ b_rows, float* __restrict__ m_rows,
                       const float* __restrict__ part_kmax, const float* __restrict__ part_qmax,
                       float* __restrict__ kmax, float* __restrict__ bmax,
                       uint8_t* __restrict__ elig) {
  __shared__ float k_s;
  ptx::griddep_wait();  // the chunk maxima and row values come from pass B
  const int bh = blockIdx.y, a = blockIdx.x;
  const float* pk = part_kmax + static_cast<size_t>(bh) * nchunk;
  auto window_max = [&](int f) {
    float kh = 0.f;
    for (int g = 0; g < nchunk; ++g)
      if (frames_interact(f, g, F, w, R, flags)) kh = fmaxf(kh, pk[g]);
    return kh;
  };
  if (threadIdx.x < 32) {  // the warp's lanes take the key frames g = lane, lane + 32, ...
    float kh = 0.f;
    for (int g = threadIdx.x; g < nchunk; g += 32)
      if (frames_interact(a, g, F, w, R, flags)) kh = fmaxf(kh, pk[g]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) kh = fmaxf(kh, __shfl_xor_sync(0xffffffffu, kh, o));
    if (threadIdx.x == 0) k_s = kh;
  }
  __syncthreads();
  const float kh = k_s;
  const int64_t r0 = static_cast<int64_t>(a) * rpc;
  const int64_t r1 = min(n, r0 + rpc);
  const size_t base = static_cast<size_t>(bh) * n;
  for (int64_t r = r0 + threadIdx.x; r < r1; r += kPrepThreads) {
    const float b = (scale * b_rows[base + r]) * kh;  // b_rows holds ||q_i|| here
    b_rows[base + r] = b;
    m_rows[base + r] = b + m_rows[base + r];          // m_rows holds c_i here
  }
  if (a == 0 && threadIdx.x < 32) {  // lanes take the query frames; max is order-free
    float kg = 0.f, bm = 0.f;
    for (int f = threadIdx.x; f < nchunk; f += 32) {
      kg = fmaxf(kg, pk[f]);
      bm = fmaxf(bm, (scale * part_qmax[static_cast<size_t>(bh) * nchunk + f]) * window_max(f));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      kg = fmaxf(kg, __shfl_xor_sync(0xffffffffu, kg, o));
      bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    }
    if (threadIdx.x != 0) return;
    const float underflow_limit = 126.0f * 0.693147180559945309f;
    kmax[bh] = kg;
    bmax[bh] = bm;
    elig[bh] = static_cast<uint8_t>(bm <= tau && 2.0f * bm < underflow_limit);
  }
}

}  // namespace

void prepare_chunking(int BH, int64_t N, int num_sms, int* nchunk, int* rows_per_chunk) {
  // One wave of pass B (its registers fit three 256-thread CTAs per SM):
  // 3 * SMs CTAs over the heads, at least 64 rows per CTA.  A partial second
  // wave would leave most SMs idle for its whole length.
  int64_t want = 3LL * num_sms / BH;
  int64_t max_chunks = (N + 63) / 64;
  if (want > max_chunks) want = max_chunks;
  if (want < 1) want = 1;
  int64_t rpc = (N + want - 1) / want;
  rpc = (rpc + 15) / 16 * 16;
  *rows_per_chunk = static_cast<int>(rpc);
  *nchunk = static_cast<int>((N + rpc - 1) / rpc);
}

cudaError_t launch_prepare(const void* q, const void* k, int BH, int64_t N, int D, float scale,
                           float tau, const PrepBuffers& b, const FrameWindow* win,
                           const float* key_sums, cudaStream_t stream) {
  const dim3 grid(b.nchunk, BH);
  const uint16_t* q16 = static_cast<const uint16_t*>(q);
  const uint16_t* k16 = static_cast<const uint16_t*>(k);
  // key column sums: pass A's per-chunk sums, or the producer's partial rows
  const float* sums = key_sums ? key_sums : b.part_sum;
  const int nsum = key_sums ? kKeySumRows : b.nchunk;
  // every pass may start while its predecessor finishes and waits for it
  // on the device
  cudaError_t e = cudaSuccess;
  if (D == 128) {
    if (!key_sums)
      e = launch_dependent(prep_pass_a<128>, grid, dim3(kPrepThreads), 0, stream, k16, N,
                           b.rows_per_chunk, b.nchunk, b.part_sum);
    if (e != cudaSuccess) return e;
    e = launch_dependent(prep_pass_b<128>, grid, dim3(kPrepThreads), 0, stream, q16, k16, N,
                         b.rows_per_chunk, b.nchunk, scale, sums, nsum, b.mu, b.b_rows, b.m_rows,
                         b.part_kmax, b.part_qmax);
  } else {
    if (!key_sums)
      e = launch_dependent(prep_pass_a<64>, grid, dim3(kPrepThreads), 0, stream, k16, N,
                           b.rows_per_chunk, b.nchunk, b.part_sum);
    if (e != cudaSuccess) return e;
    e = launch_dependent(prep_pass_b<64>, grid, dim3(kPrepThreads), 0, stream, q16, k16, N,
                         b.rows_per_chunk, b.nchunk, scale, sums, nsum, b.mu, b.b_rows, b.m_rows,
                         b.part_kmax, b.part_qmax);
  }
  if (e != cudaSuccess) return e;
  if (win) {
    e = launch_dependent(prep_pass_c_window, grid, dim3(kPrepThreads), 0, stream, N,
                         b.rows_per_chunk, b.nchunk, win->F, win->R, win->w, win->flags, scale,
                         tau, b.b_rows, b.m_rows, b.part_kmax, b.part_qmax, b.kmax, b.bmax,
                         b.elig);
  } else {
    e = launch_dependent(prep_pass_c, grid, dim3(kPrepThreads), 0, stream, N, b.rows_per_chunk,
                         b.nchunk, scale, tau, b.b_rows, b.m_rows, b.part_kmax, b.part_qmax,
                         b.kmax, b.bmax, b.elig);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace wsattn
