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
// Two HBM-bound passes over [BH, N, D] bf16, each CTA owning one chunk of
// rows of one (b, h); every reduction runs in a fixed order, so the results
// are bit-reproducible:
//   A  per-chunk key column sums                                (reads k)
//   B  mu = ordered sum of the chunk sums / N; key norms ||k_j - mu|| and
//      their per-chunk max; query norms ||q_i||, c_i, per-chunk max query
//      norm (row norms reduced with warp shuffles)        (reads k and q).
//      The last CTA of each head to finish (a per-head counter) then takes
//      K_h = max of the chunk maxima (with window bounds, where the chunks
//      are the frames: for each query frame, the max over the frames it
//      attends), B_h = (scale max ||q_i||) K_h, which equals max_i b_i because
//      the expression is monotone in ||q_i||, and
//      eligible = B_h <= tau and 2 B_h < 126 ln 2.
// The row bound b_i = (scale ||q_i||) K and the fixed max m_i = b_i + c_i are
// not written out on the hot path: the forward forms m_i from ||q_i||, c_i
// and its frame's K when it starts a tile.  finalize_rows writes b_i and m_i
// for the readers of the statistics.
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

// Per-head statistics, computed by the last CTA of the head in pass B once
// every chunk's maxima are written.  Global bound: K_h for every query
// frame.  Window bound (win.nf > 0; chunk g is frame g): K_a = the largest
// maximum over the frames query frame a attends, for each a; kmax keeps the
// head's global maximum; B_h = max_a (scale max_{i in a} ||q_i||) K_a.
struct HeadOut {
  float* kq;
  int nfq;
  float* kmax;
  float* bmax;
  uint8_t* elig;
};

__device__ void head_finish(int bh, int nchunk, float scale, float tau, const FrameWindow& win,
                            const float* part_kmax, const float* part_qmax, const HeadOut& o,
                            float* scratch) {
  const float* pk = part_kmax + static_cast<size_t>(bh) * nchunk;
  const float* pq = part_qmax + static_cast<size_t>(bh) * nchunk;
  // the other CTAs' maxima: read from L2, past any stale L1 line
  float kg = 0.f, bm = 0.f;
  if (win.nf == 0) {
    float qm = 0.f;
    for (int g = threadIdx.x; g < nchunk; g += kPrepThreads) {
      kg = fmaxf(kg, __ldcg(pk + g));
      qm = fmaxf(qm, __ldcg(pq + g));
    }
    kg = block_max(kg, scratch);
    __syncthreads();
    qm = block_max(qm, scratch);
    if (threadIdx.x == 0) {
      scratch[0] = kg;
      bm = (scale * qm) * kg;
    }
    __syncthreads();
    const float kh = scratch[0];
    for (int a = threadIdx.x; a < o.nfq; a += kPrepThreads)
      o.kq[static_cast<size_t>(bh) * o.nfq + a] = kh;
  } else {
    for (int a = threadIdx.x; a < nchunk; a += kPrepThreads) {
      float ka = 0.f;
      for (int g = 0; g < nchunk; ++g)
        if (frames_interact(a, g, win.F, win.w, win.R, win.flags)) ka = fmaxf(ka, __ldcg(pk + g));
      o.kq[static_cast<size_t>(bh) * o.nfq + a] = ka;
      kg = fmaxf(kg, __ldcg(pk + a));
      bm = fmaxf(bm, (scale * __ldcg(pq + a)) * ka);
    }
    kg = block_max(kg, scratch);
    __syncthreads();
    bm = block_max(bm, scratch);
  }
  if (threadIdx.x == 0) {
    const float underflow_limit = 126.0f * 0.693147180559945309f;
    o.kmax[bh] = kg;
    o.bmax[bh] = bm;
    o.elig[bh] = static_cast<uint8_t>(bm <= tau && 2.0f * bm < underflow_limit);
  }
}

template <int D>
__global__ void __launch_bounds__(kPrepThreads)
    prep_pass_b(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k, int64_t n, int rpc,
                int nchunk, float scale, float tau, const float* __restrict__ part_sum, int nsum,
                float* __restrict__ mu_out, float* __restrict__ qn, float* __restrict__ crow,
                float* __restrict__ part_kmax, float* __restrict__ part_qmax,
                int* __restrict__ head_count, FrameWindow win, HeadOut ho) {
  constexpr int kLanes = D / 8;
  constexpr int kRows = kPrepThreads / kLanes;
  __shared__ float mu_s[D];
  __shared__ float wmax[kPrepThreads / 32];
  __shared__ int last;
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
    // publish this chunk's maxima, then count it; the head's last chunk
    // (in whatever order they end) finishes the head
    __threadfence();
    last = atomicAdd(head_count + bh, 1) == nchunk - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  head_finish(bh, nchunk, scale, tau, win, part_kmax, part_qmax, ho, wmax);
  if (threadIdx.x == 0) head_count[bh] = 0;  // ready for the next launch
}

// b_i and m_i of every row from ||q_i||, c_i and the row's frame bound
// (in place when the outputs are the inputs).
__global__ void __launch_bounds__(kPrepThreads)
    prep_finalize_rows(const float* qn, const float* crow, const float* __restrict__ kq, int nfq,
                       int64_t tq, int64_t n, int64_t total, float scale, float* b_out,
                       float* m_out) {
  ptx::griddep_wait();  // the statistics come from pass B
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kPrepThreads + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * kPrepThreads) {
    const int64_t bh = i / n, r = i - bh * n;
    const float kb = kq[bh * nfq + r / tq];
    const float b = row_bound(scale, qn[i], kb);
    const float c = crow[i];
    b_out[i] = b;
    m_out[i] = __fadd_rn(b, c);
  }
}

}  // namespace

void prepare_chunking(int BH, int64_t N, int num_sms, int* nchunk, int* rows_per_chunk) {
  // One wave of pass B (its 64 registers per thread fit four 256-thread
  // CTAs per SM): 4 * SMs CTAs over the heads, at least 64 rows per CTA.  A
  // partial second wave would leave most SMs idle for its whole length.
  // Measured at the SR shape: 3 per SM 73.9 us, 4 per SM 70.5, 8 per SM
  // 76.3 (dense shape: 250, 224, 216).
  int64_t want = 4LL * num_sms / BH;
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
  const FrameWindow fw = win ? *win : FrameWindow{0, 0, 0, 0, 0};
  const HeadOut ho{b.kq, b.nfq, b.kmax, b.bmax, b.elig};
  // every pass may start while its predecessor finishes and waits for it
  // on the device
  cudaError_t e = cudaSuccess;
  if (D == 128) {
    if (!key_sums)
      e = launch_dependent(prep_pass_a<128>, grid, dim3(kPrepThreads), 0, stream, k16, N,
                           b.rows_per_chunk, b.nchunk, b.part_sum);
    if (e != cudaSuccess) return e;
    e = launch_dependent(prep_pass_b<128>, grid, dim3(kPrepThreads), 0, stream, q16, k16, N,
                         b.rows_per_chunk, b.nchunk, scale, tau, sums, nsum, b.mu, b.qn_rows,
                         b.c_rows, b.part_kmax, b.part_qmax, b.head_count, fw, ho);
  } else {
    if (!key_sums)
      e = launch_dependent(prep_pass_a<64>, grid, dim3(kPrepThreads), 0, stream, k16, N,
                           b.rows_per_chunk, b.nchunk, b.part_sum);
    if (e != cudaSuccess) return e;
    e = launch_dependent(prep_pass_b<64>, grid, dim3(kPrepThreads), 0, stream, q16, k16, N,
                         b.rows_per_chunk, b.nchunk, scale, tau, sums, nsum, b.mu, b.qn_rows,
                         b.c_rows, b.part_kmax, b.part_qmax, b.head_count, fw, ho);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_finalize_rows(const PrepBuffers& b, int BH, int64_t N, float scale,
                                 float* b_out, float* m_out, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(BH) * N;
  int64_t blocks = (total + kPrepThreads - 1) / kPrepThreads;
  if (blocks > 4096) blocks = 4096;
  const cudaError_t e =
      launch_dependent(prep_finalize_rows, dim3(static_cast<unsigned>(blocks)), dim3(kPrepThreads),
                       0, stream, static_cast<const float*>(b.qn_rows),
                       static_cast<const float*>(b.c_rows), static_cast<const float*>(b.kq), b.nfq,
                       b.tq, N, total, scale, b_out, m_out);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace wsattn
