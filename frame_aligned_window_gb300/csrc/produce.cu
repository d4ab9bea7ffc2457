// Pre-attention producer: RMS normalisation, QKV projection, rotary
// embedding and head packing in one tcgen05 GEMM whose epilogue writes the
// attention's input layout directly.
//
// Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
// TPUs", section "Layout is ABI" and Figure 5: the attention inputs come out
// of a chain of small ops (normalisation, rotary embedding, projection, head
// packing); fused into one kernel, that kernel writes its output in the
// layout the next consumer reads, and the copies that repacked it vanish.
// The readings taken here (the pages name the ops only):
//   xh_t = x_t / sqrt(mean_c x_tc^2 + eps)        RMS normalisation, no gain
//   y_t  = W xh_t = (W x_t) / rms_t               projection, no bias
//   q, k: dims (2p, 2p+1) of token t turn by the angle of table entry (t, p)
//   q, k, v stored bf16 [B, H, N, D]
// The row scale commutes with the projection, so the GEMM multiplies the
// caller's x and the epilogue applies 1 / rms_t (from a small pre-pass).
//
// The epilogue also sums the stored (bf16) keys over each 32-row group, per
// column, in a fixed butterfly order: the key mean that the fixed-max
// statistics need (section "Breaking softmax's dependency chain") then comes
// from these sums, and the prepare pass that re-read k for it is skipped.
//
// Kernel shape (one CTA per SM, persistent): tiles of 128 tokens x BN
// features (BN = 256, or 128 when H * D is not a multiple of 256), 64-wide
// model-dim stages in a 4-deep TMA ring, two TMEM accumulators so the MMA of
// one tile overlaps the epilogue of the previous one.  Each CTA loads its
// own x tile and W tile for every stage.
//   warp 0  TMA producer (x tile 128 x 64, W tile BN x 64)
//   warp 1  MMA issuer: 4 x tcgen05.mma M=128 N=BN K=16 per stage
//   warp 2  TMEM allocation
//   warps 4-7 epilogue: thread = token row (TMEM lane)
// W is loaded evict-last (it is re-read for every token tile) and q, k, v
// are stored evict-first.  The GEMM is a dependent launch after the RMS
// pre-pass: its main loop reads only x and W, and only the epilogue waits
// for the pre-pass's 1/rms values.  Every wait is bounded; after an expired
// one the TMA producer waits (bounded) for its loads in flight.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace wsattn {
namespace {

using namespace ptx;

constexpr int kPStages = 4;
constexpr int kPThreads = 256;
constexpr int kPEpiWarp0 = 4;
constexpr uint32_t kPABytes = kProdTileM * kProdTileK * 2;  // 16 KB
constexpr uint32_t kPOutChunk = 32 * 64 * 2;                // one warp's 32 rows x 64 columns
constexpr long long kPWaitLimit = 1LL << 31;                // about one second

enum : int {
  PB_FULL0 = 0,
  PB_EMPTY0 = kPStages,
  PB_ACCFULL0 = 2 * kPStages,
  PB_ACCEMPTY0 = 2 * kPStages + 2,
  PB_COUNT = 2 * kPStages + 4
};

struct PShared {
  uint32_t stages;   // kPStages x (A tile, B tile)
  uint32_t ostage;   // 4 epilogue warps x 2 staging chunks
  uint32_t bars;
  volatile int* abort_flag;
  int* status;
};

__device__ __forceinline__ uint32_t pbar(const PShared& s, int i) {
  return s.bars + 8u * static_cast<uint32_t>(i);
}

__device__ __noinline__ bool pwait_slow(const PShared& s, uint32_t b, uint32_t parity, int code) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(b, parity)) return true;
    if (*s.abort_flag) return false;
    if (clock64() - t0 > kPWaitLimit) {
      atomicOr(s.status, code);
      *s.abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool pwait(const PShared& s, uint32_t b, uint32_t parity, int code) {
  if (mbar_try_wait(b, parity)) return true;
  return pwait_slow(s, b, parity, code);
}

struct PTile {
  int b, mt, nt;
};

// Work unit t: feature tile nt of token tile mt of batch element b, token
// tile major (the feature tiles of one x slice are consecutive units, so the
// CTAs running at one time share that slice in L2).
__device__ __forceinline__ PTile decode(const ProdParams& p, int t) {
  PTile r;
  r.nt = t % p.ntiles;
  const int rest = t / p.ntiles;
  r.mt = rest % p.mtiles;
  r.b = rest / p.mtiles;
  return r;
}

template <int BN>
__device__ void p_producer(const ProdParams& p, const PShared& s, int total, int cl, int ncl) {
  constexpr uint32_t kStage = kPABytes + BN * kProdTileK * 2;
  const int ksteps = p.c / kProdTileK;
  // W is re-read for every token tile: keep it in L2 ahead of the streams
  const uint64_t keep = policy_evict_last();
  uint32_t slot = 0, phase = 0;
  uint32_t last_phase = 0, issued = 0;  // per slot: parity of its last load, loaded yet
  // after an expired wait: the loads already issued land whatever the
  // consumers do; wait (bounded) for each slot's last one before leaving
  auto drain = [&]() {
    for (int i = 0; i < kPStages; ++i) {
      if (!(issued >> i & 1u)) continue;
      const long long t0 = clock64();
      while (!mbar_try_wait(pbar(s, PB_FULL0 + i), last_phase >> i & 1u))
        if (clock64() - t0 > kPWaitLimit) break;
    }
  };
  for (int t = cl; t < total; t += ncl) {
    const PTile tl = decode(p, t);
    for (int kt = 0; kt < ksteps; ++kt) {
      if (!pwait(s, pbar(s, PB_EMPTY0 + slot), phase ^ 1u, kStatusTimeoutProducer))
        return drain();
      const uint32_t dst = s.stages + slot * kStage;
      mbar_arrive_expect_tx(pbar(s, PB_FULL0 + slot), kStage);
      tma_load_3d(dst, &p.tm_x, pbar(s, PB_FULL0 + slot), kt * kProdTileK, tl.mt * kProdTileM,
                  tl.b);
      tma_load_2d_hint(dst + kPABytes, &p.tm_w, pbar(s, PB_FULL0 + slot), kt * kProdTileK,
                       tl.nt * BN, keep);
      last_phase = (last_phase & ~(1u << slot)) | (phase << slot);
      issued |= 1u << slot;
      if (++slot == kPStages) {
        slot = 0;
        phase ^= 1u;
      }
    }
  }
}

template <int BN>
__device__ void p_mma(const ProdParams& p, const PShared& s, int total, uint32_t tbase, int cl,
                      int ncl) {
  constexpr uint32_t kStage = kPABytes + BN * kProdTileK * 2;
  constexpr uint32_t idesc = idesc_bf16_f32(kProdTileM, BN, false);
  const int ksteps = p.c / kProdTileK;
  uint32_t slot = 0, phase = 0, it = 0;
  for (int t = cl; t < total; t += ncl, ++it) {
    const uint32_t ab = it & 1u, use = it >> 1;
    if (!pwait(s, pbar(s, PB_ACCEMPTY0 + ab), (use & 1u) ^ 1u, kStatusTimeoutMma)) return;
    tc_fence_after();
    const uint32_t d = tbase + ab * BN;
    for (int kt = 0; kt < ksteps; ++kt) {
      if (!pwait(s, pbar(s, PB_FULL0 + slot), phase, kStatusTimeoutMma)) return;
      tc_fence_after();
      const uint32_t a_addr = s.stages + slot * kStage;
      // K-major tiles, 128-byte rows: 16 bf16 of K are 32 bytes further on
      const uint64_t ad = sdesc_sw128(a_addr, 16, 1024);
      const uint64_t bd = sdesc_sw128(a_addr + kPABytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kProdTileK / 16; ++kk)
        mma_ss(d, ad + 2 * kk, bd + 2 * kk, idesc, (kt | kk) != 0 ? 1u : 0u);
      tc_commit(pbar(s, PB_EMPTY0 + slot));  // the slot may be refilled
      if (++slot == kPStages) {
        slot = 0;
        phase ^= 1u;
      }
    }
    tc_commit(pbar(s, PB_ACCFULL0 + ab));
  }
}

// 64 consecutive fp32 columns of this thread's TMEM lane (one wait).
__device__ __forceinline__ void ld64(uint32_t taddr, float (&y)[64]) {
  uint32_t r0[16], r1[16], r2[16], r3[16];
  tmem_ld16(taddr, r0);
  tmem_ld16(taddr + 16, r1);
  tmem_ld16(taddr + 32, r2);
  tmem_ld16(taddr + 48, r3);
  tmem_wait_ld16(r0);
  reg_fence16(r1);
  reg_fence16(r2);
  reg_fence16(r3);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    y[i] = __uint_as_float(r0[i]);
    y[16 + i] = __uint_as_float(r1[i]);
    y[32 + i] = __uint_as_float(r2[i]);
    y[48 + i] = __uint_as_float(r3[i]);
  }
}

// Column sums over the warp's 32 rows of the 64 columns each lane holds
// (a reduce-scatter: at each step a lane keeps half of its columns and adds
// its partner's copy of them).  Lane l returns the sums of columns 2l, 2l+1.
__device__ __forceinline__ float2 warp_colsum64(float (&a)[64]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < 2 * o; ++i) {
      const float keep = upper ? a[i + 2 * o] : a[i];
      const float send = upper ? a[i] : a[i + 2 * o];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return make_float2(a[0], a[1]);
}

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D, int BN>
__device__ void p_epilogue(const ProdParams& p, const PShared& s, int total, uint32_t tbase,
                           int cl, int ncl) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int wq = warp - kPEpiWarp0;  // TMEM lanes 32 wq .. 32 wq + 31
  const int r = 32 * wq + lane;
  const uint32_t tlane = tbase + (static_cast<uint32_t>(32 * wq) << 16);
  const int hd = p.heads * D;
  const uint64_t stream_out = policy_evict_first();  // q, k, v are not read again here
  griddep_wait();  // 1/rms comes from the pre-pass, which may still be running
  uint32_t it = 0, ob = 0;
  for (int t = cl; t < total; t += ncl, ++it) {
    const PTile tl = decode(p, t);
    const uint32_t ab = it & 1u, use = it >> 1;
    const bool ok = pwait(s, pbar(s, PB_ACCFULL0 + ab), use & 1u, kStatusTimeoutSoftmax);
    if (!__all_sync(0xffffffffu, ok)) return;
    tc_fence_after();
    const int tok = tl.mt * kProdTileM + r;
    // the tile lies in the problem: batch element, token tile, feature tile
    const bool tile_ok = WSATTN_BOUNDS(p.status, tl.b >= 0 && tl.b < p.batch && tl.mt >= 0 &&
                                                     tl.mt < p.mtiles && tl.nt >= 0 &&
                                                     tl.nt < p.ntiles);
    const bool valid = tok < p.n && tile_ok;
    const float inv = valid ? p.inv_rms[static_cast<size_t>(tl.b) * p.n + tok] : 0.f;
    const int f0 = tl.nt * BN;
    const int kind = f0 / hd;  // 0 q, 1 k, 2 v
    const int h0 = (f0 - kind * hd) / D;
    const int row0 = tl.mt * kProdTileM + 32 * wq;  // first token of this warp's rows
    const bool any_row = row0 < p.n;
#pragma unroll 1
    for (int j = 0; j < BN / 64; ++j) {
      float y[64];
      ld64(tlane + ab * BN + 64 * j, y);
      if (j == BN / 64 - 1) {  // the accumulator is read: the next tile may use it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pbar(s, PB_ACCEMPTY0 + ab));
      }
      const int h = h0 + (64 * j) / D;
      const int d0 = (64 * j) % D;
#pragma unroll
      for (int i = 0; i < 64; ++i) y[i] *= inv;
      if (kind < 2 && valid) {
        const size_t toff = static_cast<size_t>(tok) * (D / 2) + d0 / 2;
        const float4* cp = reinterpret_cast<const float4*>(p.rope_cos + toff);
        const float4* sp = reinterpret_cast<const float4*>(p.rope_sin + toff);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float4 c4 = __ldg(cp + g), s4 = __ldg(sp + g);
          const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
          const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 2 * (4 * g + e);
            const float a = y[i], b = y[i + 1];
            y[i] = fmaf(a, cs[e], -b * sn[e]);
            y[i + 1] = fmaf(a, sn[e], b * cs[e]);
          }
        }
      }
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = bf16x2(y[2 * i], y[2 * i + 1]);
      const size_t slot = (static_cast<size_t>(tl.b) * p.heads + h) * p.nparts +
                          static_cast<size_t>(tl.mt) * 4 + wq;
      if (kind == 1 && tile_ok &&
          WSATTN_BOUNDS(p.status, h >= 0 && h < p.heads && d0 + 64 <= D &&
                                      slot < static_cast<size_t>(p.batch) * p.heads * p.nparts)) {
        // sums of the stored (rounded) keys; rows past N hold zeros
        float a[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          a[2 * i] = __uint_as_float(pk[i] << 16);
          a[2 * i + 1] = __uint_as_float(pk[i] & 0xFFFF0000u);
        }
        const float2 cs = warp_colsum64(a);
        reinterpret_cast<float2*>(p.part_sum + slot * D + d0)[lane] = cs;
      }
      if (any_row && tile_ok && WSATTN_BOUNDS(p.status, kind >= 0 && kind < 3 && h < p.heads)) {
        // 128-byte swizzle: 16-byte unit u of row l sits at unit u ^ (l & 7)
        const uint32_t buf = s.ostage + (static_cast<uint32_t>(wq) * 2 + ob) * kPOutChunk;
        if (lane == 0) bulk_wait_read_1();  // this buffer's previous store has read it
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(buf + 128u * lane + 16u * (u ^ (lane & 7)), pk[4 * u], pk[4 * u + 1],
                       pk[4 * u + 2], pk[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d_hint(&p.tm_out[kind], buf, d0, row0, tl.b * p.heads + h, stream_out);
          bulk_commit_group();
        }
        ob ^= 1u;
      }
    }
  }
}

template <int D, int BN>
__global__ void __launch_bounds__(kPThreads, 1) produce_kernel(const __grid_constant__ ProdParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr uint32_t kStage = kPABytes + BN * kProdTileK * 2;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  PShared s;
  s.stages = base;
  s.ostage = base + kPStages * kStage;  // 1024-aligned: every stage is a multiple of 1 KB
  s.bars = s.ostage + 8u * kPOutChunk;
  uint8_t* gb = smem_raw + (s.bars - raw);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(gb + 8 * PB_COUNT);
  s.abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  s.status = p.status;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int total = p.batch * p.mtiles * p.ntiles;  // work units
  const int cl = static_cast<int>(blockIdx.x), ncl = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(pbar(s, PB_FULL0 + i), 1);
      mbar_init(pbar(s, PB_EMPTY0 + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(pbar(s, PB_ACCFULL0 + i), 1);
      mbar_init(pbar(s, PB_ACCEMPTY0 + i), 4);  // one arrival per epilogue warp
    }
    *s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.tm_x);
    prefetch_tensormap(&p.tm_w);
    for (int i = 0; i < 3; ++i) prefetch_tensormap(&p.tm_out[i]);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tslot), 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0) p_producer<BN>(p, s, total, cl, ncl);
  } else if (warp == 1) {
    if (lane == 0) p_mma<BN>(p, s, total, tbase, cl, ncl);
  } else if (warp >= kPEpiWarp0) {
    p_epilogue<D, BN>(p, s, total, tbase, cl, ncl);
    if (lane == 0) bulk_wait_all();  // the tile stores must be complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, 2 * BN);
}

// One warp per token: 1 / sqrt(mean_c x_c^2 + eps).  The squares of bf16
// values are exact in fp32; each lane sums its 16-byte words in order and
// the lanes combine in a fixed butterfly, so the result is reproducible.
__global__ void __launch_bounds__(256) rms_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                  int C, float eps, float* __restrict__ inv) {
  // the GEMM that follows reads only x and W until its epilogue: let it start
  griddep_launch_dependents();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * C);
  float ss = 0.f;
#pragma unroll 4
  for (int i = lane; i < C / 8; i += 32) {
    const uint4 u = __ldg(xr + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
      ss = fmaf(lo, lo, ss);
      ss = fmaf(hi, hi, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) inv[row] = 1.0f / sqrtf(ss / static_cast<float>(C) + eps);
}

// Key column sums per head: the epilogue's 32-row group sums reduced to
// kKeySumRows partial rows (the statistics pass adds those in order).  CTA
// (x, bh, z) takes 32 columns of one head and the z-th share of its groups;
// thread (g, c) sums groups g, g + 16, ... of the share into eight
// interleaved accumulators (independent loads in flight), then the
// accumulators and the 16 thread rows combine in a fixed order.
constexpr int kRedRows = 16;
__global__ void __launch_bounds__(32 * kRedRows) reduce_key_sums(const float* __restrict__ parts,
                                                                 int nparts, int D,
                                                                 float* __restrict__ out) {
  __shared__ float red[kRedRows][32];
  griddep_wait();  // the group sums come from the GEMM's epilogue
  const int bh = blockIdx.y, c = 32 * blockIdx.x + threadIdx.x, g = threadIdx.y;
  const int per = (nparts + kKeySumRows - 1) / kKeySumRows;
  const int p0 = static_cast<int>(blockIdx.z) * per;
  const int p1 = min(nparts, p0 + per);
  const float* src = parts + static_cast<size_t>(bh) * nparts * D + c;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  int i = p0 + g;
  for (; i + 7 * kRedRows < p1; i += 8 * kRedRows) {
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] += src[static_cast<size_t>(i + kRedRows * u) * D];
  }
#pragma unroll
  for (int u = 0; u < 8; ++u)
    if (i + kRedRows * u < p1) acc[u] += src[static_cast<size_t>(i + kRedRows * u) * D];
  float sum = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) sum += acc[u];
  red[g][threadIdx.x] = sum;
  __syncthreads();
  if (g == 0) {
    float t = 0.f;
    for (int r = 0; r < kRedRows; ++r) t += red[r][threadIdx.x];
    out[(static_cast<size_t>(bh) * kKeySumRows + blockIdx.z) * D + c] = t;
  }
}

// A persistent grid: one CTA per SM, at most one per work unit.
template <int D, int BN>
cudaError_t launch_gemm(const ProdParams& p, int max_ctas, cudaStream_t stream) {
  static bool attr_set[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  const size_t smem = produce_smem_bytes(BN);
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        produce_kernel<D, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int units = p.batch * p.mtiles * p.ntiles;
  int grid = max_ctas < units ? max_ctas : units;
  if (grid < 1) grid = 1;
  // dependent launch: the GEMM's main loop (x and W only) overlaps the RMS
  // pre-pass; the epilogue waits for its 1/rms values
  return launch_dependent(produce_kernel<D, BN>, dim3(grid), dim3(kPThreads), smem, stream, p);
}

}  // namespace

int produce_tile_n(int heads, int head_dim) {
  const int hd = heads * head_dim;
  if (hd % 256 == 0) return 256;
  if (hd % 128 == 0) return 128;
  return 0;
}

size_t produce_smem_bytes(int bn) {
  const size_t stage = kPABytes + static_cast<size_t>(bn) * kProdTileK * 2;
  return 1024 + kPStages * stage + 8 * kPOutChunk + 8 * PB_COUNT + 16;
}

cudaError_t launch_produce(const ProdParams& p, const uint16_t* x, float eps, int D, int bn,
                           int grid, float* inv_rms, float* key_sums, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.batch) * p.n;
  rms_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(x, rows, p.c, eps,
                                                                       inv_rms);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (D == 128)
    e = bn == 256 ? launch_gemm<128, 256>(p, grid, stream) : launch_gemm<128, 128>(p, grid, stream);
  else
    e = bn == 256 ? launch_gemm<64, 256>(p, grid, stream) : launch_gemm<64, 128>(p, grid, stream);
  if (e != cudaSuccess) return e;
  const int BH = p.batch * p.heads;
  return launch_dependent(reduce_key_sums, dim3(D / 32, BH, kKeySumRows), dim3(32, kRedRows), 0,
                          stream,
                          static_cast<const float*>(p.part_sum), p.nparts, D, key_sums);
}

}  // namespace wsattn
