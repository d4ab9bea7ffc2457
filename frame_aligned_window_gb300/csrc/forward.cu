// Fused frame-aligned window-sparse attention forward for sm_103a.
//
// Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
// TPUs":
//   - "Deleting the mask" (Fig. 3): key blocks divide the frame span, so each
//     query tile visits only fully active key blocks -- reference frame and
//     window alike, in one pass -- with no mask predicate and no padding.
//   - "Breaking softmax's dependency chain" (Fig. 4): on eligible heads the
//     row bound is the softmax max, so a block's probabilities are
//     p = exp(scale*s - m_i) with no running max and no rescale in the loop
//     (m_i = b_i + scale q_i.mu: the bound of the centered logits, shifted
//     back to the logits of the keys as given);
//     ineligible heads run the online max (rescaling O and l) in the same
//     kernel, chosen per tile.
//   - "Proving pixels unchanged": the PV product takes P in bf16.
//
// Persistent kernel, one CTA per SM, 8 warps:
//   warp 0      TMA producer: Q tile (128 x D) into a staging buffer; K and V
//               blocks (bk x D) into two rings, all 128-byte swizzled.
//   warp 1      MMA issuer (one thread): S = Q K^T and O += P V with
//               tcgen05.mma kind::f16 (bf16 in, fp32 accumulate in TMEM).
//               Q and P are read from TMEM, K and V from shared memory.
//   warps 4-7   softmax + epilogue warpgroup: thread i owns row i of the
//               tile (TMEM lane i), so row sums are thread-local.
// Tensor memory (512 columns): O [0, D), S0/S1 double buffer of bk columns
// each (P aliases the first bk/2 columns of its S buffer as bf16 pairs), Q
// (D/2 columns of bf16 pairs).  While the softmax works on S(j), the tensor
// core runs PV(j-1) and QK(j+1).
//
// Every wait is bounded: on expiry the kernel sets a bit in the status word,
// raises a CTA-wide abort flag, and all roles leave their loops; TMEM is
// released on the way out.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace wsattn {
namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr long long kWaitLimitCycles = 1LL << 31;  // about one second
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;

// mbarrier slots
enum : int {
  B_QFULL = 0,   // TMA -> softmax: Q tile staged in smem
  B_QEMPTY,      // softmax -> TMA: Q staging buffer free
  B_QTFULL,      // softmax -> MMA: Q tile in TMEM
  B_OBAR,        // MMA -> softmax: PV(j) done (online path only)
  B_OFULL,       // MMA -> softmax: last PV of the tile done
  B_SFULL0,      // MMA -> softmax: S buffer 0 / 1 written
  B_SFULL1,
  B_PFULL0,      // softmax -> MMA: P buffer 0 / 1 written
  B_PFULL1,
  B_KFULL0,
  B_KEMPTY0 = B_KFULL0 + 4,
  B_VFULL0 = B_KEMPTY0 + 4,
  B_VEMPTY0 = B_VFULL0 + 4,
  B_COUNT = B_VEMPTY0 + 4
};

struct Shared {
  uint32_t q, k, v, bars;  // shared-window addresses
  volatile int* abort_flag;
  int* status;
};

__device__ __forceinline__ uint32_t bar(const Shared& s, int i) {
  return s.bars + 8u * static_cast<uint32_t>(i);
}

__device__ __noinline__ bool wait_slow(const Shared& s, uint32_t b, uint32_t parity, int code) {
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(b, parity)) return true;
    if (*s.abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicOr(s.status, code);
      *s.abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool wait(const Shared& s, uint32_t b, uint32_t parity, int code) {
  if (mbar_try_wait(b, parity)) return true;
  return wait_slow(s, b, parity, code);
}

// Warp-uniform wait for the softmax warps: every lane waits, then the warp
// agrees (and reconverges) before any .sync.aligned tcgen05 instruction.
__device__ __forceinline__ bool wait_warp(const Shared& s, uint32_t b, uint32_t parity) {
  const bool ok = wait(s, b, parity, kStatusTimeoutSoftmax);
  return __all_sync(0xffffffffu, ok);
}

struct TmemCols {
  uint32_t o, s0, s1, q;
};

template <int D>
__device__ __forceinline__ TmemCols tmem_cols(int bk) {
  const uint32_t spad = (static_cast<uint32_t>(bk) + 31u) & ~31u;
  return TmemCols{0u, static_cast<uint32_t>(D), static_cast<uint32_t>(D) + spad,
                  static_cast<uint32_t>(D) + 2u * spad};
}

// ------------------------------------------------------------------ producer
template <int D>
__device__ void producer(const FwdParams& p, const Shared& s) {
  constexpr int kBoxes = D / 64;
  const uint32_t box_bytes = static_cast<uint32_t>(p.bk) * 128u;
  const uint32_t stage_bytes = box_bytes * kBoxes;
  const int n_items = p.n_tiles * p.bh;
  uint32_t kc = 0, vc = 0, qc = 0;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const WorkTile t = p.tiles[it / p.bh];
    const int y0 = (it % p.bh) * p.n;
    if (!wait(s, bar(s, B_QEMPTY), (qc & 1u) ^ 1u, kStatusTimeoutProducer)) return;
    mbar_arrive_expect_tx(bar(s, B_QFULL), kTileM * D * 2);
#pragma unroll
    for (int c = 0; c < kBoxes; ++c)
      tma_load_2d(s.q + c * (kTileM * 128), &p.tm_q, bar(s, B_QFULL), c * 64, y0 + t.row0);
    ++qc;
    const int nblk = t.kend - t.kbeg;
    // Issue order follows consumption: K0, K1, V0, K2, V1, ...
    for (int j = 0; j <= nblk; ++j) {
      if (j < nblk) {
        const int row = y0 + p.kcol[t.kbeg + j] * p.bk;
        const uint32_t slot = kc % static_cast<uint32_t>(p.stages_k);
        const uint32_t ph = (kc / static_cast<uint32_t>(p.stages_k)) & 1u;
        if (!wait(s, bar(s, B_KEMPTY0 + slot), ph ^ 1u, kStatusTimeoutProducer)) return;
        mbar_arrive_expect_tx(bar(s, B_KFULL0 + slot), stage_bytes);
#pragma unroll
        for (int c = 0; c < kBoxes; ++c)
          tma_load_2d(s.k + slot * stage_bytes + c * box_bytes, &p.tm_k, bar(s, B_KFULL0 + slot),
                      c * 64, row);
        ++kc;
      }
      if (j >= 1) {
        const int row = y0 + p.kcol[t.kbeg + j - 1] * p.bk;
        const uint32_t slot = vc % static_cast<uint32_t>(p.stages_v);
        const uint32_t ph = (vc / static_cast<uint32_t>(p.stages_v)) & 1u;
        if (!wait(s, bar(s, B_VEMPTY0 + slot), ph ^ 1u, kStatusTimeoutProducer)) return;
        mbar_arrive_expect_tx(bar(s, B_VFULL0 + slot), stage_bytes);
#pragma unroll
        for (int c = 0; c < kBoxes; ++c)
          tma_load_2d(s.v + slot * stage_bytes + c * box_bytes, &p.tm_v, bar(s, B_VFULL0 + slot),
                      c * 64, row);
        ++vc;
      }
    }
  }
}

// ---------------------------------------------------------------- MMA issuer
template <int D>
__device__ void mma_issuer(const FwdParams& p, const Shared& s, uint32_t tbase) {
  constexpr int kBoxes = D / 64;
  const int bk = p.bk;
  const uint32_t box_bytes = static_cast<uint32_t>(bk) * 128u;
  const uint32_t stage_bytes = box_bytes * kBoxes;
  const TmemCols tc_ = tmem_cols<D>(bk);
  const uint32_t t_o = tbase + tc_.o, t_s0 = tbase + tc_.s0, t_s1 = tbase + tc_.s1;
  const uint32_t t_q = tbase + tc_.q;
  const uint32_t id_qk = idesc_bf16_f32(kTileM, bk, false);
  const uint32_t id_pv = idesc_bf16_f32(kTileM, D, true);
  const int n_items = p.n_tiles * p.bh;
  uint32_t kc = 0, vc = 0, pc0 = 0, pc1 = 0, tiles_done = 0;

  // S(j) = Q K_j^T into S buffer (j & 1).
  auto issue_qk = [&](int j) -> bool {
    const uint32_t slot = kc % static_cast<uint32_t>(p.stages_k);
    const uint32_t ph = (kc / static_cast<uint32_t>(p.stages_k)) & 1u;
    if (!wait(s, bar(s, B_KFULL0 + slot), ph, kStatusTimeoutMma)) return false;
    tc_fence_after();
    const uint32_t kbase = s.k + slot * stage_bytes;
    const uint32_t d_s = (j & 1) ? t_s1 : t_s0;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint64_t bdesc = sdesc_sw128(kbase + (kk / 4) * box_bytes + (kk % 4) * 32, 16, 1024);
      mma_ts(d_s, t_q + kk * 8, bdesc, id_qk, kk > 0 ? 1u : 0u);
    }
    tc_commit(bar(s, B_KEMPTY0 + slot));
    tc_commit(bar(s, (j & 1) ? B_SFULL1 : B_SFULL0));
    ++kc;
    return true;
  };

  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const WorkTile t = p.tiles[it / p.bh];
    const int bh = it % p.bh;
    const int nblk = t.kend - t.kbeg;
    const bool online = p.force_path >= 0 ? (p.force_path == 1) : (p.elig[bh] == 0);
    if (!wait(s, bar(s, B_QTFULL), tiles_done & 1u, kStatusTimeoutMma)) return;
    tc_fence_after();
    for (int j = 0; j < nblk && j < 2; ++j)
      if (!issue_qk(j)) return;
    for (int j = 0; j < nblk; ++j) {
      const int sb = j & 1;
      uint32_t par;
      if (sb) { par = pc1 & 1u; ++pc1; } else { par = pc0 & 1u; ++pc0; }
      if (!wait(s, bar(s, B_PFULL0 + sb), par, kStatusTimeoutMma)) return;
      tc_fence_after();
      const uint32_t vslot = vc % static_cast<uint32_t>(p.stages_v);
      const uint32_t vph = (vc / static_cast<uint32_t>(p.stages_v)) & 1u;
      if (!wait(s, bar(s, B_VFULL0 + vslot), vph, kStatusTimeoutMma)) return;
      tc_fence_after();
      const uint32_t vbase = s.v + vslot * stage_bytes;
      const uint32_t a_p = sb ? t_s1 : t_s0;
      for (int kk = 0; kk < bk / 16; ++kk) {
        // V is MN-major: 16 key rows per step (2 KB), D split in 64-wide
        // boxes box_bytes apart (leading byte offset), 8-row groups 1 KB apart.
        const uint64_t bdesc = sdesc_sw128(vbase + kk * 2048, box_bytes, 1024);
        mma_ts(t_o, a_p + kk * 8, bdesc, id_pv, (j > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(bar(s, B_VEMPTY0 + vslot));
      ++vc;
      if (online && j + 1 < nblk) tc_commit(bar(s, B_OBAR));
      if (j + 2 < nblk && !issue_qk(j + 2)) return;
    }
    tc_commit(bar(s, B_OFULL));
    ++tiles_done;
  }
}

// -------------------------------------------------------------- softmax WG
// Copies this thread's Q row from the swizzled staging tile into TMEM (bf16
// pairs, column c holds elements 2c, 2c+1); rows past the frame are zeroed.
template <int D>
__device__ bool load_q(const Shared& s, uint32_t t_q, int r, int nvalid, uint32_t& qc) {
  if (!wait_warp(s, bar(s, B_QFULL), qc & 1u)) return false;
  ++qc;
  const bool zero = r >= nvalid;
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint32_t row_addr = s.q + c * (kTileM * 128) + r * 128;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t m = static_cast<uint32_t>(2 * h + e);
        const uint4 v = ld_shared_v4(row_addr + ((m ^ static_cast<uint32_t>(r & 7)) << 4));
        w[4 * e + 0] = zero ? 0u : v.x;
        w[4 * e + 1] = zero ? 0u : v.y;
        w[4 * e + 2] = zero ? 0u : v.z;
        w[4 * e + 3] = zero ? 0u : v.w;
      }
      tmem_st8(t_q + c * 32 + h * 8, w);
    }
  }
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(bar(s, B_QTFULL));
  mbar_arrive(bar(s, B_QEMPTY));
  return true;
}

// p = 2^(s*c + nb) for 16 logits; adds them to l (pairwise) and stores the
// bf16 pairs as 8 TMEM columns at taddr.
__device__ __forceinline__ void exp_pack_store(const uint32_t (&sv)[16], float c, float nb,
                                               float& l, uint32_t taddr) {
  uint32_t w[8];
  float ps[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float p0 = ex2_approx(fmaf(__uint_as_float(sv[2 * i]), c, nb));
    const float p1 = ex2_approx(fmaf(__uint_as_float(sv[2 * i + 1]), c, nb));
    ps[i] = p0 + p1;
    const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  tmem_st8(taddr, w);
  l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
}

// Fixed-max path: nb = -m_i * log2(e).
__device__ __forceinline__ bool fixed_block(uint32_t sa, int nch, float c, float nb, float& l0,
                                            float& l1) {
  uint32_t ra[16], rb[16];
  tmem_ld16(sa, ra);
  tmem_wait_ld16(ra);
  for (int k = 0; k < nch; k += 2) {
    const bool has_b = k + 1 < nch;
    if (has_b) tmem_ld16(sa + (k + 1) * 16, rb);
    exp_pack_store(ra, c, nb, l0, sa + k * 8);
    if (has_b) {
      tmem_wait_ld16(rb);
      const bool has_a = k + 2 < nch;
      if (has_a) tmem_ld16(sa + (k + 2) * 16, ra);
      exp_pack_store(rb, c, nb, l1, sa + (k + 1) * 8);
      if (has_a) tmem_wait_ld16(ra);
    }
  }
  return true;
}

template <int D>
__device__ void softmax_wg(const FwdParams& p, const Shared& s, uint32_t tbase) {
  const int warp = threadIdx.x / 32;
  const int r = threadIdx.x - kSoftmaxWarp0 * 32;  // tile row == TMEM lane
  const uint32_t lane = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const TmemCols tc_ = tmem_cols<D>(p.bk);
  const int nch = p.bk / 16;
  const float c = p.scale_log2;
  const int n_items = p.n_tiles * p.bh;
  uint32_t qc = 0, sc0 = 0, sc1 = 0, oc = 0, tiles_done = 0;

  int it = blockIdx.x;
  if (it >= n_items) return;
  if (!load_q<D>(s, lane + tc_.q, r, p.tiles[it / p.bh].nvalid, qc)) return;
  while (true) {
    const WorkTile t = p.tiles[it / p.bh];
    const int bh = it % p.bh;
    const int nblk = t.kend - t.kbeg;
    const bool online = p.force_path >= 0 ? (p.force_path == 1) : (p.elig[bh] == 0);
    const bool valid = r < t.nvalid;
    const size_t grow = static_cast<size_t>(bh) * p.n + t.row0 + r;
    float l = 0.f;
    if (!online) {
      const float nb = valid ? -p.m_rows[grow] * kLog2e : 0.f;
      float l0 = 0.f, l1 = 0.f;
      for (int j = 0; j < nblk; ++j) {
        const int sb = j & 1;
        uint32_t par;
        if (sb) { par = sc1 & 1u; ++sc1; } else { par = sc0 & 1u; ++sc0; }
        if (!wait_warp(s, bar(s, B_SFULL0 + sb), par)) return;
        tc_fence_after();
        fixed_block(lane + (sb ? tc_.s1 : tc_.s0), nch, c, nb, l0, l1);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(s, B_PFULL0 + sb));
      }
      l = l0 + l1;
    } else {
      float m = -INFINITY;
      for (int j = 0; j < nblk; ++j) {
        const int sb = j & 1;
        uint32_t par;
        if (sb) { par = sc1 & 1u; ++sc1; } else { par = sc0 & 1u; ++sc0; }
        if (!wait_warp(s, bar(s, B_SFULL0 + sb), par)) return;
        tc_fence_after();
        const uint32_t sa = lane + (sb ? tc_.s1 : tc_.s0);
        float mx = -INFINITY;
        for (int k = 0; k < nch; ++k) {
          uint32_t ra[16];
          tmem_ld16(sa + k * 16, ra);
          tmem_wait_ld16(ra);
#pragma unroll
          for (int i = 0; i < 16; ++i) mx = fmaxf(mx, __uint_as_float(ra[i]));
        }
        const float m_new = fmaxf(m, mx * c);
        const float alpha = ex2_approx(m - m_new);
        float ls = 0.f;
        for (int k = 0; k < nch; ++k) {
          uint32_t ra[16];
          tmem_ld16(sa + k * 16, ra);
          tmem_wait_ld16(ra);
          exp_pack_store(ra, c, -m_new, ls, sa + k * 8);
        }
        l = l * alpha + ls;
        m = m_new;
        if (j > 0) {
          // O += P(j-1) V must have landed before it is rescaled.
          if (!wait_warp(s, bar(s, B_OBAR), oc & 1u)) return;
          ++oc;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha < 1.f)) {
            for (int k = 0; k < D / 16; ++k) {
              uint32_t ra[16];
              tmem_ld16(lane + tc_.o + k * 16, ra);
              tmem_wait_ld16(ra);
#pragma unroll
              for (int i = 0; i < 16; ++i) ra[i] = __float_as_uint(__uint_as_float(ra[i]) * alpha);
              tmem_st16(lane + tc_.o + k * 16, ra);
            }
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(s, B_PFULL0 + sb));
      }
    }

    // Stage the next tile's Q so its first QK products overlap this epilogue.
    const int nxt = it + static_cast<int>(gridDim.x);
    if (nxt < n_items && !load_q<D>(s, lane + tc_.q, r, p.tiles[nxt / p.bh].nvalid, qc)) return;

    if (!wait_warp(s, bar(s, B_OFULL), tiles_done & 1u)) return;
    ++tiles_done;
    tc_fence_after();
    const float inv = 1.f / l;
    float* orow = p.out + grow * D;
#pragma unroll 1
    for (int k = 0; k < D / 16; ++k) {
      uint32_t v[16];
      tmem_ld16(lane + tc_.o + k * 16, v);
      tmem_wait_ld16(v);
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(orow + k * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                               __uint_as_float(v[4 * i + 2]) * inv,
                               __uint_as_float(v[4 * i + 3]) * inv);
      }
    }
    if (nxt >= n_items) break;
    it = nxt;
  }
}

// -------------------------------------------------------------------- kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1) wsattn_fwd_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t stage_bytes = static_cast<uint32_t>(p.bk) * D * 2u;
  Shared s;
  s.q = base;
  s.k = base + kTileM * D * 2;
  s.v = s.k + static_cast<uint32_t>(p.stages_k) * stage_bytes;
  s.bars = s.v + static_cast<uint32_t>(p.stages_v) * stage_bytes;
  uint8_t* gbars = smem_raw + (s.bars - raw);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(gbars + 8 * B_COUNT);
  s.abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  s.status = p.status;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(bar(s, B_QFULL), 1);
    mbar_init(bar(s, B_QEMPTY), kTileM);
    mbar_init(bar(s, B_QTFULL), kTileM);
    mbar_init(bar(s, B_OBAR), 1);
    mbar_init(bar(s, B_OFULL), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(s, B_SFULL0 + i), 1);
      mbar_init(bar(s, B_PFULL0 + i), kTileM);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(s, B_KFULL0 + i), 1);
      mbar_init(bar(s, B_KEMPTY0 + i), 1);
      mbar_init(bar(s, B_VFULL0 + i), 1);
      mbar_init(bar(s, B_VEMPTY0 + i), 1);
    }
    *s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.tm_q);
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tslot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0) producer<D>(p, s);
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<D>(p, s, tbase);
  } else if (warp >= kSoftmaxWarp0) {
    softmax_wg<D>(p, s, tbase);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, kTmemCols);
}

__global__ void timeout_selftest_kernel(long long limit_cycles, int* status) {
  __shared__ __align__(8) uint64_t b;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&b), 1);
    fence_barrier_init();
    int st = 0;
    const long long t0 = clock64();
    // Nothing ever arrives on b: this wait can only end by the limit.
    while (!mbar_try_wait(smem_u32(&b), 0)) {
      if (clock64() - t0 > limit_cycles) {
        st = kStatusTimeoutSelftest;
        break;
      }
    }
    *status = st;
  }
}

}  // namespace

size_t forward_smem_bytes(int D, int bk, int stages_k, int stages_v) {
  const size_t stage = static_cast<size_t>(bk) * D * 2;
  return 1024 + static_cast<size_t>(kTileM) * D * 2 + (stages_k + stages_v) * stage +
         8 * B_COUNT + 16;
}

void forward_stages(int D, int bk, size_t smem_optin, int* stages_k, int* stages_v) {
  int st = 4;
  while (st > 1 && forward_smem_bytes(D, bk, st, st) > smem_optin) --st;
  *stages_k = st;
  *stages_v = st;
}

cudaError_t launch_forward(const FwdParams& p, int D, int grid, size_t smem, cudaStream_t stream) {
  static bool attr_set[2] = {false, false};
  const int idx = D == 128 ? 1 : 0;
  cudaError_t e = cudaSuccess;
  if (!attr_set[idx]) {
    e = D == 128 ? cudaFuncSetAttribute(wsattn_fwd_kernel<128>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, 232448)
                 : cudaFuncSetAttribute(wsattn_fwd_kernel<64>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set[idx] = true;
  }
  if (D == 128)
    wsattn_fwd_kernel<128><<<grid, kThreads, smem, stream>>>(p);
  else
    wsattn_fwd_kernel<64><<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_timeout_selftest(long long limit_cycles, int* status, cudaStream_t stream) {
  timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_cycles, status);
  return cudaGetLastError();
}

}  // namespace wsattn
