// Fused frame-aligned window-sparse attention forward for sm_103a.
//
// Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
// TPUs":
//   - "Deleting the mask" (Fig. 3): key blocks divide the frame span, so each
//     query tile visits only fully active key blocks -- reference frame and
//     window alike, in one pass -- with no mask predicate and no padding.
//     Frames whose token span is not a multiple of 128 end in short tails;
//     consecutive frames' tails share one tile whose key list is the union
//     of theirs.  There, and only there, a row zeroes the 16-key chunks of
//     the union that its own frame does not attend (still whole chunks of
//     fully active or skipped blocks, never single elements).
//   - "Breaking softmax's dependency chain" (Fig. 4): on eligible heads the
//     row bound is the softmax max, so a block's probabilities are
//     p = exp(scale*s - m_i) with no running max and no rescale in the loop
//     (m_i = b_i + scale q_i.mu: the bound of the centered logits, shifted
//     back to the logits of the keys as given); ineligible heads run the
//     online max (rescaling O and l) in the same kernel, chosen per tile.
//   - "Proving pixels unchanged": the PV product takes P in bf16.
//
// Persistent kernel, one CTA per SM, 12 warps:
//   warps 0, 2  TMA producers (one thread each): warp 0 loads the Q tile
//               (128 x D) into a staging buffer and the K steps, warp 2 the V
//               steps, into two rings, all 128-byte swizzled.
//   warps 1, 3  MMA issuers (whole warps, one elected lane issuing each
//               instruction): S = Q K^T and O += P V with
//               tcgen05.mma kind::f16 (bf16 in, fp32 accumulate in TMEM).
//               Q and P are read from TMEM, K and V from shared memory.
//               Warp 2 also allocates and frees tensor memory.
//   warps 4-11  two softmax + epilogue warpgroups (kNumWG).  Thread i of a
//               warpgroup owns row i of the tile (TMEM lane i); the 16-column
//               chunks of a key step are split over the warpgroups in order
//               (warpgroup 0 takes ceil(chunks / 2)), so each SMSP runs two
//               softmax warps.
//
// Keys are consumed in steps of up to G consecutive active blocks of one run
// (G * bk <= 160 keys): the step's rows are consecutive, so K and V arrive as
// one TMA box per 64-column slab, and each MMA covers the whole step.
//
// Tensor memory (512 columns at D = 128, 160-key steps): O [0, D), one S
// buffer (step columns), two P buffers (step/2 columns of bf16 pairs each),
// Q (D/2 columns of bf16 pairs).  A softmax warp starts a step by loading its
// S columns into registers and signalling that S is free, so QK^T(j+1)
// refills S while the softmax of step j computes; P(j) goes to its own
// buffer (j mod 2), which the PV of step j reads while the softmax already
// writes P(j+1) to the other one.  The only round trip through the tensor
// core that the softmax waits on is thus load S(j) -> QK^T(j+1) -> S full,
// and PV runs beside it.
//
// Work items (tile, b*h) are ordered class by class (tiles with equal key
// lists, longest first) and head by head inside a class, so the CTAs running
// at one time stream the same head's keys and values through L2.  They are
// dealt out on the device: a CTA's TMA warp takes the next index from a
// global counter two key steps before it has loaded the current item's last
// keys, decodes it (tile, b*h and the tile's record) and passes it to the
// CTA's other roles through a small queue in shared memory, so the items go
// to whichever CTA is free first (list scheduling in the longest-first order)
// and the deal adapts to the actual cost of each item (online heads are
// slower).  The next item's Q tile is loaded while the current one runs.
// The last CTA to finish resets the counter.  The kernel is a dependent
// launch: its prologue overlaps the end of the statistics pass before it.
//
// Every wait is bounded: on expiry the kernel sets a bit in the status word,
// raises a CTA-wide abort flag, and all roles leave their loops; the TMA
// producer first waits (bounded) for the loads it has in flight, and TMEM is
// released on the way out.
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace wsattn {
namespace {

using namespace ptx;

constexpr int kNumWG = 2;  // softmax warpgroups (3 and 4 measured slower: more arrivals, fewer registers)
constexpr int kSoftmaxWarp0 = 4;
constexpr int kSoftmaxWarps = 4 * kNumWG;
constexpr int kThreads = 32 * (kSoftmaxWarp0 + kSoftmaxWarps);
constexpr int kMaxChunksAll = (10 + kNumWG - 1) / kNumWG;   // chunks a warpgroup takes at 160 keys
constexpr long long kWaitLimitCycles = 1LL << 31;  // about one second
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyMax = 8.f;  // online path: rescale when the max grows by > 2^8
constexpr uint32_t kTmemCols = 512;
// Work items are dealt out on the device: the TMA warp takes the next index
// from a global counter and passes it to the CTA's other roles through a
// small queue in shared memory.
constexpr int kItemQueue = 4;
// A queue slot: the item index (-1: none left), its tile and b*h, and the
// tile's record, decoded once by the TMA warp.
constexpr int kQWords = 4 + static_cast<int>(sizeof(WorkTile) / 4);
constexpr uint32_t kItemReaders = 3 + kSoftmaxWarps;  // V producer, both issuers, every softmax warp

// mbarrier slots
enum : int {
  B_QFULL = 0,   // TMA -> softmax: Q tile staged in smem
  B_QEMPTY,      // softmax -> TMA: Q staging buffer free
  B_QTFULL,      // softmax -> MMA: Q tile in TMEM
  B_OFULL,       // MMA -> softmax: last PV of the tile done
  B_XCH,         // softmax <-> softmax: row maxima / row sums exchanged
  B_SFULL,       // MMA -> softmax: S written (one phase per key step)
  B_SEMPTY,      // softmax -> MMA: every softmax warp holds its S columns
  B_PFULL0,      // softmax -> MMA: P buffer 0 / 1 written
  B_PFULL1,
  B_PVDONE0,     // MMA -> softmax: the PV that read P buffer 0 / 1 done
  B_PVDONE1,
  B_KFULL0,
  B_KEMPTY0 = B_KFULL0 + 4,
  B_VFULL0 = B_KEMPTY0 + 4,
  B_VEMPTY0 = B_VFULL0 + 4,
  B_IQFULL0 = B_VEMPTY0 + 4,     // TMA warp -> the other roles: work item in queue slot
  B_IQEMPTY0 = B_IQFULL0 + kItemQueue,  // every role has read the slot
  B_COUNT = B_IQEMPTY0 + kItemQueue
};
// Exchange area after the barriers: row maxima and row sums of the
// warpgroups, double-buffered: float [2 parity][kNumWG][128 rows] each.
constexpr uint32_t kXchBytes = 2 * 2 * kNumWG * 128 * 4;
// Epilogue staging after the exchange area (128-byte aligned): one 32-row x
// 16-column fp32 chunk (2 KB) per softmax warp, written row by row and sent
// to global memory by one TMA store.
constexpr uint32_t kOChunkBytes = 32 * 16 * 4;
constexpr uint32_t kOStageBytes = kSoftmaxWarps * kOChunkBytes;

struct Shared {
  uint32_t q, k, v, bars;  // shared-window addresses
  uint32_t ostage;         // epilogue staging chunks (kOChunkBytes per softmax warp)
  float* xch_m;            // [2][kNumWG][128]
  volatile int32_t* iq;    // [kItemQueue][kQWords] decoded work items
  float* xch_l;            // [2][kNumWG][128]
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

// Position in the work-item queue.
struct ItemPos {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == kItemQueue) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Arrival of one softmax warp: the warp's threads synchronise (ordering
// every lane's prior shared-memory writes and fenced tcgen05 operations
// before it) and lane 0 arrives.  Barriers the softmax warps signal count
// one arrival per warp: 256 arrivals on one mbarrier serialise in the
// shared-memory atomic unit and stall the warps' next barrier operation for
// hundreds of cycles.
__device__ __forceinline__ void warp_arrive(uint32_t b) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(b);
}

struct Item {
  int tile, bh;
};

// Work item -> (tile, b*h): classes in order, heads in order inside a class.
__device__ __forceinline__ Item map_item(const FwdParams& p, int it) {
  int c = 0;
  while (c + 1 < p.n_cls && it >= p.bh * __ldg(p.cls + c + 1)) ++c;
  const int beg = __ldg(p.cls + c);
  const int n = __ldg(p.cls + c + 1) - beg;
  const int o = it - p.bh * beg;
  return Item{beg + o % n, o / n};
}

// TMA warp: takes the next work item from the launch's counter, decodes it
// and posts it to the queue.  Returns the item, -1 once none is left (posted
// too, so the other roles stop), -2 on an expired wait.
__device__ __forceinline__ int post_item(const FwdParams& p, const Shared& s, ItemPos& q,
                                         int n_items, Item& im, WorkTile& t) {
  if (!wait(s, bar(s, B_IQEMPTY0 + q.slot), q.phase ^ 1u, kStatusTimeoutProducer)) return -2;
  int it = atomicAdd(p.work, 1);
  if (it >= n_items) it = -1;
  volatile int32_t* e = s.iq + q.slot * kQWords;
  if (it >= 0) {
    im = map_item(p, it);
    if (!WSATTN_BOUNDS(p.status, im.tile >= 0 && im.tile < p.n_tiles && im.bh >= 0 &&
                                     im.bh < p.bh))
      im = Item{0, 0};
    t = p.tiles[im.tile];
    e[1] = im.tile;
    e[2] = im.bh;
    const int32_t* tw = reinterpret_cast<const int32_t*>(&t);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(WorkTile) / 4); ++i) e[4 + i] = tw[i];
  }
  e[0] = it;
  mbar_arrive(bar(s, B_IQFULL0 + q.slot));
  q.next();
  return it;
}

// The decoded item of a queue slot.
__device__ __forceinline__ int slot_item(const Shared& s, uint32_t slot, Item& im, WorkTile& t) {
  const volatile int32_t* e = s.iq + slot * kQWords;
  const int it = e[0];
  if (it >= 0) {
    im.tile = e[1];
    im.bh = e[2];
    int32_t* tw = reinterpret_cast<int32_t*>(&t);
#pragma unroll
    for (int i = 0; i < static_cast<int>(sizeof(WorkTile) / 4); ++i) tw[i] = e[4 + i];
  }
  return it;
}

// An issuer thread's next work item (-1: none left, -2: expired wait).
__device__ __forceinline__ int read_item(const Shared& s, ItemPos& q, int code, Item& im,
                                         WorkTile& t) {
  if (!wait(s, bar(s, B_IQFULL0 + q.slot), q.phase, code)) return -2;
  const int it = slot_item(s, q.slot, im, t);
  mbar_arrive(bar(s, B_IQEMPTY0 + q.slot));
  q.next();
  return it;
}

// The MMA issuers are whole warps (each instruction issued by one elected
// lane): every lane waits, and the warp reconverges before the next MMA.
__device__ __forceinline__ bool wait_issuer(const Shared& s, uint32_t b, uint32_t parity) {
  return __all_sync(0xffffffffu, wait(s, b, parity, kStatusTimeoutMma));
}

// An issuer warp's next work item: every lane waits and reads, one arrives.
__device__ __forceinline__ int read_item_issuer(const Shared& s, ItemPos& q, Item& im,
                                                WorkTile& t) {
  if (!wait_issuer(s, bar(s, B_IQFULL0 + q.slot), q.phase)) return -2;
  const int it = slot_item(s, q.slot, im, t);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar(s, B_IQEMPTY0 + q.slot));
  q.next();
  return it;
}

// A softmax warp's next work item (warp-uniform; one arrival per warp).
__device__ __forceinline__ int read_item_warp(const Shared& s, ItemPos& q, Item& im,
                                             WorkTile& t) {
  if (!wait_warp(s, bar(s, B_IQFULL0 + q.slot), q.phase)) return -2;
  const int it = slot_item(s, q.slot, im, t);
  warp_arrive(bar(s, B_IQEMPTY0 + q.slot));
  q.next();
  return it;
}

// Barrier of the two softmax warpgroups (every warp arrives, then waits for
// the phase), bounded like every other wait; the arrival publishes the
// exchange values written before it.
__device__ __forceinline__ bool xch_sync(const Shared& s, uint32_t& xc) {
  warp_arrive(bar(s, B_XCH));
  const bool ok = wait_warp(s, bar(s, B_XCH), xc & 1u);
  ++xc;
  return ok;
}

// The share of warpgroup w when n units (16-column chunks of a key step, or
// 16-element groups of D) are split over the warpgroups: the earlier
// warpgroups take the larger shares; first = units before w's.
__device__ __forceinline__ void wg_share(int n, int w, int& first, int& count) {
  first = 0;
#pragma unroll
  for (int v = 0; v < kNumWG - 1; ++v)
    if (v < w) first += (n + kNumWG - 1 - v) / kNumWG;
  count = (n + kNumWG - 1 - w) / kNumWG;
}

// Tensor-memory columns: O [0, D), S [D, D + step), P buffers of step/2
// columns from D + step, Q (D/2 columns) after them.
struct TmemCols {
  uint32_t o, s, p, pstride, q;
};

template <int D>
__device__ __forceinline__ TmemCols tmem_cols(int step_keys) {
  const uint32_t st = static_cast<uint32_t>(step_keys);
  return TmemCols{0u, static_cast<uint32_t>(D), static_cast<uint32_t>(D) + st, st / 2u,
                  static_cast<uint32_t>(D) + 2u * st};
}

// Position in a ring of `n` stages: slot and the parity of its current use.
// Advanced by increments only (no division in the per-step loops).
struct Ring {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Walks a tile's key blocks G at a time: the first run's blocks, then the
// second's, as one sequence, so a step may end the first run and start the
// second (no half-empty step at the end of the first run).
struct Steps {
  int j, nblk, run0, len0, run1;
  __device__ __forceinline__ void init(const WorkTile& t) {
    j = 0;
    nblk = t.nblk;
    run0 = t.run0;
    len0 = t.len0;
    run1 = t.run1;
  }
  // Key block at walk position i.
  __device__ __forceinline__ int block(int i) const {
    return i < len0 ? run0 + i : run1 + (i - len0);
  }
  // Walk position of the next step's first block; nb receives its block count.
  __device__ __forceinline__ int next(int G, int& nb) {
    const int first = j;
    nb = nblk - j < G ? nblk - j : G;
    j += nb;
    return first;
  }
  // Whether the step at walk position `first` with nb blocks spans both runs.
  __device__ __forceinline__ bool spans(int first, int nb) const {
    return first < len0 && first + nb > len0;
  }
};

// ------------------------------------------------------------------ producer
// A step's G blocks are normally consecutive rows of one run, so the step is
// one TMA box per 64-column slab (G * bk rows).  The shorter last step of a
// tile loads the whole box too: the rows past it are never read by an MMA.
// A step that ends the first run and starts the second is loaded one block
// (bk rows) per box into consecutive rows of the stage.
// After an expired wait: the TMA loads this producer issued land in shared
// memory whatever the consumers do, so wait (bounded) for each slot's last
// load before the CTA may leave.
// Bit i of `issued` marks slot i as loaded at least once, bit i of `phase`
// the parity of its last load.
__device__ __noinline__ void drain_loads(uint32_t full0, int n, uint32_t phase, uint32_t issued) {
  for (int i = 0; i < n; ++i) {
    if (!(issued >> i & 1u)) continue;
    const long long t0 = clock64();
    while (!mbar_try_wait(full0 + 8u * static_cast<uint32_t>(i), phase >> i & 1u))
      if (clock64() - t0 > kWaitLimitCycles) break;
  }
}

// Two producer threads: one loads each tile's Q and its K steps, the other
// its V steps.  With one thread issuing in consumption order (K0, K1, V0, K2,
// V1, ...), a K load waited behind the V load before it, whose slot frees
// later (PV runs behind QK), and K arrived with half its lead.
template <int D>
__device__ void producer_qk(const FwdParams& p, const Shared& s) {
  constexpr int kBoxes = D / 64;
  const int bk = p.bk, G = p.G;
  const uint32_t ns = static_cast<uint32_t>(G * bk);     // rows of a step
  const uint32_t box_pitch = ns * 128u;                  // a 64-column box of a stage
  const uint32_t stage_bytes = box_pitch * kBoxes;
  const uint32_t nk = static_cast<uint32_t>(p.stages_k);
  Ring kr;
  uint32_t qc = 0;
  // parity of the last load issued into each K slot (for drain_loads)
  uint32_t kph = 0, kiss = 0;
  auto drain = [&]() {
    drain_loads(bar(s, B_KFULL0), static_cast<int>(nk), kph, kiss);
    drain_loads(bar(s, B_QFULL), 1, (qc - 1u) & 1u, qc > 0 ? 1u : 0u);
  };
  const int n_items = p.n_tiles * p.bh;
  ItemPos iq;
  [[maybe_unused]] const int rows = p.bh * p.n;
  // Takes the next item from the counter; false on an expired wait.
  auto take = [&](int& it, Item& im, WorkTile& t) {
    it = post_item(p, s, iq, n_items, im, t);
    return it != -2;
  };
  // A merged tail tile's Q comes one row group at a time (gsz rows from
  // token row0 + i*T into tile rows i*gsz onwards; gsz*128 bytes is a
  // multiple of 1024, so every box starts on the swizzle's period).
  auto load_qtile = [&](const Item& im, const WorkTile& t) {
    const int ng = t.gsz ? t.nvalid / t.gsz : 0;
    mbar_arrive_expect_tx(bar(s, B_QFULL), (t.gsz ? t.nvalid : kTileM) * D * 2);
    if (WSATTN_BOUNDS(p.status, t.row0 >= 0 && t.nvalid > 0 && t.nvalid <= kTileM &&
                                    (t.gsz ? t.nvalid % t.gsz == 0 &&
                                                 t.row0 + (ng - 1) * p.tq + t.gsz <= p.n
                                           : t.row0 + t.nvalid <= p.n))) {
      if (t.gsz == 0) {
#pragma unroll
        for (int c = 0; c < kBoxes; ++c)
          tma_load_2d(s.q + c * (kTileM * 128), &p.tm_q, bar(s, B_QFULL), c * 64,
                      im.bh * p.n + t.row0);
      } else {
        for (int i = 0; i < ng; ++i) {
#pragma unroll
          for (int c = 0; c < kBoxes; ++c)
            tma_load_2d(s.q + c * (kTileM * 128) + static_cast<uint32_t>(i * t.gsz) * 128u,
                        &p.tm_qg, bar(s, B_QFULL), c * 64, im.bh * p.n + t.row0 + i * p.tq);
        }
      }
    }
    ++qc;
  };
  // The next item is taken kLookahead K steps before the current item's last
  // one, and its Q tile is loaded as soon as the staging buffer is free
  // (tested without blocking, so the K loads never wait for it): the Q tile
  // is then resident when the softmax warps finish the current item.
  constexpr int kLookahead = 2;
  int it;
  Item im{};
  WorkTile t{};
  if (!take(it, im, t)) return drain();
  bool q_pending = it >= 0;
  while (it >= 0) {
    const int y0 = im.bh * p.n;
    if (q_pending) {
      if (!wait(s, bar(s, B_QEMPTY), (qc & 1u) ^ 1u, kStatusTimeoutProducer)) return drain();
      load_qtile(im, t);
    }
    int nxt = -1;
    Item nim{};
    WorkTile nt{};
    bool nq_pending = false;
    const int post_at = t.nstep > kLookahead ? t.nstep - kLookahead : 0;
    Steps ks;
    ks.init(t);
    for (int j = 0; j < t.nstep; ++j) {
      if (j == post_at) {
        if (!take(nxt, nim, nt)) return drain();
        nq_pending = nxt >= 0;
      }
      if (nq_pending && mbar_test_wait(bar(s, B_QEMPTY), (qc & 1u) ^ 1u)) {
        load_qtile(nim, nt);
        nq_pending = false;
      }
      int nb;
      const int first = ks.next(G, nb);
      const bool split = ks.spans(first, nb);
      const int row = y0 + ks.block(first) * bk;
      if (!wait(s, bar(s, B_KEMPTY0 + kr.slot), kr.phase ^ 1u, kStatusTimeoutProducer))
        return drain();
      const uint32_t fb = bar(s, B_KFULL0 + kr.slot);
      const uint32_t tx = split ? static_cast<uint32_t>(nb * bk) * 128u * kBoxes : stage_bytes;
      mbar_arrive_expect_tx(fb, tx);
      const uint32_t dst = s.k + kr.slot * stage_bytes;
      if (!split) {
        // the step's keys lie in the head (rows past them, to the box end,
        // are loaded but never read)
        if (WSATTN_BOUNDS(p.status, nb >= 1 && nb <= G && row >= y0 && row + nb * bk <= y0 + p.n &&
                                        row + nb * bk <= rows)) {
#pragma unroll
          for (int c = 0; c < kBoxes; ++c)
            tma_load_2d(dst + c * box_pitch, &p.tm_k, fb, c * 64, row);
        }
      } else {
        for (int i = 0; i < nb; ++i) {
          const int bro = y0 + ks.block(first + i) * bk;
          if (WSATTN_BOUNDS(p.status, nb <= G && bro >= y0 && bro + bk <= y0 + p.n)) {
#pragma unroll
            for (int c = 0; c < kBoxes; ++c)
              tma_load_2d(dst + c * box_pitch + static_cast<uint32_t>(i * bk) * 128u, &p.tm_k1, fb,
                          c * 64, bro);
          }
        }
      }
      kph = (kph & ~(1u << kr.slot)) | (kr.phase << kr.slot);
      kiss |= 1u << kr.slot;
      kr.next(nk);
    }
    it = nxt;
    im = nim;
    t = nt;
    q_pending = nq_pending;
  }
}

template <int D>
__device__ void producer_v(const FwdParams& p, const Shared& s) {
  constexpr int kBoxes = D / 64;
  const int bk = p.bk, G = p.G;
  const uint32_t ns = static_cast<uint32_t>(G * bk);
  const uint32_t box_pitch = ns * 128u;
  const uint32_t stage_bytes = box_pitch * kBoxes;
  const uint32_t nv = static_cast<uint32_t>(p.stages_v);
  Ring vr;
  uint32_t vph = 0, viss = 0;
  auto drain = [&]() { drain_loads(bar(s, B_VFULL0), static_cast<int>(nv), vph, viss); };
  ItemPos iq;
  while (true) {
    Item im;
    WorkTile t;
    const int it = read_item(s, iq, kStatusTimeoutProducer, im, t);
    if (it == -2) return drain();
    if (it < 0) break;
    const int y0 = im.bh * p.n;
    Steps vs;
    vs.init(t);
    for (int j = 0; j < t.nstep; ++j) {
      int nb;
      const int first = vs.next(G, nb);
      const bool split = vs.spans(first, nb);
      const int row = y0 + vs.block(first) * bk;
      if (!wait(s, bar(s, B_VEMPTY0 + vr.slot), vr.phase ^ 1u, kStatusTimeoutProducer))
        return drain();
      const uint32_t fb = bar(s, B_VFULL0 + vr.slot);
      const uint32_t tx = split ? static_cast<uint32_t>(nb * bk) * 128u * kBoxes : stage_bytes;
      mbar_arrive_expect_tx(fb, tx);
      const uint32_t dst = s.v + vr.slot * stage_bytes;
      if (!split) {
        if (WSATTN_BOUNDS(p.status, nb >= 1 && nb <= G && row >= y0 && row + nb * bk <= y0 + p.n)) {
#pragma unroll
          for (int c = 0; c < kBoxes; ++c)
            tma_load_2d(dst + c * box_pitch, &p.tm_v, fb, c * 64, row);
        }
      } else {
        for (int i = 0; i < nb; ++i) {
          const int bro = y0 + vs.block(first + i) * bk;
          if (WSATTN_BOUNDS(p.status, nb <= G && bro >= y0 && bro + bk <= y0 + p.n)) {
#pragma unroll
            for (int c = 0; c < kBoxes; ++c)
              tma_load_2d(dst + c * box_pitch + static_cast<uint32_t>(i * bk) * 128u, &p.tm_v1, fb,
                          c * 64, bro);
          }
        }
      }
      vph = (vph & ~(1u << vr.slot)) | (vr.phase << vr.slot);
      viss |= 1u << vr.slot;
      vr.next(nv);
    }
  }
}

// ---------------------------------------------------------------- MMA issue
// Two issuer warps feed the tensor core: warp 1 issues S = Q K^T, warp 3
// issues O += P V, each instruction from one elected lane of the converged
// warp.  A tcgen05.mma blocks its issuing thread while the MMA queue is
// full, so with one issuer every barrier wait and every bit of bookkeeping
// between MMA groups left the tensor core idle; with two, one issuer's waits
// overlap the other's MMAs.  QK^T(j+1) waits only until every softmax warp
// holds S(j) in registers; PV(j) waits for P(j).
// Descriptor bases are computed once; each MMA adds a constant to the
// start-address field (bits 0-13, address >> 4), and the k-step loops are
// unrolled.
template <int D>
__device__ void qk_issuer(const FwdParams& p, const Shared& s, uint32_t tbase) {
  constexpr int kBoxes = D / 64;
  const int bk = p.bk, G = p.G;
  const int ns = G * bk;
  const uint32_t box_pitch = static_cast<uint32_t>(ns) * 128u;
  const uint32_t stage_bytes = box_pitch * kBoxes;
  const TmemCols tc_ = tmem_cols<D>(ns);
  const uint32_t t_s = tbase + tc_.s, t_q = tbase + tc_.q;
  const uint32_t id_qk0 = idesc_bf16_f32(kTileM, 0, false);  // N filled per step
  // K is K-major (SBO 1 KB)
  const uint64_t kdesc0 = sdesc_sw128(s.k, 16, 1024);
  const uint64_t box16 = box_pitch >> 4, stage16 = stage_bytes >> 4;
  const uint32_t nk = static_cast<uint32_t>(p.stages_k);
  Ring kr;
  uint32_t su = 0;  // parity of the current use of S
  uint32_t tiles_done = 0;
  Steps qs;
  ItemPos iq;
  while (true) {
    Item im;
    WorkTile t;
    if (read_item_issuer(s, iq, im, t) < 0) break;
    qs.init(t);
    if (!wait_issuer(s, bar(s, B_QTFULL), tiles_done & 1u)) return;
    tc_fence_after();
    for (int j = 0; j < t.nstep; ++j) {
      int nb;
      qs.next(G, nb);
      const uint32_t keys = static_cast<uint32_t>(nb * bk);
      const uint32_t slot = kr.slot;
      // K is normally resident long before S is free: wait for it first, so
      // the wait that gates the MMAs is the softmax's.
      if (!wait_issuer(s, bar(s, B_KFULL0 + slot), kr.phase)) return;
      // the softmax warps must hold the previous S in registers
      if (!wait_issuer(s, bar(s, B_SEMPTY), su ^ 1u)) return;
      tc_fence_after();
      const uint64_t kd = kdesc0 + slot * stage16;
      const uint32_t id = id_qk0 | ((keys >> 3) << 17);
      // S (keys columns) and Q (D/2 columns) inside the allocation, N a
      // multiple of 16 no larger than a step, the K stage inside its ring
      if (WSATTN_BOUNDS(p.status, keys >= 16 && keys % 16 == 0 && keys <= static_cast<uint32_t>(ns) &&
                                      tc_.s + keys <= kTmemCols && tc_.q + D / 2 <= kTmemCols &&
                                      slot < nk)) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts_warp(t_s, t_q + kk * 8, kd + (kk / 4) * box16 + (kk % 4) * 2, id, kk > 0 ? 1u : 0u);
      }
      tc_commit_warp(bar(s, B_KEMPTY0 + slot));
      tc_commit_warp(bar(s, B_SFULL));
      kr.next(nk);
      su ^= 1u;
    }
    ++tiles_done;
  }
}

template <int D, int MAXC>
__device__ void pv_issuer(const FwdParams& p, const Shared& s, uint32_t tbase) {
  constexpr int kBoxes = D / 64;
  const int bk = p.bk, G = p.G;
  const int ns = G * bk;
  const uint32_t box_pitch = static_cast<uint32_t>(ns) * 128u;
  const uint32_t stage_bytes = box_pitch * kBoxes;
  const TmemCols tc_ = tmem_cols<D>(ns);
  const uint32_t t_o = tbase + tc_.o, t_p = tbase + tc_.p;
  const uint32_t id_pv = idesc_bf16_f32(kTileM, D, true);
  // V is MN-major (LBO = the 64-column box pitch)
  const uint64_t vdesc0 = sdesc_sw128(s.v, box_pitch, 1024);
  const uint64_t stage16 = stage_bytes >> 4;
  const uint32_t nv = static_cast<uint32_t>(p.stages_v);
  Ring vr, pr;
  Steps ps;
  ItemPos iq;
  while (true) {
    Item im;
    WorkTile t;
    if (read_item_issuer(s, iq, im, t) < 0) break;
    const int nstep = t.nstep;
    ps.init(t);
    for (int j = 0; j < nstep; ++j) {
      int nb;
      ps.next(G, nb);
      const int keys = nb * bk;
      const int nks = keys / 16;
      const uint32_t pb = pr.slot;
      if (!wait_issuer(s, bar(s, B_PFULL0 + pb), pr.phase)) return;
      const uint32_t vslot = vr.slot;
      if (!wait_issuer(s, bar(s, B_VFULL0 + vslot), vr.phase)) return;
      tc_fence_after();
      const uint64_t vd = vdesc0 + vslot * stage16;
      const uint32_t a_p = t_p + pb * tc_.pstride;
      // P (8 columns per k-step) and O (D columns) inside the allocation,
      // the V stage inside its ring, the k-steps inside the unrolled range
      if (WSATTN_BOUNDS(p.status, nks >= 1 && nks <= kNumWG * MAXC &&
                                      tc_.p + pb * tc_.pstride + 8u * nks <= kTmemCols &&
                                      tc_.o + D <= kTmemCols && vslot < nv)) {
        // 16 key rows (2 KB of V, 8 P columns) per k-step
        mma_ts_warp(t_o, a_p, vd, id_pv, j > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < kNumWG * MAXC; ++kk)
          if (kk < nks) mma_ts_warp(t_o, a_p + kk * 8, vd + kk * 128, id_pv, 1u);
      }
      tc_commit_warp(bar(s, B_VEMPTY0 + vslot));
      tc_commit_warp(bar(s, B_PVDONE0 + pb));
      vr.next(nv);
      pr.next(2);
    }
    tc_commit_warp(bar(s, B_OFULL));
  }
}

// -------------------------------------------------------------- softmax WGs
// Copies this thread's share of its Q row (the warpgroup's 16-element groups
// of D) from the swizzled staging tile into TMEM (column c holds elements 2c
// and 2c+1); rows past the frame are zeroed.
template <int D>
__device__ bool load_q(const Shared& s, uint32_t t_q, int wg, int r, int nvalid, uint32_t& qc) {
  if (!wait_warp(s, bar(s, B_QFULL), qc & 1u)) return false;
  ++qc;
  const bool zero = r >= nvalid;
  int g0, ng;
  wg_share(D / 16, wg, g0, ng);
#pragma unroll
  for (int h = 0; h < (D / 16 + kNumWG - 1) / kNumWG; ++h) {
    if (h >= ng) break;
    const int e0 = 16 * (g0 + h);  // first element of this 16-element group
    const uint32_t row_addr = s.q + (e0 / 64) * (kTileM * 128) + r * 128;
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t m = static_cast<uint32_t>((e0 % 64) / 8 + e);
      const uint4 v = ld_shared_v4(row_addr + ((m ^ static_cast<uint32_t>(r & 7)) << 4));
      w[4 * e + 0] = zero ? 0u : v.x;
      w[4 * e + 1] = zero ? 0u : v.y;
      w[4 * e + 2] = zero ? 0u : v.z;
      w[4 * e + 3] = zero ? 0u : v.w;
    }
    tmem_st8(t_q + e0 / 2, w);
  }
  tmem_wait_st();
  tc_fence_before();
  warp_arrive(bar(s, B_QTFULL));
  warp_arrive(bar(s, B_QEMPTY));
  return true;
}

// p = 2^(s*c + nb) for 16 logits (two lanes at a time); adds them to the
// packed row sums and stores the bf16 pairs as 8 TMEM columns at taddr.
__device__ __forceinline__ void exp_pack_store(const uint32_t (&sv)[16], uint64_t c2, uint64_t nb2,
                                               uint64_t& la, uint64_t& lb, uint32_t taddr) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 t = f2_unpack(
        f2_fma(f2_pack(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1])), c2, nb2));
    const float p0 = ex2_approx(t.x);
    const float p1 = ex2_approx(t.y);
    if (i & 1)
      lb = f2_add(lb, f2_pack(p0, p1));
    else
      la = f2_add(la, f2_pack(p0, p1));
    const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  tmem_st8(taddr, w);
}

// Loads this warpgroup's S columns of the step (MAXC chunks of 16 from sa)
// into registers with one wait.  Chunks past the step's own (a shorter last
// step of a run) read neighbouring tensor-memory columns and are ignored.
template <int MAXC>
__device__ __forceinline__ void load_s(uint32_t sa, uint32_t (&sv)[MAXC][16]) {
#pragma unroll
  for (int c = 0; c < MAXC; ++c) tmem_ld16(sa + 16 * c, sv[c]);
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < MAXC; ++c) reg_fence16(sv[c]);
}

// p = 2^(s*c + nb) for the first n16 chunks: stores their bf16 pairs at
// pa + 8c and adds them to the packed row sums.  Chunks whose bit in vis is
// clear (keys the row's frame does not attend, in a merged tail tile) get
// the bias -inf, so their p is exactly 0.
template <int MAXC, bool kMasked>
__device__ __forceinline__ void exp_chunks(const uint32_t (&sv)[MAXC][16], int n16, uint64_t c2,
                                           uint64_t nb2, uint64_t& la, uint64_t& lb,
                                           uint32_t pa, uint32_t vis) {
  const uint64_t ninf2 = f2_pack(-INFINITY, -INFINITY);
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    if (c < n16)
      exp_pack_store(sv[c], c2, !kMasked || ((vis >> c) & 1u) ? nb2 : ninf2, la, lb, pa + 8 * c);
  }
}

// A softmax thread's view of a work item: the tile, its path, and the
// statistics behind its own row's fixed max.  Formed for the next item before
// the current item's epilogue, so that the global loads of the row and frame
// statistics complete while the epilogue runs rather than in front of the
// next item's first key step.
struct RowItem {
  Item im;
  WorkTile t;
  size_t grow;
  float qn, kq, c;  // ||q_i||, the frame's key-norm bound, c_i (0 for rows past the frame)
  bool online, valid;
  // -m_i in log2 units: the row's fixed max m_i = b_i + c_i, b_i = (scale ||q_i||) K
  __device__ __forceinline__ float nb_fixed(float scale) const {
    return valid ? -__fadd_rn(row_bound(scale, qn, kq), c) * kLog2e : 0.f;
  }
};

// Bit c set: chunk f16 + c of the step starting at walk position `first`
// (cpb 16-key chunks per block) lies in one of the row's own key runs.
__device__ __forceinline__ uint32_t chunk_vis(const int (&own)[kGroupInts], const Steps& st,
                                              int first, int f16, int n16, int cpb) {
  uint32_t vis = 0;
  for (int c = 0; c < n16; ++c) {
    const int b = st.block(first + (f16 + c) / cpb);
    if ((b >= own[0] && b < own[0] + own[1]) || (b >= own[2] && b < own[2] + own[3]))
      vis |= 1u << c;
  }
  return vis;
}

__device__ __forceinline__ RowItem row_item(const FwdParams& p, const Item& im,
                                            const WorkTile& t, int r) {
  RowItem x;
  x.im = im;
  x.t = t;
  x.online = p.force_path >= 0 ? (p.force_path == 1) : (p.elig[x.im.bh] == 0);
  const int64_t tok = tile_row_token(t, r, p.tq);
  x.grow = static_cast<size_t>(x.im.bh) * p.n + tok;
  x.valid = r < x.t.nvalid && WSATTN_BOUNDS(p.status, x.grow < static_cast<size_t>(p.bh) * p.n);
  // loads only: their values are first used when the item starts
  x.qn = x.valid ? p.qn_rows[x.grow] : 0.f;
  x.kq = x.valid ? p.kq[static_cast<size_t>(x.im.bh) * p.nfq + tok / p.tq] : 0.f;
  x.c = x.valid ? p.c_rows[x.grow] : 0.f;
  return x;
}

template <int D, int MAXC>
__device__ void softmax_wg(const FwdParams& p, const Shared& s, uint32_t tbase) {
  const int warp = threadIdx.x / 32;
  const int wg = (warp - kSoftmaxWarp0) / 4;
  const int r = (threadIdx.x - kSoftmaxWarp0 * 32) % kTileM;  // tile row == TMEM lane
  const uint32_t lane = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const int bk = p.bk, G = p.G;
  const TmemCols tc_ = tmem_cols<D>(G * bk);
  int og0, nog;  // this warpgroup's 16-column groups of O
  wg_share(D / 16, wg, og0, nog);
  const uint32_t ocol = tc_.o + static_cast<uint32_t>(16 * og0);
  const float c = p.scale_log2;
  const uint64_t c2 = f2_pack(c, c);
  // The output is not read again here: its L2 lines go first, so they are
  // written back while this kernel runs (it does not bind on DRAM) instead
  // of during the next call's statistics passes, whose reads would evict
  // them.
  const uint64_t out_policy = policy_evict_first();
  uint32_t qc = 0, tiles_done = 0, xpar = 0, xc = 0;
  uint32_t su = 0;  // parity of the current use of S
  Ring pr;          // P buffer

  ItemPos iq;
  Item im0;
  WorkTile t0;
  if (read_item_warp(s, iq, im0, t0) < 0) return;
  RowItem cur = row_item(p, im0, t0, r);
  if (!load_q<D>(s, lane + tc_.q, wg, r, cur.t.nvalid, qc)) return;
  while (true) {
    const Item im = cur.im;
    const WorkTile t = cur.t;
    const bool online = cur.online;
    const size_t grow = cur.grow;
    const bool valid = cur.valid;
    const float nb_fixed = cur.nb_fixed(p.scale);
    Steps st;
    st.init(t);
    float l = 0.f;
    float m = -INFINITY;
    // The step loops, compiled once for ordinary tiles and once for merged
    // tail tiles (whose rows see only their own frames' key chunks).
    auto fixed_path = [&](auto masked_tag) -> bool {
      constexpr bool kMasked = decltype(masked_tag)::value;
      // merged tail tile: the row's own frame's key runs (rows past the
      // groups see the whole union)
      int own[kGroupInts] = {0, 0x3fffffff, 0, 0};
      if (kMasked && valid) {
#pragma unroll
        for (int i = 0; i < kGroupInts; ++i)
          own[i] = p.grp[static_cast<size_t>(t.gtab + r / t.gsz) * kGroupInts + i];
      }
      // Fixed max: every step is load, exp, pack, store; the row sum
      // accumulates.
      const uint64_t nb2 = f2_pack(nb_fixed, nb_fixed);
      uint64_t la = f2_pack(0.f, 0.f), lb = la;
      for (int j = 0; j < t.nstep; ++j) {
        int nblk;
        const int pos = st.next(G, nblk);  // walk position of the step's first block
        const int keys = nblk * bk;
        int f16, n16;  // this warpgroup's 16-column chunks of the step
        wg_share(keys / 16, wg, f16, n16);
        const uint32_t vis = kMasked ? chunk_vis(own, st, pos, f16, n16, bk / 16) : ~0u;
        const uint32_t c0 = static_cast<uint32_t>(16 * f16);  // first S column
        const uint32_t pb = pr.slot;
        // the S columns read and the P columns written lie in the allocation
        // and P stays inside its own buffer
        const bool cols_ok = WSATTN_BOUNDS(
            p.status, tc_.s + c0 + 16u * MAXC <= kTmemCols && n16 <= MAXC &&
                          c0 / 2 + 8u * n16 <= tc_.pstride && tc_.p + 2u * tc_.pstride <= kTmemCols);
        if (!wait_warp(s, bar(s, B_SFULL), su)) return false;
        tc_fence_after();
        uint32_t sv[MAXC][16];
        if (cols_ok) load_s<MAXC>(lane + tc_.s + c0, sv);
        tc_fence_before();
        warp_arrive(bar(s, B_SEMPTY));
        su ^= 1u;
        // the PV that read this P buffer two steps back must be done
        if (!wait_warp(s, bar(s, B_PVDONE0 + pb), pr.phase ^ 1u)) return false;
        tc_fence_after();
        if (cols_ok)
          exp_chunks<MAXC, kMasked>(sv, n16, c2, nb2, la, lb,
                                    lane + tc_.p + pb * tc_.pstride + c0 / 2, vis);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar(s, B_PFULL0 + pb));
        pr.next(2);
      }
      const float2 a = f2_unpack(f2_add(la, lb));
      l = a.x + a.y;
      return true;
    };
    auto online_path = [&](auto masked_tag) -> bool {
      constexpr bool kMasked = decltype(masked_tag)::value;
      // merged tail tile: the row's own frame's key runs (rows past the
      // groups see the whole union)
      int own[kGroupInts] = {0, 0x3fffffff, 0, 0};
      if (kMasked && valid) {
#pragma unroll
        for (int i = 0; i < kGroupInts; ++i)
          own[i] = p.grp[static_cast<size_t>(t.gtab + r / t.gsz) * kGroupInts + i];
      }
      for (int j = 0; j < t.nstep; ++j) {
        int nblk;
        const int pos = st.next(G, nblk);  // walk position of the step's first block
        const int keys = nblk * bk;
        int f16, n16;
        wg_share(keys / 16, wg, f16, n16);
        const uint32_t vis = kMasked ? chunk_vis(own, st, pos, f16, n16, bk / 16) : ~0u;
        const uint32_t c0 = static_cast<uint32_t>(16 * f16);
        const bool cols_ok = WSATTN_BOUNDS(
            p.status, tc_.s + c0 + 16u * MAXC <= kTmemCols && n16 <= MAXC &&
                          c0 / 2 + 8u * n16 <= tc_.pstride && tc_.p + 2u * tc_.pstride <= kTmemCols &&
                          ocol + 16u * nog <= kTmemCols);
        if (!wait_warp(s, bar(s, B_SFULL), su)) return false;
        tc_fence_after();
        uint32_t sv[MAXC][16];
        if (cols_ok) {
          load_s<MAXC>(lane + tc_.s + c0, sv);
        } else {
#pragma unroll
          for (int k = 0; k < MAXC; ++k)
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[k][i] = 0u;
        }
        tc_fence_before();
        warp_arrive(bar(s, B_SEMPTY));
        su ^= 1u;
        // row max of this step over both warpgroups' columns
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < MAXC; ++k) {
          if (k < n16 && (!kMasked || ((vis >> k) & 1u))) {
#pragma unroll
            for (int i = 0; i < 16; ++i) mx = fmaxf(mx, __uint_as_float(sv[k][i]));
          }
        }
        s.xch_m[(xpar * kNumWG + wg) * kTileM + r] = mx;
        if (!xch_sync(s, xc)) return false;
        float mall = mx;
#pragma unroll
        for (int v = 0; v < kNumWG; ++v) mall = fmaxf(mall, s.xch_m[(xpar * kNumWG + v) * kTileM + r]);
        xpar ^= 1u;
        // Lazy rescale: the running max moves only when the step's max
        // exceeds it by more than kLazyMax (log2 units), so p <= 2^kLazyMax
        // (exact enough in fp32 and bf16) and O and l are rescaled rarely;
        // O / l is unchanged in exact arithmetic whatever max is used.
        const float m_top = fmaxf(m, mall * c);
        const float m_new = m_top > m + kLazyMax ? m_top : m;
        const float alpha = m_new == m ? 1.f : ex2_approx(m - m_new);
        const uint32_t pb = pr.slot;
        if (!wait_warp(s, bar(s, B_PVDONE0 + pb), pr.phase ^ 1u)) return false;
        tc_fence_after();
        uint64_t sa2 = f2_pack(0.f, 0.f), sb2 = sa2;
        if (cols_ok)
          exp_chunks<MAXC, kMasked>(sv, n16, c2, f2_pack(-m_new, -m_new), sa2, sb2,
                           lane + tc_.p + pb * tc_.pstride + c0 / 2, vis);
        const float2 a = f2_unpack(f2_add(sa2, sb2));
        l = l * alpha + (a.x + a.y);
        m = m_new;
        if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f) && cols_ok) {
          // O += P(j-1) V must have landed before O is rescaled: PV(j-1)
          // read the other P buffer, whose PV-done barrier is at most one
          // use behind (its next use needs P(j+1)), so one parity wait is
          // exact.  Ring position of step j-1: the other slot, same phase
          // when this slot is 1, flipped when it is 0.
          const uint32_t prev_phase = pb == 1u ? pr.phase : pr.phase ^ 1u;
          if (!wait_warp(s, bar(s, B_PVDONE0 + (pb ^ 1u)), prev_phase)) return false;
          tc_fence_after();
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
          for (int k = 0; k < nog; ++k) {
            uint32_t ra[16];
            tmem_ld16(lane + ocol + k * 16, ra);
            tmem_wait_ld16(ra);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 o2 = f2_unpack(f2_mul(
                  f2_pack(__uint_as_float(ra[2 * i]), __uint_as_float(ra[2 * i + 1])), a2));
              ra[2 * i] = __float_as_uint(o2.x);
              ra[2 * i + 1] = __float_as_uint(o2.y);
            }
            tmem_st16(lane + ocol + k * 16, ra);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(bar(s, B_PFULL0 + pb));
        pr.next(2);
      }
        return true;
    };
    const bool steps_ok =
        !online ? (t.gsz ? fixed_path(std::true_type{}) : fixed_path(std::false_type{}))
                : (t.gsz ? online_path(std::true_type{}) : online_path(std::false_type{}));
    if (!steps_ok) return;

    // Stage the next tile's Q so its first QK products overlap this epilogue,
    // and start the loads of its row parameters.
    Item nim;
    WorkTile ntl;
    const int nxt = read_item_warp(s, iq, nim, ntl);
    if (nxt == -2) return;
    RowItem nx;
    if (nxt >= 0) {
      nx = row_item(p, nim, ntl, r);
      if (!load_q<D>(s, lane + tc_.q, wg, r, nx.t.nvalid, qc)) return;
    }

    if (!wait_warp(s, bar(s, B_OFULL), tiles_done & 1u)) return;
    // the row sum is the sum of the warpgroups' partial sums (fixed order)
    const uint32_t lpar = tiles_done & 1u;
    ++tiles_done;
    s.xch_l[(lpar * kNumWG + wg) * kTileM + r] = l;
    if (!xch_sync(s, xc)) return;
    float lsum = 0.f;
#pragma unroll
    for (int g = 0; g < kNumWG; ++g) lsum += s.xch_l[(lpar * kNumWG + g) * kTileM + r];
    tc_fence_after();
    const float inv = 1.f / lsum;
    float* orow = p.out + grow * D + 16 * og0;
    // A warp whose 32 rows are 32 consecutive output tokens (every full warp
    // of an ordinary tile; in a merged tail tile, when its row groups hold a
    // multiple of 32 rows) stages each 16-column group in its shared chunk
    // (its rows 64 bytes apart) and sends it with one TMA store: the
    // per-thread row stores below touch 32 rows per instruction.  The chunk
    // uses the 64-byte swizzle (16-byte unit u of row r sits at unit
    // u ^ ((r >> 1) & 3)), so each quarter-warp's 16-byte stores fall in eight
    // different bank groups.  Other warps store their valid rows themselves.
    const int wq = warp & 3;
    // O's columns lie in the allocation; a full warp's 32 rows in the output
    const bool o_ok = WSATTN_BOUNDS(p.status, ocol + 16u * nog <= kTmemCols);
    const int64_t wtok = tile_row_token(t, 32 * wq, p.tq);
    const bool warp_full =
        32 * wq + 32 <= t.nvalid && t.gsz % 32 == 0 &&
        WSATTN_BOUNDS(p.status, im.bh * p.n + wtok + 32 <= static_cast<int64_t>(p.bh) * p.n);
    const uint32_t chunk = s.ostage + static_cast<uint32_t>(warp - kSoftmaxWarp0) * kOChunkBytes;
    const int lid = threadIdx.x & 31;
#pragma unroll 1
    for (int k = 0; k < (o_ok ? nog : 0); ++k) {
      uint32_t v[16];
      tmem_ld16(lane + ocol + k * 16, v);
      tmem_wait_ld16(v);
      if (warp_full) {
        // the chunk's previous store must have read it
        if (lid == 0) bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_shared_v4(chunk + 64u * lid + 16u * (i ^ ((lid >> 1) & 3)),
                       __float_as_uint(__uint_as_float(v[4 * i]) * inv),
                       __float_as_uint(__uint_as_float(v[4 * i + 1]) * inv),
                       __float_as_uint(__uint_as_float(v[4 * i + 2]) * inv),
                       __float_as_uint(__uint_as_float(v[4 * i + 3]) * inv));
        fence_proxy_async_smem();
        __syncwarp();
        if (lid == 0) {
          tma_store_2d_hint(&p.tm_o, chunk, 16 * (og0 + k),
                            static_cast<int32_t>(im.bh * p.n + wtok), out_policy);
          bulk_commit_group();
        }
      } else if (valid) {
        float4* dst = reinterpret_cast<float4*>(orow + k * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_global_v4_hint(dst + i, __uint_as_float(v[4 * i]) * inv,
                            __uint_as_float(v[4 * i + 1]) * inv, __uint_as_float(v[4 * i + 2]) * inv,
                            __uint_as_float(v[4 * i + 3]) * inv, out_policy);
      }
    }
    if (nxt < 0) break;
    cur = nx;
  }
}

// -------------------------------------------------------------------- kernel
// MAXC = 16-column chunks per warpgroup and key step: ceil(G * bk / 16 / kNumWG).
template <int D, int MAXC>
__global__ void __launch_bounds__(kThreads, 1) wsattn_fwd_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t stage_bytes = static_cast<uint32_t>(p.G * p.bk) * D * 2u;
  Shared s;
  s.q = base;
  s.k = base + kTileM * D * 2;
  s.v = s.k + static_cast<uint32_t>(p.stages_k) * stage_bytes;
  s.bars = s.v + static_cast<uint32_t>(p.stages_v) * stage_bytes;
  uint8_t* gbars = smem_raw + (s.bars - raw);
  s.xch_m = reinterpret_cast<float*>(gbars + 8 * B_COUNT + 16);
  s.xch_l = s.xch_m + 2 * kNumWG * kTileM;
  s.iq = reinterpret_cast<volatile int32_t*>(s.xch_l + 2 * kNumWG * kTileM);
  s.ostage = (s.bars + 8u * B_COUNT + 16u + kXchBytes + 4u * kQWords * kItemQueue + 511u) & ~511u;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(gbars + 8 * B_COUNT);
  s.abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  s.status = p.status;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(bar(s, B_QFULL), 1);
    mbar_init(bar(s, B_QEMPTY), kSoftmaxWarps);
    mbar_init(bar(s, B_QTFULL), kSoftmaxWarps);
    mbar_init(bar(s, B_OFULL), 1);
    mbar_init(bar(s, B_SFULL), 1);
    mbar_init(bar(s, B_SEMPTY), kSoftmaxWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(s, B_PFULL0 + i), kSoftmaxWarps);
      mbar_init(bar(s, B_PVDONE0 + i), 1);
    }
    mbar_init(bar(s, B_XCH), kSoftmaxWarps);
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(s, B_KFULL0 + i), 1);
      mbar_init(bar(s, B_KEMPTY0 + i), 1);
      mbar_init(bar(s, B_VFULL0 + i), 1);
      mbar_init(bar(s, B_VEMPTY0 + i), 1);
    }
    for (int i = 0; i < kItemQueue; ++i) {
      mbar_init(bar(s, B_IQFULL0 + i), 1);
      mbar_init(bar(s, B_IQEMPTY0 + i), kItemReaders);
    }
    *s.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&p.tm_q);
    prefetch_tensormap(&p.tm_k);
    prefetch_tensormap(&p.tm_v);
    prefetch_tensormap(&p.tm_o);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tslot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  griddep_wait();  // the row maxima and eligibility come from the kernel before
#ifdef WSATTN_DEBUG
  uint32_t dsmem = 0;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dsmem));
  // the shared-memory layout fits the launch's dynamic shared memory, the
  // rings are at most 4 deep (the barriers there are), the tensor-memory
  // layout fits the allocation
  const bool layout_ok = WSATTN_BOUNDS(
      p.status, (s.ostage + kOStageBytes) - raw <= dsmem && p.stages_k >= 1 && p.stages_k <= 4 &&
                    p.stages_v >= 1 && p.stages_v <= 4 &&
                    tmem_cols<D>(p.G * p.bk).q + D / 2 <= kTmemCols);
#else
  constexpr bool layout_ok = true;
#endif

  if (!layout_ok) {
  } else if (warp == 0) {
    if (lane == 0) producer_qk<D>(p, s);
  } else if (warp == 2) {
    if (lane == 0) producer_v<D>(p, s);
  } else if (warp == 1) {
    qk_issuer<D>(p, s, tbase);
  } else if (warp == 3) {
    pv_issuer<D, MAXC>(p, s, tbase);
  } else if (warp >= kSoftmaxWarp0) {
    softmax_wg<D, MAXC>(p, s, tbase);
    // the epilogue's tile stores must be complete before the CTA exits
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tbase, kTmemCols);
  // The last CTA to finish (every CTA has drawn its last item by now) resets
  // the work counter for the next launch.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.work + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      p.work[0] = 0;
      p.work[1] = 0;
      __threadfence();
    }
  }
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

template <int D, int MAXC>
cudaError_t launch_one(const FwdParams& p, int grid, size_t smem, cudaStream_t stream) {
  static bool attr_set[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(
        wsattn_fwd_kernel<D, MAXC>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // dependent launch: the prologue (barriers, TMEM, tensor maps) overlaps
  // the end of the statistics pass before it
  return launch_dependent(wsattn_fwd_kernel<D, MAXC>, dim3(grid), dim3(kThreads), smem, stream,
                          p);
}

template <int D, int M>
cudaError_t launch_m(const FwdParams& p, int maxc, int grid, size_t smem, cudaStream_t stream) {
  if constexpr (M > kMaxChunksAll) {
    return cudaErrorInvalidValue;
  } else {
    if (maxc == M) return launch_one<D, M>(p, grid, smem, stream);
    return launch_m<D, M + 1>(p, maxc, grid, smem, stream);
  }
}

template <int D>
cudaError_t launch_d(const FwdParams& p, int grid, size_t smem, cudaStream_t stream) {
  const int chunks = p.G * p.bk / 16;  // 16-column chunks of a full step
  return launch_m<D, 1>(p, (chunks + kNumWG - 1) / kNumWG, grid, smem, stream);
}

}  // namespace

size_t forward_smem_bytes(int D, int step_keys, int stages_k, int stages_v) {
  const size_t stage = static_cast<size_t>(step_keys) * D * 2;
  return 1024 + static_cast<size_t>(kTileM) * D * 2 + (stages_k + stages_v) * stage +
         8 * B_COUNT + 16 + kXchBytes + 4 * kQWords * kItemQueue + 512 + kOStageBytes;
}

void forward_stages(int D, int step_keys, size_t smem_optin, int* stages_k, int* stages_v) {
  int st = 4;
  while (st > 1 && forward_smem_bytes(D, step_keys, st, st) > smem_optin) --st;
  *stages_k = st;
  *stages_v = st;
}

cudaError_t launch_forward(const FwdParams& p, int D, int grid, size_t smem, cudaStream_t stream) {
  static_assert(kMaxChunksAll * 16 * kNumWG >= kStepKeys, "chunk instantiations must cover a step");
  return D == 128 ? launch_d<128>(p, grid, smem, stream) : launch_d<64>(p, grid, smem, stream);
}

cudaError_t launch_timeout_selftest(long long limit_cycles, int* status, cudaStream_t stream) {
  timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_cycles, status);
  return cudaGetLastError();
}

}  // namespace wsattn
