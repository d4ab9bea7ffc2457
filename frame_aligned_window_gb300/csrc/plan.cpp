// Block-map builder (host only).
//
// Google Developers Blog post "HeyGen x Google Cloud: Bringing Avatar IV to
// TPUs", section "Deleting the mask" (Fig. 3): the mask is frame-aligned, so
// with block sizes that are multiples of 16 and divide the frame token span T
// every block lies inside one query frame and one key frame and is therefore
// entirely active or entirely skipped.  The map is built at frame granularity
// and expanded to blocks; no element of the mask is ever materialised.
//
// Frame rule (frames_interact in internal.h; token-order frame indices):
// query frame a sees key frame c iff c is a reference frame, a is a reference
// frame (reference queries are global), or the video frames are at most w
// apart; the mask variants make the window causal (c in a - w .. a), move the
// reference frames after the video frames, or confine reference queries to
// reference keys.
#include <algorithm>
#include <new>
#include <utility>

#include "internal.h"

namespace wsattn {

static bool valid_block(int b, int T) { return b >= 16 && b % 16 == 0 && T % b == 0; }

namespace {

// A frame's key blocks: at most two runs of consecutive blocks.
struct FrameKeys {
  int64_t frame;
  int32_t kbeg, nblk;
  int32_t run[2], len[2];
};

// Key steps of a tile: its two runs are walked as one sequence of blocks,
// G at a time (a step may end the first run and start the second).
int32_t key_steps(int32_t len0, int32_t len1, int G) { return (len0 + len1 + G - 1) / G; }

// The union of the key blocks of f[0 .. m), as at most two runs; false if it
// takes more.
bool union_runs(const FrameKeys* f, int m, int32_t (&run)[2], int32_t (&len)[2]) {
  std::vector<std::pair<int32_t, int32_t>> iv;  // [begin, end)
  for (int i = 0; i < m; ++i)
    for (int r = 0; r < 2; ++r)
      if (f[i].len[r] > 0) iv.emplace_back(f[i].run[r], f[i].run[r] + f[i].len[r]);
  std::sort(iv.begin(), iv.end());
  std::vector<std::pair<int32_t, int32_t>> u;
  for (const auto& x : iv) {
    if (!u.empty() && x.first <= u.back().second)
      u.back().second = std::max(u.back().second, x.second);
    else
      u.push_back(x);
  }
  if (u.empty() || u.size() > 2) return false;
  run[0] = u[0].first;
  len[0] = u[0].second - u[0].first;
  run[1] = u.size() == 2 ? u[1].first : 0;
  len[1] = u.size() == 2 ? u[1].second - u[1].first : 0;
  return true;
}

}  // namespace

// The forward kernel streams keys in steps of floor(kStepKeys / bk) blocks,
// so the automatic size is the valid block whose step holds the most keys;
// ties go to the larger block (fewer TMA boxes per step).
int auto_block(int T) {
  int best = 0, best_step = 0;
  for (int b = 16; b <= kStepKeys && b <= T; b += 16) {
    if (T % b != 0) continue;
    const int step = (kStepKeys / b) * b;
    if (step >= best_step) {
      best = b;
      best_step = step;
    }
  }
  return best;
}

int build_host_plan(int frames, int tokens_per_frame, int window, int ref_frames, int heads,
                    int head_dim, int block_q, int block_k, int mask_flags, HostPlan* out) {
  if (!out) return WSATTN_ERR_BAD_ARG;
  const int all_flags = WSATTN_MASK_CAUSAL | WSATTN_MASK_REF_SUFFIX | WSATTN_MASK_REF_LOCAL;
  if (mask_flags & ~all_flags) return WSATTN_ERR_BAD_ARG;
  if (frames < 1 || ref_frames < 0 || window < 0 || heads < 1) return WSATTN_ERR_BAD_ARG;
  if (tokens_per_frame < 16 || tokens_per_frame % 16 != 0) return WSATTN_ERR_BAD_BLOCK;
  if (head_dim != 64 && head_dim != 128) return WSATTN_ERR_UNSUPPORTED;
  const int T = tokens_per_frame;
  const int64_t nf = static_cast<int64_t>(frames) + ref_frames;
  const int64_t N = nf * T;
  // Query rows and key coordinates are int32 inside the kernels.
  if (N > (int64_t(1) << 30)) return WSATTN_ERR_BAD_ARG;
  const int bq = block_q ? block_q : auto_block(T);
  const int bk = block_k ? block_k : auto_block(T);
  if (block_q < 0 || block_k < 0) return WSATTN_ERR_BAD_BLOCK;
  if (!valid_block(bq, T) || !valid_block(bk, T)) return WSATTN_ERR_BAD_BLOCK;

  HostPlan& p = *out;
  p = HostPlan{};
  p.F = frames; p.T = T; p.w = window; p.R = ref_frames; p.H = heads; p.D = head_dim;
  p.flags = mask_flags;
  p.bq = bq; p.bk = bk; p.N = N;
  p.nqb = N / bq;
  p.nkb = N / bk;
  p.G = bk <= kStepKeys ? kStepKeys / bk : 1;
  try {
    // Bitmap and CSR.
    p.bitmap.assign(static_cast<size_t>(p.nqb * p.nkb), 0);
    p.row_ptr.assign(static_cast<size_t>(p.nqb + 1), 0);
    for (int64_t qb = 0; qb < p.nqb; ++qb) {
      const int a = static_cast<int>(qb * bq / T);
      for (int64_t kb = 0; kb < p.nkb; ++kb) {
        const int c = static_cast<int>(kb * bk / T);
        if (frames_interact(a, c, frames, window, ref_frames, mask_flags)) {
          p.bitmap[static_cast<size_t>(qb * p.nkb + kb)] = 1;
          p.col.push_back(static_cast<int32_t>(kb));
        }
      }
      p.row_ptr[static_cast<size_t>(qb + 1)] = static_cast<int32_t>(p.col.size());
    }
    // Active element pairs per (b, h): T*T per interacting frame pair.
    int64_t pairs = 0;
    for (int64_t a = 0; a < nf; ++a)
      for (int64_t c = 0; c < nf; ++c)
        if (frames_interact(static_cast<int>(a), static_cast<int>(c), frames, window, ref_frames,
                            mask_flags))
          pairs++;
    p.active_pairs = pairs * T * T;

    // Work list: every 128-row query tile of every frame, with the frame's key
    // blocks.  The key list of frame a is the CSR row of its first q-block
    // (all q-blocks of a frame share it).  Frames' short tail tiles are
    // collected and merged below.
    const int tiles_per_frame = (T + kTileM - 1) / kTileM;
    const int tail = T % kTileM;
    std::vector<FrameKeys> tails;
    for (int64_t a = 0; a < nf; ++a) {
      const int64_t qb0 = a * T / bq;
      const int32_t kbeg = static_cast<int32_t>(p.kcol.size());
      for (int32_t e = p.row_ptr[static_cast<size_t>(qb0)];
           e < p.row_ptr[static_cast<size_t>(qb0 + 1)]; ++e)
        p.kcol.push_back(p.col[static_cast<size_t>(e)]);
      const int32_t kend = static_cast<int32_t>(p.kcol.size());
      // Split the (increasing) key-block list into runs of consecutive blocks.
      int32_t run[2] = {0, 0}, len[2] = {0, 0};
      int nrun = 0;
      for (int32_t e = kbeg; e < kend; ++e) {
        const int32_t kb = p.kcol[static_cast<size_t>(e)];
        if (nrun > 0 && kb == run[nrun - 1] + len[nrun - 1]) {
          ++len[nrun - 1];
        } else {
          if (nrun == 2) return WSATTN_ERR_UNSUPPORTED;  // not produced by this mask family
          run[nrun] = kb;
          len[nrun] = 1;
          ++nrun;
        }
      }
      if (nrun == 0) return WSATTN_ERR_BAD_ARG;  // every frame sees at least itself
      for (int t = 0; t < tiles_per_frame; ++t) {
        if (tail && t == tiles_per_frame - 1) {
          tails.push_back(FrameKeys{a, kbeg, kend - kbeg, {run[0], nrun == 2 ? run[1] : 0},
                                    {len[0], len[1]}});
          continue;
        }
        WorkTile wt{};
        wt.row0 = static_cast<int32_t>(a * T + t * kTileM);
        wt.nvalid = std::min(kTileM, T - t * kTileM);
        wt.nblk = kend - kbeg;
        wt.run0 = run[0];
        wt.len0 = len[0];
        wt.run1 = nrun == 2 ? run[1] : 0;
        wt.nstep = key_steps(len[0], len[1], p.G);
        wt.kbeg = kbeg;
        p.tiles.push_back(wt);
      }
    }
    // Tail tiles: up to g = 128 / tail consecutive frames' tails share one
    // tile when the union of their key blocks is still two runs at most and
    // takes fewer key steps than the tails one by one (greedily, in token
    // order).  The first group's rows are the first frame's tail.
    const int g = tail ? kTileM / tail : 0;
    for (size_t i = 0; i < tails.size();) {
      int m = static_cast<int>(std::min<size_t>(static_cast<size_t>(g), tails.size() - i));
      int32_t urun[2] = {0, 0}, ulen[2] = {0, 0};
      for (; m >= 2; --m) {
        int32_t sep = 0;
        for (int j = 0; j < m; ++j) sep += key_steps(tails[i + j].len[0], tails[i + j].len[1], p.G);
        if (union_runs(&tails[i], m, urun, ulen) && key_steps(ulen[0], ulen[1], p.G) < sep) break;
      }
      const FrameKeys& f0 = tails[i];
      WorkTile wt{};
      wt.row0 = static_cast<int32_t>(f0.frame * T + (tiles_per_frame - 1) * kTileM);
      wt.kbeg = f0.kbeg;
      if (m >= 2) {
        wt.nvalid = m * tail;
        wt.nblk = ulen[0] + ulen[1];
        wt.run0 = urun[0];
        wt.len0 = ulen[0];
        wt.run1 = urun[1];
        wt.nstep = key_steps(ulen[0], ulen[1], p.G);
        wt.gsz = tail;
        wt.gtab = static_cast<int32_t>(p.grp.size() / kGroupInts);
        for (int j = 0; j < m; ++j) {
          const FrameKeys& f = tails[i + j];
          p.grp.insert(p.grp.end(), {f.run[0], f.len[0], f.run[1], f.len[1]});
        }
        p.gsz = tail;
        i += static_cast<size_t>(m);
      } else {
        wt.nvalid = tail;
        wt.nblk = f0.nblk;
        wt.run0 = f0.run[0];
        wt.len0 = f0.len[0];
        wt.run1 = f0.run[1];
        wt.nstep = key_steps(f0.len[0], f0.len[1], p.G);
        ++i;
      }
      p.tiles.push_back(wt);
    }
    // Longest first (the reference frame's tiles see every key block); the
    // order among equal lengths stays the token order.
    std::stable_sort(p.tiles.begin(), p.tiles.end(), [](const WorkTile& x, const WorkTile& y) {
      return x.nblk > y.nblk;
    });
    p.cls.push_back(0);
    for (size_t i = 1; i < p.tiles.size(); ++i)
      if (p.tiles[i].nblk != p.tiles[i - 1].nblk) p.cls.push_back(static_cast<int32_t>(i));
    p.cls.push_back(static_cast<int32_t>(p.tiles.size()));
  } catch (const std::bad_alloc&) {
    return WSATTN_ERR_NO_MEMORY;
  }
  return WSATTN_OK;
}

}  // namespace wsattn
