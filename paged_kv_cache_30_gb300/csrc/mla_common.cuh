// mla_common.cuh -- the unit of work of the MLA verify kernels and its
// decoding from the planning kernel's table (shared by the bf16/FP8 and the
// native-FP8 verify kernels).
#pragma once
#include "pkv_internal.h"

namespace pkv {
namespace mla {

struct Unit {
  int b, split, t, half, nsplit;
  int L, lim;
  int tile0, ntiles;  // tiles [tile0, tile0 + ntiles) of this CTA
};

__device__ __forceinline__ int clamped_len(const MlaParams& p, int b) {
  int L = __ldg(p.seq_lens + b);
  if (L < 0) L = 0;
  if ((long long)L > (long long)p.max_blocks * p.page_size) L = p.max_blocks * p.page_size;
  return L;
}

// Splits of a request of L keys when a split holds at least min_tiles tiles
// (at most p.cap; the planning kernel picks min_tiles and writes the count
// into every entry, so the verify kernels never recompute it).
__device__ __forceinline__ int split_count(const MlaParams& p, int L, int min_tiles) {
  const int req_tiles = (L + kMlaTile - 1) / kMlaTile;
  const int ns = (req_tiles + min_tiles - 1) / min_tiles;
  return ns < 1 ? 1 : (ns > p.cap ? p.cap : ns);
}

// Tiles of the largest split of a request of L keys.
__device__ __forceinline__ int split_tiles(const MlaParams& p, int L, int min_tiles) {
  const int req_tiles = (L + kMlaTile - 1) / kMlaTile;
  const int ns = split_count(p, L, min_tiles);
  return (req_tiles + ns - 1) / ns;
}

// Plan entry of (request b, row t, half, split of nsplit): row t is a verify
// token, or a token pair for CTA-pair launches; split, nsplit - 1 < 16.
__device__ __forceinline__ int plan_entry(int rows, int b, int t, int half, int split, int nsplit) {
  return ((((b * rows + t) * 2 + half) << 4 | split) << 4) | (nsplit - 1);
}

// The unit of this CTA, from the plan the planning kernel wrote (see
// plan_entry), or -1 (returned as split 0 of nsplit 0: no unit).
__device__ __forceinline__ Unit decode_unit(const MlaParams& p) {
  Unit u;
  const int v = __ldg(p.plan + blockIdx.x);
  if (v < 0) {
    u.split = 0;
    u.nsplit = 0;
    return u;
  }
  u.split = (v >> 4) & 15;
  const int ns = (v & 15) + 1;
  const int ch = v >> 8;
  u.half = ch & 1;
  const int rt = ch >> 1;
  u.b = rt / p.qlen;
  u.t = rt - u.b * p.qlen;
  const int L = clamped_len(p, u.b);
  int Lr = p.real_seq_lens ? __ldg(p.real_seq_lens + u.b) : L;
  int lim = L - p.qlen + 1 + u.t;
  if (Lr < lim) lim = Lr;
  if (lim < 0) lim = 0;
  u.L = L;
  u.lim = lim;
  const int req_tiles = (L + kMlaTile - 1) / kMlaTile;
  u.nsplit = ns;
  const int a = (int)((long long)req_tiles * u.split / ns);
  const int e = (int)((long long)req_tiles * (u.split + 1) / ns);
  const int lim_tiles = (lim + kMlaTile - 1) / kMlaTile;
  u.tile0 = a;
  u.ntiles = max(0, min(e, lim_tiles) - a);
  return u;
}

__device__ __forceinline__ int counter_index(const MlaParams& p, const Unit& u) {
  return (u.b * p.qlen + u.t) * 2 + u.half;
}

__device__ __forceinline__ long long slot_of(const MlaParams& p, const Unit& u, int split) {
  return ((long long)(u.b * p.cap + split) * p.qlen + u.t) * 2 + u.half;
}

}  // namespace mla
}  // namespace pkv
