// gqa_decode.cu -- split-KV paged GQA decode attention for sm_103a.
//
// Computes, for every request b and query head h (kv head h / 8),
//   out = sum_j softmax_j(scale * q.k_j) v_j, with an optional sink logit in
//   the denominator, and lse = log sum_j exp(scale * q.k_j) (keys only),
// over keys [max(L - window, 0), L) gathered through block_table
// ("vllm.models.flint.ops.decode_attention": flint_decode_attention and the
// module's numerics paragraph; block-table indexing as in the transformers
// "Atencion paginada" decode path).
//
// Design: persistent, two CTAs per SM, each 2 producer warps + 4 consumer warps.
//  * Work items are (request, kv head, split) triples.  Every CTA derives the
//    same item list in its prologue from seq_lens alone: request b's n_b
//    attended pages are cut into s_b = min(cap, ceil(n_b / chunk)) contiguous
//    page ranges, with chunk chosen from the total so that the launch has about
//    target_items items (shorter requests use fewer splits).  CTA c starts
//    with item c; the rest come from a global queue (an atomic head; every CTA
//    fetches until it draws an index past the end, so the launch makes a known
//    number of fetches and the CTA that draws the last one resets the head to
//    zero), so the launch shape depends only on the device and the batch.  A
//    CTA claims its next item only when the current one has a few tiles left
//    to issue, so when the queue runs dry no CTA still holds an unstarted item.
//  * Programmatic dependent launch: the prologue, the first item's descriptor,
//    its block-table entries and up to one ring of its leading tiles (never
//    the page holding position L - 1) are done before griddepcontrol.wait, so
//    they overlap the tail of the kernel before; q, the queue, the workspace
//    and the outputs come after it.
//  * The first producer warp takes items from the queue, writes each item's
//    descriptor and bulk-copies its 8 query rows into a descriptor slot.  Both
//    producer warps read block-table entries 32 at a time and stream the
//    16-token tiles of every page with one TMA operation each -- the first the
//    even pages, the second the odd ones (one issuing thread tops out near
//    31 GB/s of 8 KB tiles, two reach ~49 GB/s) -- through a 5-D view of the
//    cache (64 dims, token, 4 chunks of 64 dims, kv head, block) whose box
//    lands the tile chunk-major as four 16 x 128-byte slabs (K lo, K hi, V lo,
//    V hi) with 128-byte swizzle, into an 8-stage ring (8 KB stages) guarded
//    by full/empty mbarriers.  They run ahead across item boundaries.
//  * Consumer warp w takes tiles w, w+4, ... of the item.  It pulls the tile's
//    K and V fragments into registers with ldmatrix (conflict-free thanks to
//    the swizzle), frees the stage at once (after a generic-to-async proxy
//    fence: the next TMA write into the stage must not overtake these reads),
//    then
//      S[8 heads x 16 tok] = Q K^T          mma.m16n8k16, heads on the M side
//                                             (rows 8..15 zero)
//      online softmax, exp2 domain, running max in unscaled logits
//      O^T[128 dims x 8 heads] += V^T P^T   mma.m16n8k16; P^T is S's
//                                             accumulator layout rounded to bf16
//  * The four warps' (O, m, l) merge in shared memory.  A single-split item
//    writes out / lse directly.  Otherwise the fp32 partial is published and
//    a per-group arrival counter (groups of up to 16 splits) is bumped with a
//    release atomic; the last CTA of a group merges the group, and with more
//    than one group the last group merges the group results.  Every counter is
//    reset to zero by the CTA that consumed it.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarps = 2;     // even and odd tiles
constexpr int kThreads = kConsumers + 32 * kProducerWarps;
constexpr int kCtasPerSm = 2;
constexpr int kStageBytes = 16 * 512;  // one 16-token tile: 16 x [K | V] x bf16
constexpr int kStages = 8;
constexpr int kBoxBytes = 16 * 128;    // one 64-element-wide TMA box of a tile
constexpr int kItemSlots = 4;
constexpr int kQBytes = kGqaGroup * kGqaHeadDim * 2;
constexpr int kWbRow = 132;            // padded O row of the combine buffer (floats)
constexpr int kWbFloats = kGqaGroup * kWbRow + 2 * kGqaGroup;  // O[8][132], m[8], l[8]
constexpr int kMergeGroup = 16;        // splits merged by one CTA at the first level
constexpr int kClaimTiles = 4;         // claim the next item this many tiles before the end
constexpr float kLog2e = 1.4426950408889634f;

struct ItemDesc {
  // pe: pages [p0, pe) of a CTA's first item are streamed before the
  // programmatic-dependent-launch wait (pe == p0 for later items)
  int item, b, kvh, split, nsplit, p0, p1, start_tok, L, seq_base, pe, pad1;
};

// shared-memory carve-up (offsets from a 1024-aligned base)
constexpr int kOffWbuf = kStages * kStageBytes;
constexpr int kOffQ = kOffWbuf + kConsumerWarps * kWbFloats * 4;
constexpr int kOffPrefix = kOffQ + kItemSlots * kQBytes;
constexpr int kOffItems = kOffPrefix + ((kGqaMaxBatch + 1) * 4 + 15) / 16 * 16;
constexpr int kOffBars = kOffItems + kItemSlots * (int)sizeof(ItemDesc);
constexpr int kNumBars = 2 * kStages + 3 * kItemSlots;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
static_assert(kOffWbuf % 1024 == 0 && kOffQ % 16 == 0 && kOffPrefix % 16 == 0 &&
                  kOffItems % 16 == 0 && kOffBars % 16 == 0 && kOffMisc % 16 == 0,
              "shared-memory offsets");
static_assert(kCtasPerSm * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
static_assert(kMergeGroup * kGqaMlFloats <= kConsumerWarps * kWbFloats, "merge scratch");
static_assert(kStages % (2 * kProducerWarps) == 0, "each stage is refilled by one producer warp");

// Exclusive scan of one int per thread over the CTA; `scratch` holds one int
// per warp plus one.  Returns the exclusive prefix; *total = the sum.
__device__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      const int s = scratch[w];
      scratch[w] = run;
      run += s;
    }
    scratch[kThreads / 32] = run;
  }
  __syncthreads();
  const int res = scratch[warp] + incl - v;
  *total = scratch[kThreads / 32];
  __syncthreads();
  return res;
}

template <int P>
__device__ __forceinline__ int clamp_len(const GqaParams& p, int b) {
  int L = __ldg(p.seq_lens + b);
  if (L < 0) L = 0;
  if (L > p.max_blocks * P) L = p.max_blocks * P;
  return L;
}

__device__ __forceinline__ int window_start(const GqaParams& p, int L) {
  return (p.window > 0 && L > p.window) ? L - p.window : 0;
}

// Out row slice [d0, d0 + 8) of one (request, head), and its lse.
__device__ __forceinline__ void finalize(const GqaParams& p, int b, int head, int d0,
                                         const float (&o)[8], float m, float l) {
  float inv = 0.f;
  if (l > 0.f) {
    float den = l;
    if (p.sinks) den += ex2(__fmaf_rn(__ldg(p.sinks + head), kLog2e, -m * p.scale_log2));
    inv = 1.f / den;
  }
  uint4 v;
  v.x = pack_bf16(o[0] * inv, o[1] * inv);
  v.y = pack_bf16(o[2] * inv, o[3] * inv);
  v.z = pack_bf16(o[4] * inv, o[5] * inv);
  v.w = pack_bf16(o[6] * inv, o[7] * inv);
  *reinterpret_cast<uint4*>(p.out + b * p.o_sb + head * p.o_sh + d0) = v;
  if (d0 == 0 && p.lse)
    p.lse[b * p.lse_sb + head * p.lse_sh] = (l > 0.f) ? m * p.scale + logf(l) : -INFINITY;
}

// Merge n published partials (slots slot0, slot0 + stride, ...) into
// (o[8], M, L) for this thread's head eh and dims [ed, ed + 8).  `sml` is
// shared scratch for n x 16 floats; all consumer threads take part.
__device__ __forceinline__ void merge_slots(const GqaParams& p, long long slot0, int stride,
                                            int n, float* sml, int eh, int ed, float (&o)[8],
                                            float& M, float& Ls) {
  const int ct = threadIdx.x;
  for (int i = ct; i < n * kGqaMlFloats; i += kConsumers) {
    const int s = i / kGqaMlFloats, k = i % kGqaMlFloats;
    sml[i] = __ldcg(p.part_ml + (slot0 + (long long)s * stride) * kGqaMlFloats + k);
  }
  named_bar_sync(1, kConsumers);
  M = -INFINITY;
  for (int s = 0; s < n; ++s) M = fmaxf(M, sml[s * kGqaMlFloats + eh]);
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
  Ls = 0.f;
  const float c2 = p.scale_log2;
#pragma unroll 4
  for (int s = 0; s < n; ++s) {
    const float* src =
        p.part_o + (slot0 + (long long)s * stride) * kGqaPartialFloats + eh * kGqaHeadDim + ed;
    const float4 a = ldcg_f4(src), b = ldcg_f4(src + 4);
    const float ms = sml[s * kGqaMlFloats + eh];
    const float w = (ms == -INFINITY) ? 0.f : ex2((ms - M) * c2);
    Ls = __fmaf_rn(w, sml[s * kGqaMlFloats + kGqaGroup + eh], Ls);
    o[0] = __fmaf_rn(w, a.x, o[0]); o[1] = __fmaf_rn(w, a.y, o[1]);
    o[2] = __fmaf_rn(w, a.z, o[2]); o[3] = __fmaf_rn(w, a.w, o[3]);
    o[4] = __fmaf_rn(w, b.x, o[4]); o[5] = __fmaf_rn(w, b.y, o[5]);
    o[6] = __fmaf_rn(w, b.z, o[6]); o[7] = __fmaf_rn(w, b.w, o[7]);
  }
}

__device__ __forceinline__ void store_partial(const GqaParams& p, long long slot, int eh, int ed,
                                              const float (&o)[8], float m, float l) {
  float* dst = p.part_o + slot * kGqaPartialFloats + eh * kGqaHeadDim + ed;
  *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
  *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
  if (ed == 0) {
    p.part_ml[slot * kGqaMlFloats + eh] = m;
    p.part_ml[slot * kGqaMlFloats + kGqaGroup + eh] = l;
  }
}

template <int P, bool kCluster>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    gqa_decode_kernel(const __grid_constant__ GqaParams p,
                      const __grid_constant__ CUtensorMap kv_map) {
  constexpr int TPP = P / 16;  // 16-token tiles per page
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);

  const uint32_t ring = base_u32;
  float* wbuf = reinterpret_cast<float*>(base + kOffWbuf);
  const uint32_t qbuf = base_u32 + kOffQ;
  int* prefix = reinterpret_cast<int*>(base + kOffPrefix);
  ItemDesc* items = reinterpret_cast<ItemDesc*>(base + kOffItems);
  const uint32_t bars = base_u32 + kOffBars;
  int* misc = reinterpret_cast<int*>(base + kOffMisc);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto ifull_bar = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto iempty_bar = [&](int s) { return bars + 8u * (2 * kStages + kItemSlots + s); };
  // descriptor written (no query bytes): what the second producer waits for
  auto dfull_bar = [&](int s) { return bars + 8u * (2 * kStages + 2 * kItemSlots + s); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(ifull_bar(s), 1);
      mbar_init(iempty_bar(s), kConsumerWarps + 1);  // + the second producer
      mbar_init(dfull_bar(s), 1);
    }
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) tma_prefetch_desc(&kv_map);
  // Programmatic dependent launch.  Before griddepcontrol.wait (i.e. while the
  // grid this launch depends on, e.g. the previous call or layer, may still be
  // running) the kernel reads only seq_lens, block_table and the leading KV
  // pages of its first item -- never the page holding position L - 1, which
  // an append kernel may just have written -- and writes only shared memory
  // (and error bits).  q, sinks, the workspace (queue, counters, partials)
  // and every output are touched after the wait.

  // ---- prologue: the item list, identical in every CTA -------------------
  const int B = p.B;
  // With a split cap of 1, or a window that spans at most min_pages pages
  // (no request then reaches two splits: chunk >= min_pages), item i is
  // (request i / Hkv, kv head i % Hkv) and no scan is needed.  A window of W
  // tokens touches at most (W + 2P - 2) / P pages.
  const bool one_split = p.cap <= 1 || (p.window > 0 && (p.window + 2 * P - 2) / P <= p.min_pages);
  int total_items = B * p.Hkv;
  if (!kCluster && !one_split) {
    int local_pages = 0;
    for (int b = tid; b < B; b += kThreads) {
      const int raw = __ldg(p.seq_lens + b);
      if ((long long)raw > (long long)p.max_blocks * P) atomicOr(p.err, DEVERR_SEQ_TOO_LONG);
      const int L = clamp_len<P>(p, b);
      local_pages += (L + P - 1) / P - window_start(p, L) / P;
    }
    int total_pages;
    block_exclusive_scan(local_pages, misc, &total_pages);
    const long long total_ph = (long long)total_pages * p.Hkv;
    int chunk = (int)((total_ph + p.target_items - 1) / p.target_items);
    if (chunk < p.min_pages) chunk = p.min_pages;
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = tid * per;
    int my_items = 0;
    for (int i = 0; i < per && b0 + i < B; ++i) {
      const int L = clamp_len<P>(p, b0 + i);
      const int n = (L + P - 1) / P - window_start(p, L) / P;
      const int s = max(1, min(p.cap, (n + chunk - 1) / chunk));
      my_items += s * p.Hkv;
    }
    int run = block_exclusive_scan(my_items, misc, &total_items);
    for (int i = 0; i < per && b0 + i < B; ++i) {
      prefix[b0 + i] = run;
      const int L = clamp_len<P>(p, b0 + i);
      const int n = (L + P - 1) / P - window_start(p, L) / P;
      run += max(1, min(p.cap, (n + chunk - 1) / chunk)) * p.Hkv;
    }
    if (tid == 0) prefix[B] = total_items;
  }
  // one-split items and the cluster mode write no partials
  if (!kCluster && !one_split && (long long)total_items > p.max_items) {
    if (tid == 0) atomicOr(p.err, DEVERR_ITEM_OVERFLOW);
    total_items = (int)p.max_items;
  }
  __syncthreads();

  // Streams the tiles of pages [p0, p1) of (request row bt_row, kv head kvh)
  // that fall to producer `mine`: whole pages, alternating (an item's first
  // tile number `seq` is a multiple of TPP, so a page's tiles share a parity
  // of seq / TPP and every ring stage is refilled by one producer only).
  // At page claim_at (if in range) it calls on_page() first: the first
  // producer claims its next item there.
  auto stream_tiles = [&](const int32_t* bt_row, int kvh, int p0, int p1, uint32_t seq,
                          uint32_t mine, int claim_at, auto&& on_page) {
    for (int pb = p0; pb < p1; pb += 32) {
      const int cnt = min(32, p1 - pb);
      int blk = 0;
      if (lane < cnt) {
        blk = __ldg(bt_row + pb + lane);
        if (blk < 0 || blk >= p.num_blocks) atomicOr(p.err, DEVERR_BAD_BLOCK);
      }
      for (int i = 0; i < cnt; ++i) {
        if (pb + i == claim_at) on_page();
        const int blk_i = __shfl_sync(0xffffffffu, blk, i);
#pragma unroll
        for (int sub = 0; sub < TPP; ++sub) {
          if (lane == 0 && ((seq / TPP) & 1u) == mine) {
            const int stage = seq % kStages;
            mbar_wait(empty_bar(stage), ((seq / kStages) & 1) ^ 1u, p.err);
            mbar_arrive_expect_tx(full_bar(stage), kStageBytes);
            const uint32_t dst = ring + stage * kStageBytes;
            // one box: 16 tokens x 4 chunks of 64 dims (K lo, K hi, V lo, V hi),
            // landing chunk-major
            tma_load_5d(dst, &kv_map, full_bar(stage), 0, 16 * sub, 0, kvh, blk_i);
          }
          ++seq;
        }
      }
    }
  };

  // cluster mode: the split this CTA's consumers left in shared memory
  int cl_nsplit = 0, cl_b = 0, cl_kvh = 0;
  const int eh = (tid & (kConsumers - 1)) >> 4, ed = (tid & 15) * 8;  // epilogue: head, 8 dims

  if (warp == kConsumerWarps + 1) {
    // ===================== second producer warp: odd tiles =====================
    for (int it = 0;; ++it) {
      const int slot = it % kItemSlots;
      mbar_wait(dfull_bar(slot), (it / kItemSlots) & 1, p.err);
      const ItemDesc d = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(iempty_bar(slot));
      if (d.item < 0) break;
      const int32_t* bt_row = p.bt + (long long)d.b * p.bt_sb;
      stream_tiles(bt_row, d.kvh, d.p0, d.pe, (uint32_t)d.seq_base, 1u, -1, [] {});
      if (it == 0) griddep_wait();  // the pages from pe on only after the wait
      stream_tiles(bt_row, d.kvh, d.pe, d.p1, (uint32_t)(d.seq_base + (d.pe - d.p0) * TPP), 1u,
                   -1, [] {});
    }
  } else if (warp == kConsumerWarps) {
    // ============ first producer warp: the queue, descriptors, even tiles ============
    // CTA c's first item is item c (static: known before the wait, so its
    // leading tiles are requested then); the queue deals items gridDim.x on.
    // A CTA claims its next item when the current one has kClaimTiles tiles
    // left to issue (enough to hide the atomic): a claimed item waits for the
    // current one to end, so claiming at its start would leave a CTA holding
    // up to two items when the queue runs dry.  Every CTA draws exactly one
    // queue index past the end, so the launch makes (items beyond the static
    // ones) + CTAs fetches, and the fetch that returns the last of them resets
    // the head.
    const int grid = (int)gridDim.x;
    const int last_fetch = max(total_items - grid, 0) + grid - 1;
    int fetched = 0;  // lane 0's claim (a queue index), not yet examined
    uint32_t seq = 0;
    for (int it = 0;; ++it) {
      int item = (int)blockIdx.x;
      // cluster mode: one item, split blockIdx.x of (request, kv head) blockIdx.y
      int b = 0, nsplit = 1, kvh = 0, split = 0, L = 0;
      if (kCluster) {
        const int pair = (int)blockIdx.y;
        b = pair / p.Hkv;
        kvh = pair - b * p.Hkv;
        split = (int)blockIdx.x;
        L = clamp_len<P>(p, b);
        if (lane == 0 && kvh == 0 && split == 0 &&
            (long long)__ldg(p.seq_lens + b) > (long long)p.max_blocks * P)
          atomicOr(p.err, DEVERR_SEQ_TOO_LONG);
        const int n = (L + P - 1) / P - window_start(p, L) / P;
        nsplit = max(1, min(p.cluster, (n + p.min_pages - 1) / p.min_pages));
        item = (it == 0 && split < nsplit) ? pair : total_items;
      } else if (it > 0) {
        const int k = __shfl_sync(0xffffffffu, fetched, 0);
        if (lane == 0 && k == last_fetch) atomicExch(&p.sched[0], 0);
        item = grid + k;
      }
      const int slot = it % kItemSlots;
      if (lane == 0) mbar_wait(iempty_bar(slot), ((it / kItemSlots) & 1) ^ 1u, p.err);
      __syncwarp();
      // no CTA can take more items than the launch has: the item loop is bounded
      const bool runaway = it > total_items;
      if (item >= total_items || runaway) {
        if (!kCluster && it == 0) {
          // no static item: this CTA still draws its one index past the end
          griddep_wait();
          if (lane == 0) {
            const int k = atomicAdd(&p.sched[0], 1);
            if (k == last_fetch) atomicExch(&p.sched[0], 0);
          }
        }
        if (lane == 0) {
          if (runaway) atomicOr(p.err, DEVERR_QUEUE);
          griddep_launch_dependents();  // the queue is empty: this CTA only drains now
          items[slot].item = -1;
          mbar_arrive(dfull_bar(slot));
          mbar_arrive(ifull_bar(slot));
        }
        break;
      }
      if (kCluster) {
        // (b, kvh, split, nsplit, L) decoded above
      } else if (one_split) {
        b = item / p.Hkv;
        kvh = item - b * p.Hkv;
        nsplit = 1;
        split = 0;
        // the check the scanning prologue makes, once per request
        if (lane == 0 && kvh == 0 && (long long)__ldg(p.seq_lens + b) > (long long)p.max_blocks * P)
          atomicOr(p.err, DEVERR_SEQ_TOO_LONG);
      } else {
        int lo = 0, hi = B - 1;  // request = last b with prefix[b] <= item
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
        }
        b = lo;
        nsplit = (prefix[b + 1] - prefix[b]) / p.Hkv;
        const int local = item - prefix[b];
        kvh = local / nsplit;
        split = local % nsplit;
      }
      if (!kCluster) L = clamp_len<P>(p, b);
      const int start_tok = window_start(p, L);
      const int sp = start_tok / P;
      const int n = (L + P - 1) / P - sp;
      const int p0 = sp + (int)((long long)n * split / nsplit);
      const int p1 = sp + (int)((long long)n * (split + 1) / nsplit);
      // First item: pages before the one holding position L - 1, at most one
      // ring's worth (both producers together issue at most kStages tiles, so
      // neither waits for a free stage before the consumers can start).
      const int pe = it == 0 ? max(p0, min(min(p1, p0 + kStages / TPP), (L - 1) / P)) : p0;
      if (lane == 0) {
        ItemDesc& d = items[slot];
        d.item = item; d.b = b; d.kvh = kvh; d.split = split; d.nsplit = nsplit;
        d.p0 = p0; d.p1 = p1; d.start_tok = start_tok; d.L = L; d.seq_base = (int)seq;
        d.pe = pe;
        // the descriptor stores are released by this arrive
        mbar_arrive(dfull_bar(slot));
      }
      const int32_t* bt_row = p.bt + (long long)b * p.bt_sb;
      stream_tiles(bt_row, kvh, p0, pe, seq, 0u, -1, [] {});
      if (it == 0) griddep_wait();
      if (lane == 0) {
        // the consumers' phase also waits for the 8 query rows
        mbar_arrive_expect_tx(ifull_bar(slot), kQBytes);
        const uint16_t* qrow = p.q + b * p.q_sb + (long long)(kvh * kGqaGroup) * p.q_sh;
#pragma unroll
        for (int h = 0; h < kGqaGroup; ++h)
          bulk_load(qbuf + slot * kQBytes + h * kGqaHeadDim * 2, qrow + h * p.q_sh,
                    kGqaHeadDim * 2, ifull_bar(slot));
      }
      // claim_at lies in [pe, p1) whenever pages remain after pe; otherwise the
      // claim is made right away
      // (the cluster mode has no queue: one item per CTA)
      const int claim_at = kCluster ? -1 : max(pe, p1 - max(1, kClaimTiles / TPP));
      stream_tiles(bt_row, kvh, pe, p1, seq + (uint32_t)((pe - p0) * TPP), 0u, claim_at, [&] {
        if (lane == 0) fetched = atomicAdd(&p.sched[0], 1);
      });
      if (!kCluster && p1 <= pe && lane == 0) fetched = atomicAdd(&p.sched[0], 1);
      seq += (uint32_t)((p1 - p0) * TPP);
    }
    if (lane == 0) {
      // every issued copy (of both producer warps) has landed before the CTA
      // may exit (the consumers waited on them already unless a wait gave up)
      const uint32_t recent = seq < (uint32_t)kStages ? seq : (uint32_t)kStages;
      for (uint32_t k = seq - recent; k < seq; ++k)
        mbar_wait(full_bar(k % kStages), (k / kStages) & 1, p.err);
    }
  } else {
  // ============================ consumer warps ============================
  griddep_wait();  // outputs, partials and counters only after the wait
  const int g = lane >> 2, t = lane & 3;
  // ldmatrix addressing: matrix mi = lane / 8 supplies row r = lane % 8 of
  // tile rows 0..7 (mi = 0, 1) or 8..15 (mi = 2, 3); odd mi read the upper
  // 16-byte unit of a 16-element k-step.  The 128-byte swizzle XORs the unit
  // index with the row index mod 8.
  const int mi = lane >> 3, r = lane & 7;
  const uint32_t row_off = (uint32_t)(r + 8 * (mi >> 1)) * 128u;
  const int ubit = mi & 1;
  float* my_wb = wbuf + warp * kWbFloats;
  const float c2 = p.scale_log2;

  for (int it = 0;; ++it) {
    const int slot = it % kItemSlots;
    mbar_wait(ifull_bar(slot), (it / kItemSlots) & 1, p.err);
    const ItemDesc d = items[slot];
    // Q as the A operand: rows = the 8 heads of this kv head (rows 8..15 zero)
    uint32_t qa[8][2];
    if (d.item >= 0) {
      const uint8_t* qs = base + kOffQ + slot * kQBytes + g * kGqaHeadDim * 2;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        qa[s][0] = *reinterpret_cast<const uint32_t*>(qs + (16 * s + 2 * t) * 2);
        qa[s][1] = *reinterpret_cast<const uint32_t*>(qs + (16 * s + 8 + 2 * t) * 2);
      }
    }
    fence_proxy_async_smem();  // the Q slot is refilled by a bulk copy
    __syncwarp();
    if (lane == 0) mbar_arrive(iempty_bar(slot));
    if (d.item < 0) break;

    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    // m: running max (raw logits); msc: the exponent reference m * c2 as
    // rounded once when m last grew -- every term and rescale uses it, and the
    // rescale factor is exactly 1 while m holds (a factor recomputed from the
    // unrounded m * c2 would be 2^(rounding error) != 1 and would compound over
    // the 8192 tiles of a 131072-key split).  l is a compensated (Neumaier)
    // sum; lcomp carries the rounding error of its additions.
    float m = -INFINITY, msc = 0.f, l = 0.f, lcomp = 0.f;

    const int ntiles = (d.p1 - d.p0) * TPP;
    for (int k = warp; k < ntiles; k += kConsumerWarps) {
      const uint32_t seq = (uint32_t)d.seq_base + (uint32_t)k;
      const int stage = seq % kStages;
      mbar_wait(full_bar(stage), (seq / kStages) & 1, p.err);
      const uint32_t tile = ring + stage * kStageBytes + row_off;
      // K fragments (B operand of S = Q K^T) and V fragments (A operand of
      // O^T += V^T P^T) for the whole tile, then the stage is released.
      uint32_t kf[8][4], vf[8][4];
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t unit = (uint32_t)((2 * (s & 3) + ubit) ^ r);
        ldsm_x4(tile + (s >> 2) * kBoxBytes + (unit << 4), kf[s][0], kf[s][1], kf[s][2], kf[s][3]);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t unit = (uint32_t)((2 * (j & 3) + ubit) ^ r);
        ldsm_x4_trans(tile + (2 + (j >> 2)) * kBoxBytes + (unit << 4), vf[j][0], vf[j][1],
                      vf[j][2], vf[j][3]);
      }
      fence_proxy_async_smem();  // the stage is refilled by TMA
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(stage));

      const int tok0 = (d.p0 + k / TPP) * P + 16 * (k % TPP);
      // ---- S = Q K^T over 128 dims, 4 independent accumulator chains ----
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        if (s & 1) {
          mma_bf16_16816(sb, qa[s][0], 0u, qa[s][1], 0u, kf[s][0], kf[s][1]);
          mma_bf16_16816(sd, qa[s][0], 0u, qa[s][1], 0u, kf[s][2], kf[s][3]);
        } else {
          mma_bf16_16816(sa, qa[s][0], 0u, qa[s][1], 0u, kf[s][0], kf[s][1]);
          mma_bf16_16816(sc, qa[s][0], 0u, qa[s][1], 0u, kf[s][2], kf[s][3]);
        }
      }
      // lane (g, t): head g; tile tokens 2t, 2t+1 (x0, x1) and 8+2t, 9+2t (x2, x3)
      float x0 = sa[0] + sb[0], x1 = sa[1] + sb[1];
      float x2 = sc[0] + sd[0], x3 = sc[1] + sd[1];
      const int pa = tok0 + 2 * t;
      const bool v0 = pa >= d.start_tok && pa < d.L;
      const bool v1 = pa + 1 >= d.start_tok && pa + 1 < d.L;
      const bool v2 = pa + 8 >= d.start_tok && pa + 8 < d.L;
      const bool v3 = pa + 9 >= d.start_tok && pa + 9 < d.L;
      x0 = v0 ? x0 : -INFINITY;
      x1 = v1 ? x1 : -INFINITY;
      x2 = v2 ? x2 : -INFINITY;
      x3 = v3 ? x3 : -INFINITY;
      // ---- online softmax (exp2 domain, running max in raw logits) ----
      float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m, mx);
      const bool grew = mn > m;  // false while no key has been seen
      const float msc_new = grew ? mn * c2 : msc;
      const float alpha = grew ? ((m == -INFINITY) ? 0.f : ex2(msc - msc_new)) : 1.f;
      msc = msc_new;
      const float e0 = ex2(__fmaf_rn(x0, c2, -msc));
      const float e1 = ex2(__fmaf_rn(x1, c2, -msc));
      const float e2 = ex2(__fmaf_rn(x2, c2, -msc));
      const float e3 = ex2(__fmaf_rn(x3, c2, -msc));
      {
        const float ls = __fmul_rn(l, alpha), x = (e0 + e1) + (e2 + e3);
        const float tsum = __fadd_rn(ls, x);
        const bool lbig = fabsf(ls) >= fabsf(x);
        const float err = __fadd_rn(__fsub_rn(lbig ? ls : x, tsum), lbig ? x : ls);
        lcomp = __fadd_rn(__fmul_rn(lcomp, alpha), err);
        l = tsum;
      }
      m = mn;
      // O^T columns are heads 2t, 2t+1: their rescale factors live on lanes 8t, 8t+4
      const float al0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
      const float al1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[j][0] *= al0; acc[j][1] *= al1; acc[j][2] *= al0; acc[j][3] *= al1;
      }
      const uint32_t pb0 = pack_bf16(e0, e1), pb1 = pack_bf16(e2, e3);
      // V rows outside [start_tok, L) are zeroed: stale cache contents (NaN,
      // Inf) must not reach P.V even with P = 0.
      if ((tok0 < d.start_tok) || (tok0 + 16 > d.L)) {
        const uint32_t mlo = (v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u);
        const uint32_t mhi = (v2 ? 0x0000ffffu : 0u) | (v3 ? 0xffff0000u : 0u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          vf[j][0] &= mlo; vf[j][1] &= mlo; vf[j][2] &= mhi; vf[j][3] &= mhi;
        }
      }
      // ---- O^T += V^T P^T: 8 m-tiles of 16 dims ----
#pragma unroll
      for (int j = 0; j < 8; ++j)
        mma_bf16_16816(acc[j], vf[j][0], vf[j][1], vf[j][2], vf[j][3], pb0, pb1);
    }

    // ---- merge the warps' (O, m, l) in shared memory ----
    l = __fadd_rn(l, lcomp);
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int d0 = 16 * j + g;
      my_wb[(2 * t) * kWbRow + d0] = acc[j][0];
      my_wb[(2 * t + 1) * kWbRow + d0] = acc[j][1];
      my_wb[(2 * t) * kWbRow + d0 + 8] = acc[j][2];
      my_wb[(2 * t + 1) * kWbRow + d0 + 8] = acc[j][3];
    }
    if (t == 0) {
      my_wb[kGqaGroup * kWbRow + g] = m;
      my_wb[kGqaGroup * kWbRow + kGqaGroup + g] = l;
    }
    named_bar_sync(1, kConsumers);
    float mc = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w)
      mc = fmaxf(mc, wbuf[w * kWbFloats + kGqaGroup * kWbRow + eh]);
    float o[8], lc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float* wb = wbuf + w * kWbFloats;
      const float mw = wb[kGqaGroup * kWbRow + eh];
      const float cw = (mw == -INFINITY) ? 0.f : ex2((mw - mc) * c2);
      lc = __fmaf_rn(cw, wb[kGqaGroup * kWbRow + kGqaGroup + eh], lc);
      const float4 a = *reinterpret_cast<const float4*>(wb + eh * kWbRow + ed);
      const float4 bq = *reinterpret_cast<const float4*>(wb + eh * kWbRow + ed + 4);
      o[0] = __fmaf_rn(cw, a.x, o[0]); o[1] = __fmaf_rn(cw, a.y, o[1]);
      o[2] = __fmaf_rn(cw, a.z, o[2]); o[3] = __fmaf_rn(cw, a.w, o[3]);
      o[4] = __fmaf_rn(cw, bq.x, o[4]); o[5] = __fmaf_rn(cw, bq.y, o[5]);
      o[6] = __fmaf_rn(cw, bq.z, o[6]); o[7] = __fmaf_rn(cw, bq.w, o[7]);
    }
    const int head = d.kvh * kGqaGroup + eh;
    if (d.nsplit == 1) {
      finalize(p, d.b, head, ed, o, mc, lc);
    } else if (kCluster) {
      // leave this split's (O, m, l) in shared memory, where the cluster's
      // first CTA reads it after the cluster barrier below
      named_bar_sync(1, kConsumers);  // every warp is done reading wbuf
      float* cp = wbuf + eh * kGqaHeadDim + ed;
      *reinterpret_cast<float4*>(cp) = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4*>(cp + 4) = make_float4(o[4], o[5], o[6], o[7]);
      if (ed == 0) {
        wbuf[kGqaPartialFloats + eh] = mc;
        wbuf[kGqaPartialFloats + kGqaGroup + eh] = lc;
      }
      cl_nsplit = d.nsplit;
      cl_b = d.b;
      cl_kvh = d.kvh;
    } else {
      // publish this split, then count arrivals in its group of <= 16 splits
      store_partial(p, d.item, eh, ed, o, mc, lc);
      const long long first = d.item - d.split;
      const int gi = d.split / kMergeGroup;
      const long long gfirst = first + gi * kMergeGroup;
      const int gsize = min(kMergeGroup, d.nsplit - gi * kMergeGroup);
      const int ngroups = (d.nsplit + kMergeGroup - 1) / kMergeGroup;
      int* gcnt = p.group_counters + gfirst;
      named_bar_sync(1, kConsumers);
      if (tid == 0) misc[12] = atomic_add_acq_rel_gpu(gcnt, 1);
      named_bar_sync(1, kConsumers);
      if (misc[12] == gsize - 1) {
        float M, Ls;
        merge_slots(p, gfirst, 1, gsize, wbuf, eh, ed, o, M, Ls);
        if (tid == 0) store_relaxed_gpu(gcnt, 0);
        if (ngroups == 1) {
          finalize(p, d.b, head, ed, o, M, Ls);
        } else {
          store_partial(p, gfirst, eh, ed, o, M, Ls);  // the group result
          int* tcnt = p.counters + d.b * p.Hkv + d.kvh;
          named_bar_sync(1, kConsumers);
          if (tid == 0) misc[13] = atomic_add_acq_rel_gpu(tcnt, 1);
          named_bar_sync(1, kConsumers);
          if (misc[13] == ngroups - 1) {
            merge_slots(p, first, kMergeGroup, ngroups, wbuf, eh, ed, o, M, Ls);
            if (tid == 0) store_relaxed_gpu(tcnt, 0);
            finalize(p, d.b, head, ed, o, M, Ls);
          }
        }
      }
    }
    named_bar_sync(1, kConsumers);  // wbuf and misc are reused by the next item
  }
  }  // consumer warps

  if constexpr (kCluster) {
    // Split merge through distributed shared memory (the Flint page's cluster
    // reduction): after the first barrier every CTA's partial is visible; the
    // cluster's first CTA merges them in split order (the result does not
    // depend on timing) and writes out / lse; the second barrier keeps every
    // CTA, and so its shared memory, alive until those reads are done.  Every
    // thread of every CTA reaches both barriers (all earlier waits are bounded).
    cluster_sync();
    if (warp < kConsumerWarps && cl_nsplit > 1 && blockIdx.x == 0) {
      const uint32_t wb0 = smem_u32(wbuf);
      float o[8], M = -INFINITY, Ls = 0.f;
      float ms[kGqaMaxCluster];
#pragma unroll
      for (int r = 0; r < kGqaMaxCluster; ++r)
        ms[r] = r < cl_nsplit
                    ? ld_cluster_f32(map_shared_rank(wb0 + 4u * (kGqaPartialFloats + eh), r))
                    : -INFINITY;
#pragma unroll
      for (int r = 0; r < kGqaMaxCluster; ++r) M = fmaxf(M, ms[r]);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = 0.f;
      const float c2 = p.scale_log2;
#pragma unroll
      for (int r = 0; r < kGqaMaxCluster; ++r) {
        if (r < cl_nsplit) {
          const uint32_t base_r = map_shared_rank(wb0, r);
          const float w = (ms[r] == -INFINITY) ? 0.f : ex2((ms[r] - M) * c2);
          const float lr = ld_cluster_f32(base_r + 4u * (kGqaPartialFloats + kGqaGroup + eh));
          const float4 a = ld_cluster_f4(base_r + 4u * (eh * kGqaHeadDim + ed));
          const float4 c = ld_cluster_f4(base_r + 4u * (eh * kGqaHeadDim + ed + 4));
          Ls = __fmaf_rn(w, lr, Ls);
          o[0] = __fmaf_rn(w, a.x, o[0]); o[1] = __fmaf_rn(w, a.y, o[1]);
          o[2] = __fmaf_rn(w, a.z, o[2]); o[3] = __fmaf_rn(w, a.w, o[3]);
          o[4] = __fmaf_rn(w, c.x, o[4]); o[5] = __fmaf_rn(w, c.y, o[5]);
          o[6] = __fmaf_rn(w, c.z, o[6]); o[7] = __fmaf_rn(w, c.w, o[7]);
        }
      }
      finalize(p, cl_b, cl_kvh * kGqaGroup + eh, ed, o, M, Ls);
    }
    cluster_sync();
  }
}

template <int P, bool kCluster>
cudaError_t launch_page(const GqaParams& p, const CUtensorMap& kv_map, int grid,
                        cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  const cudaError_t e =
      set_smem_attr_once(gqa_decode_kernel<P, kCluster>, kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  // launched as a programmatic dependent of the previous kernel on the stream:
  // its launch and pre-wait prologue overlap that kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = kCluster ? dim3(p.cluster, p.B * p.Hkv) : dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCluster ? p.cluster : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kCluster ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gqa_decode_kernel<P, kCluster>, p, kv_map);
}

}  // namespace

int gqa_ctas_per_sm() { return kCtasPerSm; }

cudaError_t launch_gqa_decode(const GqaParams& p, const CUtensorMap& kv_map, int page_size,
                              int grid, cudaStream_t stream) {
  if (p.cluster > 1) {
    if (p.cluster > kGqaMaxCluster) return cudaErrorInvalidValue;
    return page_size == 16 ? launch_page<16, true>(p, kv_map, grid, stream)
                           : launch_page<32, true>(p, kv_map, grid, stream);
  }
  return page_size == 16 ? launch_page<16, false>(p, kv_map, grid, stream)
                         : launch_page<32, false>(p, kv_map, grid, stream);
}

}  // namespace pkv
