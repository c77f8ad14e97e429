// gqa_decode.cu -- split-KV paged GQA decode attention for sm_103a.
//
// Computes, for every request b and query head h (kv head h / 8),
//   out = sum_j softmax_j(scale * q.k_j) v_j  with an optional sink logit in
//   the denominator, lse = natural-log sum over keys of exp(scale * q.k_j),
// over keys [max(L - window, 0), L) gathered through block_table
// ("vllm.models.flint.ops.decode_attention": flint_decode_attention and the
// module's numerics paragraph; block-table indexing as in the transformers
// "Atencion paginada" decode path).
//
// Design (one persistent CTA per SM, 1 producer warp + 8 consumer warps):
//  * Work items are (request, kv head, split) triples.  Every CTA derives the
//    same item list in its prologue from seq_lens alone: request b's n_b
//    attended pages are cut into s_b = min(cap, ceil(n_b / chunk)) contiguous
//    splits, with chunk chosen from the total so that the launch has about
//    target_items items (shorter requests use fewer splits).  CTAs pull items
//    from a global queue (atomic head, reset by the last CTA to exit).
//  * The producer warp reads block-table entries 32 at a time and streams each
//    page of an item as four 128-byte-wide TMA tiles (K lo, K hi, V lo, V hi)
//    with 128-byte swizzle into a 128 KB ring of page stages guarded by
//    full/empty mbarriers; it runs ahead across item boundaries.
//  * Consumer warp w handles pages w, w+8, ... of the item.  Per 16-token tile:
//      S[8 heads x 16 tok] = Q K^T      mma.m16n8k16 (heads are the M side,
//                                         rows 8..15 zero), K via ldmatrix
//      online softmax in the exp2 domain (running max in unscaled logits),
//      O^T[128 dims x 8 heads] += V^T P^T  mma.m16n8k16 with V via
//                                         ldmatrix.trans and P^T taken
//                                         straight from S's accumulator layout
//    The 128-byte swizzle makes every ldmatrix phase conflict-free.
//  * The 8 warps' (O, m, l) are merged through shared memory.  A single-split
//    item writes out / lse directly; otherwise it publishes an fp32 partial and
//    bumps the (request, kv head) arrival counter; the CTA that arrives last
//    merges all partials and resets the counter to zero.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kRingBytes = 128 * 1024;
constexpr int kItemSlots = 4;
constexpr int kWbRow = 132;                                  // padded O row (floats)
constexpr int kWbFloats = kGqaGroup * kWbRow + 2 * kGqaGroup;  // O[8][132], m[8], l[8]
constexpr float kLog2e = 1.4426950408889634f;

struct ItemDesc {
  int item, b, kvh, split, nsplit, p0, p1, start_tok, L, seq_base, pad0, pad1;
};

template <int P>
struct Cfg {
  static constexpr int kStageBytes = P * 512;  // P tokens x [K | V] x bf16
  static constexpr int kStages = kRingBytes / kStageBytes;
  static constexpr int kTiles = P / 16;
  static constexpr int kChunkBytes = P * 128;  // one 64-element-wide TMA tile
  // shared-memory carve-up (offsets from a 1024-aligned base, 16-aligned)
  static constexpr int kOffWbuf = kRingBytes;
  static constexpr int kOffPrefix = kOffWbuf + kConsumerWarps * kWbFloats * 4;
  static constexpr int kOffLens = kOffPrefix + ((kGqaMaxBatch + 1) * 4 + 15) / 16 * 16;
  static constexpr int kOffItems = kOffLens + kGqaMaxBatch * 4;
  static constexpr int kOffBars = kOffItems + kItemSlots * (int)sizeof(ItemDesc);
  static constexpr int kNumBars = 2 * kStages + 2 * kItemSlots;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kOffWbuf % 16 == 0 && kOffPrefix % 16 == 0 && kOffLens % 16 == 0 &&
                    kOffItems % 16 == 0 && kOffBars % 16 == 0 && kOffMisc % 16 == 0,
                "shared-memory offsets must stay 16-byte aligned");
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

// Exclusive scan of one int per thread over the whole CTA; `scratch` holds
// one int per warp plus one.  Returns the exclusive prefix; *total = sum.
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

// Writes the final bf16 output row slice and lse of one (request, head).
__device__ __forceinline__ void finalize(const GqaParams& p, int b, int head, int d4, float o0,
                                         float o1, float o2, float o3, float m, float l,
                                         bool write_lse) {
  float inv = 0.f;
  if (l > 0.f) {
    float den = l;
    if (p.sinks) den += ex2(__fmaf_rn(p.sinks[head], kLog2e, -m * p.scale_log2));
    inv = 1.f / den;
  }
  uint2 v;
  v.x = pack_bf16(o0 * inv, o1 * inv);
  v.y = pack_bf16(o2 * inv, o3 * inv);
  *reinterpret_cast<uint2*>(p.out + b * p.o_sb + head * p.o_sh + d4) = v;
  if (write_lse && p.lse)
    p.lse[b * p.lse_sb + head * p.lse_sh] = (l > 0.f) ? m * p.scale + logf(l) : -INFINITY;
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_decode_kernel(const __grid_constant__ GqaParams p, const __grid_constant__ CUtensorMap kv_map) {
  using C = Cfg<P>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);

  const uint32_t ring = base_u32;
  float* wbuf = reinterpret_cast<float*>(base + C::kOffWbuf);
  int* prefix = reinterpret_cast<int*>(base + C::kOffPrefix);
  int* lens = reinterpret_cast<int*>(base + C::kOffLens);
  ItemDesc* items = reinterpret_cast<ItemDesc*>(base + C::kOffItems);
  const uint32_t bars = base_u32 + C::kOffBars;
  int* misc = reinterpret_cast<int*>(base + C::kOffMisc);
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
  auto ifull_bar = [&](int s) { return bars + 8u * (2 * C::kStages + s); };
  auto iempty_bar = [&](int s) { return bars + 8u * (2 * C::kStages + kItemSlots + s); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(ifull_bar(s), 1);
      mbar_init(iempty_bar(s), kConsumerWarps);
    }
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) tma_prefetch_desc(&kv_map);

  // ---- prologue: the item list, identical in every CTA -------------------
  // pass 1: clamp lengths, count attended pages.
  const int B = p.B;
  long long local_pages = 0;
  for (int b = tid; b < B; b += kThreads) {
    int L = p.seq_lens[b];
    if (L < 0) L = 0;
    if ((long long)(L + P - 1) / P > p.max_blocks) {
      atomicOr(p.err, DEVERR_SEQ_TOO_LONG);
      L = p.max_blocks * P;
    }
    lens[b] = L;
    const int start_tok = (p.window > 0 && L > p.window) ? L - p.window : 0;
    local_pages += (L + P - 1) / P - start_tok / P;
  }
  {
    int lp = (int)local_pages;
    int tot;
    block_exclusive_scan(lp, misc, &tot);
    local_pages = tot;
  }
  const long long total_pages = local_pages * p.Hkv;
  int chunk = (int)((total_pages + p.target_items - 1) / p.target_items);
  if (chunk < p.min_pages) chunk = p.min_pages;
  // pass 2: splits per request, exclusive prefix of items over requests.
  const int per = (B + kThreads - 1) / kThreads;
  const int b0 = tid * per;
  int my_items = 0;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    if (b >= B) break;
    const int L = lens[b];
    const int start_tok = (p.window > 0 && L > p.window) ? L - p.window : 0;
    const int n = (L + P - 1) / P - start_tok / P;
    int s = (n + chunk - 1) / chunk;
    s = s < 1 ? 1 : (s > p.cap ? p.cap : s);
    my_items += s * p.Hkv;
  }
  int total_items;
  int run = block_exclusive_scan(my_items, misc, &total_items);
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    if (b >= B) break;
    prefix[b] = run;
    const int L = lens[b];
    const int start_tok = (p.window > 0 && L > p.window) ? L - p.window : 0;
    const int n = (L + P - 1) / P - start_tok / P;
    int s = (n + chunk - 1) / chunk;
    s = s < 1 ? 1 : (s > p.cap ? p.cap : s);
    run += s * p.Hkv;
  }
  if (tid == 0) prefix[B] = total_items;
  if ((long long)total_items > p.max_items) {
    if (tid == 0) atomicOr(p.err, DEVERR_ITEM_OVERFLOW);
    total_items = (int)p.max_items;
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ===================== producer warp =====================
    int next = 0;
    if (lane == 0) next = atomicAdd(&p.sched[0], 1);
    next = __shfl_sync(0xffffffffu, next, 0);
    uint32_t seq = 0;
    for (int it = 0;; ++it) {
      const int item = next;
      if (item < total_items) {
        if (lane == 0) next = atomicAdd(&p.sched[0], 1);
        next = __shfl_sync(0xffffffffu, next, 0);
      }
      const int slot = it % kItemSlots;
      const uint32_t par = (it / kItemSlots) & 1;
      if (lane == 0) mbar_wait(iempty_bar(slot), par ^ 1u, p.err);
      __syncwarp();
      if (item >= total_items) {
        if (lane == 0) {
          items[slot].item = -1;
          mbar_arrive(ifull_bar(slot));
        }
        break;
      }
      // decode: request = last b with prefix[b] <= item
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
      }
      const int b = lo;
      const int nsplit = (prefix[b + 1] - prefix[b]) / p.Hkv;
      const int local = item - prefix[b];
      const int kvh = local / nsplit, split = local % nsplit;
      const int L = lens[b];
      const int start_tok = (p.window > 0 && L > p.window) ? L - p.window : 0;
      const int sp = start_tok / P;
      const int n = (L + P - 1) / P - sp;
      const int p0 = sp + (int)((long long)n * split / nsplit);
      const int p1 = sp + (int)((long long)n * (split + 1) / nsplit);
      if (lane == 0) {
        ItemDesc& d = items[slot];
        d.item = item; d.b = b; d.kvh = kvh; d.split = split; d.nsplit = nsplit;
        d.p0 = p0; d.p1 = p1; d.start_tok = start_tok; d.L = L; d.seq_base = (int)seq;
        mbar_arrive(ifull_bar(slot));  // release: the descriptor is visible to waiters
      }
      const int32_t* bt_row = p.bt + (long long)b * p.bt_sb;
      for (int pb = p0; pb < p1; pb += 32) {
        const int cnt = min(32, p1 - pb);
        int blk = 0;
        if (lane < cnt) {
          blk = __ldg(bt_row + pb + lane);
          if (blk < 0 || blk >= p.num_blocks) atomicOr(p.err, DEVERR_BAD_BLOCK);
        }
        for (int i = 0; i < cnt; ++i) {
          const int blk_i = __shfl_sync(0xffffffffu, blk, i);
          if (lane == 0) {
            const int stage = seq % C::kStages;
            const uint32_t ph = (seq / C::kStages) & 1;
            mbar_wait(empty_bar(stage), ph ^ 1u, p.err);
            mbar_arrive_expect_tx(full_bar(stage), C::kStageBytes);
            const uint32_t dst = ring + stage * C::kStageBytes;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              tma_load_4d(dst + c * C::kChunkBytes, &kv_map, full_bar(stage), 64 * c, 0, kvh, blk_i);
          }
          ++seq;
        }
      }
    }
    // Every issued copy has landed before the CTA may exit (the consumers
    // waited on them already unless a wait gave up).
    if (lane == 0) {
      const uint32_t n_recent = seq < (uint32_t)C::kStages ? seq : (uint32_t)C::kStages;
      for (uint32_t k = seq - n_recent; k < seq; ++k)
        mbar_wait(full_bar(k % C::kStages), (k / C::kStages) & 1, p.err);
    }
    // last CTA out resets the queue for the next launch
    if (lane == 0) {
      __threadfence();
      const int old = atomicAdd(&p.sched[1], 1);
      if (old == (int)gridDim.x - 1) {
        atomicExch(&p.sched[0], 0);
        atomicExch(&p.sched[1], 0);
      }
    }
    return;
  }

  // ======================= consumer warps =======================
  const int g = lane >> 2, t = lane & 3;
  // ldmatrix lane addressing: matrix mi = lane / 8 supplies row r = lane % 8;
  // matrices 0,1: tile rows 0..7; 2,3: rows 8..15; odd matrices: the upper
  // 8 elements (next 16-byte unit) of a 16-element k-step.
  const int mi = lane >> 3, r = lane & 7;
  const uint32_t row_off = (uint32_t)(r + 8 * (mi >> 1)) * 128u;
  const int ubit = mi & 1;
  float* my_wb = wbuf + warp * kWbFloats;
  const int ct = tid;  // consumer thread index 0..255
  const int eh = ct >> 5, ed = (ct & 31) * 4;  // epilogue: head, first of 4 dims

  for (int it = 0;; ++it) {
    const int slot = it % kItemSlots;
    mbar_wait(ifull_bar(slot), (it / kItemSlots) & 1, p.err);
    const ItemDesc d = items[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(iempty_bar(slot));
    if (d.item < 0) break;

    // Q as the A operand (rows = the 8 heads of this kv head; rows 8..15 zero).
    uint32_t qa[8][2];
    {
      const uint16_t* qrow = p.q + d.b * p.q_sb + (d.kvh * kGqaGroup + g) * p.q_sh;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        qa[s][0] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * s + 2 * t));
        qa[s][1] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * s + 8 + 2 * t));
      }
    }
    float acc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    float m = -INFINITY, l = 0.f;
    const float c2 = p.scale_log2;

    const int npages = d.p1 - d.p0;
    for (int k = warp; k < npages; k += kConsumerWarps) {
      const uint32_t seq = (uint32_t)d.seq_base + (uint32_t)k;
      const int stage = seq % C::kStages;
      mbar_wait(full_bar(stage), (seq / C::kStages) & 1, p.err);
      const uint32_t st = ring + stage * C::kStageBytes;
      const int page = d.p0 + k;
#pragma unroll
      for (int u = 0; u < C::kTiles; ++u) {
        const int tok0 = page * P + 16 * u;
        const uint32_t tile = st + 16u * u * 128u + row_off;
        // ---- S = Q K^T over 128 dims: 4 independent accumulator chains ----
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const uint32_t unit = (uint32_t)((2 * (s & 3) + ubit) ^ r);
          uint32_t k0, k1, k2, k3;
          ldsm_x4(tile + (s >> 2) * C::kChunkBytes + (unit << 4), k0, k1, k2, k3);
          if (s & 1) {
            mma_bf16_16816(sb, qa[s][0], 0u, qa[s][1], 0u, k0, k1);
            mma_bf16_16816(sd, qa[s][0], 0u, qa[s][1], 0u, k2, k3);
          } else {
            mma_bf16_16816(sa, qa[s][0], 0u, qa[s][1], 0u, k0, k1);
            mma_bf16_16816(sc, qa[s][0], 0u, qa[s][1], 0u, k2, k3);
          }
        }
        // lane (g, t): head g, tile tokens 2t, 2t+1 (x0, x1) and 8+2t, 9+2t (x2, x3)
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
        const float msc = (mn == -INFINITY) ? 0.f : mn * c2;
        const float alpha = ex2(__fmaf_rn(m, c2, -msc));
        const float e0 = ex2(__fmaf_rn(x0, c2, -msc));
        const float e1 = ex2(__fmaf_rn(x1, c2, -msc));
        const float e2 = ex2(__fmaf_rn(x2, c2, -msc));
        const float e3 = ex2(__fmaf_rn(x3, c2, -msc));
        l = __fmaf_rn(l, alpha, (e0 + e1) + (e2 + e3));
        m = mn;
        // O^T columns are heads 2t, 2t+1: fetch their rescale factors
        const float al0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
        const float al1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[j][0] *= al0; acc[j][1] *= al1; acc[j][2] *= al0; acc[j][3] *= al1;
        }
        // P^T as the B operand: exactly S's accumulator pairs, rounded to bf16
        const uint32_t pb0 = pack_bf16(e0, e1), pb1 = pack_bf16(e2, e3);
        // V rows outside [start_tok, L) are zeroed: stale cache contents
        // (NaN, Inf) must not reach P.V even with P = 0.
        const bool edge = (tok0 < d.start_tok) || (tok0 + 16 > d.L);
        const uint32_t mlo = (v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u);
        const uint32_t mhi = (v2 ? 0x0000ffffu : 0u) | (v3 ? 0xffff0000u : 0u);
        // ---- O^T += V^T P^T: 8 m-tiles of 16 dims ----
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t unit = (uint32_t)((2 * (j & 3) + ubit) ^ r);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(tile + (2 + (j >> 2)) * C::kChunkBytes + (unit << 4), a0, a1, a2, a3);
          if (edge) { a0 &= mlo; a1 &= mlo; a2 &= mhi; a3 &= mhi; }
          mma_bf16_16816(acc[j], a0, a1, a2, a3, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(stage));
    }

    // ---- merge the 8 warps' (O, m, l) through shared memory ----
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
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f, lc = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float* wb = wbuf + w * kWbFloats;
      const float mw = wb[kGqaGroup * kWbRow + eh];
      const float cw = (mw == -INFINITY) ? 0.f : ex2((mw - mc) * c2);
      lc = __fmaf_rn(cw, wb[kGqaGroup * kWbRow + kGqaGroup + eh], lc);
      const float4 ov = *reinterpret_cast<const float4*>(wb + eh * kWbRow + ed);
      o0 = __fmaf_rn(cw, ov.x, o0); o1 = __fmaf_rn(cw, ov.y, o1);
      o2 = __fmaf_rn(cw, ov.z, o2); o3 = __fmaf_rn(cw, ov.w, o3);
    }
    const int head = d.kvh * kGqaGroup + eh;
    if (d.nsplit == 1) {
      finalize(p, d.b, head, ed, o0, o1, o2, o3, mc, lc, ed == 0);
    } else {
      float* po = p.part_o + (long long)d.item * kGqaPartialFloats + eh * kGqaHeadDim + ed;
      *reinterpret_cast<float4*>(po) = make_float4(o0, o1, o2, o3);
      if (ed == 0) {
        p.part_ml[(long long)d.item * kGqaMlFloats + eh] = mc;
        p.part_ml[(long long)d.item * kGqaMlFloats + kGqaGroup + eh] = lc;
      }
      __threadfence();
      named_bar_sync(1, kConsumers);
      int* counter = p.counters + d.b * p.Hkv + d.kvh;
      if (ct == 0) misc[8] = atomicAdd(counter, 1);
      named_bar_sync(1, kConsumers);
      if (misc[8] == d.nsplit - 1) {
        __threadfence();
        const long long first = d.item - d.split;
        float M = -INFINITY;
        for (int s = 0; s < d.nsplit; ++s)
          M = fmaxf(M, __ldcg(p.part_ml + (first + s) * kGqaMlFloats + eh));
        o0 = o1 = o2 = o3 = 0.f;
        float Ls = 0.f;
#pragma unroll 4
        for (int s = 0; s < d.nsplit; ++s) {
          const float ms = __ldcg(p.part_ml + (first + s) * kGqaMlFloats + eh);
          const float ls = __ldcg(p.part_ml + (first + s) * kGqaMlFloats + kGqaGroup + eh);
          const float4 ov = ldcg_f4(p.part_o + (first + s) * kGqaPartialFloats + eh * kGqaHeadDim + ed);
          const float w = (ms == -INFINITY) ? 0.f : ex2((ms - M) * c2);
          Ls = __fmaf_rn(w, ls, Ls);
          o0 = __fmaf_rn(w, ov.x, o0); o1 = __fmaf_rn(w, ov.y, o1);
          o2 = __fmaf_rn(w, ov.z, o2); o3 = __fmaf_rn(w, ov.w, o3);
        }
        finalize(p, d.b, head, ed, o0, o1, o2, o3, M, Ls, ed == 0);
        if (ct == 0) *counter = 0;  // self-reset for the next launch
      }
    }
    named_bar_sync(1, kConsumers);  // wbuf and misc[8] are reused by the next item
  }
}

}  // namespace

size_t gqa_smem_bytes(int page_size) {
  return page_size == 16 ? Cfg<16>::kBytes : Cfg<32>::kBytes;
}

template <int P>
static cudaError_t launch_page(const GqaParams& p, const CUtensorMap& kv_map, int grid,
                               cudaStream_t stream) {
  static bool attr_set = false;  // per process; the attribute is per device function
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        gqa_decode_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<P>::kBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  gqa_decode_kernel<P><<<grid, kThreads, Cfg<P>::kBytes, stream>>>(p, kv_map);
  return cudaGetLastError();
}

cudaError_t launch_gqa_decode(const GqaParams& p, const CUtensorMap& kv_map, int page_size,
                              int grid, cudaStream_t stream) {
  return page_size == 16 ? launch_page<16>(p, kv_map, grid, stream)
                         : launch_page<32>(p, kv_map, grid, stream);
}

}  // namespace pkv
