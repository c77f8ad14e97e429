// mla_verify_pair.cu -- causal MLA verify over a paged bf16 latent cache on
// CTA pairs (tcgen05 cta_group::2), for an even number of verify tokens.
//
// Computes what mla_verify.cu computes (see there, and
// "vllm.v1.attention.ops.triton_decode_attention", decode_attention_fwd_verify:
// parameters): for verify token t of request b and each of the 128 heads,
// out = softmax over keys [0, lim_t) of scale * q.K_j, applied to K_j[:512],
// lim_t = max(min(L - qlen + 1 + t, L_real), 0), and lse; splits of a request
// publish fp32 (O half, m, l) partials that the last split merges.
//
// The two verify tokens 2tp and 2tp + 1 of a request see the same keys, so a
// cluster of two CTAs shares every key tile between them: CTA rank r handles
// token 2tp + r and one half of the 512 output dims (the same half in both).
//  * A tile is 64 keys.  Each CTA loads its 32-key half of the tile (all 576
//    dims, four TMA boxes of 8 keys x 9 chunks, 36 KB, into a 3-slot ring
//    released as soon as the tile's S is done) and, for P V, all 64 keys of
//    its 128 V dims (four boxes of 16 keys x 2 chunks, 16 KB, into a 3-slot
//    ring released after P V).  Both CTAs' key loads complete on the even
//    CTA's barrier; each CTA's V loads on its own.
//  * S = Q K^T is one M = 256 (128 heads x 2 tokens) x N = 64 (keys) MMA
//    chain issued by the even CTA: rows of token 2tp + r live in CTA r's TMEM
//    (query dims 0..383, 24 K16 steps) or shared memory (dims 384..575, 12
//    steps); keys 0..31 of the tile come from the even CTA's shared memory,
//    32..63 from the odd one's.  O += P V is M = 256 x N = 256 (this half's
//    dims, 128 from each CTA) x K = 64.  Commits arrive in both CTAs.
//  * Eight softmax warps per CTA, two per TMEM lane quarter, each taking 32
//    of the 64 score columns; the row max of a tile is combined through shared
//    memory; exp2-domain softmax with a lazily updated reference max (O is
//    rescaled in TMEM only when the max grows by more than 2^8).
// TMEM (512 columns, allocated by the pair): O half [0, 256), S [256, 320),
// query dims 0..383 as bf16 pairs [320, 512).
#include "pkv_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"
#include "mla_common.cuh"

namespace pkv {
namespace {
using namespace mla;

constexpr int kThreads = 384;       // warp 0 loads, warp 1 MMA, warps 4..11 softmax
constexpr int kSoftmaxWarp0 = 4;
constexpr int kSoftmaxThreads = 256;
constexpr int kTile = 64;           // keys per tile of the pair
constexpr int kChunks = kMlaLk / 64;
constexpr int kQtChunks = 6;        // query dims [0, 384) in TMEM
constexpr int kQsChunks = kChunks - kQtChunks;
constexpr int kQChunkBytes = kMlaHeads * 128;
constexpr int kQsBytes = kQsChunks * kQChunkBytes;       // 49152
constexpr int kGroupBytes = kChunks * 1024;              // 9216: 8 keys x 576 dims
constexpr int kKBytes = 4 * kGroupBytes;                 // 36864: this CTA's 32 keys
constexpr int kVBoxBytes = 16 * 2 * 128;                 // 4096: 16 keys x 2 chunks
constexpr int kVBytes = 4 * kVBoxBytes;                  // 16384: 64 keys x 128 dims
constexpr int kStages = 3;                               // slots of each ring
constexpr int kPBytes = kMlaHeads * kTile * 2;           // 16384 (128-byte rows)
constexpr int kOffK = kQsBytes;
constexpr int kOffV = kOffK + kStages * kKBytes;
constexpr int kOffP = kOffV + kStages * kVBytes;
constexpr int kOffBars = kOffP + kPBytes;
constexpr int kOffRed = kOffBars + 256;                  // [3][2][128] floats
constexpr int kSmemBytes = kOffRed + 3 * 2 * 128 * 4 + 1024;  // + alignment slack
static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0 &&
                  kKBytes % 1024 == 0 && kVBytes % 1024 == 0,
              "swizzle atoms need 1024 B alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
// At a unit's start the query dims [0, 384) land by TMA in a staging area over
// key slot 2, the V ring and P (free until the first tiles are consumed).
constexpr int kOffStaging = kOffK + 2 * kKBytes;
constexpr int kQtBytes = kQtChunks * kQChunkBytes;       // 98304
static_assert(kOffStaging + kQtBytes <= kOffP + kPBytes && kOffStaging % 1024 == 0,
              "query staging area");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
constexpr uint32_t kTmemQ = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

// barriers (same offsets in both CTAs; the ones marked "even" are used in
// the even CTA only, with arrivals from both)
enum {
  kQFull = 0,     // this CTA's query landed (TMA: dims 384..575, and 0..383 staged)
  kQtReady = 1,   // query dims 0..383 moved from staging into TMEM (256 arrivals)
  kQReady = 2,    // even: both CTAs' query ready (2 arrivals)
  kKFull = 3,     // even: key slot s of both CTAs landed (2 arrivals + bytes), 3 slots
  kKEmpty = 6,    // key slot s free (pair commit after S), 3 slots
  kVFull = 9,     // this CTA's V slot s landed, 3 slots
  kVEmpty = 12,   // V slot s free (pair commit after P V), 3 slots
  kSFull = 15,    // S in TMEM (pair commit)
  kSFree = 16,    // even: S read by all softmax warps of both CTAs (16 arrivals)
  kPFull = 17,    // even: P of both CTAs written, their V slots ready (2 arrivals)
  kPvDone = 18,   // P V done (pair commit)
  kNumBars = 19
};

struct PairUnit {
  int b, split, t, half, nsplit;
  int L, lim, lim_max;  // this token's row limit; the pair's largest
  int tile0, ntiles;    // 64-key tiles [tile0, tile0 + ntiles) of this split
  bool valid;
};

// The unit of this CTA's cluster from the plan (plan_entry: request b, token
// pair tp, half, split and split count; or -1), and this CTA's token 2tp + rank.
__device__ __forceinline__ PairUnit decode_pair_unit(const MlaParams& p, int rank) {
  PairUnit u;
  const int v = __ldg(p.plan + (blockIdx.x >> 1));
  u.valid = v >= 0;
  if (!u.valid) return u;
  u.split = (v >> 4) & 15;
  const int ns = (v & 15) + 1;
  const int ch = v >> 8;
  u.half = ch & 1;
  const int rt = ch >> 1, npairs = p.qlen >> 1;
  u.b = rt / npairs;
  const int tp = rt - u.b * npairs;
  u.t = 2 * tp + rank;
  const int L = clamped_len(p, u.b);
  const int Lr = p.real_seq_lens ? __ldg(p.real_seq_lens + u.b) : L;
  auto lim_of = [&](int t) { return max(min(L - p.qlen + 1 + t, Lr), 0); };
  u.L = L;
  u.lim = lim_of(u.t);
  u.lim_max = max(lim_of(2 * tp), lim_of(2 * tp + 1));
  const int req_tiles = (L + kTile - 1) / kTile;
  u.nsplit = ns;
  const int a = (int)((long long)req_tiles * u.split / ns);
  const int e = (int)((long long)req_tiles * (u.split + 1) / ns);
  u.tile0 = a;
  u.ntiles = max(0, min(e, (u.lim_max + kTile - 1) / kTile) - a);
  return u;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_verify_pair_kernel(const __grid_constant__ MlaParams p,
                           const __grid_constant__ CUtensorMap q_map,
                           const __grid_constant__ CUtensorMap kv_map,
                           const __grid_constant__ CUtensorMap v_map) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sQ = base_u32, sP = base_u32 + kOffP;
  auto sK = [&](int st) { return base_u32 + kOffK + st * kKBytes; };
  auto sV = [&](int st) { return base_u32 + kOffV + st * kVBytes; };
  const uint32_t bars = base_u32 + kOffBars;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + kOffBars + 8 * kNumBars);
  int* flag = reinterpret_cast<int*>(base + kOffBars + 8 * kNumBars + 8);
  float* red = reinterpret_cast<float*>(base + kOffRed);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  if (tid == 0) {
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQtReady), kSoftmaxThreads);
    mbar_init(bar(kQReady), 2);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(kKFull + s), 2);
      mbar_init(bar(kKEmpty + s), 1);
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    mbar_init(bar(kSFull), 1);
    mbar_init(bar(kSFree), 2 * (kSoftmaxThreads / 32));
    mbar_init(bar(kPFull), 2);
    mbar_init(bar(kPvDone), 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&q_map);
    tma_prefetch_desc(&kv_map);
    tma_prefetch_desc(&v_map);
  }
  // Programmatic dependent launch: the plan comes from the kernel before.
  griddep_wait();
  griddep_launch_dependents();
  const PairUnit u = decode_pair_unit(p, (int)rank);
  if (!u.valid) return;  // both CTAs of the cluster read the same entry

  if (warp == 1) tc::tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
  tc::fence_before_sync();
  cluster_sync();  // both CTAs' barriers initialised and the pair's TMEM allocated
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  auto even_bar = [&](int i) { return map_shared_rank(bar(i), 0); };
  const float c2 = p.scale * kLog2e;
  const int n = u.ntiles;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (n > 0) {
      const int qrow = u.b * p.qlen + u.t;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(kQFull), kQsBytes + kQtBytes);
        for (int c = 0; c < kQsChunks; ++c)
          tma_load_3d(sQ + c * kQChunkBytes, &q_map, bar(kQFull), 64 * (kQtChunks + c), 0, qrow);
        for (int c = 0; c < kQtChunks; ++c)
          tma_load_3d(base_u32 + kOffStaging + c * kQChunkBytes, &q_map, bar(kQFull), 64 * c, 0,
                      qrow);
      }
      const int32_t* bt_row = p.bt + (long long)u.b * p.bt_sb;
      const int vchunk = 4 * u.half + 2 * (int)rank;
      for (int g = 0; g < n; g += 8) {
        // lane l: block id and page offset of 16-key piece l % 4 of tile g + l / 4
        // (pieces past the request read as zeros: their page lies past the cache)
        const int gt = g + (lane >> 2);
        const int piece_tok = (u.tile0 + gt) * kTile + 16 * (lane & 3);
        int blk = p.num_pages, off = 0;
        if (gt < n && piece_tok < u.L) {
          blk = __ldg(bt_row + piece_tok / p.page_size);
          off = piece_tok % p.page_size;
          if (blk < 0 || blk >= p.num_pages) atomicOr(p.err, DEVERR_BAD_BLOCK);
        }
        for (int i = g; i < min(n, g + 8); ++i) {
          const int j = 4 * (i - g);
          int pb[4], po[4], pb1[4], po1[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            pb[q] = __shfl_sync(0xffffffffu, blk, j + q);
            po[q] = __shfl_sync(0xffffffffu, off, j + q);
            pb1[q] = __shfl_sync(0xffffffffu, blk, (j + 4 + q) & 31);  // tile i + 1 (used at i == 0)
            po1[q] = __shfl_sync(0xffffffffu, off, (j + 4 + q) & 31);
          }
          if (lane == 0) {
            // this CTA's 32 keys: pieces 2 rank, 2 rank + 1, two 8-key boxes each
            auto issue_k = [&](int t, const int (&b)[4], const int (&o)[4]) {
              const int sk = t % kStages;
              mbar_wait(bar(kKEmpty + sk), ((t / kStages) & 1) ^ 1u, p.err);
              const uint32_t full = even_bar(kKFull + sk);
              mbar_arrive_expect_tx_cluster(full, kKBytes);
              const uint32_t dk = sK(sk);
              const int h0 = 2 * (int)rank, h1 = h0 + 1;
              tma_load_4d_pair(dk, &kv_map, full, 0, o[h0], 0, b[h0]);
              tma_load_4d_pair(dk + kGroupBytes, &kv_map, full, 0, o[h0] + 8, 0, b[h0]);
              tma_load_4d_pair(dk + 2 * kGroupBytes, &kv_map, full, 0, o[h1], 0, b[h1]);
              tma_load_4d_pair(dk + 3 * kGroupBytes, &kv_map, full, 0, o[h1] + 8, 0, b[h1]);
            };
            if (i != 1) issue_k(i, pb, po);  // key tile 1 goes out with tile 0
            if (i == 0) {
              if (n > 1) issue_k(1, pb1, po1);
              // key slot 2, the V ring and P held the staged query until it
              // was moved into TMEM
              mbar_wait(bar(kQtReady), 0, p.err);
            }
            // all 64 keys of this CTA's 128 V dims: box q = keys 16q.., 2 chunks
            const int st = i % kStages;
            mbar_wait(bar(kVEmpty + st), ((i / kStages) & 1) ^ 1u, p.err);
            mbar_arrive_expect_tx(bar(kVFull + st), kVBytes);
            const uint32_t dv = sV(st);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              tma_load_4d(dv + q * kVBoxBytes, &v_map, bar(kVFull + st), 0, po[q], vchunk, pb[q]);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ==================== query handshake; MMA issue (even CTA) ====================
    if (n > 0) {
      mbar_wait(bar(kQFull), 0, p.err);
      mbar_wait(bar(kQtReady), 0, p.err);
      tc::fence_after_sync();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(even_bar(kQReady));
      if (rank == 0) {
        const uint32_t id_s = tc::idesc_bf16_f32(256, kTile, false, false);
        const uint32_t id_pv = tc::idesc_bf16_f32(256, kMlaHalf, false, true);
        mbar_wait(bar(kQReady), 0, p.err);
        tc::fence_after_sync();
        auto do_pv = [&](int j) {
          // P of both CTAs written and both CTAs' V slot landed (and zeroed
          // where no token attends)
          mbar_wait(bar(kPFull), j & 1, p.err);
          tc::fence_after_sync();
          const uint32_t vst = sV(j % kStages);
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks)
            tc::mma_pair_ss_elect(tmem + kTmemO, tc::smem_desc(sP + ks * 32, 16, 1024, tc::kSwizzle128),
                                  tc::smem_desc(vst + ks * kVBoxBytes, 2048, 1024, tc::kSwizzle128),
                                  id_pv, j > 0 || ks > 0);
          tc::commit_pair_elect(bar(kPvDone));
          // only slots the producer will refill get a release (every arrive
          // reaches a CTA that is still waiting for it)
          if (j + kStages < n) tc::commit_pair_elect(bar(kVEmpty + j % kStages));
        };
        for (int i = 0; i < n; ++i) {
          const int st = i % kStages;
          mbar_wait(bar(kKFull + st), (i / kStages) & 1, p.err);
          if (i > 0) mbar_wait(bar(kSFree), (i - 1) & 1, p.err);
          tc::fence_after_sync();
          const uint32_t kst = sK(st);
#pragma unroll 1
          for (int c = 0; c < kQtChunks; ++c) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_pair_ts_elect(
                  tmem + kTmemS, tmem + kTmemQ + (4 * c + ks) * 8,
                  tc::smem_desc(kst + c * 1024 + ks * 32, 16, kGroupBytes, tc::kSwizzle128), id_s,
                  (c | ks) != 0);
          }
#pragma unroll 1
          for (int c = kQtChunks; c < kChunks; ++c) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_pair_ss_elect(
                  tmem + kTmemS,
                  tc::smem_desc(sQ + (c - kQtChunks) * kQChunkBytes + ks * 32, 16, 1024,
                                tc::kSwizzle128),
                  tc::smem_desc(kst + c * 1024 + ks * 32, 16, kGroupBytes, tc::kSwizzle128), id_s,
                  true);
          }
          tc::commit_pair_elect(bar(kSFull));
          // the key slot is free once S is done (P V reads the V ring)
          if (i + kStages < n) tc::commit_pair_elect(bar(kKEmpty + st));
          if (i > 0) do_pv(i - 1);
        }
        do_pv(n - 1);
      }
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ============ softmax (one thread per head, half of the columns) + epilogue ============
    const int sw = warp - kSoftmaxWarp0, quarter = sw & 3, chalf = sw >> 2;
    const int row = 32 * quarter + lane;  // head = TMEM lane
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    if (n > 0) {
      // query dims [0, 384) from the staging area into TMEM: this warp writes
      // lanes 32 quarter .., chunks 3 chalf .. + 2 (row `row` of each 16 KB
      // chunk, 128-byte swizzle: 16-byte unit k at k ^ (row % 8))
      const int c0 = 3 * chalf;
      mbar_wait(bar(kQFull), 0, p.err);
      const uint8_t* stg = base + kOffStaging + (row / 8) * 1024 + (row % 8) * 128;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        uint32_t v[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 w = *reinterpret_cast<const uint4*>(stg + (c0 + j) * kQChunkBytes +
                                                          ((k ^ (row % 8)) * 16));
          v[4 * k] = w.x;
          v[4 * k + 1] = w.y;
          v[4 * k + 2] = w.z;
          v[4 * k + 3] = w.w;
        }
        tc::st_32x32b_x32(tmem + lane_base + kTmemQ + 32 * (c0 + j), v);
      }
      fence_proxy_async_smem();  // the staging area is refilled by TMA after this
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(bar(kQtReady));
    }
    float m_used = -INFINITY, l = 0.f;  // l: this warp's 32 columns of every tile
    uint8_t* p_row = base + kOffP + (row / 8) * 1024 + (row % 8) * 128;
    const int sidx = sw * 32 + lane;  // 0 .. 255
    for (int i = 0; i < n; ++i) {
      mbar_wait(bar(kSFull), i & 1, p.err);
      __syncwarp();  // tcgen05.ld is warp-collective
      tc::fence_after_sync();
      uint32_t xr[32];
      tc::ld_32x32b_x32(tmem + lane_base + kTmemS + 32 * chalf, xr);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(even_bar(kSFree)) : "memory");
      const int kb = (u.tile0 + i) * kTile;  // first key of the tile
      const int nvalid = min(32, u.lim - kb - 32 * chalf);
      float mo = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (c < nvalid) mo = fmaxf(mo, __uint_as_float(xr[c]));
      float* rb = red + (i & 1) * 256;
      rb[chalf * 128 + row] = mo;
      named_bar_sync(1, kSoftmaxThreads);
      const float mt = fmaxf(rb[row], rb[128 + row]);
      // lazy max (see mla_verify.cu): both warps of a lane quarter see the same
      // mt and m_used, so they take the same decisions
      bool waited = false;
      const bool need =
          mt > -INFINITY && (m_used == -INFINITY || (mt - m_used) * c2 > kRescaleLog2);
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_used;
        const float alpha =
            (m_used == -INFINITY) ? 0.f : (need ? ex2((m_used - m_new) * c2) : 1.f);
        if (i > 0) {
          // every P V so far must be done before O is rescaled in place
          mbar_wait(bar(kPvDone), (i - 1) & 1, p.err);
          waited = true;
          __syncwarp();
          tc::fence_after_sync();
          for (int j = 0; j < 4; ++j) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kTmemO + 128 * chalf + 32 * j;
            tc::ld_32x32b_x32(ta, o);
            tc::wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            tc::st_32x32b_x32(ta, o);
          }
          tc::wait_st();
        }
        l *= alpha;
        m_used = m_new;
      }
      const float msc = (m_used == -INFINITY) ? 0.f : m_used * c2;
      uint32_t pk[16];
      float lt = 0.f;
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const float e0 = (c < nvalid) ? ex2(__fmaf_rn(__uint_as_float(xr[c]), c2, -msc)) : 0.f;
        const float e1 =
            (c + 1 < nvalid) ? ex2(__fmaf_rn(__uint_as_float(xr[c + 1]), c2, -msc)) : 0.f;
        lt += e0 + e1;
        pk[c / 2] = pack_bf16(e0, e1);
      }
      l += lt;
      // the P buffer (and the stage's V rows) are free once P V of the
      // previous tile is done
      if (i > 0 && !waited) mbar_wait(bar(kPvDone), (i - 1) & 1, p.err);
#pragma unroll
      for (int uq = 0; uq < 4; ++uq)
        *reinterpret_cast<uint4*>(p_row + (((4 * chalf + uq) ^ (row % 8)) * 16)) =
            make_uint4(pk[4 * uq], pk[4 * uq + 1], pk[4 * uq + 2], pk[4 * uq + 3]);
      const int vvalid = u.lim_max - kb;  // keys of the tile either token attends
      mbar_wait(bar(kVFull + i % kStages), (i / kStages) & 1, p.err);  // this CTA's V slot
      if (vvalid < kTile) {
        // keys no token of the pair attends: zero their V rows (this CTA's 128
        // dims) so stale or poisoned cache contents never meet P = 0 in the MMA
        uint8_t* vst = base + kOffV + (i % kStages) * kVBytes;
        const int z0 = max(vvalid, 0), nz = kTile - z0;
        for (int q = sidx; q < nz * 16; q += kSoftmaxThreads) {
          const int key = z0 + q / 16, c = (q / 8) & 1, un = q & 7;
          *reinterpret_cast<uint4*>(vst + (key / 16) * kVBoxBytes + c * 2048 + (key % 16) * 128 +
                                    un * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();  // P and zeroed V rows are read by the MMA (async proxy)
      tc::fence_before_sync();   // and any in-place O rescale precedes the next P V
      __syncwarp();
      named_bar_sync(1, kSoftmaxThreads);
      if (sidx == 0) mbar_arrive_cluster(even_bar(kPFull));
    }

    // ------------------------------ epilogue ------------------------------
    if (n > 0) {
      mbar_wait(bar(kPvDone), (n - 1) & 1, p.err);
      __syncwarp();  // the TMEM loads below are warp-collective
      tc::fence_after_sync();
    }
    float* lr = red + 512;
    lr[chalf * 128 + row] = l;
    named_bar_sync(1, kSoftmaxThreads);
    const float lsum = lr[row] + lr[128 + row];
    const long long r = (long long)u.b * p.qlen + u.t;
    const int dim0 = u.half * kMlaHalf + 128 * chalf;  // this warp's 128 output dims
    uint16_t* out_row = p.out + r * p.o_sr + row * p.o_sh + dim0;
    const bool write_lse = u.half == 0 && chalf == 0;
    if (u.nsplit == 1) {
      const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
      for (int j = 0; j < 4; ++j) {
        uint32_t o[32];
        if (n > 0) {
          tc::ld_32x32b_x32(tmem + lane_base + kTmemO + 128 * chalf + 32 * j, o);
          tc::wait_ld();
        }
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint4 v;
          v.x = n > 0 ? pack_bf16(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv) : 0u;
          v.y = n > 0 ? pack_bf16(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv) : 0u;
          v.z = n > 0 ? pack_bf16(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv) : 0u;
          v.w = n > 0 ? pack_bf16(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv) : 0u;
          *reinterpret_cast<uint4*>(out_row + 32 * j + c) = v;
        }
      }
      if (write_lse)
        p.lse[r * p.lse_sr + row * p.lse_sh] = (lsum > 0.f) ? m_used * p.scale + logf(lsum) : -INFINITY;
    } else {
      // publish this split's partial: O half (fp32, [64 dim quads][128 heads][4]), m, l
      Unit uu;
      uu.b = u.b;
      uu.t = u.t;
      uu.half = u.half;
      const long long slot = slot_of(p, uu, u.split);
      float* po = p.partials + slot * kMlaPartialFloats + 4 * row;
      for (int j = 0; j < 4; ++j) {
        uint32_t o[32];
        if (n > 0) {
          tc::ld_32x32b_x32(tmem + lane_base + kTmemO + 128 * chalf + 32 * j, o);
          tc::wait_ld();
        }
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4*>(po + ((128 * chalf + 32 * j + c) / 4) * (4 * kMlaHeads)) =
              n > 0 ? make_float4(__uint_as_float(o[c]), __uint_as_float(o[c + 1]),
                                  __uint_as_float(o[c + 2]), __uint_as_float(o[c + 3]))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float* pml = p.partials + slot * kMlaPartialFloats + kMlaHeads * kMlaHalf;
      if (chalf == 0) {
        pml[row] = m_used;
        pml[kMlaHeads + row] = lsum;
      }
      __syncwarp();
      named_bar_sync(1, kSoftmaxThreads);
      int* cnt = p.counters + counter_index(p, uu);
      if (sidx == 0) *flag = atomic_add_acq_rel_gpu(cnt, 1);
      named_bar_sync(1, kSoftmaxThreads);
      if (*flag == u.nsplit - 1) {
        // last split of this (request, token, half): merge every split's
        // partial in split order (the same bits whichever split merges); this
        // split's own O is still in tensor memory
        const int ns = u.nsplit;
        float ms_[16], ls_[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          if (s < ns && s != u.split) {
            const float* ml =
                p.partials + slot_of(p, uu, s) * kMlaPartialFloats + kMlaHeads * kMlaHalf;
            ms_[s] = __ldcg(ml + row);
            ls_[s] = __ldcg(ml + kMlaHeads + row);
          } else {
            ms_[s] = m_used;
            ls_[s] = lsum;
          }
        }
        float M = -INFINITY;
#pragma unroll
        for (int s = 0; s < 16; ++s)
          if (s < ns) M = fmaxf(M, ms_[s]);
        float Ls = 0.f;
        float w[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          w[s] = 0.f;
          if (s < ns) {
            w[s] = (ms_[s] == -INFINITY) ? 0.f : ex2((ms_[s] - M) * c2);
            Ls = __fmaf_rn(w[s], ls_[s], Ls);
          }
        }
        const float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
        for (int j = 0; j < 128; j += 32) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
#pragma unroll 4
          for (int s = 0; s < ns; ++s) {
            float4 v[8];
            if (s == u.split) {
              uint32_t o[32];
              tc::ld_32x32b_x32(tmem + lane_base + kTmemO + 128 * chalf + j, o);
              tc::wait_ld();
#pragma unroll
              for (int k = 0; k < 8; ++k)
                v[k] = n > 0 ? make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                           __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
              const float* src = p.partials + slot_of(p, uu, s) * kMlaPartialFloats + 4 * row +
                                 ((128 * chalf + j) / 4) * (4 * kMlaHeads);
#pragma unroll
              for (int k = 0; k < 8; ++k) v[k] = ldcg_f4(src + k * (4 * kMlaHeads));
            }
            const float ws = w[s];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              acc[4 * k] = __fmaf_rn(ws, v[k].x, acc[4 * k]);
              acc[4 * k + 1] = __fmaf_rn(ws, v[k].y, acc[4 * k + 1]);
              acc[4 * k + 2] = __fmaf_rn(ws, v[k].z, acc[4 * k + 2]);
              acc[4 * k + 3] = __fmaf_rn(ws, v[k].w, acc[4 * k + 3]);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = pack_bf16(acc[8 * k] * inv, acc[8 * k + 1] * inv);
            v.y = pack_bf16(acc[8 * k + 2] * inv, acc[8 * k + 3] * inv);
            v.z = pack_bf16(acc[8 * k + 4] * inv, acc[8 * k + 5] * inv);
            v.w = pack_bf16(acc[8 * k + 6] * inv, acc[8 * k + 7] * inv);
            *reinterpret_cast<uint4*>(out_row + j + 8 * k) = v;
          }
        }
        if (write_lse)
          p.lse[r * p.lse_sr + row * p.lse_sh] = (Ls > 0.f) ? M * p.scale + logf(Ls) : -INFINITY;
        if (sidx == 0) store_relaxed_gpu(cnt, 0);
      }
    }
  }

  // Neither CTA leaves while the other may still use its shared memory or
  // barriers; then the pair frees its TMEM.  Every thread of both CTAs gets
  // here (all waits above are bounded).
  tc::fence_before_sync();
  __syncwarp();
  cluster_sync();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_mla_verify_pair(const MlaParams& p, const CUtensorMap& q_map,
                                   const CUtensorMap& kv_map, const CUtensorMap& v_map, int grid,
                                   cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_attr_once(mla_verify_pair_kernel, kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  e = launch_mla_plan(p, grid / 2, stream, true);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mla_verify_pair_kernel, p, q_map, kv_map, v_map);
}

}  // namespace pkv
