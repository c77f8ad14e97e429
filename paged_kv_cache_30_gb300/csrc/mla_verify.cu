// mla_verify.cu -- causal MLA verify over a paged latent cache, on tcgen05.
//
// Computes, for verify token t of request b (row r = b * qlen + t) and each
// of the 128 query heads h,
//   out[r, h, :] = sum_{j < lim} softmax_j(scale * q[r, h, :] . K_j) K_j[:512]
//   lse[r, h]    = log sum_{j < lim} exp(scale * q . K_j)   (-inf, out 0 if lim == 0)
// with lim = max(min(L - qlen + 1 + t, L_real), 0) and K_j the 576-wide latent
// row of key j gathered through block_table; V is the first 512 dims of K
// ("vllm.v1.attention.ops.triton_decode_attention", decode_attention_fwd_verify:
// parameters).  An FP8 e4m3 cache is dequantised by the scalar k_scale.
//
// One CTA per unit = (request, split, verify token, half of the 512 output
// dims).  A one-CTA planning kernel first writes each CTA's unit: largest
// splits first, a request's units side by side, the CTAs without a unit
// (the launch is sized for the largest split count) at the end, where they
// return at once.  Tensor memory (512 columns) holds the
// CTA's output half O[128 x 256] (fp32), two score buffers S[128 x 32] and
// query dims [0, 384) as bf16 pairs (the A operand of 24 of the 36 K16 steps
// of S: an MMA with A in TMEM reads only B from shared memory, and shared
// memory bandwidth is what bounds these N = 32 MMAs).
//   warp 0      TMA: query dims [384, 576) of the token once (48 KB), then
//               32-key tiles of the latent cache into a 4-stage ring (FP8:
//               e4m3 into a 2-stage ring, converted into a 3-stage bf16 ring
//               by warps 2, 3, 8..11).  The cache is read as a 4-D tensor
//               (64 dims, token, 9 chunks of 64 dims, page): one box of 8
//               tokens x 9 chunks (16 for e4m3) lands chunk-major, so a tile
//               is 4 groups of 8 keys, 9216 bytes apart, and chunk c of group
//               g is one 1024-byte 128-byte-swizzle atom at g * 9216 + c * 1024
//               -- both the K-major S operand and the MN-major V operand are
//               plain descriptors over it (stride 9216 between 8-key groups).
//   warp 1      TMEM allocation; MMA issue (one elected lane, warp-uniform
//               descriptors): S = Q K^T (M 128 heads, N 32 keys, K 576: 24
//               K16 steps with A from TMEM, 12 with A from shared memory) and
//               O += P V (M 128, N 256, K 32; P K-major with 64-byte swizzle,
//               V = the same smem tile read MN-major).
//   warps 4..7  softmax, one thread per
//               head: S from TMEM, mask j >= lim, exp2-domain online softmax
//               with a lazily updated max (O in TMEM is rescaled only when
//               the max grows by more than 2^8), P rounded to bf16 into
//               shared memory; epilogue.
// Warps 0..7 first share the load of query dims [0, 384) into TMEM (one
// round of 16-byte loads per thread; the producer's share comes after it has
// issued the ring's first fill).
// The two halves both compute S (576-wide Q K^T) and each does half of P V.
// Splits of a request publish fp32 (O half, m, l) partials; the last CTA of a
// (request, token, half) merges them with its own O, still in tensor memory,
// and resets its arrival counter.
#include "pkv_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"
#include "mla_common.cuh"

#include <cuda_fp16.h>

namespace pkv {
namespace {
using namespace mla;

constexpr int kSoftmaxWarp0 = 4;
constexpr int kChunks = kMlaLk / 64;            // 9 64-dim chunks of a latent row
constexpr int kQtChunks = 6;                    // query dims [0, 384) live in TMEM
constexpr int kQsChunks = kChunks - kQtChunks;  // dims [384, 576) in shared memory
constexpr int kQChunkBytes = kMlaHeads * 128;   // 16 KB: 128 rows x 64 dims
constexpr int kQsBytes = kQsChunks * kQChunkBytes;  // 49152
constexpr int kGroupBytes = kChunks * 1024;     // 9216: 8 keys x 576 dims, chunk-major
constexpr int kStageBytes = kMlaTile / 8 * kGroupBytes;  // 36864: one bf16 tile
constexpr int kF8StageBytes = kStageBytes / 2;      // 18432: one e4m3 tile
constexpr int kPBytes = kMlaHeads * kMlaTile * 2;   // 8192 (64-byte rows)

// Shared memory: [query dims 384..575 | bf16 tile stages | e4m3 tile stages
// (FP8 only) | P | barriers].  The bf16 path keeps 4 tiles in flight; the FP8
// path lands e4m3 tiles in a 2-stage ring and converts each into one of 3
// bf16 stages.
template <bool kFp8>
struct Cfg {
  static constexpr int kThreads = kFp8 ? 384 : 256;  // FP8: warps 2, 3, 8..11 convert
  static constexpr int kStages = kFp8 ? 3 : 4;        // bf16 tiles the MMAs read
  static constexpr int kF8Stages = kFp8 ? 2 : 0;      // e4m3 tiles TMA lands
  static constexpr int kF8Ring = kFp8 ? kF8Stages : 1;  // ring modulus (1 when unused)
  static constexpr int kOffStages = kQsBytes;
  static constexpr int kOffF8 = kOffStages + kStages * kStageBytes;
  static constexpr int kOffP = kOffF8 + kF8Stages * kF8StageBytes;
  static constexpr int kOffBars = kOffP + kPBytes;
  static constexpr int kSmemBytes = kOffBars + 256 + 1024;
  // At a unit's start the query dims [0, 384) land by TMA in a staging area
  // over bf16 stages 1..3 (bf16 cache: stage 0 takes the first tile at once)
  // or 0..2 (FP8: the e4m3 ring takes the first tiles; the converters wait).
  static constexpr int kOffStaging = kFp8 ? kOffStages : kOffStages + kStageBytes;
  static constexpr int kQtBytes = kQtChunks * kQChunkBytes;  // 98304
  static_assert(kOffStages % 1024 == 0 && kOffF8 % 1024 == 0 && kOffP % 1024 == 0,
                "swizzle atoms need 1024 B alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  static_assert(kOffStaging + kQtBytes <= (kFp8 ? kOffF8 : kOffP), "query staging area");
};

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;     // columns [0, 256): O half
constexpr uint32_t kTmemS = 256;   // columns [256, 320): two S buffers of 32
constexpr uint32_t kTmemQ = 320;   // columns [320, 512): query dims [0, 384), bf16 pairs
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // rescale O only when the max grows by > 2^8

// barrier indices
enum { kQFull = 0, kQtReady = 1, kKvFull = 2, kKvEmpty = 6, kSFull = 10, kSFree = 12, kPFull = 14,
       kPvDone = 15, kF8Full = 16, kF8Empty = 20, kNumBars = 24 };
constexpr int kMaxStages = 4;
constexpr int kConverters = 192;  // FP8: six converter warps

template <bool kFp8>
__global__ void __launch_bounds__(Cfg<kFp8>::kThreads, 1)
    mla_verify_kernel(const __grid_constant__ MlaParams p, const __grid_constant__ CUtensorMap q_map,
                      const __grid_constant__ CUtensorMap kv_map) {
  using C = Cfg<kFp8>;
  constexpr int kStages = C::kStages;
  // Programmatic dependent launch: nothing is read before the grids this
  // launch depends on have completed; the next grid may be scheduled as soon
  // as every CTA of this one has started (it waits for this grid the same way).
  griddep_wait();
  griddep_launch_dependents();
  const Unit u = decode_unit(p);
  if (u.split >= u.nsplit) return;  // no unit for this CTA

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sQ = base_u32, sK = base_u32 + C::kOffStages, sP = base_u32 + C::kOffP;
  const uint32_t sF8 = base_u32 + C::kOffF8;
  const uint32_t bars = base_u32 + C::kOffBars;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile uint32_t* tmem_slot =
      reinterpret_cast<volatile uint32_t*>(base + C::kOffBars + 8 * kNumBars);
  int* flag = reinterpret_cast<int*>(base + C::kOffBars + 8 * kNumBars + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  static_assert(C::kStages <= kMaxStages && C::kF8Stages <= kMaxStages, "barrier slots");
  if (tid == 0) {
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQtReady), 256);
    for (int s = 0; s < kMaxStages; ++s) {  // every barrier either path may touch
      mbar_init(bar(kKvFull + s), 1);
      mbar_init(bar(kKvEmpty + s), 1);
      mbar_init(bar(kF8Full + s), 1);
      mbar_init(bar(kF8Empty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kSFree + s), 128);
    }
    mbar_init(bar(kPFull), 1);
    mbar_init(bar(kPvDone), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  float scale_eff = p.scale, out_scale = 1.f;
  if (kFp8 && p.k_scale) {
    out_scale = __ldg(p.k_scale);  // V = raw e4m3 x k_scale
    scale_eff *= out_scale;
  }
  const float c2 = scale_eff * kLog2e;
  const int n = u.ntiles;

  // Query dims [0, 384) into TMEM (the A operand of the first 24 K16 steps of
  // S = Q K^T), shared by warps 0..7: warp w writes TMEM lanes (heads)
  // 32 (w % 4) .. + 31, 64-dim chunks 3 (w / 4) .. + 2, read from the staging
  // area the producer's TMA filled (row = head of each 16 KB chunk, 128-byte
  // swizzle: 16-byte unit k at k ^ (head % 8)); 256 arrivals on kQtReady, after
  // which the staging area may be refilled.  (Per-thread global loads at a
  // 1152-byte lane stride took ~8 us here.)
  auto load_qt_share = [&]() {
    const int head = 32 * (warp & 3) + lane, c0 = 3 * ((warp >> 2) & 1);
    mbar_wait(bar(kQFull), 0, p.err);
    const uint8_t* stg = base + C::kOffStaging + (head / 8) * 1024 + (head % 8) * 128;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      uint32_t v[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 w =
            *reinterpret_cast<const uint4*>(stg + (c0 + j) * kQChunkBytes + ((k ^ (head % 8)) * 16));
        v[4 * k] = w.x;
        v[4 * k + 1] = w.y;
        v[4 * k + 2] = w.z;
        v[4 * k + 3] = w.w;
      }
      tc::st_32x32b_x32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kTmemQ + 32 * (c0 + j), v);
    }
    fence_proxy_async_smem();  // the staging area is refilled by the async proxy
    tc::wait_st();
    tc::fence_before_sync();
    mbar_arrive(bar(kQtReady));
  };

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (n > 0) {
      const int qrow = u.b * p.qlen + u.t;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(kQFull), kQsBytes + C::kQtBytes);
        for (int c = 0; c < kQsChunks; ++c)
          tma_load_3d(sQ + c * kQChunkBytes, &q_map, bar(kQFull), 64 * (kQtChunks + c), 0, qrow);
        for (int c = 0; c < kQtChunks; ++c)
          tma_load_3d(base_u32 + C::kOffStaging + c * kQChunkBytes, &q_map, bar(kQFull), 64 * c, 0,
                      qrow);
      }
      const int32_t* bt_row = p.bt + (long long)u.b * p.bt_sb;
      // lane l holds the block id / page offset of 16-key piece l of the tiles
      // [gg, gg + 16); out-of-range pieces point past the cache (TMA fills zeros).
      // (An L2 prefetch of the tiles ahead, 18 more TMA operations per tile,
      // measured slower: the TMA unit's operation rate, not latency, limits.)
      auto piece = [&](int gg, int& blk, int& off) {
        const int piece_tok = (u.tile0 + gg) * kMlaTile + 16 * lane;
        blk = p.num_pages;
        off = 0;
        if (gg < n && piece_tok < u.L && lane < 2 * (n - gg)) {
          blk = __ldg(bt_row + piece_tok / p.page_size);
          off = piece_tok % p.page_size;
          if (blk < 0 || blk >= p.num_pages) atomicOr(p.err, DEVERR_BAD_BLOCK);
        }
      };
      for (int g = 0; g < n; g += 16) {
        int blk, off;
        piece(g, blk, off);
        for (int i = g; i < min(n, g + 16); ++i) {
          // bf16: stage 0 needs no wait; stages 1..3 held the staged query, so
          // the producer first moves its share and waits for everyone's.
          // FP8: the e4m3 ring is outside the staging area.
          if (kFp8 ? i == min(n, C::kF8Ring) : i == 1) {
            load_qt_share();
            if (!kFp8) mbar_wait(bar(kQtReady), 0, p.err);
          }
          const int b0 = __shfl_sync(0xffffffffu, blk, 2 * (i - g));
          const int o0 = __shfl_sync(0xffffffffu, off, 2 * (i - g));
          const int b1 = __shfl_sync(0xffffffffu, blk, 2 * (i - g) + 1);
          const int o1 = __shfl_sync(0xffffffffu, off, 2 * (i - g) + 1);
          if (lane == 0 && !kFp8) {
            const int st = i % kStages;
            mbar_wait(bar(kKvEmpty + st), ((i / kStages) & 1) ^ 1u, p.err);
            mbar_arrive_expect_tx(bar(kKvFull + st), kStageBytes);
            const uint32_t dst = sK + st * kStageBytes;
            // four boxes of 8 keys x 9 chunks: group g at g * 9216, chunk c of it
            // at + c * 1024 (one 128-byte-swizzle atom)
            tma_load_4d(dst, &kv_map, bar(kKvFull + st), 0, o0, 0, b0);
            tma_load_4d(dst + kGroupBytes, &kv_map, bar(kKvFull + st), 0, o0 + 8, 0, b0);
            tma_load_4d(dst + 2 * kGroupBytes, &kv_map, bar(kKvFull + st), 0, o1, 0, b1);
            tma_load_4d(dst + 3 * kGroupBytes, &kv_map, bar(kKvFull + st), 0, o1 + 8, 0, b1);
          } else if (lane == 0) {
            // e4m3 boxes of 16 keys x 64 dims, unswizzled: box (piece h, chunk c)
            // at (h * 9 + c) * 1 KB, 64-byte rows
            const int st = i % C::kF8Ring;
            mbar_wait(bar(kF8Empty + st), ((i / C::kF8Ring) & 1) ^ 1u, p.err);
            mbar_arrive_expect_tx(bar(kF8Full + st), kF8StageBytes);
            const uint32_t dst = sF8 + st * kF8StageBytes;
            // two boxes of 16 keys x 9 chunks: piece h at h * 9216, chunk c of it
            // at + c * 1024, 64-byte rows
            tma_load_4d(dst, &kv_map, bar(kF8Full + st), 0, o0, 0, b0);
            tma_load_4d(dst + kGroupBytes, &kv_map, bar(kF8Full + st), 0, o1, 0, b1);
          }
        }
      }
      if (n <= (kFp8 ? C::kF8Ring : 1)) load_qt_share();
    }
  } else if (warp == 1) {
    // ============================= MMA issuer =============================
    if (n > 0) {
      const uint32_t id_s = tc::idesc_bf16_f32(128, kMlaTile, false, false);
      const uint32_t id_pv = tc::idesc_bf16_f32(128, kMlaHalf, false, true);
      load_qt_share();
      mbar_wait(bar(kQFull), 0, p.err);
      mbar_wait(bar(kQtReady), 0, p.err);
      auto do_pv = [&](int j) {
        mbar_wait(bar(kPFull), j & 1, p.err);
        tc::fence_after_sync();
        const uint32_t v0 = sK + (j % kStages) * kStageBytes + (4 * u.half) * 1024;
#pragma unroll
        for (int ks = 0; ks < kMlaTile / 16; ++ks)
          tc::mma_bf16_elect(tmem + kTmemO, tc::smem_desc(sP + ks * 32, 16, 512, tc::kSwizzle64),
                             tc::smem_desc(v0 + ks * 2 * kGroupBytes, 1024, kGroupBytes,
                                           tc::kSwizzle128),
                             id_pv, j > 0 || ks > 0);
        tc::commit_elect(bar(kPvDone));
        tc::commit_elect(bar(kKvEmpty + j % kStages));
      };
      for (int i = 0; i < n; ++i) {
        const int st = i % kStages, sb = i & 1;
        mbar_wait(bar(kKvFull + st), (i / kStages) & 1, p.err);
        mbar_wait(bar(kSFree + sb), ((i >> 1) & 1) ^ 1u, p.err);
        tc::fence_after_sync();
        const uint32_t kst = sK + st * kStageBytes;
        const uint32_t d = tmem + kTmemS + sb * kMlaTile;
        // dims [0, 384): A = query from TMEM (8 columns per K16 step)
#pragma unroll 1
        for (int c = 0; c < kQtChunks; ++c) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16_ts_elect(
                d, tmem + kTmemQ + (4 * c + ks) * 8,
                tc::smem_desc(kst + c * 1024 + ks * 32, 16, kGroupBytes, tc::kSwizzle128), id_s,
                (c | ks) != 0);
        }
        // dims [384, 576): A = query from shared memory
#pragma unroll 1
        for (int c = kQtChunks; c < kChunks; ++c) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16_elect(
                d, tc::smem_desc(sQ + (c - kQtChunks) * kQChunkBytes + ks * 32, 16, 1024,
                                 tc::kSwizzle128),
                tc::smem_desc(kst + c * 1024 + ks * 32, 16, kGroupBytes, tc::kSwizzle128), id_s,
                true);
        }
        tc::commit_elect(bar(kSFull + sb));
        if (i > 0) do_pv(i - 1);
      }
      do_pv(n - 1);
    }
  } else if (!kFp8 && (warp == 2 || warp == 3)) {
    if (n > 0) load_qt_share();
  } else if (kFp8 && (warp == 2 || warp == 3 || warp >= 8)) {
    // ============ FP8: e4m3 tile -> bf16 tile in the MMA's swizzled layout ============
    // Exact: every e4m3 value is a bf16 value.  k_scale is applied to the scores
    // and to the output instead.
    const int ct = (warp < 8) ? tid - 64 : tid - 256 + 64;  // 0 .. 191
    if (warp < 8 && n > 0) load_qt_share();
    // the bf16 stages held the staged query
    if (n > 0) mbar_wait(bar(kQtReady), 0, p.err);
    for (int i = 0; i < n; ++i) {
      const int sf = i % C::kF8Ring, st = i % kStages;
      mbar_wait(bar(kF8Full + sf), (i / C::kF8Ring) & 1, p.err);
      // the bf16 stage is free once P V of its previous tile is done
      mbar_wait(bar(kKvEmpty + st), ((i / kStages) & 1) ^ 1u, p.err);
      const uint8_t* src = base + C::kOffF8 + sf * kF8StageBytes;
      uint8_t* dst = base + C::kOffStages + st * kStageBytes;
      // 1152 items: (piece h, chunk c, key row rr of 16, 16-byte e4m3 unit q of 4)
      for (int it = ct; it < 2 * kChunks * 16 * 4; it += kConverters) {
        const int q = it & 3, rr = (it >> 2) & 15, hc = it >> 6;  // hc = h * 9 + c
        const int h = hc / kChunks, c = hc % kChunks;
        const uint4 w =
            *reinterpret_cast<const uint4*>(src + h * kGroupBytes + c * 1024 + rr * 64 + q * 16);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const uint16_t pair = (uint16_t)(wv[k] >> (16 * hh));
            uint32_t f16x2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
            const __half2 hv = *reinterpret_cast<const __half2*>(&f16x2);
            const float2 fv = __half22float2(hv);
            o[2 * k + hh] = pack_bf16(fv.x, fv.y);
          }
        }
        const int row = 16 * h + rr;  // key row of the tile
        uint8_t* rowp = dst + (row / 8) * kGroupBytes + c * 1024 + (row % 8) * 128;
        // e4m3 unit q holds dims 16q .. 16q + 15 = bf16 units 2q, 2q + 1
        *reinterpret_cast<uint4*>(rowp + (((2 * q) ^ (row % 8)) * 16)) =
            make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(rowp + (((2 * q + 1) ^ (row % 8)) * 16)) =
            make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();  // the MMA reads the bf16 tile through the async proxy
      __syncwarp();
      named_bar_sync(2, kConverters);
      if (ct == 0) {
        mbar_arrive(bar(kF8Empty + sf));
        mbar_arrive(bar(kKvFull + st));
      }
    }
  } else if (warp >= kSoftmaxWarp0 && warp < 8) {
    // ================= softmax (one thread per head) + epilogue ============
    const int row = tid - kSoftmaxWarp0 * 32;           // head 0..127
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    float m_used = -INFINITY, l = 0.f;
    uint8_t* p_row = base + C::kOffP + (row / 8) * 512 + (row % 8) * 64;
    const int pswz = (row % 8) >> 1;
    if (n > 0) {
      load_qt_share();
    }
    for (int i = 0; i < n; ++i) {
      const int sb = i & 1;
      mbar_wait(bar(kSFull + sb), (i >> 1) & 1, p.err);
      __syncwarp();  // tcgen05.ld is warp-collective
      tc::fence_after_sync();
      uint32_t xr[32];
      tc::ld_32x32b_x32(tmem + lane_base + kTmemS + sb * kMlaTile, xr);
      tc::wait_ld();
      tc::fence_before_sync();
      mbar_arrive(bar(kSFree + sb));
      const int tok0 = (u.tile0 + i) * kMlaTile;
      const int nvalid = min(kMlaTile, u.lim - tok0);
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMlaTile; ++c)
        if (c < nvalid) mt = fmaxf(mt, __uint_as_float(xr[c]));
      // Lazy max: a row moves its reference max only when the tile's max
      // exceeds it by more than 2^8 (or on its first key).  The TMEM accesses
      // of the rescale are warp-collective, so the whole warp rescales when
      // any of its rows needs to; each row uses its own factor (1 if unchanged).
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
          for (int j = 0; j < kMlaHalf / 32; ++j) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kTmemO + 32 * j;
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
      for (int c = 0; c < kMlaTile; c += 2) {
        const float e0 = (c < nvalid) ? ex2(__fmaf_rn(__uint_as_float(xr[c]), c2, -msc)) : 0.f;
        const float e1 =
            (c + 1 < nvalid) ? ex2(__fmaf_rn(__uint_as_float(xr[c + 1]), c2, -msc)) : 0.f;
        lt += e0 + e1;
        pk[c / 2] = pack_bf16(e0, e1);
      }
      l += lt;
      // the P buffer (and, at the tail, the V rows) are free once P V of the
      // previous tile is done
      if (i > 0 && !waited) mbar_wait(bar(kPvDone), (i - 1) & 1, p.err);
#pragma unroll
      for (int uq = 0; uq < 4; ++uq)
        *reinterpret_cast<uint4*>(p_row + ((uq ^ pswz) & 3) * 16) =
            make_uint4(pk[4 * uq], pk[4 * uq + 1], pk[4 * uq + 2], pk[4 * uq + 3]);
      if (nvalid < kMlaTile) {
        // keys past the row limit: zero their V rows (this CTA's 256 dims) so
        // stale or poisoned cache contents never meet P = 0 in the MMA
        uint8_t* vst =
            base + C::kOffStages + (i % kStages) * kStageBytes + 4 * u.half * 1024;
        const int nz = kMlaTile - max(nvalid, 0);
        for (int q = row; q < nz * 4 * 8; q += 128) {
          const int rr = max(nvalid, 0) + q / 32, ch = (q / 8) % 4, un = q % 8;
          *reinterpret_cast<uint4*>(vst + (rr / 8) * kGroupBytes + ch * 1024 + (rr % 8) * 128 +
                                    un * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();  // P and zeroed V rows are read by the MMA (async proxy)
      tc::fence_before_sync();   // and any in-place O rescale precedes the next P V
      __syncwarp();
      named_bar_sync(1, 128);
      if (row == 0) mbar_arrive(bar(kPFull));
    }

    // ------------------------------ epilogue ------------------------------
    if (n > 0) {
      mbar_wait(bar(kPvDone), (n - 1) & 1, p.err);
      __syncwarp();  // the TMEM loads below are warp-collective
      tc::fence_after_sync();
    }
    const long long r = (long long)u.b * p.qlen + u.t;
    uint16_t* out_row = p.out + r * p.o_sr + row * p.o_sh + u.half * kMlaHalf;
    if (u.nsplit == 1) {
      const float inv = (l > 0.f) ? out_scale / l : 0.f;
      for (int j = 0; j < kMlaHalf / 32; ++j) {
        uint32_t o[32];
        if (n > 0) {
          tc::ld_32x32b_x32(tmem + lane_base + kTmemO + 32 * j, o);
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
      if (u.half == 0)
        p.lse[r * p.lse_sr + row * p.lse_sh] = (l > 0.f) ? m_used * scale_eff + logf(l) : -INFINITY;
    } else {
      // publish the split's partial: O half (fp32, as [64 dim quads][128 heads][4]:
      // a warp's float4 stores cover 512 contiguous bytes), m, l
      const long long slot = slot_of(p, u, u.split);
      float* po = p.partials + slot * kMlaPartialFloats + 4 * row;
      for (int j = 0; j < kMlaHalf / 32; ++j) {
        uint32_t o[32];
        if (n > 0) {
          tc::ld_32x32b_x32(tmem + lane_base + kTmemO + 32 * j, o);
          tc::wait_ld();
        }
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<float4*>(po + (8 * j + c / 4) * (4 * kMlaHeads)) =
              n > 0 ? make_float4(__uint_as_float(o[c]), __uint_as_float(o[c + 1]),
                                  __uint_as_float(o[c + 2]), __uint_as_float(o[c + 3]))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float* pml = p.partials + slot * kMlaPartialFloats + kMlaHeads * kMlaHalf;
      pml[row] = m_used;
      pml[kMlaHeads + row] = l;
      __syncwarp();
      named_bar_sync(1, 128);
      int* cnt = p.counters + counter_index(p, u);
      if (row == 0) *flag = atomic_add_acq_rel_gpu(cnt, 1);
      __syncwarp();
      named_bar_sync(1, 128);
      if (*flag == u.nsplit - 1) {
        // last split of this (request, token, half): merge every partial
        // (m, l) of every split first (independent loads), then O in 32-dim
        // chunks with the loads of several splits in flight
        const int ns = u.nsplit;
        float ms_[16], ls_[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          if (s < ns && s != u.split) {
            const float* ml =
                p.partials + slot_of(p, u, s) * kMlaPartialFloats + kMlaHeads * kMlaHalf;
            ms_[s] = __ldcg(ml + row);
            ls_[s] = __ldcg(ml + kMlaHeads + row);
          } else {  // this split's own (m, l); its O is still in tensor memory
            ms_[s] = m_used;
            ls_[s] = l;
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
        const float inv = (Ls > 0.f) ? out_scale / Ls : 0.f;
        for (int j = 0; j < kMlaHalf; j += 32) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
          // splits in index order, whichever of them merges (the result is the
          // same bits every call); this split's own O comes from tensor memory
#pragma unroll 4
          for (int s = 0; s < ns; ++s) {
            float4 v[8];
            if (s == u.split) {
              uint32_t o[32];
              tc::ld_32x32b_x32(tmem + lane_base + kTmemO + j, o);
              tc::wait_ld();
#pragma unroll
              for (int k = 0; k < 8; ++k)
                v[k] = n > 0 ? make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                           __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3]))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
              const float* src = p.partials + slot_of(p, u, s) * kMlaPartialFloats + 4 * row +
                                 (j / 4) * (4 * kMlaHeads);
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
        if (u.half == 0)
          p.lse[r * p.lse_sr + row * p.lse_sh] = (Ls > 0.f) ? M * scale_eff + logf(Ls) : -INFINITY;
        if (row == 0) store_relaxed_gpu(cnt, 0);
      }
    }
  }

  tc::fence_before_sync();
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ work plan --
// One CTA writes every verify CTA's unit (plan_entry: request, split and
// split count, verify token -- or token pair for CTA-pair launches -- and
// half) or -1.  The units (split < the request's split count) come in order
// of decreasing split size, i.e. tiles per split, ties by request index
// (beyond kPlanSortMax requests: request order), so the CTAs that start last
// are the short ones; a request's units are consecutive (split-major, then
// verify token, then half: the CTAs that read the same keys run side by
// side); -1 fills the rest of the launch.  A split holds at least
// kMlaMinTiles tiles, or kMlaMinTilesWide for CTA-pair launches whose batch
// still has a unit for every CTA pair at that size: each unit costs ~8 us
// beyond its tiles, so fewer, longer units win once the GPU is full.
constexpr int kPlanThreads = 1024;
constexpr int kPlanSortMax = 8192;

__global__ void __launch_bounds__(kPlanThreads, 1)
    mla_plan_kernel(const __grid_constant__ MlaParams p, int grid, int pair) {
  // Before the dependency wait only seq_lens is read (complete before the
  // kernel this launch depends on, like the block table); the plan, which the
  // previous call's verify kernel may still be reading, is written after it.
  griddep_launch_dependents();
  extern __shared__ unsigned long long keys[];  // [P2] (length, request) sort keys
  __shared__ int warp_sums[kPlanThreads / 32];
  __shared__ int s_total;
  const int B = p.B, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // one entry per CTA (row t = verify token), or per CTA pair (t = token pair)
  const int rows = pair ? p.qlen / 2 : p.qlen;
  const int per_split = rows * 2;
  // the minimum split: CTA pairs take the wider one when the batch still has
  // a unit for every CTA pair at that size
  int min_tiles = kMlaMinTiles;
  if (pair) {
    int mine = 0;
    for (int b = tid; b < B; b += kPlanThreads)
      mine += split_count(p, clamped_len(p, b), kMlaMinTilesWide);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
    if (lane == 0) warp_sums[wid] = mine;
    __syncthreads();
    if (wid == 0) {
      int v = warp_sums[lane];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) s_total = v;
    }
    __syncthreads();
    if ((long long)s_total * per_split >= p.pair_slots) min_tiles = kMlaMinTilesWide;
    __syncthreads();  // warp_sums and s_total are reused below
  }
  auto entry = [&](int b, int split, int ns, int t, int half) {
    return plan_entry(rows, b, t, half, split, ns);
  };
  if (B > kPlanSortMax) {  // request order, a fixed slot per (request, split)
    griddep_wait();
    for (int x = tid; x < grid; x += kPlanThreads) {
      const int per_b = p.cap * per_split;
      const int b = x / per_b, rem = x - b * per_b;
      const int split = rem / per_split, th = rem - split * per_split;
      const int ns = split_count(p, clamped_len(p, b), min_tiles);
      p.plan[x] = split < ns ? entry(b, split, ns, th >> 1, th & 1) : -1;
    }
    return;
  }
  int P2 = 1;
  while (P2 < B) P2 <<= 1;
  for (int i = tid; i < P2; i += kPlanThreads) {
    unsigned long long k = ~0ull;
    if (i < B)
      k = ((unsigned long long)(0x7fffffff - split_tiles(p, clamped_len(p, i), min_tiles)) << 32) |
          (unsigned)i;
    keys[i] = k;
  }
  __syncthreads();
  for (int k = 2; k <= P2; k <<= 1)  // bitonic sort, ascending
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P2; i += kPlanThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x0 = keys[i], x1 = keys[ixj];
          if ((x0 > x1) == ((i & k) == 0)) {
            keys[i] = x1;
            keys[ixj] = x0;
          }
        }
      }
      __syncthreads();
    }
  // ranks [r0, r0 + R) of this thread; exclusive scan of their unit counts
  const int R = (B + kPlanThreads - 1) / kPlanThreads;
  const int r0 = min(B, tid * R), r1 = min(B, r0 + R);
  int mine = 0;
  for (int r = r0; r < r1; ++r)
    mine += split_count(p, clamped_len(p, (int)(keys[r] & 0xffffffffu)), min_tiles) * per_split;
  int incl = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int v = warp_sums[lane];
    int wi = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += t;
    }
    warp_sums[lane] = wi - v;
    if (lane == 31) s_total = wi;
  }
  __syncthreads();
  int x = warp_sums[wid] + incl - mine;
  griddep_wait();
  for (int r = r0; r < r1; ++r) {
    const int b = (int)(keys[r] & 0xffffffffu);
    const int ns = split_count(p, clamped_len(p, b), min_tiles);
    for (int split = 0; split < ns; ++split)
      for (int th = 0; th < per_split; ++th) p.plan[x++] = entry(b, split, ns, th >> 1, th & 1);
  }
  for (int y = s_total + tid; y < grid; y += kPlanThreads) p.plan[y] = -1;
}

template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel* fn, int grid, int threads, int smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, args...);
}

template <bool kFp8>
cudaError_t launch_t(const MlaParams& p, const CUtensorMap& q_map, const CUtensorMap& kv_map,
                     int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_attr_once(mla_verify_kernel<kFp8>, Cfg<kFp8>::kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  e = launch_mla_plan(p, grid, stream, false);
  if (e != cudaSuccess) return e;
  return launch_pdl(mla_verify_kernel<kFp8>, grid, Cfg<kFp8>::kThreads, Cfg<kFp8>::kSmemBytes,
                    stream, p, q_map, kv_map);
}

}  // namespace

cudaError_t launch_mla_plan(const MlaParams& p, int grid, cudaStream_t stream, bool pair) {
  static std::atomic<uint64_t> plan_attr_done{0};
  cudaError_t e = set_smem_attr_once(mla_plan_kernel, kPlanSortMax * 8, plan_attr_done);
  if (e != cudaSuccess) return e;
  int p2 = 1;
  while (p2 < p.B) p2 <<= 1;
  return launch_pdl(mla_plan_kernel, 1, kPlanThreads, p.B > kPlanSortMax ? 0 : p2 * 8, stream, p,
                    grid, pair ? 1 : 0);
}

cudaError_t launch_mla_verify(const MlaParams& p, const CUtensorMap& q_map,
                              const CUtensorMap& kv_map, bool fp8, int grid,
                              cudaStream_t stream) {
  return fp8 ? launch_t<true>(p, q_map, kv_map, grid, stream)
             : launch_t<false>(p, q_map, kv_map, grid, stream);
}

}  // namespace pkv
