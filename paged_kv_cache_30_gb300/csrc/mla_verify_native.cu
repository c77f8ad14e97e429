// mla_verify_native.cu -- MLA causal verify over an e4m3 latent cache with the
// query quantised to e4m3 too, so that S = Q K^T runs on kind::f8f6f4 MMAs.
//
// Same result definition as mla_verify.cu ("vllm.v1.attention.ops.
// triton_decode_attention", decode_attention_fwd_verify: parameters), with the
// query of (row r, head h) taken as code value x q_scale[r, h] (per-(row, head)
// e4m3 quantisation, mla_quantize_q below): the "native FP8 MLA MMA" step,
// which trades the bf16 query for half-size tensor operands.
//
// Kernel shape (one CTA per unit, the planning kernel of mla_verify.cu orders
// the units):
//   tensor memory: O half [0, 256) fp32, two score buffers [256, 320), the
//   whole e4m3 query (576 bytes = 144 columns per head) at [320, 464): every
//   one of the 18 K32 steps of S reads A from tensor memory.
//   warp 0      TMA: 32-key e4m3 tiles as four boxes of 8 keys x 9 chunks of
//               64 dims with 64-byte swizzle (group g at g * 4608, chunk c of
//               it at + c * 512) into a 4-stage ring; S reads them directly.
//   warp 1      MMA: S = Q8 K8^T (M 128 heads, N 32 keys, 18 x K32 e4m3 steps,
//               A from TMEM, B K-major 64-byte swizzle, SBO 4608); O_half +=
//               P V_half (bf16, as in mla_verify.cu).
//   warps 2, 3, 8..11  expand this CTA's V half (4 chunks) of each tile from
//               e4m3 to bf16 (exact) into a 3-stage ring, zeroing the rows of
//               keys past the row limit.
//   warps 4..7  softmax, one thread per head, scores scaled by the head's
//               q_scale x k_scale x scale; epilogue and split merge as in
//               mla_verify.cu.
#include "pkv_internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"
#include "mla_common.cuh"

#include <cuda_fp16.h>

namespace pkv {
namespace {
using namespace mla;

constexpr int kSoftmaxWarp0 = 4;
constexpr int kChunks = kMlaLk / 64;          // 9 chunks of 64 dims
constexpr int kF8Group = kChunks * 512;       // 4608: 8 keys x 576 e4m3, chunk-major
constexpr int kF8Tile = kMlaTile / 8 * kF8Group;   // 18432
constexpr int kVGroup = 4 * 1024;             // 4096: 8 keys x 256 bf16 (this CTA's V half)
constexpr int kVTile = kMlaTile / 8 * kVGroup;     // 16384
constexpr int kPBytes = kMlaHeads * kMlaTile * 2;  // 8192 (64-byte rows)
constexpr int kF8Stages = 4, kVStages = 3;
constexpr int kThreads = 384;
constexpr int kConverters = 192;
constexpr int kOffF8 = 0;
constexpr int kOffV = kOffF8 + kF8Stages * kF8Tile;  // 73728
constexpr int kOffP = kOffV + kVStages * kVTile;     // 122880
constexpr int kOffBars = kOffP + 2 * kPBytes;        // 139264: P of tile i in buffer i % 2
constexpr int kSmemBytes = kOffBars + 256 + 1024;
static_assert(kOffV % 1024 == 0 && kOffP % 1024 == 0, "swizzle atoms need 1024 B alignment");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;
constexpr uint32_t kTmemQ = 320;      // 144 columns: 576 e4m3 per head
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;

// barrier indices: a tile's e4m3 stage is free once S has read it (MMA commit)
// and the converters have expanded its V half (count 2)
enum { kQReady = 0, kF8Full = 1, kF8Empty = 5, kVFull = 9, kVEmpty = 12, kSFull = 15,
       kSFree = 17, kPFull = 19, kPFree = 21, kPvDone = 23, kNumBars = 24 };

__global__ void __launch_bounds__(kThreads, 1)
    mla_verify_native_kernel(const __grid_constant__ MlaParams p,
                             const __grid_constant__ CUtensorMap kv_map) {
  griddep_wait();
  griddep_launch_dependents();
  const Unit u = decode_unit(p);
  if (u.split >= u.nsplit) return;  // no unit for this CTA

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  const uint32_t sF8 = base_u32 + kOffF8, sV = base_u32 + kOffV, sP = base_u32 + kOffP;
  const uint32_t bars = base_u32 + kOffBars;
  auto bar = [&](int i) { return bars + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(base + kOffBars + 8 * kNumBars);
  int* flag = reinterpret_cast<int*>(base + kOffBars + 8 * kNumBars + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(bar(kQReady), 256);
    for (int s = 0; s < kF8Stages; ++s) {
      mbar_init(bar(kF8Full + s), 1);
      mbar_init(bar(kF8Empty + s), 2);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kSFree + s), 128);
      mbar_init(bar(kPFull + s), 1);
      mbar_init(bar(kPFree + s), 1);
    }
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
  const float k_scale = p.k_scale ? __ldg(p.k_scale) : 1.f;
  const int n = u.ntiles;
  const long long qrow = (long long)u.b * p.qlen + u.t;

  // The e4m3 query into TMEM, shared by warps 0..7: warp w writes lanes (heads)
  // 32 (w % 4) .. + 31; warps 0..3 bytes 0..255 of each head (columns 320..383),
  // warps 4..7 bytes 256..575 (columns 384..463), every store starting on a
  // 32-column boundary; 256 arrivals on kQReady.
  auto load_q8_share = [&]() {
    const int head = 32 * (warp & 3) + lane, half = (warp >> 2) & 1;
    const uint4* src = reinterpret_cast<const uint4*>(p.q8 + qrow * p.q8_sr + (long long)head * p.q8_sh +
                                                      256 * half);
    const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kTmemQ + 64 * half;
    uint4 w[20];
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = __ldg(src + k);
    if (half) {
#pragma unroll
      for (int k = 16; k < 20; ++k) w[k] = __ldg(src + k);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t v[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[4 * k] = w[8 * j + k].x;
        v[4 * k + 1] = w[8 * j + k].y;
        v[4 * k + 2] = w[8 * j + k].z;
        v[4 * k + 3] = w[8 * j + k].w;
      }
      tc::st_32x32b_x32(ta + 32 * j, v);
    }
    if (half) {
      uint32_t v16[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v16[4 * k] = w[16 + k].x;
        v16[4 * k + 1] = w[16 + k].y;
        v16[4 * k + 2] = w[16 + k].z;
        v16[4 * k + 3] = w[16 + k].w;
      }
      tc::st_32x32b_x16(ta + 64, v16);
    }
    tc::wait_st();
    tc::fence_before_sync();
    mbar_arrive(bar(kQReady));
  };

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (n > 0) {
      const int32_t* bt_row = p.bt + (long long)u.b * p.bt_sb;
      // lane l holds the block id / page offset of 16-key piece l of the tiles
      // [gg, gg + 16); out-of-range pieces point past the cache (TMA fills zeros)
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
      const int first_wait = min(n, kF8Stages);
      for (int g = 0; g < n; g += 16) {
        int blk, off;
        piece(g, blk, off);
        for (int i = g; i < min(n, g + 16); ++i) {
          const int b0 = __shfl_sync(0xffffffffu, blk, 2 * (i - g));
          const int o0 = __shfl_sync(0xffffffffu, off, 2 * (i - g));
          const int b1 = __shfl_sync(0xffffffffu, blk, 2 * (i - g) + 1);
          const int o1 = __shfl_sync(0xffffffffu, off, 2 * (i - g) + 1);
          if (i == first_wait) load_q8_share();  // the ring's first fill needs no wait
          if (lane == 0) {
            const int st = i % kF8Stages;
            mbar_wait(bar(kF8Empty + st), ((i / kF8Stages) & 1) ^ 1u, p.err);
            mbar_arrive_expect_tx(bar(kF8Full + st), kF8Tile);
            const uint32_t dst = sF8 + st * kF8Tile;
            tma_load_4d(dst, &kv_map, bar(kF8Full + st), 0, o0, 0, b0);
            tma_load_4d(dst + kF8Group, &kv_map, bar(kF8Full + st), 0, o0 + 8, 0, b0);
            tma_load_4d(dst + 2 * kF8Group, &kv_map, bar(kF8Full + st), 0, o1, 0, b1);
            tma_load_4d(dst + 3 * kF8Group, &kv_map, bar(kF8Full + st), 0, o1 + 8, 0, b1);
          }
        }
      }
      if (n <= first_wait) load_q8_share();
    }
  } else if (warp == 1) {
    // ============================= MMA issuer =============================
    if (n > 0) {
      const uint32_t id_s = tc::idesc_e4m3_f32(128, kMlaTile);
      const uint32_t id_pv = tc::idesc_bf16_f32(128, kMlaHalf, false, true);
      load_q8_share();
      mbar_wait(bar(kQReady), 0, p.err);
      auto do_pv = [&](int j) {
        const int sv = j % kVStages, pb = j & 1;
        mbar_wait(bar(kVFull + sv), (j / kVStages) & 1, p.err);
        mbar_wait(bar(kPFull + pb), (j >> 1) & 1, p.err);
        tc::fence_after_sync();
        const uint32_t v0 = sV + sv * kVTile;
#pragma unroll
        for (int ks = 0; ks < kMlaTile / 16; ++ks)
          tc::mma_bf16_elect(tmem + kTmemO,
                             tc::smem_desc(sP + pb * kPBytes + ks * 32, 16, 512, tc::kSwizzle64),
                             tc::smem_desc(v0 + ks * 2 * kVGroup, 1024, kVGroup, tc::kSwizzle128),
                             id_pv, j > 0 || ks > 0);
        tc::commit_elect(bar(kPvDone));
        tc::commit_elect(bar(kPFree + pb));
        tc::commit_elect(bar(kVEmpty + sv));
      };
      for (int i = 0; i < n; ++i) {
        const int st = i % kF8Stages, sb = i & 1;
        mbar_wait(bar(kF8Full + st), (i / kF8Stages) & 1, p.err);
        mbar_wait(bar(kSFree + sb), ((i >> 1) & 1) ^ 1u, p.err);
        tc::fence_after_sync();
        const uint32_t kst = sF8 + st * kF8Tile;
        const uint32_t d = tmem + kTmemS + sb * kMlaTile;
        // 18 K32 steps: chunk c = s / 2, half-row (32 bytes) s % 2
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
            tc::mma_e4m3_ts_elect(d, tmem + kTmemQ + (2 * c + h2) * 8,
                                  tc::smem_desc(kst + c * 512 + h2 * 32, 16, kF8Group, tc::kSwizzle64),
                                  id_s, (c | h2) != 0);
        }
        tc::commit_elect(bar(kSFull + sb));
        tc::commit_elect(bar(kF8Empty + st));  // S is done with the e4m3 tile
        if (i > 0) do_pv(i - 1);
      }
      do_pv(n - 1);
    }
  } else if (warp == 2 || warp == 3 || warp >= 8) {
    // ===== V half of each tile: e4m3 -> bf16 (exact), keys past the limit zeroed =====
    const int ct = (warp < 8) ? tid - 64 : tid - 256 + 64;  // 0 .. 191
    if (warp < 8 && n > 0) load_q8_share();
    for (int i = 0; i < n; ++i) {
      const int sf = i % kF8Stages, sv = i % kVStages;
      mbar_wait(bar(kF8Full + sf), (i / kF8Stages) & 1, p.err);
      mbar_wait(bar(kVEmpty + sv), ((i / kVStages) & 1) ^ 1u, p.err);
      const uint8_t* src = base + kOffF8 + sf * kF8Tile;
      uint8_t* dst = base + kOffV + sv * kVTile;
      const int nvalid = min(kMlaTile, u.lim - (u.tile0 + i) * kMlaTile);
      // 512 items: (key row r of 32, chunk c of this half, 16-byte e4m3 unit q of 4)
      for (int it = ct; it < kMlaTile * 4 * 4; it += kConverters) {
        const int q = it & 3, c = (it >> 2) & 3, r = it >> 4;
        uint32_t o[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (r < nvalid) {
          const int cc = 4 * u.half + c;
          const uint4 w = *reinterpret_cast<const uint4*>(
              src + (r / 8) * kF8Group + cc * 512 + (r % 8) * 64 + (((q ^ ((r % 8) >> 1)) & 3) * 16));
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
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
        }
        uint8_t* rowp = dst + (r / 8) * kVGroup + c * 1024 + (r % 8) * 128;
        // e4m3 unit q holds dims 16q .. 16q + 15 = bf16 units 2q, 2q + 1
        *reinterpret_cast<uint4*>(rowp + (((2 * q) ^ (r % 8)) * 16)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(rowp + (((2 * q + 1) ^ (r % 8)) * 16)) =
            make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();  // the MMA reads the bf16 V half through the async proxy
      __syncwarp();
      named_bar_sync(2, kConverters);
      if (ct == 0) {
        mbar_arrive(bar(kF8Empty + sf));
        mbar_arrive(bar(kVFull + sv));
      }
    }
  } else if (warp >= kSoftmaxWarp0 && warp < 8) {
    // ================= softmax (one thread per head) + epilogue ============
    const int row = tid - kSoftmaxWarp0 * 32;  // head 0..127
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    // scores of this head: S x q_scale x k_scale x scale
    const float s_eff = __ldg(p.q_scale + qrow * p.qs_sr + (long long)row * p.qs_sh) * k_scale * p.scale;
    const float c2 = s_eff * kLog2e;
    float m_used = -INFINITY, l = 0.f;
    // P row of this head in buffer b (64-byte swizzle)
    auto p_row = [&](int b) { return base + kOffP + b * kPBytes + (row / 8) * 512 + (row % 8) * 64; };
    const int pswz = (row % 8) >> 1;
    if (n > 0) load_q8_share();
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
      // P buffer i % 2 is free once P V of tile i - 2 is done.  Waiting here,
      // before any kPvDone wait, also keeps kPvDone within one phase of the
      // P V this thread waits for (parity waits cannot alias).
      const int pb = i & 1;
      mbar_wait(bar(kPFree + pb), ((i >> 1) & 1) ^ 1u, p.err);
      const int nvalid = min(kMlaTile, u.lim - (u.tile0 + i) * kMlaTile);
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMlaTile; ++c)
        if (c < nvalid) mt = fmaxf(mt, __uint_as_float(xr[c]));
      // lazy max, as in mla_verify.cu (the warp rescales its O rows together)
      const bool need =
          mt > -INFINITY && (m_used == -INFINITY || (mt - m_used) * c2 > kRescaleLog2);
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_used;
        const float alpha =
            (m_used == -INFINITY) ? 0.f : (need ? ex2((m_used - m_new) * c2) : 1.f);
        if (i > 0) {
          mbar_wait(bar(kPvDone), (i - 1) & 1, p.err);
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
      // Last tile: P V of tile n - 2 must be done before P n - 1 is published.
      // kPvDone is then one phase short of the end when the epilogue waits for
      // the last phase; were both last P V done by then, a wait for the parity
      // of phase n - 2 would alias the never-completing phase n.
      if (i == n - 1 && i > 0) mbar_wait(bar(kPvDone), (i - 1) & 1, p.err);
#pragma unroll
      for (int uq = 0; uq < 4; ++uq)
        *reinterpret_cast<uint4*>(p_row(pb) + ((uq ^ pswz) & 3) * 16) =
            make_uint4(pk[4 * uq], pk[4 * uq + 1], pk[4 * uq + 2], pk[4 * uq + 3]);
      fence_proxy_async_smem();  // P is read by the MMA (async proxy)
      tc::fence_before_sync();   // and any in-place O rescale precedes the next P V
      __syncwarp();
      named_bar_sync(1, 128);
      if (row == 0) mbar_arrive(bar(kPFull + pb));
    }

    // ------------------------------ epilogue ------------------------------
    if (n > 0) {
      // P V of tile n - 2 is done (waited for above): kPvDone is at most one
      // phase short of the end
      mbar_wait(bar(kPvDone), (n - 1) & 1, p.err);
      __syncwarp();
      tc::fence_after_sync();
    }
    const long long r = qrow;
    uint16_t* out_row = p.out + r * p.o_sr + row * p.o_sh + u.half * kMlaHalf;
    if (u.nsplit == 1) {
      const float inv = (l > 0.f) ? k_scale / l : 0.f;
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
        p.lse[r * p.lse_sr + row * p.lse_sh] = (l > 0.f) ? m_used * s_eff + logf(l) : -INFINITY;
    } else {
      // publish the split's partial: O half as [64 dim quads][128 heads][4], m, l
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
        // last split: merge every split in index order (the same bits whichever
        // split is last), this split's own O read from tensor memory
        const int ns = u.nsplit;
        float ms_[16], ls_[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
          if (s < ns && s != u.split) {
            const float* ml =
                p.partials + slot_of(p, u, s) * kMlaPartialFloats + kMlaHeads * kMlaHalf;
            ms_[s] = __ldcg(ml + row);
            ls_[s] = __ldcg(ml + kMlaHeads + row);
          } else {
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
        const float inv = (Ls > 0.f) ? k_scale / Ls : 0.f;
        for (int j = 0; j < kMlaHalf; j += 32) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
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
          p.lse[r * p.lse_sr + row * p.lse_sh] = (Ls > 0.f) ? M * s_eff + logf(Ls) : -INFINITY;
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

// ------------------------------------------------------ query quantisation --
// One warp per (row, head): 576 bf16 = 72 16-byte units (lanes take units
// lane, lane + 32, lane + 64 < 72); absmax by warp reduction; scale =
// absmax / 448 (1 for an all-zero row); code = e4m3(q / scale), quotient
// rounded to nearest even in fp32, conversion to nearest even, saturating.
__global__ void __launch_bounds__(256)
    mla_quantize_q_kernel(const __grid_constant__ QuantParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const long long pair = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (pair >= (long long)p.R * p.H) return;
  const int lane = threadIdx.x & 31;
  const long long r = pair / p.H;
  const int h = (int)(pair % p.H);
  const uint4* src = reinterpret_cast<const uint4*>(p.q + r * p.q_sr + (long long)h * p.q_sh);
  uint4 w[3];
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int unit = lane + 32 * k;
    w[k] = unit < 72 ? __ldg(src + unit) : make_uint4(0, 0, 0, 0);
    const uint32_t wv[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      amax = fmaxf(amax, fabsf(__uint_as_float(wv[e] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(wv[e] & 0xffff0000u)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  if (lane == 0) p.q_scale[r * p.qs_sr + h] = sc;
  uint8_t* dst = p.q8 + r * p.q8_sr + (long long)h * kMlaLk;
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int unit = lane + 32 * k;
    if (unit >= 72) continue;
    const uint32_t wv[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
    uint32_t packed[2];
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      // four elements: (lo, hi) of word e and of word e + 1
      const float x0 = __fdiv_rn(__uint_as_float(wv[e] << 16), sc);
      const float x1 = __fdiv_rn(__uint_as_float(wv[e] & 0xffff0000u), sc);
      const float x2 = __fdiv_rn(__uint_as_float(wv[e + 1] << 16), sc);
      const float x3 = __fdiv_rn(__uint_as_float(wv[e + 1] & 0xffff0000u), sc);
      uint16_t lo, hi;
      // cvt.rn.satfinite.e4m3x2.f32 d, a, b: a lands in the upper byte
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
      packed[e / 2] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint2*>(dst + 8 * unit) = make_uint2(packed[0], packed[1]);
  }
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

}  // namespace

cudaError_t launch_mla_verify_native(const MlaParams& p, const CUtensorMap& kv_map, int grid,
                                     cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = set_smem_attr_once(mla_verify_native_kernel, kSmemBytes, attr_done);
  if (e != cudaSuccess) return e;
  e = launch_mla_plan(p, grid, stream, false);
  if (e != cudaSuccess) return e;
  return launch_pdl(mla_verify_native_kernel, grid, kThreads, kSmemBytes, stream, p, kv_map);
}

cudaError_t launch_mla_quantize_q(const QuantParams& p, cudaStream_t stream) {
  const long long pairs = (long long)p.R * p.H;
  if (pairs == 0) return cudaSuccess;
  return launch_pdl(mla_quantize_q_kernel, (int)((pairs + 7) / 8), 256, 0, stream, p);
}

}  // namespace pkv
