// kv_append.cu -- the paged-cache write that precedes a decode or verify call.
//
// "Atencion paginada" (transformers), decode path: the cache is updated in
// place through block_table; a sequence with n cached tokens puts its new token
// at logical position n, i.e. page block_table[b][n / P], slot n % P.  With the
// decode kernel's seq_lens (lengths including the current token) that position
// is seq_lens[b] - 1; an MLA verify row t sits at seq_lens[b] - qlen + t.
//
// One warp per written row: 512 bytes (GQA: 16 lanes of K, 16 of V, 16 bytes
// each) or 1152 bytes (MLA bf16) copied with 16-byte loads and stores; an e4m3
// MLA cache gets e4m3(x / k_scale), converted by `cvt.rn.satfinite`.  A page
// entry outside the table or the cache is never written: it raises a bit of
// the device error word instead.
#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 8;  // rows per 256-thread CTA

// Physical byte offset of position `pos` of request b, or -1 (and an error bit).
__device__ __forceinline__ long long row_offset(const AppendParams& p, int b, long long pos) {
  const long long pg = pos / p.page_size;
  if (pg >= p.max_blocks) {
    atomicOr(p.err, DEVERR_SEQ_TOO_LONG);
    return -1;
  }
  const int blk = __ldg(p.bt + (long long)b * p.bt_sb + pg);
  if (blk < 0 || blk >= p.num_blocks) {
    atomicOr(p.err, DEVERR_BAD_BLOCK);
    return -1;
  }
  return (long long)blk * p.c_sblk + (pos % p.page_size) * p.c_stok;
}

__global__ void __launch_bounds__(kWarps * 32) gqa_kv_append_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (w >= (long long)p.B * p.Hkv) return;
  const int b = (int)(w / p.Hkv), h = (int)(w % p.Hkv);
  const int L = __ldg(p.seq_lens + b);
  if (L <= 0) return;
  const long long off = row_offset(p, b, (long long)L - 1);
  if (off < 0) return;
  // lanes 0..15: K dims 8*lane .. +8; lanes 16..31: V dims 8*(lane-16) .. +8
  const uint16_t* src = (lane < 16 ? p.k : p.v) + b * p.s_sb + h * p.s_sh + 8 * (lane & 15);
  const uint4 x = *reinterpret_cast<const uint4*>(src);
  *reinterpret_cast<uint4*>(p.cache + off + h * p.c_sh + 16 * lane) = x;
}

// Two fp32 values to packed e4m3 (lo in the low byte), nearest even, saturating.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kWarps * 32) mla_kv_append_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (r >= (long long)p.B * p.qlen) return;
  const int b = (int)(r / p.qlen), t = (int)(r % p.qlen);
  const long long pos = (long long)__ldg(p.seq_lens + b) - p.qlen + t;
  if (pos < 0) return;
  const long long off = row_offset(p, b, pos);
  if (off < 0) return;
  const uint16_t* src = p.k + r * p.s_sb;
  if (!p.fp8) {
    for (int i = lane; i < kMlaLk / 8; i += 32)  // 72 units of 16 bytes
      *reinterpret_cast<uint4*>(p.cache + off + 16 * i) =
          *reinterpret_cast<const uint4*>(src + 8 * i);
    return;
  }
  const float ks = p.k_scale ? __ldg(p.k_scale) : 1.f;
  for (int i = lane; i < kMlaLk / 16; i += 32) {  // 36 units of 16 e4m3 bytes
    const uint4 a = *reinterpret_cast<const uint4*>(src + 16 * i);
    const uint4 c = *reinterpret_cast<const uint4*>(src + 16 * i + 8);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      // bf16 pairs (w[2k], w[2k+1]) hold elements 4k .. 4k+3, low half first
      const float x0 = __uint_as_float(w[2 * k] << 16), x1 = __uint_as_float(w[2 * k] & 0xFFFF0000u);
      const float x2 = __uint_as_float(w[2 * k + 1] << 16),
                  x3 = __uint_as_float(w[2 * k + 1] & 0xFFFF0000u);
      const uint16_t lo = e4m3x2(__fdiv_rn(x0, ks), __fdiv_rn(x1, ks));
      const uint16_t hi = e4m3x2(__fdiv_rn(x2, ks), __fdiv_rn(x3, ks));
      o[k] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint4*>(p.cache + off + 16 * i) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

// Failure-detection self-test: one CTA waits on an mbarrier that nothing ever
// arrives on, through the bounded wait every kernel of the library uses; the
// wait gives up after ~2^31 cycles, raises DEVERR_WAIT_TIMEOUT in `err` and the
// kernel returns (no fault, no hang).
__global__ void wait_selftest_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(b, 0, err);
  __syncthreads();
}

cudaError_t launch_wait_selftest(int* err, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_gqa_kv_append(const AppendParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.Hkv;
  const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
  gqa_kv_append_kernel<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_mla_kv_append(const AppendParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.qlen;
  const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
  mla_kv_append_kernel<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
