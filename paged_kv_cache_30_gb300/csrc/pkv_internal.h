// pkv_internal.h -- declarations shared by the host launcher (api.cpp) and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cuda.h>

#include <atomic>
#include <cuda_runtime.h>
#include <stdint.h>

struct pkv_tensor;  // include/pkv.h

namespace pkv {

// Device-side error bits, OR-ed into the workspace error word and read back by
// pkv_check_errors().
enum : int {
  DEVERR_BAD_BLOCK = 1,      // a block-table entry outside [0, num_blocks)
  DEVERR_SEQ_TOO_LONG = 2,   // seq_len needs more pages than the block table holds
  DEVERR_WAIT_TIMEOUT = 4,   // a pipeline wait gave up (the kernel drained and returned)
  DEVERR_ITEM_OVERFLOW = 8,  // more work items than the workspace holds
  DEVERR_QUEUE = 16,         // a CTA drew more items than the launch has (it stopped)
};

// Per-device workspace carved out of one allocation (see api.cpp).
struct Workspace {
  void* base = nullptr;
  size_t bytes = 0;
  float* partials = nullptr;  // split partials, reused by both paths
  size_t partial_bytes = 0;
  int* counters = nullptr;    // self-resetting arrival counters
  int64_t num_counters = 0;
  int* sched = nullptr;       // [0] work-queue head (self-resetting)
  int* err = nullptr;         // device error word
  int num_sms = 0;
};

// ---------------------------------------------------------------- GQA --
constexpr int kGqaHeadDim = 128;
constexpr int kGqaGroup = 8;         // query heads per kv head
constexpr int kGqaMaxBatch = 2048;   // requests per call (device-side scheduler table)
constexpr int kGqaPartialFloats = kGqaGroup * kGqaHeadDim;  // O partial of one work item
constexpr int kGqaMlFloats = 2 * kGqaGroup;                 // m[8], l[8] of one work item

struct GqaParams {
  const uint16_t* q;  // bf16 [B, Hq, 128]
  int64_t q_sb, q_sh;
  const int32_t* bt;
  int64_t bt_sb;
  int max_blocks;
  int num_blocks;
  const int32_t* seq_lens;
  const float* sinks;  // [Hq] or null
  uint16_t* out;       // bf16 [B, Hq, 128]
  int64_t o_sb, o_sh;
  float* lse;          // [B, Hq] or null
  int64_t lse_sb, lse_sh;
  int B, Hkv;
  int window;          // <= 0: all keys
  float scale_log2;    // scale * log2(e)
  float scale;
  int cap;             // max splits per (request, kv head)
  int min_pages;       // fewest pages a split may hold
  int target_items;    // desired number of work items per launch
  float* part_o;       // [max_items][8][128]
  float* part_ml;      // [max_items][16]
  int64_t max_items;
  int* counters;       // [B * Hkv] arrival counters of the last merge level
  int* group_counters; // [max_items] arrival counters of split groups (by first item)
  int* sched;
  int* err;
  int cluster;         // > 1: cluster mode with this many splits per cluster (see below)
};

// Launch the GQA decode kernel for page size 16 or 32.  p.cluster <= 1: the
// persistent kernel on `grid` CTAs.  p.cluster = C in [2, 8]: the cluster
// mode, grid (C, B * Hkv) in clusters of C CTAs, CTA r of a cluster taking
// split r of one (request, kv head); the splits merge through distributed
// shared memory (no workspace partials, counters or queue).
cudaError_t launch_gqa_decode(const GqaParams& p, const CUtensorMap& kv_map, int page_size,
                              int grid, cudaStream_t stream);
constexpr int kGqaMaxCluster = 8;
int gqa_ctas_per_sm();

// A validated GQA decode call: kernel parameters (without workspace pointers)
// and the KV-cache tensor map.
struct GqaCall {
  GqaParams p;
  CUtensorMap map;  // CUtensorMap carries its own 64-byte alignment
  int64_t pairs;   // B * Hkv
  int cap_req;     // num_kv_splits as given (0 = library's choice)
  int page_size;
  int device;      // the device holding q (current, and the stream's device)
};

// Defined in api.cpp, for entry points implemented in other files.
// Validates every argument (shapes, dtypes, strides, alignment, overlap of
// outputs with inputs, the device of q against the current device and the
// stream's) and fills `call`; B == 0 returns PKV_OK with call->pairs == 0
// before any CUDA call.
int prepare_gqa_call(const ::pkv_tensor* q, const ::pkv_tensor* kv_cache,
                     const ::pkv_tensor* block_table, const ::pkv_tensor* seq_lens,
                     const ::pkv_tensor* sinks, int window, float scale, int page_size,
                     int num_kv_splits, const ::pkv_tensor* out, const ::pkv_tensor* lse,
                     cudaStream_t stream, GqaCall* call);

// Launch shape of a GQA decode call on scratch that holds max_items split
// partials and max_pairs (request, kv head) counters: the split cap (0 = the
// most that fit, at most 256), the grid (CTAs per SM x SMs, or fewer for
// small calls) and the kernel's target item count.  PKV_ERR_WORKSPACE when
// the call does not fit.  Every entry point launching the GQA kernel uses it.
struct GqaShape {
  int cap, grid, target_items;
  int cluster;    // > 1: cluster mode with this many splits per (request, kv head) at most
  int min_pages;  // fewest pages a split may hold
};
int gqa_launch_shape(int64_t pairs, int cap_req, int64_t max_items, int64_t max_pairs,
                     int num_sms, int max_blocks, int page_size, GqaShape* shape);
// Device address of the error word of pkv_paged_decode_attn_noalloc's static
// scratch on `device`, or null before that device's first such call.
int* noalloc_error_word(int device);
int abi_fail(int code, const char* message);
int abi_cuda_fail(cudaError_t e, const char* what);

// ---------------------------------------------------------------- MLA --
constexpr int kMlaHeads = 128;
constexpr int kMlaLk = 576;
constexpr int kMlaLv = 512;
constexpr int kMlaHalf = kMlaLv / 2;        // output dims per CTA
constexpr int kMlaTile = 32;                // keys per pipeline tile
constexpr int kMlaMinTiles = 128;           // a split holds at least 4096 keys
// CTA-pair launches split more coarsely (6144 keys) when the batch still has
// a unit for every CTA pair at that size: each unit costs ~8 us of start,
// query load and merge on top of its tiles, and on B = 32 qlen 4 batches
// (lengths U[512, 8192], four seeds, same process) 128 -> 192 measured
// 223.2 / 221.2 / 221.2 / 202.8 -> 200.7 / 210.9 / 200.7 / 184.3 us.
constexpr int kMlaMinTilesWide = 192;
constexpr int64_t kMlaPartialFloats = int64_t(kMlaHeads) * kMlaHalf + 2 * kMlaHeads;

struct MlaParams {
  const uint16_t* q;             // bf16 [B*qlen, 128, 576]
  int64_t q_sr, q_sh;
  const uint8_t* kv;             // latent cache base
  int64_t kv_stok, kv_spage;     // token / page strides in bytes
  const int32_t* bt;
  int64_t bt_sb;
  int max_blocks;
  int num_pages;
  const int32_t* seq_lens;
  const int32_t* real_seq_lens;  // or null
  const float* k_scale;          // device scalar or null (FP8 only)
  uint16_t* out;                 // bf16 [B*qlen, 128, 512]
  int64_t o_sr, o_sh;
  float* lse;                    // [B*qlen, 128]
  int64_t lse_sr, lse_sh;
  int B, qlen, cap, page_size;
  float scale;
  int pair_slots;                // CTA pairs that run at once (SMs / 2)
  float* partials;               // [slots][128*256 + 256]
  int64_t max_slots;
  int* counters;                 // [(b*qlen + t)*2 + half]
  int* plan;                     // [grid] unit of each CTA (written by the planning kernel)
  int* err;
  // native FP8 (e4m3 query): codes [B*qlen, 128, 576] and fp32 scales [B*qlen, 128]
  const uint8_t* q8;
  int64_t q8_sr, q8_sh;
  const float* q_scale;
  int64_t qs_sr, qs_sh;
};

// The planning kernel: writes p.plan[0, grid) (one CTA; programmatic dependent
// launch): one entry per verify CTA, or with `pair` one per CTA pair (a pair
// takes two consecutive verify tokens).
cudaError_t launch_mla_plan(const MlaParams& p, int grid, cudaStream_t stream, bool pair);
// bf16 latent cache, even qlen: the planning kernel, then the verify kernel on
// CTA pairs (grid CTAs, clusters of 2; v_map: the cache as (64 dims, token,
// 9 chunks, page) with a box of (64, 16, 2, 1), 128-byte swizzle).
cudaError_t launch_mla_verify_pair(const MlaParams& p, const CUtensorMap& q_map,
                                   const CUtensorMap& kv_map, const CUtensorMap& v_map, int grid,
                                   cudaStream_t stream);
cudaError_t launch_mla_verify(const MlaParams& p, const CUtensorMap& q_map,
                              const CUtensorMap& kv_map, bool fp8, int grid, cudaStream_t stream);
// Native FP8: planning kernel, then the verify kernel with S = Q8 K8^T on
// kind::f8f6f4 (kv_map: the e4m3 cache as (64 dims, token, 9 chunks, page) with
// a box of (64, 8, 9, 1) and 64-byte swizzle).
cudaError_t launch_mla_verify_native(const MlaParams& p, const CUtensorMap& kv_map, int grid,
                                     cudaStream_t stream);

// Per-(row, head) e4m3 quantisation of an MLA query: scale = absmax / 448,
// code = e4m3(q / scale) (round to nearest even, saturating).
struct QuantParams {
  const uint16_t* q;      // bf16 [R, H, 576]
  int64_t q_sr, q_sh;     // element strides
  uint8_t* q8;            // [R, H, 576], row stride q8_sr, head stride 576
  int64_t q8_sr;
  float* q_scale;         // [R, H], row stride qs_sr, head stride 1
  int64_t qs_sr;
  int R, H;
};
cudaError_t launch_mla_quantize_q(const QuantParams& p, cudaStream_t stream);

// ---------------------------------------------------------- KV append --
struct AppendParams {
  const uint16_t* k;     // GQA: k [B, Hkv, 128]; MLA: latent [B*qlen, 576]
  const uint16_t* v;     // GQA: v [B, Hkv, 128]; MLA: unused
  int64_t s_sb, s_sh;    // source strides (elements): GQA [b, h]; MLA [row, -]
  uint8_t* cache;        // cache base
  int64_t c_sblk, c_sh, c_stok;  // bytes: block/page, kv head (GQA), token
  int num_blocks;
  const int32_t* bt;
  int64_t bt_sb;
  int max_blocks;
  const int32_t* seq_lens;
  int B, Hkv, qlen, page_size;
  int fp8;               // MLA: e4m3 cache
  const float* k_scale;  // MLA FP8: device scalar or null
  int* err;
};
cudaError_t launch_gqa_kv_append(const AppendParams& p, cudaStream_t stream);
// one CTA whose bounded mbarrier wait runs out and raises DEVERR_WAIT_TIMEOUT in err
cudaError_t launch_wait_selftest(int* err, cudaStream_t stream);
cudaError_t launch_mla_kv_append(const AppendParams& p, cudaStream_t stream);

// Large dynamic shared memory is an attribute of a kernel on the current
// device: set it the first time a kernel launches on each device.
template <typename Kernel>
inline cudaError_t set_smem_attr_once(Kernel* fn, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// The counter region of the workspace holds 2^20 ints: the first half for
// (request, kv head) counters, the second half for split-group counters.
constexpr int64_t kTopCounters = int64_t(1) << 19;

}  // namespace pkv
