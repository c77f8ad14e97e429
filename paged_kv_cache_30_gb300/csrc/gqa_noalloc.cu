// gqa_noalloc.cu -- pkv_paged_decode_attn_noalloc: the GQA decode kernel run
// on scratch memory that the library never allocates.
//
// Some callers cannot let a library call cudaMalloc: an inference server that
// hands all of HBM to its own KV-cache pool up front and treats any other
// device allocation as an out-of-memory risk, or a host framework whose memory
// manager must own every device buffer.  pkv_paged_decode_attn allocates its
// workspace on first use; this entry point instead keeps the kernel's scratch
// (split partials, arrival counters, work-queue words) in one file-scope
// __device__ array of fixed size, which the CUDA module holds on every device
// that loads the library until the process exits.
#include "../../include/pkv.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "pkv_internal.h"

namespace {

// Limits of the static scratch.
constexpr int64_t kMaxPairs = 4096;  // (request, kv head) pairs per call
constexpr int64_t kMaxItems = 2048;  // split partials per call: B * Hkv * splits
constexpr int64_t kCounterInts = 64 + kMaxPairs + kMaxItems;  // queue/error words + counters
constexpr int64_t kItemBytes = int64_t(pkv::kGqaPartialFloats + pkv::kGqaMlFloats) * 4;
constexpr size_t kScratchBytes = size_t(kCounterInts * 4 + kMaxItems * kItemBytes);

// About 8.2 MiB: [queue words, error word | top counters | group counters |
// partial O | partial m, l].
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceScratch {
  bool ready = false;
  unsigned char* ptr = nullptr;  // device address of g_scratch on this device
  int num_sms = 0;
};
std::mutex g_mu;
DeviceScratch g_dev[64];

}  // namespace

namespace pkv {

// The device error word of the static scratch on `device`, or null when no
// call has set that device up yet (read by pkv_check_errors).
int* noalloc_error_word(int device) {
  if (device < 0 || device >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  return g_dev[device].ready ? reinterpret_cast<int*>(g_dev[device].ptr) + 32 : nullptr;
}

}  // namespace pkv

extern "C" PKV_API int pkv_paged_decode_attn_noalloc(
    const pkv_tensor* q, const pkv_tensor* kv_cache, const pkv_tensor* block_table,
    const pkv_tensor* seq_lens, const pkv_tensor* sinks, int window, float scale, int page_size,
    int num_kv_splits, const pkv_tensor* out, const pkv_tensor* lse, void* stream_ptr) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  pkv::GqaCall call;
  int rc = pkv::prepare_gqa_call(q, kv_cache, block_table, seq_lens, sinks, window, scale,
                                 page_size, num_kv_splits, out, lse, stream, &call);
  if (rc != PKV_OK || call.pairs == 0) return rc;

  // Set-up, once per device with that device current (prepare_gqa_call has
  // checked that q's device is current): the device address of the scratch
  // array (in host code its name is only a host-side stand-in) and the SM count.
  const int dev = call.device;
  DeviceScratch st;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev[dev].ready) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
      if (e != cudaSuccess) return pkv::abi_cuda_fail(e, "cudaGetSymbolAddress(scratch)");
      int sms = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return pkv::abi_cuda_fail(e, "cudaDeviceGetAttribute");
      g_dev[dev].ptr = static_cast<unsigned char*>(ptr);
      g_dev[dev].num_sms = sms;
      g_dev[dev].ready = true;
    }
    st = g_dev[dev];
  }
  // The same launch shape as pkv_paged_decode_attn, on the array's limits.
  pkv::GqaShape shape;
  if ((rc = pkv::gqa_launch_shape(call.pairs, call.cap_req, kMaxItems, kMaxPairs, st.num_sms,
                                  call.p.max_blocks, call.page_size, &shape)))
    return rc;

  pkv::GqaParams& p = call.p;
  int* words = reinterpret_cast<int*>(st.ptr);
  p.sched = words;                      // [0] queue head
  p.err = words + 32;                   // device error bits (pkv_check_errors reads them)
  p.counters = words + 64;              // [kMaxPairs]
  p.group_counters = words + 64 + kMaxPairs;  // [kMaxItems]
  p.part_o = reinterpret_cast<float*>(st.ptr + kCounterInts * 4);
  p.part_ml = p.part_o + kMaxItems * pkv::kGqaPartialFloats;
  p.max_items = kMaxItems;
  p.cap = shape.cluster > 1 ? shape.cluster : shape.cap;
  p.cluster = shape.cluster;
  p.min_pages = shape.min_pages;
  p.target_items = shape.target_items;

  // The array keeps the previous call's contents: the queue words, the error
  // word and every arrival counter must start this call at zero.
  cudaError_t e = cudaMemsetAsync(st.ptr, 0, size_t(kCounterInts) * 4, stream);
  if (e != cudaSuccess) return pkv::abi_cuda_fail(e, "clearing the scratch counters");
  e = pkv::launch_gqa_decode(p, call.map, call.page_size, shape.grid, stream);
  if (e != cudaSuccess) return pkv::abi_cuda_fail(e, "gqa decode launch (no-alloc)");
  return PKV_OK;
}
