// api.cpp -- the C ABI of libpkv (see include/pkv.h): argument validation,
// per-device workspace, tensor-map encoding, the static split-cap heuristic
// and kernel launches.  No allocation happens after a device's workspace
// exists, so every launch can be captured in a CUDA graph.
#include "../../include/pkv.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <initializer_list>
#include <string>
#include <utility>

#include "pkv_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
constexpr size_t kDefaultWorkspace = size_t(1) << 30;
constexpr int64_t kNumCounters = int64_t(1) << 20;

struct DeviceState {
  pkv::Workspace ws;
  cudaEvent_t order_event = nullptr;
  cudaStream_t last_stream = nullptr;
  bool has_last = false;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// ------------------------------------------------------------ workspace --
int init_locked(int device, size_t partial_bytes) {
  DeviceState& st = g_dev[device];
  if (st.ws.base) return PKV_OK;
  if (partial_bytes == 0) partial_bytes = kDefaultWorkspace;
  partial_bytes = (partial_bytes + 255) / 256 * 256;
  const size_t head = 512 + size_t(kNumCounters) * 4;  // err + sched, counters
  const size_t total = head + partial_bytes;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  void* base = nullptr;
  e = cudaMalloc(&base, total);
  if (e != cudaSuccess) {
    cudaSetDevice(prev);
    return cuda_fail(e, "workspace cudaMalloc");
  }
  e = cudaMemset(base, 0, head);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st.order_event, cudaEventDisableTiming);
  int sms = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(base);
    cudaSetDevice(prev);
    return cuda_fail(e, "workspace init");
  }
  uint8_t* b = static_cast<uint8_t*>(base);
  st.ws.base = base;
  st.ws.bytes = total;
  st.ws.err = reinterpret_cast<int*>(b);
  st.ws.sched = reinterpret_cast<int*>(b + 256);
  st.ws.counters = reinterpret_cast<int*>(b + 512);
  st.ws.num_counters = kNumCounters;
  st.ws.partials = reinterpret_cast<float*>(b + head);
  st.ws.partial_bytes = partial_bytes;
  st.ws.num_sms = sms;
  cudaSetDevice(prev);
  return PKV_OK;
}

// Workspace of `dev` (the device of the call's tensors, which the caller has
// checked is current), allocating it on first use (refused while the stream
// is being captured: allocation would not be part of the graph).
int workspace_for(int dev, cudaStream_t stream, DeviceState** out, bool* capturing) {
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device %d", dev);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  *capturing = cs != cudaStreamCaptureStatusNone;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_dev[dev].ws.base) {
    if (*capturing)
      return fail(PKV_ERR_CAPTURE,
                  "the workspace of device %d must be allocated (pkv_init or one eager call) "
                  "before CUDA graph capture", dev);
    const int rc = init_locked(dev, 0);
    if (rc != PKV_OK) return rc;
  }
  *out = &g_dev[dev];
  return PKV_OK;
}

// Launches sharing a workspace must be ordered: a call on a new stream first
// waits for the stream of the previous call (outside graph capture).
int order_streams(DeviceState* st, cudaStream_t stream, bool capturing) {
  if (capturing) return PKV_OK;
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->has_last && st->last_stream != stream) {
    cudaError_t e = cudaEventRecord(st->order_event, st->last_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, st->order_event, 0);
    if (e != cudaSuccess) return cuda_fail(e, "cross-stream ordering");
  }
  st->last_stream = stream;
  st->has_last = true;
  return PKV_OK;
}

// ------------------------------------------------------------ validation --
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_tensor(const pkv_tensor* t, const char* name, int dtype, int ndim) {
  if (!t) return fail(PKV_ERR_INVALID_ARG, "%s is NULL", name);
  if (!t->data) return fail(PKV_ERR_INVALID_ARG, "%s has a NULL data pointer", name);
  if (t->dtype != dtype)
    return fail(PKV_ERR_INVALID_ARG, "%s has dtype %d, expected %d", name, t->dtype, dtype);
  if (t->ndim != ndim)
    return fail(PKV_ERR_INVALID_ARG, "%s has %d dims, expected %d", name, t->ndim, ndim);
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0 || t->stride[i] < 0)
      return fail(PKV_ERR_INVALID_ARG, "%s has a negative size or stride", name);
  return PKV_OK;
}

int elem_bytes(int dtype) {
  switch (dtype) {
    case PKV_DTYPE_BF16: return 2;
    case PKV_DTYPE_F32: return 4;
    case PKV_DTYPE_I32: return 4;
    case PKV_DTYPE_FP8_E4M3: return 1;
    default: return 1;
  }
}

// Byte range [lo, hi) a strided view spans (empty when any size is 0).
void byte_span(const pkv_tensor* t, uintptr_t* lo, uintptr_t* hi) {
  *lo = *hi = reinterpret_cast<uintptr_t>(t->data);
  int64_t last = 0;
  for (int i = 0; i < t->ndim; ++i) {
    if (t->shape[i] == 0) return;
    last += (t->shape[i] - 1) * t->stride[i];
  }
  *hi = *lo + uintptr_t((last + 1) * elem_bytes(t->dtype));
}

// True when two views share any byte.
bool overlaps(const pkv_tensor* a, const pkv_tensor* b) {
  if (!a || !b) return false;
  uintptr_t a0, a1, b0, b1;
  byte_span(a, &a0, &a1);
  byte_span(b, &b0, &b1);
  return a0 < a1 && b0 < b1 && a0 < b1 && b0 < a1;
}

// Outputs may not share memory with any input or with each other: the kernels
// read inputs of one request after writing outputs of another.
int check_no_overlap(std::initializer_list<std::pair<const pkv_tensor*, const char*>> outputs,
                     std::initializer_list<std::pair<const pkv_tensor*, const char*>> inputs) {
  for (auto o = outputs.begin(); o != outputs.end(); ++o) {
    for (const auto& i : inputs)
      if (overlaps(o->first, i.first))
        return fail(PKV_ERR_INVALID_ARG, "%s overlaps %s", o->second, i.second);
    for (auto o2 = o + 1; o2 != outputs.end(); ++o2)
      if (overlaps(o->first, o2->first))
        return fail(PKV_ERR_INVALID_ARG, "%s overlaps %s", o->second, o2->second);
  }
  return PKV_OK;
}

// Requests hold at most max_blocks x page_size keys; the kernels keep that
// product in 32-bit integers.
int check_table_width(const pkv_tensor* block_table, int page_size) {
  if (block_table->shape[1] < 1 || block_table->shape[1] * int64_t(page_size) >= (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "block_table width %lld x page_size %d must be in [1, 2^31)",
                (long long)block_table->shape[1], page_size);
  return PKV_OK;
}

// The device whose memory holds `t` (the call's device): it must be the
// current device and the device of `stream`.  While `stream` is being
// captured the pointer and stream queries are not made (they would end the
// capture); the call's device is then the current one.
int device_of(const pkv_tensor* t, const char* name, cudaStream_t stream, int* device) {
  int cur = 0;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  if (cs != cudaStreamCaptureStatusNone) {
    if (cur < 0 || cur >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device %d", cur);
    *device = cur;
    return PKV_OK;
  }
  cudaPointerAttributes a;
  e = cudaPointerGetAttributes(&a, t->data);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)
    return fail(PKV_ERR_INVALID_ARG, "%s is not device memory", name);
  const int dev = a.type == cudaMemoryTypeDevice ? a.device : cur;
  if (dev != cur)
    return fail(PKV_ERR_INVALID_ARG, "%s is on device %d but device %d is current", name, dev, cur);
  int sdev = 0;
  e = cudaStreamGetDevice(stream, &sdev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamGetDevice");
  if (sdev != dev)
    return fail(PKV_ERR_INVALID_ARG, "the stream belongs to device %d, %s to device %d", sdev, name,
                dev);
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_UNSUPPORTED, "device %d", dev);
  *device = dev;
  return PKV_OK;
}

// ---------------------------------------------------------- tensor maps --
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int get_encoder(EncodeTiledFn* fn) {
  static EncodeTiledFn cached = nullptr;
  static std::once_flag once;
  static cudaError_t status = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    status = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                              cudaEnableDefault, &q);
    if (status == cudaSuccess && q == cudaDriverEntryPointSuccess) cached = (EncodeTiledFn)p;
  });
  if (!cached) {
    if (status != cudaSuccess) return cuda_fail(status, "cuTensorMapEncodeTiled lookup");
    return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  }
  *fn = cached;
  return PKV_OK;
}

// The GQA cache [blocks, Hkv, P, 256] viewed as (64 dims, token, 4 chunks of 64
// dims, kv head, block): a box of (64, 16, 4, 1, 1) is one 16-token tile of one
// kv head, landing chunk-major (K lo, K hi, V lo, V hi; 16 rows of 128 bytes
// each, 128-byte swizzle) -- one TMA operation per 8 KB tile.
int encode_gqa_kv_map(EncodeTiledFn encode, const pkv_tensor* kv_cache, int page_size,
                      CUtensorMap* map) {
  const cuuint64_t gdim[5] = {64, cuuint64_t(page_size), 4, cuuint64_t(kv_cache->shape[1]),
                              cuuint64_t(kv_cache->shape[0])};
  const cuuint64_t gstride[4] = {cuuint64_t(kv_cache->stride[2]) * 2, 128,
                                 cuuint64_t(kv_cache->stride[1]) * 2,
                                 cuuint64_t(kv_cache->stride[0]) * 2};
  const cuuint32_t box[5] = {64, 16, 4, 1, 1};
  const cuuint32_t estride[5] = {1, 1, 1, 1, 1};
  const CUresult cr = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, kv_cache->data, gdim,
                             gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS)
    return fail(PKV_ERR_INVALID_ARG, "cuTensorMapEncodeTiled rejected the kv_cache layout (%d)",
                (int)cr);
  return PKV_OK;
}

}  // namespace

// =================================================================== ABI ==
extern "C" {

PKV_API int pkv_version(void) { return 100; }

PKV_API const char* pkv_last_error(void) { return g_last_error.c_str(); }

PKV_API int pkv_init(int device, size_t workspace_bytes) {
  if (device < 0 || device >= kMaxDevices) return fail(PKV_ERR_INVALID_ARG, "device %d", device);
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
  if (device >= count) return fail(PKV_ERR_INVALID_ARG, "device %d of %d", device, count);
  // refuse while the legacy stream of the device is capturing
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(device);
  e = cudaStreamIsCapturing(cudaStreamPerThread, &cs);
  cudaSetDevice(prev);
  if (e == cudaSuccess && cs != cudaStreamCaptureStatusNone)
    return fail(PKV_ERR_CAPTURE, "pkv_init during stream capture");
  std::lock_guard<std::mutex> lk(g_mu);
  return init_locked(device, workspace_bytes);
}

PKV_API int pkv_shutdown(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  int prev = 0;
  cudaGetDevice(&prev);
  for (int d = 0; d < kMaxDevices; ++d) {
    DeviceState& st = g_dev[d];
    if (!st.ws.base) continue;
    cudaSetDevice(d);
    cudaDeviceSynchronize();
    cudaFree(st.ws.base);
    if (st.order_event) cudaEventDestroy(st.order_event);
    st = DeviceState();
  }
  cudaSetDevice(prev);
  return PKV_OK;
}

PKV_API int pkv_check_errors(int device, int32_t* flags) {
  if (!flags) return fail(PKV_ERR_INVALID_ARG, "flags is NULL");
  *flags = 0;
  if (device < 0 || device >= kMaxDevices) return fail(PKV_ERR_INVALID_ARG, "device %d", device);
  // the error word of pkv_paged_decode_attn_noalloc's static scratch, if set up
  int* noalloc_err = pkv::noalloc_error_word(device);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[device];
  if (!st.ws.base && !noalloc_err) return PKV_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(device);
  int32_t v = 0, w = 0;
  cudaError_t e = cudaDeviceSynchronize();
  for (int* word : {static_cast<int*>(st.ws.err), noalloc_err}) {
    if (!word || e != cudaSuccess) continue;
    e = cudaMemcpy(&w, word, 4, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(word, 0, 4);
    v |= w;
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  cudaSetDevice(prev);
  if (e != cudaSuccess) return cuda_fail(e, "pkv_check_errors");
  *flags = v;
  if (v == 0) return PKV_OK;
  if (v & (pkv::DEVERR_BAD_BLOCK | pkv::DEVERR_SEQ_TOO_LONG))
    return fail(PKV_ERR_BAD_BLOCK_TABLE, "device error word 0x%x: bad block table or seq_lens", v);
  return fail(PKV_ERR_CUDA, "device error word 0x%x", v);
}

PKV_API int pkv_selftest_wait_timeout(int device, void* stream_ptr) {
  if (device < 0 || device >= kMaxDevices) return fail(PKV_ERR_INVALID_ARG, "device %d", device);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[device];
  if (!st.ws.base) return fail(PKV_ERR_INVALID_ARG, "device %d has no workspace: call pkv_init", device);
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(device);
  const cudaError_t e =
      pkv::launch_wait_selftest(static_cast<int*>(st.ws.err), static_cast<cudaStream_t>(stream_ptr));
  cudaSetDevice(prev);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
  return PKV_OK;
}

PKV_API int pkv_check_counters(int device, int64_t* nonzero) {
  if (!nonzero) return fail(PKV_ERR_INVALID_ARG, "nonzero is NULL");
  *nonzero = 0;
  if (device < 0 || device >= kMaxDevices) return fail(PKV_ERR_INVALID_ARG, "device %d", device);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[device];
  if (!st.ws.base) return PKV_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(device);
  const size_t n = 64 + size_t(st.ws.num_counters);
  int32_t* host = static_cast<int32_t*>(malloc(n * 4));
  if (!host) {
    cudaSetDevice(prev);
    return fail(PKV_ERR_INVALID_ARG, "host allocation failed");
  }
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(host, st.ws.sched, 64 * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess)
    e = cudaMemcpy(host + 64, st.ws.counters, size_t(st.ws.num_counters) * 4,
                   cudaMemcpyDeviceToHost);
  cudaSetDevice(prev);
  if (e != cudaSuccess) {
    free(host);
    return cuda_fail(e, "pkv_check_counters");
  }
  int64_t c = 0;
  for (size_t i = 0; i < n; ++i) c += host[i] != 0;
  free(host);
  *nonzero = c;
  return PKV_OK;
}

PKV_API int pkv_num_kv_splits(int max_seq_len, int batch, int qlen, int num_heads, int sm_count,
                              int block_h, double occupancy, int min_work_per_split,
                              int max_splits) {
  if (sm_count <= 0 || block_h <= 0 || qlen <= 0 || num_heads <= 0 || !(occupancy >= 0.0))
    return fail(PKV_ERR_INVALID_ARG, "pkv_num_kv_splits: bad argument");
  auto cdiv = [](long long a, long long b) { return (a + b - 1) / b; };
  const long long row_blocks = cdiv((long long)qlen * num_heads, block_h);
  const long long per_split = (long long)(batch > 1 ? batch : 1) * row_blocks;
  const long long ideal =
      cdiv(max_seq_len > 1 ? max_seq_len : 1, min_work_per_split > 1 ? min_work_per_split : 1);
  long long slots = (long long)(occupancy * sm_count);
  if (slots < 1) slots = 1;
  long long n;
  if (per_split <= slots) {
    n = slots / per_split;  // one dispatch round holds this many splits of every request
  } else {
    long long hi = ideal < max_splits ? ideal : max_splits;
    if (hi < 1) hi = 1;
    // cost(n) = rounds(n) / n: the idle tail of the last dispatch round
    double best = 1e300;
    for (long long k = 1; k <= hi; ++k) {
      const double c = double(cdiv(k * per_split, slots)) / double(k);
      if (c < best) best = c;
    }
    n = 1;
    for (long long k = 1; k <= hi; ++k) {
      const double c = double(cdiv(k * per_split, slots)) / double(k);
      if (c <= best * 1.05) {
        n = k;
        break;
      }
    }
  }
  long long r = n;
  if (ideal < r) r = ideal;
  if (2LL * sm_count < r) r = 2LL * sm_count;
  if (r < 1) r = 1;
  return (int)r;
}

PKV_API int pkv_paged_decode_attn(const pkv_tensor* q, const pkv_tensor* kv_cache,
                                  const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                                  const pkv_tensor* sinks, int window, float scale,
                                  int page_size, int num_kv_splits, const pkv_tensor* out,
                                  const pkv_tensor* lse, void* stream_ptr) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  pkv::GqaCall call;
  int rc = pkv::prepare_gqa_call(q, kv_cache, block_table, seq_lens, sinks, window, scale,
                                 page_size, num_kv_splits, out, lse, stream, &call);
  if (rc != PKV_OK || call.pairs == 0) return rc;
  DeviceState* st = nullptr;
  bool capturing = false;
  if ((rc = workspace_for(call.device, stream, &st, &capturing))) return rc;
  const pkv::Workspace& ws = st->ws;
  // partial slots: bounded by the partial bytes and by the split-group counters
  const int64_t item_bytes = int64_t(pkv::kGqaPartialFloats + pkv::kGqaMlFloats) * 4;
  const int64_t max_items =
      std::min<int64_t>(int64_t(ws.partial_bytes) / item_bytes, ws.num_counters - pkv::kTopCounters);
  pkv::GqaShape shape;
  if ((rc = pkv::gqa_launch_shape(call.pairs, call.cap_req, max_items, pkv::kTopCounters,
                                  ws.num_sms, call.p.max_blocks, page_size, &shape)))
    return rc;
  pkv::GqaParams& p = call.p;
  p.cap = shape.cluster > 1 ? shape.cluster : shape.cap;
  p.cluster = shape.cluster;
  p.min_pages = shape.min_pages;
  p.target_items = shape.target_items;
  p.part_o = ws.partials;
  p.part_ml = ws.partials + max_items * pkv::kGqaPartialFloats;
  p.max_items = max_items;
  p.counters = ws.counters;
  p.group_counters = ws.counters + pkv::kTopCounters;
  p.sched = ws.sched;
  p.err = ws.err;
  if ((rc = order_streams(st, stream, capturing))) return rc;
  const cudaError_t e = pkv::launch_gqa_decode(p, call.map, page_size, shape.grid, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gqa decode launch");
  return PKV_OK;
}

// Both MLA verify entry points: q (bf16) for pkv_mla_verify_attn, or q8 (e4m3
// codes) + q_scale for pkv_mla_verify_attn_fp8_native (native == true).
static int mla_verify_impl(const pkv_tensor* q, const pkv_tensor* q8, const pkv_tensor* q_scale,
                           bool native, const pkv_tensor* latent_cache,
                           const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                           const pkv_tensor* real_seq_lens, int qlen, float scale, int page_size,
                           const pkv_tensor* k_scale, const pkv_tensor* out, const pkv_tensor* lse,
                           int num_kv_splits, void* stream_ptr) {
  int rc;
  if (native) {
    if ((rc = check_tensor(q8, "q8", PKV_DTYPE_FP8_E4M3, 3))) return rc;
    if ((rc = check_tensor(q_scale, "q_scale", PKV_DTYPE_F32, 2))) return rc;
    if (q8->stride[2] != 1 || q8->stride[0] % 16 || q8->stride[1] % 16 || !aligned16(q8->data))
      return fail(PKV_ERR_ALIGNMENT, "q8 rows must be contiguous and 16-byte aligned");
    if (q_scale->shape[0] != q8->shape[0] || q_scale->shape[1] != q8->shape[1])
      return fail(PKV_ERR_INVALID_ARG, "q_scale must be [B*qlen, 128]");
    q = q8;
  } else if ((rc = check_tensor(q, "q", PKV_DTYPE_BF16, 3))) {
    return rc;
  }
  if (!latent_cache) return fail(PKV_ERR_INVALID_ARG, "latent_cache is NULL");
  const bool fp8 = latent_cache->dtype == PKV_DTYPE_FP8_E4M3;
  if (native && !fp8)
    return fail(PKV_ERR_UNSUPPORTED, "the native-FP8 path needs an e4m3 latent cache");
  if ((rc = check_tensor(latent_cache, "latent_cache", fp8 ? PKV_DTYPE_FP8_E4M3 : PKV_DTYPE_BF16,
                         latent_cache->ndim == 3 ? 3 : 4)))
    return rc;
  if ((rc = check_tensor(block_table, "block_table", PKV_DTYPE_I32, 2))) return rc;
  if ((rc = check_tensor(seq_lens, "seq_lens", PKV_DTYPE_I32, 1))) return rc;
  if (real_seq_lens && (rc = check_tensor(real_seq_lens, "real_seq_lens", PKV_DTYPE_I32, 1)))
    return rc;
  if ((rc = check_tensor(out, "out", PKV_DTYPE_BF16, 3))) return rc;
  if ((rc = check_tensor(lse, "lse", PKV_DTYPE_F32, 2))) return rc;
  if (k_scale) {
    if (!k_scale->data || k_scale->dtype != PKV_DTYPE_F32 ||
        !(k_scale->ndim == 0 || (k_scale->ndim == 1 && k_scale->shape[0] == 1)))
      return fail(PKV_ERR_INVALID_ARG, "k_scale must be an fp32 scalar on the device");
  }
  if (qlen < 1) return fail(PKV_ERR_INVALID_ARG, "qlen %d < 1", qlen);
  const int64_t R = q->shape[0], H = q->shape[1], Lk = q->shape[2];
  if (H != pkv::kMlaHeads) return fail(PKV_ERR_UNSUPPORTED, "%lld heads (128 are built)", (long long)H);
  if (Lk != pkv::kMlaLk) return fail(PKV_ERR_UNSUPPORTED, "Lk %lld (576 is built)", (long long)Lk);
  if (R % qlen) return fail(PKV_ERR_INVALID_ARG, "q rows %lld not a multiple of qlen %d", (long long)R, qlen);
  const int64_t B = R / qlen;
  if (page_size != 16 && page_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "page_size %d (16 and 32 are built)", page_size);
  // latent cache: [num_pages, P, 1, 576] or [num_pages * P, 1, 576]
  int64_t num_pages, s_page, s_tok;
  if (latent_cache->ndim == 4) {
    if (latent_cache->shape[1] != page_size || latent_cache->shape[2] != 1 ||
        latent_cache->shape[3] != Lk)
      return fail(PKV_ERR_INVALID_ARG, "latent_cache must be [num_pages, %d, 1, 576]", page_size);
    num_pages = latent_cache->shape[0];
    s_page = latent_cache->stride[0];
    s_tok = latent_cache->stride[1];
    if (latent_cache->stride[3] != 1)
      return fail(PKV_ERR_INVALID_ARG, "latent rows must be contiguous");
  } else {
    if (latent_cache->shape[1] != 1 || latent_cache->shape[2] != Lk ||
        latent_cache->shape[0] % page_size)
      return fail(PKV_ERR_INVALID_ARG, "latent_cache must be [num_pages * P, 1, 576]");
    num_pages = latent_cache->shape[0] / page_size;
    s_tok = latent_cache->stride[0];
    s_page = s_tok * page_size;
    if (latent_cache->stride[2] != 1)
      return fail(PKV_ERR_INVALID_ARG, "latent rows must be contiguous");
  }
  const int esz = fp8 ? 1 : 2;
  if (num_pages < 1 || num_pages >= (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_pages %lld", (long long)num_pages);
  if ((s_tok * esz) % 16 || (s_page * esz) % 16 || !aligned16(latent_cache->data))
    return fail(PKV_ERR_ALIGNMENT, "latent cache rows and pages must be 16-byte aligned");
  if (block_table->shape[0] != B || seq_lens->shape[0] != B ||
      (real_seq_lens && real_seq_lens->shape[0] != B))
    return fail(PKV_ERR_INVALID_ARG, "block_table / seq_lens / real_seq_lens batch mismatch");
  if (block_table->shape[1] < 1 || (block_table->stride[1] != 1 && block_table->shape[1] > 1))
    return fail(PKV_ERR_INVALID_ARG, "block_table rows must be non-empty and contiguous");
  if ((seq_lens->stride[0] != 1 && B > 1) ||
      (real_seq_lens && real_seq_lens->stride[0] != 1 && B > 1))
    return fail(PKV_ERR_INVALID_ARG, "seq_lens must be contiguous");
  if (out->shape[0] != R || out->shape[1] != H || out->shape[2] != pkv::kMlaLv)
    return fail(PKV_ERR_INVALID_ARG, "out must be [B*qlen, 128, 512]");
  if (lse->shape[0] != R || lse->shape[1] != H)
    return fail(PKV_ERR_INVALID_ARG, "lse must be [B*qlen, 128]");
  if (q->stride[2] != 1 || out->stride[2] != 1)
    return fail(PKV_ERR_INVALID_ARG, "q and out last dims must be contiguous");
  if ((!native && (q->stride[0] % 8 || q->stride[1] % 8 || !aligned16(q->data))) ||
      out->stride[0] % 8 || out->stride[1] % 8 || !aligned16(out->data))
    return fail(PKV_ERR_ALIGNMENT, "q and out must be 16-byte aligned with strides %% 8 == 0");
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (num_kv_splits < 0) return fail(PKV_ERR_INVALID_ARG, "num_kv_splits < 0");
  if ((rc = check_table_width(block_table, page_size))) return rc;
  if ((rc = check_no_overlap({{out, "out"}, {lse, "lse"}},
                             {{q, native ? "q8" : "q"}, {q_scale, "q_scale"},
                              {latent_cache, "latent_cache"}, {block_table, "block_table"},
                              {seq_lens, "seq_lens"}, {real_seq_lens, "real_seq_lens"},
                              {k_scale, "k_scale"}})))
    return rc;
  if (B == 0) return PKV_OK;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if ((rc = device_of(q, native ? "q8" : "q", stream, &dev))) return rc;
  DeviceState* st = nullptr;
  bool capturing = false;
  if ((rc = workspace_for(dev, stream, &st, &capturing))) return rc;
  const pkv::Workspace& ws = st->ws;
  // splits: at most 16 per (request, token, half); the device uses fewer for
  // short requests (at least 4096 keys per split, or 6144 on CTA pairs when
  // the batch is large enough: the planning kernel's choice)
  int64_t cap = num_kv_splits == 0 ? 16 : std::min<int64_t>(num_kv_splits, 16);
  // each slot: one partial plus one plan entry (the plan sits at the end)
  const int64_t max_slots = int64_t(ws.partial_bytes) / (pkv::kMlaPartialFloats * 4 + 4);
  const int64_t units = B * qlen * 2;
  if (units > pkv::kTopCounters)
    return fail(PKV_ERR_WORKSPACE, "%lld (row, half) units exceed the counters", (long long)units);
  if (num_kv_splits == 0) cap = std::max<int64_t>(1, std::min<int64_t>(cap, max_slots / units));
  if (units * cap > max_slots || units * cap >= (int64_t(1) << 31))
    return fail(PKV_ERR_WORKSPACE, "workspace holds %lld MLA partials, %lld needed",
                (long long)max_slots, (long long)(units * cap));
  {
    // no request holds more than max_blocks * page_size keys, so none uses
    // more splits than that many keys need: fewer CTAs with nothing to do
    const int64_t max_keys =
        std::min<int64_t>(block_table->shape[1], int64_t(1) << 30) * int64_t(page_size);
    const int64_t max_tiles = (max_keys + pkv::kMlaTile - 1) / pkv::kMlaTile;
    const int64_t need = (max_tiles + pkv::kMlaMinTiles - 1) / pkv::kMlaMinTiles;
    cap = std::max<int64_t>(1, std::min<int64_t>(cap, need));
  }

  EncodeTiledFn encode = nullptr;
  if ((rc = get_encoder(&encode))) return rc;
  CUtensorMap q_map, kv_map, v_map;
  // bf16 cache and an even number of verify tokens: tokens 2tp and 2tp + 1
  // share every key tile on a CTA pair
  const bool pair = !native && !fp8 && qlen % 2 == 0;
  if (native) {
    // the e4m3 cache as (64 dims, tokens, 9 chunks of 64 dims, pages): a box of
    // (64, 8, 9, 1) lands chunk-major, 8 rows of 64 bytes per chunk, 64-byte swizzle
    const cuuint64_t gdim[4] = {64, cuuint64_t(page_size), 9, cuuint64_t(num_pages)};
    const cuuint64_t gstr[3] = {cuuint64_t(s_tok), 64, cuuint64_t(s_page)};
    const cuuint32_t box[4] = {64, 8, 9, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult cr = encode(&kv_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, latent_cache->data, gdim, gstr,
                         box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS)
      return fail(PKV_ERR_INVALID_ARG, "latent cache tensor map rejected (%d)", (int)cr);
  } else {
    {
      const cuuint64_t gdim[3] = {cuuint64_t(Lk), cuuint64_t(H), cuuint64_t(R)};
      const cuuint64_t gstr[2] = {cuuint64_t(q->stride[1]) * 2, cuuint64_t(q->stride[0]) * 2};
      const cuuint32_t box[3] = {64, 128, 1};
      const cuuint32_t es[3] = {1, 1, 1};
      CUresult cr = encode(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q->data, gdim, gstr, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (cr != CUDA_SUCCESS) return fail(PKV_ERR_INVALID_ARG, "q tensor map rejected (%d)", (int)cr);
    }
    {
      // the cache viewed as (64 dims, tokens, 9 chunks of 64 dims, pages): a box
      // of (64, n tokens, 9, 1) lands chunk-major, n rows of 128 (bf16, 128-byte
      // swizzle) or 64 (e4m3, plain) bytes per chunk
      const cuuint64_t gdim[4] = {64, cuuint64_t(page_size), 9, cuuint64_t(num_pages)};
      const cuuint64_t gstr[3] = {cuuint64_t(s_tok) * esz, cuuint64_t(64 * esz),
                                  cuuint64_t(s_page) * esz};
      const cuuint32_t box[4] = {64, fp8 ? 16u : 8u, 9, 1};
      const cuuint32_t es[4] = {1, 1, 1, 1};
      CUresult cr = encode(&kv_map,
                           fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                           latent_cache->data, gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (cr != CUDA_SUCCESS)
        return fail(PKV_ERR_INVALID_ARG, "latent cache tensor map rejected (%d)", (int)cr);
    }
    if (pair) {
      // the same view, boxes of 16 tokens x 2 chunks: 128 V dims of 16 keys,
      // landing chunk-major (two 2 KB slabs of 16 rows of 128 bytes)
      const cuuint64_t gdim[4] = {64, cuuint64_t(page_size), 9, cuuint64_t(num_pages)};
      const cuuint64_t gstr[3] = {cuuint64_t(s_tok) * 2, 128, cuuint64_t(s_page) * 2};
      const cuuint32_t box[4] = {64, 16, 2, 1};
      const cuuint32_t es[4] = {1, 1, 1, 1};
      CUresult cr = encode(&v_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, latent_cache->data, gdim,
                           gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (cr != CUDA_SUCCESS)
        return fail(PKV_ERR_INVALID_ARG, "latent cache V tensor map rejected (%d)", (int)cr);
    }
  }
  pkv::MlaParams p;
  std::memset(&p, 0, sizeof p);
  if (native) {
    p.q8 = static_cast<const uint8_t*>(q8->data);
    p.q8_sr = q8->stride[0];
    p.q8_sh = q8->stride[1];
    p.q_scale = static_cast<const float*>(q_scale->data);
    p.qs_sr = q_scale->stride[0];
    p.qs_sh = q_scale->stride[1];
  } else {
    p.q = static_cast<const uint16_t*>(q->data);
    p.q_sr = q->stride[0];
    p.q_sh = q->stride[1];
  }
  p.kv = static_cast<const uint8_t*>(latent_cache->data);
  p.kv_stok = s_tok * esz;
  p.kv_spage = s_page * esz;
  p.bt = static_cast<const int32_t*>(block_table->data);
  p.bt_sb = block_table->stride[0];
  p.max_blocks = int(std::min<int64_t>(block_table->shape[1], int64_t(1) << 30));
  p.num_pages = int(num_pages);
  p.seq_lens = static_cast<const int32_t*>(seq_lens->data);
  p.real_seq_lens = real_seq_lens ? static_cast<const int32_t*>(real_seq_lens->data) : nullptr;
  p.k_scale = k_scale ? static_cast<const float*>(k_scale->data) : nullptr;
  p.out = static_cast<uint16_t*>(out->data);
  p.o_sr = out->stride[0];
  p.o_sh = out->stride[1];
  p.lse = static_cast<float*>(lse->data);
  p.lse_sr = lse->stride[0];
  p.lse_sh = lse->stride[1];
  p.B = int(B);
  p.qlen = qlen;
  p.cap = int(cap);
  p.page_size = page_size;
  p.scale = scale;
  p.pair_slots = ws.num_sms / 2;
  p.partials = ws.partials;
  p.max_slots = max_slots;
  p.counters = ws.counters;
  p.plan = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ws.partials) + ws.partial_bytes) -
           units * cap;
  p.err = ws.err;
  if ((rc = order_streams(st, stream, capturing))) return rc;
  const cudaError_t e =
      native ? pkv::launch_mla_verify_native(p, kv_map, int(units * cap), stream)
      : pair ? pkv::launch_mla_verify_pair(p, q_map, kv_map, v_map, int(units * cap), stream)
             : pkv::launch_mla_verify(p, q_map, kv_map, fp8, int(units * cap), stream);
  if (e != cudaSuccess) return cuda_fail(e, "mla verify launch");
  return PKV_OK;
}

PKV_API int pkv_mla_verify_attn(const pkv_tensor* q, const pkv_tensor* latent_cache,
                                const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                                const pkv_tensor* real_seq_lens, int qlen, float scale,
                                int page_size, const pkv_tensor* k_scale, const pkv_tensor* out,
                                const pkv_tensor* lse, int num_kv_splits, void* stream_ptr) {
  return mla_verify_impl(q, nullptr, nullptr, false, latent_cache, block_table, seq_lens,
                         real_seq_lens, qlen, scale, page_size, k_scale, out, lse, num_kv_splits,
                         stream_ptr);
}

PKV_API int pkv_mla_verify_attn_fp8_native(const pkv_tensor* q8, const pkv_tensor* q_scale,
                                           const pkv_tensor* latent_cache,
                                           const pkv_tensor* block_table,
                                           const pkv_tensor* seq_lens,
                                           const pkv_tensor* real_seq_lens, int qlen, float scale,
                                           int page_size, const pkv_tensor* k_scale,
                                           const pkv_tensor* out, const pkv_tensor* lse,
                                           int num_kv_splits, void* stream_ptr) {
  return mla_verify_impl(nullptr, q8, q_scale, true, latent_cache, block_table, seq_lens,
                         real_seq_lens, qlen, scale, page_size, k_scale, out, lse, num_kv_splits,
                         stream_ptr);
}

PKV_API int pkv_mla_quantize_q(const pkv_tensor* q, const pkv_tensor* q8,
                               const pkv_tensor* q_scale, void* stream_ptr) {
  int rc;
  if ((rc = check_tensor(q, "q", PKV_DTYPE_BF16, 3))) return rc;
  if ((rc = check_tensor(q8, "q8", PKV_DTYPE_FP8_E4M3, 3))) return rc;
  if ((rc = check_tensor(q_scale, "q_scale", PKV_DTYPE_F32, 2))) return rc;
  const int64_t R = q->shape[0], H = q->shape[1], Lk = q->shape[2];
  if (H != pkv::kMlaHeads) return fail(PKV_ERR_UNSUPPORTED, "%lld heads (128 are built)", (long long)H);
  if (Lk != pkv::kMlaLk) return fail(PKV_ERR_UNSUPPORTED, "Lk %lld (576 is built)", (long long)Lk);
  if (q8->shape[0] != R || q8->shape[1] != H || q8->shape[2] != Lk || q_scale->shape[0] != R ||
      q_scale->shape[1] != H)
    return fail(PKV_ERR_INVALID_ARG, "q8 must be [R, 128, 576] and q_scale [R, 128]");
  if (q->stride[2] != 1 || q->stride[0] % 8 || q->stride[1] % 8 || !aligned16(q->data))
    return fail(PKV_ERR_ALIGNMENT, "q rows must be contiguous and 16-byte aligned");
  if (q8->stride[2] != 1 || q8->stride[1] != Lk || q8->stride[0] % 16 || !aligned16(q8->data))
    return fail(PKV_ERR_ALIGNMENT, "q8 heads must be contiguous rows of 576 bytes, 16-byte aligned");
  if (q_scale->stride[1] != 1 && H > 1)
    return fail(PKV_ERR_INVALID_ARG, "q_scale rows must be contiguous");
  if (R == 0) return PKV_OK;
  if (R * H >= (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "%lld (row, head) pairs", (long long)(R * H));
  if ((rc = check_no_overlap({{q8, "q8"}, {q_scale, "q_scale"}}, {{q, "q"}}))) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if ((rc = device_of(q, "q", stream, &dev))) return rc;
  DeviceState* st = nullptr;
  bool capturing = false;
  if ((rc = workspace_for(dev, stream, &st, &capturing))) return rc;
  pkv::QuantParams p;
  p.q = static_cast<const uint16_t*>(q->data);
  p.q_sr = q->stride[0];
  p.q_sh = q->stride[1];
  p.q8 = static_cast<uint8_t*>(q8->data);
  p.q8_sr = q8->stride[0];
  p.q_scale = static_cast<float*>(q_scale->data);
  p.qs_sr = q_scale->stride[0];
  p.R = int(R);
  p.H = int(H);
  if ((rc = order_streams(st, stream, capturing))) return rc;
  const cudaError_t e = pkv::launch_mla_quantize_q(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "mla quantize launch");
  return PKV_OK;
}

PKV_API int pkv_gqa_kv_append(const pkv_tensor* k, const pkv_tensor* v, const pkv_tensor* kv_cache,
                              const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                              int page_size, void* stream_ptr) {
  int rc;
  if ((rc = check_tensor(k, "k", PKV_DTYPE_BF16, 3))) return rc;
  if ((rc = check_tensor(v, "v", PKV_DTYPE_BF16, 3))) return rc;
  if ((rc = check_tensor(kv_cache, "kv_cache", PKV_DTYPE_BF16, 4))) return rc;
  if ((rc = check_tensor(block_table, "block_table", PKV_DTYPE_I32, 2))) return rc;
  if ((rc = check_tensor(seq_lens, "seq_lens", PKV_DTYPE_I32, 1))) return rc;
  const int64_t B = k->shape[0], Hkv = k->shape[1], D = k->shape[2];
  const int64_t nb = kv_cache->shape[0];
  if (D != pkv::kGqaHeadDim)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %lld (only 128 is built)", (long long)D);
  if (v->shape[0] != B || v->shape[1] != Hkv || v->shape[2] != D)
    return fail(PKV_ERR_INVALID_ARG, "v must have the shape of k");
  if (kv_cache->shape[1] != Hkv || kv_cache->shape[3] != 2 * D)
    return fail(PKV_ERR_INVALID_ARG, "kv_cache must be [num_blocks, Hkv, P, 256]");
  if (page_size != 16 && page_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "page_size %d (16 and 32 are built)", page_size);
  if (kv_cache->shape[2] != page_size)
    return fail(PKV_ERR_INVALID_ARG, "kv_cache.shape[2] %lld != page_size %d",
                (long long)kv_cache->shape[2], page_size);
  if (nb < 1 || nb >= (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_blocks %lld", (long long)nb);
  if (block_table->shape[0] != B || seq_lens->shape[0] != B)
    return fail(PKV_ERR_INVALID_ARG, "block_table / seq_lens batch mismatch");
  if (block_table->shape[1] < 1 || block_table->shape[1] > (int64_t(1) << 30) ||
      (block_table->stride[1] != 1 && block_table->shape[1] > 1))
    return fail(PKV_ERR_INVALID_ARG, "block_table rows must be non-empty and contiguous");
  if (seq_lens->stride[0] != 1 && B > 1)
    return fail(PKV_ERR_INVALID_ARG, "seq_lens must be contiguous");
  if (k->stride[2] != 1 || v->stride[2] != 1 || kv_cache->stride[3] != 1)
    return fail(PKV_ERR_INVALID_ARG, "k/v last dim and kv_cache rows must be contiguous");
  if (k->stride[0] != v->stride[0] || k->stride[1] != v->stride[1])
    return fail(PKV_ERR_INVALID_ARG, "k and v must share strides");
  if (k->stride[0] % 8 || k->stride[1] % 8 || kv_cache->stride[0] % 8 ||
      kv_cache->stride[1] % 8 || kv_cache->stride[2] % 8)
    return fail(PKV_ERR_ALIGNMENT, "strides of k, v and kv_cache must be multiples of 8");
  if (!aligned16(k->data) || !aligned16(v->data) || !aligned16(kv_cache->data))
    return fail(PKV_ERR_ALIGNMENT, "k, v and kv_cache must be 16-byte aligned");
  if ((rc = check_table_width(block_table, page_size))) return rc;
  if ((rc = check_no_overlap({{kv_cache, "kv_cache"}},
                             {{k, "k"}, {v, "v"}, {block_table, "block_table"},
                              {seq_lens, "seq_lens"}})))
    return rc;
  if (B == 0) return PKV_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if ((rc = device_of(kv_cache, "kv_cache", stream, &dev))) return rc;
  DeviceState* st = nullptr;
  bool capturing = false;
  if ((rc = workspace_for(dev, stream, &st, &capturing))) return rc;
  pkv::AppendParams p;
  std::memset(&p, 0, sizeof p);
  p.k = static_cast<const uint16_t*>(k->data);
  p.v = static_cast<const uint16_t*>(v->data);
  p.s_sb = k->stride[0];
  p.s_sh = k->stride[1];
  p.cache = static_cast<uint8_t*>(kv_cache->data);
  p.c_sblk = kv_cache->stride[0] * 2;
  p.c_sh = kv_cache->stride[1] * 2;
  p.c_stok = kv_cache->stride[2] * 2;
  p.num_blocks = int(nb);
  p.bt = static_cast<const int32_t*>(block_table->data);
  p.bt_sb = block_table->stride[0];
  p.max_blocks = int(block_table->shape[1]);
  p.seq_lens = static_cast<const int32_t*>(seq_lens->data);
  p.B = int(B);
  p.Hkv = int(Hkv);
  p.qlen = 1;
  p.page_size = page_size;
  p.err = st->ws.err;
  if (B * Hkv >= (int64_t(1) << 31)) return fail(PKV_ERR_UNSUPPORTED, "B x Hkv too large");
  const cudaError_t e = pkv::launch_gqa_kv_append(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "gqa kv append launch");
  return PKV_OK;
}

PKV_API int pkv_mla_kv_append(const pkv_tensor* latent, const pkv_tensor* latent_cache,
                              const pkv_tensor* block_table, const pkv_tensor* seq_lens, int qlen,
                              int page_size, const pkv_tensor* k_scale, void* stream_ptr) {
  int rc;
  if ((rc = check_tensor(latent, "latent", PKV_DTYPE_BF16, 2))) return rc;
  if (!latent_cache) return fail(PKV_ERR_INVALID_ARG, "latent_cache is NULL");
  const bool fp8 = latent_cache->dtype == PKV_DTYPE_FP8_E4M3;
  if ((rc = check_tensor(latent_cache, "latent_cache", fp8 ? PKV_DTYPE_FP8_E4M3 : PKV_DTYPE_BF16,
                         latent_cache->ndim == 4 ? 4 : 3)))
    return rc;
  if ((rc = check_tensor(block_table, "block_table", PKV_DTYPE_I32, 2))) return rc;
  if ((rc = check_tensor(seq_lens, "seq_lens", PKV_DTYPE_I32, 1))) return rc;
  if (k_scale) {
    if ((rc = check_tensor(k_scale, "k_scale", PKV_DTYPE_F32, k_scale->ndim))) return rc;
    if (!(k_scale->ndim == 0 || (k_scale->ndim == 1 && k_scale->shape[0] == 1)))
      return fail(PKV_ERR_INVALID_ARG, "k_scale must be an fp32 scalar on the device");
  }
  if (qlen < 1) return fail(PKV_ERR_INVALID_ARG, "qlen %d < 1", qlen);
  const int64_t R = latent->shape[0], Lk = latent->shape[1];
  if (Lk != pkv::kMlaLk) return fail(PKV_ERR_UNSUPPORTED, "Lk %lld (576 is built)", (long long)Lk);
  if (R % qlen) return fail(PKV_ERR_INVALID_ARG, "latent rows %lld not a multiple of qlen %d",
                            (long long)R, qlen);
  const int64_t B = R / qlen;
  if (page_size != 16 && page_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "page_size %d (16 and 32 are built)", page_size);
  int64_t num_pages, s_page, s_tok;
  if (latent_cache->ndim == 4) {
    if (latent_cache->shape[1] != page_size || latent_cache->shape[2] != 1 ||
        latent_cache->shape[3] != Lk || latent_cache->stride[3] != 1)
      return fail(PKV_ERR_INVALID_ARG, "latent_cache must be [num_pages, %d, 1, 576], rows contiguous",
                  page_size);
    num_pages = latent_cache->shape[0];
    s_page = latent_cache->stride[0];
    s_tok = latent_cache->stride[1];
  } else {
    if (latent_cache->shape[1] != 1 || latent_cache->shape[2] != Lk ||
        latent_cache->shape[0] % page_size || latent_cache->stride[2] != 1)
      return fail(PKV_ERR_INVALID_ARG, "latent_cache must be [num_pages * P, 1, 576], rows contiguous");
    num_pages = latent_cache->shape[0] / page_size;
    s_tok = latent_cache->stride[0];
    s_page = s_tok * page_size;
  }
  const int esz = fp8 ? 1 : 2;
  if (num_pages < 1 || num_pages >= (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_pages %lld", (long long)num_pages);
  if ((s_tok * esz) % 16 || (s_page * esz) % 16 || !aligned16(latent_cache->data))
    return fail(PKV_ERR_ALIGNMENT, "latent cache rows and pages must be 16-byte aligned");
  if (latent->stride[1] != 1 || latent->stride[0] % 8 || !aligned16(latent->data))
    return fail(PKV_ERR_ALIGNMENT, "latent rows must be contiguous and 16-byte aligned");
  if (block_table->shape[0] != B || seq_lens->shape[0] != B)
    return fail(PKV_ERR_INVALID_ARG, "block_table / seq_lens batch mismatch");
  if (block_table->shape[1] < 1 || block_table->shape[1] > (int64_t(1) << 30) ||
      (block_table->stride[1] != 1 && block_table->shape[1] > 1))
    return fail(PKV_ERR_INVALID_ARG, "block_table rows must be non-empty and contiguous");
  if (seq_lens->stride[0] != 1 && B > 1)
    return fail(PKV_ERR_INVALID_ARG, "seq_lens must be contiguous");
  if (R >= (int64_t(1) << 31)) return fail(PKV_ERR_UNSUPPORTED, "too many latent rows");
  if ((rc = check_table_width(block_table, page_size))) return rc;
  if ((rc = check_no_overlap({{latent_cache, "latent_cache"}},
                             {{latent, "latent"}, {block_table, "block_table"},
                              {seq_lens, "seq_lens"}, {k_scale, "k_scale"}})))
    return rc;
  if (B == 0) return PKV_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if ((rc = device_of(latent_cache, "latent_cache", stream, &dev))) return rc;
  DeviceState* st = nullptr;
  bool capturing = false;
  if ((rc = workspace_for(dev, stream, &st, &capturing))) return rc;
  pkv::AppendParams p;
  std::memset(&p, 0, sizeof p);
  p.k = static_cast<const uint16_t*>(latent->data);
  p.s_sb = latent->stride[0];
  p.cache = static_cast<uint8_t*>(latent_cache->data);
  p.c_sblk = s_page * esz;
  p.c_stok = s_tok * esz;
  p.num_blocks = int(num_pages);
  p.bt = static_cast<const int32_t*>(block_table->data);
  p.bt_sb = block_table->stride[0];
  p.max_blocks = int(block_table->shape[1]);
  p.seq_lens = static_cast<const int32_t*>(seq_lens->data);
  p.B = int(B);
  p.Hkv = 1;
  p.qlen = qlen;
  p.page_size = page_size;
  p.fp8 = fp8 ? 1 : 0;
  p.k_scale = (fp8 && k_scale) ? static_cast<const float*>(k_scale->data) : nullptr;
  p.err = st->ws.err;
  const cudaError_t e = pkv::launch_mla_kv_append(p, stream);
  if (e != cudaSuccess) return cuda_fail(e, "mla kv append launch");
  return PKV_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Shared with entry points implemented in other translation units.
namespace pkv {

int abi_fail(int code, const char* message) { return fail(code, "%s", message); }

int abi_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }

int prepare_gqa_call(const pkv_tensor* q, const pkv_tensor* kv_cache,
                     const pkv_tensor* block_table, const pkv_tensor* seq_lens,
                     const pkv_tensor* sinks, int window, float scale, int page_size,
                     int num_kv_splits, const pkv_tensor* out, const pkv_tensor* lse,
                     cudaStream_t stream, GqaCall* call) {
  int rc;
  if ((rc = check_tensor(q, "q", PKV_DTYPE_BF16, 3))) return rc;
  if ((rc = check_tensor(kv_cache, "kv_cache", PKV_DTYPE_BF16, 4))) return rc;
  if ((rc = check_tensor(block_table, "block_table", PKV_DTYPE_I32, 2))) return rc;
  if ((rc = check_tensor(seq_lens, "seq_lens", PKV_DTYPE_I32, 1))) return rc;
  if ((rc = check_tensor(out, "out", PKV_DTYPE_BF16, 3))) return rc;
  if (sinks && (rc = check_tensor(sinks, "sinks", PKV_DTYPE_F32, 1))) return rc;
  if (lse && (rc = check_tensor(lse, "lse", PKV_DTYPE_F32, 2))) return rc;
  const int64_t B = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t nb = kv_cache->shape[0], Hkv = kv_cache->shape[1];
  if (D != kGqaHeadDim)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %lld (only 128 is built)", (long long)D);
  if (kv_cache->shape[3] != 2 * D)
    return fail(PKV_ERR_INVALID_ARG, "kv_cache last dim %lld, expected [K | V] = 256",
                (long long)kv_cache->shape[3]);
  if (Hkv <= 0 || Hq != kGqaGroup * Hkv)
    return fail(PKV_ERR_UNSUPPORTED, "num_q_heads %lld must be 8 x num_kv_heads %lld",
                (long long)Hq, (long long)Hkv);
  if (page_size != 16 && page_size != 32)
    return fail(PKV_ERR_UNSUPPORTED, "page_size %d (16 and 32 are built)", page_size);
  if (kv_cache->shape[2] != page_size)
    return fail(PKV_ERR_INVALID_ARG, "kv_cache.shape[2] %lld != page_size %d",
                (long long)kv_cache->shape[2], page_size);
  if (nb < 1 || nb >= (int64_t(1) << 31))
    return fail(PKV_ERR_INVALID_ARG, "num_blocks %lld", (long long)nb);
  if (block_table->shape[0] != B || seq_lens->shape[0] != B)
    return fail(PKV_ERR_INVALID_ARG, "block_table / seq_lens batch mismatch");
  if (out->shape[0] != B || out->shape[1] != Hq || out->shape[2] != D)
    return fail(PKV_ERR_INVALID_ARG, "out shape mismatch");
  if (sinks && sinks->shape[0] != Hq) return fail(PKV_ERR_INVALID_ARG, "sinks must be [Hq]");
  if (sinks && sinks->shape[0] > 1 && sinks->stride[0] != 1)
    return fail(PKV_ERR_INVALID_ARG, "sinks must be contiguous");
  if (lse && (lse->shape[0] != B || lse->shape[1] != Hq))
    return fail(PKV_ERR_INVALID_ARG, "lse must be [B, Hq]");
  if ((rc = check_table_width(block_table, page_size))) return rc;
  if (block_table->stride[1] != 1 && block_table->shape[1] > 1)
    return fail(PKV_ERR_INVALID_ARG, "block_table rows must be contiguous");
  if (seq_lens->stride[0] != 1 && B > 1)
    return fail(PKV_ERR_INVALID_ARG, "seq_lens must be contiguous");
  if (!std::isfinite(scale)) return fail(PKV_ERR_INVALID_ARG, "scale is not finite");
  if (num_kv_splits < 0) return fail(PKV_ERR_INVALID_ARG, "num_kv_splits < 0");
  if (B > kGqaMaxBatch)
    return fail(PKV_ERR_UNSUPPORTED, "batch %lld > %d", (long long)B, kGqaMaxBatch);
  // layout rules of the HND page cache and 16-byte vector access
  if (q->stride[2] != 1 || out->stride[2] != 1 || kv_cache->stride[3] != 1 ||
      kv_cache->stride[2] != 2 * D)
    return fail(PKV_ERR_INVALID_ARG, "q/out last dim and kv_cache rows must be contiguous");
  if (q->stride[0] % 8 || q->stride[1] % 8 || out->stride[0] % 8 || out->stride[1] % 8 ||
      kv_cache->stride[0] % 8 || kv_cache->stride[1] % 8)
    return fail(PKV_ERR_ALIGNMENT, "strides of q, out and kv_cache must be multiples of 8");
  if (!aligned16(q->data) || !aligned16(out->data) || !aligned16(kv_cache->data))
    return fail(PKV_ERR_ALIGNMENT, "q, out and kv_cache must be 16-byte aligned");
  if ((rc = check_no_overlap({{out, "out"}, {lse, "lse"}},
                             {{q, "q"}, {kv_cache, "kv_cache"}, {block_table, "block_table"},
                              {seq_lens, "seq_lens"}, {sinks, "sinks"}})))
    return rc;

  std::memset(call, 0, sizeof *call);
  call->pairs = B * Hkv;
  call->cap_req = num_kv_splits;
  call->page_size = page_size;
  if (B == 0) return PKV_OK;
  if ((rc = device_of(q, "q", stream, &call->device))) return rc;

  EncodeTiledFn encode = nullptr;
  if ((rc = get_encoder(&encode))) return rc;
  if ((rc = encode_gqa_kv_map(encode, kv_cache, page_size, &call->map))) return rc;
  GqaParams& p = call->p;
  p.q = static_cast<const uint16_t*>(q->data);
  p.q_sb = q->stride[0];
  p.q_sh = q->stride[1];
  p.bt = static_cast<const int32_t*>(block_table->data);
  p.bt_sb = block_table->stride[0];
  p.max_blocks = int(block_table->shape[1]);
  p.num_blocks = int(nb);
  p.seq_lens = static_cast<const int32_t*>(seq_lens->data);
  p.sinks = sinks ? static_cast<const float*>(sinks->data) : nullptr;
  p.out = static_cast<uint16_t*>(out->data);
  p.o_sb = out->stride[0];
  p.o_sh = out->stride[1];
  p.lse = lse ? static_cast<float*>(lse->data) : nullptr;
  p.lse_sb = lse ? lse->stride[0] : 0;
  p.lse_sh = lse ? lse->stride[1] : 0;
  p.B = int(B);
  p.Hkv = int(Hkv);
  p.window = window;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.scale = scale;
  return PKV_OK;
}

int gqa_launch_shape(int64_t pairs, int cap_req, int64_t max_items, int64_t max_pairs,
                     int num_sms, int max_blocks, int page_size, GqaShape* shape) {
  if (pairs > max_pairs)
    return fail(PKV_ERR_WORKSPACE, "%lld (request, kv head) pairs exceed the %lld counters",
                (long long)pairs, (long long)max_pairs);
  // At most 256 splits per (request, kv head): the merge runs in at most two
  // levels of at most 16 partials each.
  int64_t cap = cap_req == 0 ? max_items / pairs : cap_req;
  if (cap > 256) cap = 256;
  if (cap < 1) cap = 1;
  // A launch whose requests cannot split writes no partials and no counters.
  if (cap > 1 && pairs * cap > max_items)
    return fail(PKV_ERR_WORKSPACE, "scratch holds %lld split partials, %lld x %lld needed",
                (long long)max_items, (long long)pairs, (long long)cap);
  const int64_t grid = std::max<int64_t>(
      1, std::min<int64_t>(int64_t(num_sms) * gqa_ctas_per_sm(), pairs * cap));
  shape->cap = int(cap);
  shape->grid = int(grid);
  // About four items per CTA (A/B on the Flint batch: best of 2..24), but no
  // more than 16 per (request, kv head) while that still gives every CTA one:
  // a few long requests then stream fewer, larger splits, each merged in a
  // single 16-way level (one 131072-token request, auto cap, on GB300:
  // 118.7 -> 106.5 us; eight of them 632.8 -> 627.4 us).
  shape->target_items = int(std::max<int64_t>(grid, std::min<int64_t>(grid * 4, pairs * 16)));
  // A split streams at least 256 keys (128 KB per kv head).  Cluster mode
  // (splits merged through distributed shared memory, no queue and no
  // workspace partials) for small launches whose requests are short:
  // C = splits a request of the block table's full width can use (at most 8,
  // at least 128 keys each: then a CTA's whole split is usually among the
  // tiles it requests before the dependency wait; A/B on the tiny batch,
  // graph-replayed: 256 -> 128 keys 5.4 -> 4.0 us per call, 64 keys no
  // better), when every (request, kv head) gets its own cluster in a single
  // wave and no split can exceed 64 pages.
  shape->min_pages = 256 / page_size;
  const int64_t cl_min = 128 / page_size;
  const int64_t c = std::min<int64_t>(std::min<int64_t>(cap, kGqaMaxCluster),
                                      (int64_t(max_blocks) + cl_min - 1) / cl_min);
  shape->cluster = 0;
  if (c >= 2 && c * pairs <= int64_t(num_sms) * gqa_ctas_per_sm() &&
      (int64_t(max_blocks) + c - 1) / c <= 64) {
    shape->cluster = int(c);
    shape->min_pages = int(cl_min);
  }
  return PKV_OK;
}

}  // namespace pkv
