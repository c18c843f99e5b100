// static_workspace.cu -- an attention entry point that allocates nothing.
//
// Some callers cannot allocate device memory at the point where they run
// attention: a serving loop whose device memory was fully reserved at start
// (for instance a KV-cache pool sized to fill the GPU), code running inside a
// host framework that hands out no scratch buffers, or a path that must not
// call cudaMalloc because it would synchronise the device.  For them this
// file keeps the attention workspace (work list, split-KV partial states,
// merge counters, flag word) in one fixed array that lives inside the
// library: every GPU that loads the library holds it until the process exits.
//
// Host code only knows the array's host-side stand-in name; its device
// address is looked up with cudaGetSymbolAddress, with the calling device
// current, on every call made outside a stream capture (a device reset in
// the process cannot leave a stale address behind).  Inside a capture the
// address looked up by the device's last uncaptured call is used.
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "nvfp4kv.h"

namespace nvfp4kv {
int set_error_detail(int status, const char* message);
int validate_run(const nvfp4kv_plan_info* info, const void* q, int64_t qst, int64_t qsh,
                 const nvfp4kv_paged_cache* cache, const int32_t* kv_indices,
                 const void* workspace, uint64_t workspace_bytes, const void* out);
}

namespace {

constexpr uint64_t kStaticWorkspaceBytes = 16ull << 20;  // 16 MiB

static __device__ __align__(256) uint8_t g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_device_address[kMaxDevices] = {};

// The array's device address on the current device (see the file comment).
int static_address(cudaStream_t stream, void** out) {
  using nvfp4kv::set_error_detail;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error_detail(NVFP4KV_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return set_error_detail(NVFP4KV_ERR_UNSUPPORTED, "device index beyond 127");
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return set_error_detail(NVFP4KV_ERR_CUDA, cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess) return set_error_detail(NVFP4KV_ERR_CUDA, cudaGetErrorString(e));
    g_device_address[dev] = ptr;
  } else if (!g_device_address[dev]) {
    return set_error_detail(NVFP4KV_ERR_INVALID_ARGUMENT,
                            "first static-workspace call on this device is inside a stream "
                            "capture; make one call before capturing");
  }
  *out = g_device_address[dev];
  return NVFP4KV_OK;
}

}  // namespace

extern "C" int nvfp4kv_decode_run_static(const nvfp4kv_plan_info* info, const void* plan_host,
                                         const void* q_bf16, int64_t q_stride_tok,
                                         int64_t q_stride_head,
                                         const nvfp4kv_paged_cache* cache,
                                         const int32_t* kv_indices, float sm_scale,
                                         void* out_bf16, float* lse, cudaStream_t stream) {
  using nvfp4kv::set_error_detail;
  if (!info || info->magic != nvfp4kv::kPlanMagic)
    return set_error_detail(NVFP4KV_ERR_INVALID_ARGUMENT, "info is not a plan");
  if (info->workspace_bytes > kStaticWorkspaceBytes)
    return set_error_detail(NVFP4KV_ERR_WORKSPACE_TOO_SMALL,
                            "the plan needs more workspace than the 16 MiB static "
                            "workspace holds; use nvfp4kv_decode_run with a caller "
                            "workspace, or plan fewer splits");
  if (info->plan_host_bytes > 0 && !plan_host)
    return set_error_detail(NVFP4KV_ERR_INVALID_ARGUMENT, "plan_host is null");
  void* ws = nullptr;
  if (int st = static_address(stream, &ws)) return st;
  // every argument check of the run first: a rejected call enqueues nothing
  if (int st = nvfp4kv::validate_run(info, q_bf16, q_stride_tok, q_stride_head, cache,
                                     kv_indices, ws, kStaticWorkspaceBytes, out_bf16))
    return st;
  uint8_t* base = static_cast<uint8_t*>(ws);
  // the array keeps the previous call's contents: the flag word and the merge
  // counters must start at zero, the work list is this plan's
  cudaError_t e = cudaMemsetAsync(base, 0, info->off_units, stream);
  if (e == cudaSuccess && info->plan_host_bytes > 0)
    e = cudaMemcpyAsync(base + info->off_units, plan_host, info->plan_host_bytes,
                        cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return set_error_detail(NVFP4KV_ERR_CUDA, cudaGetErrorString(e));
  return nvfp4kv_decode_run(info, q_bf16, q_stride_tok, q_stride_head, cache, kv_indices,
                            sm_scale, ws, kStaticWorkspaceBytes, out_bf16, lse, stream);
}

extern "C" int nvfp4kv_static_workspace_flags(const nvfp4kv_plan_info* info, uint32_t* flags,
                                              int32_t clear, cudaStream_t stream) {
  using nvfp4kv::set_error_detail;
  if (!info || info->magic != nvfp4kv::kPlanMagic || !flags)
    return set_error_detail(NVFP4KV_ERR_INVALID_ARGUMENT, "info is not a plan, or flags is null");
  void* ws = nullptr;
  if (int st = static_address(stream, &ws)) return st;
  return nvfp4kv_workspace_flags(info, ws, flags, clear, stream);
}
