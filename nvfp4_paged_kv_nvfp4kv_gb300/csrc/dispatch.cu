// dispatch.cu -- launching the attention kernels through their descriptions.
#include <mutex>
#include <set>

#include <cuda_runtime.h>

#include "internal.h"

namespace nvfp4kv {

// Opt a kernel into its dynamic shared-memory size (once per kernel and
// device; the runtime keeps the attribute per function per device).
cudaError_t prepare_kernel(const AttendConfig& cfg) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({cfg.func, dev})) return cudaSuccess;
  e = cudaFuncSetAttribute(cfg.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           cfg.smem_bytes);
  if (e == cudaSuccess) done.insert({cfg.func, dev});
  return e;
}

cudaError_t launch_attend(const AttendConfig& cfg, const AttendParams& p, int grid_x,
                          int grid_y, cudaStream_t stream) {
  void* args[] = {const_cast<AttendParams*>(&p)};
  const int upc = cfg.units_per_cta > 1 ? cfg.units_per_cta : 1;
  return cudaLaunchKernel(cfg.func, dim3((grid_x + upc - 1) / upc, grid_y),
                          dim3(cfg.warps * 32), args, cfg.smem_bytes, stream);
}

}  // namespace nvfp4kv
