// api.cu - library-wide entry points (workspace sizes, status names) and the per-device host
// caches every entry point shares.
#include <map>
#include <mutex>
#include <utility>

#include "dspark_common.cuh"
#include "host_common.h"

namespace {
std::mutex ds_cache_mu;
std::map<int, int> ds_sms_by_device;
std::map<std::pair<int, const void*>, size_t> ds_smem_by_kernel;
}  // namespace

int ds_num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 148;
  }
  std::lock_guard<std::mutex> lock(ds_cache_mu);
  auto it = ds_sms_by_device.find(dev);
  if (it != ds_sms_by_device.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    return 148;                                   // not cached: asked again next time
  }
  ds_sms_by_device[dev] = n;
  return n;
}

cudaError_t ds_ensure_smem(const void* func, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(ds_cache_mu);
  size_t& have = ds_smem_by_kernel[std::make_pair(dev, func)];
  if (bytes <= have) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
  if (e == cudaSuccess) have = bytes;
  return e;
}

// Per-op workspace layouts are defined next to their kernels; these sizes must cover them.
extern "C" size_t dspark_internal_ws_sample(int64_t R, int32_t B, int64_t V);
extern "C" size_t dspark_internal_ws_dense_walk(int64_t R, int32_t B, int64_t V);
extern "C" size_t dspark_internal_ws_verify(int64_t R, int32_t B, int64_t V);
extern "C" size_t dspark_internal_ws_lattice_row(int64_t R, int32_t B, int64_t V);

extern "C" size_t dspark_workspace_size(dspark_op op, int64_t R, int32_t B, int64_t V, int32_t K) {
  (void)K;
  if (R < 0 || B < 0 || V < 0) return 0;
  switch (op) {
    case DSPARK_OP_D2T_CHECK:
      return size_t(ds_ceil_div(V, 32)) * sizeof(uint32_t) + 256;
    case DSPARK_OP_TOPK:
      return 0;
    case DSPARK_OP_SAMPLE:
      return dspark_internal_ws_sample(R, B, V);
    case DSPARK_OP_DENSE_WALK:
      return dspark_internal_ws_dense_walk(R, B, V);
    case DSPARK_OP_VERIFY:
      return dspark_internal_ws_verify(R, B, V);
    case DSPARK_OP_LATTICE_ROW:
      return dspark_internal_ws_lattice_row(R, B, V);
    default:
      return 0;
  }
}

extern "C" const char* dspark_status_string(dspark_status s) {
  switch (s) {
    case DSPARK_OK: return "ok";
    case DSPARK_EINVAL: return "invalid argument";
    case DSPARK_ERANGE: return "d2t or token id out of range";
    case DSPARK_EDUP: return "d2t is not one-to-one";
    case DSPARK_EPROPOSAL: return "recorded proposal probability of a drafted token is zero";
    case DSPARK_ENONFINITE: return "non-finite row maximum";
    case DSPARK_ETIMEOUT: return "bounded device wait ran out";
    case DSPARK_ECUDA: return "CUDA error";
    case DSPARK_EWORKSPACE: return "workspace missing, misaligned or too small";
    default: return "unknown status";
  }
}
