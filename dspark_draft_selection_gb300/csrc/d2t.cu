// d2t.cu - pruned-vocabulary map validation (dspark_d2t_check).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"), commit on the d2t checks: d2t needs an entry for every draft
// logit, every mapped id must lie inside the target vocabulary, and sampled drafting needs the
// map to be one-to-one (two draft tokens on one target id would repeat ids in a proposal);
// greedy drafting accepts any mapping. optimum-intel PR #2099, Pruned draft vocabulary:
// draft token i is target token i + d2t[i].
//
// Two passes so that a range error always wins over a duplicate: the range pass, then (only if
// the status word is still clear) a pass that sets one bit per target id in a workspace bitmap
// and reports an id whose bit was already set.
#include "dspark_common.cuh"
#include "host_common.h"

namespace {

__global__ void d2t_range_kernel(const int64_t* d2t, int64_t V_d, int64_t V_t, int32_t* status) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < V_d; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t t = i + d2t[i];
    if (t < 0 || t >= V_t) ds_set_error(status, DSPARK_ERANGE);
  }
}

__global__ void d2t_dup_kernel(const int64_t* d2t, int64_t V_d, uint32_t* bitmap, int32_t* status) {
  if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < V_d; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t t = i + d2t[i];
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&bitmap[t >> 5], bit) & bit) ds_set_error(status, DSPARK_EDUP);
  }
}

}  // namespace

extern "C" dspark_status dspark_d2t_check(const int64_t* d2t, int64_t V_d, int64_t V_t,
                                          int32_t require_injective, void* ws, size_t ws_bytes,
                                          int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(d2t && dev_status && V_d >= 1 && V_t >= 1 && V_t <= 0x7FFFFFFF);
  const size_t need = size_t(ds_ceil_div(V_t, 32)) * sizeof(uint32_t);
  if (require_injective) {
    if (!ws || ws_bytes < need || !ds_aligned(ws, 256)) return DSPARK_EWORKSPACE;
  }
  const int threads = 256;
  const unsigned blocks = unsigned(std::min<int64_t>(ds_ceil_div(V_d, threads), int64_t(ds_num_sms()) * 8));
  d2t_range_kernel<<<blocks, threads, 0, stream>>>(d2t, V_d, V_t, dev_status);
  if (require_injective) {
    DS_CUDA_TRY(cudaMemsetAsync(ws, 0, need, stream));
    d2t_dup_kernel<<<blocks, threads, 0, stream>>>(d2t, V_d, reinterpret_cast<uint32_t*>(ws), dev_status);
  }
  return ds_launch_status();
}

// ------------------------------------------------------------------------------------------------
// Allocation-free variant. Some callers cannot hand the library a device workspace: runtimes that
// allocate nothing once serving has started, or hosts whose device memory belongs to another
// allocator. For them the duplicate bitmap is a static array in this library's device image,
// sized for target vocabularies of up to D2T_NOALLOC_MAX_VT ids (128 KB). Host code cannot use the
// array's name as a device address, so every call asks the runtime for the array's address in the
// context current at the call (a host-side query that allocates nothing; the first one on a
// device loads the module there). The bitmap is cleared on the caller's stream at every call;
// calls that overlap on the GPU share it and race.
// ------------------------------------------------------------------------------------------------
namespace {

constexpr int64_t D2T_NOALLOC_MAX_VT = int64_t(1) << 20;

__device__ __align__(256) uint32_t d2t_noalloc_bitmap[D2T_NOALLOC_MAX_VT / 32];

// The bitmap's device address in the current context, or nullptr.
uint32_t* d2t_noalloc_bitmap_ptr() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, d2t_noalloc_bitmap) != cudaSuccess || ptr == nullptr) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return static_cast<uint32_t*>(ptr);
}

}  // namespace

extern "C" dspark_status dspark_d2t_check_noalloc(const int64_t* d2t, int64_t V_d, int64_t V_t,
                                                  int32_t require_injective, int32_t* dev_status,
                                                  dspark_stream_t stream) {
  DS_REQUIRE(d2t && dev_status && V_d >= 1 && V_t >= 1);
  if (V_t > D2T_NOALLOC_MAX_VT) return DSPARK_EINVAL;
  uint32_t* bitmap = d2t_noalloc_bitmap_ptr();
  if (bitmap == nullptr) return DSPARK_ECUDA;
  const int threads = 256;
  const unsigned blocks = unsigned(std::min<int64_t>(ds_ceil_div(V_d, threads), int64_t(ds_num_sms()) * 8));
  d2t_range_kernel<<<blocks, threads, 0, stream>>>(d2t, V_d, V_t, dev_status);
  if (require_injective) {
    DS_CUDA_TRY(cudaMemsetAsync(bitmap, 0, size_t(ds_ceil_div(V_t, 32)) * sizeof(uint32_t), stream));
    d2t_dup_kernel<<<blocks, threads, 0, stream>>>(d2t, V_d, bitmap, dev_status);
  }
  return ds_launch_status();
}
