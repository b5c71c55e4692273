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
