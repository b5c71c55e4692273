// host_common.h - argument checks and launch helpers for the libdspark entry points.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <utility>
#include <stdint.h>

#include "../../include/dspark.h"

#define DS_REQUIRE(cond)                 \
  do {                                   \
    if (!(cond)) return DSPARK_EINVAL;   \
  } while (0)

#define DS_CUDA_TRY(expr)                        \
  do {                                           \
    if ((expr) != cudaSuccess) {                 \
      (void)cudaGetLastError();                  \
      return DSPARK_ECUDA;                       \
    }                                            \
  } while (0)

static inline dspark_status ds_launch_status() {
  return (cudaGetLastError() == cudaSuccess) ? DSPARK_OK : DSPARK_ECUDA;
}

static inline int ds_dtype_size(dspark_dtype d) { return d == DSPARK_BF16 ? 2 : 4; }
static inline bool ds_dtype_ok(dspark_dtype d) { return d == DSPARK_BF16 || d == DSPARK_F32; }

static inline int64_t ds_ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static inline bool ds_aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Poll limit of the first wait for a tile's tensor-core MMAs (lattice and dense walk); lowered only
// by the test hook dspark_test_set_first_wait_polls.
extern std::atomic<uint32_t> g_ds_first_wait_polls;

// Streaming multiprocessors of the current device (cached per device; thread-safe).
int ds_num_sms();

// Raises `func`'s dynamic shared-memory limit on the current device to at least `bytes` (each
// (device, kernel) pair is configured once; thread-safe). Kernel attributes are per device, so a
// process driving several GPUs, or calling from several threads, configures each one it uses.
cudaError_t ds_ensure_smem(const void* func, size_t bytes);

// Launches `kern` on `stream` with programmatic stream serialization: it may start while the
// previous kernel on the stream is still running (see ds_pdl_trigger / ds_pdl_wait).
template <typename... KArgs, typename... Args>
static inline cudaError_t ds_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
