// host_common.h - argument checks and launch helpers for the libdspark entry points.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
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

// Streaming multiprocessors of the current device (cached per device; thread-safe).
int ds_num_sms();

// Raises `func`'s dynamic shared-memory limit on the current device to at least `bytes` (each
// (device, kernel) pair is configured once; thread-safe). Kernel attributes are per device, so a
// process driving several GPUs, or calling from several threads, configures each one it uses.
cudaError_t ds_ensure_smem(const void* func, size_t bytes);
