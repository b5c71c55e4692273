// api.cu - library-wide entry points: workspace sizes and status names.
#include "dspark_common.cuh"
#include "host_common.h"

// Per-op workspace layouts are defined next to their kernels; these sizes must cover them.
extern "C" size_t dspark_internal_ws_sample(int64_t R, int32_t B, int64_t V);
extern "C" size_t dspark_internal_ws_dense_walk(int64_t R, int32_t B, int64_t V);
extern "C" size_t dspark_internal_ws_verify(int64_t R, int32_t B, int64_t V);

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
