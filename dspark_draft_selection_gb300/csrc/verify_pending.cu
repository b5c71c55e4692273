// verify_pending.cu - dspark_verify until its kernels land: refuses every call.
#include "dspark_common.cuh"
#include "host_common.h"

extern "C" size_t dspark_internal_ws_verify(int64_t, int32_t, int64_t) { return 0; }
extern "C" dspark_status dspark_verify(const void*, dspark_dtype, int64_t, int32_t, int64_t, int64_t,
                                       const int64_t*, const int32_t*, const int32_t*,
                                       const dspark_qrecord*, int64_t, float, float, const uint64_t*,
                                       const uint64_t*, int32_t*, int32_t*, float*, void*, size_t,
                                       int32_t*, dspark_stream_t) {
  return DSPARK_EINVAL;
}
