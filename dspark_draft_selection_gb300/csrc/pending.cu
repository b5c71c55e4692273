// pending.cu - entry points whose kernels are not built yet; they refuse every call.
#include "dspark_common.cuh"
#include "host_common.h"

extern "C" size_t dspark_internal_ws_sample(int64_t, int32_t, int64_t) { return 0; }
extern "C" size_t dspark_internal_ws_dense_walk(int64_t, int32_t, int64_t) { return 0; }
extern "C" size_t dspark_internal_ws_verify(int64_t, int32_t, int64_t) { return 0; }

extern "C" dspark_status dspark_sample(const void*, dspark_dtype, int64_t, int32_t, int64_t, int64_t,
                                       const int64_t*, const int64_t*, int64_t, float, float, float,
                                       float, const uint64_t*, const uint64_t*, int32_t*, int32_t*,
                                       const dspark_qrecord*, void*, size_t, int32_t*, dspark_stream_t) {
  return DSPARK_EINVAL;
}
extern "C" dspark_status dspark_dense_walk(const void*, dspark_dtype, int64_t, int32_t, int64_t, int64_t,
                                           const int64_t*, const int32_t*, const void*, const void*,
                                           dspark_dtype, int32_t, int64_t, const int64_t*, const void*,
                                           const void*, dspark_dtype, int32_t, int64_t, float, float,
                                           float, float, const uint64_t*, const uint64_t*, int32_t*,
                                           int32_t*, const dspark_qrecord*, void*, size_t, int32_t*,
                                           dspark_stream_t) {
  return DSPARK_EINVAL;
}
extern "C" dspark_status dspark_verify(const void*, dspark_dtype, int64_t, int32_t, int64_t, int64_t,
                                       const int64_t*, const int32_t*, const int32_t*,
                                       const dspark_qrecord*, int64_t, float, float, const uint64_t*,
                                       const uint64_t*, int32_t*, int32_t*, float*, void*, size_t,
                                       int32_t*, dspark_stream_t) {
  return DSPARK_EINVAL;
}
