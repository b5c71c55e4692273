// conv.cu - DFlash-2 grouped dynamic convolution over packed block rows (dspark_grouped_conv).
//
// Method: optimum-intel PR #2098 ("Export DFlash v2 and DSpark drafts for PagedAttention and
// continuous batching"), What does this PR do > DFlash v2, and its commit on the per-row DFlash
// backbone: the grouped dynamic convolution of a DFlash-2 draft runs over the packed block rows
// of several requests, shifts its taps back along those rows and masks each tap to the block of
// the row it produces. openvino.genai PR #4847 (block sampler commit): every block follows at
// least one context row, which keeps the blocks of different requests apart in those rows.
//
//   y[i, c] = sum over t < L of k[i, g(c), t] * x[i - t, c], a tap counting only when row i - t
//             exists and belongs to row i's block; g(c) = c / (C / G).
//
// One thread produces eight consecutive channels of one row (16-byte loads of bf16 rows, two of
// float32 rows) and adds its taps in order t = 0, 1, ... with float32 FMAs. The rows a tap reads
// were read by the threads of the rows before, so apart from the taps every input byte comes from
// HBM once and every output byte goes there once: the kernel is bound by HBM bandwidth.
#include "dspark_common.cuh"
#include "host_common.h"

namespace {

constexpr int CV_THREADS = 256;
constexpr int CV_MAXL = 16;

template <typename T>
DS_DEV void cv_ld8(const T* p, float (&v)[8]) {
  if constexpr (sizeof(T) == 2) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = ds_vec_elem<T>(u, e);
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Vector path: C % 8 == 0, every group a multiple of eight channels, rows 16-byte aligned.
template <typename T>
__global__ void __launch_bounds__(CV_THREADS) conv_vec_kernel(const T* x, int64_t ldx, int64_t N, int64_t C,
                                                              int32_t G, int32_t L, const float* k,
                                                              const int32_t* block, float* y, int64_t ldy) {
  ds_pdl_trigger();
  ds_pdl_wait();                                     // the rows may come from the kernel before
  const int64_t nvec = C / 8;
  const int64_t gs = C / G;
  for (int64_t u = blockIdx.x * int64_t(CV_THREADS) + threadIdx.x; u < N * nvec; u += int64_t(gridDim.x) * CV_THREADS) {
    const int64_t i = u / nvec, c0 = (u - i * nvec) * 8;
    const int64_t g = c0 / gs;
    const int32_t bi = block[i];
    const float* ki = k + (i * G + g) * L;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int t = 0; t < L && t <= i; ++t) {
      if (block[i - t] != bi) continue;              // masked: another block's row
      const float kt = __ldg(ki + t);
      float v[8];
      cv_ld8<T>(x + (i - t) * ldx + c0, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = __fmaf_rn(kt, v[e], acc[e]);
    }
    float4* yo = reinterpret_cast<float4*>(y + i * ldy + c0);
    yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// Any shape: one thread per output element.
template <typename T>
__global__ void __launch_bounds__(CV_THREADS) conv_any_kernel(const T* x, int64_t ldx, int64_t N, int64_t C,
                                                              int32_t G, int32_t L, const float* k,
                                                              const int32_t* block, float* y, int64_t ldy) {
  ds_pdl_trigger();
  ds_pdl_wait();
  const int64_t gs = C / G;
  for (int64_t u = blockIdx.x * int64_t(CV_THREADS) + threadIdx.x; u < N * C; u += int64_t(gridDim.x) * CV_THREADS) {
    const int64_t i = u / C, c = u - i * C;
    const int32_t bi = block[i];
    const float* ki = k + (i * G + c / gs) * L;
    float acc = 0.0f;
    for (int t = 0; t < L && t <= i; ++t)
      if (block[i - t] == bi) acc = __fmaf_rn(__ldg(ki + t), ds_load_elem<T>(x + (i - t) * ldx + c), acc);
    y[i * ldy + c] = acc;
  }
}

}  // namespace

extern "C" dspark_status dspark_grouped_conv(const void* x, dspark_dtype dtype, int64_t N, int64_t C, int64_t ldx,
                                             int32_t G, int32_t L, const float* k, const int32_t* block, float* y,
                                             int64_t ldy, dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype) && N >= 0 && C >= 1 && ldx >= C && ldy >= C && G >= 1 && C % G == 0);
  DS_REQUIRE(L >= 1 && L <= CV_MAXL);
  if (N == 0) return DSPARK_OK;
  DS_REQUIRE(x && k && block && y && ds_aligned(x, ds_dtype_size(dtype)) && ds_aligned(y, 4) && ds_aligned(k, 4));
  const int esz = ds_dtype_size(dtype);
  const bool vec = C % 8 == 0 && (C / G) % 8 == 0 && ds_aligned(x, 16) && (ldx * esz) % 16 == 0 &&
                   ds_aligned(y, 16) && (ldy * 4) % 16 == 0;
  const int64_t work = vec ? N * (C / 8) : N * C;
  const unsigned grid = unsigned(std::max<int64_t>(1, std::min<int64_t>(ds_ceil_div(work, CV_THREADS), int64_t(ds_num_sms()) * 8)));
  cudaStream_t st = stream;
  if (dtype == DSPARK_BF16) {
    const __nv_bfloat16* xp = reinterpret_cast<const __nv_bfloat16*>(x);
    if (vec)
      DS_CUDA_TRY(ds_launch(conv_vec_kernel<__nv_bfloat16>, dim3(grid), dim3(CV_THREADS), 0, st, xp, ldx, N, C, G, L, k, block, y, ldy));
    else
      DS_CUDA_TRY(ds_launch(conv_any_kernel<__nv_bfloat16>, dim3(grid), dim3(CV_THREADS), 0, st, xp, ldx, N, C, G, L, k, block, y, ldy));
  } else {
    const float* xp = reinterpret_cast<const float*>(x);
    if (vec)
      DS_CUDA_TRY(ds_launch(conv_vec_kernel<float>, dim3(grid), dim3(CV_THREADS), 0, st, xp, ldx, N, C, G, L, k, block, y, ldy));
    else
      DS_CUDA_TRY(ds_launch(conv_any_kernel<float>, dim3(grid), dim3(CV_THREADS), 0, st, xp, ldx, N, C, G, L, k, block, y, ldy));
  }
  return DSPARK_OK;
}
