// rowsample.cuh - building blocks of the full-vocabulary row sampler (sample.cu), which the
// dense Markov walk and verification reuse.
//
// Sums of weights: each thread adds the weights of its elements with the error-free 2Sum
// transformation in float32 pairs (about 48 significant bits), then converts to double; every
// larger sum is in double. A double accumulation per element would run on the GPU's narrow
// FP64 pipe; the float pairs keep the running sums within ~1e-14 of the exact value, far below
// the spacing of any decision.
#pragma once

#include "dspark_common.cuh"

namespace rs {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr int MAXVEC = 65536;    // 16-byte vectors per row (262,144 float32 or 524,288 bf16 elements)

// float pair (hi + lo) accumulator
struct FF {
  float hi, lo;
};
DS_DEV void ff_add(FF& a, float b) {
  const float s = __fadd_rn(a.hi, b);
  const float bb = __fsub_rn(s, a.hi);
  const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  a.hi = s;
  a.lo = __fadd_rn(a.lo, err);
}
DS_DEV double ff_value(const FF& a) { return double(a.hi) + double(a.lo); }
DS_DEV void ff_acc(FF& m, const FF& v) {   // m += v for float pairs
  const float lo = __fadd_rn(m.lo, v.lo);
  m.lo = 0.0f;
  ff_add(m, v.hi);
  m.lo = __fadd_rn(m.lo, lo);
}

// Two float-pair accumulators in packed float32 registers (lanes of the f32x2 operations): the
// same 2Sum steps as ff_add on two independent sums at once.
struct FF2 {
  uint64_t hi, lo;
};
DS_DEV void ff2_add(FF2& a, uint64_t b) {
  const uint64_t s = ds_add2(a.hi, b);
  const uint64_t bb = ds_sub2(s, a.hi);
  const uint64_t err = ds_add2(ds_sub2(a.hi, ds_sub2(s, bb)), ds_sub2(b, bb));
  a.hi = s;
  a.lo = ds_add2(a.lo, err);
}
// The two lanes folded into one float pair.
DS_DEV FF ff2_fold(const FF2& a) {
  FF r{ds_f2lo(a.hi), ds_f2lo(a.lo)};
  const float lo = __fadd_rn(r.lo, ds_f2hi(a.lo));
  r.lo = 0.0f;
  ff_add(r, ds_f2hi(a.hi));
  r.lo = __fadd_rn(r.lo, lo);
  return r;
}

// Sum of a float pair over a warp in float pairs (FP32 shuffles and 2Sum only; every lane gets
// it). The GPU's FP64 pipe is narrow, so callers convert the result once per warp, not per lane.
DS_DEV FF warp_ff_reduce(FF v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xFFFFFFFFu, v.hi, o), ol = __shfl_xor_sync(0xFFFFFFFFu, v.lo, o);
    const float lo = __fadd_rn(v.lo, ol);
    v.lo = 0.0f;
    ff_add(v, oh);
    v.lo = __fadd_rn(v.lo, lo);
  }
  return v;
}

// 1 when a V-element row is within the sampler's row length, else -1 (the row-length check the
// entry points make before any launch).
inline int cluster_size_for(int64_t V, int elem_bytes) {
  const int64_t epv = 16 / elem_bytes;
  return (V / epv + 1 <= int64_t(MAXVEC)) ? 1 : -1;
}

// ---- block reductions (all threads call; result valid in every thread) ------------------------
struct BlockScratch {
  double tot;
  double d[WARPS];
  float f[WARPS];
  unsigned long long u[WARPS];
};

DS_DEV double block_sum(double v, BlockScratch& s) {
  v = ds_warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.d[threadIdx.x >> 5] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) t += s.d[w];
  return t;
}
// Block sum of per-thread float pairs, as a double (warp sums in float pairs, one conversion per
// warp, the final 16 additions in one thread).
static __device__ __noinline__ double block_sum_ff(FF v, BlockScratch& s) {
  v = warp_ff_reduce(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.d[threadIdx.x >> 5] = ff_value(v);
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) t += s.d[w];
    s.tot = t;
  }
  __syncthreads();
  return s.tot;
}

// Block sum of per-thread counts (exact in 32 bits).
DS_DEV uint32_t block_count(uint32_t v, BlockScratch& s) {
  v = __reduce_add_sync(0xFFFFFFFFu, v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.u[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) t += uint32_t(s.u[w]);
  return t;
}

DS_DEV float block_max(float v, BlockScratch& s) {
  v = ds_warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.f[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = -INFINITY;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) t = fmaxf(t, s.f[w]);
  return t;
}
DS_DEV unsigned long long block_max_u64(unsigned long long v, BlockScratch& s) {
  v = ds_warp_max_u64(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s.u[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long t = 0;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) t = max(t, s.u[w]);
  return t;
}

// Exclusive prefix (in thread order) of a per-thread double, plus the block total.
DS_DEV double block_exclusive_scan(double v, double* total, BlockScratch& s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) s.d[warp] = incl;
  __syncthreads();
  double before = 0.0, all = 0.0;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) {
    if (w < warp) before += s.d[w];
    all += s.d[w];
  }
  *total = all;
  return before + incl - v;
}

// Arguments of the row sampler (dspark_sample, and the dense walk on its biased rows).
struct SampleArgs {
  const void* rows;
  int64_t V, ld;
  const int64_t* row_start;
  int64_t row_base, row_mul; // source row = row_base + row_id * row_mul when row_start is NULL
  int32_t B, C;              // C: 1 when the row length was checked by the caller
  float mult, softcap, T, top_p;
  const uint64_t* seed;
  const uint64_t* step;
  int32_t position;          // >= 0: counter position for every row; < 0: j = row_id % B
  const int64_t* d2t;
  int64_t V_t;
  int32_t* out_tgt;
  int32_t* out_idx;
  int64_t out_mul, out_add;  // output slot = row_id * out_mul + out_add
  int32_t* prev_out;         // dense walk: next position's previous token, per request
  dspark_qrecord q;
  int q_mode;                // 0 none, 1 sparse, 2 dense
  int write_z;
  int64_t q_row_mul, q_row_add;  // record row = row_id * mul + add
  // verification hooks: skip the draw; report the weight of a probed index and the argmax
  int no_draw;
  const int32_t* probe_tgt;      // [R, B - 1] drafted target ids probed in row j < n_draft[r]
  const int32_t* n_draft;        // [R]; rows j > n_draft[r] are skipped
  float* probe_w;                // [rows] weight of the probed id if kept, else 0
  int32_t* amax_out;             // [rows] argmax index (lowest on ties)
  int32_t* status;
};

// Launches the row sampler (defined in sample.cu).
cudaError_t sample_rows(const SampleArgs& a, int64_t rows, int is_bf16, int xform, cudaStream_t stream);

}  // namespace rs
