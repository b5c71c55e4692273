// rowsample.cuh - building blocks of the full-vocabulary row sampler (sample.cu), which the
// dense Markov walk and verification reuse.
//
// Sums of weights: each thread adds the weights of its elements with the error-free 2Sum
// transformation in float32 pairs (about 48 significant bits). A double operation costs about as
// much as 64 float32 ones on this part (its FP64 pipe is narrow), so per-element and running sums
// stay in float pairs; the row sampler converts block totals to double, the draws of the dense walk
// and of verification keep float pairs to the decision (pick_cell, warp_pick). The float pairs keep
// the running sums within ~1e-14 of the exact value, far below the spacing of any decision.
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

// ---- float-pair decisions ---------------------------------------------------------------------
// A double operation costs about as much as 64 float32 ones on this part, so the running sums and
// comparisons that pick a token are float pairs; a comparison is right unless the two values agree
// to about 2^-48 relative, where a double sum in another order could fall either way as well.

// a - b as one float, whose sign is the sign of the difference (2Sum on the leading terms)
DS_DEV float ff_diff(const FF& a, const FF& b) {
  const float s = __fsub_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(-b.hi, bb));
  return __fadd_rn(s, __fadd_rn(err, __fsub_rn(a.lo, b.lo)));
}
DS_DEV FF ff_neg(const FF& a) { return FF{-a.hi, -a.lo}; }
// a * b as a float pair (the leading product's error from an FMA)
DS_DEV FF ff_mul(const FF& a, const FF& b) {
  const float p = __fmul_rn(a.hi, b.hi);
  const float e = __fmaf_rn(a.hi, b.hi, -p);
  const float t = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, e));
  const float s = __fadd_rn(p, t);
  return FF{s, __fsub_rn(t, __fsub_rn(s, p))};
}
// The uniform m * 2^-53 of ds_uniform as a float pair: the top 24 bits of m exactly, the other 29
// rounded to 24 (within 2^-49 of the double).
DS_DEV FF ff_uniform(uint64_t seed, uint64_t step, uint32_t position, uint32_t purpose, uint32_t draw = 0) {
  const uint64_t m = ds_uniform_bits(seed, step, position, purpose, draw);
  return FF{__fmul_rn(__uint2float_rn(uint32_t(m >> 29)), 0x1p-24f),
            __fmul_rn(__uint2float_rn(uint32_t(m & 0x1FFFFFFFull)), 0x1p-53f)};
}

// Shared state of pick_cell.
template <int NTHREADS>
struct PickShared {
  FF wsum[NTHREADS / 32];
  FF total, tau;
  unsigned long long cell;   // the crossing cell (~0 when none)
  int tinf;                  // rounding fallback: the last cell with mass, every running sum below tau
};

// Whole block: the cell whose running sum first exceeds target = u * total over `ncell` float-pair
// cell masses (each thread a contiguous run of cells), and tau = target minus the mass before it.
// Without such a cell (rounding), the last cell with mass and tinf.
template <int NTHREADS>
DS_DEV void pick_cell(const float2* cells, int64_t ncell, const FF& u, PickShared<NTHREADS>& s) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (ncell + NTHREADS - 1) / NTHREADS;
  const int64_t c0 = min(ncell, tid * per), c1 = min(ncell, c0 + per);
  FF mf{0.0f, 0.0f};
  for (int64_t c = c0; c < c1; ++c) {
    const float2 cv = __ldcg(cells + c);
    ff_acc(mf, FF{cv.x, cv.y});
  }
  FF incl = mf;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF nb{__shfl_up_sync(0xFFFFFFFFu, incl.hi, o), __shfl_up_sync(0xFFFFFFFFu, incl.lo, o)};
    if (lane >= o) ff_acc(incl, nb);
  }
  FF before{__shfl_up_sync(0xFFFFFFFFu, incl.hi, 1), __shfl_up_sync(0xFFFFFFFFu, incl.lo, 1)};
  if (lane == 0) before = FF{0.0f, 0.0f};
  if (lane == 31) s.wsum[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    FF run{0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < NTHREADS / 32; ++w) {
      const FF x = s.wsum[w];
      s.wsum[w] = run;
      ff_acc(run, x);
    }
    s.total = run;
    s.cell = ~0ull;
    s.tinf = 0;
  }
  __syncthreads();
  ff_acc(before, s.wsum[warp]);
  const FF target = ff_mul(u, s.total);
  FF end = before;
  ff_acc(end, mf);
  if (mf.hi > 0.0f && ff_diff(target, before) >= 0.0f && ff_diff(target, end) < 0.0f) {
    FF acc = before;
    for (int64_t c = c0; c < c1; ++c) {
      const float2 cv = __ldcg(cells + c);
      FF nxt = acc;
      ff_acc(nxt, FF{cv.x, cv.y});
      if (cv.x > 0.0f && ff_diff(target, nxt) < 0.0f) {
        atomicMin(&s.cell, static_cast<unsigned long long>(c));
        break;
      }
      acc = nxt;
    }
  }
  __syncthreads();
  if (s.cell != ~0ull && int64_t(s.cell) >= c0 && int64_t(s.cell) < c1) {   // the owner: tau
    FF acc = before;
    for (int64_t c = c0; c < int64_t(s.cell); ++c) {
      const float2 cv = __ldcg(cells + c);
      ff_acc(acc, FF{cv.x, cv.y});
    }
    FF tau = target;
    ff_acc(tau, ff_neg(acc));
    s.tau = tau;
  }
  if (tid == 0 && s.cell == ~0ull) {                   // rounding: the last cell with mass
    for (int64_t c = ncell - 1; c >= 0; --c) {
      if (__ldcg(cells + c).x > 0.0f) {
        s.cell = static_cast<unsigned long long>(c);
        s.tinf = 1;
        break;
      }
    }
  }
  __syncthreads();
}

// One warp: lane l holds the N masses v[e] of indices base + N l + e (in index order). The first
// index whose running sum exceeds tau; with tinf, or when no running sum does, the last index with
// mass; -1 when there is none. Every lane gets the result.
template <int N>
DS_DEV int64_t warp_pick(const FF (&v)[N], const FF& tau, bool tinf, int64_t base) {
  static_assert(N <= 32, "one bit per mass");
  const int lane = threadIdx.x & 31;
  FF ls{0.0f, 0.0f};
#pragma unroll
  for (int e = 0; e < N; ++e) ff_acc(ls, v[e]);
  FF li = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF nb{__shfl_up_sync(0xFFFFFFFFu, li.hi, o), __shfl_up_sync(0xFFFFFFFFu, li.lo, o)};
    if (lane >= o) ff_acc(li, nb);
  }
  FF lx{__shfl_up_sync(0xFFFFFFFFu, li.hi, 1), __shfl_up_sync(0xFFFFFFFFu, li.lo, 1)};
  if (lane == 0) lx = FF{0.0f, 0.0f};
  const bool has = ls.hi > 0.0f;
  const unsigned withm = __ballot_sync(0xFFFFFFFFu, has);
  const int lastl = withm ? 31 - __clz(int(withm)) : -1;
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, !tinf && has && ff_diff(tau, lx) >= 0.0f && ff_diff(tau, li) < 0.0f);
  const int hl = hit ? __ffs(int(hit)) - 1 : lastl;
  int64_t pick = -1;
  if (lane == hl) {
    FF run = lx;
    uint32_t gt = 0u, nz = 0u;
#pragma unroll
    for (int e = 0; e < N; ++e) {
      ff_acc(run, v[e]);
      gt |= uint32_t(!tinf && ff_diff(run, tau) > 0.0f) << e;
      nz |= uint32_t(v[e].hi > 0.0f) << e;
    }
    gt &= nz;
    const int64_t b = base + int64_t(N) * lane;
    pick = gt ? b + (__ffs(int(gt)) - 1) : (nz ? b + (31 - __clz(int(nz))) : -1);
  }
  return hl >= 0 ? __shfl_sync(0xFFFFFFFFu, pick, hl) : -1;
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
  float mult, softcap, T, top_p, min_p;
  const float* T_r;          // [requests] per-request temperature (<= 0: greedy), or null
  const float* top_p_r;      // [requests] per-request top-p, or null
  const float* min_p_r;      // [requests] per-request min-p, or null
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
  // top-p rows: a block's scratch row for the weights of its row's vectors (block b at
  // wscr + b * wscr_ld), so the nucleus passes after the first read them instead of recomputing
  // them; null: recomputed
  float* wscr;
  int64_t wscr_ld;
};

// Launches the row sampler (defined in sample.cu).
cudaError_t sample_rows(const SampleArgs& a, int64_t rows, int is_bf16, int xform, cudaStream_t stream);

}  // namespace rs
