// rowsample.cuh - one-row-per-cluster building blocks for full-vocabulary sampling.
//
// A row of V elements is held in registers by a cluster of C CTAs x 512 threads. CTA c owns the
// contiguous vector chunk [c * nvc, (c + 1) * nvc) of the row's 16-byte vectors; thread t of
// CTA c holds the vectors c * nvc + k * 512 + t (k < MAXV, "round" k). Scalar elements before
// the first 16-byte boundary (head) sit on CTA 0, threads t < head; the ragged tail on CTA C-1,
// threads t < ntail. Index order therefore walks: head, CTA 0 rounds 0.., CTA 1 rounds 0.., ...,
// tail - which is how the draw's running sums are laid out.
//
// Sums of weights: each thread adds the weights of one vector with the error-free 2Sum
// transformation in float32 pairs (about 48 significant bits), then converts to double; every
// larger sum is in double. A double accumulation per element would run on the GPU's narrow
// FP64 pipe; the float pairs keep the running sums within ~1e-14 of the exact value, far below
// the spacing of any decision.
#pragma once

#include <cooperative_groups.h>

#include "dspark_common.cuh"

namespace cg = cooperative_groups;

namespace rs {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr int MAXV = 8;          // 16-byte vectors per thread
constexpr int MAXC = 16;         // CTAs per cluster
constexpr int SEGS = MAXV + 2;   // head, rounds, tail

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

// Geometry of one row as seen by this thread.
struct RowGeom {
  int64_t head, nvec, tail0, ntail, nvc;
  int C, crank;
  __device__ int64_t vec_index(int k) const {           // -1 when this thread has no round-k vector
    const int64_t v = int64_t(crank) * nvc + int64_t(k) * THREADS + threadIdx.x;
    const int64_t end = min(nvec, int64_t(crank + 1) * nvc);
    return v < end ? v : -1;
  }
  __device__ bool has_head() const { return crank == 0 && threadIdx.x < head; }
  __device__ bool has_tail() const { return crank == C - 1 && threadIdx.x < ntail; }
};

template <typename T>
DS_DEV RowGeom row_geom(const T* row, int64_t V, int C, int crank) {
  constexpr int EPV = 16 / sizeof(T);
  RowGeom g;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  g.head = int64_t(((16u - (addr & 15u)) & 15u) / sizeof(T));
  if (g.head > V) g.head = V;
  g.nvec = (V - g.head) / EPV;
  g.tail0 = g.head + g.nvec * EPV;
  g.ntail = V - g.tail0;
  g.nvc = (g.nvec + C - 1) / C;
  g.C = C;
  g.crank = crank;
  return g;
}

// Smallest power-of-two cluster that holds a V-element row within MAXV vectors per thread.
inline int cluster_size_for(int64_t V, int elem_bytes) {
  const int64_t epv = 16 / elem_bytes;
  const int64_t nvec = V / epv + 1;
  int C = 1;
  while (C <= MAXC && (nvec + C - 1) / C > int64_t(THREADS) * MAXV) C <<= 1;
  return C <= MAXC ? C : -1;
}

// ---- block reductions (all threads call; result valid in every thread) ------------------------
struct BlockScratch {
  double d[WARPS];
  float f[WARPS];
  unsigned long long u[WARPS];
  double seg[SEGS];
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

// ---- cluster reductions through the leader CTA's shared slots --------------------------------
// Every thread of every CTA calls these with its CTA's value (uniform control flow). Slots are
// double buffered: a CTA can be at most one reduction ahead of another, because every reduction
// ends with a cluster barrier.
struct ClusterRed {
  double d[2][MAXC];
  unsigned long long u[2][MAXC];
  double bd[2];
  unsigned long long bu;
  int phase;
};

DS_DEV void cred_init(ClusterRed& r) {
  if (threadIdx.x == 0) r.phase = 0;
}

// Sum over CTAs (op 0), max over CTAs (op 1), or exclusive prefix over CTA rank + total (op 2).
DS_DEV double cluster_sum_d(cg::cluster_group& cl, ClusterRed& r, double v, int op = 0, double* total = nullptr) {
  __syncthreads();
  const int ph = r.phase;
  double* lead = cl.map_shared_rank(&r.d[ph][0], 0);
  const int C = int(cl.num_blocks()), me = int(cl.block_rank());
  if (threadIdx.x == 0) lead[me] = v;
  cl.sync();
  if (threadIdx.x == 0) {
    double acc = (op == 1) ? -INFINITY : 0.0, before = 0.0;
    for (int c = 0; c < C; ++c) {
      const double x = lead[c];
      if (op == 1) acc = fmax(acc, x);
      else acc += x;
      if (c < me) before += x;
    }
    r.bd[0] = (op == 2) ? before : acc;
    r.bd[1] = acc;
    r.phase = ph ^ 1;
  }
  __syncthreads();
  if (total) *total = r.bd[1];
  return r.bd[0];
}

DS_DEV unsigned long long cluster_max_u64(cg::cluster_group& cl, ClusterRed& r, unsigned long long v) {
  __syncthreads();
  const int ph = r.phase;
  unsigned long long* lead = cl.map_shared_rank(&r.u[ph][0], 0);
  const int C = int(cl.num_blocks()), me = int(cl.block_rank());
  if (threadIdx.x == 0) lead[me] = v;
  cl.sync();
  if (threadIdx.x == 0) {
    unsigned long long acc = 0;
    for (int c = 0; c < C; ++c) acc = max(acc, lead[c]);
    r.bu = acc;
    r.phase = ph ^ 1;
  }
  __syncthreads();
  return r.bu;
}

// Arguments of the row sampler (dspark_sample, and the dense walk on its biased rows).
struct SampleArgs {
  const void* rows;
  int64_t V, ld;
  const int64_t* row_start;
  int64_t row_base, row_mul; // source row = row_base + row_id * row_mul when row_start is NULL
  int32_t B, C;
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
