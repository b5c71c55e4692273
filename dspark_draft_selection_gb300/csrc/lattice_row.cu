// lattice_row.cu - the block sampler's lattice-row branch (dspark_lattice_row_sample).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"), block-sampler commit: a greedy request whose logit processors
// keep the argmax walks the lattice greedily, a sampled one walks it with its draft RNG, and any
// other request samples the lattice row after the token before, ending the block at a token
// outside the candidates. Here that row is the whole draft vocabulary's transformed row with every
// candidate's entry replaced by its walk value fl32(u_j[b] + A_j[prev, b]) (position 0: A_0's row
// 0), drawn like a full-row multinomial request.
//
// Per position j, in stream order:
//  1. lr_copy_kernel - the transformed logits of every request still drafting into a float32 row
//     of the workspace (HBM streaming, 16-byte loads where aligned);
//  2. lr_patch_kernel - the K candidates' walk values over it; requests whose block has ended get
//     empty outputs at j;
//  3. the row sampler of sample.cu on those rows (temperature, top-p, min-p, Philox draw at
//     position j, q record, d2t), skipping ended requests;
//  4. lr_end_kernel - the drawn index's rank among position j's candidates becomes the previous
//     rank, or, when the index is not a candidate, the block ends at j + 1.
#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int LR_THREADS = 256;

struct LrArgs {
  const void* logits;
  int64_t ld;
  const int64_t* row_start;
  int32_t B, K, j;
  int64_t V;
  const int32_t* cand_draft;   // [R, B, K]
  const float* cand_val;       // [R, B, K]
  const float* trans;          // [R, B, K, K]
  float mult, softcap;
  float* zw;                   // [R, V] the rows to sample
  int32_t* act;                // [R] 0 while the block is drafting, -1 once it has ended
  int32_t* prev_rank;          // [R]
  int32_t* out_tgt;            // [R, B]
  int32_t* out_idx;            // [R, B]
  int32_t* n_drafted;          // [R]
  int32_t* q_n;                // [R * B] sparse record counts, or null
};

__global__ void lr_init_kernel(int32_t* act, int32_t* prev_rank, int32_t* n_drafted, int32_t B, int64_t R) {
  ds_pdl_trigger();
  ds_pdl_wait();
  for (int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; r < R; r += int64_t(gridDim.x) * blockDim.x) {
    act[r] = 0;
    prev_rank[r] = 0;
    n_drafted[r] = B;
  }
}

template <typename T, bool XFORM>
DS_DEV float lr_xform(const T* p, float mult, float softcap) {
  float x = ds_load_elem<T>(p);
  if (XFORM) {
    if (mult != 1.0f) x = __fmul_rn(x, mult);
    if (softcap > 0.0f) x = __fmul_rn(softcap, tanhf(__fdiv_rn(x, softcap)));
  }
  return x;
}

// grid (parts, R): part p of request r's row j
template <typename T, bool XFORM>
__global__ void __launch_bounds__(LR_THREADS) lr_copy_kernel(const LrArgs a) {
  ds_pdl_trigger();
  ds_pdl_wait();                                   // act comes from the last position's end kernel
  const int64_t r = blockIdx.y;
  if (a.act[r] < 0) return;
  const T* row = reinterpret_cast<const T*>(a.logits) + (a.row_start ? a.row_start[r] + a.j : r * a.B + a.j) * a.ld;
  float* z = a.zw + r * a.V;
  for (int64_t i = blockIdx.x * int64_t(LR_THREADS) + threadIdx.x; i < a.V; i += int64_t(gridDim.x) * LR_THREADS)
    z[i] = lr_xform<T, XFORM>(row + i, a.mult, a.softcap);
}

// one block per request: the candidates' walk values, or the empty outputs of an ended block
__global__ void __launch_bounds__(64) lr_patch_kernel(const LrArgs a) {
  ds_pdl_trigger();
  ds_pdl_wait();
  const int64_t r = blockIdx.x;
  const int64_t slot = r * a.B + a.j;
  if (a.act[r] < 0) {
    if (threadIdx.x == 0) {
      a.out_tgt[slot] = -1;
      a.out_idx[slot] = -1;
      if (a.q_n) a.q_n[slot] = 0;
    }
    return;
  }
  const int64_t cb = (r * a.B + a.j) * a.K;
  const float* Arow = a.trans + (cb * a.K) + (a.j == 0 ? 0 : int64_t(a.prev_rank[r]) * a.K);
  for (int b = threadIdx.x; b < a.K; b += blockDim.x) {
    const int32_t i = a.cand_draft[cb + b];
    if (i >= 0 && i < a.V) a.zw[r * a.V + i] = __fadd_rn(a.cand_val[cb + b], Arow[b]);
  }
}

// one thread per request: the drawn index's candidate rank, or the end of the block
__global__ void lr_end_kernel(const LrArgs a, int64_t R) {
  ds_pdl_trigger();
  ds_pdl_wait();                                   // the drawn indices come from the row sampler
  const int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (r >= R || a.act[r] < 0) return;
  const int32_t tok = a.out_idx[r * a.B + a.j];
  const int32_t* c = a.cand_draft + (r * a.B + a.j) * a.K;
  int rank = -1;
  for (int b = 0; b < a.K && rank < 0; ++b)
    if (c[b] == tok) rank = b;
  if (rank >= 0) {
    a.prev_rank[r] = rank;
  } else {
    a.act[r] = -1;
    a.n_drafted[r] = a.j + 1;
  }
}

size_t lr_align(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" size_t dspark_internal_ws_lattice_row(int64_t R, int32_t B, int64_t V) {
  return lr_align(size_t(R) * size_t(V) * sizeof(float)) + 2 * lr_align(size_t(R) * sizeof(int32_t)) +
         lr_align(size_t(R) * size_t(B) * sizeof(int32_t));
}

extern "C" dspark_status dspark_lattice_row_sample(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                                                   int64_t V_d, int64_t ld, const int64_t* row_start,
                                                   const int32_t* cand_draft, const float* cand_val, const float* trans,
                                                   int32_t K, const int64_t* d2t, int64_t V_t, float mult,
                                                   float softcap, float temperature, float top_p, float min_p,
                                                   const uint64_t* seed, const uint64_t* step, int32_t* out_tgt,
                                                   int32_t* out_idx, int32_t* n_drafted, const dspark_qrecord* q,
                                                   void* ws, size_t ws_bytes, int32_t* dev_status,
                                                   dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype) && R >= 0 && B >= 1 && B <= 100 && V_d >= 1 && ld >= V_d && V_d <= 0x7FFFFFFF);
  DS_REQUIRE(K >= 1 && K <= 64 && K <= V_d && R * B <= 0x7FFFFFFF);
  DS_REQUIRE(logits && cand_draft && cand_val && trans && out_tgt && n_drafted && dev_status &&
             ds_aligned(logits, ds_dtype_size(dtype)));
  DS_REQUIRE(temperature == temperature && top_p == top_p && top_p > 0.0f && min_p >= 0.0f && min_p <= 1.0f);
  DS_REQUIRE(mult == mult && softcap == softcap && softcap >= 0.0f);
  if (temperature > 0.0f) DS_REQUIRE(seed && step);
  if (d2t) DS_REQUIRE(V_t >= 1);
  const int C = rs::cluster_size_for(V_d, 4);
  DS_REQUIRE(C > 0);
  if (R == 0) return DSPARK_OK;
  const size_t need = dspark_internal_ws_lattice_row(R, B, V_d);
  if (!ws || ws_bytes < need || !ds_aligned(ws, 256)) return DSPARK_EWORKSPACE;
  uint8_t* p = reinterpret_cast<uint8_t*>(ws);
  LrArgs a = {};
  a.zw = reinterpret_cast<float*>(p);
  p += lr_align(size_t(R) * size_t(V_d) * sizeof(float));
  a.act = reinterpret_cast<int32_t*>(p);
  p += lr_align(size_t(R) * sizeof(int32_t));
  a.prev_rank = reinterpret_cast<int32_t*>(p);
  p += lr_align(size_t(R) * sizeof(int32_t));
  a.out_idx = out_idx ? out_idx : reinterpret_cast<int32_t*>(p);
  a.logits = logits;
  a.ld = ld;
  a.row_start = row_start;
  a.B = B;
  a.K = K;
  a.V = V_d;
  a.cand_draft = cand_draft;
  a.cand_val = cand_val;
  a.trans = trans;
  a.mult = mult;
  a.softcap = softcap;
  a.out_tgt = out_tgt;
  a.n_drafted = n_drafted;

  rs::SampleArgs sa = {};
  sa.rows = a.zw;
  sa.V = V_d;
  sa.ld = V_d;
  sa.row_mul = 1;
  sa.B = 1;                                        // one row per request, its status in act
  sa.C = C;
  sa.mult = 1.0f;                                  // the rows are already transformed
  sa.softcap = 0.0f;
  sa.T = temperature;
  sa.top_p = top_p;
  sa.min_p = min_p;
  sa.seed = seed;
  sa.step = step;
  sa.d2t = d2t;
  sa.V_t = V_t;
  sa.out_tgt = out_tgt;
  sa.out_idx = a.out_idx;
  sa.out_mul = B;
  sa.n_draft = a.act;                              // -1: the request's block has ended
  sa.status = dev_status;
  if (q) {
    sa.q = *q;
    sa.q_row_mul = B;
    if (q->z) {
      DS_REQUIRE(q->zmax && q->wsum && q->wcut && q->icut && q->ldz >= V_d);
      sa.q_mode = 2;
      sa.write_z = 1;
    } else {
      DS_REQUIRE(q->ids && q->p && q->n && q->cap >= 1);
      sa.q_mode = 1;
      a.q_n = q->n;
    }
  }
  cudaStream_t st = stream;
  DS_CUDA_TRY(ds_launch(lr_init_kernel, dim3(unsigned((R + 255) / 256)), dim3(256), 0, st, a.act, a.prev_rank,
                        n_drafted, B, R));
  const bool xform = (mult != 1.0f) || (softcap > 0.0f);
  const unsigned parts = unsigned(std::max<int64_t>(1, std::min<int64_t>(ds_ceil_div(V_d, 8 * LR_THREADS),
                                                                         int64_t(ds_num_sms()) * 4 / std::max<int64_t>(R, 1) + 1)));
  for (int32_t j = 0; j < B; ++j) {
    a.j = j;
    if (dtype == DSPARK_BF16)
      DS_CUDA_TRY(xform ? ds_launch(lr_copy_kernel<__nv_bfloat16, true>, dim3(parts, unsigned(R)), dim3(LR_THREADS), 0, st, a)
                        : ds_launch(lr_copy_kernel<__nv_bfloat16, false>, dim3(parts, unsigned(R)), dim3(LR_THREADS), 0, st, a));
    else
      DS_CUDA_TRY(xform ? ds_launch(lr_copy_kernel<float, true>, dim3(parts, unsigned(R)), dim3(LR_THREADS), 0, st, a)
                        : ds_launch(lr_copy_kernel<float, false>, dim3(parts, unsigned(R)), dim3(LR_THREADS), 0, st, a));
    DS_CUDA_TRY(ds_launch(lr_patch_kernel, dim3(unsigned(R)), dim3(64), 0, st, a));
    sa.position = j;
    sa.out_add = j;
    sa.q_row_add = j;
    DS_CUDA_TRY(rs::sample_rows(sa, R, 0, 0, st));
    DS_CUDA_TRY(ds_launch(lr_end_kernel, dim3(unsigned((R + 127) / 128)), dim3(128), 0, st, a, R));
  }
  return DSPARK_OK;
}
