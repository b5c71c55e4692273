// dense_walk.cu - dense Markov walk, markov_head_top_k = 0 (dspark_dense_walk).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"), Change > Markov heads: the dense Markov walk corrects every
// drafted position with one head inference per position; block-sampler commit: a dense step
// biases the scaled rows by the token drafted before, greedy takes the best biased token.
// optimum-intel PR #2099 ("... DSpark drafts with a pruned vocabulary"), Markov head: the
// next-token table is over the target vocabulary, so draft index i reads row i + d2t[i].
//
// Per position j (B positions run in sequence; position j + 1 needs the token drawn at j):
//  1. dense_walk_gemm_kernel - persistent CTAs sweep the draft vocabulary in 128-row tiles:
//     W rows m(i) are gathered into the 128-byte swizzled K-major layout and multiplied on the
//     tensor cores (tcgen05.mma, M = 128 vocabulary rows, N = requests padded to 16, K = rank)
//     against E[prev_r] of every request, which each CTA stages once. The epilogue reads the
//     accumulators from TMEM and writes z = (s + gamma * tau) / T for every (request, index):
//     straight into the dense proposal record when one is kept, else into the workspace.
//  2. the row sampler of sample.cu over those z rows (argmax when greedy), which also writes the
//     token back as the next position's previous token.
#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int DW_THREADS = 128;
constexpr int DW_M = 128;
constexpr int DW_MAXR = 128;

struct DwArgs {
  const void* logits;
  int64_t ld;
  const int64_t* row_start;
  int32_t B, j, R, Npad, rank;
  int64_t V, V_t, ntiles;
  const int32_t* prev_cur;
  const __nv_bfloat16* E;
  const __nv_bfloat16* W;
  const int64_t* d2t;
  const float* gate;
  float mult, softcap, Tz;
  float* z;
  int64_t ldz, z_row_mul, z_row_add;
  int32_t* status;
  uint32_t first_wait;       // polls of the first MMA-completion wait of a tile
};

template <bool XFORM>
DS_DEV float dw_xform(float x, float mult, float softcap) {
  if (XFORM) {
    if (mult != 1.0f) x = __fmul_rn(x, mult);
    if (softcap > 0.0f) x = __fmul_rn(softcap, tanhf(__fdiv_rn(x, softcap)));
  }
  return x;
}

// gamma_{r,j} for every (request, position), and the first position's previous tokens
template <typename HT>
__global__ void __launch_bounds__(128) dense_walk_gate_kernel(const HT* hidden, const HT* g, int H, int64_t ldh,
                                                              const int64_t* row_start, int32_t B,
                                                              const int32_t* prev, int32_t* prev_cur, float* gate) {
  __shared__ float s_red[4];
  const int tile = blockIdx.x;
  const int r = tile / B, j = tile % B;
  float gamma = 1.0f;
  if (hidden != nullptr) {
    const int64_t hrow = row_start ? row_start[r] + j : int64_t(tile);
    gamma = ds_block_gate(hidden + hrow * ldh, g, H, s_red);
  }
  if (threadIdx.x == 0) {
    gate[tile] = gamma;
    if (j == 0) prev_cur[r] = prev[r];
  }
}

template <typename T, bool XFORM>
__global__ void __launch_bounds__(DW_THREADS, 1) dense_walk_gemm_kernel(const DwArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int32_t s_arow[DW_M];
  __shared__ int32_t s_prev[DW_MAXR];
  __shared__ float s_gate[DW_MAXR];
  __shared__ int64_t s_lrow[DW_MAXR];

  const int rank = a.rank, nkb = rank / 64, Npad = a.Npad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                          // nkb x [128 rows x 128 B]
  uint8_t* sB = base + nkb * (DW_M * 128);     // nkb x [Npad rows x 128 B]
  const uint32_t ncols = Npad <= 32 ? 32 : Npad <= 64 ? 64 : 128;

  if (warp == 0) ds_tmem_alloc(&s_tmem, ncols);
  if (threadIdx.x == 0) ds_mbar_init(&s_bar, 1);
  for (int r = threadIdx.x; r < Npad; r += DW_THREADS) {
    int32_t p = -1;
    if (r < a.R) {
      p = a.prev_cur[r];
      if (p < 0 || p >= a.V_t) {
        ds_set_error(a.status, DSPARK_ERANGE);
        p = -1;
      }
      s_gate[r] = a.gate[int64_t(r) * a.B + a.j];
      s_lrow[r] = a.row_start ? a.row_start[r] + a.j : int64_t(r) * a.B + a.j;
    }
    s_prev[r] = p;
  }
  __syncthreads();
  const int cpr = rank / 8;
  for (int t = threadIdx.x; t < Npad * cpr; t += DW_THREADS) {
    const int m = t / cpr, c = t % cpr, kb = c >> 3, cc = c & 7;
    uint8_t* dst = sB + kb * (Npad * 128) + m * 128 + ((cc ^ (m & 7)) << 4);
    const int32_t id = s_prev[m];
    if (id >= 0) ds_cp_async16(dst, a.E + int64_t(id) * rank + c * 8);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  ds_tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = ds_idesc_bf16_f32(DW_M, Npad);
  const T* logits = reinterpret_cast<const T*>(a.logits);
  uint32_t phase = 0;
  bool alive = true;

  for (int64_t tile = blockIdx.x; tile < a.ntiles && alive; tile += gridDim.x) {
    const int64_t i0 = tile * DW_M;
    for (int m = threadIdx.x; m < DW_M; m += DW_THREADS) {
      const int64_t i = i0 + m;
      int64_t t = -1;
      if (i < a.V) {
        t = a.d2t ? i + a.d2t[i] : i;
        if (t < 0 || t >= a.V_t) {
          ds_set_error(a.status, DSPARK_ERANGE);
          t = -1;
        }
      }
      s_arow[m] = int32_t(t);
    }
    __syncthreads();
    for (int t = threadIdx.x; t < DW_M * cpr; t += DW_THREADS) {
      const int m = t / cpr, c = t % cpr, kb = c >> 3, cc = c & 7;
      uint8_t* dst = sA + kb * (DW_M * 128) + m * 128 + ((cc ^ (m & 7)) << 4);
      const int32_t id = s_arow[m];
      if (id >= 0) ds_cp_async16(dst, a.W + int64_t(id) * rank + c * 8);
      else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    ds_cp_async_wait_all();
    ds_fence_proxy_async_smem();
    __syncthreads();
    ds_tc_fence_after();
    if (threadIdx.x == 0) {
      const uint32_t aaddr = ds_smem_addr(sA), baddr = ds_smem_addr(sB);
      for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const uint64_t ad = ds_smem_desc_sw128(aaddr + kb * (DW_M * 128) + s * 32);
          const uint64_t bd = ds_smem_desc_sw128(baddr + kb * (Npad * 128) + s * 32);
          ds_umma_f16(tmem, ad, bd, idesc, (kb | s) != 0);
        }
      }
      ds_umma_commit(&s_bar);
    }
    __syncwarp();
    bool ok = ds_mbar_wait(&s_bar, phase, a.first_wait);
    if (!ok) {
      ds_set_error(a.status, DSPARK_ETIMEOUT);
      (void)ds_mbar_wait(&s_bar, phase, DS_WAIT_LIMIT);  // let in-flight MMAs drain; the CTA stops
    }
    ok = __syncthreads_and(ok) != 0;                     // one verdict for the whole CTA
    alive = ok;
    phase ^= 1;
    ds_tc_fence_after();
    if (ok) {
      const int64_t i = i0 + warp * 32 + lane;
      for (int c0 = 0; c0 < Npad; c0 += 32) {
        float acc[32];
        ds_tmem_ld_32x32b_x32(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c0), acc);
        if (i < a.V) {
          // the 32 requests' logits first (read-only loads, all in flight together), then z
          float sv[32];
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int r = c0 + cc;
            sv[cc] = 0.0f;
            if (r < a.R) {
              if constexpr (sizeof(T) == 2) {
                sv[cc] = ds_bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(logits + s_lrow[r] * a.ld + i)));
              } else {
                sv[cc] = __ldg(reinterpret_cast<const float*>(logits + s_lrow[r] * a.ld + i));
              }
            }
          }
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int r = c0 + cc;
            if (r < a.R) {
              const float s = dw_xform<XFORM>(sv[cc], a.mult, a.softcap);
              const float v = __fmaf_rn(s_gate[r], acc[cc], s);
              a.z[(int64_t(r) * a.z_row_mul + a.z_row_add) * a.ldz + i] = ds_temper(v, a.Tz);
            }
          }
        }
      }
    }
    ds_tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) {
    ds_tc_fence_after();
    ds_tmem_dealloc(tmem, ncols);
  }
}

template <typename T, bool XFORM>
cudaError_t dw_launch_gemm(const DwArgs& a, cudaStream_t stream) {
  auto kern = dense_walk_gemm_kernel<T, XFORM>;
  const size_t smem = size_t(a.rank / 64) * (DW_M + a.Npad) * 128 + 1024;
  const cudaError_t e = ds_ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int per_sm = smem <= 110 * 1024 ? 2 : 1;
  const int64_t grid = std::min<int64_t>(a.ntiles, int64_t(ds_num_sms()) * per_sm);
  kern<<<unsigned(grid), DW_THREADS, smem, stream>>>(a);
  return cudaGetLastError();
}

size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" size_t dspark_internal_ws_dense_walk(int64_t R, int32_t B, int64_t V) {
  return ws_align(size_t(R) * B * sizeof(float)) + ws_align(size_t(R) * sizeof(int32_t)) +
         ws_align(size_t(std::min<int64_t>(R, DW_MAXR)) * V * sizeof(float));
}

extern "C" dspark_status dspark_dense_walk(const void* logits, dspark_dtype dtype, int64_t R, int32_t B, int64_t V_d,
                                           int64_t ld, const int64_t* row_start, const int32_t* prev, const void* E,
                                           const void* W, dspark_dtype table_dtype, int32_t rank, int64_t V_t,
                                           const int64_t* d2t, const void* hidden, const void* g,
                                           dspark_dtype hidden_dtype, int32_t H, int64_t ldh, float mult,
                                           float softcap, float temperature, float top_p, const uint64_t* seed,
                                           const uint64_t* step, int32_t* out_tgt, int32_t* out_idx,
                                           const dspark_qrecord* q, void* ws, size_t ws_bytes, int32_t* dev_status,
                                           dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype) && R >= 0 && B >= 1 && B <= 100 && V_d >= 1 && ld >= V_d);
  DS_REQUIRE(V_d <= 0x7FFFFFFF && V_t >= 1 && V_t <= 0x7FFFFFFF);
  DS_REQUIRE(logits && prev && E && W && out_tgt && dev_status && ds_aligned(logits, ds_dtype_size(dtype)));
  DS_REQUIRE(table_dtype == DSPARK_BF16 && rank % 64 == 0 && rank >= 64 && rank <= 256);
  DS_REQUIRE(ds_aligned(E, 16) && ds_aligned(W, 16));
  DS_REQUIRE(temperature == temperature && top_p == top_p && top_p > 0.0f && softcap >= 0.0f && mult == mult);
  if (!d2t) DS_REQUIRE(V_t >= V_d);
  if (temperature > 0.0f) DS_REQUIRE(seed && step);
  if (hidden) DS_REQUIRE(g && H >= 1 && ldh >= H && ds_dtype_ok(hidden_dtype));
  const bool record = q != nullptr;
  if (record) DS_REQUIRE(q->z && q->zmax && q->wsum && q->wcut && q->icut && q->ldz >= V_d);
  if (R == 0) return DSPARK_OK;
  const size_t need = dspark_internal_ws_dense_walk(R, B, V_d);
  if (!ws || ws_bytes < need || !ds_aligned(ws, 256)) return DSPARK_EWORKSPACE;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(ws);
  float* gate = reinterpret_cast<float*>(wsb);
  int32_t* prev_cur = reinterpret_cast<int32_t*>(wsb + ws_align(size_t(R) * B * sizeof(float)));
  float* zscr = reinterpret_cast<float*>(wsb + ws_align(size_t(R) * B * sizeof(float)) +
                                         ws_align(size_t(R) * sizeof(int32_t)));
  cudaStream_t st = stream;

  if (hidden && hidden_dtype == DSPARK_BF16)
    dense_walk_gate_kernel<__nv_bfloat16><<<unsigned(R * B), 128, 0, st>>>(
        reinterpret_cast<const __nv_bfloat16*>(hidden), reinterpret_cast<const __nv_bfloat16*>(g), H, ldh, row_start,
        B, prev, prev_cur, gate);
  else
    dense_walk_gate_kernel<float><<<unsigned(R * B), 128, 0, st>>>(
        reinterpret_cast<const float*>(hidden), reinterpret_cast<const float*>(g), H, ldh, row_start, B, prev,
        prev_cur, gate);
  DS_CUDA_TRY(cudaGetLastError());

  const bool xform = (mult != 1.0f) || (softcap > 0.0f);
  const int64_t Vs = V_d;
  const int Cz = rs::cluster_size_for(Vs, 4);
  DS_REQUIRE(Cz > 0);
  for (int64_t c0 = 0; c0 < R; c0 += DW_MAXR) {
    const int32_t Rc = int32_t(std::min<int64_t>(DW_MAXR, R - c0));
    DwArgs a = {};
    a.logits = reinterpret_cast<const uint8_t*>(logits) + (row_start ? 0 : c0 * B * ld * ds_dtype_size(dtype));
    a.ld = ld;
    a.row_start = row_start ? row_start + c0 : nullptr;
    a.B = B;
    a.R = Rc;
    a.Npad = ((Rc + 15) / 16) * 16;
    a.rank = rank;
    a.V = V_d;
    a.V_t = V_t;
    a.ntiles = (V_d + DW_M - 1) / DW_M;
    a.prev_cur = prev_cur + c0;
    a.E = reinterpret_cast<const __nv_bfloat16*>(E);
    a.W = reinterpret_cast<const __nv_bfloat16*>(W);
    a.d2t = d2t;
    a.gate = gate + c0 * B;
    a.mult = mult;
    a.softcap = softcap;
    a.Tz = temperature > 0.0f ? temperature : 1.0f;
    a.status = dev_status;
    a.first_wait = g_ds_first_wait_polls.load(std::memory_order_relaxed);
    if (record) {
      a.z = q->z + c0 * B * q->ldz;
      a.ldz = q->ldz;
      a.z_row_mul = B;
    } else {
      a.z = zscr;
      a.ldz = V_d;
      a.z_row_mul = 1;
    }
    rs::SampleArgs sa = {};
    sa.rows = a.z;
    sa.V = V_d;
    sa.ld = a.ldz;
    sa.row_mul = a.z_row_mul;
    sa.B = 1;
    sa.C = Cz;
    sa.mult = 1.0f;
    sa.softcap = 0.0f;
    sa.T = temperature > 0.0f ? 1.0f : 0.0f;     // the rows already hold z = v / T
    sa.top_p = top_p;
    sa.seed = seed ? seed + c0 : nullptr;
    sa.step = step ? step + c0 : nullptr;
    sa.d2t = d2t;
    sa.V_t = V_t;
    sa.out_tgt = out_tgt + c0 * B;
    sa.out_idx = out_idx ? out_idx + c0 * B : nullptr;
    sa.out_mul = B;
    sa.prev_out = prev_cur + c0;
    sa.status = dev_status;
    if (record) {
      sa.q = *q;
      sa.q.zmax = q->zmax + c0 * B;
      sa.q.wsum = q->wsum + c0 * B;
      sa.q.wcut = q->wcut + c0 * B;
      sa.q.icut = q->icut + c0 * B;
      sa.q_mode = 2;
      sa.q_row_mul = B;
    }
    for (int32_t j = 0; j < B; ++j) {
      a.j = j;
      a.z_row_add = record ? j : 0;
      cudaError_t e;
      if (dtype == DSPARK_BF16)
        e = xform ? dw_launch_gemm<__nv_bfloat16, true>(a, st) : dw_launch_gemm<__nv_bfloat16, false>(a, st);
      else
        e = xform ? dw_launch_gemm<float, true>(a, st) : dw_launch_gemm<float, false>(a, st);
      DS_CUDA_TRY(e);
      sa.row_base = record ? j : 0;
      sa.position = j;
      sa.out_add = j;
      sa.q_row_add = j;
      DS_CUDA_TRY(rs::sample_rows(sa, Rc, 0, 0, st));
    }
  }
  return DSPARK_OK;
}
