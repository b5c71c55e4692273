// lattice.cu - Markov-head transition lattice (dspark_lattice_score).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"), Change > Markov heads (the Top-K scorer rates the candidates of
// neighbouring positions in one inference for all requests); optimum-intel PR #2098 ("Export
// DFlash v2 and DSpark drafts ..."), What does this PR do > DFlash v2 (packed Top-K lattice,
// transitions gated by the draft hidden states); optimum-intel PR #2099 ("... pruned
// vocabulary"), Markov head (the next-token table is indexed by target ids). Head form:
// tau(a, b) = E[a] . W[b]; gate gamma = sigmoid(h . g).
//
// One CTA per (request, position) tile. The candidate rows of E (previous position) and W
// (this position) are gathered from HBM with 16-byte cp.async straight into the 128-byte
// swizzled K-major shared-memory layout that tcgen05.mma reads; one thread issues the
// rank/16 MMAs (M = 128 with the unused A rows zeroed, N = 64, fp32 accumulators in TMEM);
// four warps read the 128 x 64 accumulator tile back with tcgen05.ld, scale it by the
// gate and store it. float32 tables (or ranks the tensor-core layout does not take) use a
// CUDA-core FMA kernel instead.
#include "dspark_common.cuh"
#include "host_common.h"

namespace {

constexpr int LT_THREADS = 128;
constexpr int LT_M = 128;      // MMA rows (A: previous candidates, zero-padded)
constexpr int LT_N = 64;       // MMA columns (B: this position's candidates, zero-padded)

struct LatticeArgs {
  const int32_t* cand_tgt;
  const int32_t* prev;
  int32_t B, K, rank, H;
  const void* E;
  const void* W;
  int64_t V_t;
  const void* hidden;
  const void* g;
  int64_t ldh;
  const int64_t* row_start;
  float* trans;
  float* gate;
  int32_t* status;
  int hidden_bf16;
};

DS_DEV float lt_gate_any(const LatticeArgs& a, int64_t hrow, float* s_red) {
  if (a.hidden == nullptr) return 1.0f;
  if (a.hidden_bf16)
    return ds_block_gate(reinterpret_cast<const __nv_bfloat16*>(a.hidden) + hrow * a.ldh,
                         reinterpret_cast<const __nv_bfloat16*>(a.g), a.H, s_red);
  return ds_block_gate(reinterpret_cast<const float*>(a.hidden) + hrow * a.ldh, reinterpret_cast<const float*>(a.g),
                       a.H, s_red);
}

// ---------------------------------------------------------------------------------------
// tensor-core path: bf16 tables, rank % 64 == 0, rank <= 512
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(LT_THREADS) lattice_tc_kernel(const LatticeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int32_t s_ida[LT_M];
  __shared__ int32_t s_idb[LT_N];
  __shared__ float s_red[LT_THREADS / 32];

  const int tile = blockIdx.x;                       // r * B + j
  const int r = tile / a.B, j = tile % a.B;
  const int K = a.K, rank = a.rank;
  const int nkb = rank / 64;                         // 64-element (128-byte) K chunks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                                // nkb x [128 rows x 128 B]
  uint8_t* sB = base + nkb * (LT_M * 128);           // nkb x [ 64 rows x 128 B]

  if (warp == 0) ds_tmem_alloc(&s_tmem, 64);
  if (threadIdx.x == 0) ds_mbar_init(&s_bar, 1);

  const int Ka = (j == 0) ? 1 : K;
  const int32_t* ct = a.cand_tgt + int64_t(tile) * K;
  for (int i = threadIdx.x; i < LT_M; i += LT_THREADS) {
    int32_t id = -1;
    if (i < Ka) id = (j == 0) ? a.prev[r] : ct[i - K];  // previous position's candidates
    if (i < Ka && (id < 0 || id >= a.V_t)) {
      ds_set_error(a.status, DSPARK_ERANGE);
      id = -1;
    }
    s_ida[i] = id;
  }
  for (int i = threadIdx.x; i < LT_N; i += LT_THREADS) {
    int32_t id = (i < K) ? ct[i] : -1;
    if (i < K && (id < 0 || id >= a.V_t)) {
      ds_set_error(a.status, DSPARK_ERANGE);
      id = -1;
    }
    s_idb[i] = id;
  }
  __syncthreads();

  // gather rows into the swizzled K-major layout: row m, 16-byte chunk c of K-chunk kb lives at
  // kb * (rows * 128) + m * 128 + ((c ^ (m & 7)) * 16)
  const int cpr = rank / 8;                          // 16-byte chunks per table row
  const __nv_bfloat16* E = reinterpret_cast<const __nv_bfloat16*>(a.E);
  const __nv_bfloat16* W = reinterpret_cast<const __nv_bfloat16*>(a.W);
  // rows past Ka (A) and K (B) only feed accumulator rows/columns that are never read, so they
  // are left as they are; a live row with an out-of-range id is zeroed (zero transitions)
  for (int t = threadIdx.x; t < Ka * cpr; t += LT_THREADS) {
    const int m = t / cpr, c = t % cpr, kb = c >> 3, cc = c & 7;
    uint8_t* dst = sA + kb * (LT_M * 128) + m * 128 + ((cc ^ (m & 7)) << 4);
    const int32_t id = s_ida[m];
    if (id >= 0) ds_cp_async16(dst, E + int64_t(id) * rank + c * 8);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  for (int t = threadIdx.x; t < K * cpr; t += LT_THREADS) {
    const int m = t / cpr, c = t % cpr, kb = c >> 3, cc = c & 7;
    uint8_t* dst = sB + kb * (LT_N * 128) + m * 128 + ((cc ^ (m & 7)) << 4);
    const int32_t id = s_idb[m];
    if (id >= 0) ds_cp_async16(dst, W + int64_t(id) * rank + c * 8);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  // the gate overlaps the gathers in flight
  const int64_t hrow = a.row_start ? a.row_start[r] + j : int64_t(tile);
  const float gamma = lt_gate_any(a, hrow, s_red);
  ds_cp_async_wait_all();
  ds_fence_proxy_async_smem();
  __syncthreads();
  ds_tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = ds_idesc_bf16_f32(LT_M, LT_N);
    const uint32_t aaddr = ds_smem_addr(sA), baddr = ds_smem_addr(sB);
    for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t ad = ds_smem_desc_sw128(aaddr + kb * (LT_M * 128) + s * 32);
        const uint64_t bd = ds_smem_desc_sw128(baddr + kb * (LT_N * 128) + s * 32);
        ds_umma_f16(tmem, ad, bd, idesc, (kb | s) != 0);
      }
    }
    ds_umma_commit(&s_bar);
  }
  __syncwarp();
  bool ok = ds_mbar_wait(&s_bar, 0, DS_WAIT_LIMIT);
  if (!ok) {
    ds_set_error(a.status, DSPARK_ETIMEOUT);
    ok = ds_mbar_wait(&s_bar, 0, DS_WAIT_LIMIT);     // let in-flight MMAs drain before freeing TMEM
  }
  ok = __syncthreads_and(ok) != 0;                 // one verdict for the whole CTA
  ds_tc_fence_after();
  // each thread owns accumulator row `arow` (TMEM lane): scale it by the gate and store it
  // straight from registers (16-byte stores when the row is 16-byte aligned)
  if (ok) {
    float v[64];
    ds_tmem_ld_32x32b_x64(tmem + (uint32_t(warp * 32) << 16), v);
    const int arow = warp * 32 + lane;
    if (arow < K) {
      float* out = a.trans + (int64_t(tile) * K + arow) * K;
      const bool live = arow < Ka;
#pragma unroll
      for (int b = 0; b < 64; ++b) v[b] = live ? __fmul_rn(gamma, v[b]) : 0.0f;
      if ((K & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
#pragma unroll
        for (int b4 = 0; b4 < 16; ++b4)
          if (4 * b4 < K) reinterpret_cast<float4*>(out)[b4] = make_float4(v[4 * b4], v[4 * b4 + 1], v[4 * b4 + 2], v[4 * b4 + 3]);
      } else {
#pragma unroll
        for (int b = 0; b < 64; ++b)
          if (b < K) out[b] = v[b];
      }
    }
  }
  if (threadIdx.x == 0 && a.gate) a.gate[tile] = gamma;
  ds_tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ds_tc_fence_after();
    ds_tmem_dealloc(tmem, 64);
  }
}

// ---------------------------------------------------------------------------------------
// CUDA-core path: any table dtype / rank
// ---------------------------------------------------------------------------------------
template <typename TT>
__global__ void __launch_bounds__(256) lattice_fma_kernel(const LatticeArgs a) {
  __shared__ float sA[64][65];
  __shared__ float sB[64][65];
  __shared__ int32_t s_ida[64], s_idb[64];
  __shared__ float s_red[8];
  const int tile = blockIdx.x;
  const int r = tile / a.B, j = tile % a.B;
  const int K = a.K, rank = a.rank;
  const int Ka = (j == 0) ? 1 : K;
  const int32_t* ct = a.cand_tgt + int64_t(tile) * K;
  if (threadIdx.x < 64) {
    const int i = threadIdx.x;
    int32_t ia = -1, ib = -1;
    if (i < Ka) ia = (j == 0) ? a.prev[r] : ct[i - K];
    if (i < K) ib = ct[i];
    if (i < Ka && (ia < 0 || ia >= a.V_t)) { ds_set_error(a.status, DSPARK_ERANGE); ia = -1; }
    if (i < K && (ib < 0 || ib >= a.V_t)) { ds_set_error(a.status, DSPARK_ERANGE); ib = -1; }
    s_ida[i] = ia;
    s_idb[i] = ib;
  }
  const int64_t hrow = a.row_start ? a.row_start[r] + j : int64_t(tile);
  const float gamma = lt_gate_any(a, hrow, s_red);
  __syncthreads();
  const TT* E = reinterpret_cast<const TT*>(a.E);
  const TT* W = reinterpret_cast<const TT*>(a.W);
  const int arow = threadIdx.x >> 2, b0 = (threadIdx.x & 3) * 16;
  float acc[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) acc[q] = 0.0f;
  for (int k0 = 0; k0 < rank; k0 += 64) {
    for (int t = threadIdx.x; t < 64 * 64; t += 256) {
      const int m = t >> 6, kk = t & 63, k = k0 + kk;
      const int32_t ia = s_ida[m], ib = s_idb[m];
      sA[m][kk] = (ia >= 0 && k < rank) ? ds_load_elem<TT>(E + int64_t(ia) * rank + k) : 0.0f;
      sB[m][kk] = (ib >= 0 && k < rank) ? ds_load_elem<TT>(W + int64_t(ib) * rank + k) : 0.0f;
    }
    __syncthreads();
    for (int kk = 0; kk < 64; ++kk) {
      const float x = sA[arow][kk];
#pragma unroll
      for (int q = 0; q < 16; ++q) acc[q] = __fmaf_rn(x, sB[b0 + q][kk], acc[q]);
    }
    __syncthreads();
  }
  if (arow < K) {
    float* out = a.trans + (int64_t(tile) * K + arow) * K;
    const bool live = arow < Ka;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      if (b0 + q < K) out[b0 + q] = live ? __fmul_rn(gamma, acc[q]) : 0.0f;
  }
  if (threadIdx.x == 0 && a.gate) a.gate[tile] = gamma;
}

}  // namespace

extern "C" dspark_status dspark_lattice_score(const int32_t* cand_tgt, const int32_t* prev, int64_t R,
                                              int32_t B, int32_t K, const void* E, const void* W,
                                              dspark_dtype table_dtype, int64_t V_t, int32_t rank,
                                              const void* hidden, const void* g,
                                              dspark_dtype hidden_dtype, int32_t H, int64_t ldh,
                                              const int64_t* row_start, float* trans, float* gate,
                                              int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(R >= 0 && B >= 1 && K >= 1 && K <= 64 && rank >= 1 && V_t >= 1);
  DS_REQUIRE(R * B <= 0x7FFFFFFF && V_t <= 0x7FFFFFFF);
  DS_REQUIRE(cand_tgt && prev && E && W && trans && dev_status);
  DS_REQUIRE(ds_dtype_ok(table_dtype));
  if (hidden) {
    DS_REQUIRE(g && H >= 1 && ldh >= H && ds_dtype_ok(hidden_dtype));
  }
  if (R == 0) return DSPARK_OK;
  LatticeArgs a;
  a.cand_tgt = cand_tgt;
  a.prev = prev;
  a.B = B;
  a.K = K;
  a.rank = rank;
  a.H = H;
  a.E = E;
  a.W = W;
  a.V_t = V_t;
  a.hidden = hidden;
  a.g = g;
  a.ldh = ldh;
  a.row_start = row_start;
  a.trans = trans;
  a.gate = gate;
  a.status = dev_status;
  a.hidden_bf16 = hidden_dtype == DSPARK_BF16;
  const unsigned tiles = unsigned(R * B);
  const bool tc = table_dtype == DSPARK_BF16 && rank % 64 == 0 && rank <= 512 &&
                  ds_aligned(E, 16) && ds_aligned(W, 16);
  if (tc) {
    const size_t smem = std::max<size_t>(size_t(rank / 64) * (LT_M + LT_N) * 128, 64 * 65 * 4) + 1024;
    DS_CUDA_TRY(ds_ensure_smem(reinterpret_cast<const void*>(lattice_tc_kernel), smem));
    lattice_tc_kernel<<<tiles, LT_THREADS, smem, stream>>>(a);
  } else if (table_dtype == DSPARK_BF16) {
    lattice_fma_kernel<__nv_bfloat16><<<tiles, 256, 0, stream>>>(a);
  } else {
    lattice_fma_kernel<float><<<tiles, 256, 0, stream>>>(a);
  }
  return ds_launch_status();
}
