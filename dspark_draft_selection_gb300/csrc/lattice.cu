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
// four warps read the 128 x 64 accumulator tile back with tcgen05.ld and scale it by the
// gate. float32 tables (or ranks the tensor-core layout does not take) use a CUDA-core FMA
// kernel instead.
//
// dspark_lattice_chain fuses the lattice with the greedy chain rules (max-sum, walk) for blocks
// of up to 8 positions: the B tile CTAs of a request form one thread-block cluster, each keeps
// its tile in its own shared memory, and the cluster's first CTA runs the chain recurrence of
// dspark_chain_select (same float32 operations, same tie rules) reading the other tiles through
// distributed shared memory. The lattice never makes a round trip through HBM.
#include <atomic>

#include <cooperative_groups.h>

#include "dspark_common.cuh"
#include "host_common.h"

namespace cg = cooperative_groups;

// Poll limit of the first wait for the tile's MMAs (a test hook can lower it; see
// dspark_test_set_first_wait_polls). The wait after a first wait that ran out keeps the full
// limit, so tensor memory is never freed while MMAs are in flight.
std::atomic<uint32_t> g_ds_first_wait_polls{DS_WAIT_LIMIT};

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
  uint32_t first_wait;       // polls of the first MMA-completion wait
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
struct LtShared {
  uint64_t bar;
  uint32_t tmem;
  int32_t ida[LT_M];
  int32_t idb[LT_N];
  float red[LT_THREADS / 32];
};

// Tile (r, j) on the tensor cores. Afterwards thread (warp, lane) holds accumulator row
// warp * 32 + lane, scaled by the gate, in v (rows past the tile's live rows are zero), and the
// tile's tensor memory is freed. Returns false (DSPARK_ETIMEOUT set, v zero) if the MMA wait ran
// out. `base`: 1024-byte aligned dynamic shared memory of nkb * (LT_M + LT_N) * 128 bytes.
DS_DEV bool lt_tile_tc(const LatticeArgs& a, int r, int j, uint8_t* base, LtShared& sh, float (&v)[64],
                       float& gamma) {
  const int tile = r * a.B + j;
  const int K = a.K, rank = a.rank;
  const int nkb = rank / 64;                         // 64-element (128-byte) K chunks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* sA = base;                                // nkb x [128 rows x 128 B]
  uint8_t* sB = base + nkb * (LT_M * 128);           // nkb x [ 64 rows x 128 B]

  if (warp == 0) ds_tmem_alloc(&sh.tmem, 64);
  if (threadIdx.x == 0) ds_mbar_init(&sh.bar, 1);

  const int Ka = (j == 0) ? 1 : K;
  const int32_t* ct = a.cand_tgt + int64_t(tile) * K;
  for (int i = threadIdx.x; i < LT_M; i += LT_THREADS) {
    int32_t id = -1;
    if (i < Ka) id = (j == 0) ? a.prev[r] : ct[i - K];  // previous position's candidates
    if (i < Ka && (id < 0 || id >= a.V_t)) {
      ds_set_error(a.status, DSPARK_ERANGE);
      id = -1;
    }
    sh.ida[i] = id;
  }
  for (int i = threadIdx.x; i < LT_N; i += LT_THREADS) {
    int32_t id = (i < K) ? ct[i] : -1;
    if (i < K && (id < 0 || id >= a.V_t)) {
      ds_set_error(a.status, DSPARK_ERANGE);
      id = -1;
    }
    sh.idb[i] = id;
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
    const int32_t id = sh.ida[m];
    if (id >= 0) ds_cp_async16(dst, E + int64_t(id) * rank + c * 8);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  for (int t = threadIdx.x; t < K * cpr; t += LT_THREADS) {
    const int m = t / cpr, c = t % cpr, kb = c >> 3, cc = c & 7;
    uint8_t* dst = sB + kb * (LT_N * 128) + m * 128 + ((cc ^ (m & 7)) << 4);
    const int32_t id = sh.idb[m];
    if (id >= 0) ds_cp_async16(dst, W + int64_t(id) * rank + c * 8);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  // the gate overlaps the gathers in flight
  const int64_t hrow = a.row_start ? a.row_start[r] + j : int64_t(tile);
  gamma = lt_gate_any(a, hrow, sh.red);
  ds_cp_async_wait_all();
  ds_fence_proxy_async_smem();
  __syncthreads();
  ds_tc_fence_after();
  const uint32_t tmem = sh.tmem;

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
    ds_umma_commit(&sh.bar);
  }
  __syncwarp();
  bool ok = ds_mbar_wait(&sh.bar, 0, a.first_wait);
  if (!ok) {
    ds_set_error(a.status, DSPARK_ETIMEOUT);
    (void)ds_mbar_wait(&sh.bar, 0, DS_WAIT_LIMIT);    // let in-flight MMAs drain before freeing TMEM
  }
  ok = __syncthreads_and(ok) != 0;                 // one verdict for the whole CTA
  ds_tc_fence_after();
  if (ok) {
    ds_tmem_ld_32x32b_x64(tmem + (uint32_t(warp * 32) << 16), v);
    const bool live = warp * 32 + lane < Ka;
#pragma unroll
    for (int b = 0; b < 64; ++b) v[b] = live ? __fmul_rn(gamma, v[b]) : 0.0f;
  } else {
#pragma unroll
    for (int b = 0; b < 64; ++b) v[b] = 0.0f;
  }
  ds_tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ds_tc_fence_after();
    ds_tmem_dealloc(tmem, 64);
  }
  return ok;
}

// Stores row `arow` of tile `tile` (16-byte stores when the row is 16-byte aligned).
DS_DEV void lt_store_row(const LatticeArgs& a, int tile, int arow, const float (&v)[64]) {
  const int K = a.K;
  float* out = a.trans + (int64_t(tile) * K + arow) * K;
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

__global__ void __launch_bounds__(LT_THREADS) lattice_tc_kernel(const LatticeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ LtShared sh;
  const int tile = blockIdx.x;                       // r * B + j
  const int r = tile / a.B, j = tile % a.B;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ds_pdl_trigger();
  ds_pdl_wait();                                     // the candidates come from the previous kernel;
                                                     // no CTA holds tensor memory while it waits
  float v[64];
  float gamma;
  const bool ok = lt_tile_tc(a, r, j, base, sh, v, gamma);
  const int arow = threadIdx.x;                      // warp * 32 + lane: the thread's TMEM lane
  if (ok && arow < a.K) lt_store_row(a, tile, arow, v);
  if (threadIdx.x == 0 && a.gate) a.gate[tile] = gamma;
}

// ---------------------------------------------------------------------------------------
// lattice + greedy chain, one cluster of B tile CTAs per request (B <= 8)
// ---------------------------------------------------------------------------------------
constexpr int LC_MAXB = 8;
constexpr uint32_t LC_TILE_BYTES = 64 * 64 * 4;

struct ChainOut {
  const float* u;                                    // [R, B, K] unary scores
  int mode;
  int32_t* chain_rank;
  int32_t* chain_tgt;
  float* score;
};

// Float offset of element (a, b) in a 64 x 64 tile: rows of 64 floats, the 16-byte groups of row a
// permuted by a & 15 (row-wise 16-byte stores and column-wise reads are both free of bank conflicts).
DS_DEV int lc_off(int a, int b) { return a * 64 + ((((b >> 2) ^ (a & 15))) << 2) + (b & 3); }

// The chain recurrence of dspark_chain_select for one request, run by the cluster's first CTA on
// tiles in its shared memory: position 0's row in s_row0, position jj >= 1 at rx + (jj - 1) * 4096.
DS_DEV void lc_chain(const ChainOut& c, int r, int B, int K, const float* s_row0, const float* rx, const float* s_u,
                     const int32_t* s_ct, float* s_delta, float (*s_bv)[64], int (*s_ba)[64], uint8_t (*s_back)[64],
                     int* s_path) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  if (c.mode == DSPARK_MAXSUM) {
    if (t < K) s_delta[t] = __fadd_rn(s_u[t], s_row0[t]);        // delta_0 = u_0 + A_0[0, :]
    __syncthreads();
    for (int jj = 1; jj < B; ++jj) {
      const float* At = rx + (jj - 1) * 4096;
      const float* uj = s_u + jj * K;
      const int b = t & 63, part = t >> 6;         // two threads per column, 32 predecessors each
      if (b < K) {
        const int a0 = part * 32, na = min(K - a0, 32);
        float vv[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) vv[q] = (q < na) ? __fadd_rn(s_delta[a0 + q], At[lc_off(a0 + q, b)]) : -INFINITY;
        float best = vv[0];
        int ba = (na > 0) ? a0 : -1;
#pragma unroll
        for (int q = 1; q < 32; ++q)
          if (q < na && vv[q] > best) {
            best = vv[q];
            ba = a0 + q;
          }
        s_bv[part][b] = best;
        s_ba[part][b] = ba;
      }
      __syncthreads();
      float nd = 0.0f;
      if (t < K) {
        float best = s_bv[0][t];
        int ba = s_ba[0][t];
        if (s_ba[1][t] >= 0 && (ba < 0 || s_bv[1][t] > best)) {
          best = s_bv[1][t];
          ba = s_ba[1][t];
        }
        nd = __fadd_rn(uj[t], best);
        s_back[jj][t] = uint8_t(ba < 0 ? 0 : ba);
      }
      __syncthreads();
      if (t < K) s_delta[t] = nd;
      __syncthreads();
    }
    if (warp == 0) {
      uint64_t kbest = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = lane + 32 * h;
        if (k < K) {
          const uint64_t kk = ds_key64(ds_canon_zero(s_delta[k]), uint32_t(k));
          kbest = kk > kbest ? kk : kbest;
        }
      }
      kbest = ds_warp_max_u64(kbest);
      if (lane == 0) {
        int bb = int(ds_key64_idx(kbest));
        c.score[r] = s_delta[bb];
        for (int jj = B - 1; jj >= 0; --jj) {
          s_path[jj] = bb;
          if (jj > 0) bb = s_back[jj][bb];
        }
      }
    }
    __syncthreads();
    if (t < B) {
      const int bb = s_path[t];
      c.chain_rank[r * B + t] = bb;
      c.chain_tgt[r * B + t] = s_ct[t * K + bb];
    }
  } else if (warp == 0) {                            // greedy walk: the best candidate after the one before
    int prevb = 0;
    double score = 0.0;
    for (int jj = 0; jj < B; ++jj) {
      float w2[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = lane + 32 * h;
        const float ab = (b < K) ? (jj == 0 ? s_row0[b] : rx[(jj - 1) * 4096 + lc_off(prevb, b)]) : 0.0f;
        w2[h] = (b < K) ? __fadd_rn(s_u[jj * K + b], ab) : -INFINITY;
      }
      const uint64_t k0 = (lane < K) ? ds_key64(ds_canon_zero(w2[0]), lane) : 0;
      const uint64_t k1 = (lane + 32 < K) ? ds_key64(ds_canon_zero(w2[1]), lane + 32) : 0;
      const int pick = int(ds_key64_idx(ds_warp_max_u64(k0 > k1 ? k0 : k1)));
      const float vp = __shfl_sync(0xFFFFFFFFu, pick < 32 ? w2[0] : w2[1], pick & 31);
      score += double(vp);
      if (lane == 0) {
        c.chain_rank[r * B + jj] = pick;
        c.chain_tgt[r * B + jj] = s_ct[jj * K + pick];
      }
      prevb = pick;
    }
    if (lane == 0) c.score[r] = float(score);
  }
}

// Each CTA computes its position's tile; the CTAs of positions 1..B-1 then push their tiles into
// the first CTA's operand buffers (free once its own MMAs are done) with one bulk copy each,
// completing on the first CTA's mbarrier, and leave; the first CTA runs the chain on chip.
__global__ void __launch_bounds__(LT_THREADS) lattice_chain_kernel(const LatticeArgs a, const ChainOut c) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ LtShared sh;
  __shared__ __align__(8) uint64_t s_rx;            // tiles received by the first CTA
  __shared__ float s_row0[64];
  __shared__ float s_u[LC_MAXB * 64];
  __shared__ int32_t s_ct[LC_MAXB * 64];
  __shared__ float s_delta[64];
  __shared__ float s_bv[2][64];
  __shared__ int s_ba[2][64];
  __shared__ uint8_t s_back[LC_MAXB][64];
  __shared__ int s_path[LC_MAXB];
  cg::cluster_group cl = cg::this_cluster();
  const int j = int(cl.block_rank());                // cluster dims (B, 1, 1): rank = position
  const int tile = blockIdx.x, r = tile / a.B;
  const int K = a.K, B = a.B, t = threadIdx.x;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* s_tile = reinterpret_cast<float*>(base);
  if (j == 0 && t == 0) {
    ds_mbar_init(&s_rx, 1);
    ds_fence_mbar_init_cluster();
  }
  ds_pdl_trigger();
  ds_pdl_wait();
  float v[64];
  float gamma;
  const bool ok = lt_tile_tc(a, r, j, base, sh, v, gamma);
  if (a.trans && ok && t < K) lt_store_row(a, tile, t, v);
  if (t == 0 && a.gate) a.gate[tile] = gamma;
  if (j == 0) {
    for (int i = t; i < B * K; i += LT_THREADS) {
      s_u[i] = c.u[int64_t(r) * B * K + i];
      s_ct[i] = a.cand_tgt[int64_t(r) * B * K + i];
    }
    if (t == 0) {
#pragma unroll
      for (int b = 0; b < 64; ++b) s_row0[b] = v[b];
      ds_mbar_arrive_expect_tx(&s_rx, uint32_t(B - 1) * LC_TILE_BYTES);
    }
  } else if (t < 64) {
    // the tile into this CTA's operand buffers (its MMAs are done), rows of 64 floats
#pragma unroll
    for (int k4 = 0; k4 < 16; ++k4)
      *reinterpret_cast<float4*>(s_tile + t * 64 + ((k4 ^ (t & 15)) << 2)) =
          make_float4(v[4 * k4], v[4 * k4 + 1], v[4 * k4 + 2], v[4 * k4 + 3]);
    ds_fence_proxy_async_smem();                     // the bulk copy reads what the threads wrote
  }
  cl.sync();                                         // every tile is formed; the first CTA can receive
  if (j != 0) {
    if (t == 0) {
      const uint32_t dst = ds_mapa(ds_smem_addr(base) + uint32_t(j - 1) * LC_TILE_BYTES, 0);
      ds_bulk_s2s_cluster(dst, ds_smem_addr(s_tile), LC_TILE_BYTES, ds_mapa(ds_smem_addr(&s_rx), 0));
      ds_bulk_wait_read_all();                       // the source must outlive the copy's reads
    }
    return;
  }
  bool got = ds_mbar_wait(&s_rx, 0, DS_WAIT_LIMIT);
  if (!got) {
    ds_set_error(a.status, DSPARK_ETIMEOUT);
    got = ds_mbar_wait(&s_rx, 0, DS_WAIT_LIMIT);     // copies still landing here must finish first
  }
  if (__syncthreads_and(got) == 0) return;
  lc_chain(c, r, B, K, s_row0, s_tile, s_u, s_ct, s_delta, s_bv, s_ba, s_back, s_path);
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
  ds_pdl_trigger();
  ds_pdl_wait();
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
  LatticeArgs a = {};
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
  a.first_wait = g_ds_first_wait_polls.load(std::memory_order_relaxed);
  const unsigned tiles = unsigned(R * B);
  const bool tc = table_dtype == DSPARK_BF16 && rank % 64 == 0 && rank <= 512 &&
                  ds_aligned(E, 16) && ds_aligned(W, 16);
  if (tc) {
    const size_t smem = std::max<size_t>(size_t(rank / 64) * (LT_M + LT_N) * 128, 64 * 65 * 4) + 1024;
    DS_CUDA_TRY(ds_ensure_smem(reinterpret_cast<const void*>(lattice_tc_kernel), smem));
    DS_CUDA_TRY(ds_launch(lattice_tc_kernel, dim3(tiles), dim3(LT_THREADS), smem, stream, a));
  } else if (table_dtype == DSPARK_BF16) {
    DS_CUDA_TRY(ds_launch(lattice_fma_kernel<__nv_bfloat16>, dim3(tiles), dim3(256), 0, stream, a));
  } else {
    DS_CUDA_TRY(ds_launch(lattice_fma_kernel<float>, dim3(tiles), dim3(256), 0, stream, a));
  }
  return DSPARK_OK;
}

extern "C" void dspark_test_set_first_wait_polls(uint32_t polls) {
  g_ds_first_wait_polls.store(polls == 0xFFFFFFFFu ? DS_WAIT_LIMIT : polls, std::memory_order_relaxed);
}

extern "C" dspark_status dspark_lattice_chain(const float* cand_val, const int32_t* cand_tgt, const int32_t* prev,
                                              int64_t R, int32_t B, int32_t K, const void* E, const void* W,
                                              dspark_dtype table_dtype, int64_t V_t, int32_t rank,
                                              const void* hidden, const void* g, dspark_dtype hidden_dtype,
                                              int32_t H, int64_t ldh, const int64_t* row_start,
                                              dspark_chain_mode mode, float* trans, float* gate,
                                              int32_t* chain_rank, int32_t* chain_tgt, float* score,
                                              int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(R >= 0 && B >= 1 && K >= 1 && K <= 64 && rank >= 1 && V_t >= 1);
  DS_REQUIRE(R * B <= 0x7FFFFFFF && V_t <= 0x7FFFFFFF);
  DS_REQUIRE(cand_val && cand_tgt && prev && E && W && chain_rank && chain_tgt && score && dev_status);
  DS_REQUIRE(ds_dtype_ok(table_dtype) && (mode == DSPARK_MAXSUM || mode == DSPARK_WALK));
  if (hidden) DS_REQUIRE(g && H >= 1 && ldh >= H && ds_dtype_ok(hidden_dtype));
  const bool fused = table_dtype == DSPARK_BF16 && rank % 64 == 0 && rank <= 512 && B <= LC_MAXB &&
                     ds_aligned(E, 16) && ds_aligned(W, 16);
  if (!fused) {
    // the two-launch path needs the lattice in memory
    DS_REQUIRE(trans != nullptr);
    const dspark_status st = dspark_lattice_score(cand_tgt, prev, R, B, K, E, W, table_dtype, V_t, rank, hidden, g,
                                                  hidden_dtype, H, ldh, row_start, trans, gate, dev_status, stream);
    if (st != DSPARK_OK) return st;
    return dspark_chain_select(cand_val, trans, cand_tgt, R, B, K, mode, 0.0f, 1.0f, 0.0f, nullptr, nullptr, nullptr,
                               nullptr, nullptr, nullptr, chain_rank,
                               chain_tgt, score, nullptr, dev_status, stream);
  }
  if (R == 0) return DSPARK_OK;
  LatticeArgs a = {};
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
  a.first_wait = g_ds_first_wait_polls.load(std::memory_order_relaxed);
  ChainOut c;
  c.u = cand_val;
  c.mode = int(mode);
  c.chain_rank = chain_rank;
  c.chain_tgt = chain_tgt;
  c.score = score;
  const size_t smem = std::max<size_t>(size_t(rank / 64) * (LT_M + LT_N) * 128, size_t(B - 1) * LC_TILE_BYTES) + 1024;
  DS_CUDA_TRY(ds_ensure_smem(reinterpret_cast<const void*>(lattice_chain_kernel), smem));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(R * B));
  cfg.blockDim = dim3(LT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(B);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  DS_CUDA_TRY(cudaLaunchKernelEx(&cfg, lattice_chain_kernel, a, c));
  return DSPARK_OK;
}
