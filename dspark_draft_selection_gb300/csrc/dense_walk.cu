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
//  1. dense_walk_gemm_kernel - a persistent, warp-specialised tcgen05 GEMM over the draft
//     vocabulary in 128-row tiles. The W rows m(i) of a tile go into a ring of 128-byte swizzled
//     K-chunks, one stage per mbarrier, with an L2 evict-last policy (the table is read again at
//     every position): one TMA copy per stage when the rows are contiguous (no d2t), else four
//     producer warps gathering them with cp.async; one thread issues the MMAs (M = 128 request rows
//     of E[prev_r], staged once; N = the tile's 128 vocabulary rows; K = rank) into one of two TMEM
//     accumulators; the epilogue warps drain the other accumulator, one request per TMEM lane, so
//     each lane reads its logits and writes z = (s + gamma tau) / T into the dense record (or the
//     workspace) as contiguous vectors, and keeps its request's largest (z, lowest index) key in a
//     register (then reduced across the CTA and the GPU).
//  2. sampled positions without a nucleus: dense_walk_draw_kernel - the z rows in parts over many
//     CTAs: weights of z - zmax, the kept mass of every cell of 256 indices; the part that finishes
//     last draws the token (double running sums over the cells, then the cell's elements) and
//     writes it as the next position's previous token. Greedy positions finish with the argmax key
//     (dense_walk_greedy_kernel); nucleus positions use the row sampler of sample.cu on the z rows.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int DW_M = 128;                    // vocabulary rows per tile (MMA M)
constexpr int DW_MAXR = 128;                 // requests per GEMM launch (MMA N <= 128)
constexpr int DW_NS = 8;                     // K-chunk stages in the ring (16 KB each)
constexpr int DW_PROD = 128;                 // producer threads (warps 0-3)
constexpr int DW_MMA_WARP = 4;
constexpr int DW_EPI_WARP0 = 5;              // epilogue warps 5..12
constexpr int DW_EPI = 256;
constexpr int DW_THREADS = DW_PROD + 32 + DW_EPI;
constexpr uint32_t DW_STAGE = DW_M * 128;    // bytes of one K-chunk of a tile

struct DwArgs {
  const void* logits;
  int64_t ld;
  const int64_t* row_start;
  int32_t B, j, R, rank;
  int64_t V, V_t, ntiles;
  const int32_t* prev_cur;
  const __nv_bfloat16* E;
  const __nv_bfloat16* W;
  const int64_t* d2t;
  const float* gate;
  float mult, softcap, Tz;
  float* z;
  int64_t ldz, z_row_mul, z_row_add;
  unsigned long long* zkey;  // [R, B] largest (z, lowest index) key of each request and position
  int32_t* status;
  uint32_t first_wait;       // polls of the epilogue's first wait for an accumulator
  int use_tma;               // W rows are contiguous (no d2t): one TMA load fills a stage
};

template <bool XFORM>
DS_DEV float dw_xform(float x, float mult, float softcap) {
  if (XFORM) {
    if (mult != 1.0f) x = __fmul_rn(x, mult);
    if (softcap > 0.0f) x = __fmul_rn(softcap, tanhf(__fdiv_rn(x, softcap)));
  }
  return x;
}

// gamma_{r,j} for every (request, position); also the first position's previous tokens, the
// per-position maximum keys (cleared) and the draw tickets (cleared)
template <typename HT>
__global__ void __launch_bounds__(128) dense_walk_gate_kernel(const HT* hidden, const HT* g, int H, int64_t ldh,
                                                              const int64_t* row_start, int32_t B,
                                                              const int32_t* prev, int32_t* prev_cur, float* gate,
                                                              unsigned long long* zkey, int32_t* ticket) {
  __shared__ float s_red[4];
  const int tile = blockIdx.x;
  const int r = tile / B, j = tile % B;
  ds_pdl_trigger();
  ds_pdl_wait();
  float gamma = 1.0f;
  if (hidden != nullptr) {
    const int64_t hrow = row_start ? row_start[r] + j : int64_t(tile);
    gamma = ds_block_gate(hidden + hrow * ldh, g, H, s_red);
  }
  if (threadIdx.x == 0) {
    gate[tile] = gamma;
    zkey[tile] = 0ull;
    if (j == 0) {
      prev_cur[r] = prev[r];
      ticket[r] = 0;
    }
  }
}

// Eight consecutive logits of a row as float (vector load when aligned and whole; zero past V)
template <typename T>
DS_DEV void dw_ld8(const T* p, int64_t i, int64_t V, float (&x)[8]) {
  if (i + 8 <= V && (reinterpret_cast<uintptr_t>(p + i) & 15) == 0) {
    if constexpr (sizeof(T) == 2) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p + i));
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = ds_vec_elem<T>(v, e);
    } else {
      const uint4 v0 = __ldcs(reinterpret_cast<const uint4*>(p + i)), v1 = __ldcs(reinterpret_cast<const uint4*>(p + i) + 1);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] = ds_vec_elem<T>(v0, e);
        x[e + 4] = ds_vec_elem<T>(v1, e);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (i + e < V) ? ds_load_elem<T>(p + i + e) : 0.0f;
  }
}

// D[request, vocabulary] = E[prev] . W[m(i)]^T: TMEM lanes are requests (M = 128, rows past R
// zero), columns the tile's 128 vocabulary indices, so an epilogue lane owns one request: its logits
// and z are contiguous vectors and its maximum is a running value in a register.
template <typename T, bool XFORM, bool TONE>
__global__ void __launch_bounds__(DW_THREADS, 1) dense_walk_gemm_kernel(const DwArgs a,
                                                                       const __grid_constant__ CUtensorMap tmW) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_full[DW_NS], s_empty[DW_NS], s_accf[2], s_acce[2], s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int32_t s_prev[DW_MAXR];
  __shared__ float s_gate[DW_MAXR];
  __shared__ int64_t s_lrow[DW_MAXR];
  __shared__ unsigned long long s_kmax[DW_MAXR];

  const int rank = a.rank, nkb = rank / 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;                                  // nkb x [128 request rows x 128 B]
  uint8_t* sB = base + nkb * (DW_MAXR * 128);          // DW_NS x [128 vocabulary rows x 128 B]
  constexpr uint32_t ncols = 2 * DW_M;                 // two accumulators of 128 columns

  ds_pdl_trigger();
  ds_pdl_wait();                                       // previous tokens come from the last position
  if (tid == 0) {
    for (int s = 0; s < DW_NS; ++s) {
      ds_mbar_init(&s_full[s], a.use_tma ? 1 : DW_PROD);
      ds_mbar_init(&s_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ds_mbar_init(&s_accf[b], 1);
      ds_mbar_init(&s_acce[b], DW_EPI / 32);
    }
    ds_mbar_init(&s_drain, 1);
    s_abort = 0;
  }
  if (warp == DW_MMA_WARP) ds_tmem_alloc(&s_tmem, ncols);
  for (int r = tid; r < DW_MAXR; r += DW_THREADS) {
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
    s_kmax[r] = 0ull;
  }
  __syncthreads();
  // the A operand: E[prev_r] of every request (zero rows past R and for bad ids), once. With at
  // most 64 requests, rows 64..127 repeat rows 0..63, so every TMEM lane quarter holds requests.
  const bool dup = a.R <= 64;
  const int cpr = rank / 8;
  for (int t = tid; t < DW_MAXR * cpr; t += DW_THREADS) {
    const int m = t / cpr, c = t % cpr, kb = c >> 3, cc = c & 7;
    uint8_t* dst = sA + kb * (DW_MAXR * 128) + m * 128 + ((cc ^ (m & 7)) << 4);
    const int32_t id = s_prev[dup ? (m & 63) : m];
    if (id >= 0) ds_cp_async16(dst, a.E + int64_t(id) * rank + c * 8);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  ds_cp_async_wait_all();
  ds_fence_proxy_async_smem();
  __syncthreads();
  ds_tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp < DW_PROD / 32 && a.use_tma) {
    // ---- producer: one thread loads each K-chunk of a tile (128 contiguous W rows x 128 bytes,
    // 128-byte swizzle) with one TMA copy; rows past the table read as zero ----
    if (tid == 0) {
      const uint64_t pol = ds_policy_evict_last();
      uint32_t g = 0;
      for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const uint32_t s = g % DW_NS, ph = (g / DW_NS) & 1u;
          if (!ds_mbar_wait_or_abort(&s_empty[s], ph ^ 1u, DS_WAIT_LIMIT, &s_abort)) {
            if (!*reinterpret_cast<volatile int*>(&s_abort)) ds_set_error(a.status, DSPARK_ETIMEOUT);
            s_abort = 1;
          }
          if (*reinterpret_cast<volatile int*>(&s_abort)) break;
          ds_mbar_arrive_expect_tx(&s_full[s], DW_STAGE);
          ds_tma_load_2d(sB + s * DW_STAGE, &tmW, kb * 64, int32_t(tile * DW_M), &s_full[s], pol);
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
      }
      // every TMA copy this thread issued lands before the CTA leaves (or the wait gives up)
      for (uint32_t k = (g > DW_NS ? g - DW_NS : 0); k < g; ++k)
        (void)ds_mbar_wait(&s_full[k % DW_NS], (k / DW_NS) & 1u, DS_WAIT_LIMIT);
    }
    __syncwarp();
  } else if (warp < DW_PROD / 32) {
    // ---- producers: thread p copies 16-byte column p % 8 of rows p / 8 + 16 kk of each K-chunk ----
    const uint64_t pol = ds_policy_evict_last();
    const int cc = tid & 7, m0 = tid >> 3;
    uint32_t g = 0;                                    // K-chunks issued by this CTA
    for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
      const int64_t i0 = tile * DW_M;
      int64_t rid[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int64_t i = i0 + m0 + 16 * kk;
        int64_t t = -2;                                // -2: past the vocabulary (column never read)
        if (i < a.V) {
          t = a.d2t ? i + a.d2t[i] : i;
          if (t < 0 || t >= a.V_t) {
            ds_set_error(a.status, DSPARK_ERANGE);
            t = -1;                                    // -1: zero row (zero transitions)
          }
        }
        rid[kk] = t;
      }
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        const uint32_t s = g % DW_NS, ph = (g / DW_NS) & 1u;
        if (!ds_mbar_wait_or_abort(&s_empty[s], ph ^ 1u, DS_WAIT_LIMIT, &s_abort)) {
          if (!*reinterpret_cast<volatile int*>(&s_abort)) ds_set_error(a.status, DSPARK_ETIMEOUT);
          s_abort = 1;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        uint8_t* stage = sB + s * DW_STAGE;
        bool zeroed = false;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int m = m0 + 16 * kk;
          uint8_t* dst = stage + m * 128 + ((cc ^ (m & 7)) << 4);
          if (rid[kk] >= 0) {
            ds_cp_async16_hint(dst, a.W + rid[kk] * rank + kb * 64 + cc * 8, pol);
          } else if (rid[kk] == -1) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            zeroed = true;
          }
        }
        if (zeroed) ds_fence_proxy_async_smem();
        ds_cp_async_mbar_arrive(&s_full[s]);
      }
      if (*reinterpret_cast<volatile int*>(&s_abort)) break;
    }
    ds_cp_async_wait_all();                            // no copy lands after the CTA is gone
  } else if (warp == DW_MMA_WARP) {
    // ---- one thread issues the MMAs; the accumulator buffers alternate by tile ----
    if (lane == 0) {
      constexpr uint32_t idesc = ds_idesc_bf16_f32(DW_MAXR, DW_M);
      const uint32_t aaddr = ds_smem_addr(sA), baddr = ds_smem_addr(sB);
      uint32_t g = 0, k = 0;
      for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++k) {
        const uint32_t b = k & 1u, use = k >> 1;
        if (!ds_mbar_wait_or_abort(&s_acce[b], (use & 1u) ^ 1u, DS_WAIT_LIMIT, &s_abort)) {
          if (!*reinterpret_cast<volatile int*>(&s_abort)) ds_set_error(a.status, DSPARK_ETIMEOUT);
          s_abort = 1;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        ds_tc_fence_after();
        const uint32_t dacc = tmem + b * uint32_t(DW_M);
        bool stop = false;
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const uint32_t s = g % DW_NS, ph = (g / DW_NS) & 1u;
          if (!ds_mbar_wait_or_abort(&s_full[s], ph, DS_WAIT_LIMIT, &s_abort)) {
            if (!*reinterpret_cast<volatile int*>(&s_abort)) ds_set_error(a.status, DSPARK_ETIMEOUT);
            s_abort = 1;
          }
          if (*reinterpret_cast<volatile int*>(&s_abort)) {
            stop = true;
            break;
          }
          ds_tc_fence_after();
#pragma unroll
          for (int sub = 0; sub < 4; ++sub) {
            const uint64_t ad = ds_smem_desc_sw128(aaddr + kb * (DW_MAXR * 128) + sub * 32);
            const uint64_t bd = ds_smem_desc_sw128(baddr + s * DW_STAGE + sub * 32);
            ds_umma_f16(dacc, ad, bd, idesc, (kb | sub) != 0);
          }
          ds_umma_commit(&s_empty[s]);                 // the stage is free once these MMAs are done
        }
        if (stop) break;
        ds_umma_commit(&s_accf[b]);                    // the tile's accumulator is complete
      }
      // every MMA this thread issued completes before tensor memory is released
      ds_umma_commit(&s_drain);
      (void)ds_mbar_wait(&s_drain, 0, DS_WAIT_LIMIT);
    }
    __syncwarp();
  } else {
    // ---- epilogue: warp ew reads TMEM lanes 32 (warp % 4) .. (requests). With duplicated request
    // rows every warp owns one 32-column chunk of each tile and prefetches the next tile's logits
    // for it; otherwise the quarters holding requests take chunks h and h + 2, h = ew / 4 ----
    constexpr int VPC = 32 * int(sizeof(T)) / 16;      // 16-byte vectors of logits per chunk
    const int ew = warp - DW_EPI_WARP0, q = warp & 3, h = ew >> 2;
    const int r = dup ? (q & 1) * 32 + lane : q * 32 + lane;   // this lane's request
    const bool live = r < a.R;
    const bool any = dup || q * 32 < a.R;              // warp-uniform: the quarter holds requests
    const int ch0 = dup ? (q >> 1) * 2 + h : h, chs = dup ? 4 : 2;
    const T* lrow = live ? reinterpret_cast<const T*>(a.logits) + s_lrow[r] * a.ld : nullptr;
    float* zrow = live ? a.z + (int64_t(r) * a.z_row_mul + a.z_row_add) * a.ldz : nullptr;
    const float gam = live ? s_gate[r] : 0.0f;
    const bool vec_l = live && (reinterpret_cast<uintptr_t>(lrow) & 15) == 0;
    const bool vec_z = live && (reinterpret_cast<uintptr_t>(zrow) & 15) == 0;
    auto fetch = [&](int64_t i0, uint4 (&buf)[VPC]) {  // one chunk's logits, whole vectors only
      if (vec_l && i0 + 32 <= a.V) {
#pragma unroll
        for (int v = 0; v < VPC; ++v) buf[v] = __ldcs(reinterpret_cast<const uint4*>(lrow + i0) + v);
      }
    };
    auto chunk = [&](int64_t i0, const uint4 (&buf)[VPC], float (&acc)[32], unsigned long long& kb) {
      constexpr int EPV = 16 / int(sizeof(T));
      const bool whole = vec_l && i0 + 32 <= a.V;
#pragma unroll
      for (int c = 0; c < 32; ++c) {                   // z in place of the accumulator
        const float sv = whole ? ds_vec_elem<T>(buf[c / EPV], c % EPV) : ((i0 + c < a.V) ? ds_load_elem<T>(lrow + i0 + c) : 0.0f);
        acc[c] = ds_temper_t<TONE>(__fmaf_rn(gam, acc[c], dw_xform<XFORM>(sv, a.mult, a.softcap)), a.Tz);
        if (i0 + c < a.V) {
          const unsigned long long key = ds_key64(ds_canon_zero(acc[c]), uint32_t(i0 + c));
          kb = key > kb ? key : kb;
        }
      }
      if (vec_z && i0 + 32 <= a.V) {
#pragma unroll
        for (int v = 0; v < 8; ++v)
          reinterpret_cast<float4*>(zrow + i0)[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (i0 + c < a.V) zrow[i0 + c] = acc[c];
      }
    };
    // the next tile's logits are prefetched into registers for bf16 rows (the register budget of
    // 13 warps, 128 a thread, does not hold two float32 chunks)
    constexpr bool PREF = sizeof(T) == 2;
    unsigned long long kbest = 0ull;
    uint4 pf[VPC];
    if (PREF && dup && live) fetch(int64_t(blockIdx.x) * DW_M + ch0 * 32, pf);
    uint32_t k = 0;
    bool first = true;
    for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++k) {
      const uint32_t b = k & 1u, use = k >> 1;
      uint4 cur[VPC];
      if (PREF && dup) {                               // this tile's logits; fetch the next tile's
#pragma unroll
        for (int v = 0; v < VPC; ++v) cur[v] = pf[v];
        if (live && tile + gridDim.x < a.ntiles) fetch((tile + gridDim.x) * DW_M + ch0 * 32, pf);
      }
      const bool ok =
          ds_mbar_wait_or_abort(&s_accf[b], use & 1u, first ? a.first_wait : DS_WAIT_LIMIT, &s_abort);
      first = false;
      if (!ok) {
        if (!*reinterpret_cast<volatile int*>(&s_abort)) ds_set_error(a.status, DSPARK_ETIMEOUT);
        s_abort = 1;
      }
      if (*reinterpret_cast<volatile int*>(&s_abort)) break;
      ds_tc_fence_after();
      if (any) {
#pragma unroll 1
        for (int ch = ch0; ch < DW_M / 32; ch += chs) {
          float acc[32];
          ds_tmem_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + b * uint32_t(DW_M) + uint32_t(ch * 32), acc);
          const int64_t i0 = tile * DW_M + ch * 32;
          if (live && i0 < a.V) {
            if (!(PREF && dup)) fetch(i0, cur);
            chunk(i0, cur, acc, kbest);
          }
        }
      }
      ds_tc_fence_before();
      __syncwarp();
      if (lane == 0) ds_mbar_arrive(&s_acce[b]);
    }
    if (live && kbest != 0ull) atomicMax(&s_kmax[r], kbest);
    ds_named_sync(1, DW_EPI);                          // every epilogue warp has folded its keys
    for (int rr = tid - DW_EPI_WARP0 * 32; rr < a.R; rr += DW_EPI)
      if (s_kmax[rr] != 0ull) atomicMax(&a.zkey[int64_t(rr) * a.B + a.j], s_kmax[rr]);
  }
  __syncthreads();
  if (warp == DW_MMA_WARP) {
    ds_tc_fence_after();
    ds_tmem_dealloc(tmem, ncols);
  }
}

// ---- sampled positions without a nucleus: draws over the z rows ------------------------------
constexpr int DD_THREADS = 512;
constexpr int DD_WARPS = DD_THREADS / 32;
constexpr int DD_CELL = 256;                 // indices per cell: one warp, eight consecutive a lane
constexpr int DD_PART = 32768;               // indices per CTA (128 cells)

struct DwDraw {
  const float* z;
  int64_t ldz, z_row_mul, z_row_add;         // z row of request r: (r * mul + add) * ldz
  int64_t V, V_t;
  int32_t B, j;
  const unsigned long long* zkey;            // [R, B]
  const uint64_t* seed;
  const uint64_t* step;
  const int64_t* d2t;
  int32_t* out_tgt;                          // [R, B]
  int32_t* out_idx;
  int32_t* prev_cur;                         // [R]
  dspark_qrecord q;                          // dense record statistics (zmax, wsum, wcut, icut) or none
  int has_q;
  int64_t q_row_mul, q_row_add;
  float2* cells;                             // [R, ncell]
  int64_t ncell;
  int32_t* ticket;                           // [R]
  int32_t* status;
};

DS_DEV void dd_emit(const DwDraw& d, int64_t r, int64_t pick, float zmax, double wsum, float wcut, int64_t icut) {
  int64_t tgt = pick;
  if (pick >= 0 && d.d2t) {
    tgt = pick + d.d2t[pick];
    if (tgt < 0 || tgt >= d.V_t) {
      ds_set_error(d.status, DSPARK_ERANGE);
      tgt = -1;
    }
  }
  if (d.out_idx) d.out_idx[r * d.B + d.j] = int32_t(pick);
  d.out_tgt[r * d.B + d.j] = int32_t(tgt);
  d.prev_cur[r] = int32_t(tgt);
  if (d.has_q) {
    const int64_t qrow = r * d.q_row_mul + d.q_row_add;
    d.q.zmax[qrow] = zmax;
    d.q.wsum[qrow] = wsum;
    d.q.wcut[qrow] = wcut;
    d.q.icut[qrow] = int32_t(icut);
  }
}

// Weights of eight z values (zero past V)
DS_DEV void dd_w8(const float* zr, int64_t t, int64_t V, float zmax, float (&w)[8]) {
  float x[8];
  if (t + 8 <= V && (reinterpret_cast<uintptr_t>(zr + t) & 15) == 0) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(zr + t));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(zr + t) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (t + e < V) ? __ldcg(zr + t + e) : -INFINITY;
  }
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 w2 = ds_weight2(__fsub_rn(x[e], zmax), __fsub_rn(x[e + 1], zmax));
    w[e] = w2.x;
    w[e + 1] = w2.y;
  }
}

__global__ void __launch_bounds__(DD_THREADS) dense_walk_draw_kernel(const DwDraw d) {
  __shared__ double s_run[DD_THREADS + 1];
  __shared__ int s_last;
  __shared__ int64_t s_cell, s_pick;
  __shared__ double s_tau;
  ds_pdl_trigger();
  ds_pdl_wait();                                       // z and the maximum keys come from the GEMM
  const int64_t r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float zmax = ds_key64_val(d.zkey[r * d.B + d.j]);
  if (!(zmax > -INFINITY && zmax < INFINITY)) {
    if (blockIdx.x == 0 && tid == 0) {
      ds_set_error(d.status, DSPARK_ENONFINITE);
      if (d.out_idx) d.out_idx[r * d.B + d.j] = -1;
      d.out_tgt[r * d.B + d.j] = -1;
      d.prev_cur[r] = -1;
    }
    return;
  }
  const float* zr = d.z + (r * d.z_row_mul + d.z_row_add) * d.ldz;
  float2* cells = d.cells + r * d.ncell;
  const int64_t t0 = int64_t(blockIdx.x) * DD_PART;
  constexpr int CPP = DD_PART / DD_CELL;
  for (int k0 = warp; k0 < CPP; k0 += 4 * DD_WARPS) {  // four cells per warp in flight
    float w[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t t = t0 + int64_t(k0 + u * DD_WARPS) * DD_CELL + lane * 8;
      if (t < d.V) dd_w8(zr, t, d.V, zmax, w[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = t0 / DD_CELL + k0 + u * DD_WARPS;
      if (c * DD_CELL >= d.V) continue;                // warp-uniform
      const int64_t t = c * DD_CELL + lane * 8;
      rs::FF m{0.0f, 0.0f};
      if (t < d.V) {
#pragma unroll
        for (int e = 0; e < 8; ++e) rs::ff_add(m, w[u][e]);
      }
      const rs::FF cw = rs::warp_ff_reduce(m);
      if (lane == 0) cells[c] = make_float2(cw.hi, cw.lo);
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&d.ticket[r], 1) == int(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the last part: the first kept index whose running sum exceeds u * W_kept
  const int64_t ncell = d.ncell;
  const int64_t per = (ncell + DD_THREADS - 1) / DD_THREADS;
  const int64_t c0 = min(ncell, tid * per), c1 = min(ncell, c0 + per);
  rs::FF mf{0.0f, 0.0f};
  for (int64_t c = c0; c < c1; ++c) {
    const float2 cv = __ldcg(cells + c);
    rs::ff_acc(mf, rs::FF{cv.x, cv.y});
  }
  const double mine = rs::ff_value(mf);
  s_run[tid] = mine;
  __syncthreads();
  if (tid < 32) {
    constexpr int PT = DD_THREADS / 32;
    double loc = 0.0;
#pragma unroll
    for (int q = 0; q < PT; ++q) loc += s_run[lane * PT + q];
    double incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double nb = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += nb;
    }
    double run = incl - loc;
#pragma unroll
    for (int q = 0; q < PT; ++q) {
      const double x = s_run[lane * PT + q];
      s_run[lane * PT + q] = run;
      run += x;
    }
    if (lane == 31) s_run[DD_THREADS] = incl;
  }
  __syncthreads();
  const double before = s_run[tid], total = s_run[DD_THREADS];
  const double u = ds_uniform(d.seed[r], d.step[r], uint32_t(d.j), DS_PURPOSE_DRAFT);
  const double target = u * total;
  if (tid == 0) {
    s_cell = -1;
    s_pick = -1;
    d.ticket[r] = 0;                                   // ready for the next position
  }
  __syncthreads();
  if (mine > 0.0 && target >= before && target < before + mine) {
    double acc = before;
    for (int64_t c = c0; c < c1; ++c) {
      const float2 cv2 = __ldcg(cells + c);
      const double cv = double(cv2.x) + double(cv2.y);
      if (cv > 0.0 && target < acc + cv) {
        s_cell = c;
        s_tau = target - acc;
        break;
      }
      acc += cv;
    }
  }
  __syncthreads();
  if (tid == 0 && s_cell < 0) {                        // rounding: the last cell with mass
    for (int64_t c = ncell - 1; c >= 0; --c) {
      const float2 cv2 = __ldcg(cells + c);
      if (double(cv2.x) + double(cv2.y) > 0.0) {
        s_cell = c;
        s_tau = INFINITY;
        break;
      }
    }
  }
  __syncthreads();
  const int64_t cell = s_cell;
  if (cell >= 0 && warp == 0) {
    const int64_t t = cell * DD_CELL + lane * 8;
    const double tau = s_tau;
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = 0.0f;
    if (t < d.V) dd_w8(zr, t, d.V, zmax, w);
    rs::FF lm{0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < 8; ++e) rs::ff_add(lm, w[e]);
    const double ls = rs::ff_value(lm);
    double incl = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double nb = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += nb;
    }
    const double ex = incl - ls;
    const unsigned withm = __ballot_sync(0xFFFFFFFFu, ls > 0.0);
    const int lastl = withm ? 31 - __clz(int(withm)) : -1;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, ls > 0.0 && tau >= ex && tau < incl);
    const int hl = hit ? __ffs(hit) - 1 : lastl;
    if (lane == hl) {
      double run = ex;
      int64_t pick = -1, last = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (pick < 0 && w[e] > 0.0f) {
          run += double(w[e]);
          last = t + e;
          if (run > tau) pick = t + e;
        }
      }
      s_pick = pick >= 0 ? pick : last;
    }
  }
  __syncthreads();
  if (tid == 0) dd_emit(d, r, s_pick, zmax, total, 0.0f, -1);
}

// Greedy positions: the argmax key is the token (lowest index among equal maxima).
__global__ void dense_walk_greedy_kernel(const DwDraw d, int32_t R) {
  ds_pdl_trigger();
  ds_pdl_wait();
  const int64_t r = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= R) return;
  const unsigned long long key = d.zkey[r * d.B + d.j];
  const float zmax = ds_key64_val(key);
  if (!(zmax > -INFINITY && zmax < INFINITY)) {
    ds_set_error(d.status, DSPARK_ENONFINITE);
    if (d.out_idx) d.out_idx[r * d.B + d.j] = -1;
    d.out_tgt[r * d.B + d.j] = -1;
    d.prev_cur[r] = -1;
    return;
  }
  const int64_t pick = ds_key64_idx(key);
  dd_emit(d, r, pick, zmax, 1.0, 1.0f, pick);
}

// cuTensorMapEncodeTiled, from the driver through the runtime (no link against the driver library)
using DwEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
DwEncodeFn dw_encode_fn() {
  static std::once_flag once;
  static DwEncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<DwEncodeFn>(p);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

// Tensor map of W [V_t, rank] bf16 for stage loads: box 64 elements (128 bytes) x 128 rows.
bool dw_tensor_map(CUtensorMap* m, const void* W, int64_t V_t, int rank) {
  const DwEncodeFn fn = dw_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cuuint64_t(rank), cuuint64_t(V_t)};
  const cuuint64_t strides[1] = {cuuint64_t(rank) * 2};
  const cuuint32_t box[2] = {64, uint32_t(DW_M)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, bool XFORM, bool TONE>
cudaError_t dw_launch_gemm_t(const DwArgs& a, const CUtensorMap& tm, cudaStream_t stream) {
  auto kern = dense_walk_gemm_kernel<T, XFORM, TONE>;
  const size_t smem = size_t(a.rank / 64) * DW_MAXR * 128 + size_t(DW_NS) * DW_STAGE + 1024;
  const cudaError_t e = ds_ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(a.ntiles, int64_t(ds_num_sms()));
  return ds_launch(kern, dim3(unsigned(grid)), dim3(DW_THREADS), smem, stream, a, tm);
}

template <typename T, bool XFORM>
cudaError_t dw_launch_gemm(const DwArgs& a, const CUtensorMap& tm, cudaStream_t stream) {
  return a.Tz == 1.0f ? dw_launch_gemm_t<T, XFORM, true>(a, tm, stream) : dw_launch_gemm_t<T, XFORM, false>(a, tm, stream);
}

size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }

struct DwWs {
  float* gate;                 // [R, B]
  int32_t* prev_cur;           // [R]
  unsigned long long* zkey;    // [R, B]
  int32_t* ticket;             // [R]
  float2* cells;               // [min(R, DW_MAXR), ncell]
  float* zscr;                 // [min(R, DW_MAXR), V] z rows when no record is kept
};

DwWs dw_layout(void* base, int64_t R, int32_t B, int64_t V, size_t* total) {
  const int64_t Rc = std::min<int64_t>(R, DW_MAXR);
  const size_t ncell = size_t((V + DD_CELL - 1) / DD_CELL);
  uint8_t* p = reinterpret_cast<uint8_t*>(base);
  size_t off = 0;
  DwWs w = {};
  auto take = [&](size_t bytes) {
    uint8_t* q = p ? p + off : nullptr;
    off += ws_align(bytes);
    return q;
  };
  w.gate = reinterpret_cast<float*>(take(size_t(R) * B * sizeof(float)));
  w.prev_cur = reinterpret_cast<int32_t*>(take(size_t(R) * sizeof(int32_t)));
  w.zkey = reinterpret_cast<unsigned long long*>(take(size_t(R) * B * sizeof(unsigned long long)));
  w.ticket = reinterpret_cast<int32_t*>(take(size_t(R) * sizeof(int32_t)));
  w.cells = reinterpret_cast<float2*>(take(size_t(Rc) * ncell * sizeof(float2)));
  w.zscr = reinterpret_cast<float*>(take(size_t(Rc) * size_t(V) * sizeof(float)));
  *total = off;
  return w;
}

}  // namespace

extern "C" size_t dspark_internal_ws_dense_walk(int64_t R, int32_t B, int64_t V) {
  size_t total = 0;
  dw_layout(nullptr, R, B, V, &total);
  return total;
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
  size_t need = 0;
  dw_layout(nullptr, R, B, V_d, &need);
  if (!ws || ws_bytes < need || !ds_aligned(ws, 256)) return DSPARK_EWORKSPACE;
  const DwWs w = dw_layout(ws, R, B, V_d, &need);
  cudaStream_t st = stream;
  const bool greedy = !(temperature > 0.0f);
  const bool nucleus = !greedy && top_p < 1.0f;

  if (hidden && hidden_dtype == DSPARK_BF16)
    DS_CUDA_TRY(ds_launch(dense_walk_gate_kernel<__nv_bfloat16>, dim3(unsigned(R * B)), dim3(128), 0, st,
                          reinterpret_cast<const __nv_bfloat16*>(hidden), reinterpret_cast<const __nv_bfloat16*>(g), H,
                          ldh, row_start, B, prev, w.prev_cur, w.gate, w.zkey, w.ticket));
  else
    DS_CUDA_TRY(ds_launch(dense_walk_gate_kernel<float>, dim3(unsigned(R * B)), dim3(128), 0, st,
                          reinterpret_cast<const float*>(hidden), reinterpret_cast<const float*>(g), H, ldh, row_start,
                          B, prev, w.prev_cur, w.gate, w.zkey, w.ticket));

  const bool xform = (mult != 1.0f) || (softcap > 0.0f);
  // contiguous W rows (no d2t) are loaded by TMA; the map is encoded once per call
  alignas(64) CUtensorMap tm;
  memset(&tm, 0, sizeof(tm));
  const bool use_tma = d2t == nullptr && dw_tensor_map(&tm, W, V_t, rank);
  const int Cz = rs::cluster_size_for(V_d, 4);
  DS_REQUIRE(Cz > 0);
  const int64_t ncell = (V_d + DD_CELL - 1) / DD_CELL;
  for (int64_t c0 = 0; c0 < R; c0 += DW_MAXR) {
    const int32_t Rc = int32_t(std::min<int64_t>(DW_MAXR, R - c0));
    DwArgs a = {};
    a.logits = reinterpret_cast<const uint8_t*>(logits) + (row_start ? 0 : c0 * B * ld * ds_dtype_size(dtype));
    a.ld = ld;
    a.row_start = row_start ? row_start + c0 : nullptr;
    a.B = B;
    a.R = Rc;
    a.rank = rank;
    a.V = V_d;
    a.V_t = V_t;
    a.ntiles = (V_d + DW_M - 1) / DW_M;
    a.prev_cur = w.prev_cur + c0;
    a.E = reinterpret_cast<const __nv_bfloat16*>(E);
    a.W = reinterpret_cast<const __nv_bfloat16*>(W);
    a.d2t = d2t;
    a.gate = w.gate + c0 * B;
    a.mult = mult;
    a.softcap = softcap;
    a.Tz = temperature > 0.0f ? temperature : 1.0f;
    a.zkey = w.zkey + c0 * B;
    a.status = dev_status;
    a.first_wait = g_ds_first_wait_polls.load(std::memory_order_relaxed);
    a.use_tma = use_tma ? 1 : 0;
    if (record) {
      a.z = q->z + c0 * B * q->ldz;
      a.ldz = q->ldz;
      a.z_row_mul = B;
    } else {
      a.z = w.zscr;
      a.ldz = V_d;
      a.z_row_mul = 1;
    }
    // draws without a nucleus, and greedy positions
    DwDraw d = {};
    d.z = a.z;
    d.ldz = a.ldz;
    d.z_row_mul = a.z_row_mul;
    d.V = V_d;
    d.V_t = V_t;
    d.B = B;
    d.zkey = a.zkey;
    d.seed = seed ? seed + c0 : nullptr;
    d.step = step ? step + c0 : nullptr;
    d.d2t = d2t;
    d.out_tgt = out_tgt + c0 * B;
    d.out_idx = out_idx ? out_idx + c0 * B : nullptr;
    d.prev_cur = w.prev_cur + c0;
    d.cells = w.cells;
    d.ncell = ncell;
    d.ticket = w.ticket + c0;
    d.status = dev_status;
    if (record) {
      d.q = *q;
      d.q.zmax = q->zmax + c0 * B;
      d.q.wsum = q->wsum + c0 * B;
      d.q.wcut = q->wcut + c0 * B;
      d.q.icut = q->icut + c0 * B;
      d.has_q = 1;
      d.q_row_mul = B;
    }
    // nucleus positions: the row sampler over the z rows
    rs::SampleArgs sa = {};
    sa.rows = a.z;
    sa.V = V_d;
    sa.ld = a.ldz;
    sa.row_mul = a.z_row_mul;
    sa.B = 1;
    sa.C = Cz;
    sa.mult = 1.0f;
    sa.softcap = 0.0f;
    sa.T = 1.0f;                                   // the rows already hold z = v / T
    sa.top_p = top_p;
    sa.seed = d.seed;
    sa.step = d.step;
    sa.d2t = d2t;
    sa.V_t = V_t;
    sa.out_tgt = d.out_tgt;
    sa.out_idx = d.out_idx;
    sa.out_mul = B;
    sa.prev_out = d.prev_cur;
    sa.status = dev_status;
    if (record) {
      sa.q = d.q;
      sa.q_mode = 2;
      sa.q_row_mul = B;
    }
    for (int32_t j = 0; j < B; ++j) {
      a.j = j;
      a.z_row_add = record ? j : 0;
      cudaError_t e;
      if (dtype == DSPARK_BF16)
        e = xform ? dw_launch_gemm<__nv_bfloat16, true>(a, tm, st) : dw_launch_gemm<__nv_bfloat16, false>(a, tm, st);
      else
        e = xform ? dw_launch_gemm<float, true>(a, tm, st) : dw_launch_gemm<float, false>(a, tm, st);
      DS_CUDA_TRY(e);
      d.j = j;
      d.z_row_add = a.z_row_add;
      d.q_row_add = j;
      if (greedy) {
        DS_CUDA_TRY(ds_launch(dense_walk_greedy_kernel, dim3(unsigned((Rc + 127) / 128)), dim3(128), 0, st, d, Rc));
      } else if (!nucleus) {
        const dim3 grid(unsigned((V_d + DD_PART - 1) / DD_PART), unsigned(Rc));
        DS_CUDA_TRY(ds_launch(dense_walk_draw_kernel, grid, dim3(DD_THREADS), 0, st, d));
      } else {
        sa.row_base = record ? j : 0;
        sa.position = j;
        sa.out_add = j;
        sa.q_row_add = j;
        DS_CUDA_TRY(rs::sample_rows(sa, Rc, 0, 0, st));
      }
    }
  }
  return DSPARK_OK;
}
