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
//     vocabulary in 128-row tiles, D[vocabulary, request] = W[m(i)] . E[prev]^T: TMEM lanes are the
//     tile's vocabulary rows, columns the requests. The W rows m(i) of a tile go into a ring of
//     128-byte swizzled K-chunks, one stage per mbarrier (one TMA copy per stage when the rows are
//     contiguous, no d2t; else two producer warps gathering them with cp.async). Two loader warps
//     stage the tile's logits of every request into shared memory. One thread issues the MMAs
//     (M = 128 vocabulary rows, N = the requests rounded up to 16, K = rank) into one of two or
//     four TMEM accumulators; the epilogue warps drain another, one vocabulary index per lane, so
//     each load and store of a warp is one contiguous stretch of one request's row, and write
//     z = (s + gamma tau) / T into the dense record (or the workspace). Every lane keeps the running
//     largest (z, lowest index) key of its index for each request (or the warp reduces them per
//     tile), then the CTA and the GPU fold them. The table, the logits and z are all streamed once
//     per position with an L2 evict-first policy: the 78 MB table does not stay in L2 next to the
//     other streams, and marking it evict-last only pushes out the z rows the draw reads next.
//  2. sampled positions without a nucleus: dense_walk_draw_kernel - the z rows (mostly from L2)
//     in parts over one wave of CTAs: weights of z - zmax, the kept mass of every cell of 1024
//     indices; the part that finishes last draws the token with float-pair running sums over the
//     cells, then the cell's elements, and writes it as the next position's previous token. Greedy
//     positions finish with the argmax key (dense_walk_greedy_kernel); nucleus positions use the
//     row sampler of sample.cu on the z rows.
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int DW_M = 128;                    // vocabulary rows per tile (MMA M)
constexpr int DW_MAXR = 128;                 // requests per GEMM launch with bf16 logits (MMA N <= 128)
constexpr int DW_MAXR_F32 = 64;              // with float32 logits (their staged tiles are twice as large)
constexpr int DW_NS_MAX = 8;                 // K-chunk stages of the W ring (16 KB each)
constexpr int DW_NL_MAX = 4;                 // staged logits tiles
constexpr int DW_WPROD = 64;                 // W producers (warps 0-1; thread 0 alone with TMA)
constexpr int DW_LOAD0 = 64;                 // logits loaders (warps 2-3)
constexpr int DW_LOAD = 64;
constexpr int DW_MMA_WARP = 4;
constexpr int DW_EPI_WARP0 = 5;              // epilogue warps 5..12
constexpr int DW_EPI = 256;
constexpr int DW_THREADS = DW_WPROD + DW_LOAD + 32 + DW_EPI;
constexpr uint32_t DW_STAGE = DW_M * 128;    // bytes of one K-chunk of a tile
constexpr size_t DW_SMEM_BUDGET = 216 * 1024;

struct DwArgs {
  const void* logits;
  int64_t ld;
  const int64_t* row_start;
  int32_t B, j, R, Rp, rank, ns, nl;
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
  int lvec;                  // every logits row starts on a 16-byte boundary
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

// D[vocabulary, request] = W[m(i)] . E[prev]^T: TMEM lanes are the tile's 128 vocabulary rows and
// columns the requests (N = R rounded up to 16), so an epilogue lane owns one vocabulary index and
// every load and store of a warp is one contiguous stretch of one request's row.
template <typename T, bool XFORM, bool TONE>
__global__ void __launch_bounds__(DW_THREADS, 1) dense_walk_gemm_kernel(const DwArgs a,
                                                                       const __grid_constant__ CUtensorMap tmW) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_full[DW_NS_MAX], s_empty[DW_NS_MAX], s_lfull[DW_NL_MAX], s_lempty[DW_NL_MAX];
  __shared__ uint64_t s_accf[4], s_acce[4], s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int32_t s_prev[DW_MAXR];
  __shared__ float s_gate[DW_MAXR];
  __shared__ int64_t s_lrow[DW_MAXR];
  __shared__ unsigned long long s_kmax[DW_MAXR];

  const int R = a.R, Rp = a.Rp, ns = a.ns, nl = a.nl, nkb = a.rank / 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = base;                                           // ns x [128 vocabulary rows x 128 B]
  uint8_t* sA = sW + size_t(ns) * DW_STAGE;                     // nkb x [Rp request rows x 128 B]
  T* sL = reinterpret_cast<T*>(sA + size_t(nkb) * Rp * 128);    // nl x [Rp requests x 128 logits]
  const size_t lstride = size_t(Rp) * DW_M;                     // elements of one staged logits tile
  constexpr uint32_t ncols = 2 * DW_M;                          // tensor memory columns taken
  const uint32_t acs = Rp <= 64 ? 64u : 128u;                   // columns of one accumulator
  const uint32_t nacc = ncols / acs;                            // 4 or 2 accumulators

  ds_pdl_trigger();
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      ds_mbar_init(&s_full[s], a.use_tma ? 1 : DW_WPROD);
      ds_mbar_init(&s_empty[s], 1);
    }
    for (int l = 0; l < nl; ++l) {
      ds_mbar_init(&s_lfull[l], DW_LOAD);
      ds_mbar_init(&s_lempty[l], DW_EPI / 32);
    }
    for (uint32_t b = 0; b < nacc; ++b) {
      ds_mbar_init(&s_accf[b], 1);
      ds_mbar_init(&s_acce[b], DW_EPI / 32);
    }
    ds_mbar_init(&s_drain, 1);
    s_abort = 0;
  }
  for (int r = tid; r < DW_MAXR; r += DW_THREADS) {
    if (r < R) s_lrow[r] = a.row_start ? a.row_start[r] + a.j : int64_t(r) * a.B + a.j;
    s_kmax[r] = 0ull;
  }
  __syncthreads();
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(&s_abort) != 0; };
  auto wait = [&](uint64_t* bar, uint32_t parity, uint32_t limit) {
    if (!ds_mbar_wait_or_abort(bar, parity, limit, &s_abort)) {
      if (!aborted()) ds_set_error(a.status, DSPARK_ETIMEOUT);
      s_abort = 1;
    }
    return !aborted();
  };

  // The table and the logits are inputs that no kernel of this library writes, so the producers
  // and loaders start before the wait for the previous kernel; the previous tokens (the B operand),
  // the gates and everything written come after it.
  if (warp < DW_WPROD / 32 && a.use_tma) {
    // ---- W producer: one thread loads each K-chunk of a tile (128 contiguous W rows x 128 bytes,
    // 128-byte swizzle) with one TMA copy; rows past the table read as zero ----
    if (tid == 0) {
      const uint64_t pol = ds_policy_evict_first();
      uint32_t g = 0;
      for (int64_t tile = blockIdx.x; tile < a.ntiles && !aborted(); tile += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const uint32_t s = g % ns, ph = (g / ns) & 1u;
          if (!wait(&s_empty[s], ph ^ 1u, DS_WAIT_LIMIT)) break;
          ds_mbar_arrive_expect_tx(&s_full[s], DW_STAGE);
          ds_tma_load_2d(sW + s * DW_STAGE, &tmW, kb * 64, int32_t(tile * DW_M), &s_full[s], pol);
        }
      }
      // every TMA copy this thread issued lands before the CTA leaves (or the wait gives up)
      for (uint32_t k = (g > uint32_t(ns) ? g - ns : 0); k < g; ++k)
        (void)ds_mbar_wait(&s_full[k % ns], (k / ns) & 1u, DS_WAIT_LIMIT);
    }
    __syncwarp();
  } else if (warp < DW_WPROD / 32) {
    // ---- W producers (gathered rows m(i) = i + d2t[i]): thread p copies 16-byte column p % 8 of
    // rows p / 8 + 8 kk of each K-chunk ----
    const uint64_t pol = ds_policy_evict_first();
    const int cc = tid & 7, m0 = tid >> 3;
    uint32_t g = 0;
    for (int64_t tile = blockIdx.x; tile < a.ntiles && !aborted(); tile += gridDim.x) {
      const int64_t i0 = tile * DW_M;
      int64_t rid[16];
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const int64_t i = i0 + m0 + 8 * kk;
        int64_t t = -2;                                // -2: past the vocabulary (row never read)
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
        const uint32_t s = g % ns, ph = (g / ns) & 1u;
        if (!wait(&s_empty[s], ph ^ 1u, DS_WAIT_LIMIT)) break;
        uint8_t* stage = sW + s * DW_STAGE;
        bool zeroed = false;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const int m = m0 + 8 * kk;
          uint8_t* dst = stage + m * 128 + ((cc ^ (m & 7)) << 4);
          if (rid[kk] >= 0) {
            ds_cp_async16_hint(dst, a.W + rid[kk] * a.rank + kb * 64 + cc * 8, pol);
          } else if (rid[kk] == -1) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            zeroed = true;
          }
        }
        if (zeroed) ds_fence_proxy_async_smem();
        ds_cp_async_mbar_arrive(&s_full[s]);
      }
    }
    ds_cp_async_wait_all();                            // no copy lands after the CTA is gone
  } else if (warp < (DW_WPROD + DW_LOAD) / 32) {
    // ---- logits loaders: the tile's 128 logits of every request into [request][128], read once
    // (L2 evict first); a ragged last tile or unaligned rows go element by element ----
    const uint64_t pol = ds_policy_evict_first();
    const int lt = tid - DW_LOAD0;
    constexpr int EPV = 16 / int(sizeof(T));           // elements per 16-byte copy
    constexpr int CPR = DW_M / EPV;                    // copies per request row
    const T* lg = reinterpret_cast<const T*>(a.logits);
    uint32_t k = 0;
    for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++k) {
      const uint32_t lb = k % nl, ph = (k / nl) & 1u;
      if (!wait(&s_lempty[lb], ph ^ 1u, DS_WAIT_LIMIT)) break;
      T* dst = sL + lb * lstride;
      const int64_t v0 = tile * DW_M;
      if (a.lvec && v0 + DW_M <= a.V) {
        for (int t = lt; t < R * CPR; t += DW_LOAD) {
          const int cr = t / CPR, c = t % CPR;
          ds_cp_async16_hint(dst + cr * DW_M + c * EPV, lg + s_lrow[cr] * a.ld + v0 + c * EPV, pol);
        }
        ds_cp_async_mbar_arrive(&s_lfull[lb]);
      } else {
        for (int t = lt; t < R * DW_M; t += DW_LOAD) {
          const int cr = t / DW_M, c = t % DW_M;
          dst[cr * DW_M + c] = (v0 + c < a.V) ? lg[s_lrow[cr] * a.ld + v0 + c] : T(0.0f);
        }
        ds_cp_async_wait_all();
        ds_mbar_arrive(&s_lfull[lb]);
      }
    }
    ds_cp_async_wait_all();
  } else {
    // ---- after the previous kernel: the MMA warp takes tensor memory, the epilogue warps stage
    // the B operand E[prev_r] (zero rows past R and for bad ids) ----
    ds_pdl_wait();
    if (warp == DW_MMA_WARP) {
      ds_tmem_alloc(&s_tmem, ncols);
    } else {
      const int et = tid - DW_EPI_WARP0 * 32;
      for (int r = et; r < Rp; r += DW_EPI) {
        int32_t p = -1;
        float gm = 0.0f;
        if (r < R) {
          p = a.prev_cur[r];
          if (p < 0 || p >= a.V_t) {
            ds_set_error(a.status, DSPARK_ERANGE);
            p = -1;
          }
          gm = a.gate[int64_t(r) * a.B + a.j];
        }
        s_prev[r] = p;
        s_gate[r] = gm;
      }
      ds_named_sync(1, DW_EPI);
      const int cpr = a.rank / 8;
      for (int t = et; t < Rp * cpr; t += DW_EPI) {
        const int m = t / cpr, c = t % cpr, kb = c >> 3, cc = c & 7;
        uint8_t* dst = sA + kb * (Rp * 128) + m * 128 + ((cc ^ (m & 7)) << 4);
        const int32_t id = s_prev[m];
        if (id >= 0) ds_cp_async16(dst, a.E + int64_t(id) * a.rank + c * 8);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
      ds_cp_async_wait_all();
      ds_fence_proxy_async_smem();
    }
    ds_tc_fence_before();
    ds_named_sync(2, 32 + DW_EPI);
    ds_tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == DW_MMA_WARP) {
      // ---- one thread issues the MMAs; the accumulator buffers alternate by tile ----
      if (lane == 0) {
        const uint32_t idesc = ds_idesc_bf16_f32(DW_M, Rp);
        const uint32_t waddr = ds_smem_addr(sW), aaddr = ds_smem_addr(sA);
        uint32_t g = 0, k = 0;
        for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++k) {
          const uint32_t b = k % nacc, use = k / nacc;
          if (!wait(&s_acce[b], (use & 1u) ^ 1u, DS_WAIT_LIMIT)) break;
          ds_tc_fence_after();
          const uint32_t dacc = tmem + b * acs;
          bool stop = false;
          for (int kb = 0; kb < nkb; ++kb, ++g) {
            const uint32_t s = g % ns, ph = (g / ns) & 1u;
            if (!wait(&s_full[s], ph, DS_WAIT_LIMIT)) {
              stop = true;
              break;
            }
            ds_tc_fence_after();
#pragma unroll
            for (int sub = 0; sub < 4; ++sub) {
              const uint64_t wd = ds_smem_desc_sw128(waddr + s * DW_STAGE + sub * 32);
              const uint64_t ed = ds_smem_desc_sw128(aaddr + kb * (Rp * 128) + sub * 32);
              ds_umma_f16(dacc, wd, ed, idesc, (kb | sub) != 0);
            }
            ds_umma_commit(&s_empty[s]);               // the stage is free once these MMAs are done
          }
          if (stop) break;
          ds_umma_commit(&s_accf[b]);                  // the tile's accumulator is complete
        }
        // every MMA this thread issued completes before tensor memory is released
        ds_umma_commit(&s_drain);
        (void)ds_mbar_wait(&s_drain, 0, DS_WAIT_LIMIT);
      }
      __syncwarp();
    } else {
      // ---- epilogue: warp (q, h) reads TMEM lanes 32 q.. (vocabulary rows) and the 32-request
      // column chunks h, h + 2; per request the warp reduces its 32 keys (largest z, lowest index)
      // and lane c keeps the running best of request 32 kc + c ----
      const int q = warp & 3, h = (warp - DW_EPI_WARP0) >> 2;
      const int ql = q * 32 + lane;
      const int64_t zstep = a.z_row_mul * a.ldz;
      // With one chunk a warp (R <= 64) and at most 255 tiles a CTA, every lane keeps the running
      // best key of its own index for each of the chunk's 32 requests, with the tile ordinal of
      // that best in a byte, and the warp reduces them once at the end; otherwise each request's
      // 32 keys are reduced across the warp at every tile.
      const bool regmax = Rp <= 64 && (a.ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x <= 255;
      uint32_t bk[32], bt[8];
#pragma unroll
      for (int c = 0; c < 32; ++c) bk[c] = 0u;
#pragma unroll
      for (int c = 0; c < 8; ++c) bt[c] = 0u;
      uint32_t best[2] = {0u, 0u}, bidx[2] = {0u, 0u};
      uint32_t k = 0;
      bool first = true;
      for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x, ++k) {
        const uint32_t b = k % nacc, use = k / nacc, lb = k % nl;
        if (!wait(&s_accf[b], use & 1u, first ? a.first_wait : DS_WAIT_LIMIT)) break;
        first = false;
        if (!wait(&s_lfull[lb], (k / nl) & 1u, DS_WAIT_LIMIT)) break;
        ds_tc_fence_after();
        const int64_t v = tile * DW_M + ql;
        const bool valid = v < a.V;
        const T* L = sL + lb * lstride + ql;
        float* zv = a.z + a.z_row_add * a.ldz + v;
        if (regmax) {
          if (h * 32 < R) {                            // warp-uniform
            float acc[32];
            ds_tmem_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + b * acs + uint32_t(h * 32), acc);
            float* zp = zv + int64_t(h * 32) * zstep;
#pragma unroll
            for (int c = 0; c < 32; ++c, zp += zstep) {
              const int cr = h * 32 + c;
              if (cr >= R) break;                      // warp-uniform
              const float x = dw_xform<XFORM>(ds_load_elem<T>(L + cr * DW_M), a.mult, a.softcap);
              const float zc = ds_temper_t<TONE>(__fmaf_rn(s_gate[cr], acc[c], x), a.Tz);
              if (valid) *zp = zc;
              const uint32_t ob = valid ? ds_key32(ds_canon_zero(zc)) : 0u;
              const bool up = ob > bk[c];              // ties keep the earlier tile (lower index)
              bk[c] = up ? ob : bk[c];
              bt[c >> 2] = up ? ((bt[c >> 2] & ~(0xFFu << (8 * (c & 3)))) | (k << (8 * (c & 3)))) : bt[c >> 2];
            }
          }
        } else {
#pragma unroll
          for (int sc = 0; sc < 2; ++sc) {
            const int kc = h + 2 * sc;
            if (kc * 32 >= R) break;                   // warp-uniform
            float acc[32];
            ds_tmem_ld_32x32b_x32(tmem + (uint32_t(q * 32) << 16) + b * acs + uint32_t(kc * 32), acc);
            float* zp = zv + int64_t(kc * 32) * zstep;
            uint32_t tmx = 0u, tbal = 0u;              // lane c: the tile's best of request 32 kc + c
#pragma unroll
            for (int c = 0; c < 32; ++c, zp += zstep) {
              const int cr = kc * 32 + c;
              if (cr >= R) break;                      // warp-uniform
              const float x = dw_xform<XFORM>(ds_load_elem<T>(L + cr * DW_M), a.mult, a.softcap);
              const float zc = ds_temper_t<TONE>(__fmaf_rn(s_gate[cr], acc[c], x), a.Tz);
              if (valid) *zp = zc;
              const uint32_t ob = valid ? ds_key32(ds_canon_zero(zc)) : 0u;
              const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, ob);
              const unsigned bal = __ballot_sync(0xFFFFFFFFu, ob == mx);
              tmx = lane == c ? mx : tmx;
              tbal = lane == c ? bal : tbal;
            }
            if (tmx > best[sc]) {                      // ties keep the earlier tile (lower indices)
              best[sc] = tmx;
              bidx[sc] = uint32_t(tile * DW_M + q * 32 + __ffs(int(tbal)) - 1);
            }
          }
        }
        ds_tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ds_mbar_arrive(&s_acce[b]);
          ds_mbar_arrive(&s_lempty[lb]);
        }
      }
      if (regmax) {
        // per request: the largest (key, lowest index) over the warp's lanes
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int cr = h * 32 + c;
          if (cr >= R) break;                          // warp-uniform
          const uint32_t kt = (bt[c >> 2] >> (8 * (c & 3))) & 0xFFu;
          const uint32_t vi = uint32_t((int64_t(blockIdx.x) + int64_t(kt) * gridDim.x) * DW_M + ql);
          unsigned long long key = bk[c] ? ((static_cast<unsigned long long>(bk[c]) << 32) | (0xFFFFFFFFull - vi)) : 0ull;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, key, o);
            key = other > key ? other : key;
          }
          if (lane == 0 && key != 0ull) atomicMax(&s_kmax[cr], key);
        }
      } else {
#pragma unroll
        for (int sc = 0; sc < 2; ++sc) {
          const int cr = (h + 2 * sc) * 32 + lane;
          if (cr < R && best[sc] != 0u)
            atomicMax(&s_kmax[cr], (static_cast<unsigned long long>(best[sc]) << 32) | (0xFFFFFFFFull - bidx[sc]));
        }
      }
      ds_named_sync(1, DW_EPI);                        // every epilogue warp has folded its keys
      for (int rr = tid - DW_EPI_WARP0 * 32; rr < R; rr += DW_EPI)
        if (s_kmax[rr] != 0ull) atomicMax(&a.zkey[int64_t(rr) * a.B + a.j], s_kmax[rr]);
    }
  }
  __syncthreads();
  if (warp == DW_MMA_WARP) {
    ds_tc_fence_after();
    ds_tmem_dealloc(s_tmem, ncols);
  }
}

// ---- sampled positions without a nucleus: draws over the z rows ------------------------------
constexpr int DD_THREADS = 256;
constexpr int DD_WARPS = DD_THREADS / 32;
constexpr int DD_CELL = 1024;                // indices per cell: one warp, 32 a lane

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
  int64_t ncell, part_cells;                 // cells of a row, cells of one CTA
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

// Four z values from t on (minus infinity past V; a vector load when whole and aligned)
DS_DEV float4 dd_ld4(const float* zr, int64_t t, int64_t V, bool vec) {
  if (vec && t + 4 <= V) return __ldcg(reinterpret_cast<const float4*>(zr + t));
  float4 x;
  x.x = (t < V) ? __ldcg(zr + t) : -INFINITY;
  x.y = (t + 1 < V) ? __ldcg(zr + t + 1) : -INFINITY;
  x.z = (t + 2 < V) ? __ldcg(zr + t + 2) : -INFINITY;
  x.w = (t + 3 < V) ? __ldcg(zr + t + 3) : -INFINITY;
  return x;
}

// Kept mass of cell c (indices c * 1024 ..): lane l weighs the four values at k * 128 + 4 l for
// k = 0..7 (each load of the warp is 512 contiguous bytes) and the warp adds its float pairs.
DS_DEV rs::FF dd_cell_mass(const float* zr, int64_t c, int64_t V, float zmax, bool vec, int lane) {
  float4 x[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = dd_ld4(zr, c * DD_CELL + k * 128 + lane * 4, V, vec);
  rs::FF2 acc{0ull, 0ull};
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 w01 = ds_weight2(__fsub_rn(x[k].x, zmax), __fsub_rn(x[k].y, zmax));
    const float2 w23 = ds_weight2(__fsub_rn(x[k].z, zmax), __fsub_rn(x[k].w, zmax));
    rs::ff2_add(acc, ds_f2(w01.x, w01.y));
    rs::ff2_add(acc, ds_f2(w23.x, w23.y));
  }
  return rs::warp_ff_reduce(rs::ff2_fold(acc));
}

__global__ void __launch_bounds__(DD_THREADS, 3) dense_walk_draw_kernel(const DwDraw d) {
  __shared__ rs::PickShared<DD_THREADS> s_pk;
  __shared__ int s_last;
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
  const int64_t cbeg = int64_t(blockIdx.x) * d.part_cells, cend = min(d.ncell, cbeg + d.part_cells);
  const bool vec = (reinterpret_cast<uintptr_t>(zr) & 15) == 0;
  for (int64_t c = cbeg + warp; c < cend; c += DD_WARPS) {
    const rs::FF cw = dd_cell_mass(zr, c, d.V, zmax, vec, lane);
    if (lane == 0) cells[c] = make_float2(cw.hi, cw.lo);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&d.ticket[r], 1) == int(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the last part: the first kept index whose running sum exceeds u * W_kept (float pairs)
  if (tid == 0) d.ticket[r] = 0;                       // ready for the next position
  rs::pick_cell<DD_THREADS>(cells, d.ncell, rs::ff_uniform(d.seed[r], d.step[r], uint32_t(d.j), DS_PURPOSE_DRAFT), s_pk);
  const int64_t cell = s_pk.cell == ~0ull ? -1 : int64_t(s_pk.cell);
  if (warp == 0) {
    int64_t pick = -1;
    if (cell >= 0) {
      // the cell in index order: lane l holds indices t .. t + 31, t = cell * 1024 + 32 l
      const int64_t t = cell * DD_CELL + lane * 32;
      rs::FF w[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float4 x = dd_ld4(zr, t + 4 * k, d.V, vec);
        const float2 w01 = ds_weight2(__fsub_rn(x.x, zmax), __fsub_rn(x.y, zmax));
        const float2 w23 = ds_weight2(__fsub_rn(x.z, zmax), __fsub_rn(x.w, zmax));
        w[4 * k] = rs::FF{w01.x, 0.0f};
        w[4 * k + 1] = rs::FF{w01.y, 0.0f};
        w[4 * k + 2] = rs::FF{w23.x, 0.0f};
        w[4 * k + 3] = rs::FF{w23.y, 0.0f};
      }
      pick = rs::warp_pick<32>(w, s_pk.tau, s_pk.tinf != 0, cell * DD_CELL);
    }
    if (lane == 0) dd_emit(d, r, pick, zmax, rs::ff_value(s_pk.total), 0.0f, -1);
  }
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

// Shared memory of one GEMM CTA: the W ring, the B operand and the staged logits tiles. The ring
// and the logits tiles take what the budget leaves after the B operand (at least 4 and 2).
void dw_plan_smem(DwArgs& a, size_t elem) {
  const size_t abytes = size_t(a.rank / 64) * a.Rp * 128, lbytes = size_t(a.Rp) * DW_M * elem;
  int nl = DW_NL_MAX;
  while (nl > 2 && abytes + nl * lbytes + 4 * size_t(DW_STAGE) > DW_SMEM_BUDGET) --nl;
  a.nl = nl;
  a.ns = int(std::min<size_t>(DW_NS_MAX, (DW_SMEM_BUDGET - abytes - nl * lbytes) / DW_STAGE));
}
size_t dw_smem_bytes(const DwArgs& a, size_t elem) {
  return size_t(a.ns) * DW_STAGE + size_t(a.rank / 64) * a.Rp * 128 + size_t(a.nl) * a.Rp * DW_M * elem + 1024;
}

template <typename T, bool XFORM, bool TONE>
cudaError_t dw_launch_gemm_t(const DwArgs& a, const CUtensorMap& tm, cudaStream_t stream) {
  auto kern = dense_walk_gemm_kernel<T, XFORM, TONE>;
  const size_t smem = dw_smem_bytes(a, sizeof(T));
  const cudaError_t e = ds_ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(a.ntiles, int64_t(ds_num_sms()));
  return ds_launch(kern, dim3(unsigned(grid)), dim3(DW_THREADS), smem, stream, a, tm);
}

template <typename T, bool XFORM>
cudaError_t dw_launch_gemm(const DwArgs& a, const CUtensorMap& tm, cudaStream_t stream) {
  return a.Tz == 1.0f ? dw_launch_gemm_t<T, XFORM, true>(a, tm, stream) : dw_launch_gemm_t<T, XFORM, false>(a, tm, stream);
}

// Draw CTAs resident on the whole GPU at once
int dd_ctas_per_wave() {
  static std::once_flag once;
  static int per_sm = 1;
  std::call_once(once, [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dense_walk_draw_kernel, DD_THREADS, 0) == cudaSuccess && n > 0)
      per_sm = n;
    else
      (void)cudaGetLastError();
  });
  return per_sm * ds_num_sms();
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
  const int64_t G = dtype == DSPARK_BF16 ? DW_MAXR : DW_MAXR_F32;   // requests per GEMM launch
  const size_t esz = ds_dtype_size(dtype);
  const bool lvec = ds_aligned(logits, 16) && (ld * int64_t(esz)) % 16 == 0;
  for (int64_t c0 = 0; c0 < R; c0 += G) {
    const int32_t Rc = int32_t(std::min<int64_t>(G, R - c0));
    DwArgs a = {};
    a.logits = reinterpret_cast<const uint8_t*>(logits) + (row_start ? 0 : c0 * B * ld * ds_dtype_size(dtype));
    a.ld = ld;
    a.row_start = row_start ? row_start + c0 : nullptr;
    a.B = B;
    a.R = Rc;
    a.Rp = (Rc + 15) / 16 * 16;
    a.rank = rank;
    dw_plan_smem(a, esz);
    a.lvec = lvec ? 1 : 0;
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
    {  // one wave of draw CTAs: the parts of a row split the cells evenly
      const int64_t parts = std::max<int64_t>(1, std::min<int64_t>(ncell, int64_t(dd_ctas_per_wave()) / Rc));
      d.part_cells = (ncell + parts - 1) / parts;
    }
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
        const dim3 grid(unsigned((ncell + d.part_cells - 1) / d.part_cells), unsigned(Rc));
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
