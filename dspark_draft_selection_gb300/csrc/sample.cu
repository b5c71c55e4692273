// sample.cu - full-row multinomial drafting with the proposal record (dspark_sample), and the
// row sampler the dense Markov walk reuses on its biased rows.
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"): Change > Sampled drafting (draw with the draft RNG, record the
// distribution q of every candidate); the commit on the thresholded TopPFilter (nucleus = shortest
// prefix of tokens ordered by probability, ties by index, whose mass exceeds top_p; candidates
// gathered by thresholds p_max e^-10, e^-20, e^-40, then all; exponents below -64 flushed); the
// commit on double-precision multinomial sums; the commit on the double uniform.
//
// One block of 512 threads per row, persistent over rows (two blocks per SM on the plain path,
// one with a nucleus, a transform or a sparse record). When the rows are fewer than the blocks
// that fit, each row is split into P = 2, 4 or 8 parts run by the blocks of one cluster, which
// exchange their maxima and masses through distributed shared memory. The row streams through
// the block in passes (16-byte loads, several chunks in flight per thread; repeated passes mostly
// hit L2): the maximum of z = s / T (and the dense record's z row), the nucleus when top-p < 1
// (a radix select on the weight bits by mass, then the few weights of the crossing digit sorted in
// shared memory), then the kept mass of every cell of 32 vectors as a
// float pair (2Sum), turned into double once per thread rather than once per cell, since the
// FP64 pipe is costly per warp instruction. A block scan over the cells locates the one whose
// running sum crosses u * W_kept; its warp re-reads those 32 vectors and finds the lane, then
// the element.
#include <cfloat>

#include <cooperative_groups.h>

#include "host_common.h"
#include "rowsample.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int SP_CAP = 1024;   // nucleus candidates sorted at the cut



template <bool XFORM>
DS_DEV float sp_xform(float x, float mult, float softcap) {
  if (XFORM) {
    if (mult != 1.0f) x = __fmul_rn(x, mult);
    if (softcap > 0.0f) x = __fmul_rn(softcap, tanhf(__fdiv_rn(x, softcap)));
  }
  return x;
}

DS_DEV bool sp_keep(float w, int64_t i, float wcut, int64_t icut) {
  return w > 0.0f && (w > wcut || (w == wcut && i <= icut));
}

// Geometry of one row: scalar head up to 16-byte alignment, vectors in chunks of SR_THREADS (one
// per thread), scalar tail. Index order: head, chunk 0 (thread order), chunk 1, ..., tail; the
// vectors of warp w in chunk c form cell c * WARPS + w.
constexpr int SR_THREADS = rs::THREADS;
constexpr int SR_WARPS = rs::WARPS;
constexpr int SR_U = 4;                      // chunks loaded together by a thread (bytes in flight)
constexpr int SR_MAXCHUNK = 128;             // rows of up to 128 x 512 vectors
constexpr int SR_CELLS = SR_MAXCHUNK * SR_WARPS;
constexpr int SR_MAXP = 8;                   // parts (cluster blocks) per row
// nucleus scratch: candidate keys, then 16 digit accumulators (float pair + count) per thread
constexpr size_t SP_NUC_BYTES = sizeof(uint64_t) * SP_CAP + size_t(16) * SR_THREADS * (sizeof(float2) + sizeof(uint32_t));

template <typename T>
struct SrRow {
  const T* row;
  int64_t head, nvec, tail0, ntail;
  int nchunk;
  int c_lo, c_hi;                  // this block's chunks (a part of the row when P > 1)
  bool own_head, own_tail;
};

template <typename T>
DS_DEV SrRow<T> sr_row(const T* row, int64_t V) {
  constexpr int EPV = 16 / sizeof(T);
  SrRow<T> g;
  g.row = row;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  g.head = int64_t(((16u - (addr & 15u)) & 15u) / sizeof(T));
  if (g.head > V) g.head = V;
  g.nvec = (V - g.head) / EPV;
  g.tail0 = g.head + g.nvec * EPV;
  g.ntail = V - g.tail0;
  g.nchunk = int((g.nvec + SR_THREADS - 1) / SR_THREADS);
  g.c_lo = 0;
  g.c_hi = g.nchunk;
  g.own_head = g.own_tail = true;
  return g;
}

// Restricts a row to part p of P (contiguous chunk ranges; the head goes with part 0, the tail
// with part P - 1).
template <typename T>
DS_DEV void sr_part(SrRow<T>& g, int p, int P) {
  const int per = (g.nchunk + P - 1) / P;
  g.c_lo = min(g.nchunk, p * per);
  g.c_hi = min(g.nchunk, g.c_lo + per);
  g.own_head = p == 0;
  g.own_tail = p == P - 1;
}

// Calls f(raw value, index, chunk) for every element this thread holds (head elements with chunk
// -1, tail elements with chunk nchunk), and fc(chunk) after each chunk, with every thread of the
// block taking part (fc may use warp collectives). SR_U chunks are loaded at a time.
// Exclusive prefix (thread order) of per-thread doubles and their total: staged in shared memory and
// scanned by warp 0 alone (16 values per lane), so the narrow FP64 pipe sees a few hundred adds.
__device__ __noinline__ double sr_prefix(double v, double* total, double* s_run) {
  const int tid = threadIdx.x, lane = tid & 31;
  s_run[tid] = v;
  __syncthreads();
  if (tid < 32) {
    constexpr int PER = SR_THREADS / 32;
    double loc = 0.0;
#pragma unroll
    for (int q = 0; q < PER; ++q) loc += s_run[lane * PER + q];
    double incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double nb = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += nb;
    }
    double run = incl - loc;
#pragma unroll
    for (int q = 0; q < PER; ++q) {
      const double x = s_run[lane * PER + q];
      s_run[lane * PER + q] = run;
      run += x;
    }
    if (lane == 31) s_run[SR_THREADS] = incl;
  }
  __syncthreads();
  *total = s_run[SR_THREADS];
  const double r = s_run[tid];
  __syncthreads();                                        // s_run is reused by the next call
  return r;
}

template <typename T, typename F, typename FC>
DS_DEV void sr_pass(const SrRow<T>& g, F&& f, FC&& fc) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x;
  if (g.own_head && tid < g.head) f(ds_load_elem<T>(g.row + tid), int64_t(tid), -1);
  const uint4* vp = reinterpret_cast<const uint4*>(g.row + g.head);
  for (int c0 = g.c_lo; c0 < g.c_hi; c0 += SR_U) {
    uint4 buf[SR_U];
#pragma unroll
    for (int u = 0; u < SR_U; ++u) {
      const int64_t v = int64_t(c0 + u) * SR_THREADS + tid;
      if (c0 + u < g.c_hi && v < g.nvec) buf[u] = __ldg(vp + v);
    }
#pragma unroll
    for (int u = 0; u < SR_U; ++u) {
      if (c0 + u >= g.c_hi) break;
      const int64_t v = int64_t(c0 + u) * SR_THREADS + tid;
      if (v < g.nvec) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) f(ds_vec_elem<T>(buf[u], e), g.head + v * EPV + e, c0 + u);
      }
      fc(c0 + u);
    }
  }
  if (g.own_tail && tid < g.ntail) f(ds_load_elem<T>(g.row + g.tail0 + tid), g.tail0 + tid, g.nchunk);
}

// The same over the weights of the row: those of its vectors read from the block's scratch row wr
// (vector v's weights at wr + v * EPV, stored by an earlier pass), those of the few head and tail
// elements computed by wf from the row; calls f(weight, index).
template <typename T, typename WF, typename F>
DS_DEV void sr_wpass(const SrRow<T>& g, const float* wr, WF&& wf, F&& f) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int NF4 = EPV / 4;                 // 16-byte weight loads per vector
  const int tid = threadIdx.x;
  if (g.own_head && tid < g.head) f(wf(ds_load_elem<T>(g.row + tid)), int64_t(tid));
  const float4* wv = reinterpret_cast<const float4*>(wr);
  for (int c0 = g.c_lo; c0 < g.c_hi; c0 += SR_U) {
    float4 buf[SR_U][NF4];
#pragma unroll
    for (int u = 0; u < SR_U; ++u) {
      const int64_t v = int64_t(c0 + u) * SR_THREADS + tid;
      if (c0 + u < g.c_hi && v < g.nvec) {
#pragma unroll
        for (int h = 0; h < NF4; ++h) buf[u][h] = __ldcg(wv + v * NF4 + h);
      }
    }
#pragma unroll
    for (int u = 0; u < SR_U; ++u) {
      const int64_t v = int64_t(c0 + u) * SR_THREADS + tid;
      if (c0 + u < g.c_hi && v < g.nvec) {
        const int64_t i0 = g.head + v * EPV;
#pragma unroll
        for (int h = 0; h < NF4; ++h) {
          f(buf[u][h].x, i0 + 4 * h);
          f(buf[u][h].y, i0 + 4 * h + 1);
          f(buf[u][h].z, i0 + 4 * h + 2);
          f(buf[u][h].w, i0 + 4 * h + 3);
        }
      }
    }
  }
  if (g.own_tail && tid < g.ntail) f(wf(ds_load_elem<T>(g.row + g.tail0 + tid)), g.tail0 + tid);
}

// NUC: rows may need a top-p nucleus; SPQ: a sparse record is written. The common case (neither)
// is compiled separately with a register budget for two blocks per SM.
template <typename T, bool XFORM, bool NUC, bool SPQ>
__global__ void __launch_bounds__(SR_THREADS, (NUC || SPQ || XFORM) ? 1 : 2)
    sample_row_kernel(const rs::SampleArgs a, int64_t rows) {
  constexpr int EPV = 16 / sizeof(T);
  extern __shared__ __align__(16) uint8_t dsm[];
  double* s_cell = reinterpret_cast<double*>(dsm);                        // [SR_CELLS] per-cell values
  float2* s_cellf = reinterpret_cast<float2*>(dsm);                       // ... as float pairs
  // nucleus scratch after the cells: candidate keys [SP_CAP], then per-thread digit masses and
  // counts; per-cell counts of a sparse record after that
  uint64_t* s_keys = reinterpret_cast<uint64_t*>(dsm + sizeof(double) * SR_CELLS);   // [SP_CAP]
  uint8_t* s_nuc = dsm + sizeof(double) * SR_CELLS + sizeof(uint64_t) * SP_CAP;
  uint32_t* s_cnt32 = reinterpret_cast<uint32_t*>(dsm + sizeof(double) * SR_CELLS + (NUC ? SP_NUC_BYTES : 0));
  __shared__ rs::BlockScratch bs;
  __shared__ uint32_t s_cnt;
  __shared__ int s_cellpick;
  __shared__ double s_tau, s_cut[2];
  __shared__ double s_digm[16];
  __shared__ uint32_t s_digc[16];
  __shared__ int s_cutk;
  // exchange slots of the row's parts (a cluster of P blocks), one per part
  __shared__ float s_xf[SR_MAXP];
  __shared__ unsigned long long s_xu[SR_MAXP];
  __shared__ double s_xd[SR_MAXP];
  __shared__ double s_run[SR_THREADS + 1];
  cg::cluster_group cl = cg::this_cluster();
  const int P = int(cl.num_blocks()), part = int(cl.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  bool greedy = !(a.T > 0.0f);
  float Tz = greedy ? 1.0f : a.T, top_p = a.top_p, min_p = a.min_p;
  auto zof = [&](float raw) { return ds_temper(sp_xform<XFORM>(raw, a.mult, a.softcap), Tz); };

  for (int64_t row_id = blockIdx.x / P; row_id < rows; row_id += gridDim.x / P) {
    const int64_t r = row_id / a.B, j = row_id % a.B;
    if (a.n_draft) {                                      // every part of the row skips it
      const int32_t nd = a.n_draft[r];                    // rows past n, and every row of a request
      if (nd < 0 || nd > a.B - 1 || j > nd) continue;     // whose n is out of range, are not needed
    }
    if (a.T_r) {                                          // a mixed batch: this request's values
      const float Tq = a.T_r[r];
      greedy = !(Tq > 0.0f);
      Tz = greedy ? 1.0f : Tq;
    }
    if (a.top_p_r) top_p = a.top_p_r[r];
    if (a.min_p_r) min_p = a.min_p_r[r];
    if (!(Tz == Tz) || !(top_p > 0.0f) || !(min_p >= 0.0f && min_p <= 1.0f)) {   // out of contract:
      if (tid == 0 && part == 0) ds_set_error(a.status, DSPARK_EINVAL);          // greedy, reported
      greedy = true;
      Tz = 1.0f;
      top_p = 1.0f;
      min_p = 0.0f;
    }
    if (a.no_draw && greedy) {                            // verification statistics of a greedy
      greedy = false;                                     // request: its temperature-1 row, no
      Tz = 1.0f;                                          // nucleus (the argmax comes from the
      top_p = 1.0f;                                       // kept-mass pass)
      min_p = 0.0f;
    }
    const int64_t prow = a.row_start ? a.row_start[r] + j : a.row_base + row_id * a.row_mul;
    SrRow<T> g = sr_row<T>(reinterpret_cast<const T*>(a.rows) + prow * a.ld, a.V);
    if (P > 1) sr_part(g, part, P);
    const int64_t qrow = row_id * a.q_row_mul + a.q_row_add;
    float* zr = (a.q_mode == 2 && a.write_z) ? a.q.z + qrow * a.q.ldz : nullptr;
    const int ncells = (g.c_hi - g.c_lo) * SR_WARPS;      // this block's cells

    // ---- pass 1: maximum of z and the argmax key (lowest index on ties); the z row of a dense
    // record is written on the way ----
    float tmax = -INFINITY;
    unsigned long long best = 0;
    // the argmax key per element only when greedy; a sampled row finds its argmax (lowest index
    // with z == zmax) in the kept-mass pass
    const bool want_key = greedy;
    if (!want_key && zr == nullptr) {
      // the common case: the maximum only
      sr_pass(g, [&](float raw, int64_t, int) { tmax = fmaxf(tmax, zof(raw)); }, [](int) {});
    } else {
      sr_pass(g,
              [&](float raw, int64_t i, int) {
                const float z = zof(raw);
                tmax = fmaxf(tmax, z);
                if (want_key) best = max(best, (unsigned long long)ds_key64(ds_canon_zero(z), uint32_t(i)));
                if (zr) zr[i] = z;
              },
              [](int) {});
    }
    if (want_key) best = rs::block_max_u64(best, bs);
    if (P > 1) {
      // the parts' maxima: every block posts into slot `part` of every block, then reads them
      const float bt = rs::block_max(tmax, bs);
      if (tid < P) {
        *cl.map_shared_rank(&s_xf[part], tid) = bt;
        *cl.map_shared_rank(&s_xu[part], tid) = best;
      }
      cl.sync();
      tmax = -INFINITY;
      best = 0;
      for (int q = 0; q < P; ++q) {
        tmax = fmaxf(tmax, s_xf[q]);
        best = max(best, s_xu[q]);
      }
    }

    int64_t pick = -1;
    float zmax, wcut = 0.0f;
    int64_t icut = -1;
    double wkept = 1.0;
    if (greedy) {
      zmax = ds_key64_val(best);
      wcut = 1.0f;
      icut = ds_key64_idx(best);
      if (tid == 0 && part == 0) pick = icut;
    } else {
      zmax = rs::block_max(tmax, bs);
      if (!(zmax > -INFINITY && zmax < INFINITY)) {
        if (tid == 0) {
          ds_set_error(a.status, DSPARK_ENONFINITE);
          if (a.out_idx) a.out_idx[row_id * a.out_mul + a.out_add] = -1;
          a.out_tgt[row_id * a.out_mul + a.out_add] = -1;
          if (a.prev_out) a.prev_out[r] = -1;
        }
        __syncthreads();
        if (P > 1) cl.sync();                              // every part takes this branch
        continue;
      }
      auto wof = [&](float raw) { return ds_weight(__fsub_rn(zof(raw), zmax)); };
      float* wr = nullptr;                               // the block's scratch row of weights
      bool wready = false;                               // ... once written

      // ---- top-p nucleus: the cut (wcut, icut) of the (weight desc, index asc) order. A radix
      // select on the weight bits by mass: each pass sorts the weights that match the digits fixed
      // so far into 16 digit buckets (per-thread float-pair masses and counts in shared memory, so
      // the sums are deterministic), and the digit where the mass from the top crosses top_p * W
      // is fixed. Once that digit holds at most SP_CAP weights they are sorted by (weight desc,
      // index asc) and cut by a block scan. Only more than SP_CAP equal weights at the cut (a
      // flat row) fall back to a bisection over (weight, index) keys ----
      if (NUC && top_p < 1.0f) {
        float2* s_accm = reinterpret_cast<float2*>(s_nuc);                    // [16][SR_THREADS]
        uint32_t* s_accc = reinterpret_cast<uint32_t*>(s_accm + 16 * SR_THREADS);
        uint32_t prefix = 0, pmask = 0, dcount = 0;
        double above = 0.0, target = 0.0;
        int shift = 30;                                // weights <= 1: bit 30 and up are zero
        bool first = true;
        wr = a.wscr ? a.wscr + int64_t(blockIdx.x) * a.wscr_ld : nullptr;
        while (true) {
          const int width = min(4, shift);
          shift -= width;
          const uint32_t dmask = (1u << width) - 1u;
#pragma unroll
          for (int d = 0; d < 16; ++d) {
            s_accm[d * SR_THREADS + tid] = make_float2(0.0f, 0.0f);
            s_accc[d * SR_THREADS + tid] = 0u;
          }
          auto radix = [&](float w) {
            const uint32_t kb = __float_as_uint(w);
            if (w > 0.0f && (kb & pmask) == prefix) {
              const int o = int((kb >> shift) & dmask) * SR_THREADS + tid;
              const float2 m = s_accm[o];
              rs::FF f{m.x, m.y};
              rs::ff_add(f, w);
              s_accm[o] = make_float2(f.hi, f.lo);
              s_accc[o] += 1u;
            }
          };
          if (wready) {
            sr_wpass(g, wr, wof, [&](float w, int64_t) { radix(w); });
          } else {
            // the first pass computes the weights (and keeps those of the vectors in the scratch row)
            sr_pass(g,
                    [&](float raw, int64_t i, int c) {
                      const float w = wof(raw);
                      if (wr && c >= 0 && c < g.nchunk) wr[i - g.head] = w;
                      radix(w);
                    },
                    [](int) {});
          }
          __syncthreads();
          wready = wr != nullptr;
          {                                            // digit `warp`'s mass and count
            rs::FF f{0.0f, 0.0f};
            uint32_t c = 0;
            for (int k = lane; k < SR_THREADS; k += 32) {
              const float2 m = s_accm[warp * SR_THREADS + k];
              const float lo = __fadd_rn(f.lo, m.y);
              f.lo = 0.0f;
              rs::ff_add(f, m.x);
              f.lo = __fadd_rn(f.lo, lo);
              c += s_accc[warp * SR_THREADS + k];
            }
            f = rs::warp_ff_reduce(f);
            c = __reduce_add_sync(0xFFFFFFFFu, c);
            if (lane == 0) {
              s_digm[warp] = rs::ff_value(f);
              s_digc[warp] = c;
            }
          }
          __syncthreads();
          if (first) {                                 // the first pass sees every positive weight
            double W = 0.0;
            for (int d = 0; d < 16; ++d) W += s_digm[d];
            target = double(top_p) * W;
            first = false;
          }
          // the digit where the running mass from the top first exceeds the target (rounding can
          // leave it unreached: then the lowest non-empty digit)
          int dsel = -1;
          double run = above;
          for (int d = int(dmask); d >= 0; --d) {
            if (s_digc[d] == 0u) continue;
            if (run + s_digm[d] > target) {
              dsel = d;
              break;
            }
            run += s_digm[d];
          }
          if (dsel < 0) {
            run = above;
            for (int d = int(dmask); d >= 0; --d) {
              if (s_digc[d] == 0u) continue;
              dsel = d;
              run += s_digm[d];
            }
            run -= s_digm[dsel];
          }
          above = run;
          prefix |= uint32_t(dsel) << shift;
          pmask |= dmask << shift;
          dcount = s_digc[dsel];
          __syncthreads();                             // digit totals are rewritten next pass
          if (dcount <= uint32_t(SP_CAP) || shift == 0) break;
        }
        if (dcount <= uint32_t(SP_CAP)) {
          // the weights of the selected digit, sorted, and the first whose running mass crosses
          if (tid == 0) s_cnt = 0;
          __syncthreads();
          auto collect = [&](float w, int64_t i) {
            if (w > 0.0f && (__float_as_uint(w) & pmask) == prefix) {
              const uint32_t slot = atomicAdd(&s_cnt, 1u);
              if (slot < uint32_t(SP_CAP)) s_keys[slot] = ds_key64(w, uint32_t(i));
            }
          };
          if (wready) sr_wpass(g, wr, wof, collect);
          else sr_pass(g, [&](float raw, int64_t i, int) { collect(wof(raw), i); }, [](int) {});
          __syncthreads();
          const int n = int(min(s_cnt, uint32_t(SP_CAP)));
          int n2 = 1;
          while (n2 < n) n2 <<= 1;
          for (int i = n + tid; i < n2; i += SR_THREADS) s_keys[i] = 0;
          if (tid == 0) s_cutk = n - 1;                // rounding: the last one
          __syncthreads();
          ds_block_sort_desc(s_keys, n2);
          const int k0 = 2 * tid;
          const double w0 = k0 < n ? double(ds_key64_val(s_keys[k0])) : 0.0;
          const double w1 = k0 + 1 < n ? double(ds_key64_val(s_keys[k0 + 1])) : 0.0;
          double tot = 0.0;
          const double before = above + rs::block_exclusive_scan(w0 + w1, &tot, bs);
          if (k0 < n && before + w0 > target) atomicMin(&s_cutk, k0);
          else if (k0 + 1 < n && before + w0 + w1 > target) atomicMin(&s_cutk, k0 + 1);
          __syncthreads();
          if (tid == 0) {
            const uint64_t kc = s_keys[max(s_cutk, 0)];
            s_cut[0] = double(ds_key64_val(kc));
            s_cut[1] = double(ds_key64_idx(kc));
          }
        } else {
          // more than SP_CAP equal weights at the cut: the largest (weight, index) key whose upper
          // set has mass above the target, by bisection over the 64 key bits
          unsigned long long res = 0;
          for (int b = 63; b >= 0; --b) {
            const unsigned long long cand = res | (1ull << b);
            rs::FF mm{0.0f, 0.0f};
            sr_pass(g,
                    [&](float raw, int64_t i, int) {
                      const float w = wof(raw);
                      if ((unsigned long long)ds_key64(w, uint32_t(i)) >= cand) rs::ff_add(mm, w);
                    },
                    [](int) {});
            const double mb = rs::block_sum_ff(mm, bs);
            if (mb > target) res = cand;
          }
          if (tid == 0) {
            s_cut[0] = double(ds_key64_val(res));
            s_cut[1] = double(ds_key64_idx(res));
          }
        }
        __syncthreads();
        wcut = float(s_cut[0]);
        icut = int64_t(s_cut[1]);
      }

      // ---- min-p after top-p: where it cuts inside the nucleus (or there is none) the cut becomes
      // (min_p, the largest int32), which the cut's rule reads as w >= min_p ----
      const bool mp_on = min_p > 0.0f;
      if (mp_on && !(wcut >= min_p)) {
        wcut = min_p;
        icut = 0x7FFFFFFF;
      }
      // ---- pass: kept mass per cell (float pairs per thread, double per warp), head and tail.
      // Without a nucleus or min-p every positive weight is kept ----
      auto keep = [&](float w, int64_t i) { return (NUC || mp_on) ? sp_keep(w, i, wcut, icut) : (w > 0.0f); };
      rs::FF mh{0.0f, 0.0f}, mt{0.0f, 0.0f};
      const bool want_amax = a.amax_out != nullptr;
      uint32_t amin = 0xFFFFFFFFu;                         // lowest index with z == zmax
      if (g.own_head && tid < g.head) {
        const float z = zof(ds_load_elem<T>(g.row + tid)), w = ds_weight(__fsub_rn(z, zmax));
        if (keep(w, tid)) rs::ff_add(mh, w);
        if (z == zmax) amin = min(amin, uint32_t(tid));
      }
      if (g.own_tail && tid < g.ntail) {
        const float z = zof(ds_load_elem<T>(g.row + g.tail0 + tid)), w = ds_weight(__fsub_rn(z, zmax));
        if (keep(w, g.tail0 + tid)) rs::ff_add(mt, w);
        if (z == zmax) amin = min(amin, uint32_t(g.tail0 + tid));
      }
      if (wready && !want_amax) {
        // the weights of the vectors from the scratch row
        constexpr int NF4 = EPV / 4;
        const float4* wv = reinterpret_cast<const float4*>(wr);
        for (int cb = g.c_lo; cb < g.c_hi; cb += SR_U) {
          float4 wb[SR_U][NF4];
#pragma unroll
          for (int u = 0; u < SR_U; ++u) {
            const int64_t v = int64_t(cb + u) * SR_THREADS + tid;
            if (cb + u < g.c_hi && v < g.nvec) {
#pragma unroll
              for (int h = 0; h < NF4; ++h) wb[u][h] = __ldcg(wv + v * NF4 + h);
            }
          }
#pragma unroll
          for (int u = 0; u < SR_U; ++u) {
            if (cb + u >= g.c_hi) break;
            const int64_t v = int64_t(cb + u) * SR_THREADS + tid;
            rs::FF m{0.0f, 0.0f};
            if (v < g.nvec) {
              const int64_t i0 = g.head + v * EPV;
#pragma unroll
              for (int h = 0; h < NF4; ++h) {
                const float w4[4] = {wb[u][h].x, wb[u][h].y, wb[u][h].z, wb[u][h].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (keep(w4[e], i0 + 4 * h + e)) rs::ff_add(m, w4[e]);
              }
            }
            const rs::FF cw = rs::warp_ff_reduce(m);
            if (lane == 0) s_cellf[(cb + u - g.c_lo) * SR_WARPS + warp] = make_float2(cw.hi, cw.lo);
          }
        }
      } else {
        const uint4* vp = reinterpret_cast<const uint4*>(g.row + g.head);
        for (int cb = g.c_lo; cb < g.c_hi; cb += SR_U) {
          uint4 buf[SR_U];
#pragma unroll
          for (int u = 0; u < SR_U; ++u) {
            const int64_t v = int64_t(cb + u) * SR_THREADS + tid;
            if (cb + u < g.c_hi && v < g.nvec) buf[u] = __ldg(vp + v);
          }
#pragma unroll
          for (int u = 0; u < SR_U; ++u) {
            if (cb + u >= g.c_hi) break;
            const int64_t v = int64_t(cb + u) * SR_THREADS + tid;
            rs::FF m{0.0f, 0.0f};
            if (v < g.nvec) {
#pragma unroll
              for (int e = 0; e < EPV; ++e) {
                const float z = zof(ds_vec_elem<T>(buf[u], e)), w = ds_weight(__fsub_rn(z, zmax));
                if (keep(w, g.head + v * EPV + e)) rs::ff_add(m, w);
                if (want_amax && z == zmax) amin = min(amin, uint32_t(g.head + v * EPV + e));
              }
            }
            const rs::FF cw = rs::warp_ff_reduce(m);              // kept as a float pair: the
            if (lane == 0) s_cellf[(cb + u - g.c_lo) * SR_WARPS + warp] = make_float2(cw.hi, cw.lo);
          }
        }
      }
      const double Hm = rs::block_sum_ff(mh, bs);              // (also orders the cell writes)
      const double Tm = rs::block_sum_ff(mt, bs);
      if (want_amax) {
        // the row's argmax: the lowest index of weight 1 over the block, then over the parts
        best = ~rs::block_max_u64(~(unsigned long long)amin, bs);   // minimum via max of the complement
        if (P > 1) {
          if (tid < P) *cl.map_shared_rank(&s_xu[part], tid) = best;
          cl.sync();
          for (int q = 0; q < P; ++q) best = min(best, s_xu[q]);
        }
      }
      // cells: each thread owns a contiguous run of cells; exclusive prefix over threads
      const int per = (ncells + SR_THREADS - 1) / SR_THREADS;
      const int c0 = tid * per, c1 = min(ncells, c0 + per);
      // (FP64 pipe costs a warp instruction per use whatever the active lanes: one conversion
      // per thread here, not one per warp and cell)
      rs::FF mf{0.0f, 0.0f};
      for (int c = c0; c < c1; ++c) {
        const float2 cv = s_cellf[c];
        const float lo = __fadd_rn(mf.lo, cv.y);
        mf.lo = 0.0f;
        rs::ff_add(mf, cv.x);
        mf.lo = __fadd_rn(mf.lo, lo);
      }
      const double mine = rs::ff_value(mf);
      double ctot = 0.0;
      const double before = sr_prefix(mine, &ctot, s_run);
      // this part's mass, the parts before it and the row's total (one exchange when P > 1)
      const double ptot = Hm + ctot + Tm;
      double pbase = 0.0;
      wkept = ptot;
      if (P > 1) {
        if (tid < P) *cl.map_shared_rank(&s_xd[part], tid) = ptot;
        cl.sync();
        wkept = 0.0;
        for (int q = 0; q < P; ++q) {
          if (q < part) pbase += s_xd[q];
          wkept += s_xd[q];
        }
      }

      if (a.probe_w && part == 0) {
        const int64_t x = (a.probe_tgt && j < a.n_draft[r]) ? int64_t(a.probe_tgt[r * (a.B - 1) + j]) : -1;
        if (tid == 0) {
          float pw = 0.0f;
          if (x >= 0 && x < a.V) {
            const float w = wof(ds_load_elem<T>(g.row + x));
            pw = sp_keep(w, x, wcut, icut) ? w : 0.0f;
          }
          a.probe_w[row_id] = pw;
        }
      }

      // ---- draw: the first kept index whose running sum exceeds u * W_kept ----
      if (!a.no_draw) {
        const double u = ds_uniform(a.seed[r], a.step[r], uint32_t(a.position >= 0 ? a.position : int32_t(j)),
                                    DS_PURPOSE_DRAFT);
        const double gtarget = u * wkept;
        // the part whose mass holds the target works in its own frame; past the total (rounding)
        // the last part takes the last kept index
        const bool mine_p = (gtarget >= pbase && gtarget < pbase + ptot) || (part == P - 1 && gtarget >= wkept);
        const double target = gtarget - pbase;
        if (tid == 0) s_cellpick = mine_p ? -3 : -5;          // -5 another part, -3 none, -1 head, -2 tail
        __syncthreads();
        if (!mine_p) {
        } else if (target < Hm) {
          if (tid == 0) s_cellpick = -1;
        } else if (target >= Hm + ctot) {
          if (tid == 0) s_cellpick = (target < ptot) ? -2 : -4;    // -4: rounding left it past the end
        } else {
          const double t_in = target - Hm;
          if (t_in >= before && t_in < before + mine) {
            double acc = before;
            int found = -1;
            for (int c = c0; c < c1; ++c) {
              const double cv = double(s_cellf[c].x) + double(s_cellf[c].y);
              if (found < 0 && t_in < acc + cv && cv > 0.0) {
                found = c;
                s_tau = t_in - acc;
              }
              acc += cv;
            }
            if (found < 0) {                                  // rounding: the last cell with mass
              for (int c = c1 - 1; c >= c0; --c)
                if (double(s_cellf[c].x) + double(s_cellf[c].y) > 0.0) {
                  found = c;
                  s_tau = INFINITY;
                  break;
                }
            }
            s_cellpick = found;
          }
        }
        __syncthreads();
        const int cp = s_cellpick;
        if (cp == -1 || cp == -2) {
          // the few scalar head or tail elements, walked by one thread
          if (tid == 0) {
            double run = (cp == -1) ? 0.0 : Hm + ctot;        // in this part's frame, as `target`
            const int64_t i0 = (cp == -1) ? 0 : g.tail0, i1 = (cp == -1) ? g.head : a.V;
            int64_t lastmine = -1;
            for (int64_t i = i0; i < i1 && pick < 0; ++i) {
              const float w = wof(ds_load_elem<T>(g.row + i));
              if (sp_keep(w, i, wcut, icut)) {
                run += double(w);
                lastmine = i;
                if (run > target) pick = i;
              }
            }
            if (pick < 0) pick = lastmine;
          }
        } else if (cp == -4 || cp == -3) {
          // rounding left the target at the very end: the last kept index of the row (this is the
          // last part), found by a backward scan
          if (tid == 0) {
            for (int64_t i = a.V - 1; i >= 0 && pick < 0; --i)
              if (keep(wof(ds_load_elem<T>(g.row + i)), i)) pick = i;
          }
        } else if (cp >= 0 && warp == cp % SR_WARPS) {
          // the crossing cell: its warp re-reads its 32 vectors and finds the lane, then the element
          const int c = g.c_lo + cp / SR_WARPS;
          const double tau = s_tau;
          const int64_t v = int64_t(c) * SR_THREADS + tid;
          uint4 w4 = make_uint4(0, 0, 0, 0);
          if (v < g.nvec) w4 = __ldg(reinterpret_cast<const uint4*>(g.row + g.head) + v);
          rs::FF lm{0.0f, 0.0f};
          if (v < g.nvec) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              const float w = wof(ds_vec_elem<T>(w4, e));
              if (sp_keep(w, g.head + v * EPV + e, wcut, icut)) rs::ff_add(lm, w);
            }
          }
          const double mv = rs::ff_value(lm);
          double incl = mv;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const double nb = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += nb;
          }
          const double ex = incl - mv;
          const unsigned withm = __ballot_sync(0xFFFFFFFFu, mv > 0.0);
          const int lastl = withm ? 31 - __clz(int(withm)) : -1;
          if (mv > 0.0 && ((tau >= ex && tau < incl) || (lane == lastl && tau >= incl))) {
            double run = ex;
            int64_t lastmine = -1;
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
              const int64_t i = g.head + v * EPV + e;
              const float w = wof(ds_vec_elem<T>(w4, e));
              if (pick < 0 && sp_keep(w, i, wcut, icut)) {
                run += double(w);
                lastmine = i;
                if (run > tau) pick = i;
              }
            }
            if (pick < 0) pick = lastmine;
          }
        }
      }

      // ---- sparse record: kept tokens in ascending index order with q = w / W_kept ----
      if (SPQ && a.q_mode == 1) {
        // counts per cell (reusing the cell array), then positions by the same contiguous scan
        __syncthreads();
        uint32_t kc = 0, kh = 0, kt = 0;
        sr_pass(g,
                [&](float raw, int64_t i, int c) {
                  if (sp_keep(wof(raw), i, wcut, icut)) {
                    if (c < 0) ++kh;
                    else if (c >= g.nchunk) ++kt;
                    else ++kc;
                  }
                },
                [&](int c) {
                  const uint32_t n = __reduce_add_sync(0xFFFFFFFFu, kc);
                  if (lane == 0) s_cnt32[c * SR_WARPS + warp] = n;
                  kc = 0;
                });
        const double nh = double(rs::block_count(kh, bs)), nt = double(rs::block_count(kt, bs));
        double cmine = 0.0;
        for (int c = c0; c < c1; ++c) cmine += double(s_cnt32[c]);
        double cnt_tot = 0.0;
        const double cbefore = sr_prefix(cmine, &cnt_tot, s_run);
        const double ntot = nh + cnt_tot + nt;
        if (ntot > double(a.q.cap)) {
          if (tid == 0) {
            a.q.n[qrow] = -1;
            ds_set_error(a.status, DSPARK_EINVAL);
          }
        } else {
          if (tid == 0) a.q.n[qrow] = int32_t(ntot);
          // cell bases: each thread rewrites its own cells as exclusive prefixes
          double acc = nh + cbefore;
          for (int c = c0; c < c1; ++c) {
            const double n = double(s_cnt32[c]);
            s_cell[c] = acc;                                  // the cell's first output position
            acc += n;
          }
          __syncthreads();
          auto emit = [&](float w, int64_t i, int64_t pos) {
            int64_t tg = i;
            if (a.d2t) tg = i + a.d2t[i];
            const int64_t o = qrow * a.q.cap + pos;
            a.q.ids[o] = int32_t(tg);
            a.q.p[o] = float(double(w) / wkept);
          };
          if (tid == 0) {
            int64_t pos = 0;
            for (int64_t i = 0; i < g.head; ++i) {
              const float w = wof(ds_load_elem<T>(g.row + i));
              if (sp_keep(w, i, wcut, icut)) emit(w, i, pos++);
            }
            pos = int64_t(nh + cnt_tot);
            for (int64_t i = g.tail0; i < a.V; ++i) {
              const float w = wof(ds_load_elem<T>(g.row + i));
              if (sp_keep(w, i, wcut, icut)) emit(w, i, pos++);
            }
          }
          const unsigned below = (1u << lane) - 1u;
          for (int c = 0; c < g.nchunk; ++c) {
            const int64_t v = int64_t(c) * SR_THREADS + tid;
            uint4 w4 = make_uint4(0, 0, 0, 0);
            if (v < g.nvec) w4 = __ldg(reinterpret_cast<const uint4*>(g.row + g.head) + v);
            uint32_t mk = 0;
            if (v < g.nvec) {
#pragma unroll
              for (int e = 0; e < EPV; ++e)
                if (sp_keep(wof(ds_vec_elem<T>(w4, e)), g.head + v * EPV + e, wcut, icut)) mk |= 1u << e;
            }
            const uint32_t nk = uint32_t(__popc(mk));
            uint32_t pre = nk;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, pre, o);
              if (lane >= o) pre += y;
            }
            int64_t pos = int64_t(s_cell[c * SR_WARPS + warp]) + int64_t(pre - nk);
            (void)below;
#pragma unroll
            for (int e = 0; e < EPV; ++e)
              if (mk & (1u << e)) emit(wof(ds_vec_elem<T>(w4, e)), g.head + v * EPV + e, pos++);
          }
        }
      }
    }

    if (a.amax_out && tid == 0 && part == 0)
      a.amax_out[row_id] = greedy ? int32_t(ds_key64_idx(best)) : int32_t(best);

    // ---- outputs (the thread that picked) ----
    if (pick >= 0) {
      int64_t tgt = pick;
      if (a.d2t) {
        tgt = pick + a.d2t[pick];
        if (tgt < 0 || tgt >= a.V_t) {
          ds_set_error(a.status, DSPARK_ERANGE);
          tgt = -1;
        }
      }
      if (a.out_idx) a.out_idx[row_id * a.out_mul + a.out_add] = int32_t(pick);
      a.out_tgt[row_id * a.out_mul + a.out_add] = int32_t(tgt);
      if (a.prev_out) a.prev_out[r] = int32_t(tgt);
      if (a.q_mode == 1 && greedy) {
        a.q.n[qrow] = 1;
        a.q.ids[qrow * a.q.cap] = int32_t(tgt);
        a.q.p[qrow * a.q.cap] = 1.0f;
      }
    }
    if (a.q_mode == 2 && tid == 0 && part == 0) {
      a.q.zmax[qrow] = zmax;
      a.q.wsum[qrow] = greedy ? 1.0 : wkept;
      a.q.wcut[qrow] = wcut;
      a.q.icut[qrow] = int32_t(icut);
    }
    __syncthreads();                                       // the next row reuses the shared arrays
    if (P > 1) cl.sync();                                  // ... and the other parts' slots
  }
}

template <typename T, bool XFORM, bool NUC, bool SPQ>
cudaError_t sp_launch_v(const rs::SampleArgs& a, int64_t rows, cudaStream_t stream) {
  auto kern = sample_row_kernel<T, XFORM, NUC, SPQ>;
  // the nucleus' candidate keys are only needed with NUC
  const size_t smem = sizeof(double) * SR_CELLS + (NUC ? SP_NUC_BYTES : 0) +
                      (SPQ ? sizeof(uint32_t) * SR_CELLS : 0);
  const cudaError_t e = ds_ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const int per_sm = (NUC || SPQ || XFORM) ? 1 : 2;
  const int64_t slots = int64_t(per_sm) * ds_num_sms();
  if (rows <= 0) return cudaSuccess;
  // few rows: split each row over P blocks of a cluster so that every SM streams (common case only)
  int P = 1;
  if (!NUC && !SPQ) {
    const int64_t nchunk = (a.V * int64_t(sizeof(T)) / 16 + SR_THREADS) / SR_THREADS;
    while (P < SR_MAXP && rows * (2 * P) <= slots && nchunk >= int64_t(4 * 2 * P)) P *= 2;
  }
  if (P == 1) {
    const int64_t grid = std::min<int64_t>(rows, slots);
    kern<<<unsigned(grid), SR_THREADS, smem, stream>>>(a, rows);
    return cudaGetLastError();
  }
  const int64_t grid = std::min<int64_t>(rows, slots / P) * P;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(SR_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(P);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, rows);
}

template <typename T, bool XFORM>
cudaError_t sp_launch(const rs::SampleArgs& a, int64_t rows, cudaStream_t stream) {
  const bool nuc = (a.T > 0.0f && a.top_p < 1.0f) || a.T_r != nullptr || a.top_p_r != nullptr;
  const bool spq = a.q_mode == 1;
  if (nuc) return spq ? sp_launch_v<T, XFORM, true, true>(a, rows, stream) : sp_launch_v<T, XFORM, true, false>(a, rows, stream);
  return spq ? sp_launch_v<T, XFORM, false, true>(a, rows, stream) : sp_launch_v<T, XFORM, false, false>(a, rows, stream);
}

}  // namespace

// Shared with the dense walk: one launch of the row sampler over `rows` rows.
cudaError_t rs::sample_rows(const rs::SampleArgs& a, int64_t rows, int is_bf16, int xform, cudaStream_t stream) {
  if (is_bf16) return xform ? sp_launch<__nv_bfloat16, true>(a, rows, stream) : sp_launch<__nv_bfloat16, false>(a, rows, stream);
  return xform ? sp_launch<float, true>(a, rows, stream) : sp_launch<float, false>(a, rows, stream);
}

// The nucleus path's scratch rows: one per resident block (one block per SM), each the row length
// rounded up to 64 floats.
int64_t sp_wscr_ld(int64_t V) { return (V + 63) / 64 * 64; }

extern "C" size_t dspark_internal_ws_sample(int64_t, int32_t, int64_t V) {
  if (V <= 0) return 0;
  return size_t(ds_num_sms()) * size_t(sp_wscr_ld(V)) * sizeof(float);
}

extern "C" dspark_status dspark_sample(const void* logits, dspark_dtype dtype, int64_t R, int32_t B, int64_t V_d,
                                       int64_t ld, const int64_t* row_start, const int64_t* d2t, int64_t V_t,
                                       float mult, float softcap, float temperature, float top_p,
                                       float min_p, const float* temperature_r, const float* top_p_r,
                                       const float* min_p_r,
                                       const uint64_t* seed, const uint64_t* step, int32_t* out_tgt,
                                       int32_t* out_idx, const dspark_qrecord* q, void* ws, size_t ws_bytes,
                                       int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype));
  DS_REQUIRE(R >= 0 && B >= 1 && V_d >= 1 && ld >= V_d && V_d <= 0x7FFFFFFF && R * B <= 0x7FFFFFFF);
  DS_REQUIRE(logits && out_tgt && dev_status && ds_aligned(logits, ds_dtype_size(dtype)));
  DS_REQUIRE(temperature == temperature && top_p == top_p && top_p > 0.0f && min_p >= 0.0f && min_p <= 1.0f);
  DS_REQUIRE(mult == mult && softcap == softcap && softcap >= 0.0f);
  if (temperature > 0.0f || temperature_r) DS_REQUIRE(seed && step);
  if (d2t) DS_REQUIRE(V_t >= 1);
  rs::SampleArgs a = {};
  a.T_r = temperature_r;
  a.top_p_r = top_p_r;
  a.min_p = min_p;
  a.min_p_r = min_p_r;
  a.rows = logits;
  a.V = V_d;
  a.ld = ld;
  a.row_start = row_start;
  a.B = B;
  a.C = rs::cluster_size_for(V_d, ds_dtype_size(dtype));
  DS_REQUIRE(a.C > 0);
  a.mult = mult;
  a.softcap = softcap;
  a.T = temperature;
  a.top_p = top_p;
  a.seed = seed;
  a.step = step;
  a.position = -1;
  a.d2t = d2t;
  a.V_t = V_t;
  a.out_tgt = out_tgt;
  a.out_idx = out_idx;
  a.status = dev_status;
  a.q_row_mul = 1;
  a.row_mul = 1;
  a.out_mul = 1;
  if (q) {
    if (q->z) {
      DS_REQUIRE(q->zmax && q->wsum && q->wcut && q->icut && q->ldz >= V_d);
      a.q = *q;
      a.q_mode = 2;
      a.write_z = 1;
    } else {
      DS_REQUIRE(q->ids && q->p && q->n && q->cap >= 1);
      a.q = *q;
      a.q_mode = 1;
    }
  }
  if (R == 0) return DSPARK_OK;
  // with the workspace, top-p rows keep their weights in it between the nucleus passes
  const size_t wbytes = dspark_internal_ws_sample(R, B, V_d);
  if (ws && ws_bytes >= wbytes && ds_aligned(ws, 16)) {
    a.wscr = static_cast<float*>(ws);
    a.wscr_ld = sp_wscr_ld(V_d);
  }
  const int xform = (mult != 1.0f) || (softcap > 0.0f);
  const cudaError_t e = rs::sample_rows(a, R * B, dtype == DSPARK_BF16, xform, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}
