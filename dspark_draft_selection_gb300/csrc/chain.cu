// chain.cu - chain selection over the K'xK' lattice (dspark_chain_select).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"), block-sampler commit: a greedy request walks the lattice taking
// the best candidate after the token before; a sampled request walks it with its draft RNG; the
// sampled candidates carry their proposal q (Change > Sampled drafting). The max-sum chain is
// the Viterbi recurrence over the same lattice. Sampling follows the thresholded top-p commit
// (nucleus = shortest prefix of (probability desc, index asc) whose mass exceeds top_p), the
// double-sum commit and the double-uniform commit; the candidate rank is the row index.
//
// One CTA of 256 threads per request. The unary scores and candidate ids, then the K'xK' tiles
// of up to 16 positions at once, are requested together with 16-byte cp.async copies (the next
// batch as soon as one is consumed), so the lattice is read once and its latency is paid once per
// batch rather than once per position; odd K' or unaligned lattices take double-buffered tiles.
// Max-sum uses all threads (4 threads per column b, 16 predecessors each); the walks use warp 0
// with the row after the previous choice, except that every thread helps with the sampled walk's
// top-p nucleus (4 threads per candidate sum the weights of the keys above its key), and the
// draws' uniforms are made ahead of the walk.
#include "dspark_common.cuh"
#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int CH_THREADS = 256;
constexpr int CH_MAXK = 64;
constexpr int CH_MAXB = 128;
constexpr int CH_MAXNS = 16;          // tiles requested together (batch path)
constexpr int CH_MAXH = 1024;         // history ids staged in shared memory (the rest read from L2)

struct ChainArgs {
  const float* u;
  const float* trans;
  const int32_t* cand_tgt;
  int32_t B, K, mode;
  float T, top_p, min_p;
  const float* T_r;                   // [R] per-request temperature (<= 0: greedy), or null
  const float* top_p_r;               // [R] per-request top-p, or null
  const float* min_p_r;               // [R] per-request min-p, or null
  const int32_t* hist_ids;            // [R, hist_cap] penalty history (target ids), or null
  const int32_t* hist_n;              // [R]
  int32_t hist_cap;
  float rep, pres;                    // repetition (1: off) and presence (0: off) penalties
  const uint64_t* seed;
  const uint64_t* step;
  int32_t* chain_rank;
  int32_t* chain_tgt;
  float* score;
  int32_t* q_ids;
  float* q_p;
  int32_t* q_n;
  int32_t q_cap;
  int32_t* status;
  int32_t ns;                         // tiles per batch (batch path)
};

// cp.async one position's K x K tile (K*K floats; K*K*4 is a multiple of 16 when K % 2 == 0,
// otherwise the tail goes element-wise)
DS_DEV void ch_load_tile(float* dst, const float* src, int n) {
  const int nvec = ((reinterpret_cast<uintptr_t>(src) & 15) == 0) ? n / 4 : 0;
  for (int i = threadIdx.x; i < nvec; i += CH_THREADS) ds_cp_async16(dst + 4 * i, src + 4 * i);
  for (int i = 4 * nvec + threadIdx.x; i < n; i += CH_THREADS) dst[i] = src[i];
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// cp.async of one tile (K*K floats, 16-byte aligned, K*K % 4 == 0) without committing the group
DS_DEV void ch_issue_tile(float* dst, const float* src, int n) {
  for (int i = threadIdx.x; i < n / 4; i += CH_THREADS) ds_cp_async16(dst + 4 * i, src + 4 * i);
}

DS_DEV void ch_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
DS_DEV void ch_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// warp inclusive scan of float pairs (the running sums of the sampled walk: a double instruction
// costs about 64 single-precision ones on this part)
DS_DEV rs::FF ch_warp_scan(rs::FF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const rs::FF n{__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
    if (lane >= o) rs::ff_acc(v, n);
  }
  return v;
}
DS_DEV rs::FF ch_shfl(const rs::FF& v, int src) {
  return rs::FF{__shfl_sync(0xFFFFFFFFu, v.hi, src), __shfl_sync(0xFFFFFFFFu, v.lo, src)};
}

template <bool RING>
__global__ void __launch_bounds__(CH_THREADS) chain_kernel(const ChainArgs a) {
  // RING: batches of NS [K*K] tiles, each batch requested at once, else [2][K*K] double-buffered;
  // then [B*K] unary scores
  extern __shared__ __align__(128) float ch_dyn[];
  __shared__ float s_delta[CH_MAXK];
  __shared__ float s_bv[4][CH_MAXK];
  __shared__ int s_ba[4][CH_MAXK];
  __shared__ uint8_t s_back[CH_MAXB][CH_MAXK];

  const int r = blockIdx.x, K = a.K, B = a.B, t = threadIdx.x;
  const int KK = K * K;
  ds_pdl_trigger();
  ds_pdl_wait();                                   // the lattice and candidates come from before
  const int KKp = (KK + 3) & ~3;
  const int NS = RING ? a.ns : 2;
  float* s_tile0 = ch_dyn;
  float* s_tile1 = ch_dyn + KKp;
  float* s_u = ch_dyn + size_t(NS) * KKp;
  const float* u = a.u + int64_t(r) * B * K;
  const float* A = a.trans + int64_t(r) * B * KK;
  // the request's candidate ids (for the outputs) and unary scores come in with the first
  // tiles, asynchronously, so no thread stalls on a load
  int32_t* s_ct = reinterpret_cast<int32_t*>(s_u + ((B * K + 3) & ~3));
  const int32_t* ctg = a.cand_tgt + int64_t(r) * B * K;
  const bool uvec = ((B * K) & 3) == 0 && (reinterpret_cast<uintptr_t>(u) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(ctg) & 15) == 0;
  if (uvec) {
    for (int i = t; i < (B * K) / 4; i += CH_THREADS) {
      ds_cp_async16(s_u + 4 * i, u + 4 * i);
      ds_cp_async16(s_ct + 4 * i, ctg + 4 * i);
    }
  } else {
    for (int i = t; i < B * K; i += CH_THREADS) {
      s_u[i] = u[i];
      s_ct[i] = ctg[i];
    }
  }
  if (RING) {
    // the first batch of tiles is requested at once by every thread: the lattice's latency is paid
    // once per batch of NS positions instead of once per position
    for (int i = 0; i < NS && i < B; ++i) ch_issue_tile(ch_dyn + size_t(i) * KKp, A + int64_t(i) * KK, KK);
    asm volatile("cp.async.commit_group;" ::: "memory");
  } else {
    ch_load_tile(s_tile0, A, KK);                  // commits the ids and scores with tile 0
  }

  const bool maxsum = a.mode == DSPARK_MAXSUM;
  // this request's sampling parameters: a mixed batch gives them per request
  float Tq = a.T_r ? a.T_r[r] : a.T, tpq = a.top_p_r ? a.top_p_r[r] : a.top_p;
  float mpq = a.min_p_r ? a.min_p_r[r] : a.min_p;
  if (a.mode == DSPARK_SAMPLE && !(Tq == Tq && tpq > 0.0f && mpq >= 0.0f && mpq <= 1.0f)) {   // out of
    if (t == 0) ds_set_error(a.status, DSPARK_EINVAL);                                        // contract:
    Tq = 0.0f;                                                                                // greedy,
    tpq = 1.0f;                                                                               // reported
    mpq = 0.0f;
  }
  const bool sample = (a.mode == DSPARK_SAMPLE) && (Tq > 0.0f);
  const uint64_t seed = sample ? a.seed[r] : 0, step = sample ? a.step[r] : 0;
  const int warp = t >> 5, lane = t & 31;
  int prevb = 0;
  // penalties: which candidates' target ids are in the request's history (a bit per (position,
  // rank)); tokens drafted at earlier positions are added as the walk goes
  __shared__ uint32_t s_hitw[CH_MAXB * CH_MAXK / 32];
  __shared__ int32_t s_hist[CH_MAXH];
  __shared__ int32_t s_drafted[CH_MAXB];
  const bool pen = a.hist_ids != nullptr;
  if (pen) {
    const int hn = max(0, min(a.hist_n[r], a.hist_cap));
    const int32_t* hg = a.hist_ids + int64_t(r) * a.hist_cap;
    for (int i = t; i < min(hn, CH_MAXH); i += CH_THREADS) s_hist[i] = hg[i];
    for (int i = t; i < (B * K + 31) / 32; i += CH_THREADS) s_hitw[i] = 0u;
    ch_wait_all();                               // the candidate ids (and the first tiles) are in
    __syncthreads();
    for (int i = t; i < B * K; i += CH_THREADS) {
      const int32_t c = s_ct[i];
      bool hit = false;
      for (int k = 0; k < hn && !hit; ++k) hit = (k < CH_MAXH ? s_hist[k] : hg[k]) == c;
      if (hit) atomicOr(&s_hitw[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
  }
  double score = 0.0;
  // the draws' uniforms, which the walk's path does not change, ahead of the walk (visible after
  // the first position's barrier)
  __shared__ float2 s_ud[CH_MAXB];
  if (sample)
    for (int j = t; j < B; j += CH_THREADS) {
      const rs::FF uj = rs::ff_uniform(seed, step, uint32_t(j), DS_PURPOSE_DRAFT);
      s_ud[j] = make_float2(uj.hi, uj.lo);
    }
  // the nucleus of a sampled position: the keys and weights of its candidates, the mass bound
  // top_p * W and the membership that every thread helps to find
  __shared__ uint64_t s_nk[CH_MAXK];
  __shared__ float s_nw[CH_MAXK];
  __shared__ float s_tp[2];
  __shared__ uint8_t s_keep[CH_MAXK];

  for (int j = 0; j < B; ++j) {
    const float* Aj;
    if (RING) {
      if (j % NS == 0) {
        ch_wait_all();
        __syncthreads();
      }
      Aj = ch_dyn + size_t(j % NS) * KKp;
    } else {
      if (j + 1 < B) {
        ch_load_tile(((j + 1) & 1) ? s_tile1 : s_tile0, A + int64_t(j + 1) * KK, KK);
        ch_wait_prev();
      } else {
        ch_wait_all();
      }
      __syncthreads();
      Aj = (j & 1) ? s_tile1 : s_tile0;
    }
    const float* uj = s_u + j * K;
    if (maxsum) {
      if (j == 0) {
        if (t < K) s_delta[t] = __fadd_rn(uj[t], Aj[t]);          // delta_0 = u_0 + A_0[0, :]
      } else {
        const int b = t & 63, part = t >> 6;
        if (b < K) {
          // the 16 predecessors of this part: loads first (independent), then the running max
          // (first maximum kept: lowest predecessor index among equal sums)
          const int a0 = part * 16, na = min(K - a0, 16);
          float v[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = (q < na) ? __fadd_rn(s_delta[a0 + q], Aj[(a0 + q) * K + b]) : -INFINITY;
          float best = v[0];
          int ba = (na > 0) ? a0 : -1;
#pragma unroll
          for (int q = 1; q < 16; ++q)
            if (q < na && v[q] > best) {
              best = v[q];
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
          for (int p = 1; p < 4; ++p) {
            if (s_ba[p][t] >= 0 && (ba < 0 || s_bv[p][t] > best)) {
              best = s_bv[p][t];
              ba = s_ba[p][t];
            }
          }
          nd = __fadd_rn(uj[t], best);
          s_back[j][t] = uint8_t(ba < 0 ? 0 : ba);
        }
        __syncthreads();
        if (t < K) s_delta[t] = nd;
      }
    } else {
      // ---- warp 0: the row's values (penalties applied) and, when sampling, the weights and
      // their total ----
      const bool nuc = sample && tpq < 1.0f;
      float v[2] = {-INFINITY, -INFINITY}, w[2] = {0.0f, 0.0f};
      rs::FF wall{0.0f, 0.0f};
      if (warp == 0) {
      const float* row = (j == 0) ? Aj : Aj + prevb * K;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = lane + 32 * h;
        v[h] = (b < K) ? __fadd_rn(uj[b], row[b]) : -INFINITY;
        if (pen && b < K) {
          // repetition, then presence, on candidates in the history or drafted before
          const int i = j * K + b;
          const int32_t c = s_ct[i];
          bool hit = (s_hitw[i >> 5] >> (i & 31)) & 1u;
          for (int k = 0; k < j && !hit; ++k) hit = s_drafted[k] == c;
          if (hit) {
            if (a.rep != 1.0f) v[h] = v[h] > 0.0f ? __fdiv_rn(v[h], a.rep) : __fmul_rn(v[h], a.rep);
            if (a.pres != 0.0f) v[h] = __fsub_rn(v[h], a.pres);
          }
        }
      }
      if (sample) {
        float zmax = -INFINITY, z[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          z[h] = (lane + 32 * h < K) ? ds_temper(v[h], Tq) : -INFINITY;
          zmax = fmaxf(zmax, z[h]);
        }
        zmax = ds_warp_max(zmax);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int b = lane + 32 * h;
          w[h] = (b < K) ? ds_weight(__fsub_rn(z[h], zmax)) : 0.0f;
        }
        __syncwarp();
        rs::FF wsum2{w[0], 0.0f};
        rs::ff_add(wsum2, w[1]);
        wall = rs::warp_ff_reduce(wsum2);
        if (nuc) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int b = lane + 32 * h;
            s_nk[b] = (b < K) ? ds_key64(w[h], uint32_t(b)) : 0ull;
            s_nw[b] = w[h];
          }
          if (lane == 0) {
            const rs::FF tp = rs::ff_mul(rs::FF{tpq, 0.0f}, wall);
            s_tp[0] = tp.hi;
            s_tp[1] = tp.lo;
          }
        }
      }
      }
      // ---- every thread: top-p nucleus membership. Candidate i is kept when the mass of the
      // candidates before it in the (weight desc, rank asc) order - the keys above its key - is at
      // most top_p * W; then the first candidate whose running mass exceeds top_p * W is the last
      // kept one. Four threads share a candidate's sum (16 keys each, in float pairs) ----
      if (nuc) {
        __syncthreads();
        const int i = t >> 2, qq = t & 3;
        rs::FF e0{0.0f, 0.0f}, e1{0.0f, 0.0f};
        const uint64_t ki = (i < CH_MAXK) ? s_nk[i] : 0ull;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const int k0 = qq * 16 + k;
          if (s_nk[k0] > ki) rs::ff_add(e0, s_nw[k0]);
          if (s_nk[k0 + 1] > ki) rs::ff_add(e1, s_nw[k0 + 1]);
        }
        rs::ff_acc(e0, e1);
        rs::ff_acc(e0, rs::FF{__shfl_xor_sync(0xFFFFFFFFu, e0.hi, 1), __shfl_xor_sync(0xFFFFFFFFu, e0.lo, 1)});
        rs::ff_acc(e0, rs::FF{__shfl_xor_sync(0xFFFFFFFFu, e0.hi, 2), __shfl_xor_sync(0xFFFFFFFFu, e0.lo, 2)});
        if (qq == 0 && i < CH_MAXK)
          s_keep[i] = (ki != 0ull && s_nw[i] > 0.0f && !(rs::ff_diff(e0, rs::FF{s_tp[0], s_tp[1]}) > 0.0f)) ? 1 : 0;
        __syncthreads();
      }
      if (warp == 0) {
      int pick;
      const int64_t qrow = int64_t(r) * B + j;
      if (!sample) {
        const uint64_t k0 = (lane < K) ? ds_key64(ds_canon_zero(v[0]), lane) : 0;
        const uint64_t k1 = (lane + 32 < K) ? ds_key64(ds_canon_zero(v[1]), lane + 32) : 0;
        pick = int(ds_key64_idx(ds_warp_max_u64(k0 > k1 ? k0 : k1)));
        if (a.mode == DSPARK_SAMPLE && lane == 0 && a.q_n) {
          a.q_n[qrow] = 1;
          a.q_ids[qrow * a.q_cap] = s_ct[j * K + pick];
          a.q_p[qrow * a.q_cap] = 1.0f;
        }
      } else {
        // kept[h]: membership of candidate lane + 32h (positive weight, the nucleus)
        bool kept[2] = {w[0] > 0.0f, w[1] > 0.0f};
        if (nuc) {
          kept[0] = kept[0] && s_keep[lane] != 0;
          kept[1] = kept[1] && s_keep[lane + 32] != 0;
        }
        // min-p after top-p: candidates whose weight is at least min_p times the top one's (1)
        if (mpq > 0.0f) {
          kept[0] = kept[0] && w[0] >= mpq;
          kept[1] = kept[1] && w[1] >= mpq;
        }
        // draw: kept candidates in ascending rank order; running sums by warp scan
        // (lane holds ranks lane and lane + 32: scan the first half, then the second)
        const rs::FF inc0 = ch_warp_scan(rs::FF{kept[0] ? w[0] : 0.0f, 0.0f});
        rs::FF inc1 = ch_warp_scan(rs::FF{kept[1] ? w[1] : 0.0f, 0.0f});
        rs::ff_acc(inc1, ch_shfl(inc0, 31));
        const rs::FF wkf = ch_shfl(inc1, 31);
        const rs::FF target = rs::ff_mul(rs::FF{s_ud[j].x, s_ud[j].y}, wkf);
        const unsigned c0 = __ballot_sync(0xFFFFFFFFu, kept[0] && rs::ff_diff(inc0, target) > 0.0f);
        const unsigned c1 = __ballot_sync(0xFFFFFFFFu, kept[1] && rs::ff_diff(inc1, target) > 0.0f);
        // q = w / W_kept rounded to float: q0 = w / W_hi, then the remainder w - q0 W (an FMA and the
        // low term) corrects it to the nearest float of the float-pair quotient
        auto qdiv = [&](float wv) {
          const float q0 = __fdiv_rn(wv, wkf.hi);
          const float rem = __fsub_rn(__fmaf_rn(-q0, wkf.hi, wv), __fmul_rn(q0, wkf.lo));
          return __fadd_rn(q0, __fdiv_rn(rem, wkf.hi));
        };
        if (c0) pick = __ffs(c0) - 1;
        else if (c1) pick = 32 + __ffs(c1) - 1;
        else {
          const unsigned l0 = __ballot_sync(0xFFFFFFFFu, kept[0]), l1 = __ballot_sync(0xFFFFFFFFu, kept[1]);
          pick = l1 ? 32 + (31 - __clz(int(l1))) : (l0 ? 31 - __clz(int(l0)) : 0);
        }
        if (a.q_n) {
          // kept candidates in ascending rank order with q = w / W_kept
          const unsigned m0 = __ballot_sync(0xFFFFFFFFu, kept[0]), m1 = __ballot_sync(0xFFFFFFFFu, kept[1]);
          const unsigned below = (1u << lane) - 1u;
          const int n0 = __popc(m0);
          if (kept[0]) {
            const int o = __popc(m0 & below);
            if (o < a.q_cap) {
              a.q_ids[qrow * a.q_cap + o] = s_ct[j * K + lane];
              a.q_p[qrow * a.q_cap + o] = qdiv(w[0]);
            }
          }
          if (kept[1]) {
            const int o = n0 + __popc(m1 & below);
            if (o < a.q_cap) {
              a.q_ids[qrow * a.q_cap + o] = s_ct[j * K + lane + 32];
              a.q_p[qrow * a.q_cap + o] = qdiv(w[1]);
            }
          }
          if (lane == 0) a.q_n[qrow] = n0 + __popc(m1);
        }
      }
      const float vp = __shfl_sync(0xFFFFFFFFu, pick < 32 ? v[0] : v[1], pick & 31);
      score += double(vp);
      if (lane == 0) {
        a.chain_rank[r * B + j] = pick;
        a.chain_tgt[r * B + j] = s_ct[j * K + pick];
        s_drafted[j] = s_ct[j * K + pick];
      }
      __syncwarp();
      prevb = pick;
      }
    }
    __syncthreads();
    if (RING && j % NS == NS - 1 && j + 1 < B) {
      // the batch is consumed: request the next one
      for (int i = j + 1; i < j + 1 + NS && i < B; ++i)
        ch_issue_tile(ch_dyn + size_t(i % NS) * KKp, A + int64_t(i) * KK, KK);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  }
  if (maxsum) {
    // best final score (first maximum) by warp 0, then the backtrack by thread 0 into shared
    // memory, then every position's outputs in parallel
    __shared__ int s_path[CH_MAXB];
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
        a.score[r] = s_delta[bb];
        for (int j = B - 1; j >= 0; --j) {
          s_path[j] = bb;
          if (j > 0) bb = s_back[j][bb];
        }
      }
    }
    __syncthreads();
    for (int j = t; j < B; j += CH_THREADS) {
      const int bb = s_path[j];
      a.chain_rank[r * B + j] = bb;
      a.chain_tgt[r * B + j] = s_ct[j * K + bb];
    }
  }
  if (!maxsum && t == 0) a.score[r] = float(score);
}

}  // namespace

extern "C" dspark_status dspark_chain_select(const float* cand_val, const float* trans,
                                             const int32_t* cand_tgt, int64_t R, int32_t B, int32_t K,
                                             dspark_chain_mode mode, float temperature, float top_p,
                                             float min_p, const float* temperature_r, const float* top_p_r,
                                             const float* min_p_r, const dspark_penalties* penalties,
                                             const uint64_t* seed, const uint64_t* step,
                                             int32_t* chain_rank, int32_t* chain_tgt, float* score,
                                             const dspark_qrecord* q, int32_t* dev_status,
                                             dspark_stream_t stream) {
  DS_REQUIRE(R >= 0 && B >= 1 && B <= CH_MAXB && K >= 1 && K <= CH_MAXK);
  DS_REQUIRE(R <= 0x7FFFFFFF);
  DS_REQUIRE(cand_val && trans && cand_tgt && chain_rank && chain_tgt && score && dev_status);
  DS_REQUIRE(mode == DSPARK_MAXSUM || mode == DSPARK_WALK || mode == DSPARK_SAMPLE);
  ChainArgs a = {};
  a.u = cand_val;
  a.trans = trans;
  a.cand_tgt = cand_tgt;
  a.B = B;
  a.K = K;
  a.mode = int(mode);
  a.T = temperature;
  a.top_p = top_p;
  a.min_p = min_p;
  a.T_r = mode == DSPARK_SAMPLE ? temperature_r : nullptr;
  a.top_p_r = mode == DSPARK_SAMPLE ? top_p_r : nullptr;
  a.min_p_r = mode == DSPARK_SAMPLE ? min_p_r : nullptr;
  if (penalties) {
    // penalties change a walk's rows by the tokens drafted before: walks only, not max-sum
    DS_REQUIRE(mode != DSPARK_MAXSUM && penalties->ids && penalties->n && penalties->cap >= 0);
    DS_REQUIRE(penalties->repetition > 0.0f && penalties->repetition < INFINITY && penalties->presence == penalties->presence);
    a.hist_ids = penalties->ids;
    a.hist_n = penalties->n;
    a.hist_cap = penalties->cap;
    a.rep = penalties->repetition;
    a.pres = penalties->presence;
  }
  a.seed = seed;
  a.step = step;
  a.chain_rank = chain_rank;
  a.chain_tgt = chain_tgt;
  a.score = score;
  a.status = dev_status;
  if (mode == DSPARK_SAMPLE) {
    DS_REQUIRE(temperature == temperature && top_p > 0.0f && top_p == top_p && min_p >= 0.0f && min_p <= 1.0f);
    if (temperature > 0.0f || temperature_r) DS_REQUIRE(seed && step);
    if (q) {
      DS_REQUIRE(q->ids && q->p && q->n && q->cap >= K);
      a.q_ids = q->ids;
      a.q_p = q->p;
      a.q_n = q->n;
      a.q_cap = q->cap;
    }
  }
  if (R == 0) return DSPARK_OK;
  const size_t tile = size_t((K * K + 3) & ~3) * sizeof(float);
  const size_t ubytes = 2 * size_t((B * K + 3) & ~3) * sizeof(float);   // scores + candidate ids
  // the batch path copies 16-byte pieces: tiles 16-byte aligned, K*K a multiple of 4 (K even)
  const bool ring = (K % 2 == 0) && ds_aligned(trans, 16);
  constexpr size_t kBudget = 192 * 1024;                   // dynamic shared memory for tiles + scores
  int ns = 2;
  if (ring) {
    ns = int(std::min<size_t>({size_t(B), size_t(CH_MAXNS), (kBudget - std::min(kBudget, ubytes)) / tile}));
    if (ns < 1) ns = 1;
  }
  a.ns = ns;
  const size_t smem = size_t(ns) * tile + ubytes;
  if (smem > kBudget + 16 * 1024) return DSPARK_EINVAL;
  if (ring) {
    if (smem > 48 * 1024)
      DS_CUDA_TRY(ds_ensure_smem(reinterpret_cast<const void*>(chain_kernel<true>), smem));
    DS_CUDA_TRY(ds_launch(chain_kernel<true>, dim3(unsigned(R)), dim3(CH_THREADS), smem, stream, a));
  } else {
    if (smem > 48 * 1024)
      DS_CUDA_TRY(ds_ensure_smem(reinterpret_cast<const void*>(chain_kernel<false>), smem));
    DS_CUDA_TRY(ds_launch(chain_kernel<false>, dim3(unsigned(R)), dim3(CH_THREADS), smem, stream, a));
  }
  return ds_launch_status();
}
