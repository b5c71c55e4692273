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
// One CTA per request; the lattice is read once (coalesced over candidates b).
#include "dspark_common.cuh"
#include "host_common.h"

namespace {

constexpr int CH_THREADS = 256;
constexpr int CH_MAXK = 64;
constexpr int CH_MAXB = 128;

struct ChainArgs {
  const float* u;
  const float* trans;
  const int32_t* cand_tgt;
  int32_t B, K, mode;
  float T, top_p;
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
};

__global__ void __launch_bounds__(CH_THREADS) chain_maxsum_kernel(const ChainArgs a) {
  __shared__ float s_delta[CH_MAXK];
  __shared__ float s_bv[4][CH_MAXK];
  __shared__ int s_ba[4][CH_MAXK];
  __shared__ uint8_t s_back[CH_MAXB][CH_MAXK];
  const int r = blockIdx.x, K = a.K, B = a.B, t = threadIdx.x;
  const float* u = a.u + int64_t(r) * B * K;
  const float* A = a.trans + int64_t(r) * B * K * K;
  if (t < K) s_delta[t] = __fadd_rn(u[t], A[t]);        // delta_0 = u_0 + A_0[0, :]
  __syncthreads();
  const int b = t & 63, part = t >> 6;
  for (int j = 1; j < B; ++j) {
    const float* Aj = A + int64_t(j) * K * K;
    if (b < K) {
      float best = -INFINITY;
      int ba = -1;
      const int a0 = part * 16, a1 = min(K, a0 + 16);
      for (int aa = a0; aa < a1; ++aa) {
        const float v = __fadd_rn(s_delta[aa], Aj[aa * K + b]);
        if (v > best || ba < 0) {
          best = v;
          ba = aa;
        }
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
      nd = __fadd_rn(u[j * K + t], best);
      s_back[j][t] = uint8_t(ba < 0 ? 0 : ba);
    }
    __syncthreads();
    if (t < K) s_delta[t] = nd;
    __syncthreads();
  }
  if (t == 0) {
    int bb = 0;
    float best = s_delta[0];
    for (int k = 1; k < K; ++k)
      if (s_delta[k] > best) {
        best = s_delta[k];
        bb = k;
      }
    a.score[r] = best;
    for (int j = B - 1; j >= 0; --j) {
      a.chain_rank[r * B + j] = bb;
      a.chain_tgt[r * B + j] = a.cand_tgt[(int64_t(r) * B + j) * K + bb];
      if (j > 0) bb = s_back[j][bb];
    }
  }
}

// Greedy and sampled walks: warp 0 of the CTA walks the lattice position by position.
__global__ void __launch_bounds__(32) chain_walk_kernel(const ChainArgs a) {
  __shared__ float s_w[CH_MAXK];
  __shared__ int s_order[CH_MAXK];
  __shared__ uint8_t s_kept[CH_MAXK];
  const int r = blockIdx.x, K = a.K, B = a.B, lane = threadIdx.x;
  const float* u = a.u + int64_t(r) * B * K;
  const float* A = a.trans + int64_t(r) * B * K * K;
  const bool sample = (a.mode == DSPARK_SAMPLE) && (a.T > 0.0f);
  const uint64_t seed = sample ? a.seed[r] : 0, step = sample ? a.step[r] : 0;
  int prevb = 0;
  double score = 0.0;
  for (int j = 0; j < B; ++j) {
    const float* row = (j == 0) ? A : A + (int64_t(j) * K + prevb) * K;
    float v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int b = lane + 32 * h;
      v[h] = (b < K) ? __fadd_rn(u[j * K + b], row[b]) : -INFINITY;
    }
    int pick;
    const int64_t qrow = int64_t(r) * B + j;
    if (!sample) {
      uint64_t k0 = (lane < K) ? ds_key64(ds_canon_zero(v[0]), lane) : 0;
      uint64_t k1 = (lane + 32 < K) ? ds_key64(ds_canon_zero(v[1]), lane + 32) : 0;
      pick = int(ds_key64_idx(ds_warp_max_u64(k0 > k1 ? k0 : k1)));
      if (a.mode == DSPARK_SAMPLE && lane == 0 && a.q_n) {
        a.q_n[qrow] = 1;
        a.q_ids[qrow * a.q_cap] = a.cand_tgt[qrow * K + pick];
        a.q_p[qrow * a.q_cap] = 1.0f;
      }
    } else {
      float z[2], zmax = -INFINITY;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        z[h] = (lane + 32 * h < K) ? ds_temper(v[h], a.T) : -INFINITY;
        zmax = fmaxf(zmax, z[h]);
      }
      zmax = ds_warp_max(zmax);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = lane + 32 * h;
        if (b < K) {
          s_w[b] = ds_weight(__fsub_rn(z[h], zmax));
          s_kept[b] = 0;
        }
      }
      __syncwarp();
      if (a.top_p < 1.0f) {
        // rank of every candidate in (weight desc, rank asc) order
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int b = lane + 32 * h;
          if (b < K) {
            const float wb = s_w[b];
            int rk = 0;
            for (int c = 0; c < K; ++c) {
              const float wc = s_w[c];
              rk += (wc > wb || (wc == wb && c < b)) ? 1 : 0;
            }
            s_order[rk] = b;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        double wall = 0.0;
        for (int b = 0; b < K; ++b) wall += double(s_w[b]);
        if (a.top_p < 1.0f) {
          double cum = 0.0;
          const double tp = double(a.top_p);
          bool over = false;
          for (int k = 0; k < K; ++k) {
            const int b = s_order[k];
            if (!(s_w[b] > 0.0f)) break;
            cum += double(s_w[b]) / wall;
            s_kept[b] = 1;
            if (cum > tp) {
              over = true;
              break;
            }
          }
          if (!over)
            for (int b = 0; b < K; ++b) s_kept[b] = s_w[b] > 0.0f;
        } else {
          for (int b = 0; b < K; ++b) s_kept[b] = s_w[b] > 0.0f;
        }
        double wk = 0.0;
        int last = -1, nk = 0;
        for (int b = 0; b < K; ++b)
          if (s_kept[b]) {
            wk += double(s_w[b]);
            last = b;
          }
        const double target = ds_uniform(seed, step, uint32_t(j), DS_PURPOSE_DRAFT) * wk;
        double c = 0.0;
        int chosen = last;
        for (int b = 0; b < K; ++b)
          if (s_kept[b]) {
            c += double(s_w[b]);
            if (c > target) {
              chosen = b;
              break;
            }
          }
        if (a.q_n) {
          for (int b = 0; b < K; ++b)
            if (s_kept[b]) {
              if (nk < a.q_cap) {
                a.q_ids[qrow * a.q_cap + nk] = a.cand_tgt[qrow * K + b];
                a.q_p[qrow * a.q_cap + nk] = float(double(s_w[b]) / wk);
              }
              ++nk;
            }
          a.q_n[qrow] = nk;
        }
        s_order[0] = chosen < 0 ? 0 : chosen;
      }
      __syncwarp();
      pick = s_order[0];
      __syncwarp();
    }
    const float vp = __shfl_sync(0xFFFFFFFFu, pick < 32 ? v[0] : v[1], pick & 31);
    score += double(vp);
    if (lane == 0) {
      a.chain_rank[r * B + j] = pick;
      a.chain_tgt[r * B + j] = a.cand_tgt[(int64_t(r) * B + j) * K + pick];
    }
    prevb = pick;
  }
  if (lane == 0) a.score[r] = float(score);
}

}  // namespace

extern "C" dspark_status dspark_chain_select(const float* cand_val, const float* trans,
                                             const int32_t* cand_tgt, int64_t R, int32_t B, int32_t K,
                                             dspark_chain_mode mode, float temperature, float top_p,
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
  a.seed = seed;
  a.step = step;
  a.chain_rank = chain_rank;
  a.chain_tgt = chain_tgt;
  a.score = score;
  a.status = dev_status;
  if (mode == DSPARK_SAMPLE) {
    DS_REQUIRE(temperature == temperature && top_p > 0.0f && top_p == top_p);
    if (temperature > 0.0f) DS_REQUIRE(seed && step);
    if (q) {
      DS_REQUIRE(q->ids && q->p && q->n && q->cap >= K);
      a.q_ids = q->ids;
      a.q_p = q->p;
      a.q_n = q->n;
      a.q_cap = q->cap;
    }
  }
  if (R == 0) return DSPARK_OK;
  if (mode == DSPARK_MAXSUM)
    chain_maxsum_kernel<<<unsigned(R), CH_THREADS, 0, stream>>>(a);
  else
    chain_walk_kernel<<<unsigned(R), 32, 0, stream>>>(a);
  return ds_launch_status();
}
