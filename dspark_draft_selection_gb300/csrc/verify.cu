// verify.cu - rejection-sampling verification of drafted tokens (dspark_verify).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"): commit on exact sampled speculative decoding - each window
// position is checked against the target's post-filter p, accepted with probability min(1, p/q),
// otherwise a sample of norm(max(0, p - q)) is emitted and the later candidates dropped;
// accepted tokens report the target's log-probability; ids beyond a model's row have zero
// probability; q is recorded sparse over the kept tokens or dense, in target ids; sums in double.
// Commit on the double uniform (acceptance test and draws). Description > Fixes > Split
// validation windows: row j validates candidate j; row n is the bonus row. This is the
// speculative sampling rule of Leviathan et al. (2023) and Chen et al. (2023).
//
// Launches:
//  0. pruned dense records only: the inverse map t2d over the target vocabulary (target id ->
//     draft index of the record, -1 outside the draft vocabulary).
//  1. statistics of every needed target row: the maximum, the top-p cut and the kept mass of p_j,
//     the weight of the drafted token x_j, and the argmax (greedy requests) - verify_stats_kernel
//     when there is no nucleus, else the row sampler of sample.cu in statistics mode. The target
//     logits are read from HBM once here. The acceptance tests of a request run once its rows are
//     done (in the statistics kernel, by the CTA that finishes the last of them; after the row
//     sampler, in verify_accept_kernel): one warp, one lane per window position - the tests
//     u_j < p_j(x_j) / q_j(x_j) of different positions are independent, and the first failing
//     position (a ballot) ends the window. They leave at most one draw: the residual at the first
//     rejection, or the bonus draw at n (greedy requests need none).
//  2. verify_draw_kernel - one CTA per part of a request's draw row (as many parts as keep all
//     requests' parts in one wave of resident CTAs; 8,192 ids with a sparse record) forms
//     rho = max(0, p - q) (p alone for the bonus draw) scaled by W_p * W_q, so no element needs a
//     division, as float pairs, and writes the mass of every cell of VM_CELL consecutive ids; the
//     part that finishes last scans all cells in double, finds the cell whose running sum crosses
//     u * sum(rho), re-evaluates that cell's ids and emits the token.
#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int VM_THREADS = 512;            // residual-mass CTAs
constexpr int VM_CELL = 256;               // ids per cell: one warp, eight consecutive ids a lane
constexpr int VM_PART_MIN_CELLS = 16;      // the smallest dense part (4,096 ids)
constexpr int VM_PART_SPARSE = 8192;       // ... for sparse records (staged in shared memory by id)

enum : int32_t { JOB_NONE = 0, JOB_RESIDUAL = 1, JOB_BONUS = 2 };
// proposal record forms
enum : int { QF_NONE = 0, QF_SPARSE = 1, QF_DENSE = 2, QF_DENSE_PRUNED = 3 };

struct VerifyWs {
  float* zmax;       // [R * (B + 1)] target row statistics
  double* wsum;
  float* wcut;
  int32_t* icut;
  float* probe_w;
  int32_t* amax;
  int32_t* job_kind; // [R] the draw job of each request (from the acceptance tests)
  int32_t* job_j;
  int32_t* tk_stats; // [R] rows of a request whose statistics are done
  int32_t* tk_draw;  // [R] parts of a request's draw row that are done
  float2* cells;     // [R, ncell] residual mass per cell (float pair)
  int32_t* t2d;      // [V] record index of each target id (pruned dense records)
};

struct VerifyArgs {
  const void* logits;
  int64_t V, ld;
  const int64_t* row_start;
  int32_t B;
  const int32_t* draft_tgt;
  const int32_t* n_draft;
  dspark_qrecord q;
  int q_form;
  int64_t V_q;
  float T, top_p, min_p;
  const float* T_r;          // [R] per-request temperature (<= 0: greedy), or null
  const float* top_p_r;      // [R] per-request top-p, or null
  const float* min_p_r;      // [R] per-request min-p, or null
  const uint64_t* vseed;
  const uint64_t* step;
  int32_t* out_tokens;
  int32_t* n_accepted;
  float* logprob;
  int32_t* status;
  int64_t ncell;
  int32_t part_cells;  // cells per draw CTA (dense and no record; sparse records use VM_PART_SPARSE)
  VerifyWs ws;
};

// Request r's temperature: a mixed batch gives it per request (a NaN one counts as greedy; the
// host or the statistics pass reports it)
DS_DEV float vf_T(const VerifyArgs& a, int64_t r) {
  const float T = a.T_r ? a.T_r[r] : a.T;
  return T == T ? T : 0.0f;
}

// Request r's min-p (0 when out of [0, 1]; the host or the statistics pass reports it)
DS_DEV float vf_mp(const VerifyArgs& a, int64_t r) {
  const float m = a.min_p_r ? a.min_p_r[r] : a.min_p;
  return (m >= 0.0f && m <= 1.0f) ? m : 0.0f;
}

DS_DEV bool vf_keep(float w, int64_t i, float wcut, int64_t icut) {
  return w > 0.0f && (w > wcut || (w == wcut && i <= icut));
}

// Record index of target id x for a dense record (-1: not in the record)
DS_DEV int64_t vf_qindex(const VerifyArgs& a, int64_t x) {
  if (x < 0) return -1;
  if (a.q_form == QF_DENSE_PRUNED) return x < a.V ? int64_t(a.ws.t2d[x]) : -1;
  return x < a.V_q ? x : -1;
}

// Kept weight of record index i of a dense record row
DS_DEV float vf_wq(const VerifyArgs& a, int64_t qrow, int64_t i) {
  if (i < 0) return 0.0f;
  const float w = ds_weight(__fsub_rn(a.q.z[qrow * a.q.ldz + i], a.q.zmax[qrow]));
  return vf_keep(w, i, a.q.wcut[qrow], a.q.icut[qrow]) ? w : 0.0f;
}

// A double as a float pair (its leading 48 bits)
DS_DEV rs::FF vf_ff(double x) {
  const float hi = float(x);
  return rs::FF{hi, float(x - double(hi))};
}

// q_j(x) = num / den from the record: a sparse record's probability over 1, a dense record's kept
// weight over the row's kept mass; ids outside the record have num = 0
DS_DEV float vf_qnum(const VerifyArgs& a, int64_t qrow, int64_t x) {
  if (x < 0) return 0.0f;
  if (a.q_form == QF_SPARSE) {
    const int n = a.q.n[qrow];
    for (int k = 0; k < n && k < a.q.cap; ++k)
      if (a.q.ids[qrow * a.q.cap + k] == x) return a.q.p[qrow * a.q.cap + k];
    return 0.0f;
  }
  return vf_wq(a, qrow, vf_qindex(a, x));
}

__global__ void verify_t2d_kernel(const int64_t* d2t, int64_t V_d, int64_t V_t, int32_t* t2d, int32_t* status) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < V_d; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t t = i + d2t[i];
    if (t < 0 || t >= V_t) {
      ds_set_error(status, DSPARK_ERANGE);
      continue;
    }
    t2d[t] = int32_t(i);
  }
}

// The acceptance tests of request r by one warp, one lane per window position: the tests of
// different positions are independent, so every lane decides its own and the first position that is
// not accepted (a ballot) ends the window. With `write`, the accepted tokens, their log-probabilities
// and n_accepted are written (and the greedy correction or bonus). Returns the draw job through
// *kind / *jj: none (greedy, an error, or a proposal error), the residual at the first rejection, or
// the bonus draw at n.
DS_DEV void vf_accept_warp(const VerifyArgs& a, int64_t r, bool write, int* kind, int* jj) {
  const int lane = threadIdx.x & 31;
  const int B = a.B, n = a.n_draft[r];
  const int64_t obase = r * (B + 1), rbase = r * (B + 1);
  if (n < 0 || n > B) {                                    // out of contract: an error, no indexing
    if (write) {
      if (lane == 0) {
        ds_set_error(a.status, DSPARK_EINVAL);
        a.n_accepted[r] = -1;
        a.ws.job_kind[r] = JOB_NONE;
      }
      for (int k = lane; k <= B; k += 32) {
        a.out_tokens[obase + k] = -1;
        a.logprob[obase + k] = 0.0f;
      }
    }
    *kind = JOB_NONE;
    return;
  }
  const bool greedy = !(vf_T(a, r) > 0.0f);
  const uint64_t vseed = greedy ? 0 : a.vseed[r], step = greedy ? 0 : a.step[r];
  int first = n;                                           // first position that is not accepted
  bool first_zero_q = false;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    bool ev = false, zq = false;
    if (j < n) {
      const int64_t rid = rbase + j;
      const int32_t x = a.draft_tgt[r * B + j];
      if (greedy) {
        ev = x != a.ws.amax[rid];
      } else {
        const float qn = vf_qnum(a, r * B + j, x);
        zq = !(qn > 0.0f);
        if (!zq) {
          // u < p(x) / q(x) with p = w_p / W_p and q = qn / W_q (W_q = 1 for a sparse record),
          // cross-multiplied: u qn W_p < w_p W_q, in float pairs
          const rs::FF ua = rs::ff_uniform(vseed, step, uint32_t(j), DS_PURPOSE_ACCEPT);
          const rs::FF lhs = rs::ff_mul(rs::ff_mul(ua, rs::FF{qn, 0.0f}), vf_ff(a.ws.wsum[rid]));
          const rs::FF wp{a.ws.probe_w[rid], 0.0f};
          const rs::FF rhs = a.q_form == QF_SPARSE ? wp : rs::ff_mul(wp, vf_ff(a.q.wsum[r * B + j]));
          ev = !(rs::ff_diff(lhs, rhs) < 0.0f);
        }
        ev = ev || zq;
      }
    }
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, ev);
    if (bal) {
      const int l = __ffs(bal) - 1;
      first = j0 + l;
      first_zero_q = __shfl_sync(0xFFFFFFFFu, zq, l);
      break;
    }
  }
  if (first_zero_q) {                                      // the proposal gave a drafted token q = 0
    if (write) {
      if (lane == 0) {
        ds_set_error(a.status, DSPARK_EPROPOSAL);
        a.n_accepted[r] = -1;
        a.ws.job_kind[r] = JOB_NONE;
      }
      for (int k = lane; k <= B; k += 32) a.out_tokens[obase + k] = -1;
    }
    *kind = JOB_NONE;
    return;
  }
  const int acc = first;
  if (write) {
    for (int k = lane; k <= B; k += 32) {
      if (k < acc) {
        const int64_t rid = rbase + k;
        a.out_tokens[obase + k] = a.draft_tgt[r * B + k];
        a.logprob[obase + k] = __fsub_rn(logf(a.ws.probe_w[rid]), logf(float(a.ws.wsum[rid])));
      } else if (k > acc) {
        a.out_tokens[obase + k] = -1;
        a.logprob[obase + k] = 0.0f;
      } else if (greedy) {
        // the correction or bonus is the argmax of its row; it reports the temperature-1 log-prob
        // (the argmax has weight 1)
        const int64_t rid = rbase + acc;
        a.out_tokens[obase + acc] = a.ws.amax[rid];
        a.logprob[obase + acc] = -logf(float(a.ws.wsum[rid]));
      }
    }
    if (lane == 0) a.n_accepted[r] = acc;
  }
  *kind = greedy ? JOB_NONE : (acc < n ? JOB_RESIDUAL : JOB_BONUS);
  *jj = acc;
  if (write && lane == 0) {
    a.ws.job_kind[r] = *kind;
    a.ws.job_j[r] = acc;
  }
}

// ---- statistics of the target rows (no nucleus: top_p >= 1, or greedy) --------------------------
// One CTA per row at a time, persistent over rows, several CTAs per SM. Pass 1 takes the row's
// maximum over the raw 16-byte vectors (the maximum of z = s / T is fl(max s / T) for T > 0);
// pass 2 (the row again, mostly from L2) sums the weights of z - zmax with the packed weight
// function into two float pairs per thread, and finds the argmax of greedy rows. The probed
// drafted token's weight is evaluated once.
constexpr int VS_THREADS = 256;
constexpr int VS_WARPS = VS_THREADS / 32;
constexpr int VS_PER_SM = 3;

template <typename T>
DS_DEV float vs_vec_max(const uint4& v) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162*>(&w[0]);
#pragma unroll
    for (int k = 1; k < 4; ++k) m = __hmax2(m, *reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    return fmaxf(__low2float(m), __high2float(m));
  } else {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
}

template <typename T>
__global__ void __launch_bounds__(VS_THREADS, VS_PER_SM) verify_stats_kernel(const VerifyArgs a, int64_t rows) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int BATCH = 8;
  __shared__ float s_f[VS_WARPS];
  __shared__ rs::FF s_d[VS_WARPS];
  __shared__ uint32_t s_u[VS_WARPS];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ds_pdl_trigger();
  ds_pdl_wait();                                   // drafted tokens and counts may come from before
  for (int64_t rid = blockIdx.x; rid < rows; rid += gridDim.x) {
    const int64_t r = rid / (a.B + 1);
    const int j = int(rid - r * (a.B + 1));
    const float Tq = vf_T(a, r);
    const bool greedy = !(Tq > 0.0f);
    const float Tz = greedy ? 1.0f : Tq;
    const float mp = greedy ? 0.0f : vf_mp(a, r);   // min-p: the kept weights are those >= mp
    const int32_t n = a.n_draft[r];
    if (n < 0 || n > a.B) {                        // out of contract: the first row's CTA reports it
      if (j == 0 && warp == 0) {
        int kind = JOB_NONE, jj = 0;
        vf_accept_warp(a, r, true, &kind, &jj);
      }
      continue;
    }
    if (j > n) continue;                           // not needed
    const int64_t prow = a.row_start ? a.row_start[r] + j : rid;
    const T* row = reinterpret_cast<const T*>(a.logits) + prow * a.ld;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    int64_t head = int64_t(((16u - (addr & 15u)) & 15u) / sizeof(T));
    if (head > a.V) head = a.V;
    const int64_t nvec = (a.V - head) / EPV, tail0 = head + nvec * EPV;
    const uint4* rv = reinterpret_cast<const uint4*>(row + head);
    // pass 1: the maximum of the raw values
    float mx = -INFINITY;
    if (tid < head) mx = ds_load_elem<T>(row + tid);
    if (tid < a.V - tail0) mx = fmaxf(mx, ds_load_elem<T>(row + tail0 + tid));
    for (int64_t v0 = tid; v0 < nvec; v0 += int64_t(BATCH) * VS_THREADS) {
      uint4 w[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u)
        if (v0 + u * VS_THREADS < nvec) w[u] = __ldg(rv + v0 + u * VS_THREADS);
#pragma unroll
      for (int u = 0; u < BATCH; ++u)
        if (v0 + u * VS_THREADS < nvec) mx = fmaxf(mx, vs_vec_max<T>(w[u]));
    }
    mx = ds_warp_max(mx);
    if (lane == 0) s_f[warp] = mx;
    __syncthreads();
    float rmax = s_f[0];
#pragma unroll
    for (int k = 1; k < VS_WARPS; ++k) rmax = fmaxf(rmax, s_f[k]);
    const float zmax = ds_temper(rmax, Tz);
    const bool finite = zmax > -INFINITY && zmax < INFINITY;   // else reported, with no mass
    // pass 2: the sum of the weights (two float pairs per thread) and the argmax of greedy rows
    rs::FF2 acc{0, 0};
    rs::FF sc{0.0f, 0.0f};
    uint32_t amin = 0xFFFFFFFFu;
    auto scalar = [&](int64_t i) {
      const float z = ds_temper(ds_load_elem<T>(row + i), Tz);
      const float wi = ds_weight(__fsub_rn(z, zmax));
      rs::ff_add(sc, wi >= mp ? wi : 0.0f);
      if (greedy && z == zmax) amin = min(amin, uint32_t(i));
    };
    if (finite && tid < head) scalar(tid);
    if (finite && tid < a.V - tail0) scalar(tail0 + tid);
    for (int64_t v0 = tid; finite && v0 < nvec; v0 += int64_t(4) * VS_THREADS) {
      uint4 w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + u * VS_THREADS < nvec) w[u] = __ldg(rv + v0 + u * VS_THREADS);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t v = v0 + u * VS_THREADS;
        if (v < nvec) {
#pragma unroll
          for (int e = 0; e < EPV; e += 2) {
            const float z0 = ds_temper(ds_vec_elem<T>(w[u], e), Tz), z1 = ds_temper(ds_vec_elem<T>(w[u], e + 1), Tz);
            const float2 w2 = ds_weight2(__fsub_rn(z0, zmax), __fsub_rn(z1, zmax));
            rs::ff2_add(acc, ds_f2(w2.x >= mp ? w2.x : 0.0f, w2.y >= mp ? w2.y : 0.0f));
            if (greedy) {
              const uint32_t i0 = uint32_t(head + v * EPV + e);
              if (z0 == zmax) amin = min(amin, i0);
              if (z1 == zmax) amin = min(amin, i0 + 1);
            }
          }
        }
      }
    }
    rs::FF f = rs::ff2_fold(acc);
    rs::ff_acc(f, sc);
    f = rs::warp_ff_reduce(f);
    amin = __reduce_min_sync(0xFFFFFFFFu, amin);
    if (lane == 0) {
      s_d[warp] = f;
      s_u[warp] = amin;
    }
    __syncthreads();
    if (tid == 0) {
      rs::FF Wf{0.0f, 0.0f};
      uint32_t am = 0xFFFFFFFFu;
      for (int k = 0; k < VS_WARPS; ++k) {
        rs::ff_acc(Wf, s_d[k]);
        am = min(am, s_u[k]);
      }
      const double W = rs::ff_value(Wf);
      if (!finite) ds_set_error(a.status, DSPARK_ENONFINITE);
      a.ws.zmax[rid] = zmax;
      a.ws.wsum[rid] = W;
      a.ws.wcut[rid] = mp > 0.0f ? mp : 0.0f;          // min-p's cut (min_p, largest int32): w >= mp
      a.ws.icut[rid] = mp > 0.0f ? 0x7FFFFFFF : -1;
      if (greedy) a.ws.amax[rid] = int32_t(am);
      float pw = 0.0f;
      if (finite && j < n) {
        const int64_t x = a.draft_tgt[r * a.B + j];
        if (x >= 0 && x < a.V) pw = ds_weight(__fsub_rn(ds_temper(ds_load_elem<T>(row + x), Tz), zmax));
        if (pw < mp) pw = 0.0f;
      }
      a.ws.probe_w[rid] = pw;
      // the CTA that completes the request's last needed row runs its acceptance tests
      __threadfence();
      s_last = atomicAdd(&a.ws.tk_stats[r], 1) == n;
    }
    __syncthreads();
    if (s_last && warp == 0) {
      __threadfence();
      int kind = JOB_NONE, jj = 0;
      vf_accept_warp(a, r, true, &kind, &jj);
    }
    __syncthreads();                                 // the reduction slots are reused by the next row
  }
}

// The acceptance tests after the row sampler's statistics (rows with a nucleus): one warp per request.
__global__ void __launch_bounds__(128) verify_accept_kernel(const VerifyArgs a, int64_t R) {
  const int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  ds_pdl_trigger();
  ds_pdl_wait();
  if (r >= R) return;                                      // whole warps leave together
  int kind = JOB_NONE, jj = 0;
  vf_accept_warp(a, r, true, &kind, &jj);
}

// ---- residual masses ---------------------------------------------------------------------------
// Per job: the target row's statistics and the record row, so that rho'(t) = rho(t) * W_p * W_q
// needs no division: max(0, w_p(t) W_q - w_q(t) W_p) for a dense q, max(0, w_p(t) - q(t) W_p) for a
// sparse q, and w_p(t) when drawing from p. Each is a float pair (about 48 significant bits).
template <typename T>
struct VfJob {
  const T* row;
  float zmax, wcut;
  int64_t icut;
  double Wp;
  float wp_hi, wp_lo, wq_hi, wq_lo;
  int64_t qrow;
  bool use_q;
  float Tq;                  // the request's temperature
};

template <typename T>
DS_DEV VfJob<T> vf_job(const VerifyArgs& a, int64_t r, int j, bool use_q) {
  VfJob<T> g;
  const int64_t rid = r * (a.B + 1) + j;
  const int64_t prow = a.row_start ? a.row_start[r] + j : rid;
  g.row = reinterpret_cast<const T*>(a.logits) + prow * a.ld;
  g.zmax = a.ws.zmax[rid];
  g.wcut = a.ws.wcut[rid];
  g.icut = a.ws.icut[rid];
  g.Wp = a.ws.wsum[rid];
  g.qrow = r * a.B + j;
  g.use_q = use_q;
  g.Tq = vf_T(a, r);
  g.wp_hi = float(g.Wp);
  g.wp_lo = float(g.Wp - double(g.wp_hi));
  const double Wq = (use_q && a.q_form >= QF_DENSE) ? a.q.wsum[g.qrow] : 1.0;
  g.wq_hi = float(Wq);
  g.wq_lo = float(Wq - double(g.wq_hi));
  return g;
}

DS_DEV rs::FF vf_ff_mul(float x, float dh, float dl) {     // x * (dh + dl) as a float pair
  const float pr = __fmul_rn(x, dh);
  return rs::FF{pr, __fadd_rn(__fmaf_rn(x, dh, -pr), __fmul_rn(x, dl))};
}

// rho' of one id from its target weight and its q term (a dense record's kept weight, or a sparse
// record's probability)
template <typename T>
DS_DEV rs::FF vf_rho(const VerifyArgs& a, const VfJob<T>& g, float wp, float qterm) {
  if (!g.use_q) return rs::FF{wp, 0.0f};
  rs::FF av, bv;
  if (a.q_form >= QF_DENSE) {
    av = vf_ff_mul(wp, g.wq_hi, g.wq_lo);
    bv = vf_ff_mul(qterm, g.wp_hi, g.wp_lo);
  } else {
    av = rs::FF{wp, 0.0f};
    bv = vf_ff_mul(qterm, g.wp_hi, g.wp_lo);
  }
  // a - b with the rounding error of the leading difference kept (2Sum)
  const float sd = __fsub_rn(av.hi, bv.hi);
  const float bb = __fsub_rn(sd, av.hi);
  const float err = __fadd_rn(__fsub_rn(av.hi, __fsub_rn(sd, bb)), __fsub_rn(-bv.hi, bb));
  const float lo = __fadd_rn(err, __fsub_rn(av.lo, bv.lo));
  if (!(__fadd_rn(sd, lo) > 0.0f)) return rs::FF{0.0f, 0.0f};
  return rs::FF{sd, lo};
}

// Eight consecutive elements t..t+7 of a row (t % 8 == 0), zero past `n`; 16-byte loads when the
// eight are whole and aligned.
template <typename T>
DS_DEV void vf_ld8(const T* p, int64_t t, int64_t n, float (&x)[8]) {
  const T* q = p + t;
  if (t + 8 <= n && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
    if constexpr (sizeof(T) == 2) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(q));
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = ds_vec_elem<T>(v, e);
    } else {
      const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(q)), v1 = __ldg(reinterpret_cast<const uint4*>(q) + 1);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] = ds_vec_elem<T>(v0, e);
        x[e + 4] = ds_vec_elem<T>(v1, e);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (t + e < n) ? ds_load_elem<T>(q + e) : 0.0f;
  }
}

DS_DEV void vf_ld8_i32(const int32_t* p, int64_t t, int64_t n, int32_t (&x)[8]) {
  const int32_t* q = p + t;
  if (t + 8 <= n && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
    const int4 v0 = __ldg(reinterpret_cast<const int4*>(q)), v1 = __ldg(reinterpret_cast<const int4*>(q) + 1);
    x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
    x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = (t + e < n) ? __ldg(q + e) : -1;
  }
}

// rho' of the eight ids t..t+7 (zero past V). s_q: a sparse record's q by id, indexed from s_q0.
template <typename T, int QF, bool TONE>
DS_DEV void vf_rho8(const VerifyArgs& a, const VfJob<T>& g, int64_t t, const float* s_q, int64_t s_q0,
                    rs::FF (&out)[8]) {
  float x[8];
  vf_ld8<T>(g.row, t, a.V, x);
  float qt[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) qt[e] = 0.0f;
  if (g.use_q) {
    if constexpr (QF == QF_SPARSE) {
#pragma unroll
      for (int e = 0; e < 8; ++e) qt[e] = (t + e < a.V) ? s_q[t + e - s_q0] : 0.0f;
    } else if constexpr (QF == QF_DENSE) {
      float zq[8];
      vf_ld8<float>(a.q.z + g.qrow * a.q.ldz, t, a.V_q, zq);
      const float zm = a.q.zmax[g.qrow], wc = a.q.wcut[g.qrow];
      const int64_t ic = a.q.icut[g.qrow];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float2 w2 = ds_weight2(__fsub_rn(zq[e], zm), __fsub_rn(zq[e + 1], zm));
        if (t + e < a.V_q) qt[e] = vf_keep(w2.x, t + e, wc, ic) ? w2.x : 0.0f;
        if (t + e + 1 < a.V_q) qt[e + 1] = vf_keep(w2.y, t + e + 1, wc, ic) ? w2.y : 0.0f;
      }
    } else if constexpr (QF == QF_DENSE_PRUNED) {
      int32_t ii[8];
      vf_ld8_i32(a.ws.t2d, t, a.V, ii);
#pragma unroll
      for (int e = 0; e < 8; ++e) qt[e] = vf_wq(a, g.qrow, ii[e]);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const float2 w2 = ds_weight2(__fsub_rn(ds_temper_t<TONE>(x[e], g.Tq), g.zmax),
                                 __fsub_rn(ds_temper_t<TONE>(x[e + 1], g.Tq), g.zmax));
    float wp0 = w2.x, wp1 = w2.y;
    if (!(t + e < a.V) || !vf_keep(wp0, t + e, g.wcut, g.icut)) wp0 = 0.0f;
    if (!(t + e + 1 < a.V) || !vf_keep(wp1, t + e + 1, g.wcut, g.icut)) wp1 = 0.0f;
    out[e] = vf_rho<T>(a, g, wp0, qt[e]);
    out[e + 1] = vf_rho<T>(a, g, wp1, qt[e + 1]);
  }
}

// Stages a sparse record's q for ids [lo, lo + len) into s_q (zero elsewhere); whole block.
DS_DEV void vf_stage_sparse(const VerifyArgs& a, int64_t qrow, int64_t lo, int len, float* s_q) {
  for (int i = threadIdx.x; i < len; i += blockDim.x) s_q[i] = 0.0f;
  __syncthreads();
  const int n = min(a.q.n[qrow], a.q.cap);
  for (int k = threadIdx.x; k < n; k += blockDim.x) {
    const int64_t id = a.q.ids[qrow * a.q.cap + k];
    if (id >= lo && id < lo + len) s_q[id - lo] = a.q.p[qrow * a.q.cap + k];
  }
  __syncthreads();
}

// One CTA per (part of a draw row, request). Warp 0 first runs the request's acceptance tests
// (the same decisions in every part; part 0 writes the accepted tokens), which name the draw job;
// the CTA then writes the residual mass of every cell of its part, and the part that finishes last
// (a ticket per request) picks the token: it scans all the row's cells in double, finds the cell
// whose running sum crosses u * sum(rho), and re-evaluates that cell's ids.
template <typename T, int QF, bool TONE>
__global__ void __launch_bounds__(VM_THREADS, 2) verify_draw_kernel(const VerifyArgs a) {
  const int CPP = (QF == QF_SPARSE) ? VM_PART_SPARSE / VM_CELL : a.part_cells;   // cells per part
  const int64_t PART = int64_t(CPP) * VM_CELL;
  constexpr int WARPS = VM_THREADS / 32;
  __shared__ float s_q[QF == QF_SPARSE ? VM_PART_SPARSE : 1];
  __shared__ rs::PickShared<VM_THREADS> s_pk;
  __shared__ int s_last;
  ds_pdl_trigger();
  ds_pdl_wait();
  const int64_t r = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t kind = a.ws.job_kind[r];
  if (kind == JOB_NONE) return;                            // the whole request has no draw
  const int j = a.ws.job_j[r];
  const int64_t t0 = int64_t(blockIdx.x) * PART;
  VfJob<T> g = vf_job<T>(a, r, j, kind == JOB_RESIDUAL);
  if (QF == QF_SPARSE && g.use_q) vf_stage_sparse(a, g.qrow, t0, PART, s_q);
  float2* cells = a.ws.cells + r * a.ncell;
  for (int k0 = warp; k0 < CPP; k0 += 2 * WARPS) {        // two cells per warp in flight
    rs::FF v[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int cl = k0 + u * WARPS;
      const int64_t t = t0 + int64_t(cl) * VM_CELL + lane * 8;
      if (cl < CPP && t < a.V) vf_rho8<T, QF, TONE>(a, g, t, s_q, t0, v[u]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int cl = k0 + u * WARPS;
      const int64_t c = t0 / VM_CELL + cl;
      if (cl >= CPP || c * VM_CELL >= a.V) continue;       // warp-uniform
      const int64_t t = c * VM_CELL + lane * 8;
      rs::FF m{0.0f, 0.0f};
      if (t < a.V) {
#pragma unroll
        for (int e = 0; e < 8; ++e) rs::ff_acc(m, v[u][e]);
      }
      const rs::FF cw = rs::warp_ff_reduce(m);
      if (lane == 0) cells[c] = make_float2(cw.hi, cw.lo);
    }
  }
  // the last part to finish picks the token
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&a.ws.tk_draw[r], 1) == int(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // the crossing cell: the first whose running sum exceeds u * total (float pairs)
  const rs::FF u = rs::ff_uniform(a.vseed[r], a.step[r], uint32_t(j), DS_PURPOSE_RESIDUAL);
  rs::pick_cell<VM_THREADS>(cells, a.ncell, u, s_pk);
  if (!(s_pk.total.hi > 0.0f)) {
    // the residual has no mass (possible only through rounding): draw from p, whose cells this CTA
    // recomputes over the whole row (rare)
    g.use_q = false;
    for (int64_t c = warp; c < a.ncell; c += WARPS) {
      const int64_t t = c * VM_CELL + lane * 8;
      rs::FF v[8];
      rs::FF m{0.0f, 0.0f};
      if (t < a.V) {
        vf_rho8<T, QF, TONE>(a, g, t, s_q, 0, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) rs::ff_acc(m, v[e]);
      }
      const rs::FF cw = rs::warp_ff_reduce(m);
      if (lane == 0) cells[c] = make_float2(cw.hi, cw.lo);
    }
    __threadfence_block();
    __syncthreads();
    rs::pick_cell<VM_THREADS>(cells, a.ncell, u, s_pk);
  }
  const int64_t cell = s_pk.cell == ~0ull ? -1 : int64_t(s_pk.cell);
  int64_t pick = -1;
  if (cell >= 0) {
    if (QF == QF_SPARSE && g.use_q) vf_stage_sparse(a, g.qrow, cell * VM_CELL, VM_CELL, s_q);
    if (warp == 0) {
      const int64_t t = cell * VM_CELL + lane * 8;
      rs::FF v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = rs::FF{0.0f, 0.0f};
      if (t < a.V) vf_rho8<T, QF, TONE>(a, g, t, s_q, cell * VM_CELL, v);
      pick = rs::warp_pick<8>(v, s_pk.tau, s_pk.tinf != 0, cell * VM_CELL);
    }
  }
  if (tid == 0) {
    float w = 0.0f;
    if (pick >= 0) {
      const float x = ds_load_elem<T>(g.row + pick);
      w = ds_weight(__fsub_rn(ds_temper_t<TONE>(x, g.Tq), g.zmax));
    }
    a.out_tokens[r * (a.B + 1) + j] = int32_t(pick);
    a.logprob[r * (a.B + 1) + j] = __fsub_rn(logf(w), logf(g.wp_hi));
  }
}

size_t vf_align(size_t x) { return (x + 255) & ~size_t(255); }

VerifyWs vf_layout(void* base, int64_t R, int32_t B, int64_t V, size_t* total) {
  const size_t rows = size_t(R) * (B + 1);
  const size_t ncell = size_t((V + VM_CELL - 1) / VM_CELL);
  uint8_t* p = reinterpret_cast<uint8_t*>(base);
  size_t off = 0;
  VerifyWs w = {};
  auto take = [&](size_t bytes) {
    uint8_t* q = p ? p + off : nullptr;
    off += vf_align(bytes);
    return q;
  };
  w.zmax = reinterpret_cast<float*>(take(rows * 4));
  w.wsum = reinterpret_cast<double*>(take(rows * 8));
  w.wcut = reinterpret_cast<float*>(take(rows * 4));
  w.icut = reinterpret_cast<int32_t*>(take(rows * 4));
  w.probe_w = reinterpret_cast<float*>(take(rows * 4));
  w.amax = reinterpret_cast<int32_t*>(take(rows * 4));
  w.job_kind = reinterpret_cast<int32_t*>(take(size_t(R) * 4));
  w.job_j = reinterpret_cast<int32_t*>(take(size_t(R) * 4));
  w.tk_stats = reinterpret_cast<int32_t*>(take(size_t(R) * 2 * 4));   // both ticket arrays, cleared together
  w.tk_draw = w.tk_stats ? w.tk_stats + R : nullptr;
  w.cells = reinterpret_cast<float2*>(take(size_t(R) * ncell * sizeof(float2)));
  w.t2d = reinterpret_cast<int32_t*>(take(size_t(V) * 4));
  *total = off;
  return w;
}

template <typename T, int QF, bool TONE>
cudaError_t vf_launch_draws(const VerifyArgs& a, int64_t R, cudaStream_t stream) {
  VerifyArgs b = a;
  if (QF == QF_SPARSE) {
    b.part_cells = VM_PART_SPARSE / VM_CELL;
  } else {
    // as many parts per request as leave every request's parts in one wave of resident CTAs (two
    // per SM): a second, nearly empty wave would double the kernel's time
    const int64_t slots = int64_t(2) * ds_num_sms();
    int64_t np = std::max<int64_t>(1, slots / std::max<int64_t>(R, 1));
    np = std::min<int64_t>(np, std::max<int64_t>(1, a.ncell / VM_PART_MIN_CELLS));
    b.part_cells = int32_t((a.ncell + np - 1) / np);
  }
  const dim3 grid(unsigned((b.ncell + b.part_cells - 1) / b.part_cells), unsigned(R));
  return ds_launch(verify_draw_kernel<T, QF, TONE>, grid, dim3(VM_THREADS), 0, stream, b);
}

template <typename T, bool TONE>
cudaError_t vf_launch_draws_form(const VerifyArgs& a, int64_t R, cudaStream_t stream) {
  switch (a.q_form) {
    case QF_SPARSE: return vf_launch_draws<T, QF_SPARSE, TONE>(a, R, stream);
    case QF_DENSE: return vf_launch_draws<T, QF_DENSE, TONE>(a, R, stream);
    default: return vf_launch_draws<T, QF_DENSE_PRUNED, TONE>(a, R, stream);
  }
}

template <typename T>
cudaError_t vf_launch_draws_any(const VerifyArgs& a, int64_t R, cudaStream_t stream) {
  return (a.T == 1.0f && !a.T_r) ? vf_launch_draws_form<T, true>(a, R, stream) : vf_launch_draws_form<T, false>(a, R, stream);
}

}  // namespace

extern "C" size_t dspark_internal_ws_verify(int64_t R, int32_t B, int64_t V) {
  size_t total = 0;
  vf_layout(nullptr, R, B, V, &total);
  return total;
}

extern "C" dspark_status dspark_verify(const void* tgt_logits, dspark_dtype dtype, int64_t R, int32_t B, int64_t V_t,
                                       int64_t ld, const int64_t* row_start, const int32_t* draft_tgt,
                                       const int32_t* n_draft, const dspark_qrecord* q, int64_t V_q,
                                       const int64_t* q_d2t, float temperature, float top_p, float min_p,
                                       const float* temperature_r, const float* top_p_r, const float* min_p_r,
                                       const uint64_t* vseed,
                                       const uint64_t* step, int32_t* out_tokens, int32_t* n_accepted, float* logprob,
                                       void* ws, size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype) && R >= 0 && B >= 1 && B <= 100 && V_t >= 1 && ld >= V_t);
  DS_REQUIRE(V_t <= 0x7FFFFFFF && R * (B + 1) <= 0x7FFFFFFF);
  DS_REQUIRE(tgt_logits && draft_tgt && n_draft && out_tokens && n_accepted && logprob && dev_status);
  DS_REQUIRE(ds_aligned(tgt_logits, ds_dtype_size(dtype)));
  DS_REQUIRE(temperature == temperature && top_p == top_p && top_p > 0.0f && min_p >= 0.0f && min_p <= 1.0f);
  const bool greedy = !(temperature > 0.0f) && !temperature_r;   // every request greedy
  int q_form = QF_NONE;
  if (!greedy) {
    DS_REQUIRE(vseed && step && q);
    if (q->z) {
      DS_REQUIRE(q->zmax && q->wsum && q->wcut && q->icut && q->ldz >= V_q && V_q >= 1 && V_q <= 0x7FFFFFFF);
      q_form = q_d2t ? QF_DENSE_PRUNED : QF_DENSE;
    } else {
      DS_REQUIRE(q->ids && q->p && q->n && q->cap >= 1 && !q_d2t);
      q_form = QF_SPARSE;
    }
  }
  const int C = rs::cluster_size_for(V_t, ds_dtype_size(dtype));
  DS_REQUIRE(C > 0);
  if (R == 0) return DSPARK_OK;
  size_t need = 0;
  vf_layout(nullptr, R, B, V_t, &need);
  if (!ws || ws_bytes < need || !ds_aligned(ws, 256)) return DSPARK_EWORKSPACE;
  VerifyArgs a = {};
  a.logits = tgt_logits;
  a.V = V_t;
  a.ld = ld;
  a.row_start = row_start;
  a.B = B;
  a.draft_tgt = draft_tgt;
  a.n_draft = n_draft;
  if (q) a.q = *q;
  a.q_form = q_form;
  a.V_q = V_q;
  a.T = temperature;
  a.top_p = top_p;
  a.T_r = temperature_r;
  a.top_p_r = top_p_r;
  a.min_p = min_p;
  a.min_p_r = min_p_r;
  a.vseed = vseed;
  a.step = step;
  a.out_tokens = out_tokens;
  a.n_accepted = n_accepted;
  a.logprob = logprob;
  a.status = dev_status;
  a.ncell = (V_t + VM_CELL - 1) / VM_CELL;
  a.ws = vf_layout(ws, R, B, V_t, &need);

  // 0. inverse map of a pruned dense record
  if (q_form == QF_DENSE_PRUNED) {
    DS_CUDA_TRY(cudaMemsetAsync(a.ws.t2d, 0xFF, size_t(V_t) * sizeof(int32_t), stream));
    const unsigned blocks = unsigned(std::min<int64_t>(ds_ceil_div(V_q, 256), int64_t(ds_num_sms()) * 8));
    verify_t2d_kernel<<<blocks, 256, 0, stream>>>(q_d2t, V_q, V_t, a.ws.t2d, dev_status);
    DS_CUDA_TRY(cudaGetLastError());
  }

  DS_CUDA_TRY(cudaMemsetAsync(a.ws.tk_stats, 0, size_t(R) * 2 * sizeof(int32_t), stream));
  // 1. statistics of every needed target row, and the acceptance tests
  const bool lean = greedy || (!(top_p < 1.0f) && !top_p_r);
  if (lean) {
    const int64_t grid = std::min<int64_t>(R * (B + 1), int64_t(ds_num_sms()) * VS_PER_SM);
    if (dtype == DSPARK_BF16)
      DS_CUDA_TRY(ds_launch(verify_stats_kernel<__nv_bfloat16>, dim3(unsigned(grid)), dim3(VS_THREADS), 0, stream, a,
                            R * (B + 1)));
    else
      DS_CUDA_TRY(ds_launch(verify_stats_kernel<float>, dim3(unsigned(grid)), dim3(VS_THREADS), 0, stream, a,
                            R * (B + 1)));
  } else {
  rs::SampleArgs sa = {};
  sa.rows = tgt_logits;
  sa.V = V_t;
  sa.ld = ld;
  sa.row_start = row_start;
  sa.row_mul = 1;
  sa.B = B + 1;
  sa.C = C;
  sa.mult = 1.0f;
  sa.softcap = 0.0f;
  sa.T = greedy ? 1.0f : temperature;
  sa.top_p = greedy ? 1.0f : top_p;
  sa.T_r = temperature_r;
  sa.top_p_r = top_p_r;
  sa.min_p = greedy ? 0.0f : min_p;
  sa.min_p_r = min_p_r;
  sa.position = -1;
  sa.out_mul = 1;
  sa.status = dev_status;
  sa.q.zmax = a.ws.zmax;
  sa.q.wsum = a.ws.wsum;
  sa.q.wcut = a.ws.wcut;
  sa.q.icut = a.ws.icut;
  sa.q_mode = 2;
  sa.q_row_mul = 1;
  sa.no_draw = 1;
  sa.probe_tgt = draft_tgt;
  sa.n_draft = n_draft;
  sa.probe_w = a.ws.probe_w;
  sa.amax_out = (greedy || temperature_r) ? a.ws.amax : nullptr;
  DS_CUDA_TRY(rs::sample_rows(sa, R * (B + 1), dtype == DSPARK_BF16, 0, stream));
  DS_CUDA_TRY(ds_launch(verify_accept_kernel, dim3(unsigned((R * 32 + 127) / 128)), dim3(128), 0, stream, a, R));
  }

  if (greedy) return DSPARK_OK;
  // 2. residual or bonus draws
  const cudaError_t e = dtype == DSPARK_BF16 ? vf_launch_draws_any<__nv_bfloat16>(a, R, stream)
                                             : vf_launch_draws_any<float>(a, R, stream);
  DS_CUDA_TRY(e);
  return DSPARK_OK;
}
