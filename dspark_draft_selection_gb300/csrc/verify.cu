// verify.cu - rejection-sampling verification of drafted tokens (dspark_verify).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"): commit on exact sampled speculative decoding - each window
// position is checked against the target's post-filter p, accepted with probability min(1, p/q),
// otherwise a sample of norm(max(0, p - q)) is emitted and the later candidates dropped;
// accepted tokens report the target's log-probability; ids beyond a model's row have zero
// probability; sums in double. Commit on the double uniform (acceptance test and draws).
// Description > Fixes > Split validation windows: row j validates candidate j; row n is the
// bonus row. This is the speculative sampling rule of Leviathan et al. (2023) and Chen et al.
// (2023).
//
// Three launches:
//  1. the row sampler of sample.cu in statistics mode over every needed target row:
//     the maximum, the top-p cut and the kept mass of p_j, the weight of the drafted token x_j,
//     and the argmax (greedy requests). The target logits are read from HBM once here.
//  2. verify_accept_kernel - one thread per request runs the sequential tests
//     u_j < p_j(x_j) / q_j(x_j) and leaves at most one draw job (residual at j*, or bonus at n).
//  3. verify_draw_kernel - one 1024-thread CTA per request with a job re-reads that one row
//     (and the dense q row), forms rho = max(0, p - q) (or p) scaled by W_p * W_q so that no
//     element needs a division (float pairs per element, double per warp), and finds the
//     crossing of u * sum(rho) with per-(round, warp) sums and short scans.
#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int VD_THREADS = 1024;
constexpr int VD_WARPS = VD_THREADS / 32;
constexpr int VD_MAXROUNDS = 256;        // rows up to 262,144 ids
constexpr int VD_SPARSE_MAX = 1024;      // sparse q entries staged per draw

enum : int32_t { JOB_NONE = 0, JOB_RESIDUAL = 1, JOB_BONUS = 2 };

struct VerifyWs {
  float* zmax;       // [R * (B + 1)]
  double* wsum;
  float* wcut;
  int32_t* icut;
  float* probe_w;
  int32_t* amax;
  int32_t* job_kind; // [R]
  int32_t* job_j;
};

struct VerifyArgs {
  const void* logits;
  int64_t V, ld;
  const int64_t* row_start;
  int32_t B;
  const int32_t* draft_tgt;
  const int32_t* n_draft;
  dspark_qrecord q;
  int q_dense;
  int64_t V_q;
  float T, top_p;
  const uint64_t* vseed;
  const uint64_t* step;
  int32_t* out_tokens;
  int32_t* n_accepted;
  float* logprob;
  int32_t* status;
  VerifyWs ws;
};

DS_DEV bool vf_keep(float w, int64_t i, float wcut, int64_t icut) {
  return w > 0.0f && (w > wcut || (w == wcut && i <= icut));
}

// q_j(x) from the record (double); ids outside the record's width have probability zero
DS_DEV double vf_q(const VerifyArgs& a, int64_t qrow, int64_t x) {
  if (x < 0) return 0.0;
  if (a.q_dense) {
    if (x >= a.V_q) return 0.0;
    const float w = ds_weight(__fsub_rn(a.q.z[qrow * a.q.ldz + x], a.q.zmax[qrow]));
    return vf_keep(w, x, a.q.wcut[qrow], a.q.icut[qrow]) ? double(w) / a.q.wsum[qrow] : 0.0;
  }
  const int n = a.q.n[qrow];
  for (int k = 0; k < n && k < a.q.cap; ++k)
    if (a.q.ids[qrow * a.q.cap + k] == x) return double(a.q.p[qrow * a.q.cap + k]);
  return 0.0;
}

__global__ void verify_accept_kernel(const VerifyArgs a, int64_t R) {
  const int64_t r = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
  if (r >= R) return;
  const int B = a.B, n = a.n_draft[r];
  const int64_t obase = r * (B + 1), rbase = r * (B + 1);
  const bool greedy = !(a.T > 0.0f);
  const uint64_t vseed = greedy ? 0 : a.vseed[r], step = greedy ? 0 : a.step[r];
  int acc = 0;
  int32_t kind = JOB_BONUS, jj = n;
  for (int j = 0; j < n; ++j) {
    const int64_t rid = rbase + j;
    const int32_t x = a.draft_tgt[r * B + j];
    const double lw = log(double(a.ws.probe_w[rid])) - log(a.ws.wsum[rid]);
    if (greedy) {
      if (x == a.ws.amax[rid]) {
        a.out_tokens[obase + acc] = x;
        a.logprob[obase + acc] = float(lw);
        ++acc;
        continue;
      }
      kind = JOB_RESIDUAL;
      jj = j;
      break;
    }
    const double qx = vf_q(a, r * B + j, x);
    if (!(qx > 0.0)) {
      ds_set_error(a.status, DSPARK_EPROPOSAL);
      a.n_accepted[r] = -1;
      for (int k = 0; k <= B; ++k) a.out_tokens[obase + k] = -1;
      a.ws.job_kind[r] = JOB_NONE;
      return;
    }
    const double px = double(a.ws.probe_w[rid]) / a.ws.wsum[rid];
    const double ua = ds_uniform(vseed, step, uint32_t(j), DS_PURPOSE_ACCEPT);
    if (ua < px / qx) {
      a.out_tokens[obase + acc] = x;
      a.logprob[obase + acc] = float(lw);
      ++acc;
      continue;
    }
    kind = JOB_RESIDUAL;
    jj = j;
    break;
  }
  a.n_accepted[r] = acc;
  for (int k = acc + 1; k <= B; ++k) {
    a.out_tokens[obase + k] = -1;
    a.logprob[obase + k] = 0.0f;
  }
  if (greedy) {
    // the correction or bonus is the argmax of its row; it reports the temperature-1 log-prob
    const int64_t rid = rbase + jj;
    a.out_tokens[obase + acc] = a.ws.amax[rid];
    a.logprob[obase + acc] = float(-log(a.ws.wsum[rid]));   // the argmax has weight 1
    a.ws.job_kind[r] = JOB_NONE;
  } else {
    a.ws.job_kind[r] = kind;
    a.ws.job_j[r] = jj;
  }
}

template <typename T>
__global__ void __launch_bounds__(VD_THREADS, 1) verify_draw_kernel(const VerifyArgs a) {
  extern __shared__ __align__(16) float2 s_rwf[];         // [rounds][VD_WARPS] float pairs
  __shared__ double s_scan[VD_MAXROUNDS];
  __shared__ double s_wtot[VD_WARPS];
  __shared__ int32_t s_sid[VD_SPARSE_MAX];
  __shared__ float s_sq[VD_SPARSE_MAX];
  __shared__ int s_pick, s_round, s_warp;
  __shared__ double s_tau;

  const int64_t r = blockIdx.x;
  const int32_t kind = a.ws.job_kind[r];
  if (kind == JOB_NONE) return;
  const int B = a.B, j = a.ws.job_j[r];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rid = r * (B + 1) + j;
  const int64_t prow = a.row_start ? a.row_start[r] + j : rid;
  const T* row = reinterpret_cast<const T*>(a.logits) + prow * a.ld;
  const float zmax = a.ws.zmax[rid], wcut = a.ws.wcut[rid];
  const int64_t icut = a.ws.icut[rid];
  const double wsum = a.ws.wsum[rid];
  const int64_t qrow = r * B + j;
  const bool resid = kind == JOB_RESIDUAL;
  const int64_t V = a.V;
  const int nrounds = int((V + VD_THREADS - 1) / VD_THREADS);

  // sparse q of this position, staged (ids are looked up by scan; the record holds few entries)
  int ns = 0;
  if (resid && !a.q_dense) {
    ns = min(a.q.n[qrow], min(a.q.cap, VD_SPARSE_MAX));
    for (int k = tid; k < ns; k += VD_THREADS) {
      s_sid[k] = a.q.ids[qrow * a.q.cap + k];
      s_sq[k] = a.q.p[qrow * a.q.cap + k];
    }
    __syncthreads();
  }
  auto pval = [&](int64_t t, float* wout) -> double {
    const float z = ds_temper(ds_load_elem<T>(row + t), a.T);
    const float w = ds_weight(__fsub_rn(z, zmax));
    if (wout) *wout = w;
    return vf_keep(w, t, wcut, icut) ? double(w) / wsum : 0.0;
  };
  // Residual masses scaled by W_p * W_q, so that no element needs a division (the draw only
  // needs the masses up to a common factor): rho'(t) = max(0, w_p(t) W_q - w_q(t) W_p) for a
  // dense q, max(0, w_p(t) - q(t) W_p) for a sparse q, and w_p(t) when drawing from p. Each is a
  // float pair (about 48 bits); the double pipe only sees per-warp sums.
  const double Wq = (resid && a.q_dense) ? a.q.wsum[qrow] : 1.0;
  const float wp_hi = float(wsum), wp_lo = float(wsum - double(float(wsum)));
  const float wq_hi = float(Wq), wq_lo = float(Wq - double(float(Wq)));
  auto ff_mul = [](float x, float dh, float dl) {        // x * (dh + dl) as a float pair
    const float pr = __fmul_rn(x, dh);
    return rs::FF{pr, __fadd_rn(__fmaf_rn(x, dh, -pr), __fmul_rn(x, dl))};
  };
  auto rho_ff = [&](int64_t t, bool use_q) -> rs::FF {
    float wp = ds_weight(__fsub_rn(ds_temper(ds_load_elem<T>(row + t), a.T), zmax));
    if (!vf_keep(wp, t, wcut, icut)) wp = 0.0f;
    if (!use_q) return rs::FF{wp, 0.0f};
    rs::FF av, bv;
    if (a.q_dense) {
      float wq = 0.0f;
      if (t < a.V_q) {
        wq = ds_weight(__fsub_rn(a.q.z[qrow * a.q.ldz + t], a.q.zmax[qrow]));
        if (!vf_keep(wq, t, a.q.wcut[qrow], a.q.icut[qrow])) wq = 0.0f;
      }
      av = ff_mul(wp, wq_hi, wq_lo);
      bv = ff_mul(wq, wp_hi, wp_lo);
    } else {
      float q = 0.0f;
      for (int k = 0; k < ns; ++k)
        if (s_sid[k] == t) q = s_sq[k];
      av = rs::FF{wp, 0.0f};
      bv = ff_mul(q, wp_hi, wp_lo);
    }
    // a - b with the rounding error of the leading difference kept (2Sum)
    const float sd = __fsub_rn(av.hi, bv.hi);
    const float bb = __fsub_rn(sd, av.hi);
    const float err = __fadd_rn(__fsub_rn(av.hi, __fsub_rn(sd, bb)), __fsub_rn(-bv.hi, bb));
    const float lo = __fadd_rn(err, __fsub_rn(av.lo, bv.lo));
    if (!(__fadd_rn(sd, lo) > 0.0f)) return rs::FF{0.0f, 0.0f};
    return rs::FF{sd, lo};
  };
  auto rho = [&](int64_t t, bool use_q) -> double { return rs::ff_value(rho_ff(t, use_q)); };

  const double u = ds_uniform(a.vseed[r], a.step[r], uint32_t(j), DS_PURPOSE_RESIDUAL);
  bool use_q = resid;
  for (int attempt = 0; attempt < 2; ++attempt) {
    // per-(round, warp) sums in index order
    // four rounds at a time: their masses are formed first (all loads in flight together), then
    // summed per warp
    for (int k0 = 0; k0 < nrounds; k0 += 4) {
      rs::FF f[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t t = int64_t(k0 + u) * VD_THREADS + tid;
        f[u] = (k0 + u < nrounds && t < V) ? rho_ff(t, use_q) : rs::FF{0.0f, 0.0f};
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (k0 + u >= nrounds) break;
        const rs::FF v = rs::warp_ff_reduce(f[u]);          // kept as a float pair (no FP64 here)
        if (lane == 0) s_rwf[(k0 + u) * VD_WARPS + warp] = make_float2(v.hi, v.lo);
      }
    }
    __syncthreads();
    // round totals in float pairs, one double per round, and their running sums
    for (int k = tid; k < nrounds; k += VD_THREADS) {
      rs::FF sum{0.0f, 0.0f};
      for (int w = 0; w < VD_WARPS; ++w) {
        const float2 c = s_rwf[k * VD_WARPS + w];
        const float lo = __fadd_rn(sum.lo, c.y);
        sum.lo = 0.0f;
        rs::ff_add(sum, c.x);
        sum.lo = __fadd_rn(sum.lo, lo);
      }
      s_scan[k] = rs::ff_value(sum);
    }
    __syncthreads();
    if (tid == 0) {
      double accum = 0.0;
      for (int k = 0; k < nrounds; ++k) {
        const double nx = accum + s_scan[k];
        s_scan[k] = accum;                 // exclusive prefix
        accum = nx;
      }
      s_wtot[0] = accum;
    }
    __syncthreads();
    const double total = s_wtot[0];
    if (total > 0.0 || attempt == 1) break;
    use_q = false;                         // the residual has no mass (rounding): draw from p
    __syncthreads();
  }
  const double total = s_wtot[0];
  const double target = u * total;
  if (tid == 0) {
    int kr = -1, kw = -1;
    double tau = 0.0;
    for (int k = 0; k < nrounds && kr < 0; ++k) {
      const double next = (k + 1 < nrounds) ? s_scan[k + 1] : total;
      if (!(target < next)) continue;                  // the crossing is in a later round
      double acc = s_scan[k];
      for (int w = 0; w < VD_WARPS; ++w) {
        const double cw = double(s_rwf[k * VD_WARPS + w].x) + double(s_rwf[k * VD_WARPS + w].y);
        const double nx = acc + cw;
        if (target < nx && cw > 0.0) {
          kr = k;
          kw = w;
          tau = target - acc;
          break;
        }
        acc = nx;
      }
    }
    s_round = kr;
    s_warp = kw;
    s_tau = tau;
    s_pick = -1;
  }
  __syncthreads();
  if (s_round >= 0 && warp == s_warp) {
    const int64_t t = int64_t(s_round) * VD_THREADS + tid;
    const double v = (t < V) ? rho(t, use_q) : 0.0;
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double nn = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += nn;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, v > 0.0 && incl > s_tau);
    const unsigned pos = __ballot_sync(0xFFFFFFFFu, v > 0.0);
    if (lane == 0) s_pick = hit ? int(s_round * VD_THREADS + warp * 32 + __ffs(hit) - 1)
                               : (pos ? int(s_round * VD_THREADS + warp * 32 + 31 - __clz(int(pos))) : -1);
  }
  __syncthreads();
  if (tid == 0) {
    int64_t pick = s_pick;
    if (pick < 0) {
      // the target fell past the last boundary by rounding: the last id with positive mass
      for (int64_t t = V - 1; t >= 0; --t)
        if (rho(t, use_q) > 0.0) {
          pick = t;
          break;
        }
    }
    const int acc = a.n_accepted[r];
    float w = 0.0f;
    if (pick >= 0) pval(pick, &w);
    a.out_tokens[r * (B + 1) + acc] = int32_t(pick);
    a.logprob[r * (B + 1) + acc] = float(log(double(w)) - log(wsum));
  }
}

size_t vf_align(size_t x) { return (x + 255) & ~size_t(255); }

VerifyWs vf_layout(void* base, int64_t R, int32_t B, size_t* total) {
  const size_t rows = size_t(R) * (B + 1);
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
  *total = off;
  return w;
}

}  // namespace

extern "C" size_t dspark_internal_ws_verify(int64_t R, int32_t B, int64_t V) {
  (void)V;
  size_t total = 0;
  vf_layout(nullptr, R, B, &total);
  return total;
}

extern "C" dspark_status dspark_verify(const void* tgt_logits, dspark_dtype dtype, int64_t R, int32_t B, int64_t V_t,
                                       int64_t ld, const int64_t* row_start, const int32_t* draft_tgt,
                                       const int32_t* n_draft, const dspark_qrecord* q, int64_t V_q,
                                       float temperature, float top_p, const uint64_t* vseed, const uint64_t* step,
                                       int32_t* out_tokens, int32_t* n_accepted, float* logprob, void* ws,
                                       size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype) && R >= 0 && B >= 1 && B <= 100 && V_t >= 1 && ld >= V_t);
  DS_REQUIRE(V_t <= int64_t(VD_MAXROUNDS) * VD_THREADS && R * (B + 1) <= 0x7FFFFFFF);
  DS_REQUIRE(tgt_logits && draft_tgt && n_draft && out_tokens && n_accepted && logprob && dev_status);
  DS_REQUIRE(ds_aligned(tgt_logits, ds_dtype_size(dtype)));
  DS_REQUIRE(temperature == temperature && top_p == top_p && top_p > 0.0f);
  const bool greedy = !(temperature > 0.0f);
  int q_dense = 0;
  if (!greedy) {
    DS_REQUIRE(vseed && step && q);
    if (q->z) {
      DS_REQUIRE(q->zmax && q->wsum && q->wcut && q->icut && q->ldz >= V_q && V_q >= 1);
      q_dense = 1;
    } else {
      DS_REQUIRE(q->ids && q->p && q->n && q->cap >= 1);
    }
  }
  if (R == 0) return DSPARK_OK;
  size_t need = 0;
  vf_layout(nullptr, R, B, &need);
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
  a.q_dense = q_dense;
  a.V_q = V_q;
  a.T = temperature;
  a.top_p = top_p;
  a.vseed = vseed;
  a.step = step;
  a.out_tokens = out_tokens;
  a.n_accepted = n_accepted;
  a.logprob = logprob;
  a.status = dev_status;
  a.ws = vf_layout(ws, R, B, &need);

  // 1. statistics of every needed target row
  rs::SampleArgs sa = {};
  sa.rows = tgt_logits;
  sa.V = V_t;
  sa.ld = ld;
  sa.row_start = row_start;
  sa.row_mul = 1;
  sa.B = B + 1;
  sa.C = rs::cluster_size_for(V_t, ds_dtype_size(dtype));
  DS_REQUIRE(sa.C > 0);
  sa.mult = 1.0f;
  sa.softcap = 0.0f;
  sa.T = greedy ? 1.0f : temperature;
  sa.top_p = greedy ? 1.0f : top_p;
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
  sa.amax_out = greedy ? a.ws.amax : nullptr;
  DS_CUDA_TRY(rs::sample_rows(sa, R * (B + 1), dtype == DSPARK_BF16, 0, stream));

  // 2. sequential acceptance tests, one thread per request
  verify_accept_kernel<<<unsigned((R + 127) / 128), 128, 0, stream>>>(a, R);
  DS_CUDA_TRY(cudaGetLastError());

  // 3. residual or bonus draws
  if (!greedy) {
    const int nrounds = int((V_t + VD_THREADS - 1) / VD_THREADS);
    const size_t smem = size_t(nrounds) * VD_WARPS * sizeof(double);
    static size_t configured[2] = {0, 0};
    const int di = dtype == DSPARK_BF16 ? 0 : 1;
    if (smem > configured[di]) {
      if (di == 0)
        DS_CUDA_TRY(cudaFuncSetAttribute(verify_draw_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
      else
        DS_CUDA_TRY(cudaFuncSetAttribute(verify_draw_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
      configured[di] = smem;
    }
    if (di == 0) verify_draw_kernel<__nv_bfloat16><<<unsigned(R), VD_THREADS, smem, stream>>>(a);
    else verify_draw_kernel<float><<<unsigned(R), VD_THREADS, smem, stream>>>(a);
    DS_CUDA_TRY(cudaGetLastError());
  }
  return DSPARK_OK;
}
