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
// One cluster of C CTAs per row (layout in rowsample.cuh); the row is read from HBM once and
// stays in registers through: the maximum of z = s / T, the nucleus (threshold rounds with the
// candidates sorted in the leader CTA; a 64-step bisection over (weight, index) keys when the
// candidates overflow the leader), the kept mass per (thread, segment), the cluster prefix that
// locates the CTA, segment and thread whose running sum crosses u * W_kept, and the walk over that
// thread's <= 8 elements.
#include <cfloat>

#include "host_common.h"
#include "rowsample.cuh"

namespace {

constexpr int SP_CAP = 4096;   // nucleus candidates sorted in the leader CTA



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

template <typename T, bool XFORM>
__global__ void __launch_bounds__(rs::THREADS, 1) sample_cluster_kernel(const rs::SampleArgs a) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr int SEGS = rs::SEGS;
  extern __shared__ __align__(16) uint8_t dsm[];
  double(*s_mass)[rs::THREADS] = reinterpret_cast<double(*)[rs::THREADS]>(dsm);
  uint64_t* s_keys = reinterpret_cast<uint64_t*>(dsm + sizeof(double) * SEGS * rs::THREADS);
  __shared__ rs::BlockScratch bs;
  __shared__ rs::ClusterRed cr;
  __shared__ uint32_t s_cnt;
  __shared__ int s_seg;
  __shared__ double s_tau, s_cut[2];

  cg::cluster_group cl = cg::this_cluster();
  const int C = a.C, crank = int(cl.block_rank());
  const int64_t row_id = blockIdx.x / C;
  const int64_t r = row_id / a.B, j = row_id % a.B;
  const int64_t prow = a.row_start ? a.row_start[r] + j : a.row_base + row_id * a.row_mul;
  if (a.n_draft && j > a.n_draft[r]) return;        // every CTA of the cluster leaves together
  const T* row = reinterpret_cast<const T*>(a.rows) + prow * a.ld;
  const rs::RowGeom g = rs::row_geom<T>(row, a.V, C, crank);
  const int tid = threadIdx.x;
  rs::cred_init(cr);
  if (tid == 0) s_cnt = 0;

  uint4 buf[rs::MAXV];
#pragma unroll
  for (int k = 0; k < rs::MAXV; ++k) {
    const int64_t v = g.vec_index(k);
    if (v >= 0) buf[k] = ds_ld_stream(reinterpret_cast<const uint4*>(row + g.head) + v);
  }
  const float rh = g.has_head() ? ds_load_elem<T>(row + tid) : 0.0f;
  const float rt = g.has_tail() ? ds_load_elem<T>(row + g.tail0 + tid) : 0.0f;
  const bool greedy = !(a.T > 0.0f);
  const float Tz = greedy ? 1.0f : a.T;
  auto zof = [&](float raw) { return ds_temper(sp_xform<XFORM>(raw, a.mult, a.softcap), Tz); };
  const int64_t ih = tid, it = g.tail0 + tid;

  int64_t pick = -1;
  float zmax = 0.0f, wcut = 0.0f;
  int64_t icut = -1;
  double wkept = 1.0;

  if (greedy) {
    // argmax, lowest index on ties
    unsigned long long best = 0;
#pragma unroll
    for (int k = 0; k < rs::MAXV; ++k) {
      const int64_t v = g.vec_index(k);
      if (v >= 0) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const unsigned long long kk = ds_key64(ds_canon_zero(zof(ds_vec_elem<T>(buf[k], e))), uint32_t(g.head + v * EPV + e));
          best = max(best, kk);
        }
      }
    }
    if (g.has_head()) best = max(best, (unsigned long long)ds_key64(ds_canon_zero(zof(rh)), uint32_t(ih)));
    if (g.has_tail()) best = max(best, (unsigned long long)ds_key64(ds_canon_zero(zof(rt)), uint32_t(it)));
    best = rs::cluster_max_u64(cl, cr, rs::block_max_u64(best, bs));
    zmax = ds_key64_val(best);
    wcut = 1.0f;
    icut = ds_key64_idx(best);
    if (crank == 0 && tid == 0) pick = icut;
  } else {
    // ---- maximum of z ----
    float tmax = -INFINITY;
#pragma unroll
    for (int k = 0; k < rs::MAXV; ++k)
      if (g.vec_index(k) >= 0) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) tmax = fmaxf(tmax, zof(ds_vec_elem<T>(buf[k], e)));
      }
    if (g.has_head()) tmax = fmaxf(tmax, zof(rh));
    if (g.has_tail()) tmax = fmaxf(tmax, zof(rt));
    zmax = float(rs::cluster_sum_d(cl, cr, double(rs::block_max(tmax, bs)), 1));
    if (!(zmax > -INFINITY && zmax < INFINITY)) {
      if (tid == 0 && crank == 0) {
        ds_set_error(a.status, DSPARK_ENONFINITE);
        if (a.out_idx) a.out_idx[row_id * a.out_mul + a.out_add] = -1;
        a.out_tgt[row_id * a.out_mul + a.out_add] = -1;
        if (a.prev_out) a.prev_out[r] = -1;
      }
      cl.sync();
      return;
    }
    auto wof = [&](float raw) { return ds_weight(__fsub_rn(zof(raw), zmax)); };

    // ---- top-p nucleus: the cut (wcut, icut) of the (weight desc, index asc) order ----
    if (a.top_p < 1.0f) {
      rs::FF acc{0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < rs::MAXV; ++k)
        if (g.vec_index(k) >= 0) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) rs::ff_add(acc, wof(ds_vec_elem<T>(buf[k], e)));
        }
      if (g.has_head()) rs::ff_add(acc, wof(rh));
      if (g.has_tail()) rs::ff_add(acc, wof(rt));
      const double wall = rs::cluster_sum_d(cl, cr, rs::block_sum(rs::ff_value(acc), bs));
      const double tp = double(a.top_p);
      for (int round = 0; round < 4; ++round) {
        const float tau = round == 0 ? ds_weight(-10.0f) : round == 1 ? ds_weight(-20.0f)
                        : round == 2 ? ds_weight(-40.0f) : FLT_MIN;
        rs::FF m{0.0f, 0.0f};
        double cnt = 0.0;
        auto visit = [&](float w) {
          if (w >= tau) {
            rs::ff_add(m, w);
            cnt += 1.0;
          }
        };
#pragma unroll
        for (int k = 0; k < rs::MAXV; ++k)
          if (g.vec_index(k) >= 0) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) visit(wof(ds_vec_elem<T>(buf[k], e)));
          }
        if (g.has_head()) visit(wof(rh));
        if (g.has_tail()) visit(wof(rt));
        const double mass = rs::cluster_sum_d(cl, cr, rs::block_sum(rs::ff_value(m), bs));
        const double ncand = rs::cluster_sum_d(cl, cr, rs::block_sum(cnt, bs));
        if (round < 3 && !(mass / wall > tp + 1e-12)) continue;
        if (ncand <= double(SP_CAP)) {
          // candidates (a prefix of the sorted order) sorted in the leader, walked in order
          uint32_t* lcnt = cl.map_shared_rank(&s_cnt, 0);
          uint64_t* lkeys = cl.map_shared_rank(s_keys, 0);
          auto push = [&](float w, int64_t i) {
            if (w >= tau) {
              const uint32_t slot = atomicAdd(lcnt, 1u);
              if (slot < SP_CAP) lkeys[slot] = ds_key64(w, uint32_t(i));
            }
          };
#pragma unroll
          for (int k = 0; k < rs::MAXV; ++k) {
            const int64_t v = g.vec_index(k);
            if (v >= 0) {
#pragma unroll
              for (int e = 0; e < EPV; ++e) push(wof(ds_vec_elem<T>(buf[k], e)), g.head + v * EPV + e);
            }
          }
          if (g.has_head()) push(wof(rh), ih);
          if (g.has_tail()) push(wof(rt), it);
          cl.sync();
          if (crank == 0) {
            const int n = int(min(s_cnt, uint32_t(SP_CAP)));
            int n2 = 1;
            while (n2 < n) n2 <<= 1;
            for (int i = n + tid; i < n2; i += blockDim.x) s_keys[i] = 0;
            __syncthreads();
            ds_block_sort_desc(s_keys, n2);
            if (tid == 0) {
              double cum = 0.0;
              s_cut[0] = 0.0;
              s_cut[1] = -1.0;
              for (int k = 0; k < n; ++k) {
                const float w = ds_key64_val(s_keys[k]);
                cum += double(w) / wall;
                if (cum > tp) {
                  s_cut[0] = double(w);
                  s_cut[1] = double(ds_key64_idx(s_keys[k]));
                  break;
                }
              }
              s_cnt = 0;
            }
          }
        } else {
          // bisection for the largest (weight, index) key whose upper set has mass > top_p
          unsigned long long res = 0;
          for (int b = 63; b >= 0; --b) {
            const unsigned long long cand = res | (1ull << b);
            rs::FF mm{0.0f, 0.0f};
            auto vis2 = [&](float w, int64_t i) {
              if ((unsigned long long)ds_key64(w, uint32_t(i)) >= cand) rs::ff_add(mm, w);
            };
#pragma unroll
            for (int k = 0; k < rs::MAXV; ++k) {
              const int64_t v = g.vec_index(k);
              if (v >= 0) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) vis2(wof(ds_vec_elem<T>(buf[k], e)), g.head + v * EPV + e);
              }
            }
            if (g.has_head()) vis2(wof(rh), ih);
            if (g.has_tail()) vis2(wof(rt), it);
            const double mb = rs::cluster_sum_d(cl, cr, rs::block_sum(rs::ff_value(mm), bs));
            if (mb / wall > tp) res = cand;
          }
          if (tid == 0) {
            s_cut[0] = double(ds_key64_val(res));
            s_cut[1] = double(ds_key64_idx(res));
          }
        }
        break;
      }
      wcut = float(rs::cluster_sum_d(cl, cr, crank == 0 ? s_cut[0] : 0.0));
      icut = int64_t(rs::cluster_sum_d(cl, cr, crank == 0 ? s_cut[1] : 0.0));
    }

    // ---- kept mass per (thread, segment): segment 0 head, 1 + k round k, SEGS - 1 tail ----
    double mine = 0.0;
    unsigned long long lastk = 0;
    {
      double mh = 0.0;
      if (g.has_head()) {
        const float w = wof(rh);
        if (sp_keep(w, ih, wcut, icut)) {
          mh = double(w);
          lastk = max(lastk, (unsigned long long)(ih + 1));
        }
      }
      s_mass[0][tid] = mh;
      mine += mh;
    }
#pragma unroll
    for (int k = 0; k < rs::MAXV; ++k) {
      const int64_t v = g.vec_index(k);
      rs::FF m{0.0f, 0.0f};
      if (v >= 0) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          const float w = wof(ds_vec_elem<T>(buf[k], e));
          const int64_t i = g.head + v * EPV + e;
          if (sp_keep(w, i, wcut, icut)) {
            rs::ff_add(m, w);
            lastk = max(lastk, (unsigned long long)(i + 1));
          }
        }
      }
      s_mass[1 + k][tid] = rs::ff_value(m);
      mine += s_mass[1 + k][tid];
    }
    {
      double mt = 0.0;
      if (g.has_tail()) {
        const float w = wof(rt);
        if (sp_keep(w, it, wcut, icut)) {
          mt = double(w);
          lastk = max(lastk, (unsigned long long)(it + 1));
        }
      }
      s_mass[SEGS - 1][tid] = mt;
      mine += mt;
    }
    const double ctot = rs::block_sum(mine, bs);
    double wtot = 0.0;
    const double cpre = rs::cluster_sum_d(cl, cr, ctot, 2, &wtot);
    const int64_t last_kept = int64_t(rs::cluster_max_u64(cl, cr, rs::block_max_u64(lastk, bs))) - 1;
    wkept = wtot;
    if (a.amax_out) {
      // argmax of z (lowest index on ties), for greedy verification
      unsigned long long best = 0;
#pragma unroll
      for (int k = 0; k < rs::MAXV; ++k) {
        const int64_t v = g.vec_index(k);
        if (v >= 0) {
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            best = max(best, (unsigned long long)ds_key64(ds_canon_zero(zof(ds_vec_elem<T>(buf[k], e))), uint32_t(g.head + v * EPV + e)));
        }
      }
      if (g.has_head()) best = max(best, (unsigned long long)ds_key64(ds_canon_zero(zof(rh)), uint32_t(ih)));
      if (g.has_tail()) best = max(best, (unsigned long long)ds_key64(ds_canon_zero(zof(rt)), uint32_t(it)));
      best = rs::cluster_max_u64(cl, cr, rs::block_max_u64(best, bs));
      if (crank == 0 && tid == 0) a.amax_out[row_id] = int32_t(ds_key64_idx(best));
    }
    if (a.probe_w) {
      const int64_t x = (a.probe_tgt && j < a.n_draft[r]) ? int64_t(a.probe_tgt[r * (a.B - 1) + j]) : -1;
      if (crank == 0 && tid == 0 && (x < 0 || x >= a.V)) a.probe_w[row_id] = 0.0f;
      if (x >= 0 && x < a.V) {
        auto probe = [&](float raw, int64_t i) {
          if (i == x) {
            const float w = wof(raw);
            a.probe_w[row_id] = sp_keep(w, i, wcut, icut) ? w : 0.0f;
          }
        };
        if (g.has_head()) probe(rh, ih);
        if (g.has_tail()) probe(rt, it);
#pragma unroll
        for (int k = 0; k < rs::MAXV; ++k) {
          const int64_t v = g.vec_index(k);
          if (v >= 0 && x >= g.head + v * EPV && x < g.head + (v + 1) * EPV) {
#pragma unroll
            for (int e = 0; e < EPV; ++e) probe(ds_vec_elem<T>(buf[k], e), g.head + v * EPV + e);
          }
        }
      }
    }
    const double u = a.no_draw ? 2.0 : ds_uniform(a.seed[r], a.step[r], uint32_t(a.position >= 0 ? a.position : int32_t(j)),
                                DS_PURPOSE_DRAFT);
    const double target = u * wtot;
    if (!a.no_draw && target >= cpre && target < cpre + ctot) {
      // this CTA holds the crossing: find the segment, then the thread, then the element
      const int warp = tid >> 5, lane = tid & 31;
      if (warp < SEGS) {
        double sacc = 0.0;
        for (int i = lane; i < rs::THREADS; i += 32) sacc += s_mass[warp][i];
        sacc = ds_warp_sum(sacc);
        if (lane == 0) bs.seg[warp] = sacc;
      }
      __syncthreads();
      if (tid == 0) {
        double acc = cpre;
        int sfound = -1;
        double tau = 0.0;
        int slast = -1;
        for (int s = 0; s < SEGS; ++s) {
          if (bs.seg[s] > 0.0) slast = s;
          const double nxt = acc + bs.seg[s];
          if (sfound < 0 && target < nxt && bs.seg[s] > 0.0) {
            sfound = s;
            tau = target - acc;
          }
          acc = nxt;
        }
        if (sfound < 0) {
          sfound = slast;
          tau = INFINITY;
        }
        s_seg = sfound;
        s_tau = tau;
      }
      __syncthreads();
      const int seg = s_seg;
      const double tau = s_tau;
      // inclusive / exclusive running sums over threads with excl[t+1] == incl[t] exactly
      const double mv = (seg >= 0) ? s_mass[seg][tid] : 0.0;
      double incl = mv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
      }
      __syncthreads();
      if (lane == 31) bs.d[warp] = incl;
      __syncthreads();
      double before = 0.0;
      for (int w = 0; w < warp; ++w) before += bs.d[w];
      const double prev_incl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
      const double ex = before + (lane > 0 ? prev_incl : 0.0);
      const double in = before + incl;
      bool last_thread_with_mass = false;
      {
        // the thread that holds the segment's last positive mass takes the rounding remainder
        const unsigned ball = __ballot_sync(0xFFFFFFFFu, mv > 0.0);
        __syncthreads();
        if (lane == 0) bs.u[warp] = ball;
        __syncthreads();
        int lw = -1;
        for (int w = rs::WARPS - 1; w >= 0; --w)
          if (bs.u[w]) {
            lw = w;
            break;
          }
        last_thread_with_mass = (lw == warp) && (mv > 0.0) && (31 - __clz(unsigned(bs.u[lw])) == lane);
      }
      if (seg >= 0 && mv > 0.0 && ((tau >= ex && tau < in) || (last_thread_with_mass && tau >= in))) {
        double run = ex;
        int64_t lastmine = -1;
        auto walk = [&](float w, int64_t i) {
          if (pick < 0 && sp_keep(w, i, wcut, icut)) {
            run += double(w);
            lastmine = i;
            if (run > tau) pick = i;
          }
        };
        if (seg == 0) {
          walk(wof(rh), ih);
        } else if (seg == SEGS - 1) {
          walk(wof(rt), it);
        } else {
          const int k = seg - 1;
          const int64_t v = g.vec_index(k);
#pragma unroll
          for (int kk = 0; kk < rs::MAXV; ++kk)
            if (kk == k) {
#pragma unroll
              for (int e = 0; e < EPV; ++e) walk(wof(ds_vec_elem<T>(buf[kk], e)), g.head + v * EPV + e);
            }
        }
        if (pick < 0) pick = lastmine;
      }
    } else if (!a.no_draw && crank == C - 1 && tid == 0 && !(target < wtot)) {
      pick = last_kept;      // rounding left the target at the very end
    }
  }

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
      const int64_t qr = row_id * a.q_row_mul + a.q_row_add;
      a.q.n[qr] = 1;
      a.q.ids[qr * a.q.cap] = int32_t(tgt);
      a.q.p[qr * a.q.cap] = 1.0f;
    }
  }

  // ---- proposal record ----
  const int64_t qrow = row_id * a.q_row_mul + a.q_row_add;
  if (a.q_mode == 2) {
    if (crank == 0 && tid == 0) {
      a.q.zmax[qrow] = zmax;
      a.q.wsum[qrow] = greedy ? 1.0 : wkept;
      a.q.wcut[qrow] = wcut;
      a.q.icut[qrow] = int32_t(icut);
    }
    if (a.write_z) {
      float* zr = a.q.z + qrow * a.q.ldz;
#pragma unroll
      for (int k = 0; k < rs::MAXV; ++k) {
        const int64_t v = g.vec_index(k);
        if (v >= 0) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) zr[g.head + v * EPV + e] = zof(ds_vec_elem<T>(buf[k], e));
        }
      }
      if (g.has_head()) zr[ih] = zof(rh);
      if (g.has_tail()) zr[it] = zof(rt);
    }
  } else if (a.q_mode == 1 && !greedy) {
    // sparse record: kept tokens in ascending index order with q = w / W_kept
    auto wof = [&](float raw) { return ds_weight(__fsub_rn(zof(raw), zmax)); };
    double cnt_seg[rs::SEGS];
    double mine = 0.0;
    cnt_seg[0] = (g.has_head() && sp_keep(wof(rh), ih, wcut, icut)) ? 1.0 : 0.0;
#pragma unroll
    for (int k = 0; k < rs::MAXV; ++k) {
      double c = 0.0;
      const int64_t v = g.vec_index(k);
      if (v >= 0) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) c += sp_keep(wof(ds_vec_elem<T>(buf[k], e)), g.head + v * EPV + e, wcut, icut) ? 1.0 : 0.0;
      }
      cnt_seg[1 + k] = c;
    }
    cnt_seg[SEGS - 1] = (g.has_tail() && sp_keep(wof(rt), it, wcut, icut)) ? 1.0 : 0.0;
#pragma unroll
    for (int s = 0; s < SEGS; ++s) mine += cnt_seg[s];
    const double ccnt = rs::block_sum(mine, bs);
    double ntot = 0.0;
    const double cbase = rs::cluster_sum_d(cl, cr, ccnt, 2, &ntot);
    if (ntot > double(a.q.cap)) {
      if (crank == 0 && tid == 0) {
        a.q.n[qrow] = -1;
        ds_set_error(a.status, DSPARK_EINVAL);
      }
    } else {
      if (crank == 0 && tid == 0) a.q.n[qrow] = int32_t(ntot);
      double base = cbase;
#pragma unroll
      for (int s = 0; s < SEGS; ++s) {
        double segtot = 0.0;
        double pos = base + rs::block_exclusive_scan(cnt_seg[s], &segtot, bs);
        auto emit = [&](float w, int64_t i) {
          if (sp_keep(w, i, wcut, icut)) {
            int64_t tg = i;
            if (a.d2t) tg = i + a.d2t[i];
            const int64_t o = qrow * a.q.cap + int64_t(pos);
            a.q.ids[o] = int32_t(tg);
            a.q.p[o] = float(double(w) / wkept);
            pos += 1.0;
          }
        };
        if (s == 0) {
          if (g.has_head()) emit(wof(rh), ih);
        } else if (s == SEGS - 1) {
          if (g.has_tail()) emit(wof(rt), it);
        } else {
          const int64_t v = g.vec_index(s - 1);
          if (v >= 0) {
#pragma unroll
            for (int kk = 0; kk < rs::MAXV; ++kk)
              if (kk == s - 1) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) emit(wof(ds_vec_elem<T>(buf[kk], e)), g.head + v * EPV + e);
              }
          }
        }
        base += segtot;
      }
    }
  }
  cl.sync();
}

template <typename T, bool XFORM>
cudaError_t sp_launch(const rs::SampleArgs& a, int64_t rows, cudaStream_t stream) {
  auto kern = sample_cluster_kernel<T, XFORM>;
  const size_t smem = sizeof(double) * rs::SEGS * rs::THREADS + sizeof(uint64_t) * SP_CAP;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(rows * a.C), 1, 1);
  cfg.blockDim = dim3(rs::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(a.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

// Shared with the dense walk: one launch of the row sampler over `rows` rows.
cudaError_t rs::sample_rows(const rs::SampleArgs& a, int64_t rows, int is_bf16, int xform, cudaStream_t stream) {
  if (is_bf16) return xform ? sp_launch<__nv_bfloat16, true>(a, rows, stream) : sp_launch<__nv_bfloat16, false>(a, rows, stream);
  return xform ? sp_launch<float, true>(a, rows, stream) : sp_launch<float, false>(a, rows, stream);
}

extern "C" size_t dspark_internal_ws_sample(int64_t, int32_t, int64_t) { return 0; }

extern "C" dspark_status dspark_sample(const void* logits, dspark_dtype dtype, int64_t R, int32_t B, int64_t V_d,
                                       int64_t ld, const int64_t* row_start, const int64_t* d2t, int64_t V_t,
                                       float mult, float softcap, float temperature, float top_p,
                                       const uint64_t* seed, const uint64_t* step, int32_t* out_tgt,
                                       int32_t* out_idx, const dspark_qrecord* q, void* ws, size_t ws_bytes,
                                       int32_t* dev_status, dspark_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  DS_REQUIRE(ds_dtype_ok(dtype));
  DS_REQUIRE(R >= 0 && B >= 1 && V_d >= 1 && ld >= V_d && V_d <= 0x7FFFFFFF && R * B <= 0x7FFFFFFF);
  DS_REQUIRE(logits && out_tgt && dev_status && ds_aligned(logits, ds_dtype_size(dtype)));
  DS_REQUIRE(temperature == temperature && top_p == top_p && top_p > 0.0f);
  DS_REQUIRE(mult == mult && softcap == softcap && softcap >= 0.0f);
  if (temperature > 0.0f) DS_REQUIRE(seed && step);
  if (d2t) DS_REQUIRE(V_t >= 1);
  rs::SampleArgs a = {};
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
  const int xform = (mult != 1.0f) || (softcap > 0.0f);
  const cudaError_t e = rs::sample_rows(a, R * B, dtype == DSPARK_BF16, xform, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}
