// topk.cu - row transform + exact Top-K' + d2t map (dspark_topk).
//
// Method: openvino.genai PR #4847 ("Add DSpark and DFlash v2 drafts and sampled drafting to
// DFlash speculative decoding"), Change > Markov heads (the scorer takes the K best backbone
// candidates of every block position) and the block-sampler commit (rows are the backbone
// logits times the output multiplier, soft-capped); optimum-intel PR #2099 ("... DSpark drafts
// with a pruned vocabulary"), Markov head (top_k = min(64, draft_vocab_size)) and Pruned
// draft vocabulary (target id i + d2t[i]). optimum-intel PR #2098 runs this selection with the
// OpenVINO GPU plugin's radix TopK; this kernel is a different, exact design for sm_103a.
//
// Design: persistent CTAs (two per SM) each take whole rows, streaming a row in chunks of up to
// 42 KB through a 2-stage shared-memory ring filled by bulk asynchronous copies (cp.async.bulk +
// mbarrier transaction counts); the ring runs on across rows, so HBM keeps streaming while a
// chunk is screened. The logits are read once and no other CTA is involved in a row.
// Per row the CTA keeps the exact top-K' keys seen so far (64-bit keys: value, then lower index
// first), sorted, in shared memory, and a bound B that K' elements already seen reach:
//  1. Chunk 0: each warp takes the m-th largest of its lanes' maxima (m = ceil(K'/8), warp REDUX
//     rounds); every lane maximum is a distinct element, so 8 warps x m >= K' elements are >= the
//     minimum T over the warps. Elements >= T survive (a few K'); B = T.
//  2. Later chunks: every element of the chunk comes after the K' elements behind B, so an equal
//     value loses on the index and only values strictly above B can enter: one packed compare
//     of each vector's maximum, survivors rare and never a flood of ties.
//  3. Screening is one sweep without side effects that marks the vectors holding a survivor;
//     the marked vectors are then taken apart by the whole warp (8-bit masks from packed
//     compares, one survivor per lane per pass, one shared-memory atomic per pass).
//  4. Once 2K' survivors have gathered (and at the row's end) they merge into the running list:
//     a key's position is the number of keys above it in both lists; the list keeps its first
//     K' entries and B rises to its K'-th value.
//  5. A chunk whose survivors overflow the buffer (ties in chunk 0, or a rising row) is first cut
//     to its own exact top-K' by a bisection over its keys in shared memory.
// After the last chunk the list is the row's top-K', written in order with the d2t map.
#include <type_traits>

#include "dspark_common.cuh"
#include "host_common.h"

namespace {

constexpr int TK_THREADS = 256;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_STAGES = 2;
constexpr int TK_STAGE_VEC = 2688;      // 16-byte vectors per chunk (42 KB)
constexpr int TK_NEW_CAP = 1024;        // survivors of one chunk before the exact cut
constexpr int TK_KMAX = 64;
constexpr int TK_ROUNDS = (TK_STAGE_VEC + TK_THREADS - 1) / TK_THREADS;   // vectors per lane per chunk

struct TopkArgs {
  const void* logits;
  int64_t V, ld;
  const int64_t* row_start;
  int32_t B, Kp;
  int32_t rows;
  float mult, softcap;
  const int64_t* d2t;
  int64_t V_t;
  int32_t* cand_draft;
  int32_t* cand_tgt;
  float* cand_val;
  int32_t* status;
};

DS_DEV __nv_bfloat162 tk_b2(uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); }

template <bool XFORM>
DS_DEV float tk_xform(float x, float mult, float softcap) {
  if (XFORM) {
    if (mult != 1.0f) x = __fmul_rn(x, mult);
    if (softcap > 0.0f) x = __fmul_rn(softcap, tanhf(__fdiv_rn(x, softcap)));
  }
  return x;
}

// Block-wide sum of a per-thread count.
DS_DEV uint32_t tk_block_sum(uint32_t c, uint32_t* s_red) {
  c = __reduce_add_sync(0xFFFFFFFFu, c);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = c;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int w = 0; w < TK_WARPS; ++w) t += s_red[w];
  return t;
}

// Geometry of one row: scalar head up to 16-byte alignment, vectors, scalar tail, chunks.
struct TkRow {
  const void* row;
  int64_t head, nvec, tail0;
  int nch;
};

template <typename T>
DS_DEV TkRow tk_row(const TopkArgs& a, uint32_t row_id) {
  constexpr int EPV = 16 / sizeof(T);
  int64_t prow = row_id;
  if (a.row_start) {
    const uint32_t r = row_id / uint32_t(a.B);
    prow = a.row_start[r] + (row_id - r * uint32_t(a.B));
  }
  TkRow g;
  const T* row = reinterpret_cast<const T*>(a.logits) + prow * a.ld;
  g.row = row;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  g.head = int64_t(((16u - (addr & 15u)) & 15u) / sizeof(T));
  if (g.head > a.V) g.head = a.V;
  g.nvec = (a.V - g.head) / EPV;
  g.tail0 = g.head + g.nvec * EPV;
  g.nch = g.nvec > 0 ? int((g.nvec + TK_STAGE_VEC - 1) / TK_STAGE_VEC) : 1;
  return g;
}

// Writes candidate `rank` of a row: draft index, target id (d2t, range-checked) and value.
DS_DEV void tk_emit(const TopkArgs& a, uint32_t row_id, int rank, uint64_t k64) {
  const int64_t o = int64_t(row_id) * a.Kp + rank;
  const uint32_t idx = ds_key64_idx(k64);
  int64_t tgt = idx;
  if (a.d2t) {
    tgt = int64_t(idx) + a.d2t[idx];
    if (tgt < 0 || tgt >= a.V_t) {
      ds_set_error(a.status, DSPARK_ERANGE);
      tgt = -1;
    }
  }
  a.cand_draft[o] = int32_t(idx);
  a.cand_tgt[o] = int32_t(tgt);
  a.cand_val[o] = ds_key64_val(k64);
}

// The chunk's own top-K' among the elements that pass the screen (x > thr when `strict`, else
// x >= thr): the K'-th largest passing key by bisection over the 64 key bits (chunk read from
// shared memory), then every passing key at or above it (exactly K' keys) into s_new[base...].
// Only for a chunk whose survivors overflow the buffer. Returns base + the keys written.
template <typename T, bool XFORM>
__device__ __noinline__ uint32_t tk_chunk_exact(const TopkArgs& a, const uint4* sv, int nv, int64_t e0,
                                                int64_t iextra, float xextra, float thr, bool strict,
                                                uint64_t* s_new, uint32_t base, uint32_t* s_red, uint32_t* s_n) {
  constexpr int EPV = 16 / sizeof(T);
  auto pass = [&](float x) { return strict ? (x > thr) : (x >= thr); };
  uint64_t kres = 0;
  for (int b = 63; b >= 0; --b) {
    const uint64_t cand = kres | (1ull << b);
    uint32_t c = 0;
    for (int e = threadIdx.x; e < nv; e += TK_THREADS) {
      const uint4 w = sv[e];
#pragma unroll
      for (int x = 0; x < EPV; ++x) {
        const float v = ds_canon_zero(tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap));
        c += (pass(v) && ds_key64(v, uint32_t(e0 + int64_t(e) * EPV + x)) >= cand) ? 1u : 0u;
      }
    }
    if (iextra >= 0) {
      const float v = ds_canon_zero(xextra);
      c += (pass(v) && ds_key64(v, uint32_t(iextra)) >= cand) ? 1u : 0u;
    }
    if (tk_block_sum(c, s_red) >= uint32_t(a.Kp)) kres = cand;
  }
  __syncthreads();
  if (threadIdx.x == 0) *s_n = base;
  __syncthreads();
  for (int e = threadIdx.x; e < nv; e += TK_THREADS) {
    const uint4 w = sv[e];
#pragma unroll
    for (int x = 0; x < EPV; ++x) {
      const float v = ds_canon_zero(tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap));
      const uint64_t k = ds_key64(v, uint32_t(e0 + int64_t(e) * EPV + x));
      if (pass(v) && k >= kres) {
        const uint32_t slot = atomicAdd(s_n, 1u);
        if (slot < TK_NEW_CAP) s_new[slot] = k;
      }
    }
  }
  if (iextra >= 0) {
    const float v = ds_canon_zero(xextra);
    const uint64_t k = ds_key64(v, uint32_t(iextra));
    if (pass(v) && k >= kres) {
      const uint32_t slot = atomicAdd(s_n, 1u);
      if (slot < TK_NEW_CAP) s_new[slot] = k;
    }
  }
  __syncthreads();
  return min(*s_n, uint32_t(TK_NEW_CAP));
}

template <typename T, bool XFORM>
__global__ void __launch_bounds__(TK_THREADS, 2) topk_row_kernel(const TopkArgs a) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr bool PACKED = std::is_same<T, __nv_bfloat16>::value && !XFORM;
  constexpr int PRODUCER = TK_THREADS - 32;               // lane 0 of the last warp issues the copies
  extern __shared__ __align__(128) uint8_t tk_dyn[];      // TK_STAGES x TK_STAGE_VEC x 16 bytes
  __shared__ uint64_t s_full[TK_STAGES];
  __shared__ uint64_t s_top[2][TK_KMAX];                  // running top-K' keys, sorted
  __shared__ uint64_t s_new[TK_NEW_CAP];                  // survivors not yet merged
  __shared__ uint32_t s_red[TK_WARPS];
  __shared__ float s_wthr[TK_WARPS];
  __shared__ uint32_t s_n;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint4* stages = reinterpret_cast<const uint4*>(tk_dyn);

  // producer: the CTA's (row, chunk) sequence, TK_STAGES items ahead of the consumer
  int p_ri = 0, p_c = 0, issued = 0;
  auto issue_next = [&]() {
    const int64_t row_id = int64_t(blockIdx.x) + int64_t(p_ri) * gridDim.x;
    if (row_id >= a.rows) return;
    const TkRow g = tk_row<T>(a, uint32_t(row_id));
    const int64_t v0 = int64_t(p_c) * TK_STAGE_VEC, v1 = min(g.nvec, v0 + TK_STAGE_VEC);
    const uint32_t bytes = v1 > v0 ? uint32_t((v1 - v0) * 16) : 0u;
    const int s = issued % TK_STAGES;
    ds_mbar_arrive_expect_tx(&s_full[s], bytes);
    if (bytes)
      ds_bulk_g2s(tk_dyn + size_t(s) * TK_STAGE_VEC * 16,
                  reinterpret_cast<const uint8_t*>(g.row) + g.head * int64_t(sizeof(T)) + v0 * 16, bytes, &s_full[s]);
    ++issued;
    if (++p_c == g.nch) {
      p_c = 0;
      ++p_ri;
    }
  };

  if (tid == PRODUCER) {
    for (int s = 0; s < TK_STAGES; ++s) ds_mbar_init(&s_full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int s = 0; s < TK_STAGES; ++s) issue_next();
  }
  if (tid == 0) s_n = 0;
  __syncthreads();

  const int m = (a.Kp + TK_WARPS - 1) / TK_WARPS;
  int n = 0;                                               // items consumed
  for (int64_t row_id = blockIdx.x; row_id < a.rows; row_id += gridDim.x) {
    const TkRow g = tk_row<T>(a, uint32_t(row_id));
    const T* row = reinterpret_cast<const T*>(g.row);
    int cur = 0, ntop = 0;
    float bound = -INFINITY;                               // every later element must beat it strictly
    for (int c = 0; c < g.nch; ++c, ++n) {
      const int s = n % TK_STAGES;
      const int64_t v0 = int64_t(c) * TK_STAGE_VEC, v1 = min(g.nvec, v0 + TK_STAGE_VEC);
      const int nv = v1 > v0 ? int(v1 - v0) : 0;
      const int64_t e0 = g.head + v0 * EPV;                 // index of the chunk's first vector element
      const uint4* sv = stages + size_t(s) * TK_STAGE_VEC;

      // scalar head (chunk 0) and tail (last chunk) elements, loaded directly
      int64_t iextra = -1;
      if (c == 0 && tid < g.head) iextra = tid;
      if (c == g.nch - 1 && tid >= 8 && tid - 8 < a.V - g.tail0) iextra = g.tail0 + (tid - 8);
      const float xextra = iextra >= 0 ? tk_xform<XFORM>(ds_load_elem<T>(row + iextra), a.mult, a.softcap) : -INFINITY;

      bool ok = ds_mbar_wait(&s_full[s], uint32_t(n / TK_STAGES) & 1u, DS_WAIT_LIMIT);
      ok = __syncthreads_and(ok) != 0;
      if (!ok) {
        // a copy never completed: report it, let the copies in flight land (bounded), stop
        if (tid == PRODUCER) {
          ds_set_error(a.status, DSPARK_ETIMEOUT);
          for (int j = n; j < issued; ++j)
            (void)ds_mbar_wait(&s_full[j % TK_STAGES], uint32_t(j / TK_STAGES) & 1u, DS_WAIT_LIMIT);
        }
        return;
      }
      const uint32_t nbase = s_n;                          // survivors of earlier chunks not merged yet

      // ---- screen: one sweep without side effects marks the vectors holding a survivor (all
      // loads in flight together), then the marked vectors are taken apart ----
      float thr;
      bool strict;
      uint32_t hits = 0;
      if (c == 0) {
        // bound from the chunk itself: the m-th largest lane maximum of every warp
        strict = false;
        float tmax = xextra;
        float vmax[TK_ROUNDS];
        __nv_bfloat162 vmax2[TK_ROUNDS];
        if constexpr (PACKED) {
          __nv_bfloat162 acc = __float2bfloat162_rn(-INFINITY);
#pragma unroll
          for (int k = 0; k < TK_ROUNDS; ++k) {
            const int e = tid + k * TK_THREADS;
            vmax2[k] = __float2bfloat162_rn(-INFINITY);
            if (e < nv) {
              const uint4 w = sv[e];
              vmax2[k] = __hmax2(__hmax2(tk_b2(w.x), tk_b2(w.y)), __hmax2(tk_b2(w.z), tk_b2(w.w)));
              acc = __hmax2(acc, vmax2[k]);
            }
          }
          tmax = fmaxf(tmax, fmaxf(__low2float(acc), __high2float(acc)));
        } else {
#pragma unroll
          for (int k = 0; k < TK_ROUNDS; ++k) {
            const int e = tid + k * TK_THREADS;
            vmax[k] = -INFINITY;
            if (e < nv) {
              const uint4 w = sv[e];
#pragma unroll
              for (int x = 0; x < EPV; ++x)
                vmax[k] = fmaxf(vmax[k], tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap));
              tmax = fmaxf(tmax, vmax[k]);
            }
          }
        }
        uint32_t key = ds_key32(ds_canon_zero(tmax)), kth = 0;
#pragma unroll
        for (int t = 0; t < (TK_KMAX + TK_WARPS - 1) / TK_WARPS; ++t) {
          if (t < m) {
            kth = __reduce_max_sync(0xFFFFFFFFu, key);
            const unsigned who = __ballot_sync(0xFFFFFFFFu, key == kth);
            if (lane == __ffs(who) - 1) key = 0;
          }
        }
        if (lane == 0) s_wthr[warp] = (kth <= ds_key32(-INFINITY)) ? -INFINITY : ds_key32_to_float(kth);
        __syncthreads();
        thr = s_wthr[0];
#pragma unroll
        for (int w = 1; w < TK_WARPS; ++w) thr = fminf(thr, s_wthr[w]);
        const __nv_bfloat162 thr2 = __float2bfloat162_rn(thr);   // exact for bf16 rows: an element value
#pragma unroll
        for (int k = 0; k < TK_ROUNDS; ++k) {
          bool any;
          if constexpr (PACKED) any = (tid + k * TK_THREADS < nv) && __hge2_mask(vmax2[k], thr2) != 0u;
          else any = (tid + k * TK_THREADS < nv) && vmax[k] >= thr;
          hits |= any ? (1u << k) : 0u;
        }
      } else {
        // bound from the elements before the chunk: only values strictly above it can enter
        strict = true;
        thr = bound;
        const __nv_bfloat162 thr2 = __float2bfloat162_rn(thr);   // exact for bf16 rows: an element value
#pragma unroll
        for (int k = 0; k < TK_ROUNDS; ++k) {
          const int e = tid + k * TK_THREADS;
          if (e < nv) {
            const uint4 w = sv[e];
            bool any;
            if constexpr (PACKED) {
              const __nv_bfloat162 mx = __hmax2(__hmax2(tk_b2(w.x), tk_b2(w.y)), __hmax2(tk_b2(w.z), tk_b2(w.w)));
              any = __hgt2_mask(mx, thr2) != 0u;
            } else {
              float mx = -INFINITY;
#pragma unroll
              for (int x = 0; x < EPV; ++x) mx = fmaxf(mx, tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap));
              any = mx > thr;
            }
            hits |= any ? (1u << k) : 0u;
          }
        }
      }
      // the marked vectors, one per lane at a time: 8-bit survivor masks drained by the whole warp
      // (one survivor per lane per pass, one shared-memory atomic per pass)
      {
        const unsigned below = (1u << lane) - 1u;
        const __nv_bfloat162 thr2 = __float2bfloat162_rn(thr);
        while (__any_sync(0xFFFFFFFFu, hits != 0u)) {
          uint32_t m8 = 0;
          int e = 0;
          if (hits) {
            e = tid + (__ffs(hits) - 1) * TK_THREADS;
            hits &= hits - 1u;
            const uint4 w = sv[e];
            if constexpr (PACKED) {
              uint32_t c0, c1, c2, c3;
              if (strict) {
                c0 = __hgt2_mask(tk_b2(w.x), thr2), c1 = __hgt2_mask(tk_b2(w.y), thr2);
                c2 = __hgt2_mask(tk_b2(w.z), thr2), c3 = __hgt2_mask(tk_b2(w.w), thr2);
              } else {
                c0 = __hge2_mask(tk_b2(w.x), thr2), c1 = __hge2_mask(tk_b2(w.y), thr2);
                c2 = __hge2_mask(tk_b2(w.z), thr2), c3 = __hge2_mask(tk_b2(w.w), thr2);
              }
              // bytes [e0 e1 e2 e3] and [e4 e5 e6 e7] (0x00 / 0xFF), then one bit per element
              const uint32_t w01 = __byte_perm(c0, c1, 0x6420), w23 = __byte_perm(c2, c3, 0x6420);
              uint32_t f = (w01 & 0x08040201u) | (w23 & 0x80402010u);
              f |= f >> 16;
              f |= f >> 8;
              m8 = f & 0xFFu;
            } else {
#pragma unroll
              for (int x = 0; x < EPV; ++x) {
                const float v = tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap);
                m8 |= (strict ? v > thr : v >= thr) ? (1u << x) : 0u;
              }
            }
          }
          while (true) {
            const unsigned act = __ballot_sync(0xFFFFFFFFu, m8 != 0u);
            if (act == 0u) break;
            uint32_t slot = 0;
            const int leader = __ffs(act) - 1;
            if (lane == leader) slot = atomicAdd(&s_n, uint32_t(__popc(act)));
            slot = __shfl_sync(0xFFFFFFFFu, slot, leader) + uint32_t(__popc(act & below));
            if (m8 != 0u) {
              const int x = __ffs(m8) - 1;
              m8 &= m8 - 1u;
              const float v = tk_xform<XFORM>(ds_load_elem<T>(reinterpret_cast<const T*>(sv + e) + x), a.mult, a.softcap);
              if (slot < TK_NEW_CAP) s_new[slot] = ds_key64(ds_canon_zero(v), uint32_t(e0 + int64_t(e) * EPV + x));
            }
          }
        }
      }
      if (iextra >= 0 && (strict ? xextra > thr : xextra >= thr)) {
        const uint32_t slot = atomicAdd(&s_n, 1u);
        if (slot < TK_NEW_CAP) s_new[slot] = ds_key64(ds_canon_zero(xextra), uint32_t(iextra));
      }
      if (c == 0) bound = thr;      // K' elements of chunk 0 are >= thr and precede every later one
      __syncthreads();
      uint32_t N = s_n;
      if (N > uint32_t(TK_NEW_CAP))
        N = tk_chunk_exact<T, XFORM>(a, sv, nv, e0, iextra, xextra, thr, strict, s_new, nbase, s_red, &s_n);
      // the stage is free: refill it with the item TK_STAGES ahead
      if (tid == PRODUCER) {
        ds_fence_proxy_async_smem();
        issue_next();
      }

      // ---- merge the survivors into the running list once enough have gathered (and at the end
      // of the row): a key's position is the number of keys above it in both lists (binary
      // search in the sorted list, a count over the new keys) ----
      if (N >= uint32_t(2 * a.Kp) || c == g.nch - 1) {
        const uint64_t* old = s_top[cur];
        uint64_t* out = s_top[cur ^ 1];
        const uint32_t nt = uint32_t(ntop);
        for (uint32_t t = tid; t < N + nt; t += TK_THREADS) {
          const bool is_new = t < N;
          const uint64_t k = is_new ? s_new[t] : old[t - N];
          uint32_t pos = 0;
          if (is_new) {
            uint32_t lo = 0, hi = nt;                      // first old key below k
            while (lo < hi) {
              const uint32_t mid = (lo + hi) >> 1;
              if (old[mid] > k) lo = mid + 1;
              else hi = mid;
            }
            pos = lo;
          } else {
            pos = t - N;
          }
          uint32_t u = 0;
          for (; u + 8 <= N; u += 8) {
            uint32_t cnt = 0;
#pragma unroll
            for (int r = 0; r < 8; ++r) cnt += (s_new[u + r] > k) ? 1u : 0u;
            pos += cnt;
          }
          for (; u < N; ++u) pos += (s_new[u] > k) ? 1u : 0u;
          if (pos < uint32_t(a.Kp)) out[pos] = k;
        }
        __syncthreads();
        cur ^= 1;
        ntop = int(min(uint32_t(ntop) + N, uint32_t(a.Kp)));
        if (ntop == a.Kp) bound = fmaxf(bound, ds_key64_val(s_top[cur][a.Kp - 1]));
        if (tid == 0) s_n = 0;
      }
    }
    if (tid < a.Kp) {
      if (tid < ntop) {
        tk_emit(a, uint32_t(row_id), tid, s_top[cur][tid]);
      } else {                                             // unreachable: every row holds >= K' elements
        ds_set_error(a.status, DSPARK_EINVAL);
        const int64_t o = row_id * a.Kp + tid;
        a.cand_draft[o] = -1;
        a.cand_tgt[o] = -1;
        a.cand_val[o] = -INFINITY;
      }
    }
  }
}

template <typename T, bool XFORM>
cudaError_t tk_launch(const TopkArgs& a, cudaStream_t stream) {
  auto kern = topk_row_kernel<T, XFORM>;
  const size_t smem = size_t(TK_STAGES) * TK_STAGE_VEC * 16;
  static int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  const int grid = int(std::min<int64_t>(a.rows, int64_t(2) * ds_num_sms()));
  kern<<<unsigned(grid), TK_THREADS, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

extern "C" dspark_status dspark_topk(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                                     int64_t V_d, int64_t ld, const int64_t* row_start, int32_t K,
                                     float mult, float softcap, const int64_t* d2t, int64_t V_t,
                                     int32_t* cand_draft, int32_t* cand_tgt, float* cand_val,
                                     int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype));
  DS_REQUIRE(R >= 0 && B >= 1 && V_d >= 1 && ld >= V_d && K >= 1 && K <= TK_KMAX);
  DS_REQUIRE(V_d <= 0x7FFFFFFF && R * B <= 0x7FFFFFFF);
  DS_REQUIRE(logits && cand_draft && cand_tgt && cand_val && dev_status);
  DS_REQUIRE(ds_aligned(logits, ds_dtype_size(dtype)));
  DS_REQUIRE(mult == mult && softcap == softcap && softcap >= 0.0f);
  if (d2t) DS_REQUIRE(V_t >= 1);
  if (R == 0) return DSPARK_OK;
  TopkArgs a;
  a.logits = logits;
  a.V = V_d;
  a.ld = ld;
  a.row_start = row_start;
  a.B = B;
  a.Kp = int32_t(K < V_d ? K : V_d);
  a.rows = int32_t(R * B);
  a.mult = mult;
  a.softcap = softcap;
  a.d2t = d2t;
  a.V_t = V_t;
  a.cand_draft = cand_draft;
  a.cand_tgt = cand_tgt;
  a.cand_val = cand_val;
  a.status = dev_status;
  const bool xform = (mult != 1.0f) || (softcap > 0.0f);
  cudaError_t e;
  if (dtype == DSPARK_BF16)
    e = xform ? tk_launch<__nv_bfloat16, true>(a, stream) : tk_launch<__nv_bfloat16, false>(a, stream);
  else
    e = xform ? tk_launch<float, true>(a, stream) : tk_launch<float, false>(a, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}
