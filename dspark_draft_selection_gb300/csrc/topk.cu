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
// Design: one CTA of 512 threads per row, persistent over rows (two CTAs per SM). Thread t owns
// the row's 16-byte vectors t, t + 512, t + 1024, ..., so each batch of the CTA is one contiguous
// stretch of the row and every load is coalesced. The logits go from HBM to registers once;
// nothing is staged in shared memory and no barrier falls inside the stream.
//  1. Stream: each thread loads its vectors in two alternating half-batches of 4 (one in flight
//     while the other is folded in) and keeps the keys (vector maximum, vector number) of its 6
//     largest vectors, sorted, with a branch-free min/max network.
//  2. Bound: each warp pops its m = ceil(2K'/16) largest tracked maxima (REDUX rounds) and one
//     warp finds T, the K'-th largest pop, by a bisection over the value key. The pops are maxima
//     of distinct vectors, so K' distinct elements are >= T and every top-K' element is >= T.
//  3. Gather: only a vector whose maximum reaches T can hold an element >= T. A thread whose
//     sixth tracked maximum is below T knows all its other vectors are below T and re-reads only
//     its tracked vectors that reach T (from L2); otherwise its warp re-reads all of them.
//     Elements >= T go to a shared list (about K' + 3 on Gaussian rows).
//  4. Select: a listed key's rank is the number of listed keys above it (64-bit keys: value, then
//     lower index first); the first K' ranks are written in order with the d2t map.
//  5. A list that overflows its 2048 slots (ties at T, as in a constant row) is cut exactly by a
//     bisection over the 64 key bits, counting the whole row once per bit.
// Launched with programmatic dependent launch: the stream of the logits may overlap the previous
// kernel on the stream; the candidates are written only after that kernel has completed.
#include <type_traits>

#include "dspark_common.cuh"
#include "host_common.h"

namespace {

constexpr int TK_THREADS = 512;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_TRACK = 6;             // largest vectors remembered per thread
constexpr int TK_CAP = 2048;            // listed keys
constexpr int TK_KMAX = 64;
constexpr int TK_POPS = 16;             // tracked maxima a warp offers to the bound (at most)
constexpr int64_t TK_SHORT_V = int64_t(8) * TK_THREADS * 65536;   // rows a 16-bit vector number covers

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

// Geometry of one row: scalar head up to 16-byte alignment, vectors, scalar tail.
struct TkRow {
  const void* row;
  int64_t head, nvec, tail0;
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

// Keys of tracked vectors: the order key of the vector's maximum (-0.0 folded onto +0.0) in the
// high half, the thread's vector number in the low half; 0 marks an empty slot. Rows of bf16
// without transform and at most TK_SHORT_V elements use 16 + 16 bits, other rows 32 + 32 bits.
template <bool SHORT>
struct TkKey {
  using K = uint32_t;
  static constexpr bool narrow = true;
  static constexpr int VBITS = 16;
  DS_DEV static K make(float vmax, uint32_t j) { return (ds_key32(ds_canon_zero(vmax)) & 0xFFFF0000u) | j; }
  DS_DEV static uint32_t val(K k) { return k >> 16; }
  DS_DEV static uint32_t num(K k) { return k & 0xFFFFu; }
  DS_DEV static float to_float(uint32_t v) { return ds_key32_to_float((v << 16) | ((v & 0x8000u) ? 0u : 0xFFFFu)); }
};
template <>
struct TkKey<false> {
  using K = uint64_t;
  static constexpr bool narrow = false;
  static constexpr int VBITS = 32;
  DS_DEV static K make(float vmax, uint32_t j) { return (uint64_t(ds_key32(ds_canon_zero(vmax))) << 32) | j; }
  DS_DEV static uint32_t val(K k) { return uint32_t(k >> 32); }
  DS_DEV static uint32_t num(K k) { return uint32_t(k); }
  DS_DEV static float to_float(uint32_t v) { return ds_key32_to_float(v); }
};

// The largest (transformed) element of a 16-byte vector.
template <typename T, bool XFORM>
DS_DEV float tk_vec_max(const uint4& w, float mult, float softcap) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value && !XFORM) {
    const __nv_bfloat162 m2 = __hmax2(__hmax2(tk_b2(w.x), tk_b2(w.y)), __hmax2(tk_b2(w.z), tk_b2(w.w)));
    return __bfloat162float(__hmax(m2.x, m2.y));
  } else {
    constexpr int EPV = 16 / sizeof(T);
    float m = -INFINITY;
#pragma unroll
    for (int x = 0; x < EPV; ++x) m = fmaxf(m, tk_xform<XFORM>(ds_vec_elem<T>(w, x), mult, softcap));
    return m;
  }
}

// Lists every element >= thr of the row's vector e, loaded as w (thr2: the bound as a bf16 pair).
template <typename T, bool XFORM>
DS_DEV void tk_take(const TopkArgs& a, const uint4& w, int64_t e, int64_t head, float thr,
                    __nv_bfloat162 thr2, uint64_t* s_list, uint32_t* s_n) {
  constexpr int EPV = 16 / sizeof(T);
  const int64_t i0 = head + e * EPV;
  if constexpr (std::is_same<T, __nv_bfloat16>::value && !XFORM) {
    // bytes [e0 e1 e2 e3] and [e4 e5 e6 e7] (0x00 / 0xFF) from packed compares, then one bit each
    const uint32_t c0 = __hge2_mask(tk_b2(w.x), thr2), c1 = __hge2_mask(tk_b2(w.y), thr2);
    const uint32_t c2 = __hge2_mask(tk_b2(w.z), thr2), c3 = __hge2_mask(tk_b2(w.w), thr2);
    const uint32_t w01 = __byte_perm(c0, c1, 0x6420), w23 = __byte_perm(c2, c3, 0x6420);
    uint32_t f = (w01 & 0x08040201u) | (w23 & 0x80402010u);
    f |= f >> 16;
    f |= f >> 8;
    uint32_t m8 = f & 0xFFu;
    while (m8) {
      const int x = __ffs(m8) - 1;
      m8 &= m8 - 1u;
      const uint32_t slot = atomicAdd(s_n, 1u);
      if (slot < uint32_t(TK_CAP)) s_list[slot] = ds_key64(ds_canon_zero(ds_vec_elem<T>(w, x)), uint32_t(i0 + x));
    }
  } else {
#pragma unroll
    for (int x = 0; x < EPV; ++x) {
      const float v = tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap);
      if (v >= thr) {
        const uint32_t slot = atomicAdd(s_n, 1u);
        if (slot < uint32_t(TK_CAP)) s_list[slot] = ds_key64(ds_canon_zero(v), uint32_t(i0 + x));
      }
    }
  }
}

// The K'-th largest of the warps' pops (s_pop[w * TK_POPS + r], r < s_wcnt[w], m per warp at most)
// by a bisection over the VBITS-bit value key, two bits a round, run by one warp: lane l holds the
// pops at flat positions l, l + 32, ... of the 16 x m grid (NV >= ceil(16 m / 32)).
template <int NV, int VBITS>
DS_DEV uint32_t tk_kth_pop(const uint32_t* s_pop, const uint32_t* s_wcnt, int m, uint32_t Kp) {
  const int lane = threadIdx.x & 31;
  uint32_t pv[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int f = lane + 32 * k;
    const int w = f / m, r = f - w * m;
    pv[k] = (w < TK_WARPS && uint32_t(r) < s_wcnt[w]) ? s_pop[w * TK_POPS + r] : 0u;
  }
  uint32_t kth = 0;
#pragma unroll 1
  for (int b = VBITS - 2; b >= 0; b -= 2) {               // two bits a round: three counts
    const uint32_t c1 = kth | (1u << b), c2 = kth | (2u << b), c3 = kth | (3u << b);
    uint32_t n1 = 0, n2 = 0, n3 = 0;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      n1 += pv[k] >= c1 ? 1u : 0u;
      n2 += pv[k] >= c2 ? 1u : 0u;
      n3 += pv[k] >= c3 ? 1u : 0u;
    }
    n1 = __reduce_add_sync(0xFFFFFFFFu, n1);
    n2 = __reduce_add_sync(0xFFFFFFFFu, n2);
    n3 = __reduce_add_sync(0xFFFFFFFFu, n3);
    kth |= ((n1 >= Kp ? 1u : 0u) + (n2 >= Kp ? 1u : 0u) + (n3 >= Kp ? 1u : 0u)) << b;
  }
  return kth;
}

// The row's exact top-K' keys into s_list[0..K'), for a row whose list overflowed: the K'-th
// largest key by bisection over the 64 key bits (the whole row counted per bit, from global
// memory), then every key at or above it. Returns K'.
template <typename T, bool XFORM>
__device__ __noinline__ uint32_t tk_row_exact(const TopkArgs& a, const uint4* rv, int nvt, int64_t head,
                                              int64_t iextra, float xextra, uint64_t* s_list,
                                              uint32_t* s_red, uint32_t* s_n) {
  constexpr int EPV = 16 / sizeof(T);
  const int tid = threadIdx.x;
  uint64_t kres = 0;
  for (int b = 63; b >= 0; --b) {
    const uint64_t cand = kres | (1ull << b);
    uint32_t c = 0;
    for (int j = 0; j < nvt; ++j) {
      const int64_t e = tid + int64_t(j) * TK_THREADS;
      const uint4 w = __ldg(rv + e);
#pragma unroll
      for (int x = 0; x < EPV; ++x) {
        const float v = ds_canon_zero(tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap));
        c += ds_key64(v, uint32_t(head + e * EPV + x)) >= cand ? 1u : 0u;
      }
    }
    if (iextra >= 0) c += ds_key64(ds_canon_zero(xextra), uint32_t(iextra)) >= cand ? 1u : 0u;
    if (tk_block_sum(c, s_red) >= uint32_t(a.Kp)) kres = cand;
  }
  __syncthreads();
  if (tid == 0) *s_n = 0;
  __syncthreads();
  for (int j = 0; j < nvt; ++j) {
    const int64_t e = tid + int64_t(j) * TK_THREADS;
    const uint4 w = __ldg(rv + e);
#pragma unroll
    for (int x = 0; x < EPV; ++x) {
      const float v = ds_canon_zero(tk_xform<XFORM>(ds_vec_elem<T>(w, x), a.mult, a.softcap));
      const uint64_t k = ds_key64(v, uint32_t(head + e * EPV + x));
      if (k >= kres) s_list[atomicAdd(s_n, 1u)] = k;     // exactly K' keys pass
    }
  }
  if (iextra >= 0) {
    const uint64_t k = ds_key64(ds_canon_zero(xextra), uint32_t(iextra));
    if (k >= kres) s_list[atomicAdd(s_n, 1u)] = k;
  }
  __syncthreads();
  return *s_n;
}

template <typename T, bool XFORM, bool SHORT>
__global__ void __launch_bounds__(TK_THREADS, 2) topk_row_kernel(const TopkArgs a) {
  using KK = TkKey<SHORT>;
  using K = typename KK::K;
  constexpr int EPV = 16 / sizeof(T);
  __shared__ uint64_t s_list[TK_CAP];
  __shared__ uint64_t s_top[TK_KMAX];
  __shared__ uint32_t s_red[TK_WARPS];
  __shared__ uint32_t s_pop[TK_WARPS * TK_POPS];
  __shared__ uint32_t s_wcnt[TK_WARPS];
  __shared__ uint32_t s_n, s_tv;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  ds_pdl_trigger();
  bool waited = false;                                     // the previous kernel's completion
  for (int64_t row_id = blockIdx.x; row_id < a.rows; row_id += gridDim.x) {
    const TkRow g = tk_row<T>(a, uint32_t(row_id));
    const T* row = reinterpret_cast<const T*>(g.row);
    const uint4* rv = reinterpret_cast<const uint4*>(row + g.head);
    const int nvt = tid < g.nvec ? int((g.nvec - 1 - tid) / TK_THREADS) + 1 : 0;

    // scalar head and tail elements, one per thread
    int64_t iextra = -1;
    if (tid < g.head) iextra = tid;
    else if (tid >= 8 && tid - 8 < a.V - g.tail0) iextra = g.tail0 + (tid - 8);
    const float xextra = iextra >= 0 ? tk_xform<XFORM>(ds_load_elem<T>(row + iextra), a.mult, a.softcap) : -INFINITY;

    // ---- 1. stream: the six largest vectors of the thread. Two half-batches alternate, so one is
    // always in flight while the other is folded into the tracked keys ----
    constexpr int TK_HALF = KK::narrow ? 4 : 2;             // vectors per half-batch
    K t[TK_TRACK];
#pragma unroll
    for (int i = 0; i < TK_TRACK; ++i) t[i] = 0;
    uint4 wa[TK_HALF], wb[TK_HALF];
    auto load = [&](uint4 (&w)[TK_HALF], int j0) {
#pragma unroll
      for (int u = 0; u < TK_HALF; ++u)
        if (j0 + u < nvt) w[u] = __ldg(rv + (tid + int64_t(j0 + u) * TK_THREADS));
    };
    auto fold = [&](const uint4 (&w)[TK_HALF], int j0) {
#pragma unroll
      for (int u = 0; u < TK_HALF; ++u) {
        if (j0 + u < nvt) {
          K x = KK::make(tk_vec_max<T, XFORM>(w[u], a.mult, a.softcap), uint32_t(j0 + u));
#pragma unroll
          for (int i = 0; i < TK_TRACK; ++i) {
            const K hi = t[i] > x ? t[i] : x;
            x = t[i] > x ? x : t[i];
            t[i] = hi;
          }
        }
      }
    };
    load(wa, 0);
    load(wb, TK_HALF);
    for (int j0 = 0; j0 < nvt; j0 += 2 * TK_HALF) {
      fold(wa, j0);
      load(wa, j0 + 2 * TK_HALF);
      fold(wb, j0 + TK_HALF);
      load(wb, j0 + 3 * TK_HALF);
    }

    // ---- 2. bound: each warp pops its m largest tracked maxima, m = ceil(2K' / warps holding
    // vectors) (at most 16); T is the K'-th largest of all pops, found by one warp. Rows too short
    // for K' pops (under 800 elements) list every element ----
    const int64_t busy = g.nvec < TK_THREADS ? g.nvec : TK_THREADS;
    const int aw = int((busy + 31) / 32);
    const int m_pop = aw > 0 ? min(TK_POPS, (2 * a.Kp + aw - 1) / aw) : 0;
    {
      K c[TK_TRACK];
#pragma unroll
      for (int i = 0; i < TK_TRACK; ++i) c[i] = t[i];
      uint32_t cnt = 0;
      for (int r = 0; r < m_pop; ++r) {
        const uint32_t head = KK::val(c[0]);
        uint32_t top;
        int owner;
        if constexpr (KK::narrow) {                        // value and lane in one 21-bit key
          const uint32_t pk = __reduce_max_sync(0xFFFFFFFFu, (head << 5) | uint32_t(lane));
          top = pk >> 5;
          owner = int(pk & 31u);
        } else {
          top = __reduce_max_sync(0xFFFFFFFFu, head);
          owner = __ffs(__ballot_sync(0xFFFFFFFFu, head == top)) - 1;
        }
        if (top == 0u) break;                              // the warp's tracked vectors are used up
        if (lane == 0) s_pop[warp * TK_POPS + r] = top;
        ++cnt;
        if (lane == owner) {
#pragma unroll
          for (int i = 0; i + 1 < TK_TRACK; ++i) c[i] = c[i + 1];
          c[TK_TRACK - 1] = 0;
        }
      }
      if (lane == 0) s_wcnt[warp] = cnt;
    }
    if (tid == 0) s_n = 0;
    __syncthreads();
    if (warp == 0) {
      uint32_t pops = 0, kth = 0;
#pragma unroll
      for (int w = 0; w < TK_WARPS; ++w) pops += s_wcnt[w];
      if (pops >= uint32_t(a.Kp))                          // else no bound: every element is listed
        kth = tk_kth_pop<TK_POPS / 2, KK::VBITS>(s_pop, s_wcnt, m_pop, uint32_t(a.Kp));
      if (lane == 0) s_tv = kth;
    }
    __syncthreads();
    const uint32_t tv = s_tv;
    const float thr = tv == 0u ? -INFINITY : KK::to_float(tv);
    const __nv_bfloat162 thr2 = __float2bfloat162_rn(thr);   // exact: thr is a bf16 value on packed rows

    // ---- 3. gather the elements >= T ----
    // a thread whose last tracked maximum is below T re-reads only its tracked vectors that reach
    // T (usually none or one); the vectors of the other threads are re-read by their whole warp,
    // one lane per vector
    const bool full = KK::val(t[TK_TRACK - 1]) >= tv;
    if (!full) {
#pragma unroll
      for (int i = 0; i < TK_TRACK; ++i) {
        if (KK::val(t[i]) >= tv) {
          const int64_t e = tid + int64_t(KK::num(t[i])) * TK_THREADS;
          tk_take<T, XFORM>(a, __ldg(rv + e), e, g.head, thr, thr2, s_list, &s_n);
        }
      }
    }
    for (unsigned fm = __ballot_sync(0xFFFFFFFFu, full); fm != 0u; fm &= fm - 1u) {
      const int src = __ffs(fm) - 1;
      const int stid = (tid & ~31) + src;
      const int snvt = __shfl_sync(0xFFFFFFFFu, nvt, src);
      for (int j = lane; j < snvt; j += 32) {
        const int64_t e = stid + int64_t(j) * TK_THREADS;
        tk_take<T, XFORM>(a, __ldg(rv + e), e, g.head, thr, thr2, s_list, &s_n);
      }
    }
    if (iextra >= 0 && xextra >= thr) {
      const uint32_t slot = atomicAdd(&s_n, 1u);
      if (slot < uint32_t(TK_CAP)) s_list[slot] = ds_key64(ds_canon_zero(xextra), uint32_t(iextra));
    }
    __syncthreads();
    uint32_t N = s_n;
    if (N > uint32_t(TK_CAP)) N = tk_row_exact<T, XFORM>(a, rv, nvt, g.head, iextra, xextra, s_list, s_red, &s_n);

    // ---- 4. rank the listed keys: P threads share a key's count (P = 1, 2, 4 or 8) ----
    {
      uint32_t P = 1;
      while (P < 8u && N * P * 2u <= uint32_t(TK_THREADS)) P *= 2u;
      const uint32_t sub = tid & (P - 1u), per = uint32_t(TK_THREADS) / P;
      for (uint32_t base = 0; base < N; base += per) {
        if (base + uint32_t(warp * 32) / P >= N) continue;   // no key for this warp
        const uint32_t q = base + tid / P;
        const uint64_t k = q < N ? s_list[q] : ~0ull;
        uint32_t pos = 0, u = sub;
        for (; u + 7u * P < N; u += 8u * P) {
          uint32_t cnt = 0;
#pragma unroll
          for (int r = 0; r < 8; ++r) cnt += (s_list[u + r * P] > k) ? 1u : 0u;
          pos += cnt;
        }
        for (; u < N; u += P) pos += (s_list[u] > k) ? 1u : 0u;
        for (uint32_t o = 1; o < P; o <<= 1) pos += __shfl_xor_sync(0xFFFFFFFFu, pos, o);
        if (q < N && sub == 0u && pos < uint32_t(a.Kp)) s_top[pos] = k;
      }
    }
    __syncthreads();
    if (!waited) {                                         // the logits were read before it; the
      ds_pdl_wait();                                       // outputs are written after it
      waited = true;
    }
    if (tid < a.Kp) {
      if (uint32_t(tid) < N) {
        tk_emit(a, uint32_t(row_id), tid, s_top[tid]);
      } else {                                             // unreachable: every row holds >= K' elements
        ds_set_error(a.status, DSPARK_EINVAL);
        const int64_t o = row_id * a.Kp + tid;
        a.cand_draft[o] = -1;
        a.cand_tgt[o] = -1;
        a.cand_val[o] = -INFINITY;
      }
    }
    __syncthreads();                                       // the lists are rebuilt for the next row
  }
  (void)EPV;
}

template <typename T, bool XFORM, bool SHORT>
cudaError_t tk_launch(const TopkArgs& a, cudaStream_t stream) {
  const int grid = int(std::min<int64_t>(a.rows, int64_t(2) * ds_num_sms()));
  return ds_launch(topk_row_kernel<T, XFORM, SHORT>, dim3(unsigned(grid)), dim3(TK_THREADS), 0, stream, a);
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
  if (dtype == DSPARK_BF16 && !xform)
    e = V_d <= TK_SHORT_V ? tk_launch<__nv_bfloat16, false, true>(a, stream)
                          : tk_launch<__nv_bfloat16, false, false>(a, stream);
  else if (dtype == DSPARK_BF16)
    e = tk_launch<__nv_bfloat16, true, false>(a, stream);
  else
    e = xform ? tk_launch<float, true, false>(a, stream) : tk_launch<float, false, false>(a, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}
