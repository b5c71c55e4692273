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
// Design: every row is split into P parts handled by independent CTAs (no CTA ever waits for
// another), so the logits stream from HBM at full occupancy; the logits are read once.
//  1. A part's 16-byte vectors are dealt round-robin to the CTA's 256 threads (coalesced
//     streaming loads, <= 8 vectors per thread held in registers).
//  2. Each warp takes the m-th largest of its lanes' maxima (m = ceil(K'/8), warp REDUX rounds):
//     each lane maximum is a distinct element, so 8 warps x m >= K' elements are >= the minimum
//     T_p over the warps; T_p bounds the part's K'-th largest value from below.
//  3. Elements >= T_p survive (a few K' per part) and go, as 64-bit (value, lower index first)
//     keys, to a small per-part slot of the workspace.
//  4. The last CTA of the row to finish (a ticket counter) merges: max_p T_p bounds the row's
//     K'-th value, a 32-step bisection over the surviving values finds the exact K'-th value,
//     and a short bitonic sort orders the few keys at or above it. Ties that overflow the
//     per-part slots send the row to an exact bisection over the row itself (slow, rare).
#include <type_traits>

#include "dspark_common.cuh"
#include "host_common.h"

namespace {

constexpr int TK_THREADS = 256;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_MAXV = 8;         // 16-byte vectors per thread
constexpr int TK_PART_CAP = 256;   // survivor keys kept per part
constexpr int TK_MERGE_CAP = 2048; // keys gathered by the merging CTA
constexpr int TK_MAXP = 64;
static_assert(TK_PART_CAP <= TK_MERGE_CAP, "part survivors are staged in the merge buffer");

struct TopkArgs {
  const void* logits;
  int64_t V, ld;
  const int64_t* row_start;
  int32_t B, Kp, P;
  int64_t nvp;                     // vectors per part
  float mult, softcap;
  const int64_t* d2t;
  int64_t V_t;
  int32_t* cand_draft;
  int32_t* cand_tgt;
  float* cand_val;
  int32_t* status;
  uint64_t* ws_keys;               // [rows * P * TK_PART_CAP]
  uint32_t* ws_cnt;                // [rows * P]
  float* ws_thr;                   // [rows * P]
  uint32_t* ws_ticket;             // [rows], zero between calls
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

// The part's exact K'-th largest value key, by bisection over the part re-read from memory (only
// for a part whose survivors overflow their slot).
template <typename T, bool XFORM>
__device__ __noinline__ uint32_t tk_part_kth(const TopkArgs& a, const T* row, int64_t head, int64_t v0, int64_t v1,
                                             int64_t iextra, uint32_t* s_red) {
  constexpr int EPV = 16 / sizeof(T);
  uint32_t vres = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = vres | (1u << b);
    uint32_t c = 0;
    if (iextra >= 0)
      c += (ds_key32(ds_canon_zero(tk_xform<XFORM>(ds_load_elem<T>(row + iextra), a.mult, a.softcap))) >= cand) ? 1u : 0u;
    for (int64_t i = (head + v0 * EPV) + threadIdx.x; i < head + v1 * EPV; i += TK_THREADS)
      c += (ds_key32(ds_canon_zero(tk_xform<XFORM>(ds_load_elem<T>(row + i), a.mult, a.softcap))) >= cand) ? 1u : 0u;
    if (tk_block_sum(c, s_red) >= uint32_t(a.Kp)) vres = cand;
  }
  return vres;
}

template <typename T, bool XFORM>
__device__ __noinline__ float tk_part_refine(const TopkArgs& a, const T* row, int64_t head, int64_t v0, int64_t v1,
                                             int64_t iextra, uint64_t* s_keys, uint32_t* s_red, uint32_t* s_n) {
  constexpr int EPV = 16 / sizeof(T);
  const uint32_t vres = tk_part_kth<T, XFORM>(a, row, head, v0, v1, iextra, s_red);
  const float thr = ds_key32_to_float(vres);
  __syncthreads();
  if (threadIdx.x == 0) *s_n = 0;
  __syncthreads();
  auto visit = [&](int64_t i) {
    const float x = tk_xform<XFORM>(ds_load_elem<T>(row + i), a.mult, a.softcap);
    if (x >= thr) {
      const uint32_t slot = atomicAdd(s_n, 1u);
      if (slot < TK_PART_CAP) s_keys[slot] = ds_key64(ds_canon_zero(x), uint32_t(i));
    }
  };
  if (iextra >= 0) visit(iextra);
  for (int64_t i = (head + v0 * EPV) + threadIdx.x; i < head + v1 * EPV; i += TK_THREADS) visit(i);
  __syncthreads();
  return thr;
}

// Exact top-K' of the whole row by bisection over 64-bit keys (ties flooding the buffers).
template <typename T, bool XFORM>
__device__ __noinline__ int tk_row_exact(const TopkArgs& a, const T* row, uint64_t* s_keys, uint32_t* s_red, uint32_t* s_n) {
  uint64_t kres = 0;
  for (int b = 63; b >= 0; --b) {
    const uint64_t cand = kres | (1ull << b);
    uint32_t c = 0;
    for (int64_t i = threadIdx.x; i < a.V; i += TK_THREADS) {
      const float x = ds_canon_zero(tk_xform<XFORM>(ds_load_elem<T>(row + i), a.mult, a.softcap));
      c += (ds_key64(x, uint32_t(i)) >= cand) ? 1u : 0u;
    }
    if (tk_block_sum(c, s_red) >= uint32_t(a.Kp)) kres = cand;
  }
  if (threadIdx.x == 0) *s_n = 0;
  __syncthreads();
  for (int64_t i = threadIdx.x; i < a.V; i += TK_THREADS) {
    const float x = ds_canon_zero(tk_xform<XFORM>(ds_load_elem<T>(row + i), a.mult, a.softcap));
    const uint64_t k = ds_key64(x, uint32_t(i));
    if (k >= kres) {
      const uint32_t slot = atomicAdd(s_n, 1u);
      if (slot < TK_MERGE_CAP) s_keys[slot] = k;
    }
  }
  __syncthreads();
  return int(min(*s_n, uint32_t(TK_MERGE_CAP)));
}

template <typename T, bool XFORM>
__global__ void __launch_bounds__(TK_THREADS, 4) topk_part_kernel(const TopkArgs a) {
  constexpr int EPV = 16 / sizeof(T);
  __shared__ uint64_t s_keys[TK_MERGE_CAP];
  __shared__ uint32_t s_red[TK_WARPS];
  __shared__ float s_wthr[TK_WARPS];
  __shared__ uint32_t s_n;
  __shared__ int s_last;

  const int P = a.P;                                  // a power of two
  const uint32_t row_id = blockIdx.x >> (31 - __clz(P));   // r * B + j
  const int p = int(blockIdx.x & uint32_t(P - 1));
  int64_t prow = row_id;
  if (a.row_start) {
    const uint32_t r = row_id / uint32_t(a.B);
    prow = a.row_start[r] + (row_id - r * uint32_t(a.B));
  }
  const T* row = reinterpret_cast<const T*>(a.logits) + prow * a.ld;
  const int64_t V = a.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // row = scalar head (until 16-byte alignment) + vectors + scalar tail; head on part 0, tail on P-1
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  int64_t head = int64_t(((16u - (addr & 15u)) & 15u) / sizeof(T));
  if (head > V) head = V;
  const int64_t nvec = (V - head) / EPV;
  const int64_t tail0 = head + nvec * EPV;
  const int64_t v0 = int64_t(p) * a.nvp, v1 = min(nvec, v0 + a.nvp);
  const uint4* vbase = reinterpret_cast<const uint4*>(row + head);

  const int32_t lv0 = int32_t(v0) + tid, lv1 = int32_t(v1);   // this lane's vector indices (V < 2^31)
  uint4 buf[TK_MAXV];
#pragma unroll
  for (int k = 0; k < TK_MAXV; ++k) {
    if (lv0 + k * TK_THREADS < lv1) buf[k] = ds_ld_stream(vbase + (lv0 + k * TK_THREADS));
  }
  float xextra = -INFINITY;
  int64_t iextra = -1;
  if (p == 0 && tid < head) iextra = tid;
  if (p == P - 1 && tid >= 8 && tid - 8 < V - tail0) iextra = tail0 + (tid - 8);
  if (iextra >= 0) xextra = tk_xform<XFORM>(ds_load_elem<T>(row + iextra), a.mult, a.softcap);
  if (tid == 0) s_n = 0;

  // lane maximum (bf16 rows without a transform stay packed: two elements per instruction)
  constexpr bool PACKED = std::is_same<T, __nv_bfloat16>::value && !XFORM;
  float tmax = xextra;
  if constexpr (PACKED) {
    __nv_bfloat162 m2 = __float2bfloat162_rn(-INFINITY);
#pragma unroll
    for (int k = 0; k < TK_MAXV; ++k) {
      if (lv0 + k * TK_THREADS < lv1) {
        m2 = __hmax2(m2, tk_b2(buf[k].x));
        m2 = __hmax2(m2, tk_b2(buf[k].y));
        m2 = __hmax2(m2, tk_b2(buf[k].z));
        m2 = __hmax2(m2, tk_b2(buf[k].w));
      }
    }
    tmax = fmaxf(tmax, fmaxf(__low2float(m2), __high2float(m2)));
  } else {
#pragma unroll
    for (int k = 0; k < TK_MAXV; ++k) {
      if (lv0 + k * TK_THREADS < lv1) {
#pragma unroll
        for (int e = 0; e < EPV; ++e)
          tmax = fmaxf(tmax, tk_xform<XFORM>(ds_vec_elem<T>(buf[k], e), a.mult, a.softcap));
      }
    }
  }
  // the warp's m-th largest lane maximum (removed lanes drop to key 0, below every value)
  const int m = (a.Kp + TK_WARPS - 1) / TK_WARPS;
  uint32_t key = ds_key32(ds_canon_zero(tmax));
  uint32_t kth = 0;
#pragma unroll
  for (int t = 0; t < (64 + TK_WARPS - 1) / TK_WARPS; ++t) {
    if (t < m) {
      kth = __reduce_max_sync(0xFFFFFFFFu, key);
      const unsigned who = __ballot_sync(0xFFFFFFFFu, key == kth);
      if (lane == __ffs(who) - 1) key = 0;
    }
  }
  if (lane == 0) s_wthr[warp] = (kth <= ds_key32(-INFINITY)) ? -INFINITY : ds_key32_to_float(kth);
  __syncthreads();
  float thr = s_wthr[0];
#pragma unroll
  for (int w = 1; w < TK_WARPS; ++w) thr = fminf(thr, s_wthr[w]);

  // survivors: elements >= thr. Every round k adds an 8-bit mask of this lane's survivors to one
  // 64-bit mask (packed compares, no branches); the warp then drains all masks together, one
  // survivor per lane per pass with one shared-memory atomic per pass, so a lane's rare
  // survivors do not hold the whole warp in a per-element loop.
  {
    const __nv_bfloat162 thr2 = __float2bfloat162_rn(thr);   // exact: thr is an element value or -inf
    const int32_t vv0 = lv0, vv1 = lv1;
    unsigned long long mm = 0;
#pragma unroll
    for (int k = 0; k < TK_MAXV; ++k) {
      uint32_t m8 = 0;
      if (vv0 + k * TK_THREADS < vv1) {
        if constexpr (PACKED) {
          const uint32_t c0 = __hge2_mask(tk_b2(buf[k].x), thr2), c1 = __hge2_mask(tk_b2(buf[k].y), thr2);
          const uint32_t c2 = __hge2_mask(tk_b2(buf[k].z), thr2), c3 = __hge2_mask(tk_b2(buf[k].w), thr2);
          // bytes [e0 e1 e2 e3] and [e4 e5 e6 e7] (0x00 / 0xFF), then one bit per element
          const uint32_t w01 = __byte_perm(c0, c1, 0x6420), w23 = __byte_perm(c2, c3, 0x6420);
          uint32_t f = (w01 & 0x08040201u) | (w23 & 0x80402010u);
          f |= f >> 16;
          f |= f >> 8;
          m8 = f & 0xFFu;
        } else {
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            m8 |= (tk_xform<XFORM>(ds_vec_elem<T>(buf[k], e), a.mult, a.softcap) >= thr) ? (1u << e) : 0u;
        }
      }
      mm |= (unsigned long long)m8 << (8 * k);
    }
    const unsigned below = (1u << lane) - 1u;
    while (true) {
      const unsigned act = __ballot_sync(0xFFFFFFFFu, mm != 0ull);
      if (act == 0u) break;
      uint32_t slot = 0;
      const int leader = __ffs(act) - 1;
      if (lane == leader) slot = atomicAdd(&s_n, uint32_t(__popc(act)));
      slot = __shfl_sync(0xFFFFFFFFu, slot, leader) + uint32_t(__popc(act & below));
      if (mm != 0ull) {
        const int bit = __ffsll(mm) - 1;
        mm &= mm - 1ull;
        const int k = bit >> 3, e = bit & 7;
        uint4 q = buf[0];
#pragma unroll
        for (int kk = 1; kk < TK_MAXV; ++kk)
          if (k == kk) q = buf[kk];
        const float x = tk_xform<XFORM>(ds_vec_elem<T>(q, e), a.mult, a.softcap);
        if (slot < TK_PART_CAP)
          s_keys[slot] = ds_key64(ds_canon_zero(x), uint32_t(head) + uint32_t(vv0 + k * TK_THREADS) * EPV + uint32_t(e));
      }
    }
    if (iextra >= 0 && xextra >= thr) {
      const uint32_t slot = atomicAdd(&s_n, 1u);
      if (slot < TK_PART_CAP) s_keys[slot] = ds_key64(ds_canon_zero(xextra), uint32_t(iextra));
    }
  }
  __syncthreads();
  if (s_n > uint32_t(TK_PART_CAP)) {
    // the survivors overflow the slot: tighten thr to the part's own exact K'-th largest value
    // and collect again (rare; both from memory)
    thr = tk_part_refine<T, XFORM>(a, row, head, v0, v1, iextra, s_keys, s_red, &s_n);
  }
  __syncthreads();
  const uint32_t n = s_n;
  const int64_t part = int64_t(row_id) * P + p;
  for (uint32_t i = tid; i < min(n, uint32_t(TK_PART_CAP)); i += TK_THREADS) a.ws_keys[part * TK_PART_CAP + i] = s_keys[i];
  if (tid == 0) {
    a.ws_cnt[part] = n;
    a.ws_thr[part] = thr;
    __threadfence();
    const uint32_t old = atomicAdd(&a.ws_ticket[row_id], 1u);
    s_last = (old == uint32_t(P - 1));
  }
  __syncthreads();
  if (!s_last) return;

  // ---- merge: this CTA finished last for its row ----
  __threadfence();
  __shared__ uint32_t s_off[TK_MAXP + 1];
  __shared__ float s_rthr;
  __shared__ int s_bad;
  if (tid == 0) {
    float rthr = -INFINITY;
    uint32_t off = 0;
    int bad = 0;
    for (int q = 0; q < P; ++q) {
      const uint32_t c = __ldcg(&a.ws_cnt[int64_t(row_id) * P + q]);
      rthr = fmaxf(rthr, __ldcg(&a.ws_thr[int64_t(row_id) * P + q]));
      bad |= c > uint32_t(TK_PART_CAP);
      s_off[q] = off;
      off += min(c, uint32_t(TK_PART_CAP));
    }
    s_off[P] = off;
    s_rthr = rthr;
    s_bad = bad;
  }
  __syncthreads();
  const float rthr = s_rthr;
  // keys >= the row bound, gathered from every part's slot into shared memory
  if (tid == 0) s_n = 0;
  __syncthreads();
  {
    int q = 0;
    for (uint32_t g = tid; g < s_off[P]; g += TK_THREADS) {
      while (g >= s_off[q + 1]) ++q;
      const uint64_t k = __ldcg(&a.ws_keys[(int64_t(row_id) * P + q) * TK_PART_CAP + (g - s_off[q])]);
      if (ds_key64_val(k) >= rthr) {
        const uint32_t slot = atomicAdd(&s_n, 1u);
        if (slot < TK_MERGE_CAP) s_keys[slot] = k;
      }
    }
  }
  __syncthreads();
  const uint32_t ngot = s_n;
  int nk;
  if (!s_bad && ngot <= uint32_t(TK_MERGE_CAP)) {
    // exact K'-th largest value among them, by bisection on the value key
    // (bf16 values without a transform have keys whose low 16 bits carry no order, so the
    // bisection stops after the top 16 bits)
    uint32_t vres = 0;
    const int blo = PACKED ? 16 : 0;
    for (int b = 31; b >= blo; --b) {
      const uint32_t cand = vres | (1u << b);
      uint32_t c = 0;
      for (uint32_t i = tid; i < ngot; i += TK_THREADS) c += (uint32_t(s_keys[i] >> 32) >= cand) ? 1u : 0u;
      if (tk_block_sum(c, s_red) >= uint32_t(a.Kp)) vres = cand;
    }
    // compact the keys at or above it to the front (in place: the block walks the buffer in
    // passes of TK_THREADS so that no thread overwrites a key another thread has not read yet)
    if (tid == 0) s_n = 0;
    __syncthreads();
    for (uint32_t i0 = 0; i0 < ngot; i0 += TK_THREADS) {
      const uint32_t i = i0 + tid;
      const uint64_t k = (i < ngot) ? s_keys[i] : 0;
      const bool keep = (i < ngot) && uint32_t(k >> 32) >= vres;
      __syncthreads();
      if (keep) s_keys[atomicAdd(&s_n, 1u)] = k;
      __syncthreads();
    }
    nk = int(s_n);
  } else {
    nk = tk_row_exact<T, XFORM>(a, row, s_keys, s_red, &s_n);
  }
  int n2 = 1;
  while (n2 < nk) n2 <<= 1;
  for (int i = nk + tid; i < n2; i += TK_THREADS) s_keys[i] = 0;
  __syncthreads();
  ds_block_sort_desc(s_keys, n2);
  if (tid < a.Kp && tid >= nk) {               // unreachable: >= K' keys always reach the sort
    ds_set_error(a.status, DSPARK_EINVAL);
    const int64_t o = int64_t(row_id) * a.Kp + tid;
    a.cand_draft[o] = -1;
    a.cand_tgt[o] = -1;
    a.cand_val[o] = -INFINITY;
  } else if (tid < a.Kp) {
    const uint64_t k64 = s_keys[tid];
    const uint32_t idx = ds_key64_idx(k64);
    int64_t tgt = idx;
    if (a.d2t) {
      tgt = int64_t(idx) + a.d2t[idx];
      if (tgt < 0 || tgt >= a.V_t) {
        ds_set_error(a.status, DSPARK_ERANGE);
        tgt = -1;
      }
    }
    const int64_t o = int64_t(row_id) * a.Kp + tid;
    a.cand_draft[o] = int32_t(idx);
    a.cand_tgt[o] = int32_t(tgt);
    a.cand_val[o] = ds_key64_val(k64);
  }
  if (tid == 0) a.ws_ticket[row_id] = 0;
}

size_t tk_align(size_t x) { return (x + 255) & ~size_t(255); }

struct TopkLayout {
  int P;
  int64_t nvp;
  size_t keys, cnt, thr, ticket, total;
};

TopkLayout tk_layout(int64_t rows, int64_t V, int elem_bytes) {
  TopkLayout L = {};
  const int64_t epv = 16 / elem_bytes;
  const int64_t nvec = V / epv + 1;
  int P = 1;
  while (P < TK_MAXP && ds_ceil_div(nvec, P) > int64_t(TK_THREADS) * TK_MAXV) P <<= 1;
  L.P = P;
  L.nvp = ds_ceil_div(nvec, P);
  L.keys = tk_align(size_t(rows) * P * TK_PART_CAP * sizeof(uint64_t));
  L.cnt = tk_align(size_t(rows) * P * sizeof(uint32_t));
  L.thr = tk_align(size_t(rows) * P * sizeof(float));
  L.ticket = tk_align(size_t(rows) * sizeof(uint32_t));
  L.total = L.keys + L.cnt + L.thr + L.ticket;
  return L;
}

template <typename T, bool XFORM>
cudaError_t tk_launch(const TopkArgs& a, int64_t rows, cudaStream_t stream) {
  topk_part_kernel<T, XFORM><<<unsigned(rows * a.P), TK_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

extern "C" size_t dspark_internal_ws_topk(int64_t R, int32_t B, int64_t V) {
  // float32 rows hold 4 elements per 16-byte vector, so they split into the most parts
  return std::max(tk_layout(R * B, V, 4).total, tk_layout(R * B, V, 2).total);
}

extern "C" dspark_status dspark_topk(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                                     int64_t V_d, int64_t ld, const int64_t* row_start, int32_t K,
                                     float mult, float softcap, const int64_t* d2t, int64_t V_t,
                                     int32_t* cand_draft, int32_t* cand_tgt, float* cand_val, void* ws,
                                     size_t ws_bytes, int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype));
  DS_REQUIRE(R >= 0 && B >= 1 && V_d >= 1 && ld >= V_d && K >= 1 && K <= 64);
  DS_REQUIRE(V_d <= 0x7FFFFFFF && R * B <= 0x7FFFFFFF);
  DS_REQUIRE(logits && cand_draft && cand_tgt && cand_val && dev_status);
  DS_REQUIRE(ds_aligned(logits, ds_dtype_size(dtype)));
  DS_REQUIRE(mult == mult && softcap == softcap && softcap >= 0.0f);
  if (d2t) DS_REQUIRE(V_t >= 1);
  if (R == 0) return DSPARK_OK;
  const int64_t rows = R * B;
  const TopkLayout L = tk_layout(rows, V_d, ds_dtype_size(dtype));
  DS_REQUIRE(int64_t(L.P) * TK_THREADS * TK_MAXV >= L.nvp * L.P);
  if (!ws || ws_bytes < L.total || !ds_aligned(ws, 256)) return DSPARK_EWORKSPACE;
  uint8_t* w = reinterpret_cast<uint8_t*>(ws);
  TopkArgs a;
  a.logits = logits;
  a.V = V_d;
  a.ld = ld;
  a.row_start = row_start;
  a.B = B;
  a.Kp = int32_t(K < V_d ? K : V_d);
  a.P = L.P;
  a.nvp = L.nvp;
  a.mult = mult;
  a.softcap = softcap;
  a.d2t = d2t;
  a.V_t = V_t;
  a.cand_draft = cand_draft;
  a.cand_tgt = cand_tgt;
  a.cand_val = cand_val;
  a.status = dev_status;
  a.ws_keys = reinterpret_cast<uint64_t*>(w);
  a.ws_cnt = reinterpret_cast<uint32_t*>(w + L.keys);
  a.ws_thr = reinterpret_cast<float*>(w + L.keys + L.cnt);
  a.ws_ticket = reinterpret_cast<uint32_t*>(w + L.keys + L.cnt + L.thr);
  const bool xform = (mult != 1.0f) || (softcap > 0.0f);
  cudaError_t e;
  if (dtype == DSPARK_BF16)
    e = xform ? tk_launch<__nv_bfloat16, true>(a, rows, stream) : tk_launch<__nv_bfloat16, false>(a, rows, stream);
  else
    e = xform ? tk_launch<float, true>(a, rows, stream) : tk_launch<float, false>(a, rows, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}
