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
// Design: persistent CTAs (two per SM) stream row parts of up to 42 KB through a 2-stage
// shared-memory ring filled by bulk asynchronous copies (cp.async.bulk + mbarrier transaction
// counts), so HBM keeps streaming while a part is processed; the logits are read once.
// Per part (~85 elements per lane):
//  1. Each warp takes the m-th largest of its lanes' maxima (m = ceil(K'/8), warp REDUX rounds):
//     each lane maximum is a distinct element, so 8 warps x m >= K' elements are >= the minimum
//     T_p over the warps; T_p bounds the part's K'-th largest value from below.
//  2. Elements >= T_p survive (a few K' per part). The vectors whose maximum (kept from the first
//     pass) clears T_p are queued per warp; the warp takes them 32 at a time, builds 8-bit
//     survivor masks with packed bf16x2 compares and drains them together (one survivor per lane
//     per pass, one shared-memory atomic per pass), reading values back from shared memory.
//  3. Survivors go, as 64-bit (value, lower index first) keys, to a per-part workspace slot.
//  4. A second kernel merges each row (one CTA per row): max_p T_p bounds the row's K'-th value;
//     the m-th largest per-thread maximum of the keys above it per warp tightens the bound; each
//     key left (about 2K') is ranked by counting the keys above it and written to its slot. A part whose survivors overflow its slot first tightens T_p
//     to its own exact K'-th value; ties that still overflow send the row to an exact bisection
//     over the row itself (slow, rare). No CTA waits for another and the workspace keeps no state.
#include <type_traits>

#include "dspark_common.cuh"
#include "host_common.h"

namespace {

constexpr int TK_THREADS = 256;
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_STAGES = 2;
constexpr int TK_STAGE_VEC = 2688;      // 16-byte vectors per stage (42 KB)
constexpr int TK_PART_CAP = 512;        // survivor keys kept per part
constexpr int TK_MERGE_CAP = 2048;      // keys gathered by the merging CTA
constexpr int TK_SEL_CAP = 512;         // keys ranked by the merging CTA
constexpr int TK_ROUNDS = (TK_STAGE_VEC + TK_THREADS - 1) / TK_THREADS;   // vectors per lane per part
constexpr int TK_QCAP = 32 * TK_ROUNDS;  // per-warp queue of candidate vectors
static_assert(TK_PART_CAP <= TK_MERGE_CAP, "part survivors are staged in the merge buffer");

struct TopkArgs {
  const void* logits;
  int64_t V, ld;
  const int64_t* row_start;
  int32_t B, Kp, P;
  int32_t nvp;                     // vectors per part
  int32_t nitems;                  // rows * P
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

// The part's exact K'-th largest value key, by bisection over the part re-read from memory (only
// for a part whose survivors overflow their slot), then the survivors at or above it. Elements
// [e0, e1) and [x0, x1) form the part.
template <typename T, bool XFORM>
__device__ __noinline__ float tk_part_refine(const TopkArgs& a, const T* row, int64_t e0, int64_t e1, int64_t x0,
                                             int64_t x1, uint64_t* s_keys, uint32_t* s_red, uint32_t* s_n) {
  auto val = [&](int64_t i) { return ds_canon_zero(tk_xform<XFORM>(ds_load_elem<T>(row + i), a.mult, a.softcap)); };
  uint32_t vres = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = vres | (1u << b);
    uint32_t c = 0;
    for (int64_t i = e0 + threadIdx.x; i < e1; i += TK_THREADS) c += (ds_key32(val(i)) >= cand) ? 1u : 0u;
    for (int64_t i = x0 + threadIdx.x; i < x1; i += TK_THREADS) c += (ds_key32(val(i)) >= cand) ? 1u : 0u;
    if (tk_block_sum(c, s_red) >= uint32_t(a.Kp)) vres = cand;
  }
  const float thr = ds_key32_to_float(vres);
  __syncthreads();
  if (threadIdx.x == 0) *s_n = 0;
  __syncthreads();
  auto visit = [&](int64_t i) {
    const float x = val(i);
    if (x >= thr) {
      const uint32_t slot = atomicAdd(s_n, 1u);
      if (slot < TK_PART_CAP) s_keys[slot] = ds_key64(x, uint32_t(i));
    }
  };
  for (int64_t i = e0 + threadIdx.x; i < e1; i += TK_THREADS) visit(i);
  for (int64_t i = x0 + threadIdx.x; i < x1; i += TK_THREADS) visit(i);
  __syncthreads();
  return thr;
}

// Exact top-K' of the whole row by bisection over 64-bit keys (ties flooding the buffers).
template <typename T, bool XFORM>
__device__ __noinline__ int tk_row_exact(const TopkArgs& a, const T* row, uint64_t* s_keys, uint32_t* s_red,
                                         uint32_t* s_n) {
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
__global__ void __launch_bounds__(TK_THREADS, 2) topk_stream_kernel(const TopkArgs a) {
  constexpr int EPV = 16 / sizeof(T);
  constexpr bool PACKED = std::is_same<T, __nv_bfloat16>::value && !XFORM;
  extern __shared__ __align__(128) uint8_t tk_dyn[];      // TK_STAGES x TK_STAGE_VEC x 16 bytes
  __shared__ uint64_t s_full[TK_STAGES];
  __shared__ uint64_t s_keys[TK_MERGE_CAP];
  __shared__ uint32_t s_red[TK_WARPS];
  __shared__ float s_wthr[TK_WARPS];
  __shared__ uint32_t s_n;
  __shared__ uint16_t s_queue[TK_WARPS][TK_QCAP];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = a.P;
  const uint4* stages = reinterpret_cast<const uint4*>(tk_dyn);

  // producer: thread 0 issues the bulk copy of an item's vectors into a stage
  auto issue = [&](int item, int s) {
    const uint32_t row_id = uint32_t(item) / uint32_t(P);
    const int p = item - int(row_id) * P;
    const TkRow g = tk_row<T>(a, row_id);
    const int64_t v0 = int64_t(p) * a.nvp, v1 = min(g.nvec, v0 + a.nvp);
    const uint32_t bytes = v1 > v0 ? uint32_t((v1 - v0) * 16) : 0u;
    ds_mbar_arrive_expect_tx(&s_full[s], bytes);
    if (bytes)
      ds_bulk_g2s(tk_dyn + size_t(s) * TK_STAGE_VEC * 16,
                  reinterpret_cast<const uint8_t*>(g.row) + g.head * int64_t(sizeof(T)) + v0 * 16, bytes, &s_full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < TK_STAGES; ++s) ds_mbar_init(&s_full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    for (int s = 0; s < TK_STAGES; ++s) {
      const int item = blockIdx.x + s * gridDim.x;
      if (item < a.nitems) issue(item, s);
    }
  }
  const unsigned below = (1u << lane) - 1u;
  const int m = (a.Kp + TK_WARPS - 1) / TK_WARPS;

  int n = 0;
  for (int item = blockIdx.x; item < a.nitems; item += gridDim.x, ++n) {
    const int s = n % TK_STAGES;
    const uint32_t parity = uint32_t(n / TK_STAGES) & 1u;
    const uint32_t row_id = uint32_t(item) / uint32_t(P);
    const int p = item - int(row_id) * P;
    const TkRow g = tk_row<T>(a, row_id);
    const T* row = reinterpret_cast<const T*>(g.row);
    const int64_t v0 = int64_t(p) * a.nvp, v1 = min(g.nvec, v0 + a.nvp);
    const int nv = v1 > v0 ? int(v1 - v0) : 0;
    const uint4* sv = stages + size_t(s) * TK_STAGE_VEC;

    // scalar head (first part) and tail (last part) elements, loaded directly
    int64_t iextra = -1;
    if (p == 0 && tid < g.head) iextra = tid;
    if (p == P - 1 && tid >= 8 && tid - 8 < a.V - g.tail0) iextra = g.tail0 + (tid - 8);
    const float xextra = iextra >= 0 ? tk_xform<XFORM>(ds_load_elem<T>(row + iextra), a.mult, a.softcap) : -INFINITY;
    if (tid == 0) s_n = 0;

    bool ok = ds_mbar_wait(&s_full[s], parity, DS_WAIT_LIMIT);
    ok = __syncthreads_and(ok) != 0;
    if (!ok) {
      // a copy never completed: report it and stop (copies still in flight target this CTA's
      // shared memory only, which stays allocated until they land or the kernel ends)
      if (tid == 0) ds_set_error(a.status, DSPARK_ETIMEOUT);
      for (int t = 0; t < TK_STAGES; ++t) (void)ds_mbar_wait(&s_full[t], parity, DS_WAIT_LIMIT);
      return;
    }

    // lane maximum, keeping every vector's own maximum for the screening pass
    float tmax = xextra;
    float vmax[TK_ROUNDS];
#pragma unroll
    for (int k = 0; k < TK_ROUNDS; ++k) {
      const int i = tid + k * TK_THREADS;
      vmax[k] = -INFINITY;
      if (i < nv) {
        const uint4 w = sv[i];
        if constexpr (PACKED) {
          const __nv_bfloat162 m2 = __hmax2(__hmax2(tk_b2(w.x), tk_b2(w.y)), __hmax2(tk_b2(w.z), tk_b2(w.w)));
          vmax[k] = fmaxf(__low2float(m2), __high2float(m2));
        } else {
#pragma unroll
          for (int e = 0; e < EPV; ++e) vmax[k] = fmaxf(vmax[k], tk_xform<XFORM>(ds_vec_elem<T>(w, e), a.mult, a.softcap));
        }
        tmax = fmaxf(tmax, vmax[k]);
      }
    }
    // the warp's m-th largest lane maximum (removed lanes drop to key 0, below every value)
    uint32_t key = ds_key32(ds_canon_zero(tmax)), kth = 0;
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

    // survivors: vectors whose maximum clears thr (a few percent) are queued per warp; the warp
    // then takes them 32 at a time, builds each one's 8-bit survivor mask from packed compares, and
    // drains the masks together (one survivor per lane per pass, one shared-memory atomic per pass)
    uint16_t* q = s_queue[warp];
    int qn = 0;
#pragma unroll
    for (int k = 0; k < TK_ROUNDS; ++k) {
      const bool cand = (tid + k * TK_THREADS < nv) && vmax[k] >= thr;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, cand);
      if (cand) q[qn + __popc(bal & below)] = uint16_t(tid + k * TK_THREADS);
      qn += __popc(bal);
    }
    __syncwarp();
    const __nv_bfloat162 thr2 = __float2bfloat162_rn(thr);   // exact for bf16 rows: thr is an element value
    for (int q0 = 0; q0 < qn; q0 += 32) {
      const int qi = q0 + lane;
      uint32_t m8 = 0;
      int i = 0;
      if (qi < qn) {
        i = q[qi];
        const uint4 w = sv[i];
        if constexpr (PACKED) {
          const uint32_t c0 = __hge2_mask(tk_b2(w.x), thr2), c1 = __hge2_mask(tk_b2(w.y), thr2);
          const uint32_t c2 = __hge2_mask(tk_b2(w.z), thr2), c3 = __hge2_mask(tk_b2(w.w), thr2);
          // bytes [e0 e1 e2 e3] and [e4 e5 e6 e7] (0x00 / 0xFF), then one bit per element
          const uint32_t w01 = __byte_perm(c0, c1, 0x6420), w23 = __byte_perm(c2, c3, 0x6420);
          uint32_t f = (w01 & 0x08040201u) | (w23 & 0x80402010u);
          f |= f >> 16;
          f |= f >> 8;
          m8 = f & 0xFFu;
        } else {
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            m8 |= (tk_xform<XFORM>(ds_vec_elem<T>(w, e), a.mult, a.softcap) >= thr) ? (1u << e) : 0u;
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
          const int e = __ffs(m8) - 1;
          m8 &= m8 - 1u;
          const float x = tk_xform<XFORM>(ds_load_elem<T>(reinterpret_cast<const T*>(sv + i) + e), a.mult, a.softcap);
          if (slot < TK_PART_CAP)
            s_keys[slot] = ds_key64(ds_canon_zero(x), uint32_t(g.head + (v0 + i) * EPV + e));
        }
      }
    }
    if (iextra >= 0 && xextra >= thr) {
      const uint32_t slot = atomicAdd(&s_n, 1u);
      if (slot < TK_PART_CAP) s_keys[slot] = ds_key64(ds_canon_zero(xextra), uint32_t(iextra));
    }
    __syncthreads();
    // the stage is free: refill it with the item TK_STAGES rounds ahead
    if (tid == 0) {
      const int next = item + TK_STAGES * int(gridDim.x);
      if (next < a.nitems) issue(next, s);
    }
    if (s_n > uint32_t(TK_PART_CAP)) {
      // the survivors overflow the slot: tighten thr to the part's own exact K'-th largest value
      const int64_t e0 = g.head + v0 * EPV, e1 = g.head + v1 * EPV;
      const int64_t x0 = (p == 0) ? 0 : (p == P - 1 ? g.tail0 : 0);
      const int64_t x1 = (p == 0) ? g.head : (p == P - 1 ? a.V : 0);
      thr = tk_part_refine<T, XFORM>(a, row, e0, e1, x0, x1, s_keys, s_red, &s_n);
      if (p == 0 && p == P - 1) {
        // a single-part row: its tail was not in [x0, x1); add those at or above thr
        if (iextra >= g.tail0 && xextra >= thr) {
          const uint32_t slot = atomicAdd(&s_n, 1u);
          if (slot < TK_PART_CAP) s_keys[slot] = ds_key64(ds_canon_zero(xextra), uint32_t(iextra));
        }
        __syncthreads();
      }
    }
    const uint32_t ns = s_n;
    const int64_t part = int64_t(row_id) * P + p;
    for (uint32_t i = tid; i < min(ns, uint32_t(TK_PART_CAP)); i += TK_THREADS) a.ws_keys[part * TK_PART_CAP + i] = s_keys[i];
    if (tid == 0) {
      a.ws_cnt[part] = ns;
      a.ws_thr[part] = thr;
    }
    __syncthreads();
  }
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

// One CTA per row merges the row's part survivors: max_p T_p bounds the row's K'-th value, the
// per-warp m-th largest thread maximum of the keys above it tightens the bound, and each key left
// is ranked by counting the keys above it.
template <typename T, bool XFORM>
__global__ void __launch_bounds__(TK_THREADS) topk_merge_kernel(const TopkArgs a) {
  constexpr bool PACKED = std::is_same<T, __nv_bfloat16>::value && !XFORM;
  __shared__ uint64_t s_keys[TK_MERGE_CAP];
  __shared__ uint64_t s_sel[TK_SEL_CAP];
  __shared__ unsigned long long s_wkey[TK_WARPS];
  __shared__ uint32_t s_red[2][TK_WARPS];
  __shared__ uint32_t s_off[65];
  __shared__ uint32_t s_n, s_n2;
  __shared__ int s_bad;
  __shared__ float s_rthr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int P = a.P;
  const uint32_t row_id = blockIdx.x;
  if (tid == 0) {
    float rthr = -INFINITY;
    uint32_t off = 0;
    int bad = 0;
    for (int q = 0; q < P; ++q) {
      const uint32_t c = a.ws_cnt[int64_t(row_id) * P + q];
      rthr = fmaxf(rthr, a.ws_thr[int64_t(row_id) * P + q]);
      bad |= c > uint32_t(TK_PART_CAP);
      s_off[q] = off;
      off += min(c, uint32_t(TK_PART_CAP));
    }
    s_off[P] = off;
    s_rthr = rthr;
    s_bad = bad;
    s_n = 0;
  }
  __syncthreads();
  const float rthr = s_rthr;
  {
    int q = 0;
    for (uint32_t gi = tid; gi < s_off[P]; gi += TK_THREADS) {
      while (gi >= s_off[q + 1]) ++q;
      const uint64_t k = a.ws_keys[(int64_t(row_id) * P + q) * TK_PART_CAP + (gi - s_off[q])];
      if (ds_key64_val(k) >= rthr) {
        const uint32_t slot = atomicAdd(&s_n, 1u);
        if (slot < TK_MERGE_CAP) s_keys[slot] = k;
      }
    }
  }
  __syncthreads();
  const uint32_t ngot = min(s_n, uint32_t(TK_MERGE_CAP));
  const TkRow g = tk_row<T>(a, row_id);
  const T* row = reinterpret_cast<const T*>(g.row);
  // a tighter row bound: the m-th largest per-thread maximum of the gathered keys in every warp
  // (m = ceil(K'/8)); 8 warps x m distinct keys are >= its minimum over the warps
  unsigned long long mx = 0;
  for (uint32_t i = tid; i < ngot; i += TK_THREADS) mx = max(mx, (unsigned long long)s_keys[i]);
  {
    const int m = (a.Kp + TK_WARPS - 1) / TK_WARPS;
    unsigned long long key = mx, kth = 0;
#pragma unroll
    for (int t = 0; t < (64 + TK_WARPS - 1) / TK_WARPS; ++t) {
      if (t < m) {
        kth = __reduce_max_sync(0xFFFFFFFFu, uint32_t(key >> 32)) == uint32_t(key >> 32) ? key : 0ull;
        kth = ds_warp_max_u64(kth);   // the largest full key among the lanes holding the top value
        const unsigned who = __ballot_sync(0xFFFFFFFFu, key == kth);
        if (lane == __ffs(who) - 1) key = 0;
      }
    }
    if (lane == 0) s_wkey[warp] = kth;
  }
  __syncthreads();
  unsigned long long bound = s_wkey[0];
#pragma unroll
  for (int w = 1; w < TK_WARPS; ++w) bound = min(bound, s_wkey[w]);
  // compact the keys >= bound (ballot per warp, one barrier), then each key's rank is the number
  // of compacted keys above it: rank < K' goes straight to its output slot
  uint32_t nsel = 0;
  if (!s_bad && s_n <= uint32_t(TK_MERGE_CAP)) {
    if (tid == 0) s_n2 = 0;
    __syncthreads();
    for (uint32_t i0 = 0; i0 < ngot; i0 += TK_THREADS) {
      const uint32_t i = i0 + tid;
      const uint64_t k = (i < ngot) ? s_keys[i] : 0;
      const bool keep = (i < ngot) && k >= bound;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
      uint32_t base = 0;
      if (lane == 0 && bal) base = atomicAdd(&s_n2, uint32_t(__popc(bal)));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (keep && base + __popc(bal & ((1u << lane) - 1u)) < uint32_t(TK_SEL_CAP))
        s_sel[base + __popc(bal & ((1u << lane) - 1u))] = k;
    }
    __syncthreads();
    nsel = s_n2;
  }
  if (!s_bad && s_n <= uint32_t(TK_MERGE_CAP) && nsel <= uint32_t(TK_SEL_CAP)) {
    for (uint32_t i = tid; i < nsel; i += TK_THREADS) {
      const uint64_t k = s_sel[i];
      uint32_t rank = 0;
      for (uint32_t j = 0; j < nsel; ++j) rank += (s_sel[j] > k) ? 1u : 0u;
      if (rank < uint32_t(a.Kp)) tk_emit(a, row_id, int(rank), k);
    }
  } else {
    // ties flooded the buffers: exact selection over the row itself, then sort
    const int nk = tk_row_exact<T, XFORM>(a, row, s_keys, s_red[0], &s_n);
    int n2 = 1;
    while (n2 < nk) n2 <<= 1;
    for (int i = nk + tid; i < n2; i += TK_THREADS) s_keys[i] = 0;
    __syncthreads();
    ds_block_sort_desc(s_keys, n2);
    if (tid < a.Kp) {
      if (tid >= nk) {                              // unreachable: >= K' keys always reach the sort
        ds_set_error(a.status, DSPARK_EINVAL);
        const int64_t o = int64_t(row_id) * a.Kp + tid;
        a.cand_draft[o] = -1;
        a.cand_tgt[o] = -1;
        a.cand_val[o] = -INFINITY;
      } else {
        tk_emit(a, row_id, tid, s_keys[tid]);
      }
    }
  }
}

size_t tk_align(size_t x) { return (x + 255) & ~size_t(255); }

struct TopkLayout {
  int P, nvp;
  size_t keys, cnt, thr, total;
};

TopkLayout tk_layout(int64_t rows, int64_t V, int elem_bytes) {
  TopkLayout L = {};
  const int64_t epv = 16 / elem_bytes;
  const int64_t nvec = V / epv + 1;
  L.P = int(std::max<int64_t>(1, ds_ceil_div(nvec, TK_STAGE_VEC)));
  L.nvp = int(ds_ceil_div(nvec, L.P));
  L.keys = tk_align(size_t(rows) * L.P * TK_PART_CAP * sizeof(uint64_t));
  L.cnt = tk_align(size_t(rows) * L.P * sizeof(uint32_t));
  L.thr = tk_align(size_t(rows) * L.P * sizeof(float));
  L.total = L.keys + L.cnt + L.thr;
  return L;
}

template <typename T, bool XFORM>
cudaError_t tk_launch(const TopkArgs& a, cudaStream_t stream) {
  auto kern = topk_stream_kernel<T, XFORM>;
  const size_t smem = size_t(TK_STAGES) * TK_STAGE_VEC * 16;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int grid = std::min(a.nitems, 2 * ds_num_sms());
  kern<<<unsigned(grid), TK_THREADS, smem, stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_merge_kernel<T, XFORM><<<unsigned(a.nitems / a.P), TK_THREADS, 0, stream>>>(a);
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
  DS_REQUIRE(L.P <= 64 && L.nvp <= TK_STAGE_VEC && rows * L.P <= 0x7FFFFFFF);
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
  a.nitems = int32_t(rows * L.P);
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
