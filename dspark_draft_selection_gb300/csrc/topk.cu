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
// Design (one thread-block cluster of C CTAs per row; the logits are read from HBM once):
//  1. The row's 16-byte vectors are dealt round-robin to the C*512 threads of the cluster and
//     held in registers (coalesced streaming loads, <= 8 vectors per thread).
//  2. Every thread's maximum is one element of the row. Each CTA finds the m-th largest of its
//     512 thread maxima, m = ceil(K'/C): C*m >= K' distinct elements are >= each CTA's value,
//     so the minimum T over the cluster (exchanged through distributed shared memory) is a
//     lower bound of the row's K'-th largest value.
//  3. Elements >= T survive (typically ~2K' of them) and are appended, as 64-bit keys
//     (value, then lower index first), to the leader CTA's shared memory.
//  4. The leader sorts the survivors (bitonic) and writes the first K'. If ties flood the
//     survivor buffer, the leader finds the exact K'-th key by bisection over the row instead.
#include <cooperative_groups.h>

#include "dspark_common.cuh"
#include "host_common.h"

namespace cg = cooperative_groups;

namespace {

constexpr int TK_THREADS = 512;
constexpr int TK_MAXV = 8;      // 16-byte vectors held per thread
constexpr int TK_CAP = 2048;    // survivor capacity of the leader CTA
constexpr int TK_MAXC = 16;

struct TopkArgs {
  const void* logits;
  int64_t V, ld;
  const int64_t* row_start;
  int32_t B, Kp, C;
  float mult, softcap;
  const int64_t* d2t;
  int64_t V_t;
  int32_t* cand_draft;
  int32_t* cand_tgt;
  float* cand_val;
  int32_t* status;
};

template <bool XFORM>
DS_DEV float tk_xform(float x, float mult, float softcap) {
  if (XFORM) {
    if (mult != 1.0f) x = __fmul_rn(x, mult);
    if (softcap > 0.0f) x = __fmul_rn(softcap, tanhf(__fdiv_rn(x, softcap)));
  }
  return x;
}

// Count of row elements whose 64-bit key is >= kmin (whole block; slow path only).
template <typename T, bool XFORM>
DS_DEV uint32_t tk_block_count_ge(const T* row, int64_t V, float mult, float softcap,
                                  uint64_t kmin, uint32_t* s_acc) {
  uint32_t c = 0;
  for (int64_t i = threadIdx.x; i < V; i += blockDim.x) {
    const float x = ds_canon_zero(tk_xform<XFORM>(ds_load_elem<T>(row + i), mult, softcap));
    c += (ds_key64(x, uint32_t(i)) >= kmin) ? 1u : 0u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
  __syncthreads();
  if (threadIdx.x == 0) *s_acc = 0;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) atomicAdd(s_acc, c);
  __syncthreads();
  return *s_acc;
}

template <typename T, bool XFORM>
__global__ void __launch_bounds__(TK_THREADS, 2) topk_cluster_kernel(const TopkArgs a) {
  constexpr int EPV = 16 / sizeof(T);
  __shared__ uint64_t s_keys[TK_CAP];
  __shared__ uint32_t s_tc[TK_MAXC];
  __shared__ uint32_t s_count;
  __shared__ uint32_t s_t;
  __shared__ uint32_t s_acc;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = a.C;
  const int crank = int(cluster.block_rank());
  const int64_t row_id = blockIdx.x / C;             // r * B + j
  const int64_t r = row_id / a.B, j = row_id % a.B;
  const int64_t prow = a.row_start ? a.row_start[r] + j : row_id;
  const T* row = reinterpret_cast<const T*>(a.logits) + prow * a.ld;
  const int64_t V = a.V;

  // split the row into a scalar head (until 16-byte alignment), full vectors, scalar tail
  const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
  int64_t head = int64_t(((16u - (addr & 15u)) & 15u) / sizeof(T));
  if (head > V) head = V;
  const int64_t nvec = (V - head) / EPV;
  const int64_t tail0 = head + nvec * EPV;
  const int64_t nextra = head + (V - tail0);
  const uint4* vbase = reinterpret_cast<const uint4*>(row + head);
  const int64_t gthr = int64_t(crank) * TK_THREADS + threadIdx.x;
  const int64_t stride = int64_t(C) * TK_THREADS;

  uint4 buf[TK_MAXV];
#pragma unroll
  for (int k = 0; k < TK_MAXV; ++k) {
    const int64_t v = gthr + k * stride;
    if (v < nvec) buf[k] = ds_ld_stream(vbase + v);
  }
  float xextra = -INFINITY;
  int64_t iextra = -1;
  if (gthr < nextra) {
    iextra = (gthr < head) ? gthr : tail0 + (gthr - head);
    xextra = tk_xform<XFORM>(ds_load_elem<T>(row + iextra), a.mult, a.softcap);
  }
  if (crank == 0 && threadIdx.x == 0) s_count = 0;

  // pass 1: this thread's maximum
  float tmax = xextra;
#pragma unroll
  for (int k = 0; k < TK_MAXV; ++k) {
    if (gthr + k * stride < nvec) {
#pragma unroll
      for (int e = 0; e < EPV; ++e)
        tmax = fmaxf(tmax, tk_xform<XFORM>(ds_vec_elem<T>(buf[k], e), a.mult, a.softcap));
    }
  }
  // this CTA's m-th largest thread maximum, by bisection on the ordering key
  const int m = (a.Kp + C - 1) / C;
  const uint32_t key = ds_key32(ds_canon_zero(tmax));
  uint32_t res = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = res | (1u << b);
    if (__syncthreads_count(key >= cand) >= m) res = cand;
  }
  uint32_t* leader_tc = cluster.map_shared_rank(s_tc, 0);
  if (threadIdx.x == 0) leader_tc[crank] = res;
  cluster.sync();
  if (threadIdx.x == 0) {
    uint32_t t = 0xFFFFFFFFu;
    for (int c = 0; c < C; ++c) t = min(t, leader_tc[c]);
    s_t = t;
  }
  __syncthreads();
  const uint32_t tkey = s_t;
  const float thr = (tkey <= ds_key32(-INFINITY)) ? -INFINITY : ds_key32_to_float(tkey);

  // pass 2: survivors >= thr go to the leader as (value, lower index first) keys
  uint32_t* leader_count = cluster.map_shared_rank(&s_count, 0);
  uint64_t* leader_keys = cluster.map_shared_rank(s_keys, 0);
#pragma unroll
  for (int k = 0; k < TK_MAXV; ++k) {
    const int64_t v = gthr + k * stride;
    if (v < nvec) {
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float x = tk_xform<XFORM>(ds_vec_elem<T>(buf[k], e), a.mult, a.softcap);
        if (x >= thr) {
          const uint32_t slot = atomicAdd(leader_count, 1u);
          if (slot < TK_CAP) leader_keys[slot] = ds_key64(ds_canon_zero(x), uint32_t(head + v * EPV + e));
        }
      }
    }
  }
  if (iextra >= 0 && xextra >= thr) {
    const uint32_t slot = atomicAdd(leader_count, 1u);
    if (slot < TK_CAP) leader_keys[slot] = ds_key64(ds_canon_zero(xextra), uint32_t(iextra));
  }
  cluster.sync();
  if (crank != 0) return;

  // leader: exact order of the survivors
  uint32_t n = s_count;
  if (n > TK_CAP) {
    // slow path (ties flooded the buffer): bisection for the exact K'-th key over the row
    uint64_t kres = 0;
    for (int b = 63; b >= 0; --b) {
      const uint64_t cand = kres | (1ull << b);
      if (tk_block_count_ge<T, XFORM>(row, V, a.mult, a.softcap, cand, &s_acc) >= uint32_t(a.Kp))
        kres = cand;
    }
    if (threadIdx.x == 0) s_count = 0;
    __syncthreads();
    for (int64_t i = threadIdx.x; i < V; i += blockDim.x) {
      const float x = ds_canon_zero(tk_xform<XFORM>(ds_load_elem<T>(row + i), a.mult, a.softcap));
      const uint64_t k64 = ds_key64(x, uint32_t(i));
      if (k64 >= kres) {
        const uint32_t slot = atomicAdd(&s_count, 1u);
        if (slot < TK_CAP) s_keys[slot] = k64;
      }
    }
    __syncthreads();
    n = min(s_count, uint32_t(TK_CAP));
  }
  int n2 = 1;
  while (n2 < int(n)) n2 <<= 1;
  for (int i = int(n) + threadIdx.x; i < n2; i += blockDim.x) s_keys[i] = 0;
  __syncthreads();
  ds_block_sort_desc(s_keys, n2);
  if (threadIdx.x < a.Kp) {
    const uint64_t k64 = s_keys[threadIdx.x];
    const uint32_t idx = ds_key64_idx(k64);
    int64_t tgt = idx;
    if (a.d2t) {
      tgt = int64_t(idx) + a.d2t[idx];
      if (tgt < 0 || tgt >= a.V_t) {
        ds_set_error(a.status, DSPARK_ERANGE);
        tgt = -1;
      }
    }
    const int64_t o = row_id * a.Kp + threadIdx.x;
    a.cand_draft[o] = int32_t(idx);
    a.cand_tgt[o] = int32_t(tgt);
    a.cand_val[o] = ds_key64_val(k64);
  }
}

template <typename T, bool XFORM>
cudaError_t tk_launch(const TopkArgs& a, int64_t rows, cudaStream_t stream) {
  auto kern = topk_cluster_kernel<T, XFORM>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(rows * a.C), 1, 1);
  cfg.blockDim = dim3(TK_THREADS, 1, 1);
  cfg.dynamicSmemBytes = 0;
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

// Smallest power-of-two cluster whose threads hold a row within TK_MAXV vectors each.
extern "C" int dspark_internal_topk_cluster_size(int64_t V, int32_t elem_bytes) {
  const int64_t epv = 16 / elem_bytes;
  const int64_t need = ds_ceil_div(V / epv + 2, int64_t(TK_THREADS) * TK_MAXV);
  int C = 1;
  while (C < need) C <<= 1;
  return C <= TK_MAXC ? C : -1;
}

extern "C" dspark_status dspark_topk(const void* logits, dspark_dtype dtype, int64_t R, int32_t B,
                                     int64_t V_d, int64_t ld, const int64_t* row_start, int32_t K,
                                     float mult, float softcap, const int64_t* d2t, int64_t V_t,
                                     int32_t* cand_draft, int32_t* cand_tgt, float* cand_val,
                                     int32_t* dev_status, dspark_stream_t stream) {
  DS_REQUIRE(ds_dtype_ok(dtype));
  DS_REQUIRE(R >= 0 && B >= 1 && V_d >= 1 && ld >= V_d && K >= 1 && K <= 64);
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
  a.C = dspark_internal_topk_cluster_size(V_d, ds_dtype_size(dtype));
  DS_REQUIRE(a.C > 0);
  a.mult = mult;
  a.softcap = softcap;
  a.d2t = d2t;
  a.V_t = V_t;
  a.cand_draft = cand_draft;
  a.cand_tgt = cand_tgt;
  a.cand_val = cand_val;
  a.status = dev_status;
  const bool xform = (mult != 1.0f) || (softcap > 0.0f);
  const int64_t rows = R * B;
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
