// dspark_common.cuh - device helpers shared by the libdspark kernels (sm_103a).
//
// Status words, bf16 widening, order-preserving float keys, the Philox4x32-10 stream and
// its double uniform, the float32 softmax weight, warp reductions, and the inline-PTX
// wrappers for mbarriers and the tcgen05 tensor-core path.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"

#define DS_DEV __device__ __forceinline__

// Wall-clock bound of one mbarrier wait (2 s): far above any wait of a working kernel.
#define DS_WAIT_NS 2000000000ull

// ----------------------------------------------------------------------------------------
// status
// ----------------------------------------------------------------------------------------
// First error wins: a status word only ever moves from 0 to one nonzero code.
DS_DEV void ds_set_error(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------------------------------
// programmatic dependent launch: every library kernel lets the next kernel on its stream launch
// as soon as all of its own CTAs are running (trigger), and waits for the previous kernel to
// complete, with its memory visible, before it reads any buffer a library call writes and before
// it writes anything (wait). Before the wait a kernel reads only the caller's model inputs
// (logits, hidden states, head tables, d2t, row starts). Without a programmatic launch both are
// no-ops.
// ----------------------------------------------------------------------------------------
DS_DEV void ds_pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
DS_DEV void ds_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------------------------------
// element access
// ----------------------------------------------------------------------------------------
DS_DEV float ds_bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

template <typename T>
DS_DEV float ds_load_elem(const T* p);
template <>
DS_DEV float ds_load_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return ds_bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(p));
}
template <>
DS_DEV float ds_load_elem<float>(const float* p) { return *p; }

// Element e of a 16-byte vector holding bf16 (8 per vector) or float (4 per vector).
template <typename T>
DS_DEV float ds_vec_elem(const uint4& v, int e);
template <>
DS_DEV float ds_vec_elem<__nv_bfloat16>(const uint4& v, int e) {
  const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
  return (e & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
}
template <>
DS_DEV float ds_vec_elem<float>(const uint4& v, int e) {
  const uint32_t w = (e == 0) ? v.x : (e == 1) ? v.y : (e == 2) ? v.z : v.w;
  return __uint_as_float(w);
}

// Streaming 16-byte load (read once: evict-first in L1 and L2).
DS_DEV uint4 ds_ld_stream(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }

// ----------------------------------------------------------------------------------------
// ordering keys: larger float <-> larger unsigned key; -0.0 is folded onto +0.0 first
// ----------------------------------------------------------------------------------------
DS_DEV float ds_canon_zero(float x) { return __fadd_rn(x, 0.0f); }
DS_DEV uint32_t ds_key32(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
DS_DEV float ds_key32_to_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}
// (value descending, index ascending) as one descending 64-bit key
DS_DEV uint64_t ds_key64(float x, uint32_t idx) {
  return (uint64_t(ds_key32(x)) << 32) | uint64_t(0xFFFFFFFFu - idx);
}
DS_DEV uint32_t ds_key64_idx(uint64_t k) { return 0xFFFFFFFFu - uint32_t(k & 0xFFFFFFFFull); }
DS_DEV float ds_key64_val(uint64_t k) { return ds_key32_to_float(uint32_t(k >> 32)); }

// ----------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) and the 53-bit double uniform
// ----------------------------------------------------------------------------------------
struct DsU4 {
  uint32_t x, y, z, w;
};

DS_DEV DsU4 ds_philox4x32_10(DsU4 c, uint32_t k0, uint32_t k1) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(M0, c.x), lo0 = M0 * c.x;
    const uint32_t hi1 = __umulhi(M1, c.z), lo1 = M1 * c.z;
    c = DsU4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
    k0 += W0;
    k1 += W1;
  }
  return c;
}

enum : uint32_t { DS_PURPOSE_DRAFT = 0, DS_PURPOSE_ACCEPT = 1, DS_PURPOSE_RESIDUAL = 2 };

// The 53-bit integer m of the uniform u = m * 2^-53 for (seed, step, position, purpose, draw):
// m = (x0 >> 5) * 2^26 + (x1 >> 6) from the first two Philox outputs.
DS_DEV uint64_t ds_uniform_bits(uint64_t seed, uint64_t step, uint32_t position, uint32_t purpose,
                                uint32_t draw = 0) {
  const DsU4 c{uint32_t(step), position, (purpose << 20) + draw, uint32_t(step >> 32)};
  const DsU4 o = ds_philox4x32_10(c, uint32_t(seed), uint32_t(seed >> 32));
  return (uint64_t(o.x >> 5) << 26) | uint64_t(o.y >> 6);
}
// Double uniform in [0, 1) for (seed, step, position, purpose, draw).
DS_DEV double ds_uniform(uint64_t seed, uint64_t step, uint32_t position, uint32_t purpose,
                         uint32_t draw = 0) {
  return double(ds_uniform_bits(seed, step, position, purpose, draw)) * (1.0 / 9007199254740992.0);
}

// ----------------------------------------------------------------------------------------
// softmax weight of an exponent d = z - zmax <= 0, in float32 (flush below -64):
//   t = fl32(d log2 e), n = rint(t), f = t - n (exact), w = 2^n * P(f),
//   P = degree-7 Taylor polynomial of 2^f = e^(f ln 2), coefficients (ln 2)^k / k!
//   rounded to float32, evaluated with correctly rounded FMAs.
// Every step is one correctly rounded float32 operation, so the CPU reference computes the
// same bits.
// ----------------------------------------------------------------------------------------
DS_DEV float ds_weight(float d) {
  if (!(d >= -64.0f)) return 0.0f;
  const float t = __fmul_rn(d, 0x1.715476p+0f);   // 1 / ln 2
  const float n = rintf(t);
  const float f = __fsub_rn(t, n);
  float p = 0x1.ffcbfcp-17f;                       // (ln 2)^7 / 7!
  p = __fmaf_rn(p, f, 0x1.430912p-13f);            // (ln 2)^6 / 6!
  p = __fmaf_rn(p, f, 0x1.5d87fep-10f);            // (ln 2)^5 / 5!
  p = __fmaf_rn(p, f, 0x1.3b2ab6p-7f);             // (ln 2)^4 / 4!
  p = __fmaf_rn(p, f, 0x1.c6b08ep-5f);             // (ln 2)^3 / 3!
  p = __fmaf_rn(p, f, 0x1.ebfbe0p-3f);             // (ln 2)^2 / 2!
  p = __fmaf_rn(p, f, 0x1.62e430p-1f);             // ln 2
  p = __fmaf_rn(p, f, 1.0f);
  const int ni = int(n);                           // -93 <= n <= 0: 2^n is a normal float
  return __fmul_rn(p, __int_as_float((ni + 127) << 23));
}

// ---- packed float32 pairs (sm_100 family f32x2): each lane is one IEEE round-to-nearest
// operation, so a packed evaluation gives the same bits as two scalar ones. There is no packed
// multiply here: a packed product feeding a packed add can come out fused (unrounded), so a
// rounded product is an FMA with a zero addend ----
DS_DEV uint64_t ds_f2(float lo, float hi) {
  return (uint64_t(__float_as_uint(hi)) << 32) | uint64_t(__float_as_uint(lo));
}
DS_DEV float ds_f2lo(uint64_t v) { return __uint_as_float(uint32_t(v)); }
DS_DEV float ds_f2hi(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }
DS_DEV uint64_t ds_fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
DS_DEV uint64_t ds_add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
DS_DEV uint64_t ds_sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ds_weight of two exponents at once, with the same bits: t = fl(d / ln 2) is an explicit FMA
// with a zero addend (the product's rounding; a packed multiply feeding the packed add below could
// come out fused, unrounded), rint(t) is taken by adding and removing 1.5 * 2^23 (round to nearest,
// ties to even, for |t| < 2^22), and 2^n * P(f) adds n to the exponent field of P(f) (P(f) in
// [0.70, 1.42] and n >= -93, so the result is a normal float); the integer n sits in the low
// mantissa bits of t + 1.5 * 2^23, so (bits << 23) is n << 23.
DS_DEV float2 ds_weight2(float d0, float d1) {
  const uint64_t M = ds_f2(12582912.0f, 12582912.0f);
  const uint64_t t = ds_fma2(ds_f2(d0, d1), ds_f2(0x1.715476p+0f, 0x1.715476p+0f), ds_f2(0.0f, 0.0f));
  const uint64_t tm = ds_add2(t, M);
  const uint64_t f = ds_sub2(t, ds_sub2(tm, M));
  uint64_t p = ds_f2(0x1.ffcbfcp-17f, 0x1.ffcbfcp-17f);
  p = ds_fma2(p, f, ds_f2(0x1.430912p-13f, 0x1.430912p-13f));
  p = ds_fma2(p, f, ds_f2(0x1.5d87fep-10f, 0x1.5d87fep-10f));
  p = ds_fma2(p, f, ds_f2(0x1.3b2ab6p-7f, 0x1.3b2ab6p-7f));
  p = ds_fma2(p, f, ds_f2(0x1.c6b08ep-5f, 0x1.c6b08ep-5f));
  p = ds_fma2(p, f, ds_f2(0x1.ebfbe0p-3f, 0x1.ebfbe0p-3f));
  p = ds_fma2(p, f, ds_f2(0x1.62e430p-1f, 0x1.62e430p-1f));
  p = ds_fma2(p, f, ds_f2(1.0f, 1.0f));
  const uint32_t w0 = uint32_t(p) + (uint32_t(tm) << 23);
  const uint32_t w1 = uint32_t(p >> 32) + (uint32_t(tm >> 32) << 23);
  return make_float2((d0 >= -64.0f) ? __uint_as_float(w0) : 0.0f, (d1 >= -64.0f) ? __uint_as_float(w1) : 0.0f);
}

// z = s / T in float32 (the identity for T == 1)
DS_DEV float ds_temper(float s, float T) { return (T == 1.0f) ? s : __fdiv_rn(s, T); }
// the same with the T == 1 case decided at compile time (no division is evaluated for it)
template <bool TONE>
DS_DEV float ds_temper_t(float s, float T) {
  if constexpr (TONE) return s;
  else return __fdiv_rn(s, T);
}

// ----------------------------------------------------------------------------------------
// warp helpers
// ----------------------------------------------------------------------------------------
DS_DEV float ds_warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
DS_DEV double ds_warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
DS_DEV float ds_warp_sumf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
DS_DEV uint64_t ds_warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = (w > v) ? w : v;
  }
  return v;
}

// ----------------------------------------------------------------------------------------
// gate gamma = sigmoid(h . g) of one hidden row, whole block: float32 partial dots per thread
// (16-byte loads, four pairs in flight, when both rows are 16-byte aligned), summed in double;
// s_red holds one float per warp.
// ----------------------------------------------------------------------------------------
template <typename HT>
DS_DEV float ds_block_gate(const HT* h, const HT* g, int H, float* s_red) {
  constexpr int EPV = 16 / sizeof(HT);
  constexpr int U = 4;
  float acc = 0.0f;
  int k0 = 0;
  if (((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(g)) & 15u) == 0) {
    const int nv = H / EPV;
    const uint4* hv = reinterpret_cast<const uint4*>(h);
    const uint4* gv = reinterpret_cast<const uint4*>(g);
    for (int v0 = threadIdx.x; v0 < nv; v0 += U * int(blockDim.x)) {
      uint4 x[U], y[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * int(blockDim.x);
        if (v < nv) {
          x[u] = __ldg(hv + v);
          y[u] = __ldg(gv + v);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (v0 + u * int(blockDim.x) < nv) {
#pragma unroll
          for (int e = 0; e < EPV; ++e) acc = __fmaf_rn(ds_vec_elem<HT>(x[u], e), ds_vec_elem<HT>(y[u], e), acc);
        }
      }
    }
    k0 = nv * EPV;
  }
  for (int k = k0 + int(threadIdx.x); k < H; k += blockDim.x) acc = __fmaf_rn(ds_load_elem<HT>(h + k), ds_load_elem<HT>(g + k), acc);
  acc = ds_warp_sumf(acc);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = acc;
  __syncthreads();
  double dot = 0.0;
  for (int w = 0; w < int(blockDim.x >> 5); ++w) dot += double(s_red[w]);
  __syncthreads();
  return float(1.0 / (1.0 + exp(-dot)));
}

// ----------------------------------------------------------------------------------------
// shared-memory bitonic sort of n2 (power of two) 64-bit keys, descending; whole block
// ----------------------------------------------------------------------------------------
DS_DEV void ds_block_sort_desc(uint64_t* s, int n2) {
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = s[i], b = s[ixj];
          const bool desc = ((i & k) == 0);
          if (desc ? (a < b) : (a > b)) {
            s[i] = b;
            s[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// ----------------------------------------------------------------------------------------
// mbarrier + tcgen05 inline PTX (sm_100 family). Every wait is bounded.
// ----------------------------------------------------------------------------------------
DS_DEV uint32_t ds_smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

DS_DEV void ds_mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(ds_smem_addr(bar)), "r"(count)
               : "memory");
}

DS_DEV uint64_t ds_globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of an mbarrier to complete; gives up after `limit` polls or about
// DS_WAIT_NS nanoseconds, whichever comes first (a poll may suspend the thread for a while).
DS_DEV bool ds_mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
  const uint32_t a = ds_smem_addr(bar);
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 63u) == 63u) {
      const uint64_t t = ds_globaltimer();
      if (t0 == 0) t0 = t;
      else if (t - t0 > DS_WAIT_NS) return false;
    }
  }
  return false;
}

// ds_mbar_wait that also gives up as soon as *abort becomes nonzero (another role of the CTA
// stopped).
DS_DEV bool ds_mbar_wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t limit, const int* abort) {
  const uint32_t a = ds_smem_addr(bar);
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 63u) == 63u) {
      if (*reinterpret_cast<const volatile int*>(abort)) return false;
      const uint64_t t = ds_globaltimer();
      if (t0 == 0) t0 = t;
      else if (t - t0 > DS_WAIT_NS) return false;
    }
  }
  return false;
}

// Arrive on an mbarrier and add `bytes` to the transaction count its phase waits for.
DS_DEV void ds_mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(ds_smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Bulk asynchronous copy global -> shared (16-byte aligned, size a multiple of 16) that
// completes `bytes` of the mbarrier's transaction count.
DS_DEV void ds_bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          ds_smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(ds_smem_addr(bar))
      : "memory");
}

// --- thread-block clusters ---
// Address of the same shared-memory location in CTA `rank` of the cluster (shared::cluster window).
DS_DEV uint32_t ds_mapa(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

// Bulk copy from this CTA's shared memory to another CTA's shared memory in the cluster
// (16-byte aligned, size a multiple of 16), completing `bytes` on the destination's mbarrier.
DS_DEV void ds_bulk_s2s_cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes, uint32_t mbar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(mbar_cluster)
      : "memory");
}

// Waits until this thread's bulk copies have finished reading their sources.
DS_DEV void ds_bulk_wait_read_all() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Makes an mbarrier initialisation visible to the other CTAs of the cluster.
DS_DEV void ds_fence_mbar_init_cluster() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

DS_DEV void ds_fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMEM allocation: one full warp executes these.
DS_DEV void ds_tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   ds_smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
DS_DEV void ds_tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

DS_DEV void ds_tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
DS_DEV void ds_tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate); one thread.
DS_DEV void ds_umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread complete.
DS_DEV void ds_umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          ds_smem_addr(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle layout
// (8-row x 128-byte atoms, atoms 1024 bytes apart along M/N).
DS_DEV uint64_t ds_smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr & 0x3FFFFu) >> 4);        // start address
  d |= uint64_t(1) << 16;                        // leading byte offset (unused with swizzle)
  d |= uint64_t(1024 >> 4) << 32;                // stride byte offset: 8 rows x 128 B
  d |= uint64_t(1) << 46;                        // descriptor version
  d |= uint64_t(2) << 61;                        // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t ds_idesc_bf16_f32(int M, int N) {
  return (1u << 4)                    // D format: f32
         | (1u << 7)                  // A format: bf16
         | (1u << 10)                 // B format: bf16
         | (uint32_t(N >> 3) << 17)   // N / 8
         | (uint32_t(M >> 4) << 24);  // M / 16
}

// 32 lanes x 32 bits, 64 consecutive columns into 64 registers (one warp).
DS_DEV void ds_tmem_ld_32x32b_x64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
        "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
        "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
        "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]),
        "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]),
        "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 bits, 32 consecutive columns into 32 registers (one warp).
DS_DEV void ds_tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Ampere-style 16-byte async copy global -> shared (any 16-byte-aligned destination).
DS_DEV void ds_cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(ds_smem_addr(smem_dst)),
               "l"(gmem_src)
               : "memory");
}
// 2-D tiled TMA load of box (x = inner coordinate in elements, y = row) into shared memory,
// completing its bytes on an mbarrier, with an L2 cache policy. x * element size must be a
// multiple of 16 bytes; rows outside the tensor read as zero.
DS_DEV void ds_tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(ds_smem_addr(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(ds_smem_addr(bar)), "l"(pol)
      : "memory");
}

// An L2 policy that keeps lines (evict last), for data read again by later launches.
DS_DEV uint64_t ds_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// An L2 policy that lets lines go first (evict first), for data read once.
DS_DEV uint64_t ds_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
DS_DEV void ds_cp_async16_hint(void* smem_dst, const void* gmem_src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(ds_smem_addr(smem_dst)),
               "l"(gmem_src), "l"(pol)
               : "memory");
}
// Arrive on an mbarrier once this thread's earlier cp.async copies have landed (counted in its
// expected arrivals).
DS_DEV void ds_cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(ds_smem_addr(bar)) : "memory");
}
DS_DEV void ds_mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ds_smem_addr(bar)) : "memory");
}
// Named barrier over `count` threads (a multiple of 32).
DS_DEV void ds_named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

DS_DEV void ds_cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Bounded-wait limits (polls); a wait that runs out reports DSPARK_ETIMEOUT.
#define DS_WAIT_LIMIT (1u << 26)
