// Scan core: affine pairs, their composition, lane/warp scans and the PTX
// helpers the kernels need (relaxed and acquire/release global accesses for
// the look-back, mbarrier, cp.async.bulk, L2 bulk prefetch, programmatic
// dependent launch, globaltimer).
//
// The recurrence (rl-triton technical summary, Methodology 1):
//   backward  A_t = alpha_t + beta_t * A_{t+1}
//   forward   e_t = alpha_t + beta_t * e_{t-1}
// A pair P = (m, c) stands for the affine map x -> c + m*x: the value of a
// segment's first (backward) or last (forward) step as a function of the
// value just outside it. One step is (beta_t, alpha_t). Composition follows
// the page's operator (alpha_B + beta_B*alpha_A, beta_A*beta_B), where B is
// the segment nearer the output's time origin (earlier in time for backward
// scans, later in time for forward ones):
//   outer ∘ inner = (m_o * m_i, c_o + m_o * c_i).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rlcs {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Pairs
// ---------------------------------------------------------------------------
struct FPair {
  float m, c;
};
// Integer pairs for the episodic prefix sum: m is 0 or 1 (reset or carry),
// c wraps modulo 2^32 like int32 two's-complement addition.
struct IPair {
  uint32_t m, c;
};

__device__ __forceinline__ FPair identity(FPair) { return {1.0f, 0.0f}; }
__device__ __forceinline__ IPair identity(IPair) { return {1u, 0u}; }

// outer ∘ inner: the map "apply inner first, then outer".
__device__ __forceinline__ FPair compose(FPair o, FPair i) {
  return {o.m * i.m, fmaf(o.m, i.c, o.c)};
}
__device__ __forceinline__ IPair compose(IPair o, IPair i) {
  return {o.m & i.m, o.c + (o.m ? i.c : 0u)};
}

__device__ __forceinline__ float apply(FPair p, float x) {
  return fmaf(p.m, x, p.c);
}
__device__ __forceinline__ uint32_t apply(IPair p, uint32_t x) {
  return p.c + (p.m ? x : 0u);
}

template <class P>
__device__ __forceinline__ P shfl_down(P p, int off) {
  P q;
  q.m = __shfl_down_sync(kFull, p.m, off);
  q.c = __shfl_down_sync(kFull, p.c, off);
  return q;
}
template <class P>
__device__ __forceinline__ P shfl_up(P p, int off) {
  P q;
  q.m = __shfl_up_sync(kFull, p.m, off);
  q.c = __shfl_up_sync(kFull, p.c, off);
  return q;
}
template <class P>
__device__ __forceinline__ P shfl_idx(P p, int src) {
  P q;
  q.m = __shfl_sync(kFull, p.m, src);
  q.c = __shfl_sync(kFull, p.c, src);
  return q;
}

// ---------------------------------------------------------------------------
// Warp scans over one pair per lane (lane order = time order).
// ---------------------------------------------------------------------------

// Backward (suffix) inclusive scan: lane l ends with P_l ∘ P_{l+1} ∘ ... ∘ P_31.
template <class P>
__device__ __forceinline__ P warp_suffix_scan(P p, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    P q = shfl_down(p, off);
    if (lane + off < 32) p = compose(p, q);
  }
  return p;
}

// Forward (prefix) inclusive scan: lane l ends with P_l ∘ P_{l-1} ∘ ... ∘ P_0.
template <class P>
__device__ __forceinline__ P warp_prefix_scan(P p, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    P q = shfl_up(p, off);
    if (lane >= off) p = compose(p, q);
  }
  return p;
}

// Ordered reduction of one pair per lane into lane 0:
// P_0 ∘ P_1 ∘ ... ∘ P_31 (lane 0 outermost). Other lanes hold partials.
template <class P>
__device__ __forceinline__ P warp_reduce_outer_first(P p) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    P q = shfl_down(p, off);
    p = compose(p, q);  // lanes past the end compose garbage they never use
  }
  return p;
}

// ---------------------------------------------------------------------------
// PTX helpers (sm_90+ forms, valid on sm_103a)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Strong (relaxed, gpu-scope) 64-bit accesses: single-copy atomic for a
// naturally aligned word, and served by L2, so never a stale L1 line.
__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t *p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t *p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// mbarrier in shared memory (one phase used per launch).
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
      "l"(src), "r"(bytes), "r"(b)
      : "memory");
}

// Bulk prefetch of [src, src+bytes) into L2 (no data returned to the thread).
// src 16-byte aligned, bytes a multiple of 16. L2 is the device's point of
// coherence, so prefetching a range that an earlier grid is still writing
// can never yield stale data: later loads see whatever L2 holds by then.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid in the stream
// (and its memory) before touching global memory; let the next grid start
// its launch early.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace rlcs
