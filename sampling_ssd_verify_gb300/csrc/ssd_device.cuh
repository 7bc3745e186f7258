// ssd_device.cuh -- device helpers: inline-PTX wrappers for mbarriers and
// bulk copies, bounded waits, Philox-4x32-10, exponent and reduction helpers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_internal.cuh"

namespace ssd {

// ---- shared-memory addressing, mbarriers, bulk copies ---------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread for up to `ns` nanoseconds while the
// phase is incomplete (the thread resumes when the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete, for at most
// kWaitLimitNs.  On time-out the error flag is raised (shared flag and the
// caller's device status) and false is returned; the caller then carries on
// without the data so that every thread still reaches every barrier.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* s_err,
                                          int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (*s_err) return false;
    if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      *s_err = 1;
      if (status) atomicOr(status, SSD_DEV_TIMEOUT);
      return false;
    }
  }
}

// A flag another CTA of the launch sets once: release store / acquire load
// at GPU scope.
__device__ __forceinline__ void flag_release(int* f) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(f), "r"(1) : "memory");
}
__device__ __forceinline__ int flag_acquire(const int* f) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}

// Wait (bounded, like mbar_wait) until the counter reaches `target`; false
// on a timeout or when the CTA has already met an error.  One thread.
__device__ __forceinline__ bool count_wait(const int* f, int target, volatile int* s_err,
                                           int32_t* status) {
  if (flag_acquire(f) >= target) return true;
  const unsigned long long t0 = global_ns();
  while (true) {
    if (*s_err) return false;
    __nanosleep(256);
    if (flag_acquire(f) >= target) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      *s_err = 1;
      if (status) atomicOr(status, SSD_DEV_TIMEOUT);
      return false;
    }
  }
}

// Wait (bounded) until the flag is set.
__device__ __forceinline__ bool flag_wait(const int* f, volatile int* s_err, int32_t* status) {
  return count_wait(f, 1, s_err, status);
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
// dst, src and bytes must be multiples of 16.  The streamed rows are read
// once (or re-read soon after), so their L2 lines are marked evict-first:
// they displace one another rather than the kernel's code, its counters and
// its per-row results, which the rarer paths (draws, decisions) would
// otherwise fetch again from HBM.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "{.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], pol;}" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// ---- thread-block clusters ---------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives, then waits; the
// release/acquire pair orders the shared (local and remote) and global
// accesses made before the barrier with those made after it.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The split form: every CTA arrives at launch and waits before its first
// store to another CTA's shared memory, so that no store reaches a CTA of the
// cluster that has not started.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// The address of *local in CTA `rank`'s shared memory (shared::cluster window).
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(ra)
               : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  return ra;
}
// Stores into another CTA's shared memory (addresses from cluster_addr).
__device__ __forceinline__ void st_cluster_f64(double* local, uint32_t rank, double v) {
  asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(cluster_addr(local, rank)), "d"(v)
               : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t ra, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}


// Relaxed / acquire loads and release stores of 32-bit words that other
// CTAs of the launch write (draw-queue counters and entries).
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* f) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* f) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* f) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_s32(int* f, int v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_s32(int* f, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

// Atomic add / or with acquire-release semantics at GPU scope: the thread's
// earlier writes (and those ordered before them) are published with the
// update, and the writes published by earlier updates are visible after it.
__device__ __forceinline__ int atom_add_acq_rel(int* f, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(f), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_or_acq_rel(unsigned long long* f,
                                                              unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(f), "l"(v)
               : "memory");
  return old;
}

// Warp-wide maximum of a float (redux.sync .f32, sm_100 family); -inf is an
// ordinary value, NaN inputs are not expected.
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Named barrier over the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// ---- optional bounds checks (compile with -DSSD_CHECKS) ---------------------------
// A failed check records (code, a, b, block, thread) once in the workspace's
// debug record, counts the failure and skips the guarded access.
#ifdef SSD_CHECKS
__device__ __forceinline__ bool ssd_chk(bool ok, unsigned long long* dbg, int code, long long a,
                                        long long b) {
  if (ok) return true;
  if (dbg != nullptr) {
    if (atomicCAS(dbg, 0ull, (unsigned long long)code) == 0ull) {
      dbg[1] = (unsigned long long)a;
      dbg[2] = (unsigned long long)b;
      dbg[3] = blockIdx.x;
      dbg[4] = threadIdx.x;
    }
    atomicAdd(dbg + 5, 1ull);
  }
  return false;
}
#define SSD_CHK(ok, dbg, code, a, b) ::ssd::ssd_chk((ok), (dbg), (code), (long long)(a), (long long)(b))
#else
#define SSD_CHK(ok, dbg, code, a, b) true
#endif

__device__ __forceinline__ bool in_range(uintptr_t a0, uintptr_t a1, const char* lo,
                                         const char* hi) {
  return a0 >= (uintptr_t)lo && a1 <= (uintptr_t)hi && a0 <= a1;
}

// ---- element access ---------------------------------------------------------------
template <int DT>
struct Elem;
template <>
struct Elem<0> {  // bf16
  static constexpr int kSize = 2;
  static constexpr int kVec = 8;
  __device__ __forceinline__ static float load(const void* base, int64_t i) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + i);
    return __uint_as_float(((uint32_t)h) << 16);
  }
  __device__ __forceinline__ static float load_cg(const void* base, int64_t i) {
    const unsigned short h = __ldcg(reinterpret_cast<const unsigned short*>(base) + i);
    return __uint_as_float(((uint32_t)h) << 16);
  }
  __device__ __forceinline__ static float smem(const void* base, int i) {
    const unsigned short h = reinterpret_cast<const unsigned short*>(base)[i];
    return __uint_as_float(((uint32_t)h) << 16);
  }
  __device__ __forceinline__ static void unpack(const uint4 v, float* x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
};
template <>
struct Elem<1> {  // fp32
  static constexpr int kSize = 4;
  static constexpr int kVec = 4;
  __device__ __forceinline__ static float load(const void* base, int64_t i) {
    return __ldg(reinterpret_cast<const float*>(base) + i);
  }
  __device__ __forceinline__ static float load_cg(const void* base, int64_t i) {
    return __ldcg(reinterpret_cast<const float*>(base) + i);
  }
  __device__ __forceinline__ static float smem(const void* base, int i) {
    return reinterpret_cast<const float*>(base)[i];
  }
  __device__ __forceinline__ static void unpack(const uint4 v, float* x) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
};

// A lane's run of VEC elements from y as a 16-byte vector: one load when the
// row is aligned and the run lies inside it, else element by element (zero
// bits beyond V).
template <int DT>
__device__ __forceinline__ uint4 load_run(const char* row, int y, int V, bool vec) {
  constexpr int VEC = Elem<DT>::kVec;
  if (vec && y + VEC <= V) return __ldg(reinterpret_cast<const uint4*>(row) + y / VEC);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if constexpr (DT == 0) {
    const unsigned short* h = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
    for (int k = 0; k < VEC; ++k)
      if (y + k < V) w[k >> 1] |= (uint32_t)__ldg(h + y + k) << (16 * (k & 1));
  } else {
    const uint32_t* f = reinterpret_cast<const uint32_t*>(row);
#pragma unroll
    for (int k = 0; k < VEC; ++k)
      if (y + k < V) w[k] = __ldg(f + y + k);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Element k (runtime index) of a 16-byte vector, without spilling the vector.
template <int DT>
__device__ __forceinline__ float vec_elem(const uint4 v, int k) {
  if constexpr (DT == 0) {
    const uint32_t w = (k < 4) ? ((k < 2) ? v.x : v.y) : ((k < 6) ? v.z : v.w);
    return __uint_as_float((k & 1) ? (w & 0xFFFF0000u) : (w << 16));
  } else {
    const uint32_t w = (k < 2) ? ((k == 0) ? v.x : v.y) : ((k == 2) ? v.z : v.w);
    return __uint_as_float(w);
  }
}

__device__ __forceinline__ const char* row_ptr(const void* base, int64_t row, int64_t stride,
                                               int esize) {
  return reinterpret_cast<const char*>(base) + row * stride * esize;
}

// ---- arithmetic helpers -------------------------------------------------------------
// 2^x with the SFU (ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats as one 64-bit register pair (the operands of the packed f32x2
// instructions) and back.
__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// max(a, b, c) in one instruction (three-operand max.f32 of sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Error-free sum of two floats (Knuth): a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// Compensated pair addition (hi, lo) += (bhi, blo).
__device__ __forceinline__ void pair_add(float& hi, float& lo, float bhi, float blo) {
  float s, e;
  two_sum(hi, bhi, s, e);
  e += lo + blo;
  hi = s + e;
  lo = e - (hi - s);
}

// Scale a compensated pair by f (keeps the product's rounding error).
__device__ __forceinline__ void pair_scale(float& hi, float& lo, float f) {
  const float p = hi * f;
  const float perr = fmaf(hi, f, -p);
  lo = fmaf(lo, f, perr);
  hi = p;
}

// ---- Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) ---------------------------------
// Round: (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
// key += (0x9E3779B9, 0xBB67AE85) between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    k.x += 0x9E3779B9u;
    k.y += 0xBB67AE85u;
  }
  return c;
}

// u = (out0 >> 8) * 2^-24 for key = seed, counter = (c0, c1, stream, round).
__device__ __forceinline__ double uniform24(uint64_t seed, uint32_t c0, uint32_t c1,
                                            uint32_t stream, uint32_t round) {
  const uint4 o = philox4x32_10(make_uint4(c0, c1, stream, round),
                                make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
  return (double)(o.x >> 8) * (1.0 / 16777216.0);
}

// ---- candidate lists (top-F by raw logit, ties to the lower index) -----------------------
__device__ __forceinline__ bool cand_before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// Warp-wide merge of (max, compensated sum) partials.  Each lane holds
// (m, mc = fl(m*c), hi, lo) with the sum taken relative to mc; returns the
// warp maximum M and the sum relative to fl(M*c) in every lane.
__device__ __forceinline__ void warp_softmax_merge(float m, float mc, float hi, float lo, float c,
                                                   float& M, float& MC, float& Shi,
                                                   float& Slo) {
  M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  MC = __fmul_rn(M, c);
  float h = hi, l = lo;
  if (m == __int_as_float(0xff800000)) {
    h = 0.f;
    l = 0.f;
  } else if (mc != MC) {
    pair_scale(h, l, exp2f(mc - MC));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, h, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    pair_add(h, l, h2, l2);
  }
  Shi = h;
  Slo = l;
}

}  // namespace ssd
