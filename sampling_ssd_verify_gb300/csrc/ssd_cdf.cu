// ssd_cdf.cu -- the inverse-CDF draw over one vocabulary row per group.
//
// After the streaming pass every group (a verified sequence, or a Saguaro
// branch row) has its draw parameters: the bonus weight
//   w(y) = (p_k(y) - q'_k(y))^+   when a draft was rejected at k < K,
//   w(y) = p_K(y)                 when every draft was accepted
// ([SD-7.3] §7.3.3 for the residual, §7.3.2 for the all-accepted bonus), or
// the Saguaro draft distribution w(y) = q'(y) for a continuation draw
// ([SSD-note] §"Saguaro 优化二：Saguaro 采样").  The token drawn is the
// smallest y with sum_{y'<=y} w(y') > u * Z, Z = sum_y w(y).
//
// Work is split into 512-element units over (group, unit); one persistent
// CTA per SM streams its share of units of the one or two rows a group needs
// through a bulk-copy ring, each consumer warp reduces one unit to its
// weight sum, and the last CTA to finish a group (atomic arrival counter)
// locates the unit holding u*Z by a prefix over the unit sums and scans that
// unit in vocabulary order.
//
// Sources: [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈";
// [SD-7.3] "7.3 Speculative Decoding：投机采样加速".

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_device.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr float kPosInf = INFINITY;

// One row half of a stage: where element y lives (shared memory or global).
struct Half {
  const char* row;   // row base (global)
  int ei0, ei1;      // elements [ei0, ei1) are in shared memory
  const char* sm;    // shared memory copy of element ei0
};

template <int DT>
__device__ __forceinline__ float fetch(const Half& h, int y, const CdfParams& p, bool is_t) {
  if (y >= h.ei0 && y < h.ei1) {
    if (!SSD_CHK((y - h.ei0) * Elem<DT>::kSize < kUnitsPerStageB * kUnitB * Elem<DT>::kSize,
                 p.dbg, 24, y, h.ei0))
      return 0.f;
    return Elem<DT>::smem(h.sm, y - h.ei0);
  }
  const uintptr_t a = (uintptr_t)(h.row + (int64_t)y * Elem<DT>::kSize);
  if (!SSD_CHK(in_range(a, a + Elem<DT>::kSize, is_t ? p.t_lo : p.d_lo, is_t ? p.t_hi : p.d_hi),
               p.dbg, 22, y, (int64_t)(a - (uintptr_t)(is_t ? p.t_lo : p.d_lo))))
    return 0.f;
  return Elem<DT>::load(h.row, y);
}

// The draw weight of token y given its target logit zt and draft logit zd.
__device__ __forceinline__ float weight(const GroupParams& gp, float c, int y, float zt,
                                        float zd) {
  float p = 0.f;
  if (gp.use_t) p = ex2(fmaf(zt, c, -gp.mc_t)) * gp.inv_st;
  if (!gp.use_d) return p;
  const bool inS = zd > gp.theta || (zd == gp.theta && y <= gp.itheta);
  const float q = ex2(fmaf(zd, c, -gp.mc_d)) * (inS ? gp.scale_in : gp.scale_out);
  return gp.sign_d > 0 ? q : fmaxf(p - q, 0.f);
}

template <int DT>
__device__ __forceinline__ float weight_global(const CdfParams& p, const GroupParams& gp,
                                               const char* rt, const char* rd, int y) {
  const uintptr_t at = (uintptr_t)(rt + (int64_t)y * Elem<DT>::kSize);
  const uintptr_t ad = (uintptr_t)(rd + (int64_t)y * Elem<DT>::kSize);
  const float zt = (gp.use_t && SSD_CHK(in_range(at, at + Elem<DT>::kSize, p.t_lo, p.t_hi), p.dbg,
                                         26, y, gp.row_t)) ? Elem<DT>::load(rt, y) : 0.f;
  const float zd = (gp.use_d && SSD_CHK(in_range(ad, ad + Elem<DT>::kSize, p.d_lo, p.d_hi), p.dbg,
                                         27, y, gp.row_d)) ? Elem<DT>::load(rd, y) : 0.f;
  return weight(gp, p.c, y, zt, zd);
}

__device__ __forceinline__ double warp_incl_scan(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Scan [e0, e1) in vocabulary order for the first y with run + cumsum > rem.
// Returns -1 if none; *lastpos gets the last y with positive weight.
template <int DT>
__device__ int scan_range(const CdfParams& p, const GroupParams& gp, const char* rt,
                          const char* rd, int e0, int e1, double rem, double* run_io,
                          int* lastpos) {
  const int lane = threadIdx.x & 31;
  double run = *run_io;
  int last = -1;
  int t = -1;
  for (int base = e0; base < e1; base += 32) {
    const int y = base + lane;
    const float w = y < e1 ? weight_global<DT>(p, gp, rt, rd, y) : 0.f;
    if (w > 0.f) last = y;
    const double incl = warp_incl_scan((double)w);
    const unsigned m = __ballot_sync(0xffffffffu, y < e1 && run + incl > rem);
    if (m) {
      t = base + __ffs(m) - 1;
      break;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
  *run_io = run;
  *lastpos = last;
  return t;
}

// Full two-pass draw over the whole row by one warp (degenerate residual).
template <int DT>
__device__ int full_row_draw(const CdfParams& p, const GroupParams& gp, const char* rt,
                             const char* rd, double* Zout) {
  const int lane = threadIdx.x & 31;
  double loc = 0.0;
  for (int y = lane; y < p.V; y += 32) loc += (double)weight_global<DT>(p, gp, rt, rd, y);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) loc += __shfl_xor_sync(0xffffffffu, loc, off);
  const double Z = loc;
  *Zout = Z;
  double run = 0.0;
  int last = -1;
  int t = scan_range<DT>(p, gp, rt, rd, 0, p.V, gp.u * Z, &run, &last);
  if (t < 0) t = last >= 0 ? last : 0;
  return t;
}

// The draw for group g (warp 0 of the last CTA to finish the group).
template <int DT>
__device__ void group_draw(const CdfParams& p, int64_t g) {
  const int lane = threadIdx.x & 31;
  if (!SSD_CHK(g < p.groups, p.dbg, 20, g, p.groups)) return;
  const GroupParams gp = p.gp[g];
  const int esz = Elem<DT>::kSize;
  const char* rt = gp.use_t ? row_ptr(p.tgt, gp.row_t, p.t_stride, esz) : nullptr;
  const char* rd = gp.use_d ? row_ptr(p.dft, gp.row_d, p.d_stride, esz) : nullptr;
  const float* sub = p.subsum + g * p.nsub;
  const int per = (p.nsub + 31) / 32;
  const int lo = min(lane * per, p.nsub);
  const int hi = min(lo + per, p.nsub);
  double loc = 0.0;
  for (int u = lo; u < hi; ++u)
    if (SSD_CHK(g * p.nsub + u < (int64_t)p.groups * p.nsub, p.dbg, 23, g, u))
      loc += (double)__ldcg(sub + u);
  const double incl = warp_incl_scan(loc);
  double Z = __shfl_sync(0xffffffffu, incl, 31);
  int t;
  float wt;
  if (!(Z > 1e-30)) {
    // The residual vanished in rounding (exact arithmetic forbids it after a
    // rejection): draw the bonus from p_k instead and report it.
    if (lane == 0 && p.status) atomicOr(p.status, SSD_DEV_ZERO_RESIDUAL);
    GroupParams gp2 = gp;
    gp2.use_d = 0;
    gp2.use_t = gp.use_t;
    if (!gp2.use_t) {  // Saguaro rows always have Z ~ 1; keep a defined result
      gp2.use_d = 1;
      gp2.sign_d = 1;
    }
    t = full_row_draw<DT>(p, gp2, rt, rd, &Z);
    wt = weight_global<DT>(p, gp2, rt, rd, t);
  } else {
    const double thr = gp.u * Z;
    const unsigned m = __ballot_sync(0xffffffffu, incl > thr && lo < hi);
    int unit = -1;
    double before = 0.0;
    if (m) {
      const int L = __ffs(m) - 1;
      if (lane == L) {
        double run = incl - loc;
        for (int u = lo; u < hi; ++u) {
          const double nx = run + (double)__ldcg(sub + u);
          if (nx > thr) {
            unit = u;
            before = run;
            break;
          }
          run = nx;
        }
        if (unit < 0) {  // rounding: the lane's own running sum never exceeded thr;
                         // fall back to the last positive weight of its range
          for (int u = hi - 1; u >= lo; --u)
            if (__ldcg(sub + u) > 0.f) {
              unit = u;
              break;
            }
          before = -INFINITY;
        }
      }
      unit = __shfl_sync(0xffffffffu, unit, L);
      before = __shfl_sync(0xffffffffu, before, L);
    }
    if (unit < 0) {  // no prefix exceeded u*Z: take the last unit with weight
      int cand = -1;
      for (int u = hi - 1; u >= lo; --u)
        if (__ldcg(sub + u) > 0.f) {
          cand = u;
          break;
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        cand = max(cand, __shfl_xor_sync(0xffffffffu, cand, off));
      unit = cand >= 0 ? cand : p.nsub - 1;
      before = -INFINITY;  // no index qualifies: the last positive weight is taken
    }
    const int e0 = unit * kUnitB;
    const int e1 = min(e0 + kUnitB, p.V);
    double run = 0.0;
    int last = -1;
    t = scan_range<DT>(p, gp, rt, rd, e0, e1, thr - before, &run, &last);
    if (t < 0) t = last >= 0 ? last : e0;
    wt = weight_global<DT>(p, gp, rt, rd, t);
  }
  if (lane != 0) return;
  if (!SSD_CHK(g < p.groups && t >= 0 && t < p.V, p.dbg, 25, g, t)) return;
  p.out_token[g] = t;
  if (p.out_mass) p.out_mass[g] = (float)Z;
  if (p.out_qprime) p.out_qprime[g] = (float)((double)wt / Z);
  if (p.out_guess) {
    const RowResult* rr = p.rowres + g * p.rpg + p.nt;
    int n = 0;
    for (int k = 0; k < kMaxTopK && n < p.F; ++k) {
      const int i = __ldcg(&rr->ti[k]);
      if (i < 0 || i == t) continue;
      p.out_guess[g * p.F + n] = i;
      ++n;
    }
    for (; n < p.F; ++n) p.out_guess[g * p.F + n] = -1;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 1) cdf_kernel(const __grid_constant__ CdfParams p) {
  constexpr int ES = Elem<DT>::kSize;
  constexpr int HALF = kUnitsPerStageB * kUnitB * ES;
  constexpr int STAGE = 2 * HALF;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStagesB * STAGE);
  uint64_t* empty = full + kStagesB;
  __shared__ int s_err;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t u_begin = (int64_t)blockIdx.x * p.upc;
  const int64_t u_end = min(u_begin + p.upc, p.total_units);
  if (u_begin >= u_end) return;

  if (tid == 0) {
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    s_err = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      int n = 0;
      for (int64_t u = u_begin; u < u_end;) {
        const int64_t g = u / p.nsub;
        const int64_t uge = min((g + 1) * (int64_t)p.nsub, u_end);
        if (!SSD_CHK(g < p.groups, p.dbg, 20, g, p.groups)) break;
        const GroupParams& gp = p.gp[g];
        const int use_t = gp.use_t, use_d = gp.use_d;
        const char* rt = use_t ? row_ptr(p.tgt, gp.row_t, p.t_stride, ES) : nullptr;
        const char* rd = use_d ? row_ptr(p.dft, gp.row_d, p.d_stride, ES) : nullptr;
        for (int64_t un = 0; u < uge; u = un) {
          un = min(u + (int64_t)kUnitsPerStageB, uge);
          const int e0 = (int)((u - g * p.nsub) * kUnitB);
          const int e1 = (int)min((int64_t)p.V, (un - g * p.nsub) * kUnitB);
          const int slot = n % kStagesB;
          if (n >= kStagesB) mbar_wait(empty + slot, ((n / kStagesB) - 1) & 1, &s_err, p.status);
          uintptr_t a0[2] = {0, 0}, a1[2] = {0, 0};
          uint32_t bytes = 0;
          for (int h = 0; h < 2; ++h) {
            const char* r = h == 0 ? rt : rd;
            if (r == nullptr) continue;
            const uintptr_t b0 = (uintptr_t)(r + (int64_t)e0 * ES);
            const uintptr_t b1 = (uintptr_t)(r + (int64_t)e1 * ES);
            a0[h] = (b0 + 15) & ~(uintptr_t)15;
            a1[h] = b1 & ~(uintptr_t)15;
            if (a1[h] > a0[h]) bytes += (uint32_t)(a1[h] - a0[h]);
          }
          bool srcok = true;
          for (int h = 0; h < 2; ++h)
            if (a1[h] > a0[h])
              srcok &= SSD_CHK(in_range(a0[h], a1[h], h == 0 ? p.t_lo : p.d_lo,
                                        h == 0 ? p.t_hi : p.d_hi), p.dbg, 21, a0[h], h);
          if (bytes > 0 && !s_err && srcok) {
            mbar_arrive_expect_tx(full + slot, bytes);
            for (int h = 0; h < 2; ++h)
              if (a1[h] > a0[h])
                bulk_g2s(ring + slot * STAGE + h * HALF, reinterpret_cast<const void*>(a0[h]),
                         (uint32_t)(a1[h] - a0[h]), full + slot);
          } else {
            mbar_arrive(full + slot);
          }
          ++n;
        }
      }
      for (int q = max(0, n - kStagesB); q < n; ++q)
        mbar_wait(full + (q % kStagesB), (q / kStagesB) & 1, &s_err, p.status);
    }
    return;
  }

  // ---------------- consumers ----------------
  int n = 0;
  for (int64_t u = u_begin; u < u_end;) {
    const int64_t g = u / p.nsub;
    const int64_t uge = min((g + 1) * (int64_t)p.nsub, u_end);
    const int64_t ug0 = u;
    const GroupParams gp = p.gp[g];
    const char* rt = gp.use_t ? row_ptr(p.tgt, gp.row_t, p.t_stride, ES) : nullptr;
    const char* rd = gp.use_d ? row_ptr(p.dft, gp.row_d, p.d_stride, ES) : nullptr;
    for (int64_t un = 0; u < uge; u = un) {
      un = min(u + (int64_t)kUnitsPerStageB, uge);
      const int e0 = (int)((u - g * p.nsub) * kUnitB);
      const int e1 = (int)min((int64_t)p.V, (un - g * p.nsub) * kUnitB);
      const int slot = n % kStagesB;
      mbar_wait(full + slot, (n / kStagesB) & 1, &s_err, p.status);
      Half ht, hd;
      for (int h = 0; h < 2; ++h) {
        Half& H = h == 0 ? ht : hd;
        const char* r = h == 0 ? rt : rd;
        H.row = r;
        H.sm = reinterpret_cast<const char*>(ring + slot * STAGE + h * HALF);
        H.ei0 = H.ei1 = e0;
        if (r != nullptr) {
          const uintptr_t b0 = (uintptr_t)(r + (int64_t)e0 * ES);
          const uintptr_t b1 = (uintptr_t)(r + (int64_t)e1 * ES);
          const uintptr_t A0 = (b0 + 15) & ~(uintptr_t)15;
          const uintptr_t A1 = b1 & ~(uintptr_t)15;
          if (A1 > A0) {
            H.ei0 = e0 + (int)((A0 - b0) / ES);
            H.ei1 = H.ei0 + (int)((A1 - A0) / ES);
          }
        }
      }
      const int64_t uu = u + warp;
      if (uu < un) {
        const int ue0 = (int)((uu - g * p.nsub) * kUnitB);
        const int ue1 = min(ue0 + kUnitB, p.V);
        float s = 0.f;
#pragma unroll 4
        for (int m = 0; m < kUnitB / 32; ++m) {
          const int y = ue0 + lane + 32 * m;
          if (y < ue1) {
            const float zt = gp.use_t ? fetch<DT>(ht, y, p, true) : 0.f;
            const float zd = gp.use_d ? fetch<DT>(hd, y, p, false) : 0.f;
            s += weight(gp, p.c, y, zt, zd);
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0 && SSD_CHK(uu < (int64_t)p.groups * p.nsub, p.dbg, 23, uu, g)) {
          p.subsum[g * p.nsub + (uu - g * p.nsub)] = s;
          __threadfence();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + slot);
      ++n;
    }
    // this CTA's units of group g are summed: arrival
    consumer_sync();
    if (warp == 0) {
      int last = 0;
      if (lane == 0) {
        __threadfence();
        last = SSD_CHK(g < p.groups, p.dbg, 28, g, p.groups)
                   ? atomicAdd(p.cnt + g, (int)(uge - ug0)) + (int)(uge - ug0) == p.nsub
                   : 0;
        if (last) __threadfence();
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) group_draw<DT>(p, g);
    }
  }
}

}  // namespace

int cdf_smem_bytes(int dtype) {
  const int es = dtype == SSD_BF16 ? 2 : 4;
  return kStagesB * 2 * kUnitsPerStageB * kUnitB * es + 2 * kStagesB * (int)sizeof(uint64_t);
}

cudaError_t launch_cdf(const CdfParams& p, int dtype, int grid, cudaStream_t s) {
  const int smem = cdf_smem_bytes(dtype);
  cudaError_t e;
  if (dtype == SSD_BF16) {
    e = cudaFuncSetAttribute(cdf_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cdf_kernel<0><<<grid, kThreads, smem, s>>>(p);
  } else {
    e = cudaFuncSetAttribute(cdf_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cdf_kernel<1><<<grid, kThreads, smem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace ssd
