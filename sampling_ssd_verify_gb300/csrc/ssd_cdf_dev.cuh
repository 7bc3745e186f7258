// ssd_cdf_dev.cuh -- device code of the inverse-CDF draw, which the
// streaming kernel (ssd_stream_kernel.cuh) runs after the rows in the same launch.
//
// The bonus weight of a verified sequence is w(y) = (p_k(y) - q'_k(y))^+
// after a rejection at k < K and w(y) = p_K(y) when every draft was accepted
// ([SD-7.3] §7.3.3 for the residual, §7.3.2 for the all-accepted bonus); a
// Saguaro continuation draws from w(y) = q'(y) ([SSD-note] §"Saguaro
// 优化二：Saguaro 采样").  The token drawn is the smallest y with
// sum_{y'<=y} w(y') > u * Z, Z = sum_y w(y).
//
// Work is split into kUnitB-element units; the sum of the weights of each
// unit is stored, and the chunk that completes a group runs its draw: the
// unit holding u*Z by a prefix over the unit sums, then a vocabulary-order
// scan of that unit.
//
// Sources: [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈";
// [SD-7.3] "7.3 Speculative Decoding：投机采样加速".
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_cache_dev.cuh"
#include "ssd_device.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

// One row half of a stage: where element y lives (shared memory or global).
struct Half {
  const char* row;   // row base (global)
  int ei0, ei1;      // elements [ei0, ei1) are in shared memory
  const char* sm;    // shared memory copy of element ei0
};

template <int DT>
__device__ __forceinline__ float fetch(const Half& h, int y, const CdfParams& p, bool is_t,
                                       int half) {
  if (y >= h.ei0 && y < h.ei1) {
    if (!SSD_CHK((y - h.ei0) * Elem<DT>::kSize < half, p.dbg, 24, y, h.ei0))
      return 0.f;
    return Elem<DT>::smem(h.sm, y - h.ei0);
  }
  const uintptr_t a = (uintptr_t)(h.row + (int64_t)y * Elem<DT>::kSize);
  if (!SSD_CHK(in_range(a, a + Elem<DT>::kSize, is_t ? p.t_lo : p.d_lo, is_t ? p.t_hi : p.d_hi),
               p.dbg, 22, y, (int64_t)(a - (uintptr_t)(is_t ? p.t_lo : p.d_lo))))
    return 0.f;
  return Elem<DT>::load(h.row, y);
}

// A group's draw parameters, read from L2: another CTA of the same launch
// may have written them.
__device__ __forceinline__ GroupParams load_gp(const GroupParams* src) {
  static_assert(sizeof(GroupParams) % 8 == 0, "GroupParams is read as 8-byte words");
  GroupParams gp;
  const unsigned long long* a = reinterpret_cast<const unsigned long long*>(src);
  unsigned long long* b = reinterpret_cast<unsigned long long*>(&gp);
#pragma unroll
  for (int i = 0; i < (int)(sizeof(GroupParams) / 8); ++i) b[i] = __ldcg(a + i);
  return gp;
}

// The draw weight of token y given its target logit zt and draft logit zd.
// The three kinds of draw, as separate formulas so that unit loops can be
// specialised; weight() dispatches.  kind_of() classifies a group.
enum DrawKind : int { kResidual = 0, kTarget = 1, kSaguaro = 2 };

__device__ __forceinline__ int kind_of(const GroupParams& gp) {
  return gp.use_d ? (gp.sign_d > 0 ? kSaguaro : kResidual) : kTarget;
}

template <bool HAS_S>
__device__ __forceinline__ float q_scale(const GroupParams& gp, int y, float zd) {
  if (!HAS_S) return gp.scale_out;
  const bool inS = zd > gp.theta || (zd == gp.theta && y <= gp.itheta);
  return inS ? gp.scale_in : gp.scale_out;
}

template <int KIND, bool HAS_S>
__device__ __forceinline__ float weight_k(const GroupParams& gp, float c, int y, float zt,
                                          float zd) {
  if (KIND == kTarget) return ex2(fmaf(zt, c, -gp.mc_t)) * gp.inv_st;
  const float q = ex2(fmaf(zd, c, -gp.mc_d)) * q_scale<HAS_S>(gp, y, zd);
  if (KIND == kSaguaro) return q;
  const float pt = ex2(fmaf(zt, c, -gp.mc_t)) * gp.inv_st;
  return fmaxf(pt - q, 0.f);
}

__device__ __forceinline__ float weight(const GroupParams& gp, float c, int y, float zt,
                                        float zd) {
  const bool has_s = gp.theta != INFINITY;
  switch (kind_of(gp)) {
    case kTarget: return weight_k<kTarget, false>(gp, c, y, zt, zd);
    case kSaguaro:
      return has_s ? weight_k<kSaguaro, true>(gp, c, y, zt, zd)
                   : weight_k<kSaguaro, false>(gp, c, y, zt, zd);
    default:
      return has_s ? weight_k<kResidual, true>(gp, c, y, zt, zd)
                   : weight_k<kResidual, false>(gp, c, y, zt, zd);
  }
}

// The weights of 16 consecutive tokens y0 .. y0+15 (0 from e1 on), with one
// dispatch on the kind of draw for the whole run.
template <int KIND, bool HAS_S>
__device__ __forceinline__ void weights16_k(const GroupParams& gp, float c, int y0, int e1,
                                            const float* zt, const float* zd, float* w) {
#pragma unroll
  for (int k = 0; k < 16; ++k)
    w[k] = y0 + k < e1 ? weight_k<KIND, HAS_S>(gp, c, y0 + k, zt[k], zd[k]) : 0.f;
}

__device__ __forceinline__ void weights16(const GroupParams& gp, float c, int y0, int e1,
                                          const float* zt, const float* zd, float* w) {
  const bool has_s = gp.theta != INFINITY;
  switch (kind_of(gp)) {
    case kTarget: weights16_k<kTarget, false>(gp, c, y0, e1, zt, zd, w); break;
    case kSaguaro:
      if (has_s) weights16_k<kSaguaro, true>(gp, c, y0, e1, zt, zd, w);
      else weights16_k<kSaguaro, false>(gp, c, y0, e1, zt, zd, w);
      break;
    default:
      if (has_s) weights16_k<kResidual, true>(gp, c, y0, e1, zt, zd, w);
      else weights16_k<kResidual, false>(gp, c, y0, e1, zt, zd, w);
  }
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
  return weight(gp, gp.c, y, zt, zd);
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
__device__ __noinline__ int full_row_draw(const CdfParams& p, const GroupParams& gp, const char* rt,
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

// ---- double-float arithmetic for the draw ------------------------------------------
// A non-negative value hi + lo held as a normalised pair of floats (|lo| at
// most half an ulp of hi): about 48 significant bits at any magnitude, on the
// fp32 pipes.  The draw's sums, prefixes and comparisons use it; sums of
// non-negative terms only, so the two-sum based add stays accurate.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF df_of(float x) { return DF{x, 0.f}; }

__device__ __forceinline__ DF df_add(DF a, DF b) {
  pair_add(a.hi, a.lo, b.hi, b.lo);
  return a;
}

// a * u for 0 <= u < 1 (exact product of the high part, then normalised).
__device__ __forceinline__ DF df_scale(DF a, float u) {
  const float p = a.hi * u;
  const float e = fmaf(a.lo, u, fmaf(a.hi, u, -p));
  DF r;
  r.hi = p + e;
  r.lo = e - (r.hi - p);
  return r;
}

// a > b for normalised pairs.
__device__ __forceinline__ bool df_gt(DF a, DF b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ DF df_shfl(DF v, int src) {
  return DF{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

__device__ __forceinline__ DF df_shfl_up(DF v, int off) {
  return DF{__shfl_up_sync(0xffffffffu, v.hi, off), __shfl_up_sync(0xffffffffu, v.lo, off)};
}

// Inclusive warp prefix sum over the first `width` lanes (a power of two;
// lanes beyond take part with whatever they hold and are ignored).
__device__ __forceinline__ DF df_warp_scan(DF v, int width = 32) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    if (off >= width) break;
    const DF o = df_shfl_up(v, off);
    if (lane >= off) v = df_add(v, o);
  }
  return v;
}

// Pairwise sum of 16 floats (depth 4).
__device__ __forceinline__ DF df_sum16(const float* x) {
  DF t[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float s, e;
    two_sum(x[2 * k], x[2 * k + 1], s, e);
    t[k].hi = s + e;
    t[k].lo = e - (t[k].hi - s);
  }
#pragma unroll
  for (int w = 4; w > 0; w >>= 1)
#pragma unroll
    for (int k = 0; k < w; ++k) t[k] = df_add(t[k], t[k + w]);
  return t[0];
}

// Lane L's 16 values x[0..15], in order: the first k with x[k] > 0 and
// base + x[0] + ... + x[k] > thr, found with lanes 0..15 holding one value
// each (a shuffle per value, then a 16-lane scan).  Returns k, or -1 if no
// prefix exceeds thr; *before gets base + x[0] + ... + x[k-1], and *lastpos
// the last k with x[k] > 0 (-1 if none).  Called by all 32 lanes.
__device__ __forceinline__ int lane_search16(const float* x, int L, DF base, DF thr, DF* before,
                                             int* lastpos) {
  const int lane = threadIdx.x & 31;
  float mine = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float o = __shfl_sync(0xffffffffu, x[k], L);
    if (lane == k) mine = o;
  }
  const DF incl = df_warp_scan(df_of(lane < 16 ? mine : 0.f), 16);
  const DF up = df_shfl_up(incl, 1);  // every lane takes part in the shuffle
  const DF excl = lane == 0 ? DF{0.f, 0.f} : up;
  const unsigned pos = __ballot_sync(0xffffffffu, lane < 16 && mine > 0.f);
  const unsigned hit =
      __ballot_sync(0xffffffffu, lane < 16 && mine > 0.f && df_gt(df_add(base, incl), thr));
  *lastpos = pos ? 31 - __clz(pos) : -1;
  const int k = hit ? __ffs(hit) - 1 : -1;
  *before = df_add(base, df_shfl(excl, k >= 0 ? k : 0));
  return k;
}

// Sixteen consecutive logits of row `r` starting at y0 (< e1), vectorised
// when the address is 16-byte aligned and the run is complete.
template <int DT>
__device__ __forceinline__ void load16(const CdfParams& p, const char* r, bool is_t, int y0,
                                       int e1, float* z) {
  constexpr int ES = Elem<DT>::kSize;
  constexpr int VEC = Elem<DT>::kVec;
  const uintptr_t a = (uintptr_t)(r + (int64_t)y0 * ES);
  if (y0 + 16 <= e1 && (a & 15) == 0 &&
      SSD_CHK(in_range(a, a + 16 * ES, is_t ? p.t_lo : p.d_lo, is_t ? p.t_hi : p.d_hi), p.dbg, 29,
              y0, e1)) {
    const uint4* v = reinterpret_cast<const uint4*>(a);
#pragma unroll
    for (int k = 0; k < 16 / VEC; ++k) Elem<DT>::unpack(__ldg(v + k), z + k * VEC);
  } else {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int y = y0 + k;
      const uintptr_t ay = (uintptr_t)(r + (int64_t)y * ES);
      (void)ay;  // read by the bounds-checked build only
      z[k] = (y < e1 && SSD_CHK(in_range(ay, ay + ES, is_t ? p.t_lo : p.d_lo,
                                         is_t ? p.t_hi : p.d_hi), p.dbg, 29, y, e1))
                 ? Elem<DT>::load(r, y) : 0.f;
    }
  }
}

// Saguaro row g's guesses: its top list minus the drawn token t, truncated
// to the row's fan-out, padded with -1 to p.F columns.  One thread.
__device__ __forceinline__ void write_guesses(const CdfParams& p, int64_t g, const RowResult* rr,
                                              int t) {
  const int F = p.F_rows ? min(max(__ldg(p.F_rows + g), 0), p.F) : p.F;
  int n = 0;
  for (int k = 0; k < kMaxTopK && n < F; ++k) {
    const int i = __ldcg(&rr->ti[k]);
    if (i < 0 || i == t) continue;
    p.out_guess[g * p.F + n] = i;
    ++n;
  }
  for (; n < p.F; ++n) p.out_guess[g * p.F + n] = -1;
}

// The draw for group g (one warp of the CTA that completes the group).
// 1. Z = sum of the group's unit sums (each lane holds 16 units at once).
// 2. The unit holding u*Z: lane prefix + warp scan, then inside the lane
//    that crosses u*Z.
// 3. Inside that unit: each lane takes 16 consecutive tokens, lane prefix +
//    warp scan in vocabulary order; the first token whose cumulative weight
//    exceeds u*Z is the draw.
// Sums and prefixes are double-float pairs (see DF); a row whose weights
// vanish in rounding falls back to the fp64 two-pass draw.
template <int DT>
__device__ __noinline__ void group_draw(const CdfParams& p, int64_t g) {
  constexpr int R = 16;  // unit sums per lane per round
  const int lane = threadIdx.x & 31;
  if (!SSD_CHK(g < p.groups, p.dbg, 20, g, p.groups)) return;
  const float* sub = p.subsum + g * p.nsub;
  const int nsub = p.nsub;
  const int rounds = (nsub + 32 * R - 1) / (32 * R);
  float v[R];
  auto load_round = [&](int rnd) {
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int u = rnd * 32 * R + lane * R + k;
      v[k] = (u < nsub && SSD_CHK(g * nsub + u < (int64_t)p.groups * nsub, p.dbg, 23, g, u))
                 ? __ldcg(sub + u) : 0.f;
    }
  };
  load_round(0);  // in flight together with the group's parameters
  const GroupParams gp = load_gp(p.gp + g);
  if (no_draw(gp)) return;  // the group's epilogue wrote its outputs
  const int esz = Elem<DT>::kSize;
  const char* rt = gp.use_t ? row_ptr(p.tgt, gp.row_t, p.t_stride, esz) : nullptr;
  const char* rd = gp.use_d ? row_ptr(p.dft, gp.row_d, p.d_stride, esz) : nullptr;
  DF loc0 = df_sum16(v);  // round 0's lane sum, reused by the search
  DF Zl = loc0;
  for (int rnd = 1; rnd < rounds; ++rnd) {
    load_round(rnd);
    Zl = df_add(Zl, df_sum16(v));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const DF o{__shfl_xor_sync(0xffffffffu, Zl.hi, off), __shfl_xor_sync(0xffffffffu, Zl.lo, off)};
    Zl = df_add(Zl, o);
  }
  const DF Z = Zl;  // the same in every lane (the pairwise adds commute)
  double Zd = (double)Z.hi + (double)Z.lo;
  int t;
  float wt;
  if (!(Zd > 1e-30)) {
    // The residual vanished in rounding (exact arithmetic forbids it after a
    // rejection): draw the bonus from p_k instead and report it.
    if (lane == 0 && p.status) atomicOr(p.status, SSD_DEV_ZERO_RESIDUAL);
    GroupParams gp2 = gp;
    gp2.use_d = 0;
    if (!gp2.use_t) {  // Saguaro rows always have Z ~ 1; keep a defined result
      gp2.use_d = 1;
      gp2.sign_d = 1;
    }
    t = full_row_draw<DT>(p, gp2, rt, rd, &Zd);
    wt = weight_global<DT>(p, gp2, rt, rd, t);
  } else {
    // u has 24 fraction bits: exact as a float
    const DF thr = df_scale(Z, (float)gp.u);
    int unit = -1;
    DF before{0.f, 0.f};
    bool any_before = true;  // false: take the last positive weight
    DF run{0.f, 0.f};
    for (int rnd = 0; rnd < rounds && unit < 0; ++rnd) {
      DF loc = loc0;
      if (rounds > 1) {  // v holds the last round's sums after Z
        load_round(rnd);
        if (rnd > 0) loc = df_sum16(v);
      }
      const DF incl = df_warp_scan(loc);
      const DF up = df_shfl_up(incl, 1);
      const DF excl = lane == 0 ? DF{0.f, 0.f} : up;
      const unsigned m = __ballot_sync(0xffffffffu, df_gt(df_add(run, incl), thr));
      if (m) {
        const int L = __ffs(m) - 1;
        // prefix before lane L's first unit
        const DF base = df_add(run, df_shfl(excl, L));
        DF bk;
        int lastk;
        int uk = lane_search16(v, L, base, thr, &bk, &lastk);
        if (uk < 0) {  // rounding inside the lane: its last positive unit
          uk = lastk;
          any_before = false;
        }
        if (uk >= 0) {
          unit = rnd * 32 * R + L * R + uk;
          before = bk;
        }
      }
      run = df_add(run, df_shfl(incl, 31));
    }
    if (unit < 0) {  // no prefix exceeded u*Z: the last unit with weight
      int cand = -1;
      for (int rnd = 0; rnd < rounds; ++rnd) {
        load_round(rnd);
#pragma unroll
        for (int k = 0; k < R; ++k)
          if (v[k] > 0.f) cand = rnd * 32 * R + lane * R + k;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        cand = max(cand, __shfl_xor_sync(0xffffffffu, cand, off));
      unit = cand >= 0 ? cand : nsub - 1;
      any_before = false;
    }
    // vocabulary-order scan of the unit: lane l holds tokens e0 + 16 l ...
    const int e0 = unit * kUnitB;
    const int e1 = min(e0 + kUnitB, p.V);
    const int y0 = e0 + lane * 16;
    float zt[16], zd[16], w[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) zt[k] = zd[k] = 0.f;
    if (gp.use_t) load16<DT>(p, rt, true, y0, e1, zt);
    if (gp.use_d) load16<DT>(p, rd, false, y0, e1, zd);
    int lastpos = -1;
    weights16(gp, gp.c, y0, e1, zt, zd, w);
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (w[k] > 0.f) lastpos = y0 + k;
    const DF incl = df_warp_scan(df_sum16(w));
    const DF up = df_shfl_up(incl, 1);
    const DF excl = lane == 0 ? DF{0.f, 0.f} : up;
    t = -1;
    const unsigned m =
        __ballot_sync(0xffffffffu, any_before && df_gt(df_add(before, incl), thr));
    if (m) {
      const int L = __ffs(m) - 1;
      const DF base = df_add(before, df_shfl(excl, L));
      DF bt;
      int lastk;
      int tk = lane_search16(w, L, base, thr, &bt, &lastk);
      if (tk < 0) tk = lastk;  // rounding inside the lane: its last positive weight
      if (tk >= 0) t = e0 + L * 16 + tk;
    }
    if (t < 0) {  // rounding left no index: the last positive weight of the unit
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
      t = lastpos >= 0 ? lastpos : e0;
    }
    const int owner = (t - e0) >> 4;
    float wown = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (y0 + k == t) wown = w[k];
    wt = __shfl_sync(0xffffffffu, wown, owner & 31);
  }
  if (lane != 0) return;
  if (!SSD_CHK(g < p.groups && t >= 0 && t < p.V, p.dbg, 25, g, t)) return;
  p.out_token[g] = t;
  if (p.rc.table != nullptr)  // the round's cache: look the outcome (k, t) up
    round_outcome(static_cast<const Slot*>(p.rc.table), p.rc.cap, g, gp.k, t, p.groups,
                  p.rc.branch, p.rc.all_hit, p.rc.cnt);
  if (p.out_mass) p.out_mass[g] = (float)Zd;
  if (p.out_qprime) p.out_qprime[g] = (float)((double)wt / Zd);
  if (p.out_guess) write_guesses(p, g, p.rowres + g * p.rpg + p.nt, t);
}

// Sum of the draw weights of one unit (SPLIT: of half h of it) whose
// elements sit 16-byte aligned in shared memory (vectorised fast path of one
// warp), specialised per kind of draw.
template <int DT, int KIND, bool HAS_S, bool SPLIT>
__device__ __forceinline__ float unit_sum_k(const CdfParams& p, const GroupParams& gp,
                                            const Half& ht, const Half& hd, int ue0, int h) {
  constexpr int VEC = Elem<DT>::kVec;
  constexpr int NV = kUnitB / VEC / 32 / (SPLIT ? 2 : 1);
  static_assert(NV >= 1, "a half unit is at least one vector per lane");
  const int lane = threadIdx.x & 31;
  if (SPLIT) ue0 += h * (kUnitB / 2);
  const uint4* st4 = reinterpret_cast<const uint4*>(ht.sm + (ue0 - ht.ei0) * Elem<DT>::kSize);
  const uint4* sd4 = reinterpret_cast<const uint4*>(hd.sm + (ue0 - hd.ei0) * Elem<DT>::kSize);
  uint4 rt[NV], rd[NV];
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    if (KIND != kSaguaro) rt[m] = st4[lane + 32 * m];
    if (KIND != kTarget) rd[m] = sd4[lane + 32 * m];
  }
  float s = 0.f;
#pragma unroll
  for (int m = 0; m < NV; ++m) {
    const int vi = lane + 32 * m;
    float zt[VEC], zd[VEC];
    if (KIND != kSaguaro) Elem<DT>::unpack(rt[m], zt);
    if (KIND != kTarget) Elem<DT>::unpack(rd[m], zd);
    float sv = 0.f;
    if constexpr (KIND == kResidual) {
      // (p - q')^+ with the two exponent arguments and the two scalings as
      // packed f32x2 operations (the roundings of weight_k, element by
      // element); the set S's larger scale only where a draft logit reaches
      // theta (S holds the top F logits, theta the F-th)
      bool inS_any = false;
      if (HAS_S) {
        float mx = zd[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) mx = fmaxf(mx, zd[e]);
        inS_any = mx >= gp.theta;
      }
      if (!inS_any) {
        const unsigned long long cc = pack2(gp.c, gp.c), mm = pack2(-gp.mc_t, -gp.mc_d);
        const unsigned long long sc = pack2(gp.inv_st, gp.scale_out);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          unsigned long long a, w;
          asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(a) : "l"(pack2(zt[e], zd[e])), "l"(cc),
              "l"(mm));
          float at, ad;
          unpack2(a, at, ad);
          asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(w) : "l"(pack2(ex2(at), ex2(ad))), "l"(sc));
          float pt, q;
          unpack2(w, pt, q);
          sv += fmaxf(pt - q, 0.f);
        }
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
          sv += weight_k<KIND, HAS_S>(gp, gp.c, ue0 + vi * VEC + e, zt[e], zd[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e)
        sv += weight_k<KIND, HAS_S>(gp, gp.c, ue0 + vi * VEC + e, KIND != kSaguaro ? zt[e] : 0.f,
                                    KIND != kTarget ? zd[e] : 0.f);
    }
    s += sv;
  }
  return s;
}

template <int DT, bool SPLIT>
__device__ __forceinline__ float unit_sum_fast(const CdfParams& p, const GroupParams& gp,
                                               const Half& ht, const Half& hd, int ue0, int h) {
  const bool has_s = gp.theta != INFINITY;
  switch (kind_of(gp)) {
    case kTarget: return unit_sum_k<DT, kTarget, false, SPLIT>(p, gp, ht, hd, ue0, h);
    case kSaguaro:
      return has_s ? unit_sum_k<DT, kSaguaro, true, SPLIT>(p, gp, ht, hd, ue0, h)
                   : unit_sum_k<DT, kSaguaro, false, SPLIT>(p, gp, ht, hd, ue0, h);
    default:
      return has_s ? unit_sum_k<DT, kResidual, true, SPLIT>(p, gp, ht, hd, ue0, h)
                   : unit_sum_k<DT, kResidual, false, SPLIT>(p, gp, ht, hd, ue0, h);
  }
}

// Chunk c of the draws: group g and its units [u0, u1), group by group.
__device__ __forceinline__ void cdf_chunk_geom(const CdfParams& p, long long c, int64_t& g,
                                               int& u0, int& u1) {
  g = c / p.cpg;
  u0 = (int)(c - g * p.cpg) * p.cu;
  u1 = min(u0 + p.cu, p.nsub);
}

// Layout of a draw stage in a ring slot of kStageBytes: a weight that reads
// both rows gets half the slot for each (target run first); a weight that
// reads one row gets the whole slot, so it takes twice the units per stage.
struct DrawLayout {
  int ups;    // units per stage
  int cap;    // bytes of one row's run
  int off_d;  // offset of the draft run
};

template <int DT>
__device__ __forceinline__ DrawLayout draw_layout(const GroupParams& gp) {
  const bool two = gp.use_t && gp.use_d;
  const int cap = two ? kStageBytes / 2 : kStageBytes;
  return DrawLayout{cap / (kUnitB * Elem<DT>::kSize), cap, two ? kStageBytes / 2 : 0};
}

// Bulk copies of units [u, un) of a group's target row rt and draft row rd
// (null: not part of the weight) into one stage: the target run at dst, the
// draft run at dst + lay.off_d, each from its first 16-byte boundary to its
// last; completion is counted on `bar`.  One thread.
template <int DT>
__device__ __forceinline__ void cdf_issue_stage(const CdfParams& p, const char* rt,
                                                const char* rd, int u, int un,
                                                unsigned char* dst, const DrawLayout& lay,
                                                uint64_t* bar, volatile int* s_err) {
  constexpr int ES = Elem<DT>::kSize;
  const int e0 = u * kUnitB;
  const int e1 = min(p.V, un * kUnitB);
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
      srcok &= SSD_CHK(in_range(a0[h], a1[h], h == 0 ? p.t_lo : p.d_lo, h == 0 ? p.t_hi : p.d_hi),
                       p.dbg, 21, a0[h], h);
  srcok &= SSD_CHK((un - u) * kUnitB * ES <= lay.cap, p.dbg, 28, un - u, lay.cap);
  if (bytes > 0 && !*s_err && srcok) {
    mbar_arrive_expect_tx(bar, bytes);
    for (int h = 0; h < 2; ++h)
      if (a1[h] > a0[h])
        bulk_g2s(dst + (h == 0 ? 0 : lay.off_d), reinterpret_cast<const void*>(a0[h]),
                 (uint32_t)(a1[h] - a0[h]), bar);
  } else {
    mbar_arrive(bar);
  }
}

// The weight sums of units [u, un) of group g, staged by cdf_issue_stage at
// `stage`: consumer warp `warp` takes units u + warp, u + warp + 16, ...,
// and its lane 0 stores each sum.  A stage of at most half as many units as
// consumer warps (fp32 rows read together) gives each unit two warps, one
// per half: their sums meet in `half` (shared memory, [kConsumerWarps]) and
// the first half's warp adds them, in that order.  Units whose elements are
// not all in shared memory, 16-byte aligned (row ends, unaligned rows), read
// the missing ones from global memory.  All consumer warps call it.
template <int DT>
__device__ __forceinline__ void cdf_consume_stage(const CdfParams& p, int64_t g,
                                                  const GroupParams& gp, const char* rt,
                                                  const char* rd, int u, int un,
                                                  const unsigned char* stage,
                                                  const DrawLayout& lay, int warp,
                                                  float* half) {
  if (no_draw(gp)) return;
  constexpr int kPair = kConsumerWarps / 2;
  const bool split = 2 * (un - u) <= kConsumerWarps;  // the same in every consumer warp
  if (!split && u + warp >= un) return;
  const int e0 = u * kUnitB;
  const int e1 = min(p.V, un * kUnitB);
  Half ht, hd;
  constexpr int ES = Elem<DT>::kSize;
  for (int h = 0; h < 2; ++h) {
    Half& H = h == 0 ? ht : hd;
    const char* r = h == 0 ? rt : rd;
    H.row = r;
    H.sm = reinterpret_cast<const char*>(stage + (h == 0 ? 0 : lay.off_d));
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
  const int lane = threadIdx.x & 31;
  constexpr int VEC = Elem<DT>::kVec;
  auto fast_unit = [&](int ue0, int ue1) {
    bool fast = ue1 - ue0 == kUnitB;
    if (gp.use_t) fast &= ue0 >= ht.ei0 && ue1 <= ht.ei1 && (ue0 - ht.ei0) % VEC == 0;
    if (gp.use_d) fast &= ue0 >= hd.ei0 && ue1 <= hd.ei1 && (ue0 - hd.ei0) % VEC == 0;
    return fast;
  };
  // the elements [y0, y1) one by one (lane-strided)
  auto slow_sum = [&](int y0, int y1) {
    float s = 0.f;
    for (int y = y0 + lane; y < y1; y += 32) {
      const float zt = gp.use_t ? fetch<DT>(ht, y, p, true, lay.cap) : 0.f;
      const float zd = gp.use_d ? fetch<DT>(hd, y, p, false, lay.cap) : 0.f;
      s += weight(gp, gp.c, y, zt, zd);
    }
    return s;
  };
  if (split) {
    const int uu = u + warp % kPair, h = warp / kPair;
    float s = 0.f;
    if (uu < un) {
      const int ue0 = uu * kUnitB;
      const int ue1 = min(ue0 + kUnitB, p.V);
      if (fast_unit(ue0, ue1)) {
        s = unit_sum_fast<DT, true>(p, gp, ht, hd, ue0, h);
      } else {
        const int m = ue0 + kUnitB / 2;
        s = h == 0 ? slow_sum(ue0, min(m, ue1)) : slow_sum(m, ue1);
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) half[warp] = s;
    consumer_sync();
    if (h == 0 && uu < un && lane == 0 && SSD_CHK(uu < p.nsub && g < p.groups, p.dbg, 23, uu, g))
      p.subsum[g * p.nsub + uu] = half[warp] + half[warp + kPair];
    return;
  }
  for (int uu = u + warp; uu < un; uu += kConsumerWarps) {
    const int ue0 = uu * kUnitB;
    const int ue1 = min(ue0 + kUnitB, p.V);
    float s = fast_unit(ue0, ue1) ? unit_sum_fast<DT, false>(p, gp, ht, hd, ue0, 0)
                                  : slow_sum(ue0, ue1);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0 && SSD_CHK(uu < p.nsub && g < p.groups, p.dbg, 23, uu, g))
      p.subsum[g * p.nsub + uu] = s;
  }
}

// A finished chunk of group g (nu units, their sums stored): count it into
// the group's arrivals; the warp whose chunk completes the group runs the
// draw.  One warp.
template <int DT>
__device__ __forceinline__ void cdf_chunk_done(const CdfParams& p, int64_t g, int nu) {
  const int lane = threadIdx.x & 31;
  if (!SSD_CHK(g < p.groups, p.dbg, 20, g, p.groups)) return;
  int last = 0;
  if (lane == 0) {
    __threadfence();
    last = atomicAdd(p.cnt + g, nu) + nu == p.nsub;
    if (last) __threadfence();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) group_draw<DT>(p, g);
}


// ---- one-term draws straight from the streaming pass ---------------------------------
// The weight of a Saguaro row (q', [SSD-note] §"Saguaro 优化二") or of the
// all-accepted bonus (p_K, [SD-7.3] §7.3.2) has one term, so the streaming
// pass can sum it per block while the row goes by: bs[b] = (sum of
// exp2(z*c - off) over block b, off).  Block b is consumer warp b % 16's
// share of stage b / 16 of an aligned row: elements [s*E + w*BE, +BE).
// The draw then needs only the block holding u*Z, read again from L2:
//   W_b = bs[b].sum * 2^(off_b - mc) * scale (+ for a Saguaro set S, the
//         difference of the in-S and out-of-S weights of its tokens in b),
//   Z = sum_b W_b, the block where the prefix crosses u*Z, then the tokens
//   of that block in vocabulary order.
// Sums and prefixes are double-float pairs, as in group_draw.  One warp;
// rr (Saguaro: the row's top list, null for p_K) gives S and the guesses.
template <int DT>
__device__ __noinline__ void direct_draw(const CdfParams& p, const float2* bs, int nblk, const GroupParams& gp,
                            int64_t g, const RowResult* rr, int F) {
  constexpr int R = 16;  // block sums per lane per round
  constexpr int ES = Elem<DT>::kSize;
  constexpr int VEC = Elem<DT>::kVec;
  constexpr int BE = kVecsPerWarp * VEC;                 // elements per block
  constexpr int E = units_per_stage(ES) * kUnitA;        // elements per stage
  constexpr int PL = BE / 32;                            // elements per lane in a block
  static_assert(PL == 8 || PL == 16 || PL == 32, "a lane's run is half, one or two 16-element halves");
  constexpr int PW = PL < 16 ? 16 : PL;                  // held per lane (zero weights beyond PL)
  const int lane = threadIdx.x & 31;
  if (!SSD_CHK(g < p.groups, p.dbg, 50, g, p.groups)) return;
  const bool tgt = gp.use_t != 0;
  const float mc = tgt ? gp.mc_t : gp.mc_d;
  const float sc = tgt ? gp.inv_st : gp.scale_out;
  const bool has_s = !tgt && gp.theta != INFINITY && rr != nullptr;
  const int nS = has_s ? F : 0;
  const float dsc = gp.scale_in - gp.scale_out;
  const char* row = tgt ? row_ptr(p.tgt, gp.row_t, p.t_stride, ES) : row_ptr(p.dft, gp.row_d, p.d_stride, ES);
  const int rounds = (nblk + 32 * R - 1) / (32 * R);
  // the cached set S (lane f < nS: token f, its block and weight difference),
  // loaded at once
  int s_blk = -1;
  float s_d = 0.f;
  if (lane < nS) {
    const int tok = __ldcg(&rr->ti[lane]);
    const float tv = __ldcg(&rr->tv[lane]);
    if (tok >= 0) {
      s_blk = (tok / E) * kConsumerWarps + (tok % E) / BE;
      s_d = dsc * ex2(fmaf(tv, gp.c, -mc));
    }
  }
  float v[R];
  auto load_round = [&](int rnd) {
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int b = rnd * 32 * R + lane * R + k;
      float w = 0.f;
      if (b < nblk) {
        const float2 e = __ldcg(bs + b);
        if (e.x > 0.f) w = e.x * ex2(e.y - mc) * sc;
      }
      v[k] = w;
    }
    // the cached set's tokens move from the out-of-S to the in-S weight
    for (int f = 0; f < nS; ++f) {
      const int b = __shfl_sync(0xffffffffu, s_blk, f);
      const float d = __shfl_sync(0xffffffffu, s_d, f);
      if (b < 0) continue;
      const int k = b - rnd * 32 * R - lane * R;
      if (k >= 0 && k < R) {
#pragma unroll
        for (int q = 0; q < R; ++q)
          if (q == k) v[q] = fmaxf(v[q] + d, 0.f);
      }
    }
  };
  load_round(0);
  DF loc0 = df_sum16(v);
  DF Zl = loc0;
  for (int rnd = 1; rnd < rounds; ++rnd) {
    load_round(rnd);
    Zl = df_add(Zl, df_sum16(v));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const DF o{__shfl_xor_sync(0xffffffffu, Zl.hi, off), __shfl_xor_sync(0xffffffffu, Zl.lo, off)};
    Zl = df_add(Zl, o);
  }
  const DF Z = Zl;
  double Zd = (double)Z.hi + (double)Z.lo;
  int t;
  float wt;
  if (!(Zd > 1e-30)) {
    // a one-term weight sums to about 1; keep a defined result anyway
    if (lane == 0 && p.status) atomicOr(p.status, SSD_DEV_ZERO_RESIDUAL);
    t = full_row_draw<DT>(p, gp, tgt ? row : nullptr, tgt ? nullptr : row, &Zd);
    wt = weight_global<DT>(p, gp, tgt ? row : nullptr, tgt ? nullptr : row, t);
  } else {
    const DF thr = df_scale(Z, (float)gp.u);
    int blk = -1;
    DF before{0.f, 0.f};
    bool any_before = true;
    DF run{0.f, 0.f};
    for (int rnd = 0; rnd < rounds && blk < 0; ++rnd) {
      DF loc = loc0;
      if (rounds > 1) {
        load_round(rnd);
        if (rnd > 0) loc = df_sum16(v);
      }
      const DF incl = df_warp_scan(loc);
      const DF up = df_shfl_up(incl, 1);
      const DF excl = lane == 0 ? DF{0.f, 0.f} : up;
      const unsigned m = __ballot_sync(0xffffffffu, df_gt(df_add(run, incl), thr));
      if (m) {
        const int L = __ffs(m) - 1;
        const DF base = df_add(run, df_shfl(excl, L));
        DF bk;
        int lastk;
        int uk = lane_search16(v, L, base, thr, &bk, &lastk);
        if (uk < 0) {
          uk = lastk;
          any_before = false;
        }
        if (uk >= 0) {
          blk = rnd * 32 * R + L * R + uk;
          before = bk;
        }
      }
      run = df_add(run, df_shfl(incl, 31));
    }
    if (blk < 0) {  // no prefix exceeded u*Z: the last block with weight
      int cand = -1;
      for (int rnd = 0; rnd < rounds; ++rnd) {
        load_round(rnd);
#pragma unroll
        for (int k = 0; k < R; ++k)
          if (v[k] > 0.f) cand = rnd * 32 * R + lane * R + k;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cand = max(cand, __shfl_xor_sync(0xffffffffu, cand, off));
      blk = cand >= 0 ? cand : 0;
      any_before = false;
    }
    // the block's tokens in vocabulary order: lane l holds PL consecutive ones
    const int e_lo = (blk / kConsumerWarps) * E + (blk % kConsumerWarps) * BE;
    const int e_hi = min(p.V, e_lo + BE);
    const int y0 = e_lo + lane * PL;
    float z[PW], w[PW];
#pragma unroll
    for (int k = PL; k < PW; ++k) z[k] = w[k] = 0.f;
#pragma unroll
    for (int k = 0; k < PL; k += VEC) {
      const uintptr_t a = (uintptr_t)(row + (int64_t)(y0 + k) * ES);
      uint4 r4 = make_uint4(0, 0, 0, 0);
      const bool in = y0 + k + VEC <= e_hi &&
                      SSD_CHK(in_range(a, a + 16, tgt ? p.t_lo : p.d_lo, tgt ? p.t_hi : p.d_hi),
                              p.dbg, 51, y0 + k, g);
      if (in) r4 = __ldg(reinterpret_cast<const uint4*>(a));
      Elem<DT>::unpack(r4, z + k);
#pragma unroll
      for (int q = 0; q < VEC; ++q) {
        const int y = y0 + k + q;
        float wy = 0.f;
        if (in) {
          const float e = ex2(fmaf(z[k + q], gp.c, -mc));
          wy = tgt ? e * gp.inv_st : e * q_scale<true>(gp, y, z[k + q]);
        }
        w[k + q] = wy;
      }
    }
    int lastpos = -1;
#pragma unroll
    for (int k = 0; k < PL; ++k)
      if (w[k] > 0.f) lastpos = y0 + k;
    DF lsum = df_sum16(w);
    if constexpr (PL == 32) lsum = df_add(lsum, df_sum16(w + 16));
    const DF incl = df_warp_scan(lsum);
    const DF up = df_shfl_up(incl, 1);
    const DF excl = lane == 0 ? DF{0.f, 0.f} : up;
    t = -1;
    const unsigned m = __ballot_sync(0xffffffffu, any_before && df_gt(df_add(before, incl), thr));
    if (m) {
      const int L = __ffs(m) - 1;
      const DF base = df_add(before, df_shfl(excl, L));
      DF bt;
      int lastk;
      int tk;
      if constexpr (PL == 32) {
        // the first half of lane L's run, then (if it does not cross) the second
        const DF half = df_shfl(df_sum16(w), L);
        if (df_gt(df_add(base, half), thr)) {
          tk = lane_search16(w, L, base, thr, &bt, &lastk);
          if (tk < 0) tk = lastk;
        } else {
          tk = lane_search16(w + 16, L, df_add(base, half), thr, &bt, &lastk);
          if (tk < 0) tk = lastk;
          if (tk >= 0) tk += 16;
          else {  // rounding: the last positive weight of the first half
            int lk2;
            DF b2;
            (void)lane_search16(w, L, base, thr, &b2, &lk2);
            tk = lk2;
          }
        }
      } else {
        tk = lane_search16(w, L, base, thr, &bt, &lastk);
        if (tk < 0) tk = lastk;
      }
      if (tk >= 0) t = e_lo + L * PL + tk;
    }
    if (t < 0) {  // rounding left no index: the last positive weight of the block
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
      t = lastpos >= 0 ? lastpos : e_lo;
    }
    const int owner = (t - e_lo) / PL;
    float wown = 0.f;
#pragma unroll
    for (int k = 0; k < PL; ++k)
      if (y0 + k == t) wown = w[k];
    wt = __shfl_sync(0xffffffffu, wown, owner & 31);
  }
  if (lane != 0) return;
  if (!SSD_CHK(t >= 0 && t < p.V, p.dbg, 52, g, t)) return;
  p.out_token[g] = t;
  if (p.rc.table != nullptr)  // the round's cache: look the outcome (k, t) up
    round_outcome(static_cast<const Slot*>(p.rc.table), p.rc.cap, g, gp.k, t, p.groups,
                  p.rc.branch, p.rc.all_hit, p.rc.cnt);
  if (p.out_mass) p.out_mass[g] = (float)Zd;
  if (p.out_qprime) p.out_qprime[g] = (float)((double)wt / Zd);
  if (p.out_guess && rr != nullptr) write_guesses(p, g, rr, t);
}

}  // namespace
}  // namespace ssd
