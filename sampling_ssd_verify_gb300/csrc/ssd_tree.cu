// ssd_tree.cu -- verification of tree-shaped drafts.
//
// [SD-7.3] "7.3 Speculative Decoding：投机采样加速" §7.3.9 item 3 names tree drafts
// (several candidate continuations per position) as the next step; the
// per-token rule of §7.3.3 is applied to each candidate in turn, with the
// residual renormalised after every rejection (multi-candidate rejection
// sampling):
//   at node u with residual r (r = p_u on arrival), child v (in increasing
//   index order) is accepted with probability min(1, r(x_v) / q_u(x_v));
//   accepted: move to v; rejected: r = (r - q_u)^+ / sum (r - q_u)^+;
//   no child accepted (or a leaf): the bonus is drawn from r.
// After m rejections at node u the residual is (p_u - c q_u)^+ / P with
// c = 1 + P_1 + ... + P_{m-1} and P = W(c) = sum_y (p_u(y) - c q_u(y))^+
// (each step maps (c, P) to (c + P, W(c + P))), so one pass over the rows
// p_u and q_u per rejection gives the next residual exactly.
//
// Two launches: the streaming kernel (ssd_stream_kernel.cuh) computes every
// row's normaliser; then a cluster of CTAs per tree walks it.
//  * Every CTA of the cluster loads, once, the decision inputs of every edge
//    (p_u(x_v), q_u(x_v), the uniform) and every node's normalisers, so the
//    accept/reject steps are shared-memory arithmetic that each thread
//    repeats (same inputs, same instructions: every thread of the cluster
//    takes the same branch).
//  * A pass over the rows is split over the cluster by 512-element units
//    (16-byte loads where both rows are 16-byte aligned); each CTA's partial
//    of W goes to every CTA's shared memory (st.shared::cluster), one
//    cluster barrier per pass, and every CTA adds the partials in rank order.
//  * The pass for the last child's rejection also writes the unit sums of
//    the bonus weight (p_u - c' q_u)^+, so the bonus costs no further pass;
//    a walk that ends by acceptance at a leaf makes one pass over p_leaf.
//  * Rank 0's first warp draws the bonus (ssd_cdf_dev.cuh's group_draw).

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_cdf_dev.cuh"
#include "ssd_device.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kTreeConsumers = 16;               // warps that sum the weights
constexpr int kTreeWarps = kTreeConsumers + 1;   // + one warp that issues the copies
constexpr int kTreeThreads = kTreeWarps * 32;
constexpr int kTreeRingBytes = 192 * 1024;       // the copy ring (dynamic shared memory)

// A stage holds kTreeConsumers units (one per consumer warp) of the target
// row and, after it, of the draft row.
template <int DT>
struct TreeRing {
  static constexpr int kRowBytes = kTreeConsumers * kUnitB * Elem<DT>::kSize;
  static constexpr int kStageBytes = 2 * kRowBytes;
  static constexpr int kStages = kTreeRingBytes / kStageBytes;
  static_assert(kStages >= 2, "the ring holds at least two stages");
};

// The weight of one element: p_u(y) (no draft term) or (p_u(y) - s q_u(y))^+,
// with p = exp2(fl(z c - mc_t)) inv_st and s q = exp2(fl(z c - mc_d)) scale --
// the same expressions as the bonus draw's weight (ssd_cdf_dev.cuh).
struct PassW {
  float c, mc_t, inv_st, mc_d, scale;
};

template <bool USE_D>
__device__ __forceinline__ float pass_weight(const PassW& w, float zt, float zd) {
  const float pt = ex2(fmaf(zt, w.c, -w.mc_t)) * w.inv_st;
  if (!USE_D) return pt;
  return fmaxf(pt - ex2(fmaf(zd, w.c, -w.mc_d)) * w.scale, 0.f);
}

// The weight sum of unit `un` (elements un * 512 ...), in every lane.  Lane
// l's runs are the VEC elements from un * 512 + (l + 32 j) VEC; a run that
// starts below `send` is read from shared memory (ps, qs: the unit's first
// element there), the others from the rows.
template <int DT, bool USE_D>
__device__ __forceinline__ float unit_sum(const char* prow, const char* qrow, int V, bool vec,
                                          const PassW& w, int un, const char* ps, const char* qs,
                                          int send) {
  constexpr int VEC = Elem<DT>::kVec;
  constexpr int J = kUnitB / (32 * VEC);  // runs per lane per unit
  const int lane = threadIdx.x & 31;
  uint4 rt[J], rd[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int y = un * kUnitB + (lane + 32 * j) * VEC;
    if (y < send) {
      rt[j] = *reinterpret_cast<const uint4*>(ps + (lane + 32 * j) * 16);
      if (USE_D) rd[j] = *reinterpret_cast<const uint4*>(qs + (lane + 32 * j) * 16);
    } else {
      rt[j] = load_run<DT>(prow, y, V, vec);
      if (USE_D) rd[j] = load_run<DT>(qrow, y, V, vec);
    }
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int y = un * kUnitB + (lane + 32 * j) * VEC;
    float zt[VEC], zd[VEC];
    Elem<DT>::unpack(rt[j], zt);
    if (USE_D) Elem<DT>::unpack(rd[j], zd);
#pragma unroll
    for (int k = 0; k < VEC; ++k)
      if (y + k < V) s += pass_weight<USE_D>(w, zt[k], USE_D ? zd[k] : 0.f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

// What one CTA needs for its share of a pass.
struct Share {
  const char* prow;
  const char* qrow;
  int V, ulo, uhi;  // units [ulo, uhi) of the rows
  float* sub;       // unit sums out (null: none)
};

// This CTA's share read straight from the rows (rows not 16-byte aligned):
// consumer warp w takes units ulo + w, ulo + w + 16, ...  Returns the
// partial of the warp (lane 0).
template <int DT, bool USE_D>
__device__ double share_ldg(const Share& sh, const PassW& w) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  double acc = 0.0;
  for (int un = sh.ulo + warp; un < sh.uhi; un += kTreeConsumers) {
    const float s = unit_sum<DT, USE_D>(sh.prow, sh.qrow, sh.V, false, w, un, nullptr, nullptr, 0);
    if (sh.sub != nullptr && lane == 0) sh.sub[un] = s;
    acc += (double)s;
  }
  return acc;
}

// This CTA's share through the copy ring (rows 16-byte aligned): the copy
// warp's lane 0 brings stage after stage (kTreeConsumers units of each row,
// the byte count rounded down to 16; the few elements beyond are read from
// the rows), consumer warp w sums unit w of each stage.  `gs` counts the
// stages this CTA has used (the ring's phase), the same in every thread.
template <int DT, bool USE_D>
__device__ double share_ring(const Share& sh, const PassW& w, char* ring, uint64_t* full,
                             uint64_t* empty, uint32_t& gs, volatile int* s_err, int32_t* status) {
  using RG = TreeRing<DT>;
  constexpr int ES = Elem<DT>::kSize;
  constexpr int SE = kTreeConsumers * kUnitB;  // elements of a row per stage
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nst = (sh.uhi - sh.ulo + kTreeConsumers - 1) / kTreeConsumers;
  double acc = 0.0;
  auto stage_bytes = [&](int st) {  // bytes of each row brought by stage st
    const int e0 = (sh.ulo + st * kTreeConsumers) * kUnitB;
    const int e1 = min(min(e0 + SE, sh.uhi * kUnitB), sh.V);
    return (uint32_t)((e1 - e0) * ES) & ~15u;
  };
  if (warp == kTreeConsumers) {
    if (lane == 0) {
      for (int st = 0; st < nst; ++st) {
        const uint32_t n = gs + (uint32_t)st;
        const int slot = (int)(n % RG::kStages);
        if (n >= (uint32_t)RG::kStages)
          mbar_wait(empty + slot, ((n / RG::kStages) - 1) & 1, s_err, status);
        const uint32_t bytes = stage_bytes(st);
        const int64_t off = (int64_t)(sh.ulo + st * kTreeConsumers) * kUnitB * ES;
        mbar_arrive_expect_tx(full + slot, bytes * (USE_D ? 2u : 1u));
        if (bytes > 0) {
          char* dst = ring + (size_t)slot * RG::kStageBytes;
          bulk_g2s(dst, sh.prow + off, bytes, full + slot);
          if (USE_D) bulk_g2s(dst + RG::kRowBytes, sh.qrow + off, bytes, full + slot);
        }
      }
    }
  } else {
    for (int st = 0; st < nst; ++st) {
      const uint32_t n = gs + (uint32_t)st;
      const int slot = (int)(n % RG::kStages);
      mbar_wait(full + slot, (n / RG::kStages) & 1, s_err, status);
      const int un = sh.ulo + st * kTreeConsumers + warp;
      if (un < sh.uhi) {
        const int send = (sh.ulo + st * kTreeConsumers) * kUnitB + (int)(stage_bytes(st) / ES);
        const char* ps = ring + (size_t)slot * RG::kStageBytes + (size_t)warp * kUnitB * ES;
        const float s = unit_sum<DT, USE_D>(sh.prow, sh.qrow, sh.V, true, w, un, ps,
                                            ps + RG::kRowBytes, send);
        if (sh.sub != nullptr && lane == 0) sh.sub[un] = s;
        acc += (double)s;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + slot);
    }
  }
  gs += (uint32_t)nst;
  return acc;
}

struct TreeShared {
  // per node u: normalisers of p_u and q_u
  float mct[kMaxTreeNodes], mcd[kMaxTreeNodes];
  double st[kMaxTreeNodes], sd[kMaxTreeNodes];
  // per node v >= 1 (the edge from its parent u): logits of x_v in p_u, q_u,
  // then p_u(x_v), q_u(x_v) and the uniform of its test
  float lp[kMaxTreeNodes], lq[kMaxTreeNodes];
  double pv[kMaxTreeNodes], qv[kMaxTreeNodes], uv[kMaxTreeNodes];
  double red[kTreeWarps];
  double part[2][kTreeMaxCluster];  // the cluster's partials, double-buffered by pass
};

template <int DT>
__global__ void __launch_bounds__(kTreeThreads, 1)
    tree_walk_kernel(const __grid_constant__ TreeParams tp) {
  constexpr int ES = Elem<DT>::kSize;
  const int cs = tp.cluster;
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / cs;
  const int N = tp.N;
  const int V = tp.V;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const CdfParams& q = tp.q;
  using RG = TreeRing<DT>;
  __shared__ TreeShared sh;
  __shared__ __align__(8) uint64_t full[RG::kStages], empty[RG::kStages];
  __shared__ int s_err;
  extern __shared__ __align__(128) char ring[];
  cluster_arrive_relaxed();
  if (tid == 0) {
    s_err = 0;
    for (int i = 0; i < RG::kStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kTreeConsumers);
    }
    fence_barrier_init();
  }
  const float cf = tp.c;
  const double c = (double)cf;
  const RowResult* rr = tp.rowres + (int64_t)b * 2 * N;
  const int nE = tp.child_off[N];

  // ---- decision inputs of every edge and normalisers of every node ----
  auto row_t = [&](int u) { return row_ptr(tp.tgt, (int64_t)b * N + u, tp.t_stride, ES); };
  auto row_d = [&](int u) { return row_ptr(tp.dft, (int64_t)b * N + u, tp.d_stride, ES); };
  auto rows_ok = [&](int u) {
    const uintptr_t a = (uintptr_t)row_t(u), d = (uintptr_t)row_d(u);
    return SSD_CHK(in_range(a, a + (uintptr_t)V * ES, q.t_lo, q.t_hi), q.dbg, 60, b, u) &&
           SSD_CHK(in_range(d, d + (uintptr_t)V * ES, q.d_lo, q.d_hi), q.dbg, 61, b, u);
  };
  if (tid < N) {
    sh.mct[tid] = __ldcg(&rr[tid].mc);
    sh.st[tid] = __ldcg(&rr[tid].s);
    sh.mcd[tid] = __ldcg(&rr[N + tid].mc);
    sh.sd[tid] = __ldcg(&rr[N + tid].s);
  }
  int pu = -1, pvn = -1;  // this thread's edge: parent, child
  if (tid < nE) {
    pvn = tp.child[tid];
    int lo = 0, hi = N - 1;  // the u with child_off[u] <= tid < child_off[u + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tp.child_off[mid] <= tid) lo = mid;
      else hi = mid - 1;
    }
    pu = lo;
    int x = __ldg(tp.tokens + (int64_t)b * N + pvn);
    if (x < 0 || x >= V) {
      if (tp.status && rank == 0) atomicOr(tp.status, SSD_DEV_BAD_TOKEN);
      x = 0;
    }
    const bool ok = rows_ok(pu);
    sh.lp[pvn] = ok ? Elem<DT>::load(row_t(pu), x) : 0.f;
    sh.lq[pvn] = ok ? Elem<DT>::load(row_d(pu), x) : 0.f;
  }
  __syncthreads();
  if (tid < nE) {
    sh.pv[pvn] = exp2((double)sh.lp[pvn] * c - (double)sh.mct[pu]) / sh.st[pu];
    sh.qv[pvn] = exp2((double)sh.lq[pvn] * c - (double)sh.mcd[pu]) / sh.sd[pu];
    sh.uv[pvn] = uniform24(tp.seeds[b], (uint32_t)b, (uint32_t)(pvn - 1), 0u, tp.round);
  }
  __syncthreads();

  // ---- one pass over rows of node u, split over the cluster ----
  uint32_t gs = 0;  // stages through the ring so far
  const int ulo = (int)((int64_t)rank * q.nsub / cs), uhi = (int)((int64_t)(rank + 1) * q.nsub / cs);
  int npass = 0;
  float* sub_b = q.subsum + (int64_t)b * q.nsub;
  // W = sum of the weights of node u's rows (the same value in every thread
  // of the cluster); sub: write the unit sums of the bonus draw
  auto pass = [&](int u, bool use_d, const PassW& w, bool sub) -> double {
    const char* pr = row_t(u);
    const char* qr = row_d(u);
    const bool ok = rows_ok(u);
    const bool vec = (((uintptr_t)pr | (use_d ? (uintptr_t)qr : 0)) & 15) == 0;
    float* dst = sub && SSD_CHK(b < q.groups, q.dbg, 62, b, q.groups) ? sub_b : nullptr;
    const Share shr{pr, qr, V, ulo, uhi, dst};
    double part = 0.0;
    if (ok && vec) {
      part = use_d ? share_ring<DT, true>(shr, w, ring, full, empty, gs, &s_err, tp.status)
                   : share_ring<DT, false>(shr, w, ring, full, empty, gs, &s_err, tp.status);
    } else if (ok && warp < kTreeConsumers) {
      part = use_d ? share_ldg<DT, true>(shr, w) : share_ldg<DT, false>(shr, w);
    }
    if (lane == 0) sh.red[warp] = part;
    if (npass == 0) cluster_wait();  // every CTA of the cluster has started
    __syncthreads();
    const int buf = npass & 1;
    if (tid < cs) {
      double t = 0.0;
      for (int i = 0; i < kTreeWarps; ++i) t += sh.red[i];
      st_cluster_f64(&sh.part[buf][rank], (uint32_t)tid, t);
    }
    if (sub) __threadfence();  // the unit sums, for rank 0's draw
    cluster_barrier();
    double W = 0.0;
    for (int r = 0; r < cs; ++r) W += sh.part[buf][r];
    ++npass;
    return W;
  };
  auto bonus_gp = [&](int u, int depth, double cc) {
    GroupParams gp = {};
    gp.k = depth;
    gp.use_t = 1;
    gp.row_t = (int64_t)b * N + u;
    gp.mc_t = sh.mct[u];
    gp.inv_st = (float)(1.0 / sh.st[u]);
    gp.sign_d = -1;
    gp.theta = INFINITY;
    gp.itheta = -1;
    if (cc > 0.0) {
      gp.use_d = 1;
      gp.row_d = (int64_t)b * N + u;
      gp.mc_d = sh.mcd[u];
      gp.scale_out = gp.scale_in = (float)(cc / sh.sd[u]);
    }
    gp.u = uniform24(tp.seeds[b], (uint32_t)b, (uint32_t)u, 1u, tp.round);
    gp.c = cf;
    return gp;
  };
  auto bonus_pass = [&](int u, int depth, double cc) -> double {
    const GroupParams gp = bonus_gp(u, depth, cc);
    if (rank == 0 && tid == 0) tp.gparams[b] = gp;
    const PassW w{cf, gp.mc_t, gp.inv_st, gp.mc_d, gp.scale_out};
    return pass(u, gp.use_d != 0, w, true);
  };

  // ---- the walk (every thread of the cluster takes the same steps) ----
  int u = 0, depth = 0;
  double cc = 0.0, P = 1.0, Zlast = -1.0;
  bool drawn = false;  // the bonus unit sums are written
  bool zero = false;   // a residual vanished (reported once)
  // u grows at every move (children have larger indices): at most N moves
  for (int iter = 0; iter < N && !drawn; ++iter) {
    const int c0 = tp.child_off[u], c1 = tp.child_off[u + 1];
    bool moved = false;
    for (int ci = c0; ci < c1; ++ci) {
      const int v = tp.child[ci];
      const double pv = sh.pv[v], qv = sh.qv[v];
      const double rv = cc == 0.0 ? pv : fmax(pv - cc * qv, 0.0) / P;
      if (sh.uv[v] < rv / qv) {
        if (rank == 0 && tid == 0 && tp.path && depth < tp.Dmax)
          tp.path[(int64_t)b * tp.Dmax + depth] = v;
        depth += 1;
        u = v;
        cc = 0.0;
        P = 1.0;
        Zlast = -1.0;
        moved = true;
        break;
      }
      // rejected: the next residual, (p - c' q)^+ / W(c') with c' = c + P
      const double cn = cc + P;
      double W;
      if (ci + 1 < c1) {
        const PassW w{cf, sh.mct[u], (float)(1.0 / sh.st[u]), sh.mcd[u], (float)(cn / sh.sd[u])};
        W = pass(u, true, w, false);
      } else {
        W = bonus_pass(u, depth, cn);  // the last child: the bonus's unit sums too
        drawn = W > 1e-300;
      }
      if (W > 1e-300) {
        Zlast = W / P;
        cc = cn;
        P = W;
      } else {
        zero = true;
        Zlast = 0.0;
      }
    }
    if (!moved) break;
  }
  if (!drawn) bonus_pass(u, depth, cc);  // a leaf, or the last residual vanished
  if (zero && rank == 0 && tid == 0 && tp.status) atomicOr(tp.status, SSD_DEV_ZERO_RESIDUAL);
  // no copy into this CTA's shared memory is left in flight
  if (warp == kTreeConsumers && lane == 0)
    for (uint32_t n = gs > (uint32_t)RG::kStages ? gs - RG::kStages : 0u; n < gs; ++n)
      mbar_wait(full + n % RG::kStages, (n / RG::kStages) & 1, &s_err, tp.status);
  if (rank != 0) return;
  if (warp == 0) group_draw<DT>(q, b);
  if (tid == 0) {
    tp.accept_len[b] = depth;
    if (tp.path)
      for (int d = depth; d < tp.Dmax; ++d) tp.path[(int64_t)b * tp.Dmax + d] = -1;
    // the last residual step's mass; 1 (the mass of p_u) when u rejected nothing
    if (tp.resid_mass) tp.resid_mass[b] = Zlast >= 0.0 ? (float)Zlast : 1.f;
  }
}

}  // namespace

template <int DT>
cudaError_t launch_tree_dt(const TreeParams& tp, cudaStream_t s) {
  const int cs = tp.cluster;
  if (cs < 1 || cs > kTreeMaxCluster || (cs & (cs - 1)) != 0) return cudaErrorInvalidValue;
  const int ring = TreeRing<DT>::kStages * TreeRing<DT>::kStageBytes;
  const cudaError_t e =
      cudaFuncSetAttribute(tree_walk_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, ring);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tp.B * cs));
  cfg.blockDim = dim3(kTreeThreads);
  cfg.dynamicSmemBytes = (size_t)ring;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)cs;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_walk_kernel<DT>, tp);
}

template cudaError_t launch_tree_dt<0>(const TreeParams& tp, cudaStream_t s);
template cudaError_t launch_tree_dt<1>(const TreeParams& tp, cudaStream_t s);

}  // namespace ssd
