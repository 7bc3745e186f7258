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
// row's normaliser; then one CTA per tree walks it, reading the rows it needs
// for each residual and for the bonus draw (ssd_cdf_dev.cuh's group_draw).

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_cdf_dev.cuh"
#include "ssd_device.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kTreeThreads = 256;

// Compensated (Kahan) fp32 accumulation of non-negative terms.
struct KSum {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float v) {
    const float y = v - lo;
    const float t = hi + y;
    lo = (t - hi) - y;
    hi = t;
  }
};

// Block-wide sum of per-thread compensated pairs, as a double (all threads).
__device__ double block_sum(KSum k, double* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double v = (double)k.hi - (double)k.lo;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < kTreeThreads / 32; ++w) t += s_red[w];
  __syncthreads();
  return t;
}

template <int DT>
__device__ __forceinline__ float logit_at(const char* row, int y) {
  return Elem<DT>::load(row, y);
}

template <int DT>
__global__ void __launch_bounds__(kTreeThreads)
    tree_walk_kernel(const __grid_constant__ TreeParams tp) {
  const int b = blockIdx.x;
  const int N = tp.N;
  const int V = tp.V;
  constexpr int ES = Elem<DT>::kSize;
  __shared__ double s_red[kTreeThreads / 32];
  __shared__ int s_u, s_depth, s_acc;
  __shared__ double s_c, s_P, s_Zlast;
  if (threadIdx.x == 0) {
    s_u = 0;
    s_depth = 0;
    s_c = 0.0;
    s_P = 1.0;
    s_Zlast = -1.0;
  }
  __syncthreads();
  const float cf = tp.c;
  const double c = (double)cf;
  const RowResult* rr = tp.rowres + (int64_t)b * 2 * N;
  for (int iter = 0; iter <= N; ++iter) {
    const int u = s_u;
    const RowResult* rt = rr + u;
    const RowResult* rd = rr + N + u;
    const char* prow = row_ptr(tp.tgt, (int64_t)b * N + u, tp.t_stride, ES);
    const char* qrow = row_ptr(tp.dft, (int64_t)b * N + u, tp.d_stride, ES);
    const float mct = __ldcg(&rt->mc), mcd = __ldcg(&rd->mc);
    const double st = __ldcg(&rt->s), sd = __ldcg(&rd->s);
    bool moved = false;
    for (int ci = tp.child_off[u]; ci < tp.child_off[u + 1]; ++ci) {
      const int v = tp.child[ci];
      if (threadIdx.x == 0) {
        int x = __ldg(tp.tokens + (int64_t)b * N + v);
        if (x < 0 || x >= V) {
          if (tp.status) atomicOr(tp.status, SSD_DEV_BAD_TOKEN);
          x = 0;
        }
        const double pv = exp2((double)logit_at<DT>(prow, x) * c - (double)mct) / st;
        const double qv = exp2((double)logit_at<DT>(qrow, x) * c - (double)mcd) / sd;
        const double rv = s_c == 0.0 ? pv : fmax(pv - s_c * qv, 0.0) / s_P;
        const double uv = uniform24(tp.seeds[b], (uint32_t)b, (uint32_t)(v - 1), 0u, tp.round);
        s_acc = uv < rv / qv ? 1 : 0;
      }
      __syncthreads();
      if (s_acc) {
        if (threadIdx.x == 0) {
          if (tp.path && s_depth < tp.Dmax) tp.path[(int64_t)b * tp.Dmax + s_depth] = v;
          s_depth += 1;
          s_u = v;
          s_c = 0.0;
          s_P = 1.0;
          s_Zlast = -1.0;
        }
        moved = true;
        __syncthreads();
        break;
      }
      // rejected: the next residual, (p - c' q)^+ / W(c') with c' = c + P
      const double cn = s_c + s_P;
      const float cnf = (float)cn;
      KSum k;
      for (int y = threadIdx.x; y < V; y += kTreeThreads) {
        const float pp = ex2(fmaf(logit_at<DT>(prow, y), cf, -mct)) * (float)(1.0 / st);
        const float qq = ex2(fmaf(logit_at<DT>(qrow, y), cf, -mcd)) * (float)(1.0 / sd);
        k.add(fmaxf(pp - cnf * qq, 0.f));
      }
      const double W = block_sum(k, s_red);
      if (threadIdx.x == 0) {
        if (W > 1e-300) {
          s_Zlast = W / s_P;
          s_c = cn;
          s_P = W;
        } else {
          if (tp.status) atomicOr(tp.status, SSD_DEV_ZERO_RESIDUAL);
          s_Zlast = 0.0;
        }
      }
      __syncthreads();
    }
    if (!moved) break;
  }
  // the bonus from the final residual: w = (p_u - c q_u)^+ (c = 0: p_u)
  const int u = s_u;
  const RowResult* rt = rr + u;
  const RowResult* rd = rr + N + u;
  const CdfParams& q = tp.q;
  if (threadIdx.x == 0) {
    GroupParams gp = {};
    gp.k = s_depth;
    gp.use_t = 1;
    gp.row_t = (int64_t)b * N + u;
    gp.mc_t = __ldcg(&rt->mc);
    gp.inv_st = (float)(1.0 / __ldcg(&rt->s));
    gp.sign_d = -1;
    gp.theta = INFINITY;
    gp.itheta = -1;
    if (s_c > 0.0) {
      gp.use_d = 1;
      gp.row_d = (int64_t)b * N + u;
      gp.mc_d = __ldcg(&rd->mc);
      gp.scale_out = gp.scale_in = (float)(s_c / __ldcg(&rd->s));
    }
    gp.u = uniform24(tp.seeds[b], (uint32_t)b, (uint32_t)u, 1u, tp.round);
    gp.c = cf;
    tp.gparams[b] = gp;
  }
  __syncthreads();
  const GroupParams gp = load_gp(tp.gparams + b);
  const char* prow = row_ptr(tp.tgt, gp.row_t, tp.t_stride, ES);
  const char* qrow = gp.use_d ? row_ptr(tp.dft, gp.row_d, tp.d_stride, ES) : nullptr;
  // unit sums of the draw weight: warp w takes units w, w + 8, ...
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int un = warp; un < q.nsub; un += kTreeThreads / 32) {
    float sacc = 0.f;
    for (int m = 0; m < kUnitB / 32; ++m) {
      const int y = un * kUnitB + lane + 32 * m;
      if (y < V)
        sacc += weight(gp, gp.c, y, logit_at<DT>(prow, y), qrow ? logit_at<DT>(qrow, y) : 0.f);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, off);
    if (lane == 0) q.subsum[(int64_t)b * q.nsub + un] = sacc;
  }
  __threadfence_block();
  __syncthreads();
  if (warp == 0) group_draw<DT>(q, b);
  if (threadIdx.x == 0) {
    tp.accept_len[b] = s_depth;
    if (tp.path)
      for (int d = s_depth; d < tp.Dmax; ++d) tp.path[(int64_t)b * tp.Dmax + d] = -1;
    // the last residual step's mass; 1 (the mass of p_u) when u rejected nothing
    if (tp.resid_mass) tp.resid_mass[b] = s_Zlast >= 0.0 ? (float)s_Zlast : 1.f;
  }
}

}  // namespace

template <int DT>
cudaError_t launch_tree_dt(const TreeParams& tp, cudaStream_t s) {
  tree_walk_kernel<DT><<<tp.B, kTreeThreads, 0, s>>>(tp);
  return cudaGetLastError();
}

template cudaError_t launch_tree_dt<0>(const TreeParams& tp, cudaStream_t s);
template cudaError_t launch_tree_dt<1>(const TreeParams& tp, cudaStream_t s);

}  // namespace ssd
