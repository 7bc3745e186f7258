// ssd_stream.cu -- the streaming pass over full-vocabulary logit rows.
//
// One persistent CTA per SM takes an equal, contiguous share of the
// flattened (row, 1024-element unit) space.  A producer warp streams the
// share through a ring of 16 KB shared-memory stages with 1-D bulk copies
// (cp.async.bulk + mbarrier transaction counts); eight consumer warps reduce
// each row piece to
//   * the online-softmax normaliser: max raw logit m and
//     s = sum_y 2^(z_y * c - fl(m*c)), c = log2(e)/T, accumulated with
//     per-thread compensated sums ([SD-7.3] §7.3.2: the target and draft
//     distributions at every position);
//   * for draft rows, the top-(F_j+1) raw logits (ties to the lower index):
//     the bonus-token guesses and the Saguaro cached set
//     ([SSD-note] §"怎么猜奖励 token", §"Saguaro 优化二：Saguaro 采样").
// Rows split across CTAs are merged by the last CTA to finish them (atomic
// arrival counter); the last row of a sequence to be finalised runs the
// sequence epilogue: the warp-parallel accept test min(1, p/q') with the
// first-rejection scan ([SD-7.3] §7.3.3; [SD-blog] §"三、接受概率为什么是对的"),
// or, for Saguaro sampling, the parameters of the continuation draw.
//
// Sources: [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈";
// [SD-7.3] "7.3 Speculative Decoding：投机采样加速";
// [SD-blog] "推测解码：用一个“小模型”骗出 3 倍推理速度".

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd_cache_dev.cuh"
#include "ssd_cdf_dev.cuh"
#include "ssd_device.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

constexpr float kNegInf = -INFINITY;
constexpr float kPosInf = INFINITY;

template <int TOPK>
struct alignas(16) PieceRed {
  long long chunk;  // the piece's chunk, -1: no more pieces
  float c;          // log2(e) / T of the piece's sequence
  float m[kConsumerWarps];
  float hi[kConsumerWarps];
  float lo[kConsumerWarps];
  float tv[kConsumerWarps][TOPK > 0 ? TOPK : 1];
  int ti[kConsumerWarps][TOPK > 0 ? TOPK : 1];
};

// Geometry of one pipeline stage: the element range [e0, e1) of row `row`
// and its 16-byte-aligned interior [a0, a1) (byte addresses).
struct Stage {
  int e0, e1;
  uintptr_t b0, a0, a1;
};

// What the consumer warps need of a stage, written by the producer next to
// the stage and published by the same mbarrier arrival: the aligned vectors
// in shared memory (nvec, holding elements ei0 ...), and for the unaligned
// head and tail the element range [e0, e1) at global address b0.
struct StageDesc {
  int nvec, ei0, e0, e1;
  uintptr_t b0;
};

template <int DT>
__device__ __forceinline__ const void* tensor_of(const StreamParams& p, int64_t row,
                                                 int64_t& trow, bool& is_t) {
  const int64_t g = row / p.rpg;
  const int jr = (int)(row - g * p.rpg);
  is_t = jr < p.nt;
  if (is_t) {
    trow = g * (p.K + 1) + jr;
    return p.tgt;
  }
  trow = g * p.Kq + (jr - p.nt);
  return p.dft;
}

// Row-level geometry, computed once per row piece.
struct RowGeom {
  const char* rp;  // address of element 0 of the row
  int64_t ur;      // first unit of the row in the flattened unit space
  bool is_t;       // target row (else draft row)
};

template <int DT>
__device__ __forceinline__ RowGeom row_geom(const StreamParams& p, int64_t row) {
  RowGeom rg;
  int64_t trow;
  const void* base = tensor_of<DT>(p, row, trow, rg.is_t);
  rg.rp = row_ptr(base, trow, rg.is_t ? p.t_stride : p.d_stride, Elem<DT>::kSize);
  rg.ur = row * p.upr;
  return rg;
}

// Stage of units [u, un) of the row: element range and aligned interior.
template <int DT>
__device__ __forceinline__ Stage stage_of(const RowGeom& rg, int V, int64_t u, int64_t un) {
  Stage st;
  st.e0 = (int)((u - rg.ur) * kUnitA);
  st.e1 = (int)min((int64_t)V, (un - rg.ur) * kUnitA);
  st.b0 = (uintptr_t)(rg.rp + (int64_t)st.e0 * Elem<DT>::kSize);
  const uintptr_t b1 = (uintptr_t)(rg.rp + (int64_t)st.e1 * Elem<DT>::kSize);
  st.a0 = (st.b0 + 15) & ~(uintptr_t)15;
  st.a1 = b1 & ~(uintptr_t)15;
  if (st.a1 <= st.a0) st.a0 = st.a1 = st.b0;  // no aligned interior: all scalar
  return st;
}

// Per-thread accumulator of one row piece.
template <int TOPK>
struct Acc {
  float m, mc, hi, lo;
  float tv[TOPK > 0 ? TOPK : 1];
  int ti[TOPK > 0 ? TOPK : 1];
  __device__ __forceinline__ void reset() {
    m = kNegInf;
    mc = kNegInf;
    hi = 0.f;
    lo = 0.f;
#pragma unroll
    for (int k = 0; k < (TOPK > 0 ? TOPK : 1); ++k) {
      tv[k] = kNegInf;
      ti[k] = 0x7fffffff;
    }
  }
  // Raise the running maximum to vm (rescaling the sum).
  __device__ __forceinline__ void raise_max(float vm, float c) {
    const float mcn = __fmul_rn(vm, c);
    if (m != kNegInf) pair_scale(hi, lo, exp2f(mc - mcn));
    m = vm;
    mc = mcn;
  }
  // Kahan-style compensated accumulation of a (positive) partial sum.
  __device__ __forceinline__ void add(float v) {
    const float y = v - lo;
    const float t = hi + y;
    lo = (t - hi) - y;
    hi = t;
  }
};

// Two floats as one 64-bit register pair, for the packed f32x2 instructions.
__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// Softmax accumulator of one consumer thread: running maximum m, its scaled
// offset mc = fl(m*c) and the compensated sum (hi, lo) of 2^(z*c - mc).
struct SAcc {
  float m, mc, hi, lo;
  __device__ __forceinline__ void reset() {
    m = kNegInf;
    mc = kNegInf;
    hi = 0.f;
    lo = 0.f;
  }
  __device__ __forceinline__ void raise_max(float vm, float c) {
    const float mcn = __fmul_rn(vm, c);
    if (m != kNegInf) pair_scale(hi, lo, exp2f(mc - mcn));
    m = vm;
    mc = mcn;
  }
  __device__ __forceinline__ void add(float v) {
    const float y = v - lo;
    const float t = hi + y;
    lo = (t - hi) - y;
    hi = t;
  }
  // n logits (all finite, or -inf padding) whose maximum is vm.  For n a
  // multiple of 4 the exponent arguments and the pairwise tree sum use the
  // packed f32x2 FMA / add (the same roundings, in the same order).
  template <int N>
  __device__ __forceinline__ void take(const float* x, float vm, float c) {
    if (vm > m) raise_max(vm, c);
    float e[N];
    if constexpr (N % 4 == 0) {
      const unsigned long long cc = pack2(c, c), mm = pack2(-mc, -mc);
#pragma unroll
      for (int k = 0; k < N; k += 2) {
        unsigned long long d;
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pack2(x[k], x[k + 1])), "l"(cc),
            "l"(mm));
        float a0, a1;
        unpack2(d, a0, a1);
        e[k] = ex2(a0);
        e[k + 1] = ex2(a1);
      }
#pragma unroll
      for (int w = N / 2; w > 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; k += 2) {
          unsigned long long t;
          asm("add.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(pack2(e[k], e[k + 1])),
              "l"(pack2(e[k + w], e[k + w + 1])));
          unpack2(t, e[k], e[k + 1]);
        }
      e[0] += e[1];
    } else {
#pragma unroll
      for (int k = 0; k < N; ++k) e[k] = ex2(fmaf(x[k], c, -mc));
#pragma unroll
      for (int w = N / 2; w > 0; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) e[k] += e[k + w];
      if (N % 2 == 1 && N > 1) e[0] += e[N - 1];
    }
    add(e[0]);
  }
  // As take<N> for NV vectors of N / NV logits each, also returning each
  // vector's sum (at this thread's offset mc after the call); the thread's
  // total is the sum of the vector sums.
  template <int N, int NV>
  __device__ __forceinline__ void take_split(const float* x, float vm, float c, float* vs) {
    constexpr int W = N / NV;
    if (vm > m) raise_max(vm, c);
    float e[N];
#pragma unroll
    for (int k = 0; k < N; ++k) e[k] = ex2(fmaf(x[k], c, -mc));
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      float* v = e + q * W;
#pragma unroll
      for (int w = W / 2; w > 0; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) v[k] += v[k + w];
      vs[q] = v[0];
    }
    float t[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) t[q] = vs[q];
#pragma unroll
    for (int w = NV / 2; w > 0; w >>= 1)
#pragma unroll
      for (int q = 0; q < w; ++q) t[q] += t[q + w];
    add(t[0]);
  }
};

// The warp's sums of NV sub-units (one 32-vector run each, lane l holding
// vector l's sum vs[q] at its own offset mc): rescaled to the warp's largest
// offset and stored with it as (sum, offset) for sub-units su0 + q * step of
// row `row`.  Called by all 32 lanes.
template <int NV>
__device__ __forceinline__ void store_subunits(const StreamParams& p, int64_t row, int su0,
                                               int step, const float* vs, float mc) {
  const int lane = threadIdx.x & 31;
  const float mcw = unord_float(__reduce_max_sync(0xffffffffu, ord_float(mc)));
  const float sc = (mc == -INFINITY || mcw == -INFINITY) ? 0.f : ex2(mc - mcw);
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    float v = vs[q] * sc;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int su = su0 + q * step;
    if (lane == 0 && SSD_CHK(su < p.nsu && row < p.NR, p.dbg, 11, su, row))
      p.usum[row * p.nsu + su] = make_float2(v, mcw);
  }
}

// One warp-wide top list: lane l < TOPK holds the l-th best candidate by
// (logit desc, index asc); (cv, ci) is the TOPK-th entry, known to all lanes.
// Candidates are offered by ballot and inserted cooperatively, so a lane's
// rare candidate costs the warp a handful of shuffles instead of a predicated
// per-thread insertion.
template <int TOPK>
struct WarpList {
  float lv, cv;
  int li, ci;
  float hv;  // the head (best entry), known to all lanes
  int R;     // entries the row needs (F_j + 1 <= TOPK); the cut is entry R - 1
  __device__ __forceinline__ void reset(int need) {
    lv = cv = hv = kNegInf;
    li = ci = 0x7fffffff;
    R = need;
  }
  // -inf marks padding (empty lanes, partial vectors): never a candidate.
  __device__ __forceinline__ bool qualifies(float x, int i, float ccut) const {
    return x != kNegInf && cand_before(x, i, cv, ci) && x >= ccut;
  }
  __device__ __forceinline__ void insert(float v, int i) {
    const int lane = threadIdx.x & 31;
    const bool before = lane < R && cand_before(lv, li, v, i);
    const int pos = __popc(__ballot_sync(0xffffffffu, before));
    if (pos >= R) return;  // warp-uniform
    if (pos == 0) hv = v;
    const float upv = __shfl_up_sync(0xffffffffu, lv, 1);
    const int upi = __shfl_up_sync(0xffffffffu, li, 1);
    if (lane > pos && lane < R) {
      lv = upv;
      li = upi;
    } else if (lane == pos) {
      lv = v;
      li = i;
    }
    cv = __shfl_sync(0xffffffffu, lv, R - 1);
    ci = __shfl_sync(0xffffffffu, li, R - 1);
  }
  // A lower bound on the TOPK-th largest logit of a block: the TOPK-th
  // largest of the 32 lane maxima (at least TOPK logits of the block reach
  // it).  Used while the list is still empty, so that the first block does not
  // flood it with candidates.
  __device__ __forceinline__ float boot_bound(float vm) const {
    const int lane = threadIdx.x & 31;
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float o = __shfl_sync(0xffffffffu, vm, j);
      rank += (o > vm || (o == vm && j < lane)) ? 1 : 0;
    }
    const unsigned m = __ballot_sync(0xffffffffu, rank == R - 1);
    return __shfl_sync(0xffffffffu, vm, __ffs(m) - 1);
  }
  // Offer the lane's logits held as NV raw 16-byte vectors raw[q] (element k
  // of vector q has index idx0 + q * kstride + k; vm is the maximum over all
  // of them, vq[q] the maximum of vector q; padding is -inf).  Called by all
  // 32 lanes.  The common case -- no lane holds a candidate -- costs one vote.
  template <int DT, int NV>
  __device__ __forceinline__ void offer(const uint4* raw, const float* vq, float vm, int idx0,
                                        int kstride, float ccut);
  // The rare path: locate candidates vector by vector (one vote each), then
  // element by element with a runtime index.
  template <int DT, int NV>
  __device__ __forceinline__ void offer_rare(const uint4* raw, const float* vq, int idx0,
                                             int kstride, float ccut, bool anyq) {
    constexpr int VEC = Elem<DT>::kVec;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const uint4 rq = raw[q];
      const float mq = vq[q];
      if (!__any_sync(0xffffffffu, anyq && mq != kNegInf && mq >= cv && mq >= ccut)) continue;
#pragma unroll 1
      for (int k = 0; k < VEC; ++k) {
        const float xk = vec_elem<DT>(rq, k);
        const int ik = idx0 + q * kstride + k;
        unsigned m = __ballot_sync(0xffffffffu, anyq && mq != kNegInf && qualifies(xk, ik, ccut));
        while (m) {
          const int L = __ffs(m) - 1;
          const float v = __shfl_sync(0xffffffffu, xk, L);
          const int i = __shfl_sync(0xffffffffu, ik, L);
          insert(v, i);
          m &= m - 1;
        }
      }
    }
  }
  // One logit per lane (unaligned stage fragments); -inf is padding.
  __device__ __forceinline__ void offer1(float x, int idx, float ccut) {
    unsigned m = __ballot_sync(0xffffffffu, qualifies(x, idx, ccut));
    while (m) {
      const int L = __ffs(m) - 1;
      insert(__shfl_sync(0xffffffffu, x, L), __shfl_sync(0xffffffffu, idx, L));
      m &= m - 1;
    }
  }
};

template <int TOPK>
template <int DT, int NV>
__device__ __forceinline__ void WarpList<TOPK>::offer(const uint4* raw, const float* vq, float vm,
                                                      int idx0, int kstride, float ccut) {
  const bool anyq = vm != kNegInf && vm >= cv && vm >= ccut;
  if (!__any_sync(0xffffffffu, anyq)) return;
  offer_rare<DT, NV>(raw, vq, idx0, kstride, ccut, anyq);
}

// The R-th largest list head of piece `piece` on the CTA's board (one entry
// per consumer warp, (piece << 32) | ordered float), or -inf when fewer than
// R warps have published one.  Called by all 32 lanes.
__device__ __forceinline__ float heads_cut(const unsigned long long* board, uint32_t piece,
                                           int R) {
  const int lane = threadIdx.x & 31;
  const unsigned long long hw =
      lane < kConsumerWarps ? *reinterpret_cast<const volatile unsigned long long*>(&board[lane])
                            : ~0ull;
  const float h = (hw >> 32) == piece ? unord_float((uint32_t)hw) : kNegInf;
  int rank = 0;
#pragma unroll
  for (int j = 0; j < kConsumerWarps; ++j) {
    const float o = __shfl_sync(0xffffffffu, h, j);
    rank += (o > h || (o == h && j < lane)) ? 1 : 0;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < kConsumerWarps && rank == R - 1);
  return hit ? __shfl_sync(0xffffffffu, h, __ffs(hit) - 1) : kNegInf;
}

// Fold one stored partial into a lane's accumulator (row merges).
template <int TOPK>
__device__ __forceinline__ void fold_partial(Acc<TOPK>& a, const RowPartial* pp, float c,
                                             bool top) {
  const float m2 = __ldcg(&pp->m);
  const float h2 = __ldcg(&pp->s_hi);
  const float l2 = __ldcg(&pp->s_lo);
  if (m2 != kNegInf) {
    float hh = h2, ll = l2;
    const float mc2 = __fmul_rn(m2, c);
    if (m2 > a.m) {
      a.raise_max(m2, c);
    } else if (mc2 != a.mc) {
      pair_scale(hh, ll, exp2f(mc2 - a.mc));
    }
    pair_add(a.hi, a.lo, hh, ll);
  }
  if constexpr (TOPK > 0) {
    if (top) {
#pragma unroll
      for (int k = 0; k < TOPK; ++k) {
        const float v = __ldcg(&pp->tv[k]);
        const int i = __ldcg(&pp->ti[k]);
        if (v != kNegInf) topk_insert_ordered<TOPK>(a.tv, a.ti, v, i);
      }
    }
  }
}

// Warp roles: warps 0..kConsumerWarps-1 reduce staged data, warp
// kConsumerWarps takes chunks from the global counter and issues their bulk
// copies, and kEpilogueWarps epilogue warps (piece p to warp p mod
// kEpilogueWarps) merge each piece's per-warp results and do all
// global-memory epilogue work, so the consumer warps never wait for it.
// Piece results pass through a queue of kPieceSlots shared-memory slots
// guarded by mbarriers.
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarp = kConsumerWarps + 1;  // the first epilogue warp
constexpr int kEpilogueWarps = 2;
constexpr int kStreamThreads = (kConsumerWarps + 1 + kEpilogueWarps) * 32;

// ---- per-sequence temperature -----------------------------------------------------------
// A sequence is greedy (the limit T -> 0) when its temperature is 0 -- or
// negative or not finite, which also sets SSD_DEV_BAD_TEMPERATURE.  A greedy
// sequence's sums (unused) take T = 1.
__device__ __forceinline__ bool seq_greedy(const StreamParams& p, int64_t g) {
  if (p.T_rows == nullptr) return p.greedy_all != 0;
  const float T = __ldg(p.T_rows + g);
  return !(T > 0.f && T <= 3.402823466e38f);
}

// log2(e) / T rounded once from fp64, as the host computes the scale of a
// single temperature (kept out of line: the fp64 division is long).
__device__ __noinline__ float scale_of_temperature(float T) {
  return (T > 0.f && T <= 3.402823466e38f) ? (float)(1.4426950408889634 / (double)T)
                                           : 1.4426950408889634f;
}

// log2(e) / T of sequence g: the scale of every exponent of its rows.
__device__ __forceinline__ float seq_scale(const StreamParams& p, int64_t g) {
  if (p.T_rows == nullptr) return p.c;
  return scale_of_temperature(__ldg(p.T_rows + g));
}

// Top-list entries row `row` (row jr of sequence g) needs: F_j + 1 on a draft
// row that feeds guesses or a Saguaro set, 1 (its argmax) on a target row of
// a greedy sequence, otherwise none.
__device__ __forceinline__ int row_need(const StreamParams& p, int64_t g, int jr) {
  if (jr < p.nt) return p.mode == kModeVerify && seq_greedy(p, g) ? 1 : 0;
  const int F = p.F[jr - p.nt];
  return (p.need_top && F > 0) ? F + 1 : 0;
}

// Greedy verification of sequence g (the limit T -> 0): x_i is accepted iff
// it is the argmax of target row i (ties to the lower index); the bonus is
// the argmax of the first rejected target row, or of row K when every draft
// is accepted.  Nothing is left to draw.  Warp 0 of the finishing CTA.
__device__ void greedy_epilogue(const StreamParams& p, int64_t g) {
  const int lane = threadIdx.x & 31;
  const int K = p.K;
  bool acc = true;
  if (lane < K) {
    const RowResult* rt = p.rowres + g * p.rpg + lane;
    acc = __ldcg(&rt->x) == __ldcg(&rt->ti[0]);
  }
  const unsigned rej = ~__ballot_sync(0xffffffffu, acc) & (K >= 32 ? 0xffffffffu : ((1u << K) - 1u));
  const int k = rej ? __ffs(rej) - 1 : K;
  if (lane != 0) return;
  if (!SSD_CHK(g < p.B && k >= 0 && k <= K, p.dbg, 8, g, k)) return;
  p.accept_len[g] = k;
  const int t = __ldcg(&p.rowres[g * p.rpg + k].ti[0]);
  p.bonus[g] = t;
  if (p.resid_mass) p.resid_mass[g] = 1.f;
  if (p.rc.table != nullptr)  // the round's cache: look the outcome (k, t) up
    round_outcome(static_cast<const Slot*>(p.rc.table), p.rc.cap, g, k, t, p.B, p.rc.branch,
                  p.rc.all_hit, p.rc.cnt);
  if (p.T_rows != nullptr && p.status) {
    const float T = __ldg(p.T_rows + g);
    if (T != 0.f) atomicOr(p.status, SSD_DEV_BAD_TEMPERATURE);
  }
  GroupParams gp = {};
  gp.use_t = 0;  // no draw
  gp.use_d = 0;
  gp.theta = kPosInf;
  gp.itheta = -1;
  p.gparams[g] = gp;
  if (p.grp_ready) {
    __threadfence();
    flag_release(p.grp_ready + g);
  }
}

// ---- the sequence epilogue of ssd_verify (warp 0 of the finishing CTA) -----------------
__device__ void verify_epilogue(const StreamParams& p, int64_t g, float cf) {
  if (seq_greedy(p, g)) {
    greedy_epilogue(p, g);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int K = p.K;
  const double c = (double)cf;
  bool acc = true;
  if (lane < K) {
    const RowResult* rt = p.rowres + g * p.rpg + lane;
    const RowResult* rd = p.rowres + g * p.rpg + p.nt + lane;
    const int x = __ldcg(&rt->x);
    const double pt = exp2((double)__ldcg(&rt->zx) * c - (double)__ldcg(&rt->mc)) / __ldcg(&rt->s);
    const double sq = __ldcg(&rd->s);
    const double mcq = (double)__ldcg(&rd->mc);
    double qp = exp2((double)__ldcg(&rd->zx) * c - mcq) / sq;
    const int F = p.F[lane];
    const float Cl = p.C[lane];
    if (Cl < 1.f && F > 0) {
      double QS = 0.0;
      bool inS = false;
      for (int f = 0; f < F; ++f) {
        QS += (double)exp2f(fmaf(__ldcg(&rd->tv[f]), cf, -__ldcg(&rd->mc)));
        inS |= __ldcg(&rd->ti[f]) == x;
      }
      QS /= sq;
      qp = qp * (inS ? (double)Cl : 1.0) / (1.0 - (1.0 - (double)Cl) * QS);
    }
    const double r = pt / qp;
    const double u = uniform24(p.seeds[g], (uint32_t)g, (uint32_t)lane, 0u, p.round);
    acc = u < r;
  }
  const unsigned rej = ~__ballot_sync(0xffffffffu, acc) & (K >= 32 ? 0xffffffffu : ((1u << K) - 1u));
  const int k = rej ? __ffs(rej) - 1 : K;
  if (lane == 0) {
    if (!SSD_CHK(g < p.B && k >= 0 && k <= K, p.dbg, 8, g, k)) return;
    p.accept_len[g] = k;
    GroupParams gp;
    const RowResult* rt = p.rowres + g * p.rpg + k;
    gp.k = k;
    gp.use_t = 1;
    gp.row_t = g * (int64_t)(K + 1) + k;
    gp.mc_t = __ldcg(&rt->mc);
    gp.inv_st = (float)(1.0 / __ldcg(&rt->s));
    gp.sign_d = -1;
    gp.theta = kPosInf;
    gp.itheta = -1;
    if (k < K) {
      const RowResult* rd = p.rowres + g * p.rpg + p.nt + k;
      gp.use_d = 1;
      gp.row_d = g * (int64_t)p.Kq + k;
      gp.mc_d = __ldcg(&rd->mc);
      const double sq = __ldcg(&rd->s);
      double scale_out = 1.0 / sq, scale_in = 1.0 / sq;
      const int F = p.F[k];
      const float Ck = p.C[k];
      if (Ck < 1.f && F > 0) {
        double QS = 0.0;
        for (int f = 0; f < F; ++f)
          QS += (double)exp2f(fmaf(__ldcg(&rd->tv[f]), cf, -gp.mc_d));
        QS /= sq;
        const double gn = 1.0 / (1.0 - (1.0 - (double)Ck) * QS);
        scale_out = gn / sq;
        scale_in = gn * (double)Ck / sq;
        gp.theta = __ldcg(&rd->tv[F - 1]);
        gp.itheta = __ldcg(&rd->ti[F - 1]);
      }
      gp.scale_out = (float)scale_out;
      gp.scale_in = (float)scale_in;
    } else {
      gp.use_d = 0;
      gp.row_d = 0;
      gp.mc_d = 0.f;
      gp.scale_out = gp.scale_in = 0.f;
    }
    gp.u = uniform24(p.seeds[g], (uint32_t)g, (uint32_t)k, 1u, p.round);
    gp.c = cf;
    p.gparams[g] = gp;
    if (p.grp_ready) {
      __threadfence();
      flag_release(p.grp_ready + g);  // the group's draw may start
    }
  }
}

// Saguaro continuation draw: parameters of q' for branch row g.
__device__ void saguaro_epilogue(const StreamParams& p, int64_t g, const RowResult& rr,
                                 float cf) {
  GroupParams gp;
  gp.k = 0;
  gp.use_t = 0;
  gp.use_d = 1;
  gp.sign_d = 1;
  gp.row_t = 0;
  gp.row_d = g;
  gp.mc_t = 0.f;
  gp.inv_st = 0.f;
  gp.mc_d = rr.mc;
  gp.theta = kPosInf;
  gp.itheta = -1;
  double scale_out = 1.0 / rr.s, scale_in = 1.0 / rr.s;
  const int F = p.F[0];
  const float C = p.C[0];
  if (C < 1.f && F > 0) {
    double QS = 0.0;
    for (int f = 0; f < F; ++f) QS += (double)exp2f(fmaf(rr.tv[f], cf, -rr.mc));
    QS /= rr.s;
    const double gn = 1.0 / (1.0 - (1.0 - (double)C) * QS);
    scale_out = gn / rr.s;
    scale_in = gn * (double)C / rr.s;
    gp.theta = rr.tv[F - 1];
    gp.itheta = rr.ti[F - 1];
  }
  gp.scale_out = (float)scale_out;
  gp.scale_in = (float)scale_in;
  gp.u = uniform24(p.seeds[g], (uint32_t)g, (uint32_t)p.jpos, 2u, p.round);
  gp.c = cf;
  p.gparams[g] = gp;
  if (p.grp_ready) {
    __threadfence();
    flag_release(p.grp_ready + g);  // the row's draw may start
  }
}

// The unit sums of a Saguaro row's draw weight q'(y), from the sub-unit sums
// the streaming pass wrote: each sub-unit rescaled from its offset to the
// row's, times the weight outside the cached set S, plus the difference of
// the weights for the tokens of S (the top F of the row).  One warp; the
// row's draw parameters are published by lane 0 before.
template <int DT>
__device__ void saguaro_unit_sums(const StreamParams& p, const CdfParams& cq, int64_t g,
                                  const RowResult& rr, float c) {
  const int lane = threadIdx.x & 31;
  constexpr int kSpu = kUnitB / (32 * Elem<DT>::kVec);  // sub-units per unit
  const GroupParams gp = load_gp(cq.gp + g);
  const float2* us = p.usum + g * p.nsu;
  const int F = gp.theta != kPosInf ? p.F[0] : 0;
  for (int u = lane; u < cq.nsub; u += 32) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kSpu; ++k) {
      const int su = u * kSpu + k;
      if (su < p.nsu) {
        const float2 v = __ldcg(us + su);
        if (v.x > 0.f) sum += v.x * ex2(v.y - gp.mc_d);
      }
    }
    float w = sum * gp.scale_out;
    for (int f = 0; f < F; ++f)
      if (rr.ti[f] >= 0 && rr.ti[f] / kUnitB == u)
        w += (gp.scale_in - gp.scale_out) * ex2(fmaf(rr.tv[f], c, -gp.mc_d));
    if (SSD_CHK(g < cq.groups && u < cq.nsub, p.dbg, 12, g, u))
      cq.subsum[g * cq.nsub + u] = fmaxf(w, 0.f);
  }
  __syncwarp();
}

// Finalise row `row` from the merged (M, MC, S, top list) held by warp 0.
template <int DT, int TOPK>
__device__ void finalize_row(const StreamParams& p, const CdfParams& cq, int64_t row, float c,
                             float M, float MC, float Shi, float Slo, const Acc<TOPK>& a,
                             bool top, bool* cleared, volatile int* s_err) {
  const int lane = threadIdx.x & 31;
  const int64_t g = row / p.rpg;
  const int jr = (int)(row - g * p.rpg);
  const bool is_t = jr < p.nt;
  const int j = is_t ? jr : jr - p.nt;
  RowResult rr;
  rr.m = M;
  rr.mc = MC;
  rr.s = (double)Shi + (double)Slo;
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    const bool valid = TOPK > 0 && top && k < TOPK && a.tv[k < TOPK ? k : 0] != kNegInf;
    rr.tv[k] = valid ? a.tv[k < TOPK ? k : 0] : kNegInf;
    rr.ti[k] = valid ? a.ti[k < TOPK ? k : 0] : -1;
  }
  rr.x = -1;
  rr.zx = 0.f;
  if (p.tokens != nullptr && j < p.tokK) {
    int x = SSD_CHK(g < p.B && j < p.tokK, p.dbg, 3, g, j) ? p.tokens[g * p.tokK + j] : 0;
    if (x < 0 || x >= p.V) {
      if (lane == 0 && p.status) atomicOr(p.status, SSD_DEV_BAD_TOKEN);
      x = 0;
    }
    int64_t trow;
    bool it;
    const void* base = tensor_of<DT>(p, row, trow, it);
    const char* rp = row_ptr(base, trow, it ? p.t_stride : p.d_stride, Elem<DT>::kSize);
    rr.x = x;
    const uintptr_t ga = (uintptr_t)(rp + (int64_t)x * Elem<DT>::kSize);
    rr.zx = SSD_CHK(in_range(ga, ga + Elem<DT>::kSize, it ? p.t_lo : p.d_lo, it ? p.t_hi : p.d_hi),
                    p.dbg, 4, row, x) ? Elem<DT>::load_cg(rp, x) : 0.f;
  }
  if (lane == 0 && SSD_CHK(row < p.NR, p.dbg, 5, row, p.NR)) p.rowres[row] = rr;
  // bonus guesses: top-(F_j+1) minus the sampled token, truncated to F_j
  if (!is_t && p.guesses != nullptr && lane == 0) {
    const bool greedy = p.mode == kModeVerify && seq_greedy(p, g);
    const int F = p.F[j];
    int n = 0;
    const int64_t o = (g * p.nd + j) * (int64_t)p.Fmax;
    for (int k = 0; k < kMaxTopK && n < F; ++k) {
      if (rr.ti[k] < 0 || rr.ti[k] == rr.x) continue;
      if (!SSD_CHK(o + n < (int64_t)p.B * p.nd * p.Fmax && n < p.Fmax, p.dbg, 7, o + n, n)) break;
      p.guesses[o + n] = rr.ti[k];
      if (p.guess_q)
        p.guess_q[o + n] = greedy ? (rr.ti[k] == rr.ti[0] ? 1.f : 0.f)
                                  : (float)((double)exp2f(fmaf(rr.tv[k], c, -MC)) / rr.s);
      ++n;
    }
    for (; n < p.Fmax; ++n) {
      if (!SSD_CHK(o + n < (int64_t)p.B * p.nd * p.Fmax, p.dbg, 7, o + n, n)) break;
      p.guesses[o + n] = -1;
      if (p.guess_q) p.guess_q[o + n] = 0.f;
    }
  }
  if (!is_t && p.rc.table != nullptr && p.guesses != nullptr && p.F[j] > 0) {
    // the round's cache: guess f of this row (entry f of the list, or f + 1
    // once the drafted token is passed) -> key (sequence, position, guess),
    // value its index in the guesses array; one lane per guess, after every
    // CTA has cleared its slice of the table
    const int F = p.F[j];
    if (!*cleared) {
      int ok = 0;
      if (lane == 0)
        ok = count_wait(p.rc.cleared, (int)gridDim.x * kEpilogueWarps, s_err, p.status);
      *cleared = __shfl_sync(0xffffffffu, ok, 0) != 0;
    }
    int sx = kMaxTopK;
    for (int k = F; k >= 0; --k)
      if (rr.ti[k] == rr.x) sx = k;
    if (*cleared && lane < F) {
      const int e = lane < sx ? lane : lane + 1;
      const int tok = e < kMaxTopK ? rr.ti[e] : -1;
      if (tok >= 0)
        cache_insert(static_cast<Slot*>(p.rc.table), p.rc.cap, pack_key((int)g, j, tok),
                     (int)((g * p.nd + j) * p.Fmax + lane), p.status);
    }
  }
  if (p.mode == kModeTopF) return;
  // sequence arrival
  int last = 0;
  if (lane == 0) {
    __threadfence();
    last = SSD_CHK(g < p.B, p.dbg, 9, g, p.B) ? atomicAdd(p.grp_cnt + g, 1) == p.rpg - 1 : 0;
    if (last) __threadfence();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  if (p.mode == kModeVerify) {
    verify_epilogue(p, g, c);
  } else {
    if (lane == 0) saguaro_epilogue(p, g, rr, c);
    if (p.usum != nullptr) {
      // the row's unit sums from the streaming pass, then its draw
      __syncwarp();
      saguaro_unit_sums<DT>(p, cq, g, rr, c);
      group_draw<DT>(cq, g);
    }
  }
}

constexpr int kPieceSlots = 4;
static_assert(kPieceSlots % kEpilogueWarps == 0, "a slot belongs to one epilogue warp");
// Chunk of each piece, written by the producer before the piece's first
// stage is published.  The producer runs at most kStagesA + 1 pieces ahead
// of the consumer warps, so a queue this long is never overwritten early.
constexpr int kPieceQueue = 16;
static_assert(kPieceQueue > kStagesA + 1, "piece queue shorter than the pipeline");

// A piece as the producer hands it to the consumer warps (chunk -1: the end).
struct PieceDesc {
  long long chunk;
  // a chunk of rows
  int64_t row, pu0, pu1;
  const char* rp;  // element 0 of the row
  int jr;          // row within its group
  int kch;         // chunk of the row
  float c;         // log2(e) / T of the row's sequence
  int need;        // top-list entries the row needs
  // the row's group; for a chunk of the draws also its units [u0, u1) and
  // the group's parameters
  int64_t g;
  int u0, u1;
  GroupParams gp;
};

// Units [pu0, pu1) of row `row` that chunk c covers (chunks in the order
// (chunk of row, row), so a row's later chunks start long after its first).
__device__ __forceinline__ void chunk_geom(const StreamParams& p, long long c, int64_t& row,
                                           int& k, int64_t& pu0, int64_t& pu1) {
  k = (int)(c / p.NR);
  row = c - (int64_t)k * p.NR;
  pu0 = row * p.upr + (int64_t)k * p.clen;
  pu1 = min(pu0 + p.clen, (row + 1) * p.upr);
}

template <int DT, int TOPK>
__global__ void __launch_bounds__(kStreamThreads, 1)
    stream_kernel(const __grid_constant__ VerifyParams vp) {
  const StreamParams& p = vp.s;
  const CdfParams& cq = vp.q;  // the draws (cq.nchunks == 0: none)
  const long long nS = p.nchunks;
  const long long ntot = nS + cq.nchunks;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStagesA * kStageBytes);
  uint64_t* empty = full + kStagesA;
  uint64_t* pfull = empty + kStagesA;
  uint64_t* pempty = pfull + kPieceSlots;
  PieceRed<TOPK>* slots = reinterpret_cast<PieceRed<TOPK>*>(pempty + kPieceSlots);
  __shared__ int s_err;
  // Top-list pruning bound shared by the CTA's warps: (piece << 32) |
  // ordered float.  Piece numbers only increase within a CTA, so a value of
  // another piece is never mistaken for the current piece's.
  __shared__ unsigned long long s_cut;
  // Each consumer warp's list head, (piece << 32) | ordered float: the heads
  // of one piece are distinct logits of its row, so the R-th largest of them
  // is a lower bound on the row's R-th best.
  __shared__ unsigned long long s_head[kConsumerWarps];
  __shared__ PieceDesc s_pq[kPieceQueue];
  __shared__ StageDesc s_sd[kStagesA];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int ups = kStageBytes / (kUnitA * Elem<DT>::kSize);  // units per stage

  if (tid == 0) {
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    for (int i = 0; i < kPieceSlots; ++i) {
      mbar_init(pfull + i, kConsumerWarps);
      mbar_init(pempty + i, 1);
    }
    s_err = 0;
    s_cut = 0ull;
    for (int i = 0; i < kConsumerWarps; ++i) s_head[i] = ~0ull;  // a tag no piece has
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int n = 0;
      // the first round of chunks is static (chunk = CTA): a CTA's first
      // copy does not wait behind every CTA's atomic on the counter
      unsigned long long next = blockIdx.x;
      for (int piece = 0;; ++piece) {
        long long c = next < (unsigned long long)ntot ? (long long)next : -1ll;
        PieceDesc& d = s_pq[piece % kPieceQueue];
        if (c >= nS) {
          // a chunk of the draws: wait until the epilogue of its group has
          // published the group's parameters
          int64_t g;
          int u0, u1;
          cdf_chunk_geom(cq, c - nS, g, u0, u1);
          if (!(g >= 0 && g < cq.groups && u0 < u1) ||
              !flag_wait(p.grp_ready + g, &s_err, p.status)) {
            c = -1;
          } else {
            d.g = g;
            d.u0 = u0;
            d.u1 = u1;
            d.gp = load_gp(cq.gp + g);
          }
        }
        d.chunk = c;
        if (c < 0) {
          // end marker: one stage without data
          const int slot = n % kStagesA;
          if (n >= kStagesA) mbar_wait(empty + slot, ((n / kStagesA) - 1) & 1, &s_err, p.status);
          mbar_arrive(full + slot);
          ++n;
          break;
        }
        // the following chunk, fetched early (the counter hands out chunks
        // after the static first round)
        next = gridDim.x + atomicAdd(p.chunk_ctr, 1ull);
        if (c >= nS) {
          constexpr int ES = Elem<DT>::kSize;
          const char* rt = d.gp.use_t ? row_ptr(cq.tgt, d.gp.row_t, cq.t_stride, ES) : nullptr;
          const char* rd = d.gp.use_d ? row_ptr(cq.dft, d.gp.row_d, cq.d_stride, ES) : nullptr;
          const DrawLayout lay = draw_layout<DT>(d.gp);
          for (int u = d.u0, un = 0; u < d.u1; u = un) {
            un = min(u + lay.ups, d.u1);
            const int slot = n % kStagesA;
            if (n >= kStagesA) mbar_wait(empty + slot, ((n / kStagesA) - 1) & 1, &s_err, p.status);
            cdf_issue_stage<DT>(cq, rt, rd, u, un, ring + slot * kStageBytes, lay, full + slot,
                                &s_err);
            ++n;
          }
          continue;
        }
        int64_t row, pu0, pu1;
        int k;
        chunk_geom(p, c, row, k, pu0, pu1);
        const RowGeom rg = row_geom<DT>(p, row);
        // published to the consumers by the arrival on the piece's first stage
        d.row = row;
        d.pu0 = pu0;
        d.pu1 = pu1;
        d.rp = rg.rp;
        const int64_t g = row / p.rpg;
        d.g = g;
        d.jr = (int)(row - g * p.rpg);
        d.kch = k;
        d.c = seq_scale(p, g);
        d.need = TOPK > 0 ? row_need(p, g, d.jr) : 0;
        for (int64_t u = pu0, un = 0; u < pu1; u = un) {
          un = min(u + ups, pu1);
          const Stage st = stage_of<DT>(rg, p.V, u, un);
          const int slot = n % kStagesA;
          if (n >= kStagesA) mbar_wait(empty + slot, ((n / kStagesA) - 1) & 1, &s_err, p.status);
          StageDesc& sd = s_sd[slot];
          sd.nvec = (int)((st.a1 - st.a0) >> 4);
          sd.ei0 = st.e0 + (int)((st.a0 - st.b0) / Elem<DT>::kSize);
          sd.e0 = st.e0;
          sd.e1 = st.e1;
          sd.b0 = st.b0;
          const uint32_t bytes = (uint32_t)(st.a1 - st.a0);
          const bool tsrc = rg.is_t;
          (void)tsrc;  // read by the bounds-checked build only
          if (bytes > 0 && !s_err &&
              SSD_CHK(in_range(st.a0, st.a1, tsrc ? p.t_lo : p.d_lo, tsrc ? p.t_hi : p.d_hi),
                      p.dbg, 1, st.a0, st.a1)) {
            mbar_arrive_expect_tx(full + slot, bytes);
            bulk_g2s(ring + slot * kStageBytes, reinterpret_cast<const void*>(st.a0), bytes,
                     full + slot);
          } else {
            mbar_arrive(full + slot);
          }
          ++n;
        }
      }
      // do not leave while copies into this CTA's shared memory are in flight
      for (int q = max(0, n - kStagesA); q < n; ++q)
        mbar_wait(full + (q % kStagesA), (q / kStagesA) & 1, &s_err, p.status);
    }
    return;
  }

  if (warp >= kEpilogueWarp) {
    // ---------------- epilogue: merge, publish, finalise ----------------
    bool cleared = true;  // the round's cache table is cleared (or there is none)
    if (p.rc.table != nullptr) {
      // clear this warp's share of the CTA's slice of the table before the
      // first piece arrives; inserts wait until every share is done
      const int64_t per = (p.rc.cap + gridDim.x - 1) / gridDim.x;
      const int64_t s0 = (int64_t)blockIdx.x * per;
      const int64_t s1 = min(p.rc.cap, s0 + per);
      Slot* tab = static_cast<Slot*>(p.rc.table);
      for (int64_t i = s0 + (warp - kEpilogueWarp) * 32 + lane; i < s1; i += kEpilogueWarps * 32)
        slot_clear(tab + i);
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        atomicAdd(p.rc.cleared, 1);
      }
      cleared = false;
    }
    for (int piece = warp - kEpilogueWarp;; piece += kEpilogueWarps) {
      const int slot = piece % kPieceSlots;
      if (!mbar_wait(pfull + slot, (piece / kPieceSlots) & 1, &s_err, p.status)) break;
      const PieceRed<TOPK>& R = slots[slot];
      const long long chunk = R.chunk;
      if (chunk < 0) break;
      if (chunk >= nS) {
        // a chunk of the draws: its unit sums are stored; count it into its
        // group, and draw if it completes the group
        int64_t g;
        int u0, u1;
        cdf_chunk_geom(cq, chunk - nS, g, u0, u1);
        __syncwarp();
        if (lane == 0) mbar_arrive(pempty + slot);
        cdf_chunk_done<DT>(cq, g, u1 - u0);
        continue;
      }
      int64_t row, pu0, pu1;
      int kch;
      chunk_geom(p, chunk, row, kch, pu0, pu1);
      const int64_t g = row / p.rpg;
      const int jr = (int)(row - g * p.rpg);
      const float c = R.c;
      const int need = TOPK > 0 ? row_need(p, g, jr) : 0;  // list entries the row needs
      const bool top = need > 0;
      Acc<TOPK> b;
      b.reset();
      if (lane < kConsumerWarps) {
        b.m = R.m[lane];
        b.mc = b.m == kNegInf ? kNegInf : __fmul_rn(b.m, c);
        b.hi = R.hi[lane];
        b.lo = R.lo[lane];
        if (TOPK > 0 && top) {
#pragma unroll
          for (int k = 0; k < (TOPK > 0 ? TOPK : 1); ++k) {
            b.tv[k] = R.tv[lane][k];
            b.ti[k] = R.ti[lane][k];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(pempty + slot);  // the slot may be refilled
      float M, MC, Shi, Slo;
      warp_softmax_merge(b.m, b.mc, b.hi, b.lo, c, M, MC, Shi, Slo);
      if constexpr (TOPK > 0) {
        if (top) warp_topk_merge<TOPK>(b.tv, b.ti, need);
      }
      if (p.nch == 1) {
        finalize_row<DT, TOPK>(p, cq, row, c, M, MC, Shi, Slo, b, top, &cleared, &s_err);
        continue;
      }
      if constexpr (TOPK > 0) {
        // the chunk's R-th best logit bounds the row's cut: later chunks of
        // the row start from it
        if (top && lane == 0) {
          float v = kNegInf;
#pragma unroll
          for (int k = 0; k < (TOPK > 0 ? TOPK : 1); ++k) v = k == need - 1 ? b.tv[k] : v;
          if (v != kNegInf) atomicMax(p.row_cut + row, ord_float(v));
        }
      }
      // row split into chunks: publish the partial, the last arrival merges
      if (!SSD_CHK(row < p.NR && kch < p.nch, p.dbg, 6, row, kch)) continue;
      RowPartial* slotp = p.partials + (row * p.nch + kch);
      if (lane == 0) {
        slotp->m = M;
        slotp->s_hi = Shi;
        slotp->s_lo = Slo;
#pragma unroll
        for (int k = 0; k < (TOPK > 0 ? TOPK : 1); ++k) {
          slotp->tv[k] = (TOPK > 0 && top) ? b.tv[k] : kNegInf;
          slotp->ti[k] = (TOPK > 0 && top) ? b.ti[k] : 0x7fffffff;
        }
      }
      int last = 0;
      if (lane == 0) {
        __threadfence();
        last = atomicAdd(p.row_cnt + row, 1) == p.nch - 1;
        if (last) __threadfence();
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      Acc<TOPK> mrg;
      mrg.reset();
      for (int cc = lane; cc < p.nch; cc += 32)
        fold_partial<TOPK>(mrg, p.partials + (row * p.nch + cc), c, top);
      warp_softmax_merge(mrg.m, mrg.mc, mrg.hi, mrg.lo, c, M, MC, Shi, Slo);
      if constexpr (TOPK > 0) {
        if (top) warp_topk_merge<TOPK>(mrg.tv, mrg.ti, need);
      }
      finalize_row<DT, TOPK>(p, cq, row, c, M, MC, Shi, Slo, mrg, top, &cleared, &s_err);
    }
    return;
  }

  // ---------------- consumers ----------------
  SAcc a;
  WarpList<(TOPK > 0 ? TOPK : 1)> wl;
  constexpr int VEC = Elem<DT>::kVec;
  int slot = 0;         // ring stage of the next stage
  uint32_t phase = 0;   // its mbarrier phase parity
  for (int piece = 0;; ++piece) {
    // the piece's first stage (or the end marker) publishes its chunk
    bool ok = mbar_wait(full + slot, phase, &s_err, p.status);
    const volatile PieceDesc& d = s_pq[piece % kPieceQueue];
    const long long chunk = ok ? d.chunk : -1ll;
    const int ps = piece % kPieceSlots;
    if (chunk < 0) {
      // hand an end marker to every epilogue warp (the next kEpilogueWarps pieces)
      for (int q = piece; q < piece + kEpilogueWarps; ++q) {
        const int qs = q % kPieceSlots;
        if (lane == 0 && q >= kPieceSlots)
          mbar_wait(pempty + qs, ((q / kPieceSlots) - 1) & 1, &s_err, p.status);
        if (warp == 0 && lane == 0) slots[qs].chunk = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull + qs);
      }
      break;
    }
    if (chunk >= nS) {
      // ---- a chunk of the draws: the weight sums of its units ----
      const PieceDesc& dn = s_pq[piece % kPieceQueue];  // published by the stage's arrival
      const int64_t g = dn.g;
      const int u0 = dn.u0, u1 = dn.u1;
      const GroupParams gp = dn.gp;
      constexpr int ES = Elem<DT>::kSize;
      const char* rt = gp.use_t ? row_ptr(cq.tgt, gp.row_t, cq.t_stride, ES) : nullptr;
      const char* rd = gp.use_d ? row_ptr(cq.dft, gp.row_d, cq.d_stride, ES) : nullptr;
      const DrawLayout lay = draw_layout<DT>(gp);
      for (int u = u0, un = 0; u < u1; u = un) {
        un = min(u + lay.ups, u1);
        if (u != u0) mbar_wait(full + slot, phase, &s_err, p.status);
        cdf_consume_stage<DT>(cq, g, gp, rt, rd, u, un, ring + slot * kStageBytes, lay, warp);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
        if (++slot == kStagesA) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // hand the chunk to its epilogue warp
      if (lane == 0 && piece >= kPieceSlots)
        mbar_wait(pempty + ps, ((piece / kPieceSlots) - 1) & 1, &s_err, p.status);
      __syncwarp();
      if (warp == 0 && lane == 0) slots[ps].chunk = chunk;
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull + ps);
      continue;
    }
    const int64_t row = d.row, pu0 = d.pu0, pu1 = d.pu1;
    const int kch = d.kch;
    const int jr = d.jr;
    const bool is_t = jr < p.nt;
    (void)is_t;  // read by the bounds-checked build only
    const float c = d.c;
    const int need = d.need;
    const bool top = TOPK > 0 && need > 0;
    a.reset();
    wl.reset(top ? need : 1);
    // pruning bound for this row's top list: what earlier chunks of the row
    // established, then the CTA's warps' cuts
    float ccut = kNegInf;
    if (TOPK > 0 && top && kch > 0) {
      const uint32_t rc = __ldcg(p.row_cut + row);
      if (rc != 0u) ccut = unord_float(rc);
    }
    float published = kNegInf;   // this warp's last published cut
    float hpublished = kNegInf;  // and list head
    bool booted = false;         // the piece's first full stage is done
    const unsigned long long tag = (unsigned long long)(uint32_t)piece << 32;
    const int nst = (int)((pu1 - pu0 + ups - 1) / ups);  // stages of the piece
    for (int s = 0; s < nst; ++s) {
      if (s != 0) mbar_wait(full + slot, phase, &s_err, p.status);
      const int nvec = s_sd[slot].nvec;
      const int ei0 = s_sd[slot].ei0;
      const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kStageBytes);
      constexpr int kVecs = kStageBytes / 16;
      constexpr int kVpt = kVecs / kConsumers;
      if (nvec == kVecs) {
        // full stage: this thread's kVpt vectors, loaded first
        uint4 raw[kVpt];
#pragma unroll
        for (int k = 0; k < kVpt; ++k) raw[k] = sv[tid + k * kConsumers];
        constexpr int N = kVpt * VEC;
        float x[N];
#pragma unroll
        for (int k = 0; k < kVpt; ++k) Elem<DT>::unpack(raw[k], x + k * VEC);
        float vq[kVpt];
#pragma unroll
        for (int q = 0; q < kVpt; ++q) {
          float t = fmaxf(x[q * VEC], x[q * VEC + 1]);
#pragma unroll
          for (int k = 2; k < VEC; k += 2) t = fmax3(t, x[q * VEC + k], x[q * VEC + k + 1]);
          vq[q] = t;
        }
        float vm = vq[0];
#pragma unroll
        for (int q = 1; q < kVpt; ++q) vm = fmaxf(vm, vq[q]);
        if (p.usum != nullptr) {
          // the sums of the warp's four 32-vector runs, for the row's draw
          float vs[kVpt];
          a.take_split<N, kVpt>(x, vm, c, vs);
          store_subunits<kVpt>(p, row, ei0 / (32 * VEC) + warp, kConsumerWarps, vs, a.mc);
        } else {
          a.take<N>(x, vm, c);
        }
        if (TOPK > 0 && top) {
          if (!booted) {
            // First full stage of the piece: bound the row's R-th best by the
            // R-th largest lane maximum, and publish the warp's maximum as
            // its head at once, so that warps that reach this stage later
            // start from the R-th largest head already published.
            booted = true;
            const float bm = unord_float(__reduce_max_sync(0xffffffffu, ord_float(vm)));
            if (lane == 0)
              *reinterpret_cast<volatile unsigned long long*>(&s_head[warp]) = tag | ord_float(bm);
            hpublished = bm;
            __syncwarp();
            ccut = fmaxf(ccut, fmaxf(wl.boot_bound(vm), heads_cut(s_head, (uint32_t)piece, wl.R)));
          }
          wl.template offer<DT, kVpt>(raw, vq, vm, ei0 + tid * VEC, kConsumers * VEC, ccut);
        }
      } else {
        // partial stage: warp-strided vectors so that every lane takes part
        for (int v0 = warp * 32; v0 < nvec; v0 += kConsumers) {
          const int v = v0 + lane;
          float x[VEC];
          float vm = kNegInf;
          uint4 rv = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
          if (DT == 1) rv = make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
          float vs1 = 0.f;
          if (v < nvec && SSD_CHK(v < kVecs, p.dbg, 10, v, nvec)) {
            rv = sv[v];
            Elem<DT>::unpack(rv, x);
            vm = x[0];
#pragma unroll
            for (int k = 1; k < VEC; ++k) vm = fmaxf(vm, x[k]);
            if (p.usum != nullptr)
              a.take_split<VEC, 1>(x, vm, c, &vs1);
            else
              a.take<VEC>(x, vm, c);
          }
          if (p.usum != nullptr) store_subunits<1>(p, row, (ei0 + v0 * VEC) / (32 * VEC), 0, &vs1, a.mc);
          if (TOPK > 0 && top) wl.template offer<DT, 1>(&rv, &vm, vm, ei0 + v * VEC, 0, ccut);
        }
      }
      // unaligned head / tail elements (fewer than 32) by warp 0, from global memory
      if (warp == 0) {
        const StageDesc st = s_sd[slot];
        const int hc = nvec > 0 ? ei0 - st.e0 : st.e1 - st.e0;
        const int ei1 = ei0 + nvec * VEC;
        const int tc = nvec > 0 ? st.e1 - ei1 : 0;
        for (int f0 = 0; f0 < hc + tc; f0 += 32) {
          const int f = f0 + lane;
          float x = kNegInf;
          int idx = 0;
          if (f < hc + tc) {
            idx = f < hc ? st.e0 + f : ei1 + (f - hc);
            const uintptr_t fa = st.b0 + (uintptr_t)(idx - st.e0) * Elem<DT>::kSize;
            if (SSD_CHK(in_range(fa, fa + Elem<DT>::kSize, is_t ? p.t_lo : p.d_lo,
                                 is_t ? p.t_hi : p.d_hi), p.dbg, 2, idx, st.e0)) {
              x = Elem<DT>::load(reinterpret_cast<const void*>(st.b0), (int64_t)(idx - st.e0));
              a.take<1>(&x, x, c);
            }
          }
          if (TOPK > 0 && top) wl.offer1(x, idx, ccut);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + slot);
      if (++slot == kStagesA) {
        slot = 0;
        phase ^= 1u;
      }
      if (TOPK > 0 && top) {
        // The warp holds R candidates >= its cut cv, so no logit strictly
        // below the largest cut of the CTA's warps (for this row) can enter
        // the row's top list.  A warp publishes its cut only when it rose
        // (cv is warp-uniform); every lane then reads the CTA-wide value.
        if (wl.cv != kNegInf && wl.cv > published) {
          if (lane == 0) atomicMax(&s_cut, tag | ord_float(wl.cv));
          published = wl.cv;
        }
        if (wl.hv > hpublished) {
          // A new head: publish it, then raise the cut to the R-th largest
          // of this piece's heads (R distinct logits of the row reach it).
          hpublished = wl.hv;
          if (lane == 0) *reinterpret_cast<volatile unsigned long long*>(&s_head[warp]) =
              tag | ord_float(wl.hv);
          __syncwarp();
          const float hr = heads_cut(s_head, (uint32_t)piece, wl.R);
          if (lane == 0 && hr != kNegInf) atomicMax(&s_cut, tag | ord_float(hr));
        }
        __syncwarp();
        const unsigned long long w = *reinterpret_cast<volatile unsigned long long*>(&s_cut);
        if ((w >> 32) == (uint32_t)piece) ccut = fmaxf(ccut, unord_float((uint32_t)w));
      }
    }

    // ---- hand the piece's per-warp results to the epilogue warp ----
    float M, MC, Shi, Slo;
    warp_softmax_merge(a.m, a.mc, a.hi, a.lo, c, M, MC, Shi, Slo);
    if (lane == 0 && piece >= kPieceSlots)
      mbar_wait(pempty + ps, ((piece / kPieceSlots) - 1) & 1, &s_err, p.status);
    __syncwarp();
    PieceRed<TOPK>& R = slots[ps];
    if (lane == 0) {
      R.m[warp] = M;
      R.hi[warp] = Shi;
      R.lo[warp] = Slo;
      if (warp == 0) {
        R.chunk = chunk;
        R.c = c;
      }
    }
    if (lane < (TOPK > 0 ? TOPK : 1)) {
      R.tv[warp][lane] = (TOPK > 0 && top) ? wl.lv : kNegInf;
      R.ti[warp][lane] = (TOPK > 0 && top) ? wl.li : 0x7fffffff;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(pfull + ps);
  }
}

template <int DT, int TOPK>
cudaError_t launch_t(const VerifyParams& p, int grid, cudaStream_t s) {
  const int smem = stream_smem_bytes();
  auto kern = stream_kernel<DT, TOPK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // CTAs wait for groups that other CTAs complete: all of them must be
  // resident at once, which a cooperative launch guarantees
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = p.q.nchunks > 0 ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int DT>
cudaError_t launch_dt(const VerifyParams& p, int topk, int grid, cudaStream_t s) {
  switch (topk) {
    case 0: return launch_t<DT, 0>(p, grid, s);
    case 2: return launch_t<DT, 2>(p, grid, s);
    case 4: return launch_t<DT, 4>(p, grid, s);
    case 8: return launch_t<DT, 8>(p, grid, s);
    case 16: return launch_t<DT, 16>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int stream_smem_bytes() {
  return kStagesA * kStageBytes + 2 * (kStagesA + kPieceSlots) * (int)sizeof(uint64_t) +
         kPieceSlots * (int)sizeof(PieceRed<kMaxTopK>);
}

cudaError_t launch_stream(const VerifyParams& p, int dtype, int topk, int grid, cudaStream_t s) {
  return dtype == SSD_BF16 ? launch_dt<0>(p, topk, grid, s) : launch_dt<1>(p, topk, grid, s);
}

}  // namespace ssd
