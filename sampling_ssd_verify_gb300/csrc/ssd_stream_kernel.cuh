// ssd_stream_kernel.cuh -- the streaming pass over full-vocabulary logit
// rows and the draws that follow it, in one persistent launch (instantiated
// per element type by ssd_stream_bf16.cu and ssd_stream_f32.cu).
//
// Work: one persistent CTA per SM (a cooperative launch: CTAs wait on work
// other CTAs do).  Its producer warp takes row chunks from a global counter
// (the first round static: chunk = CTA) and draw chunks from a ticket queue,
// and streams them through a ring of kStagesA 32 KB shared-memory stages with
// 1-D bulk copies (cp.async.bulk, mbarrier transaction counts, L2
// evict-first).  Sixteen consumer warps reduce each stage; each owns one
// block of 128 consecutive 16-byte vectors of the stage.  Three epilogue
// warps take pieces in turn (piece p to warp p mod 3) and do every
// global-memory epilogue step, so the consumers never wait for one.
//
// A row chunk gives, per row ([SD-7.3] §7.3.2: the target and draft
// distributions of every position):
//   * the online-softmax normaliser: max raw logit m and
//     s = sum_y 2^(z_y * c - fl(m*c)), c = log2(e)/T, compensated fp32 sums
//     per thread, merged per warp and per row;
//   * the logit of the row's draft token, picked out of the staged data;
//   * the top-(F_j+1) raw logits (ties to the lower index) of the draft rows
//     ([SSD-note] §"怎么猜奖励 token", §"Saguaro 优化二：Saguaro 采样"): the
//     consumers record each block's and each warp's maximum; at the end of
//     the piece theta = the R-th largest warp maximum (R warps hold a logit
//     >= theta, so no logit below it is in the top R), each warp reads its
//     blocks whose maximum reaches theta again and lists their logits
//     >= theta; the epilogue keeps the best R in a warp-wide sorted list;
//   * for rows whose draw weight has one term (Saguaro rows, target row K),
//     each block's sum, so that the draw needs no second pass.
//
// Sequences are verified as their positions complete: row chunks are handed
// out position by position, and when the target and draft rows of position
// i are both final the accept test u_i < p_i(x_i)/q'_i(x_i) runs at once
// ([SD-7.3] §7.3.3; [SD-blog] §"三、接受概率为什么是对的").  A sequence is
// decided when its first rejection k has every earlier position accepted (or
// all K are accepted and target row K is done).  The all-accepted bonus is
// drawn at once from target row K's block sums; a residual (p - q')^+ draw
// is cut into chunks pushed to a ticket queue, which producers serve before
// their next row chunk, while later positions are still streaming.
//
// Sources: [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈";
// [SD-7.3] "7.3 Speculative Decoding：投机采样加速";
// [SD-blog] "推测解码：用一个“小模型”骗出 3 倍推理速度".
#pragma once

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

// Warp roles: warps 0..kConsumerWarps-1 reduce staged data, warp
// kConsumerWarps takes chunks and issues their bulk copies, and
// kEpilogueWarps epilogue warps (piece p to warp p mod kEpilogueWarps) merge
// each piece's per-warp results and do all global-memory epilogue work.
// Piece results pass through a queue of kPieceSlots shared-memory slots
// guarded by mbarriers; the consumers take a piece's slot when the piece
// starts (the block maxima are written into it stage by stage).
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarp = kConsumerWarps + 1;  // the first epilogue warp
constexpr int kEpilogueWarps = 3;
constexpr int kStreamThreads = (kConsumerWarps + 1 + kEpilogueWarps) * 32;
constexpr int kPieceSlots = 3;
static_assert(kPieceSlots % kEpilogueWarps == 0, "a slot belongs to one epilogue warp");
// The producer runs at most kStagesA + 1 pieces ahead of the consumer
// warps, so a descriptor queue this long is never overwritten early.
constexpr int kPieceQueue = 16;
constexpr int kMaxCand = 64;  // top-list candidates a piece hands to its epilogue
static_assert(kPieceQueue > kStagesA + 1, "piece queue shorter than the pipeline");

struct alignas(16) PieceRed {
  long long chunk;  // the piece (row chunk, or nchunks + draw chunk), -1: no more pieces
  float c;          // log2(e) / T of the piece's sequence
  int nst;          // stages of the piece
  float zx;         // logit of the row's draft token, when the piece holds it
  float m[kConsumerWarps];
  float hi[kConsumerWarps];
  float lo[kConsumerWarps];
  float wmax[kConsumerWarps];  // each consumer warp's largest logit of the piece
  float bmax[kMaxBlocks];  // block maxima, (stage of the piece) * kConsumerWarps + warp
  // The piece's top-list candidates: every logit >= theta of the blocks
  // whose maximum reaches theta, found by the consumer warps at the end of
  // the piece (ncand > kMaxCand: too many, the epilogue reads the blocks).
  int ncand;
  float cand_v[kMaxCand];
  int cand_i[kMaxCand];
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

template <int DT>
__device__ __forceinline__ const char* row_address(const StreamParams& p, int64_t row, bool& is_t) {
  int64_t trow;
  const void* base = tensor_of<DT>(p, row, trow, is_t);
  return row_ptr(base, trow, is_t ? p.t_stride : p.d_stride, Elem<DT>::kSize);
}

// Stage s of a row at rp: element range and aligned interior.
template <int DT>
__device__ __forceinline__ Stage stage_of(const char* rp, int V, int s) {
  constexpr int E = units_per_stage(Elem<DT>::kSize) * kUnitA;  // elements per stage
  Stage st;
  st.e0 = s * E;
  st.e1 = min(V, st.e0 + E);
  st.b0 = (uintptr_t)(rp + (int64_t)st.e0 * Elem<DT>::kSize);
  const uintptr_t b1 = (uintptr_t)(rp + (int64_t)st.e1 * Elem<DT>::kSize);
  st.a0 = (st.b0 + 15) & ~(uintptr_t)15;
  st.a1 = b1 & ~(uintptr_t)15;
  if (st.a1 <= st.a0) st.a0 = st.a1 = st.b0;  // no aligned interior: all scalar
  return st;
}

// Named barrier 2: the consumer warps wait (bar.sync) until the epilogue
// warps have loaded the draft tokens into shared memory (bar.arrive).
constexpr int kTokBarThreads = kConsumers + kEpilogueWarps * 32;
__device__ __forceinline__ void tok_bar_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(kTokBarThreads) : "memory");
}
__device__ __forceinline__ void tok_bar_arrive() {
  asm volatile("bar.arrive 2, %0;" ::"n"(kTokBarThreads) : "memory");
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
  // n logits (finite, or -inf padding) whose maximum vm is finite.  For n a
  // multiple of 4 the exponent arguments and the pairwise tree sum use the
  // packed f32x2 FMA / add (the same roundings, in the same order).  Returns
  // the sum added (relative to the offset mc after the call).
  template <int N>
  __device__ __forceinline__ float take(const float* x, float vm, float c) {
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
    return e[0];
  }
};

// One warp-wide top list: lane l < R holds the l-th best candidate by
// (logit desc, index asc); (cv, ci) is entry R - 1, known to all lanes.
// Candidates are offered by ballot and inserted cooperatively.
struct WarpList {
  float lv, cv;
  int li, ci;
  int R;  // entries kept (<= 32)
  __device__ __forceinline__ void reset(int need) {
    lv = cv = kNegInf;
    li = ci = 0x7fffffff;
    R = need;
  }
  __device__ __forceinline__ bool qualifies(float x, int i) const {
    return x != kNegInf && cand_before(x, i, cv, ci);
  }
  __device__ __forceinline__ void insert(float v, int i) {
    const int lane = threadIdx.x & 31;
    const bool before = lane < R && cand_before(lv, li, v, i);
    const int pos = __popc(__ballot_sync(0xffffffffu, before));
    if (pos >= R) return;  // warp-uniform
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
  // Offer one logit per lane (-inf: nothing); all 32 lanes call.
  __device__ __forceinline__ void offer(float x, int idx, bool valid) {
    unsigned m = __ballot_sync(0xffffffffu, valid && qualifies(x, idx));
    while (m) {
      const int L = __ffs(m) - 1;
      insert(__shfl_sync(0xffffffffu, x, L), __shfl_sync(0xffffffffu, idx, L));
      m &= m - 1;
    }
  }
};

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

// Fan-out of Saguaro row r (per-row array clamped to [0, Fmax], a bad value
// reported), or F_j of draft position j.
__device__ __forceinline__ int saguaro_F(const StreamParams& p, int64_t r) {
  if (p.F_rows == nullptr) return p.F[0];
  const int f = __ldg(p.F_rows + r);
  return min(max(f, 0), p.Fmax);
}

// Top-list entries row `row` (row jr of group g) needs: F_j + 1 on a draft
// row that feeds guesses or a Saguaro set, 1 (its argmax) on a target row of
// a greedy sequence, otherwise none.
__device__ __forceinline__ int row_need(const StreamParams& p, int64_t g, int jr) {
  if (jr < p.nt) return p.mode == kModeVerify && seq_greedy(p, g) ? 1 : 0;
  const int F = p.mode == kModeSaguaro ? saguaro_F(p, g) : p.F[jr - p.nt];
  return (p.need_top && F > 0) ? F + 1 : 0;
}

// Row chunk c: its row, chunk of the row and units [pu0, pu1).  Order 0:
// (chunk of row, row).  Order 1 (verify, position-major): for position
// i < K, chunk-of-row major, then sequence, then (target i, draft i); for
// position K, the draft rows K first, then the target rows K.
__device__ __forceinline__ void chunk_geom(const StreamParams& p, long long c, int64_t& row,
                                           int& kch, int64_t& pu0, int64_t& pu1) {
  if (p.order == 0) {
    kch = (int)(c / p.NR);
    row = c - (int64_t)kch * p.NR;
  } else {
    const long long B = p.B;
    const long long per = 2 * B * p.nch;  // chunks of one position i < K
    const long long lo = (long long)p.K * per;
    int i, mem;  // mem 0: target row, 1: draft row
    long long g;
    if (c < lo) {
      i = (int)(c / per);
      const long long o = c - i * per;
      kch = (int)(o / (2 * B));
      const long long r = o - (long long)kch * 2 * B;
      g = r >> 1;
      mem = (int)(r & 1);
    } else {
      i = p.K;
      const long long mK = p.Kq > p.K ? 2 : 1;
      const long long o = c - lo;
      kch = (int)(o / (mK * B));
      const long long r = o - (long long)kch * mK * B;
      mem = (mK == 2 && r < B) ? 1 : 0;
      g = (mK == 2 && r >= B) ? r - B : r;
    }
    row = g * p.rpg + (mem == 0 ? i : p.nt + i);
  }
  pu0 = row * p.upr + (int64_t)kch * p.clen;
  pu1 = min(pu0 + p.clen, (row + 1) * p.upr);
}

// A piece as the producer hands it to the consumer warps (chunk -1: the end).
struct PieceDesc {
  long long chunk;
  // a chunk of rows
  int64_t row, pu0, pu1;
  const char* rp;  // element 0 of the row
  int jr;          // row within its group
  int s0;          // stage of the row the piece starts at
  float c;         // log2(e) / T of the row's sequence
  int need;        // top-list entries the row needs
  int wsum;        // the row's block sums are stored (one-term draw)
  // the row's group; for a chunk of the draws also its units [u0, u1) and
  // the group's parameters
  int64_t g;
  int u0, u1;
  GroupParams gp;
};

// ---- the top list of a row chunk (epilogue warp) ------------------------------------------
// Block b of a row chunk is consumer warp b % W's share of stage s0 + b / W
// (W = kConsumerWarps): vectors [kVecsPerWarp w, kVecsPerWarp (w + 1)) of
// the stage's aligned interior, plus the
// unaligned head and tail of the stage for w = 0.  The consumers record each
// block's maximum and each warp's maximum over the chunk.
//
// theta = the R-th largest of the W warp maxima: R different warps hold a
// logit >= theta, so no logit below it is in the top R.  Every block whose
// maximum reaches theta is read again (from L2: the chunk was just
// streamed) and its logits >= theta are offered to the warp list.

// Offer the logits >= th of 16-byte vector r (element e has index
// idx0 + e), one vector per lane: each lane marks its qualifying elements,
// then the warp inserts them one by one (usually one or none per block).
template <int DT>
__device__ __forceinline__ void offer_vector(WarpList& wl, uint4 r, bool valid, int idx0,
                                             float th) {
  constexpr int VEC = Elem<DT>::kVec;
  float x[VEC];
  Elem<DT>::unpack(r, x);
  unsigned bits = 0;
#pragma unroll
  for (int e = 0; e < VEC; ++e)
    bits |= (valid && x[e] >= th && wl.qualifies(x[e], idx0 + e)) ? (1u << e) : 0u;
  unsigned lanes = __ballot_sync(0xffffffffu, bits != 0);
  while (lanes) {
    const int L = __ffs(lanes) - 1;
    const unsigned bL = __shfl_sync(0xffffffffu, bits, L);
    const int e = __ffs(bL) - 1;
    const float v = __shfl_sync(0xffffffffu, vec_elem<DT>(r, e), L);
    const int i = __shfl_sync(0xffffffffu, idx0 + e, L);
    wl.insert(v, i);
    if ((threadIdx.x & 31) == L) bits &= bits - 1;
    lanes = __ballot_sync(0xffffffffu, bits != 0);
  }
}

// Read block b of the chunk again and offer its logits >= th.
template <int DT>
__device__ __forceinline__ void reread_block(const StreamParams& p, const char* rp, int s0, int b,
                                             const char* lo, const char* hi, int64_t row,
                                             float th, WarpList& wl) {
  constexpr int VEC = Elem<DT>::kVec;
  const int lane = threadIdx.x & 31;
  const int wb = b % kConsumerWarps;
  const Stage st = stage_of<DT>(rp, p.V, s0 + b / kConsumerWarps);
  const int nvec = (int)((st.a1 - st.a0) >> 4);
  const int ei0 = st.e0 + (int)((st.a0 - st.b0) / Elem<DT>::kSize);
  uint4 raw[kVpt];
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int vi = wb * kVecsPerWarp + lane + 32 * k;
    const uintptr_t a = st.a0 + (uintptr_t)vi * 16;
    raw[k] = make_uint4(0, 0, 0, 0);
    if (vi < nvec && SSD_CHK(in_range(a, a + 16, lo, hi), p.dbg, 30, row, vi))
      raw[k] = __ldg(reinterpret_cast<const uint4*>(a));
  }
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int vi = wb * kVecsPerWarp + lane + 32 * k;
    offer_vector<DT>(wl, raw[k], vi < nvec, ei0 + vi * VEC, th);
  }
  if (wb == 0) {
    // the stage's unaligned head and tail
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
        if (SSD_CHK(in_range(fa, fa + Elem<DT>::kSize, lo, hi), p.dbg, 31, row, idx))
          x = Elem<DT>::load_cg(reinterpret_cast<const void*>(st.b0), (int64_t)(idx - st.e0));
      }
      wl.offer(x, idx, x >= th);
    }
  }
}

// Consumer warp wb lists the logits >= th of its block of stage s (read
// again from global memory) in the piece's candidate list.
template <int DT>
__device__ __forceinline__ void list_block(const StreamParams& p, const char* rp, bool is_t, int s,
                                           int wb, float th, int64_t row, PieceRed& R) {
  constexpr int VEC = Elem<DT>::kVec;
  const int lane = threadIdx.x & 31;
  const char* lo = is_t ? p.t_lo : p.d_lo;
  const char* hi = is_t ? p.t_hi : p.d_hi;
  (void)lo;
  (void)hi;  // read by the bounds-checked build only
  const Stage st = stage_of<DT>(rp, p.V, s);
  const int nvec = (int)((st.a1 - st.a0) >> 4);
  const int ei0 = st.e0 + (int)((st.a0 - st.b0) / Elem<DT>::kSize);
  uint4 raw[kVpt];
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int vi = wb * kVecsPerWarp + lane + 32 * k;
    const uintptr_t a = st.a0 + (uintptr_t)vi * 16;
    raw[k] = make_uint4(0, 0, 0, 0);
    if (vi < nvec && SSD_CHK(in_range(a, a + 16, lo, hi), p.dbg, 32, row, vi))
      raw[k] = __ldg(reinterpret_cast<const uint4*>(a));
  }
  auto put = [&](float x, int idx, bool ok) {
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (!m) return;
    int base = 0;
    if (lane == 0) base = atomicAdd(&R.ncand, __popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int pos = base + __popc(m & ((1u << lane) - 1u));
    if (ok && pos < kMaxCand) {
      R.cand_v[pos] = x;
      R.cand_i[pos] = idx;
    }
  };
#pragma unroll
  for (int k = 0; k < kVpt; ++k) {
    const int vi = wb * kVecsPerWarp + lane + 32 * k;
    float x[VEC];
    Elem<DT>::unpack(raw[k], x);
    float vm = x[0];
#pragma unroll
    for (int e = 1; e < VEC; ++e) vm = fmaxf(vm, x[e]);
    if (!__any_sync(0xffffffffu, vi < nvec && vm >= th)) continue;
#pragma unroll
    for (int e = 0; e < VEC; ++e) put(x[e], ei0 + vi * VEC + e, vi < nvec && x[e] >= th);
  }
  if (wb == 0) {
    // the stage's unaligned head and tail
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
        if (SSD_CHK(in_range(fa, fa + Elem<DT>::kSize, lo, hi), p.dbg, 33, row, idx))
          x = Elem<DT>::load(reinterpret_cast<const void*>(st.b0), (int64_t)(idx - st.e0));
      }
      put(x, idx, x != kNegInf && x >= th);
    }
  }
}

// The chunk's top list: wm = lane w's warp maximum (lanes >= W: -inf),
// v[j] = the maximum of block lane + 32 j.
template <int DT>
__device__ __noinline__ void chunk_top(const StreamParams& p, int64_t row, int s0, float wm,
                          const float (&v)[kBlkPerLane], WarpList& wl) {
  const int lane = threadIdx.x & 31;
  // theta: the R-th largest warp maximum (-inf when fewer than R warps saw data)
  float th = kNegInf;
  float m = wm;
  for (int r = 0; r < wl.R; ++r) {
    const float mx = warp_max_f32(m);
    if (mx == kNegInf) {
      th = kNegInf;
      break;
    }
    th = mx;
    const unsigned who = __ballot_sync(0xffffffffu, m == mx);
    if (lane == __ffs(who) - 1) m = kNegInf;
  }
  bool is_t;
  const char* rp = row_address<DT>(p, row, is_t);
  const char* lo = is_t ? p.t_lo : p.d_lo;
  const char* hi = is_t ? p.t_hi : p.d_hi;
  (void)lo;
  (void)hi;  // read by the bounds-checked build only
  // the candidate blocks, lane by lane in order
  unsigned cmask = 0;
#pragma unroll
  for (int j = 0; j < kBlkPerLane; ++j) cmask |= (v[j] != kNegInf && v[j] >= th) ? (1u << j) : 0u;
  unsigned lanes = __ballot_sync(0xffffffffu, cmask != 0);
  while (lanes) {
    const int L = __ffs(lanes) - 1;
    const unsigned mL = __shfl_sync(0xffffffffu, cmask, L);
    const int j = __ffs(mL) - 1;
    if (lane == L) cmask &= cmask - 1;
    reread_block<DT>(p, rp, s0, L + 32 * j, lo, hi, row, th, wl);
    lanes = __ballot_sync(0xffffffffu, cmask != 0);
  }
}

// Fold a stored chunk partial into a lane's softmax accumulator (row
// merges); the partial's list entries go to the warp list.
__device__ __forceinline__ void fold_partial(SAcc& a, const RowPartial* pp, float c) {
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
}

// ---- target rows past a rejection ---------------------------------------------------------
// No output depends on target row j of a sequence once one of its positions
// before j is rejected: the first rejection, which decides the sequence, is
// then before j, and the accept tests stop there ([SD-7.3] §7.3.3).  Draft
// rows always stream (their top lists give the guesses of every position).
// The producer reads the sequence's state word when it fetches a chunk id
// and drops the chunk when it is such a row; a state read too early only
// streams a row that is not needed.

// The state word of row chunk c's sequence when c is a target row past
// position 0 of a verify launch (loaded now, used at the next claim), else 0.
__device__ __forceinline__ unsigned long long chunk_state(const StreamParams& p, long long c,
                                                          long long nS) {
  if (p.mode != kModeVerify || c >= nS) return 0ull;
  int64_t row, pu0, pu1;
  int kch;
  chunk_geom(p, c, row, kch, pu0, pu1);
  const int64_t g = row / p.rpg;
  const int jr = (int)(row - g * p.rpg);
  if (jr == 0 || jr >= p.nt) return 0ull;
  return ld_relaxed_u64(p.seq_state + g);
}

// Whether row chunk c is a target row past a rejection recorded in st; if
// so its bytes are added to the launch's count of bytes not streamed.
template <int DT>
__device__ __forceinline__ bool chunk_past_rejection(const StreamParams& p, long long c,
                                                     unsigned long long st) {
  if (st >> 32 == 0ull) return false;
  int64_t row, pu0, pu1;
  int kch;
  chunk_geom(p, c, row, kch, pu0, pu1);
  const int64_t g = row / p.rpg;
  const int jr = (int)(row - g * p.rpg);
  if (jr == 0 || jr >= p.nt) return false;
  const unsigned below = jr >= 32 ? 0xffffffffu : ((1u << jr) - 1u);
  if (((unsigned)(st >> 32) & below) == 0u) return false;
  const int64_t e0 = (pu0 - row * p.upr) * kUnitA;
  const int64_t e1 = min((pu1 - row * p.upr) * kUnitA, (int64_t)p.V);
  atomicAdd(p.skipped, (unsigned long long)((e1 - e0) * Elem<DT>::kSize));
  return true;
}

// ---- the sequence outcome (verify) ------------------------------------------------------
// State word of a sequence: bit i = position i accepted, bit 32 + i =
// rejected (i < K <= 32).
__device__ __forceinline__ unsigned maskK(int K) { return K >= 32 ? 0xffffffffu : ((1u << K) - 1u); }
// Decided by a rejection: the first rejected position k with every earlier
// position accepted; returns k or -1.
__device__ __forceinline__ int rejected_at(unsigned long long s, int K) {
  const unsigned R = (unsigned)(s >> 32) & maskK(K);
  if (R == 0) return -1;
  const int k = __ffs(R) - 1;
  const unsigned low = k >= 32 ? 0xffffffffu : ((1u << k) - 1u);
  return ((unsigned)s & low) == low ? k : -1;
}
__device__ __forceinline__ bool all_accepted(unsigned long long s, int K) {
  return ((unsigned)s & maskK(K)) == maskK(K);
}

// The accept test of position i of sequence g (one lane): u_i < p_i(x_i) /
// q'_i(x_i) with q' the Saguaro-biased draft distribution, or, greedy, x_i
// is the argmax of target row i.  The ratio is first formed in fp32 (error
// a few 1e-6 relative); only when u lies within 1e-4 of it is the decision
// taken from the fp64 ratio, so the result is that of the fp64 test.
__device__ bool accept_test(const StreamParams& p, int64_t g, int i, float cf) {
  const RowResult* rt = p.rowres + g * p.rpg + i;
  const RowResult* rd = p.rowres + g * p.rpg + p.nt + i;
  const int x = __ldcg(&rt->x);
  if (seq_greedy(p, g)) return x == __ldcg(&rt->ti[0]);
  const float zt = __ldcg(&rt->zx), mct = __ldcg(&rt->mc);
  const double st = __ldcg(&rt->s);
  const float zd = __ldcg(&rd->zx), mcd = __ldcg(&rd->mc);
  const double sq = __ldcg(&rd->s);
  const double u = uniform24(p.seeds[g], (uint32_t)g, (uint32_t)i, 0u, p.round);
  const int F = p.F[i];
  const float Cl = p.C[i];
  const bool sag = Cl < 1.f && F > 0;
  float QS32 = 0.f;
  bool inS = false;
  if (sag) {
    for (int f = 0; f < F; ++f) {
      QS32 += ex2(fmaf(__ldcg(&rd->tv[f]), cf, -mcd));
      inS |= __ldcg(&rd->ti[f]) == x;
    }
  }
  const float pt32 = ex2(fmaf(zt, cf, -mct)) / (float)st;
  float qp32 = ex2(fmaf(zd, cf, -mcd)) / (float)sq;
  if (sag) qp32 = qp32 * (inS ? Cl : 1.f) / (1.f - (1.f - Cl) * (QS32 / (float)sq));
  const float r32 = pt32 / qp32;
  const float uf = (float)u;  // exact: 24-bit uniform
  if (fabsf(uf - r32) > 1e-4f * fmaxf(1.f, r32)) return uf < r32;
  const double c = (double)cf;
  const double pt = exp2((double)zt * c - (double)mct) / st;
  double qp = exp2((double)zd * c - (double)mcd) / sq;
  if (sag) {
    double QS = 0.0;
    for (int f = 0; f < F; ++f) QS += (double)exp2f(fmaf(__ldcg(&rd->tv[f]), cf, -mcd));
    QS /= sq;
    qp = qp * (inS ? (double)Cl : 1.0) / (1.0 - (1.0 - (double)Cl) * QS);
  }
  return u < pt / qp;
}

// Queue the draw chunks of group g (one lane): one fence orders the group's
// parameters before everything that follows, the tickets are reserved, and
// the entries are written with plain (relaxed) stores, back to back; a
// producer that reads an entry fences before it reads the parameters.
__device__ __forceinline__ void push_draw(const StreamParams& p, const CdfParams& cq, int64_t g) {
  __threadfence();
  const unsigned base = atomicAdd(p.dq_tail, (unsigned)cq.cpg);
  for (int c = 0; c < cq.cpg; ++c) {
    const int64_t e = (int64_t)base + c;
    if (SSD_CHK(e < (int64_t)cq.groups * cq.cpg, p.dbg, 40, e, g))
      st_relaxed_s32(p.dq_entry + e, (int)(g * cq.cpg + c) + 1);
  }
}

// The group counts as decided once its draw is queued or done (one lane).
__device__ __forceinline__ void mark_decided(const StreamParams& p) {
  __threadfence();
  atomicAdd(p.decided, 1);
}

// The bonus draw's parameters for sequence g decided with accept length k:
// the residual (p_k - q'_k)^+ (q' biased by the Saguaro set of draft row k),
// or p_K when every draft was accepted.  Every lane of a warp computes the
// same value from the same loads.
__device__ __forceinline__ GroupParams draw_params(const StreamParams& p, int64_t g, int k,
                                                   float cf) {
  const int K = p.K;
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
      float tvs[kMaxTopK];  // the set's logits, loaded together
#pragma unroll
      for (int f = 0; f < kMaxTopK; ++f) tvs[f] = f < F ? __ldcg(&rd->tv[f]) : 0.f;
      double QS = 0.0;
#pragma unroll
      for (int f = 0; f < kMaxTopK; ++f)
        if (f < F) QS += (double)exp2f(fmaf(tvs[f], cf, -gp.mc_d));
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
  return gp;
}

// The outputs of greedy sequence g with accept length k (one lane): the
// bonus is target row k's argmax; no draw (its parameters say so).
__device__ __forceinline__ void greedy_outcome(const StreamParams& p, int64_t g, int k) {
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
  gp.theta = kPosInf;
  gp.itheta = -1;
  p.gparams[g] = gp;
}

// Sequence g is decided with accept length k (warp of the deciding CTA):
// write k, then either the greedy outputs, a direct draw of p_K from the
// streaming pass's block sums, or the draw's chunks to the ticket queue.
template <int DT>
__device__ __noinline__ void decide(const StreamParams& p, const CdfParams& cq, int64_t g, int k,
                                   float cf) {
  const int lane = threadIdx.x & 31;
  const int K = p.K;
  if (!SSD_CHK(g < p.B && k >= 0 && k <= K, p.dbg, 8, g, k)) return;
  if (seq_greedy(p, g)) {
    if (lane == 0) {
      greedy_outcome(p, g, k);
      mark_decided(p);
    }
    return;
  }
  // the draw's parameters, computed by every lane (the same loads, the same
  // arithmetic); lane 0 stores them
  const GroupParams gp = draw_params(p, g, k, cf);
  if (lane == 0) {
    p.accept_len[g] = k;
    p.gparams[g] = gp;
  }
  if (k == K && p.bsum != nullptr) {
    // all accepted: the bonus is drawn from p_K with the block sums that the
    // streaming pass stored for target row K (no ticket: count it as decided
    // first, so that idle producers need not wait for the draw)
    if (lane == 0) mark_decided(p);
    direct_draw<DT>(cq, p.bsum + g * p.nblk, p.nblk, gp, g, nullptr, 0);
    return;
  }
  if (lane == 0) {
    push_draw(p, cq, g);
    mark_decided(p);
  }
}

// Saguaro continuation draw of branch row g: the parameters of q', then the
// draw from the block sums (aligned rows) or the draw's chunks queued.
template <int DT>
__device__ __noinline__ void saguaro_finish(const StreamParams& p, const CdfParams& cq, int64_t g,
                               const RowResult& rr, float cf) {
  const int lane = threadIdx.x & 31;
  const int F = saguaro_F(p, g);
  if (lane == 0 && p.F_rows != nullptr && p.status) {
    const int f = __ldg(p.F_rows + g);
    if (f < 0 || f > p.Fmax) atomicOr(p.status, SSD_DEV_BAD_FANOUT);
  }
  // q''s parameters, computed by every lane (rr is the same in every lane);
  // lane 0 stores them
  GroupParams gp;
  {
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
  }
  if (lane == 0) p.gparams[g] = gp;
  if (p.bsum != nullptr) {
    // counted only where producers wait for queued draws
    if (lane == 0 && cq.cpg > 0) mark_decided(p);
    direct_draw<DT>(cq, p.bsum + g * p.nblk, p.nblk, gp, g, p.rowres + g, F);
    return;
  }
  if (lane == 0) {
    push_draw(p, cq, g);
    mark_decided(p);
  }
}

// The bonus guesses of draft row j of group g (one warp; lane l < R of wl
// holds list entry l): top-(F_j+1) minus the sampled token, truncated to F_j;
// lane f writes guess f (entry f of the list, or f + 1 once the drafted
// token is passed), and, with the round's cache (table_ready: cleared),
// inserts its key (sequence, position, guess) -> index in the guesses array.
__device__ __forceinline__ void row_guesses(const StreamParams& p, int64_t g, int j,
                                            const RowResult& rr, const WarpList& wl, int need,
                                            float c, float MC, bool table_ready) {
  const int lane = threadIdx.x & 31;
  if (p.guesses != nullptr) {
    const bool greedy = p.mode == kModeVerify && seq_greedy(p, g);
    const int F = p.F[j];
    const unsigned hitx =
        __ballot_sync(0xffffffffu, lane < F + 1 && lane < need && wl.li == rr.x && rr.x >= 0);
    const int sx = hitx ? __ffs(hitx) - 1 : 32;
    const int e = lane < sx ? lane : lane + 1;
    const float ev = __shfl_sync(0xffffffffu, wl.lv, e & 31);
    const int ei = __shfl_sync(0xffffffffu, wl.li, e & 31);
    const int i0 = __shfl_sync(0xffffffffu, wl.li, 0);
    const bool valid = lane < F && e < need && ev != kNegInf;
    const int64_t o = (g * p.nd + j) * (int64_t)p.Fmax;
    if (lane < p.Fmax && SSD_CHK(o + lane < (int64_t)p.B * p.nd * p.Fmax, p.dbg, 7, o + lane, lane)) {
      p.guesses[o + lane] = valid ? ei : -1;
      if (p.guess_q)
        p.guess_q[o + lane] = !valid ? 0.f
                              : greedy ? (ei == i0 ? 1.f : 0.f)
                                       : ex2(fmaf(ev, c, -MC)) / (float)rr.s;
    }
  }
  if (p.rc.table != nullptr && p.guesses != nullptr && p.F[j] > 0 && table_ready) {
    const int F = p.F[j];
    int sx = kMaxTopK;
    for (int k = F; k >= 0; --k)
      if (rr.ti[k] == rr.x) sx = k;
    if (lane < F) {
      const int e = lane < sx ? lane : lane + 1;
      const int tok = e < kMaxTopK ? rr.ti[e] : -1;
      if (tok >= 0)
        cache_insert(static_cast<Slot*>(p.rc.table), p.rc.cap, pack_key((int)g, j, tok),
                     (int)((g * p.nd + j) * p.Fmax + lane), p.status);
    }
  }
}

// Finalise row `row` from the merged (M, MC, S) and top list (lane l < R
// holds entry l).  Writes the row's result, its guesses and cache keys, then
// counts the row into its position (verify) or draws (Saguaro).
// xs / zxs: the row's draft token and its logit when the streaming pass
// captured them (have_x), else they are read here.
template <int DT>
__device__ __noinline__ void finalize_row(const StreamParams& p, const CdfParams& cq, int64_t row, float c,
                             float M, float MC, float Shi, float Slo, const WarpList& wl,
                             int need, bool have_x, int xs, float zxs, bool* cleared,
                             volatile int* s_err) {
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
    const float v = __shfl_sync(0xffffffffu, wl.lv, k);
    const int i = __shfl_sync(0xffffffffu, wl.li, k);
    const bool valid = k < need && v != kNegInf;
    rr.tv[k] = valid ? v : kNegInf;
    rr.ti[k] = valid ? i : -1;
  }
  rr.x = -1;
  rr.zx = 0.f;
  if (have_x) {
    rr.x = xs;
    rr.zx = zxs;
  } else if (p.tokens != nullptr && j < p.tokK) {
    int x = SSD_CHK(g < p.B && j < p.tokK, p.dbg, 3, g, j) ? p.tokens[g * p.tokK + j] : 0;
    if (x < 0 || x >= p.V) {
      if (lane == 0 && p.status) atomicOr(p.status, SSD_DEV_BAD_TOKEN);
      x = 0;
    }
    bool it;
    const char* rp = row_address<DT>(p, row, it);
    rr.x = x;
    const uintptr_t ga = (uintptr_t)(rp + (int64_t)x * Elem<DT>::kSize);
    rr.zx = SSD_CHK(in_range(ga, ga + Elem<DT>::kSize, it ? p.t_lo : p.d_lo, it ? p.t_hi : p.d_hi),
                    p.dbg, 4, row, x) ? Elem<DT>::load_cg(rp, x) : 0.f;
  }
  if (lane == 0 && SSD_CHK(row < p.NR, p.dbg, 5, row, p.NR)) p.rowres[row] = rr;
  if (!is_t) {
    bool ready = p.rc.table == nullptr || p.guesses == nullptr || p.F[j] == 0 || *cleared;
    if (!ready) {
      // the round's cache takes keys after every CTA has cleared its slice
      int ok = 0;
      if (lane == 0)
        ok = count_wait(p.rc.cleared, (int)gridDim.x * kEpilogueWarps, s_err, p.status);
      *cleared = ready = __shfl_sync(0xffffffffu, ok, 0) != 0;
    }
    row_guesses(p, g, j, rr, wl, need, c, MC, ready);
  }
  // orders every lane's stores (results, guesses, cache keys and values)
  // before lane 0's release arrival below
  __syncwarp();
  if (p.mode == kModeTopF) return;
  if (p.mode == kModeSaguaro) {
    saguaro_finish<DT>(p, cq, g, rr, c);
    return;
  }
  // verify: count the row into its position; the position's last row runs
  // the accept test and updates the sequence's state
  const int K = p.K;
  const int size = j < K ? 2 : (p.Kq > K ? 2 : 1);
  int dk = -1;
  if (lane == 0) {
    // acquire-release arrivals: this row's results (and, through the warp
    // barrier above, the cache keys of its lanes) are published with the
    // arrival, and the position's last row sees its partner's
    const int64_t pc = g * (K + 1) + j;
    const bool last = SSD_CHK(g < p.B && j <= K, p.dbg, 9, g, j)
                          ? atom_add_acq_rel(p.pair_cnt + pc, 1) == size - 1 : false;
    if (last) {
      if (j < K) {
        const bool acc = accept_test(p, g, j, c);
        const unsigned long long bits = acc ? (1ull << j) : (1ull << (32 + j));
        const unsigned long long old = atom_or_acq_rel(p.seq_state + g, bits);
        const unsigned long long nw = old | bits;
        const int kr = rejected_at(nw, K);
        if (kr >= 0 && rejected_at(old, K) < 0) {
          dk = kr;
        } else if (all_accepted(nw, K) && !all_accepted(old, K)) {
          if (atom_add_acq_rel(p.kcnt + g, 1) == 1) dk = K;
        }
      } else {
        if (atom_add_acq_rel(p.kcnt + g, 1) == 1) dk = K;
      }
    }
  }
  dk = __shfl_sync(0xffffffffu, dk, 0);
  if (dk >= 0) decide<DT>(p, cq, g, dk, c);
}

template <int DT>
__global__ void __launch_bounds__(kStreamThreads, 1)
    stream_kernel(const __grid_constant__ VerifyParams vp) {
  const StreamParams& p = vp.s;
  const CdfParams& cq = vp.q;  // the draws (cq.cpg == 0: none)
  const long long nS = p.nchunks;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStagesA * kStageBytes);
  uint64_t* empty = full + kStagesA;
  uint64_t* pfull = empty + kStagesA;
  uint64_t* pempty = pfull + kPieceSlots;
  PieceRed* slots = reinterpret_cast<PieceRed*>(pempty + kPieceSlots);
  __shared__ int s_err;
  __shared__ PieceDesc s_pq[kPieceQueue];
  __shared__ StageDesc s_sd[kStagesA];
  // The draft tokens of the launch, when they fit: the consumers pick each
  // row's draft-token logit out of the staged data, so the epilogue needs no
  // global gather.
  __shared__ int s_tok[kTokCache];
  // half-unit sums of a draw stage (two buffers: consecutive stages alternate,
  // kStagesA being even)
  static_assert(kStagesA % 2 == 0, "ring slots alternate in parity");
  __shared__ float s_half[2 * kConsumerWarps];
  const bool tok_smem = p.tokens != nullptr && (int64_t)p.B * p.tokK <= kTokCache;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  constexpr int ups = units_per_stage(Elem<DT>::kSize);  // units per stage

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
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int n = 0;
      const bool draws = cq.cpg > 0;
      const unsigned maxT = draws ? (unsigned)cq.groups * (unsigned)cq.cpg : 0u;
      // the first round of row chunks is static (chunk = CTA): a CTA's first
      // copy does not wait behind every CTA's atomic on the counter
      unsigned long long next = blockIdx.x;
      unsigned long long next_st = 0ull;  // its sequence's state (nothing decided yet)
      // Draw tickets.  At a piece boundary a producer that saw queued draws
      // nobody has taken claims a ticket (the first producer to reach a
      // boundary takes a new draw); a claimed ticket whose draw is not yet
      // published is held and read again at the next boundary.  The queue
      // counters and the held entry are loaded before the wait for a free
      // ring slot and read after it.
      long long ticket = -1;
      bool ticket_ok = draws;  // tickets may still carry draws
      bool slot_held = false;  // the ring slot of stage n is free
      for (int piece = 0;; ++piece) {
        long long c = -1;
        int e = 0;
        unsigned qh = 0, qt = 0;
        if (ticket >= 0) {
          e = (int)ld_relaxed_u32(reinterpret_cast<const unsigned*>(p.dq_entry + ticket));
        } else if (ticket_ok) {
          qh = ld_relaxed_u32(p.dq_head);
          qt = ld_relaxed_u32(p.dq_tail);
        }
        // the ring slot of the piece's first stage
        if (n >= kStagesA) mbar_wait(empty + n % kStagesA, ((n / kStagesA) - 1) & 1, &s_err, p.status);
        slot_held = true;
        if (ticket < 0 && ticket_ok && qh < qt) {
          const unsigned t = atomicAdd(p.dq_head, 1u);
          if (t < maxT) {
            ticket = t;
            e = (int)ld_relaxed_u32(reinterpret_cast<const unsigned*>(p.dq_entry + t));
          } else {
            ticket_ok = false;
          }
        }
        // 1. a draw chunk whose ticket is ready goes first
        if (e > 0) {
          __threadfence();  // acquire: the group's parameters after its entry
          c = nS + (e - 1);
          ticket = -1;
        }
        // 2. the next row chunk (its id and its sequence's state were fetched
        //    one piece ago); a target row past a known rejection is dropped
        while (c < 0 && next < (unsigned long long)nS) {
          const long long cand = (long long)next;
          const unsigned long long st = next_st;
          next = gridDim.x + atomicAdd(p.chunk_ctr, 1ull);
          next_st = chunk_state(p, (long long)next, nS);
          if (!chunk_past_rejection<DT>(p, cand, st)) c = cand;
        }
        // 3. nothing left to stream: wait for the draws still to come.  The
        //    producer leaves once every group is decided (no more draws can
        //    be queued) and its ticket has no draw.
        if (c < 0 && draws) {
          const unsigned long long t0 = global_ns();
          while (!s_err) {
            if (ticket < 0 && ticket_ok) {
              const unsigned t = atomicAdd(p.dq_head, 1u);
              if (t < maxT) ticket = t;
              else ticket_ok = false;
            }
            // one round trip per poll: the words are loaded together (relaxed)
            const int ev = ticket >= 0 ? (int)ld_relaxed_u32(
                                             reinterpret_cast<const unsigned*>(p.dq_entry + ticket))
                                       : 0;
            const int dec = (int)ld_relaxed_u32(reinterpret_cast<const unsigned*>(p.decided));
            if (ev > 0) {
              __threadfence();  // acquire: the group's parameters after its entry
              c = nS + (ev - 1);
              ticket = -1;
              break;
            }
            // every group decided: the tail is final (each push precedes its
            // group's decided count), read after an acquire fence
            if (dec >= cq.groups) {
              __threadfence();
              if (ticket < 0 || (unsigned)ticket >= ld_acquire_u32(p.dq_tail)) break;
            }
            // a producer without a ticket only waits for the end
            __nanosleep(ticket >= 0 ? 128 : 1024);
            if (global_ns() - t0 > kWaitLimitNs) {
              s_err = 1;
              if (p.status) atomicOr(p.status, SSD_DEV_TIMEOUT);
              break;
            }
          }
        }
        PieceDesc& d = s_pq[piece % kPieceQueue];
        if (c >= nS) {
          int64_t g;
          int u0, u1;
          cdf_chunk_geom(cq, c - nS, g, u0, u1);
          if (!(g >= 0 && g < cq.groups && u0 < u1)) {
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
          // end marker: one stage without data (its slot is held)
          mbar_arrive(full + n % kStagesA);
          ++n;
          break;
        }
        if (c >= nS) {
          constexpr int ES = Elem<DT>::kSize;
          const char* rt = d.gp.use_t ? row_ptr(cq.tgt, d.gp.row_t, cq.t_stride, ES) : nullptr;
          const char* rd = d.gp.use_d ? row_ptr(cq.dft, d.gp.row_d, cq.d_stride, ES) : nullptr;
          const DrawLayout lay = draw_layout<DT>(d.gp);
          for (int u = d.u0, un = 0; u < d.u1; u = un) {
            un = min(u + lay.ups, d.u1);
            const int slot = n % kStagesA;
            if (!slot_held && n >= kStagesA)
              mbar_wait(empty + slot, ((n / kStagesA) - 1) & 1, &s_err, p.status);
            slot_held = false;
            cdf_issue_stage<DT>(cq, rt, rd, u, un, ring + slot * kStageBytes, lay, full + slot,
                                &s_err);
            ++n;
          }
          continue;
        }
        int64_t row, pu0, pu1;
        int k;
        chunk_geom(p, c, row, k, pu0, pu1);
        bool is_t;
        const char* rp = row_address<DT>(p, row, is_t);
        const int64_t g = row / p.rpg;
        // published to the consumers by the arrival on the piece's first stage
        d.row = row;
        d.pu0 = pu0;
        d.pu1 = pu1;
        d.rp = rp;
        d.g = g;
        d.jr = (int)(row - g * p.rpg);
        d.s0 = (int)((pu0 - row * p.upr) / ups);
        d.c = seq_scale(p, g);
        d.need = row_need(p, g, d.jr);
        d.wsum = p.bsum != nullptr &&
                 (p.mode == kModeSaguaro || (p.mode == kModeVerify && d.jr == p.K));
        for (int64_t u = pu0, un = 0; u < pu1; u = un) {
          un = min(u + ups, pu1);
          const Stage st = stage_of<DT>(rp, p.V, (int)((u - row * p.upr) / ups));
          const int slot = n % kStagesA;
          if (!slot_held && n >= kStagesA)
            mbar_wait(empty + slot, ((n / kStagesA) - 1) & 1, &s_err, p.status);
          slot_held = false;
          StageDesc& sd = s_sd[slot];
          sd.nvec = (int)((st.a1 - st.a0) >> 4);
          sd.ei0 = st.e0 + (int)((st.a0 - st.b0) / Elem<DT>::kSize);
          sd.e0 = st.e0;
          sd.e1 = st.e1;
          sd.b0 = st.b0;
          const uint32_t bytes = (uint32_t)(st.a1 - st.a0);
          if (bytes > 0 && !s_err &&
              SSD_CHK(in_range(st.a0, st.a1, is_t ? p.t_lo : p.d_lo, is_t ? p.t_hi : p.d_hi),
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
    if (tok_smem) {
      // eight loads in flight per thread, then their checks and stores
      constexpr int kU = 8;
      const int nt = p.B * p.tokK;
      const int t0 = (warp - kEpilogueWarp) * 32 + lane;
      constexpr int kStep = kEpilogueWarps * 32;
      for (int i0 = t0; i0 < nt; i0 += kU * kStep) {
        int xs[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) xs[k] = i0 + k * kStep < nt ? __ldg(p.tokens + i0 + k * kStep) : 0;
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          int x = xs[k];
          if (x < 0 || x >= p.V) {
            if (p.status) atomicOr(p.status, SSD_DEV_BAD_TOKEN);
            x = 0;
          }
          if (i0 + k * kStep < nt) s_tok[i0 + k * kStep] = x;
        }
      }
      tok_bar_arrive();
    }
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
      const PieceRed& R = slots[slot];
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
      const int need = row_need(p, g, jr);  // list entries the row needs
      SAcc b;
      b.reset();
      if (lane < kConsumerWarps) {
        b.m = R.m[lane];
        b.mc = b.m == kNegInf ? kNegInf : __fmul_rn(b.m, c);
        b.hi = R.hi[lane];
        b.lo = R.lo[lane];
      }
      const int nb = R.nst * kConsumerWarps;
      float v[kBlkPerLane];
#pragma unroll
      for (int j = 0; j < kBlkPerLane; ++j) {
        const int bb = lane + 32 * j;
        v[j] = (need > 0 && bb < nb) ? R.bmax[bb] : kNegInf;
      }
      const float wmx = (need > 0 && lane < kConsumerWarps) ? R.wmax[lane] : kNegInf;
      const int ncand = need > 0 ? R.ncand : 0;
      float cvv[kMaxCand / 32];
      int cvi[kMaxCand / 32];
#pragma unroll
      for (int q = 0; q < kMaxCand / 32; ++q) {
        const int i = q * 32 + lane;
        cvv[q] = i < ncand && i < kMaxCand ? R.cand_v[i] : kNegInf;
        cvi[q] = i < ncand && i < kMaxCand ? R.cand_i[i] : 0;
      }
      // the row's draft token and, when this piece holds it, its logit
      const int jx = jr < p.nt ? jr : jr - p.nt;
      const int x = (tok_smem && jx < p.tokK) ? s_tok[g * p.tokK + jx] : -1;
      const bool in_piece = x >= 0 && (int64_t)x >= (pu0 - row * p.upr) * kUnitA &&
                            (int64_t)x < (pu1 - row * p.upr) * kUnitA;
      const float zx = in_piece ? R.zx : 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(pempty + slot);  // the slot may be refilled
      float M, MC, Shi, Slo;
      warp_softmax_merge(b.m, b.mc, b.hi, b.lo, c, M, MC, Shi, Slo);
      WarpList wl;
      wl.reset(need > 0 ? need : 1);
      if (need > 0) {
        if (ncand <= kMaxCand) {
          // the candidates the consumer warps listed
          for (int i0 = 0; i0 < ncand; i0 += 32) {
            const bool ok = i0 + lane < ncand;
            wl.offer(ok ? cvv[i0 / 32] : kNegInf, ok ? cvi[i0 / 32] : 0, ok);
          }
        } else {
          chunk_top<DT>(p, row, (int)((pu0 - row * p.upr) / (int64_t)ups), wmx, v, wl);
        }
      }
      if (p.nch == 1) {
        finalize_row<DT>(p, cq, row, c, M, MC, Shi, Slo, wl, need, x >= 0, x, zx, &cleared,
                         &s_err);
        continue;
      }
      // row split into chunks: publish the partial, the last arrival merges
      if (!SSD_CHK(row < p.NR && kch < p.nch, p.dbg, 6, row, kch)) continue;
      RowPartial* slotp = p.partials + (row * p.nch + kch);
      if (lane == 0) {
        slotp->m = M;
        slotp->s_hi = Shi;
        slotp->s_lo = Slo;
        slotp->zx = zx;
        slotp->has_zx = in_piece ? 1 : 0;
      }
      if (lane < kMaxTopK) {
        const bool ok = need > 0 && lane < need;
        slotp->tv[lane] = ok ? wl.lv : kNegInf;
        slotp->ti[lane] = ok ? wl.li : 0x7fffffff;
      }
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence();
        last = atomicAdd(p.row_cnt + row, 1) == p.nch - 1;
        if (last) __threadfence();
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      SAcc mrg;
      mrg.reset();
      for (int cc = lane; cc < p.nch; cc += 32) fold_partial(mrg, p.partials + (row * p.nch + cc), c);
      warp_softmax_merge(mrg.m, mrg.mc, mrg.hi, mrg.lo, c, M, MC, Shi, Slo);
      // the chunk that held the draft token gives its logit
      float zxm = 0.f;
      if (x >= 0) {
        bool mine = false;
        for (int cc = lane; cc < p.nch; cc += 32) {
          const RowPartial* pp = p.partials + (row * p.nch + cc);
          if (__ldcg(&pp->has_zx)) {
            zxm = __ldcg(&pp->zx);
            mine = true;
          }
        }
        const unsigned hz = __ballot_sync(0xffffffffu, mine);
        zxm = hz ? __shfl_sync(0xffffffffu, zxm, __ffs(hz) - 1) : 0.f;
      }
      WarpList rl;
      rl.reset(need > 0 ? need : 1);
      if (need > 0) {
        // the chunks' lists, eight chunks' loads in flight at a time
        constexpr int kB = 8;
        for (int c0 = 0; c0 < p.nch; c0 += kB) {
          float xs[kB];
          int is[kB];
#pragma unroll
          for (int q = 0; q < kB; ++q) {
            const bool ok = c0 + q < p.nch && lane < need;
            const RowPartial* pp = p.partials + (row * p.nch + c0 + q);
            xs[q] = ok ? __ldcg(&pp->tv[lane]) : kNegInf;
            is[q] = ok ? __ldcg(&pp->ti[lane]) : 0x7fffffff;
          }
#pragma unroll
          for (int q = 0; q < kB; ++q) rl.offer(xs[q], is[q], xs[q] != kNegInf);
        }
      }
      finalize_row<DT>(p, cq, row, c, M, MC, Shi, Slo, rl, need, x >= 0, x, zxm, &cleared,
                       &s_err);
    }
    return;
  }

  // ---------------- consumers ----------------
  SAcc a;
  constexpr int VEC = Elem<DT>::kVec;
  constexpr int N = kVpt * VEC;
  int slot = 0;         // ring stage of the next stage
  uint32_t phase = 0;   // its mbarrier phase parity
  if (tok_smem) tok_bar_sync();
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
        __syncwarp();
        if (warp == 0 && lane == 0) slots[qs].chunk = -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull + qs);
      }
      break;
    }
    // take the piece's result slot (its epilogue warp is done with it)
    if (lane == 0 && piece >= kPieceSlots)
      mbar_wait(pempty + ps, ((piece / kPieceSlots) - 1) & 1, &s_err, p.status);
    __syncwarp();
    PieceRed& R = slots[ps];
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
        cdf_consume_stage<DT>(cq, g, gp, rt, rd, u, un, ring + slot * kStageBytes, lay, warp,
                              s_half + (slot & 1) * kConsumerWarps);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
        if (++slot == kStagesA) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // the unit sums may be read by another CTA (the group's last chunk)
      if (cq.cpg > 1 && lane == 0) __threadfence();
      __syncwarp();
      if (warp == 0 && lane == 0) R.chunk = chunk;
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull + ps);
      continue;
    }
    const int64_t row = d.row, pu0 = d.pu0, pu1 = d.pu1;
    const int jr = d.jr;
    const bool is_t = jr < p.nt;
    (void)is_t;  // read by the bounds-checked build only
    const float c = d.c;
    const bool top = d.need > 0;
    const bool wsum = d.wsum != 0;
    const int s0 = d.s0;
    const int64_t g = d.g;
    const int jx = jr < p.nt ? jr : jr - p.nt;
    const int xtok = (tok_smem && jx < p.tokK) ? s_tok[g * p.tokK + jx] : -1;
    a.reset();
    float wmax = kNegInf;  // this warp's largest logit of the piece
    float mybm = kNegInf;  // lane s: this warp's block maximum of stage s of the piece
    if (top && warp == 0 && lane == 0) R.ncand = 0;
    const int nst = (int)((pu1 - pu0 + ups - 1) / ups);  // stages of the piece
    for (int s = 0; s < nst; ++s) {
      if (s != 0) mbar_wait(full + slot, phase, &s_err, p.status);
      // the stage's description and data are read first and the slot is
      // released before the arithmetic, so that the producer refills it
      // while this stage is reduced
      const StageDesc st = s_sd[slot];
      const int nvec = st.nvec;
      const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kStageBytes);
      const int vb = warp * kVecsPerWarp + lane;
      uint4 raw[kVpt];
      if (nvec == kStageVecs) {
#pragma unroll
        for (int k = 0; k < kVpt; ++k) raw[k] = sv[vb + 32 * k];
      } else {
        // partial stage: -inf padding beyond the staged vectors
        const uint4 pad = DT == 0 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                  : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
#pragma unroll
        for (int k = 0; k < kVpt; ++k)
          raw[k] = (vb + 32 * k < nvec && SSD_CHK(vb + 32 * k < kStageVecs, p.dbg, 10, vb, nvec))
                       ? sv[vb + 32 * k] : pad;
      }
      if (xtok >= 0 && lane == 0) {
        // the row's draft-token logit, from this warp's block of the stage
        const int xe = xtok - st.ei0;
        if (xe >= warp * kVecsPerWarp * VEC && xe < min((warp + 1) * kVecsPerWarp, nvec) * VEC)
          R.zx = Elem<DT>::smem(ring + slot * kStageBytes, xe);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + slot);
      if (++slot == kStagesA) {
        slot = 0;
        phase ^= 1u;
      }
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
      float vm = fmaxf(fmaxf(vq[0], vq[1]), fmaxf(vq[2], vq[3]));
      float ssum = 0.f;
      if (vm != kNegInf) ssum = a.take<N>(x, vm, c);
      if (wsum) {
        // the block's sum for the row's one-term draw: each lane's sum at
        // its own offset, rescaled to the warp's largest offset
        const float mcw = warp_max_f32(a.mc);
        float bs = (a.mc == kNegInf || ssum == 0.f) ? 0.f : ssum * ex2(a.mc - mcw);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) bs += __shfl_xor_sync(0xffffffffu, bs, off);
        const int64_t bi = (int64_t)(s0 + s) * kConsumerWarps + warp;
        if (lane == 0 && SSD_CHK(bi < p.nblk && g < cq.groups, p.dbg, 11, bi, g))
          p.bsum[g * p.nblk + bi] = make_float2(bs, mcw);
      }
      // unaligned head / tail elements (fewer than 32) by warp 0, from global memory
      if (warp == 0) {
        const int ei0 = st.ei0;
        const int hc = nvec > 0 ? ei0 - st.e0 : st.e1 - st.e0;
        const int ei1 = ei0 + nvec * VEC;
        const int tc = nvec > 0 ? st.e1 - ei1 : 0;
        for (int f0 = 0; f0 < hc + tc; f0 += 32) {
          const int f = f0 + lane;
          float xh = kNegInf;
          int idx = 0;
          if (f < hc + tc) {
            idx = f < hc ? st.e0 + f : ei1 + (f - hc);
            const uintptr_t fa = st.b0 + (uintptr_t)(idx - st.e0) * Elem<DT>::kSize;
            if (SSD_CHK(in_range(fa, fa + Elem<DT>::kSize, is_t ? p.t_lo : p.d_lo,
                                 is_t ? p.t_hi : p.d_hi), p.dbg, 2, idx, st.e0)) {
              xh = Elem<DT>::load(reinterpret_cast<const void*>(st.b0), (int64_t)(idx - st.e0));
              a.take<1>(&xh, xh, c);
              vm = fmaxf(vm, xh);
              if (idx == xtok) R.zx = xh;
            }
          }
        }
      }
      if (top) {
        const float bm = warp_max_f32(vm);
        wmax = fmaxf(wmax, bm);
        if (lane == s) mybm = bm;
        if (lane == 0) R.bmax[s * kConsumerWarps + warp] = bm;
      }
    }

    if (top) {
      // The piece's top-list candidates.  theta = the R-th largest of the W
      // warp maxima (R warps hold a logit >= theta, so no logit below it is
      // in the top R); each warp reads its own blocks whose maximum reaches
      // theta again and lists their logits >= theta.
      if (lane == 0) R.wmax[warp] = wmax;
      consumer_sync();
      float m = lane < kConsumerWarps ? R.wmax[lane] : kNegInf;
      float th = kNegInf;
      for (int r = 0; r < d.need; ++r) {
        const float mx = warp_max_f32(m);
        if (mx == kNegInf) {
          th = kNegInf;
          break;
        }
        th = mx;
        const unsigned who = __ballot_sync(0xffffffffu, m == mx);
        if (lane == __ffs(who) - 1) m = kNegInf;
      }
      unsigned cs = __ballot_sync(0xffffffffu, lane < nst && mybm != kNegInf && mybm >= th);
      while (cs) {
        const int sc = __ffs(cs) - 1;
        cs &= cs - 1;
        list_block<DT>(p, d.rp, is_t, s0 + sc, warp, th, row, R);
      }
    }
    // ---- hand the piece's per-warp results to the epilogue warp ----
    float M, MC, Shi, Slo;
    warp_softmax_merge(a.m, a.mc, a.hi, a.lo, c, M, MC, Shi, Slo);
    if (lane == 0) {
      R.m[warp] = M;
      R.hi[warp] = Shi;
      R.lo[warp] = Slo;
      if (warp == 0) {
        R.chunk = chunk;
        R.c = c;
        R.nst = nst;
      }
      // block sums of a split row are read by another CTA
      if (wsum && p.nch > 1) __threadfence();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(pfull + ps);
  }
}

}  // namespace

template <int DT>
cudaError_t launch_stream_dt(const VerifyParams& p, int grid, cudaStream_t s) {
  const int smem = stream_smem_bytes();
  auto kern = stream_kernel<DT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // CTAs wait for work that other CTAs do (draw tickets, split rows, the
  // round cache): all of them must be resident at once, which a cooperative
  // launch guarantees
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace ssd
