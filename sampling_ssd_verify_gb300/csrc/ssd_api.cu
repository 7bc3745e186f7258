// ssd_api.cu -- the C-ABI entry points: argument validation, workspace
// layout, launch configuration.  All arithmetic runs in the kernels of
// ssd_stream_kernel.cuh (the streaming pass with the draws of
// ssd_cdf_dev.cuh, instantiated by ssd_stream_bf16.cu / ssd_stream_f32.cu),
// ssd_tree.cu and ssd_cache.cu; the one host computation is the fan-out
// helper.
//
// Sources: [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈";
// [SD-7.3] "7.3 Speculative Decoding：投机采样加速".

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "ssd.h"
#include "ssd_internal.cuh"

namespace ssd {

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

namespace {

int esize_of(int32_t dtype) { return dtype == SSD_BF16 ? 2 : 4; }

bool logits_ok(const ssd_logits* L, int V) {
  if (L == nullptr || L->ptr == nullptr) return false;
  if (L->dtype != SSD_BF16 && L->dtype != SSD_F32) return false;
  if (L->pad_ != 0) return false;
  if (L->row_stride < V) return false;
  if (((uintptr_t)L->ptr) % esize_of(L->dtype) != 0) return false;
  return true;
}

bool finite_pos(float x) { return std::isfinite(x) && x > 0.f; }

ssd_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SSD_OK;
  cudaGetLastError();  // clear a sticky launch-configuration error
  return SSD_ERR_CUDA;
}

int64_t stream_grid0() {
  int sms = num_sms();
  if (sms <= 0) sms = 1;
  return std::min<int64_t>(sms, kMaxGrid);
}

int units_per_row(int V) { return (V + kUnitA - 1) / kUnitA; }

// Chunking of the streaming pass: nch chunks of clen units per row.  CTAs
// take chunks from a global counter, so a CTA that meets costlier rows takes
// fewer.  Whole rows when there are at least two per CTA (a row split over
// CTAs costs a partial merge); otherwise rows are cut into chunks of whole
// stages: about four per CTA in all, or, for a few rows (a latency-bound
// pass), at most one per CTA.  A chunk has at most kMaxChunkStages stages
// (its block maxima live in shared memory).  The launch and the workspace
// size both use it.
void stream_chunking(int64_t NR, int V, int esize, int& nch, int& clen) {
  const int64_t grid0 = stream_grid0();
  const int ups = units_per_stage(esize);
  const int upr = units_per_row(V);
  const int spr = (upr + ups - 1) / ups;
  int64_t want = 1;
  if (2 * NR <= grid0) {
    want = grid0 / NR;
  } else if (NR < 2 * grid0) {
    want = (4 * grid0 + NR - 1) / NR;
  }
  want = std::max<int64_t>(want, (spr + kMaxChunkStages - 1) / kMaxChunkStages);
  want = std::max<int64_t>(1, std::min<int64_t>(want, spr));
  const int sper = (int)((spr + want - 1) / want);  // stages per chunk
  clen = sper * ups;
  nch = (upr + clen - 1) / clen;
  if (nch == 1) clen = upr;
}

// Chunks per group of the draws: enough for about one per CTA when groups
// are few, and at most about 16 stages each (a draw chunk occupies its CTA's
// ring while rows wait), each at least one stage.
int draw_chunks_per_group(int groups, int V, int esize) {
  const int64_t grid0 = stream_grid0();
  const int nsub = (V + kUnitB - 1) / kUnitB;
  const int ups = fused_units_per_stage(esize);
  const int stages = (nsub + ups - 1) / ups;
  int64_t cpg = std::max<int64_t>((grid0 + groups - 1) / groups, (stages + 15) / 16);
  cpg = std::max<int64_t>(1, std::min<int64_t>(cpg, stages));
  const int cu = (int)((nsub + cpg - 1) / cpg);
  return (nsub + cu - 1) / cu;
}

WsLayout layout_for(int groups, int rpg, int K, int V, int esize, bool draws, bool bsum) {
  int nch, clen;
  stream_chunking((int64_t)groups * rpg, V, esize, nch, clen);
  const int cpg = draws ? draw_chunks_per_group(groups, V, esize) : 0;
  return ws_layout(groups, rpg, K, V, esize, nch, cpg, bsum);
}

// Workspace bytes for either element type.
size_t layout_bytes(int groups, int rpg, int K, int V, bool draws, bool bsum) {
  return std::max(layout_for(groups, rpg, K, V, 2, draws, bsum).total,
                  layout_for(groups, rpg, K, V, 4, draws, bsum).total);
}

// The 16-byte-aligned rows of whole vectors whose one-term draws can use the
// streaming pass's block sums.
bool rows_aligned(const ssd_logits* L, int V) {
  const int es = esize_of(L->dtype);
  return ((uintptr_t)L->ptr % 16) == 0 && (L->row_stride * es) % 16 == 0 && (V * es) % 16 == 0;
}

struct Common {
  StreamParams sp;
  CdfParams cp;
};

// Shared set-up of a launch over `groups` groups of rpg = nt + nd rows: the
// workspace layout, its counters cleared on the stream, the parameter
// blocks of the streaming pass and of the draws.
ssd_status setup(const ssd_logits* target, const ssd_logits* draft, int groups, int K, int Kq,
                 int nt, int nd, int V, float T, void* workspace, size_t ws_bytes,
                 cudaStream_t stream, Common& cm, bool draws, bool bsum) {
  const int rpg = nt + nd;
  const int es = esize_of(draft->dtype);
  int nch, clen;
  stream_chunking((int64_t)groups * rpg, V, es, nch, clen);
  const int cpg = draws ? draw_chunks_per_group(groups, V, es) : 0;
  const WsLayout L = ws_layout(groups, rpg, K, V, es, nch, cpg, bsum);
  if (workspace == nullptr || ((uintptr_t)workspace & 255) != 0 || ws_bytes < L.total)
    return SSD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws + L.cnt_off, 0, L.cnt_bytes, stream);
  if (e != cudaSuccess) return cuda_status(e);
  int* cnt = reinterpret_cast<int*>(ws + L.cnt_off);
  unsigned long long* w8 = reinterpret_cast<unsigned long long*>(ws + L.cnt_off + L.ctr_off);
  StreamParams& p = cm.sp;
  p = StreamParams{};
  p.tgt = target ? target->ptr : nullptr;
  p.t_stride = target ? target->row_stride : 0;
  p.dft = draft->ptr;
  p.d_stride = draft->row_stride;
  p.B = groups;
  p.K = K;
  p.Kq = Kq;
  p.V = V;
  p.nt = nt;
  p.nd = nd;
  p.rpg = rpg;
  p.NR = L.NR;
  p.upr = units_per_row(V);
  p.spr = L.nblk / kConsumerWarps;
  p.nblk = L.nblk;
  p.nch = nch;
  p.clen = clen;
  p.nchunks = L.NR * nch;
  p.order = 0;
  p.c = (float)(1.4426950408889634 / (double)T);  // log2(e) / T
  p.row_cnt = cnt + L.o_row_cnt;
  p.pair_cnt = cnt + L.o_pair;
  p.kcnt = cnt + L.o_kcnt;
  p.dq_entry = cnt + L.o_dq;
  p.seq_state = reinterpret_cast<unsigned long long*>(ws + L.cnt_off) + L.o_state;
  p.chunk_ctr = w8;
  p.dq_tail = reinterpret_cast<unsigned int*>(w8 + 3 * kCtrStride);
  p.dq_head = reinterpret_cast<unsigned int*>(w8 + 4 * kCtrStride);
  p.decided = reinterpret_cast<int*>(w8 + 5 * kCtrStride);
  p.skipped = w8 + 6 * kCtrStride;
  p.partials = reinterpret_cast<RowPartial*>(ws + L.part_off);
  p.rowres = reinterpret_cast<RowResult*>(ws + L.rowres_off);
  p.gparams = reinterpret_cast<GroupParams*>(ws + L.gp_off);
  p.bsum = bsum ? reinterpret_cast<float2*>(ws + L.bsum_off) : nullptr;
  if (target != nullptr) {
    p.t_lo = static_cast<const char*>(target->ptr);
    p.t_hi = p.t_lo + ((int64_t)(groups * (K + 1) - 1) * target->row_stride + V) * es;
  }
  p.d_lo = static_cast<const char*>(draft->ptr);
  p.d_hi = p.d_lo + ((int64_t)(groups * Kq - 1) * draft->row_stride + V) * es;
  // the bounds-check record of SSD_CHECKS builds: the caller's last 256
  // bytes (8-byte aligned), whatever layout this launch uses
  const size_t dbg_at = (ws_bytes - 256) & ~(size_t)7;
  p.dbg = reinterpret_cast<unsigned long long*>(ws + dbg_at);
#ifdef SSD_CHECKS
  e = cudaMemsetAsync(ws + dbg_at, 0, 256, stream);
  if (e != cudaSuccess) return cuda_status(e);
#endif
  CdfParams& q = cm.cp;
  q = CdfParams{};
  q.tgt = p.tgt;
  q.t_stride = p.t_stride;
  q.dft = p.dft;
  q.d_stride = p.d_stride;
  q.groups = groups;
  q.V = V;
  q.nsub = L.nsub;
  q.total_units = (int64_t)groups * L.nsub;
  q.cpg = cpg;
  q.cu = cpg > 0 ? (L.nsub + cpg - 1) / cpg : 0;
  q.nchunks = (int64_t)groups * cpg;
  q.gp = p.gparams;
  q.rowres = p.rowres;
  q.rpg = rpg;
  q.nt = nt;
  q.subsum = reinterpret_cast<float*>(ws + L.sub_off);
  q.cnt = cnt + L.o_grp_cnt;
  q.t_lo = p.t_lo;
  q.t_hi = p.t_hi;
  q.d_lo = p.d_lo;
  q.d_hi = p.d_hi;
  q.dbg = p.dbg;
  return SSD_OK;
}

// The launch: one CTA per SM, at most one per chunk of work.
ssd_status run_pass(Common& cm, int dtype, cudaStream_t s) {
  VerifyParams vp;
  vp.s = cm.sp;
  vp.q = cm.cp;
  const int grid =
      (int)std::max<int64_t>(1, std::min<int64_t>(stream_grid0(), vp.s.nchunks + vp.q.nchunks));
  const cudaError_t e = dtype == SSD_BF16 ? launch_stream_dt<0>(vp, grid, s)
                                          : launch_stream_dt<1>(vp, grid, s);
  return cuda_status(e);
}

int64_t capacity_of(size_t table_bytes) {
  int64_t cap = 1;
  while ((cap << 1) * 16 <= (int64_t)table_bytes) cap <<= 1;
  return cap * 16 <= (int64_t)table_bytes ? cap : 0;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

const char* ssd_status_string(int status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "beyond the compiled limits of the library";
    case SSD_ERR_TABLE_FULL: return "cache table too small (capacity must be >= 2 n)";
    case SSD_ERR_DUPLICATE_KEY: return "duplicate cache key";
    case SSD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SSD_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int ssd_version(void) { return 100; }

ssd_status ssd_fanout(int K, int budget, double a, double r, int32_t* F_out) {
  if (K < 0 || K > 4096 || budget < 0 || !(a > 0.0) || !std::isfinite(a) || !(r >= 0.0) ||
      !std::isfinite(r) || F_out == nullptr)
    return SSD_ERR_INVALID_ARG;
  // shares w_k = a^(k/(1+r)), normalised to the budget
  std::vector<double> share(K + 1);
  double total = 0.0;
  for (int k = 0; k <= K; ++k) total += (share[k] = std::exp(std::log(a) * k / (1.0 + r)));
  std::vector<int> order(K + 1);
  int given = 0;
  for (int k = 0; k <= K; ++k) {
    share[k] = share[k] * budget / total;
    F_out[k] = (int32_t)std::floor(share[k]);
    given += F_out[k];
    share[k] -= F_out[k];
    order[k] = k;
  }
  // remaining units to the largest fractional parts, ties to the lower k
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return share[x] > share[y]; });
  for (int i = 0; i < budget - given && i <= K; ++i) F_out[order[i]] += 1;
  return SSD_OK;
}

size_t ssd_verify_workspace_size(int B, int K, int Kq, int V) {
  if (B < 1 || K < 1 || K > SSD_MAX_K || (Kq != K && Kq != K + 1) || V < 2 || V > SSD_MAX_V)
    return 0;
  return layout_bytes(B, K + 1 + Kq, K, V, true, true);
}

ssd_status ssd_verify_skipped_bytes(const void* workspace, size_t workspace_bytes, int B, int K,
                                    int Kq, int V, int dtype, uint64_t* out, void* stream) {
  if (B < 1 || K < 1 || K > SSD_MAX_K || (Kq != K && Kq != K + 1) || V < 2 || V > SSD_MAX_V ||
      (dtype != SSD_BF16 && dtype != SSD_F32) || out == nullptr)
    return SSD_ERR_INVALID_ARG;
  if (workspace == nullptr || ((uintptr_t)workspace & 255) != 0 ||
      workspace_bytes < ssd_verify_workspace_size(B, K, Kq, V))
    return SSD_ERR_WORKSPACE;
  // the counter's place in the layout the call used (the counters do not
  // depend on the block-sum room)
  const WsLayout L = layout_for(B, K + 1 + Kq, K, V, esize_of(dtype), true, false);
  const char* ctr = static_cast<const char*>(workspace) + L.cnt_off + L.ctr_off +
                    6 * kCtrStride * sizeof(unsigned long long);
  return cuda_status(cudaMemcpyAsync(out, ctr, sizeof(uint64_t), cudaMemcpyDeviceToDevice,
                                     static_cast<cudaStream_t>(stream)));
}

size_t ssd_topf_workspace_size(int B, int Kq, int V) {
  if (B < 1 || Kq < 1 || Kq > SSD_MAX_K + 1 || V < 2 || V > SSD_MAX_V) return 0;
  return layout_bytes(B, Kq, 0, V, false, false);
}

size_t ssd_saguaro_workspace_size(int R, int V) {
  if (R < 1 || V < 2 || V > SSD_MAX_V) return 0;
  return layout_bytes(R, 1, 0, V, true, true);
}

}  // extern "C"

namespace {

// The outcome cache of a round built and probed in the verify launch.
struct RoundArgs {
  void* table;
  size_t table_bytes;
  int32_t* out_branch;
  int32_t* all_hit;
};

// ssd_verify with a Saguaro factor per draft position (Cv[0..K-1], host),
// when T_rows (device [B]) is given a temperature per sequence instead of T
// (T = 0 is the greedy limit), and when ra is given the round's cache.
ssd_status verify_impl(const ssd_logits* target, const ssd_logits* draft, int B, int K, int Kq,
                       int V, float T, const float* T_rows, const RoundArgs* ra,
                       const int32_t* draft_tokens, const uint64_t* seeds,
                       uint32_t round, const int32_t* fanout, const float* Cv,
                       int32_t* accept_len, int32_t* bonus, float* resid_mass, int32_t* guesses,
                       float* guess_q, int Fmax, void* workspace, size_t workspace_bytes,
                       int32_t* dev_status, void* stream) {
  if (B < 1 || K < 1 || K > SSD_MAX_K || (Kq != K && Kq != K + 1) || V < 2 || V > SSD_MAX_V)
    return SSD_ERR_INVALID_ARG;
  if (!logits_ok(target, V) || !logits_ok(draft, V) || target->dtype != draft->dtype)
    return SSD_ERR_INVALID_ARG;
  if (T_rows == nullptr && !(std::isfinite(T) && T >= 0.f)) return SSD_ERR_INVALID_ARG;
  if (Cv == nullptr) return SSD_ERR_INVALID_ARG;
  for (int j = 0; j < K; ++j)
    if (!std::isfinite(Cv[j]) || !(Cv[j] > 0.f) || Cv[j] > 1.f) return SSD_ERR_INVALID_ARG;
  if (!draft_tokens || !seeds || !accept_len || !bonus) return SSD_ERR_INVALID_ARG;
  if (guess_q && !guesses) return SSD_ERR_INVALID_ARG;
  int F[SSD_MAX_K + 1] = {0};
  int maxF = 0;
  if (fanout) {
    for (int j = 0; j < Kq; ++j) {
      if (fanout[j] < 0 || fanout[j] + 1 > V) return SSD_ERR_INVALID_ARG;
      if (fanout[j] > SSD_MAX_F) return SSD_ERR_UNSUPPORTED;
      F[j] = fanout[j];
      maxF = std::max(maxF, F[j]);
    }
  }
  if (guesses && (Fmax < 1 || Fmax < maxF)) return SSD_ERR_INVALID_ARG;
  int64_t cache_cap = 0;
  if (ra != nullptr) {
    if (!guesses || !ra->out_branch || !ra->table || ((uintptr_t)ra->table & 15) != 0)
      return SSD_ERR_INVALID_ARG;
    cache_cap = capacity_of(ra->table_bytes);
    if (cache_cap < 2 * (int64_t)B * Kq * Fmax) return SSD_ERR_TABLE_FULL;
  }
  // top lists are needed for the guesses and for every position that biases
  bool biased = false;
  for (int j = 0; j < K; ++j) biased |= Cv[j] < 1.f && F[j] > 0;
  const bool need_top = (guesses && maxF > 0) || biased;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Common cm;
  // a greedy sequence's (unused) sums take T = 1
  const bool greedy_all = T_rows == nullptr && T == 0.f;
  // all-accepted bonus draws of p_K from the streaming pass's block sums
  const bool direct = rows_aligned(target, V);
  ssd_status st = setup(target, draft, B, K, Kq, K + 1, Kq, V, T > 0.f ? T : 1.f, workspace,
                        workspace_bytes, s, cm, true, direct);
  if (st != SSD_OK) return st;
  StreamParams& p = cm.sp;
  for (int j = 0; j <= SSD_MAX_K; ++j) {
    p.F[j] = F[j];
    p.C[j] = j < K ? Cv[j] : 1.f;
  }
  p.order = 1;  // position-major: outcomes are decided while later positions stream
  p.T_rows = T_rows;
  p.greedy_all = greedy_all ? 1 : 0;
  p.bonus = bonus;
  p.resid_mass = resid_mass;
  if (ra != nullptr) {
    unsigned long long* w8 = p.chunk_ctr;
    p.rc.table = ra->table;
    p.rc.cap = cache_cap;
    p.rc.branch = ra->out_branch;
    p.rc.all_hit = ra->all_hit;
    p.rc.cnt = w8 + 1 * kCtrStride;
    p.rc.cleared = reinterpret_cast<int*>(w8 + 2 * kCtrStride);
    cm.cp.rc = p.rc;
  }
  p.need_top = need_top ? 1 : 0;
  p.tokens = draft_tokens;
  p.tokK = K;
  p.seeds = seeds;
  p.round = round;
  p.mode = kModeVerify;
  p.accept_len = accept_len;
  p.guesses = guesses;
  p.guess_q = guess_q;
  p.Fmax = Fmax;
  p.status = dev_status;
  CdfParams& q = cm.cp;
  q.mode = kModeVerify;
  q.out_token = bonus;
  q.out_mass = resid_mass;
  q.status = dev_status;
  return run_pass(cm, target->dtype, s);
}

}  // namespace

extern "C" {

ssd_status ssd_verify(const ssd_logits* target, const ssd_logits* draft, int B, int K, int Kq,
                      int V, float T, const int32_t* draft_tokens, const uint64_t* seeds,
                      uint32_t round, const int32_t* fanout, float C, int32_t* accept_len,
                      int32_t* bonus, float* resid_mass, int32_t* guesses, float* guess_q,
                      int Fmax, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      void* stream) {
  if (K < 1 || K > SSD_MAX_K) return SSD_ERR_INVALID_ARG;
  float Cv[SSD_MAX_K];
  for (int j = 0; j < K; ++j) Cv[j] = C;
  return verify_impl(target, draft, B, K, Kq, V, T, nullptr, nullptr, draft_tokens, seeds, round,
                     fanout, Cv,
                     accept_len, bonus, resid_mass, guesses, guess_q, Fmax, workspace,
                     workspace_bytes, dev_status, stream);
}

ssd_status ssd_verify_ck(const ssd_logits* target, const ssd_logits* draft, int B, int K,
                         int Kq, int V, float T, const int32_t* draft_tokens,
                         const uint64_t* seeds, uint32_t round, const int32_t* fanout,
                         const float* C_pos, int32_t* accept_len, int32_t* bonus,
                         float* resid_mass, int32_t* guesses, float* guess_q, int Fmax,
                         void* workspace, size_t workspace_bytes, int32_t* dev_status,
                         void* stream) {
  if (K < 1 || K > SSD_MAX_K || C_pos == nullptr) return SSD_ERR_INVALID_ARG;
  return verify_impl(target, draft, B, K, Kq, V, T, nullptr, nullptr, draft_tokens, seeds, round,
                     fanout, C_pos, accept_len, bonus, resid_mass, guesses, guess_q, Fmax, workspace,
                     workspace_bytes, dev_status, stream);
}

ssd_status ssd_verify_round(const ssd_logits* target, const ssd_logits* draft, int B, int K,
                            int Kq, int V, float T, const int32_t* draft_tokens,
                            const uint64_t* seeds, uint32_t round, const int32_t* fanout, float C,
                            int32_t* accept_len, int32_t* bonus, float* resid_mass,
                            int32_t* guesses, float* guess_q, int Fmax, void* table,
                            size_t table_bytes, int32_t* out_branch, int32_t* all_hit,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            void* stream) {
  if (K < 1 || K > SSD_MAX_K) return SSD_ERR_INVALID_ARG;
  float Cv[SSD_MAX_K];
  for (int j = 0; j < K; ++j) Cv[j] = C;
  const RoundArgs ra{table, table_bytes, out_branch, all_hit};
  return verify_impl(target, draft, B, K, Kq, V, T, nullptr, &ra, draft_tokens, seeds, round,
                     fanout, Cv, accept_len, bonus, resid_mass, guesses, guess_q, Fmax, workspace,
                     workspace_bytes, dev_status, stream);
}

ssd_status ssd_verify_ex(const ssd_logits* target, const ssd_logits* draft, int B, int K,
                         int Kq, int V, const float* T_rows, const int32_t* draft_tokens,
                         const uint64_t* seeds, uint32_t round, const int32_t* fanout,
                         const float* C_pos, int32_t* accept_len, int32_t* bonus,
                         float* resid_mass, int32_t* guesses, float* guess_q, int Fmax,
                         void* workspace, size_t workspace_bytes, int32_t* dev_status,
                         void* stream) {
  if (K < 1 || K > SSD_MAX_K || T_rows == nullptr) return SSD_ERR_INVALID_ARG;
  float Cv[SSD_MAX_K];
  for (int j = 0; j < K; ++j) Cv[j] = C_pos ? C_pos[j] : 1.f;
  return verify_impl(target, draft, B, K, Kq, V, 1.f, T_rows, nullptr, draft_tokens, seeds, round,
                     fanout, Cv, accept_len, bonus, resid_mass, guesses, guess_q, Fmax, workspace,
                     workspace_bytes, dev_status, stream);
}

ssd_status ssd_topf_bonus(const ssd_logits* draft, int B, int Kq, int V, float T,
                          const int32_t* draft_tokens, int K, const int32_t* fanout, int Fmax,
                          int32_t* guesses, float* guess_q, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (B < 1 || Kq < 1 || Kq > SSD_MAX_K + 1 || V < 2 || V > SSD_MAX_V) return SSD_ERR_INVALID_ARG;
  if (!logits_ok(draft, V) || !finite_pos(T) || !fanout || !guesses) return SSD_ERR_INVALID_ARG;
  if (draft_tokens && (K < 0 || K > Kq)) return SSD_ERR_INVALID_ARG;
  int F[SSD_MAX_K + 1] = {0};
  int maxF = 0;
  for (int j = 0; j < Kq; ++j) {
    if (fanout[j] < 0 || fanout[j] + 1 > V) return SSD_ERR_INVALID_ARG;
    if (fanout[j] > SSD_MAX_F) return SSD_ERR_UNSUPPORTED;
    F[j] = fanout[j];
    maxF = std::max(maxF, F[j]);
  }
  if (Fmax < 1 || Fmax < maxF) return SSD_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Common cm;
  ssd_status st = setup(nullptr, draft, B, 0, Kq, 0, Kq, V, T, workspace, workspace_bytes, s, cm,
                        false, false);
  if (st != SSD_OK) return st;
  StreamParams& p = cm.sp;
  for (int j = 0; j <= SSD_MAX_K; ++j) {
    p.F[j] = F[j];
    p.C[j] = 1.f;
  }
  p.need_top = maxF > 0;
  p.tokens = draft_tokens;
  p.tokK = draft_tokens ? K : 0;
  p.mode = kModeTopF;
  p.guesses = guesses;
  p.guess_q = guess_q;
  p.Fmax = Fmax;
  p.status = dev_status;
  return run_pass(cm, draft->dtype, s);
}

ssd_status ssd_saguaro_sample(const ssd_logits* draft, int R, int V, float T, float C,
                              const int32_t* F_row, int Fmax, const uint64_t* seeds, int j,
                              uint32_t round, int32_t* out_token, float* out_qprime,
                              int32_t* out_guess, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, void* stream) {
  if (R < 1 || V < 2 || V > SSD_MAX_V || !logits_ok(draft, V)) return SSD_ERR_INVALID_ARG;
  if (!finite_pos(T) || !std::isfinite(C) || !(C > 0.f) || C > 1.f) return SSD_ERR_INVALID_ARG;
  if (Fmax < 0 || Fmax + 1 > V || !seeds || !out_token || j < 0) return SSD_ERR_INVALID_ARG;
  if (Fmax > SSD_MAX_F) return SSD_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Common cm;
  // Aligned rows of whole 16-byte vectors: the streaming pass writes the
  // block sums the draw needs, and each row draws as soon as it is done,
  // without reading the row again.
  const bool direct = rows_aligned(draft, V);
  ssd_status st = setup(nullptr, draft, R, 0, 1, 0, 1, V, T, workspace, workspace_bytes, s, cm,
                        !direct, direct);
  if (st != SSD_OK) return st;
  StreamParams& p = cm.sp;
  p.F[0] = Fmax;
  p.F_rows = F_row;
  p.Fmax = Fmax;
  for (int i = 0; i <= SSD_MAX_K; ++i) p.C[i] = i == 0 ? C : 1.f;
  p.need_top = Fmax > 0;
  p.seeds = seeds;
  p.round = round;
  p.jpos = j;
  p.mode = kModeSaguaro;
  p.status = dev_status;
  CdfParams& q = cm.cp;
  q.mode = kModeSaguaro;
  q.out_token = out_token;
  q.out_qprime = out_qprime;
  q.out_guess = Fmax > 0 ? out_guess : nullptr;
  q.F = Fmax;
  q.F_rows = F_row;
  q.status = dev_status;
  return run_pass(cm, draft->dtype, s);
}

size_t ssd_tree_workspace_size(int B, int N, int V) {
  if (B < 1 || N < 1 || N > kMaxTreeNodes || V < 2 || V > SSD_MAX_V) return 0;
  return layout_bytes(B, 2 * N, N - 1, V, false, false);
}

ssd_status ssd_tree_verify(const ssd_logits* target, const ssd_logits* draft, int B, int N, int V,
                           float T, const int32_t* parent, const int32_t* tokens,
                           const uint64_t* seeds, uint32_t round, int32_t* accept_len,
                           int32_t* path, int Dmax, int32_t* bonus, float* resid_mass,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream) {
  if (B < 1 || N < 1 || N > kMaxTreeNodes || V < 2 || V > SSD_MAX_V) return SSD_ERR_INVALID_ARG;
  if (!logits_ok(target, V) || !logits_ok(draft, V) || target->dtype != draft->dtype)
    return SSD_ERR_INVALID_ARG;
  if (!finite_pos(T) || !parent || !tokens || !seeds || !accept_len || !bonus)
    return SSD_ERR_INVALID_ARG;
  if (parent[0] != -1) return SSD_ERR_INVALID_ARG;
  int depth[kMaxTreeNodes] = {0};
  int dmax = 0;
  for (int u = 1; u < N; ++u) {
    if (parent[u] < 0 || parent[u] >= u) return SSD_ERR_INVALID_ARG;
    depth[u] = depth[parent[u]] + 1;
    dmax = std::max(dmax, depth[u]);
  }
  if (path && Dmax < dmax) return SSD_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Common cm;
  // every node's target and draft row: group b holds target rows b*N .. and
  // draft rows b*N .. (K + 1 = Kq = N)
  ssd_status st = setup(target, draft, B, N - 1, N, N, N, V, T, workspace, workspace_bytes, s, cm,
                        false, false);
  if (st != SSD_OK) return st;
  StreamParams& p = cm.sp;
  for (int j = 0; j <= SSD_MAX_K; ++j) {
    p.F[j] = 0;
    p.C[j] = 1.f;
  }
  p.mode = kModeTopF;
  p.status = dev_status;
  st = run_pass(cm, target->dtype, s);
  if (st != SSD_OK) return st;
  TreeParams tp{};
  tp.B = B;
  tp.N = N;
  tp.V = V;
  // CTAs per tree: the most (up to 8) that keep every tree's cluster resident
  // at once (one 512-thread CTA per SM)
  tp.cluster = kTreeMaxCluster;
  while (tp.cluster > 1 && (int64_t)B * tp.cluster > (int64_t)std::max(num_sms(), 1))
    tp.cluster >>= 1;
  tp.c = p.c;
  tp.tgt = p.tgt;
  tp.t_stride = p.t_stride;
  tp.dft = p.dft;
  tp.d_stride = p.d_stride;
  tp.tokens = tokens;
  tp.seeds = seeds;
  tp.round = round;
  tp.rowres = p.rowres;
  tp.gparams = p.gparams;
  int n = 0;
  for (int u = 0; u < N; ++u) {
    tp.child_off[u] = n;
    for (int v = u + 1; v < N; ++v)
      if (parent[v] == u) tp.child[n++] = v;
  }
  tp.child_off[N] = n;
  tp.accept_len = accept_len;
  tp.path = path;
  tp.Dmax = Dmax;
  tp.resid_mass = resid_mass;
  tp.status = dev_status;
  tp.q = cm.cp;
  tp.q.mode = kModeVerify;
  tp.q.out_token = bonus;
  tp.q.status = dev_status;
  const cudaError_t e = target->dtype == SSD_BF16 ? launch_tree_dt<0>(tp, s) : launch_tree_dt<1>(tp, s);
  return cuda_status(e);
}

size_t ssd_cache_bytes(int n_keys) {
  if (n_keys < 0) return 0;
  int64_t cap = 16;
  while (cap < 2 * (int64_t)n_keys) cap <<= 1;
  return (size_t)cap * 16;
}

ssd_status ssd_cache_build(void* table, size_t table_bytes, const int32_t* row, const int32_t* k,
                           const int32_t* t, const int32_t* branch, int n, int32_t* dev_status,
                           void* stream) {
  if (table == nullptr || ((uintptr_t)table & 15) != 0 || n < 0) return SSD_ERR_INVALID_ARG;
  if (n > 0 && (!row || !k || !t || !branch)) return SSD_ERR_INVALID_ARG;
  const int64_t cap = capacity_of(table_bytes);
  if (cap < 2 * (int64_t)n || cap < 1) return SSD_ERR_TABLE_FULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ssd_status st = cuda_status(launch_cache_clear(table, cap, s));
  if (st != SSD_OK) return st;
  return cuda_status(launch_cache_insert(table, cap, row, k, t, branch, n, nullptr, 0, 0, 0,
                                         dev_status, s));
}

ssd_status ssd_cache_build_guesses(void* table, size_t table_bytes, const int32_t* guesses, int B,
                                   int Kq, int Fmax, int32_t* dev_status, void* stream) {
  if (table == nullptr || ((uintptr_t)table & 15) != 0 || !guesses || B < 1 || Kq < 1 ||
      Kq > 255 || Fmax < 1)
    return SSD_ERR_INVALID_ARG;
  const int64_t n = (int64_t)B * Kq * Fmax;
  if (n > (int64_t)0x3fffffff) return SSD_ERR_INVALID_ARG;
  const int64_t cap = capacity_of(table_bytes);
  if (cap < 2 * n) return SSD_ERR_TABLE_FULL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ssd_status st = cuda_status(launch_cache_clear(table, cap, s));
  if (st != SSD_OK) return st;
  return cuda_status(launch_cache_insert(table, cap, nullptr, nullptr, nullptr, nullptr, 0,
                                         guesses, B, Kq, Fmax, dev_status, s));
}

ssd_status ssd_cache_lookup(const void* table, size_t table_bytes, const int32_t* accept_len,
                            const int32_t* bonus, int B, int32_t* out_branch, int32_t* all_hit,
                            void* stream) {
  if (table == nullptr || ((uintptr_t)table & 15) != 0 || !accept_len || !bonus || B < 1 ||
      !out_branch)
    return SSD_ERR_INVALID_ARG;
  const int64_t cap = capacity_of(table_bytes);
  if (cap < 1) return SSD_ERR_INVALID_ARG;
  return cuda_status(launch_cache_lookup(table, cap, accept_len, bonus, B, out_branch, all_hit,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
