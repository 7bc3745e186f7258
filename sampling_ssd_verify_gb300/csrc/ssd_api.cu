// ssd_api.cu -- the C-ABI entry points: argument validation, workspace
// layout, launch configuration.  All arithmetic runs in the kernels of
// ssd_stream.cu (the streaming pass with the draws of ssd_cdf_dev.cuh) and
// ssd_cache.cu; the one host computation is the fan-out helper.
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

int topk_for(int maxF) {
  const int need = maxF + 1;
  if (need <= 2) return 2;
  if (need <= 4) return 4;
  if (need <= 8) return 8;
  return 16;
}

ssd_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SSD_OK;
  cudaGetLastError();  // clear a sticky launch-configuration error
  return SSD_ERR_CUDA;
}

// Chunks per row of the streaming pass.  CTAs take chunks from a global
// counter, so a CTA that meets costlier rows (more top-list insertions)
// takes fewer.  Whole rows when there are at least two per CTA (a row split
// over CTAs costs a partial merge and restarts its top-list pruning);
// otherwise rows are cut into up to kMaxChunks equal non-empty chunks: about
// four per CTA in all, or, for a few rows (a latency-bound pass), at most
// one per CTA.  The launch and the workspace size both use it.
int64_t stream_grid0() {
  int sms = num_sms();
  if (sms <= 0) sms = 1;
  return std::min<int64_t>(sms, kMaxGrid);
}

int stream_chunk_len(int64_t NR, int upr) {
  const int64_t grid0 = stream_grid0();
  int64_t nch = 1;
  if (2 * NR <= grid0) {
    // a few rows (small batches): latency-bound, so one round of chunks
    nch = grid0 / NR;
  } else if (NR < 2 * grid0) {
    nch = (4 * grid0 + NR - 1) / NR;
  }
  nch = std::max<int64_t>(1, std::min<int64_t>({nch, (int64_t)kMaxChunks, (int64_t)upr}));
  return (int)((upr + nch - 1) / nch);
}

int stream_chunks_per_row(int64_t NR, int upr) {
  const int clen = stream_chunk_len(NR, upr);
  return (upr + clen - 1) / clen;
}

int units_per_row(int V) { return (V + kUnitA - 1) / kUnitA; }

struct Common {
  StreamParams sp;
  CdfParams cp;
};

// Shared set-up of the streaming pass and the CDF pass over `groups` groups of
// rpg = nt + nd rows.
ssd_status setup(const ssd_logits* target, const ssd_logits* draft, int groups, int K, int Kq,
                 int nt, int nd, int V, float T, void* workspace, size_t ws_bytes,
                 cudaStream_t stream, Common& cm, WsLayout& L, bool usum = false) {
  const int rpg = nt + nd;
  L = ws_layout(groups, rpg, V,
                stream_chunks_per_row((int64_t)groups * rpg, units_per_row(V)), usum);
  if (workspace == nullptr || ((uintptr_t)workspace & 255) != 0 || ws_bytes < L.total)
    return SSD_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws + L.cnt_off, 0, L.cnt_bytes, stream);
  if (e != cudaSuccess) return cuda_status(e);
  int* cnt = reinterpret_cast<int*>(ws + L.cnt_off);
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
  p.total_units = L.NR * p.upr;
  p.c = (float)(1.4426950408889634 / (double)T);  // log2(e) / T
  p.row_cnt = cnt;
  p.grp_cnt = cnt + L.NR;
  p.row_cut = reinterpret_cast<uint32_t*>(cnt + L.NR + 2 * groups);
  p.grp_ready = cnt + 2 * L.NR + 2 * groups;
  p.chunk_ctr = reinterpret_cast<unsigned long long*>(ws + L.cnt_off + L.ctr_off);
  p.partials = reinterpret_cast<RowPartial*>(ws + L.part_off);
  p.rowres = reinterpret_cast<RowResult*>(ws + L.rowres_off);
  p.gparams = reinterpret_cast<GroupParams*>(ws + L.gp_off);
  if (usum) {
    p.usum = reinterpret_cast<float2*>(ws + L.usum_off);
    const int su = 32 * (16 / esize_of(draft->dtype));  // 32 vectors of 16 bytes
    p.nsu = (V + su - 1) / su;
  }
  const int es = esize_of(draft->dtype);
  if (target != nullptr) {
    p.t_lo = static_cast<const char*>(target->ptr);
    p.t_hi = p.t_lo + ((int64_t)(groups * (K + 1) - 1) * target->row_stride + V) * es;
  }
  p.d_lo = static_cast<const char*>(draft->ptr);
  p.d_hi = p.d_lo + ((int64_t)(groups * Kq - 1) * draft->row_stride + V) * es;
  p.dbg = reinterpret_cast<unsigned long long*>(ws + L.dbg_off);
#ifdef SSD_CHECKS
  e = cudaMemsetAsync(ws + L.dbg_off, 0, 256, stream);
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
  q.gp = p.gparams;
  q.rowres = p.rowres;
  q.rpg = rpg;
  q.nt = nt;
  q.subsum = reinterpret_cast<float*>(ws + L.sub_off);
  q.cnt = cnt + L.NR + groups;
  q.t_lo = p.t_lo;
  q.t_hi = p.t_hi;
  q.d_lo = p.d_lo;
  q.d_hi = p.d_hi;
  q.dbg = p.dbg;
  return SSD_OK;
}

// Chunking of the streaming pass and, when `draws`, of the draws that follow
// it in the same launch; then the launch.
//
// Draws: units of kUnitB elements, fused_units_per_stage per ring stage, cut
// into chunks of cu units -- about four per CTA in all, at most eight stages
// each (a small pass, latency-bound, takes one round) -- and taken group by
// group, the order in which the streaming pass completes the groups, so
// that a chunk rarely waits for its group's parameters.
ssd_status run_pass(Common& cm, int dtype, int topk, bool draws, cudaStream_t s) {
  StreamParams& p = cm.sp;
  CdfParams& q = cm.cp;
  const int64_t grid0 = stream_grid0();
  p.clen = stream_chunk_len(p.NR, p.upr);
  p.nch = (p.upr + p.clen - 1) / p.clen;
  p.nchunks = p.NR * p.nch;
  q.nchunks = 0;
  if (draws) {
    const int ups = fused_units_per_stage(esize_of(dtype));
    int64_t cu = q.total_units >= 8 * grid0 ? (q.total_units + 4 * grid0 - 1) / (4 * grid0)
                                            : (q.total_units + grid0 - 1) / grid0;
    cu = std::max<int64_t>(1, std::min<int64_t>({cu, 8 * (int64_t)ups, (int64_t)q.nsub}));
    q.cu = (int)cu;
    q.cpg = (q.nsub + q.cu - 1) / q.cu;
    q.nchunks = (int64_t)q.groups * q.cpg;
  } else {
    p.grp_ready = nullptr;
  }
  VerifyParams vp;
  vp.s = p;
  vp.q = q;
  const int grid = (int)std::min<int64_t>(grid0, p.nchunks + q.nchunks);
  return cuda_status(launch_stream(vp, dtype, topk, grid, s));
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
    case SSD_ERR_UNSUPPORTED: return "unsupported by this build";
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
  return ws_layout(B, K + 1 + Kq, V,
                   stream_chunks_per_row((int64_t)B * (K + 1 + Kq), units_per_row(V))).total;
}

size_t ssd_topf_workspace_size(int B, int Kq, int V) {
  if (B < 1 || Kq < 1 || Kq > SSD_MAX_K + 1 || V < 2 || V > SSD_MAX_V) return 0;
  return ws_layout(B, Kq, V, stream_chunks_per_row((int64_t)B * Kq, units_per_row(V))).total;
}

size_t ssd_saguaro_workspace_size(int R, int V) {
  if (R < 1 || V < 2 || V > SSD_MAX_V) return 0;
  return ws_layout(R, 1, V, stream_chunks_per_row((int64_t)R, units_per_row(V)), true).total;
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
  WsLayout L;
  // a greedy sequence's (unused) sums take T = 1
  const bool greedy_all = T_rows == nullptr && T == 0.f;
  ssd_status st = setup(target, draft, B, K, Kq, K + 1, Kq, V, T > 0.f ? T : 1.f, workspace,
                        workspace_bytes, s, cm, L);
  if (st != SSD_OK) return st;
  StreamParams& p = cm.sp;
  for (int j = 0; j <= SSD_MAX_K; ++j) {
    p.F[j] = F[j];
    p.C[j] = j < K ? Cv[j] : 1.f;
  }
  p.T_rows = T_rows;
  p.greedy_all = greedy_all ? 1 : 0;
  p.bonus = bonus;
  p.resid_mass = resid_mass;
  if (ra != nullptr) {
    p.rc.table = ra->table;
    p.rc.cap = cache_cap;
    p.rc.branch = ra->out_branch;
    p.rc.all_hit = ra->all_hit;
    p.rc.cnt = p.chunk_ctr + 1;
    p.rc.cleared = reinterpret_cast<int*>(p.chunk_ctr + 2);
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
  // greedy sequences keep a one-entry list (the argmax) on their target rows
  int topk = need_top ? topk_for(maxF) : 0;
  if (T_rows != nullptr || greedy_all) topk = std::max(topk, 2);
  return run_pass(cm, target->dtype, topk, true, s);
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
  WsLayout L;
  ssd_status st = setup(nullptr, draft, B, 0, Kq, 0, Kq, V, T, workspace, workspace_bytes, s, cm, L);
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
  return run_pass(cm, draft->dtype, maxF > 0 ? topk_for(maxF) : 0, false, s);
}

ssd_status ssd_saguaro_sample(const ssd_logits* draft, int R, int V, float T, float C, int F,
                              const uint64_t* seeds, int j, uint32_t round, int32_t* out_token,
                              float* out_qprime, int32_t* out_guess, void* workspace,
                              size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (R < 1 || V < 2 || V > SSD_MAX_V || !logits_ok(draft, V)) return SSD_ERR_INVALID_ARG;
  if (!finite_pos(T) || !std::isfinite(C) || !(C > 0.f) || C > 1.f) return SSD_ERR_INVALID_ARG;
  if (F < 0 || F + 1 > V || !seeds || !out_token || j < 0) return SSD_ERR_INVALID_ARG;
  if (F > SSD_MAX_F) return SSD_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Common cm;
  WsLayout L;
  // Aligned rows of whole 16-byte vectors: the streaming pass writes the
  // sub-unit sums the draw needs, and each row draws as soon as it is done,
  // without reading the row again.
  const int es = esize_of(draft->dtype);
  const bool direct = ((uintptr_t)draft->ptr % 16) == 0 && (draft->row_stride * es) % 16 == 0 &&
                      (V * es) % 16 == 0;
  ssd_status st = setup(nullptr, draft, R, 0, 1, 0, 1, V, T, workspace, workspace_bytes, s, cm, L,
                        direct);
  if (st != SSD_OK) return st;
  StreamParams& p = cm.sp;
  p.F[0] = F;
  for (int j = 0; j <= SSD_MAX_K; ++j) p.C[j] = j == 0 ? C : 1.f;
  const bool need_top = F > 0;
  p.need_top = need_top;
  p.seeds = seeds;
  p.round = round;
  p.jpos = j;
  p.mode = kModeSaguaro;
  p.status = dev_status;
  CdfParams& q = cm.cp;
  q.mode = kModeSaguaro;
  q.out_token = out_token;
  q.out_qprime = out_qprime;
  q.out_guess = F > 0 ? out_guess : nullptr;
  q.F = F;
  q.status = dev_status;
  return run_pass(cm, draft->dtype, need_top ? topk_for(F) : 0, !direct, s);
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
