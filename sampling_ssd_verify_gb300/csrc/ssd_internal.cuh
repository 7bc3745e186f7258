// ssd_internal.cuh -- shared definitions of the CUDA library (not part of
// the public ABI): tuning constants, kernel parameter blocks, workspace
// records and small device helpers (PTX wrappers, Philox, reductions).
//
// Sources, cited by page title and section:
//   [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈"
//   [SD-7.3]   "7.3 Speculative Decoding：投机采样加速"
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// ---- tuning ------------------------------------------------------------------
constexpr int kConsumerWarps = 16;                  // warps that reduce staged data
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;           // + one producer (bulk-copy) warp
constexpr int kUnitA = 1024;                        // elements per work unit, streaming pass
constexpr int kStageBytes = 32768;                  // bytes per pipeline stage
constexpr int kStagesA = 6;                         // ring depth, streaming pass
constexpr int kUnitB = 512;                         // elements per unit, CDF pass
// units of the draws per stage of the streaming ring (target and draft runs
// of kStageBytes / 2 each)
__host__ __device__ constexpr int fused_units_per_stage(int esize) { return kStageBytes / 2 / (kUnitB * esize); }
constexpr int kMaxTopK = 16;                        // per-row candidate list (F + 1 <= 16)
constexpr int kMaxGrid = 4096;                      // bound on CTAs of one launch
constexpr int kMaxChunks = 16;                      // bound on chunks per row (streaming pass)
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s

enum Mode : int { kModeVerify = 0, kModeTopF = 1, kModeSaguaro = 2 };

// Per-(CTA, row piece) partial of the streaming pass.
struct RowPartial {
  float m;        // max raw logit of the piece
  float pad;
  float s_hi;     // sum of exp2(z*c - fl(m*c)) as a compensated pair
  float s_lo;
  float tv[kMaxTopK];
  int ti[kMaxTopK];
};

// Final per-row statistics.
struct RowResult {
  float m;        // max raw logit
  float mc;       // fl32(m * c): the offset every exponent of the row used
  double s;       // sum_y exp2(fl(z_y*c - mc))
  float zx;       // logit of the row's draft token (if the row has one)
  int x;
  float tv[kMaxTopK];  // top raw logits, descending, ties to the lower index
  int ti[kMaxTopK];
};

// Per-group (sequence / branch row) parameters of the CDF pass, written by
// the group epilogue of the streaming pass.
struct GroupParams {
  int k;            // verify: accept length; rows read by the CDF pass: see below
  int use_t;        // the CDF weight has a target term p(y)
  int use_d;        // the CDF weight has a draft term q'(y)
  int sign_d;       // +1: w = q'(y) (Saguaro draw), -1: w = (p(y) - q'(y))^+
  int64_t row_t;    // target row index (into the target tensor)
  int64_t row_d;    // draft row index (into the draft tensor)
  float mc_t, inv_st;        // p(y) = exp2(fl(z*c - mc_t)) * inv_st
  float mc_d, scale_out, scale_in;  // q'(y) = exp2(fl(z*c - mc_d)) * (in S ? scale_in : scale_out)
  float theta;      // S = { y : z > theta or (z == theta and y <= itheta) }
  int itheta;
  float c;          // log2(e) / T of the group
  double u;         // uniform of the draw
};
// A group whose outputs its epilogue already wrote (a greedy sequence): its
// draw chunks do nothing.
__host__ __device__ inline bool no_draw(const GroupParams& gp) { return !gp.use_t && !gp.use_d; }

// The outcome cache of one round built and probed inside the verify launch
// (ssd_verify_round): each draft row's guesses are inserted as the row is
// finalised, and each sequence looks its outcome up once its bonus is known.
// The epilogue warps clear the table at the start of the launch; inserts
// wait (bounded) until every CTA has cleared its slice.
struct RoundCache {
  void* table;               // Slot[cap] (ssd_cache_dev.cuh), or null: no cache
  int64_t cap;
  int32_t* branch;           // [B] out
  int32_t* all_hit;          // out (or null)
  unsigned long long* cnt;   // (finished sequences << 32) | hits, zeroed per call
  int* cleared;              // epilogue warps done clearing, zeroed per call
};

struct StreamParams {
  const void* tgt;
  int64_t t_stride;
  const void* dft;
  int64_t d_stride;
  int B, K, Kq, V;
  int nt, nd, rpg;          // target rows, draft rows per group, rows per group
  int64_t NR;               // rows in total
  int upr;                  // units per row
  int64_t total_units;
  // Rows are cut into nch chunks of clen units (the last one shorter); CTAs
  // take chunks in the order (chunk of row, row) from a global counter.
  int nch, clen;
  int64_t nchunks;
  unsigned long long* chunk_ctr;
  uint32_t* row_cut;        // per row: ordered-float lower bound on its top-list cut (0: none)
  float c;                  // log2(e) / T
  // Per-sequence temperature (device [B]) or null: then every sequence uses
  // T, greedy when greedy_all.  T = 0 is the greedy limit.
  const float* T_rows;
  int greedy_all;
  float C[SSD_MAX_K + 1];   // Saguaro factor per draft position (a continuation draw: C[0])
  int F[SSD_MAX_K + 1];
  int need_top;             // draft rows keep a top list
  const int32_t* tokens;    // [groups, tokK] or null
  int tokK;
  const uint64_t* seeds;
  uint32_t round;
  int jpos;                 // Saguaro: continuation position
  int mode;
  int32_t* accept_len;
  int32_t* bonus;           // written by the epilogue of a greedy sequence
  float* resid_mass;
  RoundCache rc;
  int32_t* guesses;         // [groups, nd, Fmax]
  float* guess_q;
  int Fmax;
  int* row_cnt;
  int* grp_cnt;
  int* grp_ready;           // per group: 1 once its draw parameters are published
  RowPartial* partials;     // slot row * nch + chunk of row
  // One-row draws whose unit sums the streaming pass writes (Saguaro rows,
  // aligned): per 32-vector sub-unit of each row, (sum of exp2(z*c - off),
  // off); null when the draws read the rows again.
  float2* usum;
  int nsu;                  // sub-units per row
  RowResult* rowres;
  GroupParams* gparams;
  int32_t* status;
  // bounds of the inputs and the debug record (used by SSD_CHECKS builds)
  const char* t_lo;
  const char* t_hi;
  const char* d_lo;
  const char* d_hi;
  unsigned long long* dbg;
};

struct CdfParams {
  const void* tgt;
  int64_t t_stride;
  const void* dft;
  int64_t d_stride;
  int groups, V, nsub;
  int64_t total_units;
  // Each group's nsub units are cut into cpg chunks of cu units (the last one
  // shorter), taken group by group.
  int cu, cpg;
  int64_t nchunks;
  int mode;
  const GroupParams* gp;
  const RowResult* rowres;  // Saguaro: the branch row's top list
  int rpg, nt;
  float* subsum;            // [groups, nsub]
  int* cnt;                 // [groups]
  int32_t* out_token;
  float* out_mass;          // verify: resid mass
  float* out_qprime;        // Saguaro: q'(x)
  int32_t* out_guess;       // Saguaro: [groups, F]
  int F;
  RoundCache rc;
  int32_t* status;
  const char* t_lo;
  const char* t_hi;
  const char* d_lo;
  const char* d_hi;
  unsigned long long* dbg;
};

// The streaming pass and the draws in one persistent launch: logical chunks
// [0, s.nchunks) stream rows, [s.nchunks, s.nchunks + q.nchunks) are chunks
// of the draws (none when q.nchunks is 0), all taken from the one counter
// s.chunk_ctr.  A chunk of the draws waits until its group's
// parameters are published (s.grp_ready), so the launch is cooperative.
struct VerifyParams {
  StreamParams s;
  CdfParams q;
};

// ---- workspace layout ----------------------------------------------------------
struct WsLayout {
  size_t cnt_off, cnt_bytes;       // counters (cleared each call)
  size_t ctr_off;                  // the chunk counter, within the counters
  size_t part_off, rowres_off, gp_off, sub_off, usum_off, dbg_off, total;
  int64_t NR;
  int groups, nsub;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// nch: chunks per row of the streaming pass; split rows (nch > 1) need one
// partial slot per chunk.  usum: room for the streaming pass's sub-unit sums
// of every row (sub-units of at least 128 elements).
inline WsLayout ws_layout(int groups, int rpg, int V, int nch, bool usum = false) {
  WsLayout L;
  L.groups = groups;
  L.NR = (int64_t)groups * rpg;
  L.nsub = (V + kUnitB - 1) / kUnitB;
  // counters: row arrivals [NR], group arrivals [groups], CDF arrivals
  // [groups], row cuts [NR], group-ready flags [groups], then 8-byte
  // counters: chunks, round-cache outcomes, round-cache clearing
  size_t ncnt = 2 * (size_t)L.NR + 3 * (size_t)groups;
  L.cnt_off = 0;
  L.ctr_off = (ncnt * sizeof(int) + 7) & ~(size_t)7;
  // chunk counter, round-cache outcomes, round-cache clearing
  L.cnt_bytes = align256(L.ctr_off + 3 * sizeof(unsigned long long));
  L.part_off = L.cnt_bytes;
  const size_t slots = nch > 1 ? (size_t)L.NR * nch : 1;
  L.rowres_off = L.part_off + align256(slots * sizeof(RowPartial));
  L.gp_off = L.rowres_off + align256((size_t)L.NR * sizeof(RowResult));
  L.sub_off = L.gp_off + align256((size_t)groups * sizeof(GroupParams));
  L.usum_off = L.sub_off + align256((size_t)groups * L.nsub * sizeof(float));
  const size_t usum_bytes = usum ? (size_t)L.NR * ((V + 127) / 128) * 2 * sizeof(float) : 0;
  L.dbg_off = L.usum_off + align256(usum_bytes);
  L.total = L.dbg_off + 256;  // bounds-check record of SSD_CHECKS builds
  return L;
}

// ---- launchers (defined in ssd_stream.cu / ssd_cdf.cu / ssd_cache.cu) -----------
cudaError_t launch_stream(const VerifyParams& p, int dtype, int topk, int grid,
                          cudaStream_t s);
cudaError_t launch_cache_clear(void* table, int64_t capacity, cudaStream_t s);
cudaError_t launch_cache_insert(void* table, int64_t capacity, const int32_t* row,
                                const int32_t* k, const int32_t* t, const int32_t* branch, int n,
                                const int32_t* guesses, int B, int Kq, int Fmax,
                                int32_t* status, cudaStream_t s);
cudaError_t launch_cache_lookup(const void* table, int64_t capacity, const int32_t* accept_len,
                                const int32_t* bonus, int B, int32_t* out_branch,
                                int32_t* all_hit, cudaStream_t s);
int stream_smem_bytes();
int num_sms();

}  // namespace ssd
