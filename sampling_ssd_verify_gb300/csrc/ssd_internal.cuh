// ssd_internal.cuh -- shared definitions of the CUDA library (not part of
// the public ABI): tuning constants, kernel parameter blocks, workspace
// records and the launcher declarations.
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
constexpr int kUnitA = 1024;                        // elements per work unit, streaming pass
constexpr int kStageBytes = 32768;                  // bytes per pipeline stage
constexpr int kStagesA = 6;                         // ring depth
constexpr int kStageVecs = kStageBytes / 16;        // 16-byte vectors per stage
constexpr int kVecsPerWarp = kStageVecs / kConsumerWarps;  // one block: 128 vectors
constexpr int kVpt = kVecsPerWarp / 32;             // vectors per consumer thread and stage
constexpr int kUnitB = 512;                         // elements per unit of the draws
constexpr int kMaxTopK = 16;                        // per-row candidate list (F + 1 <= 16)
constexpr int kMaxChunkStages = 32;                 // stages of one row chunk (block maxima in smem)
constexpr int kMaxBlocks = kMaxChunkStages * kConsumerWarps;
constexpr int kBlkPerLane = kMaxBlocks / 32;            // block maxima per lane of a warp
static_assert(kMaxBlocks % 32 == 0 && kBlkPerLane <= 32, "block maxima fit one mask per lane");
constexpr int kMaxGrid = 4096;                      // bound on CTAs of one launch
constexpr int kTokCache = 4096;                     // draft tokens kept in shared memory
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // bounded waits: 2 s

// units of the draws per stage when both rows are read (target and draft
// runs of kStageBytes / 2 each)
__host__ __device__ constexpr int fused_units_per_stage(int esize) {
  return kStageBytes / 2 / (kUnitB * esize);
}
// units of the streaming pass per stage
__host__ __device__ constexpr int units_per_stage(int esize) {
  return kStageBytes / (kUnitA * esize);
}

enum Mode : int { kModeVerify = 0, kModeTopF = 1, kModeSaguaro = 2 };

// Per-(row chunk) partial of the streaming pass, merged by the last chunk
// of the row to finish.
struct RowPartial {
  float m;        // max raw logit of the chunk
  float zx;       // logit of the row's draft token, when the chunk holds it
  float s_hi;     // sum of exp2(z*c - fl(m*c)) as a compensated pair
  float s_lo;
  int has_zx;
  float tv[kMaxTopK];  // the chunk's exact top list (value desc, index asc)
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

// Per-group (sequence / branch row) parameters of a draw, written by the
// thread that decides the group's outcome.
struct GroupParams {
  int k;            // verify: accept length
  int use_t;        // the draw weight has a target term p(y)
  int use_d;        // the draw weight has a draft term q'(y)
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
// A group whose outputs its epilogue already wrote (a greedy sequence): no draw.
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
  int upr;                  // units (kUnitA elements) per row
  int spr;                  // stages per row
  int nblk;                 // blocks (one consumer warp's share of a stage) per row
  // Rows are cut into nch chunks of clen units (a multiple of the stage
  // length, the last one shorter); CTAs take chunks from a global counter.
  // order 0: chunk c is (chunk c / NR of row c % NR); order 1 (verify):
  // position-major -- for each draft position i, every sequence's target
  // and draft rows of position i, so that outcomes are decided (and their
  // draws run, from L2) while later positions stream.
  int nch, clen;
  int order;
  int64_t nchunks;
  unsigned long long* chunk_ctr;
  float c;                  // log2(e) / T
  // Per-sequence temperature (device [B]) or null: then every sequence uses
  // T, greedy when greedy_all.  T = 0 is the greedy limit.
  const float* T_rows;
  int greedy_all;
  float C[SSD_MAX_K + 1];   // Saguaro factor per draft position (a continuation draw: C[0])
  int F[SSD_MAX_K + 1];
  const int32_t* F_rows;    // Saguaro: device [R] fan-out per row, or null: F[0]
  int need_top;             // draft rows keep a top list
  const int32_t* tokens;    // [groups, tokK] or null
  int tokK;
  const uint64_t* seeds;
  uint32_t round;
  int jpos;                 // Saguaro: continuation position
  int mode;
  int32_t* accept_len;
  int32_t* bonus;           // written directly for greedy sequences and direct draws
  float* resid_mass;
  RoundCache rc;
  int32_t* guesses;         // [groups, nd, Fmax]
  float* guess_q;
  int Fmax;
  int* row_cnt;             // [NR] chunk arrivals of split rows
  RowPartial* partials;     // slot row * nch + chunk of row
  RowResult* rowres;
  GroupParams* gparams;
  // One-row draws straight from the streaming pass (aligned rows: Saguaro
  // rows, and target row K of a verified sequence): per (group, block) the
  // sum of exp2(z*c - off) over the block and its offset off; null when
  // those draws read their row again.
  float2* bsum;
  // Sequence outcomes (verify): per (sequence, position) arrivals of the
  // position's rows, per sequence the state word (bit i: position i
  // accepted, bit 32 + i: rejected) and the all-accepted counter.
  int* pair_cnt;
  unsigned long long* seq_state;
  int* kcnt;
  // Draw queue: a decided group's chunks are pushed as tickets (entry =
  // chunk id + 1, 0 while unwritten); producers claim tickets in order.
  int* dq_entry;
  unsigned int* dq_tail;
  unsigned int* dq_head;
  int* decided;             // groups whose draw is queued or done
  unsigned long long* skipped;  // bytes of target rows not streamed (past a rejection)
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
  // shorter); chunk id = group * cpg + chunk.
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
  int32_t* out_guess;       // Saguaro: [groups, Fmax]
  int F;                    // Saguaro: Fmax (columns of out_guess)
  const int32_t* F_rows;    // Saguaro: per-row fan-out, or null: F
  RoundCache rc;
  int32_t* status;
  const char* t_lo;
  const char* t_hi;
  const char* d_lo;
  const char* d_hi;
  unsigned long long* dbg;
};

// The streaming pass and the draws in one persistent launch: row chunks
// [0, s.nchunks) from the counter s.chunk_ctr, draw chunks from the ticket
// queue as groups are decided.  CTAs wait for one another (draw tickets,
// split rows, the round cache), so the launch is cooperative.
struct VerifyParams {
  StreamParams s;
  CdfParams q;
};

// Tree-draft verification (ssd_tree.cu): one cluster of `cluster` CTAs per
// tree walks it after the streaming pass has normalised every row (row u of
// tree b: target at rowres[b * 2N + u], draft at rowres[b * 2N + N + u]).
constexpr int kMaxTreeNodes = 256;
constexpr int kTreeMaxCluster = 8;
struct TreeParams {
  int B, N, V;
  int cluster;              // CTAs per tree: 1, 2, 4 or 8
  float c;                  // log2(e) / T
  const void* tgt;
  int64_t t_stride;
  const void* dft;
  int64_t d_stride;
  const int32_t* tokens;    // [B, N]
  const uint64_t* seeds;
  uint32_t round;
  const RowResult* rowres;
  GroupParams* gparams;     // [B]
  // children of node u: child[child_off[u] .. child_off[u+1]), in index order
  int child_off[kMaxTreeNodes + 1];
  int child[kMaxTreeNodes];
  int32_t* accept_len;
  int32_t* path;            // [B, Dmax] or null
  int Dmax;
  float* resid_mass;
  int32_t* status;
  CdfParams q;              // the bonus draw (unit sums, group_draw)
};

// ---- workspace layout ----------------------------------------------------------
struct WsLayout {
  size_t cnt_off, cnt_bytes;       // counters (cleared each call)
  size_t ctr_off;                  // the 8-byte counters, within the counters
  size_t part_off, rowres_off, gp_off, sub_off, bsum_off, dbg_off, total;
  // offsets (in ints) of the int counters
  size_t o_row_cnt, o_grp_cnt, o_pair, o_kcnt, o_dq, o_state;
  int64_t NR;
  int groups, nsub, nblk, cpg;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// spacing of the 8-byte counters (in 8-byte words): one 128-byte line each
constexpr int kCtrStride = 16;

// groups of rpg rows (nt target rows, K positions), V elements per row of
// esize bytes, nch chunks per row, cpg draw chunks per group; bsum: room for
// the one-row draws' block sums (one row per group).
inline WsLayout ws_layout(int groups, int rpg, int K, int V, int esize, int nch, int cpg,
                          bool bsum) {
  WsLayout L;
  L.groups = groups;
  L.NR = (int64_t)groups * rpg;
  L.nsub = (V + kUnitB - 1) / kUnitB;
  const int ups = units_per_stage(esize);
  const int upr = (V + kUnitA - 1) / kUnitA;
  L.nblk = ((upr + ups - 1) / ups) * kConsumerWarps;
  L.cpg = cpg;
  // int counters: row arrivals [NR], draw arrivals [groups], position
  // arrivals [groups * (K+1)], all-accepted events [groups], draw tickets
  // [groups * cpg]; then 8-byte words: sequence states [groups], the chunk
  // counter, round-cache outcomes, round-cache clearing, queue tail / head,
  // decided groups, bytes of target rows skipped
  L.o_row_cnt = 0;
  L.o_grp_cnt = L.o_row_cnt + (size_t)L.NR;
  L.o_pair = L.o_grp_cnt + (size_t)groups;
  L.o_kcnt = L.o_pair + (size_t)groups * (K + 1);
  L.o_dq = L.o_kcnt + (size_t)groups;
  const size_t nint = L.o_dq + (size_t)groups * cpg;
  L.cnt_off = 0;
  L.o_state = ((nint * sizeof(int) + 7) & ~(size_t)7) / 8;  // in 8-byte words
  // each 8-byte counter on its own 128-byte line: CTAs poll some of them
  // while others are incremented
  L.ctr_off = ((L.o_state + (size_t)groups) * 8 + 127) & ~(size_t)127;
  L.cnt_bytes = align256(L.ctr_off + 7 * kCtrStride * sizeof(unsigned long long));
  L.part_off = L.cnt_bytes;
  const size_t slots = nch > 1 ? (size_t)L.NR * nch : 1;
  L.rowres_off = L.part_off + align256(slots * sizeof(RowPartial));
  L.gp_off = L.rowres_off + align256((size_t)L.NR * sizeof(RowResult));
  L.sub_off = L.gp_off + align256((size_t)groups * sizeof(GroupParams));
  L.bsum_off = L.sub_off + align256((size_t)groups * L.nsub * sizeof(float));
  const size_t bsum_bytes = bsum ? (size_t)groups * L.nblk * sizeof(float2) : 0;
  L.dbg_off = L.bsum_off + align256(bsum_bytes);
  L.total = L.dbg_off + 256;  // bounds-check record of SSD_CHECKS builds
  return L;
}

// ---- launchers (ssd_stream_*.cu / ssd_cache.cu) ----------------------------------
template <int DT>
cudaError_t launch_stream_dt(const VerifyParams& p, int grid, cudaStream_t s);
cudaError_t launch_cache_clear(void* table, int64_t capacity, cudaStream_t s);
cudaError_t launch_cache_insert(void* table, int64_t capacity, const int32_t* row,
                                const int32_t* k, const int32_t* t, const int32_t* branch, int n,
                                const int32_t* guesses, int B, int Kq, int Fmax,
                                int32_t* status, cudaStream_t s);
cudaError_t launch_cache_lookup(const void* table, int64_t capacity, const int32_t* accept_len,
                                const int32_t* bonus, int B, int32_t* out_branch,
                                int32_t* all_hit, cudaStream_t s);
template <int DT>
cudaError_t launch_tree_dt(const TreeParams& tp, cudaStream_t s);
int stream_smem_bytes();
int num_sms();

}  // namespace ssd
