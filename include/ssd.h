/*
 * ssd.h -- C ABI of the GB300 (sm_103a) speculative-decoding sampling library.
 *
 * The library implements the data-parallel sampling step of speculative
 * decoding and of speculative speculative decoding (SSD / Saguaro) over
 * full-vocabulary logits that already sit in device memory:
 *   - the per-position accept test min(1, p(x)/q(x)) up to the first
 *     rejection and the bonus token drawn from normalize((p - q)^+);
 *   - the top-F bonus-token guesses per draft position;
 *   - Saguaro sampling (cached tokens' draft probability times C, then
 *     renormalised);
 *   - the outcome-cache build and lookup keyed by (row, k accepted, bonus t);
 *   - the geometric fan-out allocation of the cache budget (host helper).
 *
 * Sources, cited by page title and section:
 *   [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈"
 *   [SD-7.3]   "7.3 Speculative Decoding：投机采样加速"
 *   [SD-blog]  "推测解码：用一个“小模型”骗出 3 倍推理速度"
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless the comment says "host".
 *   - The caller owns all memory; the library never allocates.  Scratch
 *     space comes from a caller-provided workspace sized by the matching
 *     *_workspace_size() call.  The first bytes of the workspace (counters)
 *     are cleared on the stream at the start of every call, so a workspace
 *     needs no initialisation and may be reused by any entry point, but two
 *     calls that run concurrently must not share one.  Sizes depend on the
 *     current device's SM count (small batches split rows over more CTAs):
 *     query them with the device current that the call will run on.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  The library keeps no global state, so
 *     calls are thread-safe.
 *   - The return value reports argument errors (checked on the host before
 *     anything is enqueued) and launch errors.  Errors found on the device
 *     are OR-ed as SSD_DEV_* bits into *dev_status when dev_status is not
 *     NULL; the library never traps and every wait on the device is bounded.
 *   - Logit rows are contiguous over the vocabulary (V elements); successive
 *     rows are `row_stride` elements apart.  Any element-aligned pointer and
 *     stride is accepted; 16-byte aligned rows take the bulk-copy fast path.
 *   - Philox-4x32-10 uniforms: key = (seed lo32, seed hi32), counter =
 *     (c0, c1, stream, round), u = (out0 >> 8) * 2^-24 in [0, 1).
 *     Streams: 0 = accept test, 1 = bonus draw, 2 = draft / Saguaro sample.
 */
#ifndef SSD_H
#define SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1,   /* an argument is out of range or inconsistent */
  SSD_ERR_UNSUPPORTED = 2,   /* valid, but beyond the library's compiled limits (e.g. F > 15) */
  SSD_ERR_TABLE_FULL = 3,    /* host-detectable: cache capacity below 2 n */
  SSD_ERR_DUPLICATE_KEY = 4, /* reserved; duplicates are reported via dev_status */
  SSD_ERR_WORKSPACE = 5,     /* workspace NULL, misaligned or too small */
  SSD_ERR_CUDA = 6           /* a CUDA runtime call failed */
} ssd_status;

/* Bits OR-ed into *dev_status by device code. */
#define SSD_DEV_BAD_TOKEN 0x1      /* a draft token outside [0, V); treated as token 0 */
#define SSD_DEV_ZERO_RESIDUAL 0x2  /* residual mass underflowed; bonus drawn from p_k */
#define SSD_DEV_TIMEOUT 0x4        /* a bounded wait gave up; outputs are undefined */
#define SSD_DEV_TABLE_FULL 0x8     /* cache insert found no free slot */
#define SSD_DEV_DUPLICATE_KEY 0x10 /* cache insert met an existing key */
#define SSD_DEV_BAD_TEMPERATURE 0x20 /* a per-sequence temperature negative or not
                                        finite; that sequence is verified greedily */
#define SSD_DEV_BAD_FANOUT 0x40    /* a per-row fan-out outside [0, Fmax]; clamped */

typedef enum { SSD_BF16 = 0, SSD_F32 = 1 } ssd_dtype;

/* A batch of logit rows in device memory. */
typedef struct {
  const void* ptr;    /* device pointer to the first element of row 0 */
  int32_t dtype;      /* ssd_dtype */
  int32_t pad_;       /* must be 0 */
  int64_t row_stride; /* elements between the starts of consecutive rows, >= V */
} ssd_logits;

/* Compiled limits of the library. */
#define SSD_MAX_K 32       /* draft tokens per sequence */
#define SSD_MAX_F 15       /* bonus guesses per position */
#define SSD_MAX_V 16777215 /* vocabulary size (token ids and 24-bit uniforms stay exact) */

/* Static message for a status code. */
const char* ssd_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int ssd_version(void);

/* ---------------------------------------------------------------------------
 * ssd_verify -- rejection-sampling verification of K drafts per sequence.
 * [SD-7.3] §7.3.2 / §7.3.3; [SD-blog] §"三、接受概率为什么是对的";
 * [SSD-note] §"接受-拒绝机制", §"Saguaro 优化二：Saguaro 采样".
 *
 * For sequence b (0 <= b < B) with drafts x_0..x_{K-1}:
 *   p_i = softmax(z_target[b,i,:] / T),  i = 0..K   (position K: all accepted)
 *   q_j = softmax(z_draft[b,j,:] / T),   j = 0..Kq-1
 *   S_j = top-F_j of z_draft[b,j,:] (raw logit desc, ties to the lower index)
 *   q'_j(y) = q_j(y) * (C if y in S_j else 1) / (1 - (1-C) * q_j(S_j))
 *   accept x_i iff u_i < p_i(x_i) / q'_i(x_i),  u_i = U(seeds[b]; b, i, 0, round);
 *   k = the first rejected position, or K when every draft is accepted;
 *   w = (p_k - q'_k)^+ if k < K, else p_K;  Z = sum_y w(y);
 *   bonus t = smallest y with sum_{y'<=y} w(y') > u' * Z,
 *             u' = U(seeds[b]; b, k, 1, round).
 *   guesses[b,j,:] = top-(F_j + 1) of z_draft[b,j,:] minus x_j (j < K),
 *                    truncated to F_j, padded with -1 to Fmax.
 * C = 1 (or all F_j = 0) is plain speculative decoding, bit for bit.
 * T = 0 is the greedy limit T -> 0 (a serving setting the pages do not
 * treat): x_i is accepted iff it is the argmax of z_target[b,i,:] (ties to
 * the lower index), the bonus is the argmax of target row k, resid_mass is
 * 1, and guess_q is 1 for the draft argmax and 0 for other guesses; no
 * uniform is drawn.
 *
 * target      [B, K+1, V] logits: row (b, i) is row b*(K+1)+i.  Target rows
 *             past a known rejection of their sequence are not read: no
 *             output depends on p_i for i > k (the accept tests stop at the
 *             first rejection, [SD-7.3] §7.3.3); a row whose sequence is not
 *             yet decided when its turn comes is read (see
 *             ssd_verify_skipped_bytes).
 * draft       [B, Kq, V] logits, Kq in {K, K+1}: row (b, j) is row b*Kq+j.
 *             Every draft row is read (the guesses of every position).
 *             Verification reads draft rows 0..K-1; row K (when Kq = K+1)
 *             only feeds the guesses for the all-accepted outcome.
 * draft_tokens device [B, K] int32.
 * seeds       device [B] uint64 Philox keys.
 * fanout      HOST [Kq] int32 F_j (F_j in [0, SSD_MAX_F], F_j + 1 <= V),
 *             or NULL for all zero.  With Kq = K, F_K does not exist.
 * C           Saguaro factor in (0, 1].
 * accept_len  device [B] int32 out: k in [0, K].
 * bonus       device [B] int32 out: t in [0, V).
 * resid_mass  device [B] float out (or NULL): Z (1 - alpha_k when k < K;
 *             sum of p_K, i.e. ~1, when k = K).
 * guesses     device [B, Kq, Fmax] int32 out (or NULL).
 * guess_q     device [B, Kq, Fmax] float out (or NULL): q_j of each guess
 *             (plain draft probability), 0 for padding.
 * Fmax        >= max F_j when guesses is given.
 * workspace   device, 256-byte aligned, >= ssd_verify_workspace_size(B,K,Kq,V).
 * dev_status  device int32 (or NULL): SSD_DEV_* bits are OR-ed in.
 * T           temperature, finite and >= 0 (0: greedy).
 * ------------------------------------------------------------------------- */
size_t ssd_verify_workspace_size(int B, int K, int Kq, int V);
ssd_status ssd_verify(const ssd_logits* target, const ssd_logits* draft, int B, int K, int Kq,
                      int V, float T, const int32_t* draft_tokens, const uint64_t* seeds,
                      uint32_t round, const int32_t* fanout, float C, int32_t* accept_len,
                      int32_t* bonus, float* resid_mass, int32_t* guesses, float* guess_q,
                      int Fmax, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                      void* stream);

/* ---------------------------------------------------------------------------
 * ssd_verify_skipped_bytes -- the bytes of target rows that the last call of
 * ssd_verify, ssd_verify_ck, ssd_verify_ex or ssd_verify_round on `workspace`
 * did not read (rows past a rejection already known when their turn came).
 * A measurement aid: the logits streamed by that call are the target and
 * draft bytes minus this count.
 *
 * workspace   the call's workspace (256-byte aligned) and its size; B, K,
 *             Kq, V and dtype (ssd_dtype) those of the call.
 * out         device uint64 out, written in stream order after the call.
 * Errors: SSD_ERR_INVALID_ARG (bad sizes, null pointers), SSD_ERR_WORKSPACE
 * (smaller than ssd_verify_workspace_size).  Enqueues one 8-byte copy.
 * ------------------------------------------------------------------------- */
ssd_status ssd_verify_skipped_bytes(const void* workspace, size_t workspace_bytes, int B, int K,
                                    int Kq, int V, int dtype, uint64_t* out, void* stream);

/* ---------------------------------------------------------------------------
 * ssd_verify_ck -- ssd_verify with one Saguaro factor per draft position.
 * [SSD-note] §"关于逐位置 C 的思考": the pages use one global C and propose a
 * factor per position (positions whose fan-out covers more can bias less).
 *
 * As ssd_verify, with q'_j built from C_pos[j] instead of C:
 *   q'_j(y) = q_j(y) * (C_j if y in S_j else 1) / (1 - (1-C_j) * q_j(S_j)).
 * The drafts x_j must have been drawn from the same q'_j (for example by
 * ssd_saguaro_sample at position j with C = C_pos[j]).
 *
 * C_pos  HOST [K] float, each in (0, 1]; read before the call returns.
 * Every C_pos[j] equal to C gives the results of ssd_verify with C, bit for
 * bit.  Other arguments, errors and outputs: ssd_verify.
 * ------------------------------------------------------------------------- */
ssd_status ssd_verify_ck(const ssd_logits* target, const ssd_logits* draft, int B, int K,
                         int Kq, int V, float T, const int32_t* draft_tokens,
                         const uint64_t* seeds, uint32_t round, const int32_t* fanout,
                         const float* C_pos, int32_t* accept_len, int32_t* bonus,
                         float* resid_mass, int32_t* guesses, float* guess_q, int Fmax,
                         void* workspace, size_t workspace_bytes, int32_t* dev_status,
                         void* stream);

/* ---------------------------------------------------------------------------
 * ssd_verify_ex -- ssd_verify with a temperature per sequence and an
 * optional Saguaro factor per draft position (the pages use one T and one C;
 * a batch of requests with their own sampling settings needs both).
 *
 * As ssd_verify_ck, with sequence b verified at temperature T_rows[b]:
 * T_rows[b] > 0 as ssd_verify at that T; T_rows[b] = 0 greedy (see
 * ssd_verify).  A negative or non-finite T_rows[b] is verified greedily and
 * sets SSD_DEV_BAD_TEMPERATURE.  A call whose T_rows are all equal to T > 0
 * gives the results of ssd_verify_ck with T.
 *
 * T_rows  device [B] float.
 * C_pos   HOST [K] float in (0, 1], or NULL for C = 1 at every position.
 * Other arguments, errors and outputs: ssd_verify.
 * ------------------------------------------------------------------------- */
ssd_status ssd_verify_ex(const ssd_logits* target, const ssd_logits* draft, int B, int K,
                         int Kq, int V, const float* T_rows, const int32_t* draft_tokens,
                         const uint64_t* seeds, uint32_t round, const int32_t* fanout,
                         const float* C_pos, int32_t* accept_len, int32_t* bonus,
                         float* resid_mass, int32_t* guesses, float* guess_q, int Fmax,
                         void* workspace, size_t workspace_bytes, int32_t* dev_status,
                         void* stream);

/* ---------------------------------------------------------------------------
 * ssd_verify_round -- one SSD round in one launch: ssd_verify, the outcome
 * cache of the round's guesses (ssd_cache_build_guesses) and its lookup with
 * every sequence's outcome (ssd_cache_lookup).  [SSD-note] §"SSD 的核心思想":
 * the drafter prepares a continuation per predicted outcome (k, t) and the
 * round goes on at once when the real outcome was predicted; §"Saguaro 优化三":
 * the batch proceeds without waiting only if every sequence hits.
 *
 * Arguments and outputs of ssd_verify (guesses is required), plus:
 * table       device, 16-byte aligned, table_bytes >= ssd_cache_bytes(B*Kq*Fmax);
 *             its previous content is discarded (the launch clears it before
 *             inserting); afterwards it holds the round's guesses in the
 *             format of ssd_cache_build_guesses, so ssd_cache_lookup can read
 *             it.  Too small: SSD_ERR_TABLE_FULL.
 * out_branch  device [B] int32 out: (b*Kq + k)*Fmax + f of the guess that
 *             equals the outcome (k, t) = (accept_len[b], bonus[b]), or -1.
 * all_hit     device int32 out (or NULL): 1 if every sequence hit, else 0.
 * The results equal those of the three calls in sequence; outputs are
 * undefined after SSD_DEV_TIMEOUT.
 * ------------------------------------------------------------------------- */
ssd_status ssd_verify_round(const ssd_logits* target, const ssd_logits* draft, int B, int K,
                            int Kq, int V, float T, const int32_t* draft_tokens,
                            const uint64_t* seeds, uint32_t round, const int32_t* fanout, float C,
                            int32_t* accept_len, int32_t* bonus, float* resid_mass,
                            int32_t* guesses, float* guess_q, int Fmax, void* table,
                            size_t table_bytes, int32_t* out_branch, int32_t* all_hit,
                            void* workspace, size_t workspace_bytes, int32_t* dev_status,
                            void* stream);

/* ---------------------------------------------------------------------------
 * ssd_verify_noalloc -- ssd_verify without a caller workspace.  The pages have
 * no counterpart: this is a deployment convenience.
 *
 * For callers that cannot allocate device memory where they call the library
 * (a plugin of an inference runtime whose enqueue hook may not allocate, a
 * process whose device memory belongs to a pool allocator, a decode loop that
 * cannot pay for cudaMalloc and its implicit synchronisation).  The scratch
 * space is a SSD_NOALLOC_SCRATCH_BYTES array compiled into the library; every
 * GPU that loads the library holds it until the process exits.  Arguments and
 * results are those of ssd_verify.
 *   - Requests whose ssd_verify_workspace_size(B, K, Kq, V) exceeds
 *     SSD_NOALLOC_SCRATCH_BYTES return SSD_ERR_WORKSPACE (use ssd_verify with
 *     your own workspace); nothing is enqueued.  4 MiB covers, for example,
 *     B = 256 sequences with K = 8 at V = 151936.
 *   - The first call on a device looks up the array's address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture on the device.  The cache is
 *     keyed on the current context: after cudaDeviceReset the next call
 *     looks the address up again (make it, too, outside stream capture).
 *   - All calls on a device share the array; the parts that must start at
 *     zero are cleared at the start of each call.  Calls whose work overlaps
 *     on the GPU (different streams or host threads) race on the array and
 *     must be serialised by the caller.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library
 *     routine is called.
 * ------------------------------------------------------------------------- */
#define SSD_NOALLOC_SCRATCH_BYTES (4u << 20)
ssd_status ssd_verify_noalloc(const ssd_logits* target, const ssd_logits* draft, int B, int K,
                              int Kq, int V, float T, const int32_t* draft_tokens,
                              const uint64_t* seeds, uint32_t round, const int32_t* fanout,
                              float C, int32_t* accept_len, int32_t* bonus, float* resid_mass,
                              int32_t* guesses, float* guess_q, int Fmax, int32_t* dev_status,
                              void* stream);

/* ---------------------------------------------------------------------------
 * ssd_topf_bonus -- bonus-token guesses alone.  [SSD-note] §"怎么猜奖励 token":
 * the top-F_j draft logits of position j, excluding the token already sampled
 * there.
 *
 * draft        [B, Kq, V] logits.
 * draft_tokens device [B, K] int32 (or NULL = no exclusion); positions
 *              j < K exclude draft_tokens[b, j].
 * fanout       HOST [Kq] int32.
 * guesses      device [B, Kq, Fmax] int32 out, -1 padded.
 * guess_q      device [B, Kq, Fmax] float out (or NULL): q_j(guess) at T.
 * ------------------------------------------------------------------------- */
size_t ssd_topf_workspace_size(int B, int Kq, int V);
ssd_status ssd_topf_bonus(const ssd_logits* draft, int B, int Kq, int V, float T,
                          const int32_t* draft_tokens, int K, const int32_t* fanout, int Fmax,
                          int32_t* guesses, float* guess_q, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------
 * ssd_saguaro_sample -- one continuation step of the SSD cache build: every
 * branch row draws its next draft token from the Saguaro distribution.
 * [SSD-note] §"Saguaro 优化二：Saguaro 采样" and §"实现细节：缓存怎么建"; the
 * fan-out of a branch row is that of the outcome position it continues
 * (§"最优扇出度分配"), so it is given per row.
 *
 * For branch row r (0 <= r < R) with F = F_row[r]:
 *   S = top-F of z[r,:];  q' = Saguaro(softmax(z[r,:]/T), S, C);
 *   x = smallest y with sum_{y'<=y} q'(y') > u * sum(q'),
 *       u = U(seeds[r]; r, j, 2, round);
 *   guesses = top-(F+1) of z[r,:] minus x, truncated to F.
 *
 * draft       [R, V] logits.
 * T           temperature, finite and > 0.
 * C           Saguaro factor in (0, 1] (the factor of position j when the
 *             caller uses one per position).
 * F_row       device [R] int32 cached-set size / guesses per row, each in
 *             [0, Fmax] (a value outside is clamped and sets
 *             SSD_DEV_BAD_FANOUT), or NULL: F = Fmax for every row.
 * Fmax        0..SSD_MAX_F, Fmax + 1 <= V: the largest F and the column
 *             count of out_guess.
 * seeds       device [R] uint64.   j: continuation position (counter word).
 * out_token   device [R] int32 out.
 * out_qprime  device [R] float out (or NULL): q'(x).
 * out_guess   device [R, Fmax] int32 out (or NULL), -1 padded.
 * ------------------------------------------------------------------------- */
size_t ssd_saguaro_workspace_size(int R, int V);
ssd_status ssd_saguaro_sample(const ssd_logits* draft, int R, int V, float T, float C,
                              const int32_t* F_row, int Fmax, const uint64_t* seeds, int j,
                              uint32_t round, int32_t* out_token, float* out_qprime,
                              int32_t* out_guess, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------
 * ssd_tree_verify -- verification of tree-shaped drafts.  [SD-7.3] §7.3.9
 * item 3 (树形草稿: several candidate continuations per position instead of
 * one chain); the pages give no algorithm, and the per-token rule of §7.3.3
 * is applied to each candidate in turn (multi-candidate rejection sampling):
 *
 * The tree has N nodes, the same for the whole batch: node 0 is the last
 * verified position, node u >= 1 has parent parent[u] < u and holds draft
 * token tokens[b, u], drawn from the draft distribution q_{parent(u)} of its
 * parent.  Target row u of tree b is p_u, the target distribution after node
 * u's path; draft row u is q_u.  For tree b:
 *   u = 0, r = p_0 = softmax(z_target[b,0,:] / T);
 *   for each child v of u in increasing index order:
 *     accept x_v iff U(seeds[b]; b, v-1, 0, round) < r(x_v) / q_u(x_v):
 *       then u = v, r = p_v, and continue with v's children;
 *     else r = (r - q_u)^+ / sum (r - q_u)^+;
 *   when no child of u is accepted (or u is a leaf): bonus t = smallest y
 *   with sum_{y'<=y} r(y') > U(seeds[b]; b, u, 1, round) * sum(r).
 * A chain (parent[u] = u - 1) gives ssd_verify's results with C = 1, F = 0
 * (accept_len, bonus; drafts drawn with counter (b, v-1, 2, round)).
 *
 * target, draft  [B, N, V] logits, same dtype: row (b, u) is row b*N + u.
 * parent      HOST [N] int32: parent[0] = -1, 0 <= parent[u] < u.
 * tokens      device [B, N] int32 (entry 0 of a tree is ignored).
 * accept_len  device [B] int32 out: depth of the last accepted node.
 * path        device [B, Dmax] int32 out (or NULL): the accepted nodes, -1
 *             padded; Dmax >= the tree's depth.
 * bonus       device [B] int32 out.
 * resid_mass  device [B] float out (or NULL): sum (r - q_u)^+ of the last
 *             rejection at the final node, 1 when it rejected nothing.
 * T           temperature, finite and > 0.   N <= 256.
 * workspace   >= ssd_tree_workspace_size(B, N, V), 256-byte aligned.
 * Two launches on `stream`: the streaming pass normalises every row, then
 * one thread-block cluster per tree walks it: its CTAs share the tree's row
 * passes; 8 CTAs, halved while B times the cluster size exceeds the SM
 * count (one CTA per tree when B does).
 * ------------------------------------------------------------------------- */
size_t ssd_tree_workspace_size(int B, int N, int V);
ssd_status ssd_tree_verify(const ssd_logits* target, const ssd_logits* draft, int B, int N, int V,
                           float T, const int32_t* parent, const int32_t* tokens,
                           const uint64_t* seeds, uint32_t round, int32_t* accept_len,
                           int32_t* path, int Dmax, int32_t* bonus, float* resid_mass,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream);

/* ---------------------------------------------------------------------------
 * Outcome cache.  [SSD-note] §"SSD 的核心思想": the verification outcome is the
 * pair (k accepted, bonus t); the drafter keeps a continuation per predicted
 * outcome.  Keys are (row, k, t), values are branch ids.
 *
 * The table is an open-addressed hash table of 16-byte slots (64-bit packed
 * key, 32-bit value) with a power-of-two capacity >= 2 n; probing is linear
 * and bounded by the capacity, so a full table can never loop.
 *
 * ssd_cache_bytes(n)  bytes of a table for n keys.
 * ssd_cache_build     clears the table and inserts n keys row[i], k[i], t[i]
 *                     -> branch[i] (all device [n] int32).  Duplicate keys set
 *                     SSD_DEV_DUPLICATE_KEY (the first value is kept).
 * ssd_cache_build_guesses  clears and inserts every non-negative guess
 *                     g = guesses[b, k, f] of a [B, Kq, Fmax] table as key
 *                     (b, k, g) -> branch (b*Kq + k)*Fmax + f.
 * ssd_cache_lookup    out_branch[b] = value of key (b, accept_len[b], bonus[b])
 *                     or -1; *all_hit = 1 if every row hit, else 0 (device
 *                     int32).  [SSD-note] §"Saguaro 优化三": a batch proceeds
 *                     without waiting only if every sequence hits.
 * ------------------------------------------------------------------------- */
size_t ssd_cache_bytes(int n_keys);
ssd_status ssd_cache_build(void* table, size_t table_bytes, const int32_t* row, const int32_t* k,
                           const int32_t* t, const int32_t* branch, int n, int32_t* dev_status,
                           void* stream);
ssd_status ssd_cache_build_guesses(void* table, size_t table_bytes, const int32_t* guesses, int B,
                                   int Kq, int Fmax, int32_t* dev_status, void* stream);
ssd_status ssd_cache_lookup(const void* table, size_t table_bytes, const int32_t* accept_len,
                            const int32_t* bonus, int B, int32_t* out_branch, int32_t* all_hit,
                            void* stream);

/* ---------------------------------------------------------------------------
 * ssd_fanout -- geometric fan-out (host only, no device work).
 * [SSD-note] §"最优扇出度分配": with acceptance P(k) ~ a^k and a per-position
 * miss rate falling as F_k^-r, the Lagrange optimum under sum F_k = budget is
 * F_k ~ a^(k/(1+r)).  Real-valued shares budget * w_k / sum(w) are rounded
 * down, then the remaining units go to the largest fractional parts (ties to
 * the lower k).
 * F_out HOST [K+1] int32 out.  K >= 0, budget >= 0, a > 0, r >= 0.
 * ------------------------------------------------------------------------- */
ssd_status ssd_fanout(int K, int budget, double a, double r, int32_t* F_out);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H */
