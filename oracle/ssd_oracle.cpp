// ssd_oracle.cpp -- plain, slow, fp64 CPU oracle of the speculative-decoding
// verify path (accept/reject, residual bonus, top-F bonus guesses, Saguaro
// sampling, outcome cache, geometric fan-out).
//
// TEST INFRASTRUCTURE ONLY.  This file is the correctness reference and the
// timed CPU baseline.  It shares no code, header, table or helper with the
// CUDA library; only the tests, the smoke check and the benchmark's CPU
// baseline leg may load it.
//
// Every function follows one passage of the source pages, cited by page
// title and section:
//   [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈"
//   [SD-7.3]   "7.3 Speculative Decoding：投机采样加速"
//   [SD-blog]  "推测解码：用一个“小模型”骗出 3 倍推理速度"
// Where the pages leave a step open (their formulas were lost), the reading
// taken is stated next to the code.
//
// Pins (tests/test_oracle_*.py): exact-enumeration losslessness, closed-form
// acceptance law, chi-square bonus law, top-F vs a library sort, Saguaro
// closed forms, inverse CDF vs a library search, Philox round structure vs
// numpy's Philox4x64, Lagrange optimum of the fan-out vs numerical
// minimisation.  "parity unpinned": the fan-out *objective* itself (its
// formula is missing from the page; only its stated shape is pinned).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <thread>
#include <tuple>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Philox-4xW-10 counter-based generator (Salmon, Moraes, Dror, Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).  One round maps
// counter (c0,c1,c2,c3) and key (k0,k1) to
//   (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
// the key is bumped by the Weyl constants (W0, W1) between rounds.
// ---------------------------------------------------------------------------
template <typename W> struct PhiloxConst;
template <> struct PhiloxConst<uint32_t> {
  static constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  static constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
};
template <> struct PhiloxConst<uint64_t> {
  static constexpr uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  static constexpr uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
};

inline void mulhilo(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
  uint64_t p = (uint64_t)a * (uint64_t)b;
  hi = (uint32_t)(p >> 32);
  lo = (uint32_t)p;
}
inline void mulhilo(uint64_t a, uint64_t b, uint64_t& hi, uint64_t& lo) {
  unsigned __int128 p = (unsigned __int128)a * (unsigned __int128)b;
  hi = (uint64_t)(p >> 64);
  lo = (uint64_t)p;
}

template <typename W>
void philox4_10(const W ctr_in[4], const W key_in[2], W out[4]) {
  W c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  W k[2] = {key_in[0], key_in[1]};
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k[0] += PhiloxConst<W>::W0;
      k[1] += PhiloxConst<W>::W1;
    }
    W hi0, lo0, hi1, lo1;
    mulhilo(PhiloxConst<W>::M0, c[0], hi0, lo0);
    mulhilo(PhiloxConst<W>::M1, c[2], hi1, lo1);
    W n0 = hi1 ^ c[1] ^ k[0];
    W n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
  for (int i = 0; i < 4; ++i) out[i] = c[i];
}

// Uniform in [0,1) with 24 random bits: exact in fp32 and fp64, so the CUDA
// path and this oracle hold the same value.  key = (seed lo, seed hi),
// counter = (c0, c1, stream, round).  Streams: 0 accept test, 1 bonus draw,
// 2 draft / Saguaro sample.
double uniform24(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t stream, uint32_t round) {
  uint32_t ctr[4] = {c0, c1, stream, round};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4_10<uint32_t>(ctr, key, out);
  return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

// ---------------------------------------------------------------------------
// Logit access: bf16 (dtype 0) or fp32 (dtype 1), widened exactly to fp64.
// ---------------------------------------------------------------------------
double logit_at(const void* base, int dtype, int64_t off) {
  if (dtype == 0) {
    uint16_t h = ((const uint16_t*)base)[off];
    uint32_t u = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
  }
  return (double)((const float*)base)[off];
}

std::vector<double> load_row(const void* base, int dtype, int64_t row_off, int V) {
  std::vector<double> z(V);
  for (int y = 0; y < V; ++y) z[y] = logit_at(base, dtype, row_off + y);
  return z;
}

// Temperature softmax p = softmax(z / T) with max subtraction.
// [SD-7.3] §7.3.2 (target and draft distributions compared per position);
// T divides the logits before the softmax (reading: the pages name high
// temperature but give no formula).
std::vector<double> softmax(const std::vector<double>& z, double T) {
  double m = -INFINITY;
  for (double v : z) m = std::max(m, v);
  std::vector<double> p(z.size());
  double s = 0.0;
  for (size_t y = 0; y < z.size(); ++y) {
    p[y] = std::exp((z[y] - m) / T);
    s += p[y];
  }
  for (auto& v : p) v /= s;
  return p;
}

// Indices of the n largest raw logits, ordered by (logit desc, index asc).
// [SSD-note] §"怎么猜奖励 token": the bonus guesses are the top logits of the
// drafter's full-vocabulary distribution.
std::vector<int> top_n(const std::vector<double>& z, int n) {
  std::vector<int> idx(z.size());
  for (size_t y = 0; y < z.size(); ++y) idx[y] = (int)y;
  n = std::min<int>(n, (int)z.size());
  auto before = [&](int a, int b) { return z[a] > z[b] || (z[a] == z[b] && a < b); };
  std::partial_sort(idx.begin(), idx.begin() + n, idx.end(), before);
  idx.resize(n);
  return idx;
}

// Saguaro draft distribution: the probability of every cached token (set S)
// is multiplied by C, all others are left unchanged, then the result is
// renormalised.  [SSD-note] §"Saguaro 优化二：Saguaro 采样" / "解法：操纵草稿分布".
std::vector<double> saguaro(const std::vector<double>& q, const std::vector<int>& S, double C) {
  std::vector<double> qp(q);
  if (C == 1.0) return qp;  // plain speculative decoding
  for (int y : S) qp[y] = C * q[y];
  double total = 0.0;
  for (double v : qp) total += v;
  for (auto& v : qp) v /= total;
  return qp;
}

// Accept probability min(1, p(x)/q(x)).  [SD-7.3] §7.3.3;
// [SD-blog] §"三、接受概率为什么是对的".
double accept_prob(double px, double qx) {
  if (qx <= 0.0) return 1.0;
  return std::min(1.0, px / qx);
}

// Residual w = (p - q)^+, returns Z = sum w.  [SD-7.3] §7.3.3;
// [SSD-note] §"接受-拒绝机制".
double residual(const std::vector<double>& p, const std::vector<double>& q, std::vector<double>& w) {
  w.assign(p.size(), 0.0);
  double Z = 0.0;
  for (size_t y = 0; y < p.size(); ++y) {
    w[y] = std::max(0.0, p[y] - q[y]);
    Z += w[y];
  }
  return Z;
}

// Inverse CDF in vocabulary order: the smallest y with cumsum_y(w) > u*Z
// (strict).  If rounding leaves none, the largest y with w(y) > 0.
// margin = min(cumsum_t - uZ, uZ - cumsum_{t-1}) / Z (near-tie measure).
int inverse_cdf(const std::vector<double>& w, double Z, double u, double* margin) {
  const double thr = u * Z;
  double cum = 0.0;
  for (size_t y = 0; y < w.size(); ++y) {
    double prev = cum;
    cum += w[y];
    if (cum > thr) {
      if (margin) *margin = std::min(cum - thr, thr - prev) / Z;
      return (int)y;
    }
  }
  for (int y = (int)w.size() - 1; y >= 0; --y) {
    if (w[y] > 0.0) {
      if (margin) *margin = 0.0;
      return y;
    }
  }
  if (margin) *margin = 0.0;
  return (int)w.size() - 1;
}

// Bonus guesses for position j: the top F_j + 1 draft logits, minus the token
// already sampled at j (if any), truncated to F_j.  [SSD-note] §"怎么猜奖励 token".
std::vector<int> guesses_from(const std::vector<int>& topF1, int F, int exclude) {
  std::vector<int> g;
  for (int y : topF1) {
    if (y == exclude) continue;
    if ((int)g.size() == F) break;
    g.push_back(y);
  }
  return g;
}

template <typename Fn>
void parallel_rows(int n, int nthreads, Fn fn) {
  if (nthreads <= 1 || n <= 1) {
    for (int r = 0; r < n; ++r) fn(r);
    return;
  }
  nthreads = std::min(nthreads, n);
  std::vector<std::thread> th;
  for (int t = 0; t < nthreads; ++t)
    th.emplace_back([&, t] {
      for (int r = t; r < n; r += nthreads) fn(r);
    });
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

// ---- Philox ----------------------------------------------------------------
void orc_philox4x32(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4_10<uint32_t>(ctr, key, out);
}
void orc_philox4x64(const uint64_t* ctr, const uint64_t* key, uint64_t* out) {
  philox4_10<uint64_t>(ctr, key, out);
}
double orc_uniform(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t stream, uint32_t round) {
  return uniform24(seed, c0, c1, stream, round);
}
void orc_uniform_batch(uint64_t seed, uint32_t c1, uint32_t stream, uint32_t round, int n,
                       double* out) {
  for (int i = 0; i < n; ++i) out[i] = uniform24(seed, (uint32_t)i, c1, stream, round);
}

// ---- single steps (exposed for the enumeration / closed-form pins) ---------
void orc_softmax(const double* z, int V, double T, double* p) {
  std::vector<double> zz(z, z + V);
  auto pp = softmax(zz, T);
  std::copy(pp.begin(), pp.end(), p);
}
void orc_top_n(const double* z, int V, int n, int32_t* idx) {
  std::vector<double> zz(z, z + V);
  auto t = top_n(zz, n);
  for (size_t i = 0; i < t.size(); ++i) idx[i] = t[i];
}
// q' for a draft row: S = top-F of the raw logits.
void orc_saguaro_dist(const double* z, int V, double T, int F, double C, double* qp) {
  std::vector<double> zz(z, z + V);
  auto q = softmax(zz, T);
  auto S = top_n(zz, F);
  auto r = saguaro(q, S, C);
  std::copy(r.begin(), r.end(), qp);
}
double orc_accept_prob(double px, double qx) { return accept_prob(px, qx); }
double orc_residual(const double* p, const double* q, int V, double* w) {
  std::vector<double> pp(p, p + V), qq(q, q + V), ww;
  double Z = residual(pp, qq, ww);
  std::copy(ww.begin(), ww.end(), w);
  return Z;
}
int orc_inverse_cdf(const double* w, int V, double Z, double u, double* margin) {
  std::vector<double> ww(w, w + V);
  return inverse_cdf(ww, Z, u, margin);
}

// ---- a1..a5: batched verify --------------------------------------------------
// target: [B, K+1, V] rows at (b*(K+1)+i)*t_stride; draft: [B, Kq, V] rows at
// (b*Kq+j)*d_stride.  F: [Kq] fan-out (F[K] used only when Kq == K+1).
// For sequence b:
//   p_i = softmax(z_p[i]/T), q_j = softmax(z_q[j]/T)
//   S_j = top-F_j of z_q[j];  q'_j = Saguaro(q_j, S_j, C_j)
//   (C: one Saguaro factor per draft position j = 0..K-1 -- a single C for
//   every position is the pages' setting, a factor per position the
//   extension [SSD-note] §"关于逐位置 C 的思考" proposes)
//   i = 0..K-1: u = U(seed_b; b, i, 0, round); accept iff u < p_i(x_i)/q'_i(x_i),
//               else k = i and stop ([SD-7.3] §7.3.2 step 4: later drafts dropped);
//               all accepted -> k = K
//   k < K: w = (p_k - q'_k)^+;  k = K: w = p_K  ([SD-7.3] §7.3.2: gamma+1 tokens
//               from one target forward when every draft is accepted)
//   t = inverse CDF of w at u' = U(seed_b; b, k, 1, round)
//   guesses_j = top-(F_j+1) of z_q[j] minus x_j (j < K), truncated to F_j.
// Reading: verification uses q', the distribution the drafts were drawn from
// ([SSD-note] §"解法：操纵草稿分布": lowering q on cached tokens raises (p-q)^+).
// row_ids (or NULL = 0..B-1) give each row's Philox counter word 0, so a
// sample of rows of a larger batch can be checked one by one.
//
// T_rows (or NULL: T for every row) gives each sequence its own temperature.
// T = 0 is the greedy limit T -> 0 (a common serving setting; the pages do
// not treat it): p_i and q_j become one-hot at the argmax of their logits
// (ties to the lower index, the top-n order), so
//   x_i is accepted iff x_i = argmax z_p[i] (p_i(x_i) / q'_i(x_i) is 1 for a
//   greedy draft on the target's argmax and 0 otherwise; Saguaro's factor
//   leaves a one-hot q unchanged),
//   the bonus is argmax z_p[k] (the residual of a one-hot p_k against a
//   one-hot q'_k at another token is p_k itself; all accepted: p_K),
//   resid_mass = 1, both margins = +inf (no random decision), and guess_q is
//   the limit of q_j: 1 for the draft argmax, 0 for every other guess.
// Returns 0, or 1 if a draft token lies outside [0, V).
int orc_verify(const void* target, const void* draft, int dtype, int64_t t_stride,
               int64_t d_stride, int B, int K, int Kq, int V, double T,
               const int32_t* tokens, const uint64_t* seeds, uint32_t round,
               const int32_t* F, const double* C, int Fmax, int32_t* accept_len, int32_t* bonus,
               double* resid_mass, int32_t* guesses, double* guess_q, double* margin_accept,
               double* margin_cdf, int nthreads, const int32_t* row_ids, const double* T_rows) {
  for (int i = 0; i < B * K; ++i)
    if (tokens[i] < 0 || tokens[i] >= V) return 1;
  parallel_rows(B, nthreads, [&](int b) {
    const double Tb = T_rows ? T_rows[b] : T;
    std::vector<std::vector<double>> zq(Kq), q(Kq);
    std::vector<std::vector<int>> top1(Kq);
    for (int j = 0; j < Kq; ++j) {
      zq[j] = load_row(draft, dtype, ((int64_t)b * Kq + j) * d_stride, V);
      if (Tb > 0.0) q[j] = softmax(zq[j], Tb);
      top1[j] = top_n(zq[j], F[j] + 1);
    }
    const int32_t* x = tokens + (int64_t)b * K;
    if (Tb == 0.0) {
      int k = K;
      for (int i = 0; i < K; ++i) {
        auto zp = load_row(target, dtype, ((int64_t)b * (K + 1) + i) * t_stride, V);
        if (x[i] != top_n(zp, 1)[0]) {
          k = i;
          break;
        }
      }
      auto zk = load_row(target, dtype, ((int64_t)b * (K + 1) + k) * t_stride, V);
      accept_len[b] = k;
      bonus[b] = top_n(zk, 1)[0];
      if (resid_mass) resid_mass[b] = 1.0;
      if (margin_accept) margin_accept[b] = INFINITY;
      if (margin_cdf) margin_cdf[b] = INFINITY;
      if (guesses) {
        for (int j = 0; j < Kq; ++j) {
          int excl = j < K ? x[j] : -1;
          auto g = guesses_from(top1[j], F[j], excl);
          const int amax = top_n(zq[j], 1)[0];
          for (int f = 0; f < Fmax; ++f) {
            int64_t o = ((int64_t)b * Kq + j) * Fmax + f;
            guesses[o] = f < (int)g.size() ? g[f] : -1;
            if (guess_q) guess_q[o] = (f < (int)g.size() && g[f] == amax) ? 1.0 : 0.0;
          }
        }
      }
      return;
    }
    const uint32_t rid = row_ids ? (uint32_t)row_ids[b] : (uint32_t)b;  // Philox counter word 0
    int k = K;
    double mA = INFINITY;
    std::vector<double> p_k;
    std::vector<double> qp_k;
    for (int i = 0; i < K; ++i) {
      auto zp = load_row(target, dtype, ((int64_t)b * (K + 1) + i) * t_stride, V);
      auto p = softmax(zp, Tb);
      std::vector<int> S(top1[i].begin(), top1[i].begin() + std::min<int>(F[i], top1[i].size()));
      auto qp = saguaro(q[i], S, C[i]);
      double r = p[x[i]] / qp[x[i]];
      double u = uniform24(seeds[b], rid, (uint32_t)i, 0u, round);
      mA = std::min(mA, std::fabs(u - r));
      if (!(u < r)) {
        k = i;
        p_k = std::move(p);
        qp_k = std::move(qp);
        break;
      }
    }
    std::vector<double> w;
    double Z;
    if (k < K) {
      Z = residual(p_k, qp_k, w);
    } else {
      auto zp = load_row(target, dtype, ((int64_t)b * (K + 1) + K) * t_stride, V);
      w = softmax(zp, Tb);
      Z = 0.0;
      for (double v : w) Z += v;
    }
    double mC = 0.0;
    double u2 = uniform24(seeds[b], rid, (uint32_t)k, 1u, round);
    int t;
    if (Z > 1e-30) {
      t = inverse_cdf(w, Z, u2, &mC);
    } else {
      // degenerate residual (cannot happen in exact arithmetic): draw from p_k
      auto zp = load_row(target, dtype, ((int64_t)b * (K + 1) + k) * t_stride, V);
      auto p = softmax(zp, Tb);
      double Zp = 0.0;
      for (double v : p) Zp += v;
      t = inverse_cdf(p, Zp, u2, &mC);
    }
    accept_len[b] = k;
    bonus[b] = t;
    if (resid_mass) resid_mass[b] = Z;
    if (margin_accept) margin_accept[b] = mA;
    if (margin_cdf) margin_cdf[b] = mC;
    if (guesses) {
      for (int j = 0; j < Kq; ++j) {
        int excl = j < K ? x[j] : -1;
        auto g = guesses_from(top1[j], F[j], excl);
        for (int f = 0; f < Fmax; ++f) {
          int64_t o = ((int64_t)b * Kq + j) * Fmax + f;
          guesses[o] = f < (int)g.size() ? g[f] : -1;
          if (guess_q) guess_q[o] = f < (int)g.size() ? q[j][g[f]] : 0.0;
        }
      }
    }
  });
  return 0;
}

// ---- a2 alone: bonus guesses per draft position ----------------------------
int orc_topf_bonus(const void* draft, int dtype, int64_t d_stride, int B, int Kq, int V,
                   double T, const int32_t* tokens, int K, const int32_t* F, int Fmax,
                   int32_t* guesses, double* guess_q, int nthreads) {
  parallel_rows(B, nthreads, [&](int b) {
    for (int j = 0; j < Kq; ++j) {
      auto z = load_row(draft, dtype, ((int64_t)b * Kq + j) * d_stride, V);
      auto q = softmax(z, T);
      auto top1 = top_n(z, F[j] + 1);
      int excl = (tokens && j < K) ? tokens[(int64_t)b * K + j] : -1;
      auto g = guesses_from(top1, F[j], excl);
      for (int f = 0; f < Fmax; ++f) {
        int64_t o = ((int64_t)b * Kq + j) * Fmax + f;
        guesses[o] = f < (int)g.size() ? g[f] : -1;
        if (guess_q) guess_q[o] = f < (int)g.size() ? q[g[f]] : 0.0;
      }
    }
  });
  return 0;
}

// ---- a6: Saguaro continuation sampling -------------------------------------
// For each branch row r: S = top-F_r of the row's draft logits; x ~ q' by
// inverse CDF at u = U(seed_r; r, j, 2, round); guesses = top-(F_r+1) minus x,
// truncated to F_r.  [SSD-note] §"Saguaro 优化二" and §"实现细节：缓存怎么建"
// (all branches' continuations are drafted as one batch).  A branch row's
// fan-out is that of the outcome position it continues (§"最优扇出度分配"),
// so F_rows (or NULL: F for every row) gives one per row; out_guess has F
// columns (F >= every F_r), padded with -1.
int orc_saguaro_sample(const void* draft, int dtype, int64_t stride, int R, int V, double T,
                       double C, int F, const int32_t* F_rows, const uint64_t* seeds, int j,
                       uint32_t round, int32_t* out_token, double* out_qprime, int32_t* out_guess,
                       double* margin_cdf, int nthreads, const int32_t* row_ids) {
  parallel_rows(R, nthreads, [&](int r) {
    const int Fr = F_rows ? F_rows[r] : F;
    auto z = load_row(draft, dtype, (int64_t)r * stride, V);
    auto q = softmax(z, T);
    auto top1 = top_n(z, Fr + 1);
    std::vector<int> S(top1.begin(), top1.begin() + std::min<int>(Fr, top1.size()));
    auto qp = saguaro(q, S, C);
    double Z = 0.0;
    for (double v : qp) Z += v;
    const uint32_t rid = row_ids ? (uint32_t)row_ids[r] : (uint32_t)r;
    double u = uniform24(seeds[r], rid, (uint32_t)j, 2u, round);
    double m = 0.0;
    int x = inverse_cdf(qp, Z, u, &m);
    out_token[r] = x;
    if (out_qprime) out_qprime[r] = qp[x];
    if (margin_cdf) margin_cdf[r] = m;
    if (out_guess) {
      auto g = guesses_from(top1, Fr, x);
      for (int f = 0; f < F; ++f) out_guess[(int64_t)r * F + f] = f < (int)g.size() ? g[f] : -1;
    }
  });
  return 0;
}

// ---- tree drafts ------------------------------------------------------------
// [SD-7.3] §7.3.9 item 3 names tree-shaped drafts (树形草稿: several candidate
// continuations per position instead of one chain) as the next step.  The
// pages give no algorithm; the reading taken is multi-candidate rejection
// sampling with recursive residuals, the plain generalisation of the
// per-token rule of §7.3.3 to several candidates:
//   * a tree of N nodes shared by the batch: parent[0] = -1 (node 0 is the
//     last verified position), 0 <= parent[u] < u; node u >= 1 holds draft
//     token x_u, drawn from q_{parent(u)}, the draft distribution at its
//     parent; the children of a node are tried in increasing index order;
//   * target row u is p_u (the target distribution after node u's path),
//     draft row u is q_u;
//   * at node u with current residual r (r = p_u on arrival), child v is
//     accepted with probability min(1, r(x_v) / q_u(x_v)) (uniform
//     U(seed_b; b, v-1, 0, round)); accepted: move to v with r = p_v;
//     rejected: r = (r - q_u)^+ / sum (r - q_u)^+ and try the next child;
//   * no child accepted (or u is a leaf): the bonus t ~ r by inverse CDF at
//     U(seed_b; b, u, 1, round).
// A chain (every node has one child) is the linear verification with C = 1,
// uniform for uniform.  Outputs: accept_len = depth of the final node, path
// = the accepted nodes (-1 padded to Dmax), bonus, resid_mass = the mass of
// the last residual step (the sum of p_u, about 1, when the final node
// rejected nothing).
int orc_tree_verify(const void* target, const void* draft, int dtype, int64_t t_stride,
                    int64_t d_stride, int B, int N, int V, double T, const int32_t* parent,
                    const int32_t* tokens, const uint64_t* seeds, uint32_t round,
                    int32_t* accept_len, int32_t* path, int Dmax, int32_t* bonus,
                    double* resid_mass, double* margin_accept, double* margin_cdf,
                    int nthreads) {
  for (int u = 1; u < N; ++u)
    if (parent[u] < 0 || parent[u] >= u) return 3;
  for (int64_t i = 0; i < (int64_t)B * N; ++i)
    if (i % N != 0 && (tokens[i] < 0 || tokens[i] >= V)) return 1;
  parallel_rows(B, nthreads, [&](int b) {
    const int32_t* x = tokens + (int64_t)b * N;
    int u = 0, depth = 0;
    double mA = INFINITY;
    std::vector<double> r = softmax(load_row(target, dtype, ((int64_t)b * N) * t_stride, V), T);
    double Zlast = -1.0;
    for (int d = 0; d < Dmax; ++d) path[(int64_t)b * Dmax + d] = -1;
    while (true) {
      std::vector<double> q;
      bool moved = false;
      Zlast = -1.0;  // no rejection at this node yet
      for (int v = u + 1; v < N && !moved; ++v) {
        if (parent[v] != u) continue;
        if (q.empty())
          q = softmax(load_row(draft, dtype, ((int64_t)b * N + u) * d_stride, V), T);
        const double ratio = q[x[v]] > 0.0 ? r[x[v]] / q[x[v]] : INFINITY;
        const double uv = uniform24(seeds[b], (uint32_t)b, (uint32_t)(v - 1), 0u, round);
        mA = std::min(mA, std::fabs(uv - ratio));
        if (uv < ratio) {
          u = v;
          if (depth < Dmax) path[(int64_t)b * Dmax + depth] = v;
          ++depth;
          r = softmax(load_row(target, dtype, ((int64_t)b * N + v) * t_stride, V), T);
          moved = true;
        } else {
          std::vector<double> w;
          const double Z = residual(r, q, w);
          if (Z > 1e-300) {
            for (auto& e : w) e /= Z;
            r = std::move(w);
          }
          Zlast = Z;
        }
      }
      if (!moved) break;
    }
    double total = 0.0;
    for (double e : r) total += e;
    double mC = 0.0;
    const double ub = uniform24(seeds[b], (uint32_t)b, (uint32_t)u, 1u, round);
    bonus[b] = inverse_cdf(r, total, ub, &mC);
    accept_len[b] = depth;
    if (resid_mass) resid_mass[b] = Zlast < 0.0 ? total : Zlast;
    if (margin_accept) margin_accept[b] = mA;
    if (margin_cdf) margin_cdf[b] = mC;
  });
  return 0;
}

// Draft tokens of a tree: x_v ~ q_{parent(v)} by inverse CDF at
// U(seed_b; b, v-1, 2, round) -- for a chain, the same draws as the linear
// drafts at positions j = v-1.
int orc_tree_draft(const void* draft, int dtype, int64_t d_stride, int B, int N, int V, double T,
                   const int32_t* parent, const uint64_t* seeds, uint32_t round, int32_t* tokens,
                   int nthreads) {
  for (int u = 1; u < N; ++u)
    if (parent[u] < 0 || parent[u] >= u) return 3;
  parallel_rows(B, nthreads, [&](int b) {
    tokens[(int64_t)b * N] = -1;
    for (int v = 1; v < N; ++v) {
      auto q = softmax(load_row(draft, dtype, ((int64_t)b * N + parent[v]) * d_stride, V), T);
      double Z = 0.0;
      for (double e : q) Z += e;
      const double uv = uniform24(seeds[b], (uint32_t)b, (uint32_t)(v - 1), 2u, round);
      tokens[(int64_t)b * N + v] = inverse_cdf(q, Z, uv, nullptr);
    }
  });
  return 0;
}

// ---- a7: outcome cache -----------------------------------------------------
// The speculation cache maps a verification outcome (row, k accepted, bonus t)
// to the branch pre-drafted for it.  [SSD-note] §"SSD 的核心思想".
// Returns 0, or 2 if two entries share a key.
int orc_cache_lookup(const int32_t* row, const int32_t* k, const int32_t* t,
                     const int32_t* branch, int n, const int32_t* accept_len,
                     const int32_t* bonus, int B, int32_t* out_branch, int32_t* all_hit) {
  std::map<std::tuple<int, int, int>, int> cache;
  for (int i = 0; i < n; ++i) {
    auto key = std::make_tuple(row[i], k[i], t[i]);
    if (cache.count(key)) return 2;
    cache[key] = branch[i];
  }
  int all = 1;
  for (int b = 0; b < B; ++b) {
    auto it = cache.find(std::make_tuple(b, accept_len[b], bonus[b]));
    out_branch[b] = it == cache.end() ? -1 : it->second;
    if (out_branch[b] < 0) all = 0;
  }
  *all_hit = all;
  return 0;
}

// ---- a8: geometric fan-out -------------------------------------------------
// [SSD-note] §"最优扇出度分配": acceptance count is geometric, P(k) ~ a^k; the
// cache miss rate at position k falls as a power of the fan-out, F_k^-r; the
// Lagrange optimum of sum_k P(k) F_k^-r under sum_k F_k = budget is
// F_k ~ P(k)^(1/(1+r)) = a^(k/(1+r)) (constant factor absorbed).
// Reading: the same weight law is used for every k = 0..K.  Real-valued
// allocation x_k = budget * w_k / sum(w); integerised by largest remainder
// (floor, then +1 to the largest fractional parts, ties to the lower k).
int orc_fanout_real(int K, int budget, double a, double r, double* x) {
  if (K < 0 || budget < 0 || !(a > 0.0) || !(r >= 0.0)) return 1;
  double sw = 0.0;
  std::vector<double> w(K + 1);
  for (int k = 0; k <= K; ++k) {
    w[k] = std::pow(a, (double)k / (1.0 + r));
    sw += w[k];
  }
  for (int k = 0; k <= K; ++k) x[k] = budget * w[k] / sw;
  return 0;
}
int orc_fanout(int K, int budget, double a, double r, int32_t* F) {
  std::vector<double> x(K + 1);
  if (orc_fanout_real(K, budget, a, r, x.data())) return 1;
  int used = 0;
  std::vector<std::pair<double, int>> frac;
  for (int k = 0; k <= K; ++k) {
    F[k] = (int32_t)std::floor(x[k]);
    used += F[k];
    frac.push_back({x[k] - F[k], k});
  }
  std::stable_sort(frac.begin(), frac.end(),
                   [](const std::pair<double, int>& A, const std::pair<double, int>& Bp) {
                     return A.first > Bp.first;
                   });
  for (int i = 0; i < budget - used; ++i) F[frac[i].second] += 1;
  return 0;
}

}  // extern "C"
