// Plain CPU oracle for the speculative-decoding verify step.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
// call this file: it exists so that tests, the package's smoke check and the
// benchmark's CPU-baseline leg can compare the CUDA kernels against an
// obviously correct, slow, single-threaded restatement of the method.  It
// shares no code, header, table or constant generator with the CUDA library.
//
// Everything is computed in double.  bf16 inputs are widened exactly.
//
// Sources (web pages; the method is stated in prose there, no formulas):
//  [SD]    "What is speculative decoding" explainer (lotook.com), section on
//          the four-stage loop (draft K tokens, verify in one pass,
//          accept/reject left to right, resample at the first rejection or
//          take a bonus token) and the FAQ on losslessness.
//  [SSD]   "Speculative Speculative Decoding" blog (jiwasawa.github.io),
//          section "Saguaro 1. Outcome Prediction": bonus-token candidates
//          taken from the draft logits' top tokens with a fan-out per
//          position, keyed by the verify outcome.
//  [D3D]   "LLMの生成を5倍速くする「D3D」を図で読む" (animemo.app),
//          sections 検証のしくみ③ / 検証のまとめ (greedy verify worked
//          example, tau), 答え:ありうる結果すべてに、先回りして下書きする
//          (the drafter's own 2nd/3rd candidates per rejection position,
//          plus one all-accepted key), ヒット / ミス (hit test).
//
// Readings where the pages are silent (each is listed in the design notes):
//  * acceptance: accept d_j iff u_j <= p_j(d_j) / q_j(d_j)  (min(1,p/q));
//  * residual:  w_i = max(0, p_i - q_i), sampled by inverse CDF in index
//    order; if sum w == 0 sample from p instead;
//  * temperature enters as softmax(l / T); T == 0 is greedy (argmax,
//    lowest index on ties); T < 0 or NaN marks the row invalid;
//  * uniforms: Philox4x32-10, key = seed, counter = (row, position, slot, 0),
//    word 0 -> u = ((x0 >> 8) + 1) * 2^-24 in (0, 1]; slot 0 = accept test,
//    slot 1 = residual / bonus sample;
//  * outcome-prediction keys: top-f_k draft tokens at position k by raw
//    draft logit excluding the drafted token d_k (ties -> lowest index,
//    -inf logits never become keys); position K uses an optional draft
//    "bonus" row with no exclusion.
//
// Parity pins (see tests/test_oracle_*.py): worked greedy example, bonus
// case, exact enumeration of the output law at V=4, K=2 (losslessness),
// chi-square at V=8 over 10^6 Philox rounds, closed-form invariants, brute
// force compaction / top-F, key counts from the D3D preparation table, and
// Philox against an independent implementation plus a published
// known-answer vector.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#include <algorithm>

namespace {

// ---------------------------------------------------------------- Philox ----
// Philox4x32 with 10 rounds, from J. Salmon, M. Moraes, R. Dror, D. Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): each round
// multiplies counter words 0 and 2 by the two round multipliers, keeps the
// 64-bit products' halves, xors the high halves with the other counter words
// and the key, and bumps the key by the Weyl constants.
struct Philox4x32 {
  static void round(uint32_t c[4], const uint32_t k[2]) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    const uint32_t n0 = hi1 ^ c[1] ^ k[0];
    const uint32_t n1 = lo1;
    const uint32_t n2 = hi0 ^ c[3] ^ k[1];
    const uint32_t n3 = lo0;
    c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
  }
  static void run(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
      round(c, k);
      k[0] += 0x9E3779B9u;
      k[1] += 0xBB67AE85u;
    }
    std::memcpy(out, c, sizeof(c));
  }
};

double uniform_from_philox(uint64_t seed, uint32_t row, uint32_t pos, uint32_t slot) {
  const uint32_t ctr[4] = {row, pos, slot, 0u};
  const uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  Philox4x32::run(ctr, key, out);
  // top 24 bits of word 0, shifted into (0, 1]; exact in float and double.
  return (double)((out[0] >> 8) + 1u) * (1.0 / 16777216.0);
}

// ------------------------------------------------------------ logit rows ----
enum { DT_F32 = 0, DT_BF16 = 1 };

double widen(const void *base, int dtype, int64_t i) {
  if (dtype == DT_F32) return (double)((const float *)base)[i];
  const uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
  float f;
  std::memcpy(&f, &bits, sizeof(f));
  return (double)f;
}

std::vector<double> load_row(const void *base, int dtype, int64_t row, int V) {
  std::vector<double> l((size_t)V);
  for (int i = 0; i < V; ++i) l[(size_t)i] = widen(base, dtype, row * (int64_t)V + i);
  return l;
}

// index of the largest logit; ties go to the lowest index.
int argmax_lowest(const std::vector<double> &l) {
  int best = 0;
  for (int i = 1; i < (int)l.size(); ++i)
    if (l[(size_t)i] > l[(size_t)best]) best = i;
  return best;
}

// softmax(l / T) written out: p_i = exp((l_i - m)/T) / sum_t exp((l_t - m)/T)
// with m = max l.  Also returns Z = sum_t exp((l_t - m)/T) and m.
std::vector<double> softmax_T(const std::vector<double> &l, double T, double *Z_out, double *m_out) {
  double m = -std::numeric_limits<double>::infinity();
  for (double v : l) m = std::max(m, v);
  std::vector<double> e(l.size());
  double Z = 0.0;
  for (size_t i = 0; i < l.size(); ++i) {
    e[i] = std::exp((l[i] - m) / T);
    Z += e[i];
  }
  for (double &v : e) v /= Z;
  if (Z_out) *Z_out = Z;
  if (m_out) *m_out = m;
  return e;
}

const double kGuard = 1e-6;

// Inverse-CDF draw from unnormalised weights w (all >= 0) with uniform u:
// the smallest i with C_i = sum_{t<=i} w_t > u*S, S = sum w, scanning in
// index order.  If rounding leaves no such i, the largest i with w_i > 0.
// *near is set when the chosen bin's nearer edge is within 1e-6*S of u*S.
int inverse_cdf(const std::vector<double> &w, double u, bool *near) {
  double S = 0.0;
  for (double v : w) S += v;
  const double target = u * S;
  double C = 0.0;
  for (size_t i = 0; i < w.size(); ++i) {
    const double prev = C;
    C += w[i];
    if (C > target) {
      *near = std::min(C - target, target - prev) < kGuard * S;
      return (int)i;
    }
  }
  int last = -1;
  for (size_t i = 0; i < w.size(); ++i)
    if (w[i] > 0.0) last = (int)i;
  *near = true;  // the draw fell past the rounded total: a boundary case
  return last < 0 ? 0 : last;
}

struct RowResult {
  int n_acc = 0, tau = 0, token = -1;
  int guard_pos = -1;       // first position with a near-boundary decision
  bool valid = true;
  bool nonfinite = false;   // invalid because a row it reads is not finite
  bool hit = false;
};

// A logit row fails the finiteness check when it holds a NaN or +inf, or
// when every value is -inf (no distribution can be formed from it); single
// -inf values are allowed and carry zero weight.
bool row_not_finite(const void *base, int dtype, int64_t row, int V) {
  bool any_finite = false;
  for (int i = 0; i < V; ++i) {
    const double v = widen(base, dtype, row * (int64_t)V + i);
    if (std::isnan(v) || v == std::numeric_limits<double>::infinity()) return true;
    if (v != -std::numeric_limits<double>::infinity()) any_finite = true;
  }
  return !any_finite;
}

// Optional finiteness check of the rows a verify call reads for one
// sequence: the K+1 target rows; draft row j when the sequence is sampled or
// keys are built at position j (keys_at[j] != 0); the bonus draft row when
// keys are built at position K.
struct FiniteCheck {
  bool on = false;
  const int32_t *keys_at = nullptr;  // [K+1] or null: no keys
  const void *bonus = nullptr;       // bonus draft rows [B][V] or null
  int64_t bonus_row = 0;
};

// One sequence of the verify step with the uniforms given explicitly.
//   target: [K+1][V] logits, draft: [K][V] logits, tokens: [K] drafted ids.
//   u_accept[j]: uniform of the accept test at position j (slot 0).
//   u_sample[j]: uniform of the residual (j < K) or bonus (j == K) draw.
// Optional per-position outputs (may be null): ratio/p_tok/q_tok [K],
// argmax [K+1], Zt [K+1], Zd [K].
RowResult verify_one(int K, int V, int dtype, const void *target, int64_t trow0,
                     const void *draft, int64_t drow0, const int32_t *tokens, double T,
                     const double *u_accept, const double *u_sample,
                     double *ratio, double *p_tok, double *q_tok, int32_t *argmax_out,
                     double *Zt_out, double *Zd_out, int32_t *out_tokens,
                     const FiniteCheck &fc = FiniteCheck()) {
  RowResult res;
  for (int j = 0; j <= K; ++j) out_tokens[j] = -1;
  bool tokens_ok = true;
  for (int j = 0; j < K; ++j)
    if (tokens[j] < 0 || tokens[j] >= V) tokens_ok = false;
  const bool temp_ok = !(T < 0.0) && !std::isnan(T) && !std::isinf(T);
  if (!tokens_ok || !temp_ok) {
    res.valid = false;
    res.tau = 0;
    res.n_acc = 0;
    return res;
  }
  if (fc.on) {
    bool bad = false;
    for (int j = 0; j <= K && !bad; ++j) bad = row_not_finite(target, dtype, trow0 + j, V);
    for (int j = 0; j < K && !bad; ++j)
      if (T > 0.0 || (fc.keys_at && fc.keys_at[j] > 0))
        bad = row_not_finite(draft, dtype, drow0 + j, V);
    if (!bad && fc.bonus && fc.keys_at && fc.keys_at[K] > 0)
      bad = row_not_finite(fc.bonus, dtype, fc.bonus_row, V);
    if (bad) {
      res.valid = false;
      res.nonfinite = true;
      return res;
    }
  }

  // target rows j = 0..K: argmax, and softmax for T > 0.
  std::vector<std::vector<double>> p((size_t)K + 1), q((size_t)K);
  std::vector<int> amax((size_t)K + 1);
  for (int j = 0; j <= K; ++j) {
    std::vector<double> l = load_row(target, dtype, trow0 + j, V);
    amax[(size_t)j] = argmax_lowest(l);
    if (argmax_out) argmax_out[j] = amax[(size_t)j];
    if (T > 0.0) {
      double Z;
      p[(size_t)j] = softmax_T(l, T, &Z, nullptr);
      if (Zt_out) Zt_out[j] = Z;
    }
  }

  if (T == 0.0) {
    // Greedy: accept d_j while it equals the target's top choice; at the
    // first mismatch emit the target's choice there; if none, the bonus
    // row's choice ([D3D] 検証のしくみ③, 検証のまとめ; [SD] FAQ).
    int m = K;
    for (int j = 0; j < K; ++j)
      if (tokens[j] != amax[(size_t)j]) { m = j; break; }
    res.n_acc = m;
    res.token = amax[(size_t)m];
  } else {
    // draft rows j = 0..K-1
    for (int j = 0; j < K; ++j) {
      std::vector<double> l = load_row(draft, dtype, drow0 + j, V);
      double Z;
      q[(size_t)j] = softmax_T(l, T, &Z, nullptr);
      if (Zd_out) Zd_out[j] = Z;
    }
    // per-position acceptance ratio p(d)/q(d); q(d) == 0 counts as +inf.
    std::vector<double> r((size_t)K);
    for (int j = 0; j < K; ++j) {
      const double pd = p[(size_t)j][(size_t)tokens[j]];
      const double qd = q[(size_t)j][(size_t)tokens[j]];
      r[(size_t)j] = qd > 0.0 ? pd / qd : std::numeric_limits<double>::infinity();
      if (ratio) ratio[j] = r[(size_t)j];
      if (p_tok) p_tok[j] = pd;
      if (q_tok) q_tok[j] = qd;
    }
    // Left-to-right accept/reject ([SD] the four-stage loop): a token the
    // target likes at least as much as the draft is always kept, otherwise
    // kept with probability p/q; stop at the first rejection.
    int m = K;
    for (int j = 0; j < K; ++j) {
      const double u = u_accept[j];
      if (res.guard_pos < 0 && std::fabs(u - r[(size_t)j]) < kGuard) res.guard_pos = j;
      if (!(u <= r[(size_t)j])) { m = j; break; }
    }
    // Correction token at the first rejection from the residual max(0,p-q),
    // else the bonus token from the last target row.
    std::vector<double> w((size_t)V);
    if (m < K) {
      double S = 0.0;
      for (int i = 0; i < V; ++i) {
        w[(size_t)i] = std::max(0.0, p[(size_t)m][(size_t)i] - q[(size_t)m][(size_t)i]);
        S += w[(size_t)i];
      }
      if (S == 0.0) w = p[(size_t)m];
    } else {
      w = p[(size_t)K];
    }
    bool near = false;
    res.token = inverse_cdf(w, u_sample[m], &near);
    if (near && res.guard_pos < 0) res.guard_pos = m;
    res.n_acc = m;
  }
  res.tau = res.n_acc + 1;
  for (int j = 0; j < res.n_acc; ++j) out_tokens[j] = tokens[j];
  out_tokens[res.n_acc] = res.token;
  return res;
}

struct Cand {
  double v;
  int i;
};

}  // namespace

extern "C" {

// Raw Philox4x32-10 block, for pinning against other implementations.
void oracle_philox4x32_10(const uint32_t *ctr4, const uint32_t *key2, uint32_t *out4) {
  Philox4x32::run(ctr4, key2, out4);
}

double oracle_uniform(uint64_t seed, uint32_t row, uint32_t pos, uint32_t slot) {
  return uniform_from_philox(seed, row, pos, slot);
}

// One row with explicit uniforms (used by the enumeration pins).
// Returns tau (0 for an invalid row).  out_tokens: [K+1].
int oracle_verify_row_u(int K, int V, int dtype, const void *target, const void *draft,
                        const int32_t *tokens, double T, const double *u_accept,
                        const double *u_sample, int32_t *out_tokens, int32_t *n_acc,
                        int32_t *guard_pos, double *ratio, double *p_tok, double *q_tok,
                        int32_t *argmax_out) {
  RowResult r = verify_one(K, V, dtype, target, 0, draft, 0, tokens, T, u_accept, u_sample,
                           ratio, p_tok, q_tok, argmax_out, nullptr, nullptr, out_tokens);
  if (n_acc) *n_acc = r.n_acc;
  if (guard_pos) *guard_pos = r.guard_pos;
  return r.tau;
}

// Full batch with Philox uniforms.  Rows are numbered row_base + b for the
// uniform counters.  keys (optional): [B][n_keys][2] cache keys (k, token);
// hit (optional): [B].  Per-position optional outputs as in verify_one,
// laid out [B][K] (ratio, p_tok, q_tok, Zd) and [B][K+1] (argmax, Zt).
// Returns the number of invalid rows.
// check_finite (optional): with it, rows the call reads are checked as
// FiniteCheck describes; fanout [K+1] (or null) marks the positions whose
// draft rows are read for keys, draft_bonus [B][V] (or null) the bonus draft
// rows; nonfinite [B] (optional) receives 1 for each sequence the check
// made invalid.
int oracle_verify_checked(int B, int K, int V, int dtype, const void *target, const void *draft,
                          const int32_t *tokens, const float *temperature, uint64_t seed,
                          int64_t row_base, const int32_t *keys, int n_keys,
                          int32_t *num_accepted, int32_t *out_tokens, int32_t *tau, uint8_t *hit,
                          int32_t *guard_pos, double *ratio, double *p_tok, double *q_tok,
                          int32_t *argmax_out, double *Zt, double *Zd, int check_finite,
                          const int32_t *fanout, const void *draft_bonus, uint8_t *nonfinite) {
  int invalid = 0;
  std::vector<double> ua((size_t)std::max(K, 1)), us((size_t)K + 1);
  for (int b = 0; b < B; ++b) {
    const uint32_t row = (uint32_t)(row_base + b);
    for (int j = 0; j < K; ++j) ua[(size_t)j] = uniform_from_philox(seed, row, (uint32_t)j, 0u);
    for (int j = 0; j <= K; ++j) us[(size_t)j] = uniform_from_philox(seed, row, (uint32_t)j, 1u);
    const size_t pk = (size_t)b * (size_t)K, pk1 = (size_t)b * (size_t)(K + 1);
    FiniteCheck fc;
    fc.on = check_finite != 0;
    fc.keys_at = fanout;
    fc.bonus = draft_bonus;
    fc.bonus_row = b;
    RowResult r = verify_one(
        K, V, dtype, target, (int64_t)b * (K + 1), draft, (int64_t)b * K, tokens + pk,
        (double)temperature[b], ua.data(), us.data(), ratio ? ratio + pk : nullptr,
        p_tok ? p_tok + pk : nullptr, q_tok ? q_tok + pk : nullptr,
        argmax_out ? argmax_out + pk1 : nullptr, Zt ? Zt + pk1 : nullptr, Zd ? Zd + pk : nullptr,
        out_tokens + pk1, fc);
    if (!r.valid) ++invalid;
    if (nonfinite) nonfinite[b] = r.nonfinite ? 1 : 0;
    num_accepted[b] = r.n_acc;
    tau[b] = r.tau;
    if (guard_pos) guard_pos[b] = r.guard_pos;
    if (hit) {
      bool h = false;
      if (r.valid && keys)
        for (int k = 0; k < n_keys; ++k) {
          const int32_t *key = keys + ((size_t)b * (size_t)n_keys + (size_t)k) * 2;
          if (key[0] == r.n_acc && key[1] == r.token) h = true;
        }
      hit[b] = h ? 1 : 0;
    }
  }
  return invalid;
}

int oracle_verify(int B, int K, int V, int dtype, const void *target, const void *draft,
                  const int32_t *tokens, const float *temperature, uint64_t seed,
                  int64_t row_base, const int32_t *keys, int n_keys, int32_t *num_accepted,
                  int32_t *out_tokens, int32_t *tau, uint8_t *hit, int32_t *guard_pos,
                  double *ratio, double *p_tok, double *q_tok, int32_t *argmax_out,
                  double *Zt, double *Zd) {
  return oracle_verify_checked(B, K, V, dtype, target, draft, tokens, temperature, seed, row_base,
                               keys, n_keys, num_accepted, out_tokens, tau, hit, guard_pos, ratio,
                               p_tok, q_tok, argmax_out, Zt, Zd, 0, nullptr, nullptr, nullptr);
}

// Outcome prediction ([SSD] Saguaro outcome prediction; [D3D] 先回りして
// 下書きする): for each position k < K the fanout[k] highest draft logits
// at k, skipping the drafted token d_k (it carries no residual mass after
// a rejection) and -inf logits, ties to the lowest index; for k == K the
// fanout[K] highest logits of the optional bonus draft row.  Missing
// candidates leave (-1, -1).  keys: [B][n_keys][2] with
// n_keys = sum(fanout).  Returns n_keys.
int oracle_outcome_predict(int B, int K, int V, int dtype, const void *draft,
                           const int32_t *tokens, const void *draft_bonus,
                           const int32_t *fanout, int32_t *keys) {
  int n_keys = 0;
  for (int k = 0; k <= K; ++k) n_keys += fanout[k];
  for (int b = 0; b < B; ++b) {
    int slot = 0;
    for (int k = 0; k <= K; ++k) {
      std::vector<Cand> cand;
      if (k < K || draft_bonus) {
        const int excl = k < K ? tokens[(size_t)b * K + k] : -1;
        for (int i = 0; i < V; ++i) {
          const double v = k < K ? widen(draft, dtype, ((int64_t)b * K + k) * V + i)
                                 : widen(draft_bonus, dtype, (int64_t)b * V + i);
          if (i == excl || v == -std::numeric_limits<double>::infinity() || std::isnan(v)) continue;
          cand.push_back({v, i});
        }
        std::stable_sort(cand.begin(), cand.end(),
                         [](const Cand &a, const Cand &c) { return a.v > c.v; });
      }
      for (int f = 0; f < fanout[k]; ++f, ++slot) {
        int32_t *key = keys + ((size_t)b * (size_t)n_keys + (size_t)slot) * 2;
        if (f < (int)cand.size()) {
          key[0] = k;
          key[1] = cand[(size_t)f].i;
        } else {
          key[0] = -1;
          key[1] = -1;
        }
      }
    }
  }
  return n_keys;
}

// Compaction: offsets[b] = sum_{b' < b} tau[b'] (B+1 entries) and
// packed[offsets[b] + i] = out_tokens[b][i] for i < tau[b].
void oracle_compact(int B, int K, const int32_t *out_tokens, const int32_t *tau,
                    int32_t *offsets, int32_t *packed) {
  int32_t acc = 0;
  for (int b = 0; b < B; ++b) {
    offsets[b] = acc;
    for (int i = 0; i < tau[b]; ++i) packed[acc + i] = out_tokens[(size_t)b * (K + 1) + i];
    acc += tau[b];
  }
  offsets[B] = acc;
}

// Packing of the drafter's next pass ([D3D] パック:24ブロックを1回の計算で
// and the list of continuations before it).  One block is K+1 tokens: an
// anchor (already confirmed) and K drafted tokens.  The pack holds the block
// under verification (block 0) and one continuation block per outcome key:
//  * block 0: anchor[b], then d_0..d_{K-1}, at positions anchor_pos[b] + i;
//  * key (k, c), 0 <= k <= K: a rejection at k (or, k == K, all accepted)
//    confirms the anchor and d_0..d_{k-1}, and c takes position
//    anchor_pos[b] + 1 + k; its block is c followed by K mask tokens at the
//    next K positions;
//  * an empty key (or k outside [0, K]) leaves its block empty: tokens,
//    positions and ctx all -1.
// ctx[b][i]: how many tokens of block 0 block i sees besides the shared
// prefix ("each block sees the text before it and itself"): 0 for block 0
// (it sees itself), k + 1 for the continuation of key (k, c).
// tokens / positions: [B][1 + n_keys][K + 1]; ctx: [B][1 + n_keys].
void oracle_d3d_pack(int B, int K, int n_keys, const int32_t *keys, const int32_t *draft_tokens,
                     const int32_t *anchor, const int32_t *anchor_pos, int32_t mask_token,
                     int32_t *tokens, int32_t *positions, int32_t *ctx) {
  const int L = K + 1, nb = 1 + n_keys;
  for (int b = 0; b < B; ++b) {
    for (int blk = 0; blk < nb; ++blk) {
      int32_t *t = tokens + ((size_t)b * nb + blk) * L;
      int32_t *p = positions + ((size_t)b * nb + blk) * L;
      int32_t &c = ctx[(size_t)b * nb + blk];
      if (blk == 0) {
        for (int i = 0; i < L; ++i) {
          t[i] = i == 0 ? anchor[b] : draft_tokens[(size_t)b * K + (i - 1)];
          p[i] = anchor_pos[b] + i;
        }
        c = 0;
        continue;
      }
      const int32_t *key = keys + ((size_t)b * n_keys + (blk - 1)) * 2;
      const int k = key[0];
      if (k < 0 || k > K || key[1] < 0) {
        for (int i = 0; i < L; ++i) t[i] = p[i] = -1;
        c = -1;
        continue;
      }
      for (int i = 0; i < L; ++i) {
        t[i] = i == 0 ? key[1] : mask_token;
        p[i] = anchor_pos[b] + 1 + k + i;
      }
      c = k + 1;
    }
  }
}

// N-gram / prompt-lookup drafting ([SD] FAQ "is a separate draft model
// always needed?": the engine finds a matching span in the prompt and recent
// output and copies the tokens that follow it as drafts; [SSD] Saguaro
// fallback: an n-gram model as the light fallback drafter at large batch).
// For each row b with history h[0..len): for n = n_max down to n_min, the
// last n tokens h[len-n..len) are searched for at earlier places: the
// latest i with i + n < len (the span must be followed by at least one
// token) and h[i..i+n) == h[len-n..len).  The first n that has such an i
// wins; the drafts are h[i+n .. min(i+n+K, len)), the remaining slots -1.
// No match: count 0, all -1, match_pos and match_n -1.
// history: [B][L] (row b uses its first len[b] tokens); drafts: [B][K].
void oracle_ngram_draft(int B, int L, int K, int n_max, int n_min, const int32_t *history,
                        const int32_t *len, int32_t *drafts, int32_t *count, int32_t *match_pos,
                        int32_t *match_n) {
  for (int b = 0; b < B; ++b) {
    const int32_t *h = history + (size_t)b * L;
    const int n_tok = len[b];
    int best_i = -1, best_n = -1;
    for (int n = n_max; n >= n_min && best_i < 0; --n) {
      if (n > n_tok) continue;
      for (int i = n_tok - n - 1; i >= 0; --i) {  // latest first; i + n < n_tok
        bool same = true;
        for (int t = 0; t < n && same; ++t) same = h[i + t] == h[n_tok - n + t];
        if (same) {
          best_i = i;
          best_n = n;
          break;
        }
      }
    }
    int c = 0;
    for (int j = 0; j < K; ++j) {
      int v = -1;
      if (best_i >= 0 && best_i + best_n + j < n_tok) {
        v = h[best_i + best_n + j];
        ++c;
      }
      drafts[(size_t)b * K + j] = v;
    }
    count[b] = c;
    match_pos[b] = best_i;
    match_n[b] = best_n;
  }
}

// KV-cache rollback after a round ([SD] FAQ on speculative decoding and the
// KV cache: when the target rejects the drafts after some position, the
// engine rolls both models' KV caches back and truncates them, dropping the
// rejected entries before the next cycle).  Row b's cache holds kv_len[b]
// entries in pages of page_size entries listed in block_table[b][0..); the
// round appended `appended` of them (the verify pass: the anchor and the K
// drafts, K + 1) and confirms the first tau[b] (the anchor and the accepted
// drafts; the correction or bonus token has no entry yet; 0 for an invalid
// row).  new_len = kv_len - appended + min(tau, appended) (appended and the
// kept entries clamped to the entries the row holds).  The pages past
// ceil(new_len / page_size), up to ceil(kv_len / page_size), are freed: their
// ids go, row after row, to freed[free_offsets[b] ...] and their table
// slots become -1.  free_offsets has B + 1 entries.
void oracle_kv_rollback(int B, int page_size, int max_pages, int appended, const int32_t *kv_len,
                        const int32_t *tau, int32_t *block_table, int32_t *new_len,
                        int32_t *freed, int32_t *free_offsets) {
  int32_t acc = 0;
  for (int b = 0; b < B; ++b) {
    const int before = std::max(kv_len[b] - appended, 0);    // entries older than the round
    const int keep = std::min(std::min(std::max(tau[b], 0), appended), kv_len[b] - before);
    const int n_new = before + keep;
    const int used = (kv_len[b] + page_size - 1) / page_size;
    const int still = (n_new + page_size - 1) / page_size;
    new_len[b] = n_new;
    free_offsets[b] = acc;
    for (int p = still; p < used && p < max_pages; ++p) {
      freed[acc++] = block_table[(size_t)b * max_pages + p];
      block_table[(size_t)b * max_pages + p] = -1;
    }
  }
  free_offsets[B] = acc;
}

}  // extern "C"
