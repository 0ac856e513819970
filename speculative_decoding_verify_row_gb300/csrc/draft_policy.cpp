// Host-side draft proposal and window-shape policy (no GPU work).
//
// (1) Prompt-lookup proposal: an n-gram index private to the request, over
//     its whole context, proposes what followed earlier occurrences of the
//     last `match` tokens ("Speculative decoding on RDNA" §06, N-gram takeovers: default
//     match 5, propose 3).  Several matches become the branches of one token
//     tree ("One RDNA4 verify pass has slack for about two dozen speculative
//     tokens", "Spend the budget on a tree": the best few matches, a few
//     branches six to eight tokens deep).
// (2) Window pricing: window cost = a + b per extra row, fitted to measured
//     windows; the draft depth that maximises expected emitted tokens per
//     unit of cost, with one token per step (no drafts) as the fallback
//     (same page, §05); a takeover has to price at least as well as the
//     native window (§06); the AR floor's keep-or-retire decision (§07).
//
// All arithmetic is IEEE double in a fixed order; the library is built with
// floating-point contraction off, so results are the same on every host.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <map>
#include <vector>

#include "verifyrow.h"

namespace {

struct Continuation {
  std::vector<int32_t> toks;
  int count;        // occurrences proposing exactly these tokens
  int last_start;   // start of the most recent such occurrence
};

bool is_fin(double x) { return std::isfinite(x); }

// 1 + sum_{j=1..k} prod_{i<=j} alpha_i: the expected number of emitted
// tokens of a window with k drafts whose i-th draft is accepted with
// probability alpha[i-1] once the drafts before it were.
double expected_emitted(const double* alpha, int k) {
  double e = 1.0, run = 1.0;
  for (int j = 0; j < k; ++j) {
    run *= alpha[j];
    e += run;
  }
  return e;
}

bool valid_alpha(const double* alpha, int k) {
  if (k > 0 && !alpha) return false;
  for (int j = 0; j < k; ++j)
    if (!is_fin(alpha[j]) || alpha[j] < 0.0 || alpha[j] > 1.0) return false;
  return true;
}

// a + b k must be a positive cost for every depth 0..kmax
bool valid_cost(double a, double b, int kmax) {
  if (!is_fin(a) || !is_fin(b) || a <= 0.0) return false;
  return a + b * kmax > 0.0;
}

}  // namespace

extern "C" {

int vr_ngram_propose(const int32_t* context, int len, int match, int propose, int branches,
                     int max_nodes, int32_t* out_tokens, int32_t* out_parent,
                     int32_t* out_n_nodes) {
  if (len < 0 || (len > 0 && !context)) return VR_ERR_ARG;
  if (!out_tokens || !out_parent || !out_n_nodes) return VR_ERR_ARG;
  if (match < 1 || propose < 1 || branches < 1) return VR_ERR_ARG;
  if (max_nodes < 0 || max_nodes > VR_MAX_WINDOW_ROWS - 1) return VR_ERR_ARG;
  *out_n_nodes = 0;
  if (len <= match) return VR_OK;

  // every earlier occurrence of the last `match` tokens (the suffix itself
  // excluded) and the up to `propose` tokens that followed it
  const int32_t* key = context + (len - match);
  std::vector<Continuation> conts;
  std::map<std::vector<int32_t>, size_t> seen;
  for (int s = 0; s + match < len; ++s) {
    if (!std::equal(key, key + match, context + s)) continue;
    const int c0 = s + match;
    const int c1 = std::min(len, c0 + propose);
    std::vector<int32_t> toks(context + c0, context + c1);
    auto it = seen.find(toks);
    if (it == seen.end()) {
      seen.emplace(toks, conts.size());
      conts.push_back({std::move(toks), 1, s});
    } else {
      conts[it->second].count += 1;
      conts[it->second].last_start = s;
    }
  }

  // the most frequent continuations first, the most recent among equals
  std::sort(conts.begin(), conts.end(), [](const Continuation& x, const Continuation& y) {
    if (x.count != y.count) return x.count > y.count;
    return x.last_start > y.last_start;
  });

  // the kept continuations as one tree: shared prefixes share nodes, new
  // nodes are appended (so every parent precedes its children), at most
  // max_nodes nodes
  int n = 0;
  const int keep = std::min<int>(branches, static_cast<int>(conts.size()));
  for (int b = 0; b < keep; ++b) {
    int cur = -1;
    for (const int32_t t : conts[b].toks) {
      int next = -1;
      for (int j = 0; j < n; ++j)
        if (out_parent[j] == cur && out_tokens[j] == t) {
          next = j;
          break;
        }
      if (next < 0) {
        if (n == max_nodes) break;
        out_tokens[n] = t;
        out_parent[n] = cur;
        next = n++;
      }
      cur = next;
    }
  }
  *out_n_nodes = n;
  return VR_OK;
}

int vr_cost_fit(const int32_t* rows, const double* ms, int n, double* out_a, double* out_b) {
  if (!rows || !ms || !out_a || !out_b || n < 2) return VR_ERR_ARG;
  double sx = 0.0, sy = 0.0;
  for (int i = 0; i < n; ++i) {
    if (rows[i] < 1 || !is_fin(ms[i])) return VR_ERR_ARG;
    sx += static_cast<double>(rows[i] - 1);
    sy += ms[i];
  }
  const double mx = sx / n, my = sy / n;
  double sxx = 0.0, sxy = 0.0;
  for (int i = 0; i < n; ++i) {
    const double dx = static_cast<double>(rows[i] - 1) - mx;
    sxx += dx * dx;
    sxy += dx * (ms[i] - my);
  }
  if (sxx == 0.0) return VR_ERR_ARG;   // every sample has the same row count
  const double b = sxy / sxx;
  *out_b = b;
  *out_a = my - b * mx;
  return VR_OK;
}

int vr_choose_depth(const double* alpha, int kmax, double a, double b, int32_t* out_k,
                    double* out_tokens_per_ms) {
  if (!out_k || kmax < 0 || kmax > VR_MAX_WINDOW_ROWS - 1) return VR_ERR_ARG;
  if (!valid_alpha(alpha, kmax) || !valid_cost(a, b, kmax)) return VR_ERR_ARG;
  int best = 0;
  double best_rate = 1.0 / a;
  for (int k = 1; k <= kmax; ++k) {
    const double rate = expected_emitted(alpha, k) / (a + b * k);
    if (rate > best_rate) {
      best = k;
      best_rate = rate;
    }
  }
  *out_k = best;
  if (out_tokens_per_ms) *out_tokens_per_ms = best_rate;
  return VR_OK;
}

int vr_takeover(const double* alpha_native, int k_native, const double* alpha_ngram, int k_ngram,
                double a, double b, int32_t* out_take) {
  if (!out_take || k_native < 0 || k_ngram < 1) return VR_ERR_ARG;
  if (k_native > VR_MAX_WINDOW_ROWS - 1 || k_ngram > VR_MAX_WINDOW_ROWS - 1) return VR_ERR_ARG;
  if (!valid_alpha(alpha_native, k_native) || !valid_alpha(alpha_ngram, k_ngram)) return VR_ERR_ARG;
  if (!valid_cost(a, b, std::max(k_native, k_ngram))) return VR_ERR_ARG;
  const double native = expected_emitted(alpha_native, k_native) / (a + b * k_native);
  const double ngram = expected_emitted(alpha_ngram, k_ngram) / (a + b * k_ngram);
  *out_take = ngram >= native ? 1 : 0;
  return VR_OK;
}

int vr_ar_floor(double ar_ms, const double* window_ms, const int32_t* emitted, int n,
                int32_t* out_speculate) {
  if (!out_speculate || n < 1 || !window_ms || !emitted) return VR_ERR_ARG;
  *out_speculate = 0;
  if (!is_fin(ar_ms) || ar_ms <= 0.0) return VR_OK;        // invalid timing: retire
  for (int i = 0; i < n; ++i)
    if (!is_fin(window_ms[i]) || window_ms[i] <= 0.0 || emitted[i] < 1) return VR_OK;
  for (int i = 0; i < n; ++i)
    if (window_ms[i] / emitted[i] < ar_ms) *out_speculate = 1;
  return VR_OK;
}

}  // extern "C"
