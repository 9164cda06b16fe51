// Width controller (host).
//
// "GPU-Resident Speculative Decoding ..." (Design > Feedback Control of Speculation Width):
// the step cost T(N) of every tree size is measured at load time; the acceptance kernel
// records the accepted nodes of every step and the drafter the match length of its best
// candidate; between windows the controller estimates the expected accepted tokens of each
// width from the recent match lengths, using the acceptance observed for the same match
// length, and picks the width that maximises expected tokens per unit time; like a
// congestion controller it probes a wider tree after a period of plain decoding, with a
// spacing that follows the measured costs; the completion interval of consecutive windows
// refines T(N) through an exponential moving average.
//
// Readings (the page gives no constants): history of the last 32 steps; prior of 2
// pseudo-steps at 1 + 0.5 * min(N - 1, match length) tokens; a match length of 2 assumed
// before any step; probe spacing ceil(4 * T(N_2) / T(N_1)) windows clamped to [2, 64], doubled
// (up to 64) after each probe that accepts no draft and reset by one that accepts any, as a
// congestion controller backs off; moving-average weight 0.25.
#include <algorithm>
#include <cmath>
#include <deque>
#include <vector>

#include "../../include/w4a8.h"

#define W4A8_API extern "C" __attribute__((visibility("default")))

namespace {
constexpr int kMaxLen = 8;
constexpr int kHistory = 32;
constexpr double kPriorSteps = 2.0;
constexpr double kPriorPerMatch = 0.5;
constexpr int kAssumedMatch = 2;
constexpr double kAlpha = 0.25;
}  // namespace

struct w4a8_controller {
  std::vector<int> widths;
  std::vector<double> cost;
  std::vector<double> sum_tok, cnt;  // [width index][match length 0..8]
  std::deque<int> recent;
  int low_streak = 0;
  int base_every = 4;      // probe spacing from the measured costs
  int probe_every = 4;     // current spacing (backs off after failed probes)
  int pending_probes = 0;  // probes chosen whose windows have not been observed
  bool probing = false;

  double prior(int w, int ell) const { return 1.0 + kPriorPerMatch * std::min(w - 1, ell); }
  double est(size_t i, int ell) const {
    const size_t k = i * (kMaxLen + 1) + ell;
    return (sum_tok[k] + kPriorSteps * prior(widths[i], ell)) / (cnt[k] + kPriorSteps);
  }
  double expected(size_t i) const {
    if (widths[i] == 1) return 1.0;
    if (recent.empty()) return est(i, kAssumedMatch);
    double s = 0.0;
    for (int ell : recent) s += est(i, ell);
    return s / (double)recent.size();
  }
  size_t best() const {
    size_t b = 0;
    double bv = -1.0;
    for (size_t i = 0; i < widths.size(); ++i) {
      const double v = expected(i) / cost[i];
      if (v > bv * (1.0 + 1e-12)) {
        bv = v;
        b = i;
      }
    }
    return b;
  }
  int index_of(int w) const {
    for (size_t i = 0; i < widths.size(); ++i)
      if (widths[i] == w) return (int)i;
    return -1;
  }
};

W4A8_API w4a8_status w4a8_controller_create(const int* widths, const float* t_us, int n, w4a8_controller** out) {
  if (!widths || !t_us || !out || n <= 0 || n > 8) return W4A8_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    if (widths[i] < 1 || widths[i] > 16 || !(t_us[i] > 0.0f)) return W4A8_ERR_ARG;
    if (i > 0 && widths[i] <= widths[i - 1]) return W4A8_ERR_ARG;
  }
  w4a8_controller* c = new (std::nothrow) w4a8_controller();
  if (!c) return W4A8_ERR_NOMEM;
  c->widths.assign(widths, widths + n);
  c->cost.assign(t_us, t_us + n);
  c->sum_tok.assign((size_t)n * (kMaxLen + 1), 0.0);
  c->cnt.assign((size_t)n * (kMaxLen + 1), 0.0);
  if (n > 1) {
    const double ratio = c->cost[1] / c->cost[0];
    c->base_every = std::min(64, std::max(2, (int)std::ceil(4.0 * ratio)));
    c->probe_every = c->base_every;
  }
  *out = c;
  return W4A8_OK;
}

W4A8_API void w4a8_controller_destroy(w4a8_controller* c) { delete c; }

W4A8_API int w4a8_controller_choose(w4a8_controller* c) {
  if (!c) return 1;
  size_t b = c->best();
  c->probing = false;
  if (b == 0 && c->widths.size() > 1) {
    if (++c->low_streak >= c->probe_every) {
      c->low_streak = 0;
      c->probing = true;
      ++c->pending_probes;
      b = 1;  // probe the next wider tree once
    }
  } else {
    c->low_streak = 0;
  }
  return c->widths[b];
}

W4A8_API w4a8_status w4a8_controller_observe(w4a8_controller* c, int width, const w4a8_step_stats* stats, int n,
                                             double interval_us) {
  if (!c || (n > 0 && !stats) || n < 0) return W4A8_ERR_ARG;
  const int i = c->index_of(width);
  if (i == 1 && n > 0 && c->pending_probes > 0) {
    // the window of a probe (windows complete in the order they were chosen): back off while
    // probes find nothing to accept, return to the cost-based spacing when one does
    --c->pending_probes;
    int accepted = 0;
    for (int k = 0; k < n; ++k) accepted += std::max(0, (int)stats[k].n_emitted - 1);
    c->probe_every = accepted > 0 ? c->base_every : std::min(64, 2 * c->probe_every);
  }
  for (int k = 0; k < n; ++k) {
    const int ell = std::min<int>(kMaxLen, stats[k].best_match_len);
    if (i >= 0 && stats[k].n_emitted > 0) {
      const size_t idx = (size_t)i * (kMaxLen + 1) + ell;
      c->sum_tok[idx] += stats[k].n_emitted;
      c->cnt[idx] += 1.0;
    }
    c->recent.push_back(ell);
    while ((int)c->recent.size() > kHistory) c->recent.pop_front();
  }
  if (i >= 0 && n > 0 && interval_us > 0.0) c->cost[i] = (1.0 - kAlpha) * c->cost[i] + kAlpha * (interval_us / n);
  return W4A8_OK;
}

W4A8_API double w4a8_controller_expected_tokens(const w4a8_controller* c, int width) {
  if (!c) return 0.0;
  const int i = c->index_of(width);
  return i < 0 ? 0.0 : c->expected((size_t)i);
}

W4A8_API double w4a8_controller_cost(const w4a8_controller* c, int width) {
  if (!c) return 0.0;
  const int i = c->index_of(width);
  return i < 0 ? 0.0 : c->cost[(size_t)i];
}
