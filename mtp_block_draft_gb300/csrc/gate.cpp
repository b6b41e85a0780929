// Draft-depth gate (host only): value(k) = E(k) / cost(k) from running acceptance and
// measured forward times, as the colibri speculative-decoding doc's gate paragraph and
// its paragraph on each step's own drafts define it; readings in dmtp_gate.h.
#include <cmath>
#include <new>

#include "dmtp_gate.h"

namespace {

constexpr double kAvg = 1.0 / 16.0;  // weight of a new measurement in a running average
constexpr int kProbeEvery = 16;      // every 16th pick tries one draft deeper
constexpr int kPlainEvery = 64;      // forwards without a plain step before one is taken
constexpr double kRho0 = 0.5;

bool is_fin(double x) { return std::isfinite(x); }

double avg(double old, bool have, double x) { return have ? old + (x - old) * kAvg : x; }

int bin_of(double p) {
  const int b = (int)std::floor(p * DMTP_GATE_BINS);
  return b < 0 ? 0 : (b > DMTP_GATE_BINS - 1 ? DMTP_GATE_BINS - 1 : b);
}

// E(k) = 1 + a_1 + a_1 a_2 + ... over acc[0..k-1]
double expected_tokens(const double* acc, int k) {
  double e = 1.0, run = 1.0;
  for (int j = 0; j < k; ++j) {
    run *= acc[j];
    e += run;
  }
  return e;
}

}  // namespace

struct dmtp_gate {
  int K;
  double a[DMTP_GATE_MAX_DRAFTS];
  double t[DMTP_GATE_MAX_ROWS + 1];
  bool has_t[DMTP_GATE_MAX_ROWS + 1];
  double d;
  bool has_d;
  long long picks, since_plain;
  long long bin_judged[DMTP_GATE_BINS], bin_accepted[DMTP_GATE_BINS];

  double rho() const {
    if (!has_t[1]) return kRho0;
    double sxy = 0.0, sxx = 0.0;
    bool any = false;
    for (int n = 2; n <= DMTP_GATE_MAX_ROWS; ++n) {
      if (!has_t[n]) continue;
      const double x = (double)(n - 1), y = t[n] / t[1] - 1.0;
      sxy += x * y;
      sxx += x * x;
      any = true;
    }
    return any ? sxy / sxx : kRho0;
  }
  // T(n) / T(1): measured where both are, else 1 + (n - 1) rho
  double t_rel(int n) const {
    if (has_t[1] && n <= DMTP_GATE_MAX_ROWS && has_t[n]) return t[n] / t[1];
    return 1.0 + (n - 1) * rho();
  }
  double cost(int k, bool count_drafting) const {
    double c = t_rel(k + 1);
    if (count_drafting && k >= 1 && has_d && has_t[1]) c += (k - 1) * d / t[1];
    return c;
  }
  double bin_estimate(int b) const {
    const double centre = (b + 0.5) / DMTP_GATE_BINS;
    return (2.0 * centre + (double)bin_accepted[b]) / (2.0 + (double)bin_judged[b]);
  }
  // values[k - 1] = value(k), k = 1..proposed
  void decide(int proposed, const double* values, int* k, double* value) {
    ++picks;
    int pick = 0;
    double v = 1.0;
    if (since_plain < kPlainEvery && proposed > 0) {
      int best = 0;
      double best_v = 1.0;
      for (int j = 1; j <= proposed; ++j)
        if (values[j - 1] > best_v) {
          best = j;
          best_v = values[j - 1];
        }
      pick = best;
      v = best_v;
      if (picks % kProbeEvery == 0) {
        pick = best + 1 < proposed ? best + 1 : proposed;
        v = pick ? values[pick - 1] : 1.0;
      }
    }
    *k = pick;
    if (value) *value = v;
  }
};

extern "C" {

int dmtp_gate_create(int max_drafts, const double* priors, dmtp_gate** out) {
  if (!out) return DMTP_EINVAL;
  *out = nullptr;
  if (max_drafts < 1 || max_drafts > DMTP_GATE_MAX_DRAFTS) return DMTP_EINVAL;
  if (priors)
    for (int j = 0; j < max_drafts; ++j)
      if (!is_fin(priors[j]) || priors[j] < 0.0 || priors[j] > 1.0) return DMTP_EINVAL;
  dmtp_gate* g = new (std::nothrow) dmtp_gate();
  if (!g) return DMTP_ENOMEM;
  g->K = max_drafts;
  for (int j = 0; j < max_drafts; ++j)
    g->a[j] = priors ? priors[j] : (j == 0 ? 0.8 : (j == 1 ? 0.6 : 0.5));
  *out = g;
  return DMTP_OK;
}

int dmtp_gate_forward(dmtp_gate* g, int rows, double seconds) {
  if (!g || rows < 1 || rows > DMTP_GATE_MAX_ROWS || !is_fin(seconds) || !(seconds > 0.0))
    return DMTP_EINVAL;
  g->t[rows] = avg(g->t[rows], g->has_t[rows], seconds);
  g->has_t[rows] = true;
  g->since_plain = rows == 1 ? 0 : g->since_plain + 1;
  return DMTP_OK;
}

int dmtp_gate_draft_cost(dmtp_gate* g, double seconds) {
  if (!g || !is_fin(seconds) || !(seconds >= 0.0)) return DMTP_EINVAL;
  g->d = avg(g->d, g->has_d, seconds);
  g->has_d = true;
  return DMTP_OK;
}

int dmtp_gate_result(dmtp_gate* g, int judged, int accepted, const double* p) {
  if (!g || accepted < 0 || judged < accepted || judged > accepted + 1 || judged > g->K)
    return DMTP_EINVAL;
  if (p)
    for (int j = 0; j < judged; ++j)
      if (!is_fin(p[j]) || p[j] < 0.0 || p[j] > 1.0) return DMTP_EINVAL;
  for (int j = 0; j < judged; ++j) {
    const bool acc = j < accepted;
    g->a[j] = avg(g->a[j], true, acc ? 1.0 : 0.0);
    if (p) {
      const int b = bin_of(p[j]);
      ++g->bin_judged[b];
      if (acc) ++g->bin_accepted[b];
    }
  }
  return DMTP_OK;
}

int dmtp_gate_pick(dmtp_gate* g, int proposed, int* k, double* value) {
  if (!g || !k || proposed < 0) return DMTP_EINVAL;
  if (proposed > g->K) proposed = g->K;
  double values[DMTP_GATE_MAX_DRAFTS];
  for (int j = 1; j <= proposed; ++j)
    values[j - 1] = expected_tokens(g->a, j) / g->cost(j, true);
  g->decide(proposed, values, k, value);
  return DMTP_OK;
}

int dmtp_gate_pick_p(dmtp_gate* g, int proposed, const double* p, int* k, double* value) {
  if (!g || !k || proposed < 0 || (proposed > 0 && !p)) return DMTP_EINVAL;
  if (proposed > g->K) proposed = g->K;
  double acc[DMTP_GATE_MAX_DRAFTS], values[DMTP_GATE_MAX_DRAFTS];
  for (int j = 0; j < proposed; ++j) {
    if (!is_fin(p[j]) || p[j] < 0.0 || p[j] > 1.0) return DMTP_EINVAL;
    acc[j] = g->bin_estimate(bin_of(p[j]));
  }
  for (int j = 1; j <= proposed; ++j)
    values[j - 1] = expected_tokens(acc, j) / g->cost(j, false);
  g->decide(proposed, values, k, value);
  return DMTP_OK;
}

int dmtp_gate_read(const dmtp_gate* g, dmtp_gate_stats* out) {
  if (!g || !out) return DMTP_EINVAL;
  *out = dmtp_gate_stats{};
  out->max_drafts = g->K;
  for (int j = 0; j < g->K; ++j) out->a[j] = g->a[j];
  for (int n = 1; n <= DMTP_GATE_MAX_ROWS; ++n) out->t[n] = g->has_t[n] ? g->t[n] : 0.0;
  out->d = g->has_d ? g->d : 0.0;
  out->d_measured = g->has_d ? 1 : 0;
  out->rho = g->rho();
  out->picks = g->picks;
  out->since_plain = g->since_plain;
  for (int b = 0; b < DMTP_GATE_BINS; ++b) {
    out->bin_judged[b] = g->bin_judged[b];
    out->bin_accepted[b] = g->bin_accepted[b];
  }
  return DMTP_OK;
}

void dmtp_gate_free(dmtp_gate* g) { delete g; }

}  // extern "C"
