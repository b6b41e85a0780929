/*
 * dmtp_gate.h — draft-depth gate: the number of drafts each verify checks.
 *
 * Source: colibri speculative-decoding doc, the draft-depth gate paragraph and its
 * per-step refinement. A verify of k drafts is scored as value(k) = E(k) / cost(k) plain
 * decode steps, with
 *   E(k)    = 1 + a_1 + a_1 a_2 + ... + a_1 ... a_k,
 *   cost(k) = (T(k+1) + (k - 1) d) / T(1),
 * where a_j estimates how often draft j survives given that the earlier drafts did,
 * T(n) is the observed duration of an n-row forward and d the observed extra time of
 * one more draft. The depth of highest value is verified when its value is above 1
 * (else a plain step); unobserved row counts follow T(1)(1 + (n - 1) rho); every 16th
 * decision looks one draft deeper and a plain step is forced after 64 multi-row
 * forwards in a row. In the per-step form, each draft's own probability selects the
 * acceptance observed for drafts of similar probability (ten bins) and only the verify
 * is priced.
 *
 * Readings where the page leaves a step open (the same in the test oracle):
 *   - running averages (a_j, T(n), d) are exponential with weight 1/16; the first
 *     measurement of T(n) or d sets it;
 *   - rho is the least-squares slope through the origin of T(n)/T(1) - 1 against n - 1
 *     over the measured n >= 2 (summed in increasing n), 0.5 until T(1) and one
 *     multi-row forward are measured; while T(1) is unmeasured cost(k) = 1 + k rho;
 *   - equal values go to the smaller k; the probe (every 16th pick, counted from the
 *     first) takes min(proposed, best + 1) with best = 0 when the gate declines; the
 *     forced plain step takes precedence;
 *   - bin i holds p in [i/10, (i+1)/10) (p = 1 in bin 9), starting at (i + 1/2)/10 with
 *     the weight of two verifies: estimate = (2 centre + accepted) / (2 + judged);
 *   - default priors a_1 = 0.8, a_2 = 0.6, a_j = 0.5 beyond (the page's MTP-head priors).
 *
 * Host-only: no device memory, no CUDA calls. A gate belongs to one draft source and to
 * one caller at a time (not thread-safe). Every int-returning call returns DMTP_OK or a
 * negative DMTP_E* code (dmtp.h); a call that fails leaves the gate unchanged.
 */
#ifndef DMTP_GATE_H
#define DMTP_GATE_H

#include "dmtp.h"

#ifdef __cplusplus
extern "C" {
#endif

#define DMTP_GATE_MAX_DRAFTS 32 /* drafts a verify may carry                       */
#define DMTP_GATE_MAX_ROWS 64   /* row counts a forward may report to the gate     */
#define DMTP_GATE_BINS 10       /* probability bins of the per-step form           */

typedef struct dmtp_gate dmtp_gate; /* opaque, owned by the library */

typedef struct {
  int max_drafts;
  double a[DMTP_GATE_MAX_DRAFTS];      /* a_1 .. a_max_drafts                          */
  double t[DMTP_GATE_MAX_ROWS + 1];    /* t[n]: averaged seconds of an n-row forward;
                                          0 where none was reported (t[0] unused)     */
  double d;                            /* averaged seconds per draft past the first   */
  int d_measured;                      /* 0 until dmtp_gate_draft_cost was called     */
  double rho;                          /* the current slope (0.5 until fitted)         */
  long long picks;                     /* picks so far (both forms)                    */
  long long since_plain;               /* forwards since the last one-row forward      */
  long long bin_judged[DMTP_GATE_BINS];
  long long bin_accepted[DMTP_GATE_BINS];
} dmtp_gate_stats;

/* A gate for verifies of at most max_drafts (1..DMTP_GATE_MAX_DRAFTS) drafts. priors:
 * host array [max_drafts] of a_1.. in [0, 1], or NULL for the defaults. */
int dmtp_gate_create(int max_drafts, const double* priors, dmtp_gate** out);

/* After every forward, plain steps (rows = 1) too: rows in 1..DMTP_GATE_MAX_ROWS,
 * seconds > 0 (finite). */
int dmtp_gate_forward(dmtp_gate* g, int rows, double seconds);

/* Time spent writing one draft past the first: seconds >= 0 (finite). */
int dmtp_gate_draft_cost(dmtp_gate* g, double seconds);

/* A settled verify: `accepted` drafts accepted and `judged` drafts settled (accepted,
 * plus 1 after a rejection): 0 <= accepted <= judged <= min(accepted + 1, max_drafts).
 * p: NULL, or host array [judged] of the drafts' probabilities in [0, 1] (feeds the
 * bins of the per-step form). */
int dmtp_gate_result(dmtp_gate* g, int judged, int accepted, const double* p);

/* How many of `proposed` (>= 0; more than max_drafts counts as max_drafts) drafts to
 * carry: *k in 0..proposed (0: a plain step), *value = value(*k) (1 for a plain step;
 * value may be NULL). */
int dmtp_gate_pick(dmtp_gate* g, int proposed, int* k, double* value);

/* The per-step form: p = host array [proposed] of this step's drafts' probabilities in
 * [0, 1] (NULL only when proposed = 0); only their verify is priced. */
int dmtp_gate_pick_p(dmtp_gate* g, int proposed, const double* p, int* k, double* value);

/* A copy of the gate's state. */
int dmtp_gate_read(const dmtp_gate* g, dmtp_gate_stats* out);

/* Never fails; NULL is a no-op. */
void dmtp_gate_free(dmtp_gate* g);

#ifdef __cplusplus
}
#endif
#endif /* DMTP_GATE_H */
