// Draft-cap controller: host code, no device work.
//
// mlx-dspark PyPI page, "The Apple-Silicon speedup ceiling": throughput is
// about A / (drafter + overhead + verify cost) for accept length A and draft
// cap C, and the verify cost of a wider round is measured on the device, not
// assumed.  Wiki page, "Key techniques": a controller picks each round's cap
// from the measured curves and a live acceptance estimate, with
// expected committed tokens 1 + sum_i p^i, and parks speculation (cap 0) when
// it loses; PyPI page, "Tuning": while parked it runs plain steps plus
// periodic probe rounds.
//
// The acceptance estimate is the exponentially weighted maximum-likelihood
// estimate of a geometric acceptance model: a round that verified C drafts and
// accepted a contributes a successes and, if a < C, one failure; S and F are
// EWMAs of those counts and p = S / (S + F).
#include <cmath>

#include "sv_internal.h"

namespace sv {

static double expected_committed(double p, int cap) {
  double total = 0.0, term = 1.0;
  for (int i = 0; i <= cap; ++i) {
    total += term;
    term *= p;
  }
  return total;
}

// Best cap for acceptance p: maximises E(C) / T(C), the smallest C on ties.
static int best_cap(double p, int max_cap, const double* verify_us, const double* draft_us, double overhead_us,
                    double* rate_out) {
  int best = 0;
  double best_rate = -1.0;
  for (int c = 0; c <= max_cap; ++c) {
    const double rate = expected_committed(p, c) / (draft_us[c] + overhead_us + verify_us[c]);
    if (rate > best_rate) {
      best = c;
      best_rate = rate;
    }
  }
  if (rate_out) *rate_out = best_rate;
  return best;
}

static int check_curves(int max_cap, const double* verify_us, const double* draft_us, double overhead_us) {
  if (max_cap < 0 || max_cap > SV_CAP_MAX) return fail(SV_EINVAL, "max_cap must be in [0, %d] (got %d)", SV_CAP_MAX, max_cap);
  if (!verify_us || !draft_us) return fail(SV_EINVAL, "verify_us and draft_us must be non-null");
  if (!(overhead_us >= 0.0) || std::isinf(overhead_us)) return fail(SV_EINVAL, "overhead_us must be finite and >= 0");
  for (int c = 0; c <= max_cap; ++c) {
    if (!(verify_us[c] > 0.0) || std::isinf(verify_us[c]))
      return fail(SV_EINVAL, "verify_us[%d] must be finite and > 0", c);
    if (!(draft_us[c] >= 0.0) || std::isinf(draft_us[c]))
      return fail(SV_EINVAL, "draft_us[%d] must be finite and >= 0", c);
  }
  return SV_OK;
}

}  // namespace sv

using namespace sv;

extern "C" {

double sv_expected_committed(double p, int cap) {
  if (!(p >= 0.0 && p <= 1.0) || cap < 0) return NAN;
  return expected_committed(p, cap);
}

int sv_best_cap(double p, int max_cap, const double* verify_us, const double* draft_us, double overhead_us, int* cap,
                double* rate) {
  int st = check_curves(max_cap, verify_us, draft_us, overhead_us);
  if (st) return st;
  if (!(p >= 0.0 && p <= 1.0)) return fail(SV_EINVAL, "p must be in [0, 1]");
  if (!cap) return fail(SV_EINVAL, "cap must be non-null");
  *cap = best_cap(p, max_cap, verify_us, draft_us, overhead_us, rate);
  return SV_OK;
}

int sv_verify_knee(const double* verify_us, int n, double tol, int* width) {
  if (!verify_us || n < 1 || !width) return fail(SV_EINVAL, "verify_us, n >= 1 and width are required");
  if (!(tol >= 0.0)) return fail(SV_EINVAL, "tol must be >= 0");
  int m = 1;
  for (int c = 0; c < n; ++c) {
    if (verify_us[c] <= (1.0 + tol) * verify_us[0])
      m = c + 1;
    else
      break;
  }
  *width = m;
  return SV_OK;
}

int sv_cap_init(sv_cap_controller* ctl, int max_cap, const double* verify_us, const double* draft_us,
                double overhead_us, double alpha, int probe_every, int probe_cap, double p0) {
  if (!ctl) return fail(SV_EINVAL, "controller must be non-null");
  int st = check_curves(max_cap, verify_us, draft_us, overhead_us);
  if (st) return st;
  if (!(alpha > 0.0 && alpha <= 1.0)) return fail(SV_EINVAL, "alpha must be in (0, 1]");
  if (probe_every < 1) return fail(SV_EINVAL, "probe_every must be >= 1");
  if (probe_cap < 1 || probe_cap > max_cap) return fail(SV_EINVAL, "probe_cap must be in [1, max_cap]");
  if (!(p0 >= 0.0 && p0 <= 1.0)) return fail(SV_EINVAL, "p0 must be in [0, 1]");
  ctl->max_cap = max_cap;
  for (int c = 0; c <= SV_CAP_MAX; ++c) {
    ctl->verify_us[c] = c <= max_cap ? verify_us[c] : 0.0;
    ctl->draft_us[c] = c <= max_cap ? draft_us[c] : 0.0;
  }
  ctl->overhead_us = overhead_us;
  ctl->alpha = alpha;
  ctl->probe_every = probe_every;
  ctl->probe_cap = probe_cap;
  ctl->S = p0;  // the prior counts as one round's worth of evidence
  ctl->F = 1.0 - p0;
  ctl->parked = 0;
  ctl->since_probe = 0;
  return SV_OK;
}

double sv_cap_acceptance(const sv_cap_controller* ctl) {
  if (!ctl) return NAN;
  const double tot = ctl->S + ctl->F;
  return tot > 0.0 ? ctl->S / tot : 0.0;
}

int sv_cap_next(sv_cap_controller* ctl, int* cap) {
  if (!ctl || !cap) return fail(SV_EINVAL, "controller and cap must be non-null");
  if (ctl->parked) {
    if (++ctl->since_probe >= ctl->probe_every) {
      ctl->since_probe = 0;
      *cap = ctl->probe_cap;
    } else {
      *cap = 0;
    }
    return SV_OK;
  }
  const int c = best_cap(sv_cap_acceptance(ctl), ctl->max_cap, ctl->verify_us, ctl->draft_us, ctl->overhead_us,
                         nullptr);
  if (c == 0) {
    ctl->parked = 1;
    ctl->since_probe = 0;
  }
  *cap = c;
  return SV_OK;
}

int sv_cap_update(sv_cap_controller* ctl, int cap, int accepted) {
  if (!ctl) return fail(SV_EINVAL, "controller must be non-null");
  if (cap < 0 || cap > ctl->max_cap || accepted < 0 || accepted > cap)
    return fail(SV_EINVAL, "need 0 <= accepted <= cap <= max_cap (got cap %d, accepted %d)", cap, accepted);
  if (cap == 0) return SV_OK;  // a plain step says nothing about acceptance
  const double a = ctl->alpha;
  ctl->S = (1.0 - a) * ctl->S + a * accepted;
  ctl->F = (1.0 - a) * ctl->F + a * (accepted < cap ? 1.0 : 0.0);
  if (ctl->parked &&
      best_cap(sv_cap_acceptance(ctl), ctl->max_cap, ctl->verify_us, ctl->draft_us, ctl->overhead_us, nullptr) > 0)
    ctl->parked = 0;
  return SV_OK;
}

}  // extern "C"
