// I/O-aware dynamic verification width ("Resource-Efficient Speculative
// Decoding for Long-Context LLM Serving", section 4.2, paragraph "I/O-aware
// dynamic verification widths"): the next round's width is
// argmin_q T_round_hat(q) / U_hat(q) over the candidate widths, from recent
// per-width statistics, after an initial sampling phase, switching only when
// the estimated gain exceeds a threshold.  Host-side logic.
#include <algorithm>
#include <new>
#include <vector>

#include "svx.h"

namespace {
struct Stats {
  int64_t n = 0;
  double t_draft = 0, t_h2d = 0, t_attn = 0, t_correct = 0, committed = 0;
};
}  // namespace

struct svx_width_s {
  std::vector<int32_t> widths;
  std::vector<Stats> stats;
  double ema = 0.25, threshold = 0.0;
  int32_t n_init = 1;
  int32_t current = 0;

  int index(int32_t q) const {
    for (size_t i = 0; i < widths.size(); ++i)
      if (widths[i] == q) return static_cast<int>(i);
    return -1;
  }
  // T_round_hat / U_hat; transfer and the attention it overlaps are counted once.  < 0: no estimate.
  double cost(int i) const {
    const Stats& s = stats[static_cast<size_t>(i)];
    if (s.n == 0 || !(s.committed > 0.0)) return -1.0;
    return (s.t_draft + std::max(s.t_h2d, s.t_attn) + s.t_correct) / s.committed;
  }
};

extern "C" {

svx_status svx_width_create(const int32_t* widths, int32_t n, double ema, double threshold, int32_t n_init,
                            svx_width* out) {
  if (!widths || n < 1 || !out || !(ema > 0.0 && ema <= 1.0) || !(threshold >= 0.0) || n_init < 1)
    return SVX_ERR_INVALID_ARG;
  svx_width w = new (std::nothrow) svx_width_s();
  if (!w) return SVX_ERR_OOM;
  w->widths.assign(widths, widths + n);
  w->stats.assign(static_cast<size_t>(n), Stats());
  w->ema = ema;
  w->threshold = threshold;
  w->n_init = n_init;
  w->current = widths[0];
  *out = w;
  return SVX_OK;
}

svx_status svx_width_destroy(svx_width w) {
  delete w;
  return SVX_OK;
}

svx_status svx_width_record(svx_width w, int32_t q, double t_draft, double t_h2d, double t_attn, double t_correct,
                            double committed) {
  if (!w) return SVX_ERR_INVALID_ARG;
  const int i = w->index(q);
  if (i < 0) return SVX_ERR_INVALID_ARG;
  Stats& s = w->stats[static_cast<size_t>(i)];
  auto upd = [&](double& x, double v) { x = (s.n == 0) ? v : x + w->ema * (v - x); };
  upd(s.t_draft, t_draft);
  upd(s.t_h2d, t_h2d);
  upd(s.t_attn, t_attn);
  upd(s.t_correct, t_correct);
  upd(s.committed, committed);
  ++s.n;
  return SVX_OK;
}

svx_status svx_width_next(svx_width w, int32_t* q_out) {
  if (!w || !q_out) return SVX_ERR_INVALID_ARG;
  for (size_t i = 0; i < w->widths.size(); ++i)  // limited initial sampling
    if (w->stats[i].n < w->n_init) {
      w->current = w->widths[i];
      *q_out = w->current;
      return SVX_OK;
    }
  int best = -1;
  double best_cost = 0.0;
  for (size_t i = 0; i < w->widths.size(); ++i) {
    const double c = w->cost(static_cast<int>(i));
    if (c >= 0.0 && (best < 0 || c < best_cost)) {
      best = static_cast<int>(i);
      best_cost = c;
    }
  }
  const double cur = w->cost(w->index(w->current));
  if (best >= 0 && (cur < 0.0 || best_cost < (1.0 - w->threshold) * cur)) w->current = w->widths[static_cast<size_t>(best)];
  *q_out = w->current;
  return SVX_OK;
}

svx_status svx_width_cost(svx_width w, int32_t q, double* cost_out) {
  if (!w || !cost_out) return SVX_ERR_INVALID_ARG;
  const int i = w->index(q);
  if (i < 0) return SVX_ERR_INVALID_ARG;
  *cost_out = w->cost(i);
  return SVX_OK;
}

}  // extern "C"
