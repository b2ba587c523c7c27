// Target-priority admission of Draft steps ("Resource-Efficient Speculative
// Decoding for Long-Context LLM Serving", section 4.3, "Target-priority
// scheduling" and the paragraphs after it).  Host-side decision logic only:
// the caller runs the Draft steps (e.g. on a low-priority stream or on a
// restricted set of SMs) and reports their completion and the Target's
// observed latency.
#include <cstdint>
#include <new>
#include <unordered_map>

#include "svx.h"

struct svx_sched_s {
  svx_sched_config cfg;
  double t_D, dT;
  bool paused = false;
  std::unordered_map<int64_t, int64_t> in_flight;  // request -> sequence number of its unfinished step
  std::unordered_map<int64_t, int64_t> seq;
};

extern "C" {

svx_status svx_sched_create(const svx_sched_config* cfg, svx_sched* out) {
  if (!cfg || !out || !(cfg->ema > 0.0 && cfg->ema <= 1.0) || !(cfg->delta >= 0.0) || !(cfg->t_draft >= 0.0) ||
      !(cfg->eps_target >= 0.0))
    return SVX_ERR_INVALID_ARG;
  svx_sched s = new (std::nothrow) svx_sched_s();
  if (!s) return SVX_ERR_OOM;
  s->cfg = *cfg;
  s->t_D = cfg->t_draft;
  s->dT = cfg->delta_target;
  *out = s;
  return SVX_OK;
}

svx_status svx_sched_destroy(svx_sched s) {
  delete s;
  return SVX_OK;
}

svx_status svx_sched_new_round(svx_sched s) {
  if (!s) return SVX_ERR_INVALID_ARG;
  if (s->paused && s->dT <= s->cfg.eps_target) s->paused = false;
  return SVX_OK;
}

svx_status svx_sched_try_admit(svx_sched s, int64_t req, int64_t round, double now, double window,
                               svx_draft_instr* out, int32_t* admitted) {
  if (!s || !out || !admitted) return SVX_ERR_INVALID_ARG;
  *admitted = 0;
  if (s->paused || s->in_flight.count(req)) return SVX_OK;
  // dT_hat <= eps_T and t_D_hat + delta <= S_hat
  if (!(s->dT <= s->cfg.eps_target && s->t_D + s->cfg.delta <= window)) return SVX_OK;
  const int64_t q = ++s->seq[req];
  s->in_flight[req] = q;
  *out = svx_draft_instr{req, round, q, s->cfg.alloc, now + window - s->t_D - s->cfg.delta};
  *admitted = 1;
  return SVX_OK;
}

svx_status svx_sched_check_start(svx_sched s, const svx_draft_instr* ins, int64_t cur_req, int64_t cur_round,
                                 double now, int32_t* ok) {
  if (!s || !ins || !ok) return SVX_ERR_INVALID_ARG;
  *ok = (ins->req == cur_req && ins->round == cur_round && now <= ins->t_latest) ? 1 : 0;
  if (!*ok) {  // expired or mismatched: not executed, and the request may be scheduled again
    auto it = s->in_flight.find(ins->req);
    if (it != s->in_flight.end() && it->second == ins->seq) s->in_flight.erase(it);
  }
  return SVX_OK;
}

svx_status svx_sched_ack(svx_sched s, int64_t req, int64_t seq, double t_draft_observed, int32_t* accepted) {
  if (!s || !accepted) return SVX_ERR_INVALID_ARG;
  *accepted = 0;
  auto it = s->in_flight.find(req);
  if (it == s->in_flight.end() || it->second != seq) return SVX_OK;  // stale or unknown ACK
  s->in_flight.erase(it);
  s->t_D = s->t_D + s->cfg.ema * (t_draft_observed - s->t_D);
  *accepted = 1;
  return SVX_OK;
}

svx_status svx_sched_observe_target(svx_sched s, double t_co, double t_alone) {
  if (!s || !(t_alone > 0.0)) return SVX_ERR_INVALID_ARG;
  const double d = (t_co - t_alone) / t_alone;
  s->dT = s->dT + s->cfg.ema * (d - s->dT);
  if (d > s->cfg.eps_target) s->paused = true;  // stop submitting; exclusive Target execution resumes
  return SVX_OK;
}

svx_status svx_sched_estimates(svx_sched s, double* t_draft, double* delta_target, int32_t* paused) {
  if (!s || !t_draft || !delta_target || !paused) return SVX_ERR_INVALID_ARG;
  *t_draft = s->t_D;
  *delta_target = s->dT;
  *paused = s->paused ? 1 : 0;
  return SVX_OK;
}

}  // extern "C"
