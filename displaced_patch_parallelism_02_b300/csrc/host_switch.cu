// Adaptive parallelism switching (Hydiff summaries: gist.science, section
// "自适应并行切换"; Avetisyan, "Адаптивное переключение"): a host-side
// state machine over the per-step denoising discrepancy (rel-MAE of the
// conditional vs the unconditional noise estimate, from dpp_cfg_combine).
//
//   stage 0  warm-up           run the two branches serially;
//   stage 1  parallel          run them in parallel;
//   stage 2  fully connecting  serial again, to the last step.
//
// 0 -> 1 at tau1, where the discrepancy's decline has flattened: for
// `patience` consecutive steps the relative drop (prev - d) / prev stays
// below flat_tol (a rise counts as flat).  1 -> 2 at tau2, where it starts
// rising: for `patience` consecutive steps d exceeds the lowest value seen
// in the parallel stage by more than the fraction rise_tol.  The pages give
// no thresholds; these rules are the plainest reading of "the decline
// flattens" and "the discrepancy starts rising".
#include "../../include/dpp.h"

extern "C" {

void dpp_switch_init(dpp_switch_state *s, double flat_tol, double rise_tol, int patience) {
  if (!s) return;
  s->flat_tol = flat_tol;
  s->rise_tol = rise_tol;
  s->patience = patience < 1 ? 1 : patience;
  s->stage = DPP_STAGE_WARMUP;
  s->run = 0;
  s->steps = 0;
  s->prev = 0.0;
  s->min_d = 0.0;
}

int dpp_switch_update(dpp_switch_state *s, double d) {
  if (!s) return -1;
  if (!(d >= 0.0)) return s->stage;  // NaN or negative: no information, no change
  if (s->stage == DPP_STAGE_WARMUP) {
    if (s->steps > 0) {
      const double drop = s->prev > 0.0 ? (s->prev - d) / s->prev : 0.0;
      s->run = drop < s->flat_tol ? s->run + 1 : 0;
      if (s->run >= s->patience) {
        s->stage = DPP_STAGE_PARALLEL;
        s->run = 0;
        s->min_d = d;
      }
    }
  } else if (s->stage == DPP_STAGE_PARALLEL) {
    if (d < s->min_d) s->min_d = d;
    s->run = d > s->min_d * (1.0 + s->rise_tol) ? s->run + 1 : 0;
    if (s->run >= s->patience) {
      s->stage = DPP_STAGE_FULLY_CONNECTING;
      s->run = 0;
    }
  }
  s->prev = d;
  ++s->steps;
  return s->stage;
}

}  // extern "C"
