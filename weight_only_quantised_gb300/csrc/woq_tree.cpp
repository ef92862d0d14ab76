// Adaptive draft-tree planner (host code; see include/woq_tree.h for the definition).
//
// "Doubling LLM token rates in ComfyUI", section "Adaptive tree MTP": decayed counts of
// the accepted token's rank per draft level, timed draft and verify phases, and every
// 32 steps a score of all 64 chains of widths that lay out seven draft rows, with a 3 %
// margin before switching.  The scoring walks each shape once, accumulating the
// probability of reaching each level, so a re-plan is 64 x 7 multiply-adds.
#include <math.h>
#include <string.h>

#include "woq_tree.h"

namespace woq {
namespace {

constexpr int kRows = WOQ_TREE_ROWS;
constexpr int kBins = WOQ_TREE_BINS;
constexpr int kNone = kBins - 1;

// widths of composition `index` of 7: bit i of index cuts after unit i + 1
int shape_of(int index, int* widths) {
  int depth = 0, w = 0;
  for (int unit = 0; unit < kRows; ++unit) {
    ++w;
    if (unit == kRows - 1 || ((index >> unit) & 1)) {
      widths[depth++] = w;
      w = 0;
    }
  }
  return depth;
}

bool valid_shape(const int* widths, int depth) {
  if (!widths || depth < 1 || depth > kRows) return false;
  int s = 0;
  for (int d = 0; d < depth; ++d) {
    if (widths[d] < 1) return false;
    s += widths[d];
  }
  return s == kRows;
}

double expected_tokens(const woq_tree_planner& p, const int* widths, int depth) {
  double reach = 1.0, tokens = 1.0;  // the verify pass always yields one token of its own
  for (int d = 0; d < depth; ++d) {
    double mass = 0.0;
    for (int b = 0; b < kBins; ++b) mass += p.counts[d][b];
    if (mass <= 0.0) break;  // no statistics for this level yet: it adds nothing
    double hit = 0.0;
    for (int r = 0; r < widths[d]; ++r) hit += p.counts[d][r];
    tokens += reach * (hit / mass);
    reach *= p.counts[d][0] / mass;
  }
  return tokens;
}

double score_of(const woq_tree_planner& p, const int* widths, int depth, double* tokens_out) {
  const double tokens = expected_tokens(p, widths, depth);
  if (tokens_out) *tokens_out = tokens;
  const double cost = p.verify_ms + depth * p.draft_ms;
  return cost > 0.0 ? tokens / cost : 0.0;
}

}  // namespace
}  // namespace woq

using namespace woq;

extern "C" {

int woq_tree_init(woq_tree_planner* p, double decay, double hysteresis, int replan_every) {
  if (!p) return WOQ_ERR_NULL;
  if (decay == 0.0) decay = exp2(-1.0 / 64.0);
  if (hysteresis < 0.0) hysteresis = 0.03;
  if (replan_every <= 0) replan_every = 32;
  if (!(decay > 0.0 && decay <= 1.0) || !(hysteresis < 10.0)) return WOQ_ERR_SHAPE;
  memset(p, 0, sizeof(*p));
  p->decay = decay;
  p->hysteresis = hysteresis;
  p->replan_every = replan_every;
  p->depth = kRows;  // the plain chain
  for (int d = 0; d < kRows; ++d) p->widths[d] = 1;
  return WOQ_OK;
}

int woq_tree_shape(int index, int* widths, int* depth) {
  if (!widths || !depth) return WOQ_ERR_NULL;
  if (index < 0 || index >= WOQ_TREE_SHAPES) return WOQ_ERR_SHAPE;
  *depth = shape_of(index, widths);
  return WOQ_OK;
}

int woq_tree_score(const woq_tree_planner* p, const int* widths, int depth, double* expected, double* score) {
  if (!p || !widths || !score) return WOQ_ERR_NULL;
  if (!valid_shape(widths, depth)) return WOQ_ERR_SHAPE;
  *score = score_of(*p, widths, depth, expected);
  return WOQ_OK;
}

int woq_tree_replan(woq_tree_planner* p, int* best_index, double* best_score, int* switched) {
  if (!p) return WOQ_ERR_NULL;
  int best = -1;
  double best_s = -1.0;
  int w[kRows];
  for (int i = 0; i < WOQ_TREE_SHAPES; ++i) {
    const int depth = shape_of(i, w);
    const double s = score_of(*p, w, depth, nullptr);
    if (s > best_s) {  // ties keep the first in enumeration order
      best_s = s;
      best = i;
    }
  }
  const double current = score_of(*p, p->widths, p->depth, nullptr);
  int sw = 0;
  int bw[kRows];
  const int bdepth = shape_of(best, bw);
  bool same = bdepth == p->depth;
  for (int d = 0; same && d < bdepth; ++d) same = bw[d] == p->widths[d];
  if (!same && best_s >= (1.0 + p->hysteresis) * current && best_s > 0.0) {
    p->depth = bdepth;
    for (int d = 0; d < kRows; ++d) p->widths[d] = d < bdepth ? bw[d] : 0;
    sw = 1;
  }
  if (best_index) *best_index = best;
  if (best_score) *best_score = best_s;
  if (switched) *switched = sw;
  return WOQ_OK;
}

int woq_tree_observe(woq_tree_planner* p, int levels_reached, const int* ranks, double draft_ms, double verify_ms,
                     int* switched) {
  if (!p) return WOQ_ERR_NULL;
  if (levels_reached < 0 || levels_reached > p->depth) return WOQ_ERR_SHAPE;
  if (levels_reached > 0 && !ranks) return WOQ_ERR_NULL;
  for (int d = 0; d < levels_reached; ++d)
    if (ranks[d] < 0 || ranks[d] > kRows || (d + 1 < levels_reached && ranks[d] != 1)) return WOQ_ERR_SHAPE;
  for (int d = 0; d < kRows; ++d)
    for (int b = 0; b < kBins; ++b) p->counts[d][b] *= p->decay;
  for (int d = 0; d < levels_reached; ++d) p->counts[d][ranks[d] == 0 ? kNone : ranks[d] - 1] += 1.0;
  if (draft_ms >= 0.0 && verify_ms >= 0.0) {
    if (!p->times_seen) {
      p->draft_ms = draft_ms;
      p->verify_ms = verify_ms;
      p->times_seen = 1;
    } else {
      p->draft_ms = p->decay * p->draft_ms + (1.0 - p->decay) * draft_ms;
      p->verify_ms = p->decay * p->verify_ms + (1.0 - p->decay) * verify_ms;
    }
  }
  ++p->steps;
  if (switched) *switched = 0;
  if (p->steps % p->replan_every == 0) return woq_tree_replan(p, nullptr, nullptr, switched);
  return WOQ_OK;
}

}  // extern "C"
