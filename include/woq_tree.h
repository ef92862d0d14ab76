/* Adaptive draft-tree planner for multi-token-prediction verification.
 *
 * "Doubling LLM token rates in ComfyUI" (blog.comfy.org), section "Adaptive tree
 * MTP": the verify pass carries eight rows (the committed token and seven draft
 * tokens).  At each draft level the head's top choice continues the chain and a
 * few runner-up choices are kept as sibling leaves; the shape of the tree is a
 * chain of widths w_1 .. w_D with w_1 + ... + w_D = 7 (the 64 compositions of 7).
 * The planner keeps exponentially decayed counts of the rank the accepted token
 * had at each level (first choice, second, ..., seventh, or none) and measured
 * durations of the draft and verify phases; at each 32nd step it scores every
 * shape by
 *
 *     expected tokens per step / (verify_ms + D * draft_ms)
 *
 * switching only when the best shape beats the current one by at least 3 %.
 *
 * Readings where the section is silent (stated here, kept by the oracle):
 *   - counts at level d are updated only on steps whose chain reached level d
 *     (levels 1 .. d-1 accepted their first choice), so p_d(r) = c_d[r] / sum_r'
 *     c_d[r'] over the 8 bins is a conditional probability; a level with no mass
 *     yet has p_d(r) = 0;
 *   - expected tokens of shape w: 1 + sum_d P_d * sum_{r <= w_d} p_d(r), P_1 = 1,
 *     P_{d+1} = P_d * p_d(1): a hit on a sibling ends the step, and the verify pass
 *     always yields one token of its own;
 *   - decayed counts: c <- decay * c + observation each step; the phase times are
 *     decayed means with the same factor (default decay 2^(-1/64), a 64-step
 *     half-life);
 *   - ties between shapes go to the first in the enumeration order (w_1 first, a
 *     composition listed by its bit pattern of cuts, ascending);
 *   - the first shape is the plain chain (1, 1, 1, 1, 1, 1, 1).
 * Host code only: no GPU, no allocation, plain C structs owned by the caller.
 */
#ifndef WOQ_TREE_H
#define WOQ_TREE_H

#include <stddef.h>
#include <stdint.h>

#include "woq.h"

#ifdef __cplusplus
extern "C" {
#endif

#define WOQ_TREE_ROWS 7   /* draft rows per verify pass (eight rows with the committed token) */
#define WOQ_TREE_BINS 8   /* accepted-token rank 1..7, or none */
#define WOQ_TREE_SHAPES 64

typedef struct {
  double counts[WOQ_TREE_ROWS][WOQ_TREE_BINS]; /* decayed rank counts per level; bin 7 = none */
  double draft_ms;                              /* decayed mean time of one draft level */
  double verify_ms;                             /* decayed mean time of one verify pass */
  double decay;                                 /* per-step decay factor in (0, 1] */
  double hysteresis;                            /* switch when best >= (1 + hysteresis) * current */
  int replan_every;                             /* steps between re-plans */
  int steps;                                    /* observed steps */
  int times_seen;                               /* whether phase times have been observed */
  int widths[WOQ_TREE_ROWS];                    /* current shape: widths of levels 1..depth */
  int depth;                                    /* number of levels of the current shape */
} woq_tree_planner;

/* Start a planner: decay (0 = default 2^(-1/64)), hysteresis (< 0 = default 0.03),
 * replan_every (<= 0 = default 32).  WOQ_ERR_NULL / WOQ_ERR_SHAPE on bad arguments. */
WOQ_API int woq_tree_init(woq_tree_planner* p, double decay, double hysteresis, int replan_every);

/* The i-th shape (0 <= i < 64) of the enumeration: widths[0 .. *depth - 1], sum 7. */
WOQ_API int woq_tree_shape(int index, int* widths, int* depth);

/* Expected tokens per step and score (tokens / (verify_ms + depth draft_ms)) of a
 * shape under the planner's statistics.  score is 0 when the cost is not positive. */
WOQ_API int woq_tree_score(const woq_tree_planner* p, const int* widths, int depth, double* expected_tokens,
                           double* score);

/* One step's outcome.  levels_reached: how many levels were verified against
 * (1 + the number of leading first-choice hits, at most the current depth);
 * ranks[d] (d < levels_reached): rank 1..7 of the accepted token among the head's
 * candidates at level d + 1, or 0 for none.  draft_ms / verify_ms: this step's
 * measured phase times (< 0: not measured).  Every replan_every steps the planner
 * re-plans; *switched (may be NULL) tells whether the shape changed. */
WOQ_API int woq_tree_observe(woq_tree_planner* p, int levels_reached, const int* ranks, double draft_ms,
                             double verify_ms, int* switched);

/* Re-plan now: score all 64 shapes, adopt the best if it beats the current shape
 * by the hysteresis margin.  Writes the best shape's index and score. */
WOQ_API int woq_tree_replan(woq_tree_planner* p, int* best_index, double* best_score, int* switched);

#ifdef __cplusplus
}
#endif

#endif /* WOQ_TREE_H */
