"""Oracle of the adaptive draft-tree planner (test infrastructure).

Only the test suite and the CPU-baseline legs of ``bench.py`` may import this module.
It restates "Doubling LLM token rates in ComfyUI" (blog.comfy.org), section
"Adaptive tree MTP", in plain Python with fp64 arithmetic, and shares no code with
the library's planner:

- the verify pass carries the committed token and seven draft tokens; a shape is a
  chain of widths (w_1, ..., w_D), w_1 + ... + w_D = 7: at level d the head's first
  choice continues the chain, choices 2 .. w_d are sibling leaves;
- per level the planner keeps exponentially decayed counts of the rank the accepted
  token had (1 .. 7, or none), and decayed means of the draft and verify times;
- at each 32nd step all 64 shapes get a score, expected tokens per step over
  verify_ms + D * draft_ms, and the planner changes shape only for a winner at least
  3 % above the current one.

Readings where the section is silent (the same list is in include/woq_tree.h):
counts at level d change only on steps that reached level d, so the estimated
probabilities are conditional on reaching it; a level without counts contributes
nothing; a step yields the accepted draft tokens plus the verify pass's own token;
counts decay by a factor per step (default 2^(-1/64)); ties go to the first shape of
the enumeration (by the bit pattern of cuts, ascending); the first shape is the plain
chain of seven levels.
"""
from __future__ import annotations

ROWS = 7
BINS = 8  # ranks 1..7, then none


def shapes():
    """The 64 compositions of 7: shape i cuts after unit u + 1 where bit u of i is set."""
    out = []
    for mask in range(1 << (ROWS - 1)):
        parts, run = [], 0
        for unit in range(ROWS):
            run += 1
            if unit == ROWS - 1 or mask & (1 << unit):
                parts.append(run)
                run = 0
        out.append(tuple(parts))
    return out


def level_probabilities(counts):
    """p[d][b] = counts[d][b] / sum_b counts[d][b] (None for a level without counts)."""
    probs = []
    for row in counts:
        total = sum(row)
        probs.append([c / total for c in row] if total > 0 else None)
    return probs


def expected_tokens(counts, widths):
    """1 + sum over levels of P(reach level) * P(accepted token within the level's width)."""
    probs = level_probabilities(counts)
    tokens = 1.0
    reach = 1.0
    for d, w in enumerate(widths):
        p = probs[d]
        if p is None:
            break
        tokens += reach * sum(p[:w])
        reach *= p[0]
    return tokens


def score(counts, draft_ms, verify_ms, widths):
    cost = verify_ms + len(widths) * draft_ms
    return expected_tokens(counts, widths) / cost if cost > 0 else 0.0


class Planner:
    def __init__(self, decay=None, hysteresis=0.03, replan_every=32):
        self.decay = 2.0 ** (-1.0 / 64.0) if decay is None else decay
        self.hysteresis = hysteresis
        self.replan_every = replan_every
        self.counts = [[0.0] * BINS for _ in range(ROWS)]
        self.draft_ms = 0.0
        self.verify_ms = 0.0
        self.times_seen = False
        self.steps = 0
        self.shape = (1,) * ROWS

    def replan(self):
        """(index of the best shape, its score, whether the shape changed)."""
        all_shapes = shapes()
        scores = [score(self.counts, self.draft_ms, self.verify_ms, s) for s in all_shapes]
        best = 0
        for i in range(1, len(scores)):
            if scores[i] > scores[best]:
                best = i
        current = score(self.counts, self.draft_ms, self.verify_ms, self.shape)
        changed = False
        if all_shapes[best] != self.shape and scores[best] > 0 and scores[best] >= (1 + self.hysteresis) * current:
            self.shape = all_shapes[best]
            changed = True
        return best, scores[best], changed

    def observe(self, ranks, draft_ms=None, verify_ms=None):
        """ranks: accepted-token rank (1..7, 0 = none) at each level the step reached."""
        assert len(ranks) <= len(self.shape)
        for d in range(ROWS):
            for b in range(BINS):
                self.counts[d][b] *= self.decay
        for d, r in enumerate(ranks):
            self.counts[d][BINS - 1 if r == 0 else r - 1] += 1.0
        if draft_ms is not None and verify_ms is not None:
            if not self.times_seen:
                self.draft_ms, self.verify_ms, self.times_seen = draft_ms, verify_ms, True
            else:
                self.draft_ms = self.decay * self.draft_ms + (1 - self.decay) * draft_ms
                self.verify_ms = self.decay * self.verify_ms + (1 - self.decay) * verify_ms
        self.steps += 1
        if self.steps % self.replan_every == 0:
            return self.replan()[2]
        return False


def simulate_step(level_rank_probs, widths, rng):
    """One step of the drafting process of the section, sampled: at each level draw the
    accepted token's rank; a first-choice hit continues the chain, a sibling hit (rank
    2 .. w) ends it with one more token, a miss ends it.  Returns (tokens, ranks)."""
    tokens, ranks = 1, []
    for d, w in enumerate(widths):
        p = level_rank_probs[d]
        u = rng.random()
        acc, rank = 0.0, 0
        for r in range(1, ROWS + 1):
            acc += p[r - 1]
            if u < acc:
                rank = r
                break
        ranks.append(rank)
        if rank == 1:
            tokens += 1
            continue
        if 1 < rank <= w:
            tokens += 1
        break
    return tokens, ranks


def decayed_mass(decay, n):
    """Closed form of n unit observations under per-step decay, starting from zero."""
    return (1 - decay ** n) / (1 - decay) if decay != 1 else float(n)


__all__ = ["ROWS", "BINS", "shapes", "expected_tokens", "score", "Planner", "simulate_step", "decayed_mass",
           "level_probabilities"]
