// spec.cpp -- host side of speculative decoding without a draft model.
//
// "Writing an LLM inference engine from scratch in Rust", "Speculative decoding without
// a draft model": guesses come from the context itself (prompt lookup): the last few
// tokens are looked up earlier in the context, and whatever followed that earlier
// occurrence is proposed; up to 4 tokens are checked in one batched pass, kept up to the
// first the model disagrees with.  Two refinements from the same section: a match must
// be at least 2 tokens long, and an acceptance gate pauses speculation while guesses
// keep failing.
#include <cstdint>
#include <cstring>

#include "../../include/mie.h"

namespace mie {
mie_status fail(mie_status s, const char *fmt, ...);
}

// The tokens that followed the most recent earlier occurrence of the context's last g
// tokens, for the longest g in [min_ngram, max_ngram] that occurs earlier (the earlier
// occurrence must end before the last g tokens begin); at most k of them, never past the
// end of the context.  Returns how many were written to out (0: no match).
extern "C" int mie_lookup_propose(const int32_t *ids, int n, int min_ngram, int max_ngram, int k, int32_t *out) {
  if (!ids || !out || n < 1 || k < 1 || min_ngram < 1 || max_ngram < min_ngram) return 0;
  const int g_hi = max_ngram < n ? max_ngram : n;
  for (int g = g_hi; g >= min_ngram; --g) {
    const int32_t *suffix = ids + (n - g);
    for (int start = n - 2 * g; start >= 0; --start) {
      if (std::memcmp(ids + start, suffix, sizeof(int32_t) * (size_t)g) != 0) continue;
      const int from = start + g;
      int cnt = n - from < k ? n - from : k;
      for (int j = 0; j < cnt; ++j) out[j] = ids[from + j];
      return cnt;
    }
  }
  return 0;
}

// Acceptance gate: the acceptance of the last `window` attempts (accepted / proposed
// guesses); when a full window falls below `threshold`, speculation pauses for the
// current pause length and that length doubles, up to `pause_max`; once a full window is
// back at or above the threshold, the length returns to `pause`.  READING: the window
// keeps its attempts across a pause, so an attempt right after a pause that leaves the
// rate below the threshold starts the next, doubled, pause ("each consecutive pause
// doubles").
struct mie_spec_gate {
  int window, pause, pause_max;
  float threshold;
  int hist_acc[64], hist_prop[64];
  int n_hist, head;
  int paused_for;   // passes still to skip
  int next_pause;   // length of the next pause
};

extern "C" size_t mie_spec_gate_bytes(void) { return sizeof(mie_spec_gate); }

extern "C" void mie_spec_gate_init(mie_spec_gate *g, int window, float threshold, int pause, int pause_max) {
  std::memset(g, 0, sizeof *g);
  g->window = window < 1 ? 1 : (window > 64 ? 64 : window);
  g->threshold = threshold;
  g->pause = pause < 0 ? 0 : pause;
  g->pause_max = pause_max < g->pause ? g->pause : pause_max;
  g->next_pause = g->pause;
}

// 1 when this pass may speculate; a paused gate counts the pass off.
extern "C" int mie_spec_gate_open(mie_spec_gate *g) {
  if (g->paused_for > 0) {
    --g->paused_for;
    return 0;
  }
  return 1;
}

// Records one attempt: `proposed` > 0 guesses, `accepted` of them kept.
extern "C" void mie_spec_gate_record(mie_spec_gate *g, int proposed, int accepted) {
  if (proposed <= 0) return;
  g->hist_prop[g->head] = proposed;
  g->hist_acc[g->head] = accepted;
  g->head = (g->head + 1) % g->window;
  if (g->n_hist < g->window) ++g->n_hist;
  if (g->n_hist < g->window) return;
  long p = 0, a = 0;
  for (int i = 0; i < g->window; ++i) {
    p += g->hist_prop[i];
    a += g->hist_acc[i];
  }
  if ((float)a < g->threshold * (float)p) {
    g->paused_for = g->next_pause;
    g->next_pause = g->next_pause * 2 > g->pause_max ? g->pause_max : g->next_pause * 2;
  } else {
    g->next_pause = g->pause;
  }
}
