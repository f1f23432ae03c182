// Kernel-variant choice per (kind, uplo, n).  Written by the offline tuner
// (symmetric_matrix_vector_gb300/tune.py) from timings on GB300; an entry
// applies to every n up to and including n_max, the first match wins.
#pragma once

namespace xsymv {

struct TunedEntry {
  char kind;
  int upper;   // 1 'U', 0 'L', -1 either
  int n_max;
  int variant;
};

// BEGIN TUNED TABLE
static const TunedEntry kTuned[] = {
    {'s', -1, 2147483647, 0},
    {'d', -1, 2147483647, 0},
    {'c', -1, 2147483647, 0},
    {'z', -1, 2147483647, 0},
    {'w', -1, 2147483647, 0},
};
// END TUNED TABLE

inline int tuned_variant(char kind, int upper, int n) {
  for (const TunedEntry& e : kTuned)
    if (e.kind == kind && (e.upper < 0 || e.upper == upper) && n <= e.n_max) return e.variant;
  return 0;
}

}  // namespace xsymv
