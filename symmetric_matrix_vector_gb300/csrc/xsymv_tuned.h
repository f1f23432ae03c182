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
    {'s', 1, 6144, 1},   // vr1_u2_r0_w8 1814.5 GB/s at n=4096
    {'s', 1, 12288, 0},   // vr1_u4_r0_w8 3617.0 GB/s at n=8192
    {'s', 1, 20480, 11},   // vr1_u2_r0_w8_b6_g7 5338.3 GB/s at n=16384
    {'s', 1, 28672, 11},   // vr1_u2_r0_w8_b6_g7 5956.3 GB/s at n=24576
    {'s', 1, 2147483647, 7},   // vr1_u2_r0_w8_b6 6100.1 GB/s at n=32768
    {'s', 0, 6144, 3},   // vr1_u4_r0_w4 1811.4 GB/s at n=4096
    {'s', 0, 12288, 11},   // vr1_u2_r0_w8_b6_g7 3621.1 GB/s at n=8192
    {'s', 0, 20480, 11},   // vr1_u2_r0_w8_b6_g7 5398.0 GB/s at n=16384
    {'s', 0, 28672, 7},   // vr1_u2_r0_w8_b6 5758.0 GB/s at n=24576
    {'s', 0, 2147483647, 11},   // vr1_u2_r0_w8_b6_g7 6132.9 GB/s at n=32768
    {'d', 1, 16384, 10},   // vr2_u4_r0_w8_b0_g5 1721.7 GB/s at n=8192
    {'d', 1, 2147483647, 8},   // vr4_u2_r0_w8_b0_g5 1978.2 GB/s at n=24576
    {'d', 0, 16384, 10},   // vr2_u4_r0_w8_b0_g5 1714.6 GB/s at n=8192
    {'d', 0, 2147483647, 8},   // vr4_u2_r0_w8_b0_g5 1976.2 GB/s at n=24576
    {'c', 1, 12288, 9},   // vr1_u4_r0_w8_b0_g7 4798.9 GB/s at n=8192
    {'c', 1, 2147483647, 10},   // vr2_u2_r0_w8_b0_g7 6057.9 GB/s at n=16384
    {'c', 0, 12288, 9},   // vr1_u4_r0_w8_b0_g7 4838.8 GB/s at n=8192
    {'c', 0, 2147483647, 10},   // vr2_u2_r0_w8_b0_g7 6069.8 GB/s at n=16384
    {'z', 1, 12288, 7},   // vr4_u2_r0_w8_b0_g5 968.3 GB/s at n=8192
    {'z', 1, 2147483647, 6},   // vr4_u2_r0_w8_b0_g4 1004.5 GB/s at n=16384
    {'z', 0, 12288, 7},   // vr4_u2_r0_w8_b0_g5 968.1 GB/s at n=8192
    {'z', 0, 2147483647, 6},   // vr4_u2_r0_w8_b0_g4 1005.9 GB/s at n=16384
    {'w', 1, 6144, 5},   // vr4_u2_r0_w8_b0_g4 106.3 GB/s at n=4096
    {'w', 1, 2147483647, 5},   // vr4_u2_r0_w8_b0_g4 118.6 GB/s at n=8192
    {'w', 0, 6144, 5},   // vr4_u2_r0_w8_b0_g4 106.8 GB/s at n=4096
    {'w', 0, 2147483647, 5},   // vr4_u2_r0_w8_b0_g4 118.6 GB/s at n=8192
};
// END TUNED TABLE

inline int tuned_variant(char kind, int upper, int n) {
  for (const TunedEntry& e : kTuned)
    if (e.kind == kind && (e.upper < 0 || e.upper == upper) && n <= e.n_max) return e.variant;
  return 0;
}

}  // namespace xsymv
