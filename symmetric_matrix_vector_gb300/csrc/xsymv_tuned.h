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
    {'s', 1, 6144, 3},   // vr1_u4_r0_w4 1739.3 GB/s at n=4096
    {'s', 1, 12288, 2},   // vr1_u2_r0_w8 3514.6 GB/s at n=8192
    {'s', 1, 20480, 2},   // vr1_u2_r0_w8 4788.7 GB/s at n=16384
    {'s', 1, 28672, 0},   // vr1_u4_r0_w8 5243.6 GB/s at n=24576
    {'s', 1, 2147483647, 0},   // vr1_u4_r0_w8 5421.6 GB/s at n=32768
    {'s', 0, 6144, 2},   // vr1_u2_r0_w8 1637.0 GB/s at n=4096
    {'s', 0, 12288, 2},   // vr1_u2_r0_w8 3198.7 GB/s at n=8192
    {'s', 0, 20480, 2},   // vr1_u2_r0_w8 4511.5 GB/s at n=16384
    {'s', 0, 28672, 2},   // vr1_u2_r0_w8 4909.5 GB/s at n=24576
    {'s', 0, 2147483647, 0},   // vr1_u4_r0_w8 5241.5 GB/s at n=32768
    {'d', 1, 16384, 3},   // vr4_u2_r0_w8 1554.6 GB/s at n=8192
    {'d', 1, 2147483647, 3},   // vr4_u2_r0_w8 1953.1 GB/s at n=24576
    {'d', 0, 16384, 3},   // vr4_u2_r0_w8 1554.1 GB/s at n=8192
    {'d', 0, 2147483647, 3},   // vr4_u2_r0_w8 1913.6 GB/s at n=24576
    {'c', 1, 12288, 2},   // vr1_u4_r0_w8 4550.8 GB/s at n=8192
    {'c', 1, 2147483647, 2},   // vr1_u4_r0_w8 5442.8 GB/s at n=16384
    {'c', 0, 12288, 2},   // vr1_u4_r0_w8 4298.1 GB/s at n=8192
    {'c', 0, 2147483647, 2},   // vr1_u4_r0_w8 5468.3 GB/s at n=16384
    {'z', 1, 12288, 0},   // vr4_u2_r0_w8 922.9 GB/s at n=8192
    {'z', 1, 2147483647, 0},   // vr4_u2_r0_w8 994.5 GB/s at n=16384
    {'z', 0, 12288, 0},   // vr4_u2_r0_w8 922.6 GB/s at n=8192
    {'z', 0, 2147483647, 0},   // vr4_u2_r0_w8 993.8 GB/s at n=16384
    {'w', 1, 6144, 4},   // vr4_u2_a4_w4 99.0 GB/s at n=4096
    {'w', 1, 2147483647, 5},   // vr4_u2_t4_w4 116.3 GB/s at n=8192
    {'w', 0, 6144, 4},   // vr4_u2_a4_w4 98.7 GB/s at n=4096
    {'w', 0, 2147483647, 5},   // vr4_u2_t4_w4 115.7 GB/s at n=8192
};
// END TUNED TABLE

inline int tuned_variant(char kind, int upper, int n) {
  for (const TunedEntry& e : kTuned)
    if (e.kind == kind && (e.upper < 0 || e.upper == upper) && n <= e.n_max) return e.variant;
  return 0;
}

}  // namespace xsymv
