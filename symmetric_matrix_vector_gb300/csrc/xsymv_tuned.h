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
    {'s', 1, 6144, 2},   // vr1_u8_r0_w8 1630.7 GB/s at n=4096
    {'s', 1, 12288, 7},   // vr1_u2_r0_w8_b6 3263.3 GB/s at n=8192
    {'s', 1, 20480, 7},   // vr1_u2_r0_w8_b6 4623.0 GB/s at n=16384
    {'s', 1, 28672, 7},   // vr1_u2_r0_w8_b6 5293.2 GB/s at n=24576
    {'s', 1, 2147483647, 7},   // vr1_u2_r0_w8_b6 5531.1 GB/s at n=32768
    {'s', 0, 6144, 3},   // vr1_u4_r0_w4 1541.7 GB/s at n=4096
    {'s', 0, 12288, 7},   // vr1_u2_r0_w8_b6 3248.5 GB/s at n=8192
    {'s', 0, 20480, 1},   // vr1_u2_r0_w8 4480.8 GB/s at n=16384
    {'s', 0, 28672, 7},   // vr1_u2_r0_w8_b6 5492.8 GB/s at n=24576
    {'s', 0, 2147483647, 7},   // vr1_u2_r0_w8_b6 5769.9 GB/s at n=32768
    {'d', 1, 16384, 1},   // vr2_u4_r0_w8 1633.1 GB/s at n=8192
    {'d', 1, 2147483647, 0},   // vr4_u2_r0_w8 1971.9 GB/s at n=24576
    {'d', 0, 16384, 1},   // vr2_u4_r0_w8 1630.5 GB/s at n=8192
    {'d', 0, 2147483647, 0},   // vr4_u2_r0_w8 1974.4 GB/s at n=24576
    {'c', 1, 12288, 5},   // vr1_u2_r0_w8_b5 4463.6 GB/s at n=8192
    {'c', 1, 2147483647, 0},   // vr1_u4_r0_w8 5572.3 GB/s at n=16384
    {'c', 0, 12288, 0},   // vr1_u4_r0_w8 4478.8 GB/s at n=8192
    {'c', 0, 2147483647, 0},   // vr1_u4_r0_w8 5672.8 GB/s at n=16384
    {'z', 1, 12288, 0},   // vr4_u2_r0_w8 956.8 GB/s at n=8192
    {'z', 1, 2147483647, 0},   // vr4_u2_r0_w8 1005.2 GB/s at n=16384
    {'z', 0, 12288, 0},   // vr4_u2_r0_w8 951.8 GB/s at n=8192
    {'z', 0, 2147483647, 0},   // vr4_u2_r0_w8 1004.8 GB/s at n=16384
    {'w', 1, 6144, 0},   // vr4_u2_r0_w8 107.8 GB/s at n=4096
    {'w', 1, 2147483647, 0},   // vr4_u2_r0_w8 118.9 GB/s at n=8192
    {'w', 0, 6144, 0},   // vr4_u2_r0_w8 107.8 GB/s at n=4096
    {'w', 0, 2147483647, 0},   // vr4_u2_r0_w8 119.0 GB/s at n=8192
};
// END TUNED TABLE

inline int tuned_variant(char kind, int upper, int n) {
  for (const TunedEntry& e : kTuned)
    if (e.kind == kind && (e.upper < 0 || e.upper == upper) && n <= e.n_max) return e.variant;
  return 0;
}

}  // namespace xsymv
