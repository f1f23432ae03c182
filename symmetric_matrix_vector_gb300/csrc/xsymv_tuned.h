// Kernel-variant choice per (kind, uplo, n).  Written by the offline tuner
// (symmetric_matrix_vector_gb300/tune.py) from timings on GB300; an entry
// applies to every n up to and including n_max, the first match wins.  Each
// entry names its variant; the name is looked up in the kind's compiled
// variant list when the entry is first used, so inserting or removing a
// variant cannot silently retarget an entry.
#pragma once

namespace xsymv {

struct TunedEntry {
  char kind;
  int upper;   // 1 'U', 0 'L', -1 either
  int n_max;
  const char* variant;   // variant name ("vr..._w..."), as xsymv_variant_name reports it
};

// BEGIN TUNED TABLE
static const TunedEntry kTuned[] = {
    {'s', 1, 6144, "vr1_u2_r0_w8_b6_g11"},   // 1978.9 GB/s at n=4096
    {'s', 1, 10240, "vr2_u2_r0_w8_b4_g12"},   // 4006.5 GB/s at n=8192
    {'s', 1, 14336, "vr2_u2_r0_w8_b4_g11"},   // 5338.2 GB/s at n=12288
    {'s', 1, 18432, "vr2_u2_r0_w8_b4_g11"},   // 6161.7 GB/s at n=16384
    {'s', 1, 22528, "vr2_u2_r0_w8_b4_g12"},   // 6451.4 GB/s at n=20480
    {'s', 1, 26624, "vr2_u2_r0_w8_b4_g12"},   // 6536.7 GB/s at n=24576
    {'s', 1, 30720, "vr2_u2_r0_w8_b4_g11"},   // 6697.5 GB/s at n=28672
    {'s', 1, 2147483647, "vr2_u2_r0_w8_b4_g11"},   // 6768.2 GB/s at n=32768
    {'s', 0, 6144, "vr2_u2_r0_w8_b4_g12"},   // 1982.7 GB/s at n=4096
    {'s', 0, 10240, "vr2_u2_r0_w8_b4_g13"},   // 4029.6 GB/s at n=8192
    {'s', 0, 14336, "vr2_u2_r0_w8_b4_g11"},   // 5394.7 GB/s at n=12288
    {'s', 0, 18432, "vr2_u2_r0_w8_b4_g13"},   // 6171.4 GB/s at n=16384
    {'s', 0, 22528, "vr2_u2_r0_w8_b4_g11"},   // 6437.5 GB/s at n=20480
    {'s', 0, 26624, "vr2_u2_r0_w8_b4_g12"},   // 6588.4 GB/s at n=24576
    {'s', 0, 30720, "vr2_u2_r0_w8_b4_g12"},   // 6724.5 GB/s at n=28672
    {'s', 0, 2147483647, "vr2_u2_r0_w8_b4_g11"},   // 6809.4 GB/s at n=32768
    {'d', 1, 12288, "vr4_u2_r0_w8_b0_g5_c8"},   // 1817.5 GB/s at n=8192
    {'d', 1, 20480, "vr4_u2_r0_w8_b0_g5_c8"},   // 2120.0 GB/s at n=16384
    {'d', 1, 2147483647, "vr4_u2_r0_w8_b0_g5_c8"},   // 2170.6 GB/s at n=24576
    {'d', 0, 12288, "vr4_u2_r0_w8_b0_g5_c8"},   // 1840.6 GB/s at n=8192
    {'d', 0, 20480, "vr4_u2_r0_w8_b0_g5_c8"},   // 2116.3 GB/s at n=16384
    {'d', 0, 2147483647, "vr4_u2_r0_w8_b0_g5_c8"},   // 2175.2 GB/s at n=24576
    {'c', 1, 12288, "vr2_u2_r0_w8_b4_g13"},   // 5198.0 GB/s at n=8192
    {'c', 1, 2147483647, "vr2_u2_r0_w8_b4_g13"},   // 6447.7 GB/s at n=16384
    {'c', 0, 12288, "vr2_u2_r0_w8_b4_g11"},   // 5207.7 GB/s at n=8192
    {'c', 0, 2147483647, "vr2_u2_r0_w8_b4_g11"},   // 6536.5 GB/s at n=16384
    {'z', 1, 12288, "vr4_u2_r0_w8_b0_g5_c8"},   // 1060.8 GB/s at n=8192
    {'z', 1, 2147483647, "vr4_u2_r0_w8_b0_g5_c8"},   // 1096.4 GB/s at n=16384
    {'z', 0, 12288, "vr4_u2_r0_w8_b0_g5_c8"},   // 1061.0 GB/s at n=8192
    {'z', 0, 2147483647, "vr4_u2_r0_w8_b0_g4_c8"},   // 1101.6 GB/s at n=16384
    {'w', 1, 6144, "vr4_u2_r0_w8_b0_g4_c8"},   // 120.0 GB/s at n=4096
    {'w', 1, 2147483647, "vr8_u1_r0_w4_b0_g6_c8"},   // 132.2 GB/s at n=8192
    {'w', 0, 6144, "vr4_u2_r0_w8_b0_g4_c8"},   // 119.6 GB/s at n=4096
    {'w', 0, 2147483647, "vr8_u1_r0_w4_b0_g6_c8"},   // 132.2 GB/s at n=8192
};
// END TUNED TABLE

constexpr int kTunedCount = (int)(sizeof(kTuned) / sizeof(kTuned[0]));

// index into kTuned of the entry for (kind, upper, n), -1 if none
inline int tuned_entry(char kind, int upper, int n) {
  for (int i = 0; i < kTunedCount; ++i) {
    const TunedEntry& e = kTuned[i];
    if (e.kind == kind && (e.upper < 0 || e.upper == upper) && n <= e.n_max) return i;
  }
  return -1;
}

}  // namespace xsymv
