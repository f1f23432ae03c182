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
    {'s', 1, 768, "vr1_u2_r0_w8_b6_g7"},   // 47.6 GB/s at n=512
    {'s', 1, 1536, "vr2_u2_r0_w8_b4_g13_c2_f"},   // 171.6 GB/s at n=1024
    {'s', 1, 2560, "vr2_u2_r0_w8_b4_g13"},   // 565.9 GB/s at n=2048
    {'s', 1, 3584, "vr1_u2_r0_w8_b0_g9"},   // 1179.8 GB/s at n=3072
    {'s', 1, 6144, "vr1_u2_r0_w8_b6_g14"},   // 1776.0 GB/s at n=4096
    {'s', 1, 10240, "vr2_u2_r0_w8_b4_g12_c2_f"},   // 4016.5 GB/s at n=8192
    {'s', 1, 14336, "vr2_u2_r0_w8_b4_g12_c2_f"},   // 5329.5 GB/s at n=12288
    {'s', 1, 18432, "vr2_u2_r0_w8_b4_g13"},   // 6877.7 GB/s at n=16384
    {'s', 1, 22528, "vr2_u2_r0_w8_b4_g12"},   // 6891.1 GB/s at n=20480
    {'s', 1, 26624, "vr2_u2_r0_w8_b4_g12"},   // 6905.8 GB/s at n=24576
    {'s', 1, 30720, "vr2_u2_r0_w8_b4_g11"},   // 6941.3 GB/s at n=28672
    {'s', 1, 2147483647, "vr2_u2_r0_w8_b4_g13"},   // 6975.5 GB/s at n=32768
    {'s', 0, 768, "vr1_u2_r0_w8"},   // 48.5 GB/s at n=512
    {'s', 0, 1536, "vr1_u2_r0_w8_b6_g14_c2_f"},   // 173.3 GB/s at n=1024
    {'s', 0, 2560, "vr1_u2_r0_w8_b0_g9"},   // 628.4 GB/s at n=2048
    {'s', 0, 3584, "vr1_u2_r0_w8_b0_g9"},   // 1260.0 GB/s at n=3072
    {'s', 0, 6144, "vr1_u2_r0_w8_b6_g11"},   // 1844.0 GB/s at n=4096
    {'s', 0, 10240, "vr2_u2_r0_w8_b4_g12_c2_f"},   // 4005.0 GB/s at n=8192
    {'s', 0, 14336, "vr2_u2_r0_w8_b4_g11_c2_f"},   // 5376.3 GB/s at n=12288
    {'s', 0, 18432, "vr2_u2_r0_w8_b4_g13"},   // 6843.5 GB/s at n=16384
    {'s', 0, 22528, "vr2_u2_r0_w8_b4_g12"},   // 6863.3 GB/s at n=20480
    {'s', 0, 26624, "vr2_u2_r0_w8_b4_g12"},   // 6923.8 GB/s at n=24576
    {'s', 0, 30720, "vr2_u2_r0_w8_b4_g12"},   // 6951.2 GB/s at n=28672
    {'s', 0, 2147483647, "vr2_u2_r0_w8_b4_g13"},   // 6975.4 GB/s at n=32768
    {'d', 1, 1536, "vr4_u2_r0_w8_b0_g6"},   // 245.6 GB/s at n=1024
    {'d', 1, 3072, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 680.6 GB/s at n=2048
    {'d', 1, 6144, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 1320.2 GB/s at n=4096
    {'d', 1, 12288, "vr4_u2_r0_w8_b0_g6_c8_f"},   // 1871.8 GB/s at n=8192
    {'d', 1, 20480, "vr4_u2_r0_w8_b0_g5_c8"},   // 2179.7 GB/s at n=16384
    {'d', 1, 2147483647, "vr4_u2_r0_w8_b0_g5_c8"},   // 2214.4 GB/s at n=24576
    {'d', 0, 1536, "vr4_u2_r0_w8_b0_g6_c8"},   // 248.3 GB/s at n=1024
    {'d', 0, 3072, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 687.7 GB/s at n=2048
    {'d', 0, 6144, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 1315.8 GB/s at n=4096
    {'d', 0, 12288, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 1889.4 GB/s at n=8192
    {'d', 0, 20480, "vr4_u2_r0_w8_b0_g5_c8"},   // 2178.4 GB/s at n=16384
    {'d', 0, 2147483647, "vr4_u2_r0_w8_b0_g5_c8"},   // 2214.4 GB/s at n=24576
    {'c', 1, 1536, "vr2_u2_r0_w8_b4_g13_c2_f"},   // 321.2 GB/s at n=1024
    {'c', 1, 3072, "vr2_u2_r0_w8_b4_g10"},   // 1015.3 GB/s at n=2048
    {'c', 1, 6144, "vr2_u2_r0_w8_b4_g13_c2_f"},   // 2929.4 GB/s at n=4096
    {'c', 1, 12288, "vr2_u2_r0_w8_b4_g13_c2_f"},   // 5151.3 GB/s at n=8192
    {'c', 1, 2147483647, "vr2_u2_r0_w8_b4_g13"},   // 6854.2 GB/s at n=16384
    {'c', 0, 1536, "vr2_u2_r0_w8_b4_g13"},   // 328.4 GB/s at n=1024
    {'c', 0, 3072, "vr2_u2_r0_w8_b0_g7"},   // 1054.5 GB/s at n=2048
    {'c', 0, 6144, "vr2_u2_r0_w8_b4_g11"},   // 2899.9 GB/s at n=4096
    {'c', 0, 12288, "vr2_u2_r0_w8_b4_g10"},   // 5130.6 GB/s at n=8192
    {'c', 0, 2147483647, "vr2_u2_r0_w8_b4_g13"},   // 6858.4 GB/s at n=16384
    {'z', 1, 1536, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 333.4 GB/s at n=1024
    {'z', 1, 3072, "vr4_u2_r0_w8_b0_g6_c8_f"},   // 630.5 GB/s at n=2048
    {'z', 1, 6144, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 920.2 GB/s at n=4096
    {'z', 1, 12288, "vr4_u2_r0_w8_b0_g5_c8"},   // 1099.4 GB/s at n=8192
    {'z', 1, 2147483647, "vr4_u2_r0_w8_b0_g5_c8"},   // 1119.9 GB/s at n=16384
    {'z', 0, 1536, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 338.7 GB/s at n=1024
    {'z', 0, 3072, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 630.2 GB/s at n=2048
    {'z', 0, 6144, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 927.4 GB/s at n=4096
    {'z', 0, 12288, "vr4_u2_r0_w8_b0_g5_c8"},   // 1101.4 GB/s at n=8192
    {'z', 0, 2147483647, "vr4_u2_r0_w8_b0_g4_c8"},   // 1122.8 GB/s at n=16384
    {'w', 1, 1536, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 89.0 GB/s at n=1024
    {'w', 1, 3072, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 132.3 GB/s at n=2048
    {'w', 1, 6144, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 160.6 GB/s at n=4096
    {'w', 1, 2147483647, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 168.9 GB/s at n=8192
    {'w', 0, 1536, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 88.3 GB/s at n=1024
    {'w', 0, 3072, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 132.4 GB/s at n=2048
    {'w', 0, 6144, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 160.6 GB/s at n=4096
    {'w', 0, 2147483647, "vr4_u2_r0_w8_b0_g5_c8_f"},   // 168.8 GB/s at n=8192
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
