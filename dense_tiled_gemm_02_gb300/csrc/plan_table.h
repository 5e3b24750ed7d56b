// plan_table.h -- per-shape choice of tile width, raster group, split-K and
// operand swap.
//
// The selection key is the whole problem (M, N, K, operand type, layouts):
// a key that leaves out a dimension silently serves a tile tuned for another
// shape ("Tuning Triton" skill page, section 3, where a decode shape reusing
// the square-shape tile ran several times slower).  Rows of kTable come from
// the measured sweep of the tuning script (dense_tiled_gemm_02_gb300/tune.py); shapes without
// a row fall back to the rules in choose_plan(), which follow the regime
// split of that page's section 4 (skinny shapes get their own candidates).
#pragma once

#include <cstdint>

#include "common.h"

namespace gb300 {

struct PlanChoice {
  int bn;        // output tile width (64, 128 or 256); tile height is BM = 128
  int group_m;   // GROUP_M of the grouped raster
  int splits;    // split-K factor (1 = none)
  int swap;      // 1: compute D^T = B^T A^T (long dimension on the tensor-core M side)
  int max_ctas;  // 0 = one CTA per SM
  int pair;      // 1: CTA-pair kernel (cta_group::2), tile 256 x bn
  int ksub;      // pair kernel: 64-wide K slices per ring stage (1 or 2)
  int tail;      // pair kernel: stream-K hybrid for a partial last wave
  int no_decode; // 1: never take the decode kernel (M <= 16, K-contiguous B)
  int no_dbulk;  // 1: never take the decode kernel's bulk-copy form; -1: take it
                 // whenever the operands allow, whatever N (0: the planner decides)
  int native_i8; // int8: 1 runs the native integer mma.sync kernel instead of the
                 // exact bf16 emulation on the tcgen05 tensor cores
  int sk;        // single-CTA kernel: stream-K over all SMs, shared tiles finished
                 // in the kernel by their last piece (no split-K reduce launch)
  int kgroup;    // single-CTA kernel: consecutive K slices loaded together (0 = 1)
  int lsu;       // 16-bit operand rows off the 16-byte grid: 1 loads them with the
                 // single-CTA kernel's producer warps instead of a workspace copy
  int i8chunk;   // exact int8: K of one exact fp32 accumulation pass, a multiple of
                 // 64 up to 960 (0 = the default)
  int dmma;      // decode regime: 1 takes the tensor-core (mma.sync) form whenever
                 // the shape allows, -1 never, 0 the planner decides
  int csk;       // single-CTA kernel with split-K: 1 adds the splits' sums through the
                 // shared memory of a cluster of split CTAs instead of a reduce launch
  int skpat;     // pair kernel stream-K: -1 keeps equal runs where the chained layout
                 // would apply (0: chains where they apply)
};

struct PlanRow {
  int64_t M, N, K;
  int ab_type, layout_a, layout_b;  // -1 = any
  PlanChoice choice;
};

// Measured rows (exact shape match), from interleaved sweeps of the tuning
// script on one GB300 (median of 5 repeats; the figures are TFLOP/s or TOPS
// of the whole call).  Layouts: 0 = row-major, 1 = column-major; types as in
// common.h.
static const PlanRow kTable[] = {
    // 4096^3 bf16, B column-major: pair 256x256 with the stream-K hybrid
    // 1605, without 1579; 2 K slices per stage 1495; GROUP_M 4 / 16 within
    // 1 % of 8.  Stream-K runs in chains (at most two pieces a run): 1666
    // against 1594 with equal runs (PyTorch's GEMM 1602 on the same box).
    {4096, 4096, 4096, T_BF16, 0, 1, {256, 8, 1, 0, 0, 1, 1, 1}},
    // 4096^3 E4M3 (A row, B column-major): pair 256x224, whose 16 x 19 tiles
    // are exactly four waves of the 76 pairs (no stream-K pieces): 2507
    // TFLOPS against 2432 for 256x256 with the stream-K hybrid (cuBLAS
    // 2442).  At bf16 the 224-wide tile measured slower (1514 against 1593):
    // a 224-column MMA took as long as a 256-column one there.
    {4096, 4096, 4096, T_E4M3, 0, 1, {224, 8, 1, 0, 0, 1, 1, 1}},
    // 8192^3 bf16, B column-major: pair 256x256 with stream-K 1940, without
    // 1913; pair 256x128 1099 (1453 with 2 K slices per stage); single-CTA
    // 128x256 1486.
    {8192, 8192, 8192, T_BF16, 0, 1, {256, 8, 1, 0, 0, 1, 1, 1}},
    // 8192^3 int8: pair 256x256 1209; with 2 K slices per stage 1184;
    // single-CTA 128x128 858 (512-K exact passes).  With 960-K passes (the
    // default since): 1591, GROUP_M 16 1567, 768-K passes 1568.  Stream-K
    // pieces for the partial last wave (13.47 waves; int32 partials, chained
    // runs): 742-748 us against 749-753 without and 761 with equal runs
    // (one box, two interleaved sweeps; the spreads were 4 %).
    {8192, 8192, 8192, T_I8, 0, 0, {256, 8, 1, 0, 0, 1, 1, 1}},
    // (64, 8192, 8192) bf16, all row-major: 128x128 tiles, split 2: 246;
    // 128x256 split 4: 241; swapped 128x64 split 4: 230, split 2: 211.
    // The two splits of a tile reduced within their cluster (csk): 232
    // against 226 with the reduce launch (128x128 unsplit: 149).
    {64, 8192, 8192, T_BF16, 0, 0, {128, 8, 2, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1}},
    // (8192, 128, 4096) bf16: 128x64 tiles, no split: 370; 128x128 no
    // split: 319, split 2: 286; pair 256x128 split 4: 260.  128x128 with
    // two splits reduced within their cluster: 347 against 291 for 128x64
    // unsplit on the same box (the K loops of the 128 CTAs stream A at
    // 5.3 TB/s; 128x64 tiles read each A row twice).
    {8192, 128, 4096, T_BF16, 0, 0, {128, 8, 2, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1}},
    // Decode shapes the CUDA-core decode kernel does not take (16 rows, or
    // an N-contiguous B): the long N on the tensor-core M side (swap),
    // 128x64 tiles, K split 4 ways and reduced by the reduce kernel.
    // 16x4096x4096, B K-contiguous: 16.3-16.9 us; the same splits reduced
    // within a cluster 24.9 (the split-0 CTA's strided epilogue), 2 splits
    // 21.9, unswapped 20.0-30.1, the mma.sync decode form 23.1, cuBLAS 29-31.
    {16, 4096, 4096, T_BF16, 0, 1, {64, 8, 4, 1, 0, 0, 1, 0}},
    // 16x4096x4096, B N-contiguous: 16.3-16.8 us; cluster split 25.2, 2
    // splits 22.9, unswapped 20.0-31.9, the mma.sync form 46.7, cuBLAS 28.
    {16, 4096, 4096, T_BF16, 0, 0, {64, 8, 4, 1, 0, 0, 1, 0}},
    // 1x4096x4096, B N-contiguous: 15.6-16.2 us; cluster split 24.8, the
    // mma.sync form 20.7, cuBLAS 31.9.
    {1, 4096, 4096, T_BF16, 0, 0, {64, 8, 4, 1, 0, 0, 1, 0}},
    // (1000, 1000, 1000) bf16: 128x64: 130; 128x128: 104; pair: 105 / 84.
    {1000, 1000, 1000, T_BF16, 0, 0, {64, 8, 1, 0, 0, 0, 1, 0}},
    // 1024^3 fp16: 128x64: 202; 128x128: 174; pair 256x128: 168.
    {1024, 1024, 1024, T_F16, 0, 0, {64, 8, 1, 0, 0, 0, 1, 0}},
};

inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline PlanChoice choose_plan(int64_t M, int64_t N, int64_t K, int ab_type, int layout_a,
                              int layout_b, int num_sms) {
  for (const PlanRow& r : kTable) {
    if (r.M == M && r.N == N && r.K == K && (r.ab_type < 0 || r.ab_type == ab_type) &&
        (r.layout_a < 0 || r.layout_a == layout_a) && (r.layout_b < 0 || r.layout_b == layout_b))
      return r.choice;
  }
  PlanChoice c{256, 8, 1, 0, 0, 0, 1, 1, 0};
  // Skinny M: put the long N dimension on the 128-row tensor-core side.
  if (M < 128 && N >= 2 * M) c.swap = 1;
  const int64_t Mi = c.swap ? N : M;
  const int64_t Ni = c.swap ? M : N;
  // Tile width: the widest tile that still gives every SM a tile, else the
  // one with the most tiles in flight.
  const int64_t tm = cdiv64(Mi, 128);
  if (Ni <= 64) c.bn = 64;
  else if (Ni <= 128) c.bn = 128;
  else if (tm * cdiv64(Ni, 256) >= num_sms) c.bn = 256;
  else if (tm * cdiv64(Ni, 128) >= num_sms / 2) c.bn = 128;
  else c.bn = 64;
  // Large problems: the CTA-pair 256 x 256 tile when its tiles fill at
  // least one wave of 2-CTA clusters (measured faster than 128 x 256 per SM).
  // Exact int8 takes the same rule with the pair kernel's int8 variant.
  if (Ni > 128 && cdiv64(Mi, 256) * cdiv64(Ni, 256) >= num_sms / 2) {
    c.pair = 1;
    c.bn = 256;
    return c;
  }
  const int64_t tiles = tm * cdiv64(Ni, c.bn);
  // Split K when the tiles alone leave most SMs idle and K is long.
  const int64_t kb = cdiv64(K, ab_type == T_E4M3 || ab_type == T_E5M2 ? 128 : 64);  // K slices
  if (tiles * 2 <= num_sms && kb >= 16) {
    int64_t s = num_sms / tiles;
    if (s > kb / 8) s = kb / 8;
    if (s > 8) s = 8;
    if (s < 1) s = 1;
    c.splits = (int)s;
  }
  return c;
}

}  // namespace gb300
