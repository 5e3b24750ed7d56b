// common.h -- structures shared by the host planner and the device kernels.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GB_HD __host__ __device__ __forceinline__
#else
#define GB_HD inline
#endif

namespace gb300 {

// Element type codes (the values of gemm_dtype_t).
enum : int { T_F16 = 1, T_BF16 = 2, T_F32 = 3, T_I8 = 4, T_I32 = 5, T_E4M3 = 6, T_E5M2 = 7,
             T_MXE4M3 = 8, T_MXE5M2 = 9 };

// Tensor-memory columns of the block-scaled (mx) mode of the single-CTA
// kernel: the per-stage scale cells of A and of B (stage s at + 4 s), beside
// the two 128-column accumulators.
constexpr uint32_t SFA_COL = 256;
constexpr uint32_t SFB_COL = 320;

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4: element types
// (bits 7-9 A, 10-12 B: 0 E4M3, 1 E5M2), majors (bit 15 A, 16 B), N/8 in
// bits 17-22, scale type E8M0 (bit 23), M/16 in bits 24-28; the scale-data
// IDs (bits 4-5 B, 29-30 A) are set per instruction.
GB_HD constexpr uint32_t idesc_mxf8(uint32_t e5m2, uint32_t a_mn, uint32_t b_mn, uint32_t m,
                                    uint32_t n) {
  return (e5m2 << 7) | (e5m2 << 10) | (a_mn << 15) | (b_mn << 16) | ((n >> 3) << 17) |
         (1u << 23) | ((m >> 4) << 24);
}

// Tile geometry of the tcgen05 kernels: one CTA owns a BM x BN output tile
// and walks K in BK-wide slices (BK 16-bit elements = one 128-byte row).
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int NUM_THREADS = 192;  // warp 0: TMA loads, warp 1: MMA issue, warps 2-5: epilogue

// Device status word bits.
constexpr uint32_t STATUS_TIMEOUT = 1u;

// Debug flags (test hooks).
constexpr int DBG_SKIP_FIRST_FILL = 1;

// Kernel parameters (passed by value).  Coordinates are those of the
// internal problem, which may be the transposed problem D^T = B^T A^T.
struct KParams {
  int M, N, K;                   // internal problem
  int tiles_m, tiles_n, group_m; // output tile grid and raster group
  int splits, kb_per_split, num_kb;
  int kb_per_chunk;              // k-blocks accumulated in one TMEM pass (exact-int8 mode)
  int kgroup;                    // single-CTA kernel: K slices loaded as one group (1, 2, 4)
  // Operands whose rows the TMA unit cannot read (rows off the 16-byte
  // grid), loaded instead by the kernel's own producer warps (16-bit types):
  // internal A' (M x K) and B' (K x N) pointers and leading dimensions.
  int a_lsu, b_lsu;
  const void* a_src;
  const void* b_src;
  long long a_ld, b_ld;
  // Block-scaled 8-bit floats (mx = 1): the E8M0 exponents of the 32-element
  // K blocks, packed by pack_scales_kernel into 512-byte cells, one per
  // (128-row tile, ring stage of four K blocks): cell (t, g) holds at byte
  // 16 j + 4 c + k the exponent of row 128 t + 32 c + j and K block 4 g + k
  // (sfa for the rows of A, sfb for the columns of B; nsb4 = cells per tile).
  int mx, nsb4;
  const uint8_t* sfa;
  const uint8_t* sfb;
  int a_mn, b_mn;                // operand majors: 0 = K-major, 1 = MN-major
  uint32_t idesc;                // tcgen05 instruction descriptor
  int f8;                        // 8-bit float operands: kind::f8f6f4, 128 K a slice
  // epilogue (internal coordinates: row r < M, column c < N)
  const void* C;
  int c_type;
  long long c_rs, c_cs;          // element strides of C
  void* D;
  int d_type;
  long long d_rs, d_cs;
  int d_vec;                     // D rows contiguous and 16-byte aligned
  int d_tma;                     // 16-bit D stored through shared memory by TMA (pair kernel)
  int c_tma;                     // with d_tma: C of D's type loaded by TMA into the same
                                 // staging buffers (pair kernel, 16-bit types)
  int c_vec;                     // C rows contiguous and 16-byte aligned
  float* ws;                     // split-K partial sums (fp32), or null
  long long ws_rs, ws_cs, ws_split;
  uint32_t* status;              // device status word
  unsigned long long timeout_ns; // bound of every device-side wait
  int debug_flags;
  // Stream-K hybrid (pair kernel), when sk_len > 0: cluster c first takes
  // sk_dp whole tiles (c, c + clusters, ...), then one contiguous run of
  // K stages over the tiles from sk_start on (sk_len stages, one more for
  // clusters c < sk_rem), so that every cluster gets the same work.  A tile
  // whose stages fall to two clusters is finished by the one that reaches
  // it last (the end of its run); the other (at the start of its run)
  // leaves its fp32 partial in tail_ws[c] and raises tail_flags[c] to epoch.
  // sk_len = 0: units are dealt round-robin.
  // sk_n3 >= 0: the runs are laid out in chains instead (plan_stream_k):
  // sk_n3 chains of three runs over four tiles, then chains of two runs
  // over three tiles, so that no run holds more than two pieces.
  int sk_dp, sk_start, sk_len, sk_rem, sk_n3;
  float* tail_ws;                // [leaving cluster][CTA half][128 rows][BN] fp32
  uint32_t* tail_flags;          // [leaving cluster][CTA half]
  uint32_t epoch;                // value the flags take during this run
  // Stream-K over the single-CTA kernel's tiles (sk1 = 1): CTA c of G takes
  // the contiguous run [c*T/G, (c+1)*T/G) of the T = tiles * num_kb
  // (tile, K slice) iterations.  A tile split over several CTAs is finished
  // by the CTA holding its first K slice: that piece is the last of its
  // CTA's run, while every other piece of the tile is the first of its own
  // CTA's run.  Those leave their fp32 partials in fix_ws[c] and raise
  // fix_flag[c] to `epoch`; the finishing CTA waits for them (they wait for
  // nothing), adds them up into its idle accumulator buffer while its own
  // MMAs run, then adds its accumulator and C and stores D.
  int sk1;
  // Split-K over a cluster (csk = splits > 1, single-CTA kernel, one unit
  // per CTA, cluster of csk consecutive CTAs = the splits of one tile): the
  // tile's 32-column slices are owned round-robin by the cluster's CTAs;
  // each copies its fp32 sums of the others' slices into their shared
  // memory (distributed shared memory) and adds the sums it receives for
  // its own, in split order, then C, and stores them: no partials in global
  // memory, no reduce launch.
  int csk;
  float* fix_ws;                 // [G][BM * BN] fp32, interleaved (see tc_gemm.cuh)
  uint32_t* fix_flag;            // [G], the epoch of the run that wrote fix_ws[c]
  // Timeline hook (tests and profiling; null in normal runs): the tensor-core
  // kernels write global-timer stamps of kTraceEvents events per CTA at
  // trace[cta * kTraceEvents + event] (see trace_at in tc_gemm.cuh).
  unsigned long long* trace;
};

constexpr int kTraceEvents = 32;

// Instruction descriptor of tcgen05.mma kind::f16 and kind::f8f6f4: fp32
// accumulator (bits 4-5 = 1), A/B element type (bits 7-9, 10-12: 0 fp16,
// 1 bf16 for kind::f16; 0 E4M3, 1 E5M2 for kind::f8f6f4), operand majors
// (bit 15 A, bit 16 B: 0 K-major, 1 MN-major), N/8 in bits 17-22 and M/16
// in bits 24-28.
GB_HD constexpr uint32_t idesc_f16(uint32_t bf16, uint32_t a_mn, uint32_t b_mn,
                                                 uint32_t m, uint32_t n) {
  return (1u << 4) | (bf16 << 7) | (bf16 << 10) | (a_mn << 15) | (b_mn << 16) |
         ((n >> 3) << 17) | ((m >> 4) << 24);
}

// Grouped tile order (FlagGems "Hygon optimization", "Grouped scheduling"):
// tiles are numbered so that GROUP_M consecutive tile rows walk the tile
// columns together; the last group holds the tile rows that remain.
GB_HD void raster_tile(int64_t t, int64_t num_pid_m, int64_t num_pid_n, int64_t group_m,
                       int64_t& pid_m, int64_t& pid_n) {
  const int64_t in_group = group_m * num_pid_n;
  const int64_t group_id = t / in_group;
  const int64_t first_m = group_id * group_m;
  const int64_t rem = num_pid_m - first_m;
  const int64_t size_m = rem < group_m ? rem : group_m;
  pid_m = first_m + (t % in_group) % size_m;
  pid_n = (t % in_group) / size_m;
}

// A piece of work of one CTA (or CTA pair): the output tile at (m0, n0) and
// the K slices [kb0, kb1).
struct Unit {
  int m0, n0, kb0, kb1, split;
  int tail;  // 1: part of a tile shared by two clusters (pair kernel, stream-K) or
             // by several CTAs (single-CTA stream-K)
  int part;  // 0: adds the other cluster's partial and finishes the tile;
             // 1: leaves its partial sums
  int ti;    // partial-sum slot (the leaving cluster; single-CTA stream-K: this piece's)
  int tile;  // tile index in the grouped order
  int pieces, piece;  // single-CTA stream-K: pieces of the tile, this one's K rank
};

// Stream-K hybrid plan (pair kernel): with W = tiles / clusters full waves
// and a partial last wave, W - 1 waves run as whole tiles and the stages of
// the remaining tiles are dealt out as equal contiguous runs, one per
// cluster.  Runs are at least one tile long (the remaining tiles number at
// least `clusters`), so a tile is shared by at most two clusters.  Leaves
// the fields zero (round-robin units) when the waves are already full or a
// run would be shorter than a tile.
//
// Chains (chains = true): equal runs put both ends of many runs inside
// tiles with a whole tile between them (three pieces), and such a run's
// finishing piece waits for a partner's long leaving piece while the whole
// tile's accumulator waits behind it; those clusters end last.  When the
// S stream-K tiles over C clusters satisfy 4C/3 <= S <= 3C/2, the runs are
// laid out instead as n3 = 3C - 2S chains of three runs over four tiles
// (run ends at 4/3 and 8/3 tiles: [W, F], [L, F], [L, W]) followed by
// n2 = 3S - 4C chains of two runs over three tiles (ends at 1.5 tiles:
// [W, F], [L, W]): every run holds at most two pieces, at the price of runs
// of 4/3 and 3/2 tiles instead of S/C.  At 4096^3 (S = 104, C = 76): 20
// triples and 8 pairs, runs of 85 - 96 stages instead of 87 - 88.
GB_HD void plan_stream_k(int64_t tiles, int clusters, int num_kb, int ksub, KParams& p,
                         bool chains = true) {
  p.sk_dp = p.sk_start = p.sk_len = p.sk_rem = 0;
  p.sk_n3 = -1;
  if (clusters <= 0 || tiles < clusters || tiles % clusters == 0 || ksub <= 0 ||
      num_kb % ksub != 0 || num_kb / ksub < 2)
    return;
  const int64_t waves = tiles / clusters;
  const int64_t sk_tiles = tiles - (waves - 1) * clusters;
  const int64_t work = sk_tiles * (num_kb / ksub);
  p.sk_dp = static_cast<int>(waves - 1);
  p.sk_start = static_cast<int>((waves - 1) * clusters);
  p.sk_len = static_cast<int>(work / clusters);
  p.sk_rem = static_cast<int>(work % clusters);
  if (chains && num_kb / ksub >= 8 && 3 * sk_tiles >= 4 * static_cast<int64_t>(clusters) &&
      2 * sk_tiles <= 3 * static_cast<int64_t>(clusters))
    p.sk_n3 = static_cast<int>(3 * static_cast<int64_t>(clusters) - 2 * sk_tiles);
}

// Work of one cluster.  Round-robin: units u = cid, cid + ncl, ... of the
// tiles x splits.  Stream-K hybrid: sk_dp whole tiles, then the tile pieces
// of the cluster's run of K stages [g0, g1) (stages of ksub slices).
struct PairWork {
  int n;       // number of units
  int g0, g1;  // stream-K run (stage indices over the tiles from sk_start)
};

GB_HD PairWork pair_work(const KParams& p, int ksub, int cid, int ncl) {
  PairWork pw;
  if (p.sk_len > 0) {
    const int nks = p.num_kb / ksub;
    if (p.sk_n3 >= 0) {
      // chain of `parts` runs over `span` tiles from tile `base`; this is run r
      const int t3 = 3 * p.sk_n3;
      const int base = cid < t3 ? 4 * (cid / 3) : 4 * p.sk_n3 + 3 * ((cid - t3) / 2);
      const int r = cid < t3 ? cid % 3 : (cid - t3) % 2;
      const int span = cid < t3 ? 4 : 3, parts = cid < t3 ? 3 : 2;
      pw.g0 = base * nks + (r * span * nks) / parts;
      pw.g1 = base * nks + ((r + 1) * span * nks) / parts;
    } else {
      pw.g0 = cid * p.sk_len + (cid < p.sk_rem ? cid : p.sk_rem);
      pw.g1 = pw.g0 + p.sk_len + (cid < p.sk_rem ? 1 : 0);
    }
    pw.n = p.sk_dp + ((pw.g1 - 1) / nks - pw.g0 / nks + 1);
  } else {
    const int total = p.tiles_m * p.tiles_n * p.splits;
    pw.g0 = pw.g1 = 0;
    pw.n = cid < total ? (total - cid + ncl - 1) / ncl : 0;
  }
  return pw;
}

// The i-th unit of cluster cid; m0 counts rows of 2*BM-row pair tiles.
GB_HD Unit pair_unit(const KParams& p, const PairWork& pw, int ksub, int cid, int ncl, int i,
                     int bn) {
  Unit w;
  int t;
  w.split = 0;
  w.tail = 0;
  w.part = 0;
  w.ti = 0;
  if (p.sk_len > 0 && i >= p.sk_dp) {
    // After its sk_dp whole tiles of the full waves, a cluster takes the
    // pieces of its stream-K run (k = 0 .. n-1 in K order) as: the piece
    // that starts mid-tile (it leaves a partial for the cluster whose run
    // ends in that tile, and waits for nothing), then the piece that ends
    // mid-tile (it finishes its tile with the next cluster's partial), then
    // the whole tiles (a run is shorter than two tiles: at most one).  A
    // finishing piece thus waits only for another run's first piece, and its
    // epilogue overlaps the whole tile's MMAs.  (Taking the leaving piece
    // before the full waves was measured slower: it staggers the waves and
    // loses the grouped raster's L2 reuse.)
    const int nks = p.num_kb / ksub;
    const int j = i - p.sk_dp;
    const int n_sk = pw.n - p.sk_dp;
    const int has_l = pw.g0 % nks != 0 ? 1 : 0;
    const int has_f = (pw.g1 % nks != 0 && n_sk > has_l) ? 1 : 0;
    int k;
    if (has_l && j == 0)
      k = 0;
    else if (has_f && j == has_l)
      k = n_sk - 1;
    else
      k = j - has_f;
    const int s = pw.g0 / nks + k;
    const int st0 = pw.g0 - s * nks > 0 ? pw.g0 - s * nks : 0;
    const int st1 = pw.g1 - s * nks < nks ? pw.g1 - s * nks : nks;
    t = p.sk_start + s;
    w.kb0 = st0 * ksub;
    w.kb1 = st1 * ksub;
    // A run is at least one tile long, so a piece cannot both start and end
    // inside its tile.
    if (st0 > 0) {
      w.tail = 1;
      w.part = 1;
      w.ti = cid;
    } else if (st1 < nks) {
      w.tail = 1;
      w.part = 0;
      w.ti = cid + 1;
    }
  } else if (p.sk_len > 0) {
    t = cid + i * ncl;
    w.kb0 = 0;
    w.kb1 = p.num_kb;
  } else {
    const int u = cid + i * ncl;
    t = u / p.splits;
    w.split = u - t * p.splits;
    w.kb0 = w.split * p.kb_per_split;
    w.kb1 = w.kb0 + p.kb_per_split < p.num_kb ? w.kb0 + p.kb_per_split : p.num_kb;
  }
  int64_t pm, pn;
  raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
  w.m0 = static_cast<int>(pm) * (2 * BM);
  w.n0 = static_cast<int>(pn) * bn;
  w.tile = t;
  w.pieces = 1;
  w.piece = 0;
  return w;
}

// ---------------------------------------------------------------- single-CTA stream-K
// First iteration of CTA c's run, and the CTA whose run holds iteration i
// (T iterations over G CTAs, T >= G so that no run is empty).
GB_HD int64_t sk_start(int64_t c, int64_t T, int64_t G) { return c * T / G; }
GB_HD int64_t sk_owner(int64_t i, int64_t T, int64_t G) { return ((i + 1) * G - 1) / T; }

// The units of one CTA of the single-CTA kernel: round-robin over the
// tiles x splits, or (sk1) the pieces of its stream-K run [s, e).
struct CtaWork {
  int n;
  int64_t s, e;
};

GB_HD CtaWork cta_work(const KParams& p, int c, int G, bool allow_sk = true) {
  CtaWork cw;
  if (allow_sk && p.sk1) {
    const int64_t T = static_cast<int64_t>(p.tiles_m) * p.tiles_n * p.num_kb;
    cw.s = sk_start(c, T, G);
    cw.e = sk_start(c + 1, T, G);
    cw.n = cw.e > cw.s ? static_cast<int>((cw.e - 1) / p.num_kb - cw.s / p.num_kb + 1) : 0;
  } else {
    const int total = p.tiles_m * p.tiles_n * p.splits;
    cw.s = cw.e = 0;
    cw.n = c < total ? (total - c + G - 1) / G : 0;
  }
  return cw;
}

// The CTA that computes piece j (in K order) of tile t; for j >= 1 that
// piece starts the CTA's run, so its partial sits in slot (and flag) of
// that CTA.
GB_HD int sk_piece_cta(const KParams& p, int t, int j, int G) {
  const int64_t T = static_cast<int64_t>(p.tiles_m) * p.tiles_n * p.num_kb;
  return static_cast<int>(sk_owner(static_cast<int64_t>(t) * p.num_kb, T, G) + j);
}

// Unit i of CTA c (of G); bm x bn tiles.  allow_sk = false compiles the
// stream-K arm out (kernels that never take it).
GB_HD Unit cta_unit(const KParams& p, const CtaWork& cw, int c, int G, int i, int bm, int bn,
                    bool allow_sk = true) {
  Unit w;
  int t;
  w.split = 0;
  w.tail = 0;
  w.part = 0;
  w.ti = 0;
  w.pieces = 1;
  w.piece = 0;
  if (allow_sk && p.sk1) {
    const int64_t nkb = p.num_kb;
    const int64_t T = static_cast<int64_t>(p.tiles_m) * p.tiles_n * nkb;
    t = static_cast<int>(cw.s / nkb + i);
    const int64_t t0 = static_cast<int64_t>(t) * nkb, t1 = t0 + nkb;
    w.kb0 = static_cast<int>((cw.s > t0 ? cw.s : t0) - t0);
    w.kb1 = static_cast<int>((cw.e < t1 ? cw.e : t1) - t0);
    const int64_t cf = sk_owner(t0, T, G), cl = sk_owner(t1 - 1, T, G);
    w.pieces = static_cast<int>(cl - cf + 1);
    w.piece = static_cast<int>(c - cf);
    w.tail = w.pieces > 1 ? 1 : 0;
    w.part = w.piece > 0 ? 1 : 0;  // 1: leaves its partial; 0: finishes the tile
    w.ti = c;
  } else {
    const int u = c + i * G;
    t = u / p.splits;
    w.split = u - t * p.splits;
    w.kb0 = w.split * p.kb_per_split;
    w.kb1 = w.kb0 + p.kb_per_split < p.num_kb ? w.kb0 + p.kb_per_split : p.num_kb;
  }
  int64_t pm, pn;
  raster_tile(t, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
  w.m0 = static_cast<int>(pm) * bm;
  w.n0 = static_cast<int>(pn) * bn;
  w.tile = t;
  return w;
}

}  // namespace gb300
