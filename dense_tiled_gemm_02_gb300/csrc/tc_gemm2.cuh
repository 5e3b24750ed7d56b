// tc_gemm2.cuh -- the CTA-pair (tcgen05 cta_group::2) variant of the GEMM.
//
// A cluster of two CTAs on neighbouring SMs owns a 256 x BN output tile.
// Each CTA stages its own 128 rows of A and half of the tile's BN columns of
// B per K-slice; the even CTA issues one 256 x BN x 16 pair MMA per 16-wide
// K step, which reads A from both CTAs' shared memory and the two B halves
// from both, and writes each CTA's 128 accumulator rows into that CTA's
// tensor memory.  Per SM this halves the B bytes that must be staged for the
// same work as the single-CTA 128 x BN tile.
//
// A ring stage holds KSUB 64-wide K slices (one 128-byte swizzle atom each),
// so one barrier wait and one commit cover 4*KSUB MMAs: the single issuing
// thread has little time between MMAs (the tensor core queues only a few),
// and every instruction it spends per stage is taken from that slack.
//
// Roles per CTA (192 threads) are those of tc_gemm.cuh:
//   warp 0  TMA producer (both CTAs): waits for its own free stage, loads its
//           A rows and B half; completion bytes of both CTAs are counted on
//           the even CTA's "full" barrier, which the even producer arms with
//           the pair's byte count.
//   warp 1  MMA issuer (even CTA only; both CTAs own the tensor memory).
//           Each stage is released to both producers, and each finished
//           accumulator announced to both epilogues, by one commit that
//           arrives on the same barrier of both CTAs.
//   warps 2-5 epilogue (both CTAs): drain their 128 rows, then tell the even
//           CTA's MMA warp that the accumulator buffer is free.
// All waits are bounded (ptx.cuh); the kernel ends with a cluster barrier so
// neither CTA leaves while its partner may still signal it.
#pragma once

#include "tc_gemm.cuh"

namespace gb300 {

template <int BN, int KSUB, bool I8X = false>
struct PairCfg {
  static constexpr int BNH = BN / 2;                        // B columns staged per CTA
  static constexpr uint32_t A_ATOM = BM * BK * 2;           // 128 rows x 64 K: 16 KiB
  static constexpr uint32_t B_ATOM = BNH * BK * 2;
  static constexpr uint32_t A_BYTES = KSUB * A_ATOM;        // per stage
  static constexpr uint32_t B_BYTES = KSUB * B_ATOM;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t PAIR_TX = 2 * STAGE_BYTES;      // bytes both CTAs land per stage
  // Two fp32 accumulators of BN columns each.
  static constexpr uint32_t TMEM_COLS = (2 * BN <= 256) ? 256 : 512;
  // Epilogue warps: four (one per 32-lane quarter of tensor memory), or
  // eight for exact int8, where two warps share a quarter and each keeps the
  // int32 sums of half the tile's columns in registers.
  static constexpr int EPI_WARPS = I8X ? 8 : 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  // 224: 16 x 19 tiles at 4096^2 are exactly four waves of 76 pairs
  static_assert(BN == 128 || BN == 224 || BN == 256, "pair tile width");
  static_assert(!I8X || BN == 256, "the int8 pair variant uses 256-wide tiles");
  static_assert(B_ATOM % 1024 == 0, "stage alignment");
};

// Staging for the TMA store of D: two buffers of 128 rows x 64 16-bit
// columns (one 128-byte swizzle row each).  The exact-int8 variant has four:
// two 4 KB buffers (32 rows x 32 int32) per epilogue warp for C and D.
constexpr uint32_t D_STAGE_BYTES = BM * 64 * 2;

// Exact int8: accumulator columns each epilogue thread reads from tensor
// memory per wait while draining a finished pass (two 16-column loads; 64
// columns no longer fit the registers beside the 128 int32 sums).
constexpr int I8_DRAIN = 32;

template <bool I8X>
__host__ __device__ constexpr uint32_t pair_stage_bytes() {
  return (I8X ? 4 : 2) * D_STAGE_BYTES;
}

template <int BN, int STAGES, int KSUB, bool I8X = false>
constexpr uint32_t pair_smem_bytes() {
  return STAGES * PairCfg<BN, KSUB>::STAGE_BYTES + pair_stage_bytes<I8X>() + 512 + 1024;
}

// ---------------------------------------------------------------- the chunk that crosses N
// A TMA store writes whole 16-byte units at the right edge of the tensor: a
// D whose N is not a multiple of 8 (16-bit) but whose rows are padded to
// one would get up to 7 elements of its padding overwritten.  The staged
// 32 x 64 chunk that crosses N is therefore stored by the warp itself, by
// rows: lane l takes columns 2l and 2l+1 of every row, so each warp access
// covers 128 contiguous bytes of one row, with element masks at N.

// Byte offset, in a swizzled chunk, of row i's columns 2*lane and 2*lane+1.
__device__ __forceinline__ uint32_t chunk_off(int i, int lane) {
  return static_cast<uint32_t>(i * 128 + (((lane >> 2) ^ (i & 7)) * 16) + (lane & 3) * 4);
}

// The warp's staged 32 x 64 D chunk to global memory at (y0, x0), masked to
// M x N; a word store where the row's address allows it, else two halves.
__device__ __forceinline__ void st_d_chunk_rows(const uint8_t* chunk, uint16_t* D, long long d_rs,
                                                int y0, int x0, int M, int N, int lane) {
  const int col = x0 + 2 * lane;
#pragma unroll 4
  for (int i = 0; i < 32; ++i) {
    if (y0 + i >= M) break;
    const uint32_t w = *reinterpret_cast<const uint32_t*>(chunk + chunk_off(i, lane));
    uint16_t* dst = D + static_cast<long long>(y0 + i) * d_rs + col;
    if (col + 1 < N && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
      *reinterpret_cast<uint32_t*>(dst) = w;
    } else {
      if (col < N) dst[0] = static_cast<uint16_t>(w);
      if (col + 1 < N) dst[1] = static_cast<uint16_t>(w >> 16);
    }
  }
}

// kb0/kb1 count 64-wide K slices; a stage covers KSUB of them.
//
// I8X: exact int8 GEMM on the bf16 tensor pipe (operands widened to bf16
// beforehand, which is exact for |v| <= 128).  Each run of kb_per_chunk K
// slices (960 K by default) is accumulated afresh in fp32, where every partial
// sum is an integer of magnitude at most 960 * 2^14 < 2^24 and therefore
// exact; the epilogue converts each finished chunk to int32 and adds it to
// running sums held in registers (eight epilogue warps, 128 columns each),
// while the MMA fills the other accumulator with the next chunk.  After the last chunk C is
// added and the sums are stored as int32.
template <int BN, int STAGES, int KSUB, bool I8X>
__global__ void __launch_bounds__(PairCfg<BN, KSUB, I8X>::THREADS, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmD,
                        const __grid_constant__ CUtensorMap tmC, const KParams p) {
  using Cfg = PairCfg<BN, KSUB, I8X>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
  uint8_t* sD = sB + STAGES * Cfg::B_BYTES;  // staging buffers, 1024-aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(sD + pair_stage_bytes<I8X>());
  // ring full/empty, accumulator full/empty, done; C-load barriers of the
  // epilogue warps' two staging buffers
  constexpr int NBARS = 2 * STAGES + 5 + 2 * Cfg::EPI_WARPS;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* ep_go = abort_flag + 1;  // the epilogue leader's verdict for its warps

  if (threadIdx.x == 0) trace_at(p, 0);
  const uint32_t bar0 = smem_u32(bars);
  auto full = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
  auto acc_full = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acc_empty = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
  auto cbar = [&](int e, int b) { return bar0 + 8u * (2 * STAGES + 5 + 2 * e + b); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 2 * Cfg::EPI_WARPS);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(done_bar, 1);
    for (int e = 0; e < Cfg::EPI_WARPS; ++e) {
      mbar_init(cbar(e, 0), 1);
      mbar_init(cbar(e, 1), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.d_tma) tma_prefetch_desc(&tmD);
    if ((I8X && p.d_tma && p.C) || (!I8X && p.c_tma)) tma_prefetch_desc(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), Cfg::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // The work split and the load thread's first unit depend on the kernel
  // parameters only: computed before the wait, so that the first loads go
  // out as soon as it returns.
  const int cid = blockIdx.x >> 1;
  const int ncl = gridDim.x >> 1;
  const PairWork pw = pair_work(p, KSUB, cid, ncl);
  Unit w_first{};
  if (threadIdx.x == 0 && pw.n > 0) w_first = pair_unit(p, pw, KSUB, cid, ncl, 0, BN);
  // This CTA's TMA loads of one ring stage: K slices kb .. kb+KSUB-1 of unit
  // w into slot s, counted on the even CTA's barrier (armed by the even CTA
  // with both CTAs' bytes).
  auto issue_stage = [&](const Unit& w, const int kb, const uint32_t s) {
    const int am = w.m0 + BM * static_cast<int>(rank);
    const int bn0 = w.n0 + Cfg::BNH * static_cast<int>(rank);
    const uint32_t fb = map_shared_rank(full(s), 0);
    if (leader) mbar_arrive_expect_tx(full(s), Cfg::PAIR_TX);
#pragma unroll
    for (int j = 0; j < KSUB; ++j) {
      // a K slice past the end still lands (as zeros) and is counted
      const int k0 = (kb + j) * (p.f8 ? 2 * BK : BK);  // a 128-byte row: 64 or 128 K
      const uint32_t a_dst = smem_u32(sA + s * Cfg::A_BYTES + j * Cfg::A_ATOM);
      const uint32_t b_dst = smem_u32(sB + s * Cfg::B_BYTES + j * Cfg::B_ATOM);
      if (!p.a_mn) {
        tma_load_2d_pair(a_dst, &tmA, k0, am, fb);
      } else {
#pragma unroll
        for (int i = 0; i < BM / 64; ++i)
          tma_load_2d_pair(a_dst + i * 8192u, &tmA, am + 64 * i, k0, fb);
      }
      if (!p.b_mn) {
        tma_load_2d_pair(b_dst, &tmB, k0, bn0, fb);
      } else {
#pragma unroll
        for (int i = 0; i < Cfg::BNH / 64; ++i)
          tma_load_2d_pair(b_dst + i * 8192u, &tmB, bn0 + 64 * i, k0, fb);
      }
    }
  };
  // The first stage goes out right after the wait below, before the load
  // loop's code is first fetched; the loop then starts at the second.
  const bool early = !(p.debug_flags & DBG_SKIP_FIRST_FILL) && pw.n > 0 &&
                     w_first.kb0 < w_first.kb1;
  // Everything above touches only on-chip state: it overlaps the previous
  // kernel in the stream; global memory is read and written only after it.
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    trace_at(p, 1);
    if (early) {
      issue_stage(w_first, w_first.kb0, 0u);
      trace_at(p, 2);
    }
  }

  const uint64_t tmo = p.timeout_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      // it: stages issued; (s, ph): ring slot and phase (STAGES >= 2)
      uint32_t it = early ? 1u : 0u, s = early ? 1u : 0u, ph = 0;
      int64_t skipped = -1;
      bool stop = false;
      for (int i = 0; i < pw.n && !stop; ++i) {
        const Unit w = i == 0 ? w_first : pair_unit(p, pw, KSUB, cid, ncl, i, BN);
        for (int kb = (i == 0 && early) ? w.kb0 + KSUB : w.kb0; kb < w.kb1; kb += KSUB) {
          if (!bounded_wait(empty(s), ph ^ 1u, abort_flag, p.status, STATUS_TIMEOUT, tmo)) {
            stop = true;
            break;
          }
          if (leader && (p.debug_flags & DBG_SKIP_FIRST_FILL) && it == 0) {
            skipped = 0;  // test hook: never arm stage 0, so the MMA wait on it expires
          } else {
            issue_stage(w, kb, s);
          }
          if (it == 0) trace_at(p, 2);
          ++it;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (leader) {
        // Both CTAs' copies of the last stages are counted here: let them land.
        for (uint32_t j = it > STAGES ? it - STAGES : 0; j < it; ++j) {
          if (static_cast<int64_t>(j) == skipped) continue;
          drain_wait(full(j % STAGES), (j / STAGES) & 1u, 200000000ull);
        }
      } else if (stop) {
        // The odd CTA cannot watch the even CTA's barrier: give copies it
        // issued before giving up time to land.
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 1000000ull) __nanosleep(1000);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      const uint32_t a_lo0 = sdesc_lo(smem_u32(sA), p.a_mn ? 8192u : 16u);
      const uint32_t b_lo0 = sdesc_lo(smem_u32(sB), p.b_mn ? 8192u : 16u);
      const uint32_t dhi = sdesc_hi_sw128(1024u);
      // Offsets (16-byte units) of the 4*KSUB K steps of a stage: 32 bytes
      // along a K-major row or 16 rows of an MN-major tile per step, one
      // swizzle atom per 64-wide slice.
      uint32_t a_off[4 * KSUB], b_off[4 * KSUB];
#pragma unroll
      for (int kk = 0; kk < 4 * KSUB; ++kk) {
        a_off[kk] = (kk / 4) * (Cfg::A_ATOM >> 4) + (kk % 4) * (p.a_mn ? 128u : 2u);
        b_off[kk] = (kk / 4) * (Cfg::B_ATOM >> 4) + (kk % 4) * (p.b_mn ? 128u : 2u);
      }
      uint32_t s = 0, ph = 0, acc_it = 0;
      bool stop = false;
      const bool f8 = !I8X && p.f8 != 0;
      // One pass of the K loop into accumulator buffer `buf`.
      bool first_stage = true;
      auto k_loop = [&](const int kc, const int ke, const uint32_t buf) {
        const uint32_t d_tmem = tmem_base + buf * BN;
        uint32_t accumulate = 0;
        for (int kb = kc; kb < ke; kb += KSUB) {
          if (!bounded_wait(full(s), ph, abort_flag, p.status, STATUS_TIMEOUT, tmo)) {
            stop = true;
            return;
          }
          if (first_stage) {
            trace_at(p, 3);
            first_stage = false;
          }
          const uint32_t a_lo = a_lo0 + s * (Cfg::A_BYTES >> 4);
          const uint32_t b_lo = b_lo0 + s * (Cfg::B_BYTES >> 4);
          if (f8) {  // 8-bit operands: 32 K per 32-byte step (both K-major)
#pragma unroll
            for (int kk = 0; kk < 4 * KSUB; ++kk)
              mma_f8_ss_pair(d_tmem, sdesc(dhi, a_lo + a_off[kk]), sdesc(dhi, b_lo + b_off[kk]),
                             p.idesc, accumulate | kk);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4 * KSUB; ++kk)
              mma_f16_ss_pair(d_tmem, sdesc(dhi, a_lo + a_off[kk]), sdesc(dhi, b_lo + b_off[kk]),
                              p.idesc, accumulate | kk);
          }
          accumulate = 1;
          mma_commit_pair_both(empty(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      };
      for (int i = 0; i < pw.n && !stop; ++i) {
        const Unit w = pair_unit(p, pw, KSUB, cid, ncl, i, BN);
        if constexpr (I8X) {
          // a fresh accumulator for every chunk of kb_per_chunk K slices
          for (int kc = w.kb0; kc < w.kb1 && !stop; kc += p.kb_per_chunk) {
            const uint32_t buf = acc_it & 1u;
            if (!bounded_wait(acc_empty(buf), ((acc_it >> 1) & 1u) ^ 1u, abort_flag, p.status,
                              STATUS_TIMEOUT, tmo)) {
              stop = true;
              break;
            }
            tc_fence_after();
            k_loop(kc, min(w.kb1, kc + p.kb_per_chunk), buf);
            if (stop) break;
            mma_commit_pair_both(acc_full(buf));
            ++acc_it;
          }
        } else {
          const uint32_t buf = acc_it & 1u;
          if (!bounded_wait(acc_empty(buf), ((acc_it >> 1) & 1u) ^ 1u, abort_flag, p.status,
                            STATUS_TIMEOUT, tmo))
            break;
          tc_fence_after();
          if (i < 11) trace_at(p, 10 + 2 * i);
          k_loop(w.kb0, w.kb1, buf);
          if (stop) break;
          mma_commit_pair_both(acc_full(buf));
          if (i < 11) trace_at(p, 11 + 2 * i);
          ++acc_it;
        }
      }
      trace_at(p, 4);
      mma_commit_pair_both(done_bar);
      drain_wait(done_bar, 0, 200000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // One thread (the epilogue leader) waits for each accumulator and tells
    // the other 127 through a named barrier, so that all of them always take
    // the same path through the barriers below.  The per-tile loop over
    // 32-column slices is kept rolled: unrolled, its code no longer fits the
    // instruction cache next to the producer and MMA loops, and every slice
    // then waits on instruction fetch.
    const int q = warp & 3;
    const int row_local = q * 32 + lane;  // this thread's row of the CTA's 128
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const bool ep_leader = threadIdx.x == 64;
    uint32_t acc_it = 0, staged = 0;
    if constexpr (I8X) {
      // Exact int8.  Warps 2-9: warp w reads TMEM lanes 32*(w%4).. and the
      // columns [HC*half, HC*half + HC) of each accumulator.  Per chunk,
      // each fp32 value (an integer below 2^24, so cvt.rni is exact) is
      // added to the thread's int32 sums; after the last chunk C is added
      // and the row segment stored.
      constexpr int HC = BN / 2;
      const int half = (warp - 2) >> 2;
      const uint32_t col0 = static_cast<uint32_t>(half * HC);
      // With p.d_tma the tile's C and D move through two 4 KB shared-memory
      // buffers of this warp (32 rows x 32 int32, 128-byte swizzle) by TMA:
      // per-thread row accesses would put 32 rows in every warp access.
      const int e = warp - 2;
      uint8_t* const stg = sD + e * 8192;
      uint32_t cph[2] = {0u, 0u};      // parity of the next completion of cbar(e, b)
      bool c_pending[2] = {false, false};
      auto load_c = [&](int b, int gx, int gy) {  // lane 0: slice into buffer b
        bulk_wait_read_all();                       // earlier stores have read it
        mbar_arrive_expect_tx(cbar(e, b), 32 * 32 * 4);
        tma_load_2d(smem_u32(stg + b * 4096), &tmC, gx, gy, cbar(e, b));
      };
      int isum[HC];
      bool ok = true;
      for (int i = 0; i < pw.n && ok; ++i) {
        const Unit w = pair_unit(p, pw, KSUB, cid, ncl, i, BN);
        const int r = w.m0 + BM * static_cast<int>(rank) + row_local;
        const int nch = (w.kb1 - w.kb0 + p.kb_per_chunk - 1) / p.kb_per_chunk;
        const int gy = w.m0 + BM * static_cast<int>(rank) + 32 * q;  // this warp's rows
        const int gx0 = w.n0 + static_cast<int>(col0);
        // Stream-K pieces of a shared tile: the leaving piece stores its
        // int32 sums (as the 16-bit path stores its fp32 ones: int4 of
        // column group g of row i at [g][i]) and raises its flag; the
        // finishing piece adds them, then C, and stores D.  Integer sums:
        // the result is the same bits as without stream-K.
        const bool leaves = w.tail && w.part == 1;
#pragma unroll
        for (int j = 0; j < HC; ++j) isum[j] = 0;
        for (int ch = 0; ch < nch; ++ch) {
          const uint32_t buf = acc_it & 1u;
          if (p.d_tma && p.C && !leaves && ch == nch - 1) {
            // C of the tile's first two slices, while the last chunk runs
            if (lane == 0) {
              load_c(0, gx0, gy);
              load_c(1, gx0 + 32, gy);
            }
            c_pending[0] = c_pending[1] = true;
          }
          if (ep_leader)
            *ep_go = bounded_wait(acc_full(buf), (acc_it >> 1) & 1u, abort_flag, p.status,
                                  STATUS_TIMEOUT, tmo) ? 1 : 0;
          named_barrier_sync(1, 32 * Cfg::EPI_WARPS);
          ok = *ep_go != 0;
          named_barrier_sync(1, 32 * Cfg::EPI_WARPS);
          if (!ok) break;
          tc_fence_after();
          // I8_DRAIN columns per tensor-memory round trip: the loads of a
          // batch are all issued before the one wait, so the latency of a
          // load is paid once per batch, not once per 16 columns (the 128
          // sums already hold most of the registers a thread of this
          // 320-thread block may have, which bounds the batch).
          constexpr int DC = I8_DRAIN;
#pragma unroll
          for (int c = 0; c < HC / DC; ++c) {
            uint32_t v[DC];
#pragma unroll
            for (int x = 0; x < DC / 16; ++x)
              tmem_ld_32x32b_x16(tmem_base + lane_base + buf * BN + col0 + c * DC + 16 * x,
                                 *reinterpret_cast<uint32_t(*)[16]>(v + 16 * x));
            tmem_ld_wait();
            if (c == HC / DC - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(map_shared_rank(acc_empty(buf), 0));
            }
#pragma unroll
            for (int j = 0; j < DC; ++j) isum[c * DC + j] += __float2int_rn(__uint_as_float(v[j]));
          }
          ++acc_it;
        }
        if (!ok) break;
        // (the piece's slot and flag, computed here so that they are not
        // held across the chunk loop)
        int4* const pbase = w.tail ? reinterpret_cast<int4*>(
                                         p.tail_ws + static_cast<size_t>(w.ti * 2 + rank) * BM * BN) +
                                         row_local
                                   : nullptr;
        uint32_t* const flag = w.tail ? p.tail_flags + w.ti * 2 + rank : nullptr;
        if (leaves) {
#pragma unroll
          for (int g = 0; g < HC / 4; ++g)
            pbase[(static_cast<int>(col0) / 4 + g) * BM] =
                make_int4(isum[4 * g], isum[4 * g + 1], isum[4 * g + 2], isum[4 * g + 3]);
          // Publish: every epilogue thread of this CTA has written its row.
          __threadfence();
          named_barrier_sync(1, 32 * Cfg::EPI_WARPS);
          if (ep_leader) {
            __threadfence();
            st_release_gpu(flag, p.epoch);
          }
          continue;
        }
        if (w.tail && w.part == 0) {
          if (ep_leader)
            *ep_go = bounded_flag_wait(flag, p.epoch, abort_flag, p.status, STATUS_TIMEOUT, tmo)
                         ? 1 : 0;
          named_barrier_sync(1, 32 * Cfg::EPI_WARPS);
          ok = *ep_go != 0;
          named_barrier_sync(1, 32 * Cfg::EPI_WARPS);
          if (!ok) break;
          // four 16-byte loads in flight per batch (the 128 sums hold most
          // of the registers)
#pragma unroll
          for (int g0 = 0; g0 < HC / 4; g0 += 4) {
            int4 v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              v[k] = __ldcg(pbase + (static_cast<int>(col0) / 4 + g0 + k) * BM);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              isum[4 * (g0 + k)] += v[k].x;
              isum[4 * (g0 + k) + 1] += v[k].y;
              isum[4 * (g0 + k) + 2] += v[k].z;
              isum[4 * (g0 + k) + 3] += v[k].w;
            }
          }
        }
        if (p.d_tma) {
#pragma unroll
          for (int c = 0; c < HC / 32; ++c) {
            const int b = c & 1;
            uint8_t* const sbuf = stg + b * 4096;
            const int gx = gx0 + 32 * c;
            if (!p.C) {
              // the store issued from this buffer two slices ago has read it
              if (lane == 0) bulk_wait_read_le1();
              __syncwarp();
            } else {
              if (!bounded_wait(cbar(e, b), cph[b], abort_flag, p.status, STATUS_TIMEOUT, tmo)) {
                ok = false;
                break;
              }
              cph[b] ^= 1u;
              c_pending[b] = false;
            }
            // this thread's row: 8 units of 16 bytes, unit u at (u ^ row % 8)
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              int4* const ptr = reinterpret_cast<int4*>(sbuf + lane * 128 + ((u ^ (lane & 7)) * 16));
              int4 x = p.C ? *ptr : make_int4(0, 0, 0, 0);
              x.x += isum[c * 32 + 4 * u];
              x.y += isum[c * 32 + 4 * u + 1];
              x.z += isum[c * 32 + 4 * u + 2];
              x.w += isum[c * 32 + 4 * u + 3];
              *ptr = x;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (gx < p.N && gy < p.M)  // boxes entirely outside D are skipped
                tma_store_2d(&tmD, smem_u32(sbuf), gx, gy);
              bulk_commit();
              if (p.C && c + 2 < HC / 32) load_c(b, gx + 64, gy);
            }
            if (p.C && c + 2 < HC / 32) c_pending[b] = true;
          }
          if (!ok) break;
        } else {
#pragma unroll
          for (int c = 0; c < HC / 32; ++c)
            store_d_i32(p, r, w.n0 + static_cast<int>(col0) + c * 32,
                        *reinterpret_cast<int(*)[32]>(isum + c * 32));
        }
      }
      // C loads still in flight (after a timeout) land before the CTA
      // leaves, and so do the stores that read the staging buffers.
      if (lane == 0) {
        for (int b = 0; b < 2; ++b)
          if (c_pending[b]) drain_wait(cbar(e, b), cph[b], 200000000ull);
        bulk_wait_all();
      }
    } else {
    // C by TMA (p.c_tma): each warp loads its 32 rows x 64 columns of C per
    // chunk into the staging buffer that the chunk's D then leaves from, D
    // written over C in place.  Chunks 0 and 1 of a tile are requested
    // before the accumulator wait (under the tile's MMAs), chunk j + 2 once
    // chunk j's store has read the buffer.  Register-held C waited on DRAM
    // once every two 32-column slices: about 7 of a 256-wide tile's 7.5 us.
    const int ew = warp - 2;  // this epilogue warp's C barriers
    // 64-column chunks of a tile (a 224-wide tile ends in a 32-column one)
    constexpr int NCHUNK = (BN + 63) / 64;
    // bit b of ctw: parity of the next wait on buffer b; byte b of ctn: loads
    // into buffer b not waited for yet
    uint32_t ctw = 0u, ctn = 0u;
    auto load_ct = [&](int b, int x, int y) {  // lane 0: one 32 x 64 box into buffer b
      mbar_arrive_expect_tx(cbar(ew, b), 32 * 128);
      tma_load_2d(smem_u32(sD + b * D_STAGE_BYTES + q * 32 * 128), &tmC, x, y, cbar(ew, b));
    };
    for (int i = 0; i < pw.n; ++i) {
      const Unit w = pair_unit(p, pw, KSUB, cid, ncl, i, BN);
      const int r = w.m0 + BM * static_cast<int>(rank) + row_local;
      const bool leaves_partial = w.tail && w.part == 1;
      const bool staged_store = p.d_tma && !leaves_partial && p.splits == 1;
      const bool use_ctma = p.c_tma && staged_store;
      const int y0w = w.m0 + BM * static_cast<int>(rank) + 32 * q;  // the warp's first row
      // C of a slice comes as four 16-byte loads of this thread's row, issued
      // one slice ahead (the first one before the accumulator wait); in a
      // tile that crosses N the groups past N are masked (ld_c8), and a row
      // past M reads nothing and adds zeros.
      const bool c_rows = !use_ctma && !leaves_partial && p.C != nullptr && p.c_vec &&
                          p.c_type != T_F32 && r < p.M;
      const int c_ncols = min(BN, p.N - w.n0);
      const uint16_t* crow =
          c_rows ? static_cast<const uint16_t*>(p.C) + r * p.c_rs + w.n0 : nullptr;
      // Two slices of C in flight: slice c lives in cb[c & 1] and is
      // reloaded with slice c + 2 once used (a loop unrolled by two keeps the
      // buffers in fixed registers).
      const uint32_t buf = acc_it & 1u;
      uint32_t* flag = w.tail ? p.tail_flags + w.ti * 2 + rank : nullptr;
      // The fp32 partial sums of a shared tile (one CTA half), stored so that
      // the 128 threads' float4s of each 4-column group are adjacent: a warp
      // then moves 512 contiguous bytes per access instead of 32 pieces.
      float4* pbase = w.tail ? reinterpret_cast<float4*>(
                                   p.tail_ws + static_cast<size_t>(w.ti * 2 + rank) * BM * BN) +
                                   row_local
                             : nullptr;
      // When a unit that finishes a shared tile is the last of its cluster,
      // the MMA no longer needs the other accumulator buffer: while this
      // unit's MMAs run, the other cluster's partial is copied into those
      // tensor-memory columns, and the final epilogue reads both sums there.
      // Otherwise the partial is read from global memory slice by slice,
      // while the MMAs of the cluster's next unit run.
      const bool adds = w.tail && w.part == 0;
      const bool preloaded = adds && i == pw.n - 1;
      const uint32_t pcol = tmem_base + lane_base + (buf ^ 1u) * BN;
      if (adds) {
        if (ep_leader)
          *ep_go = bounded_flag_wait(flag, p.epoch, abort_flag, p.status, STATUS_TIMEOUT, tmo)
                       ? 1 : 0;
        named_barrier_sync(1, 128);
        const bool fok = *ep_go != 0;
        named_barrier_sync(1, 128);
        if (!fok) break;
        if (preloaded) {
          // two 32-column slices per batch: 16 loads in flight per thread
          // (a 224-wide tile ends in one single slice)
#pragma unroll 1
          for (int c = 0; c < BN / 32; c += 2) {
            const int nh = c + 1 < BN / 32 ? 2 : 1;
            uint32_t x[2][32];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 q = h < nh ? pbase[((c + h) * 8 + j) * BM]
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                x[h][4 * j] = __float_as_uint(q.x);
                x[h][4 * j + 1] = __float_as_uint(q.y);
                x[h][4 * j + 2] = __float_as_uint(q.z);
                x[h][4 * j + 3] = __float_as_uint(q.w);
              }
            tmem_st_32x32b_x32(pcol + c * 32, x[0]);
            if (nh == 2) tmem_st_32x32b_x32(pcol + (c + 1) * 32, x[1]);
          }
          tmem_st_wait();
        }
      }
      if (use_ctma) {
        const uint32_t s0 = staged;  // chunk j of this tile uses buffer (s0 + j) & 1
        if (lane == 0) {
          bulk_wait_read_all();  // the previous tile's stores have read the buffers
          for (int j = 0; j < 2 && j < NCHUNK; ++j) load_ct((s0 + j) & 1u, w.n0 + 64 * j, y0w);
        }
        for (int j = 0; j < 2 && j < NCHUNK; ++j) ctn += 1u << (8u * ((s0 + j) & 1u));
      }
      uint4 cb0[4], cb1[4];
      if (c_rows) {
#pragma unroll
        for (int k = 0; k < 4; ++k) cb0[k] = ld_c8(crow, 8 * k, c_ncols);
#pragma unroll
        for (int k = 0; k < 4; ++k) cb1[k] = ld_c8(crow, 32 + 8 * k, c_ncols);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) cb0[k] = cb1[k] = make_uint4(0u, 0u, 0u, 0u);
      }
      // The other cluster's partial, when it is read from global memory:
      // like C, two slices in flight (slice c in pb[c & 1]).
      const bool adds_global = adds && !preloaded;
      float4 pb0[8], pb1[8];
      if (adds_global) {
#pragma unroll
        for (int j = 0; j < 8; ++j) pb0[j] = pbase[j * BM];
#pragma unroll
        for (int j = 0; j < 8; ++j) pb1[j] = pbase[(8 + j) * BM];
      }
      if (ep_leader) {
        *ep_go = bounded_wait(acc_full(buf), (acc_it >> 1) & 1u, abort_flag, p.status,
                              STATUS_TIMEOUT, tmo) ? 1 : 0;
        trace_at(p, 5);
      }
      named_barrier_sync(1, 128);
      const bool go = *ep_go != 0;
      named_barrier_sync(1, 128);
      if (!go) break;
      tc_fence_after();
      // One 32-column slice; CT/DT are the C and D element types when known
      // at compile time (0: no C), -1 for the generic run-time path.
      // Once slice c's C has been added, its buffer takes slice c + 2.
      auto reload_c = [&](const int c, uint4 (&cbuf)[4]) {
        if (c_rows && c + 2 < BN / 32) {
#pragma unroll
          for (int k = 0; k < 4; ++k) cbuf[k] = ld_c8(crow, 32 * (c + 2) + 8 * k, c_ncols);
        }
      };
      auto slice = [&](const int c, uint4 (&cbuf)[4], float4 (&pbuf)[8], auto ct_tag,
                       auto dt_tag) {
        constexpr int CT = decltype(ct_tag)::value;
        constexpr int DT = decltype(dt_tag)::value;
        const int h = c & 1;  // which half of a 64-column staging chunk
        // Each warp stages its own 32 rows and stores them itself, so the
        // chunk loop needs no barrier across warps.
        uint8_t* stage = sD + (staged & 1u) * D_STAGE_BYTES;
        if (use_ctma && h == 0) {
          // this chunk's C has landed in its buffer
          const uint32_t b = staged & 1u;
          bounded_wait(cbar(ew, b), (ctw >> b) & 1u, abort_flag, p.status, STATUS_TIMEOUT, tmo);
          ctw ^= 1u << b;
          ctn -= 1u << (8u * b);
        } else if (staged_store && h == 0 && staged >= 2) {
          // the store this warp issued from this buffer two chunks ago must have read it
          if (lane == 0) bulk_wait_read_le1();
          __syncwarp();
        }
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + lane_base + buf * BN + c * 32, v);
        tmem_ld_wait();
        if (c == BN / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(map_shared_rank(acc_empty(buf), 0));
        }
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
        const int c0 = w.n0 + c * 32;
        if (leaves_partial) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            pbase[(c * 8 + j) * BM] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2],
                                                  f[4 * j + 3]);
          return;
        }
        if (preloaded) {
          uint32_t q[32];
          tmem_ld_32x32b_x32(pcol + c * 32, q);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) f[j] += __uint_as_float(q[j]);
        } else if (adds_global) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            f[4 * j] += pbuf[j].x;
            f[4 * j + 1] += pbuf[j].y;
            f[4 * j + 2] += pbuf[j].z;
            f[4 * j + 3] += pbuf[j].w;
          }
          if (c + 2 < BN / 32) {
#pragma unroll
            for (int j = 0; j < 8; ++j) pbuf[j] = pbase[((c + 2) * 8 + j) * BM];
          }
        }
        if (CT < 0) {
          if (p.splits > 1) {
            store_partial(p, r, c0, w.split, f);
            return;
          }
          if (c_rows) {
            add_c_prefetched(p.c_type, cbuf, f);
            reload_c(c, cbuf);
          } else {
            add_c_f(p, r, c0, f);
          }
          if (!staged_store) {
            store_d_f(p, r, c0, f);
            return;
          }
        } else if (CT != 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // C from the staging buffer (the unit D takes below), else from registers
            const uint4 cv = use_ctma ? *reinterpret_cast<const uint4*>(
                                            stage + row_local * 128 +
                                            (((h * 4 + k) ^ (row_local & 7)) * 16))
                                      : cbuf[k];
            const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float lo, hi;
              unpack2_t<CT>(cw[e], lo, hi);
              f[8 * k + 2 * e] += lo;
              f[8 * k + 2 * e + 1] += hi;
            }
          }
          if (!use_ctma) reload_c(c, cbuf);
        }
        // 16 bytes = 8 outputs per swizzle unit; the unit's position in the
        // 128-byte row is XORed with row % 8 (the TMA's 128B swizzle), which
        // also spreads a warp's stores over all banks.
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 x;
          if constexpr (DT < 0) {
            x.x = pack2(p.d_type, f[8 * k + 0], f[8 * k + 1]);
            x.y = pack2(p.d_type, f[8 * k + 2], f[8 * k + 3]);
            x.z = pack2(p.d_type, f[8 * k + 4], f[8 * k + 5]);
            x.w = pack2(p.d_type, f[8 * k + 6], f[8 * k + 7]);
          } else {
            x.x = pack2_t<DT>(f[8 * k + 0], f[8 * k + 1]);
            x.y = pack2_t<DT>(f[8 * k + 2], f[8 * k + 3]);
            x.z = pack2_t<DT>(f[8 * k + 4], f[8 * k + 5]);
            x.w = pack2_t<DT>(f[8 * k + 6], f[8 * k + 7]);
          }
          const int unit = (h * 4 + k) ^ (row_local & 7);
          *reinterpret_cast<uint4*>(stage + row_local * 128 + unit * 16) = x;
        }
        // a chunk is stored after its second slice, or after its only one
        // (the 32-column chunk that ends a 224-wide tile)
        const bool half = (BN % 64) != 0 && c == BN / 32 - 1;
        if (h == 1 || half) {
          const int x0 = w.n0 + 32 * (c - h);
          if (!half && (x0 + 64 <= p.N || (p.N & 7) == 0)) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && x0 < p.N && y0w < p.M)  // boxes entirely outside D are skipped
              tma_store_2d(&tmD, smem_u32(stage + q * 32 * 128), x0, y0w);
            if (lane == 0) bulk_commit();
          } else {
            // by rows: the chunk that crosses an N off the 16-byte grid, or
            // the half chunk (a 64-column box would reach into the next tile)
            __syncwarp();
            st_d_chunk_rows(stage + q * 32 * 128, static_cast<uint16_t*>(p.D), p.d_rs, y0w, x0,
                            p.M, half ? min(p.N, x0 + 32) : p.N, lane);
            __syncwarp();  // read out before the buffer takes a later chunk
          }
          const int j = c >> 1;  // this chunk
          if (use_ctma && j + 2 < NCHUNK) {
            // chunk j + 2's C into this buffer once the store has read it
            if (lane == 0) {
              bulk_wait_read_all();
              load_ct(staged & 1u, w.n0 + 64 * (j + 2), y0w);
            }
            ctn += 1u << (8u * (staged & 1u));
          }
          ++staged;
        }
      };
      // Typed paths: staged 16-bit D with C of the same type read by rows,
      // or no C; everything else takes the generic path.  The choice must be
      // the same for all 128 threads (the slices hold warp-wide barriers):
      // it depends on the call only, and ragged tiles take it too (their C
      // loads are masked; D is clipped at M by the TMA store and at N by the
      // TMA store or, for the chunk that crosses an N off 16 bytes, by rows).
      const bool c_typed = p.C != nullptr && p.c_vec && p.c_type == p.d_type;
      const bool typed = staged_store && (p.C == nullptr || c_typed);
      const int kind = !typed ? 0 : (p.C ? 1 : 2) + (p.d_type == T_F16 ? 2 : 0);
#pragma unroll 1
      for (int c = 0; c < BN / 32; c += 2) {
        switch (kind) {
          case 1:
            slice(c, cb0, pb0, IntTag<T_BF16>{}, IntTag<T_BF16>{});
            if (c + 1 < BN / 32) slice(c + 1, cb1, pb1, IntTag<T_BF16>{}, IntTag<T_BF16>{});
            break;
          case 2:
            slice(c, cb0, pb0, IntTag<0>{}, IntTag<T_BF16>{});
            if (c + 1 < BN / 32) slice(c + 1, cb1, pb1, IntTag<0>{}, IntTag<T_BF16>{});
            break;
          case 3:
            slice(c, cb0, pb0, IntTag<T_F16>{}, IntTag<T_F16>{});
            if (c + 1 < BN / 32) slice(c + 1, cb1, pb1, IntTag<T_F16>{}, IntTag<T_F16>{});
            break;
          case 4:
            slice(c, cb0, pb0, IntTag<0>{}, IntTag<T_F16>{});
            if (c + 1 < BN / 32) slice(c + 1, cb1, pb1, IntTag<0>{}, IntTag<T_F16>{});
            break;
          default:
            slice(c, cb0, pb0, IntTag<-1>{}, IntTag<-1>{});
            if (c + 1 < BN / 32) slice(c + 1, cb1, pb1, IntTag<-1>{}, IntTag<-1>{});
            break;
        }
      }
      if (leaves_partial) {
        // Publish: every epilogue thread of this CTA has written its row.
        __threadfence();
        named_barrier_sync(1, 128);
        if (ep_leader) {
          __threadfence();
          st_release_gpu(flag, p.epoch);
        }
      }
      ++acc_it;
    }
    // Shared memory must outlive the stores that read it and the C loads
    // still in flight (after a timeout) must land.
    if (lane == 0) {
      for (uint32_t b = 0; b < 2; ++b)
        if ((ctn >> (8u * b)) & 0xFFu) drain_wait(cbar(ew, b), (ctw >> b) & 1u, 200000000ull);
      bulk_wait_all();
    }
    }
  }

  if (threadIdx.x == 64) trace_at(p, 6);
  tc_fence_before();
  cluster_sync_all();
  if (threadIdx.x == 64) trace_at(p, 7);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace gb300
