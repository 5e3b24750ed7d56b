// i8_mma.cu -- exact int8 GEMM on the native integer matrix instruction.
//
// D = A*B + C with int8 operands, int32 accumulation and int32 C and D, on
// the warp-level mma.sync.m16n8k32.s32.s8.s8.s32 instruction: every product
// and every partial sum is an exact integer (|sum| <= K * 2^14 stays far below
// 2^31 for K <= 2^16), so the result is exact with no chunking.  The pages
// compare a compiler builtin with hand-written inline assembly for the matrix
// instruction of their DCU ("DCU K100" article, section 5.3); this kernel is
// the inline-assembly form on this GPU's integer instruction, kept beside
// the exact-int8 path on the bf16 tensor cores (tcgen05) so that the two can
// be measured against each other.
//
// Tiles of 128 x 128 outputs, K in 64-byte slices through a 4-stage
// cp.async ring (zero fill beyond M, N and K: the masked K tail of the
// "Hopper Support in Triton" slides 14-15), eight warps of 64 x 32 outputs,
// operand fragments read with ldmatrix from 16-byte-chunk-swizzled rows, the
// grouped GROUP_M tile order (FlagGems "Hygon optimization").  Both operands
// are read K-contiguous; to_kmajor_i8_kernel makes such copies of operands
// stored the other way (or with rows off the 16-byte grid).
#include <cuda_runtime.h>

#include <cstdint>

#include "common.h"
#include "ptx.cuh"
#include "tc_launch.h"

namespace gb300 {

namespace {

constexpr int kTile = 128;        // output tile (both dimensions)
constexpr int kSlice = 64;        // K bytes per ring stage
constexpr int kStages = 4;
constexpr int kThreads = 256;     // 8 warps: 2 along M x 4 along N
constexpr uint32_t kOperandBytes = kTile * kSlice;       // one operand of one stage: 8 KB
constexpr uint32_t kStageBytes = 2 * kOperandBytes;
constexpr uint32_t kSmemBytes = kStages * kStageBytes;   // 64 KB

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// d += a * b over a 16 x 8 x 32 block; int8 operands, int32 accumulators.
__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A stage holds an operand as 128 rows of 64 bytes (four 16-byte chunks);
// chunk c of row r sits at chunk position c ^ ((r >> 1) & 3), so that the
// eight rows an ldmatrix reads at one logical chunk fall on distinct banks.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return static_cast<uint32_t>(r * kSlice + ((c ^ ((r >> 1) & 3)) << 4));
}

}  // namespace

__global__ void __launch_bounds__(kThreads) i8_mma_kernel(const I8Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  int64_t pm, pn;
  raster_tile(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
  const int m0 = static_cast<int>(pm) * kTile;
  const int n0 = static_cast<int>(pn) * kTile;
  const int nk = (p.K + kSlice - 1) / kSlice;
  const uint32_t s0 = smem_u32(smem);

  // Each thread copies two 16-byte chunks of A and two of B per stage:
  // chunk q = tid + 256 i is row q / 4, chunk q % 4.  Bytes past K, and rows
  // past M or N, read nothing and land as zeros.
  auto load_stage = [&](int kb, int s) {
    const uint32_t sa = s0 + s * kStageBytes;
    const uint32_t sb = sa + kOperandBytes;
    const int k0 = kb * kSlice;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int q = tid + i * kThreads;
      const int r = q >> 2;
      const int c = q & 3;
      const int k = k0 + c * 16;
      const int kb_left = min(16, max(0, p.K - k));
      const int ra = m0 + r;
      const int na = ra < p.M ? kb_left : 0;
      cp_async16(sa + sw_off(r, c), na > 0 ? p.A + static_cast<long long>(ra) * p.lda + k : p.A,
                 na);
      const int rb = n0 + r;
      const int nb = rb < p.N ? kb_left : 0;
      cp_async16(sb + sw_off(r, c), nb > 0 ? p.B + static_cast<long long>(rb) * p.ldb + k : p.B,
                 nb);
    }
  };

  const int wm = warp >> 2;  // rows wm*64 .. +63 of the tile
  const int wn = warp & 3;   // columns wn*32 .. +31
  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nk) load_stage(s, s);
    cp_async_commit();
  }
  for (int kb = 0; kb < nk; ++kb) {
    cp_async_wait<kStages - 2>();
    __syncthreads();  // stage kb has landed for all; stage kb - 1 is free again
    if (kb + kStages - 1 < nk) load_stage(kb + kStages - 1, (kb + kStages - 1) % kStages);
    cp_async_commit();
    const uint32_t sa = s0 + (kb % kStages) * kStageBytes;
    const uint32_t sb = sa + kOperandBytes;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {  // two 32-byte K steps per slice
      uint32_t a[4][4], b[4][2];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        // matrices: rows 0-7 / 8-15 of the 16-row block, K bytes 0-15 / 16-31
        const int r = wm * 64 + mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = 2 * ks + (lane >> 4);
        ldsm_x4(sa + sw_off(r, c), a[mi][0], a[mi][1], a[mi][2], a[mi][3]);
      }
#pragma unroll
      for (int nj = 0; nj < 2; ++nj) {
        // matrices: columns 0-7 at K bytes 0-15 and 16-31, then columns 8-15
        const int r = wn * 32 + nj * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int c = 2 * ks + ((lane >> 3) & 1);
        ldsm_x4(sb + sw_off(r, c), b[2 * nj][0], b[2 * nj][1], b[2 * nj + 1][0],
                b[2 * nj + 1][1]);
      }
#pragma unroll
      for (int mi = 0; mi < 4; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) mma_s8(acc[mi][ni], a[mi], b[ni][0], b[ni][1]);
    }
  }
  cp_async_wait<0>();

  // Thread (g = lane / 4, t = lane % 4) holds, per 16 x 8 block, rows g and
  // g + 8 at columns 2t and 2t + 1.  D = sum + C in int32.
  const int g = lane >> 2;
  const int t = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 4; ++mi)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = m0 + wm * 64 + mi * 16 + g + 8 * h;
      if (r >= p.M) continue;
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int c = n0 + wn * 32 + ni * 8 + 2 * t;
        int v0 = acc[mi][ni][2 * h];
        int v1 = acc[mi][ni][2 * h + 1];
        if (p.vec && c + 1 < p.N) {
          if (p.C) {
            const int2 cv = *reinterpret_cast<const int2*>(p.C + r * p.c_rs + c);
            v0 += cv.x;
            v1 += cv.y;
          }
          *reinterpret_cast<int2*>(p.D + r * p.d_rs + c) = make_int2(v0, v1);
        } else {
          if (c < p.N) {
            if (p.C) v0 += p.C[r * p.c_rs + c * p.c_cs];
            p.D[r * p.d_rs + c * p.d_cs] = v0;
          }
          if (c + 1 < p.N) {
            if (p.C) v1 += p.C[r * p.c_rs + (c + 1) * p.c_cs];
            p.D[r * p.d_rs + (c + 1) * p.d_cs] = v1;
          }
        }
      }
    }
}

// dst[r * ld_dst + k] = src[r * rs + k * ks] for r < rows, k < cols: an int8
// operand copied K-contiguous.  A block moves a 64 x 64 tile through shared
// memory, reading along the source's contiguous dimension and writing along
// K, so both sides are coalesced.
__global__ void __launch_bounds__(256) to_kmajor_i8_kernel(const int8_t* __restrict__ src,
                                                           long long rs, long long ks,
                                                           long long rows, long long cols,
                                                           int8_t* __restrict__ dst,
                                                           long long ld_dst) {
  __shared__ int8_t tile[64][65];
  pdl_wait();
  pdl_trigger();
  const long long k0 = static_cast<long long>(blockIdx.x) * 64;
  const bool r_fast = rs == 1 && ks != 1;  // the source is contiguous along r
  const long long row_tiles = (rows + 63) / 64;
  for (long long rt = blockIdx.y; rt < row_tiles; rt += gridDim.y) {
    const long long r0 = rt * 64;
#pragma unroll 4
    for (int i = threadIdx.x; i < 64 * 64; i += 256) {
      const int a = i & 63, b = i >> 6;
      const int rr = r_fast ? a : b, kk = r_fast ? b : a;
      const long long r = r0 + rr, k = k0 + kk;
      tile[rr][kk] = (r < rows && k < cols) ? src[r * rs + k * ks] : int8_t(0);
    }
    __syncthreads();
#pragma unroll 4
    for (int i = threadIdx.x; i < 64 * 64; i += 256) {
      const int kk = i & 63, rr = i >> 6;
      const long long r = r0 + rr, k = k0 + kk;
      if (r < rows && k < cols) dst[r * ld_dst + k] = tile[rr][kk];
    }
    __syncthreads();  // the tile is read out before the next rows land in it
  }
}

cudaError_t prepare_i8_mma() {
  return cudaFuncSetAttribute(i8_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kSmemBytes);
}

cudaError_t launch_i8_mma(const I8Params& p, cudaStream_t st) {
  const int grid = p.tiles_m * p.tiles_n;
  return launch_pdl(i8_mma_kernel, dim3(grid), dim3(kThreads), kSmemBytes, st, p);
}

cudaError_t launch_to_kmajor_i8(const int8_t* src, long long rs, long long ks, long long rows,
                                long long cols, int8_t* dst, long long ld_dst, cudaStream_t st) {
  const long long row_tiles = (rows + 63) / 64;
  const dim3 grid(static_cast<unsigned>((cols + 63) / 64),
                  static_cast<unsigned>(row_tiles < 65535 ? row_tiles : 65535));
  return launch_pdl(to_kmajor_i8_kernel, grid, dim3(256), 0, st, src, rs, ks, rows, cols, dst,
                    ld_dst);
}

}  // namespace gb300
