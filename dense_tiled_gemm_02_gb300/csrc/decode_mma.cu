// decode_mma.cu -- the decode regime on the warp-level tensor-core
// instruction: D = A*B + C for M <= 16 rows, B in either layout.
//
// At a handful of rows the multiply is bound by reading B once (2*N*K
// bytes); the arithmetic per B element grows with M (16 multiply-adds at
// M = 16, more than the CUDA cores sustain at HBM speed), so the products go
// to the tensor core, but through mma.sync.m16n8k16 (fp16 or bf16 in, fp32
// accumulate) fed straight from registers: each thread loads its B fragment
// elements from global memory with 16-byte loads, A's rows (zero-padded to 8
// or 16) come from shared memory, and no B tile is staged anywhere.  A 128-row
// tcgen05 tile would stage B through shared memory for 16 useful rows.
//
// The sum over K is the Triton loop of the "Hopper Support in Triton" slide 5
// (acc += dot(a, b) per K block), split over blocks ("SPLIT_K", slides 14-15);
// D = sum + C ("DCU K100" article, 5.2).
//
// Because a sum over K may visit K in any order, the fragment positions of
// K are assigned to whatever memory positions make the loads long and
// contiguous; A is read with the same assignment, so every product pairs
// A(m, k) with B(k, n) of the same k.  Likewise the n of a fragment is mapped
// to whichever column the thread loaded, and D is stored through the same map.
//
// Two forms:
//  * K-contiguous B (element (k, n) at B[n * ldb + k], a weight stored N x K):
//    warp w of a block owns 8 columns; per step thread (g, t) (g = lane / 4,
//    t = lane % 4) loads 32 consecutive K of column g, so a warp reads 256
//    contiguous bytes of each of its 8 columns' rows; the 32 K feed 8 MMAs.
//  * N-contiguous B (element (k, n) at B[k * ldb + n]): the block's 4 warps
//    share 128 columns and interleave over K in 16-row steps; thread (g, t)
//    loads columns 16g .. 16g+15 of rows 2t, 2t+1, 2t+8, 2t+9 of the step (a
//    warp reads 256 contiguous bytes of each of 16 rows) and pairs the rows'
//    16-bit elements with a byte permute, one MMA per column j: MMA j covers
//    the columns 16g' + j of all eight g'.  The warps' sums are added in
//    shared memory in warp order.
//
// Each block writes the fp32 partial sums of its K slice; the last of a
// column block's slices (a counter) adds them in slice order, adds C, stores
// D and resets the counter, as in decode.cu: deterministic, one launch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.h"
#include "ptx.cuh"
#include "tc_launch.h"

namespace gb300 {

namespace {

constexpr int DM_KC_THREADS = 256;  // K-contiguous form: 8 warps x 8 columns
constexpr int DM_KC_COLS = 64;
constexpr int DM_KC_STEP = 128;     // K per warp step (4 threads x 32)
constexpr int DM_NC_THREADS = 128;  // N-contiguous form: 4 warps on 128 columns
constexpr int DM_NC_COLS = 128;
constexpr int DM_NC_STEP = 16;      // K per warp step
constexpr int DM_PAD = 8;           // elements of padding per A row in shared memory

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ float dm_load(const void* base, int t, long long off) {
  if (t == T_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[off]);
  if (t == T_F16) return __half2float(static_cast<const __half*>(base)[off]);
  return static_cast<const float*>(base)[off];
}

__device__ __forceinline__ void dm_store(void* base, int t, long long off, float v) {
  if (t == T_BF16)
    static_cast<__nv_bfloat16*>(base)[off] = __float2bfloat16_rn(v);
  else if (t == T_F16)
    static_cast<__half*>(base)[off] = __float2half_rn(v);
  else
    static_cast<float*>(base)[off] = v;
}

// A's rows 0 .. MT-1 over K [k0, k0 + kn) into shared memory (row stride
// kc + DM_PAD elements); rows at or past M and K past kn are zeros.
template <int MT>
__device__ __forceinline__ void stage_a(const DecodeArgs& d, uint16_t* sA, int k0, int kn,
                                        int nthreads) {
  const int ld = d.kc + DM_PAD;
  const bool vec = d.a_cs == 1 && (d.M == 1 || d.a_rs % 8 == 0) &&
                   (reinterpret_cast<uintptr_t>(d.A) & 15u) == 0 && (k0 & 7) == 0 && (kn & 7) == 0;
  if (vec) {
    const int cpr = d.kc / 8;  // 16-byte chunks per row
    for (int i = threadIdx.x; i < MT * cpr; i += nthreads) {
      const int m = i / cpr, c = i - m * cpr;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < d.M && 8 * c < kn)
        v = *reinterpret_cast<const uint4*>(d.A + m * d.a_rs + k0 + 8 * c);  // kn % 8 == 0
      *reinterpret_cast<uint4*>(sA + m * ld + 8 * c) = v;
    }
  } else {
    for (int i = threadIdx.x; i < MT * d.kc; i += nthreads) {
      const int m = i / d.kc, kk = i - m * d.kc;
      sA[m * ld + kk] = (m < d.M && kk < kn)
                            ? d.A[m * d.a_rs + static_cast<long long>(k0 + kk) * d.a_cs]
                            : uint16_t(0);
    }
  }
}

// The last block of column block `cb` (after every slice wrote its partials)
// adds the partials in slice order, adds C, stores D, resets the counter.
__device__ __forceinline__ void finish_columns(const DecodeArgs& d, int n_begin, int ncols,
                                               int nthreads) {
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned old = atomicAdd(d.counters + blockIdx.x, 1u);
    last = old == static_cast<unsigned>(d.splits) - 1u;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int i = threadIdx.x; i < d.M * ncols; i += nthreads) {
    const int m = i / ncols, n = n_begin + (i - m * ncols);
    if (n >= d.N) continue;
    float v = 0.f;
    for (int sl = 0; sl < d.splits; ++sl)
      v += d.ws[sl * d.ws_split + m * d.ws_rs + static_cast<long long>(n) * d.ws_cs];
    if (d.C) v += dm_load(d.C, d.c_type, m * d.c_rs + static_cast<long long>(n) * d.c_cs);
    dm_store(d.D, d.d_type, m * d.d_rs + static_cast<long long>(n) * d.d_cs, v);
  }
  if (threadIdx.x == 0) d.counters[blockIdx.x] = 0u;  // ready for the next call
}

// ---------------------------------------------------------------- K-contiguous B
// VEC: B 16-byte aligned with ldb a multiple of 8 (16-byte loads), else
// 2-byte loads of the same elements.
template <bool BF16, int MT, bool VEC>
__global__ void __launch_bounds__(DM_KC_THREADS) decode_mma_kc_kernel(const DecodeArgs d) {
  extern __shared__ __align__(16) uint16_t sA[];  // [MT][kc + DM_PAD]
  pdl_wait();
  pdl_trigger();
  const int k0 = blockIdx.y * d.kc;
  const int kn = min(d.kc, d.K - k0);
  stage_a<MT>(d, sA, k0, kn, DM_KC_THREADS);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n = blockIdx.x * DM_KC_COLS + warp * 8 + g;  // the column this thread loads
  const bool n_ok = n < d.N;
  const uint16_t* brow = d.B + static_cast<long long>(n_ok ? n : 0) * d.ldb + k0;
  const int ld = d.kc + DM_PAD;
  const uint16_t* a_lo = sA + g * ld;
  const uint16_t* a_hi = sA + (g + 8) * ld;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};

  // Two steps' loads in flight before the first use.
  constexpr int U = 2;
  for (int kb = 0; kb < kn; kb += U * DM_KC_STEP) {
    uint4 b[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int kk = kb + u * DM_KC_STEP + 32 * t + 8 * q;
        if (!n_ok || kk >= kn) {
          b[u][q] = make_uint4(0u, 0u, 0u, 0u);
        } else if (VEC) {
          b[u][q] = ld_global_v4_pinned(brow + kk);
        } else {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = brow[kk + 2 * e] | (static_cast<uint32_t>(brow[kk + 2 * e + 1]) << 16);
          b[u][q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ks = kb + u * DM_KC_STEP + 32 * t;  // this thread's 32 K of the step
      if (kb + u * DM_KC_STEP >= kn) break;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 alo = *reinterpret_cast<const uint4*>(a_lo + ks + 8 * q);
        const uint4 ahi = MT > 8 ? *reinterpret_cast<const uint4*>(a_hi + ks + 8 * q)
                                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int h = 0; h < 2; ++h)  // MMA j = 2q + h: elements 4j .. 4j+3 of the 32
          mma16816<BF16>(acc, word(alo, 2 * h), word(ahi, 2 * h), word(alo, 2 * h + 1),
                         word(ahi, 2 * h + 1), word(b[u][q], 2 * h), word(b[u][q], 2 * h + 1));
      }
    }
  }
  // acc: rows g and g + 8, columns 2t and 2t + 1 of the warp's 8.
  float* out = d.ws + blockIdx.y * d.ws_split;
  const int nc = blockIdx.x * DM_KC_COLS + warp * 8 + 2 * t;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = g + 8 * (i >> 1), c = nc + (i & 1);
    if (m < d.M && c < d.N) out[m * d.ws_rs + static_cast<long long>(c) * d.ws_cs] = acc[i];
  }
  finish_columns(d, blockIdx.x * DM_KC_COLS, DM_KC_COLS, DM_KC_THREADS);
}

// ---------------------------------------------------------------- N-contiguous B
// VEC: B 16-byte aligned with ldb and N multiples of 8 (16-byte loads), else
// 2-byte loads.
template <bool BF16, int MT, bool VEC>
__global__ void __launch_bounds__(DM_NC_THREADS) decode_mma_nc_kernel(const DecodeArgs d) {
  extern __shared__ __align__(16) uint16_t sA[];  // [MT][kc + DM_PAD], then the warp sums
  pdl_wait();
  pdl_trigger();
  const int k0 = blockIdx.y * d.kc;
  const int kn = min(d.kc, d.K - k0);
  stage_a<MT>(d, sA, k0, kn, DM_NC_THREADS);
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int c0 = blockIdx.x * DM_NC_COLS + 16 * g;  // this thread's 16 columns
  const int ld = d.kc + DM_PAD;
  const uint16_t* a_lo = sA + g * ld;
  const uint16_t* a_hi = sA + (g + 8) * ld;
  float acc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

  // 16 columns of row r (K index within the slice) as two 16-byte words.
  auto load_row = [&](int r, uint4& lo, uint4& hi) {
    lo = hi = make_uint4(0u, 0u, 0u, 0u);
    if (r >= kn) return;
    const uint16_t* p = d.B + static_cast<long long>(k0 + r) * d.ldb + c0;
    if (VEC) {
      if (c0 < d.N) lo = ld_global_v4_pinned(p);
      if (c0 + 8 < d.N) hi = ld_global_v4_pinned(p + 8);
    } else {
      uint32_t w[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t x0 = c0 + 2 * e < d.N ? p[2 * e] : 0u;
        const uint32_t x1 = c0 + 2 * e + 1 < d.N ? p[2 * e + 1] : 0u;
        w[e] = x0 | (x1 << 16);
      }
      lo = make_uint4(w[0], w[1], w[2], w[3]);
      hi = make_uint4(w[4], w[5], w[6], w[7]);
    }
  };

  constexpr int U = 2;  // steps whose loads are in flight together
  const int nsteps = (kn + DM_NC_STEP - 1) / DM_NC_STEP;
  for (int s0 = warp; s0 < nsteps; s0 += U * 4) {
    uint4 rw[U][4][2];  // [step][row 2t, 2t+1, 2t+8, 2t+9][columns 0-7, 8-15]
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int kb = (s0 + 4 * u) * DM_NC_STEP;
      const int rows[4] = {kb + 2 * t, kb + 2 * t + 1, kb + 2 * t + 8, kb + 2 * t + 9};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (s0 + 4 * u < nsteps)
          load_row(rows[i], rw[u][i][0], rw[u][i][1]);
        else
          rw[u][i][0] = rw[u][i][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (s0 + 4 * u >= nsteps) break;
      const int kb = (s0 + 4 * u) * DM_NC_STEP;
      const uint32_t a0 = *reinterpret_cast<const uint32_t*>(a_lo + kb + 2 * t);
      const uint32_t a2 = *reinterpret_cast<const uint32_t*>(a_lo + kb + 2 * t + 8);
      const uint32_t a1 = MT > 8 ? *reinterpret_cast<const uint32_t*>(a_hi + kb + 2 * t) : 0u;
      const uint32_t a3 = MT > 8 ? *reinterpret_cast<const uint32_t*>(a_hi + kb + 2 * t + 8) : 0u;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int half = j >> 3, wi = (j & 7) >> 1;
        const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;  // upper or lower 16 bits
        const uint32_t b0 = __byte_perm(word(rw[u][0][half], wi), word(rw[u][1][half], wi), sel);
        const uint32_t b1 = __byte_perm(word(rw[u][2][half], wi), word(rw[u][3][half], wi), sel);
        mma16816<BF16>(acc[j], a0, a1, a2, a3, b0, b1);
      }
    }
  }
  // Add the four warps' sums in warp order (shared memory after A's rows).
  float* red = reinterpret_cast<float*>(sA + MT * ld + 8);  // 16-byte aligned (ld % 8 == 0)
  __syncthreads();
  if (warp > 0) {
    float* dst = red + ((warp - 1) * 32 + lane) * 64;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      *reinterpret_cast<float4*>(dst + 4 * j) =
          make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
  }
  __syncthreads();
  if (warp == 0) {
    for (int w = 1; w < 4; ++w) {
      const float* src = red + ((w - 1) * 32 + lane) * 64;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(src + 4 * j);
        acc[j][0] += v.x;
        acc[j][1] += v.y;
        acc[j][2] += v.z;
        acc[j][3] += v.w;
      }
    }
    // MMA j: acc rows g (0, 1) and g + 8 (2, 3); logical columns 2t and
    // 2t + 1, which are the block's columns 16 * (2t) + j and 16 * (2t+1) + j.
    float* out = d.ws + blockIdx.y * d.ws_split;
    const int cb = blockIdx.x * DM_NC_COLS;
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int m = g + 8 * (i >> 1), c = cb + 16 * (2 * t + (i & 1)) + j;
        if (m < d.M && c < d.N) out[m * d.ws_rs + static_cast<long long>(c) * d.ws_cs] = acc[j][i];
      }
  }
  finish_columns(d, blockIdx.x * DM_NC_COLS, DM_NC_COLS, DM_NC_THREADS);
}

template <typename K>
cudaError_t launch_dm(K kernel, const DecodeArgs& d, int cols, int threads, size_t smem,
                      cudaStream_t st) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return cudaGetLastError();
  const dim3 grid(static_cast<unsigned>((d.N + cols - 1) / cols), static_cast<unsigned>(d.splits));
  return launch_pdl(kernel, grid, dim3(threads), smem, st, d);
}

template <bool BF16, int MT>
cudaError_t launch_mt(const DecodeArgs& d, cudaStream_t st) {
  const size_t smem = decode_mma_smem(d.M, d.kc, d.b_kcontig);
  const bool b16 = (reinterpret_cast<uintptr_t>(d.B) & 15u) == 0 && d.ldb % 8 == 0;
  if (d.b_kcontig) {
    return b16 ? launch_dm(decode_mma_kc_kernel<BF16, MT, true>, d, DM_KC_COLS, DM_KC_THREADS,
                           smem, st)
               : launch_dm(decode_mma_kc_kernel<BF16, MT, false>, d, DM_KC_COLS, DM_KC_THREADS,
                           smem, st);
  }
  return b16 && d.N % 8 == 0
             ? launch_dm(decode_mma_nc_kernel<BF16, MT, true>, d, DM_NC_COLS, DM_NC_THREADS,
                         smem, st)
             : launch_dm(decode_mma_nc_kernel<BF16, MT, false>, d, DM_NC_COLS, DM_NC_THREADS,
                         smem, st);
}

}  // namespace

int decode_mma_cols(bool b_kcontig) { return b_kcontig ? DM_KC_COLS : DM_NC_COLS; }
int decode_mma_kstep(bool b_kcontig) { return b_kcontig ? DM_KC_STEP : DM_NC_STEP; }

size_t decode_mma_smem(int M, int kc, bool b_kcontig) {
  const size_t mt = M <= 8 ? 8 : 16;
  const size_t a = mt * static_cast<size_t>(kc + DM_PAD) * sizeof(uint16_t);
  // N-contiguous form: three warps' 16 x 4 sums per lane after A's rows
  return b_kcontig ? a : a + 16 + 3 * 32 * 64 * sizeof(float);
}

cudaError_t launch_decode_mma(const DecodeArgs& d, cudaStream_t st) {
  const int step = decode_mma_kstep(d.b_kcontig);
  if (d.M < 1 || d.M > kDecodeMmaMaxRows || d.K < 1 || d.N < 1 || d.kc < step ||
      d.kc % step != 0 || d.splits < 1 || static_cast<long long>(d.kc) * d.splits < d.K ||
      (d.b_kcontig && d.K % 8 != 0))
    return cudaErrorInvalidValue;
  if (d.M <= 8) return d.bf16 ? launch_mt<true, 8>(d, st) : launch_mt<false, 8>(d, st);
  return d.bf16 ? launch_mt<true, 16>(d, st) : launch_mt<false, 16>(d, st);
}

}  // namespace gb300
