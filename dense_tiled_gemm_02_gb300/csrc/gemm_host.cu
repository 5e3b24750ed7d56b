// gemm_host.cu -- the C ABI: validation, plan selection, workspace, tensor
// maps and launches.  See include/gemm.h for the contract of each entry.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "common.h"
#include "gemm.h"
#include "plan_table.h"
#include "tc_launch.h"

using namespace gb300;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per device-side wait

int elem_size(int t) {
  switch (t) {
    case T_F16:
    case T_BF16: return 2;
    case T_F32:
    case T_I32: return 4;
    case T_I8:
    case T_E4M3:
    case T_E5M2:
    case T_MXE4M3:
    case T_MXE5M2: return 1;
    default: return 0;
  }
}

bool is_f16ish(int t) { return t == T_F16 || t == T_BF16; }
bool is_mx(int t) { return t == T_MXE4M3 || t == T_MXE5M2; }
bool is_f8(int t) { return t == T_E4M3 || t == T_E5M2 || is_mx(t); }

// One operand as the kernel sees it: storage pointer (user's or workspace),
// storage layout and leading dimension, logical rows x cols.
struct Operand {
  int layout;          // storage order of the internal operand
  int64_t ld;          // leading dimension (elements)
  int64_t rows, cols;  // logical extent (A': M' x K, B': K x N')
  bool repack;         // copy into ws before the TMA can read it
  bool lsu = false;    // read by the kernel's producer warps instead (rows off 16 bytes)
  int64_t ws_ld;       // leading dimension inside the workspace
  size_t ws_off;       // byte offset of its workspace copy
};

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// cluster = 0: a variant without cluster split-K; cluster >= 2: the one
// with the smallest cluster capacity that holds `cluster` splits.
const TcVariant* find_variant(int bn, bool i8x, int pw = 0, int cluster = 0) {
  const TcVariant* tabs[3] = {kVariantsBN256, kVariantsBN128, kVariantsBN64};
  const int counts[3] = {kNumVariantsBN256, kNumVariantsBN128, kNumVariantsBN64};
  const TcVariant* best = nullptr;
  for (int t = 0; t < 3; ++t)
    for (int i = 0; i < counts[t]; ++i) {
      const TcVariant& v = tabs[t][i];
      if (v.bn != bn || v.i8x != i8x || v.pw != pw) continue;
      if (cluster == 0 ? v.cs == 1 : (v.cs >= cluster && (!best || v.cs < best->cs))) {
        if (cluster == 0) return &v;
        best = &v;
      }
    }
  return best;
}

const PairVariant* find_pair(int bn, int ksub, bool i8x) {
  for (int i = 0; i < kNumPairVariants; ++i)
    if (kPairVariants[i].bn == bn && kPairVariants[i].ksub == ksub && kPairVariants[i].i8x == i8x)
      return &kPairVariants[i];
  return nullptr;
}

}  // namespace

struct gemm_plan {
  gemm_desc_t desc;
  int device = 0, num_sms = 0;
  PlanChoice choice{};
  const TcVariant* variant = nullptr;
  const PairVariant* pair = nullptr;  // set when the CTA-pair kernel runs the plan
  bool i8x = false;
  bool f8 = false;              // 8-bit float operands (kind::f8f6f4, K-major)
  bool mx = false;              // block-scaled 8-bit floats (kind::mxf8f6f4, gemm_run_mx)
  size_t ws_sfa_off = 0, ws_sfb_off = 0;  // packed scale cells of A and B
  int mab_type = T_BF16;        // type the tensor cores read (bf16 for int8 input)
  int64_t M = 0, N = 0, K = 0;  // internal problem
  Operand a{}, b{};
  int c_layout = 0, d_layout = 0;
  int64_t ldc = 0, ldd = 0;
  int grid = 0;
  KParams kp{};                 // everything but pointers
  void* ws = nullptr;
  size_t ws_bytes = 0;
  size_t ws_partial_off = 0;
  size_t ws_tail_off = 0, ws_flags_off = 0;  // last-wave partials and their flags
  size_t ws_fix_off = 0, ws_fixflag_off = 0;  // single-CTA stream-K partials and their flags
  // Native int8 (i8_mma.cu): the integer mma.sync kernel; A and B read
  // K-contiguous, copied so first when stored otherwise (a.repack, b.repack).
  bool native_i8 = false;
  // Decode regime (decode.cu): a handful of rows against a K-contiguous B.
  bool decode = false;
  int decode_kc = 0;
  // Bulk-copy form of the decode kernel (taken at run time when A and B are
  // 16-byte aligned; otherwise the split-K form planned beside it runs).
  bool decode_bulk = false;
  int decode_cpb = 0, decode_stages = 0, decode_cps = 0;
  // Tensor-core form of the decode regime (decode_mma.cu): M <= 16 rows, B
  // K-contiguous (decode_bk) or N-contiguous.
  bool decode_mma = false, decode_bk = true;
  // 16-bit C / D whose rows are not 16-byte aligned: aligned workspace copies
  // (leading dimension stage_ld) that the kernel reads / writes instead.
  bool c_stage = false, d_stage = false;
  size_t ws_c_off = 0, ws_d_off = 0;
  int64_t stage_ld = 0;
  uint32_t epoch = 0;                         // flag value of the latest run
  uint32_t* status = nullptr;
  int debug_flags = 0;
  unsigned long long* trace = nullptr;  // timeline hook (gemm_trace_set)
  uint64_t timeout_ns = kDefaultTimeoutNs;
  // Tensor maps of recently seen operand addresses (a few entries per
  // operand, replaced round-robin): encoding one costs microseconds of host
  // time, which short GEMMs cannot hide.
  static constexpr int kMapCache = 8;
  const void* map_ptr[4][kMapCache] = {};  // A', B', D, C
  CUtensorMap map[4][kMapCache] = {};
  int map_next[4] = {0, 0, 0, 0};
  std::string plan_str;
  // Kernel timing: event pairs recorded around the tensor-core launch of the
  // next timing_n runs (created by gemm_timing_enable, never by gemm_run).
  std::vector<cudaEvent_t> timing_ev;
  int timing_n = 0, timing_used = 0;
  // Host-buffer calls (gemm_host_io_enable / gemm_run_host_batch): two sets
  // of device copies of A, B, C, D, and three streams (copies in, GEMM,
  // copy out) with per-set events, so that one call's input copies overlap
  // the previous call's GEMM and output copy.
  bool io_ready = false;
  void* io_buf[2][4] = {};  // [set][A, B, C, D]
  size_t io_bytes[4] = {};
  cudaStream_t io_stream[3] = {};
  cudaEvent_t io_ev[2][3] = {};  // [set][inputs landed, GEMM done, D copied out]
  cudaEvent_t io_start = nullptr, io_end = nullptr;
  uint64_t io_calls = 0;
};

namespace {

int64_t packed_ld(int layout, int64_t rows, int64_t cols) {
  return layout == GEMM_ROW_MAJOR ? cols : rows;
}

bool valid_ld(int layout, int64_t ld, int64_t rows, int64_t cols) {
  const int64_t need = packed_ld(layout, rows, cols);
  return ld >= std::max<int64_t>(need, 1);
}

int validate(const gemm_desc_t& d) {
  if (d.M < 0 || d.N < 0 || d.K < 0) return GEMM_ERR_INVALID_ARG;
  if (d.M > INT32_MAX / 2 || d.N > INT32_MAX / 2 || d.K > INT32_MAX / 2) return GEMM_ERR_INVALID_ARG;
  for (int l : {d.layout_a, d.layout_b, d.layout_c, d.layout_d})
    if (l != GEMM_ROW_MAJOR && l != GEMM_COL_MAJOR) return GEMM_ERR_INVALID_ARG;
  const int ab = d.ab_type, c = d.c_type, o = d.d_type;
  if (is_f16ish(ab)) {
    if (!(is_f16ish(o) || o == T_F32)) return GEMM_ERR_UNSUPPORTED;
    if (!(is_f16ish(c) || c == T_F32 || c == 0)) return GEMM_ERR_UNSUPPORTED;
  } else if (ab == T_I8) {
    if (o != T_I32 || !(c == T_I32 || c == 0)) return GEMM_ERR_UNSUPPORTED;
  } else if (is_f8(ab)) {
    // 8-bit float operands (plain or block-scaled), read K-major only (A
    // row-major, B column-major)
    if (!(is_f16ish(o) || o == T_F32)) return GEMM_ERR_UNSUPPORTED;
    if (!(is_f16ish(c) || c == T_F32 || c == 0)) return GEMM_ERR_UNSUPPORTED;
    if (d.layout_a != GEMM_ROW_MAJOR || d.layout_b != GEMM_COL_MAJOR) return GEMM_ERR_UNSUPPORTED;
  } else {
    return GEMM_ERR_UNSUPPORTED;
  }
  if (!valid_ld(d.layout_a, d.lda, d.M, d.K) || !valid_ld(d.layout_b, d.ldb, d.K, d.N) ||
      !valid_ld(d.layout_c, d.ldc, d.M, d.N) || !valid_ld(d.layout_d, d.ldd, d.M, d.N))
    return GEMM_ERR_INVALID_ARG;
  return GEMM_OK;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

void apply_force_plan(PlanChoice& c) {
  const char* s = std::getenv("GEMM_FORCE_PLAN");
  if (!s) return;
  std::string str(s);
  size_t pos = 0;
  while (pos < str.size()) {
    size_t end = str.find(',', pos);
    if (end == std::string::npos) end = str.size();
    const std::string kv = str.substr(pos, end - pos);
    const size_t eq = kv.find('=');
    if (eq != std::string::npos) {
      const std::string k = kv.substr(0, eq);
      const int v = std::atoi(kv.c_str() + eq + 1);
      if (k == "bn") c.bn = v;
      else if (k == "splits") c.splits = v;
      else if (k == "group") c.group_m = v;
      else if (k == "swap") c.swap = v;
      else if (k == "grid") c.max_ctas = v;
      else if (k == "pair") c.pair = v;
      else if (k == "ksub") c.ksub = v;
      else if (k == "tail") c.tail = v;
      else if (k == "decode") c.no_decode = v ? 0 : 1;
      else if (k == "dbulk") c.no_dbulk = v ? -1 : 1;
      else if (k == "native_i8") c.native_i8 = v;
      else if (k == "sk") c.sk = v;
      else if (k == "kgroup") c.kgroup = v;
      else if (k == "lsu") c.lsu = v;
      else if (k == "i8chunk") c.i8chunk = v;
      else if (k == "dmma") c.dmma = v ? 1 : -1;
      else if (k == "csk") c.csk = v;
      else if (k == "skpat") c.skpat = v ? 0 : -1;
    }
    pos = end + 1;
  }
}

void make_plan_string(gemm_plan* h) {
  char buf[512];
  std::snprintf(buf, sizeof buf,
                "M=%lld N=%lld K=%lld decode=%d dbulk=%d swap=%d pair=%d bn=%d ksub=%d stages=%d "
                "group_m=%d splits=%d kb_per_split=%d tail=%d grid=%d i8x=%d a_mn=%d b_mn=%d "
                "repack_a=%d repack_b=%d stage_c=%d stage_d=%d ws_bytes=%zu native_i8=%d "
                "sk=%d kgroup=%d lsu_a=%d lsu_b=%d mx=%d i8chunk=%d dmma=%d csk=%d skchain=%d",
                (long long)h->desc.M, (long long)h->desc.N, (long long)h->desc.K, (int)h->decode,
                (int)h->decode_bulk,
                h->choice.swap,
                h->pair ? 1 : 0, h->choice.bn, h->choice.ksub,
                h->pair ? h->pair->stages : (h->variant ? h->variant->stages : 0), h->kp.group_m,
                h->kp.splits,
                h->kp.kb_per_split,
                h->kp.sk_len > 0 ? h->kp.tiles_m * h->kp.tiles_n - h->kp.sk_start : 0,
                h->grid, (int)h->i8x, h->kp.a_mn, h->kp.b_mn,
                (int)h->a.repack, (int)h->b.repack, (int)h->c_stage, (int)h->d_stage,
                h->ws_bytes, (int)h->native_i8, h->kp.sk1, h->kp.kgroup, (int)h->a.lsu,
                (int)h->b.lsu, (int)h->mx, h->choice.i8chunk, (int)h->decode_mma, h->kp.csk,
                h->kp.sk_n3);
  h->plan_str = buf;
}

// Plan of the decode kernel (no operand swap, no tensor maps): K split into
// slices so that about four blocks per SM stream B, the slices' fp32
// partials in the workspace, finished by the last block of each column
// block.  mma: the tensor-core form (decode_mma.cu) for up to 16 rows and
// either B layout.  Leaves h's workspace and status word allocated, or frees
// them and returns an error.
int plan_decode(gemm_plan* h, int sms, bool mma) {
  const gemm_desc_t& d = h->desc;
  h->decode = true;
  h->M = d.M;
  h->N = d.N;
  h->K = d.K;
  h->c_layout = d.layout_c;
  h->d_layout = d.layout_d;
  h->ldc = d.ldc;
  h->ldd = d.ldd;
  KParams& kp = h->kp;
  kp.M = (int)d.M;
  kp.N = (int)d.N;
  kp.K = (int)d.K;
  kp.c_type = d.c_type;
  kp.d_type = d.d_type;
  kp.c_rs = d.layout_c == GEMM_ROW_MAJOR ? d.ldc : 1;
  kp.c_cs = d.layout_c == GEMM_ROW_MAJOR ? 1 : d.ldc;
  kp.d_rs = d.layout_d == GEMM_ROW_MAJOR ? d.ldd : 1;
  kp.d_cs = d.layout_d == GEMM_ROW_MAJOR ? 1 : d.ldd;
  int64_t col_blocks = 0, s = 1, kc = 0;
  if (mma) {
    // Tensor-core form: blocks of decode_mma_cols() columns, K slices of a
    // whole number of warp steps, about three blocks per SM (two for the
    // N-contiguous form, whose partials hold all 128 columns of a block);
    // a slice of A (16 rows at most) stays below 64 KB of shared memory.
    h->decode_mma = true;
    h->decode_bk = d.layout_b == GEMM_COL_MAJOR;
    const int64_t cols = decode_mma_cols(h->decode_bk);
    const int64_t step = decode_mma_kstep(h->decode_bk);
    col_blocks = (d.N + cols - 1) / cols;
    const int64_t target = (int64_t)sms * (h->decode_bk ? 3 : 2);
    s = std::max<int64_t>(1, (target + col_blocks / 2) / col_blocks);
    s = std::min<int64_t>(s, std::max<int64_t>(1, (d.K + step - 1) / step));
    kc = round_up((d.K + s - 1) / s, step);
    kc = std::min<int64_t>(kc, 1920);
    s = (d.K + kc - 1) / kc;
  } else {
    // Slices of kc K elements (a multiple of 256, the width of one warp step;
    // at most 2048: a slice of A is at most 4 rows x 2048 x 2 bytes of shared
    // memory), as many as fill one wave of resident blocks: a second, partial
    // wave would double the time of the ones in it.
    col_blocks = (d.N + decode_columns_per_block() - 1) / decode_columns_per_block();
    const int64_t slots = (int64_t)sms * decode_blocks_per_sm((int)d.M, 1024);
    s = std::max<int64_t>(1, slots / col_blocks);
    s = std::min<int64_t>(s, std::max<int64_t>(1, d.K / 256));
    kc = round_up((d.K + s - 1) / s, 256);
    kc = std::min<int64_t>(kc, 2048);
    s = (d.K + kc - 1) / kc;
  }
  h->decode_kc = (int)kc;
  kp.splits = (int)s;
  // Bulk-copy form: when A's and B's rows are K-contiguous with strides of
  // whole 16-byte units, and N gives every SM at least four columns (below
  // that, the split-K form's parallelism over K wins), blocks of cpb whole
  // columns, as many as make whole waves of one block per SM.
  const bool a_k_rows = (d.layout_a == GEMM_ROW_MAJOR && (d.M == 1 || d.lda % 8 == 0)) ||
                        (d.M == 1 && d.layout_a == GEMM_COL_MAJOR && d.lda == 1);
  const int64_t cmax = 32;  // columns per block: four per consumer warp at most
  const int64_t waves = (d.N + cmax * sms - 1) / (cmax * sms);
  const int64_t cpb = std::min<int64_t>(cmax, (d.N + sms * waves - 1) / (sms * waves));
  int cps = 0;
  const int stages = decode_bulk_ring((int)d.M, d.K, (int)cpb, &cps);
  if (!mma && h->choice.no_dbulk != 1 && a_k_rows && d.ldb % 8 == 0 &&
      (stages * cps >= cpb || stages >= 2) &&
      (h->choice.no_dbulk == -1 || d.N >= 4 * (int64_t)sms)) {
    h->decode_bulk = true;
    h->decode_cpb = (int)cpb;
    h->decode_stages = stages;
    h->decode_cps = cps;
  }
  kp.kb_per_split = 0;
  const bool row = d.layout_d == GEMM_ROW_MAJOR;
  kp.ws_rs = row ? d.N : 1;
  kp.ws_cs = row ? 1 : d.M;
  kp.ws_split = d.M * d.N;
  h->ws_partial_off = 0;
  h->ws_flags_off = (size_t)round_up(s * d.M * d.N * 4, 256);  // per-column-block counters
  h->ws_bytes = h->ws_flags_off + (size_t)round_up(col_blocks * 4, 256);
  h->grid = (int)(col_blocks * s);
  if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    h->ws = nullptr;
    return GEMM_ERR_ALLOC_FAILED;
  }
  if (cudaMemset(static_cast<char*>(h->ws) + h->ws_flags_off, 0, col_blocks * 4) !=
      cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->ws);
    return GEMM_ERR_CUDA;
  }
  if (cudaMalloc(&h->status, 256) != cudaSuccess || cudaMemset(h->status, 0, 256) != cudaSuccess) {
    cudaGetLastError();
    if (h->status) cudaFree(h->status);
    cudaFree(h->ws);
    return GEMM_ERR_ALLOC_FAILED;
  }
  make_plan_string(h);
  return GEMM_OK;
}

// Plan of the native int8 kernel: 128 x 128 tiles in the grouped order, no
// split and no swap; A (M x K) and B (read as N rows of K) copied to
// K-contiguous workspace rows (128-byte lines) unless they already are
// K-contiguous with 16-byte rows.  Leaves h's workspace and status word
// allocated, or returns an error with nothing held.
int plan_native_i8(gemm_plan* h) {
  const gemm_desc_t& d = h->desc;
  PlanChoice& c = h->choice;
  h->native_i8 = true;
  c.swap = 0;
  c.pair = 0;
  c.splits = 1;
  c.tail = 0;
  c.bn = 128;
  c.ksub = 1;
  h->M = d.M;
  h->N = d.N;
  h->K = d.K;
  h->c_layout = d.layout_c;
  h->d_layout = d.layout_d;
  h->ldc = d.ldc;
  h->ldd = d.ldd;
  h->a = Operand{d.layout_a, d.lda, d.M, d.K, false, 0, 0};
  h->b = Operand{d.layout_b, d.ldb, d.K, d.N, false, 0, 0};
  h->a.repack = !(d.layout_a == GEMM_ROW_MAJOR && d.lda % 16 == 0);
  h->b.repack = !(d.layout_b == GEMM_COL_MAJOR && d.ldb % 16 == 0);
  const int64_t ldk = round_up(std::max<int64_t>(d.K, 1), 128);
  size_t off = 0;
  if (h->a.repack) {
    h->a.ws_ld = ldk;
    h->a.ws_off = off;
    off += (size_t)round_up(ldk * d.M, 256);
  }
  if (h->b.repack) {
    h->b.ws_ld = ldk;
    h->b.ws_off = off;
    off += (size_t)round_up(ldk * d.N, 256);
  }
  KParams& kp = h->kp;
  kp.M = (int)d.M;
  kp.N = (int)d.N;
  kp.K = (int)d.K;
  const int64_t tm = (d.M + 127) / 128, tn = (d.N + 127) / 128;
  if (tm * tn > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  kp.tiles_m = (int)tm;
  kp.tiles_n = (int)tn;
  kp.group_m = std::max(1, std::min(c.group_m, kp.tiles_m));
  kp.splits = 1;
  kp.num_kb = (int)((d.K + 63) / 64);
  kp.kb_per_split = kp.num_kb;
  kp.c_type = d.c_type;
  kp.d_type = d.d_type;
  kp.c_rs = d.layout_c == GEMM_ROW_MAJOR ? d.ldc : 1;
  kp.c_cs = d.layout_c == GEMM_ROW_MAJOR ? 1 : d.ldc;
  kp.d_rs = d.layout_d == GEMM_ROW_MAJOR ? d.ldd : 1;
  kp.d_cs = d.layout_d == GEMM_ROW_MAJOR ? 1 : d.ldd;
  h->grid = (int)(tm * tn);
  if (prepare_i8_mma() != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  h->ws_bytes = off;
  if (off > 0 && cudaMalloc(&h->ws, off) != cudaSuccess) {
    cudaGetLastError();
    h->ws = nullptr;
    return GEMM_ERR_ALLOC_FAILED;
  }
  if (cudaMalloc(&h->status, 256) != cudaSuccess || cudaMemset(h->status, 0, 256) != cudaSuccess) {
    cudaGetLastError();
    if (h->status) cudaFree(h->status);
    if (h->ws) cudaFree(h->ws);
    h->ws = nullptr;
    h->status = nullptr;
    return GEMM_ERR_ALLOC_FAILED;
  }
  make_plan_string(h);
  return GEMM_OK;
}

// Build the tiled tensor map of an internal operand (es-byte elements: 2,
// or 1 for 8-bit floats, which are K-major only).  K-major storage: dims
// {K, rows}, box {128 / es, box_rows} (one 128-byte row of K); MN-major
// storage (16-bit): dims {MN, K}, box {64, BK}; 128-byte swizzle; reads
// outside the tensor return zeros.
int encode_operand(CUtensorMap* tm, const void* base, int64_t ld, bool k_major, int64_t mn,
                   int64_t K, int box_rows, int es) {
  EncodeFn enc = get_encode();
  if (!enc) return GEMM_ERR_CUDA;
  cuuint64_t dims[2], strides[1];
  cuuint32_t box[2], estr[2] = {1, 1};
  if (k_major) {
    dims[0] = (cuuint64_t)K;
    dims[1] = (cuuint64_t)mn;
    box[0] = (cuuint32_t)(128 / es);
    box[1] = (cuuint32_t)box_rows;
  } else {
    dims[0] = (cuuint64_t)mn;
    dims[1] = (cuuint64_t)K;
    box[0] = 64;
    box[1] = BK;
  }
  strides[0] = (cuuint64_t)ld * es;
  CUresult r = enc(tm, es == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                   const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Tensor map of a row-contiguous 16-bit D (internal coordinates): dims
// {N, M}, box {64, 32} with 128-byte swizzle, for the per-warp stores from
// the staging buffers of the pair kernel.
int encode_store_d(CUtensorMap* tm, void* base, int64_t ld, int64_t M, int64_t N) {
  EncodeFn enc = get_encode();
  if (!enc) return GEMM_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Tensor map of a row-contiguous int32 C or D (internal coordinates): dims
// {N, M}, box {32, 32} (128 bytes x 32 rows) with 128-byte swizzle, for the
// exact-int8 pair kernel's per-warp C loads and D stores.
int encode_i32_tile(CUtensorMap* tm, const void* base, int64_t ld, int64_t M, int64_t N) {
  EncodeFn enc = get_encode();
  if (!enc) return GEMM_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// The cached tensor map of slot `which` for base (encoded on a miss).
template <typename Enc>
const CUtensorMap* cached_map(gemm_plan* h, int which, const void* base, Enc encode) {
  for (int i = 0; i < gemm_plan::kMapCache; ++i)
    if (h->map_ptr[which][i] == base) return &h->map[which][i];
  const int slot = h->map_next[which];
  h->map_next[which] = (slot + 1) % gemm_plan::kMapCache;
  h->map_ptr[which][slot] = nullptr;
  if (encode(&h->map[which][slot]) != GEMM_OK) return nullptr;
  h->map_ptr[which][slot] = base;
  return &h->map[which][slot];
}

}  // namespace

namespace {
int run_impl(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
             const uint8_t* SA, const uint8_t* SB, gemm_stream_t stream);
}  // namespace

extern "C" {

const char* gemm_strerror(int s) {
  switch (s) {
    case GEMM_OK: return "success";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported type combination";
    case GEMM_ERR_MISALIGNED: return "misaligned operand pointer";
    case GEMM_ERR_CUDA: return "CUDA call or launch failed";
    case GEMM_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired";
    case GEMM_ERR_ALLOC_FAILED: return "allocation failed";
    case GEMM_ERR_NO_DEVICE: return "no sm_103 device is current";
    default: return "unknown status";
  }
}

int gemm_raster_tile(int64_t t, int64_t num_pid_m, int64_t num_pid_n, int64_t group_m,
                     int64_t* pid_m, int64_t* pid_n) {
  if (num_pid_m <= 0 || num_pid_n <= 0 || group_m <= 0 || !pid_m || !pid_n) return GEMM_ERR_INVALID_ARG;
  if (t < 0 || t >= num_pid_m * num_pid_n) return GEMM_ERR_INVALID_ARG;
  raster_tile(t, num_pid_m, num_pid_n, group_m, *pid_m, *pid_n);
  return GEMM_OK;
}

int gemm_decode_ring(int M, int64_t K, int cpb, int* cps, int64_t* smem_bytes) {
  if (M < 1 || M > kDecodeMaxRows || K <= 0 || cpb < 1 || cpb > 32 || !cps || !smem_bytes)
    return GEMM_ERR_INVALID_ARG;
  const int stages = decode_bulk_ring(M, K, cpb, cps);
  *smem_bytes = decode_bulk_smem(M, K, stages, *cps);
  return stages;
}

int gemm_pair_schedule(int64_t tiles_m, int64_t tiles_n, int64_t group_m, int num_kb, int ksub,
                       int clusters, int stream_k, int cid, int i, int64_t* out) {
  if (tiles_m <= 0 || tiles_n <= 0 || group_m <= 0 || num_kb <= 0 || ksub <= 0 ||
      clusters <= 0 || cid < 0 || cid >= clusters || i < 0)
    return GEMM_ERR_INVALID_ARG;
  KParams p{};
  p.tiles_m = (int)tiles_m;
  p.tiles_n = (int)tiles_n;
  p.group_m = (int)group_m;
  p.num_kb = num_kb;
  p.splits = 1;
  p.kb_per_split = num_kb;
  if (stream_k) plan_stream_k(tiles_m * tiles_n, clusters, num_kb, ksub, p, stream_k == 2);
  const PairWork pw = pair_work(p, ksub, cid, clusters);
  if (!out) return pw.n;
  if (i >= pw.n) return GEMM_ERR_INVALID_ARG;
  const Unit w = pair_unit(p, pw, ksub, cid, clusters, i, 1);
  out[0] = w.m0 / (2 * BM);  // tile row
  out[1] = w.n0;             // tile column (bn = 1)
  out[2] = w.kb0;
  out[3] = w.kb1;
  out[4] = w.tail;
  out[5] = w.part;
  out[6] = w.ti;
  return pw.n;
}

int gemm_cta_schedule(int64_t tiles_m, int64_t tiles_n, int64_t group_m, int num_kb, int splits,
                      int grid, int stream_k, int cta, int i, int64_t* out) {
  if (tiles_m <= 0 || tiles_n <= 0 || group_m <= 0 || num_kb <= 0 || splits <= 0 ||
      grid <= 0 || cta < 0 || cta >= grid || i < 0 || tiles_m * tiles_n > INT32_MAX / num_kb)
    return GEMM_ERR_INVALID_ARG;
  KParams p{};
  p.tiles_m = (int)tiles_m;
  p.tiles_n = (int)tiles_n;
  p.group_m = (int)group_m;
  p.num_kb = num_kb;
  p.sk1 = stream_k ? 1 : 0;
  p.splits = stream_k ? 1 : splits;
  p.kb_per_split = (num_kb + p.splits - 1) / p.splits;
  if (p.sk1 && (int64_t)grid > tiles_m * tiles_n * num_kb) return GEMM_ERR_INVALID_ARG;
  const CtaWork cw = cta_work(p, cta, grid);
  if (!out) return cw.n;
  if (i >= cw.n) return GEMM_ERR_INVALID_ARG;
  const Unit w = cta_unit(p, cw, cta, grid, i, 1, 1);
  out[0] = w.tile;
  out[1] = w.m0;  // tile row (bm = 1)
  out[2] = w.n0;  // tile column (bn = 1)
  out[3] = w.kb0;
  out[4] = w.kb1;
  out[5] = w.pieces;
  out[6] = w.piece;
  out[7] = (w.tail && w.part == 1) ? w.ti : -1;
  out[8] = w.tail ? sk_piece_cta(p, w.tile, w.piece, grid) : -1;
  return cw.n;
}

int gemm_create(gemm_handle_t* out, const gemm_desc_t* desc) {
  if (!out || !desc) return GEMM_ERR_INVALID_ARG;
  gemm_desc_t d = *desc;
  if (d.lda == 0) d.lda = packed_ld(d.layout_a, d.M, d.K);
  if (d.ldb == 0) d.ldb = packed_ld(d.layout_b, d.K, d.N);
  if (d.ldc == 0) d.ldc = packed_ld(d.layout_c, d.M, d.N);
  if (d.ldd == 0) d.ldd = packed_ld(d.layout_d, d.M, d.N);
  int v = validate(d);
  if (v != GEMM_OK) return v;

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GEMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;

  gemm_plan* h = new (std::nothrow) gemm_plan();
  if (!h) return GEMM_ERR_ALLOC_FAILED;
  h->desc = d;
  h->device = dev;
  h->num_sms = sms;
  h->i8x = (static_cast<int>(d.ab_type) == T_I8);
  h->f8 = is_f8(static_cast<int>(d.ab_type));
  h->mx = is_mx(static_cast<int>(d.ab_type));
  h->mab_type = h->i8x ? static_cast<int>(T_BF16)
                       : (h->mx ? (static_cast<int>(d.ab_type) == T_MXE5M2 ? static_cast<int>(T_E5M2)
                                                                          : static_cast<int>(T_E4M3))
                                : static_cast<int>(d.ab_type));

  if (d.M == 0 || d.N == 0) {
    // An empty D: nothing to read, compute or store (gemm_run returns at
    // once).  No plan, no workspace; the status word keeps gemm_get_status
    // uniform.  The planners below divide by tile and column-block counts.
    h->M = d.M;
    h->N = d.N;
    h->K = d.K;
    if (cudaMalloc(&h->status, 256) != cudaSuccess ||
        cudaMemset(h->status, 0, 256) != cudaSuccess) {
      cudaGetLastError();
      if (h->status) cudaFree(h->status);
      delete h;
      return GEMM_ERR_ALLOC_FAILED;
    }
    make_plan_string(h);
    *out = h;
    return GEMM_OK;
  }
  h->choice = choose_plan(d.M, d.N, d.K, d.ab_type, d.layout_a, d.layout_b, sms);
  apply_force_plan(h->choice);
  if (h->mx) {
    // Block-scaled 8-bit floats: the single-CTA kernel's 128 x 128 tile with
    // the producer warps that place the scales (no swap, split or stream-K).
    PlanChoice& m = h->choice;
    m.pair = 0;
    m.bn = 128;
    m.swap = 0;
    m.splits = 1;
    m.sk = 0;
    m.kgroup = 1;
    m.lsu = 0;
    m.no_decode = 1;
  }
  // Decode regime: a handful of rows, 16-bit operands.  Up to four rows
  // against a K-contiguous B take the CUDA-core forms (decode.cu).  The
  // warp-level tensor-core form (decode_mma.cu: up to 16 rows, B of either
  // layout) runs only when asked for (dmma=1): it measured slower than the
  // tcgen05 path at 1 and 16 rows with either B layout at N = K = 4096
  // (16 x 4096 x 4096: 23.1 against 16.3 us with K-contiguous B, 46.7
  // against 16.8 with N-contiguous B; 1 x 4096 x 4096 N-contiguous: 20.7
  // against 16.0) and slower than the bulk-copy form at one row (14.7
  // against 9.7).
  const bool f16ab = d.ab_type == GEMM_F16 || d.ab_type == GEMM_BF16;
  const bool dec_cuda = f16ab && d.M >= 1 && d.M <= kDecodeMaxRows &&
                        d.layout_b == GEMM_COL_MAJOR && d.K % 8 == 0 && d.K >= 256;
  const bool dec_mma = f16ab && d.M >= 1 && d.M <= kDecodeMmaMaxRows && d.K >= 1 &&
                       (d.layout_b == GEMM_ROW_MAJOR || d.K % 8 == 0);
  const bool use_mma = dec_mma && h->choice.dmma == 1;
  if (!h->choice.no_decode && (use_mma || dec_cuda)) {
    const int rc = plan_decode(h, sms, use_mma);
    if (rc != GEMM_OK) {
      delete h;
      return rc;
    }
    *out = h;
    return GEMM_OK;
  }
  if (h->i8x && h->choice.native_i8) {
    const int rc = plan_native_i8(h);
    if (rc != GEMM_OK) {
      delete h;
      return rc;
    }
    const char* lg = std::getenv("GEMM_LOG");
    if (lg && lg[0] == '1') std::fprintf(stderr, "[gemm] plan: %s\n", h->plan_str.c_str());
    *out = h;
    return GEMM_OK;
  }
  if (h->i8x) {
    // The exact-int8 kernels: the pair kernel's 256 x 256 tile or the
    // single-CTA 128 x 128 tile (each epilogue thread keeps 128 int32 sums in
    // registers), with no K split; the pair kernel's stream-K pieces pass
    // int32 partials.
    h->choice.bn = h->choice.pair ? 256 : 128;
    h->choice.splits = 1;
    if (!h->choice.pair) h->choice.tail = 0;
  }
  PlanChoice& c = h->choice;
  const bool swap = c.swap != 0;
  h->M = swap ? d.N : d.M;
  h->N = swap ? d.M : d.N;
  h->K = d.K;
  auto flip = [](int l) { return l == GEMM_ROW_MAJOR ? GEMM_COL_MAJOR : GEMM_ROW_MAJOR; };
  // Internal operands: A' is M' x K, B' is K x N'.  With the swap,
  // A' = B^T and B' = A^T read the user's buffers in the other order.
  h->a.layout = swap ? flip(d.layout_b) : d.layout_a;
  h->a.ld = swap ? d.ldb : d.lda;
  h->a.rows = h->M;
  h->a.cols = h->K;
  h->b.layout = swap ? flip(d.layout_a) : d.layout_b;
  h->b.ld = swap ? d.lda : d.ldb;
  h->b.rows = h->K;
  h->b.cols = h->N;
  h->c_layout = swap ? flip(d.layout_c) : d.layout_c;
  h->d_layout = swap ? flip(d.layout_d) : d.layout_d;
  h->ldc = d.ldc;
  h->ldd = d.ldd;

  // The pair kernel stages bn/2 columns of B per CTA; an N-major B needs
  // whole 64-column swizzle atoms there.
  const bool b_n_major = h->b.layout == GEMM_ROW_MAJOR;
  if (c.pair && b_n_major && (c.bn / 2) % 64 != 0) c.pair = 0;
  if (c.pair) {
    h->pair = find_pair(c.bn, c.ksub, h->i8x);
    if (!h->pair) h->pair = find_pair(c.bn, 1, h->i8x);
    if (!h->pair) c.pair = 0;
  }
  c.ksub = h->pair ? h->pair->ksub : 1;
  if (!c.pair && c.bn == 224) c.bn = 256;  // 224-wide tiles exist for the pair kernel only
  // In-kernel loads of 16-bit operand rows that are off the 16-byte grid
  // (instead of workspace copies): single-CTA kernel, 128- or 256-wide tiles.
  const bool lsu_ok = c.lsu && !c.pair && is_f16ish(d.ab_type) && (c.bn == 128 || c.bn == 256);
  h->a.lsu = lsu_ok && (h->a.ld * 2) % 16 != 0;
  h->b.lsu = lsu_ok && (h->b.ld * 2) % 16 != 0;
  if (!c.pair) {
    h->variant = find_variant(c.bn, h->i8x, (h->a.lsu || h->b.lsu || h->mx) ? 4 : 0);
    if (!h->variant) {
      delete h;
      return GEMM_ERR_UNSUPPORTED;
    }
  }
  const int tile_m = c.pair ? 2 * BM : BM;

  // Tile grid and K split.
  KParams& kp = h->kp;
  kp.M = (int)h->M;
  kp.N = (int)h->N;
  kp.K = (int)h->K;
  kp.tiles_m = (int)((h->M + tile_m - 1) / tile_m);
  kp.tiles_n = (int)((h->N + c.bn - 1) / c.bn);
  kp.group_m = std::max(1, std::min(c.group_m, kp.tiles_m));
  const int bk_el = h->f8 ? 2 * BK : BK;  // K per 128-byte row
  kp.num_kb = (int)((h->K + bk_el - 1) / bk_el);
  kp.f8 = h->f8 ? 1 : 0;
  int splits = std::max(1, std::min(c.splits, std::max(1, kp.num_kb)));
  kp.kb_per_split = kp.num_kb > 0 ? (kp.num_kb + splits - 1) / splits : 0;
  // a ring stage covers ksub K slices: splits start on stage boundaries
  kp.kb_per_split = (int)round_up(kp.kb_per_split, c.ksub);
  if (kp.kb_per_split > 0) splits = (kp.num_kb + kp.kb_per_split - 1) / kp.kb_per_split;
  kp.splits = splits;
  c.splits = splits;
  // Exact int8: K slices of one fp32 accumulation pass.  Every partial sum
  // of a pass is an integer of magnitude at most (pass K) * 2^14, exactly
  // representable in fp32 while below 2^24: at most 1023 K, so at most 15
  // slices of 64; a whole number of ring stages (ksub slices each).  The
  // longest pass is the default: every pass ends in a drain of the whole
  // accumulator, and 960-K passes measured 1591 TOPS at 8192^3 against
  // 1389 for 512-K passes (768: 1568).
  if (h->i8x) {
    const int want = c.i8chunk > 0 ? c.i8chunk / BK : 15;
    kp.kb_per_chunk = std::max(1, std::min(15, want)) / c.ksub * c.ksub;
    kp.kb_per_chunk = std::max(c.ksub, kp.kb_per_chunk);
    c.i8chunk = kp.kb_per_chunk * BK;
  } else {
    kp.kb_per_chunk = std::max(1, kp.num_kb);
    c.i8chunk = 0;
  }
  kp.kgroup = (c.kgroup == 2 || c.kgroup == 4) ? c.kgroup : 1;
  c.kgroup = kp.kgroup;
  kp.a_mn = h->a.layout == GEMM_COL_MAJOR ? 1 : 0;  // A' contiguous along M'
  kp.b_mn = h->b.layout == GEMM_ROW_MAJOR ? 1 : 0;  // B' contiguous along N'
  // element type code 1: bf16 (kind::f16) or E5M2 (kind::f8f6f4)
  kp.idesc = idesc_f16(h->mab_type == T_BF16 || h->mab_type == T_E5M2 ? 1u : 0u,
                       (uint32_t)kp.a_mn, (uint32_t)kp.b_mn, (uint32_t)tile_m, (uint32_t)c.bn);
  kp.mx = h->mx ? 1 : 0;
  if (h->mx) {
    kp.idesc = idesc_mxf8(h->mab_type == T_E5M2 ? 1u : 0u, (uint32_t)kp.a_mn, (uint32_t)kp.b_mn,
                          (uint32_t)tile_m, (uint32_t)c.bn);
    kp.nsb4 = kp.num_kb;  // a ring stage covers 128 K: four 32-element scale blocks
  }
  kp.c_type = d.c_type;
  kp.d_type = d.d_type;
  kp.c_rs = h->c_layout == GEMM_ROW_MAJOR ? h->ldc : 1;
  kp.c_cs = h->c_layout == GEMM_ROW_MAJOR ? 1 : h->ldc;
  kp.d_rs = h->d_layout == GEMM_ROW_MAJOR ? h->ldd : 1;
  kp.d_cs = h->d_layout == GEMM_ROW_MAJOR ? 1 : h->ldd;
  int max_ctas = sms;
  if (c.max_ctas > 0) max_ctas = std::min(max_ctas, c.max_ctas);
  // Single-CTA stream-K: one equal run of (tile, K slice) iterations per
  // CTA over every SM (at most one CTA per iteration, so no run is empty).
  kp.sk1 = 0;
  if (!c.pair && c.sk && !h->i8x) {
    const int64_t iters = (int64_t)kp.tiles_m * kp.tiles_n * std::max(1, kp.num_kb);
    if (iters <= INT32_MAX && kp.num_kb > 0) {
      kp.sk1 = 1;
      splits = 1;
      kp.splits = 1;
      c.splits = 1;
      kp.kb_per_split = kp.num_kb;
    }
  }
  const int64_t units = (int64_t)kp.tiles_m * kp.tiles_n *
                        (kp.sk1 ? std::max(1, kp.num_kb) : kp.splits);
  if (!c.pair) h->grid = (int)std::max<int64_t>(1, std::min<int64_t>(units, max_ctas));
  // Split-K over clusters: every unit its own CTA (no persistent loop), the
  // splits of a tile one cluster, their sums added through shared memory.
  kp.csk = 0;
  if (c.csk && !c.pair && !h->i8x && !kp.sk1 && !h->mx && !h->a.lsu && !h->b.lsu &&
      kp.splits >= 2 && units <= max_ctas) {
    const TcVariant* v = find_variant(c.bn, false, 0, kp.splits);
    if (v) {
      h->variant = v;
      kp.csk = kp.splits;
      h->grid = (int)units;
    }
  }

  // Kernel attributes and, for the pair kernel, how many 2-CTA clusters
  // can be resident at once (the persistent grid).
  const cudaError_t prep = h->pair ? h->pair->prepare() : h->variant->prepare();
  int clusters = 0;
  if (prep == cudaSuccess && h->pair) {
    clusters = h->pair->max_clusters();
    if (c.max_ctas > 0) clusters = std::min(clusters, c.max_ctas / 2);
  }
  if (prep != cudaSuccess || (h->pair && clusters <= 0)) {
    cudaGetLastError();
    delete h;
    return GEMM_ERR_CUDA;
  }
  // Stream-K hybrid: when the tiles leave a partial last wave, all full
  // waves but one run as whole tiles and the rest of the tiles' K stages
  // are dealt out as equal contiguous runs, one per cluster, so that the
  // clusters finish together.  Each run is at least one tile long, so a
  // tile is shared by at most two clusters.
  const int64_t tiles = (int64_t)kp.tiles_m * kp.tiles_n;
  kp.sk_dp = kp.sk_start = kp.sk_len = kp.sk_rem = 0;
  kp.sk_n3 = -1;
  if (h->pair && c.tail && kp.splits == 1)
    plan_stream_k(tiles, clusters, kp.num_kb, c.ksub, kp, c.skpat >= 0);
  const int64_t sk_slots = kp.sk_len > 0 ? clusters : 0;
  if (h->pair) h->grid = 2 * (int)std::max<int64_t>(1, std::min<int64_t>(
                                 kp.sk_len > 0 ? clusters : units, clusters));

  // Workspace: operand copies the TMA unit can read, split-K partials, and
  // the last-wave partials with their flags.
  size_t off = 0;
  auto plan_copy = [&](Operand& o, int64_t in_es) {
    const int64_t inner = o.layout == GEMM_ROW_MAJOR ? o.cols : o.rows;
    const int64_t outer = o.layout == GEMM_ROW_MAJOR ? o.rows : o.cols;
    o.repack = !o.lsu && (h->i8x || ((o.ld * in_es) % 16 != 0));
    if (!o.repack) return;
    const int64_t ws_es = h->f8 ? 1 : 2;  // bf16 (16-bit or widened int8) or 8-bit copies
    // Rows start on 128-byte lines: a TMA row of 128 bytes then reads four
    // 32-byte sectors, not five (measured: a B whose rows sat 16 bytes off
    // the line cost 10 % of the kernel time at 4096 x 4097 x 4096).
    o.ws_ld = round_up(std::max<int64_t>(inner, 1), 128 / ws_es);
    o.ws_off = off;
    off += (size_t)round_up(o.ws_ld * outer * ws_es, 256);
  };
  const int64_t in_es = elem_size(d.ab_type);
  plan_copy(h->a, in_es);
  plan_copy(h->b, in_es);
  if (kp.splits > 1 && !kp.csk) {
    h->ws_partial_off = off;
    off += (size_t)round_up((int64_t)kp.splits * h->M * h->N * 4, 256);
    const bool row = h->d_layout == GEMM_ROW_MAJOR;
    kp.ws_rs = row ? h->N : 1;
    kp.ws_cs = row ? 1 : h->M;
    kp.ws_split = h->M * h->N;
  }
  if (h->mx) {
    h->ws_sfa_off = off;
    off += (size_t)round_up((int64_t)kp.tiles_m * kp.nsb4 * 512, 256);
    h->ws_sfb_off = off;
    off += (size_t)round_up((int64_t)kp.tiles_n * kp.nsb4 * 512, 256);
  }
  if (kp.sk1) {
    h->ws_fix_off = off;
    off += (size_t)round_up((int64_t)h->grid * BM * c.bn * 4, 256);
    h->ws_fixflag_off = off;
    off += (size_t)round_up((int64_t)h->grid * 4, 256);
  }
  if (sk_slots > 0) {
    h->ws_tail_off = off;
    off += (size_t)round_up(sk_slots * 2 * BM * c.bn * 4, 256);
    h->ws_flags_off = off;
    off += (size_t)round_up(sk_slots * 2 * 4, 256);
  }
  // C and D rows (along the internal N) that are not 16-byte aligned keep
  // the kernels off their vector and TMA paths; an aligned copy costs one
  // extra pass over C or D, far less than scattered 2-byte accesses from
  // the epilogue (measured: the pair kernel moving such rows itself, one
  // row per warp access through its staging chunks, took 306 us at
  // 4095 x 4097 x 4099 against 121 us plus the copies).  Split-K plans
  // write D from the reduce kernel, which streams it anyway.
  auto is16 = [](int t) { return t == GEMM_F16 || t == GEMM_BF16; };
  if (kp.splits == 1) {
    h->c_stage = is16(d.c_type) && h->c_layout == GEMM_ROW_MAJOR && (h->ldc * 2) % 16 != 0;
    h->d_stage = is16(d.d_type) && h->d_layout == GEMM_ROW_MAJOR && (h->ldd * 2) % 16 != 0;
  }
  if (h->c_stage || h->d_stage) {
    h->stage_ld = round_up(std::max<int64_t>(h->N, 1), 64);  // 128-byte rows, as above
    const size_t bytes = (size_t)round_up(h->stage_ld * h->M * 2, 256);
    if (h->c_stage) {
      h->ws_c_off = off;
      off += bytes;
    }
    if (h->d_stage) {
      h->ws_d_off = off;
      off += bytes;
    }
  }
  h->ws_bytes = off;
  if (off > 0 && cudaMalloc(&h->ws, off) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return GEMM_ERR_ALLOC_FAILED;
  }
  if ((sk_slots > 0 &&
       cudaMemset(static_cast<char*>(h->ws) + h->ws_flags_off, 0, sk_slots * 2 * 4) !=
           cudaSuccess) ||
      (kp.sk1 && cudaMemset(static_cast<char*>(h->ws) + h->ws_fixflag_off, 0,
                            (size_t)h->grid * 4) != cudaSuccess)) {
    cudaGetLastError();
    cudaFree(h->ws);
    delete h;
    return GEMM_ERR_CUDA;
  }
  if (cudaMalloc(&h->status, 256) != cudaSuccess || cudaMemset(h->status, 0, 256) != cudaSuccess) {
    cudaGetLastError();
    if (h->status) cudaFree(h->status);
    if (h->ws) cudaFree(h->ws);
    delete h;
    return GEMM_ERR_ALLOC_FAILED;
  }
  make_plan_string(h);
  const char* lg = std::getenv("GEMM_LOG");
  if (lg && lg[0] == '1') std::fprintf(stderr, "[gemm] plan: %s\n", h->plan_str.c_str());
  *out = h;
  return GEMM_OK;
}

int gemm_run(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
             gemm_stream_t stream) {
  if (!h || h->mx) return GEMM_ERR_INVALID_ARG;  // block-scaled handles run with gemm_run_mx
  return run_impl(h, A, B, C, D, nullptr, nullptr, stream);
}

int gemm_run_mx(gemm_handle_t h, const void* A, const uint8_t* SA, const void* B,
                const uint8_t* SB, const void* C, void* D, gemm_stream_t stream) {
  if (!h || !h->mx) return GEMM_ERR_INVALID_ARG;
  if (h->desc.M > 0 && h->desc.N > 0 && h->desc.K > 0 && (!SA || !SB)) return GEMM_ERR_INVALID_ARG;
  return run_impl(h, A, B, C, D, SA, SB, stream);
}

}  // extern "C"

namespace {
int run_impl(gemm_handle_t h, const void* A, const void* B, const void* C, void* D,
             const uint8_t* SA, const uint8_t* SB, gemm_stream_t stream) {
  if (h->desc.M == 0 || h->desc.N == 0) return GEMM_OK;  // an empty D: nothing to do
  if (!D || (h->desc.K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  const gemm_desc_t& d = h->desc;
  const int es_ab = elem_size(d.ab_type);
  const int es_c = elem_size(d.c_type);
  const int es_d = elem_size(d.d_type);
  auto mis = [](const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
  if ((A && mis(A, es_ab)) || (B && mis(B, es_ab)) || (C && mis(C, es_c)) || mis(D, es_d))
    return GEMM_ERR_MISALIGNED;
  if (C && d.c_type == 0) return GEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) return GEMM_ERR_INVALID_ARG;

  KParams kp = h->kp;
  kp.C = C;
  kp.D = D;
  kp.status = h->status;
  kp.timeout_ns = h->timeout_ns;
  kp.debug_flags = h->debug_flags;
  h->debug_flags = 0;  // test hooks apply to one run
  kp.trace = h->trace;
  const bool row_order = h->d_layout == GEMM_ROW_MAJOR;
  auto set_vec = [&]() {
    kp.c_vec = (kp.C && kp.c_cs == 1 && (reinterpret_cast<uintptr_t>(kp.C) % 16) == 0 &&
                (kp.c_rs * es_c) % 16 == 0) ? 1 : 0;
    kp.d_vec = (kp.d_cs == 1 && (reinterpret_cast<uintptr_t>(kp.D) % 16) == 0 &&
                (kp.d_rs * es_d) % 16 == 0) ? 1 : 0;
  };
  set_vec();

  if (d.K == 0) {  // D = C
    kp.splits = 0;
    return launch_reduce(kp, row_order, h->num_sms, st) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
  }
  if (h->native_i8) {
    // A as M rows of K, B as N rows of K; copied K-contiguous when planned so.
    char* ws = static_cast<char*>(h->ws);
    const int8_t* ka = static_cast<const int8_t*>(A);
    const int8_t* kb = static_cast<const int8_t*>(B);
    if (h->a.repack) {
      int8_t* dst = reinterpret_cast<int8_t*>(ws + h->a.ws_off);
      const bool row = d.layout_a == GEMM_ROW_MAJOR;
      if (launch_to_kmajor_i8(ka, row ? d.lda : 1, row ? 1 : d.lda, d.M, d.K, dst, h->a.ws_ld,
                              st) != cudaSuccess)
        return GEMM_ERR_CUDA;
      ka = dst;
    } else if (mis(A, 16)) {
      return GEMM_ERR_MISALIGNED;
    }
    if (h->b.repack) {
      int8_t* dst = reinterpret_cast<int8_t*>(ws + h->b.ws_off);
      const bool col = d.layout_b == GEMM_COL_MAJOR;  // element (k, n) at B[k + n * ldb]
      if (launch_to_kmajor_i8(kb, col ? d.ldb : 1, col ? 1 : d.ldb, d.N, d.K, dst, h->b.ws_ld,
                              st) != cudaSuccess)
        return GEMM_ERR_CUDA;
      kb = dst;
    } else if (mis(B, 16)) {
      return GEMM_ERR_MISALIGNED;
    }
    I8Params ip;
    ip.M = kp.M;
    ip.N = kp.N;
    ip.K = kp.K;
    ip.tiles_m = kp.tiles_m;
    ip.tiles_n = kp.tiles_n;
    ip.group_m = kp.group_m;
    ip.A = ka;
    ip.lda = h->a.repack ? h->a.ws_ld : d.lda;
    ip.B = kb;
    ip.ldb = h->b.repack ? h->b.ws_ld : d.ldb;
    ip.C = static_cast<const int32_t*>(C);
    ip.c_rs = kp.c_rs;
    ip.c_cs = kp.c_cs;
    ip.D = static_cast<int32_t*>(D);
    ip.d_rs = kp.d_rs;
    ip.d_cs = kp.d_cs;
    ip.vec = (kp.d_cs == 1 && kp.d_rs % 2 == 0 && !mis(D, 8) &&
              (!C || (kp.c_cs == 1 && kp.c_rs % 2 == 0 && !mis(C, 8)))) ? 1 : 0;
    const bool timed = h->timing_used < h->timing_n;
    if (timed && cudaEventRecord(h->timing_ev[2 * h->timing_used], st) != cudaSuccess)
      return GEMM_ERR_CUDA;
    if (launch_i8_mma(ip, st) != cudaSuccess) return GEMM_ERR_CUDA;
    if (timed) {
      if (cudaEventRecord(h->timing_ev[2 * h->timing_used + 1], st) != cudaSuccess)
        return GEMM_ERR_CUDA;
      ++h->timing_used;
    }
    return GEMM_OK;
  }
  if (h->decode) {
    DecodeArgs a;
    a.A = static_cast<const uint16_t*>(A);
    a.a_rs = d.layout_a == GEMM_ROW_MAJOR ? d.lda : 1;
    a.a_cs = d.layout_a == GEMM_ROW_MAJOR ? 1 : d.lda;
    a.B = static_cast<const uint16_t*>(B);
    a.ldb = d.ldb;
    a.M = (int)d.M;
    a.N = (int)d.N;
    a.K = (int)d.K;
    a.kc = h->decode_kc;
    a.splits = kp.splits;
    a.bf16 = d.ab_type == GEMM_BF16;
    a.ws = static_cast<float*>(h->ws);
    a.ws_split = kp.ws_split;
    a.ws_rs = kp.ws_rs;
    a.ws_cs = kp.ws_cs;
    a.counters = reinterpret_cast<unsigned*>(static_cast<char*>(h->ws) + h->ws_flags_off);
    a.C = C;
    a.c_type = d.c_type;
    a.c_rs = kp.c_rs;
    a.c_cs = kp.c_cs;
    a.D = D;
    a.d_type = d.d_type;
    a.d_rs = kp.d_rs;
    a.d_cs = kp.d_cs;
    a.bulk = h->decode_bulk && reinterpret_cast<uintptr_t>(A) % 16 == 0 &&
             reinterpret_cast<uintptr_t>(B) % 16 == 0;
    a.cpb = h->decode_cpb;
    a.stages = h->decode_stages;
    a.cps = h->decode_cps;
    a.status = h->status;
    a.timeout_ns = h->timeout_ns;
    a.debug_flags = kp.debug_flags;
    a.mma = h->decode_mma;
    a.b_kcontig = h->decode_bk;
    const bool timed = h->timing_used < h->timing_n;
    if (timed && cudaEventRecord(h->timing_ev[2 * h->timing_used], st) != cudaSuccess)
      return GEMM_ERR_CUDA;
    if ((a.mma ? launch_decode_mma(a, st) : launch_decode(a, st)) != cudaSuccess)
      return GEMM_ERR_CUDA;
    if (timed) {
      if (cudaEventRecord(h->timing_ev[2 * h->timing_used + 1], st) != cudaSuccess)
        return GEMM_ERR_CUDA;
      ++h->timing_used;
    }
    return GEMM_OK;
  }
  char* ws = static_cast<char*>(h->ws);
  uint16_t* d_staged = nullptr;
  // The 16-bit copies before the GEMM (C staging, operand copies) go out
  // as one launch.
  CopyJob16 jobs[kMaxCopyJobs];
  int njobs = 0;
  if (h->c_stage && C) {
    uint16_t* cs = reinterpret_cast<uint16_t*>(ws + h->ws_c_off);
    jobs[njobs++] = CopyJob16{static_cast<const uint16_t*>(C), kp.c_rs, cs, h->stage_ld, h->M,
                              h->N};
    kp.C = cs;
    kp.c_rs = h->stage_ld;
  }
  if (h->d_stage) {
    d_staged = reinterpret_cast<uint16_t*>(ws + h->ws_d_off);
    kp.D = d_staged;
    kp.d_rs = h->stage_ld;
  }
  set_vec();

  const bool swap = h->choice.swap != 0;
  const void* pa = swap ? B : A;  // storage of A'
  const void* pb = swap ? A : B;  // storage of B'
  const void* ta = pa;
  const void* tb = pb;
  // Operands the TMA unit cannot read in place go through the workspace.
  for (int which = 0; which < 2; ++which) {
    Operand& o = which == 0 ? h->a : h->b;
    const void* src = which == 0 ? pa : pb;
    if (o.lsu) continue;  // read in place by the kernel's producer warps
    const bool need = o.repack || mis(src, 16);
    if (!need) continue;
    if (!o.repack) return GEMM_ERR_MISALIGNED;  // no workspace was planned for this operand
    const int64_t inner = o.layout == GEMM_ROW_MAJOR ? o.cols : o.rows;
    const int64_t outer = o.layout == GEMM_ROW_MAJOR ? o.rows : o.cols;
    uint16_t* dst = reinterpret_cast<uint16_t*>(ws + o.ws_off);
    if (d.ab_type == GEMM_I8 || h->f8) {  // int8 widened to bf16; 8-bit floats as bytes
      if (launch_repack(src, d.ab_type, o.ld, dst, o.ws_ld, outer, inner, h->num_sms, st) !=
          cudaSuccess)
        return GEMM_ERR_CUDA;
    } else {
      jobs[njobs++] = CopyJob16{static_cast<const uint16_t*>(src), o.ld, dst, o.ws_ld, outer,
                                inner};
    }
    (which == 0 ? ta : tb) = dst;
  }
  if (njobs > 0 && launch_copy16(jobs, njobs, h->num_sms, st) != cudaSuccess)
    return GEMM_ERR_CUDA;
  const int64_t lda_eff = h->a.repack ? h->a.ws_ld : h->a.ld;
  const int64_t ldb_eff = h->b.repack ? h->b.ws_ld : h->b.ld;

  const int b_box = h->pair ? h->choice.bn / 2 : h->choice.bn;  // B rows staged per CTA
  const CUtensorMap* tm[2] = {nullptr, nullptr};
  static const CUtensorMap kNoMap = {};  // an operand the TMA unit does not read
  kp.a_lsu = h->a.lsu ? 1 : 0;
  kp.b_lsu = h->b.lsu ? 1 : 0;
  kp.a_src = pa;
  kp.b_src = pb;
  kp.a_ld = h->a.ld;
  kp.b_ld = h->b.ld;
  for (int which = 0; which < 2; ++which) {
    const void* base = which == 0 ? ta : tb;
    if ((which == 0 ? h->a : h->b).lsu) {
      tm[which] = &kNoMap;
      continue;
    }
    for (int i = 0; i < gemm_plan::kMapCache; ++i)
      if (h->map_ptr[which][i] == base) tm[which] = &h->map[which][i];
    if (tm[which]) continue;
    const int slot = h->map_next[which];
    h->map_next[which] = (slot + 1) % gemm_plan::kMapCache;
    h->map_ptr[which][slot] = nullptr;
    const int rc = which == 0
                       ? encode_operand(&h->map[0][slot], ta, lda_eff, kp.a_mn == 0, h->M, h->K, BM,
                                        h->f8 ? 1 : 2)
                       : encode_operand(&h->map[1][slot], tb, ldb_eff, kp.b_mn == 0, h->N, h->K,
                                        b_box, h->f8 ? 1 : 2);
    if (rc != GEMM_OK) return GEMM_ERR_CUDA;
    h->map_ptr[which][slot] = base;
    tm[which] = &h->map[which][slot];
  }
  if (h->mx) {
    uint8_t* ca = reinterpret_cast<uint8_t*>(ws + h->ws_sfa_off);
    uint8_t* cb = reinterpret_cast<uint8_t*>(ws + h->ws_sfb_off);
    const int nsb = (int)((d.K + 31) / 32);
    if (launch_pack_scales(SA, (int)h->M, nsb, kp.nsb4, kp.tiles_m, ca, st) != cudaSuccess ||
        launch_pack_scales(SB, (int)h->N, nsb, kp.nsb4, kp.tiles_n, cb, st) != cudaSuccess)
      return GEMM_ERR_CUDA;
    kp.sfa = ca;
    kp.sfb = cb;
  }
  if (kp.splits > 1 && !kp.csk) kp.ws = reinterpret_cast<float*>(ws + h->ws_partial_off);
  if (kp.sk1) {
    kp.fix_ws = reinterpret_cast<float*>(ws + h->ws_fix_off);
    kp.fix_flag = reinterpret_cast<uint32_t*>(ws + h->ws_fixflag_off);
    if (++h->epoch == 0) h->epoch = 1;  // flags start at 0: never reuse it
    kp.epoch = h->epoch;
  }
  if (kp.sk_len > 0) {
    kp.tail_ws = reinterpret_cast<float*>(ws + h->ws_tail_off);
    kp.tail_flags = reinterpret_cast<uint32_t*>(ws + h->ws_flags_off);
    if (++h->epoch == 0) h->epoch = 1;  // flags start at 0: never reuse it
    kp.epoch = h->epoch;
  }
  // The pair kernel stores a 16-bit, row-contiguous D with TMA from swizzled
  // shared memory (rows 16-byte aligned, as TMA requires); its exact-int8
  // mode moves an int32 C and D that way.
  const CUtensorMap* tmd = tm[0];  // placeholder arguments when unused
  const CUtensorMap* tmc = tm[0];
  // A TMA store writes whole 16-byte units at the right edge of the tensor
  // (measured: a 700-column bf16 D in rows of 704 had columns 700-703
  // written).  The 16-bit path stores the chunk that crosses such an N by
  // rows instead (in the kernel); the int32 path of exact int8 takes TMA
  // only when N fills whole units.
  if (h->i8x) {
    kp.d_tma = (h->pair && kp.splits == 1 && kp.d_vec && (!C || kp.c_vec) && h->N % 4 == 0) ? 1
                                                                                            : 0;
    if (kp.d_tma) {
      void* dp = kp.D;
      const int64_t drs = kp.d_rs;
      tmd = cached_map(h, 2, dp, [&](CUtensorMap* m) {
        return encode_i32_tile(m, dp, drs, h->M, h->N);
      });
      if (!tmd) return GEMM_ERR_CUDA;
      if (C) {
        const void* cp = kp.C;
        const int64_t crs = kp.c_rs;
        tmc = cached_map(h, 3, cp, [&](CUtensorMap* m) {
          return encode_i32_tile(m, cp, crs, h->M, h->N);
        });
        if (!tmc) return GEMM_ERR_CUDA;
      }
    }
  } else {
    kp.d_tma = (h->pair && kp.splits == 1 && kp.d_vec &&
                (d.d_type == GEMM_BF16 || d.d_type == GEMM_F16)) ? 1 : 0;
    kp.c_tma = 0;
    if (kp.d_tma) {
      void* dp = kp.D;
      const int64_t drs = kp.d_rs;
      tmd = cached_map(h, 2, dp, [&](CUtensorMap* m) {
        return encode_store_d(m, dp, drs, h->M, h->N);
      });
      if (!tmd) return GEMM_ERR_CUDA;
      // A C of D's type with 16-byte rows comes in by TMA into the staging
      // buffers (the same 32 x 64 boxes, 128-byte swizzle).
      if (kp.C && kp.c_vec && d.c_type == d.d_type) {
        void* cp = const_cast<void*>(kp.C);
        const int64_t crs = kp.c_rs;
        tmc = cached_map(h, 3, cp, [&](CUtensorMap* m) {
          return encode_store_d(m, cp, crs, h->M, h->N);
        });
        if (!tmc) return GEMM_ERR_CUDA;
        kp.c_tma = 1;
      }
    }
  }
  const bool timed = h->timing_used < h->timing_n;
  if (timed && cudaEventRecord(h->timing_ev[2 * h->timing_used], st) != cudaSuccess)
    return GEMM_ERR_CUDA;
  const cudaError_t le = h->pair ? h->pair->launch(*tm[0], *tm[1], *tmd, *tmc, kp, h->grid, st)
                                 : h->variant->launch(*tm[0], *tm[1], kp, h->grid, st);
  if (le != cudaSuccess) return GEMM_ERR_CUDA;
  if (timed) {
    if (cudaEventRecord(h->timing_ev[2 * h->timing_used + 1], st) != cudaSuccess)
      return GEMM_ERR_CUDA;
    ++h->timing_used;
  }
  if (kp.splits > 1 && !kp.csk && launch_reduce(kp, row_order, h->num_sms, st) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (d_staged && launch_copy_out16(d_staged, h->stage_ld, static_cast<uint16_t*>(D), h->ldd,
                                    h->M, h->N, h->num_sms, st) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_get_status(gemm_handle_t h, gemm_stream_t stream) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaMemcpy(&word, h->status, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (word != 0 && cudaMemset(h->status, 0, sizeof word) != cudaSuccess) return GEMM_ERR_CUDA;
  return (word & STATUS_TIMEOUT) ? GEMM_ERR_DEVICE_TIMEOUT : GEMM_OK;
}

int gemm_destroy(gemm_handle_t h) {
  if (!h) return GEMM_OK;
  int rc = GEMM_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) rc = GEMM_ERR_CUDA;
  if (h->ws) cudaFree(h->ws);
  if (h->status) cudaFree(h->status);
  for (cudaEvent_t e : h->timing_ev) cudaEventDestroy(e);
  for (auto& set : h->io_buf)
    for (void* b : set)
      if (b) cudaFree(b);
  for (cudaStream_t s : h->io_stream)
    if (s) cudaStreamDestroy(s);
  for (auto& set : h->io_ev)
    for (cudaEvent_t e : set)
      if (e) cudaEventDestroy(e);
  if (h->io_start) cudaEventDestroy(h->io_start);
  if (h->io_end) cudaEventDestroy(h->io_end);
  delete h;
  return rc;
}

namespace {
// Bytes from an operand's first element to one past its last, in storage
// order (rows x cols, leading dimension ld).
size_t span_bytes(int layout, int64_t rows, int64_t cols, int64_t ld, int es) {
  if (rows <= 0 || cols <= 0) return 0;
  const int64_t outer = layout == GEMM_ROW_MAJOR ? rows : cols;
  const int64_t inner = layout == GEMM_ROW_MAJOR ? cols : rows;
  return (size_t)((outer - 1) * ld + inner) * (size_t)es;
}
}  // namespace

int gemm_host_io_enable(gemm_handle_t h) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  if (h->io_ready) return GEMM_OK;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) return GEMM_ERR_INVALID_ARG;
  const gemm_desc_t& d = h->desc;
  h->io_bytes[0] = span_bytes(d.layout_a, d.M, d.K, d.lda, elem_size(d.ab_type));
  h->io_bytes[1] = span_bytes(d.layout_b, d.K, d.N, d.ldb, elem_size(d.ab_type));
  h->io_bytes[2] = d.c_type ? span_bytes(d.layout_c, d.M, d.N, d.ldc, elem_size(d.c_type)) : 0;
  h->io_bytes[3] = span_bytes(d.layout_d, d.M, d.N, d.ldd, elem_size(d.d_type));
  if (d.M == 0 || d.N == 0)  // an empty D reads nothing: no operand is copied
    for (size_t& b : h->io_bytes) b = 0;
  bool ok = true;
  for (int s = 0; s < 2 && ok; ++s)
    for (int k = 0; k < 4 && ok; ++k)
      if (h->io_bytes[k]) ok = cudaMalloc(&h->io_buf[s][k], h->io_bytes[k]) == cudaSuccess;
  for (int k = 0; k < 3 && ok; ++k)
    ok = cudaStreamCreateWithFlags(&h->io_stream[k], cudaStreamNonBlocking) == cudaSuccess;
  for (int s = 0; s < 2 && ok; ++s)
    for (int k = 0; k < 3 && ok; ++k)
      ok = cudaEventCreateWithFlags(&h->io_ev[s][k], cudaEventDisableTiming) == cudaSuccess;
  if (ok) ok = cudaEventCreateWithFlags(&h->io_start, cudaEventDisableTiming) == cudaSuccess;
  if (ok) ok = cudaEventCreateWithFlags(&h->io_end, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return GEMM_ERR_ALLOC_FAILED;  // what was created is released by gemm_destroy
  }
  h->io_ready = true;
  return GEMM_OK;
}

int gemm_run_host_batch(gemm_handle_t h, int n, const void* const* A, const void* const* B,
                        const void* const* C, void* const* D, gemm_stream_t stream) {
  if (!h || n < 0 || (n > 0 && (!A || !B || !D))) return GEMM_ERR_INVALID_ARG;
  if (!h->io_ready) return GEMM_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)  // nothing is enqueued unless every pointer needed is there
    if ((h->io_bytes[0] && !A[i]) || (h->io_bytes[1] && !B[i]) || (h->io_bytes[3] && !D[i]))
      return GEMM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t s_in = h->io_stream[0], s_gemm = h->io_stream[1], s_out = h->io_stream[2];
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // Everything enqueued on `stream` before this call comes first.
  if (!ok(cudaEventRecord(h->io_start, st)) || !ok(cudaStreamWaitEvent(s_in, h->io_start, 0)))
    return GEMM_ERR_CUDA;
  for (int i = 0; i < n; ++i) {
    const int set = (int)(h->io_calls++ & 1u);
    void* const* buf = h->io_buf[set];
    cudaEvent_t* ev = h->io_ev[set];
    const void* hc = (C && h->io_bytes[2]) ? C[i] : nullptr;
    // The set's inputs are free once the GEMM that read them is done, its D
    // once that D has been copied out (an event never recorded is complete).
    if (!ok(cudaStreamWaitEvent(s_in, ev[1], 0))) return GEMM_ERR_CUDA;
    // An empty operand (M, N or K zero) has no device copy and is not copied.
    if ((h->io_bytes[0] &&
         !ok(cudaMemcpyAsync(buf[0], A[i], h->io_bytes[0], cudaMemcpyHostToDevice, s_in))) ||
        (h->io_bytes[1] &&
         !ok(cudaMemcpyAsync(buf[1], B[i], h->io_bytes[1], cudaMemcpyHostToDevice, s_in))))
      return GEMM_ERR_CUDA;
    if (hc && !ok(cudaMemcpyAsync(buf[2], hc, h->io_bytes[2], cudaMemcpyHostToDevice, s_in)))
      return GEMM_ERR_CUDA;
    if (!ok(cudaEventRecord(ev[0], s_in)) || !ok(cudaStreamWaitEvent(s_gemm, ev[0], 0)) ||
        !ok(cudaStreamWaitEvent(s_gemm, ev[2], 0)))
      return GEMM_ERR_CUDA;
    const int rc = gemm_run(h, buf[0], buf[1], hc ? buf[2] : nullptr, buf[3], s_gemm);
    if (rc != GEMM_OK) return rc;
    if (!ok(cudaEventRecord(ev[1], s_gemm)) || !ok(cudaStreamWaitEvent(s_out, ev[1], 0)) ||
        (h->io_bytes[3] &&
         !ok(cudaMemcpyAsync(D[i], buf[3], h->io_bytes[3], cudaMemcpyDeviceToHost, s_out))) ||
        !ok(cudaEventRecord(ev[2], s_out)))
      return GEMM_ERR_CUDA;
  }
  // `stream` continues once the last output copy has landed.
  if (!ok(cudaEventRecord(h->io_end, s_out)) || !ok(cudaStreamWaitEvent(st, h->io_end, 0)))
    return GEMM_ERR_CUDA;
  return GEMM_OK;
}

int gemm_plan_string(gemm_handle_t h, char* buf, size_t n) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  if (buf && n > 0) {
    std::strncpy(buf, h->plan_str.c_str(), n - 1);
    buf[n - 1] = '\0';
  }
  return (int)h->plan_str.size();
}

int64_t gemm_workspace_bytes(gemm_handle_t h) { return h ? (int64_t)h->ws_bytes : -1; }

int gemm_debug_set(gemm_handle_t h, int flags, uint64_t timeout_ns) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  h->debug_flags = flags;
  h->timeout_ns = timeout_ns ? timeout_ns : kDefaultTimeoutNs;
  return GEMM_OK;
}

int gemm_trace_set(gemm_handle_t h, uint64_t* dev_buf) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  h->trace = reinterpret_cast<unsigned long long*>(dev_buf);
  return GEMM_OK;
}

int gemm_timing_enable(gemm_handle_t h, int n) {
  if (!h || n < 0) return GEMM_ERR_INVALID_ARG;
  for (cudaEvent_t e : h->timing_ev) cudaEventDestroy(e);
  h->timing_ev.clear();
  h->timing_n = h->timing_used = 0;
  if (n == 0) return GEMM_OK;
  if (cudaSetDevice(h->device) != cudaSuccess) return GEMM_ERR_CUDA;
  h->timing_ev.resize(2 * static_cast<size_t>(n));
  for (auto& e : h->timing_ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      gemm_timing_enable(h, 0);
      return GEMM_ERR_CUDA;
    }
  }
  h->timing_n = n;
  return GEMM_OK;
}

int gemm_timing_read(gemm_handle_t h, float* ms, int n) {
  if (!h || (n > 0 && !ms)) return GEMM_ERR_INVALID_ARG;
  const int k = std::min(n, h->timing_used);
  for (int i = 0; i < k; ++i) {
    if (cudaEventSynchronize(h->timing_ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms[i], h->timing_ev[2 * i], h->timing_ev[2 * i + 1]) !=
            cudaSuccess)
      return GEMM_ERR_CUDA;
  }
  return k;
}

}  // extern "C"
