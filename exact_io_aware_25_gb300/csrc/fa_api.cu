// fa_api.cu -- host side of libfa.so: argument validation, TMA tensor-map
// encoding, kernel launches on the caller's stream and the device error word.
// The C ABI is declared in include/fa.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_kernels.cuh"

namespace fa {

// Device error word written by kernels whose bounded waits ran out.
__device__ int g_dev_error;

// The two driver calls are resolved through the runtime's entry-point query,
// like cuTensorMapEncodeTiled, so that the library loads (for its host-side
// checks) on a machine without the driver.
unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext *);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c) return 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultTimeoutNs = 2000000000LL;

std::mutex g_mu;
long long g_timeout_ns = kDefaultTimeoutNs;
int g_starve_next = 0;
cudaEvent_t g_bwd_ev_start = nullptr, g_bwd_ev_stop = nullptr;
// Device address of the error word, per device, with the identifier of the
// context it was looked up in (the address is only valid in that context).
int *g_err_ptr[kMaxDevices] = {};
unsigned long long g_err_ctx[kMaxDevices] = {};
int g_dev_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Current device, checked to be sm_103; fills the error-word pointer.
fa_status device_setup(int *dev_out, int **err_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    g_dev_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_dev_ok[dev] != 1) return FA_ERR_UNSUPPORTED;
  // looked up again whenever the current context is not the one the cached
  // address came from (another context made current, or the device reset)
  const unsigned long long ctx = current_context_id();
  if (!g_err_ptr[dev] || ctx == 0 || ctx != g_err_ctx[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess || !p) return FA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int *>(p);
    g_err_ctx[dev] = current_context_id();  // the lookup creates the primary context if needed
  }
  *dev_out = dev;
  *err_out = g_err_ptr[dev];
  return FA_OK;
}

// [B*H, N, d] bf16 viewed as a 3-D tensor {d, N, B*H}; 128-row x 64-column
// boxes (one 128-byte swizzle span; a d = 128 tile is two boxes), 128-byte
// swizzle; rows past N read as zeros and are dropped on store.
bool encode_bhnd(CUtensorMap *m, const void *ptr, int BH, int N, int d = kHeadDim,
                 int box_rows = kTile) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 [rows, d] dQ accumulators as a 2-D tensor {d, rows}; boxes of 32
// columns (128 bytes) by 128 rows (d = 64) or 64 rows (d = 128, whose
// backward steps cover 64 queries), 128-byte swizzle.
bool encode_dq_acc(CUtensorMap *m, const void *ptr, size_t rows, int d) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(d == kHeadDimWide ? 64 : kTile)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status validate_common(int B, int H, int N, int d, float scale, const uint8_t *block_mask) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows >= (1LL << 31) || static_cast<long long>(B) * H >= 65536) return FA_ERR_INVALID_ARG;
  if (d != kHeadDim && d != kHeadDimWide) return FA_ERR_UNSUPPORTED;
  const int nt = (N + kTile - 1) / kTile;
  if (nt > kMaxGridTiles) return FA_ERR_UNSUPPORTED;
  if (block_mask && nt > kMaxMaskTiles) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Dropout threshold for drop probability p: p * 256 rounded to nearest (ties
// to even, the default rounding mode), at most 255; -1 for p outside [0, 1).
int drop_threshold(float p) {
  if (!std::isfinite(p) || p < 0.f || p >= 1.f) return -1;
  const long r = std::lrintf(p * 256.f);
  return r > 255 ? 255 : static_cast<int>(r);
}

// Largest N whose query / key pair indices (i >> 1, j >> 1) fit the 16-bit
// halves of the dropout hash counter.
constexpr int kMaxDropN = 131072;

Problem make_problem(int B, int H, int N, float scale, int causal, const int32_t *kv_len,
                     const uint8_t *block_mask, int *err, int p8 = 0,
                     unsigned long long seed = 0) {
  Problem p{};
  p.B = B;
  p.H = H;
  p.N = N;
  p.Nk = N;
  p.d = kHeadDim;
  p.nt = (N + kTile - 1) / kTile;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.kv_len = kv_len;
  p.block_mask = block_mask;
  std::lock_guard<std::mutex> lk(g_mu);
  p.wait.err = err;
  p.wait.timeout_ns = static_cast<uint64_t>(g_timeout_ns);
  p.drop_p8 = static_cast<uint32_t>(p8);
  p.seed_lo = static_cast<uint32_t>(seed & 0xffffffffull);
  p.seed_hi = static_cast<uint32_t>(seed >> 32);
  p.keep_scale = 256.f / static_cast<float>(256 - p8);
  p.head_group = B * H;
  return p;
}

// Heads per scheduling group (Problem::head_group): as many as fit their
// re-read rows, per_head_bytes each, into about half of the 129 MB L2.
int heads_per_group(int B, int H, size_t per_head_bytes) {
  constexpr size_t kL2Budget = size_t(64) << 20;
  const size_t bh = static_cast<size_t>(B) * H;
  size_t g = per_head_bytes > 0 ? kL2Budget / per_head_bytes : bh;
  if (g < 1) g = 1;
  if (g > bh) g = bh;
  return static_cast<int>(g);
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t dsum, lse2, dq_acc, col_cnt, col_idx, kt_order, sched, total;
};

// Workspace: D and base-2 lse [B*H, n_pad] fp32, dQ accumulators
// [B*H, n_pad, d] fp32, and the block-sparse column lists (key tile ->
// ascending query tiles): counts int32 [nt], indices int16 [nt, nt] and the
// key tiles by descending count int16 [nt]; one int32 work counter for the
// persistent main kernel.
WsLayout ws_layout(int B, int H, int N, int d) {
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t n_pad = align_up(static_cast<size_t>(N), kTile);
  const size_t nt = n_pad / kTile;
  WsLayout w{};
  w.dsum = 0;
  w.lse2 = align_up(w.dsum + bh * n_pad * sizeof(float), 256);
  w.dq_acc = align_up(w.lse2 + bh * n_pad * sizeof(float), 256);
  // column lists exist only with a block mask, which limits nt to kMaxMaskTiles
  const size_t nl = nt < static_cast<size_t>(kMaxMaskTiles) ? nt : kMaxMaskTiles;
  w.col_cnt = align_up(w.dq_acc + bh * n_pad * static_cast<size_t>(d) * sizeof(float), 256);
  w.col_idx = align_up(w.col_cnt + nl * sizeof(int), 256);
  w.kt_order = align_up(w.col_idx + nl * nl * sizeof(int16_t), 256);
  w.sched = align_up(w.kt_order + nl * sizeof(int16_t), 256);
  w.total = align_up(w.sched + sizeof(int), 256);
  return w;
}

// Split-KV forward: the number of key-range splits (0 = choose) and the
// scratch it needs.
int splitkv_splits(int B, int H, int Nq, int Nk, int num_splits) {
  const int nq_tiles = (Nq + kTile - 1) / kTile, nk_tiles = (Nk + kTile - 1) / kTile;
  int s = num_splits;
  if (s <= 0) {
    // about two CTAs per SM of a 152-SM GB300, at most one split per key tile
    const long long units = static_cast<long long>(B) * H * nq_tiles;
    s = static_cast<int>((2LL * 152 + units - 1) / units);
    if (s > 256) s = 256;
  }
  if (s > nk_tiles) s = nk_tiles;
  return s < 1 ? 1 : s;
}

struct SplitWs {
  size_t part_o, part_lse, total;
  int nq_pad;
};

SplitWs splitkv_ws(int B, int H, int Nq, int d, int S) {
  SplitWs w{};
  w.nq_pad = static_cast<int>(align_up(static_cast<size_t>(Nq), kTile));
  const size_t rows = static_cast<size_t>(S) * B * H * w.nq_pad;
  w.part_o = 0;
  w.part_lse = align_up(rows * static_cast<size_t>(d) * sizeof(float), 256);
  w.total = align_up(w.part_lse + rows * sizeof(float), 256);
  return w;
}

fa_status validate_splitkv(int B, int H, int Nq, int Nk, int d, float scale, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > 1024) return FA_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh >= 65536 || bh * Nq >= (1LL << 31) || bh * Nk >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  if (d != kHeadDim && d != kHeadDimWide) return FA_ERR_UNSUPPORTED;
  if ((Nq + kTile - 1) / kTile > kMaxGridTiles) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Optional parts of a forward call beyond fa_fwd_dropout's arguments.
struct FwdExtra {
  float *row_m = nullptr, *row_l = nullptr;             // row statistics
  const int32_t *csr_ptr = nullptr, *csr_idx = nullptr;  // CSR block mask
  int csr_nnz = 0;
  int Nk = 0;                                            // key rows (0: N)
};

fa_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int N, int d, float scale, int causal, const int32_t *kv_len,
                   const uint8_t *block_mask, float p, unsigned long long seed,
                   const FwdExtra &x, void *stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = validate_common(B, H, N, d, scale, block_mask);
  if (st != FA_OK) return st;
  if (x.csr_ptr && (N + kTile - 1) / kTile > kMaxMaskTiles) return FA_ERR_UNSUPPORTED;
  const int Nk = x.Nk > 0 ? x.Nk : N;
  if (static_cast<long long>(B) * H * Nk >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  const int p8 = drop_threshold(p);
  if (p8 < 0) return FA_ERR_INVALID_ARG;
  if (p8 > 0 && (N > kMaxDropN || Nk > kMaxDropN)) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  if ((x.row_m && !aligned16(x.row_m)) || (x.row_l && !aligned16(x.row_l)))
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int *err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv, to;
  if (!encode_bhnd(&tq, q, BH, N, d) || !encode_bhnd(&tk, k, BH, Nk, d) ||
      !encode_bhnd(&tv, v, BH, Nk, d) ||
      (d == kHeadDimWide && !encode_bhnd(&to, o, BH, N, d)))   // the d = 128 forward stores O by TMA
    return FA_ERR_CUDA;
  FwdArgs a{};
  a.pr = make_problem(B, H, N, scale, causal, kv_len, block_mask, err, p8, seed);
  a.pr.d = d;
  a.pr.Nk = Nk;
  a.pr.causal_off = Nk - N;
  // the rows every query tile re-reads: K and V of its head
  a.pr.head_group = heads_per_group(B, H, 4 * static_cast<size_t>(Nk) * d);
  a.lse = lse;
  a.o = static_cast<uint16_t *>(o);
  a.row_m = x.row_m;
  a.row_l = x.row_l;
  a.csr_ptr = x.csr_ptr;
  a.csr_idx = x.csr_idx;
  a.csr_nnz = x.csr_nnz;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    a.starve = g_starve_next;
    g_starve_next = 0;
  }
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d == kHeadDimWide ? launch_fwd_d128(tq, tk, tv, to, a, cs)
                                          : launch_fwd(tq, tk, tv, a, cs);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// CSR block mask arguments: row_ptr [nb + 1] always, col_idx [nnz] when nnz > 0.
fa_status validate_csr(const int32_t *row_ptr, const int32_t *col_idx, int nnz) {
  if (!row_ptr || nnz < 0 || (nnz > 0 && !col_idx)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int H, int N, int d, float scale, int causal,
                         const int32_t *kv_len, const uint8_t *block_mask, float p,
                         unsigned long long seed, void *stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, kv_len, block_mask, p, seed,
                  FwdExtra{}, stream);
}

fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                 int N, int d, float scale, int causal, const int32_t *kv_len,
                 const uint8_t *block_mask, void *stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, kv_len, block_mask, 0.f, 0ull,
                  FwdExtra{}, stream);
}

fa_status fa_fwd_stats(const void *q, const void *k, const void *v, void *o, float *lse,
                       float *row_max, float *row_sum, int B, int H, int N, int d, float scale,
                       int causal, const int32_t *kv_len, const uint8_t *block_mask,
                       void *stream) {
  if (!row_max || !row_sum) return FA_ERR_INVALID_ARG;
  FwdExtra x;
  x.row_m = row_max;
  x.row_l = row_sum;
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, kv_len, block_mask, 0.f, 0ull, x,
                  stream);
}

fa_status fa_fwd_csr(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                     int H, int N, int d, float scale, int causal, const int32_t *kv_len,
                     const int32_t *row_ptr, const int32_t *col_idx, int nnz, void *stream) {
  const fa_status st = validate_csr(row_ptr, col_idx, nnz);
  if (st != FA_OK) return st;
  FwdExtra x;
  x.csr_ptr = row_ptr;
  x.csr_idx = col_idx;
  x.csr_nnz = nnz;
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, kv_len, nullptr, 0.f, 0ull, x,
                  stream);
}

fa_status fa_fwd_qk(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int H, int Nq, int Nk, int d, float scale, int causal, const int32_t *kv_len,
                    void *stream) {
  if (Nk < 1) return FA_ERR_INVALID_ARG;
  FwdExtra x;
  x.Nk = Nk;
  return fwd_impl(q, k, v, o, lse, B, H, Nq, d, scale, causal, kv_len, nullptr, 0.f, 0ull, x,
                  stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (validate_common(B, H, N, d, 1.f, nullptr) != FA_OK) return 0;
  return ws_layout(B, H, N, d).total;
}

}  // extern "C"

namespace fa {
namespace {

// The backward of every entry point: N query rows, Nk key rows (Nk = N
// except in fa_bwd_qk, which passes no block mask and no dropout).
fa_status bwd_impl(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int Nk,
                   int d, float scale, int causal, const int32_t *kv_len,
                   const uint8_t *block_mask, float p, unsigned long long seed, void *workspace,
                   size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  fa_status st = validate_common(B, H, N, d, scale, block_mask);
  if (st != FA_OK) return st;
  if (Nk < 1 || static_cast<long long>(B) * H * Nk >= (1LL << 31)) return FA_ERR_INVALID_ARG;
  const int p8 = drop_threshold(p);
  if (p8 < 0) return FA_ERR_INVALID_ARG;
  if (p8 > 0 && N > kMaxDropN) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  const WsLayout wl = ws_layout(B, H, N, d);
  if (!workspace || !aligned16(workspace) || workspace_bytes < wl.total) return FA_ERR_WORKSPACE;
  int dev = 0;
  int *err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  const int BH = B * H;
  // the d = 128 backward steps over 64 query rows at a time
  const int qrows = d == kHeadDimWide ? 64 : kTile;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if (!encode_bhnd(&tq, q, BH, N, d, qrows) || !encode_bhnd(&tk, k, BH, Nk, d) ||
      !encode_bhnd(&tv, v, BH, Nk, d) || !encode_bhnd(&tdo, dout, BH, N, d, qrows) ||
      !encode_bhnd(&tdk, dk, BH, Nk, d) || !encode_bhnd(&tdv, dv, BH, Nk, d))
    return FA_ERR_CUDA;
  BwdArgs a{};
  a.pr = make_problem(B, H, N, scale, causal, kv_len, block_mask, err, p8, seed);
  a.pr.d = d;
  a.pr.Nk = Nk;
  a.pr.causal_off = Nk - N;
  // the rows every key tile re-reads: Q and dO (bf16) and the fp32 dQ
  // accumulators of its head
  a.pr.head_group = heads_per_group(B, H, 8 * static_cast<size_t>(N) * d);
  a.n_pad = static_cast<int>(align_up(static_cast<size_t>(N), kTile));
  a.nkt = (Nk + kTile - 1) / kTile;
  a.o = static_cast<const uint16_t *>(o);
  a.dout = static_cast<const uint16_t *>(dout);
  a.lse = lse;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.dsum = reinterpret_cast<float *>(ws + wl.dsum);
  a.lse2 = reinterpret_cast<float *>(ws + wl.lse2);
  a.dq_acc = reinterpret_cast<float *>(ws + wl.dq_acc);
  a.col_cnt = reinterpret_cast<int *>(ws + wl.col_cnt);
  a.col_idx = reinterpret_cast<int16_t *>(ws + wl.col_idx);
  a.kt_order = reinterpret_cast<int16_t *>(ws + wl.kt_order);
  a.sched = reinterpret_cast<int *>(ws + wl.sched);
  a.dq = static_cast<uint16_t *>(dq);
  CUtensorMap tdq_acc;
  if (!encode_dq_acc(&tdq_acc, a.dq_acc, static_cast<size_t>(BH) * a.n_pad, d)) return FA_ERR_CUDA;
  cudaEvent_t ev0, ev1;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ev0 = g_bwd_ev_start;
    ev1 = g_bwd_ev_stop;
  }
  return launch_bwd(tq, tk, tv, tdo, tdk, tdv, tdq_acc, a, static_cast<cudaStream_t>(stream), ev0,
                    ev1) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                         int H, int N, int d, float scale, int causal, const int32_t *kv_len,
                         const uint8_t *block_mask, float p, unsigned long long seed,
                         void *workspace, size_t workspace_bytes, void *stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, N, d, scale, causal, kv_len,
                  block_mask, p, seed, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_qk(const void *q, const void *k, const void *v, const void *o, const float *lse,
                    const void *dout, void *dq, void *dk, void *dv, int B, int H, int Nq, int Nk,
                    int d, float scale, int causal, const int32_t *kv_len, void *workspace,
                    size_t workspace_bytes, void *stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, kv_len,
                  nullptr, 0.f, 0ull, workspace, workspace_bytes, stream);
}

size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (validate_splitkv(B, H, Nq, Nk, d, 1.f, num_splits) != FA_OK) return 0;
  return splitkv_ws(B, H, Nq, d, splitkv_splits(B, H, Nq, Nk, num_splits)).total;
}

fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                         int H, int Nq, int Nk, int d, float scale, const int32_t *kv_len,
                         int num_splits, void *workspace, size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = validate_splitkv(B, H, Nq, Nk, d, scale, num_splits);
  if (st != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  const int S = splitkv_splits(B, H, Nq, Nk, num_splits);
  const SplitWs wl = splitkv_ws(B, H, Nq, d, S);
  if (!workspace || !aligned16(workspace) || workspace_bytes < wl.total) return FA_ERR_WORKSPACE;
  int dev = 0;
  int *err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  if (!encode_bhnd(&tq, q, BH, Nq, d) || !encode_bhnd(&tk, k, BH, Nk, d) ||
      !encode_bhnd(&tv, v, BH, Nk, d))
    return FA_ERR_CUDA;
  FwdArgs a{};
  a.pr = make_problem(B, H, Nq, scale, 0, kv_len, nullptr, err);
  a.pr.Nk = Nk;
  a.pr.d = d;
  a.lse = lse;
  a.n_split = S;
  a.nq_pad = wl.nq_pad;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.part_o = reinterpret_cast<float *>(ws + wl.part_o);
  a.part_lse = reinterpret_cast<float *>(ws + wl.part_lse);
  a.o = static_cast<uint16_t *>(o);
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t e = d == kHeadDimWide ? launch_fwd_splitkv_d128(tq, tk, tv, a, cs)
                                          : launch_fwd_splitkv(tq, tk, tv, a, cs);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                 float scale, int causal, const int32_t *kv_len, const uint8_t *block_mask,
                 void *workspace, size_t workspace_bytes, void *stream) {
  return fa_bwd_dropout(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, kv_len,
                        block_mask, 0.f, 0ull, workspace, workspace_bytes, stream);
}

size_t fa_bwd_csr_workspace_size(int B, int H, int N, int d) {
  if (validate_common(B, H, N, d, 1.f, nullptr) != FA_OK) return 0;
  const size_t nt = (static_cast<size_t>(N) + kTile - 1) / kTile;
  if (nt > static_cast<size_t>(kMaxMaskTiles)) return 0;
  return ws_layout(B, H, N, d).total + align_up(nt * nt, 256);
}

fa_status fa_bwd_csr(const void *q, const void *k, const void *v, const void *o,
                     const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                     int H, int N, int d, float scale, int causal, const int32_t *kv_len,
                     const int32_t *row_ptr, const int32_t *col_idx, int nnz, void *workspace,
                     size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  fa_status st = validate_csr(row_ptr, col_idx, nnz);
  if (st != FA_OK) return st;
  if ((st = validate_common(B, H, N, d, scale, nullptr)) != FA_OK) return st;
  const size_t need = fa_bwd_csr_workspace_size(B, H, N, d);
  if (need == 0) return FA_ERR_UNSUPPORTED;  // more than 1024 tiles per row
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int *err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  // the dense copy of the mask sits after the backward's own workspace
  const size_t own = ws_layout(B, H, N, d).total;
  uint8_t *dense = static_cast<uint8_t *>(workspace) + own;
  const int nb = (N + kTile - 1) / kTile;
  if (launch_csr_to_dense(row_ptr, col_idx, nnz, nb, dense, err,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return fa_bwd_dropout(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, kv_len,
                        dense, 0.f, 0ull, workspace, own, stream);
}

fa_status fa_check(void *stream) {
  int dev = 0;
  int *err = nullptr;
  fa_status st = device_setup(&dev, &err);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return FA_ERR_CUDA;
    return h == kDevTimeout ? FA_ERR_TIMEOUT : h == kDevBadArg ? FA_ERR_INVALID_ARG : FA_ERR_CUDA;
  }
  return FA_OK;
}

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer, bad size or bad scale";
    case FA_ERR_UNSUPPORTED:
      return "FA_ERR_UNSUPPORTED: head dim (64 or 128), size limit or device (sm_103)";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: tensor pointers must be 16-byte aligned";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel's bounded wait ran out";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    default: return "unknown fa_status";
  }
}

void fa_set_wait_timeout_ns(long long ns) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timeout_ns = ns > 0 ? ns : kDefaultTimeoutNs;
}

void fa_set_bwd_main_events(void *start_event, void *stop_event) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_bwd_ev_start = static_cast<cudaEvent_t>(start_event);
  g_bwd_ev_stop = static_cast<cudaEvent_t>(stop_event);
}

void fa_debug_starve_next_fwd(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_starve_next = enable ? 1 : 0;
}

}  // extern "C"
