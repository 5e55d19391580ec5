// fa_kernels.cuh -- parameter blocks and launch entry points shared between
// the host launcher (fa_api.cu) and the kernels (fa_fwd.cu, fa_bwd.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_sm103.cuh"

namespace fa {

constexpr int kTile = 128;      // B_r = B_c = 128 query / key rows per tile
constexpr int kHeadDim = 64;    // d of the main kernels; the forward also has a d = 128 kernel
constexpr int kHeadDimWide = 128;
constexpr int kMaxMaskTiles = 1024;  // block-sparse: at most 1024 tiles per row (N <= 131072)
// Query tiles per head: the limit the host checks (at most 65535 tiles, 8M rows).
constexpr int kMaxGridTiles = 65535;

struct Problem {
  int B, H, N;            // N: query rows (and key rows, except in the split-KV forward)
  int Nk;                 // key rows
  int d;                  // head dimension (64 or 128)
  int nt;                 // ceil(N / 128) query tiles per head
  float scale;            // S = scale * Q K^T
  float scale_log2;       // scale * log2(e)
  int causal;
  int causal_off;         // causal keeps key j for query i iff j <= i + causal_off (Nk - Nq)
  const int32_t *kv_len;  // device [B] or nullptr
  const uint8_t *block_mask;  // device [nt * nt] or nullptr
  WaitCtl wait;
  // Dropout: element (i, j) of head bh is kept iff its hash byte >= drop_p8
  // (0 = no dropout); kept values are scaled by keep_scale = 256 / (256 - drop_p8).
  uint32_t drop_p8;
  uint32_t seed_lo, seed_hi;
  float keep_scale;
  // Work order (see work_order): heads are taken in groups of head_group
  // whose re-read rows fit in L2 together (1 <= head_group <= B * H).
  int head_group;
};

// The order in which the forward's CTAs and the backward's work items are
// handed out: heads in groups of p.head_group, and within a group by rank
// (query tile from the last, or key tile from the first: the longest first
// under causal) with the group's heads varying fastest.  Unit u in
// [0, B*H*per_head) maps to head bh and rank.  head_group = B*H gives one
// global longest-first order; smaller groups keep the rows that the
// resident CTAs re-read (K, V in the forward; Q, dO and the fp32 dQ
// accumulators in the backward) to a few heads, so that they stay in L2.
__device__ __forceinline__ void work_order(const Problem &p, int u, int per_head, int &bh,
                                           int &rank) {
  const int BH = p.B * p.H;
  const int span = p.head_group * per_head;
  const int gi = u / span;
  const int g0 = gi * p.head_group;
  const int gs = min(p.head_group, BH - g0);
  const int rem = u - gi * span;
  rank = rem / gs;
  bh = g0 + (rem - rank * gs);
}

// The 32-bit PCG hash (Jarzynski and Olano, "Hash Functions for GPU
// Rendering", JCGT 9(3), 2020): an LCG step followed by the RXS-M-XS output
// permutation of the PCG generator.
__device__ __forceinline__ uint32_t pcg_hash(uint32_t x) {
  const uint32_t st = x * 747796405u + 2891336453u;
  const uint32_t w = ((st >> ((st >> 28) + 4u)) ^ st) * 277803737u;
  return (w >> 22) ^ w;
}

// Dropout key of head bh; the keep byte of element (i, j) is byte
// 2 * (i & 1) + (j & 1) of pcg_hash(key ^ ((i >> 1) << 16 | (j >> 1))).
__device__ __forceinline__ uint32_t drop_head_key(const Problem &pr, int bh) {
  return pcg_hash(pcg_hash(pcg_hash(pr.seed_lo) ^ pr.seed_hi) ^ static_cast<uint32_t>(bh));
}

// Dropout keep bits of 32 query columns of one key row in the backward
// (thread = key row): column e is kept iff keep_bit(bits, e), i.e. Z(q0 + e,
// key) = 1.  kk = head key ^ (key >> 1); sh = 8 * (key & 1) selects the key's
// byte among each 2x2 block word (even queries: bytes 0-1, odd: 2-3); p8 is
// 1..255.  Called by a converged warp.
__device__ __forceinline__ uint32_t keep_bits32(uint32_t kk, uint32_t sh, uint32_t p8, int q0) {
  // keys 2m and 2m + 1 sit in adjacent lanes and draw on the same hash word
  // of each 2x2 block: each lane of the pair hashes half of the 16 query
  // pairs (the even lane pairs 0-7, the odd lane 8-15) and the two swap their
  // words with one shuffle (the warp is converged here)
  const uint32_t odd = threadIdx.x & 1u;
  // byte x >= p8 iff x + (256 - p8) carries out of the byte: the low seven
  // bits of each byte are added without crossing bytes, and the carry out of
  // bit 7 is the majority of the two top bits and the carry into it
  const uint32_t qq = (256u - p8) * 0x01010101u;
  // the four keep bytes of this key for query columns [2k, 2k + 16, 2k + 1,
  // 2k + 17], picked in one byte permute from {own word, partner's word}:
  // columns 2k, 2k + 1 are in the word of query pair k (the even lane's),
  // 16 + 2k, 17 + 2k in that of pair 8 + k (the odd lane's); the key's byte
  // in a word is sh / 8 (even query) and 2 + sh / 8 (odd query)
  const uint32_t b = sh >> 3, lo = odd ? 4u : 0u, hi = odd ? 0u : 4u;
  const uint32_t sel = (lo + b) | ((hi + b) << 4) | ((lo + 2u + b) << 8) | ((hi + 2u + b) << 12);
  uint32_t bits = 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t qp = static_cast<uint32_t>((q0 + 2 * k + 16 * static_cast<int>(odd)) >> 1);
    const uint32_t w = pcg_hash(kk ^ (qp << 16));
    const uint32_t o = __shfl_xor_sync(0xffffffffu, w, 1);
    const uint32_t x = prmt(w, o, sel);
    const uint32_t sum7 = (x & 0x7f7f7f7fu) + (qq & 0x7f7f7f7fu);
    const uint32_t carry = (x & qq) | ((x | qq) & sum7);
    // their carries (bit 7 of each byte) to bits k, 8 + k, 16 + k, 24 + k
    bits |= (carry & 0x80808080u) >> (7 - k);
  }
  return bits;
}

// Bit of keep_bits32's word that holds column e (0..31): columns 2k and
// 2k + 1 at bits k and 16 + k, columns 16 + 2k and 17 + 2k at 8 + k and 24 + k.
__device__ __forceinline__ constexpr int keep_pos(int e) {
  return ((e >> 4) << 3) + ((e & 1) << 4) + ((e & 15) >> 1);
}
__device__ __forceinline__ bool keep_bit(uint32_t bits, int e) {
  return (bits >> keep_pos(e)) & 1u;
}

struct FwdArgs {
  Problem pr;
  float *lse;             // [B, H, N]
  int starve;             // test hook: producer issues no K/V loads
  // Split-KV: n_split > 0 splits each row's key tiles into n_split contiguous
  // ranges (blockIdx.z); each CTA writes its normalised partial O and its lse
  // to the workspace instead of O and lse, and a merge kernel combines them.
  int n_split;
  int nq_pad;             // query rows per head in the partial arrays (N rounded up to 128)
  float *part_o;          // [n_split, B*H, nq_pad, d] fp32
  float *part_lse;        // [n_split, B*H, nq_pad] fp32, natural log
  uint16_t *o;            // [B, H, N, d] bf16: written by the d = 64 forward's softmax warps,
                          // or by the merge kernel in split-KV mode
  // Optional row statistics (plain forward): row max m_i of S and the
  // exponential sum l_i = sum_j exp(s_ij - m_i), fp32 [B, H, N].
  float *row_m;
  float *row_l;
  // Block-sparse mask given as CSR over query tiles (instead of
  // pr.block_mask): key tiles of query tile I are csr_idx[csr_ptr[I] ..
  // csr_ptr[I + 1]), in any order, duplicates allowed.
  const int32_t *csr_ptr;
  const int32_t *csr_idx;
  int csr_nnz;
};

struct BwdArgs {
  Problem pr;
  int n_pad;              // N rounded up to a multiple of 128
  int nkt;                // key tiles per head: ceil(Nk / 128) (work items per head)
  const uint16_t *o;      // [B, H, N, d] bf16
  const uint16_t *dout;   // [B, H, N, d] bf16
  const float *lse;       // [B, H, N]
  float *dsum;            // workspace -D  [B*H, n_pad] (D = rowsum(dO o O), negated)
  float *lse2;            // workspace lse * log2(e) [B*H, n_pad] (+inf in padding rows)
  float *dq_acc;          // workspace dQ accumulators [B*H, n_pad, d]
  int *col_cnt;           // workspace, block mask only: query tiles per key tile [nt]
  int16_t *col_idx;       // workspace, block mask only: their indices [nt][nt], ascending
  int16_t *kt_order;      // workspace, block mask only: key tiles by descending count [nt]
  int *sched;             // workspace: work counter of the persistent main kernel
  uint16_t *dq;           // [B, H, N, d] bf16
};

// Item t of a backward main kernel: head bh and key tile kt.  work_order
// gives the key tile's rank; under a block mask the rank indexes the key
// tiles sorted by their number of query tiles, largest first (written by the
// preprocess), so that the items handed out last are the shortest.
__device__ __forceinline__ void bwd_item(const BwdArgs &a, int t, int &bh, int &kt) {
  int rank;
  work_order(a.pr, t, a.nkt, bh, rank);
  kt = a.pr.block_mask ? static_cast<int>(__ldg(a.kt_order + rank)) : rank;
}

// First query tile with a query that sees a key of key tile kt under the
// causal rule (key j is kept for query i iff j <= i + causal_off): the tile
// of query kt * 128 - causal_off, or tile 0.
__device__ __forceinline__ int causal_first_qtile(const Problem &p, int kt) {
  const int q0 = kt * kTile - p.causal_off;
  return q0 <= 0 ? 0 : q0 / kTile;
}

// Causal offset of the tile pair (query tile i, key tile kt): the element of
// tile rows (key kr, query qc) is masked iff kr > qc + causal_delta.
__device__ __forceinline__ int causal_delta(const Problem &p, int i, int kt) {
  return (i - kt) * kTile + p.causal_off;
}

// Key bound of batch b: kv_len[b] clamped to [0, Nk].
__device__ __forceinline__ int key_bound(const Problem &p, int b) {
  if (!p.kv_len) return p.Nk;
  int L = __ldg(p.kv_len + b);
  return L < 0 ? 0 : (L > p.Nk ? p.Nk : L);
}

// Programmatic dependent launch: a kernel of this library may begin launching
// while the previous kernel on the stream drains.  Each kernel calls
// pdl_wait() before it reads anything (so results of the previous kernel
// are complete and visible) and pdl_trigger() to let its own successor
// start launching.  A successor starts only once every CTA of this kernel
// has triggered, so it never takes SMs that this kernel still needs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

size_t fwd_smem_bytes();
size_t bwd_smem_bytes();

// Unique identifier of the CUDA context current on the calling host thread
// (cuCtxGetId), 0 when there is none yet.  A device address looked up with
// cudaGetSymbolAddress is valid only in the context it was looked up in; the
// host code caches such addresses together with this identifier.
unsigned long long current_context_id();

// Expands a CSR block mask (row_ptr [nb + 1], col_idx [nnz]) into the dense
// nb x nb uint8 form (fa_bwd.cu); bad entries are skipped and recorded as
// kDevBadArg in *err.
cudaError_t launch_csr_to_dense(const int32_t *row_ptr, const int32_t *col_idx, int nnz, int nb,
                                uint8_t *dense, int *err, cudaStream_t st);

// (the d = 64 forward writes O from registers: no O tensor map)
cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdArgs &a, cudaStream_t st);
cudaError_t launch_fwd_splitkv(const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tv, const FwdArgs &a, cudaStream_t st);
// The same two entry points for d = 128 (fa_fwd_d128.cu); the tensor maps
// have 128 x 64 boxes, two per tile.
cudaError_t launch_fwd_d128(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &to, const FwdArgs &a, cudaStream_t st);
cudaError_t launch_fwd_splitkv_d128(const CUtensorMap &tq, const CUtensorMap &tk,
                                    const CUtensorMap &tv, const FwdArgs &a, cudaStream_t st);

// The d = 128 main backward kernel (fa_bwd_d128.cu), launched by launch_bwd
// between its preprocess and dQ-convert kernels.  Tensor maps: tq, tdo with
// 64-row x 64-column boxes; tk, tv, tdk, tdv with 128 x 64 boxes; tdq_acc
// {128, rows} fp32 with 64-row x 32-column boxes.
cudaError_t launch_bwd_main_d128(const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &tdo,
                                 const CUtensorMap &tdk, const CUtensorMap &tdv,
                                 const CUtensorMap &tdq_acc, const BwdArgs &a, cudaStream_t st,
                                 cudaEvent_t ev_start, cudaEvent_t ev_stop);

// ev_start / ev_stop (may be null) are recorded around the main kernel.
// tdq_acc: the fp32 dQ accumulators [B*H*n_pad, 64] as a 2-D map with 128 x 32
// boxes and 128-byte swizzle (target of the TMA reduce-adds).
cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &tdk, const CUtensorMap &tdv,
                       const CUtensorMap &tdq_acc, const BwdArgs &a, cudaStream_t st,
                       cudaEvent_t ev_start, cudaEvent_t ev_stop);

}  // namespace fa
