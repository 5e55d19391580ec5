// fa_fwd_common.cuh -- pieces of the forward shared by
// the d = 64 and d = 128 forward kernels.
//
// "FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness" (explainer page), "Method", steps 2-3: block row max,
// exponentials against the running max, row sums; masked entries are set
// to -inf before the max so that they contribute exactly zero.
#pragma once

#include "fa_kernels.cuh"

namespace fa {

// The running reference max of a row is only moved when the row max exceeds
// it by more than this (base-2 units), so P~ <= 2^8 and the O rescale is rare.
// Exact: O / l and lse use the same reference.
constexpr float kLazyRescale = 8.f;

// Dropout state of one query row: the hash key with the row pair folded in.
// (Which two bytes of each block word are the row's follows from the row's
// parity, which is the parity of its thread; the threshold p8 is passed from
// the kernel's parameters where it is used.)
struct RowDrop {
  uint32_t key;  // head key ^ ((i >> 1) << 16)
};

// Exponentials of 64 consecutive S columns sv[0..64) of a row: sv[c] <-
// 2^(sv[c]*sl2 - m), accumulated into the eight partial sums (before
// dropout) and packed to bf16 pairs in pk, with dropped elements packed as 0
// when kDrop (jp0 = key pair index of sv[0]).  Called by a converged warp
// whose lanes hold consecutive rows, even rows in even lanes.
template <bool kDrop>
__device__ __forceinline__ void exp64(float *sv, float sl2, float m, float (&rs8)[8],
                                      uint32_t (&pk)[32], const RowDrop &rd, uint32_t p8,
                                      uint32_t jp0) {
  // byte x >= p8 (1..255) iff x + (256 - p8) carries out of the byte
  const uint32_t qq = kDrop ? (256u - p8) * 0x01010101u : 0u;
  // a row's keep bytes in each block word: bytes 0-1 (even row), 2-3 (odd);
  // this row's, and its partner's in the adjacent lane (rows 2i and 2i + 1
  // are threads 2i' and 2i' + 1)
  const bool odd_row = (threadIdx.x & 1u) != 0u;
  const uint32_t sel = odd_row ? 0x7632u : 0x5410u;
  const uint32_t sel_partner = odd_row ? 0x5410u : 0x7632u;
#pragma unroll
  for (int c = 0; c < 64; c += 8) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; u += 2)
      fma2(x[u], x[u + 1], sv[c + u], sv[c + u + 1], sl2, sl2, -m, -m);
#pragma unroll
    for (int u = 0; u < 8; ++u) sv[c + u] = ex2_approx(x[u]);
    // (the dropout instantiation sums into four partials, not eight: its
    // hashing needs the registers)
#pragma unroll
    for (int u = 0; u < 8; u += 2) {
      const int r = kDrop ? (u & 2) : u;
      add2(rs8[r], rs8[r + 1], rs8[r], rs8[r + 1], sv[c + u], sv[c + u + 1]);
    }
    // the block words of key pairs (c >> 1) + 0..3 (keys c + u and c + u + 1
    // share one): rows 2i and 2i + 1 sit in adjacent lanes and draw on the
    // same words, so each lane of the pair hashes two of the four (the even
    // lane pairs 0-1, the odd lane 2-3), keeps its own row's bytes of them
    // and hands its partner the partner's with one shuffle
    uint32_t km[4] = {~0u, ~0u, ~0u, ~0u};  // per bf16 pair: 0xffff over each kept column
    if (kDrop) {
      const uint32_t odd = threadIdx.x & 1u;
      const uint32_t p = jp0 + static_cast<uint32_t>(c >> 1) + 2u * odd;
      const uint32_t w0 = pcg_hash(rd.key ^ p), w1 = pcg_hash(rd.key ^ (p + 1u));
      const uint32_t own = prmt(w0, w1, sel);
      const uint32_t got = __shfl_xor_sync(0xffffffffu, prmt(w0, w1, sel_partner), 1);
      // the keep bytes of columns c .. c + 3 and c + 4 .. c + 7, four per
      // word, compared with p8 at once: bit 7 of each byte is the carry
      const uint32_t x0 = odd ? got : own, x1 = odd ? own : got;
      const uint32_t s0 = (x0 & 0x7f7f7f7fu) + (qq & 0x7f7f7f7fu);
      const uint32_t s1 = (x1 & 0x7f7f7f7fu) + (qq & 0x7f7f7f7fu);
      const uint32_t k0 = (x0 & qq) | ((x0 | qq) & s0);
      const uint32_t k1 = (x1 & qq) | ((x1 | qq) & s1);
      // each column's carry replicated over its half of the bf16 pair
      km[0] = prmt(k0, 0u, 0x9988u);
      km[1] = prmt(k0, 0u, 0xbbaau);
      km[2] = prmt(k1, 0u, 0x9988u);
      km[3] = prmt(k1, 0u, 0xbbaau);
    }
#pragma unroll
    for (int u = 0; u < 8; u += 2)
      pk[(c + u) >> 1] = pack_bf16(sv[c + u], sv[c + u + 1]) & km[u >> 1];
  }
}

// exp64 on the 64-column half `half` of a 128-column row (jp0: the tile's
// first key pair).
template <bool kDrop>
__device__ __forceinline__ void exp_half(float (&sv)[kTile], int half, float sl2, float m,
                                         float (&rs8)[8], uint32_t (&pk)[32], const RowDrop &rd,
                                         uint32_t p8, uint32_t jp0) {
  exp64<kDrop>(sv + half * 64, sl2, m, rs8, pk, rd, p8, jp0 + static_cast<uint32_t>(half * 32));
}


// Masks of C consecutive S columns of a row on an edge tile: columns at or
// past lim_kv are padding, columns past lim_c lie in the future of the row
// (causal); both become -inf.  Limits count from the first of the C columns.
template <int C>
__device__ __forceinline__ void mask_cols(float (&sv)[C], int lim_kv, int lim_c) {
#pragma unroll
  for (int c = 0; c < C; ++c)
    if (c >= lim_kv || c > lim_c) sv[c] = -INFINITY;
}

__device__ __forceinline__ void mask_row(float (&sv)[kTile], int lim_kv, int lim_c) {
  mask_cols<kTile>(sv, lim_kv, lim_c);
}

// Max of C values (C a multiple of 16): eight independent chains of
// three-input maxima, then a tree.
template <int C>
__device__ __forceinline__ float max_cols(const float (&sv)[C]) {
  float mx8[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) mx8[u] = fmaxf(sv[u], sv[8 + u]);
#pragma unroll
  for (int c = 16; c < C; c += 16)
#pragma unroll
    for (int u = 0; u < 8; ++u) mx8[u] = fmax3(mx8[u], sv[c + u], sv[c + 8 + u]);
  return fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
}

__device__ __forceinline__ float row_max(const float (&sv)[kTile]) { return max_cols<kTile>(sv); }

// Block-sparse: writes the key tiles j < j_end whose mask byte in `row` is
// nonzero to tiles[], ascending, and returns their count (one warp; j_end <=
// kMaxMaskTiles).  Lane l takes the contiguous bytes [l * per, (l + 1) * per)
// and issues all its loads before using any, so the row costs one memory
// latency; a warp prefix sum of the per-lane counts places each lane's tiles.
__device__ __forceinline__ int compact_mask_row(const uint8_t *row, int j_end, int16_t *tiles,
                                                int lane) {
  const int per = (j_end + 31) >> 5;  // at most 32 bytes per lane
  const int j0 = lane * per;
  uint32_t bits = 0u;
  // 16 loads in flight at a time (one round up to 512 tiles, two beyond)
  for (int r = 0; r < per; r += 16) {
    uint32_t v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      v[e] = (r + e < per && j0 + r + e < j_end) ? static_cast<uint32_t>(__ldg(row + j0 + r + e))
                                                 : 0u;
#pragma unroll
    for (int e = 0; e < 16; ++e) bits |= (v[e] != 0u ? 1u : 0u) << (r + e);
  }
  const int cnt = __popc(bits);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int off = incl - cnt;
  while (bits) {
    const int e = __ffs(static_cast<int>(bits)) - 1;
    bits &= bits - 1u;
    tiles[off++] = static_cast<int16_t>(j0 + e);
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}


// Block-sparse from a CSR row: the entries col_idx[row_ptr[qt] ..
// row_ptr[qt + 1]) of query tile qt are marked in a bitmap (any order;
// duplicates merge), then the marked key tiles j < j_end are listed
// ascending in tiles[] and counted, as compact_mask_row does for the dense
// form.  A row range outside [0, nnz] or a tile index outside [0, nb) is
// skipped and recorded as kDevBadArg.  One warp; bits holds ceil(nb / 32)
// words of shared memory.
__device__ __forceinline__ int compact_csr_row(const int32_t *row_ptr, const int32_t *col_idx,
                                               int nnz, int qt, int nb, int j_end, uint32_t *bits,
                                               int16_t *tiles, int lane, const WaitCtl &w) {
  for (int i = lane; i < (nb + 31) / 32; i += 32) bits[i] = 0u;
  __syncwarp();
  int beg = __ldg(row_ptr + qt), end = __ldg(row_ptr + qt + 1);
  bool bad = false;
  if (beg < 0 || end < beg || end > nnz) {
    bad = true;
    beg = end = 0;
  }
  for (int e = beg + lane; e < end; e += 32) {
    const int c = __ldg(col_idx + e);
    if (c < 0 || c >= nb) bad = true;
    else if (c < j_end) atomicOr(&bits[c >> 5], 1u << (c & 31));
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(w, kDevBadArg);
  __syncwarp();
  int count = 0;
  for (int base = 0; base < j_end; base += 32) {
    const int j = base + lane;
    const bool keep = j < j_end && ((bits[base >> 5] >> lane) & 1u) != 0u;
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    if (keep) tiles[count + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(j);
    count += __popc(bal);
  }
  return count;
}

// Causal: one past the last key tile any row of query tile qt may see
// (keys j <= i + off), clamped to the n_kv tiles below the key bound.
__device__ __forceinline__ int causal_tile_end(int qt, int off, int n_kv) {
  const int last = qt * kTile + kTile - 1 + off;
  return last < 0 ? 0 : min(n_kv, last / kTile + 1);
}

// Split-KV merge ([MATH] §4: the softmax-weighted sum over the keys splits
// into independent ranges whose (max, sum, output) states combine by
// rescaling).  Each split s left O_s = (sum over its keys of P~ V) / l_s and
// lse_s = m_s + ln l_s; then lse = ln sum_s e^{lse_s} and
// O = sum_s e^{lse_s - lse} O_s.  8 threads per query row, D / 8 columns each.
template <int D>
__global__ void __launch_bounds__(256) fa_fwd_merge_kernel(const FwdArgs a) {
  pdl_wait();
  pdl_trigger();
  const int bh = blockIdx.y;
  const int row = blockIdx.x * 32 + static_cast<int>(threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;
  if (row >= a.pr.N) return;
  const int S = a.n_split, BH = a.pr.B * a.pr.H;
  const size_t stride = static_cast<size_t>(BH) * a.nq_pad;   // between splits
  const size_t base = static_cast<size_t>(bh) * a.nq_pad + row;
  float mx = -INFINITY;
  for (int sp = 0; sp < S; ++sp) mx = fmaxf(mx, a.part_lse[base + sp * stride]);
  constexpr int kC = D / 8;  // columns per thread
  float acc[kC];
#pragma unroll
  for (int c = 0; c < kC; ++c) acc[c] = 0.f;
  float den = 0.f;
  if (mx != -INFINITY) {
    for (int sp = 0; sp < S; ++sp) {
      const float ls = a.part_lse[base + sp * stride];
      if (ls == -INFINITY) continue;
      const float w = __expf(ls - mx);
      den += w;
      const float4 *src =
          reinterpret_cast<const float4 *>(a.part_o + (base + sp * stride) * D + sub * kC);
#pragma unroll
      for (int c4 = 0; c4 < kC / 4; ++c4) {
        const float4 x = src[c4];
        acc[4 * c4] = fmaf(w, x.x, acc[4 * c4]);
        acc[4 * c4 + 1] = fmaf(w, x.y, acc[4 * c4 + 1]);
        acc[4 * c4 + 2] = fmaf(w, x.z, acc[4 * c4 + 2]);
        acc[4 * c4 + 3] = fmaf(w, x.w, acc[4 * c4 + 3]);
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const size_t orow = static_cast<size_t>(bh) * a.pr.N + row;
#pragma unroll
  for (int c8 = 0; c8 < kC / 8; ++c8) {
    uint4 out;
    out.x = pack_bf16(acc[8 * c8] * inv, acc[8 * c8 + 1] * inv);
    out.y = pack_bf16(acc[8 * c8 + 2] * inv, acc[8 * c8 + 3] * inv);
    out.z = pack_bf16(acc[8 * c8 + 4] * inv, acc[8 * c8 + 5] * inv);
    out.w = pack_bf16(acc[8 * c8 + 6] * inv, acc[8 * c8 + 7] * inv);
    *reinterpret_cast<uint4 *>(a.o + orow * D + sub * kC + 8 * c8) = out;
  }
  if (sub == 0) a.lse[orow] = den > 0.f ? mx + __logf(den) : -INFINITY;
}

}  // namespace fa
