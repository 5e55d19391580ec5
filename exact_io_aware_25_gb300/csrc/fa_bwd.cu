// fa_bwd.cu -- backward kernels of exact tiled attention for sm_103a.
//
// The backward recomputes S and P tile by tile from Q, K, V and the stored
// per-row statistic instead of reading a stored N x N matrix ("FlashAttention:
// Fast and Memory-Efficient Exact Attention with IO-Awareness" explainer,
// "Key ideas", recomputation; "Mathematical Properties Behind FlashAttention",
// section 5, re-materialization).  The gradient formulas are the textbook
// ones for O = softmax(scale Q K^T) V:
//   dV = P^T dO, dP = dO V^T, D_i = <dO_i, O_i>, dS = P o (dP - D),
//   dQ = scale dS K, dK = scale dS^T Q.
//
// Three kernels on the caller's stream:
//   fa_bwd_pre_kernel   D_i, lse_i * log2(e) (+inf on padding / empty rows)
//                       into the workspace, and zeroes the fp32 dQ
//                       accumulators.  HBM-bound.
//   fa_bwd_main_kernel  persistent, one CTA per SM claiming work items (key
//                       tile j, b*h) from a counter in the workspace; per item
//                       K_j, V_j stay in shared memory while the allowed query
//                       tiles stream past:
//                         S^T = K_j Q_i^T, dP^T = V_j dO_i^T  (tcgen05, TMEM)
//                         P^T = 2^(S^T scale log2e - lse2_i), dS^T = P^T o (dP^T - D_i)
//                         dV += P^T dO_i, dK += dS^T Q_i      (TMEM accumulators)
//                         dQ_i partial = dS K_j -> TMA reduce-add (fp32) into
//                         the workspace accumulators
//   fa_bwd_dq_kernel    dQ = scale * accumulator -> bf16.
#include "fa_kernels.cuh"

namespace fa {
namespace {

constexpr int kStages = 3;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;  // 16 KiB bf16 tile
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- preprocess

// Preprocess.  The fp32 dQ accumulators are zeroed either by its first
// n_zero blocks (kZeroPerThread float4 per thread, 64 KiB per block), or, when
// n_zero is 0, row by row by the blocks below.  Nothing in the zeroing depends
// on the previous kernel on the stream, so the zeroing blocks store without
// waiting for it, on whatever SMs that kernel's tail leaves idle, and exit.
// (The accumulators' previous reader, the dQ conversion of an earlier call,
// lets its successors launch only after its reads.)  The other blocks wait,
// then take one (b, h) per n_pad / 128 blocks: 8 threads per row, each
// reading 8 bf16 of O and dO (16 bytes each).  Each thread takes
// kRowsPerThread rows, spaced one block-row apart, and issues all their loads
// before using any, so enough requests are in flight.  Rows past N (up to
// the 128-row padding) get D = 0 and lse2 = +inf.
constexpr int kRowsPerThread = 4;
constexpr int kRowsPerBlock = 256 / 8;  // rows one pass of a block covers
constexpr int kZeroPerThread = 16;
constexpr size_t kZeroPerBlock = 256 * kZeroPerThread;  // float4 per zeroing block
constexpr int kZeroAheadMaxN = 2048;

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdArgs a, unsigned n_zero,
                                                         size_t n4) {
  pdl_trigger();
  if (blockIdx.x < n_zero) {
    float4 *acc = reinterpret_cast<float4 *>(a.dq_acc);
    const size_t base = blockIdx.x * kZeroPerBlock + threadIdx.x;
#pragma unroll
    for (int u = 0; u < kZeroPerThread; ++u) {
      const size_t i = base + static_cast<size_t>(u) * 256;
      if (i < n4) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  pdl_wait();
  constexpr int kV = D / 64;  // 16-byte words of O (and of dO) per thread and row
  const Problem &pr = a.pr;
  const int blocks_per_head = a.n_pad / (kRowsPerBlock * kRowsPerThread);
  const int blk = static_cast<int>(blockIdx.x - n_zero);
  const int bh = blk / blocks_per_head, bx = blk - bh * blocks_per_head;
  const int sub = threadIdx.x & 7;
  const int r0 = bx * (kRowsPerBlock * kRowsPerThread) + (threadIdx.x >> 3);
  if (blk == 0 && threadIdx.x == 0) *a.sched = 0;
  if (pr.block_mask && blk == 0) {
    // the key tiles by descending number of query tiles (counting sort; ties
    // in any order): the main kernel hands out each head group's items
    // longest first, so that the ones left for the end are the shortest
    __shared__ int bins[kMaxMaskTiles + 1];
    const int nt = pr.nt;
    for (int c = threadIdx.x; c <= nt; c += blockDim.x) bins[c] = 0;
    __syncthreads();
    for (int kt = threadIdx.x; kt < nt; kt += blockDim.x) atomicAdd(&bins[a.col_cnt[kt]], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
      int pos = 0;
      for (int c = nt; c >= 0; --c) {
        const int k = bins[c];
        bins[c] = pos;
        pos += k;
      }
    }
    __syncthreads();
    for (int kt = threadIdx.x; kt < nt; kt += blockDim.x)
      a.kt_order[atomicAdd(&bins[a.col_cnt[kt]], 1)] = static_cast<int16_t>(kt);
  }
  const uint16_t *o_head = a.o + static_cast<size_t>(bh) * pr.N * D;
  const uint16_t *do_head = a.dout + static_cast<size_t>(bh) * pr.N * D;
  const size_t ws_row0 = static_cast<size_t>(bh) * a.n_pad;
  uint4 ov[kRowsPerThread][kV], dv[kRowsPerThread][kV];
#pragma unroll
  for (int u = 0; u < kRowsPerThread; ++u) {
    const int i = r0 + u * kRowsPerBlock;
#pragma unroll
    for (int w = 0; w < kV; ++w) {
      ov[u][w] = make_uint4(0u, 0u, 0u, 0u);
      dv[u][w] = make_uint4(0u, 0u, 0u, 0u);
      if (i < pr.N) {
        ov[u][w] = __ldg(reinterpret_cast<const uint4 *>(o_head + i * D + (sub * kV + w) * 8));
        dv[u][w] = __ldg(reinterpret_cast<const uint4 *>(do_head + i * D + (sub * kV + w) * 8));
      }
    }
  }
  // n_pad is a multiple of 128 and the grid covers it exactly: every row
  // below is in the padded range, and all 32 lanes reach the shuffles.
#pragma unroll
  for (int u = 0; u < kRowsPerThread; ++u) {
    const int i = r0 + u * kRowsPerBlock;
    float dsum = 0.f;
#pragma unroll
    for (int w = 0; w < kV; ++w) {
      const uint32_t ow[4] = {ov[u][w].x, ov[u][w].y, ov[u][w].z, ov[u][w].w};
      const uint32_t dw[4] = {dv[u][w].x, dv[u][w].y, dv[u][w].z, dv[u][w].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        dsum = fmaf(__uint_as_float(ow[t] << 16), __uint_as_float(dw[t] << 16), dsum);
        dsum = fmaf(__uint_as_float(ow[t] & 0xFFFF0000u), __uint_as_float(dw[t] & 0xFFFF0000u),
                    dsum);
      }
    }
    dsum += __shfl_xor_sync(0xffffffffu, dsum, 1);
    dsum += __shfl_xor_sync(0xffffffffu, dsum, 2);
    dsum += __shfl_xor_sync(0xffffffffu, dsum, 4);
    const size_t g = ws_row0 + i;
    if (n_zero == 0) {
      float4 *acc = reinterpret_cast<float4 *>(a.dq_acc + g * D + sub * (D / 8));
#pragma unroll
      for (int w = 0; w < D / 32; ++w) acc[w] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (sub == 0) {
      a.dsum[g] = -dsum;   // stored negated: the main kernels add it
      float l2 = INFINITY;  // padding rows and rows with no allowed key: P = 0
      if (i < pr.N) {
        const float lse = a.lse[static_cast<size_t>(bh) * pr.N + i];
        if (lse != -INFINITY) l2 = lse * kLog2e;
      }
      a.lse2[g] = l2;
    }
  }
}

// ---------------------------------------------------------------- dQ convert

// dQ = scale * accumulator -> bf16, one (b, h) per blockIdx.y; a thread
// converts 8 consecutive values of a row (chunk c: row c / 8, part c % 8) for
// kRowsPerThread chunks spaced one block apart.  Its successors may launch
// only once every block is past its reads of the accumulators (the next
// call's zeroing writes them without waiting).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdArgs a) {
  pdl_wait();
  const Problem &pr = a.pr;
  const int bh = blockIdx.y;
  const int chunks = pr.N * (D / 8);
  const int c0 = blockIdx.x * (256 * kRowsPerThread) + threadIdx.x;
  const float *acc_head = a.dq_acc + static_cast<size_t>(bh) * a.n_pad * D;
  uint16_t *dq_head = a.dq + static_cast<size_t>(bh) * pr.N * D;
  float4 x[kRowsPerThread], y[kRowsPerThread];
#pragma unroll
  for (int u = 0; u < kRowsPerThread; ++u) {
    const int c = c0 + u * 256;
    if (c < chunks) {
      // the accumulator rows are padded but contiguous within the head, so
      // chunk c sits at element 8 c
      const float4 *src = reinterpret_cast<const float4 *>(acc_head + static_cast<size_t>(c) * 8);
      x[u] = __ldcs(src);
      y[u] = __ldcs(src + 1);
    }
  }
  const float s = pr.scale;
#pragma unroll
  for (int u = 0; u < kRowsPerThread; ++u) {
    const int c = c0 + u * 256;
    if (c >= chunks) break;
    uint4 out;
    out.x = pack_bf16(x[u].x * s, x[u].y * s);
    out.y = pack_bf16(x[u].z * s, x[u].w * s);
    out.z = pack_bf16(y[u].x * s, y[u].y * s);
    out.w = pack_bf16(y[u].z * s, y[u].w * s);
    *reinterpret_cast<uint4 *>(dq_head + static_cast<size_t>(c) * 8) = out;
  }
  pdl_trigger();
}

// ---------------------------------------------------------------- block-sparse column lists

// For each key tile kt: the query tiles i >= i_begin with block_mask[i][kt]
// != 0, ascending, and their count.  Built once per call; the main kernel
// reads the list of the key tile it is working on.  A block takes
// kColsPerBlock adjacent key tiles, one warp each.  It first copies the
// mask's nt x kColsPerBlock byte slab for them into shared memory, all of its
// loads issued before any is stored (a warp instruction reads four rows of
// eight adjacent bytes), then each warp compacts its column 32 rows per
// ballot.  Few blocks, so the launch may overlap the previous kernel's tail
// without crowding it.
constexpr int kColsPerBlock = 8;
constexpr int kColsLoads = 16;  // slab bytes a thread loads per round

__global__ void __launch_bounds__(256) fa_bwd_cols_kernel(const BwdArgs a) {
  __shared__ uint8_t slab[kMaxMaskTiles * kColsPerBlock];
  pdl_wait();
  pdl_trigger();
  const Problem &pr = a.pr;
  const int nt = pr.nt, c0 = static_cast<int>(blockIdx.x) * kColsPerBlock;
  const int tid = threadIdx.x, c = tid & (kColsPerBlock - 1);
  constexpr int kRowsPerPass = 256 / kColsPerBlock;
  const bool col_ok = c0 + c < nt;
  const uint8_t *src = pr.block_mask + c0 + c;
  for (int r0 = tid / kColsPerBlock; r0 < nt; r0 += kRowsPerPass * kColsLoads) {
    uint8_t v[kColsLoads];
#pragma unroll
    for (int u = 0; u < kColsLoads; ++u) {
      const int r = r0 + u * kRowsPerPass;
      v[u] = col_ok && r < nt ? __ldg(src + static_cast<size_t>(r) * nt) : 0;
    }
#pragma unroll
    for (int u = 0; u < kColsLoads; ++u) {
      const int r = r0 + u * kRowsPerPass;
      if (r < nt) slab[r * kColsPerBlock + c] = v[u];
    }
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31, kt = c0 + warp;
  if (kt >= nt) return;
  const int i_begin = pr.causal ? kt : 0;
  int16_t *out = a.col_idx + static_cast<size_t>(kt) * nt;
  int cnt = 0;
  for (int base = i_begin & ~31; base < nt; base += 32) {
    const int i = base + lane;
    const bool keep = i >= i_begin && i < nt && slab[i * kColsPerBlock + warp] != 0;
    const uint32_t bal = __ballot_sync(0xffffffffu, keep);
    if (keep) out[cnt + __popc(bal & ((1u << lane) - 1u))] = static_cast<int16_t>(i);
    cnt += __popc(bal);
  }
  if (lane == 0) a.col_cnt[kt] = cnt;
}

// ---------------------------------------------------------------- main kernel

// Persistent: one CTA per SM walks the work items (key tile kt, head b*h).
// Its first item is t = blockIdx.x; later ones are claimed from a global
// counter by the producer warp and handed to the other roles through a small
// ring in shared memory, so CTAs that drew short items take more of them.
// Items are numbered by work_order: groups of heads whose Q, dO and fp32 dQ
// accumulators fit in L2 together, and within a group key tile by key tile
// (the longest causal items, small kt, first) with the group's heads
// fastest.  On long sequences a group is one or two heads, so the dQ
// reduce-adds and the Q / dO re-reads stay in L2; on short ones it is every
// head, which keeps one global longest-first order.
// K_j and V_j are double-buffered across items and every ring runs on one
// step counter for the whole CTA, so the next item's loads and first
// S^T / dP^T overlap the current item's last step and epilogue.
//
// Warp roles (16 warps, four warpgroups):
//   warpgroup 0 (warps 0-3)   P^T / dS^T for queries 0-63 of the step (thread = key row),
//                             then the dV half of the item's epilogue
//   warpgroup 1 (warps 4-7)   the same for queries 64-127, then the dK half
//   warpgroup 2 (warps 8-11)  dQ partial: TMEM -> swizzled shared tile -> TMA
//                             reduce-add into the fp32 accumulators (thread = query row)
//   warpgroup 3: warp 12      TMA producer
//                warp 13      TMEM owner and MMA issuer
//                warp 14      dK / dV stores (TMA) from the staging buffer
//                warp 15      idle
// Launched at 128 registers per thread; the elementwise warpgroups then take
// 160 (room for all 64 S^T and dP^T columns of a thread), the dQ warpgroup and
// the producer / MMA warpgroup 96 each: 160 + 160 + 96 + 96 = 4 x 128.
constexpr int kMainThreads = 512;
constexpr uint32_t kRegsElementwise = 160, kRegsDq = 96, kRegsControl = 96;

// One work item: key tile kt of head bh and the query tiles that attend to
// it (from causal_first_qtile under causal, the block mask's column kt, none
// at all when the tile lies past kv_len).
struct Item {
  int kt, bh, n, rot, i_begin;
  int kv_bound;
};

struct __align__(1024) BwdSmem {
  uint8_t kv[2][2][kTileBytes];          // [item parity][K_j | V_j]; later dK / dV staging
  uint8_t q[kStages][kTileBytes];
  uint8_t dout[kStages][kTileBytes];
  uint8_t dst[2][kTileBytes];            // dS^T bf16 [query half], rows = keys
  uint8_t dq_stage[kTileBytes];          // dQ partial fp32, 32 columns at a time, rows = queries
  float lse2[kStages][kTile];
  float dsum[kStages][kTile];
  uint64_t bar_kv[2];
  uint64_t bar_kv_free[2];
  uint64_t bar_q_full[kStages];
  uint64_t bar_q_empty[kStages];
  uint64_t bar_s_full;
  uint64_t bar_st_read;    // elementwise warps hold S^T / dP^T in registers
  uint64_t bar_p_full;     // P^T of the step is in TMEM
  uint64_t bar_ds_full;    // dS^T of the step is in shared memory
  uint64_t bar_pt_free;   // dropout only: dV has read P^T
  uint64_t bar_ds_free;
  uint64_t bar_dq_full;
  uint64_t bar_dq_free;
  uint64_t bar_done;
  uint64_t bar_final;
  uint64_t bar_epi_full[2];   // dK / dV of the item staged in kv[parity]
  int epi_item[2];            // its item id, -1 = no more items
  uint64_t bar_item_full[4];
  uint64_t bar_item_empty[4];
  int item_ring[4];
  Item item_info[4];   // the items, as the producer computed them (the others read them here)
  uint32_t tmem_base;
  int abort;
};

// Barriers between roles count warps, not threads: each warp arrives once,
// from lane 0 after a __syncwarp, so that 256 arrivals do not queue on one
// shared-memory word every step.
constexpr uint32_t kEwWarps = 8, kDqWarps = 4;
// Consumers of the item ring: the MMA warp, the elementwise warps and the dQ
// warps each release a slot once they have read it.
constexpr uint32_t kItemConsumers = 1 + kEwWarps + kDqWarps;

__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// TMEM columns: S^T, dP^T (fp32, lanes = keys), dV, dK (fp32 accumulators,
// lanes = keys), dQ partial (fp32, lanes = queries), P^T (bf16 pairs).
constexpr uint32_t kColST = 0, kColDPT = 128, kColDV = 256, kColDK = 320, kColDQ = 384,
                   kColPT = 448;
constexpr uint32_t kTmemCols = 512;


__device__ __forceinline__ Item item_at(const BwdArgs &a, int t) {
  const Problem &pr = a.pr;
  Item it;
  bwd_item(a, t, it.bh, it.kt);
  it.kv_bound = key_bound(pr, it.bh / pr.H);
  it.i_begin = pr.causal ? causal_first_qtile(pr, it.kt) : 0;
  if (it.kt * kTile >= it.kv_bound) it.n = 0;
  else if (pr.block_mask) it.n = __ldg(a.col_cnt + it.kt);
  else it.n = pr.nt > it.i_begin ? pr.nt - it.i_begin : 0;
  // the key tiles of one head start at different query tiles, so their
  // concurrent dQ reduce-adds land on different accumulator rows
  it.rot = it.n > 0 ? it.kt % it.n : 0;
  return it;
}

// Query tile of step k of the item.
__device__ __forceinline__ int qtile_of(const BwdArgs &a, const Item &it, int k) {
  int j = k + it.rot;
  if (j >= it.n) j -= it.n;
  return a.pr.block_mask ? static_cast<int>(__ldg(a.col_idx + static_cast<size_t>(it.kt) * a.pr.nt + j))
                         : it.i_begin + j;
}

// Elementwise phase 1 for 32 query columns starting at qc: S^T values in
// `v` are replaced, in place, by P^T = 2^(S^T * scale * log2(e) - lse2_q).
// kMask selects the edge-tile body (keys past kv_len, causal diagonal: kr is
// the key row less the tile pair's causal_delta); the common body carries no
// masking work at all.
template <bool kMask>
__device__ __forceinline__ void p_from_s32(uint32_t (&v)[32], int qc, int kr, bool key_ok,
                                           bool diag, float sl2, uint32_t lse2) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float4 l4 = ld_shared_f4(lse2 + (qc + 4 * g) * 4);
    float x[4];
    fma2(x[0], x[1], __uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]), sl2, sl2, -l4.x,
         -l4.y);
    fma2(x[2], x[3], __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]), sl2, sl2,
         -l4.z, -l4.w);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float p = ex2_approx(x[u]);
      if (kMask) {
        const bool masked = !key_ok || (diag && kr > qc + 4 * g + u);
        p = masked ? 0.f : p;
      }
      v[4 * g + u] = __float_as_uint(p);
    }
  }
}

// P^T of 32 columns as bf16 pairs into the TMEM P^T columns; with dropout,
// the dropped columns as 0 (the keep scale is applied to dV at the end).
template <bool kDrop>
__device__ __forceinline__ void store_p32(const uint32_t (&v)[32], int qc, uint32_t tmem_pt,
                                          uint32_t keep) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t pw[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int e = 16 * c + 2 * t;
      float x0 = __uint_as_float(v[e]), x1 = __uint_as_float(v[e + 1]);
      if (kDrop) {
        x0 = keep_bit(keep, e) ? x0 : 0.f;
        x1 = keep_bit(keep, e + 1) ? x1 : 0.f;
      }
      pw[t] = pack_bf16(x0, x1);
    }
    tmem_st8(tmem_pt + ((qc + 16 * c) >> 1), pw);
  }
}

// Elementwise phase 2: dS^T = P^T o (dP^T - D_q) for 32 columns, bf16 into
// row kr of this warpgroup's 128-byte-swizzled dS^T tile.  With dropout,
// dP^T is first multiplied by Z * keep_scale.
template <bool kDrop>
__device__ __forceinline__ void ds_store32(const uint32_t (&pv)[32], const uint32_t (&dv)[32],
                                           int qc, int half, int kr, uint32_t dsum,
                                           uint32_t ds_row, uint32_t keep, float keep_scale) {
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t dw[8];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int e0 = 16 * c + 4 * g;
      const float4 d4 = ld_shared_f4(dsum + (qc + e0) * 4);
      float dp[4], ds[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) dp[u] = __uint_as_float(dv[e0 + u]);
      if (kDrop) {
        // dP^T * Z * keep_scale - D in one packed multiply-add per pair
        float zs[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) zs[u] = keep_bit(keep, e0 + u) ? keep_scale : 0.f;
        fma2(dp[0], dp[1], dp[0], dp[1], zs[0], zs[1], d4.x, d4.y);
        fma2(dp[2], dp[3], dp[2], dp[3], zs[2], zs[3], d4.z, d4.w);
      } else {
        add2(dp[0], dp[1], dp[0], dp[1], d4.x, d4.y);   // (the stored D is negated)
        add2(dp[2], dp[3], dp[2], dp[3], d4.z, d4.w);
      }
      mul2(ds[0], ds[1], __uint_as_float(pv[e0]), __uint_as_float(pv[e0 + 1]), dp[0], dp[1]);
      mul2(ds[2], ds[3], __uint_as_float(pv[e0 + 2]), __uint_as_float(pv[e0 + 3]), dp[2], dp[3]);
      dw[2 * g] = pack_bf16(ds[0], ds[1]);
      dw[2 * g + 1] = pack_bf16(ds[2], ds[3]);
    }
    const uint32_t ch0 = static_cast<uint32_t>((qc + 16 * c - half * 64) >> 3);
    st_shared_v4(ds_row + ((ch0 ^ (kr & 7)) << 4), dw[0], dw[1], dw[2], dw[3]);
    st_shared_v4(ds_row + (((ch0 + 1) ^ (kr & 7)) << 4), dw[4], dw[5], dw[6], dw[7]);
  }
}

template <bool kDrop>
__global__ void __launch_bounds__(kMainThreads, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                       const __grid_constant__ CUtensorMap tm_dq_acc, const BwdArgs a) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  BwdSmem &s = *reinterpret_cast<BwdSmem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Problem &pr = a.pr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.nkt * pr.B * pr.H;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.bar_kv[i], 1);
      mbar_init(&s.bar_kv_free[i], 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.bar_q_full[i], 1);
      mbar_init(&s.bar_q_empty[i], 1);
    }
    mbar_init(&s.bar_s_full, 1);
    mbar_init(&s.bar_st_read, kEwWarps);
    mbar_init(&s.bar_p_full, kEwWarps);
    mbar_init(&s.bar_ds_full, kEwWarps);
    mbar_init(&s.bar_pt_free, 1);
    mbar_init(&s.bar_ds_free, 1);
    mbar_init(&s.bar_dq_full, 1);
    mbar_init(&s.bar_dq_free, kDqWarps);
    mbar_init(&s.bar_done, 1);
    mbar_init(&s.bar_final, 1);
    for (int i = 0; i < 2; ++i) mbar_init(&s.bar_epi_full[i], kEwWarps);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s.bar_item_full[i], 1);
      mbar_init(&s.bar_item_empty[i], kItemConsumers);
    }
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 13) tmem_alloc(&s.tmem_base, kTmemCols);
  if (warp == 12 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp < 8) {
    setmaxnreg_inc<kRegsElementwise>();
    // ------------------------------------------------------------ elementwise
    const int half = warp >> 2;            // query columns 64*half .. 64*half+63
    const int kr = (warp & 3) * 32 + lane; // TMEM lane: key row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = pr.scale_log2;
    // Per-item waits take one decision for all eight warps (a named-barrier
    // reduction), so the barriers of the per-item epilogue are reached by all
    // of them, on a timeout as well.  Inside an item each warp waits on its own
    // (a reduction per wait cost about 200 cycles); the outcome is reduced
    // once after the item's last step.
    auto wg_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return named_bar_and(1, 256, mbar_wait_warp(bar, parity, pr.wait, &s.abort));
    };
    // usually complete by the time a warp gets there, else within a few
    // hundred cycles: polled (waking from the hardware suspend measured slower)
    auto w_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return mbar_spin_warp(bar, parity, pr.wait, &s.abort);
    };
    bool ok = true;
    int g = 0;          // step counter of this CTA
    uint32_t done_par = 0;
    int last_v = 0;     // items handed to the store warp
    for (int v = 0; ok; ++v) {
      if (!wg_wait(&s.bar_item_full[v & 3], (v >> 2) & 1)) break;
      const int t = s.item_ring[v & 3];
      const Item itm = s.item_info[v & 3];
      warp_arrive(&s.bar_item_empty[v & 3]);
      if (t >= n_items) break;
      const bool key_ok = itm.kt * kTile + kr < itm.kv_bound;
      uint32_t drop_kk = 0u, drop_sh = 0u;
      if (kDrop) {
        const uint32_t key = static_cast<uint32_t>(itm.kt * kTile + kr);
        drop_kk = drop_head_key(pr, itm.bh) ^ (key >> 1);
        drop_sh = 8u * (key & 1u);
      }
      for (int k = 0; k < itm.n; ++k, ++g) {
        const int st = g % kStages;
        // the step's query tile: a global load under a block mask, so looked up
        // only where it is used (the causal diagonal, the dropout keep bits),
        // not on every step's path
        const int i = (pr.causal || kDrop) ? qtile_of(a, itm, k) : 0;
        // dropout keep bits of this step's 64 query columns, before S^T arrives
        uint32_t keep_a = 0u, keep_b = 0u;
        if (kDrop) {
          keep_a = keep_bits32(drop_kk, drop_sh, pr.drop_p8, i * kTile + half * 64);
          keep_b = keep_bits32(drop_kk, drop_sh, pr.drop_p8, i * kTile + half * 64 + 32);
          asm volatile("" : "+r"(keep_a), "+r"(keep_b));  // evaluated here, before S^T / dP^T
        }
        // causal: this warp's block (keys kr0..kr0+31, queries half*64..+63)
        // holds a masked element iff its largest kr - qc exceeds the pair's
        // delta.  Without dropout decided before the wait, off the path from
        // S^T to its loads (with dropout, whose keep bits already sit there,
        // that measured slower).
        int delta = 0, kr_rel = 0;
        bool diag = false, need_mask = false;
        auto decide_mask = [&] {
          delta = causal_delta(pr, i, itm.kt);
          diag = pr.causal && ((warp & 3) * 32 + 31 - half * 64 > delta);
          kr_rel = kr - delta;
          need_mask = diag || !__all_sync(0xffffffffu, key_ok);
        };
        if (!kDrop) decide_mask();
        if (!w_wait(&s.bar_s_full, g & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (kDrop) decide_mask();
        const uint32_t t_s = tmem + lane_base + kColST + half * 64;
        const uint32_t t_dp = tmem + lane_base + kColDPT + half * 64;
        uint32_t sa[32], da[32], sb[32], db[32];
        tmem_ld32(t_s, sa);
        tmem_ld32(t_dp, da);
        // the step's lse2 and D (the Q / dO stage; the S^T MMA already waited
        // for its Q), checked while the TMEM loads are in flight
        if (!w_wait(&s.bar_q_full[st], (g / kStages) & 1)) {
          tmem_wait_ld_tied32(sa, da);
          ok = false;
          break;
        }
        tmem_wait_ld_tied32(sa, da);
        tmem_ld32(t_s + 32, sb);   // second half in flight while the first is computed
        tmem_ld32(t_dp + 32, db);
        const uint32_t lse2_a = smem_u32(s.lse2[st]), dsum_a = smem_u32(s.dsum[st]);
        // phase 1: P^T, in place over the S^T registers
        if (need_mask) p_from_s32<true>(sa, half * 64, kr_rel, key_ok, diag, sl2, lse2_a);
        else p_from_s32<false>(sa, half * 64, kr, key_ok, diag, sl2, lse2_a);
        tmem_wait_ld_tied32(sb, db);
        tc_fence_before();
        warp_arrive(&s.bar_st_read);  // S^T / dP^T TMEM columns may be overwritten
        if (need_mask) p_from_s32<true>(sb, half * 64 + 32, kr_rel, key_ok, diag, sl2, lse2_a);
        else p_from_s32<false>(sb, half * 64 + 32, kr, key_ok, diag, sl2, lse2_a);
        // The previous step's MMAs are done with the P^T columns (dV) and the
        // dS^T tile (dK, dQ): without dropout one wait on the later of the two
        // commits, which the MMA thread issues after both (an mbarrier
        // operation costs about as much as the wait it saves); with dropout,
        // whose longer step leaves dQ later, a wait for dV alone here.
        if (g > 0 && !w_wait(kDrop ? &s.bar_pt_free : &s.bar_ds_free, (g - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_pt = tmem + lane_base + kColPT;
        store_p32<kDrop>(sa, half * 64, t_pt, keep_a);
        store_p32<kDrop>(sb, half * 64 + 32, t_pt, keep_b);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&s.bar_p_full);   // dV of this step may start
        // phase 2: dS^T (without dropout its tile was found free before the P^T store)
        if (kDrop && g > 0 && !w_wait(&s.bar_ds_free, (g - 1) & 1)) {
          ok = false;
          break;
        }
        const uint32_t ds_row = smem_u32(s.dst[half]) + kr * 128;
        ds_store32<kDrop>(sa, da, half * 64, half, kr, dsum_a, ds_row, keep_a, pr.keep_scale);
        ds_store32<kDrop>(sb, db, half * 64 + 32, half, kr, dsum_a, ds_row, keep_b, pr.keep_scale);
        fence_proxy_async_smem();
        warp_arrive(&s.bar_ds_full);  // dK, dQ of this step may start
      }
      // every warp gets here, from the last step or from a failed wait
      ok = named_bar_and(1, 256, ok);
      if (!ok) break;
      // -------------------------------------------------------- epilogue: dV (warpgroup 0), dK (1)
      if (itm.n > 0) {
        if (!wg_wait(&s.bar_done, done_par)) {
          ok = false;
          break;
        }
        done_par ^= 1u;
        tc_fence_after();
      }
      const uint32_t col = half == 0 ? kColDV : kColDK;
      const float mul = half == 0 ? (kDrop ? pr.keep_scale : 1.f) : pr.scale;
      const int kb = v & 1;
      // the store of the item two back has read this staging buffer (implied
      // by done for items with steps; waited here for the others too)
      if (v >= 2 && !w_wait(&s.bar_kv_free[kb], ((v - 2) >> 1) & 1)) {
        ok = false;
        break;
      }
      const uint32_t dst = smem_u32(s.kv[kb][half == 0 ? 1 : 0]) + kr * 128;
      uint32_t r0[32], r1[32];
      if (itm.n > 0) {
        tmem_ld32(tmem + lane_base + col, r0);
        tmem_ld32(tmem + lane_base + col + 32, r1);
        tmem_wait_ld_tied32(r0, r1);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) r0[c] = r1[c] = 0u;
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const uint32_t *r = h2 == 0 ? r0 : r1;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int c0 = ch * 8;
          st_shared_v4(dst + (((h2 * 4 + ch) ^ (kr & 7)) << 4),
                       pack_bf16(__uint_as_float(r[c0]) * mul, __uint_as_float(r[c0 + 1]) * mul),
                       pack_bf16(__uint_as_float(r[c0 + 2]) * mul, __uint_as_float(r[c0 + 3]) * mul),
                       pack_bf16(__uint_as_float(r[c0 + 4]) * mul, __uint_as_float(r[c0 + 5]) * mul),
                       pack_bf16(__uint_as_float(r[c0 + 6]) * mul, __uint_as_float(r[c0 + 7]) * mul));
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      // the store warp takes it from here
      if (tid == 0) s.epi_item[kb] = t;
      warp_arrive(&s.bar_epi_full[kb]);
      last_v = v + 1;
    }
    // tell the store warp there is nothing more (after it is done with the
    // staging buffer's previous use, whose item id shares the slot)
    if (ok) {
      const int kb = last_v & 1;
      if (last_v < 2 || w_wait(&s.bar_kv_free[kb], ((last_v - 2) >> 1) & 1)) {
        if (tid == 0) s.epi_item[kb] = -1;
        warp_arrive(&s.bar_epi_full[kb]);
      }
    }
  } else if (warp < 12) {
    setmaxnreg_dec<kRegsDq>();
    // ------------------------------------------------------------ dQ partials (rows = queries)
    const int qr = tid - 256;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    int g = 0;
    for (int v = 0; ok; ++v) {
      if (!named_bar_and(2, 128, mbar_wait_warp(&s.bar_item_full[v & 3], (v >> 2) & 1, pr.wait,
                                                &s.abort)))
        break;
      const int t = s.item_ring[v & 3];
      const Item itm = s.item_info[v & 3];
      warp_arrive(&s.bar_item_empty[v & 3]);
      if (t >= n_items) break;
      for (int k = 0; k < itm.n; ++k, ++g) {
        // the accumulator rows of this step (looked up before the wait)
        const int row0 = itm.bh * a.n_pad + qtile_of(a, itm, k) * kTile;
        // one decision for all four warps: the barriers below must see all of them
        if (!named_bar_and(2, 128, mbar_wait_warp(&s.bar_dq_full, g & 1, pr.wait, &s.abort))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lane_base + kColDQ, r0);
        tmem_ld32(tmem + lane_base + kColDQ + 32, r1);
        tmem_wait_ld_tied32(r0, r1);
        tc_fence_before();
        warp_arrive(&s.bar_dq_free);
        // Columns 0-31, then 32-63, go through the one staging tile: each time
        // the previous reduce-add must have finished reading it.
        const uint32_t stage = smem_u32(s.dq_stage);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          if (qr == 0) bulk_wait_read_all();
          named_bar_sync(2, 128);
          const uint32_t *r = h2 == 0 ? r0 : r1;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(stage + sw128_offset(qr, ch), r[4 * ch], r[4 * ch + 1], r[4 * ch + 2],
                         r[4 * ch + 3]);
          fence_proxy_async_smem();
          named_bar_sync(2, 128);
          if (qr == 0) {
            tma_reduce_add_2d(&tm_dq_acc, s.dq_stage, h2 * 32, row0);
            bulk_commit();
          }
        }
      }
    }
    if (qr == 0) bulk_wait_all();
  } else {
    setmaxnreg_dec<kRegsControl>();
    // The producer and MMA warps run converged, whole-warp: every wait is
    // one decision for the warp and an elected lane issues each operation.
    if (warp == 12) {
      // ---------------------------------------------------------- producer
      bool ok = true;
      int g = 0;
      for (int v = 0; ok; ++v) {
        // claim the next item and publish it to the other roles
        const int slot = v & 3;
        if (v >= 4 &&
            !mbar_wait_warp(&s.bar_item_empty[slot], ((v - 4) >> 2) & 1, pr.wait, &s.abort))
          break;
        int t = static_cast<int>(blockIdx.x);
        if (v > 0) {
          int c = 0;
          if (lane == 0) c = atomicAdd(a.sched, 1);
          t = static_cast<int>(gridDim.x) + __shfl_sync(0xffffffffu, c, 0);
        }
        const int kb = v & 1;
        // The item two back has stored its dK / dV out of this buffer.  Taken
        // for every item (those without steps stage zeros in the buffer too),
        // and before item v is published, so that no later phase of the
        // barrier (item v's own store) can complete before this wait looks.
        if (v >= 2 && !mbar_wait_warp(&s.bar_kv_free[kb], ((v - 2) >> 1) & 1, pr.wait, &s.abort))
          break;
        // the item's schedule, computed once here (its global lookups: the
        // longest-first order, the column count, kv_len) and handed over with it
        Item itm{};
        if (t < n_items) itm = item_at(a, t);
        if (lane == 0) {
          s.item_ring[slot] = t;
          s.item_info[slot] = itm;
          mbar_arrive(&s.bar_item_full[slot]);
        }
        __syncwarp();
        if (t >= n_items) {
          // no item left for this CTA: the dQ conversion may launch once
          // every CTA got here (released at the start instead, it measured
          // 0.2-0.4% slower steps on the long workloads)
          pdl_trigger();
          break;
        }
        if (itm.n == 0) continue;
        mbar_arrive_expect_tx_w(&s.bar_kv[kb], 2 * kTileBytes);
        tma_load_3d_w(s.kv[kb][0], &tm_k, &s.bar_kv[kb], 0, itm.kt * kTile, itm.bh);
        tma_load_3d_w(s.kv[kb][1], &tm_v, &s.bar_kv[kb], 0, itm.kt * kTile, itm.bh);
        for (int k = 0; k < itm.n; ++k, ++g) {
          const int st = g % kStages;
          const uint32_t use = g / kStages;
          const int i = qtile_of(a, itm, k);  // (a global load under a block mask: before the wait)
          if (use > 0 && !mbar_wait_warp(&s.bar_q_empty[st], (use - 1) & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          const size_t stat = static_cast<size_t>(itm.bh) * a.n_pad + static_cast<size_t>(i) * kTile;
          mbar_arrive_expect_tx_w(&s.bar_q_full[st], 2 * kTileBytes + 2 * kTile * 4);
          tma_load_3d_w(s.q[st], &tm_q, &s.bar_q_full[st], 0, i * kTile, itm.bh);
          tma_load_3d_w(s.dout[st], &tm_do, &s.bar_q_full[st], 0, i * kTile, itm.bh);
          bulk_load_w(s.lse2[st], a.lse2 + stat, kTile * 4, &s.bar_q_full[st]);
          bulk_load_w(s.dsum[st], a.dsum + stat, kTile * 4, &s.bar_q_full[st]);
        }
      }
    } else if (warp == 13) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);  // S^T, dP^T
      constexpr uint32_t id_acc = idesc_bf16(128, 64, false, true);  // dV, dK
      constexpr uint32_t id_dq = idesc_bf16(128, 64, true, true);    // dQ (A = dS, MN-major)
      // shared-memory descriptors of the fixed buffers (start address in 16-byte
      // units in the low bits: an offset of o bytes adds o / 16)
      const uint64_t d_dst_k = sdesc_sw128(smem_u32(s.dst[0]), 16, 1024);         // dS^T, K-major
      const uint64_t d_dst_mn = sdesc_sw128(smem_u32(s.dst[0]), kTileBytes, 1024);  // dS, MN-major
      bool ok = true;
      int g = 0;
      uint32_t kv_use[2] = {0u, 0u};
      for (int v = 0; ok; ++v) {
        if (!mbar_wait_warp(&s.bar_item_full[v & 3], (v >> 2) & 1, pr.wait, &s.abort)) break;
        const int t = s.item_ring[v & 3];
        const Item itm = s.item_info[v & 3];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.bar_item_empty[v & 3]);
        __syncwarp();
        if (t >= n_items) break;
        if (itm.n == 0) continue;
        const int kb = v & 1;
        const uint32_t k_addr = smem_u32(s.kv[kb][0]), v_addr = smem_u32(s.kv[kb][1]);
        const uint64_t d_k = sdesc_sw128(k_addr, 16, 1024), d_v = sdesc_sw128(v_addr, 16, 1024);
        const uint64_t d_k_mn = sdesc_sw128(k_addr, 1024, 1024);
        if (!mbar_wait_warp(&s.bar_kv[kb], kv_use[kb] & 1, pr.wait, &s.abort)) break;
        ++kv_use[kb];
        // S^T = K_j Q_i^T and dP^T = V_j dO_i^T for step gs.
        auto issue_s = [&](int gs) -> bool {
          const int st = gs % kStages;
          if (!mbar_wait_warp(&s.bar_q_full[st], (gs / kStages) & 1, pr.wait, &s.abort))
            return false;
          tc_fence_after();
          const uint64_t d_q = sdesc_sw128(smem_u32(s.q[st]), 16, 1024);
          const uint64_t d_do = sdesc_sw128(smem_u32(s.dout[st]), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            mma_bf16_ss_w(tmem + kColST, d_k + kk * 2, d_q + kk * 2, id_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            mma_bf16_ss_w(tmem + kColDPT, d_v + kk * 2, d_do + kk * 2, id_s, kk > 0);
          mma_commit_w(&s.bar_s_full);
          return true;
        };
        // the previous step's S^T / dP^T are in registers before they are overwritten
        if (g > 0 && !mbar_wait_warp(&s.bar_st_read, (g - 1) & 1, pr.wait, &s.abort)) break;
        tc_fence_after();
        if (!issue_s(g)) break;
        for (int k = 0; k < itm.n; ++k, ++g) {
          const int st = g % kStages;
          if (k + 1 < itm.n) {
            if (!mbar_wait_warp(&s.bar_st_read, g & 1, pr.wait, &s.abort) ||
                (tc_fence_after(), !issue_s(g + 1))) {
              ok = false;
              break;
            }
          }
          // P^T of this step is in TMEM.
          if (!mbar_wait_warp(&s.bar_p_full, g & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t d_q_mn = sdesc_sw128(smem_u32(s.q[st]), 1024, 1024);
          const uint64_t d_do_mn = sdesc_sw128(smem_u32(s.dout[st]), 1024, 1024);
          const uint32_t acc0 = k > 0 ? 1u : 0u;
          // dV += P^T dO_i: A = P^T from TMEM (16 queries = 8 columns per
          // instruction), B = dO_i (queries x d, d contiguous: MN-major).
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ts_w(tmem + kColDV, tmem + kColPT + kk * 8, d_do_mn + kk * 128, id_acc,
                          kk > 0 ? 1u : acc0);
          if (kDrop) mma_commit_w(&s.bar_pt_free);
          // dS^T of this step is in shared memory.
          if (!mbar_wait_warp(&s.bar_ds_full, g & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dK += dS^T Q_i: A = dS^T (K-major over queries, two 64-query
          // halves 16 KiB apart), B = Q_i (MN-major).
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss_w(tmem + kColDK, d_dst_k + (kk >> 2) * (kTileBytes >> 4) + (kk & 3) * 2,
                          d_q_mn + kk * 128, id_acc, kk > 0 ? 1u : acc0);
          mma_commit_w(&s.bar_q_empty[st]);
          if (g > 0 && !mbar_wait_warp(&s.bar_dq_free, (g - 1) & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dQ_i = dS K_j: A = dS read from the dS^T tile as an MN-major
          // operand (queries contiguous, two 64-query halves 16 KiB apart);
          // B = K_j, MN-major (d contiguous).  K dimension = keys.
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss_w(tmem + kColDQ, d_dst_mn + kk * 128, d_k_mn + kk * 128, id_dq, kk > 0);
          mma_commit_w(&s.bar_dq_full);
          mma_commit_w(&s.bar_ds_free);
        }
        // after the item's last dQ, not its last dK: dQ reads K_j from the
        // buffer the epilogue then overwrites with the dK / dV staging
        if (ok) mma_commit_w(&s.bar_done);
      }
      mma_commit_w(&s.bar_final);
      mbar_wait_drain(&s.bar_final, 0, pr.wait);
      __syncwarp();
    } else if (warp == 14) {
      // ---------------------------------------------------------- dK / dV store
      for (int u = 0;; ++u) {
        const int kb = u & 1;
        if (!mbar_wait_warp(&s.bar_epi_full[kb], (u >> 1) & 1, pr.wait, &s.abort)) break;
        const int t = s.epi_item[kb];
        if (t < 0) break;
        int bh, kt;
        bwd_item(a, t, bh, kt);
        if (lane == 0) {
          tma_store_3d(&tm_dv, s.kv[kb][1], 0, kt * kTile, bh);
          tma_store_3d(&tm_dk, s.kv[kb][0], 0, kt * kTile, bh);
          bulk_commit();
          bulk_wait_read_all();  // the staging buffer may be reloaded now
          mbar_arrive(&s.bar_kv_free[kb]);
        }
        __syncwarp();
      }
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t bwd_smem_bytes() { return sizeof(BwdSmem) + 1024; }

cudaError_t launch_bwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, const CUtensorMap &tdk, const CUtensorMap &tdv,
                       const CUtensorMap &tdq_acc, const BwdArgs &a, cudaStream_t st,
                       cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  static int configured_dev = -1;
  static int num_sms = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = bwd_smem_bytes();
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(fa_bwd_main_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_bwd_main_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  if (a.pr.block_mask &&
      (e = launch_pdl(fa_bwd_cols_kernel, dim3((a.pr.nt + kColsPerBlock - 1) / kColsPerBlock),
                      dim3(256), 0, st, a)) != cudaSuccess)
    return e;
  // preprocess: n_pad / (32 rows x 4) blocks per head, which cover the padded
  // rows exactly, after the zeroing blocks (every padded row of every head)
  // at d = 128 and, at d = 64, on sequences of up to kZeroAheadMaxN.  The
  // zeroing blocks run during the previous kernel's tail; on long sequences
  // behind the persistent d = 64 forward their stores evict the forward's K / V
  // from L2 while its last units still read them (0.3% slower steps at 64K;
  // behind the d = 128 forward, 0.9% faster at 4K)
  const size_t n4 = static_cast<size_t>(a.pr.B) * a.pr.H * a.n_pad * (a.pr.d / 4);
  const unsigned n_zero = a.pr.N <= kZeroAheadMaxN || a.pr.d == kHeadDimWide
                              ? static_cast<unsigned>((n4 + kZeroPerBlock - 1) / kZeroPerBlock)
                              : 0u;
  const dim3 pre_grid(n_zero + static_cast<unsigned>(a.n_pad / (kRowsPerBlock * kRowsPerThread)) *
                                   static_cast<unsigned>(a.pr.B * a.pr.H));
  if ((e = a.pr.d == kHeadDimWide
               ? launch_pdl(fa_bwd_pre_kernel<kHeadDimWide>, pre_grid, dim3(256), 0, st, a, n_zero,
                            n4)
               : launch_pdl(fa_bwd_pre_kernel<kHeadDim>, pre_grid, dim3(256), 0, st, a, n_zero,
                            n4)) != cudaSuccess)
    return e;
  if (a.pr.d == kHeadDimWide) {
    if ((e = launch_bwd_main_d128(tq, tk, tv, tdo, tdk, tdv, tdq_acc, a, st, ev_start, ev_stop)) !=
        cudaSuccess)
      return e;
    const int chunks = a.pr.N * (kHeadDimWide / 8);
    const dim3 dq_grid((chunks + 256 * kRowsPerThread - 1) / (256 * kRowsPerThread),
                       a.pr.B * a.pr.H);
    return launch_pdl(fa_bwd_dq_kernel<kHeadDimWide>, dq_grid, dim3(256), 0, st, a);
  }
  const int n_items = a.nkt * a.pr.B * a.pr.H;
  const dim3 grid(n_items < num_sms ? n_items : num_sms);
  if (ev_start && ev_stop && (e = cudaEventRecord(ev_start, st)) != cudaSuccess) return e;
  e = a.pr.drop_p8 > 0
          ? launch_pdl(fa_bwd_main_kernel<true>, grid, dim3(kMainThreads), smem, st, tq, tk, tv,
                       tdo, tdk, tdv, tdq_acc, a)
          : launch_pdl(fa_bwd_main_kernel<false>, grid, dim3(kMainThreads), smem, st, tq, tk, tv,
                       tdo, tdk, tdv, tdq_acc, a);
  if (e != cudaSuccess) return e;
  if (ev_start && ev_stop && (e = cudaEventRecord(ev_stop, st)) != cudaSuccess) return e;
  const int chunks = a.pr.N * (kHeadDim / 8);
  const dim3 dq_grid((chunks + 256 * kRowsPerThread - 1) / (256 * kRowsPerThread), a.pr.B * a.pr.H);
  return launch_pdl(fa_bwd_dq_kernel<kHeadDim>, dq_grid, dim3(256), 0, st, a);
}


namespace {

// CSR block mask -> dense nb x nb bytes; one CTA per query tile (row):
// the row is cleared, then every in-range entry sets its byte.  Duplicate
// entries write the same value.  Out-of-range rows or columns are skipped
// and recorded as kDevBadArg.
__global__ void __launch_bounds__(256) fa_csr_to_dense_kernel(const int32_t *row_ptr,
                                                               const int32_t *col_idx, int nnz,
                                                               int nb, uint8_t *dense, int *err) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  uint8_t *row = dense + static_cast<size_t>(r) * nb;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) row[j] = 0;
  __syncthreads();
  int beg = __ldg(row_ptr + r), end = __ldg(row_ptr + r + 1);
  bool bad = false;
  if (beg < 0 || end < beg || end > nnz) {
    bad = true;
    beg = end = 0;
  }
  for (int e = beg + static_cast<int>(threadIdx.x); e < end; e += blockDim.x) {
    const int c = __ldg(col_idx + e);
    if (c < 0 || c >= nb) bad = true;
    else row[c] = 1;
  }
  if (bad) atomicCAS(err, 0, kDevBadArg);
}

}  // namespace

cudaError_t launch_csr_to_dense(const int32_t *row_ptr, const int32_t *col_idx, int nnz, int nb,
                                uint8_t *dense, int *err, cudaStream_t st) {
  return launch_pdl(fa_csr_to_dense_kernel, dim3(nb), dim3(256), 0, st, row_ptr, col_idx, nnz, nb,
                    dense, err);
}

}  // namespace fa
