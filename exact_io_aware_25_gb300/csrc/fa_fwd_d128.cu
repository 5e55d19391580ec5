// fa_fwd_d128.cu -- forward kernel of exact tiled attention for head
// dimension d = 128 on sm_103a.
//
// Same method as the d = 64 kernel ("FlashAttention: Fast and
// Memory-Efficient Exact Attention with IO-Awareness" (explainer page),
// "Method": S_ij on chip, running max and exponential sum, rescaled partial
// output, only O and lse written), with a layout for the wider head:
//
// One CTA per (query tile, b*h) and per SM (199 KiB of shared memory, all
// 512 TMEM columns); 10 warps:
//   warp 8   TMA producer: Q once, K_j (3-stage ring, two tiles ahead) and
//            V_j (2-stage ring).  Each 128 x 128 bf16 tile is two 128 x 64
//            boxes (the 128-byte swizzle spans 64 bf16), 16 KiB apart.
//   warp 9   TMEM owner and MMA issuer: S_j = Q K_j^T (M=128, N=128, K=128)
//            into S buffer j & 1, and O += P~_j V_j (M=128, N=128, K=128)
//            with P~_j from P~ buffer j & 1 in TMEM.  Per tile j it waits
//            for P~_j (which implies S_j has been read), issues PV_j and then
//            S_{j+2} into S_j's buffer, so the commit that announces S_{j+2}
//            also covers PV_j: when the softmax sees S_{j+2} ready, P~ buffer
//            j & 1 is free again.  S_{j+1} is computed while the softmax
//            works on S_j.  (Issuing S_{j+2} ahead of PV_j was measured
//            slower.)
//   warps 0-7 softmax: warps w and w + 4 own query rows 32 (w & 3) .. + 31
//            and split their 128 key columns (64 each; see below).  Per tile
//            one wait (S_j ready), one pair barrier and one arrival (P~_j
//            stored); the O rescale, when the lazily moved max requires one,
//            first waits for PV_{j-1}.
// TMEM columns: S buffers 0-127 and 128-255, P~ buffers 256-319 and
// 320-383 (bf16 pairs), O accumulator 384-511.
#include "fa_kernels.cuh"
#include "fa_fwd_common.cuh"

namespace fa {
namespace {

constexpr int kD = kHeadDimWide;
constexpr int kKStages = 3, kVStages = 2;
constexpr int kThreads = 320;
constexpr uint32_t kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr uint32_t kHalfBytes = kTile * 64 * 2;  // 128 rows x 64 bf16: one swizzle span
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // 32 KiB: d 0-63, then d 64-127

struct __align__(1024) Fwd128Smem {
  uint8_t q[kTileBytes];  // Q_i; reused to stage O for the TMA stores
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[kVStages][kTileBytes];
  uint64_t bar_q;
  uint64_t bar_k_full[kKStages];
  uint64_t bar_k_empty[kKStages];
  uint64_t bar_v_full[kVStages];
  uint64_t bar_v_empty[kVStages];
  uint64_t bar_s_full[2];
  uint64_t bar_p_full[2];
  uint64_t bar_o_done[2];
  uint64_t bar_final;
  uint32_t tmem_base;
  int abort;
  int n_tiles;
  int tile0;
  int16_t tiles[kMaxMaskTiles];
  uint32_t bits[kMaxMaskTiles / 32];  // CSR block mask: the row's tiles as a bitmap
  float xmax[2][2][kTile];            // [step parity][column half][row]: partial row maxima
  float xl[2][kTile];                 // [column half][row]: partial row sums, at the end
};

// one CTA per SM: the buffers plus the 1 KiB alignment slack within 227 KiB
static_assert(sizeof(Fwd128Smem) + 1024 <= 227 * 1024, "shared memory");

constexpr uint32_t kColS = 0, kColP = 256, kColO = 384, kTmemCols = 512;

__device__ __forceinline__ int tile_at(const Fwd128Smem &s, bool sparse, int it) {
  return sparse ? static_cast<int>(s.tiles[it]) : s.tile0 + it;
}

template <bool kDrop, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_d128_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o, const FwdArgs args) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  Fwd128Smem &s = *reinterpret_cast<Fwd128Smem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Problem &pr = args.pr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // launch order (work_order): groups of heads whose K and V fit in L2,
  // within a group the last (heaviest causal) query tiles first
  int bh, qrank;
  work_order(pr, static_cast<int>(blockIdx.x), pr.nt, bh, qrank);
  const int qt = pr.nt - 1 - qrank;
  const int b = bh / pr.H;
  const int kv_bound = key_bound(pr, b);
  const int n_kv = (kv_bound + kTile - 1) / kTile;
  int j_begin = 0, j_end = pr.causal ? causal_tile_end(qt, pr.causal_off, n_kv) : n_kv;
  if (kSplit) {
    const int per = (n_kv + args.n_split - 1) / args.n_split;
    j_begin = min(n_kv, static_cast<int>(blockIdx.y) * per);
    j_end = min(n_kv, j_begin + per);
  }
  const bool sparse = pr.block_mask != nullptr || args.csr_ptr != nullptr;

  // The producer warp initialises the barriers and, for a row without a
  // block mask, issues its first loads (Q, K_0, V_0) at once, so that their
  // memory latency overlaps the TMEM allocation and the CTA-wide setup.
  const bool early = !sparse && j_end > j_begin && !args.starve;
  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_init(&s.bar_q, 1);
      for (int i = 0; i < kKStages; ++i) {
        mbar_init(&s.bar_k_full[i], 1);
        mbar_init(&s.bar_k_empty[i], 1);
      }
      for (int i = 0; i < kVStages; ++i) {
        mbar_init(&s.bar_v_full[i], 1);
        mbar_init(&s.bar_v_empty[i], 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.bar_s_full[i], 1);
        mbar_init(&s.bar_p_full[i], kSoftmaxWarps);
        mbar_init(&s.bar_o_done[i], 1);
      }
      mbar_init(&s.bar_final, 1);
      s.abort = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_o);
    }
    __syncwarp();
    if (early) {
      const int row = j_begin * kTile;
      mbar_arrive_expect_tx_w(&s.bar_q, kTileBytes);
      tma_load_3d_w(s.q, &tm_q, &s.bar_q, 0, qt * kTile, bh);
      tma_load_3d_w(s.q + kHalfBytes, &tm_q, &s.bar_q, 64, qt * kTile, bh);
      mbar_arrive_expect_tx_w(&s.bar_k_full[0], kTileBytes);
      tma_load_3d_w(s.k[0], &tm_k, &s.bar_k_full[0], 0, row, bh);
      tma_load_3d_w(s.k[0] + kHalfBytes, &tm_k, &s.bar_k_full[0], 64, row, bh);
      mbar_arrive_expect_tx_w(&s.bar_v_full[0], kTileBytes);
      tma_load_3d_w(s.v[0], &tm_v, &s.bar_v_full[0], 0, row, bh);
      tma_load_3d_w(s.v[0] + kHalfBytes, &tm_v, &s.bar_v_full[0], 64, row, bh);
    }
  }
  if (warp == kMmaWarp) tmem_alloc(&s.tmem_base, kTmemCols);
  if (warp == 0) {
    const int count =
        !sparse ? j_end - j_begin
        : args.csr_ptr
            ? compact_csr_row(args.csr_ptr, args.csr_idx, args.csr_nnz, qt, pr.nt, j_end, s.bits,
                              s.tiles, lane, pr.wait)
            : compact_mask_row(pr.block_mask + static_cast<size_t>(qt) * pr.nt, j_end, s.tiles,
                               lane);
    if (lane == 0) {
      s.n_tiles = count;
      s.tile0 = j_begin;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int n = s.n_tiles;
  const uint32_t tmem = s.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (n > 0) {
      if (!early) {
        mbar_arrive_expect_tx_w(&s.bar_q, kTileBytes);
        tma_load_3d_w(s.q, &tm_q, &s.bar_q, 0, qt * kTile, bh);
        tma_load_3d_w(s.q + kHalfBytes, &tm_q, &s.bar_q, 64, qt * kTile, bh);
      }
      if (!args.starve) {
        auto load_k = [&](int it) -> bool {
          const int st = it % kKStages;
          const uint32_t use = it / kKStages;
          if (use > 0 && !mbar_wait_warp(&s.bar_k_empty[st], (use - 1) & 1, pr.wait, &s.abort))
            return false;
          const int row = tile_at(s, sparse, it) * kTile;
          mbar_arrive_expect_tx_w(&s.bar_k_full[st], kTileBytes);
          tma_load_3d_w(s.k[st], &tm_k, &s.bar_k_full[st], 0, row, bh);
          tma_load_3d_w(s.k[st] + kHalfBytes, &tm_k, &s.bar_k_full[st], 64, row, bh);
          return true;
        };
        bool ok = early || load_k(0);   // K_0 and V_0 went out with Q when early
        if (ok && n > 1) ok = load_k(1);
        for (int it = 0; ok && it < n; ++it) {
          if (it + 2 < n && !load_k(it + 2)) break;
          if (early && it == 0) continue;
          const int st = it % kVStages;
          const uint32_t use = it / kVStages;
          if (use > 0 && !mbar_wait_warp(&s.bar_v_empty[st], (use - 1) & 1, pr.wait, &s.abort))
            break;
          const int row = tile_at(s, sparse, it) * kTile;
          mbar_arrive_expect_tx_w(&s.bar_v_full[st], kTileBytes);
          tma_load_3d_w(s.v[st], &tm_v, &s.bar_v_full[st], 0, row, bh);
          tma_load_3d_w(s.v[st] + kHalfBytes, &tm_v, &s.bar_v_full[st], 64, row, bh);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (n > 0) {
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 128, false, true);
      const uint64_t d_q0 = sdesc_sw128(smem_u32(s.q), 16, 1024);
      const uint64_t d_q1 = sdesc_sw128(smem_u32(s.q + kHalfBytes), 16, 1024);
      bool ok = mbar_wait_warp(&s.bar_q, 0, pr.wait, &s.abort);
      // S_it = Q K_it^T into S buffer it & 1: K = 128 as two 64-wide halves.
      auto issue_s = [&](int it) -> bool {
        const int st = it % kKStages;
        if (!mbar_wait_warp(&s.bar_k_full[st], (it / kKStages) & 1, pr.wait, &s.abort))
          return false;
        tc_fence_after();
        const uint64_t d_k0 = sdesc_sw128(smem_u32(s.k[st]), 16, 1024);
        const uint64_t d_k1 = sdesc_sw128(smem_u32(s.k[st] + kHalfBytes), 16, 1024);
        const uint32_t dst = tmem + kColS + static_cast<uint32_t>(it & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss_w(dst, d_q0 + kk * 2, d_k0 + kk * 2, idesc_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_bf16_ss_w(dst, d_q1 + kk * 2, d_k1 + kk * 2, idesc_s, 1u);
        mma_commit_w(&s.bar_s_full[it & 1]);
        mma_commit_w(&s.bar_k_empty[st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int it = 0; ok && it < n; ++it) {
        const int bf = it & 1;
        const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
        // P~_it stored (so S_it has been read into registers as well)
        if (!mbar_wait_warp(&s.bar_p_full[bf], ph, pr.wait, &s.abort)) break;
        const int st = it % kVStages;
        if (!mbar_wait_warp(&s.bar_v_full[st], (it / kVStages) & 1, pr.wait, &s.abort)) break;
        tc_fence_after();
        // A = P~_it from TMEM (16 keys = 8 packed columns per step); B = V_j,
        // [keys][d] with d contiguous: MN-major, two 64-wide swizzle spans
        // along N (leading offset 16 KiB), 8-key groups 1024 bytes apart.
        const uint64_t d_v = sdesc_sw128(smem_u32(s.v[st]), kHalfBytes, 1024);
        const uint32_t pa = tmem + kColP + static_cast<uint32_t>(bf) * 64;
        const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_bf16_ts_w(tmem + kColO, pa + kk * 8, d_v + kk * 128, idesc_o, kk > 0 ? 1u : acc0);
        mma_commit_w(&s.bar_o_done[bf]);
        mma_commit_w(&s.bar_v_empty[st]);
        // S_{it+2} into S_it's buffer, behind PV_it: the commit that
        // announces it also covers PV_it, so P~ buffer bf is then free
        if (it + 2 < n && !issue_s(it + 2)) break;
      }
    }
    mma_commit_w(&s.bar_final);
    mbar_wait_drain(&s.bar_final, 0, pr.wait);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (half rows)
    // Warps w and w + 4 share TMEM lanes 32 (w & 3) .. + 31 (query rows) and
    // split each row's 128 key columns: warp w takes columns 0-63, warp w + 4
    // columns 64-127.  The pair combines its two partial row maxima through
    // shared memory at a 64-thread named barrier (id 2 + (w & 3)), which also
    // carries each warp's wait outcome so that both leave the loop together.
    // Each warp keeps the row sum of its own columns; the two are added in the
    // epilogue, where warp w writes O columns 0-63 and warp w + 4 columns 64-127.
    const int row = (warp & 3) * 32 + lane;
    const int ch = warp >> 2;                  // column half
    const uint32_t pair_bar = 2u + static_cast<uint32_t>(warp & 3);
    const int qrow = qt * kTile + row;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = pr.scale_log2;
    float m = -INFINITY;
    float l = 0.f;           // sum over this warp's columns
    float m_hi = -INFINITY;  // exact running row max (m may lag it by up to kLazyRescale)
    RowDrop rd{0u};
    if (kDrop) rd.key = drop_head_key(pr, bh) ^ (static_cast<uint32_t>(qrow >> 1) << 16);
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int bf = it & 1;
      const uint32_t ph = static_cast<uint32_t>(it >> 1) & 1u;
      const int j = tile_at(s, sparse, it);
      // S_it ready; PV_{it-2}, the last reader of P~ buffer bf, has completed
      const bool got = mbar_wait_warp_fast(&s.bar_s_full[bf], ph, pr.wait, &s.abort);
      float sv[64];
      const int key0 = j * kTile;
      const int kc0 = key0 + ch * 64;          // key of this warp's first column
      const bool edge =
          (key0 + kTile > kv_bound) || (pr.causal && key0 + kTile - 1 > qt * kTile + pr.causal_off);
      float mx_part = -INFINITY;
      if (got) {
        tc_fence_after();
        uint32_t raw[64];
        const uint32_t t0 = tmem + lane_base + kColS + static_cast<uint32_t>(bf) * 128 + ch * 64;
        tmem_ld32(t0, raw);
        tmem_ld32(t0 + 32, raw + 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = __uint_as_float(raw[c]);
        if (edge)
          mask_cols<64>(sv, kv_bound - kc0, pr.causal ? (qrow + pr.causal_off - kc0) : 64);
        mx_part = max_cols<64>(sv);
      }
      s.xmax[bf][ch][row] = mx_part;
      ok = named_bar_and(pair_bar, 64, ok && got);
      if (!ok) break;
      const float mxs = fmaxf(mx_part, s.xmax[bf][ch ^ 1][row]) * sl2;
      m_hi = fmaxf(m_hi, mxs);
      const float m_cand = fmaxf(m, mxs);
      const bool bump = (m == -INFINITY) || (m_cand > m + kLazyRescale);
      const float m_ref = bump ? m_cand : m;
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float alpha = bump ? ex2_approx(m - m_use) : 1.f;
      float rs8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) rs8[u] = 0.f;
      {
        uint32_t pk[32];
        const uint32_t jp0 = static_cast<uint32_t>(kc0 >> 1);
        exp64<kDrop>(sv, sl2, m_use, rs8, pk, rd, pr.drop_p8, jp0);
        tmem_st32(tmem + lane_base + kColP + static_cast<uint32_t>(bf) * 64 + ch * 32, pk);
      }
      const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
      // both warps of the pair hold the same alpha, so they take this branch together
      if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O must hold every PV up to it-1 before it is rescaled
        const int pb = (it - 1) & 1;
        if (mbar_wait_warp(&s.bar_o_done[pb], static_cast<uint32_t>((it - 1) >> 1) & 1u, pr.wait,
                           &s.abort)) {
          tc_fence_after();
          const uint32_t to = tmem + lane_base + kColO + ch * 64;
          uint32_t ov[32];
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            tmem_ld32(to + q2 * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(to + q2 * 32, ov);
          }
        } else {
          ok = false;  // reported to the partner at the next step's barrier
        }
      }
      tmem_wait_st();
      l = l * alpha + rs;
      m = m_ref;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.bar_p_full[bf]);
    }
    // ---------------------------------------------------------- epilogue
    // the pair adds its two partial row sums
    s.xl[ch][row] = l;
    ok = named_bar_and(pair_bar, 64, ok);
    l += s.xl[ch ^ 1][row];
    if (ok && n > 0) {
      // the last PV's commit also covers every earlier MMA of the issuer
      ok = mbar_wait_warp(&s.bar_o_done[(n - 1) & 1], static_cast<uint32_t>((n - 1) >> 1) & 1u,
                          pr.wait, &s.abort);
      tc_fence_after();
    }
    if (ok) {
      const float inv = (n > 0 && l > 0.f) ? (kDrop ? pr.keep_scale : 1.f) / l : 0.f;
      const float lse = (n > 0 && l > 0.f) ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      size_t prow = 0;
      if (kSplit)
        prow = (static_cast<size_t>(blockIdx.y) * (pr.B * pr.H) + bh) *
                   static_cast<size_t>(args.nq_pad) + qrow;
      float ov[64];
      if (n > 0) {
        uint32_t raw[64];
        const uint32_t to = tmem + lane_base + kColO + ch * 64;
        tmem_ld32(to, raw);
        tmem_ld32(to + 32, raw + 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 64; ++c) ov[c] = __uint_as_float(raw[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) ov[c] = 0.f;
      }
      if (kSplit) {
        if (qrow < pr.N) {
          float4 *dst = reinterpret_cast<float4 *>(args.part_o + prow * kD + ch * 64);
#pragma unroll
          for (int c4 = 0; c4 < 16; ++c4)
            dst[c4] = make_float4(ov[4 * c4] * inv, ov[4 * c4 + 1] * inv, ov[4 * c4 + 2] * inv,
                                  ov[4 * c4 + 3] * inv);
          if (ch == 0) args.part_lse[prow] = lse;
        }
      } else {
        const uint32_t q_base = smem_u32(s.q + ch * kHalfBytes) + row * 128;
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const float *x = ov + c8 * 8;
          st_shared_v4(q_base + ((c8 ^ (row & 7)) << 4), pack_bf16(x[0] * inv, x[1] * inv),
                       pack_bf16(x[2] * inv, x[3] * inv), pack_bf16(x[4] * inv, x[5] * inv),
                       pack_bf16(x[6] * inv, x[7] * inv));
        }
        fence_proxy_async_smem();
        if (ch == 0 && qrow < pr.N) {
          args.lse[static_cast<size_t>(bh) * pr.N + qrow] = lse;
          if (args.row_m) {
            // the pages' row statistics: m = max_j s_ij, l = sum_j exp(s_ij - m)
            const bool any = n > 0 && l > 0.f;
            const size_t r = static_cast<size_t>(bh) * pr.N + qrow;
            args.row_m[r] = any ? m_hi * 0.69314718055994531f : -INFINITY;
            args.row_l[r] = any ? l * ex2_approx(m - m_hi) : 0.f;
          }
        }
      }
    }
    named_bar_sync(1, 32 * kSoftmaxWarps);
    if (!kSplit && tid == 0 && ok && !s.abort) {
      tma_store_3d(&tm_o, s.q, 0, qt * kTile, bh);
      tma_store_3d(&tm_o, s.q + kHalfBytes, 64, qt * kTile, bh);
      bulk_commit();
      // the CTA may leave once the stores have read shared memory; the grid's
      // completion covers the global writes
      bulk_wait_read_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t fwd_d128_smem_bytes() { return sizeof(Fwd128Smem) + 1024; }

namespace {
cudaError_t launch_fwd_d128_config() {
  static int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    const int smem = static_cast<int>(fwd_d128_smem_bytes());
    e = cudaFuncSetAttribute(fa_fwd_d128_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_fwd_d128_kernel<true, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_fwd_d128_kernel<false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_fwd_d128(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const CUtensorMap &to, const FwdArgs &a, cudaStream_t st) {
  cudaError_t e = launch_fwd_d128_config();
  if (e != cudaSuccess) return e;
  const size_t smem = fwd_d128_smem_bytes();
  const dim3 grid(a.pr.nt * a.pr.B * a.pr.H);
  if (a.pr.drop_p8 > 0)
    return launch_pdl(fa_fwd_d128_kernel<true, false>, grid, dim3(kThreads), smem, st, tq, tk, tv,
                      to, a);
  return launch_pdl(fa_fwd_d128_kernel<false, false>, grid, dim3(kThreads), smem, st, tq, tk, tv,
                    to, a);
}

cudaError_t launch_fwd_splitkv_d128(const CUtensorMap &tq, const CUtensorMap &tk,
                                    const CUtensorMap &tv, const FwdArgs &a, cudaStream_t st) {
  cudaError_t e = launch_fwd_d128_config();
  if (e != cudaSuccess) return e;
  const dim3 grid(a.pr.nt * a.pr.B * a.pr.H, a.n_split);
  e = launch_pdl(fa_fwd_d128_kernel<false, true>, grid, dim3(kThreads), fwd_d128_smem_bytes(), st,
                 tq, tk, tv, tq, a);
  if (e != cudaSuccess) return e;
  const dim3 mgrid((a.pr.N + 31) / 32, a.pr.B * a.pr.H);
  return launch_pdl(fa_fwd_merge_kernel<kD>, mgrid, dim3(256), 0, st, a);
}

}  // namespace fa
