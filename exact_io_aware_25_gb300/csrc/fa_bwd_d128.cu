// fa_bwd_d128.cu -- main backward kernel for head dimension d = 128.
//
// Same recomputation scheme and gradient formulas as the d = 64 kernel
// ("FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness" explainer, "Key ideas", recomputation):
//   dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q,
// with S and P rebuilt per tile from Q, K and the stored lse.  The layout
// changes so that the two 128 x 128 fp32 accumulators dK and dV fit in TMEM
// next to the per-step matrices: a step covers 64 queries (not 128), and the
// dQ partial is produced transposed, dQ^T = K^T dS^T (M = d = 128, N = 64
// queries), so it needs 64 TMEM columns instead of 128.
//
// Persistent, one CTA per SM walking the work items (key tile kt, head b*h),
// numbered by work_order, from a global counter like the d = 64 kernel; K_j and V_j (32 KiB each)
// have a single buffer, which also stages dK / dV for the store.
//
// Warp roles (16 warps):
//   warpgroup 0 (warps 0-3)   P^T / dS^T for queries 0-31 of the step (thread = key row),
//                             then the dV half of the item's epilogue
//   warpgroup 1 (warps 4-7)   the same for queries 32-63, then the dK half
//   warpgroup 2 (warps 8-11)  dQ^T partial: thread = one d index; its 64
//                             query values -> the warp's fp32 staging tile
//                             (queries x 32 d) -> TMA reduce-add into the
//                             accumulators
//   warp 12 TMA producer, warp 13 TMEM owner and MMA issuer, warp 14 dK / dV
//   stores, warp 15 idle.
//
// TMEM columns (512): S^T 0-63, dP^T 64-127 (fp32, lanes = keys), P^T
// 128-159 (bf16 pairs), dQ^T 160-223 (fp32, lanes = d), dV 256-383, dK
// 384-511 (fp32, lanes = keys).
#include "fa_kernels.cuh"

namespace fa {
namespace {

constexpr int kQStep = 64;                          // queries per step
constexpr int kStages = 3;
constexpr uint32_t kKvHalf = kTile * 64 * 2;        // 128 rows x 64 bf16 = 16 KiB
constexpr uint32_t kKvBytes = 2 * kKvHalf;          // K_j or V_j: d 0-63, then d 64-127
constexpr uint32_t kQHalf = kQStep * 64 * 2;        // 64 rows x 64 bf16 = 8 KiB
constexpr uint32_t kQBytes = 2 * kQHalf;            // Q_i or dO_i of one step
constexpr uint32_t kDsBytes = kTile * kQStep * 2;   // dS^T: 128 keys x 64 queries bf16
constexpr uint32_t kDqWarpStage = kQStep * 32 * 4;  // 64 queries x 32 d fp32 = 8 KiB

constexpr int kMainThreads = 512;
constexpr uint32_t kRegsElementwise = 160, kRegsDq = 96, kRegsControl = 96;
constexpr uint32_t kEwWarps = 8, kDqWarps = 4;
constexpr uint32_t kItemConsumers = 1 + kEwWarps + kDqWarps;

// One work item: key tile kt of head bh and its query steps (two per query
// tile that attends to the key tile: from causal_first_qtile under causal,
// the block mask's column kt, none past kv_len).
struct Item {
  int kt, bh, n, rot, i_begin;
  int kv_bound;
};

struct __align__(1024) Bwd128Smem {
  uint8_t kv[2][kKvBytes];                // K_j | V_j; later dK | dV staging
  uint8_t q[kStages][kQBytes];
  uint8_t dout[kStages][kQBytes];
  uint8_t dst[kDsBytes];                  // dS^T, rows = keys, 64 queries (one swizzle span)
  uint8_t dq_stage[kDqWarps][kDqWarpStage];
  float lse2[kStages][kQStep];
  float dsum[kStages][kQStep];
  uint64_t bar_kv;
  uint64_t bar_kv_free;
  uint64_t bar_q_full[kStages];
  uint64_t bar_q_empty[kStages];
  uint64_t bar_s_full;
  uint64_t bar_st_read;
  uint64_t bar_p_full;
  uint64_t bar_ds_full;
  uint64_t bar_ds_free;
  uint64_t bar_dq_full;
  uint64_t bar_dq_free;
  uint64_t bar_done;
  uint64_t bar_final;
  uint64_t bar_epi_full;
  int epi_item;
  uint64_t bar_item_full[4];
  uint64_t bar_item_empty[4];
  int item_ring[4];
  Item item_info[4];   // the items, as the producer computed them (the others read them here)
  uint32_t tmem_base;
  int abort;
};

// one CTA per SM: the buffers plus the 1 KiB alignment slack within 227 KiB
static_assert(sizeof(Bwd128Smem) + 1024 <= 227 * 1024, "shared memory");

constexpr uint32_t kColST = 0, kColDPT = 64, kColPT = 128, kColDQT = 160, kColDV = 256,
                   kColDK = 384, kTmemCols = 512;

__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}


__device__ __forceinline__ Item item_at(const BwdArgs &a, int t) {
  const Problem &pr = a.pr;
  Item it;
  bwd_item(a, t, it.bh, it.kt);
  it.kv_bound = key_bound(pr, it.bh / pr.H);
  it.i_begin = pr.causal ? causal_first_qtile(pr, it.kt) : 0;
  int tiles;
  if (it.kt * kTile >= it.kv_bound) tiles = 0;
  else if (pr.block_mask) tiles = __ldg(a.col_cnt + it.kt);
  else tiles = pr.nt > it.i_begin ? pr.nt - it.i_begin : 0;
  it.n = 2 * tiles;
  // start the key tiles of one head at different query tiles, so that their
  // concurrent dQ reduce-adds land on different accumulator rows
  it.rot = tiles > 0 ? 2 * (it.kt % tiles) : 0;
  return it;
}

// Query step (64-row block index) of step k of the item.
__device__ __forceinline__ int qstep_of(const BwdArgs &a, const Item &it, int k) {
  int j = k + it.rot;
  if (j >= it.n) j -= it.n;
  const int tile = a.pr.block_mask
                       ? static_cast<int>(__ldg(a.col_idx + static_cast<size_t>(it.kt) * a.pr.nt +
                                                (j >> 1)))
                       : it.i_begin + (j >> 1);
  return 2 * tile + (j & 1);
}

// P^T = 2^(S^T * scale * log2(e) - lse2_q) for this thread's 32 query
// columns (qc: first column within the step, for lse2; qm: the same column
// within its 128-query tile, for the causal diagonal, against kr = the key
// row less the tile pair's causal_delta), in place.
template <bool kMask>
__device__ __forceinline__ void p_from_s32(uint32_t (&v)[32], int qc, int qm, int kr, bool key_ok,
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
        const bool masked = !key_ok || (diag && kr > qm + 4 * g + u);
        p = masked ? 0.f : p;
      }
      v[4 * g + u] = __float_as_uint(p);
    }
  }
}

// P^T of 32 columns (qc = first column within the step) as bf16 pairs into
// the P^T columns; dropped elements as 0.
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

// dS^T = P^T o (dP^T - D_q) for 32 columns (qc within the step), bf16 into
// row kr of the 128-byte-swizzled dS^T tile.  With dropout, dP^T is first
// multiplied by Z * keep_scale.
template <bool kDrop>
__device__ __forceinline__ void ds_store32(const uint32_t (&pv)[32], const uint32_t (&dv)[32],
                                           int qc, int kr, uint32_t dsum, uint32_t ds_row,
                                           uint32_t keep, float keep_scale) {
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
    const uint32_t ch0 = static_cast<uint32_t>((qc + 16 * c) >> 3);
    st_shared_v4(ds_row + ((ch0 ^ (kr & 7)) << 4), dw[0], dw[1], dw[2], dw[3]);
    st_shared_v4(ds_row + (((ch0 + 1) ^ (kr & 7)) << 4), dw[4], dw[5], dw[6], dw[7]);
  }
}

template <bool kDrop>
__global__ void __launch_bounds__(kMainThreads, 1)
    fa_bwd_d128_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk,
                       const __grid_constant__ CUtensorMap tm_dv,
                       const __grid_constant__ CUtensorMap tm_dq_acc, const BwdArgs a) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  Bwd128Smem &s = *reinterpret_cast<Bwd128Smem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Problem &pr = a.pr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = a.nkt * pr.B * pr.H;

  if (tid == 0) {
    mbar_init(&s.bar_kv, 1);
    mbar_init(&s.bar_kv_free, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.bar_q_full[i], 1);
      mbar_init(&s.bar_q_empty[i], 1);
    }
    mbar_init(&s.bar_s_full, 1);
    mbar_init(&s.bar_st_read, kEwWarps);
    mbar_init(&s.bar_p_full, kEwWarps);
    mbar_init(&s.bar_ds_full, kEwWarps);
    mbar_init(&s.bar_ds_free, 1);
    mbar_init(&s.bar_dq_full, 1);
    mbar_init(&s.bar_dq_free, kDqWarps);
    mbar_init(&s.bar_done, 1);
    mbar_init(&s.bar_final, 1);
    mbar_init(&s.bar_epi_full, kEwWarps);
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
    const int half = warp >> 2;             // query columns 32*half .. 32*half+31 of the step
    const int qc = half * 32;
    const int kr = (warp & 3) * 32 + lane;  // TMEM lane: key row
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = pr.scale_log2;
    auto wg_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return named_bar_and(1, 256, mbar_wait_warp(bar, parity, pr.wait, &s.abort));
    };
    auto w_wait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return mbar_wait_warp_fast(bar, parity, pr.wait, &s.abort);
    };
    bool ok = true;
    int g = 0;
    uint32_t done_par = 0;
    int last_v = 0;
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
        // the step's query block: a global load under a block mask, so looked
        // up only where it is used (the causal diagonal, the dropout keep bits)
        const int i64 = (pr.causal || kDrop) ? qstep_of(a, itm, k) : 0;
        uint32_t keep = 0u;
        if (kDrop) {
          keep = keep_bits32(drop_kk, drop_sh, pr.drop_p8, i64 * kQStep + qc);
          asm volatile("" : "+r"(keep));  // evaluated here, before the step's registers fill
        }
        // causal: query step i64 lies in query tile i64 / 2; this warp's block
        // (keys kr0..kr0+31, tile columns qm..qm+31) holds a masked element iff
        // its largest kr - qm exceeds the tile pair's delta.  Without dropout
        // decided before the wait, off the path from S^T to its loads.
        const int qm = (i64 & 1) * kQStep + qc;
        int delta = 0, kr_rel = 0;
        bool diag = false, need_mask = false;
        auto decide_mask = [&] {
          delta = causal_delta(pr, i64 >> 1, itm.kt);
          diag = pr.causal && ((warp & 3) * 32 + 31 - qm > delta);
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
        uint32_t sa[32], da[32];
        tmem_ld32(tmem + lane_base + kColST + qc, sa);
        tmem_ld32(tmem + lane_base + kColDPT + qc, da);
        // the step's lse2 and D (the Q / dO stage; the S^T MMA already waited
        // for its Q), checked while the TMEM loads are in flight
        if (!w_wait(&s.bar_q_full[st], (g / kStages) & 1)) {
          tmem_wait_ld_tied32(sa, da);
          ok = false;
          break;
        }
        tmem_wait_ld_tied32(sa, da);
        tc_fence_before();
        warp_arrive(&s.bar_st_read);  // S^T / dP^T TMEM columns may be overwritten
        const uint32_t lse2_a = smem_u32(s.lse2[st]), dsum_a = smem_u32(s.dsum[st]);
        if (need_mask) p_from_s32<true>(sa, qc, qm, kr_rel, key_ok, diag, sl2, lse2_a);
        else p_from_s32<false>(sa, qc, qm, kr, key_ok, diag, sl2, lse2_a);
        // The previous step's MMAs are done with the P^T columns (dV) and the
        // dS^T tile (dK, dQ^T): one wait on the later of the two commits, which
        // the MMA thread issues after both.
        if (g > 0 && !w_wait(&s.bar_ds_free, (g - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        store_p32<kDrop>(sa, qc, tmem + lane_base + kColPT, keep);
        tmem_wait_st();
        tc_fence_before();
        warp_arrive(&s.bar_p_full);   // dV of this step may start
        ds_store32<kDrop>(sa, da, qc, kr, dsum_a, smem_u32(s.dst) + kr * 128, keep,
                          pr.keep_scale);
        fence_proxy_async_smem();
        warp_arrive(&s.bar_ds_full);  // dK, dQ^T of this step may start
      }
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
      // the previous item's store has read the staging buffer (for items
      // with steps it is implied: the producer waited for it before loading
      // this item's K and V)
      if (v >= 1 && !w_wait(&s.bar_kv_free, (v - 1) & 1)) {
        ok = false;
        break;
      }
      const uint32_t col = half == 0 ? kColDV : kColDK;
      const float mul = half == 0 ? (kDrop ? pr.keep_scale : 1.f) : pr.scale;
      const uint32_t dst = smem_u32(s.kv[half == 0 ? 1 : 0]) + kr * 128;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {   // d 0-63, then d 64-127
        uint32_t r0[32], r1[32];
        if (itm.n > 0) {
          tmem_ld32(tmem + lane_base + col + h2 * 64, r0);
          tmem_ld32(tmem + lane_base + col + h2 * 64 + 32, r1);
          tmem_wait_ld_tied32(r0, r1);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) r0[c] = r1[c] = 0u;
        }
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          const uint32_t *r = q2 == 0 ? r0 : r1;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const int c0 = ch * 8;
            st_shared_v4(dst + h2 * kKvHalf + (((q2 * 4 + ch) ^ (kr & 7)) << 4),
                         pack_bf16(__uint_as_float(r[c0]) * mul, __uint_as_float(r[c0 + 1]) * mul),
                         pack_bf16(__uint_as_float(r[c0 + 2]) * mul, __uint_as_float(r[c0 + 3]) * mul),
                         pack_bf16(__uint_as_float(r[c0 + 4]) * mul, __uint_as_float(r[c0 + 5]) * mul),
                         pack_bf16(__uint_as_float(r[c0 + 6]) * mul, __uint_as_float(r[c0 + 7]) * mul));
          }
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      if (tid == 0) s.epi_item = t;
      warp_arrive(&s.bar_epi_full);
      last_v = v + 1;
    }
    // tell the store warp there is nothing more, once it has taken the last item
    if (ok && (last_v < 1 || w_wait(&s.bar_kv_free, (last_v - 1) & 1))) {
      if (tid == 0) s.epi_item = -1;
      warp_arrive(&s.bar_epi_full);
    }
  } else if (warp < 12) {
    setmaxnreg_dec<kRegsDq>();
    // ------------------------------------------------------------ dQ^T partials (thread = d index)
    const int dw = warp & 3;                      // d chunk 32*dw .. 32*dw+31
    const uint32_t lane_base = static_cast<uint32_t>(dw * 32) << 16;
    const uint32_t stage = smem_u32(s.dq_stage[dw]);
    bool ok = true;
    int g = 0;
    for (int v = 0; ok; ++v) {
      if (!mbar_wait_warp(&s.bar_item_full[v & 3], (v >> 2) & 1, pr.wait, &s.abort)) break;
      const int t = s.item_ring[v & 3];
      const Item itm = s.item_info[v & 3];
      warp_arrive(&s.bar_item_empty[v & 3]);
      if (t >= n_items) break;
      for (int k = 0; k < itm.n; ++k, ++g) {
        // the accumulator rows of this step (looked up before the wait)
        const int row0 = itm.bh * a.n_pad + qstep_of(a, itm, k) * kQStep;
        if (!mbar_wait_warp(&s.bar_dq_full, g & 1, pr.wait, &s.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r0[32], r1[32];
        tmem_ld32(tmem + lane_base + kColDQT, r0);
        tmem_ld32(tmem + lane_base + kColDQT + 32, r1);
        tmem_wait_ld_tied32(r0, r1);
        tc_fence_before();
        warp_arrive(&s.bar_dq_free);
        // this warp's previous reduce-add has finished reading its staging tile
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        // element (query q, d lane) of the 64 x 32 fp32 tile, 128-byte rows,
        // 16-byte chunks swizzled by q & 7: a warp writes one full row per q
#pragma unroll
        for (int q = 0; q < kQStep; ++q) {
          const uint32_t x = q < 32 ? r0[q] : r1[q - 32];
          const uint32_t addr = stage + q * 128 + ((((lane >> 2) ^ (q & 7)) << 4) | ((lane & 3) << 2));
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(x) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_2d(&tm_dq_acc, s.dq_stage[dw], dw * 32, row0);
          bulk_commit();
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    setmaxnreg_dec<kRegsControl>();
    if (warp == 12) {
      // ---------------------------------------------------------- producer
      bool ok = true;
      int g = 0;
      for (int v = 0; ok; ++v) {
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
        // The previous item's dK / dV have been stored out of the buffer.
        // Waited before item v is published, so that no later phase of the
        // barrier (item v's own store) can complete before this wait looks.
        if (v >= 1 && !mbar_wait_warp(&s.bar_kv_free, (v - 1) & 1, pr.wait, &s.abort)) break;
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
        mbar_arrive_expect_tx_w(&s.bar_kv, 2 * kKvBytes);
        tma_load_3d_w(s.kv[0], &tm_k, &s.bar_kv, 0, itm.kt * kTile, itm.bh);
        tma_load_3d_w(s.kv[0] + kKvHalf, &tm_k, &s.bar_kv, 64, itm.kt * kTile, itm.bh);
        tma_load_3d_w(s.kv[1], &tm_v, &s.bar_kv, 0, itm.kt * kTile, itm.bh);
        tma_load_3d_w(s.kv[1] + kKvHalf, &tm_v, &s.bar_kv, 64, itm.kt * kTile, itm.bh);
        for (int k = 0; k < itm.n; ++k, ++g) {
          const int st = g % kStages;
          const uint32_t use = g / kStages;
          const int i64 = qstep_of(a, itm, k);  // (a global load under a block mask: before the wait)
          if (use > 0 && !mbar_wait_warp(&s.bar_q_empty[st], (use - 1) & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          const size_t stat = static_cast<size_t>(itm.bh) * a.n_pad + static_cast<size_t>(i64) * kQStep;
          mbar_arrive_expect_tx_w(&s.bar_q_full[st], 2 * kQBytes + 2 * kQStep * 4);
          tma_load_3d_w(s.q[st], &tm_q, &s.bar_q_full[st], 0, i64 * kQStep, itm.bh);
          tma_load_3d_w(s.q[st] + kQHalf, &tm_q, &s.bar_q_full[st], 64, i64 * kQStep, itm.bh);
          tma_load_3d_w(s.dout[st], &tm_do, &s.bar_q_full[st], 0, i64 * kQStep, itm.bh);
          tma_load_3d_w(s.dout[st] + kQHalf, &tm_do, &s.bar_q_full[st], 64, i64 * kQStep, itm.bh);
          bulk_load_w(s.lse2[st], a.lse2 + stat, kQStep * 4, &s.bar_q_full[st]);
          bulk_load_w(s.dsum[st], a.dsum + stat, kQStep * 4, &s.bar_q_full[st]);
        }
      }
    } else if (warp == 13) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);   // S^T, dP^T (N = 64 queries)
      constexpr uint32_t id_acc = idesc_bf16(128, 128, false, true); // dV, dK (N = d)
      constexpr uint32_t id_dq = idesc_bf16(128, 64, true, true);    // dQ^T = K^T dS^T
      const uint32_t k_addr = smem_u32(s.kv[0]), v_addr = smem_u32(s.kv[1]);
      // K_j / V_j as K-major A operands (K = d, two 64-wide halves 16 KiB apart)
      const uint64_t d_k0 = sdesc_sw128(k_addr, 16, 1024), d_k1 = sdesc_sw128(k_addr + kKvHalf, 16, 1024);
      const uint64_t d_v0 = sdesc_sw128(v_addr, 16, 1024), d_v1 = sdesc_sw128(v_addr + kKvHalf, 16, 1024);
      // K_j^T as an MN-major A operand (M = d: the two halves are the two
      // 64-wide column blocks; K = keys, 8-key groups 1024 bytes apart)
      const uint64_t d_kt = sdesc_sw128(k_addr, kKvHalf, 1024);
      const uint64_t d_ds_k = sdesc_sw128(smem_u32(s.dst), 16, 1024);   // dS^T, K-major over queries
      const uint64_t d_ds_mn = sdesc_sw128(smem_u32(s.dst), 16, 1024);  // dS^T, MN-major (N = queries)
      bool ok = true;
      int g = 0;
      uint32_t kv_use = 0u;
      for (int v = 0; ok; ++v) {
        if (!mbar_wait_warp(&s.bar_item_full[v & 3], (v >> 2) & 1, pr.wait, &s.abort)) break;
        const int t = s.item_ring[v & 3];
        const Item itm = s.item_info[v & 3];
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.bar_item_empty[v & 3]);
        __syncwarp();
        if (t >= n_items) break;
        if (itm.n == 0) continue;
        if (!mbar_wait_warp(&s.bar_kv, kv_use & 1, pr.wait, &s.abort)) break;
        ++kv_use;
        // S^T = K_j Q_i^T and dP^T = V_j dO_i^T for step gs (N = 64 queries, K = d).
        auto issue_s = [&](int gs) -> bool {
          const int st = gs % kStages;
          if (!mbar_wait_warp(&s.bar_q_full[st], (gs / kStages) & 1, pr.wait, &s.abort))
            return false;
          tc_fence_after();
          const uint32_t qa = smem_u32(s.q[st]), oa = smem_u32(s.dout[st]);
          const uint64_t d_q0 = sdesc_sw128(qa, 16, 1024), d_q1 = sdesc_sw128(qa + kQHalf, 16, 1024);
          const uint64_t d_o0 = sdesc_sw128(oa, 16, 1024), d_o1 = sdesc_sw128(oa + kQHalf, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss_w(tmem + kColST, d_k0 + kk * 2, d_q0 + kk * 2, id_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss_w(tmem + kColST, d_k1 + kk * 2, d_q1 + kk * 2, id_s, 1u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss_w(tmem + kColDPT, d_v0 + kk * 2, d_o0 + kk * 2, id_s, kk > 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss_w(tmem + kColDPT, d_v1 + kk * 2, d_o1 + kk * 2, id_s, 1u);
          mma_commit_w(&s.bar_s_full);
          return true;
        };
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
          if (!mbar_wait_warp(&s.bar_p_full, g & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Q_i, dO_i as MN-major B operands (N = d: two 64-wide halves 8 KiB
          // apart; K = queries, 8-query groups 1024 bytes apart)
          const uint64_t d_q_mn = sdesc_sw128(smem_u32(s.q[st]), kQHalf, 1024);
          const uint64_t d_do_mn = sdesc_sw128(smem_u32(s.dout[st]), kQHalf, 1024);
          const uint32_t acc0 = k > 0 ? 1u : 0u;
          // dV += P^T dO_i: A = P^T from TMEM (16 queries = 8 columns per step)
#pragma unroll
          for (int kk = 0; kk < kQStep / 16; ++kk)
            mma_bf16_ts_w(tmem + kColDV, tmem + kColPT + kk * 8, d_do_mn + kk * 128, id_acc,
                          kk > 0 ? 1u : acc0);
          if (!mbar_wait_warp(&s.bar_ds_full, g & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dK += dS^T Q_i: A = dS^T (K-major over the 64 queries of one
          // swizzle span), B = Q_i (MN-major)
#pragma unroll
          for (int kk = 0; kk < kQStep / 16; ++kk)
            mma_bf16_ss_w(tmem + kColDK, d_ds_k + kk * 2, d_q_mn + kk * 128, id_acc,
                          kk > 0 ? 1u : acc0);
          mma_commit_w(&s.bar_q_empty[st]);
          if (g > 0 && !mbar_wait_warp(&s.bar_dq_free, (g - 1) & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // dQ^T = K_j^T dS^T: A = K_j^T (MN-major), B = dS^T (MN-major over
          // the queries); K dimension = keys, 16 per step = 2048 bytes
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_bf16_ss_w(tmem + kColDQT, d_kt + kk * 128, d_ds_mn + kk * 128, id_dq, kk > 0);
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
        if (!mbar_wait_warp(&s.bar_epi_full, u & 1, pr.wait, &s.abort)) break;
        const int t = s.epi_item;
        if (t < 0) break;
        int bh, kt;
        bwd_item(a, t, bh, kt);
        if (lane == 0) {
          tma_store_3d(&tm_dv, s.kv[1], 0, kt * kTile, bh);
          tma_store_3d(&tm_dv, s.kv[1] + kKvHalf, 64, kt * kTile, bh);
          tma_store_3d(&tm_dk, s.kv[0], 0, kt * kTile, bh);
          tma_store_3d(&tm_dk, s.kv[0] + kKvHalf, 64, kt * kTile, bh);
          bulk_commit();
          bulk_wait_read_all();  // the buffer may be reloaded now
          mbar_arrive(&s.bar_kv_free);
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

cudaError_t launch_bwd_main_d128(const CUtensorMap &tq, const CUtensorMap &tk,
                                 const CUtensorMap &tv, const CUtensorMap &tdo,
                                 const CUtensorMap &tdk, const CUtensorMap &tdv,
                                 const CUtensorMap &tdq_acc, const BwdArgs &a, cudaStream_t st,
                                 cudaEvent_t ev_start, cudaEvent_t ev_stop) {
  static int configured_dev = -1;
  static int num_sms = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(Bwd128Smem) + 1024;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(fa_bwd_d128_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_bwd_d128_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  const int n_items = a.nkt * a.pr.B * a.pr.H;
  const dim3 grid(n_items < num_sms ? n_items : num_sms);
  if (ev_start && ev_stop && (e = cudaEventRecord(ev_start, st)) != cudaSuccess) return e;
  e = a.pr.drop_p8 > 0
          ? launch_pdl(fa_bwd_d128_kernel<true>, grid, dim3(kMainThreads), smem, st, tq, tk, tv,
                       tdo, tdk, tdv, tdq_acc, a)
          : launch_pdl(fa_bwd_d128_kernel<false>, grid, dim3(kMainThreads), smem, st, tq, tk, tv,
                       tdo, tdk, tdv, tdq_acc, a);
  if (e != cudaSuccess) return e;
  if (ev_start && ev_stop && (e = cudaEventRecord(ev_stop, st)) != cudaSuccess) return e;
  return cudaSuccess;
}

}  // namespace fa
