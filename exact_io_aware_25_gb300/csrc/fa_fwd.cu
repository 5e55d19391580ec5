// fa_fwd.cu -- forward kernel of exact tiled attention for sm_103a.
//
// Follows "FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness" (explainer page), "Method": for query tile i and each allowed
// key/value tile j,
//   1. S_ij = Q_i K_j^T on chip (here scaled: S = scale * Q K^T),
//   2. block row max / exponentials / row sums,
//   3. running max m and exponential sum l updated with the merge rule of
//      "online softmax tracking",
//   4. the partial output rescaled and P~_ij V_j accumulated,
// then only O and the per-row statistic (lse = m + ln l) are written.
//
// GB300 mapping (one CTA per (query tile, b*h); 6 warps; two CTAs share an SM:
// 256 TMEM columns and 100 KiB of shared memory each):
//   warp 4   TMA producer: Q once, then K_j (3-stage ring, one tile ahead) and
//            V_j (2-stage ring).
//   warp 5   TMEM owner and MMA issuer: S = Q K_j^T (M=128, N=128, K=64)
//            into TMEM, and O += P~ V_j (M=128, N=64, K=128) with P~ read
//            straight from TMEM (A operand in tensor memory).  S_{j+1} is
//            issued as soon as the softmax has pulled S_j into registers, so
//            the tensor core overlaps the exponentials.
//   warps 0-3 softmax: thread t owns query row t.  Reads its S row from TMEM,
//            applies the masks, keeps (m, l) in base-2 units, writes
//            P~ = 2^(S*scale*log2e - m) as packed bf16 pairs back into TMEM,
//            rescales its O row in TMEM when m grew, and runs the epilogue
//            (O / l -> bf16 -> its row of O in global memory, lse).
// Division by l is deferred to the epilogue; the result equals the pages'
// per-step normalised update because both use the same running max.
#include "fa_kernels.cuh"
#include "fa_fwd_common.cuh"

namespace fa {
namespace {

// K ring 3 deep (a slot frees as soon as S = Q K^T has read it), V ring 2
// deep (frees after PV); the producer keeps K one tile ahead of V.
constexpr int kKStages = 3, kVStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;  // 16 KiB bf16 tile

// One unit of work: query tile qt of head bh and its key-tile range.  id is
// the CTA index it was launched as (blockIdx.x), mapped by work_order.
struct Unit {
  int qt, bh, kv_bound, j_begin, j_end;
};

struct __align__(1024) FwdSmem {
  uint8_t q[kTileBytes];              // Q_i of the current unit
  uint8_t k[kKStages][kTileBytes];
  uint8_t v[kVStages][kTileBytes];
  uint64_t bar_q;
  uint64_t bar_q_empty;               // the unit's last S MMA has completed: Q may be replaced
  uint64_t bar_k_full[kKStages];
  uint64_t bar_k_empty[kKStages];
  uint64_t bar_v_full[kVStages];
  uint64_t bar_v_empty[kVStages];
  uint64_t bar_s_full;
  uint64_t bar_s_free;
  uint64_t bar_p_full;
  uint64_t bar_o_done;
  uint64_t bar_o_read;                // the softmax has read a unit's O: the next unit's PV may start
  uint64_t bar_final;
  uint64_t bar_unit_full[2];          // unit ring (producer -> MMA and softmax warps)
  uint64_t bar_unit_empty[2];
  uint64_t bar_clc;                   // completion of a launch-cancel request
  uint4 clc_resp;                     // its 16-byte response
  int unit_id[2];                     // CTA index of the unit in the slot, -1: no more units
  int unit_n[2];                      // its number of key tiles
  Unit unit_info[2];                  // the unit as the producer computed it
  uint32_t tmem_base;
  int abort;
  int16_t tiles[2][kMaxMaskTiles];    // block-sparse: the unit's key tiles, per ring slot
  uint32_t bits[kMaxMaskTiles / 32];  // CSR block mask: the row's tiles as a bitmap
};

// TMEM columns: S (fp32) at 0, P~ (bf16 pairs) at 128, O accumulator at 192.
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192, kTmemCols = 256;

constexpr uint32_t kSoftmaxWarps = 4;
// Consumers of the unit ring: the MMA warp and the four softmax warps.
constexpr uint32_t kUnitConsumers = 1 + kSoftmaxWarps;


template <bool kSplit>
__device__ __forceinline__ Unit unit_at(const FwdArgs &args, int id) {
  const Problem &pr = args.pr;
  Unit u;
  int qrank;
  work_order(pr, id, pr.nt, u.bh, qrank);
  u.qt = pr.nt - 1 - qrank;
  u.kv_bound = key_bound(pr, u.bh / pr.H);
  const int n_kv = (u.kv_bound + kTile - 1) / kTile;
  u.j_begin = 0;
  u.j_end = pr.causal ? causal_tile_end(u.qt, pr.causal_off, n_kv) : n_kv;
  if (kSplit) {
    // split-KV (no causal, no block mask): this CTA's contiguous range of key tiles
    const int per = (n_kv + args.n_split - 1) / args.n_split;
    u.j_begin = min(n_kv, static_cast<int>(blockIdx.y) * per);
    u.j_end = min(n_kv, u.j_begin + per);
  }
  return u;
}

// Launch-cancel request (cluster launch control, PTX ISA "clusterlaunchcontrol"):
// asks the hardware to cancel the launch of one CTA of this grid that has
// not started yet; the 16-byte response lands in resp and completes 16
// transaction bytes on bar.  Issued by one elected lane.
__device__ __forceinline__ void clc_try_cancel_w(uint4 *resp, uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], 16;\n\t"
      "@e clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
      "[%0], [%1];\n\t}" ::"r"(smem_u32(resp)),
      "r"(smem_u32(bar))
      : "memory");
}

// Decodes a completed response: the x index of the cancelled CTA, or -1 when
// none was left to cancel.
__device__ __forceinline__ int clc_cancelled_x(const uint4 *resp) {
  uint32_t ok, x;
  asm volatile(
      "{\n\t.reg .b128 rr;\n\t.reg .pred p;\n\t"
      "ld.shared.b128 rr, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, rr;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "mov.u32 %1, 0;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, rr;\n\t}"
      : "=r"(ok), "=r"(x)
      : "r"(smem_u32(resp))
      : "memory");
  return ok ? static_cast<int>(x) : -1;
}

// kDrop: fused dropout; kSplit: split-KV partial (key range per blockIdx.y,
// fp32 partial outputs for the merge kernel).
//
// Without split, a CTA that is about to finish its unit takes over the unit
// of a CTA of the same grid that has not been launched yet (a launch-cancel
// request), so that each of the two CTAs per SM keeps working through units
// with the next unit's schedule, Q and first K / V loads and first S
// overlapping the current unit's last tiles and epilogue, instead of paying
// a CTA launch, barrier and TMEM setup and an empty pipeline per unit.  The
// hardware hands each cancelled CTA to exactly one requester, so every unit
// is processed exactly once whatever else runs on the GPU.
template <bool kDrop, bool kSplit>
__global__ void __launch_bounds__(kThreads, 2)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdArgs args) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  FwdSmem &s = *reinterpret_cast<FwdSmem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const Problem &pr = args.pr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool sparse = pr.block_mask != nullptr || args.csr_ptr != nullptr;
  const bool persist = !kSplit && !args.starve;

  // The producer warp initialises the barriers and, for a first unit without
  // a block mask, issues its first loads (Q, K_0, V_0) at once, so that their
  // memory latency overlaps the TMEM allocation and the CTA-wide setup.
  const Unit u0 = unit_at<kSplit>(args, static_cast<int>(blockIdx.x));
  const bool early = !sparse && u0.j_end > u0.j_begin && !args.starve;
  if (warp == 4) {
    if (lane == 0) {
      mbar_init(&s.bar_q, 1);
      mbar_init(&s.bar_q_empty, 1);
      for (int i = 0; i < kKStages; ++i) {
        mbar_init(&s.bar_k_full[i], 1);
        mbar_init(&s.bar_k_empty[i], 1);
      }
      for (int i = 0; i < kVStages; ++i) {
        mbar_init(&s.bar_v_full[i], 1);
        mbar_init(&s.bar_v_empty[i], 1);
      }
      mbar_init(&s.bar_s_full, 1);
      mbar_init(&s.bar_s_free, kSoftmaxWarps);   // one arrival per softmax warp
      mbar_init(&s.bar_p_full, kSoftmaxWarps);
      mbar_init(&s.bar_o_done, 1);
      mbar_init(&s.bar_o_read, kSoftmaxWarps);
      mbar_init(&s.bar_final, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.bar_unit_full[i], 1);
        mbar_init(&s.bar_unit_empty[i], kUnitConsumers);
      }
      mbar_init(&s.bar_clc, 1);
      s.abort = 0;
      fence_mbar_init();
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    __syncwarp();
    if (early) {
      mbar_arrive_expect_tx_w(&s.bar_q, kTileBytes);
      tma_load_3d_w(s.q, &tm_q, &s.bar_q, 0, u0.qt * kTile, u0.bh);
      mbar_arrive_expect_tx_w(&s.bar_k_full[0], kTileBytes);
      tma_load_3d_w(s.k[0], &tm_k, &s.bar_k_full[0], 0, u0.j_begin * kTile, u0.bh);
      mbar_arrive_expect_tx_w(&s.bar_v_full[0], kTileBytes);
      tma_load_3d_w(s.v[0], &tm_v, &s.bar_v_full[0], 0, u0.j_begin * kTile, u0.bh);
    }
  }
  if (warp == 5) tmem_alloc(&s.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  // The producer and MMA warps run converged, whole-warp: waits are one
  // decision per warp and an elected lane issues each copy and MMA.
  if (warp == 4) {
    // ------------------------------------------------------------ producer
    int id = static_cast<int>(blockIdx.x);
    Unit u = u0;
    int g = 0;           // key tiles loaded so far (K / V ring position)
    int qn = 0;          // units with key tiles so far (Q buffer uses)
    uint32_t clc_par = 0;
    bool ok = true;
    for (int v = 0; ok; ++v) {
      // schedule of the unit ([EXPL] "Extension: Block-Sparse FlashAttention":
      // only the nonzero blocks of the row are evaluated), published to the
      // MMA and softmax warps through ring slot v & 1
      const int slot = v & 1;
      if (v >= 2 && !mbar_wait_warp(&s.bar_unit_empty[slot], ((v - 2) >> 1) & 1, pr.wait, &s.abort))
        break;
      int n = 0;
      if (id >= 0) {
        n = !sparse ? u.j_end - u.j_begin
            : args.csr_ptr
                ? compact_csr_row(args.csr_ptr, args.csr_idx, args.csr_nnz, u.qt, pr.nt, u.j_end,
                                  s.bits, s.tiles[slot], lane, pr.wait)
                : compact_mask_row(pr.block_mask + static_cast<size_t>(u.qt) * pr.nt, u.j_end,
                                   s.tiles[slot], lane);
      }
      if (lane == 0) {
        s.unit_id[slot] = id;
        s.unit_n[slot] = n;
        s.unit_info[slot] = u;   // (its kv_len lookup is not repeated by the softmax warps)
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.bar_unit_full[slot]);
      __syncwarp();
      if (id < 0) break;
      if (n > 0 && !args.starve) {
        auto tile_of = [&](int it) -> int {
          return sparse ? static_cast<int>(s.tiles[slot][it]) : u.j_begin + it;
        };
        const bool pre = early && v == 0;   // Q, K_0 and V_0 went out before the setup
        if (!pre) {
          // the previous unit's last S has completed: the Q buffer is free
          if (qn > 0 && !mbar_wait_warp(&s.bar_q_empty, (qn - 1) & 1, pr.wait, &s.abort)) break;
          mbar_arrive_expect_tx_w(&s.bar_q, kTileBytes);
          tma_load_3d_w(s.q, &tm_q, &s.bar_q, 0, u.qt * kTile, u.bh);
        }
        ++qn;
        auto load_k = [&](int it) -> bool {
          const int gt = g + it;
          const int st = gt % kKStages;
          const uint32_t use = gt / kKStages;
          if (use > 0 && !mbar_wait_warp(&s.bar_k_empty[st], (use - 1) & 1, pr.wait, &s.abort))
            return false;
          mbar_arrive_expect_tx_w(&s.bar_k_full[st], kTileBytes);
          tma_load_3d_w(s.k[st], &tm_k, &s.bar_k_full[st], 0, tile_of(it) * kTile, u.bh);
          return true;
        };
        ok = pre || load_k(0);
        for (int it = 0; ok && it < n; ++it) {
          if (it + 1 < n && !load_k(it + 1)) {
            ok = false;
            break;
          }
          if (pre && it == 0) continue;
          const int gt = g + it;
          const int st = gt % kVStages;
          const uint32_t use = gt / kVStages;
          if (use > 0 && !mbar_wait_warp(&s.bar_v_empty[st], (use - 1) & 1, pr.wait, &s.abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx_w(&s.bar_v_full[st], kTileBytes);
          tma_load_3d_w(s.v[st], &tm_v, &s.bar_v_full[st], 0, tile_of(it) * kTile, u.bh);
        }
        if (!ok) break;
        g += n;
      }
      // the next unit: taken over from a CTA of this grid not yet launched
      id = -1;
      if (persist) {
        clc_try_cancel_w(&s.clc_resp, &s.bar_clc);
        if (!mbar_wait_warp(&s.bar_clc, clc_par, pr.wait, &s.abort)) break;
        clc_par ^= 1u;
        id = clc_cancelled_x(&s.clc_resp);
        if (id >= 0) u = unit_at<kSplit>(args, id);
      }
      // no unit left for this CTA: the next kernel on the stream may launch
      // once every CTA got here.  (Triggered at the start instead, the next
      // kernel's blocks sat waiting beside the CTAs for the whole forward:
      // 1% slower steps at N = 4096.)
      if (id < 0) pdl_trigger();
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(128, 64, false, true);
    const uint64_t d_q = sdesc_sw128(smem_u32(s.q), 16, 1024);
    int g = 0, qn = 0;
    bool ok = true;
    // S of key tile gt (global count) = Q K^T into the S columns.
    auto issue_s = [&](int gt) -> bool {
      const int st = gt % kKStages;
      if (!mbar_wait_warp(&s.bar_k_full[st], (gt / kKStages) & 1, pr.wait, &s.abort))
        return false;
      tc_fence_after();
      const uint64_t d_k = sdesc_sw128(smem_u32(s.k[st]), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        mma_bf16_ss_w(tmem + kColS, d_q + kk * 2, d_k + kk * 2, idesc_s, kk > 0);
      mma_commit_w(&s.bar_s_full);
      mma_commit_w(&s.bar_k_empty[st]);
      return true;
    };
    for (int v = 0; ok; ++v) {
      const int slot = v & 1;
      if (!mbar_wait_warp(&s.bar_unit_full[slot], (v >> 1) & 1, pr.wait, &s.abort)) break;
      const int id = s.unit_id[slot], n = s.unit_n[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.bar_unit_empty[slot]);
      __syncwarp();
      if (id < 0) break;
      if (n == 0) continue;
      // Q of this unit; the S columns are free (the softmax has loaded the
      // previous unit's last S before that unit's last PV was issued)
      if (!mbar_wait_warp(&s.bar_q, qn & 1, pr.wait, &s.abort)) break;
      tc_fence_after();
      if (!issue_s(g)) break;
      for (int it = 0; ok && it < n; ++it) {
        const int gt = g + it;
        // the softmax has copied S_gt into registers: the S columns are free
        if (!mbar_wait_warp(&s.bar_s_free, gt & 1, pr.wait, &s.abort)) {
          ok = false;
          break;
        }
        if (it + 1 < n) {
          if (!issue_s(gt + 1)) {
            ok = false;
            break;
          }
        } else {
          mma_commit_w(&s.bar_q_empty);   // the unit's last S has been issued
        }
        if (!mbar_wait_warp(&s.bar_p_full, gt & 1, pr.wait, &s.abort)) {
          ok = false;
          break;
        }
        const int st = gt % kVStages;
        if (!mbar_wait_warp(&s.bar_v_full[st], (gt / kVStages) & 1, pr.wait, &s.abort)) {
          ok = false;
          break;
        }
        // the first PV of a unit overwrites O: the softmax has read the
        // previous unit's O by then
        if (it == 0 && qn > 0 && !mbar_wait_warp(&s.bar_o_read, (qn - 1) & 1, pr.wait, &s.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // A = P~ from TMEM (16 keys = 8 packed columns per step); V_j is
        // [keys][d] with d contiguous: an MN-major B operand, one 64-wide
        // swizzle atom along N, 8-key groups 1024 bytes apart.
        const uint64_t d_v = sdesc_sw128(smem_u32(s.v[st]), 1024, 1024);
        const uint32_t acc0 = it > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_bf16_ts_w(tmem + kColO, tmem + kColP + kk * 8, d_v + kk * 128, idesc_o,
                        kk > 0 ? 1u : acc0);
        mma_commit_w(&s.bar_o_done);
        mma_commit_w(&s.bar_v_empty[st]);
      }
      g += n;
      ++qn;
    }
    // make sure no MMA is in flight before TMEM is released
    mma_commit_w(&s.bar_final);
    mbar_wait_drain(&s.bar_final, 0, pr.wait);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (rows)
    const int row = tid;                   // 0..127 == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = pr.scale_log2;
    int g = 0;
    bool ok = true;
    for (int v = 0; ok; ++v) {
      const int slot = v & 1;
      if (!mbar_wait_warp(&s.bar_unit_full[slot], (v >> 1) & 1, pr.wait, &s.abort)) break;
      const int id = s.unit_id[slot], n = s.unit_n[slot];
      if (id < 0) break;
      const Unit u = s.unit_info[slot];
      const int qt = u.qt, bh = u.bh, kv_bound = u.kv_bound;
      const int qrow = qt * kTile + row;
      float m = -INFINITY;     // running max of S*scale*log2e
      float l = 0.f;           // running sum of 2^(S*scale*log2e - m)
      float m_hi = -INFINITY;  // exact running row max (m may lag it by up to kLazyRescale)
      RowDrop rd{0u};
      if (kDrop) rd.key = drop_head_key(pr, bh) ^ (static_cast<uint32_t>(qrow >> 1) << 16);
      for (int it = 0; it < n; ++it) {
        const int gt = g + it;
        const int j = sparse ? static_cast<int>(s.tiles[slot][it]) : u.j_begin + it;
        if (!mbar_wait_warp_fast(&s.bar_s_full, gt & 1, pr.wait, &s.abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[kTile];
        {
          uint32_t raw[kTile];
          const uint32_t t0 = tmem + lane_base + kColS;
          tmem_ld32(t0 + 0, raw + 0);
          tmem_ld32(t0 + 32, raw + 32);
          tmem_ld32(t0 + 64, raw + 64);
          tmem_ld32(t0 + 96, raw + 96);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < kTile; ++c) sv[c] = __uint_as_float(raw[c]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.bar_s_free);
        const int key0 = j * kTile;
        const bool edge =
            (key0 + kTile > kv_bound) || (pr.causal && key0 + kTile - 1 > qt * kTile + pr.causal_off);
        if (edge) {
          // keys >= kv_bound are padding; keys > qrow are in the future
          mask_row(sv, kv_bound - key0, pr.causal ? (qrow + pr.causal_off - key0) : kTile);
        }
        const float mxs = row_max(sv) * sl2;
        m_hi = fmaxf(m_hi, mxs);
        const float m_cand = fmaxf(m, mxs);
        const bool bump = (m == -INFINITY) || (m_cand > m + kLazyRescale);
        const float m_ref = bump ? m_cand : m;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float alpha = bump ? ex2_approx(m - m_use) : 1.f;  // 0 when m = -inf
        float rs8[8];
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) rs8[w8] = 0.f;
        // P~ in two 64-key halves; the wait for the previous PV of this unit
        // (which still reads the P~ columns and accumulates into O) sits
        // between them.  (Before a unit's first tile the previous unit's last
        // PV has completed: its epilogue waited for it.)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
          const uint32_t jp0 = static_cast<uint32_t>(key0 >> 1);
          exp_half<kDrop>(sv, half, sl2, m_use, rs8, pk, rd, pr.drop_p8, jp0);  // exact zeros where masked
          if (half == 0 && it > 0) {
            if (!mbar_wait_warp_fast(&s.bar_o_done, (gt - 1) & 1, pr.wait, &s.abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          tmem_st32(tmem + lane_base + kColP + half * 32, pk);
        }
        if (!ok) break;
        const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t to = tmem + lane_base + kColO;
          uint32_t ov[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            tmem_ld32(to + half * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(to + half * 32, ov);
          }
        }
        tmem_wait_st();
        l = l * alpha + rs;
        m = m_ref;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.bar_p_full);
      }
      if (!ok) break;
      // -------------------------------------------------------- epilogue of the unit
      float ov[kHeadDim];
      if (n > 0) {
        if (!mbar_wait_warp(&s.bar_o_done, (g + n - 1) & 1, pr.wait, &s.abort)) break;
        tc_fence_after();
        uint32_t raw[kHeadDim];
        const uint32_t to = tmem + lane_base + kColO;
        tmem_ld32(to, raw);
        tmem_ld32(to + 32, raw + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.bar_o_read);   // the next unit's PV may overwrite O
#pragma unroll
        for (int c = 0; c < kHeadDim; ++c) ov[c] = __uint_as_float(raw[c]);
      } else {
#pragma unroll
        for (int c = 0; c < kHeadDim; ++c) ov[c] = 0.f;
      }
      // the unit's schedule (and its tile list) is no longer needed
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.bar_unit_empty[slot]);
      const float inv = (n > 0 && l > 0.f) ? (kDrop ? pr.keep_scale : 1.f) / l : 0.f;
      const float lse = (n > 0 && l > 0.f) ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (qrow < pr.N) {
        if (kSplit) {
          // split-KV partial: O_s = O / l_s (fp32) and lse_s of this row, for the merge
          const size_t prow = (static_cast<size_t>(blockIdx.y) * (pr.B * pr.H) + bh) *
                                  static_cast<size_t>(args.nq_pad) + qrow;
          float4 *dst = reinterpret_cast<float4 *>(args.part_o + prow * kHeadDim);
#pragma unroll
          for (int c4 = 0; c4 < kHeadDim / 4; ++c4)
            dst[c4] = make_float4(ov[4 * c4] * inv, ov[4 * c4 + 1] * inv, ov[4 * c4 + 2] * inv,
                                  ov[4 * c4 + 3] * inv);
          args.part_lse[prow] = lse;
        } else {
          // O / l -> bf16, the row's 128 bytes straight from registers
          const size_t r = static_cast<size_t>(bh) * pr.N + qrow;
          uint4 *dst = reinterpret_cast<uint4 *>(args.o + r * kHeadDim);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const float *x = ov + ch * 8;
            dst[ch] = make_uint4(pack_bf16(x[0] * inv, x[1] * inv), pack_bf16(x[2] * inv, x[3] * inv),
                                 pack_bf16(x[4] * inv, x[5] * inv), pack_bf16(x[6] * inv, x[7] * inv));
          }
          args.lse[r] = lse;
          if (args.row_m) {
            // the pages' row statistics: m = max_j s_ij, l = sum_j exp(s_ij - m)
            const bool any = n > 0 && l > 0.f;
            args.row_m[r] = any ? m_hi * 0.69314718055994531f : -INFINITY;
            args.row_l[r] = any ? l * ex2_approx(m - m_hi) : 0.f;
          }
        }
      }
      g += n;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t fwd_smem_bytes() { return sizeof(FwdSmem) + 1024; }

// Opts both forward instantiations into their dynamic shared memory (once per device).
cudaError_t launch_fwd_config() {
  static int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    const int smem = static_cast<int>(fwd_smem_bytes());
    e = cudaFuncSetAttribute(fa_fwd_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_fwd_kernel<true, false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(fa_fwd_kernel<false, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  return cudaSuccess;
}

cudaError_t launch_fwd(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const FwdArgs &a, cudaStream_t st) {
  cudaError_t e = launch_fwd_config();
  if (e != cudaSuccess) return e;
  const size_t smem = fwd_smem_bytes();
  dim3 grid(a.pr.nt * a.pr.B * a.pr.H);
  if (a.pr.drop_p8 > 0)
    return launch_pdl(fa_fwd_kernel<true, false>, grid, dim3(kThreads), smem, st, tq, tk, tv, a);
  return launch_pdl(fa_fwd_kernel<false, false>, grid, dim3(kThreads), smem, st, tq, tk, tv, a);
}

cudaError_t launch_fwd_splitkv(const CUtensorMap &tq, const CUtensorMap &tk,
                               const CUtensorMap &tv, const FwdArgs &a, cudaStream_t st) {
  cudaError_t e = launch_fwd_config();
  if (e != cudaSuccess) return e;
  const dim3 grid(a.pr.nt * a.pr.B * a.pr.H, a.n_split);
  e = launch_pdl(fa_fwd_kernel<false, true>, grid, dim3(kThreads), fwd_smem_bytes(), st, tq, tk, tv,
                 a);
  if (e != cudaSuccess) return e;
  const dim3 mgrid((a.pr.N + 31) / 32, a.pr.B * a.pr.H);
  return launch_pdl(fa_fwd_merge_kernel<kHeadDim>, mgrid, dim3(256), 0, st, a);
}

}  // namespace fa
