// fa_host.cu -- host-buffer entry points (fa_fwd_host, fa_fwd_bwd_host).
//
// The attention of one (b, h) depends on that head's Q, K, V (and dO) alone
// ("FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness" explainer, "Method": every head is an independent N x d
// problem), so a call on host tensors is cut into contiguous groups of heads
// and pipelined over three streams: the host-to-device copies of group c + 1
// and the device-to-host copies of group c - 1 run while the kernels of group
// c run on the caller's stream.  Each group is an ordinary fa_fwd / fa_bwd
// call on a sub-problem, so every group's result is what those entry points
// compute for its heads.
#include <cmath>
#include <mutex>

#include "fa.h"
#include "fa_kernels.cuh"

namespace fa {
namespace {

constexpr int kMaxHostChunks = 64;
constexpr int kMaxHostDevices = 64;
// events per call: start, per group (inputs copied, forward done, backward done), end
constexpr int kHostEvents = 3 * kMaxHostChunks + 2;

// The two copy streams and an event pool of one device, created on the first
// host-buffer call in a context (and again in a new context).
struct CopyEngine {
  unsigned long long ctx = 0;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev[kHostEvents] = {};
};

CopyEngine g_engine[kMaxHostDevices];
// Held while a call enqueues its work: calls share the copy streams and the
// event pool (a wait captures an event's state when it is enqueued, so the
// pool may be re-recorded by the next call at once).
std::mutex g_host_mu;

fa_status copy_engine(CopyEngine **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxHostDevices) return FA_ERR_CUDA;
  CopyEngine &c = g_engine[dev];
  const unsigned long long ctx = current_context_id();
  if (!c.h2d || ctx == 0 || ctx != c.ctx) {
    // handles of an earlier context died with it; they are not destroyed here
    c = CopyEngine{};
    if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess) {
      c = CopyEngine{};
      return FA_ERR_CUDA;
    }
    for (int i = 0; i < kHostEvents; ++i)
      if (cudaEventCreateWithFlags(&c.ev[i], cudaEventDisableTiming) != cudaSuccess) {
        c = CopyEngine{};
        return FA_ERR_CUDA;
      }
    c.ctx = current_context_id();
  }
  *out = &c;
  return FA_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Arena: device copies of q, k, v, dout, o, dq, dk, dv, lse, kv_len and the
// block mask, then the backward workspace of the whole problem (a group
// needs at most that).  The lse region gives every group its own segment
// starting on a 256-byte boundary (a group's rows need not start on one
// inside a contiguous [B, H, N] array), hence the slack of one boundary per
// group.
struct Arena {
  size_t q, k, v, dout, o, dq, dk, dv, lse, kv_len, mask, ws, ws_bytes, total;
};

Arena arena_layout(int B, int H, int N, int d) {
  const size_t t = static_cast<size_t>(B) * H * N * d * 2;
  const size_t nb = (static_cast<size_t>(N) + kTile - 1) / kTile;
  Arena a{};
  size_t off = 0;
  size_t *tensors[8] = {&a.q, &a.k, &a.v, &a.dout, &a.o, &a.dq, &a.dk, &a.dv};
  for (size_t *p : tensors) {
    *p = off;
    off += round256(t);
  }
  a.lse = off;
  off += round256(static_cast<size_t>(B) * H * N * 4) + 256 * static_cast<size_t>(kMaxHostChunks);
  a.kv_len = off;
  off += round256(static_cast<size_t>(B) * 4);
  a.mask = off;
  off += nb <= static_cast<size_t>(kMaxMaskTiles) ? round256(nb * nb) : 0;
  a.ws = off;
  a.ws_bytes = fa_bwd_workspace_size(B, H, N, d);
  a.total = off + a.ws_bytes;
  return a;
}

// One group of heads: batches [b0, b0 + nb) with all H heads, or heads
// [h0, h0 + nh) of batch b0 alone (nb = 1); either way a contiguous slab of
// the [B, H, N, d] tensors.
struct Group {
  int b0, nb, h0, nh;
};

// Cuts n units into k groups (1 <= k <= n) at first[0..k]: the first and
// the last group half as large as the others (k >= 3), so that the first
// group's inputs arrive, and the last group's results leave, with less of the
// pipeline idle.
void taper_cuts(int n, int k, int *first) {
  first[0] = 0;
  first[k] = n;
  for (int i = 1; i < k; ++i) {
    int c = k <= 2 ? static_cast<int>(static_cast<long long>(i) * n / k)
                   : static_cast<int>((static_cast<double>(n) * (i - 0.5)) / (k - 1) + 0.5);
    if (c < first[i - 1] + 1) c = first[i - 1] + 1;
    if (c > n - (k - i)) c = n - (k - i);
    first[i] = c;
  }
}

// Cuts B * H heads into about `want` groups (1 <= want <= kMaxHostChunks):
// whole batches when want <= B, else heads of one batch (tapered when B = 1);
// never more than kMaxHostChunks groups.
int plan_groups(int B, int H, int want, Group *g) {
  int first[kMaxHostChunks + 1];
  int n = 0;
  if (want <= B) {
    taper_cuts(B, want, first);
    for (int c = 0; c < want; ++c) g[n++] = Group{first[c], first[c + 1] - first[c], 0, H};
  } else if (B == 1) {
    const int k = want < H ? want : H;
    taper_cuts(H, k, first);
    for (int c = 0; c < k; ++c) g[n++] = Group{0, 1, first[c], first[c + 1] - first[c]};
  } else {
    int per = (want + B - 1) / B;
    if (per > H) per = H;
    if (per > kMaxHostChunks / B) per = kMaxHostChunks / B;   // B < want <= kMaxHostChunks
    for (int b = 0; b < B; ++b)
      for (int c = 0; c < per; ++c) {
        const int h0 = c * H / per, h1 = (c + 1) * H / per;
        if (h1 > h0) g[n++] = Group{b, 1, h0, h1 - h0};
      }
  }
  return n;
}

// Groups to use: n_chunks when given, else one per about 384 query tiles of
// 128 rows (measured on GB300: fewer groups leave the copies exposed, smaller
// ones run the kernels on too few tiles to fill the GPU), two to five; never
// more than B * H or kMaxHostChunks.
int group_count(int B, int H, int N, int n_chunks) {
  const long long bh = static_cast<long long>(B) * H;
  long long want = n_chunks;
  if (want <= 0) {
    const long long tiles = bh * ((N + kTile - 1) / kTile);
    want = (tiles + 192) / 384;
    if (want < 2) want = 2;
    if (want > 5) want = 5;
  }
  if (want > bh) want = bh;
  if (want > kMaxHostChunks) want = kMaxHostChunks;
  return static_cast<int>(want < 1 ? 1 : want);
}

fa_status host_impl(const void *q, const void *k, const void *v, const void *dout, void *o,
                    float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                    float scale, int causal, const int32_t *kv_len, const uint8_t *block_mask,
                    int n_chunks, void *arena, size_t arena_bytes, void *stream) {
  const bool bwd = dout != nullptr || dq != nullptr || dk != nullptr || dv != nullptr;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (bwd && (!dout || !dq || !dk || !dv)) return FA_ERR_INVALID_ARG;
  if (n_chunks < 0 || n_chunks > kMaxHostChunks) return FA_ERR_INVALID_ARG;
  // fa_fwd's checks, in its order
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * N >= (1LL << 31) || static_cast<long long>(B) * H >= 65536)
    return FA_ERR_INVALID_ARG;
  if (d != kHeadDim && d != kHeadDimWide) return FA_ERR_UNSUPPORTED;
  const int nb = (N + kTile - 1) / kTile;
  if (nb > kMaxGridTiles || (block_mask && nb > kMaxMaskTiles)) return FA_ERR_UNSUPPORTED;
  const size_t need = fa_host_arena_size(B, H, N, d);
  if (need == 0) return FA_ERR_UNSUPPORTED;
  if (!arena || (reinterpret_cast<uintptr_t>(arena) & 255u) != 0 || arena_bytes < need)
    return FA_ERR_WORKSPACE;
  const Arena al = arena_layout(B, H, N, d);
  uint8_t *base = static_cast<uint8_t *>(arena);
  const size_t head_elems = static_cast<size_t>(N) * d;  // bf16 words per head
  const size_t head_bytes = head_elems * 2;

  Group groups[kMaxHostChunks];
  const int ng = plan_groups(B, H, group_count(B, H, N, n_chunks), groups);
  size_t lse_seg[kMaxHostChunks];   // offset of each group's lse segment in the lse region
  size_t lse_off = 0;
  for (int c = 0; c < ng; ++c) {
    lse_seg[c] = lse_off;
    lse_off += round256(static_cast<size_t>(groups[c].nb) * groups[c].nh * N * 4);
  }

  std::lock_guard<std::mutex> lk(g_host_mu);
  CopyEngine *ce = nullptr;
  fa_status st = copy_engine(&ce);
  if (st != FA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaEvent_t *ev = ce->ev;
  cudaEvent_t ev_start = ev[0], ev_end = ev[1];
  auto ev_in = [&](int c) { return ev[2 + 3 * c]; };
  auto ev_fwd = [&](int c) { return ev[3 + 3 * c]; };
  auto ev_bwd = [&](int c) { return ev[4 + 3 * c]; };
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };

  // the copies follow the work already on the caller's stream (which may
  // still read or write the arena)
  if (!ok(cudaEventRecord(ev_start, cs)) || !ok(cudaStreamWaitEvent(ce->h2d, ev_start, 0)) ||
      !ok(cudaStreamWaitEvent(ce->d2h, ev_start, 0)))
    return FA_ERR_CUDA;
  const int32_t *kv_dev = nullptr;
  const uint8_t *mask_dev = nullptr;
  if (kv_len) {
    if (!ok(cudaMemcpyAsync(base + al.kv_len, kv_len, static_cast<size_t>(B) * 4,
                            cudaMemcpyHostToDevice, ce->h2d)))
      return FA_ERR_CUDA;
    kv_dev = reinterpret_cast<const int32_t *>(base + al.kv_len);
  }
  if (block_mask) {
    if (!ok(cudaMemcpyAsync(base + al.mask, block_mask, static_cast<size_t>(nb) * nb,
                            cudaMemcpyHostToDevice, ce->h2d)))
      return FA_ERR_CUDA;
    mask_dev = base + al.mask;
  }
  // host -> device: a group's input slabs, one copy per tensor
  auto copy_in = [&](int c) -> bool {
    const Group &g = groups[c];
    const size_t h0 = static_cast<size_t>(g.b0) * H + g.h0;
    const size_t heads = static_cast<size_t>(g.nb) * g.nh;
    const size_t off = h0 * head_bytes, bytes = heads * head_bytes;
    const void *src[4] = {q, k, v, dout};
    const size_t dst[4] = {al.q, al.k, al.v, al.dout};
    for (int t = 0; t < (bwd ? 4 : 3); ++t)
      if (!ok(cudaMemcpyAsync(base + dst[t] + off, static_cast<const uint8_t *>(src[t]) + off,
                              bytes, cudaMemcpyHostToDevice, ce->h2d)))
        return false;
    return ok(cudaEventRecord(ev_in(c), ce->h2d));
  };
  // device -> host: O and lse after the group's forward, the gradients after its backward
  auto copy_out = [&](int c) -> bool {
    const Group &g = groups[c];
    const size_t h0 = static_cast<size_t>(g.b0) * H + g.h0;
    const size_t heads = static_cast<size_t>(g.nb) * g.nh;
    const size_t off = h0 * head_bytes, bytes = heads * head_bytes;
    if (!ok(cudaStreamWaitEvent(ce->d2h, ev_fwd(c), 0)) ||
        !ok(cudaMemcpyAsync(static_cast<uint8_t *>(o) + off, base + al.o + off, bytes,
                            cudaMemcpyDeviceToHost, ce->d2h)) ||
        !ok(cudaMemcpyAsync(reinterpret_cast<uint8_t *>(lse) + h0 * N * 4,
                            base + al.lse + lse_seg[c], heads * N * 4, cudaMemcpyDeviceToHost,
                            ce->d2h)))
      return false;
    if (bwd) {
      if (!ok(cudaStreamWaitEvent(ce->d2h, ev_bwd(c), 0))) return false;
      void *dst[3] = {dq, dk, dv};
      const size_t srcoff[3] = {al.dq, al.dk, al.dv};
      for (int t = 0; t < 3; ++t)
        if (!ok(cudaMemcpyAsync(static_cast<uint8_t *>(dst[t]) + off, base + srcoff[t] + off,
                                bytes, cudaMemcpyDeviceToHost, ce->d2h)))
          return false;
    }
    return true;
  };
  // Enqueue order: the inputs of the first two groups; then per group its
  // kernels, its copies back and the inputs of the group two ahead, so that
  // each copy is queued as soon as what it waits for is.
  for (int c = 0; c < ng && c < 2; ++c)
    if (!copy_in(c)) return FA_ERR_CUDA;
  for (int c = 0; c < ng; ++c) {
    const Group &g = groups[c];
    const size_t h0 = static_cast<size_t>(g.b0) * H + g.h0;
    const size_t off = h0 * head_bytes;
    const int32_t *kvg = kv_dev ? kv_dev + g.b0 : nullptr;
    if (!ok(cudaStreamWaitEvent(cs, ev_in(c), 0))) return FA_ERR_CUDA;
    float *lse_dev = reinterpret_cast<float *>(base + al.lse + lse_seg[c]);
    st = fa_fwd(base + al.q + off, base + al.k + off, base + al.v + off, base + al.o + off,
                lse_dev, g.nb, g.nh, N, d, scale, causal, kvg, mask_dev, stream);
    if (st != FA_OK) return st;
    if (!ok(cudaEventRecord(ev_fwd(c), cs))) return FA_ERR_CUDA;
    if (bwd) {
      st = fa_bwd(base + al.q + off, base + al.k + off, base + al.v + off, base + al.o + off,
                  lse_dev, base + al.dout + off, base + al.dq + off, base + al.dk + off,
                  base + al.dv + off, g.nb, g.nh, N, d, scale, causal, kvg, mask_dev,
                  base + al.ws, al.ws_bytes, stream);
      if (st != FA_OK) return st;
      if (!ok(cudaEventRecord(ev_bwd(c), cs))) return FA_ERR_CUDA;
    }
    if (!copy_out(c)) return FA_ERR_CUDA;
    if (c + 2 < ng && !copy_in(c + 2)) return FA_ERR_CUDA;
  }
  // the caller's stream completes only after the last copy back
  if (!ok(cudaEventRecord(ev_end, ce->d2h)) || !ok(cudaStreamWaitEvent(cs, ev_end, 0)))
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

size_t fa_host_arena_size(int B, int H, int N, int d) {
  if (fa_bwd_workspace_size(B, H, N, d) == 0) return 0;
  return arena_layout(B, H, N, d).total;
}

fa_status fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                      int H, int N, int d, float scale, int causal, const int32_t *kv_len,
                      const uint8_t *block_mask, int n_chunks, void *arena, size_t arena_bytes,
                      void *stream) {
  return host_impl(q, k, v, nullptr, o, lse, nullptr, nullptr, nullptr, B, H, N, d, scale, causal,
                   kv_len, block_mask, n_chunks, arena, arena_bytes, stream);
}

fa_status fa_fwd_bwd_host(const void *q, const void *k, const void *v, const void *dout, void *o,
                          float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d,
                          float scale, int causal, const int32_t *kv_len,
                          const uint8_t *block_mask, int n_chunks, void *arena,
                          size_t arena_bytes, void *stream) {
  if (!dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  return host_impl(q, k, v, dout, o, lse, dq, dk, dv, B, H, N, d, scale, causal, kv_len,
                   block_mask, n_chunks, arena, arena_bytes, stream);
}

}  // extern "C"
