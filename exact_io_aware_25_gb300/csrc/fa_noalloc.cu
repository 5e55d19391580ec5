// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass without a caller-provided
// workspace, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) when they
// run the backward pass: for example a plugin inside a host application that
// owns every device allocation itself, or a latency-critical loop that must
// not pay for an allocation or the device synchronisation cudaMalloc may
// imply.  For them this entry point takes its scratch from a fixed array
// that lives in the library's device image (64 MiB).
//
// The array is reserved in device memory when the module that holds it is
// loaded into a context.  Under CUDA's default lazy module loading that is
// the first call of this entry point on each device (the address lookup
// below loads it); with eager loading it is when the context is created.
// Either way the memory stays reserved until the context is destroyed, and
// the first call can fail with FA_ERR_CUDA when the device has no 64 MiB to
// spare; it may also synchronise.  Make that first call outside
// latency-critical code and before any stream capture.
//
// The array's host-side name is only a stand-in for the device symbol, so
// host code never passes it to a kernel; the device address is looked up
// with cudaGetSymbolAddress with the device current and cached per device
// together with the identifier of the context it belongs to, so a call made
// in another context (or after the device was reset) looks it up again.
// Calls that overlap on the GPU (on different streams, or from different
// host threads) share the one array and race; the caller must order them.
// Each call rewrites every scratch byte it reads (the preprocessing kernel
// clears the dQ accumulators and writes D and the base-2 log-sum-exp), so the
// previous call's contents never matter.
#include <mutex>

#include "fa.h"
#include "fa_kernels.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};

}  // namespace

extern "C" {

size_t fa_bwd_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv, int B,
                         int H, int N, int d, float scale, int causal, const int32_t *kv_len,
                         const uint8_t *block_mask, void *stream) {
  // fa_bwd checks every argument before it looks at the workspace and
  // launches nothing without one: called with none, it returns exactly the
  // status it gives these arguments, or FA_ERR_WORKSPACE when they are valid.
  const fa_status pre = fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal,
                               kv_len, block_mask, nullptr, 0, stream);
  if (pre != FA_ERR_WORKSPACE) return pre;
  if (fa_bwd_workspace_size(B, H, N, d) > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    const unsigned long long ctx = fa::current_context_id();
    if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return FA_ERR_CUDA;
      g_noalloc_ptr[dev] = p;
      g_noalloc_ctx[dev] = fa::current_context_id();
    }
    scratch = g_noalloc_ptr[dev];
  }
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, causal, kv_len, block_mask,
                scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
