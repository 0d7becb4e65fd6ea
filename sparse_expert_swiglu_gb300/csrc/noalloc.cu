// moe_route_topk_noalloc: the router entry point for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain a device buffer: code that runs where
// cudaMalloc is not allowed or not wanted (a plugin handed only input and output
// pointers by its host framework, a runtime whose memory is a fixed pre-sized pool,
// a latency-critical path where an allocation would synchronise the device).  This
// entry point gives them the router without a caller workspace: its scratch (the
// control block with the cross-CTA counter, and the kernel's copy of the top-k
// result) lives in a file-scope device array that every GPU loading the library
// holds until the process exits.  The router kernel and its launch are the same as
// moe_route_topk's; only where its scratch lives differs.
#include <atomic>

#include "params.cuh"

using namespace sesg;

namespace {

constexpr int kNoAllocMaxPairs = MOE_ROUTE_NOALLOC_MAX_PAIRS;  // tokens x experts per token
constexpr size_t kCtrlBytes = 256;
constexpr size_t kScratchBytes = kCtrlBytes + (size_t)kNoAllocMaxPairs * (sizeof(int32_t) + sizeof(float));

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) uint8_t g_route_scratch[kScratchBytes];

// Device address of g_route_scratch per device (its name is only a host-side stand-in).
constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

inline bool aligned16(const void* p) { return ((uintptr_t)p % 16) == 0; }

}  // namespace

extern "C" moe_status_t moe_route_topk_noalloc(const uint16_t* x, int32_t B, int32_t d,
                                               const uint16_t* w_router, int32_t E, int32_t k,
                                               int32_t renorm, int32_t* topk_idx, float* topk_w,
                                               int32_t* expert_count, void* stream) {
  if (B < 0 || d <= 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (B > 1024 || E > 256 || k > kMaxTok || d % 256 || d > 7936) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)B * k > kNoAllocMaxPairs) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (B == 0) return MOE_OK;
  if (!x || !w_router || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router)) return MOE_ERR_ALIGNMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED_SHAPE;
  void* base = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!base) {
    // once per device, with that device current
    if (cudaGetSymbolAddress(&base, g_route_scratch) != cudaSuccess || !base) return MOE_ERR_CUDA;
    g_scratch_addr[dev].store(base, std::memory_order_release);
  }
  uint8_t* ws = static_cast<uint8_t*>(base);
  cudaStream_t st = (cudaStream_t)stream;
  // the cross-CTA counter and the status word must start at zero
  if (cudaMemsetAsync(ws, 0, sizeof(Ctrl), st) != cudaSuccess) return MOE_ERR_CUDA;
  RouteParams rp = {};
  rp.x = reinterpret_cast<const __half*>(x);
  rp.w_router = reinterpret_cast<const __half*>(w_router);
  rp.B = B;
  rp.d = d;
  rp.E = E;
  rp.k = k;
  rp.renorm = renorm ? 1 : 0;
  rp.group = 0;
  rp.gcap = kMaxTok;
  rp.topk_idx = reinterpret_cast<int32_t*>(ws + kCtrlBytes);
  rp.topk_w = reinterpret_cast<float*>(ws + kCtrlBytes + (size_t)kNoAllocMaxPairs * sizeof(int32_t));
  rp.user_idx = topk_idx;
  rp.user_w = topk_w;
  rp.expert_count = expert_count;
  rp.ctrl = reinterpret_cast<Ctrl*>(ws);
  return launch_route(rp, st, true) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
