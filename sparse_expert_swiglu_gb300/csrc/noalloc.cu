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
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "params.cuh"

using namespace sesg;

namespace {

constexpr int kNoAllocMaxPairs = MOE_ROUTE_NOALLOC_MAX_PAIRS;  // tokens x experts per token
constexpr size_t kCtrlBytes = 256;
constexpr size_t kScratchBytes = kCtrlBytes + (size_t)kNoAllocMaxPairs * (sizeof(int32_t) + sizeof(float));

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) uint8_t g_route_scratch[kScratchBytes];

// Device address of g_route_scratch per device (its name is only a host-side stand-in),
// with the id of the context it was looked up in: a context created later on the device
// (after cudaDeviceReset, say) loads the module again, possibly elsewhere, so the address
// is looked up again when the current context's id differs.
constexpr int kMaxDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// The current context's id, through the driver entry points the runtime hands out (the
// library links no driver library).  0 if unavailable.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static std::atomic<void*> get_current{nullptr}, get_id{nullptr};
  void* gc = get_current.load(std::memory_order_acquire);
  void* gi = get_id.load(std::memory_order_acquire);
  if (!gc || !gi) {
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &gc, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &gi, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !gc || !gi)
      return 0;
    get_current.store(gc, std::memory_order_release);
    get_id.store(gi, std::memory_order_release);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (reinterpret_cast<GetCurrent>(gc)(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (reinterpret_cast<GetId>(gi)(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

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
  // (the caller's device pointers imply a current context; without one, or without the
  // driver entry points, the id is 0 and the address is looked up on every call)
  const unsigned long long ctx = current_context_id();
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry& en = g_scratch[dev];
    if (!en.addr || en.ctx_id != ctx || ctx == 0) {
      // once per device and context, with that device current
      if (cudaGetSymbolAddress(&en.addr, g_route_scratch) != cudaSuccess || !en.addr) {
        en.addr = nullptr;
        return MOE_ERR_CUDA;
      }
      en.ctx_id = ctx;
    }
    base = en.addr;
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
