// Inter-expert prefetch: the packed up projections of predicted experts, into L2.
//
// FloE's dual sparsity predictor guesses, from an earlier hidden state, which experts a
// later layer will route to, so that their weights can be moved closer before the layer
// runs.  This file is the move.  The prediction is the caller's (the library's router
// on a predictor weight, for instance).  Only the packed up projection is moved: it is
// the part of an expert that every token routed to it reads whole.  The gate and down
// rows it will read depend on that token's mask, which is known only inside the layer.
//
// One warp per CTA and no shared memory beyond the expert list, so the CTAs fit beside
// a running decode layer on every SM.  The expert list is built again by every CTA
// (n <= 1024 ids), and the experts' bytes are spread over the grid in 16 KB bulk L2
// prefetches.  Each SM's copy engine then queues only its own share.
#include "params.cuh"

namespace sesg {
namespace {

constexpr int kPfThreads = 32;
constexpr uint32_t kPfChunk = 16384;
constexpr int kPfMaxE = 256;

__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__global__ void __launch_bounds__(kPfThreads) expert_prefetch_kernel(const uint8_t* __restrict__ up,
                                                                     size_t up_bytes, int E,
                                                                     const int32_t* __restrict__ idx, int n,
                                                                     int max_experts) {
  __shared__ uint32_t flags[kPfMaxE / 32];
  __shared__ int16_t list[kPfMaxE];
  const int lane = threadIdx.x;
  if (lane < kPfMaxE / 32) flags[lane] = 0u;
  __syncwarp();
  for (int j = lane; j < n; j += kPfThreads) {
    const int e = idx[j];
    if (e >= 0 && e < E) atomicOr(&flags[e >> 5], 1u << (e & 31));
  }
  __syncwarp();
  // the distinct experts in ascending order: lane w owns flag word w
  int cnt = lane < kPfMaxE / 32 ? __popc(flags[lane]) : 0;
  int before = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, before, off);
    if (lane >= off) before += o;
  }
  before -= cnt;
  const int nu = min(__shfl_sync(0xffffffffu, before + cnt, 31), max_experts);
  if (lane < kPfMaxE / 32) {
    uint32_t w = flags[lane];
    for (int r = before; w != 0u; ++r) {
      const int b = __ffs(w) - 1;
      w &= w - 1u;
      list[r] = (int16_t)(lane * 32 + b);
    }
  }
  __syncwarp();
  const size_t per = (up_bytes + kPfChunk - 1) / kPfChunk;
  const size_t total = (size_t)nu * per;
  for (size_t c = (size_t)blockIdx.x * kPfThreads + lane; c < total; c += (size_t)gridDim.x * kPfThreads) {
    const size_t u = c / per, off = (c - u * per) * kPfChunk;
    const uint32_t bytes = (uint32_t)min((size_t)kPfChunk, up_bytes - off);
    bulk_prefetch_l2(up + (size_t)list[u] * up_bytes + off, bytes);
  }
}

}  // namespace

cudaError_t launch_expert_prefetch(const uint8_t* up, size_t up_bytes, int E, const int32_t* idx, int n,
                                   int max_experts, int P, cudaStream_t st) {
  expert_prefetch_kernel<<<P, kPfThreads, 0, st>>>(up, up_bytes, E, idx, n, max_experts);
  return cudaGetLastError();
}

}  // namespace sesg
