// Shared device-side definitions of the sparse-SwiGLU MoE decode library (sm_103a).
//
// Layout constants, the device copies of the public structs, the work-descriptor
// types that the kernels exchange through the caller's workspace, and thin inline
// PTX wrappers (mma.sync, mbarrier, cp.async.bulk, programmatic dependent launch).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sparse_expert_swiglu.h"

namespace sesg {

// ---------------------------------------------------------------------------
// Packed INT2 W^up layout (one expert; see expert_int2_up_packed_bytes()).
//
// The expert is cut into blocks of 16 output columns (an "M-tile", the M side of
// an m16n8k16 tensor-core tile) by 512 input rows (a "superblock" of 8 quantiser
// groups of 64).  Blocks are stored M-tile major, so the whole d-strip of one
// M-tile is contiguous.  A block is 2560 bytes:
//   [0, 2048)    codes: uint4 u (0..3) x lane (0..31), 16 bytes each, i.e. the
//                A-operand fragments of one warp for 4 k-steps of every group
//   [2048, 2560) (scale, zero) fp16 pairs: [16 columns][8 groups]
// Lane l = 4*gl + c, word w = 4*u + r of its uint4s holds, for each group slot
// n (0..7) of the superblock, two codes at bits 2n (low half) and 16+2n (high
// half): q[k][j] and q[k+1][j] with
//   j = 16*mtile + gl + 8*(r & 1)
//   k = 512*sb + 64*n + 16*u + 2*c + 8*(r >> 1)
// which are exactly the (row, k) pairs of A-fragment register r of an
// m16n8k16 f16 mma for k-step u of group n.
// ---------------------------------------------------------------------------
constexpr int kGroup = 64;
constexpr int kSuper = 512;
constexpr int kMTile = 16;
constexpr int kBlkCodeBytes = 2048;
constexpr int kBlkBytes = 2560;
constexpr int kMaxTok = 8;       // tokens of one expert handled together
constexpr int kMaxSlots = 16;    // k + n_shared per token

__host__ __device__ inline int n_superblocks(int d) { return (d + kSuper - 1) / kSuper; }
__host__ __device__ inline size_t packed_bytes_per_expert(int d, int f) {
  return (size_t)(f / kMTile) * n_superblocks(d) * kBlkBytes;
}

// Codes of one block word as an mma A-operand register.
template <int GI>
__device__ __forceinline__ uint32_t code_pair(uint32_t w) {
  // Two 2-bit codes of group slot GI as an fp16x2 of subnormals q * 4^pos * 2^-24
  // (exact); the power of two is removed after the mma.  Slots 5..7 sit above the
  // 10-bit mantissa and are shifted down first.
  if constexpr (GI < 5) return w & (0x00030003u << (2 * GI));
  else return (w >> 10) & (0x00030003u << (2 * (GI - 5)));
}

__device__ __forceinline__ float pos_scale(int gi) {
  const int pos = gi < 5 ? gi : gi - 5;
  return __int_as_float((127 + 24 - 2 * pos) << 23);  // 2^(24 - 2 pos)
}

// Device copy of moe_experts_t.
struct ExpertSet {
  int E, d, f;
  const uint8_t* up;
  const __half* gate_t;
  const __half* down;
  const float* thr;
  size_t up_stride;  // bytes per expert of the packed up projection
  int rs;            // elements between consecutive gate (and down) rows: d, or 2d when
                     // gate and down rows are interleaved in one buffer (down == gate_t + d)
};

// One unit of expert work: an expert and up to 8 of the tokens routed to it.
struct GroupDesc {
  int expert;        // < routed.E: routed expert; else shared expert expert - routed.E
  int n_tok;         // 1..8
  int tok[kMaxTok];  // token index into x / y
  int slot[kMaxTok]; // which of the token's k (+ shared) experts this is
  float w[kMaxTok];  // combine weight (router weight, 1 for shared experts)
};

// Workspace control block (zeroed by moe_workspace_init; kernels leave it reusable).
struct Ctrl {
  int status;        // first device-side error, MOE_OK if none
  int route_done;    // last-CTA counter of the router
  int G;             // number of groups of the current call
  int reserved0;     // unused (keeps the block's layout)
  int N;             // total kept items of the current call (written by the gather kernel)
  int reserved1;     // unused
  int gdone;         // decode gather CTAs that have added their share of y
  int pad1;
};

__device__ inline void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ld_nc_v2(const void* p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ uint32_t ld_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// b * m for fp16x2 b and m = (1, 1) or (0, 0): b or zeros, exactly (x is finite).  Used to
// zero an mma B operand on the FMA pipe rather than by a select on the integer pipe.
__device__ __forceinline__ uint32_t hmul2_mask(uint32_t b, uint32_t m) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(b), "r"(m));
  return r;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000000;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: every try_wait suspends for at most ~1 ms, so the bound is a few
// seconds of wall time; on expiry the caller records MOE_ERR_TIMEOUT and bails out.
constexpr uint32_t kWaitTries = 4000;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitTries; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// 1-D bulk copy global -> shared, completion counted on an mbarrier (bytes, dst, src 16-B aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + __expf(-g)); }

}  // namespace sesg
