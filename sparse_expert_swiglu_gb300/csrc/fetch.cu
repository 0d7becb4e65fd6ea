// FloE's on-the-fly mode ("FloE: On-the-Fly MoE Inference on Memory-constrained GPU",
// sec. 三 "系统协同优化" and its expert-offloading setting): the experts' gate and down
// rows stay in page-locked host memory and only the rows that the masks keep cross to the
// GPU.  This kernel runs between the decode up kernel (which has listed the kept columns
// of every up CTA) and the decode gather kernel: CTA c copies the kept rows of up CTA c,
// in list order, to rows [prefix(c), prefix(c) + count(c)) of a staging area in device
// memory, 4d bytes per row (gate row, then down row).  That is the global kept-row order
// in which the gather kernel's CTAs split the rows, so the gather streams row r of the
// staging area where it would read column r's rows from the experts.
//
// Host memory is read with plain 16-byte loads through the unified address space (the
// NVLink-C2C or PCIe link); each warp copies one row at a time, every lane keeping 8
// loads in flight.
#include "params.cuh"

namespace sesg {

constexpr int kFetchThreads = 512;
constexpr int kFetchUnroll = 8;

__global__ void __launch_bounds__(kFetchThreads) decode_fetch_kernel(DecodeParams p) {
  __shared__ int s_pre;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  const int c = blockIdx.x;
  griddep_wait();
  griddep_launch_dependents();
  // rows of the up CTAs before this one (exclusive prefix of their kept counts)
  if (warp == 0) {
    int part = 0;
    for (int i = lane; i < c; i += 32) part += min(__ldcg(p.cta_total + i), p.kcap);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) s_pre = part;
  }
  __syncthreads();
  const int n = min(__ldcg(p.cta_total + c), p.kcap);  // a list holds at most kcap entries
  const int d = p.d;
  const int cpr = d / 4;   // 16-byte chunks per row
  const int half = d / 8;  // chunks of the gate row
  const int4* list = p.klist + (size_t)c * p.kcap;
  uint4* dst = reinterpret_cast<uint4*>(p.staging) + (size_t)s_pre * cpr;
  for (int j = warp; j < n; j += nw) {
    const int e = __ldcg(&list[j].x);
    const int col = e & 0xffff, g = e >> 16;
    const int expert = __ldcg(&p.groups[g].expert);
    const bool routed = expert < p.routed.E;
    const ExpertSet& es = routed ? p.routed : p.shared;
    const int el = routed ? expert : expert - p.routed.E;
    const size_t roff = ((size_t)el * es.f + col) * es.rs;
    const uint4* gsrc = reinterpret_cast<const uint4*>(es.gate_t + roff);
    const uint4* dsrc = reinterpret_cast<const uint4*>(es.down + roff);
    uint4* out = dst + (size_t)j * cpr;
    for (int q0 = lane; q0 < cpr; q0 += 32 * kFetchUnroll) {
      uint4 v[kFetchUnroll];
#pragma unroll
      for (int u = 0; u < kFetchUnroll; ++u) {
        const int q = q0 + 32 * u;
        if (q < cpr) v[u] = q < half ? gsrc[q] : dsrc[q - half];
      }
#pragma unroll
      for (int u = 0; u < kFetchUnroll; ++u) {
        const int q = q0 + 32 * u;
        if (q < cpr) out[q] = v[u];
      }
    }
  }
}

cudaError_t launch_decode_fetch(const DecodeParams& p, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.P);
  cfg.blockDim = dim3(kFetchThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, decode_fetch_kernel, p);
}

}  // namespace sesg
