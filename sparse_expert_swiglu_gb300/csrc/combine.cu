// Combination of the experts of a token, y_b = sum_j w_bj E_j(x_b) + sum_s E_s(x_b)
// (the router weights are already folded into the gather kernel's partial outputs),
// the single fp16 rounding of y, and, for stacked layers, the RMSNorm
// y / sqrt(mean(y^2) + 1e-6) that hands the hidden state to the next layer.
//
// Grid: 8 CTAs per token, each owning d/8 hidden elements.  The partial rows of
// every (gather CTA, group) pair that holds the token are added in a fixed order,
// so the result is bitwise reproducible.  With RMSNorm the 8 CTAs of a token form a
// thread-block cluster and exchange their sums of squares through distributed
// shared memory.
#include <cooperative_groups.h>

#include "params.cuh"

namespace cg = cooperative_groups;

namespace sesg {

// Threads per CTA: 1024 up to 8 tokens (more subsets of the partial rows, one round of
// loads), 256 above (several CTAs per SM, so that 8 CTAs per token still run in one
// wave); 256 threads cover the d / 32 float4 columns of a CTA for d <= 8192.
__host__ __device__ constexpr int comb_threads(int B) { return B <= 8 ? 1024 : 256; }
constexpr int kCombSlices = 8;

__device__ __forceinline__ long long cta_first_item(long long N, int c, int P) { return N * c / P; }
__device__ __forceinline__ int cta_of_item(long long i, long long N, int P) {
  return (int)(((i + 1) * P + N - 1) / N) - 1;
}

template <bool RMS, int kCombThreads>
__global__ void __launch_bounds__(kCombThreads) combine_kernel(ExpertParams p) {
  extern __shared__ float4 comb_smem[];
  const int P = p.P3;
  float4* s_red = comb_smem;                                   // [kCombThreads]
  int* s_bound = reinterpret_cast<int*>(comb_smem + kCombThreads);  // [P+1] first item of every gather CTA
  int* s_gtot = s_bound + P + 1;            // [G_max+1] group item offsets
  int* s_list = s_gtot + p.G_max + 1;       // [n_slots * P] partial rows (-1: empty range)
  __shared__ int s_slot[kMaxSlots][4];      // c_lo, count, group, tau
  __shared__ int s_off[kMaxSlots + 1];
  __shared__ int s_tg[kMaxSlots];
  __shared__ int s_meta[2];
  __shared__ float s_ss[32];
  __shared__ float s_cluster_ss;
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.y, slice = blockIdx.x;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int d = p.d;
  const int sw = d / kCombSlices;           // hidden elements of this CTA
  const int F4 = sw / 4;
  const int NS = min(32, kCombThreads / F4);  // subsets of the partial rows
  const int f4 = t % F4, sub = t / F4;

  // one round of loads: call size, group totals, the token's (group, slot) pairs
  if (t == 0) {
    s_meta[0] = *reinterpret_cast<volatile int*>(&p.ctrl->N);
    s_meta[1] = *reinterpret_cast<volatile int*>(&p.ctrl->G);
  }
  for (int g = t; g < p.G_max; g += kCombThreads) s_gtot[g] = __ldcg(p.group_total + g);
  if (t < p.n_slots) s_tg[t] = p.tok_groups[b * kMaxSlots + t];
  __syncthreads();
  const long long N = s_meta[0];
  const int G = s_meta[1];
  for (int c = t; c <= P; c += kCombThreads) s_bound[c] = (int)cta_first_item(N, c, P);
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < G; base += 32) {
      const int i = base + lane;
      const int v = i < G ? s_gtot[i] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      __syncwarp();
      if (i < G) s_gtot[i] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_gtot[G] = carry;
  }
  __syncthreads();
  if (t < p.n_slots) {
    const int tg = s_tg[t];
    const int g = tg >> 3;
    const long long s0 = s_gtot[g], s1 = s_gtot[g + 1];
    int lo = 0, cnt = 0;
    if (s1 > s0) {
      lo = cta_of_item(s0, N, P);
      cnt = cta_of_item(s1 - 1, N, P) - lo + 1;
    }
    s_slot[t][0] = lo;
    s_slot[t][1] = cnt;
    s_slot[t][2] = g;
    s_slot[t][3] = tg & 7;
  }
  __syncthreads();
  if (t == 0) {
    int o = 0;
    for (int j = 0; j < p.n_slots; ++j) {
      s_off[j] = o;
      o += s_slot[j][1];
    }
    s_off[p.n_slots] = o;
  }
  __syncthreads();
  const int total = s_off[p.n_slots];
  for (int i = t; i < total; i += kCombThreads) {
    int j = 0;
    while (s_off[j + 1] <= i) ++j;
    const int c = s_slot[j][0] + (i - s_off[j]);
    s_list[i] = (s_bound[c] == s_bound[c + 1]) ? -1 : (c + s_slot[j][2]) * kMaxTok + s_slot[j][3];
  }
  __syncthreads();

  // the partial rows, NS subsets in parallel, 8 loads in flight per thread
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int col = slice * sw + f4 * 4;
  if (sub < NS) {
    constexpr int LU = 8;
    for (int i0 = sub; i0 < total; i0 += NS * LU) {
      float4 v[LU];
#pragma unroll
      for (int u = 0; u < LU; ++u) {
        const int i = i0 + u * NS;
        const int row = i < total ? s_list[i] : -1;
        v[u] = row < 0 ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : __ldcg(reinterpret_cast<const float4*>(p.part + (size_t)row * d + col));
      }
#pragma unroll
      for (int u = 0; u < LU; ++u) {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
    s_red[sub * F4 + f4] = acc;
  }
  __syncthreads();
  float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
  if (sub == 0) {
    y = s_red[f4];
    for (int s = 1; s < NS; ++s) {
      const float4 v = s_red[s * F4 + f4];
      y.x += v.x;
      y.y += v.y;
      y.z += v.z;
      y.w += v.w;
    }
  }
  float rinv = 1.f;
  if constexpr (RMS) {
    float ss = sub == 0 ? y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) s_ss[warp] = ss;
    __syncthreads();
    if (t == 0) {
      float tot = 0.f;
      for (int w = 0; w < kCombThreads / 32; ++w) tot += s_ss[w];
      s_cluster_ss = tot;
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (t == 0) {
      float tot = 0.f;
      for (int r = 0; r < kCombSlices; ++r) tot += *cluster.map_shared_rank(&s_cluster_ss, r);
      s_ss[0] = rsqrtf(tot / (float)d + 1e-6f);
    }
    cluster.sync();  // every CTA has read the others' sums before any of them exits
    rinv = s_ss[0];
  }
  if (sub == 0) {
    __half2* yo = reinterpret_cast<__half2*>(p.y + (size_t)b * d + col);
    yo[0] = __floats2half2_rn(y.x * rinv, y.y * rinv);
    yo[1] = __floats2half2_rn(y.z * rinv, y.w * rinv);
  }
}

size_t combine_smem_bytes(const ExpertParams& p) {
  const size_t ints = (size_t)p.P3 + 1 + p.G_max + 1 + (size_t)p.n_slots * p.P3 + 4;
  return ints * 4 + (size_t)comb_threads(p.B) * 16;
}

template <bool RMS, int NT>
static cudaError_t launch_comb(cudaLaunchConfig_t& cfg, const ExpertParams& p, size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(combine_kernel<RMS, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, combine_kernel<RMS, NT>, p);
}

cudaError_t launch_combine(const ExpertParams& p, cudaStream_t st, bool pdl) {
  const size_t smem = combine_smem_bytes(p);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCombSlices, p.B);
  cfg.blockDim = dim3(comb_threads(p.B));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.rmsnorm) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = kCombSlices;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (p.rmsnorm) {
    return comb_threads(p.B) == 1024 ? launch_comb<true, 1024>(cfg, p, smem) : launch_comb<true, 256>(cfg, p, smem);
  }
  return comb_threads(p.B) == 1024 ? launch_comb<false, 1024>(cfg, p, smem) : launch_comb<false, 256>(cfg, p, smem);
}

}  // namespace sesg
