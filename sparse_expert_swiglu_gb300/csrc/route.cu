// Router GEMV + softmax top-k of every token, and the grouping of (token, expert)
// pairs into expert work groups.
//
// "MoE-Lightning: High-Throughput MoE Inference on Memory-constrained GPUs", sec. 三
// "MoE 模型架构": a gating network chooses the top-k experts of every token;
// "MOE-INFINITY ...", sec. A3 background: Mixtral-8x7B routes each token to 2 of
// its 8 experts.  Ties between equal logits go to the lower expert index; the
// chosen experts are listed by logit descending; renorm selects softmax over the
// chosen logits (1) or the full softmax over all experts (0).
#include "params.cuh"

namespace sesg {


constexpr int kRouteThreads = 512;

// Logits of one token: each thread owns EV consecutive experts and a strided set of
// rows; the rows are fetched RU at a time so that their loads are in flight together.
template <int EV>
__device__ void router_logits(const RouteParams& p, int b, float* logits, float* red) {
  constexpr int RU = 16;
  const int tid = threadIdx.x;
  const int nchunk = p.E / EV;             // expert chunks
  const int nrs = kRouteThreads / nchunk;  // row slots
  const int ec = tid % nchunk, rs = tid / nchunk;
  float acc[EV];
#pragma unroll
  for (int i = 0; i < EV; ++i) acc[i] = 0.f;
  if (rs < nrs) {
    const __half* xb = p.x + (size_t)b * p.d;
    // (a CTA of kRouteThreads covers nrs * RU rows per pass: every load of a pass is
    // in flight at once)
    for (int r0 = rs; r0 < p.d; r0 += nrs * RU) {
      float xv[RU];
      uint4 wv[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int r = r0 + u * nrs;
        xv[u] = 0.f;
        wv[u] = make_uint4(0, 0, 0, 0);
        if (r < p.d) {
          xv[u] = __half2float(xb[r]);
          const __half* wrow = p.w_router + (size_t)r * p.E + ec * EV;
          if constexpr (EV == 8) wv[u] = *reinterpret_cast<const uint4*>(wrow);
          else wv[u].x = (uint32_t)__half_as_ushort(wrow[0]);
        }
      }
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        if constexpr (EV == 8) {
          const __half2* h2 = reinterpret_cast<const __half2*>(&wv[u]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 wf = __half22float2(h2[i]);
            acc[2 * i] = fmaf(xv[u], wf.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(xv[u], wf.y, acc[2 * i + 1]);
          }
        } else {
          acc[0] = fmaf(xv[u], __half2float(__ushort_as_half((unsigned short)wv[u].x)), acc[0]);
        }
      }
    }
  }
  // red[rs][e], then a fixed-order sum over the row slots: warp w adds the slots of
  // experts w, w + 16, ... with its lanes taking every 32nd slot, then a butterfly
  if (rs < nrs) {
#pragma unroll
    for (int i = 0; i < EV; ++i) red[rs * p.E + ec * EV + i] = acc[i];
  }
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5, nwarps = kRouteThreads / 32;
  for (int e = warp; e < p.E; e += nwarps) {
    float s0 = 0.f, s1 = 0.f;
    int r = lane;
    for (; r + 32 < nrs; r += 64) {
      s0 += red[r * p.E + e];
      s1 += red[(r + 32) * p.E + e];
    }
    if (r < nrs) s0 += red[r * p.E + e];
    float s = s0 + s1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) logits[e] = s;
  }
  __syncthreads();
}

// Warp 0: k rounds of arg-max (larger logit, then lower index), softmax weights.
__device__ void router_topk(const RouteParams& p, int b, const float* logits, int* s_idx_out,
                            float* s_w_out) {
  const int lane = threadIdx.x & 31;
  constexpr int kPer = 8;  // E <= 256
  float l[kPer];
  bool taken[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    // a NaN logit (from a non-finite token) ranks as -inf, so that the k chosen experts
    // are always k distinct valid ones
    const float le = e < p.E ? logits[e] : -INFINITY;
    l[i] = isnan(le) ? -INFINITY : le;
    taken[i] = e >= p.E;
  }
  float lmax = -INFINITY;
  int sel_idx[8];
  float sel_l[8];
  for (int j = 0; j < p.k; ++j) {
    float best = -INFINITY;
    int bidx = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && (l[i] > best || (l[i] == best && e < bidx))) {
        best = l[i];
        bidx = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, off);
      if (ob > best || (ob == best && oi < bidx)) {
        best = ob;
        bidx = oi;
      }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i == bidx) taken[i] = true;
    sel_idx[j] = bidx;
    sel_l[j] = best;
    if (j == 0) lmax = best;
  }
  float denom = 0.f;
  if (p.renorm) {
    for (int j = 0; j < p.k; ++j) denom += expf(sel_l[j] - lmax);
  } else {
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i < p.E) part += expf(l[i] - lmax);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    denom = part;
  }
  if (lane == 0) {
    for (int j = 0; j < p.k; ++j) {
      const float w = expf(sel_l[j] - lmax) / denom;
      p.topk_idx[b * p.k + j] = sel_idx[j];
      p.topk_w[b * p.k + j] = w;
      if (s_idx_out) {
        s_idx_out[b * p.k + j] = sel_idx[j];
        s_w_out[b * p.k + j] = w;
      }
      if (p.user_idx) p.user_idx[b * p.k + j] = sel_idx[j];
      if (p.user_w) p.user_w[b * p.k + j] = w;
    }
  }
}

// Last CTA: counting of tokens per expert and the expert work groups.  Every pair sets
// its token's bit in its expert's token mask (a token's k experts are distinct), so an
// expert's count is a popcount and its tokens come out in ascending order by walking
// the set bits: no loop over all pairs per expert.
__device__ void router_group(const RouteParams& p, bool local) {
  extern __shared__ float dyn[];
  int* s_idx = reinterpret_cast<int*>(dyn);   // [B*k]
  int* s_list = s_idx + p.B * p.k;            // [B*k] (token << 4 | slot) grouped by expert
  float* s_w = reinterpret_cast<float*>(s_list + p.B * p.k);  // [B*k]
  uint32_t* s_em = reinterpret_cast<uint32_t*>(s_w + p.B * p.k);  // [E][ceil(B/32)] token masks
  const int nw = (p.B + 31) / 32;
  __shared__ int s_cnt[256], s_off[257], s_goff[257];
  const int tid = threadIdx.x;
  const int npair = p.B * p.k;
  if (!local) {  // top-k results of other CTAs: read them back through L2
    for (int i = tid; i < npair; i += kRouteThreads) {
      s_idx[i] = __ldcg(p.topk_idx + i);
      s_w[i] = __ldcg(p.topk_w + i);
    }
  }
  for (int w = tid; w < p.E * nw; w += kRouteThreads) s_em[w] = 0u;
  __syncthreads();
  for (int i = tid; i < npair; i += kRouteThreads) {
    const int b = i / p.k;
    atomicOr(&s_em[s_idx[i] * nw + (b >> 5)], 1u << (b & 31));
  }
  __syncthreads();
  for (int e = tid; e < p.E; e += kRouteThreads) {
    int c = 0;
    for (int w = 0; w < nw; ++w) c += __popc(s_em[e * nw + w]);
    s_cnt[e] = c;
    if (p.expert_count) p.expert_count[e] = c;
  }
  __syncthreads();
  if (tid < 32) {
    // exclusive prefixes of the pair counts and of the group counts (warp scans)
    int o = 0, go = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + tid;
      const int c = e < p.E ? s_cnt[e] : 0, gc = (c + p.gcap - 1) / p.gcap;
      int ic = c, ig = gc;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int oc = __shfl_up_sync(0xffffffffu, ic, off), og = __shfl_up_sync(0xffffffffu, ig, off);
        if (tid >= off) {
          ic += oc;
          ig += og;
        }
      }
      if (e < p.E) {
        s_off[e] = o + ic - c;
        s_goff[e] = go + ig - gc;
      }
      o += __shfl_sync(0xffffffffu, ic, 31);
      go += __shfl_sync(0xffffffffu, ig, 31);
    }
    if (tid == 0) {
      s_off[p.E] = o;
      s_goff[p.E] = go;
    }
  }
  __syncthreads();
  if (!p.group) return;
  // tokens of expert e in ascending order, each with the slot j where it chose e
  for (int e = tid; e < p.E; e += kRouteThreads) {
    int o = s_off[e];
    for (int w = 0; w < nw; ++w) {
      uint32_t m = s_em[e * nw + w];
      while (m) {
        const int b = w * 32 + __ffs(m) - 1;
        m &= m - 1;
        int j = 0;
        while (j + 1 < p.k && s_idx[b * p.k + j] != e) ++j;
        s_list[o++] = (b << 4) | j;
      }
    }
  }
  __syncthreads();
  const int g_routed = s_goff[p.E];
  const int g_per_shared = (p.B + p.gcap - 1) / p.gcap;
  const int G = g_routed + p.n_shared * g_per_shared;
  for (int e = tid; e < p.E; e += kRouteThreads) {
    const int n = s_cnt[e];
    for (int q = 0; q * p.gcap < n; ++q) {
      GroupDesc gd;
      gd.expert = e;
      gd.n_tok = min(p.gcap, n - q * p.gcap);
      const int g = s_goff[e] + q;
      for (int t = 0; t < kMaxTok; ++t) {
        if (t < gd.n_tok) {
          const int pr = s_list[s_off[e] + q * p.gcap + t];
          const int b = pr >> 4, j = pr & 15;
          gd.tok[t] = b;
          gd.slot[t] = j;
          gd.w[t] = s_w[b * p.k + j];
          p.tok_groups[b * kMaxSlots + j] = (g << 3) | t;
        } else {
          gd.tok[t] = 0;
          gd.slot[t] = 0;
          gd.w[t] = 0.f;
        }
      }
      p.groups[g] = gd;
    }
  }
  for (int q = tid; q < p.n_shared * g_per_shared; q += kRouteThreads) {
    const int s = q / g_per_shared, qq = q % g_per_shared;
    GroupDesc gd;
    gd.expert = p.E + s;
    gd.n_tok = min(p.gcap, p.B - qq * p.gcap);
    const int g = g_routed + q;
    for (int t = 0; t < kMaxTok; ++t) {
      const int b = qq * p.gcap + t;
      gd.tok[t] = t < gd.n_tok ? b : 0;
      gd.slot[t] = t < gd.n_tok ? p.k + s : 0;
      gd.w[t] = t < gd.n_tok ? 1.f : 0.f;
      if (t < gd.n_tok) p.tok_groups[b * kMaxSlots + p.k + s] = (g << 3) | t;
    }
    p.groups[g] = gd;
  }
  for (int g = tid; g < p.G_max; g += kRouteThreads) p.group_total[g] = 0;
  if (tid == 0) p.ctrl->G = G;
}

template <int EV>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteParams p) {
  __shared__ float s_logits[256];
  __shared__ float s_red[kRouteThreads * 8];
  __shared__ int s_last;
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ float dyn[];
  const bool local = gridDim.x == 1;
  int* s_idx = reinterpret_cast<int*>(dyn);
  float* s_w = reinterpret_cast<float*>(s_idx + 2 * p.B * p.k);
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    router_logits<EV>(p, b, s_logits, s_red);
    if (threadIdx.x < 32) router_topk(p, b, s_logits, local ? s_idx : nullptr, local ? s_w : nullptr);
    __syncthreads();
  }
  if (gridDim.x > 1) {
    // the last CTA to finish groups the pairs of every token.  The barrier orders this
    // CTA's top-k stores before thread 0's count, whose release publishes them and whose
    // acquire (in the last CTA) makes the other CTAs' stores visible to its reads below.
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned old;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(&p.ctrl->route_done) : "memory");
      s_last = old == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
  }
  router_group(p, local);
  if (threadIdx.x == 0) p.ctrl->route_done = 0;
}

// Single expert: groups of up to 8 consecutive tokens, weight 1.
__global__ void expert_prep_kernel(int expert, int n, int gcap, GroupDesc* groups,
                                   int* tok_groups, int* group_total, Ctrl* ctrl) {
  griddep_wait();
  griddep_launch_dependents();
  const int G = (n + gcap - 1) / gcap;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    GroupDesc gd;
    gd.expert = expert;
    gd.n_tok = min(gcap, n - g * gcap);
    for (int t = 0; t < kMaxTok; ++t) {
      const bool on = t < gd.n_tok;
      gd.tok[t] = on ? g * gcap + t : 0;
      gd.slot[t] = 0;
      gd.w[t] = on ? 1.f : 0.f;
      if (on) tok_groups[(g * gcap + t) * kMaxSlots] = (g << 3) | t;
    }
    groups[g] = gd;
    group_total[g] = 0;
  }
  if (threadIdx.x == 0) ctrl->G = G;
}

size_t route_group_smem(int B, int k, int E) {
  return (size_t)3 * B * k * sizeof(int) + (size_t)E * ((B + 31) / 32) * sizeof(uint32_t);
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.B);  // one CTA per token; the last one groups the pairs
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = route_group_smem(p.B, p.k, p.E);
  cfg.stream = st;
  {
    // always: the kernel's static shared memory counts against the default 48 KB too
    cudaError_t e = cudaFuncSetAttribute(
        p.E % 8 == 0 ? (const void*)route_kernel<8> : (const void*)route_kernel<1>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.E % 8 == 0) return cudaLaunchKernelEx(&cfg, route_kernel<8>, p);
  return cudaLaunchKernelEx(&cfg, route_kernel<1>, p);
}

cudaError_t launch_expert_prep(int expert, int n, int gcap, GroupDesc* groups, int* tok_groups,
                               int* group_total, Ctrl* ctrl, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(128);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, expert_prep_kernel, expert, n, gcap, groups, tok_groups,
                            group_total, ctrl);
}

}  // namespace sesg
