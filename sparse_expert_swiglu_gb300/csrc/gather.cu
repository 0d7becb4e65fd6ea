// Steps 3 and 4 of Algorithm 1 "Efficient Sparse Kernel" of "FloE: On-the-Fly MoE
// Inference on Memory-constrained GPU" (sec. 三 "系统协同优化") over the kept columns
// only: x' = SiLU(x W^gate[:, mask]) (.) v[mask] and out = x' W^down[mask, :], with
// W^gate stored as rows gate_t[i] and W^down stored transposed (row i contiguous) so
// that a kept column costs two contiguous d-vectors and masked-out bytes are never
// read; SiLU is fused with the product (the kernel optimisation list of that section).
//
// Each CTA takes an equal share of the kept items of the whole call (in the fixed
// order group, M-tile, column).  One producer thread brings the gate row, the down
// row and the v values of every item into a shared-memory ring with 1-D bulk copies
// (TMA).  The consumer warps form NGRP independent groups; group q handles items
// q, q + NGRP, ...: its threads own interleaved 16-byte chunks of the hidden
// dimension, form the partial dot products x . gate, sum them across the group
// (double-buffered, one named barrier per item), apply SiLU * v * (router weight)
// and accumulate h * down in fp32 registers.  At the end of every expert group the
// NGRP accumulators are added in a fixed order and written as this CTA's partial
// output; the combine kernel adds the partials.
#include "params.cuh"

namespace sesg {

constexpr int kChunk = 8;  // fp16 elements per 16-byte chunk

struct GatherLayout {
  size_t off_full, off_empty, off_stage, off_lslot, off_lcol, off_lgrp, off_red, off_accred, off_tmp,
      off_goff, total, stage_bytes;
};

__host__ __device__ inline int gather_ngrp(int d, int nt) {
  const int ncw = d / 256;
  const int maxg = nt == 1 ? 4 : nt == 2 ? 2 : 1;
  for (int g = maxg; g > 1; g >>= 1)
    if (ncw % g == 0) return g;
  return 1;
}

__host__ __device__ inline GatherLayout gather_layout(int d, int stages, int nt, int list_cap,
                                                      int g_max) {
  GatherLayout L;
  const int ncw = d / 256, ngrp = gather_ngrp(d, nt);
  size_t o = 0;
  L.off_full = o;
  o += 8 * (size_t)stages;
  L.off_empty = o;
  o += 8 * (size_t)stages;
  o = (o + 127) & ~(size_t)127;
  L.stage_bytes = (size_t)4 * d + 32;
  L.off_stage = o;
  o += L.stage_bytes * stages;
  L.off_lslot = o;
  o += (size_t)list_cap * 4;
  L.off_lcol = o;
  o += (size_t)list_cap * 4;
  L.off_lgrp = o;
  o += (size_t)list_cap * 4;
  L.off_red = o;  // [ngrp][2][warps per group][kMaxTok]
  o += (size_t)2 * ncw * kMaxTok * 4;
  o = (o + 15) & ~(size_t)15;
  L.off_accred = o;  // cross-group reduction buffer [nt][d]
  o += ngrp > 1 ? (size_t)nt * d * 4 : 0;
  L.off_tmp = o;  // block-scan scratch
  o += (size_t)1040 * 4;
  L.off_goff = o;  // kept-item offsets of the groups [G_max + 1]
  o += ((size_t)g_max + 1) * 4;
  L.total = o;
  return L;
}

// In-place exclusive prefix sum of data[0..n) (data[n] = total), all threads of the
// block; tmp holds blockDim.x + 1 ints.
__device__ void block_exclusive_scan(int* data, int n, int* tmp) {
  const int nthr = blockDim.x, t = threadIdx.x;
  const int per = (n + nthr - 1) / nthr;
  const int lo = min(n, t * per), hi = min(n, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += data[i];
  tmp[t] = s;
  __syncthreads();
  if (t < 32) {
    int carry = 0;
    for (int b = 0; b < nthr; b += 32) {
      const int i = b + t;
      const int v = i < nthr ? tmp[i] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (t >= off) incl += o;
      }
      if (i < nthr) tmp[i] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (t == 0) tmp[nthr] = carry;
  }
  __syncthreads();
  int run = tmp[t];
  for (int i = lo; i < hi; ++i) {
    const int v = data[i];
    data[i] = run;
    run += v;
  }
  if (t == 0) data[n] = tmp[nthr];
  __syncthreads();
}

template <int NT, int NGRP, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) gather_kernel(ExpertParams p) {
  extern __shared__ __align__(128) uint8_t gsm[];
  const int d = p.d;
  const int ncw = d / 256;          // consumer warps
  const int nct = ncw * 32;         // consumer threads
  constexpr int ngrp = NGRP;
  const int wg = ncw / ngrp;        // warps per consumer group
  const int tpg = wg * 32;          // threads per consumer group
  const int S = p.stages;
  const GatherLayout L = gather_layout(d, S, NT, p.list_cap, p.G_max);
  uint64_t* full = reinterpret_cast<uint64_t*>(gsm + L.off_full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(gsm + L.off_empty);
  uint8_t* stage = gsm + L.off_stage;
  int* lslot = reinterpret_cast<int*>(gsm + L.off_lslot);
  int* lcol = reinterpret_cast<int*>(gsm + L.off_lcol);
  int* lgrp = reinterpret_cast<int*>(gsm + L.off_lgrp);
  float* red = reinterpret_cast<float*>(gsm + L.off_red);
  float* accred = reinterpret_cast<float*>(gsm + L.off_accred);
  int* tmp = reinterpret_cast<int*>(gsm + L.off_tmp);
  __shared__ int s_abort, s_issued, s_consumed;
  __shared__ GroupDesc s_gd;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == ncw;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], wg);
    }
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
  }
  griddep_wait();
  griddep_launch_dependents();

  // ---- prologue: this CTA's range of the global kept-item order (group, M-tile, column)
  const int G = *reinterpret_cast<volatile int*>(&p.ctrl->G);
  const int MT = p.f / kMTile;
  int* goff = reinterpret_cast<int*>(gsm + L.off_goff);  // [G+1]
  int* uoff = reinterpret_cast<int*>(stage);  // scratch in the idle stage ring: [MT+1]
  for (int g = tid; g < G; g += blockDim.x) goff[g] = __ldcg(p.group_total + g);
  __syncthreads();
  block_exclusive_scan(goff, G, tmp);
  const long long N = goff[G];
  if (blockIdx.x == 0 && tid == 0) p.ctrl->N = (int)N;
  const int a = (int)(N * blockIdx.x / p.P3), b = (int)(N * (blockIdx.x + 1) / p.P3);

  // consumer-group geometry
  const int q = producer ? 0 : warp / wg;        // consumer group
  const int tg = producer ? 0 : tid - q * tpg;   // thread within the group
  const int wig = tg >> 5;                       // warp within the group
  float acc[NT][kChunk * NGRP];
  uint4 xr[NT][NGRP];
  float wt[NT];

  for (int wa = a; wa < b; wa += p.list_cap) {
    const int wb = min(b, wa + p.list_cap);
    int g = 0;
    {
      int lo = 0, hi = G - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (goff[mid + 1] > wa) hi = mid;
        else lo = mid + 1;
      }
      g = lo;
    }
    for (; g < G && goff[g] < wb; ++g) {
      if (goff[g + 1] == goff[g]) continue;
      const uint8_t* cnt = p.unit_cnt + (size_t)g * MT;
      for (int i = tid; i < MT; i += blockDim.x) uoff[i] = __ldcg(cnt + i);
      __syncthreads();
      block_exclusive_scan(uoff, MT, tmp);
      const int gbase = goff[g];
      for (int m = tid; m < MT; m += blockDim.x) {
        const int s0 = gbase + uoff[m], s1 = gbase + uoff[m + 1];
        for (int i = max(s0, wa); i < min(s1, wb); ++i) {
          lslot[i - wa] = ((g * MT) + m) * 16 + (i - s0);
          lgrp[i - wa] = g;
        }
      }
      __syncthreads();
    }
    const int n = wb - wa;
    const int base = wa - a;  // items issued / consumed by this CTA before this window
    for (int i = tid; i < n; i += blockDim.x) lcol[i] = __ldcg(p.item_col + lslot[i]);
    fence_proxy_async_smem();  // order the prologue's generic writes to the ring before TMA reuses it
    __syncthreads();

    if (producer) {
      // two producer lanes (even / odd items): two bulk-copy transactions in flight per SM
      if (lane < 2) {
        const uint64_t pol = policy_evict_first();
        int last_g = -1;
        const __half* gbase_ptr = nullptr;
        const __half* dbase_ptr = nullptr;
        int row_stride = d;
        for (int i = lane; i < n; i += 2) {
          const int gidx = base + i;
          const int s = gidx % S;
          if (gidx >= S && !mbar_wait(&empty[s], ((gidx / S) - 1) & 1)) {
            set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
            break;
          }
          if (*reinterpret_cast<volatile int*>(&s_abort)) break;
          const int gi = lgrp[i];
          if (gi != last_g) {
            last_g = gi;
            int el;
            const ExpertSet& es = expert_set(p, p.groups[gi].expert, el);
            gbase_ptr = es.gate_t + (size_t)el * es.f * es.rs;
            dbase_ptr = es.down + (size_t)el * es.f * es.rs;
            row_stride = es.rs;
          }
          const size_t roff = (size_t)lcol[i] * row_stride;
          uint8_t* st = stage + (size_t)s * L.stage_bytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(4 * d + 32));
          bulk_g2s(st, gbase_ptr + roff, (uint32_t)(2 * d), &full[s], pol);
          bulk_g2s(st + 2 * d, dbase_ptr + roff, (uint32_t)(2 * d), &full[s], pol);
          bulk_g2s(st + 4 * d, p.item_v + (size_t)lslot[i] * 8, 32u, &full[s], pol);
          atomicMax(&s_issued, gidx + 1);
        }
      }
    } else {
      // ---- consumers: segments of equal group, items of a segment dealt round-robin
      int i = 0;
      int local = 0;  // items this consumer group has processed (red buffer parity)
      while (i < n) {
        const int g = lgrp[i];
        int e = i;
        while (e < n && lgrp[e] == g) ++e;
        // segment start: the group's tokens, weights, x chunks
        named_barrier(1, nct);
        if (tid == 0) s_gd = p.groups[g];
        named_barrier(1, nct);
        const int ntok = s_gd.n_tok;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          wt[t] = t < ntok ? s_gd.w[t] : 0.f;
#pragma unroll
          for (int k = 0; k < NGRP; ++k) {
            xr[t][k] = make_uint4(0, 0, 0, 0);
            if (t < ntok)
              xr[t][k] = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)s_gd.tok[t] * d) + tg + k * tpg);
          }
#pragma unroll
          for (int e2 = 0; e2 < kChunk * NGRP; ++e2) acc[t][e2] = 0.f;
        }
        for (int ii = i + q; ii < e; ii += ngrp) {
          const int gidx = base + ii;
          const int s = gidx % S;
          const bool ok = mbar_wait(&full[s], (gidx / S) & 1);
          const uint8_t* st = stage + (size_t)s * L.stage_bytes;
          // x . gate over this thread's chunks, summed over the warp
          float dot[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) dot[t] = 0.f;
#pragma unroll
          for (int k = 0; k < NGRP; ++k) {
            {
              uint4 gr = make_uint4(0, 0, 0, 0);
              if (ok) gr = reinterpret_cast<const uint4*>(st)[tg + k * tpg];
              const __half2* gh = reinterpret_cast<const __half2*>(&gr);
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                if (t < ntok) {
                  const __half2* xh = reinterpret_cast<const __half2*>(&xr[t][k]);
#pragma unroll
                  for (int e2 = 0; e2 < 4; ++e2) {
                    const float2 gf = __half22float2(gh[e2]);
                    const float2 xf = __half22float2(xh[e2]);
                    dot[t] = fmaf(xf.x, gf.x, dot[t]);
                    dot[t] = fmaf(xf.y, gf.y, dot[t]);
                  }
                }
              }
            }
          }
          float* rb = red + ((size_t)(q * 2 + (local & 1)) * wg) * kMaxTok;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t < ntok) {
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) dot[t] += __shfl_xor_sync(0xffffffffu, dot[t], off);
              if (lane == 0) rb[wig * kMaxTok + t] = dot[t];
            }
          }
          // one barrier per item within the group; any failed wait ends the group
          int fail;
          asm volatile(
              "{\n\t.reg .pred pin, pout;\n\t"
              "setp.ne.u32 pin, %1, 0;\n\t"
              "barrier.red.or.pred pout, %2, %3, pin;\n\t"
              "selp.u32 %0, 1, 0, pout;\n\t}"
              : "=r"(fail)
              : "r"((unsigned)(!ok)), "r"(2 + q), "r"(tpg)
              : "memory");
          if (fail) {
            if (tg == 0) {
              set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
              atomicExch(&s_abort, 1);
            }
            break;
          }
          const float* hv = reinterpret_cast<const float*>(st + 4 * d);
          float h[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            h[t] = 0.f;
            if (t < ntok) {
              float gsum = 0.f;
              for (int w = 0; w < wg; ++w) gsum += rb[w * kMaxTok + t];
              h[t] = silu_f(gsum) * hv[t] * wt[t];
            }
          }
          // down rows: acc += h * down[kept row]
#pragma unroll
          for (int k = 0; k < NGRP; ++k) {
            {
              const uint4 dr = reinterpret_cast<const uint4*>(st + 2 * d)[tg + k * tpg];
              const __half2* dh = reinterpret_cast<const __half2*>(&dr);
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const float2 df = __half22float2(dh[e2]);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                  acc[t][k * kChunk + 2 * e2] = fmaf(h[t], df.x, acc[t][k * kChunk + 2 * e2]);
                  acc[t][k * kChunk + 2 * e2 + 1] = fmaf(h[t], df.y, acc[t][k * kChunk + 2 * e2 + 1]);
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          ++local;
        }
        // segment end: add the groups' accumulators in a fixed order, write the partial
        named_barrier(1, nct);
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        float* dst = p.part + ((size_t)(blockIdx.x + g) * kMaxTok) * d;
        for (int r = 0; r < ngrp; ++r) {
          if (q == r) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (t < ntok) {
#pragma unroll
                for (int k = 0; k < NGRP; ++k) {
                  {
                    const int c = tg + k * tpg;
                    float4* ar = reinterpret_cast<float4*>(accred + (size_t)t * d + c * kChunk);
                    float4 v0 = make_float4(acc[t][k * 8 + 0], acc[t][k * 8 + 1], acc[t][k * 8 + 2], acc[t][k * 8 + 3]);
                    float4 v1 = make_float4(acc[t][k * 8 + 4], acc[t][k * 8 + 5], acc[t][k * 8 + 6], acc[t][k * 8 + 7]);
                    if (r > 0) {
                      const float4 p0 = ar[0], p1 = ar[1];
                      v0 = make_float4(p0.x + v0.x, p0.y + v0.y, p0.z + v0.z, p0.w + v0.w);
                      v1 = make_float4(p1.x + v1.x, p1.y + v1.y, p1.z + v1.z, p1.w + v1.w);
                    }
                    if (r + 1 < ngrp) {
                      ar[0] = v0;
                      ar[1] = v1;
                    } else {
                      float4* o = reinterpret_cast<float4*>(dst + (size_t)t * d + c * kChunk);
                      o[0] = v0;
                      o[1] = v1;
                    }
                  }
                }
              }
            }
          }
          if (ngrp > 1) named_barrier(1, nct);
        }
        if (tid == 0) s_consumed = base + e;
        i = e;
      }
    }
    __syncthreads();
    if (s_abort) break;
  }
  // on an abort, wait (bounded) for copies still in flight before the CTA exits
  if (s_abort && tid == 0)
    for (int i = max(s_consumed, s_issued - S); i < s_issued; ++i)
      (void)mbar_wait(&full[i % S], (i / S) & 1);
}

size_t gather_smem_bytes(int d, int stages, int nt, int list_cap, int g_max) {
  return gather_layout(d, stages, nt, list_cap, g_max).total;
}

cudaError_t launch_gather(const ExpertParams& p, int nt, cudaStream_t st, bool pdl) {
  const int ncw = p.d / 256;
  const size_t smem = gather_smem_bytes(p.d, p.stages, nt, p.list_cap, p.G_max);
  const int ngrp = gather_ngrp(p.d, nt);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.P3);
  cfg.blockDim = dim3((ncw + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
#define SESG_G(NTV, NG, MT)                                                                        \
  if ((ncw + 1) * 32 > MT) return cudaErrorInvalidConfiguration;                                  \
  e = cudaFuncSetAttribute(gather_kernel<NTV, NG, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                             \
  if (e != cudaSuccess) return e;                                                                  \
  return cudaLaunchKernelEx(&cfg, gather_kernel<NTV, NG, MT>, p);
  const bool small = (ncw + 1) * 32 <= 544;  // d <= 4096: more registers per thread
  if (nt == 1 && ngrp == 4) { if (small) { SESG_G(1, 4, 544) } SESG_G(1, 4, 1024) }
  if (nt == 1 && ngrp == 2) { if (small) { SESG_G(1, 2, 544) } SESG_G(1, 2, 1024) }
  if (nt == 1) { if (small) { SESG_G(1, 1, 544) } SESG_G(1, 1, 1024) }
  if (nt == 2 && ngrp == 2) { if (small) { SESG_G(2, 2, 544) } SESG_G(2, 2, 1024) }
  if (nt == 2) { if (small) { SESG_G(2, 1, 544) } SESG_G(2, 1, 1024) }
  if (nt == 4) { if (small) { SESG_G(4, 1, 544) } SESG_G(4, 1, 800) }
  SESG_G(8, 1, 544)
#undef SESG_G
}

}  // namespace sesg
