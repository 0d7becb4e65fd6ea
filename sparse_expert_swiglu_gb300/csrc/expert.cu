// Sparse SwiGLU experts: Algorithm 1 "Efficient Sparse Kernel" of "FloE: On-the-Fly
// MoE Inference on Memory-constrained GPU" (sec. 三 "系统协同优化"), as three kernels:
//
//   up_kernel      step 1 (v = x W^up from the INT2 codes) and step 2 (mask = |v| > t),
//                  with the kept columns compacted into an item list
//   gather_kernel  steps 3 and 4 over kept columns only: the gate row and the down
//                  row of every kept column are brought into shared memory by 1-D
//                  bulk copies (TMA), SiLU(x . gate) * v is fused with the product,
//                  and the down rows are accumulated in fp32
//   combine_kernel the deterministic sum of the per-CTA partial outputs, the fp16
//                  rounding and (for stacked layers) the RMSNorm
//
// The work unit is a "group": one expert and up to 8 of the tokens routed to it, so
// each expert's weights are read once for all of its tokens.
#include "params.cuh"

namespace sesg {


__device__ __forceinline__ const ExpertSet& expert_set(const ExpertParams& p, int expert,
                                                       int& local) {
  if (expert < p.routed.E) {
    local = expert;
    return p.routed;
  }
  local = expert - p.routed.E;
  return p.shared;
}

// ===========================================================================
// up_kernel
// ===========================================================================
constexpr int kUpWarps = 8;
constexpr int kUpThreads = kUpWarps * 32;

template <int GI>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t wsh) {
  // Two 2-bit codes of group slot GI as an fp16x2 of subnormals q * 4^pos * 2^-24
  // (exact); the power of two is removed after the mma.
  if constexpr (GI < 5) return w & (0x00030003u << (2 * GI));
  else return wsh & (0x00030003u << (2 * (GI - 5)));
}

__device__ __forceinline__ float pos_scale(int gi) {
  const int pos = gi < 5 ? gi : gi - 5;
  return __int_as_float((127 + 24 - 2 * pos) << 23);  // 2^(24 - 2 pos)
}

// One warp, one (group, M-tile): v for 16 columns and the group's tokens.
//
// Tensor-core mapping (mma.sync m16n8k16, f16 in, f32 accumulate): M = 16 output
// columns, K = 16 inputs, N = 8 slots.  A slot is a (token, group class) pair:
// with T tokens (padded to a power of two) there are G = 8/T classes, and a
// k-step of quantiser group gi only feeds the slots of class gi % G, whose B
// column carries that token's x; the other B columns are zero.  So one
// accumulator tile collects G quantiser groups side by side, and the per-group
// scale/zero correction  v += s * (A_g - z * X_g)  (X_g = sum of x over the
// group) is applied once per G groups instead of once per group.
template <int T>
__device__ void up_unit(const ExpertParams& p, const GroupDesc& gd, long long u, int mt,
                        const uint4* __restrict__ bfrag, const float* __restrict__ xg,
                        float* __restrict__ vbuf) {
  constexpr int G = 8 / T;
  const int lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
  const int d = p.d, nsb = n_superblocks(d), ngrp = d / kGroup;
  int el;
  const ExpertSet& es = expert_set(p, gd.expert, el);
  const uint8_t* strip = es.up + (size_t)el * es.up_stride + (size_t)mt * nsb * kBlkBytes;

  // (scale, zero) table entries this lane needs per phase: slots 2c, 2c+1
  const int gi_lane = (G >= 2) ? (2 * c) % G : 0;
  using SZ = typename std::conditional<G >= 2, uint2, uint32_t>::type;

  float vacc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  uint4 cw[4];
  SZ sz[T][2];
  auto load_sb = [&](int sb, uint4 (&cwo)[4], SZ (&szo)[T][2]) {
    const uint8_t* blk = strip + (size_t)sb * kBlkBytes;
#pragma unroll
    for (int q = 0; q < 4; ++q) cwo[q] = ld_stream_v4(blk + (q * 32 + lane) * 16);
#pragma unroll
    for (int ph = 0; ph < T; ++ph)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = gl + 8 * r;
        const int gi0 = (G >= 2) ? ph * G + gi_lane : ph;
        const uint8_t* a = blk + kBlkCodeBytes + (row * 8 + gi0) * 4;
        if constexpr (G >= 2) szo[ph][r] = ld_nc_v2(a);
        else szo[ph][r] = ld_nc_u32(a);
      }
  };
  load_sb(0, cw, sz);

  for (int sb = 0; sb < nsb; ++sb) {
    uint4 w[4];
    SZ szc[T][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = cw[q];
#pragma unroll
    for (int ph = 0; ph < T; ++ph)
#pragma unroll
      for (int r = 0; r < 2; ++r) szc[ph][r] = sz[ph][r];
    if (sb + 1 < nsb) load_sb(sb + 1, cw, sz);

    const int ng = min(8, (d - sb * kSuper) / kGroup);
    uint4 wsh[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      wsh[q] = make_uint4(w[q].x >> 10, w[q].y >> 10, w[q].z >> 10, w[q].w >> 10);
    const uint4* bf = bfrag + (size_t)(sb * 16) * 32 + lane;

#pragma unroll
    for (int ph = 0; ph < T; ++ph) {
      float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int gam = 0; gam < G; ++gam) {
        const int gi = ph * G + gam;
        if (gi < ng) {
          const uint4 b01 = bf[(gi * 2 + 0) * 32];
          const uint4 b23 = bf[(gi * 2 + 1) * 32];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint4 wt = w[t], st = wsh[t];
            uint32_t a[4];
            // gi is a compile-time constant after unrolling
#define SESG_CASE(GIV)                      \
  case GIV:                                 \
    a[0] = code_pair<GIV>(wt.x, st.x);      \
    a[1] = code_pair<GIV>(wt.y, st.y);      \
    a[2] = code_pair<GIV>(wt.z, st.z);      \
    a[3] = code_pair<GIV>(wt.w, st.w);      \
    break;
            switch (gi) {
              SESG_CASE(0) SESG_CASE(1) SESG_CASE(2) SESG_CASE(3)
              SESG_CASE(4) SESG_CASE(5) SESG_CASE(6) default: SESG_CASE(7)
            }
#undef SESG_CASE
            const uint4 bb = (t < 2) ? b01 : b23;
            if (t & 1) mma_16816(D, a, bb.z, bb.w);
            else mma_16816(D, a, bb.x, bb.y);
          }
        }
      }
      // fold this phase's G groups into v
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int gi = (G >= 2) ? ph * G + gi_lane + s : ph;
        const int tau = (G >= 2) ? (2 * c) / G : 2 * c + s;
        if (gi < ng) {
          const float cs = pos_scale(gi);
          const float X = xg[tau * ngrp + sb * 8 + gi];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            float sf, zf;
            if constexpr (G >= 2) {
              const uint32_t pr = s ? szc[ph][r].y : szc[ph][r].x;
              const __half2 h = *reinterpret_cast<const __half2*>(&pr);
              sf = __low2float(h);
              zf = __high2float(h);
            } else {
              const __half2 h = *reinterpret_cast<const __half2*>(&szc[ph][r]);
              sf = __low2float(h);
              zf = __high2float(h);
            }
            const float tval = fmaf(-zf, X, D[2 * r + s] * cs);
            vacc[r][s] = fmaf(sf, tval, vacc[r][s]);
          }
        }
      }
    }
  }

  // per-token v of rows gl and gl+8 -> vbuf[16][8]
  if constexpr (G >= 2) {
    float v0 = vacc[0][0] + vacc[0][1];
    float v1 = vacc[1][0] + vacc[1][1];
    if constexpr (G >= 4) {
      v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
    }
    if constexpr (G == 8) {
      v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
      v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
    }
    const int tau = (2 * c) / G;
    if ((c % (G / 2)) == 0) {
      vbuf[gl * 8 + tau] = v0;
      vbuf[(gl + 8) * 8 + tau] = v1;
    }
  } else {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      vbuf[gl * 8 + 2 * c + s] = vacc[0][s];
      vbuf[(gl + 8) * 8 + 2 * c + s] = vacc[1][s];
    }
  }
  __syncwarp();

  // step 2: mask = |v| > t; union over the group's tokens; compaction by ballot
  const float thr = es.thr[el];
  float vv[kMaxTok];
  uint32_t mbits = 0;
#pragma unroll
  for (int t = 0; t < kMaxTok; ++t) {
    vv[t] = 0.f;
    if (t < gd.n_tok && lane < 16) {
      vv[t] = vbuf[lane * 8 + t];
      if (fabsf(vv[t]) > thr) mbits |= 1u << t;
    }
  }
  const bool kept = mbits != 0;
  const uint32_t bal = __ballot_sync(0xffffffffu, kept);
  if (kept) {
    const int rank = __popc(bal & ((1u << lane) - 1u));
    const long long slot = u * 16 + rank;
    p.item_col[slot] = mt * kMTile + lane;
    float hv[kMaxTok];
#pragma unroll
    for (int t = 0; t < kMaxTok; ++t) hv[t] = ((mbits >> t) & 1u) ? vv[t] : 0.f;
    float4* dst = reinterpret_cast<float4*>(p.item_v + slot * 8);
    dst[0] = make_float4(hv[0], hv[1], hv[2], hv[3]);
    dst[1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
  }
  if (lane == 0) {
    p.unit_cnt[u] = (uint8_t)__popc(bal);
    const int g = (int)(u / (p.f / kMTile));
    if (bal) atomicAdd(&p.group_total[g], __popc(bal));
  }
  if (p.dbg_v || p.dbg_mask) {
#pragma unroll
    for (int t = 0; t < kMaxTok; ++t) {
      if (t < gd.n_tok) {
        const size_t row = (size_t)gd.tok[t] * p.n_slots + gd.slot[t];
        if (p.dbg_v && lane < 16) p.dbg_v[row * p.f + mt * kMTile + lane] = vv[t];
        const uint32_t mb = __ballot_sync(0xffffffffu, (mbits >> t) & 1u) & 0xffffu;
        if (p.dbg_mask && lane == 0)
          reinterpret_cast<uint16_t*>(p.dbg_mask)[row * (size_t)(2 * ((p.f + 31) / 32)) + mt] =
              (uint16_t)mb;
      }
    }
  }
  __syncwarp();
}

// B fragments of the current group (zero where a slot's class does not match the
// k-step's group) and the per-group sums X_g of every token.
__device__ void build_bfrag(const ExpertParams& p, const GroupDesc& gd, int T, uint4* bfrag,
                            float* xg) {
  const int d = p.d, G = 8 / T;
  for (int idx = threadIdx.x; idx < d; idx += blockDim.x) {  // d/32 k-step pairs x 32 lanes
    const int ks2 = idx >> 5, lane = idx & 31, gl = lane >> 2, c = lane & 3;
    uint32_t r[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ks = 2 * ks2 + h;
      const int gi = (ks & 31) >> 2;
      uint32_t b0 = 0, b1 = 0;
      const int tau = gl / G;
      if ((gl % G) == (gi % G) && tau < gd.n_tok) {
        const __half* xr = p.x + (size_t)gd.tok[tau] * d + 16 * ks + 2 * c;
        b0 = *reinterpret_cast<const uint32_t*>(xr);
        b1 = *reinterpret_cast<const uint32_t*>(xr + 8);
      }
      r[2 * h] = b0;
      r[2 * h + 1] = b1;
    }
    bfrag[idx] = make_uint4(r[0], r[1], r[2], r[3]);
  }
  const int ngrp = d / kGroup;
  for (int idx = threadIdx.x; idx < kMaxTok * ngrp; idx += blockDim.x) {
    const int tau = idx / ngrp, grp = idx % ngrp;
    float s = 0.f;
    if (tau < gd.n_tok) {
      const __half2* xr = reinterpret_cast<const __half2*>(p.x + (size_t)gd.tok[tau] * d + grp * kGroup);
      for (int r = 0; r < kGroup / 2; ++r) {
        const float2 v = __half22float2(xr[r]);
        s += v.x;
        s += v.y;
      }
    }
    xg[idx] = s;
  }
}

__global__ void __launch_bounds__(kUpThreads, 2) up_kernel(ExpertParams p) {
  extern __shared__ __align__(16) uint8_t up_smem[];
  uint4* bfrag = reinterpret_cast<uint4*>(up_smem);                 // [d/32][32]
  float* xg = reinterpret_cast<float*>(bfrag + p.d);                // [8][d/64]
  float* vbuf = xg + kMaxTok * (p.d / kGroup);                      // [8 warps][16][8]
  __shared__ GroupDesc s_gd;
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int G = *reinterpret_cast<volatile int*>(&p.ctrl->G);
  const int MT = p.f / kMTile;
  const long long U = (long long)G * MT;
  const long long u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  for (long long ub = u0; ub < u1;) {
    const int g = (int)(ub / MT);
    const long long ue = min(u1, (long long)(g + 1) * MT);
    __syncthreads();
    if (threadIdx.x == 0) s_gd = p.groups[g];
    __syncthreads();
    const int n = s_gd.n_tok;
    const int T = n <= 1 ? 1 : n <= 2 ? 2 : n <= 4 ? 4 : 8;
    build_bfrag(p, s_gd, T, bfrag, xg);
    __syncthreads();
    float* vb = vbuf + warp * 16 * 8;
    for (long long u = ub + warp; u < ue; u += kUpWarps) {
      const int mt = (int)(u - (long long)g * MT);
      switch (T) {
        case 1: up_unit<1>(p, s_gd, u, mt, bfrag, xg, vb); break;
        case 2: up_unit<2>(p, s_gd, u, mt, bfrag, xg, vb); break;
        case 4: up_unit<4>(p, s_gd, u, mt, bfrag, xg, vb); break;
        default: up_unit<8>(p, s_gd, u, mt, bfrag, xg, vb); break;
      }
    }
    ub = ue;
  }
}

size_t up_smem_bytes(int d) {
  return (size_t)d * 16 + (size_t)kMaxTok * (d / kGroup) * 4 + (size_t)kUpWarps * 16 * 8 * 4;
}

// ===========================================================================
// gather_kernel
// ===========================================================================
constexpr int kEPT = 8;   // hidden elements per consumer thread (one 16-byte chunk of a row)
constexpr int kBatch = 4; // kept columns per reduction round

struct GatherSmem {
  // carved out of dynamic shared memory by offsets computed on both sides
  size_t off_full, off_empty, off_stage, off_x, off_lslot, off_lcol, off_lgrp, off_red, off_h,
      total;
  size_t stage_bytes;
};

__host__ __device__ inline GatherSmem gather_layout(int d, int stages, int ncw, int nt,
                                                    int list_cap) {
  GatherSmem L;
  size_t o = 0;
  L.off_full = o;
  o += 8 * (size_t)stages;
  L.off_empty = o;
  o += 8 * (size_t)stages;
  o = (o + 127) & ~(size_t)127;
  L.stage_bytes = (size_t)4 * d + 32;
  L.off_stage = o;
  o += L.stage_bytes * stages;
  L.off_x = o;
  o += (size_t)nt * d * 2;
  L.off_lslot = o;
  o += (size_t)list_cap * 4;
  L.off_lcol = o;
  o += (size_t)list_cap * 4;
  L.off_lgrp = o;
  o += (size_t)list_cap * 4;
  L.off_red = o;
  o += (size_t)ncw * kBatch * kMaxTok * 4;
  L.off_h = o;
  o += (size_t)kBatch * kMaxTok * 4;
  L.total = o;
  return L;
}

// Exclusive prefix of the kept-item totals of groups: out[0..G] (warp 0).
__device__ void warp_exclusive_scan(const int* in, int* out, int n) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    int v = i < n ? in[i] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (i < n) out[i] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) out[n] = carry;
}

template <int NT, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) gather_kernel(ExpertParams p) {
  constexpr int KB = (NT >= 4) ? 2 : kBatch;  // kept columns per reduction round
  extern __shared__ __align__(128) uint8_t gsm[];
  const int d = p.d;
  const int ncw = d / (32 * kEPT);                 // consumer warps
  const int nct = ncw * 32;                        // consumer threads
  const int S = p.stages;
  const GatherSmem L = gather_layout(d, S, ncw, NT, p.list_cap);
  uint64_t* full = reinterpret_cast<uint64_t*>(gsm + L.off_full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(gsm + L.off_empty);
  uint8_t* stage = gsm + L.off_stage;
  __half* xs = reinterpret_cast<__half*>(gsm + L.off_x);
  int* lslot = reinterpret_cast<int*>(gsm + L.off_lslot);
  int* lcol = reinterpret_cast<int*>(gsm + L.off_lcol);
  int* lgrp = reinterpret_cast<int*>(gsm + L.off_lgrp);
  float* red = reinterpret_cast<float*>(gsm + L.off_red);
  float* hsm = reinterpret_cast<float*>(gsm + L.off_h);
  __shared__ int s_abort, s_issued, s_consumed;
  __shared__ GroupDesc s_gd;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == ncw;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ncw);
    }
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
  }
  griddep_wait();
  griddep_launch_dependents();

  // ---- prologue: my range of the global kept-item order (group, M-tile, column)
  const int G = *reinterpret_cast<volatile int*>(&p.ctrl->G);
  const int MT = p.f / kMTile;
  int* scan = reinterpret_cast<int*>(stage);       // scratch: [G+1] group offsets, then [MT+1]
  int* goff = scan;
  int* uoff = scan + G + 1;
  int* gtot = uoff + MT + 1;                       // [G] copy of the group totals
  for (int g = tid; g < G; g += blockDim.x) gtot[g] = __ldcg(p.group_total + g);
  __syncthreads();
  if (warp == 0) warp_exclusive_scan(gtot, goff, G);
  __syncthreads();
  const long long N = goff[G];
  if (blockIdx.x == 0 && tid == 0) p.ctrl->N = (int)N;
  const int a = (int)(N * blockIdx.x / p.P3), b = (int)(N * (blockIdx.x + 1) / p.P3);

  float acc[NT][kEPT];
  int cur_g = -1;
  for (int wa = a; wa < b; wa += p.list_cap) {
    const int wb = min(b, wa + p.list_cap);
    // groups overlapping [wa, wb): fill the list
    int g = 0;
    {
      // first group with goff[g+1] > wa
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
      __syncthreads();
      // exclusive scan of the group's per-M-tile counts (uint8) into uoff
      {
        const uint8_t* cnt = p.unit_cnt + (size_t)g * MT;
        for (int i = tid; i < MT; i += blockDim.x) uoff[i] = __ldcg(cnt + i);
        __syncthreads();
        if (warp == 0) {
          // in place: use gtot region after it as temporary
          int carry = 0;
          for (int base = 0; base < MT; base += 32) {
            const int i = base + lane;
            const int v = i < MT ? uoff[i] : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
              const int o = __shfl_up_sync(0xffffffffu, incl, off);
              if (lane >= off) incl += o;
            }
            __syncwarp();
            if (i < MT) uoff[i] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
          }
          if (lane == 0) uoff[MT] = carry;
        }
        __syncthreads();
      }
      const int gbase = goff[g];
      for (int m = tid; m < MT; m += blockDim.x) {
        const int s0 = gbase + uoff[m], s1 = gbase + uoff[m + 1];
        for (int i = max(s0, wa); i < min(s1, wb); ++i) {
          const int slot = ((g * MT) + m) * 16 + (i - s0);
          lslot[i - wa] = slot;
          lcol[i - wa] = __ldcg(p.item_col + slot);
          lgrp[i - wa] = g;
        }
      }
    }
    __syncthreads();
    const int n = wb - wa;
    const int base = wa - a;  // items issued / consumed by this CTA before this window

    if (producer) {
      if (lane == 0) {
        const uint64_t pol = policy_evict_first();
        int last_g = -1;
        const __half* gbase_ptr = nullptr;
        const __half* dbase_ptr = nullptr;
        int issued = 0;
        for (int i = 0; i < n; ++i) {
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
            gbase_ptr = es.gate_t + (size_t)el * es.f * d;
            dbase_ptr = es.down + (size_t)el * es.f * d;
          }
          const size_t roff = (size_t)lcol[i] * d;
          uint8_t* st = stage + (size_t)s * L.stage_bytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(4 * d + 32));
          bulk_g2s(st, gbase_ptr + roff, (uint32_t)(2 * d), &full[s], pol);
          bulk_g2s(st + 2 * d, dbase_ptr + roff, (uint32_t)(2 * d), &full[s], pol);
          bulk_g2s(st + 4 * d, p.item_v + (size_t)lslot[i] * 8, 32u, &full[s], pol);
          ++issued;
        }
        s_issued = base + issued;
      }
    } else {
      // ---- consumers
      const int tc = tid;  // 0..nct-1, owns hidden elements [tc*8, tc*8+8)
      for (int i0 = 0; i0 < n;) {
        const int g = lgrp[i0];
        int nb = 1;
        while (nb < KB && i0 + nb < n && lgrp[i0 + nb] == g) ++nb;
        if (g != cur_g) {
          if (cur_g >= 0) {
            float* dst = p.part + ((size_t)(blockIdx.x + cur_g) * kMaxTok) * d + tc * kEPT;
#pragma unroll
            for (int t = 0; t < NT; ++t)
              if (t < s_gd.n_tok) {
                float4* o = reinterpret_cast<float4*>(dst + (size_t)t * d);
                o[0] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
                o[1] = make_float4(acc[t][4], acc[t][5], acc[t][6], acc[t][7]);
              }
          }
          named_barrier(1, nct);
          if (tc == 0) s_gd = p.groups[g];
          named_barrier(1, nct);
          for (int idx = tc; idx < s_gd.n_tok * d / 8; idx += nct) {
            const int t = idx / (d / 8), o = idx % (d / 8);
            reinterpret_cast<uint4*>(xs + (size_t)t * d)[o] =
                reinterpret_cast<const uint4*>(p.x + (size_t)s_gd.tok[t] * d)[o];
          }
          named_barrier(1, nct);
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < kEPT; ++e) acc[t][e] = 0.f;
          cur_g = g;
        }
        const int ntok = s_gd.n_tok;
        bool ok = true;
        for (int q = 0; q < nb; ++q) {
          const int i = base + i0 + q;
          ok = ok && mbar_wait(&full[i % S], (i / S) & 1);
        }
        // gate chunks of the batch, then per token: x chunk, dot products, warp sums
        float gf[KB][kEPT];
#pragma unroll
        for (int q = 0; q < KB; ++q) {
          uint4 gr = make_uint4(0, 0, 0, 0);
          if (q < nb && ok)
            gr = reinterpret_cast<const uint4*>(stage + (size_t)((base + i0 + q) % S) * L.stage_bytes)[tc];
          const __half2* h = reinterpret_cast<const __half2*>(&gr);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f2 = __half22float2(h[e]);
            gf[q][2 * e] = f2.x;
            gf[q][2 * e + 1] = f2.y;
          }
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < ntok) {
            const uint4 xr = reinterpret_cast<const uint4*>(xs + (size_t)t * d)[tc];
            const __half2* h = reinterpret_cast<const __half2*>(&xr);
            float xf[kEPT];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f2 = __half22float2(h[e]);
              xf[2 * e] = f2.x;
              xf[2 * e + 1] = f2.y;
            }
#pragma unroll
            for (int q = 0; q < KB; ++q) {
              if (q < nb) {
                float sdot = 0.f;
#pragma unroll
                for (int e = 0; e < kEPT; ++e) sdot = fmaf(xf[e], gf[q][e], sdot);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, off);
                if (lane == 0) red[(warp * kBatch + q) * kMaxTok + t] = sdot;
              }
            }
          }
        }
        // barrier with an OR-reduction of the failures
        int any_fail;
        asm volatile(
            "{\n\t.reg .pred pin, pout;\n\t"
            "setp.ne.u32 pin, %1, 0;\n\t"
            "barrier.red.or.pred pout, 1, %2, pin;\n\t"
            "selp.u32 %0, 1, 0, pout;\n\t}"
            : "=r"(any_fail)
            : "r"((unsigned)(!ok)), "r"(nct)
            : "memory");
        if (any_fail) {
          if (tc == 0) {
            set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          break;
        }
        if (tc < nb * kMaxTok) {
          const int q = tc / kMaxTok, t = tc % kMaxTok;
          float h = 0.f;
          if (t < ntok) {
            float gsum = 0.f;
            for (int w = 0; w < ncw; ++w) gsum += red[(w * kBatch + q) * kMaxTok + t];
            const float* hv = reinterpret_cast<const float*>(
                stage + (size_t)((base + i0 + q) % S) * L.stage_bytes + 4 * d);
            h = silu_f(gsum) * hv[t] * s_gd.w[t];
          }
          hsm[q * kMaxTok + t] = h;
        }
        named_barrier(1, nct);
        // down rows: acc += h * down[kept row]
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
          if (q < nb) {
            const uint8_t* st = stage + (size_t)((base + i0 + q) % S) * L.stage_bytes;
            const uint4 dr = reinterpret_cast<const uint4*>(st + 2 * d)[tc];
            const __half2* h = reinterpret_cast<const __half2*>(&dr);
            float df[kEPT];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f2 = __half22float2(h[e]);
              df[2 * e] = f2.x;
              df[2 * e + 1] = f2.y;
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              if (t < ntok) {
                const float hq = hsm[q * kMaxTok + t];
#pragma unroll
                for (int e = 0; e < kEPT; ++e) acc[t][e] = fmaf(hq, df[e], acc[t][e]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0)
          for (int q = 0; q < nb; ++q) mbar_arrive(&empty[(base + i0 + q) % S]);
        i0 += nb;
        if (tc == 0) s_consumed = base + i0;
      }
    }
    __syncthreads();
    if (s_abort) break;
  }
  // flush the last group (consumers)
  if (!producer && cur_g >= 0 && !s_abort) {
    float* dst = p.part + ((size_t)(blockIdx.x + cur_g) * kMaxTok) * d + tid * kEPT;
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if (t < s_gd.n_tok) {
        float4* o = reinterpret_cast<float4*>(dst + (size_t)t * d);
        o[0] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
        o[1] = make_float4(acc[t][4], acc[t][5], acc[t][6], acc[t][7]);
      }
  }
  // on an abort, wait (bounded) for copies still in flight before the CTA exits
  if (s_abort && tid == 0) {
    for (int i = s_consumed; i < s_issued; ++i) (void)mbar_wait(&full[i % S], (i / S) & 1);
  }
}

// ===========================================================================
// combine_kernel: y[b] = sum of the partial outputs of every (group, CTA) that
// holds token b, in a fixed order; optional RMSNorm; fp16 output.
// ===========================================================================
constexpr int kCombWarps = 8;
constexpr int kCombSlice = 128;  // hidden elements per CTA (32 lanes x float4)

__device__ __forceinline__ long long cta_first_item(long long N, int c, int P) {
  return N * c / P;
}
__device__ __forceinline__ int cta_of_item(long long i, long long N, int P) {
  return (int)(((i + 1) * P + N - 1) / N) - 1;
}

__global__ void __launch_bounds__(kCombWarps * 32) combine_kernel(ExpertParams p) {
  __shared__ float4 s_acc[kCombWarps][32];
  __shared__ int s_goff[kMaxSlots][2];
  __shared__ int s_last;
  __shared__ float s_red[kCombWarps];
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.y, slice = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = p.d;
  const long long N = *reinterpret_cast<volatile int*>(&p.ctrl->N);
  const int P = p.P3;
  // item range of each group holding token b
  if (threadIdx.x < p.n_slots) {
    const int tg = p.tok_groups[b * kMaxSlots + threadIdx.x];
    const int g = tg >> 3;
    int s0 = 0;
    for (int q = 0; q < g; ++q) s0 += __ldcg(p.group_total + q);
    s_goff[threadIdx.x][0] = s0;
    s_goff[threadIdx.x][1] = s0 + __ldcg(p.group_total + g);
  }
  __syncthreads();
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int cnt = 0;
  const int col = slice * kCombSlice + lane * 4;
  for (int j = 0; j < p.n_slots; ++j) {
    const int tg = p.tok_groups[b * kMaxSlots + j];
    const int g = tg >> 3, tau = tg & 7;
    const long long s0 = s_goff[j][0], s1 = s_goff[j][1];
    if (s1 <= s0) continue;
    const int c_lo = cta_of_item(s0, N, P), c_hi = cta_of_item(s1 - 1, N, P);
    for (int c = c_lo; c <= c_hi; ++c) {
      if (cta_first_item(N, c, P) == cta_first_item(N, c + 1, P)) continue;  // empty range
      if ((cnt++ % kCombWarps) != warp) continue;
      const float4 v = __ldcg(reinterpret_cast<const float4*>(
          p.part + ((size_t)(c + g) * kMaxTok + tau) * d + col));
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
  }
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float4 t = s_acc[0][lane];
    for (int w = 1; w < kCombWarps; ++w) {
      const float4 v = s_acc[w][lane];
      t.x += v.x;
      t.y += v.y;
      t.z += v.z;
      t.w += v.w;
    }
    if (!p.rmsnorm) {
      __half2* yo = reinterpret_cast<__half2*>(p.y + (size_t)b * d + col);
      yo[0] = __floats2half2_rn(t.x, t.y);
      yo[1] = __floats2half2_rn(t.z, t.w);
    } else {
      *reinterpret_cast<float4*>(p.yacc + (size_t)b * d + col) = t;
      float ss = t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) p.sumsq[(size_t)b * gridDim.x + slice] = ss;
    }
  }
  if (!p.rmsnorm) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&p.tok_ctr[b], 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (threadIdx.x == 0) {
    float ss = 0.f;
    for (int s = 0; s < (int)gridDim.x; ++s) ss += __ldcg(p.sumsq + (size_t)b * gridDim.x + s);
    s_red[0] = rsqrtf(ss / (float)d + 1e-6f);
    p.tok_ctr[b] = 0;
  }
  __syncthreads();
  const float rinv = s_red[0];
  for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(p.yacc + (size_t)b * d) + i);
    __half2* yo = reinterpret_cast<__half2*>(p.y + (size_t)b * d + 4 * i);
    yo[0] = __floats2half2_rn(v.x * rinv, v.y * rinv);
    yo[1] = __floats2half2_rn(v.z * rinv, v.w * rinv);
  }
}

// ===========================================================================
// launches
// ===========================================================================
static cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                                   cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

cudaError_t launch_up(const ExpertParams& p, int grid, cudaStream_t st, bool pdl) {
  const size_t smem = up_smem_bytes(p.d);
  cudaError_t e = cudaFuncSetAttribute(up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(grid), dim3(kUpThreads), smem, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, up_kernel, p);
}

size_t gather_smem_bytes(int d, int stages, int nt, int list_cap) {
  return gather_layout(d, stages, d / (32 * kEPT), nt, list_cap).total;
}

cudaError_t launch_gather(const ExpertParams& p, int nt, cudaStream_t st, bool pdl) {
  const int ncw = p.d / (32 * kEPT);
  const size_t smem = gather_smem_bytes(p.d, p.stages, nt, p.list_cap);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(p.P3), dim3((ncw + 1) * 32), smem, st, pdl, attr);
  cudaError_t e;
#define SESG_G(NTV, MT)                                                                        \
  if ((ncw + 1) * 32 > MT) return cudaErrorInvalidConfiguration;                              \
  e = cudaFuncSetAttribute(gather_kernel<NTV, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           (int)smem);                                                         \
  if (e != cudaSuccess) return e;                                                              \
  return cudaLaunchKernelEx(&cfg, gather_kernel<NTV, MT>, p);
  switch (nt) {
    case 1: SESG_G(1, 1024)
    case 2: SESG_G(2, 1024)
    case 4: SESG_G(4, 800)
    default: SESG_G(8, 544)
  }
#undef SESG_G
}

cudaError_t launch_combine(const ExpertParams& p, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg =
      make_cfg(dim3(p.d / kCombSlice, p.B), dim3(kCombWarps * 32), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace sesg
