// Steps 1 and 2 of Algorithm 1 "Efficient Sparse Kernel" of "FloE: On-the-Fly MoE
// Inference on Memory-constrained GPU" (sec. 三 "系统协同优化"): v = x W^up from the INT2
// codes (the intra-expert predictor of sec. "双稀疏预测器" reuses exactly this product),
// then mask = |v| > t, with the kept columns of every 16-column tile compacted into
// an item list for the gather kernel.
//
// Work unit: (group, M-tile) = one expert, up to 8 of its tokens, 16 output columns.
// Each CTA takes a contiguous range of units.  One producer thread streams the
// units' packed strips (contiguous in memory) into a 4-stage shared-memory ring
// with 1-D bulk copies (TMA).  Consumer warp w owns superblock sb = w % nsb of
// M-tile slot w / nsb, reads the B fragments (the group's tokens) of its superblock
// from the group's x in shared memory as each k-step comes, and runs the INT2 dot
// products on the tensor cores (mma.sync m16n8k16, fp16 in, fp32 accumulate).  Partial v of the superblocks are summed in
// a fixed order by one warp per M-tile, which also applies the threshold.
#include "params.cuh"

namespace sesg {

constexpr int kUpMaxStages = 4;
constexpr size_t kUpSmemBudget = 220 * 1024;
// compute warps per CTA (up to): with the B fragments read from shared memory, 16
// warps (two M-tiles of 8 superblocks per step at d = 4096) hide the dependent mma and
// code-extraction latencies that 8 warps left exposed; at most kUpMaxMpar M-tiles per
// step, since one finalize warp sums and thresholds all of them
constexpr int kUpWarps = 16;
constexpr int kUpMaxMpar = 4;
constexpr int kXPad = 8;  // halves after each token's x row (rows 16 bytes off the banks)

struct UpLayout {
  int nsb, mpar, nwc, spp, stages;
  size_t strip, stage_bytes, off_full, off_empty, off_stage, off_x, off_xg, off_vpart, off_vbuf, total;
};

// Geometry: nwc compute warps (one superblock of one of mpar M-tiles each), one finalize
// warp, one producer warp.  A ring stage holds spp steps of mpar M-tile strips, so that
// every bulk-copy transaction moves >= 32 KB (smaller ones cost the same fixed time).
__host__ __device__ inline UpLayout up_layout(int d, int max_tok) {
  UpLayout L;
  L.nsb = n_superblocks(d);
  if (L.nsb <= 8) {
    L.mpar = kUpWarps / L.nsb;
    if (L.mpar > kUpMaxMpar) L.mpar = kUpMaxMpar;
    if (L.mpar < 1) L.mpar = 1;
    L.nwc = L.mpar * L.nsb;
  } else {
    L.mpar = 1;
    L.nwc = L.nsb;
  }
  L.strip = (size_t)L.nsb * kBlkBytes;
  const size_t step = L.strip * L.mpar;
  L.spp = step >= 32768 ? 1 : (int)((32768 + step - 1) / step);
  size_t fixed = 256 + (size_t)max_tok * (d + kXPad) * 2 + (size_t)kMaxTok * (d / kGroup) * 4 +
                 (size_t)2 * L.nwc * 32 * 16 + (size_t)L.mpar * 16 * kMaxTok * 4 + 64;
  while (L.spp > 1 && fixed + 2 * step * L.spp > kUpSmemBudget) --L.spp;
  L.stage_bytes = step * L.spp;
  L.stages = (int)((kUpSmemBudget - fixed) / L.stage_bytes);
  L.stages = L.stages > kUpMaxStages ? kUpMaxStages : (L.stages < 2 ? 2 : L.stages);
  size_t o = 0;
  L.off_full = o;
  o += 8 * kUpMaxStages;
  L.off_empty = o;
  o += 8 * kUpMaxStages;
  o = (o + 127) & ~(size_t)127;
  L.off_stage = o;
  o += L.stage_bytes * L.stages;
  L.off_x = o;
  o += (size_t)max_tok * (d + kXPad) * 2;
  o = (o + 15) & ~(size_t)15;
  L.off_xg = o;
  o += (size_t)kMaxTok * (d / kGroup) * 4;
  o = (o + 15) & ~(size_t)15;
  L.off_vpart = o;
  o += (size_t)2 * L.nwc * 32 * 16;
  L.off_vbuf = o;
  o += (size_t)L.mpar * 16 * kMaxTok * 4;
  L.total = o;
  return L;
}

// Where lane (gl, c) finds its B operand: token gl / G's x at the superblock's input
// 16 ks + 2 c (and + 8) for k-step ks, used when the k-step's quantiser group class
// gi % G is the lane's slot class gl % G and the token exists, else zero.
struct BSrc {
  const __half* row;  // the token's x at the superblock start + 2 c (a valid address)
  int cls;            // gl % G
  bool tok;           // token gl / G is one of the group's
};

// k-steps of quantiser group GI (compile time): 4 mma into the 4 accumulator chains.
template <int G, int GI>
__device__ __forceinline__ void up_group(const uint4 (&w)[4], const BSrc& bs, float (&D)[4][4]) {
  const bool on = bs.tok && bs.cls == GI % G;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    uint32_t a[4];
    a[0] = code_pair<GI>(w[t].x);
    a[1] = code_pair<GI>(w[t].y);
    a[2] = code_pair<GI>(w[t].z);
    a[3] = code_pair<GI>(w[t].w);
    const __half* xr = bs.row + 16 * (GI * 4 + t);
    const uint32_t b0 = on ? *reinterpret_cast<const uint32_t*>(xr) : 0u;
    const uint32_t b1 = on ? *reinterpret_cast<const uint32_t*>(xr + 8) : 0u;
    mma_16816(D[t], a, b0, b1);
  }
}

template <int T, int PH, int GAM>
__device__ __forceinline__ void up_phase_groups(const uint4 (&w)[4], const BSrc& bs, float (&D)[4][4],
                                                int ng) {
  constexpr int G = 8 / T;
  if constexpr (GAM < G) {
    constexpr int GI = PH * G + GAM;
    if (GI < ng) up_group<G, GI>(w, bs, D);
    up_phase_groups<T, PH, GAM + 1>(w, bs, D, ng);
  }
}

// Fold the accumulators of phase PH (G quantiser groups side by side) into v.
template <int T, int PH>
__device__ __forceinline__ void up_phase(const uint4 (&w)[4], const BSrc& bs, const uint8_t* __restrict__ szt,
                                         const float* __restrict__ xg, int sb, int ng, int ngrp,
                                         float (&vacc)[2][2]) {
  constexpr int G = 8 / T;
  const int lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
  float D[4][4];
#pragma unroll
  for (int t = 0; t < 4; ++t) D[t][0] = D[t][1] = D[t][2] = D[t][3] = 0.f;
  up_phase_groups<T, PH, 0>(w, bs, D, ng);
  const int gi_lane = (G >= 2) ? (2 * c) % G : 0;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int gi = (G >= 2) ? PH * G + gi_lane + s : PH;
    const int tau = (G >= 2) ? (2 * c) / G : 2 * c + s;
    if (gi < ng) {
      const float cs = pos_scale(gi);
      const float X = xg[tau * ngrp + sb * 8 + gi];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const __half2 h = *reinterpret_cast<const __half2*>(szt + ((gl + 8 * r) * 8 + gi) * 4);
        const float sf = __low2float(h), zf = __high2float(h);
        const float acc = (D[0][2 * r + s] + D[1][2 * r + s]) + (D[2][2 * r + s] + D[3][2 * r + s]);
        vacc[r][s] = fmaf(sf, fmaf(-zf, X, acc * cs), vacc[r][s]);
      }
    }
  }
}

template <int T, int PH>
__device__ __forceinline__ void up_phases(const uint4 (&w)[4], const BSrc& bs, const uint8_t* __restrict__ szt,
                                          const float* __restrict__ xg, int sb, int ng, int ngrp,
                                          float (&vacc)[2][2]) {
  if constexpr (PH < T) {
    up_phase<T, PH>(w, bs, szt, xg, sb, ng, ngrp, vacc);
    up_phases<T, PH + 1>(w, bs, szt, xg, sb, ng, ngrp, vacc);
  }
}

// One warp: partial v of its superblock of one M-tile.
//
// Tensor-core mapping: M = 16 output columns, K = 16 inputs, N = 8 slots.  A slot
// is a (token, group class) pair: with T tokens (padded to a power of two) there
// are G = 8/T classes, and a k-step of quantiser group gi only feeds the slots of
// class gi % G, whose B column carries that token's x; the other B columns are
// zero.  One accumulator tile therefore collects G quantiser groups side by side,
// and the per-group correction v += s * (A_g - z * X_g) (X_g = sum of x over the
// group) is applied once per G groups.  Four accumulator chains (one per k-step of a
// group) shorten the mma dependency chain.  Every group index is a compile-time
// constant, so the codes and accumulators stay in registers.
template <int T>
__device__ __forceinline__ void up_superblock(const uint8_t* __restrict__ blk, const BSrc& bs,
                                              const float* __restrict__ xg, int sb, int ng,
                                              int ngrp, float (&vacc)[2][2]) {
  const int lane = threadIdx.x & 31;
  uint4 w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = reinterpret_cast<const uint4*>(blk)[q * 32 + lane];
  up_phases<T, 0>(w, bs, blk + kBlkCodeBytes, xg, sb, ng, ngrp, vacc);
}

// One warp, after the superblock partials are summed: per-token v of the M-tile's
// 16 columns, step 2 (mask = |v| > t, union over the group's tokens), compaction of
// the kept columns by ballot, and the optional debug outputs.
template <int T>
__device__ __forceinline__ void up_finalize(const ExpertParams& p, const GroupDesc& gd, int g,
                                            long long u, int mt, float thr, const float (&vacc)[2][2],
                                            float* __restrict__ vbuf) {
  constexpr int G = 8 / T;
  const int lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
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
  __syncwarp();
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
}

__device__ __forceinline__ int barrier_or(int id, int nthreads, bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.u32 pin, %1, 0;\n\t"
      "barrier.red.or.pred pout, %2, %3, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}"
      : "=r"(r)
      : "r"((unsigned)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r;
}

template <int MAXT>
__global__ void __launch_bounds__(MAXT, 1) up_kernel(ExpertParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int d = p.d;
  const UpLayout L = up_layout(d, p.max_tok);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.off_empty);
  uint8_t* stage = smem + L.off_stage;
  __half* xs = reinterpret_cast<__half*>(smem + L.off_x);
  float* xg = reinterpret_cast<float*>(smem + L.off_xg);
  float4* vpart = reinterpret_cast<float4*>(smem + L.off_vpart);
  float* vbuf = reinterpret_cast<float*>(smem + L.off_vbuf);
  __shared__ GroupDesc s_gd;
  __shared__ int s_abort, s_issued, s_consumed;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwc = L.nwc, nsb = L.nsb, S = L.stages, spp = L.spp;
  const int fin_warp = nwc, prod_warp = nwc + 1;
  const int nbar = (nwc + 1) * 32;  // compute warps + the finalize warp
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nwc);
    }
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  const int G = *reinterpret_cast<volatile int*>(&p.ctrl->G);
  const int MT = p.f / kMTile;
  const long long U = (long long)G * MT;
  const long long u0 = U * blockIdx.x / gridDim.x, u1 = U * (blockIdx.x + 1) / gridDim.x;
  const int ngrp = d / kGroup;
  // steps: up to mpar consecutive units of one group; stage = up to spp consecutive steps

  if (warp == prod_warp) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      // stage st (ring slot s, parity ph) and the group g of unit us, advanced without
      // divisions
      int st = 0, s = 0, ph = 0;
      long long g_lo = u0 >= 0 ? (u0 / MT) * MT : 0;  // first unit of us's group
      for (long long us = u0; us < u1;) {
        if (st >= S && !mbar_wait(&empty[s], ph ^ 1)) {
          set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
        // the stage's steps and bytes
        long long ends[4];
        uint32_t bytes = 0;
        int nst = 0;
        {
          long long glo = g_lo;
          for (long long v = us; v < u1 && nst < spp; ++nst) {
            if (v >= glo + MT) glo += MT;
            ends[nst] = min(min(v + L.mpar, u1), glo + MT);
            bytes += (uint32_t)((ends[nst] - v) * L.strip);
            v = ends[nst];
          }
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        for (int q = 0; q < nst; ++q) {
          const long long ue = ends[q];
          if (us >= g_lo + MT) g_lo += MT;
          const int g = (int)(g_lo / MT);
          int el;
          const ExpertSet& es = expert_set(p, p.groups[g].expert, el);
          const uint8_t* src = es.up + (size_t)el * es.up_stride + (size_t)(us - g_lo) * L.strip;
          bulk_g2s(stage + (size_t)s * L.stage_bytes + (size_t)q * L.mpar * L.strip, src,
                   (uint32_t)((ue - us) * L.strip), &full[s], pol);
          us = ue;
        }
        s_issued = st + 1;
        ++st;
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  } else {
    // ---- compute warps (w < nwc) and the finalize warp (w == nwc)
    const bool fin = warp == fin_warp;
    const int m_slot = fin ? 0 : warp / nsb, sb = fin ? 0 : warp % nsb;
    const int ng = min(8, (d - sb * kSuper) / kGroup);
    int cur_g = -1, T = 1;
    float thr = 0.f;
    BSrc bs{xs, 0, false};
    const int xstride = d + kXPad;
    // step position: jj within the stage, stage st (ring slot s, parity ph); the group g
    // of unit us and its first unit g_lo; all advanced without divisions
    int jj = 0, st = 0, s = 0, ph = 0, jpar = 0;
    int g = (int)(u0 / MT);
    long long g_lo = (long long)g * MT;
    for (long long us = u0; us < u1;) {
      if (us >= g_lo + MT) {
        g_lo += MT;
        ++g;
      }
      const long long ue = min(min(us + L.mpar, u1), g_lo + MT);
      if (g != cur_g) {
        named_barrier(1, nbar);
        if (threadIdx.x == 0) s_gd = p.groups[g];
        named_barrier(1, nbar);
        const int n_tok = s_gd.n_tok;
        for (int i = threadIdx.x; i < n_tok * (d / 8); i += nbar) {
          const int t = i / (d / 8), o = i % (d / 8);
          reinterpret_cast<uint4*>(xs + (size_t)t * xstride)[o] =
              __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)s_gd.tok[t] * d) + o);
        }
        int el;
        const ExpertSet& es = expert_set(p, s_gd.expert, el);
        thr = es.thr[el];
        named_barrier(1, nbar);
        for (int i = threadIdx.x; i < kMaxTok * ngrp; i += nbar) {
          const int t = i / ngrp, grp = i % ngrp;
          float sum = 0.f;
          if (t < n_tok) {
            const uint4* xr = reinterpret_cast<const uint4*>(xs + (size_t)t * xstride + grp * kGroup);
#pragma unroll
            for (int r = 0; r < kGroup / 8; ++r) {
              const uint4 v = xr[r];
              const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f2 = __half22float2(h2[e]);
                sum += f2.x;
                sum += f2.y;
              }
            }
          }
          xg[i] = sum;
        }
        T = n_tok <= 1 ? 1 : n_tok <= 2 ? 2 : n_tok <= 4 ? 4 : 8;
        {
          const int Gc = 8 / T, gl = lane >> 2, tau = gl / Gc;
          bs.tok = tau < n_tok;
          bs.cls = gl % Gc;
          bs.row = xs + (size_t)(bs.tok ? tau : 0) * xstride + sb * kSuper + 2 * (lane & 3);
        }
        named_barrier(1, nbar);
        cur_g = g;
      }
      const bool first = jj == 0;
      const bool last = jj == spp - 1 || ue >= u1;
      bool ok = true;
      if (!fin) {
        if (first) ok = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));  // the mma below is warp-wide
        const bool active = us + m_slot < ue;
        float vacc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if (active && ok) {
          const uint8_t* blk = stage + (size_t)s * L.stage_bytes +
                               ((size_t)jj * L.mpar + m_slot) * L.strip + (size_t)sb * kBlkBytes;
          switch (T) {
            case 1: up_superblock<1>(blk, bs, xg, sb, ng, ngrp, vacc); break;
            case 2: up_superblock<2>(blk, bs, xg, sb, ng, ngrp, vacc); break;
            case 4: up_superblock<4>(blk, bs, xg, sb, ng, ngrp, vacc); break;
            default: up_superblock<8>(blk, bs, xg, sb, ng, ngrp, vacc); break;
          }
        }
        vpart[((jpar & 1) * nwc + warp) * 32 + lane] =
            make_float4(vacc[0][0], vacc[0][1], vacc[1][0], vacc[1][1]);
        __syncwarp();
        if (last && lane == 0) mbar_arrive(&empty[s]);
      }
      if (barrier_or(1, nbar, !ok)) {
        if (threadIdx.x == 0) {
          set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
        break;
      }
      if (threadIdx.x == 0 && last) s_consumed = st + 1;  // stages 0..st are free
      if (fin) {
        // sum the superblock partials of every M-tile of step j; threshold and compaction
        for (int m = 0; m < L.mpar; ++m) {
          if (us + m >= ue) break;
          float v[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
          for (int q = 0; q < nsb; ++q) {
            const float4 pv = vpart[((jpar & 1) * nwc + m * nsb + q) * 32 + lane];
            v[0][0] += pv.x;
            v[0][1] += pv.y;
            v[1][0] += pv.z;
            v[1][1] += pv.w;
          }
          const long long u = us + m;
          const int mt = (int)(u - g_lo);
          float* vb = vbuf + m * 16 * kMaxTok;
          switch (T) {
            case 1: up_finalize<1>(p, s_gd, g, u, mt, thr, v, vb); break;
            case 2: up_finalize<2>(p, s_gd, g, u, mt, thr, v, vb); break;
            case 4: up_finalize<4>(p, s_gd, g, u, mt, thr, v, vb); break;
            default: up_finalize<8>(p, s_gd, g, u, mt, thr, v, vb); break;
          }
        }
      }
      us = ue;
      ++jpar;
      if (++jj == spp || ue >= u1) {
        jj = 0;
        ++st;
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  }
  __syncthreads();
  // on an abort, wait (bounded) for copies still in flight before the CTA exits
  if (s_abort && threadIdx.x == 0)
    for (int q = max(s_consumed, s_issued - S); q < s_issued; ++q) (void)mbar_wait(&full[q % S], (q / S) & 1);
}

size_t up_smem_bytes(int d, int max_tok) { return up_layout(d, max_tok).total; }
int up_threads(int d) { return (up_layout(d, 1).nwc + 2) * 32; }

// Register budget: up to 10 warps, up to 14 (d <= 6144: one warp per superblock) or up to
// 18 (d <= 4096: 16 compute warps; beyond 6144) warps per CTA.
static const void* up_kernel_for(int d) {
  const int t = up_threads(d);
  return t <= 320 ? (const void*)up_kernel<320> : t <= 448 ? (const void*)up_kernel<448> : (const void*)up_kernel<576>;
}

int up_blocks_per_sm(int d, int max_tok) {
  const size_t smem = up_smem_bytes(d, max_tok);
  const void* fn = up_kernel_for(d);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, up_threads(d), smem) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_up(const ExpertParams& p, int grid, cudaStream_t st, bool pdl) {
  const size_t smem = up_smem_bytes(p.d, p.max_tok);
  const void* fn = up_kernel_for(p.d);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(up_threads(p.d));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const int t = up_threads(p.d);
  if (t <= 320) return cudaLaunchKernelEx(&cfg, up_kernel<320>, p);
  if (t <= 448) return cudaLaunchKernelEx(&cfg, up_kernel<448>, p);
  return cudaLaunchKernelEx(&cfg, up_kernel<576>, p);
}

}  // namespace sesg
