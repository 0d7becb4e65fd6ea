// Decode path for one or two tokens: the MoE layer of "FloE: On-the-Fly MoE
// Inference on Memory-constrained GPU" (sec. 三 "系统协同优化", Algorithm 1
// "Efficient Sparse Kernel" for every chosen expert) as two kernels chained by
// programmatic dependent launch:
//
//   decode_up_kernel      one CTA per SM.  Routes the tokens (router GEMV on router
//                         rows loaded into registers before the previous kernel
//                         ends, softmax top-k, expert groups; every CTA redundantly,
//                         the result is identical), then steps 1-2 of Algorithm 1 on a
//                         fixed, equal share of the work units (16 output columns of
//                         one expert): packed INT2 strips stream through a TMA ring;
//                         16 warps, one 512-input superblock each, two units in
//                         flight; per unit lane a finalize warp adds each unit's
//                         superblock partials in a fixed order, applies
//                         mask = |v| > t and stages the unit's kept columns; at the
//                         end the CTA writes them as one list in unit order.
//   decode_gather_kernel  one CTA per SM.  An equal share of all kept columns, in
//                         (group, column) order: their gate and down rows stream
//                         through a TMA ring; 16 warps form x . gate for a batch of
//                         rows (one barrier per batch), h = SiLU(.) * v * router
//                         weight, acc += h * down; each CTA adds its share of y to
//                         the fp32 accumulator (kDecYRep copies) with vector atomics
//                         (fewer additions per address) and the last CTA to
//                         finish rounds y to fp16 once, after the RMSNorm of stacked
//                         layers.
//
// Every CTA's share and every order inside a CTA are fixed; only the order in which
// the CTAs' shares reach the fp32 accumulator varies, so y can differ between calls
// in the last bits of the fp32 sum (and by one fp16 ulp where that sum sits on a
// rounding boundary).  Every wait is bounded; on expiry a CTA records
// MOE_ERR_TIMEOUT, stops, and waits (bounded) for its copies in flight before it
// exits.
#include <type_traits>

#include "params.cuh"

namespace sesg {

namespace {

constexpr int kDecMaxG = 24;     // groups: 2 tokens x 8 experts + 8 shared experts
constexpr int kDecMaxE = 64;     // routed experts of the in-kernel router
constexpr int kDecMaxSb = 12;    // superblocks of 512 inputs (d <= 6144)
// unit slots of superblock partials (a power of two): the up warps run up to kDecNV units
// ahead of the finalize warps; 2 measured faster than 4 (Mixtral-8x7B one-token layer at
// 70 %: 44.47 against 44.73 us), 8 does not fit the one-kernel layer's shared memory
constexpr int kDecNV = 2;
constexpr int kDecMaxSu = 12;    // up-ring stages
constexpr int kDecMaxSr = 16;    // row-ring stages (the h warp's descriptor ring needs kDecMaxSr + 3 kDecRows <= kHD)
constexpr int kDecMaxUnits = 128;  // units per CTA
constexpr int kDecRows = 4;      // kept rows per gather batch
// producer lanes that issue the kept rows' bulk copies, in rounds of one row per lane: one
// thread issues about 2.8 bulk copies per us whatever their size (measured on all SMs at
// once: 8 KB copies 22.7 GB/s per SM from one lane, 33-38 GB/s from four).  Two lanes
// measured best on the one-token Mixtral-8x7B layer (70 %: 42.7 us, four lanes 42.9-43.3,
// one 44.4); rounds aligned to the gather batches or lanes that run independently of
// each other were slower.
constexpr int kRowLanes = 2;
constexpr int kDecMaxGw = 24;    // gather warps
// up kernel: two unit lanes of up to 8 superblock warps (d <= 4096) or one lane of up to 12,
// plus the strip producer and one finalize warp per lane
__host__ __device__ constexpr int dec_lanes(int nsb) { return nsb <= 8 ? 2 : 1; }
constexpr int kUpThreads = (2 * 8 + 3) * 32;
static_assert((kDecMaxSb + 2) * 32 <= kUpThreads, "one-lane up kernel block");
// register cap of the up kernel: 96 per thread, so that 5 warps fit one SM sub-partition
constexpr int kUpRegThreads = 640;
static_assert(kUpThreads <= kUpRegThreads, "up kernel block exceeds its register budget");
constexpr int kGaThreads = (kDecMaxGw + 1) * 32;      // gather warps + the row producer warp
constexpr int kGaSmallThreads = (16 + 1) * 32;       // d <= 4096: 96 registers per thread
constexpr int kDecMaxD = 6144;

__host__ __device__ inline size_t al16(size_t o) { return (o + 15) & ~(size_t)15; }

// ---- up kernel shared memory
struct UpMisc {
  int abort;
  int G;
  int pend[kDecMaxSu];         // strip in flight in the stage (issue index + 1) or 0
  int total;                   // kept columns of this CTA's units
  int tidx[2][kMaxTok];
  float tw[2][kMaxTok];
  float vbuf[kDecNV][16 * 2];
  int ucnt[kDecMaxUnits];      // kept columns of each unit, then their list offsets
};

struct UpLayoutD {
  int nsb, nwarps, su;
  size_t strip, ring;
  size_t off_bar, off_misc, off_ring, off_x, off_vpart, off_xg, off_grp, off_lred, off_ent, total;
};

// umax: units per CTA, at most
__host__ __device__ inline UpLayoutD up_layout_d(int d, int B, int E, int su, int umax) {
  UpLayoutD L;
  L.nsb = n_superblocks(d);
  L.nwarps = dec_lanes(L.nsb) * (L.nsb + 1) + 1;
  L.su = su;
  L.strip = (size_t)L.nsb * kBlkBytes;
  L.ring = L.strip * su;
  size_t o = 0;
  L.off_bar = o;
  o += 8 * (size_t)(2 * kDecMaxSu + 2 * kDecNV);
  o = al16(o);
  L.off_misc = o;
  o += al16(sizeof(UpMisc));
  o = (o + 127) & ~(size_t)127;
  L.off_ring = o;
  o += al16(L.ring);
  L.off_x = o;
  o += al16((size_t)B * d * 2);
  L.off_vpart = o;
  o += (size_t)kDecNV * L.nsb * 32 * 16;
  L.off_xg = o;
  o += (size_t)2 * L.nsb * 16 * 4;
  L.off_grp = o;
  o += al16(sizeof(GroupDesc) * kDecMaxG);
  L.off_lred = o;
  o += (size_t)L.nwarps * 2 * E * 4;
  L.off_ent = o;
  o += (size_t)umax * 16 * 16;
  L.total = o;
  return L;
}

// ---- gather kernel shared memory
struct GaRow {
  int col;    // kept column
  int g;      // group
  float v[2]; // v per group token (0 where that token drops the column)
};

struct GaMisc {
  int abort;
  int last;                    // this CTA finished last
  int G;
  int issued;                  // rows issued (0 .. issued-1)
  int consumed;                // rows whose stages are free again
  int tmap[kDecMaxG][2];       // group token of batch token b, -1 if none
  float tw[kDecMaxG][2];       // its combine weight
};

struct GaLayoutD {
  int ngw, nwarps, sr, cap;
  size_t row;
  size_t off_bar, off_misc, off_ring, off_list, off_red, off_pre, off_grp, total;
};

__host__ __device__ inline GaLayoutD ga_layout_d(int d, int sr, int cap, int P) {
  GaLayoutD L;
  L.ngw = d / 256;
  L.nwarps = L.ngw + 1;
  L.sr = sr;
  L.cap = cap;
  L.row = (size_t)4 * d;
  size_t o = 0;
  L.off_bar = o;
  o += 8 * (size_t)(2 * kDecMaxSr);
  o = al16(o);
  L.off_misc = o;
  o += al16(sizeof(GaMisc));
  o = (o + 127) & ~(size_t)127;
  L.off_ring = o;
  o += L.row * sr;
  L.off_list = o;
  o += sizeof(GaRow) * (size_t)cap;
  L.off_red = o;
  o += (size_t)2 * kDecRows * 2 * kDecMaxGw * 4 + (size_t)2 * kDecRows * 2 * 4;
  L.off_pre = o;
  o += al16(4 * ((size_t)P + 1));
  L.off_grp = o;
  o += al16(sizeof(GroupDesc) * kDecMaxG);
  L.total = o;
  return L;
}

__device__ __forceinline__ const ExpertSet& dec_set(const DecodeParams& p, int expert, int& local) {
  if (expert < p.routed.E) {
    local = expert;
    return p.routed;
  }
  local = expert - p.routed.E;
  return p.shared;
}

__device__ __forceinline__ int vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

__device__ __forceinline__ void dec_fail(const DecodeParams& p, int* abort_flag) {
  set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
  atomicExch(abort_flag, 1);
}

__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// SiLU with the fast division (2 ulp): g / (1 + e^-g)
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ long long muldiv(long long a, long long b, long long c) { return a * b / c; }

// ---------------------------------------------------------------------------
// Routing (all threads of the CTA): logits, softmax top-k, groups.  Ties between
// equal logits go to the lower expert index; groups are the chosen experts in
// ascending index order, then the shared experts.
//
// Thread t owns the router rows rs + u * nrs (u < kRouteRows per pass) of expert chunk
// ec (8 experts, 16 bytes per row); the first pass's rows are loaded before the
// dependency wait (the router weight is not written by the previous kernel).  The
// products x * W_r are formed by fma.rn.f32.f16 on the fp16 values as stored: the
// exact product rounded once into the fp32 sum, without conversions.
// ---------------------------------------------------------------------------
constexpr int kRouteRows = 8;

template <int HA, int HB>
__device__ __forceinline__ float fma_f16(uint32_t a, uint32_t b, float c) {
  float r;
  if constexpr (HA == 0 && HB == 0)
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %3;\n\t}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  else if constexpr (HA == 0 && HB == 1)
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b1, %3;\n\t}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  else if constexpr (HA == 1 && HB == 0)
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a1, b0, %3;\n\t}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  else
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\tmov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %3;\n\t}" : "=f"(r) : "r"(a), "r"(b), "f"(c));
  return r;
}

struct RouteSplit {
  int nchunk, ec, rs, nrs;
};

__device__ __forceinline__ RouteSplit route_split(int E, int nthreads) {
  RouteSplit r;
  r.nchunk = E / 8;
  r.ec = (int)threadIdx.x % r.nchunk;
  r.rs = (int)threadIdx.x / r.nchunk;
  r.nrs = nthreads / r.nchunk;
  return r;
}

// the first pass's router rows of this thread (zero past d)
__device__ __forceinline__ void route_prefetch(const DecodeParams& p, const RouteSplit& rt, uint4 (&wv)[kRouteRows]) {
  const int E = p.routed.E, d = p.d;
#pragma unroll
  for (int u = 0; u < kRouteRows; ++u) {
    const int r = rt.rs + u * rt.nrs;
    wv[u] = r < d ? __ldg(reinterpret_cast<const uint4*>(p.w_router + (size_t)r * E + rt.ec * 8))
                  : make_uint4(0, 0, 0, 0);
  }
}

template <int B, typename Misc>
__device__ __forceinline__ void dec_route(const DecodeParams& p, int nthreads, const RouteSplit& rt,
                                          const uint4 (&wv0)[kRouteRows], const __half* xs, float* lred,
                                          Misc* m, GroupDesc* grp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = nthreads / 32;
  const int E = p.routed.E, d = p.d, k = p.k;
  const int nchunk = rt.nchunk;
  float acc[B][8];
#pragma unroll
  for (int b = 0; b < B; ++b)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[b][i] = 0.f;
  for (int r0 = rt.rs, pass = 0; r0 < d; r0 += kRouteRows * rt.nrs, ++pass) {
    uint4 wv[kRouteRows];
#pragma unroll
    for (int u = 0; u < kRouteRows; ++u) {
      const int r = r0 + u * rt.nrs;
      wv[u] = pass == 0 ? wv0[u]
                        : (r < d ? __ldg(reinterpret_cast<const uint4*>(p.w_router + (size_t)r * E + rt.ec * 8))
                                 : make_uint4(0, 0, 0, 0));
    }
#pragma unroll
    for (int u = 0; u < kRouteRows; ++u) {
      const int r = r0 + u * rt.nrs;
      if (r < d) {
        const uint32_t w4[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
#pragma unroll
        for (int b = 0; b < B; ++b) {
          const uint32_t xh = *reinterpret_cast<const unsigned short*>(xs + (size_t)b * d + r);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[b][2 * i] = fma_f16<0, 0>(xh, w4[i], acc[b][2 * i]);
            acc[b][2 * i + 1] = fma_f16<0, 1>(xh, w4[i], acc[b][2 * i + 1]);
          }
        }
      }
    }
  }
  // warp sums by recursive halving: across lane bits 4, 3, 2 every lane keeps half of
  // its experts and adds its partner's copy of them (8 values -> 1), then the lanes
  // that still share an expert (bits 1 and 0 not used by the expert chunk) add up.
  const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0, u4 = (lane & 4) != 0;
  const int e_in = (u16 ? 4 : 0) + (u8 ? 2 : 0) + (u4 ? 1 : 0);
#pragma unroll
  for (int b = 0; b < B; ++b) {
    float w4[4], w2[2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w4[i] = (u16 ? acc[b][i + 4] : acc[b][i]) + __shfl_xor_sync(0xffffffffu, u16 ? acc[b][i] : acc[b][i + 4], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      w2[i] = (u8 ? w4[i + 2] : w4[i]) + __shfl_xor_sync(0xffffffffu, u8 ? w4[i] : w4[i + 2], 8);
    if (nchunk == 8) {
      // lane bits 0-2 name the chunk: every lane keeps two experts of its chunk
      const int e2 = (u16 ? 4 : 0) + (u8 ? 2 : 0);
      lred[(warp * B + b) * E + (lane & 7) * 8 + e2] = w2[0];
      lred[(warp * B + b) * E + (lane & 7) * 8 + e2 + 1] = w2[1];
      continue;
    }
    float v = (u4 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, u4 ? w2[0] : w2[1], 4);
    if (nchunk <= 2) v += __shfl_xor_sync(0xffffffffu, v, 2);
    if (nchunk == 1) v += __shfl_xor_sync(0xffffffffu, v, 1);
    if ((lane & 3) < nchunk) lred[(warp * B + b) * E + (lane % nchunk) * 8 + e_in] = v;
  }
  __syncthreads();
  if (warp == 0) {
  for (int b = 0; b < B; ++b) {
    // lane j: the logits of experts j and j + 32 (E <= 64), the warps' partial sums
    // added in a fixed order
    float l[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = lane + 32 * h;
      if (e < E) {
        float s = 0.f;
#pragma unroll 6
        for (int w = 0; w < nw; ++w) s += lred[(w * B + b) * E + e];
        // a NaN logit (from a non-finite token) ranks as -inf: the ranks then stay a
        // total order and the k chosen experts k distinct valid ones
        l[h] = isnan(s) ? -INFINITY : s;
      }
    }
    // top-k by rank: an expert's rank counts the experts with a larger logit, or an
    // equal one and a lower index; ranks 0..k-1 are chosen, listed by rank
    int rank[2] = {0, 0};
    for (int e = 0; e < E; ++e) {
      const float le = __shfl_sync(0xffffffffu, e < 32 ? l[0] : l[1], e & 31);
#pragma unroll
      for (int h = 0; h < 2; ++h) rank[h] += (le > l[h] || (le == l[h] && e < lane + 32 * h)) ? 1 : 0;
    }
    bool chosen[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) chosen[h] = lane + 32 * h < E && rank[h] < k;
    // the largest logit (that of the rank-0 expert)
    float lmax = fmaxf(l[0], l[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
    // softmax over the chosen experts (renormalised top-k) or over all E; the
    // denominator is a fixed-order butterfly sum
    float ex[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
      ex[h] = (lane + 32 * h < E && (chosen[h] || !p.renorm)) ? expf(l[h] - lmax) : 0.f;
    float denom = ex[0] + ex[1];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (chosen[h]) {
        const int e = lane + 32 * h, r = rank[h];
        const float w = ex[h] / denom;
        m->tidx[b][r] = e;
        m->tw[b][r] = w;
        if (blockIdx.x == 0) {
          p.topk_idx[b * k + r] = e;
          p.topk_w[b * k + r] = w;
          if (p.user_idx) p.user_idx[b * k + r] = e;
          if (p.user_w) p.user_w[b * k + r] = w;
        }
      }
    }
    __syncwarp();
  }
    // groups
    const int np = B * k;
    int e = -1, bb = 0, jj = 0;
    float ww = 0.f;
    if (lane < np) {
      bb = lane / k;
      jj = lane % k;
      e = m->tidx[bb][jj];
      ww = m->tw[bb][jj];
    }
    bool first = lane < np;
    int pos = 0, cnt = 0;
    for (int q = 0; q < np; ++q) {
      const int eq = __shfl_sync(0xffffffffu, e, q), bq = __shfl_sync(0xffffffffu, bb, q);
      if (lane < np && eq == e) {
        ++cnt;
        if (bq < bb) {
          first = false;
          ++pos;
        }
      }
    }
    const unsigned fm = __ballot_sync(0xffffffffu, first);
    int gi = 0;
    for (int q = 0; q < np; ++q) {
      const int eq = __shfl_sync(0xffffffffu, e, q);
      if (((fm >> q) & 1u) && eq < e) ++gi;
    }
    const int GR = __popc(fm);
    if (lane < np) {
      GroupDesc& gd = grp[gi];
      gd.tok[pos] = bb;
      gd.slot[pos] = jj;
      gd.w[pos] = ww;
      if (first) {
        gd.expert = e;
        gd.n_tok = cnt;
        for (int t = cnt; t < kMaxTok; ++t) {
          gd.tok[t] = 0;
          gd.slot[t] = 0;
          gd.w[t] = 0.f;
        }
      }
    }
    if (lane < p.n_shared) {
      GroupDesc& gd = grp[GR + lane];
      gd.expert = E + lane;
      gd.n_tok = B;
      for (int t = 0; t < kMaxTok; ++t) {
        gd.tok[t] = t < B ? t : 0;
        gd.slot[t] = t < B ? k + lane : 0;
        gd.w[t] = t < B ? 1.f : 0.f;
      }
    }
    if (lane == 0) m->G = GR + p.n_shared;
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// Up projection of one superblock (one warp).
//
// Tensor-core mapping as in the up kernel of the general path: M = 16 output
// columns, K = 16 inputs, N = 8 slots; slot n is (token n / G, class n % G) with
// G = 8 / T classes, and a k-step of quantiser group gi feeds only the slots of
// class gi % G.  A lane supplies B column gl, so it only ever holds x of its own
// token and class: T x 4 k-steps x 2 registers, selected (or zeroed) per mma.
// ---------------------------------------------------------------------------
template <int T>
__device__ __forceinline__ void dec_up_setup(const __half* xs, int d, const GroupDesc& gd, int sb,
                                             int ng, uint32_t (&xr)[T][4][2], float* xgw) {
  constexpr int G = 8 / T;
  const int lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
  const int tau = gl / G, cl = gl % G;
  const int n_tok = gd.n_tok;
#pragma unroll
  for (int jj = 0; jj < T; ++jj) {
    const int gi = cl + G * jj;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      uint32_t b0 = 0, b1 = 0;
      if (tau < n_tok && gi < ng) {
        const __half* xp = xs + (size_t)gd.tok[tau] * d + sb * kSuper + gi * kGroup + 16 * t + 2 * c;
        b0 = *reinterpret_cast<const uint32_t*>(xp);
        b1 = *reinterpret_cast<const uint32_t*>(xp + 8);
      }
      xr[jj][t][0] = b0;
      xr[jj][t][1] = b1;
    }
  }
  // X[tau][gi] = sum of x over quantiser group gi of this superblock (4 / T lanes each)
  constexpr int LPS = 4 / T;
  const int q = lane / LPS, part = lane % LPS;
  const int qt = q / 8, qg = q % 8;
  float s = 0.f;
  if (qt < n_tok && qg < ng) {
    const uint4* src = reinterpret_cast<const uint4*>(xs + (size_t)gd.tok[qt] * d + sb * kSuper +
                                                      qg * kGroup + part * (16 * T));
#pragma unroll
    for (int mm = 0; mm < 2 * T; ++mm) {
      const uint4 v = src[mm];
      const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f2 = __half22float2(h2[e]);
        s += f2.x;
        s += f2.y;
      }
    }
  }
#pragma unroll
  for (int off = 1; off < LPS; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (part == 0) xgw[qt * 8 + qg] = s;
  __syncwarp();
}

// FULL: all 8 quantiser groups of the superblock exist (no per-group test)
template <int T, int PH, int GAM, bool FULL>
__device__ __forceinline__ void dec_groups(const uint4 (&w)[4], const uint32_t (&xr)[T][4][2],
                                           int cl, float (&D)[4][4], int ng) {
  constexpr int G = 8 / T;
  if constexpr (GAM < G) {
    constexpr int GI = PH * G + GAM;
    if (FULL || GI < ng) {
      // x only in the slots of class GAM (the integer pipe is busy unpacking the codes)
      const uint32_t on = cl == GAM ? 0x3C003C00u : 0u;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        uint32_t a[4];
        a[0] = code_pair<GI>(w[t].x);
        a[1] = code_pair<GI>(w[t].y);
        a[2] = code_pair<GI>(w[t].z);
        a[3] = code_pair<GI>(w[t].w);
        mma_16816(D[t], a, hmul2_mask(xr[PH][t][0], on), hmul2_mask(xr[PH][t][1], on));
      }
    }
    dec_groups<T, PH, GAM + 1, FULL>(w, xr, cl, D, ng);
  }
}

template <int T, int PH, bool FULL>
__device__ __forceinline__ void dec_phases(const uint4 (&w)[4], const uint32_t (&xr)[T][4][2],
                                           const uint32_t (&sz)[T][2][2], const float* xgw,
                                           int ng, float (&vacc)[2][2]) {
  if constexpr (PH < T) {
    constexpr int G = 8 / T;
    const int lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
    float D[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) D[t][0] = D[t][1] = D[t][2] = D[t][3] = 0.f;
    dec_groups<T, PH, 0, FULL>(w, xr, gl % G, D, ng);
    const int gi_lane = (2 * c) % G, tau = (2 * c) / G;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int gi = PH * G + gi_lane + s;
      if (FULL || gi < ng) {
        const float cs = pos_scale(gi);
        const float X = xgw[tau * 8 + gi];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const __half2 h = *reinterpret_cast<const __half2*>(&sz[PH][s][r]);
          const float sf = __low2float(h), zf = __high2float(h);
          const float acc = (D[0][2 * r + s] + D[1][2 * r + s]) + (D[2][2 * r + s] + D[3][2 * r + s]);
          vacc[r][s] = fmaf(sf, fmaf(-zf, X, acc * cs), vacc[r][s]);
        }
      }
    }
    dec_phases<T, PH + 1, FULL>(w, xr, sz, xgw, ng, vacc);
  }
}

// This lane's codes and (scale, zero) pairs of one superblock block, copied out of the
// stage so that the stage can be refilled while the dot products run.
template <int T>
__device__ __forceinline__ void dec_load_block(const uint8_t* __restrict__ blk, uint4 (&w)[4],
                                               uint32_t (&sz)[T][2][2]) {
  constexpr int G = 8 / T;
  const int lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = reinterpret_cast<const uint4*>(blk)[q * 32 + lane];
  const uint8_t* szt = blk + kBlkCodeBytes;
  const int gi_lane = (2 * c) % G;
#pragma unroll
  for (int ph = 0; ph < T; ++ph)
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int r = 0; r < 2; ++r)
        sz[ph][s][r] = *reinterpret_cast<const uint32_t*>(szt + ((gl + 8 * r) * 8 + ph * G + gi_lane + s) * 4);
}

// The superblock partials of one unit added in a fixed order, per-token v of its 16
// columns, mask = |v| > t (union over the group's tokens) and the unit's kept columns,
// appended at out in ascending order: {column | group << 16, v per group token (0 for a
// token that drops the column)}.  Returns the number of kept columns.
template <int T>
__device__ __forceinline__ int dec_finalize(const DecodeParams& p, const float4* vpart, int nsb, const GroupDesc& gd,
                            int g, int mt, float thr, float* vbuf, int4* out) {
  constexpr int G = 8 / T;
  const int lane = threadIdx.x & 31, gl = lane >> 2, c = lane & 3;
  float v00 = 0.f, v01 = 0.f, v10 = 0.f, v11 = 0.f;
  for (int q = 0; q < nsb; ++q) {
    const float4 pv = vpart[q * 32 + lane];
    v00 += pv.x;
    v01 += pv.y;
    v10 += pv.z;
    v11 += pv.w;
  }
  float v0 = v00 + v01, v1 = v10 + v11;
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
    vbuf[gl * 2 + tau] = v0;
    vbuf[(gl + 8) * 2 + tau] = v1;
  }
  __syncwarp();
  float vv[T];
  uint32_t mbits = 0;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    vv[t] = 0.f;
    if (t < gd.n_tok && lane < 16) {
      vv[t] = vbuf[lane * 2 + t];
      if (fabsf(vv[t]) > thr) mbits |= 1u << t;
    }
  }
  __syncwarp();
  const uint32_t bal = __ballot_sync(0xffffffffu, mbits != 0);
  if (mbits) {
    const int rank = __popc(bal & ((1u << lane) - 1u));
    const float v0 = (mbits & 1u) ? vv[0] : 0.f;
    const float v1 = (T > 1 && ((mbits >> 1) & 1u)) ? vv[T > 1 ? 1 : 0] : 0.f;
    out[rank] = make_int4((mt * kMTile + lane) | (g << 16), __float_as_int(v0), __float_as_int(v1), 0);
  }
  const int cnt = __popc(bal);
  if (p.dbg_v || p.dbg_mask) {
#pragma unroll
    for (int t = 0; t < T; ++t) {
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
  return cnt;
}

// The shared-memory objects of the up phase, common to the up kernel of the two-kernel
// decode path and to the one-kernel decode layer.
struct UpShared {
  uint64_t *full, *empty;     // strip ring: [su] data landed / stage free (nsb warps)
  uint64_t *vfull, *vfree;    // unit slots: [kDecNV] partials in (nsb warps) / finalized
  int* abort;
  int* pend;                  // [kDecMaxSu] strip in flight in the stage (issue index + 1) or 0
  float (*vbuf)[16 * 2];      // [kDecNV] per-slot v staging of the finalize warps
  int* ucnt;                  // [kDecMaxUnits] kept columns of each unit
  uint8_t* ring;
  const __half* xs;
  float4* vpart;
  float* xg;
  const GroupDesc* grp;
  int4* ent;                  // [unit][16] kept columns of each unit
  size_t strip;
  int su, nsb;
  uint64_t* ufin;             // [kDecMaxUnits] single-use: unit j finalized (NULL: not signalled)
};

// Strip producer (one lane): the packed strips of units u0 .. u0 + n - 1, in order.
__device__ __forceinline__ void dec_issue_strips(const DecodeParams& p, const UpShared& S, int u0, int n, int MT) {
  const uint64_t pol = policy_evict_first();
  int s = 0, ph = 0, g = u0 / MT, mt = u0 - g * MT;
  for (int j = 0; j < n; ++j) {
    if (j >= S.su && !mbar_wait(&S.empty[s], ph ^ 1)) {
      dec_fail(p, S.abort);
      break;
    }
    if (vload(S.abort)) break;
    int el;
    const ExpertSet& es = dec_set(p, S.grp[g].expert, el);
    S.pend[s] = j + 1;
    mbar_arrive_expect_tx(&S.full[s], (uint32_t)S.strip);
    bulk_g2s(S.ring + (size_t)s * S.strip, es.up + (size_t)el * es.up_stride + (size_t)mt * S.strip,
             (uint32_t)S.strip, &S.full[s], pol);
    if (++s == S.su) {
      s = 0;
      ph ^= 1;
    }
    if (++mt == MT) {
      mt = 0;
      ++g;
    }
  }
}

// Finalize warp fl of NL: units j = fl, fl + NL, ... once all their superblock partials
// are in; the unit's kept columns go to its 16 entries, then its count is published.
template <int B>
__device__ __forceinline__ void dec_finalize_units(const DecodeParams& p, const UpShared& S, int fl, int NL,
                                                   int u0, int n, int MT) {
  const int lane = threadIdx.x & 31;
  int g = (u0 + fl) / MT, mt = (u0 + fl) - g * MT, cur_g = -1;
  float thr = 0.f;
  for (int j = fl; j < n; j += NL) {
    const int slot = j & (kDecNV - 1);
    if (!__all_sync(0xffffffffu, mbar_wait(&S.vfull[slot], (j / kDecNV) & 1))) {
      if (lane == 0) dec_fail(p, S.abort);
      break;
    }
    if (g != cur_g) {
      int el;
      const ExpertSet& es = dec_set(p, S.grp[g].expert, el);
      thr = es.thr[el];
      cur_g = g;
    }
    const int cnt = dec_finalize<B>(p, S.vpart + (size_t)slot * S.nsb * 32, S.nsb, S.grp[g], g, mt, thr,
                                    S.vbuf[slot], S.ent + (size_t)j * 16);
    __syncwarp();
    if (lane == 0) {
      // the entries before the count: the row producer of the one-kernel layer reads
      // the count without a block barrier
      __threadfence_block();
      *reinterpret_cast<volatile int*>(S.ucnt + j) = cnt;
      if (S.ufin) mbar_arrive(&S.ufin[j]);
      mbar_arrive(&S.vfree[slot]);
    }
    mt += NL;
    while (mt >= MT) {
      mt -= MT;
      ++g;
    }
  }
}

// Superblock warp (warp index uw < NL * nsb): unit lane ug = uw / nsb (units j = ug,
// ug + NL, ...), superblock sb = uw % nsb of every unit.
template <int B>
__device__ __forceinline__ void dec_up_units(const DecodeParams& p, const UpShared& S, int NL, int u0, int n,
                                             int MT) {
  const int d = p.d, lane = threadIdx.x & 31, uw = threadIdx.x >> 5;
  const int nsb = S.nsb, SU = S.su, ug = uw / nsb, sb = uw % nsb;
  const int ng = min(8, (d - sb * kSuper) / kGroup);
  float* xgw = S.xg + uw * 16;
  uint32_t xr[B][4][2];
  int cur_g = -1;
  // stage s = j % SU with full-barrier parity ph = (j / SU) & 1, and unit u = u0 + j as
  // (group g, M-tile mt), all advanced by NL units per iteration without divisions
  int s = ug % SU, ph = (ug / SU) & 1;
  int g = (u0 + ug) / MT, mt = (u0 + ug) - g * MT;
  for (int j = ug; j < n; j += NL) {
    const int slot = j & (kDecNV - 1);
    const bool ab = vload(S.abort) != 0;
    bool ok = __all_sync(0xffffffffu, !ab && mbar_wait(&S.full[s], ph));
    if (!ok) {
      if (!ab && lane == 0) dec_fail(p, S.abort);
      break;
    }
    if (g != cur_g) {
      dec_up_setup<B>(S.xs, d, S.grp[g], sb, ng, xr, xgw);
      cur_g = g;
    }
    uint4 w[4];
    uint32_t sz[B][2][2];
    dec_load_block<B>(S.ring + (size_t)s * S.strip + (size_t)sb * kBlkBytes, w, sz);
    __syncwarp();
    if (lane == 0) {
      if (sb == 0) S.pend[s] = 0;
      mbar_arrive(&S.empty[s]);  // release: the copies above are done before the stage is reused
    }
    float vacc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    if (ng == 8)
      dec_phases<B, 0, true>(w, xr, sz, xgw, ng, vacc);
    else
      dec_phases<B, 0, false>(w, xr, sz, xgw, ng, vacc);
    // the slot's previous unit must have been finalized
    if (j >= kDecNV && !__all_sync(0xffffffffu, mbar_wait(&S.vfree[slot], ((j / kDecNV) - 1) & 1))) {
      if (lane == 0) dec_fail(p, S.abort);
      break;
    }
    S.vpart[((size_t)slot * nsb + sb) * 32 + lane] = make_float4(vacc[0][0], vacc[0][1], vacc[1][0], vacc[1][1]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.vfull[slot]);
    s += NL;
    if (s >= SU) {
      s -= SU;
      ph ^= 1;
    }
    mt += NL;
    while (mt >= MT) {
      mt -= MT;
      ++g;
    }
  }
}

// The last CTA to finish: y = fp16(sum of the accumulator copies) or, for stacked
// layers, the RMSNorm y / sqrt(mean(y^2) + 1e-6) of it.  It leaves the copies zeroed
// and the finish counter reset for the next call on the workspace (every CTA's additions
// and count precede this, and the next call starts after this kernel ends).
// ss: [B][32] floats of shared memory; called by every thread of the CTA.
template <int B>
__device__ __forceinline__ void dec_last_cta(const DecodeParams& p, int nwarps, float* ss) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, d = p.d;
  float4 v[B][2];
  float sq[B];
#pragma unroll
  for (int b = 0; b < B; ++b) {
    v[b][0] = v[b][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid < d / 8) {
#pragma unroll
      for (int r = 0; r < kDecYRep; ++r) {
        float4* src = reinterpret_cast<float4*>(p.yacc + ((size_t)r * B + b) * d + tid * 8);
        const float4 a0 = __ldcg(src), a1 = __ldcg(src + 1);
        v[b][0] = make_float4(v[b][0].x + a0.x, v[b][0].y + a0.y, v[b][0].z + a0.z, v[b][0].w + a0.w);
        v[b][1] = make_float4(v[b][1].x + a1.x, v[b][1].y + a1.y, v[b][1].z + a1.z, v[b][1].w + a1.w);
        __stcg(src, make_float4(0.f, 0.f, 0.f, 0.f));
        __stcg(src + 1, make_float4(0.f, 0.f, 0.f, 0.f));
      }
    }
    const float4 v0 = v[b][0], v1 = v[b][1];
    sq[b] = ((v0.x * v0.x + v0.y * v0.y) + (v0.z * v0.z + v0.w * v0.w)) +
            ((v1.x * v1.x + v1.y * v1.y) + (v1.z * v1.z + v1.w * v1.w));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sq[b] += __shfl_xor_sync(0xffffffffu, sq[b], off);
    if (lane == 0) ss[b * 32 + warp] = sq[b];
  }
  __syncthreads();
#pragma unroll
  for (int b = 0; b < B; ++b) {
    float rinv = 1.f;
    if (p.rmsnorm) {
      float t = 0.f;
      for (int w = 0; w < nwarps; ++w) t += ss[b * 32 + w];
      rinv = rsqrtf(t / (float)d + 1e-6f);
    }
    if (tid < d / 8) {
      const float4 v0 = v[b][0], v1 = v[b][1];
      __half2* yo = reinterpret_cast<__half2*>(p.y + (size_t)b * d + tid * 8);
      yo[0] = __floats2half2_rn(v0.x * rinv, v0.y * rinv);
      yo[1] = __floats2half2_rn(v0.z * rinv, v0.w * rinv);
      yo[2] = __floats2half2_rn(v1.x * rinv, v1.y * rinv);
      yo[3] = __floats2half2_rn(v1.z * rinv, v1.w * rinv);
    }
  }
  if (tid == 0) p.ctrl->gdone = 0;
}

}  // namespace

// ---------------------------------------------------------------------------
// Up kernel.  B = tokens (1 or 2), also the group width of the tensor-core mapping.
// ---------------------------------------------------------------------------
template <int B>
__global__ void __launch_bounds__(kUpRegThreads, 1) decode_up_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t usm[];
  const int d = p.d, SU = p.su;
  const UpLayoutD L = up_layout_d(d, B, p.routed.E, SU, p.umax);
  uint64_t* full = reinterpret_cast<uint64_t*>(usm + L.off_bar);
  uint64_t* empty = full + kDecMaxSu;
  uint64_t* vfull = empty + kDecMaxSu;
  uint64_t* vfree = vfull + kDecNV;
  UpMisc* m = reinterpret_cast<UpMisc*>(usm + L.off_misc);
  uint8_t* ring = usm + L.off_ring;
  __half* xs = reinterpret_cast<__half*>(usm + L.off_x);
  float4* vpart = reinterpret_cast<float4*>(usm + L.off_vpart);
  float* xg = reinterpret_cast<float*>(usm + L.off_xg);
  GroupDesc* grp = reinterpret_cast<GroupDesc*>(usm + L.off_grp);
  float* lred = reinterpret_cast<float*>(usm + L.off_lred);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsb = L.nsb, nthreads = L.nwarps * 32;
  if (tid == 0) {
    for (int s = 0; s < SU; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nsb);
    }
    for (int v = 0; v < kDecNV; ++v) {
      mbar_init(&vfull[v], nsb);
      mbar_init(&vfree[v], 1);
    }
    fence_barrier_init();
    m->abort = 0;
    m->total = 0;
    for (int s = 0; s < kDecMaxSu; ++s) m->pend[s] = 0;
  }
  for (int j = tid; j < kDecMaxUnits; j += nthreads) m->ucnt[j] = 0;
  // the router weight is not written by the previous kernel: load this thread's rows
  // of it before waiting
  const RouteSplit rt = route_split(p.routed.E, nthreads);
  uint4 wv[kRouteRows];
  route_prefetch(p, rt, wv);
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  // the gather kernel's fp32 accumulator of y and its finish counter start at zero
  // (the previous kernel, which may be the last call's gather kernel, has finished)
  for (int i = blockIdx.x * nthreads + tid; i < kDecYRep * p.B * p.d / 4; i += gridDim.x * nthreads)
    reinterpret_cast<float4*>(p.yacc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (blockIdx.x == 0 && tid == 0) p.ctrl->gdone = 0;
  for (int i = tid; i < B * d / 8; i += nthreads)
    reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(p.x) + i);
  __syncthreads();
  dec_route<B>(p, nthreads, rt, wv, xs, lred, m, grp);
  const int G = m->G;
  if (blockIdx.x == 0) {
    for (int i = tid; i < G * (int)(sizeof(GroupDesc) / 4); i += nthreads)
      reinterpret_cast<int*>(p.groups)[i] = reinterpret_cast<const int*>(grp)[i];
    if (tid == 0) p.ctrl->G = G;
  }
  const int MT = p.f / kMTile;
  const int U = G * MT;
  const int u0 = (int)muldiv(U, blockIdx.x, gridDim.x), u1 = (int)muldiv(U, blockIdx.x + 1, gridDim.x);
  const int n = u1 - u0;

  int4* ent = reinterpret_cast<int4*>(usm + L.off_ent);  // [unit][16] kept columns
  const int NL = dec_lanes(nsb);
  const UpShared S{full, empty, vfull, vfree, &m->abort, m->pend, m->vbuf, m->ucnt, ring, xs, vpart, xg, grp,
                   ent, L.strip, SU, nsb, nullptr};
  if (warp > NL * nsb) {
    // ---- finalize warps, one per unit lane
    dec_finalize_units<B>(p, S, warp - NL * nsb - 1, NL, u0, n, MT);
  } else if (warp == NL * nsb) {
    // ---- producer warp: the strips of this CTA's units, in order
    if (lane == 0) dec_issue_strips(p, S, u0, n, MT);
  } else {
    // ---- up warps
    dec_up_units<B>(p, S, NL, u0, n, MT);
  }
  __syncthreads();
  // this CTA's list: the units' kept columns in unit order
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < n; base += 32) {
      const int c = base + lane;
      const int v = c < n ? m->ucnt[c] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (c < n) m->ucnt[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) m->total = carry;
  }
  __syncthreads();
  int4* out = p.klist + (size_t)blockIdx.x * p.kcap;
  for (int j = warp; j < n; j += L.nwarps) {
    const int o = m->ucnt[j], c = (j + 1 < n ? m->ucnt[j + 1] : m->total) - o;
    if (lane < c) out[o + lane] = ent[(size_t)j * 16 + lane];
  }
  if (tid == 0) {
    if (m->abort) {
      // wait (bounded) for the strips still in flight before the CTA exits
      for (int s = 0; s < SU; ++s) {
        const int q = m->pend[s];
        if (q > 0) (void)mbar_wait(&full[s], ((q - 1) / SU) & 1);
      }
    }
    p.cta_total[blockIdx.x] = m->total;
  }
}

// ---------------------------------------------------------------------------
// Gather kernel.  A producer warp streams the kept rows through the ring; the gather
// warps release a stage once every warp is done with its row.  A kept column whose
// gate and down rows are interleaved in one buffer costs one 4d-byte copy, else two
// 2d-byte copies.
// ---------------------------------------------------------------------------
// STAGED: the rows come from the staging area that the fetch kernel filled (host-resident
// gate/down rows) instead of from the experts; a separate build, so that the usual one
// carries no code for it.
template <int B, int MAXT, bool STAGED>
__global__ void __launch_bounds__(MAXT, 1) decode_gather_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t gsm[];
  const int d = p.d, SR = p.sr, P = gridDim.x;
  const GaLayoutD L = ga_layout_d(d, SR, p.list_cap, P);
  uint64_t* full = reinterpret_cast<uint64_t*>(gsm + L.off_bar);
  uint64_t* empty = full + kDecMaxSr;
  GaMisc* m = reinterpret_cast<GaMisc*>(gsm + L.off_misc);
  uint8_t* ring = gsm + L.off_ring;
  GaRow* list = reinterpret_cast<GaRow*>(gsm + L.off_list);
  float* red = reinterpret_cast<float*>(gsm + L.off_red);
  int* pre = reinterpret_cast<int*>(gsm + L.off_pre);
  GroupDesc* grp = reinterpret_cast<GroupDesc*>(gsm + L.off_grp);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ngw = L.ngw, nct = ngw * 32, nthreads = nct + 32;
  if (tid == 0) {
    for (int s = 0; s < SR; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ngw);
    }
    fence_barrier_init();
    m->abort = 0;
    m->issued = 0;
    m->consumed = 0;
  }
  for (int i = tid; i < 2 * kDecRows * 2 * kDecMaxGw; i += nthreads) red[i] = 0.f;
  // this thread's 8 hidden elements of the tokens, fp16 pairs (x precedes the up kernel)
  uint32_t xh[B][4];
#pragma unroll
  for (int b = 0; b < B; ++b) {
    const uint4 xv = tid < nct ? __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)b * d) + tid)
                               : make_uint4(0, 0, 0, 0);
    xh[b][0] = xv.x;
    xh[b][1] = xv.y;
    xh[b][2] = xv.z;
    xh[b][3] = xv.w;
  }
  griddep_wait();
  griddep_launch_dependents();

  // ---- prologue: this CTA's rows [a, bnd) of the kept columns in unit order.  The
  // per-CTA kept counts, the group count and the group descriptors are loaded at once.
  for (int c = tid; c < P; c += nthreads) pre[c] = __ldcg(p.cta_total + c);
  {
    const int nwords = min(p.gmax, kDecMaxG) * (int)(sizeof(GroupDesc) / 4);
    for (int i = tid; i < nwords; i += nthreads)
      reinterpret_cast<int*>(grp)[i] = __ldcg(reinterpret_cast<const int*>(p.groups) + i);
    if (tid == 0) m->G = __ldcg(&p.ctrl->G);
  }
  __syncthreads();
  if (tid < 32) {
    // exclusive prefix of the counts, in place; pre[P] = all kept columns
    int carry = 0;
    for (int base = 0; base < P; base += 32) {
      const int c = base + lane;
      const int v = c < P ? pre[c] : 0;
      int incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (c < P) pre[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pre[P] = carry;
  }
  __syncthreads();
  const int N = pre[P], G = m->G;
  const int a = (int)muldiv(N, blockIdx.x, P), bnd = (int)muldiv(N, blockIdx.x + 1, P);
  const int nrows = bnd - a;
  if (tid < G * 2) {
    const int g = tid >> 1, b = tid & 1;
    const GroupDesc& gd = grp[g];
    int t_of_b = -1;
    float w = 0.f;
    for (int t = 0; t < gd.n_tok; ++t)
      if (gd.tok[t] == b) {
        t_of_b = t;
        w = gd.w[t];
      }
    m->tmap[g][b] = t_of_b;
    m->tw[g][b] = w;
  }
  // rows [a, bnd): row r is entry r - pre[c] of up CTA c, the last c with pre[c] <= r
  for (int r = a + tid; r < bnd; r += nthreads) {
    int lo = 0, hi = P - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int4 e = __ldcg(p.klist + (size_t)lo * p.kcap + (r - pre[lo]));
    GaRow gr;
    gr.col = e.x & 0xffff;
    gr.g = e.x >> 16;
    gr.v[0] = __int_as_float(e.y);
    gr.v[1] = __int_as_float(e.z);
    list[r - a] = gr;
  }
  __syncthreads();
  if (warp == ngw) {
    // ---- producer warp: the kept rows, in order, in rounds of up to kRowLanes rows (one
    // per lane); a round is issued only once every lane has its row's stage, so the
    // issued rows stay contiguous
    const uint64_t pol = policy_evict_first();
    int s = 0, ph = 0;  // stage and parity of row i0
    for (int i0 = 0; i0 < nrows; i0 += kRowLanes) {
      const int nr = min(kRowLanes, nrows - i0);
      int sq = s + lane, pq = ph;
      if (sq >= SR) {
        sq -= SR;
        pq ^= 1;
      }
      const bool w = lane >= nr || i0 + lane < SR || mbar_wait(&empty[sq], pq ^ 1);
      if (!__all_sync(0xffffffffu, w && !vload(&m->abort))) {
        if (lane == 0) dec_fail(p, &m->abort);
        break;
      }
      if (lane < nr) {
        uint8_t* st = ring + (size_t)sq * L.row;
        if constexpr (STAGED) {
          // rows copied from host memory: row a + i of the staging area
          mbar_arrive_expect_tx(&full[sq], (uint32_t)L.row);
          bulk_g2s(st, p.staging + (size_t)(a + i0 + lane) * (4 * d), (uint32_t)(4 * d), &full[sq], pol);
        } else {
          const GaRow gr = list[i0 + lane];
          int el;
          const ExpertSet& es = dec_set(p, grp[gr.g].expert, el);
          const size_t roff = ((size_t)el * es.f + gr.col) * es.rs;
          mbar_arrive_expect_tx(&full[sq], (uint32_t)L.row);
          if (es.rs == 2 * d) {
            bulk_g2s(st, es.gate_t + roff, (uint32_t)(4 * d), &full[sq], pol);
          } else {
            bulk_g2s(st, es.gate_t + roff, (uint32_t)(2 * d), &full[sq], pol);
            bulk_g2s(st + 2 * d, es.down + roff, (uint32_t)(2 * d), &full[sq], pol);
          }
        }
      }
      if (lane == 0) m->issued = i0 + nr;
      s += nr;
      if (s >= SR) {
        s -= SR;
        ph ^= 1;
      }
    }
  } else {
  // ---- batches of up to kDecRows rows, one barrier per batch, software-pipelined:
  // all warps form the dot products of batch k and publish per-warp sums; after the
  // barrier warp 0 alone turns them into h = SiLU(.) * v * w for batch k while every
  // warp applies batch k-1 (whose h warp 0 wrote before the barrier) to its rows.
  float acc[B][8];
#pragma unroll
  for (int b = 0; b < B; ++b)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[b][e] = 0.f;
  float* hbuf = red + 2 * kDecRows * 2 * kDecMaxGw;  // [2][kDecRows][2]
  int s0 = 0, ph0 = 0;  // stage and full-barrier parity of row i0
  int prev_nb = 0;      // rows of the batch whose h warp 0 computed last
  bool stop = false;
  auto bar_or = [&](bool bad) -> bool {
    int fail;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "barrier.red.or.pred pout, 1, %2, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(fail)
        : "r"((unsigned)bad), "r"(nct)
        : "memory");
    return fail != 0;
  };
  // acc += h (batch in parity slot par) * this thread's down slices
  auto apply = [&](int par, int nbq, const uint4 (&dn)[kDecRows]) {
    const float* hb = hbuf + par * kDecRows * 2;
#pragma unroll
    for (int q = 0; q < kDecRows; ++q) {
      if (q < nbq) {
        const float2 hq = *reinterpret_cast<const float2*>(hb + q * 2);
        const float hv[2] = {hq.x, hq.y};
        const __half2* dh = reinterpret_cast<const __half2*>(&dn[q]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 df = __half22float2(dh[e]);
#pragma unroll
          for (int b = 0; b < B; ++b) {
            acc[b][2 * e] = fmaf(hv[b], df.x, acc[b][2 * e]);
            acc[b][2 * e + 1] = fmaf(hv[b], df.y, acc[b][2 * e + 1]);
          }
        }
      }
    }
  };
  auto step = [&](int i0, int bt, uint4 (&dcur)[kDecRows], const uint4 (&dprev)[kDecRows]) {
    const int nb = min(kDecRows, nrows - i0);
    int st[kDecRows];
    bool ok = !vload(&m->abort);
#pragma unroll
    for (int q = 0; q < kDecRows; ++q) {
      int sq = s0 + q, pq = ph0;
      if (sq >= SR) {
        sq -= SR;
        pq ^= 1;
      }
      st[q] = sq;
      if (q < nb) ok = ok && mbar_wait(&full[sq], pq);
    }
    s0 += kDecRows;
    if (s0 >= SR) {
      s0 -= SR;
      ph0 ^= 1;
    }
    float dot[kDecRows][B];
#pragma unroll
    for (int q = 0; q < kDecRows; ++q) {
#pragma unroll
      for (int b = 0; b < B; ++b) dot[q][b] = 0.f;
      if (q < nb && ok) {
        const uint4 gr = reinterpret_cast<const uint4*>(ring + (size_t)st[q] * L.row)[tid];
        const uint32_t gw[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
#pragma unroll
          for (int b = 0; b < B; ++b) {
            dot[q][b] = fma_f16<0, 0>(xh[b][e], gw[e], dot[q][b]);
            dot[q][b] = fma_f16<1, 1>(xh[b][e], gw[e], dot[q][b]);
          }
        }
      }
    }
    // this thread's slice of every down row, then the stages can be refilled at once
#pragma unroll
    for (int q = 0; q < kDecRows; ++q)
      dcur[q] = (q < nb && ok) ? reinterpret_cast<const uint4*>(ring + (size_t)st[q] * L.row + 2 * d)[tid]
                               : make_uint4(0, 0, 0, 0);
    __syncwarp();
    if (lane == 0)
      for (int q = 0; q < nb; ++q) mbar_arrive(&empty[st[q]]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int q = 0; q < kDecRows; ++q)
#pragma unroll
        for (int b = 0; b < B; ++b) dot[q][b] += __shfl_xor_sync(0xffffffffu, dot[q][b], off);
    float* rb = red + (size_t)(bt & 1) * kDecRows * 2 * kDecMaxGw;
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < kDecRows; ++q)
#pragma unroll
        for (int b = 0; b < B; ++b) rb[(q * 2 + b) * kDecMaxGw + warp] = dot[q][b];
    }
    if (bar_or(!ok)) {
      if (tid == 0) dec_fail(p, &m->abort);
      stop = true;
      return;
    }
    if (tid == 0) m->consumed = i0 + nb;
    // the previous batch, with the h warp 0 wrote before this barrier
    if (bt > 0) apply((bt - 1) & 1, prev_nb, dprev);
    if (warp == 0) {
      // h of this batch: lane q * 2 + b
      if (lane < kDecRows * 2) {
        const int q = lane >> 1, b = lane & 1;
        float hq = 0.f;
        if (q < nb && b < B) {
          const GaRow gr = list[i0 + q];
          const int t = m->tmap[gr.g][b];
          if (t >= 0) {
            const float4* pr = reinterpret_cast<const float4*>(rb + (q * 2 + b) * kDecMaxGw);
            const float4 p0 = pr[0], p1 = pr[1], p2 = pr[2], p3 = pr[3];  // unused slots hold 0
            float gs = (((p0.x + p0.y) + (p0.z + p0.w)) + ((p1.x + p1.y) + (p1.z + p1.w))) +
                       (((p2.x + p2.y) + (p2.z + p2.w)) + ((p3.x + p3.y) + (p3.z + p3.w)));
            if (ngw > 16) {
              const float4 p4 = pr[4], p5 = pr[5];
              gs += ((p4.x + p4.y) + (p4.z + p4.w)) + ((p5.x + p5.y) + (p5.z + p5.w));
            }
            hq = silu_fast(gs) * (t == 0 ? gr.v[0] : gr.v[1]) * m->tw[gr.g][b];
          }
        }
        hbuf[(bt & 1) * kDecRows * 2 + lane] = hq;
      }
      __syncwarp();
    }
    prev_nb = nb;
  };
  uint4 dA[kDecRows], dB[kDecRows];
  int bt = 0;
  for (int i0 = 0; i0 < nrows && !stop; i0 += 2 * kDecRows) {
    step(i0, bt++, dA, dB);
    if (!stop && i0 + kDecRows < nrows) step(i0 + kDecRows, bt++, dB, dA);
  }
  // the last batch: its h is written once warp 0 reaches the barrier
  if (!stop && bt > 0 && !bar_or(false)) apply((bt - 1) & 1, prev_nb, (bt & 1) ? dA : dB);
  // this CTA's share of y, added in fp32 into copy blockIdx.x % kDecYRep of the
  // accumulator (the order of the CTAs' additions varies)
#pragma unroll
  for (int b = 0; b < B; ++b) {
    float* dst = p.yacc + ((size_t)(blockIdx.x % kDecYRep) * B + b) * d + tid * 8;
    red_add_v4(dst, acc[b][0], acc[b][1], acc[b][2], acc[b][3]);
    red_add_v4(dst + 4, acc[b][4], acc[b][5], acc[b][6], acc[b][7]);
  }
  }
  // the last CTA to finish: y = fp16(sum) or, for stacked layers, the RMSNorm
  // y / sqrt(mean(y^2) + 1e-6) of it.  The barrier orders every thread's additions
  // before thread 0's count, an acq_rel atomic: its release publishes them, and in the
  // last CTA its acquire, followed by the barrier, orders the reads below after every
  // other CTA's additions.
  __syncthreads();
  if (tid == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(&p.ctrl->gdone) : "memory");
    m->last = old == gridDim.x - 1;
  }
  __syncthreads();
  if (m->last) dec_last_cta<B>(p, L.nwarps, red);
  if (m->abort && tid == 0) {
    // wait (bounded) for the rows still in flight before the CTA exits
    for (int i = max(m->consumed, m->issued - SR); i < m->issued; ++i)
      (void)mbar_wait(&full[i % SR], (i / SR) & 1);
  }
}

// ---------------------------------------------------------------------------
// One-kernel decode layer (d <= 4096).  The up kernel's routing and up phase, then, in
// the same CTA, the gather of exactly the kept columns of this CTA's own units: the row
// producer warp streams a unit's kept rows as soon as its finalize warp has published
// them, while the strip producer warp still streams the later units' strips, and the
// compute warps turn from superblocks to rows when their units are done.  There is no grid-wide
// step between the up projection and the gather: a CTA never waits for another one.
// Each CTA adds its share of y into the fp32 accumulator, and the last one to finish
// rounds y (after the RMSNorm of stacked layers), leaving the accumulator zeroed.
// ---------------------------------------------------------------------------
namespace {

constexpr int kHB = 4;   // gather batches in flight between the gather warps and the h warp
constexpr int kHD = 64;  // row descriptors kept for the h warp (rows ahead of it: < SR + 3 kDecRows)
static_assert(kDecMaxSr + 3 * kDecRows <= kHD, "the row producer may run kDecMaxSr + 3 kDecRows rows ahead of the h warp");

// Sums of v[q][b] over the warp's lanes by recursive halving (one value kept per lane
// and round): for one token lane 8q + i ends with row q, for two tokens lane 8q + 4b + i
// with (row q, token b).
template <int B>
__device__ __forceinline__ float warp_sum_rows(const float (&v)[kDecRows][B]) {
  static_assert(kDecRows == 4, "four rows per batch");
  const int lane = threadIdx.x & 31;
  const bool u16 = (lane & 16) != 0, u8 = (lane & 8) != 0;
  if constexpr (B == 1) {
    const float a0 = (u16 ? v[2][0] : v[0][0]) + __shfl_xor_sync(0xffffffffu, u16 ? v[0][0] : v[2][0], 16);
    const float a1 = (u16 ? v[3][0] : v[1][0]) + __shfl_xor_sync(0xffffffffu, u16 ? v[1][0] : v[3][0], 16);
    float c = (u8 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, u8 ? a0 : a1, 8);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
  } else {
    const bool u4 = (lane & 4) != 0;
    // rows (u16 ? 2 : 0) + {0, 1}, both tokens
    const float a0 = (u16 ? v[2][0] : v[0][0]) + __shfl_xor_sync(0xffffffffu, u16 ? v[0][0] : v[2][0], 16);
    const float a1 = (u16 ? v[2][1] : v[0][1]) + __shfl_xor_sync(0xffffffffu, u16 ? v[0][1] : v[2][1], 16);
    const float a2 = (u16 ? v[3][0] : v[1][0]) + __shfl_xor_sync(0xffffffffu, u16 ? v[1][0] : v[3][0], 16);
    const float a3 = (u16 ? v[3][1] : v[1][1]) + __shfl_xor_sync(0xffffffffu, u16 ? v[1][1] : v[3][1], 16);
    // row (u16 ? 2 : 0) + (u8 ? 1 : 0), both tokens
    const float c0 = (u8 ? a2 : a0) + __shfl_xor_sync(0xffffffffu, u8 ? a0 : a2, 8);
    const float c1 = (u8 ? a3 : a1) + __shfl_xor_sync(0xffffffffu, u8 ? a1 : a3, 8);
    // token u4
    float e = (u4 ? c1 : c0) + __shfl_xor_sync(0xffffffffu, u4 ? c0 : c1, 4);
    e += __shfl_xor_sync(0xffffffffu, e, 2);
    e += __shfl_xor_sync(0xffffffffu, e, 1);
    return e;
  }
}

struct LyMisc {
  int abort;
  int G;
  int last;                     // this CTA finished last
  int rissued;                  // rows issued into the row ring
  int rconsumed;                // rows whose stages the gather warps have released
  int known;                    // rows of the units finalized so far (the row producer's count)
  int allknown;                 // 1 once every unit is finalized (known is then final)
  int pend[kDecMaxSu];          // strip in flight in the stage (issue index + 1) or 0
  int tidx[2][kMaxTok];
  float tw[2][kMaxTok];
  float vbuf[kDecNV][16 * 2];
  int ucnt[kDecMaxUnits];       // kept columns of unit j once it is finalized, -1 before
  int tmap[kDecMaxG][2];        // group token of batch token b, -1 if none
  float gw[kDecMaxG][2];        // its combine weight
};

struct LyLayoutD {
  int nsb, nup, ngw, nc, nwarps, su, sr;
  size_t strip, row;
  size_t off_bar, off_misc, off_nbs, off_ring, off_rring, off_hdesc, off_x, off_vpart, off_xg, off_grp,
      off_lred, off_ent, off_red, total;
};

// warps: nc = max(up warps, gather warps) compute warps, then the strip producer, one
// finalize warp per unit lane, and the row producer.  umax: units per CTA, at most.
__host__ __device__ inline LyLayoutD ly_layout_d(int d, int B, int E, int su, int sr, int umax) {
  LyLayoutD L;
  L.nsb = n_superblocks(d);
  L.nup = dec_lanes(L.nsb) * L.nsb;
  L.ngw = d / 256;
  L.nc = L.nup > L.ngw ? L.nup : L.ngw;
  L.nwarps = L.nc + 1 + dec_lanes(L.nsb) + 1;
  L.su = su;
  L.sr = sr;
  L.strip = (size_t)L.nsb * kBlkBytes;
  L.row = (size_t)4 * d;
  size_t o = 0;
  L.off_bar = o;
  o += 8 * (size_t)(2 * kDecMaxSu + 2 * kDecNV + 2 * kDecMaxSr + 2 * kHB + 1 + kDecMaxUnits);
  o = al16(o);
  L.off_misc = o;
  o += al16(sizeof(LyMisc));
  L.off_nbs = o;
  o += al16(4 * (size_t)kHB);
  o = (o + 127) & ~(size_t)127;
  L.off_ring = o;
  o += L.strip * su;
  L.off_rring = o;
  o += L.row * sr;
  L.off_hdesc = o;
  o += 16 * (size_t)kHD;
  L.off_x = o;
  o += al16((size_t)B * d * 2);
  L.off_vpart = o;
  o += (size_t)kDecNV * L.nsb * 32 * 16;
  L.off_xg = o;
  o += (size_t)2 * L.nsb * 16 * 4;
  L.off_grp = o;
  o += al16(sizeof(GroupDesc) * kDecMaxG);
  L.off_lred = o;
  o += al16((size_t)L.nwarps * 2 * E * 4);
  L.off_ent = o;
  o += (size_t)umax * 16 * 16;
  L.off_red = o;
  o += (size_t)kHB * kDecRows * 2 * (kDecMaxGw + 1) * 4;
  L.total = o;
  return L;
}


}  // namespace

template <int B>
__global__ void __launch_bounds__(kUpRegThreads, 1) decode_layer_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t lsm[];
  const int d = p.d, SU = p.su, SR1 = p.sr;
  const LyLayoutD L = ly_layout_d(d, B, p.routed.E, SU, SR1, p.umax);
  // row ring: SR1 stages of its own, then, once every up warp is done with the strip
  // ring, as many more stages in the strip ring's space
  const int SR = min(kDecMaxSr, SR1 + (int)(L.strip * SU / L.row));
  uint64_t* full = reinterpret_cast<uint64_t*>(lsm + L.off_bar);
  uint64_t* empty = full + kDecMaxSu;
  uint64_t* vfull = empty + kDecMaxSu;
  uint64_t* vfree = vfull + kDecNV;
  uint64_t* rfull = vfree + kDecNV;
  uint64_t* rempty = rfull + kDecMaxSr;
  uint64_t* dotsb = rempty + kDecMaxSr;  // [kHB] a batch's dot partials are in (gather warps)
  uint64_t* hrdy = dotsb + kHB;          // [kHB] its h values are in (the h warp)
  uint64_t* updone = hrdy + kHB;         // every up warp is done with the strip ring
  uint64_t* ufin = updone + 1;           // [kDecMaxUnits] single-use: unit j finalized
  LyMisc* m = reinterpret_cast<LyMisc*>(lsm + L.off_misc);
  uint8_t* ring = lsm + L.off_ring;
  uint8_t* rring = lsm + L.off_rring;
  // stage s of the row ring
  auto rstage = [&](int s) -> uint8_t* {
    return s < SR1 ? rring + (size_t)s * L.row : ring + (size_t)(s - SR1) * L.row;
  };
  int4* hdesc = reinterpret_cast<int4*>(lsm + L.off_hdesc);  // [kHD] descriptor of row i at i % kHD (for the h warp)
  __half* xs = reinterpret_cast<__half*>(lsm + L.off_x);
  float4* vpart = reinterpret_cast<float4*>(lsm + L.off_vpart);
  float* xg = reinterpret_cast<float*>(lsm + L.off_xg);
  GroupDesc* grp = reinterpret_cast<GroupDesc*>(lsm + L.off_grp);
  float* lred = reinterpret_cast<float*>(lsm + L.off_lred);
  int4* ent = reinterpret_cast<int4*>(lsm + L.off_ent);
  float* red = reinterpret_cast<float*>(lsm + L.off_red);
  float* part = red;                                       // [kHB][kDecRows][2][kDecMaxGw] dot partials
  float* hbuf = red + kHB * kDecRows * 2 * kDecMaxGw;      // [kHB][kDecRows][2] h values
  int* nbs = reinterpret_cast<int*>(lsm + L.off_nbs);      // [kHB] rows of a batch
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsb = L.nsb, NL = dec_lanes(nsb), nup = L.nup, ngw = L.ngw, NC = L.nc;
  const int nthreads = L.nwarps * 32, nct = ngw * 32;
  if (tid == 0) {
    for (int s = 0; s < SU; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nsb);
    }
    for (int v = 0; v < kDecNV; ++v) {
      mbar_init(&vfull[v], nsb);
      mbar_init(&vfree[v], 1);
    }
    for (int s = 0; s < SR; ++s) {
      mbar_init(&rfull[s], 1);
      mbar_init(&rempty[s], ngw);
    }
    for (int h = 0; h < kHB; ++h) {
      mbar_init(&dotsb[h], ngw);
      mbar_init(&hrdy[h], 1);
    }
    mbar_init(updone, nup);
    fence_barrier_init();
    m->abort = 0;
    m->rissued = 0;
    m->rconsumed = 0;
    m->known = 0;
    m->allknown = 0;
    for (int s = 0; s < kDecMaxSu; ++s) m->pend[s] = 0;
  }
  for (int j = tid; j < kDecMaxUnits; j += nthreads) {
    m->ucnt[j] = -1;
    mbar_init(&ufin[j], 1);
  }
  if (tid < kDecMaxUnits) fence_barrier_init();
  for (int i = tid; i < kHB * kDecRows * 2 * (kDecMaxGw + 1); i += nthreads) red[i] = 0.f;
  // the router weight is not written by the previous kernel: load this thread's rows
  // of it before waiting
  const RouteSplit rt = route_split(p.routed.E, nthreads);
  uint4 wv[kRouteRows];
  route_prefetch(p, rt, wv);
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  for (int i = tid; i < B * d / 8; i += nthreads)
    reinterpret_cast<uint4*>(xs)[i] = __ldg(reinterpret_cast<const uint4*>(p.x) + i);
  __syncthreads();
  dec_route<B>(p, nthreads, rt, wv, xs, lred, m, grp);
  const int G = m->G;
  if (tid < G * 2) {
    const int g = tid >> 1, b = tid & 1;
    const GroupDesc& gd = grp[g];
    int t_of_b = -1;
    float w = 0.f;
    for (int t = 0; t < gd.n_tok; ++t)
      if (gd.tok[t] == b) {
        t_of_b = t;
        w = gd.w[t];
      }
    m->tmap[g][b] = t_of_b;
    m->gw[g][b] = w;
  }
  __syncthreads();
  const int MT = p.f / kMTile;
  const int U = G * MT;
  const int u0 = (int)muldiv(U, blockIdx.x, gridDim.x), u1 = (int)muldiv(U, blockIdx.x + 1, gridDim.x);
  const int n = u1 - u0;
  const UpShared S{full, empty, vfull, vfree, &m->abort, m->pend, m->vbuf, m->ucnt, ring, xs, vpart, xg, grp,
                   ent, L.strip, SU, nsb, ufin};

  if (warp == NC) {
    // ---- strip producer: the packed strips of this CTA's units, in order
    if (lane == 0) dec_issue_strips(p, S, u0, n, MT);
  } else if (warp == NC + NL + 1) {
    // ---- row producer: the kept rows of each unit once its finalize warp has published
    // them, in unit order.  It first adds the unit's rows to the known count (the gather
    // warps size their batches by it), and sets allknown after the last unit.  A stage's
    // first use: its own stages at once, those in the strip ring's space once the up phase
    // is over; later uses: once the gather warps have released it.  Rows go out in rounds
    // of up to kRowLanes, one per lane: every lane waits for its row's stage, and the round
    // is issued only if all of them got theirs, so the issued rows stay contiguous.
    const uint64_t pol = policy_evict_first();
    int rs = 0, rph = 0, issued = 0, known = 0;  // stage and parity of row `issued`
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&ufin[j], 0))) {
        ok = false;
        break;
      }
      const int c = m->ucnt[j];
      if (c == 0) continue;
      known += c;
      if (lane == 0) *reinterpret_cast<volatile int*>(&m->known) = known;
      // the unit's expert rows (every entry of a unit has the same group)
      const int g = ent[j * 16].x >> 16;
      int el;
      const ExpertSet& es = dec_set(p, grp[g].expert, el);
      const size_t rsb = (size_t)es.rs * 2;
      const uint8_t* gbase = reinterpret_cast<const uint8_t*>(es.gate_t + (size_t)el * es.f * es.rs);
      const uint8_t* dbase = reinterpret_cast<const uint8_t*>(es.down + (size_t)el * es.f * es.rs);
      const bool inter = es.rs == 2 * d;
      for (int r0 = 0; r0 < c; r0 += kRowLanes) {
        const int nr = min(kRowLanes, c - r0);
        int sq = rs + lane, pq = rph;  // this lane's row issued + lane
        if (sq >= SR) {
          sq -= SR;
          pq ^= 1;
        }
        bool w = true;
        if (lane < nr) w = issued + lane >= SR ? mbar_wait(&rempty[sq], pq ^ 1) : (sq < SR1 || mbar_wait(updone, 0));
        if (!__all_sync(0xffffffffu, w && !vload(&m->abort))) {
          ok = false;
          break;
        }
        if (lane < nr) {
          const int4 e = ent[j * 16 + r0 + lane];
          const size_t off = (size_t)(e.x & 0xffff) * rsb;
          uint8_t* st = rstage(sq);
          hdesc[(issued + lane) & (kHD - 1)] = e;
          mbar_arrive_expect_tx(&rfull[sq], (uint32_t)L.row);
          if (inter) {
            bulk_g2s(st, gbase + off, (uint32_t)(4 * d), &rfull[sq], pol);
          } else {
            bulk_g2s(st, gbase + off, (uint32_t)(2 * d), &rfull[sq], pol);
            bulk_g2s(st + 2 * d, dbase + off, (uint32_t)(2 * d), &rfull[sq], pol);
          }
        }
        issued += nr;
        rs += nr;
        if (rs >= SR) {
          rs -= SR;
          rph ^= 1;
        }
      }
    }
    if (lane == 0) {
      m->rissued = issued;
      if (ok) {
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&m->allknown) = 1;
        // end marker: a plain arrival on the stage of row `issued` (no row comes there), so
        // that a gather warp waiting for that row wakes and sees allknown; the stage's
        // previous row must have been consumed first, as for a row
        if (issued >= SR && !mbar_wait(&rempty[rs], rph ^ 1))
          ok = false;
        else
          mbar_arrive(&rfull[rs]);
      }
      if (!ok) dec_fail(p, &m->abort);
    }
  } else if (warp > NC) {
    // ---- finalize warps, one per unit lane; then the first one forms the gather's h
    dec_finalize_units<B>(p, S, warp - NC - 1, NL, u0, n, MT);
    if (warp == NC + 1) {
      // batch k (rows 4k ..): sum the gather warps' dot partials of each (row, token), then
      // h = SiLU(sum) * v * router weight, for lane q * 2 + b; rows past the batch's count
      // get h = 0
      for (int k = 0;; ++k) {
        const int hs = k & (kHB - 1);
        if (!__all_sync(0xffffffffu, !vload(&m->abort) && mbar_wait(&dotsb[hs], (k / kHB) & 1))) break;
        const int nbw = vload(&nbs[hs]);
        const int nb = nbw & 0xff;
        if (lane < kDecRows * 2) {
          const int q = lane >> 1, b = lane & 1;
          float hq = 0.f;
          if (q < nb && b < B) {
            const int4 e = hdesc[(k * kDecRows + q) & (kHD - 1)];
            const int g = e.x >> 16;
            const int t = m->tmap[g][b];
            if (t >= 0) {
              const float4* pr = reinterpret_cast<const float4*>(part + ((hs * kDecRows + q) * 2 + b) * kDecMaxGw);
              const float4 p0 = pr[0], p1 = pr[1], p2 = pr[2], p3 = pr[3];  // unused slots hold 0
              float gs = (((p0.x + p0.y) + (p0.z + p0.w)) + ((p1.x + p1.y) + (p1.z + p1.w))) +
                         (((p2.x + p2.y) + (p2.z + p2.w)) + ((p3.x + p3.y) + (p3.z + p3.w)));
              if (ngw > 16) {
                const float4 p4 = pr[4], p5 = pr[5];
                gs += ((p4.x + p4.y) + (p4.z + p4.w)) + ((p5.x + p5.y) + (p5.z + p5.w));
              }
              hq = silu_fast(gs) * __int_as_float(t == 0 ? e.y : e.z) * m->gw[g][b];
            }
          }
          hbuf[hs * kDecRows * 2 + lane] = hq;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hrdy[hs]);
        if (nbw & 0x100) break;  // the last batch
      }
    }
  } else {
    // ---- compute warps: the superblocks of this CTA's units, then its kept rows
    if (warp < nup) {
      dec_up_units<B>(p, S, NL, u0, n, MT);
      __syncwarp();
      if (lane == 0) mbar_arrive(updone);
    }
    if (warp < ngw) {
      float acc[B][8];
#pragma unroll
      for (int b = 0; b < B; ++b)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[b][e] = 0.f;
      // this thread's 8 hidden elements of the tokens, fp16 pairs
      uint32_t xh[B][4];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const uint4 xv = reinterpret_cast<const uint4*>(xs + (size_t)b * d)[tid];
        xh[b][0] = xv.x;
        xh[b][1] = xv.y;
        xh[b][2] = xv.z;
        xh[b][3] = xv.w;
      }
      int s0 = 0, ph0 = 0;  // stage and full-barrier parity of the batch's first row
      int cons = 0;         // rows consumed
      // acc += h of batch k * this thread's slices of its down rows (all four: rows past a
      // batch's count have h = 0 and zero slices), once the h warp has published that h
      auto apply = [&](int k, const uint4 (&dn)[kDecRows]) -> bool {
        const int hs = k & (kHB - 1);
        if (!__all_sync(0xffffffffu, mbar_wait(&hrdy[hs], (k / kHB) & 1))) return false;
        const float* hb = hbuf + hs * kDecRows * 2;
#pragma unroll
        for (int q = 0; q < kDecRows; ++q) {
          const float2 hq = *reinterpret_cast<const float2*>(hb + q * 2);
          const float hv[2] = {hq.x, hq.y};
          const __half2* dh = reinterpret_cast<const __half2*>(&dn[q]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 df = __half22float2(dh[e]);
#pragma unroll
            for (int b = 0; b < B; ++b) {
              acc[b][2 * e] = fmaf(hv[b], df.x, acc[b][2 * e]);
              acc[b][2 * e + 1] = fmaf(hv[b], df.y, acc[b][2 * e + 1]);
            }
          }
        }
        return true;
      };
      // batch k: kDecRows rows when that many more are known, else (once every unit is
      // finalized) the remaining 0 .. kDecRows - 1 rows as the last batch.  Dot partials of
      // this warp into slot k % kHB, then the previous batch applied; no warp waits for
      // another one.  Returns the batch's rows plus 0x100 for the last batch, or -1.
      auto step = [&](auto full_t, int k, int nb, uint4 (&dcur)[kDecRows], const uint4 (&dprev)[kDecRows]) -> int {
        constexpr bool FULLB = decltype(full_t)::value;
        const int hs = k & (kHB - 1);
        int st[kDecRows];
        bool ok = true;
#pragma unroll
        for (int q = 0; q < kDecRows; ++q) {
          int sq = s0 + q, pq = ph0;
          if (sq >= SR) {
            sq -= SR;
            pq ^= 1;
          }
          st[q] = sq;
          if (FULLB || q < nb) ok = mbar_wait(&rfull[sq], pq) && ok;
        }
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) {
            dec_fail(p, &m->abort);
            mbar_arrive(&dotsb[hs]);
          }
          return -1;
        }
        if (warp == 0 && lane == 0) nbs[hs] = FULLB ? kDecRows : (nb | 0x100);
        float dot[kDecRows][B];
#pragma unroll
        for (int q = 0; q < kDecRows; ++q) {
#pragma unroll
          for (int b = 0; b < B; ++b) dot[q][b] = 0.f;
          if (FULLB || q < nb) {
            const uint4 gr = reinterpret_cast<const uint4*>(rstage(st[q]))[tid];
            const uint32_t gw4[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
#pragma unroll
              for (int b = 0; b < B; ++b) {
                dot[q][b] = fma_f16<0, 0>(xh[b][e], gw4[e], dot[q][b]);
                dot[q][b] = fma_f16<1, 1>(xh[b][e], gw4[e], dot[q][b]);
              }
            }
          }
        }
        // this thread's slice of every down row, then the stages can be refilled at once
#pragma unroll
        for (int q = 0; q < kDecRows; ++q)
          dcur[q] = (FULLB || q < nb) ? reinterpret_cast<const uint4*>(rstage(st[q]) + 2 * d)[tid]
                                      : make_uint4(0, 0, 0, 0);
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < kDecRows; ++q)
            if (FULLB || q < nb) mbar_arrive(&rempty[st[q]]);
        }
        // the warp's sums by recursive halving: lane 8q (+ 4b for two tokens) ends with
        // (row q, token b)
        const float r = warp_sum_rows<B>(dot);
        if ((lane & (B == 1 ? 7 : 3)) == 0) {
          const int q = lane >> 3, b = B == 1 ? 0 : (lane >> 2) & 1;
          part[((hs * kDecRows + q) * 2 + b) * kDecMaxGw + warp] = r;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&dotsb[hs]);
        if (k > 0 && !apply(k - 1, dprev)) {
          if (lane == 0) dec_fail(p, &m->abort);
          return -1;
        }
        s0 += FULLB ? kDecRows : nb;
        if (s0 >= SR) {
          s0 -= SR;
          ph0 ^= 1;
        }
        cons += FULLB ? kDecRows : nb;
        return FULLB ? kDecRows : (nb | 0x100);
      };
      // rows of the next batch: kDecRows if known, else the rest once all are known.  While
      // neither, wait for row kn (the first one not known yet) to land: the row producer
      // publishes a unit's count before issuing its rows, and after the last unit it puts
      // an end marker on the stage of the row past the last one.
      auto next_rows = [&]() -> int {
        for (uint32_t tries = 0;; ++tries) {
          int ak = 0, kn = 0;
          if (lane == 0) {
            ak = vload(&m->allknown);
            __threadfence_block();
            kn = vload(&m->known);
          }
          ak = __shfl_sync(0xffffffffu, ak, 0);
          kn = __shfl_sync(0xffffffffu, kn, 0);
          if (kn - cons >= kDecRows) return kDecRows;
          if (ak) return kn - cons;
          if (__any_sync(0xffffffffu, vload(&m->abort)) || tries > (uint32_t)kDecMaxUnits * 16) return -1;
          int sq = s0 + (kn - cons), pq = ph0;
          if (sq >= SR) {
            sq -= SR;
            pq ^= 1;
          }
          if (!__all_sync(0xffffffffu, mbar_wait(&rfull[sq], pq))) return -1;
        }
      };
      uint4 dA[kDecRows], dB[kDecRows];
      int k = 0, res = 0;
      const std::integral_constant<bool, true> kFull;
      const std::integral_constant<bool, false> kPart;
      for (;;) {
        int nb = next_rows();
        if (nb < 0) {
          res = -1;
          if (lane == 0) dec_fail(p, &m->abort);
          break;
        }
        res = nb == kDecRows ? step(kFull, k, nb, dA, dB) : step(kPart, k, nb, dA, dB);
        if (res < 0) break;
        ++k;
        if (res & 0x100) break;
        nb = next_rows();
        if (nb < 0) {
          res = -1;
          if (lane == 0) dec_fail(p, &m->abort);
          break;
        }
        res = nb == kDecRows ? step(kFull, k, nb, dB, dA) : step(kPart, k, nb, dB, dA);
        if (res < 0) break;
        ++k;
        if (res & 0x100) break;
      }
      // the last batch (k - 1), whose rows' down slices are in dA if k - 1 is even
      if (res >= 0 && !apply(k - 1, ((k - 1) & 1) ? dB : dA) && lane == 0) dec_fail(p, &m->abort);
      if (tid == 0) m->rconsumed = cons;
      // this CTA's share of y, added in fp32 into copy blockIdx.x % kDecYRep of the
      // accumulator (the order of the CTAs' additions varies)
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float* dst = p.yacc + ((size_t)(blockIdx.x % kDecYRep) * B + b) * d + tid * 8;
        red_add_v4(dst, acc[b][0], acc[b][1], acc[b][2], acc[b][3]);
        red_add_v4(dst + 4, acc[b][4], acc[b][5], acc[b][6], acc[b][7]);
      }
    }
  }
  // the last CTA to finish rounds y: the barrier orders every thread's additions before
  // thread 0's count, an acq_rel atomic whose release publishes them; in the last CTA its
  // acquire, followed by the barrier, orders the reads after every other CTA's additions
  __syncthreads();
  if (tid == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(&p.ctrl->gdone) : "memory");
    m->last = old == gridDim.x - 1;
  }
  __syncthreads();
  if (m->last) dec_last_cta<B>(p, L.nwarps, red);
  if (m->abort && tid == 0) {
    // wait (bounded) for the strips and rows still in flight before the CTA exits
    for (int s = 0; s < SU; ++s) {
      const int q = m->pend[s];
      if (q > 0) (void)mbar_wait(&full[s], ((q - 1) / SU) & 1);
    }
    for (int i = max(m->rconsumed, m->rissued - SR); i < m->rissued; ++i)
      (void)mbar_wait(&rfull[i % SR], (i / SR) & 1);
  }
}

bool decode_supported(int B, int d, int f, int E, int k, int n_shared, int P) {
  // the in-kernel router splits the experts into 1, 2, 4 or 8 chunks of 8
  if (!(B >= 1 && B <= 2 && d <= kDecMaxD && d % 256 == 0 && (E == 8 || E == 16 || E == 32 || E == 64) &&
        k <= kMaxTok && B * k + n_shared <= kDecMaxG && n_shared <= 8 && P >= 1))
    return false;
  const long long units = (long long)(B * k + n_shared) * (f / kMTile);
  return (units + P - 1) / P <= kDecMaxUnits;
}

int decode_units_max(int B, int f, int k, int n_shared, int P) {
  const long long units = (long long)(B * k + n_shared) * (f / kMTile);
  return (int)((units + P - 1) / P);
}

int decode_list_cap(int B, int f, int k, int n_shared, int P) {
  const long long rows = (long long)(B * k + n_shared) * f;
  return (int)((rows + P - 1) / P) + 1;
}

int decode_plan(int B, int d, int E, int umax, int list_cap, int P, int smem_optin, int& su, int& sr) {
  su = sr = 0;
  const UpLayoutD u0 = up_layout_d(d, B, E, 0, umax);
  const size_t strip = u0.strip;
  size_t fixed = u0.total - al16(u0.ring);
  int s = (int)(((size_t)smem_optin - fixed - 256) / strip);
  if (s > kDecMaxSu) s = kDecMaxSu;
  // a multiple of the unit lanes: stage s then only ever holds strips of lane s % lanes,
  // so a warp's wait on a stage is always for the phase after the one it last waited for
  // (a parity wait cannot tell a phase from the one two back)
  s -= s % dec_lanes(u0.nsb);
  if (s < 2 || up_layout_d(d, B, E, s, umax).total > (size_t)smem_optin) return 0;
  su = s;
  const GaLayoutD g0 = ga_layout_d(d, 0, list_cap, P);
  const size_t row = (size_t)4 * d;
  if (g0.total + 4 * row > (size_t)smem_optin) return 0;
  int r = (int)(((size_t)smem_optin - g0.total) / row);
  sr = r > kDecMaxSr ? kDecMaxSr : r;
  return 1;
}

size_t decode_up_smem(const DecodeParams& p) { return up_layout_d(p.d, p.B, p.routed.E, p.su, p.umax).total; }
size_t decode_gather_smem(const DecodeParams& p) { return ga_layout_d(p.d, p.sr, p.list_cap, p.P).total; }

static cudaLaunchConfig_t pdl_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                  cudaLaunchAttribute* attr, bool pdl) {
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

cudaError_t launch_decode_up(const DecodeParams& p, cudaStream_t st, bool pdl) {
  const UpLayoutD L = up_layout_d(p.d, p.B, p.routed.E, p.su, p.umax);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3(p.P), dim3(L.nwarps * 32), L.total, st, attr, pdl);
  const void* fn = p.B == 1 ? (const void*)decode_up_kernel<1> : (const void*)decode_up_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
  if (e != cudaSuccess) return e;
  if (p.B == 1) return cudaLaunchKernelEx(&cfg, decode_up_kernel<1>, p);
  return cudaLaunchKernelEx(&cfg, decode_up_kernel<2>, p);
}

template <int B, int MAXT, bool STAGED>
static cudaError_t launch_ga(cudaLaunchConfig_t& cfg, const DecodeParams& p, size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(decode_gather_kernel<B, MAXT, STAGED>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_gather_kernel<B, MAXT, STAGED>, p);
}

template <int B, int MAXT>
static cudaError_t launch_ga(cudaLaunchConfig_t& cfg, const DecodeParams& p, size_t smem) {
  return p.staging ? launch_ga<B, MAXT, true>(cfg, p, smem) : launch_ga<B, MAXT, false>(cfg, p, smem);
}

cudaError_t launch_decode_gather(const DecodeParams& p, cudaStream_t st, bool pdl) {
  const GaLayoutD L = ga_layout_d(p.d, p.sr, p.list_cap, p.P);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3(p.P), dim3(L.nwarps * 32), L.total, st, attr, pdl);
  // d <= 4096: at most 17 warps (96 registers per thread); above, up to 25 warps
  if (L.nwarps * 32 <= kGaSmallThreads)
    return p.B == 1 ? launch_ga<1, kGaSmallThreads>(cfg, p, L.total) : launch_ga<2, kGaSmallThreads>(cfg, p, L.total);
  return p.B == 1 ? launch_ga<1, kGaThreads>(cfg, p, L.total) : launch_ga<2, kGaThreads>(cfg, p, L.total);
}

// ring space of the one-kernel layer given to the strips, in tenths; own row stages, at least
constexpr int kLyStripShare = 4;
constexpr int kLyMinRowStages = kDecRows + 2;

int decode_layer_plan(int B, int d, int E, int umax, int smem_optin, int& su, int& sr) {
  su = sr = 0;
  // one token, d <= 4096.  Two tokens take the two-kernel path: their up phase is twice
  // as long, and the gather kernel's globally balanced rows then win (Mixtral-8x7B at
  // 70 %: 85.6 against 96.3 us per layer)
  if (d > 4096 || B != 1) return 0;
  const LyLayoutD z = ly_layout_d(d, B, E, 0, 0, umax);
  if (z.nwarps * 32 > kUpRegThreads || z.total + 1024 > (size_t)smem_optin) return 0;
  const size_t budget = (size_t)smem_optin - z.total - 256;
  // strips: about 40 % of the ring space, rounded up to a multiple of the unit lanes (stage
  // s then only ever holds strips of lane s % lanes, so a warp's wait on a stage is always
  // for the phase after the one it last waited for: a parity wait cannot tell a phase from
  // the one two back); rows: the rest
  const int NL = dec_lanes(z.nsb);
  int s = (int)(budget * kLyStripShare / 10 / z.strip);
  s += (NL - s % NL) % NL;
  if (s < 2 * NL) s = 2 * NL;
  if (s > kDecMaxSu) s = kDecMaxSu - kDecMaxSu % NL;
  if ((size_t)s * z.strip >= budget) return 0;
  int r = (int)((budget - (size_t)s * z.strip) / z.row);
  if (r > kDecMaxSr) r = kDecMaxSr;
  if (r < kLyMinRowStages) return 0;
  if (ly_layout_d(d, B, E, s, r, umax).total > (size_t)smem_optin) return 0;
  su = s;
  sr = r;
  return 1;
}

size_t decode_layer_smem(const DecodeParams& p) {
  return ly_layout_d(p.d, p.B, p.routed.E, p.su, p.sr, p.umax).total;
}

cudaError_t launch_decode_layer(const DecodeParams& p, cudaStream_t st, bool pdl) {
  const LyLayoutD L = ly_layout_d(p.d, p.B, p.routed.E, p.su, p.sr, p.umax);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_cfg(dim3(p.P), dim3(L.nwarps * 32), L.total, st, attr, pdl);
  if (p.B != 1) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute((const void*)decode_layer_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L.total);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<1>, p);
}

}  // namespace sesg
