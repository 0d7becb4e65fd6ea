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
// (TMA).  The consumer warps own interleaved 16-byte chunks of the hidden dimension;
// per group segment they hold the group's x (fp32) and its output accumulators in
// registers.  Items go in batches (one barrier per batch): every warp forms the
// partial dot products x . gate of a batch (packed fp32 FMAs, one recursive-halving
// warp reduction for all items and tokens), warp 0 turns the per-warp sums into
// h = SiLU(.) * v * (router weight) while the others apply the previous batch,
// acc += h * down.  At the end of a segment the accumulators are this CTA's partial
// output of the group; the combine kernel adds the partials.
#include "params.cuh"

namespace sesg {

constexpr int kChunk = 8;  // fp16 elements per 16-byte chunk

struct GatherLayout {
  size_t off_full, off_empty, off_stage, off_lslot, off_lcol, off_lgrp, off_red, off_hbuf, off_goff,
      off_x, off_h16, total, stage_bytes;
};

// Tensor-core consumers (groups of up to 8 tokens, d <= 4096): the group's x in shared
// memory, 4 or 8 rows (the group size bound) of d + 8 halves (the padding spreads the
// rows over the banks).
constexpr int kMmaTok = 8;
constexpr int kMmaBatch = 4;  // kept rows per batch
__host__ __device__ inline bool gather_mma(int d, int nt) { return d <= 4096 && nt >= 2; }
__host__ __device__ inline int gather_mma_xrows(int nt) { return nt <= 4 ? 4 : 8; }

// Scratch of the prologue inside the (then idle) stage ring: the tile counts of one
// group [MT + 1] and the block scan's [threads + 1].
__host__ __device__ inline size_t gather_scan_tmp_off(int MT) { return ((size_t)(MT + 1) * 4 + 15) & ~(size_t)15; }
__host__ __device__ inline size_t gather_scan_bytes(int MT, int threads) {
  return gather_scan_tmp_off(MT) + (size_t)(threads + 1) * 4;
}


constexpr int kGaBatchTok = 16;  // items per batch x tokens per group, at most

// Two 8x8 fp16 matrices from shared memory (rows given by lanes 0-7 and 8-15), as
// mma operand fragments; .trans delivers them transposed.
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(addr));
}

// Warp sums of V values (V a power of two <= 32) by recursive halving: at each of the
// first log2(V) levels every lane keeps half of its values and adds its partner's copy
// of them; the last levels add the one remaining value.  Returns the sum of value
// `idx` over the 32 lanes, where idx is set from the lane's bits 4, 3, ... .
template <int V>
__device__ __forceinline__ float warp_sum_halving(float (&a)[V], int lane, int& idx) {
  idx = 0;
  int cnt = V;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (cnt > 1) {
      const int h = cnt / 2;
      const bool up = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < h && i < V / 2; ++i)
        a[i] = (up ? a[i + h] : a[i]) + __shfl_xor_sync(0xffffffffu, up ? a[i] : a[i + h], off);
      if (up) idx += h;
      cnt = h;
    } else {
      a[0] += __shfl_xor_sync(0xffffffffu, a[0], off);
    }
  }
  return a[0];
}

__host__ __device__ inline GatherLayout gather_layout(int d, int stages, int nt, int list_cap,
                                                      int g_max) {
  GatherLayout L;
  const int ncw = d / 256;
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
  o = (o + 15) & ~(size_t)15;
  L.off_red = o;  // [2][items][tokens][consumer warps] partial dot products
  o += (size_t)2 * kGaBatchTok * ncw * 4;
  o = (o + 15) & ~(size_t)15;
  L.off_hbuf = o;  // [2][items][tokens] h of a batch
  o += (size_t)2 * kGaBatchTok * 4;
  L.off_goff = o;  // kept-item offsets of the groups [G_max + 1]
  o += ((size_t)g_max + 1) * 4;
  o = (o + 127) & ~(size_t)127;
  L.off_x = L.off_h16 = o;
  if (gather_mma(d, nt)) {
    L.off_x = o;  // [4 or 8][d + 8] fp16
    o += (size_t)gather_mma_xrows(nt) * (d + 8) * 2;
    o = (o + 127) & ~(size_t)127;
    L.off_h16 = o;  // [8 tokens][16 k] fp16: k = row (hi), 4 + row (lo), 8..15 zero
    o += (size_t)kMmaTok * 16 * 2;
  }
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

template <int NT, int MAXT, bool MMA>
__global__ void __launch_bounds__(MAXT, 1) gather_kernel(ExpertParams p) {
  extern __shared__ __align__(128) uint8_t gsm[];
  // items per batch (one barrier per batch), within the register budget
  constexpr int kR = NT >= 4 ? 2 : (MAXT > 640 && NT == 2) ? 2 : 4;
  static_assert(MMA || kR * NT <= kGaBatchTok, "batch buffers");
  const int d = p.d;
  const int ncw = d / 256;   // consumer warps
  const int nct = ncw * 32;  // consumer threads
  const int S = p.stages;
  const GatherLayout L = gather_layout(d, S, NT, p.list_cap, p.G_max);
  uint64_t* full = reinterpret_cast<uint64_t*>(gsm + L.off_full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(gsm + L.off_empty);
  uint8_t* stage = gsm + L.off_stage;
  int* lslot = reinterpret_cast<int*>(gsm + L.off_lslot);
  int* lcol = reinterpret_cast<int*>(gsm + L.off_lcol);
  int* lgrp = reinterpret_cast<int*>(gsm + L.off_lgrp);
  float* red = reinterpret_cast<float*>(gsm + L.off_red);    // [2][kR][NT][ncw] partial dots
  float* hbuf = reinterpret_cast<float*>(gsm + L.off_hbuf);  // [2][kR][NT]
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

  // ---- prologue: this CTA's range of the global kept-item order (group, M-tile, column)
  const int G = *reinterpret_cast<volatile int*>(&p.ctrl->G);
  const int MT = p.f / kMTile;
  int* goff = reinterpret_cast<int*>(gsm + L.off_goff);  // [G+1]
  int* uoff = reinterpret_cast<int*>(stage);  // scratch in the idle stage ring: [MT+1]
  int* tmp = reinterpret_cast<int*>(stage + gather_scan_tmp_off(MT));  // [threads + 1]
  for (int g = tid; g < G; g += blockDim.x) goff[g] = __ldcg(p.group_total + g);
  __syncthreads();
  block_exclusive_scan(goff, G, tmp);
  const long long N = goff[G];
  if (blockIdx.x == 0 && tid == 0) p.ctrl->N = (int)N;
  const int a = (int)(N * blockIdx.x / p.P3), b = (int)(N * (blockIdx.x + 1) / p.P3);

  // ring positions: the producer's next stage and the consumers' next stage, each with
  // its barrier parity, advanced one item at a time (no divisions in the loops)
  int ps = 0, pph = 0, cs = 0, cph = 0;
  float2 acc[MMA ? 1 : NT][kChunk / 2];
  float2 xf[MMA ? 1 : NT][kChunk / 2];
  float wt[MMA ? 1 : NT];
  if constexpr (MMA) {
    // the h buffer's k = 8..15 stay zero
    __half* h16 = reinterpret_cast<__half*>(gsm + L.off_h16);
    for (int i = tid; i < kMmaTok * 16; i += blockDim.x) h16[i] = __float2half(0.f);
    __syncthreads();
  }

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
      if (lane == 0) {
        const uint64_t pol = policy_evict_first();
        int last_g = -1;
        const __half* gbase_ptr = nullptr;
        const __half* dbase_ptr = nullptr;
        int row_stride = d;
        for (int i = 0; i < n; ++i) {
          if (base + i >= S && !mbar_wait(&empty[ps], pph ^ 1)) {
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
          uint8_t* st = stage + (size_t)ps * L.stage_bytes;
          mbar_arrive_expect_tx(&full[ps], (uint32_t)(4 * d + 32));
          if (row_stride == 2 * d) {
            bulk_g2s(st, gbase_ptr + roff, (uint32_t)(4 * d), &full[ps], pol);
          } else {
            bulk_g2s(st, gbase_ptr + roff, (uint32_t)(2 * d), &full[ps], pol);
            bulk_g2s(st + 2 * d, dbase_ptr + roff, (uint32_t)(2 * d), &full[ps], pol);
          }
          bulk_g2s(st + 4 * d, p.item_v + (size_t)lslot[i] * 8, 32u, &full[ps], pol);
          s_issued = base + i + 1;
          if (++ps == S) {
            ps = 0;
            pph ^= 1;
          }
        }
      }
    } else if constexpr (MMA) {
      // ---- consumers on the tensor cores, for groups of up to 8 tokens.  Warp w owns
      // the hidden slice [256 w, 256 w + 256).  Per batch of up to 4 kept rows:
      //   dots   D[row][token] += G[row][k] . X[k][token]: mma.m16n8k16 with the gate
      //          rows as A (ldmatrix from the stages; rows 4..15 absent) and the group's x
      //          as B (shared memory), 16 k-steps over the warp's slice;
      //   h      warp 0 adds the 16 warps' partial dots, h = SiLU(.) * v * w, split into
      //          fp16 hi + lo (hi + lo carries h to about 22 bits);
      //   down   acc[col][token] += Down^T[col][k] . H[k][token] with k = 0..3 the batch's
      //          rows times hi and k = 4..7 the same rows times lo: ldmatrix.trans of the
      //          down rows as A (lanes 4..7 address rows 0..3 again), one mma per 16
      //          columns.
      __half* xs = reinterpret_cast<__half*>(gsm + L.off_x);
      __half* h16 = reinterpret_cast<__half*>(gsm + L.off_h16);  // [8 tokens][16 k]
      float* redm = red;  // [ncw][4 rows][8 tokens]
      const int xstride = d + 8;
      const int gid = lane >> 2, c = lane & 3;
      const int kw = warp * 256;
      const int lit = lane & 7, lhalf = (lane >> 3) & 1;  // ldmatrix: row, 8-column half
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
      bool stop = false;
      int i = 0;
      while (i < n && !stop) {
        const int g = lgrp[i];
        int e = i;
        while (e < n && lgrp[e] == g) ++e;
        // segment start: the group, and its tokens' x in shared memory (zero rows after
        // the last token)
        named_barrier(1, nct);
        if (tid == 0) s_gd = p.groups[g];
        named_barrier(1, nct);
        const int ntok = s_gd.n_tok;
        constexpr int XR = NT <= 4 ? 4 : 8;  // x rows held (the group size bound)
#pragma unroll
        for (int t = 0; t < XR; ++t) {
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (t < ntok) xv = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)s_gd.tok[t] * d) + tid);
          reinterpret_cast<uint4*>(xs + (size_t)t * xstride)[tid] = xv;
        }
        const float wtl = (lane & 7) < ntok ? s_gd.w[lane & 7] : 0.f;  // warp 0: token lane % 8

        float accm[16][4];
#pragma unroll
        for (int j = 0; j < 16; ++j) accm[j][0] = accm[j][1] = accm[j][2] = accm[j][3] = 0.f;
        named_barrier(1, nct);
        for (int i0 = i; i0 < e; i0 += kMmaBatch) {
          const int nb = min(kMmaBatch, e - i0);
          int sq0 = cs, sq1 = cs, sq2 = cs, sq3 = cs;
          bool ok = !*reinterpret_cast<volatile int*>(&s_abort);
#pragma unroll
          for (int q = 0; q < kMmaBatch; ++q) {
            if (q < nb) {
              if (q == 0) sq0 = cs;
              if (q == 1) sq1 = cs;
              if (q == 2) sq2 = cs;
              if (q == 3) sq3 = cs;
              ok = ok && mbar_wait(&full[cs], cph);
              if (++cs == S) {
                cs = 0;
                cph ^= 1;
              }
            }
          }
          // this lane's ldmatrix row: kept row lit of the batch.  Absent rows repeat row
          // 0 (same address: no bank conflict; finite weights whose dot products are not
          // used and whose down contributions are multiplied by h = 0)
          const int sl = (lit < nb) ? (lit == 1 ? sq1 : lit == 2 ? sq2 : lit == 3 ? sq3 : sq0) : sq0;
          const int ld = lit & 3;  // down operand: k = lit holds row lit % 4
          const int sld = (ld < nb) ? (ld == 1 ? sq1 : ld == 2 ? sq2 : ld == 3 ? sq3 : sq0) : sq0;
          const uint32_t garow = smem_addr(stage + (size_t)sl * L.stage_bytes) + (uint32_t)(kw + lhalf * 8) * 2u;
          const uint32_t darow = smem_addr(stage + (size_t)sld * L.stage_bytes) + (uint32_t)(2 * d) +
                                 (uint32_t)(kw + lhalf * 8) * 2u;
          // two accumulator chains (even and odd k-steps) halve the dependent mma latency
          float dd[4] = {0.f, 0.f, 0.f, 0.f}, de[4] = {0.f, 0.f, 0.f, 0.f};
          ok = __all_sync(0xffffffffu, ok);  // the mma below is warp-wide: one decision for all lanes
          if (ok) {
            // B column gid = token gid (zero beyond the x rows held)
            const bool xon = gid < XR;
            const __half* xg = xs + (size_t)(xon ? gid : 0) * xstride + kw + 2 * c;
            auto xb = [&](int off) -> uint32_t {
              if constexpr (XR == kMmaTok) return *reinterpret_cast<const uint32_t*>(xg + off);
              return xon ? *reinterpret_cast<const uint32_t*>(xg + off) : 0u;
            };
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              uint32_t a[4], a2[4];
              ldsm_x2(garow + j * 32u, a[0], a[2]);
              ldsm_x2(garow + (j + 1) * 32u, a2[0], a2[2]);
              a[1] = a[3] = a2[1] = a2[3] = 0u;
              mma_16816(dd, a, xb(j * 16), xb(j * 16 + 8));
              mma_16816(de, a2, xb((j + 1) * 16), xb((j + 1) * 16 + 8));
            }
            dd[0] += de[0];
            dd[1] += de[1];
          }
          if (gid < kMmaBatch) {
            redm[(warp * kMmaBatch + gid) * kMmaTok + 2 * c] = dd[0];
            redm[(warp * kMmaBatch + gid) * kMmaTok + 2 * c + 1] = dd[1];
          }
          if (bar_or(!ok)) {
            if (tid == 0) {
              set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
              atomicExch(&s_abort, 1);
            }
            stop = true;
            break;
          }
          if (warp == 0) {
            // lane = row * 8 + token
            const int it = lane >> 3, t = lane & 7;
            float hq = 0.f;
            if (it < nb && t < ntok) {
              float s0 = 0.f, s1 = 0.f;
              int w = 0;
              for (; w + 1 < ncw; w += 2) {
                s0 += redm[(w * kMmaBatch + it) * kMmaTok + t];
                s1 += redm[((w + 1) * kMmaBatch + it) * kMmaTok + t];
              }
              if (w < ncw) s0 += redm[(w * kMmaBatch + it) * kMmaTok + t];
              const int si = it == 0 ? sq0 : it == 1 ? sq1 : it == 2 ? sq2 : sq3;
              const float* hv = reinterpret_cast<const float*>(stage + (size_t)si * L.stage_bytes + 4 * d);
              hq = silu_f(s0 + s1) * hv[t] * wtl;
            }
            const __half hi = __float2half_rn(hq);
            const __half lo = __float2half_rn(hq - __half2float(hi));
            h16[t * 16 + it] = hi;
            h16[t * 16 + kMmaBatch + it] = lo;
          }
          named_barrier(1, nct);
          {
            const uint32_t bh = *reinterpret_cast<const uint32_t*>(h16 + gid * 16 + 2 * c);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              uint32_t a[4];
              ldsm_x2_trans(darow + j * 32u, a[0], a[1]);
              a[2] = a[3] = 0u;
              mma_16816(accm[j], a, bh, 0u);
            }
          }
          // the batch's stages are free once every warp has read them
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&empty[sq0]);
            if (nb > 1) mbar_arrive(&empty[sq1]);
            if (nb > 2) mbar_arrive(&empty[sq2]);
            if (nb > 3) mbar_arrive(&empty[sq3]);
          }
          if (tid == 0) s_consumed = base + i0 + nb;
        }
        // segment end: this CTA's partial output of the group; accm[j] holds columns
        // kw + 16 j + gid (+ 8) of tokens 2c and 2c + 1
        if (!stop) {
          float* dst = p.part + ((size_t)(blockIdx.x + g) * kMaxTok) * d;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = kw + 16 * j + gid;
            if (2 * c < ntok) {
              dst[(size_t)(2 * c) * d + col] = accm[j][0];
              dst[(size_t)(2 * c) * d + col + 8] = accm[j][2];
            }
            if (2 * c + 1 < ntok) {
              dst[(size_t)(2 * c + 1) * d + col] = accm[j][1];
              dst[(size_t)(2 * c + 1) * d + col + 8] = accm[j][3];
            }
          }
        }
        if (tid == 0) s_consumed = base + e;
        i = e;
      }
    } else {
      // ---- consumers: segments of equal group; in a segment, batches of up to kR
      // items with one barrier each, software-pipelined: every warp forms the dot
      // products of batch k, then (after the barrier) applies batch k-1 while warp 0
      // turns batch k's sums into h = SiLU(.) * v * w.
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
      // acc += h (batch parity par) * this thread's down slices of the batch's stages
      auto apply = [&](int par, int nbq, const int (&sq)[kR]) {
        const float* hb = hbuf + par * kR * NT;
#pragma unroll
        for (int q = 0; q < kR; ++q) {
          if (q < nbq) {
            const uint8_t* st = stage + (size_t)sq[q] * L.stage_bytes;
            const uint4 dr = reinterpret_cast<const uint4*>(st + 2 * d)[tid];
            const __half2* dh = reinterpret_cast<const __half2*>(&dr);
            float2 hv[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) hv[t] = make_float2(hb[q * NT + t], hb[q * NT + t]);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float2 df = __half22float2(dh[e2]);
#pragma unroll
              for (int t = 0; t < NT; ++t) acc[t][e2] = __ffma2_rn(hv[t], df, acc[t][e2]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int q = 0; q < kR; ++q)
            if (q < nbq) mbar_arrive(&empty[sq[q]]);
        }
      };
      bool stop = false;
      int i = 0;
      while (i < n && !stop) {
        const int g = lgrp[i];
        int e = i;
        while (e < n && lgrp[e] == g) ++e;
        // segment start: the group's tokens, weights, x
        named_barrier(1, nct);
        if (tid == 0) s_gd = p.groups[g];
        named_barrier(1, nct);
        const int ntok = s_gd.n_tok;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          wt[t] = t < ntok ? s_gd.w[t] : 0.f;
          uint4 xv = make_uint4(0, 0, 0, 0);
          if (t < ntok) xv = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)s_gd.tok[t] * d) + tid);
          const __half2* xh = reinterpret_cast<const __half2*>(&xv);
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            xf[t][e2] = __half22float2(xh[e2]);
            acc[t][e2] = make_float2(0.f, 0.f);
          }
        }
        int prev_s[kR];
        int prev_nb = 0, bt = 0;
        for (int i0 = i; i0 < e; i0 += kR) {
          const int nb = min(kR, e - i0);
          int sq[kR];
          bool ok = !*reinterpret_cast<volatile int*>(&s_abort);
#pragma unroll
          for (int q = 0; q < kR; ++q) {
            sq[q] = cs;
            if (q < nb) {
              ok = ok && mbar_wait(&full[cs], cph);
              if (++cs == S) {
                cs = 0;
                cph ^= 1;
              }
            }
          }
          float dot[kR * NT];
#pragma unroll
          for (int q = 0; q < kR; ++q) {
            float2 d2[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) d2[t] = make_float2(0.f, 0.f);
            if (q < nb && ok) {
              const uint4 gr = reinterpret_cast<const uint4*>(stage + (size_t)sq[q] * L.stage_bytes)[tid];
              const __half2* gh = reinterpret_cast<const __half2*>(&gr);
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const float2 gf = __half22float2(gh[e2]);
#pragma unroll
                for (int t = 0; t < NT; ++t) d2[t] = __ffma2_rn(xf[t][e2], gf, d2[t]);
              }
            }
#pragma unroll
            for (int t = 0; t < NT; ++t) dot[q * NT + t] = d2[t].x + d2[t].y;
          }
          // warp sums of the kR x NT dot products; lanes 0, 4, ... hold one each
          int vi;
          const float vs = warp_sum_halving<kR * NT>(dot, lane, vi);
          float* rb = red + (size_t)(bt & 1) * kR * NT * ncw;
          if ((lane & (32 / (kR * NT) - 1)) == 0) rb[vi * ncw + warp] = vs;
          if (bar_or(!ok)) {
            if (tid == 0) {
              set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
              atomicExch(&s_abort, 1);
            }
            stop = true;
            break;
          }
          // the previous batch, with the h warp 0 wrote before this barrier
          if (bt > 0) apply((bt - 1) & 1, prev_nb, prev_s);
          if (tid == 0) s_consumed = base + i0;  // the stages before this batch are free
          if (warp == 0 && lane < kR * NT) {
            const int q = lane / NT, t = lane - (lane / NT) * NT;
            float hq = 0.f;
            int sl = sq[0];
#pragma unroll
            for (int qq = 1; qq < kR; ++qq)
              if (q == qq) sl = sq[qq];
            float wtt = wt[0];
#pragma unroll
            for (int tt = 1; tt < NT; ++tt)
              if (t == tt) wtt = wt[tt];
            if (q < nb && t < ntok) {
              // the consumer warps' partial sums, four at a time (independent loads)
              const float* pr = rb + lane * ncw;
              float gs = 0.f;
              int w = 0;
              if ((ncw & 3) == 0) {
                float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
                for (; w < ncw; w += 4) {
                  const float4 v4 = *reinterpret_cast<const float4*>(pr + w);
                  s4 = make_float4(s4.x + v4.x, s4.y + v4.y, s4.z + v4.z, s4.w + v4.w);
                }
                gs = (s4.x + s4.y) + (s4.z + s4.w);
              }
              for (; w < ncw; ++w) gs += pr[w];
              const float* hv = reinterpret_cast<const float*>(stage + (size_t)sl * L.stage_bytes + 4 * d);
              hq = silu_f(gs) * hv[t] * wtt;
            }
            hbuf[(bt & 1) * kR * NT + lane] = hq;
          }
#pragma unroll
          for (int q = 0; q < kR; ++q) prev_s[q] = sq[q];
          prev_nb = nb;
          ++bt;
        }
        // the segment's last batch
        if (!stop && bt > 0) {
          if (bar_or(false)) {
            stop = true;
          } else {
            apply((bt - 1) & 1, prev_nb, prev_s);
          }
        }
        // segment end: this CTA's partial output of the group
        if (!stop) {
          float* dst = p.part + ((size_t)(blockIdx.x + g) * kMaxTok) * d;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (t < ntok) {
              float4* o = reinterpret_cast<float4*>(dst + (size_t)t * d + tid * kChunk);
              o[0] = make_float4(acc[t][0].x, acc[t][0].y, acc[t][1].x, acc[t][1].y);
              o[1] = make_float4(acc[t][2].x, acc[t][2].y, acc[t][3].x, acc[t][3].y);
            }
          }
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

// Ring depth for the tensor-core consumers: a multiple of 4 stages.  Stage k starts at
// 32 k bytes modulo 128, so the 4 rows of any batch then sit in distinct bank quarters
// for ldmatrix, also across the ring's wrap.
int gather_round_stages(int d, int nt, int stages) {
  return gather_mma(d, nt) && stages >= 8 ? stages & ~3 : stages;
}

// Bytes of the stage ring that the prologue borrows (checked against the ring size).
size_t gather_ring_scratch_bytes(int d, int f) { return gather_scan_bytes(f / kMTile, (d / 256 + 1) * 32); }

cudaError_t launch_gather(const ExpertParams& p, int nt, cudaStream_t st, bool pdl) {
  const int ncw = p.d / 256;
  const size_t smem = gather_smem_bytes(p.d, p.stages, nt, p.list_cap, p.G_max);
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
#define SESG_G(NTV, MT, MM)                                                                        \
  if ((ncw + 1) * 32 > MT) return cudaErrorInvalidConfiguration;                                     \
  e = cudaFuncSetAttribute(gather_kernel<NTV, MT, MM>, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                           (int)smem);                                                                \
  if (e != cudaSuccess) return e;                                                                     \
  return cudaLaunchKernelEx(&cfg, gather_kernel<NTV, MT, MM>, p);
  // register caps: 96 per thread up to 640 threads (d <= 4096), 72 up to 800 (d <= 6144),
  // 64 above
  const bool small = (ncw + 1) * 32 <= 640;
  const bool mid = (ncw + 1) * 32 <= 800;
  if (gather_mma(p.d, nt)) {
    if (nt <= 4) { SESG_G(4, 640, true) }
    SESG_G(8, 640, true)
  }
  if (nt == 1) { if (small) { SESG_G(1, 640, false) } if (mid) { SESG_G(1, 800, false) } SESG_G(1, 1024, false) }
  if (nt == 2) { if (small) { SESG_G(2, 640, false) } if (mid) { SESG_G(2, 800, false) } SESG_G(2, 1024, false) }
  if (nt == 4 && small) { SESG_G(4, 640, false) }
  return cudaErrorInvalidConfiguration;
#undef SESG_G
}

}  // namespace sesg
