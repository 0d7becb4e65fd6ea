// Batched decode / prefill contraction: steps 3 and 4 of Algorithm 1 "Efficient Sparse
// Kernel" ("FloE: On-the-Fly MoE Inference on Memory-constrained GPU", sec. 三) for
// 16 to 64 tokens, with every kept gate and down row read once per expert however many
// of the call's tokens the expert serves.  (FloE's limitations name decode-only
// sparsity; MoE-Lightning sec. 三 notes that an FFN's arithmetic intensity grows with
// the batch.)  The router and the INT2 up projection are the general path's; the up
// kernel also writes every token's dense v and mask words.  Then:
//
//   seg    one CTA per expert (routed, then shared): its tokens in ascending order, and
//          the union of their masks as a list of kept columns;
//   gate   H[r][t] = SiLU(x_t . gate[col_r]) * v_t[col_r] * mask_t[col_r] * w_t for
//          each expert's tokens in groups of 16: whole gate rows streamed by bulk copies,
//          mma.m16n8k16 with the group's x as A (in registers) and 8 kept rows as B; h is
//          stored as fp16 hi + lo (about 22 bits);
//   down   Y^T[c][t] = sum_r down[col_r][c] * H[r][t] for one 2048-column chunk of d and
//          one part of 512 kept rows per tile: the rows' chunks streamed by bulk copies
//          in batches of 16, ldmatrix.trans of the down rows as A, H hi and lo as B, the
//          accumulators (2048 columns x 16 tokens over the warps) in registers; each
//          (part, token, slot) output row belongs to one tile, so plain stores;
//   final  y = sum over a token's slots and parts (the weights are inside h), RMSNorm
//          if asked, fp16.
//
// Every sum has a fixed order: the batched path is bitwise reproducible.
#include "params.cuh"

namespace sesg {

namespace {

constexpr int kBtMaxTok = 64;     // tokens per call (and so per expert), at most
constexpr int kSegThreads = 256;
constexpr int kBtMaxSeg = 264;    // routed + shared experts
constexpr int kBtPartRows = 512;  // down: kept rows per part (a multiple of the batch rows)

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2b(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// In-place exclusive prefix sum of a[0..n) (a[n] = total) by one block; tmp holds
// blockDim.x + 1 ints.
__device__ void bt_block_scan(int* a, int n, int* tmp) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (n + nt - 1) / nt, lo = min(n, tid * per), hi = min(n, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += a[i];
  tmp[tid] = s;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < nt; ++i) {
      const int c = tmp[i];
      tmp[i] = run;
      run += c;
    }
    tmp[nt] = run;
  }
  __syncthreads();
  int run = tmp[tid];
  for (int i = lo; i < hi; ++i) {
    const int c = a[i];
    a[i] = run;
    run += c;
  }
  if (tid == 0) a[n] = tmp[nt];
  __syncthreads();
}

__device__ __forceinline__ const ExpertSet& bt_set(const BatchParams& p, int e, int& local) {
  if (e < p.routed.E) {
    local = e;
    return p.routed;
  }
  local = e - p.routed.E;
  return p.shared;
}

// ---- seg: expert e's tokens and the union of their masks -------------------------
__global__ void __launch_bounds__(kSegThreads) batch_seg_kernel(BatchParams p) {
  __shared__ int s_flag[kBtMaxTok + 1];
  __shared__ int s_tmp[kSegThreads + 1];
  __shared__ int s_tok[kBtMaxTok], s_slot[kBtMaxTok];
  extern __shared__ int s_words[];  // [fw + 1] kept-column counts per mask word
  griddep_wait();
  const int e = blockIdx.x, tid = threadIdx.x, B = p.B, k = p.k;
  const bool routed = e < p.routed.E;
  // this token's slot for expert e, or -1
  if (tid < B) {
    int slot = -1;
    if (routed) {
      for (int j = 0; j < k; ++j)
        if (p.topk_idx[tid * k + j] == e) slot = j;
    } else {
      slot = k + (e - p.routed.E);
    }
    s_slot[tid] = slot;
    s_flag[tid] = slot >= 0 ? 1 : 0;
  }
  __syncthreads();
  bt_block_scan(s_flag, B, s_tmp);
  const int T = s_flag[B];
  int tok_slot = -1, tok_pos = 0;
  if (tid < B) {
    tok_slot = s_slot[tid];
    tok_pos = s_flag[tid];
  }
  __syncthreads();
  if (tid < B && tok_slot >= 0) {
    s_tok[tok_pos] = tid;
    s_slot[tok_pos] = tok_slot;  // every thread read its own entry before the barrier
  }
  __syncthreads();
  if (tid < T) {
    const int b = s_tok[tid], sl = s_slot[tid];
    p.seg_tok[e * kBtMaxTok + tid] = b;
    p.seg_slot[e * kBtMaxTok + tid] = sl;
    p.seg_w[e * kBtMaxTok + tid] = routed ? p.topk_w[b * k + sl] : 1.f;
  }
  // union of the T tokens' masks, word by word (bits past f dropped)
  const int fw = p.fw, f = p.f;
  for (int m = tid; m < fw; m += blockDim.x) {
    uint32_t u = 0u;
    for (int t = 0; t < T; ++t) u |= p.mask[((size_t)s_tok[t] * p.n_slots + s_slot[t]) * fw + m];
    const int valid = f - 32 * m;
    if (valid < 32) u &= valid > 0 ? ((1u << valid) - 1u) : 0u;
    s_words[m] = __popc(u);
  }
  __syncthreads();
  bt_block_scan(s_words, fw, s_tmp);
  for (int m = tid; m < fw; m += blockDim.x) {
    uint32_t u = 0u;
    for (int t = 0; t < T; ++t) u |= p.mask[((size_t)s_tok[t] * p.n_slots + s_slot[t]) * fw + m];
    const int valid = f - 32 * m;
    if (valid < 32) u &= valid > 0 ? ((1u << valid) - 1u) : 0u;
    int o = s_words[m];
    while (u) {
      const int b = __ffs(u) - 1;
      u &= u - 1u;
      p.seg_col[(size_t)e * f + o++] = 32 * m + b;
    }
  }
  if (tid == 0) {
    p.seg_t[e] = T;
    p.seg_n[e] = s_words[fw];
  }
  griddep_launch_dependents();
}

__device__ __forceinline__ int bt_find(const int* pre, int nseg, int tile) {
  int lo = 0, hi = nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Barrier of the first n threads (id 1) that also ORs `bad` over them: every consumer
// warp learns of a failed wait at the same barrier, so none is left waiting at a later one.
__device__ __forceinline__ bool bar_or(bool bad, int n) {
  int any;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.u32 pin, %1, 0;\n\t"
      "barrier.red.or.pred pout, 1, %2, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}"
      : "=r"(any)
      : "r"((unsigned)bad), "r"(n)
      : "memory");
  return any != 0;
}

// ---- gate: h for the kept rows of one expert and one group of 16 of its tokens ------
// Warps 0 .. ncw - 1 (ncw = d / 256) own 256-input slices of d and hold the group's x
// there as mma A fragments (16 tokens x 256 inputs = 64 registers); warp ncw's lanes
// stream whole gate rows (2d bytes, one bulk copy each, lane i the batch's row i) into a
// ring.  Per batch of 8 kept rows every warp forms D[16 tokens][8 rows] over its slice
// (the rows as B via ldmatrix), the partials meet in shared memory and the first 128
// consumer threads turn their sums into h = SiLU(.) * v * mask * w, one (row, token)
// each, stored at ht[expert][group][row][hi/lo][16 tokens].  (One warp forming all 128
// took 2,300 cycles a batch and held up every stage release behind it.)  Warp ncw + 1
// builds each tile's table of v * mask * w, one tile ahead of the consumers, in a second
// buffer.
// ring stages (one gate row each): 32 where they fit (d <= 2048), else 16.  Rows take
// about 6 us from issue to arrival here (a cycle trace); 32 stages instead of 16 at
// DeepSeek-V2-Lite's shape, and 24 at Mixtral's, changed the pass by under 1 %.
constexpr int kGateSTMax = 32;
__host__ __device__ __forceinline__ int gate_stages(int d) { return d <= 2048 ? 32 : 16; }
constexpr int kGateWarps = 16;         // consumer warps, at most (d <= 4096)
constexpr int kGateBatch = 8;          // kept rows per batch (the mma N)
constexpr int kBtGroupTok = 16;        // tokens per group (the mma M)
constexpr int kBtMaxGroups = kBtMaxTok / kBtGroupTok;
constexpr int kBtTileRows = 64;        // gate tiles: kept rows per tile

__device__ __forceinline__ int bt_groups(int T) { return (T + kBtGroupTok - 1) / kBtGroupTok; }

__device__ __forceinline__ size_t bt_ht_index(int e, int g, int f, int r) {
  return ((((size_t)e * kBtMaxGroups + g) * f + r) * 2) * kBtGroupTok;
}

__global__ void __launch_bounds__((kGateWarps + 2) * 32, 1) batch_gate_kernel(BatchParams p) {
  extern __shared__ __align__(128) uint8_t bsm[];
  __shared__ int s_pre[kBtMaxSeg + 1];
  __shared__ int s_abort;
  // the tile tables: v * mask * w of each (kept row, group token); table k of this CTA
  // in buffer k % 2, filled by the table warp (tbl_full) and released by the consumers
  // (tbl_free) once the tile's last h is formed
  __shared__ float s_vmw[2][kBtTileRows][kBtGroupTok];
  __shared__ __align__(8) uint64_t tbl_full[2], tbl_free[2];
  const int d = p.d, f = p.f, ncw = d / 256, nct = ncw * 32;
  const size_t stage_b = (size_t)2 * d + 16;  // a gate row, padded against bank conflicts
  const int ST = gate_stages(d);
  uint64_t* full = reinterpret_cast<uint64_t*>(bsm);
  uint64_t* empty = full + kGateSTMax;
  float* red = reinterpret_cast<float*>(bsm + 2 * kGateSTMax * 8);       // [2][ncw][128]
  uint8_t* ring = bsm + 2 * kGateSTMax * 8 + 2 * kGateWarps * 128 * 4;
  const int nseg = p.routed.E + p.n_shared, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ncw);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tbl_full[b], 1);
      mbar_init(&tbl_free[b], 1);
    }
    fence_barrier_init();
    s_abort = 0;
  }
  griddep_wait();
  // tiles (expert, group, 64 kept rows)
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < nseg; ++e) {
      s_pre[e] = run;
      run += bt_groups(p.seg_t[e]) * ((p.seg_n[e] + kBtTileRows - 1) / kBtTileRows);
    }
    s_pre[nseg] = run;
  }
  __syncthreads();
  const int ntiles = s_pre[nseg];
  auto tile_of = [&](int tile, int& e, int& g, int& r0, int& nr) {
    e = bt_find(s_pre, nseg, tile);
    const int K = p.seg_n[e], nb = (K + kBtTileRows - 1) / kBtTileRows, i = tile - s_pre[e];
    g = i / nb;
    r0 = (i % nb) * kBtTileRows;
    nr = min(kBtTileRows, K - r0);
  };
  if (warp == ncw) {
    // ---- producer: the gate rows of this CTA's tiles, in order, in the consumers'
    // batches of 8: lane i copies the batch's row i into its own stage
    const uint64_t pol = policy_evict_first();
    int issued = 0;
    bool stop = false;
    for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x) {
      int e, g, r0, nr, el;
      tile_of(tile, e, g, r0, nr);
      const ExpertSet& es = bt_set(p, e, el);
      const __half* gbase = es.gate_t + (size_t)el * es.f * es.rs;
      for (int rb = 0; rb < nr && !stop; rb += kGateBatch) {
        const int cnt = min(kGateBatch, nr - rb);
        bool ok = !*reinterpret_cast<volatile int*>(&s_abort);
        if (ok && lane < cnt) {
          const int q = issued + lane, st = q % ST;
          if (q >= ST) ok = mbar_wait(&empty[st], ((q / ST) & 1) ^ 1);
          if (ok) {
            const int col = p.seg_col[(size_t)e * f + r0 + rb + lane];
            mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * d));
            bulk_g2s(ring + (size_t)st * stage_b, gbase + (size_t)col * es.rs, (uint32_t)(2 * d), &full[st], pol);
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) atomicExch(&s_abort, 1);
          stop = true;
        }
        issued += cnt;
      }
    }
  } else if (warp == ncw + 1) {
    // ---- table warp: lane l fills token l % 16's column of rows 2 j + l / 16, in three
    // rounds of independent loads (the rows' columns, their mask words, the kept v)
    const int tl = lane & (kBtGroupTok - 1), rh = lane / kBtGroupTok;
    int k = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
      const int b = k & 1;
      if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(&tbl_free[b], ((k >> 1) - 1) & 1))) {
        if (lane == 0) atomicExch(&s_abort, 1);
        break;
      }
      if (__any_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&s_abort) != 0)) break;
      int e, g, r0, nr;
      tile_of(tile, e, g, r0, nr);
      const int t0 = g * kBtGroupTok, Tg = min(kBtGroupTok, p.seg_t[e] - t0);
      const bool tok = tl < Tg;
      const int tk = tok ? p.seg_tok[e * kBtMaxTok + t0 + tl] : 0, sl = tok ? p.seg_slot[e * kBtMaxTok + t0 + tl] : 0;
      const float tw = tok ? p.seg_w[e * kBtMaxTok + t0 + tl] : 0.f;
      const size_t row = (size_t)tk * p.n_slots + sl;
      const int* cols = p.seg_col + (size_t)e * f + r0;
      int c[kBtTileRows / 2];
#pragma unroll
      for (int j = 0; j < kBtTileRows / 2; ++j) c[j] = (tok && 2 * j + rh < nr) ? cols[2 * j + rh] : -1;
      uint32_t kept = 0u;
#pragma unroll
      for (int j = 0; j < kBtTileRows / 2; ++j)
        if (c[j] >= 0 && ((p.mask[row * p.fw + (c[j] >> 5)] >> (c[j] & 31)) & 1u)) kept |= 1u << j;
#pragma unroll
      for (int j = 0; j < kBtTileRows / 2; ++j)
        s_vmw[b][2 * j + rh][tl] = ((kept >> j) & 1u) ? p.v[row * f + c[j]] * tw : 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tbl_full[b]);
    }
  } else {
    // ---- consumers
    const int gid = lane >> 2, c4 = lane & 3;
    int cs = 0, cph = 0, nbatch = 0, k = 0;
    bool failed = false;
    for (int tile = blockIdx.x; tile < ntiles && !failed; tile += gridDim.x, ++k) {
      int e, g, r0, nr;
      tile_of(tile, e, g, r0, nr);
      const int T = p.seg_t[e], t0 = g * kBtGroupTok, Tg = min(kBtGroupTok, T - t0), K = p.seg_n[e];
      named_barrier(1, nct);  // the h of the previous tile's last batch is formed
      if (tid == 0 && k > 0) mbar_arrive(&tbl_free[(k - 1) & 1]);
      // this tile's table (one decision for all consumer threads)
      if (bar_or(!mbar_wait(&tbl_full[k & 1], (k >> 1) & 1), nct)) {
        if (tid == 0) {
          set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
        failed = true;
        break;
      }
      const float(*tab)[kBtGroupTok] = s_vmw[k & 1];
      // this warp's x slice of the group's tokens as A fragments (zero past Tg)
      uint32_t xa[16][4];
      {
        const int ta = t0 + gid, tb = t0 + gid + 8;
        const __half* xa_p = p.x + (size_t)(gid < Tg ? p.seg_tok[e * kBtMaxTok + ta] : 0) * d + 256 * warp + 2 * c4;
        const __half* xb_p = p.x + (size_t)(gid + 8 < Tg ? p.seg_tok[e * kBtMaxTok + tb] : 0) * d + 256 * warp + 2 * c4;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          xa[ks][0] = gid < Tg ? __ldg(reinterpret_cast<const uint32_t*>(xa_p + 16 * ks)) : 0u;
          xa[ks][1] = gid + 8 < Tg ? __ldg(reinterpret_cast<const uint32_t*>(xb_p + 16 * ks)) : 0u;
          xa[ks][2] = gid < Tg ? __ldg(reinterpret_cast<const uint32_t*>(xa_p + 16 * ks + 8)) : 0u;
          xa[ks][3] = gid + 8 < Tg ? __ldg(reinterpret_cast<const uint32_t*>(xb_p + 16 * ks + 8)) : 0u;
        }
      }
      for (int b0 = 0; b0 < nr; b0 += kGateBatch) {
        const int nv = min(kGateBatch, nr - b0);
        // the batch's stages: row i in stage (cs + i) mod ST
        bool ok = !*reinterpret_cast<volatile int*>(&s_abort);
        for (int i = 0; i < nv && ok; ++i) {
          int sq = cs + i, pq = cph;
          if (sq >= ST) {
            sq -= ST;
            pq ^= 1;
          }
          ok = mbar_wait(&full[sq], pq);
        }
        ok = __all_sync(0xffffffffu, ok);
        // B: lanes 0-7 address kept row (lane & 7) (row 0 again past nv) at k, 8-15 at k + 8
        const int ri = (lane & 7) < nv ? (lane & 7) : 0;
        int sr = cs + ri;
        if (sr >= ST) sr -= ST;
        const uint32_t bbase = smem_addr(ring + (size_t)sr * stage_b) + (uint32_t)(256 * warp + ((lane >> 3) & 1) * 8) * 2u;
        float dacc[4] = {0.f, 0.f, 0.f, 0.f};
        if (ok) {
#pragma unroll
          for (int ks = 0; ks < 16; ++ks) {
            uint32_t bb0, bb1;
            ldsm_x2b(bbase + ks * 32u, bb0, bb1);
            mma_16816(dacc, xa[ks], bb0, bb1);
          }
        }
        __syncwarp();
        if (lane == 0 && ok)
          for (int i = 0; i < nv; ++i) {
            int sq = cs + i;
            if (sq >= ST) sq -= ST;
            mbar_arrive(&empty[sq]);
          }
        cs += nv;
        if (cs >= ST) {
          cs -= ST;
          cph ^= 1;
        }
        float* rb = red + (size_t)(nbatch & 1) * kGateWarps * 128;
        *reinterpret_cast<float4*>(rb + warp * 128 + lane * 4) = make_float4(dacc[0], dacc[1], dacc[2], dacc[3]);
        if (bar_or(!ok, nct)) {
          if (tid == 0) {
            set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          failed = true;
          break;
        }
        // h of the batch's 128 (row, token) values, one per consumer thread (the first
        // 128): value q is accumulator entry q & 3 of lane q >> 2, i.e. token
        // (q >> 4) + 8 (q >> 1 & 1) and row 2 (q >> 2 & 3) + (q & 1); the warps' partials
        // added in warp order
        for (int q = tid; q < 128; q += nct) {
          float sum = 0.f;
#pragma unroll
          for (int w = 0; w < kGateWarps; ++w)
            if (w < ncw) sum += rb[w * 128 + q];
          const int ql = q >> 2, i = q & 3;
          const int tl = (ql >> 2) + (i >= 2 ? 8 : 0), rl = b0 + 2 * (ql & 3) + (i & 1);
          if (tl < Tg && rl < nr) {
            const int r = r0 + rl;
            const float vmw = tab[rl][tl];
            const float h = vmw != 0.f ? silu_f(sum) * vmw : 0.f;
            const __half hi = __float2half_rn(h);
            const __half lo = __float2half_rn(h - __half2float(hi));
            __half* dst = p.ht + bt_ht_index(e, g, f, r);
            dst[tl] = hi;
            dst[kBtGroupTok + tl] = lo;
          }
        }
        ++nbatch;
      }
      // the down pass reads 16-row batches whole: rows K .. roundup16(K) of the last tile
      // and the tokens past Tg of every row get h = 0 (written by this CTA only)
      if (warp == 0 && !failed) {
        for (int r = r0 + lane; r < r0 + kBtTileRows && r < f; r += 32) {
          __half* dst = p.ht + bt_ht_index(e, g, f, r);
          if (r >= K) {
            if (r < ((K + 15) & ~15))
              for (int j = 0; j < 2 * kBtGroupTok; ++j) dst[j] = __float2half_rn(0.f);
          } else {
            for (int j = Tg; j < kBtGroupTok; ++j) {
              dst[j] = __float2half_rn(0.f);
              dst[kBtGroupTok + j] = __float2half_rn(0.f);
            }
          }
        }
      }
    }
  }
  __syncthreads();
  griddep_launch_dependents();
}

// ---- down: one 2048-column chunk of d for one part (512 rows) of one (expert, group) --
// Warps 0 .. ncw - 1 (ncw = W / 128, W = min(d, 2048)) own 128 columns of the chunk and
// accumulate Y^T[128 columns][16 tokens] in registers; warp ncw streams batches of 16
// kept rows (each row's chunk, 2W bytes, one bulk copy, lane i row i) with their h (1 KB,
// lane 16).  The part's sums go to ypart[part][token][slot], added in order by the final
// kernel.
constexpr int kDownST = 3;
constexpr int kDownRowsB = 16;   // kept rows per batch (the mma K)
constexpr int kDownWarps = 16;
__host__ __device__ __forceinline__ int bt_chunk(int d) { return d < 2048 ? d : 2048; }

__global__ void __launch_bounds__((kDownWarps + 1) * 32, 1) batch_down_kernel(BatchParams p) {
  extern __shared__ __align__(128) uint8_t bsm[];
  __shared__ int s_pre[kBtMaxSeg + 1];
  __shared__ int s_abort;
  __shared__ int s_row[kBtGroupTok];  // the group tokens' output rows (token * slots + slot)
  const int d = p.d, f = p.f, W = bt_chunk(d), nchunk = d / W, ncw = W / 128;
  const size_t row_b = (size_t)2 * W + 16;                          // a row's chunk, padded
  const size_t stage_b = (size_t)kDownRowsB * row_b + 2 * kBtGroupTok * 2 * kDownRowsB;  // + h [16][2][16]
  uint64_t* full = reinterpret_cast<uint64_t*>(bsm);
  uint64_t* empty = full + kDownST;
  uint8_t* ring = bsm + 128;
  const int nseg = p.routed.E + p.n_shared, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kDownST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ncw);
    }
    fence_barrier_init();
    s_abort = 0;
  }
  griddep_wait();
  if (tid == 0) {
    int run = 0;
    for (int e = 0; e < nseg; ++e) {
      s_pre[e] = run;
      const int parts = max(1, (p.seg_n[e] + kBtPartRows - 1) / kBtPartRows);
      run += bt_groups(p.seg_t[e]) * nchunk * parts;
    }
    s_pre[nseg] = run;
  }
  __syncthreads();
  const int ntiles = s_pre[nseg];
  // tile -> expert, group, chunk, part and its rows [rb, re)
  auto tile_of = [&](int tile, int& e, int& g, int& c, int& part, int& rb, int& re) {
    e = bt_find(s_pre, nseg, tile);
    const int K = p.seg_n[e], parts = max(1, (K + kBtPartRows - 1) / kBtPartRows), i = tile - s_pre[e];
    part = i % parts;
    c = (i / parts) % nchunk;
    g = i / (parts * nchunk);
    rb = part * kBtPartRows;
    re = min(K, rb + kBtPartRows);
  };
  if (warp == ncw) {
    // ---- producer: per batch, lane 0 arms the stage, then lanes 0-15 copy one row each
    // and lane 16 the batch's h
    const uint64_t pol = policy_evict_first();
    int s = 0, ph = 0, issued = 0;
    bool stop = false;
    for (int tile = blockIdx.x; tile < ntiles && !stop; tile += gridDim.x) {
      int e, g, c, part, rb, re, el;
      tile_of(tile, e, g, c, part, rb, re);
      const ExpertSet& es = bt_set(p, e, el);
      const __half* dbase = es.down + (size_t)el * es.f * es.rs + (size_t)c * W;
      for (int r0 = rb; r0 < re && !stop; r0 += kDownRowsB) {
        bool ok = !*reinterpret_cast<volatile int*>(&s_abort);
        if (lane == 0 && ok) {
          if (issued >= kDownST) ok = mbar_wait(&empty[s], ph ^ 1);
          if (ok)
            mbar_arrive_expect_tx(&full[s], (uint32_t)(kDownRowsB * 2 * W + 2 * kBtGroupTok * 2 * kDownRowsB));
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          if (lane == 0) atomicExch(&s_abort, 1);
          stop = true;
          break;
        }
        uint8_t* st = ring + (size_t)s * stage_b;
        if (lane < kDownRowsB) {
          // rows past the part's end (only at K): a real row with h = 0 (finite * 0)
          const int r = r0 + lane < re ? r0 + lane : re - 1;
          const int col = p.seg_col[(size_t)e * f + r];
          bulk_g2s(st + (size_t)lane * row_b, dbase + (size_t)col * es.rs, (uint32_t)(2 * W), &full[s], pol);
        } else if (lane == kDownRowsB) {
          bulk_g2s(st + kDownRowsB * row_b, p.ht + bt_ht_index(e, g, f, r0),
                   (uint32_t)(2 * kBtGroupTok * 2 * kDownRowsB), &full[s], pol);
        }
        ++issued;
        if (++s == kDownST) {
          s = 0;
          ph ^= 1;
        }
      }
    }
  } else {
    const int gid = lane >> 2, c4 = lane & 3;
    int cs = 0, cph = 0;
    bool stop = false;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      int e, g, c, part, rb, re;
      tile_of(tile, e, g, c, part, rb, re);
      const int T = p.seg_t[e], t0 = g * kBtGroupTok, Tg = min(kBtGroupTok, T - t0);
      // the previous tile's epilogue is done with the table, and every warp learns of a
      // failed wait in it
      if (bar_or(stop, ncw * 32)) {
        if (tid == 0) set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
        break;
      }
      if (tid < kBtGroupTok && tid < Tg)
        s_row[tid] = p.seg_tok[e * kBtMaxTok + t0 + tid] * p.n_slots + p.seg_slot[e * kBtMaxTok + t0 + tid];
      named_barrier(1, ncw * 32);
      float acc[8][2][4];
#pragma unroll
      for (int mi = 0; mi < 8; ++mi)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) acc[mi][nb][0] = acc[mi][nb][1] = acc[mi][nb][2] = acc[mi][nb][3] = 0.f;
      for (int r0 = rb; r0 < re; r0 += kDownRowsB) {
        if (!__all_sync(0xffffffffu, !*reinterpret_cast<volatile int*>(&s_abort) && mbar_wait(&full[cs], cph))) {
          if (lane == 0) {
            set_status(&p.ctrl->status, MOE_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          stop = true;
          break;
        }
        const uint8_t* st = ring + (size_t)cs * stage_b;
        const uint8_t* hh = st + kDownRowsB * row_b;  // [16 rows][hi/lo][16 tokens]
        // B = H (rows x tokens, row-major): ldmatrix.trans, lanes 0-7 rows 0-7, 8-15 rows 8-15
        const uint32_t bh = smem_addr(hh + (size_t)((lane & 7) + ((lane >> 3) & 1) * 8) * 64);
        uint32_t bhi[2][2], blo[2][2];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                       : "=r"(bhi[nb][0]), "=r"(bhi[nb][1]) : "r"(bh + nb * 16u));
          asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                       : "=r"(blo[nb][0]), "=r"(blo[nb][1]) : "r"(bh + 32u + nb * 16u));
        }
        // A = down^T (columns x rows) through ldmatrix.trans: lanes 0-7 a0 (columns m..,
        // rows 0-7), 8-15 a1 (columns m + 8..), 16-23 a2 (rows 8-15), 24-31 a3
        const int kr = (lane & 7) + ((lane >> 4) & 1) * 8;
        const uint32_t abase = smem_addr(st + (size_t)kr * row_b) + (uint32_t)(128 * warp + ((lane >> 3) & 1) * 8) * 2u;
#pragma unroll
        for (int mi = 0; mi < 8; ++mi) {
          uint32_t a[4];
          ldsm_x4_trans(abase + mi * 32u, a);
#pragma unroll
          for (int nb = 0; nb < 2; ++nb) {
            mma_16816(acc[mi][nb], a, bhi[nb][0], bhi[nb][1]);
            mma_16816(acc[mi][nb], a, blo[nb][0], blo[nb][1]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[cs]);
        if (++cs == kDownST) {
          cs = 0;
          cph ^= 1;
        }
      }
      if (stop) continue;  // the next tile's barrier tells the other warps
      // column 128 warp + 16 mi + gid (+ 8) of the chunk, token nb * 8 + 2 c4 (+ 1)
#pragma unroll
      for (int mi = 0; mi < 8; ++mi)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = c * W + 128 * warp + 16 * mi + gid + (i >= 2 ? 8 : 0);
            const int tl = nb * 8 + 2 * c4 + (i & 1);
            if (tl < Tg) p.ypart[((size_t)part * p.B * p.n_slots + s_row[tl]) * d + col] = acc[mi][nb][i];
          }
    }
  }
  __syncthreads();
  griddep_launch_dependents();
}

// ---- final: y = sum over a token's slots and their parts (fixed order), RMSNorm ----
constexpr int kFinalThreads = 512;
__global__ void __launch_bounds__(kFinalThreads) batch_final_kernel(BatchParams p) {
  __shared__ float s_red[kFinalThreads / 32];
  __shared__ int s_parts[kMaxSlots];
  griddep_wait();
  const int b = blockIdx.x, tid = threadIdx.x, d = p.d, S = p.n_slots;
  if (tid < S) {
    // the slot's expert and its number of parts
    const int e = tid < p.k ? p.topk_idx[b * p.k + tid] : p.routed.E + (tid - p.k);
    s_parts[tid] = max(1, (p.seg_n[e] + kBtPartRows - 1) / kBtPartRows);
  }
  __syncthreads();
  // 8 consecutive columns per thread (d <= 4096)
  const int i0 = tid * 8;
  float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (i0 < d) {
    for (int sl = 0; sl < S; ++sl)
      for (int q = 0; q < s_parts[sl]; ++q) {
        const float4* src = reinterpret_cast<const float4*>(p.ypart + (((size_t)q * p.B + b) * S + sl) * d + i0);
        const float4 a0 = src[0], a1 = src[1];
        v[0] += a0.x;
        v[1] += a0.y;
        v[2] += a0.z;
        v[3] += a0.w;
        v[4] += a1.x;
        v[5] += a1.y;
        v[6] += a1.z;
        v[7] += a1.w;
      }
  }
  float rinv = 1.f;
  if (p.rmsnorm) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) ss += v[j] * v[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) s_red[tid >> 5] = ss;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < kFinalThreads / 32; ++w) t += s_red[w];
    rinv = rsqrtf(t / (float)d + 1e-6f);
  }
  if (i0 < d) {
    __half2* yo = reinterpret_cast<__half2*>(p.y + (size_t)b * d + i0);
#pragma unroll
    for (int j = 0; j < 4; ++j) yo[j] = __floats2half2_rn(v[2 * j] * rinv, v[2 * j + 1] * rinv);
  }
  griddep_launch_dependents();
}

}  // namespace

size_t batch_gate_smem(int d) {
  return (size_t)2 * kGateSTMax * 8 + (size_t)2 * kGateWarps * 128 * 4 + (size_t)gate_stages(d) * (2 * d + 16);
}
size_t batch_down_smem(int d) {
  const size_t W = bt_chunk(d);
  return 128 + (size_t)kDownST * (kDownRowsB * (2 * W + 16) + 2 * kBtGroupTok * 2 * kDownRowsB);
}
// Parts of 512 rows an expert's down pass has, at most (the ypart buffer's first index).
int batch_max_parts(int f) { return (f + kBtPartRows - 1) / kBtPartRows; }

cudaError_t launch_batched(const BatchParams& p, int P, cudaStream_t st) {
  const int nseg = p.routed.E + p.n_shared;
  if (nseg > kBtMaxSeg || p.B > kBtMaxTok || p.d % 256 || p.d > 4096 || p.n_slots > kMaxSlots ||
      bt_chunk(p.d) % 128 || p.f % 16)
    return cudaErrorInvalidValue;
  batch_seg_kernel<<<nseg, kSegThreads, (size_t)(p.fw + 1) * sizeof(int), st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t gs = batch_gate_smem(p.d), ds = batch_down_smem(p.d);
  e = cudaFuncSetAttribute(batch_gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gs);
  if (e != cudaSuccess) return e;
  batch_gate_kernel<<<P, (p.d / 256 + 2) * 32, gs, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(batch_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ds);
  if (e != cudaSuccess) return e;
  batch_down_kernel<<<P, (bt_chunk(p.d) / 128 + 1) * 32, ds, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  batch_final_kernel<<<p.B, kFinalThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sesg
