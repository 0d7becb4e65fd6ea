// Kernel parameter blocks and launchers shared by the library's translation units.
#pragma once

#include "common.cuh"

namespace sesg {

struct RouteParams {
  const __half* x;         // [B][d]
  const __half* w_router;  // [d][E]
  int B, d, E, k, renorm;
  int n_shared;            // always-on shared experts (grouping only)
  int group;               // 1: build groups for the expert kernels
  int gcap;                // tokens per group (<= 8)
  int32_t* topk_idx;       // [B][k] (workspace copy, always written)
  float* topk_w;           // [B][k]
  int32_t* user_idx;       // optional copies
  float* user_w;
  int32_t* expert_count;   // optional [E]
  Ctrl* ctrl;
  GroupDesc* groups;       // grouping outputs
  int* tok_groups;         // [B][kMaxSlots]: (group << 3) | local token index
  int* group_total;        // [G_max] zeroed here for the expert kernels
  int G_max;
};

struct ExpertParams {
  ExpertSet routed, shared;
  const __half* x;          // [B][d]
  int B, d, f;
  const GroupDesc* groups;
  Ctrl* ctrl;
  uint8_t* unit_cnt;        // [G_max * MT] kept columns per (group, M-tile)
  int* item_col;            // [G_max * MT * 16]
  float* item_v;            // [G_max * MT * 16][8]: v of kept columns, 0 for tokens that drop them
  int* group_total;         // [G_max] kept items per group
  float* part;              // [(P3 + G_max)][8][d] per-CTA partial outputs
  const int* tok_groups;    // [B][16]
  int n_slots;              // slots per token in the debug outputs
  float* dbg_v;             // [B][n_slots][f] or NULL
  uint32_t* dbg_mask;       // [B][n_slots][f/32] or NULL
  __half* y;                // [B][d]
  int rmsnorm;
  int P3;                   // gather CTAs
  int stages;               // gather pipeline depth
  int list_cap;             // gather item-list capacity per CTA window
  int G_max;
  int max_tok;              // largest group of this call (sizes the up kernel's x buffer)
};

// The decode path (one or two tokens): up kernel (routing, up projection, mask, kept
// lists) and gather kernel (kept gate/down rows, the weighted sum and RMSNorm).
// copies of the decode paths' fp32 accumulator of y, CTA c adding into copy c % kDecYRep.
// More copies mean fewer atomic additions per address, but the last CTA reads and clears
// every copy; one copy measured fastest (Mixtral-8x7B one-token layer at 70 %: 1 copy
// 44.6 us, 2 copies 45.2, 4 copies 46.6, 8 copies 49.4).
constexpr int kDecYRep = 1;

struct DecodeParams {
  const __half* x;          // [B][d]
  const __half* w_router;   // [d][E]
  int B, d, f, k, renorm, n_shared;
  ExpertSet routed, shared;
  Ctrl* ctrl;
  GroupDesc* groups;        // [<= 24] written by CTA 0 of the up kernel
  int4* klist;              // [P][kcap] kept columns of every up CTA, in unit order:
                            // {column | group << 16, v of group token 0, 1 (float bits), 0}
  int kcap;                 // entries per up CTA
  int gmax;                 // group descriptors the workspace holds
  int umax;                 // units per up CTA, at most
  int* cta_total;           // [P] kept columns per up CTA
  float* yacc;              // [kDecYRep][B][d] fp32 sums of the CTAs' shares, CTA c adding
                            // into copy c % kDecYRep (left zeroed by the last CTA)
  int P;                    // CTAs of the up and gather kernels (one per SM)
  int list_cap;             // rows per gather CTA, at most
  int32_t* topk_idx;        // [B][k] workspace copies (written by CTA 0)
  float* topk_w;
  int32_t* user_idx;        // optional copies for the caller
  float* user_w;
  int n_slots;              // k + n_shared (debug row stride)
  float* dbg_v;             // [B][n_slots][f] or NULL
  uint32_t* dbg_mask;       // [B][n_slots][f/32] or NULL
  int su, sr;               // depths of the up-strip ring and of the row ring
  __half* y;                // [B][d]
  int rmsnorm;
  uint8_t* staging;         // or NULL: the kept rows in global kept order, 4d bytes each (gate
                            // row, down row), copied from host memory by the fetch kernel;
                            // the gather kernel then streams these instead of the experts
};

// The batched path (16 to 64 tokens): per-expert kept-row lists over the union of the
// expert's tokens' masks, then a gate pass and a down pass that read every kept row
// once per expert (batched.cu).
struct BatchParams {
  ExpertSet routed, shared;
  const __half* x;          // [B][d]
  int B, d, f, k, n_shared, n_slots;  // n_slots = k + n_shared
  const int32_t* topk_idx;  // [B][k] the router's choice
  const float* topk_w;      // [B][k]
  const float* v;           // [B][n_slots][f] dense v of the up kernel
  const uint32_t* mask;     // [B][n_slots][fw] mask words of the up kernel
  int fw;                   // (f + 31) / 32
  int* seg_n;               // [E + n_shared] kept rows of each expert
  int* seg_t;               // [E + n_shared] its tokens
  int* seg_tok;             // [E + n_shared][64] token, ascending
  int* seg_slot;            // [E + n_shared][64] the token's slot for the expert
  float* seg_w;             // [E + n_shared][64] combine weight (1 for shared experts)
  int* seg_col;             // [E + n_shared][f] kept columns, ascending
  __half* ht;               // [E + n_shared][4 groups][f][hi/lo][16 tokens] h as fp16 hi + lo
  float* ypart;             // [parts][B][n_slots][d] each (token, slot)'s weighted expert
                            // output, one row per 512-kept-row part of the expert
  __half* y;                // [B][d]
  int rmsnorm;
  Ctrl* ctrl;               // status of a timed-out wait
};

__device__ __forceinline__ const ExpertSet& expert_set(const ExpertParams& p, int expert,
                                                       int& local) {
  if (expert < p.routed.E) {
    local = expert;
    return p.routed;
  }
  local = expert - p.routed.E;
  return p.shared;
}

// pack.cu
cudaError_t launch_pack(const __half* w, int d, int f, uint8_t* packed, cudaStream_t st);
cudaError_t launch_unpack(const uint8_t* packed, int d, int f, uint8_t* q, __half* scale,
                          __half* zero, cudaStream_t st);
// route.cu
cudaError_t launch_route(const RouteParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_expert_prep(int expert, int n, int gcap, GroupDesc* groups, int* tok_groups,
                               int* group_total, Ctrl* ctrl, cudaStream_t st, bool pdl);
// up.cu
size_t up_smem_bytes(int d, int max_tok);
int up_threads(int d);
int up_blocks_per_sm(int d, int max_tok);
cudaError_t launch_up(const ExpertParams& p, int grid, cudaStream_t st, bool pdl);
// gather.cu
size_t gather_smem_bytes(int d, int stages, int nt, int list_cap, int g_max);
cudaError_t launch_gather(const ExpertParams& p, int nt, cudaStream_t st, bool pdl);
// combine.cu
size_t combine_smem_bytes(const ExpertParams& p);
cudaError_t launch_combine(const ExpertParams& p, cudaStream_t st, bool pdl);
// decode.cu
bool decode_supported(int B, int d, int f, int E, int k, int n_shared, int P);
int decode_list_cap(int B, int f, int k, int n_shared, int P);
int decode_units_max(int B, int f, int k, int n_shared, int P);
int decode_plan(int B, int d, int E, int umax, int list_cap, int P, int smem_optin, int& su, int& sr);
cudaError_t launch_decode_up(const DecodeParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_decode_gather(const DecodeParams& p, cudaStream_t st, bool pdl);
int decode_layer_plan(int B, int d, int E, int umax, int smem_optin, int& su, int& sr);
cudaError_t launch_decode_layer(const DecodeParams& p, cudaStream_t st, bool pdl);
// fetch.cu
cudaError_t launch_decode_fetch(const DecodeParams& p, cudaStream_t st, bool pdl);
// batched.cu
constexpr int kBatchMinTok = 16;  // the batched path serves 16 ..
constexpr int kBatchMaxTok = 64;  // .. 64 tokens (and d <= 4096)
int batch_max_parts(int f);
cudaError_t launch_batched(const BatchParams& p, int P, cudaStream_t st);

}  // namespace sesg
