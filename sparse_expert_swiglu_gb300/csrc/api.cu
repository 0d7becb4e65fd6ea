// extern "C" entry points: argument checks, workspace carving and kernel launches.
#include <string.h>

#include "params.cuh"

using namespace sesg;

namespace sesg {
size_t gather_ring_scratch_bytes(int d, int f);  // gather.cu
cudaError_t launch_expert_prefetch(const uint8_t* up, size_t up_bytes, int E, const int32_t* idx, int n,
                                   int max_experts, int P, cudaStream_t st);  // prefetch.cu
int gather_round_stages(int d, int nt, int stages);  // gather.cu
}

namespace {

constexpr size_t kWsAlign = 256;
constexpr int kMaxB = 1024;
constexpr int kMaxD = 7936;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
};

cudaError_t device_info(DeviceInfo& di) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
}

// Tokens of one expert handled together: their fp32 accumulators must fit in the
// gather kernel's registers (8 x 8 floats per thread up to d = 4096, 4 x 8 up to 6144).
// tokens per expert group: up to 8 where the gather kernel runs on the tensor cores
// (d <= 4096), 2 where it keeps x and the outputs of a group in registers
int group_cap(int d) { return d <= 4096 ? 8 : 2; }

int groups_max_routed(int B, int E, int k, int gcap) {
  const long long pairs = (long long)B * k;
  const long long bound = (pairs + gcap - 1) / gcap + (E < pairs ? E : pairs);
  return (int)(pairs < bound ? pairs : bound);
}

// Workspace carving shared by every entry point.
struct WsLayout {
  size_t ctrl, groups, tok_groups, topk_idx, topk_w, group_total, unit_cnt, item_col, item_v,
      part, yacc, cta_total, klist, total;
  // the batched path only (0 otherwise): dense v and masks, per-expert lists, h, outputs
  size_t bv = 0, bmask = 0, seg_n = 0, seg_t = 0, seg_tok = 0, seg_slot = 0, seg_w = 0, seg_col = 0,
         ht = 0, ypart = 0;
  int G_max, P3, list_cap;
};

WsLayout ws_layout(int B, int npairs, int G_max, int d, int f, int P3) {
  WsLayout L;
  const int MT = f / kMTile;
  const int list_cap = (int)(((long long)G_max * f + P3 - 1) / P3 + 1);
  L.G_max = G_max;
  L.P3 = P3;
  L.list_cap = list_cap < 2048 ? list_cap : 2048;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, kWsAlign);
    return at;
  };
  L.ctrl = take(sizeof(Ctrl));
  // the decode paths' fp32 accumulator of y, zero between calls (each call leaves it so):
  // at the same offset for every B, so that calls with different token counts can share
  // a workspace
  L.yacc = take(sizeof(float) * (size_t)kDecYRep * B * d);
  L.groups = take(sizeof(GroupDesc) * (size_t)(G_max > 0 ? G_max : 1));
  L.tok_groups = take(sizeof(int) * (size_t)B * kMaxSlots);
  L.topk_idx = take(sizeof(int) * (size_t)(npairs > 0 ? npairs : 1));
  L.topk_w = take(sizeof(float) * (size_t)(npairs > 0 ? npairs : 1));
  L.group_total = take(sizeof(int) * (size_t)(G_max > 0 ? G_max : 1));
  L.unit_cnt = take((size_t)G_max * MT);
  L.item_col = take(sizeof(int) * (size_t)G_max * MT * 16);
  L.item_v = take(sizeof(float) * (size_t)G_max * MT * 16 * 8);
  L.part = take(sizeof(float) * (size_t)(P3 + G_max) * kMaxTok * d);
  L.cta_total = take(sizeof(int) * (size_t)P3);
  // decode path: per up CTA, 16 entries of 16 bytes for each of its units
  L.klist = take((size_t)P3 * (((size_t)G_max * MT + P3 - 1) / P3) * 16 * 16);
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(ws) + off);
}

moe_status_t check_experts(const moe_experts_t* ex, int d, int f, bool may_be_empty) {
  if (!ex) return MOE_ERR_INVALID_ARG;
  if (ex->E == 0 && may_be_empty) return MOE_OK;
  if (ex->E < 1 || ex->E > 256) return ex->E < 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  if (ex->d != d || ex->f != f) return MOE_ERR_INVALID_ARG;
  if (!ex->up_packed || !ex->gate_t || !ex->down || !ex->thr) return MOE_ERR_INVALID_ARG;
  if (!aligned(ex->up_packed, 16) || !aligned(ex->gate_t, 16) || !aligned(ex->down, 16) ||
      !aligned(ex->thr, 4))
    return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

moe_status_t check_dims(int d, int f) {
  if (d <= 0 || f <= 0) return MOE_ERR_INVALID_ARG;
  if (d % 256 || d > kMaxD || f % kMTile || f > 65536) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

ExpertSet to_set(const moe_experts_t& ex) {
  ExpertSet s;
  s.E = ex.E;
  s.d = ex.d;
  s.f = ex.f;
  s.up = reinterpret_cast<const uint8_t*>(ex.up_packed);
  s.gate_t = reinterpret_cast<const __half*>(ex.gate_t);
  s.down = reinterpret_cast<const __half*>(ex.down);
  s.thr = ex.thr;
  s.up_stride = packed_bytes_per_expert(ex.d, ex.f);
  s.rs = (s.down == s.gate_t + ex.d) ? 2 * ex.d : ex.d;
  return s;
}

struct Plan {
  int up_grid;
  int stages;
  int nt;
};

// Grid of the up kernel, depth of the gather pipeline.
moe_status_t plan(const DeviceInfo& di, const WsLayout& L, int d, int f, int max_tok, Plan& pl) {
  const size_t up_smem = up_smem_bytes(d, max_tok);
  if (up_smem + 1024 > (size_t)di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int occ = up_blocks_per_sm(d, max_tok);
  if (occ < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  pl.up_grid = di.sms * occ;
  pl.nt = max_tok <= 1 ? 1 : max_tok <= 2 ? 2 : max_tok <= 4 ? 4 : 8;
  const size_t fixed = gather_smem_bytes(d, 0, pl.nt, L.list_cap, L.G_max) + 2048;
  const size_t stage = (size_t)4 * d + 32 + 16;
  if (fixed + 2 * stage > (size_t)di.smem_optin) return MOE_ERR_UNSUPPORTED_SHAPE;
  int S = (int)((di.smem_optin - fixed) / stage);
  S = gather_round_stages(d, pl.nt, S > 16 ? 16 : S);
  // the gather prologue borrows the stage buffers for the scan of one group's tile counts
  if ((size_t)S * (4 * d + 32) < gather_ring_scratch_bytes(d, f)) return MOE_ERR_UNSUPPORTED_SHAPE;
  pl.stages = S;
  return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Optional per-kernel timing events of moe_debug_t (index 0..4).
cudaError_t record(const moe_debug_t* dbg, int i, cudaStream_t st) {
  if (!dbg || !dbg->events || !dbg->events[i]) return cudaSuccess;
  // Inside stream capture an external record becomes an event-record node of the
  // graph; outside it the plain record is the one that applies.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const cudaError_t q = cudaStreamIsCapturing(st, &cs);
  if (q != cudaSuccess) return q;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags((cudaEvent_t)dbg->events[i], st, cudaEventRecordExternal);
  return cudaEventRecord((cudaEvent_t)dbg->events[i], st);
}

}  // namespace

extern "C" {

size_t expert_int2_up_packed_bytes(int32_t d, int32_t f) {
  if (d <= 0 || f <= 0 || d % kGroup || f % kMTile) return 0;
  return packed_bytes_per_expert(d, f);
}

moe_status_t expert_pack_int2_up(const uint16_t* w_up, int32_t d, int32_t f, void* up_packed,
                                 void* stream) {
  if (!w_up || !up_packed || d <= 0 || f <= 0) return MOE_ERR_INVALID_ARG;
  if (d % kGroup || f % kMTile) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(w_up, 16) || !aligned(up_packed, 16)) return MOE_ERR_ALIGNMENT;
  return cuda_status(launch_pack(reinterpret_cast<const __half*>(w_up), d, f,
                                 reinterpret_cast<uint8_t*>(up_packed), (cudaStream_t)stream));
}

moe_status_t expert_unpack_int2_up(const void* up_packed, int32_t d, int32_t f, uint8_t* q,
                                   uint16_t* scale, uint16_t* zero, void* stream) {
  if (!up_packed || d <= 0 || f <= 0) return MOE_ERR_INVALID_ARG;
  if (d % kGroup || f % kMTile) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(up_packed, 16)) return MOE_ERR_ALIGNMENT;
  return cuda_status(launch_unpack(reinterpret_cast<const uint8_t*>(up_packed), d, f, q,
                                   reinterpret_cast<__half*>(scale),
                                   reinterpret_cast<__half*>(zero), (cudaStream_t)stream));
}

size_t moe_route_workspace_bytes(int32_t B, int32_t E, int32_t k) {
  if (B < 0 || E < 1 || k < 1) return 0;
  return ws_layout(B, B * k, 0, 256, kMTile, 1).total;
}

moe_status_t moe_route_topk(const uint16_t* x, int32_t B, int32_t d, const uint16_t* w_router,
                            int32_t E, int32_t k, int32_t renorm, int32_t* topk_idx, float* topk_w,
                            int32_t* expert_count, void* ws, size_t ws_bytes, void* stream) {
  if (B < 0 || d <= 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (B > kMaxB || E > 256 || k > kMaxTok || d % 256 || d > kMaxD) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (B == 0) return MOE_OK;
  if (!x || !w_router || !topk_idx || !topk_w || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16)) return MOE_ERR_ALIGNMENT;
  if (!aligned(ws, kWsAlign)) return MOE_ERR_ALIGNMENT;
  const WsLayout L = ws_layout(B, B * k, 0, 256, kMTile, 1);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  RouteParams rp = {};
  rp.x = reinterpret_cast<const __half*>(x);
  rp.w_router = reinterpret_cast<const __half*>(w_router);
  rp.B = B;
  rp.d = d;
  rp.E = E;
  rp.k = k;
  rp.renorm = renorm ? 1 : 0;
  rp.group = 0;
  rp.gcap = kMaxTok;
  rp.topk_idx = at<int32_t>(ws, L.topk_idx);
  rp.topk_w = at<float>(ws, L.topk_w);
  rp.user_idx = topk_idx;
  rp.user_w = topk_w;
  rp.expert_count = expert_count;
  rp.ctrl = at<Ctrl>(ws, L.ctrl);
  return cuda_status(launch_route(rp, (cudaStream_t)stream, true));
}

// ---------------------------------------------------------------------------

static moe_status_t expert_params(const uint16_t* x, int B, const moe_experts_t* routed,
                                  const moe_experts_t* shared, int n_slots, uint16_t* y, int rmsnorm,
                                  const moe_debug_t* dbg, void* ws, const WsLayout& L, const DeviceInfo& di,
                                  int max_tok, ExpertParams& p, Plan& pl) {
  moe_status_t s = plan(di, L, routed->d, routed->f, max_tok, pl);
  if (s != MOE_OK) return s;
  p = ExpertParams{};
  p.routed = to_set(*routed);
  if (shared && shared->E > 0) p.shared = to_set(*shared);
  p.x = reinterpret_cast<const __half*>(x);
  p.B = B;
  p.d = routed->d;
  p.f = routed->f;
  p.groups = at<GroupDesc>(ws, L.groups);
  p.ctrl = at<Ctrl>(ws, L.ctrl);
  p.unit_cnt = at<uint8_t>(ws, L.unit_cnt);
  p.item_col = at<int>(ws, L.item_col);
  p.item_v = at<float>(ws, L.item_v);
  p.group_total = at<int>(ws, L.group_total);
  p.part = at<float>(ws, L.part);
  p.tok_groups = at<int>(ws, L.tok_groups);
  p.n_slots = n_slots;
  p.dbg_v = dbg ? dbg->v : nullptr;
  p.dbg_mask = dbg ? dbg->mask : nullptr;
  p.y = reinterpret_cast<__half*>(y);
  p.rmsnorm = rmsnorm;
  p.P3 = L.P3;
  p.stages = pl.stages;
  p.list_cap = L.list_cap;
  p.G_max = L.G_max;
  p.max_tok = max_tok;
  return MOE_OK;
}

static moe_status_t run_experts(const uint16_t* x, int B, const moe_experts_t* routed,
                                const moe_experts_t* shared, int n_slots, uint16_t* y,
                                int rmsnorm, const moe_debug_t* dbg, void* ws,
                                const WsLayout& L, const DeviceInfo& di, int max_tok,
                                cudaStream_t st) {
  ExpertParams p;
  Plan pl;
  moe_status_t s = expert_params(x, B, routed, shared, n_slots, y, rmsnorm, dbg, ws, L, di, max_tok, p, pl);
  if (s != MOE_OK) return s;
  cudaError_t e = record(dbg, 1, st);
  if (e == cudaSuccess) e = launch_up(p, pl.up_grid, st, true);
  if (e == cudaSuccess) e = record(dbg, 2, st);
  if (e == cudaSuccess) e = launch_gather(p, pl.nt, st, true);
  if (e == cudaSuccess) e = record(dbg, 3, st);
  if (e == cudaSuccess) e = launch_combine(p, st, true);
  if (e == cudaSuccess) e = record(dbg, 4, st);
  return cuda_status(e);
}

size_t moe_expert_workspace_bytes(int32_t n, int32_t d, int32_t f) {
  if (n < 0 || check_dims(d, f) != MOE_OK) return 0;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return 0;
  const int gcap = group_cap(d);
  return ws_layout(n, n, (n + gcap - 1) / gcap, d, f, di.sms).total;
}

moe_status_t moe_expert_sparse_swiglu(const uint16_t* x, int32_t n, const moe_experts_t* experts,
                                      int32_t expert, uint16_t* y, const moe_debug_t* dbg, void* ws,
                                      size_t ws_bytes, void* stream) {
  if (n < 0 || !experts) return MOE_ERR_INVALID_ARG;
  moe_status_t s = check_dims(experts->d, experts->f);
  if (s != MOE_OK) return s;
  if (n > kMaxB) return MOE_ERR_UNSUPPORTED_SHAPE;
  s = check_experts(experts, experts->d, experts->f, false);
  if (s != MOE_OK) return s;
  if (expert < 0 || expert >= experts->E) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!x || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_ALIGNMENT;
  if (!aligned(ws, kWsAlign)) return MOE_ERR_ALIGNMENT;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return MOE_ERR_CUDA;
  const int gcap = group_cap(experts->d);
  const WsLayout L = ws_layout(n, n, (n + gcap - 1) / gcap, experts->d, experts->f, di.sms);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  if (record(dbg, 0, st) != cudaSuccess) return MOE_ERR_CUDA;
  cudaError_t e = launch_expert_prep(expert, n, gcap, at<GroupDesc>(ws, L.groups),
                                     at<int>(ws, L.tok_groups), at<int>(ws, L.group_total),
                                     at<Ctrl>(ws, L.ctrl), st, true);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return run_experts(x, n, experts, nullptr, 1, y, 0, dbg, ws, L, di, n < gcap ? n : gcap, st);
}

static moe_status_t check_layer(const moe_layer_t* layer, int B) {
  if (!layer || B < 0) return MOE_ERR_INVALID_ARG;
  const moe_experts_t& r = layer->routed;
  moe_status_t s = check_dims(r.d, r.f);
  if (s != MOE_OK) return s;
  s = check_experts(&r, r.d, r.f, false);
  if (s != MOE_OK) return s;
  s = check_experts(&layer->shared, r.d, r.f, true);
  if (s != MOE_OK) return s;
  if (layer->shared.E > 8) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (layer->k < 1 || layer->k > r.E) return MOE_ERR_INVALID_ARG;
  if (layer->k > kMaxTok || B > kMaxB) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!layer->w_router) return MOE_ERR_INVALID_ARG;
  if (!aligned(layer->w_router, 16)) return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

// The batched path applies: 16 to 64 tokens, d <= 4096, and at least 6 tokens per routed
// expert on average (B k / E >= 6).  There the general path splits many experts' tokens
// (and every shared expert's) into groups of 8 and reads their kept rows once per group.
// Measured per layer, general against batched: Mixtral-8x7B at 70 %, 16 tokens (4 per
// expert) 474 against 495 us, 32 tokens 720 against 622 us; DeepSeek-V2-Lite at 64 tokens
// (6 per expert) 558 / 530 / 307 against 493 / 490 / 335 us at 0 / 50 / 90 %.
static bool use_batched(const moe_layer_t* layer, int B) {
  return B >= kBatchMinTok && B <= kBatchMaxTok && layer->routed.d <= 4096 &&
         (long long)B * layer->k >= 6LL * layer->routed.E;
}

static WsLayout layer_layout(const moe_layer_t* layer, int B, int sms) {
  const int k = layer->k, E = layer->routed.E, ns = layer->shared.E;
  const int gcap = group_cap(layer->routed.d);
  const int G_max = groups_max_routed(B, E, k, gcap) + ns * ((B + gcap - 1) / gcap);
  WsLayout L = ws_layout(B, B * k, G_max, layer->routed.d, layer->routed.f, sms);
  if (use_batched(layer, B)) {
    const size_t d = layer->routed.d, f = layer->routed.f, S = k + ns, fw = (f + 31) / 32, nseg = E + ns;
    size_t o = L.total;
    auto take = [&](size_t bytes) {
      const size_t at = o;
      o = align_up(o + bytes, kWsAlign);
      return at;
    };
    L.bv = take(4 * (size_t)B * S * f);
    L.bmask = take(4 * (size_t)B * S * fw);
    L.seg_n = take(4 * nseg);
    L.seg_t = take(4 * nseg);
    L.seg_tok = take(4 * nseg * kBatchMaxTok);
    L.seg_slot = take(4 * nseg * kBatchMaxTok);
    L.seg_w = take(4 * nseg * kBatchMaxTok);
    L.seg_col = take(4 * nseg * f);
    L.ht = take(2 * nseg * kBatchMaxTok * 2 * f);  // [nseg][4 groups][f][2][16] halves
    L.ypart = take(4 * (size_t)batch_max_parts((int)f) * B * S * d);
    L.total = o;
  }
  return L;
}

// The decode path applies: shapes it handles and a shared-memory plan that fits.
static bool use_decode_path(const moe_layer_t* layer, int B, const DeviceInfo& di, int& su, int& sr,
                            int& cap, int& umax) {
  const int k = layer->k, P = di.sms;
  cap = decode_list_cap(B, layer->routed.f, k, layer->shared.E, P);
  umax = decode_units_max(B, layer->routed.f, k, layer->shared.E, P);
  return decode_supported(B, layer->routed.d, layer->routed.f, layer->routed.E, k, layer->shared.E, P) &&
         decode_plan(B, layer->routed.d, layer->routed.E, umax, cap, P, di.smem_optin, su, sr);
}

// A few tokens more than the decode path takes run through it two at a time (the
// tokens are independent: routing, experts and RMSNorm act per token); the experts two
// pairs share are then read twice, and it still measured faster than the general path
// up to 6 tokens with at most 16 routed experts (Mixtral-8x7B at 70 %, 4 / 5 / 6 / 7
// tokens: 171 / 218 / 255 / 304 against 216 / 251 / 277 / 308 us; 8 tokens: 340 against
// 329) and up to 4 with more, where every call routes over all of them (DeepSeek-V2-Lite,
// 0 / 50 / 90 %: 4 tokens 138 / 103 / 70 against 170 / 119 / 68 us; 7 tokens 252 / 190 /
// 131 against 239 / 169 / 93).
static bool use_decode_pairs(const moe_layer_t* layer, int B, const DeviceInfo& di) {
  const int pair_max = layer->routed.E <= 16 ? 6 : 4;
  int su = 0, sr = 0, cap = 0, umax = 0;
  return B > 2 && B <= pair_max && !use_decode_path(layer, B, di, su, sr, cap, umax) &&
         use_decode_path(layer, 2, di, su, sr, cap, umax);
}

size_t moe_layer_workspace_bytes(const moe_layer_t* layer, int32_t B) {
  if (check_layer(layer, B) != MOE_OK) return 0;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return 0;
  const size_t t = layer_layout(layer, B, di.sms).total;
  if (!use_decode_pairs(layer, B, di)) return t;
  const size_t t2 = layer_layout(layer, 2, di.sms).total;
  return t > t2 ? t : t2;
}

// The decode path runs as one kernel: the shapes of use_decode_path with d <= 4096 whose
// one-kernel shared-memory plan fits.
static bool use_layer_kernel(const moe_layer_t* layer, int B, const DeviceInfo& di, int umax, int& su,
                             int& sr) {
  return decode_layer_plan(B, layer->routed.d, layer->routed.E, umax, di.smem_optin, su, sr) != 0;
}

int32_t moe_layer_path(const moe_layer_t* layer, int32_t B) {
  moe_status_t s = check_layer(layer, B);
  if (s != MOE_OK) return s;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return MOE_ERR_CUDA;
  int su = 0, sr = 0, cap = 0, umax = 0;
  if (use_decode_pairs(layer, B, di)) return 4;
  if (!(B >= 1 && use_decode_path(layer, B, di, su, sr, cap, umax))) return use_batched(layer, B) ? 3 : 0;
  return use_layer_kernel(layer, B, di, umax, su, sr) ? 2 : 1;
}

// Kept-column entries each up CTA's list holds (16 per unit of its share).
static int decode_kcap(const WsLayout& L, int f, int P) {
  return (int)((((long long)L.G_max * (f / kMTile)) + P - 1) / P) * 16;
}

// Decode-path parameters of one layer call (workspace carving, plan, debug outputs).
static void fill_decode_params(DecodeParams& dp, const uint16_t* x, int B, const moe_layer_t* layer,
                               uint16_t* y, int rmsnorm_out, const moe_debug_t* dbg, void* ws,
                               const WsLayout& L, int P, int su, int sr, int cap, int umax) {
  const int k = layer->k;
  dp = DecodeParams{};
  dp.x = reinterpret_cast<const __half*>(x);
  dp.w_router = reinterpret_cast<const __half*>(layer->w_router);
  dp.B = B;
  dp.d = layer->routed.d;
  dp.f = layer->routed.f;
  dp.k = k;
  dp.renorm = layer->renorm ? 1 : 0;
  dp.n_shared = layer->shared.E;
  dp.routed = to_set(layer->routed);
  if (layer->shared.E > 0) dp.shared = to_set(layer->shared);
  dp.ctrl = at<Ctrl>(ws, L.ctrl);
  dp.groups = at<GroupDesc>(ws, L.groups);
  dp.gmax = L.G_max;
  dp.umax = umax;
  dp.klist = at<int4>(ws, L.klist);
  dp.kcap = decode_kcap(L, layer->routed.f, P);
  dp.cta_total = at<int>(ws, L.cta_total);
  dp.yacc = at<float>(ws, L.yacc);
  dp.P = P;
  dp.list_cap = cap;
  dp.topk_idx = at<int32_t>(ws, L.topk_idx);
  dp.topk_w = at<float>(ws, L.topk_w);
  dp.user_idx = dbg ? dbg->topk_idx : nullptr;
  dp.user_w = dbg ? dbg->topk_w : nullptr;
  dp.n_slots = k + layer->shared.E;
  dp.dbg_v = dbg ? dbg->v : nullptr;
  dp.dbg_mask = dbg ? dbg->mask : nullptr;
  dp.su = su;
  dp.sr = sr;
  dp.y = reinterpret_cast<__half*>(y);
  dp.rmsnorm = rmsnorm_out ? 1 : 0;
}

// The decode path on B = 1 or 2 tokens (use_decode_path holds): one kernel, or the up
// and gather kernels.  ev: record the debug events.
static moe_status_t run_decode(const uint16_t* x, int B, const moe_layer_t* layer, uint16_t* y,
                               int rmsnorm_out, const moe_debug_t* dbg, void* ws, const WsLayout& L,
                               const DeviceInfo& di, int su, int sr, int cap, int umax, cudaStream_t st,
                               bool ev) {
  const moe_debug_t* de = ev ? dbg : nullptr;
  DecodeParams dp;
  fill_decode_params(dp, x, B, layer, y, rmsnorm_out, dbg, ws, L, di.sms, su, sr, cap, umax);
  int lsu = 0, lsr = 0;
  if (use_layer_kernel(layer, B, di, umax, lsu, lsr)) {
    // one kernel: events 0 and 1 mark its start, events 2, 3 and 4 its end
    dp.su = lsu;
    dp.sr = lsr;
    cudaError_t e = record(de, 0, st);
    if (e == cudaSuccess) e = record(de, 1, st);
    if (e == cudaSuccess) e = launch_decode_layer(dp, st, true);
    if (e == cudaSuccess) e = record(de, 2, st);
    if (e == cudaSuccess) e = record(de, 3, st);
    if (e == cudaSuccess) e = record(de, 4, st);
    return cuda_status(e);
  }
  // two kernels: the router runs inside the up kernel and the combination inside the
  // gather kernel: events 0 and 1, and 3 and 4, mark the same points
  cudaError_t e = record(de, 0, st);
  if (e == cudaSuccess) e = record(de, 1, st);
  if (e == cudaSuccess) e = launch_decode_up(dp, st, true);
  if (e == cudaSuccess) e = record(de, 2, st);
  if (e == cudaSuccess) e = launch_decode_gather(dp, st, true);
  if (e == cudaSuccess) e = record(de, 3, st);
  if (e == cudaSuccess) e = record(de, 4, st);
  return cuda_status(e);
}

moe_status_t moe_layer_decode(const uint16_t* x, int32_t B, const moe_layer_t* layer, uint16_t* y,
                              int32_t rmsnorm_out, const moe_debug_t* dbg, void* ws,
                              size_t ws_bytes, void* stream) {
  moe_status_t s = check_layer(layer, B);
  if (s != MOE_OK) return s;
  if (B == 0) return MOE_OK;
  if (!x || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_ALIGNMENT;
  if (!aligned(ws, kWsAlign)) return MOE_ERR_ALIGNMENT;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return MOE_ERR_CUDA;
  const WsLayout L = layer_layout(layer, B, di.sms);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = (cudaStream_t)stream;
  const int k = layer->k;
  int su = 0, sr = 0, cap = 0, umax = 0;
  if (use_decode_path(layer, B, di, su, sr, cap, umax))
    return run_decode(x, B, layer, y, rmsnorm_out, dbg, ws, L, di, su, sr, cap, umax, st, true);
  if (use_decode_pairs(layer, B, di)) {
    // tokens 2i and 2i + 1 (the last one alone for odd B) through the decode path, one
    // call after the other on the workspace; each call's debug outputs at its tokens.
    // Events 0 and 1 before the first call, 2 after it, 3 and 4 after the last.
    if (ws_bytes < layer_layout(layer, 2, di.sms).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    const size_t d = layer->routed.d, f = layer->routed.f, S = k + layer->shared.E, fw = (f + 31) / 32;
    cudaError_t e = record(dbg, 0, st);
    if (e == cudaSuccess) e = record(dbg, 1, st);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    for (int t0 = 0; t0 < B; t0 += 2) {
      const int Bc = B - t0 < 2 ? B - t0 : 2;
      moe_debug_t dc = {};
      if (dbg) {
        dc.topk_idx = dbg->topk_idx ? dbg->topk_idx + (size_t)t0 * k : nullptr;
        dc.topk_w = dbg->topk_w ? dbg->topk_w + (size_t)t0 * k : nullptr;
        dc.v = dbg->v ? dbg->v + (size_t)t0 * S * f : nullptr;
        dc.mask = dbg->mask ? dbg->mask + (size_t)t0 * S * fw : nullptr;
      }
      if (!use_decode_path(layer, Bc, di, su, sr, cap, umax)) return MOE_ERR_UNSUPPORTED_SHAPE;
      s = run_decode(x + (size_t)t0 * d, Bc, layer, y + (size_t)t0 * d, rmsnorm_out, dbg ? &dc : nullptr, ws,
                     layer_layout(layer, Bc, di.sms), di, su, sr, cap, umax, st, false);
      if (s != MOE_OK) return s;
      if (t0 == 0 && record(dbg, 2, st) != cudaSuccess) return MOE_ERR_CUDA;
    }
    e = record(dbg, 3, st);
    if (e == cudaSuccess) e = record(dbg, 4, st);
    return cuda_status(e);
  }
  RouteParams rp = {};
  rp.x = reinterpret_cast<const __half*>(x);
  rp.w_router = reinterpret_cast<const __half*>(layer->w_router);
  rp.B = B;
  rp.d = layer->routed.d;
  rp.E = layer->routed.E;
  rp.k = k;
  rp.renorm = layer->renorm ? 1 : 0;
  rp.n_shared = layer->shared.E;
  rp.group = 1;
  rp.gcap = group_cap(layer->routed.d);
  rp.topk_idx = at<int32_t>(ws, L.topk_idx);
  rp.topk_w = at<float>(ws, L.topk_w);
  rp.user_idx = dbg ? dbg->topk_idx : nullptr;
  rp.user_w = dbg ? dbg->topk_w : nullptr;
  rp.expert_count = nullptr;
  rp.ctrl = at<Ctrl>(ws, L.ctrl);
  rp.groups = at<GroupDesc>(ws, L.groups);
  rp.tok_groups = at<int>(ws, L.tok_groups);
  rp.group_total = at<int>(ws, L.group_total);
  rp.G_max = L.G_max;
  if (record(dbg, 0, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_route(rp, st, true) != cudaSuccess) return MOE_ERR_CUDA;
  const int n_slots = k + layer->shared.E;
  const int max_tok = B < rp.gcap ? B : rp.gcap;
  if (!use_batched(layer, B))
    return run_experts(x, B, &layer->routed, &layer->shared, n_slots, y, rmsnorm_out ? 1 : 0, dbg, ws, L, di,
                       max_tok, st);
  // batched: the up kernel writes dense v and masks into the workspace, then the
  // per-expert kept-row lists, the gate pass, the down pass and the final sum
  ExpertParams p;
  Plan pl;
  s = expert_params(x, B, &layer->routed, &layer->shared, n_slots, y, rmsnorm_out ? 1 : 0, nullptr, ws, L, di,
                    max_tok, p, pl);
  if (s != MOE_OK) return s;
  const size_t f = layer->routed.f, fw = (f + 31) / 32;
  p.dbg_v = at<float>(ws, L.bv);
  p.dbg_mask = at<uint32_t>(ws, L.bmask);
  BatchParams bp = {};
  bp.routed = p.routed;
  bp.shared = p.shared;
  bp.x = p.x;
  bp.B = B;
  bp.d = layer->routed.d;
  bp.f = (int)f;
  bp.k = k;
  bp.n_shared = layer->shared.E;
  bp.n_slots = n_slots;
  bp.topk_idx = rp.topk_idx;
  bp.topk_w = rp.topk_w;
  bp.v = p.dbg_v;
  bp.mask = p.dbg_mask;
  bp.fw = (int)fw;
  bp.seg_n = at<int>(ws, L.seg_n);
  bp.seg_t = at<int>(ws, L.seg_t);
  bp.seg_tok = at<int>(ws, L.seg_tok);
  bp.seg_slot = at<int>(ws, L.seg_slot);
  bp.seg_w = at<float>(ws, L.seg_w);
  bp.seg_col = at<int>(ws, L.seg_col);
  bp.ht = at<__half>(ws, L.ht);
  bp.ypart = at<float>(ws, L.ypart);
  bp.ctrl = at<Ctrl>(ws, L.ctrl);
  bp.y = reinterpret_cast<__half*>(y);
  bp.rmsnorm = rmsnorm_out ? 1 : 0;
  cudaError_t e = record(dbg, 1, st);
  if (e == cudaSuccess) e = launch_up(p, pl.up_grid, st, true);
  if (e == cudaSuccess) e = record(dbg, 2, st);
  if (e == cudaSuccess) e = launch_batched(bp, di.sms, st);
  if (e == cudaSuccess) e = record(dbg, 3, st);
  if (e == cudaSuccess) e = record(dbg, 4, st);
  // the caller's copies of v and the masks
  if (e == cudaSuccess && dbg && dbg->v)
    e = cudaMemcpyAsync(dbg->v, p.dbg_v, 4 * (size_t)B * n_slots * f, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && dbg && dbg->mask)
    e = cudaMemcpyAsync(dbg->mask, p.dbg_mask, 4 * (size_t)B * n_slots * fw, cudaMemcpyDeviceToDevice, st);
  return cuda_status(e);
}

// Staging area of a host-rows call: one 4d-byte row for every entry the up CTAs' lists
// can hold (at least every column of every (token, expert) pair: the dense worst case).
static size_t host_rows_staging_bytes(const moe_layer_t* layer, const WsLayout& L, int P) {
  return (size_t)P * decode_kcap(L, layer->routed.f, P) * 4 * layer->routed.d;
}

size_t moe_layer_host_rows_workspace_bytes(const moe_layer_t* layer, int32_t B) {
  if (check_layer(layer, B) != MOE_OK) return 0;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return 0;
  const WsLayout L = layer_layout(layer, B, di.sms);
  return align_up(L.total, kWsAlign) + host_rows_staging_bytes(layer, L, di.sms);
}

// The device's address of a buffer of `bytes` bytes in page-locked host memory (or in
// device memory): both its first and its last byte must be registered, in one mapping
// (the last byte's device address is the first one's plus the distance), so that every
// row the fetch kernel may read is covered.
static moe_status_t device_view(const __half* p, size_t bytes, const __half*& out) {
  cudaPointerAttributes a, z;
  const char* last = reinterpret_cast<const char*>(p) + (bytes ? bytes - 1 : 0);
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess || cudaPointerGetAttributes(&z, last) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeUnregistered || a.devicePointer == nullptr) return MOE_ERR_INVALID_ARG;
  if (z.type == cudaMemoryTypeUnregistered || z.devicePointer == nullptr) return MOE_ERR_INVALID_ARG;
  if (static_cast<const char*>(z.devicePointer) != static_cast<const char*>(a.devicePointer) + (bytes ? bytes - 1 : 0))
    return MOE_ERR_INVALID_ARG;
  out = reinterpret_cast<const __half*>(a.devicePointer);
  return MOE_OK;
}

// gate_t and down of a set: E * f rows of rs elements each from the buffer start (an
// interleaved down buffer starts d elements later and ends where gate_t ends).
static moe_status_t device_view_rows(ExpertSet& es) {
  const size_t span = (size_t)es.E * es.f * es.rs * sizeof(__half);
  const size_t down_off = (size_t)(es.down - es.gate_t) * sizeof(__half);
  const bool inter = es.rs == 2 * es.d;
  moe_status_t s = device_view(es.gate_t, span, es.gate_t);
  if (s == MOE_OK) s = device_view(es.down, inter ? span - down_off : span, es.down);
  return s;
}

moe_status_t moe_layer_decode_host_rows(const uint16_t* x, int32_t B, const moe_layer_t* layer,
                                        uint16_t* y, int32_t rmsnorm_out, const moe_debug_t* dbg,
                                        void* ws, size_t ws_bytes, void* stream) {
  moe_status_t s = check_layer(layer, B);
  if (s != MOE_OK) return s;
  if (B == 0) return MOE_OK;
  if (!x || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return MOE_ERR_ALIGNMENT;
  if (!aligned(ws, kWsAlign)) return MOE_ERR_ALIGNMENT;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return MOE_ERR_CUDA;
  const WsLayout L = layer_layout(layer, B, di.sms);
  const size_t off_staging = align_up(L.total, kWsAlign);
  if (ws_bytes < off_staging + host_rows_staging_bytes(layer, L, di.sms)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int P = di.sms;
  int su = 0, sr = 0, cap = 0, umax = 0;
  if (!use_decode_path(layer, B, di, su, sr, cap, umax)) return MOE_ERR_UNSUPPORTED_SHAPE;
  DecodeParams dp;
  fill_decode_params(dp, x, B, layer, y, rmsnorm_out, dbg, ws, L, P, su, sr, cap, umax);
  s = device_view_rows(dp.routed);
  if (s == MOE_OK && layer->shared.E > 0) s = device_view_rows(dp.shared);
  if (s != MOE_OK) return s;
  dp.staging = at<uint8_t>(ws, off_staging);
  cudaStream_t st = (cudaStream_t)stream;
  // up kernel, fetch kernel, gather kernel; event 2 marks the start of the fetch
  cudaError_t e = record(dbg, 0, st);
  if (e == cudaSuccess) e = record(dbg, 1, st);
  if (e == cudaSuccess) e = launch_decode_up(dp, st, true);
  if (e == cudaSuccess) e = record(dbg, 2, st);
  if (e == cudaSuccess) e = launch_decode_fetch(dp, st, true);
  if (e == cudaSuccess) e = launch_decode_gather(dp, st, true);
  if (e == cudaSuccess) e = record(dbg, 3, st);
  if (e == cudaSuccess) e = record(dbg, 4, st);
  return cuda_status(e);
}

moe_status_t moe_prefetch_experts(const moe_experts_t* experts, const int32_t* idx, int32_t n,
                                  size_t max_bytes, void* stream) {
  if (!experts || n < 0) return MOE_ERR_INVALID_ARG;
  if (n > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_status_t s = check_dims(experts->d, experts->f);
  if (s != MOE_OK) return s;
  if (experts->E < 1 || experts->E > 256) return experts->E < 0 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED_SHAPE;
  if (!experts->up_packed) return MOE_ERR_INVALID_ARG;
  if (!aligned(experts->up_packed, 16)) return MOE_ERR_ALIGNMENT;
  if (n == 0) return MOE_OK;
  if (!idx) return MOE_ERR_INVALID_ARG;
  if (!aligned(idx, 4)) return MOE_ERR_ALIGNMENT;
  const size_t per = packed_bytes_per_expert(experts->d, experts->f);
  long long max_experts = 256;
  if (max_bytes > 0) max_experts = (long long)(max_bytes / per);
  if (max_experts == 0) return MOE_OK;
  DeviceInfo di;
  if (device_info(di) != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_expert_prefetch(reinterpret_cast<const uint8_t*>(experts->up_packed), per,
                                            experts->E, idx, n, (int)(max_experts > 256 ? 256 : max_experts),
                                            di.sms, (cudaStream_t)stream));
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, kWsAlign)) return MOE_ERR_ALIGNMENT;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

moe_status_t moe_get_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  int status = 0;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws);  // the control block is always first
  if (cudaMemcpy(&status, &ctrl->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (status != 0) {
    const int zero = 0;
    if (cudaMemcpy(&ctrl->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return status;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_OOM: return "out of memory";
    default: return "unknown status";
  }
}

}  // extern "C"
