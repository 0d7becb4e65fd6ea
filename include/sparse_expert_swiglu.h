/*
 * sparse_expert_swiglu.h -- C ABI of the GB300 (sm_103a) decode-time MoE library
 * with contextually sparse SwiGLU experts.
 *
 * What it computes (page title, section):
 *   - "FloE: On-the-Fly MoE Inference on Memory-constrained GPU", sec. 三
 *     "MoE 专家前向计算": a SwiGLU expert a_E(x) = (SiLU(x W^gate) (.) x W^up) W^down;
 *     "混合压缩策略": W^up stored INT2, W^gate / W^down sparsified by activation;
 *     "系统协同优化", Algorithm 1 "Efficient Sparse Kernel":
 *        v = x W^up;  mask = |v| > t_ij;  x' = SiLU(x W^gate[:, mask]) (.) v[mask];
 *        out = x' W^down[mask, :]
 *     with W^down stored transposed (one contiguous d-vector per intermediate
 *     column), only selected columns loaded, SiLU fused with the product.
 *   - "MoE-Lightning: High-Throughput MoE Inference on Memory-constrained GPUs",
 *     sec. 三 "MoE 模型架构": a gating network chooses the top-k experts of each
 *     token; "MOE-INFINITY ...", sec. A3 background: Mixtral-8x7B has 8 experts
 *     and routes each token to 2 of them.
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller, unless the
 *     comment says "host".  The library allocates nothing; all scratch lives in the
 *     caller's workspace, except the static scratch of moe_route_topk_noalloc.
 *   - fp16 tensors are IEEE binary16 bit patterns passed as uint16_t.  All
 *     arrays are dense, row-major, and start on a 16-byte boundary.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it and returns without
 *     synchronising, except moe_get_status().
 *   - Return value: MOE_OK (0) or a negative moe_status_t.  Argument errors
 *     are detected on the host before anything is enqueued.  Errors found on
 *     the device (a bounded wait that ran out) are recorded in the workspace
 *     and reported by moe_get_status().
 *   - Thread safety: calls may be made from several host threads as long as
 *     concurrent calls use different workspaces.
 */
#ifndef SPARSE_EXPERT_SWIGLU_H
#define SPARSE_EXPERT_SWIGLU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int moe_status_t;
enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,        /* NULL where a pointer is required, negative size, k > E ... */
  MOE_ERR_UNSUPPORTED_SHAPE = -2,  /* see "Shape limits" below */
  MOE_ERR_ALIGNMENT = -3,          /* a pointer is not 16-byte aligned (workspace: 256-byte) */
  MOE_ERR_WORKSPACE_TOO_SMALL = -4,
  MOE_ERR_CUDA = -5,               /* a CUDA runtime call or a launch failed */
  MOE_ERR_TIMEOUT = -6,            /* a bounded device-side wait ran out (moe_get_status) */
  MOE_ERR_OOM = -7
};

/*
 * Shape limits (MOE_ERR_UNSUPPORTED_SHAPE otherwise):
 *   hidden size d: multiple of 256, 256 <= d <= 7936
 *   intermediate size f (per expert): multiple of 16, 16 <= f <= 65536
 *   routed experts E: 1..256; top-k: 1 <= k <= min(E, 8); shared experts: 0..8
 *   tokens per call B (or n): 0..1024 (0 is a no-op that returns MOE_OK)
 */

/* One stack of equally shaped experts of one layer. */
typedef struct {
  int32_t E;                 /* number of experts in the stack */
  int32_t d;                 /* hidden size */
  int32_t f;                 /* intermediate size of one expert */
  const void* up_packed;     /* [E][expert_int2_up_packed_bytes(d, f)] from expert_pack_int2_up */
  const uint16_t* gate_t;    /* fp16 [E][f][d]: row i = column i of W^gate */
  const uint16_t* down;      /* fp16 [E][f][d]: row i = row i of W^down (the transposed,
                                column-major W^down of FloE's kernel optimisation list).
                                Interleaved form: one buffer [E][f][2][d] holding gate row i
                                then down row i; pass gate_t = buffer, down = buffer + d.
                                The two rows of a kept column are then one contiguous read. */
  const float* thr;          /* fp32 [E]: threshold t_ij of Algorithm 1, one per expert */
} moe_experts_t;

/* One MoE layer. */
typedef struct {
  int32_t k;                 /* experts per token */
  int32_t renorm;            /* 1: weights = softmax over the k chosen logits;
                                0: full softmax over E, read at the chosen experts */
  const uint16_t* w_router;  /* fp16 [d][E] router (gating network) weight */
  moe_experts_t routed;      /* routed experts */
  moe_experts_t shared;      /* always-on shared experts, weight 1 (E = 0: none);
                                same d and f as `routed` */
} moe_layer_t;

/* Optional outputs of moe_layer_decode / moe_expert_sparse_swiglu for tests and
 * inspection.  Any member may be NULL.  S = k + shared.E (1 for the single-expert
 * call); slot j < k is the token's j-th routed expert, slot k + s shared expert s. */
typedef struct {
  int32_t* topk_idx;   /* [B][k] chosen experts, by logit descending, ties to the lower index */
  float* topk_w;       /* [B][k] combine weights */
  uint32_t* mask;      /* [B][S][ceil(f/32)] bit i%32 of word i/32 = (|v_i| > t) */
  float* v;            /* [B][S][f] fp32 v = x W~^up (step 1 of Algorithm 1) */
  void** events;       /* 5 cudaEvent_t (as void*), recorded on `stream` before the router
                          (or the single-expert set-up), before the up-projection kernel,
                          before the gather kernel, before the combine kernel and after it;
                          for per-kernel timing.  Recording them serialises the kernels.
                          On the decode path (moe_layer_decode with 1 or 2 tokens) the
                          router runs inside the up-projection kernel and the combination
                          inside the gather kernel: events 0 and 1, and events 3 and 4,
                          are recorded back to back. */
} moe_debug_t;

/* ---------------- INT2 up projection ---------------- */

/* Bytes of one packed expert: (f/16) * ceil(d/512) * 2560.  0 for unsupported shapes. */
size_t expert_int2_up_packed_bytes(int32_t d, int32_t f);

/*
 * expert_pack_int2_up -- quantise one W^up to INT2 (FloE "混合压缩策略": Q(.) on the
 * up projection) and store it in the layout the expert kernels read.
 *   w_up      fp16 [d][f] (x . W^up gives the f intermediate values); finite values
 *   up_packed out, expert_int2_up_packed_bytes(d, f) bytes
 * Scheme (the pages name only "INT2"): one fp16 (scale, zero) per 64-row group and
 * column, computed with fp32 IEEE operations:
 *   scale = fp16((max - min) / 3), replaced by 1 if it rounds to 0;
 *   zero  = fp16(clamp(-min / scale, +-65504));  q = clamp(rint(w / scale + zero), 0, 3)
 * and W~^up = scale * (q - zero).  Deterministic: the same input gives the same bytes.
 */
moe_status_t expert_pack_int2_up(const uint16_t* w_up, int32_t d, int32_t f, void* up_packed,
                                 void* stream);

/*
 * expert_unpack_int2_up -- inverse of the storage step of expert_pack_int2_up, for
 * tests and inspection: writes the codes q uint8 [d][f] (values 0..3), scale and
 * zero fp16 [d/64][f].  Any of the three outputs may be NULL.
 */
moe_status_t expert_unpack_int2_up(const void* up_packed, int32_t d, int32_t f, uint8_t* q,
                                   uint16_t* scale, uint16_t* zero, void* stream);

/* ---------------- routing ---------------- */

/*
 * moe_route_topk -- router GEMV and softmax top-k of every token (MoE-Lightning
 * sec. 三 "MoE 模型架构"; MOE-INFINITY sec. A3).
 *   x        fp16 [B][d];  w_router fp16 [d][E]
 *   topk_idx out int32 [B][k]: experts by logit descending, equal logits to the lower index
 *   topk_w   out fp32 [B][k]: renorm ? softmax over the k chosen logits
 *                                   : full softmax over E at the chosen experts
 *   expert_count out int32 [E] or NULL: tokens routed to each expert (one row of
 *            MOE-INFINITY's iteration-level expert activation matrix)
 *   ws / ws_bytes: workspace of at least moe_route_workspace_bytes(B, E, k) bytes,
 *            256-byte aligned, zero-filled once before its first use (moe_workspace_init).
 */
size_t moe_route_workspace_bytes(int32_t B, int32_t E, int32_t k);
moe_status_t moe_route_topk(const uint16_t* x, int32_t B, int32_t d, const uint16_t* w_router,
                            int32_t E, int32_t k, int32_t renorm, int32_t* topk_idx, float* topk_w,
                            int32_t* expert_count, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_route_topk_noalloc -- moe_route_topk without a caller workspace.  The
 * papers have no counterpart to this call: it is a deployment convenience.
 * It serves callers that cannot allocate device memory (a plugin given only its
 * input and output pointers, a runtime with a fixed memory pool, a path where an
 * allocation would synchronise the device).  Its scratch is a static device array
 * inside the library, one per device, sized for at most
 * MOE_ROUTE_NOALLOC_MAX_PAIRS = B * k (token, expert) pairs.
 *   Arguments, layouts and results are those of moe_route_topk.
 *   B * k > MOE_ROUTE_NOALLOC_MAX_PAIRS: MOE_ERR_WORKSPACE_TOO_SMALL, nothing enqueued.
 *   The first call on a device looks up the scratch address (with that device
 *   current); make it before capturing a stream.  The address is kept per device and
 *   context: the first call in a context created later on the device (after
 *   cudaDeviceReset, say) looks it up again.  Every call clears the scratch's
 *   control block on `stream` before the kernel.  Calls that overlap in time on
 *   one device (different streams or host threads) share the scratch and race:
 *   order them on one stream.
 */
#define MOE_ROUTE_NOALLOC_MAX_PAIRS 2048
moe_status_t moe_route_topk_noalloc(const uint16_t* x, int32_t B, int32_t d,
                                    const uint16_t* w_router, int32_t E, int32_t k,
                                    int32_t renorm, int32_t* topk_idx, float* topk_w,
                                    int32_t* expert_count, void* stream);

/* ---------------- one expert ---------------- */

/*
 * moe_expert_sparse_swiglu -- Algorithm 1 of FloE for one expert of `experts` on n
 * tokens, weight 1:  y[b] = sum over i with |v_bi| > thr[e] of
 *                           SiLU(x_b . gate_t[e][i]) * v_bi * down[e][i][:]
 * with v = x . W~^up (dequantised INT2).  Only the gate and down rows of kept
 * columns are read.  fp32 accumulation; y is rounded to fp16 once.
 *   x  fp16 [n][d];  y out fp16 [n][d];  dbg: optional (topk members unused; S = 1)
 *   ws / ws_bytes: at least moe_expert_workspace_bytes(n, d, f) bytes, 256-byte
 *   aligned, zero-filled once before its first use (moe_workspace_init).
 */
size_t moe_expert_workspace_bytes(int32_t n, int32_t d, int32_t f);
moe_status_t moe_expert_sparse_swiglu(const uint16_t* x, int32_t n, const moe_experts_t* experts,
                                      int32_t expert, uint16_t* y, const moe_debug_t* dbg, void* ws,
                                      size_t ws_bytes, void* stream);

/* ---------------- one layer ---------------- */

/*
 * moe_layer_decode -- one MoE decode layer on B tokens:
 *   y[b] = sum_j topk_w[b][j] * E_{topk_idx[b][j]}(x[b]) + sum_s E^shared_s(x[b])
 * where every expert is the sparse SwiGLU expert above (routed and shared experts
 * use their own thresholds).  With rmsnorm_out = 1 the result is replaced by
 * y / sqrt(mean(y^2) + 1e-6) (unit weight) before the fp16 rounding: the hidden
 * state handed to the next layer of a stack.  Routing stays on the device.
 *   x fp16 [B][d];  y out fp16 [B][d] (may not alias x);  layer: host pointer to the
 *   description (its tensor members are device pointers);  dbg: optional.
 *   ws / ws_bytes: at least moe_layer_workspace_bytes(layer, B) bytes, 256-byte
 *   aligned, zero-filled once before its first use (moe_workspace_init).  Calls with
 *   different B may share a workspace that is large enough for each of them.
 */
size_t moe_layer_workspace_bytes(const moe_layer_t* layer, int32_t B);
moe_status_t moe_layer_decode(const uint16_t* x, int32_t B, const moe_layer_t* layer, uint16_t* y,
                              int32_t rmsnorm_out, const moe_debug_t* dbg, void* ws,
                              size_t ws_bytes, void* stream);

/*
 * moe_layer_path -- which kernels moe_layer_decode runs for this layer and B tokens on
 * the current device: 2 = the one-kernel decode path (one token, 8/16/32/64 routed
 * experts, d <= 4096: one kernel routes, projects, thresholds, gathers the kept rows
 * and combines), 1 = the two-kernel decode path (two tokens with those experts and
 * d <= 6144, or one token with 4096 < d <= 6144: an up-projection kernel that also
 * routes and a gather kernel that also combines), 3 = the batched path (16 to 64
 * tokens, d <= 4096, B k >= 6 E: the router and the up-projection kernel, then per expert the
 * union of its tokens' masks as one kept-row list, a gate pass and a down pass that read
 * every kept row once per expert, and a per-token sum; bitwise reproducible), 4 = the
 * decode path in pairs (three to six tokens of a shape that paths 1 and 2 take, three
 * or four with more than 16 routed experts: tokens
 * 2i and 2i + 1 through the decode path, one call after the other, the last token of an
 * odd count alone; the tokens are independent, and two pairs that route to one expert
 * read its rows twice), 0 = the general path (router, up-projection, gather and combine
 * kernels), or a negative moe_status_t for an invalid layer.  Every path computes the
 * same layer.  The general path is bitwise reproducible; on the decode paths the CTAs'
 * shares reach the fp32 sum of y in a varying order, so two calls can differ in the
 * last bits of that sum (at most one fp16 ulp of y).
 */
int32_t moe_layer_path(const moe_layer_t* layer, int32_t B);

/*
 * moe_layer_decode_host_rows -- moe_layer_decode with the experts' gate and down rows
 * in page-locked host memory: FloE's on-the-fly setting ("FloE: On-the-Fly MoE
 * Inference on Memory-constrained GPU", sec. 三 "系统协同优化"), where only the compressed
 * up projection stays in GPU memory and only the rows that the masks keep are brought
 * over.  Same arguments and result as moe_layer_decode, except:
 *   layer: the router weight, up_packed and thr of both expert sets are device
 *     pointers; gate_t and down (routed and shared) are host pointers to memory from
 *     cudaHostAlloc / cudaMallocHost or registered with cudaHostRegister (device
 *     pointers are accepted too), the whole extent of each (E * f rows) in one mapping;
 *     any other memory, or a buffer registered only in part, returns MOE_ERR_INVALID_ARG.
 *   ws / ws_bytes: at least moe_layer_host_rows_workspace_bytes(layer, B) bytes: the
 *     workspace of moe_layer_decode followed by a staging area for the kept rows (4d
 *     bytes per row, room for at least (B k + shared E) f rows: the dense worst case).
 * Only the decode shapes are supported (moe_layer_path(layer, B) == 1 or 2; the
 * two-kernel form runs either way); other shapes return MOE_ERR_UNSUPPORTED_SHAPE.
 * Three kernels run: the up-projection kernel, a
 * fetch kernel that copies each kept row (4d bytes) from host memory into the staging
 * area, and the gather kernel, which streams the staging area.  dbg->events[2] marks
 * the start of the fetch kernel.  The host rows must not change while the call runs.
 */
size_t moe_layer_host_rows_workspace_bytes(const moe_layer_t* layer, int32_t B);
moe_status_t moe_layer_decode_host_rows(const uint16_t* x, int32_t B, const moe_layer_t* layer,
                                        uint16_t* y, int32_t rmsnorm_out, const moe_debug_t* dbg,
                                        void* ws, size_t ws_bytes, void* stream);

/*
 * moe_prefetch_experts -- the data movement behind an inter-expert predictor ("FloE:
 * On-the-Fly MoE Inference on Memory-constrained GPU", sec. "双稀疏预测器", Inter-expert
 * Predictor).  FloE's predictor guesses a later layer's experts from an earlier hidden
 * state.  The page gives its core observation: consecutive MoE layers' hidden states
 * have cosine similarity above 0.95.  This call L2-prefetches the packed up projections
 * of the predicted experts, the part that every token routed to an expert reads whole,
 * so that the layer's up-projection reads hit in L2.  The prediction is the caller's:
 * a trained predictor, or moe_route_topk on the current hidden state with the next
 * layer's router weight.  The call only enqueues bulk L2 prefetches on `stream` and
 * returns.  No result of any call changes; only timing can.
 *   experts    the expert stack of the layer that the prediction is for (d, f, E and
 *              up_packed are read; gate_t, down and thr are not)
 *   idx        device int32 [n]: predicted expert ids; repeats and ids outside [0, E)
 *              are ignored
 *   n          0..1024 (0: nothing is enqueued, idx may be NULL)
 *   max_bytes  prefetch whole experts in ascending id order while the total stays
 *              <= max_bytes (0: no limit); GB300's L2 holds 129 MB
 *   stream     cudaStream_t or NULL.  The kernel uses one warp per SM and no workspace,
 *              so it can run on a second stream beside a decode layer
 * Errors: MOE_ERR_INVALID_ARG (experts NULL, n < 0, up_packed NULL, idx NULL with
 * n > 0), MOE_ERR_UNSUPPORTED_SHAPE (n > 1024, E outside 1..256, d or f outside the
 * shape limits), MOE_ERR_ALIGNMENT (up_packed not 16-byte or idx not 4-byte aligned),
 * MOE_ERR_CUDA.  Argument errors are found before any CUDA call.
 */
moe_status_t moe_prefetch_experts(const moe_experts_t* experts, const int32_t* idx, int32_t n,
                                  size_t max_bytes, void* stream);

/* ---------------- expert activation tracking and expert cache (host) ----------------
 *
 * "MoE-Infinity" (sec. 4.3, 4.5, 4.7 Algorithm 1 "专家缓存检索", appendix B.1): request-level
 * expert activation matrices, their collection, the activation prediction from it and
 * the sparsity-aware expert cache.  Host functions on caller-owned host memory (no GPU,
 * no allocation, no internal locking: one thread per structure at a time).
 *
 * An EAM is int32 [L][E], row-major: cell [i][j] = tokens routed to expert j of MoE layer
 * i.  One iteration's row i is the expert_count that moe_route_topk returns for layer i;
 * a request's EAM is the sum over its iterations (moe_eam_add_counts).
 */

/* eam[layer][j] += counts[j] for j < E. */
moe_status_t moe_eam_add_counts(int32_t* eam, int32_t L, int32_t E, int32_t layer, const int32_t* counts);

/*
 * EAMC: at most `capacity` past request EAMs.  moe_eamc_bytes sizes the caller's buffer
 * (0 for invalid sizes); moe_eamc_init formats it (empty).  moe_eamc_insert appends
 * `ream` while there is room, else overwrites the stored entry nearest to it (smallest
 * cosine distance of the flattened matrices; ties: the lowest index); *slot (optional)
 * receives the index written.  moe_eamc_size returns the entry count (negative status
 * for an invalid buffer); moe_eamc_entry copies entry i out.
 */
size_t moe_eamc_bytes(int32_t L, int32_t E, int32_t capacity);
moe_status_t moe_eamc_init(void* eamc, size_t bytes, int32_t L, int32_t E, int32_t capacity);
moe_status_t moe_eamc_insert(void* eamc, const int32_t* ream, int32_t* slot);
int32_t moe_eamc_size(const void* eamc);
moe_status_t moe_eamc_entry(const void* eamc, int32_t i, int32_t* eam);

/*
 * moe_eamc_match -- the n_match stored entries nearest to `cur` (cosine distance
 * 1 - a.b / (|a| |b|) in double, 1 when either matrix is all zero), by (distance,
 * index) ascending: idx[n_match] and dist[n_match]; slots past the entry count get -1
 * and +inf; *n_found (optional) = entries returned.
 *
 * moe_eamc_predict -- PredictEAM for current layer `layer` (0 <= layer < L): the nearest
 * n_match entries (1 <= n_match <= 1024) summed cell by cell, each row normalised to sum
 * 1 (rows summing to 0 stay 0), row i multiplied by 1 - (i - layer) / L.
 * p_eam: double [L][E] out.  An empty EAMC predicts all zeros.
 */
moe_status_t moe_eamc_match(const void* eamc, const int32_t* cur, int32_t n_match, int32_t* idx,
                            double* dist, int32_t* n_found);
moe_status_t moe_eamc_predict(const void* eamc, const int32_t* cur, int32_t layer, int32_t n_match,
                              double* p_eam);

/*
 * Expert cache (Algorithm 1): at most `capacity` experts, identified by (layer, expert),
 * kept in insertion order.  moe_expert_cache_lookup requests expert `expert` of layer
 * `layer`, the layer now running, with `cur` the current EAM:
 *   hit            -> *hit = 1, nothing changes;
 *   miss, room     -> *hit = 0, the expert is appended (the caller fetches it);
 *   miss, full     -> *hit = 0; p = moe_eamc_predict(eamc, cur, layer, n_match); the cached
 *                     expert e with the smallest (p[e.layer][e.expert] + eps) / n_token *
 *                     (1 - e.layer / L), n_token = sum of row e.layer of p (1 where that
 *                     row sums to 0), is removed (ties: the earliest inserted) and the
 *                     requested expert appended.
 * evicted[2] receives the removed (layer, expert), or (-1, -1).  The EAMC must have the
 * cache's L and E; a miss on a full cache needs L * E <= 4096 and n_match <= 1024
 * (MOE_ERR_UNSUPPORTED_SHAPE otherwise, nothing changed).  moe_expert_cache_contents copies the (layer, expert) pairs in
 * insertion order to layer_expert[2 * n] (optional) and sets *n.
 */
size_t moe_expert_cache_bytes(int32_t capacity);
moe_status_t moe_expert_cache_init(void* cache, size_t bytes, int32_t capacity, int32_t L, int32_t E);
moe_status_t moe_expert_cache_lookup(void* cache, const void* eamc, const int32_t* cur, int32_t layer,
                                     int32_t expert, int32_t n_match, double eps, int32_t* hit,
                                     int32_t* evicted);
moe_status_t moe_expert_cache_contents(const void* cache, int32_t* layer_expert, int32_t* n);

/* ---------------- workspace and status ---------------- */

/* Zero-fills `ws` on `stream` (required once after allocating a workspace). */
moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, then returns and clears the first device-side error
 * recorded in `ws` since the last call (MOE_OK if none; MOE_ERR_CUDA if the
 * synchronisation itself failed).
 */
moe_status_t moe_get_status(void* ws, void* stream);

/* Static string for a status code. */
const char* moe_status_string(moe_status_t status);

/*
 * moe_selftest_wait_timeout -- diagnostic of the timeout path of every kernel: enqueues
 * on `stream` one thread that waits on a barrier nothing completes, for at most `tries`
 * (1..4000) try_wait rounds of at most about 1 ms each, then records MOE_ERR_TIMEOUT in
 * `ws` the way the kernels do.  moe_get_status then returns MOE_ERR_TIMEOUT (and clears
 * it); the context stays usable.  ws: any workspace of this library (its control block
 * is first), 256-byte aligned.  Nothing faults or hangs.
 */
moe_status_t moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t tries, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_EXPERT_SWIGLU_H */
