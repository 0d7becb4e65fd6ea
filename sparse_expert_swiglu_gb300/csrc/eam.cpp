// Expert activation tracking and the sparsity-aware expert cache of "MOE-INFINITY:
// Efficient MoE Inference on Personal Machines with Sparsity-Aware Expert Cache" (sec. 4.3
// "解码过程中激活预测的形式化", 4.5 "请求级稀疏激活追踪", 4.7 Algorithm 1 "专家缓存检索",
// appendix B.1 "预测器运行时效率").  Host code: the data structures live in caller-owned host
// memory; nothing is allocated here.
//
//   EAM       L x E int32 matrix, cell [i][j] = tokens routed to expert j of MoE layer i.
//             A request's EAM (rEAM) is the sum of its iterations' EAMs (iEAM); one row of
//             an iEAM is exactly the per-expert token count that moe_route_topk returns.
//   EAMC      a fixed-capacity collection of past rEAMs.  A new entry is appended while
//             there is room, else it replaces the stored entry nearest to it (cosine
//             distance of the flattened matrices).
//   PredictEAM the entries nearest to the current EAM are summed cell by cell, every row
//             is normalised to sum 1, and row i is scaled by 1 - (i - l)/L for the current
//             layer l.
//   cache     Algorithm 1: on a miss with a full cache, the cached expert e with the
//             smallest (p[e.layer][e.expert] + eps) / n_token * (1 - e.layer / L) is
//             evicted, n_token being the sum of row e.layer of the prediction.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "../../include/sparse_expert_swiglu.h"

namespace {

constexpr int32_t kEamcMagic = 0x45414d43;   // "EAMC"
constexpr int32_t kCacheMagic = 0x45434348;  // "ECCH"

struct EamcHeader {
  int32_t magic, L, E, capacity, size, pad[3];
};
struct CacheHeader {
  int32_t magic, capacity, L, E, size, pad[3];
};

// Layout: header, then the entries cell-major, int32 [L * E][capacity] (cell t of entry i
// at t * capacity + i, so that one cell of all entries is contiguous), then the entries'
// squared norms, int64 [capacity].
size_t eamc_entries_bytes(int64_t L, int64_t E, int64_t capacity) {
  return ((size_t)(capacity * L * E) * sizeof(int32_t) + 7) & ~(size_t)7;
}
size_t eamc_bytes(int64_t L, int64_t E, int64_t capacity) {
  return sizeof(EamcHeader) + eamc_entries_bytes(L, E, capacity) + (size_t)capacity * sizeof(int64_t);
}

int32_t* eamc_cells(EamcHeader* h) { return reinterpret_cast<int32_t*>(h + 1); }
const int32_t* eamc_cells(const EamcHeader* h) { return reinterpret_cast<const int32_t*>(h + 1); }
int32_t eamc_cell(const EamcHeader* h, int32_t i, int t) { return eamc_cells(h)[(size_t)t * h->capacity + i]; }
int64_t* eamc_norms(EamcHeader* h) {
  return reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(h + 1) + eamc_entries_bytes(h->L, h->E, h->capacity));
}
const int64_t* eamc_norms(const EamcHeader* h) {
  return reinterpret_cast<const int64_t*>(reinterpret_cast<const uint8_t*>(h + 1) +
                                          eamc_entries_bytes(h->L, h->E, h->capacity));
}

const EamcHeader* eamc_of(const void* p) {
  const EamcHeader* h = reinterpret_cast<const EamcHeader*>(p);
  return (h && h->magic == kEamcMagic) ? h : nullptr;
}

// Exact squared norm of a flattened EAM.
int64_t sqnorm(const int32_t* a, int n) {
  int64_t s = 0;
  for (int t = 0; t < n; ++t) s += (int64_t)a[t] * a[t];
  return s;
}

// Cosine distance 1 - a.b / (|a| |b|) from the exact integer products, in double; 1 when
// either matrix is all zero (no direction to compare).
double cosine_distance(int64_t ab, int64_t aa, int64_t bb) {
  if (aa == 0 || bb == 0) return 1.0;
  return 1.0 - (double)ab / (sqrt((double)aa) * sqrt((double)bb));
}

// The n nearest entries to cur, by (distance, index) ascending; returns how many.  The
// dot products of a block of 256 entries accumulate cell by cell over cur's nonzero
// cells (a contiguous run of the block per cell).  Token counts are integers far below
// 2^26, so every product and partial sum is an integer below 2^53: exact in double.
int nearest(const EamcHeader* h, const int32_t* cur, int n, int32_t* idx, double* dist) {
  constexpr int kBlock = 256;
  const int cells = h->L * h->E;
  const int64_t cc = sqnorm(cur, cells);
  const int64_t* norms = eamc_norms(h);
  const int32_t* data = eamc_cells(h);
  int m = 0;
  double acc[kBlock];
  for (int32_t b = 0; b < h->size; b += kBlock) {
    const int nb = h->size - b < kBlock ? h->size - b : kBlock;
    for (int u = 0; u < nb; ++u) acc[u] = 0.0;
    for (int t = 0; t < cells; ++t) {
      if (cur[t] == 0) continue;
      const double ct = (double)cur[t];
      const int32_t* col = data + (size_t)t * h->capacity + b;
      for (int u = 0; u < nb; ++u) acc[u] += ct * (double)col[u];
    }
    for (int u = 0; u < nb; ++u) {
      const int32_t i = b + u;
      const double di = cosine_distance((int64_t)acc[u], cc, norms[i]);
      // insertion into the sorted prefix [0, m) of at most n entries
      int pos = m;
      while (pos > 0 && dist[pos - 1] > di) --pos;  // equal distances keep the lower index first
      if (pos >= n) continue;
      const int last = m < n ? m : n - 1;
      for (int t = last; t > pos; --t) {
        dist[t] = dist[t - 1];
        idx[t] = idx[t - 1];
      }
      dist[pos] = di;
      idx[pos] = i;
      if (m < n) ++m;
    }
  }
  return m;
}

}  // namespace

extern "C" {

size_t moe_eamc_bytes(int32_t L, int32_t E, int32_t capacity) {
  if (L < 1 || E < 1 || capacity < 1) return 0;
  return eamc_bytes(L, E, capacity);
}

moe_status_t moe_eamc_init(void* eamc, size_t bytes, int32_t L, int32_t E, int32_t capacity) {
  if (!eamc || L < 1 || E < 1 || capacity < 1) return MOE_ERR_INVALID_ARG;
  if (bytes < eamc_bytes(L, E, capacity)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  EamcHeader* h = reinterpret_cast<EamcHeader*>(eamc);
  memset(h, 0, sizeof(*h));
  h->magic = kEamcMagic;
  h->L = L;
  h->E = E;
  h->capacity = capacity;
  h->size = 0;
  return MOE_OK;
}

int32_t moe_eamc_size(const void* eamc) {
  const EamcHeader* h = eamc_of(eamc);
  return h ? h->size : MOE_ERR_INVALID_ARG;
}

moe_status_t moe_eamc_entry(const void* eamc, int32_t i, int32_t* eam) {
  const EamcHeader* h = eamc_of(eamc);
  if (!h || !eam || i < 0 || i >= h->size) return MOE_ERR_INVALID_ARG;
  for (int t = 0; t < h->L * h->E; ++t) eam[t] = eamc_cell(h, i, t);
  return MOE_OK;
}

moe_status_t moe_eamc_insert(void* eamc, const int32_t* ream, int32_t* slot) {
  EamcHeader* h = const_cast<EamcHeader*>(eamc_of(eamc));
  if (!h || !ream) return MOE_ERR_INVALID_ARG;
  int32_t s = h->size;
  if (h->size == h->capacity) {
    // replace the stored entry nearest to the new one (ties: the lowest index)
    int32_t i0 = 0;
    double d0 = 0.0;
    (void)nearest(h, ream, 1, &i0, &d0);
    s = i0;
  } else {
    ++h->size;
  }
  int32_t* data = eamc_cells(h);
  for (int t = 0; t < h->L * h->E; ++t) data[(size_t)t * h->capacity + s] = ream[t];
  eamc_norms(h)[s] = sqnorm(ream, h->L * h->E);
  if (slot) *slot = s;
  return MOE_OK;
}

moe_status_t moe_eamc_match(const void* eamc, const int32_t* cur, int32_t n_match, int32_t* idx,
                            double* dist, int32_t* n_found) {
  const EamcHeader* h = eamc_of(eamc);
  if (!h || !cur || !idx || !dist || n_match < 1) return MOE_ERR_INVALID_ARG;
  const int m = nearest(h, cur, n_match, idx, dist);
  for (int t = m; t < n_match; ++t) {
    idx[t] = -1;
    dist[t] = INFINITY;
  }
  if (n_found) *n_found = m;
  return MOE_OK;
}

moe_status_t moe_eamc_predict(const void* eamc, const int32_t* cur, int32_t layer, int32_t n_match,
                              double* p_eam) {
  const EamcHeader* h = eamc_of(eamc);
  if (!h || !cur || !p_eam || n_match < 1) return MOE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= h->L) return MOE_ERR_INVALID_ARG;
  if (n_match > 1024) return MOE_ERR_UNSUPPORTED_SHAPE;
  const int L = h->L, E = h->E;
  int32_t idx[1024];
  double dist[1024];
  const int m = nearest(h, cur, n_match, idx, dist);
  for (int i = 0; i < L; ++i) {
    double* row = p_eam + (size_t)i * E;
    double rs = 0.0;
    for (int j = 0; j < E; ++j) {
      double c = 0.0;
      for (int t = 0; t < m; ++t) c += eamc_cell(h, idx[t], i * E + j);
      row[j] = c;
      rs += c;
    }
    const double scale = 1.0 - (double)(i - layer) / (double)L;
    for (int j = 0; j < E; ++j) row[j] = rs > 0.0 ? row[j] / rs * scale : 0.0;
  }
  return MOE_OK;
}

size_t moe_expert_cache_bytes(int32_t capacity) {
  if (capacity < 1) return 0;
  return sizeof(CacheHeader) + (size_t)capacity * 2 * sizeof(int32_t);
}

moe_status_t moe_expert_cache_init(void* cache, size_t bytes, int32_t capacity, int32_t L, int32_t E) {
  if (!cache || capacity < 1 || L < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (bytes < moe_expert_cache_bytes(capacity)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  CacheHeader* c = reinterpret_cast<CacheHeader*>(cache);
  memset(c, 0, sizeof(*c));
  c->magic = kCacheMagic;
  c->capacity = capacity;
  c->L = L;
  c->E = E;
  return MOE_OK;
}

moe_status_t moe_expert_cache_contents(const void* cache, int32_t* layer_expert, int32_t* n) {
  const CacheHeader* c = reinterpret_cast<const CacheHeader*>(cache);
  if (!c || c->magic != kCacheMagic || !n) return MOE_ERR_INVALID_ARG;
  if (layer_expert) memcpy(layer_expert, c + 1, (size_t)c->size * 2 * sizeof(int32_t));
  *n = c->size;
  return MOE_OK;
}

moe_status_t moe_expert_cache_lookup(void* cache, const void* eamc, const int32_t* cur, int32_t layer,
                                     int32_t expert, int32_t n_match, double eps, int32_t* hit,
                                     int32_t* evicted) {
  CacheHeader* c = reinterpret_cast<CacheHeader*>(cache);
  const EamcHeader* h = eamc_of(eamc);
  if (!c || c->magic != kCacheMagic || !h || !cur || !hit || !evicted) return MOE_ERR_INVALID_ARG;
  if (h->L != c->L || h->E != c->E || layer < 0 || layer >= c->L || expert < 0 || expert >= c->E)
    return MOE_ERR_INVALID_ARG;
  int32_t* ent = reinterpret_cast<int32_t*>(c + 1);  // [size][2] (layer, expert), insertion order
  evicted[0] = evicted[1] = -1;
  for (int t = 0; t < c->size; ++t) {
    if (ent[2 * t] == layer && ent[2 * t + 1] == expert) {
      *hit = 1;
      return MOE_OK;
    }
  }
  *hit = 0;
  if (c->size == c->capacity) {
    const int L = c->L, E = c->E;
    double p_stack[4096];
    if ((size_t)L * E > 4096) return MOE_ERR_UNSUPPORTED_SHAPE;
    moe_status_t s = moe_eamc_predict(eamc, cur, layer, n_match, p_stack);
    if (s != MOE_OK) return s;
    int victim = 0;
    double p_min = INFINITY;
    for (int t = 0; t < c->size; ++t) {
      const int li = ent[2 * t], ej = ent[2 * t + 1];
      double n_token = 0.0;
      for (int j = 0; j < E; ++j) n_token += p_stack[(size_t)li * E + j];
      if (n_token == 0.0) n_token = 1.0;  // a row without prediction: the bare eps
      const double pr = (p_stack[(size_t)li * E + ej] + eps) / n_token * (1.0 - (double)li / (double)L);
      if (pr < p_min) {
        p_min = pr;
        victim = t;
      }
    }
    evicted[0] = ent[2 * victim];
    evicted[1] = ent[2 * victim + 1];
    memmove(ent + 2 * victim, ent + 2 * (victim + 1), (size_t)(c->size - victim - 1) * 2 * sizeof(int32_t));
    --c->size;
  }
  ent[2 * c->size] = layer;
  ent[2 * c->size + 1] = expert;
  ++c->size;
  return MOE_OK;
}

moe_status_t moe_eam_add_counts(int32_t* eam, int32_t L, int32_t E, int32_t layer, const int32_t* counts) {
  if (!eam || !counts || layer < 0 || layer >= L || E < 1) return MOE_ERR_INVALID_ARG;
  for (int j = 0; j < E; ++j) eam[(size_t)layer * E + j] += counts[j];
  return MOE_OK;
}

}  // extern "C"
