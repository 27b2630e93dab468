// Host planner: turns cu_doclens into per-token metadata, tile work lists and
// RoPE tables, and owns their device copies.
//
// Method: "When Precision Meets Position: BFloat16 Breaks Down RoPE in
// Long-Context Training", architecture page, §3.4 "AnchorAttention: The Shared
// Anchor Design" ("Mask construction": anchor column visible to every row,
// intra-document causal attention, cross-document pairs masked) and §3.4
// "Document Token Indexing" (continuous vs reset position IDs). The pages fix
// the mask; the tiling and the work order are this library's.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <map>
#include <new>
#include <string>

#include "aa_internal.h"

namespace aa {

static thread_local std::string g_last_error;

aa_status fail(aa_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

aa_status cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return AA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

aa_status check_compute_plan(const aa_plan_s* p) {
  if (!p) return fail(AA_ERR_INVALID_ARG, "plan is NULL");
  if (p->host_only) return fail(AA_ERR_INVALID_ARG, "plan was built with host_only = 1");
  return AA_OK;
}

// Visible-interval metadata. Row i sees keys [row_lo[i], i] through the tile
// path; key j is seen by rows [j, key_hi[j]]. With the anchor handled
// separately (ANCHOR mode) key 0 is removed from both: row_lo >= 1, the anchor
// row's interval is empty, and key_hi[0] = -1.
static void build_token_metadata(aa_plan_s* p) {
  const int T = p->T;
  p->doc_id.assign(T, 0);
  p->pos_id.assign(T, 0);
  p->row_lo.assign(T, 0);
  p->key_hi.assign(T, T - 1);
  const int mode = p->cfg.mask_mode;
  const bool continuous = mode == AA_MASK_CAUSAL || p->cfg.pos_mode == AA_POS_CONTINUOUS;
  if (mode == AA_MASK_CAUSAL) {
    for (int i = 0; i < T; ++i) p->pos_id[i] = i + p->cfg.pos_shift;
    return;
  }
  // anchor token
  p->doc_id[0] = 0;
  p->pos_id[0] = p->cfg.pos_shift;
  p->row_lo[0] = p->anchor ? 1 : 0;   // ANCHOR: empty tile interval [1, 0]
  p->key_hi[0] = p->anchor ? -1 : 0;  // INTRA_DOC: the anchor sees only itself
  const int K = (int)p->cu.size() - 1;
  for (int k = 1; k <= K; ++k) {
    const int a = p->cu[k - 1], b = p->cu[k];
    for (int i = a; i < b; ++i) {
      p->doc_id[i] = k;
      p->pos_id[i] = (continuous ? i : (i - a + 1)) + p->cfg.pos_shift;
      p->row_lo[i] = a;
      p->key_hi[i] = b - 1;
    }
  }
}

static void build_stats_and_work(aa_plan_s* p) {
  const int T = p->T, nt = p->n_tiles;
  // pair count: closed form per mode
  if (p->cfg.mask_mode == AA_MASK_CAUSAL) {
    p->unmasked_pairs = (int64_t)T * (T + 1) / 2;
  } else {
    int64_t s = 1;  // the anchor's own pair
    for (size_t k = 1; k < p->cu.size(); ++k) {
      const int64_t n = p->cu[k] - p->cu[k - 1];
      s += n * (n + 1) / 2;
      if (p->anchor) s += n;  // one anchor edge per document token
    }
    p->unmasked_pairs = s;
  }
  p->causal_tiles = (int64_t)nt * (nt + 1) / 2;
  p->live_tiles = 0;
  p->fwd_items.clear();
  p->bwd_items.clear();
  std::vector<WorkItem> q_ranges(nt);
  for (int a = 0; a < nt; ++a) {
    const int r0 = a * kTile, r1 = std::min(T, r0 + kTile) - 1;
    int lo = -1;
    for (int i = r0; i <= r1; ++i)
      if (p->row_lo[i] <= i) { lo = p->row_lo[i]; break; }  // row_lo is non-decreasing
    // every tile holds at least one row that sees itself
    const int kt_lo = lo / kTile;
    q_ranges[a] = WorkItem{a, 0, kt_lo, a};
    int64_t live = a - kt_lo + 1;
    if (p->anchor && kt_lo > 0) live += 1;  // the anchor column's block
    p->live_tiles += live;
  }
  // forward: an item fills the attention kernel's two query-tile slots.
  // With an even number of query heads per kv head, one query tile of two
  // heads that share their K/V: both slots see the same key tiles. Otherwise
  // the pair of query tiles (2a, 2a+1) of one head, visiting the union of
  // their key ranges (tile 2a+1 has one more key tile, its diagonal).
  p->qtile_klo.assign(nt, 0);
  for (int a = 0; a < nt; ++a) p->qtile_klo[a] = q_ranges[a].lo;
  p->fwd_head_pairs = p->group >= 2 && p->group % 2 == 0;
  if (p->fwd_head_pairs) {
    for (int h = 0; h < p->Hq; h += 2)
      for (int a = 0; a < nt; ++a) p->fwd_items.push_back(WorkItem{a, h, q_ranges[a].lo, a});
  } else {
    for (int h = 0; h < p->Hq; ++h)
      for (int a = 0; 2 * a < nt; ++a) {
        const int t0 = 2 * a, t1 = std::min(nt - 1, 2 * a + 1);
        p->fwd_items.push_back(WorkItem{a, h, std::min(q_ranges[t0].lo, q_ranges[t1].lo), t1});
      }
  }
  for (int g = 0; g < p->Hkv; ++g)
    for (int b = 0; b < nt; ++b) {
      const int j0 = b * kTile, j1 = std::min(T, j0 + kTile) - 1;
      int hi = -1;
      for (int j = j0; j <= j1; ++j) hi = std::max(hi, p->key_hi[j]);
      if (hi < j0) continue;  // no key of this tile is seen through the tile path
      p->bwd_items.push_back(WorkItem{b, g, b, hi / kTile});
    }
  // Work order. Items that read the same document run together, so its
  // tiles are fetched from HBM about once and re-read from L2, and groups
  // run longest first (LPT over groups). Ties resolve in a fixed order so
  // plans are reproducible.
  //  - backward: one group per (document, head), items in tile order: the
  //    document's Q/dO tiles and dQ accumulator rows stay in L2 while they
  //    are re-read and reduced into (otherwise the fp32 accumulator, 1 GiB
  //    at 64K x 32 heads, goes to HBM and back on every reduction);
  //  - forward: one group per document with its heads interleaved, items
  //    longest first: the CTAs running together read neighbouring head
  //    slices of the same K/V rows (a [T, H, D] row holds every head), which
  //    a group per (document, head) does not.
  auto order = [&](std::vector<WorkItem>& items, bool fwd) {
    auto doc_of = [&](const WorkItem& w) {
      const int row = (fwd && !p->fwd_head_pairs) ? 2 * w.tile * kTile : w.tile * kTile;
      return p->doc_id[std::min(row + (row == 0 && T > 1 ? 1 : 0), T - 1)];
    };
    std::vector<int64_t> key_doc(items.size());
    std::map<std::pair<int, int>, int64_t> group_cost;
    auto group = [&](size_t n) { return std::make_pair((int)key_doc[n], fwd ? 0 : items[n].head); };
    for (size_t n = 0; n < items.size(); ++n) {
      key_doc[n] = doc_of(items[n]);
      group_cost[group(n)] += items[n].hi - items[n].lo + 1;
    }
    std::vector<size_t> idx(items.size());
    for (size_t n = 0; n < idx.size(); ++n) idx[n] = n;
    std::stable_sort(idx.begin(), idx.end(), [&](size_t a, size_t b) {
      const WorkItem &x = items[a], &y = items[b];
      const int64_t cx = group_cost[group(a)], cy = group_cost[group(b)];
      if (cx != cy) return cx > cy;
      if (key_doc[a] != key_doc[b]) return key_doc[a] < key_doc[b];
      if (fwd) {
        const int lx = x.hi - x.lo, ly = y.hi - y.lo;
        if (lx != ly) return lx > ly;
        if (x.tile != y.tile) return x.tile < y.tile;
        return x.head < y.head;
      }
      if (x.head != y.head) return x.head < y.head;
      return x.tile < y.tile;
    });
    std::vector<WorkItem> sorted;
    sorted.reserve(items.size());
    for (size_t n : idx) sorted.push_back(items[n]);
    items.swap(sorted);
  };
  order(p->fwd_items, true);
  order(p->bwd_items, false);
  p->fwd_tiles = 0;
  for (int a = 0; a < nt; ++a) p->fwd_tiles += (int64_t)(q_ranges[a].hi - q_ranges[a].lo + 1) * p->Hq;
  p->bwd_tiles = 0;
  for (auto& w : p->bwd_items) p->bwd_tiles += (int64_t)(w.hi - w.lo + 1) * p->group;
}

// Two-level cos/sin tables for Eq. 6: pos = 32*h + l, so
// (cos, sin)(pos*theta_p) is the complex product of rope_hi[h][p] and
// rope_lo[p][l]. Entries are computed in fp64 and rounded once to fp32.
// rope_lo (16 KB at D = 128) stays in L1; a 128-row tile touches only a few
// rope_hi rows, and rope_lo is p-major so consecutive positions read
// consecutive entries.
static void build_rope_tables(aa_plan_s* p) {
  const int half = p->D / 2;
  int max_pos = 0;
  for (int v : p->pos_id) max_pos = std::max(max_pos, v);
  p->n_hi = max_pos / kRopeSplit + 1;
  const std::vector<double>& theta = p->theta;
  p->rope_hi.resize((size_t)p->n_hi * half);
  p->rope_lo.resize((size_t)kRopeSplit * half);
  for (int h = 0; h < p->n_hi; ++h)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)h * kRopeSplit * theta[i];
      p->rope_hi[(size_t)h * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
  p->rope_step.resize(half);
  for (int i = 0; i < half; ++i)
    p->rope_step[i] = make_float2((float)std::cos(theta[i]), (float)std::sin(theta[i]));
  for (int i = 0; i < half; ++i)
    for (int l = 0; l < kRopeSplit; ++l) {
      const double ang = (double)l * theta[i];
      p->rope_lo[(size_t)i * kRopeSplit + l] = make_float2((float)std::cos(ang), (float)std::sin(ang));
    }
}

template <class T>
static aa_status upload(T** dst, const std::vector<T>& src, cudaStream_t s, const char* what) {
  const size_t bytes = std::max<size_t>(src.size(), 1) * sizeof(T);
  cudaError_t e = cudaMalloc((void**)dst, bytes);
  if (e != cudaSuccess) {
    *dst = nullptr;
    return e == cudaErrorMemoryAllocation ? fail(AA_ERR_NO_MEMORY, std::string("cudaMalloc ") + what)
                                          : cuda_fail(e, what);
  }
  if (!src.empty()) {
    e = cudaMemcpyAsync(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, what);
  }
  return AA_OK;
}

static void free_device(aa_plan_s* p) {
  DevicePlan& d = p->dev;
  void* ptrs[] = {d.pos_id,    d.row_lo, d.key_hi, d.fwd_items, d.bwd_items, d.qtile_klo,
                  d.rope_hi,   d.rope_lo, d.rope_step, d.err,   d.perm,      d.pos_orig};
  for (void* q : ptrs)
    if (q) cudaFree(q);
  d = DevicePlan{};
}

static aa_status validate(const aa_config* c, const int32_t* cu, int32_t num_docs, const double* theta) {
  if (!c) return fail(AA_ERR_INVALID_ARG, "config is NULL");
  if (c->total_tokens < 2 || c->total_tokens >= (1 << 30))
    return fail(AA_ERR_INVALID_ARG, "total_tokens must be in [2, 2^30)");
  if (c->num_q_heads < 1 || c->num_kv_heads < 1 || c->num_q_heads % c->num_kv_heads)
    return fail(AA_ERR_INVALID_ARG, "need Hq >= 1, Hkv >= 1 and Hq % Hkv == 0");
  if ((int64_t)c->num_q_heads * c->total_tokens >= (1ll << 31))
    return fail(AA_ERR_INVALID_ARG, "Hq * T must stay below 2^31");
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(AA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c->mask_mode < AA_MASK_CAUSAL || c->mask_mode > AA_MASK_ANCHOR)
    return fail(AA_ERR_INVALID_ARG, "unknown mask_mode");
  if (c->pos_mode != AA_POS_RESET && c->pos_mode != AA_POS_CONTINUOUS)
    return fail(AA_ERR_INVALID_ARG, "unknown pos_mode");
  if (c->rope_layout < AA_ROPE_ADJACENT || c->rope_layout > AA_ROPE_NONE)
    return fail(AA_ERR_INVALID_ARG, "unknown rope_layout");
  if (theta) {
    for (int i = 0; i < c->head_dim / 2; ++i)
      if (!(theta[i] >= 0.0 && std::isfinite(theta[i])))
        return fail(AA_ERR_INVALID_ARG, "theta[" + std::to_string(i) + "] must be finite and >= 0");
  } else if (c->rope_layout != AA_ROPE_NONE && !(c->rope_base > 1.0 && std::isfinite(c->rope_base))) {
    return fail(AA_ERR_INVALID_ARG, "rope_base must be finite and > 1");
  }
  if (c->pos_shift < 0 || (int64_t)c->pos_shift + c->total_tokens >= (1ll << 30))
    return fail(AA_ERR_INVALID_ARG, "pos_shift must be >= 0 and keep positions below 2^30");
  if (!std::isfinite(c->softmax_scale)) return fail(AA_ERR_INVALID_ARG, "softmax_scale is not finite");
  if (c->mask_mode != AA_MASK_CAUSAL) {
    if (!cu || num_docs < 1) return fail(AA_ERR_INVALID_ARG, "cu_doclens with >= 1 document required");
    if (cu[0] != 1) return fail(AA_ERR_INVALID_ARG, "cu_doclens[0] must be 1 (token 0 is the anchor)");
    if (cu[num_docs] != c->total_tokens) return fail(AA_ERR_INVALID_ARG, "cu_doclens[num_docs] must equal T");
    for (int k = 1; k <= num_docs; ++k)
      if (cu[k] <= cu[k - 1]) return fail(AA_ERR_INVALID_ARG, "cu_doclens must increase strictly");
  }
  return AA_OK;
}

}  // namespace aa

using namespace aa;

// Segment plans: group the tokens by document (documents in order of first
// appearance, tokens in their order inside a document; the anchor stays
// first). The grouped layout is an ordinary contiguous packing with the same
// visible pairs (same document and j <= i keep their meaning because the order
// inside a document is kept) and the same positions (RESET: rank inside the
// document; CONTINUOUS: the caller's token index, set explicitly below).
static aa_status group_segments(const aa_config* cfg, const int32_t* doc_of_token, std::vector<int32_t>* perm,
                                std::vector<int32_t>* cu) {
  const int T = cfg->total_tokens;
  if (!doc_of_token) return fail(AA_ERR_INVALID_ARG, "doc_of_token is NULL");
  if (cfg->mask_mode == AA_MASK_CAUSAL)
    return fail(AA_ERR_INVALID_ARG, "segment plans need mask_mode ANCHOR or INTRA_DOC");
  if (doc_of_token[0] != 0) return fail(AA_ERR_INVALID_ARG, "doc_of_token[0] must be 0 (token 0 is the anchor)");
  std::map<int32_t, int> group_of;  // document id -> group index (first appearance)
  std::vector<std::vector<int32_t>> groups;
  for (int i = 1; i < T; ++i) {
    const int32_t d = doc_of_token[i];
    if (d < 1) return fail(AA_ERR_INVALID_ARG, "doc_of_token[" + std::to_string(i) + "] must be >= 1");
    auto it = group_of.find(d);
    if (it == group_of.end()) {
      it = group_of.emplace(d, (int)groups.size()).first;
      groups.emplace_back();
    }
    groups[it->second].push_back(i);
  }
  perm->assign(1, 0);
  cu->assign(1, 1);
  for (auto& g : groups) {
    perm->insert(perm->end(), g.begin(), g.end());
    cu->push_back(cu->back() + (int32_t)g.size());
  }
  return AA_OK;
}

static aa_status make_plan(const aa_config* cfg, const int32_t* cu_doclens_host, int32_t num_docs,
                           const double* theta, const int32_t* doc_of_token, aa_stream_t stream, aa_plan_t* out) {
  if (!out) return fail(AA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  std::vector<int32_t> perm, seg_cu;
  if (doc_of_token) {
    if (!cfg) return fail(AA_ERR_INVALID_ARG, "config is NULL");
    if (cfg->total_tokens < 2 || cfg->total_tokens >= (1 << 30))
      return fail(AA_ERR_INVALID_ARG, "total_tokens must be in [2, 2^30)");
    aa_status gs = group_segments(cfg, doc_of_token, &perm, &seg_cu);
    if (gs != AA_OK) return gs;
    cu_doclens_host = seg_cu.data();
    num_docs = (int32_t)seg_cu.size() - 1;
  }
  aa_status st = validate(cfg, cu_doclens_host, num_docs, theta);
  if (st != AA_OK) return st;
  aa_plan_s* p = new (std::nothrow) aa_plan_s();
  if (!p) return fail(AA_ERR_NO_MEMORY, "plan allocation");
  p->cfg = *cfg;
  p->T = cfg->total_tokens;
  p->Hq = cfg->num_q_heads;
  p->Hkv = cfg->num_kv_heads;
  p->group = p->Hq / p->Hkv;
  p->D = cfg->head_dim;
  p->n_tiles = (p->T + kTile - 1) / kTile;
  p->scale = cfg->softmax_scale > 0.f ? cfg->softmax_scale : (float)(1.0 / std::sqrt((double)p->D));
  p->anchor = cfg->mask_mode == AA_MASK_ANCHOR;
  p->host_only = cfg->host_only != 0;
  if (cfg->mask_mode != AA_MASK_CAUSAL) p->cu.assign(cu_doclens_host, cu_doclens_host + num_docs + 1);
  p->theta.resize(p->D / 2);
  for (int i = 0; i < p->D / 2; ++i)  // Eq. 6: theta_p = base^(-2p/D), unless the caller supplies them
    p->theta[i] = theta ? theta[i] : std::pow(cfg->rope_base, -2.0 * (double)i / (double)p->D);
  build_token_metadata(p);
  if (doc_of_token) {
    p->segmented = true;
    p->perm = perm;
    p->seg_doc.assign(doc_of_token, doc_of_token + p->T);
    if (cfg->pos_mode == AA_POS_CONTINUOUS)  // the caller's token index, not the grouped one
      for (int t = 0; t < p->T; ++t) p->pos_id[t] = perm[t] + cfg->pos_shift;
    p->seg_pos.assign(p->T, 0);
    for (int t = 0; t < p->T; ++t) p->seg_pos[perm[t]] = p->pos_id[t];
  }
  build_stats_and_work(p);
  build_rope_tables(p);
  if (p->host_only) {
    *out = p;
    return AA_OK;
  }
  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) {
    delete p;
    return cuda_fail(e, "device query");
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<int32_t> zero(1, 0);
  DevicePlan& d = p->dev;
  if ((st = upload(&d.pos_id, p->pos_id, s, "pos_id")) != AA_OK ||
      (st = upload(&d.row_lo, p->row_lo, s, "row_lo")) != AA_OK ||
      (st = upload(&d.key_hi, p->key_hi, s, "key_hi")) != AA_OK ||
      (st = upload(&d.fwd_items, p->fwd_items, s, "fwd work list")) != AA_OK ||
      (st = upload(&d.bwd_items, p->bwd_items, s, "bwd work list")) != AA_OK ||
      (st = upload(&d.qtile_klo, p->qtile_klo, s, "query-tile key ranges")) != AA_OK ||
      (st = upload(&d.rope_hi, p->rope_hi, s, "rope table (hi)")) != AA_OK ||
      (st = upload(&d.rope_lo, p->rope_lo, s, "rope table (lo)")) != AA_OK ||
      (st = upload(&d.rope_step, p->rope_step, s, "rope step table")) != AA_OK ||
      (st = upload(&d.err, zero, s, "error word")) != AA_OK ||
      (p->segmented && ((st = upload(&d.perm, p->perm, s, "segment permutation")) != AA_OK ||
                        (st = upload(&d.pos_orig, p->seg_pos, s, "segment positions")) != AA_OK))) {
    cudaStreamSynchronize(s);
    free_device(p);
    delete p;
    return st;
  }
  // the host vectors must outlive the asynchronous copies
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    free_device(p);
    delete p;
    return cuda_fail(e, "plan upload");
  }
  *out = p;
  return AA_OK;
}

extern "C" aa_status aa_plan(const aa_config* cfg, const int32_t* cu_doclens_host, int32_t num_docs,
                             aa_stream_t stream, aa_plan_t* out) {
  return make_plan(cfg, cu_doclens_host, num_docs, nullptr, nullptr, stream, out);
}

extern "C" aa_status aa_plan_segments(const aa_config* cfg, const int32_t* doc_of_token_host, aa_stream_t stream,
                                      aa_plan_t* out) {
  if (!doc_of_token_host) return fail(AA_ERR_INVALID_ARG, "doc_of_token is NULL");
  return make_plan(cfg, nullptr, 0, nullptr, doc_of_token_host, stream, out);
}

extern "C" aa_status aa_plan_with_theta(const aa_config* cfg, const int32_t* cu_doclens_host, int32_t num_docs,
                                        const double* theta, aa_stream_t stream, aa_plan_t* out) {
  if (!theta) return fail(AA_ERR_INVALID_ARG, "theta is NULL (use aa_plan for base^(-2p/D))");
  return make_plan(cfg, cu_doclens_host, num_docs, theta, nullptr, stream, out);
}

extern "C" aa_status aa_plan_destroy(aa_plan_t p) {
  if (!p) return AA_OK;
  if (!p->host_only) {
    cudaDeviceSynchronize();
    free_device(p);
  }
  delete p;
  return AA_OK;
}

extern "C" aa_status aa_plan_metadata(aa_plan_t p, int32_t* doc_id_host, int32_t* pos_id_host) {
  if (!p) return fail(AA_ERR_INVALID_ARG, "plan is NULL");
  // segment plans report the caller's document ids and token order
  const std::vector<int32_t>& doc = p->segmented ? p->seg_doc : p->doc_id;
  const std::vector<int32_t>& pos = p->segmented ? p->seg_pos : p->pos_id;
  if (doc_id_host) std::memcpy(doc_id_host, doc.data(), sizeof(int32_t) * p->T);
  if (pos_id_host) std::memcpy(pos_id_host, pos.data(), sizeof(int32_t) * p->T);
  return AA_OK;
}

extern "C" aa_status aa_plan_stats(aa_plan_t p, int64_t* pairs, int64_t* live, int64_t* causal) {
  if (!p) return fail(AA_ERR_INVALID_ARG, "plan is NULL");
  if (pairs) *pairs = p->unmasked_pairs;
  if (live) *live = p->live_tiles;
  if (causal) *causal = p->causal_tiles;
  return AA_OK;
}

extern "C" aa_status aa_plan_work(aa_plan_t p, int64_t* fwd_tiles, int64_t* bwd_tiles) {
  if (!p) return fail(AA_ERR_INVALID_ARG, "plan is NULL");
  if (fwd_tiles) *fwd_tiles = p->fwd_tiles;
  if (bwd_tiles) *bwd_tiles = p->bwd_tiles;
  return AA_OK;
}

extern "C" aa_status aa_set_wait_limit(aa_plan_t p, uint64_t ns) {
  if (!p) return fail(AA_ERR_INVALID_ARG, "plan is NULL");
  p->wait_limit_ns = ns;
  return AA_OK;
}

extern "C" aa_status aa_set_bwd_timing_events(aa_plan_t p, void* start, void* stop) {
  if (!p) return fail(AA_ERR_INVALID_ARG, "plan is NULL");
  if ((start == nullptr) != (stop == nullptr))
    return fail(AA_ERR_INVALID_ARG, "give both timing events or neither");
  p->bwd_ev_start = static_cast<cudaEvent_t>(start);
  p->bwd_ev_stop = static_cast<cudaEvent_t>(stop);
  return AA_OK;
}

extern "C" aa_status aa_check_device_error(aa_plan_t p, aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, p->dev.err, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (word != 0) {
    e = cudaMemsetAsync(p->dev.err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    char buf[96];
    std::snprintf(buf, sizeof buf, "device-side wait timed out or launch check failed (site code %d)", (int)word);
    return fail(AA_ERR_TIMEOUT, buf);
  }
  return AA_OK;
}

// ---------------------------------------------------------------- sharding
// Documents are independent apart from the anchor column ("Mask
// construction": nothing crosses documents; every row sees token 0), so a
// packing splits across ranks along documents and heads. A piece is one
// document with a range of kv heads (and their query heads); its cost is the
// visible pairs it covers: (N(N+1)/2 + N) per query head (intra-document
// causal pairs plus one anchor edge per token). Pieces are dealt longest
// first to the least-loaded shard (LPT). A document whose all-head cost
// exceeds one shard's share of the total is cut into that many kv-head ranges
// (as even as the kv heads allow) before dealing, so no rank holds a
// disproportionate document and no piece needs another rank's keys.
extern "C" aa_status aa_shard_plan(const int32_t* cu, int32_t num_docs, int32_t num_kv_heads, int32_t group,
                                   int32_t num_shards, aa_shard_piece* pieces, int32_t max_pieces,
                                   int32_t* num_pieces, int64_t* shard_cost) {
  if (!cu || !num_pieces) return fail(AA_ERR_INVALID_ARG, "aa_shard_plan: cu_doclens and num_pieces are required");
  if (num_docs < 1 || num_kv_heads < 1 || group < 1 || num_shards < 1)
    return fail(AA_ERR_INVALID_ARG, "aa_shard_plan: num_docs, num_kv_heads, group and num_shards must be >= 1");
  if (cu[0] != 1) return fail(AA_ERR_INVALID_ARG, "aa_shard_plan: cu_doclens[0] must be 1 (token 0 is the anchor)");
  for (int k = 1; k <= num_docs; ++k)
    if (cu[k] <= cu[k - 1]) return fail(AA_ERR_INVALID_ARG, "aa_shard_plan: cu_doclens must increase strictly");
  auto pair_cost = [&](int d) {  // one query head of document d (0-based)
    const int64_t n = cu[d + 1] - cu[d];
    return n * (n + 1) / 2 + n;
  };
  int64_t total = 0;
  for (int d = 0; d < num_docs; ++d) total += pair_cost(d) * num_kv_heads * group;
  const double share = (double)total / num_shards;
  std::vector<aa_shard_piece> out;
  for (int d = 0; d < num_docs; ++d) {
    const int64_t all = pair_cost(d) * num_kv_heads * group;
    int parts = (int)std::min<int64_t>(num_kv_heads, std::max<int64_t>(1, (int64_t)std::ceil(all / share - 1e-9)));
    for (int j = 0; j < parts; ++j) {
      const int g0 = (int)((int64_t)num_kv_heads * j / parts), g1 = (int)((int64_t)num_kv_heads * (j + 1) / parts);
      out.push_back(aa_shard_piece{-1, d + 1, g0, g1, pair_cost(d) * (g1 - g0) * group});
    }
  }
  if ((int64_t)out.size() > max_pieces || (!pieces && max_pieces > 0)) {
    *num_pieces = (int32_t)out.size();
    return fail(AA_ERR_INVALID_ARG, "aa_shard_plan: pieces[] is too small (num_pieces holds the count needed)");
  }
  std::vector<size_t> order(out.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) { return out[a].cost > out[b].cost; });
  std::vector<int64_t> load(num_shards, 0);
  for (size_t i : order) {
    int best = 0;
    for (int r = 1; r < num_shards; ++r)
      if (load[r] < load[best]) best = r;
    out[i].shard = best;
    load[best] += out[i].cost;
  }
  std::stable_sort(out.begin(), out.end(), [](const aa_shard_piece& a, const aa_shard_piece& b) {
    if (a.shard != b.shard) return a.shard < b.shard;
    if (a.kv_head_begin != b.kv_head_begin) return a.kv_head_begin < b.kv_head_begin;
    return a.doc < b.doc;
  });
  for (size_t i = 0; i < out.size(); ++i) pieces[i] = out[i];
  *num_pieces = (int32_t)out.size();
  if (shard_cost)
    for (int r = 0; r < num_shards; ++r) shard_cost[r] = load[r];
  return AA_OK;
}

extern "C" const char* aa_status_string(aa_status s) {
  switch (s) {
    case AA_OK: return "AA_OK";
    case AA_ERR_INVALID_ARG: return "AA_ERR_INVALID_ARG";
    case AA_ERR_UNSUPPORTED: return "AA_ERR_UNSUPPORTED";
    case AA_ERR_CUDA: return "AA_ERR_CUDA";
    case AA_ERR_NO_MEMORY: return "AA_ERR_NO_MEMORY";
    case AA_ERR_TIMEOUT: return "AA_ERR_TIMEOUT";
  }
  return "AA_ERR_UNKNOWN";
}

extern "C" const char* aa_last_error(void) { return g_last_error.c_str(); }
