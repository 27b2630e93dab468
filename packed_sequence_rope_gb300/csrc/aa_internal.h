// Internal declarations shared by the host planner and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <string>
#include <vector>

#include "../../include/anchorattn.h"

namespace aa {

constexpr int kTile = 128;      // rows of a query tile and of a key tile
constexpr int kRopeSplit = 32;  // position split of the two-level cos/sin tables

// One unit of forward work: query tile `tile` of query head `head`, visiting
// key tiles [lo, hi] (inclusive). One unit of backward work: key tile `tile`
// of kv head `head`, visiting query tiles [lo, hi] for every query head of
// the group.
struct WorkItem {
  int32_t tile, head, lo, hi;
};

struct DevicePlan {
  int32_t* pos_id = nullptr;   // [T] rotation index (shift included)
  int32_t* row_lo = nullptr;   // [T] first key of row i's tile-path interval [row_lo, i]
  int32_t* key_hi = nullptr;   // [T] last query row that sees key j in the tile path
  WorkItem* fwd_items = nullptr;  // grouped by document, longest group first (claimed in that order)
  WorkItem* bwd_items = nullptr;  // in work-list order (claimed by the CTAs in that order)
  int32_t* qtile_klo = nullptr;  // [n_tiles] first live key tile of each query tile
  float2* rope_hi = nullptr;   // [n_hi][D/2]  cos/sin((32*h) * theta_p)
  float2* rope_lo = nullptr;   // [D/2][32]    cos/sin(l * theta_p), p-major
  float2* rope_step = nullptr; // [D/2]        cos/sin(theta_p)
  int32_t* err = nullptr;      // device error word (0 = ok)
  int32_t* perm = nullptr;     // segment plans: [T] caller token of each grouped position
  int32_t* pos_orig = nullptr; // segment plans: [T] rotation index in the caller's token order
};

}  // namespace aa

struct aa_plan_s {
  aa_config cfg;
  int32_t T = 0, Hq = 0, Hkv = 0, D = 0, n_tiles = 0, group = 1;
  float scale = 0.f;
  bool anchor = false;          // anchor column handled outside the tile path
  bool host_only = false;
  std::vector<int32_t> cu;      // document boundaries (empty in CAUSAL mode)
  std::vector<int32_t> doc_id, pos_id, row_lo, key_hi;  // in the kernels' (grouped) token order
  // Segment plans (aa_plan_segments): documents given per token, possibly in
  // interleaved chunks. The kernels run on the stable grouping of the tokens
  // by document; perm[t] is the caller's token at grouped position t.
  bool segmented = false;
  std::vector<int32_t> perm, seg_doc, seg_pos;  // seg_*: the caller's order
  // fwd: one item per (query-tile pair, head), or with fwd_head_pairs (an even
  // number of query heads per kv head) one per (query tile, two heads of one
  // kv group), whose two tiles then see the same key tiles
  std::vector<aa::WorkItem> fwd_items, bwd_items;
  bool fwd_head_pairs = false;
  std::vector<int32_t> qtile_klo;
  std::vector<double> theta;    // [D/2] rotation frequency of each pair (Eq. 6's theta_p)
  std::vector<float2> rope_hi, rope_lo, rope_step;
  int32_t n_hi = 0;
  int64_t unmasked_pairs = 0, live_tiles = 0, causal_tiles = 0;
  int64_t fwd_tiles = 0, bwd_tiles = 0;
  uint64_t wait_limit_ns = 2000000000ull;
  cudaEvent_t bwd_ev_start = nullptr, bwd_ev_stop = nullptr;
  int device = 0, num_sms = 0;
  aa::DevicePlan dev;
};

namespace aa {
constexpr int kMaxDevices = 64;

// Per-device one-time host set-up (a kernel attribute, an occupancy query):
// `fn` runs once for each device ordinal, thread-safely, and every later call
// returns its first result. Ordinals outside [0, kMaxDevices) run `fn` every
// time.
template <class R, class Fn>
R once_per_device(std::once_flag (&flags)[kMaxDevices], R (&results)[kMaxDevices], int device, Fn fn) {
  if (device < 0 || device >= kMaxDevices) return fn();
  std::call_once(flags[device], [&] { results[device] = fn(); });
  return results[device];
}

// Record a failure message for aa_last_error() and return `s`.
aa_status fail(aa_status s, const std::string& msg);
aa_status cuda_fail(cudaError_t e, const char* what);
bool aligned16(const void* p);
aa_status check_compute_plan(const aa_plan_s* p);
// Rotate x [T, H, D] into y with the canonical tile rotation (no checks);
// positions from `pos` (default: the plan's kernel-order pos_id); y's row t
// reads x's row src_rows[t] (default: row t).
aa_status launch_rope(const aa_plan_s* p, const void* x, void* y, int H, int inverse, cudaStream_t s,
                      const int32_t* pos = nullptr, const int32_t* src_rows = nullptr);
// Forward kernels with an already-validated workspace. rows (segment plans):
// q and k are in the caller's order and are read through rows[t] (the caller
// token at kernel position t) by the rotation passes, v is already in kernel
// order, and o / lse are written at the caller's rows. NULL: all in kernel
// order.
aa_status launch_fwd_with_workspace(aa_plan_s* p, const void* q, const void* k, const void* v, void* o, float* lse,
                                    void* workspace, cudaStream_t s, const int32_t* rows = nullptr);
size_t fwd_base_workspace_bytes(const aa_plan_s* p);
// Where a forward workspace keeps the rotated Q and K (kernel token order);
// only meaningful when the plan rotates (rope_layout != AA_ROPE_NONE).
void fwd_rotated_operands(const aa_plan_s* p, const void* fwd_workspace, const void** qr, const void** kr);
// with_rot = false: the caller supplies the rotated Q and K (aa_bwd_from_fwd)
size_t bwd_base_workspace_bytes(const aa_plan_s* p, bool with_rot = true);
// Segment plans: extra workspace behind the base one, and the gather / run /
// scatter wrappers (segments.cu).
size_t seg_fwd_extra_bytes(const aa_plan_s* p);
size_t seg_bwd_extra_bytes(const aa_plan_s* p, bool with_qk = true);
aa_status seg_fwd(aa_plan_s* p, const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                  cudaStream_t s);
// qr / kr / vg (all or none): rotated Q and K and the grouped V already in
// the kernels' token order (a forward workspace), replacing q and k (which
// may then be NULL) and v.
aa_status seg_bwd(aa_plan_s* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, void* workspace, cudaStream_t s,
                  const void* qr = nullptr, const void* kr = nullptr, const void* vg = nullptr);
// Segment plans: where a forward workspace keeps the grouped V.
const void* fwd_grouped_v(const aa_plan_s* p, const void* fwd_workspace);
// Launch the backward kernels with an already-validated workspace pointer;
// qr / kr as for seg_bwd. rows (segment plans): q, k, o, lse, dout, dq, dk,
// dv are in the caller's order (read and written through rows[t], the
// caller token at kernel position t), v is in kernel order, and dout_g
// receives dout in kernel order (written by the preprocess kernel, read by
// the tile kernel). NULL: all in kernel order.
aa_status launch_bwd_with_workspace(aa_plan_s* p, const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                    void* workspace, cudaStream_t s, const void* qr = nullptr,
                                    const void* kr = nullptr, const int32_t* rows = nullptr,
                                    void* dout_g = nullptr);
}  // namespace aa
