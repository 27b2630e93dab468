// Forward pass of fused RoPE + AnchorAttention on sm_103a.
//
// What it computes ("When Precision Meets Position", architecture page §3.4
// "AnchorAttention: The Shared Anchor Design", "Mask construction"; RoPE per
// Eq. 6 of §3.4 "Rotary Positional Embedding (RoPE)"): for every query row i
// of head h,
//   O_i   = sum_{j visible} softmax_j(scale * (R_i q_i).(R_j k_j)) v_j
//   LSE_i = ln sum_{j visible} exp(scale * (R_i q_i).(R_j k_j))
// with the visible set {0} U [row_lo_i, i] (ANCHOR) or [row_lo_i, i].
//
// How. Q and K are rotated once per call by the standalone RoPE kernel into
// the workspace: every query tile of a document re-reads K, and a Q tile
// rotated inside the attention kernel would put the rotation between one
// item's last products and the next item's first. The attention kernel is
// persistent: one CTA per SM; the CTAs claim (pair of 128-row query tiles,
// head) items — with an even number of query heads per kv head, (query tile,
// two heads of one kv group) items — from a counter in work-list order
// (grouped by document with the heads interleaved, longest document first),
// 384 threads:
//   warp 0      claims the next item (published to the other roles through a
//               2-slot shared-memory ring) and is the TMA producer: each
//               item's rotated Q0/Q1 as soon as the previous item's last S
//               product of that tile has run, and the rotated K / V tiles
//               through a 2-stage ring that runs on across items
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 4-7   query tile 0: online softmax (thread = query row = TMEM lane)
//               and epilogue
//   warps 8-11  the same for query tile 1
// Between items nothing drains: the next item's loads and first products
// overlap the last key tiles and the epilogues, and group 0 writes its O
// while group 1 finishes.
// Tensor-memory columns: S0 [0,128) S1 [128,256) O0, O1 (D columns each). The
// softmax writes P as packed bf16 over the first 64 columns of its S, and the
// PV product reads it straight from TMEM (tcgen05.mma with A in TMEM).
// The MMA issue order S0(j), PV1(j-1), S1(j), PV0(j) lets each softmax group
// work while the tensor core runs the other group's products. Only the key
// tiles that overlap a query tile's row intervals are visited; the anchor
// column enters as the online softmax's start state (m = s_i0, l = 1) and its
// value row is added in the epilogue.
#include "kcommon.cuh"

namespace aa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: O is rescaled only when the max grows by > 2^8
constexpr uint64_t kDrainLimitNs = 1000000000ull;
constexpr int kStages = 2;
constexpr int kThreads = 384;

// One item as the roles see it: query tiles qt0 and qt0 + 1 (when it exists)
// of head h over key tiles [kt_lo, kt_hi]; query tile t visits [lo[t], hi[t]].
struct FwdItem {
  int h, qt0, kt_lo, kt_hi, lo[2], hi[2];
  bool has1;
};

// A claimed item as the producer publishes it: the work-list index (-1: none
// left), its decoded description and the anchor's rotated key and value rows
// for the item's kv head (bf16 pairs), so that no role starts an item with
// dependent global loads.
template <int HD>
struct ItemSlot {
  alignas(16) uint32_t k0[HD / 2];
  alignas(16) uint32_t v0[HD / 2];
  FwdItem w;
  int it;
};

template <int HD>
struct FwdSmem {
  static constexpr int kB = HD / 64;
  alignas(1024) uint8_t q[2][kB][16384];
  alignas(1024) uint8_t k[kStages][kB][16384];
  alignas(1024) uint8_t v[kStages][kB][16384];
  uint64_t q_full[2], q_free[2];
  uint64_t item_full[2], item_empty[2];
  ItemSlot<HD> slot[2];
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2], drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct FwdParams {
  const __nv_bfloat16* kr;  // rotated K [T, Hkv, D] (or K itself without RoPE)
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* pos_id;
  const int32_t* row_lo;
  const int32_t* qtile_klo;
  const int32_t* out_rows;   // caller row of each kernel row for O / LSE (NULL: the same row)
  const WorkItem* items;     // the work list: grouped by document, longest group first
  int32_t* next_item;        // next unclaimed index (zeroed before the launch)
  int n_items;
  const float2* rope_hi;
  const float2* rope_lo;
  const float2* rope_step;
  int32_t* err;
  uint64_t wait_limit_ns;
  int T, Hq, Hkv, group, layout, anchor, n_tiles;
  int head_pairs;  // items are (query tile, two heads of one kv group) instead of (two query tiles, head)
  float scale;
};


__device__ __forceinline__ FwdItem load_fwd_item(const FwdParams& P, int it) {
  const WorkItem w = P.items[it];
  FwdItem f;
  f.h = w.head;
  if (P.head_pairs) {
    f.qt0 = w.tile;
    f.kt_lo = w.lo;
    f.kt_hi = w.hi;
    f.has1 = true;
    f.lo[0] = f.lo[1] = __ldg(P.qtile_klo + w.tile);
    f.hi[0] = f.hi[1] = w.tile;
    return f;
  }
  f.qt0 = 2 * w.tile;
  f.kt_lo = w.lo;
  f.kt_hi = w.hi;
  f.has1 = f.qt0 + 1 < P.n_tiles;
  f.lo[0] = __ldg(P.qtile_klo + f.qt0);
  f.hi[0] = f.qt0;
  f.lo[1] = f.has1 ? __ldg(P.qtile_klo + f.qt0 + 1) : 1;  // empty range for a missing second tile
  f.hi[1] = f.has1 ? f.qt0 + 1 : 0;
  return f;
}

// Bounded wait that also gives up as soon as another role of the CTA aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const FwdParams& P,
                                              volatile int* abort_flag, int site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::global_timer_ns() - t0 >= P.wait_limit_ns) {
      atomicCAS(P.err, 0, site);
      *abort_flag = 1;
      return false;
    }
  }
}

// The li-th item this CTA runs (its work-list index, or -1 when the list is
// exhausted or the CTA aborted), as the producer published it in slot li & 1.
// warp_read: the whole (converged) warp waits. Each reader frees the slot
// (release_fwd_item) once it no longer reads it: the MMA thread after the
// item's last product, the softmax warps after the epilogue (it reads v_0
// from the slot). Slot readers: the MMA thread and the 8 softmax warps.
constexpr int kFwdItemReaders = 9;
static_assert(kFwdItemReaders == 1 + (kThreads / 32 - 4), "item readers: the MMA thread and warps 4-11");

template <class Smem>
__device__ __forceinline__ int read_fwd_item(Smem& sm, int li, const FwdParams& P, volatile int* abort_flag,
                                             bool warp_read, int site) {
  const int slot = li & 1;
  bool ok = wait_or_abort(&sm.item_full[slot], (li >> 1) & 1, P, abort_flag, site);
  if (warp_read) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return -1;
  return *reinterpret_cast<volatile int*>(&sm.slot[slot].it);
}

template <class Smem>
__device__ __forceinline__ void release_fwd_item(Smem& sm, int li, bool warp_read) {
  if (warp_read) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&sm.item_empty[li & 1]);
  } else {
    ptx::mbar_arrive(&sm.item_empty[li & 1]);
  }
}

// Barrier phases: the item ring counts the CTA's items; the K/V ring counts
// the CTA's key-tile steps across its items; s_full / p_full count each query tile's softmax steps; q_full,
// q_free and o_full count the items in which the query tile exists.
// The roles synchronise through mbarriers only (every wait bounded), so an
// abort in one role never strands another at a named barrier; inside a warp
// each wait's outcome is made uniform by a vote before any warp-collective
// step, so no lane leaves a loop that the rest of its warp stays in.
// kRows: O and LSE rows go to P.out_rows (segment plans); the contiguous
// instantiation carries no row map.
template <int HD, bool kRows>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (ptx::smem_u32(smem_raw) & 1023u) {  // swizzled tiles need a 1 KB aligned base
    if (threadIdx.x == 0) atomicCAS(P.err, 0, 398);
    return;
  }
  FwdSmem<HD>& sm = *reinterpret_cast<FwdSmem<HD>*>(smem_raw);
  constexpr uint32_t kTileBytes = 128 * HD * 2;
  constexpr int kTmemCols = 512;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sm.abort_flag;

  if (tid == 0) {
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(&sm.q_full[t], 1);
      ptx::mbar_init(&sm.q_free[t], 128);
      ptx::mbar_init(&sm.s_full[t], 1);
      ptx::mbar_init(&sm.p_full[t], 128);
      ptx::mbar_init(&sm.o_full[t], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sm.kv_full[s], 1);
      ptx::mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.item_full[s], 1);
      ptx::mbar_init(&sm.item_empty[s], kFwdItemReaders);
    }
    ptx::mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int nq[2] = {0, 0}, ks = 0;
      bool ok = true;
      for (int li = 0; ok; ++li) {
        // claim the next work-list item once every reader has taken slot li & 1
        const int slot = li & 1;
        if (li >= 2) ok = wait_or_abort(&sm.item_empty[slot], ((li >> 1) - 1) & 1, P, abort_flag, 302);
        if (!ok) break;
        int it = atomicAdd(P.next_item, 1);
        if (it >= P.n_items) it = -1;
        ItemSlot<HD>& sl = sm.slot[slot];
        sl.it = it;
        FwdItem w{};
        if (it >= 0) {
          w = load_fwd_item(P, it);
          sl.w = w;
          if (P.anchor) {
            const size_t row0 = (size_t)(w.h / P.group) * HD;
            const uint4* ks = reinterpret_cast<const uint4*>(P.kr + row0);
            const uint4* vs = reinterpret_cast<const uint4*>(P.v + row0);
            uint4 kq[HD / 8], vq[HD / 8];
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) {
              kq[c] = __ldg(ks + c);
              vq[c] = __ldg(vs + c);
            }
#pragma unroll
            for (int c = 0; c < HD / 8; ++c) {
              reinterpret_cast<uint4*>(sl.k0)[c] = kq[c];
              reinterpret_cast<uint4*>(sl.v0)[c] = vq[c];
            }
          }
        }
        ptx::mbar_arrive(&sm.item_full[slot]);  // release: the slot is written
        if (it < 0) break;
        const int g = w.h / P.group;
        for (int t = 0; t < (w.has1 ? 2 : 1) && ok; ++t) {
          // the tile's previous Q has had its last S product and its anchor dot
          if (nq[t] > 0) ok = wait_or_abort(&sm.q_free[t], (nq[t] - 1) & 1, P, abort_flag, 300);
          if (!ok) break;
          ptx::mbar_arrive_expect_tx(&sm.q_full[t], kTileBytes);
          for (int b = 0; b < HD / 64; ++b)
            ptx::tma_load_3d(sm.q[t][b], &tmQ, &sm.q_full[t], b * 64, w.h + (P.head_pairs ? t : 0),
                             (w.qt0 + (P.head_pairs ? 0 : t)) * kTile);
          ++nq[t];
        }
        for (int kt = w.kt_lo; kt <= w.kt_hi && ok; ++kt) {
          const int s = ks % kStages;
          if (ks >= kStages) ok = wait_or_abort(&sm.kv_empty[s], ((ks / kStages) - 1) & 1, P, abort_flag, 301);
          if (!ok) break;
          ptx::mbar_arrive_expect_tx(&sm.kv_full[s], 2 * kTileBytes);
          for (int b = 0; b < HD / 64; ++b) {
            ptx::tma_load_3d(sm.k[s][b], &tmK, &sm.kv_full[s], b * 64, g, kt * kTile);
            ptx::tma_load_3d(sm.v[s][b], &tmV, &sm.kv_full[s], b * 64, g, kt * kTile);
          }
          ++ks;
        }
      }
      // let every issued copy land before the CTA can exit (each earlier
      // phase of these barriers completed before the buffer was refilled)
      for (int t = 0; t < 2; ++t)
        if (nq[t] > 0) ptx::mbar_wait(&sm.q_full[t], (nq[t] - 1) & 1, kDrainLimitNs, P.err, 309);
      for (int u = (ks > kStages ? ks - kStages : 0); u < ks; ++u)
        ptx::mbar_wait(&sm.kv_full[u % kStages], (u / kStages) & 1, kDrainLimitNs, P.err, 309);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, 0, 0);
      constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, HD, 0, 1);
      const uint32_t t_s[2] = {tmem, tmem + 128};
      const uint32_t t_o[2] = {tmem + 256, tmem + 256 + HD};
      uint32_t ph_p[2] = {0, 0};
      int nq[2] = {0, 0}, ks = 0;
      bool first_pv[2] = {true, true}, ready[2] = {false, false};
      auto issue_s = [&](int t, int s) -> bool {
        if (!ready[t]) {  // this item's Q tile t has landed (first use only)
          if (!wait_or_abort(&sm.q_full[t], nq[t] & 1, P, abort_flag, 312)) return false;
          ready[t] = true;
          ptx::tc_fence_after();
        }
        const uint64_t qd = ptx::smem_desc_sw128(ptx::smem_u32(sm.q[t][0]), 16, 1024);
        const uint64_t kd = ptx::smem_desc_sw128(ptx::smem_u32(sm.k[s][0]), 16, 1024);
        if constexpr (HD == 128)
          ptx::mma8_ss_kk(t_s[t], qd, kd, idesc_s, 0);
        else
          ptx::mma4_ss_kk(t_s[t], qd, kd, idesc_s, 0);
        ptx::mma_commit(&sm.s_full[t]);
        return true;
      };
      auto issue_pv = [&](int t, int s) -> bool {
        if (!wait_or_abort(&sm.p_full[t], ph_p[t], P, abort_flag, 311)) return false;
        ph_p[t] ^= 1;
        ptx::tc_fence_after();
        ptx::mma8_ts_seq(t_o[t], t_s[t], ptx::smem_desc_sw128(ptx::smem_u32(sm.v[s][0]), 16384, 1024), idesc_pv,
                         first_pv[t] ? 0u : 1u);
        first_pv[t] = false;
        return true;
      };
      bool ok = true;
      for (int li = 0; ok; ++li) {
        const int it = read_fwd_item(sm, li, P, abort_flag, false, 310);
        if (it < 0) break;
        const FwdItem w = sm.slot[li & 1].w;
        first_pv[0] = first_pv[1] = true;
        ready[0] = false;
        ready[1] = !w.has1;
        int pend1 = -1;  // stage whose PV1 is still to be issued
        int kstep = 0;   // key-tile step within the item
        // issue order S0(j), PV1(j-1), S1(j), PV0(j): each softmax group works
        // while the tensor core runs the other group's products
        for (int kt = w.kt_lo; kt <= w.kt_hi && ok; ++kt, ++kstep, ++ks) {
          const int s = ks % kStages;
          ok = wait_or_abort(&sm.kv_full[s], (ks / kStages) & 1, P, abort_flag, 313);
          if (!ok) break;
          ptx::tc_fence_after();
          const bool in0 = kt >= w.lo[0] && kt <= w.hi[0], in1 = kt >= w.lo[1] && kt <= w.hi[1];
          if (in0 && !(ok = issue_s(0, s))) break;
          if (pend1 >= 0) {
            if (!(ok = issue_pv(1, pend1))) break;
            pend1 = -1;
          }
          if (kstep > 0) ptx::mma_commit(&sm.kv_empty[(ks - 1) % kStages]);
          if (in1 && !(ok = issue_s(1, s))) break;
          if (in0) {
            if (!(ok = issue_pv(0, s))) break;
            if (kt == w.hi[0]) ptx::mma_commit(&sm.o_full[0]);  // O0 complete
          }
          if (in1) pend1 = s;
        }
        if (ok && pend1 >= 0) {
          ok = issue_pv(1, pend1);
          if (ok) ptx::mma_commit(&sm.o_full[1]);
        }
        if (ok) ptx::mma_commit(&sm.kv_empty[(ks - 1) % kStages]);
        release_fwd_item(sm, li, false);
        ++nq[0];
        if (w.has1) ++nq[1];
      }
      // every issued MMA must finish before TMEM is released
      ptx::mma_commit(&sm.drain);
      ptx::mbar_wait(&sm.drain, 0, kDrainLimitNs, P.err, 319);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax
    const int t = (warp - 4) >> 2;
    const int r = tid & 127;
    const float sl2 = P.scale * kLog2e;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + 128 * t + lane_off, t_o = tmem + 256 + HD * t + lane_off;
    uint32_t ph_s = 0;
    int nq = 0;
    bool ok = true;
    for (int li = 0; ok; ++li) {
      const int it = read_fwd_item(sm, li, P, abort_flag, true, 320);
      if (it < 0) break;
      const ItemSlot<HD>& sl = sm.slot[li & 1];
      const FwdItem w = sl.w;
      if (t == 1 && !w.has1) {
        release_fwd_item(sm, li, true);
        continue;
      }
      const int h = w.h + (P.head_pairs ? t : 0);
      const int lo_t = w.lo[t], hi_t = w.hi[t];
      const int i = (w.qt0 + (P.head_pairs ? 0 : t)) * kTile + r;
      const bool row_valid = i < P.T;
      const int lo = row_valid ? __ldg(P.row_lo + i) : 1;
      const int hi = row_valid ? i : 0;
      float m = -INFINITY, l = 0.f, s0 = 0.f;
      if (P.anchor) {
        ok = __all_sync(0xffffffffu, wait_or_abort(&sm.q_full[t], nq & 1, P, abort_flag, 324));
        if (!ok) break;
        // s_i0 = q~_i . k~_0 with the rotated anchor key the producer staged
        const uint4* k0 = reinterpret_cast<const uint4*>(sl.k0);
        float acc = 0.f;
#pragma unroll 4
        for (int c8 = 0; c8 < HD / 8; ++c8) {
          const uint4 kq = k0[c8];
          const uint4 qq = *reinterpret_cast<const uint4*>(sm.q[t][0] + (c8 >> 3) * 16384 + sw128_chunk(r, c8 & 7));
          const uint32_t ka[4] = {kq.x, kq.y, kq.z, kq.w}, qa[4] = {qq.x, qq.y, qq.z, qq.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = ptx::unpack_bf16x2(ka[e]), qf = ptx::unpack_bf16x2(qa[e]);
            acc = fmaf(qf.x, kf.x, acc);
            acc = fmaf(qf.y, kf.y, acc);
          }
        }
        s0 = acc * sl2;
        m = s0;
        l = 1.f;
      }
      for (int kt = lo_t; kt <= hi_t && ok; ++kt) {
        ok = __all_sync(0xffffffffu, wait_or_abort(&sm.s_full[t], ph_s, P, abort_flag, 322));
        if (!ok) break;
        ph_s ^= 1;
        ptx::tc_fence_after();
        // the item's last S product for this tile is done and the anchor dot
        // read Q long before: the producer may refill the Q buffer
        if (kt == hi_t) ptx::mbar_arrive(&sm.q_free[t]);
        const int j0 = kt * kTile;
        // tiles every row of the warp sees entirely skip the per-element mask
        const bool full = __all_sync(0xffffffffu, lo <= j0 && j0 + kTile - 1 <= hi);
        // the row's logits, read from TMEM once (one wait) and kept in registers
        // for both passes
        float sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) ptx::tmem_ld32(t_s + c * 32, sv + c * 32);
        ptx::tmem_wait_ld();
        // keys this row does not see become -inf (their P is 2^-inf = 0)
        if (!full) {
#pragma unroll
          for (int e = 0; e < 128; ++e) sv[e] = (j0 + e >= lo && j0 + e <= hi) ? sv[e] : -INFINITY;
        }
        // pass 1: row max of the visible logits (scaled once at the end)
        float mt = -INFINITY;
#pragma unroll
        for (int e = 0; e < 128; e += 2) mt = fmaxf(mt, fmaxf(sv[e], sv[e + 1]));
        mt *= sl2;
        // TMEM access is warp-collective, so a rescale of O is decided per warp
        const bool need = (mt > m + kRescaleThreshold) || (m == -INFINITY && mt > -INFINITY);
        if (__any_sync(0xffffffffu, need)) {
          const float mn = fmaxf(m, mt);
          const float f = (m == -INFINITY) ? 0.f : exp2f(m - mn);
          l *= f;
          if (kt > lo_t) {  // O holds earlier tiles: S(kt) done implies their PV is done
#pragma unroll 1
            for (int c = 0; c < HD / 16; ++c) {
              float ov[16];
              ptx::tmem_ld16(t_o + c * 16, ov);
              ptx::tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) ov[e] *= f;
              ptx::tmem_st16f(t_o + c * 16, ov);
            }
          }
          m = mn;
        }
        // pass 2: P = exp2(s - m) as packed bf16 over the first 64 columns of S
        float rs = 0.f;
        const float mm = (m == -INFINITY) ? 0.f : m;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float* sc = sv + c * 32;
          uint32_t pw[16];
          const float2 sl22 = make_float2(sl2, sl2), nm2 = make_float2(-mm, -mm);
          float2 rs2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 a = __ffma2_rn(make_float2(sc[2 * e], sc[2 * e + 1]), sl22, nm2);
            const float2 pp = make_float2(ptx::ex2(a.x), ptx::ex2(a.y));
            rs2 = __fadd2_rn(rs2, pp);
            pw[e] = ptx::pack_bf16x2(pp.x, pp.y);
          }
          rs += rs2.x + rs2.y;
          ptx::tmem_st16(t_s + c * 16, pw);
        }
        l += rs;
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&sm.p_full[t]);
      }
      if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&sm.o_full[t], nq & 1, P, abort_flag, 323));
      if (!ok) break;
      // ---- epilogue. Its TMEM reads complete (tmem_wait_ld) before this
      // thread's next p_full arrival, which the next item's first PV of this
      // tile (overwriting O) waits for.
      ptx::tc_fence_after();
      const float w0 = P.anchor ? exp2f(s0 - m) : 0.f;
      const float inv_l = 1.f / l;
      const int i_out = !row_valid ? 0 : kRows ? __ldg(P.out_rows + i) : i;
      __nv_bfloat16* orow = P.o + ((size_t)i_out * P.Hq + h) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float ov[32];
        ptx::tmem_ld32(t_o + c * 32, ov);
        ptx::tmem_wait_ld();
        if (row_valid) {
          uint32_t ow[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float2 v0 = make_float2(0.f, 0.f);
            if (P.anchor)
              v0 = ptx::unpack_bf16x2(sl.v0[c * 16 + e]);
            const float a = (ov[2 * e] + w0 * v0.x) * inv_l;
            const float b = (ov[2 * e + 1] + w0 * v0.y) * inv_l;
            ow[e] = ptx::pack_bf16x2(a, b);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(ow[4 * e], ow[4 * e + 1], ow[4 * e + 2], ow[4 * e + 3]);
        }
      }
      if (row_valid) P.lse[(size_t)h * P.T + i_out] = (m + log2f(l)) * 0.69314718055994531f;
      release_fwd_item(sm, li, true);
      ++nq;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// Forward workspace: [rotated K][rotated Q] (with RoPE), then 256 bytes
// holding the attention kernel's work counter.
size_t fwd_k_bytes(const aa_plan_s* p) { return ((size_t)p->T * p->Hkv * p->D * 2 + 255) & ~size_t(255); }
size_t fwd_rot_bytes(const aa_plan_s* p) {
  if (p->cfg.rope_layout == AA_ROPE_NONE) return 0;
  return fwd_k_bytes(p) + (((size_t)p->T * p->Hq * p->D * 2 + 255) & ~size_t(255));
}
int32_t* fwd_counter(const aa_plan_s* p, void* workspace) {
  return reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + fwd_rot_bytes(p));
}

template <int HD>
aa_status launch_fwd(aa_plan_s* p, const void* q, const void* k, const void* v, void* o, float* lse,
                     void* workspace, cudaStream_t s, const int32_t* rows) {
  CUtensorMap tq, tk, tv;
  aa_status st;
  const void* qr = q;
  const void* kr = k;
  if (p->cfg.rope_layout != AA_ROPE_NONE) {
    fwd_rotated_operands(p, workspace, &qr, &kr);  // they stay there for aa_bwd_from_fwd
    if ((st = launch_rope(p, k, workspace, p->Hkv, 0, s, nullptr, rows)) != AA_OK) return st;
    if ((st = launch_rope(p, q, const_cast<void*>(qr), p->Hq, 0, s, nullptr, rows)) != AA_OK) return st;
  }
  if ((st = make_tile_map(&tq, qr, p->T, p->Hq, HD)) != AA_OK) return st;
  if ((st = make_tile_map(&tk, kr, p->T, p->Hkv, HD)) != AA_OK) return st;
  if ((st = make_tile_map(&tv, v, p->T, p->Hkv, HD)) != AA_OK) return st;
  FwdParams P;
  P.kr = static_cast<const __nv_bfloat16*>(kr);
  P.v = static_cast<const __nv_bfloat16*>(v);
  P.o = static_cast<__nv_bfloat16*>(o);
  P.lse = lse;
  P.pos_id = p->dev.pos_id;
  P.row_lo = p->dev.row_lo;
  P.qtile_klo = p->dev.qtile_klo;
  P.out_rows = rows;
  P.items = p->dev.fwd_items;
  P.next_item = fwd_counter(p, workspace);
  P.n_items = (int)p->fwd_items.size();
  P.rope_hi = p->dev.rope_hi;
  P.rope_lo = p->dev.rope_lo;
  P.rope_step = p->dev.rope_step;
  P.err = p->dev.err;
  P.wait_limit_ns = p->wait_limit_ns;
  P.T = p->T;
  P.Hq = p->Hq;
  P.Hkv = p->Hkv;
  P.group = p->group;
  P.layout = p->cfg.rope_layout;
  P.anchor = p->anchor ? 1 : 0;
  P.n_tiles = p->n_tiles;
  P.head_pairs = p->fwd_head_pairs ? 1 : 0;
  P.scale = p->scale;
  const size_t smem = sizeof(FwdSmem<HD>);
  static std::once_flag attr_once[kMaxDevices];
  static cudaError_t attr_result[kMaxDevices];
  cudaError_t e = once_per_device(attr_once, attr_result, p->device, [&] {
    cudaError_t r = cudaFuncSetAttribute(attn_fwd_kernel<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(attn_fwd_kernel<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return r;
  });
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_kernel smem attribute");
  // persistent: one CTA per SM (fewer for short work lists), claiming the
  // items in work-list order from the counter in this call's workspace
  if (p->fwd_items.empty()) return AA_OK;
  if ((e = cudaMemsetAsync(P.next_item, 0, sizeof(int32_t), s)) != cudaSuccess)
    return cuda_fail(e, "resetting the forward work counter");
  const unsigned n_cta = (unsigned)std::min<size_t>(p->fwd_items.size(), (size_t)std::max(p->num_sms, 1));
  if (rows)
    attn_fwd_kernel<HD, true><<<n_cta, kThreads, smem, s>>>(tq, tk, tv, P);
  else
    attn_fwd_kernel<HD, false><<<n_cta, kThreads, smem, s>>>(tq, tk, tv, P);
  e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "attn_fwd_kernel launch");
}

}  // namespace

void fwd_rotated_operands(const aa_plan_s* p, const void* fwd_workspace, const void** qr, const void** kr) {
  *kr = fwd_workspace;
  *qr = static_cast<const uint8_t*>(fwd_workspace) + fwd_k_bytes(p);
}

size_t fwd_base_workspace_bytes(const aa_plan_s* p) {
  if (!p) return 0;
  return fwd_rot_bytes(p) + 256;
}

aa_status launch_fwd_with_workspace(aa_plan_s* p, const void* q, const void* k, const void* v, void* o, float* lse,
                                    void* workspace, cudaStream_t s, const int32_t* rows) {
  return p->D == 128 ? launch_fwd<128>(p, q, k, v, o, lse, workspace, s, rows)
                     : launch_fwd<64>(p, q, k, v, o, lse, workspace, s, rows);
}

}  // namespace aa

using namespace aa;

extern "C" size_t aa_fwd_workspace_bytes(aa_plan_t p) {
  if (!p) return 0;
  return fwd_base_workspace_bytes(p) + (p->segmented ? seg_fwd_extra_bytes(p) : 0);
}

extern "C" aa_status aa_fwd(aa_plan_t p, const void* q, const void* k, const void* v, void* o, float* lse,
                            void* workspace, size_t workspace_bytes, aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  if (!q || !k || !v || !o || !lse) return fail(AA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(AA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(AA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  if (workspace_bytes < aa_fwd_workspace_bytes(p))
    return fail(AA_ERR_INVALID_ARG, "workspace is smaller than aa_fwd_workspace_bytes()");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->segmented) return seg_fwd(p, q, k, v, o, lse, workspace, s);
  return launch_fwd_with_workspace(p, q, k, v, o, lse, workspace, s);
}
