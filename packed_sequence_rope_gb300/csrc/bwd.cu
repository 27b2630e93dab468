// Backward pass of fused RoPE + AnchorAttention on sm_103a.
//
// Gradients of the forward defined in fwd.cu ("When Precision Meets
// Position", architecture page §3.4 "AnchorAttention: The Shared Anchor
// Design" for the mask, Eq. 6 of §3.4 "Rotary Positional Embedding (RoPE)"
// for the rotation) with respect to the un-rotated q, k, v:
//   P_ij  = exp(scale * q~_i.k~_j - LSE_i)            (recomputed)
//   dv_j  = sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i.v_j - D_i),  D_i = dO_i.O_i
//   dq~_i = scale sum_j dS_ij k~_j,  dk~_j = scale sum_i dS_ij q~_i
//   dq = R^T dq~,  dk = R^T dk~
//
// Kernels, in stream order:
//   1. bwd_prep: D_i, and the anchor column for every row (P_i0, dS_i0): the
//      fp32 dQ accumulator is initialised with scale*dS_i0*k~_0 (so it needs
//      no separate clearing pass) and per-chunk partial sums of dv_0, dk~_0
//      are written.
//   2. attn_bwd: persistent, one CTA per SM claiming (key tile, kv head)
//      items in work-list order; per item K~/V stay in shared memory while it
//      loops over the group's query heads and the live query tiles. Five tcgen05 MMAs per tile (S^T, dP^T, dV, dK, dQ) with fp32
//      TMEM accumulators; dQ~ is added into the fp32 accumulator (TMA bulk
//      reductions for D = 128, vector atomics for D = 64); dK/dV are rotated
//      back and written once.
//   3. dq_finalize: dq = bf16(R^T dq~).
//   4. anchor_finalize: dk_0 / dv_0 = fixed-order sums of the partials.
#include "kcommon.cuh"

namespace aa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainLimitNs = 1000000000ull;
// Row chunks of the anchor partial sums: one prep block per (head, chunk).
// 64 blocks of about 1K rows per head ran the prep pass faster than 256 short
// ones (fewer block prologues and epilogue reductions).
constexpr int kPrepChunks = 64;

struct Workspace {
  __nv_bfloat16* qr;  // [T, Hq, D] rotated Q (unused without RoPE)
  __nv_bfloat16* kr;  // [T, Hkv, D] rotated K (unused without RoPE)
  float* dq_acc;   // [T, Hq, D] fp32
  float* dsum;     // [Hq, T] fp32 (D_i)
  float* part_dv;  // [kPrepChunks, Hq, D]
  float* part_dk;  // [kPrepChunks, Hq, D]
  int32_t* next_item;  // the attention kernel's work counter (reset by bwd_prep)
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// with_rot = false: the rotated Q and K come from the caller (a forward
// workspace), so the workspace holds no copies of them
Workspace carve(void* base, const aa_plan_s* p, size_t* total, bool with_rot = true) {
  Workspace w;
  size_t off = 0;
  uint8_t* b = static_cast<uint8_t*>(base);
  const bool rot = with_rot && p->cfg.rope_layout != AA_ROPE_NONE;
  w.qr = reinterpret_cast<__nv_bfloat16*>(b + off);
  if (rot) off = align256(off + (size_t)p->T * p->Hq * p->D * 2);
  w.kr = reinterpret_cast<__nv_bfloat16*>(b + off);
  if (rot) off = align256(off + (size_t)p->T * p->Hkv * p->D * 2);
  w.dq_acc = reinterpret_cast<float*>(b + off);
  off = align256(off + (size_t)p->T * p->Hq * p->D * 4);
  w.dsum = reinterpret_cast<float*>(b + off);
  off = align256(off + (size_t)p->Hq * p->T * 4);
  w.part_dv = reinterpret_cast<float*>(b + off);
  off = align256(off + (size_t)kPrepChunks * p->Hq * p->D * 4);
  w.part_dk = reinterpret_cast<float*>(b + off);
  off = align256(off + (size_t)kPrepChunks * p->Hq * p->D * 4);
  w.next_item = reinterpret_cast<int32_t*>(b + off);
  off = align256(off + sizeof(int32_t));
  if (total) *total = off;
  return w;
}

// ---------------------------------------------------------------- 1. prep
// 256 threads per (row chunk, head). A row is handled by HD/8 lanes holding
// 8 channels (one 16-byte load per tensor) each, so a warp covers 32/(HD/8)
// rows per pass and every load is a full 16-byte vector.
constexpr int kPrepThreads = 256;

template <int HD>
__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const __nv_bfloat16* __restrict__ q,
                                                                const __nv_bfloat16* __restrict__ k,
                                                                const __nv_bfloat16* __restrict__ v,
                                                                const __nv_bfloat16* __restrict__ o,
                                                                const __nv_bfloat16* __restrict__ dout,
                                                                const float* __restrict__ lse, Workspace ws, int T,
                                                                int Hq, int group, int anchor, float scale,
                                                                const int32_t* __restrict__ rows,
                                                                __nv_bfloat16* __restrict__ dout_g) {
  // rows (segment plans): o, dout and lse are in the caller's order, kernel
  // row i reading caller row rows[i]; dout_g then receives dout in kernel
  // order for the tile kernel. q (rotated) and every output are in kernel
  // order.
  constexpr int LPR = HD / 8;          // lanes per row
  constexpr int RPW = 32 / LPR;        // rows per warp pass
  constexpr int NW = kPrepThreads / 32;
  // heads are the fast grid index: blocks resident together read whole
  // [Hq, D] token rows rather than one head's rows at a stride
  const int h = blockIdx.x, g = h / group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the attention kernel, next in stream order, claims its items from here
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ws.next_item = 0;
  const int sub = lane / LPR, c0 = (lane % LPR) * 8;
  const int rows_per_chunk = (T + kPrepChunks - 1) / kPrepChunks;
  const int r_begin = blockIdx.y * rows_per_chunk;
  const int r_end = min(T, r_begin + rows_per_chunk);
  __shared__ float red_dv[NW][HD], red_dk[NW][HD];

  auto unpack8 = [](const uint4& u, float* x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = ptx::unpack_bf16x2(w[j]);
      x[2 * j] = f.x;
      x[2 * j + 1] = f.y;
    }
  };
  // the anchor key k~_0 (k is the rotated K, the forward's operand) and v_0
  // for this lane's channels
  float k0[8], v0[8];
  if (anchor) {
    unpack8(*reinterpret_cast<const uint4*>(k + (size_t)g * HD + c0), k0);
    unpack8(*reinterpret_cast<const uint4*>(v + (size_t)g * HD + c0), v0);
  }
  float pdv[8], pdk[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) pdv[e] = pdk[e] = 0.f;

  // sum over the LPR lanes of one row
  auto row_sum = [](float x) {
#pragma unroll
    for (int s = LPR / 2; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
    return x;
  };

  // NB passes per iteration, all their loads issued before any arithmetic
  // (enough bytes in flight per SM to cover HBM latency); the pass base is
  // warp-uniform so every lane takes part in the shuffles
  constexpr int NB = 4;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int ib = r_begin + warp * RPW; ib < r_end; ib += NB * NW * RPW) {
    uint4 ro[NB], rd[NB], rq[NB];
    float lse_v[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int i = ib + b * NW * RPW + sub;
      const bool valid = i < r_end;
      const size_t base = ((size_t)i * Hq + h) * HD + c0;
      const int is = valid && rows ? __ldg(rows + i) : i;  // the caller's row
      const size_t sbase = ((size_t)is * Hq + h) * HD + c0;
      ro[b] = valid ? *reinterpret_cast<const uint4*>(o + sbase) : z;
      rd[b] = valid ? *reinterpret_cast<const uint4*>(dout + sbase) : z;
      rq[b] = valid && anchor ? *reinterpret_cast<const uint4*>(q + base) : z;
      lse_v[b] = valid && anchor ? __ldg(lse + (size_t)h * T + is) : 0.f;
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int i = ib + b * NW * RPW + sub;
      const bool valid = i < r_end;
      const size_t base = ((size_t)i * Hq + h) * HD + c0;
      if (dout_g && valid) *reinterpret_cast<uint4*>(dout_g + base) = rd[b];
      float ov[8], dov[8];
      unpack8(ro[b], ov);
      unpack8(rd[b], dov);
      float dsum = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) dsum = fmaf(ov[e], dov[e], dsum);
      dsum = row_sum(dsum);
      if (valid && c0 == 0) ws.dsum[(size_t)h * T + i] = dsum;
      float4* acc = reinterpret_cast<float4*>(ws.dq_acc + base);
      if (anchor) {
        float qv[8];  // q~_i: q is the rotated Q here
        unpack8(rq[b], qv);
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          s = fmaf(qv[e], k0[e], s);
          dp = fmaf(dov[e], v0[e], dp);
        }
        s = row_sum(s);
        dp = row_sum(dp);
        const float p0 = valid ? exp2f((s * scale - lse_v[b]) * kLog2e) : 0.f;
        const float ds0 = p0 * (dp - dsum);
        const float sd = scale * ds0;
        if (valid) {
          acc[0] = make_float4(sd * k0[0], sd * k0[1], sd * k0[2], sd * k0[3]);
          acc[1] = make_float4(sd * k0[4], sd * k0[5], sd * k0[6], sd * k0[7]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          pdv[e] = fmaf(p0, dov[e], pdv[e]);
          pdk[e] = fmaf(sd, qv[e], pdk[e]);
        }
      } else if (valid) {
        acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  if (!anchor) return;
  // fold the warp's row slots (same channels), then the warps in a fixed order
#pragma unroll
  for (int e = 0; e < 8; ++e) {
#pragma unroll
    for (int s = LPR; s < 32; s <<= 1) {
      pdv[e] += __shfl_xor_sync(0xffffffffu, pdv[e], s);
      pdk[e] += __shfl_xor_sync(0xffffffffu, pdk[e], s);
    }
  }
  if (sub == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      red_dv[warp][c0 + e] = pdv[e];
      red_dk[warp][c0 + e] = pdk[e];
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < HD; c += blockDim.x) {
    float sdv = 0.f, sdk = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      sdv += red_dv[w][c];
      sdk += red_dk[w][c];
    }
    ws.part_dv[((size_t)blockIdx.y * Hq + h) * HD + c] = sdv;
    ws.part_dk[((size_t)blockIdx.y * Hq + h) * HD + c] = sdk;
  }
}

// ---------------------------------------------------------------- 2. main
// Persistent: one CTA per SM. The CTAs claim (key tile, kv head) items from a
// global counter in work-list order, so the items in flight at any moment are
// neighbours in the planner's (document, head) grouping and share their Q~/dO
// tiles and dQ accumulator rows in L2. An item keeps K~/V stationary in
// shared memory and loops over the group's query heads and live query tiles.
// 512 threads:
//   warp 0      claims the next item (published to the other roles through
//               a 2-slot ring in shared memory) and is the TMA producer: an
//               item's K, V once it may overwrite them; Q_i, dO_i through a
//               2-stage ring that runs on across items
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2-3   staging of each query tile's -LSE*log2(e) and -D rows into
//               shared memory (Q and K arrive rotated from the workspace: a
//               rotation in the tile load cost more than the once-per-call
//               pass, since most items run only a handful of tiles)
//   warps 4-11  P/dS: two groups (query columns 0-63 and 64-127), thread = key
//               row = TMEM lane; P^T packed bf16 into TMEM for the dV product,
//               dS^T bf16 into shared memory, each group in two 32-column
//               chunks: the first chunks of both groups release half of the
//               dV / dK~ products while the second chunks are computed; at
//               the end of an item they read dV and dK~ out of TMEM and write
//               dv and dk = R^T (scale dK~): group 0 dv and half of dk,
//               group 1 the other half
//   warps 12-15 dQ drain: dQ~ from TMEM into the fp32 accumulator. For
//               D = 128 the MMA produces dQ~^T (lane = channel); the drain
//               copies it into the step's dead Q~/dO stage buffers, releases
//               TMEM at once and adds the copy with TMA bulk reductions that
//               overlap the next tile; for D = 64 it uses vector atomics.
// Between items nothing drains: the next item's K~/V load waits only for the
// last MMA that reads the old ones, and its first S^T / dP^T products run
// while the P/dS warps are still writing the previous item's dk, dv. The
// next item's first dV / dK~ products need those TMEM columns back; they come
// after the P/dS warps' first arrival of that item, which follows their
// epilogue reads.
// TMEM columns: S^T [0,128) (P^T over [0,32) and [64,96)), dP^T [128,256) (dQ~
// or dQ~^T reuses [128,256) once dS is formed), dV [256,256+D), dK~ [256+D,256+2D).
constexpr int kBwdThreads = 512;

template <int HD>
struct BwdSmem {
  static constexpr int kB = HD / 64;
  alignas(1024) uint8_t k[kB][16384];
  alignas(1024) uint8_t v[kB][16384];
  alignas(1024) uint8_t q[2][kB][16384];
  alignas(1024) uint8_t dout[2][kB][16384];
  alignas(1024) uint8_t dst[2][16384];  // dS^T: 128 keys x 128 query rows, bf16
  float lse2[2][128];                   // -LSE * log2(e) of each stage's query rows
  float dsum[2][128];                   // -D of each stage's query rows
  uint64_t kv_full, kv_free;
  uint64_t item_full[2], item_empty[2];
  int item_slot[2];  // claimed work-list index (-1: none left)
  uint64_t qd_full[2], q_ready[2], qd_empty[2];
  uint64_t st_full, p_full[2], dq_full, dq_free, o_full, drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdParams {
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* lse;
  Workspace ws;
  const int32_t* pos_id;
  const int32_t* key_hi;
  const int32_t* rows;        // caller row of each kernel row for lse, dk, dv (NULL: the same row)
  const WorkItem* items;      // the work list, in the planner's order
  int32_t* next_item;         // next unclaimed index (zeroed by bwd_prep)
  int n_items;
  const float2* rope_hi;
  const float2* rope_lo;
  const float2* rope_step;
  int32_t* err;
  uint64_t wait_limit_ns;
  int T, Hq, Hkv, group, layout;
  float scale;
};

// One item as the roles see it: key tile kt of kv head g; step s (0 <= s <
// n_steps) is query head g * group + s / n_qt, query tile lo + s % n_qt.
struct BwdItem {
  int kt, g, lo, n_qt, n_steps;
  __device__ int head(int step, int group) const { return g * group + step / n_qt; }
  __device__ int qtile(int step) const { return lo + step % n_qt; }
};

__device__ __forceinline__ BwdItem load_item(const BwdParams& P, int it) {
  const WorkItem w = P.items[it];
  const int n_qt = w.hi - w.lo + 1;
  return BwdItem{w.tile, w.head, w.lo, n_qt, n_qt * P.group};
}

__device__ __forceinline__ bool bwd_wait(uint64_t* bar, uint32_t parity, const BwdParams& P,
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
// warp_read: the whole (converged) warp reads it and lane 0 frees the slot;
// otherwise the calling thread alone. Slot readers: the MMA thread and the
// 14 warps of the P/dS, staging and drain roles.
constexpr int kItemReaders = 15;

template <class Smem>
__device__ __forceinline__ int read_item(Smem& sm, int li, const BwdParams& P, volatile int* abort_flag,
                                         bool warp_read, int site) {
  const int slot = li & 1;
  bool ok = bwd_wait(&sm.item_full[slot], (li >> 1) & 1, P, abort_flag, site);
  if (warp_read) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return -1;
  const int it = *reinterpret_cast<volatile int*>(&sm.item_slot[slot]);
  if (warp_read) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&sm.item_empty[slot]);
  } else {
    ptx::mbar_arrive(&sm.item_empty[slot]);
  }
  return it;
}

// Barrier phases: per-step barriers count the CTA's steps across all its
// items (gs); per-item barriers (item_full, item_empty, kv_full, kv_free,
// o_full) count its items (li). Every wait is bounded; a timeout records the site in the error word
// and stops every role of the CTA. Waits followed by warp-collective steps
// are made warp-uniform by a vote (the drain group by a barrier reduction).
template <int HD>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams P) {
  // the layout fills the 227 KB limit exactly, so it relies on a 1 KB aligned
  // dynamic shared-memory base (checked: swizzled tiles need it)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (ptx::smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(P.err, 0, 498);
    return;
  }
  BwdSmem<HD>& sm = *reinterpret_cast<BwdSmem<HD>*>(smem_raw);
  constexpr int kTmemCols = 512;
  constexpr uint32_t kTileBytes = 128 * HD * 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sm.abort_flag;

  if (tid == 0) {
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
    ptx::tma_prefetch_desc(&tmDO);
    ptx::mbar_init(&sm.kv_full, 1);
    ptx::mbar_init(&sm.kv_free, 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.item_full[s], 1);
      ptx::mbar_init(&sm.item_empty[s], kItemReaders);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.qd_full[s], 1);
      ptx::mbar_init(&sm.q_ready[s], 64);
      ptx::mbar_init(&sm.qd_empty[s], 1);
    }
    ptx::mbar_init(&sm.st_full, 1);
    ptx::mbar_init(&sm.p_full[0], 256);
    ptx::mbar_init(&sm.p_full[1], 256);
    ptx::mbar_init(&sm.dq_full, 1);
    ptx::mbar_init(&sm.dq_free, 128);
    ptx::mbar_init(&sm.o_full, 1);
    ptx::mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t t_s = tmem, t_dp = tmem + 128, t_dq = tmem + 128, t_dv = tmem + 256, t_dk = tmem + 256 + HD;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int gs = 0, n_issued = 0, li_loaded = -1;
      bool ok = true;
      for (int li = 0; ok; ++li) {
        // claim the next work-list item once every role has read slot li & 1
        const int slot = li & 1;
        if (li >= 2) ok = bwd_wait(&sm.item_empty[slot], ((li >> 1) - 1) & 1, P, abort_flag, 402);
        if (!ok) break;
        int it = atomicAdd(P.next_item, 1);
        if (it >= P.n_items) it = -1;
        sm.item_slot[slot] = it;
        ptx::mbar_arrive(&sm.item_full[slot]);  // release: the slot is written
        if (it < 0) break;
        const BwdItem w = load_item(P, it);
        // the previous item's last MMA has read K~/V
        if (li > 0) ok = bwd_wait(&sm.kv_free, (li - 1) & 1, P, abort_flag, 400);
        if (!ok) break;
        ptx::mbar_arrive_expect_tx(&sm.kv_full, 2 * kTileBytes);
        for (int b = 0; b < HD / 64; ++b) {
          ptx::tma_load_3d(sm.k[b], &tmK, &sm.kv_full, b * 64, w.g, w.kt * kTile);
          ptx::tma_load_3d(sm.v[b], &tmV, &sm.kv_full, b * 64, w.g, w.kt * kTile);
        }
        li_loaded = li;
        for (int step = 0; step < w.n_steps; ++step, ++gs) {
          const int s = gs & 1;
          if (gs >= 2) ok = bwd_wait(&sm.qd_empty[s], ((gs >> 1) - 1) & 1, P, abort_flag, 401);
          if (!ok) break;
          const int h = w.head(step, P.group), qt = w.qtile(step);
          ptx::mbar_arrive_expect_tx(&sm.qd_full[s], 2 * kTileBytes);
          for (int b = 0; b < HD / 64; ++b) {
            ptx::tma_load_3d(sm.q[s][b], &tmQ, &sm.qd_full[s], b * 64, h, qt * kTile);
            ptx::tma_load_3d(sm.dout[s][b], &tmDO, &sm.qd_full[s], b * 64, h, qt * kTile);
          }
          n_issued = gs + 1;
        }
      }
      // no copy may be in flight when the CTA exits (matters after an abort);
      // every earlier phase of these barriers completed before the next
      // copy into the same buffer was issued
      if (li_loaded >= 0) ptx::mbar_wait(&sm.kv_full, li_loaded & 1, kDrainLimitNs, P.err, 409);
      for (int u = (n_issued > 2 ? n_issued - 2 : 0); u < n_issued; ++u)
        ptx::mbar_wait(&sm.qd_full[u & 1], (u >> 1) & 1, kDrainLimitNs, P.err, 409);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_kt = ptx::idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t idesc_kd = ptx::idesc_bf16_f32(128, HD, 0, 1);   // dV, dK
      constexpr uint32_t idesc_qd = ptx::idesc_bf16_f32(128, HD, 1, 1);   // dQ
      const uint32_t sk = ptx::smem_u32(sm.k[0]), sv = ptx::smem_u32(sm.v[0]);
      const uint32_t sds = ptx::smem_u32(sm.dst[0]);
      int gs = 0;
      bool ok = true;
      for (int li = 0; ok; ++li) {
        const int it = read_item(sm, li, P, abort_flag, false, 410);
        if (it < 0) break;
        const int n_steps = load_item(P, it).n_steps;
        ok = bwd_wait(&sm.kv_full, li & 1, P, abort_flag, 411);
        for (int step = 0; step < n_steps && ok; ++step, ++gs) {
          const int s = gs & 1;
          const uint32_t sq = ptx::smem_u32(sm.q[s][0]), sdo = ptx::smem_u32(sm.dout[s][0]);
          // the products need only the tiles; the LSE/D rows are for P/dS
          ok = bwd_wait(&sm.qd_full[s], (gs >> 1) & 1, P, abort_flag, 412);
          if (!ok) break;
          ptx::tc_fence_after();
          if constexpr (HD == 128)
            ptx::mma8_ss_kk(t_s, ptx::smem_desc_sw128(sk, 16, 1024), ptx::smem_desc_sw128(sq, 16, 1024), idesc_kt, 0);
          else
            ptx::mma4_ss_kk(t_s, ptx::smem_desc_sw128(sk, 16, 1024), ptx::smem_desc_sw128(sq, 16, 1024), idesc_kt, 0);
          if (gs > 0) {
            // dQ~ of the previous tile must be drained before dP^T overwrites it
            ok = bwd_wait(&sm.dq_free, (gs - 1) & 1, P, abort_flag, 413);
            if (!ok) break;
            ptx::tc_fence_after();
          }
          if constexpr (HD == 128)
            ptx::mma8_ss_kk(t_dp, ptx::smem_desc_sw128(sv, 16, 1024), ptx::smem_desc_sw128(sdo, 16, 1024), idesc_kt, 0);
          else
            ptx::mma4_ss_kk(t_dp, ptx::smem_desc_sw128(sv, 16, 1024), ptx::smem_desc_sw128(sdo, 16, 1024), idesc_kt, 0);
          ptx::mma_commit(&sm.st_full);
          // dV += P^T dO (P^T from TMEM: q 0-63 at cols 0-31, 64-127 at
          // 64-95) and dK~ += dS^T Q~, each in two parts: the P/dS warps
          // finish query columns 0-31 and 64-95 first (part 0), so those
          // products run while they compute the rest (part 1). Part 0 of an
          // item's first step also means the P/dS warps have read the
          // previous item's dV / dK~ out of TMEM.
          const uint64_t dv_b = ptx::smem_desc_sw128(sdo, 16384, 1024);
          const uint64_t dk_a = ptx::smem_desc_sw128(sds, 16, 1024), dk_b = ptx::smem_desc_sw128(sq, 16384, 1024);
          ok = bwd_wait(&sm.p_full[0], gs & 1, P, abort_flag, 414);
          if (!ok) break;
          ptx::tc_fence_after();
          ptx::mma4_ts_part0(t_dv, t_s, dv_b, idesc_kd, step > 0 ? 1u : 0u);
          ptx::mma4_ss_part0(t_dk, dk_a, dk_b, idesc_kd, step > 0 ? 1u : 0u);
          ok = bwd_wait(&sm.p_full[1], gs & 1, P, abort_flag, 416);
          if (!ok) break;
          ptx::tc_fence_after();
          ptx::mma4_ts_part1(t_dv, t_s, dv_b, idesc_kd, 1u);
          ptx::mma4_ss_part1(t_dk, dk_a, dk_b, idesc_kd, 1u);
          if constexpr (HD == 128) {
            // dQ~^T = K~^T dS^T: TMEM lanes = channels, columns = query rows, so
            // the drain's reductions are 128-byte coalesced per warp
            constexpr uint32_t idesc_qt = ptx::idesc_bf16_f32(128, 128, 1, 1);
            ptx::mma8_ss_mm(t_dq, ptx::smem_desc_sw128(sk, 16384, 1024), ptx::smem_desc_sw128(sds, 16384, 1024),
                            idesc_qt, 0);
          } else {
            // dQ~ = dS K~ (TMEM lanes = query rows)
            ptx::mma8_ss_mm(t_dq, ptx::smem_desc_sw128(sds, 16384, 1024), ptx::smem_desc_sw128(sk, 16384, 1024),
                            idesc_qd, 0);
          }
          ptx::mma_commit(&sm.dq_full);  // the drain hands stage s back to the producer
        }
        if (ok) {
          ptx::mma_commit(&sm.kv_free);  // K~/V read for the last time
          ptx::mma_commit(&sm.o_full);   // dV, dK~ complete
        }
      }
      ptx::mma_commit(&sm.drain);
      ptx::mbar_wait(&sm.drain, 0, kDrainLimitNs, P.err, 419);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ P / dS
    const int r = tid & 127;
    const int cq = (warp - 4) >> 2;  // query columns [64 cq, 64 cq + 64)
    const float sl2 = P.scale * kLog2e;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int gs = 0;
    bool ok = true;
    for (int li = 0; ok; ++li) {
      const int it = read_item(sm, li, P, abort_flag, true, 424);
      if (it < 0) break;
      const BwdItem w = load_item(P, it);
      const int j = w.kt * kTile + r;
      const bool key_valid = j < P.T;
      const int jhi = key_valid ? __ldg(P.key_hi + j) : -1;  // rows [j, jhi] see key j
      for (int step = 0; step < w.n_steps && ok; ++step, ++gs) {
        const int s = gs & 1, i0 = w.qtile(step) * kTile;
        const bool full = __all_sync(0xffffffffu, j <= i0 && i0 + kTile - 1 <= jhi);
        ok = bwd_wait(&sm.q_ready[s], (gs >> 1) & 1, P, abort_flag, 420);  // LSE/D staged
        if (ok) ok = bwd_wait(&sm.st_full, gs & 1, P, abort_flag, 421);
        ok = __all_sync(0xffffffffu, ok);  // the warp leaves (or stays) as one
        if (!ok) break;
        ptx::tc_fence_after();
        const float4* lse_s = reinterpret_cast<const float4*>(sm.lse2[s]);
        const float4* d_s = reinterpret_cast<const float4*>(sm.dsum[s]);
#pragma unroll 1
        for (int c = 2 * cq; c < 2 * cq + 2; ++c) {
          float sv[32], dpv[32];
          ptx::tmem_ld32(t_s + lane_off + c * 32, sv);
          ptx::tmem_ld32(t_dp + lane_off + c * 32, dpv);
          // the first 8 columns' -LSE log2(e) and -D, read while TMEM answers;
          // each group's values are read one group ahead
          float4 na0 = lse_s[c * 8], na1 = lse_s[c * 8 + 1], nb0 = d_s[c * 8], nb1 = d_s[c * 8 + 1];
          ptx::tmem_wait_ld();
          // query columns this key row is not seen by become -inf (P = 2^-inf = 0, dS = 0)
          if (!full) {
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              const int i = i0 + c * 32 + x;
              sv[x] = (i >= j && i <= jhi) ? sv[x] : -INFINITY;
            }
          }
#pragma unroll
          for (int gq = 0; gq < 4; ++gq) {  // 8 query columns at a time
            const int cb = c * 32 + gq * 8;
            float lse2[8], dd[8];
            lse2[0] = na0.x; lse2[1] = na0.y; lse2[2] = na0.z; lse2[3] = na0.w;
            lse2[4] = na1.x; lse2[5] = na1.y; lse2[6] = na1.z; lse2[7] = na1.w;
            dd[0] = nb0.x; dd[1] = nb0.y; dd[2] = nb0.z; dd[3] = nb0.w;
            dd[4] = nb1.x; dd[5] = nb1.y; dd[6] = nb1.z; dd[7] = nb1.w;
            if (gq < 3) {
              na0 = lse_s[(cb + 8) >> 2];
              na1 = lse_s[(cb + 12) >> 2];
              nb0 = d_s[(cb + 8) >> 2];
              nb1 = d_s[(cb + 12) >> 2];
            }
            uint32_t pw[4], dw[4];
            const float2 sl22 = make_float2(sl2, sl2);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int x = gq * 8 + e;
              const float2 a = __ffma2_rn(make_float2(sv[x], sv[x + 1]), sl22, make_float2(lse2[e], lse2[e + 1]));
              const float2 pp = make_float2(ptx::ex2(a.x), ptx::ex2(a.y));
              const float2 dd2 =
                  __fmul2_rn(pp, __fadd2_rn(make_float2(dpv[x], dpv[x + 1]), make_float2(dd[e], dd[e + 1])));
              pw[e / 2] = ptx::pack_bf16x2(pp.x, pp.y);
              dw[e / 2] = ptx::pack_bf16x2(dd2.x, dd2.y);
            }
            // P^T packs over S^T columns this group has already read: query
            // columns [64 cq, 64 cq + 64) land in TMEM columns [64 cq, 64 cq + 32)
            ptx::tmem_st4(t_s + lane_off + 64 * cq + (c - 2 * cq) * 16 + gq * 4, pw);
            const int c8 = c * 4 + gq;  // 16-byte chunk along the 128 query columns
            *reinterpret_cast<uint4*>(sm.dst[c8 >> 3] + sw128_chunk(r, c8 & 7)) =
                make_uint4(dw[0], dw[1], dw[2], dw[3]);
          }
          // this chunk's P^T and dS^T are in place: part c - 2 cq of the dV and
          // dK~ products may run
          ptx::tmem_wait_st();
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&sm.p_full[c - 2 * cq]);
        }
      }
      if (ok) ok = bwd_wait(&sm.o_full, li & 1, P, abort_flag, 423);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // ---- epilogue: dV and dk = R^T (scale dK~) for this thread's key row.
      // Its TMEM reads all complete (tmem_wait_ld) before this thread's next
      // p_full arrival, which the next item's dV / dK~ products wait for.
      ptx::tc_fence_after();
      const int j_out = key_valid ? (P.rows ? __ldg(P.rows + j) : j) : 0;
      __nv_bfloat16* dvrow = P.dv + ((size_t)j_out * P.Hkv + w.g) * HD;
      __nv_bfloat16* dkrow = P.dk + ((size_t)j_out * P.Hkv + w.g) * HD;
      const int pos = key_valid ? __ldg(P.pos_id + j) : 0;
      auto store32 = [&](__nv_bfloat16* row, int c0, const float* x) {
        uint4* dst = reinterpret_cast<uint4*>(row + c0);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c] = make_uint4(ptx::pack_bf16x2(x[8 * c], x[8 * c + 1]), ptx::pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                              ptx::pack_bf16x2(x[8 * c + 4], x[8 * c + 5]),
                              ptx::pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
      };
      // dk unit u: 32 channels (adjacent pairs or no rotation) or, for the
      // half-split pairing, channels [32u, 32u + 32) with their partners D/2 on
      auto dk_unit = [&](int u) {
        if (P.layout != 1) {
          float x[32];
          ptx::tmem_ld32(t_dk + lane_off + u * 32, x);
          ptx::tmem_wait_ld();
          if (key_valid) {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] *= P.scale;
            if (P.layout == 0) {
              // rope_cs's composition, with each half-unit's 8 pairs of table
              // entries requested together
              const float4* hrow =
                  reinterpret_cast<const float4*>(P.rope_hi + (size_t)(pos >> 5) * (HD / 2) + u * 16);
              const float2* lcol = P.rope_lo + (size_t)(u * 16) * kRopeSplit + (pos & (kRopeSplit - 1));
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                float4 hv[4];
                float2 lv[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) hv[e] = __ldg(hrow + hh * 4 + e);
#pragma unroll
                for (int e = 0; e < 8; ++e) lv[e] = __ldg(lcol + (size_t)(hh * 8 + e) * kRopeSplit);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const float2 a = (e & 1) ? make_float2(hv[e >> 1].z, hv[e >> 1].w)
                                           : make_float2(hv[e >> 1].x, hv[e >> 1].y);
                  const float c = __fmaf_rn(a.x, lv[e].x, -__fmul_rn(a.y, lv[e].y));
                  const float sn = __fmaf_rn(a.y, lv[e].x, __fmul_rn(a.x, lv[e].y));
                  rope_pair(x[16 * hh + 2 * e], x[16 * hh + 2 * e + 1], c, -sn);
                }
              }
            }
            store32(dkrow, u * 32, x);
          }
        } else {
          float x[32], y[32];
          ptx::tmem_ld32(t_dk + lane_off + u * 32, x);
          ptx::tmem_ld32(t_dk + lane_off + HD / 2 + u * 32, y);
          ptx::tmem_wait_ld();
          if (key_valid) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              x[e] *= P.scale;
              y[e] *= P.scale;
              const float2 cs = rope_cs(P.rope_hi, P.rope_lo, pos, u * 32 + e, HD / 2);
              rope_pair(x[e], y[e], cs.x, -cs.y);
            }
            store32(dkrow, u * 32, x);
            store32(dkrow, HD / 2 + u * 32, y);
          }
        }
      };
      // group 0 writes dv and, when there are four dk units (D = 128, adjacent
      // pairs), the first two; group 1 the other dk units
      if (cq == 0) {
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float x[32];
          ptx::tmem_ld32(t_dv + lane_off + c * 32, x);
          ptx::tmem_wait_ld();
          if (key_valid) store32(dvrow, c * 32, x);
        }
        const int nd = P.layout == 1 ? HD / 64 : HD / 32, sp = nd >= 4 ? 2 : 0;  // dk units: all, group 0's
#pragma unroll 1
        for (int u = 0; u < sp; ++u) dk_unit(u);
      } else {
        const int nd = P.layout == 1 ? HD / 64 : HD / 32, sp = nd >= 4 ? 2 : 0;
#pragma unroll 1
        for (int u = sp; u < nd; ++u) dk_unit(u);
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ drain
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int gs = 0;
    bool ok = true;
    for (int li = 0; ok; ++li) {
      int it = read_item(sm, li, P, abort_flag, true, 430);
      if (!ptx::bar_and(3, 128, it >= 0)) break;  // the drain group moves on (or stops) as one
      const BwdItem w = load_item(P, it);
      for (int step = 0; step < w.n_steps && ok; ++step, ++gs) {
        const int h = w.head(step, P.group), i0 = w.qtile(step) * kTile;
        ok = bwd_wait(&sm.dq_full, gs & 1, P, abort_flag, 431);
        ok = ptx::bar_and(3, 128, ok);  // the drain group moves on (or stops) as one
        if (!ok) break;
        ptx::tc_fence_after();
        if constexpr (HD == 128) {
          // lane r = channel. The step's Q~ / dO stage buffers are dead once its
          // MMAs are done, so they hold scale*dQ~ as two [128 rows][64 channels]
          // fp32 blocks: TMEM is released as soon as it is read, and two TMA
          // bulk reductions add the blocks to the accumulator while the next
          // tile computes. The stage returns to the producer once read.
          const int s = gs & 1;
          float* stage = reinterpret_cast<float*>((r >> 6) == 0 ? sm.q[s][0] : sm.dout[s][0]);
          const int ch = r & 63;
          // query rows 0-63, then 64-127: the second pair of TMEM reads is
          // signalled (dq_free) before its shared-memory stores, so the next
          // dP^T product starts as soon as TMEM has been read
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
            float dq[64];
            ptx::tmem_ld32(t_dq + lane_off + hh * 64, dq);
            ptx::tmem_ld32(t_dq + lane_off + hh * 64 + 32, dq + 32);
            ptx::tmem_wait_ld();
            if (hh == 1) {
              ptx::tc_fence_before();
              ptx::mbar_arrive(&sm.dq_free);
            }
#pragma unroll
            for (int e = 0; e < 64; ++e) stage[(hh * 64 + e) * 64 + ch] = P.scale * dq[e];
          }
          ptx::fence_proxy_async_smem();
          asm volatile("bar.sync 3, 128;" ::: "memory");
          if (r == 0) {
            ptx::tma_reduce_add_3d(&tmDQ, sm.q[s][0], 0, h, i0);
            ptx::tma_reduce_add_3d(&tmDQ, sm.dout[s][0], 64, h, i0);
            ptx::bulk_commit();
            ptx::bulk_wait_read0();
            ptx::mbar_arrive(&sm.qd_empty[s]);
          }
          continue;
        } else {
          if (r == 0) ptx::mbar_arrive(&sm.qd_empty[gs & 1]);  // the step's MMAs are done
          const int i = i0 + r;
          float* dst = P.ws.dq_acc + ((size_t)(i < P.T ? i : 0) * P.Hq + h) * HD;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            float dq[32];
            ptx::tmem_ld32(t_dq + lane_off + c * 32, dq);
            ptx::tmem_wait_ld();
            if (i < P.T) {
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                ptx::red_add_v4(dst + c * 32 + e, P.scale * dq[e], P.scale * dq[e + 1], P.scale * dq[e + 2],
                                P.scale * dq[e + 3]);
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&sm.dq_free);
      }
    }
    if constexpr (HD == 128) {
      // the reductions must have read their shared-memory sources before the
      // CTA exits; their global writes complete with the kernel
      if (r == 0) ptx::bulk_wait_read0();
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ LSE/D staging
    const int t = tid - 64;
    int gs = 0;
    bool ok = true;
    for (int li = 0; ok; ++li) {
      const int it = read_item(sm, li, P, abort_flag, true, 440);
      if (it < 0) break;
      const BwdItem w = load_item(P, it);
      for (int step = 0; step < w.n_steps && ok; ++step, ++gs) {
        const int s = gs & 1;
        const int i0 = w.qtile(step) * kTile;
        const size_t hrow = (size_t)w.head(step, P.group) * P.T;
        // the step's rows are read from global memory while its tiles land
        float a[kTile / 64], b[kTile / 64];
#pragma unroll
        for (int u = 0; u < kTile / 64; ++u) {
          const int i = i0 + t + 64 * u;
          const int is = i < P.T && P.rows ? __ldg(P.rows + i) : i;
          a[u] = i < P.T ? -__ldg(P.lse + hrow + is) * kLog2e : -INFINITY;  // -LSE log2(e)
          b[u] = i < P.T ? -__ldg(P.ws.dsum + hrow + i) : 0.f;             // -D
        }
        ok = bwd_wait(&sm.qd_full[s], (gs >> 1) & 1, P, abort_flag, 442);
        if (!ok) break;
#pragma unroll
        for (int u = 0; u < kTile / 64; ++u) {
          sm.lse2[s][t + 64 * u] = a[u];
          sm.dsum[s][t + 64 * u] = b[u];
        }
        ptx::mbar_arrive(&sm.q_ready[s]);
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- 3. dq
// quads = D/8 threads per [T*H] row, each on one channel quad (4 rotation
// pairs, 32 bytes of fp32); a thread takes NB rows per pass and issues all
// their loads first. The rotations of the pass's tokens are composed once
// into shared memory and shared by the token's heads (composing them per row
// made the table lookups, not HBM, the limit).
constexpr int kFinNB = 4;

template <int HD>
__global__ void __launch_bounds__(256) dq_finalize_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                          const int32_t* __restrict__ pos_id,
                                                          const float2* __restrict__ hi_tab,
                                                          const float2* __restrict__ lo_tab, int rows, int H,
                                                          int layout, const int32_t* __restrict__ out_tok) {
  // out_tok (segment plans): the caller token of each kernel token, where
  // its dq row is written (NULL: the same token)
  constexpr int half = HD / 2, quads = half / 4;
  constexpr int RPB = 256 / quads;          // rows per block sub-pass
  constexpr int PASS = kFinNB * RPB;        // rows per pass: at most PASS tokens
  __shared__ float2 cs_s[PASS][half];
  const int qd = threadIdx.x % quads, rsub = threadIdx.x / quads;
  // rows < 2^31, but a pass start plus the grid stride need not be
  for (int64_t p0 = (int64_t)blockIdx.x * PASS; p0 < rows; p0 += (int64_t)gridDim.x * PASS) {
    const int r0 = (int)p0;
    const int r_last = (int)(p0 + PASS < rows ? p0 + PASS - 1 : rows - 1);  // the pass's last row
    float4 u[kFinNB], w[kFinNB];
#pragma unroll
    for (int b = 0; b < kFinNB; ++b) {
      const int64_t ra = p0 + b * RPB + rsub;
      const float* a = acc + (size_t)(ra < rows ? ra : rows - 1) * HD;
      if (layout == 1) {
        u[b] = *reinterpret_cast<const float4*>(a + qd * 4);
        w[b] = *reinterpret_cast<const float4*>(a + half + qd * 4);
      } else {
        u[b] = *reinterpret_cast<const float4*>(a + qd * 8);
        w[b] = *reinterpret_cast<const float4*>(a + qd * 8 + 4);
      }
    }
    const int t_first = r0 / H;
    if (layout != 2) {
      const int n = r_last / H - t_first + 1;
      for (int e = threadIdx.x; e < n * half; e += blockDim.x) {
        const int tt = e / half, pr = e % half;
        cs_s[tt][pr] = rope_cs(hi_tab, lo_tab, __ldg(pos_id + t_first + tt), pr, half);
      }
      __syncthreads();
    }
#pragma unroll
    for (int b = 0; b < kFinNB; ++b) {
      if (p0 + b * RPB + rsub >= rows) break;
      const int row = r0 + b * RPB + rsub;
      __nv_bfloat16* y = dq + (out_tok ? ((size_t)__ldg(out_tok + row / H) * H + row % H) : (size_t)row) * HD;
      float x0[4], x1[4];
      if (layout == 1) {
        x0[0] = u[b].x; x0[1] = u[b].y; x0[2] = u[b].z; x0[3] = u[b].w;
        x1[0] = w[b].x; x1[1] = w[b].y; x1[2] = w[b].z; x1[3] = w[b].w;
      } else {
        x0[0] = u[b].x; x1[0] = u[b].y; x0[1] = u[b].z; x1[1] = u[b].w;
        x0[2] = w[b].x; x1[2] = w[b].y; x0[3] = w[b].z; x1[3] = w[b].w;
      }
      if (layout != 2) {
        const float2* cs = cs_s[row / H - t_first] + qd * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) rope_pair(x0[e], x1[e], cs[e].x, -cs[e].y);
      }
      if (layout == 1) {
        *reinterpret_cast<uint2*>(y + qd * 4) =
            make_uint2(ptx::pack_bf16x2(x0[0], x0[1]), ptx::pack_bf16x2(x0[2], x0[3]));
        *reinterpret_cast<uint2*>(y + half + qd * 4) =
            make_uint2(ptx::pack_bf16x2(x1[0], x1[1]), ptx::pack_bf16x2(x1[2], x1[3]));
      } else {
        *reinterpret_cast<uint4*>(y + qd * 8) =
            make_uint4(ptx::pack_bf16x2(x0[0], x1[0]), ptx::pack_bf16x2(x0[1], x1[1]),
                       ptx::pack_bf16x2(x0[2], x1[2]), ptx::pack_bf16x2(x0[3], x1[3]));
      }
    }
    if (layout != 2) __syncthreads();  // cs_s is rewritten by the next pass
  }
}

// ---------------------------------------------------------------- 4. anchor
// One block per kv head. The kPrepChunks row chunks are split into runs of
// consecutive chunks, each summed by its own thread (many loads in flight
// instead of one long dependent walk), and the runs are combined in run
// order, so the sums are run-to-run deterministic.
constexpr int kAnchorThreads = 512;
static_assert(kPrepChunks % (kAnchorThreads / 64) == 0, "row chunks split evenly into runs at D = 64 and 128");

__global__ void __launch_bounds__(kAnchorThreads)
    anchor_finalize_kernel(Workspace ws, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                           const int32_t* __restrict__ pos_id, const float2* __restrict__ hi_tab,
                           const float2* __restrict__ lo_tab, int Hq, int Hkv, int D, int layout) {
  const int g = blockIdx.x, group = Hq / Hkv;
  const int runs = kAnchorThreads / D;  // 4 at D = 128, 8 at D = 64
  const int per = kPrepChunks / runs;
  const int c = threadIdx.x % D, run = threadIdx.x / D;
  extern __shared__ float sh[];  // [2][runs][D] run sums, then [2][D] totals (dv, dk)
  float sdv = 0.f, sdk = 0.f;
  const size_t stride = (size_t)Hq * D;
  for (int hh = 0; hh < group; ++hh) {
    const float* pv = ws.part_dv + (size_t)(g * group + hh) * D + c;
    const float* pk = ws.part_dk + (size_t)(g * group + hh) * D + c;
#pragma unroll 8
    for (int b = run * per; b < (run + 1) * per; ++b) {
      sdv += pv[b * stride];
      sdk += pk[b * stride];
    }
  }
  sh[run * D + c] = sdv;
  sh[(runs + run) * D + c] = sdk;
  __syncthreads();
  float* tot = sh + 2 * runs * D;
  if (threadIdx.x < D) {
    float a = 0.f, b = 0.f;
    for (int q = 0; q < runs; ++q) {
      a += sh[q * D + c];
      b += sh[(runs + q) * D + c];
    }
    tot[c] = a;
    tot[D + c] = b;
  }
  __syncthreads();
  const int pos = __ldg(pos_id);
  for (int p = threadIdx.x; p < D / 2; p += blockDim.x) {
    const int ia = layout == 1 ? p : 2 * p, ib = layout == 1 ? p + D / 2 : 2 * p + 1;
    float a = tot[D + ia], b = tot[D + ib];
    if (layout != 2) {
      const float2 cs = rope_cs(hi_tab, lo_tab, pos, p, D / 2);
      rope_pair(a, b, cs.x, -cs.y);
    }
    dk[(size_t)g * D + ia] = __float2bfloat16_rn(a);
    dk[(size_t)g * D + ib] = __float2bfloat16_rn(b);
    dv[(size_t)g * D + ia] = __float2bfloat16_rn(tot[ia]);
    dv[(size_t)g * D + ib] = __float2bfloat16_rn(tot[ib]);
  }
}

template <int HD>
aa_status launch_bwd(aa_plan_s* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, void* workspace, cudaStream_t s,
                     const void* qr_in, const void* kr_in, const int32_t* rows, void* dout_g) {
  size_t need = 0;
  const bool given = qr_in != nullptr;  // rotated Q and K from a forward workspace
  Workspace ws = carve(workspace, p, &need, !given);
  cudaError_t e;
  const int rope_layout = p->cfg.rope_layout;
  // Q is the streaming operand of the key-stationary tile loop: rotate it
  // once here rather than on every visit (or take the forward's rotation)
  const void* qr = given ? qr_in : q;
  const void* kr = given ? kr_in : k;
  if (rope_layout != AA_ROPE_NONE && !given) {
    aa_status rs = launch_rope(p, q, ws.qr, p->Hq, 0, s, nullptr, rows);
    if (rs == AA_OK) rs = launch_rope(p, k, ws.kr, p->Hkv, 0, s, nullptr, rows);
    if (rs != AA_OK) return rs;
    qr = ws.qr;
    kr = ws.kr;
  }
  bwd_prep_kernel<HD><<<dim3(p->Hq, kPrepChunks), kPrepThreads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(qr), static_cast<const __nv_bfloat16*>(kr),
      static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(o),
      static_cast<const __nv_bfloat16*>(dout), lse, ws, p->T, p->Hq, p->group, p->anchor ? 1 : 0, p->scale, rows,
      rows ? static_cast<__nv_bfloat16*>(dout_g) : nullptr);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "bwd_prep_kernel launch");

  CUtensorMap tq, tk, tv, tdo;
  aa_status st;
  if ((st = make_tile_map(&tq, qr, p->T, p->Hq, HD)) != AA_OK) return st;
  if ((st = make_tile_map(&tk, kr, p->T, p->Hkv, HD)) != AA_OK) return st;
  if ((st = make_tile_map(&tv, v, p->T, p->Hkv, HD)) != AA_OK) return st;
  if ((st = make_tile_map(&tdo, rows ? dout_g : dout, p->T, p->Hq, HD)) != AA_OK) return st;
  CUtensorMap tdq;
  if ((st = make_f32_map(&tdq, ws.dq_acc, p->T, p->Hq, HD, 64, kTile)) != AA_OK) return st;
  BwdParams P;
  P.dk = static_cast<__nv_bfloat16*>(dk);
  P.dv = static_cast<__nv_bfloat16*>(dv);
  P.lse = lse;
  P.ws = ws;
  P.pos_id = p->dev.pos_id;
  P.key_hi = p->dev.key_hi;
  P.rows = rows;
  P.items = p->dev.bwd_items;
  P.next_item = ws.next_item;
  P.n_items = (int)p->bwd_items.size();
  P.rope_hi = p->dev.rope_hi;
  P.rope_lo = p->dev.rope_lo;
  P.rope_step = p->dev.rope_step;
  P.err = p->dev.err;
  P.wait_limit_ns = p->wait_limit_ns;
  P.T = p->T;
  P.Hq = p->Hq;
  P.Hkv = p->Hkv;
  P.group = p->group;
  P.layout = rope_layout;
  P.scale = p->scale;
  const size_t smem = sizeof(BwdSmem<HD>);
  static std::once_flag attr_once[kMaxDevices];
  static cudaError_t attr_result[kMaxDevices];
  e = once_per_device(attr_once, attr_result, p->device, [&] {
    return cudaFuncSetAttribute(attn_bwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd_kernel smem attribute");
  if (p->bwd_ev_start && (e = cudaEventRecord(p->bwd_ev_start, s)) != cudaSuccess)
    return cuda_fail(e, "recording the bwd start event");
  // persistent: one CTA per SM (fewer for short work lists)
  const unsigned n_cta = (unsigned)std::min<size_t>(p->bwd_items.size(), (size_t)std::max(p->num_sms, 1));
  if (!p->bwd_items.empty()) {
    attn_bwd_kernel<HD><<<n_cta, kBwdThreads, smem, s>>>(tq, tk, tv, tdo, tdq, P);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "attn_bwd_kernel launch");
  }
  if (p->bwd_ev_stop && (e = cudaEventRecord(p->bwd_ev_stop, s)) != cudaSuccess)
    return cuda_fail(e, "recording the bwd stop event");

  // one full wave of resident blocks, grid-striding over the rows
  static std::once_flag occ_once[kMaxDevices];
  static int occ_result[kMaxDevices];
  const int occ = once_per_device(occ_once, occ_result, p->device, [] {
    int n = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dq_finalize_kernel<HD>, 256, 0) == cudaSuccess && n > 0
               ? n
               : 4;
  });
  const int rows_total = p->T * p->Hq;  // below 2^31: the plan checks T * Hq
  const int per_block = kFinNB * (256 / (HD / 8));
  const int64_t blocks =
      std::min<int64_t>((rows_total + per_block - 1) / per_block, (int64_t)p->num_sms * std::max(occ, 1));
  dq_finalize_kernel<HD><<<(unsigned)blocks, 256, 0, s>>>(ws.dq_acc, static_cast<__nv_bfloat16*>(dq),
                                                          p->dev.pos_id, p->dev.rope_hi, p->dev.rope_lo, rows_total,
                                                          p->Hq, rope_layout, rows);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "dq_finalize_kernel launch");
  if (p->anchor) {
    anchor_finalize_kernel<<<p->Hkv, kAnchorThreads, (2 * kAnchorThreads + 2 * HD) * sizeof(float), s>>>(
        ws, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), p->dev.pos_id, p->dev.rope_hi,
        p->dev.rope_lo, p->Hq, p->Hkv, HD, rope_layout);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "anchor_finalize_kernel launch");
  }
  return AA_OK;
}

}  // namespace

aa_status launch_bwd_with_workspace(aa_plan_s* p, const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                    void* workspace, cudaStream_t s, const void* qr, const void* kr,
                                    const int32_t* rows, void* dout_g) {
  return p->D == 128 ? launch_bwd<128>(p, q, k, v, o, lse, dout, dq, dk, dv, workspace, s, qr, kr, rows, dout_g)
                     : launch_bwd<64>(p, q, k, v, o, lse, dout, dq, dk, dv, workspace, s, qr, kr, rows, dout_g);
}

size_t bwd_base_workspace_bytes(const aa_plan_s* p, bool with_rot) {
  if (!p) return 0;
  size_t total = 0;
  carve(nullptr, p, &total, with_rot);
  return total;
}

}  // namespace aa

using namespace aa;

extern "C" size_t aa_bwd_workspace_bytes(aa_plan_t p) {
  if (!p) return 0;
  return bwd_base_workspace_bytes(p) + (p->segmented ? seg_bwd_extra_bytes(p) : 0);
}

extern "C" aa_status aa_bwd(aa_plan_t p, const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                            size_t workspace_bytes, aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* x : ptrs) {
    if (!x) return fail(AA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(x)) return fail(AA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  }
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(AA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  if (workspace_bytes < aa_bwd_workspace_bytes(p))
    return fail(AA_ERR_INVALID_ARG, "workspace is smaller than aa_bwd_workspace_bytes()");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->segmented) return seg_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, workspace, s);
  return launch_bwd_with_workspace(p, q, k, v, o, lse, dout, dq, dk, dv, workspace, s);
}

extern "C" size_t aa_bwd_from_fwd_workspace_bytes(aa_plan_t p) {
  if (!p) return 0;
  return bwd_base_workspace_bytes(p, false) + (p->segmented ? seg_bwd_extra_bytes(p, false) : 0);
}

extern "C" aa_status aa_bwd_from_fwd(aa_plan_t p, const void* fwd_workspace, const void* v, const void* o,
                                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                     void* workspace, size_t workspace_bytes, aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  if (p->cfg.rope_layout == AA_ROPE_NONE)
    return fail(AA_ERR_UNSUPPORTED, "with AA_ROPE_NONE aa_fwd keeps no rotated operands: call aa_bwd");
  const void* ptrs[] = {v, o, lse, dout, dq, dk, dv};
  for (const void* x : ptrs) {
    if (!x) return fail(AA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(x)) return fail(AA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  }
  if (!fwd_workspace || (reinterpret_cast<uintptr_t>(fwd_workspace) & 255u))
    return fail(AA_ERR_INVALID_ARG, "fwd_workspace must be the 256-byte aligned workspace of an aa_fwd call");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(AA_ERR_INVALID_ARG, "workspace must be a 256-byte aligned device pointer");
  if (workspace_bytes < aa_bwd_from_fwd_workspace_bytes(p))
    return fail(AA_ERR_INVALID_ARG, "workspace is smaller than aa_bwd_from_fwd_workspace_bytes()");
  const void *qr = nullptr, *kr = nullptr;
  fwd_rotated_operands(p, fwd_workspace, &qr, &kr);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->segmented)
    return seg_bwd(p, nullptr, nullptr, v, o, lse, dout, dq, dk, dv, workspace, s, qr, kr,
                   fwd_grouped_v(p, fwd_workspace));
  return launch_bwd_with_workspace(p, nullptr, nullptr, v, o, lse, dout, dq, dk, dv, workspace, s, qr, kr);
}
