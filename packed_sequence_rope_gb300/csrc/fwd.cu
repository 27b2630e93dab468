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
// How: one CTA per (query tile of 128 rows, head) work item, items in
// longest-first order. Q and K/V tiles arrive by TMA (128-byte swizzle), are
// rotated in shared memory in fp32 and rounded to bf16 (RoPE fused into the
// tile load), S = Q~ K~^T and O += P V run on the tcgen05 tensor cores with
// fp32 accumulators in TMEM, and the online softmax runs one query row per
// thread straight from TMEM. Only the key tiles that overlap the row
// intervals of the tile are visited; the anchor column is folded into the
// softmax's starting state on the CUDA cores (m = s_i0, l = 1, weight of v_0),
// so fully cross-document tiles are never touched.
#include "kcommon.cuh"

namespace aa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

template <int HD>
struct FwdSmem {
  static constexpr int kBlocks = HD / 64;
  alignas(1024) uint8_t q[kBlocks][16384];
  alignas(1024) uint8_t k[kBlocks][16384];
  alignas(1024) uint8_t v[kBlocks][16384];
  alignas(1024) uint8_t p[2][16384];  // P tile: 128 query rows x 128 keys, bf16
  float k0[HD];                       // rotated anchor key (bf16-rounded)
  float v0[HD];                       // anchor value
  uint64_t bar_q, bar_kv, bar_mma;
  uint32_t tmem_base;
};

struct FwdParams {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  const int32_t* pos_id;
  const int32_t* row_lo;
  const WorkItem* items;
  const float2* rope_hi;
  const float2* rope_lo;
  int32_t* err;
  uint64_t wait_limit_ns;
  int T, Hq, Hkv, group, layout, anchor;
  float scale;
};

constexpr uint64_t kDrainLimitNs = 1000000000ull;

template <int HD>
__global__ void __launch_bounds__(128, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams P) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem<HD>& sm = *reinterpret_cast<FwdSmem<HD>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                    ~uintptr_t(1023));
  constexpr int kTmemCols = 256;  // S: 128 columns, O: HD columns
  constexpr uint32_t kTileBytes = 128 * HD * 2;
  const int tid = threadIdx.x, warp = tid >> 5;
  const WorkItem item = P.items[blockIdx.x];
  const int qt = item.tile, h = item.head, g = h / P.group;
  const int row0 = qt * kTile;

  if (tid == 0) {
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
    ptx::mbar_init(&sm.bar_q, 1);
    ptx::mbar_init(&sm.bar_kv, 1);
    ptx::mbar_init(&sm.bar_mma, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 128;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  // thread 0 tracks what is in flight so an aborted CTA can drain it
  bool kv_pending = false, mma_pending = false, q_pending = false;
  uint32_t kv_phase = 0, mma_phase = 0;

  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(&sm.bar_q, kTileBytes);
    for (int b = 0; b < HD / 64; ++b) ptx::tma_load_3d(sm.q[b], &tmQ, &sm.bar_q, b * 64, h, row0);
    ptx::mbar_arrive_expect_tx(&sm.bar_kv, 2 * kTileBytes);
    for (int b = 0; b < HD / 64; ++b) {
      ptx::tma_load_3d(sm.k[b], &tmK, &sm.bar_kv, b * 64, g, item.lo * kTile);
      ptx::tma_load_3d(sm.v[b], &tmV, &sm.bar_kv, b * 64, g, item.lo * kTile);
    }
    q_pending = kv_pending = true;
  }

  // anchor key (rotated like any key, rounded to bf16) and value
  if (P.anchor) {
    const int pos0 = __ldg(P.pos_id);
    const __nv_bfloat16* k0 = P.k + (size_t)g * HD;
    const __nv_bfloat16* v0 = P.v + (size_t)g * HD;
    for (int c = tid; c < HD; c += 128) sm.v0[c] = __bfloat162float(v0[c]);
    if (tid < HD / 2) {
      int ia, ib;
      if (P.layout == 1) { ia = tid; ib = tid + HD / 2; } else { ia = 2 * tid; ib = 2 * tid + 1; }
      float x = __bfloat162float(k0[ia]), y = __bfloat162float(k0[ib]);
      if (P.layout != 2) {
        const float2 cs = rope_cs(P.rope_hi, P.rope_lo, pos0, tid, HD / 2);
        rope_pair(x, y, cs.x, cs.y);
      }
      sm.k0[ia] = __bfloat162float(__float2bfloat16_rn(x));
      sm.k0[ib] = __bfloat162float(__float2bfloat16_rn(y));
    }
  }

  const int r = tid;  // this thread's query row within the tile == TMEM lane
  const int i = row0 + r;
  const bool row_valid = i < P.T;
  const int lo = row_valid ? __ldg(P.row_lo + i) : 1;
  const int hi = row_valid ? i : 0;
  const float sl2 = P.scale * kLog2e;

  bool ok = ptx::mbar_wait(&sm.bar_q, 0, P.wait_limit_ns, P.err, 101);
  if (__syncthreads_or(!ok)) goto abort;
  if (tid == 0) q_pending = false;
  if (row_valid) rope_row_smem<HD>(sm.q[0], r, __ldg(P.pos_id + i), P.layout, false, P.rope_hi, P.rope_lo);
  ptx::fence_proxy_async_smem();
  __syncthreads();

  {
    // online-softmax state in log2 units
    float m = -INFINITY, l = 0.f, s0 = 0.f;
    if (P.anchor) {
      float acc = 0.f;
      for (int c = 0; c < HD; ++c) acc = fmaf(tile_elem(sm.q[0], r, c), sm.k0[c], acc);
      s0 = acc * sl2;
      m = s0;
      l = 1.f;
    }
    constexpr uint32_t idesc_s = ptx::idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(128, HD, 0, 1);
    const int n_iter = item.hi - item.lo + 1;
    for (int it = 0; it < n_iter; ++it) {
      const int kt = item.lo + it;
      ok = ptx::mbar_wait(&sm.bar_kv, kv_phase, P.wait_limit_ns, P.err, 102);
      if (__syncthreads_or(!ok)) goto abort;
      if (tid == 0) kv_pending = false;
      kv_phase ^= 1;
      {
        const int j = kt * kTile + r;
        if (j < P.T) rope_row_smem<HD>(sm.k[0], r, __ldg(P.pos_id + j), P.layout, false, P.rope_hi, P.rope_lo);
      }
      ptx::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t a = ptx::smem_desc_sw128(ptx::smem_u32(sm.q[0]) + off, 16, 1024);
          const uint64_t b = ptx::smem_desc_sw128(ptx::smem_u32(sm.k[0]) + off, 16, 1024);
          ptx::mma_bf16(tmem_s, a, b, idesc_s, kk > 0);
        }
        ptx::mma_commit(&sm.bar_mma);
        mma_pending = true;
      }
      ok = ptx::mbar_wait(&sm.bar_mma, mma_phase, P.wait_limit_ns, P.err, 103);
      if (__syncthreads_or(!ok)) goto abort;
      if (tid == 0) mma_pending = false;
      mma_phase ^= 1;
      ptx::tc_fence_after();

      // ---- softmax on this thread's row
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tmem_s + lane_off + c * 32, sv + c * 32);
      ptx::tmem_wait_ld();
      const int j0 = kt * kTile;
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const int j = j0 + c;
        const bool vis = (j >= lo) && (j <= hi);
        sv[c] = vis ? sv[c] * sl2 : -INFINITY;
        mt = fmaxf(mt, sv[c]);
      }
      // TMEM loads/stores are warp-collective, so the rescale decision is
      // taken per warp: if any row of the warp needs it, every row of the
      // warp moves to max(m, mt) (a factor of 1 where the max did not grow)
      const bool need = (mt > m + kRescaleThreshold) || (m == -INFINITY && mt > -INFINITY);
      if (__any_sync(0xffffffffu, need)) {
        const float mn = fmaxf(m, mt);
        const float f = (m == -INFINITY) ? 0.f : exp2f(m - mn);
        l *= f;
        if (it > 0) {
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) {
            float ov[32];
            ptx::tmem_ld32(tmem_o + lane_off + c * 32, ov);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] *= f;
            ptx::tmem_st32(tmem_o + lane_off + c * 32, ov);
          }
          ptx::tmem_wait_st();
        }
        m = mn;
      }
      float rs = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < 16; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = (m == -INFINITY) ? 0.f : exp2f(sv[c8 * 8 + 2 * e] - m);
          const float p1 = (m == -INFINITY) ? 0.f : exp2f(sv[c8 * 8 + 2 * e + 1] - m);
          rs += p0 + p1;
          w[e] = ptx::pack_bf16x2(p0, p1);
        }
        *reinterpret_cast<uint4*>(sm.p[c8 >> 3] + sw128_chunk(r, c8 & 7)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      l += rs;
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t a = ptx::smem_desc_sw128(ptx::smem_u32(sm.p[0]) + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          const uint64_t b = ptx::smem_desc_sw128(ptx::smem_u32(sm.v[0]) + kk * 2048, 16384, 1024);
          ptx::mma_bf16(tmem_o, a, b, idesc_pv, (it > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&sm.bar_mma);
        mma_pending = true;
      }
      ok = ptx::mbar_wait(&sm.bar_mma, mma_phase, P.wait_limit_ns, P.err, 104);
      if (__syncthreads_or(!ok)) goto abort;
      mma_phase ^= 1;
      if (tid == 0) {
        mma_pending = false;
        if (it + 1 < n_iter) {
          ptx::mbar_arrive_expect_tx(&sm.bar_kv, 2 * kTileBytes);
          for (int b = 0; b < HD / 64; ++b) {
            ptx::tma_load_3d(sm.k[b], &tmK, &sm.bar_kv, b * 64, g, (kt + 1) * kTile);
            ptx::tma_load_3d(sm.v[b], &tmV, &sm.bar_kv, b * 64, g, (kt + 1) * kTile);
          }
          kv_pending = true;
        }
      }
      ptx::tc_fence_after();
    }

    // ---- epilogue: O = (O_tiles + w0 * v0) / l, LSE = ln(l) + m ln 2
    const float w0 = P.anchor ? exp2f(s0 - m) : 0.f;
    const float inv_l = 1.f / l;
    __nv_bfloat16* orow = P.o + ((size_t)(row_valid ? i : 0) * P.Hq + h) * HD;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float ov[32];
      ptx::tmem_ld32(tmem_o + lane_off + c * 32, ov);  // warp-collective: every lane loads
      ptx::tmem_wait_ld();
      if (row_valid) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a = (ov[2 * e] + w0 * sm.v0[c * 32 + 2 * e]) * inv_l;
          const float b = (ov[2 * e + 1] + w0 * sm.v0[c * 32 + 2 * e + 1]) * inv_l;
          w[e] = ptx::pack_bf16x2(a, b);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
      }
    }
    if (row_valid) P.lse[(size_t)h * P.T + i] = (m + log2f(l)) * 0.69314718055994531f;
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
  return;

abort:
  // a bounded wait ran out: let in-flight copies and MMAs land, free TMEM, return
  if (tid == 0) {
    if (q_pending) ptx::mbar_wait(&sm.bar_q, 0, kDrainLimitNs, P.err, 199);
    if (kv_pending) ptx::mbar_wait(&sm.bar_kv, kv_phase, kDrainLimitNs, P.err, 199);
    if (mma_pending) ptx::mbar_wait(&sm.bar_mma, mma_phase, kDrainLimitNs, P.err, 199);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) ptx::tmem_dealloc(tmem, kTmemCols);
}

template <int HD>
aa_status launch_fwd(aa_plan_s* p, const void* q, const void* k, const void* v, void* o, float* lse,
                     cudaStream_t s) {
  CUtensorMap tq, tk, tv;
  aa_status st;
  if ((st = make_tile_map(&tq, q, p->T, p->Hq, HD)) != AA_OK) return st;
  if ((st = make_tile_map(&tk, k, p->T, p->Hkv, HD)) != AA_OK) return st;
  if ((st = make_tile_map(&tv, v, p->T, p->Hkv, HD)) != AA_OK) return st;
  FwdParams P;
  P.k = static_cast<const __nv_bfloat16*>(k);
  P.v = static_cast<const __nv_bfloat16*>(v);
  P.o = static_cast<__nv_bfloat16*>(o);
  P.lse = lse;
  P.pos_id = p->dev.pos_id;
  P.row_lo = p->dev.row_lo;
  P.items = p->dev.fwd_items;
  P.rope_hi = p->dev.rope_hi;
  P.rope_lo = p->dev.rope_lo;
  P.err = p->dev.err;
  P.wait_limit_ns = p->wait_limit_ns;
  P.T = p->T;
  P.Hq = p->Hq;
  P.Hkv = p->Hkv;
  P.group = p->group;
  P.layout = p->cfg.rope_layout;
  P.anchor = p->anchor ? 1 : 0;
  P.scale = p->scale;
  const size_t smem = sizeof(FwdSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_kernel smem attribute");
  const unsigned n_items = (unsigned)p->fwd_items.size();
  attn_fwd_kernel<HD><<<n_items, 128, smem, s>>>(tq, tk, tv, P);
  e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "attn_fwd_kernel launch");
}

}  // namespace
}  // namespace aa

using namespace aa;

extern "C" aa_status aa_fwd(aa_plan_t p, const void* q, const void* k, const void* v, void* o, float* lse,
                            aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  if (!q || !k || !v || !o || !lse) return fail(AA_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(AA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return p->D == 128 ? launch_fwd<128>(p, q, k, v, o, lse, s) : launch_fwd<64>(p, q, k, v, o, lse, s);
}
