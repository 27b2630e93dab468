// Shift-discrepancy diagnostics ("When Precision Meets Position", architecture
// page, §3.4 "Diagnostic Methodology: Measuring the Breakdown"):
//   Eq. 4  D       = sum_h sum_j n_j sum_i |ATTN_ij(Δ1) - ATTN_ij(Δ2)|,
//                    n_j = 1 / (rows that may attend to key j)
//   Eq. 5  D_logit = (1/T) sum_h sum_i |A_{i,first}(Δ1) - A_{i,first}(Δ2)|
// for one input under two shifts of every position (Eq. 3 says both are zero
// under exact arithmetic). The rotated operands are the library's own bf16
// Q~, K~ from the RoPE kernel (fp32 rotation, rounded to bf16), so the numbers
// measure this library's arithmetic.
//
// This runs once per evaluation, not per training step: the logits are
// recomputed on CUDA cores (bf16 products are exact in fp32, fp32 sums, as
// the tensor-core path does) in two passes over the visible keys, the first
// for each row's softmax statistics under both shifts, the second for
// |ATTN(Δ1) - ATTN(Δ2)| summed into per-key columns.
#include "kcommon.cuh"

namespace aa {
namespace {

constexpr int kRows = 32;    // query rows per CTA
constexpr int kKeys = 32;    // keys per shared-memory chunk
constexpr int kThreads = 256;

template <int HD>
struct DiagSmem {
  static constexpr int kPitch = HD + 8;  // bf16 elements per row: 16-byte pad spreads banks
  __nv_bfloat16 q[2][kRows][kPitch];
  __nv_bfloat16 k[2][kKeys][kPitch];
  float col[kKeys];
};

// dot(a, b) over HD bf16 channels in fp32, 16 bytes at a time
template <int HD>
__device__ __forceinline__ float dot_bf16(const __nv_bfloat16* a, const __nv_bfloat16* b) {
  float acc = 0.f;
#pragma unroll 4
  for (int c = 0; c < HD; c += 8) {
    const uint4 x = *reinterpret_cast<const uint4*>(a + c), y = *reinterpret_cast<const uint4*>(b + c);
    const uint32_t xa[4] = {x.x, x.y, x.z, x.w}, ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 u = ptx::unpack_bf16x2(xa[e]), v = ptx::unpack_bf16x2(ya[e]);
      acc = fmaf(u.x, v.x, acc);
      acc = fmaf(u.y, v.y, acc);
    }
  }
  return acc;
}

struct DiagParams {
  const __nv_bfloat16* q[2];  // rotated Q under shift 1 / shift 2, [T, Hq, D]
  const __nv_bfloat16* k[2];  // rotated K, [T, Hkv, D]
  const int32_t* row_lo;      // row i sees keys [row_lo_i, i] (plus key 0 with the anchor)
  float* col;                 // [Hq, T] sum_i |ATTN_ij(Δ1) - ATTN_ij(Δ2)|, zeroed by the host
  float* first;               // [Hq, T] |A_i0(Δ1) - A_i0(Δ2)| (0 where row i cannot see key 0)
  int T, Hq, Hkv, group, anchor;
  float scale;
};

// One CTA per (32 query rows, query head); thread = (row r = tid / 8, key
// slot kg = tid % 8), covering keys kg, kg + 8, kg + 16, kg + 24 of a chunk.
template <int HD>
__global__ void __launch_bounds__(kThreads) shift_diag_kernel(const DiagParams P) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  DiagSmem<HD>& sm = *reinterpret_cast<DiagSmem<HD>*>(smem_raw);
  const int tid = threadIdx.x, r = tid >> 3, kg = tid & 7;
  const int h = blockIdx.y, g = h / P.group;
  const int R0 = blockIdx.x * kRows;
  const int i = R0 + r;
  const bool row_valid = i < P.T;
  const int lo = row_valid ? __ldg(P.row_lo + i) : 1;
  const int hi = row_valid ? i : 0;

  // the block's query rows under both shifts
  for (int e = tid; e < 2 * kRows * (HD / 8); e += kThreads) {
    const int s = e / (kRows * (HD / 8)), rr = (e / (HD / 8)) % kRows, c8 = e % (HD / 8);
    const int ii = R0 + rr;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (ii < P.T) v = *reinterpret_cast<const uint4*>(P.q[s] + ((size_t)ii * P.Hq + h) * HD + c8 * 8);
    *reinterpret_cast<uint4*>(&sm.q[s][rr][c8 * 8]) = v;
  }
  // key chunks: [first visible key of the block, last row], plus the chunk
  // holding key 0 when the anchor is visible from outside that range
  const int k_first = __ldg(P.row_lo + R0) / kKeys;  // row_lo is non-decreasing
  const int k_last = min(P.T - 1, R0 + kRows - 1) / kKeys;
  const bool extra0 = P.anchor && k_first > 0;
  const int n_chunks = (k_last - k_first + 1) + (extra0 ? 1 : 0);
  auto chunk_base = [&](int c) { return extra0 ? (c == 0 ? 0 : (k_first + c - 1) * kKeys) : (k_first + c) * kKeys; };
  auto visible = [&](int j) { return row_valid && ((j >= lo && j <= hi) || (P.anchor && j == 0)); };
  auto load_keys = [&](int j0) {
    __syncthreads();  // the previous chunk is no longer read
    for (int e = tid; e < 2 * kKeys * (HD / 8); e += kThreads) {
      const int s = e / (kKeys * (HD / 8)), kk = (e / (HD / 8)) % kKeys, c8 = e % (HD / 8);
      const int j = j0 + kk;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (j < P.T) v = *reinterpret_cast<const uint4*>(P.k[s] + ((size_t)j * P.Hkv + g) * HD + c8 * 8);
      *reinterpret_cast<uint4*>(&sm.k[s][kk][c8 * 8]) = v;
    }
    __syncthreads();
  };

  // pass 1: per-thread online softmax statistics for both shifts
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, a0[2] = {0.f, 0.f};
  bool sees0 = false;
  for (int c = 0; c < n_chunks; ++c) {
    const int j0 = chunk_base(c);
    load_keys(j0);
#pragma unroll
    for (int t = 0; t < kKeys / 8; ++t) {
      const int kk = kg + 8 * t, j = j0 + kk;
      if (!visible(j)) continue;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const float a = P.scale * dot_bf16<HD>(&sm.q[s][r][0], &sm.k[s][kk][0]);
        if (j == 0) a0[s] = a;
        const float mn = fmaxf(m[s], a);
        l[s] = l[s] * expf(m[s] - mn) + expf(a - mn);
        m[s] = mn;
      }
      if (j == 0) sees0 = true;
    }
  }
  // combine the row's 8 threads (consecutive lanes)
  float lse[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[s], off), lo_ = __shfl_xor_sync(0xffffffffu, l[s], off);
      const float mn = fmaxf(m[s], mo);
      l[s] = (mn == -INFINITY) ? 0.f : l[s] * expf(m[s] - mn) + lo_ * expf(mo - mn);
      m[s] = mn;
    }
    lse[s] = m[s] + logf(l[s]);
  }
  // Eq. 5: the first token's logit under both shifts (held by the thread of key 0)
  // (the output was cleared, so rows that cannot see key 0 keep 0)
  if (sees0) P.first[(size_t)h * P.T + i] = fabsf(a0[0] - a0[1]);

  // pass 2: |ATTN(Δ1) - ATTN(Δ2)| summed into the key columns
  for (int c = 0; c < n_chunks; ++c) {
    const int j0 = chunk_base(c);
    if (tid < kKeys) sm.col[tid] = 0.f;
    load_keys(j0);
#pragma unroll
    for (int t = 0; t < kKeys / 8; ++t) {
      const int kk = kg + 8 * t, j = j0 + kk;
      if (!visible(j)) continue;
      const float p1 = expf(P.scale * dot_bf16<HD>(&sm.q[0][r][0], &sm.k[0][kk][0]) - lse[0]);
      const float p2 = expf(P.scale * dot_bf16<HD>(&sm.q[1][r][0], &sm.k[1][kk][0]) - lse[1]);
      atomicAdd(&sm.col[kk], fabsf(p1 - p2));
    }
    __syncthreads();
    if (tid < kKeys && j0 + tid < P.T && sm.col[tid] != 0.f) atomicAdd(P.col + (size_t)h * P.T + j0 + tid, sm.col[tid]);
  }
}

// One CTA: per head D_h = sum_j col_hj / count_j and L_h = sum_i first_hi,
// then D = sum_h D_h and D_logit = (1/T) sum_h L_h; fixed-order fp64 sums.
// count_j = rows that may attend to key j = key_hi_j - j + 1, or T for the
// anchor key.
__global__ void __launch_bounds__(kThreads) shift_diag_reduce_kernel(const float* __restrict__ col,
                                                                     const float* __restrict__ first,
                                                                     const int32_t* __restrict__ key_hi, int T,
                                                                     int Hq, int anchor, double* out) {
  __shared__ double red[2][kThreads];
  double tot_d = 0.0, tot_l = 0.0;
  for (int h = 0; h < Hq; ++h) {
    double sd = 0.0, sl = 0.0;
    for (int j = threadIdx.x; j < T; j += kThreads) {
      const int cnt = (anchor && j == 0) ? T : __ldg(key_hi + j) - j + 1;
      if (cnt > 0) sd += (double)col[(size_t)h * T + j] / cnt;
      sl += (double)first[(size_t)h * T + j];
    }
    red[0][threadIdx.x] = sd;
    red[1][threadIdx.x] = sl;
    __syncthreads();
    for (int w = kThreads / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w) {
        red[0][threadIdx.x] += red[0][threadIdx.x + w];
        red[1][threadIdx.x] += red[1][threadIdx.x + w];
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      out[2 + 2 * h] = red[0][0];
      out[3 + 2 * h] = red[1][0];
      tot_d += red[0][0];
      tot_l += red[1][0];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    out[0] = tot_d;
    out[1] = tot_l / T;
  }
}

bool same_problem(const aa_plan_s* a, const aa_plan_s* b) {
  return a->T == b->T && a->Hq == b->Hq && a->Hkv == b->Hkv && a->D == b->D &&
         a->cfg.mask_mode == b->cfg.mask_mode && a->cfg.pos_mode == b->cfg.pos_mode &&
         a->cfg.rope_layout == b->cfg.rope_layout && a->theta == b->theta && a->scale == b->scale &&
         a->cu == b->cu && a->device == b->device;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace aa

using namespace aa;

extern "C" size_t aa_shift_diag_workspace_bytes(aa_plan_t p) {
  if (!p || p->cfg.rope_layout == AA_ROPE_NONE) return 0;
  return 2 * (align256((size_t)p->T * p->Hq * p->D * 2) + align256((size_t)p->T * p->Hkv * p->D * 2));
}

extern "C" aa_status aa_shift_diag(aa_plan_t p1, aa_plan_t p2, const void* q, const void* k, float* col_absdiff,
                                   float* first_logit_absdiff, double* result, void* workspace,
                                   size_t workspace_bytes, aa_stream_t stream) {
  aa_status st = check_compute_plan(p1);
  if (st != AA_OK) return st;
  if ((st = check_compute_plan(p2)) != AA_OK) return st;
  if (p1->segmented || p2->segmented)
    return fail(AA_ERR_UNSUPPORTED, "aa_shift_diag: segment plans are not supported");
  if (!same_problem(p1, p2))
    return fail(AA_ERR_INVALID_ARG, "aa_shift_diag: the two plans must differ only in pos_shift");
  if (!q || !k || !col_absdiff || !first_logit_absdiff || !result)
    return fail(AA_ERR_INVALID_ARG, "aa_shift_diag: q, k, col_absdiff, first_logit_absdiff and result are required");
  if (!aligned16(q) || !aligned16(k)) return fail(AA_ERR_INVALID_ARG, "aa_shift_diag: q and k must be 16-byte aligned");
  const size_t need = aa_shift_diag_workspace_bytes(p1);
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return fail(AA_ERR_INVALID_ARG, "aa_shift_diag: workspace missing, unaligned or smaller than "
                                    "aa_shift_diag_workspace_bytes()");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int T = p1->T, Hq = p1->Hq, Hkv = p1->Hkv, D = p1->D;
  DiagParams P;
  if (need) {
    uint8_t* w = static_cast<uint8_t*>(workspace);
    const size_t qb = align256((size_t)T * Hq * D * 2), kb = align256((size_t)T * Hkv * D * 2);
    auto* q1 = reinterpret_cast<__nv_bfloat16*>(w);
    auto* k1 = reinterpret_cast<__nv_bfloat16*>(w + qb);
    auto* q2 = reinterpret_cast<__nv_bfloat16*>(w + qb + kb);
    auto* k2 = reinterpret_cast<__nv_bfloat16*>(w + 2 * qb + kb);
    if ((st = launch_rope(p1, q, q1, Hq, 0, s)) != AA_OK || (st = launch_rope(p1, k, k1, Hkv, 0, s)) != AA_OK ||
        (st = launch_rope(p2, q, q2, Hq, 0, s)) != AA_OK || (st = launch_rope(p2, k, k2, Hkv, 0, s)) != AA_OK)
      return st;
    P.q[0] = q1; P.q[1] = q2; P.k[0] = k1; P.k[1] = k2;
  } else {
    P.q[0] = P.q[1] = static_cast<const __nv_bfloat16*>(q);
    P.k[0] = P.k[1] = static_cast<const __nv_bfloat16*>(k);
  }
  cudaError_t e = cudaMemsetAsync(col_absdiff, 0, (size_t)Hq * T * sizeof(float), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(first_logit_absdiff, 0, (size_t)Hq * T * sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e, "aa_shift_diag: clearing the outputs");
  P.row_lo = p1->dev.row_lo;
  P.col = col_absdiff;
  P.first = first_logit_absdiff;
  P.T = T; P.Hq = Hq; P.Hkv = Hkv; P.group = p1->group; P.anchor = p1->anchor ? 1 : 0;
  P.scale = p1->scale;
  const dim3 grid((unsigned)((T + kRows - 1) / kRows), (unsigned)Hq);
  if (D == 128)
    shift_diag_kernel<128><<<grid, kThreads, sizeof(DiagSmem<128>), s>>>(P);
  else
    shift_diag_kernel<64><<<grid, kThreads, sizeof(DiagSmem<64>), s>>>(P);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "shift_diag_kernel launch");
  shift_diag_reduce_kernel<<<1, kThreads, 0, s>>>(col_absdiff, first_logit_absdiff, p1->dev.key_hi, T, Hq,
                                                  p1->anchor ? 1 : 0, result);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "shift_diag_reduce_kernel launch");
  return AA_OK;
}
