// Segment plans: documents given per token ("When Precision Meets Position",
// architecture page, §3.4 "AnchorAttention with Interleaved Chunks": documents
// split into chunks that are shuffled and recombined with the order inside each
// document kept; §3.4 "Mask construction" for what each token may see).
//
// A token sees the anchor and the earlier tokens of its own document, wherever
// they sit in the packing. The planner groups the tokens by document (stable:
// the order inside a document is kept), which turns the problem into an
// ordinary contiguous packing with the same visible pairs and the same
// positions; aa_fwd / aa_bwd gather their inputs into that order, run the
// usual kernels, and scatter the outputs back. The gathers and scatters are
// HBM-bound copies of whole token rows.
#include "kcommon.cuh"

namespace aa {
namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Row permutation of a [T, row] tensor in 16-byte vectors: gather
// (dst[t] = src[perm[t]]) or scatter (dst[perm[t]] = src[t]).
__global__ void __launch_bounds__(256) permute_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           const int32_t* __restrict__ perm, int T, int row_vecs,
                                                           int scatter) {
  const int64_t n = (int64_t)T * row_vecs;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(e / row_vecs), c = (int)(e - (int64_t)t * row_vecs);
    const int64_t o = (int64_t)__ldg(perm + t) * row_vecs + c;
    if (scatter)
      dst[o] = src[e];
    else
      dst[e] = src[o];
  }
}

// Column permutation of a [H, T] fp32 array (the LSE rows).
__global__ void __launch_bounds__(256) permute_cols_kernel(const float* __restrict__ src, float* __restrict__ dst,
                                                           const int32_t* __restrict__ perm, int T, int H,
                                                           int scatter) {
  const int64_t n = (int64_t)T * H;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int h = (int)(e / T), t = (int)(e - (int64_t)h * T);
    const int64_t o = (int64_t)h * T + __ldg(perm + t);
    if (scatter)
      dst[o] = src[e];
    else
      dst[e] = src[o];
  }
}

aa_status permute_rows(const aa_plan_s* p, const void* src, void* dst, int H, int scatter, cudaStream_t s) {
  const int row_vecs = H * p->D * 2 / 16;
  const int64_t n = (int64_t)p->T * row_vecs;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)p->num_sms * 8);
  permute_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                       p->dev.perm, p->T, row_vecs, scatter);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "permute_rows_kernel launch");
}

aa_status permute_cols(const aa_plan_s* p, const float* src, float* dst, int scatter, cudaStream_t s) {
  const int64_t n = (int64_t)p->T * p->Hq;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)p->num_sms * 8);
  permute_cols_kernel<<<(unsigned)blocks, 256, 0, s>>>(src, dst, p->dev.perm, p->T, p->Hq, scatter);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "permute_cols_kernel launch");
}

size_t tensor_bytes(const aa_plan_s* p, int H) { return align256((size_t)p->T * H * p->D * 2); }
size_t lse_bytes(const aa_plan_s* p) { return align256((size_t)p->Hq * p->T * 4); }

}  // namespace

// Forward extras: grouped Q, K, V, O and LSE.
size_t seg_fwd_extra_bytes(const aa_plan_s* p) {
  return 2 * tensor_bytes(p, p->Hq) + 2 * tensor_bytes(p, p->Hkv) + lse_bytes(p);
}

// Backward extras: grouped Q, K (unless the rotated ones are given), V, O,
// dO, LSE and dQ, dK, dV.
size_t seg_bwd_extra_bytes(const aa_plan_s* p, bool with_qk) {
  const int n = with_qk ? 4 : 3;
  return n * tensor_bytes(p, p->Hq) + n * tensor_bytes(p, p->Hkv) + lse_bytes(p);
}

aa_status seg_fwd(aa_plan_s* p, const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                  cudaStream_t s) {
  uint8_t* w = static_cast<uint8_t*>(workspace) + fwd_base_workspace_bytes(p);
  const size_t tq = tensor_bytes(p, p->Hq), tk = tensor_bytes(p, p->Hkv);
  void* qg = w;
  void* kg = w + tq;
  void* vg = w + tq + tk;
  void* og = w + tq + 2 * tk;
  float* lg = reinterpret_cast<float*>(w + 2 * tq + 2 * tk);
  aa_status st;
  if ((st = permute_rows(p, q, qg, p->Hq, 0, s)) != AA_OK || (st = permute_rows(p, k, kg, p->Hkv, 0, s)) != AA_OK ||
      (st = permute_rows(p, v, vg, p->Hkv, 0, s)) != AA_OK)
    return st;
  if ((st = launch_fwd_with_workspace(p, qg, kg, vg, og, lg, workspace, s)) != AA_OK) return st;
  if ((st = permute_rows(p, og, o, p->Hq, 1, s)) != AA_OK) return st;
  return permute_cols(p, lg, lse, 1, s);
}

aa_status seg_bwd(aa_plan_s* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, void* workspace, cudaStream_t s, const void* qr,
                  const void* kr) {
  // qr / kr: the forward's rotated Q and K, already in the grouped order
  const bool given = qr != nullptr;
  uint8_t* w = static_cast<uint8_t*>(workspace) + bwd_base_workspace_bytes(p, !given);
  const size_t tq = tensor_bytes(p, p->Hq), tk = tensor_bytes(p, p->Hkv);
  void* og = w;
  void* dog = w + tq;
  void* dqg = w + 2 * tq;
  void* vg = w + 3 * tq;
  void* dkg = w + 3 * tq + tk;
  void* dvg = w + 3 * tq + 2 * tk;
  float* lg = reinterpret_cast<float*>(w + 3 * tq + 3 * tk);
  void* qg = w + 3 * tq + 3 * tk + lse_bytes(p);  // only without qr / kr
  void* kg = static_cast<uint8_t*>(qg) + tq;
  aa_status st;
  if (!given &&
      ((st = permute_rows(p, q, qg, p->Hq, 0, s)) != AA_OK || (st = permute_rows(p, k, kg, p->Hkv, 0, s)) != AA_OK))
    return st;
  if ((st = permute_rows(p, v, vg, p->Hkv, 0, s)) != AA_OK || (st = permute_rows(p, o, og, p->Hq, 0, s)) != AA_OK ||
      (st = permute_rows(p, dout, dog, p->Hq, 0, s)) != AA_OK || (st = permute_cols(p, lse, lg, 0, s)) != AA_OK)
    return st;
  st = given ? launch_bwd_with_workspace(p, nullptr, nullptr, vg, og, lg, dog, dqg, dkg, dvg, workspace, s, qr, kr)
             : launch_bwd_with_workspace(p, qg, kg, vg, og, lg, dog, dqg, dkg, dvg, workspace, s);
  if (st != AA_OK) return st;
  if ((st = permute_rows(p, dqg, dq, p->Hq, 1, s)) != AA_OK || (st = permute_rows(p, dkg, dk, p->Hkv, 1, s)) != AA_OK)
    return st;
  return permute_rows(p, dvg, dv, p->Hkv, 1, s);
}

}  // namespace aa
