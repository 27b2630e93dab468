// Segment plans: documents given per token ("When Precision Meets Position",
// architecture page, §3.4 "AnchorAttention with Interleaved Chunks": documents
// split into chunks that are shuffled and recombined with the order inside each
// document kept; §3.4 "Mask construction" for what each token may see).
//
// A token sees the anchor and the earlier tokens of its own document, wherever
// they sit in the packing. The planner groups the tokens by document (stable:
// the order inside a document is kept), which turns the problem into an
// ordinary contiguous packing with the same visible pairs and the same
// positions. The kernels run on that grouped order and meet the caller's
// order only at their edges: the rotation passes read q and k through the
// permutation, the backward's preprocess kernel reads o, dout and lse through
// it (and leaves a grouped dout for the tile kernel), and every output row
// (O, LSE, dq, dk, dv) is written at its caller position by the kernel that
// produces it. Only V is gathered, once per forward (the training step's
// backward reads the forward's copy).
#include "kcommon.cuh"

namespace aa {
namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Row gather of a [T, row] tensor in 16-byte vectors: dst[t] = src[perm[t]].
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                          const int32_t* __restrict__ perm, int T, int row_vecs) {
  const int64_t n = (int64_t)T * row_vecs;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(e / row_vecs), c = (int)(e - (int64_t)t * row_vecs);
    dst[e] = src[(int64_t)__ldg(perm + t) * row_vecs + c];
  }
}

aa_status gather_rows(const aa_plan_s* p, const void* src, void* dst, int H, cudaStream_t s) {
  const int row_vecs = H * p->D * 2 / 16;
  const int64_t n = (int64_t)p->T * row_vecs;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)p->num_sms * 8);
  gather_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                      p->dev.perm, p->T, row_vecs);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "gather_rows_kernel launch");
}

size_t tensor_bytes(const aa_plan_s* p, int H) { return align256((size_t)p->T * H * p->D * 2); }

}  // namespace

// Forward extras: the grouped V, which stays there for aa_bwd_from_fwd (and,
// without RoPE, grouped Q and K: no rotation pass reads them through the
// permutation then).
size_t seg_fwd_extra_bytes(const aa_plan_s* p) {
  const bool rope = p->cfg.rope_layout != AA_ROPE_NONE;
  return tensor_bytes(p, p->Hkv) + (rope ? 0 : tensor_bytes(p, p->Hq) + tensor_bytes(p, p->Hkv));
}

const void* fwd_grouped_v(const aa_plan_s* p, const void* fwd_workspace) {
  return static_cast<const uint8_t*>(fwd_workspace) + fwd_base_workspace_bytes(p);
}

// Backward extras: the grouped dO (written by the preprocess kernel) and,
// unless the forward's grouped V is given (aa_bwd_from_fwd), the grouped V;
// without RoPE also grouped Q and K.
size_t seg_bwd_extra_bytes(const aa_plan_s* p, bool with_qk) {
  const bool rope = p->cfg.rope_layout != AA_ROPE_NONE;
  size_t n = tensor_bytes(p, p->Hq);
  if (with_qk) n += tensor_bytes(p, p->Hkv);
  if (with_qk && !rope) n += tensor_bytes(p, p->Hq) + tensor_bytes(p, p->Hkv);
  return n;
}

// The kernels run on the grouped token order. Q and K are read through the
// permutation by the rotation passes (or gathered, without RoPE), V is
// gathered once per forward, and every output (O, LSE, dq, dk, dv) is written
// straight to the caller's rows by the kernel that produces it.
aa_status seg_fwd(aa_plan_s* p, const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                  cudaStream_t s) {
  uint8_t* w = static_cast<uint8_t*>(workspace) + fwd_base_workspace_bytes(p);
  const size_t tq = tensor_bytes(p, p->Hq), tk = tensor_bytes(p, p->Hkv);
  void* vg = w;
  aa_status st;
  if ((st = gather_rows(p, v, vg, p->Hkv, s)) != AA_OK) return st;
  if (p->cfg.rope_layout == AA_ROPE_NONE) {
    void* qg = w + tk;
    void* kg = w + tk + tq;
    if ((st = gather_rows(p, q, qg, p->Hq, s)) != AA_OK || (st = gather_rows(p, k, kg, p->Hkv, s)) != AA_OK)
      return st;
    q = qg;
    k = kg;
  }
  return launch_fwd_with_workspace(p, q, k, vg, o, lse, workspace, s, p->dev.perm);
}

aa_status seg_bwd(aa_plan_s* p, const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, void* workspace, cudaStream_t s, const void* qr,
                  const void* kr, const void* vg_in) {
  // qr / kr / vg_in: the forward's rotated Q, K and grouped V, already in the
  // grouped order
  const bool given = qr != nullptr;
  uint8_t* w = static_cast<uint8_t*>(workspace) + bwd_base_workspace_bytes(p, !given);
  const size_t tq = tensor_bytes(p, p->Hq), tk = tensor_bytes(p, p->Hkv);
  void* dog = w;
  aa_status st;
  const void* vg = vg_in;
  if (!given) {
    void* vgw = w + tq;
    if ((st = gather_rows(p, v, vgw, p->Hkv, s)) != AA_OK) return st;
    vg = vgw;
    if (p->cfg.rope_layout == AA_ROPE_NONE) {
      void* qg = w + tq + tk;
      void* kg = w + 2 * tq + tk;
      if ((st = gather_rows(p, q, qg, p->Hq, s)) != AA_OK || (st = gather_rows(p, k, kg, p->Hkv, s)) != AA_OK)
        return st;
      q = qg;
      k = kg;
    }
  }
  return launch_bwd_with_workspace(p, q, k, vg, o, lse, dout, dq, dk, dv, workspace, s, qr, kr, p->dev.perm, dog);
}

}  // namespace aa
