// Standalone RoPE (Eq. 6 of "When Precision Meets Position", architecture
// page §3.4 "Rotary Positional Embedding (RoPE): The Theoretical Promise";
// fp32 rotation then a cast to bf16 as in §3.2 "Big-Picture Architecture")
// and the host-side TMA descriptor helper.
//
// HBM-bound: one read and one write of x. Each thread rotates four pairs
// (16 bytes of bf16 for the adjacent layout), grid-strided over the whole
// tensor with a grid sized to the SM count.
#include <cudaTypedefs.h>

#include <mutex>

#include "kcommon.cuh"

namespace aa {

__global__ void __launch_bounds__(256) rope_apply_kernel(const __nv_bfloat16* __restrict__ x,
                                                         __nv_bfloat16* __restrict__ y,
                                                         const int32_t* __restrict__ pos_id,
                                                         const float2* __restrict__ hi_tab,
                                                         const float2* __restrict__ lo_tab, int64_t T, int H,
                                                         int D, int layout, int inverse) {
  const int half = D / 2;
  const int quads = half / 4;  // groups of 4 pairs per (token, head)
  const int64_t n = T * H * quads;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int qd = (int)(idx % quads);
    const int64_t row = idx / quads;  // token * H + head
    const int t = (int)(row / H);
    const int pos = __ldg(pos_id + t);
    const __nv_bfloat16* xr = x + row * D;
    __nv_bfloat16* yr = y + row * D;
    if (layout == 0) {
      uint4 w = *reinterpret_cast<const uint4*>(xr + qd * 8);
      uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 cs = rope_cs(hi_tab, lo_tab, pos, qd * 4 + e, half);
        if (inverse) cs.y = -cs.y;
        float2 v = ptx::unpack_bf16x2(u[e]);
        rope_pair(v.x, v.y, cs.x, cs.y);
        u[e] = ptx::pack_bf16x2(v.x, v.y);
      }
      *reinterpret_cast<uint4*>(yr + qd * 8) = w;
    } else {
      uint2 wa = *reinterpret_cast<const uint2*>(xr + qd * 4);
      uint2 wb = *reinterpret_cast<const uint2*>(xr + half + qd * 4);
      __nv_bfloat16* a = reinterpret_cast<__nv_bfloat16*>(&wa);
      __nv_bfloat16* b = reinterpret_cast<__nv_bfloat16*>(&wb);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 cs = rope_cs(hi_tab, lo_tab, pos, qd * 4 + e, half);
        if (inverse) cs.y = -cs.y;
        float u = __bfloat162float(a[e]), v = __bfloat162float(b[e]);
        rope_pair(u, v, cs.x, cs.y);
        a[e] = __float2bfloat16_rn(u);
        b[e] = __float2bfloat16_rn(v);
      }
      *reinterpret_cast<uint2*>(yr + qd * 4) = wa;
      *reinterpret_cast<uint2*>(yr + half + qd * 4) = wb;
    }
  }
}

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

aa_status make_tile_map(CUtensorMap* m, const void* base, int T, int H, int D) {
  auto enc = get_encode_fn();
  if (!enc) return fail(AA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kTile};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(AA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  return AA_OK;
}

}  // namespace aa

using namespace aa;

extern "C" aa_status aa_rope_apply(aa_plan_t p, const void* x, void* y, int32_t num_heads, int32_t inverse,
                                   aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  if (!x || !y) return fail(AA_ERR_INVALID_ARG, "x and y must be device pointers");
  if (!aligned16(x) || !aligned16(y)) return fail(AA_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (num_heads < 1) return fail(AA_ERR_INVALID_ARG, "num_heads must be >= 1");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t T = p->T;
  const int D = p->D;
  if (p->cfg.rope_layout == AA_ROPE_NONE) {
    if (x == y) return AA_OK;
    cudaError_t e = cudaMemcpyAsync(y, x, (size_t)T * num_heads * D * 2, cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? AA_OK : cuda_fail(e, "aa_rope_apply copy");
  }
  const int64_t n = T * num_heads * (D / 8);
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  const int64_t cap = (int64_t)p->num_sms * 8;
  if (blocks > cap) blocks = cap;
  rope_apply_kernel<<<(unsigned)blocks, threads, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), p->dev.pos_id, p->dev.rope_hi,
      p->dev.rope_lo, T, num_heads, D, p->cfg.rope_layout, inverse ? 1 : 0);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "rope_apply_kernel launch");
}
