// Standalone RoPE (Eq. 6 of "When Precision Meets Position", architecture
// page §3.4 "Rotary Positional Embedding (RoPE): The Theoretical Promise";
// fp32 rotation then a cast to bf16 as in §3.2 "Big-Picture Architecture")
// and the host-side TMA descriptor helper.
//
// HBM-bound: one read and one write of x, one CTA per (128-row tile, head).
// The attention entry points run the same kernel once per call on Q and K,
// so aa_rope_apply and the operands the attention kernels read agree bit for
// bit.
#include <cudaTypedefs.h>

#include <mutex>

#include "kcommon.cuh"

namespace aa {

// Accessor over one head of a [T, H, D] bf16 tensor in global memory, rows
// relative to a 128-row tile; reads from x, writes to y (which may equal x).
template <int HD, int L, bool kRows>
struct GlobalTile {
  using Raw = QuadRaw;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  int row0, H, head;
  const int32_t* src_rows;  // x row of each y row (kRows only)
  __device__ __forceinline__ size_t off(int r, int e) const { return ((size_t)(row0 + r) * H + head) * HD + e; }
  __device__ __forceinline__ size_t src_off(int r, int e) const {
    const int row = kRows ? __ldg(src_rows + row0 + r) : row0 + r;
    return ((size_t)row * H + head) * HD + e;
  }
  __device__ __forceinline__ QuadRaw load_raw(int r, int qd) const {
    QuadRaw q;
    if (L == 0) {
      q.w = *reinterpret_cast<const uint4*>(x + src_off(r, 8 * qd));
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(x + src_off(r, 4 * qd));
      const uint2 b = *reinterpret_cast<const uint2*>(x + src_off(r, HD / 2 + 4 * qd));
      q.w = make_uint4(a.x, a.y, b.x, b.y);
    }
    return q;
  }
  __device__ __forceinline__ void store_raw(int r, int qd, const QuadRaw& q) const {
    if (L == 0) {
      *reinterpret_cast<uint4*>(y + off(r, 8 * qd)) = q.w;
    } else {
      *reinterpret_cast<uint2*>(y + off(r, 4 * qd)) = make_uint2(q.w.x, q.w.y);
      *reinterpret_cast<uint2*>(y + off(r, HD / 2 + 4 * qd)) = make_uint2(q.w.z, q.w.w);
    }
  }
  __device__ __forceinline__ static void unpack(const QuadRaw& q, float* a, float* b) { quad_unpack(L, q, a, b); }
  __device__ __forceinline__ static QuadRaw pack(const float* a, const float* b) { return quad_pack(L, a, b); }
};

// One CTA of 128 threads per (128-row tile, head): the canonical tile
// rotation of kcommon.cuh, straight from and to global memory.
template <int HD, int L, bool kRows>
__global__ void __launch_bounds__(128) rope_apply_kernel(const __nv_bfloat16* __restrict__ x,
                                                         __nv_bfloat16* y, const int32_t* __restrict__ pos_id,
                                                         const float2* __restrict__ hi_tab,
                                                         const float2* __restrict__ lo_tab,
                                                         const float2* __restrict__ step_tab, int T, int H,
                                                         int inverse, const int32_t* __restrict__ src_rows) {
  GlobalTile<HD, L, kRows> tile{x, y, (int)blockIdx.x * kTile, H, (int)blockIdx.y, src_rows};
  RopeUnits<HD, 128> st;
  st.begin(tile.row0, T, pos_id, inverse != 0, hi_tab, lo_tab, threadIdx.x);
  st.run(tile, inverse != 0, hi_tab, lo_tab, step_tab, threadIdx.x);
}

template <int HD>
void launch_rope_apply(const aa_plan_s* p, const void* x, void* y, int H, int inverse, cudaStream_t s,
                       const int32_t* pos, const int32_t* src_rows) {
  const dim3 grid((unsigned)p->n_tiles, (unsigned)H);
  const auto* xi = static_cast<const __nv_bfloat16*>(x);
  auto* yo = static_cast<__nv_bfloat16*>(y);
  const bool adj = p->cfg.rope_layout == AA_ROPE_ADJACENT;
  auto k = adj ? (src_rows ? rope_apply_kernel<HD, 0, true> : rope_apply_kernel<HD, 0, false>)
               : (src_rows ? rope_apply_kernel<HD, 1, true> : rope_apply_kernel<HD, 1, false>);
  k<<<grid, 128, 0, s>>>(xi, yo, pos, p->dev.rope_hi, p->dev.rope_lo, p->dev.rope_step, p->T, H, inverse, src_rows);
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

aa_status launch_rope(const aa_plan_s* p, const void* x, void* y, int H, int inverse, cudaStream_t s,
                      const int32_t* pos, const int32_t* src_rows) {
  if (!pos) pos = p->dev.pos_id;
  if (p->D == 128)
    launch_rope_apply<128>(p, x, y, H, inverse, s, pos, src_rows);
  else
    launch_rope_apply<64>(p, x, y, H, inverse, s, pos, src_rows);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "rope_apply_kernel launch");
}

aa_status make_f32_map(CUtensorMap* m, const void* base, int T, int H, int D, int box_c, int box_t) {
  auto enc = get_encode_fn();
  if (!enc) return fail(AA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
  cuuint32_t box[3] = {(cuuint32_t)box_c, 1, (cuuint32_t)box_t};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(AA_ERR_CUDA, "cuTensorMapEncodeTiled (fp32) failed");
  return AA_OK;
}

// One warp waits on a barrier that expects one arrival and never gets it.
__global__ void bounded_wait_selftest_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) ptx::mbar_wait(&bar, 0, limit_ns, err, 900);
}

}  // namespace aa

using namespace aa;

extern "C" aa_status aa_selftest_bounded_wait(aa_plan_t p, aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  bounded_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p->dev.err, p->wait_limit_ns);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? AA_OK : cuda_fail(e, "bounded_wait_selftest_kernel launch");
}

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
  // a segment plan's tensors arrive in the caller's token order
  return launch_rope(p, x, y, num_heads, inverse ? 1 : 0, s, p->segmented ? p->dev.pos_orig : p->dev.pos_id);
}
