// aa_bwd_static_workspace: the backward pass for callers that cannot allocate
// device memory. The scratch that aa_bwd normally takes from the caller lives
// here, in one fixed-size array in the library's own device memory.
#include <cstdio>
#include <mutex>

#include "aa_internal.h"

namespace aa {
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(64) << 20;  // 64 MiB per device

// Reserved on every GPU that loads this module and kept until the process
// exits. Host code must not use the name as an address: the device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on `device`, looked up once per device and
// kept for the life of the process (a reset of the device's primary context
// would invalidate it; the header tells callers not to reset). The caller has
// made `device` current.
aa_status static_workspace_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return fail(AA_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[device]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_workspace);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static workspace");
    g_addr[device] = ptr;
  }
  *out = g_addr[device];
  return AA_OK;
}

}  // namespace
}  // namespace aa

using namespace aa;

extern "C" aa_status aa_bwd_static_workspace(aa_plan_t p, const void* q, const void* k, const void* v,
                                             const void* o, const float* lse, const void* dout, void* dq,
                                             void* dk, void* dv, aa_stream_t stream) {
  aa_status st = check_compute_plan(p);
  if (st != AA_OK) return st;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
  for (const void* x : ptrs) {
    if (!x) return fail(AA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(x)) return fail(AA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  }
  const size_t need = aa_bwd_workspace_bytes(p);
  if (need > kStaticWorkspaceBytes) {
    char buf[200];
    std::snprintf(buf, sizeof buf,
                  "this plan needs %zu bytes of backward scratch; the static workspace holds %zu bytes "
                  "(%zu MiB): use aa_bwd with a caller-provided workspace",
                  need, kStaticWorkspaceBytes, kStaticWorkspaceBytes >> 20);
    return fail(AA_ERR_INVALID_ARG, buf);
  }
  int current = -1;
  cudaError_t e = cudaGetDevice(&current);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (current != p->device) return fail(AA_ERR_INVALID_ARG, "the plan's device must be the current device");
  void* ws = nullptr;
  if ((st = static_workspace_address(current, &ws)) != AA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->segmented) return seg_bwd(p, q, k, v, o, lse, dout, dq, dk, dv, ws, s);
  return launch_bwd_with_workspace(p, q, k, v, o, lse, dout, dq, dk, dv, ws, s);
}
