// mcs_group_noalloc: query grouping for callers that cannot allocate device
// memory.  Its scratch is a fixed array compiled into the library instead of
// a caller-provided workspace; see the declaration in include/mcs.h.
#include "internal.h"
#include "mcs.h"

namespace {

// Size of the built-in scratch.  Every GPU on which the library's grouping
// module is loaded keeps this much device memory until the process exits.
constexpr size_t kNoallocScratchBytes = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// In host code `g_noalloc_scratch` only names a host-side shadow of the
// array; kernels must be given its device address.  The address is looked up
// on every call, with the caller's device current: a cached address would go
// stale if the device's context were destroyed and created again (after
// cudaDeviceReset the module is loaded anew and the array may move).  The
// first lookup on a device loads the library's kernels there.
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" mcs_status mcs_group_noalloc(const mcs_params* p, const void* q, int32_t* perm,
                                        cudaStream_t stream) {
  const mcs_status st = mcs::check_params(p, false);
  if (st != MCS_OK) return st;
  if (q == nullptr || perm == nullptr) return MCS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15u) != 0) return MCS_ERR_INVALID_ARG;
  const int BH = p->B * p->H, N = p->N, D = p->D, C = p->C;
  const int G = (N + C - 1) / C;
  const int iters = p->pddp_iters > 0 ? p->pddp_iters : 32;

  // Heads are grouped a batch at a time through the fixed scratch.
  const size_t one = mcs::pddp_workspace_bytes(1, N, D, C);
  if (one > kNoallocScratchBytes) return MCS_ERR_WORKSPACE;  // too large for the built-in scratch
  int batch = static_cast<int>(kNoallocScratchBytes / one);
  if (batch > BH) batch = BH;
  while (batch > 1 && mcs::pddp_workspace_bytes(batch, N, D, C) > kNoallocScratchBytes) --batch;

  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return mcs::record_cuda_error(e, "cudaGetSymbolAddress(noalloc scratch)");
  unsigned* status = nullptr;
  if ((e = mcs::device_status_word(&status)) != cudaSuccess)
    return mcs::record_cuda_error(e, "status word");

  // The kernels address q's rows by global head (either layout).
  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(q);
  for (int h0 = 0; h0 < BH; h0 += batch) {
    const int hc = BH - h0 < batch ? BH - h0 : batch;
    e = mcs::launch_pddp(qb, p->layout, p->H, h0, hc, N, D, C, iters,
                         perm + static_cast<size_t>(h0) * G * C, scratch, kNoallocScratchBytes,
                         status, stream);
    if (e != cudaSuccess) return mcs::record_cuda_error(e, "noalloc grouping launch");
  }
  return MCS_OK;
}
