// C-ABI entry points of libmcs.so: argument checks, TMA tensor maps and
// dispatch to the kernels.  Declarations and per-call documentation live in
// include/mcs.h.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "internal.h"
#include "mcs.h"

namespace {

__device__ unsigned g_mcs_status = 0;

thread_local char t_last_error[256] = "no error";

mcs_status cuda_fail(cudaError_t e, const char* what) {
  snprintf(t_last_error, sizeof(t_last_error), "%s: %s", what, cudaGetErrorString(e));
  return MCS_ERR_CUDA;
}

// cuTensorMapEncodeTiled fetched through the runtime, so that the library
// needs no link-time dependency on libcuda.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// A q/k/v-shaped bf16 tensor viewed as 4-D (d, token, h, b) whatever its
// layout ([B,H,N,D] or [B,N,H,D]: only the strides differ), box
// {64, 128, 1, 1}: 128-token tiles of one head, tokens past N zero-filled.
bool make_tile_map(CUtensorMap* m, const void* base, const mcs_params* p) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  const cuuint64_t D = p->D, N = p->N, H = p->H, row = D * 2;
  cuuint64_t dims[4] = {D, N, H, (cuuint64_t)p->B};
  cuuint64_t strides[3];
  if (p->layout == MCS_LAYOUT_BNHD) {
    strides[0] = H * row;      // token
    strides[1] = row;          // head
  } else {
    strides[0] = row;
    strides[1] = N * row;
  }
  strides[2] = N * H * row;    // batch
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH*N][D] bf16 viewed as 2-D with a one-row box {64, 1}, for gather4.
bool make_gather_map(CUtensorMap* m, const void* base, int BH, int N, int D) {
  EncodeTiledFn f = encode_fn();
  if (!f) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)BH * (cuuint64_t)N};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t es[2] = {1, 1};
  return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mcs_status check_shape(const mcs_params* p, bool need_k) {
  if (p == nullptr) return MCS_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->N < 1) return MCS_ERR_INVALID_ARG;
  if ((long long)p->B * p->H > 65535) return MCS_ERR_INVALID_ARG;
  if ((long long)p->B * p->H * p->N > 0x7fffffffLL) return MCS_ERR_INVALID_ARG;
  if (p->D != 64 && p->D != 128) return MCS_ERR_UNSUPPORTED;
  if (p->C != 64 && p->C != 128) return MCS_ERR_UNSUPPORTED;
  if (need_k && (p->K < 1 || p->K > p->N)) return MCS_ERR_INVALID_ARG;
  if (p->scale < 0.f || !isfinite(p->scale)) return MCS_ERR_INVALID_ARG;
  if (p->pddp_iters < 0) return MCS_ERR_INVALID_ARG;
  if (p->layout != MCS_LAYOUT_BHND && p->layout != MCS_LAYOUT_BNHD) return MCS_ERR_INVALID_ARG;
  return MCS_OK;
}

float scale_of(const mcs_params* p) {
  return p->scale > 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->D));
}
int iters_of(const mcs_params* p) { return p->pddp_iters > 0 ? p->pddp_iters : 32; }
int groups_of(const mcs_params* p) { return (p->N + p->C - 1) / p->C; }

mcs_status status_ptr(unsigned** out) {
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_mcs_status);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
  return MCS_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

// Test-only fault injection for the attention kernels: with the environment
// variable MCS_TEST_FAULT=stall_load the producers stop after the first K/V
// tile, so the MMA thread's next bounded wait expires (MCS_ERR_TIMEOUT) and
// the kernel's teardown path runs.  Read at every call; unset in normal use.
int fault_from_env() {
  const char* f = getenv("MCS_TEST_FAULT");
  return (f != nullptr && strcmp(f, "stall_load") == 0) ? 1 : 0;
}

// Paired-mode requirements (pair lists, see PairLayout): C = 64, K small
// enough for the union kernel's shared memory, tokens below 2^28.
mcs_status check_pairs(const mcs_params* p) {
  mcs_status s = check_shape(p, true);
  if (s != MCS_OK) return s;
  if (p->C != 64 || p->K > mcs::kPairMaxK || p->N >= (1 << mcs::kPairTokenBits))
    return MCS_ERR_UNSUPPORTED;
  return MCS_OK;
}

mcs_status run_sparse(const mcs_params* p, const void* q, const void* k, const void* v,
                      const int32_t* perm, const int32_t* idx, const void* aux, void* out,
                      int mode, cudaStream_t stream, const void* pairs = nullptr) {
  mcs_status s = check_shape(p, true);
  if (s != MCS_OK) return s;
  if (pairs && (s = check_pairs(p)) != MCS_OK) return s;
  if (!q || !k || !v || !perm || (!idx && !pairs) || !out) return MCS_ERR_INVALID_ARG;
  if (pairs && (reinterpret_cast<uintptr_t>(pairs) & 255u) != 0) return MCS_ERR_INVALID_ARG;
  if (mode != mcs::kSparse && !aux) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (aux && !aligned16(aux)))
    return MCS_ERR_INVALID_ARG;
  const int BH = p->B * p->H;
  CUtensorMap tq, tk, tv;
  if (!make_gather_map(&tq, q, BH, p->N, p->D) || !make_gather_map(&tk, k, BH, p->N, p->D) ||
      !make_gather_map(&tv, v, BH, p->N, p->D))
    return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(gather)");
  mcs::AttnArgs a{};
  a.H = p->H;
  a.layout = p->layout;
  a.N = p->N;
  a.C = p->C;
  a.G = groups_of(p);
  a.K = p->K;
  a.scale_log2 = scale_of(p) * kLog2e;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = nullptr;
  a.perm = perm;
  a.idx = idx;
  a.aux_in = static_cast<const __nv_bfloat16*>(aux);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.fault = fault_from_env();
  if (pairs) {
    const mcs::PairLayout l = mcs::pair_layout(BH, a.G, p->K);
    a.P = l.P;
    a.cap = l.cap;
    a.plen = static_cast<const int32_t*>(pairs);
    a.pidx = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(pairs) + l.entries_off);
    mode |= mcs::kPaired;
  }
  if ((s = status_ptr(&a.status)) != MCS_OK) return s;
  cudaError_t e = mcs::launch_attention(p->D, mode, &tq, &tk, &tv, a, BH, stream);
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention launch");
  return MCS_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t mass_head_bytes(const mcs_params* p) {
  return static_cast<size_t>(groups_of(p)) * static_cast<size_t>(p->N) * sizeof(float);
}

// Workspace per head of the anchor step's selection: the group masses and
// their digit histograms (kMassHistBins words per group).
size_t hist_head_bytes(const mcs_params* p) {
  return static_cast<size_t>(groups_of(p)) * mcs::kMassHistBins * sizeof(uint32_t);
}
size_t select_head_bytes(const mcs_params* p) {
  return round_up(mass_head_bytes(p), 256) + round_up(hist_head_bytes(p), 256);
}

// a3 for heads [h0, h0 + hc), with (hist != null) or without the histograms.
mcs_status run_group_mass(const mcs_params* p, const void* q, const void* k, const float* lse,
                          const int32_t* perm, int h0, int hc, float* mass, uint32_t* hist,
                          cudaStream_t stream) {
  const int BH = p->B * p->H;
  CUtensorMap tq, tk;
  if (!make_gather_map(&tq, q, BH, p->N, p->D) || !make_tile_map(&tk, k, p))
    return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(mass)");
  mcs::MassArgs a{};
  a.H = p->H;
  a.layout = p->layout;
  a.N = p->N;
  a.C = p->C;
  a.G = groups_of(p);
  a.head0 = h0;
  a.scale_log2 = scale_of(p) * kLog2e;
  a.perm = perm;
  a.lse = lse;
  a.mass = mass;
  a.hist = hist;
  mcs_status s;
  if ((s = status_ptr(&a.status)) != MCS_OK) return s;
  cudaError_t e = mcs::launch_group_mass(p->D, &tq, &tk, a, hc, stream);
  if (e != cudaSuccess) return cuda_fail(e, "group mass launch");
  return MCS_OK;
}

mcs_status run_topk(const mcs_params* p, const float* mass, const uint32_t* hist, int rows,
                    int32_t* idx, float* retained, cudaStream_t stream) {
  unsigned* st;
  mcs_status s;
  if ((s = status_ptr(&st)) != MCS_OK) return s;
  cudaError_t e = mcs::launch_topk(mass, hist, rows, p->N, p->K, idx, retained, st, stream);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return MCS_OK;
}

}  // namespace

namespace mcs {

mcs_status record_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }
mcs_status check_params(const mcs_params* p, bool need_k) { return check_shape(p, need_k); }

cudaError_t device_status_word(unsigned** out) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_mcs_status);
}
}  // namespace mcs

extern "C" {

const char* mcs_status_string(mcs_status s) {
  switch (s) {
    case MCS_OK: return "MCS_OK";
    case MCS_ERR_INVALID_ARG: return "MCS_ERR_INVALID_ARG";
    case MCS_ERR_UNSUPPORTED: return "MCS_ERR_UNSUPPORTED";
    case MCS_ERR_WORKSPACE: return "MCS_ERR_WORKSPACE";
    case MCS_ERR_CUDA: return "MCS_ERR_CUDA";
    case MCS_ERR_TIMEOUT: return "MCS_ERR_TIMEOUT";
    case MCS_ERR_BOUNDS: return "MCS_ERR_BOUNDS";
  }
  return "MCS_ERR_UNKNOWN";
}

const char* mcs_last_cuda_error(void) { return t_last_error; }

mcs_status mcs_device_status(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_mcs_status, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol(status)");
  if (v != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_mcs_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol(status)");
  }
  if (v & mcs::DEV_TIMEOUT) return MCS_ERR_TIMEOUT;
  if (v & mcs::DEV_BOUNDS) return MCS_ERR_BOUNDS;
  return MCS_OK;
}

size_t mcs_group_workspace(const mcs_params* p) {
  if (check_shape(p, false) != MCS_OK) return 0;
  return mcs::pddp_workspace_bytes(p->B * p->H, p->N, p->D, p->C);
}

size_t mcs_anchor_workspace(const mcs_params* p) {
  if (check_shape(p, false) != MCS_OK) return 0;
  const size_t per_head = select_head_bytes(p);
  const size_t BH = static_cast<size_t>(p->B) * p->H;
  size_t heads = std::max<size_t>(1, (size_t(1) << 32) / per_head);
  heads = std::min(heads, BH);
  return std::max(per_head * heads, mcs_group_workspace(p));
}

mcs_status mcs_group(const mcs_params* p, const void* q, int32_t* perm, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
  mcs_status s = check_shape(p, false);
  if (s != MCS_OK) return s;
  if (!q || !perm || !aligned16(q)) return MCS_ERR_INVALID_ARG;
  const size_t need = mcs_group_workspace(p);
  if (ws_bytes < need || (need > 0 && ws == nullptr) || !aligned16(ws)) return MCS_ERR_WORKSPACE;
  const int BH = p->B * p->H;
  unsigned* st;
  if ((s = status_ptr(&st)) != MCS_OK) return s;
  cudaError_t e = mcs::launch_pddp(static_cast<const __nv_bfloat16*>(q), p->layout, p->H, 0, BH,
                                   p->N, p->D, p->C, iters_of(p), perm, ws, ws_bytes, st, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pddp launch");
  return MCS_OK;
}

mcs_status mcs_dense_attn(const mcs_params* p, const void* q, const void* k, const void* v,
                          void* out, float* lse, cudaStream_t stream) {
  mcs_status s = check_shape(p, false);
  if (s != MCS_OK) return s;
  if (!q || !k || !v || !out) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return MCS_ERR_INVALID_ARG;
  const int BH = p->B * p->H;
  CUtensorMap tq, tk, tv;
  if (!make_tile_map(&tq, q, p) || !make_tile_map(&tk, k, p) || !make_tile_map(&tv, v, p))
    return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(tile)");
  mcs::AttnArgs a{};
  a.H = p->H;
  a.layout = p->layout;
  a.N = p->N;
  a.C = p->C;
  a.G = groups_of(p);
  a.K = p->N;
  a.scale_log2 = scale_of(p) * kLog2e;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse = lse;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.fault = fault_from_env();
  if ((s = status_ptr(&a.status)) != MCS_OK) return s;
  cudaError_t e = mcs::launch_attention(p->D, mcs::kDense, &tq, &tk, &tv, a, BH, stream);
  if (e != cudaSuccess) return cuda_fail(e, "dense attention launch");
  return MCS_OK;
}

mcs_status mcs_group_mass(const mcs_params* p, const void* q, const void* k, const float* lse,
                          const int32_t* perm, int head_begin, int head_count, float* mass,
                          cudaStream_t stream) {
  mcs_status s = check_shape(p, false);
  if (s != MCS_OK) return s;
  if (!q || !k || !lse || !perm || !mass) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k)) return MCS_ERR_INVALID_ARG;
  const int BH = p->B * p->H;
  if (head_begin < 0 || head_count < 1 || head_begin + head_count > BH) return MCS_ERR_INVALID_ARG;
  return run_group_mass(p, q, k, lse, perm, head_begin, head_count, mass, nullptr, stream);
}

mcs_status mcs_topk(const mcs_params* p, const float* mass, int rows, int32_t* idx,
                    float* retained, cudaStream_t stream) {
  if (p == nullptr || p->N < 1 || p->K < 1 || p->K > p->N) return MCS_ERR_INVALID_ARG;
  if (rows < 0 || (rows > 0 && (!mass || !idx))) return MCS_ERR_INVALID_ARG;
  return run_topk(p, mass, nullptr, rows, idx, retained, stream);
}

mcs_status mcs_sparse_attn(const mcs_params* p, const void* q, const void* k, const void* v,
                           const int32_t* perm, const int32_t* idx, const void* residual,
                           void* out, cudaStream_t stream) {
  return run_sparse(p, q, k, v, perm, idx, residual, out,
                    residual ? mcs::kSparseAdd : mcs::kSparse, stream);
}

mcs_status mcs_sparse_attn_record(const mcs_params* p, const void* q, const void* k,
                                  const void* v, const int32_t* perm, const int32_t* idx,
                                  const void* dense_out, void* residual, cudaStream_t stream) {
  return run_sparse(p, q, k, v, perm, idx, dense_out, residual, mcs::kSparseRecord, stream);
}

mcs_status mcs_quantize_e4m3(const void* x, size_t n, float scale, void* x8,
                             cudaStream_t stream) {
  if (n > 0 && (!x || !x8 || !aligned16(x) || !aligned16(x8))) return MCS_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return MCS_ERR_INVALID_ARG;
  cudaError_t e = mcs::launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(x), n, scale,
                                            static_cast<uint8_t*>(x8), stream);
  if (e != cudaSuccess) return cuda_fail(e, "e4m3 quantize launch");
  return MCS_OK;
}

mcs_status mcs_sparse_attn_e4m3(const mcs_params* p, const void* q, const void* k8,
                                const void* v8, float k_scale, float v_scale,
                                const int32_t* perm, const int32_t* idx, const void* residual,
                                void* out, cudaStream_t stream) {
  mcs_status s = check_shape(p, true);
  if (s != MCS_OK) return s;
  if (!q || !k8 || !v8 || !perm || !idx || !out) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k8) || !aligned16(v8) || !aligned16(out) ||
      (residual && !aligned16(residual)))
    return MCS_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !isfinite(k_scale) || !(v_scale > 0.f) || !isfinite(v_scale))
    return MCS_ERR_INVALID_ARG;
  const int BH = p->B * p->H;
  // the sparse modes read rows with plain loads; the maps are kernel
  // parameters only
  CUtensorMap tq;
  if (!make_gather_map(&tq, q, BH, p->N, p->D))
    return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(gather)");
  mcs::AttnArgs a{};
  a.H = p->H;
  a.layout = p->layout;
  a.N = p->N;
  a.C = p->C;
  a.G = groups_of(p);
  a.K = p->K;
  a.scale_log2 = scale_of(p) * kLog2e * k_scale;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.perm = perm;
  a.idx = idx;
  a.aux_in = static_cast<const __nv_bfloat16*>(residual);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k8 = static_cast<const uint8_t*>(k8);
  a.v8 = static_cast<const uint8_t*>(v8);
  a.v_scale = v_scale;
  a.fault = fault_from_env();
  if ((s = status_ptr(&a.status)) != MCS_OK) return s;
  const int mode = (residual ? mcs::kSparseAdd : mcs::kSparse) | mcs::kE4M3;
  cudaError_t e = mcs::launch_attention(p->D, mode, &tq, &tq, &tq, a, BH, stream);
  if (e != cudaSuccess) return cuda_fail(e, "e4m3 sparse attention launch");
  return MCS_OK;
}

size_t mcs_pair_bytes(const mcs_params* p) {
  if (check_pairs(p) != MCS_OK) return 0;
  return mcs::pair_layout(p->B * p->H, groups_of(p), p->K).total;
}

mcs_status mcs_pair_lists(const mcs_params* p, const int32_t* idx, void* pairs,
                          size_t pairs_bytes, cudaStream_t stream) {
  mcs_status s = check_pairs(p);
  if (s != MCS_OK) return s;
  if (!idx || !pairs) return MCS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(pairs) & 255u) != 0) return MCS_ERR_INVALID_ARG;
  if (pairs_bytes < mcs_pair_bytes(p)) return MCS_ERR_WORKSPACE;
  unsigned* st;
  if ((s = status_ptr(&st)) != MCS_OK) return s;
  cudaError_t e =
      mcs::launch_pair_union(idx, p->B * p->H, groups_of(p), p->K, p->N, pairs, st, stream);
  if (e != cudaSuccess) return cuda_fail(e, "pair lists launch");
  return MCS_OK;
}

mcs_status mcs_sparse_attn_pairs(const mcs_params* p, const void* q, const void* k,
                                 const void* v, const int32_t* perm, const void* pairs,
                                 const void* residual, void* out, cudaStream_t stream) {
  if (!pairs) return MCS_ERR_INVALID_ARG;
  return run_sparse(p, q, k, v, perm, nullptr, residual, out,
                    residual ? mcs::kSparseAdd : mcs::kSparse, stream, pairs);
}

mcs_status mcs_sparse_attn_pairs_record(const mcs_params* p, const void* q, const void* k,
                                        const void* v, const int32_t* perm, const void* pairs,
                                        const void* dense_out, void* residual,
                                        cudaStream_t stream) {
  if (!pairs) return MCS_ERR_INVALID_ARG;
  return run_sparse(p, q, k, v, perm, nullptr, dense_out, residual, mcs::kSparseRecord, stream,
                    pairs);
}

mcs_status mcs_select(const mcs_params* p, const void* q, const void* k, const float* lse,
                      const int32_t* perm, int32_t* idx, float* retained, void* ws,
                      size_t ws_bytes, cudaStream_t stream) {
  mcs_status s = check_shape(p, true);
  if (s != MCS_OK) return s;
  if (!q || !k || !lse || !perm || !idx) return MCS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k)) return MCS_ERR_INVALID_ARG;
  const size_t per_head = select_head_bytes(p);
  if (!ws || !aligned16(ws) || ws_bytes < per_head) return MCS_ERR_WORKSPACE;
  const int BH = p->B * p->H;
  const int G = groups_of(p);
  // a chunk of heads at a time through the workspace: the masses [chunk, G, N],
  // then their digit histograms [chunk, G, kMassHistBins]
  const int chunk = static_cast<int>(std::min<size_t>(BH, ws_bytes / per_head));
  float* mass = static_cast<float*>(ws);
  uint32_t* hist = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) +
                                               round_up(chunk * mass_head_bytes(p), 256));
  for (int h0 = 0; h0 < BH; h0 += chunk) {
    const int hc = std::min(chunk, BH - h0);
    if ((s = run_group_mass(p, q, k, lse, perm, h0, hc, mass, hist, stream)) != MCS_OK) return s;
    int32_t* idx_h = idx + static_cast<size_t>(h0) * G * p->K;
    float* ret_h = retained ? retained + static_cast<size_t>(h0) * G : nullptr;
    if ((s = run_topk(p, mass, hist, hc * G, idx_h, ret_h, stream)) != MCS_OK) return s;
  }
  return MCS_OK;
}

mcs_status mcs_anchor_select(const mcs_params* p, const void* q, const void* k, const void* v,
                             int32_t* perm, int32_t* idx, void* dense_out, float* lse,
                             void* residual, float* retained, void* ws, size_t ws_bytes,
                             cudaStream_t stream) {
  mcs_status s = check_shape(p, true);
  if (s != MCS_OK) return s;
  if (!q || !k || !v || !perm || !idx || !dense_out || !lse || !residual)
    return MCS_ERR_INVALID_ARG;
  if (!ws || !aligned16(ws) || ws_bytes < std::max(select_head_bytes(p), mcs_group_workspace(p)))
    return MCS_ERR_WORKSPACE;
  // a1
  if ((s = mcs_group(p, q, perm, ws, ws_bytes, stream)) != MCS_OK) return s;
  // a2
  if ((s = mcs_dense_attn(p, q, k, v, dense_out, lse, stream)) != MCS_OK) return s;
  // a3 + a4
  if ((s = mcs_select(p, q, k, lse, perm, idx, retained, ws, ws_bytes, stream)) != MCS_OK) return s;
  // a5, anchor form
  return mcs_sparse_attn_record(p, q, k, v, perm, idx, dense_out, residual, stream);
}

}  // extern "C"
