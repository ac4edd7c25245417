// Diagnostic selectors and error measures (not on the reuse-step path).
//
// The pages separate the dense-sparse gap by comparing selectors that keep
// the same number of KV tokens (wispaper.ai, "The gap has three separable
// sources"; ai.info AI summary, "Methodology in Plain English"): mean-pooled
// block-sparse attention, whose score for a query group and a KV block is the
// dot product of the group's mean query with the block's mean key (wispaper.ai,
// "Mean-pooled block scoring misses high-mass tokens"); a block oracle that
// keeps whole KV blocks by their exact group mass; the token oracle (the exact
// group-mass selection of select.cu); and a per-query oracle (a group of one
// query).  They are compared by attention recall and by the relative L1 error
// of the output (ai.info AI summary, "Main Findings").
//
// KV blocks are the full blocks [b*block, (b+1)*block); the partial block at
// the end of the sequence is never selected.  Both block selectors rank
// blocks with the radix top-K of select.cu (ties to the lower block), then
// expand the kept blocks to their tokens.  These kernels move little data
// (group masses are read once; pooled operands are a few MB) and are written
// plainly: one warp per block sum, one CTA per pooled row.
#include <math.h>

#include <algorithm>

#include "internal.h"

namespace mcs {
namespace {

// bmass[r, b] = sum of mass[r, b*block .. b*block + block) over full blocks.
// One warp per block; lanes read consecutive masses.
__global__ void block_mass_kernel(const float* __restrict__ mass, int n, int block, int nb,
                                  float* __restrict__ bmass) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const size_t row = blockIdx.y;
  if (warp >= nb) return;
  const float* src = mass + row * n + static_cast<size_t>(warp) * block;
  float s = 0.f;
  for (int t = lane; t < block; t += 32) s += src[t];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) bmass[row * nb + warp] = s;
}

// idx[r, j*block + t] = bidx[r, j]*block + t
__global__ void expand_blocks_kernel(const int32_t* __restrict__ bidx, int kb, int block,
                                     long long total, int32_t* __restrict__ idx) {
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long K = static_cast<long long>(kb) * block;
    const long long r = e / K;
    const int within = static_cast<int>(e - r * K);
    idx[e] = bidx[r * kb + within / block] * block + within % block;
  }
}

// qbar[bh, g, :] = mean of the group's query rows (padding slots skipped).
// One CTA of D threads per (group, head).
__global__ void pool_queries_kernel(const __nv_bfloat16* __restrict__ q,
                                    const int32_t* __restrict__ perm, int N, int D, int C, int G,
                                    int layout, int H, float* __restrict__ qbar, unsigned* status) {
  const int g = blockIdx.x, bh = blockIdx.y, d = threadIdx.x;
  const RowMap rm = row_map(layout, H, N, bh);
  const int32_t* pg = perm + (static_cast<size_t>(bh) * G + g) * C;
  float s = 0.f;
  int cnt = 0;
  for (int p = 0; p < C; ++p) {
    const int t = __ldg(pg + p);
    if (t < 0) continue;
    if (t >= N) {
      if (d == 0) atomicOr(status, DEV_BOUNDS);
      continue;
    }
    s += __bfloat162float(q[static_cast<size_t>(rm.rbase + t * rm.rstride) * D + d]);
    ++cnt;
  }
  qbar[(static_cast<size_t>(bh) * G + g) * D + d] = cnt > 0 ? s / cnt : 0.f;
}

// kbar[bh, b, :] = mean of the key rows of full block b.  One CTA of D
// threads per (block, head).
__global__ void pool_keys_kernel(const __nv_bfloat16* __restrict__ k, int N, int D, int block,
                                 int nb, int layout, int H, float* __restrict__ kbar) {
  const int b = blockIdx.x, bh = blockIdx.y, d = threadIdx.x;
  const RowMap rm = row_map(layout, H, N, bh);
  float s = 0.f;
  for (int t = b * block; t < (b + 1) * block; ++t)
    s += __bfloat162float(k[static_cast<size_t>(rm.rbase + t * rm.rstride) * D + d]);
  kbar[(static_cast<size_t>(bh) * nb + b) * D + d] = s / block;
}

// Order-preserving map of a float to an unsigned key (larger float, larger
// key), so that the radix top-K, which ranks unsigned bit patterns, ranks
// scores of either sign.
__device__ __forceinline__ uint32_t float_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// keys[bh*G + g, b] = float_key(scale * qbar[bh, g] . kbar[bh, b]).  One CTA
// per (group, head); qbar row staged in shared memory.
__global__ void pooled_scores_kernel(const float* __restrict__ qbar,
                                     const float* __restrict__ kbar, int D, int G, int nb,
                                     float scale, uint32_t* __restrict__ keys) {
  __shared__ float sq[128];
  const int g = blockIdx.x, bh = blockIdx.y;
  if (threadIdx.x < D) sq[threadIdx.x] = qbar[(static_cast<size_t>(bh) * G + g) * D + threadIdx.x];
  __syncthreads();
  uint32_t* out = keys + (static_cast<size_t>(bh) * G + g) * nb;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    const float4* kr = reinterpret_cast<const float4*>(kbar + (static_cast<size_t>(bh) * nb + b) * D);
    float s = 0.f;
    for (int d4 = 0; d4 < D / 4; ++d4) {
      const float4 kv = kr[d4];
      s += sq[4 * d4] * kv.x + sq[4 * d4 + 1] * kv.y + sq[4 * d4 + 2] * kv.z +
           sq[4 * d4 + 3] * kv.w;
    }
    out[b] = float_key(scale * s);
  }
}

// retained[r] = sum of mass[r, idx[r, t]] over t.  One CTA per row.
__global__ void gather_mass_kernel(const float* __restrict__ mass, int n,
                                   const int32_t* __restrict__ idx, int K,
                                   float* __restrict__ retained, unsigned* status) {
  __shared__ float red[32];
  const size_t row = blockIdx.x;
  float s = 0.f;
  bool bad = false;
  for (int t = threadIdx.x; t < K; t += blockDim.x) {
    const int j = idx[row * K + t];
    if (j < 0 || j >= n) {
      bad = true;
      continue;
    }
    s += mass[row * n + j];
  }
  if (bad) atomicOr(status, DEV_BOUNDS);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) retained[row] = v;
  }
}

// sums[0] += sum |got - want|, sums[1] += sum |want| over the D elements of
// each listed row (rows == null: every row of `total_rows`).
__global__ void rel_l1_kernel(const __nv_bfloat16* __restrict__ got,
                              const __nv_bfloat16* __restrict__ want,
                              const int32_t* __restrict__ rows, long long nrows, int D,
                              long long total_rows, double* sums, unsigned* status) {
  __shared__ double red[2][32];
  double e = 0.0, w = 0.0;
  const long long total = nrows * D;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long rr = i / D;
    long long r = rr;
    if (rows != nullptr) {
      r = rows[rr];
      if (r < 0 || r >= total_rows) {
        atomicOr(status, DEV_BOUNDS);
        continue;
      }
    }
    const size_t off = static_cast<size_t>(r) * D + (i - rr * D);
    const double a = __bfloat162float(got[off]), b = __bfloat162float(want[off]);
    e += fabs(a - b);
    w += fabs(b);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    e += __shfl_xor_sync(0xffffffffu, e, o);
    w += __shfl_xor_sync(0xffffffffu, w, o);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = e;
    red[1][threadIdx.x >> 5] = w;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const bool in = threadIdx.x < (blockDim.x >> 5);
    double a = in ? red[0][threadIdx.x] : 0.0, b = in ? red[1][threadIdx.x] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (threadIdx.x == 0) {
      atomicAdd(sums, a);
      atomicAdd(sums + 1, b);
    }
  }
}

}  // namespace

namespace {

constexpr size_t kAlign = 256;
size_t rup(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct DiagLayout {
  size_t keys, bidx, qbar, kbar, total;
};

// Workspace of the block selectors for all B*H*G group rows.
DiagLayout diag_layout(const mcs_params* p, int block) {
  const size_t BH = static_cast<size_t>(p->B) * p->H;
  const size_t G = (static_cast<size_t>(p->N) + p->C - 1) / p->C;
  const size_t nb = static_cast<size_t>(p->N) / block, kb = static_cast<size_t>(p->K) / block;
  DiagLayout l;
  l.keys = 0;
  l.bidx = rup(BH * G * nb * 4);
  l.qbar = l.bidx + rup(BH * G * kb * 4);
  l.kbar = l.qbar + rup(BH * G * p->D * 4);
  l.total = l.kbar + rup(BH * nb * p->D * 4);
  return l;
}

// K must be a positive multiple of block, at most N / block full blocks.
mcs_status check_block(const mcs_params* p, int block) {
  mcs_status s = check_params(p, true);
  if (s != MCS_OK) return s;
  if (block < 1 || block > 1024 || p->K % block != 0 || p->K / block > p->N / block)
    return MCS_ERR_INVALID_ARG;
  return MCS_OK;
}

cudaError_t expand(const int32_t* bidx, int rows, int kb, int block, int32_t* idx,
                   cudaStream_t stream) {
  const long long total = static_cast<long long>(rows) * kb * block;
  const long long blocks = std::min<long long>((total + 255) / 256, 152LL * 32);
  expand_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(bidx, kb, block, total,
                                                                          idx);
  return cudaGetLastError();
}

}  // namespace
}  // namespace mcs

extern "C" {

size_t mcs_block_workspace(const mcs_params* p, int block) {
  if (mcs::check_block(p, block) != MCS_OK) return 0;
  return mcs::diag_layout(p, block).total;
}

mcs_status mcs_block_topk(const mcs_params* p, const float* mass, int rows, int block,
                          int32_t* idx, float* retained, void* ws, size_t ws_bytes,
                          cudaStream_t stream) {
  mcs_status s = mcs::check_block(p, block);
  if (s != MCS_OK) return s;
  const long long G = (p->N + p->C - 1) / p->C;
  if (rows < 1 || rows > static_cast<long long>(p->B) * p->H * G || !mass || !idx)
    return MCS_ERR_INVALID_ARG;
  const mcs::DiagLayout l = mcs::diag_layout(p, block);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % 16) != 0 || ws_bytes < l.total)
    return MCS_ERR_WORKSPACE;
  unsigned* st;
  cudaError_t e = mcs::device_status_word(&st);
  if (e != cudaSuccess) return mcs::record_cuda_error(e, "status word");
  char* w = static_cast<char*>(ws);
  float* bmass = reinterpret_cast<float*>(w + l.keys);
  int32_t* bidx = reinterpret_cast<int32_t*>(w + l.bidx);
  const int nb = p->N / block, kb = p->K / block;
  for (int r0 = 0; r0 < rows; r0 += 65535) {
    const int rc = std::min(65535, rows - r0);
    mcs::block_mass_kernel<<<dim3((nb + 7) / 8, rc), 256, 0, stream>>>(
        mass + static_cast<size_t>(r0) * p->N, p->N, block, nb, bmass + static_cast<size_t>(r0) * nb);
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) e = mcs::launch_topk(bmass, nullptr, rows, nb, kb, bidx, retained, st, stream);
  if (e == cudaSuccess) e = mcs::expand(bidx, rows, kb, block, idx, stream);
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, "block top-k launch");
}

mcs_status mcs_pooled_block_select(const mcs_params* p, const void* q, const void* k,
                                   const int32_t* perm, int block, int32_t* idx, void* ws,
                                   size_t ws_bytes, cudaStream_t stream) {
  mcs_status s = mcs::check_block(p, block);
  if (s != MCS_OK) return s;
  if (!q || !k || !perm || !idx) return MCS_ERR_INVALID_ARG;
  const mcs::DiagLayout l = mcs::diag_layout(p, block);
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % 16) != 0 || ws_bytes < l.total)
    return MCS_ERR_WORKSPACE;
  unsigned* st;
  cudaError_t e = mcs::device_status_word(&st);
  if (e != cudaSuccess) return mcs::record_cuda_error(e, "status word");
  char* w = static_cast<char*>(ws);
  uint32_t* keys = reinterpret_cast<uint32_t*>(w + l.keys);
  int32_t* bidx = reinterpret_cast<int32_t*>(w + l.bidx);
  float* qbar = reinterpret_cast<float*>(w + l.qbar);
  float* kbar = reinterpret_cast<float*>(w + l.kbar);
  const int BH = p->B * p->H, G = (p->N + p->C - 1) / p->C;
  const int nb = p->N / block, kb = p->K / block;
  const float scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->D));
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kbf = static_cast<const __nv_bfloat16*>(k);
  mcs::pool_queries_kernel<<<dim3(G, BH), p->D, 0, stream>>>(qb, perm, p->N, p->D, p->C, G,
                                                             p->layout, p->H, qbar, st);
  mcs::pool_keys_kernel<<<dim3(nb, BH), p->D, 0, stream>>>(kbf, p->N, p->D, block, nb, p->layout,
                                                           p->H, kbar);
  mcs::pooled_scores_kernel<<<dim3(G, BH), 256, 0, stream>>>(qbar, kbar, p->D, G, nb, scale,
                                                             keys);
  e = cudaGetLastError();
  // the keys are unsigned patterns, ranked by the top-K as they are
  if (e == cudaSuccess)
    e = mcs::launch_topk(reinterpret_cast<const float*>(keys), nullptr, BH * G, nb, kb, bidx,
                         nullptr, st, stream);
  if (e == cudaSuccess) e = mcs::expand(bidx, BH * G, kb, block, idx, stream);
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, "pooled block select launch");
}

mcs_status mcs_gather_mass(const mcs_params* p, const float* mass, int rows, const int32_t* idx,
                           float* retained, cudaStream_t stream) {
  mcs_status s = mcs::check_params(p, true);
  if (s != MCS_OK) return s;
  if (rows < 0 || (rows > 0 && (!mass || !idx || !retained))) return MCS_ERR_INVALID_ARG;
  if (rows == 0) return MCS_OK;
  unsigned* st;
  cudaError_t e = mcs::device_status_word(&st);
  if (e == cudaSuccess) {
    mcs::gather_mass_kernel<<<rows, 256, 0, stream>>>(mass, p->N, idx, p->K, retained, st);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, "gather mass launch");
}

mcs_status mcs_rel_l1(const mcs_params* p, const void* got, const void* want, const int32_t* rows,
                      int nrows, double* sums, cudaStream_t stream) {
  mcs_status s = mcs::check_params(p, false);
  if (s != MCS_OK) return s;
  if (!got || !want || !sums || nrows < 0 || (nrows > 0 && !rows)) return MCS_ERR_INVALID_ARG;
  const long long total_rows = static_cast<long long>(p->B) * p->H * p->N;
  const long long n = rows ? nrows : total_rows;
  unsigned* st;
  cudaError_t e = mcs::device_status_word(&st);
  if (e == cudaSuccess) e = cudaMemsetAsync(sums, 0, 2 * sizeof(double), stream);
  if (e == cudaSuccess && n > 0) {
    const long long blocks = std::min<long long>((n * p->D + 255) / 256, 152LL * 16);
    mcs::rel_l1_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(got), static_cast<const __nv_bfloat16*>(want), rows, n,
        p->D, total_rows, sums, st);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, "relative L1 launch");
}

}  // extern "C"
