// Sibling-pair key lists for C = 64 groups.
//
// A C = 64 group fills only half of the 128-row query tile of a tcgen05 MMA
// (an M = 64 MMA takes as long as an M = 128 one).  Groups 2u and 2u+1 are
// siblings in the grouping tree (PDDP splits a node into them last), so their
// queries are similar and their selected KV sets overlap heavily.  The sparse
// kernel's paired mode runs both groups in one 128-row tile over the UNION of
// their index sets, and a per-row mask (-2^20 added through one more MMA step
// to the scores of keys the row's group did not select) keeps each query's
// softmax over its own group's K tokens only: the same attention as two
// separate groups (wispaper.ai, "Token-level selection needs tile-aligned
// query groups"), with |A u B| <= 2K key columns per 128 rows instead of 2K.
//
// This file builds the union lists from idx (sorted rows), one CTA per pair:
// both rows in shared memory; for a in A its rank among B (binary search)
// and whether B holds it; an exclusive prefix of those duplicates; then
//   position of A[i] = i + rank_B(A[i]) - dups(A[0..i))
//   position of B[j] not in A = j + rank_A(B[j]) - dups(A[0..rank_A(B[j])))
// which is its place in the ascending union without repeats.
#include "internal.h"

namespace mcs {
namespace {

constexpr int kPairThreads = 512;

// number of entries of s[0..n) smaller than x (s ascending)
__device__ __forceinline__ int lower_bound_s(const int32_t* s, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kPairThreads)
    pair_union_kernel(const int32_t* __restrict__ idx, int G, int K, int N, int P, int cap,
                      int32_t* __restrict__ lens, int32_t* __restrict__ entries,
                      unsigned* status) {
  extern __shared__ int32_t psm[];
  int32_t* sA = psm;          // [K]
  int32_t* sB = psm + K;      // [K]
  int32_t* pre = psm + 2 * K;  // [K + 1]: duplicates among A[0..i)
  __shared__ int32_t wsum[kPairThreads / 32];
  const int u = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  const bool hasB = 2 * u + 1 < G;
  const int32_t* A = idx + ((size_t)bh * G + 2 * u) * K;
  const int32_t* B = A + K;
  bool bad = false;
  for (int i = tid; i < K; i += kPairThreads) {
    int32_t a = __ldg(A + i);
    if (a < 0 || a >= N) { bad = true; a = 0; }
    sA[i] = a;
    if (hasB) {
      int32_t b = __ldg(B + i);
      if (b < 0 || b >= N) { bad = true; b = 0; }
      sB[i] = b;
    }
  }
  __syncthreads();
  // duplicates of A in B over contiguous per-thread ranges, then a block scan
  const int per = (K + kPairThreads - 1) / kPairThreads;
  const int lo = min(K, tid * per), hi = min(K, lo + per);
  int cnt = 0;
  if (hasB) {
    for (int i = lo; i < hi; ++i) {
      const int rb = lower_bound_s(sB, K, sA[i]);
      cnt += (rb < K && sB[rb] == sA[i]) ? 1 : 0;
    }
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int v = 0; v < kPairThreads / 32; ++v) {
    before += v < w ? wsum[v] : 0;
    total += wsum[v];
  }
  int run = before + incl - cnt;
  for (int i = lo; i < hi; ++i) {
    pre[i] = run;
    if (hasB) {
      const int rb = lower_bound_s(sB, K, sA[i]);
      run += (rb < K && sB[rb] == sA[i]) ? 1 : 0;
    }
  }
  if (tid == 0) pre[K] = total;
  __syncthreads();
  const int len = hasB ? 2 * K - total : K;
  int32_t* out = entries + ((size_t)bh * P + u) * cap;
  constexpr uint32_t kInA = 1u << kPairTokenBits, kInB = 2u << kPairTokenBits;
  for (int i = tid; i < K; i += kPairThreads) {
    const int32_t a = sA[i];
    int rb = 0;
    bool dup = false;
    if (hasB) {
      rb = lower_bound_s(sB, K, a);
      dup = rb < K && sB[rb] == a;
    }
    const int pos = i + rb - pre[i];
    if (pos >= 0 && pos < cap)
      out[pos] = static_cast<int32_t>(static_cast<uint32_t>(a) | kInA | (dup ? kInB : 0u));
  }
  if (hasB) {
    for (int j = tid; j < K; j += kPairThreads) {
      const int32_t b = sB[j];
      const int ra = lower_bound_s(sA, K, b);
      if (ra < K && sA[ra] == b) continue;  // written with A's entry
      const int pos = j + ra - pre[ra];
      if (pos >= 0 && pos < cap) out[pos] = static_cast<int32_t>(static_cast<uint32_t>(b) | kInB);
    }
  }
  for (int q = len + tid; q < cap; q += kPairThreads) out[q] = 0;  // token 0, in neither group
  if (tid == 0) lens[(size_t)bh * P + u] = len;
  if (bad) atomicOr(status, DEV_BOUNDS);
}

}  // namespace

cudaError_t launch_pair_union(const int32_t* idx, int BH, int G, int K, int N, void* pairs,
                              unsigned* status, cudaStream_t stream) {
  const PairLayout l = pair_layout(BH, G, K);
  const int smem = (3 * K + 1) * 4;
  cudaError_t e =
      cudaFuncSetAttribute(pair_union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  uint8_t* base = static_cast<uint8_t*>(pairs);
  pair_union_kernel<<<dim3(l.P, BH), kPairThreads, smem, stream>>>(
      idx, G, K, N, l.P, l.cap, reinterpret_cast<int32_t*>(base),
      reinterpret_cast<int32_t*>(base + l.entries_off), status);
  return cudaGetLastError();
}

}  // namespace mcs
