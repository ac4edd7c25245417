// Fast PDDP: median-split principal direction divisive partitioning of the
// queries of every head into groups of exactly C (the short group last).
//
// Sources: wispaper.ai, "Token-level selection needs tile-aligned query
// groups" (project each group onto its principal direction, split the
// ordered queries at the median, recurse until every group holds C);
// ai.info AI summary, "Methodology in Plain English" and "Key
// Contributions" (batched power iteration across all heads at each tree
// depth, only index arrays passed between levels).
//
// Tree shape.  A node of n rows has g = ceil(n/C) groups; its left child
// takes the C*floor(g/2) rows of smallest projection, the right child the
// rest.  Node sizes therefore depend only on (N, C): at depth d, slot s
// (d bits, most significant first = the path from the root) is found by
// walking those bits from the root.  Every depth works on all heads and all
// nodes at once; between depths only the permutation array (token index per
// position) moves, nodes being contiguous position ranges.
//
// One depth = four launches:
//   pddp_moments   per (head, node, chunk of <= kChunkRows rows): X^T X and
//                  sum x of the chunk's rows on tcgen05 (A = X^T, B = X, both
//                  MN-major views of the same gathered tile), fp32 in TMEM
//   pddp_power     per (head, node): sum the chunk partials in fixed order,
//                  Cov = X^T X - s s^T / n, then `iters` steps v <- Cov v/|Cov v|
//                  from (1,..,1)/sqrt(D); sign: largest |v_d| positive
//   pddp_project   per position: t = (x - mu).v, key = (ordered bits of t, token)
//   pddp_split     per (head, node): radix-select the C*floor(g/2)-th smallest
//                  key, stable partition of the positions (leaves are copied)
// and finally pddp_finalize sorts each group's indices ascending and pads the
// short group with -1.
#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int kChunkRows = 1024;  // rows per moments CTA (8 tiles of 128)
constexpr int kMomThreads = 192;

struct Node {
  int start, n;
};

// Node of `slot` at `depth` (slot's bits from the most significant one are
// the left(0)/right(1) path).  n == 0: no node (a leaf reached earlier).
__host__ __device__ inline Node node_at(int N, int C, int depth, int slot) {
  Node nd{0, N};
  for (int b = depth - 1; b >= 0; --b) {
    const int bit = (slot >> b) & 1;
    const int g = (nd.n + C - 1) / C;
    if (g <= 1) {
      if (bit) nd.n = 0;
      if (nd.n == 0) return nd;
      continue;
    }
    const int nl = C * (g / 2);
    if (bit) {
      nd.start += nl;
      nd.n -= nl;
    } else {
      nd.n = nl;
    }
  }
  return nd;
}

int depth_count(int N, int C) {
  const int G = (N + C - 1) / C;
  int d = 0;
  while ((1 << d) < G) ++d;
  return d;
}

// Largest node at a depth, and the largest number of moments chunks of a node.
int max_node_rows(int N, int C, int depth) {
  int m = 0;
  for (int s = 0; s < (1 << depth); ++s) {
    const Node nd = node_at(N, C, depth, s);
    if (nd.n > m) m = nd.n;
  }
  return m;
}

struct WsLayout {
  size_t perm_a, perm_b, keys, partials, nodevec, total;
  int max_chunks_slots;  // max over depths of slots * chunks per node
  int max_slots;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

WsLayout ws_layout(int BH, int N, int D, int C) {
  WsLayout w{};
  const int depths = depth_count(N, C);
  int mcs = 1, ms = 1;
  for (int d = 0; d < depths; ++d) {
    const int chunks = (max_node_rows(N, C, d) + kChunkRows - 1) / kChunkRows;
    if ((1 << d) * chunks > mcs) mcs = (1 << d) * chunks;
    if ((1 << d) > ms) ms = 1 << d;
  }
  w.max_chunks_slots = mcs;
  w.max_slots = ms;
  size_t off = 0;
  w.perm_a = off;
  off += align256(sizeof(int32_t) * (size_t)BH * N);
  w.perm_b = off;
  off += align256(sizeof(int32_t) * (size_t)BH * N);
  w.keys = off;
  off += align256(sizeof(uint64_t) * (size_t)BH * N);
  w.partials = off;
  off += align256(sizeof(float) * (size_t)BH * mcs * (D * D + D));
  w.nodevec = off;
  off += align256(sizeof(float) * (size_t)BH * ms * 2 * D);
  w.total = off;
  return w;
}

// ---------------------------------------------------------------- init

__global__ void pddp_init_kernel(int32_t* perm, int N, int BH) {
  const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (i < (size_t)BH * N) perm[i] = static_cast<int32_t>(i % N);
}

// ---------------------------------------------------------------- moments

template <int D>
struct MomLayout {
  // Each stage: two 16 KB sub-tiles [128 rows x 128 B].  For D = 128 they
  // hold columns 0-63 and 64-127; for D = 64 the second one stays zero so
  // the M = 128 MMA (A = X^T, M = feature) sees zero rows 64-127.
  static constexpr int kSubBytes = 128 * 128;
  static constexpr int kStage = 2 * kSubBytes;
  static constexpr int kBars = 2 * kStage;
  static constexpr int kUsed = kBars + 128 + 1024;
  // three CTAs per SM: 3 x ~67 KB of shared memory, 3 x 128 TMEM columns
  static constexpr int kSmem = kUsed;
};

__device__ __forceinline__ float smem_x(const uint8_t* stage, int row, int col) {
  // element (row, col) of a 128B-swizzled tile pair
  const int sub = col >> 6;
  const int c = col & 63;
  const int chunk = (c >> 3) ^ (row & 7);
  const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(
      stage + sub * (128 * 128) + row * 128 + chunk * 16 + (c & 7) * 2);
  return __bfloat162float(*p);
}

template <int D>
__global__ void __launch_bounds__(kMomThreads, 3)
    pddp_moments_kernel(const __grid_constant__ CUtensorMap tq, const int32_t* __restrict__ perm,
                        int N, int C, int depth, int slots, int max_chunks, float* partials,
                        unsigned* status, int layout, int H, int head0) {
  using L = MomLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* full = bars + 0;   // [2]
  uint64_t* ready = bars + 2;  // [2]
  uint64_t* empty = bars + 4;  // [2]
  uint64_t* done = bars + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 7);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int chunk = blockIdx.x, slot = blockIdx.y, bh = blockIdx.z;
  const Node nd = node_at(N, C, depth, slot);
  if ((nd.n + C - 1) / C <= 1 || chunk * kChunkRows >= nd.n) return;  // uniform exit
  const int rows = min(kChunkRows, nd.n - chunk * kChunkRows);
  const int ntiles = (rows + 127) / 128;
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(full + s, 1);
      mbar_init(ready + s, 4);
      mbar_init(empty + s, 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (D == 64 && warp < 4) {
    // zero the second sub-tile of both stages
    for (int i = threadIdx.x; i < 2 * (128 * 128) / 16; i += 128) {
      const int st = i / ((128 * 128) / 16), o = i % ((128 * 128) / 16);
      reinterpret_cast<uint4*>(smem + st * L::kStage + L::kSubBytes)[o] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int32_t* pos = perm + (size_t)bh * N + nd.start + chunk * kChunkRows;
  const RowMap rm = row_map(layout, H, N, head0 + bh);  // rows of q in either layout

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    bool bad = false;
    int issued = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      int r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = j * 128 + 4 * lane + i;
        int t = rr < rows ? __ldg(pos + rr) : 0;
        if (t < 0 || t >= N) { bad = true; t = 0; }
        r[i] = rm.rbase + t * rm.rstride;
      }
      if (j >= 2) {
        bool ok = mbar_wait(empty + st, ((j >> 1) - 1) & 1, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      if (lane == 0) mbar_expect_tx(full + st, (D / 64) * L::kSubBytes);
      __syncwarp();
      for (int s = 0; s < D / 64; ++s)
        tma_gather4(smem + st * L::kStage + s * L::kSubBytes + lane * 4 * 128, &tq, s * 64, r[0],
                    r[1], r[2], r[3], full + st);
      ++issued;
    }
    if (bad) atomicOr(status, DEV_BOUNDS);
    if (*abort_flag && lane == 0) {
      for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
        const long long t0 = clock64();
        while (!mbar_try_wait(full + (j & 1), (j >> 1) & 1))
          if (clock64() - t0 > kWaitLimitCycles) break;
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA
    // whole warp in the loop, one elected lane issues (a lane-0-only branch
    // issues MMAs much more slowly)
    constexpr uint32_t idesc = idesc_bf16(128, D, true, true);
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      const bool ok = mbar_wait(ready + st, (j >> 1) & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t base = smem_u32(smem + st * L::kStage);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t d = sdesc_sw128(base + kk * 16 * 128, L::kSubBytes, 1024);
          umma_ss(tmem, d, d, idesc, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(empty + st);
      }
    }
    if (elect_one()) umma_commit(done);
    __syncwarp();
    const long long t0 = clock64();
    while (!mbar_try_wait(done, 0))
      if (clock64() - t0 > kWaitLimitCycles) break;
  } else {
    // ------------------------------------------------------------ row sums, tails, epilogue
    const int t = threadIdx.x;  // 0..127
    float colsum = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      bool w = mbar_wait(full + st, (j >> 1) & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      uint8_t* stage = smem + st * L::kStage;
      const int valid = min(128, rows - j * 128);
      if (valid < 128) {
        // rows past the node end were gathered from row 0: zero them
        for (int i = t; i < (128 - valid) * 8 * (D / 64); i += 128) {
          const int r = valid + i / (8 * (D / 64));
          const int rem = i % (8 * (D / 64));
          const int s = rem / 8, c16 = rem % 8;
          *reinterpret_cast<uint4*>(stage + s * L::kSubBytes + r * 128 + c16 * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
      if (t < D) {
        for (int r = 0; r < valid; ++r) colsum += smem_x(stage, r, t);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ready + st);
      // the producer may overwrite this stage only after the MMA's commit,
      // which follows every compute warp's arrival
    }
    if (ok) {
      bool w = mbar_wait(done, 0, abort_flag, status);
      ok = __all_sync(0xffffffffu, w);
    }
    if (ok) {
      tc_fence_after();
      float* out = partials + ((size_t)(bh * slots + slot) * max_chunks + chunk) * (D * D + D);
      const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + c * 32, v);
        tmem_ld_wait();
        if (t < D) {
#pragma unroll
          for (int i = 0; i < 32; ++i) out[t * D + c * 32 + i] = __uint_as_float(v[i]);
        }
      }
      if (t < D) out[D * D + t] = colsum;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------- power iteration

constexpr int kPowThreads = 256;

// One CTA per node.  Thread t owns row a = t / TPR of the node's covariance
// and the contiguous columns [part*SEG, (part+1)*SEG) of it (SEG = D / TPR),
// kept in registers for every iteration; an iteration reads only the current
// vector from shared memory, as 16-byte broadcast loads, and sums its
// products in four independent chains.  (Re-reading the D x D matrix from
// shared memory every iteration made the deep tree levels, with thousands of
// nodes, shared-memory bound.)
template <int D>
__global__ void __launch_bounds__(kPowThreads, 2)
    pddp_power_kernel(const float* __restrict__ partials, int N, int C, int depth, int slots,
                      int max_chunks, int iters, float* __restrict__ nodevec) {
  constexpr int TPR = kPowThreads / D;  // threads per row: 2 (D=128) or 4 (D=64)
  constexpr int SEG = D / TPR;          // columns per thread: 64 or 16
  static_assert(SEG % 4 == 0 && 32 % TPR == 0, "row segments are float4 vectors in one warp");
  __shared__ __align__(16) float s[D];
  __shared__ __align__(16) float v[D];
  __shared__ float w[D], red[kPowThreads / 32];
  __shared__ int lead;
  const int slot = blockIdx.x, bh = blockIdx.y;
  const Node nd = node_at(N, C, depth, slot);
  if ((nd.n + C - 1) / C <= 1) return;
  const int nchunks = (nd.n + kChunkRows - 1) / kChunkRows;
  const int tid = threadIdx.x;
  const int a = tid / TPR, part = tid % TPR, b0 = part * SEG;
  constexpr int DD = D * D + D;  // one chunk's partials: X^T X, then the column sums
  const float* base = partials + (size_t)(bh * slots + slot) * max_chunks * DD;
  // this thread's covariance segment and (first D threads) the column sums,
  // summed over the node's chunks in chunk order
  float c[SEG];
#pragma unroll
  for (int k = 0; k < SEG; ++k) c[k] = 0.f;
  float sacc = 0.f;
  for (int ch = 0; ch < nchunks; ++ch) {
    const float* pc = base + (size_t)ch * DD;
    const float4* row = reinterpret_cast<const float4*>(pc + a * D + b0);
#pragma unroll
    for (int k4 = 0; k4 < SEG / 4; ++k4) {
      const float4 x = __ldg(row + k4);
      c[4 * k4] += x.x;
      c[4 * k4 + 1] += x.y;
      c[4 * k4 + 2] += x.z;
      c[4 * k4 + 3] += x.w;
    }
    if (tid < D) sacc += __ldg(pc + D * D + tid);
  }
  if (tid < D) {
    s[tid] = sacc;
    v[tid] = rsqrtf(static_cast<float>(D));
  }
  __syncthreads();
  const float inv_n = 1.f / static_cast<float>(nd.n);
  const float sa = s[a];
#pragma unroll
  for (int k = 0; k < SEG; ++k) c[k] -= sa * s[b0 + k] * inv_n;  // Cov = X^T X - s s^T / n
  const float4* v4 = reinterpret_cast<const float4*>(v + b0);
  for (int it = 0; it < iters; ++it) {
    float acc4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k4 = 0; k4 < SEG / 4; ++k4) {
      const float4 x = v4[k4];
      acc4[0] = fmaf(c[4 * k4], x.x, acc4[0]);
      acc4[1] = fmaf(c[4 * k4 + 1], x.y, acc4[1]);
      acc4[2] = fmaf(c[4 * k4 + 2], x.z, acc4[2]);
      acc4[3] = fmaf(c[4 * k4 + 3], x.w, acc4[3]);
    }
    float acc = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    float sq = (part == 0) ? acc * acc : 0.f;
    if (part == 0) w[a] = acc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((tid & 31) == 0) red[tid >> 5] = sq;
    __syncthreads();
    float norm2 = 0.f;
#pragma unroll
    for (int i = 0; i < kPowThreads / 32; ++i) norm2 += red[i];
    if (norm2 == 0.f) break;  // uniform: every thread sums the same values
    const float nrm = sqrtf(norm2);
    if (tid < D) v[tid] = w[tid] / nrm;
    __syncthreads();
  }
  __syncthreads();
  if (tid == 0) {
    int best = 0;
    float bv = fabsf(v[0]);
    for (int i = 1; i < D; ++i)
      if (fabsf(v[i]) > bv) { bv = fabsf(v[i]); best = i; }
    lead = best;
  }
  __syncthreads();
  const float sign = v[lead] < 0.f ? -1.f : 1.f;
  float* out = nodevec + (size_t)(bh * slots + slot) * 2 * D;
  if (tid < D) {
    out[tid] = sign * v[tid];
    out[D + tid] = s[tid] * inv_n;  // mean
  }
}

// ---------------------------------------------------------------- projection

template <int D>
__global__ void __launch_bounds__(256)
    pddp_project_kernel(const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ perm,
                        int N, int C, int depth, int slots, const float* __restrict__ nodevec,
                        uint64_t* __restrict__ keys, int layout, int H, int head0) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  const int bh = blockIdx.y;
  if (p >= N) return;
  // find the node holding position p
  Node nd{0, N};
  int slot = 0;
  for (int b = 0; b < depth; ++b) {
    const int g = (nd.n + C - 1) / C;
    if (g <= 1) return;  // leaf: nothing to project
    const int nl = C * (g / 2);
    if (p - nd.start < nl) {
      nd.n = nl;
      slot = slot << 1;
    } else {
      nd.start += nl;
      nd.n -= nl;
      slot = (slot << 1) | 1;
    }
  }
  if ((nd.n + C - 1) / C <= 1) return;
  const int token = perm[(size_t)bh * N + p];
  const float* vec = nodevec + (size_t)(bh * slots + slot) * 2 * D;
  const RowMap rm = row_map(layout, H, N, head0 + bh);
  const uint4* row = reinterpret_cast<const uint4*>(q + (size_t)(rm.rbase + token * rm.rstride) * D);
  float t = 0.f;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 w = __ldg(row + c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      const int d = c * 8 + 2 * e;
      t = fmaf(f.x - __ldg(vec + D + d), __ldg(vec + d), t);
      t = fmaf(f.y - __ldg(vec + D + d + 1), __ldg(vec + d + 1), t);
    }
  }
  uint32_t u = __float_as_uint(t);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // unsigned order == float order
  keys[(size_t)bh * N + p] = (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(token);
}

// ---------------------------------------------------------------- select + partition

constexpr int kSplitThreads = 512;

__device__ __forceinline__ uint32_t block_scan_incl(uint32_t v, uint32_t* wsum, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kSplitThreads / 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) wsum[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t x = lane < kWarps ? wsum[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += n;
    }
    if (lane < kWarps) wsum[lane] = x;
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? wsum[warp - 1] : 0u;
  *total = wsum[kWarps - 1];
  __syncthreads();
  return v + before;
}

__global__ void __launch_bounds__(kSplitThreads)
    pddp_split_kernel(const uint64_t* __restrict__ keys, const int32_t* __restrict__ perm_in,
                      int32_t* __restrict__ perm_out, int N, int C, int depth, unsigned* status) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t sel_digit, sel_below;
  const int slot = blockIdx.x, bh = blockIdx.y;
  const Node nd = node_at(N, C, depth, slot);
  if (nd.n == 0) return;
  const int tid = threadIdx.x;
  const int32_t* in = perm_in + (size_t)bh * N + nd.start;
  int32_t* out = perm_out + (size_t)bh * N + nd.start;
  const int g = (nd.n + C - 1) / C;
  if (g <= 1) {
    for (int i = tid; i < nd.n; i += kSplitThreads) out[i] = in[i];
    return;
  }
  const int nl = C * (g / 2);
  const uint64_t* kk = keys + (size_t)bh * N + nd.start;
  // radix select of the nl-th smallest key, 8 bits at a time from the top
  uint64_t prefix = 0, mask = 0;
  uint32_t remaining = static_cast<uint32_t>(nl);
  uint64_t T = ~0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += kSplitThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < nd.n; i += kSplitThreads) {
      const uint64_t k = kk[i];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    uint32_t mine = tid < 256 ? hist[tid] : 0u;
    uint32_t total;
    const uint32_t incl = block_scan_incl(mine, wsum, &total);
    if (tid < 256) {
      const uint32_t below = incl - mine;
      if (below < remaining && remaining <= incl) {
        sel_digit = tid;
        sel_below = below;
      }
    }
    __syncthreads();
    const uint32_t cnt = hist[sel_digit];
    prefix |= static_cast<uint64_t>(sel_digit) << shift;
    mask |= 255ull << shift;
    remaining -= sel_below;
    __syncthreads();
    if (remaining == cnt) {  // the whole bucket is at or below the threshold
      T = prefix | ~mask;
      break;
    }
    if (shift == 0) T = prefix;
  }
  // stable partition by position: key <= T left, else right
  uint32_t run_left = 0, run_right = 0;
  for (int base = 0; base < nd.n; base += kSplitThreads) {
    const int i = base + tid;
    bool valid = i < nd.n, left = false;
    if (valid) left = kk[i] <= T;
    const uint32_t packed = valid ? (left ? (1u << 16) : 1u) : 0u;
    uint32_t total;
    const uint32_t incl = block_scan_incl(packed, wsum, &total);
    const uint32_t excl = incl - packed;
    if (valid) {
      const int dst = left ? static_cast<int>(run_left + (excl >> 16))
                           : nl + static_cast<int>(run_right + (excl & 0xFFFFu));
      if (dst < nd.n && (left ? dst < nl : dst >= nl))
        out[dst] = in[i];
      else
        atomicOr(status, DEV_BOUNDS);
    }
    run_left += total >> 16;
    run_right += total & 0xFFFFu;
  }
}

// ---------------------------------------------------------------- finalize

__global__ void __launch_bounds__(128)
    pddp_finalize_kernel(const int32_t* __restrict__ perm_work, int32_t* __restrict__ perm_out,
                         int N, int C, int G) {
  __shared__ int32_t buf[128];
  const int g = blockIdx.x, bh = blockIdx.y, t = threadIdx.x;
  const int n = min(C, N - g * C);
  int v = 0x7fffffff;
  if (t < n) v = perm_work[(size_t)bh * N + g * C + t];
  buf[t] = v;
  __syncthreads();
  // bitonic sort of 128 values, ascending
  for (int k = 2; k <= 128; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int ixj = t ^ j;
      if (ixj > t) {
        const int a = buf[t], b = buf[ixj];
        const bool up = (t & k) == 0;
        if ((a > b) == up) {
          buf[t] = b;
          buf[ixj] = a;
        }
      }
      __syncthreads();
    }
  }
  if (t < C) perm_out[((size_t)bh * G + g) * C + t] = t < n ? buf[t] : -1;
}

template <int D>
cudaError_t run_pddp(const __nv_bfloat16* q, const CUtensorMap* tq, int layout, int H, int head0,
                     int BH, int N, int C, int iters, int32_t* perm_out, void* ws,
                     unsigned* status, cudaStream_t stream) {
  const WsLayout w = ws_layout(BH, N, D, C);
  uint8_t* base = static_cast<uint8_t*>(ws);
  int32_t* pa = reinterpret_cast<int32_t*>(base + w.perm_a);
  int32_t* pb = reinterpret_cast<int32_t*>(base + w.perm_b);
  uint64_t* keys = reinterpret_cast<uint64_t*>(base + w.keys);
  float* partials = reinterpret_cast<float*>(base + w.partials);
  float* nodevec = reinterpret_cast<float*>(base + w.nodevec);
  const int G = (N + C - 1) / C;
  const int depths = depth_count(N, C);

  const size_t total = (size_t)BH * N;
  pddp_init_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(pa, N, BH);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int msmem = MomLayout<D>::kSmem;
  e = cudaFuncSetAttribute(pddp_moments_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           msmem);
  if (e != cudaSuccess) return e;
  const int psmem = 0;  // the power kernel's shared memory is static

  for (int d = 0; d < depths; ++d) {
    const int slots = 1 << d;
    const int chunks = (max_node_rows(N, C, d) + kChunkRows - 1) / kChunkRows;
    pddp_moments_kernel<D><<<dim3(chunks, slots, BH), kMomThreads, msmem, stream>>>(
        *tq, pa, N, C, d, slots, chunks, partials, status, layout, H, head0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pddp_power_kernel<D><<<dim3(slots, BH), kPowThreads, psmem, stream>>>(partials, N, C, d, slots,
                                                                          chunks, iters, nodevec);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pddp_project_kernel<D><<<dim3((N + 255) / 256, BH), 256, 0, stream>>>(
        q, pa, N, C, d, slots, nodevec, keys, layout, H, head0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pddp_split_kernel<<<dim3(slots, BH), kSplitThreads, 0, stream>>>(keys, pa, pb, N, C, d,
                                                                     status);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    int32_t* t = pa;
    pa = pb;
    pb = t;
  }
  pddp_finalize_kernel<<<dim3(G, BH), 128, 0, stream>>>(pa, perm_out, N, C, G);
  return cudaGetLastError();
}

}  // namespace

size_t pddp_workspace_bytes(int BH, int N, int D, int C) { return ws_layout(BH, N, D, C).total; }

cudaError_t launch_pddp(const __nv_bfloat16* q, const CUtensorMap* tq_gather, int layout, int H,
                        int head0, int BH, int N, int D, int C, int iters, int32_t* perm_out,
                        void* ws, size_t ws_bytes, unsigned* status, cudaStream_t stream) {
  if (ws_bytes < pddp_workspace_bytes(BH, N, D, C)) return cudaErrorInvalidValue;
  if (D == 128)
    return run_pddp<128>(q, tq_gather, layout, H, head0, BH, N, C, iters, perm_out, ws, status,
                         stream);
  if (D == 64)
    return run_pddp<64>(q, tq_gather, layout, H, head0, BH, N, C, iters, perm_out, ws, status,
                        stream);
  return cudaErrorInvalidValue;
}

}  // namespace mcs
