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
//   pddp_moments   per (head, node, chunk of <= kChunkRows rows): the rows,
//                  gathered in position order with 16-byte cp.async into a
//                  swizzled two-stage ring; X^T X on tcgen05 (A = X^T, B = X,
//                  both MN-major views of the same tile), fp32 in TMEM; the
//                  column sums on the CUDA cores (16-byte shared loads)
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
constexpr int kMomProducers = 4;  // cp.async producer warps of the moments kernel
constexpr int kMomMmaWarp = 4 + kMomProducers;
constexpr int kMomThreads = 32 * (kMomMmaWarp + 1);

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
  static constexpr int kSmem = kUsed;
};

// Byte offset of 16-byte chunk `seg` of row r in a stage of two 128-byte-
// swizzled sub-tiles [128 rows x 128 B] (columns 0-63, 64-127).
__device__ __forceinline__ int mom_swz(int r, int seg) {
  return (seg >> 3) * (128 * 128) + r * 128 + (((seg & 7) ^ (r & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kMomThreads, 3)
    pddp_moments_kernel(const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ perm,
                        int N, int C, int depth, int slots, int max_chunks, float* partials,
                        unsigned* status, int layout, int H, int head0) {
  using L = MomLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* full = bars + 0;   // [2] rows landed (every producer thread)
  uint64_t* ready = bars + 2;  // [2] column sums taken (4 warp arrivals)
  uint64_t* empty = bars + 4;  // [2] MMA done with the stage
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
      mbar_init(full + s, kMomProducers * 32);
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
  if (warp == kMomMmaWarp) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int32_t* pos = perm + (size_t)bh * N + nd.start + chunk * kChunkRows;
  const RowMap rm = row_map(layout, H, N, head0 + bh);  // rows of q in either layout

  if (warp >= 4 && warp < kMomMmaWarp) {
    // ------------------------------------------------------------ producers
    // Producer warp pw copies rows 32 pw .. 32 pw + 31 of each tile with
    // 16-byte cp.async (kRPI whole rows per warp instruction, written in the
    // swizzled layout); lane l reads the token of row 32 pw + l once and
    // broadcasts it.  Rows past the node end are zero-filled.
    constexpr int kSegs = D * 2 / 16;  // 16-byte segments per row
    constexpr int kRPI = 32 / kSegs;   // rows per warp instruction
    const int pw = warp - 4;
    const int sub = lane / kSegs, seg = lane % kSegs;
    bool bad = false;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      const int rr = j * 128 + pw * 32 + lane;
      int t = rr < rows ? __ldg(pos + rr) : -1;
      if (t >= N || (rr < rows && t < 0)) { bad = true; t = -1; }
      const int myrow = t < 0 ? -1 : rm.rbase + t * rm.rstride;
      if (j >= 2) {
        bool ok = mbar_wait(empty + st, ((j >> 1) - 1) & 1, abort_flag, status);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      uint8_t* stage = smem + st * L::kStage;
#pragma unroll
      for (int i = 0; i < 32 / kRPI; ++i) {
        const int row = __shfl_sync(0xffffffffu, myrow, i * kRPI + sub);
        const int r = pw * 32 + i * kRPI + sub;
        cp_async16_zfill(stage + mom_swz(r, seg),
                         q + (size_t)(row < 0 ? 0 : row) * D + seg * 8, row >= 0);
      }
      cp_async_arrive(full + st);
    }
    if (bad) atomicOr(status, DEV_BOUNDS);
    asm volatile("cp.async.wait_all;" ::: "memory");  // every copy lands before exit
  } else if (warp == kMomMmaWarp) {
    // ------------------------------------------------------------ MMA
    // whole warp in the loop, one elected lane issues (a lane-0-only branch
    // issues MMAs much more slowly)
    constexpr uint32_t idesc = idesc_bf16(128, D, true, true);
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      const bool ok = mbar_wait(ready + st, (j >> 1) & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, ok)) break;
      fence_proxy_async_smem();  // rows written by cp.async, read by the MMA
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
    // ------------------------------------------------------------ column sums, epilogue
    // Thread t sums the 16-byte chunk cc = t % kCC (8 columns) over the rows
    // of row group t / kCC of every tile (rows past the node end are zero);
    // the row groups' partial sums are added at the end.
    constexpr int kCC = D / 8;        // 16-byte chunks per row
    constexpr int kRG = 128 / kCC;    // row groups
    constexpr int kRPG = 128 / kRG;   // rows per group
    const int t = threadIdx.x;  // 0..127
    const int cc = t % kCC, rgp = t / kCC;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      bool w = mbar_wait(full + st, (j >> 1) & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      const uint8_t* stage = smem + st * L::kStage;
#pragma unroll 4
      for (int i = 0; i < kRPG; ++i) {
        const int r = rgp * kRPG + i;
        const uint4 v = *reinterpret_cast<const uint4*>(stage + mom_swz(r, cc));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h[e]);
          acc[2 * e] += f.x;
          acc[2 * e + 1] += f.y;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ready + st);
      // the producers may overwrite this stage only after the MMA's commit,
      // which follows every compute warp's arrival
    }
    // partial column sums of the row groups -> shared memory (the first
    // stage: every copy into it has landed and the MMA reads it no more
    // once `done` completes), summed below in row-group order
    float colsum = 0.f;
    if (ok) {
      bool w = mbar_wait(done, 0, abort_flag, status);
      ok = __all_sync(0xffffffffu, w);
    }
    float* red = reinterpret_cast<float*>(smem);
    asm volatile("bar.sync 1, 128;" ::: "memory");  // warps 0-3: stage 0 free of readers
    if (ok) {
#pragma unroll
      for (int e = 0; e < 8; ++e) red[rgp * D + cc * 8 + e] = acc[e];
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (ok && t < D) {
      for (int g = 0; g < kRG; ++g) colsum += red[g * D + t];
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
          float4* o4 = reinterpret_cast<float4*>(out + t * D + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
      }
      if (t < D) out[D * D + t] = colsum;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMomMmaWarp) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------- power iteration

constexpr int kPowThreads = 256;

// One CTA per node.  Thread t owns row a = t / TPR of the node's covariance
// and the contiguous columns [part*SEG, (part+1)*SEG) of it (SEG = D / TPR),
// kept in registers as packed fp32 pairs for every iteration; an iteration
// reads only the current vector from shared memory (16-byte broadcast loads)
// and multiplies with packed f32x2 FMAs.  The matrix is first divided by its
// trace (largest eigenvalue <= 1, so the iterate cannot overflow), and the
// iterate is normalised after the first step, every kNormEvery steps and at
// the end instead of every step: power iteration's direction does not depend
// on the scale of the iterate, and a node whose covariance sends the start
// vector to zero is caught at the first step (it keeps the start vector).
// One block barrier per step.  (Re-reading the D x D matrix from shared
// memory every iteration made the deep tree levels, with thousands of nodes,
// shared-memory bound.)
template <int D>
__global__ void __launch_bounds__(kPowThreads, 2)
    pddp_power_kernel(const float* __restrict__ partials, int N, int C, int depth, int slots,
                      int max_chunks, int iters, float* __restrict__ nodevec) {
  constexpr int TPR = kPowThreads / D;  // threads per row: 2 (D=128) or 4 (D=64)
  constexpr int SEG = D / TPR;          // columns per thread: 64 or 16
  constexpr int kNormEvery = 8;
  static_assert(SEG % 4 == 0 && 32 % TPR == 0, "row segments are float4 vectors in one warp");
  __shared__ __align__(16) float s[D];
  __shared__ __align__(16) float vb[2][D];  // the iterate, double-buffered
  __shared__ float red[kPowThreads / 32];
  __shared__ int lead;
  const int slot = blockIdx.x, bh = blockIdx.y;
  const Node nd = node_at(N, C, depth, slot);
  if ((nd.n + C - 1) / C <= 1) return;
  const int nchunks = (nd.n + kChunkRows - 1) / kChunkRows;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int a = tid / TPR, part = tid % TPR, b0 = part * SEG;
  constexpr int DD = D * D + D;  // one chunk's partials: X^T X, then the column sums
  const float* base = partials + (size_t)(bh * slots + slot) * max_chunks * DD;
  // this thread's covariance segment (packed pairs) and (first D threads)
  // the column sums, summed over the node's chunks in chunk order
  uint64_t cp[SEG / 2];
#pragma unroll
  for (int k = 0; k < SEG / 2; ++k) cp[k] = 0ull;
  float sacc = 0.f, dacc = 0.f;
  for (int ch = 0; ch < nchunks; ++ch) {
    const float* pc = base + (size_t)ch * DD;
    const ulonglong2* row = reinterpret_cast<const ulonglong2*>(pc + a * D + b0);
#pragma unroll
    for (int k4 = 0; k4 < SEG / 4; ++k4) {
      const ulonglong2 x = __ldg(row + k4);
      cp[2 * k4] = f2_add(cp[2 * k4], x.x);
      cp[2 * k4 + 1] = f2_add(cp[2 * k4 + 1], x.y);
    }
    if (tid < D) sacc += __ldg(pc + D * D + tid);
    if (part == 0) dacc += __ldg(pc + a * D + a);  // the diagonal, for the trace
  }
  if (tid < D) {
    s[tid] = sacc;
    vb[0][tid] = rsqrtf(static_cast<float>(D));
  }
  __syncthreads();
  const float inv_n = 1.f / static_cast<float>(nd.n);
  const float sa = s[a] * inv_n;
  const uint64_t nsa = f2_pack(-sa, -sa);
#pragma unroll
  for (int k = 0; k < SEG / 2; ++k)
    cp[k] = f2_fma(nsa, f2_pack(s[b0 + 2 * k], s[b0 + 2 * k + 1]), cp[k]);  // Cov = X^T X - s s^T / n
  float diag = part == 0 ? dacc - sa * s[a] : 0.f;
  // trace of Cov, then Cov / trace
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) diag += __shfl_xor_sync(0xffffffffu, diag, o);
  if (lane == 0) red[wid] = diag;
  __syncthreads();
  float tr = 0.f;
#pragma unroll
  for (int i = 0; i < kPowThreads / 32; ++i) tr += red[i];
  const float inv_tr = tr > 0.f ? 1.f / tr : 1.f;
  const uint64_t itr2 = f2_pack(inv_tr, inv_tr);
#pragma unroll
  for (int k = 0; k < SEG / 2; ++k) cp[k] = f2_fma(cp[k], itr2, 0ull);
  int cur = 0;
  for (int it = 0; it < iters; ++it) {
    uint64_t acc0 = 0ull, acc1 = 0ull;
    const ulonglong2* v2 = reinterpret_cast<const ulonglong2*>(vb[cur] + b0);
#pragma unroll
    for (int k4 = 0; k4 < SEG / 4; ++k4) {
      const ulonglong2 x = v2[k4];
      acc0 = f2_fma(cp[2 * k4], x.x, acc0);
      acc1 = f2_fma(cp[2 * k4 + 1], x.y, acc1);
    }
    float a0, a1, a2, a3;
    f2_unpack(acc0, a0, a1);
    f2_unpack(acc1, a2, a3);
    float acc = (a0 + a1) + (a2 + a3);
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (part == 0) vb[cur ^ 1][a] = acc;
    __syncthreads();
    cur ^= 1;
    if (it == 0 || (it + 1) % kNormEvery == 0 || it == iters - 1) {
      const float x = tid < D ? vb[cur][tid] : 0.f;
      float sq = x * x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      __syncthreads();  // every thread has read red[] of the trace step or of the last norm
      if (lane == 0) red[wid] = sq;
      __syncthreads();
      float norm2 = 0.f;
#pragma unroll
      for (int i = 0; i < kPowThreads / 32; ++i) norm2 += red[i];
      if (norm2 == 0.f) {  // uniform: C v = 0, keep the previous vector
        cur ^= 1;
        break;
      }
      const float inv = rsqrtf(norm2);
      if (tid < D) vb[cur][tid] = x * inv;
      __syncthreads();
    }
  }
  __syncthreads();
  const float* v = vb[cur];
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

constexpr int kProjThreads = 256;

template <int D>
constexpr int proj_smem_bytes() { return (kProjThreads / 32) * 32 * D * 2; }

// One warp per 32 consecutive positions of a head.  The warp copies its 32
// rows into shared memory with 16-byte cp.async (all loads in flight at
// once), then lane l takes elements [l*E, (l+1)*E) of every row, forms its
// partial (x - mu).v for all 32 rows with the node's mean and direction in
// registers, and a butterfly transpose reduction leaves row l's projection
// in lane l.
template <int D>
__global__ void __launch_bounds__(kProjThreads)
    pddp_project_kernel(const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ perm,
                        int N, int C, int depth, int slots, const float* __restrict__ nodevec,
                        uint64_t* __restrict__ keys, int layout, int H, int head0) {
  constexpr int E = D / 32;          // elements of a row per lane: 4 (D = 128) or 2 (D = 64)
  constexpr int kSegs = D * 2 / 16;  // 16-byte chunks per row
  static_assert(E == 2 || E == 4, "D must be 64 or 128");
  extern __shared__ __align__(16) uint8_t proj_smem[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int p0 = (blockIdx.x * (kProjThreads / 32) + wid) * 32;
  const int bh = blockIdx.y;
  if (p0 >= N) return;  // whole warp
  uint8_t* buf = proj_smem + wid * 32 * D * 2;
  const int p = p0 + lane;
  // node holding position p; -1 for positions past N and for leaves
  int slot = -1;
  if (p < N) {
    Node nd{0, N};
    int s = 0;
    bool leaf = false;
    for (int b = 0; b < depth; ++b) {
      const int g = (nd.n + C - 1) / C;
      if (g <= 1) { leaf = true; break; }
      const int nl = C * (g / 2);
      if (p - nd.start < nl) {
        nd.n = nl;
        s = s << 1;
      } else {
        nd.start += nl;
        nd.n -= nl;
        s = (s << 1) | 1;
      }
    }
    if (!leaf && (nd.n + C - 1) / C > 1) slot = s;
  }
  const int token = slot >= 0 ? perm[(size_t)bh * N + p] : -1;
  const RowMap rm = row_map(layout, H, N, head0 + bh);
  const int myrow = token >= 0 ? rm.rbase + token * rm.rstride : -1;
  // rows -> shared memory: chunk c = lane + 32 i is segment c % kSegs of row c / kSegs
#pragma unroll
  for (int i = 0; i < kSegs; ++i) {
    const int c = lane + 32 * i;
    const int r = c / kSegs, sg = c % kSegs;
    const int row = __shfl_sync(0xffffffffu, myrow, r);
    cp_async16_zfill(buf + r * D * 2 + sg * 16, q + (size_t)(row < 0 ? 0 : row) * D + sg * 8,
                     row >= 0);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncwarp();
  float acc[32];
  int cached = -1;
  float vs[E], ms[E];
#pragma unroll
  for (int e = 0; e < E; ++e) vs[e] = ms[e] = 0.f;
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    const int sr = __shfl_sync(0xffffffffu, slot, r);
    acc[r] = 0.f;
    if (sr >= 0) {  // the same for the whole warp
      if (sr != cached) {
        const float* vec = nodevec + (size_t)(bh * slots + sr) * 2 * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          vs[e] = __ldg(vec + e);
          ms[e] = __ldg(vec + D + e);
        }
        cached = sr;
      }
      const __nv_bfloat162* x =
          reinterpret_cast<const __nv_bfloat162*>(buf + r * D * 2 + lane * E * 2);
      float t = 0.f;
#pragma unroll
      for (int h = 0; h < E / 2; ++h) {
        const float2 f = __bfloat1622float2(x[h]);
        t = fmaf(f.x - ms[2 * h], vs[2 * h], t);
        t = fmaf(f.y - ms[2 * h + 1], vs[2 * h + 1], t);
      }
      acc[r] = t;
    }
  }
  // transpose reduction: after the step of width w, a lane keeps the w rows
  // whose index has its lane's bit w, summed with its partner's
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? acc[i] : acc[i + w];
      const float keep = upper ? acc[i + w] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  if (slot >= 0) {
    uint32_t u = __float_as_uint(acc[0]);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // unsigned order == float order
    keys[(size_t)bh * N + p] = (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(token);
  }
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
  // stable partition by position: key <= T left, else right.  Warp w owns
  // the contiguous positions [w*len, (w+1)*len): it counts its left keys,
  // the warps' counts are scanned, then each warp writes its range in order
  // with ballots (no block barrier inside the loop).
  constexpr int kWarps = kSplitThreads / 32;
  const int lane = tid & 31, w = tid >> 5;
  const int len = (nd.n + kWarps - 1) / kWarps;
  const int lo = min(nd.n, w * len), hi = min(nd.n, lo + len);
  uint32_t nleft = 0;
  for (int b = lo; b < hi; b += 32) {
    const int i = b + lane;
    nleft += __popc(__ballot_sync(0xffffffffu, i < hi && kk[i] <= T));
  }
  __shared__ uint32_t wleft[kWarps];
  if (lane == 0) wleft[w] = nleft;
  __syncthreads();
  uint32_t before_left = 0;
  for (int v = 0; v < w; ++v) before_left += wleft[v];
  uint32_t run_left = before_left, run_right = static_cast<uint32_t>(lo) - before_left;
  const unsigned lt = (1u << lane) - 1u;
  for (int b = lo; b < hi; b += 32) {
    const int i = b + lane;
    const bool valid = i < hi;
    const bool left = valid && kk[i] <= T;
    const unsigned ml = __ballot_sync(0xffffffffu, left);
    const unsigned mr = __ballot_sync(0xffffffffu, valid && !left);
    if (valid) {
      const int dst = left ? static_cast<int>(run_left + __popc(ml & lt))
                           : nl + static_cast<int>(run_right + __popc(mr & lt));
      if (dst < nd.n && (left ? dst < nl : dst >= nl))
        out[dst] = in[i];
      else
        atomicOr(status, DEV_BOUNDS);
    }
    run_left += __popc(ml);
    run_right += __popc(mr);
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
cudaError_t run_pddp(const __nv_bfloat16* q, int layout, int H, int head0,
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
  e = cudaFuncSetAttribute(pddp_project_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           proj_smem_bytes<D>());
  if (e != cudaSuccess) return e;

  for (int d = 0; d < depths; ++d) {
    const int slots = 1 << d;
    const int chunks = (max_node_rows(N, C, d) + kChunkRows - 1) / kChunkRows;
    pddp_moments_kernel<D><<<dim3(chunks, slots, BH), kMomThreads, msmem, stream>>>(
        q, pa, N, C, d, slots, chunks, partials, status, layout, H, head0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pddp_power_kernel<D><<<dim3(slots, BH), kPowThreads, psmem, stream>>>(partials, N, C, d, slots,
                                                                          chunks, iters, nodevec);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    pddp_project_kernel<D><<<dim3((N + kProjThreads - 1) / kProjThreads, BH), kProjThreads,
                             proj_smem_bytes<D>(), stream>>>(q, pa, N, C, d, slots, nodevec, keys,
                                                             layout, H, head0);
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

cudaError_t launch_pddp(const __nv_bfloat16* q, int layout, int H, int head0, int BH, int N,
                        int D, int C, int iters, int32_t* perm_out, void* ws, size_t ws_bytes,
                        unsigned* status, cudaStream_t stream) {
  if (ws_bytes < pddp_workspace_bytes(BH, N, D, C)) return cudaErrorInvalidValue;
  if (D == 128)
    return run_pddp<128>(q, layout, H, head0, BH, N, C, iters, perm_out, ws, status, stream);
  if (D == 64) return run_pddp<64>(q, layout, H, head0, BH, N, C, iters, perm_out, ws, status, stream);
  return cudaErrorInvalidValue;
}

}  // namespace mcs
