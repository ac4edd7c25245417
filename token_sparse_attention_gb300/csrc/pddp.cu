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
// One depth = four to six launches:
//   pddp_moments   per (head, node, chunk of <= kChunkRows rows): the rows,
//                  gathered in position order with 16-byte cp.async into a
//                  swizzled two-stage ring; X^T X on tcgen05 (A = X^T, B = X,
//                  both MN-major views of the same tile), fp32 in TMEM; the
//                  column sums by one more MMA against a block of ones
//   pddp_reduce    (nodes of many chunks) sum the chunk partials in chunk order
//   pddp_power     per (head, node): (sum a few chunk partials in chunk order)
//                  Cov = X^T X - s s^T / n, then `iters` steps v <- Cov v/|Cov v|
//                  from (1,..,1)/sqrt(D); sign: largest |v_d| positive
//   pddp_project   per position: t = (x - mu).v, key = (ordered bits of t, token)
//   pddp_split     per (head, node): radix-select the C*floor(g/2)-th smallest
//                  key, stable partition of the positions; one CTA per big node,
//                  one warp per small node (a new leaf is copied once)
// and finally pddp_finalize sorts each group's indices ascending and pads the
// short group with -1.
#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int kChunkRows = 1024;  // rows per moments CTA (8 tiles of 128)
constexpr int kMomProducers = 8;  // cp.async producer warps of the moments kernel (0-7)
constexpr int kMomStages = 3;     // ring stages of the moments kernel (two CTAs per SM)
constexpr int kMomMmaWarp = kMomProducers;
constexpr int kMomThreads = 32 * (kMomMmaWarp + 1);

struct Node {
  int start, n;
};

// Node of `slot` at `depth` (slot's bits from the most significant one are
// the left(0)/right(1) path).  n == 0: no node (a leaf reached earlier).
// *stale (optional): the walk passed a leaf above `depth` (the node is that
// leaf, carried down along its 0 path).
__host__ __device__ inline Node node_at(int N, int C, int depth, int slot,
                                        bool* stale = nullptr) {
  Node nd{0, N};
  for (int b = depth - 1; b >= 0; --b) {
    const int bit = (slot >> b) & 1;
    const int g = (nd.n + C - 1) / C;
    if (g <= 1) {
      if (stale) *stale = true;
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
  size_t perm_a, perm_b, keys, partials, nodevec, table, total;
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
  w.table = off;  // per depth: the slots of the nodes that split, ascending
  off += align256(sizeof(int32_t) * (size_t)(depths > 0 ? depths : 1) * ms);
  w.total = off;
  return w;
}

// Number of nodes that split at `depth` (g > 1); the same for every head.
int split_count(int N, int C, int depth) {
  int k = 0;
  for (int s = 0; s < (1 << depth); ++s) {
    const Node nd = node_at(N, C, depth, s);
    if ((nd.n + C - 1) / C > 1) ++k;
  }
  return k;
}

// ---------------------------------------------------------------- init

// Block d lists, ascending, the slots of the nodes that split at depth d, so
// that the per-node kernels of a depth launch one CTA per such node (the deep
// levels hold many empty slots and leaves).
constexpr int kTableThreads = 256;

__global__ void __launch_bounds__(kTableThreads)
    pddp_table_kernel(int N, int C, int max_slots, int32_t* __restrict__ table) {
  __shared__ int wcount[kTableThreads / 32];
  const int d = blockIdx.x, slots = 1 << d;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int run = 0;  // entries written by earlier rounds
  for (int base = 0; base < slots; base += kTableThreads) {
    const int s = base + tid;
    bool split = false;
    if (s < slots) {
      const Node nd = node_at(N, C, d, s);
      split = (nd.n + C - 1) / C > 1;
    }
    const unsigned m = __ballot_sync(0xffffffffu, split);
    if (lane == 0) wcount[w] = __popc(m);
    __syncthreads();
    int before = run, total = run;
    for (int v = 0; v < kTableThreads / 32; ++v) {
      if (v < w) before += wcount[v];
      total += wcount[v];
    }
    if (split) table[(size_t)d * max_slots + before + __popc(m & ((1u << lane) - 1u))] = s;
    run = total;
    __syncthreads();  // wcount is rewritten by the next round
  }
}

__global__ void pddp_init_kernel(int32_t* perm, int N, int BH) {
  const size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (i < (size_t)BH * N) perm[i] = static_cast<int32_t>(i % N);
}

// ---------------------------------------------------------------- moments

template <int D>
struct MomLayout {
  // Each stage: two 16 KB sub-tiles [128 rows x 128 B].  For D = 128 they
  // hold columns 0-63 and 64-127; for D = 64 the second one stays zero so
  // the M = 128 MMA (A = X^T, M = feature) sees zero rows 64-127.  After the
  // barriers: a 16 x 16 block of bf16 ones, the B operand of the column sums.
  static constexpr int kSubBytes = 128 * 128;
  static constexpr int kStage = 2 * kSubBytes;
  static constexpr int kBars = kMomStages * kStage;
  static constexpr int kOnes = kBars + 128;
  static constexpr int kUsed = kOnes + 512 + 1024;
  static constexpr int kSmem = kUsed;
};

// Byte offset of 16-byte chunk `seg` of row r in a stage of two 128-byte-
// swizzled sub-tiles [128 rows x 128 B] (columns 0-63, 64-127).
__device__ __forceinline__ int mom_swz(int r, int seg) {
  return (seg >> 3) * (128 * 128) + r * 128 + (((seg & 7) ^ (r & 7)) << 4);
}

// Per (head, node, chunk): X^T X of the chunk's rows into TMEM columns 0-127
// and the column sums, X^T 1, into columns 128-143 (one more N = 16 MMA per
// K step against a block of ones), so that a stage is free again as soon as
// its MMAs complete.  Warps 0-7 copy rows; warp 8 issues the MMAs; warps 0-3
// then write the chunk's partial (X^T X, then the column sums).  Two CTAs per
// SM (256 TMEM columns each).
template <int D>
__global__ void __launch_bounds__(kMomThreads, 2)
    pddp_moments_kernel(const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ perm,
                        const int32_t* __restrict__ slot_tab, int N, int C, int depth, int slots,
                        int max_chunks, float* partials, unsigned* status, int layout, int H,
                        int head0) {
  using L = MomLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* full = bars + 0;            // [kMomStages] rows landed (every producer thread)
  uint64_t* empty = bars + kMomStages;  // [kMomStages] MMA done with the stage
  uint64_t* done = bars + 2 * kMomStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMomStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int chunk = blockIdx.x, slot = slot_tab[blockIdx.y], bh = blockIdx.z;
  const Node nd = node_at(N, C, depth, slot);
  if ((nd.n + C - 1) / C <= 1 || chunk * kChunkRows >= nd.n) return;  // uniform exit
  const int rows = min(kChunkRows, nd.n - chunk * kChunkRows);
  const int ntiles = (rows + 127) / 128;
  const int warp = warp_id(), lane = lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMomStages; ++s) {
      mbar_init(full + s, kMomProducers * 32);
      mbar_init(empty + s, 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp < 4) {
    // the ones block (bf16 1.0 = 0x3F80), and for D = 64 zeros in the second
    // sub-tile of both stages
    if (threadIdx.x < 32)
      reinterpret_cast<uint4*>(smem + L::kOnes)[threadIdx.x] =
          make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    if (D == 64) {
      for (int i = threadIdx.x; i < kMomStages * (128 * 128) / 16; i += 128) {
        const int st = i / ((128 * 128) / 16), o = i % ((128 * 128) / 16);
        reinterpret_cast<uint4*>(smem + st * L::kStage + L::kSubBytes)[o] = make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async_smem();
  }
  if (warp == kMomMmaWarp) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int32_t* pos = perm + (size_t)bh * N + nd.start + chunk * kChunkRows;
  const RowMap rm = row_map(layout, H, N, head0 + bh);  // rows of q in either layout

  bool ok = true;
  if (warp < kMomProducers) {
    // ------------------------------------------------------------ producers
    // Producer warp pw copies rows 16 pw .. 16 pw + 15 of each tile with
    // 16-byte cp.async (kRPI whole rows per warp instruction, written in the
    // swizzled layout); lane l < 16 reads the token of row 16 pw + l (the
    // next tile's one tile ahead) and broadcasts it.  Rows past the node end
    // are zero-filled.
    constexpr int kRows = 128 / kMomProducers;  // rows of a tile per warp
    constexpr int kSegs = D * 2 / 16;           // 16-byte segments per row
    constexpr int kRPI = 32 / kSegs;            // rows per warp instruction
    static_assert(kRows % kRPI == 0, "whole rows per warp instruction");
    const int pw = warp;
    const int sub = lane / kSegs, seg = lane % kSegs;
    const int myr = pw * kRows + (lane % kRows);
    bool bad = false;
    int tnext = myr < rows ? __ldg(pos + myr) : -1;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kMomStages;
      const int rr = j * 128 + myr;
      int t = tnext;
      if (j + 1 < ntiles) tnext = rr + 128 < rows ? __ldg(pos + rr + 128) : -1;
      if (t >= N || (rr < rows && t < 0)) { bad = true; t = -1; }
      const int myrow = t < 0 ? -1 : rm.rbase + t * rm.rstride;
      if (j >= kMomStages) {  // the stage's previous tile, j - kMomStages, is multiplied
        bool w = mbar_wait(empty + st, (j / kMomStages - 1) & 1, abort_flag, status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      }
      uint8_t* stage = smem + st * L::kStage;
#pragma unroll
      for (int i = 0; i < kRows / kRPI; ++i) {
        const int row = __shfl_sync(0xffffffffu, myrow, i * kRPI + sub);
        const int r = pw * kRows + i * kRPI + sub;
        cp_async16_zfill(stage + mom_swz(r, seg),
                         q + (size_t)(row < 0 ? 0 : row) * D + seg * 8, row >= 0);
      }
      cp_async_arrive(full + st);
    }
    if (bad) atomicOr(status, DEV_BOUNDS);
    asm volatile("cp.async.wait_all;" ::: "memory");  // every copy lands before exit
  } else {
    // ------------------------------------------------------------ MMA
    // whole warp in the loop, one elected lane issues (a lane-0-only branch
    // issues MMAs much more slowly)
    constexpr uint32_t idesc = idesc_bf16(128, D, true, true);
    constexpr uint32_t idesc_sum = idesc_bf16(128, 16, true, false);
    const uint64_t ones = sdesc_none(smem_u32(smem + L::kOnes), 128, 256);
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % kMomStages;
      const bool w = mbar_wait(full + st, (j / kMomStages) & 1, abort_flag, status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      fence_proxy_async_smem();  // rows written by cp.async, read by the MMA
      tc_fence_after();
      const uint32_t base = smem_u32(smem + st * L::kStage);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t d = sdesc_sw128(base + kk * 16 * 128, L::kSubBytes, 1024);
          const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
          umma_ss(tmem, d, d, idesc, acc);
          umma_ss(tmem + 128, d, ones, idesc_sum, acc);
        }
        umma_commit(empty + st);
      }
      __syncwarp();
    }
    if (elect_one()) umma_commit(done);  // after every MMA issued (or none)
    __syncwarp();
  }

  // ------------------------------------------------------------ epilogue
  // warps 0-3: TMEM lane t = feature row t
  if (warp < 4) {
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      const bool w = mbar_wait(done, 0, abort_flag, status);
      ok = __all_sync(0xffffffffu, w);
    }
    if (ok) {
      tc_fence_after();
      const int t = threadIdx.x;  // 0..127
      float* out = partials + ((size_t)(bh * slots + slot) * max_chunks + chunk) * (D * D + D);
      const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
      // thread t holds row t of X^T X; the matrix is symmetric, so it stores
      // its 32 columns c*32+i as column t of rows c*32+i: one coalesced
      // 128-byte row segment per warp and store
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + c * 32, v);
        tmem_ld_wait();
        if (t < D) {
#pragma unroll
          for (int i = 0; i < 32; ++i) out[(c * 32 + i) * D + t] = __uint_as_float(v[i]);
        }
      }
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + 128, v);
      tmem_ld_wait();
      if (t < D) out[D * D + t] = __uint_as_float(v[0]);
    }
  } else if (warp == kMomMmaWarp) {
    // drain: every MMA this CTA issued completes before TMEM is freed
    const long long t0 = clock64();
    while (!mbar_try_wait(done, 0))
      if (clock64() - t0 > kWaitLimitCycles) break;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMomMmaWarp) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------- power iteration

// Nodes of more than kChunkRows rows leave one partial (X^T X, column sums)
// per chunk.  Nodes of at least kReduceChunks chunks have them summed into
// chunk 0 here, in chunk order, one float4 of the partial per thread, so that
// the power kernel (one CTA per node) reads a single partial; the power
// kernel sums fewer chunks itself, in the same order.
constexpr int kReduceThreads = 256;
constexpr int kReduceChunks = 4;

template <int D>
__global__ void __launch_bounds__(kReduceThreads)
    pddp_reduce_kernel(float* __restrict__ partials, const int32_t* __restrict__ slot_tab, int N,
                       int C, int depth, int slots, int max_chunks) {
  constexpr int DD = D * D + D;
  static_assert(DD % 4 == 0, "partials are float4 vectors");
  const int q4 = blockIdx.x * kReduceThreads + threadIdx.x;
  const int slot = slot_tab[blockIdx.y], bh = blockIdx.z;
  if (q4 * 4 >= DD) return;
  const Node nd = node_at(N, C, depth, slot);
  const int nchunks = (nd.n + kChunkRows - 1) / kChunkRows;
  if ((nd.n + C - 1) / C <= 1 || nchunks < kReduceChunks) return;
  float4* base = reinterpret_cast<float4*>(partials + (size_t)(bh * slots + slot) * max_chunks * DD);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int ch = 0; ch < nchunks; ++ch) {
    const float4 x = __ldg(base + (size_t)ch * (DD / 4) + q4);
    acc.x += x.x;
    acc.y += x.y;
    acc.z += x.z;
    acc.w += x.w;
  }
  base[q4] = acc;
}

constexpr int kPowThreads = 256;

// One CTA per node.  The D x D covariance is cut into 16 x 16 blocks of
// R = D/16 rows by 4*J = D/16 columns: half-warp h of warp w holds row block
// 2w + h, its lane c the columns [64j + 4c, 64j + 4c + 4) of those rows
// (j < J), all in registers as packed fp32 pairs for every iteration.  A step
// reads J 16-byte pieces of the iterate from shared memory, multiplies with
// packed f32x2 FMAs (R partial dot products per thread), and a reduce-scatter
// across the 16 lanes of the half-warp (shuffles) leaves each row's sum in
// 2 (D = 128) or 4 (D = 64) lanes, one of which stores it.  A lane holds its
// rows in the order i ^ sigma (sigma from its lane bits), so that at every
// halving level it keeps the first half and its partner's second half is the
// same rows: no selects.  The matrix is first divided by
// its trace (largest eigenvalue <= 1, so the iterate cannot overflow), and
// the iterate is normalised after the first step, every kNormEvery steps and
// at the end instead of every step: power iteration's direction does not
// depend on the scale of the iterate, and a node whose covariance sends the
// start vector to zero is caught at the first step (it keeps the start
// vector).  One block barrier per step.  (One covariance row per thread pair
// made every thread read D/2 iterate entries per step: the shared-memory
// pipe, not the FMAs, set the pace of the deep levels.)
template <int D>
__global__ void __launch_bounds__(kPowThreads, 2)
    pddp_power_kernel(const float* __restrict__ partials, const int32_t* __restrict__ slot_tab,
                      int N, int C, int depth, int slots, int max_chunks, int iters,
                      float* __restrict__ nodevec) {
  constexpr int R = D / 16;  // rows per thread: 8 (D = 128) or 4 (D = 64)
  constexpr int J = D / 64;  // 4-column pieces per thread: 2 or 1
  constexpr int kNormEvery = 8;
  constexpr int DD = D * D + D;  // one partial: X^T X, then the column sums
  static_assert(kPowThreads == 256 && (D == 64 || D == 128), "16 x 16 blocks over 8 warps");
  __shared__ __align__(16) float s[D];
  __shared__ __align__(16) float vb[2][D];  // the iterate, double-buffered
  __shared__ float red[kPowThreads / 32];
  __shared__ int lead;
  const int slot = slot_tab[blockIdx.x], bh = blockIdx.y;
  const Node nd = node_at(N, C, depth, slot);
  if ((nd.n + C - 1) / C <= 1) return;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int cb = lane & 15, r0 = (wid * 2 + (lane >> 4)) * R;
  // sigma: the row offset a lane's reduce-scatter ends on; wmask: the lane
  // bits of the plain butterfly levels (the lane stores if they are zero)
  int sigma = 0, wmask = 0;
  {
    int len = R;
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) {
      if (len > 1) {
        len >>= 1;
        if (lane & m) sigma += len;
      } else {
        wmask |= m;
      }
    }
  }
  const float* pc = partials + (size_t)(bh * slots + slot) * max_chunks * DD;
  const int nchunks = (nd.n + kChunkRows - 1) / kChunkRows;
  const int nsum = nchunks >= kReduceChunks ? 1 : nchunks;  // chunk 0 holds the sum, or sum here
  uint64_t cp[R][2 * J];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const ulonglong2 x =
          __ldg(reinterpret_cast<const ulonglong2*>(pc + (r0 + (i ^ sigma)) * D + 64 * j + 4 * cb));
      cp[i][2 * j] = x.x;
      cp[i][2 * j + 1] = x.y;
    }
  float diag = 0.f, colsum = 0.f;
  if (tid < D) {
    colsum = __ldg(pc + D * D + tid);
    diag = __ldg(pc + tid * D + tid);
  }
#pragma unroll 1
  for (int ch = 1; ch < nsum; ++ch) {
    const float* pk = pc + (size_t)ch * DD;
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const ulonglong2 x = __ldg(
            reinterpret_cast<const ulonglong2*>(pk + (r0 + (i ^ sigma)) * D + 64 * j + 4 * cb));
        cp[i][2 * j] = f2_add(cp[i][2 * j], x.x);
        cp[i][2 * j + 1] = f2_add(cp[i][2 * j + 1], x.y);
      }
    if (tid < D) {
      colsum += __ldg(pk + D * D + tid);
      diag += __ldg(pk + tid * D + tid);
    }
  }
  if (tid < D) {
    s[tid] = colsum;
    vb[0][tid] = rsqrtf(static_cast<float>(D));
  }
  __syncthreads();
  const float inv_n = 1.f / static_cast<float>(nd.n);
  // Cov = X^T X - s s^T / n
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const float sa = s[r0 + (i ^ sigma)] * inv_n;
    const uint64_t nsa = f2_pack(-sa, -sa);
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const float4 sb = *reinterpret_cast<const float4*>(s + 64 * j + 4 * cb);
      cp[i][2 * j] = f2_fma(nsa, f2_pack(sb.x, sb.y), cp[i][2 * j]);
      cp[i][2 * j + 1] = f2_fma(nsa, f2_pack(sb.z, sb.w), cp[i][2 * j + 1]);
    }
  }
  // trace of Cov, then Cov / trace
  if (tid < D) diag -= s[tid] * inv_n * s[tid];
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
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int k = 0; k < 2 * J; ++k) cp[i][k] = f2_fma(cp[i][k], itr2, 0ull);
  const bool writer = (lane & wmask) == 0;
  int cur = 0;
  for (int it = 0; it < iters; ++it) {
    ulonglong2 vv[J];
#pragma unroll
    for (int j = 0; j < J; ++j)
      vv[j] = *reinterpret_cast<const ulonglong2*>(vb[cur] + 64 * j + 4 * cb);
    float acc[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      uint64_t a2 = 0ull;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        a2 = f2_fma(cp[i][2 * j], vv[j].x, a2);
        a2 = f2_fma(cp[i][2 * j + 1], vv[j].y, a2);
      }
      float lo, hi;
      f2_unpack(a2, lo, hi);
      acc[i] = lo + hi;
    }
    // reduce-scatter over the half-warp: halve the row set per level while
    // more than one row is left, then plain butterfly sums
    int len = R;
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) {
      if (len > 1) {
        const int half = len >> 1;
#pragma unroll
        for (int k = 0; k < half; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k + half], m);
        len = half;
      } else {
        acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], m);
      }
    }
    if (writer) vb[cur ^ 1][r0 + sigma] = acc[0];
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
  if (wid == 0) {  // largest |v_d|, lowest d on ties
    float bv = -1.f;
    int bi = 0;
#pragma unroll
    for (int k = lane; k < D; k += 32) {
      const float a = fabsf(v[k]);
      if (a > bv) {
        bv = a;
        bi = k;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > bv || (ob == bv && oi < bi)) {
        bv = ob;
        bi = oi;
      }
    }
    if (lane == 0) lead = bi;
  }
  __syncthreads();
  const float sign = v[lead] < 0.f ? -1.f : 1.f;
  float* out = nodevec + (size_t)(bh * slots + slot) * 2 * D;
  if (tid < D) {
    out[tid] = sign * v[tid];
    out[D + tid] = s[tid] * inv_n;  // mean
  }
}

// Power iteration for the depths whose nodes fit one moments chunk (the deep
// levels, thousands of nodes).  The covariance is symmetric, so a node keeps
// only its upper-triangle 8 x 8 blocks, one per thread (136 threads at
// D = 128): half the registers of the full matrix, four nodes per SM instead
// of two.  A step: block (a, b), a <= b, adds B v_b to rows 8a.. and, off the
// diagonal, B^T v_a to rows 8b..; each contribution goes to its own slot of
// a shared array part[row block][column block][8] (every slot written by
// exactly one thread), and thread t < D sums row t's D/8 slots in column-block
// order.  Normalisation, trace scaling and the sign rule as pddp_power_kernel.
template <int D>
constexpr int sym_threads() { return ((D / 8) * (D / 8 + 1) / 2 + 31) / 32 * 32; }

template <int D>
__global__ void __launch_bounds__(sym_threads<D>(), D == 128 ? 4 : 8)
    pddp_power_sym_kernel(const float* __restrict__ partials, const int32_t* __restrict__ slot_tab,
                          int N, int C, int depth, int slots, int max_chunks, int iters,
                          float* __restrict__ nodevec) {
  constexpr int NB = D / 8;                 // block rows
  constexpr int NBLK = NB * (NB + 1) / 2;   // blocks of the upper triangle
  constexpr int T = sym_threads<D>();
  constexpr int kPad = NB * 8 + 8;          // floats per row block of part[] (bank spread)
  constexpr int kNormEvery = 8;
  constexpr int DD = D * D + D;
  static_assert(D == 64 || D == 128, "D must be 64 or 128");
  __shared__ __align__(16) float s[D];
  __shared__ __align__(16) float vb[2][D];  // the iterate, double-buffered
  __shared__ __align__(16) float part[NB * kPad];
  __shared__ float red[T / 32];
  __shared__ int lead;
  const int slot = slot_tab[blockIdx.x], bh = blockIdx.y;
  const Node nd = node_at(N, C, depth, slot);
  if ((nd.n + C - 1) / C <= 1) return;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // this thread's block (a, b): row block a holds the NB - a blocks b = a .. NB-1
  const bool has_blk = tid < NBLK;
  int a = 0, b = 0;
  if (has_blk) {
    int t = tid;
    while (t >= NB - a) {
      t -= NB - a;
      ++a;
    }
    b = a + t;
  }
  const bool diag = a == b;
  const float* pc = partials + (size_t)(bh * slots + slot) * max_chunks * DD;  // one chunk
  uint64_t B[8][4];  // rows 8a + i, columns 8b .. 8b + 7 as packed pairs
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (has_blk) {
      const ulonglong2* r = reinterpret_cast<const ulonglong2*>(pc + (8 * a + i) * D + 8 * b);
      const ulonglong2 x0 = __ldg(r), x1 = __ldg(r + 1);
      B[i][0] = x0.x;
      B[i][1] = x0.y;
      B[i][2] = x1.x;
      B[i][3] = x1.y;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) B[i][k] = 0ull;
    }
  }
  float diag_v = 0.f;
  if (tid < D) {
    s[tid] = __ldg(pc + D * D + tid);
    diag_v = __ldg(pc + tid * D + tid);
    vb[0][tid] = rsqrtf(static_cast<float>(D));
  }
  __syncthreads();
  const float inv_n = 1.f / static_cast<float>(nd.n);
  // Cov = X^T X - s s^T / n
  if (has_blk) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float sa = s[8 * a + i] * inv_n;
      const uint64_t nsa = f2_pack(-sa, -sa);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        B[i][k] = f2_fma(nsa, f2_pack(s[8 * b + 2 * k], s[8 * b + 2 * k + 1]), B[i][k]);
    }
  }
  // trace of Cov, then Cov / trace
  if (tid < D) diag_v -= s[tid] * inv_n * s[tid];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) diag_v += __shfl_xor_sync(0xffffffffu, diag_v, o);
  if (lane == 0) red[wid] = diag_v;
  __syncthreads();
  float tr = 0.f;
#pragma unroll
  for (int i = 0; i < T / 32; ++i) tr += red[i];
  const float inv_tr = tr > 0.f ? 1.f / tr : 1.f;
  const uint64_t itr2 = f2_pack(inv_tr, inv_tr);
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) B[i][k] = f2_fma(B[i][k], itr2, 0ull);
  int cur = 0;
  for (int it = 0; it < iters; ++it) {
    if (has_blk) {
      const ulonglong2 p0 = *reinterpret_cast<const ulonglong2*>(vb[cur] + 8 * b);
      const ulonglong2 p1 = *reinterpret_cast<const ulonglong2*>(vb[cur] + 8 * b + 4);
      const uint64_t vbp[4] = {p0.x, p0.y, p1.x, p1.y};
      float y1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint64_t acc = 0ull;
#pragma unroll
        for (int k = 0; k < 4; ++k) acc = f2_fma(B[i][k], vbp[k], acc);
        float lo, hi;
        f2_unpack(acc, lo, hi);
        y1[i] = lo + hi;
      }
      float* dst = part + a * kPad + b * 8;
      *reinterpret_cast<float4*>(dst) = make_float4(y1[0], y1[1], y1[2], y1[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(y1[4], y1[5], y1[6], y1[7]);
      if (!diag) {
        const float4 q0 = *reinterpret_cast<const float4*>(vb[cur] + 8 * a);
        const float4 q1 = *reinterpret_cast<const float4*>(vb[cur] + 8 * a + 4);
        const float va[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint64_t y2[4] = {0ull, 0ull, 0ull, 0ull};  // columns 8b + 2k, 8b + 2k + 1
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint64_t vi = f2_pack(va[i], va[i]);
#pragma unroll
          for (int k = 0; k < 4; ++k) y2[k] = f2_fma(B[i][k], vi, y2[k]);
        }
        float z[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) f2_unpack(y2[k], z[2 * k], z[2 * k + 1]);
        float* dst2 = part + b * kPad + a * 8;
        *reinterpret_cast<float4*>(dst2) = make_float4(z[0], z[1], z[2], z[3]);
        *reinterpret_cast<float4*>(dst2 + 4) = make_float4(z[4], z[5], z[6], z[7]);
      }
    }
    __syncthreads();
    if (tid < D) {
      const float* src = part + (tid >> 3) * kPad + (tid & 7);
      float y = 0.f;
#pragma unroll
      for (int c = 0; c < NB; ++c) y += src[c * 8];
      vb[cur ^ 1][tid] = y;
    }
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
      for (int i = 0; i < T / 32; ++i) norm2 += red[i];
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
  if (wid == 0) {  // largest |v_d|, lowest d on ties
    float bv = -1.f;
    int bi = 0;
#pragma unroll
    for (int k = lane; k < D; k += 32) {
      const float x = fabsf(v[k]);
      if (x > bv) {
        bv = x;
        bi = k;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > bv || (ob == bv && oi < bi)) {
        bv = ob;
        bi = oi;
      }
    }
    if (lane == 0) lead = bi;
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

constexpr int kProjThreads = 32;  // one warp per CTA: a finished warp's slot is refilled at once

template <int D>
constexpr int proj_smem_bytes() { return (kProjThreads / 32) * 32 * D * 2; }

// One warp per 32 consecutive positions of a head.  The warp copies its 32
// rows into shared memory with 16-byte cp.async (all loads in flight at
// once); each half-warp then takes every other row, its lane hl the elements
// [hl*D/16, (hl+1)*D/16) of each, forms the partial (x - mu).v of its 16
// rows with the node's mean and direction in registers, and a butterfly
// transpose reduction over the half-warp leaves one row's projection per
// lane.
template <int D, int C>
__global__ void __launch_bounds__(kProjThreads)
    pddp_project_kernel(const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ perm,
                        int N, int depth, int slots, const float* __restrict__ nodevec,
                        uint64_t* __restrict__ keys, int layout, int H, int head0) {
  // C is a template argument: the node walk of every position divides by it
  constexpr int kSegs = D * 2 / 16;  // 16-byte chunks per row
  static_assert(D == 64 || D == 128, "D must be 64 or 128");
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
  // half-warp hp takes rows 2i + hp (i < 16); its lane hl the elements
  // [hl*E2, hl*E2 + E2) of each (one 16-byte (D = 128) or 8-byte shared load)
  constexpr int E2 = D / 16;
  const int hl = lane & 15, hp = lane >> 4;
  float acc[16];
  int cached = -1;
  float vs[E2], ms[E2];
#pragma unroll
  for (int e = 0; e < E2; ++e) vs[e] = ms[e] = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = 2 * i + hp;
    const int sr = __shfl_sync(0xffffffffu, slot, r);
    acc[i] = 0.f;
    if (sr >= 0) {
      if (sr != cached) {
        const float* vec = nodevec + (size_t)(bh * slots + sr) * 2 * D + hl * E2;
#pragma unroll
        for (int e = 0; e < E2; ++e) {
          vs[e] = __ldg(vec + e);
          ms[e] = __ldg(vec + D + e);
        }
        cached = sr;
      }
      const __nv_bfloat162* x =
          reinterpret_cast<const __nv_bfloat162*>(buf + r * D * 2 + hl * E2 * 2);
      float t = 0.f;
#pragma unroll
      for (int h = 0; h < E2 / 2; ++h) {
        const float2 f = __bfloat1622float2(x[h]);
        t = fmaf(f.x - ms[2 * h], vs[2 * h], t);
        t = fmaf(f.y - ms[2 * h + 1], vs[2 * h + 1], t);
      }
      acc[i] = t;
    }
  }
  // transpose reduction over the half-warp: after the step of width w, a lane
  // keeps the w rows whose index has its lane's bit w, summed with its
  // partner's; lane hl ends with row index i = hl, i.e. row 2 hl + hp
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool upper = (hl & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? acc[i] : acc[i + w];
      const float keep = upper ? acc[i + w] : acc[i];
      acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  const int r = 2 * hl + hp;
  const int s_r = __shfl_sync(0xffffffffu, slot, r);
  const int tok_r = __shfl_sync(0xffffffffu, token, r);
  if (s_r >= 0) {
    uint32_t u = __float_as_uint(acc[0]);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // unsigned order == float order
    keys[(size_t)bh * N + p0 + r] = (static_cast<uint64_t>(u) << 32) | static_cast<uint32_t>(tok_r);
  }
}

// ---------------------------------------------------------------- select + partition
//
// Each splitting node finds T, the C*floor(g/2)-th smallest of its keys (keys
// are distinct: the token is the low word), by radix select over 8-bit digits
// from the top, then partitions its positions stably: key <= T left, the rest
// right.  Nodes of more than kSmallNode rows take one CTA each and stream
// their keys from global memory (kUnroll independent loads in flight per
// thread); smaller nodes take one warp each, with the keys in shared memory
// and no block barrier.  A leaf is copied to the output buffer once, at the
// depth where it appears; from then on both buffers hold its final positions.

constexpr int kSmallNode = 1024;
constexpr int kSplitWide = 16384;  // nodes above this many rows split with 1024 threads
constexpr int kSmallWarps = 1;  // nodes (warps) per CTA

template <int kWarps>
__device__ __forceinline__ uint32_t block_scan_incl(uint32_t v, uint32_t* wsum, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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

// Nodes of more than kSmallNode rows: one CTA of kSplitThreads threads each,
// kUnroll keys per thread in flight.  1024 threads for the top depths (a few
// nodes of tens of thousands of rows), 256 below (more nodes, more CTAs per SM).
template <int kSplitThreads, int kUnroll>
__global__ void __launch_bounds__(kSplitThreads)
    pddp_split_kernel(const uint64_t* __restrict__ keys, const int32_t* __restrict__ perm_in,
                      int32_t* __restrict__ perm_out, const int32_t* __restrict__ slot_tab, int N,
                      int C, int depth, unsigned* status) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t wsum[32];
  __shared__ uint32_t sel_digit, sel_below;
  const int slot = slot_tab[blockIdx.x], bh = blockIdx.y;
  const Node nd = node_at(N, C, depth, slot);
  const int g = (nd.n + C - 1) / C;
  if (g <= 1 || nd.n <= kSmallNode) return;  // leaves and small nodes: the warp path
  const int tid = threadIdx.x;
  const int32_t* in = perm_in + (size_t)bh * N + nd.start;
  int32_t* out = perm_out + (size_t)bh * N + nd.start;
  const int n = nd.n, nl = C * (g / 2);
  const uint64_t* kk = keys + (size_t)bh * N + nd.start;
  // radix select of the nl-th smallest key, 8 bits at a time from the top
  uint64_t prefix = 0, mask = 0;
  uint32_t remaining = static_cast<uint32_t>(nl);
  uint64_t T = ~0ull;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = tid; b < 256; b += kSplitThreads) hist[b] = 0;
    if (tid == 0) sel_digit = 256;  // none yet
    __syncthreads();
    for (int i0 = tid; i0 < n; i0 += kUnroll * kSplitThreads) {
      uint64_t k[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = i0 + u * kSplitThreads;
        k[u] = i < n ? kk[i] : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (i0 + u * kSplitThreads < n && (k[u] & mask) == prefix)
          atomicAdd(&hist[(k[u] >> shift) & 255u], 1u);
    }
    __syncthreads();
    uint32_t mine = tid < 256 ? hist[tid] : 0u;
    uint32_t total;
    const uint32_t incl = block_scan_incl<kSplitThreads / 32>(mine, wsum, &total);
    if (tid < 256) {
      const uint32_t below = incl - mine;
      if (below < remaining && remaining <= incl) {
        sel_digit = tid;
        sel_below = below;
      }
    }
    __syncthreads();
    if (sel_digit >= 256u) {  // cannot happen with distinct keys (block-uniform)
      if (tid == 0) atomicOr(status, DEV_BOUNDS);
      return;
    }
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
  // with ballots (no block barrier inside the loop), kUnroll batches of 32
  // positions loaded at a time.
  constexpr int kWarps = kSplitThreads / 32;
  const int lane = tid & 31, w = tid >> 5;
  const int len = (n + kWarps - 1) / kWarps;
  const int lo = min(n, w * len), hi = min(n, lo + len);
  uint32_t nleft = 0;
  for (int b = lo; b < hi; b += 32 * kUnroll) {
    bool left[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = b + 32 * u + lane;
      left[u] = i < hi && kk[i] <= T;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) nleft += __popc(__ballot_sync(0xffffffffu, left[u]));
  }
  __shared__ uint32_t wleft[kWarps];
  if (lane == 0) wleft[w] = nleft;
  __syncthreads();
  uint32_t before_left = 0;
  for (int v = 0; v < w; ++v) before_left += wleft[v];
  uint32_t run_left = before_left, run_right = static_cast<uint32_t>(lo) - before_left;
  const unsigned lt = (1u << lane) - 1u;
  for (int b = lo; b < hi; b += 32 * kUnroll) {
    bool left[kUnroll];
    int32_t val[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = b + 32 * u + lane;
      left[u] = i < hi && kk[i] <= T;
      val[u] = i < hi ? in[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = b + 32 * u + lane;
      const bool valid = i < hi;
      const unsigned ml = __ballot_sync(0xffffffffu, left[u]);
      const unsigned mr = __ballot_sync(0xffffffffu, valid && !left[u]);
      if (valid) {
        const int dst = left[u] ? static_cast<int>(run_left + __popc(ml & lt))
                                : nl + static_cast<int>(run_right + __popc(mr & lt));
        if (dst < n && (left[u] ? dst < nl : dst >= nl))
          out[dst] = val[u];
        else
          atomicOr(status, DEV_BOUNDS);
      }
      run_left += __popc(ml);
      run_right += __popc(mr);
    }
  }
}

// One warp per node of at most kSmallNode rows (and per new leaf, which it
// copies).  The node's keys go to shared memory once; the digit histogram is
// per warp; a lane scans 8 consecutive bins.
__global__ void __launch_bounds__(32 * kSmallWarps)
    pddp_split_small_kernel(const uint64_t* __restrict__ keys, const int32_t* __restrict__ perm_in,
                            int32_t* __restrict__ perm_out, int N, int C, int depth, int slots,
                            unsigned* status) {
  __shared__ uint64_t skeys[kSmallWarps][kSmallNode];
  __shared__ uint32_t shist[kSmallWarps][256];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int slot = blockIdx.x * kSmallWarps + w, bh = blockIdx.y;
  if (slot >= slots) return;  // whole warp
  bool stale = false;
  const Node nd = node_at(N, C, depth, slot, &stale);
  if (nd.n == 0 || stale || nd.n > kSmallNode) return;
  const int32_t* in = perm_in + (size_t)bh * N + nd.start;
  int32_t* out = perm_out + (size_t)bh * N + nd.start;
  const int n = nd.n, g = (n + C - 1) / C;
  if (g <= 1) {  // a leaf appearing at this depth
    for (int i = lane; i < n; i += 32) out[i] = in[i];
    return;
  }
  const int nl = C * (g / 2);
  const uint64_t* kk = keys + (size_t)bh * N + nd.start;
  uint64_t* sk = skeys[w];
  uint32_t* h = shist[w];
  for (int i = lane; i < n; i += 32) sk[i] = kk[i];
  __syncwarp();
  uint64_t prefix = 0, mask = 0, T = ~0ull;
  uint32_t remaining = static_cast<uint32_t>(nl);
  for (int shift = 56; shift >= 0; shift -= 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) h[lane * 8 + e] = 0;
    __syncwarp();
    for (int i = lane; i < n; i += 32) {
      const uint64_t k = sk[i];
      if ((k & mask) == prefix) atomicAdd(&h[(k >> shift) & 255u], 1u);
    }
    __syncwarp();
    uint32_t c[8], tot = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      c[e] = h[lane * 8 + e];
      tot += c[e];
    }
    uint32_t incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    uint32_t below = incl - tot;
    int dsel = -1;
    uint32_t bsel = 0, csel = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (below < remaining && remaining <= below + c[e]) {
        dsel = lane * 8 + e;
        bsel = below;
        csel = c[e];
      }
      below += c[e];
    }
    const unsigned found = __ballot_sync(0xffffffffu, dsel >= 0);
    if (found == 0u) {  // cannot happen with distinct keys
      if (lane == 0) atomicOr(status, DEV_BOUNDS);
      return;
    }
    const int src = __ffs(found) - 1;
    dsel = __shfl_sync(0xffffffffu, dsel, src);
    bsel = __shfl_sync(0xffffffffu, bsel, src);
    csel = __shfl_sync(0xffffffffu, csel, src);
    prefix |= static_cast<uint64_t>(dsel) << shift;
    mask |= 255ull << shift;
    remaining -= bsel;
    if (remaining == csel) {
      T = prefix | ~mask;
      break;
    }
    if (shift == 0) T = prefix;
    __syncwarp();  // every lane has read h before the next pass clears it
  }
  uint32_t run_left = 0, run_right = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int b = 0; b < n; b += 32) {
    const int i = b + lane;
    const bool valid = i < n;
    const bool left = valid && sk[i] <= T;
    const unsigned ml = __ballot_sync(0xffffffffu, left);
    const unsigned mr = __ballot_sync(0xffffffffu, valid && !left);
    if (valid) {
      const int dst = left ? static_cast<int>(run_left + __popc(ml & lt))
                           : nl + static_cast<int>(run_right + __popc(mr & lt));
      if (dst < n && (left ? dst < nl : dst >= nl))
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
  int32_t* table = reinterpret_cast<int32_t*>(base + w.table);
  const int G = (N + C - 1) / C;
  const int depths = depth_count(N, C);

  const size_t total = (size_t)BH * N;
  pddp_init_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(pa, N, BH);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (depths > 0) {
    pddp_table_kernel<<<depths, kTableThreads, 0, stream>>>(N, C, w.max_slots, table);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  const int msmem = MomLayout<D>::kSmem;
  e = cudaFuncSetAttribute(pddp_moments_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           msmem);
  if (e != cudaSuccess) return e;
  const int psmem = 0;  // the power kernel's shared memory is static
  auto project = C == 64 ? pddp_project_kernel<D, 64> : pddp_project_kernel<D, 128>;
  e = cudaFuncSetAttribute(project, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           proj_smem_bytes<D>());
  if (e != cudaSuccess) return e;

  for (int d = 0; d < depths; ++d) {
    const int slots = 1 << d;
    const int chunks = (max_node_rows(N, C, d) + kChunkRows - 1) / kChunkRows;
    const int nsplit = split_count(N, C, d);  // >= 1 below depth_count
    const int32_t* tab = table + (size_t)d * w.max_slots;
    pddp_moments_kernel<D><<<dim3(chunks, nsplit, BH), kMomThreads, msmem, stream>>>(
        q, pa, tab, N, C, d, slots, chunks, partials, status, layout, H, head0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (chunks >= kReduceChunks) {
      constexpr int kQ4 = (D * D + D) / 4;
      pddp_reduce_kernel<D><<<dim3((kQ4 + kReduceThreads - 1) / kReduceThreads, nsplit, BH),
                              kReduceThreads, 0, stream>>>(partials, tab, N, C, d, slots, chunks);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (chunks == 1)  // every node in one chunk: the half-matrix kernel, four nodes per SM
      pddp_power_sym_kernel<D><<<dim3(nsplit, BH), sym_threads<D>(), 0, stream>>>(
          partials, tab, N, C, d, slots, chunks, iters, nodevec);
    else
      pddp_power_kernel<D><<<dim3(nsplit, BH), kPowThreads, psmem, stream>>>(
          partials, tab, N, C, d, slots, chunks, iters, nodevec);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    project<<<dim3((N + kProjThreads - 1) / kProjThreads, BH), kProjThreads, proj_smem_bytes<D>(),
              stream>>>(q, pa, N, d, slots, nodevec, keys, layout, H, head0);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (max_node_rows(N, C, d) > kSmallNode) {
      if (max_node_rows(N, C, d) > kSplitWide)
        pddp_split_kernel<1024, 8><<<dim3(nsplit, BH), 1024, 0, stream>>>(keys, pa, pb, tab, N, C,
                                                                          d, status);
      else
        pddp_split_kernel<256, 4><<<dim3(nsplit, BH), 256, 0, stream>>>(keys, pa, pb, tab, N, C, d,
                                                                        status);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    pddp_split_small_kernel<<<dim3((slots + kSmallWarps - 1) / kSmallWarps, BH),
                              32 * kSmallWarps, 0, stream>>>(keys, pa, pb, N, C, d, slots, status);
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
