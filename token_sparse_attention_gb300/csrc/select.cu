// Exact group-mass selection (the anchor step's second pass) and per-group
// top-K.
//
// The selector's second pass recomputes the QK scores, recovers the exact
// attention probabilities exp(s - lse) from the first pass's log-sum-exp,
// sums them over each query group and keeps the K KV tokens of largest group
// mass (ai.info AI summary, "Methodology in Plain English"; agihunt.info
// summary, paragraph on the selection objective).
//
// group_mass_kernel: one CTA per (head, group).  The scores are computed
// transposed, S^T = K_tile Q_g^T (M = 128 KV rows, N = C queries), so that
// TMEM lane t holds KV row t and each thread sums its row's C probabilities
// in registers: no cross-thread reduction and no running max (lse is known).
//   warps 0-3  exp + sum, one KV row per thread, write mass[g, j]
//   warp 4     producer: gather4 of the group's Q rows, TMA tiles of K
//   warp 5     TMEM allocation and MMA issue (one elected lane)
// Two K stages and two TMEM score buffers let the MMA of tile j+1 run while
// tile j is exponentiated.
//
// Top-K: one CTA per (head, group) row of masses, selecting on the float bit
// pattern (masses are >= 0, so unsigned order of the bits is numeric order),
// ties to the lower index, indices written ascending.  Within the anchor step
// the mass kernel also counts each row's masses by their top 12 bits; from
// that histogram topk_hist_kernel knows the bucket of the K-th largest mass
// before it reads the row, and selects in one read of the masses.  (The
// second pass fuses group aggregation with top-K: ai.info AI summary,
// "Methodology in Plain English".  The masses still go through HBM here: one
// row of N fp32 masses does not fit in shared memory.)
// topk_kernel (no histogram) runs a 12+12+8-bit radix select and an ordered
// compaction: four reads of the row.
#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int kMassThreads = 192;
// Histogram digit of a mass: the float's top 12 bits (sign, exponent, three
// mantissa bits; masses are >= 0, so the digit grows with the mass), clamped
// to the last bin (kMassHistBins in internal.h).
constexpr int kHistBins = kMassHistBins;
__device__ __forceinline__ uint32_t mass_digit(uint32_t bits) {
  return min(bits >> 20, static_cast<uint32_t>(kHistBins - 1));
}

// GP groups per CTA: 1, or 2 sibling C = 64 groups sharing one 128-query
// tile (a 64-column MMA costs nearly as much as a 128-column one, and the K
// tiles are then loaded once for both groups); each group keeps its own mass
// row and histogram.
template <int D, int CQ, int GP>
struct MassLayout {
  static constexpr int kSub = D / 64;
  static constexpr int kQSub = CQ * 128;        // CQ rows x 128 B
  static constexpr int kKSub = 128 * 128;       // 128 rows x 128 B
  static constexpr int kQ = 0;
  static constexpr int kK0 = kSub * kQSub;      // 1024-aligned (CQ multiple of 8)
  static constexpr int kKStage = kSub * kKSub;
  // the bias step's operands: a ones tile (128 KV rows x 16) and the
  // queries' bias parts (CQ rows x 16), K-major without swizzle, 8-row x
  // 16-byte core matrices, the two K halves of an 8-row group adjacent
  static constexpr int kOnes = kK0 + 2 * kKStage;
  static constexpr int kQb = kOnes + 128 * 32;
  static constexpr int kHist = kQb + CQ * 32;            // mass histogram (kHistBins words)
  static constexpr int kBars = kHist + GP * kHistBins * 4;
  static constexpr int kUsed = kBars + 128 + 1024;
  // at most two CTAs per SM (TMEM: 2 x 256 columns)
  static constexpr int kSmem = kUsed > 80 * 1024 ? kUsed : 80 * 1024;
  static_assert(2 * (kSmem + 1024) <= 228 * 1024, "two CTAs per SM");
  static constexpr int kTmemCols = 2 * CQ < 32 ? 32 : 2 * CQ;
};

__device__ __forceinline__ bool warp_wait_m(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                            unsigned* status) {
  bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void drain_wait_m(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

template <int D, int CQ, int GP>
__global__ void __launch_bounds__(kMassThreads, 2)
    group_mass_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const MassArgs a) {
  using L = MassLayout<D, CQ, GP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sq = smem + L::kQ;
  uint8_t* sk = smem + L::kK0;
  uint8_t* sones = smem + L::kOnes;
  uint8_t* sqb = smem + L::kQb;
  uint32_t* shist = reinterpret_cast<uint32_t*>(smem + L::kHist);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;   // [2]
  uint64_t* k_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;   // [2]
  uint64_t* s_empty = bars + 7;  // [2]
  uint64_t* done = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  const int g = blockIdx.x * GP;             // the CTA's first group
  const int ng = min(GP, a.G - g);           // its groups (the last CTA may have one)
  const int qrows = ng * a.C;                // their query rows, adjacent in perm
  const int hc = blockIdx.y;          // head within the chunk
  const int bh = a.head0 + hc;        // global head
  const int ntiles = (a.N + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full + s, 1);
      mbar_init(k_empty + s, 1);
      mbar_init(s_full + s, 1);
      mbar_init(s_empty + s, 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  // The bias of query p enters the scores through the MMA: one more K step of
  // 16 multiplies a ones tile (KV rows) by the query's -lse/scale, split into
  // three bf16 parts whose sum is exact to ~2^-24 relative, so that the exp
  // warps compute exp2(scale*log2(e) * S') with S' = q.k - lse/scale straight
  // from TMEM.  Padding slots get a large negative bias (probability 0).
  if (threadIdx.x < 128) {
    const int r = threadIdx.x;
    const int core = ((r >> 3) * 2) * 128 + (r & 7) * 16;  // K half 0; half 1 at +128
    const __nv_bfloat16 one = __float2bfloat16_rn(1.f), zero = __float2bfloat16_rn(0.f);
    __nv_bfloat162 v01 = __halves2bfloat162(one, one), v23 = __halves2bfloat162(one, zero);
    uint4 w0;
    w0.x = *reinterpret_cast<uint32_t*>(&v01);
    w0.y = *reinterpret_cast<uint32_t*>(&v23);
    w0.z = 0u;
    w0.w = 0u;
    *reinterpret_cast<uint4*>(sones + core) = w0;
    *reinterpret_cast<uint4*>(sones + core + 128) = make_uint4(0u, 0u, 0u, 0u);
    if (r < CQ) {
      constexpr float kLog2e = 1.4426950408889634f;
      const int p = (r < qrows) ? __ldg(a.perm + (static_cast<size_t>(bh) * a.G + g) * a.C + r) : -1;
      float b = -1e30f;
      if (p >= 0 && p < a.N)
        b = -(__ldg(a.lse + static_cast<size_t>(bh) * a.N + p) * kLog2e) / a.scale_log2;
      const __nv_bfloat16 h0 = __float2bfloat16_rn(b);
      const float r1 = b - __bfloat162float(h0);
      const __nv_bfloat16 h1 = __float2bfloat16_rn(r1);
      const __nv_bfloat16 h2 = __float2bfloat16_rn(r1 - __bfloat162float(h1));
      __nv_bfloat162 p01 = __halves2bfloat162(h0, h1), p23 = __halves2bfloat162(h2, zero);
      uint4 wb;
      wb.x = *reinterpret_cast<uint32_t*>(&p01);
      wb.y = *reinterpret_cast<uint32_t*>(&p23);
      wb.z = 0u;
      wb.w = 0u;
      *reinterpret_cast<uint4*>(sqb + core) = wb;
      *reinterpret_cast<uint4*>(sqb + core + 128) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();  // generic writes -> tensor-core operand reads
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int32_t* perm_g = a.perm + (static_cast<size_t>(bh) * a.G + g) * a.C;
    const RowMap rm = row_map(a.layout, a.H, a.N, bh);  // rows of q in either layout
    bool bad = false;
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_expect_tx(q_full, L::kSub * L::kQSub);
    }
    __syncwarp();
    for (int r4 = lane; r4 < CQ / 4; r4 += 32) {
      int r[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int p = 4 * r4 + i;
        int t = (p < qrows) ? __ldg(perm_g + p) : 0;
        if (t < 0) t = 0;
        if (t >= a.N) { bad = true; t = 0; }
        r[i] = rm.rbase + t * rm.rstride;
      }
      for (int s = 0; s < L::kSub; ++s)
        tma_gather4(sq + s * L::kQSub + r4 * 4 * 128, &tq, s * 64, r[0], r[1], r[2], r[3], q_full);
    }
    if (bad) atomicOr(a.status, DEV_BOUNDS);
    // K tiles: the whole warp runs the loop, an elected lane issues (a
    // lane-0-only branch issues TMA and MMA instructions much more slowly)
    int issued = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      if (j >= 2 && !warp_wait_m(k_empty + st, ((j >> 1) - 1) & 1, abort_flag, a.status)) break;
      if (elect_one()) {
        mbar_expect_tx(k_full + st, L::kKStage);
        for (int s = 0; s < L::kSub; ++s)
          tma_load_4d(sk + st * L::kKStage + s * L::kKSub, &tk, s * 64, j * 128, bh % a.H,
                      bh / a.H, k_full + st);
      }
      ++issued;
    }
    if (*abort_flag) {
      for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
        drain_wait_m(k_full + (j & 1), (j >> 1) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // whole warp in the loop, one elected lane issues each tile's MMAs
    constexpr uint32_t idesc = idesc_bf16(128, CQ, false, false);
    const uint32_t q_addr = smem_u32(sq), k_addr = smem_u32(sk);
    const uint64_t ones_desc = sdesc_none(smem_u32(sones), 128, 256);
    const uint64_t qb_desc = sdesc_none(smem_u32(sqb), 128, 256);
    bool ok = warp_wait_m(q_full, 0, abort_flag, a.status);
    for (int j = 0; ok && j < ntiles; ++j) {
      const int st = j & 1;
      if (!warp_wait_m(k_full + st, (j >> 1) & 1, abort_flag, a.status)) break;
      if (j >= 2 && !warp_wait_m(s_empty + st, ((j >> 1) - 1) & 1, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t kb = k_addr + st * L::kKStage;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * L::kKSub + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * L::kQSub + (kk & 3) * 32;
          umma_ss(tmem + st * CQ, sdesc_sw128(kb + ko, 16, 1024), sdesc_sw128(q_addr + qo, 16, 1024),
                  idesc, kk > 0);
        }
        umma_ss(tmem + st * CQ, ones_desc, qb_desc, idesc, 1u);  // + bias of each query
        umma_commit(s_full + st);
        umma_commit(k_empty + st);
      }
    }
    if (elect_one()) umma_commit(done);
    __syncwarp();
    drain_wait_m(done, 0);
  } else {
    // ------------------------------------------------------------ exp + sum
    const int t = threadIdx.x;  // 0..127: KV row within the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    if (a.hist != nullptr)
      for (int b = t; b < GP * kHistBins; b += 128) shist[b] = 0;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const float sl2 = a.scale_log2;
    float* mass_row = a.mass + (static_cast<size_t>(hc) * a.G + g) * a.N;
    constexpr int kCols = CQ / GP;  // score columns (queries) of one group
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      if (!warp_wait_m(s_full + st, (j >> 1) & 1, abort_flag, a.status)) break;
      tc_fence_after();
      float acc[GP];
#pragma unroll
      for (int gi = 0; gi < GP; ++gi) acc[gi] = 0.f;
#pragma unroll
      for (int c = 0; c < CQ / 32; ++c) {
        uint32_t s[32];
        tmem_ld32(tmem + st * CQ + lane_off + c * 32, s);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[(c * 32) / kCols] += ex2(__uint_as_float(s[i]) * sl2);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + st);
      const int jrow = j * 128 + t;
      if (jrow < a.N) {
#pragma unroll
        for (int gi = 0; gi < GP; ++gi) {
          if (gi < ng) {
            mass_row[static_cast<size_t>(gi) * a.N + jrow] = acc[gi];
            if (a.hist != nullptr)
              atomicAdd(&shist[gi * kHistBins + mass_digit(__float_as_uint(acc[gi]))], 1u);
          }
        }
      }
    }
    if (a.hist != nullptr) {
      asm volatile("bar.sync 1, 128;" ::: "memory");
      uint32_t* hist_row = a.hist + (static_cast<size_t>(hc) * a.G + g) * kHistBins;
      for (int b = t; b < ng * kHistBins; b += 128) hist_row[b] = shist[b];
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, L::kTmemCols);
}

template <int D, int CQ, int GP>
cudaError_t launch_mass_one(const CUtensorMap* tq, const CUtensorMap* tk, const MassArgs& a,
                            int heads, cudaStream_t stream) {
  auto kern = group_mass_kernel<D, CQ, GP>;
  const int smem = MassLayout<D, CQ, GP>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3((a.G + GP - 1) / GP, heads), kMassThreads, smem, stream>>>(*tq, *tk, a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- top-K

constexpr int kTopkThreads = 1024;
// Candidate capacity of the one-read path: rows whose threshold bucket holds
// more masses than this (ties en masse, degenerate inputs) take the
// multi-pass path instead.
constexpr int kCandCap = 4096;

// Inclusive scan over the block of a packed value; returns the block total in *total.
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = warp > 0 ? warp_sums[warp - 1] : 0u;
  *total = warp_sums[31];
  __syncthreads();
  return v + before;
}

// Block sum of acc, stored to *dst by thread 0 (every thread must call).
__device__ __forceinline__ void block_sum_store(float acc, float* red, float* dst) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = red[threadIdx.x];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) *dst = v;
  }
}

// Number of entries of the ascending array a[0, n) below x.
__device__ __forceinline__ uint32_t count_below(const uint32_t* a, uint32_t n, uint32_t x) {
  uint32_t lo = 0, hi = n;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// One row, multi-pass: radix select of the K-th largest key in 12+12+8-bit
// digits (three reads of the row), then one ordered compaction (a fourth
// read) that keeps every larger key and the lowest-index ties.  hist holds
// 4096 words, scal 2.
__device__ void topk_row_multipass(const uint32_t* __restrict__ keys, int n, int K,
                                   int32_t* __restrict__ out, float* retained_row, unsigned* status,
                                   uint32_t* hist, uint32_t* warp_sums, uint32_t* scal,
                                   float* red) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, prefix_mask = 0, remaining = static_cast<uint32_t>(K);
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
#pragma unroll
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const int nb = 1 << widths[pass];
    for (int b = tid; b < nb; b += kTopkThreads) hist[b] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      const uint32_t k = __ldg(keys + i);
      if ((k & prefix_mask) == prefix) atomicAdd(&hist[(k >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // thread t owns the bins [per*t, per*t + per) counted from the TOP digit down
    const int per = nb / kTopkThreads > 0 ? nb / kTopkThreads : 1;
    uint32_t mine = 0;
    const int first = nb - 1 - per * tid;  // highest bin of this thread
    if (per * tid < nb)
      for (int q = 0; q < per; ++q) mine += hist[first - q];
    uint32_t total;
    const uint32_t incl = block_inclusive_scan(mine, warp_sums, &total);
    uint32_t above = incl - mine;  // count in higher bins
    if (per * tid < nb) {
      for (int q = 0; q < per; ++q) {
        const uint32_t c = hist[first - q];
        if (above < remaining && remaining <= above + c) {
          scal[0] = static_cast<uint32_t>(first - q);
          scal[1] = above;
        }
        above += c;
      }
    }
    __syncthreads();
    prefix |= scal[0] << shift;
    prefix_mask |= static_cast<uint32_t>(nb - 1) << shift;
    remaining -= scal[1];
    __syncthreads();
  }
  // prefix == the K-th largest key; take every larger key and the first
  // `remaining` keys equal to it, in ascending index order.
  const uint32_t T = prefix;
  const uint32_t need_eq = remaining;
  uint32_t run_gt = 0, run_eq = 0;
  float acc = 0.f;
  for (int base = 0; base < n; base += kTopkThreads) {
    const int i = base + tid;
    uint32_t k = 0;
    bool gt = false, eq = false;
    if (i < n) {
      k = __ldg(keys + i);
      gt = k > T;
      eq = k == T;
    }
    const uint32_t packed = (gt ? (1u << 16) : 0u) | (eq ? 1u : 0u);
    uint32_t total;
    const uint32_t incl = block_inclusive_scan(packed, warp_sums, &total);
    const uint32_t excl = incl - packed;
    const uint32_t gt_before = run_gt + (excl >> 16);
    const uint32_t eq_before = run_eq + (excl & 0xFFFFu);
    if (gt || (eq && eq_before < need_eq)) {
      const uint32_t pos = gt_before + min(eq_before, need_eq);
      if (pos < static_cast<uint32_t>(K)) {
        out[pos] = i;
        acc += __uint_as_float(k);
      } else {
        atomicOr(status, DEV_BOUNDS);
      }
    }
    run_gt += total >> 16;
    run_eq += total & 0xFFFFu;
  }
  if (retained_row != nullptr) block_sum_store(acc, red, retained_row);
}

__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ mass, int n, int K, int32_t* __restrict__ idx,
                float* __restrict__ retained, unsigned* status) {
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t scal[2];
  __shared__ float red[32];
  const size_t row = blockIdx.x;
  topk_row_multipass(reinterpret_cast<const uint32_t*>(mass + row * n), n, K, idx + row * K,
                     retained ? retained + row : nullptr, status, hist, warp_sums, scal, red);
}

// Dynamic shared memory of topk_hist_kernel, in 32-bit words.
__host__ __device__ constexpr int topk_hist_words(int K) { return 72 + 1024 + K + 2 * kCandCap; }

// One row per CTA, given the row's digit histogram (mass_digit counts).
//  1. From the histogram: the digit d of the K-th largest mass and the count A
//     of masses with a larger digit; the M masses of digit d are candidates.
//  2. One read of the row: indices of digit > d go, in order, to above[0, A);
//     candidates (key, index), in order, to ckey/cidx.
//  3. Radix select over the candidates' 20 low bits (two 10-bit digits) gives
//     the K-th largest key T and how many keys equal to T to keep; the kept
//     candidates are compacted in order (larger keys, then the lowest-index
//     ties).
//  4. The two ascending index lists are merged into the output.
// A row whose bucket exceeds kCandCap, whose digit is the clamped top one, or
// whose masses do not match the histogram takes topk_row_multipass.
__global__ void __launch_bounds__(kTopkThreads, 2)
    topk_hist_kernel(const float* __restrict__ mass, const uint32_t* __restrict__ hist, int n,
                     int K, int32_t* __restrict__ idx, float* __restrict__ retained,
                     unsigned* status) {
  extern __shared__ uint32_t tsm[];
  uint32_t* warp_sums = tsm;                        // 32
  uint32_t* scal = tsm + 32;                        // 8
  float* red = reinterpret_cast<float*>(tsm + 40);  // 32
  uint32_t* h = tsm + 72;                           // 1024 (and 4096 for the fallback)
  uint32_t* above = h + 1024;                       // K
  uint32_t* ckey = above + K;                       // kCandCap
  uint32_t* cidx = ckey + kCandCap;                 // kCandCap

  const int tid = threadIdx.x;
  const size_t row = blockIdx.x;
  const uint32_t* keys = reinterpret_cast<const uint32_t*>(mass + row * n);
  int32_t* out = idx + row * K;
  float* ret_row = retained ? retained + row : nullptr;
  const uint32_t uK = static_cast<uint32_t>(K);

  // 1. threshold digit (two bins per thread, counted from the top)
  const uint32_t* hrow = hist + row * kHistBins;
  static_assert(2 * kTopkThreads >= kHistBins, "two bins per thread cover the histogram");
  const int first = kHistBins - 1 - 2 * tid;  // < 0 for the threads past the last bin
  const uint32_t c0 = first >= 0 ? hrow[first] : 0u, c1 = first >= 1 ? hrow[first - 1] : 0u;
  if (tid == 0) {
    scal[0] = kHistBins;  // not found
    scal[1] = 0;
  }
  uint32_t total;
  const uint32_t incl = block_inclusive_scan(c0 + c1, warp_sums, &total);
  const uint32_t ab = incl - (c0 + c1);
  if (ab < uK && uK <= ab + c0) {
    scal[0] = first;
    scal[1] = ab;
  } else if (ab + c0 < uK && uK <= ab + c0 + c1) {
    scal[0] = first - 1;
    scal[1] = ab + c0;
  }
  __syncthreads();
  const uint32_t d = scal[0], A = scal[1];
  const uint32_t M = d < kHistBins ? hrow[d] : 0u;
  bool fast = d < kHistBins - 1 && M <= kCandCap && total == static_cast<uint32_t>(n);

  // 2. one read of the row, eight contiguous masses per thread per chunk (two
  // 16-byte loads in flight per thread)
  float acc = 0.f;
  if (fast) {
    const bool vec = (reinterpret_cast<uintptr_t>(keys) & 15) == 0;
    constexpr int kPer = 8;
    auto load = [&](int i0, uint32_t* u) {
      if (vec && i0 + kPer - 1 < n) {
        const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(keys + i0));
        const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(keys + i0 + 4));
        u[0] = v0.x;
        u[1] = v0.y;
        u[2] = v0.z;
        u[3] = v0.w;
        u[4] = v1.x;
        u[5] = v1.y;
        u[6] = v1.z;
        u[7] = v1.w;
      } else {
#pragma unroll
        for (int e = 0; e < kPer; ++e) u[e] = i0 + e < n ? __ldg(keys + i0 + e) : 0u;
      }
    };
    constexpr int kChunk = kPer * kTopkThreads;
    // digit > d  <=>  bits >= hiT;  digit == d  <=>  loT <= bits < hiT (d is
    // below the clamped top digit on this path); positions past n load 0 and
    // are excluded only in the last, partial chunk
    const uint32_t loT = d << 20, hiT = (d + 1u) << 20;
    uint32_t run_a = 0, run_c = 0;
    for (int base = 0; base < n; base += kChunk) {
      const int i0 = base + kPer * tid;
      const bool tail = base + kChunk > n;
      uint32_t cur[kPer];
      load(i0, cur);
      uint32_t na = 0, nge = 0;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        const bool valid = !tail || i0 + e < n;
        na += (valid && cur[e] >= hiT) ? 1u : 0u;
        nge += (valid && cur[e] >= loT) ? 1u : 0u;
      }
      const uint32_t packed = (na << 16) | (nge - na);
      uint32_t tot;
      const uint32_t excl = block_inclusive_scan(packed, warp_sums, &tot) - packed;
      uint32_t pa = run_a + (excl >> 16), pc = run_c + (excl & 0xFFFFu);
      if (nge != 0) {
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          if (cur[e] < loT || (tail && i0 + e >= n)) continue;
          if (cur[e] >= hiT) {
            if (pa < A) above[pa] = static_cast<uint32_t>(i0 + e);
            ++pa;
            acc += __uint_as_float(cur[e]);
          } else {
            if (pc < M) {
              ckey[pc] = cur[e];
              cidx[pc] = static_cast<uint32_t>(i0 + e);
            }
            ++pc;
          }
        }
      }
      run_a += tot >> 16;
      run_c += tot & 0xFFFFu;
    }
    // block-uniform: the histogram must describe exactly these masses
    fast = run_a == A && run_c == M;
  }
  __syncthreads();
  if (!fast) {
    topk_row_multipass(keys, n, K, out, ret_row, status, h, warp_sums, scal, red);
    return;
  }

  // 3. the (K - A)-th largest candidate key, two 10-bit digits below d
  uint32_t pref = d << 20, pmask = 0xFFF00000u, R = uK - A;
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    h[tid] = 0;
    __syncthreads();
    for (uint32_t c = tid; c < M; c += kTopkThreads) {
      const uint32_t u = ckey[c];
      if ((u & pmask) == pref) atomicAdd(&h[(u >> shift) & 1023u], 1u);
    }
    __syncthreads();
    const uint32_t bin = 1023u - tid;
    const uint32_t mine = h[bin];
    uint32_t tot;
    const uint32_t below = block_inclusive_scan(mine, warp_sums, &tot) - mine;
    if (below < R && R <= below + mine) {
      scal[2] = bin;
      scal[3] = below;
    }
    __syncthreads();
    pref |= scal[2] << shift;
    pmask |= 1023u << shift;
    R -= scal[3];
    __syncthreads();
  }
  // keep candidates > T and the first need_eq equal to T, compacted in place
  // (a kept candidate moves to a position no later than its own)
  const uint32_t T = pref, need_eq = R;
  uint32_t run_gt = 0, run_eq = 0;
  for (uint32_t base = 0; base < M; base += kTopkThreads) {
    const uint32_t c = base + tid;
    uint32_t u = 0, id = 0;
    bool gt = false, eq = false;
    if (c < M) {
      u = ckey[c];
      id = cidx[c];
      gt = u > T;
      eq = u == T;
    }
    const uint32_t packed = (gt ? (1u << 16) : 0u) | (eq ? 1u : 0u);
    uint32_t tot;
    const uint32_t excl = block_inclusive_scan(packed, warp_sums, &tot) - packed;
    const uint32_t gb = run_gt + (excl >> 16), eb = run_eq + (excl & 0xFFFFu);
    if (gt || (eq && eb < need_eq)) {
      cidx[gb + min(eb, need_eq)] = id;
      acc += __uint_as_float(u);
    }
    run_gt += tot >> 16;
    run_eq += tot & 0xFFFFu;
  }
  __syncthreads();

  // 4. merge the ascending lists above[0, A) and cidx[0, Rk) into out[0, K)
  // The kept candidates go to their final slots (binary search in the above
  // list) and mark them in a bitmap over out; every other slot p then takes
  // above[p - (marked slots before p)], found from per-word prefix counts.
  const uint32_t Rk = uK - A;
  if (run_gt + min(run_eq, need_eq) != Rk) atomicOr(status, DEV_BOUNDS);  // cannot happen
  const uint32_t nw = (uK + 31) / 32;  // <= kCandCap / 2 whenever this path runs
  uint32_t* bits = ckey;               // the candidate keys are no longer needed
  uint32_t* wpre = ckey + nw;
  for (uint32_t w = tid; w < nw; w += kTopkThreads) bits[w] = 0;
  __syncthreads();
  for (uint32_t q = tid; q < Rk; q += kTopkThreads) {
    const uint32_t x = cidx[q];
    const uint32_t f = q + count_below(above, A, x);
    out[f] = static_cast<int32_t>(x);
    atomicOr(&bits[f >> 5], 1u << (f & 31));
  }
  __syncthreads();
  uint32_t run = 0;
  for (uint32_t base = 0; base < nw; base += kTopkThreads) {
    const uint32_t w = base + tid;
    const uint32_t c = w < nw ? static_cast<uint32_t>(__popc(bits[w])) : 0u;
    uint32_t tot;
    const uint32_t incl = block_inclusive_scan(c, warp_sums, &tot);
    if (w < nw) wpre[w] = run + incl - c;
    run += tot;
  }
  __syncthreads();
  for (uint32_t pos = tid; pos < uK; pos += kTopkThreads) {
    const uint32_t word = bits[pos >> 5], bit = 1u << (pos & 31);
    if ((word & bit) == 0u)
      out[pos] = static_cast<int32_t>(
          above[pos - (wpre[pos >> 5] + static_cast<uint32_t>(__popc(word & (bit - 1u))))]);
  }
  if (ret_row != nullptr) block_sum_store(acc, red, ret_row);
}
}  // namespace

cudaError_t launch_group_mass(int D, const CUtensorMap* tq, const CUtensorMap* tk,
                              const MassArgs& a, int heads, cudaStream_t stream) {
  // C = 64, D = 64: two sibling groups per CTA (at D = 128 the paired
  // layout's shared memory would allow only one CTA per SM)
  if (D == 128 && a.C == 128) return launch_mass_one<128, 128, 1>(tq, tk, a, heads, stream);
  if (D == 128 && a.C == 64) return launch_mass_one<128, 64, 1>(tq, tk, a, heads, stream);
  if (D == 64 && a.C == 128) return launch_mass_one<64, 128, 1>(tq, tk, a, heads, stream);
  if (D == 64 && a.C == 64) return launch_mass_one<64, 128, 2>(tq, tk, a, heads, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const float* mass, const uint32_t* hist, int rows, int n, int K,
                        int32_t* idx, float* retained, unsigned* status, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(topk_hist_words(K)) * 4;
  if (hist != nullptr && smem <= 227 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_hist_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    topk_hist_kernel<<<rows, kTopkThreads, smem, stream>>>(mass, hist, n, K, idx, retained, status);
    return cudaGetLastError();
  }
  topk_kernel<<<rows, kTopkThreads, 0, stream>>>(mass, n, K, idx, retained, status);
  return cudaGetLastError();
}

}  // namespace mcs
