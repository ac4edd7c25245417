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
// topk_kernel: one CTA per (head, group) row of masses.  Radix select of the
// K-th largest value on the float bit pattern (masses are >= 0, so unsigned
// order of the bits is numeric order), 12+12+8-bit digits, then one ordered
// compaction pass that keeps every larger value and the lowest-index ties,
// writing indices ascending.
#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int kMassThreads = 192;

template <int D, int CQ>
struct MassLayout {
  static constexpr int kSub = D / 64;
  static constexpr int kQSub = CQ * 128;        // CQ rows x 128 B
  static constexpr int kKSub = 128 * 128;       // 128 rows x 128 B
  static constexpr int kQ = 0;
  static constexpr int kK0 = kSub * kQSub;      // 1024-aligned (CQ multiple of 8)
  static constexpr int kKStage = kSub * kKSub;
  static constexpr int kBias = kK0 + 2 * kKStage;
  static constexpr int kBars = kBias + CQ * 4;
  static constexpr int kUsed = kBars + 128 + 1024;
  // at most two CTAs per SM (TMEM: 2 x 256 columns)
  static constexpr int kSmem = kUsed > 80 * 1024 ? kUsed : 80 * 1024;
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

template <int D, int CQ>
__global__ void __launch_bounds__(kMassThreads, 2)
    group_mass_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const MassArgs a) {
  using L = MassLayout<D, CQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sq = smem + L::kQ;
  uint8_t* sk = smem + L::kK0;
  float* bias = reinterpret_cast<float*>(smem + L::kBias);
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
  const int g = blockIdx.x;
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    const int32_t* perm_g = a.perm + (static_cast<size_t>(bh) * a.G + g) * a.C;
    const int rowbase = bh * a.N;
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
        int t = (p < a.C) ? __ldg(perm_g + p) : 0;
        if (t < 0) t = 0;
        if (t >= a.N) { bad = true; t = 0; }
        r[i] = rowbase + t;
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
          tma_load_3d(sk + st * L::kKStage + s * L::kKSub, &tk, s * 64, j * 128, bh, k_full + st);
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
    constexpr float kLog2e = 1.4426950408889634f;
    if (t < CQ) {
      const int p = (t < a.C) ? __ldg(a.perm + (static_cast<size_t>(bh) * a.G + g) * a.C + t) : -1;
      bias[t] = (p >= 0 && p < a.N) ? __ldg(a.lse + static_cast<size_t>(bh) * a.N + p) * kLog2e
                                    : INFINITY;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const float sl2 = a.scale_log2;
    float* mass_row = a.mass + (static_cast<size_t>(hc) * a.G + g) * a.N;
    const float4* bias4 = reinterpret_cast<const float4*>(bias);
    for (int j = 0; j < ntiles; ++j) {
      const int st = j & 1;
      if (!warp_wait_m(s_full + st, (j >> 1) & 1, abort_flag, a.status)) break;
      tc_fence_after();
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < CQ / 32; ++c) {
        uint32_t s[32];
        tmem_ld32(tmem + st * CQ + lane_off + c * 32, s);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 b = bias4[(c * 32 + i) >> 2];
          acc += ex2(fmaf(__uint_as_float(s[i + 0]), sl2, -b.x));
          acc += ex2(fmaf(__uint_as_float(s[i + 1]), sl2, -b.y));
          acc += ex2(fmaf(__uint_as_float(s[i + 2]), sl2, -b.z));
          acc += ex2(fmaf(__uint_as_float(s[i + 3]), sl2, -b.w));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + st);
      const int jrow = j * 128 + t;
      if (jrow < a.N) mass_row[jrow] = acc;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, L::kTmemCols);
}

template <int D, int CQ>
cudaError_t launch_mass_one(const CUtensorMap* tq, const CUtensorMap* tk, const MassArgs& a,
                            int heads, cudaStream_t stream) {
  auto kern = group_mass_kernel<D, CQ>;
  const int smem = MassLayout<D, CQ>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(a.G, heads), kMassThreads, smem, stream>>>(*tq, *tk, a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- top-K

constexpr int kTopkThreads = 1024;

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

__global__ void __launch_bounds__(kTopkThreads)
    topk_kernel(const float* __restrict__ mass, int n, int K, int32_t* __restrict__ idx,
                float* __restrict__ retained, unsigned* status) {
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t sel_digit, sel_above;
  __shared__ float red[32];

  const int tid = threadIdx.x;
  const size_t row = blockIdx.x;
  const uint32_t* keys = reinterpret_cast<const uint32_t*>(mass + row * n);

  uint32_t prefix = 0, prefix_mask = 0, remaining = static_cast<uint32_t>(K);
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
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
          sel_digit = static_cast<uint32_t>(first - q);
          sel_above = above;
        }
        above += c;
      }
    }
    __syncthreads();
    prefix |= sel_digit << shift;
    prefix_mask |= static_cast<uint32_t>(nb - 1) << shift;
    remaining -= sel_above;
    __syncthreads();
  }
  // prefix == the K-th largest key; take every larger key and the first
  // `remaining` keys equal to it, in ascending index order.
  const uint32_t T = prefix;
  const uint32_t need_eq = remaining;
  uint32_t run_gt = 0, run_eq = 0;
  float acc = 0.f;
  int32_t* out = idx + row * K;
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
  if (retained != nullptr) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((tid & 31) == 0) red[tid >> 5] = acc;
    __syncthreads();
    if (tid < 32) {
      float v = red[tid];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (tid == 0) retained[row] = v;
    }
  }
}

}  // namespace

cudaError_t launch_group_mass(int D, const CUtensorMap* tq, const CUtensorMap* tk,
                              const MassArgs& a, int heads, cudaStream_t stream) {
  if (D == 128 && a.C == 128) return launch_mass_one<128, 128>(tq, tk, a, heads, stream);
  if (D == 128 && a.C == 64) return launch_mass_one<128, 64>(tq, tk, a, heads, stream);
  if (D == 64 && a.C == 128) return launch_mass_one<64, 128>(tq, tk, a, heads, stream);
  if (D == 64 && a.C == 64) return launch_mass_one<64, 64>(tq, tk, a, heads, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_topk(const float* mass, int rows, int n, int K, int32_t* idx, float* retained,
                        unsigned* status, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  topk_kernel<<<rows, kTopkThreads, 0, stream>>>(mass, n, K, idx, retained, status);
  return cudaGetLastError();
}

}  // namespace mcs
