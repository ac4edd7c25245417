// Dense and token-sparse attention forward on tcgen05 tensor cores.
//
// Token-sparse attention: each tile-aligned group of C queries of one head
// attends only to its own K selected KV tokens, gathered by index across
// block boundaries without repacking (MC-Sparse, wispaper.ai, "Token-level
// selection needs tile-aligned query groups"); at reuse steps the cached
// dense-minus-sparse residual is added, at anchors it is recorded
// (wispaper.ai, "Residual correction recovers the discarded tail").  Dense
// attention with row LSE is the selector's first pass (ai.info AI summary,
// "Methodology in Plain English") and the speedup denominator.
//
// One CTA = one 128-row query tile (dense) or one query group (sparse) of one
// head; two CTAs share an SM so that one's softmax overlaps the other's MMAs.
//   warps 0-3  softmax + epilogue: thread t owns query row t = TMEM lane t
//   warp 4     producer: TMA tile loads (dense) or TMA gather4 (sparse)
//   warp 5     TMEM allocation and the single MMA-issuing thread
// TMEM (256 columns): S = Q K^T in columns [0,128) (fp32), overwritten in
// place by P (bf16 pairs) in columns [0,64); O accumulator in [128, 128+D).
// Online softmax in base 2 with lazy rescaling (O is only rescaled when the
// running max grows by more than 8, i.e. P stays <= 256).
#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int BM = 128;  // query rows per CTA (MMA M)
constexpr int BN = 128;  // KV rows per tile (MMA N of QK^T, K of PV)
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct AttnLayout {
  static constexpr int kSub = D / 64;             // 128-byte column sub-tiles per row
  static constexpr int kSubBytes = 128 * 128;     // one sub-tile: 128 rows x 128 B
  static constexpr int kTileBytes = kSub * kSubBytes;
  static constexpr int kQ = 0;
  static constexpr int kK = kTileBytes;
  static constexpr int kV = 2 * kTileBytes;
  static constexpr int kBars = 3 * kTileBytes;
  // At most two CTAs per SM: each holds 256 TMEM columns of the SM's 512.
  static constexpr int kUsed = kBars + 128 + 1024;
  static constexpr int kSmem = kUsed > 80 * 1024 ? kUsed : 80 * 1024;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* status) {
  bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Wait used only while tearing down after an abort: bounded by time alone.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const AttnArgs a) {
  using L = AttnLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sq = smem + L::kQ;
  uint8_t* sk = smem + L::kK;
  uint8_t* sv = smem + L::kV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 2;
  uint64_t* v_full = bars + 3;
  uint64_t* v_empty = bars + 4;
  uint64_t* s_full = bars + 5;
  uint64_t* p_full = bars + 6;
  uint64_t* o_full = bars + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  const int tile = blockIdx.x;
  const int bh = blockIdx.y;
  const int kv_total = (MODE == kDense) ? a.N : a.K;
  const int nkv = (kv_total + BN - 1) / BN;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(o_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;
  const uint32_t tO = tmem + 128;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    int k_issued = 0, v_issued = 0;
    if (MODE == kDense) {
      if (lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        mbar_expect_tx(q_full, L::kTileBytes);
        for (int s = 0; s < L::kSub; ++s)
          tma_load_3d(sq + s * L::kSubBytes, &tq, s * 64, tile * BM, bh, q_full);
        for (int j = 0; j < nkv; ++j) {
          if (j > 0 && !mbar_wait(k_empty, (j - 1) & 1, abort_flag, a.status)) break;
          mbar_expect_tx(k_full, L::kTileBytes);
          for (int s = 0; s < L::kSub; ++s)
            tma_load_3d(sk + s * L::kSubBytes, &tk, s * 64, j * BN, bh, k_full);
          ++k_issued;
          if (j > 0 && !mbar_wait(v_empty, (j - 1) & 1, abort_flag, a.status)) break;
          mbar_expect_tx(v_full, L::kTileBytes);
          for (int s = 0; s < L::kSub; ++s)
            tma_load_3d(sv + s * L::kSubBytes, &tv, s * 64, j * BN, bh, v_full);
          ++v_issued;
        }
        if (*abort_flag) {
          if (k_issued) drain_wait(k_full, (k_issued - 1) & 1);
          if (v_issued) drain_wait(v_full, (v_issued - 1) & 1);
        }
      }
    } else {
      // Sparse: Q rows by perm, K/V rows by idx, 4 rows per gather4; lane l
      // fetches rows 4l..4l+3 of every tile.
      const size_t grp = static_cast<size_t>(bh) * a.G + tile;
      const int32_t* perm_g = a.perm + grp * a.C;
      const int32_t* idx_g = a.idx + grp * a.K;
      const int rowbase = bh * a.N;
      int r[4];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int p = 4 * lane + i;
        int t = (p < a.C) ? __ldg(perm_g + p) : 0;
        if (t < 0) t = 0;  // padding slot of the short last group
        if (t >= a.N) { bad = true; t = 0; }
        r[i] = rowbase + t;
      }
      if (lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        mbar_expect_tx(q_full, L::kTileBytes);
      }
      __syncwarp();
      for (int s = 0; s < L::kSub; ++s)
        tma_gather4(sq + s * L::kSubBytes + lane * 4 * 128, &tq, s * 64, r[0], r[1], r[2], r[3],
                    q_full);
      for (int j = 0; j < nkv; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          int c = j * BN + 4 * lane + i;
          c = c < a.K ? c : a.K - 1;  // tail columns repeat a valid row; masked in softmax
          int t = __ldg(idx_g + c);
          if (t < 0 || t >= a.N) { bad = true; t = 0; }
          r[i] = rowbase + t;
        }
        if (j > 0 && !warp_wait(k_empty, (j - 1) & 1, abort_flag, a.status)) break;
        if (lane == 0) mbar_expect_tx(k_full, L::kTileBytes);
        __syncwarp();
        for (int s = 0; s < L::kSub; ++s)
          tma_gather4(sk + s * L::kSubBytes + lane * 4 * 128, &tk, s * 64, r[0], r[1], r[2], r[3],
                      k_full);
        ++k_issued;
        if (j > 0 && !warp_wait(v_empty, (j - 1) & 1, abort_flag, a.status)) break;
        if (lane == 0) mbar_expect_tx(v_full, L::kTileBytes);
        __syncwarp();
        for (int s = 0; s < L::kSub; ++s)
          tma_gather4(sv + s * L::kSubBytes + lane * 4 * 128, &tv, s * 64, r[0], r[1], r[2], r[3],
                      v_full);
        ++v_issued;
      }
      if (bad) atomicOr(a.status, DEV_BOUNDS);
      if (*abort_flag) {
        if (k_issued) drain_wait(k_full, (k_issued - 1) & 1);
        if (v_issued) drain_wait(v_full, (v_issued - 1) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, false, true);
      const uint32_t q_addr = smem_u32(sq), k_addr = smem_u32(sk), v_addr = smem_u32(sv);
      bool ok = mbar_wait(q_full, 0, abort_flag, a.status);
      for (int j = 0; ok && j < nkv; ++j) {
        if (!mbar_wait(k_full, j & 1, abort_flag, a.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kSubBytes + (kk & 3) * 32;
          umma_ss(tS, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                  idesc_qk, kk > 0);
        }
        umma_commit(s_full);
        umma_commit(k_empty);
        if (!mbar_wait(p_full, j & 1, abort_flag, a.status)) break;
        if (!mbar_wait(v_full, j & 1, abort_flag, a.status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          umma_ts(tO, tS + kk * 8, sdesc_sw128(v_addr + kk * 16 * 128, L::kSubBytes, 1024),
                  idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(v_empty);
      }
      umma_commit(o_full);
      drain_wait(o_full, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_f32 = 0.f, l_b16 = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!warp_wait(s_full, j & 1, abort_flag, a.status)) { ok = false; break; }
      tc_fence_after();
      float s[BN];
      uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + lane_off + c * 32, su + c * 32);
      tmem_ld_wait();
      const int valid = kv_total - j * BN;
      if (valid < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= valid) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < BN; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = mx * sl2;
      // Lazy rescaling: a row's reference max only moves when the tile max
      // exceeds it by more than the threshold.  TMEM loads/stores are
      // warp-collective, so the whole warp enters the rescale when any of its
      // rows needs it (f = 1 for the others).
      const bool need = (j > 0) && (m_new > m_run + kRescaleThreshold);
      if (j == 0) m_run = m_new;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? ex2(m_run - m_new) : 1.f;
        l_f32 *= f;
        l_b16 *= f;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t o[16];
          tmem_ld16(tO + lane_off + c * 16, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(f * __uint_as_float(o[i]));
          tmem_st16(tO + lane_off + c * 16, o);
        }
        if (need) m_run = m_new;
      }
      float sum_f = 0.f, sum_b = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = ex2(fmaf(s[32 * c + 2 * i], sl2, -m_run));
          const float p1 = ex2(fmaf(s[32 * c + 2 * i + 1], sl2, -m_run));
          pk[i] = pack_bf16(p0, p1);
          sum_f += p0 + p1;
          // the output is normalised by the sum of the bf16 weights the PV
          // product actually uses; the LSE by the fp32 sum
          sum_b += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xFFFF0000u);
        }
        tmem_st16(tS + lane_off + c * 16, pk);
      }
      l_f32 += sum_f;
      l_b16 += sum_b;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && warp_wait(o_full, 0, abort_flag, a.status)) {
      tc_fence_after();
      const float inv_l = 1.f / l_b16;
      int token;
      if (MODE == kDense) {
        token = tile * BM + row;
        if (token >= a.N) token = -1;
      } else {
        token = (row < a.C) ? __ldg(a.perm + (static_cast<size_t>(bh) * a.G + tile) * a.C + row)
                            : -1;
        if (token >= a.N) token = -1;
      }
      const size_t row_off = (static_cast<size_t>(bh) * a.N + (token < 0 ? 0 : token)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_ld_wait();
        if (token >= 0) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * inv_l;
          if (MODE == kSparseAdd || MODE == kSparseRecord) {
            const uint4* src = reinterpret_cast<const uint4*>(a.aux_in + row_off + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w = __ldg(src + q4);
              const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float2 f2 = __bfloat1622float2(h[e]);
                const int i0 = q4 * 8 + 2 * e;
                if (MODE == kSparseAdd) {
                  v[i0] += f2.x;
                  v[i0 + 1] += f2.y;
                } else {
                  v[i0] = f2.x - v[i0];
                  v[i0 + 1] = f2.y - v[i0 + 1];
                }
              }
            }
          }
          uint4* dst = reinterpret_cast<uint4*>(a.out + row_off + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16(v[q4 * 8 + 0], v[q4 * 8 + 1]);
            w.y = pack_bf16(v[q4 * 8 + 2], v[q4 * 8 + 3]);
            w.z = pack_bf16(v[q4 * 8 + 4], v[q4 * 8 + 5]);
            w.w = pack_bf16(v[q4 * 8 + 6], v[q4 * 8 + 7]);
            dst[q4] = w;
          }
        }
      }
      if (MODE == kDense && a.lse != nullptr && token >= 0)
        a.lse[static_cast<size_t>(bh) * a.N + token] = (m_run + __log2f(l_f32)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 256);
}

template <int D, int MODE>
cudaError_t launch_one(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                       const AttnArgs& a, int BH, cudaStream_t stream) {
  auto kern = attn_fwd_kernel<D, MODE>;
  const int smem = AttnLayout<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int gx = (MODE == kDense) ? (a.N + BM - 1) / BM : a.G;
  kern<<<dim3(gx, BH), kThreads, smem, stream>>>(*tq, *tk, *tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(int D, int mode, const CUtensorMap* tq, const CUtensorMap* tk,
                             const CUtensorMap* tv, const AttnArgs& a, int BH,
                             cudaStream_t stream) {
#define MCS_ATTN_CASE(DD, MM) \
  if (D == DD && mode == MM) return launch_one<DD, MM>(tq, tk, tv, a, BH, stream);
  MCS_ATTN_CASE(128, kDense)
  MCS_ATTN_CASE(128, kSparse)
  MCS_ATTN_CASE(128, kSparseAdd)
  MCS_ATTN_CASE(128, kSparseRecord)
  MCS_ATTN_CASE(64, kDense)
  MCS_ATTN_CASE(64, kSparse)
  MCS_ATTN_CASE(64, kSparseAdd)
  MCS_ATTN_CASE(64, kSparseRecord)
#undef MCS_ATTN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mcs
