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
// One CTA per SM; one CTA = one 128-row query tile (dense) or one query group
// (sparse) of one head.
//   warps 0-3  softmax + epilogue: thread t owns query row t = TMEM lane t
//   warps 4-10 producers: K and V tiles into a ring of kStages shared-memory
//              stages, as far ahead as the ring allows.  Dense: one thread
//              issues TMA tile loads.  Sparse: the 224 producer threads copy
//              the indexed K/V rows with 16-byte cp.async (two whole 256-byte
//              rows per warp instruction), writing them straight into the
//              128-byte-swizzled layout the MMA reads; each thread arrives
//              on the stage's mbarrier when its copies land.  (TMA gather4,
//              used for the one-time Q tile, issues too slowly per warp to
//              keep up with the tensor core here.)
//   warp 11    TMEM allocation and the single MMA-issuing thread
// TMEM (512 columns): two score buffers S0/S1 (128 fp32 columns each; P is
// written over S as bf16 pairs) and the O accumulator.  The MMA order
//   QK(0), QK(1), PV(0), QK(2), PV(1), QK(3), ...
// lets the tensor core compute S(j+1) and PV(j-1) while the softmax warps
// work on S(j).  Online softmax in base 2 with lazy rescaling (O is rescaled
// only when a row's running max grows by more than 8, so P <= 256).
#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int BM = 128;  // query rows per CTA (MMA M)
constexpr int BN = 128;  // KV rows per tile (MMA N of QK^T, K of PV)
constexpr int kProducers = 7;
constexpr int kFirstProducer = 4;
constexpr int kMmaWarp = 4 + kProducers;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct AttnLayout {
  static constexpr int kSub = D / 64;          // 128-byte column sub-tiles per row
  static constexpr int kSubBytes = 128 * 128;  // one sub-tile: 128 rows x 128 B
  static constexpr int kTileBytes = kSub * kSubBytes;
  static constexpr int kStages = D == 128 ? 7 : 14;  // K/V ring depth (tiles)
  static constexpr int kRing = 0;
  static constexpr int kBars = kRing + kStages * kTileBytes;
  static constexpr int kNumBars = 2 * kStages + 7;
  static constexpr int kSmem = kBars + kNumBars * 8 + 16 + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Sum of the eight fp32 partials held in four packed pairs.
__device__ __forceinline__ float sum8(const uint64_t* acc) {
  float a0, a1, a2, a3, a4, a5, a6, a7;
  f2_unpack(acc[0], a0, a1);
  f2_unpack(acc[1], a2, a3);
  f2_unpack(acc[2], a4, a5);
  f2_unpack(acc[3], a6, a7);
  return ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
}

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
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const AttnArgs a) {
  using L = AttnLayout<D>;
  constexpr int NS = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem + L::kRing;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* full = bars;              // [NS] stage loaded
  uint64_t* empty = bars + NS;        // [NS] stage consumed by its MMA
  uint64_t* q_full = bars + 2 * NS;   // Q tile written to TMEM (4 warp arrivals)
  uint64_t* s_full = q_full + 1;      // [2] S(j) in buffer j&1 computed
  uint64_t* p_full = q_full + 3;      // [2] P(j) written (4 warp arrivals)
  uint64_t* o_done = q_full + 5;      // PV(j) complete
  uint64_t* o_full = q_full + 6;      // every MMA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  const int tile = blockIdx.x;
  const int bh = blockIdx.y;
  const int kv_total = (MODE == kDense) ? a.N : a.K;
  const int nkv = (kv_total + BN - 1) / BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full + s, MODE == kDense ? 1 : 32 * kProducers);  // sparse: every producer thread
      mbar_init(empty + s, 1);
    }
    mbar_init(q_full, 4);
    mbar_init(s_full + 0, 1);
    mbar_init(s_full + 1, 1);
    mbar_init(p_full + 0, 4);
    mbar_init(p_full + 1, 4);
    mbar_init(o_done, 1);
    mbar_init(o_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 256;      // S0 at +0, S1 at +128
  const uint32_t tQ = tmem + 256 + D;  // Q tile, bf16 pairs (D/2 columns)

  if (warp >= 4 && warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    // Ring item i = 2j (K tile j) or 2j+1 (V tile j) goes to stage i % NS.
    int issued = 0;
    if (MODE == kDense) {
      if (warp == 4) {  // the whole warp waits; an elected lane issues the loads
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        for (int i = 0; i < 2 * nkv; ++i) {
          if (a.fault && i >= 2) break;  // test-only: starve the MMA thread
          const int st = i % NS;
          if (i >= NS && !warp_wait(empty + st, ((i / NS) - 1) & 1, abort_flag, a.status)) break;
          if (elect_one()) {
            mbar_expect_tx(full + st, L::kTileBytes);
            const CUtensorMap* tm = (i & 1) ? &tv : &tk;
            uint8_t* dst = ring + st * L::kTileBytes;
            for (int s = 0; s < L::kSub; ++s)
              tma_load_3d(dst + s * L::kSubBytes, tm, s * 64, (i >> 1) * BN, bh, full + st);
          }
          __syncwarp();
          ++issued;
        }
        if (*abort_flag) {
          for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
            drain_wait(full + (i % NS), (i / NS) & 1);
        }
      }
    } else {
      // Sparse.  Tile rows are token indices idx[j*128 + r]; a tile is
      // kChunks 16-byte chunks (row r = c / kSegs, segment c % kSegs) and
      // producer thread t copies chunks t, t + kPT, t + 2*kPT, ...
      constexpr int kPT = 32 * kProducers;
      constexpr int kSegs = D * 2 / 16;                 // 16-byte segments per row
      constexpr int kChunks = BN * kSegs;
      constexpr int kPer = (kChunks + kPT - 1) / kPT;   // chunks per thread (at most)
      const size_t grp = static_cast<size_t>(bh) * a.G + tile;
      const int32_t* idx_g = a.idx + grp * a.K;
      const int rowbase = bh * a.N;
      const int tid = (warp - kFirstProducer) * 32 + lane;
      bool bad = false;
      // Token indices of this thread's rows, loaded two tiles ahead so that
      // their latency (the index array is read once, from HBM) stays off the
      // critical path.
      auto load_rows = [&](int j, int* out) {
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int c = tid + kPT * k;
          int col = j * BN + (c < kChunks ? c / kSegs : 0);
          col = col < a.K ? col : a.K - 1;  // tail rows repeat a valid row; masked in softmax
          out[k] = __ldg(idx_g + col);
        }
      };
      int cur[kPer], nxt[kPer];
      load_rows(0, cur);
      if (nkv > 1) load_rows(1, nxt);
      bool stop = false;
      for (int j = 0; j < nkv && !stop; ++j) {
        if (a.fault && j >= 1) break;  // test-only: starve the MMA thread
        int ahead[kPer];
        if (j + 2 < nkv) load_rows(j + 2, ahead);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          if (cur[k] < 0 || cur[k] >= a.N) { bad = true; cur[k] = 0; }
        }
        for (int kv = 0; kv < 2; ++kv) {
          const int it = 2 * j + kv;
          const int st = it % NS;
          if (it >= NS && !warp_wait(empty + st, ((it / NS) - 1) & 1, abort_flag, a.status)) {
            stop = true;
            break;
          }
          const __nv_bfloat16* src = kv ? a.v : a.k;
          uint8_t* stage = ring + st * L::kTileBytes;
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int c = tid + kPT * k;
            if (c < kChunks) {
              const int r = c / kSegs, seg = c % kSegs;
              uint8_t* dst = stage + (seg >> 3) * L::kSubBytes + r * 128 +
                             (((seg & 7) ^ (r & 7)) << 4);
              cp_async16(dst, src + static_cast<size_t>(rowbase + cur[k]) * D + seg * 8);
            }
          }
          cp_async_arrive(full + st);
          ++issued;
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          cur[k] = nxt[k];
          nxt[k] = ahead[k];
        }
      }
      if (bad) atomicOr(a.status, DEV_BOUNDS);
      if (*abort_flag) asm volatile("cp.async.wait_all;" ::: "memory");  // copies land first
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (every branch warp-uniform) and one lane,
    // chosen by elect.sync right before each batch, issues the MMAs.  Issuing
    // from a lane-0-only branch instead is several times slower per MMA
    // (measured: 8 MMAs took ~400 cycles to issue from a divergent branch,
    // 69 from an elected lane), too slow to keep the tensor core fed.
    constexpr uint32_t idesc_qk = idesc_bf16(BM, BN, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16(BM, D, false, true);
    const uint32_t ring_addr = smem_u32(ring);
    auto issue_qk = [&](int j) -> bool {
      const int i = 2 * j, st = i % NS;
      if (!warp_wait(full + st, (i / NS) & 1, abort_flag, a.status)) return false;
      if (MODE != kDense) fence_proxy_async_smem();  // rows written by cp.async
      tc_fence_after();
      const uint32_t kb = ring_addr + st * L::kTileBytes;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {  // A = Q from TMEM, B = K tile
          const uint32_t off = (kk >> 2) * L::kSubBytes + (kk & 3) * 32;
          umma_ts(tmem + (j & 1) * 128, tQ + kk * 8, sdesc_sw128(kb + off, 16, 1024), idesc_qk,
                  kk > 0);
        }
        umma_commit(s_full + (j & 1));
        umma_commit(empty + st);
      }
      __syncwarp();
      return true;
    };
    bool ok = warp_wait(q_full, 0, abort_flag, a.status) && issue_qk(0);
    for (int j = 0; ok && j < nkv; ++j) {
      // S(j+1) goes into the other buffer, whose P(j-1) was consumed by
      // PV(j-1), issued earlier (MMAs of one thread execute in order).
      if (j + 1 < nkv && !issue_qk(j + 1)) break;
      if (!warp_wait(p_full + (j & 1), (j >> 1) & 1, abort_flag, a.status)) break;
      const int i = 2 * j + 1, st = i % NS;
      if (!warp_wait(full + st, (i / NS) & 1, abort_flag, a.status)) break;
      if (MODE != kDense) fence_proxy_async_smem();  // rows written by cp.async
      tc_fence_after();
      const uint32_t vb = ring_addr + st * L::kTileBytes;
      const uint32_t tP = tmem + (j & 1) * 128;
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          umma_ts(tO, tP + kk * 8, sdesc_sw128(vb + kk * 16 * 128, L::kSubBytes, 1024), idesc_pv,
                  (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(o_done);
        umma_commit(empty + st);
      }
      __syncwarp();
    }
    if (elect_one()) umma_commit(o_full);
    __syncwarp();
    drain_wait(o_full, 0);
  } else {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_f32 = 0.f, l_b16 = 0.f;
    bool ok = true;
    {
      // Q tile -> TMEM (the QK MMA's A operand, read from TMEM every tile
      // instead of shared memory): row `row` holds its D bf16 values as D/2
      // 32-bit columns, lower index in the low half.  Missing rows are zero.
      int src = -1;
      if (MODE == kDense) {
        src = tile * BM + row;
        if (src >= a.N) src = -1;
      } else if (row < a.C) {
        src = __ldg(a.perm + (static_cast<size_t>(bh) * a.G + tile) * a.C + row);
        if (src >= a.N) {
          atomicOr(a.status, DEV_BOUNDS);
          src = -1;
        }
      }
      const uint4* qrow = reinterpret_cast<const uint4*>(
          a.q + (static_cast<size_t>(bh) * a.N + (src < 0 ? 0 : src)) * D);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {  // 32 columns (64 values) at a time
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x = src >= 0 ? __ldg(qrow + c * 8 + i) : make_uint4(0, 0, 0, 0);
          w[4 * i + 0] = x.x;
          w[4 * i + 1] = x.y;
          w[4 * i + 2] = x.z;
          w[4 * i + 3] = x.w;
        }
        tmem_st32(tQ + lane_off + c * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }
    for (int j = 0; j < nkv; ++j) {
      if (!warp_wait(s_full + (j & 1), (j >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem + (j & 1) * 128 + lane_off;
      float s[BN];
      uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + c * 32, su + c * 32);
      tmem_ld_wait();
      const int valid = kv_total - j * BN;
      if (valid < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= valid) s[c] = -INFINITY;
      }
      // row max: four independent chains of 3-input max (short latency chain)
      float mc0 = s[0], mc1 = s[1], mc2 = s[2], mc3 = s[3];
#pragma unroll
      for (int c = 4; c < BN; c += 8) {
        mc0 = fmax3(mc0, s[c + 0], s[c + 1]);
        mc1 = fmax3(mc1, s[c + 2], s[c + 3]);
        mc2 = fmax3(mc2, s[c + 4 < BN ? c + 4 : 0], s[c + 5 < BN ? c + 5 : 0]);
        mc3 = fmax3(mc3, s[c + 6 < BN ? c + 6 : 0], s[c + 7 < BN ? c + 7 : 0]);
      }
      const float mx = fmaxf(fmaxf(mc0, mc1), fmaxf(mc2, mc3));
      const float m_new = mx * sl2;
      // Lazy rescaling: a row's reference max only moves when the tile max
      // exceeds it by more than the threshold.  TMEM loads/stores are
      // warp-collective, so the whole warp enters the rescale when any of its
      // rows needs it (f = 1 for the others).  O may still be accumulating
      // PV(j-1): wait for it first (PV(j) cannot start before this P(j)).
      const bool need = (j > 0) && (m_new > m_run + kRescaleThreshold);
      if (j == 0) m_run = m_new;
      if (__any_sync(0xffffffffu, need)) {
        if (!warp_wait(o_done, (j - 1) & 1, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
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
      // p = 2^(s*c - m): packed FFMA2 for the argument, MUFU ex2, bf16 pack.
      // Two row sums, each in four packed accumulators: the fp32 weights (for
      // the LSE) and the bf16 weights the PV product actually multiplies by
      // (the output is normalised by those, which keeps its error smaller).
      const uint64_t c2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_run, -m_run);
      uint64_t accf[4] = {0ull, 0ull, 0ull, 0ull}, accb[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), c2, nm2), x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          pk[i] = pack_bf16(p0, p1);
          accf[i & 3] = f2_add(accf[i & 3], f2_pack(p0, p1));
          accb[i & 3] = f2_add(accb[i & 3], f2_pack(__uint_as_float(pk[i] << 16),
                                                    __uint_as_float(pk[i] & 0xFFFF0000u)));
        }
        tmem_st16(tS + c * 16, pk);
      }
      l_f32 += sum8(accf);
      l_b16 += sum8(accb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + (j & 1));
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
        a.lse[static_cast<size_t>(bh) * a.N + token] =
            (m_run + __log2f(l_f32)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
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
