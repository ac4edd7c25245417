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
// One CTA per SM works on TWO query units of one head at once, a and b:
// query tiles 2x and 2x+1 (dense) or query groups 2x and 2x+1 (sparse).  The
// two units form independent softmax -> PV -> QK chains, so the tensor core
// runs one unit's products while the other unit's softmax warps work; with a
// single unit per CTA the softmax, the MMA completion latency and the
// hand-offs of every tile sat on the critical path.
//   warps 0-3   softmax + epilogue of unit a; thread t owns query row t
//   warps 4-7   the same for unit b
//   warps 8-14  producers.  Dense: one warp issues TMA tile loads of Q and of
//               the K/V tiles both units share.  Sparse: the 224 producer
//               threads copy each unit's query rows (by perm) and indexed K/V
//               rows (by idx) with 16-byte cp.async straight into the
//               128-byte-swizzled layout the MMA reads, and arrive on the
//               stage's mbarrier when their copies land.  Each warp reads the
//               indices of its rows of a tile once (one per lane, coalesced)
//               and broadcasts them with shuffles.
//   warp 15     TMEM allocation and MMA issue (one elected lane)
// Shared memory: Q_a and Q_b (the QK A-operands) and a ring of K/V tiles.
// TMEM (512 columns): S_a, S_b (128 fp32 columns each; P is written over S
// as bf16 pairs) and the accumulators O_a, O_b.  MMA order
//   QK_a(0) QK_b(0) | PV_a(0) QK_a(1) PV_b(0) QK_b(1) | PV_a(1) QK_a(2) ...
// QK_x(j+1) overwrites S_x only after PV_x(j), which read P_x(j), in the
// in-order MMA stream; and a commit signals completion of every earlier MMA,
// so a softmax warp that sees S_x(j) complete knows PV_x(j-1) is done too.
// Online softmax in base 2 with lazy rescaling (O is rescaled only when a
// row's running max grows by more than 16, so P <= 2^16; P is bf16 (relative
// rounding whatever its size) and O and the row sums are fp32, whose range
// that bound leaves untouched: 2^16 * N * |v| stays far below 2^127).
//
// E4M3 K/V (mode flag kE4M3; the pages leave low-precision attention open:
// ai.info AI summary, "Future Directions"): K and V are read as E4M3 bytes,
// half the bytes of bf16.  The producers copy the E4M3 rows into the stage
// with cp.async, then read them back, convert them to f16 (exact: every E4M3
// value is an f16 value) and store them in the same swizzled layout the bf16
// gathers produce; Q is converted from bf16
// to f16 on its way in, P is written as f16, and the MMAs take f16 operands
// (kind::f16, both operands f16).  P <= 2^15 there (rescale threshold 15),
// inside the f16 range.  The K scale is folded into the softmax scale, the V
// scale into the output normalisation.
#include "internal.h"
#include "ptx.cuh"

namespace mcs {
namespace {

constexpr int BM = 128;  // query rows per unit (MMA M)
constexpr int BN = 128;  // KV rows per tile (MMA N of QK^T, K of PV)
constexpr int kSoftmaxWarps = 8;
constexpr int kProducers = 7;
constexpr int kFirstProducer = kSoftmaxWarps;
constexpr int kMmaWarp = kFirstProducer + kProducers;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr float kRescaleThreshold = 16.0f;
constexpr float kRescaleThresholdF16 = 15.0f;  // f16 P: 2^15 < 65504
// Batch-completion barriers, used round robin.  A waiter on batch n reads the
// phase parity of done[n % kDone]; that is unambiguous as long as batch
// n + kDone cannot have completed yet.  The producers lag furthest: before
// loading ring item i they wait for the last batch reading item i - NS, and
// the batches that can complete meanwhile are those whose items are all
// below i: at most NS - 1 later (dense, 2 items per step) or NS / 2 later
// (sparse, 4 items per step).  16 covers both rings (NS <= 12).
constexpr int kDone = 16;

template <int D, bool PAIRS>
struct AttnLayout {
  static constexpr int kSub = D / 64;          // 128-byte column sub-tiles per row
  static constexpr int kSubBytes = 128 * 128;  // one sub-tile: 128 rows x 128 B
  static constexpr int kTileBytes = kSub * kSubBytes;  // a 128-row tile of Q, K or V
  // paired mode: each stage also holds the mask operand of a K tile (128 keys
  // x 16 bf16, K-major without swizzle), and one more 128 x 16 operand holds
  // the rows' group selectors
  static constexpr int kMaskBytes = PAIRS ? 128 * 32 : 0;
  static constexpr int kStageBytes = kTileBytes + kMaskBytes;
  static constexpr int kStages = PAIRS ? (D == 128 ? 4 : 9) : (D == 128 ? 5 : 12);  // ring depth
  static constexpr int kQ = 0;                         // Q_a, Q_b
  static constexpr int kRowSel = 2 * kTileBytes;       // paired mode: row group selectors
  static constexpr int kRing = kRowSel + kMaskBytes;
  static constexpr int kBars = kRing + kStages * kStageBytes;
  static constexpr int kNumBars = kStages + kDone + 3;
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

// Max of 64 scores: four independent chains of 3-input max.
__device__ __forceinline__ float max64(const float* s) {
  float m0 = s[0], m1 = s[1], m2 = s[2], m3 = s[3];
#pragma unroll
  for (int c = 4; c < 60; c += 8) {
    m0 = fmax3(m0, s[c + 0], s[c + 1]);
    m1 = fmax3(m1, s[c + 2], s[c + 3]);
    m2 = fmax3(m2, s[c + 4], s[c + 5]);
    m3 = fmax3(m3, s[c + 6], s[c + 7]);
  }
  m0 = fmax3(m0, s[60], s[61]);
  m1 = fmax3(m1, s[62], s[63]);
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// Paired mode: the 16-byte K-major chunk (elements 0-7 of the mask step's K
// dimension) of row r of a 128 x 16 bf16 operand without swizzle, stored as
// 8-row x 16-byte core matrices (the two K halves of an 8-row group adjacent).
__device__ __forceinline__ int mask_row_offset(int r) { return (r >> 3) * 256 + (r & 7) * 16; }

// Mask chunk of a key by its group membership bits (bit 0: in the pair's
// first group, bit 1: in its second): elements (k0, k1) = 0 for the groups
// that selected the key and -2^20 for the others; bf16 -2^20 = 0xC980.
__device__ __align__(16) uint4 g_pair_mask[4] = {
    {0xC980C980u, 0u, 0u, 0u}, {0xC9800000u, 0u, 0u, 0u}, {0x0000C980u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}};

// Byte offset of 16-byte chunk `seg` of row r in a 128-row tile stored as
// 128-byte-swizzled K-major sub-tiles (the layout TMA writes with SW128).
__device__ __forceinline__ int swz_offset(int r, int seg) {
  return (seg >> 3) * (128 * 128) + r * 128 + (((seg & 7) ^ (r & 7)) << 4);
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const AttnArgs a) {
  constexpr bool kPairs = (MODE & kPaired) != 0;
  constexpr int kBase = MODE & 3;  // kDense, kSparse, kSparseAdd or kSparseRecord
  using L = AttnLayout<D, kPairs>;
  constexpr int NS = L::kStages;
  constexpr bool kSparseMode = MODE != kDense;
  constexpr bool kE4 = (MODE & kE4M3) != 0;
  static_assert(!kE4 || (!kPairs && (kBase == kSparse || kBase == kSparseAdd)),
                "E4M3 K/V: unpaired sparse and sparse + residual modes only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* qs = smem + L::kQ;  // Q_a, then Q_b
  uint8_t* ring = smem + L::kRing;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* full = bars;              // [NS] stage loaded
  uint64_t* done = bars + NS;         // [kDone] MMA batch n complete: done[n % kDone]
  uint64_t* q_full = done + kDone;    // Q_a and Q_b loaded
  uint64_t* p_full = q_full + 1;      // [2] P_x(j) written (4 warp arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = warp_id();
  const int lane = lane_id();
  const int pair = blockIdx.x;
  const int bh = blockIdx.y;
  const int head_h = bh % a.H, head_b = bh / a.H;    // tile-map coordinates of this head
  const RowMap rm = row_map(a.layout, a.H, a.N, bh);  // rows of q/k/v/out in either layout
  // units per head: query tiles (dense), groups (sparse) or sibling pairs of
  // C = 64 groups (paired)
  const int units = kSparseMode ? (kPairs ? a.P : a.G) : (a.N + BM - 1) / BM;
  const bool has_b = 2 * pair + 1 < units;
  const int kv_total = kSparseMode ? a.K : a.N;
  // keys per unit: a pair's union list is as long as its plen entry
  int kv_len[2] = {kv_total, kv_total};
  if (kPairs) {
    kv_len[0] = __ldg(a.plen + static_cast<size_t>(bh) * a.P + 2 * pair);
    kv_len[1] = has_b ? __ldg(a.plen + static_cast<size_t>(bh) * a.P + 2 * pair + 1) : kv_len[0];
    kv_len[0] = min(max(kv_len[0], 1), a.cap);
    kv_len[1] = min(max(kv_len[1], 1), a.cap);
  }
  const int nkv = (max(kv_len[0], kv_len[1]) + BN - 1) / BN;
  // Unpaired C = 64 groups fill half a 128-row tile: unit a's rows go to tile
  // rows 0-63 (TMEM lanes read by warps 0-1), unit b's to rows 64-127 (warps
  // 6-7), so that each scheduler runs one busy softmax warp instead of two
  // (a warp may only read its own quarter of the TMEM lanes); the warps of
  // the empty rows keep only the hand-off protocol.
  const int qoff_b = (kSparseMode && !kPairs && a.C <= BM / 2) ? BM / 2 : 0;
  auto qoff = [&](int x) { return x == 1 ? qoff_b : 0; };
  // Ring items, numbered in the order the MMA warp consumes them (item i
  // goes to stage i % NS).  Dense: K(j) = 2j, V(j) = 2j+1, each shared by
  // both units.  Sparse: K_a(0) = 0, K_b(0) = 1, then per step j
  // V_a(j) = 4j+2, K_a(j+1) = 4j+3, V_b(j) = 4j+4, K_b(j+1) = 4j+5 (the two
  // K items of the last step do not exist).  In consumption order, every
  // gather has the same lead: the NS - 1 products before it.
  auto k_item = [&](int x, int j) {
    return kSparseMode ? (j == 0 ? x : 4 * j - 1 + 2 * x) : 2 * j;
  };
  auto v_item = [&](int x, int j) { return kSparseMode ? 4 * j + 2 + 2 * x : 2 * j + 1; };
  // MMA batches, in issue order: batch 0 = QK_a(0) QK_b(0); batch 2j+x+1 =
  // PV_x(j) QK_x(j+1).  Each batch ends with ONE commit, on done[n % kDone]:
  // that commit signals completion of every earlier MMA too, so it serves
  // the softmax (S_x ready), the epilogue (O_x final) and the producers
  // (stages free).
  static_assert(kDone >= NS, "batch barriers must outnumber the producer lag");
  auto wait_batch = [&](int n) {
    return warp_wait(done + n % kDone, (n / kDone) & 1, abort_flag, a.status);
  };
  // last batch that reads ring item i (its stage is free once it is done)
  auto release_batch = [&](int i) {
    return kSparseMode ? i >> 1 : ((i & 1) ? i + 1 : i);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s)
      mbar_init(full + s, kSparseMode ? 32 * kProducers : 1);  // sparse: every producer thread
    for (int n = 0; n < kDone; ++n) mbar_init(done + n, 1);
    mbar_init(q_full, kSparseMode ? 32 * kProducers : 1);
    for (int x = 0; x < 2; ++x) mbar_init(p_full + x, 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if constexpr (kPairs) {
    // row selectors: rows 0-63 (the pair's first group) take mask element
    // k0, rows 64-127 element k1 (bf16 1.0 = 0x3F80); the stages' mask
    // operands start zeroed (their second K half stays zero)
    uint8_t* rsel = smem + L::kRowSel;
    for (int r = threadIdx.x; r < 128; r += kThreads) {
      *reinterpret_cast<uint4*>(rsel + mask_row_offset(r)) =
          make_uint4(r < 64 ? 0x3F80u : 0x3F800000u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(rsel + mask_row_offset(r) + 128) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = threadIdx.x; i < NS * (L::kMaskBytes / 16); i += kThreads) {
      const int st = i / (L::kMaskBytes / 16), o = i % (L::kMaskBytes / 16);
      reinterpret_cast<uint4*>(smem + L::kRing + st * L::kStageBytes + L::kTileBytes)[o] =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();  // generic writes -> tensor-core operand reads
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // S_a at +0, S_b at +128, O_a at +256, O_b at +256+D

  if (warp >= kFirstProducer && warp < kMmaWarp) {
    // ------------------------------------------------------------ producers
    int issued = 0;
    if (!kSparseMode) {
      if (warp == kFirstProducer) {  // the whole warp waits; an elected lane issues the loads
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        if (elect_one()) {
          // Q_a, Q_b: rows past N (and a missing unit b) are zero-filled by TMA
          mbar_expect_tx(q_full, 2 * L::kTileBytes);
          for (int x = 0; x < 2; ++x)
            for (int s = 0; s < L::kSub; ++s)
              tma_load_4d(qs + x * L::kTileBytes + s * L::kSubBytes, &tq, s * 64,
                          (2 * pair + x) * BM, head_h, head_b, q_full);
        }
        __syncwarp();
        for (int i = 0; i < 2 * nkv; ++i) {
          if (a.fault && i >= 2) break;  // test-only: starve the MMA warp
          const int st = i % NS;
          if (i >= NS && !wait_batch(release_batch(i - NS))) break;
          if (elect_one()) {
            mbar_expect_tx(full + st, L::kTileBytes);
            const CUtensorMap* tm = (i & 1) ? &tv : &tk;
            uint8_t* dst = ring + st * L::kStageBytes;
            for (int s = 0; s < L::kSub; ++s)
              tma_load_4d(dst + s * L::kSubBytes, tm, s * 64, (i >> 1) * BN, head_h, head_b,
                          full + st);
          }
          ++issued;
        }
        if (*abort_flag) {
          for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
            drain_wait(full + (i % NS), (i / NS) & 1);
        }
      }
    } else {
      // Sparse.  Q rows: a 128-row tile is kChunks 16-byte chunks (row r =
      // c / kSegs, segment c % kSegs); producer thread p copies chunks p,
      // p + kPT, ...  K/V tiles: each warp instruction copies kRPI whole rows
      // (lane -> row kRPI * rg + lane / kSegs, segment lane % kSegs); producer
      // warp pw takes the row groups rg = pw, pw + kProducers, ...  The tokens
      // of a tile's rows are read once per warp (one index per lane) and
      // broadcast with shuffles.
      constexpr int kPT = 32 * kProducers;
      constexpr int kSegs = D * 2 / 16;                 // 16-byte segments per bf16 row
      constexpr int kChunks = BM * kSegs;
      constexpr int kPer = (kChunks + kPT - 1) / kPT;   // Q chunks per thread (at most)
      constexpr int kKVSegs = kE4 ? D / 16 : kSegs;     // 16-byte segments per K/V row read
      constexpr int kRPI = 32 / kKVSegs;                // rows per warp instruction
      constexpr int kRG = BN / kRPI;                    // row groups per tile
      constexpr int kGPW = (kRG + kProducers - 1) / kProducers;  // row groups per warp
      static_assert(kGPW * kRPI <= 32, "one index per lane");
      const int tid = (warp - kFirstProducer) * 32 + lane;
      const int pw = warp - kFirstProducer;
      const int sub = lane / kKVSegs, seg = lane % kKVSegs;
      const int group[2] = {2 * pair, has_b ? 2 * pair + 1 : 2 * pair};
      bool bad = false;
      // Q rows of both units (perm order); padding slots, rows past the
      // unit's queries and a missing unit b are zero rows.  A pair's rows are
      // the perm rows of its two groups, which are adjacent in perm.
      for (int x = 0; x < 2; ++x) {
        const int32_t* perm_g =
            a.perm + (static_cast<size_t>(bh) * a.G + (kPairs ? 2 * group[x] : group[x])) * a.C;
        const int qrows = kPairs ? (2 * group[x] + 1 < a.G ? 2 : 1) * a.C : a.C;
        [[maybe_unused]] uint4 qw[kE4 ? kPer : 1];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int c = tid + kPT * k;
          if (c < kChunks) {
            const int r = c / kSegs, sg = c % kSegs;
            const int gr = r - qoff(x);  // the group's row in this tile row
            int tok = (gr >= 0 && gr < qrows && (x == 0 || has_b)) ? __ldg(perm_g + gr) : -1;
            if (tok >= a.N) { bad = true; tok = -1; }
            const __nv_bfloat16* src =
                a.q + static_cast<size_t>(rm.rbase + (tok < 0 ? 0 : tok) * rm.rstride) * D + sg * 8;
            if constexpr (kE4)  // bf16 -> f16 through registers: all loads first
              qw[k] = tok >= 0 ? __ldg(reinterpret_cast<const uint4*>(src))
                               : make_uint4(0u, 0u, 0u, 0u);
            else
              cp_async16_zfill(qs + x * L::kTileBytes + swz_offset(r, sg), src, tok >= 0);
          }
        }
        if constexpr (kE4) {
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int c = tid + kPT * k;
            if (c < kChunks) {
              const uint4 w = qw[k];
              st_shared16(qs + x * L::kTileBytes + swz_offset(c / kSegs, c % kSegs),
                          make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y),
                                     bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w)));
            }
          }
        }
      }
      if constexpr (kE4) {
        fence_proxy_async_smem();  // generic writes -> tensor-core operand reads
        mbar_arrive(q_full);
      } else {
        cp_async_arrive(q_full);
      }
      // This lane's row (RowMap) of tile j of unit x: lane l < kGPW * kRPI
      // holds the row of group pw + kProducers * (l / kRPI), sub-row l % kRPI.
      // Loaded two tiles ahead so that the index latency (the index array is
      // read once, from HBM) stays off the critical path.
      // Paired mode: the pair's union list instead (no tail clamp: lists are
      // padded to whole tiles); the entry's group bits go to *bits.
      auto load_rows = [&](int x, int j, int* bits) -> int {
        const int32_t* idx_g =
            kPairs ? a.pidx + (static_cast<size_t>(bh) * a.P + group[x]) * a.cap
                   : a.idx + (static_cast<size_t>(bh) * a.G + group[x]) * a.K;
        int out = 0;
        *bits = 0;
        if (lane < kGPW * kRPI) {
          const int rg = pw + kProducers * (lane / kRPI);
          int col = j * BN + (rg < kRG ? rg * kRPI + lane % kRPI : 0);
          if (!kPairs) col = col < a.K ? col : a.K - 1;  // tail rows repeat a valid row; masked
          int tok = __ldg(idx_g + col);
          if (kPairs) {
            *bits = static_cast<int>((static_cast<uint32_t>(tok) >> kPairTokenBits) & 3u);
            tok &= (1 << kPairTokenBits) - 1;
          }
          if (tok < 0 || tok >= a.N) { bad = true; tok = 0; }
          out = rm.rbase + tok * rm.rstride;
        }
        return out;
      };
      // Copy the rows of one K or V tile into the stage of ring item `it`;
      // paired mode, K tiles: also each key's mask chunk (by its group bits)
      // into the stage's mask operand.
      auto copy_tile = [&](int it, const __nv_bfloat16* src, int rows, int bits,
                           bool is_k) -> bool {
        const int st = it % NS;
        if (it >= NS && !wait_batch(release_batch(it - NS))) return false;
        uint8_t* stage = ring + st * L::kStageBytes;
#pragma unroll
        for (int i = 0; i < kGPW; ++i) {
          const int rg = pw + kProducers * i;
          const int row = __shfl_sync(0xffffffffu, rows, i * kRPI + sub);
          if (rg < kRG)
            cp_async16(stage + swz_offset(rg * kRPI + sub, seg),
                       src + static_cast<size_t>(row) * D + seg * 8);
          if (kPairs && is_k) {
            const int b = __shfl_sync(0xffffffffu, bits, i * kRPI + sub);
            if (rg < kRG && seg == 0)
              cp_async16_ca(stage + L::kTileBytes + mask_row_offset(rg * kRPI + sub), g_pair_mask + b);
          }
        }
        cp_async_arrive(full + st);
        ++issued;
        return true;
      };
      // Both units' index rows are read once, from HBM: pull them into L2
      // now so that the per-tile index loads below hit L2.
      for (int x = 0; x < 2; ++x) {
        const char* idx_g = reinterpret_cast<const char*>(
            kPairs ? a.pidx + (static_cast<size_t>(bh) * a.P + group[x]) * a.cap
                   : a.idx + (static_cast<size_t>(bh) * a.G + group[x]) * a.K);
        const int bytes = (kPairs ? kv_len[x] : a.K) * 4;
        for (int off = tid * 128; off < bytes; off += kPT * 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(idx_g + off));
      }
      if constexpr (kE4) {
        // E4M3 rows: each ring item's rows are copied as raw bytes (16-byte
        // cp.async, one commit group per item) into the upper half of their
        // own f16 lines in the item's stage (D = 128: line r of the second
        // 128-byte sub-tile; D = 64: bytes 64-127 of line r).  kLag items
        // later, once they have landed, the same lanes read them back,
        // convert them to f16 and store row r's f16 chunks into line r (and,
        // D = 128, line r of the first sub-tile), then arrive on the stage.
        // Only the lanes of row r touch its staging bytes and its lines, all
        // in one warp, so a __syncwarp between the reads and the writes
        // orders them.  The copies need no registers and run ahead like the
        // bf16 gathers; the conversion waits kLag items behind them.
        // the release a copy waits for needs every item up to kLag + 2
        // before it converted: kLag <= NS - 2.  Converting one item behind
        // the copies measured fastest (lags of 2 and 3 delay the stages the
        // MMA is about to need).
        constexpr int kLag = 1;
        static_assert(kLag <= NS - 2, "conversions must not wait on the releases they gate");
        int stoff[kGPW], soff[kGPW][2];
#pragma unroll
        for (int i = 0; i < kGPW; ++i) {
          const int r = (pw + kProducers * i) * kRPI + sub;
          stoff[i] = (D == 128 ? 128 * 128 : 64) + r * 128 + seg * 16;
          soff[i][0] = swz_offset(r, 2 * seg);
          soff[i][1] = swz_offset(r, 2 * seg + 1);
        }
        auto convert = [&](int it) {
          uint8_t* stage = ring + (it % NS) * L::kStageBytes;
          uint4 raw[kGPW];
#pragma unroll
          for (int i = 0; i < kGPW; ++i)
            if (pw + kProducers * i < kRG) raw[i] = ld_shared16(stage + stoff[i]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < kGPW; ++i) {
            if (pw + kProducers * i < kRG) {
              uint4 lo, hi;
              e4m3x4_to_f16x4(raw[i].x, lo.x, lo.y);
              e4m3x4_to_f16x4(raw[i].y, lo.z, lo.w);
              e4m3x4_to_f16x4(raw[i].z, hi.x, hi.y);
              e4m3x4_to_f16x4(raw[i].w, hi.z, hi.w);
              st_shared16(stage + soff[i][0], lo);
              st_shared16(stage + soff[i][1], hi);
            }
          }
          fence_proxy_async_smem();  // generic writes -> tensor-core operand reads
          mbar_arrive(full + it % NS);
        };
        int pend[kLag];  // items copied, not yet converted (oldest first; -1: none)
#pragma unroll
        for (int l = 0; l < kLag; ++l) pend[l] = -1;
        auto copy8 = [&](int it, const uint8_t* src, int rows) -> bool {
          const int st = it % NS;
          if (it >= NS && !wait_batch(release_batch(it - NS))) return false;
          uint8_t* stage = ring + st * L::kStageBytes;
#pragma unroll
          for (int i = 0; i < kGPW; ++i) {
            const int rg = pw + kProducers * i;
            const int row = __shfl_sync(0xffffffffu, rows, i * kRPI + sub);
            if (rg < kRG) cp_async16(stage + stoff[i], src + static_cast<size_t>(row) * D + seg * 16);
          }
          cp_async_commit();
          ++issued;
          if (pend[kLag - 1] >= 0) {
            cp_async_wait_group<kLag>();  // the oldest pending item has landed
            convert(pend[0]);
#pragma unroll
            for (int l = 0; l + 1 < kLag; ++l) pend[l] = pend[l + 1];
            pend[kLag - 1] = it;
          } else {
            bool placed = false;
#pragma unroll
            for (int l = 0; l < kLag; ++l)
              if (!placed && pend[l] < 0) {
                pend[l] = it;
                placed = true;
              }
          }
          return true;
        };
        int bits;  // group bits: paired mode only
        int r0[2], r1[2] = {0, 0}, r2[2] = {0, 0};
        r0[0] = load_rows(0, 0, &bits);
        r0[1] = load_rows(1, 0, &bits);
        if (nkv > 1) {
          r1[0] = load_rows(0, 1, &bits);
          r1[1] = load_rows(1, 1, &bits);
        }
        bool ok = copy8(k_item(0, 0), a.k8, r0[0]) && copy8(k_item(1, 0), a.k8, r0[1]);
        for (int j = 0; ok && j < nkv; ++j) {
          if (a.fault && j >= 1) break;  // test-only: starve the MMA warp
          const bool more = j + 1 < nkv;
          for (int x = 0; ok && x < 2; ++x)
            ok = copy8(v_item(x, j), a.v8, r0[x]) &&
                 (!more || copy8(k_item(x, j + 1), a.k8, r1[x]));
          if (j + 2 < nkv) {
            r2[0] = load_rows(0, j + 2, &bits);
            r2[1] = load_rows(1, j + 2, &bits);
          }
          r0[0] = r1[0];
          r0[1] = r1[1];
          r1[0] = r2[0];
          r1[1] = r2[1];
        }
        cp_async_wait_group<0>();
        if (ok && !a.fault) {  // the last items
#pragma unroll
          for (int l = 0; l < kLag; ++l)
            if (pend[l] >= 0) convert(pend[l]);
        }
      } else {
      // rows (and paired-mode group bits) of tiles j (V_x(j)), j+1 (K_x(j+1))
      // and j+2 (being fetched)
      int r0[2], r1[2] = {0, 0}, r2[2] = {0, 0};
      int b0[2], b1[2] = {0, 0}, b2[2] = {0, 0};
      r0[0] = load_rows(0, 0, &b0[0]);
      r0[1] = load_rows(1, 0, &b0[1]);
      if (nkv > 1) {
        r1[0] = load_rows(0, 1, &b1[0]);
        r1[1] = load_rows(1, 1, &b1[1]);
      }
      bool ok = copy_tile(k_item(0, 0), a.k, r0[0], b0[0], true) &&
                copy_tile(k_item(1, 0), a.k, r0[1], b0[1], true);
      for (int j = 0; ok && j < nkv; ++j) {
        if (a.fault && j >= 1) break;  // test-only: starve the MMA warp
        const bool more = j + 1 < nkv;
        for (int x = 0; ok && x < 2; ++x)
          ok = copy_tile(v_item(x, j), a.v, r0[x], 0, false) &&
               (!more || copy_tile(k_item(x, j + 1), a.k, r1[x], b1[x], true));
        // indices of tile j+2, after this step's copies: their load latency
        // then delays nothing already due
        if (j + 2 < nkv) {
          r2[0] = load_rows(0, j + 2, &b2[0]);
          r2[1] = load_rows(1, j + 2, &b2[1]);
        }
        r0[0] = r1[0];
        r0[1] = r1[1];
        r1[0] = r2[0];
        r1[1] = r2[1];
        b0[0] = b1[0];
        b0[1] = b1[1];
        b1[0] = b2[0];
        b1[1] = b2[1];
      }
      }
      if (bad) atomicOr(a.status, DEV_BOUNDS);
      if (*abort_flag) asm volatile("cp.async.wait_all;" ::: "memory");  // copies land first
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (every branch warp-uniform) and one lane,
    // chosen by elect.sync right before each batch, issues the MMAs; issuing
    // from a lane-0-only branch is several times slower per MMA.
    //
    // The first mbarrier operation after a batch stalls until the tensor core
    // has taken nearly the whole batch (it buffers only one or two MMAs), so
    // a wait between batches is time the tensor core may sit idle.  PV_x(j)
    // and QK_x(j+1) of a unit are therefore issued as one batch, after the
    // waits for its operands (V_x(j) and K_x(j+1), loaded well ahead) and for
    // P_x(j).
    constexpr uint32_t idesc_qk =
        kE4 ? idesc_f16(BM, BN, false, false) : idesc_bf16(BM, BN, false, false);
    constexpr uint32_t idesc_pv = kE4 ? idesc_f16(BM, D, false, true) : idesc_bf16(BM, D, false, true);
    const uint32_t ring_addr = smem_u32(ring);
    const uint32_t q_addr = smem_u32(qs);
    auto stage_addr = [&](int item) { return ring_addr + (item % NS) * L::kStageBytes; };
    auto wait_item = [&](int item) {
      return warp_wait(full + item % NS, (item / NS) & 1, abort_flag, a.status);
    };
    // S_x(j) = Q_x K(j)^T (issuing lane only); paired mode: plus one K = 16
    // step of row selectors x key masks, which adds -2^20 to the scores of
    // keys the row's group did not select (exactly 0 to the others)
    auto issue_qk = [&](int x, int j) {
      const int i = k_item(x, j);
      const uint32_t kb = stage_addr(i), qb = q_addr + x * L::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * L::kSubBytes + (kk & 3) * 32;
        umma_ss(tmem + x * 128, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                idesc_qk, kk > 0);
      }
      if (kPairs)
        umma_ss(tmem + x * 128, sdesc_none(smem_u32(smem + L::kRowSel), 128, 256),
                sdesc_none(kb + L::kTileBytes, 128, 256), idesc_qk, 1u);
    };
    // O_x (+)= P_x(j) V(j), A = P from TMEM (issuing lane only)
    auto issue_pv = [&](int x, int j) {
      const int i = v_item(x, j);
      const uint32_t vb = stage_addr(i);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        umma_ts(tmem + 256 + x * D, tmem + x * 128 + kk * 8,
                sdesc_sw128(vb + kk * 16 * 128, L::kSubBytes, 1024), idesc_pv,
                (j > 0 || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = warp_wait(q_full, 0, abort_flag, a.status) && wait_item(k_item(0, 0)) &&
              wait_item(k_item(1, 0));
    if (ok) {
      if (kSparseMode) fence_proxy_async_smem();
      tc_fence_after();
      if (elect_one()) {
        issue_qk(0, 0);
        issue_qk(1, 0);
        umma_commit(done);
      }
    }
    for (int j = 0; ok && j < nkv; ++j) {
      const bool more = j + 1 < nkv;
      for (int x = 0; ok && x < 2; ++x) {
        // Probe the batch's barriers together (their latencies overlap);
        // only if one is not complete yet wait for each in turn.
        const int iv = v_item(x, j), ik = more ? k_item(x, j + 1) : iv;
        const bool ready = mbar_try_wait(full + iv % NS, (iv / NS) & 1) &
                           mbar_try_wait(full + ik % NS, (ik / NS) & 1) &
                           mbar_try_wait(p_full + x, j & 1);
        if (!__all_sync(0xffffffffu, ready))
          ok = wait_item(iv) && wait_item(ik) && warp_wait(p_full + x, j & 1, abort_flag, a.status);
        if (!ok) break;
        if (kSparseMode) fence_proxy_async_smem();
        tc_fence_after();
        if (elect_one()) {
          const int n = 2 * j + x + 1;
          issue_pv(x, j);
          if (more) issue_qk(x, j + 1);
          umma_commit(done + n % kDone);
        }
      }
    }
    const int n_last = 2 * nkv;
    drain_wait(done + n_last % kDone, (n_last / kDone) & 1);
  } else {
    // ------------------------------------------------------------ softmax
    // Warps 4x .. 4x+3 handle unit x; warp w reads TMEM lanes 32*(w%4) ...
    // The 128 scores of a row are handled 64 at a time (the register budget
    // of 16 warps): the max over both halves first, then the exponentials of
    // columns 0-63 (kept in registers) and of columns 64-127 (loaded again).
    // P of columns 0-63 goes over S columns 0-31, already read, and P of
    // 64-127 over columns 32-63, read in the first half.
    const int x = warp >> 2;
    const int row = (warp & 3) * 32 + lane;  // 0..127 == TMEM lane
    const int kv_mine = x == 0 ? kv_len[0] : kv_len[1];  // keys of this warp's unit
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + x * 128 + lane_off;
    const uint32_t tO = tmem + 256 + x * D + lane_off;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY, l_f32 = 0.f, l_b16 = 0.f;
    bool ok = true;
    // this warp's 32 rows hold none of the unit's queries (warp-uniform)
    const bool idle = kSparseMode && !kPairs &&
                      ((warp & 3) * 32 + 32 <= qoff(x) || (warp & 3) * 32 >= qoff(x) + a.C);
    for (int j = 0; j < nkv; ++j) {
      if (!wait_batch(j == 0 ? 0 : 2 * j + x - 1)) {  // S_x(j) written
        ok = false;
        break;
      }
      tc_fence_after();
      if (idle) {  // P of these rows is never read back: hand S straight on
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + x);
        continue;
      }
      const int valid = kv_mine - j * BN;
      float s[64];
      uint32_t* su = reinterpret_cast<uint32_t*>(s);
      tmem_ld32(tS + 64, su);
      tmem_ld32(tS + 96, su + 32);
      tmem_ld_wait();
      if (valid < BN) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c + 64 >= valid) s[c] = -INFINITY;
      }
      const float mx_hi = max64(s);
      tmem_ld32(tS + 0, su);
      tmem_ld32(tS + 32, su + 32);
      tmem_ld_wait();
      if (valid < 64) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= valid) s[c] = -INFINITY;
      }
      const float m_new = fmaxf(max64(s), mx_hi) * sl2;
      // Lazy rescaling: a row's reference max only moves when the tile max
      // exceeds it by more than the threshold.  TMEM loads/stores are
      // warp-collective, so the whole warp enters the rescale when any of its
      // rows needs it (f = 1 for the others).  PV_x(j-1) has completed: it
      // was issued before QK_x(j), whose completion this warp has seen.
      const bool need = (j > 0) && (m_new > m_run + (kE4 ? kRescaleThresholdF16 : kRescaleThreshold));
      if (j == 0) m_run = m_new;
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? ex2(m_run - m_new) : 1.f;
        l_f32 *= f;
        l_b16 *= f;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t o[16];
          tmem_ld16(tO + c * 16, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(f * __uint_as_float(o[i]));
          tmem_st16(tO + c * 16, o);
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
      for (int h = 0; h < 2; ++h) {
        if (h == 1) {
          tmem_ld32(tS + 64, su);
          tmem_ld32(tS + 96, su + 32);
          tmem_ld_wait();
          if (valid < BN) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c + 64 >= valid) s[c] = -INFINITY;
          }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[32 * c + 2 * i], s[32 * c + 2 * i + 1]), c2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            pk[i] = kE4 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
            accf[i & 3] = f2_add(accf[i & 3], f2_pack(p0, p1));
            if constexpr (kE4) {
              const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&pk[i]));
              accb[i & 3] = f2_add(accb[i & 3], f2_pack(r.x, r.y));
            } else {
              accb[i & 3] = f2_add(accb[i & 3], f2_pack(__uint_as_float(pk[i] << 16),
                                                        __uint_as_float(pk[i] & 0xFFFF0000u)));
            }
          }
          tmem_st16(tS + h * 32 + c * 16, pk);
        }
      }
      l_f32 += sum8(accf);
      l_b16 += sum8(accb);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + x);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && wait_batch(2 * nkv + x - 1)) {  // the last PV_x complete
      tc_fence_after();
      const float inv_l = (kE4 ? a.v_scale : 1.f) / l_b16;
      const int unit = 2 * pair + x;
      int token;
      if (!kSparseMode) {
        token = unit * BM + row;
        if (token >= a.N) token = -1;
      } else {
        // a pair's 2C rows are the perm rows of its two groups (the second
        // may not exist when G is odd)
        const int g0 = kPairs ? 2 * unit : unit;
        const int qrows = kPairs ? (g0 + 1 < a.G ? 2 : 1) * a.C : a.C;
        const int gr = row - qoff(x);
        token = (!idle && gr >= 0 && gr < qrows && (x == 0 || has_b))
                    ? __ldg(a.perm + (static_cast<size_t>(bh) * a.G + g0) * a.C + gr)
                    : -1;
        if (token >= a.N) token = -1;
      }
      const size_t row_off =
          static_cast<size_t>(rm.rbase + (token < 0 ? 0 : token) * rm.rstride) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait();
        if (token >= 0) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * inv_l;
          if (kBase == kSparseAdd || kBase == kSparseRecord) {
            const uint4* src = reinterpret_cast<const uint4*>(a.aux_in + row_off + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w = __ldg(src + q4);
              const __nv_bfloat162* hh = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float2 f2 = __bfloat1622float2(hh[e]);
                const int i0 = q4 * 8 + 2 * e;
                if (kBase == kSparseAdd) {
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
      if (!kSparseMode && a.lse != nullptr && token >= 0)
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
  constexpr bool kPairs = (MODE & kPaired) != 0;
  const int smem = AttnLayout<D, kPairs>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int units = (MODE == kDense) ? (a.N + BM - 1) / BM : (kPairs ? a.P : a.G);
  kern<<<dim3((units + 1) / 2, BH), kThreads, smem, stream>>>(*tq, *tk, *tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(int D, int mode, const CUtensorMap* tq, const CUtensorMap* tk,
                             const CUtensorMap* tv, const AttnArgs& a, int BH,
                             cudaStream_t stream) {
#define MCS_ATTN_CASE(DD, MM) \
  if (D == (DD) && mode == (MM)) return launch_one<DD, MM>(tq, tk, tv, a, BH, stream);
  MCS_ATTN_CASE(128, kDense)
  MCS_ATTN_CASE(128, kSparse)
  MCS_ATTN_CASE(128, kSparseAdd)
  MCS_ATTN_CASE(128, kSparseRecord)
  MCS_ATTN_CASE(64, kDense)
  MCS_ATTN_CASE(64, kSparse)
  MCS_ATTN_CASE(64, kSparseAdd)
  MCS_ATTN_CASE(64, kSparseRecord)
  MCS_ATTN_CASE(128, kSparse | kPaired)
  MCS_ATTN_CASE(128, kSparseAdd | kPaired)
  MCS_ATTN_CASE(128, kSparseRecord | kPaired)
  MCS_ATTN_CASE(64, kSparse | kPaired)
  MCS_ATTN_CASE(64, kSparseAdd | kPaired)
  MCS_ATTN_CASE(64, kSparseRecord | kPaired)
  MCS_ATTN_CASE(128, kSparse | kE4M3)
  MCS_ATTN_CASE(128, kSparseAdd | kE4M3)
  MCS_ATTN_CASE(64, kSparse | kE4M3)
  MCS_ATTN_CASE(64, kSparseAdd | kE4M3)
#undef MCS_ATTN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mcs
