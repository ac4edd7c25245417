// Internal launcher declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#include "mcs.h"

namespace mcs {

// Records "what: <CUDA error string>" as the thread's last CUDA error and
// returns MCS_ERR_CUDA.
mcs_status record_cuda_error(cudaError_t e, const char* what);
// The shape checks every entry point applies (need_k: K must be in [1, N]).
mcs_status check_params(const mcs_params* p, bool need_k);

// Device status bits, OR-ed into the library's status word.
enum : unsigned {
  DEV_TIMEOUT = 1u,  // a bounded wait gave up
  DEV_BOUNDS = 2u,   // an index read from an argument was out of range
};

// Rows of the [B,H,N,D] (layout 0) or [B,N,H,D] (layout 1) bf16 tensors q, k,
// v, out, dense_out and residual, viewed as [B*H*N, D]: the vector of head
// bh = b*H + h at token t is row rbase + t * rstride.
struct RowMap {
  int rbase, rstride;
};
__host__ __device__ __forceinline__ RowMap row_map(int layout, int H, int N, int bh) {
  RowMap m;
  if (layout == 1) {
    m.rbase = (bh / H) * N * H + bh % H;
    m.rstride = H;
  } else {
    m.rbase = bh * N;
    m.rstride = 1;
  }
  return m;
}

// Attention kernel modes.
enum AttnMode : int {
  kDense = 0,         // dense attention, writes O (+ LSE)
  kSparse = 1,        // token-sparse attention, writes O' scattered to perm rows
  kSparseAdd = 2,     // token-sparse attention + cached residual (reuse step)
  kSparseRecord = 3,  // token-sparse attention, writes residual = dense_out - O' (anchor)
  kPaired = 4,        // flag on a sparse mode: C = 64 sibling pairs over their key unions
  kE4M3 = 8,          // flag on kSparse / kSparseAdd: K and V are E4M3 bytes (k8, v8)
};

// Sibling-pair key lists (C = 64): groups 2u and 2u+1 of a head form pair u
// (P = ceil(G/2) pairs; the last pair has one group when G is odd).  Each
// pair's list is the ascending union of the two groups' index sets, entry =
// token | (in group 2u) << 28 | (in group 2u+1) << 29, padded to `cap`
// entries (token 0, in neither group).  Buffer: lens [BH*P] int32, then
// entries [BH*P, cap] int32 at a 256-byte aligned offset.
struct PairLayout {
  int P, cap;
  size_t entries_off, total;
};
__host__ __device__ inline PairLayout pair_layout(int BH, int G, int K) {
  PairLayout l;
  l.P = (G + 1) / 2;
  l.cap = (2 * K + 127) / 128 * 128;
  l.entries_off = ((size_t)BH * l.P * 4 + 255) / 256 * 256;
  l.total = l.entries_off + (size_t)BH * l.P * l.cap * 4;
  return l;
}
constexpr int kPairMaxK = 16384;           // the union kernel keeps 3K + 1 ints in shared memory
constexpr int kPairTokenBits = 28;         // tokens below 2^28
constexpr float kPairMaskBias = -1048576.f;  // -2^20: added to the scores of other groups' keys

struct AttnArgs {
  int H, layout;     // heads per batch entry; tensor layout (see RowMap)
  int N;             // tokens per head
  int C;             // queries per group (sparse modes)
  int G;             // groups per head (sparse modes)
  int K;             // selected KV tokens per group (sparse modes)
  float scale_log2;  // softmax scale * log2(e)
  __nv_bfloat16* out;            // [BH, N, D]; kSparseRecord: residual out
  float* lse;                    // [BH, N] natural-log LSE (kDense, nullable)
  const int32_t* perm;           // [BH, G*C]
  const int32_t* idx;            // [BH, G, K]
  const __nv_bfloat16* aux_in;   // kSparseAdd: residual; kSparseRecord: dense_out
  const __nv_bfloat16* q;        // [BH, N, D] (rows of the query tile / group)
  const __nv_bfloat16* k;        // [BH, N, D] (sparse modes: rows gathered by idx)
  const __nv_bfloat16* v;        // [BH, N, D]
  unsigned* status;              // device status word
  int fault;                     // test-only: 1 = producers stop after the first K/V tile
  // kE4M3: K and V as E4M3 bytes [BH, N, D] (rows as for k, v); the K scale
  // is folded into scale_log2, the V scale multiplies the output
  const uint8_t* k8;
  const uint8_t* v8;
  float v_scale;
  // kPaired: pair lists (see PairLayout)
  int P, cap;
  const int32_t* plen;           // [BH, P]
  const int32_t* pidx;           // [BH, P, cap]
};

// tq/tk/tv: dense -> 4-D tile maps [B][H][N][D] in the tensors' layout, box
//           {64,128,1,1}, coordinates (d, token, h, b);
//           sparse -> 2-D gather maps [B*H*N rows][D], box {64,1}.
cudaError_t launch_attention(int D, int mode, const CUtensorMap* tq, const CUtensorMap* tk,
                             const CUtensorMap* tv, const AttnArgs& a, int BH,
                             cudaStream_t stream);

// Bins of the group-mass digit histogram: digit = top 12 bits of the fp32
// mass (sign, exponent, three mantissa bits).  A group's masses are at most
// its size C <= 128 (up to rounding), whose digits are <= 1072; larger digits
// (masses of 256 or more, infinities, NaNs) fall in the last bin.
constexpr int kMassHistBins = 1088;

struct MassArgs {
  int H, layout;          // heads per batch entry; tensor layout (see RowMap)
  int N, C, G;
  int head0;              // first (b*H+h) head of this chunk
  float scale_log2;
  const int32_t* perm;    // [BH, G*C]
  const float* lse;       // [BH, N]
  float* mass;            // [heads in chunk, G, N]
  uint32_t* hist;         // [heads in chunk, G, kMassHistBins] digit counts per mass row, or null
  unsigned* status;
};

// tq: 2-D gather map over the rows of Q; tk: 4-D tile map over K.
cudaError_t launch_group_mass(int D, const CUtensorMap* tq, const CUtensorMap* tk,
                              const MassArgs& a, int heads, cudaStream_t stream);

// rows x n masses -> rows x K ascending indices (+ retained sums, nullable).
// hist (nullable): each row's digit histogram written by the mass
// kernel; with it most rows are selected in one read of their masses.
cudaError_t launch_topk(const float* mass, const uint32_t* hist, int rows, int n, int K,
                        int32_t* idx, float* retained, unsigned* status, cudaStream_t stream);

// idx [BH, G, K] (rows ascending) -> pair lists in `pairs` (PairLayout).
cudaError_t launch_pair_union(const int32_t* idx, int BH, int G, int K, int N, void* pairs,
                              unsigned* status, cudaStream_t stream);

// x8[i] = E4M3(x[i] / scale) for n bf16 values (x and x8 16-byte aligned).
cudaError_t launch_quantize_e4m3(const __nv_bfloat16* x, size_t n, float scale, uint8_t* x8,
                                 cudaStream_t stream);

// Device address of the library's status word (for kernels' status argument).
cudaError_t device_status_word(unsigned** out);
size_t pddp_workspace_bytes(int BH, int N, int D, int C);
// Groups heads [head0, head0 + BH) of q (all B*H heads, in `layout`, H heads
// per batch entry).  perm_out points at the first of those heads' perm rows.
cudaError_t launch_pddp(const __nv_bfloat16* q, int layout, int H, int head0, int BH, int N,
                        int D, int C, int iters, int32_t* perm_out, void* ws, size_t ws_bytes,
                        unsigned* status, cudaStream_t stream);

}  // namespace mcs
