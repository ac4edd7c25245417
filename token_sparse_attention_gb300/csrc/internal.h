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

// Attention kernel modes.
enum AttnMode : int {
  kDense = 0,         // dense attention, writes O (+ LSE)
  kSparse = 1,        // token-sparse attention, writes O' scattered to perm rows
  kSparseAdd = 2,     // token-sparse attention + cached residual (reuse step)
  kSparseRecord = 3,  // token-sparse attention, writes residual = dense_out - O' (anchor)
};

struct AttnArgs {
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
};

// tq/tk/tv: dense -> 3-D tile maps [BH][N][D], box {64,128,1};
//           sparse -> 2-D gather maps [BH*N][D], box {64,1}.
cudaError_t launch_attention(int D, int mode, const CUtensorMap* tq, const CUtensorMap* tk,
                             const CUtensorMap* tv, const AttnArgs& a, int BH,
                             cudaStream_t stream);

struct MassArgs {
  int N, C, G;
  int head0;              // first (b*H+h) head of this chunk
  float scale_log2;
  const int32_t* perm;    // [BH, G*C]
  const float* lse;       // [BH, N]
  float* mass;            // [heads in chunk, G, N]
  uint32_t* hist;         // [heads in chunk, G, 2048] digit counts of each mass row, or null
  unsigned* status;
};

// tq: 2-D gather map over Q [BH*N][D]; tk: 3-D tile map over K.
cudaError_t launch_group_mass(int D, const CUtensorMap* tq, const CUtensorMap* tk,
                              const MassArgs& a, int heads, cudaStream_t stream);

// rows x n masses -> rows x K ascending indices (+ retained sums, nullable).
// hist (nullable): each row's 2048-bin digit histogram written by the mass
// kernel; with it most rows are selected in one read of their masses.
cudaError_t launch_topk(const float* mass, const uint32_t* hist, int rows, int n, int K,
                        int32_t* idx, float* retained, unsigned* status, cudaStream_t stream);

// Device address of the library's status word (for kernels' status argument).
cudaError_t device_status_word(unsigned** out);
// 2-D gather tensor map over `rows` bf16 rows of D columns (box {64, 1}).
bool encode_gather_map(CUtensorMap* m, const void* base, long long rows, int D);

size_t pddp_workspace_bytes(int BH, int N, int D, int C);
cudaError_t launch_pddp(const __nv_bfloat16* q, const CUtensorMap* tq_gather, int BH, int N, int D,
                        int C, int iters, int32_t* perm_out, void* ws, size_t ws_bytes,
                        unsigned* status, cudaStream_t stream);

}  // namespace mcs
