/*
 * mcs.h -- C ABI of the MC-Sparse token-sparse attention library (libmcs.so)
 * for NVIDIA GB300 (sm_103a).
 *
 * Method: "MC-Sparse: Deconstructing and Closing the Dense-Sparse Attention
 * Gap in Diffusion Transformers".  Each tile-aligned group of C similar
 * queries of one head attends only to its own K selected KV tokens, gathered
 * by index; groups, KV indices and the dense-minus-sparse residual are
 * computed at anchor steps and reused at the reuse steps in between.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned DEVICE memory, contiguous, row-major:
 *      q, k, v, out, dense_out, residual : [B, H, N, D] bfloat16, or
 *                                          [B, N, H, D] when p->layout is
 *                                          MCS_LAYOUT_BNHD (as DiT blocks
 *                                          hold them); results are identical
 *      lse                               : [B, H, N]    float32 (natural log)
 *      perm                              : [B, H, G*C]  int32, G = ceil(N/C)
 *      idx                               : [B, H, G, K] int32
 *      mass                              : [heads, G, N] float32
 *    Pointers to bf16 tensors must be 16-byte aligned.
 *  - perm: entry g*C + p is the original token index of query p of group g;
 *    the unused slots of the short last group (when C does not divide N) are
 *    -1.  Within a group indices are ascending.
 *  - idx: the selected KV token indices of each group, ascending.
 *  - Calls are asynchronous on `stream`; outputs are valid once the stream
 *    has reached the call.  Arguments are checked on the host before any
 *    launch; on a check failure nothing is launched and a status is returned.
 *  - Faults found on the device (an index out of range, a bounded wait that
 *    gave up) are OR-ed into a device status word read by mcs_device_status.
 *    Kernels never trap.
 *  - The library allocates no memory.  Entry points that need scratch take
 *    a caller-provided device workspace (size from the *_workspace queries).
 *    Apart from the device status word and the stager objects the caller
 *    creates and destroys (mcs_stager_*: a few CUDA events each) it holds no
 *    state between calls.
 *  - Supported: D in {64, 128}, C in {64, 128}, 1 <= K <= N, B*H <= 65535.
 */
#ifndef MCS_H_
#define MCS_H_

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MCS_OK = 0,
  MCS_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
  MCS_ERR_UNSUPPORTED = 2, /* D, C outside the supported set */
  MCS_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  MCS_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (mcs_last_cuda_error) */
  MCS_ERR_TIMEOUT = 5,     /* a device-side bounded wait gave up */
  MCS_ERR_BOUNDS = 6       /* a perm/idx entry was outside [0, N) on the device */
} mcs_status;

typedef struct {
  int B, H, N, D;  /* batch, heads, tokens per head, head dim */
  int C;           /* queries per group (the kernel's query tile) */
  int K;           /* selected KV tokens per group: round(density * N) */
  float scale;     /* softmax scale; 0 selects 1/sqrt(D) */
  int pddp_iters;  /* power-iteration steps per PDDP node; 0 selects 32 */
  int layout;      /* MCS_LAYOUT_BHND (0) or MCS_LAYOUT_BNHD (1): see below */
} mcs_params;

/* Layout of the bf16 activations q, k, v, out, dense_out and residual. */
enum { MCS_LAYOUT_BHND = 0, MCS_LAYOUT_BNHD = 1 };

/* Human-readable name of a status code (static string). */
const char* mcs_status_string(mcs_status s);

/* Message of the last CUDA error seen by this thread (static per thread). */
const char* mcs_last_cuda_error(void);

/*
 * Device status: synchronises `stream`, returns the first device-side fault
 * recorded since the previous call (MCS_ERR_TIMEOUT, MCS_ERR_BOUNDS) or
 * MCS_OK, and clears the word.
 */
mcs_status mcs_device_status(cudaStream_t stream);

/* Workspace bytes needed by mcs_group and by mcs_anchor_select. */
size_t mcs_group_workspace(const mcs_params* p);
size_t mcs_anchor_workspace(const mcs_params* p);

/*
 * a1 -- Fast PDDP query grouping.  Source: wispaper.ai, "Token-level
 * selection needs tile-aligned query groups" (median split along each
 * group's principal direction until every group holds C queries); ai.info
 * AI summary, "Methodology in Plain English" / "Key Contributions" (batched
 * power iteration over all heads per tree depth, only index arrays passed
 * between levels).
 * Reads q [B,H,N,D]; writes perm [B,H,G*C].  For a node of n rows and
 * g = ceil(n/C) groups, the left child takes the C*floor(g/2) rows of
 * smallest projection (ties by token index); the principal direction is
 * pddp_iters power-iteration steps from (1,...,1)/sqrt(D), sign fixed so its
 * largest-magnitude component is positive.  Leaves in tree order, indices
 * ascending within a group, the short group last.
 * ws: device workspace of at least mcs_group_workspace(p) bytes.
 */
mcs_status mcs_group(const mcs_params* p, const void* q, int32_t* perm, void* ws, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * a2 -- Dense attention with per-query log-sum-exp: the selector's first
 * pass, which yields both the dense output and every row's LSE (ai.info AI
 * summary, "Methodology in Plain English"), and the speedup baseline.
 * out = softmax(scale * q k^T) v  [B,H,N,D] bf16;
 * lse = log sum_j exp(scale * q_i.k_j)  [B,H,N] fp32, nullable.
 */
mcs_status mcs_dense_attn(const mcs_params* p, const void* q, const void* k, const void* v,
                          void* out, float* lse, cudaStream_t stream);

/*
 * a3 -- Exact group attention mass, the selector's second pass (ai.info AI
 * summary, "Methodology in Plain English"; agihunt.info summary, paragraph on
 * the selection objective): for heads [head_begin, head_begin + head_count)
 * (numbered b*H + h) and every group g,
 *     mass[h - head_begin, g, j] = sum_{i in group g} exp(scale*q_i.k_j - lse_i).
 * Padding slots (perm = -1) contribute nothing.  mass: [head_count, G, N] fp32.
 */
mcs_status mcs_group_mass(const mcs_params* p, const void* q, const void* k, const float* lse,
                          const int32_t* perm, int head_begin, int head_count, float* mass,
                          cudaStream_t stream);

/*
 * a4 -- Per-group top-K (agihunt.info summary, paragraph on the selection
 * objective: the K KV tokens of largest group attention weight).  For each of
 * `rows` rows of p->N non-negative masses, writes the K indices of largest
 * mass (ties to the lower index) in ascending order to idx [rows, K] and,
 * when `retained` is not NULL, the sum of their masses to retained [rows].
 */
mcs_status mcs_topk(const mcs_params* p, const float* mass, int rows, int32_t* idx,
                    float* retained, cudaStream_t stream);

/*
 * a3 + a4 as the anchor step runs them (ai.info AI summary, "Methodology in
 * Plain English": the second selector pass fuses group aggregation with
 * top-K).  From q, k, the dense pass's lse and the groups perm, writes idx
 * [B,H,G,K] (each group's K KV indices of largest mass, ties to the lower
 * index, ascending) and, when `retained` is not NULL, retained [B,H,G] (their
 * mass sums): the same results as mcs_group_mass followed by mcs_topk.  Each
 * group's masses are histogrammed by their top 12 bits as they are computed,
 * so the top-K finds the K-th mass's bucket without reading them and reads
 * them once; a group whose bucket holds more than 4096 masses (mass ties en
 * masse) is selected in four reads instead.
 * ws: device workspace through which the masses and histograms pass, heads
 * in chunks: mcs_anchor_workspace(p) bytes process every head at once (up to
 * 4 GiB); at least G*(N+1088)*4 bytes (each part rounded up to 256) are
 * needed.  Requires K <= N.
 */
mcs_status mcs_select(const mcs_params* p, const void* q, const void* k, const float* lse,
                      const int32_t* perm, int32_t* idx, float* retained, void* ws,
                      size_t ws_bytes, cudaStream_t stream);

/*
 * a5 + a6 -- Token-sparse attention (wispaper.ai, "Token-level selection
 * needs tile-aligned query groups"; "Residual correction recovers the
 * discarded tail").  For every group g of every head: the group's queries
 * attend to the K rows idx[b,h,g,:] of k and v only (softmax renormalised
 * over those K), and the result of query row perm[g*C+p] is written to that
 * row of out.  When `residual` is not NULL it is added (reuse step):
 * out = O' + residual.
 */
mcs_status mcs_sparse_attn(const mcs_params* p, const void* q, const void* k, const void* v,
                           const int32_t* perm, const int32_t* idx, const void* residual,
                           void* out, cudaStream_t stream);

/*
 * Anchor form of a5 (wispaper.ai, "Residual correction recovers the
 * discarded tail": recording the residual costs one sparse evaluation and
 * an elementwise subtraction): residual = bf16(dense_out - O'), rows in
 * original token order.
 */
mcs_status mcs_sparse_attn_record(const mcs_params* p, const void* q, const void* k,
                                  const void* v, const int32_t* perm, const int32_t* idx,
                                  const void* dense_out, void* residual, cudaStream_t stream);

/*
 * E4M3 K/V cache for the token-sparse step.  The pages leave attention over
 * low-precision operands open (ai.info AI summary, "Future Directions",
 * comparability with low-precision attention); this is the library's form of
 * it.  E4M3 is the OCP 8-bit floating point format: sign, 4 exponent bits
 * (bias 7), 3 mantissa bits, no infinities, largest finite magnitude 448.
 *
 * mcs_quantize_e4m3: x8[i] = E4M3(x[i] / scale) for n bf16 values: the
 *   quotient in fp32 (correctly rounded), rounded to the nearest E4M3 value
 *   (ties to even), magnitudes above 448 saturating to +-448, NaN to a NaN
 *   code.  x (bf16) and x8 (bytes) are device buffers, 16-byte aligned; any
 *   n (0 launches nothing).  scale > 0 and finite, else
 *   MCS_ERR_INVALID_ARG.
 * mcs_sparse_attn_e4m3: mcs_sparse_attn with K and V read from E4M3 bytes
 *   k8, v8 (same shape and layout as k and v, one byte per element, 16-byte
 *   aligned) standing for k = k_scale * k8 and v = v_scale * v8 (one scale
 *   per tensor, > 0 and finite).  The products run on f16 operands: q is
 *   converted from bf16 to f16 (exact inside the f16 range; magnitudes above
 *   65504 saturate), the K and V values are exact in f16, and the attention
 *   weights are rounded to f16.  residual NULL: out = O'; else out = O' +
 *   residual.  Same shapes, checks and device status as mcs_sparse_attn.
 */
mcs_status mcs_quantize_e4m3(const void* x, size_t n, float scale, void* x8,
                             cudaStream_t stream);
mcs_status mcs_sparse_attn_e4m3(const mcs_params* p, const void* q, const void* k8,
                                const void* v8, float k_scale, float v_scale,
                                const int32_t* perm, const int32_t* idx, const void* residual,
                                void* out, cudaStream_t stream);

/*
 * Sibling-pair key lists for C = 64 groups: a kernel layout of idx, not a
 * step of the method.  A C = 64 group fills half of the 128-row query tile of
 * the tensor-core MMA, and a 64-row MMA takes as long as a 128-row one.
 * Groups 2u and 2u+1 are siblings of the grouping tree (similar queries, so
 * their index sets overlap heavily); mcs_sparse_attn_pairs runs them as one
 * 128-row tile over the union of their index sets, adding -2^20 to the
 * scores of keys a row's group did not select (through one more tensor-core
 * step), so that every query still attends to exactly its own group's K
 * tokens (wispaper.ai, "Token-level selection needs tile-aligned query
 * groups"): results match mcs_sparse_attn up to summation order, on about
 * |A u B| / 2K of the tensor work.
 *
 * mcs_pair_bytes: size of the pair-list buffer (0 when unsupported).
 * mcs_pair_lists: idx [B,H,G,K] (rows ascending) -> pairs, a device buffer of
 *   at least mcs_pair_bytes(p) bytes, 256-byte aligned (its layout is the
 *   library's; build it once per anchor, like idx).  Requires C = 64,
 *   K <= 16384, N < 2^28 (MCS_ERR_UNSUPPORTED otherwise); an index outside
 *   [0, N) sets MCS_ERR_BOUNDS in the device status.
 * mcs_sparse_attn_pairs / _pairs_record: as mcs_sparse_attn /
 *   mcs_sparse_attn_record with the pair lists in place of idx.
 */
size_t mcs_pair_bytes(const mcs_params* p);
mcs_status mcs_pair_lists(const mcs_params* p, const int32_t* idx, void* pairs,
                          size_t pairs_bytes, cudaStream_t stream);
mcs_status mcs_sparse_attn_pairs(const mcs_params* p, const void* q, const void* k,
                                 const void* v, const int32_t* perm, const void* pairs,
                                 const void* residual, void* out, cudaStream_t stream);
mcs_status mcs_sparse_attn_pairs_record(const mcs_params* p, const void* q, const void* k,
                                        const void* v, const int32_t* perm, const void* pairs,
                                        const void* dense_out, void* residual,
                                        cudaStream_t stream);

/*
 * The whole anchor step (wispaper.ai, "Reused exact selection beats
 * recomputed mean pooling"; "Residual correction recovers the discarded
 * tail"): a1 grouping -> perm; a2 dense attention -> dense_out (the step's
 * output) and lse; a3 + a4 exact selection (as mcs_select) -> idx (and
 * retained mass [B,H,G], nullable); a5 anchor form -> residual.
 * ws: device workspace of at least mcs_anchor_workspace(p) bytes; a smaller
 * one (but at least one head's group masses and histograms, G*(N+1088)*4
 * bytes rounded up to 256-byte multiples, and the grouping workspace)
 * processes fewer heads per selection pass.
 */
mcs_status mcs_anchor_select(const mcs_params* p, const void* q, const void* k, const void* v,
                             int32_t* perm, int32_t* idx, void* dense_out, float* lse,
                             void* residual, float* retained, void* ws, size_t ws_bytes,
                             cudaStream_t stream);

/*
 * Query grouping (as mcs_group) for callers that cannot allocate device
 * memory.  No counterpart in the paper: this is a deployment variant.
 *
 * Some host programs cannot hand this library a workspace: a plugin inside
 * another framework may be given only its input and output buffers, and
 * servers that fix their memory footprint at start-up forbid any device
 * allocation afterwards.  This entry point needs neither a workspace nor an
 * allocation: its scratch is a 64 MiB array compiled into the library, which
 * every GPU that loads this part of the library keeps until the process
 * exits.  It calls no cudaMalloc, cudaFree or allocating library routine.
 *
 * Same arguments and results as mcs_group, without ws/ws_bytes; heads are
 * processed a batch at a time so that each batch fits the scratch.  Returns
 * MCS_ERR_WORKSPACE, launching nothing, when a single head needs more than
 * the 64 MiB (mcs_group_workspace for B = H = 1 exceeds 64 MiB).
 * Every call looks up the array's device address with the caller's device
 * current, so a context destroyed and created again (cudaDeviceReset) is
 * handled; the first call on each device also loads the library's kernels
 * there, so make that first call before any stream capture.  CUDA failures
 * return MCS_ERR_CUDA with the message in mcs_last_cuda_error().
 * All calls share the one array and nothing in it needs clearing between
 * calls; calls that overlap on the GPU (two streams, or two host threads)
 * race on it and must be serialised by the caller.
 */
mcs_status mcs_group_noalloc(const mcs_params* p, const void* q, int32_t* perm,
                             cudaStream_t stream);

/*
 * Metadata cache staging between host and device memory.  A layer's cached
 * metadata (groups, KV indices, residual) is produced at the anchor and read
 * at every reuse step of that layer; when device memory is short, entries of
 * inactive layers live in host memory and are prefetched one layer ahead so
 * that the copy hides behind the current layer's sparse attention (ai.info
 * AI summary, "Main Findings", on cache transfers hiding behind computation;
 * wispaper.ai, "Speedups come with negligible measured quality loss", on
 * offloading inactive cache entries to CPU memory).
 *
 * An entry is one flat buffer of mcs_meta_bytes(p) bytes holding perm
 * [B,H,G*C] int32, the selected KV indices as bitmaps [B,H,G,ceil(N/32)]
 * uint32 (bit j of group g's row set: token j kept; N/8 bytes per group
 * instead of 4K) and residual (same shape and layout as q), each at a
 * 256-byte aligned offset (mcs_meta_offsets); host and device copies share
 * the layout, so one copy moves an entry.  Both return 0 / MCS_ERR_* for
 * invalid params (K must be in [1, N]).
 */
size_t mcs_meta_bytes(const mcs_params* p);
mcs_status mcs_meta_offsets(const mcs_params* p, size_t* perm_off, size_t* idx_off,
                            size_t* residual_off);

/*
 * idx [B,H,G,K] (each row K distinct tokens in [0, N)) -> the bitmaps of the
 * device entry (256-byte aligned).  A row with an index out of range or a
 * repeated index sets MCS_ERR_BOUNDS in the device status.  N <= 1.6 M.
 */
mcs_status mcs_meta_pack(const mcs_params* p, const int32_t* idx, void* entry,
                         cudaStream_t stream);

/*
 * The bitmaps of a device entry -> idx [B,H,G,K], each row ascending.  A row
 * whose bitmap does not hold exactly K set bits sets MCS_ERR_BOUNDS in the
 * device status (it writes at most K indices).  K <= 51200.
 */
mcs_status mcs_meta_unpack(const mcs_params* p, const void* entry, int32_t* idx,
                           cudaStream_t stream);

typedef struct mcs_stager mcs_stager;

/*
 * Creates a stager over `slots` (>= 1) caller-owned device buffers of
 * mcs_meta_bytes(p) bytes each (256-byte aligned; the array is copied),
 * copying on the caller's `copy_stream`.  The stager owns one CUDA event per
 * slot plus one, freed by mcs_stager_destroy.  Host entries should be pinned
 * (page-locked) memory, or the copies are not asynchronous.  A stager is used
 * from one host thread at a time.
 */
mcs_status mcs_stager_create(const mcs_params* p, int slots, void* const* device_slots,
                             cudaStream_t copy_stream, mcs_stager** out);
void mcs_stager_destroy(mcs_stager* s);

/*
 * Queues the copy host_entry -> device slot `slot` on the copy stream, to
 * start once the work queued so far on `after` is done (pass the stream that
 * last read the slot, so that the copy does not overwrite metadata still in
 * use).  Returns without waiting.
 */
mcs_status mcs_stager_prefetch(mcs_stager* s, int slot, const void* host_entry,
                               cudaStream_t after);

/*
 * Queues the copy device slot `slot` -> host_entry on the copy stream, to
 * start once the work queued so far on `after` is done (pass the stream whose
 * work wrote the slot, e.g. the anchor step's).
 */
mcs_status mcs_stager_offload(mcs_stager* s, int slot, void* host_entry, cudaStream_t after);

/* Makes `stream` wait (on the device) for the slot's last queued copy. */
mcs_status mcs_stager_wait(mcs_stager* s, int slot, cudaStream_t stream);

/*
 * Diagnostic selectors and error measures.  The pages separate the
 * dense-sparse gap by comparing, at the same number of kept KV tokens,
 * mean-pooled block-sparse attention, a block oracle, the token oracle
 * (mcs_select) and a per-query oracle (a group of one query: mcs_group_mass +
 * mcs_topk on a perm with one query per group), by attention recall and by
 * the relative L1 error of the output (wispaper.ai, "The gap has three
 * separable sources"; wispaper.ai, "Mean-pooled block scoring misses
 * high-mass tokens"; ai.info AI summary, "Main Findings").
 *
 * KV blocks are the full blocks [b*block, (b+1)*block), b < N / block; the
 * partial block at the end is never selected.  K (p->K) must be a multiple of
 * block with K / block <= N / block, 1 <= block <= 1024.  Selected token
 * indices are ascending; ties go to the lower block.
 */
/* Workspace bytes of mcs_block_topk and mcs_pooled_block_select (all groups). */
size_t mcs_block_workspace(const mcs_params* p, int block);

/*
 * Block oracle: for each of `rows` rows of N group masses (as from
 * mcs_group_mass), keeps the K / block full KV blocks of largest summed mass;
 * idx [rows, K] (tokens of the kept blocks), retained [rows] (their mass,
 * nullable).  rows <= B*H*G.
 */
mcs_status mcs_block_topk(const mcs_params* p, const float* mass, int rows, int block,
                          int32_t* idx, float* retained, void* ws, size_t ws_bytes,
                          cudaStream_t stream);

/*
 * Mean-pooled block-sparse selection: each group (perm) scores each full KV
 * block by scale * (mean of its query rows) . (mean of the block's key rows),
 * in fp32, and keeps the K / block best; idx [B,H,G,K].
 */
mcs_status mcs_pooled_block_select(const mcs_params* p, const void* q, const void* k,
                                   const int32_t* perm, int block, int32_t* idx, void* ws,
                                   size_t ws_bytes, cudaStream_t stream);

/* retained[r] = sum_t mass[r, idx[r, t]] for rows of N masses and K indices. */
mcs_status mcs_gather_mass(const mcs_params* p, const float* mass, int rows, const int32_t* idx,
                           float* retained, cudaStream_t stream);

/*
 * Relative L1 terms of an output: sums[0] = sum |got - want|, sums[1] =
 * sum |want| (device doubles, overwritten) over the D values of each row
 * listed in rows [nrows] (indices of D-vectors in memory order: rows of the
 * bf16 tensors viewed as [B*H*N, D], in their layout), or over every row when
 * rows is NULL.
 */
mcs_status mcs_rel_l1(const mcs_params* p, const void* got, const void* want, const int32_t* rows,
                      int nrows, double* sums, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MCS_H_ */
