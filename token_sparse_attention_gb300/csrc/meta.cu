// Metadata cache entries and their staging between host and device memory.
//
// A layer's cached metadata -- the groups (perm), the selected KV indices
// (idx) and the dense-minus-sparse residual -- is written at the anchor step
// and read at each reuse step of that layer.  When device memory is short the
// entries of inactive layers are kept in host memory and prefetched one layer
// ahead, so that the copy overlaps the current layer's sparse attention (ai.info
// AI summary, "Main Findings"; wispaper.ai, "Speedups come with negligible
// measured quality loss").  On a Grace-Blackwell node the host memory sits
// behind NVLink-C2C, so an entry of a few GB moves in a fraction of a layer's
// attention time.
//
// An entry stores each group's KV indices as a bitmap of N bits (bit j set:
// token j kept) rather than K int32 values: N/8 bytes instead of 4K, 6.4x
// fewer at density 0.2, which shrinks the large workload's entry from 2.2 to
// 1.0 GB.  mcs_meta_pack writes the bitmaps from an index list after the
// anchor; mcs_meta_unpack rebuilds the ascending list on the device before a
// reuse step (one pass over the bitmaps, ~0.3 ms for the large workload).
//
// The stager only orders copies: each copy is queued on the caller's copy
// stream behind an event recorded on the stream that last used (prefetch) or
// wrote (offload) the slot, and records the slot's event when done, which
// mcs_stager_wait makes a compute stream wait for.  An entry is one flat
// buffer with the same layout on both sides, so each move is one
// cudaMemcpyAsync.
#include <new>
#include <vector>

#include "internal.h"
#include "mcs.h"

struct mcs_stager {
  size_t bytes = 0;
  cudaStream_t copy = nullptr;
  std::vector<void*> slots;
  std::vector<cudaEvent_t> copied;  // per slot: its last queued copy
  cudaEvent_t order = nullptr;      // "work queued so far on `after`"
};

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct MetaLayout {
  size_t perm, idx, residual, total;
  int words;  // bitmap words per group
};

MetaLayout meta_layout(const mcs_params* p) {
  const size_t BH = static_cast<size_t>(p->B) * p->H;
  const size_t G = (static_cast<size_t>(p->N) + p->C - 1) / p->C;
  MetaLayout m;
  m.words = (p->N + 31) / 32;
  m.perm = 0;
  m.idx = round_up(BH * G * p->C * sizeof(int32_t));
  m.residual = m.idx + round_up(BH * G * static_cast<size_t>(m.words) * sizeof(uint32_t));
  m.total = m.residual + round_up(BH * p->N * static_cast<size_t>(p->D) * 2);
  return m;
}

constexpr int kPackThreads = 256;

// One CTA per group: its K indices -> a bitmap of N bits built in shared
// memory (words of the CTA's row).  Indices out of range, or repeated (fewer
// than K bits set), are reported.
__global__ void __launch_bounds__(kPackThreads)
    meta_pack_kernel(const int32_t* __restrict__ idx, int K, int N, int W,
                     uint32_t* __restrict__ bits, unsigned* status) {
  extern __shared__ uint32_t sb[];
  __shared__ unsigned set;
  const size_t row = blockIdx.x;
  for (int w = threadIdx.x; w < W; w += kPackThreads) sb[w] = 0;
  if (threadIdx.x == 0) set = 0;
  __syncthreads();
  const int32_t* ir = idx + row * K;
  bool bad = false;
  for (int t = threadIdx.x; t < K; t += kPackThreads) {
    const int j = ir[t];
    if (j < 0 || j >= N) {
      bad = true;
      continue;
    }
    atomicOr(&sb[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  uint32_t* out = bits + row * W;
  unsigned mine = 0;
  for (int w = threadIdx.x; w < W; w += kPackThreads) {
    out[w] = sb[w];
    mine += __popc(sb[w]);
  }
  atomicAdd(&set, mine);
  __syncthreads();
  if (threadIdx.x == 0 && (bad || set != static_cast<unsigned>(K))) atomicOr(status, mcs::DEV_BOUNDS);
}

// One CTA per group: bitmap -> the K set positions, ascending.  Warp w owns
// a contiguous range of the row's words.  Pass 1 counts each warp's bits (all
// loads in flight at once); one block scan of the eight counts gives each
// warp its first output position; pass 2 re-reads the words (L1 hits) 32 at a
// time, places their positions in shared memory with warp scans only, and the
// finished list is written out with coalesced stores.  A row whose bitmap
// does not hold exactly K set bits is reported (at most K positions kept).
__global__ void __launch_bounds__(kPackThreads)
    meta_unpack_kernel(const uint32_t* __restrict__ bits, int W, int K,
                       int32_t* __restrict__ idx, unsigned* status) {
  extern __shared__ int32_t sidx[];  // K
  constexpr int kWarps = kPackThreads / 32;
  __shared__ unsigned warp_sums[kWarps];
  const size_t row = blockIdx.x;
  const uint32_t* br = bits + row * W;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per_warp = (W + kWarps - 1) / kWarps;
  const int wb = warp * per_warp;
  const int we = min(W, wb + per_warp);
  unsigned cnt = 0;
  for (int w = wb + lane; w < we; w += 32) cnt += __popc(br[w]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if (lane == 0) warp_sums[warp] = cnt;
  __syncthreads();
  unsigned run = 0, total = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    run += i < warp ? warp_sums[i] : 0u;
    total += warp_sums[i];
  }
  for (int base = wb; base < we; base += 32) {
    const int w = base + lane;
    uint32_t b = w < we ? br[w] : 0u;
    const unsigned c = __popc(b);
    unsigned incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    unsigned pos = run + incl - c;
    while (b != 0u) {
      const int bit = __ffs(b) - 1;
      b &= b - 1u;
      if (pos < static_cast<unsigned>(K)) sidx[pos] = w * 32 + bit;
      ++pos;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncthreads();
  int32_t* out = idx + row * K;
  const int n = total < static_cast<unsigned>(K) ? static_cast<int>(total) : K;
  if (n == K && (K & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const int4* src = reinterpret_cast<const int4*>(sidx);  // dynamic shared memory: 16-B aligned
    int4* dst = reinterpret_cast<int4*>(out);
    for (int t = threadIdx.x; t < K / 4; t += kPackThreads) dst[t] = src[t];
  } else {
    for (int t = threadIdx.x; t < n; t += kPackThreads) out[t] = sidx[t];
  }
  if (threadIdx.x == 0 && total != static_cast<unsigned>(K)) atomicOr(status, mcs::DEV_BOUNDS);
}

// Queue dst <- src on the copy stream after the work queued so far on `after`.
mcs_status stage_copy(mcs_stager* s, int slot, void* dst, const void* src, cudaMemcpyKind kind,
                      cudaStream_t after, const char* what) {
  cudaError_t e = cudaEventRecord(s->order, after);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s->copy, s->order, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, s->bytes, kind, s->copy);
  if (e == cudaSuccess) e = cudaEventRecord(s->copied[slot], s->copy);
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, what);
}

bool valid_slot(const mcs_stager* s, int slot) {
  return s != nullptr && slot >= 0 && slot < static_cast<int>(s->slots.size());
}

}  // namespace

extern "C" {

size_t mcs_meta_bytes(const mcs_params* p) {
  if (mcs::check_params(p, true) != MCS_OK) return 0;
  return meta_layout(p).total;
}

mcs_status mcs_meta_offsets(const mcs_params* p, size_t* perm_off, size_t* idx_off,
                            size_t* residual_off) {
  mcs_status st = mcs::check_params(p, true);
  if (st != MCS_OK) return st;
  const MetaLayout m = meta_layout(p);
  if (perm_off) *perm_off = m.perm;
  if (idx_off) *idx_off = m.idx;
  if (residual_off) *residual_off = m.residual;
  return MCS_OK;
}

mcs_status mcs_meta_pack(const mcs_params* p, const int32_t* idx, void* entry,
                         cudaStream_t stream) {
  mcs_status st = mcs::check_params(p, true);
  if (st != MCS_OK) return st;
  if (idx == nullptr || entry == nullptr || (reinterpret_cast<uintptr_t>(entry) % kAlign) != 0)
    return MCS_ERR_INVALID_ARG;
  const MetaLayout m = meta_layout(p);
  const size_t smem = static_cast<size_t>(m.words) * 4;
  if (smem > 200 * 1024) return MCS_ERR_UNSUPPORTED;  // N above ~1.6 M tokens
  unsigned* status;
  cudaError_t e = mcs::device_status_word(&status);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(meta_pack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  const long long rows = static_cast<long long>(p->B) * p->H * ((p->N + p->C - 1) / p->C);
  if (e == cudaSuccess) {
    meta_pack_kernel<<<static_cast<unsigned>(rows), kPackThreads, smem, stream>>>(
        idx, p->K, p->N, m.words,
        reinterpret_cast<uint32_t*>(static_cast<char*>(entry) + m.idx), status);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, "meta pack launch");
}

mcs_status mcs_meta_unpack(const mcs_params* p, const void* entry, int32_t* idx,
                           cudaStream_t stream) {
  mcs_status st = mcs::check_params(p, true);
  if (st != MCS_OK) return st;
  if (idx == nullptr || entry == nullptr || (reinterpret_cast<uintptr_t>(entry) % kAlign) != 0)
    return MCS_ERR_INVALID_ARG;
  const MetaLayout m = meta_layout(p);
  const size_t smem = static_cast<size_t>(p->K) * 4;
  if (smem > 200 * 1024) return MCS_ERR_UNSUPPORTED;  // K above 51200
  unsigned* status;
  cudaError_t e = mcs::device_status_word(&status);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(meta_unpack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  const long long rows = static_cast<long long>(p->B) * p->H * ((p->N + p->C - 1) / p->C);
  if (e == cudaSuccess) {
    meta_unpack_kernel<<<static_cast<unsigned>(rows), kPackThreads, smem, stream>>>(
        reinterpret_cast<const uint32_t*>(static_cast<const char*>(entry) + m.idx), m.words, p->K,
        idx, status);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, "meta unpack launch");
}

mcs_status mcs_stager_create(const mcs_params* p, int slots, void* const* device_slots,
                             cudaStream_t copy_stream, mcs_stager** out) {
  if (out == nullptr) return MCS_ERR_INVALID_ARG;
  *out = nullptr;
  mcs_status st = mcs::check_params(p, true);
  if (st != MCS_OK) return st;
  if (slots < 1 || device_slots == nullptr) return MCS_ERR_INVALID_ARG;
  for (int i = 0; i < slots; ++i)
    if (device_slots[i] == nullptr || (reinterpret_cast<uintptr_t>(device_slots[i]) % kAlign) != 0)
      return MCS_ERR_INVALID_ARG;
  mcs_stager* s = new (std::nothrow) mcs_stager;
  if (s == nullptr) return MCS_ERR_INVALID_ARG;
  s->bytes = meta_layout(p).total;
  s->copy = copy_stream;
  s->slots.assign(device_slots, device_slots + slots);
  s->copied.assign(slots, nullptr);
  cudaError_t e = cudaEventCreateWithFlags(&s->order, cudaEventDisableTiming);
  for (int i = 0; e == cudaSuccess && i < slots; ++i)
    e = cudaEventCreateWithFlags(&s->copied[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    mcs_stager_destroy(s);
    return mcs::record_cuda_error(e, "cudaEventCreate(stager)");
  }
  *out = s;
  return MCS_OK;
}

void mcs_stager_destroy(mcs_stager* s) {
  if (s == nullptr) return;
  for (cudaEvent_t ev : s->copied)
    if (ev != nullptr) cudaEventDestroy(ev);
  if (s->order != nullptr) cudaEventDestroy(s->order);
  delete s;
}

mcs_status mcs_stager_prefetch(mcs_stager* s, int slot, const void* host_entry,
                               cudaStream_t after) {
  if (!valid_slot(s, slot) || host_entry == nullptr) return MCS_ERR_INVALID_ARG;
  return stage_copy(s, slot, s->slots[slot], host_entry, cudaMemcpyHostToDevice, after,
                    "stager prefetch");
}

mcs_status mcs_stager_offload(mcs_stager* s, int slot, void* host_entry, cudaStream_t after) {
  if (!valid_slot(s, slot) || host_entry == nullptr) return MCS_ERR_INVALID_ARG;
  return stage_copy(s, slot, host_entry, s->slots[slot], cudaMemcpyDeviceToHost, after,
                    "stager offload");
}

mcs_status mcs_stager_wait(mcs_stager* s, int slot, cudaStream_t stream) {
  if (!valid_slot(s, slot)) return MCS_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamWaitEvent(stream, s->copied[slot], 0);
  return e == cudaSuccess ? MCS_OK : mcs::record_cuda_error(e, "stager wait");
}

}  // extern "C"
