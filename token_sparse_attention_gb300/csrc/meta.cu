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
};

MetaLayout meta_layout(const mcs_params* p) {
  const size_t BH = static_cast<size_t>(p->B) * p->H;
  const size_t G = (static_cast<size_t>(p->N) + p->C - 1) / p->C;
  MetaLayout m;
  m.perm = 0;
  m.idx = round_up(BH * G * p->C * sizeof(int32_t));
  m.residual = m.idx + round_up(BH * G * static_cast<size_t>(p->K) * sizeof(int32_t));
  m.total = m.residual + round_up(BH * p->N * static_cast<size_t>(p->D) * 2);
  return m;
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
