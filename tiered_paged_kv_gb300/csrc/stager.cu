// Host-resident history staging: pinned host memory holds every layer's history
// (the authoritative copy); the GPU keeps a bounded working set of n_slots
// caller-owned device buffers, filled asynchronously on the stager's own copy
// stream ("ActiveKV", host-authoritative KV tier: a per-layer staging working set
// with a stated budget, and fenced asynchronous staging with an explicit
// lifecycle, so a buffer is never reused while a copy or a kernel still touches
// it).
//
// Lifecycle of a slot: free -> staged (stage: the copy stream first waits for the
// slot's last release, then copies) -> acquired (acquire: the consumer stream
// waits for the copies) -> free (release: recorded on the consumer stream after
// the work that reads the slot).  The state is tracked on the host, and any call
// out of this order fails with TPK_ERR_INVALID instead of racing.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <vector>

#include "tpk.h"

namespace tpk {
void set_error(const char* msg);  // api.cu: sets the message tpk_last_error_string returns
}

enum SlotState { kFree = 0, kStaged = 1, kAcquired = 2 };

struct tpk_stager {
  int device = 0;
  size_t slot_bytes = 0;
  std::vector<char*> slots;
  std::vector<int> state;
  std::vector<cudaEvent_t> begun;   // recorded on the copy stream before a slot's copies (timing)
  std::vector<cudaEvent_t> ready;   // recorded on the copy stream after a slot's copies (timing)
  std::vector<cudaEvent_t> freed;   // recorded on the consumer stream at release
  std::vector<bool> timed;          // begun/ready bracket the slot's latest staging
  std::vector<bool> freed_recorded;
  cudaStream_t copy = nullptr;
  int next = 0;
};

namespace {

tpk_status sfail(tpk_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  tpk::set_error(buf);
  return s;
}

tpk_status scuda(cudaError_t e, const char* what) {
  return sfail(TPK_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void release_resources(tpk_stager* st) {
  if (st->copy) cudaStreamSynchronize(st->copy);
  for (cudaEvent_t e : st->begun)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : st->ready)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : st->freed)
    if (e) cudaEventDestroy(e);
  if (st->copy) cudaStreamDestroy(st->copy);
}

tpk_status check_device(const tpk_stager* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return sfail(TPK_ERR_CUDA, "no current device");
  if (dev != st->device)
    return sfail(TPK_ERR_INVALID, "stager belongs to device %d, current device is %d", st->device, dev);
  return TPK_OK;
}

tpk_status check_slot(const tpk_stager* st, int slot) {
  if (!st) return sfail(TPK_ERR_INVALID, "null stager");
  if (slot < 0 || slot >= (int)st->slots.size())
    return sfail(TPK_ERR_INVALID, "slot %d out of [0, %d)", slot, (int)st->slots.size());
  return check_device(st);
}

}  // namespace

extern "C" {

tpk_status tpk_stager_create(int n_slots, void* const* slots, size_t slot_bytes, tpk_stager** out) {
  if (!out) return sfail(TPK_ERR_INVALID, "null output pointer");
  *out = nullptr;
  if (n_slots < 1 || n_slots > 64) return sfail(TPK_ERR_INVALID, "n_slots %d out of [1, 64]", n_slots);
  if (!slots) return sfail(TPK_ERR_INVALID, "null slot array");
  if (slot_bytes == 0) return sfail(TPK_ERR_INVALID, "slot_bytes is 0");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return scuda(e, "cudaGetDevice");
  for (int i = 0; i < n_slots; ++i) {
    if (!slots[i]) return sfail(TPK_ERR_INVALID, "slot %d is null", i);
    if (reinterpret_cast<uintptr_t>(slots[i]) & 15u) return sfail(TPK_ERR_INVALID, "slot %d is not 16-byte aligned", i);
    cudaPointerAttributes a;
    e = cudaPointerGetAttributes(&a, slots[i]);
    if (e != cudaSuccess) return scuda(e, "cudaPointerGetAttributes (slot)");
    if (a.type != cudaMemoryTypeDevice || a.device != dev)
      return sfail(TPK_ERR_INVALID, "slot %d is not device memory of the current device %d", i, dev);
  }
  tpk_stager* st = new tpk_stager;
  st->device = dev;
  st->slot_bytes = slot_bytes;
  for (int i = 0; i < n_slots; ++i) st->slots.push_back(static_cast<char*>(slots[i]));
  st->state.assign(n_slots, kFree);
  st->begun.assign(n_slots, nullptr);
  st->ready.assign(n_slots, nullptr);
  st->freed.assign(n_slots, nullptr);
  st->freed_recorded.assign(n_slots, false);
  st->timed.assign(n_slots, false);
  e = cudaStreamCreateWithFlags(&st->copy, cudaStreamNonBlocking);
  for (int i = 0; e == cudaSuccess && i < n_slots; ++i) {
    e = cudaEventCreate(&st->begun[i]);
    if (e == cudaSuccess) e = cudaEventCreate(&st->ready[i]);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st->freed[i], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {
    release_resources(st);
    delete st;
    return scuda(e, "stager stream or event creation");
  }
  *out = st;
  return TPK_OK;
}

tpk_status tpk_stager_destroy(tpk_stager* st) {
  if (!st) return TPK_OK;
  tpk_status s = check_device(st);
  if (s != TPK_OK) return s;
  cudaError_t e = cudaStreamSynchronize(st->copy);
  release_resources(st);
  delete st;
  if (e != cudaSuccess) return scuda(e, "stager copy stream");
  return TPK_OK;
}

tpk_status tpk_stager_stage(tpk_stager* st, int n_regions, const void* const* host_src, const size_t* slot_offset,
                            const size_t* bytes, int* slot_out, void** slot_dev_out) {
  if (!st) return sfail(TPK_ERR_INVALID, "null stager");
  tpk_status s = check_device(st);
  if (s != TPK_OK) return s;
  if (n_regions < 0) return sfail(TPK_ERR_INVALID, "n_regions %d < 0", n_regions);
  if (n_regions > 0 && (!host_src || !slot_offset || !bytes)) return sfail(TPK_ERR_INVALID, "null region array");
  const int slot = st->next;
  if (st->state[slot] != kFree)
    return sfail(TPK_ERR_INVALID, "slot %d is still %s: release it before staging into it again", slot,
                 st->state[slot] == kStaged ? "staged" : "acquired");
  for (int i = 0; i < n_regions; ++i) {
    if (bytes[i] == 0) continue;
    if (!host_src[i]) return sfail(TPK_ERR_INVALID, "region %d: null source", i);
    if (slot_offset[i] > st->slot_bytes || bytes[i] > st->slot_bytes - slot_offset[i])
      return sfail(TPK_ERR_INVALID, "region %d: [%zu, +%zu) outside the %zu-byte slot", i, slot_offset[i], bytes[i],
                   st->slot_bytes);
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, host_src[i]);
    if (e != cudaSuccess) return scuda(e, "cudaPointerGetAttributes (source)");
    if (a.type != cudaMemoryTypeHost)
      return sfail(TPK_ERR_INVALID, "region %d: the source is not pinned host memory (the copy would not be asynchronous)", i);
  }
  // The copies into this slot start only after the work that read it last has
  // finished (its release event, recorded on the consumer stream).
  if (st->freed_recorded[slot]) {
    cudaError_t e = cudaStreamWaitEvent(st->copy, st->freed[slot], 0);
    if (e != cudaSuccess) return scuda(e, "copy stream wait for the slot's release");
  }
  cudaError_t e = cudaEventRecord(st->begun[slot], st->copy);
  if (e != cudaSuccess) return scuda(e, "copy start event");
  for (int i = 0; i < n_regions; ++i) {
    if (bytes[i] == 0) continue;
    e = cudaMemcpyAsync(st->slots[slot] + slot_offset[i], host_src[i], bytes[i], cudaMemcpyHostToDevice, st->copy);
    if (e != cudaSuccess) return scuda(e, "staging copy");
  }
  e = cudaEventRecord(st->ready[slot], st->copy);
  if (e != cudaSuccess) return scuda(e, "ready event");
  st->timed[slot] = true;
  st->state[slot] = kStaged;
  st->next = (slot + 1) % (int)st->slots.size();
  if (slot_out) *slot_out = slot;
  if (slot_dev_out) *slot_dev_out = st->slots[slot];
  return TPK_OK;
}

tpk_status tpk_stager_acquire(tpk_stager* st, int slot, tpk_stream_t stream) {
  tpk_status s = check_slot(st, slot);
  if (s != TPK_OK) return s;
  if (st->state[slot] != kStaged)
    return sfail(TPK_ERR_INVALID, "slot %d is %s, not staged", slot, st->state[slot] == kFree ? "free" : "already acquired");
  cudaError_t e = cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), st->ready[slot], 0);
  if (e != cudaSuccess) return scuda(e, "consumer stream wait for the staging copies");
  st->state[slot] = kAcquired;
  return TPK_OK;
}

tpk_status tpk_stager_release(tpk_stager* st, int slot, tpk_stream_t stream) {
  tpk_status s = check_slot(st, slot);
  if (s != TPK_OK) return s;
  if (st->state[slot] != kAcquired)
    return sfail(TPK_ERR_INVALID, "slot %d is %s, not acquired", slot, st->state[slot] == kFree ? "free" : "staged");
  cudaError_t e = cudaEventRecord(st->freed[slot], reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return scuda(e, "release event");
  st->freed_recorded[slot] = true;
  st->state[slot] = kFree;
  return TPK_OK;
}

tpk_status tpk_stager_copy_ms(tpk_stager* st, int slot, float* ms) {
  tpk_status s = check_slot(st, slot);
  if (s != TPK_OK) return s;
  if (!ms) return sfail(TPK_ERR_INVALID, "null output pointer");
  if (!st->timed[slot]) return sfail(TPK_ERR_INVALID, "slot %d has not been staged yet", slot);
  cudaError_t e = cudaEventSynchronize(st->ready[slot]);
  if (e != cudaSuccess) return scuda(e, "wait for the staging copies");
  e = cudaEventElapsedTime(ms, st->begun[slot], st->ready[slot]);
  if (e != cudaSuccess) return scuda(e, "copy time");
  return TPK_OK;
}

tpk_status tpk_stager_sync(tpk_stager* st) {
  if (!st) return sfail(TPK_ERR_INVALID, "null stager");
  tpk_status s = check_device(st);
  if (s != TPK_OK) return s;
  cudaError_t e = cudaStreamSynchronize(st->copy);
  if (e != cudaSuccess) return scuda(e, "stager copy stream");
  return TPK_OK;
}

}  // extern "C"
