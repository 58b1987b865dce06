// slot_alloc.cu -- host side of the pool: the slot allocator, the concurrency cap of a pool
// size, and the track plan of one decode step.  Plain C++ (no device code).
//
// Sources: "SGLang之KV Cache内存池机制" §8.3 (MambaPool.alloc: one state slot per request
// from the pool's free list; the pool has one row more than its usable slots, row 0 the
// padding row), "SGLang Qwen3/kimi-k3 Hybrid Linear Mamba KV cache管理" (the concurrency
// cap: the slots a request reserves, 3 as the base plus 2 ping-pong track slots with the
// overlap scheduler, one fewer with the decode-lock skip -- 80 slots at 5 per request cap
// the running requests at 16; mamba_track_interval: a request is tracked in the step where
// its length is a multiple of the interval; the extra-buffer track slots A / B alternate:
// round t reads A and writes B, round t+1 reads B and writes A).
#include <mutex>
#include <new>
#include <vector>

#include "rsc.h"

struct rsc_slot_alloc {
  std::mutex mu;
  int num_slots = 0;
  std::vector<int32_t> free_list;  // stack of free slot ids; the next one handed out at back()
  std::vector<uint8_t> used;       // used[s], s in [0, num_slots]; row 0 is never handed out
};

extern "C" {

int rsc_slot_alloc_create(int num_slots, rsc_slot_alloc **out) {
  if (!out) return RSC_EINVAL;
  *out = nullptr;
  if (num_slots < 0 || num_slots > (1 << 30)) return RSC_ERANGE;
  rsc_slot_alloc *a = new (std::nothrow) rsc_slot_alloc;
  if (!a) return RSC_ENOSPACE;
  a->num_slots = num_slots;
  a->free_list.reserve((size_t)num_slots);
  for (int s = num_slots; s >= 1; --s) a->free_list.push_back(s);  // slot 1 first
  a->used.assign((size_t)num_slots + 1, 0);
  a->used[0] = 1;
  *out = a;
  return RSC_OK;
}

int rsc_slot_alloc_destroy(rsc_slot_alloc *a) {
  delete a;
  return RSC_OK;
}

int rsc_slot_alloc_free_count(rsc_slot_alloc *a, int *count) {
  if (!a || !count) return RSC_EINVAL;
  std::lock_guard<std::mutex> lk(a->mu);
  *count = (int)a->free_list.size();
  return RSC_OK;
}

int rsc_slot_alloc_acquire(rsc_slot_alloc *a, int n, int32_t *slots) {
  if (!a || n < 0 || (n > 0 && !slots)) return RSC_EINVAL;
  std::lock_guard<std::mutex> lk(a->mu);
  if ((size_t)n > a->free_list.size()) return RSC_ENOSPACE;  // nothing taken
  for (int i = 0; i < n; ++i) {
    const int32_t s = a->free_list.back();
    a->free_list.pop_back();
    a->used[(size_t)s] = 1;
    slots[i] = s;
  }
  return RSC_OK;
}

int rsc_slot_alloc_release(rsc_slot_alloc *a, int n, const int32_t *slots) {
  if (!a || n < 0 || (n > 0 && !slots)) return RSC_EINVAL;
  std::lock_guard<std::mutex> lk(a->mu);
  // validate the whole list first (range, held, no repeats), so a bad call frees nothing
  for (int i = 0; i < n; ++i) {
    const int32_t s = slots[i];
    if (s < 1 || s > a->num_slots) return RSC_ERANGE;
    if (!a->used[(size_t)s]) return RSC_EINVAL;
    for (int k = 0; k < i; ++k)
      if (slots[k] == s) return RSC_EINVAL;
  }
  for (int i = 0; i < n; ++i) {
    a->used[(size_t)slots[i]] = 0;
    a->free_list.push_back(slots[i]);
  }
  return RSC_OK;
}

int rsc_max_running_requests(int num_slots, int overlap, int skip_decode_lock, int *out) {
  if (!out) return RSC_EINVAL;
  if (num_slots < 0) return RSC_ERANGE;
  const int per_request = 3 + (overlap ? 2 : 0) - (skip_decode_lock ? 1 : 0);
  *out = num_slots / per_request;
  return RSC_OK;
}

int rsc_track_plan(int batch, const int32_t *seq_lens, int interval, const int32_t *track_pairs,
                   int ntrack, int32_t *next_idx, uint8_t *mask, int32_t *track_slots) {
  if (batch < 0) return RSC_ERANGE;
  if (batch == 0) return RSC_OK;
  if (!seq_lens || !track_pairs || !next_idx || !mask || !track_slots) return RSC_EINVAL;
  if (interval < 1 || ntrack < 1 || ntrack > 2) return RSC_ERANGE;
  for (int b = 0; b < batch; ++b)
    if (next_idx[b] < 0 || next_idx[b] >= ntrack || seq_lens[b] < 0) return RSC_ERANGE;
  for (int b = 0; b < batch; ++b) {
    const bool due = seq_lens[b] > 0 && seq_lens[b] % interval == 0;
    mask[b] = due ? 1 : 0;
    track_slots[b] = due ? track_pairs[(size_t)b * ntrack + next_idx[b]] : 0;
    if (due) next_idx[b] = (next_idx[b] + 1) % ntrack;  // ping-pong once a snapshot is taken
  }
  return RSC_OK;
}

}  // extern "C"
