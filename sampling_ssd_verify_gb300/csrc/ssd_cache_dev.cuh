// ssd_cache_dev.cuh -- device code of the outcome cache, shared by the cache
// kernels (ssd_cache.cu) and the verify kernel that builds and probes a
// round's cache in the same launch (ssd_stream_kernel.cuh).
//
// [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈",
// §"SSD 的核心思想": the outcome of a sequence is (k accepted, bonus t); the
// drafter keeps one continuation per predicted outcome.  §"Saguaro 优化三：
// 自适应回退策略": the batch proceeds without waiting only if every sequence
// hits.
//
// Open-addressed hash table of 16-byte slots {u64 key, i32 value, pad} with a
// power-of-two capacity; the key packs (row:32 | k:8 | t:24) and the empty
// key is all ones.  Slot index = SplitMix64 finaliser of the key (Steele, Lea
// & Flood, "Fast splittable pseudorandom number generators", OOPSLA'14);
// linear probing bounded by the capacity, so a full table never loops.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {
namespace {

constexpr unsigned long long kEmptyKey = ~0ull;

struct alignas(16) Slot {
  unsigned long long key;
  int value;
  int pad;
};

__device__ __forceinline__ unsigned long long pack_key(int row, int k, int t) {
  return ((unsigned long long)(uint32_t)row << 32) | ((unsigned long long)(k & 0xFF) << 24) |
         (unsigned long long)(t & 0xFFFFFF);
}

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ void slot_clear(Slot* s) {
  s->key = kEmptyKey;
  s->value = -1;
  s->pad = 0;
}

// Insert key -> value: claim the first empty slot of the probe sequence with
// a compare-and-swap of its key.
__device__ __forceinline__ void cache_insert(Slot* tab, int64_t cap, unsigned long long key,
                                             int value, int32_t* status) {
  int64_t i = (int64_t)(mix64(key) & (unsigned long long)(cap - 1));
  for (int64_t probe = 0; probe < cap; ++probe) {
    const unsigned long long old = atomicCAS(&tab[i].key, kEmptyKey, key);
    if (old == kEmptyKey) {
      tab[i].value = value;
      return;
    }
    if (old == key) {
      if (status) atomicOr(status, SSD_DEV_DUPLICATE_KEY);
      return;
    }
    i = (i + 1) & (cap - 1);
  }
  if (status) atomicOr(status, SSD_DEV_TABLE_FULL);
}

// The value of key, or -1: probing stops at the first empty slot.  Reads go
// to L2 (the keys may have been written by other CTAs of the same launch).
__device__ __forceinline__ int cache_find(const Slot* tab, int64_t cap, unsigned long long key) {
  int64_t i = (int64_t)(mix64(key) & (unsigned long long)(cap - 1));
  for (int64_t probe = 0; probe < cap; ++probe) {
    const unsigned long long w = __ldcg(&tab[i].key);
    if (w == key) return __ldcg(&tab[i].value);
    if (w == kEmptyKey) return -1;
    i = (i + 1) & (cap - 1);
  }
  return -1;
}

// Sequence g's lookup of its outcome (k, t) in a round's cache: out_branch[g]
// and, for the last of the B sequences to finish, *all_hit.  cnt packs
// (finished sequences << 32 | hits).  One thread; every key of sequence g was
// inserted before.
__device__ __forceinline__ void round_outcome(const Slot* tab, int64_t cap, int64_t g, int k,
                                              int t, int B, int32_t* out_branch,
                                              int32_t* all_hit, unsigned long long* cnt) {
  const int v = cache_find(tab, cap, pack_key((int)g, k, t));
  out_branch[g] = v;
  const unsigned long long hit = v >= 0 ? 1ull : 0ull;
  const unsigned long long old = atomicAdd(cnt, (1ull << 32) | hit);
  if ((old >> 32) + 1 == (unsigned long long)B && all_hit)
    *all_hit = ((old & 0xFFFFFFFFull) + hit) == (unsigned long long)B ? 1 : 0;
}

}  // namespace
}  // namespace ssd
