// ssd_cache.cu -- the speculation (outcome) cache.
//
// [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈",
// §"SSD 的核心思想": the verification outcome of a sequence is the pair
// (k accepted drafts, bonus token t); the drafter keeps a continuation for each
// predicted outcome and the next round starts at once when the real outcome is
// in the cache.  §"Saguaro 优化三：自适应回退策略": the batch proceeds without
// waiting only when every sequence hits.
//
// Open-addressed hash table of 16-byte slots (ssd_cache_dev.cuh); here the
// key packs (row:32 | k:8 | t:24) and the empty key is all ones.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "ssd_cache_dev.cuh"
#include "ssd_device.cuh"
#include "ssd_internal.cuh"

namespace ssd {

namespace {

__global__ void clear_kernel(Slot* tab, int64_t cap) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < cap;
       i += (int64_t)gridDim.x * blockDim.x) {
    slot_clear(tab + i);
  }
}

__global__ void insert_kernel(Slot* tab, int64_t cap, const int32_t* row, const int32_t* k,
                              const int32_t* t, const int32_t* branch, int n,
                              const int32_t* guesses, int B, int Kq, int Fmax, int32_t* status) {
  const int64_t total = guesses ? (int64_t)B * Kq * Fmax : n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (guesses) {
      const int g = guesses[i];
      if (g < 0) continue;
      const int b = (int)(i / ((int64_t)Kq * Fmax));
      const int kk = (int)((i / Fmax) % Kq);
      cache_insert(tab, cap, pack_key(b, kk, g), (int)i, status);
    } else {
      cache_insert(tab, cap, pack_key(row[i], k[i], t[i]), branch[i], status);
    }
  }
}

__global__ void lookup_kernel(const Slot* tab, int64_t cap, const int32_t* accept_len,
                              const int32_t* bonus, int B, int32_t* out_branch,
                              int32_t* all_hit) {
  int ok = 1;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int v = cache_find(tab, cap, pack_key(b, accept_len[b], bonus[b]));
    out_branch[b] = v;
    ok &= v >= 0;
  }
  ok = __syncthreads_and(ok);
  if (threadIdx.x == 0 && all_hit) *all_hit = ok;
}

}  // namespace

cudaError_t launch_cache_clear(void* table, int64_t capacity, cudaStream_t s) {
  const int grid = (int)std::min<int64_t>(1024, (capacity + 255) / 256);
  clear_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<Slot*>(table), capacity);
  return cudaGetLastError();
}

cudaError_t launch_cache_insert(void* table, int64_t capacity, const int32_t* row,
                                const int32_t* k, const int32_t* t, const int32_t* branch, int n,
                                const int32_t* guesses, int B, int Kq, int Fmax,
                                int32_t* status, cudaStream_t s) {
  const int64_t total = guesses ? (int64_t)B * Kq * Fmax : n;
  if (total <= 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>(1024, (total + 255) / 256);
  insert_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<Slot*>(table), capacity, row, k, t, branch,
                                     n, guesses, B, Kq, Fmax, status);
  return cudaGetLastError();
}

cudaError_t launch_cache_lookup(const void* table, int64_t capacity, const int32_t* accept_len,
                                const int32_t* bonus, int B, int32_t* out_branch,
                                int32_t* all_hit, cudaStream_t s) {
  lookup_kernel<<<1, 1024, 0, s>>>(reinterpret_cast<const Slot*>(table), capacity, accept_len,
                                   bonus, B, out_branch, all_hit);
  return cudaGetLastError();
}

}  // namespace ssd
