// ssd_noalloc.cu -- ssd_verify for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: an inference
// runtime's plugin whose enqueue hook is not allowed to allocate, a process
// whose device memory is entirely owned by a pool allocator, or a
// latency-critical decode loop that cannot afford cudaMalloc and the device
// synchronisation it implies.  ssd_verify_noalloc serves them with a scratch
// area compiled into the library: a file-scope device array of
// SSD_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
// the process exits.  Nothing here calls cudaMalloc, cudaFree or any other
// allocating routine.
//
// Set-up: the array's device address is looked up with cudaGetSymbolAddress
// the first time the entry point runs on a device (with that device current)
// and cached per device and context; that first call should therefore come
// before any stream capture on the device.  After cudaDeviceReset (a new
// context) the next call looks the address up again.
//
// Sharing: every call on a device uses the same array.  The counters that
// must start at zero are cleared on the caller's stream at the start of each
// call (as ssd_verify does with a caller workspace), and the rest of the
// array is written before it is read, so the contents left by the previous
// call do not matter -- but two calls whose work overlaps on the GPU (two
// streams, or two host threads) race on the array and must be serialised by
// the caller.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ssd.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  void* ctx;  // the context the address belongs to
  void* ptr;
};
Cached g_scratch[kMaxDevices] = {};

// The calling thread's current CUDA context (the driver's cuCtxGetCurrent,
// reached through the runtime's entry-point query), or null.  A device reset
// or a re-created primary context loads the library's module again, and the
// array may then sit at another address: the cache is keyed on the context.
void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = nullptr;
  static bool looked = false;
  if (!looked) {
    looked = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<Fn>(f);
    else
      cudaGetLastError();
  }
  void* ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of the scratch array in the current context (cached).
ssd_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SSD_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  void* ctx = current_context();
  Cached& c = g_scratch[dev];
  if (c.ptr == nullptr || ctx == nullptr || c.ctx != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return SSD_ERR_CUDA;
    }
    c.ptr = ptr;
    c.ctx = current_context();  // the query made the context current if it was not
  }
  *out = c.ptr;
  return SSD_OK;
}

}  // namespace

extern "C" ssd_status ssd_verify_noalloc(const ssd_logits* target, const ssd_logits* draft,
                                         int B, int K, int Kq, int V, float T,
                                         const int32_t* draft_tokens, const uint64_t* seeds,
                                         uint32_t round, const int32_t* fanout, float C,
                                         int32_t* accept_len, int32_t* bonus, float* resid_mass,
                                         int32_t* guesses, float* guess_q, int Fmax,
                                         int32_t* dev_status, void* stream) {
  const size_t need = ssd_verify_workspace_size(B, K, Kq, V);
  if (need == 0) return SSD_ERR_INVALID_ARG;
  // the request does not fit the built-in scratch: the caller must use
  // ssd_verify with a workspace of its own
  if (need > (size_t)SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE;
  void* scratch = nullptr;
  const ssd_status st = scratch_for_current_device(&scratch);
  if (st != SSD_OK) return st;
  return ssd_verify(target, draft, B, K, Kq, V, T, draft_tokens, seeds, round, fanout, C,
                    accept_len, bonus, resid_mass, guesses, guess_q, Fmax, scratch,
                    (size_t)SSD_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
