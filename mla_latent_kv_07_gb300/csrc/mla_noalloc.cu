// mla_noalloc.cu -- mla_decode_noalloc: the dense decode of mla_decode for
// callers that cannot hand the library a workspace.
//
// Who needs it: code that may not allocate device memory at the point where
// it decodes -- for example a serving loop that forbids allocations after its
// warm-up, an embedding host or plug-in interface that only passes the input
// and output buffers in, or code running under an allocator that must not be
// re-entered.  Such callers cannot provide the scratch mla_decode needs (split
// schedule, per-split partial outputs and log-sum-exps, status word).
//
// What it does instead: the scratch is one file-scope device array of
// kScratchBytes, reserved on every GPU that loads this library until the
// process exits.  The first call on a device looks up that array's device
// address (cudaGetSymbolAddress, with the device current) and caches it; make
// that first call before starting any stream capture.  Calls whose scratch
// need exceeds kScratchBytes are refused with MLA_ERR_WORKSPACE.  Nothing here
// calls cudaMalloc, cudaFree or any allocating routine.
//
// Every call uses the same array and leaves its contents behind; the status
// word is cleared by the first kernel of each call and every other region is
// written before it is read.  Calls whose work overlaps on the GPU (different streams,
// or different host threads without ordering) race on the array: order them.
#include <mutex>

#include "../../include/mla.h"
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;   // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch array on the current device (looked up once
// per device, with that device current; host code cannot use the array's name
// as a device address).
mla_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return MLA_OK;
}

}  // namespace

namespace mla {
// mla_api.cu: mla_decode's checks and launch sequence over a given scratch
mla_status decode_in_scratch(const mla_cache* cache, const void* q_latent, const void* q_pe,
                             const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                             float softmax_scale, void* out, float* lse, void* scratch,
                             size_t scratch_bytes, void* stream);
}  // namespace mla

extern "C" {

mla_status mla_decode_noalloc(const mla_cache* c, const void* q_latent, const void* q_pe,
                              const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                              float softmax_scale, void* out, float* lse, void* stream) {
  void* scratch = nullptr;
  mla_status st = scratch_address(&scratch);
  if (st != MLA_OK) return st;
  // the array is 256-byte aligned, as a caller workspace must be; a call whose
  // B and H need more than kScratchBytes is refused with MLA_ERR_WORKSPACE
  return mla::decode_in_scratch(c, q_latent, q_pe, end_pos, max_end_pos, B, H, softmax_scale, out, lse,
                                scratch, kScratchBytes, stream);
}

}  // extern "C"
