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
// per device; host code cannot use the array's name as a device address).
mla_status scratch_address(void** out, int* sms) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  static int nsm[64] = {0};
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
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    addr[dev] = p;
    nsm[dev] = n;
  }
  *out = addr[dev];
  *sms = nsm[dev];
  return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

mla_status mla_decode_noalloc(const mla_cache* c, const void* q_latent, const void* q_pe,
                              const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                              float softmax_scale, void* out, float* lse, void* stream) {
  if (!c || !c->kv || !c->pe) return MLA_ERR_INVALID_ARG;
  if (c->fmt != MLA_KV_BF16 && c->fmt != MLA_KV_FP8_E4M3_B128 && c->fmt != MLA_KV_FP8_E4M3_B128_POW2)
    return MLA_ERR_UNSUPPORTED;
  if (c->max_batch <= 0 || c->max_seq_len <= 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c->kv) || !aligned16(c->pe)) return MLA_ERR_INVALID_ARG;
  if (c->fmt != MLA_KV_BF16 && (!c->kv_scale || !aligned16(c->kv_scale)))
    return MLA_ERR_INVALID_ARG;
  if (!(H == 16 || H == 32 || H == 64 || H == 128)) return MLA_ERR_UNSUPPORTED;
  if (B <= 0 || B > c->max_batch) return MLA_ERR_INVALID_ARG;
  if (max_end_pos <= 0 || max_end_pos > c->max_seq_len) return MLA_ERR_OUT_OF_RANGE;
  if (!q_latent || !q_pe || !end_pos || !out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_latent) || !aligned16(q_pe) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(end_pos) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale)) return MLA_ERR_INVALID_ARG;

  void* scratch = nullptr;
  int sms = 0;
  mla_status st = scratch_address(&scratch, &sms);
  if (st != MLA_OK) return st;
  const mla::Workspace need = mla::carve_workspace(nullptr, B, H, 0, sms);
  if (need.bytes > kScratchBytes) return MLA_ERR_WORKSPACE;   // the static scratch is too small
  const mla::Workspace ws = mla::carve_workspace(scratch, B, H, 0, sms);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  mla::DecodeParams p{};
  p.fmt = mla::decode_fmt(c->fmt);
  p.max_seq_len = c->max_seq_len;
  p.kv = c->kv;
  p.kv_scale = c->kv_scale;
  p.pe = c->pe;
  p.q_latent = q_latent;
  p.q_pe = q_pe;
  p.B = B;
  p.H = H;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = out;
  p.lse = lse;
  p.ws = ws;
  p.K = 0;
  p.mtp_s = 1;

  const bool tc = mla::decode_tc_supported(H);
  // the schedule kernel writes the status word afresh; every other region
  // is written before it is read
  cudaError_t e = mla::launch_schedule(
      end_pos, max_end_pos, ws, B,
      tc ? mla::decode_tc_units(mla::decode_fmt(c->fmt), false, sms) : mla::target_units_mma(H, sms),
      tc ? mla::decode_tc_granule(mla::decode_fmt(c->fmt), false) : mla::decode_mma_granule(), tc, 1,
      false, s);
  if (e == cudaSuccess) e = tc ? mla::launch_decode_tc(p, s) : mla::launch_decode_mma(p, s);
  if (e == cudaSuccess) e = mla::launch_combine(ws, B, H, out, lse, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // extern "C"
