// absorb.cu -- the two per-head matrix products on either side of the
// absorbed decode ("DeepSeek MLA architecture ...", section 4, matrix
// absorption; "DeepSeek-V3.2-Exp . KV cache", the split of wkv_b into the key
// part and the value part):
//   q_latent[b, h, :] = q_nope[b, h, :] . W_UK[h]        (128 -> 512 per head)
//   o[b, h, :]        = W_UV[h] . x[b, h, :]              (512 -> 128 per head)
// wkv_b is [H, 256, 512] bf16: rows 0..127 of head h are W_UK[h] (n x c),
// rows 128..255 are W_UV[h] (v x c).  Products accumulate in fp32 (tensor
// memory) and are rounded to bf16 once.
//
// One CTA per (head, chunk of up to 64 sequences) -- and, for the query
// absorption, per 128-column block of q_latent, so that a head's 128 KB of
// weights is pulled in by four SMs.  The weights are the MMA's A operand
// (M = 128 rows: 128 latent columns c of W_UK^T, or the 128 value rows v of
// W_UV), the chunk's sequences its N
// (64, rows past B zero-filled by TMA): a decode batch is far narrower than
// any MMA M, so the weights take that side.  W_UK^T is read straight from
// W_UK's [n][c] layout as an MN-major A operand; W_UV and the activations are
// K-major.  All tiles arrive by TMA in the 128-byte swizzled layout.
//
// The weights are constant, so their loads are issued before the wait on the
// previous kernel (programmatic dependent launch): they stream in while it
// finishes; the activations follow the wait.
// Warps: thread 0 issues the loads and the MMAs; all four warps move the
// result from tensor memory (lane = c or v) to global memory (a warp writes
// 32 consecutive bf16 of one sequence).  Waits are bounded; on expiry a
// status bit is raised and the CTA skips its writes.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>
#include <string.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kChunk = 64;                   // sequences per CTA (MMA N)
constexpr int kXBlk = kChunk * 128;          // 64 sequence rows x 64 columns, bf16
constexpr long kSpin = 1L << 26;

struct AbsorbParams {
  CUtensorMap m_w;    // wkv_b [H][256][512] (box 64 x 128 x 1, 128-byte swizzle)
  CUtensorMap m_x;    // activations [B][H][K] (box 64 x 1 x 64, 128-byte swizzle)
  void* y;            // bf16 [B][H][N_out]
  uint32_t* status;   // device status word or null
  int B, H;
};

__device__ bool wait_bounded(uint64_t* b, uint32_t parity) {
  for (long it = 0; it < kSpin; ++it)
    if (bar_try_local(b, parity)) return true;
  return false;
}

// kQ = true: q_latent = q_nope . W_UK (K = 128; the CTA's 128-column block of
//            c is blockIdx.z)
// kQ = false: o = W_UV . x (K = 512, one block of 128 v)
template <bool kQ>
__global__ void __launch_bounds__(128) absorb_kernel(const __grid_constant__ AbsorbParams ap) {
  constexpr int kK = kQ ? 128 : 512;               // contraction length
  constexpr int kMBlocks = 1;                      // 128-row output blocks per CTA
  constexpr int kXBlocks = kK / 64;                // activation blocks of 64 columns
  constexpr uint32_t kCols = kMBlocks * kChunk;    // tensor-memory columns
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wsm = sm;                   // 2 (query) or 8 (projection) blocks of 16 KB
  constexpr int kWBlocks = kQ ? 2 : 8;
  uint8_t* xsm = sm + kWBlocks * kSwBlk;   // kXBlocks blocks of 8 KB
  const int mb = kQ ? blockIdx.z : 0;      // output block: c in [128 mb, 128 mb + 128)
  __shared__ __align__(8) uint64_t full, done;
  __shared__ uint32_t tslot;
  const int h = blockIdx.x, b0 = blockIdx.y * kChunk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    bar_init(&full, 1);
    bar_init(&done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sa(&tslot)),
                 "r"(kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = tslot;
  // the weights are constant: their loads go out before the wait on the
  // previous kernel, so they stream in while it finishes
  if (threadIdx.x == 0) {
    bar_expect_tx(&full, kWBlocks * kSwBlk + kXBlocks * kXBlk);
    const int row0 = kQ ? 0 : 128;     // W_UK or W_UV rows of head h
    for (int cb = 0; cb < kWBlocks; ++cb)
      tma3(wsm + cb * kSwBlk, &ap.m_w, 64 * (cb + 2 * mb), row0, h, &full);
  }
  pdl_wait();   // the activations may come from the previous kernel
  pdl_trigger();

  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    for (int k = 0; k < kXBlocks; ++k) tma3(xsm + k * kXBlk, &ap.m_x, 64 * k, h, b0, &full);
    const bool landed = wait_bounded(&full, 0);
    if (landed) {
      tc_after();
      const uint32_t id = idesc(128, kChunk, false, kQ);
      const uint32_t wa = sa(wsm), xa = sa(xsm);
#pragma unroll 1
      for (int m = 0; m < kMBlocks; ++m) {
#pragma unroll 1
        for (int kk = 0; kk < kK / 16; ++kk) {
          // A: W_UK^T is MN-major (c contiguous): blocks 0 and 1 (LBO apart),
          //    16 rows of n per step; W_UV is K-major: block kk/4, 32 B per step
          const uint64_t a = kQ ? sdesc(wa + 2 * m * kSwBlk + 2048 * kk, kSwBlk, 1024)
                                : sdesc(wa + (kk >> 2) * kSwBlk + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc(xa + (kk >> 2) * kXBlk + (kk & 3) * 32, 16, 1024);
          mma_ss(tmem + m * kChunk, a, b, id, kk > 0 ? 1 : 0);
        }
      }
    } else {
      // the loads issued above still land in this CTA's shared memory
      for (long it = 0; it < kSpin && !bar_try_local(&full, 0); ++it) {}
    }
    s_ok = landed;
    mma_commit(&done);   // arrives once the MMAs (if any) are complete
  }
  // every warp: the products are in tensor memory (tcgen05.ld is warp-wide,
  // so a warp reads only if all its lanes saw the commit)
  const bool finished = __all_sync(0xffffffffu, wait_bounded(&done, 0));
  __syncthreads();
  const bool ok = s_ok && finished;
  if (!ok && lane == 0 && ap.status) atomicOr(ap.status, kDevTimeout);
  tc_after();
  if (ok) {
    const int nout = kQ ? 512 : 128;
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(ap.y);
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int m = 0; m < kMBlocks; ++m) {
      const int row = (mb + m) * 128 + warp * 32 + lane;   // c (query) or v (output)
#pragma unroll 1
      for (int c = 0; c < kChunk / 16; ++c) {
        uint32_t r[16];
        TC_LD16(lane_base + m * kChunk + 16 * c, r);
        tc_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int b = b0 + 16 * c + k;
          if (b < ap.B) y[((size_t)b * ap.H + h) * nout + row] = __float2bfloat16_rn(__uint_as_float(r[k]));
        }
      }
    }
  }
  tc_before();
  __syncthreads();
  if (warp == 0) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

template <bool kQ>
cudaError_t launch(const void* x, const void* wkv_b, int B, int H, void* y, uint32_t* status,
                   cudaStream_t s) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  constexpr int kK = kQ ? 128 : 512;
  AbsorbParams ap;
  memset(&ap, 0, sizeof(ap));
  {
    cuuint64_t dims[3] = {512, 256, (cuuint64_t)H};
    cuuint64_t strides[2] = {512 * 2, 512 * 2 * 256};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&ap.m_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(wkv_b), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)kK, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)kK * 2, (cuuint64_t)kK * 2 * H};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kChunk};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&ap.m_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  ap.y = y;
  ap.status = status;
  ap.B = B;
  ap.H = H;
  const size_t smem = (kQ ? 2 : 8) * kSwBlk + (kK / 64) * kXBlk + 1024;
  cudaError_t e = ensure_smem<absorb_kernel<kQ>>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(absorb_kernel<kQ>, dim3(H, (B + kChunk - 1) / kChunk, kQ ? 4 : 1), dim3(128), smem, s,
                    ap);
}

}  // namespace

cudaError_t launch_absorb_q(const void* q_nope, const void* wkv_b, int B, int H, void* q_latent,
                            uint32_t* status, cudaStream_t s) {
  return launch<true>(q_nope, wkv_b, B, H, q_latent, status, s);
}

cudaError_t launch_project_out(const void* x, const void* wkv_b, int B, int H, void* o,
                               uint32_t* status, cudaStream_t s) {
  return launch<false>(x, wkv_b, B, H, o, status, s);
}

}  // namespace mla
