// decode_mma.cu -- split-KV flash-decoding over the latent cache with warp-level
// tensor-core MMA (mma.sync m16n8k16 bf16 -> fp32).  One CTA handles one unit
// (a range of positions of one sequence) for 16 heads:
//   S[16, 32]  = Q[16, 576] . [c | k_R][32, 576]^T        (scores of one tile)
//   online softmax over the tile (running max m, running sum l, per head)
//   O[16, 512] = alpha * O + P[16, 32] . c[32, 512]        (value sum, latent)
// The unit's normalised O and its log-sum-exp go to the workspace; the
// combine kernel merges units.  Following "DeepSeek-V3.2-Exp . KV cache"
// (MQA-decode excerpt) and "DeepSeek MLA architecture ..." sections 3-4.
//
// Tiles are staged with cp.async in two stages.  FP8 tiles land as raw codes
// and scales and are expanded in shared memory to bf16(fp32(e4m3 * scale)),
// the value the cache-write excerpt defines.  Rows past the unit's end are
// zero-filled, so masked positions multiply zeros, never stale memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kTile = 32;              // positions per tile
constexpr int kHeads = 16;             // heads per CTA (one m16 row block)
constexpr int kThreads = 128;
constexpr int kRow = kDqk + 8;         // smem row stride (bf16): 1168 B, ldmatrix conflict-free
constexpr int kPRow = kTile + 8;       // P row stride (bf16): 80 B

struct Smem {
  __nv_bfloat16 q[kHeads * kRow];
  __nv_bfloat16 kv[2][kTile * kRow];
  uint8_t raw[2][kTile * kDc];         // FP8 codes (FP8 caches only)
  float raw_scale[2][kTile * kNblk];
  float s[kHeads * kTile];
  __nv_bfloat16 p[kHeads * kPRow];
  float alpha[kHeads];
  float l[kHeads];
  float m[kHeads];
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;   // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Position of row r of tile `tile` in the unit, or -1 past the unit's end.
template <bool kSparse>
__device__ __forceinline__ int tile_pos(const DecodeParams& p, const Unit& u, int tile, int r) {
  const int i = u.t0 + tile * kTile + r;
  if (i >= u.t1) return -1;
  return kSparse ? p.ws.gidx[(size_t)u.b * p.K + i] : i;
}

template <int kFmt, bool kSparse>
__device__ __forceinline__ void load_tile(const DecodeParams& p, const Unit& u, int tile,
                                          Smem& sm, int stage) {
  const int tid = threadIdx.x;
  const size_t seq_row0 = (size_t)(u.b / p.mtp_s) * p.max_seq_len;   // the cache slot
  if (kFmt == 0) {
    // 32 rows x 72 chunks of 16 B (64 latent + 8 rotary)
    for (int c = tid; c < kTile * 72; c += kThreads) {
      const int r = c / 72, k = c % 72;
      const int pos = tile_pos<kSparse>(p, u, tile, r);
      const size_t row = seq_row0 + (pos < 0 ? 0 : pos);
      const __nv_bfloat16* src =
          k < 64 ? static_cast<const __nv_bfloat16*>(p.kv) + row * kDc + k * 8
                 : static_cast<const __nv_bfloat16*>(p.pe) + row * kDr + (k - 64) * 8;
      cp_async16(&sm.kv[stage][r * kRow + k * 8], src, pos >= 0);
    }
  } else {
    // codes: 32 rows x 32 chunks; scales: 32 rows x 1 chunk; rotary: 32 x 8
    for (int c = tid; c < kTile * 41; c += kThreads) {
      const int r = c / 41, k = c % 41;
      const int pos = tile_pos<kSparse>(p, u, tile, r);
      const size_t row = seq_row0 + (pos < 0 ? 0 : pos);
      if (k < 32) {
        cp_async16(&sm.raw[stage][r * kDc + k * 16],
                   static_cast<const uint8_t*>(p.kv) + row * kDc + k * 16, pos >= 0);
      } else if (k == 32) {
        cp_async16(&sm.raw_scale[stage][r * kNblk], p.kv_scale + row * kNblk, pos >= 0);
      } else {
        cp_async16(&sm.kv[stage][r * kRow + kDc + (k - 33) * 8],
                   static_cast<const __nv_bfloat16*>(p.pe) + row * kDr + (k - 33) * 8, pos >= 0);
      }
    }
  }
}

// FP8 codes -> bf16(fp32(e4m3 * scale)) in the operand tile.
__device__ __forceinline__ void expand_fp8(Smem& sm, int stage) {
  for (int c = threadIdx.x; c < kTile * 32; c += kThreads) {
    const int r = c >> 5, k = c & 31;  // chunk of 16 codes, block k / 8
    const uint4 v = *reinterpret_cast<const uint4*>(&sm.raw[stage][r * kDc + k * 16]);
    const float sc = sm.raw_scale[stage][r * kNblk + (k >> 3)];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i >> 1] >> ((i & 1) * 16)) & 0xffffu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      const __nv_bfloat162 bb = __floats2bfloat162_rn(__fmul_rn(f.x, sc), __fmul_rn(f.y, sc));
      o[i] = *reinterpret_cast<const uint32_t*>(&bb);
    }
    uint4* dst = reinterpret_cast<uint4*>(&sm.kv[stage][r * kRow + k * 16]);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

template <int kFmt, bool kSparse>
__global__ void __launch_bounds__(kThreads) decode_mma_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  pdl_wait();   // the schedule of this call is complete
  pdl_trigger();
  const Unit u = p.ws.units[blockIdx.x];
  if (u.b < 0) return;
  const int hg = blockIdx.y;            // head group
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;

  // queries of the 16 heads: [latent | rotary] rows
  for (int c = tid; c < kHeads * 72; c += kThreads) {
    const int r = c / 72, k = c % 72;
    const size_t qrow = (size_t)u.b * p.H + hg * kHeads + r;
    const __nv_bfloat16* src =
        k < 64 ? static_cast<const __nv_bfloat16*>(p.q_latent) + qrow * kDc + k * 8
               : static_cast<const __nv_bfloat16*>(p.q_pe) + qrow * kDr + (k - 64) * 8;
    cp_async16(&sm.q[r * kRow + k * 8], src, true);
  }
  const int ntiles = (u.t1 - u.t0 + kTile - 1) / kTile;
  load_tile<kFmt, kSparse>(p, u, 0, sm, 0);
  cp_async_commit();

  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_run[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  float l_run[4] = {0.f, 0.f, 0.f, 0.f};

  for (int it = 0; it < ntiles; ++it) {
    const int st = it & 1;
    if (it + 1 < ntiles) {
      load_tile<kFmt, kSparse>(p, u, it + 1, sm, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kFmt == 1) {
      expand_fp8(sm, st);
      __syncthreads();
    }
    const __nv_bfloat16* kv = sm.kv[st];

    // ---- scores: warp w -> positions 8w..8w+7 of the tile, all 16 heads
    {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const int n0 = warp * 8;
#pragma unroll 4
      for (int kk = 0; kk < kDqk / 16; ++kk) {
        uint32_t a0, a1, a2, a3, b0, b1;
        ldsm_x4(a0, a1, a2, a3, &sm.q[(lane & 15) * kRow + kk * 16 + (lane >> 4) * 8]);
        ldsm_x2(b0, b1, &kv[(n0 + (lane & 7)) * kRow + kk * 16 + ((lane >> 3) & 1) * 8]);
        mma16816(acc, a0, a1, a2, a3, b0, b1);
      }
      sm.s[g * kTile + n0 + 2 * t] = acc[0];
      sm.s[g * kTile + n0 + 2 * t + 1] = acc[1];
      sm.s[(g + 8) * kTile + n0 + 2 * t] = acc[2];
      sm.s[(g + 8) * kTile + n0 + 2 * t + 1] = acc[3];
    }
    __syncthreads();

    // ---- online softmax: warp w -> heads 4w..4w+3, lane -> position
    {
      const bool valid = u.t0 + it * kTile + lane < u.t1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int h = warp * 4 + j;
        const float s = valid ? sm.s[h * kTile + lane] * p.scale_log2 : -INFINITY;
        const float m_new = fmaxf(m_run[j], warp_max(s));
        const float alpha = exp2f(m_run[j] - m_new);   // 0 on the first tile
        const __nv_bfloat16 pb = __float2bfloat16_rn(exp2f(s - m_new));
        const float psum = warp_sum(__bfloat162float(pb));
        l_run[j] = l_run[j] * alpha + psum;
        m_run[j] = m_new;
        sm.p[h * kPRow + lane] = pb;
        if (lane == 0) sm.alpha[h] = alpha;
      }
    }
    __syncthreads();

    // ---- value sum: warp w -> latent columns 128w..128w+127
    {
      const float a_lo = sm.alpha[g], a_hi = sm.alpha[g + 8];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        o[j][0] *= a_lo; o[j][1] *= a_lo; o[j][2] *= a_hi; o[j][3] *= a_hi;
      }
#pragma unroll
      for (int ks = 0; ks < kTile / 16; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, &sm.p[(lane & 15) * kPRow + ks * 16 + (lane >> 4) * 8]);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int c0 = warp * 128 + jj * 16;
          const int krow = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, &kv[krow * kRow + c0 + (lane >> 4) * 8]);
          mma16816(o[2 * jj], a0, a1, a2, a3, b0, b1);
          mma16816(o[2 * jj + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  // ---- epilogue: normalised partial output and log-sum-exp of the unit
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sm.l[warp * 4 + j] = l_run[j];
      sm.m[warp * 4 + j] = m_run[j];
    }
  }
  __syncthreads();
  const size_t ubase = (size_t)blockIdx.x * p.H + hg * kHeads;
  const float l_lo = sm.l[g], l_hi = sm.l[g + 8];
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f, inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
  float* po = p.ws.part_o;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = warp * 128 + j * 8 + 2 * t;
    *reinterpret_cast<float2*>(po + (ubase + g) * kDc + col) =
        make_float2(o[j][0] * inv_lo, o[j][1] * inv_lo);
    *reinterpret_cast<float2*>(po + (ubase + g + 8) * kDc + col) =
        make_float2(o[j][2] * inv_hi, o[j][3] * inv_hi);
  }
  if (tid < kHeads) {
    const float l = sm.l[tid], m = sm.m[tid];
    // m is in log2 units (scores were scaled by log2 e); lse in natural log
    p.ws.part_lse[ubase + tid] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
}

template <int kFmt, bool kSparse>
cudaError_t launch_variant(const DecodeParams& p, cudaStream_t s) {
  const size_t smem = sizeof(Smem);
  cudaError_t e = ensure_smem<decode_mma_kernel<kFmt, kSparse>>(smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.ws.max_units, p.H / kHeads);
  return launch_pdl(decode_mma_kernel<kFmt, kSparse>, grid, dim3(kThreads), smem, s, p);
}

}  // namespace

int decode_mma_granule() { return kTile; }

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s) {
  if (p.fmt == 0) return p.K ? launch_variant<0, true>(p, s) : launch_variant<0, false>(p, s);
  return p.K ? launch_variant<1, true>(p, s) : launch_variant<1, false>(p, s);
}

}  // namespace mla
