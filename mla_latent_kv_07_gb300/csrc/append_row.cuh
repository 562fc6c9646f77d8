// append_row.cuh -- the cache-write step of "DeepSeek-V3.2-Exp . KV cache"
// (cache-write excerpt) for one row, as device code shared by the append
// kernels, the sparse prep kernel and the dense decode kernel (which writes
// the new row itself inside the unit that reads it).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace mla {

// Smallest power of two >= s, for s > 0 or +inf (returned unchanged).  A
// normal s with a zero fraction is already one; otherwise the next exponent.
// A subnormal s is m * 2^-149 with m in [1, 2^23): the answer is 2^ceil(log2 m)
// units of 2^-149, whose bit pattern is that single bit (2^23 units = the
// smallest normal, bit 23, comes out the same way).
__device__ __forceinline__ float pow2_at_least(float s) {
  const uint32_t u = __float_as_uint(s);
  const uint32_t e = u >> 23, m = u & 0x7fffffu;
  if (e == 0) return __uint_as_float(1u << (32 - __clz(m - 1)));
  return (m == 0 || e == 0xffu) ? s : __uint_as_float((e + 1) << 23);
}

// Row b of the new rows into cache row `row` of slot b, by 128 threads of
// the calling CTA that form four whole warps; t in [0, 128) is the thread's
// index among them.  Warp t / 32 owns latent block t / 32 (128 values, 4 per
// lane): amax by shuffle, scale = amax / 448 (IEEE fp32 division; format 2
// rounds it up to a power of two), codes = e4m3 of x / scale with
// round-to-nearest-even and saturation.  An all-zero block stores scale 0
// and zero codes.
__device__ __forceinline__ void append_row(const AppendRows& p, int b, int row, int t) {
  const size_t r = (size_t)b * p.max_seq_len + row;
  const int blk = t >> 5, lane = t & 31;
  const int col = blk * kBlk + lane * 4;
  const uint2 raw = *reinterpret_cast<const uint2*>(
      static_cast<const __nv_bfloat16*>(p.kv_new) + (size_t)b * kDc + col);
  if (p.fmt == 0) {
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.kv) + r * kDc + col) = raw;
  } else {
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
    const float2 x01 = __bfloat1622float2(h2[0]);
    const float2 x23 = __bfloat1622float2(h2[1]);
    float amax = fmaxf(fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    float scale = __fdiv_rn(amax, 448.0f);
    if (p.fmt == 2 && amax > 0.0f) scale = pow2_at_least(scale);
    uint32_t packed = 0;
    if (amax > 0.0f) {
      const float2 y01 = make_float2(__fdiv_rn(x01.x, scale), __fdiv_rn(x01.y, scale));
      const float2 y23 = make_float2(__fdiv_rn(x23.x, scale), __fdiv_rn(x23.y, scale));
      const uint32_t lo = __nv_cvt_float2_to_fp8x2(y01, __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_float2_to_fp8x2(y23, __NV_SATFINITE, __NV_E4M3);
      packed = (lo & 0xffffu) | (hi << 16);
    }
    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(p.kv) + r * kDc + col) = packed;
    if (lane == 0) p.kv_scale[r * kNblk + blk] = scale;
  }
  if (t < 8) {  // rotary key: 64 bf16 = 8 x 16 bytes
    const uint4 v = reinterpret_cast<const uint4*>(
        static_cast<const __nv_bfloat16*>(p.pe_new) + (size_t)b * kDr)[t];
    reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.pe) + r * kDr)[t] = v;
  }
}

// A row is appended by a dense call only where the decode reads it: end_pos
// in [1, max_end_pos] (then row end_pos - 1 < max_seq_len).
__device__ __forceinline__ bool append_row_valid(int end, int max_end_pos) {
  return end >= 1 && end <= max_end_pos;
}

}  // namespace mla
