// decode_tc.cu -- absorbed MLA decode for H = 128 heads on the 5th-generation
// tensor cores (tcgen05 + TMEM), TMA-staged, one CTA pair (cluster of 2) per
// unit of positions.
//
// What is computed ("DeepSeek-V3.2-Exp . KV cache", MQA-decode excerpt;
// "DeepSeek MLA architecture ...", sections 3-4), per unit of positions:
//   S[h, t] = q_latent[h] . c[t] + q_pe[h] . kR[t]            (128 heads)
//   online softmax of S * softmax_scale over the unit's positions
//   O[h, :] = sum_t p[h, t] c[t, :]                           (512 latent)
// followed by the log-sum-exp combine across units (combine kernel).
//
// Why a pair: an fp32 accumulator for 128 heads x 512 latent columns fills all
// of one SM's tensor memory (512 columns x 128 lanes x 4 B), leaving no room
// for the scores.  So CTA r of the pair owns latent columns [256r, 256r+256)
// and rotary columns [32r, 32r+32) of the cache and of O, and half of the
// heads for the softmax: TMEM lanes 32 q + 16 r .. 32 q + 16 r + 15 of every
// lane quadrant q (head h lives in lane h).
//   * QK: each CTA contracts its 288-wide half (Q half as the A operand held in
//     tensor memory, K half from shared memory) into a partial S for all 128
//     heads.  The partial rows of the peer's 64 heads go to the peer through
//     distributed shared memory as 24-bit codes (each fp32 partial rounded to
//     its top 24 bits; asynchronous remote stores, counted on the receiver's
//     barrier), where they are added to the peer's own fp32 partial.
//   * softmax: each CTA runs the online softmax of its own 64 heads only and
//     writes their bf16 P rows into its own P buffer and into the peer's
//     (bulk copies of whole rows, or remote stores of 16-byte chunks for
//     dense bf16), with each head's rescale factor.
//   * PV: each CTA multiplies P of all 128 heads (shared memory) by its latent
//     half V (the same shared-memory tile, read as an MN-major operand) into
//     its own O half.  When the owner of a head raised the head's reference
//     maximum, the other CTA scales its row of that head first.
// Every cache byte is fetched by exactly one CTA and there is no redundant
// tensor-core or softmax work.  Interleaving the heads by quadrant puts one
// softmax warp on each of the SM's four schedulers.
//
// Tensor memory (512 columns): O half [0,256) fp32; Q half [256,400) bf16 (2
// per column); S double buffer [400,448) and [448,496) fp32.
//
// Warp roles (512 threads; 544 for dense FP8 tiles):
//   warp 0  producer: TMA tiles (dense), or four-row TMA gathers of the
//           latent halves and 16-byte copies of the small per-row pieces (gather)
//   warp 1  QK issuer (one thread) and tensor-memory owner
//   warp 2  PV issuer (one thread); in a dense bf16 call it first works out
//           the split schedule and the pair's unit (schedule.cuh)
//   warps 4-15  the head pool, three warps per TMEM lane quadrant (a warp may
//           access lanes 32 (warp & 3) .. + 31 only), by slot:
//           4-7   softmax of the quadrant's 16 own heads (16-lane TMEM
//                 access: thread t holds two heads x 12 positions a tile);
//                 warps 4-7 first stage the query half into tensor memory
//           8-11  senders of the quadrant's 16 peer heads' partial scores,
//                 and rescalers of those heads' rows of O (served while they
//                 wait); with new rows in a dense call they first write the
//                 row (the cache-write step)
//           12-15 converter (if any)
//           Slots 4-11 stage the output half in the epilogue.
//   warps 3, 12-15 and (dense FP8) 16  converter (FP8 caches and gathers): raw rows ->
//           bf16 operand tile bf16(fp32(e4m3 * scale)) in the 128-byte
//           swizzled layout
// Distributed shared memory moves ~20-35 GB/s per SM with ~0.3 us latency on
// this part, so each tile sends 9 KB of partial scores and 6-8 KB of P rows
// per direction.
//
// Every wait is bounded; on expiry the kernel raises a status bit, stops
// issuing work, and still runs its teardown (cluster barrier, TMEM release).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>
#include <string.h>

#include "append_row.cuh"
#include "common.cuh"
#include "schedule.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace ptx;

constexpr int kHalf = kDc / 2;             // 256 latent columns per CTA
constexpr int kPeHalf = kDr / 2;           // 32 rotary columns per CTA
// log2 units: p <= 2^16 between rescales (bf16 P and the fp32 sums hold that
// with a wide margin); a larger threshold means fewer rescales, each of
// which also holds up the peer's PV for its rows of the head
constexpr float kRescaleThreshold = 16.0f;
constexpr uint32_t kTmemO = 0, kTmemQ = 256, kTmemS = 400;
constexpr long kSpinLimit = 1L << 26;   // polls (~seconds) before giving up

// Shared-memory plan per variant.  Tiles are 48 positions (MMA N for QK, K
// for PV), with two S, P and exchange buffers.  An operand stage holds the
// swizzled bf16 latent half and rotary tile the MMAs read; it is taken from
// the load (dense bf16) or the conversion (FP8, gathers) of its tile until
// PV of that tile completes.  Variants with a converter load the rows as
// stored -- FP8 codes or gathered bf16 half rows, the 4 FP8 scales of each
// row, the 64 rotary values -- into a separate ring of raw slots, which the
// converter frees as soon as it has read them.  So a load never waits for a
// PV, and the HBM latency stays out of the operand stages' cycle.  The dense
// FP8 variant fills 227 KB exactly: four operand stages (the rotary operand
// only the CTA's 32 columns), four raw slots (the ring's cycle -- a load's
// latency plus the conversion -- bounds the tile period with three), two P
// and two exchange buffers.
template <int kFmt, bool kSparse>
struct Cfg {
  static constexpr bool kConv = kFmt == 1 || kSparse;       // converter warps present
  static constexpr int kN = 48;    // positions per tile
  static constexpr int kSBufs = 2;  // S buffers (tensor memory)
  // P buffers (shared memory): three where there is room (bf16), so the
  // softmax writes P of tile i once PV of tile i-3 is done -- PV of tile i-2
  // runs behind the QK of tile i in the in-order tensor pipe
  static constexpr int kPBufs = kFmt == 0 ? 3 : 2;
  static constexpr int kXBufs = 2;   // exchange buffers
  // Warps: 0 producer, 1 QK issuer, 2 PV issuer (a dense bf16 call's split
  // schedule first), 3 converter; 4-15 the head pool, three warps per TMEM
  // lane quadrant (quadrant = warp & 3, slot = (warp - 4) >> 2: softmax,
  // sender/rescaler, converter); 16 converter.  Variants without a converter
  // stop at warp 15 (warp 3 and the pool's third slot idle), and so do the
  // gather variants: with five converter warps they run at 128 registers a
  // thread (sixteen warps; seventeen are allocated as twenty, 96 registers),
  // which measured faster for gathers (workload 5 kernel 39.8 -> 37.7 us) and
  // slower for dense FP8 tiles (workload 4 203 -> 208 us).
  static constexpr int kSmWarps = 4;   // softmax warps: one per TMEM lane quadrant
  static constexpr int kConvWarps = kSparse ? 5 : 6;   // warp 3, the pool's four slot-2 warps, warp 16
  static constexpr int kThreads = 32 * (kConv && !kSparse ? 17 : 16);
  // QK may be issued at most this many tiles past the last issued PV: enough
  // run-ahead to keep the tensor pipe busy through the exchange and softmax
  // of a tile, no more -- the pipe runs its queue in order, so each queued QK
  // delays the PV behind it.  (Measured with the head-split softmax: 4 beats 3
  // by 3% on the FP8 workloads; the two S buffers bound it anyway.)
  static constexpr int kQkAhead = 4;
  static constexpr int kBlkBytes = kN * 128;       // one 64-column swizzled block of a tile
  static constexpr int kOplBytes = 4 * kBlkBytes;  // latent half operand
  // rotary operand: dense bf16 tiles land the full 64 columns (128-byte
  // swizzle, as stored); the converter variants write only the CTA's 32
  // columns (the ones its QK reads) as 8-row x 16-byte core matrices without
  // swizzle: core (row group g, chunk c) at 512 g + 128 c
  static constexpr int kOpeBytes = kConv ? kN * 64 : kBlkBytes;
  // P: 128 heads x kN bf16, swizzled (rows of 64 positions: chunks 6 and 7 of
  // a row are padding, which carries the peer's rescale factors and flags)
  static constexpr int kPBytes = ((kN + 63) / 64) * kSwBlk;
  static_assert(kN == 48, "P rows keep chunks 6 and 7 free");
  // exchange buffer: the kN partial scores of each of the peer's 64 heads as
  // 24-bit codes (the fp32 value rounded to its top 24 bits), four values in
  // three words.  A quadrant's 16 peer heads x kN positions travel from the
  // sender thread t to the softmax thread t of the same quadrant in the peer
  // (both hold the same fragment: two heads x kN / 4 positions), 18 words a
  // thread: four 16-byte rows at q * 512 + 16 t and 8 bytes at 2048 + 8 t of
  // the quadrant's kXQuad bytes, so a warp's remote store is contiguous.
  // Buffers are kXStride apart (bf16 variants keep twice the room: the query
  // is staged across the P and exchange buffers).
  static constexpr int kXQuad = 32 * 72;
  static constexpr int kXBytes = 4 * kXQuad;
  static constexpr int kXStride = kFmt == 1 ? kXBytes : 2 * kXBytes;
  // bytes of one tile's message of P rows to the peer: variants with a
  // converter send one block of 16 whole rows (128 bytes, padding included)
  // from each quadrant's softmax warp by bulk copy; dense bf16 sends the 64
  // rows' kN positions by remote stores of 16-byte chunks, one rescale factor
  // per row and one flag word per quadrant (measured faster there)
  static constexpr uint32_t kPMsgBytes = kConv ? 4 * 16 * 128 : 64 * kN * 2 + 64 * 4 + 4 * 4;
  static constexpr int kStage = kOplBytes + kOpeBytes;
  static constexpr int kStages = kConv ? (kFmt == 1 ? 4 : 2) : 4;
  static constexpr int kRawRow = kFmt == 1 ? kHalf : kHalf * 2;  // bytes of a raw latent half row
  // FP8 scales, 16 B per row, 48 consecutive rows
  static constexpr int kScBytes = kFmt == 1 ? 1024 : 0;
  // rotary bytes per raw row: only the CTA's 32 columns (the 32 its QK reads)
  static constexpr int kRawPe = kPeHalf * 2;
  static constexpr int kRaw = kConv ? kN * kRawRow + kScBytes + kN * kRawPe : 0;
  static constexpr int kRawSlots = kConv ? (kFmt == 1 ? (kSparse ? 3 : 4) : 2) : 0;
  // the converter's ring length in index arithmetic (never zero, so the
  // converter code of the variants without one compiles cleanly)
  static constexpr int kRawRing = kRawSlots > 0 ? kRawSlots : 1;
  static constexpr int kRawOff = kStages * kStage;
  static constexpr int kPOff = kRawOff + kRawSlots * kRaw;
  static constexpr int kXOff = kPOff + kPBufs * kPBytes;
  static constexpr int kBarOff = kXOff + kXBufs * kXStride;
  // query staging (5 swizzled blocks): the P and exchange buffers, or with
  // FP8 caches operand stages 1-3, which the converter fills only once the
  // query has moved to tensor memory
  static constexpr int kQOff = kFmt == 1 ? kStage : kPOff;
  static constexpr int kSmem = kBarOff + 4096 + 1024;      // barriers/flags + base alignment slack
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kStage % 1024 == 0 && kRaw % 1024 == 0, "1 KB alignment of swizzled tiles");
  static_assert(kN % 16 == 0 && kTmemS + kSBufs * kN <= 512, "tile width");
  // the output half is staged from offset 0 (8 blocks of 32 fp32 columns)
  static_assert(kFmt == 1 ? (kStages - 1) * kStage >= 5 * kSwBlk
                          : kPBufs * kPBytes + kXBufs * kXStride >= 5 * kSwBlk,
                "query staging fits");
  static_assert(kQOff % 1024 == 0 && kPOff % 1024 == 0, "1 KB alignment of the query staging");
  static_assert(kBarOff >= 8 * kSwBlk, "output staging fits the idle buffers");
};

struct TcParams {
  DecodeParams p;
  CUtensorMap m_kv;   // bf16: latent (box 64 x N), FP8: codes (box 256 x N)
  CUtensorMap m_pe;   // rotary (dense tiles; box 64 or 32 x N)
  CUtensorMap m_sc;   // FP8 scales (dense tiles; box 4 x N)
  CUtensorMap m_ql;   // q_latent [B][128][512] (box 64 x 128, 128-byte swizzle)
  CUtensorMap m_qp;   // q_pe [B][128][64] (box 64 x 128, 128-byte swizzle)
  CUtensorMap m_po;   // partial outputs [units][128][512] fp32 (box 32 x 128, 128-byte swizzle)
  CUtensorMap m_out;  // final output [B][128][512] bf16 (box 64 x 128, 128-byte swizzle)
};

// Named barriers: 1 among the 8 epilogue warps (pool slots 0 and 1); 6 among
// warps 4-7 after the query staging; 7 among the 12 pool warps before the
// epilogue.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void qstage_sync() { asm volatile("bar.sync 6, 128;" ::: "memory"); }
__device__ __forceinline__ void pool_sync() { asm volatile("bar.sync 7, 384;" ::: "memory"); }
// Partial scores cross between the pair as the top 24 bits of the fp32 value,
// rounded (add half the dropped unit, truncate): relative error at most 2^-16
// for normal values.  Each CTA adds the peer's rounded partial to its own
// unrounded one, so the two CTAs' scores may differ in the last bits; each CTA
// keeps its own softmax state (reference maximum, row sums) for its own half
// of the output, so nothing needs them to agree.
// four fp32 bit patterns -> three words of 24-bit codes: each value rounded
// (half the dropped unit added), then its top three bytes taken in order
__device__ __forceinline__ void pack24(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t& w0,
                                       uint32_t& w1, uint32_t& w2) {
  a += 0x80u;
  b += 0x80u;
  c += 0x80u;
  d += 0x80u;
  w0 = __byte_perm(a, b, 0x5321);   // a1 a2 a3 b1
  w1 = __byte_perm(b, c, 0x6532);   // b2 b3 c1 c2
  w2 = __byte_perm(c, d, 0x7653);   // c3 d1 d2 d3
}
__device__ __forceinline__ float4 unpack24(uint32_t w0, uint32_t w1, uint32_t w2) {
  return make_float4(__uint_as_float(w0 << 8), __uint_as_float(__funnelshift_r(w0, w1, 24) << 8),
                     __uint_as_float(__funnelshift_r(w1, w2, 16) << 8), __uint_as_float(w2 & 0xFFFFFF00u));
}

// 2^x with the hardware approximation (relative error far below the bf16
// rounding P receives); 0 for -inf
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}



// Shared state of the CTA (barriers, flags) at the tail of shared memory.
struct Bars {
  uint64_t full[4];    // tile landed: stage (dense bf16) or raw slot
  uint64_t deq[4];     // operand stage converted
  uint64_t empty[4];   // PV done: operand stage free
  uint64_t rfree[4];   // raw slot read by the converter
  uint64_t sfull[2], sfree[2];
  uint64_t pfull[3];   // P rows of this CTA's heads written (its softmax warps)
  uint64_t pfree[3];   // PV of the buffer's tile done in both CTAs (one multicast commit from each)
  uint64_t rpfull[3];  // the peer's P rows (with rescale factors and flags) landed
  uint64_t xfull[2], xempty[2];
  uint64_t lpeer;      // the peer's row sums of its heads landed (epilogue)
  uint64_t drain;      // final commit of the QK issuer
  uint64_t drain_pv;   // final commit of the PV issuer
  volatile int pv_issued;   // PV issuer: tiles whose PV is issued (paces QK)
  // rescale of the peer's heads' rows of O: the PV issuer posts tile + 1 in
  // resc_req and waits until both rescaler warps have counted it in resc_done
  volatile int resc_req;
  int resc_done;
  volatile int resc_stop;   // the PV issuer has issued its last PV (or gave up)
  uint64_t qbar;    // query rows staged in shared memory
  uint64_t qready;  // query half in tensor memory
  uint64_t appended;  // the new row is in the cache (dense call with new rows)
  Unit unit;          // this pair's unit, when the kernel computes the schedule
  uint32_t tmem;
  volatile int abort;
  float l_own[128];      // epilogue: row sums of this CTA's heads (indexed by head)
  float l_peer[128];     // epilogue: row sums of the peer's heads (sent by the peer)
};
static_assert(sizeof(Bars) <= 4096, "barrier block");

struct Waiter {
  Bars* bars;
  uint32_t* status;
  long lim;   // polls before giving up
  __device__ __forceinline__ bool wait(uint64_t* b, uint32_t parity) {
    for (long it = 0; it < lim; ++it) {
      if (bar_try(b, parity)) return true;
      if (bars->abort) return false;
    }
    bars->abort = 1;
    atomicOr(status, kDevTimeout);
    return false;
  }
  __device__ __forceinline__ bool wait_local(uint64_t* b, uint32_t parity) {
    for (long it = 0; it < lim; ++it) {
      if (bar_try_local(b, parity)) return true;
      if (bars->abort) return false;
    }
    bars->abort = 1;
    atomicOr(status, kDevTimeout);
    return false;
  }
  // teardown variant: ignores the abort flag (the awaited operation was
  // issued by this thread and completes on its own), still bounded
  __device__ __forceinline__ void drain(uint64_t* b, uint32_t parity) {
    for (long it = 0; it < lim; ++it)
      if (bar_try(b, parity)) return;
    atomicOr(status, kDevTimeout);
  }
};

// FP8 codes (16) x scale -> 16 bf16 values bf16(fp32(e4m3) * scale)
__device__ __forceinline__ void dequant16(uint4 v, float sc, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i >> 1] >> ((i & 1) * 16)) & 0xffffu);
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    // a pair of IEEE fp32 products, each rounded to nearest, then to bf16
    const __nv_bfloat162 bb = __float22bfloat162_rn(__fmul2_rn(f, make_float2(sc, sc)));
    o[i] = *reinterpret_cast<const uint32_t*>(&bb);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// Scale the O half's rows of the 16 TMEM lanes from `lanes` (a tensor-memory
// address with the lane field set): lane fl = t/4 by a, lane fl + 8 by b (the
// 16-lane access touches only those rows, so warps that own the other 16
// lanes of the quadrant may scale them at the same time).  Warp-collective.
__device__ __forceinline__ void scale_rows16(uint32_t lanes, float a, float b) {
#pragma unroll 1
  for (int c = 0; c < 8; ++c) {
    uint32_t r[16];
    TC_LD16L_X4(lanes + kTmemO + 32 * c, r);
    tc_wait_ld();
#pragma unroll
    for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * ((k & 2) ? b : a));
    TC_ST16L_X4(lanes + kTmemO + 32 * c, r);
  }
  tc_wait_st();
}

// Epilogue: O columns [32 c0, 32 c1) of TMEM lane h, times inv, into the
// 128-byte swizzled output blocks c0..c1-1 (16 KB each) at `out`.
__device__ __forceinline__ void stage_output(uint32_t lane_base, uint8_t* out, int h, float inv,
                                             int c0, int c1) {
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    uint32_t r[16], q[16];
    TC_LD16(lane_base + kTmemO + 32 * c, r);
    TC_LD16(lane_base + kTmemO + 32 * c + 16, q);
    tc_wait_ld();
    uint8_t* blk = out + c * kSwBlk;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      *reinterpret_cast<float4*>(blk + swz_chunk(h, k)) =
          make_float4(__uint_as_float(r[4 * k]) * inv, __uint_as_float(r[4 * k + 1]) * inv,
                      __uint_as_float(r[4 * k + 2]) * inv, __uint_as_float(r[4 * k + 3]) * inv);
      *reinterpret_cast<float4*>(blk + swz_chunk(h, 4 + k)) =
          make_float4(__uint_as_float(q[4 * k]) * inv, __uint_as_float(q[4 * k + 1]) * inv,
                      __uint_as_float(q[4 * k + 2]) * inv, __uint_as_float(q[4 * k + 3]) * inv);
    }
  }
}

// Epilogue of a sequence's only unit: O columns [32 c0, 32 c1) of TMEM lane
// h, times inv, rounded to bf16, into 128-byte swizzled blocks of 64 columns
// (16 KB each) at `out`.
__device__ __forceinline__ void stage_output_bf16(uint32_t lane_base, uint8_t* out, int h, float inv,
                                                  int c0, int c1) {
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    uint32_t r[32];
    TC_LD16(lane_base + kTmemO + 32 * c, r);
    TC_LD16(lane_base + kTmemO + 32 * c + 16, (r + 16));
    tc_wait_ld();
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const __nv_bfloat162 two = __floats2bfloat162_rn(__uint_as_float(r[2 * k]) * inv,
                                                       __uint_as_float(r[2 * k + 1]) * inv);
      pk[k] = *reinterpret_cast<const uint32_t*>(&two);
    }
    uint8_t* blk = out + (c >> 1) * kSwBlk;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint4*>(blk + swz_chunk(h, (c & 1) * 4 + k)) =
          make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
  }
}

template <int kFmt, bool kSparse>
__global__ void __launch_bounds__(Cfg<kFmt, kSparse>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ TcParams tp) {
  using C = Cfg<kFmt, kSparse>;
  constexpr int kN = C::kN, kBlkBytes = C::kBlkBytes, kOplBytes = C::kOplBytes,
                kOpeBytes = C::kOpeBytes;
  const DecodeParams& p = tp.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + C::kBarOff);

  const int unit_id = blockIdx.x >> 1;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const uint32_t peer = rank ^ 1u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Waiter wt{bars, p.ws.status, p.spin_limit > 0 ? (long)p.spin_limit : kSpinLimit};

  // the head pool: warp & 3 is the TMEM lane quadrant the warp may access.
  // This CTA owns heads (TMEM lanes) 32 q + 16 rank .. + 15 of every quadrant
  // q, the peer the other 16: each CTA's softmax, senders and rescalers have
  // one warp per quadrant, so they spread over all four schedulers.
  const int quad = warp & 3;
  const bool pool = warp >= 4 && warp < 16;
  const int slot = (warp - 4) >> 2;   // 0 softmax, 1 sender/rescaler, 2 converter
  const int hq = 32 * quad + lane;    // this lane's head under the 32-lane access (epilogue, rescales)
  const bool own_lane = (lane >> 4) == (int)rank;
  const int own_base = 32 * quad + 16 * (int)rank, peer_base = 32 * quad + 16 * (int)peer;
  // 16-lane fragments (TC_LD16L_*): this thread holds heads base + fl and
  // base + fl + 8 at the column pairs 8k + 2 fc, 8k + 2 fc + 1
  const int fl = lane >> 2, fc = lane & 3;
  // converter warps: 3, 16 (dense FP8) and the pool's third slot (one per
  // quadrant)
  const int conv_id = warp == 3 ? 0 : warp == 16 ? 1 : (pool && slot == 2) ? C::kConvWarps - 4 + quad : -1;

  auto opl = [&](int j) { return sm + j * C::kStage; };               // operand stage j
  auto ope = [&](int j) { return sm + j * C::kStage + kOplBytes; };
  auto raw = [&](int r) { return sm + C::kRawOff + r * C::kRaw; };    // raw slot r
  auto rsc = [&](int r) { return raw(r) + kN * C::kRawRow; };
  auto rpe = [&](int r) { return raw(r) + kN * C::kRawRow + C::kScBytes; };
  auto pbuf = [&](int b) { return sm + C::kPOff + b * C::kPBytes; };
  auto xbuf = [&](int b) { return sm + C::kXOff + b * C::kXStride; };
  // tile i uses S buffer ssel(i) and P buffer psel(i); spar(i) / ppar(i) is
  // the parity of the phase that tile completes on that buffer's barriers
  auto ssel = [](int i) { return i % C::kSBufs; };
  auto spar = [](int i) { return (uint32_t)((i / C::kSBufs) & 1); };
  auto psel = [](int i) { return i % C::kPBufs; };
  auto ppar = [](int i) { return (uint32_t)((i / C::kPBufs) & 1); };
  auto xsel = [](int i) { return i % C::kXBufs; };   // the same for exchange buffers
  auto xpar = [](int i) { return (uint32_t)((i / C::kXBufs) & 1); };

  // ---------------------------------------------------------------- set-up
  if (threadIdx.x == 0) {
    for (int j = 0; j < C::kStages; ++j) {
      bar_init(&bars->full[j], kSparse ? 33 : 1);   // gathers: + the producer's 32 lanes' copies
      bar_init(&bars->deq[j], C::kConvWarps);
      bar_init(&bars->empty[j], 1);
    }
    for (int r = 0; r < C::kRawSlots; ++r) bar_init(&bars->rfree[r], C::kConvWarps);
    for (int b = 0; b < C::kPBufs; ++b) {
      bar_init(&bars->pfull[b], C::kSmWarps);
      bar_init(&bars->pfree[b], 2);    // both CTAs' PV commits
      bar_init(&bars->rpfull[b], 1);   // one arrival (with the message's bytes) from the peer
    }
    for (int b = 0; b < 2; ++b) {
      bar_init(&bars->sfull[b], 1);
      bar_init(&bars->sfree[b], C::kSmWarps + 4);   // softmax and sender warps read S
      bar_init(&bars->xfull[b], 1);    // one arrival (with the tile's bytes) from the peer
      bar_init(&bars->xempty[b], C::kSmWarps);   // the peer's softmax warps
    }
    bar_init(&bars->lpeer, 1);
    bar_init(&bars->drain, 1);
    bar_init(&bars->drain_pv, 1);
    bars->pv_issued = 0;
    bars->resc_req = 0;
    bars->resc_done = 0;
    bars->resc_stop = 0;
    bar_init(&bars->qbar, 1);
    bar_init(&bars->qready, 4);
    bar_init(&bars->appended, 4);
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
        sa(&bars->tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = bars->tmem;
  cluster_sync();  // the peer's barriers are initialised before any remote arrive

  // The set-up above may overlap the previous kernel; from here on this
  // call's schedule (and everything before it in the stream) is complete.
  pdl_wait();
  pdl_trigger();
  const Unit u = [&]() -> Unit {
    // the dense bf16 and the gather variants compute their schedule (the
    // dense FP8 variant keeps the schedule kernel; see the host launcher)
    if constexpr (!kSparse && kFmt != 0) {
      return p.ws.units[unit_id];
    } else {
      if (p.sched.end_pos == nullptr && p.sched.lengths == nullptr) return p.ws.units[unit_id];
      // warp 2 works out the schedule and this pair's unit (the first pair's
      // rank-0 CTA also writes the combine's per-sequence table, the unit
      // count and the call's status word, afresh)
      if (warp == 2) {
        const bool writer = unit_id == 0 && rank == 0;
        uint32_t flags = 0;
        int units = 0;
        const Unit mine = warp_schedule(p.sched, unit_id, &flags, &units, writer ? p.ws.seq : nullptr);
        if (lane == 0) {
          bars->unit = mine;
          if (writer) {
            *p.ws.status = flags;
            *p.ws.n_units = units;
          }
        }
      }
      __syncthreads();
      return bars->unit;
    }
  }();
  const bool live = u.b >= 0;   // both CTAs of the cluster read the same unit
  const int ntiles = live ? (u.t1 - u.t0 + kN - 1) / kN : 0;
  // A dense call with new rows: the unit the schedule flagged (the
  // sequence's last; end_pos not clamped) writes row t1 - 1 = end_pos - 1
  // before its producer loads the last tile.  Both CTAs write the whole row
  // (the same bytes), so each loads only what it wrote itself.
  const bool app = !kSparse && live && (u.flags & kUnitAppend) && p.ap.kv_new != nullptr;

  // Q half -> tensor memory (A operand of QK): lane h, 2 bf16 per column.
  // Five TMA boxes stage the 128 rows (4 latent blocks of 64 columns, the 64
  // rotary columns, 128-byte swizzled) in idle buffers, so the producer starts
  // on the cache at once.  Each thread of warps 4-7 then moves its row to its
  // TMEM lane and signals the QK issuer, and the peer that its exchange
  // buffers may be written (the bf16 variants stage the query in them).
  if (live && warp >= 4 && warp < 8) {
    const int h = threadIdx.x - 128;
    uint8_t* qs = sm + C::kQOff;
    if (h == 0) {
      bar_expect_tx(&bars->qbar, 5 * kSwBlk);
      for (int blk = 0; blk < 4; ++blk)
        tma3(qs + blk * kSwBlk, &tp.m_ql, rank * kHalf + blk * 64, 0, u.b, &bars->qbar);
      tma3(qs + 4 * kSwBlk, &tp.m_qp, 0, 0, u.b, &bars->qbar);
    }
    wt.drain(&bars->qbar, 0);
    __syncwarp();   // the tensor-memory stores below are warp-collective
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
#pragma unroll
    for (int c = 0; c < 9; ++c) {  // 144 columns = 9 x 16 = 36 chunks of 16 bytes
      uint32_t r[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int q = 4 * c + k;   // chunk of this CTA's 288-column half row
        const uint8_t* src = q < 32 ? qs + (q >> 3) * kSwBlk + swz_chunk(h, q & 7)
                                    : qs + 4 * kSwBlk + swz_chunk(h, (q - 32) + 4 * (int)rank);
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        r[4 * k] = v.x; r[4 * k + 1] = v.y; r[4 * k + 2] = v.z; r[4 * k + 3] = v.w;
      }
      TC_ST16(lane_base + kTmemQ + 16 * c, r);
    }
    tc_wait_st();
    tc_before();
    __syncwarp();
    if (lane == 0) bar_arrive(&bars->qready);
    qstage_sync();
    // phase 0 of the peer's xempty[0/1]: this CTA's exchange buffers are free
    if (h == 0) {
      bar_arrive_remote_n(mapa(&bars->xempty[0], peer), C::kSmWarps);
      bar_arrive_remote_n(mapa(&bars->xempty[1], peer), C::kSmWarps);
    }
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // dense bf16: tile i lands swizzled in operand stage i % kStages, once PV
    // of its previous tile is done; converter variants: in raw slot
    // i % kRawSlots, once the converter has read its previous tile
    constexpr int kSlots = C::kConv ? C::kRawSlots : C::kStages;
    int issued = 0;
    for (int i = 0; i < ntiles && !bars->abort; ++i) {
      const int j = i % kSlots;
      const uint32_t use = i / kSlots;
      if (!wt.wait_local(C::kConv ? &bars->rfree[j] : &bars->empty[j], (use & 1) ^ 1)) break;
      const int e0 = u.t0 + i * kN;
      const int slot = u.b / p.mtp_s;   // cache slot of the sequence (several per slot: multi-token)
      if (unit_id == 0 && i == p.withhold_tile) {
        // self-test: this tile's load is never issued, so the waits on it run
        // out (the drain below skips it)
        continue;
      }
      // the tile that holds the new row: its writers fenced their stores
      // for the tensor copies before arriving
      if (app && i == ntiles - 1 && !wt.wait_local(&bars->appended, 0)) break;
      if (!kSparse) {
        if (lane == 0) {
          if (kFmt == 0) {
            bar_expect_tx(&bars->full[j], kOplBytes + kOpeBytes);
            for (int blk = 0; blk < 4; ++blk)
              tma3(opl(j) + blk * kBlkBytes, &tp.m_kv, rank * kHalf + blk * 64, e0, slot, &bars->full[j]);
            tma3(ope(j), &tp.m_pe, 0, e0, slot, &bars->full[j]);
          } else {
            bar_expect_tx(&bars->full[j], kN * kHalf + kN * 16 + kN * C::kRawPe);
            tma3(raw(j), &tp.m_kv, rank * kHalf, e0, slot, &bars->full[j]);
            tma3(rsc(j), &tp.m_sc, 0, e0, slot, &bars->full[j]);
            tma3(rpe(j), &tp.m_pe, rank * kPeHalf, e0, slot, &bars->full[j]);
          }
        }
      } else {
        // gathered rows: the latent halves four per TMA instruction
        // (tile::gather4 on row-high boxes, lane g rows 4g..4g+3; a short
        // last group repeats its last row), the small per-row pieces -- the
        // FP8 scales, the CTA's 32 rotary columns -- by 16-byte asynchronous
        // copies from every lane, which keeps them off the copy engine whose
        // issue rate bounds the gather.  The converter ignores rows past the
        // unit.
        const int v = min(kN, u.t1 - e0);
        const int groups = (v + 3) / 4;
        // the tile's rows: lane l reads list positions l and l + 32 (one
        // round of index loads), shared by shuffles
        const int* gl = p.ws.gidx + (size_t)u.b * p.K + e0;
        const int base = u.b * p.max_seq_len;
        const int g0 = base + gl[min(lane, v - 1)], g1 = base + gl[min(lane + 32, v - 1)];
        if (lane == 0) bar_expect_tx(&bars->full[j], (uint32_t)groups * 4 * C::kRawRow);
        __syncwarp();
        int r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = min(4 * lane + k, v - 1);
          const int a0 = __shfl_sync(0xffffffffu, g0, t & 31), a1 = __shfl_sync(0xffffffffu, g1, t & 31);
          r[k] = t < 32 ? a0 : a1;
        }
        if (lane < groups)
          tma_gather4(raw(j) + 4 * lane * C::kRawRow, &tp.m_kv, rank * kHalf, r[0], r[1], r[2], r[3],
                      &bars->full[j]);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int t = lane + 32 * h2;
          if (t >= v) break;
          const size_t row = (size_t)(h2 ? g1 : g0);
          if (kFmt == 1) cp_async16(rsc(j) + t * 16, p.kv_scale + row * kNblk);
          const uint8_t* pe = static_cast<const uint8_t*>(p.pe) + row * (kDr * 2) + rank * (kPeHalf * 2);
#pragma unroll
          for (int q = 0; q < 4; ++q) cp_async16(rpe(j) + t * C::kRawPe + q * 16, pe + q * 16);
        }
        cp_async_arrive(&bars->full[j]);   // every lane, once per tile
      }
      issued = i + 1;
    }
    // copies still in flight must land before this CTA's shared memory goes
    // away; on the normal path every stage was already consumed
    if (lane == 0 && bars->abort) {
      for (int i = issued > kSlots ? issued - kSlots : 0; i < issued; ++i)
        if (!(unit_id == 0 && i == p.withhold_tile)) wt.drain(&bars->full[i % kSlots], (i / kSlots) & 1);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ PV issuer
    // P of tile i: this CTA's heads from its own softmax, the peer's heads
    // from the peer.  When the peer rescaled some of its heads in this tile,
    // the rescaler warps first scale those heads' rows of this CTA's O half.
    // The commit reaches pfree in both CTAs (each P buffer is written by
    // both), empty only here.
    if (lane == 0) {
      constexpr uint32_t id_pv = idesc(128, kHalf, true);
      const uint64_t d_v0 = sdesc(sa(opl(0)), kBlkBytes, 1024);
      const uint64_t d_p0 = sdesc(sa(pbuf(0)), 16, 1024);
      const uint32_t t_o = tmem + kTmemO;
      int nreq = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int j = i % C::kStages, b = psel(i);
        if (!wt.wait_local(&bars->pfull[b], ppar(i))) break;
        if (!wt.wait(&bars->rpfull[b], ppar(i))) break;
        // the peer's rows were written by another CTA's asynchronous stores:
        // order them before the tensor core reads the buffer
        fence_async_smem();
        const uint8_t* pb = pbuf(b);
        uint32_t flags = 0;   // one word per quadrant, in the padding of its first peer row
#pragma unroll
        for (int q = 0; q < 4; ++q)
          flags |= *reinterpret_cast<const volatile uint32_t*>(pb + swz_chunk(32 * q + 16 * (int)peer, 7));
        if (flags) {
          // the rescalers scale rows of O that PV of tile i - 1 writes
          if (i > 0 && !wt.wait(&bars->pfree[psel(i - 1)], ppar(i - 1))) break;
          ++nreq;
          asm volatile("st.release.cta.shared.b32 [%0], %1;" ::"r"(sa((const void*)&bars->resc_req)), "r"(i + 1)
                       : "memory");
          bool done = false;
          for (long it = 0; it < wt.lim && !bars->abort; ++it) {
            int d;
            asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(d) : "r"(sa(&bars->resc_done)) : "memory");
            if (d >= 4 * nreq) {
              done = true;
              break;
            }
          }
          if (!done) {
            if (!bars->abort) {
              bars->abort = 1;
              atomicOr(p.ws.status, kDevTimeout);
            }
            break;
          }
        }
        tc_after();
        const uint64_t pd = sdesc_at(d_p0, b * C::kPBytes), vd = sdesc_at(d_v0, j * C::kStage);
        if (i == 0)
          mma_ss_c<false>(t_o, pd, vd, id_pv);
        else
          mma_ss_c<true>(t_o, pd, vd, id_pv);
#pragma unroll
        for (int kk = 1; kk < kN / 16; ++kk)
          mma_ss_c<true>(t_o, sdesc_at(pd, (kk >> 2) * kSwBlk + (kk & 3) * 32), sdesc_at(vd, 2048 * kk), id_pv);
        mma_commit_mc(&bars->pfree[b], 3);
        mma_commit(&bars->empty[j]);
        bars->pv_issued = i + 1;
      }
      bars->resc_stop = 1;
      mma_commit(&bars->drain_pv);
      wt.drain(&bars->drain_pv, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc(128, kN, false);
      const uint64_t d_k0 = sdesc(sa(opl(0)), 16, 1024);
      const uint32_t t_q = tmem + kTmemQ;
      if (live && wt.wait_local(&bars->qready, 0)) tc_after();
      for (int k = 0; k < ntiles && !bars->abort; ++k) {
        const int j = k % C::kStages, b = ssel(k);
        bool paced = false;
        for (long it = 0; it < wt.lim && !bars->abort; ++it)
          if (bars->pv_issued > k - C::kQkAhead) {
            paced = true;
            break;
          }
        if (!paced) {
          if (!bars->abort) {
            bars->abort = 1;
            atomicOr(p.ws.status, kDevTimeout);
          }
          break;
        }
        if (!wt.wait_local(C::kConv ? &bars->deq[j] : &bars->full[j], (k / C::kStages) & 1)) break;
        if (!wt.wait_local(&bars->sfree[b], spar(k) ^ 1)) break;
        tc_after();
        const uint32_t sd = tmem + kTmemS + b * kN;
        const uint64_t kd = sdesc_at(d_k0, j * C::kStage);
        const uint64_t ped = C::kConv ? sdesc_plain(sa(ope(j)), 128, 512) : sdesc_at(kd, kOplBytes + rank * (kPeHalf * 2));
        constexpr uint32_t kPeStep = C::kConv ? 256 : 32;   // bytes per 16 columns
        mma_ts_c<false>(sd, t_q, kd, id_qk);
#pragma unroll
        for (int kk = 1; kk < kHalf / 16; ++kk)
          mma_ts_c<true>(sd, t_q + 8 * kk, sdesc_at(kd, (kk >> 2) * kBlkBytes + (kk & 3) * 32), id_qk);
#pragma unroll
        for (int kk = 0; kk < kPeHalf / 16; ++kk)
          mma_ts_c<true>(sd, t_q + kHalf / 2 + 8 * kk, sdesc_at(ped, kPeStep * kk), id_qk);
        mma_commit(&bars->sfull[b]);
      }
      mma_commit(&bars->drain);
      wt.drain(&bars->drain, 0);
    }
  } else if (pool && slot == 1) {
    // ------------------------------------------------------------ sender / rescaler
    // Partial S of the peer's 16 heads of this quadrant -> the peer's
    // exchange buffer, as soon as each tile's scores are computed.  (With new
    // rows in a dense call, the four warps first write the row: the
    // cache-write step, while they wait for the first scores.)
    // Rescaler duty, served inside this warp's waits: when the peer raises
    // the reference maximum of one of its heads, this CTA's row of that head
    // in O (its latent half) is scaled by the factor the peer sent with the
    // tile's P rows, before PV of that tile.  The PV issuer posts the request
    // once PV of the previous tile is complete and waits for all four warps.
    if (app) {
      append_row(p.ap, u.b, u.t1 - 1, 32 * quad + lane);
      fence_async_global();
      __syncwarp();
      if (lane == 0) bar_arrive(&bars->appended);
    }
    const uint32_t tl = tmem + ((uint32_t)peer_base << 16);
    const uint32_t off_aA = swz_chunk(peer_base + fl, 6), off_aB = swz_chunk(peer_base + fl + 8, 6);
    int handled = 0;
    // one look at the request word; true if a request was served.  Tensor-
    // memory loads and stores are warp-collective, so the whole warp takes
    // the branch when any of its 16 rows needs scaling (factor 1 for the
    // others).
    auto serve = [&]() -> bool {
      __syncwarp();
      int req;
      asm volatile("ld.acquire.cta.shared.b32 %0, [%1];" : "=r"(req) : "r"(sa((const void*)&bars->resc_req)) : "memory");
      if (req <= handled) return false;
      const int i = req - 1;
      tc_after();
      const uint8_t* pb = pbuf(psel(i));
      const float a = *reinterpret_cast<const float*>(pb + off_aA);
      const float bb = *reinterpret_cast<const float*>(pb + off_aB);
      if (__any_sync(0xffffffffu, a != 1.f || bb != 1.f)) scale_rows16(tl, a, bb);
      tc_before();
      __syncwarp();
      if (lane == 0)
        asm volatile("red.release.cta.shared.add.s32 [%0], 1;" ::"r"(sa(&bars->resc_done)) : "memory");
      handled = req;
      return true;
    };
    // a bounded wait that serves rescale requests while it polls
    auto swait_local = [&](uint64_t* bar, uint32_t parity) -> bool {
      for (long it = 0; it < wt.lim; ++it) {
        if (bar_try_local(bar, parity)) return true;
        if (bars->abort) return false;
        if (serve()) it = 0;
      }
      if (!bars->abort) {
        bars->abort = 1;
        atomicOr(p.ws.status, kDevTimeout);
      }
      return false;
    };
    auto swait = [&](uint64_t* bar, uint32_t parity) -> bool {
      for (long it = 0; it < wt.lim; ++it) {
        if (bar_try(bar, parity)) return true;
        if (bars->abort) return false;
        if (serve()) it = 0;
      }
      if (!bars->abort) {
        bars->abort = 1;
        atomicOr(p.ws.status, kDevTimeout);
      }
      return false;
    };
    // the peer's exchange buffer 0 (this thread's rows) and its xfull[0];
    // buffer b is a fixed stride further (distributed shared addresses of one
    // CTA are linear)
    const uint32_t xd0 = mapa(xbuf(0) + quad * C::kXQuad + 16 * lane, peer);
    const uint32_t xe0 = mapa(xbuf(0) + quad * C::kXQuad + 2048 + 8 * lane, peer);
    const uint32_t xf0 = mapa(&bars->xfull[0], peer);
    for (int i = 0; i < ntiles; ++i) {
      const int b = ssel(i);
      if (!swait_local(&bars->sfull[b], spar(i))) break;
      __syncwarp();
      tc_after();
      uint32_t r[24];
      TC_LD16L_X4(tl + kTmemS + b * kN, r);
      TC_LD16L_X2(tl + kTmemS + b * kN + 32, (r + 16));
      tc_wait_ld();
      tc_before();
      __syncwarp();
      if (lane == 0) bar_arrive(&bars->sfree[b]);
      const int xb = xsel(i);
      if (!swait(&bars->xempty[xb], xpar(i))) break;   // phase 0: the peer's query staging is done
      const uint32_t xd = xd0 + xb * C::kXStride, xe = xe0 + xb * C::kXStride, xf = xf0 + xb * 8u;
      uint32_t w[18];
#pragma unroll
      for (int g = 0; g < 6; ++g)
        pack24(r[4 * g], r[4 * g + 1], r[4 * g + 2], r[4 * g + 3], w[3 * g], w[3 * g + 1], w[3 * g + 2]);
      // the peer's phase completes on one arrival carrying the tile's bytes
      // and on those bytes landing, in either order
      if (quad == 0 && lane == 0) bar_arrive_expect_tx_remote(xf, C::kXBytes);
#pragma unroll
      for (int q = 0; q < 4; ++q) st_async_v4(xd + 512 * q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3], xf);
      st_async_v2(xe, w[16], w[17], xf);
    }
    // serve the remaining requests until the PV issuer is done
    for (long it = 0; it < wt.lim && !bars->abort; ++it) {
      if (serve()) {
        it = 0;
      } else if (bars->resc_stop) {
        if (!serve()) break;
      }
    }
  } else if (pool && slot == 0) {
    // ------------------------------------------------------------ softmax
    // One warp per quadrant runs the online softmax of the CTA's 16 heads of
    // that quadrant over all kN positions of a tile: thread t holds heads
    // hA = base + t/4 and hB = hA + 8 at positions 8k + 2 (t%4) and
    // 8k + 2 (t%4) + 1 (k = 0..5), 12 per head; the four threads of a head
    // agree on its tile maximum by shuffles.  P is written into this CTA's
    // buffer (4-byte pieces) and sent to the peer's: with a converter, the
    // warp's 16 rows by one bulk copy (shared memory to shared memory,
    // counted on the peer's barrier), the rows' padding carrying the rescale
    // factors and the quadrant's flag; dense bf16, as 16-byte chunks read
    // back and sent by remote stores, the factors and flag stored beside
    // them.
    const int hA = own_base + fl, hB = hA + 8;
    const uint32_t tl = tmem + ((uint32_t)own_base << 16);
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    const float ps = pos_scale ? sl2 : 1.f;   // the factor still to apply to sc in P
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    bool ok = true;
    // loop-invariant addresses: the peer's P buffer 0, rpfull[0] and
    // xempty[0] (buffer b of each is a fixed stride further), and (dense
    // bf16) the three 16-byte P chunks this thread forwards (chunk c = fc +
    // 4 j of its head pair: hA's chunks 0-5, then hB's)
    const uint32_t rp0 = mapa(pbuf(0), peer), rbar0 = mapa(&bars->rpfull[0], peer);
    const uint32_t rxe0 = mapa(&bars->xempty[0], peer);
    uint32_t fwd[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int c = fc + 4 * j;
      fwd[j] = swz_chunk(c < 6 ? hA : hB, c < 6 ? c : c - 6);
    }
    const uint32_t off_aA = swz_chunk(hA, 6), off_aB = swz_chunk(hB, 6), off_f = swz_chunk(own_base, 7);
    for (int i = 0; i < ntiles; ++i) {
      const int j = i % C::kStages, sb_i = ssel(i), b = psel(i);
      const uint32_t par = ppar(i);
      float sc[24];
      ok = ok && wt.wait_local(&bars->sfull[sb_i], spar(i));
      {
        tc_after();
        uint32_t r[24];
        TC_LD16L_X4(tl + kTmemS + sb_i * kN, r);
        TC_LD16L_X2(tl + kTmemS + sb_i * kN + 32, (r + 16));
        tc_wait_ld();
#pragma unroll
        for (int k = 0; k < 24; ++k) sc[k] = __uint_as_float(r[k]);
        tc_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&bars->sfree[sb_i]);   // QK of tile i + kSBufs may overwrite
      }
      // + the peer's partial (rounded to 24 bits), sent by the peer's sender
      // thread that holds the same fragment
      const int xb = xsel(i);
      ok = ok && wt.wait(&bars->xfull[xb], xpar(i));
      {
        const uint8_t* xr = xbuf(xb) + quad * C::kXQuad;
        uint32_t w[18];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = *reinterpret_cast<const uint4*>(xr + 512 * q + 16 * lane);
          w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
        }
        const uint2 v2 = *reinterpret_cast<const uint2*>(xr + 2048 + 8 * lane);
        w[16] = v2.x; w[17] = v2.y;
#pragma unroll
        for (int k = 0; k < 6; ++k) {
          const float4 v = unpack24(w[3 * k], w[3 * k + 1], w[3 * k + 2]);
          const float2 a = __fadd2_rn(make_float2(sc[4 * k], sc[4 * k + 1]), make_float2(v.x, v.y));
          const float2 c2 = __fadd2_rn(make_float2(sc[4 * k + 2], sc[4 * k + 3]), make_float2(v.z, v.w));
          sc[4 * k] = a.x; sc[4 * k + 1] = a.y; sc[4 * k + 2] = c2.x; sc[4 * k + 3] = c2.y;
        }
        __syncwarp();
        // the buffer may be refilled: the values read above are already in
        // registers, so no release ordering is needed
        if (lane == 0) bar_arrive_remote_relaxed(rxe0 + xb * 8u);
      }
      // masked scores and the tile maxima of the two heads.  With a positive
      // scale the scores stay unscaled here: round-to-nearest is monotone, so
      // the maximum of the scaled scores is the scaled maximum, and P below
      // takes scale and reference in one fused multiply-add.  (A scale <= 0
      // scales first.)
      const int valid = min(kN, u.t1 - (u.t0 + i * kN));
      if (!pos_scale) {
#pragma unroll
        for (int k = 0; k < 24; ++k) sc[k] *= sl2;
      }
      if (valid < kN) {   // the unit's last tile
#pragma unroll
        for (int k = 0; k < 24; ++k)
          if (8 * (k >> 2) + 2 * fc + (k & 1) >= valid) sc[k] = -INFINITY;
      }
      float xa = fmaxf(sc[0], sc[1]), xbm = fmaxf(sc[2], sc[3]);
#pragma unroll
      for (int k = 1; k < 6; ++k) {
        xa = fmaxf(xa, fmaxf(sc[4 * k], sc[4 * k + 1]));
        xbm = fmaxf(xbm, fmaxf(sc[4 * k + 2], sc[4 * k + 3]));
      }
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
      xbm = fmaxf(xbm, __shfl_xor_sync(0xffffffffu, xbm, 1));
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
      xbm = fmaxf(xbm, __shfl_xor_sync(0xffffffffu, xbm, 2));
      const float mtA = pos_scale ? xa * sl2 : xa, mtB = pos_scale ? xbm * sl2 : xbm;
      // lazy rescale of the running reference maxima
      const bool needA = ok && mtA > mA + kRescaleThreshold, needB = ok && mtB > mB + kRescaleThreshold;
      float alA = 1.f, alB = 1.f;
      if (__any_sync(0xffffffffu, needA || needB)) {
        const float nA = needA ? mtA : mA, nB = needB ? mtB : mB;
        alA = exp2f(mA - nA);   // 0 when the reference was -inf
        alB = exp2f(mB - nB);
        if (i > 0) {
          // O holds tiles < i: wait for PV of tile i-1 (its P buffer's release;
          // the previous use of that buffer is known complete, so the parity
          // wait cannot be fooled by a phase two steps back), then scale the
          // rows of this thread's two heads (the 16-lane access leaves the
          // peer's rows of the quadrant to the rescaler)
          ok = ok && wt.wait(&bars->pfree[psel(i - 1)], ppar(i - 1));
          __syncwarp();
          tc_after();
          scale_rows16(tl, alA, alB);
        }
        lA *= alA;
        lB *= alB;
        mA = nA;
        mB = nB;
      }
      // P of the two heads (bf16): the pair of positions of chunk k is 4 bytes
      // at offset 4 fc of the chunk; l sums the fp32 values before rounding
      ok = ok && wt.wait(&bars->pfree[b], par ^ 1);
      uint8_t* prow = pbuf(b);
      const float2 ps2 = make_float2(ps, ps), nA2 = make_float2(-mA, -mA), nB2 = make_float2(-mB, -mB);
      float2 sA = make_float2(0.f, 0.f), sB = sA;
#pragma unroll
      for (int k = 0; k < 6; ++k) {
        const float2 tA = __ffma2_rn(make_float2(sc[4 * k], sc[4 * k + 1]), ps2, nA2);
        const float2 tB = __ffma2_rn(make_float2(sc[4 * k + 2], sc[4 * k + 3]), ps2, nB2);
        const float2 eA = make_float2(ex2_approx(tA.x), ex2_approx(tA.y));
        const float2 eB = make_float2(ex2_approx(tB.x), ex2_approx(tB.y));
        sA = __fadd2_rn(sA, eA);
        sB = __fadd2_rn(sB, eB);
        const __nv_bfloat162 pa = __float22bfloat162_rn(eA), pb = __float22bfloat162_rn(eB);
        *reinterpret_cast<__nv_bfloat162*>(prow + swz_chunk(hA, k) + 4 * fc) = pa;
        *reinterpret_cast<__nv_bfloat162*>(prow + swz_chunk(hB, k) + 4 * fc) = pb;
      }
      lA += sA.x + sA.y;
      lB += sB.x + sB.y;
      __syncwarp();
      // the P rows (written by all the warp's threads) to the peer's buffer,
      // with the heads' rescale factors and the quadrant's "some head
      // rescaled" flag
      {
        const uint32_t rp = rp0 + b * C::kPBytes, rbar = rbar0 + b * 8u;
        // (tile 0 sets the first references: O holds nothing yet)
        const bool any = __any_sync(0xffffffffu, i > 0 && (alA != 1.f || alB != 1.f));
        if constexpr (C::kConv) {
          if (fc == 0) {
            *reinterpret_cast<float*>(prow + off_aA) = alA;
            *reinterpret_cast<float*>(prow + off_aB) = alB;
          }
          if (lane == 0) *reinterpret_cast<uint32_t*>(prow + off_f) = any ? 1u : 0u;
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (quad == 0) bar_arrive_expect_tx_remote(rbar, C::kPMsgBytes);
            bulk_s2c(rp + own_base * 128, prow + own_base * 128, 16 * 128, rbar);
          }
        } else {
          if (quad == 0 && lane == 0) bar_arrive_expect_tx_remote(rbar, C::kPMsgBytes);
#pragma unroll
          for (int jj = 0; jj < 3; ++jj) {
            const uint4 v = *reinterpret_cast<const uint4*>(prow + fwd[jj]);
            st_async_v4(rp + fwd[jj], v.x, v.y, v.z, v.w, rbar);
          }
          if (fc == 0) {
            st_async_b32(rp + off_aA, __float_as_uint(alA), rbar);
            st_async_b32(rp + off_aB, __float_as_uint(alB), rbar);
          }
          if (lane == 0) st_async_b32(rp + off_f, any ? 1u : 0u, rbar);
        }
      }
      if (!C::kConv && valid < kN) {
        // dense bf16 tail: rows past the unit hold whatever the cache holds
        // there; zero them so P = 0 never meets a non-finite value
        uint8_t* v = opl(j);
        for (int idx = 32 * quad + lane; idx < (kN - valid) * 32; idx += 128) {
          const int row = valid + idx / 32, blk = (idx / 8) & 3, ch = idx & 7;
          *reinterpret_cast<uint4*>(v + blk * kBlkBytes + swz_chunk(row, ch)) = make_uint4(0, 0, 0, 0);
        }
      }
      // (converter variants: the fence before the bulk copy already ordered
      // every generic write of this tile's P for the tensor core)
      if constexpr (!C::kConv) fence_async_smem();
      tc_before();
      __syncwarp();
      if (lane == 0) bar_arrive(&bars->pfull[b]);
    }
    // the heads' row sums (the four threads' parts), log-sum-exps, and the
    // row sums sent to the peer for its normalisation of these rows
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    if (live && fc == 0) {
      bars->l_own[hA] = lA;
      bars->l_own[hB] = lB;
      const uint32_t lbar = mapa(&bars->lpeer, peer);
      if (quad == 0 && lane == 0) bar_arrive_expect_tx_remote(lbar, 64 * 4);
      st_async_b32(mapa(&bars->l_peer[hA], peer), __float_as_uint(lA), lbar);
      st_async_b32(mapa(&bars->l_peer[hB], peer), __float_as_uint(lB), lbar);
      const bool fin = ok && !bars->abort;
      const float lseA = (fin && lA > 0.f) ? (mA + log2f(lA)) * 0.69314718055994531f : -INFINITY;
      const float lseB = (fin && lB > 0.f) ? (mB + log2f(lB)) * 0.69314718055994531f : -INFINITY;
      if (!(u.flags & kUnitDirect)) {
        p.ws.part_lse[(size_t)unit_id * p.H + hA] = lseA;
        p.ws.part_lse[(size_t)unit_id * p.H + hB] = lseB;
      } else if (p.lse) {
        p.lse[(size_t)u.b * p.H + hA] = lseA;
        p.lse[(size_t)u.b * p.H + hB] = lseB;
      }
    }
  } else if (C::kConv && conv_id >= 0) {
    // ------------------------------------------------------------ converter
    // raw slot r of tile i -> operand stage j, once the rows have landed and
    // PV of the stage's previous tile is done; C::kConvWarps warps share a tile
    const int t = 32 * conv_id + lane;
    for (int i = 0; i < ntiles; ++i) {
      const int r = i % C::kRawRing, j = i % C::kStages;
      // FP8: stages 1-3 hold the staged query until it is in tensor memory
      if (kFmt == 1 && i == 1 && !wt.wait_local(&bars->qready, 0)) break;
      if (!wt.wait_local(&bars->full[r], (i / C::kRawRing) & 1)) break;
      if (!wt.wait_local(&bars->empty[j], ((i / C::kStages) & 1) ^ 1)) break;
      const int valid = min(kN, u.t1 - (u.t0 + i * kN));
      uint8_t* dst = opl(j);
      if (kFmt == 1) {
        // 48 rows x 16 chunks of 16 codes -> 2 swizzled 16-byte chunks each
        for (int idx = t; idx < kN * 16; idx += 32 * C::kConvWarps) {
          const int row = idx >> 4, q = idx & 15;  // codes [16q, 16q + 16) of the half row
          uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
          if (row < valid) {
            const uint4 v = *reinterpret_cast<const uint4*>(raw(r) + row * kHalf + q * 16);
            const uint8_t* srow = rsc(r) + row * 16;
            const float sc = reinterpret_cast<const float*>(srow)[rank * 2 + (q >> 3)];
            dequant16(v, sc, lo, hi);
          }
          const int blk = q >> 2, ch = (q & 3) * 2;
          // odd blocks store their odd chunk first: a quarter-warp (two blocks
          // of one row) then covers all eight chunk positions of the
          // 128-byte swizzle row per store, free of bank conflicts
          const bool flip = blk & 1;
          const uint4 v1 = flip ? hi : lo, v2 = flip ? lo : hi;
          *reinterpret_cast<uint4*>(dst + blk * kBlkBytes + swz_chunk(row, ch + (flip ? 1 : 0))) = v1;
          *reinterpret_cast<uint4*>(dst + blk * kBlkBytes + swz_chunk(row, ch + (flip ? 0 : 1))) = v2;
        }
      } else {
        // gathered bf16 rows: 48 rows x 32 chunks of 8 values
        for (int idx = t; idx < kN * 32; idx += 32 * C::kConvWarps) {
          const int row = idx >> 5, q = idx & 31;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < valid) v = *reinterpret_cast<const uint4*>(raw(r) + row * C::kRawRow + q * 16);
          *reinterpret_cast<uint4*>(dst + (q >> 3) * kBlkBytes + swz_chunk(row, q & 7)) = v;
        }
      }
      // the CTA's 32 rotary columns (the only ones its QK reads) -> unswizzled
      // core matrices
      for (int idx = t; idx < kN * 4; idx += 32 * C::kConvWarps) {
        const int row = idx >> 2, q = idx & 3;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < valid) v = *reinterpret_cast<const uint4*>(rpe(r) + row * C::kRawPe + q * 16);
        *reinterpret_cast<uint4*>(ope(j) + (row >> 3) * 512 + q * 128 + (row & 7) * 16) = v;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        bar_arrive(&bars->deq[j]);
        bar_arrive(&bars->rfree[r]);
      }
    }
  }

  // -------------------------------------------------------------- epilogue
  // Every pool warp meets here once its role is done; the softmax warps have
  // stored their heads' row sums (and sent them to the peer).  The softmax
  // and sender warps of every quadrant (8 warps) then stage the O half (128
  // heads x 256 fp32), each row normalised by its head's l -- this CTA's
  // heads from its own sums, the peer's heads from the peer's -- in four
  // rounds of one 32-column block per thread: the TMA stores of the blocks a
  // round completes leave while the next round is staged.  With the last PV
  // complete in both CTAs, every stage, P and exchange buffer is idle, so the
  // half is staged from offset 0.  A sequence's only unit writes the final
  // bf16 output (4 blocks of 64 columns: two 32-column chunks each, complete
  // after rounds 1 and 3) itself.
  if (live && pool) {
    pool_sync();
    if (slot < 2) {
      bool ok = true;
      if (ntiles > 0) ok = wt.wait(&bars->pfree[psel(ntiles - 1)], ppar(ntiles - 1));
      float lt;
      if (own_lane) {
        lt = bars->l_own[hq];
      } else {
        ok = wt.wait(&bars->lpeer, 0) && ok;
        lt = bars->l_peer[hq];
      }
      __syncwarp();   // the tensor-memory loads below are warp-collective
      tc_after();
      const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
      const float inv = (ok && lt > 0.f) ? 1.f / lt : 0.f;
      const bool direct = (u.flags & kUnitDirect) != 0;
      const int sh = slot;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        if (direct)
          stage_output_bf16(lane_base, sm, hq, inv, 4 * sh + q, 4 * sh + q + 1);
        else
          stage_output(lane_base, sm, hq, inv, 4 * sh + q, 4 * sh + q + 1);
        fence_async_smem();
        epi_sync();
        if (warp == 4 && lane == 0) {
          if (!direct) {
            tma3_store(&tp.m_po, rank * kHalf + 32 * q, 0, unit_id, sm + q * kSwBlk);
            tma3_store(&tp.m_po, rank * kHalf + 32 * (4 + q), 0, unit_id, sm + (4 + q) * kSwBlk);
          } else if (q & 1) {
            const int c = q >> 1;
            tma3_store(&tp.m_out, rank * kHalf + 64 * c, 0, u.b, sm + c * kSwBlk);
            tma3_store(&tp.m_out, rank * kHalf + 64 * (2 + c), 0, u.b, sm + (2 + c) * kSwBlk);
          }
        }
      }
      if (warp == 4 && lane == 0) {
        bulk_commit();
        bulk_wait_read();
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_before();
  __syncthreads();
  cluster_sync();  // neither CTA issues remote stores any more
  if (bars->abort) {
    // The partial scores, P rows and row sums arrive by asynchronous remote
    // stores, which the cluster barrier does not wait for.  On the normal
    // path every one has landed (this CTA waited for each); after an abort
    // some the peer issued may still be in flight into this CTA's shared
    // memory, so it stays alive for a bound far above their delivery time
    // (microseconds).
    if (threadIdx.x == 0) {
      uint64_t t0, t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
      do {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      } while (t - t0 < 100000u);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool encode3(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
             uint64_t S, uint64_t B, uint32_t box0, uint32_t box1, CUtensorMapSwizzle sw) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, S, B};
  cuuint64_t strides[2] = {inner * esize, inner * esize * S};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D map over `rows` rows of `inner` elements, box `box0` x 1 row, no swizzle
bool encode2_rows(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, uint64_t inner,
                  uint64_t rows, uint32_t box0) {
  auto enc = get_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box0, 1};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kFmt, bool kSparse>
void fill_launch(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int grid, cudaStream_t s) {
  using C = Cfg<kFmt, kSparse>;
  *cfg = {};
  cfg->gridDim = dim3(grid);
  cfg->blockDim = dim3(C::kThreads);
  cfg->dynamicSmemBytes = C::kSmem;
  cfg->stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 2;
}

template <int kFmt, bool kSparse>
cudaError_t launch_tc_variant(const TcParams& tp, cudaStream_t s) {
  using C = Cfg<kFmt, kSparse>;
  cudaError_t e = ensure_smem<decode_tc_kernel<kFmt, kSparse>>(C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  fill_launch<kFmt, kSparse>(&cfg, attr, 2 * tp.p.ws.max_units, s);
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<kFmt, kSparse>, tp);
}

// CTA pairs of this variant that can be resident at once on the current
// device (cached per device); 0 if the query fails.
template <int kFmt, bool kSparse>
int resident_pairs() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    using C = Cfg<kFmt, kSparse>;
    int n = 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_launch<kFmt, kSparse>(&cfg, attr, 2, nullptr);
    cfg.numAttrs = 1;   // the cluster shape alone decides residency
    if (ensure_smem<decode_tc_kernel<kFmt, kSparse>>(C::kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<kFmt, kSparse>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev] = n > 0 ? n : -1;
  }
  return cache[dev] > 0 ? cache[dev] : 0;
}

}  // namespace

int decode_tc_granule(int fmt, bool sparse) {
  return fmt == 0 ? (sparse ? Cfg<0, true>::kN : Cfg<0, false>::kN)
                  : (sparse ? Cfg<1, true>::kN : Cfg<1, false>::kN);
}

int decode_tc_units(int fmt, bool sparse, int num_sms) {
  const int n = fmt == 0 ? (sparse ? resident_pairs<0, true>() : resident_pairs<0, false>())
                         : (sparse ? resident_pairs<1, true>() : resident_pairs<1, false>());
  const int half = num_sms / 2;
  return n > 0 && n < half ? n : half;
}

bool decode_tc_supported(int H) { return H == 128 && get_encoder() != nullptr; }

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t s) {
  TcParams tp;
  memset(&tp, 0, sizeof(tp));
  tp.p = p;
  const uint64_t S = (uint64_t)p.max_seq_len, B = (uint64_t)p.B;
  const uint64_t slots = (uint64_t)(p.B / p.mtp_s);   // cache slots the dense maps cover
  const uint32_t n = (uint32_t)decode_tc_granule(p.fmt, p.K > 0);   // tile rows
  bool ok = true;
  if (p.K) {
    // gathers: a 2D map of the latent rows [B * S], one row high, for
    // tile::gather4 (scales and rotary columns go by 16-byte copies)
    const uint64_t rows = B * S;
    ok = encode2_rows(&tp.m_kv, p.fmt == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      p.fmt == 0 ? 2 : 1, p.kv, kDc, rows, kHalf);
  } else {
    if (p.fmt == 0) {
      ok = encode3(&tp.m_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.kv, kDc, S, slots, 64, n,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
      ok = encode3(&tp.m_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.kv, kDc, S, slots, kHalf, n,
                   CU_TENSOR_MAP_SWIZZLE_NONE) &&
           encode3(&tp.m_sc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.kv_scale, kNblk, S, slots, kNblk, n,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    // bf16: straight into the operand layout; FP8: plain half rows (the
    // CTA's 32 columns) for the converter
    ok = ok && encode3(&tp.m_pe, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.pe, kDr, S, slots,
                       p.fmt == 0 ? 64 : kPeHalf, n,
                       p.fmt == 0 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  ok = ok &&
       encode3(&tp.m_ql, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.q_latent, kDc, 128, B, 64, 128,
               CU_TENSOR_MAP_SWIZZLE_128B) &&
       encode3(&tp.m_qp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.q_pe, kDr, 128, B, 64, 128,
               CU_TENSOR_MAP_SWIZZLE_128B) &&
       encode3(&tp.m_po, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.ws.part_o, kDc, 128,
               (uint64_t)p.ws.max_units, 32, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
       encode3(&tp.m_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, kDc, 128, B, 64, 128,
               CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  if (p.fmt == 0) return p.K ? launch_tc_variant<0, true>(tp, s) : launch_tc_variant<0, false>(tp, s);
  return p.K ? launch_tc_variant<1, true>(tp, s) : launch_tc_variant<1, false>(tp, s);
}

}  // namespace mla
