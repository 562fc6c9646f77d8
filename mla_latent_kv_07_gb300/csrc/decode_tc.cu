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
// and rotary columns [32r, 32r+32):
//   * QK: each CTA contracts its 288-wide half (Q half as the A operand held in
//     tensor memory, K half from shared memory) into a partial S; the two
//     partials are exchanged through distributed shared memory as 24-bit
//     codes (each fp32 partial rounded to its top 24 bits; asynchronous
//     remote stores, counted on the receiver's barrier) and added to the
//     receiver's own fp32 partial.  Each CTA runs the softmax on its sum and
//     keeps its own reference maximum and row sums for its output half.
//   * PV: each CTA multiplies P (shared memory) by its latent half V (the same
//     shared-memory tile, read as an MN-major operand) into its own O half.
// Every cache byte is fetched by exactly one CTA and there is no redundant
// tensor-core work.
//
// Tensor memory (512 columns): O half [0,256) fp32; Q half [256,400) bf16 (2
// per column); S double buffer [400,448) and [448,496) fp32.
//
// Warp roles (512 threads; 672 with a converter, 640 for gathers):
//   warp 0  producer: TMA tiles (dense) or four-row TMA gathers (gather)
//   warp 1  MMA issuer (one thread; of QK only in the dense variants) and
//           tensor-memory owner
//   dense variants: PV issuer (one thread), warp 2 (bf16) or warp 20 (FP8);
//           in a dense bf16 call warp 2 first works out the split schedule
//           and the pair's unit (schedule.cuh)
//   warps 4-7 and 12-15 (16-19 with a converter)  softmax: two threads per
//              head h <-> TMEM lane h, each half of the tile's positions;
//              online softmax (lazy rescale), P, epilogue
//   warps 8-11 exchange: partial S of each tile from TMEM -> peer (DSMEM),
//              as soon as it is computed.  (A dense call with new rows: in
//              the unit that reads the new row they first write it to the
//              cache -- the cache-write step -- before the producer loads
//              the unit's last tile.)  Distributed shared memory moves
//              ~20-35 GB/s per SM with ~0.3 us latency on this part (its
//              delivery is on the tile's critical path), so sending runs as
//              its own pipeline stage, ahead of the softmax; the softmax adds
//              the peer's partial when it reads its own.
//   warps 2-3 and 12-15 converter (FP8 caches and gathers): raw rows -> bf16
//              operand tile bf16(fp32(e4m3 * scale)) in the 128-byte
//              swizzled layout
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
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales
constexpr uint32_t kTmemO = 0, kTmemQ = 256, kTmemS = 400;
constexpr long kSpinLimit = 1L << 26;   // polls (~seconds) before giving up
constexpr int kConvWarps = 6;             // converter: warps 2-3 and 12-15

// Shared-memory plan per variant.  Tiles are 48 positions (MMA N for QK, K
// for PV), with two S, P and exchange buffers.  An operand stage holds the
// swizzled bf16 latent half and rotary tile the MMAs read; it is taken from
// the load (dense bf16) or the conversion (FP8, gathers) of its tile until
// PV of that tile completes.  Variants with a converter load the rows as
// stored -- FP8 codes or gathered bf16 half rows, the 4 FP8 scales of each
// row, the 64 rotary values -- into a separate ring of raw slots, which the
// converter frees as soon as it has read them.  So a load never waits for a
// PV, and the HBM latency stays out of the operand stages' cycle.
template <int kFmt, bool kSparse>
struct Cfg {
  static constexpr bool kConv = kFmt == 1 || kSparse;       // converter warps present
  static constexpr int kN = 48;    // positions per tile
  static constexpr int kSBufs = 2;  // S buffers (tensor memory)
  // P buffers (shared memory): three where there is room (bf16), so the
  // softmax writes P of tile i once PV of tile i-3 is done -- PV of tile i-2
  // runs behind the QK of tile i in the in-order tensor pipe
  static constexpr int kPBufs = kFmt == 0 ? 3 : 2;
  // exchange buffers: two, except with FP8 caches, whose fourth operand stage
  // takes the room of the second (the softmax reads a tile's exchange buffer
  // well before the peer's partial of the next tile is due)
  static constexpr int kXBufs = kFmt == 1 ? 1 : 2;
  // warps: 0 producer, 1 MMA, 4-7 softmax (first half), 8-11 exchange,
  // 12-15 converter (if any), then 4 warps of the softmax's second half
  static constexpr int kHiWarp = kConv ? 16 : 12;
  // QK may be issued at most this many tiles past the last issued PV: enough
  // run-ahead to keep the tensor pipe busy through the exchange and softmax
  // of a tile, no more -- the pipe runs its queue in order, so each queued QK
  // delays the PV behind it (measured: 2 starves the pipe, 3 is best).
  static constexpr int kQkAhead = 3;
  // Dense variants issue PV from a thread of its own (warp 2, idle without a
  // converter; with one, a warp of its own after the softmax's second half),
  // so a PV whose P is ready never waits behind the issue of a QK (which
  // blocks on the tensor pipe's queue for about as long as it runs).  The
  // gather variants keep one issuer: the extra warp costs them registers.
  static constexpr bool kSplitIssue = !kSparse;
  static constexpr int kPvWarp = kConv ? kHiWarp + 4 : 2;
  static constexpr int kThreads = 32 * (kHiWarp + 4 + (kConv && kSplitIssue ? 1 : 0));
  static constexpr int kBlkBytes = kN * 128;       // one 64-column swizzled block of a tile
  static constexpr int kOplBytes = 4 * kBlkBytes;  // latent half operand
  static constexpr int kOpeBytes = kBlkBytes;      // rotary operand (full 64 columns)
  static constexpr int kPBytes = ((kN + 63) / 64) * kSwBlk;  // P: 128 heads x kN bf16, swizzled
  // exchange buffer: a head's kN partial scores as 24-bit codes (the fp32
  // value rounded to its top 24 bits), four positions in three words, so
  // 3 kN / 4 words = kXRows 16-byte rows per head; row q of head h at index
  // q * 128 + h, so a warp's remote store is one contiguous 512-byte run
  static constexpr int kXRows = 3 * kN / 16;
  static constexpr int kXBytes = kXRows * 128 * 16;
  static constexpr int kStage = kOplBytes + kOpeBytes;
  static constexpr int kStages = kConv ? (kFmt == 1 ? 4 : 2) : 4;
  static constexpr int kRawRow = kFmt == 1 ? kHalf : kHalf * 2;  // bytes of a raw latent half row
  // FP8 scales, 16 B per row: dense tiles land as 48 consecutive rows; a
  // gather lands 4 rows per 128-byte slot (a tensor copy's shared-memory
  // destination is 128-byte aligned)
  static constexpr int kScBytes = kFmt == 1 ? (kSparse ? 2048 : 1024) : 0;
  // rotary bytes per raw row: dense FP8 loads only the CTA's 32 columns (the
  // 32 its QK reads); gathers land whole 128-byte rows
  static constexpr int kRawPe = (kFmt == 1 && !kSparse) ? kPeHalf * 2 : 128;
  static constexpr int kRaw = kConv ? kN * kRawRow + kScBytes + kN * kRawPe : 0;
  static constexpr int kRawSlots = kConv ? (kFmt == 1 && !kSparse ? 3 : 2) : 0;
  // the converter's ring length in index arithmetic (never zero, so the
  // converter code of the variants without one compiles cleanly)
  static constexpr int kRawRing = kRawSlots > 0 ? kRawSlots : 1;
  static constexpr int kRawOff = kStages * kStage;
  static constexpr int kPOff = kRawOff + kRawSlots * kRaw;
  static constexpr int kXOff = kPOff + kPBufs * kPBytes;
  static constexpr int kBarOff = kXOff + kXBufs * kXBytes;
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
                          : kPBufs * kPBytes + kXBufs * kXBytes >= 5 * kSwBlk,
                "query staging fits");
  static_assert(kQOff % 1024 == 0 && kPOff % 1024 == 0, "1 KB alignment of the query staging");
  static_assert(kBarOff >= 8 * kSwBlk, "output staging fits the idle buffers");
};

struct TcParams {
  DecodeParams p;
  CUtensorMap m_kv;   // bf16: latent (box 64 x N), FP8: codes (box 256 x N)
  CUtensorMap m_pe;   // rotary (box 64 x N, 128-byte swizzle)
  CUtensorMap m_sc;   // FP8 scales (box 4 x N)
  CUtensorMap m_ql;   // q_latent [B][128][512] (box 64 x 128, 128-byte swizzle)
  CUtensorMap m_qp;   // q_pe [B][128][64] (box 64 x 128, 128-byte swizzle)
  CUtensorMap m_po;   // partial outputs [units][128][512] fp32 (box 32 x 128, 128-byte swizzle)
  CUtensorMap m_out;  // final output [B][128][512] bf16 (box 64 x 128, 128-byte swizzle)
};

// named barrier 1 among the 256 softmax threads; barriers 2..5 between the
// two softmax warps that serve the same 32 heads
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void pair_sync(int q) {
  asm volatile("bar.sync %0, 64;" ::"r"(2 + q) : "memory");
}
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
  uint64_t rfree[3];   // raw slot read by the converter
  uint64_t sfull[2], sfree[2], pfull[3], pfree[3], xfull[2], xempty[2];
  uint64_t drain;   // final commit of the MMA issuer (of QK, when PV has its own)
  uint64_t drain_pv;  // final commit of the PV issuer
  volatile int pv_issued;   // PV issuer: tiles whose PV is issued (paces QK)
  uint64_t qbar;    // query rows staged in shared memory
  uint64_t qready;  // query half in tensor memory
  uint64_t appended;  // the new row is in the cache (dense call with new rows)
  Unit unit;          // this pair's unit, when the kernel computes the schedule
  uint32_t tmem;
  volatile int abort;
  float pair_max[2][256];   // softmax: tile maxima of the pair's halves, by tile parity
  float l_half[256];        // epilogue: the pair's halves of l
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

  auto opl = [&](int j) { return sm + j * C::kStage; };               // operand stage j
  auto ope = [&](int j) { return sm + j * C::kStage + kOplBytes; };
  auto raw = [&](int r) { return sm + C::kRawOff + r * C::kRaw; };    // raw slot r
  auto rsc = [&](int r) { return raw(r) + kN * C::kRawRow; };
  auto rpe = [&](int r) { return raw(r) + kN * C::kRawRow + C::kScBytes; };
  auto pbuf = [&](int b) { return sm + C::kPOff + b * C::kPBytes; };
  auto xbuf = [&](int b) { return reinterpret_cast<float*>(sm + C::kXOff + b * C::kXBytes); };
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
      bar_init(&bars->full[j], 1);
      bar_init(&bars->deq[j], kConvWarps);
      bar_init(&bars->empty[j], 1);
    }
    for (int r = 0; r < C::kRawSlots; ++r) bar_init(&bars->rfree[r], kConvWarps);
    for (int b = 0; b < C::kPBufs; ++b) {
      bar_init(&bars->pfull[b], 8);
      bar_init(&bars->pfree[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      bar_init(&bars->sfull[b], 1);
      bar_init(&bars->sfree[b], 12);   // softmax (8) and exchange (4) warps read S
      bar_init(&bars->xfull[b], 1);    // one arrival (with the tile's bytes) from the peer
      bar_init(&bars->xempty[b], 8);   // the peer's softmax warps
    }
    bar_init(&bars->drain, 1);
    bar_init(&bars->drain_pv, 1);
    bars->pv_issued = 0;
    bar_init(&bars->qbar, 1);
    bar_init(&bars->qready, 4);
    bar_init(&bars->appended, 4);   // the exchange warps
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
    // only the dense bf16 variant computes its schedule (the FP8 variant runs
    // at its register limit, where this code cost more than it saved)
    if constexpr (kSparse || kFmt != 0) {
      return p.ws.units[unit_id];
    } else {
      if (p.sched.end_pos == nullptr) return p.ws.units[unit_id];
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
  // rotary columns, 128-byte swizzled) in the P and exchange buffers, which
  // are idle until the first tile, so the producer starts on the cache at
  // once.  Each thread then moves its row to its TMEM lane and signals the MMA
  // issuer, and the peer that its exchange buffers may be written.
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
    if (lane == 0) {
      bar_arrive(&bars->qready);
      // phase 0 of the peer's xempty[0/1]: this CTA's exchange buffers are free
      bar_arrive_remote(mapa(&bars->xempty[0], peer));
      bar_arrive_remote(mapa(&bars->xempty[1], peer));
    }
  }
  // the second-half softmax warps count towards that phase too (it completes
  // only with the first half's arrivals, after the staged rows were read)
  if (live && warp >= C::kHiWarp && warp < C::kHiWarp + 4 && lane == 0) {
    bar_arrive_remote(mapa(&bars->xempty[0], peer));
    bar_arrive_remote(mapa(&bars->xempty[1], peer));
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
      if (!wt.wait(C::kConv ? &bars->rfree[j] : &bars->empty[j], (use & 1) ^ 1)) break;
      const int e0 = u.t0 + i * kN;
      const int slot = u.b / p.mtp_s;   // cache slot of the sequence (several per slot: multi-token)
      if (unit_id == 0 && i == p.withhold_tile) {
        // self-test: this tile's load is never issued, so the waits on it run
        // out (the drain below skips it)
        continue;
      }
      // the tile that holds the new row: its writers fenced their stores
      // for the tensor copies before arriving
      if (app && i == ntiles - 1 && !wt.wait(&bars->appended, 0)) break;
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
        // gathered rows, four per TMA instruction (tile::gather4 on row-high
        // boxes): lane g takes rows 4g..4g+3 of the tile -- its latent half,
        // the FP8 scales, the rotary row -- each landing 128-byte aligned.  A
        // short last group repeats its last row; the converter ignores rows
        // past the unit.
        const int v = min(kN, u.t1 - e0);
        const int groups = (v + 3) / 4;
        constexpr uint32_t kGroupBytes = 4 * (C::kRawRow + (kFmt == 1 ? 16 : 0) + 128);
        if (lane == 0) bar_expect_tx(&bars->full[j], (uint32_t)groups * kGroupBytes);
        __syncwarp();
        if (lane < groups) {
          const int* gl = p.ws.gidx + (size_t)u.b * p.K + e0;
          const int base = u.b * p.max_seq_len, c = 4 * lane;
          int r[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) r[k] = base + gl[min(c + k, v - 1)];
          tma_gather4(raw(j) + c * C::kRawRow, &tp.m_kv, rank * kHalf, r[0], r[1], r[2], r[3],
                      &bars->full[j]);
          if (kFmt == 1)
            tma_gather4(rsc(j) + lane * 128, &tp.m_sc, 0, r[0], r[1], r[2], r[3], &bars->full[j]);
          tma_gather4(rpe(j) + c * 128, &tp.m_pe, 0, r[0], r[1], r[2], r[3], &bars->full[j]);
        }
      }
      issued = i + 1;
    }
    // copies still in flight must land before this CTA's shared memory goes
    // away; on the normal path every stage was already consumed
    if (lane == 0 && bars->abort) {
      for (int i = issued > kSlots ? issued - kSlots : 0; i < issued; ++i)
        if (!(unit_id == 0 && i == p.withhold_tile)) wt.drain(&bars->full[i % kSlots], (i / kSlots) & 1);
    }
  } else if (C::kSplitIssue && warp == C::kPvWarp) {
    // ------------------------------------------------------------ PV issuer
    if (lane == 0) {
      constexpr uint32_t id_pv = idesc(128, kHalf, true);
      const uint64_t d_v0 = sdesc(sa(opl(0)), kBlkBytes, 1024);
      const uint64_t d_p0 = sdesc(sa(pbuf(0)), 16, 1024);
      const uint32_t t_o = tmem + kTmemO;
      for (int i = 0; i < ntiles; ++i) {
        const int j = i % C::kStages, b = psel(i);
        if (!wt.wait(&bars->pfull[b], ppar(i))) break;
        tc_after();
        const uint64_t pd = sdesc_at(d_p0, b * C::kPBytes), vd = sdesc_at(d_v0, j * C::kStage);
        if (i == 0)
          mma_ss_c<false>(t_o, pd, vd, id_pv);
        else
          mma_ss_c<true>(t_o, pd, vd, id_pv);
#pragma unroll
        for (int kk = 1; kk < kN / 16; ++kk)
          mma_ss_c<true>(t_o, sdesc_at(pd, (kk >> 2) * kSwBlk + (kk & 3) * 32), sdesc_at(vd, 2048 * kk), id_pv);
        mma_commit(&bars->pfree[b]);
        mma_commit(&bars->empty[j]);
        bars->pv_issued = i + 1;
      }
      mma_commit(&bars->drain_pv);
      wt.drain(&bars->drain_pv, 0);
    }
  } else if (C::kSplitIssue && warp == 1) {
    // ------------------------------------------------------------ QK issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc(128, kN, false);
      const uint64_t d_k0 = sdesc(sa(opl(0)), 16, 1024);
      const uint32_t t_q = tmem + kTmemQ;
      if (live && wt.wait(&bars->qready, 0)) tc_after();
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
        if (!wt.wait(C::kConv ? &bars->deq[j] : &bars->full[j], (k / C::kStages) & 1)) break;
        if (!wt.wait(&bars->sfree[b], spar(k) ^ 1)) break;
        tc_after();
        const uint32_t sd = tmem + kTmemS + b * kN;
        const uint64_t kd = sdesc_at(d_k0, j * C::kStage);
        const uint64_t ped = sdesc_at(kd, kOplBytes + rank * (kPeHalf * 2));
        mma_ts_c<false>(sd, t_q, kd, id_qk);
#pragma unroll
        for (int kk = 1; kk < kHalf / 16; ++kk)
          mma_ts_c<true>(sd, t_q + 8 * kk, sdesc_at(kd, (kk >> 2) * kBlkBytes + (kk & 3) * 32), id_qk);
#pragma unroll
        for (int kk = 0; kk < kPeHalf / 16; ++kk)
          mma_ts_c<true>(sd, t_q + kHalf / 2 + 8 * kk, sdesc_at(ped, 32 * kk), id_qk);
        mma_commit(&bars->sfull[b]);
      }
      mma_commit(&bars->drain);
      wt.drain(&bars->drain, 0);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    // Event-driven: QK of the next tile is issued as soon as its stage, its
    // converted operand and its S buffer are ready (at most kSBufs tiles ahead
    // of the softmax); PV of the next tile as soon as its P is written.
    // Neither waits behind the other's inputs.
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc(128, kN, false);
      constexpr uint32_t id_pv = idesc(128, kHalf, true);
      // descriptors of stage 0 and P buffer 0; a tile's are these plus
      // constant offsets (one add per MMA on this thread)
      const uint64_t d_k0 = sdesc(sa(opl(0)), 16, 1024);          // K-major operand tiles
      const uint64_t d_v0 = sdesc(sa(opl(0)), kBlkBytes, 1024);   // the latent tile read MN-major (V)
      const uint64_t d_p0 = sdesc(sa(pbuf(0)), 16, 1024);
      const uint32_t t_q = tmem + kTmemQ, t_o = tmem + kTmemO;
      int nq = 0, np = 0;
      long idle = 0;
      if (live && wt.wait(&bars->qready, 0)) tc_after();
      while (np < ntiles && !bars->abort) {
        bool did = false;
        // PV first: it is on the critical path (the softmax waits for it), and
        // issuing the 18 QK instructions takes about as long as running them
        if (np < nq) {
          const int i = np, j = i % C::kStages, b = psel(i);
          if (bar_try(&bars->pfull[b], ppar(i))) {
            tc_after();
            const uint64_t pd = sdesc_at(d_p0, b * C::kPBytes), vd = sdesc_at(d_v0, j * C::kStage);
            if (i == 0)
              mma_ss_c<false>(t_o, pd, vd, id_pv);
            else
              mma_ss_c<true>(t_o, pd, vd, id_pv);
#pragma unroll
            for (int kk = 1; kk < kN / 16; ++kk)
              mma_ss_c<true>(t_o, sdesc_at(pd, (kk >> 2) * kSwBlk + (kk & 3) * 32), sdesc_at(vd, 2048 * kk),
                             id_pv);
            mma_commit(&bars->pfree[b]);
            mma_commit(&bars->empty[j]);
            ++np;
            did = true;
          }
        }
        if (nq < ntiles && nq < np + C::kQkAhead) {
          const int k = nq, j = k % C::kStages, b = ssel(k);
          const uint32_t use = k / C::kStages;
          if (bar_try(C::kConv ? &bars->deq[j] : &bars->full[j], use & 1) &&
              bar_try(&bars->sfree[b], spar(k) ^ 1)) {
            tc_after();
            const uint32_t sd = tmem + kTmemS + b * kN;
            const uint64_t kd = sdesc_at(d_k0, j * C::kStage);
            const uint64_t ped = sdesc_at(kd, kOplBytes + rank * (kPeHalf * 2));
            mma_ts_c<false>(sd, t_q, kd, id_qk);
#pragma unroll
            for (int kk = 1; kk < kHalf / 16; ++kk)
              mma_ts_c<true>(sd, t_q + 8 * kk, sdesc_at(kd, (kk >> 2) * kBlkBytes + (kk & 3) * 32), id_qk);
#pragma unroll
            for (int kk = 0; kk < kPeHalf / 16; ++kk)
              mma_ts_c<true>(sd, t_q + kHalf / 2 + 8 * kk, sdesc_at(ped, 32 * kk), id_qk);
            mma_commit(&bars->sfull[b]);
            ++nq;
            did = true;
          }
        }
        if (did) {
          idle = 0;
        } else if (++idle > wt.lim) {
          bars->abort = 1;
          atomicOr(p.ws.status, kDevTimeout);
        }
      }
      // every MMA issued by this thread completes before tensor memory is freed
      mma_commit(&bars->drain);
      wt.drain(&bars->drain, 0);
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ exchange
    // Send only: partial S of tile i -> the peer's exchange buffer (a warp
    // writes 512 contiguous bytes per store), after releasing the S buffer.
    const int h = threadIdx.x - 256;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    if (app) {   // idle until the first scores: write the new row first
      append_row(p.ap, u.b, u.t1 - 1, h);
      fence_async_global();
      __syncwarp();
      if (lane == 0) bar_arrive(&bars->appended);
    }
    for (int i = 0; i < ntiles; ++i) {
      const int b = ssel(i);
      if (!wt.wait(&bars->sfull[b], spar(i))) break;
      tc_after();
      const uint32_t sb = lane_base + kTmemS + b * kN;
      uint32_t r[kN];
#pragma unroll
      for (int c = 0; c < kN / 16; ++c) TC_LD16(sb + 16 * c, (r + 16 * c));
      tc_wait_ld();
      tc_before();
      __syncwarp();
      if (lane == 0) bar_arrive(&bars->sfree[b]);
      const int xb = xsel(i);
      if (!wt.wait(&bars->xempty[xb], xpar(i))) break;   // phase 0: the peer's query staging is done
      const uint32_t xd = mapa(xbuf(xb) + 4 * h, peer), xf = mapa(&bars->xfull[xb], peer);
      uint32_t w[C::kXRows * 4];
#pragma unroll
      for (int g = 0; g < kN / 4; ++g)
        pack24(r[4 * g], r[4 * g + 1], r[4 * g + 2], r[4 * g + 3], w[3 * g], w[3 * g + 1], w[3 * g + 2]);
      // the peer's phase completes on one arrival carrying the tile's bytes
      // and on those bytes landing, in either order
      if (h == 0) bar_arrive_expect_tx_remote(xf, C::kXBytes);
#pragma unroll
      for (int q = 0; q < C::kXRows; ++q)
        st_async_v4(xd + 16 * 128 * q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3], xf);
    }
  } else if ((warp >= 4 && warp < 8) || (warp >= C::kHiWarp && warp < C::kHiWarp + 4)) {
    // ------------------------------------------------------------ softmax
    // Two threads per head h (TMEM lane h): half sh = 0 takes the tile's
    // positions [0,16) and [32,40), half 1 [16,32) and [40,48) (16- and
    // 8-column TMEM loads).  The pair agrees on each tile's maximum through
    // shared memory and a 64-thread barrier, so both take the same rescale
    // decisions; each rescales and, at the end, normalises half of the O row.
    const int sh = warp >= 8 ? 1 : 0;
    const int h = 32 * (warp & 3) + lane;
    const int p0 = 16 * sh, p1 = 32 + 8 * sh;   // first position of each run
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 > 0.f;
    const float ps = pos_scale ? sl2 : 1.f;   // the factor still to apply to sc in P
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int j = i % C::kStages, sb_i = ssel(i), b = psel(i);
      const uint32_t par = ppar(i);
      float sc[24];
      ok = ok && wt.wait(&bars->sfull[sb_i], spar(i));
      {
        tc_after();
        const uint32_t sb = lane_base + kTmemS + sb_i * kN;
        uint32_t r[24];
        TC_LD16(sb + p0, r);
        TC_LD8(sb + p1, (r + 16));
        tc_wait_ld();
#pragma unroll
        for (int k = 0; k < 24; ++k) sc[k] = __uint_as_float(r[k]);
        tc_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&bars->sfree[sb_i]);   // QK of tile i + kSBufs may overwrite
      }
      // + the peer's partial (rounded to 24 bits).  This half's positions p0..p0+15 are code
      // words 12 sh .. 12 sh + 11 (rows 3 sh .. 3 sh + 2), p1..p1+7 words
      // 24 + 6 sh .. 24 + 6 sh + 5 (within rows 6 + sh, 7 + sh).
      const int xb = xsel(i);
      ok = ok && wt.wait(&bars->xfull[xb], xpar(i));
      {
        const uint4* xr = reinterpret_cast<const uint4*>(xbuf(xb)) + h;
        uint32_t w[20];
#pragma unroll
        for (int q = 0; q < 5; ++q) {
          const uint4 v = xr[128 * (q < 3 ? 3 * sh + q : 6 + sh + q - 3)];
          w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int k = 0; k < 6; ++k) {
          float4 v;
          if (k < 4) {
            v = unpack24(w[3 * k], w[3 * k + 1], w[3 * k + 2]);
          } else {
            const int t = 3 * (k - 4);
            v = unpack24(sh ? w[14 + t] : w[12 + t], sh ? w[15 + t] : w[13 + t], sh ? w[16 + t] : w[14 + t]);
          }
          const float2 a = __fadd2_rn(make_float2(sc[4 * k], sc[4 * k + 1]), make_float2(v.x, v.y));
          const float2 c2 = __fadd2_rn(make_float2(sc[4 * k + 2], sc[4 * k + 3]), make_float2(v.z, v.w));
          sc[4 * k] = a.x; sc[4 * k + 1] = a.y; sc[4 * k + 2] = c2.x; sc[4 * k + 3] = c2.y;
        }
        __syncwarp();
        // my buffer b may be refilled: the values read above are already in
        // registers, so no release ordering is needed
        if (lane == 0) bar_arrive_remote_relaxed(mapa(&bars->xempty[xb], peer));
      }
      // masked scores and the tile maximum of the pair.  With a positive
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
          if ((k < 16 ? p0 + k : p1 + k - 16) >= valid) sc[k] = -INFINITY;
      }
      float mx[4] = {sc[0], sc[1], sc[2], sc[3]};
#pragma unroll
      for (int k = 4; k < 24; ++k) mx[k & 3] = fmaxf(mx[k & 3], sc[k]);
      float* pm = bars->pair_max[i & 1];
      const float mloc = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      pm[sh * 128 + h] = pos_scale ? mloc * sl2 : mloc;
      pair_sync(warp & 3);
      const float mt = fmaxf(pm[h], pm[128 + h]);
      // lazy rescale of the running reference max
      const bool need = ok && mt > m_ref + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mt : m_ref;
        const float alpha = exp2f(m_ref - m_new);   // 0 when m_ref = -inf
        if (i > 0) {
          // O holds tiles < i: wait for PV of tile i-1 (its P buffer's release;
          // the previous use of that buffer is known complete, so the parity
          // wait cannot be fooled by a phase two steps back), then scale this
          // thread's half of the lane's row
          ok = ok && wt.wait(&bars->pfree[psel(i - 1)], ppar(i - 1));
          tc_after();
#pragma unroll 1
          for (int c = 4 * sh; c < 4 * sh + 4; ++c) {
            uint32_t r[16], q[16];
            TC_LD16(lane_base + kTmemO + 32 * c, r);
            TC_LD16(lane_base + kTmemO + 32 * c + 16, q);
            tc_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
              q[k] = __float_as_uint(__uint_as_float(q[k]) * alpha);
            }
            TC_ST16(lane_base + kTmemO + 32 * c, r);
            TC_ST16(lane_base + kTmemO + 32 * c + 16, q);
          }
          tc_wait_st();
        }
        l *= alpha;
        m_ref = m_new;
      }
      // this half of head h's P row (bf16), in the 16-byte chunks p0/8,
      // p0/8 + 1 and p1/8; l sums the fp32 values before their rounding
      ok = ok && wt.wait(&bars->pfree[b], par ^ 1);
      uint8_t* prow = pbuf(b);
      float2 ls = make_float2(0.f, 0.f);
      const float2 ps2 = make_float2(ps, ps), nm2 = make_float2(-m_ref, -m_ref);
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        uint32_t pk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 t = __ffma2_rn(make_float2(sc[8 * c + 2 * k], sc[8 * c + 2 * k + 1]), ps2, nm2);
          const float2 e = make_float2(ex2_approx(t.x), ex2_approx(t.y));
          const __nv_bfloat162 two = __float22bfloat162_rn(e);
          ls = __fadd2_rn(ls, e);
          pk[k] = *reinterpret_cast<const uint32_t*>(&two);
        }
        const int chunk = c < 2 ? p0 / 8 + c : p1 / 8;
        *reinterpret_cast<uint4*>(prow + (chunk >> 3) * kSwBlk + swz_chunk(h, chunk & 7)) =
            make_uint4(pk[0], pk[1], pk[2], pk[3]);
      }
      l += ls.x + ls.y;
      if (!C::kConv && valid < kN) {
        // dense bf16 tail: rows past the unit hold whatever the cache holds
        // there; zero them so P = 0 never meets a non-finite value
        uint8_t* v = opl(j);
        for (int idx = sh * 128 + h; idx < (kN - valid) * 32; idx += 256) {
          const int row = valid + idx / 32, blk = (idx / 8) & 3, ch = idx & 7;
          *reinterpret_cast<uint4*>(v + blk * kBlkBytes + swz_chunk(row, ch)) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_async_smem();
      tc_before();
      __syncwarp();
      if (lane == 0) bar_arrive(&bars->pfull[b]);
    }
    // ------------------------------------------------------------ epilogue
    if (live) {
      if (ntiles > 0) ok = ok && wt.wait(&bars->pfree[psel(ntiles - 1)], ppar(ntiles - 1));
      tc_after();
      // O half (128 heads x 256 fp32) -> workspace, normalised by the head's
      // l (the sum of the pair's halves).  With the last PV complete, every
      // stage, P and exchange buffer is idle (the peer sent its last partial
      // before this CTA's last softmax step), so the half is staged as 8
      // swizzled blocks of 32 columns, in four rounds of one block per thread
      // of the pair: the TMA stores of the blocks a round completes leave
      // while the next round is staged.
      // A sequence's only unit writes the final bf16 output (4 blocks of 64
      // columns: two 32-column chunks each, complete after rounds 1 and 3)
      // and log-sum-exp itself.
      bars->l_half[sh * 128 + h] = l;
      softmax_sync();
      const float lt = bars->l_half[h] + bars->l_half[128 + h];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const bool direct = (u.flags & kUnitDirect) != 0;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        if (direct)
          stage_output_bf16(lane_base, sm, h, inv, 4 * sh + q, 4 * sh + q + 1);
        else
          stage_output(lane_base, sm, h, inv, 4 * sh + q, 4 * sh + q + 1);
        fence_async_smem();
        softmax_sync();
        if (sh == 0 && h == 0) {
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
      if (sh == 0 && h == 0) bulk_commit();
      if (rank == 0 && sh == 0) {
        const float lse = (ok && lt > 0.f) ? (m_ref + log2f(lt)) * 0.69314718055994531f : -INFINITY;
        if (!(u.flags & kUnitDirect))
          p.ws.part_lse[(size_t)unit_id * p.H + h] = lse;
        else if (p.lse)
          p.lse[(size_t)u.b * p.H + h] = lse;
      }
      if (sh == 0 && h == 0) bulk_wait_read();
    }
  } else if (C::kConv && (warp == 2 || warp == 3 || (warp >= 12 && warp < 16))) {
    // ------------------------------------------------------------ converter
    // raw slot r of tile i -> operand stage j, once the rows have landed and
    // PV of the stage's previous tile is done; kConvWarps warps share a tile
    const int t = warp < 4 ? threadIdx.x - 64 : threadIdx.x - 384 + 64;
    for (int i = 0; i < ntiles; ++i) {
      const int r = i % C::kRawRing, j = i % C::kStages;
      // FP8: stages 1-3 hold the staged query until it is in tensor memory
      if (kFmt == 1 && i == 1 && !wt.wait(&bars->qready, 0)) break;
      if (!wt.wait(&bars->full[r], (i / C::kRawRing) & 1)) break;
      if (!wt.wait(&bars->empty[j], ((i / C::kStages) & 1) ^ 1)) break;
      const int valid = min(kN, u.t1 - (u.t0 + i * kN));
      uint8_t* dst = opl(j);
      if (kFmt == 1) {
        // 48 rows x 16 chunks of 16 codes -> 2 swizzled 16-byte chunks each
        for (int idx = t; idx < kN * 16; idx += 32 * kConvWarps) {
          const int row = idx >> 4, q = idx & 15;  // codes [16q, 16q + 16) of the half row
          uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
          if (row < valid) {
            const uint4 v = *reinterpret_cast<const uint4*>(raw(r) + row * kHalf + q * 16);
            const uint8_t* srow = rsc(r) + (kSparse ? (row >> 2) * 128 + (row & 3) * 16 : row * 16);
            const float sc = reinterpret_cast<const float*>(srow)[rank * 2 + (q >> 3)];
            dequant16(v, sc, lo, hi);
          }
          const int blk = q >> 2, ch = (q & 3) * 2;
          *reinterpret_cast<uint4*>(dst + blk * kBlkBytes + swz_chunk(row, ch)) = lo;
          *reinterpret_cast<uint4*>(dst + blk * kBlkBytes + swz_chunk(row, ch + 1)) = hi;
        }
      } else {
        // gathered bf16 rows: 48 rows x 32 chunks of 8 values
        for (int idx = t; idx < kN * 32; idx += 32 * kConvWarps) {
          const int row = idx >> 5, q = idx & 31;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < valid) v = *reinterpret_cast<const uint4*>(raw(r) + row * C::kRawRow + q * 16);
          *reinterpret_cast<uint4*>(dst + (q >> 3) * kBlkBytes + swz_chunk(row, q & 7)) = v;
        }
      }
      // rotary rows -> swizzled operand (with half rows, the CTA's 16-byte
      // chunks 4 rank .. 4 rank + 3 of the 64-column operand row, the only
      // ones its QK reads)
      constexpr int kPeChunks = C::kRawPe / 16;
      const int pe_chunk0 = kPeChunks == 8 ? 0 : 4 * (int)rank;
      for (int idx = t; idx < kN * kPeChunks; idx += 32 * kConvWarps) {
        const int row = idx / kPeChunks, q = idx % kPeChunks;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < valid) v = *reinterpret_cast<const uint4*>(rpe(r) + row * C::kRawPe + q * 16);
        *reinterpret_cast<uint4*>(ope(j) + swz_chunk(row, pe_chunk0 + q)) = v;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        bar_arrive(&bars->deq[j]);
        bar_arrive(&bars->rfree[r]);
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_before();
  __syncthreads();
  cluster_sync();  // neither CTA issues remote stores any more
  if (bars->abort) {
    // The partial scores arrive by asynchronous remote stores, which the
    // cluster barrier does not wait for.  On the normal path every one has
    // landed (this CTA waited for each tile's); after an abort some the peer
    // issued may still be in flight into this CTA's shared memory, so it
    // stays alive for a bound far above their delivery time (microseconds).
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
    // gathers: 2D maps over all rows [B * S], one row high, for tile::gather4
    const uint64_t rows = B * S;
    ok = encode2_rows(&tp.m_kv, p.fmt == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      p.fmt == 0 ? 2 : 1, p.kv, kDc, rows, kHalf) &&
         encode2_rows(&tp.m_pe, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.pe, kDr, rows, kDr) &&
         (p.fmt == 0 || encode2_rows(&tp.m_sc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.kv_scale, kNblk,
                                     rows, kNblk));
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
