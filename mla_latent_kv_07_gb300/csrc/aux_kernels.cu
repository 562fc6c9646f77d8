// aux_kernels.cu -- the small kernels around the decode:
//   append   cache-write step with FP8 block quantisation
//            ("DeepSeek-V3.2-Exp . KV cache", cache-write excerpt)
//   prep     top-k list -> sorted, de-duplicated, valid gather list (a bitmap
//            of the sequence's positions)
//            (same page, MQA-decode excerpt: the index mask is a scatter of
//            zeros into -inf, so repeats act once and order does not matter)
//   schedule split every sequence's positions into units of about equal size
//   combine  log-sum-exp merge of the per-unit partial outputs
//   select   top-k positions per sequence from per-position scores (the
//            index lists the sparse decode takes)
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cuda.h>

#include "append_row.cuh"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using ptx::cluster_sync;
using ptx::mapa;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- append
// One CTA (4 warps) per row, positions from the host (checked there).
__global__ void __launch_bounds__(128) append_kernel(const AppendParams p) {
  pdl_wait();   // earlier kernels may still read the cache rows written here
  pdl_trigger();
  append_row(p.rows, blockIdx.x, p.pos[blockIdx.x], threadIdx.x);
}

// One CTA per sequence: row end_pos[b] - 1, where the dense decode reads it
// (the warp-MMA decode path; the tensor-memory kernel writes the row itself).
// Rows left out are flagged by the schedule kernel.
__global__ void __launch_bounds__(128) append_end_kernel(const AppendRows ap, const int* __restrict__ end_pos,
                                                         int max_end_pos) {
  pdl_wait();
  pdl_trigger();
  const int end = end_pos[blockIdx.x];
  if (append_row_valid(end, max_end_pos)) append_row(ap, blockIdx.x, end - 1, threadIdx.x);
}

// ------------------------------------------------------------ block scan
// Exclusive prefix sum over the block's threads; returns the block total.
__device__ int block_exclusive_scan(int v, int* smem /* >= 33 ints */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? smem[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nwarps) smem[lane] = w;   // inclusive warp totals
    if (lane == 31) smem[32] = w;
  }
  __syncthreads();
  int excl = x - v + (warp > 0 ? smem[warp - 1] : 0);
  *total = smem[32];
  __syncthreads();
  return excl;
}

// ------------------------------------------------------------ sparse prep
// One CTA per sequence (and, with new rows to write, one more per sequence
// for its row, so the list work does not wait for it).  The positions
// [0, T) are taken in windows of kPrepWindow: every valid list entry in the
// window sets its bit in a shared bitmap (repeats set it once), then each
// thread counts the set bits of its run of words, a block scan turns the
// counts into output offsets, and the set positions are written in
// increasing order.  Invalid entries set nothing; the list's tail is -1.
constexpr int kPrepWindow = 1 << 18;   // positions per pass: a 32 KB bitmap

__global__ void __launch_bounds__(1024) sparse_prep_kernel(const int* __restrict__ topk, int K,
                                                          const int* __restrict__ end_pos,
                                                          int max_end_pos, Workspace ws,
                                                          int* gidx_out, int* gcount_out,
                                                          const AppendRows ap, int B) {
  __shared__ uint32_t bm[kPrepWindow / 32];
  __shared__ int scan_smem[33];
  pdl_wait();   // the previous call's kernels may still read the workspace and the cache
  pdl_trigger();
  // the fused append: CTA B + b writes sequence b's new row, position
  // end_pos[b] - 1 (warps 0-3), beside the list CTAs
  if ((int)blockIdx.x >= B) {
    const int b = blockIdx.x - B, row = end_pos[b] - 1;
    if (row >= 0 && row < ap.max_seq_len && threadIdx.x < 128) append_row(ap, b, row, threadIdx.x);
    return;
  }
  const int b = blockIdx.x;
  const int end = end_pos[b];
  uint32_t flags = 0;
  if (ap.kv_new && (end - 1 < 0 || end - 1 >= ap.max_seq_len)) flags |= kDevAppendSkipped;
  int T = end;
  if (T < 0 || T > max_end_pos) {
    flags |= kDevEndPosClamped;
    T = T < 0 ? 0 : max_end_pos;
  }
  const int* list = topk + (size_t)b * K;
  int* g = ws.gidx + (size_t)b * K;
  int written = 0;
  for (int base = 0; base < T; base += kPrepWindow) {
    const int span = min(kPrepWindow, T - base);
    const int nw = (span + 31) / 32;
    for (int w = threadIdx.x; w < nw; w += blockDim.x) bm[w] = 0u;
    __syncthreads();
    for (int k = threadIdx.x; k < K; k += blockDim.x) {
      const int e = list[k];
      if (e >= base && e - base < span) atomicOr(&bm[(e - base) >> 5], 1u << ((e - base) & 31));
    }
    __syncthreads();
    const int per = (nw + blockDim.x - 1) / blockDim.x;
    const int w0 = threadIdx.x * per;
    int cnt = 0;
    for (int w = w0; w < w0 + per && w < nw; ++w) cnt += __popc(bm[w]);
    int total;
    int dst = written + block_exclusive_scan(cnt, scan_smem, &total);
    for (int w = w0; w < w0 + per && w < nw; ++w) {
      uint32_t bits = bm[w];
      while (bits) {
        const int pos = base + 32 * w + __ffs(bits) - 1;
        bits &= bits - 1u;
        g[dst] = pos;
        if (gidx_out) gidx_out[(size_t)b * K + dst] = pos;
        ++dst;
      }
    }
    written += total;
    __syncthreads();   // the bitmap is cleared for the next window
  }
  for (int k = written + threadIdx.x; k < K; k += blockDim.x) {
    g[k] = -1;
    if (gidx_out) gidx_out[(size_t)b * K + k] = -1;
  }
  if (threadIdx.x == 0) {
    ws.seq_flags[b] = flags;
    ws.lengths[b] = written;
    if (gcount_out) gcount_out[b] = written;
  }
}

// --------------------------------------------------------------- schedule
// Single CTA of 32 x ceil(B / 32) threads (at most 1024).  lengths[b] (dense:
// clamped end_pos; sparse: gather count) is cut into units of `chunk`
// positions, chunk = ceil(total / target) rounded up to the kernel's tile
// granule and grown until sum_b ceil(len_b / chunk) <= target.
__global__ void __launch_bounds__(1024) schedule_kernel(const int* __restrict__ end_pos,
                                                       int max_end_pos, Workspace ws, int B,
                                                       int target, int granule, int direct,
                                                       int mtp_s, int append) {
  __shared__ int scan_smem[33];
  __shared__ unsigned long long total_len;
  __shared__ int count_smem, max_len_smem;
  __shared__ uint32_t flags_smem;
  pdl_wait();   // the previous call's kernels may still read this workspace
  if (threadIdx.x == 0) {
    total_len = 0;
    max_len_smem = 0;
    flags_smem = 0u;
  }
  __syncthreads();
  pdl_trigger();
  const int per = (B + blockDim.x - 1) / blockDim.x;
  const int b0 = threadIdx.x * per;
  unsigned long long mine = 0;
  int longest = 0;
  uint32_t flags = 0;
  for (int b = b0; b < b0 + per && b < B; ++b) {
    int len;
    if (end_pos) {
      len = end_pos[b / mtp_s];
      // a dense call with new rows appends row end_pos - 1 where its decode reads it
      if (append && !append_row_valid(len, max_end_pos)) flags |= kDevAppendSkipped;
      if (len < 0 || len > max_end_pos) {
        flags |= kDevEndPosClamped;
        len = len < 0 ? 0 : max_end_pos;
      }
      len -= mtp_s - 1 - b % mtp_s;   // token j of the step: one position per later token fewer
      if (len < 0) len = 0;
      ws.lengths[b] = len;
    } else {
      len = ws.lengths[b];
      flags |= ws.seq_flags[b];
    }
    mine += (unsigned long long)len;
    longest = len > longest ? len : longest;
  }
  // one shared atomic per warp (a block-wide pile-up on one word serialises)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
    longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
  }
  flags = __reduce_or_sync(0xffffffffu, flags);
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&total_len, mine);
    atomicMax(&max_len_smem, longest);
    if (flags) atomicOr(&flags_smem, flags);
  }
  __syncthreads();
  // a chunk of the longest length gives every non-empty sequence one unit; no
  // larger chunk lowers the count (which may then stay above the target when
  // there are more sequences than units in a wave)
  const long long cap = max_len_smem > granule ? ((long long)max_len_smem + granule - 1) / granule * granule
                                               : (long long)granule;
  // smallest granule multiple with sum_b ceil(len_b / chunk) <= target, so
  // the units fit the launch (and, on the pair path, one wave of the GPU)
  long long chunk = ((long long)total_len + target - 1) / target;
  chunk = ((chunk + granule - 1) / granule) * granule;
  if (chunk < granule) chunk = granule;
  if (chunk > cap) chunk = cap;
  int nmine = 0;
  for (int iter = 0; iter < 64; ++iter) {
    nmine = 0;
    for (int b = b0; b < b0 + per && b < B; ++b)
      nmine += (int)((ws.lengths[b] + chunk - 1) / chunk);
    if (threadIdx.x == 0) count_smem = 0;
    __syncthreads();
    const int wsum = __reduce_add_sync(0xffffffffu, nmine);
    if ((threadIdx.x & 31) == 0) atomicAdd(&count_smem, wsum);
    __syncthreads();
    const int n = count_smem;
    __syncthreads();
    if (n <= target || chunk >= cap) break;
    long long grown = (chunk * n + target - 1) / target;
    grown = ((grown + granule - 1) / granule) * granule;
    chunk = grown > chunk + granule ? grown : chunk + granule;
    if (chunk > cap) chunk = cap;
  }
  int total_units;
  int u = block_exclusive_scan(nmine, scan_smem, &total_units);
  for (int b = b0; b < b0 + per && b < B; ++b) {
    const int len = ws.lengths[b];
    const int n = (int)((len + chunk - 1) / chunk);
    const int one = direct && n == 1;
    // the new row end_pos - 1 lies in the sequence's last unit (t1 = end_pos:
    // a valid end_pos is not clamped)
    const int app = append && end_pos && mtp_s == 1 && append_row_valid(end_pos[b], max_end_pos) ? kUnitAppend : 0;
    ws.seq[b] = make_int2(u, one ? -1 : n);
    for (int i = 0; i < n; ++i) {
      int t0 = (int)(i * chunk);
      int t1 = (int)((i + 1) * chunk < len ? (i + 1) * chunk : len);
      ws.units[u + i] = Unit{b, t0, t1, (one ? kUnitDirect : 0) | (i == n - 1 ? app : 0)};
    }
    u += n;
  }
  for (int i = total_units + threadIdx.x; i < ws.max_units; i += blockDim.x)
    ws.units[i] = Unit{-1, 0, 0, 0};
  if (threadIdx.x == 0) {
    *ws.n_units = total_units;
    *ws.status = flags_smem;   // the call's status word, written afresh
  }
}

// ---------------------------------------------------------------- combine
// CTA (h, y) combines head h of sequences y, y + gridDim.y, ...; 128 threads x
// 4 latent columns.  out = sum_i w_i O_i, w_i = exp(lse_i - lse),
// lse = log sum_i exp(lse_i).  The first warp fetches the descriptors of 32 of
// the CTA's sequences at once, so sequences the decode kernel finished itself
// (a single unit) cost one load between them, not a CTA each.  The partial
// rows are fetched eight units at a time, loads first, so their latencies
// overlap; the first eight are issued before the maximum of the lse values
// (sixteen at a time cost occupancy: slower on most workloads).
__device__ __forceinline__ void combine_one(const Workspace& ws, int H, int h, int b, int2 sq,
                                            __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  const int n = sq.y;
  const int c = threadIdx.x * 4;
  const float* pl = ws.part_lse + (size_t)sq.x * H + h;            // unit stride H
  const float* po = ws.part_o + ((size_t)sq.x * H + h) * kDc + c;  // unit stride H * 512
  const size_t ostride = (size_t)H * kDc;
  // the first kBatch partial rows are in flight while the maximum is formed
  // (the loads do not depend on it)
  constexpr int kBatch = 8;
  float4 o[kBatch];
  float l[kBatch];
#pragma unroll
  for (int k = 0; k < kBatch; ++k) {
    if (k < n) {
      o[k] = *reinterpret_cast<const float4*>(po + (size_t)k * ostride);
      l[k] = pl[(size_t)k * H];
    }
  }
  float m = -INFINITY;
  for (int i = threadIdx.x & 31; i < n; i += 32) m = fmaxf(m, pl[(size_t)i * H]);
  m = warp_max(m);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (m > -INFINITY) {
    for (int i0 = 0; i0 < n; i0 += kBatch) {
      if (i0 > 0) {
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (i0 + k < n) {
            o[k] = *reinterpret_cast<const float4*>(po + (size_t)(i0 + k) * ostride);
            l[k] = pl[(size_t)(i0 + k) * H];
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (i0 + k < n) {
          const float w = expf(l[k] - m);
          acc.x += w * o[k].x; acc.y += w * o[k].y; acc.z += w * o[k].z; acc.w += w * o[k].w;
          wsum += w;
        }
      }
    }
  }
  float lse = -INFINITY;
  if (wsum > 0.f) {
    const float inv = 1.0f / wsum;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    lse = m + logf(wsum);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + ((size_t)b * H + h) * kDc + c) = pk;
  if (lse_out && threadIdx.x == 0) lse_out[(size_t)b * H + h] = lse;
}

__global__ void __launch_bounds__(128) combine_kernel(Workspace ws, int H, int B,
                                                     __nv_bfloat16* __restrict__ out,
                                                     float* __restrict__ lse_out) {
  __shared__ int2 seq_smem[32];
  __shared__ uint32_t live_smem;
  pdl_wait();
  pdl_trigger();
  const int h = blockIdx.x, step = gridDim.y;
  for (int base = blockIdx.y; base < B; base += 32 * step) {
    if (threadIdx.x < 32) {
      const int b = base + threadIdx.x * step;
      const int2 sq = b < B ? ws.seq[b] : make_int2(0, -1);
      seq_smem[threadIdx.x] = sq;
      const uint32_t live = __ballot_sync(0xffffffffu, sq.y >= 0);
      if (threadIdx.x == 0) live_smem = live;
    }
    __syncthreads();
    for (uint32_t live = live_smem; live; live &= live - 1u) {
      const int k = __ffs(live) - 1;
      combine_one(ws, H, h, base + k * step, seq_smem[k], out, lse_out);
    }
    __syncthreads();
  }
}

// ----------------------------------------------------------- read ceiling
// Streams n16 16-byte words (8 loads in flight per thread, streaming cache
// hint) and folds them into one XOR per CTA, so no load is dead code: the
// achievable HBM read rate of this device, for comparison with the decode.
__global__ void __launch_bounds__(512) read_ceiling_kernel(const uint4* __restrict__ buf, size_t n16,
                                                          uint32_t* __restrict__ sink) {
  pdl_wait();
  pdl_trigger();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = i + k * stride < n16 ? __ldcs(buf + i + k * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  // one atomic per CTA: same-address atomics serialise in L2
  __shared__ uint32_t part[16];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t x = 0;
    for (int k = 0; k < (int)(blockDim.x >> 5); ++k) x ^= part[k];
    atomicXor(sink, x);
  }
}


// ----------------------------------------------------------- top-k select
// A cluster of kTopkCtas CTAs per sequence selects, among positions
// 0 .. end_pos-1 of its score row, the K with the largest score (equal
// scores: the lower position; -0 equals +0; NaN ranks lowest) and writes them
// in increasing order, then -1.  Scores map to order-preserving 32-bit keys;
// CTA r of the cluster holds the keys of the r-th of kTopkCtas equal runs of
// positions in shared memory (read once, 16-byte loads when aligned).  A
// radix select over the key's four bytes (most significant first) finds the
// K-th largest key t and how many keys equal to t belong to the selection:
// per pass every CTA builds a 256-bin histogram of its run, and after one
// cluster barrier each CTA sums the kTopkCtas histograms through distributed
// shared memory and takes the same decision (histograms alternate between
// two buffers by pass, so none is cleared while a peer still reads it).  A
// last pass counts, per CTA and per warp, the keys above and equal to t,
// turns the counts into offsets (the peers' through distributed shared
// memory) and writes the selected positions in order.
constexpr int kTopkCtas = 8;
constexpr int kTopkThreads = 512;
constexpr int kTopkSmemKeys = 55296;   // runs up to this many positions are staged (216 KB)

__device__ __forceinline__ uint32_t score_key(float x) {
  if (x != x) return 0u;                             // NaN: below every number
  const uint32_t u = x == 0.f ? 0u : __float_as_uint(x);   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

template <bool kSmem>
__global__ void __launch_bounds__(kTopkThreads, 1) topk_select_kernel(const float* __restrict__ scores,
                                                                     int ld, const int* __restrict__ end_pos,
                                                                     int max_end_pos, int K,
                                                                     int* __restrict__ out) {
  extern __shared__ uint32_t keys_smem[];   // kSmem: this CTA's run of keys
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t ghist[256];
  __shared__ int wgt[kTopkThreads / 32], weq[kTopkThreads / 32];
  __shared__ int cta_cnt[2];   // this CTA's keys above / equal to t (read by the peers)
  __shared__ uint32_t s_prefix;
  __shared__ int s_krem;
  pdl_wait();
  pdl_trigger();
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int b = blockIdx.x / kTopkCtas, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kWarps = kTopkThreads / 32;
  int T = end_pos[b];
  T = T < 0 ? 0 : (T > max_end_pos ? max_end_pos : T);
  const float* row = scores + (size_t)b * ld;
  int* o = out + (size_t)b * K;
  if (T <= K) {   // every valid position is selected (the same test in every CTA of the cluster)
    if (rank == 0)
      for (int k = tid; k < K; k += kTopkThreads) o[k] = k < T ? k : -1;
    return;
  }
  // this CTA's run [c0, c1): a multiple of 4 positions long except the last
  const int per = ((T + kTopkCtas - 1) / kTopkCtas + 3) & ~3;
  const int c0 = min((int)rank * per, T), c1 = min(c0 + per, T), n = c1 - c0;
  if (kSmem) {
    const float* src = row + c0;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      const int n4 = n >> 2;
      const float4* src4 = reinterpret_cast<const float4*>(src);
      for (int q0 = tid; q0 < n4; q0 += 8 * kTopkThreads) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          v[k] = q0 + k * kTopkThreads < n4 ? src4[q0 + k * kTopkThreads] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (q0 + k * kTopkThreads < n4)
            reinterpret_cast<uint4*>(keys_smem)[q0 + k * kTopkThreads] =
                make_uint4(score_key(v[k].x), score_key(v[k].y), score_key(v[k].z), score_key(v[k].w));
      }
      for (int i = 4 * n4 + tid; i < n; i += kTopkThreads) keys_smem[i] = score_key(src[i]);
    } else {
      for (int i = tid; i < n; i += kTopkThreads) keys_smem[i] = score_key(src[i]);
    }
  }
  // key of the run's i-th position
  auto key_at = [&](int i) -> uint32_t { return kSmem ? keys_smem[i] : score_key(row[c0 + i]); };

  uint32_t prefix = 0u, mask = 0u;
  int krem = K;   // selected positions still to place at or below the current prefix
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* h = hist[pass & 1];
    for (int i = tid; i < 256; i += kTopkThreads) h[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kTopkThreads) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&h[(key >> shift) & 255u], 1u);
    }
    cluster_sync();   // every CTA's histogram of this pass is complete
    for (int i = tid; i < 256; i += kTopkThreads) {
      uint32_t sum = 0;
#pragma unroll
      for (int r = 0; r < kTopkCtas; ++r) sum += ld_cluster_u32(mapa(&h[i], r));
      ghist[i] = sum;
    }
    __syncthreads();
    if (tid < 32) {
      // lane l holds bins 255 - 8 l .. 248 - 8 l (largest first)
      uint32_t cnt[8], sum = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        cnt[e] = ghist[255 - 8 * lane - e];
        sum += cnt[e];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o2);
        if (lane >= o2) incl += y;
      }
      const uint32_t before = incl - sum;   // keys in the bins above this lane's
      if (before < (uint32_t)krem && (uint32_t)krem <= incl) {
        uint32_t acc = before;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (acc + cnt[e] >= (uint32_t)krem) {
            s_prefix = prefix | ((uint32_t)(255 - 8 * lane - e) << shift);
            s_krem = krem - (int)acc;
            break;
          }
          acc += cnt[e];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    krem = s_krem;
    mask |= 255u << shift;
  }

  // prefix = the K-th largest key; krem of the keys equal to it are selected.
  // Warp w owns run positions [w R, w R + R), R a multiple of 32.
  const int R = ((n + kWarps - 1) / kWarps + 31) & ~31;
  const int q0 = warp * R, q1 = min(q0 + R, n);
  int ngt = 0, neq = 0;
  for (int i = q0 + lane; i < q1; i += 32) {
    const uint32_t key = key_at(i);
    ngt += key > prefix;
    neq += key == prefix;
  }
  ngt = __reduce_add_sync(0xffffffffu, ngt);
  neq = __reduce_add_sync(0xffffffffu, neq);
  if (lane == 0) {
    wgt[warp] = ngt;
    weq[warp] = neq;
  }
  __syncthreads();
  if (warp == 0) {   // exclusive scans of the warps' counts; this CTA's totals
    const int g = lane < kWarps ? wgt[lane] : 0, e = lane < kWarps ? weq[lane] : 0;
    int gi = g, ei = e;
#pragma unroll
    for (int o2 = 1; o2 < 32; o2 <<= 1) {
      const int yg = __shfl_up_sync(0xffffffffu, gi, o2), ye = __shfl_up_sync(0xffffffffu, ei, o2);
      if (lane >= o2) {
        gi += yg;
        ei += ye;
      }
    }
    if (lane < kWarps) {
      wgt[lane] = gi - g;
      weq[lane] = ei - e;
    }
    if (lane == kWarps - 1) {
      cta_cnt[0] = gi;
      cta_cnt[1] = ei;
    }
  }
  cluster_sync();   // every CTA's totals are in place
  int gbase = 0, ebase = 0;   // keys above / equal to t in the runs of the lower ranks
  for (int r = 0; r < (int)rank; ++r) {
    gbase += (int)ld_cluster_u32(mapa(&cta_cnt[0], r));
    ebase += (int)ld_cluster_u32(mapa(&cta_cnt[1], r));
  }
  int gt = gbase + wgt[warp], eq = ebase + weq[warp];   // before this warp's next step
  const uint32_t lt = (1u << lane) - 1u;
  for (int i0 = q0; i0 < q1; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < q1 ? key_at(i) : 0u;
    const bool is_gt = i < q1 && key > prefix, is_eq = i < q1 && key == prefix;
    const uint32_t bg = __ballot_sync(0xffffffffu, is_gt), be = __ballot_sync(0xffffffffu, is_eq);
    const int g_before = gt + __popc(bg & lt), e_before = eq + __popc(be & lt);
    if (is_gt) o[g_before + min(e_before, krem)] = c0 + i;
    if (is_eq && e_before < krem) o[g_before + e_before] = c0 + i;
    gt += __popc(bg);
    eq += __popc(be);
  }
  cluster_sync();   // no peer reads this CTA's counts any more
}
}  // namespace

cudaError_t launch_read_ceiling(const void* buf, size_t bytes, uint32_t* sink, int sms, cudaStream_t s) {
  return launch_pdl(read_ceiling_kernel, dim3(4 * sms), dim3(512), 0, s,
                    static_cast<const uint4*>(buf), bytes / 16, sink);
}

cudaError_t launch_append_host_pos(const AppendParams& p, cudaStream_t s) {
  return launch_pdl(append_kernel, dim3(p.B), dim3(128), 0, s, p);
}

cudaError_t launch_sparse_prep(const int* topk, int K, const int* end_pos, int max_end_pos,
                               const Workspace& ws, int B, int* gidx_out, int* gcount_out,
                               const AppendRows& ap, cudaStream_t s) {
  return launch_pdl(sparse_prep_kernel, dim3(ap.kv_new ? 2 * B : B), dim3(1024), 0, s, topk, K, end_pos,
                    max_end_pos, ws, gidx_out, gcount_out, ap, B);
}

cudaError_t launch_schedule(const int* end_pos, int max_end_pos, const Workspace& ws, int B,
                            int target, int granule, bool direct, int mtp_s, bool append,
                            cudaStream_t s) {
  const int threads = B >= 1024 ? 1024 : ((B + 31) / 32) * 32;
  return launch_pdl(schedule_kernel, dim3(1), dim3(threads), 0, s, end_pos, max_end_pos, ws, B,
                    target, granule, direct ? 1 : 0, mtp_s < 1 ? 1 : mtp_s, append ? 1 : 0);
}

cudaError_t launch_append_end(const AppendRows& ap, const int* end_pos, int max_end_pos, int B,
                              cudaStream_t s) {
  return launch_pdl(append_end_kernel, dim3(B), dim3(128), 0, s, ap, end_pos, max_end_pos);
}

cudaError_t launch_combine(const Workspace& ws, int B, int H, void* out, float* lse,
                           cudaStream_t s) {
  // up to 32 sequences per head in flight; a CTA walks the rest
  return launch_pdl(combine_kernel, dim3(H, B < 32 ? B : 32), dim3(128), 0, s, ws, H, B,
                    static_cast<__nv_bfloat16*>(out), lse);
}

cudaError_t launch_topk_select(const float* scores, const int* end_pos, int B, int max_end_pos, int K,
                               int* out, cudaStream_t s) {
  const int per = ((max_end_pos + kTopkCtas - 1) / kTopkCtas + 3) & ~3;   // longest run of a CTA
  const bool staged = per <= kTopkSmemKeys;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(B * kTopkCtas);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.dynamicSmemBytes = staged ? (size_t)per * 4 : 0;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTopkCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (staged) {
    cudaError_t e = ensure_smem<topk_select_kernel<true>>((size_t)kTopkSmemKeys * 4);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, topk_select_kernel<true>, scores, max_end_pos, end_pos, max_end_pos, K, out);
  }
  return cudaLaunchKernelEx(&cfg, topk_select_kernel<false>, scores, max_end_pos, end_pos, max_end_pos, K, out);
}

}  // namespace mla
