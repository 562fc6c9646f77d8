// schedule.cuh -- the split schedule of a call computed by one warp, for the
// tensor-memory decode kernel: every CTA finds its own unit from end_pos (a
// dense call) or from the gather counts the list prep wrote (a sparse call),
// so no schedule kernel (and no unit table round trip) sits between the
// call's start, or the prep, and the first cache load.  The rule is schedule_kernel's
// (aux_kernels.cu): lengths cut into units of `chunk` positions, chunk the
// smallest granule multiple with sum_b ceil(len_b / chunk) <= target, capped
// at the longest length.
#pragma once

#include "append_row.cuh"
#include "common.cuh"

namespace mla {

// Length of sequence b: clamped end_pos of its slot, less one position per
// later token of the slot (multi-token calls).
__device__ __forceinline__ int dense_len(const DenseSchedule& s, int b, uint32_t* flags) {
  int len = s.end_pos[b / s.mtp_s];
  if (len < 0 || len > s.max_end_pos) {
    *flags |= kDevEndPosClamped;
    len = len < 0 ? 0 : s.max_end_pos;
  }
  len -= s.mtp_s - 1 - b % s.mtp_s;
  return len < 0 ? 0 : len;
}

// Run by all 32 lanes of one warp, B <= kWarpScheduleMaxB.  Returns unit
// `want` of the schedule ({-1, 0, 0, 0} if the schedule has fewer units), the
// status bits the call's arguments raise (clamped end_pos, rows the append
// leaves out) and the number of units, and, with `seq` non-null, writes the
// per-sequence table the combine reads: (first unit, unit count, or -1 for a
// sequence the decode finishes itself).  Lengths are read once and kept in
// registers; the per-sequence divisions are 32-bit (lengths and chunk fit).
__device__ Unit warp_schedule(const DenseSchedule& s, int want, uint32_t* flags_out, int* units_out,
                              int2* seq) {
  const int lane = threadIdx.x & 31;
  const int nblk = (s.B + 31) >> 5;   // blocks of 32 sequences: 1..4 (warp-uniform)
  int len[4];
  uint32_t flags = 0;
  // the total as 128 * hi + lo, each part a 32-bit warp sum (len < 2^31)
  int hi = 0, lo = 0, longest = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    len[r] = 0;
    if (r < nblk) {
      const int b = lane + 32 * r;
      if (b < s.B) {
        if (s.lengths) {
          len[r] = s.lengths[b];
          flags |= s.seq_flags[b];
        } else {
          len[r] = dense_len(s, b, &flags);
          if (s.append && s.mtp_s == 1 && !append_row_valid(s.end_pos[b], s.max_end_pos)) flags |= kDevAppendSkipped;
        }
      }
      hi += len[r] >> 7;
      lo += len[r] & 127;
      longest = len[r] > longest ? len[r] : longest;
    }
  }
  hi = __reduce_add_sync(0xffffffffu, hi);
  lo = __reduce_add_sync(0xffffffffu, lo);
  longest = (int)__reduce_max_sync(0xffffffffu, (unsigned)longest);
  flags = __reduce_or_sync(0xffffffffu, flags);
  const unsigned long long total = (unsigned long long)hi * 128u + (unsigned)lo;
  const unsigned g = (unsigned)s.granule;
  const unsigned cap = (unsigned)longest > g ? ((unsigned)longest + g - 1) / g * g : g;
  unsigned long long c0 = total < 0xffff0000ull ? (unsigned)((unsigned)total + s.target - 1) / (unsigned)s.target
                                                : (total + s.target - 1) / (unsigned long long)s.target;
  c0 = (c0 + g - 1) / g * g;
  unsigned chunk = c0 < g ? g : (c0 > cap ? cap : (unsigned)c0);
  for (int iter = 0; iter < 64; ++iter) {
    int mine = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r)
      if (r < nblk) mine += (int)(((unsigned)len[r] + chunk - 1) / chunk);
    const int n = __reduce_add_sync(0xffffffffu, mine);
    if (n <= s.target || chunk >= cap) break;
    unsigned long long grown = ((unsigned long long)chunk * n + s.target - 1) / (unsigned long long)s.target;
    grown = (grown + g - 1) / g * g;
    if (grown < chunk + g) grown = chunk + g;
    chunk = grown > cap ? cap : (unsigned)grown;
  }
  // walk the sequences in order: unit numbers are an exclusive prefix sum
  Unit found{-1, 0, 0, 0};
  int carry = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    if (r >= nblk) break;
    const int b = lane + 32 * r;
    const int n = (int)(((unsigned)len[r] + chunk - 1) / chunk);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int u0 = carry + incl - n;
    const bool one = s.direct && n == 1;
    if (b < s.B && want >= u0 && want < u0 + n) {
      const int i = want - u0;
      const unsigned t1 = (unsigned)(i + 1) * chunk < (unsigned)len[r] ? (unsigned)(i + 1) * chunk : (unsigned)len[r];
      const int app = s.append && s.mtp_s == 1 && i == n - 1 && append_row_valid(s.end_pos[b], s.max_end_pos)
                          ? kUnitAppend : 0;
      found = Unit{b, (int)((unsigned)i * chunk), (int)t1, (one ? kUnitDirect : 0) | app};
    }
    if (seq && b < s.B) seq[b] = make_int2(u0, one ? -1 : n);
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  // the lane that found the unit broadcasts it
  const uint32_t hit = __ballot_sync(0xffffffffu, found.b >= 0);
  if (hit) {
    const int src = __ffs(hit) - 1;
    found.b = __shfl_sync(0xffffffffu, found.b, src);
    found.t0 = __shfl_sync(0xffffffffu, found.t0, src);
    found.t1 = __shfl_sync(0xffffffffu, found.t1, src);
    found.flags = __shfl_sync(0xffffffffu, found.flags, src);
  }
  *flags_out = flags;
  *units_out = carry;
  return found;
}

}  // namespace mla
