// common.cuh -- constants, parameter blocks, the workspace layout and the
// launch helper shared by the host API (mla_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace mla {

constexpr int kDc = 512;          // latent width (kv_lora_rank)
constexpr int kDr = 64;           // rotary key width (qk_rope_head_dim)
constexpr int kDqk = kDc + kDr;   // 576: score contraction length
constexpr int kBlk = 128;         // FP8 block width
constexpr int kNblk = kDc / kBlk; // 4 scales per row
constexpr int kMaxAppendB = 2048; // rows one append call may write
constexpr int kMaxTopK = 8192;
constexpr int kMaxMtp = 1024;     // new tokens per sequence in one multi-token call (a prefill chunk)

constexpr uint32_t kDevEndPosClamped = 0x1u;
constexpr uint32_t kDevAppendSkipped = 0x2u;
constexpr uint32_t kDevTimeout = 0x4u;

// One unit of decode work: positions [t0, t1) of sequence b (dense), or
// entries [t0, t1) of b's gather list (sparse).  b < 0: no work.  Flags:
// kUnitDirect, the unit is its sequence's only one and the decode writes the
// final output and log-sum-exp itself (the combine skips the sequence);
// kUnitAppend, a dense call with new rows whose row end_pos - 1 = t1 - 1 this
// unit writes before reading it (tensor-memory kernel).
constexpr int kUnitDirect = 1, kUnitAppend = 2;
struct Unit {
  int b, t0, t1, flags;
};

// Workspace carve-up.  Every region starts on a 256-byte boundary.
struct Workspace {
  uint32_t* status;   // device status word (MLA_DEV_* bits)
  int* n_units;       // units actually scheduled
  int2* seq;          // [B] (first unit, unit count; -1: written by the decode)
  int* lengths;       // [B] clamped end_pos (dense) or gather count (sparse);
                      // not written when the decode computes its schedule
  Unit* units;        // [max_units] written by the schedule kernel (a decode
                      // that computes its schedule keeps its unit on chip)
  float* part_lse;    // [max_units, H]
  float* part_o;      // [max_units, H, 512]
  int* gidx;          // [B, K] sorted unique gather lists (sparse only)
  uint32_t* seq_flags;  // [B] status bits the sparse prep found per sequence
                        // (the schedule ORs them into the status word)
  size_t bytes;
  int max_units;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Units the scheduler aims for.  mma.sync path: H/16 CTAs per unit, about
// two per SM.  Tensor-memory path: one CTA pair per unit, one wave.
inline int target_units_mma(int H, int num_sms) {
  int per_unit = H / 16;
  return (2 * num_sms + per_unit - 1) / per_unit;
}
inline int target_units_tc(int num_sms) { return num_sms / 2; }
inline int target_units(int H, int num_sms) {
  int a = target_units_mma(H, num_sms), b = target_units_tc(num_sms);
  return a > b ? a : b;
}

inline Workspace carve_workspace(void* base, int B, int H, int K, int num_sms) {
  Workspace w{};
  w.max_units = target_units(H, num_sms) + B;
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = p ? p + off : nullptr;
    off += align256(bytes);
    return r;
  };
  char* hdr = take(16);
  w.status = reinterpret_cast<uint32_t*>(hdr);
  w.n_units = hdr ? reinterpret_cast<int*>(hdr + 4) : nullptr;
  w.seq = reinterpret_cast<int2*>(take(sizeof(int2) * (size_t)B));
  w.lengths = reinterpret_cast<int*>(take(sizeof(int) * (size_t)B));
  w.units = reinterpret_cast<Unit*>(take(sizeof(Unit) * (size_t)w.max_units));
  w.part_lse = reinterpret_cast<float*>(take(sizeof(float) * (size_t)w.max_units * H));
  w.part_o = reinterpret_cast<float*>(take(sizeof(float) * (size_t)w.max_units * H * kDc));
  if (K > 0) {
    w.gidx = reinterpret_cast<int*>(take(sizeof(int) * (size_t)B * K));
    w.seq_flags = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t) * (size_t)B));
  }
  w.bytes = off;
  return w;
}

// Parameters of the append kernels.
// The decode kernels read formats 1 and 2 alike (fp32 scales); only the
// cache write tells them apart.
inline int decode_fmt(int fmt) { return fmt == 2 ? 1 : fmt; }

// The cache and the new rows of an append (kv_new == nullptr: no append).
struct AppendRows {
  int fmt;                // 0 bf16, 1 FP8, 2 FP8 with power-of-two scales
  int max_seq_len;
  void* kv;
  float* kv_scale;
  void* pe;
  const void* kv_new;     // bf16 [B, 512]
  const void* pe_new;     // bf16 [B, 64]
};

// Plain append: row pos[b] of slot b, positions from the host.
struct AppendParams {
  AppendRows rows;
  int B;
  int pos[kMaxAppendB];
};

// A dense call's split schedule, for kernels that compute it themselves
// (schedule.cuh); end_pos == nullptr: the schedule kernel wrote the units.
// One warp holds the lengths (four per lane), so B <= kWarpScheduleMaxB.
constexpr int kWarpScheduleMaxB = 128;
struct DenseSchedule {
  const int* end_pos;   // device [B / mtp_s]
  int max_end_pos, B, target, granule, mtp_s;
  int direct;           // a sequence with a single unit is finished by the decode
  int append;           // the call writes row end_pos - 1 (the last unit does)
  // a sparse call: the lengths are the gather counts and the status bits the
  // per-sequence flags, both written by the gather-list prep (end_pos unused)
  const int* lengths = nullptr;
  const uint32_t* seq_flags = nullptr;
};

// Parameters of the decode kernels.
struct DecodeParams {
  int fmt;
  int max_seq_len;
  const void* kv;
  const float* kv_scale;
  const void* pe;
  const void* q_latent;   // bf16 [B, H, 512]
  const void* q_pe;       // bf16 [B, H, 64]
  int B, H;
  float scale_log2;       // softmax_scale * log2(e)
  void* out;              // bf16 [B, H, 512] (sequences with a direct unit)
  float* lse;             // fp32 [B, H] or null
  Workspace ws;
  int K;                  // sparse list length (0 = dense)
  int mtp_s;              // new tokens per cache slot: sequence b reads slot b / mtp_s (1: plain decode)
  long long spin_limit = 0;   // polls a bounded wait makes before it gives up (0: the default)
  int withhold_tile = -1;     // self-test of the bounded waits: this tile of the first unit is never loaded (-1: none)
  // dense call with new rows (ap.kv_new != nullptr, one token per slot): the
  // unit flagged kUnitAppend writes row t1 - 1 before loading it
  AppendRows ap{};
  DenseSchedule sched{};   // tensor-memory dense calls: each CTA finds its unit
};

// Raise a kernel's dynamic shared memory limit once per device.  The kernel
// is a template argument, so every kernel (and every instantiation of a
// kernel template) has its own flags.
template <auto kKernel>
cudaError_t ensure_smem(size_t bytes) {
  static int done[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = 1;
  return e;
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation, so its CTAs may start while the kernel
// before it in the stream is finishing.  Each kernel calls pdl_wait() before
// its first access to global memory that an earlier kernel may write or read
// (griddepcontrol.wait returns once the previous grid has completed and its
// writes are visible), then pdl_trigger() so the next kernel may begin to
// launch.  The data dependencies stay those of plain stream order; what
// overlaps is launch latency and per-CTA set-up.  Launched without the
// attribute, both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (defined in the kernel translation units).
cudaError_t launch_append_host_pos(const AppendParams& p, cudaStream_t s);
// The sparse call's first kernel: gather lists, gather counts and per-sequence
// status bits, and (ap.kv_new != nullptr) the append of row end_pos[b] - 1.
cudaError_t launch_sparse_prep(const int* topk, int K, const int* end_pos, int max_end_pos,
                               const Workspace& ws, int B, int* gidx_out, int* gcount_out,
                               const AppendRows& ap, cudaStream_t s);
// end_pos != nullptr: dense (lengths = clamped end_pos); nullptr: the lengths
// and per-sequence status bits were written by the sparse prep.  Either way
// the schedule writes the status word afresh (the call's earlier kernels
// leave it alone), so no memset precedes a call.
// direct: a sequence that gets a single unit is finished by the decode kernel.
// append (dense): the call also writes new rows; sequences whose row it cannot
// write (end_pos outside [1, max_end_pos]) raise MLA_DEV_APPEND_SKIPPED.
// mtp_s > 1 (dense): B counts s sequences per cache slot; sequence b is token
// b % s of slot b / s and attends to end_pos[b / s] - (s - 1 - b % s) positions.
cudaError_t launch_schedule(const int* end_pos, int max_end_pos, const Workspace& ws, int B,
                            int target, int granule, bool direct, int mtp_s, bool append,
                            cudaStream_t s);
// Dense call with new rows, warp-MMA decode path: row end_pos[b] - 1 of every
// sequence with end_pos[b] in [1, max_end_pos] (schedule with append = true
// flags the others).
cudaError_t launch_append_end(const AppendRows& ap, const int* end_pos, int max_end_pos, int B,
                              cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s);
int decode_mma_granule();
// tensor-memory path (H = 128): one CTA pair per unit
cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t s);
int decode_tc_granule(int fmt, bool sparse);   // positions per tile of the variant
bool decode_tc_supported(int H);
// units for one wave of the pair kernel: min(SMs / 2, CTA pairs that can be
// resident at once), which the GPU's cluster placement may hold below SMs / 2
int decode_tc_units(int fmt, bool sparse, int num_sms);
cudaError_t launch_combine(const Workspace& ws, int B, int H, void* out, float* lse,
                           cudaStream_t s);
// per-head products around the decode (absorb.cu): q_latent = q_nope . W_UK,
// o = W_UV . x, with wkv_b [H, 256, 512] bf16 holding W_UK and W_UV per head
cudaError_t launch_absorb_q(const void* q_nope, const void* wkv_b, int B, int H, void* q_latent,
                            uint32_t* status, cudaStream_t s);
cudaError_t launch_project_out(const void* x, const void* wkv_b, int B, int H, void* o,
                               uint32_t* status, cudaStream_t s);
// streams `bytes` (a multiple of 16) of device memory, XOR-folding into *sink
cudaError_t launch_read_ceiling(const void* buf, size_t bytes, uint32_t* sink, int sms, cudaStream_t s);
// top-k position selection: scores [B][max_end_pos] fp32 -> out [B][K] int32
cudaError_t launch_topk_select(const float* scores, const int* end_pos, int B, int max_end_pos, int K,
                               int* out, cudaStream_t s);

}  // namespace mla
