// mla_api.cu -- the C ABI declared in include/mla.h: argument checks, the
// workspace carve-up and the launch sequence of each call.  Every check that
// the host can make happens before the first launch.
#include <mutex>
#include <new>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/mla.h"
#include "common.cuh"

namespace {

thread_local char g_last_error[256] = "";

mla_status cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

// Per-thread trace of the main decode kernel (see mla_trace_begin).
struct Trace {
  bool on = false;
  int cap = 0, n = 0, launches = 0;
  cudaEvent_t* ev = nullptr;  // [2 * cap]: start, stop pairs
};
thread_local Trace g_trace;

void trace_launches(int k) {
  if (g_trace.on) g_trace.launches += k;
}

bool trace_start(cudaStream_t s) {
  if (!g_trace.on || g_trace.n >= g_trace.cap) return false;
  // External records become real event nodes when the stream is being captured
  // into a graph (a plain record would only mark a dependency); outside
  // capture they behave as ordinary records.
  return cudaEventRecordWithFlags(g_trace.ev[2 * g_trace.n], s, cudaEventRecordExternal) == cudaSuccess;
}

void trace_stop(cudaStream_t s, bool started) {
  if (!started) return;
  if (cudaEventRecordWithFlags(g_trace.ev[2 * g_trace.n + 1], s, cudaEventRecordExternal) == cudaSuccess)
    ++g_trace.n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// SM count of the current device, cached per device.
int num_sms(int* out) {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return -1;
    }
    cache[dev] = n;
  }
  *out = cache[dev];
  return 0;
}

bool supported_heads(int H) { return H == 16 || H == 32 || H == 64 || H == 128; }

mla_status check_cache(const mla_cache* c) {
  if (!c || !c->kv || !c->pe) return MLA_ERR_INVALID_ARG;
  if (c->fmt != MLA_KV_BF16 && c->fmt != MLA_KV_FP8_E4M3_B128 && c->fmt != MLA_KV_FP8_E4M3_B128_POW2)
    return MLA_ERR_UNSUPPORTED;
  if (c->max_batch <= 0 || c->max_seq_len <= 0) return MLA_ERR_INVALID_ARG;
  if (!aligned16(c->kv) || !aligned16(c->pe)) return MLA_ERR_INVALID_ARG;
  if (c->fmt != MLA_KV_BF16 && (!c->kv_scale || !aligned16(c->kv_scale)))
    return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

mla::AppendRows append_rows(const mla_cache* c, const void* kv_new, const void* pe_new) {
  mla::AppendRows r{};
  r.fmt = c->fmt;
  r.max_seq_len = c->max_seq_len;
  r.kv = c->kv;
  r.kv_scale = c->kv_scale;
  r.pe = c->pe;
  r.kv_new = kv_new;
  r.pe_new = pe_new;
  return r;
}

struct DecodeArgs {
  const mla_cache* cache;
  const void* q_latent;
  const void* q_pe;
  const int32_t* end_pos;
  int32_t max_end_pos, B, H;
  float softmax_scale;
  void* out;
  float* lse;
  void* workspace;
  size_t ws_bytes;
  int32_t mtp_s;   // new tokens per sequence; B counts B / mtp_s cache slots x mtp_s
};

mla_status check_decode(const DecodeArgs& a, int K, mla::Workspace* ws) {
  mla_status st = check_cache(a.cache);
  if (st != MLA_OK) return st;
  if (!supported_heads(a.H)) return MLA_ERR_UNSUPPORTED;
  if (a.B <= 0 || a.B / a.mtp_s > a.cache->max_batch) return MLA_ERR_INVALID_ARG;
  if (a.max_end_pos <= 0 || a.max_end_pos > a.cache->max_seq_len) return MLA_ERR_OUT_OF_RANGE;
  if (!a.q_latent || !a.q_pe || !a.end_pos || !a.out) return MLA_ERR_INVALID_ARG;
  if (!aligned16(a.q_latent) || !aligned16(a.q_pe) || !aligned16(a.out) || !aligned4(a.end_pos))
    return MLA_ERR_INVALID_ARG;
  if (a.lse && !aligned4(a.lse)) return MLA_ERR_INVALID_ARG;
  if (!(a.softmax_scale == a.softmax_scale)) return MLA_ERR_INVALID_ARG;  // NaN
  int sms = 0;
  if (num_sms(&sms) != 0) return MLA_ERR_UNSUPPORTED;
  mla::Workspace need = mla::carve_workspace(nullptr, a.B, a.H, K, sms);
  if (!a.workspace || !aligned16(a.workspace) || a.ws_bytes < need.bytes) return MLA_ERR_WORKSPACE;
  *ws = mla::carve_workspace(a.workspace, a.B, a.H, K, sms);
  return MLA_OK;
}

mla::DecodeParams make_params(const DecodeArgs& a, const mla::Workspace& ws, int K) {
  mla::DecodeParams p{};
  p.fmt = mla::decode_fmt(a.cache->fmt);
  p.max_seq_len = a.cache->max_seq_len;
  p.kv = a.cache->kv;
  p.kv_scale = a.cache->kv_scale;
  p.pe = a.cache->pe;
  p.q_latent = a.q_latent;
  p.q_pe = a.q_pe;
  p.B = a.B;
  p.H = a.H;
  p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
  p.out = a.out;
  p.lse = a.lse;
  p.ws = ws;
  p.K = K;
  p.mtp_s = a.mtp_s;
  p.spin_limit = 0;
  p.withhold_tile = -1;
  return p;
}

// Decode path: the tensor-memory kernel for H = 128 unless MLA_DECODE_PATH=mma
// (read once per process) selects the warp-MMA kernel.
bool use_tc_path(int H) {
  static int forced = -1;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* v = getenv("MLA_DECODE_PATH");
    forced = (v && strcmp(v, "mma") == 0) ? 0 : 1;
  });
  return forced && mla::decode_tc_supported(H);
}

// schedule -> decode -> combine, after the lengths are known on the device.
// ap (dense, one token per slot): also write row end_pos[b] - 1 of every
// sequence from ap.kv_new / ap.pe_new -- inside the tensor-memory decode
// kernel, or by a kernel of its own ahead of the warp-MMA path.
mla_status run_decode(const DecodeArgs& a, const mla::Workspace& ws, int K, cudaStream_t s,
                      long long spin_limit = 0, int withhold_tile = -1,
                      const mla::AppendRows* ap = nullptr) {
  int sms = 0;
  num_sms(&sms);
  const bool tc = use_tc_path(a.H);
  cudaError_t e;
  if (ap && !tc) {
    e = mla::launch_append_end(*ap, a.end_pos, a.max_end_pos, a.B, s);
    if (e != cudaSuccess) return cuda_fail(e, "append");
    trace_launches(1);
  }
  const int target =
      tc ? mla::decode_tc_units(mla::decode_fmt(a.cache->fmt), K > 0, sms) : mla::target_units_mma(a.H, sms);
  const int granule = tc ? mla::decode_tc_granule(mla::decode_fmt(a.cache->fmt), K > 0) : mla::decode_mma_granule();
  // dense bf16 and sparse calls of up to kWarpScheduleMaxB sequences on the
  // tensor-memory kernel: every CTA pair works out its own unit (a sparse
  // call from the gather counts the prep kernel wrote), so no schedule kernel
  // sits between the call's start (or its prep) and the first loads.  (The
  // dense FP8 variant runs at its register limit, where the added code cost
  // more than it saved; long calls -- prefill chunks -- keep the schedule
  // kernel.)
  const bool fused_schedule =
      tc && a.B <= mla::kWarpScheduleMaxB && (K > 0 || mla::decode_fmt(a.cache->fmt) == 0);
  if (!fused_schedule) {
    e = mla::launch_schedule(K ? nullptr : a.end_pos, a.max_end_pos, ws, a.B, target, granule, tc, a.mtp_s,
                             ap != nullptr, s);
    if (e != cudaSuccess) return cuda_fail(e, "schedule");
    trace_launches(1);
  }
  const bool traced = trace_start(s);
  mla::DecodeParams p = make_params(a, ws, K);
  p.spin_limit = spin_limit;
  p.withhold_tile = withhold_tile;
  if (ap && tc) p.ap = *ap;
  if (fused_schedule && K == 0)
    p.sched = mla::DenseSchedule{a.end_pos, a.max_end_pos, a.B, target, granule, a.mtp_s, 1, ap != nullptr ? 1 : 0};
  else if (fused_schedule)
    p.sched = mla::DenseSchedule{nullptr, a.max_end_pos, a.B, target, granule, 1, 1, 0, ws.lengths, ws.seq_flags};
  e = tc ? mla::launch_decode_tc(p, s) : mla::launch_decode_mma(p, s);
  trace_stop(s, traced);
  if (e != cudaSuccess) return cuda_fail(e, "decode");
  e = mla::launch_combine(ws, a.B, a.H, a.out, a.lse, s);
  if (e != cudaSuccess) return cuda_fail(e, "combine");
  trace_launches(2);
  return MLA_OK;
}

mla_status check_absorb(const void* x, const void* wkv_b, int32_t B, int32_t H, const void* y,
                        const uint32_t* status) {
  if (!x || !wkv_b || !y || !aligned16(x) || !aligned16(wkv_b) || !aligned16(y)) return MLA_ERR_INVALID_ARG;
  if (status && !aligned4(status)) return MLA_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || B > (1 << 22) || H > (1 << 16)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}
}  // namespace

extern "C" {

mla_status mla_cache_append(const mla_cache* cache, const void* kv_new, const void* pe_new,
                            const int32_t* start_pos, int32_t B, void* stream) {
  g_last_error[0] = 0;
  mla_status st = check_cache(cache);
  if (st != MLA_OK) return st;
  if (!kv_new || !pe_new || !start_pos) return MLA_ERR_INVALID_ARG;
  if (!aligned16(kv_new) || !aligned16(pe_new)) return MLA_ERR_INVALID_ARG;
  if (B <= 0 || B > cache->max_batch || B > mla::kMaxAppendB) return MLA_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b)
    if (start_pos[b] < 0 || start_pos[b] >= cache->max_seq_len) return MLA_ERR_OUT_OF_RANGE;
  mla::AppendParams p{};
  p.rows = append_rows(cache, kv_new, pe_new);
  p.B = B;
  memcpy(p.pos, start_pos, sizeof(int32_t) * (size_t)B);
  cudaError_t e = mla::launch_append_host_pos(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append");
  trace_launches(1);
  return MLA_OK;
}

size_t mla_workspace_size(int32_t B, int32_t H, int32_t max_end_pos, int32_t topk) {
  (void)max_end_pos;
  if (B <= 0 || !supported_heads(H) || topk < 0 || topk > mla::kMaxTopK) return 0;
  int sms = 0;
  if (num_sms(&sms) != 0) return 0;
  return mla::carve_workspace(nullptr, B, H, topk, sms).bytes;
}

mla_status mla_decode(const mla_cache* cache, const void* q_latent, const void* q_pe,
                      const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                      float softmax_scale, void* out, float* lse, void* workspace,
                      size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  DecodeArgs a{cache, q_latent, q_pe, end_pos, max_end_pos, B, H, softmax_scale, out, lse,
               workspace, ws_bytes, 1};
  mla::Workspace ws;
  mla_status st = check_decode(a, 0, &ws);
  if (st != MLA_OK) return st;
  // the call's first kernel (the schedule kernel, or a decode kernel that
  // computes its own schedule) writes the status word afresh
  return run_decode(a, ws, 0, static_cast<cudaStream_t>(stream));
}

mla_status mla_decode_append(const mla_cache* cache, const void* kv_new, const void* pe_new,
                             const void* q_latent, const void* q_pe, const int32_t* end_pos,
                             int32_t max_end_pos, int32_t B, int32_t H, float softmax_scale, void* out,
                             float* lse, void* workspace, size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  if (!kv_new || !pe_new || !aligned16(kv_new) || !aligned16(pe_new)) return MLA_ERR_INVALID_ARG;
  DecodeArgs a{cache, q_latent, q_pe, end_pos, max_end_pos, B, H, softmax_scale, out, lse,
               workspace, ws_bytes, 1};
  mla::Workspace ws;
  mla_status st = check_decode(a, 0, &ws);
  if (st != MLA_OK) return st;
  const mla::AppendRows ap = append_rows(cache, kv_new, pe_new);
  return run_decode(a, ws, 0, static_cast<cudaStream_t>(stream), 0, -1, &ap);
}

}  // extern "C"

namespace mla {

// The dense decode of mla_decode with a scratch region supplied by the library
// itself (mla_noalloc.cu) instead of a caller workspace: the same argument
// checks (a scratch smaller than this B and H need -> MLA_ERR_WORKSPACE), the
// same kernels and launch sequence, the same error reporting.
mla_status decode_in_scratch(const mla_cache* cache, const void* q_latent, const void* q_pe,
                             const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                             float softmax_scale, void* out, float* lse, void* scratch,
                             size_t scratch_bytes, void* stream) {
  g_last_error[0] = 0;
  DecodeArgs a{cache, q_latent, q_pe, end_pos, max_end_pos, B, H, softmax_scale, out, lse,
               scratch, scratch_bytes, 1};
  mla::Workspace ws;
  mla_status st = check_decode(a, 0, &ws);
  if (st != MLA_OK) return st;
  return run_decode(a, ws, 0, static_cast<cudaStream_t>(stream));
}

}  // namespace mla

extern "C" {

mla_status mla_topk_select(const float* scores, const int32_t* end_pos, int32_t B, int32_t max_end_pos,
                           int32_t K, int32_t* topk_idx, void* stream) {
  g_last_error[0] = 0;
  if (!scores || !end_pos || !topk_idx || !aligned4(scores) || !aligned4(end_pos) || !aligned4(topk_idx))
    return MLA_ERR_INVALID_ARG;
  if (B < 1 || max_end_pos < 1 || K < 1 || K > mla::kMaxTopK) return MLA_ERR_INVALID_ARG;
  cudaError_t e = mla::launch_topk_select(scores, end_pos, B, max_end_pos, K, topk_idx,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "topk_select");
  trace_launches(1);
  return MLA_OK;
}

mla_status mla_selftest_decode_timeout(const mla_cache* cache, const void* q_latent, const void* q_pe,
                                       const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                                       float softmax_scale, void* out, float* lse, void* workspace,
                                       size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  DecodeArgs a{cache, q_latent, q_pe, end_pos, max_end_pos, B, H, softmax_scale, out, lse,
               workspace, ws_bytes, 1};
  mla::Workspace ws;
  mla_status st = check_decode(a, 0, &ws);
  if (st != MLA_OK) return st;
  if (!use_tc_path(H)) return MLA_ERR_UNSUPPORTED;
  // the first unit's first tile is never loaded; every wait gives up after
  // 2^16 polls (milliseconds)
  return run_decode(a, ws, 0, static_cast<cudaStream_t>(stream), 1LL << 16, 0);
}

mla_status mla_decode_mtp(const mla_cache* cache, const void* q_latent, const void* q_pe,
                          const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t s,
                          int32_t H, float softmax_scale, void* out, float* lse, void* workspace,
                          size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  if (s < 1 || s > mla::kMaxMtp || B <= 0 || B > (1 << 30) / s) return MLA_ERR_INVALID_ARG;
  // B * s sequences; sequence b * s + j is token j of cache slot b
  DecodeArgs a{cache, q_latent, q_pe, end_pos, max_end_pos, B * s, H, softmax_scale, out, lse,
               workspace, ws_bytes, s};
  mla::Workspace ws;
  mla_status st = check_decode(a, 0, &ws);
  if (st != MLA_OK) return st;
  return run_decode(a, ws, 0, static_cast<cudaStream_t>(stream));
}

mla_status mla_decode_sparse(const mla_cache* cache, const void* q_latent, const void* q_pe,
                             const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                             float softmax_scale, const int32_t* topk_idx, int32_t K,
                             const void* kv_new, const void* pe_new, void* out, float* lse,
                             int32_t* gidx_out, int32_t* gcount_out, void* workspace,
                             size_t ws_bytes, void* stream) {
  g_last_error[0] = 0;
  if (!topk_idx || K <= 0 || K > mla::kMaxTopK || !aligned4(topk_idx)) return MLA_ERR_INVALID_ARG;
  if (cache && B > 0 && (int64_t)B * cache->max_seq_len > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  if ((kv_new == nullptr) != (pe_new == nullptr)) return MLA_ERR_INVALID_ARG;
  if (kv_new && (!aligned16(kv_new) || !aligned16(pe_new) || B > mla::kMaxAppendB))
    return MLA_ERR_INVALID_ARG;
  if ((gidx_out && !aligned4(gidx_out)) || (gcount_out && !aligned4(gcount_out)))
    return MLA_ERR_INVALID_ARG;
  DecodeArgs a{cache, q_latent, q_pe, end_pos, max_end_pos, B, H, softmax_scale, out, lse,
               workspace, ws_bytes, 1};
  mla::Workspace ws;
  mla_status st = check_decode(a, K, &ws);
  if (st != MLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the prep kernel also appends the new rows (kv_new may be NULL); the
  // schedule after it writes the status word, so no memset precedes them
  cudaError_t e = mla::launch_sparse_prep(topk_idx, K, end_pos, max_end_pos, ws, B, gidx_out,
                                          gcount_out, append_rows(cache, kv_new, pe_new), s);
  if (e != cudaSuccess) return cuda_fail(e, "sparse_prep");
  trace_launches(1);
  return run_decode(a, ws, K, s);
}

mla_status mla_workspace_status(const void* workspace, uint32_t* flags, void* stream) {
  if (!workspace || !flags) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e, "status");
}

mla_status mla_absorb_q(const void* q_nope, const void* wkv_b, int32_t B, int32_t H, void* q_latent,
                        uint32_t* status, void* stream) {
  g_last_error[0] = 0;
  mla_status st = check_absorb(q_nope, wkv_b, B, H, q_latent, status);
  if (st != MLA_OK) return st;
  cudaError_t e = mla::launch_absorb_q(q_nope, wkv_b, B, H, q_latent, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "absorb_q");
  trace_launches(1);
  return MLA_OK;
}

mla_status mla_project_out(const void* x, const void* wkv_b, int32_t B, int32_t H, void* o,
                           uint32_t* status, void* stream) {
  g_last_error[0] = 0;
  mla_status st = check_absorb(x, wkv_b, B, H, o, status);
  if (st != MLA_OK) return st;
  cudaError_t e = mla::launch_project_out(x, wkv_b, B, H, o, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "project_out");
  trace_launches(1);
  return MLA_OK;
}

mla_status mla_read_ceiling(const void* buf, size_t bytes, uint32_t* sink, void* stream) {
  g_last_error[0] = 0;
  if (!buf || !sink || bytes == 0 || (bytes & 15u) || !aligned16(buf) || !aligned4(sink))
    return MLA_ERR_INVALID_ARG;
  int sms = 0;
  if (num_sms(&sms) != 0) return MLA_ERR_UNSUPPORTED;
  cudaError_t e = mla::launch_read_ceiling(buf, bytes, sink, sms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "read_ceiling");
  trace_launches(1);
  return MLA_OK;
}

const char* mla_status_string(mla_status status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_OUT_OF_RANGE: return "MLA_ERR_OUT_OF_RANGE";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
  }
  return "MLA_ERR_UNKNOWN";
}

const char* mla_last_error(void) { return g_last_error; }

mla_status mla_trace_begin(int32_t max_records) {
  if (g_trace.on || max_records < 0 || max_records > (1 << 20)) return MLA_ERR_INVALID_ARG;
  Trace t;
  t.cap = max_records;
  if (max_records > 0) {
    t.ev = new (std::nothrow) cudaEvent_t[2 * (size_t)max_records];
    if (!t.ev) return MLA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 2 * max_records; ++i) {
    cudaError_t e = cudaEventCreate(&t.ev[i]);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(t.ev[j]);
      delete[] t.ev;
      return cuda_fail(e, "trace_begin");
    }
  }
  t.on = true;
  g_trace = t;
  return MLA_OK;
}

mla_status mla_trace_end(float* main_kernel_ms, int32_t* timed_launches, int32_t* kernel_launches) {
  if (!g_trace.on) return MLA_ERR_INVALID_ARG;
  Trace t = g_trace;
  g_trace = Trace();
  mla_status st = MLA_OK;
  double total = 0.0;
  if (t.n > 0) {
    cudaError_t e = cudaEventSynchronize(t.ev[2 * t.n - 1]);
    for (int i = 0; e == cudaSuccess && i < t.n; ++i) {
      float ms = 0.f;
      e = cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]);
      total += ms;
    }
    if (e != cudaSuccess) st = cuda_fail(e, "trace_end");
  }
  for (int i = 0; i < 2 * t.cap; ++i) cudaEventDestroy(t.ev[i]);
  delete[] t.ev;   // null when only launches were counted
  if (main_kernel_ms) *main_kernel_ms = (float)total;
  if (timed_launches) *timed_launches = t.n;
  if (kernel_launches) *kernel_launches = t.launches;
  return st;
}

}  // extern "C"
