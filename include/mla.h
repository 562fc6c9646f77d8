/*
 * mla.h -- C ABI of libmla: absorbed Multi-Head Latent Attention decode over a
 * compressed latent KV cache on one NVIDIA GB300 (sm_103a).
 *
 * What the library computes (sources are web pages, cited by title/section):
 *   - "DeepSeek-V3.2-Exp . KV cache" (atlas.klimoza.dev), cache-write excerpt:
 *     each call writes the new rows of every sequence at start_pos, after
 *     rounding the 512-wide latent through FP8 with one scale per 128 values;
 *     the 64-wide rotary key is stored as is.
 *   - same page, MQA-decode excerpt: scores = (q_latent . c_KV + q_pe . k_R)
 *     * softmax_scale over cached positions 0..end_pos-1, an optional top-k
 *     index mask (positions outside the list get -inf), softmax, and the
 *     weighted sum of c_KV, which stays in the 512-wide latent space.
 *   - "DeepSeek MLA architecture: how Multi-Head Latent Attention cuts KV
 *     cache by 93%", sections 3-4: the score splits into a content term and a
 *     rotary term, and W_UK / W_UV are absorbed into the query and applied
 *     after the weighted sum (both outside this library: q_latent arrives
 *     already absorbed and the output is returned in latent space).
 *
 * Conventions shared by every call
 *   - The caller owns every buffer.  Device pointers must be device memory of
 *     the current CUDA device; "host" pointers are ordinary host memory.  The
 *     library allocates no device memory and keeps no state except cached
 *     device attributes and driver entry points.
 *   - All work is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  Nothing synchronises unless stated.
 *   - Host-checkable errors return an MLA_ERR_* code before anything is
 *     launched.  A failed launch returns MLA_ERR_CUDA.
 *   - Conditions only the device can see never trap: they are clamped or
 *     skipped and recorded in the status word of the workspace (see
 *     mla_workspace_status).
 *   - Sizes: latent width 512, rotary width 64, FP8 block 128 are fixed.
 *     H must be 16, 32, 64 or 128.  Device pointers must be 16-byte aligned.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer      */
  MLA_ERR_OUT_OF_RANGE = 2,  /* a position outside [0, max_seq_len)             */
  MLA_ERR_UNSUPPORTED = 3,   /* H, format or device not supported               */
  MLA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than required      */
  MLA_ERR_CUDA = 5           /* a CUDA runtime/driver call failed               */
} mla_status;

typedef enum {
  MLA_KV_BF16 = 0,           /* kv: bf16 [max_batch, max_seq_len, 512]          */
  MLA_KV_FP8_E4M3_B128 = 1,  /* kv: e4m3 bytes [max_batch, max_seq_len, 512] and
                                kv_scale: fp32 [max_batch, max_seq_len, 4]      */
  MLA_KV_FP8_E4M3_B128_POW2 = 2  /* the layout of format 1; every scale is a
                                power of two (the exponent-only "ue8m0" scale
                                format), still stored as fp32                   */
} mla_kv_format;

/* Cache descriptor (caller-owned device buffers, row-major, one slot per
 * sequence, as the register_buffer calls of "DeepSeek-V3.2-Exp . KV cache"
 * lay them out: [max_batch_size, max_seq_len, width]).
 *   kv       latent c_KV: bf16 or e4m3 codes, see mla_kv_format
 *   kv_scale fp32 block scales [max_batch, max_seq_len, 4] (FP8 formats
 *            only; NULL for bf16).  Scale j covers latent columns
 *            128j..128j+127 and the stored value is
 *            bf16(fp32(e4m3(code) * scale)).  The decode calls read formats 1
 *            and 2 alike; only the cache write differs.
 *   pe       rotary key k_R, bf16 [max_batch, max_seq_len, 64]            */
typedef struct {
  int32_t fmt;               /* mla_kv_format */
  int32_t max_batch;
  int32_t max_seq_len;
  void* kv;
  float* kv_scale;
  void* pe;
} mla_cache;

/* Bit flags of the device status word (OR-ed; each decode call on the
 * workspace -- mla_decode, mla_decode_append, mla_decode_mtp,
 * mla_decode_sparse -- writes the word afresh, then adds its own flags). */
#define MLA_DEV_END_POS_CLAMPED   0x1u  /* an end_pos was < 0 or > max_end_pos  */
#define MLA_DEV_APPEND_SKIPPED    0x2u  /* fused append: end_pos-1 out of range */
#define MLA_DEV_PIPELINE_TIMEOUT  0x4u  /* a bounded wait in a kernel gave up   */

/*
 * mla_cache_append -- the cache-write step of "DeepSeek-V3.2-Exp . KV cache"
 * (cache-write excerpt) and of "KV Cache Eviction Strategy in MLA ...",
 * section "Write-Back Logic and Position Tracking": for b in [0, B) write
 * kv_new[b] into row start_pos[b] of sequence slot b, and pe_new[b] into the
 * same row of pe.  bf16 caches store the row unchanged.  FP8 caches store
 * e4m3 codes and 4 fp32 scales: per 128-wide block, amax = max |x|, scale =
 * fp32(amax / 448) -- for MLA_KV_FP8_E4M3_B128_POW2 rounded up to the
 * smallest power of two not below it (the page passes a scale format to the
 * quantiser without defining it; this is the exponent-only reading) -- and
 * code = e4m3(fp32(x / scale)) with round-to-nearest-even and saturation to
 * +-448; an all-zero block stores scale 0 and code 0.
 *
 *   kv_new     device bf16 [B, 512]
 *   pe_new     device bf16 [B, 64]
 *   start_pos  HOST int32 [B]; each must be in [0, max_seq_len), otherwise
 *              MLA_ERR_OUT_OF_RANGE and nothing is written.  (The page's claim
 *              that writes past max_seq_len evict old rows does not hold for
 *              PyTorch slice assignment, which drops the new rows silently;
 *              the library refuses instead.)
 *   B          1 <= B <= min(max_batch, 2048)
 */
MLA_API mla_status mla_cache_append(const mla_cache* cache, const void* kv_new, const void* pe_new,
                            const int32_t* start_pos, int32_t B, void* stream);

/*
 * mla_workspace_size -- bytes of device workspace mla_decode (topk == 0) or
 * mla_decode_sparse (topk = K > 0) needs for B sequences and H heads.  The
 * workspace holds the split schedule, the per-split partial outputs and
 * log-sum-exps, the gather lists and the device status word.  max_end_pos is
 * accepted for interface stability; the size does not depend on it.
 * Returns 0 for unsupported arguments.
 */
MLA_API size_t mla_workspace_size(int32_t B, int32_t H, int32_t max_end_pos, int32_t topk);

/*
 * mla_decode -- absorbed MLA decode for one query token per sequence
 * ("DeepSeek-V3.2-Exp . KV cache", MQA-decode excerpt, without the index
 * mask; "DeepSeek MLA architecture ...", sections 3-4):
 *   s[b,h,t] = softmax_scale * (q_latent[b,h,:] . c[b,t,:] + q_pe[b,h,:] . kR[b,t,:])
 *   for t in [0, end_pos[b]);  p = softmax_t(s);  out[b,h,:] = sum_t p c[b,t,:]
 *   lse[b,h] = log sum_t exp(s[b,h,t])   (natural log)
 * where c is the bf16 latent or its FP8 round trip.  Work is split along t
 * across the GPU and merged by log-sum-exp.
 *
 *   q_latent    device bf16 [B, H, 512] (absorbed queries)
 *   q_pe        device bf16 [B, H, 64]  (rotated rotary queries)
 *   end_pos     device int32 [B]; positions read are 0..end_pos[b]-1.
 *               Values < 0 or > max_end_pos are clamped on the device and
 *               flagged (MLA_DEV_END_POS_CLAMPED).  end_pos[b] == 0 gives
 *               out = 0 and lse = -inf.
 *   max_end_pos host bound on every end_pos[b]; 1 <= max_end_pos <= max_seq_len
 *   out         device bf16 [B, H, 512] (round to nearest even)
 *   lse         device fp32 [B, H] or NULL
 *   workspace   device, >= mla_workspace_size(B, H, max_end_pos, 0) bytes,
 *               16-byte aligned; overwritten by the call
 */
MLA_API mla_status mla_decode(const mla_cache* cache, const void* q_latent, const void* q_pe,
                      const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                      float softmax_scale, void* out, float* lse, void* workspace,
                      size_t ws_bytes, void* stream);

/*
 * mla_decode_append -- the decoding step of "DeepSeek-V3.2-Exp . KV cache"
 * as one call: the cache-write excerpt (the new latent, rounded through the
 * cache's format, and rotary key stored at the step's position) followed by
 * the MQA-decode excerpt (mla_decode), which reads the row just written.
 * For every b with 1 <= end_pos[b] <= max_end_pos, row end_pos[b]-1 of slot
 * b receives kv_new[b] / pe_new[b] exactly as mla_cache_append would store
 * them; the decode then attends to positions 0..end_pos[b]-1.  Sequences
 * with end_pos[b] outside that range are decoded as mla_decode does (clamped,
 * flagged) and their row is not written (MLA_DEV_APPEND_SKIPPED).  With the
 * tensor-memory kernel (H = 128) the row is written inside the decode by the
 * CTA pair that reads it, so the call launches no append kernel.
 *
 *   kv_new, pe_new  device bf16 [B, 512] / [B, 64], 16-byte aligned
 *   other arguments as mla_decode (one new token per slot: B <= max_batch)
 */
MLA_API mla_status mla_decode_append(const mla_cache* cache, const void* kv_new, const void* pe_new,
                                     const void* q_latent, const void* q_pe, const int32_t* end_pos,
                                     int32_t max_end_pos, int32_t B, int32_t H, float softmax_scale,
                                     void* out, float* lse, void* workspace, size_t ws_bytes,
                                     void* stream);

/*
 * mla_topk_select -- top-k position selection per sequence: the index lists
 * that mla_decode_sparse consumes ("DeepSeek-V3.2-Exp . KV cache",
 * MQA-decode excerpt: topk_indices, one list per sequence, shared by its
 * heads).  The pages show the indexer only as a call; the selection is its
 * plainest reading, and the scores that feed it are an input here.
 *
 *   scores      device fp32 [B][max_end_pos] (row b = sequence b's score per
 *               position; row stride max_end_pos)
 *   end_pos     device int32 [B]: positions 0 .. end_pos[b]-1 compete
 *               (clamped to [0, max_end_pos])
 *   K           1 <= K <= 8192
 *   topk_idx    device int32 [B][K] (out): the K positions with the largest
 *               score, ties to the lower position, -0 equal to +0, NaN below
 *               -inf; in increasing order; fewer than K valid positions: all
 *               of them, then -1
 *
 * Errors: MLA_ERR_INVALID_ARG for null or misaligned pointers, B < 1,
 * max_end_pos < 1, K outside 1..8192.  One kernel launch on `stream`.
 */
MLA_API mla_status mla_topk_select(const float* scores, const int32_t* end_pos, int32_t B,
                                   int32_t max_end_pos, int32_t K, int32_t* topk_idx, void* stream);

/*
 * mla_selftest_decode_timeout -- self-test of the kernels' bounded waits
 *
 * Runs mla_decode (same arguments, same checks; H = 128, the tensor-memory
 * kernel) with two changes: the first unit's first tile of cache rows is
 * never loaded, and every wait in the decode kernel gives up after 2^16 polls
 * (milliseconds).  The waits on the missing tile run out, the unit's CTA pair
 * records MLA_DEV_PIPELINE_TIMEOUT in the workspace status word, drains what
 * it issued, frees its tensor memory and exits; the call completes.  Outputs
 * are unspecified; the device stays usable.  Returns MLA_ERR_UNSUPPORTED if
 * the tensor-memory kernel is not the one that would run.
 */
MLA_API mla_status mla_selftest_decode_timeout(const mla_cache* cache, const void* q_latent,
                                               const void* q_pe, const int32_t* end_pos,
                                               int32_t max_end_pos, int32_t B, int32_t H,
                                               float softmax_scale, void* out, float* lse,
                                               void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_decode_mtp -- absorbed decode of s new tokens per sequence at once
 * (multi-token decode: speculative or multi-token-prediction steps).  The s
 * new rows of cache slot b are its positions end_pos[b]-s .. end_pos[b]-1
 * (already appended); token j attends to positions 0 .. end_pos[b]-s+j:
 * causal among the step's tokens.  That is this library's reading, not a mask
 * printed on the pages -- the MQA-decode excerpt of "DeepSeek-V3.2-Exp . KV
 * cache" scores a step's tokens against all of kv_cache[:bsz, :end_pos] with
 * only the top-k index mask added; causality follows from token-by-token
 * decoding and from the `mask` argument that excerpt passes to its indexer.
 * A token with no position gets out = 0, lse = -inf.
 *
 *   q_latent    device bf16 [B, s, H, 512];  q_pe  device bf16 [B, s, H, 64]
 *   end_pos     device int32 [B]
 *   s           1 <= s <= 1024 (s = 1 is mla_decode; a large s is a prefill
 *               chunk over the cached prefix, with the same causal mask)
 *   out         device bf16 [B, s, H, 512];  lse  NULL or device fp32 [B, s, H]
 *   workspace   >= mla_workspace_size(B * s, H, max_end_pos, 0) bytes
 *   other arguments as for mla_decode (B <= cache->max_batch)
 * The B * s (sequence, token) pairs are scheduled as sequences of their own,
 * so the tokens of one slot read its rows in the same wave (the repeats come
 * from L2).
 */
MLA_API mla_status mla_decode_mtp(const mla_cache* cache, const void* q_latent, const void* q_pe,
                                  const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t s,
                                  int32_t H, float softmax_scale, void* out, float* lse,
                                  void* workspace, size_t ws_bytes, void* stream);

/*
 * mla_decode_sparse -- the same decode restricted by the DeepSeek-V3.2 top-k
 * index mask ("DeepSeek-V3.2-Exp . KV cache", MQA-decode excerpt: a tensor of
 * -inf with zeros scattered at the top-k positions is added to the scores,
 * shared by all heads).  Entries < 0 or >= end_pos[b] are skipped, repeated
 * entries count once, and only the listed rows are read.
 *
 *   topk_idx    device int32 [B, K], 1 <= K <= 8192
 *   kv_new, pe_new  NULL, or device bf16 [B, 512] / [B, 64]: first append
 *               them at row end_pos[b]-1 (the cache-write step, on the same
 *               stream), so the decode sees the newly written row.  Rows with
 *               end_pos[b]-1 outside [0, max_seq_len) are skipped and flagged
 *               (MLA_DEV_APPEND_SKIPPED).
 *   gidx_out    NULL, or device int32 [B, K]: the sorted, de-duplicated valid
 *               positions actually attended, padded with -1
 *   gcount_out  NULL, or device int32 [B]: their count
 *   workspace   >= mla_workspace_size(B, H, max_end_pos, K) bytes
 *   other arguments as for mla_decode
 * The rows are gathered by cache-row index b * max_seq_len + position, an
 * int32: B * cache->max_seq_len above 2^31 - 1 returns MLA_ERR_UNSUPPORTED.
 */
MLA_API mla_status mla_decode_sparse(const mla_cache* cache, const void* q_latent, const void* q_pe,
                             const int32_t* end_pos, int32_t max_end_pos, int32_t B, int32_t H,
                             float softmax_scale, const int32_t* topk_idx, int32_t K,
                             const void* kv_new, const void* pe_new, void* out, float* lse,
                             int32_t* gidx_out, int32_t* gcount_out, void* workspace,
                             size_t ws_bytes, void* stream);

/*
 * mla_workspace_status -- copy the device status word of a workspace used by
 * the last decode call into *flags (MLA_DEV_* bits).  Synchronises `stream`.
 */
MLA_API mla_status mla_workspace_status(const void* workspace, uint32_t* flags, void* stream);

/*
 * mla_decode_noalloc -- the dense decode of mla_decode, for callers that
 * cannot allocate device memory where they decode (for example a serving loop
 * that forbids allocations after warm-up, or a host interface that hands in
 * only the input and output buffers), and so cannot provide a workspace.  The
 * pages have no counterpart of this call.
 *
 * Instead of a caller workspace it uses one file-scope device array of
 * 32 MiB, reserved on every GPU that loads the library until the process
 * exits.  The first call on a device looks up that array's device address and
 * caches it: make that first call before starting any stream capture.  It
 * allocates nothing (no cudaMalloc, cudaFree or allocating routine).
 *
 *   arguments   as for mla_decode, without workspace and ws_bytes
 *   returns     MLA_ERR_WORKSPACE if this B and H (on this GPU's SM count)
 *               need more scratch than the 32 MiB array holds -- at H = 128 on
 *               152 SMs that is B > about 50 -- and the other MLA_ERR_* codes
 *               as mla_decode does.
 *
 * All calls share the array and leave their contents in it; each call clears
 * what must start at zero.  Calls whose GPU work overlaps (other streams, or
 * other host threads without ordering) race on it: order them.  The device
 * status word (MLA_DEV_*) of this call lives in that array and is not exposed.
 */
MLA_API mla_status mla_decode_noalloc(const mla_cache* cache, const void* q_latent,
                                      const void* q_pe, const int32_t* end_pos,
                                      int32_t max_end_pos, int32_t B, int32_t H,
                                      float softmax_scale, void* out, float* lse, void* stream);

/*
 * Tracing (no counterpart on the pages; a measurement aid).  Between
 * mla_trace_begin and mla_trace_end, on the calling host thread, every decode
 * call records a CUDA event pair around its main decode kernel on the call's
 * stream (up to max_records pairs; further calls are counted but not timed),
 * and every kernel the library launches is counted.  Calls may be captured
 * into a CUDA graph; the events then become graph nodes and are read after
 * the graph ran.  mla_trace_end synchronises on the last event and returns
 * the summed kernel time in milliseconds, the number of timed launches and
 * the number of kernel launches.  Events are created by begin and destroyed
 * by end.  max_records = 0 counts launches without recording events (an
 * event between two kernels also ends their programmatic launch overlap, so
 * a launch count of a timed run is best taken this way).  Returns
 * MLA_ERR_INVALID_ARG if tracing is already on or max_records is outside
 * [0, 2^20].
 */
MLA_API mla_status mla_trace_begin(int32_t max_records);
MLA_API mla_status mla_trace_end(float* main_kernel_ms, int32_t* timed_launches,
                                 int32_t* kernel_launches);

/*
 * mla_absorb_q -- the query side of the absorbed attention ("DeepSeek MLA
 * architecture ...", section 4: W_UK folded into the query):
 *   q_latent[b, h, c] = sum_n q_nope[b, h, n] * W_UK[h][n][c]
 * mla_project_out -- the value side (W_UV applied after the latent-space
 * attention):
 *   o[b, h, v] = sum_c W_UV[h][v][c] * x[b, h, c]
 * wkv_b is the per-head up-projection of "DeepSeek-V3.2-Exp . KV cache",
 * device bf16 [H, 256, 512]: rows 0..127 of head h are W_UK[h] (n x c), rows
 * 128..255 are W_UV[h] (v x c).
 *
 *   q_nope    device bf16 [B, H, 128]    q_latent  device bf16 [B, H, 512]
 *   x         device bf16 [B, H, 512] (e.g. the decode's out)
 *   o         device bf16 [B, H, 128]
 *   status    NULL or a device uint32 that receives MLA_DEV_PIPELINE_TIMEOUT if a
 *             bounded wait expired (the affected outputs are then not written)
 * Products accumulate in fp32 and are rounded to bf16 once.  All pointers
 * 16-byte aligned (status 4-byte), 1 <= B <= 2^22, 1 <= H <= 2^16; otherwise
 * MLA_ERR_INVALID_ARG.  Asynchronous on `stream`.
 */
MLA_API mla_status mla_absorb_q(const void* q_nope, const void* wkv_b, int32_t B, int32_t H,
                                void* q_latent, uint32_t* status, void* stream);
MLA_API mla_status mla_project_out(const void* x, const void* wkv_b, int32_t B, int32_t H, void* o,
                                   uint32_t* status, void* stream);

/*
 * mla_read_ceiling -- stream `bytes` of device memory at `buf` and XOR-fold
 * them into *sink (a measurement aid with no counterpart on the pages: the
 * HBM read rate this device achieves with plain 16-byte streaming loads, the
 * ceiling the decode's cache reads are compared with).  buf 16-byte aligned,
 * bytes a positive multiple of 16, sink a device uint32 (4-byte aligned);
 * otherwise MLA_ERR_INVALID_ARG.  Asynchronous on `stream`.
 */
MLA_API mla_status mla_read_ceiling(const void* buf, size_t bytes, uint32_t* sink, void* stream);

/* Human-readable name of a status code (static string). */
MLA_API const char* mla_status_string(mla_status status);

/* Text of the last CUDA error seen by this thread's last failing call
 * (static per-thread buffer; empty if none). */
MLA_API const char* mla_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
