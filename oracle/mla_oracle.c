/*
 * mla_oracle.c -- plain, slow, CPU reference for absorbed MLA decode over a
 * latent KV cache.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg use it; the library never calls it.  It
 * shares no code, header or table with the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [KVC]  "DeepSeek-V3.2-Exp . KV cache" (atlas.klimoza.dev): the cache
 *          write excerpt (FP8 round trip of the latent, then row writes at
 *          start_pos) and the MQA-decode excerpt (absorbed scores, top-k
 *          index mask, softmax, latent-space value sum).
 *   [ABS]  "DeepSeek MLA architecture: how Multi-Head Latent Attention cuts
 *          KV cache by 93%" (dev.to), sections 3 (decoupled RoPE: score =
 *          content term + rotary term) and 4 (matrix absorption of W_UK into
 *          the query and of W_UV after the weighted sum).
 *   [EVI]  "KV Cache Eviction Strategy in MLA ..." (instagit), section
 *          "Write-Back Logic and Position Tracking" (rows start_pos..end_pos).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - act_quant's body is not shown.  Block = 128 values; amax = max |x|;
 *     scale = fp32(amax / 448); code = e4m3(fp32(x / scale)) rounded to
 *     nearest-even with saturation to +-448.  amax == 0 gives scale 0 and
 *     all-zero codes.
 *   - The dequantised latent is bf16(fp32(e4m3_value * scale)), which is what
 *     the cache-write excerpt stores into the bf16 cache.
 *   - The cache-write excerpt passes a scale format to act_quant without
 *     defining it.  The power-of-two ("ue8m0", exponent-only) format taken
 *     here: scale = the smallest power of two >= fp32(amax / 448), so every
 *     x / scale is exact and the block still fits the e4m3 range; the codes
 *     follow as above.
 *   - Top-k entries that are negative or >= end_pos are skipped; duplicates
 *     act once (the mask is built by a scatter of zeros, which is idempotent);
 *     one index list per sequence is shared by all heads.
 *   - A sequence with no attended position yields out = 0 and lse = -inf.
 *
 * Precision: the quantiser follows the fp32 steps the page fixes; everything
 * in the attention itself is fp64.  Build with -ffp-contract=off so no step
 * is fused differently on x86-64 and aarch64.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORC_DC 512   /* kv_lora_rank: latent width                       */
#define ORC_DR 64    /* qk_rope_head_dim: rotary key width               */
#define ORC_BLK 128  /* FP8 block width along the latent                 */
#define ORC_NBLK (ORC_DC / ORC_BLK)
#define ORC_E4M3_MAX 448.0

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 bit pattern -> exact double. */
static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* fp32 -> bf16, round to nearest, ties to even, on the 16 dropped bits. */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  uint32_t upper = u >> 16, lower = u & 0xffffu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u; /* may carry into inf: correct */
  return (uint16_t)upper;
}

/* OCP FP8 E4M3 ("fn" variant): sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent field 0 holds subnormals m * 2^-9; no infinities; the only
 * NaN codes are S.1111.111; the largest finite value is 1.75 * 2^8 = 448. */
double orc_e4m3_value(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 0xf, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round y to the nearest E4M3 value (ties to the even mantissa), saturating
 * finite overflow and infinities to +-448; NaN maps to 0x7F.  All arithmetic
 * here is exact in double: y is a float, the quantum a power of two. */
uint8_t orc_e4m3_encode(float y) {
  if (isnan(y)) return 0x7f;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= ORC_E4M3_MAX) return sign | 0x7e;
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);                 /* a in [2^(e2-1), 2^e2) */
  int ex = e2 - 1;               /* floor(log2 a) */
  if (ex < -6) ex = -6;          /* below the smallest normal the spacing stays 2^-9 */
  double quantum = ldexp(1.0, ex - 3);
  double r = nearbyint(a / quantum); /* default rounding mode: nearest, ties to even */
  double v = r * quantum;        /* v <= 448 because a < 448 rounds down or onto 448 */
  if (v == 0.0) return sign;
  uint8_t code;
  if (v < ldexp(1.0, -6)) {
    code = (uint8_t)(v / ldexp(1.0, -9));             /* subnormal: m = v / 2^-9 */
  } else {
    int ev;
    frexp(v, &ev);
    int E = (ev - 1) + 7;                              /* biased exponent */
    int M = (int)((v / ldexp(1.0, ev - 1) - 1.0) * 8.0);
    code = (uint8_t)((E << 3) | M);
  }
  return sign | code;
}

/* ------------------------------------------------------------------ */
/* Cache-write step: FP8 block quantisation and its round trip [KVC]   */
/* ------------------------------------------------------------------ */

/* Smallest power of two >= s, for s > 0 (fp32 subnormals included; +inf is
 * returned as it is): frexp writes s = m * 2^e with m in [0.5, 1); s is
 * itself a power of two exactly when m == 0.5. */
static float pow2_at_least(float s) {
  if (isinf(s)) return s;
  int e;
  double m = frexp((double)s, &e);
  return (float)(m == 0.5 ? (double)s : ldexp(1.0, e));
}

/* One latent row (512 bf16) -> 512 codes + 4 fp32 scales; pow2 != 0 rounds
 * each scale up to a power of two. */
static void quantize_row(const uint16_t* x, uint8_t* q, float* scales, int pow2) {
  for (int j = 0; j < ORC_NBLK; ++j) {
    const uint16_t* xb = x + j * ORC_BLK;
    float amax = 0.0f;
    for (int i = 0; i < ORC_BLK; ++i) {
      float v = (float)fabs(bf16_to_f64(xb[i]));
      if (v > amax) amax = v;
    }
    float scale = amax / 448.0f;                 /* fp32 division */
    if (pow2 && amax > 0.0f) scale = pow2_at_least(scale);
    scales[j] = scale;
    for (int i = 0; i < ORC_BLK; ++i) {
      if (amax == 0.0f) { q[j * ORC_BLK + i] = 0; continue; }
      float y = (float)bf16_to_f64(xb[i]) / scale; /* fp32 division */
      q[j * ORC_BLK + i] = orc_e4m3_encode(y);
    }
  }
}

/* Dequantised latent element: bf16(fp32(e4m3 value * scale)). */
static uint16_t dequant_elem(uint8_t code, float scale) {
  float e = (float)orc_e4m3_value(code);       /* exact */
  float p = e * scale;                         /* fp32 multiply */
  return f32_to_bf16(p);
}

void orc_quantize_rows(const uint16_t* x, int64_t nrows, uint8_t* q, float* scales, int pow2) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r)
    quantize_row(x + r * ORC_DC, q + r * ORC_DC, scales + r * ORC_NBLK, pow2);
}

void orc_dequant_rows(const uint8_t* q, const float* scales, int64_t nrows, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < nrows; ++r)
    for (int c = 0; c < ORC_DC; ++c)
      out[r * ORC_DC + c] = dequant_elem(q[r * ORC_DC + c], scales[r * ORC_NBLK + c / ORC_BLK]);
}

void orc_e4m3_encode_array(const float* y, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(y[i]);
}

void orc_e4m3_value_array(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_value(c[i]);
}

void orc_f32_to_bf16_array(const float* f, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(f[i]);
}

/* ------------------------------------------------------------------ */
/* Attended-position set: dense = 0..T-1; sparse = valid top-k entries  */
/* ------------------------------------------------------------------ */

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Sorted, de-duplicated entries of topk[0..K) that lie in [0, T).
 * Returns the count; writes it into out[0..count). */
static int gather_list(const int32_t* topk, int K, int32_t T, int32_t* out) {
  int n = 0;
  for (int k = 0; k < K; ++k)
    if (topk[k] >= 0 && topk[k] < T) out[n++] = topk[k];
  qsort(out, (size_t)n, sizeof(int32_t), cmp_i32);
  int u = 0;
  for (int i = 0; i < n; ++i)
    if (u == 0 || out[i] != out[u - 1]) out[u++] = out[i];
  return u;
}

void orc_sparse_gather_lists(const int32_t* topk, int B, int K, const int32_t* end_pos,
                             int32_t* gidx, int32_t* gcount) {
  for (int b = 0; b < B; ++b) {
    int32_t* g = gidx + (int64_t)b * K;
    int n = gather_list(topk + (int64_t)b * K, K, end_pos[b], g);
    for (int i = n; i < K; ++i) g[i] = -1;
    gcount[b] = n;
  }
}

/* ------------------------------------------------------------------ */
/* Absorbed decode [KVC MQA-decode excerpt; ABS sections 3-4]           */
/* ------------------------------------------------------------------ */

/* Cache view.  fmt 0: kv is bf16 bits [Bmax, S, 512]; fmt 1 and 2: kv is
 * e4m3 codes [Bmax, S, 512] with kv_scale fp32 [Bmax, S, 4] (fmt 2's scales
 * are powers of two; reading them is the same).  pe is bf16 bits
 * [Bmax, S, 64] in every format. */
typedef struct {
  int fmt;
  int64_t S;
  const void* kv;
  const float* kv_scale;
  const uint16_t* pe;
} orc_cache;

/* Latent row t of sequence b as exact doubles (the values the decode
 * attends to: the bf16 cache entry, or the FP8 round trip). */
static void latent_row(const orc_cache* c, int b, int64_t t, double* row) {
  int64_t r = (int64_t)b * c->S + t;
  if (c->fmt == 0) {
    const uint16_t* kv = (const uint16_t*)c->kv + r * ORC_DC;
    for (int i = 0; i < ORC_DC; ++i) row[i] = bf16_to_f64(kv[i]);
  } else {
    const uint8_t* kv = (const uint8_t*)c->kv + r * ORC_DC;
    const float* sc = c->kv_scale + r * ORC_NBLK;
    for (int i = 0; i < ORC_DC; ++i) row[i] = bf16_to_f64(dequant_elem(kv[i], sc[i / ORC_BLK]));
  }
}

/*
 * For each requested (b, h): positions P = {0..T_b-1} (dense) or the valid
 * top-k set (sparse); s_t = sigma * (q_latent[b,h] . c_t + q_pe[b,h] . kR_t);
 * w = softmax(s) over P; out = sum_t w_t c_t (latent space); lse = log sum
 * exp(s_t).  Queries are given in fp64 so exact absorbed queries can be fed
 * in; the bf16 wrapper in Python converts bf16 inputs exactly.
 *
 * q_latent [Bq, H, 512], q_pe [Bq, H, 64] (fp64); pairs [npairs, 2] = (b, h);
 * out [npairs, 512]; lse [npairs]; w_out (optional) [npairs, wstride] holds
 * the weight of every position t < min(T_b, wstride) (0 where not attended).
 */
int orc_decode_absorbed(int fmt, int64_t S, const void* kv, const float* kv_scale,
                        const uint16_t* pe, const double* q_latent, const double* q_pe, int H,
                        const int32_t* end_pos, const int32_t* topk, int K, double sigma,
                        const int32_t* pairs, int npairs, double* out, double* lse,
                        double* w_out, int64_t wstride) {
  orc_cache c = {fmt, S, kv, kv_scale, pe};
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int p = 0; p < npairs; ++p) {
    int b = pairs[2 * p], h = pairs[2 * p + 1];
    int32_t T = end_pos[b];
    if (T > S) T = (int32_t)S;
    size_t cap = (size_t)(T > 0 ? T : 1) + (size_t)(K > 0 ? K : 1);
    int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * cap);
    double* s = (double*)malloc(sizeof(double) * cap);
    double row[ORC_DC];
    if (!pos || !s) {
#pragma omp atomic write
      err = 1;
      free(pos);
      free(s);
      continue;
    }
    int n;
    if (topk) {
      n = gather_list(topk + (int64_t)b * K, K, T, pos);
    } else {
      n = T > 0 ? T : 0;
      for (int t = 0; t < n; ++t) pos[t] = t;
    }
    const double* qL = q_latent + ((int64_t)b * H + h) * ORC_DC;
    const double* qP = q_pe + ((int64_t)b * H + h) * ORC_DR;
    double* o = out + (int64_t)p * ORC_DC;
    for (int i = 0; i < ORC_DC; ++i) o[i] = 0.0;
    if (w_out)
      for (int64_t t = 0; t < wstride; ++t) w_out[(int64_t)p * wstride + t] = 0.0;
    if (n == 0) { lse[p] = -INFINITY; free(pos); free(s); continue; }
    /* scores: content term in the latent space + rotary term */
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) {
      int64_t t = pos[i];
      latent_row(&c, b, t, row);
      const uint16_t* kR = pe + ((int64_t)b * S + t) * ORC_DR;
      double acc_c = 0.0, acc_r = 0.0;
      for (int j = 0; j < ORC_DC; ++j) acc_c += qL[j] * row[j];
      for (int j = 0; j < ORC_DR; ++j) acc_r += qP[j] * bf16_to_f64(kR[j]);
      s[i] = sigma * (acc_c + acc_r);
      if (s[i] > m) m = s[i];
    }
    /* softmax over the attended positions */
    double z = 0.0;
    for (int i = 0; i < n; ++i) z += exp(s[i] - m);
    lse[p] = m + log(z);
    /* value sum in latent space */
    for (int i = 0; i < n; ++i) {
      double w = exp(s[i] - m) / z;
      latent_row(&c, b, pos[i], row);
      for (int j = 0; j < ORC_DC; ++j) o[j] += w * row[j];
      if (w_out && pos[i] < wstride) w_out[(int64_t)p * wstride + pos[i]] = w;
    }
    free(pos);
    free(s);
  }
  return err;
}

/*
 * Naive (non-absorbed) multi-head attention over the same cache, used only
 * to check the absorption identity [ABS section 4]: per head the latent is
 * expanded to keys k_t = W_UK[h] c_t (128) and values v_t = W_UV[h] c_t
 * (128); the query is [q_nope ; q_pe] and the rotary key k_R is shared by all
 * heads [ABS section 3].  wkv_b [H, 256, 512]: rows 0..127 are W_UK[h], rows
 * 128..255 are W_UV[h] (the split of wkv_b in the MQA-decode excerpt).
 * Dense only.  q_nope [B, H, 128], q_pe [B, H, 64]; o [B, H, 128]; lse [B, H].
 */
int orc_decode_naive(int fmt, int64_t S, const void* kv, const float* kv_scale,
                     const uint16_t* pe, const double* wkv_b, const double* q_nope,
                     const double* q_pe, int B, int H, const int32_t* end_pos, double sigma,
                     double* o, double* lse) {
  orc_cache c = {fmt, S, kv, kv_scale, pe};
  const int DN = 128, DV = 128;
  for (int b = 0; b < B; ++b) {
    int32_t T = end_pos[b] < S ? end_pos[b] : (int32_t)S;
    for (int h = 0; h < H; ++h) {
      const double* Wuk = wkv_b + (int64_t)h * 256 * ORC_DC;
      const double* Wuv = Wuk + (int64_t)128 * ORC_DC;
      const double* qn = q_nope + ((int64_t)b * H + h) * DN;
      const double* qp = q_pe + ((int64_t)b * H + h) * ORC_DR;
      double* oh = o + ((int64_t)b * H + h) * DV;
      for (int d = 0; d < DV; ++d) oh[d] = 0.0;
      if (T <= 0) { lse[b * H + h] = -INFINITY; continue; }
      double* s = (double*)malloc(sizeof(double) * (size_t)T);
      double* v = (double*)malloc(sizeof(double) * (size_t)T * DV);
      if (!s || !v) { free(s); free(v); return 1; }
      double row[ORC_DC];
      double m = -INFINITY;
      for (int t = 0; t < T; ++t) {
        latent_row(&c, b, t, row);
        double dot = 0.0;
        for (int d = 0; d < DN; ++d) {
          double k = 0.0;
          for (int j = 0; j < ORC_DC; ++j) k += Wuk[(int64_t)d * ORC_DC + j] * row[j];
          dot += qn[d] * k;
        }
        const uint16_t* kR = pe + ((int64_t)b * S + t) * ORC_DR;
        for (int r = 0; r < ORC_DR; ++r) dot += qp[r] * bf16_to_f64(kR[r]);
        s[t] = sigma * dot;
        if (s[t] > m) m = s[t];
        for (int d = 0; d < DV; ++d) {
          double vv = 0.0;
          for (int j = 0; j < ORC_DC; ++j) vv += Wuv[(int64_t)d * ORC_DC + j] * row[j];
          v[(int64_t)t * DV + d] = vv;
        }
      }
      double z = 0.0;
      for (int t = 0; t < T; ++t) z += exp(s[t] - m);
      for (int t = 0; t < T; ++t) {
        double w = exp(s[t] - m) / z;
        for (int d = 0; d < DV; ++d) oh[d] += w * v[(int64_t)t * DV + d];
      }
      lse[b * H + h] = m + log(z);
      free(s);
      free(v);
    }
  }
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads of the OpenMP loops that follow (timing only; results do not
 * depend on it). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
