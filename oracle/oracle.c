/*
 * CPU oracle of one routed NVFP4 MoE decode layer-step -- TEST
 * INFRASTRUCTURE ONLY (tests, the smoke check and the bench's CPU-baseline
 * leg).  Plain loops, fp64 accumulation, one output element per loop
 * iteration; OpenMP only spreads independent output elements over cores, each
 * reduction runs sequentially in index order.  See oracle.h for the contract.
 *
 * Sources the arithmetic follows:
 *  - The step's structure: the decode executor page
 *    (vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode), module
 *    docstring "One step of b rows" (attention boundary: dual norm into the
 *    stream and the MoE input; MoE: router -> routing -> pooler -> routed
 *    experts -> tail -> unpooler; final: last gather + dual norm), and
 *    SpecializedDecode.build (fp32 stream buffer, bf16 MoE input buffer).
 *  - The dual norm's shape: the DSpark page
 *    (vllm.models.muse_spark.common.dspark), MuseSparkDSparkDecoderLayer
 *    .forward: stream = add(stream, post_norm(branch)), ffn input =
 *    pre_ffn_norm(stream).
 *  - RMSNorm: x * rsqrt(mean(x^2) + eps) * weight (the same page's fp32
 *    K-norm in precompute_and_store_context_kv).
 *  - Element formats: OCP Microscaling Formats (MX) v1.0, section 5.3.3
 *    (FP4 E2M1: bias 1, max 6) and OCP 8-bit Floating Point (OFP8) v1.0
 *    (E4M3: bias 7, no infinities, max 448).
 *  - NVFP4 two-level scaling (e4m3 scale per 16 elements, fp32 per-tensor
 *    scale = amax / (6 * 448)) and the SiLU-gated expert MLP: the stated
 *    number format and block of the routed decode workload, which the pages
 *    name but do not print; their order of operations is a reading recorded
 *    with the design notes.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ formats */

double oracle_e2m1_decode(uint8_t code) {
  /* sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0 */
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

uint8_t oracle_e2m1_encode(float v) {
  uint8_t s = signbit(v) ? 8u : 0u;
  double a = fabs((double)v);
  if (a >= 6.0) return (uint8_t)(s | 7u); /* saturate to the largest finite magnitude */
  int best = 0;
  double bd = a;
  for (int c = 1; c < 8; ++c) {
    double d = fabs(a - oracle_e2m1_decode((uint8_t)c));
    /* nearest; on a tie the code with an even mantissa bit wins */
    if (d < bd || (d == bd && (c & 1) == 0)) {
      best = c;
      bd = d;
    }
  }
  return (uint8_t)(s | best);
}

double oracle_e4m3_decode(uint8_t code) {
  /* sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0; S.1111.111 is NaN */
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7)
    mag = NAN;
  else if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

uint8_t oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t s = signbit(v) ? 0x80u : 0u;
  double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(s | 0x7E); /* saturate to 448 */
  int ex = 0;
  int e = -6; /* the subnormals share the quantum of the lowest binade */
  if (a > 0) {
    frexp(a, &ex);
    if (ex - 1 > e) e = ex - 1;
  }
  double q = ldexp(1.0, e - 3);  /* 3 mantissa bits */
  double n = nearbyint(a / q);   /* a / q is exact; ties to even */
  double val = n * q;
  if (val == 0.0) return s;
  if (val < ldexp(1.0, -6)) return (uint8_t)(s | (uint8_t)(val / ldexp(1.0, -9)));
  frexp(val, &ex);
  e = ex - 1;
  int m = (int)(val / ldexp(1.0, e) * 8.0) - 8;
  return (uint8_t)(s | (uint8_t)(((e + 7) << 3) | m));
}

uint16_t oracle_bf16_from_double(double v) {
  /* bf16: 8 significant bits, the fp32 exponent range */
  if (isnan(v)) return 0x7FC0;
  uint16_t s = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (a == 0.0) return s;
  int ex = 0;
  frexp(a, &ex);
  int e = ex - 1;
  if (e < -126) e = -126;
  double q = ldexp(1.0, e - 7);
  double val = nearbyint(a / q) * q;
  if (val >= ldexp(1.0, 128)) return (uint16_t)(s | 0x7F80u);
  float f = (float)val; /* exact: val is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(s | (uint16_t)((u >> 16) & 0x7FFFu));
}

double oracle_bf16_decode(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ---------------------------------------------------------------- quantizer */

void oracle_nvfp4_quantize(const float* v, int64_t rows, int64_t cols, uint8_t* codes,
                           uint8_t* sf, float* sg_out, float* amax_out) {
  float amax = 0.0f;
  for (int64_t i = 0; i < rows * cols; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  float sg = amax / 2688.0f; /* 2688 = 6 * 448, fp32 division */
  int64_t nb = cols / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* blk = v + r * cols + b * 16;
      float ab = 0.0f;
      for (int i = 0; i < 16; ++i) {
        float a = fabsf(blk[i]);
        if (a > ab) ab = a;
      }
      uint8_t sb = 0;
      float d = 0.0f;
      if (sg > 0.0f) {
        float q = ab / 6.0f;
        float t = q / sg;
        sb = oracle_e4m3_encode(t);
        d = (float)oracle_e4m3_decode(sb) * sg;
      }
      sf[r * nb + b] = sb;
      uint8_t* out = codes + r * (cols / 2) + b * 8;
      for (int i = 0; i < 8; ++i) {
        uint8_t lo = 0, hi = 0;
        if (d > 0.0f) {
          lo = oracle_e2m1_encode(blk[2 * i] / d);
          hi = oracle_e2m1_encode(blk[2 * i + 1] / d);
        }
        out[i] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
  if (sg_out) *sg_out = sg;
  if (amax_out) *amax_out = amax;
}

static double dequant_one(const uint8_t* codes, const uint8_t* sf, float sg, int64_t cols,
                          int64_t r, int64_t c) {
  uint8_t byte = codes[r * (cols / 2) + c / 2];
  uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
  return oracle_e2m1_decode(code) * oracle_e4m3_decode(sf[r * (cols / 16) + c / 16]) * (double)sg;
}

void oracle_nvfp4_dequantize(const uint8_t* codes, const uint8_t* sf, float sg, int64_t rows,
                             int64_t cols, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) out[r * cols + c] = dequant_one(codes, sf, sg, cols, r, c);
}

/* ----------------------------------------------------------------- boundary */

void oracle_boundary(int rows, int H, double eps, const double* branch, float* stream,
                     const float* w_post, const float* w_pre, uint16_t* x, double* x_exact) {
  for (int r = 0; r < rows; ++r) {
    const double* br = branch + (int64_t)r * H;
    float* s = stream + (int64_t)r * H;
    double ms = 0.0;
    for (int h = 0; h < H; ++h) ms += br[h] * br[h];
    ms /= H;
    double inv = 1.0 / sqrt(ms + eps);
    for (int h = 0; h < H; ++h) s[h] = (float)((double)s[h] + br[h] * inv * (double)w_post[h]);
    double ms2 = 0.0;
    for (int h = 0; h < H; ++h) ms2 += (double)s[h] * (double)s[h];
    ms2 /= H;
    double inv2 = 1.0 / sqrt(ms2 + eps);
    for (int h = 0; h < H; ++h) {
      double xe = (double)s[h] * inv2 * (double)w_pre[h];
      if (x_exact) x_exact[(int64_t)r * H + h] = xe;
      x[(int64_t)r * H + h] = oracle_bf16_from_double(xe);
    }
  }
}

/* The first layer's front (decode page, module docstring "One step of b
 * rows": the embedded tokens into the stream (fp32) and its
 * pre_qkv_proj_norm into the attention input): stream = the embedded bf16
 * values, exactly; out = bf16(stream / sqrt(mean(stream^2) + eps) * w). */
void oracle_front(int rows, int H, double eps, const uint16_t* embedded, const float* w,
                  float* stream, uint16_t* out, double* out_exact) {
  for (int r = 0; r < rows; ++r) {
    float* s = stream + (int64_t)r * H;
    double ms = 0.0;
    for (int h = 0; h < H; ++h) {
      s[h] = (float)oracle_bf16_decode(embedded[(int64_t)r * H + h]);
      ms += (double)s[h] * (double)s[h];
    }
    ms /= H;
    double inv_front = 1.0 / sqrt(ms + eps);
    for (int h = 0; h < H; ++h) {
      double xe = (double)s[h] * inv_front * (double)w[h];
      if (out_exact) out_exact[(int64_t)r * H + h] = xe;
      out[(int64_t)r * H + h] = oracle_bf16_from_double(xe);
    }
  }
}

/* out[m][n] = bf16(sum_k A[m][k] B[n][k]) over bf16 operands (a projection
 * y = W x with W [N][K] row-major and x [M][K]), summed in fp64; the sum
 * before its rounding goes to exact[m][n] when exact is not NULL. */
void oracle_bf16_linear(int M, int N, int K, const uint16_t* A, const uint16_t* B, uint16_t* out,
                        double* exact) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int m = 0; m < M; ++m) {
    for (int n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k)
        acc += oracle_bf16_decode(A[(int64_t)m * K + k]) * oracle_bf16_decode(B[(int64_t)n * K + k]);
      out[(int64_t)m * N + n] = oracle_bf16_from_double(acc);
      if (exact) exact[(int64_t)m * N + n] = acc;
    }
  }
}

/* a[r][j] = bf16(silu(g) * u) with g = gu[r][j] and u = gu[r][I + j] (the
 * gate half, then the up half of one gate_up_proj output row). */
void oracle_silu_mul(int rows, int I, const uint16_t* gu, uint16_t* a, double* exact) {
  for (int r = 0; r < rows; ++r)
    for (int j = 0; j < I; ++j) {
      double g = oracle_bf16_decode(gu[(int64_t)r * 2 * I + j]);
      double u = oracle_bf16_decode(gu[(int64_t)r * 2 * I + I + j]);
      double v = g / (1.0 + exp(-g)) * u;
      a[(int64_t)r * I + j] = oracle_bf16_from_double(v);
      if (exact) exact[(int64_t)r * I + j] = v;
    }
}

/* One dense draft layer's MLP block (the DSpark page,
 * MuseSparkDSparkDecoderLayer.forward): the attention output through
 * post_attn_norm into the fp32 stream; the feed-forward input is
 * pre_ffn_norm of the stream after a cast to bf16, the draft's compute type
 * (the layer casts the stream before every input norm); the gated MLP (gate_proj /
 * up_proj as shards 0 / 1 of gate_up_proj) in bf16: each projection's
 * output rounded to bf16, silu(gate) * up rounded to bf16, the down
 * projection rounded to bf16; its output through post_ffn_norm into the
 * stream.  Sums in fp64 over the exact bf16 operands.  x_exact (nullable)
 * receives the MLP input before its bf16 rounding. */
void oracle_dense_layer(int rows, int H, int I, double eps, const uint16_t* attn_out,
                        float* stream, const float* w_post_attn, const float* w_pre_ffn,
                        const uint16_t* w13, const uint16_t* w2, const float* w_post_ffn,
                        uint16_t* x, uint16_t* gu, uint16_t* a, uint16_t* f, double* x_exact) {
  double* br = (double*)malloc(sizeof(double) * H);
  double* t = (double*)malloc(sizeof(double) * H);
  for (int r = 0; r < rows; ++r) {
    float* s = stream + (int64_t)r * H;
    /* s1 = s + rmsnorm(attn_out) * w_post_attn */
    double ms = 0.0;
    for (int h = 0; h < H; ++h) {
      br[h] = oracle_bf16_decode(attn_out[(int64_t)r * H + h]);
      ms += br[h] * br[h];
    }
    double inv_attn = 1.0 / sqrt(ms / H + eps);
    for (int h = 0; h < H; ++h) s[h] = (float)((double)s[h] + br[h] * inv_attn * (double)w_post_attn[h]);
    /* x = bf16(rmsnorm(bf16(s1)) * w_pre_ffn) */
    double ms_ffn = 0.0;
    for (int h = 0; h < H; ++h) {
      t[h] = oracle_bf16_decode(oracle_bf16_from_double((double)s[h]));
      ms_ffn += t[h] * t[h];
    }
    double inv_ffn = 1.0 / sqrt(ms_ffn / H + eps);
    for (int h = 0; h < H; ++h) {
      double v = t[h] * inv_ffn * (double)w_pre_ffn[h];
      x[(int64_t)r * H + h] = oracle_bf16_from_double(v);
      if (x_exact) x_exact[(int64_t)r * H + h] = v;
    }
  }
  /* the gated MLP */
  oracle_bf16_linear(rows, 2 * I, H, x, w13, gu, NULL);
  oracle_silu_mul(rows, I, gu, a, NULL);
  oracle_bf16_linear(rows, H, I, a, w2, f, NULL);
  /* s2 = s1 + rmsnorm(f) * w_post_ffn */
  for (int r = 0; r < rows; ++r) {
    float* s = stream + (int64_t)r * H;
    double ms = 0.0;
    for (int h = 0; h < H; ++h) {
      br[h] = oracle_bf16_decode(f[(int64_t)r * H + h]);
      ms += br[h] * br[h];
    }
    double inv_out = 1.0 / sqrt(ms / H + eps);
    for (int h = 0; h < H; ++h) s[h] = (float)((double)s[h] + br[h] * inv_out * (double)w_post_ffn[h]);
  }
  free(br);
  free(t);
}

/* The draft's context-KV projection (the DSpark page, _project_muse_context_kv
 * and precompute_and_store_context_kv).
 *
 * Norms: fc = bf16(rmsnorm(ctx) * w_hidden) (hidden_norm), then each layer's
 * pre_qkv_proj_norm of fc: u[l] = bf16(rmsnorm(fc) * w_pre[l]).  The weights
 * are the effective ones (a zero-centred gamma is passed as 1 + gamma). */
void oracle_layer_norms(int n, int H, int L, double eps, const uint16_t* fc, const float* w_pre,
                        uint16_t* u, double* u_exact) {
  for (int r = 0; r < n; ++r) {
    const uint16_t* f = fc + (int64_t)r * H;
    double ms_fc = 0.0;
    for (int h = 0; h < H; ++h) ms_fc += oracle_bf16_decode(f[h]) * oracle_bf16_decode(f[h]);
    double inv_pre = 1.0 / sqrt(ms_fc / H + eps);
    for (int l = 0; l < L; ++l)
      for (int h = 0; h < H; ++h) {
        double v = oracle_bf16_decode(f[h]) * inv_pre * (double)w_pre[(int64_t)l * H + h];
        int64_t o = ((int64_t)l * n + r) * H + h;
        u[o] = oracle_bf16_from_double(v);
        if (u_exact) u_exact[o] = v;
      }
  }
}

void oracle_ctx_norms(int n, int H, int L, double eps, const uint16_t* ctx, const float* w_hidden,
                      const float* w_pre, uint16_t* fc, uint16_t* u, double* fc_exact, double* u_exact) {
  for (int r = 0; r < n; ++r) {
    const uint16_t* c = ctx + (int64_t)r * H;
    double ms = 0.0;
    for (int h = 0; h < H; ++h) ms += oracle_bf16_decode(c[h]) * oracle_bf16_decode(c[h]);
    double inv_hidden = 1.0 / sqrt(ms / H + eps);
    for (int h = 0; h < H; ++h) {
      double v = oracle_bf16_decode(c[h]) * inv_hidden * (double)w_hidden[h];
      fc[(int64_t)r * H + h] = oracle_bf16_from_double(v);
      if (fc_exact) fc_exact[(int64_t)r * H + h] = v;
    }
  }
  oracle_layer_norms(n, H, L, eps, fc, w_pre, u, u_exact);
}

/* The keys' RMSNorm and rotary embedding.  kv [L][n][2*KVH*D] holds each
 * layer's projection (the K heads, then the V heads).  Each K head of D
 * values is normalised in fp32 without a weight, k = bf16(k / sqrt(mean(k^2)
 * + qk_eps)), then rotated by its row's position: the rotary embedding of
 * RoFormer (Su et al., 2021) with the dimensions paired as (j, j + D/2) and
 * angle pos * theta^(-2j/D), each output rounded to bf16 once.  theta = 0
 * leaves the keys unrotated.  V passes through.  k_exact (nullable) gets the
 * rotated keys before their rounding, kn_exact (nullable) the normalised keys
 * before theirs. */
void oracle_k_norm_rope(int L, int n, int KVH, int D, double qk_eps, double theta,
                        const int64_t* positions, const uint16_t* kv, uint16_t* k_out,
                        uint16_t* v_out, double* k_exact, double* kn_exact) {
  const int KD = KVH * D, half = D / 2;
  double* kn = (double*)malloc(sizeof(double) * D);
  for (int l = 0; l < L; ++l)
    for (int r = 0; r < n; ++r) {
      const uint16_t* row = kv + ((int64_t)l * n + r) * 2 * KD;
      for (int hd = 0; hd < KVH; ++hd) {
        const uint16_t* k = row + hd * D;
        int64_t o = (((int64_t)l * n + r) * KVH + hd) * D;
        double ms = 0.0;
        for (int i = 0; i < D; ++i) ms += oracle_bf16_decode(k[i]) * oracle_bf16_decode(k[i]);
        double inv = 1.0 / sqrt(ms / D + qk_eps);
        for (int i = 0; i < D; ++i) kn[i] = oracle_bf16_decode(oracle_bf16_from_double(oracle_bf16_decode(k[i]) * inv));
        if (kn_exact)
          for (int i = 0; i < D; ++i) kn_exact[o + i] = oracle_bf16_decode(k[i]) * inv;
        for (int j = 0; j < half; ++j) {
          double x1 = kn[j], x2 = kn[j + half], y1 = x1, y2 = x2;
          if (theta > 0.0) {
            double ang = (double)positions[r] * pow(theta, -2.0 * j / D);
            y1 = x1 * cos(ang) - x2 * sin(ang);
            y2 = x2 * cos(ang) + x1 * sin(ang);
          }
          k_out[o + j] = oracle_bf16_from_double(y1);
          k_out[o + j + half] = oracle_bf16_from_double(y2);
          if (k_exact) {
            k_exact[o + j] = y1;
            k_exact[o + j + half] = y2;
          }
        }
        memcpy(v_out + o, row + KD + hd * D, sizeof(uint16_t) * D);
      }
    }
  free(kn);
}

/* The cache update: layer l's rows go to cache[l][slot][KVH][D] for slot =
 * slots[l * layer_stride + r]; a negative slot writes nothing. */
void oracle_kv_cache_write(int L, int n, int KVH, int D, const int64_t* slots, int layer_stride,
                           int64_t n_slots, const uint16_t* k, const uint16_t* v, uint16_t* k_cache,
                           uint16_t* v_cache) {
  const int64_t KD = (int64_t)KVH * D;
  for (int l = 0; l < L; ++l)
    for (int r = 0; r < n; ++r) {
      int64_t slot = slots[(int64_t)l * layer_stride + r];
      if (slot < 0 || slot >= n_slots) continue;
      memcpy(k_cache + ((int64_t)l * n_slots + slot) * KD, k + ((int64_t)l * n + r) * KD, sizeof(uint16_t) * KD);
      memcpy(v_cache + ((int64_t)l * n_slots + slot) * KD, v + ((int64_t)l * n + r) * KD, sizeof(uint16_t) * KD);
    }
}

/* ------------------------------------------------------------------ routing */

static void softmax_row(int E, const double* logit, double* p) {
  double m = logit[0];
  for (int e = 1; e < E; ++e)
    if (logit[e] > m) m = logit[e];
  double z = 0.0;
  for (int e = 0; e < E; ++e) {
    p[e] = exp(logit[e] - m);
    z += p[e];
  }
  for (int e = 0; e < E; ++e) p[e] /= z;
}

/* The n largest of p[0..E), largest first, ties to the lower index. */
static void top_n(int E, const double* p, int n, int32_t* sel) {
  for (int s = 0; s < n; ++s) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      int taken = 0;
      for (int t = 0; t < s; ++t)
        if (sel[t] == e) taken = 1;
      if (taken) continue;
      if (best < 0 || p[e] > p[best]) best = e;
    }
    sel[s] = best;
  }
}

void oracle_route(int rows, int H, int E, int k, const uint16_t* x, const uint16_t* router_w,
                  const float* bias, double* logits, double* probs, int32_t* ids, double* gates,
                  uint8_t* flags, double* gap) {
  double* lg = (double*)malloc(sizeof(double) * E);
  double* p = (double*)malloc(sizeof(double) * E);
  int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (k + 1));
  for (int r = 0; r < rows; ++r) {
    const uint16_t* xr = x + (int64_t)r * H;
    for (int e = 0; e < E; ++e) {
      const uint16_t* we = router_w + (int64_t)e * H;
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += oracle_bf16_decode(xr[h]) * oracle_bf16_decode(we[h]);
      if (bias) acc += (double)bias[e];
      lg[e] = acc;
    }
    softmax_row(E, lg, p);
    int n = (k < E) ? k + 1 : k;
    top_n(E, p, n, sel);
    double sum = 0.0;
    for (int s = 0; s < k; ++s) sum += p[sel[s]];
    for (int s = 0; s < k; ++s) {
      ids[r * k + s] = sel[s];
      gates[r * k + s] = p[sel[s]] / sum;
    }
    double g = (k < E) ? p[sel[k - 1]] - p[sel[k]] : INFINITY;
    flags[r] = (uint8_t)(g < 1e-6);
    if (gap) gap[r] = g;
    if (logits) memcpy(logits + (int64_t)r * E, lg, sizeof(double) * E);
    if (probs) memcpy(probs + (int64_t)r * E, p, sizeof(double) * E);
  }
  free(lg);
  free(p);
  free(sel);
}

/* ------------------------------------------------------------------- pooler */

void oracle_pool(int rows, int E, int k, const int32_t* ids, int32_t* count, int32_t* offset,
                 int32_t* pair_order, int32_t* active, int32_t* n_active) {
  for (int e = 0; e < E; ++e) count[e] = 0;
  for (int p = 0; p < rows * k; ++p) count[ids[p]] += 1;
  offset[0] = 0;
  for (int e = 0; e < E; ++e) offset[e + 1] = offset[e] + count[e];
  int pos = 0;
  for (int e = 0; e < E; ++e)
    for (int r = 0; r < rows; ++r)
      for (int s = 0; s < k; ++s)
        if (ids[r * k + s] == e) pair_order[pos++] = r * k + s;
  int na = 0;
  for (int e = 0; e < E; ++e)
    if (count[e] > 0) active[na++] = e;
  *n_active = na;
}

/* ------------------------------------------------------------------ experts */

static double silu(double z) { return z / (1.0 + exp(-z)); }

int oracle_gate_up(int rows, int H, int E, int k, int I, const oracle_layer_weights* w,
                   const uint8_t* x_codes, const uint8_t* x_sf, float x_sg, const int32_t* ids,
                   const int32_t* offset, const int32_t* pair_order, float* h) {
  (void)E;
  (void)offset;
  int npairs = rows * k;
  for (int pos = 0; pos < npairs; ++pos) {
    int e = ids[pair_order[pos]];
    if (!w->w13[e] || !w->w13_sf[e]) return -1; /* an active expert's weights are missing */
  }
  double* xh = (double*)malloc(sizeof(double) * (size_t)rows * H);
  oracle_nvfp4_dequantize(x_codes, x_sf, x_sg, rows, H, xh);
#pragma omp parallel for collapse(2) schedule(static)
  for (int pos = 0; pos < npairs; ++pos) {
    for (int j = 0; j < I; ++j) {
      int p = pair_order[pos];
      int r = p / k, e = ids[p];
      const uint8_t* c13 = w->w13[e];
      const uint8_t* s13 = w->w13_sf[e];
      float sg_gate = w->gscale[3 * e + 0], sg_up = w->gscale[3 * e + 1];
      const double* xr = xh + (int64_t)r * H;
      double G = 0.0, U = 0.0;
      for (int hh = 0; hh < H; ++hh) {
        G += dequant_one(c13, s13, sg_gate, H, j, hh) * xr[hh];
        U += dequant_one(c13, s13, sg_up, H, I + j, hh) * xr[hh];
      }
      h[(int64_t)pos * I + j] = (float)(silu(G) * U);
    }
  }
  free(xh);
  return 0;
}

void oracle_h_quant(int E, int I, const int32_t* offset, const float* h, uint8_t* h_codes,
                    uint8_t* h_sf, float* h_sg, float* h_amax) {
  for (int e = 0; e < E; ++e) {
    int n = offset[e + 1] - offset[e];
    h_sg[e] = 0.0f;
    h_amax[e] = 0.0f;
    if (n == 0) continue;
    oracle_nvfp4_quantize(h + (int64_t)offset[e] * I, n, I, h_codes + (int64_t)offset[e] * (I / 2),
                          h_sf + (int64_t)offset[e] * (I / 16), &h_sg[e], &h_amax[e]);
  }
}

int oracle_down(int rows, int H, int E, int k, int I, const oracle_layer_weights* w,
                const int32_t* ids, const int32_t* offset, const int32_t* pair_order,
                const uint8_t* h_codes, const uint8_t* h_sf, const float* h_sg, float* o) {
  (void)E;
  (void)offset;
  int npairs = rows * k;
  for (int pos = 0; pos < npairs; ++pos) {
    int e = ids[pair_order[pos]];
    if (!w->w2[e] || !w->w2_sf[e]) return -1;
  }
  double* hh = (double*)malloc(sizeof(double) * (size_t)npairs * I);
  /* each pooled row is dequantized with its expert's global scale */
  for (int pos = 0; pos < npairs; ++pos) {
    int e = ids[pair_order[pos]];
    oracle_nvfp4_dequantize(h_codes + (int64_t)pos * (I / 2), h_sf + (int64_t)pos * (I / 16),
                            h_sg[e], 1, I, hh + (int64_t)pos * I);
  }
#pragma omp parallel for collapse(2) schedule(static)
  for (int pos = 0; pos < npairs; ++pos) {
    for (int i = 0; i < H; ++i) {
      int p = pair_order[pos];
      int e = ids[p];
      float sg_down = w->gscale[3 * e + 2];
      const double* hr = hh + (int64_t)pos * I;
      double acc = 0.0;
      for (int j = 0; j < I; ++j) acc += dequant_one(w->w2[e], w->w2_sf[e], sg_down, I, i, j) * hr[j];
      o[(int64_t)p * H + i] = (float)acc;
    }
  }
  free(hh);
  return 0;
}

void oracle_gather(int rows, int H, int k, const double* gates, const float* o, double* y) {
  for (int r = 0; r < rows; ++r)
    for (int hh = 0; hh < H; ++hh) {
      double acc = 0.0;
      for (int s = 0; s < k; ++s) acc += gates[r * k + s] * (double)o[((int64_t)r * k + s) * H + hh];
      y[(int64_t)r * H + hh] = acc;
    }
}

/* ---------------------------------------------------------------- one layer */

/* The MoE part of a layer from its bf16 input out->x (already filled): the
   routing (optionally with the given ids), the pooler, the input's NVFP4
   quantization and the experts. */
int oracle_moe_step(int rows, int H, int E, int k, int I, const oracle_layer_weights* w,
                    const int32_t* forced_ids, oracle_layer_out* out) {
  double* p = (double*)malloc(sizeof(double) * (size_t)rows * E);
  oracle_route(rows, H, E, k, out->x, w->router_w, w->router_bias, NULL, p, out->ids, out->gates,
               out->flags, out->gap);
  if (forced_ids) {
    /* the gates of the given ids: their probabilities, renormalised */
    for (int r = 0; r < rows; ++r) {
      double sum = 0.0;
      for (int s = 0; s < k; ++s) sum += p[(int64_t)r * E + forced_ids[r * k + s]];
      for (int s = 0; s < k; ++s) {
        out->ids[r * k + s] = forced_ids[r * k + s];
        out->gates[r * k + s] = p[(int64_t)r * E + forced_ids[r * k + s]] / sum;
      }
    }
  }
  if (out->probs) memcpy(out->probs, p, sizeof(double) * (size_t)rows * E);
  free(p);
  oracle_pool(rows, E, k, out->ids, out->count, out->offset, out->pair_order, out->active,
              out->n_active);
  /* the MoE input as one NVFP4 tensor [rows, H] */
  float* xf = (float*)malloc(sizeof(float) * (size_t)rows * H);
  for (int64_t i = 0; i < (int64_t)rows * H; ++i) xf[i] = (float)oracle_bf16_decode(out->x[i]);
  oracle_nvfp4_quantize(xf, rows, H, out->x_codes, out->x_sf, out->x_sg, out->x_amax);
  free(xf);
  if (oracle_gate_up(rows, H, E, k, I, w, out->x_codes, out->x_sf, *out->x_sg, out->ids,
                     out->offset, out->pair_order, out->h))
    return -1;
  oracle_h_quant(E, I, out->offset, out->h, out->h_codes, out->h_sf, out->h_sg, out->h_amax);
  if (oracle_down(rows, H, E, k, I, w, out->ids, out->offset, out->pair_order, out->h_codes,
                  out->h_sf, out->h_sg, out->o))
    return -1;
  return 0;
}

int oracle_layer_step(int rows, int H, int E, int k, int I, double eps,
                      const oracle_layer_weights* w, const double* branch, float* stream,
                      const int32_t* forced_ids, oracle_layer_out* out) {
  oracle_boundary(rows, H, eps, branch, stream, w->w_post, w->w_pre, out->x, out->x_exact);
  return oracle_moe_step(rows, H, E, k, I, w, forced_ids, out);
}

/* Host threads the oracle's parallel loops use (n >= 1); for timing it on a
   given number of cores.  Changes no result: every reduction runs in index
   order within one output element. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
