/*
 * CPU oracle of one routed NVFP4 mixture-of-experts decode layer-step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  The GPU library never links,
 * includes or calls it, and it shares no source with the GPU library.
 *
 * What it computes (the step of one decoder layer's MoE block in the
 * specialized decode of the "Muse Spark" decode executor page,
 * vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode, module
 * docstring "One step of b rows": attention boundary = dual norm into the
 * stream and the MoE input; MoE = router -> routing -> pooler -> routed
 * experts -> unpooler; final = last gather + dual norm):
 *
 *   boundary  s' = s + rmsnorm(branch) * w_post          (fp32 stream)
 *             x  = bf16(rmsnorm(s') * w_pre)             (the MoE input)
 *   router    logit[r][e] = sum_h x[r][h] Wr[e][h] (+ bias[e])
 *   routing   p = softmax(logit[r]); top-k by p, ties to the lower expert id;
 *             gates = p_sel / sum(p_sel); flag rows whose k-th/(k+1)-th gap
 *             is below 1e-6
 *   pooler    pairs (row, slot) grouped by expert, experts ascending, rows
 *             ascending within an expert
 *   experts   x quantized to NVFP4 once ([b, H] one tensor); per pair:
 *             G = W_gate x, U = W_up x, h = silu(G) * U (fp32); h quantized
 *             to NVFP4 per expert ([n_e, I] one tensor); o = W_down h
 *   unpooler  y[r] = sum_s gate[r][s] o[pair(r, s)], slot order
 *
 * Arithmetic: fp64 everywhere except where a rounding is part of the
 * definition (the fp32 stream, bf16 MoE input, fp32 h and o, and the fp32
 * scale arithmetic of the NVFP4 quantizer).  NVFP4 dequantization is exact.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- element formats ---------------------------------------------------- */
double oracle_e2m1_decode(uint8_t code);          /* 4-bit code -> value */
uint8_t oracle_e2m1_encode(float v);              /* RNE, saturate to +-6 */
double oracle_e4m3_decode(uint8_t code);          /* OCP E4M3 (fn) byte -> value */
uint8_t oracle_e4m3_encode(float v);              /* RNE, saturate to +-448 */
uint16_t oracle_bf16_from_double(double v);       /* RNE to bf16 bits */
double oracle_bf16_decode(uint16_t bits);

/* ---- NVFP4 quantizer ------------------------------------------------------
 * One tensor v[rows][cols] (cols % 16 == 0), row-major fp32.
 *   amax = max |v|; sg = fp32(amax / 2688)   (2688 = 6 * 448)
 *   per block of 16 along a row: ab = max|v_blk|,
 *     sb = e4m3(fp32(fp32(ab / 6) / sg)), d = fp32(dec(sb) * sg),
 *     code_i = e2m1(fp32(v_i / d));   sg == 0 or d == 0 -> codes 0
 * codes [rows][cols/2], element 2j in the low nibble of byte j;
 * sf [rows][cols/16]; *sg_out and *amax_out receive the scalars. */
void oracle_nvfp4_quantize(const float* v, int64_t rows, int64_t cols, uint8_t* codes,
                           uint8_t* sf, float* sg_out, float* amax_out);
/* v_hat = dec(code) * dec(sf) * sg, exact in fp64. */
void oracle_nvfp4_dequantize(const uint8_t* codes, const uint8_t* sf, float sg, int64_t rows,
                             int64_t cols, double* out);

/* ---- step stages --------------------------------------------------------- */
/* Dual-norm boundary of `rows` rows: branch fp64 [rows][H]; stream fp32
 * [rows][H] in/out; x bf16 bits [rows][H]; x_exact (optional) receives the
 * value before bf16 rounding. */
void oracle_boundary(int rows, int H, double eps, const double* branch, float* stream,
                     const float* w_post, const float* w_pre, uint16_t* x, double* x_exact);

/* The first layer's front: stream fp32 [rows][H] = embedded (bf16 bits),
 * exactly; out bf16 bits = bf16(rmsnorm(stream) * w); out_exact (optional)
 * the value before rounding. */
void oracle_front(int rows, int H, double eps, const uint16_t* embedded, const float* w,
                  float* stream, uint16_t* out, double* out_exact);
/* Dense draft layer pieces.  oracle_bf16_linear: out [M][N] = bf16(A [M][K]
 * . B [N][K]^T), bf16 bits in and out, fp64 sums (exact [M][N], nullable).
 * oracle_silu_mul: a [rows][I] = bf16(silu(gate) * up) from gu [rows][2I]
 * (gate columns, then up columns; exact [rows][I], nullable). */
void oracle_bf16_linear(int M, int N, int K, const uint16_t* A, const uint16_t* B, uint16_t* out,
                        double* exact);
void oracle_silu_mul(int rows, int I, const uint16_t* gu, uint16_t* a, double* exact);
/* One dense draft layer's MLP block: attn_out bf16 bits [rows][H]; stream
 * fp32 [rows][H] in/out; w13 bf16 bits [2I][H] (gate rows, then up rows);
 * w2 bf16 bits [H][I].  Intermediates (bf16 bits): x [rows][H], gu
 * [rows][2I], a [rows][I], f [rows][H]; x_exact fp64 [rows][H] (nullable). */
void oracle_dense_layer(int rows, int H, int I, double eps, const uint16_t* attn_out,
                        float* stream, const float* w_post_attn, const float* w_pre_ffn,
                        const uint16_t* w13, const uint16_t* w2, const float* w_post_ffn,
                        uint16_t* x, uint16_t* gu, uint16_t* a, uint16_t* f, double* x_exact);
/* Draft context-KV projection pieces.  ctx bf16 bits [n][H]; w_pre fp32
 * [L][H]; fc bf16 bits [n][H]; u bf16 bits [L][n][H] (fc_exact, u_exact
 * nullable: the values before their rounding).
 * kv bf16 bits [L][n][2*KVH*D] (K heads, then V heads); k_out, v_out bf16
 * bits [L][n][KVH][D] (k_exact, kn_exact nullable: the rotated and the
 * normalised keys before their rounding); positions [n]; theta 0 = no rotary
 * embedding.  Caches [L][n_slots][KVH][D]; slots [L][layer_stride] (stride 0:
 * one mapping for every layer). */
void oracle_layer_norms(int n, int H, int L, double eps, const uint16_t* fc, const float* w_pre,
                        uint16_t* u, double* u_exact);
void oracle_ctx_norms(int n, int H, int L, double eps, const uint16_t* ctx, const float* w_hidden,
                      const float* w_pre, uint16_t* fc, uint16_t* u, double* fc_exact, double* u_exact);
void oracle_k_norm_rope(int L, int n, int KVH, int D, double qk_eps, double theta,
                        const int64_t* positions, const uint16_t* kv, uint16_t* k_out,
                        uint16_t* v_out, double* k_exact, double* kn_exact);
void oracle_kv_cache_write(int L, int n, int KVH, int D, const int64_t* slots, int layer_stride,
                           int64_t n_slots, const uint16_t* k, const uint16_t* v, uint16_t* k_cache,
                           uint16_t* v_cache);
/* Router + routing.  x bf16 [rows][H]; router_w bf16 [E][H]; bias fp32 [E] or
 * NULL.  Outputs: logits fp64 [rows][E] (optional), probs fp64 [rows][E]
 * (optional), ids int32 [rows][k] (slot order: descending p), gates fp64
 * [rows][k], flags uint8 [rows], gap fp64 [rows] (optional: p_k - p_k+1, or
 * +inf when k == E). */
void oracle_route(int rows, int H, int E, int k, const uint16_t* x, const uint16_t* router_w,
                  const float* bias, double* logits, double* probs, int32_t* ids, double* gates,
                  uint8_t* flags, double* gap);

/* Pooler: count [E], offset [E+1], pair_order [rows*k] (pair id r*k+s,
 * grouped by expert ascending, rows ascending), active [E] (first *n_active
 * entries used). */
void oracle_pool(int rows, int E, int k, const int32_t* ids, int32_t* count, int32_t* offset,
                 int32_t* pair_order, int32_t* active, int32_t* n_active);

typedef struct {
  const float* w_post;            /* [H] */
  const float* w_pre;             /* [H] */
  const uint16_t* router_w;       /* bf16 [E][H] */
  const float* router_bias;       /* [E] or NULL */
  const uint8_t* const* w13;      /* [E] -> e2m1x2 [2I][H/2]: gate rows, then up rows */
  const uint8_t* const* w13_sf;   /* [E] -> e4m3 [2I][H/16] */
  const uint8_t* const* w2;       /* [E] -> e2m1x2 [H][I/2] */
  const uint8_t* const* w2_sf;    /* [E] -> e4m3 [H][I/16] */
  const float* gscale;            /* [E][3]: gate, up, down global scales */
} oracle_layer_weights;

/* Experts gate/up: for each pair in pooled order, h[pos][I] (fp32) =
 * silu(G) * U over dequantized operands.  x codes/sf/sg: the NVFP4 MoE input. */
int oracle_gate_up(int rows, int H, int E, int k, int I, const oracle_layer_weights* w,
                   const uint8_t* x_codes, const uint8_t* x_sf, float x_sg, const int32_t* ids,
                   const int32_t* offset, const int32_t* pair_order, float* h);

/* h quantization: each expert's rows h[offset[e] .. offset[e+1]) form one
 * tensor.  h_codes [rows*k][I/2], h_sf [rows*k][I/16], h_sg [E], h_amax [E]
 * (experts without pairs get 0). */
void oracle_h_quant(int E, int I, const int32_t* offset, const float* h, uint8_t* h_codes,
                    uint8_t* h_sf, float* h_sg, float* h_amax);

/* Experts down: o[pair id][H] (fp32) = W_down h_hat for every pair. */
int oracle_down(int rows, int H, int E, int k, int I, const oracle_layer_weights* w,
                const int32_t* ids, const int32_t* offset, const int32_t* pair_order,
                const uint8_t* h_codes, const uint8_t* h_sf, const float* h_sg, float* o);

/* Unpooler: y[r][H] (fp64) = sum_s gates[r][s] * o[r*k+s], slot order. */
void oracle_gather(int rows, int H, int k, const double* gates, const float* o, double* y);

/* One layer (boundary .. down), every intermediate written out.  If
 * forced_ids is not NULL the routing uses those ids (the gates are then the
 * renormalised probabilities of those ids) instead of its own top-k. */
typedef struct {
  uint16_t* x; double* x_exact;
  uint8_t* x_codes; uint8_t* x_sf; float* x_sg; float* x_amax;
  double* probs; int32_t* ids; double* gates; uint8_t* flags; double* gap;
  int32_t* count; int32_t* offset; int32_t* pair_order; int32_t* active; int32_t* n_active;
  float* h; uint8_t* h_codes; uint8_t* h_sf; float* h_sg; float* h_amax;
  float* o;
} oracle_layer_out;

int oracle_layer_step(int rows, int H, int E, int k, int I, double eps,
                      const oracle_layer_weights* w, const double* branch, float* stream,
                      const int32_t* forced_ids, oracle_layer_out* out);

/* The same layer's MoE part alone, from the bf16 MoE input already in
 * out->x (x_exact is not touched): routing, pooler, the input's NVFP4
 * quantization and the experts, with forced_ids as above.  oracle_layer_step
 * is the boundary followed by this. */
int oracle_moe_step(int rows, int H, int E, int k, int I, const oracle_layer_weights* w,
                    const int32_t* forced_ids, oracle_layer_out* out);

/* Number of OpenMP threads the oracle uses (for reporting). */
void oracle_set_num_threads(int n);
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
