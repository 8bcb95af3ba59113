// Internal interface of the bf16 projection kernel on the 5th-generation
// tensor cores (tc_gemm.cu): out = X . W^T for bf16 weights W [L][R][K]
// (K-major) and activations X [rows of a layer][K], fp32 accumulation.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace moe {

enum GemmMode : int {
  kGemmPartial = 0,  // fp32 split-K partials part [S][L][n][R]; the caller sums them in split order
  kGemmBf16 = 1,     // bf16 out [L][n][R] (one split)
  kGemmGated = 2,    // gate/up of a gated MLP (L = 1, R = 2I, one split): gu [n][2I] = bf16 of
                     // both, act [n][I] = bf16(silu(gate) * up) from the bf16 values
};

struct GemmParams {
  int mode;          // GemmMode
  int L, R, K, n;    // layers, weight rows per layer, reduction length, activation rows
  int I;             // gated: gate rows 0..I-1, up rows I..2I-1 of W
  int S;             // K-splits (partials), else 1
  int KB;            // K-boxes of 64 elements: ceil(K / 64)
  int KX;            // K-boxes per pipeline stage (consecutive in K; boxes past K read zeros)
  int KST;           // stages along K: ceil(KB / KX)
  int KBS;           // stages per split (every split has at least one)
  int NT;            // activation rows per MMA tile: a multiple of 16, at most 128
  int n_tiles;       // ceil(n / NT)
  int m_tiles;       // 128-row weight tiles per layer: ceil(R / 128), gated ceil(I / 128)
  int x_layer_rows;  // rows between layers in X's map (X[l][i] is row l * x_layer_rows + i)
  int NS;            // pipeline stages
  uint32_t a_box;    // weight bytes per K-box (16 KB; gated 32 KB: gate tile, then up tile)
  uint32_t a_bytes;  // weight bytes per stage: KX * a_box
  uint32_t b_box;    // activation bytes per K-box: NT * 128
  uint32_t stage_stride;
  float* part;           // kGemmPartial
  __nv_bfloat16* out;    // kGemmBf16
  __nv_bfloat16* gu;     // kGemmGated
  __nv_bfloat16* act;    // kGemmGated
  unsigned* err;         // latched error word of the caller (a bounded wait that gave up)
  unsigned long long wait_ns;
};

// The tensor maps of one projection: the weights (box 64 elements x 128 rows)
// and the activations at each tile width (box 64 x 16t rows, t = 1..8).
struct GemmMaps {
  CUtensorMap w;
  CUtensorMap x[8];
};

// Plans mode, shapes and splits for num_sms SMs (the K-splits of a partial
// projection chosen so the busiest SM streams the fewest stages).  kx > 0
// fixes the K-boxes per stage, else the plan picks them.  Returns false if
// the shape is not served (K not a multiple of 8).
bool plan_gemm(GemmParams& p, int mode, int L, int R, int K, int n, int I, int x_layer_rows,
               int num_sms, int max_splits, int kx = 0);
// Encodes the weight map over W [L * R][K] and the activation maps over X
// [x_rows][K] (bf16, row-major, 16-byte aligned, K a multiple of 8).
cudaError_t encode_gemm_maps(GemmMaps& m, const void* W, int64_t w_rows, const void* X,
                             int64_t x_rows, int K);
size_t gemm_smem_bytes(const GemmParams& p);
cudaError_t gemm_set_smem();
cudaError_t launch_gemm(const GemmParams& p, const GemmMaps& m, int num_sms, cudaStream_t s,
                        bool pdl);

}  // namespace moe
