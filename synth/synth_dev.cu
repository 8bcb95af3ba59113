// Seeded synthetic inputs, device side.
//
// Holds no arithmetic of the MoE decode step.  It implements, from their
// published definitions and independently of the host file, the same two
// generators as synth_host.c so that large synthetic tensors (the expert
// weights: up to hundreds of GB) can be produced where they live, in HBM:
//
//  - Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11, section 4);
//  - the Irwin-Hall sum of the eight 16-bit halves of one Philox block,
//    centred and scaled by sqrt(12/8) (rounded to fp32) to unit variance.
//
// Keying: key = (seed, tag); counter = (index lo, index hi, 0, 0).
// Every fp32 operation is an explicit round-to-nearest intrinsic so that no
// multiply-add is contracted: the values match the host bit for bit.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace {

__device__ __forceinline__ void philox10(uint32_t& c0, uint32_t& c1, uint32_t& c2, uint32_t& c3,
                                         uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
}

__device__ __forceinline__ float unit_normal(uint32_t seed, uint32_t tag, uint64_t index) {
  uint32_t c0 = (uint32_t)index, c1 = (uint32_t)(index >> 32), c2 = 0u, c3 = 0u;
  philox10(c0, c1, c2, c3, seed, tag);
  const int32_t s = (int32_t)(c0 & 0xFFFFu) + (int32_t)(c0 >> 16) + (int32_t)(c1 & 0xFFFFu) +
                    (int32_t)(c1 >> 16) + (int32_t)(c2 & 0xFFFFu) + (int32_t)(c2 >> 16) +
                    (int32_t)(c3 & 0xFFFFu) + (int32_t)(c3 >> 16);
  const float z = __fmul_rn(__int2float_rn(s - 262140), 1.0f / 65536.0f);
  return __fmul_rn(z, 1.2247449f);
}

__device__ __forceinline__ float normal(uint32_t seed, uint32_t tag, uint64_t index, float mu,
                                        float sigma) {
  return __fadd_rn(mu, __fmul_rn(sigma, unit_normal(seed, tag, index)));
}

__global__ void k_normal_f32(float* __restrict__ out, uint64_t n, uint32_t seed, uint32_t tag,
                             float mu, float sigma) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = normal(seed, tag, i, mu, sigma);
}

__global__ void k_normal_bf16(__nv_bfloat16* __restrict__ out, uint64_t n, uint32_t seed,
                              uint32_t tag, float mu, float sigma) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __float2bfloat16_rn(normal(seed, tag, i, mu, sigma));
}

int grid_for(uint64_t n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  uint64_t want = (n + 255) / 256;
  uint64_t cap = (uint64_t)sms * 8;
  return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

extern "C" {

// Fills out[0..n) (device memory) with mu + sigma * z(seed, tag, i).
// Returns a cudaError_t value (0 on success).  Asynchronous on `stream`.
int synth_dev_normal_f32(float* out, uint64_t n, uint32_t seed, uint32_t tag, float mu,
                         float sigma, cudaStream_t stream) {
  if (n == 0) return 0;
  if (out == nullptr) return (int)cudaErrorInvalidValue;
  k_normal_f32<<<grid_for(n), 256, 0, stream>>>(out, n, seed, tag, mu, sigma);
  return (int)cudaGetLastError();
}

// As synth_dev_normal_f32, rounded to bf16 (round to nearest even).
int synth_dev_normal_bf16(void* out, uint64_t n, uint32_t seed, uint32_t tag, float mu,
                          float sigma, cudaStream_t stream) {
  if (n == 0) return 0;
  if (out == nullptr) return (int)cudaErrorInvalidValue;
  k_normal_bf16<<<grid_for(n), 256, 0, stream>>>((__nv_bfloat16*)out, n, seed, tag, mu, sigma);
  return (int)cudaGetLastError();
}

}  // extern "C"
