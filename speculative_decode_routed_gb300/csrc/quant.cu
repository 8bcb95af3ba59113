// Standalone NVFP4 quantizer for one fp32 tensor (two passes: the tensor's
// max |v|, then the per-16-block encode), used to prepare expert weights.
// Same scheme as the activations inside the step: tensor scale
// sg = amax / 2688; block scale sb = e4m3(fp32(ab / 6) / sg); codes
// e2m1(v / (dec(sb) * sg)), round to nearest even, saturating.
#include "common.cuh"

namespace moe {
namespace {

__global__ void amax_kernel(const float* __restrict__ v, int64_t n, unsigned* amax) {
  __shared__ float red[32];
  float m = 0.0f;
  const int64_t n4 = n / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(v) + i);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = fmaxf(t, red[w]);
    atomic_max_nonneg(amax, t);
  }
}

__global__ void encode_kernel(const float* __restrict__ v, int64_t nblocks,
                              uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
                              const unsigned* amax, float* sg_out) {
  const float sg = __fdiv_rn(__uint_as_float(*amax), 2688.0f);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    const float4* src = reinterpret_cast<const float4*>(v) + b * 4;
    float x[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = __ldg(src + i);
      x[4 * i] = f.x;
      x[4 * i + 1] = f.y;
      x[4 * i + 2] = f.z;
      x[4 * i + 3] = f.w;
    }
    uint32_t lo, hi, sb;
    quant_block16(x, sg, lo, hi, sb);
    reinterpret_cast<uint2*>(codes)[b] = make_uint2(lo, hi);
    sf[b] = (uint8_t)sb;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *sg_out = sg;
}

}  // namespace

cudaError_t launch_quantize(const float* v, int64_t rows, int64_t cols, uint8_t* codes,
                            uint8_t* sf, float* sg, float* amax, cudaStream_t s) {
  const int64_t n = rows * cols;
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  if (n == 0) return cudaMemsetAsync(sg, 0, sizeof(float), s);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  int64_t want = (n / 4 + threads - 1) / threads;
  int grid = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
  amax_kernel<<<grid, threads, 0, s>>>(v, n, reinterpret_cast<unsigned*>(amax));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t nb = n / 16;
  want = (nb + threads - 1) / threads;
  grid = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
  encode_kernel<<<grid, threads, 0, s>>>(v, nb, codes, sf, reinterpret_cast<unsigned*>(amax), sg);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_encode(const float* v, int64_t nblocks, uint8_t* codes, uint8_t* sf,
                                const unsigned* amax, float* sg, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int threads = 256;
  const int64_t want = (nblocks + threads - 1) / threads;
  const int grid = (int)(want < (int64_t)sms * 8 ? (want > 0 ? want : 1) : (int64_t)sms * 8);
  encode_kernel<<<grid, threads, 0, s>>>(v, nblocks, codes, sf, amax, sg);
  return cudaGetLastError();
}

}  // namespace moe
