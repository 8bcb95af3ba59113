// NVFP4 quantizer that allocates no device memory.
//
// moe_nvfp4_quantize needs a device scalar for the tensor's max |v|, which its
// caller allocates.  Some callers cannot allocate device memory at all: code
// that runs as a plugin or callback of another runtime which hands it only
// input and output buffers and owns every allocation itself (its memory pool
// or budget would not know about a cudaMalloc made behind its back), and
// latency-critical loops where cudaMalloc / cudaFree, which may synchronize
// the whole device, cannot be called.  This variant keeps its scratch in a
// fixed array compiled into the library instead:
//
//   g_noalloc_scratch: kNoAllocChunks fp32 partial maxima (one per chunk of
//   kNoAllocChunk elements), a CTA counter and the final max |v|, 64 KB and a
//   few bytes in all.  Every GPU that loads the library holds it until the
//   process exits.
//
// Pass 1 (one CTA per chunk) writes each chunk's max |v| to the scratch; the
// last CTA to finish reduces the partials into the tensor's max |v| and
// resets the counter.  Pass 2 is the quantizer's own encode kernel, reading
// that max from the scratch.  max is exact in any order, so the codes, block
// scales and tensor scale are bit for bit those of moe_nvfp4_quantize.
#include <mutex>

#include <cuda.h>

#include "../../include/moe_decode.h"
#include "common.cuh"
#include "moe_decode_internal.h"

namespace moe {
namespace {

constexpr int kNoAllocThreads = 256;
constexpr int64_t kNoAllocChunk = 65536;   // elements one CTA of pass 1 reduces
constexpr int kNoAllocChunks = 16384;      // partial maxima the scratch holds
constexpr size_t kOffCount = (size_t)kNoAllocChunks * sizeof(float);
constexpr size_t kOffAmax = kOffCount + sizeof(unsigned);
constexpr size_t kNoAllocScratchBytes = kOffCount + 256;
constexpr int kNoAllocMaxDevices = 64;

// The scratch.  Host code must not use this name as a device address (on the
// host it names a host-side stand-in); it gets the device address once per
// device from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

__global__ void __launch_bounds__(kNoAllocThreads)
    amax_chunks_kernel(const float* __restrict__ v, int64_t n, unsigned char* scratch) {
  __shared__ float red[kNoAllocThreads / 32];
  __shared__ int last;
  float* partial = reinterpret_cast<float*>(scratch);
  unsigned* count = reinterpret_cast<unsigned*>(scratch + kOffCount);
  unsigned* amax = reinterpret_cast<unsigned*>(scratch + kOffAmax);
  const int64_t beg = (int64_t)blockIdx.x * kNoAllocChunk;
  const int64_t end = (n - beg < kNoAllocChunk) ? n : beg + kNoAllocChunk;
  float m = 0.0f;
  for (int64_t i = beg / 4 + threadIdx.x; i < end / 4; i += kNoAllocThreads) {
    const float4 f = __ldg(reinterpret_cast<const float4*>(v) + i);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < kNoAllocThreads / 32; ++w) t = fmaxf(t, red[w]);
    partial[blockIdx.x] = t;
    __threadfence();
    last = (atomicAdd(count, 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  float t = 0.0f;
  for (int c = threadIdx.x; c < (int)gridDim.x; c += kNoAllocThreads) t = fmaxf(t, __ldcg(partial + c));
  t = warp_max(t);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.0f;
    for (int w = 0; w < kNoAllocThreads / 32; ++w) a = fmaxf(a, red[w]);
    *amax = __float_as_uint(a);
    *count = 0u;  // ready for the next call
  }
}

// Device address of the scratch, looked up once per device and context.  A
// device reset (cudaDeviceReset, or a reset of the primary context) loads the
// module again at a new address, so the cached address is kept together with
// the unique ID of the context it was taken in (a context handle may be
// reused after a reset; its ID never is) and looked up again when the current
// context's ID differs.
std::mutex g_setup_mu;
unsigned char* g_scratch_addr[kNoAllocMaxDevices] = {};
unsigned long long g_scratch_ctx_id[kNoAllocMaxDevices] = {};

// The unique ID of the calling thread's current context (0: none yet), from
// the driver's cuCtxGetCurrent and cuCtxGetId through the runtime's
// entry-point query (the library does not link the driver library itself).
CUresult current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  if (!get_current || !get_id) {
    void* p1 = nullptr;
    void* p2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 4000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return CUDA_ERROR_NOT_FOUND;
    get_current = reinterpret_cast<GetCurrent>(p1);
    get_id = reinterpret_cast<GetId>(p2);
  }
  CUcontext ctx = nullptr;
  const CUresult r = get_current(&ctx);
  if (r != CUDA_SUCCESS) return r;
  *id = 0;
  return ctx ? get_id(ctx, id) : CUDA_SUCCESS;
}

int scratch_address(unsigned char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return api_fail(MOE_ECUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return api_fail(MOE_EUNSUPPORTED, "device ordinal beyond the no-alloc quantizer's table (64)");
  unsigned long long id = 0;  // 0 before the runtime's first call on this thread
  if (current_context_id(&id) != CUDA_SUCCESS) return api_fail(MOE_ECUDA, "context query failed");
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!id || !g_scratch_addr[dev] || g_scratch_ctx_id[dev] != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the primary context current
    if (e != cudaSuccess || !p) return api_fail(MOE_ECUDA, cudaGetErrorString(e));
    if (!id && (current_context_id(&id) != CUDA_SUCCESS || !id))
      return api_fail(MOE_ECUDA, "no current CUDA context");
    g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    g_scratch_ctx_id[dev] = id;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_nvfp4_quantize_noalloc(const float* v, int64_t rows, int64_t cols,
                                          uint8_t* codes, uint8_t* sf, float* sg,
                                          void* cuda_stream) {
  using namespace moe;
  if (!v || !codes || !sf || !sg) return api_fail(MOE_EINVAL, "null pointer");
  if (rows < 0 || cols < 0 || cols % 16) return api_fail(MOE_EINVAL, "cols must be a multiple of 16");
  if (cols > 0 && rows > (kNoAllocChunk * kNoAllocChunks) / cols)
    return api_fail(MOE_EUNSUPPORTED,
                    "tensor larger than the no-alloc quantizer's limit of 2^30 elements "
                    "(16384 chunks of 65536); use moe_nvfp4_quantize");
  if (reinterpret_cast<uintptr_t>(v) % 16 || reinterpret_cast<uintptr_t>(codes) % 8 ||
      reinterpret_cast<uintptr_t>(sg) % 4)
    return api_fail(MOE_EINVAL, "v must be 16-byte, codes 8-byte and sg 4-byte aligned");
  unsigned char* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const int64_t n = rows * cols;
  // the counter must start at zero even if an earlier call was cut short
  cudaError_t e = cudaMemsetAsync(scratch + kOffCount, 0, 2 * sizeof(unsigned), s);
  if (e != cudaSuccess) return api_fail(MOE_ECUDA, cudaGetErrorString(e));
  if (n == 0) {
    e = cudaMemsetAsync(sg, 0, sizeof(float), s);
    return e == cudaSuccess ? MOE_OK : api_fail(MOE_ECUDA, cudaGetErrorString(e));
  }
  const int chunks = (int)((n + kNoAllocChunk - 1) / kNoAllocChunk);
  amax_chunks_kernel<<<chunks, kNoAllocThreads, 0, s>>>(v, n, scratch);
  e = cudaGetLastError();
  if (e != cudaSuccess) return api_fail(MOE_ECUDA, cudaGetErrorString(e));
  e = launch_nvfp4_encode(v, n / 16, codes, sf, reinterpret_cast<const unsigned*>(scratch + kOffAmax),
                          sg, s);
  if (e != cudaSuccess) return api_fail(MOE_ECUDA, cudaGetErrorString(e));
  return MOE_OK;
}
