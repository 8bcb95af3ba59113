// Dual-norm boundary (and the unpooler gather feeding it), one kernel.
//
// Page: vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode,
// module docstring "One step of b rows": the input boundary of later layers
// gathers the previous MoE's unpooler blocks and applies the dual norm into
// the stream; the attention boundary applies the dual norm into the stream
// and the MoE input; "final" is the last gather + dual norm.  The norm pair
// follows MuseSparkDSparkDecoderLayer.forward on the DSpark page:
//   stream' = stream + rmsnorm(branch) * w_post        (fp32 stream)
//   x       = bf16(rmsnorm(stream') * w_pre)
// where branch is either a bf16 tensor or the gathered expert outputs
//   y[r] = sum_s gates[r][s] * o[r*k + s]               (slot order).
// The first layer's front (same page: "the embedded tokens into the stream
// (fp32) and its pre_qkv_proj_norm into the attention input, one kernel") is
// the same kernel with one norm:  stream' = fp32(embedded), x = bf16(
// rmsnorm(stream') * w).  Boundaries that feed the drafter also copy stream'
// into an aux buffer (SpecializedDecode.build: aux buffers of the aux
// layers, and the final boundary's).
//
// GB300 layout: one thread-block cluster per row; each CTA owns H / cluster
// columns (four per thread, 128-bit accesses), and the two row sums of
// squares are reduced across the cluster through distributed shared memory,
// in a fixed order, so every CTA sees the same bit-exact total.  One atomicMax
// per CTA folds max|x| into the MoE input's NVFP4 global-scale accumulator.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace moe {
namespace {

// Block-wide sum of v (fixed order) into *slot, written by thread 0.
__device__ __forceinline__ void block_sum_to_slot(float v, float* warp_red, float* slot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) warp_red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += warp_red[w];
    *slot = t;
  }
}

// The cluster-wide sum of one shared-memory slot (after a cluster barrier):
// lanes 0..7 of warp 0 read one peer's value each (at most 8 CTAs), lane 0
// adds them in rank order -- so every CTA forms the same total bit for bit --
// and the block reads the total from its own shared memory (*total).  One
// remote read per peer and CTA, not one per thread.
__device__ __forceinline__ float cluster_slot_sum(cg::cluster_group& cluster, float* slot, float* total) {
  if (threadIdx.x < 32) {
    const unsigned n = cluster.num_blocks(), lane = threadIdx.x;
    const float v = lane < n ? *cluster.map_shared_rank(slot, lane) : 0.0f;
    float t = 0.0f;
#pragma unroll
    for (unsigned q = 0; q < 8; ++q) {
      const float vq = __shfl_sync(0xffffffffu, v, q);
      if (q < n) t += vq;
    }
    if (lane == 0) *total = t;
  }
  __syncthreads();
  return *total;
}

// KMAX: the most gather slots (k <= KMAX); 8 keeps the registers, and so
// the CTAs per SM, of the common top-8 step.
template <int KMAX>
__global__ void boundary_kernel(BoundaryParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ float warp_red[32];
  __shared__ float part[2];
  __shared__ float part_total[2];
  __shared__ float amax_red[32];

  const int r = blockIdx.y;
  const int col = blockIdx.x * p.cols_per_cta + threadIdx.x * 4;
  const bool live = (int)threadIdx.x * 4 < p.cols_per_cta;

  // Norm weights do not depend on the previous kernel: fetch them first.
  float4 wpost = make_float4(0.f, 0.f, 0.f, 0.f), wpre = wpost;
  if (live) {
    if (!p.front) wpost = __ldg(reinterpret_cast<const float4*>(p.w_post + col));
    wpre = __ldg(reinterpret_cast<const float4*>(p.w_pre + col));
  }
  grid_dep_wait();
  grid_dep_launch();
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int i = threadIdx.x; i < p.n_reset0; i += blockDim.x) p.reset0[i] = 0u;
    for (int i = threadIdx.x; i < p.n_reset1; i += blockDim.x) p.reset1[i] = 0u;
  }

  float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
  if (live) {
    if (p.branch) {
      const uint2 raw = __ldcg(reinterpret_cast<const uint2*>(p.branch + (size_t)r * p.H + col));
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
      y = make_float4(a.x, a.y, b.x, b.y);
    } else if (p.part) {
      // the branch is the split-K partials' sum in split order, as bf16;
      // eight splits' loads in flight at a time
      const size_t split = (size_t)p.rows * p.H;
      const float* src = p.part + (size_t)r * p.H + col;
      for (int s0 = 0; s0 < p.part_S; s0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[j] = (s0 + j < p.part_S) ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)(s0 + j) * split))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          y.x += v[j].x;
          y.y += v[j].y;
          y.z += v[j].z;
          y.w += v[j].w;
        }
      }
      const __nv_bfloat162 b01 = __floats2bfloat162_rn(y.x, y.y), b23 = __floats2bfloat162_rn(y.z, y.w);
      if (p.part_out) {
        uint2 packed;
        packed.x = *reinterpret_cast<const uint32_t*>(&b01);
        packed.y = *reinterpret_cast<const uint32_t*>(&b23);
        *reinterpret_cast<uint2*>(p.part_out + (size_t)r * p.H + col) = packed;
      }
      const float2 f01 = __bfloat1622float2(b01), f23 = __bfloat1622float2(b23);
      y = make_float4(f01.x, f01.y, f23.x, f23.y);
    } else {
      // all slots' loads in flight at once (k <= KMAX), summed in slot order
      float g[KMAX];
      float4 o[KMAX];
#pragma unroll
      for (int s = 0; s < KMAX; ++s) {
        if (s < p.k) {
          g[s] = __ldcg(p.gates + r * p.k + s);
          o[s] = __ldcg(reinterpret_cast<const float4*>(p.o + ((size_t)r * p.k + s) * p.H + col));
        }
      }
#pragma unroll
      for (int s = 0; s < KMAX; ++s) {
        if (s < p.k) {
          y.x = fmaf(g[s], o[s].x, y.x);
          y.y = fmaf(g[s], o[s].y, y.y);
          y.z = fmaf(g[s], o[s].z, y.z);
          y.w = fmaf(g[s], o[s].w, y.w);
        }
      }
    }
  }

  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  float* srow = p.stream + (size_t)r * p.H + col;
  if (p.front) {
    // the first layer's front: the embedded tokens are the stream
    s = y;
  } else {
    // the stream's load in flight with the branch's
    if (live)
      s = __ldcg(reinterpret_cast<const float4*>(p.stream_in ? p.stream_in + (size_t)r * p.H + col : srow));
    // rms of the branch over the whole row (cluster-wide)
    block_sum_to_slot(y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w, warp_red, &part[0]);
    cluster.sync();
    const float ss = cluster_slot_sum(cluster, &part[0], &part_total[0]);
    const float inv1 = rsqrtf(ss / (float)p.H + p.eps);
    if (live) {
      s.x += y.x * inv1 * wpost.x;
      s.y += y.y * inv1 * wpost.y;
      s.z += y.z * inv1 * wpost.z;
      s.w += y.w * inv1 * wpost.w;
    }
  }
  if (live) {
    *reinterpret_cast<float4*>(srow) = s;
    if (p.aux) *reinterpret_cast<float4*>(p.aux + (size_t)r * p.H + col) = s;
  }

  // rms of the updated stream (the dense draft layer rounds the stream to
  // bf16 before its trained input norms)
  if (p.round_norm) {
    s.x = __bfloat162float(__float2bfloat16_rn(s.x));
    s.y = __bfloat162float(__float2bfloat16_rn(s.y));
    s.z = __bfloat162float(__float2bfloat16_rn(s.z));
    s.w = __bfloat162float(__float2bfloat16_rn(s.w));
  }
  block_sum_to_slot(s.x * s.x + s.y * s.y + s.z * s.z + s.w * s.w, warp_red, &part[1]);
  cluster.sync();
  const float ss2 = cluster_slot_sum(cluster, &part[1], &part_total[1]);
  // this CTA has read its peers' shared memory for the last time: arrive now,
  // and wait only before exiting, so the barrier's latency hides behind the
  // stores below
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  const float inv2 = rsqrtf(ss2 / (float)p.H + p.eps);

  float m = 0.0f;
  if (live && p.x_out) {
    const __nv_bfloat162 x01 = __floats2bfloat162_rn(s.x * inv2 * wpre.x, s.y * inv2 * wpre.y);
    const __nv_bfloat162 x23 = __floats2bfloat162_rn(s.z * inv2 * wpre.z, s.w * inv2 * wpre.w);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&x01);
    packed.y = *reinterpret_cast<const uint32_t*>(&x23);
    *reinterpret_cast<uint2*>(p.x_out + (size_t)r * p.H + col) = packed;
    const float2 f01 = __bfloat1622float2(x01), f23 = __bfloat1622float2(x23);
    m = fmaxf(fmaxf(fabsf(f01.x), fabsf(f01.y)), fmaxf(fabsf(f23.x), fabsf(f23.y)));
  }
  if (p.x_amax) {
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) amax_red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = fmaxf(t, amax_red[w]);
      atomic_max_nonneg(p.x_amax, t);
    }
  }
  // keep this CTA's shared memory alive until every peer has read it
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace

int boundary_cluster(int H) {
  for (int c = 8; c >= 1; c >>= 1)
    if (H % (c * 128) == 0) return H / c <= 4096 ? c : 8;
  return 8;
}

cudaError_t launch_boundary(const BoundaryParams& p, int cluster, cudaStream_t s, bool pdl) {
  const int threads = ((p.cols_per_cta / 4 + 31) / 32) * 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, p.rows, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return p.k <= 8 ? cudaLaunchKernelEx(&cfg, boundary_kernel<8>, p) : cudaLaunchKernelEx(&cfg, boundary_kernel<16>, p);
}

}  // namespace moe
