// bf16 projections of a few to a few hundred activation rows on the
// 5th-generation tensor cores (tcgen05.mma kind::f16, fp32 accumulation).
//
// Pages: the DSpark page (vllm.models.muse_spark.common.dspark),
// MuseSparkDSparkDecoderLayer.forward (the dense draft layer's gate_up_proj
// and down_proj) and _project_muse_context_kv (every draft layer's stacked
// K/V projection of the context rows).  Used where the weight-streaming
// kernel (gemv.cuh, up to 8 rows) does not apply.
//
// Swap-AB, as in the routed experts: the weight rows fill the MMA's M = 128
// (operand A, streamed from HBM through a TMA ring, 128-byte swizzle) and the
// activation rows fill N (operand B, 16..128 rows per tile); K advances in
// boxes of 64 elements (128 bytes), four K = 16 MMAs each, and a pipeline
// stage holds KX consecutive boxes, so every weight row is requested in runs
// of KX * 128 contiguous bytes (with one box per stage the next 128 bytes of a
// row came a stage later, and DRAM ran half idle).  A task is one
// 128-row weight tile (of one layer; gated: 128 gate rows and the matching
// 128 up rows, two accumulators), one activation tile and one K-split; one
// persistent CTA per SM takes tasks b, b + grid, ... and keeps its ring
// streaming across task boundaries.  Warp roles:
//   warp 0  producer: the weight copies of the first stages go out before the
//           programmatic-dependency wait (the weights do not depend on the
//           kernel before), the activation copies after it;
//   warp 1  MMA issuer into one of two TMEM accumulator buffers;
//   warps 2-5 epilogue: tcgen05.ld of the accumulators (one TMEM lane per
//           weight row), stores coalesced along the weight rows: fp32 split-K
//           partials, bf16 outputs, or the gated MLP's bf16 gate/up and
//           silu(gate) * up.
// Every wait is bounded by the caller's wait limit (a latched error instead
// of a hang).
#include "tc_gemm.h"

#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kGmThreads = 32 * 6;
constexpr int kGmEpi0 = 2;            // first epilogue warp
constexpr int kGmCtrl = 1024;         // barriers and flags
constexpr int kGmMaxStages = 8;
constexpr uint32_t kGmAccCols = 256;  // TMEM columns per accumulator buffer (gate at 0, up at 128)

// kind::f16 instruction descriptor: fp32 D (bit 4), bf16 A and B (bits 7 and
// 10), both K-major, N >> 3 at bit 17, M >> 4 at bit 24 (M = 128).
__device__ __forceinline__ uint32_t gm_idesc(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void gm_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

struct GmSmem {
  uint64_t* full;       // [NS]  a stage's copies landed
  uint64_t* empty;      // [NS]  the issuer is done with a stage
  uint64_t* acc_full;   // [2]   an accumulator buffer is ready for the epilogue
  uint64_t* acc_empty;  // [2]   the epilogue has read it (4 warps)
  uint64_t* drain;      // [1]   every MMA issued has completed
  int* flag;            // the epilogue's shared verdict
  uint32_t* tmem_base;
  uint8_t* stages;
};

__device__ __forceinline__ GmSmem gm_carve(uint8_t* base) {
  GmSmem s;
  s.full = reinterpret_cast<uint64_t*>(base);
  s.empty = s.full + kGmMaxStages;
  s.acc_full = s.empty + kGmMaxStages;
  s.acc_empty = s.acc_full + 2;
  s.drain = s.acc_empty + 2;
  s.flag = reinterpret_cast<int*>(s.drain + 1);
  s.tmem_base = reinterpret_cast<uint32_t*>(s.flag + 4);
  s.stages = base + kGmCtrl;
  return s;
}

// Task t -> (layer, weight tile, split, activation tile).
struct GmTask {
  int l, m, s, nt, st0, st1;  // stages [st0, st1) along K
};

__device__ __forceinline__ GmTask gm_task(const GemmParams& p, int t) {
  GmTask k;
  k.nt = t % p.n_tiles;
  k.s = (t / p.n_tiles) % p.S;
  k.m = (t / (p.n_tiles * p.S)) % p.m_tiles;
  k.l = t / (p.n_tiles * p.S * p.m_tiles);
  k.st0 = k.s * p.KBS;
  k.st1 = min(p.KST, k.st0 + p.KBS);
  return k;
}

__global__ void __launch_bounds__(kGmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap mw,
                   const __grid_constant__ CUtensorMap mx) {
  extern __shared__ __align__(1024) uint8_t gm_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gm_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const GmSmem sm = gm_carve(base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool gated = p.mode == kGemmGated;
  const int tasks = p.L * p.m_tiles * p.S * p.n_tiles;
  const uint64_t lim = p.wait_ns;

  if (tid == 0) {
    for (int i = 0; i < p.NS; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.acc_full[i], 1);
      mbar_init(&sm.acc_empty[i], 4);
    }
    mbar_init(sm.drain, 1);
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mw)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mx)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(sm.tmem_base)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  grid_dep_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_base;
  const uint32_t bytes = p.a_bytes + (uint32_t)p.KX * p.b_box;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      auto issue_w = [&](uint8_t* st, uint64_t* full, const GmTask& k, int sk) {
        mbar_arrive_expect_tx(full, bytes);
        for (int b = 0; b < p.KX; ++b) {
          const int x = (sk * p.KX + b) * 64;
          uint8_t* dst = st + (size_t)b * p.a_box;
          if (gated) {
            tma_2d(dst, &mw, x, k.m * 128, full, pol);
            tma_2d(dst + 16384, &mw, x, p.I + k.m * 128, full, pol);
          } else {
            tma_2d(dst, &mw, x, k.l * p.R + k.m * 128, full, pol);
          }
        }
      };
      // the first stages' weights, before the dependency wait
      int pre = 0;
      for (int t = blockIdx.x; t < tasks && pre < p.NS; t += gridDim.x) {
        const GmTask k = gm_task(p, t);
        for (int sk = k.st0; sk < k.st1 && pre < p.NS; ++sk, ++pre)
          issue_w(sm.stages + (size_t)pre * p.stage_stride, &sm.full[pre], k, sk);
      }
      grid_dep_wait();
      int g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tasks && ok; t += gridDim.x) {
        const GmTask k = gm_task(p, t);
        for (int sk = k.st0; sk < k.st1; ++sk, ++g) {
          const int s = g % p.NS;
          uint8_t* st = sm.stages + (size_t)s * p.stage_stride;
          if (g >= pre) {
            if (g >= p.NS && !mbar_wait(&sm.empty[s], ((g / p.NS) - 1) & 1, lim)) {
              latch_error(p.err, kDevWaitTimeout);
              ok = false;
              break;
            }
            issue_w(st, &sm.full[s], k, sk);
          }
          for (int b = 0; b < p.KX; ++b)
            tma_2d_plain(st + p.a_bytes + (size_t)b * p.b_box, &mx, (sk * p.KX + b) * 64,
                         k.l * p.x_layer_rows + k.nt * p.NT, &sm.full[s]);
        }
      }
      // every issued copy lands before the CTA exits: the last fill of each
      // stage (it was issued only after the fills before it were consumed)
      const int issued = ok ? g : max(g, pre);
      for (int s = 0; s < p.NS && s < issued; ++s) {
        const int last = s + p.NS * ((issued - 1 - s) / p.NS);
        if (!mbar_wait(&sm.full[s], (uint32_t)(last / p.NS) & 1u, lim)) latch_error(p.err, kDevWaitTimeout);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = gm_idesc((uint32_t)p.NT);
      int g = 0;
      bool ok = true;
      int j = 0;
      for (int t = blockIdx.x; t < tasks && ok; t += gridDim.x, ++j) {
        const GmTask k = gm_task(p, t);
        const int buf = j & 1, use = j >> 1;
        if (use >= 1 && !mbar_wait(&sm.acc_empty[buf], (use - 1) & 1, lim)) {
          latch_error(p.err, kDevWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)buf * kGmAccCols;
        for (int sk = k.st0; sk < k.st1; ++sk, ++g) {
          const int s = g % p.NS;
          if (!mbar_wait(&sm.full[s], (uint32_t)(g / p.NS) & 1u, lim)) {
            latch_error(p.err, kDevWaitTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(sm.stages + (size_t)s * p.stage_stride);
          for (int b = 0; b < p.KX; ++b) {
            const uint32_t a0 = st + (uint32_t)b * p.a_box;
            const uint32_t b0 = st + p.a_bytes + (uint32_t)b * p.b_box;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint64_t bd = smem_desc(b0 + 32u * q, 16, 1024, 2);
              const bool acc = !(sk == k.st0 && b == 0 && q == 0);
              gm_mma(d0, smem_desc(a0 + 32u * q, 16, 1024, 2), bd, idesc, acc);
              if (gated) gm_mma(d0 + 128u, smem_desc(a0 + 16384u + 32u * q, 16, 1024, 2), bd, idesc, acc);
            }
          }
          tc_commit(&sm.empty[s]);
        }
        if (ok) tc_commit(&sm.acc_full[buf]);
      }
      // everything issued completes before the tensor memory is freed
      tc_commit(sm.drain);
      if (!mbar_wait(sm.drain, 0, lim)) latch_error(p.err, kDevWaitTimeout);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int t_epi = tid - 32 * kGmEpi0;  // 0..127
    const int qd = warp & 3;               // the TMEM lane quadrant this warp may read
    const int mrow = 32 * qd + lane;       // weight row within the tile
    const uint32_t lanes = (uint32_t)(32 * qd) << 16;
    int j = 0;
    for (int t = blockIdx.x; t < tasks; t += gridDim.x, ++j) {
      const GmTask k = gm_task(p, t);
      const int buf = j & 1, use = j >> 1;
      if (t_epi == 0) *sm.flag = mbar_wait(&sm.acc_full[buf], use & 1, lim) ? 1 : 0;
      named_bar(1, 128);
      const bool got = *reinterpret_cast<volatile int*>(sm.flag) != 0;
      named_bar(1, 128);
      if (!got) {
        if (t_epi == 0) latch_error(p.err, kDevWaitTimeout);
        break;
      }
      tc_fence_after();
      const int wrow = k.m * 128 + mrow;  // weight row (gated: gate / up row index j)
      const bool row_ok = wrow < (gated ? p.I : p.R);
      for (int c0 = 0; c0 < p.NT; c0 += 16) {
        uint32_t ra[16], rb[16];
        __syncwarp();  // the tensor-memory loads are warp-collective
        tc_ld16(tmem + lanes + (uint32_t)buf * kGmAccCols + (uint32_t)c0, ra);
        if (gated) tc_ld16(tmem + lanes + (uint32_t)buf * kGmAccCols + 128u + (uint32_t)c0, rb);
        tc_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (!row_ok) break;
          const int i = k.nt * p.NT + c0 + q;  // activation row
          if (i >= p.n) break;
          const float v = __uint_as_float(ra[q]);
          if (p.mode == kGemmPartial) {
            p.part[(((size_t)k.s * p.L + k.l) * p.n + i) * p.R + wrow] = v;
          } else if (p.mode == kGemmBf16) {
            p.out[((size_t)k.l * p.n + i) * p.R + wrow] = __float2bfloat16_rn(v);
          } else {
            const __nv_bfloat16 gb = __float2bfloat16_rn(v), ub = __float2bfloat16_rn(__uint_as_float(rb[q]));
            p.gu[(size_t)i * 2 * p.I + wrow] = gb;
            p.gu[(size_t)i * 2 * p.I + p.I + wrow] = ub;
            const float gv = __bfloat162float(gb), uv = __bfloat162float(ub);
            p.act[(size_t)i * p.I + wrow] = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 gemm_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 [rows][K] row-major, boxes of 64 elements x box_rows, 128-byte swizzle.
cudaError_t encode_bf16_rows(CUtensorMap* m, const void* base, int64_t rows, int K, int box_rows) {
  auto enc = gemm_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                         box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool plan_gemm(GemmParams& p, int mode, int L, int R, int K, int n, int I, int x_layer_rows,
               int num_sms, int max_splits, int kx) {
  if (K < 8 || K % 8 || n < 1 || L < 1 || R < 1) return false;
  p = GemmParams{};
  p.mode = mode;
  p.L = L;
  p.R = R;
  p.K = K;
  p.n = n;
  p.I = I;
  p.x_layer_rows = x_layer_rows;
  p.NT = n >= 128 ? 128 : (n + 15) / 16 * 16;
  p.n_tiles = (n + p.NT - 1) / p.NT;
  p.KB = (K + 63) / 64;
  p.m_tiles = mode == kGemmGated ? (I + 127) / 128 : (R + 127) / 128;
  p.a_box = mode == kGemmGated ? 32768u : 16384u;
  p.b_box = (uint32_t)p.NT * 128u;
  const uint32_t budget = 227u * 1024u - 1024u - (uint32_t)kGmCtrl;
  auto stride_of = [&](int x) { return ((uint32_t)x * (p.a_box + p.b_box) + 1023u) / 1024u * 1024u; };
  if (kx <= 0) {
    // the widest stage (up to 8 boxes, 1 KB of each weight row) that leaves
    // two in the ring and does not read far past K: measured on 33- to
    // 128-row projections at K 7168 and 28672, longer runs per row beat a
    // deeper ring (K 28672, 33 rows: 1, 2, 4 boxes at 0.58, 0.72, 0.77 of the
    // copy bandwidth with 8, 5, 2 stages)
    kx = 8;
    while (kx > 1 && kx / 2 >= p.KB) kx /= 2;
    while (kx > 1 && budget / stride_of(kx) < 2) kx /= 2;
  }
  p.KX = kx;
  p.KST = (p.KB + kx - 1) / kx;
  // K-splits (partials only): the busiest SM's stages, ceil(tasks / SMs) *
  // stages per split, as small as it gets; among counts within 3 % of the
  // best, the fewest (the caller sums the partials)
  int S = 1;
  if (mode == kGemmPartial) {
    const long long base = (long long)L * p.m_tiles * p.n_tiles;
    long long best = -1;
    for (int pass = 0; pass < 2; ++pass)
      for (int s = 1; s <= max_splits && s <= p.KST; ++s) {
        const int kbs = (p.KST + s - 1) / s;
        const long long cost = ((base * s + num_sms - 1) / num_sms) * kbs;
        if (pass == 0 && (best < 0 || cost < best)) best = cost;
        if (pass == 1 && cost * 100 <= best * 103) {
          S = s;
          pass = 2;
          break;
        }
      }
  }
  p.KBS = (p.KST + S - 1) / S;
  p.S = (p.KST + p.KBS - 1) / p.KBS;  // every split has at least one stage
  p.a_bytes = (uint32_t)kx * p.a_box;
  p.stage_stride = stride_of(kx);
  const int ns = (int)(budget / p.stage_stride);
  p.NS = ns > kGmMaxStages ? kGmMaxStages : ns;
  p.wait_ns = kDefaultWaitNs;
  return p.NS >= 2;
}

cudaError_t encode_gemm_maps(GemmMaps& m, const void* W, int64_t w_rows, const void* X, int64_t x_rows,
                             int K) {
  cudaError_t e = encode_bf16_rows(&m.w, W, w_rows, K, 128);
  for (int t = 0; t < 8 && e == cudaSuccess; ++t) e = encode_bf16_rows(&m.x[t], X, x_rows, K, 16 * (t + 1));
  return e;
}

size_t gemm_smem_bytes(const GemmParams& p) {
  return 1024 + (size_t)kGmCtrl + (size_t)p.NS * p.stage_stride;  // + alignment slack
}

cudaError_t gemm_set_smem() {
  return cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

cudaError_t launch_gemm(const GemmParams& p, const GemmMaps& m, int num_sms, cudaStream_t s, bool pdl) {
  const int tasks = p.L * p.m_tiles * p.S * p.n_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tasks < num_sms ? tasks : num_sms, 1, 1);
  cfg.blockDim = dim3(kGmThreads, 1, 1);
  cfg.dynamicSmemBytes = gemm_smem_bytes(p);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel, p, m.w, m.x[p.NT / 16 - 1]);
}

}  // namespace moe
