// The draft's context-KV projection: context rows -> every draft layer's keys
// and values, written into the KV cache.
//
// Page: vllm.models.muse_spark.common.dspark, _project_muse_context_kv and
// precompute_and_store_context_kv.  hidden_norm, then each layer's
// pre_qkv_proj_norm (bf16 outputs); each layer's stacked K/V rows of
// qkv_proj applied to its normalised rows (one batched bf16 GEMM, fp32
// accumulation, bf16 out); every key head normalised in fp32 without a weight
// and cast to bf16; the keys rotated by their positions (dimensions paired
// (j, j + D/2), angle pos * theta^(-2j/D), bf16 out); values passed through;
// keys and values scattered into the cache at their slots (negative = none).
//
// GB300 layout: three launches.  ctx_norm_kernel, one CTA per row, computes
// both norms and writes the L layer inputs.  Up to 8 rows the projection is
// the split-K weight-streaming kernel (gemv.cuh): fp32 partial sums per
// K-split, launched with programmatic dependent launch so its first weight
// loads overlap the norms; beyond 8 rows it is the library's tensor-core
// projection kernel (tc_gemm.cu), split-K partials while they fit the
// handle's buffer (summed here like the streaming kernel's), else bf16 K/V.
// kv_rope_kernel gives each (layer, row, head) one warp: it sums the partials
// in split order (or reads the GEMM's bf16 output), and the head's D values
// sit D/32 to a lane, so the key norm is a warp sum and the rotation's
// partner dimension (j + D/2) is 16 lanes away (one shuffle).  The rotation's
// cosines and sines come from a table built once at create in fp64.  After
// the streaming projection it does not wait for the whole grid: each task
// counts itself done per (layer, head) once its partials are stored, and a
// head's warps start when its count is complete (ctx_norm_kernel resets the
// counts each call, before the projection counts).

#include <cmath>
#include <cstdio>
#include <vector>

#include "../../include/moe_decode.h"
#include "common.cuh"
#include "gemv.cuh"
#include "tc_gemm.h"
#include "tc_ptx.cuh"
#include "moe_decode_internal.h"

namespace moe {
namespace {

struct CtxNormParams {
  int n, H, L;
  float eps;
  const __nv_bfloat16* ctx;  // [n][H]
  const float* w_hidden;     // [H]
  const float* w_pre;        // [L][H]
  __nv_bfloat16* fc;         // [n][H]
  __nv_bfloat16* u;          // [L][n][H]
  unsigned* done;            // the projection's per-head completion counters, reset here
  int n_done;
};

// Sum over the block, the result in every thread; red holds 32 floats.
__device__ float block_sum_all(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.0f;
  for (int i = 0; i < nw; ++i) t += red[i];
  __syncthreads();  // red is reused by the next sum
  return t;
}

__device__ __forceinline__ void unpack8(const uint4 raw, float (&v)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

constexpr int kNormChunks = 2;      // 8-column chunks per thread
constexpr int kNormPreLayers = 4;   // layers whose norm weights a thread loads up front

// One CTA per context row; chunks of 8 columns, kNormChunks per thread (thread
// t takes chunks t + j * blockDim).  Every load the thread needs -- its
// context columns, the hidden norm's weights and the first layers'
// pre-projection weights -- is issued at once, before the two reductions, so
// the kernel's latency is one memory round trip plus the reductions.
__global__ void __launch_bounds__(512, 1) ctx_norm_kernel(CtxNormParams p) {
  grid_dep_launch();  // the projection may start streaming its weights
  // this step's counters start from zero: the projection counts only after
  // this grid has completed, and its consumer launches only after that
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < p.n_done; i += blockDim.x) p.done[i] = 0u;
  __shared__ float red[32];
  const int r = blockIdx.x;
  const int nch = p.H / 8;
  uint4 craw[kNormChunks];
  float4 wh[kNormChunks][2];
  float4 wp[kNormPreLayers][kNormChunks][2];
#pragma unroll
  for (int j = 0; j < kNormChunks; ++j) {
    const int ch = threadIdx.x + j * blockDim.x, col = ch * 8;
    const bool live = ch < nch;
    craw[j] = live ? __ldg(reinterpret_cast<const uint4*>(p.ctx + (size_t)r * p.H + col)) : make_uint4(0u, 0u, 0u, 0u);
    wh[j][0] = live ? __ldg(reinterpret_cast<const float4*>(p.w_hidden + col)) : make_float4(0.f, 0.f, 0.f, 0.f);
    wh[j][1] = live ? __ldg(reinterpret_cast<const float4*>(p.w_hidden + col + 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int l = 0; l < kNormPreLayers; ++l)
      if (live && l < p.L) {
        wp[l][j][0] = __ldg(reinterpret_cast<const float4*>(p.w_pre + (size_t)l * p.H + col));
        wp[l][j][1] = __ldg(reinterpret_cast<const float4*>(p.w_pre + (size_t)l * p.H + col + 4));
      }
  }
  float c[kNormChunks][8];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < kNormChunks; ++j) {
    unpack8(craw[j], c[j]);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += c[j][i] * c[j][i];
  }
  const float inv_hidden = rsqrtf(block_sum_all(ss, red) / (float)p.H + p.eps);
  float f[kNormChunks][8];
  float ss2 = 0.0f;
#pragma unroll
  for (int j = 0; j < kNormChunks; ++j) {
    const int ch = threadIdx.x + j * blockDim.x;
    const float w[8] = {wh[j][0].x, wh[j][0].y, wh[j][0].z, wh[j][0].w,
                        wh[j][1].x, wh[j][1].y, wh[j][1].z, wh[j][1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[j][i] = __bfloat162float(__float2bfloat16_rn(c[j][i] * inv_hidden * w[i]));
      ss2 += f[j][i] * f[j][i];
    }
    if (ch < nch) *reinterpret_cast<uint4*>(p.fc + (size_t)r * p.H + ch * 8) = pack8(f[j]);
  }
  const float inv_pre = rsqrtf(block_sum_all(ss2, red) / (float)p.H + p.eps);
  auto write_layer = [&](int l, int j, float4 w0, float4 w1) {
    const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = f[j][i] * inv_pre * w[i];
    const int col = (threadIdx.x + j * blockDim.x) * 8;
    *reinterpret_cast<uint4*>(p.u + ((size_t)l * p.n + r) * p.H + col) = pack8(o);
  };
#pragma unroll
  for (int j = 0; j < kNormChunks; ++j) {
    if (threadIdx.x + j * blockDim.x >= nch) continue;
#pragma unroll
    for (int l = 0; l < kNormPreLayers; ++l)
      if (l < p.L) write_layer(l, j, wp[l][j][0], wp[l][j][1]);
    for (int l = kNormPreLayers; l < p.L; ++l) {
      const float* wl = p.w_pre + (size_t)l * p.H + (threadIdx.x + j * blockDim.x) * 8;
      write_layer(l, j, __ldg(reinterpret_cast<const float4*>(wl)), __ldg(reinterpret_cast<const float4*>(wl + 4)));
    }
  }
}

struct KvRopeParams {
  int n, L, KVH, D;
  float qk_eps;
  int max_pos;               // rows of the cos / sin table; 0 = no rotation
  const float2* cs;          // [max_pos][D/2]: (cos, sin)
  const int64_t* positions;  // [n]
  __nv_bfloat16* kv;         // [L][n][2 * KVH * D]: K heads, then V heads
  const float* part;         // [S][L][n][2 * KVH * D] split-K partials, or null: read kv
  int S;
  __nv_bfloat16* k_out;      // [L][n][KVH][D]
  __nv_bfloat16* v_out;
  const int64_t* slots;      // [L][slot_stride] (stride 0: one map), or null
  int slot_stride;
  int64_t n_slots;
  __nv_bfloat16* k_cache;  // [L][n_slots][KVH][D]
  __nv_bfloat16* v_cache;
  unsigned* err;
  // The streaming projection's per-(layer, head) completion counters, or
  // null (then the whole projection grid is waited for): a head's partials
  // are complete when its counter reaches done_target (its K and V row
  // groups times the splits).  The wait gives up after wait_ns.
  const unsigned* done;
  unsigned done_target;
  unsigned long long wait_ns;
};

constexpr unsigned kErrPosition = 3;  // a position outside the rotary table
constexpr unsigned kErrSlot = 4;      // a slot at or past n_slots

template <int E>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* src, float (&v)[E]) {
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(src + i));
    v[i] = f.x;
    v[i + 1] = f.y;
  }
}

template <int E>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* dst, const float (&v)[E]) {
#pragma unroll
  for (int i = 0; i < E; i += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + i) = __floats2bfloat162_rn(v[i], v[i + 1]);
}

// One warp per (layer, row, head); E = D / 32 values per lane.  With
// partials, the projection is their sum in split order, rounded to bf16 (and
// kept in kv); otherwise kv holds it.
template <int E>
__global__ void kv_rope_kernel(KvRopeParams p) {
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= p.L * p.n * p.KVH) return;
  const int hd = warp % p.KVH;
  const int r = (warp / p.KVH) % p.n;
  const int l = warp / (p.KVH * p.n);
  const int KD = p.KVH * p.D;
  __nv_bfloat16* row = p.kv + ((size_t)l * p.n + r) * 2 * KD;

  // The caller's positions and slots and the rotary table do not come from
  // the projection: read them before waiting for it.
  int64_t pos = 0;
  bool pos_ok = true;
  float2 t[E];
#pragma unroll
  for (int i = 0; i < E; ++i) t[i] = make_float2(1.0f, 0.0f);
  if (p.max_pos > 0) {
    pos = p.positions[r];
    pos_ok = pos >= 0 && pos < p.max_pos;
    if (pos_ok) {
      const float2* cs = p.cs + (size_t)pos * (p.D / 2) + (lane & 15) * E;
#pragma unroll
      for (int i = 0; i < E; ++i) t[i] = __ldg(cs + i);
    }
  }
  const int64_t slot = p.slots ? p.slots[(size_t)l * p.slot_stride + r] : -1;

  float k[E], v[E];
  if (p.part) {
#pragma unroll
    for (int i = 0; i < E; ++i) k[i] = v[i] = 0.0f;
    if (p.done) {
      // this head's tasks (every split of its K and V rows) have stored
      // their partials: a bounded wait on its counter, then every lane reads
      bool ok = true;
      if (lane == 0) {
        const unsigned* c = p.done + (size_t)l * p.KVH + hd;
        const uint64_t t0 = global_ns();
        while (tc::ld_acquire_u32(c) < p.done_target) {
          if (global_ns() - t0 > p.wait_ns) {
            latch_error(p.err, kDevWaitTimeout);
            ok = false;
            break;
          }
          __nanosleep(64);
        }
      }
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return;
    } else {
      grid_dep_wait();
    }
    const size_t split = (size_t)p.L * p.n * 2 * KD;
    const float* src = p.part + ((size_t)l * p.n + r) * 2 * KD + hd * p.D + lane * E;
    // eight splits' loads in flight at a time, summed in split order
    for (int s0 = 0; s0 < p.S; s0 += 8) {
      float pk[8][E], pv[8][E];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < E; ++i) {
          const bool in = s0 + j < p.S;
          pk[j][i] = in ? __ldcg(src + (size_t)(s0 + j) * split + i) : 0.0f;
          pv[j][i] = in ? __ldcg(src + (size_t)(s0 + j) * split + KD + i) : 0.0f;
        }
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < E; ++i) {
          k[i] += pk[j][i];
          v[i] += pv[j][i];
        }
    }
    store_bf16<E>(row + hd * p.D + lane * E, k);
    store_bf16<E>(row + KD + hd * p.D + lane * E, v);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      k[i] = __bfloat162float(__float2bfloat16_rn(k[i]));
      v[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
    }
  } else {
    load_bf16<E>(row + hd * p.D + lane * E, k);
    load_bf16<E>(row + KD + hd * p.D + lane * E, v);
  }
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < E; ++i) ss += k[i] * k[i];
  const float inv = rsqrtf(warp_sum(ss) / (float)p.D + p.qk_eps);
#pragma unroll
  for (int i = 0; i < E; ++i) k[i] = __bfloat162float(__float2bfloat16_rn(k[i] * inv));

  if (p.max_pos > 0) {
    if (!pos_ok) {
      if (lane == 0) latch_error(p.err, kErrPosition);
      return;
    }
    float y[E];
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float partner = __shfl_xor_sync(0xffffffffu, k[i], 16);
      // first half: x1 cos - x2 sin; second half: x2 cos + x1 sin
      y[i] = lane < 16 ? k[i] * t[i].x - partner * t[i].y : k[i] * t[i].x + partner * t[i].y;
    }
#pragma unroll
    for (int i = 0; i < E; ++i) k[i] = y[i];
  }

  const size_t o = (((size_t)l * p.n + r) * p.KVH + hd) * p.D + lane * E;
  store_bf16<E>(p.k_out + o, k);
  store_bf16<E>(p.v_out + o, v);
  if (p.slots) {
    if (slot >= p.n_slots) {
      if (lane == 0) latch_error(p.err, kErrSlot);
    } else if (slot >= 0) {
      const size_t c = (((size_t)l * p.n_slots + slot) * p.KVH + hd) * p.D + lane * E;
      store_bf16<E>(p.k_cache + c, k);
      store_bf16<E>(p.v_cache + c, v);
    }
  }
}

}  // namespace
}  // namespace moe

struct moe_ctxkv_s {
  moe_ctxkv_dims d;
  moe_ctxkv_weights w;
  moe::GemmMaps maps;               // the tensor-core projection's tensor maps (W_kv over u)
  int tc_part_rows;                 // up to this many rows its split-K partials fit the buffer
  int tc_max_splits;                // and this many splits; beyond, it writes bf16 kv directly
  void* base;                       // one allocation: the buffers below
  __nv_bfloat16 *fc, *u, *kv, *k, *v;
  float2* cs;                       // rotary table, or null
  unsigned* err;
  unsigned* done;                   // [L][KVH] the streaming projection's completion counters
  float* part;                      // split-K partials [S][L][rows][2 * KVH * D]
  int splits;                       // K-splits of the streaming projection; 0: none
  int num_sms;
  uint8_t* io;                      // host-buffer calls' copies: context [n][H] bf16,
                                    // positions [n], slots [L][n] int64 (when not mapped)
};

namespace {

constexpr size_t kCtxPartBudget = 64u << 20;  // bytes of split-K partials the handle keeps

bool ck_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int ck_cuda(cudaError_t e, const char* what) {
  char buf[200];
  snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  return moe::api_fail(MOE_ECUDA, buf);
}

struct ProjectArgs {
  int n;
  const uint16_t* context;
  const int64_t* positions;
  const int64_t* slots;
  int slot_stride;
  uint16_t* k_cache;
  uint16_t* v_cache;
  int64_t n_slots;
  uint16_t* k_out;
  uint16_t* v_out;
};

int check_project(const moe_ctxkv_t* h, const ProjectArgs& a) {
  const moe_ctxkv_dims& d = h->d;
  char buf[160];
  if (a.n < 1 || a.n > d.max_ctx) {
    snprintf(buf, sizeof(buf), "n_ctx %d outside [1, max_ctx=%d]", a.n, d.max_ctx);
    return moe::api_fail(MOE_EINVAL, buf);
  }
  if (!a.context || !ck_aligned(a.context, 16))
    return moe::api_fail(MOE_EINVAL, "context must be a 16-byte aligned device pointer");
  if (d.rope_theta > 0.0 && (!a.positions || !ck_aligned(a.positions, 8)))
    return moe::api_fail(MOE_EINVAL, "positions are required (8-byte aligned) with a rotary embedding");
  if (a.slots) {
    if (!ck_aligned(a.slots, 8)) return moe::api_fail(MOE_EINVAL, "slots must be 8-byte aligned");
    if (a.slot_stride != 0 && a.slot_stride < a.n)
      return moe::api_fail(MOE_EINVAL, "slot_stride must be 0 (one map) or at least n_ctx");
    if (!a.k_cache || !a.v_cache || a.n_slots < 1 || !ck_aligned(a.k_cache, 16) || !ck_aligned(a.v_cache, 16))
      return moe::api_fail(MOE_EINVAL, "slots need 16-byte aligned K and V caches and n_slots >= 1");
  }
  if ((a.k_out && !ck_aligned(a.k_out, 16)) || (a.v_out && !ck_aligned(a.v_out, 16)))
    return moe::api_fail(MOE_EINVAL, "k_out and v_out must be 16-byte aligned");
  return MOE_OK;
}

// The three launches on s; with ev, an event before each and after the last.
int ctxkv_enqueue(moe_ctxkv_t* h, const ProjectArgs& a, cudaStream_t s, cudaEvent_t* ev) {
  const moe_ctxkv_dims& d = h->d;
  auto mark = [&](int i) {
    if (ev) cudaEventRecord(ev[i], s);
  };
  const int KD = d.n_kv_heads * d.head_dim;
  mark(0);
  moe::CtxNormParams np{};
  np.n = a.n;
  np.H = d.hidden;
  np.L = d.n_layers;
  np.eps = d.eps;
  np.ctx = reinterpret_cast<const __nv_bfloat16*>(a.context);
  np.w_hidden = h->w.w_hidden;
  np.w_pre = h->w.w_pre;
  np.fc = h->fc;
  np.u = h->u;
  np.done = h->done;
  np.n_done = d.n_layers * d.n_kv_heads;
  const bool stream_w = h->splits > 0 && a.n <= 8;
  moe::GemmParams gp_tc;
  int tc_S = 0;  // the tensor-core projection's splits when it left partials
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n, 1, 1);
  cfg.blockDim = dim3(((d.hidden / 8 + moe::kNormChunks - 1) / moe::kNormChunks + 31) / 32 * 32, 1, 1);
  cfg.stream = s;
  cudaError_t e = cudaLaunchKernelEx(&cfg, moe::ctx_norm_kernel, np);
  if (e != cudaSuccess) return ck_cuda(e, "context norm launch");
  mark(1);
  if (stream_w) {
    moe::GemvParams gp{};
    gp.W = reinterpret_cast<const __nv_bfloat16*>(h->w.w_kv);
    gp.X = h->u;
    gp.part = h->part;
    gp.L = d.n_layers;
    gp.R = 2 * KD;
    gp.K = d.hidden;
    gp.n = a.n;
    gp.S = h->splits;
    gp.KC = d.hidden / h->splits;
    gp.done = h->done;
    gp.done_mod = KD;
    gp.done_div = d.head_dim;
    cudaLaunchConfig_t gc = {};
    gc.gridDim = dim3(h->num_sms, 1, 1);
    gc.blockDim = dim3(moe::kGemvThreads, 1, 1);
    gc.dynamicSmemBytes = moe::kGemvSmem;
    gc.stream = s;
    gc.attrs = ev ? nullptr : &pdl;  // profiled launches are timed one at a time
    gc.numAttrs = ev ? 0 : 1;
    e = cudaLaunchKernelEx(&gc, moe::gemv_bf16_kernel<false>, gp);
    if (e != cudaSuccess) return ck_cuda(e, "K/V projection launch");
  } else {
    // the tensor-core projection: split-K partials while they fit the
    // handle's buffer, else the bf16 projection itself
    const bool partial = a.n <= h->tc_part_rows;
    if (!moe::plan_gemm(gp_tc, partial ? moe::kGemmPartial : moe::kGemmBf16, d.n_layers, 2 * KD, d.hidden,
                        a.n, 0, a.n, h->num_sms, partial ? h->tc_max_splits : 1))
      return moe::api_fail(MOE_EUNSUPPORTED, "no tensor-core plan for the K/V projection");
    gp_tc.part = h->part;
    gp_tc.out = h->kv;
    gp_tc.err = h->err;
    e = moe::launch_gemm(gp_tc, h->maps, h->num_sms, s, !ev);
    if (e != cudaSuccess) return ck_cuda(e, "K/V projection launch");
    tc_S = partial ? gp_tc.S : 0;
  }
  mark(2);
  moe::KvRopeParams kp{};
  kp.n = a.n;
  kp.L = d.n_layers;
  kp.KVH = d.n_kv_heads;
  kp.D = d.head_dim;
  kp.qk_eps = d.qk_eps;
  kp.max_pos = h->cs ? d.max_position : 0;
  kp.cs = h->cs;
  kp.positions = a.positions;
  kp.kv = h->kv;
  kp.part = (stream_w || tc_S) ? h->part : nullptr;
  kp.S = stream_w ? h->splits : tc_S;
  kp.k_out = a.k_out ? reinterpret_cast<__nv_bfloat16*>(a.k_out) : h->k;
  kp.v_out = a.v_out ? reinterpret_cast<__nv_bfloat16*>(a.v_out) : h->v;
  kp.slots = a.slots;
  kp.slot_stride = a.slot_stride;
  kp.n_slots = a.n_slots;
  kp.k_cache = reinterpret_cast<__nv_bfloat16*>(a.k_cache);
  kp.v_cache = reinterpret_cast<__nv_bfloat16*>(a.v_cache);
  kp.err = h->err;
  kp.done = stream_w ? h->done : nullptr;
  kp.done_target = (unsigned)(2 * (d.head_dim / 32) * h->splits);
  kp.wait_ns = moe::kDefaultWaitNs;
  const long long warps = (long long)d.n_layers * a.n * d.n_kv_heads;
  // CTAs of 4 warps, small enough to be resident beside a streaming
  // projection CTA, so that a head's warps start as its counter completes
  cudaLaunchConfig_t rc = {};
  rc.gridDim = dim3((unsigned)((warps * 32 + 127) / 128), 1, 1);
  rc.blockDim = dim3(128, 1, 1);
  rc.stream = s;
  rc.attrs = (stream_w && !ev) ? &pdl : nullptr;
  rc.numAttrs = (stream_w && !ev) ? 1 : 0;
  switch (d.head_dim) {
    case 64: e = cudaLaunchKernelEx(&rc, moe::kv_rope_kernel<2>, kp); break;
    case 128: e = cudaLaunchKernelEx(&rc, moe::kv_rope_kernel<4>, kp); break;
    default: e = cudaLaunchKernelEx(&rc, moe::kv_rope_kernel<8>, kp); break;
  }
  if (e != cudaSuccess) return ck_cuda(e, "key norm / rotary launch");
  mark(3);
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_ctxkv_create(const moe_ctxkv_dims* dims, const moe_ctxkv_weights* w, moe_ctxkv_t** out) {
  if (!dims || !w || !out) return moe::api_fail(MOE_EINVAL, "dims, weights and out are required");
  *out = nullptr;
  const moe_ctxkv_dims d = *dims;
  if (d.hidden < 8 || d.hidden % 8 || d.hidden > 8192)
    return moe::api_fail(MOE_EUNSUPPORTED, "hidden must be a multiple of 8 in [8, 8192]");
  if (d.n_layers < 1 || d.n_layers > 256) return moe::api_fail(MOE_EUNSUPPORTED, "n_layers must be in [1, 256]");
  if (d.head_dim != 64 && d.head_dim != 128 && d.head_dim != 256)
    return moe::api_fail(MOE_EUNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (d.n_kv_heads < 1 || d.n_kv_heads * d.head_dim > 32768)
    return moe::api_fail(MOE_EUNSUPPORTED, "n_kv_heads * head_dim must be in [head_dim, 32768]");
  if (d.max_ctx < 1 || d.max_ctx > 65536) return moe::api_fail(MOE_EUNSUPPORTED, "max_ctx must be in [1, 65536]");
  if ((long long)d.n_layers * d.max_ctx * d.n_kv_heads * 32 >= (1ll << 31))
    return moe::api_fail(MOE_EUNSUPPORTED, "n_layers * max_ctx * n_kv_heads must be below 2^26");
  if (!(d.eps > 0.0f) || !(d.qk_eps > 0.0f)) return moe::api_fail(MOE_EINVAL, "eps and qk_eps must be positive");
  if (!(d.rope_theta >= 0.0)) return moe::api_fail(MOE_EINVAL, "rope_theta must be >= 0 (0: no rotary embedding)");
  if (d.rope_theta > 0.0 && (d.max_position < 1 || d.max_position > (1 << 20)))
    return moe::api_fail(MOE_EUNSUPPORTED, "max_position must be in [1, 2^20] with a rotary embedding");
  if (!w->w_hidden || !w->w_pre || !w->w_kv) return moe::api_fail(MOE_EINVAL, "a required weight pointer is NULL");
  if (!ck_aligned(w->w_hidden, 16) || !ck_aligned(w->w_pre, 16) || !ck_aligned(w->w_kv, 16))
    return moe::api_fail(MOE_EINVAL, "weight pointers must be 16-byte aligned");
  int dev = 0, major = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return ck_cuda(e, "device query");
  if (major != 10) return moe::api_fail(MOE_EUNSUPPORTED, "needs an SM 10.x GPU");

  moe_ctxkv_t* h = new moe_ctxkv_t{};
  h->d = d;
  h->w = *w;
  const size_t n = d.max_ctx, H = d.hidden, L = d.n_layers, KD = (size_t)d.n_kv_heads * d.head_dim;
  const size_t table = d.rope_theta > 0.0 ? (size_t)d.max_position * (d.head_dim / 2) : 0;
  int num_sms = 0;
  e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    delete h;
    return ck_cuda(e, "device query");
  }
  h->num_sms = num_sms;
  h->splits = moe::gemv_splits(d.n_layers, 2 * d.n_kv_heads * d.head_dim, d.hidden, num_sms);
  if (h->splits) {
    e = cudaFuncSetAttribute(moe::gemv_bf16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)moe::kGemvSmem);
    if (e != cudaSuccess) {
      delete h;
      return ck_cuda(e, "streaming projection shared memory");
    }
  }
  e = moe::gemm_set_smem();
  if (e != cudaSuccess) {
    delete h;
    return ck_cuda(e, "tensor-core projection shared memory");
  }
  // the tensor-core projection's partials: up to 128 rows and 8 splits,
  // fewer splits (or none: bf16 output) when the budget does not hold them
  h->tc_part_rows = (int)(n < 128 ? n : 128);
  const size_t per_split = L * (size_t)h->tc_part_rows * 2 * KD * sizeof(float);
  h->tc_max_splits = (int)(kCtxPartBudget / per_split < 8 ? kCtxPartBudget / per_split : 8);
  if (h->tc_max_splits == 0) h->tc_part_rows = 0;
  const size_t part_stream = h->splits ? (size_t)h->splits * L * 8 * 2 * KD * sizeof(float) : 0;
  const size_t part_tc = (size_t)h->tc_max_splits * per_split;
  const size_t b_part = part_stream > part_tc ? part_stream : part_tc;
  auto up16 = [](size_t b) { return (b + 15) & ~(size_t)15; };
  const size_t b_fc = up16(2 * n * H), b_u = up16(2 * L * n * H), b_kv = up16(2 * L * n * 2 * KD),
               b_k = up16(2 * L * n * KD), b_cs = table * sizeof(float2);
  const size_t b_io = up16(2 * n * H) + up16(8 * n) + up16(8 * L * n);
  const size_t b_done = up16(sizeof(unsigned) * L * d.n_kv_heads);
  const size_t bytes = b_part + b_fc + b_u + b_kv + 2 * b_k + b_cs + 16 + b_done + b_io;
  uint8_t* base = nullptr;
  e = cudaMalloc(&base, bytes);
  if (e != cudaSuccess) {
    cudaFree(base);
    moe_ctxkv_destroy(h);
    return moe::api_fail(MOE_ENOMEM, "context-KV workspace");
  }
  h->base = base;
  h->part = b_part ? reinterpret_cast<float*>(base) : nullptr;
  base += b_part;
  h->fc = reinterpret_cast<__nv_bfloat16*>(base);
  h->u = reinterpret_cast<__nv_bfloat16*>(base + b_fc);
  h->kv = reinterpret_cast<__nv_bfloat16*>(base + b_fc + b_u);
  h->k = reinterpret_cast<__nv_bfloat16*>(base + b_fc + b_u + b_kv);
  h->v = reinterpret_cast<__nv_bfloat16*>(base + b_fc + b_u + b_kv + b_k);
  h->cs = table ? reinterpret_cast<float2*>(base + b_fc + b_u + b_kv + 2 * b_k) : nullptr;
  h->err = reinterpret_cast<unsigned*>(base + b_fc + b_u + b_kv + 2 * b_k + b_cs);
  h->done = reinterpret_cast<unsigned*>(base + b_fc + b_u + b_kv + 2 * b_k + b_cs + 16);
  h->io = base + b_fc + b_u + b_kv + 2 * b_k + b_cs + 16 + b_done;
  e = cudaMemset(h->err, 0, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(h->done, 0, b_done);
  if (e == cudaSuccess && table) {
    // cos / sin of pos * theta^(-2j/D) in fp64, stored as fp32
    const int half = d.head_dim / 2;
    std::vector<double> freq(half);
    for (int j = 0; j < half; ++j) freq[j] = std::pow(d.rope_theta, -2.0 * j / d.head_dim);
    std::vector<float2> host(table);
    for (size_t pos = 0; pos < (size_t)d.max_position; ++pos)
      for (int j = 0; j < half; ++j) {
        const double ang = (double)pos * freq[j];
        host[pos * half + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    e = cudaMemcpy(h->cs, host.data(), b_cs, cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    moe_ctxkv_destroy(h);
    return ck_cuda(e, "context-KV set-up");
  }
  // W_kv [L * 2KD][H] over u [L * max_ctx][H]
  e = moe::encode_gemm_maps(h->maps, h->w.w_kv, (int64_t)L * 2 * KD, h->u, (int64_t)L * n, (int)H);
  if (e != cudaSuccess) {
    moe_ctxkv_destroy(h);
    return ck_cuda(e, "K/V projection tensor maps");
  }
  *out = h;
  return MOE_OK;
}

int moe_ctxkv_project(moe_ctxkv_t* h, int n_ctx, const uint16_t* context, const int64_t* positions,
                      const int64_t* slots, int slot_stride, uint16_t* k_cache, uint16_t* v_cache,
                      int64_t n_slots, uint16_t* k_out, uint16_t* v_out, void* cuda_stream) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  const ProjectArgs a{n_ctx, context, positions, slots, slot_stride, k_cache, v_cache, n_slots, k_out, v_out};
  int rc = check_project(h, a);
  if (rc) return rc;
  return ctxkv_enqueue(h, a, static_cast<cudaStream_t>(cuda_stream), nullptr);
}

int moe_ctxkv_project_host(moe_ctxkv_t* h, int n_ctx, const uint16_t* context_host,
                           const int64_t* positions_host, const int64_t* slots_host, int slot_stride,
                           uint16_t* k_cache, uint16_t* v_cache, int64_t n_slots, uint16_t* k_out_host,
                           uint16_t* v_out_host, void* cuda_stream) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  if (!context_host || !k_out_host || !v_out_host)
    return moe::api_fail(MOE_EINVAL, "context_host, k_out_host and v_out_host are required");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const moe_ctxkv_dims& d = h->d;
  const int n = n_ctx;
  if (n < 1 || n > d.max_ctx) return moe::api_fail(MOE_EINVAL, "n_ctx outside [1, max_ctx]");
  const size_t kv_bytes = (size_t)d.n_layers * n * d.n_kv_heads * d.head_dim * 2;
  const size_t slot_count = slots_host ? (size_t)(slot_stride ? d.n_layers : 1) * (slot_stride ? slot_stride : n) : 0;
  // mapped page-locked buffers are read and written by the kernels directly
  const uint16_t* ctx_d = static_cast<const uint16_t*>(moe::host_mapped(context_host));
  const int64_t* pos_d = static_cast<const int64_t*>(moe::host_mapped(positions_host));
  const int64_t* slots_d = static_cast<const int64_t*>(moe::host_mapped(slots_host));
  uint16_t* k_d = static_cast<uint16_t*>(moe::host_mapped(k_out_host));
  uint16_t* v_d = static_cast<uint16_t*>(moe::host_mapped(v_out_host));
  const bool direct = ctx_d && k_d && v_d && (!positions_host || pos_d) && (!slots_host || slots_d);
  cudaError_t e = cudaSuccess;
  if (!direct) {
    // copies in: context, positions, slots into the handle's buffers
    uint8_t* io = h->io;
    const size_t b_ctx = ((size_t)2 * d.max_ctx * d.hidden + 15) & ~(size_t)15;
    const size_t b_pos = ((size_t)8 * d.max_ctx + 15) & ~(size_t)15;
    if ((size_t)slot_count > (size_t)d.n_layers * d.max_ctx)
      return moe::api_fail(MOE_EINVAL, "slot map larger than n_layers * max_ctx");
    ctx_d = reinterpret_cast<const uint16_t*>(io);
    pos_d = positions_host ? reinterpret_cast<const int64_t*>(io + b_ctx) : nullptr;
    slots_d = slots_host ? reinterpret_cast<const int64_t*>(io + b_ctx + b_pos) : nullptr;
    e = cudaMemcpyAsync(io, context_host, (size_t)n * d.hidden * 2, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && positions_host)
      e = cudaMemcpyAsync(io + b_ctx, positions_host, (size_t)n * 8, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && slots_host)
      e = cudaMemcpyAsync(io + b_ctx + b_pos, slots_host, slot_count * 8, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return ck_cuda(e, "input copy");
    k_d = nullptr;  // the workspace's keys and values, copied out below
    v_d = nullptr;
  }
  const ProjectArgs a{n, ctx_d, pos_d, slots_d, slot_stride, k_cache, v_cache, n_slots, k_d, v_d};
  int rc = check_project(h, a);
  if (rc) return rc;
  rc = ctxkv_enqueue(h, a, s, nullptr);
  if (rc) return rc;
  if (!direct) {
    e = cudaMemcpyAsync(k_out_host, h->k, kv_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(v_out_host, h->v, kv_bytes, cudaMemcpyDeviceToHost, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return ck_cuda(e, "host-buffer projection");
  return MOE_OK;
}

int moe_ctxkv_profile(moe_ctxkv_t* h, int n_ctx, const uint16_t* context, const int64_t* positions,
                      const int64_t* slots, int slot_stride, uint16_t* k_cache, uint16_t* v_cache,
                      int64_t n_slots, void* cuda_stream, float* ms_host) {
  if (!h || !ms_host) return moe::api_fail(MOE_EINVAL, "handle and ms_host are required");
  const ProjectArgs a{n_ctx, context, positions, slots, slot_stride, k_cache, v_cache, n_slots, nullptr, nullptr};
  int rc = check_project(h, a);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaEvent_t ev[4] = {};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 4 && e == cudaSuccess; ++i) e = cudaEventCreate(&ev[i]);
  if (e == cudaSuccess) {
    rc = ctxkv_enqueue(h, a, s, ev);
    if (!rc) e = cudaEventSynchronize(ev[3]);
    for (int i = 0; i < 3 && !rc && e == cudaSuccess; ++i) e = cudaEventElapsedTime(&ms_host[i], ev[i], ev[i + 1]);
  }
  for (int i = 0; i < 4; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  if (rc) return rc;
  if (e != cudaSuccess) return ck_cuda(e, "profile events");
  return MOE_OK;
}

int moe_ctxkv_kernel_count(moe_ctxkv_t* h, int n_ctx) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  // capture one projection of n_ctx rows on a private stream (the handle's
  // own buffers as inputs, no cache write; nothing runs) and count the
  // graph's kernel nodes
  const ProjectArgs a{n_ctx, reinterpret_cast<const uint16_t*>(h->fc), reinterpret_cast<const int64_t*>(h->k),
                      nullptr, 0, nullptr, nullptr, 0, nullptr, nullptr};
  int rc = check_project(h, a);
  if (rc) return rc;
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return ck_cuda(e, "stream create");
  cudaGraph_t g = nullptr;
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    rc = ctxkv_enqueue(h, a, s, nullptr);
    e = cudaStreamEndCapture(s, &g);
  }
  int count = 0;
  size_t nn = 0;
  if (e == cudaSuccess && !rc) e = cudaGraphGetNodes(g, nullptr, &nn);
  if (e == cudaSuccess && !rc && nn) {
    std::vector<cudaGraphNode_t> nodes(nn);
    e = cudaGraphGetNodes(g, nodes.data(), &nn);
    for (size_t i = 0; i < nn && e == cudaSuccess; ++i) {
      cudaGraphNodeType t;
      e = cudaGraphNodeGetType(nodes[i], &t);
      count += (t == cudaGraphNodeTypeKernel);
    }
  }
  if (g) cudaGraphDestroy(g);
  cudaStreamDestroy(s);
  if (rc) return rc;
  if (e != cudaSuccess) return ck_cuda(e, "launch count capture");
  return count;
}

int moe_ctxkv_debug(moe_ctxkv_t* h, moe_ctxkv_debug_view* v) {
  if (!h || !v) return moe::api_fail(MOE_EINVAL, "handle and view are required");
  v->fc = h->fc;
  v->u = h->u;
  v->kv = h->kv;
  v->k = h->k;
  v->v = h->v;
  return MOE_OK;
}

int moe_ctxkv_last_error(moe_ctxkv_t* h) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return ck_cuda(e, "device synchronize");
  unsigned flag = 0;
  e = cudaMemcpy(&flag, h->err, sizeof(flag), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return ck_cuda(e, "error flag read");
  if (flag) {
    cudaMemset(h->err, 0, sizeof(unsigned));
    char buf[160];
    snprintf(buf, sizeof(buf), "device-side error %u: %s", flag,
             flag == moe::kErrPosition     ? "a position outside [0, max_position)"
             : flag == moe::kErrSlot       ? "a slot at or past n_slots"
             : flag == moe::kDevWaitTimeout ? "a bounded wait gave up"
                                           : "unknown");
    return moe::api_fail(MOE_EDEVICE, buf);
  }
  return MOE_OK;
}

void moe_ctxkv_destroy(moe_ctxkv_t* h) {
  if (!h) return;
  cudaFree(h->base);
  delete h;
}

}  // extern "C"
