// Routed NVFP4 experts: gate/up + SiLU*mul (+ the intermediate's NVFP4
// quantization) and down, as two launches of one persistent kernel.
//
// Page: vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode,
// module docstring "One step of b rows", MoE: "... pooler -> routed experts
// -> tail -> unpooler"; SpecializedDecode.build: "The routed expert ops of
// every layer"; gate_proj / up_proj stacked as shards 0 / 1 of gate_up_proj
// (MuseSparkDSparkForCausalLM weight mapping on the DSpark page).
//
// Per pair (row r, slot s) routed to expert e:
//   G_j = sum_k Wg[e][j][k] xq[r][k],  U_j = sum_k Wu[e][j][k] xq[r][k]
//   h_j = silu(G_j) * U_j                                   (fp32)
//   h quantized to NVFP4 with one global scale per expert (its pairs' rows)
//   o[pair][i] = sum_j Wd[e][i][j] hq[pair][j]              (fp32)
// with every operand NVFP4: value = e2m1 code * e4m3 block scale (per 16)
// * fp32 tensor scale.
//
// GB300 design (decode batches: the weight stream is the whole cost):
//  - One persistent CTA per SM.  Work item = (active expert, tile of weight
//    rows); each CTA takes a contiguous run of items, so it streams a long
//    contiguous stretch of each expert's weights.
//  - Each item's packed codes and e4m3 scales move global -> shared with
//    bulk async copies (evict-first in L2) into a ring of stages tracked by
//    mbarriers (complete_tx); thread 0 refills a stage as soon as the
//    per-item barrier shows every thread is done with it, so the copies of
//    the next NS-1 items (~130-190 KB per SM) are in flight ahead of the math.
//  - Sixteen warps per SM (at most 128 registers a thread).  Each thread
//    owns a fixed 16-byte column chunk (32 elements, two 16-blocks) of every
//    weight row; the expert's activation rows for that chunk stay in
//    registers.  Two exact ways to form a 16-block dot product, chosen per
//    expert by its number of rows:
//      1-2 rows: the hardware e2m1x2 -> f16x2 conversion and f16x2 fused
//        multiply-adds.  e2m1 products are multiples of 1/4 below 36, so
//        four-term partial sums (< 144) and their pairwise sums (< 288) are
//        exact in f16, and so is their fp32 total.
//      3+ rows (groups of 4): byte-permute table lookups turn codes into
//        signed bytes (2 x value) and four dp4a give the exact int32 sum.
//    The block result is scaled by the exact fp32 product of the two e4m3
//    scales and accumulated in fp32.  (Measured on GB300 from shared memory:
//    ~57 weight elements/cycle/SM for the f16 path at 1 row and 16 warps,
//    ~39 for dp4a; 29 vs 20 at 4 rows.)
//  - Partial sums are reduced across the row's threads with a warp
//    reduce-scatter (one value per lane, not one reduction per value) and a
//    fixed-order sum across warps: deterministic, no float atomics.
//  - Gate/up: the CTA that finishes an expert's last tile (threadfence +
//    per-expert counter, no spin) quantizes that expert's h rows.
//  - Down: its producer starts streaming expert weights before the
//    programmatic-dependency wait (routing is already final), so the
//    gate/up kernel's tail overlaps the down kernel's first loads.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kMaxThreads = 512;
constexpr int kMaxWarps = kMaxThreads / 32;
constexpr int kRedFloats = kMaxWarps * 32;   // one reduction buffer: 16 warps x 32 values
constexpr int kMaxPairs = 128;               // pairs of one expert <= rows <= 128
constexpr int kExpertTable = 64;             // experts of one CTA's run kept in smem
constexpr int kCtrlBytes = 512 + kExpertTable * 16 + 2 * kRedFloats * 4 + kMaxPairs * 4 + 64;
constexpr int kCtrlRounded = (kCtrlBytes + 1023) / 1024 * 1024;

// Shared memory: [barriers + stage metadata | expert table | 2 reduction
// buffers | pair ids of the current expert | flags] then the stage ring.
struct Smem {
  uint64_t* full;
  int4* meta;       // per stage: expert, tile, first pooled position, pairs
  int4* etab;       // this CTA's experts in run order: expert, first position, pairs
  float* red;       // [2][kRedFloats]
  int* pairs;       // [kMaxPairs] pair ids of the current expert (down)
  int* flag;        // last-CTA verdict of finish_expert
  int* ok;          // stage verdict of the current item
  uint8_t* stages;
};

__device__ __forceinline__ Smem carve(uint8_t* base) {
  Smem s;
  s.full = reinterpret_cast<uint64_t*>(base);        // 16 x 8 B
  s.meta = reinterpret_cast<int4*>(base + 256);      // 16 x 16 B
  s.etab = reinterpret_cast<int4*>(base + 512);      // kExpertTable x 16 B
  s.red = reinterpret_cast<float*>(base + 512 + kExpertTable * 16);
  s.pairs = reinterpret_cast<int*>(base + 512 + kExpertTable * 16 + 2 * kRedFloats * 4);
  s.flag = s.pairs + kMaxPairs;
  s.ok = s.flag + 1;
  s.stages = base + kCtrlRounded;
  return s;
}

// Reduce-scatter of V values (V a power of two <= 32) across the 32 lanes;
// lane results land in dst[index] (lanes holding the same index write once).
template <int V>
__device__ __forceinline__ void warp_reduce_scatter_store(float (&v)[V], int lane, float* dst) {
  static_assert(V >= 1 && V <= 32 && (V & (V - 1)) == 0, "V: a power of two <= 32");
  constexpr int kSteps = (V == 32) ? 5 : (V == 16 ? 4 : (V == 8 ? 3 : (V == 4 ? 2 : (V == 2 ? 1 : 0))));
  int base = 0;
#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
    const int off = 16 >> st;
    const int n = V >> st;  // values still held
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
    if (upper) base += n / 2;
  }
#pragma unroll
  for (int st = kSteps; st < 5; ++st) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16 >> st);
  const int low_bits = (1 << (5 - kSteps)) - 1;
  if ((lane & low_bits) == 0) dst[base] = v[0];
}

// e2m1 pair in the low byte -> f16x2 (exact).
__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte_in_low) {
  uint32_t r;
  const unsigned short in = static_cast<unsigned short>(byte_in_low);
  asm("{\n\t.reg .b8 t, z;\n\tmov.b16 {t, z}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "h"(in));
  return r;
}

__device__ __forceinline__ void chunk_to_f16(const uint4 c, uint32_t* h) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 16; ++q) h[q] = cvt_e2m1x2_f16x2(w[q >> 2] >> (8 * (q & 3)));
}

__device__ __forceinline__ void chunk_to_s8(const uint4 c, uint32_t* v) {
  e2m1x8_to_s8x8(c.x, v[0], v[1]);
  e2m1x8_to_s8x8(c.y, v[2], v[3]);
  e2m1x8_to_s8x8(c.z, v[4], v[5]);
  e2m1x8_to_s8x8(c.w, v[6], v[7]);
}

// Activation rows [pos0, pos0 + rb) of the expert for this thread's chunk:
// F16 layout av[a*16 + q] (f16x2 of byte q) or signed-byte layout av[a*8 + q].
template <int RB, bool kF16>
__device__ __forceinline__ void load_act(const ExpertParams& p, bool gate_up, int pos0, int rb,
                                         int cc, bool live, uint32_t (&av)[32],
                                         float (&sx)[4][2]) {
  const Workspace& ws = p.ws;
  const uint8_t* codes = gate_up ? ws.x_codes : ws.h_codes;
  const uint8_t* sf = gate_up ? ws.x_sf : ws.h_sf;
  constexpr int W = kF16 ? 16 : 8;
#pragma unroll
  for (int a = 0; a < RB; ++a) {
    if (a < rb && live) {
      const int pos = pos0 + a;
      int row = gate_up ? __ldcg(ws.pair_order + pos) / p.k : pos;
      if (!MOE_IN_BOUNDS(row >= 0 && row < p.ws_pairs, ws.err)) row = 0;
      const uint4 c = __ldcg(reinterpret_cast<const uint4*>(codes + (size_t)row * p.KB) + cc);
      if (kF16)
        chunk_to_f16(c, av + a * W);
      else
        chunk_to_s8(c, av + a * W);
      const unsigned short s2 =
          __ldcg(reinterpret_cast<const unsigned short*>(sf + (size_t)row * p.KS) + cc);
      const float2 f = e4m3x2_to_f32x2(s2);
      sx[a][0] = f.x;
      sx[a][1] = f.y;
    } else {
#pragma unroll
      for (int q = 0; q < W; ++q) av[a * W + q] = 0u;
      sx[a][0] = sx[a][1] = 0.0f;
    }
  }
}

__device__ __forceinline__ __half2 h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Dot products of this thread's chunk of the group's TW weight rows with the
// RB activation rows held in registers.
template <int TW, int RB, bool kF16>
__device__ __forceinline__ void gemv_chunk(const ExpertParams& p, const uint8_t* stage, int g,
                                           int cc, bool live, const uint32_t (&av)[32],
                                           const float (&sx)[4][2], float (&acc)[TW * RB]) {
#pragma unroll
  for (int i = 0; i < TW * RB; ++i) acc[i] = 0.0f;
  if (!live) return;
  const uint8_t* sc = stage + (size_t)cc * 16 + (size_t)g * TW * p.KB;
  const uint8_t* ss = stage + (size_t)p.T * p.KB + (size_t)cc * 2 + (size_t)g * TW * p.KS;
#pragma unroll
  for (int t = 0; t < TW; ++t) {
    const uint4 c = *reinterpret_cast<const uint4*>(sc + (size_t)t * p.KB);
    const unsigned short s2 = *reinterpret_cast<const unsigned short*>(ss + (size_t)t * p.KS);
    const float2 sw = e4m3x2_to_f32x2(s2);
    if (kF16) {
      uint32_t wh[16];
      chunk_to_f16(c, wh);
#pragma unroll
      for (int a = 0; a < RB; ++a) {
        const uint32_t* x = av + a * 16;
        // four-term exact partials, then exact pairwise sums per 16-block
        __half2 pa = __hmul2(h2(wh[0]), h2(x[0]));
        __half2 pb = __hmul2(h2(wh[4]), h2(x[4]));
        __half2 pc = __hmul2(h2(wh[8]), h2(x[8]));
        __half2 pd = __hmul2(h2(wh[12]), h2(x[12]));
#pragma unroll
        for (int q = 1; q < 4; ++q) {
          pa = __hfma2(h2(wh[q]), h2(x[q]), pa);
          pb = __hfma2(h2(wh[4 + q]), h2(x[4 + q]), pb);
          pc = __hfma2(h2(wh[8 + q]), h2(x[8 + q]), pc);
          pd = __hfma2(h2(wh[12 + q]), h2(x[12 + q]), pd);
        }
        const float2 f0 = __half22float2(__hadd2(pa, pb));
        const float2 f1 = __half22float2(__hadd2(pc, pd));
        float acc_v = acc[t * RB + a];
        acc_v = fmaf(f0.x + f0.y, sw.x * sx[a][0], acc_v);
        acc_v = fmaf(f1.x + f1.y, sw.y * sx[a][1], acc_v);
        acc[t * RB + a] = acc_v;
      }
    } else {
      uint32_t wv[8];
      chunk_to_s8(c, wv);
#pragma unroll
      for (int a = 0; a < RB; ++a) {
        const uint32_t* x = av + a * 8;
        int d0 = __dp4a((int)wv[0], (int)x[0], 0);
        d0 = __dp4a((int)wv[1], (int)x[1], d0);
        d0 = __dp4a((int)wv[2], (int)x[2], d0);
        d0 = __dp4a((int)wv[3], (int)x[3], d0);
        int d1 = __dp4a((int)wv[4], (int)x[4], 0);
        d1 = __dp4a((int)wv[5], (int)x[5], d1);
        d1 = __dp4a((int)wv[6], (int)x[6], d1);
        d1 = __dp4a((int)wv[7], (int)x[7], d1);
        float acc_v = acc[t * RB + a];
        // signed bytes carry 2 x value: the block sum is 4 x sum(w x)
        acc_v = fmaf((float)d0 * 0.25f, sw.x * sx[a][0], acc_v);
        acc_v = fmaf((float)d1 * 0.25f, sw.y * sx[a][1], acc_v);
        acc[t * RB + a] = acc_v;
      }
    }
  }
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// One activation-row group (RB rows) of one item: dot products, reduction,
// epilogue (h for gate/up, o for down).  `red` alternates between the two
// reduction buffers, so one barrier per group suffices.
template <int TW, int RB, bool kF16, bool kGU>
__device__ __forceinline__ void run_group(const ExpertParams& p, const Smem& sm, float* red,
                                          const uint8_t* stage, int tile, int pos0, int a0, int rb,
                                          int tid, int NC, const uint32_t (&av)[32],
                                          const float (&sx)[4][2], float sc0, float sc1,
                                          float& amax_out) {
  const int g = tid / p.TPG, cc = tid % p.TPG;
  const bool live = cc < p.CH;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int V = TW * RB;
  float acc[V];
  gemv_chunk<TW, RB, kF16>(p, stage, g, cc, live, av, sx, acc);
  warp_reduce_scatter_store<V>(acc, lane, red + warp * V);
  named_bar(1, NC);
  const int wpg = p.TPG / 32;
  const Workspace& ws = p.ws;
  if (kGU) {
    float m = 0.0f;
    for (int q = tid; q < p.TJ * rb; q += NC) {
      const int j = q % p.TJ, a = q / p.TJ;
      const int wg = j, wu = p.TJ + j;  // stage rows of gate j and up j
      float G = 0.0f, U = 0.0f;
      for (int i = 0; i < wpg; ++i) G += red[((wg / TW) * wpg + i) * V + (wg % TW) * RB + a];
      for (int i = 0; i < wpg; ++i) U += red[((wu / TW) * wpg + i) * V + (wu % TW) * RB + a];
      const float hv = silu(G * sc0) * (U * sc1);
      ws.h[(size_t)(pos0 + a0 + a) * p.I + tile * p.TJ + j] = hv;
      m = fmaxf(m, fabsf(hv));
    }
    amax_out = fmaxf(amax_out, m);
  } else {
    for (int q = tid; q < p.T * rb; q += NC) {
      const int w = q % p.T, a = q / p.T;
      float acc_o = 0.0f;
      for (int i = 0; i < wpg; ++i) acc_o += red[((w / TW) * wpg + i) * V + (w % TW) * RB + a];
      const int pair = sm.pairs[a0 + a];
      if (MOE_IN_BOUNDS(pair >= 0 && pair < p.ws_pairs, ws.err))
        ws.o[(size_t)pair * p.H + tile * p.T + w] = acc_o * sc0;
    }
  }
}

// The last CTA to finish an expert's gate/up tiles quantizes its h rows
// (one NVFP4 tensor per expert).
__device__ void quantize_expert_h(const ExpertParams& p, int e, int pos0, int ne, int tid,
                                  int NC) {
  const Workspace& ws = p.ws;
  const float amax = __uint_as_float(__ldcg(ws.h_amax + e));
  const float sg = __fdiv_rn(amax, 2688.0f);
  const int bpr = p.I / 16;
  const int nb = ne * bpr;
  for (int b = tid; b < nb; b += NC) {
    const int row = pos0 + b / bpr, blk = b % bpr;
    const float4* src = reinterpret_cast<const float4*>(ws.h + (size_t)row * p.I + blk * 16);
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 f = __ldcg(src + i);
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
    uint32_t lo, hi, sb;
    quant_block16(v, sg, lo, hi, sb);
    *reinterpret_cast<uint2*>(ws.h_codes + (size_t)row * (p.I / 2) + blk * 8) = make_uint2(lo, hi);
    ws.h_sf[(size_t)row * bpr + blk] = (uint8_t)sb;
  }
  if (tid == 0) ws.h_sg[e] = sg;
}

// Gate/up: this CTA is done with expert e (it ran `tiles_done` of its tiles).
// Publish its h amax, count the tiles, and if it completed the expert,
// quantize the expert's h.
__device__ void finish_expert(const ExpertParams& p, const Smem& sm, int e, int tiles_done,
                              int pos0, int ne, float amax, int tid, int NC) {
  const Workspace& ws = p.ws;
  amax = warp_max(amax);
  if ((tid & 31) == 0 && amax > 0.0f) atomic_max_nonneg(ws.h_amax + e, amax);
  __threadfence();
  named_bar(1, NC);
  if (tid == 0) {
    const unsigned old = atomicAdd(ws.done + e, (unsigned)tiles_done);
    *sm.flag = (old + (unsigned)tiles_done == (unsigned)p.tiles);
  }
  named_bar(1, NC);
  if (*sm.flag) {
    __threadfence();
    quantize_expert_h(p, e, pos0, ne, tid, NC);
    named_bar(1, NC);
    if (tid == 0) {
      ws.done[e] = 0u;
      ws.h_amax[e] = 0u;
    }
  }
  named_bar(1, NC);
}

// Issue the bulk copies of item `n` of this CTA's run into its stage
// (thread 0 only).  Stage metadata (expert, tile, first pooled position,
// pairs) rides along in shared memory.
__device__ __forceinline__ bool issue_item(const ExpertParams& p, const Smem& sm, bool gate_up,
                                           int it, int n, int ai_first, uint64_t pol) {
  const Workspace& ws = p.ws;
  const int s = n % p.NS;
  const int ai = it / p.tiles, tile = it % p.tiles;
  const int q = ai - ai_first;
  int4 et;
  if (q < kExpertTable) {
    et = sm.etab[q];
  } else {  // long runs over many experts: read the routing directly
    const int e = __ldcg(ws.active + ai);
    const int pos0 = (e >= 0 && e < p.E) ? __ldcg(ws.offset + e) : 0;
    const int ne = (e >= 0 && e < p.E) ? __ldcg(ws.offset + e + 1) - pos0 : 0;
    et = make_int4(e, pos0, ne, 0);
  }
  const int e = et.x, pos0 = et.y, ne = et.z;
  if (e < 0 || e >= p.E || pos0 < 0 || ne < 1 || ne > kMaxPairs || pos0 + ne > p.ws_pairs) {
    latch_error(ws.err, kDevBadRouting);
    return false;
  }
  sm.meta[s] = make_int4(e, tile, pos0, ne);
  uint8_t* dst = sm.stages + (size_t)s * p.stage_stride;
  // the stage was last read through the generic proxy; order that before the
  // async-proxy writes that refill it
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive_expect_tx(&sm.full[s], p.stage_bytes);
  if (gate_up) {
    const size_t rg = (size_t)e * p.RE + (size_t)tile * p.TJ;  // gate rows
    const size_t ru = rg + p.I;                                 // up rows
    const uint32_t cb = (uint32_t)(p.TJ * p.KB), sb = (uint32_t)(p.TJ * p.KS);
    bulk_g2s(dst, p.w + rg * p.KB, cb, &sm.full[s], pol);
    bulk_g2s(dst + cb, p.w + ru * p.KB, cb, &sm.full[s], pol);
    bulk_g2s(dst + 2 * cb, p.w_sf + rg * p.KS, sb, &sm.full[s], pol);
    bulk_g2s(dst + 2 * cb + sb, p.w_sf + ru * p.KS, sb, &sm.full[s], pol);
  } else {
    const size_t r0 = (size_t)e * p.RE + (size_t)tile * p.T;
    bulk_g2s(dst, p.w + r0 * p.KB, (uint32_t)(p.T * p.KB), &sm.full[s], pol);
    bulk_g2s(dst + (size_t)p.T * p.KB, p.w_sf + r0 * p.KS, (uint32_t)(p.T * p.KS), &sm.full[s],
             pol);
  }
  return true;
}

// One CTA per SM (about 200 KB of shared memory), up to 16 warps.
// Gate/up runs 8 weight rows per thread per item, down 4.
template <bool kGU>
__global__ void __launch_bounds__(kMaxThreads, 1) expert_kernel(ExpertParams p) {
  constexpr int TW = kGU ? 8 : 4;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem sm = carve(smem_raw);
  const Workspace& ws = p.ws;
  const int tid = threadIdx.x;
  const int NC = p.G * p.TPG;  // every thread computes; thread 0 also feeds the ring

  if (tid == 0) {
    for (int s = 0; s < p.NS; ++s) mbar_init(&sm.full[s], 1);
    mbar_fence_init();
  }

  // Gate/up needs the routing of the kernel before it; down's weights and
  // work list depend only on that routing (final before the gate/up kernel
  // started), so its first copies may be issued ahead of the wait.
  if (kGU) {
    grid_dep_wait();
    grid_dep_launch();
  }
  const int na = __ldcg(ws.n_active);
  const bool na_ok = na >= 0 && na <= p.E;
  const int n_items = na_ok ? na * p.tiles : 0;
  const int it0 = (int)((long long)blockIdx.x * n_items / gridDim.x);
  const int it1 = (int)((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  const int count = it1 - it0;
  const int ai_first = count > 0 ? it0 / p.tiles : 0;
  const int nai = count > 0 ? (it1 - 1) / p.tiles - ai_first + 1 : 0;
  for (int q = tid; q < nai && q < kExpertTable; q += NC) {
    const int e = __ldcg(ws.active + ai_first + q);
    const bool ok = e >= 0 && e < p.E;
    const int pos0 = ok ? __ldcg(ws.offset + e) : 0;
    sm.etab[q] = make_int4(e, pos0, ok ? __ldcg(ws.offset + e + 1) - pos0 : 0, 0);
  }
  __syncthreads();
  if (!na_ok) {
    if (tid == 0) latch_error(ws.err, kDevBadRouting);
    return;
  }

  const uint64_t pol = l2_evict_first_policy();
  int issued = 0;  // thread 0: items whose copies are in flight or landed
  if (tid == 0) {
    for (; issued < count && issued < p.NS; ++issued)
      if (!issue_item(p, sm, kGU, it0 + issued, issued, ai_first, pol)) break;
  }
  if (!kGU) {
    grid_dep_wait();  // h codes and scales come from the gate/up kernel
    grid_dep_launch();
  }

  const int cc = tid % p.TPG;
  const bool live = cc < p.CH;
  const float x_sg = kGU ? __ldcg(ws.x_sg) : 0.0f;
  uint32_t av[32];
  float sx[4][2];
  int cur_e = -1, cur_pos0 = 0, cur_ne = 0, cur_tiles = 0;
  float cur_amax = 0.0f, sc0 = 0.0f, sc1 = 0.0f;
  int gi = 0;

  for (int n = 0; n < count; ++n) {
    const int s = n % p.NS;
    // Thread 0 waits (bounded) for the stage; the barrier hands its acquire
    // and its verdict to every thread, so all take the same path and none is
    // left behind at a later barrier.  Passing the barrier also proves every
    // thread is done with item n-1, so its stage is refilled right after.
    if (tid == 0) {
      bool got = n < issued && mbar_wait(&sm.full[s], (n / p.NS) & 1, ws.wait_ns);
      if (!got) latch_error(ws.err, kDevWaitTimeout);
      *sm.ok = got ? 1 : 0;
    }
    named_bar(1, NC);
    if (*reinterpret_cast<volatile int*>(sm.ok) == 0) break;
    if (tid == 0 && n >= 1 && issued < count && issued == n - 1 + p.NS) {
      if (issue_item(p, sm, kGU, it0 + issued, issued, ai_first, pol)) ++issued;
    }
    const int4 m = sm.meta[s];
    const int e = m.x, tile = m.y, pos0 = m.z, ne = m.w;
    if (e != cur_e) {
      if (kGU && cur_e >= 0)
        finish_expert(p, sm, cur_e, cur_tiles, cur_pos0, cur_ne, cur_amax, tid, NC);
      cur_e = e;
      cur_pos0 = pos0;
      cur_ne = ne;
      cur_tiles = 0;
      cur_amax = 0.0f;
      if (kGU) {
        sc0 = __ldg(p.gscale + 3 * e + 0) * x_sg;
        sc1 = __ldg(p.gscale + 3 * e + 1) * x_sg;
      } else {
        // (the item barrier above ordered every read of the previous
        // expert's pair ids before these writes)
        sc0 = __ldg(p.gscale + 3 * e + 2) * __ldcg(ws.h_sg + e);
        for (int q = tid; q < ne; q += NC) sm.pairs[q] = __ldcg(ws.pair_order + pos0 + q);
      }
      if (ne == 1) load_act<1, true>(p, kGU, pos0, 1, cc, live, av, sx);
      else if (ne == 2) load_act<2, true>(p, kGU, pos0, 2, cc, live, av, sx);
      else if (ne <= 4) load_act<4, false>(p, kGU, pos0, ne, cc, live, av, sx);
    }
    const uint8_t* stage = sm.stages + (size_t)s * p.stage_stride;
    float* red = sm.red + (gi & 1) * kRedFloats;
    if (ne == 1) {
      ++gi;
      run_group<TW, 1, true, kGU>(p, sm, red, stage, tile, pos0, 0, 1, tid, NC, av, sx, sc0, sc1, cur_amax);
    } else if (ne == 2) {
      ++gi;
      run_group<TW, 2, true, kGU>(p, sm, red, stage, tile, pos0, 0, 2, tid, NC, av, sx, sc0, sc1, cur_amax);
    } else {
      for (int a0 = 0; a0 < ne; a0 += 4) {
        const int rb = min(4, ne - a0);
        red = sm.red + (gi & 1) * kRedFloats;
        ++gi;
        if (ne > 4) load_act<4, false>(p, kGU, pos0 + a0, rb, cc, live, av, sx);
        run_group<TW, 4, false, kGU>(p, sm, red, stage, tile, pos0, a0, rb, tid, NC, av, sx, sc0, sc1, cur_amax);
      }
    }
    ++cur_tiles;
  }
  if (kGU && cur_e >= 0) finish_expert(p, sm, cur_e, cur_tiles, cur_pos0, cur_ne, cur_amax, tid, NC);
  // every issued copy has landed before the CTA may exit (normally all were
  // consumed already; after an early stop this drains the ring)
  if (tid == 0) {
    for (int s = 0; s < p.NS && s < issued; ++s) {
      const int last = s + p.NS * ((issued - 1 - s) / p.NS);
      (void)mbar_wait(&sm.full[s], (last / p.NS) & 1, ws.wait_ns);
    }
  }
}

}  // namespace

size_t expert_ctrl_bytes() { return (size_t)kCtrlRounded; }

size_t expert_smem_bytes(const ExpertParams& p) {
  return (size_t)kCtrlRounded + (size_t)p.NS * p.stage_stride;
}

cudaError_t expert_set_smem(size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(expert_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(expert_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

cudaError_t launch_experts(const ExpertParams& p, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(p.G * p.TPG, 1, 1);
  cfg.dynamicSmemBytes = expert_smem_bytes(p);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.mode == kGateUp) return cudaLaunchKernelEx(&cfg, expert_kernel<true>, p);
  return cudaLaunchKernelEx(&cfg, expert_kernel<false>, p);
}

}  // namespace moe
