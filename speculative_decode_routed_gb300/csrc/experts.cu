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
//  - Consumer threads own a fixed 16-byte column chunk (32 elements, two
//    16-blocks) of every weight row; the expert's activation rows for that
//    chunk stay in registers as signed bytes (2 x e2m1 value, exact).  A
//    weight chunk is expanded to signed bytes with byte-permute table
//    lookups and each 16-block dot product is an exact int32 sum of four
//    dp4a; the block result is scaled by the exact fp32 product of the two
//    e4m3 scales and accumulated in fp32.
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

constexpr int kRedFloats = 8 * kTW * kMaxRB;  // one reduction buffer: 8 warps x 64 values
constexpr int kMaxPairs = 128;                 // pairs of one expert <= rows <= 128
constexpr int kExpertTable = 64;               // experts of one CTA's run kept in smem
constexpr int kCtrlBytes = 512 + kExpertTable * 16 + 2 * kRedFloats * 4 + kMaxPairs * 4 + 64;

// Shared memory: [barriers + stage metadata | 2 reduction buffers | pair ids
// of the current expert | flags] then the stage ring.
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
  s.stages = base + ((kCtrlBytes + 1023) / 1024) * 1024;
  return s;
}

// Reduce-scatter of V values (V a power of two) across the 32 lanes; lane
// results land in dst[index] (lanes holding the same index write once).
template <int V>
__device__ __forceinline__ void warp_reduce_scatter_store(float (&v)[V], int lane, float* dst) {
  constexpr int kSteps = (V >= 32) ? 5 : (V == 16 ? 4 : (V == 8 ? 3 : (V == 4 ? 2 : (V == 2 ? 1 : 0))));
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
  constexpr int kLeft = V >> kSteps;  // values per lane now (1, or V/32)
#pragma unroll
  for (int st = kSteps; st < 5; ++st) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16 >> st);
  const int low_bits = (1 << (5 - kSteps)) - 1;
  if ((lane & low_bits) == 0) {
#pragma unroll
    for (int i = 0; i < kLeft; ++i) dst[base + i] = v[i];
  }
}

// The expert's activation rows [pos0, pos0 + rb) for this thread's chunk, as
// signed bytes (2 x e2m1 value) and two fp32 block scales.
template <int RB>
__device__ __forceinline__ void load_act(const ExpertParams& p, bool gate_up, int pos0, int rb,
                                         int cc, bool live, uint32_t (&xa)[kMaxRB][8],
                                         float (&sx)[kMaxRB][2]) {
  const Workspace& ws = p.ws;
  const uint8_t* codes = gate_up ? ws.x_codes : ws.h_codes;
  const uint8_t* sf = gate_up ? ws.x_sf : ws.h_sf;
#pragma unroll
  for (int a = 0; a < RB; ++a) {
    if (a < rb && live) {
      const int pos = pos0 + a;
      const int row = gate_up ? __ldcg(ws.pair_order + pos) / p.k : pos;
      const uint4 c = __ldcg(reinterpret_cast<const uint4*>(codes + (size_t)row * p.KB) + cc);
      e2m1x8_to_s8x8(c.x, xa[a][0], xa[a][1]);
      e2m1x8_to_s8x8(c.y, xa[a][2], xa[a][3]);
      e2m1x8_to_s8x8(c.z, xa[a][4], xa[a][5]);
      e2m1x8_to_s8x8(c.w, xa[a][6], xa[a][7]);
      const unsigned short s2 =
          __ldcg(reinterpret_cast<const unsigned short*>(sf + (size_t)row * p.KS) + cc);
      const float2 f = e4m3x2_to_f32x2(s2);
      sx[a][0] = f.x;
      sx[a][1] = f.y;
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) xa[a][q] = 0u;
      sx[a][0] = sx[a][1] = 0.0f;
    }
  }
}

// Dot products of this thread's chunk of the group's kTW weight rows with the
// RB activation rows held in registers.
template <int RB>
__device__ __forceinline__ void gemv_chunk(const ExpertParams& p, const uint8_t* stage, int g,
                                           int cc, bool live, const uint32_t (&xa)[kMaxRB][8],
                                           const float (&sx)[kMaxRB][2],
                                           float (&acc)[kTW * RB]) {
#pragma unroll
  for (int i = 0; i < kTW * RB; ++i) acc[i] = 0.0f;
  if (!live) return;
  const uint8_t* sc = stage + (size_t)cc * 16 + (size_t)g * kTW * p.KB;
  const uint8_t* ss = stage + (size_t)p.T * p.KB + (size_t)cc * 2 + (size_t)g * kTW * p.KS;
#pragma unroll
  for (int t = 0; t < kTW; ++t) {
    const uint4 c = *reinterpret_cast<const uint4*>(sc + (size_t)t * p.KB);
    const unsigned short s2 = *reinterpret_cast<const unsigned short*>(ss + (size_t)t * p.KS);
    const float2 sw = e4m3x2_to_f32x2(s2);
    uint32_t wv[8];
    e2m1x8_to_s8x8(c.x, wv[0], wv[1]);
    e2m1x8_to_s8x8(c.y, wv[2], wv[3]);
    e2m1x8_to_s8x8(c.z, wv[4], wv[5]);
    e2m1x8_to_s8x8(c.w, wv[6], wv[7]);
#pragma unroll
    for (int a = 0; a < RB; ++a) {
      int d0 = __dp4a((int)wv[0], (int)xa[a][0], 0);
      d0 = __dp4a((int)wv[1], (int)xa[a][1], d0);
      d0 = __dp4a((int)wv[2], (int)xa[a][2], d0);
      d0 = __dp4a((int)wv[3], (int)xa[a][3], d0);
      int d1 = __dp4a((int)wv[4], (int)xa[a][4], 0);
      d1 = __dp4a((int)wv[5], (int)xa[a][5], d1);
      d1 = __dp4a((int)wv[6], (int)xa[a][6], d1);
      d1 = __dp4a((int)wv[7], (int)xa[a][7], d1);
      float acc_v = acc[t * RB + a];
      acc_v = fmaf((float)d0, sw.x * sx[a][0], acc_v);
      acc_v = fmaf((float)d1, sw.y * sx[a][1], acc_v);
      acc[t * RB + a] = acc_v;
    }
  }
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// One activation-row group (RB rows) of one item: dot products, reduction,
// epilogue (h for gate/up, o for down).  `red` alternates between the two
// reduction buffers, so one barrier per group suffices.
template <int RB, bool kGU>
__device__ __forceinline__ void run_group(const ExpertParams& p, const Smem& sm, float* red,
                                          const uint8_t* stage, int tile, int pos0, int a0, int rb,
                                          int tid, int NC, const uint32_t (&xa)[kMaxRB][8],
                                          const float (&sx)[kMaxRB][2], float sc0, float sc1,
                                          float& amax_out) {
  const int g = tid / p.TPG, cc = tid % p.TPG;
  const bool live = cc < p.CH;
  const int lane = tid & 31, warp = tid >> 5;
  constexpr int V = kTW * RB;
  float acc[V];
  gemv_chunk<RB>(p, stage, g, cc, live, xa, sx, acc);
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
      for (int i = 0; i < wpg; ++i) G += red[((wg / kTW) * wpg + i) * V + (wg % kTW) * RB + a];
      for (int i = 0; i < wpg; ++i) U += red[((wu / kTW) * wpg + i) * V + (wu % kTW) * RB + a];
      const float hv = silu(G * sc0) * (U * sc1);
      ws.h[(size_t)(pos0 + a0 + a) * p.I + tile * p.TJ + j] = hv;
      m = fmaxf(m, fabsf(hv));
    }
    amax_out = fmaxf(amax_out, m);
  } else {
    for (int q = tid; q < p.T * rb; q += NC) {
      const int w = q % p.T, a = q / p.T;
      float acc_o = 0.0f;
      for (int i = 0; i < wpg; ++i) acc_o += red[((w / kTW) * wpg + i) * V + (w % kTW) * RB + a];
      const int pair = sm.pairs[a0 + a];
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

// One CTA per SM by design (about 200 KB of shared memory), at most 8 warps:
// two warps per SM sub-partition leave room for up to 224 registers per
// thread, which keeps the RB = 8 path free of spills.
template <bool kGU>
__global__ void __maxnreg__(224) expert_kernel(ExpertParams p) {
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
  const int lane = tid & 31;
  const float x_sg = kGU ? __ldcg(ws.x_sg) : 0.0f;
  uint32_t xa[kMaxRB][8];
  float sx[kMaxRB][2];
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
      bool got = n < issued && mbar_wait(&sm.full[s], (n / p.NS) & 1);
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
        sc0 = __ldg(p.gscale + 3 * e + 0) * x_sg * 0.25f;
        sc1 = __ldg(p.gscale + 3 * e + 1) * x_sg * 0.25f;
      } else {
        // (the item barrier above ordered every read of the previous
        // expert's pair ids before these writes)
        sc0 = __ldg(p.gscale + 3 * e + 2) * __ldcg(ws.h_sg + e) * 0.25f;
        for (int q = tid; q < ne; q += NC) sm.pairs[q] = __ldcg(ws.pair_order + pos0 + q);
      }
      const int rb = min(kMaxRB, ne);
      if (ne <= kMaxRB) {
        if (rb == 1) load_act<1>(p, kGU, pos0, rb, cc, live, xa, sx);
        else if (rb == 2) load_act<2>(p, kGU, pos0, rb, cc, live, xa, sx);
        else if (rb <= 4) load_act<4>(p, kGU, pos0, rb, cc, live, xa, sx);
        else load_act<8>(p, kGU, pos0, rb, cc, live, xa, sx);
      }
    }
    const uint8_t* stage = sm.stages + (size_t)s * p.stage_stride;
    for (int a0 = 0; a0 < ne; a0 += kMaxRB) {
      const int rb = min(kMaxRB, ne - a0);
      float* red = sm.red + (gi & 1) * kRedFloats;
      ++gi;
      if (ne > kMaxRB) load_act<kMaxRB>(p, kGU, pos0 + a0, rb, cc, live, xa, sx);
      if (rb == 1)
        run_group<1, kGU>(p, sm, red, stage, tile, pos0, a0, rb, tid, NC, xa, sx, sc0, sc1, cur_amax);
      else if (rb == 2)
        run_group<2, kGU>(p, sm, red, stage, tile, pos0, a0, rb, tid, NC, xa, sx, sc0, sc1, cur_amax);
      else if (rb <= 4)
        run_group<4, kGU>(p, sm, red, stage, tile, pos0, a0, rb, tid, NC, xa, sx, sc0, sc1, cur_amax);
      else
        run_group<8, kGU>(p, sm, red, stage, tile, pos0, a0, rb, tid, NC, xa, sx, sc0, sc1, cur_amax);
    }
    ++cur_tiles;
  }
  if (kGU && cur_e >= 0) finish_expert(p, sm, cur_e, cur_tiles, cur_pos0, cur_ne, cur_amax, tid, NC);
  // every issued copy has landed before the CTA may exit (normally all were
  // consumed already; after an early stop this drains the ring)
  if (tid == 0) {
    for (int s = 0; s < p.NS && s < issued; ++s) {
      const int last = s + p.NS * ((issued - 1 - s) / p.NS);
      (void)mbar_wait(&sm.full[s], (last / p.NS) & 1);
    }
  }
}

}  // namespace

size_t expert_smem_bytes(const ExpertParams& p) {
  return (size_t)((kCtrlBytes + 1023) / 1024) * 1024 + (size_t)p.NS * p.stage_stride;
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
