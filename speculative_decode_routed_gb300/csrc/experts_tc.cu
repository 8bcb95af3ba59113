// Routed NVFP4 experts on the 5th-generation tensor cores (tcgen05,
// kind::mxf4nvf4 block-scaled MMA, e4m3 scales per 16 elements).
//
// Page: vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode,
// module docstring "One step of b rows", MoE: "... pooler -> routed experts
// -> tail -> unpooler"; gate_proj / up_proj stacked as shards 0 / 1 of
// gate_up_proj (the DSpark page's weight mapping).  Per pair routed to
// expert e: h = silu(Wg xq) * (Wu xq) (fp32), h quantized to NVFP4 per
// expert, o = Wd hq (fp32).
//
// Swap-AB: the expert's weight rows fill the MMA's M = 128 (operand A,
// streamed from HBM), the expert's pairs fill N (operand B, 32 rows per MMA,
// from L2).  One persistent CTA per SM, warp-specialized:
//   warp 0  TMA producer: per stage (KPS K-blocks of 256), the weight tiles
//           (tensor map, 128B swizzle), their scale atoms (one bulk copy,
//           laid out for tcgen05.cp at create time), the pooled activation
//           tiles and their scale lines (tensor maps) into a ring of stages;
//   warps 1..P  MMA issuers: issuer (type, q) -- gate or up accumulator, and
//           the stages ks = q (mod Q) of every item -- copies the stage's
//           scales into its own TMEM slot (tcgen05.cp) and issues 4 MMAs
//           (K = 64) per K-block into its own accumulator; tcgen05.commit
//           frees the stage and publishes the accumulator.  One thread's MMA
//           issue is latency-bound; independent issuers overlap.
//   4 warps epilogue: tcgen05.ld of the K-phase partial accumulators (one
//           TMEM lane per weight row) summed in a fixed order, scaled by the
//           two fp32 tensor scales, SiLU * up or the down output, coalesced
//           stores.  Accumulators are double buffered in TMEM so the epilogue
//           of item i overlaps item i+1.
// Every wait is bounded (a latched error instead of a hang).
#include <cuda.h>

#include "common.cuh"
#include "tc_internal.h"

namespace moe {
namespace {

constexpr int kTcMaxThreads = 32 * (1 + 4 + 4);  // producer, up to 4 MMA issuers, 4 epilogue warps
constexpr int kEpiThreads = 128;
constexpr int kExpertTableTc = 64;
constexpr int kMaxPairsTc = 128;
constexpr int kTcCtrl = 4096;             // barriers, tables, flags

// ---------------------------------------------------------------- PTX bits

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y,
                                       uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_2d_plain(void* dst, const CUtensorMap* map, int x, int y,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_3d_hint(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor (sm_100 form): start >> 4, leading / stride
// byte offsets >> 4, version 1, layout type (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

// kind::mxf4nvf4 instruction descriptor: A, B e2m1 (1), K-major, scales
// ue4m3 (0), M = 128, N = 32, dense.
constexpr uint32_t kIdescM128N32 = (1u << 7) | (1u << 10) | ((32u >> 3) << 17) | (0u << 23) |
                                   ((128u >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t sfa, uint32_t sfb, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdescM128N32), "r"(sfa), "r"(sfb), "r"(accumulate ? 1 : 0)
      : "memory");
}

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, const void* src) {
  const uint64_t d = smem_desc(smem_u32(src), 128, 128, 0);
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------ shared memory

struct TcSmem {
  uint64_t* full;       // [NS][Q]   TMA bytes landed, one barrier per stage and K-phase group
  uint64_t* empty;      // [NS]      every issuer that reads the stage is done (T arrivals)
  uint64_t* acc_full;   // [2]       accumulators ready for the epilogue (P arrivals)
  uint64_t* acc_empty;  // [2]       epilogue done reading them (4 arrivals)
  uint64_t* slot_free;  // [4][2]    an issuer's scale slot may be overwritten
  uint64_t* drain;      // [4]       every MMA of an issuer done
  int4* etab;           // [kExpertTableTc]
  int* pairs;           // [kMaxPairsTc]
  int* flag;
  uint32_t* tmem_base;
  uint8_t* stages;
};

__device__ __forceinline__ TcSmem tc_carve(uint8_t* base) {
  TcSmem s;
  s.full = reinterpret_cast<uint64_t*>(base);
  s.empty = s.full + 32;
  s.acc_full = s.empty + 16;
  s.acc_empty = s.acc_full + 2;
  s.slot_free = s.acc_empty + 2;
  s.drain = s.slot_free + 8;
  s.etab = reinterpret_cast<int4*>(base + 512);
  s.pairs = reinterpret_cast<int*>(base + 512 + kExpertTableTc * 16);
  s.flag = s.pairs + kMaxPairsTc;
  s.tmem_base = reinterpret_cast<uint32_t*>(s.flag + 4);
  s.stages = base + kTcCtrl;
  return s;
}

__device__ __forceinline__ int4 tc_item_expert(const TcParams& p, const TcSmem& sm, int it,
                                               int ai_first) {
  const int ai = it / p.tiles, q = ai - ai_first;
  if (q < kExpertTableTc) return sm.etab[q];
  const int e = __ldcg(p.ws.active + ai);
  const bool ok = e >= 0 && e < p.E;
  const int pos0 = ok ? __ldcg(p.ws.offset + e) : 0;
  return make_int4(e, pos0, ok ? __ldcg(p.ws.offset + e + 1) - pos0 : 0, 0);
}

__device__ __forceinline__ bool tc_item_ok(const TcParams& p, int4 et) {
  return et.x >= 0 && et.x < p.E && et.y >= 0 && et.z >= 1 && et.z <= kMaxPairsTc &&
         et.y + et.z <= p.ws_pairs;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Barrier over the four epilogue warps only (threads 64..191).
__device__ __forceinline__ void tc_named_sync() { named_bar(2, kEpiThreads); }

// The last CTA to finish an expert's gate/up tiles quantizes its h rows (one
// NVFP4 tensor per expert): codes, block scales and the per-MMA scale lines
// the down kernel streams as its B-operand scales.
__device__ void tc_quantize_expert_h(const TcParams& p, int e, int pos0, int ne, int t) {
  const Workspace& ws = p.ws;
  const float amax = __uint_as_float(__ldcg(ws.h_amax + e));
  const float sg = __fdiv_rn(amax, 2688.0f);
  const int bpr = p.I / 16;
  for (int b = t; b < ne * bpr; b += kEpiThreads) {
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
  tc_named_sync();
  // scale lines: one 16-byte line per (row, MMA of 64): bytes 0-3 = its four
  // block scales, the rest zero
  const int lpr = p.I / 64;
  for (int l = t; l < ne * lpr; l += kEpiThreads) {
    const int row = pos0 + l / lpr, m = l % lpr;
    const uint32_t w = __ldcg(reinterpret_cast<const uint32_t*>(ws.h_sf + (size_t)row * bpr) + m);
    *reinterpret_cast<uint4*>(ws.h_lines + ((size_t)m * p.ws_pairs + row) * 16) =
        make_uint4(w, 0u, 0u, 0u);
  }
  if (t == 0) ws.h_sg[e] = sg;
}

}  // namespace

// ======================================================================
// The expert kernel.  Warp 0: TMA producer.  Warps 1..P: MMA issuers (issuer
// i = type ty * Q + phase q: accumulator type ty -- gate or up -- and the
// K-blocks kb = q mod Q).  Warps P+1..P+4: epilogue.
template <bool kGU>
__global__ void __launch_bounds__(kTcMaxThreads, 1)
    tc_expert_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tm_a,
                     const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_sfb) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128B-swizzled TMA tiles need 1024-byte aligned destinations: align the
  // base explicitly (the launch adds 1 KB of slack for this)
  uint8_t* smem_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const TcSmem sm = tc_carve(smem_base);
  const Workspace& ws = p.ws;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.P;

  // A stage is read by the issuers of K-phase group q = kb mod Q.  When NS is
  // not a multiple of Q the group changes from one fill of a stage to the
  // next, and a parity wait by an issuer that skipped a phase would match the
  // stale parity of the fill before.  So each (stage, group) has its own
  // full barrier: every phase of it is consumed by the same issuers, and each
  // waiter tracks that barrier's parity itself.
  if (tid == 0) {
    for (int s = 0; s < p.NS; ++s) {
      for (int q = 0; q < p.Q; ++q) mbar_init(&sm.full[s * p.Q + q], 1);
      mbar_init(&sm.empty[s], p.T);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.acc_full[b], P);
      mbar_init(&sm.acc_empty[b], kEpiThreads / 32);
    }
    for (int i = 0; i < 8; ++i) mbar_init(&sm.slot_free[i], 1);
    for (int i = 0; i < 4; ++i) mbar_init(&sm.drain[i], 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(sm.tmem_base)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Gate/up waits for the routing and the pooled MoE input before anything;
  // down's producer issues its first weight tiles before waiting.
  if (kGU) {
    grid_dep_wait();
    grid_dep_launch();
  }
  const int na = __ldcg(ws.n_active);
  const bool na_ok = na >= 0 && na <= p.E;
  const int n_items = na_ok ? na * p.tiles : 0;
  const int it0 = (int)((long long)blockIdx.x * n_items / gridDim.x);
  const int it1 = (int)((long long)(blockIdx.x + 1) * n_items / gridDim.x);
  const int ai_first = it1 > it0 ? it0 / p.tiles : 0;
  const int nai = it1 > it0 ? (it1 - 1) / p.tiles - ai_first + 1 : 0;
  for (int q = tid; q < nai && q < kExpertTableTc; q += blockDim.x) {
    const int e = __ldcg(ws.active + ai_first + q);
    const bool ok = e >= 0 && e < p.E;
    const int pos0 = ok ? __ldcg(ws.offset + e) : 0;
    sm.etab[q] = make_int4(e, pos0, ok ? __ldcg(ws.offset + e + 1) - pos0 : 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_base;
  if (!na_ok && tid == 0) latch_error(ws.err, kDevBadRouting);

  const int KB = p.KBLK;      // K-blocks of 256 per item
  const int KPS = p.KPS;      // K-blocks per stage
  const int KS = p.KSTEPS;    // stages per item

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int g = 0;  // global stage counter = item * KS + ks
      uint32_t fbits = 0;  // per (stage, group) full barrier: parity of fills issued
      bool ok = true;
      bool waited = kGU;
      for (int it = it0; it < it1 && ok; ++it) {
        const int4 et = tc_item_expert(p, sm, it, ai_first);
        if (!tc_item_ok(p, et)) {
          latch_error(ws.err, kDevBadRouting);
          break;
        }
        const int e = et.x, tile = it % p.tiles, pos0 = et.y, ne = et.z;
        const int nt = (ne + 31) / 32;
        for (int ks = 0; ks < KS; ++ks, ++g) {
          const int kb = ks * KPS;  // first K-block of this stage
          const int nkb = min(KPS, KB - kb);
          const int s = g % p.NS;
          if (g >= p.NS && !mbar_wait(&sm.empty[s], ((g / p.NS) - 1) & 1)) {
            latch_error(ws.err, kDevWaitTimeout);
            ok = false;
            break;
          }
          uint8_t* st = sm.stages + (size_t)s * p.stage_stride;
          const int fb = s * p.Q + ks % p.Q;
          uint64_t* full = &sm.full[fb];
          fbits ^= 1u << fb;
          // weight tiles (a missing second K-block of a stage is zero filled
          // and counts in full), the present K-blocks' scale atoms, and per
          // N-tile the activation tiles and scale lines
          const uint32_t sfa_b = 2048u * (uint32_t)nkb;
          const uint32_t bytes = p.a_bytes + sfa_b * (uint32_t)p.T +
                                 (uint32_t)(nt * KPS) * (4096u + 2048u);
          mbar_arrive_expect_tx(full, bytes);
          // gate rows (gate/up) or output rows (down) of this tile
          if (KPS == 1)
            tma_2d(st, &tm_a, kb * 128, e * p.RE + tile * 128, full, pol);
          else
            tma_3d_hint(st, &tm_a, 0, e * p.RE + tile * 128, kb, full, pol);
          bulk_g2s_plain(st + p.off_sfa,
                         p.sfa + (((size_t)e * p.row_tiles + tile) * KB + kb) * 2048u, sfa_b,
                         full);
          if (kGU) {  // gate/up stages hold one K-block
            const int ru = p.I / 128 + tile;  // up rows follow the gate rows
            tma_2d(st + 16384, &tm_a, kb * 128, e * p.RE + ru * 128, full, pol);
            bulk_g2s_plain(st + p.off_sfa + 2048,
                           p.sfa + (((size_t)e * p.row_tiles + ru) * KB + kb) * 2048u, 2048u,
                           full);
          }
          if (!waited) {  // down: h and its scales come from the gate/up kernel
            grid_dep_wait();
            grid_dep_launch();
            waited = true;
          }
          for (int t = 0; t < nt; ++t) {
            if (KPS == 1)
              tma_2d_plain(st + p.off_b + t * 4096, &tm_b, kb * 128, pos0 + 32 * t, full);
            else
              tma_3d(st + p.off_b + t * 4096 * KPS, &tm_b, 0, pos0 + 32 * t, kb, full);
            tma_3d(st + p.off_sfb + t * 2048 * KPS, &tm_sfb, 0, pos0 + 32 * t, kb * 4, full);
          }
        }
      }
      if (!waited) {
        grid_dep_wait();
        grid_dep_launch();
      }
      // every issued copy lands before the CTA may exit: the last fill of a
      // stage was issued only after every earlier fill of it had been consumed
      for (int s = 0; s < p.NS && s < g; ++s) {
        const int last = s + p.NS * ((g - 1 - s) / p.NS);
        const int fb = s * p.Q + (last % KS) % p.Q;
        if (!mbar_wait(&sm.full[fb], ((fbits >> fb) & 1u) ^ 1u)) latch_error(ws.err, kDevWaitTimeout);
      }
    }
  } else if (warp <= P) {
    // --------------------------------------------------------- MMA issuers
    if (!kGU) {
      grid_dep_wait();
      grid_dep_launch();
    }
    const int i = warp - 1;
    const int ty = i / p.Q, q = i % p.Q;
    if (lane == 0) {
      const uint32_t ibase = tmem + (uint32_t)i * p.issuer_cols;
      int c = 0, item = 0;  // stages handled, items seen
      uint32_t fpar = 0;    // bit s: parity of this group's next phase of full[s][q]
      bool ok = true;
      for (int it = it0; it < it1 && ok; ++it, ++item) {
        const int4 et = tc_item_expert(p, sm, it, ai_first);
        if (!tc_item_ok(p, et)) break;
        const int nt = (et.z + 31) / 32;
        const int ab = (p.dbuf == 2) ? (item & 1) : 0;
        const int use = (p.dbuf == 2) ? (item >> 1) : item;
        if (use >= 1 && !mbar_wait(&sm.acc_empty[ab], (use - 1) & 1)) {
          latch_error(ws.err, kDevWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t dcol = ibase + (uint32_t)ab * p.acc_cols;
        bool first = true;
        for (int ks = q; ks < KS; ks += p.Q, ++c) {
          const int g = item * KS + ks;
          const int nkb = min(KPS, KB - ks * KPS);
          const int s = g % p.NS;
          const uint32_t par = (fpar >> s) & 1u;
          fpar ^= 1u << s;
          if (!mbar_wait(&sm.full[s * p.Q + q], par)) {
            latch_error(ws.err, kDevWaitTimeout);
            ok = false;
            break;
          }
          const int slot = c % p.sfslots;
          if (c >= p.sfslots &&
              !mbar_wait(&sm.slot_free[i * 2 + slot], ((c / p.sfslots) - 1) & 1)) {
            latch_error(ws.err, kDevWaitTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = sm.stages + (size_t)s * p.stage_stride;
          const uint32_t sf = ibase + (uint32_t)p.dbuf * p.acc_cols + (uint32_t)slot * p.sf_cols;
          // scales into TMEM, 4 columns per MMA (m = 4 j + k for K-block j of
          // the stage): A (this issuer's weight tile) at sf, B per N-tile at
          // sf + 16 KPS (1 + t)
          const uint32_t sfb0 = sf + 16u * (uint32_t)KPS;
          for (int m = 0; m < 4 * nkb; ++m)
            tc_cp_sf(sf + 4 * m, st + p.off_sfa + ty * 2048 * KPS + m * 512);
          for (int t = 0; t < nt; ++t)
            for (int m = 0; m < 4 * nkb; ++m)
              tc_cp_sf(sfb0 + 16 * KPS * t + 4 * m, st + p.off_sfb + t * 2048 * KPS + m * 512);
          const uint32_t a0 = smem_u32(st) + (uint32_t)(ty * 16384 * KPS), b0 = smem_u32(st + p.off_b);
          for (int m = 0; m < 4 * nkb; ++m) {
            const uint32_t kofs = (uint32_t)((m >> 2) * 16384 + 32 * (m & 3));
            const uint64_t ad = smem_desc(a0 + kofs, 16, 1024, 2);
            for (int t = 0; t < nt; ++t)
              tc_mma(dcol + 32 * t, ad,
                     smem_desc(b0 + t * 4096 * KPS + (m >> 2) * 4096 + 32 * (m & 3), 16, 1024, 2),
                     sf + 4 * m, sfb0 + 16 * KPS * t + 4 * m, !(first && m == 0));
          }
          first = false;
          tc_commit(&sm.empty[s]);
          tc_commit(&sm.slot_free[i * 2 + slot]);
        }
        if (ok) tc_commit(&sm.acc_full[ab]);  // also when this phase had no K-block
      }
      // everything this thread issued completes before TMEM is released
      tc_commit(&sm.drain[i]);
      if (!mbar_wait(&sm.drain[i], 0)) latch_error(ws.err, kDevWaitTimeout);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    if (!kGU) {
      grid_dep_wait();
      grid_dep_launch();
    }
    const int t = tid - 32 * (P + 1);   // 0..127
    const int qd = warp & 3;            // TMEM lane quadrant of this warp
    const int m = 32 * qd + lane;       // weight row within the tile
    const int nparts = KS < p.Q ? KS : p.Q;  // K-phase partial accumulators that exist
    const float x_sg = kGU ? __ldcg(ws.x_sg) : 0.0f;
    int cur_e = -1, cur_pos0 = 0, cur_ne = 0, cur_tiles = 0, item = 0;
    float cur_amax = 0.0f, sc0 = 0.0f, sc1 = 0.0f;
    for (int it = it0; it < it1; ++it, ++item) {
      const int4 et = tc_item_expert(p, sm, it, ai_first);
      if (!tc_item_ok(p, et)) break;
      const int e = et.x, tile = it % p.tiles, pos0 = et.y, ne = et.z;
      if (e != cur_e) {
        if (kGU && cur_e >= 0) {
          // publish this CTA's share of the finished expert
          float am = warp_max(cur_amax);
          if (lane == 0 && am > 0.0f) atomic_max_nonneg(ws.h_amax + cur_e, am);
          __threadfence();
          tc_named_sync();
          if (t == 0) {
            const unsigned old = atomicAdd(ws.done + cur_e, (unsigned)cur_tiles);
            *sm.flag = (old + (unsigned)cur_tiles == (unsigned)p.tiles);
          }
          tc_named_sync();
          if (*sm.flag) {
            __threadfence();
            tc_quantize_expert_h(p, cur_e, cur_pos0, cur_ne, t);
            tc_named_sync();
            if (t == 0) {
              ws.done[cur_e] = 0u;
              ws.h_amax[cur_e] = 0u;
            }
          }
          tc_named_sync();
        }
        if (!kGU) {
          tc_named_sync();  // nobody still reads the previous expert's pair ids
          for (int j = t; j < ne; j += kEpiThreads) sm.pairs[j] = __ldcg(ws.pair_order + pos0 + j);
          tc_named_sync();
        }
        cur_e = e;
        cur_pos0 = pos0;
        cur_ne = ne;
        cur_tiles = 0;
        cur_amax = 0.0f;
        if (kGU) {
          sc0 = __ldg(p.gscale + 3 * e + 0) * x_sg;
          sc1 = __ldg(p.gscale + 3 * e + 1) * x_sg;
        } else {
          sc0 = __ldg(p.gscale + 3 * e + 2) * __ldcg(ws.h_sg + e);
        }
      }
      const int ab = (p.dbuf == 2) ? (item & 1) : 0;
      const int use = (p.dbuf == 2) ? (item >> 1) : item;
      // one thread waits (bounded); the barrier hands its verdict to all four
      // epilogue warps so none is left behind at a later barrier
      if (t == 0) *sm.flag = mbar_wait(&sm.acc_full[ab], use & 1) ? 1 : 0;
      tc_named_sync();
      const bool got = *reinterpret_cast<volatile int*>(sm.flag) != 0;
      tc_named_sync();
      if (!got) {
        if (t == 0) latch_error(ws.err, kDevWaitTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t lanes = (uint32_t)(32 * qd) << 16;
      const int nt = (ne + 31) / 32;
      for (int tt = 0; tt < nt; ++tt) {
        for (int half = 0; half < 2; ++half) {
          const int c0 = 32 * tt + 16 * half;  // first pair column of this half
          const int cnt = min(16, ne - c0);
          if (cnt <= 0) break;
          // sum the K-phase partials (fixed order) of each accumulator type
          float acc0[16], acc1[16];
#pragma unroll
          for (int n = 0; n < 16; ++n) acc0[n] = acc1[n] = 0.0f;
          for (int qq = 0; qq < nparts; ++qq) {
            uint32_t r[16];
            tc_ld16(tmem + lanes + (uint32_t)qq * p.issuer_cols + (uint32_t)ab * p.acc_cols + c0, r);
            tc_wait_ld();
#pragma unroll
            for (int n = 0; n < 16; ++n) acc0[n] += __uint_as_float(r[n]);
            if (kGU) {
              tc_ld16(tmem + lanes + (uint32_t)(p.Q + qq) * p.issuer_cols +
                          (uint32_t)ab * p.acc_cols + c0,
                      r);
              tc_wait_ld();
#pragma unroll
              for (int n = 0; n < 16; ++n) acc1[n] += __uint_as_float(r[n]);
            }
          }
          if (kGU) {
            float* hrow = ws.h + (size_t)(pos0 + c0) * p.I + (size_t)tile * 128 + m;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              if (n < cnt) {
                const float hv = silu_f(acc0[n] * sc0) * (acc1[n] * sc1);
                hrow[(size_t)n * p.I] = hv;
                cur_amax = fmaxf(cur_amax, fabsf(hv));
              }
            }
          } else {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              if (n < cnt) {
                const int pair = sm.pairs[c0 + n];
                ws.o[(size_t)pair * p.H + (size_t)tile * 128 + m] = acc0[n] * sc0;
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.acc_empty[ab]);
      ++cur_tiles;
    }
    if (kGU && cur_e >= 0) {
      float am = warp_max(cur_amax);
      if (lane == 0 && am > 0.0f) atomic_max_nonneg(ws.h_amax + cur_e, am);
      __threadfence();
      tc_named_sync();
      if (t == 0) {
        const unsigned old = atomicAdd(ws.done + cur_e, (unsigned)cur_tiles);
        *sm.flag = (old + (unsigned)cur_tiles == (unsigned)p.tiles);
      }
      tc_named_sync();
      if (*sm.flag) {
        __threadfence();
        tc_quantize_expert_h(p, cur_e, cur_pos0, cur_ne, t);
        tc_named_sync();
        if (t == 0) {
          ws.done[cur_e] = 0u;
          ws.h_amax[cur_e] = 0u;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

// ======================================================================
// Pooler gather: the MoE input's codes in pooled order (the B operand of the
// gate/up MMAs) and its scale lines (one 16-byte line per row and MMA of 64:
// bytes 0-3 the four block scales), stored MMA-major [K/64][rows*k][16] so a
// 3D tensor-map box (16 B, 32 rows, 4 MMAs) lands as four tcgen05.cp atoms.
// One warp per pooled position.
__global__ void pool_gather_kernel(PoolParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const Workspace& ws = p.ws;
  const int lane = threadIdx.x & 31;
  const int pos = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (pos >= p.rows * p.k) return;
  const int row = __ldcg(ws.pair_order + pos) / p.k;
  const uint4* src = reinterpret_cast<const uint4*>(ws.x_codes + (size_t)row * (p.H / 2));
  uint4* dst = reinterpret_cast<uint4*>(ws.x_pool + (size_t)pos * (p.H / 2));
  for (int c = lane; c < p.H / 32; c += 32) dst[c] = __ldcg(src + c);
  const uint32_t* sfs = reinterpret_cast<const uint32_t*>(ws.x_sf + (size_t)row * (p.H / 16));
  uint4* lines = reinterpret_cast<uint4*>(ws.x_lines);
  for (int l = lane; l < p.H / 64; l += 32)
    lines[(size_t)l * p.ws_pairs + pos] = make_uint4(__ldcg(sfs + l), 0u, 0u, 0u);
}

// Weight scales -> per-MMA atoms for tcgen05.cp (32x128b.warpx4):
// atom (row tile, K-block, MMA k) is 512 bytes, byte 16*m0 + 4*m1 + j holds
// the scale of row m0 + 32*m1, 16-block 4k + j; zero beyond K.
__global__ void sf_atoms_kernel(const uint8_t* __restrict__ sf, int64_t rows, int ks, int kblk,
                                uint8_t* __restrict__ out) {
  const int64_t total = (rows / 128) * (int64_t)kblk * 2048;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t atom = i / 512;
    const int byte = (int)(i % 512);
    const int k = (int)(atom % 4);
    const int64_t kb = (atom / 4) % kblk;
    const int64_t rt = atom / 4 / kblk;
    const int m0 = byte / 16, m1 = (byte % 16) / 4, j = byte % 4;
    const int64_t r = rt * 128 + m0 + 32 * m1;
    const int64_t col = kb * 16 + 4 * k + j;
    out[i] = (col < ks) ? sf[r * ks + col] : (uint8_t)0;
  }
}

cudaError_t launch_tc_experts(const TcParams& p, const CUtensorMap& a, const CUtensorMap& b,
                              const CUtensorMap& sfb, int grid, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(32 * (1 + p.P + 4), 1, 1);
  cfg.dynamicSmemBytes = tc_smem_bytes(p);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.mode == kGateUp) return cudaLaunchKernelEx(&cfg, tc_expert_kernel<true>, p, a, b, sfb);
  return cudaLaunchKernelEx(&cfg, tc_expert_kernel<false>, p, a, b, sfb);
}

cudaError_t tc_set_smem(size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(tc_expert_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_expert_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

size_t tc_smem_bytes(const TcParams& p) {
  return 1024 + (size_t)kTcCtrl + (size_t)p.NS * p.stage_stride;  // + alignment slack
}

size_t tc_ctrl_bytes() { return (size_t)kTcCtrl; }

cudaError_t launch_pool_gather(const PoolParams& p, cudaStream_t s, bool pdl) {
  const int per = 4;  // warps (pooled positions) per CTA
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.rows * p.k + per - 1) / per, 1, 1);
  cfg.blockDim = dim3(32 * per, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pool_gather_kernel, p);
}

cudaError_t launch_sf_atoms(const uint8_t* sf, int64_t rows, int ks, int kblk, uint8_t* out,
                            cudaStream_t s) {
  const int64_t total = (rows / 128) * (int64_t)kblk * 2048;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  sf_atoms_kernel<<<(unsigned)blocks, 256, 0, s>>>(sf, rows, ks, kblk, out);
  return cudaGetLastError();
}

}  // namespace moe
