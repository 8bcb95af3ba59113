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
#include "routing.cuh"
#include "tc_internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int kTcMaxThreads = 32 * (1 + 4 + 4);  // producer, up to 4 MMA issuers, 4 epilogue warps
constexpr int kEpiThreads = 128;
constexpr int kMaxPairsTc = 128;
constexpr int kTcCtrl = 4096;             // barriers, tables, flags
// Named barriers of the switch from gate/up to down (2 is the epilogue's own)
constexpr int kBarSwitch = 3;    // every warp: the epilogue has read its last accumulators
constexpr int kBarDownInit = 4;  // producer and issuers: the down barriers are initialised
constexpr int kBarDownEpi = 5;   // the producer warp to the epilogue: the same

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

// ------------------------------------------------------------ shared memory

constexpr int kItemRing = 4;  // items published ahead by the producer

struct TcSmem {
  uint64_t* full;        // [NS][Q]   TMA bytes landed, one barrier per stage and K-phase group
  uint64_t* empty;       // [NS]      every issuer that reads the stage is done (T arrivals)
  uint64_t* acc_full;    // [4]       accumulator buffer ready for the epilogue (P arrivals)
  uint64_t* acc_empty;   // [4]       epilogue done reading it (4 arrivals)
  uint64_t* slot_free;   // [4][2]    an issuer's scale slot may be overwritten
  uint64_t* drain;       // [4]       every MMA of an issuer done
  uint64_t* item_full;   // [kItemRing]  an item published by the producer
  uint64_t* item_empty;  // [kItemRing]  read by every issuer and the epilogue (P + 1 arrivals)
  int4* items;           // [kItemRing]  (item, expert, first pooled position, pairs); item < 0: end
  int* pairs;            // [kMaxPairsTc]
  int* flag;
  uint32_t* tmem_base;
  unsigned* act;         // [kMaxPairsTc]  local routing: packed work item per active expert
  int* porder;           // [kMaxPairsTc]  local routing: pair id at each pooled position
  uint8_t* stages;
};

__device__ __forceinline__ TcSmem tc_carve(uint8_t* base) {
  TcSmem s;
  s.full = reinterpret_cast<uint64_t*>(base);
  s.empty = s.full + 32;
  s.acc_full = s.empty + 16;
  s.acc_empty = s.acc_full + 4;
  s.slot_free = s.acc_empty + 4;
  s.drain = s.slot_free + 8;                 // 68 barriers: 544 bytes
  s.item_full = reinterpret_cast<uint64_t*>(base + 576);
  s.item_empty = s.item_full + kItemRing;
  s.items = reinterpret_cast<int4*>(base + 640);
  s.pairs = reinterpret_cast<int*>(base + 704);
  s.flag = s.pairs + kMaxPairsTc;
  s.tmem_base = reinterpret_cast<uint32_t*>(s.flag + 4);
  s.act = reinterpret_cast<unsigned*>(base + 1280);
  s.porder = reinterpret_cast<int*>(base + 1280 + 4 * kMaxPairsTc);
  s.stages = base + kTcCtrl;
  return s;
}


// Every barrier of one projection's pipeline (init, or inval before the
// shared memory takes the other projection's layout), spread over the lanes
// of one warp: lane l takes the barriers j = l mod 32 of the list below.
__device__ void tc_barriers(const TcParams& p, const TcSmem& sm, bool init, int lane) {
  const int nfull = p.NS * p.Q, nb = nfull + p.NS + 8 + 8 + 4 + 2 * kItemRing;
  for (int j = lane; j < nb; j += 32) {
    uint64_t* b;
    uint32_t count = 1;
    int i = j;
    if (i < nfull) {
      b = &sm.full[i];
    } else if ((i -= nfull) < p.NS) {
      b = &sm.empty[i];
      count = (uint32_t)p.T;
    } else if ((i -= p.NS) < 4) {
      b = &sm.acc_full[i];
      count = (uint32_t)p.P;
    } else if ((i -= 4) < 4) {
      b = &sm.acc_empty[i];
      count = kEpiThreads / 32;
    } else if ((i -= 4) < 8) {
      b = &sm.slot_free[i];
    } else if ((i -= 8) < 4) {
      b = &sm.drain[i];
    } else if ((i -= 4) < kItemRing) {
      b = &sm.item_full[i];
    } else {
      b = &sm.item_empty[i - kItemRing];
      count = (uint32_t)p.P + 1;
    }
    if (init)
      mbar_init(b, count);
    else
      mbar_inval(b);
  }
  if (init) mbar_fence_init();
}

__device__ __forceinline__ int4 unpack_expert(unsigned w) {
  const unsigned v = w - 1u;
  return make_int4((int)(v & 1023u), (int)((v >> 10) & 4095u), (int)(v >> 22), 0);
}

__device__ __forceinline__ bool tc_item_ok(const TcParams& p, int4 et) {
  return et.x >= 0 && et.x < p.E && et.y >= 0 && et.z >= 1 && et.z <= kVirtualPairs &&
         et.y + et.z <= p.ws_pairs;
}

// Gate/up item it: tile it % tiles of virtual expert it / tiles (an active
// expert's pairs in groups of at most 32), from this CTA's own pooler when it
// routed the rows itself.
__device__ __forceinline__ int4 tc_resolve_gate_up(const TcParams& p, const TcSmem& sm, int it) {
  const unsigned w = p.local_route ? sm.act[it / p.tiles] : __ldcg(p.ws.act_info + it / p.tiles);
  return w ? unpack_expert(w) : make_int4(-1, 0, 0, 0);
}

// An item's K order: stage ks of item it reads K-stage (ks + rot) mod KSTEPS,
// rot = it mod KSTEPS -- a function of the item, so every run sums its
// products in the same order.
__device__ __forceinline__ int tc_item_rot(const TcParams& p, int it) { return it % p.KSTEPS; }
__device__ __forceinline__ int tc_stage_k(const TcParams& p, int ks, int rot) {
  const int k = ks + rot;
  return k >= p.KSTEPS ? k - p.KSTEPS : k;
}

// Stage ks of an item (expert e, output tile, nt activation tiles from row
// brow) as the gg-th stage through the ring, its slot already free; the item
// streams its K-blocks from stage rot on (tc_stage_k), so that CTAs which
// start items together do not all read the same offsets.  wts
// arms the stage's full barrier for every byte (toggling its bit in fbits)
// and issues the weight tiles and scale atoms; acts issues the activation
// (gate/up) or h (down) tiles and scale lines.
__device__ __forceinline__ void tc_issue_stage(const TcParams& p, const TcSmem& sm, const CUtensorMap* tm_a,
                                               const CUtensorMap* tm_b, const CUtensorMap* tm_sfb,
                                               uint64_t pol, bool kGU, int e, int tile, int nt, int brow,
                                               int ks, int gg, int rot, bool wts, bool acts, uint32_t& fbits) {
  const int KB = p.KBLK, KPS = p.KPS;
  const int kb = tc_stage_k(p, ks, rot) * KPS;  // first K-block of this stage
  const int nkb = min(KPS, KB - kb);
  const int s = gg % p.NS;
  uint8_t* st = sm.stages + (size_t)s * p.stage_stride;
  const int fb = s * p.Q + ks % p.Q;
  uint64_t* full = &sm.full[fb];
  if (wts) {
    fbits ^= 1u << fb;
    // weight tiles (a missing second K-block of a stage is zero filled and
    // counts in full), the present K-blocks' scale atoms, and per N-tile the
    // activation tiles and scale lines
    const uint32_t sfa_b = 2048u * (uint32_t)nkb;
    const uint32_t bytes = p.a_bytes + sfa_b * (uint32_t)p.T + (uint32_t)(nt * KPS) * (4096u + 2048u);
    mbar_arrive_expect_tx(full, bytes);
    // gate rows (gate/up) or output rows (down) of this tile
    if (p.tiled)  // tiles (e, tile, kb..kb+KPS-1) are contiguous
      tma_3d_hint(st, tm_a, 0, 0, (e * p.row_tiles + tile) * KB + kb, full, pol);
    else if (KPS == 1)
      tma_2d(st, tm_a, kb * 128, e * p.RE + tile * 128, full, pol);
    else
      tma_3d_hint(st, tm_a, 0, e * p.RE + tile * 128, kb, full, pol);
    bulk_g2s_plain(st + p.off_sfa, p.sfa + (((size_t)e * p.row_tiles + tile) * KB + kb) * 2048u, sfa_b, full);
    if (kGU) {  // gate/up stages hold one K-block
      const int ru = p.I / 128 + tile;  // up rows follow the gate rows
      if (p.tiled)
        tma_3d_hint(st + 16384, tm_a, 0, 0, (e * p.row_tiles + ru) * KB + kb, full, pol);
      else
        tma_2d(st + 16384, tm_a, kb * 128, e * p.RE + ru * 128, full, pol);
      bulk_g2s_plain(st + p.off_sfa + 2048, p.sfa + (((size_t)e * p.row_tiles + ru) * KB + kb) * 2048u, 2048u,
                     full);
    }
  }
  if (acts) {
    for (int t = 0; t < nt; ++t) {
      if (KPS == 1)
        tma_2d_plain(st + p.off_b + t * 4096, tm_b, kb * 128, brow + 32 * t, full);
      else
        tma_3d(st + p.off_b + t * 4096 * KPS, tm_b, 0, brow + 32 * t, kb, full);
      tma_3d(st + p.off_sfb + t * 2048 * KPS, tm_sfb, 0, brow + 32 * t, kb * 4, full);
    }
  }
}

// In-kernel routing and pooler (at most 8 rows, so at most 128 pairs and at
// most 8 pairs per expert: one work item per active expert).  Every CTA
// routes the rows itself, one warp per row, from the router's logits, then
// pools the pairs in shared memory with bitmaps: each pair sets its expert's
// bit in an E-bit map and its row's bit in the expert's row mask; one warp
// scan of the map's population counts numbers the active experts (ascending),
// a second scan over the active experts' pair counts gives each one's first
// pooled position, and a pair's position is that plus the number of earlier
// rows routed to the same expert -- experts ascend and rows ascend within an
// expert, as the pooler defines.  Every CTA computes the same result.  The
// first CTA also writes the workspace copies -- ids, gates, flags, logits,
// count, offset, pair order, active list, work items -- that the next
// boundary's gather and the staged checks read.  The transient arrays live
// in the stage ring, which no copy has touched yet.  Returns the number of
// work items.
__device__ int tc_local_route(const TcParams& p, const TcSmem& sm) {
  const Workspace& ws = p.ws;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = p.k, E = p.E, rows = p.rows, npairs = rows * k;
  const int EW = (E + 31) >> 5;                                // words of the expert map (<= 32)
  const bool lead = blockIdx.x == 0;
  int* sids = reinterpret_cast<int*>(sm.stages);               // [128] the routed ids
  unsigned* emap = reinterpret_cast<unsigned*>(sids + kMaxPairsTc);  // [32] bit e: expert e is active
  int* wbase = reinterpret_cast<int*>(emap + 32);              // [32] active experts below each map word
  int* aoff = wbase + 32;                                      // [129] first pooled position per active index
  unsigned* rmask = reinterpret_cast<unsigned*>(aoff + kMaxPairsTc + 1);  // [E] rows routed to each expert
  float* lg = reinterpret_cast<float*>(rmask + 1024);          // [rows][E] scratch above 256 experts
  for (int i = tid; i < EW; i += blockDim.x) emap[i] = 0u;
  for (int i = tid; i < E; i += blockDim.x) rmask[i] = 0u;
  if (warp < rows) {
    const RouteRow rr{ws.logit_part, 1, rows, E, k, nullptr,
                      lead ? ws.logits : nullptr, lead ? ws.ids : nullptr,
                      lead ? ws.gates : nullptr, lead ? ws.flags : nullptr, ws.err, sids};
    route_row(rr, warp, lg + warp * E);
  }
  __syncthreads();
  int e = -1, r = 0;
  if (tid < npairs) {
    e = sids[tid];
    r = tid / k;
    if (e >= 0 && e < E) {
      atomicOr(&emap[e >> 5], 1u << (e & 31));
      atomicOr(&rmask[e], 1u << r);
    } else {
      e = -1;                      // out of range: latched by the routing, not pooled
    }
  }
  __syncthreads();
  // the active experts below each map word (warp 0: one word per lane)
  if (warp == 0) {
    const int c = lane < EW ? __popc(emap[lane]) : 0;
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < EW) wbase[lane] = inc - c;
  }
  __syncthreads();
  const bool valid = e >= 0;
  int a = 0, rank = 0, cnt = 0;
  if (valid && MOE_IN_BOUNDS(r < 32, ws.err)) {
    a = wbase[e >> 5] + __popc(emap[e >> 5] & ((1u << (e & 31)) - 1u));  // active index of e
    const unsigned m = rmask[e];
    rank = __popc(m & ((1u << r) - 1u));                                   // earlier rows of e
    cnt = __popc(m);
    if (rank == 0) aoff[a] = cnt;
  }
  const int n_items = __syncthreads_count(valid && rank == 0);
  // first pooled position of each active expert: a scan of the pair counts
  // in active order (warp 0, four per lane)
  if (warp == 0) {
    int v[4], c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[j] = 4 * lane + j < n_items ? aoff[4 * lane + j] : 0;
      c += v[j];
    }
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    int run = inc - c;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (4 * lane + j < n_items) aoff[4 * lane + j] = run;
      run += v[j];
    }
    if (lane == 31) aoff[kMaxPairsTc] = inc;                   // every pooled pair
  }
  __syncthreads();
  const int n_valid = aoff[kMaxPairsTc];
  if (valid && MOE_IN_BOUNDS(a < kMaxPairsTc && aoff[a] + rank < npairs, ws.err)) {
    const int pos = aoff[a] + rank;
    sm.porder[pos] = tid;
    if (rank == 0) {
      const unsigned wi = pack_expert(e, aoff[a], cnt);
      sm.act[a] = wi;
      if (lead) {
        ws.active[a] = e;
        ws.act_info[a] = wi;
      }
    }
    if (lead) {
      ws.pair_order[pos] = tid;
      ws.pos_of_pair[tid] = pos;
    }
  }
  if (lead) {
    // every expert's count and first pooled position (that of the first
    // active expert at or above it)
    for (int x = tid; x < E; x += blockDim.x) {
      const int ax = wbase[x >> 5] + __popc(emap[x >> 5] & ((1u << (x & 31)) - 1u));
      ws.count[x] = __popc(rmask[x]);
      ws.offset[x] = ax < n_items ? aoff[ax] : n_valid;
    }
    if (tid == 0) {
      ws.offset[E] = n_valid;
      ws.n_active[0] = n_items;
      ws.n_virtual[0] = n_items;
    }
  }
  // the scratch was written through the generic proxy; the stage ring is
  // next written by the TMA (async proxy)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  return n_items;
}

// Down item it: tile it % tiles of virtual expert it / tiles -- under
// in-kernel routing the active expert of that index, else the one whose h
// became ready in that place.  Waits (bounded) until that expert is
// published; the acquire and the proxy fence make its h codes and scale
// lines visible to the TMA.
__device__ __forceinline__ bool tc_resolve_down(const TcParams& p, int it, int4& et) {
  const unsigned* slot = p.ws.ready_info + it / p.tiles;
  unsigned w = ld_acquire_u32(slot);
  if (!w) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
      w = ld_acquire_u32(slot);
      if (w) break;
      if ((i & 63u) == 0u && global_ns() - t0 > p.ws.wait_ns) return false;
    }
  }
  fence_proxy_async_global();
  et = unpack_expert(w);
  return true;
}

// Producer side of the item ring: publish item j (bounded wait for the slot).
__device__ __forceinline__ bool ring_put(const TcSmem& sm, int j, int4 v, uint64_t limit) {
  const int r = j % kItemRing;
  if (j >= kItemRing && !mbar_wait(&sm.item_empty[r], (uint32_t)((j / kItemRing) - 1) & 1u, limit))
    return false;
  sm.items[r] = v;
  mbar_arrive(&sm.item_full[r]);
  return true;
}

// One consumer thread's read of item j.
__device__ __forceinline__ bool ring_get(const TcSmem& sm, int j, int4& v, uint64_t limit) {
  const int r = j % kItemRing;
  if (!mbar_wait(&sm.item_full[r], (uint32_t)(j / kItemRing) & 1u, limit)) return false;
  v = sm.items[r];
  mbar_arrive(&sm.item_empty[r]);
  return true;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Barrier over the four epilogue warps only.
__device__ __forceinline__ void tc_named_sync() { named_bar(2, kEpiThreads); }

// The last CTA to finish an expert's gate/up tiles quantizes its h rows (one
// NVFP4 tensor per expert): codes, block scales and the per-MMA scale lines
// the down projection streams as its B-operand scales.
__device__ void tc_quantize_expert_h(const TcParams& p, int e, int pos0, int ne, int t) {
  const Workspace& ws = p.ws;
  const float amax = __uint_as_float(__ldcg(ws.h_amax + e));
  const float sg = __fdiv_rn(amax, 2688.0f);
  const int bpr = p.I / 16;
  // blocks 4m..4m+3 of a row sit in four adjacent lanes (bpr and the stride
  // are multiples of 4, so the four are active together): the lane of block
  // 4m gathers their scales into the row's scale line m (one 16-byte line per
  // row and MMA of 64: bytes 0-3 the four block scales, the rest zero)
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
    const unsigned mask = __activemask();
    const uint32_t s1 = __shfl_down_sync(mask, sb, 1), s2 = __shfl_down_sync(mask, sb, 2),
                   s3 = __shfl_down_sync(mask, sb, 3);
    if ((blk & 3) == 0)
      *reinterpret_cast<uint4*>(ws.h_lines + ((size_t)(blk >> 2) * p.ws_pairs + row) * 16) =
          make_uint4(sb | (s1 << 8) | (s2 << 16) | (s3 << 24), 0u, 0u, 0u);
  }
  if (t == 0) ws.h_sg[e] = sg;
}

// Gate/up epilogue: this CTA has finished `tiles` tiles of expert e (over
// any of its virtual parts).  Adds its max |h| and tile count; the CTA that
// completes the expert -- every tile of every part -- quantizes all of the
// expert's h rows and publishes its parts to the down projection.
__device__ void tc_finish_expert(const TcParams& p, const TcSmem& sm, int e, int tiles,
                                 float amax_part, int t, int pos0_local, int ne_local, int a_local) {
  const Workspace& ws = p.ws;
  // under local routing an expert is one work item: its pooled rows are the item's
  const int pos0 = p.local_route ? pos0_local : __ldcg(ws.offset + e);
  int ne = p.local_route ? ne_local : __ldcg(ws.offset + e + 1) - pos0;
  if (!MOE_IN_BOUNDS(pos0 >= 0 && ne >= 1 && pos0 + ne <= p.ws_pairs, ws.err)) ne = 0;
  const int parts = (ne + kVirtualPairs - 1) / kVirtualPairs;
  const float am = warp_max(amax_part);
  if ((t & 31) == 0 && am > 0.0f) atomic_max_nonneg(ws.h_amax + e, am);
  __threadfence();
  tc_named_sync();
  if (t == 0) {
    const unsigned old = atomicAdd(ws.done + e, (unsigned)tiles);
    *sm.flag = (old + (unsigned)tiles == (unsigned)(p.tiles * parts));
  }
  tc_named_sync();
  if (*reinterpret_cast<volatile int*>(sm.flag)) {
    __threadfence();
    tc_quantize_expert_h(p, e, pos0, ne, t);
    fence_proxy_async_global();
    __threadfence();
    tc_named_sync();
    if (t == 0) {
      ws.done[e] = 0u;
      ws.h_amax[e] = 0u;
      if (p.local_route) {
        // one part per expert (at most 8 pairs), published at its active
        // index: the down items are numbered in active order
        if (!p.withhold_ready && MOE_IN_BOUNDS(a_local >= 0 && a_local < p.E && parts == 1, ws.err))
          st_release_u32(ws.ready_info + a_local, pack_expert(e, pos0, ne));
      } else {
        const unsigned slot = atomicAdd(ws.counters + 3, (unsigned)parts);
        const unsigned cap = (unsigned)virtual_slots(p.E, p.ws_pairs);
        for (int g = 0; g < parts && !p.withhold_ready; ++g)
          if (slot + g < cap)
            st_release_u32(ws.ready_info + slot + g,
                           pack_expert(e, pos0 + kVirtualPairs * g, min(kVirtualPairs, ne - kVirtualPairs * g)));
      }
    }
  }
  tc_named_sync();
}

// ======================================================================
// One projection's pipeline over dynamically claimed items.  Warp 0:
// producer (claims items, streams their stages); warps 1..P: MMA issuers
// (issuer i = type ty * Q + phase q: accumulator type ty -- gate or up --
// and the stages ks = q mod Q); warps epi0..epi0+3: epilogue.  Issuer warps
// beyond this projection's P sit the projection out.
template <bool kGU>
__device__ __forceinline__ void tc_phase(const TcParams& p, const CUtensorMap* tm_a,
                                         const CUtensorMap* tm_b, const CUtensorMap* tm_sfb,
                                         const TcSmem& sm, uint32_t tmem, int n_items, int epi0,
                                         int first_claim = -1, const TcParams* pdn = nullptr,
                                         int* dn_claim = nullptr) {
  const Workspace& ws = p.ws;
  const uint64_t lim = ws.wait_ns;  // every wait's limit
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int KB = p.KBLK;      // K-blocks of 256 per item
  const int KPS = p.KPS;      // K-blocks per stage
  const int KS = p.KSTEPS;    // stages per item

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      unsigned* claim = ws.counters + (kGU ? 1 : 2);
      int g = 0;           // stages issued = item * KS + ks
      uint32_t fbits = 0;  // per (stage, group) full barrier: parity of fills issued
      bool ok = true;
      // the first claim may have been made already (its latency hidden under the routing)
      // gate/up items below the grid size are taken statically (item b by CTA b)
      const int cbase = kGU ? (int)gridDim.x : 0;
      int it = first_claim >= 0 ? first_claim : (int)atomicAdd(claim, 1u) + cbase;
      int nxt = 0;  // the next claim (raw: the grid offset is added only at its use)
      // Down items under in-kernel routing are numbered in active order, so
      // the expert is known at the claim: the stages' weights (and their
      // scale atoms) go out before the expert's h is published, and only the
      // h tiles wait for it.  Elsewhere down items are numbered in the order
      // the experts' h became ready.
      const bool early = !kGU && p.local_route;
      int e = 0, tile = 0, nt = 0, brow = 0, rot = 0;
      // Stage ks of the current item as the g-th stage through the ring:
      // wts arms its full barrier for every byte and issues the weight tiles
      // and scale atoms (waiting, bounded, for the slot); acts issues the
      // activation (gate/up) or h (down) tiles and scale lines.
      auto stage = [&](int ks, int gg, bool wts, bool acts) -> bool {
        const int s = gg % p.NS;
        if (wts && gg >= p.NS && !mbar_wait(&sm.empty[s], ((gg / p.NS) - 1) & 1, lim)) return false;
        tc_issue_stage(p, sm, tm_a, tm_b, tm_sfb, pol, kGU, e, tile, nt, brow, ks, gg, rot, wts, acts, fbits);
        return true;
      };
      for (int j = 0;; ++j) {
        int4 et = make_int4(-1, 0, 0, 0);
        bool live = ok && it < n_items;
        int npre = 0;  // stages whose weights went out before the item was ready
        if (live) {
          if (kGU || early) {
            et = kGU ? tc_resolve_gate_up(p, sm, it) : unpack_expert(sm.act[it / p.tiles]);
          } else if (!tc_resolve_down(p, it, et)) {
            latch_error(ws.err, kDevWaitTimeout);
            live = ok = false;
          }
          if (live && !tc_item_ok(p, et)) {
            latch_error(ws.err, kDevBadRouting);
            live = ok = false;
          }
        }
        if (live) {
          e = et.x;
          tile = it % p.tiles;
          nt = (et.z + 31) / 32;
          brow = (kGU && p.direct) ? 0 : et.y;  // first B row
          rot = tc_item_rot(p, it);
        }
        if (live && early) {
          // A ready expert takes the usual path (its stages' weights and h
          // tiles together).  Until it is ready, the weights of its stages go
          // out as ring slots come free -- only slots that earlier items
          // release: a slot this item itself holds would wait on its own h.
          const unsigned* slot = ws.ready_info + it / p.tiles;
          const int cap = min(KS, p.NS);
          unsigned w = ld_acquire_u32(slot);
          const uint64_t t0 = global_ns();
          for (uint32_t i = 1; !w; ++i) {
            for (int gg = g + npre;
                 npre < cap && (gg < p.NS || mbar_test(&sm.empty[gg % p.NS], ((gg / p.NS) - 1) & 1));
                 ++gg) {
              stage(npre, gg, true, false);  // its slot is free: no wait
              ++npre;
            }
            w = ld_acquire_u32(slot);
            if (!w && (i & 63u) == 0u && global_ns() - t0 > lim) break;
          }
          g += npre;
          if (!w) {
            latch_error(ws.err, kDevWaitTimeout);
            live = ok = false;
          } else {
            fence_proxy_async_global();
            const int4 wt = unpack_expert(w);
            if (!MOE_IN_BOUNDS(wt.x == et.x && wt.y == et.y && wt.z == et.z, ws.err)) live = ok = false;
          }
        }
        // the item is handed to the issuers and the epilogue only once it is
        // ready (the epilogue reads the expert's h scale)
        if (!ring_put(sm, j, live ? make_int4(it, et.x, et.y, et.z) : make_int4(-1, 0, 0, 0), lim)) {
          latch_error(ws.err, kDevWaitTimeout);
          break;
        }
        if (!live) {
          // gate/up claims ran out (in-kernel routing): claim this CTA's first
          // down item now -- every gate/up item is claimed -- so the claim's
          // latency hides under the CTA's last gate/up stages and epilogue
          if (kGU && ok && pdn && pdn->local_route && dn_claim) *dn_claim = (int)atomicAdd(ws.counters + 2, 1u);
          break;
        }
        for (int ks = 0; ks < npre; ++ks) stage(ks, g - npre + ks, false, true);
        // the next claim goes out once this item's first copies are issued
        // (its latency then hides under the item)
        bool claimed = false;
        if (npre > 0) {
          nxt = (int)atomicAdd(claim, 1u);
          claimed = true;
        }
        for (int ks = npre; ks < KS; ++ks, ++g) {
          if (!stage(ks, g, true, true)) {
            latch_error(ws.err, kDevWaitTimeout);
            ok = false;
            break;
          }
          if (!claimed) {
            nxt = (int)atomicAdd(claim, 1u);
            claimed = true;
          }
        }
        if (!claimed) nxt = (int)atomicAdd(claim, 1u);
        it = nxt + cbase;
      }
      // every issued copy lands before the pipeline is torn down: the last
      // fill of a stage was issued only after every earlier fill of it had
      // been consumed
      for (int s = 0; s < p.NS && s < g; ++s) {
        const int last = s + p.NS * ((g - 1 - s) / p.NS);
        const int fb = s * p.Q + (last % KS) % p.Q;
        if (!mbar_wait(&sm.full[fb], ((fbits >> fb) & 1u) ^ 1u, lim)) latch_error(ws.err, kDevWaitTimeout);
      }
      // and the issuers' releases of every stage have arrived (no commit may
      // land on a barrier after it is re-initialised for the next projection)
      if (ok)
        for (int s = 0; s < p.NS && s < g; ++s)
          if (!mbar_wait(&sm.empty[s], (uint32_t)((g - 1 - s) / p.NS) & 1u, lim))
            latch_error(ws.err, kDevWaitTimeout);
    }
  } else if (warp <= p.P) {
    // --------------------------------------------------------- MMA issuers
    const int i = warp - 1;
    const int ty = i / p.Q, q = i % p.Q;
    if (lane == 0) {
      const uint32_t ibase = tmem + (uint32_t)i * p.issuer_cols;
      int c = 0;          // stages handled
      uint32_t fpar = 0;  // bit s: parity of this group's next phase of full[s][q]
      bool ok = true;
      for (int j = 0; ok; ++j) {
        int4 v;
        if (!ring_get(sm, j, v, lim)) {
          latch_error(ws.err, kDevWaitTimeout);
          break;
        }
        if (v.x < 0) break;
        const int nt = (v.w + 31) / 32;
        const int ab = j % p.dbuf;  // accumulator buffer of item j
        const int use = j / p.dbuf;
        if (use >= 1 && !mbar_wait(&sm.acc_empty[ab], (use - 1) & 1, lim)) {
          latch_error(ws.err, kDevWaitTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t dcol = ibase + (uint32_t)ab * p.acc_cols;
        bool first = true;
        const int rot = tc_item_rot(p, v.x);
        for (int ks = q; ks < KS; ks += p.Q, ++c) {
          const int g = j * KS + ks;
          const int nkb = min(KPS, KB - tc_stage_k(p, ks, rot) * KPS);
          const int s = g % p.NS;
          const uint32_t par = (fpar >> s) & 1u;
          fpar ^= 1u << s;
          if (!mbar_wait(&sm.full[s * p.Q + q], par, lim)) {
            latch_error(ws.err, kDevWaitTimeout);
            ok = false;
            break;
          }
          const int slot = c % p.sfslots;
          if (c >= p.sfslots &&
              !mbar_wait(&sm.slot_free[i * 2 + slot], ((c / p.sfslots) - 1) & 1, lim)) {
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
      // everything this thread issued completes before the pipeline is torn
      // down, and the commits to its scale slots have arrived
      tc_commit(&sm.drain[i]);
      if (!mbar_wait(&sm.drain[i], 0, lim)) latch_error(ws.err, kDevWaitTimeout);
      if (ok)
        for (int sl = 0; sl < p.sfslots && sl < c; ++sl)
          if (!mbar_wait(&sm.slot_free[i * 2 + sl], (uint32_t)((c - 1 - sl) / p.sfslots) & 1u, lim))
            latch_error(ws.err, kDevWaitTimeout);
    }
  } else if (warp >= epi0) {
    // ----------------------------------------------------------- epilogue
    const int t = tid - 32 * epi0;      // 0..127
    const int qd = warp & 3;            // TMEM lane quadrant of this warp
    const int m = 32 * qd + lane;       // weight row within the tile
    const int nparts = KS < p.Q ? KS : p.Q;  // K-phase partial accumulators that exist
    const float x_sg = kGU ? __ldcg(ws.x_sg) : 0.0f;
    // h and o are read back soon (the h quantization and the next boundary's
    // gather): keep them in L2 while the weights stream through it
    const uint64_t keep = l2_evict_last_policy();
    int cur_e = -1, cur_pos0 = -1, cur_ne = 0, cur_tiles = 0, cur_a = -1;
    float cur_amax = 0.0f, sc0 = 0.0f, sc1 = 0.0f;
    for (int j = 0;; ++j) {
      // the next item (one thread waits, bounded; the barrier hands the slot
      // and the verdict to all four warps)
      const int r = j % kItemRing;
      if (t == 0) *sm.flag = mbar_wait(&sm.item_full[r], (uint32_t)(j / kItemRing) & 1u, lim) ? 1 : 0;
      tc_named_sync();
      const bool have = *reinterpret_cast<volatile int*>(sm.flag) != 0;
      const int4 v = have ? sm.items[r] : make_int4(-1, 0, 0, 0);
      tc_named_sync();
      if (!have) {
        if (t == 0) latch_error(ws.err, kDevWaitTimeout);
        break;
      }
      if (t == 0) mbar_arrive(&sm.item_empty[r]);
      if (v.x < 0) break;
      const int e = v.y, tile = v.x % p.tiles, pos0 = v.z, ne = v.w;
      // gate/up accumulates per expert (over its virtual parts); down and
      // direct gate/up keep the pair ids of the current virtual part
      const bool new_e = (e != cur_e), new_part = new_e || pos0 != cur_pos0;
      if (new_e && kGU && cur_e >= 0)
        tc_finish_expert(p, sm, cur_e, cur_tiles, cur_amax, t, cur_pos0, cur_ne, cur_a);
      if (new_part && (!kGU || p.direct)) {
        tc_named_sync();  // nobody still reads the previous part's pair ids
        for (int jj = t; jj < ne; jj += kEpiThreads) {
          const int pr = p.local_route ? sm.porder[pos0 + jj] : __ldcg(ws.pair_order + pos0 + jj);
          sm.pairs[jj] = MOE_IN_BOUNDS(pr >= 0 && pr < p.ws_pairs, ws.err) ? pr : -1;
        }
        tc_named_sync();
      }
      cur_pos0 = pos0;
      cur_ne = ne;
      if (new_e) {
        cur_e = e;
        cur_a = v.x / p.tiles;
        cur_tiles = 0;
        cur_amax = 0.0f;
        if (kGU) {
          sc0 = __ldg(p.gscale + 3 * e + 0) * x_sg;
          sc1 = __ldg(p.gscale + 3 * e + 1) * x_sg;
        } else {
          sc0 = __ldg(p.gscale + 3 * e + 2) * __ldcg(ws.h_sg + e);
        }
      }
      const int ab = j % p.dbuf;
      const int use = j / p.dbuf;
      if (t == 0) *sm.flag = mbar_wait(&sm.acc_full[ab], use & 1, lim) ? 1 : 0;
      tc_named_sync();
      const bool got = *reinterpret_cast<volatile int*>(sm.flag) != 0;
      tc_named_sync();
      if (!got) {
        if (t == 0) latch_error(ws.err, kDevWaitTimeout);
        break;
      }
      tc_fence_after();
      const uint32_t lanes = (uint32_t)(32 * qd) << 16;
      const int nt = (kGU && p.direct) ? 0 : (ne + 31) / 32;
      if (kGU && p.direct) {
        // the B columns are the rows: pair jj reads the column of its row
        for (int jj = 0; jj < ne; ++jj) {
          const int pr = sm.pairs[jj];
          if (kBoundsCheck && !MOE_IN_BOUNDS(pr >= 0 && pr / p.k < kVirtualPairs, ws.err)) continue;
          const uint32_t col = (uint32_t)(pr / p.k);
          float g = 0.0f, u = 0.0f;
          for (int qq = 0; qq < nparts; ++qq) {
            uint32_t ra, rb;
            tc_ld1(tmem + lanes + (uint32_t)qq * p.issuer_cols + (uint32_t)ab * p.acc_cols + col, ra);
            tc_ld1(tmem + lanes + (uint32_t)(p.Q + qq) * p.issuer_cols + (uint32_t)ab * p.acc_cols + col,
                   rb);
            tc_wait_ld();
            g += __uint_as_float(ra);
            u += __uint_as_float(rb);
          }
          const float hv = silu_f(g * sc0) * (u * sc1);
          st_keep(ws.h + (size_t)(pos0 + jj) * p.I + (size_t)tile * 128 + m, hv, keep);
          cur_amax = fmaxf(cur_amax, fabsf(hv));
        }
      }
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
            uint32_t rr[16];
            tc_ld16(tmem + lanes + (uint32_t)qq * p.issuer_cols + (uint32_t)ab * p.acc_cols + c0, rr);
            tc_wait_ld();
#pragma unroll
            for (int n = 0; n < 16; ++n) acc0[n] += __uint_as_float(rr[n]);
            if (kGU) {
              tc_ld16(tmem + lanes + (uint32_t)(p.Q + qq) * p.issuer_cols +
                          (uint32_t)ab * p.acc_cols + c0,
                      rr);
              tc_wait_ld();
#pragma unroll
              for (int n = 0; n < 16; ++n) acc1[n] += __uint_as_float(rr[n]);
            }
          }
          if (kGU) {
            float* hrow = ws.h + (size_t)(pos0 + c0) * p.I + (size_t)tile * 128 + m;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              if (n < cnt) {
                const float hv = silu_f(acc0[n] * sc0) * (acc1[n] * sc1);
                st_keep(hrow + (size_t)n * p.I, hv, keep);
                cur_amax = fmaxf(cur_amax, fabsf(hv));
              }
            }
          } else {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
              if (n < cnt) {
                const int pair = sm.pairs[c0 + n];
                if (MOE_IN_BOUNDS(pair >= 0 && pair < p.ws_pairs, ws.err))
                  st_keep(ws.o + (size_t)pair * p.H + (size_t)tile * 128 + m, acc0[n] * sc0, keep);
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
    if (kGU) {
      // its last accumulators are read: the other warps may switch the CTA to
      // the down projection while this expert's publication runs
      tc_fence_before();
      __syncwarp();
      named_bar_arrive(kBarSwitch, (int)blockDim.x);
    }
    if (kGU && cur_e >= 0) tc_finish_expert(p, sm, cur_e, cur_tiles, cur_amax, t, cur_pos0, cur_ne, cur_a);
  }
}

}  // namespace

// ======================================================================
// Routed experts of one layer in one persistent launch: every CTA claims
// gate/up items until they run out, then down items.  Under in-kernel
// routing (at most 8 rows) the down items follow the active order, which is
// also the order the gate/up items were claimed in, and a CTA streams a down
// item's weights before the expert's h is ready; beyond, an expert's down
// items are handed out in the order experts' h became ready.  Either way
// CTAs that finish gate/up early stream down weights instead of idling.  A
// CTA only ever waits for gate/up work that running CTAs have already
// claimed (no CTA claims a down item before every gate/up item is claimed),
// and gate/up work waits for nothing, so the launch needs no co-residency
// guarantee.
__global__ void __launch_bounds__(kTcMaxThreads, 1)
    tc_moe_kernel(const __grid_constant__ TcParams pg, const __grid_constant__ CUtensorMap g_a,
                  const __grid_constant__ CUtensorMap g_b, const __grid_constant__ CUtensorMap g_sfb,
                  const __grid_constant__ TcParams pd, const __grid_constant__ CUtensorMap d_a,
                  const __grid_constant__ CUtensorMap d_b, const __grid_constant__ CUtensorMap d_sfb) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128B-swizzled TMA tiles need 1024-byte aligned destinations: align the
  // base explicitly (the launch adds 1 KB of slack for this)
  uint8_t* smem_base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const TcSmem sm = tc_carve(smem_base);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int epi0 = 1 + (pg.P > pd.P ? pg.P : pd.P);

  // A stage is read by the issuers of K-phase group q = ks mod Q.  When NS is
  // not a multiple of Q the group changes from one fill of a stage to the
  // next, and a parity wait by an issuer that skipped a phase would match the
  // stale parity of the fill before.  So each (stage, group) has its own
  // full barrier: every phase of it is consumed by the same issuers, and each
  // waiter tracks that barrier's parity itself.
  if (warp == 0) tc_barriers(pg, sm, true, tid);
  if (tid == 0) {
    // every descriptor this launch will use, into the TMA unit's cache
    const CUtensorMap* maps[6] = {&g_a, &g_b, &g_sfb, &d_a, &d_b, &d_sfb};
    for (int i = 0; i < 6; ++i)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(maps[i])) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(sm.tmem_base)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // the logits (or the routing and pooled MoE input), the quantized input
  // and the zeroed item counters come from the kernels before
  grid_dep_wait();
  grid_dep_launch();
  int na;
  if (pg.local_route) {
    na = tc_local_route(pg, sm);
    // every router CTA has read max |x|: reset for the next layer's boundary
    if (blockIdx.x == 0 && tid == 0) pg.ws.x_amax[0] = 0u;
  } else {
    na = __ldcg(pg.ws.n_virtual);
  }
  // the first gate/up item of CTA b is item b; later claims count from the
  // grid size
  const int first_claim = tid == 0 ? (int)blockIdx.x : -1;
  const bool na_ok = na >= 0 && na <= virtual_slots(pg.E, pg.ws_pairs);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_base;
  if (!na_ok && tid == 0) latch_error(pg.ws.err, kDevBadRouting);
  const int n_act = na_ok ? na : 0;

  int dn_claim = -1;  // the producer's first down claim, made when gate/up claims run out
  tc_phase<true>(pg, &g_a, &g_b, &g_sfb, sm, tmem, n_act * pg.tiles, epi0, first_claim, &pd, &dn_claim);

  // Once this CTA's gate/up copies have landed, its MMAs completed and its
  // epilogue has read the last accumulators, the shared memory takes the down
  // layout, and the producer and issuers start on the down items while the
  // epilogue publishes its last expert (it joins the down phase after).
  if (warp < epi0) {
    tc_fence_before();
    __syncwarp();
    named_bar(kBarSwitch, (int)blockDim.x);
    tc_fence_after();
    if (warp == 0) {
      tc_barriers(pg, sm, false, tid);
      __syncwarp();
      tc_barriers(pd, sm, true, tid);
    }
    __syncwarp();
    named_bar(kBarDownInit, 32 * epi0);
    if (warp == 0) named_bar_arrive(kBarDownEpi, 32 + kEpiThreads);
  } else {
    __syncwarp();
    named_bar(kBarDownEpi, 32 + kEpiThreads);
    tc_fence_after();
  }

  tc_phase<false>(pd, &d_a, &d_b, &d_sfb, sm, tmem, n_act * pd.tiles, epi0, dn_claim);

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
  if (!MOE_IN_BOUNDS(row >= 0 && row < p.rows, ws.err)) return;
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

cudaError_t launch_tc_moe(const TcParams& gu, const CUtensorMap& gu_a, const CUtensorMap& gu_b,
                          const CUtensorMap& gu_sfb, const TcParams& dn, const CUtensorMap& dn_a,
                          const CUtensorMap& dn_b, const CUtensorMap& dn_sfb, int grid,
                          cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(32 * (1 + (gu.P > dn.P ? gu.P : dn.P) + 4), 1, 1);
  cfg.dynamicSmemBytes = tc_moe_smem_bytes(gu, dn);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_moe_kernel, gu, gu_a, gu_b, gu_sfb, dn, dn_a, dn_b, dn_sfb);
}

// One CTA per 16 KB tile (row tile rt = t / KB, K-block kb = t % KB), 16
// bytes per thread per step.
__global__ void tile_codes_kernel(const uint8_t* __restrict__ src, int inner, int KB,
                                  uint8_t* __restrict__ dst) {
  const int64_t t = blockIdx.x;
  const int64_t row0 = (t / KB) * 128;
  const int kb = (int)(t % KB);
  for (int q = threadIdx.x; q < 1024; q += blockDim.x) {
    const int r = q >> 3, c = (q & 7) * 16;
    const int col = kb * 128 + c;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (col + 16 <= inner) v = __ldg(reinterpret_cast<const uint4*>(src + (row0 + r) * inner + col));
    *reinterpret_cast<uint4*>(dst + t * 16384 + r * 128 + c) = v;
  }
}

cudaError_t launch_tile_codes(const uint8_t* src, int64_t rows, int inner, uint8_t* dst, cudaStream_t s) {
  const int KB = (inner + 127) / 128;
  tile_codes_kernel<<<(unsigned)(rows / 128 * KB), 256, 0, s>>>(src, inner, KB, dst);
  return cudaGetLastError();
}

cudaError_t tc_set_smem(size_t bytes) {
  return cudaFuncSetAttribute(tc_moe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)bytes);
}

size_t tc_smem_bytes(const TcParams& p) {
  return 1024 + (size_t)kTcCtrl + (size_t)p.NS * p.stage_stride;  // + alignment slack
}

size_t tc_moe_smem_bytes(const TcParams& gu, const TcParams& dn) {
  const size_t a = tc_smem_bytes(gu), b = tc_smem_bytes(dn);
  return a > b ? a : b;
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
