// Router GEMV, softmax top-k routing, pooler and the MoE input's NVFP4
// quantization, one kernel.
//
// Page: vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode,
// module docstring "One step of b rows", MoE: "router -> routing -> pooler ->
// routed experts"; SpecializedDecode.build builds one Pooler for all layers
// and batches.  Routing is softmax over all experts, top-k by probability
// (ties to the lower expert id), gates renormalised over the selected k; the
// pooler groups the (row, slot) pairs by expert, experts ascending and rows
// ascending within an expert.
//
// GB300 layout: split-K GEMV.  CTA (g, s, r) owns EG experts (one warp each),
// one H-slice and one block of 8 rows; the warp holds its expert's slice of the router weights in
// registers (fetched before the programmatic-dependency wait, since the
// weights do not depend on the previous kernel) and writes one fp32 partial
// per (row, expert).  Every CTA also quantizes a share of the MoE input's
// 16-element blocks.  The last CTA of a row block to arrive (threadfence +
// counter, no spin) sums its rows' partials in slice order and selects their
// top-k (one warp per row); the last row block to finish builds the pooler's
// arrays over every row.
#include <cooperative_groups.h>

#include "common.cuh"
#include "gemv.cuh"
#include "routing.cuh"

namespace cg = cooperative_groups;

namespace moe {
namespace {

constexpr int kRouterThreads = 256;
constexpr int kRouterWarps = kRouterThreads / 32;
constexpr int kRouterChunks = 4;   // 8-element chunks per lane per slice: slices <= 1024 wide
constexpr int kMaxTopK = 16;
constexpr int kRowBlock = 8;       // rows whose x slice is staged at once

// Shared-memory carve of the routing and pooler tails.
struct RouteSmem {
  float* lg;        // [warps][E]
  int* cnt;         // [E]
  int* off;         // [E+1]
  unsigned* mask;   // [E][RW]
  int* sids;        // [rows * k]
  int* wtot;        // [3][warps]
};

__device__ __forceinline__ RouteSmem route_carve(const RouterParams& p, uint8_t* smem) {
  RouteSmem r;
  const int RW = (p.rows + 31) / 32;
  r.lg = reinterpret_cast<float*>(smem);
  r.cnt = reinterpret_cast<int*>(r.lg + kRouterWarps * p.E);
  r.off = r.cnt + p.E;
  r.mask = reinterpret_cast<unsigned*>(r.off + p.E + 1);
  r.sids = reinterpret_cast<int*>(r.mask + p.E * RW);
  r.wtot = r.sids + p.rows * p.k;
  return r;
}

// Routing of rows [r0, r0 + nr): one warp per row (nr <= warps).
__device__ void route_rows(const RouterParams& p, const RouteSmem& rs, int r0, int nr) {
  const int warp = threadIdx.x >> 5;
  if (warp < nr) {
    const Workspace& ws = p.ws;
    // with the cluster sum the first slice holds the logits, bias included
    const RouteRow rr{ws.logit_part, p.cluster_sum ? 1 : p.S, p.rows, p.E, p.k,
                      p.cluster_sum ? nullptr : p.bias, ws.logits, ws.ids, ws.gates, ws.flags, ws.err,
                      rs.sids};
    route_row(rr, r0 + warp, rs.lg + warp * p.E);
  }
}

// After the pooler: the expert kernel's ready list and item counters start
// empty, and the router's counters are ready for the next layer.
__device__ void pool_reset(const RouterParams& p) {
  const Workspace& ws = p.ws;
  const int V = virtual_slots(p.E, p.rows * p.k);
  for (int v = threadIdx.x; v < V; v += kRouterThreads) ws.ready_info[v] = 0u;
  if (threadIdx.x == 0) {
    ws.counters[0] = 0u;
    ws.counters[1] = 0u;
    ws.counters[2] = 0u;
    ws.counters[3] = 0u;
    ws.x_amax[0] = 0u;
  }
}

// Pooler for at most kRouterThreads pairs, one thread per pair.  A pair's
// rank among its expert's pairs (pairs are in (row, slot) order, so they rank
// by row) is its warp's match count below it plus the matches in earlier
// warps; the counts come from shared-memory atomics.  One block-wide
// exclusive scan over the experts of (count, active flag, work items)
// packed 10 bits each (every field stays below 1024: at most 256 pairs)
// gives each expert its offset, active index and first work item.  The
// results equal the scanning pooler's.
__device__ void pool_small(const RouterParams& p, uint8_t* smem, bool ids_in_smem) {
  const Workspace& ws = p.ws;
  const int E = p.E, npairs = p.rows * p.k, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RouteSmem rs = route_carve(p, smem);
  int* sids = rs.sids;
  int* cnt = rs.cnt;  // counts, then offsets
  int* wtot = rs.wtot;
  for (int e = tid; e < E; e += kRouterThreads) cnt[e] = 0;
  if (!ids_in_smem)
    for (int q = tid; q < npairs; q += kRouterThreads) sids[q] = __ldcg(ws.ids + q);
  __syncthreads();
  const int eq = (tid < npairs) ? sids[tid] : -1;
  const bool valid = eq >= 0 && eq < E;
  const unsigned peers = __match_any_sync(0xffffffffu, valid ? eq : -1 - lane);
  int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid) {
    for (int q = 0; q < warp * 32; ++q) rank += (sids[q] == eq);
    atomicAdd(&cnt[eq], 1);
  }
  __syncthreads();
  const int per = (E + kRouterThreads - 1) / kRouterThreads;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int loc = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    loc += c | ((c > 0) << 10) | (((c + kVirtualPairs - 1) / kVirtualPairs) << 20);
  }
  int inc = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) wtot[warp] = inc;
  __syncthreads();
  int ex = inc - loc;
  for (int w = 0; w < warp; ++w) ex += wtot[w];
  int o = ex & 1023, a = (ex >> 10) & 1023, v = ex >> 20;
  for (int e = e0; e < e1; ++e) {
    const int c = cnt[e];
    cnt[e] = o;
    ws.offset[e] = o;
    ws.count[e] = c;
    if (c > 0) ws.active[a++] = e;
    // the expert's work items: its pairs in groups of at most kVirtualPairs
    for (int g0 = 0; g0 < c; g0 += kVirtualPairs)
      ws.act_info[v++] = pack_expert(e, o + g0, min(kVirtualPairs, c - g0));
    o += c;
  }
  if (tid == kRouterThreads - 1) {
    ws.offset[E] = o;
    ws.n_active[0] = a;
    ws.n_virtual[0] = v;
  }
  __syncthreads();
  if (valid && MOE_IN_BOUNDS(cnt[eq] + rank < npairs, ws.err)) {
    const int pos = cnt[eq] + rank;
    ws.pair_order[pos] = tid;
    ws.pos_of_pair[tid] = pos;
  }
  pool_reset(p);
}

// Pooler over every row, run by the last CTA to finish routing.  The ids are
// in shared memory when one CTA routed every row, else read back.
__device__ void pool_all(const RouterParams& p, uint8_t* smem, bool ids_in_smem) {
  const Workspace& ws = p.ws;
  const int E = p.E, k = p.k, rows = p.rows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const RouteSmem rs = route_carve(p, smem);
  int* cnt = rs.cnt;
  int* off = rs.off;
  const int RW = (rows + 31) / 32;
  unsigned* mask = rs.mask;
  int* sids = rs.sids;
  int* wtot = rs.wtot;
  if (!ids_in_smem)
    for (int q = tid; q < rows * k; q += kRouterThreads) sids[q] = __ldcg(ws.ids + q);

  for (int e = tid; e < E; e += kRouterThreads) {
    cnt[e] = 0;
    for (int w = 0; w < RW; ++w) mask[e * RW + w] = 0u;
  }
  __syncthreads();
  const int npairs = rows * k;
  for (int q = tid; q < npairs; q += kRouterThreads) {
    const int e = sids[q];
    if (e < 0 || e >= E) continue;
    const int r = q / k;
    atomicAdd(&cnt[e], 1);
    atomicOr(&mask[e * RW + (r >> 5)], 1u << (r & 31));
  }
  __syncthreads();
  {
    // block-wide exclusive scan of the counts and of the active flags; each
    // thread owns a range of experts
    const int per = (E + kRouterThreads - 1) / kRouterThreads;
    const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
    int csum = 0, asum = 0, vsum = 0;
    for (int e = e0; e < e1; ++e) {
      csum += cnt[e];
      asum += cnt[e] > 0;
      vsum += (cnt[e] + kVirtualPairs - 1) / kVirtualPairs;
    }
    int ci = csum, ai = asum, vi = vsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tc = __shfl_up_sync(0xffffffffu, ci, o);
      const int ta = __shfl_up_sync(0xffffffffu, ai, o);
      const int tv = __shfl_up_sync(0xffffffffu, vi, o);
      if (lane >= o) {
        ci += tc;
        ai += ta;
        vi += tv;
      }
    }
    if (lane == 31) {
      wtot[warp] = ci;
      wtot[kRouterWarps + warp] = ai;
      wtot[2 * kRouterWarps + warp] = vi;
    }
    __syncthreads();
    int cex = ci - csum, aex = ai - asum, vex = vi - vsum;
    for (int w = 0; w < warp; ++w) {
      cex += wtot[w];
      aex += wtot[kRouterWarps + w];
      vex += wtot[2 * kRouterWarps + w];
    }
    for (int e = e0; e < e1; ++e) {
      off[e] = cex;
      ws.offset[e] = cex;
      ws.count[e] = cnt[e];
      if (cnt[e] > 0) ws.active[aex++] = e;
      // the expert's work items: its pairs in groups of at most kVirtualPairs
      for (int g0 = 0; g0 < cnt[e]; g0 += kVirtualPairs)
        ws.act_info[vex++] = pack_expert(e, cex + g0, min(kVirtualPairs, cnt[e] - g0));
      cex += cnt[e];
    }
    if (tid == kRouterThreads - 1) {
      off[E] = cex;
      ws.offset[E] = cex;
      ws.n_active[0] = aex;
      ws.n_virtual[0] = vex;
    }
  }
  __syncthreads();
  for (int q = tid; q < npairs; q += kRouterThreads) {
    const int e = sids[q];
    if (e < 0 || e >= E) continue;
    const int r = q / k;
    int rank = 0;
    for (int w = 0; w < (r >> 5); ++w) rank += __popc(mask[e * RW + w]);
    rank += __popc(mask[e * RW + (r >> 5)] & ((1u << (r & 31)) - 1u));
    const int pos = off[e] + rank;
    if (!MOE_IN_BOUNDS(pos < npairs, ws.err)) continue;
    ws.pair_order[pos] = q;
    ws.pos_of_pair[q] = pos;
  }
  pool_reset(p);
}

// This CTA's range of the MoE input's 16-element blocks.
__device__ __forceinline__ void quant_range(const RouterParams& p, int& b0, int& b1) {
  const int ncta = gridDim.x * gridDim.y * gridDim.z;
  const int cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  const int nblk = p.rows * (p.H / 16);
  b0 = (int)((long long)cta * nblk / ncta);
  b1 = (int)((long long)(cta + 1) * nblk / ncta);
}

// This CTA's share of the MoE input's NVFP4 quantization (sg: its tensor
// scale).  pre0 / pre1: the thread's first block, already loaded (or
// loaded here when has_pre is false).
__device__ void quantize_share(const RouterParams& p, float sg, bool has_pre = false,
                               uint4 pre0 = make_uint4(0u, 0u, 0u, 0u),
                               uint4 pre1 = make_uint4(0u, 0u, 0u, 0u)) {
  // the MoE input as one NVFP4 tensor: this CTA's share of the 16-blocks,
  // one per thread.  Each block's scale also goes into its 16-byte scale
  // line ([H/64][line_rows][16]: bytes 0-3 the four scales of 64 elements,
  // the rest zero) that the tensor-core experts read when the rows
  // themselves are the MMA's N.
  const Workspace& ws = p.ws;
  const int cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  const int bpr = p.H / 16;
  int b0, b1;
  quant_range(p, b0, b1);
  for (int b = b0 + threadIdx.x; b < b1; b += blockDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)b * 16);
    const bool first = has_pre && b == b0 + (int)threadIdx.x;
    const uint4 q0 = first ? pre0 : __ldcg(src), q1 = first ? pre1 : __ldcg(src + 1);
    float v[16];
    const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&q0);
    const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&q1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f0 = __bfloat1622float2(h0[i]), f1 = __bfloat1622float2(h1[i]);
      v[2 * i] = f0.x;
      v[2 * i + 1] = f0.y;
      v[8 + 2 * i] = f1.x;
      v[8 + 2 * i + 1] = f1.y;
    }
    uint32_t lo, hi, sb;
    quant_block16(v, sg, lo, hi, sb);
    *reinterpret_cast<uint2*>(ws.x_codes + (size_t)b * 8) = make_uint2(lo, hi);
    ws.x_sf[b] = (uint8_t)sb;
    const int row = b / bpr, blk = b % bpr;
    uint8_t* line = ws.x_lines + ((size_t)(blk / 4) * p.line_rows + row) * 16;
    line[blk % 4] = (uint8_t)sb;
    if (blk % 4 == 0) {
      reinterpret_cast<uint32_t*>(line)[1] = 0u;
      reinterpret_cast<uint32_t*>(line)[2] = 0u;
      reinterpret_cast<uint32_t*>(line)[3] = 0u;
    }
  }
  if (cta == 0 && threadIdx.x == 0) ws.x_sg[0] = sg;
}

__global__ void __launch_bounds__(kRouterThreads, 1) router_kernel(RouterParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_last;
  __shared__ float s_part[kRowBlock * kRouterWarps];  // cluster sum: this CTA's [row][expert] partials
  const Workspace& ws = p.ws;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x * p.EG + warp;
  const int sl = blockIdx.y;
  const int nch = p.H / 8;
  const int c0 = sl * nch / p.S, c1 = (sl + 1) * nch / p.S;

  // the slice-0 CTA's bias for its cluster sum (static): before the wait
  const int bias_e = blockIdx.x * p.EG + (int)(threadIdx.x % kRouterWarps);
  const float bias_v = (p.cluster_sum && p.bias && sl == 0 && bias_e < p.E) ? __ldg(p.bias + bias_e) : 0.0f;
  // the expert's slice of the router weights (static): before the wait
  uint4 wv[kRouterChunks];
#pragma unroll
  for (int i = 0; i < kRouterChunks; ++i) {
    const int c = c0 + lane + 32 * i;
    wv[i] = (warp < p.EG && e < p.E && c < c1)
                ? __ldg(reinterpret_cast<const uint4*>(p.wr + (size_t)e * p.H) + c)
                : make_uint4(0u, 0u, 0u, 0u);
  }
  grid_dep_wait();
  grid_dep_launch();
  // this CTA's first quantization block and max |x| (written by the
  // boundary): loads in flight while the dot products run
  uint4 qpre0 = make_uint4(0u, 0u, 0u, 0u), qpre1 = qpre0;
  {
    int qb0, qb1;
    quant_range(p, qb0, qb1);
    const int b = qb0 + threadIdx.x;
    if (b < qb1) {
      const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)b * 16);
      qpre0 = __ldcg(src);
      qpre1 = __ldcg(src + 1);
    }
  }
  const unsigned amax_bits = __ldcg(ws.x_amax);

  // each block of 8 rows in turn: the x slice is staged in shared memory
  // (every load in flight at once, the next block's already in registers
  // while this one is multiplied), then each warp forms its expert's partial
  // dot products from registers and smem
  uint4* xs = reinterpret_cast<uint4*>(smem);  // [kRowBlock][kRouterChunks * 32]
  const int nc = c1 - c0;
  const int nrb = (p.rows + kRowBlock - 1) / kRowBlock;
  constexpr int kStage = kRowBlock * kRouterChunks * 32 / kRouterThreads;  // uint4 per thread
  uint4 pre[kStage];
  auto load_x = [&](int rb) {
    const int r0 = rb * kRowBlock, nr = min(kRowBlock, p.rows - r0);
#pragma unroll
    for (int q = 0; q < kStage; ++q) {
      const int i = threadIdx.x + q * kRouterThreads, rr = i / nc, c = i % nc;
      pre[q] = (i < nr * nc) ? __ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)(r0 + rr) * p.H) + c0 + c)
                             : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  load_x(0);
  for (int rb = 0; rb < nrb; ++rb) {
    const int r0 = rb * kRowBlock, nr = min(kRowBlock, p.rows - r0);
#pragma unroll
    for (int q = 0; q < kStage; ++q) {
      const int i = threadIdx.x + q * kRouterThreads;
      if (i < nr * nc) xs[(i / nc) * (kRouterChunks * 32) + i % nc] = pre[q];
    }
    __syncthreads();
    if (rb + 1 < nrb) load_x(rb + 1);
    if (warp < p.EG && e < p.E) {
      float acc[kRowBlock];
#pragma unroll
      for (int rr = 0; rr < kRowBlock; ++rr) {
        acc[rr] = 0.0f;
        if (rr < nr) {
#pragma unroll
          for (int i = 0; i < kRouterChunks; ++i) {
            const int c = lane + 32 * i;
            if (c < nc) acc[rr] = dot8_bf16(xs[rr * (kRouterChunks * 32) + c], wv[i], acc[rr]);
          }
        }
      }
      // reduce-scatter over the lanes: each exchange halves the rows a lane
      // keeps, so after three exchanges lanes 4m..4m+3 hold row m, and two
      // more sum those four (9 shuffles for the 8 rows, not 40)
      const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4;
      float a4[4], a2[2];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        a4[j] = (h4 ? acc[j + 4] : acc[j]) + __shfl_xor_sync(0xffffffffu, h4 ? acc[j] : acc[j + 4], 16);
#pragma unroll
      for (int j = 0; j < 2; ++j)
        a2[j] = (h3 ? a4[j + 2] : a4[j]) + __shfl_xor_sync(0xffffffffu, h3 ? a4[j] : a4[j + 2], 8);
      float v = (h2 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? a2[0] : a2[1], 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      const int row = lane >> 2;
      if ((lane & 3) == 0 && row < nr) {
        if (p.cluster_sum)
          s_part[row * kRouterWarps + warp] = v;
        else
          ws.logit_part[((size_t)sl * p.rows + r0 + row) * p.E + e] = v;
      }
    }
    __syncthreads();  // the next block's staging reuses xs
  }

  // cluster sum (one block of rows): the partials are published to the
  // cluster, and the barrier's wait hides behind this CTA's quantization
  if (p.cluster_sum) asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // this CTA's share of the MoE input's quantization, before it arrives (the
  // pooler resets max |x| for the next layer once every CTA has arrived)
  quantize_share(p, __fdiv_rn(__uint_as_float(amax_bits), 2688.0f), true, qpre0, qpre1);
  if (p.cluster_sum) {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    // the slice-0 CTA sums the S slices' partials in slice order (the cluster
    // rank is the slice) into the first slice of logit_part
    cg::cluster_group cluster = cg::this_cluster();
    if (sl == 0 && (int)threadIdx.x < p.rows * kRouterWarps) {
      const int r = threadIdx.x / kRouterWarps, wi = threadIdx.x % kRouterWarps;
      const int ee = blockIdx.x * p.EG + wi;
      float acc = 0.0f;
      for (int q = 0; q < p.S; ++q) acc += *cluster.map_shared_rank(&s_part[r * kRouterWarps + wi], q);
      if (p.bias) acc += bias_v;  // the same fp32 sum, then the bias, as the routing would add it
      if (wi < p.EG && ee < p.E) ws.logit_part[(size_t)r * p.E + ee] = acc;
    }
    // every peer keeps its partials until the sums are read
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
  // beyond one block of rows, route_kernel routes the blocks in parallel
  if (nrb > 1) return;
  // the experts kernel routes and pools (and resets max |x| once every
  // router CTA has read it); the boundary cleared its item claims and ready
  // list
  if (p.route_in_experts) return;

  // one block of rows: the last CTA to finish routes them and builds the pooler
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(ws.rg_count, 1u);
    s_last = (old == gridDim.x * gridDim.y - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const RouteSmem rs = route_carve(p, smem);
  route_rows(p, rs, 0, p.rows);
  __syncthreads();
  if (threadIdx.x == 0) ws.rg_count[0] = 0u;  // every CTA has arrived
  if (p.rows * p.k <= kRouterThreads)
    pool_small(p, smem, true);
  else
    pool_all(p, smem, true);
}

// Beyond one block of rows the router's dot products are a GEMM (rows x E x H),
// on the tensor cores: a CTA takes 16 experts and one of the S K-slices,
// each of its 8 warps an eighth of the slice.  A warp keeps its 16 experts'
// weights as mma.sync A fragments in registers for the whole launch (read
// before the dependency wait), and per block of 8 rows loads that block's x
// (the next block's loads in flight meanwhile) as B fragments, with the K
// order permuted as in the streaming projections so each thread's pieces are
// contiguous 16-byte runs; the 8 warps' 16 x 8 tiles are summed in warp order
// through shared memory into the slice's partial logits.  Needs H / S a
// multiple of 256 (a warp's columns in 32-column blocks, at most 4).
__global__ void __launch_bounds__(kRouterThreads, 1) router_mma_kernel(RouterParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float s_tile[128];  // cluster sum: this slice's [16 experts][8 rows] partials
  const Workspace& ws = p.ws;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
  const int e0 = blockIdx.x * 16, sl = blockIdx.y;
  const int W = p.H / p.S, CB = W / 256;
  const int k0 = sl * W + warp * (W / 8) + t * 8;
  uint4 a[2][4];
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int e = e0 + g + 8 * hr;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      a[hr][c] = (c < CB && e < p.E) ? __ldg(reinterpret_cast<const uint4*>(p.wr + (size_t)e * p.H + k0 + c * 32))
                                     : make_uint4(0u, 0u, 0u, 0u);
  }
  grid_dep_wait();
  grid_dep_launch();
  float* red = reinterpret_cast<float*>(smem);  // [8 warps][16 experts x 8 rows]
  const int nrb = (p.rows + kRowBlock - 1) / kRowBlock;
  uint4 bn[4];
  auto load_x = [&](int rb) {
    const int row = rb * kRowBlock + g;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      bn[c] = (c < CB && row < p.rows) ? __ldcg(reinterpret_cast<const uint4*>(p.x + (size_t)row * p.H + k0 + c * 32))
                                       : make_uint4(0u, 0u, 0u, 0u);
  };
  load_x(0);
  for (int rb = 0; rb < nrb; ++rb) {
    uint4 b[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) b[c] = bn[c];
    if (rb + 1 < nrb) load_x(rb + 1);
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (c < CB) {
        mma_16816_bf16(acc, a[0][c].x, a[1][c].x, a[0][c].y, a[1][c].y, b[c].x, b[c].y);
        mma_16816_bf16(acc, a[0][c].z, a[1][c].z, a[0][c].w, a[1][c].w, b[c].z, b[c].w);
      }
    // acc: (expert g, rows 2t, 2t + 1), (expert g + 8, rows 2t, 2t + 1)
    float* mine = red + warp * 128;
    mine[g * 8 + 2 * t] = acc[0];
    mine[g * 8 + 2 * t + 1] = acc[1];
    mine[(g + 8) * 8 + 2 * t] = acc[2];
    mine[(g + 8) * 8 + 2 * t + 1] = acc[3];
    __syncthreads();
    if (threadIdx.x < 128) {
      float v = 0.0f;
#pragma unroll
      for (int w = 0; w < kRouterWarps; ++w) v += red[w * 128 + threadIdx.x];
      const int e = e0 + (threadIdx.x >> 3), r = rb * kRowBlock + (threadIdx.x & 7);
      if (p.cluster_sum)
        s_tile[threadIdx.x] = v;
      else if (e < p.E && r < p.rows)
        ws.logit_part[((size_t)sl * p.rows + r) * p.E + e] = v;
    }
    __syncthreads();
  }
  if (!p.cluster_sum) {
    quantize_share(p, __fdiv_rn(__uint_as_float(__ldcg(ws.x_amax)), 2688.0f));
    return;
  }
  // one block of rows: the S slice CTAs of this group of 16 experts form a
  // cluster; its first CTA sums their [16 experts x 8 rows] tiles in slice
  // order and adds the bias, into logit_part's first slice (the logits), and
  // the barrier's wait hides behind this CTA's share of the quantization
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  quantize_share(p, __fdiv_rn(__uint_as_float(__ldcg(ws.x_amax)), 2688.0f));
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (sl == 0 && threadIdx.x < 128) {
    cg::cluster_group cluster = cg::this_cluster();
    const int e = e0 + (threadIdx.x >> 3), r = threadIdx.x & 7;
    float v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = q < p.S ? *cluster.map_shared_rank(&s_tile[threadIdx.x], q) : 0.0f;
    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < p.S) acc += v[q];
    if (e < p.E && r < p.rows) {
      if (p.bias) acc += __ldg(p.bias + e);
      ws.logit_part[(size_t)r * p.E + e] = acc;
    }
  }
  // every peer keeps its tile until the sums are read
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Beyond one block of rows: after the router's dot products (programmatic
// dependent launch), one CTA per block of 8 rows routes them, a warp per row;
// the last CTA to finish builds the pooler over every row.
__global__ void __launch_bounds__(kRouterThreads, 1) route_kernel(RouterParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ int s_last;
  grid_dep_wait();  // every block's logit partials
  grid_dep_launch();
  const int r0 = blockIdx.x * kRowBlock, nr = min(kRowBlock, p.rows - r0);
  const RouteSmem rs = route_carve(p, smem);
  route_rows(p, rs, r0, nr);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned old = atomicAdd(p.ws.counters, 1u);
    s_last = (old == gridDim.x - 1u);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (p.rows * p.k <= kRouterThreads)
    pool_small(p, smem, false);
  else
    pool_all(p, smem, false);
}

}  // namespace

size_t router_smem_bytes(int E, int rows) {
  const int RW = (rows + 31) / 32;
  const size_t route = (size_t)kRouterWarps * E * 4 + (size_t)E * 4 + (size_t)(E + 1) * 4 +
                       (size_t)E * RW * 4 + (size_t)rows * kMaxTopK * 4 + 3 * kRouterWarps * 4;
  const size_t xslice = (size_t)kRowBlock * kRouterChunks * 32 * 16;
  return route > xslice ? route : xslice;
}

bool router_mma_fits(const RouterParams& p) { return p.H % (p.S * 256) == 0 && p.H / p.S <= 1024; }

cudaError_t launch_router(const RouterParams& p, cudaStream_t s, bool pdl) {
  const size_t smem = router_smem_bytes(p.E, p.rows);
  static_assert(kMaxTopK <= 32, "one lane per selected expert");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_eg, p.S, 1);
  cfg.blockDim = dim3(kRouterThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = (unsigned)p.S;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  const int nrb = (p.rows + kRowBlock - 1) / kRowBlock;
  cfg.numAttrs = p.cluster_sum ? 2 : 1;
  // the tensor-core dot products beyond one block of rows, and for one block
  // when the experts kernel routes (then summed in a cluster as well)
  const bool mma = (nrb > 1 || p.route_in_experts) && router_mma_fits(p);
  if (p.cluster_sum && (nrb != 1 || p.S > 8 || (!mma && p.EG != kRouterWarps))) return cudaErrorInvalidValue;
  if (mma) cfg.gridDim = dim3((p.E + 15) / 16, p.S, 1);
  cudaError_t e = mma ? cudaLaunchKernelEx(&cfg, router_mma_kernel, p) : cudaLaunchKernelEx(&cfg, router_kernel, p);
  if (e != cudaSuccess || nrb == 1 || p.route_in_experts) return e;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(nrb, 1, 1);
  return cudaLaunchKernelEx(&cfg, route_kernel, p);
}

cudaError_t router_set_smem(size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  return e;
}

}  // namespace moe
