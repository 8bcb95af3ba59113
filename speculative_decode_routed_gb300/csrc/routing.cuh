// Softmax top-k routing of one row, shared by the router's routing tail and
// the experts kernel's in-kernel routing (every CTA routes the step's rows
// itself when there are at most 8 of them).
//
// Page: vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode,
// module docstring "One step of b rows", MoE: "router -> routing -> pooler".
// Routing is softmax over all experts, top-k by probability (ties to the
// lower expert id), gates renormalised over the selected k; a row is flagged
// when the k-th and (k+1)-th probabilities are less than 1e-6 apart.
#pragma once
#include "common.cuh"

namespace moe {

// One row's routing: the router's split-K partial logits in, the selection
// out.  Global outputs may be null (the experts kernel's CTAs other than the
// first write only the shared-memory ids).
struct RouteRow {
  const float* part;     // [S][rows][E] partial logits, summed in slice order
  int S, rows, E, k;
  const float* bias;     // [E] or null
  float* logits;         // [rows][E] or null
  int* ids;              // [rows][k] or null
  float* gates;          // [rows][k] or null
  uint8_t* flags;        // [rows] or null
  unsigned* err;         // latched error word
  int* sids;             // [rows][k] shared memory: the ids for the pooler
};

// Comparator of the routing order: higher logit first, ties to the lower id.
__device__ __forceinline__ bool route_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Shared tail of one row's routing (lane t < nsel holds the t-th selection):
// renormalised gates in slot order, the near-tie flag, ids to global and to
// shared memory for the pooler.
__device__ __forceinline__ void route_finish(const RouteRow& p, int r, int nsel, int sel_id,
                                             float sel_v, float m, float z) {
  const int k = p.k, lane = threadIdx.x & 31;
  const float ex = (lane < nsel) ? expf(sel_v - m) : 0.0f;
  float den = 0.0f;
  for (int t = 0; t < k; ++t) den += __shfl_sync(0xffffffffu, ex, t);
  const float ek = __shfl_sync(0xffffffffu, ex, k - 1);
  const float ek1 = __shfl_sync(0xffffffffu, ex, (nsel > k) ? k : 0);
  if (lane < k) {
    if (p.ids) p.ids[r * k + lane] = sel_id;
    p.sids[r * k + lane] = sel_id;
    if (p.gates) p.gates[r * k + lane] = ex / den;
    if (sel_id < 0 || sel_id >= p.E) latch_error(p.err, kDevBadRouting);
  }
  if (lane == 0 && p.flags) p.flags[r] = (nsel > k) ? (uint8_t)((ek - ek1) / z < 1e-6f) : (uint8_t)0;
}

// Order-preserving 32-bit keys of fp32 logits (larger logit, larger key);
// -0 is keyed as +0 so that equal logits tie.  Key 0 is below every logit.
__device__ __forceinline__ uint32_t logit_key(float f) {
  const uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One row's routing for E <= 256: lane owns experts e = lane + 32 i (i < 8),
// their logits in registers.  The slices' partial sums are all loaded at
// once and added in slice order.  Each lane sorts its 8 keys once; each of
// the k + 1 selections is then two warp reductions: the largest key among
// the lanes' heads (redux.sync max), then the lowest expert id among the
// lanes whose head has that key (redux.sync min), so ties go to the lower
// id; the winning lane shifts its sorted keys to the next.
__device__ inline void route_row_small(const RouteRow& p, int r) {
  const int E = p.E, k = p.k, rows = p.rows, lane = threadIdx.x & 31;
  float v[8];
  float part[8][8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const float* src = p.part + ((size_t)s * rows + r) * E;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      part[s][i] = (s < p.S && e < E) ? __ldcg(src + e) : 0.0f;
    }
  }
  uint32_t key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    float acc = 0.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < p.S) acc += part[s][i];
    if (e < E) {
      if (p.bias) acc += __ldg(p.bias + e);
      if (p.logits) p.logits[(size_t)r * E + e] = acc;
    }
    v[i] = acc;
    key[i] = (e < E) ? logit_key(acc) : 0u;
  }
  uint32_t lk = key[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) lk = max(lk, key[i]);
  const float m = key_logit(__reduce_max_sync(0xffffffffu, lk));
  float z = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (lane + 32 * i < E) z += expf(v[i] - m);
  z = warp_sum(z);
  // the lane's 8 keys sorted (largest first, ties to the lower expert id) by
  // a 19-comparator odd-even merge network; the head is then the lane's best
  uint32_t sk[8];
  int si[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    sk[i] = key[i];
    si[i] = i;
  }
  constexpr int kNet[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6},
                               {5, 7}, {1, 2}, {5, 6}, {0, 4}, {1, 5}, {2, 6}, {3, 7},
                               {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
  for (int c = 0; c < 19; ++c) {
    const int a = kNet[c][0], b = kNet[c][1];
    const bool keep = sk[a] > sk[b] || (sk[a] == sk[b] && si[a] < si[b]);
    const uint32_t ka = sk[a], kb = sk[b];
    const int ia = si[a], ib = si[b];
    sk[a] = keep ? ka : kb;
    sk[b] = keep ? kb : ka;
    si[a] = keep ? ia : ib;
    si[b] = keep ? ib : ia;
  }
  const int nsel = (k < E) ? k + 1 : k;
  int sel_id = -1;
  float sel_v = 0.0f;
  for (int t = 0; t < nsel; ++t) {
    // the largest head key, then the lowest expert id among the lanes whose
    // head has it; the winning lane moves on to its next key
    const uint32_t gk = __reduce_max_sync(0xffffffffu, sk[0]);
    const uint32_t gid =
        __reduce_min_sync(0xffffffffu, sk[0] == gk ? (uint32_t)(lane + 32 * si[0]) : 0xffffffffu);
    if (lane == t) {
      sel_id = (int)gid;
      sel_v = key_logit(gk);
    }
    if (lane == (int)(gid & 31u)) {
#pragma unroll
      for (int i = 0; i < 7; ++i) {
        sk[i] = sk[i + 1];
        si[i] = si[i + 1];
      }
      sk[7] = 0u;
    }
  }
  route_finish(p, r, nsel, sel_id, sel_v, m, z);
}

// One row's routing for any E (up to 1024): logits staged in shared memory,
// each selection a scan of the lane's experts and a warp arg-max.
__device__ inline void route_row_any(const RouteRow& p, int r, float* l) {
  const int E = p.E, k = p.k, rows = p.rows, lane = threadIdx.x & 31;
  float m = -INFINITY;
  // the lane's experts e = lane + 32 i, in groups of 8 so that the loads of
  // a slice are all in flight together; slices are summed in order
  for (int i0 = 0; i0 * 32 < E; i0 += 8) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    for (int s = 0; s < p.S; ++s) {
      const float* src = p.part + ((size_t)s * rows + r) * E;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * (i0 + i);
        if (e < E) v[i] += __ldcg(src + e);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * (i0 + i);
      if (e < E) {
        const float vb = p.bias ? v[i] + __ldg(p.bias + e) : v[i];
        l[e] = vb;
        if (p.logits) p.logits[(size_t)r * E + e] = vb;
        m = fmaxf(m, vb);
      }
    }
  }
  m = warp_max(m);
  float z = 0.0f;
  for (int e = lane; e < E; e += 32) z += expf(l[e] - m);
  z = warp_sum(z);
  __syncwarp();
  // top-(k+1) by logit (monotone in probability), ties to the lower id
  const int nsel = (k < E) ? k + 1 : k;
  int sel_id = -1;      // lane t keeps the t-th selection
  float sel_v = 0.0f;
  for (int t = 0; t < nsel; ++t) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = l[e];
      if (route_before(v, e, bv, bi)) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (route_before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == t) {
      sel_id = bi;
      sel_v = bv;
    }
    __syncwarp();
    if (lane == 0) l[bi] = -INFINITY;  // taken
    __syncwarp();
  }
  route_finish(p, r, nsel, sel_id, sel_v, m, z);
  __syncwarp();
}

// One row's routing, by the number of experts (lg: [E] shared-memory scratch
// of this warp, used above 256 experts).
__device__ __forceinline__ void route_row(const RouteRow& p, int r, float* lg) {
  if (p.E <= 256)
    route_row_small(p, r);
  else
    route_row_any(p, r, lg);
}


}  // namespace moe
