// Split-K weight streaming for projections of a few rows: out[l][i][r] =
// sum_k W[l][r][k] * X[l][i][k] for bf16 W [L][R][K] and X [L][n][K], n <= 8
// (one MMA N-tile), as fp32 partial sums per K-split, part [S][L][n][R].  The
// caller sums the S partials in split order (deterministic) in its epilogue.
//
// At a few rows the projection is bound by streaming W from HBM: it must keep
// enough bytes in flight on every SM to cover the loaded DRAM latency, not
// feed the tensor pipe.  Each warp owns one task (a layer, 32 weight rows,
// one K-split) and streams it in steps of 128 columns: 8 KB per step, each
// thread copying sixteen 16-byte pieces (four 32-column blocks of rows g and
// g + 8 of two m-tiles) with cp.async into a ring of shared-memory slots of
// its own, two steps deep, so up to 16 KB per warp and 192 KB per SM are in
// flight without holding registers.  A thread reads back only the pieces it
// copied, so the ring needs no barrier and no swizzle.  The bf16 products go
// through mma.sync m16n8k16 with fp32 accumulation; the MMA sums its 16
// K-slots in any order, so the K order is permuted to make each thread's
// weights one contiguous 16-byte run per row and block (columns 8t..8t+7:
// the first four feed one MMA, the last four the next) and X is read with
// the same permutation.  Tasks are interleaved over CTAs so every SM gets the
// same share; one CTA of 12 warps per SM.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace moe {

struct GemvParams {
  const __nv_bfloat16* W;  // [L][R][K]
  const __nv_bfloat16* X;  // [L][n][K]
  float* part;             // [S][L][n][R] (not gated)
  int L, R, K, n, S, KC;   // KC = K / S, a multiple of 128; R a multiple of 32
  // Gated (a gate/up projection, R = 2I, S = 1): a task takes 16 gate rows
  // j0.. and the matching 16 up rows I + j0.. as its two m-tiles and writes
  // gu = bf16 of both and act = bf16(silu(gate) * up) instead of partials.
  int I;
  __nv_bfloat16* gu;   // [n][2I]
  __nv_bfloat16* act;  // [n][I]
  // Completion counters (not gated; null: none).  Once a task's partials are
  // stored, done[l * (done_mod / done_div) + (row0 % done_mod) / done_div] is
  // incremented after a fence, so that a consumer can start on a group of
  // rows as soon as all of its tasks have finished.  With counters the
  // dependent grid is let launch only after this grid's dependency wait (so
  // that it never sees the counters before the predecessor has reset them).
  unsigned* done;
  int done_mod, done_div;
};

constexpr int kGemvWarps = 12;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvRows = 32;    // weight rows per task (two m-tiles)
constexpr int kGemvCols = 128;   // columns per step (four 32-column blocks)
constexpr int kGemvStages = 2;   // steps in flight per warp
constexpr int kGemvPieces = 16;  // 16-byte pieces per thread per step
constexpr size_t kGemvSmem = (size_t)kGemvWarps * kGemvStages * kGemvPieces * 32 * 16;

__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16 bytes global -> shared, bypassing L1, with 256-byte L2 fetches.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <bool kGated>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_bf16_kernel(GemvParams p) {
  extern __shared__ uint4 gemv_ring[];
  // the dependents (the epilogue kernel) may launch now and wait for this grid
  if (!p.done) grid_dep_launch();
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int warp = threadIdx.x >> 5;
  const int wid = warp * (int)gridDim.x + (int)blockIdx.x;
  const int n_warps = kGemvWarps * (int)gridDim.x;
  const int groups = kGated ? p.I / 16 : p.R / kGemvRows;
  const int tasks = p.L * groups * p.S;
  // rows of m-tile 1 relative to m-tile 0: the next 16 rows, or the up rows
  const int mt1 = kGated ? p.I : 16;
  // this thread's pieces: slot st, piece j at ring[((warp * stages + st) * 16 + j) * 32 + lane]
  uint4* mine = gemv_ring + (size_t)warp * kGemvStages * kGemvPieces * 32 + lane;
  const uint32_t mine_s = smem_u32(mine);
  bool waited = false;
  for (int task = wid; task < tasks; task += n_warps) {
    const int s = task % p.S;
    const int mg = (task / p.S) % groups;
    const int l = task / (p.S * groups);
    const int row0 = kGated ? mg * 16 : mg * kGemvRows;
    const __nv_bfloat16* w0 = p.W + ((size_t)l * p.R + row0 + g) * p.K + (size_t)s * p.KC + t * 8;
    const __nv_bfloat16* x0 = p.X + ((size_t)l * p.n + g) * p.K + (size_t)s * p.KC + t * 8;
    const int steps = p.KC / kGemvCols;
    // piece j: m-tile j >> 3, row g + 8 * ((j >> 2) & 1), 32-column block j & 3
    auto issue = [&](int it) {
      if (it < steps) {
        const uint32_t slot = mine_s + (uint32_t)((it % kGemvStages) * kGemvPieces * 32 * 16);
#pragma unroll
        for (int j = 0; j < kGemvPieces; ++j)
          cp_async16(slot + j * 32 * 16,
                     w0 + (size_t)((j >> 3) * mt1 + ((j >> 2) & 1) * 8) * p.K + it * kGemvCols + (j & 3) * 32);
      }
      cp_async_commit();  // one group per step, empty past the end
    };
#pragma unroll
    for (int it = 0; it < kGemvStages; ++it) issue(it);
    // the weights do not depend on the previous kernel; X does
    if (!waited) {
      grid_dep_wait();
      if (p.done) grid_dep_launch();
      waited = true;
    }
    auto load_x = [&](int it, uint4 (&b)[4]) {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        b[c] = g < p.n ? __ldg(reinterpret_cast<const uint4*>(x0 + it * kGemvCols + c * 32))
                       : make_uint4(0u, 0u, 0u, 0u);
    };
    float acc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mt][j] = 0.0f;
    uint4 b_next[4];
    load_x(0, b_next);
    for (int it = 0; it < steps; ++it) {
      uint4 b[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) b[c] = b_next[c];
      if (it + 1 < steps) load_x(it + 1, b_next);
      cp_async_wait<kGemvStages - 1>();  // this step's group has landed
      const uint4* slot = mine + (size_t)(it % kGemvStages) * kGemvPieces * 32;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 a[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) a[mt][hr] = slot[(mt * 8 + hr * 4 + c) * 32];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma_16816_bf16(acc[mt], a[mt][0].x, a[mt][1].x, a[mt][0].y, a[mt][1].y, b[c].x, b[c].y);
          mma_16816_bf16(acc[mt], a[mt][0].z, a[mt][1].z, a[mt][0].w, a[mt][1].w, b[c].z, b[c].w);
        }
      }
      // the slot's pieces are in registers (consumed by the MMAs): refill it
      issue(it + kGemvStages);
    }
    cp_async_wait<0>();
    if (kGated) {
      // row j of the gate and of the up projection, context row i
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = row0 + g + (q >> 1) * 8;
        const int i = 2 * t + (q & 1);
        if (i < p.n) {
          const __nv_bfloat16 gb = __float2bfloat16_rn(acc[0][q]), ub = __float2bfloat16_rn(acc[1][q]);
          p.gu[(size_t)i * 2 * p.I + j] = gb;
          p.gu[(size_t)i * 2 * p.I + p.I + j] = ub;
          const float gv = __bfloat162float(gb), uv = __bfloat162float(ub);
          p.act[(size_t)i * p.I + j] = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * uv);
        }
      }
    } else {
      float* out = p.part + ((size_t)s * p.L + l) * p.n * p.R + mg * kGemvRows;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int row = mt * 16 + g + (q >> 1) * 8;
          const int i = 2 * t + (q & 1);
          if (i < p.n) out[(size_t)i * p.R + row] = acc[mt][q];
        }
      if (p.done) {
        __threadfence();
        __syncwarp();
        if (lane == 0)
          atomicAdd(p.done + (size_t)l * (p.done_mod / p.done_div) + (row0 % p.done_mod) / p.done_div, 1u);
      }
    }
  }
}

// Splits of K for L * (R / 32) row groups over num_sms CTAs of 12 warps.  The
// time is set by the busiest SM's bytes, ceil(tasks / num_sms) * K / S, as
// long as each SM has at least 8 busy warps to cover the load latency; among
// split counts within 3 % of the best, the fewest (the epilogue sums S
// partials).  K / S stays a multiple of 128.  0 if K is not a multiple of
// 128 or R of 32.
inline int gemv_splits(int L, int R, int K, int num_sms) {
  if (K % kGemvCols || R % kGemvRows) return 0;
  const long long groups = (long long)L * (R / kGemvRows);
  long long best = 0;
  for (int pass = 0; pass < 2 && !best; ++pass)
    for (int s = 1; s <= 32; ++s) {
      if (K % (kGemvCols * s)) continue;
      const long long tasks = groups * s;
      if (pass == 0 && tasks < 8LL * num_sms) continue;
      const long long cost = ((tasks + num_sms - 1) / num_sms) * (K / s);
      if (!best || cost < best) best = cost;
    }
  for (int pass = 0; pass < 2; ++pass)
    for (int s = 1; s <= 32; ++s) {
      if (K % (kGemvCols * s)) continue;
      const long long tasks = groups * s;
      if (pass == 0 && tasks < 8LL * num_sms) continue;
      const long long cost = ((tasks + num_sms - 1) / num_sms) * (K / s);
      if (cost * 100 <= best * 103) return s;
    }
  return 0;
}

}  // namespace moe
