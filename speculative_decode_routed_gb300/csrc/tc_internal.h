// Internal interfaces of the tensor-core (tcgen05) expert path.
#pragma once
#include <cuda.h>

#include "moe_decode_internal.h"

namespace moe {

struct TcParams {
  int mode;                 // kGateUp or kDown
  int H, I, E, k;
  int K;                    // reduction length (H or I)
  int KBLK;                 // 256-wide K-blocks (the last may be half: zero filled)
  int KPS;                  // K-blocks per pipeline stage (1, or 2 when rows are whole K-blocks)
  int KSTEPS;               // stages per item: ceil(KBLK / KPS)
  int tiles;                // 128-row output tiles per expert (I/128 or H/128)
  int RE;                   // weight rows per expert (2I or H)
  int row_tiles;            // RE / 128
  int nt_max;               // 32-row activation tiles per MMA group (max pairs / 32)
  int NS;                   // pipeline stages
  int T;                    // accumulator types: 2 (gate, up) or 1 (down)
  int Q;                    // K phases: issuer q takes the K-blocks kb = q (mod Q)
  int P;                    // MMA issuer warps = T * Q, each with its own accumulators
  int dbuf;                 // accumulator buffers per issuer (2: epilogue overlaps)
  int sfslots;              // TMEM scale slots per issuer
  uint32_t acc_cols;        // TMEM columns of one accumulator (32 per N-tile)
  uint32_t sf_cols;         // TMEM columns of one scale slot (A: 16, B: 16 per N-tile)
  uint32_t issuer_cols;     // TMEM columns per issuer
  uint32_t stage_stride;    // bytes per stage (multiple of 1024)
  uint32_t a_bytes;         // weight tile bytes per stage (16 or 32 KB)
  uint32_t sfa_bytes;       // weight scale atoms per stage (2 or 4 KB)
  uint32_t off_sfa, off_b, off_sfb;  // offsets within a stage
  int ws_pairs;             // rows * k of the workspace
  int direct;               // gate/up: B is the MoE input's rows themselves (rows <= 32), not
                            // its pooled copy; each pair reads the accumulator column of its row
  int tiled;                // 1: the weight map is over tiled codes (the caller's or the
                            //    handle's copy), [E * row_tiles * KBLK][128 rows][128 B], each
                            //    box contiguous
  int withhold_ready;       // self-test of the bounded waits: completed experts are not
                            // published to the down phase, whose waits then all run out
  int local_route;          // 1 (at most 8 rows): every CTA routes the rows from the router's
                            // logits and pools their pairs in shared memory
  int rows;                 // rows of the step (local routing)
  const uint8_t* sfa;       // weight scale atoms [E][row_tiles][KBLK][2048]
  const float* gscale;      // [E][3]
  Workspace ws;
};

struct PoolParams {
  int H, k, rows;
  int ws_pairs;             // rows * k of the workspace (line stride)
  Workspace ws;
};

// Gate/up and down of one layer in one persistent launch (maps: weights,
// activation codes, activation scale lines of each projection).
cudaError_t launch_tc_moe(const TcParams& gu, const CUtensorMap& gu_a, const CUtensorMap& gu_b,
                          const CUtensorMap& gu_sfb, const TcParams& dn, const CUtensorMap& dn_a,
                          const CUtensorMap& dn_b, const CUtensorMap& dn_sfb, int grid,
                          cudaStream_t s, bool pdl);
size_t tc_moe_smem_bytes(const TcParams& gu, const TcParams& dn);
// Codes [rows][inner bytes] (rows a multiple of 128) into tiles
// [rows / 128][ceil(inner / 128)][128][128 B], the missing part of a last
// partial K-block zero.
cudaError_t launch_tile_codes(const uint8_t* src, int64_t rows, int inner, uint8_t* dst, cudaStream_t s);
cudaError_t launch_pool_gather(const PoolParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_sf_atoms(const uint8_t* sf, int64_t rows, int ks, int kblk, uint8_t* out,
                            cudaStream_t s);
cudaError_t tc_set_smem(size_t bytes);  // the fused kernel's dynamic shared memory
size_t tc_smem_bytes(const TcParams& p);
size_t tc_ctrl_bytes();

}  // namespace moe
