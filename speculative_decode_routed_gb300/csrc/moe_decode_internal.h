// Internal interfaces of the routed NVFP4 MoE decode library: the device
// workspace layout and the parameter blocks of its kernels.  Not part of the
// public C ABI (include/moe_decode.h).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <vector>

namespace moe {

// Pairs of one virtual expert: an active expert's pooled pairs in groups of
// at most this many, so that one 32-wide MMA N-tile covers each work item.
constexpr int kVirtualPairs = 32;

__host__ __device__ inline int virtual_slots(int E, int max_pairs) {
  return E + max_pairs / kVirtualPairs + 1;
}

// One expert's routing summary in a word: 1 + (expert | first pooled
// position << 10 | pairs << 22); 0 means "not published".  Experts < 1024,
// pooled positions < 4096, pairs < 256.
__host__ __device__ inline unsigned pack_expert(int e, int pos0, int ne) {
  return 1u + ((unsigned)e | ((unsigned)pos0 << 10) | ((unsigned)ne << 22));
}

// Device-side error codes latched into the workspace error word.
enum DeviceError : unsigned {
  kDevOk = 0,
  kDevWaitTimeout = 1,    // a bounded mbarrier wait gave up
  kDevBadRouting = 2,     // routing produced an out-of-range id / count
  kDevBadIndex = 3,       // bounds-check builds: a data-dependent index out of range (skipped)
  kDevCanary = 4,         // a workspace guard word changed (a write past a region's end)
};

// Library-owned scratch, sized at create for max_rows rows.
struct Workspace {
  __nv_bfloat16* x;      // [R][H]      MoE input (bf16)
  uint8_t* x_codes;      // [R][H/2]    NVFP4 codes of x (one tensor)
  uint8_t* x_sf;         // [R][H/16]   e4m3 block scales of x
  float* x_sg;           // [1]         global scale of x
  unsigned* x_amax;      // [1]         max |x| (float bits), reset by the router
  float* logit_part;     // [S][R][E]   router partial sums per H-slice
  float* logits;         // [R][E]      router logits (bias included)
  int* ids;              // [R][k]      expert of each (row, slot)
  float* gates;          // [R][k]      renormalised gates
  uint8_t* flags;        // [R]         1 if the k-th / (k+1)-th gap < 1e-6
  int* count;            // [E]         pairs per expert
  int* offset;           // [E+1]       exclusive prefix of count
  int* pair_order;       // [R*k]       pair id (r*k+s) at each pooled position
  int* pos_of_pair;      // [R*k]       pooled position of each pair id
  int* active;           // [E]         experts with pairs, ascending
  int* n_active;         // [1]
  float* h;              // [R*k][I]    silu(G)*U, pooled order
  unsigned* h_amax;      // [E]         per-expert max |h| (float bits)
  float* h_sg;           // [E]         per-expert global scale of h
  uint8_t* h_codes;      // [R*k][I/2]
  uint8_t* h_sf;         // [R*k][I/16]
  unsigned* done;        // [E]         finished gate/up tiles per expert
  float* o;              // [R*k][H]    expert outputs, pair-id order
  uint8_t* x_pool;       // [R*k][H/2]  MoE input codes in pooled order (tensor-core B operand)
  uint8_t* x_lines;      // [H/64][R*k][16]  its scales, one 16-byte line per MMA of 64 and row
                         //             (router; rows <= 32) or pooled position (pooler gather)
  uint8_t* h_lines;      // [I/64][R*k][16]  the same lines for h
  unsigned* act_info;    // [V]         per virtual expert (an active expert's pairs in groups of
                         //             at most 32): packed (expert, first pooled position, pairs)
  unsigned* ready_info;  // [V]         the same words in the order experts' h became ready (0: not yet)
  int* n_virtual;        // [1]         virtual experts of the step (V = E + rows*k/32 + 1 slots)
  unsigned* rg_count;    // [16]        router CTA arrivals per block of 8 rows
  unsigned* counters;    // [8]         [0] router row blocks routed, [1] gate/up item claims,
                         //             [2] down item claims, [3] experts ready, [4..7] unused
  unsigned* err;         // [1]         latched DeviceError; [1]: the first changed guard's index
  unsigned long long wait_ns;  // limit of every bounded wait in the kernels (a value, not a pointer)
};

// Default of Workspace::wait_ns.
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s

// ----------------------------------------------------------- boundary (K1)
struct BoundaryParams {
  int H, k, rows;
  int cols_per_cta;             // H / cluster size
  float eps;
  const __nv_bfloat16* branch;  // [rows][H] or null: gather sum_s g * o instead
  const float* o;               // [rows*k][H]
  const float* gates;           // [rows][k]
  float* stream;                // [rows][H] in/out
  const float* stream_in;       // [rows][H] read instead of stream when set (stream is still written)
  const float* w_post;          // [H]
  const float* w_pre;           // [H]
  __nv_bfloat16* x_out;         // [rows][H]
  unsigned* x_amax;             // max |x| accumulator, or null (final boundary)
  int front;                    // 1: the first layer's front -- the stream is the branch (the
                                //    embedded tokens) itself, one norm (w_pre) into x_out
  float* aux;                   // [rows][H] copy of the updated stream, or null
  unsigned* reset0;             // words zeroed once the kernel before has finished (the experts
  int n_reset0;                 //   kernel's counters and ready list when it routes itself), or
  unsigned* reset1;             //   null
  int n_reset1;
  int round_norm;               // 1: the second norm reads the stream rounded to bf16
                                // (x_out may be null: no normalised output)
  const float* part;            // [part_S][rows][H] fp32 split-K partials of a bf16 branch,
  int part_S;                   //   summed in split order and rounded to bf16 (when branch
  __nv_bfloat16* part_out;      //   is null); the rounded branch also to part_out if set
};

// ------------------------------------------------------------- router (K2)
struct RouterParams {
  int H, E, k, rows;
  int S;                        // H slices (split-K)
  int EG;                       // experts per CTA (one warp each)
  int n_eg;                     // expert groups: ceil(E / EG)
  const __nv_bfloat16* x;       // [rows][H]
  const __nv_bfloat16* wr;      // [E][H]
  const float* bias;            // [E] or null
  int line_rows;                // row stride of the scale lines (max_rows * k)
  int cluster_sum;              // 1 (at most 8 rows): the S slice CTAs of an expert group form a
                                // cluster whose first CTA sums their partials in slice order, then
                                // adds the bias, into logit_part's first slice (the logits), so
                                // routing reads one slice and no bias
  int route_in_experts;         // 1 (at most 8 rows, tensor-core experts): the experts kernel
                                // routes the rows and pools the pairs itself; the router only
                                // writes the logits and the MoE input's quantization
  Workspace ws;
};

// ------------------------------------------------------ experts (K3 / K4)
enum ExpertMode : int { kGateUp = 0, kDown = 1 };

struct ExpertParams {
  int mode;
  int H, I, E, k;
  int K, KB, KS;                // reduction length, code / scale bytes per weight row
  int T;                        // weight rows per item (gate/up: TJ gate + TJ up)
  int TJ;                       // gate/up: output columns per item; down: T
  int tiles;                    // items per expert
  int RE;                       // weight rows per expert (2I or H)
  int CH, TPG, G, TW;           // chunks/row, threads/row-group, row-groups, rows/thread
  int NS;                       // pipeline stages
  int ws_pairs;                 // rows * k of the workspace (bounds of pooled positions)
  uint32_t stage_bytes;         // bytes of one stage (codes + scales)
  uint32_t stage_stride;        // stage_bytes rounded up to 128
  const uint8_t* w;             // codes [E][RE][KB]
  const uint8_t* w_sf;          // scales [E][RE][KS]
  const float* gscale;          // [E][3]
  Workspace ws;
};

constexpr int kTWGateUp = 8;      // weight rows per thread per item (gate/up)
constexpr int kTWDown = 4;        // weight rows per thread per item (down)
constexpr int kMaxCTAThreads = 512;
constexpr int kSmemBudget = 226 * 1024;  // of the 227 KB a CTA may use

// Host-side launchers (one per kernel family).
// Cluster size of the boundary kernel for a row of H columns (H a multiple
// of 32): the largest cluster (<= 8) whose CTAs get whole 128-column slabs,
// unless that leaves a CTA more than 4096 columns (1024 threads of 4), then 8.
int boundary_cluster(int H);
cudaError_t launch_boundary(const BoundaryParams& p, int cluster, cudaStream_t s, bool pdl);
cudaError_t launch_router(const RouterParams& p, cudaStream_t s, bool pdl);
// Whether the tensor-core router's K-slices fit H (H a multiple of 256 S,
// slices at most 1024 wide).
bool router_mma_fits(const RouterParams& p);
cudaError_t launch_experts(const ExpertParams& p, int grid, cudaStream_t s, bool pdl);
cudaError_t launch_quantize(const float* v, int64_t rows, int64_t cols, uint8_t* codes,
                            uint8_t* sf, float* sg, float* amax, cudaStream_t s);
// The quantizer's encode pass alone, given the tensor's max |v| (float bits)
// in device memory.
cudaError_t launch_nvfp4_encode(const float* v, int64_t nblocks, uint8_t* codes, uint8_t* sf,
                                const unsigned* amax, float* sg, cudaStream_t s);
// Sets the calling thread's moe_decode_error_message; returns code.
int api_fail(int code, const char* msg);
// The address at which the current device may access page-locked host
// memory p (mapped into its address space), or null: the runtime reports
// none, p is not page-locked, or p is null.
void* host_mapped(const void* p);

size_t expert_smem_bytes(const ExpertParams& p);
size_t expert_ctrl_bytes();

// The library-owned graph caches (one per entry point that keeps graphs)
// hold at most kMaxCachedGraphs executables.  A lookup moves its hit to the
// back; an insert past the bound destroys the least recently used, which the
// runtime frees once it completes if it is still running.
constexpr size_t kMaxCachedGraphs = 32;

template <class Entry, class Match>
cudaGraphExec_t graph_cache_find(std::vector<Entry>& cache, Match match) {
  for (size_t i = 0; i < cache.size(); ++i)
    if (match(cache[i])) {
      const Entry hit = cache[i];
      cache.erase(cache.begin() + (std::ptrdiff_t)i);
      cache.push_back(hit);
      return hit.exec;
    }
  return nullptr;
}

template <class Entry>
void graph_cache_insert(std::vector<Entry>& cache, const Entry& entry) {
  if (cache.size() >= kMaxCachedGraphs) {
    cudaGraphExecDestroy(cache.front().exec);
    cache.erase(cache.begin());
  }
  cache.push_back(entry);
}

}  // namespace moe
