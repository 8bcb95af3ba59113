// C ABI of the routed NVFP4 MoE decode step: argument validation, the launch
// plan (tile sizes, pipeline depth, cluster shape), the workspace, the kernel
// sequence of a layer / step, and the library-owned CUDA graphs.
//
// Page: vllm.models.muse_spark.nvidia.specialized_decode.runtime (the
// deployment gate `unsupported`: the first reason a configuration cannot
// run, checked up front -- mirrored by moe_decode_create's validation and
// moe_decode_error_message) and ...runtime.decode (SpecializedDecode.run: per
// layer boundary.run -> attention -> attention_boundary.run -> moe.run, then
// final.run, replayed inside a FULL CUDA graph).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/moe_decode.h"
#include "common.cuh"
#include "moe_decode_internal.h"
#include "tc_internal.h"

// The expert path is chosen when the library is built: the tcgen05
// block-scaled tensor-core kernels by default, the CUDA-core kernels with
// -DMOE_EXPERT_FMA (kept for measurement against each other).
#ifndef MOE_EXPERT_FMA
#define MOE_EXPERT_TC 1
#else
#define MOE_EXPERT_TC 0
#endif

namespace moe {
size_t router_smem_bytes(int E, int rows);
cudaError_t router_set_smem(size_t bytes);
cudaError_t expert_set_smem(size_t bytes);
}  // namespace moe

namespace {

thread_local std::string g_msg;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_msg = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Page-locked (or registered) host memory, which a graph's copy nodes can
// move asynchronously.
bool host_pinned(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // pageable memory may report an error on older drivers
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}



// A guard of the workspace: 16 pattern bytes after a region (see Carver).
struct Guard {
  size_t offset;     // from the workspace base
  const char* name;  // the region it follows
};

struct GraphEntry {
  int rows;
  const void* branch;
  const float* stream;
  const void* out;
  cudaGraphExec_t exec;
};

}  // namespace

namespace moe {
// Records the reason of a failing call for moe_decode_error_message (entry
// points defined outside this file).
int api_fail(int code, const char* msg) { return fail(code, "%s", msg); }

void* host_mapped(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // pageable memory may report an error on older drivers
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}
}  // namespace moe

struct moe_decode_s {
  moe_decode_dims d;
  std::vector<moe_layer_weights> layers;
  const float* w_post_final = nullptr;
  const float* w_final = nullptr;
  int device = 0;
  int num_sms = 0;
  void* ws_mem = nullptr;
  size_t ws_bytes = 0;
  moe::Workspace ws{};
  int cluster = 1;
  int S = 1, EG = 8, n_eg = 1;
  moe::ExpertParams gu{}, dn{};
  cudaStream_t cap_stream = nullptr;
  std::vector<GraphEntry> graphs;
  std::vector<GraphEntry> host_graphs;  // copies in, step, copies out (pinned host buffers)
  uint16_t* io_branch = nullptr;
  float* io_stream = nullptr;
  uint16_t* io_out = nullptr;
  // tensor-core path
  moe::TcParams tgu{}, tdn{};
  std::vector<CUtensorMap> tm_w13, tm_w2;
  std::vector<uint8_t*> sfa13, sfa2;   // weight scale atoms per layer (library-owned)
  std::vector<uint8_t*> tiled13, tiled2;  // the expert codes in 16 KB tiles per layer (library-owned)
  std::vector<Guard> guards;           // the workspace's guards (offset, region)
  unsigned long long* guard_offsets = nullptr;  // device copy of their offsets
  bool tiled = false;                  // the weight maps are over tiles (the caller's or the copy)
  size_t copy_bytes = 0;               // rearranged weight copies held (scale atoms, tiled codes)
  CUtensorMap tm_xpool{}, tm_xcodes{}, tm_xlines{}, tm_hcodes{}, tm_hlines{};
};

namespace {

// Tile plan of one expert projection (see experts.cu).
int plan_experts(moe::ExpertParams& p, int mode, const moe_decode_dims& d) {
  p = moe::ExpertParams{};
  p.mode = mode;
  p.H = d.hidden;
  p.I = d.inter;
  p.E = d.n_experts;
  p.k = d.top_k;
  p.K = (mode == moe::kGateUp) ? d.hidden : d.inter;
  p.KB = p.K / 2;
  p.KS = p.K / 16;
  p.CH = p.K / 32;
  p.TPG = ((p.CH + 31) / 32) * 32;
  if (p.TPG > moe::kMaxCTAThreads) return fail(MOE_EUNSUPPORTED, "reduction length %d > 16384", p.K);
  p.TW = (mode == moe::kGateUp) ? moe::kTWGateUp : moe::kTWDown;
  // as many row-groups as fit in a CTA whose item still tiles the output
  p.G = 0;
  for (int g = moe::kMaxCTAThreads / p.TPG; g >= 1; --g) {
    const int T = p.TW * g;
    const bool fits = (mode == moe::kGateUp) ? (T % 2 == 0 && d.inter % (T / 2) == 0)
                                             : (d.hidden % T == 0);
    if (fits) {
      p.G = g;
      break;
    }
  }
  if (p.G == 0)
    return fail(MOE_EUNSUPPORTED, "no expert tile divides %s", mode == moe::kGateUp ? "inter" : "hidden");
  p.T = p.TW * p.G;
  if (mode == moe::kGateUp) {
    p.TJ = p.T / 2;
    p.tiles = d.inter / p.TJ;
    p.RE = 2 * d.inter;
  } else {
    p.TJ = p.T;
    p.tiles = d.hidden / p.T;
    p.RE = d.hidden;
  }
  p.stage_bytes = (uint32_t)(p.T * (p.KB + p.KS));
  p.stage_stride = (p.stage_bytes + 127u) / 128u * 128u;
  const size_t ctrl = moe::expert_ctrl_bytes();
  int ns = (int)((moe::kSmemBudget - ctrl) / p.stage_stride);
  if (ns > 16) ns = 16;
  if (ns < 2) return fail(MOE_EUNSUPPORTED, "expert stage of %u bytes too large", p.stage_bytes);
  p.NS = ns;
  p.ws_pairs = d.max_rows * d.top_k;
  return MOE_OK;
}

#if MOE_EXPERT_TC
// Tile plan of the tensor-core path (see experts_tc.cu).
int plan_tc(moe::TcParams& p, int mode, const moe_decode_dims& d) {
  p = moe::TcParams{};
  const bool gu = (mode == moe::kGateUp);
  p.mode = mode;
  p.H = d.hidden;
  p.I = d.inter;
  p.E = d.n_experts;
  p.k = d.top_k;
  p.K = gu ? d.hidden : d.inter;
  p.KBLK = (p.K + 255) / 256;
  p.tiles = gu ? d.inter / 128 : d.hidden / 128;
  p.RE = gu ? 2 * d.inter : d.hidden;
  p.row_tiles = p.RE / 128;
  // work items cover at most kVirtualPairs (32) pairs: one N-tile
  p.nt_max = 1;
  p.T = gu ? 2 : 1;
  p.acc_cols = 32u * (uint32_t)p.nt_max;
  // TMEM (512 columns): as many independent MMA issuers as fit, each with its
  // own accumulators and scale slots (issue latency, not the tensor core,
  // bounds one issuer; issuers overlap).  The single TMA-issuing thread costs
  // about the same per copy whatever its size, so down, whose weight tile per
  // K-block is half of gate/up's, moves two K-blocks per stage (one 3D copy
  // per operand) when its rows are whole K-blocks and TMEM still holds four
  // issuers.
  p.P = 0;
  const int qs_gu[2] = {2, 1}, qs_dn[3] = {4, 2, 1};
  const int* qs = gu ? qs_gu : qs_dn;
  const int nq = gu ? 2 : 3;
  const int kps_opts[2] = {2, 1};
  const int kps_first = (!gu && d.inter % 256 == 0) ? 0 : 1;
  const int modes[4][2] = {{2, 2}, {2, 1}, {1, 2}, {1, 1}};
  if (!gu && kps_first == 0 && (p.KBLK + 1) / 2 <= 3) {
    // down items of at most three stages (two K-blocks each): three issuers
    // with three accumulator buffers each, so that three items are in flight
    // between the MMAs and the epilogue (with two, a down item's epilogue
    // latency paced the phase, and a fourth issuer had no stage to take).
    // Measured: 8 chained layers of intermediate 1536, 133.2 against 134.4
    // µs per layer-step; with four stages per item (intermediate 2048) the
    // uneven split over three issuers cost 16 µs, so those keep four.
    const uint32_t sfc = 16u * 2u * (1u + (uint32_t)p.nt_max);
    const uint32_t cols = 3u * p.acc_cols + sfc;
    if (3u * cols <= 512u) {
      p.Q = 3;
      p.P = 3;
      p.KPS = 2;
      p.dbuf = 3;
      p.sfslots = 1;
      p.sf_cols = sfc;
      p.issuer_cols = cols;
    }
  }
  for (int qi = 0; qi < nq && !p.P; ++qi)
    for (int ki = kps_first; ki < 2 && !p.P; ++ki)
      for (int mi = 0; mi < 4 && !p.P; ++mi) {
        const int kps = kps_opts[ki];
        const uint32_t sfc = 16u * (uint32_t)kps * (1u + (uint32_t)p.nt_max);
        const uint32_t cols = (uint32_t)modes[mi][0] * p.acc_cols + (uint32_t)modes[mi][1] * sfc;
        const int P = p.T * qs[qi];
        if ((uint32_t)P * cols <= 512u) {
          p.Q = qs[qi];
          p.P = P;
          p.KPS = kps;
          p.dbuf = modes[mi][0];
          p.sfslots = modes[mi][1];
          p.sf_cols = sfc;
          p.issuer_cols = cols;
        }
      }
  if (!p.P) return fail(MOE_EUNSUPPORTED, "tensor-core plan does not fit TMEM (max_rows %d)", d.max_rows);
  p.KSTEPS = (p.KBLK + p.KPS - 1) / p.KPS;
  p.a_bytes = 16384u * (uint32_t)(p.KPS * p.T);
  p.sfa_bytes = 2048u * (uint32_t)(p.KPS * p.T);
  p.off_b = p.a_bytes;
  p.off_sfa = p.off_b + 4096u * (uint32_t)(p.KPS * p.nt_max);
  p.off_sfb = p.off_sfa + p.sfa_bytes;
  const uint32_t stage = p.off_sfb + 2048u * (uint32_t)(p.KPS * p.nt_max);
  p.stage_stride = (stage + 1023u) / 1024u * 1024u;
  int ns = (int)((227 * 1024 - 1024 - moe::tc_ctrl_bytes()) / p.stage_stride);
  if (ns > 8) ns = 8;
  if (ns < 2) return fail(MOE_EUNSUPPORTED, "tensor-core stage too large (max_rows %d)", d.max_rows);
  p.NS = ns;
  p.ws_pairs = d.max_rows * d.top_k;
  return MOE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Row-major bytes [rows][inner]: boxes of 128 bytes x box_rows, 128B swizzle.
int encode_rows(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(MOE_ECUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ECUDA, "tensor map encode failed (%d)", (int)r);
  return MOE_OK;
}

// Row-major bytes [rows][inner], inner a multiple of 128, viewed as
// [inner / 128 K-blocks][rows][128 B]: boxes of 128 bytes x box_rows x kblocks,
// landing as kblocks consecutive 128B-swizzled tiles.
int encode_rows_kb(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                   uint32_t box_rows, uint32_t kblocks) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(MOE_ECUDA, "cuTensorMapEncodeTiled is not available");
  if (inner % 128) return fail(MOE_EUNSUPPORTED, "rows of %llu bytes are not whole K-blocks",
                               (unsigned long long)inner);
  const cuuint64_t dims[3] = {128, rows, inner / 128};
  const cuuint64_t strides[2] = {inner, 128};
  const cuuint32_t box[3] = {128, box_rows, kblocks};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ECUDA, "tensor map encode failed (%d)", (int)r);
  return MOE_OK;
}

// Tiled codes [tiles][128 rows][128 B]: boxes of kblocks consecutive whole
// tiles, each one contiguous 16 KB read, landing 128B-swizzled.
int encode_tiles(CUtensorMap* m, const void* base, uint64_t tiles, uint32_t kblocks) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(MOE_ECUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {128, 128, tiles};
  const cuuint64_t strides[2] = {128, 16384};
  const cuuint32_t box[3] = {128, 128, kblocks};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ECUDA, "tensor map encode failed (%d)", (int)r);
  return MOE_OK;
}

// Scale lines [groups][rows][16 B]: boxes of 16 B x 32 rows x box_groups.
int encode_lines(CUtensorMap* m, const void* base, uint64_t rows, uint64_t groups,
                 uint32_t box_groups = 4) {
  auto enc = tensor_map_encoder();
  if (!enc) return fail(MOE_ECUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {16, rows, groups};
  const cuuint64_t strides[2] = {16, rows * 16};
  const cuuint32_t box[3] = {16, 32, box_groups};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ECUDA, "tensor map encode failed (%d)", (int)r);
  return MOE_OK;
}
#endif  // MOE_EXPERT_TC

int check_layer(const moe_layer_weights& w, int i) {
  if (!w.w_post || !w.w_pre || !w.router_w || !w.w13 || !w.w13_sf || !w.w2 || !w.w2_sf ||
      !w.w_gscale)
    return fail(MOE_EINVAL, "layer %d: a required weight pointer is NULL", i);
  const void* a16[] = {w.w_post, w.w_pre, w.router_w, w.w13, w.w13_sf, w.w2, w.w2_sf};
  for (const void* q : a16)
    if (!aligned(q, 16)) return fail(MOE_EINVAL, "layer %d: weight pointer not 16-byte aligned", i);
  if (!aligned(w.w_gscale, 4) || (w.router_bias && !aligned(w.router_bias, 4)))
    return fail(MOE_EINVAL, "layer %d: fp32 pointer not 4-byte aligned", i);
  return MOE_OK;
}

// Every region of the workspace is followed by a 256-byte guard whose first
// 16 bytes hold a pattern written at create; moe_decode_last_error checks
// them, so a kernel writing past a region's end is caught (a substitute for
// a memory sanitizer).
constexpr size_t kGuardBytes = 256;

// Region allocator over the workspace: 256-byte aligned regions, each followed
// by a guard (recorded when guards is given).
struct Carver {
  uint8_t* base;
  uint8_t* cur;
  std::vector<Guard>* guards;
  template <typename T>
  T* take(size_t count, const char* name) {
    T* p = reinterpret_cast<T*>(cur);
    cur += (count * sizeof(T) + 255) / 256 * 256;
    if (guards) guards->push_back(Guard{(size_t)(cur - base), name});
    cur += kGuardBytes;
    return p;
  }
};

__global__ void guard_kernel(uint8_t* base, const unsigned long long* offsets, int n, int check,
                             unsigned* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  uint4* g = reinterpret_cast<uint4*>(base + offsets[i]);
  const uint4 want = make_uint4(0xC0DE0000u ^ (unsigned)i, 0x5AFE0000u ^ (unsigned)i, ~(unsigned)i,
                                (unsigned)i * 2654435761u);
  if (!check) {
    *g = want;
    return;
  }
  const uint4 v = *g;
  if (v.x != want.x || v.y != want.y || v.z != want.z || v.w != want.w) {
    atomicCAS(err, 0u, (unsigned)moe::kDevCanary);
    atomicMin(err + 1, (unsigned)i);
  }
}

size_t layout_workspace(moe::Workspace& ws, uint8_t* base, const moe_decode_dims& d, int S,
                        std::vector<Guard>* guards = nullptr,
                        unsigned long long** guard_offsets = nullptr) {
  const size_t R = d.max_rows, H = d.hidden, E = d.n_experts, k = d.top_k, I = d.inter;
  Carver cv{base, base, guards};
  ws.x = cv.take<__nv_bfloat16>(R * H, "x");
  ws.x_codes = cv.take<uint8_t>(R * H / 2, "x_codes");
  ws.x_sf = cv.take<uint8_t>(R * H / 16, "x_sf");
  ws.x_sg = cv.take<float>(1, "x_sg");
  ws.x_amax = cv.take<unsigned>(1, "x_amax");
  ws.logit_part = cv.take<float>((size_t)S * R * E, "logit_part");
  ws.logits = cv.take<float>(R * E, "logits");
  ws.ids = cv.take<int>(R * k, "ids");
  ws.gates = cv.take<float>(R * k, "gates");
  ws.flags = cv.take<uint8_t>(R, "flags");
  ws.count = cv.take<int>(E, "count");
  ws.offset = cv.take<int>(E + 1, "offset");
  ws.pair_order = cv.take<int>(R * k, "pair_order");
  ws.pos_of_pair = cv.take<int>(R * k, "pos_of_pair");
  ws.active = cv.take<int>(E, "active");
  ws.n_active = cv.take<int>(1, "n_active");
  ws.h = cv.take<float>(R * k * I, "h");
  ws.h_amax = cv.take<unsigned>(E, "h_amax");
  ws.h_sg = cv.take<float>(E, "h_sg");
  ws.h_codes = cv.take<uint8_t>(R * k * I / 2, "h_codes");
  ws.h_sf = cv.take<uint8_t>(R * k * I / 16, "h_sf");
  ws.done = cv.take<unsigned>(E, "done");
  ws.o = cv.take<float>(R * k * H, "o");
  ws.x_pool = cv.take<uint8_t>(R * k * H / 2, "x_pool");
  ws.x_lines = cv.take<uint8_t>(R * k * (H / 64) * 16, "x_lines");
  ws.h_lines = cv.take<uint8_t>(R * k * (I / 64) * 16, "h_lines");
  const size_t V = (size_t)moe::virtual_slots((int)E, (int)(R * k));
  ws.act_info = cv.take<unsigned>(V, "act_info");
  ws.ready_info = cv.take<unsigned>(V, "ready_info");
  ws.n_virtual = cv.take<int>(1, "n_virtual");
  ws.rg_count = cv.take<unsigned>(16, "rg_count");
  ws.counters = cv.take<unsigned>(8, "counters");
  ws.err = cv.take<unsigned>(2, "err");
  // the guards' offsets, for the fill and check kernels (no guard after them)
  const size_t n_guards = guards ? guards->size() : 64;
  unsigned long long* offs = reinterpret_cast<unsigned long long*>(cv.cur);
  cv.cur += (n_guards * sizeof(unsigned long long) + 255) / 256 * 256;
  if (guard_offsets) *guard_offsets = offs;
  return (size_t)(cv.cur - base);
}

int check_rows(const moe_decode_t* h, int rows) {
  if (rows < 1 || rows > h->d.max_rows)
    return fail(MOE_EINVAL, "rows %d outside [1, max_rows=%d]", rows, h->d.max_rows);
  return MOE_OK;
}

int launch_layer(moe_decode_t* h, int layer, int rows, const uint16_t* branch, float* stream,
                 cudaStream_t s, cudaEvent_t* ev = nullptr, const float* stream_in = nullptr,
                 bool withhold_ready = false) {
  const bool pdl = (ev == nullptr);
  auto mark = [&](int i) {
    if (ev) cudaEventRecord(ev[i], s);
  };
  mark(0);
  const moe_decode_dims& d = h->d;
  const moe_layer_weights& w = h->layers[layer];
  moe::BoundaryParams bp{};
  bp.H = d.hidden;
  bp.k = d.top_k;
  bp.rows = rows;
  bp.cols_per_cta = d.hidden / h->cluster;
  bp.eps = d.eps;
  bp.branch = reinterpret_cast<const __nv_bfloat16*>(branch);
  bp.o = h->ws.o;
  bp.gates = h->ws.gates;
  bp.stream = stream;
  bp.stream_in = stream_in;
  bp.w_post = w.w_post;
  bp.w_pre = w.w_pre;
  bp.x_out = h->ws.x;
  bp.x_amax = h->ws.x_amax;
  // Up to 8 rows the tensor-core experts kernel routes and pools itself from
  // the router's logits.  Its item counters and ready list start at zero:
  // the boundary clears them once the previous experts kernel has finished.
  const bool local_route = MOE_EXPERT_TC && rows <= 8;
  if (local_route) {
    bp.reset0 = h->ws.counters;
    bp.n_reset0 = 8;
    bp.reset1 = h->ws.ready_info;
    bp.n_reset1 = moe::virtual_slots(d.n_experts, d.max_rows * d.top_k);
  }
  cudaError_t e = moe::launch_boundary(bp, h->cluster, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "boundary launch");
  mark(1);

  moe::RouterParams rp{};
  rp.H = d.hidden;
  rp.E = d.n_experts;
  rp.k = d.top_k;
  rp.rows = rows;
  rp.S = h->S;
  rp.EG = h->EG;
  rp.n_eg = h->n_eg;
  rp.x = h->ws.x;
  rp.wr = reinterpret_cast<const __nv_bfloat16*>(w.router_w);
  rp.bias = w.router_bias;
  rp.line_rows = d.max_rows * d.top_k;
  rp.route_in_experts = local_route ? 1 : 0;
  // one block of rows: the router's slice CTAs sum their partials in a
  // thread-block cluster (the tensor-core router's when the experts kernel
  // routes and H splits into its slices)
  rp.cluster_sum = rows <= 8 ? 1 : 0;
  rp.ws = h->ws;
  e = moe::launch_router(rp, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "router launch");
  mark(2);

#if MOE_EXPERT_TC
  // up to 32 rows the gate/up MMA's N holds the rows themselves: no pooled
  // copy of the MoE input is needed
  const bool direct = rows <= 32;
  if (!direct) {
    moe::PoolParams pp{};
    pp.H = d.hidden;
    pp.k = d.top_k;
    pp.rows = rows;
    pp.ws_pairs = d.max_rows * d.top_k;
    pp.ws = h->ws;
    e = moe::launch_pool_gather(pp, s, pdl);
    if (e != cudaSuccess) return cuda_fail(e, "pool launch");
  }
  mark(3);

  // gate/up and down in one persistent launch
  moe::TcParams tg = h->tgu;
  tg.sfa = h->sfa13[layer];
  tg.tiled = h->tiled;
  tg.gscale = w.w_gscale;
  tg.ws = h->ws;
  tg.direct = direct ? 1 : 0;
  moe::TcParams td = h->tdn;
  td.sfa = h->sfa2[layer];
  td.tiled = h->tiled;
  td.gscale = w.w_gscale;
  td.ws = h->ws;
  tg.withhold_ready = withhold_ready ? 1 : 0;
  tg.local_route = td.local_route = local_route ? 1 : 0;
  tg.rows = td.rows = rows;
  e = moe::launch_tc_moe(tg, h->tm_w13[layer], direct ? h->tm_xcodes : h->tm_xpool, h->tm_xlines,
                         td, h->tm_w2[layer],
                         h->tm_hcodes, h->tm_hlines, h->num_sms, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "experts launch");
  mark(4);
  mark(5);
  return MOE_OK;
#else
  mark(3);
  moe::ExpertParams gu = h->gu;
  gu.w = w.w13;
  gu.w_sf = w.w13_sf;
  gu.gscale = w.w_gscale;
  gu.ws = h->ws;
  e = moe::launch_experts(gu, h->num_sms, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "gate/up launch");
  mark(4);

  moe::ExpertParams dn = h->dn;
  dn.w = w.w2;
  dn.w_sf = w.w2_sf;
  dn.gscale = w.w_gscale;
  dn.ws = h->ws;
  e = moe::launch_experts(dn, h->num_sms, s, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "down launch");
  mark(5);
  return MOE_OK;
#endif
}

int launch_final(moe_decode_t* h, int rows, float* stream, uint16_t* out, cudaStream_t s,
                 float* aux = nullptr) {
  const moe_decode_dims& d = h->d;
  moe::BoundaryParams bp{};
  bp.H = d.hidden;
  bp.k = d.top_k;
  bp.rows = rows;
  bp.cols_per_cta = d.hidden / h->cluster;
  bp.eps = d.eps;
  bp.branch = nullptr;
  bp.o = h->ws.o;
  bp.gates = h->ws.gates;
  bp.stream = stream;
  bp.w_post = h->w_post_final;
  bp.w_pre = h->w_final;
  bp.x_out = reinterpret_cast<__nv_bfloat16*>(out);
  bp.x_amax = nullptr;
  bp.aux = aux;
  const cudaError_t e = moe::launch_boundary(bp, h->cluster, s, true);
  if (e != cudaSuccess) return cuda_fail(e, "final boundary launch");
  return MOE_OK;
}

int check_step_args(moe_decode_t* h, int rows, const void* branch, const float* stream,
                    const void* out) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!branch || !stream || !out) return fail(MOE_EINVAL, "branch, stream and out are required");
  if (!aligned(stream, 16) || !aligned(branch, 8) || !aligned(out, 8))
    return fail(MOE_EINVAL, "stream must be 16-byte, branch and out 8-byte aligned");
  if (!h->w_post_final || !h->w_final)
    return fail(MOE_EINVAL, "the handle was created without final norm weights");
  return MOE_OK;
}

// stream_in: where the first layer reads the stream (null: stream itself);
// aux: where the final boundary also writes the final stream (or null).
int enqueue_step(moe_decode_t* h, int rows, const uint16_t* branch, float* stream, uint16_t* out,
                 cudaStream_t s, const float* stream_in = nullptr, float* aux = nullptr) {
  for (int l = 0; l < h->d.n_layers; ++l) {
    const int rc = launch_layer(h, l, rows, l == 0 ? branch : nullptr, stream, s, nullptr,
                                l == 0 ? stream_in : nullptr);
    if (rc) return rc;
  }
  return launch_final(h, rows, stream, out, s, aux);
}

}  // namespace

extern "C" {

const char* moe_decode_error_message(void) { return g_msg.c_str(); }

const char* moe_decode_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument";
    case MOE_EUNSUPPORTED: return "unsupported shape or device";
    case MOE_ECUDA: return "CUDA runtime error";
    case MOE_ENOMEM: return "out of device memory";
    case MOE_EDEVICE: return "device-side check failed";
    default: return "unknown error";
  }
}

int moe_decode_create(const moe_decode_dims* dims, const moe_layer_weights* layers,
                      const float* w_post_final, const float* w_final, moe_decode_t** out) {
  g_msg.clear();
  if (!dims || !layers || !out) return fail(MOE_EINVAL, "dims, layers and out are required");
  *out = nullptr;
  const moe_decode_dims d = *dims;
  if (d.hidden < 128 || d.hidden % 128 || d.hidden > 8192)
    return fail(MOE_EUNSUPPORTED, "hidden %d: need a multiple of 128 in [128, 8192]", d.hidden);
  if (d.inter < 128 || d.inter % 128 || d.inter > 8192)
    return fail(MOE_EUNSUPPORTED, "inter %d: need a multiple of 128 in [128, 8192]", d.inter);
  if (d.n_experts < 1 || d.n_experts > 1024)
    return fail(MOE_EUNSUPPORTED, "n_experts %d outside [1, 1024]", d.n_experts);
  if (d.top_k < 1 || d.top_k > d.n_experts || d.top_k > 16)
    return fail(MOE_EUNSUPPORTED, "top_k %d outside [1, min(E, 16)]", d.top_k);
  if (d.max_rows < 1 || d.max_rows > 128)
    return fail(MOE_EUNSUPPORTED, "max_rows %d outside [1, 128]", d.max_rows);
  if (d.n_layers < 1 || d.n_layers > 256)
    return fail(MOE_EUNSUPPORTED, "n_layers %d outside [1, 256]", d.n_layers);
  if (!(d.eps >= 0.0f)) return fail(MOE_EINVAL, "eps must be >= 0");
  if (d.code_layout < MOE_CODES_ROW_MAJOR || d.code_layout > MOE_CODES_TILED_COPY)
    return fail(MOE_EINVAL, "code_layout %d is not a MOE_CODES_* value", d.code_layout);
  if (!MOE_EXPERT_TC && d.code_layout != MOE_CODES_ROW_MAJOR)
    return fail(MOE_EUNSUPPORTED, "the CUDA-core expert build reads row-major codes only");
  for (int i = 0; i < d.n_layers; ++i) {
    const int rc = check_layer(layers[i], i);
    if (rc) return rc;
  }
  if ((w_post_final && !aligned(w_post_final, 16)) || (w_final && !aligned(w_final, 16)))
    return fail(MOE_EINVAL, "final norm weights must be 16-byte aligned");

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major != 10)
    return fail(MOE_EUNSUPPORTED, "device %s is sm_%d%d; the library is built for the SM 10.x "
                "family (sm_103a)", prop.name, prop.major, prop.minor);

  moe_decode_t* h = new moe_decode_s();
  h->d = d;
  h->layers.assign(layers, layers + d.n_layers);
  h->w_post_final = w_post_final;
  h->w_final = w_final;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->cluster = moe::boundary_cluster(d.hidden);
  // router: one warp per expert, H split into slices of at most 1024
  h->EG = 8;
  h->n_eg = (d.n_experts + h->EG - 1) / h->EG;
  h->S = (d.hidden / 8 + 127) / 128;
  int rc = plan_experts(h->gu, moe::kGateUp, d);
  if (!rc) rc = plan_experts(h->dn, moe::kDown, d);
#if MOE_EXPERT_TC
  if (!rc) rc = plan_tc(h->tgu, moe::kGateUp, d);
  if (!rc) rc = plan_tc(h->tdn, moe::kDown, d);
#endif
  if (rc) {
    delete h;
    return rc;
  }
#if MOE_EXPERT_TC
  e = moe::tc_set_smem(moe::tc_moe_smem_bytes(h->tgu, h->tdn));
#else
  e = moe::expert_set_smem(std::max(moe::expert_smem_bytes(h->gu), moe::expert_smem_bytes(h->dn)));
#endif
  if (e == cudaSuccess) e = moe::router_set_smem(moe::router_smem_bytes(d.n_experts, d.max_rows));
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "kernel attribute");
  }
  moe::Workspace probe{};
  alignas(256) static uint8_t fake_base[256];  // sizes only: nothing is written through it
  h->ws_bytes = layout_workspace(probe, fake_base, d, h->S);
  e = cudaMalloc(&h->ws_mem, h->ws_bytes);
  if (e != cudaSuccess) {
    const size_t want = h->ws_bytes;
    delete h;
    return fail(MOE_ENOMEM, "workspace of %zu bytes: %s", want, cudaGetErrorString(e));
  }
  layout_workspace(h->ws, static_cast<uint8_t*>(h->ws_mem), d, h->S, &h->guards, &h->guard_offsets);
  h->ws.wait_ns = moe::kDefaultWaitNs;
  const size_t io = (size_t)d.max_rows * d.hidden;
  e = cudaMemset(h->ws_mem, 0, h->ws_bytes);
  // the guards: their offsets to the device, their patterns written, and the
  // error word's second slot (the first changed guard) set to "none"
  if (e == cudaSuccess) {
    std::vector<unsigned long long> offs;
    for (const Guard& g : h->guards) offs.push_back(g.offset);
    e = cudaMemcpy(h->guard_offsets, offs.data(), offs.size() * sizeof(unsigned long long),
                   cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMemset(h->ws.err + 1, 0xFF, sizeof(unsigned));
  if (e == cudaSuccess) {
    const int n = (int)h->guards.size();
    guard_kernel<<<(n + 127) / 128, 128>>>(static_cast<uint8_t*>(h->ws_mem), h->guard_offsets, n, 0,
                                           h->ws.err);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMalloc(&h->io_branch, io * 2);
  if (e == cudaSuccess) e = cudaMalloc(&h->io_stream, io * 4);
  if (e == cudaSuccess) e = cudaMalloc(&h->io_out, io * 2);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    moe_decode_destroy(h);
    return cuda_fail(e, "workspace setup");
  }
#if MOE_EXPERT_TC
  {
    const uint64_t R = (uint64_t)d.max_rows * d.top_k;
    const uint64_t H = d.hidden, I = d.inter, E = d.n_experts;
    rc = encode_rows(&h->tm_xpool, h->ws.x_pool, H / 2, R, 32);
    if (!rc) rc = encode_rows(&h->tm_xcodes, h->ws.x_codes, H / 2, (uint64_t)d.max_rows, 32);
    if (!rc) rc = encode_lines(&h->tm_xlines, h->ws.x_lines, R, H / 64);
    const uint32_t kps = (uint32_t)h->tdn.KPS;
    if (!rc) rc = kps == 1 ? encode_rows(&h->tm_hcodes, h->ws.h_codes, I / 2, R, 32)
                           : encode_rows_kb(&h->tm_hcodes, h->ws.h_codes, I / 2, R, 32, kps);
    if (!rc) rc = encode_lines(&h->tm_hlines, h->ws.h_lines, R, I / 64, 4 * kps);
    h->tm_w13.resize(d.n_layers);
    h->tm_w2.resize(d.n_layers);
    h->sfa13.assign(d.n_layers, nullptr);
    h->sfa2.assign(d.n_layers, nullptr);
    const uint64_t n13 = E * (uint64_t)h->tgu.row_tiles * h->tgu.KBLK;  // 16 KB tiles per layer
    const uint64_t n2 = E * (uint64_t)h->tdn.row_tiles * h->tdn.KBLK;
    for (int l = 0; l < d.n_layers && !rc; ++l) {
      const size_t b13 = (size_t)E * h->tgu.row_tiles * h->tgu.KBLK * 2048;
      const size_t b2 = (size_t)E * h->tdn.row_tiles * h->tdn.KBLK * 2048;
      if (!rc && cudaMalloc(&h->sfa13[l], b13) != cudaSuccess) rc = fail(MOE_ENOMEM, "scale atoms");
      if (!rc && cudaMalloc(&h->sfa2[l], b2) != cudaSuccess) rc = fail(MOE_ENOMEM, "scale atoms");
      if (!rc) h->copy_bytes += b13 + b2;
      if (!rc && moe::launch_sf_atoms(layers[l].w13_sf, (int64_t)E * 2 * I, (int)(H / 16),
                                      h->tgu.KBLK, h->sfa13[l], nullptr) != cudaSuccess)
        rc = fail(MOE_ECUDA, "scale atoms launch");
      if (!rc && moe::launch_sf_atoms(layers[l].w2_sf, (int64_t)E * H, (int)(I / 16), h->tdn.KBLK,
                                      h->sfa2[l], nullptr) != cudaSuccess)
        rc = fail(MOE_ECUDA, "scale atoms launch");
    }
    // The weight maps, by the layout of the codes.  Row-major codes are read
    // in place through 2D (or, two K-blocks per down stage, 3D) maps of
    // 128-byte x 128-row boxes; tiled codes -- the caller's, or the handle's
    // copy -- through 3D maps whose boxes are whole 16 KB tiles, each one
    // contiguous read.
    h->tiled = d.code_layout != MOE_CODES_ROW_MAJOR;
    if (!rc && d.code_layout == MOE_CODES_TILED_COPY) {
      h->tiled13.assign(d.n_layers, nullptr);
      h->tiled2.assign(d.n_layers, nullptr);
      for (int l = 0; l < d.n_layers && !rc; ++l) {
        if (cudaMalloc(&h->tiled13[l], n13 * 16384) != cudaSuccess ||
            cudaMalloc(&h->tiled2[l], n2 * 16384) != cudaSuccess) {
          cudaGetLastError();
          rc = fail(MOE_ENOMEM, "the tiled copy of layer %d's expert codes (%.2f GB): %s", l,
                    (double)(n13 + n2) * 16384.0 / 1e9,
                    "pass MOE_CODES_ROW_MAJOR, or tile the codes once (moe_tile_codes) and pass "
                    "MOE_CODES_TILED");
          break;
        }
        h->copy_bytes += (size_t)(n13 + n2) * 16384;
        if (moe::launch_tile_codes(static_cast<const uint8_t*>(layers[l].w13), (int64_t)E * 2 * I,
                                   (int)(H / 2), h->tiled13[l], nullptr) != cudaSuccess ||
            moe::launch_tile_codes(static_cast<const uint8_t*>(layers[l].w2), (int64_t)E * H,
                                   (int)(I / 2), h->tiled2[l], nullptr) != cudaSuccess)
          rc = fail(MOE_ECUDA, "code tiling launch");
      }
    }
    for (int l = 0; l < d.n_layers && !rc; ++l) {
      if (h->tiled) {
        const void* c13 = d.code_layout == MOE_CODES_TILED ? layers[l].w13 : h->tiled13[l];
        const void* c2 = d.code_layout == MOE_CODES_TILED ? layers[l].w2 : h->tiled2[l];
        rc = encode_tiles(&h->tm_w13[l], c13, n13, 1);
        if (!rc) rc = encode_tiles(&h->tm_w2[l], c2, n2, kps);
      } else {
        rc = encode_rows(&h->tm_w13[l], layers[l].w13, H / 2, E * 2 * I, 128);
        if (!rc) rc = kps == 1 ? encode_rows(&h->tm_w2[l], layers[l].w2, I / 2, E * H, 128)
                               : encode_rows_kb(&h->tm_w2[l], layers[l].w2, I / 2, E * H, 128, kps);
      }
    }
    if (!rc && cudaDeviceSynchronize() != cudaSuccess) rc = fail(MOE_ECUDA, "scale atoms");
    if (rc) {
      moe_decode_destroy(h);
      return rc;
    }
  }
#endif
  *out = h;
  return MOE_OK;
}

int moe_decode_layer(moe_decode_t* h, int layer, int rows, const uint16_t* branch, float* stream,
                     void* cuda_stream) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  if (layer < 0 || layer >= h->d.n_layers)
    return fail(MOE_EINVAL, "layer %d outside [0, %d)", layer, h->d.n_layers);
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!stream || !aligned(stream, 16)) return fail(MOE_EINVAL, "stream must be 16-byte aligned");
  if (branch && !aligned(branch, 8)) return fail(MOE_EINVAL, "branch must be 8-byte aligned");
  return launch_layer(h, layer, rows, branch, stream, static_cast<cudaStream_t>(cuda_stream));
}

int moe_decode_final(moe_decode_t* h, int rows, float* stream, uint16_t* out, float* aux,
                     void* cuda_stream) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!stream || !out || !aligned(stream, 16) || !aligned(out, 8) || !aligned(aux, 16))
    return fail(MOE_EINVAL, "stream and aux (16-byte) and out (8-byte) must be aligned device pointers");
  if (!h->w_post_final || !h->w_final)
    return fail(MOE_EINVAL, "the handle was created without final norm weights");
  return launch_final(h, rows, stream, out, static_cast<cudaStream_t>(cuda_stream), aux);
}

int moe_decode_front(moe_decode_t* h, int rows, const uint16_t* embedded, const float* w_norm,
                     float* stream, uint16_t* attn_input, float* aux, void* cuda_stream) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!embedded || !w_norm || !stream || !attn_input)
    return fail(MOE_EINVAL, "embedded, w_norm, stream and attn_input are required");
  if (!aligned(embedded, 8) || !aligned(w_norm, 16) || !aligned(stream, 16) ||
      !aligned(attn_input, 8) || !aligned(aux, 16))
    return fail(MOE_EINVAL, "w_norm, stream and aux must be 16-byte, embedded and attn_input 8-byte aligned");
  const moe_decode_dims& d = h->d;
  moe::BoundaryParams bp{};
  bp.H = d.hidden;
  bp.k = d.top_k;
  bp.rows = rows;
  bp.cols_per_cta = d.hidden / h->cluster;
  bp.eps = d.eps;
  bp.branch = reinterpret_cast<const __nv_bfloat16*>(embedded);
  bp.stream = stream;
  bp.w_pre = w_norm;
  bp.x_out = reinterpret_cast<__nv_bfloat16*>(attn_input);
  bp.front = 1;
  bp.aux = aux;
  const cudaError_t e = moe::launch_boundary(bp, h->cluster, static_cast<cudaStream_t>(cuda_stream), false);
  if (e != cudaSuccess) return cuda_fail(e, "front launch");
  return MOE_OK;
}

int moe_decode_step(moe_decode_t* h, int rows, const uint16_t* branch, float* stream,
                    uint16_t* out, void* cuda_stream) {
  const int rc = check_step_args(h, rows, branch, stream, out);
  if (rc) return rc;
  return enqueue_step(h, rows, branch, stream, out, static_cast<cudaStream_t>(cuda_stream));
}

int moe_decode_step_graph(moe_decode_t* h, int rows, const uint16_t* branch, float* stream,
                          uint16_t* out, void* cuda_stream) {
  int rc = check_step_args(h, rows, branch, stream, out);
  if (rc) return rc;
  cudaGraphExec_t exec = moe::graph_cache_find(h->graphs, [&](const GraphEntry& g) {
    return g.rows == rows && g.branch == branch && g.stream == stream && g.out == out;
  });
  if (!exec) {
    cudaError_t e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "begin capture");
    rc = enqueue_step(h, rows, branch, stream, out, h->cap_stream);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(h->cap_stream, &graph);
    if (rc) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    if (e != cudaSuccess) return cuda_fail(e, "end capture");
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return cuda_fail(e, "graph instantiate");
    moe::graph_cache_insert(h->graphs, GraphEntry{rows, branch, stream, out, exec});
  }
  const cudaError_t e = cudaGraphLaunch(exec, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "graph launch");
  return MOE_OK;
}

int moe_decode_step_host(moe_decode_t* h, int rows, const uint16_t* branch_host,
                         float* stream_host, uint16_t* out_host, void* cuda_stream) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!branch_host || !stream_host || !out_host)
    return fail(MOE_EINVAL, "branch_host, stream_host and out_host are required");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const size_t n = (size_t)rows * h->d.hidden;
  // Pinned host buffers: the copies in, the step and the copies out as one
  // cached graph, so a call is one launch and one synchronization.
  if (host_pinned(branch_host) && host_pinned(stream_host) && host_pinned(out_host)) {
    cudaGraphExec_t exec = moe::graph_cache_find(h->host_graphs, [&](const GraphEntry& g) {
      return g.rows == rows && g.branch == branch_host && g.stream == stream_host && g.out == out_host;
    });
    if (!exec) {
      cudaStream_t c = h->cap_stream;
      // mapped pinned buffers: the first boundary reads the branch and the
      // stream from host memory and the final boundary writes the output and
      // the stream back there, so the kernels make the copies themselves;
      // otherwise copy-engine copies around the step
      const uint16_t* branch_d = static_cast<const uint16_t*>(moe::host_mapped(branch_host));
      float* stream_d = static_cast<float*>(moe::host_mapped(stream_host));
      uint16_t* out_d = static_cast<uint16_t*>(moe::host_mapped(out_host));
      const bool direct = branch_d && stream_d && out_d && aligned(stream_d, 16) && aligned(branch_d, 8) &&
                          aligned(out_d, 8);
      cudaError_t e = cudaStreamBeginCapture(c, cudaStreamCaptureModeThreadLocal);
      if (e != cudaSuccess) return cuda_fail(e, "begin capture");
      int erc = 0;
      if (direct) {
        erc = enqueue_step(h, rows, branch_d, h->io_stream, out_d, c, stream_d, stream_d);
      } else {
        e = cudaMemcpyAsync(h->io_branch, branch_host, n * 2, cudaMemcpyHostToDevice, c);
        if (e == cudaSuccess) e = cudaMemcpyAsync(h->io_stream, stream_host, n * 4, cudaMemcpyHostToDevice, c);
        erc = (e == cudaSuccess) ? enqueue_step(h, rows, h->io_branch, h->io_stream, h->io_out, c)
                                 : cuda_fail(e, "input copy");
        if (!erc) {
          e = cudaMemcpyAsync(stream_host, h->io_stream, n * 4, cudaMemcpyDeviceToHost, c);
          if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, h->io_out, n * 2, cudaMemcpyDeviceToHost, c);
          if (e != cudaSuccess) erc = cuda_fail(e, "output copy");
        }
      }
      cudaGraph_t graph = nullptr;
      e = cudaStreamEndCapture(c, &graph);
      if (erc) {
        if (graph) cudaGraphDestroy(graph);
        return erc;
      }
      if (e != cudaSuccess) return cuda_fail(e, "end capture");
      e = cudaGraphInstantiate(&exec, graph, 0);
      cudaGraphDestroy(graph);
      if (e != cudaSuccess) return cuda_fail(e, "graph instantiate");
      moe::graph_cache_insert(h->host_graphs, GraphEntry{rows, branch_host, stream_host, out_host, exec});
    }
    cudaError_t e = cudaGraphLaunch(exec, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "host-buffer step");
    return MOE_OK;
  }
  cudaError_t e = cudaMemcpyAsync(h->io_branch, branch_host, n * 2, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h->io_stream, stream_host, n * 4, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "input copy");
  rc = moe_decode_step_graph(h, rows, h->io_branch, h->io_stream, h->io_out, cuda_stream);
  if (rc) return rc;
  e = cudaMemcpyAsync(stream_host, h->io_stream, n * 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, h->io_out, n * 2, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "output copy");
  return MOE_OK;
}

int moe_decode_layer_profile(moe_decode_t* h, int layer, int rows, const uint16_t* branch,
                             float* stream, void* cuda_stream, float* kernel_ms_host) {
  if (!h || !kernel_ms_host) return fail(MOE_EINVAL, "handle and kernel_ms_host are required");
  if (layer < 0 || layer >= h->d.n_layers)
    return fail(MOE_EINVAL, "layer %d outside [0, %d)", layer, h->d.n_layers);
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!stream || !aligned(stream, 16)) return fail(MOE_EINVAL, "stream must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaEvent_t ev[6] = {};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 6 && e == cudaSuccess; ++i) e = cudaEventCreate(&ev[i]);
  if (e == cudaSuccess) {
    rc = launch_layer(h, layer, rows, branch, stream, s, ev);
    if (!rc) e = cudaEventSynchronize(ev[5]);
    for (int i = 0; i < 5 && !rc && e == cudaSuccess; ++i)
      e = cudaEventElapsedTime(&kernel_ms_host[i], ev[i], ev[i + 1]);
    if (MOE_EXPERT_TC && !rc) {
      kernel_ms_host[4] = 0.0f;                  // gate/up and down share slot 3
      if (rows <= 32) kernel_ms_host[2] = 0.0f;  // no pooler gather
    }
  }
  for (int i = 0; i < 6; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  if (rc) return rc;
  if (e != cudaSuccess) return cuda_fail(e, "profile events");
  return MOE_OK;
}

int moe_decode_debug(moe_decode_t* h, moe_decode_debug_view* v) {
  if (!h || !v) return fail(MOE_EINVAL, "handle and view are required");
  const moe::Workspace& w = h->ws;
  v->x = reinterpret_cast<const uint16_t*>(w.x);
  v->x_codes = w.x_codes;
  v->x_sf = w.x_sf;
  v->x_sg = w.x_sg;
  v->logits = w.logits;
  v->ids = w.ids;
  v->gates = w.gates;
  v->flags = w.flags;
  v->count = w.count;
  v->offset = w.offset;
  v->pair_order = w.pair_order;
  v->pos_of_pair = w.pos_of_pair;
  v->active = w.active;
  v->n_active = w.n_active;
  v->h = w.h;
  v->h_sg = w.h_sg;
  v->h_codes = w.h_codes;
  v->h_sf = w.h_sf;
  v->o = w.o;
  return MOE_OK;
}

int moe_decode_last_error(moe_decode_t* h) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  // the workspace guards: a changed one latches kDevCanary and its index
  const int n = (int)h->guards.size();
  guard_kernel<<<(n + 127) / 128, 128>>>(static_cast<uint8_t*>(h->ws_mem), h->guard_offsets, n, 1,
                                         h->ws.err);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "workspace guard check");
  unsigned flag[2] = {0u, 0u};
  e = cudaMemcpy(flag, h->ws.err, sizeof(flag), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "error flag read");
  if (flag[0]) {
    const unsigned none = 0xFFFFFFFFu;
    cudaMemset(h->ws.err, 0, sizeof(unsigned));
    cudaMemcpy(h->ws.err + 1, &none, sizeof(none), cudaMemcpyHostToDevice);
    if (flag[0] == moe::kDevCanary && flag[1] < h->guards.size()) {
      // the guard is rewritten: the next check reports only new damage
      guard_kernel<<<(n + 127) / 128, 128>>>(static_cast<uint8_t*>(h->ws_mem), h->guard_offsets, n, 0,
                                             h->ws.err);
      cudaDeviceSynchronize();
      return fail(MOE_EDEVICE, "device-side error 4: the workspace guard after region '%s' changed "
                  "(a write past that region's end)", h->guards[flag[1]].name);
    }
    return fail(MOE_EDEVICE, "device-side error %u (1 = bounded wait gave up, 2 = bad routing, "
                "3 = an index out of range in a bounds-check build)", flag[0]);
  }
  return MOE_OK;
}

int moe_decode_build_info(void) {
  return (moe::kBoundsCheck ? 1 : 0) | (MOE_EXPERT_TC ? 0 : 2);
}

size_t moe_decode_workspace_bytes(const moe_decode_t* h) { return h ? h->ws_bytes : 0; }

size_t moe_decode_weight_copy_bytes(const moe_decode_t* h) { return h ? h->copy_bytes : 0; }

int moe_decode_set_wait_limit(moe_decode_t* h, uint64_t limit_ns) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  if (limit_ns < 1000ull || limit_ns > 60000000000ull)
    return fail(MOE_EINVAL, "wait limit %llu ns outside [1 us, 60 s]", (unsigned long long)limit_ns);
  // the kernels take the limit as a launch parameter: cached graphs hold the
  // old one, so they are dropped and captured again on their next use
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "device synchronize");
  for (GraphEntry& g : h->graphs) cudaGraphExecDestroy(g.exec);
  for (GraphEntry& g : h->host_graphs) cudaGraphExecDestroy(g.exec);
  h->graphs.clear();
  h->host_graphs.clear();
  h->ws.wait_ns = limit_ns;
  return MOE_OK;
}

int moe_decode_selftest_wait_timeout(moe_decode_t* h, int rows, const uint16_t* branch,
                                     float* stream, void* cuda_stream) {
  if (!h) return fail(MOE_EINVAL, "null handle");
  if (!MOE_EXPERT_TC)
    return fail(MOE_EUNSUPPORTED, "the self-test withholds the tensor-core experts kernel's ready list");
  int rc = check_rows(h, rows);
  if (rc) return rc;
  if (!branch || !stream || !aligned(stream, 16) || !aligned(branch, 8))
    return fail(MOE_EINVAL, "branch (8-byte) and stream (16-byte) aligned device pointers are required");
  return launch_layer(h, 0, rows, branch, stream, static_cast<cudaStream_t>(cuda_stream), nullptr,
                      nullptr, true);
}

int64_t moe_tiled_code_bytes(int64_t rows, int64_t row_bytes) {
  if (rows <= 0 || rows % 128 || row_bytes <= 0 || row_bytes % 16)
    return fail(MOE_EINVAL, "rows must be a positive multiple of 128 and row_bytes of 16");
  if (row_bytes > (int64_t)1 << 30 || rows / 128 > ((int64_t)1 << 31) / ((row_bytes + 127) / 128))
    return fail(MOE_EINVAL, "code tensor too large (2^31 tiles at most)");
  return rows / 128 * ((row_bytes + 127) / 128) * 16384;
}

int moe_tile_codes(const uint8_t* src, int64_t rows, int64_t row_bytes, uint8_t* dst,
                   void* cuda_stream) {
  const int64_t bytes = moe_tiled_code_bytes(rows, row_bytes);
  if (bytes < 0) return (int)bytes;
  if (!src || !dst) return fail(MOE_EINVAL, "src and dst are required");
  if (!aligned(src, 16) || !aligned(dst, 16)) return fail(MOE_EINVAL, "src and dst must be 16-byte aligned");
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
  if (s0 < d0 + (uintptr_t)bytes && d0 < s0 + (uintptr_t)(rows * row_bytes))
    return fail(MOE_EINVAL, "src and dst overlap");
  const cudaError_t e = moe::launch_tile_codes(src, rows, (int)row_bytes, dst,
                                               static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "code tiling launch");
  return MOE_OK;
}

int moe_decode_step_kernel_count(const moe_decode_t* h) {
  if (!h) return 0;
  // boundary, router and the experts (or the CUDA-core build's gate/up and
  // down), the routing kernel beyond 8 rows, and the tensor-core build's
  // pooler gather beyond 32 rows; one final boundary per step
  const int R = h->d.max_rows;
  const int per_layer = (MOE_EXPERT_TC ? 3 + (R > 32) : 4) + (R > 8);
  return per_layer * h->d.n_layers + 1;
}

void moe_decode_destroy(moe_decode_t* h) {
  if (!h) return;
  for (GraphEntry& g : h->graphs) cudaGraphExecDestroy(g.exec);
  for (GraphEntry& g : h->host_graphs) cudaGraphExecDestroy(g.exec);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  cudaFree(h->io_branch);
  cudaFree(h->io_stream);
  cudaFree(h->io_out);
  cudaFree(h->ws_mem);
  for (uint8_t* p : h->sfa13) cudaFree(p);
  for (uint8_t* p : h->tiled13) cudaFree(p);
  for (uint8_t* p : h->tiled2) cudaFree(p);
  for (uint8_t* p : h->sfa2) cudaFree(p);
  delete h;
}

int moe_nvfp4_quantize(const float* v, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf,
                       float* sg, float* amax, void* cuda_stream) {
  if (!v || !codes || !sf || !sg || !amax) return fail(MOE_EINVAL, "null pointer");
  if (rows < 0 || cols < 0 || cols % 16) return fail(MOE_EINVAL, "cols must be a multiple of 16");
  if (!aligned(v, 16) || !aligned(codes, 8) || !aligned(sg, 4) || !aligned(amax, 4))
    return fail(MOE_EINVAL, "v must be 16-byte and codes 8-byte aligned");
  const cudaError_t e = moe::launch_quantize(v, rows, cols, codes, sf, sg, amax,
                                             static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return MOE_OK;
}

}  // extern "C"
