// One dense draft layer's MLP block at decode (after its attention, which is
// not part of this library).
//
// Page: vllm.models.muse_spark.common.dspark, MuseSparkDSparkDecoderLayer
// .forward: the stream is fp32 (a plain add of each normalised branch, as
// in the routed layers); the attention output enters through post_attn_norm;
// the feed-forward reads pre_ffn_norm of the stream cast to the draft's
// compute dtype (bf16), a cast the layer makes before every input norm; its
// output enters through post_ffn_norm.  The
// feed-forward is the dense gated MLP (gate_proj / up_proj stacked as shards
// 0 / 1 of gate_up_proj, the same page's weight mapping) in bf16:
//   s1 = s + rmsnorm(attn_out) * w_post_attn                 (fp32)
//   x  = bf16(rmsnorm(bf16(s1)) * w_pre_ffn)
//   g, u = bf16(W_gate x), bf16(W_up x)                      (fp32 accumulation)
//   a  = bf16(silu(g) * u)
//   f  = bf16(W_down a)
//   s2 = s1 + rmsnorm(f) * w_post_ffn                        (fp32)
//
// GB300 layout: the norms run in the boundary kernel (cluster per row).  Up
// to 8 rows the projections are the library's weight-streaming kernel
// (gemv.cuh): gate/up pairs each gate row with its up row in one task and
// writes gu and SiLU * mul from its accumulators; the down projection leaves
// fp32 split-K partials, which the output boundary sums in split order into
// the bf16 branch.  Beyond 8 rows (or for widths the streaming kernel does
// not take) the projections are the library's tensor-core projection kernel
// (tc_gemm.cu): gate/up with SiLU * mul from its two accumulators, down as
// split-K partials the output boundary sums the same way.  Four launches
// chained by programmatic dependent launch either way.
#include <cstdio>
#include <vector>

#include "../../include/moe_decode.h"
#include "common.cuh"
#include "gemv.cuh"
#include "moe_decode_internal.h"
#include "tc_gemm.h"

namespace {
constexpr int kDenseMaxSplits = 8;  // K-splits of the tensor-core down projection
}

struct moe_dense_s {
  moe_dense_dims d;
  moe_dense_weights w;
  int cluster;
  moe::GemmMaps gu_maps, dn_maps;  // the tensor-core projections' tensor maps
  unsigned* err;                   // [2] latched device error (a bounded wait that gave up)
  __nv_bfloat16 *x, *gu, *a, *f;  // [R][H], [R][2I], [R][I], [R][H]
  float* part;                     // down projection's split-K partials [S][rows][H]
  float* io_stream;                // [R][H] the stream of a host-buffer call
  __nv_bfloat16* io_attn;          // [R][H] its attention output (when copied in)
  struct HostGraph {
    int rows;
    const void* attn;
    const void* stream;
    cudaGraphExec_t exec;
  };
  std::vector<HostGraph> host_graphs;
  int down_splits;                 // K-splits of the streamed down projection; 0: no streaming
  int num_sms;
};

namespace {

bool dense_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_err(cudaError_t e, const char* what) {
  char buf[200];
  snprintf(buf, sizeof(buf), "%s: %s", what, cudaGetErrorString(e));
  return moe::api_fail(MOE_ECUDA, buf);
}

// The dense layer's launches on s; with ev, an event before each and after
// the last (boundary, gate/up, SiLU * mul, down, boundary).
// stream_in: where the first boundary reads the stream (null: stream itself);
// aux: where the output boundary also writes the new stream (or null).
int dense_enqueue(moe_dense_t* h, int rows, const uint16_t* attn_out, float* stream,
                  cudaStream_t s, cudaEvent_t* ev, const float* stream_in = nullptr, float* aux = nullptr) {
  const moe_dense_dims& d = h->d;
  auto mark = [&](int i) {
    if (ev) cudaEventRecord(ev[i], s);
  };
  mark(0);
  moe::BoundaryParams bp{};
  bp.H = d.hidden;
  bp.k = 1;
  bp.rows = rows;
  bp.cols_per_cta = d.hidden / h->cluster;
  bp.eps = d.eps;
  bp.branch = reinterpret_cast<const __nv_bfloat16*>(attn_out);
  bp.stream = stream;
  bp.stream_in = stream_in;
  bp.w_post = h->w.w_post_attn;
  bp.w_pre = h->w.w_pre_ffn;
  bp.x_out = h->x;
  bp.round_norm = 1;
  cudaError_t e = moe::launch_boundary(bp, h->cluster, s, false);
  if (e != cudaSuccess) return cuda_err(e, "pre-ffn boundary launch");
  mark(1);
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  int part_S = 0;
  if (h->down_splits && rows <= 8) {
    // Up to 8 rows: the library's weight-streaming projections.  Gate/up
    // pairs each gate row with its up row in one task and writes gu and
    // SiLU * mul itself; the down projection leaves split-K partials that the
    // output boundary sums.  Programmatic dependent launch between the four
    // kernels (except when profiled, where each launch is timed alone).
    cudaLaunchConfig_t gc = {};
    gc.gridDim = dim3(h->num_sms, 1, 1);
    gc.blockDim = dim3(moe::kGemvThreads, 1, 1);
    gc.dynamicSmemBytes = moe::kGemvSmem;
    gc.stream = s;
    gc.attrs = ev ? nullptr : &pdl;
    gc.numAttrs = ev ? 0 : 1;
    moe::GemvParams gp{};
    gp.W = reinterpret_cast<const __nv_bfloat16*>(h->w.w13);
    gp.X = h->x;
    gp.L = 1;
    gp.R = 2 * d.inter;
    gp.K = d.hidden;
    gp.n = rows;
    gp.S = 1;
    gp.KC = d.hidden;
    gp.I = d.inter;
    gp.gu = h->gu;
    gp.act = h->a;
    e = cudaLaunchKernelEx(&gc, moe::gemv_bf16_kernel<true>, gp);
    if (e != cudaSuccess) return cuda_err(e, "gate/up projection launch");
    mark(2);
    mark(3);  // SiLU * mul is part of the gate/up projection
    moe::GemvParams dp{};
    dp.W = reinterpret_cast<const __nv_bfloat16*>(h->w.w2);
    dp.X = h->a;
    dp.part = h->part;
    dp.L = 1;
    dp.R = d.hidden;
    dp.K = d.inter;
    dp.n = rows;
    dp.S = h->down_splits;
    dp.KC = d.inter / h->down_splits;
    e = cudaLaunchKernelEx(&gc, moe::gemv_bf16_kernel<false>, dp);
    if (e != cudaSuccess) return cuda_err(e, "down projection launch");
    part_S = h->down_splits;
  } else {
    // Beyond: the tensor-core projection kernel, gate/up with SiLU * mul from
    // its two accumulators, then down as split-K partials.
    moe::GemmParams gp;
    if (!moe::plan_gemm(gp, moe::kGemmGated, 1, 2 * d.inter, d.hidden, rows, d.inter, 0, h->num_sms, 1))
      return moe::api_fail(MOE_EUNSUPPORTED, "no tensor-core plan for the gate/up projection");
    gp.gu = h->gu;
    gp.act = h->a;
    gp.err = h->err;
    e = moe::launch_gemm(gp, h->gu_maps, h->num_sms, s, !ev);
    if (e != cudaSuccess) return cuda_err(e, "gate/up projection launch");
    mark(2);
    mark(3);  // SiLU * mul is part of the gate/up projection
    moe::GemmParams dp;
    if (!moe::plan_gemm(dp, moe::kGemmPartial, 1, d.hidden, d.inter, rows, 0, 0, h->num_sms, kDenseMaxSplits))
      return moe::api_fail(MOE_EUNSUPPORTED, "no tensor-core plan for the down projection");
    dp.part = h->part;
    dp.err = h->err;
    e = moe::launch_gemm(dp, h->dn_maps, h->num_sms, s, !ev);
    if (e != cudaSuccess) return cuda_err(e, "down projection launch");
    part_S = dp.S;
  }
  mark(4);
  bp.branch = nullptr;
  bp.part = h->part;
  bp.part_S = part_S;
  bp.part_out = h->f;
  bp.w_post = h->w.w_post_ffn;
  bp.w_pre = h->w.w_post_ffn;  // read but unused: no normalised output
  bp.x_out = nullptr;
  bp.round_norm = 0;
  bp.stream_in = nullptr;
  bp.aux = aux;
  e = moe::launch_boundary(bp, h->cluster, s, !ev);
  if (e != cudaSuccess) return cuda_err(e, "post-ffn boundary launch");
  mark(5);
  return MOE_OK;
}

int check_rows_dense(const moe_dense_t* h, int rows) {
  if (rows < 1 || rows > h->d.max_rows) {
    char buf[96];
    snprintf(buf, sizeof(buf), "rows %d outside [1, max_rows=%d]", rows, h->d.max_rows);
    return moe::api_fail(MOE_EINVAL, buf);
  }
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_dense_create(const moe_dense_dims* dims, const moe_dense_weights* w, moe_dense_t** out) {
  if (!dims || !w || !out) return moe::api_fail(MOE_EINVAL, "dims, weights and out are required");
  *out = nullptr;
  const moe_dense_dims d = *dims;
  if (d.hidden <= 0 || d.hidden % 128 || d.hidden > 16384)
    return moe::api_fail(MOE_EUNSUPPORTED, "hidden must be a positive multiple of 128, at most 16384");
  if (d.inter <= 0 || d.inter % 8)
    return moe::api_fail(MOE_EUNSUPPORTED, "inter must be a positive multiple of 8");
  if (d.max_rows < 1 || d.max_rows > 128) return moe::api_fail(MOE_EUNSUPPORTED, "max_rows must be in [1, 128]");
  if (!(d.eps > 0.0f)) return moe::api_fail(MOE_EINVAL, "eps must be positive");
  if (!w->w_post_attn || !w->w_pre_ffn || !w->w13 || !w->w2 || !w->w_post_ffn)
    return moe::api_fail(MOE_EINVAL, "a required weight pointer is NULL");
  if (!dense_aligned(w->w_post_attn, 16) || !dense_aligned(w->w_pre_ffn, 16) ||
      !dense_aligned(w->w_post_ffn, 16) || !dense_aligned(w->w13, 16) || !dense_aligned(w->w2, 16))
    return moe::api_fail(MOE_EINVAL, "weight pointers must be 16-byte aligned");
  int dev = 0, major = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return cuda_err(e, "device query");
  if (major != 10) return moe::api_fail(MOE_EUNSUPPORTED, "needs an SM 10.x GPU");
  moe_dense_t* h = new moe_dense_t{};
  h->d = d;
  h->w = *w;
  h->cluster = moe::boundary_cluster(d.hidden);
  int num_sms = 0;
  e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    delete h;
    return cuda_err(e, "device query");
  }
  h->num_sms = num_sms;
  // the streamed projections need H a multiple of 128 (gate/up K) and I one
  // of 128 (down K; gate/up rows in groups of 16)
  if (d.inter % 128 == 0) h->down_splits = moe::gemv_splits(1, d.hidden, d.inter, num_sms);
  if (h->down_splits) {
    e = cudaFuncSetAttribute(moe::gemv_bf16_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)moe::kGemvSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(moe::gemv_bf16_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)moe::kGemvSmem);
    if (e != cudaSuccess) {
      delete h;
      return cuda_err(e, "streaming projection shared memory");
    }
  }
  e = moe::gemm_set_smem();
  if (e != cudaSuccess) {
    delete h;
    return cuda_err(e, "tensor-core projection shared memory");
  }
  const size_t R = (size_t)d.max_rows, H = (size_t)d.hidden, I = (size_t)d.inter;
  // the down projection's partials: the streamed path's [S][8][H] or the
  // tensor-core path's [S][R][H], whichever is larger
  const size_t part_stream = h->down_splits ? (size_t)h->down_splits * 8 * H : 0;
  const size_t part_tc = (size_t)kDenseMaxSplits * R * H;
  const size_t part_bytes = (part_stream > part_tc ? part_stream : part_tc) * sizeof(float);
  const size_t bytes = 2 * (R * H + R * 2 * I + R * I + R * H) + part_bytes + R * H * (4 + 2) + 16;
  uint8_t* base = nullptr;
  e = cudaMalloc(&base, bytes);
  if (e != cudaSuccess) {
    moe_dense_destroy(h);
    return moe::api_fail(MOE_ENOMEM, "dense layer workspace");
  }
  h->x = reinterpret_cast<__nv_bfloat16*>(base);
  h->gu = h->x + R * H;
  h->a = h->gu + R * 2 * I;
  h->f = h->a + R * I;
  h->part = reinterpret_cast<float*>(h->f + R * H);
  h->io_stream = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(h->f + R * H) + part_bytes);
  h->io_attn = reinterpret_cast<__nv_bfloat16*>(h->io_stream + R * H);
  h->err = reinterpret_cast<unsigned*>(h->io_attn + R * H);
  e = cudaMemset(h->err, 0, 2 * sizeof(unsigned));
  // the tensor-core projections' tensor maps: W13 [2I][H] over x [R][H], W2
  // [H][I] over a [R][I]
  if (e == cudaSuccess)
    e = moe::encode_gemm_maps(h->gu_maps, h->w.w13, 2 * (int64_t)I, h->x, (int64_t)R, (int)H);
  if (e == cudaSuccess) e = moe::encode_gemm_maps(h->dn_maps, h->w.w2, (int64_t)H, h->a, (int64_t)R, (int)I);
  if (e != cudaSuccess) {
    moe_dense_destroy(h);
    return cuda_err(e, "dense layer set-up");
  }
  *out = h;
  return MOE_OK;
}

int moe_dense_layer(moe_dense_t* h, int rows, const uint16_t* attn_out, float* stream,
                    void* cuda_stream) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  int rc = check_rows_dense(h, rows);
  if (rc) return rc;
  if (!attn_out || !stream || !dense_aligned(attn_out, 8) || !dense_aligned(stream, 16))
    return moe::api_fail(MOE_EINVAL, "attn_out (8-byte) and stream (16-byte) must be aligned device pointers");
  return dense_enqueue(h, rows, attn_out, stream, static_cast<cudaStream_t>(cuda_stream), nullptr);
}

int moe_dense_layer_host(moe_dense_t* h, int rows, const uint16_t* attn_host, float* stream_host,
                         void* cuda_stream) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  int rc = check_rows_dense(h, rows);
  if (rc) return rc;
  if (!attn_host || !stream_host) return moe::api_fail(MOE_EINVAL, "attn_host and stream_host are required");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  const size_t n = (size_t)rows * h->d.hidden;
  const uint16_t* attn_d = static_cast<const uint16_t*>(moe::host_mapped(attn_host));
  float* stream_d = static_cast<float*>(moe::host_mapped(stream_host));
  cudaError_t e = cudaSuccess;
  if (attn_d && stream_d && dense_aligned(attn_d, 8) && dense_aligned(stream_d, 16)) {
    // mapped page-locked buffers: the boundaries read and write host memory
    // themselves; the layer is one cached graph per (rows, buffers)
    cudaGraphExec_t exec = moe::graph_cache_find(h->host_graphs, [&](const moe_dense_s::HostGraph& g) {
      return g.rows == rows && g.attn == attn_host && g.stream == stream_host;
    });
    if (!exec) {
      cudaStream_t c = nullptr;
      e = cudaStreamCreateWithFlags(&c, cudaStreamNonBlocking);
      if (e != cudaSuccess) return cuda_err(e, "stream create");
      cudaGraph_t graph = nullptr;
      e = cudaStreamBeginCapture(c, cudaStreamCaptureModeThreadLocal);
      if (e == cudaSuccess) {
        rc = dense_enqueue(h, rows, attn_d, h->io_stream, c, nullptr, stream_d, stream_d);
        e = cudaStreamEndCapture(c, &graph);
      }
      cudaStreamDestroy(c);
      if (rc || e != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return rc ? rc : cuda_err(e, "host-buffer layer capture");
      }
      e = cudaGraphInstantiate(&exec, graph, 0);
      cudaGraphDestroy(graph);
      if (e != cudaSuccess) return cuda_err(e, "graph instantiate");
      moe::graph_cache_insert(h->host_graphs, moe_dense_s::HostGraph{rows, attn_host, stream_host, exec});
    }
    e = cudaGraphLaunch(exec, s);
  } else {
    e = cudaMemcpyAsync(h->io_attn, attn_host, n * 2, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(h->io_stream, stream_host, n * 4, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_err(e, "input copy");
    rc = dense_enqueue(h, rows, reinterpret_cast<const uint16_t*>(h->io_attn), h->io_stream, s, nullptr);
    if (rc) return rc;
    e = cudaMemcpyAsync(stream_host, h->io_stream, n * 4, cudaMemcpyDeviceToHost, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_err(e, "host-buffer layer");
  return MOE_OK;
}

int moe_dense_layer_profile(moe_dense_t* h, int rows, const uint16_t* attn_out, float* stream,
                            void* cuda_stream, float* ms_host) {
  if (!h || !ms_host) return moe::api_fail(MOE_EINVAL, "handle and ms_host are required");
  int rc = check_rows_dense(h, rows);
  if (rc) return rc;
  if (!attn_out || !stream || !dense_aligned(attn_out, 8) || !dense_aligned(stream, 16))
    return moe::api_fail(MOE_EINVAL, "attn_out (8-byte) and stream (16-byte) must be aligned device pointers");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaEvent_t ev[6] = {};
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 6 && e == cudaSuccess; ++i) e = cudaEventCreate(&ev[i]);
  if (e == cudaSuccess) {
    rc = dense_enqueue(h, rows, attn_out, stream, s, ev);
    if (!rc) e = cudaEventSynchronize(ev[5]);
    for (int i = 0; i < 5 && !rc && e == cudaSuccess; ++i)
      e = cudaEventElapsedTime(&ms_host[i], ev[i], ev[i + 1]);
  }
  for (int i = 0; i < 6; ++i)
    if (ev[i]) cudaEventDestroy(ev[i]);
  if (rc) return rc;
  if (e != cudaSuccess) return cuda_err(e, "profile events");
  return MOE_OK;
}

int moe_dense_kernel_count(moe_dense_t* h, int rows) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  int rc = check_rows_dense(h, rows);
  if (rc) return rc;
  // capture one layer on a private stream (inputs: the handle's own buffers,
  // nothing runs) and count the graph's kernel nodes
  cudaStream_t s = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_err(e, "stream create");
  cudaGraph_t g = nullptr;
  e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
  if (e == cudaSuccess) {
    rc = dense_enqueue(h, rows, reinterpret_cast<const uint16_t*>(h->x), reinterpret_cast<float*>(h->gu), s, nullptr);
    e = cudaStreamEndCapture(s, &g);
  }
  int count = 0;
  size_t n = 0;
  if (e == cudaSuccess && !rc) e = cudaGraphGetNodes(g, nullptr, &n);
  if (e == cudaSuccess && !rc && n) {
    std::vector<cudaGraphNode_t> nodes(n);
    e = cudaGraphGetNodes(g, nodes.data(), &n);
    for (size_t i = 0; i < n && e == cudaSuccess; ++i) {
      cudaGraphNodeType t;
      e = cudaGraphNodeGetType(nodes[i], &t);
      count += (t == cudaGraphNodeTypeKernel);
    }
  }
  if (g) cudaGraphDestroy(g);
  cudaStreamDestroy(s);
  if (rc) return rc;
  if (e != cudaSuccess) return cuda_err(e, "launch count capture");
  return count;
}

int moe_dense_debug(moe_dense_t* h, moe_dense_debug_view* v) {
  if (!h || !v) return moe::api_fail(MOE_EINVAL, "handle and view are required");
  v->x = h->x;
  v->gu = h->gu;
  v->a = h->a;
  v->f = h->f;
  return MOE_OK;
}

int moe_dense_last_error(moe_dense_t* h) {
  if (!h) return moe::api_fail(MOE_EINVAL, "null handle");
  cudaError_t e = cudaDeviceSynchronize();
  unsigned flag = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&flag, h->err, sizeof(flag), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_err(e, "dense layer error word");
  if (flag) {
    cudaMemset(h->err, 0, sizeof(unsigned));
    char buf[96];
    snprintf(buf, sizeof(buf), "device-side error %u (1 = a bounded wait gave up)", flag);
    return moe::api_fail(MOE_EDEVICE, buf);
  }
  return MOE_OK;
}

void moe_dense_destroy(moe_dense_t* h) {
  if (!h) return;
  for (const auto& g : h->host_graphs) cudaGraphExecDestroy(g.exec);
  cudaFree(h->x);
  delete h;
}

}  // extern "C"
