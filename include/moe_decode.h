/*
 * moe_decode.h -- C ABI of the GB300 (sm_103a) routed NVFP4 mixture-of-experts
 * decode layer-step.
 *
 * What one layer-step computes (the specialized decode executor page,
 * vllm.models.muse_spark.nvidia.specialized_decode.runtime.decode, module
 * docstring "One step of b rows" -- one request verifying 1 + 7 tokens, b
 * rows; the attention boundary "all-reduce + the dual norm into the stream
 * and the MoE input"; the MoE "router -> routing -> pooler -> routed experts
 * -> tail -> unpooler"; "final: the last gather + dual norm"; the dual norm's
 * form is MuseSparkDSparkDecoderLayer.forward on the DSpark page,
 * vllm.models.muse_spark.common.dspark):
 *
 *   stream' = stream + rmsnorm(branch) * w_post            fp32 stream
 *   x       = bf16(rmsnorm(stream') * w_pre)               MoE input
 *   logit   = x Wr^T (+ bias);  p = softmax(logit)
 *   ids     = top-k of p (ties to the lower id), slots by descending p
 *   gates   = p[ids] / sum p[ids]
 *   xq      = NVFP4(x)                 one tensor over all rows
 *   h       = silu(Wg xq) * (Wu xq)    per (row, slot), fp32
 *   hq      = NVFP4(h)                 one tensor per expert (its rows)
 *   o       = Wd hq                    per (row, slot), fp32
 *   y[r]    = sum_s gates[r][s] o[r][s]   -> the next layer's branch, or
 *   final:  stream' = stream + rmsnorm(y) * w_post_final;
 *           out = bf16(rmsnorm(stream') * w_final)
 *
 * NVFP4 (every expert weight and activation operand): element = e2m1 code
 * (4 bits) * e4m3 block scale (one per 16 consecutive elements along the
 * reduction dimension) * fp32 tensor scale; tensor scale = amax / (6 * 448);
 * block scale = e4m3(amax_blk / 6 / tensor scale), round to nearest even,
 * saturating; code = e2m1(v / (block scale * tensor scale)).
 *
 * Conventions
 *  - Every pointer is a DEVICE pointer unless the name ends in _host.  The
 *    caller owns all of them; weights must stay valid until destroy.  The
 *    library owns only its workspace, sized at create (no allocation later).
 *  - Layouts (row-major, K-major weights):
 *      router_w  bf16 [E][H]
 *      w13       e2m1x2 [E][2I][H/2]  rows 0..I-1 gate, I..2I-1 up;
 *                element 2j in the low nibble of byte j
 *      w13_sf    e4m3 [E][2I][H/16]
 *      w2        e2m1x2 [E][H][I/2],  w2_sf e4m3 [E][H][I/16]
 *      w_gscale  fp32 [E][3]          tensor scales of gate, up, down
 *      stream    fp32 [rows][H];  branch / out bf16 [rows][H]
 *  - Alignment: w13, w13_sf, w2, w2_sf, router_w 16 bytes; fp32 arrays and
 *    stream 16 bytes; branch and out 8 bytes.
 *  - Errors: functions return MOE_OK (0) or a negative MOE_E* code, checked
 *    before anything is launched; moe_decode_error_message() gives the reason
 *    of the last failure on this thread.  Faults detected on the device
 *    (a bounded wait that gave up, an out-of-range routing value) latch a
 *    flag read by moe_decode_last_error().  Nothing here traps on the device.
 *  - Asynchrony: layer / final / step calls are asynchronous on the given CUDA
 *    stream (a cudaStream_t passed as void*; NULL = the legacy default
 *    stream), allocate nothing and never synchronize, so they can be
 *    captured into a CUDA graph.  A handle serves one stream and one host
 *    thread at a time: its workspace and graph caches are not locked.
 *    Separate handles are independent.
 *  - Supported shapes: H and I multiples of 128, at most 8192;
 *    1 <= top_k <= min(E, 16); E <= 1024; 1 <= rows <= max_rows <= 128.
 *    The device must be of the SM 10.x family (built for sm_103a).
 */
#ifndef MOE_DECODE_H
#define MOE_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,        /* a null / misaligned pointer or an out-of-range argument */
  MOE_EUNSUPPORTED = -2,  /* a shape or device this library does not serve */
  MOE_ECUDA = -3,         /* a CUDA runtime call failed */
  MOE_ENOMEM = -4,        /* device memory (workspace, weight copies) could not be allocated */
  MOE_EDEVICE = -5        /* a device-side check latched an error */
};

typedef struct moe_decode_s moe_decode_t;

/* How a handle reads the expert codes (w13, w2) of moe_layer_weights.  The
 * block scales (w13_sf, w2_sf) are row-major in every case.
 *   MOE_CODES_ROW_MAJOR   the codes as laid out above, read in place.
 *   MOE_CODES_TILED       the caller's w13 / w2 already hold the codes in
 *                         16 KB tiles (moe_tile_codes), read in place: each
 *                         TMA copy of the experts kernel is then one
 *                         contiguous read (about 3 % faster at serving widths
 *                         than the row-major codes).  Tensor-core build only.
 *   MOE_CODES_TILED_COPY  the caller passes row-major codes and the handle
 *                         makes and keeps its own tiled copy, as many bytes
 *                         again as the codes; if that memory cannot be
 *                         allocated, create fails with MOE_ENOMEM.
 *                         Tensor-core build only.
 * The results are the same, bit for bit, whichever layout is read. */
enum { MOE_CODES_ROW_MAJOR = 0, MOE_CODES_TILED = 1, MOE_CODES_TILED_COPY = 2 };

typedef struct {
  int hidden;     /* H */
  int n_experts;  /* E */
  int top_k;      /* k */
  int inter;      /* I: expert intermediate width */
  int max_rows;   /* largest b any call will use */
  int n_layers;   /* L */
  float eps;      /* RMSNorm epsilon */
  int code_layout; /* MOE_CODES_*: how w13 and w2 are laid out (0: row-major) */
} moe_decode_dims;

typedef struct {
  const float* w_post;        /* [H]  norm weight of the incoming branch */
  const float* w_pre;         /* [H]  norm weight of the stream -> MoE input */
  const uint16_t* router_w;   /* bf16 [E][H] */
  const float* router_bias;   /* [E] additive logit bias, or NULL */
  const uint8_t* w13;         /* e2m1x2 [E][2I][H/2], or its tiles (MOE_CODES_TILED) */
  const uint8_t* w13_sf;      /* e4m3 [E][2I][H/16] */
  const uint8_t* w2;          /* e2m1x2 [E][H][I/2], or its tiles (MOE_CODES_TILED) */
  const uint8_t* w2_sf;       /* e4m3 [E][H][I/16] */
  const float* w_gscale;      /* [E][3] */
} moe_layer_weights;

/* Device pointers into the workspace, holding the last layer run's
 * intermediates (for staged checks).  Scalars are device pointers too. */
typedef struct {
  const uint16_t* x;          /* bf16 [rows][H]: MoE input */
  const uint8_t* x_codes;     /* [rows][H/2] */
  const uint8_t* x_sf;        /* [rows][H/16] */
  const float* x_sg;          /* [1] */
  const float* logits;        /* [rows][E] */
  const int32_t* ids;         /* [rows][k] */
  const float* gates;         /* [rows][k] */
  const uint8_t* flags;       /* [rows] */
  const int32_t* count;       /* [E] */
  const int32_t* offset;      /* [E+1] */
  const int32_t* pair_order;  /* [rows*k]: pair id r*k+s at each pooled position */
  const int32_t* pos_of_pair; /* [rows*k] */
  const int32_t* active;      /* [E] (n_active used) */
  const int32_t* n_active;    /* [1] */
  const float* h;             /* [rows*k][I], pooled order */
  const float* h_sg;          /* [E] */
  const uint8_t* h_codes;     /* [rows*k][I/2], pooled order */
  const uint8_t* h_sf;        /* [rows*k][I/16] */
  const float* o;             /* [rows*k][H], pair-id order */
} moe_decode_debug_view;

/* Validates the shapes, the device and every pointer, plans the kernels and
 * allocates the workspace.  `layers` points to dims->n_layers entries (copied).
 * w_post_final / w_final: [H] norm weights of the final boundary (may be
 * NULL if moe_decode_final / _step are never called).  The tensor-core build
 * also keeps, per layer, the weight scales rearranged for the tensor cores
 * (1/8 of the code bytes) and, with MOE_CODES_TILED_COPY, a tiled copy of
 * the expert codes (as many bytes as the codes; MOE_ENOMEM if it cannot be
 * allocated).  The caller keeps its weights alive until destroy. */
int moe_decode_create(const moe_decode_dims* dims, const moe_layer_weights* layers,
                      const float* w_post_final, const float* w_final, moe_decode_t** out);

/* One layer-step (boundary .. down) for `rows` rows.  branch: bf16 [rows][H],
 * or NULL to use the unpooled output of the previous layer call on this
 * handle (same rows) as the branch.  stream: fp32 [rows][H], updated in place. */
int moe_decode_layer(moe_decode_t* h, int layer, int rows, const uint16_t* branch, float* stream,
                     void* cuda_stream);

/* Final boundary: gathers the last layer's unpooled output into the stream
 * and writes out = bf16(rmsnorm(stream) * w_final).  aux: fp32 [rows][H]
 * receiving a copy of the updated stream (the drafter's final aux hidden
 * state; decode page, SpecializedDecode.run: final.run(final_slot, stream,
 * output, final_aux)), or NULL.  stream and aux 16-byte, out 8-byte aligned. */
int moe_decode_final(moe_decode_t* h, int rows, float* stream, uint16_t* out, float* aux,
                     void* cuda_stream);

/* The first layer's front (decode page, module docstring "One step of b
 * rows": "the embedded tokens into the stream (fp32) and its
 * pre_qkv_proj_norm into the attention input, one kernel"):
 *   stream     = fp32(embedded)                          [rows][H], written
 *   attn_input = bf16(rmsnorm(stream) * w_norm)          [rows][H]
 *   aux        = stream (a copy for the drafter), or NULL
 * embedded: bf16 [rows][H] (the embedding's output); w_norm: fp32 [H], the
 * first layer's input norm weight (caller-owned); eps is the handle's.
 * w_norm, stream and aux 16-byte, embedded and attn_input 8-byte aligned.
 * Asynchronous on cuda_stream. */
int moe_decode_front(moe_decode_t* h, int rows, const uint16_t* embedded, const float* w_norm,
                     float* stream, uint16_t* attn_input, float* aux, void* cuda_stream);

/* Every layer (layer 0 takes `branch`, later ones chain) and the final
 * boundary. */
int moe_decode_step(moe_decode_t* h, int rows, const uint16_t* branch, float* stream,
                    uint16_t* out, void* cuda_stream);

/* As moe_decode_step, replayed from a CUDA graph the library captures on the
 * first call for this (rows, branch, stream, out) and caches in the handle.
 * The first call for a new key must not itself be under stream capture.
 * Each of the library's graph caches (this one, the host-buffer step's and
 * the dense layer's) keeps the 32 most recently used graphs; an older one is
 * destroyed (freed by the runtime once it completes) and captured again if
 * its key comes back. */
int moe_decode_step_graph(moe_decode_t* h, int rows, const uint16_t* branch, float* stream,
                          uint16_t* out, void* cuda_stream);

/* End-to-end step on HOST buffers: brings branch and stream in, runs the
 * step, returns stream and out, and synchronizes the stream.  When all three
 * buffers are page-locked the step is one library-owned graph (cached per
 * rows and buffers, captured on the first call), launched once per call; if
 * the runtime also maps them into the device's address space (and stream is
 * 16-byte, branch and out 8-byte aligned), the first boundary reads branch
 * and stream from host memory and the final boundary writes stream and out
 * there, so the graph holds no copy-engine copies, else it copies in and out
 * around the step.  Pageable buffers take separate copies around the step
 * graph. */
int moe_decode_step_host(moe_decode_t* h, int rows, const uint16_t* branch_host,
                         float* stream_host, uint16_t* out_host, void* cuda_stream);

/* One layer-step with a CUDA event recorded on `cuda_stream` around each of
 * its kernels, launched without programmatic overlap so each duration is
 * that kernel's alone.  Synchronizes, then writes five durations (ms) to
 * kernel_ms_host[5]: boundary, router, pooler gather, routed experts, and a
 * fifth slot.  The tensor-core build runs gate/up and down in one kernel
 * (slot 3 holds both, slot 4 is 0) and gathers a pooled copy of the MoE
 * input only above 32 rows (slot 2 is 0 otherwise); the CUDA-core build has
 * no pooler gather (slot 2 is 0) and times gate/up (slot 3) and down
 * (slot 4) separately.  For measurement only; not capturable. */
int moe_decode_layer_profile(moe_decode_t* h, int layer, int rows, const uint16_t* branch,
                             float* stream, void* cuda_stream, float* kernel_ms_host);

/* Workspace pointers of the last layer run (see moe_decode_debug_view). */
int moe_decode_debug(moe_decode_t* h, moe_decode_debug_view* out);

/* Synchronizes the device, then returns MOE_EDEVICE if a device-side check
 * latched an error since create (and clears it), MOE_ECUDA on a CUDA error,
 * else MOE_OK.  The codes (in moe_decode_error_message): 1 a bounded wait
 * gave up, 2 routing produced an out-of-range value, 3 a data-dependent
 * index was out of range (bounds-check builds only; the access was
 * skipped), 4 a workspace guard changed.  Every region of the workspace is
 * followed by a 256-byte guard whose first 16 bytes hold a pattern written
 * at create; this call checks every guard, so a write past a region's end
 * is reported with the region's name (and the guard is rewritten). */
int moe_decode_last_error(moe_decode_t* h);

/* How this library was built: bit 0 set in a bounds-check build (compiled
 * with MOE_BOUNDS_CHECK: every index that comes from data is tested before
 * it addresses memory, latching code 3 instead of faulting); bit 1 set in
 * the CUDA-core expert build. */
int moe_decode_build_info(void);

/* The limit of every bounded wait in the handle's kernels (default 2 s):
 * a wait that runs this long gives up, the kernel latches the wait-timeout
 * code (moe_decode_last_error: MOE_EDEVICE, "device-side error 1"), lets its
 * copies in flight land, frees its tensor memory and returns.  limit_ns in
 * [1000, 6e10].  Synchronizes the device and drops the handle's cached
 * graphs (they hold the old limit; they are captured again on next use).
 * Not capturable. */
int moe_decode_set_wait_limit(moe_decode_t* h, uint64_t limit_ns);

/* Self-test of that give-up path, with no fault: one layer-step of layer 0
 * (as moe_decode_layer) whose experts kernel never publishes a finished
 * expert to its down phase, so every down item's wait for its expert runs
 * to the wait limit and gives up.  The layer's expert outputs are then left
 * unwritten; the stream is updated by the boundary as usual.  Expect
 * moe_decode_last_error to report MOE_EDEVICE (wait timeout) afterwards;
 * the handle stays usable and the next step computes normally.  Tensor-core
 * build only (MOE_EUNSUPPORTED otherwise).  Asynchronous on cuda_stream. */
int moe_decode_selftest_wait_timeout(moe_decode_t* h, int rows, const uint16_t* branch,
                                     float* stream, void* cuda_stream);

/* Bytes of device workspace (activations, routing and scratch) the handle
 * holds.  The rearranged weight copies it also holds are not counted (see
 * moe_decode_weight_copy_bytes). */
size_t moe_decode_workspace_bytes(const moe_decode_t* h);

/* Bytes of rearranged weight copies the handle holds: the scale atoms of the
 * tensor-core build (1/8 of the expert code bytes) and, with
 * MOE_CODES_TILED_COPY, the tiled copy of the codes (as many bytes as the
 * codes).  0 for a null handle. */
size_t moe_decode_weight_copy_bytes(const moe_decode_t* h);

/* The tiled layout of expert codes (MOE_CODES_TILED).  A code tensor of
 * `rows` rows of `row_bytes` bytes (w13: rows = E * 2I, row_bytes = H/2;
 * w2: rows = E * H, row_bytes = I/2) becomes
 *   tiles [rows / 128][ceil(row_bytes / 128)][128 rows][128 bytes]
 * (row tile outermost, then the 128-byte K-block), the bytes of a last
 * partial K-block beyond row_bytes zero.  Every expert's tiles are
 * contiguous: expert e's start at e * (rows_per_expert / 128) *
 * ceil(row_bytes / 128) * 16384 bytes.
 * moe_tiled_code_bytes returns the tiled size in bytes, or a negative MOE_E*
 * code if rows is not a positive multiple of 128 or row_bytes not a positive
 * multiple of 16.  moe_tile_codes writes the tiles of src (row-major, 16-byte
 * aligned) into dst (16-byte aligned, moe_tiled_code_bytes bytes, not
 * overlapping src); asynchronous on cuda_stream. */
int64_t moe_tiled_code_bytes(int64_t rows, int64_t row_bytes);
int moe_tile_codes(const uint8_t* src, int64_t rows, int64_t row_bytes, uint8_t* dst,
                   void* cuda_stream);

/* Number of kernels one moe_decode_step of max_rows rows launches: per layer
 * the boundary, the router and the experts, plus the routing kernel beyond 8
 * rows and the pooler gather beyond 32 (the CUDA-core build: gate/up and
 * down instead of the experts, no gather); one final boundary per step. */
int moe_decode_step_kernel_count(const moe_decode_t* h);

void moe_decode_destroy(moe_decode_t* h);

const char* moe_decode_strerror(int code);

/* Reason of the last failing call on this thread ("" if none). */
const char* moe_decode_error_message(void);

/* NVFP4 quantizer (the scheme above) for one fp32 tensor v[rows][cols],
 * cols % 16 == 0: writes codes [rows][cols/2], sf [rows][cols/16], the tensor
 * scale *sg and *amax (device scalars).  v 16-byte aligned, codes 8-byte
 * aligned.  Asynchronous on cuda_stream. */
int moe_nvfp4_quantize(const float* v, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* sf,
                       float* sg, float* amax, void* cuda_stream);

/* The same quantizer for callers that cannot allocate device memory: code
 * that runs inside another runtime which hands it only its input and output
 * buffers and keeps every allocation to itself, or a latency-critical loop
 * that cannot afford cudaMalloc / cudaFree (they may synchronize the whole
 * device).  The pages this library follows have no counterpart: it is a
 * deployment convenience, not part of the method.
 *
 * Same arguments and results as moe_nvfp4_quantize (codes, sf and *sg bit for
 * bit equal), minus the amax scalar: the reduction's scratch is a fixed array
 * inside the library (about 64 KB on every GPU that loads the library, held
 * until the process exits).  It allocates nothing and calls no allocating
 * routine.
 *   - At most 2^30 elements (rows * cols); larger tensors are rejected with
 *     MOE_EUNSUPPORTED before anything is launched.
 *   - The first call on each device looks up the scratch's device address
 *     (with that device current); make that first call before any stream
 *     capture on the device.  The address is kept with the unique ID of the
 *     context it was taken in: after a device reset (cudaDeviceReset, or a
 *     reset of the primary context) the next call looks it up again, and
 *     that call too should come before any capture.
 *   - v must be 16-byte, codes 8-byte and sg 4-byte aligned (MOE_EINVAL).
 *   - Every call on a device shares the one scratch array, which keeps the
 *     last call's contents (the call clears what must start at zero).  Calls
 *     that can overlap on the GPU -- on different streams, or from host
 *     threads without ordering between them -- race on it and may produce a
 *     wrong tensor scale: issue them on one stream.
 * Asynchronous on cuda_stream. */
int moe_nvfp4_quantize_noalloc(const float* v, int64_t rows, int64_t cols, uint8_t* codes,
                               uint8_t* sf, float* sg, void* cuda_stream);

/* ------------------------------------------------------------------------
 * Dense draft layer (the DSpark page, vllm.models.muse_spark.common.dspark,
 * MuseSparkDSparkDecoderLayer.forward): the MLP block of one dense layer at
 * decode, after its attention.
 *   s1 = s + rmsnorm(attn_out) * w_post_attn               (fp32 stream)
 *   x  = bf16(rmsnorm(bf16(s1)) * w_pre_ffn)   (the stream is cast to bf16,
 *                                                the draft's compute type,
 *                                                before the input norm)
 *   g, u = bf16(W_gate x), bf16(W_up x)         gate_up_proj shards 0 / 1
 *   a  = bf16(silu(g) * u);  f = bf16(W_down a)
 *   s2 = s1 + rmsnorm(f) * w_post_ffn                      (fp32 stream)
 * Up to 8 rows with H and I multiples of 128 the projections are the
 * library's own weight-streaming kernels; otherwise its tensor-core
 * projection kernel (tcgen05, bf16 operands).  Either way fp32 accumulation,
 * SiLU * mul fused into gate/up, and the down projection's split-K partials
 * summed in split order by the output boundary: four launches, all the
 * library's own.
 * ---------------------------------------------------------------------- */
typedef struct moe_dense_s moe_dense_t;

typedef struct {
  int hidden;    /* H, multiple of 128, <= 16384 */
  int inter;     /* I, multiple of 8 */
  int max_rows;  /* 1..128 */
  float eps;
} moe_dense_dims;

typedef struct {                 /* device pointers, caller-owned, 16-byte aligned */
  const float* w_post_attn;      /* [H] */
  const float* w_pre_ffn;        /* [H] */
  const uint16_t* w13;           /* bf16 [2I][H]: gate rows, then up rows */
  const uint16_t* w2;            /* bf16 [H][I] */
  const float* w_post_ffn;       /* [H] */
} moe_dense_weights;

typedef struct {                 /* device pointers into the handle's workspace */
  void* x;                       /* bf16 [rows][H]  the feed-forward input */
  void* gu;                      /* bf16 [rows][2I] gate and up projections */
  void* a;                       /* bf16 [rows][I]  silu(gate) * up */
  void* f;                       /* bf16 [rows][H]  the feed-forward output */
} moe_dense_debug_view;

/* Validates the shapes and allocates the workspace. */
int moe_dense_create(const moe_dense_dims* dims, const moe_dense_weights* w, moe_dense_t** out);

/* One layer's MLP block for `rows` rows: attn_out bf16 [rows][H] (8-byte
 * aligned), stream fp32 [rows][H] (16-byte aligned) updated in place.
 * Asynchronous on cuda_stream; a handle is used by one stream at a time. */
int moe_dense_layer(moe_dense_t* h, int rows, const uint16_t* attn_out, float* stream,
                    void* cuda_stream);

/* The same with a CUDA event around each launch (pre-ffn boundary, gate/up
 * GEMM, SiLU * mul, down GEMM, post-ffn boundary); synchronizes and writes
 * the five durations (ms) to ms_host[5].  For measurement. */
int moe_dense_layer_profile(moe_dense_t* h, int rows, const uint16_t* attn_out, float* stream,
                            void* cuda_stream, float* ms_host);

/* Workspace pointers of the last layer call (see moe_dense_debug_view). */
int moe_dense_debug(moe_dense_t* h, moe_dense_debug_view* out);

/* moe_dense_layer on HOST buffers: attn_host bf16 [rows][H] in, stream_host
 * fp32 [rows][H] in/out; synchronizes cuda_stream.  Page-locked buffers that
 * the runtime maps into the device's address space (attn 8-byte, stream
 * 16-byte aligned) are read and written by the first and last boundaries
 * themselves, the layer replayed from a graph cached per (rows, buffers);
 * other buffers are copied in and out around the layer. */
int moe_dense_layer_host(moe_dense_t* h, int rows, const uint16_t* attn_host, float* stream_host,
                         void* cuda_stream);

/* Kernels one moe_dense_layer call of `rows` rows launches: four, all the
 * library's own.
 * Counted by capturing a call into a graph on a private stream (nothing
 * runs).  Returns the count (> 0) or a negative MOE_E* code. */
int moe_dense_kernel_count(moe_dense_t* h, int rows);

/* Synchronizes the device and returns MOE_EDEVICE if a projection latched a
 * device-side error (code 1: a bounded wait gave up) since the last call (and
 * clears it), else MOE_OK. */
int moe_dense_last_error(moe_dense_t* h);

void moe_dense_destroy(moe_dense_t* h);

/* ------------------------------------------------------------------------
 * Draft context-KV projection (the DSpark page,
 * vllm.models.muse_spark.common.dspark, _project_muse_context_kv and
 * precompute_and_store_context_kv): context rows into every draft layer's
 * keys and values, and into the KV cache.
 *   fc   = bf16(rmsnorm(ctx) * w_hidden)                  hidden_norm
 *   u[l] = bf16(rmsnorm(fc) * w_pre[l])                   pre_qkv_proj_norm
 *   kv[l] = bf16(u[l] . W_kv[l]^T)      W_kv[l]: qkv_proj's K rows, then V rows
 *   k = bf16(k / sqrt(mean(k^2) + qk_eps)) per head (fp32, no weight)
 *   k = bf16(rotate(k, pos)): dimensions paired (j, j + D/2), angle
 *       pos * theta^(-2j/D) (RoFormer's rotary embedding); theta 0: none
 *   cache[l][slot] = k, v for every row with slot >= 0
 * Norm weights are the effective ones: a zero-centred gamma is passed as
 * 1 + gamma, a norm without a weight as ones.
 * ---------------------------------------------------------------------- */
typedef struct moe_ctxkv_s moe_ctxkv_t;

typedef struct {
  int hidden;        /* H: a multiple of 8, at most 8192 */
  int n_layers;      /* L: draft layers, 1..256 */
  int n_kv_heads;    /* KVH >= 1, KVH * D <= 32768 */
  int head_dim;      /* D: 64, 128 or 256 */
  int max_ctx;       /* most context rows per call, 1..65536 */
  int max_position;  /* rotary table rows: positions must lie in [0, max_position) */
  float eps;         /* hidden_norm and pre_qkv_proj_norm eps, > 0 */
  float qk_eps;      /* the key norm's eps, > 0 */
  double rope_theta; /* rotary base; 0 = no rotary embedding */
} moe_ctxkv_dims;

typedef struct {
  const float* w_hidden; /* fp32 [H] */
  const float* w_pre;    /* fp32 [L][H] */
  const uint16_t* w_kv;  /* bf16 [L][2 * KVH * D][H], K-major */
} moe_ctxkv_weights;

typedef struct {
  void* fc; /* bf16 [n][H] */
  void* u;  /* bf16 [L][n][H] */
  void* kv; /* bf16 [L][n][2 * KVH * D] */
  void* k;  /* bf16 [L][n][KVH][D] (when no k_out was given) */
  void* v;  /* bf16 [L][n][KVH][D] (when no v_out was given) */
} moe_ctxkv_debug_view;

/* Validates, allocates the workspace (about 2 * (1 + 2L) * max_ctx * H bytes
 * plus the projections) and builds the rotary table (max_position * D/2
 * cos/sin pairs, computed in fp64, stored fp32).  The caller keeps the
 * weights alive until destroy.  16-byte aligned weight pointers. */
int moe_ctxkv_create(const moe_ctxkv_dims* dims, const moe_ctxkv_weights* w, moe_ctxkv_t** out);

/* One projection of n_ctx rows, asynchronous on cuda_stream, capturable.
 *   context    bf16 [n_ctx][H], 16-byte aligned
 *   positions  int64 [n_ctx] (required with a rotary embedding)
 *   slots      int64 [L][slot_stride] (slot_stride 0: one map [n_ctx] for
 *              every layer), or NULL: no cache write.  A negative slot
 *              writes nothing; a slot >= n_slots writes nothing and latches
 *              error 4 (moe_ctxkv_last_error).
 *   k_cache, v_cache  bf16 [L][n_slots][KVH][D] (the paged cache with its
 *              blocks of 16 slots flattened), 16-byte aligned
 *   k_out, v_out  bf16 [L][n_ctx][KVH][D] or NULL (then the workspace)
 * A position outside [0, max_position) latches error 3 and leaves that row's
 * outputs unwritten.  Errors: MOE_EINVAL before any launch. */
int moe_ctxkv_project(moe_ctxkv_t* h, int n_ctx, const uint16_t* context, const int64_t* positions,
                      const int64_t* slots, int slot_stride, uint16_t* k_cache, uint16_t* v_cache,
                      int64_t n_slots, uint16_t* k_out, uint16_t* v_out, void* cuda_stream);

/* moe_ctxkv_project on HOST buffers for the context, positions, slot map and
 * the keys and values out (k_out_host, v_out_host bf16 [L][n_ctx][KVH][D],
 * required); the caches stay device memory.  Synchronizes cuda_stream.  When
 * every given host buffer is page-locked and mapped into the device's
 * address space, the kernels read and write them directly; otherwise they
 * are copied in and out (a slot map of at most n_layers * max_ctx entries). */
int moe_ctxkv_project_host(moe_ctxkv_t* h, int n_ctx, const uint16_t* context_host,
                           const int64_t* positions_host, const int64_t* slots_host, int slot_stride,
                           uint16_t* k_cache, uint16_t* v_cache, int64_t n_slots, uint16_t* k_out_host,
                           uint16_t* v_out_host, void* cuda_stream);

/* The same projection with CUDA events around its three launches (norms,
 * projection, key norm + rotation + cache write); synchronizes and writes
 * their durations (ms) to ms_host[0..2].  For measurement.  Up to 8 rows
 * (and H a multiple of 64) the projection is the library's split-K
 * weight-streaming kernel, beyond that its tensor-core projection kernel. */
int moe_ctxkv_profile(moe_ctxkv_t* h, int n_ctx, const uint16_t* context, const int64_t* positions,
                      const int64_t* slots, int slot_stride, uint16_t* k_cache, uint16_t* v_cache,
                      int64_t n_slots, void* cuda_stream, float* ms_host);

/* Workspace views of the last projection (device pointers). */
int moe_ctxkv_debug(moe_ctxkv_t* h, moe_ctxkv_debug_view* view);

/* Synchronizes the device and returns MOE_EDEVICE if a projection latched a
 * device-side error since the last call (and clears it), else MOE_OK. */
int moe_ctxkv_last_error(moe_ctxkv_t* h);

/* Kernels one moe_ctxkv_project call of n_ctx rows launches (the library's
 * three, all its own). 
 * Counted by capturing a call into a graph on a private stream (nothing
 * runs).  Returns the count (> 0) or a negative MOE_E* code. */
int moe_ctxkv_kernel_count(moe_ctxkv_t* h, int n_ctx);

void moe_ctxkv_destroy(moe_ctxkv_t* h);

#ifdef __cplusplus
}
#endif
#endif /* MOE_DECODE_H */
