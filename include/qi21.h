/*
 * qi21.h -- C ABI of the GB300 (sm_103a) Qwen-Image-2.1 single-stream DiT
 * block: prefill of the prompt prefix into a per-layer K/V cache, and the
 * denoiser step of the target rows against [cached prefix, own rows].
 *
 * Semantics follow the CPU-exact path of the docs.rs page
 * "cortiq_engine/qwen_image21.rs" (v0.8.4): Seg / Qi21Layout (positions,
 * block_ids), rope_tables, Qi21Dit::block_cpu, Qi21Dit::prefill and
 * Qi21Dit::step_cpu. The device contract (prefill keeps each layer's
 * post-RoPE K/V; step reads it) follows the module notes of
 * "gpu_wgpu/qi21.rs" (v0.8.3).
 *
 * Conventions shared by every entry point:
 *  - Pointers marked "device" are CUDA device pointers on the current
 *    device; "host" pointers are ordinary host memory. The caller owns every
 *    buffer it passes (weights, activations, workspace) and the stream. The
 *    library owns only qi21_kvcache objects.
 *  - Matrices are row-major. Weights are in nn.Linear layout [out][in].
 *  - Device work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and is asynchronous: a return of QI21_OK means
 *    "validated and enqueued".
 *  - On any error the host can detect (bad argument, shape, geometry,
 *    mask, too-small workspace) nothing is written and nothing is enqueued;
 *    the function returns a negative QI21_ERR_* and qi21_last_error()
 *    (thread-local) describes it. This mirrors the page's "decline, no
 *    partial results" convention. A pass (prefill, step, denoiser call)
 *    validates every layer and encodes every layer's tensor maps before it
 *    enqueues its first copy or kernel, so a failure found at any layer
 *    leaves the stream untouched.
 *  - Every spin-wait inside the kernels gives up after about 2 s and raises
 *    a device status word; qi21_device_status() reads and clears it.
 *  - Entry points may be called from several host threads at once, each on
 *    its own stream and buffers; the library's one-time set-up is
 *    thread-safe and kept per device (kernel attributes, SM count), so one
 *    process may drive several devices, each call working on the current
 *    one. A thread with no current CUDA context gets the current device's
 *    primary context bound on its first call (as the CUDA runtime does on a
 *    thread's first runtime call).
 *  - Every layer of a pass is bracketed by an NVTX range ("qi21 prefill
 *    layer l" / "qi21 step layer l"), visible to a profiler that collects
 *    NVTX and free otherwise.
 */
#ifndef QI21_H
#define QI21_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QI21_OK 0
#define QI21_ERR_ARG (-1)       /* null pointer, negative size, bad enum */
#define QI21_ERR_SHAPE (-2)     /* lengths/row counts that do not agree */
#define QI21_ERR_GEOM (-3)      /* geometry outside what the kernels take */
#define QI21_ERR_MASK (-4)      /* visibility not a non-decreasing leading run */
#define QI21_ERR_OOM (-5)       /* device allocation failed */
#define QI21_ERR_CUDA (-6)      /* a CUDA runtime call failed */
#define QI21_ERR_STATE (-7)     /* cache not prefilled / layer out of range */
#define QI21_ERR_WORKSPACE (-8) /* workspace too small or misaligned */
#define QI21_ERR_DEVICE (-9)    /* a kernel raised its status word (timeout) */
#define QI21_ERR_NONFINITE (-10) /* the optional finite check found NaN/Inf */

/* Segment kinds of a layout (qwen_image21.rs, enum Seg). */
#define QI21_SEG_TEXT 0  /* a = number of text rows, b unused */
#define QI21_SEG_IMAGE 1 /* a = h, b = w; h*w rows in raster order */

/* 16-bit element types (qi21_geom::dtype). */
#define QI21_DTYPE_F16 0  /* IEEE half */
#define QI21_DTYPE_BF16 1 /* bfloat16 (8-bit exponent, 7-bit mantissa) */

/* Model geometry (qwen_image21.rs, Qi21Config). Kernel limits (the page's
 * geom_ok, gpu_wgpu/qi21.rs): head_dim == 128, heads*head_dim == dim,
 * dim % 128 == 0, 128 <= dim <= 8192, mlp_hidden % 64 == 0, axes even and
 * summing to head_dim, layers >= 1, dtype QI21_DTYPE_F16 or _BF16.
 * Compute type: 16-bit operands of `dtype` (weight planes, the modulated-LN
 * rows, the qkv panel, the attention output, the SwiGLU hidden rows and
 * the K/V cache), f32 accumulation, f32 residual stream. The page's device
 * path converts F16 / Bf16 / F32 container weights into f16 planes
 * (gpu_wgpu/qi21.rs module notes, ZBlockDev::from_model_all); the bf16
 * type here keeps bf16 weights as they are, with bf16's f32-wide exponent
 * range in place of f16's range. */
typedef struct qi21_geom {
  int32_t dim;        /* H */
  int32_t heads;      /* nh */
  int32_t head_dim;   /* hd, must be 128 */
  int32_t mlp_hidden; /* I */
  int32_t layers;     /* L */
  int32_t axes[3];    /* RoPE axis widths (frame, h, w), e.g. 16, 56, 56 */
  float eps;          /* LayerNorm / RMSNorm epsilon, e.g. 1e-6 */
  float theta;        /* RoPE base, e.g. 10000 */
  int32_t dtype;      /* QI21_DTYPE_F16 (0) or QI21_DTYPE_BF16 (1) */
} qi21_geom;

/* One run of the joint sequence (qwen_image21.rs, enum Seg). The last
 * segment of a layout is the target image block; the rest is the prefix. */
typedef struct qi21_seg {
  int32_t kind;
  int32_t a;
  int32_t b;
} qi21_seg;

/* Device planes of one block, as produced by qi21_pack_layer, in the
 * geometry's 16-bit dtype (T below):
 *   wqkv  T [3H][H]  rows q (H), k (H), v (H)
 *   wo    T [H][H]
 *   w13   T [2I][H]  gate/up interleaved in 64-row blocks:
 *                    rows [128j, 128j+64) = gate rows [64j, 64j+64),
 *                    rows [128j+64, 128j+128) = up rows [64j, 64j+64)
 *   w2    T [H][I]   (down)
 *   norm_q, norm_k  f32 [128] per-head RMSNorm weights (used as is)
 * Tensor names on the page: attn.to_q/to_k/to_v, attn.to_out.0,
 * img_mlp.gate_layer (gate), img_mlp.proj (up), img_mlp.out (down),
 * attn.norm_q, attn.norm_k (qwen_image21.rs, Qi21Dit::from_cmf). */
typedef struct qi21_layer {
  const void* wqkv;
  const void* wo;
  const void* w13;
  const void* w2;
  const float* norm_q;
  const float* norm_k;
} qi21_layer;

/* Opaque per-prompt cache: L layers of post-RoPE K|V, [lp][2H] each in the
 * geometry's dtype
 * (K in columns [0, H), V in [H, 2H)), plus the layout, the prefix
 * visibility and the RoPE tables of the prefix rows and of the target rows
 * at the positions after THIS prefix (qwen_image21.rs, struct Qi21Prefix). */
typedef struct qi21_kvcache qi21_kvcache;

/* ------------------------------------------------------------- host ---- */

/* Text of the last error on this thread ("" if none). Never NULL. */
const char* qi21_last_error(void);

/* Library version string. */
const char* qi21_version(void);

/* 0 if the geometry is one the kernels take, else QI21_ERR_GEOM / _ARG. */
int qi21_geom_check(const qi21_geom* g);

/* Row counts of a layout (qwen_image21.rs, Qi21Layout::total, prefix_len,
 * target, validate): the last segment must be a non-empty image block and
 * the prefix non-empty. Any output pointer may be NULL. Host only. */
int qi21_layout_rows(const qi21_seg* segs, int32_t nseg, int32_t* total, int32_t* prefix,
                     int32_t* target);

/* Index construction of a layout, on the host (qwen_image21.rs,
 * Qi21Layout::positions, Qi21Layout::block_ids, rope_tables, and the
 * visibility end[i] of Qi21Dit::prefill). Outputs (each may be NULL):
 *   pos       int64 [total][3]   (frame, h, w)
 *   block_ids int32 [total]      -1 for text, else the image-block id
 *   vis       uint32 [prefix]    prefix row i sees keys [0, vis[i])
 *   cos, sin  f32 [total][hd/2]  hd = axes[0]+axes[1]+axes[2]; f32
 *             frequencies 1/theta^(2i/d), f32 angle, f32 cos/sin
 * Integers are exact; the tables are within a few ulp of any other f32
 * evaluation of the same formula. */
int qi21_layout_indices(const qi21_seg* segs, int32_t nseg, const int32_t axes[3], float theta,
                        int64_t* pos, int32_t* block_ids, uint32_t* vis, float* cos_,
                        float* sin_);

/* Bytes of one layer's packed planes (wqkv + wo + w13 + w2, 16-bit, each
 * 256-byte aligned). */
size_t qi21_layer_plane_bytes(const qi21_geom* g);

/* Workspace bytes of a pass over up to `max_rows` rows (prefill rows, or
 * the sum of the target rows of a step batch). */
size_t qi21_workspace_bytes(const qi21_geom* g, int32_t max_rows);

/* ----------------------------------------------------------- device ---- */

/* Pack one layer's weights (device, the geometry's dtype, nn.Linear
 * layout: wq/wk/wv/wo
 * [H][H], wgate/wup [I][H], wdown [H][I]; norm_q/norm_k device f32 [128])
 * into `planes` (device, >= qi21_layer_plane_bytes, 256-byte aligned) and
 * fill `out` with pointers into it (norm_q/norm_k are referenced, not
 * copied). Enqueued on `stream`. */
int qi21_pack_layer(const qi21_geom* g, const void* wq, const void* wk, const void* wv,
                    const void* wo, const void* wgate, const void* wup, const void* wdown,
                    const float* norm_q, const float* norm_k, void* planes, size_t plane_bytes,
                    qi21_layer* out, void* stream);

/* Allocate a cache for the layout (library-owned device memory; the
 * layout's tables are built on the host and copied synchronously). The
 * analogue of the page's per-prompt program (gpu_wgpu/qi21.rs, struct
 * Prog). Returns QI21_ERR_OOM if the device is out of memory. */
int qi21_kvcache_alloc(const qi21_geom* g, const qi21_seg* segs, int32_t nseg,
                       qi21_kvcache** out);

/* Free a cache (NULL is a no-op); synchronises the device first. The
 * analogue of release_key (gpu_wgpu/qi21.rs). */
void qi21_kvcache_free(qi21_kvcache* c);

/* Prefix rows, target rows and layers of a cache; any pointer may be NULL. */
int qi21_kvcache_info(const qi21_kvcache* c, int32_t* lp, int32_t* n, int32_t* layers);

/* Device pointer of layer `layer`'s K|V block, [lp][2H] of the geometry's
 * dtype (read-only use by the caller: parity checks, saving a prompt). */
int qi21_kvcache_layer(const qi21_kvcache* c, int32_t layer, const void** kv);

/* Prefill (qwen_image21.rs, Qi21Dit::prefill; gpu_wgpu/qi21.rs, prefill and
 * blocks()): the prefix rows x_prefix (device f32 [lp][H], read only)
 * through every block with the t = 0 modulation `mods0` (device f32 [4H],
 * raw [scale1|gate1|scale2|gate2]; the gates are tanh-ed on the device) and
 * the block-causal mask; each layer's post-RoPE K|V is written to the
 * cache. The last layer stops after its cache write (its output feeds
 * nothing). x_layers (device f32 [L][lp][H], or NULL) receives the hidden
 * state after each block 0 .. L-2. `layers` is a host array of L planes.
 * `workspace` (device, 256-byte aligned) must hold
 * qi21_workspace_bytes(g, lp). */
int qi21_prefill(const qi21_geom* g, const qi21_layer* layers, qi21_kvcache* cache,
                 const float* x_prefix, const float* mods0, float* x_layers, void* workspace,
                 size_t ws_bytes, void* stream);

/* Step (qwen_image21.rs, Qi21Dit::step_cpu, the block loop;
 * gpu_wgpu/qi21.rs, step): the target rows x_in (device f32 [n][H]) through
 * every block against [cached prefix, own rows], every key visible, with
 * the step modulation `mods` (device f32 [4H], raw). The result is written
 * to x_out (device f32 [n][H]; may equal x_in). x_layers (device f32
 * [L][n][H] or NULL) receives the hidden state after every block.
 * workspace >= qi21_workspace_bytes(g, n). */
int qi21_step(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* cache,
              const float* x_in, float* x_out, const float* mods, float* x_layers,
              void* workspace, size_t ws_bytes, void* stream);

/* Latent channels of the image tokens (qwen_image21.rs, Qi21Config::
 * in_channels / out_channels; the page's device path requires 64). */
#define QI21_LATENT_CHANNELS 64

/* Image embedding (qwen_image21.rs, Qi21Dit::embed_image; gpu_wgpu/qi21.rs,
 * zi_embed): x[n][dim] = tok[n][64] * w_in^T, no bias. tok device f32
 * [n][64], w_in device f32 [dim][64] (img_in.weight), x device f32 [n][dim].
 * in_ch must be 64; dim % 4 == 0. */
int qi21_embed(int32_t n, int32_t dim, int32_t in_ch, const float* tok, const float* w_in, float* x,
               void* stream);

/* Final layer (qwen_image21.rs, Qi21Dit::step_cpu after the blocks;
 * gpu_wgpu/qi21.rs, zi_final): out[n][64] = (LN(x) * (1 + final_scale)) *
 * w_out^T, affine-free LN with biased variance, no bias. x device f32
 * [n][dim], final_scale device f32 [dim] (raw, the norm_out scale of the
 * step), w_out device f32 [64][dim] (proj_out.weight), out device f32
 * [n][64]. out_ch must be 64; dim % 64 == 0. */
int qi21_final(int32_t n, int32_t dim, int32_t out_ch, float eps, const float* x,
               const float* final_scale, const float* w_out, float* out, void* stream);

/* One whole denoiser call of `nseq` (1..8) sequences sharing the target
 * size (qwen_image21.rs, Qi21Dit::step / step_cpu; gpu_wgpu/qi21.rs, step):
 * latent tokens tok (device f32 [nseq*n][64]) -> embed -> the blocks against
 * each sequence's cache (as qi21_step_batch) -> final layer -> velocity out
 * (device f32 [nseq*n][64]). mods device f32 [4H] raw; final_scale device
 * f32 [H] raw; w_in [H][64], w_out [64][H] device f32. The hidden state
 * lives in the workspace (>= qi21_workspace_bytes(g, nseq*n)). */
int qi21_denoise_batch(const qi21_geom* g, const qi21_layer* layers,
                       const qi21_kvcache* const* caches, int32_t nseq, const float* tok,
                       const float* w_in, const float* mods, const float* final_scale,
                       const float* w_out, float* out, void* workspace, size_t ws_bytes,
                       void* stream);

/* qi21_denoise_batch for one sequence. */
int qi21_denoise(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* cache,
                 const float* tok, const float* w_in, const float* mods, const float* final_scale,
                 const float* w_out, float* out, void* workspace, size_t ws_bytes, void* stream);

/* Size of the static device scratch behind qi21_step_noalloc: 32 MiB,
 * i.e. qi21_workspace_bytes(g, n) <= this bound (dim 4096 / mlp 12288: up to
 * 408 target rows; dim 256 / mlp 768: up to 6552). */
#define QI21_NOALLOC_SCRATCH_BYTES (32u << 20)

/* qi21_step without a caller workspace, for callers that cannot allocate
 * device memory: hosts whose device memory belongs to another allocator and
 * who have no buffer to lend, or serving loops under a no-allocation rule
 * after start-up (cudaMalloc may synchronise the device and stall every
 * other stream). The page has no counterpart; this is a library addition.
 * Same arguments and results as qi21_step without x_layers and workspace:
 * the workspace is a file-scope static device array of
 * QI21_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
 * the process exits. The entry point allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine); it returns QI21_ERR_WORKSPACE
 * when qi21_workspace_bytes(g, n) exceeds the scratch and QI21_ERR_STATE
 * while qi21_profile_enable(1) is on (profiling creates CUDA events).
 * The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture. All calls share the one scratch and it keeps
 * the last call's contents (nothing in it needs to start at zero: the step
 * writes every scratch byte it reads), so calls that overlap on the GPU --
 * concurrent streams, or two host threads -- race: serialise them. */
int qi21_step_noalloc(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* cache,
                      const float* x_in, float* x_out, const float* mods, void* stream);

/* Step of `nseq` (1..8) sequences that share the weights, the modulation
 * and the target row count n (a classifier-free-guidance pair: one latent,
 * two prompts). Sequence s has its own cache caches[s] (own prefix, own
 * target RoPE) and rows [s*n, (s+1)*n) of x_in/x_out (device f32
 * [nseq*n][H]); the GEMMs run on the stacked nseq*n rows and the attention
 * per sequence. x_layers is [L][nseq*n][H] or NULL.
 * workspace >= qi21_workspace_bytes(g, nseq*n). */
int qi21_step_batch(const qi21_geom* g, const qi21_layer* layers,
                    const qi21_kvcache* const* caches, int32_t nseq, const float* x_in,
                    float* x_out, const float* mods, float* x_layers, void* workspace,
                    size_t ws_bytes, void* stream);

#define QI21_TIMESTEP_CHANNELS 256

/* Bytes of the `work` scratch of qi21_timestep_mods: 2 * dim floats. */
#define QI21_TIMESTEP_WORK_BYTES(dim) ((size_t)(dim) * 8u)

/* The one shared modulation of a denoiser call from the model input t
 * (qwen_image21.rs, Qi21Dit::temb and Qi21Dit::mods; the page's pipeline
 * passes t = timestep / 1000, and the prefix's modulation is t = 0):
 *   e    = [cos a_i | sin a_i], a_i = 1000 t exp(-ln(10000) i / 128), i < 128
 *   temb = t_lin2 silu(t_lin1 e),   s = silu(temb)
 *   mods = modulation s  (raw [s1|g1|s2|g2], the input of qi21_step,
 *                         qi21_prefill and qi21_denoise),
 *   final_scale = norm_out s  (the input of qi21_final / qi21_denoise).
 * No biases. Device f32 weights in nn.Linear layout, 16-byte aligned:
 * t_lin1 [dim][256], t_lin2 [dim][dim], modulation [4 dim][dim], norm_out
 * [dim][dim]. work: device scratch of QI21_TIMESTEP_WORK_BYTES(dim) (h, temb
 * afterwards). Outputs mods f32 [4 dim], final_scale f32 [dim] (device;
 * must not overlap work or the weights). dim % 4 == 0, 4 <= dim <= 8192.
 * f32 arithmetic on the device (the page sums in f64 on the host). */
int qi21_timestep_mods(int32_t dim, float t, const float* t_lin1, const float* t_lin2,
                       const float* modulation, const float* norm_out, float* work, float* mods,
                       float* final_scale, void* stream);

/* Optional checks (process-wide flags). QI21_CHECK_FINITE is the page's
 * non-finite decline (gpu_wgpu/qi21.rs, step: a velocity with a NaN or an
 * infinity is refused, e.g. after an f16 overflow): with it set,
 * qi21_prefill scans the cache's K/V, qi21_step / qi21_step_batch the
 * hidden state x_out and qi21_denoise / qi21_denoise_batch the velocity
 * after the pass, synchronise the stream and return QI21_ERR_NONFINITE if
 * any value is NaN or infinite. The device buffers keep what was computed
 * (the pass already ran); the return code is the refusal. Off by default:
 * nothing synchronises. Do not set it while capturing a CUDA graph.
 * Returns the previous flags. */
#define QI21_CHECK_FINITE 1u
/* QI21_CHECK_AMAX is the page's AMAX probe (gpu_wgpu/qi21.rs, the
 * CMF_QI21_AMAX sites and read_amax): with it set, every f16 / bf16 pass
 * (prefill, step, denoiser call; not the FP8 variant) also raises, on the
 * device, the largest |value| stored at each of five 16-bit sites over all
 * of its layers: attn-in (the modulated LayerNorm before the qkv
 * projection), qkv (the panel after the qk norm and RoPE), attn-out (the
 * attention output), ffn-in (the second modulated LayerNorm) and hidden
 * (the SwiGLU rows). One extra read of each buffer per layer; nothing
 * synchronises. Flags are read when a pass is enqueued or recorded. */
#define QI21_CHECK_AMAX 2u
uint32_t qi21_set_checks(uint32_t flags);

/* The five AMAX maxima of the current device, in the site order above,
 * into out[5] (host), raised since the last reset; a NaN stored at a site
 * reads as NaN. Synchronises the device. reset != 0 zeroes them after the
 * read. */
int qi21_amax_read(float* out, int32_t reset);

/* Element types of qi21_count_nonfinite. */
#define QI21_ELEM_F16 2
#define QI21_ELEM_BF16 3
#define QI21_ELEM_F32 4

/* Number of NaN/infinite values among `count` device elements of x of type
 * elem_type (QI21_ELEM_F32, _F16 or _BF16; x aligned to its element).
 * Enqueues the scan on stream, synchronises the stream and writes the count
 * to *out_count (host). Calls from several host threads are serialised. */
int qi21_count_nonfinite(const void* x, size_t count, int32_t elem_type, uint64_t* out_count,
                         void* stream);

/* A recorded call (this library's addition: the page replays command
 * buffers it records once per prompt, gpu_wgpu/qi21.rs, Prog and
 * run_calls). qi21_graph_step_batch / qi21_graph_denoise_batch validate
 * their arguments exactly as qi21_step_batch / qi21_denoise_batch, then
 * record that call's launches into a CUDA graph (on a private stream; the
 * caller's streams are untouched, nothing runs); qi21_graph_launch replays
 * it on `stream` as one launch. The graph is bound to every pointer given
 * at capture (weights, caches, x / tokens, mods, final_scale, output,
 * workspace): between launches the caller may change the contents of those
 * buffers (new hidden states, the next timestep's mods) but not their
 * addresses, and must keep them alive until qi21_graph_free. Replays take
 * no profiling records and no finite checks; launches on one stream run in
 * order, and graphs sharing a workspace must not overlap in time. */
typedef struct qi21_graph qi21_graph;
int qi21_graph_step_batch(const qi21_geom* g, const qi21_layer* layers,
                          const qi21_kvcache* const* caches, int32_t nseq, const float* x_in,
                          float* x_out, const float* mods, void* workspace, size_t ws_bytes,
                          qi21_graph** out);
int qi21_graph_denoise_batch(const qi21_geom* g, const qi21_layer* layers,
                             const qi21_kvcache* const* caches, int32_t nseq, const float* tok,
                             const float* w_in, const float* mods, const float* final_scale,
                             const float* w_out, float* out_velocity, void* workspace,
                             size_t ws_bytes, qi21_graph** out);
int qi21_graph_launch(const qi21_graph* graph, void* stream);
void qi21_graph_free(qi21_graph* graph);

/* ------------------------------------------------------- FP8 variant ---- */
/* A generic W8A8 variant of the four projections (qkv, O, gate/up, down).
 * The page's device weights are 8- and 4-bit codecs whose formats it does
 * not give (gpu_wgpu/qi21.rs module notes), so this variant uses the OCP
 * FP8 E4M3 format: every weight row (output channel) and every activation
 * row entering a projection (xn, the attention output, the SwiGLU hidden
 * row) is scaled by a power of two 2^-e, e the smallest integer with
 * max|row| <= 448 2^e, and rounded to the nearest E4M3 value (ties to even,
 * saturating); the tensor cores multiply the codes (kind::f8f6f4, f32
 * accumulation) and the epilogue applies both scales. The attention, the
 * norms, the residual stream and the K/V cache are as in the f16 path. Not
 * the headline precision: its per-block error is set by the 3-bit mantissa
 * (about 2^-5 relative per operand element), not by the f16 bar. The FP8
 * entry points take f16 geometries only (QI21_ERR_GEOM for bf16). */

/* E4M3 planes of one layer: codes with the shapes of qi21_layer's planes
 * (wqkv [3H][H], wo [H][H], w13 [2I][H] interleaved, w2 [H][I]) and one f32
 * scale 2^e per row. */
typedef struct qi21_layer_fp8 {
  const uint8_t* wqkv;
  const uint8_t* wo;
  const uint8_t* w13;
  const uint8_t* w2;
  const float* s_qkv;
  const float* s_o;
  const float* s_13;
  const float* s_2;
  const float* norm_q;
  const float* norm_k;
} qi21_layer_fp8;

/* Bytes of one layer's E4M3 planes + scales (256-byte aligned pieces). */
size_t qi21_layer_fp8_bytes(const qi21_geom* g);

/* Quantise a layer's packed f16 planes (from qi21_pack_layer) into `mem`
 * (device, >= qi21_layer_fp8_bytes, 256-byte aligned; owned by the caller)
 * and fill *out (norm_q/norm_k are taken over). Asynchronous on stream. */
int qi21_pack_layer_fp8(const qi21_geom* g, const qi21_layer* planes, void* mem, size_t bytes,
                        qi21_layer_fp8* out, void* stream);

/* Workspace of the FP8 passes: the f16 layout plus one E4M3 row buffer
 * [rows][max(H, I)] and its row scales. */
size_t qi21_workspace_bytes_fp8(const qi21_geom* g, int32_t max_rows);

/* qi21_prefill / qi21_step_batch with the FP8 projections; same arguments,
 * layouts, errors and cache format (a cache prefilled either way can be
 * stepped either way). workspace >= qi21_workspace_bytes_fp8. */
int qi21_prefill_fp8(const qi21_geom* g, const qi21_layer_fp8* layers, qi21_kvcache* cache,
                     const float* x_prefix, const float* mods0, float* x_layers, void* workspace,
                     size_t ws_bytes, void* stream);
int qi21_step_batch_fp8(const qi21_geom* g, const qi21_layer_fp8* layers,
                        const qi21_kvcache* const* caches, int32_t nseq, const float* x_in,
                        float* x_out, const float* mods, float* x_layers, void* workspace,
                        size_t ws_bytes, void* stream);

/* The FP8 step recorded as a graph, as qi21_graph_step_batch (replay with
 * qi21_graph_launch, release with qi21_graph_free). */
int qi21_graph_step_batch_fp8(const qi21_geom* g, const qi21_layer_fp8* layers,
                              const qi21_kvcache* const* caches, int32_t nseq, const float* x_in,
                              float* x_out, const float* mods, void* workspace, size_t ws_bytes,
                              qi21_graph** out);

/* Reads and clears the device status word (0 = fine; nonzero = a kernel
 * gave up waiting). Synchronises the device. */
int qi21_device_status(void);

/* Self-test of the kernels' bounded waits: enqueues on `stream` one CTA
 * that waits on an mbarrier nothing arrives at, through the same bounded
 * wait the library's kernels use. After about 2 s the wait gives up, the
 * kernel raises the device status word and returns; the context stays
 * usable, so the next qi21_device_status() returns nonzero and the one
 * after it 0. Returns QI21_OK once enqueued. For tests of the failure
 * path; no other entry point is affected. */
int qi21_selftest_wait_timeout(void* stream);

/* Kernel classes of a pass, for qi21_profile_read. */
#define QI21_CLASS_ROWOP 0     /* modulated LayerNorm rows */
#define QI21_CLASS_QKV 1       /* qkv projection (tcgen05 GEMM, f16 panel) */
#define QI21_CLASS_QKROPE 2    /* qk RMSNorm + RoPE */
#define QI21_CLASS_KVCOPY 3    /* K|V cache write (prefill) */
#define QI21_CLASS_ATTENTION 4 /* flash attention */
#define QI21_CLASS_O 5         /* output projection + gated residual */
#define QI21_CLASS_GATEUP 6    /* gate/up projection + SwiGLU */
#define QI21_CLASS_DOWN 7      /* down projection + gated residual */
#define QI21_CLASS_MISC 8      /* modulation prep */
#define QI21_CLASS_EMBED 9     /* image embedding (qi21_denoise) */
#define QI21_CLASS_FINAL 10    /* final LN + proj_out (qi21_denoise) */
#define QI21_CLASS_TEMB 11     /* timestep conditioning (qi21_timestep_mods) */
#define QI21_CLASS_QUANT 12    /* E4M3 row quantisation (FP8 variant) */
#define QI21_NCLASS 13

/* Per-class device timing of the passes, the analogue of the page's
 * per-class step times (gpu_wgpu/qi21.rs, class_times). on != 0 starts
 * recording two CUDA events (on the launch stream) around every kernel a
 * pass launches and forgets earlier records; on == 0 stops. Host-side
 * overhead only; the kernels are unchanged. */
int qi21_profile_enable(int on);

/* Per class: ms = summed device time of the launches recorded since the
 * last enable/read (synchronises on them; NULL to skip), launches = kernels
 * launched by passes since the library was loaded (counted always).
 * Arrays of QI21_NCLASS. Clears the records. */
int qi21_profile_read(float* ms, int64_t* launches);

/* ------------------------------------------------- single operations ---- */
/* Kernel-level entry points (the same kernels the passes launch), for
 * per-operation parity checks and profiling. All pointers are device;
 * `dtype` (QI21_DTYPE_*) is the type of the 16-bit operands (T). */

/* xn = T(LN(x)(1 + scale)) per row; if y != NULL it first does
 * x += gate_t * y in place (gate_t = tanh of the raw gate, f32 [H]).
 * x f32 [rows][H], y f32 [rows][H], scale f32 [H], xn T [rows][H] (may be
 * NULL when y != NULL). qwen_image21.rs: Qi21Dit::norm_mod, gated_add;
 * gpu_wgpu/qi21.rs: qi_rowop. */
int qi21_op_rowop(int32_t dtype, int32_t rows, int32_t dim, float eps, float* x, const float* y,
                  const float* gate_t, const float* scale, void* xn, void* stream);

/* md = [s1 | tanh g1 | s2 | tanh g2] from raw mods, f32 [4H] each
 * (gpu_wgpu/qi21.rs, mods_dev). */
int qi21_op_mods_prep(int32_t dim, const float* mods, float* md, void* stream);

/* GEMM epilogues of qi21_op_gemm. */
#define QI21_EPI_F16 0    /* out T [M][ldo] = acc (T = the operands' type) */
#define QI21_EPI_F32 1    /* out f32 [M][ldo] = acc */
#define QI21_EPI_RESID 2  /* out f32 [M][ldo] += gate_t[col] * acc */
#define QI21_EPI_SWIGLU 3 /* out T [M][ldo]: col 64j+c = silu(acc[128j+c]) *
                             acc[128j+64+c] (N = 2*I on the interleaved plane) */

/* acc = A B^T with A T [M][K] (row stride K), B T [N][K] (row stride K),
 * f32 accumulation on the tensor cores; M >= 1, N % 128 == 0,
 * K % 64 == 0. */
int qi21_op_gemm(int32_t dtype, int32_t epi, int32_t M, int32_t N, int32_t K, const void* A,
                 const void* B, void* out, int32_t ldo, const float* gate_t, void* stream);

/* qi21_op_gemm with the K-split tail that the block passes use. When the
 * last wave of 256 x BN tile pairs fills only part of the GPU, each of its
 * tiles is split along K into a power-of-two number of parts (at most the
 * resident clusters / tail tiles and the k-blocks; at most 8 and BN/32,
 * or for QI21_EPI_SWIGLU at most 2) that run side by side; part p finishes
 * columns [p W, (p+1) W) of the tile (W = BN/P, for QI21_EPI_SWIGLU at
 * least one 128-column gate/up block, a part past the last block only
 * contributing its partial) after adding, in part order, every part's f32
 * partial. scratch: device, 256-byte aligned,
 * scratch_bytes >= 4096; its first 4096 bytes hold the merge flags (zeroed
 * by this call, on the stream), the rest the partials (tail tiles x parts x
 * BN x 1 KB); with too little room the call uses fewer parts, down to none.
 * *parts_out (host, may be NULL) receives the part count used (1: no
 * split). The results differ from qi21_op_gemm's only in the order of the
 * f32 additions of split tiles. Errors as qi21_op_gemm, plus
 * QI21_ERR_WORKSPACE for a null, short or misaligned scratch. */
int qi21_op_gemm_split(int32_t dtype, int32_t epi, int32_t M, int32_t N, int32_t K, const void* A,
                       const void* B, void* out, int32_t ldo, const float* gate_t, void* scratch,
                       size_t scratch_bytes, int32_t* parts_out, void* stream);

/* In place on the panel T [rows][3H] (q in columns [0, H), k in [H, 2H)):
 * per (row, head) RMSNorm * norm_q (or norm_k) over 128 values, then the
 * interleaved RoPE of pairs (2j, 2j+1) by the row's cos/sin [rows][64]
 * (qwen_image21.rs, Qi21Dit::qk_norm_rope; gpu_wgpu/qi21.rs, zi_qkrope). */
int qi21_op_qkrope(int32_t dtype, int32_t rows, int32_t heads, float eps, void* panel,
                   const float* norm_q, const float* norm_k, const float* cos_, const float* sin_,
                   void* stream);

/* FP8 variant, single operations. qi21_op_quant_rows: f16 a [rows][cols]
 * (cols % 8 == 0) -> E4M3 codes q [rows][cols] and qs[row] = 2^e.
 * qi21_op_rowop_fp8: LN(x)(1 + scale) of f32 x [rows][dim] -> codes
 * xq [rows][dim] and xs[row] = 2^e. qi21_op_gemm_fp8: acc = A B^T on codes
 * A [M][K], B [N][K] (N % 256 == 0, K % 128 == 0), times sa[row] sw[col],
 * then the epilogue (QI21_EPI_F32, _RESID or _SWIGLU, as qi21_op_gemm). */
int qi21_op_quant_rows(int32_t rows, int32_t cols, const void* a, void* q, float* qs, void* stream);
int qi21_op_rowop_fp8(int32_t rows, int32_t dim, float eps, const float* x, const float* scale,
                      void* xq, float* xs, void* stream);
int qi21_op_gemm_fp8(int32_t epi, int32_t M, int32_t N, int32_t K, const void* A, const float* sa,
                     const void* B, const float* sw, void* out, int32_t ldo, const float* gate,
                     void* stream);

/* cache [rows][2H] = panel columns [H, 3H), 16-bit elements of either
 * type (gpu_wgpu/qi21.rs, qi_kvcopy). */
int qi21_op_kvcopy(int32_t rows, int32_t dim, const void* panel, void* kv, void* stream);

/* Attention of nq query rows of the panel (q at columns [0, H) of panel
 * T [.][3H]) over n_pre keys from kv_pre (T [n_pre][2H], K then V; may be
 * NULL when n_pre == 0) followed by the panel's own keys rows [0, n_own)
 * (K at columns [H, 2H), V at [2H, 3H)). Query i sees keys [0, vis[i]) if
 * vis != NULL (uint32 [nq], non-decreasing, >= 1), else all n_pre + n_own
 * keys. out T [nq][H] (qwen_image21.rs, Qi21Dit::attention;
 * gpu_wgpu/qi21.rs, qi_flash). */
int qi21_op_attention(int32_t dtype, int32_t nq, int32_t heads, const void* panel,
                      const void* kv_pre, int32_t n_pre, int32_t n_own, const uint32_t* vis,
                      void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QI21_H */
