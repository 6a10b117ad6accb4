// Launchers shared between the kernel translation units and the C ABI
// (api.cu). Host-only declarations; no torch types anywhere.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace qi21 {

// 16-bit element type of the weight planes, the activation rows (xn, qkv
// panel, attention output, SwiGLU hidden rows) and the K/V cache; the
// residual stream is f32 either way (qi21_geom::dtype).
enum Dt : int { DT_F16 = 0, DT_BF16 = 1 };

// One-time set-up kept per CUDA device (kernel attributes, the SM count):
// the runtime applies function attributes per device, so a process that
// drives several devices initialises each on its first call there.
constexpr int kMaxDevices = 64;
template <class T>
class PerDevice {
 public:
  // The value of the current device, made by make() on its first use there
  // (thread-safe); nullptr if there is no usable current device.
  template <class F>
  const T* get(F&& make) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(once_[dev], [&] { val_[dev] = make(); });
    return &val_[dev];
  }

 private:
  std::once_flag once_[kMaxDevices];
  T val_[kMaxDevices] = {};
};

// ------------------------------------------------------------ row kernels --

// md = [s1 | tanh g1 | s2 | tanh g2]
cudaError_t launch_mods_prep(int dim, const float* mods, float* md, cudaStream_t s);

// if y: x += gate_t * y; if xn: xn = dt(LN(x)(1 + scale))
cudaError_t launch_rowop(int rows, int dim, float eps, float* x, const float* y,
                         const float* gate_t, const float* scale, void* xn, int dt, cudaStream_t s);

// Per-row RoPE table source: rows [row0, row0 + rows) use cos/sin + (r - row0)*64.
struct RopeSrc {
  const float* cos_;
  const float* sin_;
  int row0;
};
constexpr int kMaxSeq = 8;
struct RopeTables {
  int nsrc;
  RopeSrc src[kMaxSeq];
};

// In place on panel dt [rows][3H]: q, k RMSNorm * w then interleaved RoPE.
cudaError_t launch_qkrope(int rows, int heads, float eps, void* panel, int dt, const float* norm_q,
                          const float* norm_k, const RopeTables& tabs, cudaStream_t s);

// kv [rows][2H] = panel[:, H:3H] (16-bit elements)
cudaError_t launch_kvcopy(int rows, int dim, const void* panel, void* kv, cudaStream_t s);

// w13 interleave: dst [2I][H] from gate [I][H], up [I][H], 64-row blocks
// (16-bit elements).
cudaError_t launch_pack_w13(int inter, int dim, const void* gate, const void* up, void* dst,
                            cudaStream_t s);

// x[n][dim] = tok[n][64] w_in[dim][64]^T (f32)
cudaError_t launch_embed(int n, int dim, const float* tok, const float* w_in, float* x, cudaStream_t s);
// out[n][64] = (LN(x)(1 + fs)) w_out[64][dim]^T (f32)
// E4M3 row quantisation (the FP8 variant): LN(x)(1 + scale) -> codes, and
// f16 rows -> codes; xs / qs[row] = 2^e (dequantisation factor).
cudaError_t launch_rowop_q8(int rows, int dim, float eps, const float* x, const float* scale, uint8_t* xq,
                            float* xs, cudaStream_t s);
cudaError_t launch_quant_rows(int rows, int cols, const __half* a, size_t lda, uint8_t* q, size_t ldq, float* qs,
                              cudaStream_t s);
cudaError_t launch_timestep(int dim, float t, const float* t_lin1, const float* t_lin2, const float* modulation,
                            const float* norm_out, float* work, float* mods, float* final_scale, cudaStream_t s);
// Synchronous: zeroes the counter, scans on s, reads it back, syncs s.
// elem: 4 (f32), 2 (f16) or 3 (bf16, 2 bytes); x aligned to its element.
cudaError_t count_nonfinite(const void* x, size_t count, int elem, unsigned long long* out, cudaStream_t s);
cudaError_t launch_final(int n, int dim, float eps, const float* x, const float* fs, const float* w_out,
                         float* out, cudaStream_t s);

// AMAX probe: sites attn-in, qkv, attn-out, ffn-in, hidden. launch_amax
// raises slot `site` to max |x| over rows x cols 16-bit values (row stride
// ld, cols % 8 == 0, 16-byte aligned rows); amax_read synchronises the
// device, reads the slots (and zeroes them if reset).
constexpr int kAmaxSites = 5;
enum AmaxSite : int { AMAX_ATTN_IN = 0, AMAX_QKV = 1, AMAX_ATTN_OUT = 2, AMAX_FFN_IN = 3, AMAX_HIDDEN = 4 };
cudaError_t launch_amax(const void* x, size_t rows, size_t cols, size_t ld, int dt, int site, cudaStream_t s);
cudaError_t amax_read(float* out, bool reset);

// ------------------------------------------------------------------ GEMM ----

enum Epi : int { EPI_F16 = 0, EPI_F32 = 1, EPI_RESID = 2, EPI_SWIGLU = 3, EPI_QKV = 4, EPI_QKV_KV = 5 };

// Extra inputs of the EPI_QKV epilogue: per-head RMSNorm weights of q and k,
// epsilon, the model width and the RoPE tables of the rows.
struct QkvEpi {
  const float* norm_q;
  const float* norm_k;
  float eps;
  int H;
  RopeTables tabs;
  void* kv;  // EPI_QKV_KV (prefill): the layer's cache block [M][2H] (K then V), also written
};

struct GemmPlan {
  CUtensorMap tmA;  // A dt [M][K], box 64 x 128, 128B swizzle
  CUtensorMap tmB;  // B dt [N][K], box 64 x BN, 128B swizzle
  CUtensorMap tmX;  // EPI_RESID: x f32 [M][ldo], box 32 x 32, 128B swizzle
  int M, N, K, bn, epi, ldo;
  int dt;            // operand and 16-bit output type (f16 path); DT_F16 for FP8
  void* out;
  const float* gate;
  QkvEpi qkv;
  bool f8;           // E4M3 operands (tensor maps of bytes, box 128 x rows)
  const float* sa;   // FP8: per A row scale
  const float* sw;   // FP8: per B row scale
  // K-split tail (optional, set after make_gemm_plan*): scratch for the
  // partials of a partial last wave and the merge flags, which a launch sets
  // to `epoch` (>= 1; zero them before the first launch and give each launch
  // between two zeroings its own epoch)
  void* part;
  size_t part_bytes;
  int* flags;
  int epoch;
  int* parts_out;  // optional (host): the part count a launch used (1: no split)
};

// K-split tail limits: parts per tail tile, flag bytes (ints: tail tiles x
// parts x 8), and the partial bytes of `tail_tiles` tiles split in `parts`
// (one BN x 32 f32 slab per tile, part, CTA and epilogue warp).
constexpr int kMaxKParts = 8;
constexpr size_t kGemmFlagBytes = 4096;
size_t gemm_split_bytes(int bn, int tail_tiles, int parts);

// Encode the tensor maps of C = A B^T with A, B of type dt. Returns
// cudaSuccess or an error; launches nothing.
cudaError_t make_gemm_plan(GemmPlan* p, int epi, int dt, int M, int N, int K, const void* A,
                           const void* B, void* out, int ldo, const float* gate);
// The FP8 form: A, B E4M3 codes [M][K], [N][K] (row pitch K bytes), the
// accumulator scaled by sa[row] sw[col]; N % 256 == 0, K % 128 == 0.
cudaError_t make_gemm_plan_f8(GemmPlan* p, int epi, int M, int N, int K, const uint8_t* A, const float* sa,
                              const uint8_t* B, const float* sw, void* out, int ldo, const float* gate);
cudaError_t launch_gemm(const GemmPlan& p, cudaStream_t s);

// -------------------------------------------------------------- attention --

struct AttnSeq {
  const void* kv_pre;  // [n_pre][2H] K then V (dt), or null
  int n_pre;
  int q_row0;    // first query row in the panel / output
  int nq;        // query rows
  int own_row0;  // first own-key row in the panel
  int n_own;     // own keys
  const uint32_t* vis;  // [nq] leading-run visibility, or null (all keys)
};

struct AttnArgs {
  const void* panel;  // [panel_rows][3H] dt: q at 0, k at H, v at 2H
  int panel_rows;
  void* out;          // [.][H] dt
  int heads;
  int dt;
  int nseq;
  AttnSeq seq[kMaxSeq];
};

// Kernel parameters of one attention launch (tensor maps encoded).
struct AttnTcSeq {
  CUtensorMap kvmap;  // cache [n_pre][2H], box 64 x 64 (unused if n_pre == 0)
  const uint32_t* vis;
  int n_pre, pad_end, q_row0, nq, own_row0, n_own;
};

struct AttnTcParams {
  CUtensorMap panel;     // [rows][3H], box 64 x 128 (Q)
  CUtensorMap panel_kv;  // same, box 64 x 64 (K, V)
  void* out;
  int H;
  float scale_log2;
  AttnTcSeq seq[kMaxSeq];
};

struct AttnPlan {
  AttnTcParams prm;
  int dt;
  int gx, gy, gz;  // grid; gx == 0: nothing to launch
};

// Encode the maps of an attention launch (launches nothing), then launch.
cudaError_t make_attn_plan(const AttnArgs& a, AttnPlan* p);
cudaError_t launch_attn_plan(const AttnPlan& p, cudaStream_t s);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t s);

// --------------------------------------------------------------- device ----

int sm_count();
// Makes the current device's primary context current on a calling thread
// that has none yet (what the first runtime call of a thread does), for
// driver calls that need one (tensor-map encoding). True on success.
bool bind_primary_context();
// Sets the thread-local error text of qi21_last_error and returns code.
int report_error(int code, const char* msg);
// True while qi21_profile_enable(1) is in force (launches create events).
bool profiling_on();
// Each translation unit whose kernels wait on mbarriers keeps its own device
// status word; these read and clear them (after a device synchronise).
unsigned int gemm_status_read_clear();
unsigned int attn_status_read_clear();
unsigned int probe_status_read_clear();
cudaError_t launch_wait_probe(cudaStream_t s);
unsigned int read_and_clear_status();

}  // namespace qi21
