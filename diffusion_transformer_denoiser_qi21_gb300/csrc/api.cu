// C ABI of the library (include/qi21.h): argument validation, the layout
// index construction on the host, the per-prompt K/V cache object and the
// launch sequences of the prefill and the step.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/qi21.h"
#include "internal.h"
#include "ptx.cuh"

namespace qi21 {

static thread_local std::string t_err;

static int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int report_error(int code, const char* msg) { return fail(code, "%s", msg); }

static int cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? QI21_ERR_OOM : QI21_ERR_CUDA, "%s: %s", what,
              cudaGetErrorString(e));
}

#define QI21_CK(expr, what)                        \
  do {                                             \
    cudaError_t e_ = (expr);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

bool bind_primary_context() {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess;
}

int sm_count() {
  // initialised once per device, thread-safely, on first use there
  static PerDevice<int> once;
  const int* n = once.get([] {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 1;
  });
  return n ? *n : 1;
}

unsigned int read_and_clear_status() {
  cudaDeviceSynchronize();
  return gemm_status_read_clear() | attn_status_read_clear() | probe_status_read_clear();
}

// ---------------------------------------------------------- profiling ----
// Per-class device time: when enabled, every launch of a pass is bracketed
// by two CUDA events recorded on the launch stream; qi21_profile_read sums
// their elapsed times per class. Launches are counted whether or not the
// events are on.

struct ProfRec {
  int cls;
  cudaEvent_t a, b;
};

static std::mutex g_prof_mu;
static bool g_prof_on = false;
static std::vector<cudaEvent_t> g_prof_pool;
static std::vector<ProfRec> g_prof_recs;
static size_t g_prof_used = 0;
static std::atomic<long long> g_launches[QI21_NCLASS];

static cudaEvent_t prof_event() {
  if (g_prof_used == g_prof_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_prof_pool.push_back(e);
  }
  return g_prof_pool[g_prof_used++];
}

bool profiling_on() { return g_prof_on; }

// Set while this thread records a graph (qi21_graph_*): no profiling events
// and no synchronising checks go into a capture.
static thread_local bool t_capturing = false;

class ProfScope {
 public:
  ProfScope(int cls, cudaStream_t s) : cls_(cls), s_(s) {
    g_launches[cls].fetch_add(1, std::memory_order_relaxed);
    if (!g_prof_on || t_capturing) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    a_ = prof_event();
    if (a_) cudaEventRecord(a_, s_);
  }
  ~ProfScope() {
    if (!g_prof_on || a_ == nullptr) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEvent_t b = prof_event();
    if (b == nullptr) return;
    cudaEventRecord(b, s_);
    g_prof_recs.push_back(ProfRec{cls_, a_, b});
  }

 private:
  int cls_;
  cudaStream_t s_;
  cudaEvent_t a_ = nullptr;
};

// ------------------------------------------------------------- layout ----
// qwen_image21.rs: Seg, Qi21Layout::{total, prefix_len, validate, block_ids,
// positions}, rope_tables, and end[i] of Qi21Dit::prefill.

struct Layout {
  int total = 0, prefix = 0, target = 0;
};

static int layout_rows(const qi21_seg* segs, int nseg, Layout* out) {
  if (segs == nullptr || nseg <= 0) return fail(QI21_ERR_ARG, "empty layout");
  long long tot = 0;
  for (int i = 0; i < nseg; ++i) {
    const qi21_seg& s = segs[i];
    if (s.kind == QI21_SEG_TEXT) {
      if (s.a < 0) return fail(QI21_ERR_ARG, "segment %d: negative text length", i);
      tot += s.a;
    } else if (s.kind == QI21_SEG_IMAGE) {
      if (s.a < 0 || s.b < 0) return fail(QI21_ERR_ARG, "segment %d: negative image side", i);
      tot += static_cast<long long>(s.a) * s.b;
    } else {
      return fail(QI21_ERR_ARG, "segment %d: unknown kind %d", i, s.kind);
    }
    if (tot > (1LL << 30)) return fail(QI21_ERR_SHAPE, "layout too long");
  }
  const qi21_seg& last = segs[nseg - 1];
  if (last.kind != QI21_SEG_IMAGE || last.a <= 0 || last.b <= 0)
    return fail(QI21_ERR_SHAPE, "the layout must end with a non-empty target image block");
  out->total = static_cast<int>(tot);
  out->target = last.a * last.b;
  out->prefix = out->total - out->target;
  if (out->prefix == 0) return fail(QI21_ERR_SHAPE, "the prompt prefix is empty");
  return QI21_OK;
}

static void layout_positions(const qi21_seg* segs, int nseg, std::vector<int64_t>& pos,
                             std::vector<int32_t>& ids) {
  pos.clear();
  ids.clear();
  int64_t p = 0;
  int32_t bid = 0;
  for (int i = 0; i < nseg; ++i) {
    const qi21_seg& s = segs[i];
    if (s.kind == QI21_SEG_TEXT) {
      for (int r = 0; r < s.a; ++r) {
        pos.push_back(p);
        pos.push_back(p);
        pos.push_back(p);
        ids.push_back(-1);
        ++p;
      }
    } else {
      const int64_t h = s.a, w = s.b;
      for (int64_t r = 0; r < h; ++r)
        for (int64_t c = 0; c < w; ++c) {
          pos.push_back(p);
          pos.push_back(r - (h - h / 2));
          pos.push_back(c - (w - w / 2));
          ids.push_back(bid);
        }
      ++bid;
      p += h > w ? h : w;
    }
  }
}

static void prefix_vis(const std::vector<int32_t>& ids, int lp, std::vector<uint32_t>& vis) {
  vis.assign(lp, 0);
  for (int i = 0; i < lp; ++i) {
    if (ids[i] < 0) {
      vis[i] = static_cast<uint32_t>(i + 1);
    } else {
      int e = i + 1;
      while (e < lp && ids[e] == ids[i]) ++e;
      vis[i] = static_cast<uint32_t>(e);
    }
  }
}

// f32 frequencies 1/theta^(2i/d), f32 angle = f32(pos) * freq, f32 cos/sin.
static void rope_rows(const int64_t* pos, int rows, const int32_t axes[3], float theta, float* cs,
                      float* sn) {
  const int half = (axes[0] + axes[1] + axes[2]) / 2;
  std::vector<float> freq;
  std::vector<int> axis_of;
  for (int a = 0; a < 3; ++a)
    for (int i = 0; i < axes[a] / 2; ++i) {
      const float e = static_cast<float>(2 * i) / static_cast<float>(axes[a]);
      freq.push_back(1.0f / powf(theta, e));
      axis_of.push_back(a);
    }
  for (int r = 0; r < rows; ++r)
    for (int j = 0; j < half; ++j) {
      const float ang = static_cast<float>(pos[3 * r + axis_of[j]]) * freq[j];
      cs[static_cast<size_t>(r) * half + j] = cosf(ang);
      sn[static_cast<size_t>(r) * half + j] = sinf(ang);
    }
}

static int geom_check(const qi21_geom* g) {
  if (g == nullptr) return fail(QI21_ERR_ARG, "null geometry");
  if (g->head_dim != 128) return fail(QI21_ERR_GEOM, "head_dim %d (the kernels need 128)", g->head_dim);
  if (g->heads <= 0 || g->heads * g->head_dim != g->dim)
    return fail(QI21_ERR_GEOM, "heads*head_dim (%d*%d) != dim %d", g->heads, g->head_dim, g->dim);
  if (g->dim % 128 != 0 || g->dim < 128 || g->dim > 8192)
    return fail(QI21_ERR_GEOM, "dim %d (need a multiple of 128 in [128, 8192])", g->dim);
  if (g->mlp_hidden <= 0 || g->mlp_hidden % 64 != 0)
    return fail(QI21_ERR_GEOM, "mlp_hidden %d (need a positive multiple of 64)", g->mlp_hidden);
  if (g->layers <= 0) return fail(QI21_ERR_GEOM, "layers %d", g->layers);
  for (int a = 0; a < 3; ++a)
    if (g->axes[a] < 0 || g->axes[a] % 2 != 0)
      return fail(QI21_ERR_GEOM, "RoPE axis %d width %d must be even", a, g->axes[a]);
  if (g->axes[0] + g->axes[1] + g->axes[2] != g->head_dim)
    return fail(QI21_ERR_GEOM, "RoPE axes do not tile head_dim");
  if (!(g->eps > 0.f) || !(g->theta > 0.f)) return fail(QI21_ERR_GEOM, "eps and theta must be > 0");
  if (g->dtype != QI21_DTYPE_F16 && g->dtype != QI21_DTYPE_BF16)
    return fail(QI21_ERR_GEOM, "dtype %d (QI21_DTYPE_F16 or QI21_DTYPE_BF16)", g->dtype);
  return QI21_OK;
}

// The FP8 variant quantises f16 planes and f16 activation rows.
static int geom_check_fp8(const qi21_geom* g) {
  const int rc = geom_check(g);
  if (rc != QI21_OK) return rc;
  if (g->dtype != QI21_DTYPE_F16) return fail(QI21_ERR_GEOM, "the FP8 variant takes f16 geometries only");
  return QI21_OK;
}

// Element type of the geometry's 16-bit buffers for the finite scan.
static int elem_of(const qi21_geom* g) { return g->dtype == QI21_DTYPE_BF16 ? QI21_ELEM_BF16 : QI21_ELEM_F16; }

// -------------------------------------------------------------- sizes ----

static size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t x, xn, panel, att, hid, md, flags, q8, qs, total;
};

// fp8: the E4M3 activation rows (one buffer [M][max(H, I)] shared by xn,
// att and hid in turn) and their row scales, after the f16 layout.
static WsLayout ws_layout(const qi21_geom* g, int rows, bool fp8 = false) {
  const size_t M = static_cast<size_t>(rows), H = g->dim, I = g->mlp_hidden;
  WsLayout w{};
  size_t off = 0;
  w.x = off;
  off = align256(off + M * H * 4);
  w.xn = off;
  off = align256(off + M * H * 2);
  w.panel = off;
  off = align256(off + M * 3 * H * 2);
  w.att = off;
  off = align256(off + M * H * 2);
  w.hid = off;
  off = align256(off + M * I * 2);
  w.md = off;
  off = align256(off + 4 * H * 4);
  // merge flags of the GEMMs' K-split tails (zeroed at the start of a pass)
  w.flags = off;
  off = align256(off + kGemmFlagBytes);
  w.q8 = w.qs = 0;
  if (fp8) {
    w.q8 = off;
    off = align256(off + M * std::max(H, I));
    w.qs = off;
    off = align256(off + M * 4);
  }
  w.total = off;
  return w;
}

}  // namespace qi21

using namespace qi21;

// ---------------------------------------------------------------- cache ----

struct qi21_kvcache {
  qi21_geom g;
  std::vector<qi21_seg> segs;
  int lp = 0, n = 0;
  void* mem = nullptr;  // one allocation: kv, vis, tables
  void* kv = nullptr;  // [L][lp][2H] of the geometry's dtype
  uint32_t* vis = nullptr;
  float* cos_p = nullptr;
  float* sin_p = nullptr;
  float* cos_t = nullptr;
  float* sin_t = nullptr;
  bool filled = false;
};

extern "C" {

const char* qi21_last_error(void) { return t_err.c_str(); }

const char* qi21_version(void) { return "qi21-gb300 0.1 (sm_103a)"; }

int qi21_geom_check(const qi21_geom* g) { return geom_check(g); }

int qi21_layout_rows(const qi21_seg* segs, int32_t nseg, int32_t* total, int32_t* prefix,
                     int32_t* target) {
  Layout L;
  const int rc = layout_rows(segs, nseg, &L);
  if (rc != QI21_OK) return rc;
  if (total) *total = L.total;
  if (prefix) *prefix = L.prefix;
  if (target) *target = L.target;
  return QI21_OK;
}

int qi21_layout_indices(const qi21_seg* segs, int32_t nseg, const int32_t axes[3], float theta,
                        int64_t* pos, int32_t* block_ids, uint32_t* vis, float* cos_, float* sin_) {
  Layout L;
  int rc = layout_rows(segs, nseg, &L);
  if (rc != QI21_OK) return rc;
  if ((cos_ || sin_) && axes == nullptr) return fail(QI21_ERR_ARG, "null axes");
  if (cos_ || sin_) {
    for (int a = 0; a < 3; ++a)
      if (axes[a] < 0 || axes[a] % 2) return fail(QI21_ERR_GEOM, "RoPE axis widths must be even");
  }
  std::vector<int64_t> p;
  std::vector<int32_t> ids;
  layout_positions(segs, nseg, p, ids);
  if (pos) memcpy(pos, p.data(), p.size() * sizeof(int64_t));
  if (block_ids) memcpy(block_ids, ids.data(), ids.size() * sizeof(int32_t));
  if (vis) {
    std::vector<uint32_t> v;
    prefix_vis(ids, L.prefix, v);
    memcpy(vis, v.data(), v.size() * sizeof(uint32_t));
  }
  if (cos_ || sin_) {
    const int half = (axes[0] + axes[1] + axes[2]) / 2;
    std::vector<float> c(static_cast<size_t>(L.total) * half), s(c.size());
    rope_rows(p.data(), L.total, axes, theta, c.data(), s.data());
    if (cos_) memcpy(cos_, c.data(), c.size() * sizeof(float));
    if (sin_) memcpy(sin_, s.data(), s.size() * sizeof(float));
  }
  return QI21_OK;
}

size_t qi21_layer_plane_bytes(const qi21_geom* g) {
  if (geom_check(g) != QI21_OK) return 0;
  const size_t H = g->dim, I = g->mlp_hidden;
  return align256(3 * H * H * 2) + align256(H * H * 2) + align256(2 * I * H * 2) + align256(H * I * 2);
}

size_t qi21_workspace_bytes(const qi21_geom* g, int32_t max_rows) {
  if (geom_check(g) != QI21_OK || max_rows < 0) return 0;
  return ws_layout(g, max_rows).total;
}

size_t qi21_workspace_bytes_fp8(const qi21_geom* g, int32_t max_rows) {
  if (geom_check_fp8(g) != QI21_OK || max_rows < 0) return 0;
  return ws_layout(g, max_rows, true).total;
}

size_t qi21_layer_fp8_bytes(const qi21_geom* g) {
  if (geom_check_fp8(g) != QI21_OK) return 0;
  const size_t H = g->dim, I = g->mlp_hidden;
  return align256(3 * H * H) + align256(H * H) + align256(2 * I * H) + align256(H * I) + align256(3 * H * 4) +
         align256(H * 4) + align256(2 * I * 4) + align256(H * 4);
}

int qi21_pack_layer(const qi21_geom* g, const void* wq, const void* wk, const void* wv,
                    const void* wo, const void* wgate, const void* wup, const void* wdown,
                    const float* norm_q, const float* norm_k, void* planes, size_t plane_bytes,
                    qi21_layer* out, void* stream) {
  int rc = geom_check(g);
  if (rc != QI21_OK) return rc;
  if (!wq || !wk || !wv || !wo || !wgate || !wup || !wdown || !norm_q || !norm_k || !planes || !out)
    return fail(QI21_ERR_ARG, "null pointer");
  if (plane_bytes < qi21_layer_plane_bytes(g))
    return fail(QI21_ERR_SHAPE, "plane buffer %zu bytes, need %zu", plane_bytes,
                qi21_layer_plane_bytes(g));
  if (reinterpret_cast<uintptr_t>(planes) % 256)
    return fail(QI21_ERR_ARG, "planes must be 256-byte aligned");
  const size_t H = g->dim, I = g->mlp_hidden;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(planes);
  uint16_t* wqkv = reinterpret_cast<uint16_t*>(base);
  uint16_t* pwo = reinterpret_cast<uint16_t*>(base + align256(3 * H * H * 2));
  uint16_t* w13 = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(pwo) + align256(H * H * 2));
  uint16_t* w2 = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(w13) + align256(2 * I * H * 2));
  cudaError_t e;
  if ((e = cudaMemcpyAsync(wqkv, wq, H * H * 2, cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(wqkv + H * H, wk, H * H * 2, cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(wqkv + 2 * H * H, wv, H * H * 2, cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(pwo, wo, H * H * 2, cudaMemcpyDeviceToDevice, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(w2, wdown, H * I * 2, cudaMemcpyDeviceToDevice, s)) != cudaSuccess)
    return cuda_fail(e, "pack copies");
  e = launch_pack_w13(static_cast<int>(I), static_cast<int>(H), wgate, wup, w13, s);
  if (e != cudaSuccess) return cuda_fail(e, "pack_w13");
  out->wqkv = wqkv;
  out->wo = pwo;
  out->w13 = w13;
  out->w2 = w2;
  out->norm_q = norm_q;
  out->norm_k = norm_k;
  return QI21_OK;
}

int qi21_pack_layer_fp8(const qi21_geom* g, const qi21_layer* planes, void* mem, size_t bytes, qi21_layer_fp8* out,
                        void* stream) {
  int rc = geom_check_fp8(g);
  if (rc != QI21_OK) return rc;
  if (!planes || !mem || !out) return fail(QI21_ERR_ARG, "null pointer");
  if (!planes->wqkv || !planes->wo || !planes->w13 || !planes->w2 || !planes->norm_q || !planes->norm_k)
    return fail(QI21_ERR_ARG, "null plane");
  if (bytes < qi21_layer_fp8_bytes(g))
    return fail(QI21_ERR_SHAPE, "fp8 plane buffer %zu bytes, need %zu", bytes, qi21_layer_fp8_bytes(g));
  if (reinterpret_cast<uintptr_t>(mem) % 256) return fail(QI21_ERR_ARG, "mem must be 256-byte aligned");
  const size_t H = g->dim, I = g->mlp_hidden;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* p = static_cast<uint8_t*>(mem);
  auto take = [&](size_t n) {
    uint8_t* r = p;
    p += align256(n);
    return r;
  };
  uint8_t* qkv = take(3 * H * H);
  uint8_t* qo = take(H * H);
  uint8_t* q13 = take(2 * I * H);
  uint8_t* q2 = take(H * I);
  float* sqkv = reinterpret_cast<float*>(take(3 * H * 4));
  float* so = reinterpret_cast<float*>(take(H * 4));
  float* s13 = reinterpret_cast<float*>(take(2 * I * 4));
  float* s2 = reinterpret_cast<float*>(take(H * 4));
  {
    ProfScope ps(QI21_CLASS_QUANT, s);
    QI21_CK(launch_quant_rows(static_cast<int>(3 * H), static_cast<int>(H), static_cast<const __half*>(planes->wqkv),
                              H, qkv, H, sqkv, s),
            "quantise wqkv");
    QI21_CK(launch_quant_rows(static_cast<int>(H), static_cast<int>(H), static_cast<const __half*>(planes->wo), H, qo,
                              H, so, s),
            "quantise wo");
    QI21_CK(launch_quant_rows(static_cast<int>(2 * I), static_cast<int>(H), static_cast<const __half*>(planes->w13),
                              H, q13, H, s13, s),
            "quantise w13");
    QI21_CK(launch_quant_rows(static_cast<int>(H), static_cast<int>(I), static_cast<const __half*>(planes->w2), I, q2,
                              I, s2, s),
            "quantise w2");
  }
  out->wqkv = qkv;
  out->wo = qo;
  out->w13 = q13;
  out->w2 = q2;
  out->s_qkv = sqkv;
  out->s_o = so;
  out->s_13 = s13;
  out->s_2 = s2;
  out->norm_q = planes->norm_q;
  out->norm_k = planes->norm_k;
  return QI21_OK;
}

int qi21_kvcache_alloc(const qi21_geom* g, const qi21_seg* segs, int32_t nseg, qi21_kvcache** out) {
  int rc = geom_check(g);
  if (rc != QI21_OK) return rc;
  if (out == nullptr) return fail(QI21_ERR_ARG, "null output");
  *out = nullptr;
  Layout L;
  rc = layout_rows(segs, nseg, &L);
  if (rc != QI21_OK) return rc;
  std::vector<int64_t> p;
  std::vector<int32_t> ids;
  layout_positions(segs, nseg, p, ids);
  std::vector<uint32_t> vis;
  prefix_vis(ids, L.prefix, vis);
  std::vector<float> c(static_cast<size_t>(L.total) * 64), s(c.size());
  rope_rows(p.data(), L.total, g->axes, g->theta, c.data(), s.data());

  const size_t H = g->dim;
  const size_t kv_bytes = align256(static_cast<size_t>(g->layers) * L.prefix * 2 * H * 2);
  const size_t vis_bytes = align256(static_cast<size_t>(L.prefix) * 4);
  const size_t tp_bytes = align256(static_cast<size_t>(L.prefix) * 64 * 4);
  const size_t tt_bytes = align256(static_cast<size_t>(L.target) * 64 * 4);
  const size_t total = kv_bytes + vis_bytes + 2 * tp_bytes + 2 * tt_bytes;
  auto* cc = new qi21_kvcache();
  cc->g = *g;
  cc->segs.assign(segs, segs + nseg);
  cc->lp = L.prefix;
  cc->n = L.target;
  cudaError_t e = cudaMalloc(&cc->mem, total);
  if (e != cudaSuccess) {
    cudaGetLastError();
    delete cc;
    return cuda_fail(e, "kv cache allocation");
  }
  uint8_t* b = static_cast<uint8_t*>(cc->mem);
  cc->kv = b;
  cc->vis = reinterpret_cast<uint32_t*>(b + kv_bytes);
  cc->cos_p = reinterpret_cast<float*>(b + kv_bytes + vis_bytes);
  cc->sin_p = reinterpret_cast<float*>(b + kv_bytes + vis_bytes + tp_bytes);
  cc->cos_t = reinterpret_cast<float*>(b + kv_bytes + vis_bytes + 2 * tp_bytes);
  cc->sin_t = reinterpret_cast<float*>(b + kv_bytes + vis_bytes + 2 * tp_bytes + tt_bytes);
  const size_t lp64 = static_cast<size_t>(L.prefix) * 64;
  if ((e = cudaMemcpy(cc->vis, vis.data(), L.prefix * 4, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(cc->cos_p, c.data(), lp64 * 4, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(cc->sin_p, s.data(), lp64 * 4, cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(cc->cos_t, c.data() + lp64, static_cast<size_t>(L.target) * 64 * 4,
                      cudaMemcpyHostToDevice)) != cudaSuccess ||
      (e = cudaMemcpy(cc->sin_t, s.data() + lp64, static_cast<size_t>(L.target) * 64 * 4,
                      cudaMemcpyHostToDevice)) != cudaSuccess) {
    cudaFree(cc->mem);
    delete cc;
    return cuda_fail(e, "kv cache tables");
  }
  *out = cc;
  return QI21_OK;
}

void qi21_kvcache_free(qi21_kvcache* c) {
  if (c == nullptr) return;
  cudaDeviceSynchronize();
  cudaFree(c->mem);
  delete c;
}

int qi21_kvcache_info(const qi21_kvcache* c, int32_t* lp, int32_t* n, int32_t* layers) {
  if (c == nullptr) return fail(QI21_ERR_ARG, "null cache");
  if (lp) *lp = c->lp;
  if (n) *n = c->n;
  if (layers) *layers = c->g.layers;
  return QI21_OK;
}

int qi21_kvcache_layer(const qi21_kvcache* c, int32_t layer, const void** kv) {
  if (c == nullptr || kv == nullptr) return fail(QI21_ERR_ARG, "null pointer");
  if (layer < 0 || layer >= c->g.layers) return fail(QI21_ERR_STATE, "layer %d out of range", layer);
  *kv = static_cast<const uint16_t*>(c->kv) + static_cast<size_t>(layer) * c->lp * 2 * c->g.dim;
  return QI21_OK;
}

int qi21_device_status(void) { return static_cast<int>(read_and_clear_status()); }

int qi21_selftest_wait_timeout(void* stream) {
  QI21_CK(launch_wait_probe(static_cast<cudaStream_t>(stream)), "wait probe");
  return QI21_OK;
}

int qi21_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  g_prof_recs.clear();
  g_prof_used = 0;
  return QI21_OK;
}

int qi21_profile_read(float* ms, int64_t* launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (ms) {
    for (int c = 0; c < QI21_NCLASS; ++c) ms[c] = 0.f;
    for (const ProfRec& r : g_prof_recs) {
      float t = 0.f;
      if (cudaEventSynchronize(r.b) != cudaSuccess) return cuda_fail(cudaGetLastError(), "profile sync");
      if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) ms[r.cls] += t;
    }
  }
  if (launches)
    for (int c = 0; c < QI21_NCLASS; ++c) launches[c] = g_launches[c].load(std::memory_order_relaxed);
  g_prof_recs.clear();
  g_prof_used = 0;
  return QI21_OK;
}

}  // extern "C"

// --------------------------------------------------------------- passes ----

namespace {

bool same_geom(const qi21_geom& a, const qi21_geom& b) {
  return a.dim == b.dim && a.heads == b.heads && a.head_dim == b.head_dim &&
         a.mlp_hidden == b.mlp_hidden && a.layers == b.layers && a.axes[0] == b.axes[0] &&
         a.axes[1] == b.axes[1] && a.axes[2] == b.axes[2] && a.eps == b.eps && a.theta == b.theta &&
         a.dtype == b.dtype;
}

int check_layers(const qi21_geom* g, const qi21_layer* layers) {
  if (layers == nullptr) return fail(QI21_ERR_ARG, "null layers");
  for (int l = 0; l < g->layers; ++l) {
    const qi21_layer& w = layers[l];
    if (!w.wqkv || !w.wo || !w.w13 || !w.w2 || !w.norm_q || !w.norm_k)
      return fail(QI21_ERR_ARG, "layer %d: null plane", l);
    if ((reinterpret_cast<uintptr_t>(w.wqkv) | reinterpret_cast<uintptr_t>(w.wo) |
         reinterpret_cast<uintptr_t>(w.w13) | reinterpret_cast<uintptr_t>(w.w2)) % 16)
      return fail(QI21_ERR_ARG, "layer %d: planes must be 16-byte aligned", l);
  }
  return QI21_OK;
}

int check_layers_fp8(const qi21_geom* g, const qi21_layer_fp8* layers) {
  if (layers == nullptr) return fail(QI21_ERR_ARG, "null layers");
  for (int l = 0; l < g->layers; ++l) {
    const qi21_layer_fp8& w = layers[l];
    if (!w.wqkv || !w.wo || !w.w13 || !w.w2 || !w.s_qkv || !w.s_o || !w.s_13 || !w.s_2 || !w.norm_q || !w.norm_k)
      return fail(QI21_ERR_ARG, "layer %d: null plane", l);
    if ((reinterpret_cast<uintptr_t>(w.wqkv) | reinterpret_cast<uintptr_t>(w.wo) |
         reinterpret_cast<uintptr_t>(w.w13) | reinterpret_cast<uintptr_t>(w.w2) | reinterpret_cast<uintptr_t>(w.s_qkv) |
         reinterpret_cast<uintptr_t>(w.s_o) | reinterpret_cast<uintptr_t>(w.s_13) | reinterpret_cast<uintptr_t>(w.s_2)) %
        16)
      return fail(QI21_ERR_ARG, "layer %d: planes and scales must be 16-byte aligned", l);
  }
  return QI21_OK;
}


// Optional checks of qi21_set_checks (process-wide flags).
std::atomic<uint32_t> g_checks{0};

// Buffers of a pass (workspace views; x may be the caller's x_out).
struct PassBufs {
  float* x;
  void* xn;     // dt [M][H]
  void* panel;  // dt [M][3H]
  void* att;    // dt [M][H]
  void* hid;    // dt [M][I]
  float* md;
  int* flags;   // K-split tail merge flags (kGemmFlagBytes)
  uint8_t* q8;  // FP8 pass: E4M3 activation rows (xn, att, hid in turn)
  float* qs;    // FP8 pass: their row scales
};

// Everything one layer launches, with its tensor maps already encoded.
struct LayerPlan {
  GemmPlan pq, po, p13, p2;
  AttnPlan at;
  void* kv;       // prefill: the layer's cache block (written by the qkv epilogue)
  bool has_attn;  // false for the prefill's last layer (stops after its cache write)
};

static void split_scratch(GemmPlan* p, void* part, size_t bytes, int* flags, int epoch) {
  p->part = part;
  p->part_bytes = bytes;
  p->flags = flags;
  p->epoch = epoch;
}

// Plans of every layer of a pass, encoded before the pass enqueues anything
// (so an encoding failure at any layer leaves the stream untouched). Exactly
// one of layers (16-bit planes) and l8 (the FP8 variant: E4M3 planes, every
// projection on row-quantised activations) is non-null.
int plan_pass(const qi21_geom* g, const qi21_layer* layers, const qi21_layer_fp8* l8, int M, bool prefill,
              qi21_kvcache* pcache, const qi21_kvcache* const* caches, int nseq, int n, const PassBufs& b,
              std::vector<LayerPlan>& plans) {
  const bool f8 = l8 != nullptr;
  const int H = g->dim, I = g->mlp_hidden, L = g->layers, dt = g->dtype;
  const float* g1 = b.md + H;
  const float* g2 = b.md + 3 * H;
  // 16-bit hid / panel bytes; the FP8 pass keeps its 16-bit buffers too
  const size_t hid_bytes = static_cast<size_t>(M) * I * 2;
  const size_t panel_bytes = static_cast<size_t>(M) * 3 * H * 2;
  RopeTables tabs{};
  if (prefill) {
    tabs.nsrc = 1;
    tabs.src[0] = RopeSrc{pcache->cos_p, pcache->sin_p, 0};
  } else {
    tabs.nsrc = nseq;
    for (int q = 0; q < nseq; ++q) tabs.src[q] = RopeSrc{caches[q]->cos_t, caches[q]->sin_t, q * n};
  }
  plans.resize(L);
  for (int l = 0; l < L; ++l) {
    LayerPlan& lp = plans[l];
    const bool last = (l + 1 == L);
    const float* norm_q = f8 ? l8[l].norm_q : layers[l].norm_q;
    const float* norm_k = f8 ? l8[l].norm_k : layers[l].norm_k;
    // qkv projection with the qk RMSNorm + RoPE fused into its epilogue (and,
    // in a prefill, the layer's K|V cache rows written by the same store)
    const int epi_qkv = prefill ? EPI_QKV_KV : EPI_QKV;
    if (f8)
      QI21_CK(make_gemm_plan_f8(&lp.pq, epi_qkv, M, 3 * H, H, b.q8, b.qs, l8[l].wqkv, l8[l].s_qkv, b.panel, 3 * H,
                                nullptr),
              "qkv plan");
    else
      QI21_CK(make_gemm_plan(&lp.pq, epi_qkv, dt, M, 3 * H, H, b.xn, layers[l].wqkv, b.panel, 3 * H, nullptr),
              "qkv plan");
    lp.kv = prefill ? static_cast<uint16_t*>(pcache->kv) + static_cast<size_t>(l) * pcache->lp * 2 * H : nullptr;
    // a prefill's K|V cache rows are written by the qkv epilogue itself
    lp.pq.qkv = QkvEpi{norm_q, norm_k, g->eps, H, tabs, lp.kv};
    split_scratch(&lp.pq, b.hid, hid_bytes, b.flags, 4 * l + 1);
    lp.has_attn = !(prefill && last);
    if (!lp.has_attn) break;
    AttnArgs aa{};
    aa.panel = b.panel;
    aa.panel_rows = M;
    aa.out = b.att;
    aa.heads = g->heads;
    aa.dt = dt;
    if (prefill) {
      aa.nseq = 1;
      aa.seq[0] = AttnSeq{nullptr, 0, 0, M, 0, M, pcache->vis};
    } else {
      aa.nseq = nseq;
      for (int q = 0; q < nseq; ++q) {
        const qi21_kvcache* c = caches[q];
        aa.seq[q] = AttnSeq{static_cast<const uint16_t*>(c->kv) + static_cast<size_t>(l) * c->lp * 2 * H, c->lp,
                            q * n, n, q * n, n, nullptr};
      }
    }
    QI21_CK(make_attn_plan(aa, &lp.at), "attention plan");
    if (f8) {
      QI21_CK(make_gemm_plan_f8(&lp.po, EPI_RESID, M, H, H, b.q8, b.qs, l8[l].wo, l8[l].s_o, b.x, H, g1), "o plan");
      QI21_CK(make_gemm_plan_f8(&lp.p13, EPI_SWIGLU, M, 2 * I, H, b.q8, b.qs, l8[l].w13, l8[l].s_13, b.hid, I,
                                nullptr),
              "w13 plan");
      QI21_CK(make_gemm_plan_f8(&lp.p2, EPI_RESID, M, H, I, b.q8, b.qs, l8[l].w2, l8[l].s_2, b.x, H, g2),
              "down plan");
    } else {
      QI21_CK(make_gemm_plan(&lp.po, EPI_RESID, dt, M, H, H, b.att, layers[l].wo, b.x, H, g1), "o plan");
      QI21_CK(make_gemm_plan(&lp.p13, EPI_SWIGLU, dt, M, 2 * I, H, b.xn, layers[l].w13, b.hid, I, nullptr),
              "w13 plan");
      QI21_CK(make_gemm_plan(&lp.p2, EPI_RESID, dt, M, H, I, b.hid, layers[l].w2, b.x, H, g2), "down plan");
    }
    // K-split tails: the partials go to a buffer the GEMM neither reads nor
    // writes (hid during qkv and o, the panel during gate/up and down)
    split_scratch(&lp.po, b.hid, hid_bytes, b.flags, 4 * l + 2);
    split_scratch(&lp.p13, b.panel, panel_bytes, b.flags, 4 * l + 3);
    split_scratch(&lp.p2, b.panel, panel_bytes, b.flags, 4 * l + 4);
  }
  return QI21_OK;
}

// NVTX range around the launches of one layer.
class LayerRange {
 public:
  LayerRange(bool prefill, int l) {
    char name[48];
    snprintf(name, sizeof name, "qi21 %s layer %d", prefill ? "prefill" : "step", l);
    nvtxRangePushA(name);
  }
  ~LayerRange() { nvtxRangePop(); }
};

// The launches of a planned pass, in order, on stream s.
int exec_pass(const qi21_geom* g, bool f8, int M, bool prefill, const PassBufs& b,
              const std::vector<LayerPlan>& plans, float* x_layers, cudaStream_t s) {
  const int H = g->dim, I = g->mlp_hidden, L = g->layers, dt = g->dtype;
  const float* s1 = b.md;
  const float* s2 = b.md + 2 * H;
  // the AMAX probe (QI21_CHECK_AMAX, 16-bit passes): largest |value| of a
  // site's rows x cols 16-bit buffer
  const bool amax = !f8 && (g_checks.load(std::memory_order_relaxed) & QI21_CHECK_AMAX);
  auto probe = [&](const void* buf, int cols, int ld, int site) -> int {
    if (!amax) return QI21_OK;
    ProfScope ps(QI21_CLASS_MISC, s);
    QI21_CK(launch_amax(buf, static_cast<size_t>(M), static_cast<size_t>(cols), static_cast<size_t>(ld), dt, site, s),
            "amax");
    return QI21_OK;
  };
  // the modulated LayerNorm of x (16-bit xn, or E4M3 rows + scales)
  auto ln = [&](const float* scale) -> int {
    {
      ProfScope ps(QI21_CLASS_ROWOP, s);
      if (f8)
        QI21_CK(launch_rowop_q8(M, H, g->eps, b.x, scale, b.q8, b.qs, s), "rowop q8");
      else
        QI21_CK(launch_rowop(M, H, g->eps, b.x, nullptr, nullptr, scale, b.xn, dt, s), "rowop");
    }
    return probe(b.xn, H, H, scale == s1 ? AMAX_ATTN_IN : AMAX_FFN_IN);
  };
  // f16 rows -> E4M3 rows + scales (FP8 pass: att and hid)
  auto quant = [&](const void* a, int cols) -> int {
    ProfScope ps(QI21_CLASS_QUANT, s);
    QI21_CK(launch_quant_rows(M, cols, static_cast<const __half*>(a), static_cast<size_t>(cols), b.q8,
                              static_cast<size_t>(cols), b.qs, s),
            "quantise rows");
    return QI21_OK;
  };
  int rc;
  // the K-split tails' merge flags start at zero; each GEMM of the pass
  // sets them to its own epoch
  QI21_CK(cudaMemsetAsync(b.flags, 0, kGemmFlagBytes, s), "flags reset");
  if ((rc = ln(s1)) != QI21_OK) return rc;
  for (int l = 0; l < L; ++l) {
    const LayerRange range(prefill, l);
    const LayerPlan& lp = plans[l];
    const bool last = (l + 1 == L);
    {
      ProfScope ps(QI21_CLASS_QKV, s);
      QI21_CK(launch_gemm(lp.pq, s), "qkv gemm");
    }
    if ((rc = probe(b.panel, 3 * H, 3 * H, AMAX_QKV)) != QI21_OK) return rc;
    if (!lp.has_attn) break;
    {
      ProfScope ps(QI21_CLASS_ATTENTION, s);
      QI21_CK(launch_attn_plan(lp.at, s), "attention");
    }
    if ((rc = probe(b.att, H, H, AMAX_ATTN_OUT)) != QI21_OK) return rc;
    if (f8 && (rc = quant(b.att, H)) != QI21_OK) return rc;
    {
      ProfScope ps(QI21_CLASS_O, s);
      QI21_CK(launch_gemm(lp.po, s), "o gemm");
    }
    if ((rc = ln(s2)) != QI21_OK) return rc;
    {
      ProfScope ps(QI21_CLASS_GATEUP, s);
      QI21_CK(launch_gemm(lp.p13, s), "gate/up gemm");
    }
    if ((rc = probe(b.hid, I, I, AMAX_HIDDEN)) != QI21_OK) return rc;
    if (f8 && (rc = quant(b.hid, I)) != QI21_OK) return rc;
    {
      ProfScope ps(QI21_CLASS_DOWN, s);
      QI21_CK(launch_gemm(lp.p2, s), "down gemm");
    }
    if (x_layers)
      QI21_CK(cudaMemcpyAsync(x_layers + static_cast<size_t>(l) * M * H, b.x,
                              static_cast<size_t>(M) * H * 4, cudaMemcpyDeviceToDevice, s),
              "x_layers copy");
    if (!last && (rc = ln(s1)) != QI21_OK) return rc;
  }
  return QI21_OK;
}

// Per-thread plan storage, reused across calls (no allocation per step once
// it has grown to the largest layer count seen).
thread_local std::vector<LayerPlan> t_plans;

int ws_bind(const qi21_geom* g, int M, void* ws, size_t ws_bytes, PassBufs* b, bool fp8 = false) {
  if (ws == nullptr) return fail(QI21_ERR_WORKSPACE, "null workspace");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(QI21_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const WsLayout w = ws_layout(g, M, fp8);
  if (ws_bytes < w.total) return fail(QI21_ERR_WORKSPACE, "workspace %zu bytes, need %zu", ws_bytes, w.total);
  uint8_t* base = static_cast<uint8_t*>(ws);
  b->x = reinterpret_cast<float*>(base + w.x);
  b->xn = base + w.xn;
  b->panel = base + w.panel;
  b->att = base + w.att;
  b->hid = base + w.hid;
  b->md = reinterpret_cast<float*>(base + w.md);
  b->flags = reinterpret_cast<int*>(base + w.flags);
  b->q8 = fp8 ? base + w.q8 : nullptr;
  b->qs = fp8 ? reinterpret_cast<float*>(base + w.qs) : nullptr;
  return QI21_OK;
}

std::mutex g_count_mu;

int count_bad(const void* x, size_t count, int eb, unsigned long long* bad, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_count_mu);
  QI21_CK(count_nonfinite(x, count, eb, bad, s), "finite check");
  return QI21_OK;
}

// The QI21_CHECK_FINITE refusal of what a pass wrote (no-op when off).
int finite_check(const void* x, size_t count, int eb, const char* what, cudaStream_t s) {
  if (t_capturing || !(g_checks.load(std::memory_order_relaxed) & QI21_CHECK_FINITE)) return QI21_OK;
  unsigned long long bad = 0;
  const int rc = count_bad(x, count, eb, &bad, s);
  if (rc != QI21_OK) return rc;
  if (bad) return fail(QI21_ERR_NONFINITE, "%s holds %llu non-finite values", what, bad);
  return QI21_OK;
}

// A validated and planned step (the plans are in t_plans).
struct StepCall {
  PassBufs b;
  int M = 0, n = 0;
};

// Validation and planning of qi21_step_batch (nothing enqueued).
int step_prepare(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* const* caches, int32_t nseq,
                 const float* x_in, float* x_out, const float* mods, void* workspace, size_t ws_bytes,
                 const qi21_layer_fp8* l8, StepCall* sc);
// The launches of a prepared step.
int step_enqueue(const qi21_geom* g, bool f8, const StepCall& sc, const float* x_in, float* x_out,
                 const float* mods, float* x_layers, cudaStream_t s);

// qi21_step_batch without the finite check (qi21_denoise_batch checks the
// velocity instead).
int step_batch_impl(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* const* caches, int32_t nseq,
                    const float* x_in, float* x_out, const float* mods, float* x_layers, void* workspace,
                    size_t ws_bytes, void* stream, const qi21_layer_fp8* l8 = nullptr) {
  StepCall sc;
  const int rc = step_prepare(g, layers, caches, nseq, x_in, x_out, mods, workspace, ws_bytes, l8, &sc);
  if (rc != QI21_OK) return rc;
  return step_enqueue(g, l8 != nullptr, sc, x_in, x_out, mods, x_layers, static_cast<cudaStream_t>(stream));
}

int prefill_impl(const qi21_geom* g, const qi21_layer* layers, const qi21_layer_fp8* l8, qi21_kvcache* cache,
                 const float* x_prefix, const float* mods0, float* x_layers, void* workspace, size_t ws_bytes,
                 void* stream) {
  int rc = geom_check(g);
  if (rc != QI21_OK) return rc;
  if (cache == nullptr || x_prefix == nullptr || mods0 == nullptr) return fail(QI21_ERR_ARG, "null pointer");
  if (!same_geom(*g, cache->g)) return fail(QI21_ERR_SHAPE, "the cache was made for another geometry");
  if ((rc = l8 ? check_layers_fp8(g, l8) : check_layers(g, layers)) != QI21_OK) return rc;
  const int M = cache->lp;
  PassBufs b;
  if ((rc = ws_bind(g, M, workspace, ws_bytes, &b, l8 != nullptr)) != QI21_OK) return rc;
  // every layer's maps, before anything is enqueued
  if ((rc = plan_pass(g, l8 ? nullptr : layers, l8, M, true, cache, nullptr, 1, 0, b, t_plans)) != QI21_OK)
    return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t H = g->dim;
  QI21_CK(cudaMemcpyAsync(b.x, x_prefix, static_cast<size_t>(M) * H * 4, cudaMemcpyDeviceToDevice, s),
          "x copy");
  {
    ProfScope ps(QI21_CLASS_MISC, s);
    QI21_CK(launch_mods_prep(g->dim, mods0, b.md, s), "mods prep");
  }
  rc = exec_pass(g, l8 != nullptr, M, true, b, t_plans, x_layers, s);
  if (rc != QI21_OK) return rc;
  cache->filled = true;
  return finite_check(cache->kv, static_cast<size_t>(g->layers) * M * 2 * H, elem_of(g), "the K/V cache", s);
}

}  // namespace

extern "C" {

uint32_t qi21_set_checks(uint32_t flags) { return g_checks.exchange(flags); }

int qi21_amax_read(float* out, int32_t reset) {
  if (out == nullptr) return fail(QI21_ERR_ARG, "null output");
  QI21_CK(amax_read(out, reset != 0), "amax read");
  return QI21_OK;
}

int qi21_count_nonfinite(const void* x, size_t count, int32_t elem_type, uint64_t* out_count, void* stream) {
  if (elem_type != QI21_ELEM_F16 && elem_type != QI21_ELEM_BF16 && elem_type != QI21_ELEM_F32)
    return fail(QI21_ERR_ARG, "elem_type %d (QI21_ELEM_F16, _BF16 or _F32)", elem_type);
  if (out_count == nullptr || (count > 0 && x == nullptr)) return fail(QI21_ERR_ARG, "null pointer");
  const int elem_bytes = elem_type == QI21_ELEM_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(x) % elem_bytes) return fail(QI21_ERR_ARG, "x not aligned to its element");
  unsigned long long bad = 0;
  const int rc = count_bad(x, count, elem_type, &bad, static_cast<cudaStream_t>(stream));
  if (rc != QI21_OK) return rc;
  *out_count = bad;
  return QI21_OK;
}

int qi21_prefill(const qi21_geom* g, const qi21_layer* layers, qi21_kvcache* cache,
                 const float* x_prefix, const float* mods0, float* x_layers, void* workspace,
                 size_t ws_bytes, void* stream) {
  return prefill_impl(g, layers, nullptr, cache, x_prefix, mods0, x_layers, workspace, ws_bytes, stream);
}

int qi21_prefill_fp8(const qi21_geom* g, const qi21_layer_fp8* layers, qi21_kvcache* cache, const float* x_prefix,
                     const float* mods0, float* x_layers, void* workspace, size_t ws_bytes, void* stream) {
  const int gc = geom_check_fp8(g);
  if (gc != QI21_OK) return gc;
  if (layers == nullptr) return fail(QI21_ERR_ARG, "null layers");
  return prefill_impl(g, nullptr, layers, cache, x_prefix, mods0, x_layers, workspace, ws_bytes, stream);
}

int qi21_step_batch_fp8(const qi21_geom* g, const qi21_layer_fp8* layers, const qi21_kvcache* const* caches,
                        int32_t nseq, const float* x_in, float* x_out, const float* mods, float* x_layers,
                        void* workspace, size_t ws_bytes, void* stream) {
  const int gc = geom_check_fp8(g);
  if (gc != QI21_OK) return gc;
  if (layers == nullptr) return fail(QI21_ERR_ARG, "null layers");
  const int rc =
      step_batch_impl(g, nullptr, caches, nseq, x_in, x_out, mods, x_layers, workspace, ws_bytes, stream, layers);
  if (rc != QI21_OK) return rc;
  return finite_check(x_out, static_cast<size_t>(nseq) * caches[0]->n * g->dim, QI21_ELEM_F32, "the hidden state",
                      static_cast<cudaStream_t>(stream));
}

int qi21_step_batch(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* const* caches,
                    int32_t nseq, const float* x_in, float* x_out, const float* mods, float* x_layers,
                    void* workspace, size_t ws_bytes, void* stream) {
  const int rc = step_batch_impl(g, layers, caches, nseq, x_in, x_out, mods, x_layers, workspace, ws_bytes, stream);
  if (rc != QI21_OK) return rc;
  return finite_check(x_out, static_cast<size_t>(nseq) * caches[0]->n * g->dim, QI21_ELEM_F32, "the hidden state",
                      static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

int step_prepare(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* const* caches, int32_t nseq,
                 const float* x_in, float* x_out, const float* mods, void* workspace, size_t ws_bytes,
                 const qi21_layer_fp8* l8, StepCall* sc) {
  int rc = geom_check(g);
  if (rc != QI21_OK) return rc;
  if (caches == nullptr || x_in == nullptr || x_out == nullptr || mods == nullptr)
    return fail(QI21_ERR_ARG, "null pointer");
  if (nseq < 1 || nseq > kMaxSeq) return fail(QI21_ERR_ARG, "nseq %d outside [1, %d]", nseq, kMaxSeq);
  int n = -1;
  for (int q = 0; q < nseq; ++q) {
    const qi21_kvcache* c = caches[q];
    if (c == nullptr) return fail(QI21_ERR_ARG, "null cache %d", q);
    if (!same_geom(*g, c->g)) return fail(QI21_ERR_SHAPE, "cache %d was made for another geometry", q);
    if (!c->filled) return fail(QI21_ERR_STATE, "cache %d has not been prefilled", q);
    if (n < 0) n = c->n;
    if (c->n != n) return fail(QI21_ERR_SHAPE, "caches disagree on the target rows (%d vs %d)", c->n, n);
  }
  if ((rc = l8 ? check_layers_fp8(g, l8) : check_layers(g, layers)) != QI21_OK) return rc;
  sc->n = n;
  sc->M = nseq * n;
  if ((rc = ws_bind(g, sc->M, workspace, ws_bytes, &sc->b, l8 != nullptr)) != QI21_OK) return rc;
  sc->b.x = x_out;
  // every layer's maps, before anything is enqueued
  return plan_pass(g, l8 ? nullptr : layers, l8, sc->M, false, nullptr, caches, nseq, n, sc->b, t_plans);
}

int step_enqueue(const qi21_geom* g, bool f8, const StepCall& sc, const float* x_in, float* x_out,
                 const float* mods, float* x_layers, cudaStream_t s) {
  const size_t H = g->dim;
  if (x_out != x_in)
    QI21_CK(cudaMemcpyAsync(x_out, x_in, static_cast<size_t>(sc.M) * H * 4, cudaMemcpyDeviceToDevice, s),
            "x copy");
  {
    ProfScope ps(QI21_CLASS_MISC, s);
    QI21_CK(launch_mods_prep(g->dim, mods, sc.b.md, s), "mods prep");
  }
  return exec_pass(g, f8, sc.M, false, sc.b, t_plans, x_layers, s);
}

}  // namespace

extern "C" {

int qi21_embed(int32_t n, int32_t dim, int32_t in_ch, const float* tok, const float* w_in, float* x,
               void* stream) {
  if (n < 0 || dim <= 0 || dim % 4) return fail(QI21_ERR_SHAPE, "n %d dim %d", n, dim);
  if (in_ch != QI21_LATENT_CHANNELS) return fail(QI21_ERR_GEOM, "in_ch %d (the kernels take 64)", in_ch);
  if (n == 0) return QI21_OK;
  if (!tok || !w_in || !x) return fail(QI21_ERR_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(w_in) | reinterpret_cast<uintptr_t>(x)) % 16)
    return fail(QI21_ERR_ARG, "w_in and x must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope ps(QI21_CLASS_EMBED, s);
  QI21_CK(launch_embed(n, dim, tok, w_in, x, s), "embed");
  return QI21_OK;
}

int qi21_final(int32_t n, int32_t dim, int32_t out_ch, float eps, const float* x, const float* final_scale,
               const float* w_out, float* out, void* stream) {
  if (n < 0 || dim <= 0 || dim % 64) return fail(QI21_ERR_SHAPE, "n %d dim %d", n, dim);
  if (out_ch != QI21_LATENT_CHANNELS) return fail(QI21_ERR_GEOM, "out_ch %d (the kernels take 64)", out_ch);
  if (!(eps > 0.f)) return fail(QI21_ERR_ARG, "eps must be > 0");
  if (n == 0) return QI21_OK;
  if (!x || !final_scale || !w_out || !out) return fail(QI21_ERR_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(QI21_ERR_ARG, "x and out must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope ps(QI21_CLASS_FINAL, s);
  QI21_CK(launch_final(n, dim, eps, x, final_scale, w_out, out, s), "final");
  return QI21_OK;
}

int qi21_timestep_mods(int32_t dim, float t, const float* t_lin1, const float* t_lin2, const float* modulation,
                       const float* norm_out, float* work, float* mods, float* final_scale, void* stream) {
  if (dim < 4 || dim % 4 || dim > 8192) return fail(QI21_ERR_SHAPE, "dim %d", dim);
  if (!std::isfinite(t)) return fail(QI21_ERR_ARG, "t is not finite");
  if (!t_lin1 || !t_lin2 || !modulation || !norm_out || !work || !mods || !final_scale)
    return fail(QI21_ERR_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(t_lin1) | reinterpret_cast<uintptr_t>(t_lin2) |
       reinterpret_cast<uintptr_t>(modulation) | reinterpret_cast<uintptr_t>(norm_out) |
       reinterpret_cast<uintptr_t>(work)) % 16)
    return fail(QI21_ERR_ARG, "weights and work must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ProfScope ps(QI21_CLASS_TEMB, s);
  QI21_CK(launch_timestep(dim, t, t_lin1, t_lin2, modulation, norm_out, work, mods, final_scale, s), "timestep");
  return QI21_OK;
}

int qi21_denoise_batch(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* const* caches,
                       int32_t nseq, const float* tok, const float* w_in, const float* mods,
                       const float* final_scale, const float* w_out, float* out, void* workspace,
                       size_t ws_bytes, void* stream) {
  int rc = geom_check(g);
  if (rc != QI21_OK) return rc;
  if (caches == nullptr || nseq < 1 || nseq > kMaxSeq) return fail(QI21_ERR_ARG, "caches / nseq");
  if (!tok || !w_in || !mods || !final_scale || !w_out || !out) return fail(QI21_ERR_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(w_in) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(QI21_ERR_ARG, "w_in and out must be 16-byte aligned");
  for (int q = 0; q < nseq; ++q)
    if (caches[q] == nullptr) return fail(QI21_ERR_ARG, "null cache %d", q);
  const int n = caches[0]->n;
  const int M = nseq * n;
  PassBufs b;
  if ((rc = ws_bind(g, M, workspace, ws_bytes, &b)) != QI21_OK) return rc;
  // the whole step is validated and planned before anything is enqueued;
  // the embedding and the final layer take arguments checked above
  StepCall sc;
  if ((rc = step_prepare(g, layers, caches, nseq, b.x, b.x, mods, workspace, ws_bytes, nullptr, &sc)) != QI21_OK)
    return rc;
  if ((rc = qi21_embed(M, g->dim, QI21_LATENT_CHANNELS, tok, w_in, b.x, stream)) != QI21_OK) return rc;
  if ((rc = step_enqueue(g, false, sc, b.x, b.x, mods, nullptr, static_cast<cudaStream_t>(stream))) != QI21_OK)
    return rc;
  if ((rc = qi21_final(M, g->dim, QI21_LATENT_CHANNELS, g->eps, b.x, final_scale, w_out, out, stream)) != QI21_OK)
    return rc;
  return finite_check(out, static_cast<size_t>(M) * QI21_LATENT_CHANNELS, QI21_ELEM_F32, "the velocity",
                      static_cast<cudaStream_t>(stream));
}

int qi21_denoise(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* cache, const float* tok,
                 const float* w_in, const float* mods, const float* final_scale, const float* w_out, float* out,
                 void* workspace, size_t ws_bytes, void* stream) {
  if (cache == nullptr) return fail(QI21_ERR_ARG, "null cache");
  const qi21_kvcache* cs[1] = {cache};
  return qi21_denoise_batch(g, layers, cs, 1, tok, w_in, mods, final_scale, w_out, out, workspace, ws_bytes,
                            stream);
}

int qi21_step(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* cache,
              const float* x_in, float* x_out, const float* mods, float* x_layers, void* workspace,
              size_t ws_bytes, void* stream) {
  const qi21_kvcache* cs[1] = {cache};
  if (cache == nullptr) return fail(QI21_ERR_ARG, "null cache");
  return qi21_step_batch(g, layers, cs, 1, x_in, x_out, mods, x_layers, workspace, ws_bytes, stream);
}

// ------------------------------------------------------------ graphs ----
// A recorded call: the launches of one qi21_step_batch / qi21_denoise_batch
// captured into a CUDA graph on a private stream (no profiling events, no
// synchronising checks inside), then replayed as one graph launch.

}  // extern "C"

struct qi21_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

namespace {

template <class F>
int capture_graph(F&& record, qi21_graph** out) {
  if (out == nullptr) return fail(QI21_ERR_ARG, "null output");
  *out = nullptr;
  cudaStream_t cs = nullptr;
  QI21_CK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking), "capture stream");
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "begin capture");
  }
  t_capturing = true;
  const int rc = record(static_cast<void*>(cs));
  t_capturing = false;
  cudaGraph_t gr = nullptr;
  e = cudaStreamEndCapture(cs, &gr);
  cudaStreamDestroy(cs);
  if (rc != QI21_OK) {
    if (gr) cudaGraphDestroy(gr);
    return rc;
  }
  if (e != cudaSuccess) {
    if (gr) cudaGraphDestroy(gr);
    return cuda_fail(e, "end capture");
  }
  cudaGraphExec_t ex = nullptr;
  e = cudaGraphInstantiate(&ex, gr, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(gr);
    return cuda_fail(e, "graph instantiate");
  }
  auto* gg = new qi21_graph();
  gg->graph = gr;
  gg->exec = ex;
  *out = gg;
  return QI21_OK;
}

}  // namespace

extern "C" {

int qi21_graph_step_batch(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* const* caches,
                          int32_t nseq, const float* x_in, float* x_out, const float* mods, void* workspace,
                          size_t ws_bytes, qi21_graph** out) {
  return capture_graph(
      [&](void* cs) {
        return qi21_step_batch(g, layers, caches, nseq, x_in, x_out, mods, nullptr, workspace, ws_bytes, cs);
      },
      out);
}

int qi21_graph_step_batch_fp8(const qi21_geom* g, const qi21_layer_fp8* layers, const qi21_kvcache* const* caches,
                              int32_t nseq, const float* x_in, float* x_out, const float* mods, void* workspace,
                              size_t ws_bytes, qi21_graph** out) {
  return capture_graph(
      [&](void* cs) {
        return qi21_step_batch_fp8(g, layers, caches, nseq, x_in, x_out, mods, nullptr, workspace, ws_bytes, cs);
      },
      out);
}

int qi21_graph_denoise_batch(const qi21_geom* g, const qi21_layer* layers, const qi21_kvcache* const* caches,
                             int32_t nseq, const float* tok, const float* w_in, const float* mods,
                             const float* final_scale, const float* w_out, float* out_v, void* workspace,
                             size_t ws_bytes, qi21_graph** out) {
  return capture_graph(
      [&](void* cs) {
        return qi21_denoise_batch(g, layers, caches, nseq, tok, w_in, mods, final_scale, w_out, out_v, workspace,
                                  ws_bytes, cs);
      },
      out);
}

int qi21_graph_launch(const qi21_graph* gr, void* stream) {
  if (gr == nullptr || gr->exec == nullptr) return fail(QI21_ERR_ARG, "null graph");
  QI21_CK(cudaGraphLaunch(gr->exec, static_cast<cudaStream_t>(stream)), "graph launch");
  return QI21_OK;
}

void qi21_graph_free(qi21_graph* gr) {
  if (gr == nullptr) return;
  if (gr->exec) cudaGraphExecDestroy(gr->exec);
  if (gr->graph) cudaGraphDestroy(gr->graph);
  delete gr;
}

// ------------------------------------------------------ single operations --

static int dtype_check(int32_t dtype) {
  if (dtype != QI21_DTYPE_F16 && dtype != QI21_DTYPE_BF16) return fail(QI21_ERR_ARG, "dtype %d", dtype);
  return QI21_OK;
}

int qi21_op_rowop(int32_t dtype, int32_t rows, int32_t dim, float eps, float* x, const float* y, const float* gate_t,
                  const float* scale, void* xn, void* stream) {
  if (dtype_check(dtype) != QI21_OK) return QI21_ERR_ARG;
  if (rows < 0 || dim <= 0 || dim % 4 || dim > 8192) return fail(QI21_ERR_SHAPE, "rows %d dim %d", rows, dim);
  if (rows == 0) return QI21_OK;  // empty input: nothing to do
  if (x == nullptr || (y && !gate_t) || (xn && !scale) || (!y && !xn)) return fail(QI21_ERR_ARG, "null pointer");
  QI21_CK(launch_rowop(rows, dim, eps, x, y, gate_t, scale, xn, dtype, static_cast<cudaStream_t>(stream)), "rowop");
  return QI21_OK;
}

int qi21_op_mods_prep(int32_t dim, const float* mods, float* md, void* stream) {
  if (dim <= 0) return fail(QI21_ERR_SHAPE, "dim %d", dim);
  if (!mods || !md) return fail(QI21_ERR_ARG, "null pointer");
  QI21_CK(launch_mods_prep(dim, mods, md, static_cast<cudaStream_t>(stream)), "mods prep");
  return QI21_OK;
}

int qi21_op_gemm(int32_t dtype, int32_t epi, int32_t M, int32_t N, int32_t K, const void* A, const void* B,
                 void* out, int32_t ldo, const float* gate_t, void* stream) {
  if (dtype_check(dtype) != QI21_OK) return QI21_ERR_ARG;
  if (epi < 0 || epi > 3) return fail(QI21_ERR_ARG, "epilogue %d", epi);
  if (M < 0 || N <= 0 || K <= 0 || N % 128 || K % 64) return fail(QI21_ERR_SHAPE, "M %d N %d K %d", M, N, K);
  if (M == 0) return QI21_OK;
  if (!A || !B || !out || (epi == EPI_RESID && !gate_t)) return fail(QI21_ERR_ARG, "null pointer");
  const int cols = epi == EPI_SWIGLU ? N / 2 : N;
  if (ldo < cols || ldo % 8) return fail(QI21_ERR_SHAPE, "ldo %d", ldo);
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(QI21_ERR_ARG, "A, B and out must be 16-byte aligned");
  if (M == 0) return QI21_OK;
  GemmPlan p;
  QI21_CK(make_gemm_plan(&p, epi, dtype, M, N, K, A, B, out, ldo, gate_t), "gemm plan");
  QI21_CK(launch_gemm(p, static_cast<cudaStream_t>(stream)), "gemm");
  return QI21_OK;
}

int qi21_op_gemm_split(int32_t dtype, int32_t epi, int32_t M, int32_t N, int32_t K, const void* A, const void* B,
                       void* out, int32_t ldo, const float* gate_t, void* scratch, size_t scratch_bytes,
                       int32_t* parts_out, void* stream) {
  if (parts_out) *parts_out = 1;
  if (dtype_check(dtype) != QI21_OK) return QI21_ERR_ARG;
  if (epi < 0 || epi > 3) return fail(QI21_ERR_ARG, "epilogue %d", epi);
  if (M < 0 || N <= 0 || K <= 0 || N % 128 || K % 64) return fail(QI21_ERR_SHAPE, "M %d N %d K %d", M, N, K);
  if (M == 0) return QI21_OK;
  if (!A || !B || !out || (epi == EPI_RESID && !gate_t)) return fail(QI21_ERR_ARG, "null pointer");
  if (!scratch || scratch_bytes < kGemmFlagBytes) return fail(QI21_ERR_WORKSPACE, "scratch below %zu bytes", kGemmFlagBytes);
  if (reinterpret_cast<uintptr_t>(scratch) % 256) return fail(QI21_ERR_WORKSPACE, "scratch must be 256-byte aligned");
  const int cols = epi == EPI_SWIGLU ? N / 2 : N;
  if (ldo < cols || ldo % 8) return fail(QI21_ERR_SHAPE, "ldo %d", ldo);
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(QI21_ERR_ARG, "A, B and out must be 16-byte aligned");
  GemmPlan p;
  QI21_CK(make_gemm_plan(&p, epi, dtype, M, N, K, A, B, out, ldo, gate_t), "gemm plan");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int parts = 1;
  split_scratch(&p, static_cast<uint8_t*>(scratch) + kGemmFlagBytes, scratch_bytes - kGemmFlagBytes,
                static_cast<int*>(scratch), 1);
  p.parts_out = &parts;
  QI21_CK(cudaMemsetAsync(scratch, 0, kGemmFlagBytes, s), "flags reset");
  QI21_CK(launch_gemm(p, s), "gemm");
  if (parts_out) *parts_out = parts;
  return QI21_OK;
}

int qi21_op_quant_rows(int32_t rows, int32_t cols, const void* a, void* q, float* qs, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 8) return fail(QI21_ERR_SHAPE, "rows %d cols %d", rows, cols);
  if (rows == 0) return QI21_OK;
  if (!a || !q || !qs) return fail(QI21_ERR_ARG, "null pointer");
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(q)) % 16)
    return fail(QI21_ERR_ARG, "a and q must be 16-byte aligned");
  QI21_CK(launch_quant_rows(rows, cols, static_cast<const __half*>(a), static_cast<size_t>(cols),
                            static_cast<uint8_t*>(q), static_cast<size_t>(cols), qs, static_cast<cudaStream_t>(stream)),
          "quantise rows");
  return QI21_OK;
}

int qi21_op_rowop_fp8(int32_t rows, int32_t dim, float eps, const float* x, const float* scale, void* xq, float* xs,
                      void* stream) {
  if (rows < 0 || dim <= 0 || dim % 4 || dim > 8192) return fail(QI21_ERR_SHAPE, "rows %d dim %d", rows, dim);
  if (rows == 0) return QI21_OK;
  if (!x || !scale || !xq || !xs) return fail(QI21_ERR_ARG, "null pointer");
  QI21_CK(launch_rowop_q8(rows, dim, eps, x, scale, static_cast<uint8_t*>(xq), xs, static_cast<cudaStream_t>(stream)),
          "rowop q8");
  return QI21_OK;
}

int qi21_op_gemm_fp8(int32_t epi, int32_t M, int32_t N, int32_t K, const void* A, const float* sa, const void* B,
                     const float* sw, void* out, int32_t ldo, const float* gate, void* stream) {
  if (epi != EPI_F32 && epi != EPI_RESID && epi != EPI_SWIGLU) return fail(QI21_ERR_ARG, "epilogue %d", epi);
  if (M < 0 || N <= 0 || K <= 0 || N % 256 || K % 128) return fail(QI21_ERR_SHAPE, "M %d N %d K %d", M, N, K);
  if (M == 0) return QI21_OK;
  if (!A || !sa || !B || !sw || !out || (epi == EPI_RESID && !gate)) return fail(QI21_ERR_ARG, "null pointer");
  const int cols = epi == EPI_SWIGLU ? N / 2 : N;
  if (ldo < cols || ldo % 8) return fail(QI21_ERR_SHAPE, "ldo %d", ldo);
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(sw)) % 16)
    return fail(QI21_ERR_ARG, "A, B, sw and out must be 16-byte aligned");
  GemmPlan p;
  QI21_CK(make_gemm_plan_f8(&p, epi, M, N, K, static_cast<const uint8_t*>(A), sa, static_cast<const uint8_t*>(B), sw,
                            out, ldo, gate),
          "gemm plan");
  QI21_CK(launch_gemm(p, static_cast<cudaStream_t>(stream)), "gemm fp8");
  return QI21_OK;
}

int qi21_op_qkrope(int32_t dtype, int32_t rows, int32_t heads, float eps, void* panel, const float* norm_q,
                   const float* norm_k, const float* cos_, const float* sin_, void* stream) {
  if (dtype_check(dtype) != QI21_OK) return QI21_ERR_ARG;
  if (rows < 0 || heads <= 0) return fail(QI21_ERR_SHAPE, "rows %d heads %d", rows, heads);
  if (rows == 0) return QI21_OK;
  if (!panel || !norm_q || !norm_k || !cos_ || !sin_) return fail(QI21_ERR_ARG, "null pointer");
  RopeTables t{};
  t.nsrc = 1;
  t.src[0] = RopeSrc{cos_, sin_, 0};
  QI21_CK(launch_qkrope(rows, heads, eps, panel, dtype, norm_q, norm_k, t, static_cast<cudaStream_t>(stream)),
          "qkrope");
  return QI21_OK;
}

int qi21_op_kvcopy(int32_t rows, int32_t dim, const void* panel, void* kv, void* stream) {
  if (rows < 0 || dim <= 0 || dim % 8) return fail(QI21_ERR_SHAPE, "rows %d dim %d", rows, dim);
  if (rows == 0) return QI21_OK;
  if (!panel || !kv) return fail(QI21_ERR_ARG, "null pointer");
  QI21_CK(launch_kvcopy(rows, dim, panel, kv, static_cast<cudaStream_t>(stream)), "kvcopy");
  return QI21_OK;
}

int qi21_op_attention(int32_t dtype, int32_t nq, int32_t heads, const void* panel, const void* kv_pre, int32_t n_pre,
                      int32_t n_own, const uint32_t* vis, void* out, void* stream) {
  if (dtype_check(dtype) != QI21_OK) return QI21_ERR_ARG;
  if (nq < 0 || heads <= 0 || n_pre < 0 || n_own < 0) return fail(QI21_ERR_SHAPE, "bad sizes");
  if (nq > n_own) return fail(QI21_ERR_SHAPE, "nq %d > own rows %d (queries are panel rows)", nq, n_own);
  if (nq == 0) return QI21_OK;
  if (!panel || !out || (n_pre > 0 && !kv_pre)) return fail(QI21_ERR_ARG, "null pointer");
  AttnArgs a{};
  a.panel = panel;
  a.panel_rows = n_own;
  a.out = out;
  a.heads = heads;
  a.dt = dtype;
  a.nseq = 1;
  a.seq[0] = AttnSeq{kv_pre, n_pre, 0, nq, 0, n_own, vis};
  QI21_CK(launch_attention(a, static_cast<cudaStream_t>(stream)), "attention");
  return QI21_OK;
}

}  // extern "C"
