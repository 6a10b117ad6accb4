// The ends of a denoiser call: the image embedding before the blocks and
// the final modulated LayerNorm + output projection after them
// (qwen_image21.rs, Qi21Dit::embed_image and the end of Qi21Dit::step_cpu;
// gpu_wgpu/qi21.rs, zi_embed and zi_final). Both projections have 64
// latent channels on one side, so they are small f32 contractions run on
// the CUDA cores (f32 weights, as the page keeps for its device path).
// Also the timestep conditioning (qwen_image21.rs, Qi21Dit::temb and
// Qi21Dit::mods): matrix-vector products, bound by reading the f32 weights.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace qi21 {

constexpr int kLat = 64;        // latent channels
constexpr int kEmbRows = 32;    // token rows per CTA
constexpr int kEmbCols = 256;   // hidden columns per CTA (one per thread)

// x[r][c] = sum_k tok[r][k] w_in[c][k]; one thread per column c, the CTA's
// 32 token rows staged in shared memory (read as broadcasts).
__global__ void __launch_bounds__(kEmbCols) embed_kernel(int n, int dim, const float* __restrict__ tok,
                                                         const float* __restrict__ w_in,
                                                         float* __restrict__ x) {
  __shared__ float st[kEmbRows][kLat];
  const int r0 = blockIdx.x * kEmbRows;
  for (int i = threadIdx.x; i < kEmbRows * kLat; i += kEmbCols) {
    const int r = i / kLat, k = i % kLat;
    st[r][k] = (r0 + r < n) ? tok[static_cast<size_t>(r0 + r) * kLat + k] : 0.f;
  }
  __syncthreads();
  const int c = blockIdx.y * kEmbCols + threadIdx.x;
  if (c >= dim) return;
  float w[kLat];
  const float4* w4 = reinterpret_cast<const float4*>(w_in + static_cast<size_t>(c) * kLat);
#pragma unroll
  for (int i = 0; i < kLat / 4; ++i) {
    const float4 v = __ldg(w4 + i);
    w[4 * i] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
  const int rows = min(kEmbRows, n - r0);
  for (int r = 0; r < rows; ++r) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int k = 0; k < kLat; k += 4) {
      a0 = fmaf(st[r][k], w[k], a0);
      a1 = fmaf(st[r][k + 1], w[k + 1], a1);
      a2 = fmaf(st[r][k + 2], w[k + 2], a2);
      a3 = fmaf(st[r][k + 3], w[k + 3], a3);
    }
    x[static_cast<size_t>(r0 + r) * dim + c] = (a0 + a1) + (a2 + a3);
  }
}

cudaError_t launch_embed(int n, int dim, const float* tok, const float* w_in, float* x, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  dim3 grid((n + kEmbRows - 1) / kEmbRows, (dim + kEmbCols - 1) / kEmbCols);
  embed_kernel<<<grid, kEmbCols, 0, s>>>(n, dim, tok, w_in, x);
  return cudaGetLastError();
}

// out[r][o] = sum_c LN(x_r)[c] (1 + fs[c]) w_out[o][c] for 64 outputs.
// CTA = 32 rows x 64 outputs, 256 threads (2 rows x 4 outputs each). First
// the rows' mean and 1/std (two passes over each row in f32, one warp per
// 4 rows), then the contraction over dim in chunks of 64: the modulated
// LayerNorm is applied while the x chunk is staged (transposed) in shared
// memory next to the transposed w_out chunk.
constexpr int kFinRows = 32;
constexpr int kFinK = 64;

__global__ void __launch_bounds__(256) final_kernel(int n, int dim, float eps, const float* __restrict__ x,
                                                    const float* __restrict__ fs,
                                                    const float* __restrict__ w_out,
                                                    float* __restrict__ out) {
  __shared__ float mean_s[kFinRows], inv_s[kFinRows];
  __shared__ __align__(16) float at[kFinK][kFinRows + 4];  // at[k][r]
  __shared__ __align__(16) float bt[kFinK][kLat + 4];      // bt[k][o]
  const int r0 = blockIdx.x * kFinRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // row statistics
  for (int rr = 0; rr < kFinRows / 8; ++rr) {
    const int r = warp * (kFinRows / 8) + rr;
    float mean = 0.f, inv = 0.f;
    if (r0 + r < n) {
      const float* xr = x + static_cast<size_t>(r0 + r) * dim;
      float sm = 0.f;
      for (int c = lane * 4; c < dim; c += 128) {
        const float4 v = *reinterpret_cast<const float4*>(xr + c);
        sm += (v.x + v.y) + (v.z + v.w);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
      mean = sm / static_cast<float>(dim);
      float sq = 0.f;
      for (int c = lane * 4; c < dim; c += 128) {
        const float4 v = *reinterpret_cast<const float4*>(xr + c);
        const float a = v.x - mean, b = v.y - mean, cc = v.z - mean, d = v.w - mean;
        sq += (a * a + b * b) + (cc * cc + d * d);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      inv = rsqrtf(sq / static_cast<float>(dim) + eps);
    }
    if (lane == 0) {
      mean_s[r] = mean;
      inv_s[r] = inv;
    }
  }
  __syncthreads();
  const int tx = tid & 15;  // outputs 4 tx .. 4 tx + 3
  const int ty = tid >> 4;  // rows 2 ty, 2 ty + 1
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  for (int k0 = 0; k0 < dim; k0 += kFinK) {
    // stage LN(x)(1 + fs) for 32 rows x 64 columns (transposed)
    for (int i = tid; i < kFinRows * kFinK; i += 256) {
      const int r = i / kFinK, k = i % kFinK;
      float v = 0.f;
      if (r0 + r < n) v = (x[static_cast<size_t>(r0 + r) * dim + k0 + k] - mean_s[r]) * inv_s[r] * (1.f + fs[k0 + k]);
      at[k][r] = v;
    }
    for (int i = tid; i < kLat * kFinK; i += 256) {
      const int o = i / kFinK, k = i % kFinK;
      bt[k][o] = w_out[static_cast<size_t>(o) * dim + k0 + k];
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < kFinK; ++k) {
      const float2 a = *reinterpret_cast<const float2*>(&at[k][2 * ty]);
      const float4 b = *reinterpret_cast<const float4*>(&bt[k][4 * tx]);
      acc[0][0] = fmaf(a.x, b.x, acc[0][0]);
      acc[0][1] = fmaf(a.x, b.y, acc[0][1]);
      acc[0][2] = fmaf(a.x, b.z, acc[0][2]);
      acc[0][3] = fmaf(a.x, b.w, acc[0][3]);
      acc[1][0] = fmaf(a.y, b.x, acc[1][0]);
      acc[1][1] = fmaf(a.y, b.y, acc[1][1]);
      acc[1][2] = fmaf(a.y, b.z, acc[1][2]);
      acc[1][3] = fmaf(a.y, b.w, acc[1][3]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = r0 + 2 * ty + i;
    if (r < n)
      *reinterpret_cast<float4*>(out + static_cast<size_t>(r) * kLat + 4 * tx) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

cudaError_t launch_final(int n, int dim, float eps, const float* x, const float* fs, const float* w_out,
                         float* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  final_kernel<<<(n + kFinRows - 1) / kFinRows, 256, 0, s>>>(n, dim, eps, x, fs, w_out, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------ timestep ----
constexpr int kTsHalf = 128;  // the sinusoid has 2 * 128 channels

__device__ __forceinline__ float silu_f(float v) { return v / (1.f + expf(-v)); }

// h[r] = silu(sum_k t_lin1[r][k] e[k]) with e = [cos a_i | sin a_i],
// a_i = (1000 t) exp(-ln(10000) i / 128), all in f32. One warp per row;
// every CTA builds e in shared memory (128 exp + cos/sin pairs).
__global__ void __launch_bounds__(256) temb_in_kernel(int dim, float t, const float* __restrict__ w1,
                                                      float* __restrict__ h) {
  __shared__ __align__(16) float e[2 * kTsHalf];
  if (threadIdx.x < kTsHalf) {
    const float ts = 1000.f * t;
    const float f = expf(-logf(10000.f) * static_cast<float>(threadIdx.x) / static_cast<float>(kTsHalf));
    const float a = ts * f;
    e[threadIdx.x] = cosf(a);
    e[kTsHalf + threadIdx.x] = sinf(a);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 8 + warp;
  if (r >= dim) return;
  const float4* w4 = reinterpret_cast<const float4*>(w1 + static_cast<size_t>(r) * 2 * kTsHalf);
  const float4 a = __ldg(w4 + lane), b = __ldg(w4 + 32 + lane);
  const float4 ea = reinterpret_cast<const float4*>(e)[lane], eb = reinterpret_cast<const float4*>(e)[32 + lane];
  float acc = (a.x * ea.x + a.y * ea.y) + (a.z * ea.z + a.w * ea.w);
  acc += (b.x * eb.x + b.y * eb.y) + (b.z * eb.z + b.w * eb.w);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) h[r] = silu_f(acc);
}

// y = W v over two stacked weight blocks (rows [0, ra) of wa into ya, then
// rows [0, rb) of wb into yb), v = silu(x) if SILU else x, staged in shared
// memory. One warp per output row, eight 16-byte loads in flight per lane.
template <bool SILU>
__global__ void __launch_bounds__(256) gemv_kernel(int ra, int rb, int cols, const float* __restrict__ wa,
                                                   const float* __restrict__ wb, const float* __restrict__ x,
                                                   float* __restrict__ ya, float* __restrict__ yb) {
  extern __shared__ __align__(16) float v[];
  for (int c = threadIdx.x; c < cols; c += 256) v[c] = SILU ? silu_f(x[c]) : x[c];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int r = blockIdx.x * 8 + warp;
  if (r >= ra + rb) return;
  const float* w = r < ra ? wa + static_cast<size_t>(r) * cols : wb + static_cast<size_t>(r - ra) * cols;
  float* y = r < ra ? ya + r : yb + (r - ra);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  const float4* v4 = reinterpret_cast<const float4*>(v);
  const int n4 = cols / 4;
  float acc0 = 0.f, acc1 = 0.f;
  int c = lane;
  for (; c + 7 * 32 < n4; c += 8 * 32) {
    float4 q[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) q[u] = __ldg(w4 + c + u * 32);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 z = v4[c + u * 32];
      acc0 = fmaf(q[u].x, z.x, acc0);
      acc1 = fmaf(q[u].y, z.y, acc1);
      acc0 = fmaf(q[u].z, z.z, acc0);
      acc1 = fmaf(q[u].w, z.w, acc1);
    }
  }
  for (; c < n4; c += 32) {
    const float4 q = __ldg(w4 + c), z = v4[c];
    acc0 = fmaf(q.x, z.x, acc0);
    acc1 = fmaf(q.y, z.y, acc1);
    acc0 = fmaf(q.z, z.z, acc0);
    acc1 = fmaf(q.w, z.w, acc1);
  }
  float acc = acc0 + acc1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) *y = acc;
}

cudaError_t launch_timestep(int dim, float t, const float* t_lin1, const float* t_lin2, const float* modulation,
                            const float* norm_out, float* work, float* mods, float* final_scale,
                            cudaStream_t s) {
  const size_t smem = static_cast<size_t>(dim) * 4;
  float* h = work;
  float* temb = work + dim;
  temb_in_kernel<<<(dim + 7) / 8, 256, 0, s>>>(dim, t, t_lin1, h);
  gemv_kernel<false><<<(dim + 7) / 8, 256, smem, s>>>(dim, 0, dim, t_lin2, nullptr, h, temb, nullptr);
  gemv_kernel<true><<<(5 * dim + 7) / 8, 256, smem, s>>>(4 * dim, dim, dim, modulation, norm_out, temb, mods,
                                                         final_scale);
  return cudaGetLastError();
}

// ------------------------------------------------------- finite check ----
// Counts NaN/Inf values by their exponent bits (all ones), so no floating
// point is involved: f32 0x7f800000, f16 0x7c00, bf16 0x7f80. 16-byte loads
// over the aligned body, scalar loads over the unaligned head and the tail;
// one atomic per warp into a file-scope counter. KIND: 4 f32, 2 f16,
// 3 bf16.
static __device__ unsigned long long g_nonfinite;

__global__ void zero_count_kernel() { g_nonfinite = 0ull; }

template <int KIND>
__device__ __forceinline__ unsigned bad_elem(const uint8_t* p) {
  if (KIND == 4) return (*reinterpret_cast<const uint32_t*>(p) & 0x7f800000u) == 0x7f800000u;
  constexpr uint16_t m = KIND == 3 ? 0x7f80u : 0x7c00u;
  return (*reinterpret_cast<const uint16_t*>(p) & m) == m;
}

template <int KIND>
__global__ void __launch_bounds__(256) count_nonfinite_kernel(const uint8_t* __restrict__ x, size_t count,
                                                              size_t head, size_t nvec) {
  constexpr int EB = KIND == 4 ? 4 : 2;
  constexpr int kPer = 16 / EB;
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nth = static_cast<size_t>(gridDim.x) * blockDim.x;
  unsigned bad = 0;
  // elements [0, head) and [head + nvec * kPer, count) one by one
  const size_t tail0 = head + nvec * kPer;
  for (size_t i = tid; i < head + (count - tail0); i += nth) {
    const size_t e = i < head ? i : tail0 + (i - head);
    bad += bad_elem<KIND>(x + e * EB);
  }
  const uint4* v = reinterpret_cast<const uint4*>(x + head * EB);
  for (size_t i = tid; i < nvec; i += nth) {
    const uint4 q = v[i];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (KIND == 4) {
        bad += (w[k] & 0x7f800000u) == 0x7f800000u;
      } else {
        constexpr uint32_t m = KIND == 3 ? 0x7f80u : 0x7c00u;
        bad += (w[k] & m) == m;
        bad += (w[k] & (m << 16)) == (m << 16);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(&g_nonfinite, static_cast<unsigned long long>(bad));
}

cudaError_t count_nonfinite(const void* x, size_t count, int elem, unsigned long long* out, cudaStream_t s) {
  if (elem != 2 && elem != 3 && elem != 4) return cudaErrorInvalidValue;
  const int elem_bytes = elem == 4 ? 4 : 2;
  const uintptr_t a = reinterpret_cast<uintptr_t>(x);
  size_t head = ((16 - (a & 15)) & 15) / elem_bytes;
  if (head > count) head = count;
  const size_t nvec = (count - head) / (16 / elem_bytes);
  const size_t work = nvec + head + 1;
  const unsigned grid = static_cast<unsigned>(std::min<size_t>((work + 255) / 256, static_cast<size_t>(sm_count()) * 8));
  zero_count_kernel<<<1, 1, 0, s>>>();
  if (count > 0) {
    const uint8_t* xb = static_cast<const uint8_t*>(x);
    if (elem == 4)
      count_nonfinite_kernel<4><<<grid, 256, 0, s>>>(xb, count, head, nvec);
    else if (elem == 3)
      count_nonfinite_kernel<3><<<grid, 256, 0, s>>>(xb, count, head, nvec);
    else
      count_nonfinite_kernel<2><<<grid, 256, 0, s>>>(xb, count, head, nvec);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  unsigned long long h = 0;
  if ((e = cudaMemcpyFromSymbolAsync(&h, g_nonfinite, sizeof(h), 0, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return e;
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return e;
  *out = h;
  return cudaSuccess;
}

// --------------------------------------------------------------- amax ----
// Largest |value| stored at each 16-bit activation site of a pass (the
// page's CMF_QI21_AMAX probe, gpu_wgpu/qi21.rs, AMAX_SITES): one slot per
// site in a file-scope device array (each device has its own), raised with
// atomicMax on the f32 bit pattern (non-negative floats order as their
// bits; a NaN orders above every finite value and infinity).
static __device__ unsigned int g_amax[kAmaxSites];

template <bool BF>
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x, size_t rows, size_t cols,
                                                   size_t ld, int site) {
  const size_t n8 = cols / 8;  // 16-byte groups per row
  const size_t total = rows * n8;
  float m = 0.f;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = i / n8;
    const uint4 u = reinterpret_cast<const uint4*>(x + r * ld)[i - r * n8];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack2<BF>(w[k]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
      if (f.x != f.x || f.y != f.y) m = __uint_as_float(0x7fc00000u);  // keep a NaN visible
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = __uint_as_float(max(__float_as_uint(m), __shfl_xor_sync(0xffffffffu, __float_as_uint(m), o)));
  if ((threadIdx.x & 31) == 0) atomicMax(&g_amax[site], __float_as_uint(m));
}

cudaError_t launch_amax(const void* x, size_t rows, size_t cols, size_t ld, int dt, int site, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const size_t total = rows * (cols / 8);
  const unsigned grid = static_cast<unsigned>(std::min<size_t>((total + 255) / 256, static_cast<size_t>(sm_count()) * 8));
  const uint16_t* p = static_cast<const uint16_t*>(x);
  if (dt == DT_BF16)
    amax_kernel<true><<<grid, 256, 0, s>>>(p, rows, cols, ld, site);
  else
    amax_kernel<false><<<grid, 256, 0, s>>>(p, rows, cols, ld, site);
  return cudaGetLastError();
}

cudaError_t amax_read(float* out, bool reset) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  unsigned int v[kAmaxSites];
  if ((e = cudaMemcpyFromSymbol(v, g_amax, sizeof v)) != cudaSuccess) return e;
  memcpy(out, v, sizeof v);  // the slots hold f32 bit patterns
  if (reset) {
    const unsigned int z[kAmaxSites] = {};
    e = cudaMemcpyToSymbol(g_amax, z, sizeof z);
  }
  return e;
}

// ---------------------------------------------------- bounded-wait test ----
// One CTA waits on an mbarrier that nothing arrives at, with the same
// bounded wait every kernel of the library uses: it gives up after the
// limit, raises the status word and returns, leaving the context usable.
static __device__ unsigned int s_probe_status = 0;

unsigned int probe_status_read_clear() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, s_probe_status, sizeof v);
  cudaMemcpyToSymbol(s_probe_status, &z, sizeof z);
  return v;
}

__global__ void wait_probe_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // no thread ever arrives: the phase never completes
  mbar_wait(&bar, 0, &abort_flag, &s_probe_status);
}

cudaError_t launch_wait_probe(cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

}  // namespace qi21
