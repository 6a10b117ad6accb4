// Row kernels of the block: the modulation prep, the fused gated residual +
// modulated LayerNorm, the per-head qk RMSNorm + interleaved RoPE, the K/V
// cache copy and the gate/up plane interleave. All HBM-bound: 128-bit
// coalesced loads/stores, one CTA per row where a row reduction is needed.
// The 16-bit rows are f16 or bf16 (the geometry's dtype, template BF).
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace qi21 {

// ------------------------------------------------------------ mods prep ----
// [s1 | g1 | s2 | g2] -> [s1 | tanh g1 | s2 | tanh g2] (gpu_wgpu/qi21.rs,
// mods_dev: the gate chunks tanh-ed once per pass).
__global__ void mods_prep_kernel(int dim, const float* __restrict__ mods, float* __restrict__ md) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 4 * dim) return;
  const int chunk = i / dim;
  const float v = mods[i];
  md[i] = (chunk == 1 || chunk == 3) ? tanhf(v) : v;
}

cudaError_t launch_mods_prep(int dim, const float* mods, float* md, cudaStream_t s) {
  const int n = 4 * dim;
  mods_prep_kernel<<<(n + 255) / 256, 256, 0, s>>>(dim, mods, md);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- rowop ----
// 256-thread CTAs, four per SM (two at NV = 8), each taking rows
// blockIdx.x + k gridDim.x
// with the next row's x loaded while the current one is reduced; a row is
// held in registers (NV float4 per thread, NV = dim / 1024 rounded up to a
// power of two, dim <= 8192):
//   if y:  x += gate_t * y            (qwen_image21.rs, Qi21Dit::gated_add)
//   if xn: xn = LN(x) (1 + scale) rounded to f16 / bf16 (Qi21Dit::norm_mod;
//          affine-free LN, biased variance, two passes over the registers
//          in f32)
constexpr int kRowThreads = 256;

__device__ __forceinline__ float block_sum_256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  return ((red[0] + red[1]) + (red[2] + red[3])) + ((red[4] + red[5]) + (red[6] + red[7]));
}

// Two f32 lanes in one 64-bit register pair and packed f32x2 arithmetic on
// them (one instruction for both lanes).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f32x2_split(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul_x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// resident CTAs per SM: four, two for the widest rows (register budget)
constexpr int rowop_ctas_per_sm(int nv) { return nv >= 8 ? 2 : 4; }

template <int NV, bool BF>
__global__ void __launch_bounds__(kRowThreads, rowop_ctas_per_sm(NV))
    rowop_kernel(int rows, int dim, float eps, float* __restrict__ x, const float* __restrict__ y,
                 const float* __restrict__ gate_t, const float* __restrict__ scale, uint16_t* __restrict__ xn) {
  __shared__ float red[8];
  const int nv = dim >> 2;
  // rows blockIdx.x, + gridDim.x, ...: the next row's x is loaded while
  // this row is reduced and written
  float4 v[NV], nx[NV];
  auto load_row = [&](int rw, float4 (&d)[NV]) {
    const float4* src = reinterpret_cast<const float4*>(x + static_cast<size_t>(rw) * dim);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int idx = threadIdx.x + j * kRowThreads;
      if (idx < nv) d[j] = src[idx];
    }
  };
  int row = blockIdx.x;
  if (row >= rows) return;
  load_row(row, v);
  while (true) {
    const int next = row + static_cast<int>(gridDim.x);
    if (next < rows) load_row(next, nx);
    float4* x4 = reinterpret_cast<float4*>(x + static_cast<size_t>(row) * dim);
    if (y != nullptr) {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int idx = threadIdx.x + j * kRowThreads;
        if (idx < nv) {
          const float4 b = reinterpret_cast<const float4*>(y + static_cast<size_t>(row) * dim)[idx];
          const float4 g = reinterpret_cast<const float4*>(gate_t)[idx];
          v[j].x = fmaf(g.x, b.x, v[j].x);
          v[j].y = fmaf(g.y, b.y, v[j].y);
          v[j].z = fmaf(g.z, b.z, v[j].z);
          v[j].w = fmaf(g.w, b.w, v[j].w);
          x4[idx] = v[j];
        }
      }
    }
    if (xn != nullptr) {
      // the row's values as pairs of lanes (x, y), (z, w) of each float4,
      // the arithmetic packed two lanes an instruction
      uint64_t s2 = 0ull;
#pragma unroll
      for (int j = 0; j < NV; ++j)
        if (threadIdx.x + j * kRowThreads < nv)
          s2 = add_x2(s2, add_x2(f32x2(v[j].x, v[j].y), f32x2(v[j].z, v[j].w)));
      const float2 sp = f32x2_split(s2);
      const float mean = block_sum_256(sp.x + sp.y, red) / static_cast<float>(dim);
      const uint64_t nm2 = f32x2(-mean, -mean);
      uint64_t q2 = 0ull;
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        if (threadIdx.x + j * kRowThreads < nv) {
          const uint64_t a = add_x2(f32x2(v[j].x, v[j].y), nm2), b = add_x2(f32x2(v[j].z, v[j].w), nm2);
          q2 = fma_x2(a, a, q2);
          q2 = fma_x2(b, b, q2);
        }
      }
      const float2 qp = f32x2_split(q2);
      const float inv = rsqrtf(block_sum_256(qp.x + qp.y, red) / static_cast<float>(dim) + eps);
      const uint64_t one2 = f32x2(1.f, 1.f), inv2 = f32x2(inv, inv);
      uint2* o2 = reinterpret_cast<uint2*>(xn + static_cast<size_t>(row) * dim);
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int idx = threadIdx.x + j * kRowThreads;
        if (idx < nv) {
          const float4 sc = __ldg(reinterpret_cast<const float4*>(scale) + idx);
          // (v - mean) inv (1 + scale)
          const float2 lo = f32x2_split(
              mul_x2(mul_x2(add_x2(f32x2(v[j].x, v[j].y), nm2), inv2), add_x2(f32x2(sc.x, sc.y), one2)));
          const float2 hi = f32x2_split(
              mul_x2(mul_x2(add_x2(f32x2(v[j].z, v[j].w), nm2), inv2), add_x2(f32x2(sc.z, sc.w), one2)));
          uint2 out;
          out.x = pack2<BF>(lo.x, lo.y);
          out.y = pack2<BF>(hi.x, hi.y);
          o2[idx] = out;
        }
      }
    }
    if (next >= rows) break;
    row = next;
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = nx[j];
  }
}

__device__ __forceinline__ float block_max_256(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  return fmaxf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])),
               fmaxf(fmaxf(red[4], red[5]), fmaxf(red[6], red[7])));
}

// The modulated LayerNorm with an E4M3 output (the FP8 variant's xn): the
// f32 row LN(x)(1 + scale) is scaled by 2^-e, e the row's power-of-two
// exponent, and rounded to E4M3 codes; xs[row] = 2^e.
template <int NV>
__global__ void __launch_bounds__(kRowThreads) rowop_q8_kernel(int dim, float eps, const float* __restrict__ x,
                                                               const float* __restrict__ scale,
                                                               uint8_t* __restrict__ xq, float* __restrict__ xs) {
  __shared__ float red[8];
  const size_t row = blockIdx.x;
  const int nv = dim >> 2;
  const float4* x4 = reinterpret_cast<const float4*>(x + row * dim);
  float4 v[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int idx = threadIdx.x + j * kRowThreads;
    if (idx < nv) v[j] = x4[idx];
  }
  float sm = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (threadIdx.x + j * kRowThreads < nv) sm += (v[j].x + v[j].y) + (v[j].z + v[j].w);
  const float mean = block_sum_256(sm, red) / static_cast<float>(dim);
  float sq = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    if (threadIdx.x + j * kRowThreads < nv) {
      const float a = v[j].x - mean, b = v[j].y - mean, c = v[j].z - mean, d = v[j].w - mean;
      sq += (a * a + b * b) + (c * c + d * d);
    }
  }
  const float inv = rsqrtf(block_sum_256(sq, red) / static_cast<float>(dim) + eps);
  float am = 0.f;
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int idx = threadIdx.x + j * kRowThreads;
    if (idx < nv) {
      const float4 sc = __ldg(reinterpret_cast<const float4*>(scale) + idx);
      v[j].x = (v[j].x - mean) * inv * (1.f + sc.x);
      v[j].y = (v[j].y - mean) * inv * (1.f + sc.y);
      v[j].z = (v[j].z - mean) * inv * (1.f + sc.z);
      v[j].w = (v[j].w - mean) * inv * (1.f + sc.w);
      am = fmaxf(am, fmaxf(fmaxf(fabsf(v[j].x), fabsf(v[j].y)), fmaxf(fabsf(v[j].z), fabsf(v[j].w))));
    }
  }
  const int e = e4m3_row_exp(block_max_256(am, red));
  const float r = ldexpf(1.f, -e);
  uint32_t* q4 = reinterpret_cast<uint32_t*>(xq + row * dim);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const int idx = threadIdx.x + j * kRowThreads;
    if (idx < nv) q4[idx] = e4m3x4(v[j].x * r, v[j].y * r, v[j].z * r, v[j].w * r);
  }
  if (threadIdx.x == 0) xs[row] = ldexpf(1.f, e);
}

cudaError_t launch_rowop_q8(int rows, int dim, float eps, const float* x, const float* scale, uint8_t* xq,
                            float* xs, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int per = (dim / 4 + kRowThreads - 1) / kRowThreads;
  if (per <= 1)
    rowop_q8_kernel<1><<<rows, kRowThreads, 0, s>>>(dim, eps, x, scale, xq, xs);
  else if (per <= 2)
    rowop_q8_kernel<2><<<rows, kRowThreads, 0, s>>>(dim, eps, x, scale, xq, xs);
  else if (per <= 4)
    rowop_q8_kernel<4><<<rows, kRowThreads, 0, s>>>(dim, eps, x, scale, xq, xs);
  else
    rowop_q8_kernel<8><<<rows, kRowThreads, 0, s>>>(dim, eps, x, scale, xq, xs);
  return cudaGetLastError();
}

// f16 rows -> E4M3 rows with a power-of-two scale per row (the FP8
// variant's att, hid and weight planes): q = e4m3(a 2^-e), qs[row] = 2^e.
// One 256-thread CTA per row, 8 halves per thread per step; the row is read
// twice (the second pass mostly from L1).
__global__ void __launch_bounds__(kRowThreads) quant_rows_kernel(int cols, const __half* __restrict__ a, size_t lda,
                                                                 uint8_t* __restrict__ q, size_t ldq,
                                                                 float* __restrict__ qs) {
  __shared__ float red[8];
  const size_t row = blockIdx.x;
  const uint4* a8 = reinterpret_cast<const uint4*>(a + row * lda);
  const int n8 = cols >> 3;
  float am = 0.f;
  for (int i = threadIdx.x; i < n8; i += kRowThreads) {
    const uint4 u = a8[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
      am = fmaxf(am, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  const int e = e4m3_row_exp(block_max_256(am, red));
  const float r = ldexpf(1.f, -e);
  uint2* q8 = reinterpret_cast<uint2*>(q + row * ldq);
  for (int i = threadIdx.x; i < n8; i += kRowThreads) {
    const uint4 u = a8[i];
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&u.z));
    const float2 f3 = __half22float2(*reinterpret_cast<const __half2*>(&u.w));
    q8[i] = make_uint2(e4m3x4(f0.x * r, f0.y * r, f1.x * r, f1.y * r), e4m3x4(f2.x * r, f2.y * r, f3.x * r, f3.y * r));
  }
  if (threadIdx.x == 0) qs[row] = ldexpf(1.f, e);
}

cudaError_t launch_quant_rows(int rows, int cols, const __half* a, size_t lda, uint8_t* q, size_t ldq, float* qs,
                              cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  quant_rows_kernel<<<rows, kRowThreads, 0, s>>>(cols, a, lda, q, ldq, qs);
  return cudaGetLastError();
}

template <bool BF>
static void rowop_go(int rows, int dim, float eps, float* x, const float* y, const float* gate_t,
                     const float* scale, uint16_t* xn, cudaStream_t s) {
  const int per = (dim / 4 + kRowThreads - 1) / kRowThreads;  // float4 per thread
  // all CTAs resident, each walking rows with a stride of the grid
  auto grid = [&](int nv) { return std::min(rows, rowop_ctas_per_sm(nv) * sm_count()); };
  if (per <= 1)
    rowop_kernel<1, BF><<<grid(1), kRowThreads, 0, s>>>(rows, dim, eps, x, y, gate_t, scale, xn);
  else if (per <= 2)
    rowop_kernel<2, BF><<<grid(2), kRowThreads, 0, s>>>(rows, dim, eps, x, y, gate_t, scale, xn);
  else if (per <= 4)
    rowop_kernel<4, BF><<<grid(4), kRowThreads, 0, s>>>(rows, dim, eps, x, y, gate_t, scale, xn);
  else
    rowop_kernel<8, BF><<<grid(8), kRowThreads, 0, s>>>(rows, dim, eps, x, y, gate_t, scale, xn);
}

cudaError_t launch_rowop(int rows, int dim, float eps, float* x, const float* y, const float* gate_t,
                         const float* scale, void* xn, int dt, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (dt != DT_F16 && dt != DT_BF16) return cudaErrorInvalidValue;
  uint16_t* o = static_cast<uint16_t*>(xn);
  if (dt == DT_BF16)
    rowop_go<true>(rows, dim, eps, x, y, gate_t, scale, o, s);
  else
    rowop_go<false>(rows, dim, eps, x, y, gate_t, scale, o, s);
  return cudaGetLastError();
}

// --------------------------------------------------------------- qkrope ----
// One 256-thread CTA per panel row; each warp takes head vectors of q then
// k (128 values = 4 per lane), RMSNorm over the 128 values (warp shuffle),
// the weight, then rotates the pairs (2j, 2j+1) by the row's angle j
// (qwen_image21.rs, Qi21Dit::qk_norm_rope; gpu_wgpu/qi21.rs, zi_qkrope).
template <bool BF>
__global__ void __launch_bounds__(256) qkrope_kernel(int heads, float eps, uint16_t* __restrict__ panel,
                                                     const float* __restrict__ norm_q,
                                                     const float* __restrict__ norm_k,
                                                     RopeTables tabs) {
  const int row = blockIdx.x;
  int si = 0;
#pragma unroll
  for (int i = 1; i < kMaxSeq; ++i)
    if (i < tabs.nsrc && row >= tabs.src[i].row0) si = i;
  const size_t trow = static_cast<size_t>(row - tabs.src[si].row0) * 64;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const float2 c = reinterpret_cast<const float2*>(tabs.src[si].cos_ + trow)[lane];
  const float2 sn = reinterpret_cast<const float2*>(tabs.src[si].sin_ + trow)[lane];
  const float4 wq = reinterpret_cast<const float4*>(norm_q)[lane];
  const float4 wk = reinterpret_cast<const float4*>(norm_k)[lane];
  const int H = heads * 128;
  uint16_t* base = panel + static_cast<size_t>(row) * 3 * H;
  for (int v = warp; v < 2 * heads; v += 8) {
    uint2* p = reinterpret_cast<uint2*>(base + v * 128 + lane * 4);
    const uint2 raw = *p;
    const float2 lo = unpack2<BF>(raw.x);
    const float2 hi = unpack2<BF>(raw.y);
    float ss = (lo.x * lo.x + lo.y * lo.y) + (hi.x * hi.x + hi.y * hi.y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss * (1.f / 128.f) + eps);
    const float4 w = v < heads ? wq : wk;
    const float a0 = lo.x * inv * w.x, a1 = lo.y * inv * w.y;
    const float a2 = hi.x * inv * w.z, a3 = hi.y * inv * w.w;
    uint2 out;
    out.x = pack2<BF>(a0 * c.x - a1 * sn.x, a0 * sn.x + a1 * c.x);
    out.y = pack2<BF>(a2 * c.y - a3 * sn.y, a2 * sn.y + a3 * c.y);
    *p = out;
  }
}

cudaError_t launch_qkrope(int rows, int heads, float eps, void* panel, int dt, const float* norm_q,
                          const float* norm_k, const RopeTables& tabs, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (dt != DT_F16 && dt != DT_BF16) return cudaErrorInvalidValue;
  uint16_t* pp = static_cast<uint16_t*>(panel);
  if (dt == DT_BF16)
    qkrope_kernel<true><<<rows, 256, 0, s>>>(heads, eps, pp, norm_q, norm_k, tabs);
  else
    qkrope_kernel<false><<<rows, 256, 0, s>>>(heads, eps, pp, norm_q, norm_k, tabs);
  return cudaGetLastError();
}

// --------------------------------------------------------------- kvcopy ----
// The K|V columns of the panel -> the layer's cache row, 16 B per thread
// (gpu_wgpu/qi21.rs, qi_kvcopy); 16-bit elements of either type.
__global__ void kvcopy_kernel(int rows, int dim, const uint16_t* __restrict__ panel,
                              uint16_t* __restrict__ kv) {
  const int per_row = (2 * dim) / 8;  // uint4 per cache row
  const size_t total = static_cast<size_t>(rows) * per_row;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t r = i / per_row;
    const int c = static_cast<int>(i - r * per_row);
    const uint4 v = reinterpret_cast<const uint4*>(panel + r * 3 * dim + dim)[c];
    reinterpret_cast<uint4*>(kv + r * 2 * dim)[c] = v;
  }
}

cudaError_t launch_kvcopy(int rows, int dim, const void* panel, void* kv, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const size_t total = static_cast<size_t>(rows) * (2 * dim / 8);
  const int grid = static_cast<int>(std::min<size_t>((total + 255) / 256, static_cast<size_t>(sm_count()) * 16));
  kvcopy_kernel<<<grid, 256, 0, s>>>(rows, dim, static_cast<const uint16_t*>(panel), static_cast<uint16_t*>(kv));
  return cudaGetLastError();
}

// -------------------------------------------------------------- pack w13 ----
// Interleave gate and up in 64-row blocks so that every 128-row slice of the
// plane holds a matching (gate, up) pair for the SwiGLU epilogue.
__global__ void pack_w13_kernel(int inter, int dim, const uint16_t* __restrict__ gate,
                                const uint16_t* __restrict__ up, uint16_t* __restrict__ dst) {
  const int r = blockIdx.x;  // destination row in [0, 2I)
  const int j = r >> 7;
  const int w = r & 127;
  const uint16_t* src = (w < 64) ? gate + static_cast<size_t>(64 * j + w) * dim
                                 : up + static_cast<size_t>(64 * j + (w - 64)) * dim;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst + static_cast<size_t>(r) * dim);
  for (int c = threadIdx.x; c < dim / 8; c += blockDim.x) d4[c] = s4[c];
}

cudaError_t launch_pack_w13(int inter, int dim, const void* gate, const void* up, void* dst, cudaStream_t s) {
  pack_w13_kernel<<<2 * inter, 256, 0, s>>>(inter, dim, static_cast<const uint16_t*>(gate),
                                            static_cast<const uint16_t*>(up), static_cast<uint16_t*>(dst));
  return cudaGetLastError();
}

}  // namespace qi21
