// The ends of a denoiser call: the image embedding before the blocks and
// the final modulated LayerNorm + output projection after them
// (qwen_image21.rs, Qi21Dit::embed_image and the end of Qi21Dit::step_cpu;
// gpu_wgpu/qi21.rs, zi_embed and zi_final). Both projections have 64
// latent channels on one side, so they are small f32 contractions run on
// the CUDA cores (f32 weights, as the page keeps for its device path).
#include <algorithm>

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

}  // namespace qi21
