// Flash attention over [prefix cache, own panel rows] with a leading-run
// visibility mask (qwen_image21.rs, Qi21Dit::attention + softmax_prefix;
// gpu_wgpu/qi21.rs, qi_flash): query i of a sequence sees keys
// [0, lim(i)), lim(i) = vis[i] in the prefill and every key in a step.
// Keys j < n_pre come from the layer's cache [n_pre][2H] (K then V), the
// rest from the panel rows [own_row0 + j - n_pre] (K at column H, V at 2H).
//
// CTA: 8 warps x 16 query rows = 128 queries of one head and one sequence;
// K/V blocks of 64 keys double-buffered in swizzled shared memory by
// cp.async (rows past the last key are zero-filled), S = Q K^T and O += P V
// on the tensor cores (mma.m16n8k16, f16 in, f32 accumulate), the online
// softmax in f32 registers with exp2 and the 1/sqrt(128) scale folded into
// the exponent. The key-block loop stops at the visibility of the tile's
// last live query (vis is non-decreasing); masked keys get weight exactly 0.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace qi21 {

constexpr int kAttBM = 128;
constexpr int kAttBN = 64;
constexpr int kAttD = 128;
constexpr int kAttThreads = 256;
constexpr int kAttRowBytes = kAttD * 2;                 // 256 B per row
constexpr int kAttQBytes = kAttBM * kAttRowBytes;       // 32 KB
constexpr int kAttKVBytes = kAttBN * kAttRowBytes;      // 16 KB
constexpr int kAttSmem = kAttQBytes + 4 * kAttKVBytes;  // Q + 2x(K, V) = 96 KB

// byte offset of 16-byte chunk c (0..15) of row r in a swizzled tile
__device__ __forceinline__ uint32_t att_swz(int r, int c) {
  return static_cast<uint32_t>(r * kAttRowBytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct AttnKernelArgs {
  const __half* panel;
  __half* out;
  int heads;
  int dim;  // H
  float scale_log2;
  AttnSeq seq[kMaxSeq];
};

__global__ void __launch_bounds__(kAttThreads, 1) attn_mma_kernel(const AttnKernelArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const AttnSeq sq = a.seq[blockIdx.z];
  const int qt0 = blockIdx.x * kAttBM;
  if (qt0 >= sq.nq) return;
  const int h = blockIdx.y;
  const int H = a.dim;
  const int ntot = sq.n_pre + sq.n_own;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;
  const int tig = lane & 3;

  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + kAttQBytes;
  const uint32_t sV0 = sK0 + 2 * kAttKVBytes;

  // Key blocks walked: up to the last live query's visibility.
  const int q_last = min(qt0 + kAttBM, sq.nq) - 1;
  const int lim_last = sq.vis ? min(ntot, static_cast<int>(sq.vis[q_last])) : ntot;
  const int nkb = (lim_last + kAttBN - 1) / kAttBN;

  // This thread's two query rows and their limits.
  const int r0 = qt0 + warp * 16 + g;
  const int r1 = r0 + 8;
  const int lim0 = (r0 < sq.nq) ? (sq.vis ? min(ntot, static_cast<int>(sq.vis[r0])) : ntot) : ntot;
  const int lim1 = (r1 < sq.nq) ? (sq.vis ? min(ntot, static_cast<int>(sq.vis[r1])) : ntot) : ntot;

  const size_t ld_panel = static_cast<size_t>(3) * H;
  const size_t ld_pre = static_cast<size_t>(2) * H;

  // ---- Q tile -> smem (rows past nq zero-filled)
  for (int i = tid; i < kAttBM * 16; i += kAttThreads) {
    const int r = i >> 4, c = i & 15;
    const int qr = qt0 + r;
    const bool ok = qr < sq.nq;
    const __half* src = a.panel + (ok ? (static_cast<size_t>(sq.q_row0 + qr) * ld_panel) : 0) +
                        h * kAttD + c * 8;
    cp_async16(sQ + att_swz(r, c), src, ok);
  }
  auto load_kv = [&](int kb, int buf) {
    const uint32_t dK = sK0 + buf * kAttKVBytes;
    const uint32_t dV = sV0 + buf * kAttKVBytes;
    for (int i = tid; i < kAttBN * 16; i += kAttThreads) {
      const int r = i >> 4, c = i & 15;
      const int j = kb * kAttBN + r;
      const __half* ks;
      const __half* vs;
      bool ok = true;
      if (j < sq.n_pre) {
        ks = sq.kv_pre + static_cast<size_t>(j) * ld_pre + h * kAttD + c * 8;
        vs = ks + H;
      } else if (j < ntot) {
        const size_t row = static_cast<size_t>(sq.own_row0 + j - sq.n_pre) * ld_panel;
        ks = a.panel + row + H + h * kAttD + c * 8;
        vs = ks + H;
      } else {
        ks = a.panel;
        vs = a.panel;
        ok = false;
      }
      cp_async16(dK + att_swz(r, c), ks, ok);
      cp_async16(dV + att_swz(r, c), vs, ok);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  uint32_t qf[8][4];
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int kb = 0; kb < nkb; ++kb) {
    const int buf = kb & 1;
    if (kb + 1 < nkb) {
      load_kv(kb + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kb == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = 2 * kk + (lane >> 4);
        ldsm_x4(sQ + att_swz(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t sK = sK0 + buf * kAttKVBytes;
    const uint32_t sV = sV0 + buf * kAttKVBytes;

    // S = Q K^T: 16 rows x 64 keys per warp
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + att_swz(key, c), b0, b1, b2, b3);
        mma16816(s[2 * np], qf[kk], b0, b1);
        mma16816(s[2 * np + 1], qf[kk], b2, b3);
      }
    }

    // scale, mask, online softmax
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int key = kb * kAttBN + nt * 8 + 2 * tig;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kj = key + (e & 1);
        const int lim = (e < 2) ? lim0 : lim1;
        const float v = (kj < lim) ? s[nt][e] * a.scale_log2 : -INFINITY;
        s[nt][e] = v;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float al0 = exp2f(m0 - mx0);
    const float al1 = exp2f(m1 - mx1);
    m0 = mx0;
    m1 = mx1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = exp2f(s[nt][0] - mx0);
      const float p1 = exp2f(s[nt][1] - mx0);
      const float p2 = exp2f(s[nt][2] - mx1);
      const float p3 = exp2f(s[nt][3] - mx1);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      const int kk = nt >> 1;
      if ((nt & 1) == 0) {
        pa[kk][0] = pack_half2(p0, p1);
        pa[kk][1] = pack_half2(p2, p3);
      } else {
        pa[kk][2] = pack_half2(p0, p1);
        pa[kk][3] = pack_half2(p2, p3);
      }
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) {
      o[dt][0] *= al0;
      o[dt][1] *= al0;
      o[dt][2] *= al1;
      o[dt][3] *= al1;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sV + att_swz(key, c), b0, b1, b2, b3);
        mma16816(o[2 * dp], pa[kk], b0, b1);
        mma16816(o[2 * dp + 1], pa[kk], b2, b3);
      }
    }
    __syncthreads();
  }

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float i0 = 1.f / l0;
  const float i1 = 1.f / l1;
  __half* out0 = a.out + static_cast<size_t>(sq.q_row0 + r0) * H + h * kAttD + 2 * tig;
  __half* out1 = a.out + static_cast<size_t>(sq.q_row0 + r1) * H + h * kAttD + 2 * tig;
#pragma unroll
  for (int dt = 0; dt < 16; ++dt) {
    if (r0 < sq.nq)
      *reinterpret_cast<uint32_t*>(out0 + dt * 8) = pack_half2(o[dt][0] * i0, o[dt][1] * i0);
    if (r1 < sq.nq)
      *reinterpret_cast<uint32_t*>(out1 + dt * 8) = pack_half2(o[dt][2] * i1, o[dt][3] * i1);
  }
}

cudaError_t launch_attention(const AttnArgs& in, cudaStream_t s) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kAttSmem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  AttnKernelArgs a;
  a.panel = in.panel;
  a.out = in.out;
  a.heads = in.heads;
  a.dim = in.heads * kAttD;
  a.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(kAttD)));
  int maxq = 0;
  for (int i = 0; i < in.nseq; ++i) {
    a.seq[i] = in.seq[i];
    maxq = maxq > in.seq[i].nq ? maxq : in.seq[i].nq;
  }
  for (int i = in.nseq; i < kMaxSeq; ++i) a.seq[i] = AttnSeq{};
  if (maxq == 0) return cudaSuccess;
  dim3 grid((maxq + kAttBM - 1) / kAttBM, in.heads, in.nseq);
  attn_mma_kernel<<<grid, kAttThreads, kAttSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace qi21
