// tcgen05 GEMM for the block's four projections: C = A B^T with A [M][K]
// (activations) and B [N][K] (nn.Linear weights), both K-major and both f16
// or both bf16 (the geometry's dtype), f32 accumulation in TMEM, fused
// epilogues whose 16-bit outputs take the same type:
//   EPI_F16    qkv panel store                (gpu_wgpu/qi21.rs, zi_mm f16)
//   EPI_RESID  x += tanh(g) * acc on the f32 residual stream (the O and down
//              projections followed by Qi21Dit::gated_add); x moves through
//              shared memory in 32 x 32 chunks by TMA (load, update, store),
//              double-buffered per epilogue warp
//   EPI_SWIGLU silu(gate) * up on the interleaved gate/up plane
//              (qwen_image21.rs, block_cpu: silu(gate) * proj)
//   EPI_QKV    the qkv panel store with the per-head qk RMSNorm * w and the
//              interleaved RoPE applied to the q and k columns on the way out
//              (qwen_image21.rs, Qi21Dit::qk_norm_rope; each thread holds
//              whole 128-column head vectors of its row)
//   EPI_QKV_KV the same, the k and v columns also stored into the layer's
//              K|V cache rows (a prefill; gpu_wgpu/qi21.rs, qi_kvcopy, folded
//              into the store)
//   EPI_F32    plain f32 store (single-operation checks)
//
// The FP8 instance (OP = kOpF8) runs the same pipeline on E4M3 operands:
// byte-wide tensor maps with 128-byte boxes (128 elements per k-block, the
// same swizzled 128-byte rows), tcgen05.mma.kind::f8f6f4 (K = 32), and the
// accumulator multiplied by the A row scale and the B row (output channel)
// scale, both powers of two, before the epilogue above.
//
// Persistent clusters of two CTAs (one per SM) running the pair MMA
// (tcgen05.mma.cta_group::2, a 256 x BN tile per CTA pair): CTA r holds rows
// [128 r, 128 r + 128) of the A tile and rows [BN/2 r, BN/2 r + BN/2) of
// the B tile in its shared memory, and receives rows [128 r, 128 r + 128)
// of the accumulator in its TMEM. Each SM therefore holds only half of B:
// 32 KB stages instead of 48 KB, six of them, enough operand data in flight
// to cover the TMA latency. 6 warps per CTA (10 for qkv):
//   warp 0     TMA producer (both CTAs): A 128x64 and B (BN/2)x64 tiles
//              (128-byte swizzle) into a 6-stage ring; the loads of both CTAs
//              complete on the even CTA's "full" mbarrier
//   warp 1     TMEM allocation (jointly, both CTAs); in the even CTA one
//              thread issues the pair MMAs (M=256, N=BN, K=16) and commits
//              that release a stage / publish an accumulator in both CTAs
//   warps 2-5  epilogue (both CTAs): tcgen05.ld of their 32-lane quadrant,
//              fused op, 128-bit stores; two TMEM accumulators so the
//              epilogue of tile i overlaps the MMAs of tile i+1; each warp
//              reports "accumulator free" to the even CTA. The qkv
//              instances have two epilogue warps per quadrant (warps 2-9),
//              one 128-column head each.
// Schedule (tile_at): tiles in groups of G pair rows (column blocks outer,
// the pair rows of a group inner), G chosen on the host so that the group's
// A rows stay in L2 while its column blocks stream past; whole tiles of odd
// waves load their k-blocks top down (a wave starts on the k-slices its
// predecessor read last); a partial last wave is split along K into
// column-owned parts that run side by side and merge their f32 partials
// through global scratch (the K-split tail). A cluster's last item stages
// its epilogue data (x chunks, other parts' partials) in the then idle
// operand ring.
#include <algorithm>
#include <cstdio>

#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace qi21 {

// Status word of this translation unit's kernels (a wait that gave up).
static __device__ unsigned int s_gemm_status = 0;

unsigned int gemm_status_read_clear() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, s_gemm_status, sizeof v);
  cudaMemcpyToSymbol(s_gemm_status, &z, sizeof z);
  return v;
}

constexpr int kBM = 128;
constexpr int kBK = 64;

// Operand kinds of an instance: f16 or bf16 A/B (kind::f16, 16-bit
// epilogue outputs of the same type) or E4M3 codes (kind::f8f6f4, f16
// epilogue outputs).
constexpr int kOpF16 = 0;
constexpr int kOpBF16 = 1;
constexpr int kOpF8 = 2;


template <int BN, int EPI>
struct GemmCfg {
  static constexpr int kABytes = kBM * kBK * 2;        // this CTA's A rows
  static constexpr int kBBytes = (BN / 2) * kBK * 2;   // this CTA's half of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  // EPI_RESID: per epilogue warp a ring of kXBufs 32 x 32 f32 chunks of x
  // (4 KB each; kXBufs - 1 loads ahead) beside the same 192 KB of operand
  // stages (224 KB in all; four buffers with one stage fewer measured the
  // same)
  static constexpr int kXBufs = 2;
  static constexpr int kEpiBytes = EPI == EPI_RESID ? 4 * kXBufs * 4096 : 0;
  static constexpr int kStages = (192 * 1024) / kStageBytes;
  static constexpr int kEpiOff = kStages * kStageBytes;
  static constexpr int kTmemCols = 2 * BN;
  // a cluster's last work item: each epilogue warp may use 48 KB of the
  // (then idle) operand ring for its x chunks and the other K-split parts'
  // partials, and 8 single-use barriers for those x chunks
  static constexpr int kTailWarpBytes = 48 * 1024;
  static_assert(4 * kTailWarpBytes <= kStages * kStageBytes, "tail staging exceeds the operand ring");
  static_assert(BN * 128 <= kTailWarpBytes, "tail staging of one warp");
  // epilogue warps: two per TMEM lane quadrant for qkv (one 128-column head
  // each), one per quadrant otherwise
  static constexpr int kEpiWarps = (EPI == EPI_QKV || EPI == EPI_QKV_KV) ? 8 : 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kBarBytes = 512;
  static_assert((2 * kStages + 4 + 4 * kXBufs + 32) * 8 + 8 <= kBarBytes, "barrier region");
  static constexpr int kSmem = kEpiOff + kEpiBytes + kBarBytes + 1024;
};

struct EpiArgs {
  void* out;
  int ldo;
  const float* gate;
  QkvEpi qkv;
  const float* sa;  // FP8: per A row
  const float* sw;  // FP8: per B row (output column)
  // K-split tail: raw f32 partials, one slab per (tail tile, part, CTA
  // rank, epilogue warp) of [BN columns][32 rows] (a part writes the
  // columns it does not own), and one ready flag per slab, set to `epoch`
  float* part;
  int* flags;
  int parts;
  int epoch;
};

// Bounded wait (acquire) for *f == want, by one thread; false if it gave up.
__device__ __forceinline__ bool wait_flag(const int* f, int want, volatile int* abort, unsigned int* status) {
  const unsigned long long t0 = globaltimer();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v == want) return true;
    if (*abort) return false;
    __nanosleep(32);
    if (globaltimer() - t0 > kWaitTimeoutNs) {
      *abort = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void set_flag_release(int* f, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}

// 16-byte global -> shared copy (cp.async, L2 only), its group commit and
// the wait for all of this thread's groups.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// A split tail tile's owner of columns [o0, o0 + w) sums, per element of
// this thread's row, every part's value in part order (its own accumulator
// at its own place, the others' staged partials), so the result does not
// depend on which part owns the columns.
struct PartSum {
  const float* st;  // this warp's staged partials [other part][w][32], null if none
  int parts, own, w, o0;
  // kMaxP: the most parts the caller's epilogue splits into
  template <int kMaxP>
  __device__ __forceinline__ void add(uint32_t (&r)[32], int col) const {
    if (st == nullptr) return;
    const float* b = st + static_cast<size_t>(col - o0) * 32 + (threadIdx.x & 31);
    if (kMaxP == 2 || parts == 2) {  // one other part; a + b == b + a, whichever part owns
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + b[e * 32]);
      return;
    }
    const size_t slot = static_cast<size_t>(w) * 32;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float a = __uint_as_float(r[e]);
      float s = own == 0 ? a : b[e * 32];
#pragma unroll
      for (int pp = 1; pp < kMaxP; ++pp)
        if (pp < parts) s += pp == own ? a : b[(pp < own ? pp : pp - 1) * slot + e * 32];
      r[e] = __float_as_uint(s);
    }
  }
  __device__ __forceinline__ void operator()(uint32_t (&r)[32], int col) const { add<kMaxKParts>(r, col); }
};

// Owner width of a split tail tile: the qkv epilogue normalises whole
// 128-column heads and SwiGLU pairs 64 gate with 64 up columns, so their
// owners take 128 columns; the other epilogues take 32-column chunks.
// Parts: at most 2 for both (on a 128-column tile one owner and one part
// that only contributes its partial). Four SwiGLU parts (two owners and
// two contributors per 256-column tile) measured slower than two on the
// gate/up projection: the extra partial traffic outweighs the shorter tail.
template <int EPI>
constexpr int split_own_min() {
  return (EPI == EPI_QKV || EPI == EPI_QKV_KV || EPI == EPI_SWIGLU) ? 128 : 32;
}
template <int EPI>
constexpr int split_max_parts() {
  return split_own_min<EPI>() == 128 ? 2 : kMaxKParts;
}

// FP8: 32 accumulator columns starting at column `col` times sa sw[col + i]
template <int OP>
__device__ __forceinline__ void f8_scale(uint32_t (&r)[32], float sa, const float* __restrict__ sw, int col) {
  if constexpr (OP == kOpF8) {
    const float4* s4 = reinterpret_cast<const float4*>(sw + col);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 w = __ldg(s4 + j);
      r[4 * j + 0] = __float_as_uint(__uint_as_float(r[4 * j + 0]) * sa * w.x);
      r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) * sa * w.y);
      r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) * sa * w.z);
      r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) * sa * w.w);
    }
  }
}

// 32 bytes from / to global memory in one access per thread (a whole
// sector: the qkv epilogue's rows are one per thread, so a warp's accesses
// touch 32 rows); p 32-byte aligned.
__device__ __forceinline__ void ldg8(const float* p, float (&r)[8]) {
  asm("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7])
      : "l"(p));
}
__device__ __forceinline__ void stg8(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// silu(v) = v / (1 + e^-v) with the approximate exponential and divide
// (relative error ~2^-21, far below the 16-bit rounding of the output)
__device__ __forceinline__ float silu_f(float v) { return __fdividef(v, 1.f + __expf(-v)); }

// Epilogue of one row over accumulator columns [o0, o1) of the tile.
template <int BN, int EPI, int OP>
__device__ __forceinline__ void gemm_epilogue(uint32_t tbase, int row, int M, int n0, int o0, int o1,
                                              const EpiArgs& ep, const PartSum& padd) {
  constexpr bool F8 = OP == kOpF8;
  constexpr bool BF = OP == kOpBF16;  // 16-bit outputs in bf16
  const bool live = row < M;
  const float sa = (F8 && live) ? ep.sa[row] : 1.f;
  if constexpr (EPI == EPI_SWIGLU) {
    uint16_t* out = static_cast<uint16_t*>(ep.out) + static_cast<size_t>(row) * ep.ldo + n0 / 2;
#pragma unroll 1
    for (int p = o0 / 128; p < o1 / 128; ++p) {
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t g[32], u[32];
        tmem_ld32(tbase + p * 128 + c * 32, g);
        tmem_ld32(tbase + p * 128 + 64 + c * 32, u);
        tmem_ld_wait(g);
        tmem_ld_wait(u);
        padd.add<2>(g, p * 128 + c * 32);
        padd.add<2>(u, p * 128 + 64 + c * 32);
        f8_scale<OP>(g, sa, ep.sw, n0 + p * 128 + c * 32);
        f8_scale<OP>(u, sa, ep.sw, n0 + p * 128 + 64 + c * 32);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(out + p * 64 + c * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 8 * j + 2 * e;
              const float h0 = silu_f(__uint_as_float(g[i])) * __uint_as_float(u[i]);
              const float h1 = silu_f(__uint_as_float(g[i + 1])) * __uint_as_float(u[i + 1]);
              w[e] = pack2<BF>(h0, h1);
            }
            dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  } else if constexpr (EPI == EPI_QKV || EPI == EPI_QKV_KV) {
    const QkvEpi& qe = ep.qkv;
    uint16_t* out = static_cast<uint16_t*>(ep.out) + static_cast<size_t>(row) * ep.ldo;
    // this row's RoPE table (the sequence whose rows contain it)
    int si = 0;
#pragma unroll
    for (int i = 1; i < kMaxSeq; ++i)
      if (i < qe.tabs.nsrc && row >= qe.tabs.src[i].row0) si = i;
    const size_t trow = static_cast<size_t>(live ? row - qe.tabs.src[si].row0 : 0) * 64;
    const float* cs = qe.tabs.src[si].cos_ + trow;
    const float* sn = qe.tabs.src[si].sin_ + trow;
#pragma unroll 1
    for (int hc = o0 / 128; hc < o1 / 128; ++hc) {
      const int col = n0 + hc * 128;
      const int part = col / qe.H;  // 0 q, 1 k, 2 v (uniform over the tile)
      uint16_t* dst = out + col;
      // prefill: the same k / v values into the cache row (K at col - H, V at col - H)
      uint16_t* kvd = (EPI == EPI_QKV_KV && part > 0)
                          ? static_cast<uint16_t*>(qe.kv) + static_cast<size_t>(row) * 2 * qe.H + (col - qe.H)
                          : nullptr;
      // one 32-column chunk of the head: accumulator (+ the other K parts'
      // partials, x the FP8 scales) in r
      auto chunk = [&](int c, uint32_t (&r)[32]) {
        tmem_ld32(tbase + hc * 128 + c * 32, r);
        tmem_ld_wait(r);
        padd.add<2>(r, hc * 128 + c * 32);
        f8_scale<OP>(r, sa, ep.sw, col + c * 32);
      };
      if (part == 2) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          chunk(c, r);
          if (!live) continue;
#pragma unroll
          for (int j2 = 0; j2 < 2; ++j2) {
            uint32_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              v[e] = pack2<BF>(__uint_as_float(r[16 * j2 + 2 * e]), __uint_as_float(r[16 * j2 + 2 * e + 1]));
            stg8(dst + c * 32 + j2 * 16, v);
            if constexpr (EPI == EPI_QKV_KV) stg8(kvd + c * 32 + j2 * 16, v);
          }
        }
        continue;
      }
      // two passes over the head in TMEM, 32 columns in registers at a
      // time: the sum of squares, then normalise, rotate and store
      float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        chunk(c, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float v = __uint_as_float(r[e]);
          ss[e & 3] = fmaf(v, v, ss[e & 3]);
        }
      }
      const float inv = rsqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) * (1.f / 128.f) + qe.eps);
      // the norm weights (the caller's, 16-byte aligned; the same address in
      // every lane) in 16-byte loads; the per-row tables and outputs, in
      // the library's 256-byte aligned buffers, 32 bytes at a time
      const float4* w4 = reinterpret_cast<const float4*>(part == 0 ? qe.norm_q : qe.norm_k);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        chunk(c, r);
        if (!live) continue;
#pragma unroll
        for (int j2 = 0; j2 < 2; ++j2) {
          // elements 32c + 16j2 .. +15 = pairs 16c + 8j2 .. +7
          float4 w[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) w[q4] = __ldg(w4 + 8 * c + 4 * j2 + q4);
          float cv[8], sv[8];
          ldg8(cs + 16 * c + 8 * j2, cv);
          ldg8(sn + 16 * c + 8 * j2, sv);
          uint32_t v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 wq = w[e >> 1];
            const float w0 = (e & 1) ? wq.z : wq.x, w1 = (e & 1) ? wq.w : wq.y;
            const float a = __uint_as_float(r[16 * j2 + 2 * e]) * inv * w0;
            const float b = __uint_as_float(r[16 * j2 + 2 * e + 1]) * inv * w1;
            v[e] = pack2<BF>(a * cv[e] - b * sv[e], a * sv[e] + b * cv[e]);
          }
          stg8(dst + c * 32 + j2 * 16, v);
          if constexpr (EPI == EPI_QKV_KV)
            if (part == 1) stg8(kvd + c * 32 + j2 * 16, v);
        }
      }
    }
  } else {
#pragma unroll 1
    for (int c = o0 / 32; c < o1 / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tbase + c * 32, r);
      tmem_ld_wait(r);
      padd(r, c * 32);
      if (!live) continue;
      const int col = n0 + c * 32;
      f8_scale<OP>(r, sa, ep.sw, col);
      if constexpr (EPI == EPI_F16) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(ep.out) +
                                              static_cast<size_t>(row) * ep.ldo + col);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          dst[j] = make_uint4(pack2<BF>(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1])),
                              pack2<BF>(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                              pack2<BF>(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                              pack2<BF>(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
        }
      } else if constexpr (EPI == EPI_F32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(ep.out) +
                                                static_cast<size_t>(row) * ep.ldo + col);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                               __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      } else {  // EPI_RESID
        float4* xp = reinterpret_cast<float4*>(static_cast<float*>(ep.out) +
                                               static_cast<size_t>(row) * ep.ldo + col);
        const float4* gp = reinterpret_cast<const float4*>(ep.gate + col);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4 x = xp[j];
          const float4 gv = __ldg(gp + j);
          x.x = fmaf(gv.x, __uint_as_float(r[4 * j + 0]), x.x);
          x.y = fmaf(gv.y, __uint_as_float(r[4 * j + 1]), x.y);
          x.z = fmaf(gv.z, __uint_as_float(r[4 * j + 2]), x.z);
          x.w = fmaf(gv.w, __uint_as_float(r[4 * j + 3]), x.w);
          xp[j] = x;
        }
      }
    }
  }
}

// Work item t of the persistent schedule (one per cluster step): the first
// nfull items are whole 2 x (BM x BN) tiles with pair row mp (tile rows
// 2 mp and 2 mp + 1) and column block nb; when the last wave is partial,
// each of its tiles is split along K into `parts` items of k-blocks
// [part nk / parts, (part + 1) nk / parts) that run side by side in one
// shorter wave (whole tiles, so every SM streams operands at the rate of a
// full tile); parts 0 .. parts-2 store raw partials, the last part adds
// them in order and runs the epilogue.
// Full tile f lies in group f / (G nN) of G pair rows (the last group may
// be smaller); inside a group the pair rows run fastest, then the column
// blocks, so the clusters of a wave work on a band of about G pair rows and
// a few column blocks, and the group's A rows are reused from L2 across its
// column blocks. G = num_mp is plain pair-rows-fastest order.
struct TileInfo {
  int mp, n0, bn;
  int kb0, kb1;  // k-blocks of this item
  int part;      // -1 whole tile, else the part of a split tail tile
  int tail;      // index of the tail tile (split tiles only)
  bool rev;      // load the k-blocks from kb1 - 1 down (whole tiles of odd waves)
};

__device__ __forceinline__ void raster(int f, int num_mp, int nN, int G, int& mp, int& nb) {
  const int per_group = G * nN;
  const int g = f / per_group;
  const int first = g * G;
  const int gs = min(G, num_mp - first);
  const int r = f - g * per_group;
  mp = first + r % gs;
  nb = r / gs;
}

// Whole tiles of odd waves (t / nclusters odd) walk K downwards: a wave
// then starts on the k-slices of the A / B panels that the previous wave
// read last, which are the ones still in L2.
template <int BN>
__device__ __forceinline__ TileInfo tile_at(int t, int num_mp, int nN, int G, int nfull, int parts, int nk,
                                            int nclusters) {
  int mp, nb;
  if (t < nfull) {
    raster(t, num_mp, nN, G, mp, nb);
    return TileInfo{mp, nb * BN, BN, 0, nk, -1, 0, ((t / nclusters) & 1) != 0};
  }
  const int u = t - nfull;
  const int tail = u / parts;
  const int part = u - tail * parts;
  raster(nfull + tail, num_mp, nN, G, mp, nb);
  return TileInfo{mp, nb * BN, BN, part * nk / parts, (part + 1) * nk / parts, part, tail, false};
}

template <int BN, int EPI, int OP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmCfg<BN, EPI>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmX, int M, int N, int K, int group, int nfull, int num_tiles,
                   EpiArgs ep) {
  using C = GemmCfg<BN, EPI>;
  constexpr bool F8 = OP == kOpF8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kEpiOff + C::kEpiBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* xbar = tempty + 2;  // [4][kXBufs] EPI_RESID: x chunk landed, per warp and buffer
  // then 4 x 8 single-use barriers of the last item's x chunks
  uint32_t* tslot = reinterpret_cast<uint32_t*>(xbar + 4 * C::kXBufs + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_rank());
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int num_mp = ((M + kBM - 1) / kBM + 1) / 2;
  const int nN = N / BN;
  constexpr int kKE = F8 ? 128 : kBK;  // K elements per k-block (128 bytes per row)
  const int nk = K / kKE;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);   // the even CTA's producer (+ both CTAs' bytes)
      mbar_init(&empty[i], 1);  // the pair-MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * C::kEpiWarps);  // the epilogue warps of both CTAs
    }
    for (int i = 0; i < 4 * C::kXBufs + 32; ++i) mbar_init(&xbar[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI == EPI_RESID) tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc_pair(tslot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers and TMEM ready before any remote use
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = cluster; t < num_tiles && ok; t += nclusters) {
        const TileInfo ti = tile_at<BN>(t, num_mp, nN, group, nfull, ep.parts, nk, nclusters);
        const int m0 = (2 * ti.mp + rank) * kBM;
        const int bh = BN / 2;  // B rows this CTA holds
        // the even CTA's barrier counts both CTAs' A and B bytes
        const uint32_t bytes = 2u * (C::kABytes + C::kBBytes);
        for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, &s_gemm_status)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * C::kStageBytes;
          const uint32_t fb = mapa_rank(&full[s], 0);
          if (leader) mbar_arrive_expect_tx(&full[s], bytes);
          const int kc = ti.rev ? ti.kb0 + ti.kb1 - 1 - kb : kb;  // the k-block loaded into this stage
          tma_load_2d_pair(sa, &tmA, fb, kc * kKE, m0);
          tma_load_2d_pair(sa + C::kABytes, &tmB, fb, kc * kKE, ti.n0 + rank * bh);
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_f16(2 * kBM, BN, false, OP == kOpBF16);
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int t = cluster; t < num_tiles && ok; t += nclusters, ++it) {
        const TileInfo ti = tile_at<BN>(t, num_mp, nN, group, nfull, ep.parts, nk, nclusters);
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(&tempty[acc], aph ^ 1u, abort_flag, &s_gemm_status)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
        for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
          if (!mbar_wait(&full[s], ph, abort_flag, &s_gemm_status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * C::kStageBytes);
          const uint64_t adesc = sdesc_sw128(sa);
          const uint64_t bdesc = sdesc_sw128(sa + C::kABytes);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 4 x 32 bytes of each 128-byte row
            const uint32_t accumulate = (kb != ti.kb0 || k != 0) ? 1u : 0u;
            if constexpr (F8)
              tc_mma_f8_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, accumulate);
            else
              tc_mma_f16_pair(d, adesc + 2 * k, bdesc + 2 * k, idesc, accumulate);
          }
          tc_commit_pair(&empty[s], 0x3);
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) tc_commit_pair(&tfull[acc], 0x3);
      }
    }
  } else {
    const int q = warp & 3;             // TMEM lane quadrant this warp may access
    const int h = (warp - 2) >> 2;      // qkv: which of the quadrant's two epilogue warps
    int it = 0;
    int xu = 0;  // EPI_RESID: x chunks this warp has staged in its epilogue buffers
    bool eok = true;
    // a cluster's last item: this warp's share of the idle operand ring and
    // its single-use x chunk barriers
    uint8_t* const wst = smem + q * C::kTailWarpBytes;
    uint64_t* const xl = xbar + 4 * C::kXBufs + 8 * q;
    for (int t = cluster; t < num_tiles && eok; t += nclusters, ++it) {
      const TileInfo ti = tile_at<BN>(t, num_mp, nN, group, nfull, ep.parts, nk, nclusters);
      const bool last = t + nclusters >= num_tiles;
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!mbar_wait(&tfull[acc], aph, abort_flag, &s_gemm_status)) break;
      tc_fence_after();
      // every MMA of this CTA has read its operands: in the last item the
      // ring may take generic and TMA writes
      if (last) fence_proxy_async_smem();
      const uint32_t tbase = tmem + static_cast<uint32_t>(acc * BN) + (static_cast<uint32_t>(q * 32) << 16);
      // accumulator columns whose outputs this item writes: all of them, or
      // for part p of a K-split tail tile (always a cluster's last item)
      // columns [p w, (p + 1) w), w = max(BN / parts, owner width); parts
      // past the last owner only contribute partials
      const int P = ti.part >= 0 ? ep.parts : 1;
      const int w = max(ti.bn / P, split_own_min<EPI>());
      const int o0 = ti.part >= 0 ? min(ti.part * w, ti.bn) : 0, o1 = min(o0 + w, ti.bn);
      // the columns this warp finishes: with two warps per quadrant (qkv),
      // one head each of a whole tile; of a K-split part's one owned head,
      // the first warp finishes it while the second hands over the other
      // columns' partials
      int f0 = o0, f1 = o1;
      bool hand_over = true;
      if constexpr (C::kEpiWarps == 8) {
        if (ti.part < 0) {
          f0 = min(o0 + h * 128, o1);
          f1 = min(f0 + 128, o1);
        } else if (h == 1) {
          f1 = f0;
        } else {
          hand_over = false;
        }
      }
      const bool owner = f1 > f0;
      // the last item's x chunks (EPI_RESID) sit after the staged partials
      const int xoff = (P - 1) * w * 128;
      const int row0 = (2 * ti.mp + rank) * kBM + q * 32;  // this warp's first row
      if (EPI == EPI_RESID && last && lane == 0)
        for (int c = o0 / 32; c < o1 / 32; ++c) {
          mbar_arrive_expect_tx(&xl[c - o0 / 32], 4096);
          tma_load_2d(wst + xoff + (c - o0 / 32) * 4096, &tmX, &xl[c - o0 / 32], ti.n0 + 32 * c, row0);
        }
      PartSum psum{nullptr, 1, 0, 0, 0};
      if (ti.part >= 0) {
        // hand the other columns to their owners through this part's slab,
        // then sum the other parts' slices of the own columns (staged in
        // the ring) with the accumulator
        const size_t slab = static_cast<size_t>(BN) * 32;
        const size_t sbase = static_cast<size_t>(ti.tail) * P * 8 + rank * 4 + q;  // + 8 per part
        float* mine = ep.part + (sbase + ti.part * 8) * slab + lane;
        if (hand_over) {
#pragma unroll 1
          for (int c = 0; c < ti.bn / 32; ++c) {
            if (c * 32 >= o0 && c * 32 < o1) continue;
            uint32_t r[32];
            tmem_ld32(tbase + c * 32, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) __stcg(mine + static_cast<size_t>(c * 32 + e) * 32, __uint_as_float(r[e]));
          }
          __threadfence();
          __syncwarp();
          if (lane == 0) set_flag_release(ep.flags + sbase + ti.part * 8, ep.epoch);
        }
        bool got = last;  // the schedule guarantees it; anything else is refused, not raced
        if (!last && lane == 0) {
          *abort_flag = 1;
          atomicOr(&s_gemm_status, kStatusTimeout);
        }
        if (owner && lane == 0)
          for (int pp = 0; pp < P && got; ++pp)
            if (pp != ti.part) got = wait_flag(ep.flags + sbase + pp * 8, ep.epoch, abort_flag, &s_gemm_status);
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          // let the x loads issued above land before the CTA leaves
          if (EPI == EPI_RESID && last && lane == 0)
            for (int c = o0 / 32; c < o1 / 32; ++c) mbar_wait_drain(&xl[c - o0 / 32], 0);
          __syncwarp();
          eok = false;
          break;
        }
        if (owner) {
          __threadfence();
          float* st = reinterpret_cast<float*>(wst);
          int slot = 0;
          for (int pp = 0; pp < P; ++pp) {
            if (pp == ti.part) continue;
            const float* src = ep.part + (sbase + pp * 8) * slab + static_cast<size_t>(o0) * 32;
            float* dst = st + static_cast<size_t>(slot) * w * 32;
            for (int i = lane; i < w * 8; i += 32) cp_async16(dst + 4 * i, src + 4 * i);
            ++slot;
          }
          cp_async_commit_wait_all();
          __syncwarp();
          psum = PartSum{st, P, ti.part, w, o0};
        }
      }
      if constexpr (EPI == EPI_RESID) {
        // x += tanh(g) acc for this warp's 32 rows, 32 columns at a time:
        // TMA loads the x chunk (128-byte swizzled rows) into shared memory,
        // each thread updates its row there, TMA stores it back. Earlier
        // items cycle through kXBufs buffers, kXBufs - 1 loads ahead (their
        // epilogue hides behind the next item's MMAs); the last item, whose
        // epilogue nothing hides, has every chunk's load in flight at once
        // in the idle ring.
        constexpr int NB = C::kXBufs;
        uint8_t* eb = smem + C::kEpiOff + q * NB * 4096;
        uint64_t* xb = xbar + NB * q;
        const int row = row0 + lane;
        const float sa = (F8 && row < M) ? ep.sa[row] : 1.f;
        const int c0 = o0 / 32, c1 = o1 / 32;
        int issued = last ? c1 : c0;  // x chunks of this item whose loads were issued (a last item's: above)
        auto buf = [&](int c) -> uint8_t* { return last ? wst + xoff + (c - c0) * 4096 : eb + ((xu + c - c0) % NB) * 4096; };
        auto bar = [&](int c) -> uint64_t* { return last ? &xl[c - c0] : &xb[(xu + c - c0) % NB]; };
        auto par = [&](int c) -> uint32_t { return last ? 0u : static_cast<uint32_t>((xu + c - c0) / NB) & 1u; };
        auto load = [&](int c) {
          if (lane == 0) {
            if (!last) bulk_wait_read_all();  // the store that used this buffer last has read it
            mbar_arrive_expect_tx(bar(c), 4096);
            tma_load_2d(buf(c), &tmX, bar(c), ti.n0 + 32 * c, row0);
          }
          issued = c + 1;
        };
        const int ahead = last ? c1 - c0 : NB - 1;
        if (!last)
          for (int c = c0; c < c0 + ahead && c < c1; ++c) load(c);
        for (int c = c0; c < c1; ++c) {
          if (c + ahead < c1 && !*abort_flag) load(c + ahead);
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          // the gate values while the x chunk lands
          float4 gv[8];
          const float4* g4 = reinterpret_cast<const float4*>(ep.gate + ti.n0 + 32 * c);
#pragma unroll
          for (int j = 0; j < 8; ++j) gv[j] = __ldg(g4 + j);
          const bool got = mbar_wait(bar(c), par(c), abort_flag, &s_gemm_status);
          tmem_ld_wait(r);
          if (!got) {
            // another role gave up: let the x loads this warp issued land
            // before the CTA leaves (their bytes target this CTA's buffers)
            if (lane == 0)
              for (int d = c; d < issued; ++d) mbar_wait_drain(bar(d), par(d));
            __syncwarp();
            eok = false;
            break;
          }
          psum(r, 32 * c);
          f8_scale<OP>(r, sa, ep.sw, ti.n0 + 32 * c);
          // every load of the chunk before any store (a generic store would
          // otherwise order each later load behind it)
          float4* xs = reinterpret_cast<float4*>(buf(c) + lane * 128);
          float4 xv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) xv[j] = xs[j ^ (lane & 7)];  // chunk j of row `lane` under the 128-byte swizzle
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            xv[j].x = fmaf(gv[j].x, __uint_as_float(r[4 * j + 0]), xv[j].x);
            xv[j].y = fmaf(gv[j].y, __uint_as_float(r[4 * j + 1]), xv[j].y);
            xv[j].z = fmaf(gv[j].z, __uint_as_float(r[4 * j + 2]), xv[j].z);
            xv[j].w = fmaf(gv[j].w, __uint_as_float(r[4 * j + 3]), xv[j].w);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) xs[j ^ (lane & 7)] = xv[j];
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmX, buf(c), ti.n0 + 32 * c, row0);
            bulk_commit_group();
          }
        }
        if (!last) xu += c1 - c0;
      } else {
        gemm_epilogue<BN, EPI, OP>(tbase, (2 * ti.mp + rank) * kBM + q * 32 + lane, M, ti.n0, f0, f1, ep, psum);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_rank(&tempty[acc], 0));
    }
    // the x stores of this warp have completed before the CTA leaves
    if (EPI == EPI_RESID && lane == 0) bulk_wait_all();
  }
  // the partner may still be signalling this CTA's barriers: leave together
  __syncwarp();
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host ----

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // resolved once, thread-safely, on first use
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// Element types of the tensor maps.
enum MapType { MAP_F16, MAP_BF16, MAP_U8, MAP_F32 };

// 2-D tensor [outer][inner] of `type` with the given row pitch; box
// inner x outer, 128-byte swizzle.
static cudaError_t encode_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, MapType type) {
  auto fn = encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  auto encode = [&] {
    const CUtensorMapDataType dt = type == MAP_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : type == MAP_U8   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : type == MAP_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return fn(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  CUresult r = encode();
  // a host thread whose first library call this is may have no context yet
  if (r == CUDA_ERROR_INVALID_CONTEXT && bind_primary_context()) r = encode();
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// EPI_RESID: the f32 residual x [M][ldo] in 32 x 32 boxes (128-byte
// swizzled rows); other epilogues carry an unused copy of the A map.
static cudaError_t encode_x_map(GemmPlan* p) {
  if (p->epi != EPI_RESID) {
    p->tmX = p->tmA;
    return cudaSuccess;
  }
  return encode_2d(&p->tmX, p->out, p->N, p->M, static_cast<uint64_t>(p->ldo) * 4, 32, 32, MAP_F32);
}

cudaError_t make_gemm_plan(GemmPlan* p, int epi, int dt, int M, int N, int K, const void* A, const void* B,
                           void* out, int ldo, const float* gate) {
  if (dt != DT_F16 && dt != DT_BF16) return cudaErrorInvalidValue;
  const MapType mt = dt == DT_BF16 ? MAP_BF16 : MAP_F16;
  p->M = M;
  p->N = N;
  p->K = K;
  p->epi = epi;
  p->dt = dt;
  p->ldo = ldo;
  p->out = out;
  p->gate = gate;
  p->qkv = QkvEpi{};
  p->f8 = false;
  p->part = nullptr;
  p->part_bytes = 0;
  p->flags = nullptr;
  p->epoch = 1;
  p->parts_out = nullptr;
  p->sa = p->sw = nullptr;
  p->bn = (N % 256 == 0) ? 256 : 128;
  cudaError_t e = encode_2d(&p->tmA, A, K, M, static_cast<uint64_t>(K) * 2, kBK, kBM, mt);
  if (e != cudaSuccess) return e;
  // each CTA of a cluster loads half of the B tile
  e = encode_2d(&p->tmB, B, K, N, static_cast<uint64_t>(K) * 2, kBK, p->bn / 2, mt);
  if (e != cudaSuccess) return e;
  return encode_x_map(p);
}

cudaError_t make_gemm_plan_f8(GemmPlan* p, int epi, int M, int N, int K, const uint8_t* A, const float* sa,
                              const uint8_t* B, const float* sw, void* out, int ldo, const float* gate) {
  p->M = M;
  p->N = N;
  p->K = K;
  p->epi = epi;
  p->dt = DT_F16;
  p->ldo = ldo;
  p->out = out;
  p->gate = gate;
  p->qkv = QkvEpi{};
  p->f8 = true;
  p->part = nullptr;
  p->part_bytes = 0;
  p->flags = nullptr;
  p->epoch = 1;
  p->parts_out = nullptr;
  p->sa = sa;
  p->sw = sw;
  p->bn = 256;
  cudaError_t e = encode_2d(&p->tmA, A, K, M, static_cast<uint64_t>(K), 128, kBM, MAP_U8);
  if (e != cudaSuccess) return e;
  e = encode_2d(&p->tmB, B, K, N, static_cast<uint64_t>(K), 128, p->bn / 2, MAP_U8);
  if (e != cudaSuccess) return e;
  return encode_x_map(p);
}

size_t gemm_split_bytes(int bn, int tail_tiles, int parts) {
  // one [bn][32] f32 slab per (tail tile, part, CTA rank, epilogue warp)
  return parts > 1 ? static_cast<size_t>(tail_tiles) * parts * 8 * bn * 32 * sizeof(float) : 0;
}

// Pair rows per raster group: all of them while the whole A operand fits
// comfortably in L2, else as many as keep the group's A rows within
// kGroupBytes (the rest of L2 holds the streamed B column blocks).
constexpr size_t kGroupBytes = 56ull << 20;

static int raster_group(int num_mp, int K, int elem_bytes) {
  const size_t pair_bytes = static_cast<size_t>(2 * kBM) * K * elem_bytes;
  const size_t g = std::max<size_t>(1, kGroupBytes / pair_bytes);
  return static_cast<int>(std::min<size_t>(g, static_cast<size_t>(num_mp)));
}

template <int BN, int EPI, int OP = kOpF16>
static cudaError_t launch_t(const GemmPlan& p, cudaStream_t s) {
  using C = GemmCfg<BN, EPI>;
  // shared-memory opt-in and the resident cluster count, once per
  // instance and device, thread-safely, on first use there
  struct Init {
    cudaError_t e;
    int clusters;
  };
  static PerDevice<Init> once;
  const Init* init = once.get([] {
    Init r{cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI, OP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmem),
           1};
    if (r.e != cudaSuccess) return r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sm_count(), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    int n = 0;
    r.e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, EPI, OP>, &cfg);
    r.clusters = n > 0 ? n : 1;
    return r;
  });
  if (init == nullptr) return cudaErrorNoDevice;
  if (init->e != cudaSuccess) return init->e;
  const int max_clusters = init->clusters;
  const int num_mp = ((p.M + kBM - 1) / kBM + 1) / 2;
  const int pairs = num_mp * (p.N / BN);
  const int nk = p.K / (OP == kOpF8 ? 128 : kBK);
  // a partial last wave of rem tiles runs as rem x parts K-split items in
  // one shorter wave: parts a power of two <= max_clusters / rem and <= the
  // k-blocks; with 32-column owners at most 8 and BN / 32 (every part owns
  // columns), with 128-column owners (QKV, SWIGLU) at most 2 (on a
  // 128-column tile the second part only contributes its partial); only
  // when the caller gave room for the partials and the flags
  int parts = 1;
  const int rem = pairs % max_clusters;
  if (pairs > max_clusters && rem != 0 && p.part != nullptr && p.flags != nullptr) {
    const int cap = split_own_min<EPI>() == 128 ? split_max_parts<EPI>() : std::min(kMaxKParts, BN / 32);
    static_assert(split_max_parts<EPI>() <= kMaxKParts, "part cap");
    const int lim = std::min(std::min(max_clusters / rem, nk), cap);
    while (parts * 2 <= lim) parts *= 2;
    while (parts > 1 && (gemm_split_bytes(BN, rem, parts) > p.part_bytes ||
                         static_cast<size_t>(rem) * parts * 8 * sizeof(int) > kGemmFlagBytes))
      parts /= 2;
  }
  if (p.parts_out) *p.parts_out = parts;
  const int nfull = parts > 1 ? pairs - rem : pairs;
  const int total = nfull + (parts > 1 ? rem * parts : 0);
  const int clusters = std::min(total, max_clusters);
  const int group = raster_group(num_mp, p.K, OP == kOpF8 ? 1 : 2);
  EpiArgs ep{p.out, p.ldo, p.gate, p.qkv, p.sa, p.sw, static_cast<float*>(p.part), p.flags, parts, p.epoch};
  gemm_tc_kernel<BN, EPI, OP><<<2 * clusters, C::kThreads, C::kSmem, s>>>(p.tmA, p.tmB, p.tmX, p.M, p.N, p.K, group, nfull,
                                                                  total, ep);
  return cudaGetLastError();
}

template <int OP>
static cudaError_t launch_16(const GemmPlan& p, cudaStream_t s) {
  if (p.bn == 256) {
    switch (p.epi) {
      case EPI_F16: return launch_t<256, EPI_F16, OP>(p, s);
      case EPI_F32: return launch_t<256, EPI_F32, OP>(p, s);
      case EPI_RESID: return launch_t<256, EPI_RESID, OP>(p, s);
      case EPI_SWIGLU: return launch_t<256, EPI_SWIGLU, OP>(p, s);
      case EPI_QKV: return launch_t<256, EPI_QKV, OP>(p, s);
      case EPI_QKV_KV: return launch_t<256, EPI_QKV_KV, OP>(p, s);
    }
  } else {
    switch (p.epi) {
      case EPI_F16: return launch_t<128, EPI_F16, OP>(p, s);
      case EPI_F32: return launch_t<128, EPI_F32, OP>(p, s);
      case EPI_RESID: return launch_t<128, EPI_RESID, OP>(p, s);
      case EPI_SWIGLU: return launch_t<128, EPI_SWIGLU, OP>(p, s);
      case EPI_QKV: return launch_t<128, EPI_QKV, OP>(p, s);
      case EPI_QKV_KV: return launch_t<128, EPI_QKV_KV, OP>(p, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm(const GemmPlan& p, cudaStream_t s) {
  if (p.M <= 0) return cudaSuccess;
  if (p.f8) {
    if (p.bn != 256) return cudaErrorInvalidValue;
    switch (p.epi) {
      case EPI_F32: return launch_t<256, EPI_F32, kOpF8>(p, s);
      case EPI_RESID: return launch_t<256, EPI_RESID, kOpF8>(p, s);
      case EPI_SWIGLU: return launch_t<256, EPI_SWIGLU, kOpF8>(p, s);
      case EPI_QKV: return launch_t<256, EPI_QKV, kOpF8>(p, s);
      case EPI_QKV_KV: return launch_t<256, EPI_QKV_KV, kOpF8>(p, s);
    }
    return cudaErrorInvalidValue;
  }
  return p.dt == DT_BF16 ? launch_16<kOpBF16>(p, s) : launch_16<kOpF16>(p, s);
}

}  // namespace qi21
