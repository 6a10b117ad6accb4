// Flash attention over [prefix cache, own panel rows] with a leading-run
// visibility mask, on the 5th-generation tensor cores (qwen_image21.rs,
// Qi21Dit::attention + softmax_prefix; gpu_wgpu/qi21.rs, qi_flash). Q, K,
// V, P and the output are f16, or bf16 in the bf16 instance (BF), with f32
// scores, softmax and accumulation either way.
//
// Query i of a sequence sees keys [0, lim(i)), lim(i) = min(vis[i], keys)
// in the prefill (block-causal) and every key in a step. Keys j < n_pre
// come from the layer's cache [n_pre][2H] (K then V), the rest from the
// panel rows own_row0 + j - n_pre (K at column H, V at 2H).
//
// CTA = one 128-query tile of one head of one sequence, 10 warps:
//   warp 0     TMA: Q once (2 x 64-column boxes, 128-byte swizzle), then K
//              and V blocks of 192 keys into 2-stage rings, each block as
//              three 64-key boxes. The cache part of the key axis is padded
//              to a multiple of 64 so no box straddles the two sources
//              (padding keys are masked); a block may hold cache and panel
//              boxes, so at most 63 padding keys are computed per query.
//   warp 1     TMEM allocation and the single MMA-issuing thread:
//              S_j = Q K_j^T (M 128, N 192) into one of two TMEM buffers
//              (kind::f16, f32 accumulate), then O += P_j V_j (12 MMAs of
//              K 16) with P read from TMEM and V an MN-major shared-memory
//              operand.
//   warps 2-9  softmax: two warps per TMEM lane quadrant, each owning 96 of
//              the 192 key columns of its 32 query rows. Per block: read S_j
//              with tcgen05.ld, mask, exchange the partial row max with the
//              partner warp (a bounded mbarrier rendezvous), keep a running
//              max that is only raised when a block exceeds it by more than
//              2^8 (then O is rescaled in TMEM), write P_j = 2^(s - m) as
//              packed f16 pairs over the first 96 columns of S_j's buffer
//              (the A operand of P V; both warps of the quadrant have read
//              their S by then) and accumulate the row sum; at the end
//              O / l -> f16 rows of the output.
// TMEM: S buffers [0, 192), [192, 384), O [384, 512). The QK^T of block
// j+1 and the P V of block j-1 run on the tensor cores while the softmax of
// block j runs on the ALUs; 192-key blocks (against 128) spread each
// block's fixed handshake cost over 1.5x the MMA work. Every wait is
// bounded.
#include <algorithm>
#include <cstdio>

#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace qi21 {

static __device__ unsigned int s_attn_status = 0;

unsigned int attn_status_read_clear() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, s_attn_status, sizeof v);
  cudaMemcpyToSymbol(s_attn_status, &z, sizeof z);
  return v;
}

constexpr int kAQ = 128;              // queries per CTA
constexpr int kAK = 192;              // keys per block
constexpr int kAD = 128;              // head dim
constexpr int kSub = 128 * 64 * 2;    // one 128-row x 64-column f16 swizzled box: 16 KB (Q)
constexpr int kTileBytes = 2 * kSub;  // Q: 128 x 128 f16
constexpr int kKVSub = kAK * 64 * 2;  // 192 rows x 64 columns of a K or V block: 24 KB
constexpr int kKVBox = 64;            // rows per K / V box (the padding unit of the cache keys)
constexpr int kKVBytes = 2 * kKVSub;  // a K or V block: 192 x 128 f16
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;    // 2 stages
constexpr int kOffV = kOffK + 2 * kKVBytes;  // 2 stages
constexpr int kOffBar = kOffV + 2 * kKVBytes;
constexpr int kOffX = kOffBar + 256;        // partial row max / sum exchange [2][128] f32
constexpr int kAttnSmem = kOffX + 1024 + 1024;
constexpr int kAttnThreads = 320;           // 10 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 in f16

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}


__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16 columns of 32-bit stored from registers to this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}

// key index of virtual key v (cache keys, padding, then own keys), or a
// value no limit reaches for a padding key
__device__ __forceinline__ int key_index(int v, int n_pre, int pad_end) {
  return v < n_pre ? v : (v >= pad_end ? v - pad_end + n_pre : 0x7fffffff);
}

template <bool BF>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_kernel(const __grid_constant__ AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const AttnTcSeq& sq = p.seq[blockIdx.z];
  const int qt0 = blockIdx.x * kAQ;
  if (qt0 >= sq.nq) return;
  const int h = blockIdx.y;
  const int H = p.H;
  const int ntot = sq.n_pre + sq.n_own;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* qfull = bars + 0;
  uint64_t* kfull = bars + 1;    // [2]
  uint64_t* vfull = bars + 3;    // [2]
  uint64_t* kempty = bars + 5;   // [2] K stage free (its QK^T done)
  uint64_t* vempty = bars + 7;   // [2] V stage free (its P V done)
  uint64_t* sfull = bars + 9;    // [2]
  uint64_t* pfull = bars + 11;   // [2], one per P buffer
  uint64_t* pvdone = bars + 13;  // [2], one per P buffer
  uint64_t* xbar = bars + 15;    // [4], the two softmax warps of a lane quadrant
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 19);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  // key blocks this tile walks: cache blocks (padded), then own keys up to
  // the visibility of the tile's last live query (vis is non-decreasing)
  const int q_last = min(qt0 + kAQ, sq.nq) - 1;
  const int lim_last = sq.vis ? min(ntot, static_cast<int>(__ldg(sq.vis + q_last))) : ntot;
  const int own_need = max(0, lim_last - sq.n_pre);
  const int nkb = (sq.pad_end + own_need + kAK - 1) / kAK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 15; ++i) mbar_init(&bars[i], (i == 11 || i == 12) ? 256 : 1);
    for (int i = 15; i < 19; ++i) mbar_init(&bars[i], 64);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.panel);
    tma_prefetch_desc(&p.panel_kv);
    if (sq.n_pre > 0) tma_prefetch_desc(&sq.kvmap);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem;         // S buffers at columns [0, 192), [192, 384)
  const uint32_t tO = tmem + 384;   // O at columns [384, 512)
  // P_b (f16 pairs, 96 columns) over the first columns of S_b: written only
  // after both warps of a quadrant have read their S (the row-max exchange)
  const uint32_t tP = tS;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(qfull, kTileBytes);
      const int qy = sq.q_row0 + qt0;
      tma_load_2d(smem + kOffQ, &p.panel, qfull, h * kAD, qy);
      tma_load_2d(smem + kOffQ + kSub, &p.panel, qfull, h * kAD + 64, qy);
      // need order: K_{j+1} (for QK^T one block ahead), then V_j (for P V)
      // a K or V block = three 64-key boxes, each wholly from the cache
      // (keys padded to a multiple of 64) or wholly from the panel
      auto load_kv = [&](uint8_t* dst, uint64_t* bar, int j, int col_cache, int col_panel) {
#pragma unroll
        for (int sb = 0; sb < kAK / kKVBox; ++sb) {
          const int v = j * kAK + sb * kKVBox;
          uint8_t* d = dst + sb * kKVBox * 128;
          if (v < sq.n_pre) {
            tma_load_2d(d, &sq.kvmap, bar, col_cache, v);
            tma_load_2d(d + kKVSub, &sq.kvmap, bar, col_cache + 64, v);
          } else {
            const int row = sq.own_row0 + (v - sq.pad_end);
            tma_load_2d(d, &p.panel_kv, bar, col_panel, row);
            tma_load_2d(d + kKVSub, &p.panel_kv, bar, col_panel + 64, row);
          }
        }
      };
      auto load_k = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&kempty[st], ((j >> 1) & 1) ^ 1u, abort_flag, &s_attn_status)) return false;
        mbar_arrive_expect_tx(&kfull[st], kKVBytes);
        load_kv(smem + kOffK + st * kKVBytes, &kfull[st], j, h * kAD, H + h * kAD);
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&vempty[st], ((j >> 1) & 1) ^ 1u, abort_flag, &s_attn_status)) return false;
        mbar_arrive_expect_tx(&vfull[st], kKVBytes);
        load_kv(smem + kOffV + st * kKVBytes, &vfull[st], j, H + h * kAD, 2 * H + h * kAD);
        return true;
      };
      bool ok = load_k(0);
      for (int j = 0; j < nkb && ok; ++j) {
        if (j + 1 < nkb && !load_k(j + 1)) break;
        ok = load_v(j);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(128, kAK, false, BF);
      constexpr uint32_t idesc_pv = idesc_f16(128, 128, true, BF);  // V: MN-major
      const uint32_t sQ = smem_u32(smem + kOffQ);
      bool ok = mbar_wait(qfull, 0, abort_flag, &s_attn_status);
      auto issue_qk = [&](int j) -> bool {
        const int s = j & 1;
        if (!mbar_wait(&kfull[s], (j >> 1) & 1, abort_flag, &s_attn_status)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + kOffK + s * kKVBytes);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc_mma_f16(tS + (j & 1) * kAK, sdesc_sw128(sQ + (k >> 2) * kSub) + 2 * (k & 3),
                     sdesc_sw128(sK + (k >> 2) * kKVSub) + 2 * (k & 3), idesc_qk, k > 0 ? 1u : 0u);
        tc_commit(&kempty[s]);
        tc_commit(&sfull[j & 1]);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; j < nkb && ok; ++j) {
        if (j + 1 < nkb && !issue_qk(j + 1)) break;
        const int pb = j & 1;
        if (!mbar_wait(&pfull[pb], (j >> 1) & 1, abort_flag, &s_attn_status)) break;
        const int s = j & 1;
        if (!mbar_wait(&vfull[s], (j >> 1) & 1, abort_flag, &s_attn_status)) break;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + kOffV + s * kKVBytes);
#pragma unroll
        for (int k = 0; k < kAK / 16; ++k) {
          // A = P in TMEM: 128 query lanes x 16 keys = 8 columns of f16
          // pairs; B = V: 16 key rows x 128 d, d contiguous (two 64-wide
          // atoms kKVSub apart, 8-row groups 1 KB)
          const uint64_t b = sdesc(sV + k * 2048, kKVSub, 1024, 2);
          tc_mma_f16_ts(tO, tP + pb * kAK + k * 8, b, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(&vempty[s]);
        tc_commit(&pvdone[pb]);
      }
    }
  } else {
    // softmax warps: quadrant q of the TMEM lanes = query rows 32q .. 32q+31,
    // half hf = key columns [64 hf, 64 hf + 64) of every block
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const int qi = qt0 + r;
    const bool live = qi < sq.nq;
    const int lim = (sq.vis && live) ? min(ntot, static_cast<int>(__ldg(sq.vis + qi))) : lim_last;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + kOffX);  // [2][128]
    const float c = p.scale_log2;
    const uint64_t c2 = f2(c, c);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // bounded rendezvous of the two warps of this quadrant
    uint32_t xph = 0;
    auto pair_sync = [&]() -> bool {
      mbar_arrive(&xbar[q]);
      const bool r_ok = mbar_wait(&xbar[q], xph, abort_flag, &s_attn_status);
      xph ^= 1u;
      return r_ok;
    };
    for (int j = 0; j < nkb; ++j) {
      const int b = j & 1;
      if (!mbar_wait(&sfull[b], (j >> 1) & 1, abort_flag, &s_attn_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      constexpr int kHalf = kAK / 2;  // 96 key columns per warp
      uint32_t s[3][32];
#pragma unroll
      for (int cc = 0; cc < 3; ++cc) tmem_ld32(tS + b * kAK + lane_off + hf * kHalf + cc * 32, s[cc]);
#pragma unroll
      for (int cc = 0; cc < 3; ++cc) tmem_ld_wait(s[cc]);
      const int v0 = j * kAK + hf * kHalf;
      // every key of this half-block visible to this row?
      const int k0 = key_index(v0, sq.n_pre, sq.pad_end);
      const int k1 = key_index(v0 + kHalf - 1, sq.n_pre, sq.pad_end);
      const bool same_src = (v0 + kHalf <= sq.n_pre) || (v0 >= sq.pad_end);
      if (!(same_src && k1 < lim && k0 < lim)) {
#pragma unroll
        for (int cc = 0; cc < 3; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int kj = key_index(v0 + cc * 32 + e, sq.n_pre, sq.pad_end);
            if (kj >= lim) s[cc][e] = __float_as_uint(-INFINITY);
          }
      }
      float mx[6];
#pragma unroll
      for (int a = 0; a < 6; ++a) mx[a] = __uint_as_float(s[a >> 1][(a & 1) * 16]);
#pragma unroll
      for (int a = 0; a < 6; ++a)
#pragma unroll
        for (int e = 1; e < 15; e += 2)
          mx[a] = max3(mx[a], __uint_as_float(s[a >> 1][(a & 1) * 16 + e]),
                       __uint_as_float(s[a >> 1][(a & 1) * 16 + e + 1]));
#pragma unroll
      for (int a = 0; a < 6; ++a) mx[a] = fmaxf(mx[a], __uint_as_float(s[a >> 1][(a & 1) * 16 + 15]));
      const float pmax = max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), mx[0]);
      // the partner warp holds the other 64 columns of these rows
      xch[hf * 128 + r] = pmax;
      if (!pair_sync()) {
        ok = false;
        break;
      }
      const float omax = xch[(hf ^ 1) * 128 + r];
      if (!pair_sync()) {
        ok = false;
        break;
      }
      const float mb = fmaxf(pmax, omax) * c;
      // raise the running max only past the threshold (exact: O and l share
      // the stale max; P <= 2^threshold stays in f16 range)
      float alpha = 1.f;
      const bool need = mb > m + kRescaleThreshold;
      if (need) {
        alpha = ex2(m - mb);
        m = mb;
        l *= alpha;
      }
      const bool warp_rescale = __any_sync(0xffffffffu, need && j > 0);
      if (j >= 2) {
        // P buffer b was last read by the P V of block j - 2
        if (!mbar_wait(&pvdone[b], ((j - 2) >> 1) & 1, abort_flag, &s_attn_status)) {
          ok = false;
          break;
        }
      }
      // this half of the P row -> TMEM: 96 keys = 48 columns of 16-bit pairs
      // (32 + 16) over S_b
      const uint64_t nm2 = f2(-m, -m);
      uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t pk[32];
        const int npairs = part == 0 ? 32 : 16;
#pragma unroll
        for (int i = 0; i < npairs; ++i) {
          const int k = 2 * (32 * part + i);
          const uint64_t x =
              ffma2(f2(__uint_as_float(s[k >> 5][k & 31]), __uint_as_float(s[k >> 5][(k & 31) + 1])), c2, nm2);
          float x0, x1;
          unf2(x, x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          acc[i & 3] = fadd2(acc[i & 3], f2(p0, p1));
          pk[i] = pack2<BF>(p0, p1);
        }
        if (part == 0)
          tmem_st32(tP + b * kAK + hf * (kHalf / 2) + lane_off, pk);
        else
          tmem_st16(tP + b * kAK + hf * (kHalf / 2) + 32 + lane_off, pk);
      }
      {
        const uint64_t t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
        float t0, t1;
        unf2(t, t0, t1);
        l += t0 + t1;
      }
      if (warp_rescale) {
        // O is stable once the P V of block j - 1 is done
        if (!mbar_wait(&pvdone[b ^ 1], ((j - 1) >> 1) & 1, abort_flag, &s_attn_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + hf * 64 + cc * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + lane_off + hf * 64 + cc * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&pfull[b]);
    }
    if (ok && mbar_wait(&pvdone[(nkb - 1) & 1], ((nkb - 1) >> 1) & 1, abort_flag, &s_attn_status)) {
      tc_fence_after();
      xch[hf * 128 + r] = l;
      pair_sync();
      const float inv = 1.f / (l + xch[(hf ^ 1) * 128 + r]);
      uint16_t* orow = static_cast<uint16_t*>(p.out) + static_cast<size_t>(sq.q_row0 + qi) * H + h * kAD + hf * 64;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + hf * 64 + cc * 32, o);
        tmem_ld_wait(o);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
          for (int g = 0; g < 4; ++g)
            dst[g] = make_uint4(
                pack2<BF>(__uint_as_float(o[8 * g + 0]) * inv, __uint_as_float(o[8 * g + 1]) * inv),
                pack2<BF>(__uint_as_float(o[8 * g + 2]) * inv, __uint_as_float(o[8 * g + 3]) * inv),
                pack2<BF>(__uint_as_float(o[8 * g + 4]) * inv, __uint_as_float(o[8 * g + 5]) * inv),
                pack2<BF>(__uint_as_float(o[8 * g + 6]) * inv, __uint_as_float(o[8 * g + 7]) * inv));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host ----

static PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
  // resolved once, thread-safely, on first use
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

static cudaError_t encode_rows(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_rows,
                               int dt) {
  auto fn = attn_encode_fn();
  if (fn == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType type = dt == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  auto encode = [&] {
    return fn(m, type, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  CUresult r = encode();
  // a host thread whose first library call this is may have no context yet
  if (r == CUDA_ERROR_INVALID_CONTEXT && bind_primary_context()) r = encode();
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_attn_plan(const AttnArgs& in, AttnPlan* p) {
  if (in.dt != DT_F16 && in.dt != DT_BF16) return cudaErrorInvalidValue;
  memset(p, 0, sizeof *p);
  AttnTcParams& prm = p->prm;
  const int H = in.heads * kAD;
  p->dt = in.dt;
  prm.out = in.out;
  prm.H = H;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(kAD)));
  cudaError_t e = encode_rows(&prm.panel, in.panel, static_cast<uint64_t>(3) * H, in.panel_rows, kAQ, in.dt);
  if (e == cudaSuccess)
    e = encode_rows(&prm.panel_kv, in.panel, static_cast<uint64_t>(3) * H, in.panel_rows, kKVBox, in.dt);
  if (e != cudaSuccess) return e;
  int maxq = 0;
  for (int i = 0; i < in.nseq; ++i) {
    const AttnSeq& a = in.seq[i];
    AttnTcSeq& t = prm.seq[i];
    t.vis = a.vis;
    t.n_pre = a.n_pre;
    t.pad_end = (a.n_pre + kKVBox - 1) / kKVBox * kKVBox;
    t.q_row0 = a.q_row0;
    t.nq = a.nq;
    t.own_row0 = a.own_row0;
    t.n_own = a.n_own;
    if (a.n_pre > 0) {
      e = encode_rows(&t.kvmap, a.kv_pre, static_cast<uint64_t>(2) * H, a.n_pre, kKVBox, in.dt);
      if (e != cudaSuccess) return e;
    }
    maxq = std::max(maxq, a.nq);
  }
  p->gx = (maxq + kAQ - 1) / kAQ;
  p->gy = in.heads;
  p->gz = in.nseq;
  return cudaSuccess;
}

template <bool BF>
static cudaError_t launch_attn_t(const AttnPlan& p, cudaStream_t s) {
  // shared-memory opt-in, once per instance and device
  static PerDevice<cudaError_t> once;
  const cudaError_t* attr = once.get(
      [] { return cudaFuncSetAttribute(attn_tc_kernel<BF>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem); });
  if (attr == nullptr) return cudaErrorNoDevice;
  if (*attr != cudaSuccess) return *attr;
  attn_tc_kernel<BF><<<dim3(p.gx, p.gy, p.gz), kAttnThreads, kAttnSmem, s>>>(p.prm);
  return cudaGetLastError();
}

cudaError_t launch_attn_plan(const AttnPlan& p, cudaStream_t s) {
  if (p.gx == 0) return cudaSuccess;
  return p.dt == DT_BF16 ? launch_attn_t<true>(p, s) : launch_attn_t<false>(p, s);
}

cudaError_t launch_attention(const AttnArgs& in, cudaStream_t s) {
  AttnPlan p;
  const cudaError_t e = make_attn_plan(in, &p);
  if (e != cudaSuccess) return e;
  return launch_attn_plan(p, s);
}

}  // namespace qi21
