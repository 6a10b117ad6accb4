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
// A cluster of two CTAs takes two neighbouring 128-query tiles of one head
// of one sequence and runs both through the pair MMA (cta_group::2, M 256):
// each CTA holds its own Q tile and half of every key block (64 of its 128
// keys for Q K^T, 64 of the 128 head columns of V for P V), so a key block
// crosses from L2 into each SM once per 256 queries, and the MMAs read
// their operands from both CTAs' shared memory. 11 warps per CTA:
//   warp 0     TMA: Q once (2 x 64-column boxes, 128-byte swizzle), then
//              this CTA's halves of the K and V blocks in need order (K
//              two blocks ahead of V) into 6-stage rings; every
//              load signals the even CTA's barrier. The cache part of the
//              key axis is padded to a multiple of 64 so no 64-key box
//              straddles the two sources (padding keys are masked).
//   warp 1     TMEM allocation (both CTAs); in the even CTA the thread
//              issuing S_j = Q K_j^T (M 256, N 128) into one of three TMEM
//              buffers, up to two blocks ahead of P V.
//   warp 10    in the even CTA the thread issuing O += P_j V_j (8 MMAs of
//              K 16, P read from TMEM, V an MN-major operand). The two
//              issuing threads each issue synchronously, so either one's
//              waits overlap the other's MMAs; commits signal both CTAs.
//   warps 2-9  softmax, two per TMEM lane quadrant, each taking 16 of its
//              32 lanes (query rows) through the 16-lane TMEM shapes:
//              thread t holds rows base + t/4 and base + t/4 + 8 and, of
//              every 8-column group, columns 2 (t%4) and 2 (t%4) + 1, so a
//              row's 128 scores sit in 4 threads of one warp and its max
//              and sum are two shuffles. Per block: read S_j, mask, keep a
//              running max per row that is only raised when a block
//              exceeds it by more than 2^8 (then the rows of O are rescaled
//              in TMEM), write P_j = 2^(s - m) as packed 16-bit pairs over
//              the first 64 columns of S_j's buffer (the 16x128b store puts
//              each thread's key pair in its P column) and accumulate the
//              row sums; a lane per warp then signals the even CTA. At the
//              end O / l -> the rows of the output.
// TMEM (each CTA, its 128 rows): S buffers [0, 384), O [384, 512). The
// softmax of block j runs while the tensor cores work on Q K^T of j+1 and
// j+2 and P V of j-2 and j-1. Every wait is bounded.
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
constexpr int kAK = 128;              // keys per block
constexpr int kAD = 128;              // head dim
constexpr int kSub = 128 * 64 * 2;    // one 128-row x 64-column swizzled box: 16 KB (Q)
constexpr int kTileBytes = 2 * kSub;  // Q: 128 x 128
constexpr int kKVBox = 64;            // rows per K / V box (the padding unit of the cache keys)
constexpr int kBox = 64 * 64 * 2;     // one 64 x 64 box: 8 KB
constexpr int kHalf = 2 * kBox;       // this CTA's half of a K block (64 keys x 128) or V block (128 keys x 64)
constexpr int kNK = 6;                // K ring stages
constexpr int kNV = 6;                // V ring stages
constexpr int kNS = 3;                // S / P buffers in TMEM
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kNK * kHalf;
constexpr int kOffBar = kOffV + kNV * kHalf;
constexpr int kNBar = 1 + 2 * kNK + 2 * kNV + 3 * kNS;
constexpr int kAttnSmem = kOffBar + 512 + 1024;
constexpr int kAttnThreads = 352;           // 11 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8 in f16
static_assert(kNBar * 8 + 8 <= 512, "barrier area");

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

// Pair form of the A-from-TMEM MMA: each CTA of the pair supplies its 128
// lanes of A (same TMEM address) and half of B's N columns.
__device__ __forceinline__ void tc_mma_f16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on an mbarrier of the cluster without memory ordering: the data it
// announces (TMEM stores) were completed by tcgen05.wait::st and ordered
// by tcgen05.fence::before_thread_sync.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

#define QI21_A8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                   "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define QI21_I8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                   "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
#define QI21_REGS32 "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, " \
                    "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}"
#define QI21_REGS32_1 "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, " \
                      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32}"

// 16 TMEM lanes from the lane in taddr, 8 repetitions of 8 columns: thread t
// gets rows (t/4, t/4 + 8) x columns (2 (t%4), +1) of each repetition,
// in the order (row, col), (row, col + 1), (row + 8, col), (row + 8, col + 1).
__device__ __forceinline__ void tmem_ld16x256_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 " QI21_REGS32 ", [%32];"
               : QI21_A8(0), QI21_A8(8), QI21_A8(16), QI21_A8(24)
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16x256_x8(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], " QI21_REGS32_1 ";" ::"r"(taddr), QI21_I8(0),
               QI21_I8(8), QI21_I8(16), QI21_I8(24)
               : "memory");
}
// 16 TMEM lanes, 16 repetitions of 4 columns: thread t writes rows (t/4,
// t/4 + 8) of column t%4 of each repetition, row t/4 first.
__device__ __forceinline__ void tmem_st16x128_x16(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x16.b32 [%0], " QI21_REGS32_1 ";" ::"r"(taddr), QI21_I8(0),
               QI21_I8(8), QI21_I8(16), QI21_I8(24)
               : "memory");
}

// key index of virtual key v (cache keys, padding, then own keys), or a
// value no limit reaches for a padding key
__device__ __forceinline__ int key_index(int v, int n_pre, int pad_end) {
  return v < n_pre ? v : (v >= pad_end ? v - pad_end + n_pre : 0x7fffffff);
}

template <bool BF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const AttnTcSeq& sq = p.seq[blockIdx.z];
  const int rank = static_cast<int>(cluster_rank());
  const bool leader = rank == 0;
  const int pq0 = (blockIdx.x >> 1) * (2 * kAQ);  // the pair's first query
  if (pq0 >= sq.nq) return;                       // both CTAs of the pair leave
  const int qt0 = pq0 + rank * kAQ;
  const int h = blockIdx.y;
  const int H = p.H;
  const int ntot = sq.n_pre + sq.n_own;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* qfull = bars;                 // even CTA: both Q tiles landed
  uint64_t* kfull = qfull + 1;            // [kNK] even CTA: both K halves landed
  uint64_t* vfull = kfull + kNK;          // [kNV]
  uint64_t* kempty = vfull + kNV;         // [kNK] both CTAs: stage's Q K^T done
  uint64_t* vempty = kempty + kNK;        // [kNV] both CTAs: stage's P V done
  uint64_t* sfull = vempty + kNV;         // [kNS] both CTAs: S_b written
  uint64_t* pfull = sfull + kNS;          // [kNS] even CTA: both CTAs' P_b written
  uint64_t* pvdone = pfull + kNS;         // [kNS] both CTAs: P V of buffer b done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(pvdone + kNS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  // key blocks the pair walks: cache blocks (padded), then own keys up to
  // the visibility of the pair's last live query (vis is non-decreasing)
  const int q_last = min(pq0 + 2 * kAQ, sq.nq) - 1;
  const int lim_last = sq.vis ? min(ntot, static_cast<int>(__ldg(sq.vis + q_last))) : ntot;
  const int own_need = max(0, lim_last - sq.n_pre);
  const int nkb = (sq.pad_end + own_need + kAK - 1) / kAK;

  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    for (int i = 0; i < kNK; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < kNV; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], 16);  // 8 softmax warps x 2 CTAs
      mbar_init(&pvdone[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.panel);
    tma_prefetch_desc(&p.panel_kv);
    if (sq.n_pre > 0) tma_prefetch_desc(&sq.kvmap);
  }
  if (warp == 1) {
    tmem_alloc_pair(tslot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers and TMEM ready before any remote use
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tS = tmem;        // S buffers at columns [0, 384)
  const uint32_t tO = tmem + 384;  // O at columns [384, 512)
  const uint32_t tP = tS;          // P_b (16-bit pairs, 64 columns) over the first columns of S_b

  if (warp == 0) {
    if (lane == 0) {
      const uint32_t qb = mapa_rank(qfull, 0);
      if (leader) mbar_arrive_expect_tx(qfull, 2 * kTileBytes);
      const int qy = sq.q_row0 + qt0;
      tma_load_2d_pair(smem + kOffQ, &p.panel, qb, h * kAD, qy);
      tma_load_2d_pair(smem + kOffQ + kSub, &p.panel, qb, h * kAD + 64, qy);
      // one 64-key box of K or V columns [col, col + 64), wholly from the
      // cache or wholly from the panel
      auto load_box = [&](uint8_t* dst, uint32_t bar, int v, int col_cache, int col_panel) {
        if (v < sq.n_pre)
          tma_load_2d_pair(dst, &sq.kvmap, bar, col_cache, v);
        else
          tma_load_2d_pair(dst, &p.panel_kv, bar, col_panel, sq.own_row0 + (v - sq.pad_end));
      };
      // K half: keys [128 j + 64 rank, + 64), all 128 head columns
      auto load_k = [&](int j) -> bool {
        const int st = j % kNK;
        if (!mbar_wait(&kempty[st], ((j / kNK) & 1) ^ 1u, abort_flag, &s_attn_status)) return false;
        if (leader) mbar_arrive_expect_tx(&kfull[st], 2 * kHalf);
        const uint32_t fb = mapa_rank(&kfull[st], 0);
        uint8_t* d = smem + kOffK + st * kHalf;
        const int v = j * kAK + rank * kKVBox;
        load_box(d, fb, v, h * kAD, H + h * kAD);
        load_box(d + kBox, fb, v, h * kAD + 64, H + h * kAD + 64);
        return true;
      };
      // V half: all 128 keys of the block, head columns [64 rank, + 64)
      auto load_v = [&](int j) -> bool {
        const int st = j % kNV;
        if (!mbar_wait(&vempty[st], ((j / kNV) & 1) ^ 1u, abort_flag, &s_attn_status)) return false;
        if (leader) mbar_arrive_expect_tx(&vfull[st], 2 * kHalf);
        const uint32_t fb = mapa_rank(&vfull[st], 0);
        uint8_t* d = smem + kOffV + st * kHalf;
        const int c = h * kAD + rank * 64;
        load_box(d, fb, j * kAK, H + c, 2 * H + c);
        load_box(d + kBox, fb, j * kAK + kKVBox, H + c, 2 * H + c);
        return true;
      };
      // need order: K_0, K_1, then V_j before K_{j+2}
      bool ok = true;
      for (int j = 0; j < min(2, nkb) && ok; ++j) ok = load_k(j);
      for (int j = 0; j < nkb && ok; ++j) {
        ok = load_v(j);
        if (ok && j + 2 < nkb) ok = load_k(j + 2);
      }
    }
  } else if (warp == 1 || warp == 10) {
    // the even CTA's two MMA-issuing threads: Q K^T (warp 1) and P V (warp
    // 10), each issuing synchronously, so either one's waits overlap the
    // other's MMAs
    if (lane == 0 && leader) {
      bool ok = true;
      if (warp == 1) {
        constexpr uint32_t idesc_qk = idesc_f16(2 * kAQ, kAK, false, BF);
        const uint32_t sQ = smem_u32(smem + kOffQ);
        ok = mbar_wait(qfull, 0, abort_flag, &s_attn_status);
        for (int j = 0; j < nkb && ok; ++j) {
          const int b = j % kNS;
          // S_b is free once the P V that read P_{j-3} from it is done
          if (j >= kNS && !mbar_wait(&pvdone[b], ((j - kNS) / kNS) & 1, abort_flag, &s_attn_status)) break;
          const int st = j % kNK;
          if (!mbar_wait(&kfull[st], (j / kNK) & 1, abort_flag, &s_attn_status)) break;
          tc_fence_after();
          const uint32_t sK = smem_u32(smem + kOffK + st * kHalf);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc_mma_f16_pair(tS + b * kAK, sdesc_sw128(sQ + (k >> 2) * kSub) + 2 * (k & 3),
                            sdesc_sw128(sK + (k >> 2) * kBox) + 2 * (k & 3), idesc_qk, k > 0 ? 1u : 0u);
          tc_commit_pair(&kempty[st], 0x3);
          tc_commit_pair(&sfull[b], 0x3);
        }
      } else {
        constexpr uint32_t idesc_pv = idesc_f16(2 * kAQ, kAD, true, BF);  // V: MN-major
        for (int j = 0; j < nkb; ++j) {
          const int b = j % kNS;
          if (!mbar_wait(&pfull[b], (j / kNS) & 1, abort_flag, &s_attn_status)) break;
          const int st = j % kNV;
          if (!mbar_wait(&vfull[st], (j / kNV) & 1, abort_flag, &s_attn_status)) break;
          tc_fence_after();
          const uint32_t sV = smem_u32(smem + kOffV + st * kHalf);
#pragma unroll
          for (int k = 0; k < kAK / 16; ++k) {
            // A = P in TMEM: 128 query lanes x 16 keys = 8 columns of 16-bit
            // pairs; B = this CTA's 64 V columns of 16 key rows, columns
            // contiguous (128-byte rows, 8-row groups 1 KB apart)
            const uint64_t bd = sdesc(sV + k * 2048, kBox, 1024, 2);
            tc_mma_f16_ts_pair(tO, tP + b * kAK + k * 8, bd, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit_pair(&vempty[st], 0x3);
          tc_commit_pair(&pvdone[b], 0x3);
        }
      }
    }
  } else {
    // softmax: warps 2-9, two per TMEM lane quadrant, each taking 16 of its
    // 32 lanes (query rows) through the 16-lane TMEM shapes: thread t holds
    // rows r0 = base + t/4 and r1 = r0 + 8, columns 8k + 2(t%4) and + 1 of
    // each 8-column group k; a row's 128 scores sit in 4 threads of the
    // warp, whose row max and sum are two shuffles (no cross-warp step)
    const int q = warp & 3;
    const int hh = (warp - 2) >> 2;
    const int lbase = q * 32 + hh * 16;
    const int tq = lane >> 2, tj = lane & 3;
    const int r0 = lbase + tq, r1 = r0 + 8;
    const int qi0 = qt0 + r0, qi1 = qt0 + r1;
    const bool live0 = qi0 < sq.nq, live1 = qi1 < sq.nq;
    const int lim0 = (sq.vis && live0) ? min(ntot, static_cast<int>(__ldg(sq.vis + qi0))) : lim_last;
    const int lim1 = (sq.vis && live1) ? min(ntot, static_cast<int>(__ldg(sq.vis + qi1))) : lim_last;
    const uint32_t lane_off = static_cast<uint32_t>(lbase) << 16;
    const float c = p.scale_log2;
    const uint64_t c2 = f2(c, c);
    const uint32_t pf_remote = leader ? 0u : mapa_rank(pfull, 0);
    float m0 = -INFINITY, m1 = -INFINITY;
    uint64_t lacc = 0ull;  // (row r0, row r1) partial sums of this thread's columns
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      const int b = j % kNS;
      if (!mbar_wait(&sfull[b], (j / kNS) & 1, abort_flag, &s_attn_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[2][32];  // [half of the 128 columns][8 groups x (r0 c, r0 c+1, r1 c, r1 c+1)]
      tmem_ld16x256_x8(tS + b * kAK + lane_off, s[0]);
      tmem_ld16x256_x8(tS + b * kAK + 64 + lane_off, s[1]);
      tmem_ld_wait(s[0]);
      tmem_ld_wait(s[1]);
      const int v0 = j * kAK;
      const int k0 = key_index(v0, sq.n_pre, sq.pad_end);
      const int k1 = key_index(v0 + kAK - 1, sq.n_pre, sq.pad_end);
      const bool same_src = (v0 + kAK <= sq.n_pre) || (v0 >= sq.pad_end);
      if (!(same_src && k1 < min(lim0, lim1) && k0 < min(lim0, lim1))) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int g = 0; g < 8; ++g)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int col = hf * 64 + 8 * g + 2 * tj + (e & 1);
              const int kj = key_index(v0 + col, sq.n_pre, sq.pad_end);
              if (kj >= ((e & 2) ? lim1 : lim0)) s[hf][4 * g + e] = __float_as_uint(-INFINITY);
            }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, my0 = -INFINITY, my1 = -INFINITY;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int g = 0; g < 8; g += 2) {
          mx0 = max3(mx0, __uint_as_float(s[hf][4 * g + 0]), __uint_as_float(s[hf][4 * g + 1]));
          mx1 = max3(mx1, __uint_as_float(s[hf][4 * g + 2]), __uint_as_float(s[hf][4 * g + 3]));
          my0 = max3(my0, __uint_as_float(s[hf][4 * g + 4]), __uint_as_float(s[hf][4 * g + 5]));
          my1 = max3(my1, __uint_as_float(s[hf][4 * g + 6]), __uint_as_float(s[hf][4 * g + 7]));
        }
      mx0 = fmaxf(mx0, my0);
      mx1 = fmaxf(mx1, my1);
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mb0 = mx0 * c, mb1 = mx1 * c;
      // raise each row's running max only past the threshold (exact: O and
      // l share the stale max; P <= 2^threshold stays in f16 range)
      float al0 = 1.f, al1 = 1.f;
      const bool need0 = mb0 > m0 + kRescaleThreshold, need1 = mb1 > m1 + kRescaleThreshold;
      if (need0) {
        al0 = ex2(m0 - mb0);
        m0 = mb0;
      }
      if (need1) {
        al1 = ex2(m1 - mb1);
        m1 = mb1;
      }
      {
        float la, lb;
        unf2(lacc, la, lb);
        lacc = f2(la * al0, lb * al1);
      }
      const bool warp_rescale = __any_sync(0xffffffffu, (need0 || need1) && j > 0);
      // P pairs -> TMEM through the 16x128b shape: group G = 8 hf + g
      // (keys 8 G + 2 t%4, + 1) is P column 4 G + t%4, rows r0 then r1
      const uint64_t nm0 = f2(-m0, -m0), nm1 = f2(-m1, -m1);
      uint32_t pk[32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          float a0, a1, b0, b1;
          unf2(ffma2(f2(__uint_as_float(s[hf][4 * g + 0]), __uint_as_float(s[hf][4 * g + 1])), c2, nm0), a0, a1);
          unf2(ffma2(f2(__uint_as_float(s[hf][4 * g + 2]), __uint_as_float(s[hf][4 * g + 3])), c2, nm1), b0, b1);
          const float p00 = ex2(a0), p01 = ex2(a1), p10 = ex2(b0), p11 = ex2(b1);
          lacc = fadd2(lacc, f2(p00 + p01, p10 + p11));
          pk[2 * (8 * hf + g)] = pack2<BF>(p00, p01);
          pk[2 * (8 * hf + g) + 1] = pack2<BF>(p10, p11);
        }
      tmem_st16x128_x16(tP + b * kAK + lane_off, pk);
      if (warp_rescale) {
        // O is stable once the P V of block j - 1 is done
        if (!mbar_wait(&pvdone[(j - 1) % kNS], ((j - 1) / kNS) & 1, abort_flag, &s_attn_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t o[32];
          tmem_ld16x256_x8(tO + hf * 64 + lane_off, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            o[4 * g + 0] = __float_as_uint(__uint_as_float(o[4 * g + 0]) * al0);
            o[4 * g + 1] = __float_as_uint(__uint_as_float(o[4 * g + 1]) * al0);
            o[4 * g + 2] = __float_as_uint(__uint_as_float(o[4 * g + 2]) * al1);
            o[4 * g + 3] = __float_as_uint(__uint_as_float(o[4 * g + 3]) * al1);
          }
          tmem_st16x256_x8(tO + hf * 64 + lane_off, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&pfull[b]);
        else
          mbar_arrive_cluster_relaxed(pf_remote + static_cast<uint32_t>(b * 8));
      }
    }
    float l0, l1;
    unf2(lacc, l0, l1);
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (ok && nkb > 0 &&
        mbar_wait(&pvdone[(nkb - 1) % kNS], ((nkb - 1) / kNS) & 1, abort_flag, &s_attn_status)) {
      tc_fence_after();
      const float inv0 = 1.f / l0, inv1 = 1.f / l1;
      uint16_t* orow0 = static_cast<uint16_t*>(p.out) + static_cast<size_t>(sq.q_row0 + qi0) * H + h * kAD;
      uint16_t* orow1 = static_cast<uint16_t*>(p.out) + static_cast<size_t>(sq.q_row0 + qi1) * H + h * kAD;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t o[32];
        tmem_ld16x256_x8(tO + hf * 64 + lane_off, o);
        tmem_ld_wait(o);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const int col = hf * 64 + 8 * g + 2 * tj;
          if (live0)
            *reinterpret_cast<uint32_t*>(orow0 + col) =
                pack2<BF>(__uint_as_float(o[4 * g + 0]) * inv0, __uint_as_float(o[4 * g + 1]) * inv0);
          if (live1)
            *reinterpret_cast<uint32_t*>(orow1 + col) =
                pack2<BF>(__uint_as_float(o[4 * g + 2]) * inv1, __uint_as_float(o[4 * g + 3]) * inv1);
        }
      }
    }
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // neither CTA leaves while the pair's MMAs may use its memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
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
  p->gx = 2 * ((maxq + 2 * kAQ - 1) / (2 * kAQ));  // CTA pairs of two query tiles
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
