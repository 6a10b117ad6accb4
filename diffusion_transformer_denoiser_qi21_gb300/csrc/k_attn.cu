// Flash attention over [prefix cache, own panel rows] with a leading-run
// visibility mask, on the 5th-generation tensor cores (qwen_image21.rs,
// Qi21Dit::attention + softmax_prefix; gpu_wgpu/qi21.rs, qi_flash). Q, K,
// V, P and the output are f16, or bf16 in the bf16 instance (BF), with f32
// scores, softmax and accumulation either way.
//
// Query i of a sequence sees keys [0, lim(i)), lim(i) = min(vis[i], keys)
// in the prefill (block-causal) and every key in a step. Keys j < n_pre
// come from the layer's cache [n_pre][2H] (K then V), the rest from the
// panel rows own_row0 + j - n_pre (K at column H, V at 2H). The cache part
// of the key axis is padded to a multiple of 64 so that every 64-key box
// comes from one source; padding keys are masked.
//
// Work item = two 128-query tiles ("stages" 0 and 1) of one head of one
// sequence, which share every 128-key K and V block. Persistent CTAs, one
// per SM. In a step (every key visible) the items' key blocks are laid end
// to end and each CTA takes an equal run of them (stream-K): an item cut
// by a CTA boundary is done in two parts whose partial (O, max, sum) the
// part that finishes second merges. Otherwise CTA c takes items c, c + G,
// ... whole. 10 warps:
//   warp 0     TMA: the two Q tiles of each item (one buffer, reloaded per
//              stage once that stage's last Q K^T is done), then the K and
//              V blocks in need order (K_0, V_0, K_1, V_1, ...) through a
//              5-slot ring of 32 KB slots.
//   warp 1     TMEM allocation and the single MMA-issuing thread, in the
//              order  S0_j = Q0 K_j^T, O1 += P1_{j-1} V_{j-1},
//                     S1_j = Q1 K_j^T, O0 += P0_j V_j, ...
//              so that the softmax of one stage runs while the tensor cores
//              work for the other (kind::f16, f32 accumulation; P is read
//              from TMEM, V is an MN-major shared-memory operand).
//   warps 2-5  softmax of stage 0, warps 6-9 of stage 1: one thread per
//              query row, 128 keys per block. Read S with tcgen05.ld,
//              mask, row max, keep a running max that is only raised when a
//              block exceeds it by more than 2^8 (then O is rescaled in
//              TMEM), write P = 2^(s - m) as packed 16-bit pairs over the
//              first 64 columns of the stage's S buffer, accumulate the row
//              sum; after the item's last block read O, release it and store
//              O / l (or the partial).
// TMEM: S0 [0, 128), S1 [128, 256), O0 [256, 384), O1 [384, 512). Every
// wait is bounded; a role that gives up lets its in-flight copies and
// MMAs finish before the CTA leaves.
#include <algorithm>
#include <cstdio>
#include <cstring>

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

constexpr int kAQ = 128;                   // queries per stage tile
constexpr int kAK = 128;                   // keys per block
constexpr int kAD = 128;                   // head dim
constexpr int kQBox = 128 * 64 * 2;        // 128 rows x 64 columns, 16 KB
constexpr int kQTile = 2 * kQBox;          // one stage's Q: 32 KB
constexpr int kKVBox = 64;                 // keys per TMA box (the cache padding unit)
constexpr int kBoxBytes = kKVBox * 64 * 2;  // 8 KB
constexpr int kKVHalf = kAK * 64 * 2;      // 128 keys x 64 columns of a block: 16 KB
constexpr int kKVBytes = 2 * kKVHalf;      // a K or V block: 32 KB
constexpr int kSlots = 5;                  // K/V ring slots
constexpr int kOffQ = 0;
constexpr int kOffRing = 2 * kQTile;
constexpr int kOffBar = kOffRing + kSlots * kKVBytes;
constexpr int kAttnSmem = kOffBar + 256 + 1024;
constexpr int kAttnThreads = 320;          // 10 warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P <= 2^8
constexpr int kPartFloats = kAQ * kAD + 2 * kAQ;  // one stage's partial: O^T [128][128], m [128], l [128]

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

// Named barrier of the 128 threads of one softmax stage.
__device__ __forceinline__ void stage_sync(int q) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + q), "r"(128) : "memory");
}

// key index of virtual key v (cache keys, padding, then own keys), or a
// value no limit reaches for a padding key
__device__ __forceinline__ int key_index(int v, int n_pre, int pad_end) {
  return v < n_pre ? v : (v >= pad_end ? v - pad_end + n_pre : 0x7fffffff);
}

// ------------------------------------------------------------ schedule ----

struct Seg {
  int z, h, pr;  // sequence, head, query pair (queries [256 pr, 256 pr + 256))
  int b0, b1;    // key blocks [b0, b1) of the item
  int part;      // -1: the whole item; 0 / 1: its first / second part
  int slot;      // merge slot of a split item (the CTA boundary it straddles)
};

// Key blocks of item (sequence sq, pair pr): every key in a step; in the
// prefill up to the visibility of the pair's last live query.
__device__ __forceinline__ int item_blocks(const AttnTcSeq& sq, int pr) {
  if (sq.nkb > 0) return sq.nkb;
  const int ntot = sq.n_pre + sq.n_own;
  const int q_last = min(2 * kAQ * pr + 2 * kAQ - 1, sq.nq - 1);
  const int lim_last = sq.vis ? min(ntot, static_cast<int>(__ldg(sq.vis + q_last))) : ntot;
  const int own_need = max(0, lim_last - sq.n_pre);
  return (sq.pad_end + own_need + kAK - 1) / kAK;
}

// The segments this CTA works on, in order; every role walks the same
// sequence.
struct Cursor {
  long long u, u1;  // stream-K: this CTA's run of key blocks
  int item;         // whole items: the next item
};

__device__ __forceinline__ void cursor_init(const AttnTcParams& p, Cursor& c) {
  const long long cta = blockIdx.x;
  c.u = p.units * cta / p.G;
  c.u1 = p.units * (cta + 1) / p.G;
  c.item = blockIdx.x;
}

__device__ __forceinline__ bool cursor_next(const AttnTcParams& p, Cursor& c, Seg& s) {
  if (p.split) {
    if (c.u >= c.u1) return false;
    int z = 0;
    for (int k = 1; k < p.nseq; ++k)
      if (c.u >= p.seq[k].unit0) z = k;
    const AttnTcSeq& sq = p.seq[z];
    const long long lu = c.u - sq.unit0;
    const int iz = static_cast<int>(lu / sq.nkb);
    const int b = static_cast<int>(lu - static_cast<long long>(iz) * sq.nkb);
    const int take = static_cast<int>(min(static_cast<long long>(sq.nkb - b), c.u1 - c.u));
    s.z = z;
    s.h = iz / sq.pairs;
    s.pr = iz - s.h * sq.pairs;
    s.b0 = b;
    s.b1 = b + take;
    if (b == 0 && take == sq.nkb) {
      s.part = -1;
      s.slot = 0;
    } else if (b == 0) {  // ends at this CTA's run end
      s.part = 0;
      s.slot = blockIdx.x;
    } else {  // began in the previous CTA's run
      s.part = 1;
      s.slot = blockIdx.x - 1;
    }
    c.u += take;
    return true;
  }
  if (c.item >= p.items) return false;
  int z = 0;
  for (int k = 1; k < p.nseq; ++k)
    if (c.item >= p.seq[k].item0) z = k;
  const AttnTcSeq& sq = p.seq[z];
  const int iz = c.item - sq.item0;
  s.z = z;
  s.h = iz / sq.pairs;
  s.pr = iz - s.h * sq.pairs;
  s.b0 = 0;
  s.b1 = item_blocks(sq, s.pr);
  s.part = -1;
  s.slot = 0;
  c.item += p.G;
  return true;
}

// ---------------------------------------------------------------- kernel ----

// 10 warps x 200 registers fill the register file (one CTA per SM); a
// __launch_bounds__(320, 1) cap measured lower and spilled
template <bool BF>
__global__ void __maxnreg__(200) attn_tc_kernel(const __grid_constant__ AttnTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int H = p.H;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* qfull = bars + 0;    // [2] a stage's Q tile landed
  uint64_t* qempty = bars + 2;   // [2] its last Q K^T of the item done
  uint64_t* rfull = bars + 4;    // [kSlots] ring slot landed
  uint64_t* rempty = bars + 9;   // [kSlots] ring slot consumed
  uint64_t* sfull = bars + 14;   // [2] S_q in TMEM
  uint64_t* pfull = bars + 16;   // [2] P_q in TMEM (128 softmax threads)
  uint64_t* pvdone = bars + 18;  // [2] O_q += P_q V done
  uint64_t* oempty = bars + 20;  // [2] O_q read by its stage after an item (128 threads)
  uint64_t* mdone = bars + 22;   // MMAs drained (give-up path)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 23);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  volatile int* second = reinterpret_cast<volatile int*>(tslot + 2);  // [2] merge order of a split item

  if (threadIdx.x == 0) {
    for (int i = 0; i < 23; ++i) mbar_init(&bars[i], (i >= 16 && i < 18) || (i >= 20 && i < 22) ? 128 : 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.panel);
    tma_prefetch_desc(&p.panel_kv);
    for (int z = 0; z < p.nseq; ++z)
      if (p.seq[z].n_pre > 0) tma_prefetch_desc(&p.seq[z].kvmap);
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      Cursor cur;
      cursor_init(p, cur);
      Seg s;
      int si = 0;       // items (segments) started
      long long e = 0;  // ring entries issued
      bool ok = true;
      int q_issued[2] = {-1, -1};  // item whose Q tile each stage's buffer was last loaded for
      while (ok && cursor_next(p, cur, s)) {
        const AttnTcSeq& sq = p.seq[s.z];
        for (int q = 0; q < 2; ++q) {
          if (!mbar_wait(&qempty[q], (si & 1) ^ 1u, abort_flag, &s_attn_status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&qfull[q], kQTile);
          const int row = sq.q_row0 + 2 * kAQ * s.pr + kAQ * q;
          uint8_t* dq = smem + kOffQ + q * kQTile;
          tma_load_2d(dq, &p.panel, &qfull[q], s.h * kAD, row);
          tma_load_2d(dq + kQBox, &p.panel, &qfull[q], s.h * kAD + 64, row);
          q_issued[q] = si;
        }
        for (int b = s.b0; b < s.b1 && ok; ++b) {
          for (int kv = 0; kv < 2; ++kv) {
            const int slot = static_cast<int>(e % kSlots);
            if (!mbar_wait(&rempty[slot], static_cast<uint32_t>((e / kSlots) & 1) ^ 1u, abort_flag,
                           &s_attn_status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&rfull[slot], kKVBytes);
            uint8_t* dst = smem + kOffRing + slot * kKVBytes;
            const int col_cache = (kv ? H : 0) + s.h * kAD;
            const int col_panel = (kv ? 2 * H : H) + s.h * kAD;
#pragma unroll
            for (int sb = 0; sb < kAK / kKVBox; ++sb) {
              const int v = b * kAK + sb * kKVBox;
              uint8_t* d = dst + sb * kBoxBytes;
              if (v < sq.n_pre) {
                tma_load_2d(d, &sq.kvmap, &rfull[slot], col_cache, v);
                tma_load_2d(d + kKVHalf, &sq.kvmap, &rfull[slot], col_cache + 64, v);
              } else {
                const int row = sq.own_row0 + (v - sq.pad_end);
                tma_load_2d(d, &p.panel_kv, &rfull[slot], col_panel, row);
                tma_load_2d(d + kKVHalf, &p.panel_kv, &rfull[slot], col_panel + 64, row);
              }
            }
            ++e;
          }
        }
        ++si;
      }
      if (!ok) {
        // let the copies this thread started land before the CTA leaves
        for (long long d = std::max(0ll, e - kSlots); d < e; ++d)
          mbar_wait_drain(&rfull[d % kSlots], static_cast<uint32_t>((d / kSlots) & 1));
        for (int q = 0; q < 2; ++q)
          if (q_issued[q] >= 0) mbar_wait_drain(&qfull[q], static_cast<uint32_t>(q_issued[q] & 1));
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kAQ, kAK, false, BF);
      constexpr uint32_t idesc_pv = idesc_f16(kAQ, kAD, true, BF);  // V: MN-major
      Cursor cur;
      cursor_init(p, cur);
      Seg s;
      int si = 0;
      long long g = 0;  // key blocks consumed before this item
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        if (ok && !mbar_wait(bar, parity, abort_flag, &s_attn_status)) ok = false;
        return ok;
      };
      // S_q = Q_q K^T of block gb (ring entry 2 gb)
      auto issue_qk = [&](int q, long long gb) {
        const long long eK = 2 * gb;
        const uint32_t sQ = smem_u32(smem + kOffQ + q * kQTile);
        const uint32_t sK = smem_u32(smem + kOffRing + static_cast<int>(eK % kSlots) * kKVBytes);
#pragma unroll
        for (int k = 0; k < kAD / 16; ++k)
          tc_mma_f16(tmem + q * kAK, sdesc_sw128(sQ + (k >> 2) * kQBox) + 2 * (k & 3),
                     sdesc_sw128(sK + (k >> 2) * kKVHalf) + 2 * (k & 3), idesc_qk, k > 0 ? 1u : 0u);
        tc_commit(&sfull[q]);
      };
      // O_q (+)= P_q V of block gb (ring entry 2 gb + 1); first: first block of the item
      auto issue_pv = [&](int q, long long gb, bool first) {
        const long long eV = 2 * gb + 1;
        if (!wait(&pfull[q], static_cast<uint32_t>(gb & 1))) return;
        if (q == 0 && !wait(&rfull[eV % kSlots], static_cast<uint32_t>((eV / kSlots) & 1))) return;
        if (first && !wait(&oempty[q], (si & 1) ^ 1u)) return;
        tc_fence_after();
        const uint32_t sV = smem_u32(smem + kOffRing + static_cast<int>(eV % kSlots) * kKVBytes);
#pragma unroll
        for (int k = 0; k < kAK / 16; ++k) {
          // A = P in TMEM: 128 query lanes x 16 keys = 8 columns of 16-bit
          // pairs; B = V: 16 key rows x 128 d, d contiguous (two 64-wide
          // atoms kKVHalf apart, 8-row groups 1 KB)
          const uint64_t bd = sdesc(sV + k * 2048, kKVHalf, 1024, 2);
          tc_mma_f16_ts(tmem + 256 + q * kAD, tmem + q * kAK + k * 8, bd, idesc_pv, (!first || k > 0) ? 1u : 0u);
        }
        tc_commit(&pvdone[q]);
        if (q == 1) tc_commit(&rempty[eV % kSlots]);
      };
      while (ok && cursor_next(p, cur, s)) {
        const int n = s.b1 - s.b0;
        for (int j = 0; j < n && ok; ++j) {
          const long long gb = g + j;
          const long long eK = 2 * gb;
          if (!wait(&rfull[eK % kSlots], static_cast<uint32_t>((eK / kSlots) & 1))) break;
          if (j == 0 && !wait(&qfull[0], static_cast<uint32_t>(si & 1))) break;
          tc_fence_after();
          issue_qk(0, gb);
          if (j == n - 1) tc_commit(&qempty[0]);
          if (j > 0) {
            issue_pv(1, gb - 1, j == 1);
            if (!ok) break;
          }
          if (j == 0 && !wait(&qfull[1], static_cast<uint32_t>(si & 1))) break;
          tc_fence_after();
          issue_qk(1, gb);
          tc_commit(&rempty[eK % kSlots]);
          if (j == n - 1) tc_commit(&qempty[1]);
          issue_pv(0, gb, j == 0);
        }
        if (ok) issue_pv(1, g + n - 1, n == 1);
        g += n;
        ++si;
      }
      // the MMAs this thread issued have completed before the CTA leaves
      tc_commit(mdone);
      mbar_wait_drain(mdone, 0);
    }
  } else {
    // softmax: stage q, TMEM lane quadrant `quad` = query rows 32 quad .. +31
    const int q = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + q * kAK + lane_off;
    const uint32_t tO = tmem + 256 + q * kAD + lane_off;
    const float c = p.scale_log2;
    const uint64_t c2 = f2(c, c);
    Cursor cur;
    cursor_init(p, cur);
    Seg s;
    long long g = 0;
    bool ok = true;
    while (ok && cursor_next(p, cur, s)) {
      const AttnTcSeq& sq = p.seq[s.z];
      const int ntot = sq.n_pre + sq.n_own;
      const int qi = 2 * kAQ * s.pr + kAQ * q + r;
      const bool live = qi < sq.nq;
      int lim = ntot;
      if (sq.vis) {
        const int q_last = min(2 * kAQ * s.pr + 2 * kAQ - 1, sq.nq - 1);
        lim = min(ntot, static_cast<int>(__ldg(sq.vis + (live ? qi : q_last))));
      }
      const int n = s.b1 - s.b0;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        const long long gb = g + j;
        if (!mbar_wait(&sfull[q], static_cast<uint32_t>(gb & 1), abort_flag, &s_attn_status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, sv[cc]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(sv[cc]);
        const int v0 = (s.b0 + j) * kAK;
        // every key of this block visible to this row?
        const int k0 = key_index(v0, sq.n_pre, sq.pad_end);
        const int k1 = key_index(v0 + kAK - 1, sq.n_pre, sq.pad_end);
        const bool same_src = (v0 + kAK <= sq.n_pre) || (v0 >= sq.pad_end);
        if (!(same_src && k1 < lim && k0 < lim)) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int kj = key_index(v0 + cc * 32 + e, sq.n_pre, sq.pad_end);
              if (kj >= lim) sv[cc][e] = __float_as_uint(-INFINITY);
            }
        }
        float mx[4];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          mx[cc] = __uint_as_float(sv[cc][0]);
#pragma unroll
          for (int e = 1; e < 31; e += 2)
            mx[cc] = max3(mx[cc], __uint_as_float(sv[cc][e]), __uint_as_float(sv[cc][e + 1]));
          mx[cc] = fmaxf(mx[cc], __uint_as_float(sv[cc][31]));
        }
        const float mb = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c;
        // raise the running max only past the threshold (exact: O and l
        // share the stale max; P <= 2^threshold stays in range)
        float alpha = 1.f;
        const bool need = mb > m + kRescaleThreshold;
        if (need) {
          alpha = ex2(m - mb);
          m = mb;
          l *= alpha;
        }
        if (__any_sync(0xffffffffu, need && j > 0)) {
          // O_q is stable: S_q of this block completed after the P V of the
          // previous block (one issuing thread, in order)
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(tO + cc * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + cc * 32, o);
          }
        }
        // P = 2^(s c - m) as 16-bit pairs over the first 64 columns of S_q
        const uint64_t nm2 = f2(-m, -m);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int k = 64 * half + 2 * i;
            const uint64_t x =
                ffma2(f2(__uint_as_float(sv[k >> 5][k & 31]), __uint_as_float(sv[k >> 5][(k & 31) + 1])), c2, nm2);
            float x0, x1;
            unf2(x, x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            acc[i & 3] = fadd2(acc[i & 3], f2(p0, p1));
            pk[i] = pack2<BF>(p0, p1);
          }
          tmem_st32(tS + half * 32, pk);
        }
        {
          const uint64_t t = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
          float t0, t1;
          unf2(t, t0, t1);
          l += t0 + t1;
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&pfull[q]);
      }
      if (!ok) break;
      // the item's O_q: read it, release the accumulator, write the result
      const long long gl = g + n - 1;
      if (!mbar_wait(&pvdone[q], static_cast<uint32_t>(gl & 1), abort_flag, &s_attn_status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t o[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tO + cc * 32, o[cc]);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld_wait(o[cc]);
      tc_fence_before();
      mbar_arrive(&oempty[q]);
      uint16_t* orow = static_cast<uint16_t*>(p.out) + static_cast<size_t>(sq.q_row0 + qi) * H + s.h * kAD;
      if (s.part < 0) {
        const float inv = 1.f / l;
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int gq = 0; gq < 4; ++gq)
              dst[cc * 4 + gq] = make_uint4(
                  pack2<BF>(__uint_as_float(o[cc][8 * gq + 0]) * inv, __uint_as_float(o[cc][8 * gq + 1]) * inv),
                  pack2<BF>(__uint_as_float(o[cc][8 * gq + 2]) * inv, __uint_as_float(o[cc][8 * gq + 3]) * inv),
                  pack2<BF>(__uint_as_float(o[cc][8 * gq + 4]) * inv, __uint_as_float(o[cc][8 * gq + 5]) * inv),
                  pack2<BF>(__uint_as_float(o[cc][8 * gq + 6]) * inv, __uint_as_float(o[cc][8 * gq + 7]) * inv));
        }
      } else {
        // one part of a split item: store the partial (O transposed so
        // that the warp's rows are contiguous, the max and the sum); the
        // part that finishes second merges both and writes the result
        float* mine = p.part + (static_cast<size_t>(s.slot * 2 + s.part) * 2 + q) * kPartFloats;
        const float* other = p.part + (static_cast<size_t>(s.slot * 2 + (s.part ^ 1)) * 2 + q) * kPartFloats;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int e = 0; e < 32; ++e) __stcg(mine + (cc * 32 + e) * kAQ + r, __uint_as_float(o[cc][e]));
        __stcg(mine + kAQ * kAD + r, m);
        __stcg(mine + kAQ * kAD + kAQ + r, l);
        __threadfence();
        stage_sync(q);
        int* flag = p.flags + s.slot * 2 + q;
        if (r == 0) second[q] = atomicAdd(flag, 1);
        stage_sync(q);
        if (second[q] == 1) {
          __threadfence();
          const float m2 = __ldcg(other + kAQ * kAD + r);
          const float l2 = __ldcg(other + kAQ * kAD + kAQ + r);
          const float mm = fmaxf(m, m2);
          const float a1 = ex2(m - mm), a2 = ex2(m2 - mm);
          const float inv = 1.f / (l * a1 + l2 * a2);
          const float w1 = a1 * inv, w2 = a2 * inv;
          if (live) {
            uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
              for (int gq = 0; gq < 4; ++gq) {
                uint32_t w[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  const int e = 8 * gq + 2 * t;
                  const float oa = __uint_as_float(o[cc][e]) * w1 + __ldcg(other + (cc * 32 + e) * kAQ + r) * w2;
                  const float ob =
                      __uint_as_float(o[cc][e + 1]) * w1 + __ldcg(other + (cc * 32 + e + 1) * kAQ + r) * w2;
                  w[t] = pack2<BF>(oa, ob);
                }
                dst[cc * 4 + gq] = make_uint4(w[0], w[1], w[2], w[3]);
              }
          }
          if (r == 0) *flag = 0;  // both parts have arrived: ready for the next launch
        }
        // the merge-order word is reused by this stage's next split item
        stage_sync(q);
      }
      g += n;
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

size_t attn_split_bytes(int ctas) {
  return ctas > 1 ? static_cast<size_t>(ctas - 1) * 4 * kPartFloats * sizeof(float) : 0;
}

cudaError_t make_attn_plan(const AttnArgs& in, AttnPlan* p) {
  if (in.dt != DT_F16 && in.dt != DT_BF16) return cudaErrorInvalidValue;
  if (in.nseq < 1 || in.nseq > kMaxSeq) return cudaErrorInvalidValue;
  memset(p, 0, sizeof *p);
  AttnTcParams& prm = p->prm;
  const int H = in.heads * kAD;
  p->dt = in.dt;
  prm.out = in.out;
  prm.H = H;
  prm.nseq = in.nseq;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(kAD)));
  cudaError_t e = encode_rows(&prm.panel, in.panel, static_cast<uint64_t>(3) * H, in.panel_rows, kAQ, in.dt);
  if (e == cudaSuccess)
    e = encode_rows(&prm.panel_kv, in.panel, static_cast<uint64_t>(3) * H, in.panel_rows, kKVBox, in.dt);
  if (e != cudaSuccess) return e;
  bool step_mode = true;
  int items = 0, max_nkb = 0;
  long long units = 0;
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
    t.pairs = (a.nq + 2 * kAQ - 1) / (2 * kAQ);
    t.nkb = a.vis ? 0 : (t.pad_end + a.n_own + kAK - 1) / kAK;
    t.item0 = items;
    t.unit0 = units;
    if (a.vis) step_mode = false;
    items += t.pairs * in.heads;
    units += static_cast<long long>(t.pairs) * in.heads * t.nkb;
    max_nkb = std::max(max_nkb, t.nkb);
    if (a.n_pre > 0) {
      e = encode_rows(&t.kvmap, a.kv_pre, static_cast<uint64_t>(2) * H, a.n_pre, kKVBox, in.dt);
      if (e != cudaSuccess) return e;
    }
  }
  prm.items = items;
  if (items == 0) return cudaSuccess;  // gx == 0: nothing to launch
  int G = sm_count();
  if (in.max_ctas > 0) G = std::min(G, in.max_ctas);
  // stream-K when every item is a run of whole key blocks (a step), there
  // are more items than CTAs, each CTA's run is at least one item long (so
  // an item has at most two parts) and the scratch holds the partials
  const bool split = step_mode && items > G && units / G >= max_nkb && in.part != nullptr && in.flags != nullptr &&
                     attn_split_bytes(G) <= in.part_bytes && G <= kMaxAttnCtas;
  if (split) {
    prm.split = 1;
    prm.units = units;
    prm.part = static_cast<float*>(in.part);
    prm.flags = in.flags;
  } else {
    G = std::min(G, items);
  }
  prm.G = G;
  p->gx = G;
  p->gy = 1;
  p->gz = 1;
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
