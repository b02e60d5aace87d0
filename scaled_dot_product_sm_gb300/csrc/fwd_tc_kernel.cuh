// fwd_tc_kernel.cuh - bf16 prefill forward on the 5th-generation tensor cores.
//
// O = softmax(alpha Q K^T + mask + causal) V with a per-row log-sum-exp
// (course chapter "Scaled dot-product attention (forward and backward)",
// sections 2.1-2.2; stats as on the cuDNN "Attention" page), computed one
// 128-key tile at a time with a running max and sum (online softmax).
//
// A work unit = one (batch, query head) and two 128-row query tiles (256 rows)
// that share every K/V tile load.  The grid is persistent (one CTA per SM, each
// walking a list of units, or taking them from a counter when padding lengths
// make them uneven), so the next unit's Q load and first scores overlap the
// current unit's last tiles and epilogue.  Warp roles (384 threads, three
// warpgroups):
//   warps 0-3  softmax of query tile 0 (thread = row = TMEM lane)
//   warps 4-7  softmax of query tile 1
//   warp  8    TMA producer: Q tiles once, then K_0, V_0, K_1, V_1, ... through a ring
//   warp  9    TMEM allocator and tcgen05.mma issuer (see below)
//   warp  10   stages the additive mask by TMA (rows of a multiple of 4 keys), else idle
//   warp  11   idle (it completes the third warpgroup)
// The third warpgroup hands registers to the softmax warpgroups (72 -> 216 per
// thread: 4*32*72 + 8*32*216 = 64512 = 384*168, the launch's register file share).
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+Ev), O_1 [384,384+Ev).
// The softmax writes P_t as bf16 pairs over the first 64 columns of S_t, and
// O_t += P_t V reads it straight from TMEM (A operand in TMEM), so P never
// touches shared memory and the tensor core reads only K, V and Q from it.
// MMA issue order per key tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): the
// tensor core works on one query tile while the other tile's softmax runs, and
// S_t(j+1) (which overwrites P_t(j)'s columns) follows PV_t(j) in the same
// in-order MMA stream.  The commit after S_t(j+1) also covers PV_t(j), so when
// tile t sees its next scores, O_t is complete.  Exponentials are exp2 with alpha*log2(e)
// folded into the scale (with a mask, log2(e) into the exponent's FMA); O is only rescaled when a row's max grows by more
// than 2^8 (the stale max keeps every p below 256, and O/l is exact either way).
// Causal: key tiles entirely above the diagonal are neither loaded nor
// computed; only tiles that cross it test j <= i per element.
// The issuer paces the whole kernel: each tile's chain is its softmax, then
// PV_t(j) and S_t(j+1) behind the other tile's MMAs, so every cycle the issuing
// thread spends between MMA groups (barrier waits, commits, descriptor
// arithmetic) lengthens it.  The whole of warp 9 runs the issue loop, converged,
// and the lane elect.sync picked once issues each MMA and commit: the operand
// arithmetic is then warp-uniform, and the causal E = 128 forward runs 8 % faster
// than with lane 0 alone in a divergent branch (the masked one 2.7 %).
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa_impl {

namespace {

using namespace sdpa_ptx;

constexpr int BM = 128;        // query rows per tile (MMA M)
constexpr int BN = 128;        // keys per tile (MMA N of S, K of PV)
constexpr int kThreads = 384;
constexpr int kRegsLaunch = 168;   // registers per thread the kernel is compiled and launched with
constexpr int kRegsSoftmax = 216;  // after setmaxnreg.inc (warpgroups 0 and 1)
constexpr int kRegsOther = 72;     // after setmaxnreg.dec (warpgroup 2)
static_assert(8 * 32 * kRegsSoftmax + 4 * 32 * kRegsOther <= kThreads * kRegsLaunch, "register split too large");
static_assert(2 * kRegsSoftmax + kRegsOther <= 512, "per sub-partition register file exceeded");
constexpr int kChunkBytes = 128 * 128;   // one [128 rows x 64 bf16] swizzled block
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Additive mask: none, read by the softmax threads from global memory, or staged
// in shared memory by TMA (rows of a multiple of 4 keys).
constexpr int kMaskNone = 0, kMaskDirect = 1, kMaskStaged = 2;

template <int ECH, int VCH, int MK>
struct FwdCfg {
  static constexpr int E = ECH * 64, Ev = VCH * 64;
  static constexpr int kQBytes = ECH * kChunkBytes;                          // one query tile
  static constexpr int kItem = (ECH > VCH ? ECH : VCH) * kChunkBytes;       // one K or V tile
  // staged mask: one query tile's [128 rows x 128 keys] fp32 as four 32-key boxes, 128-byte swizzled
  static constexpr int kMaskBytes = MK == kMaskStaged ? BM * BN * 4 : 0;
  static constexpr int kFixed = 2 * kQBytes + kMaskBytes;
  static constexpr int kBudget = 227 * 1024 - 2048;
  static constexpr int NS = (kBudget - kFixed) / kItem > 8 ? 8 : (kBudget - kFixed) / kItem;
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kOffQ + 2 * kQBytes;
  static constexpr int kOffMask = kOffRing + NS * kItem;
  static constexpr int kOffBar = kOffMask + kMaskBytes;
  static constexpr int kBytes = kOffBar + 512 + 1024;   // barriers, unit slots + alignment slack
  static_assert(NS >= 2, "the K/V ring needs two stages");
};

template <int ECH, int VCH, int MK, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmM, FwdParams p) {
  constexpr bool MASKED = MK != kMaskNone;
  using C = FwdCfg<ECH, VCH, MK>;
  constexpr int NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* bar_q = bar;                 // 1: the unit's Q tiles landed
  uint64_t* q_free = bar + 1;            // 1: every S MMA of the previous unit complete (Q buffers free)
  uint64_t* full = bar + 2;              // NS
  uint64_t* empty = full + NS;           // NS
  uint64_t* s_full = empty + NS;         // 2: S_t(j) (and PV_t(j-1)) complete
  uint64_t* p_full = s_full + 2;         // 2: P_t(j) in TMEM (one arrival per warp)
  uint64_t* o_final = p_full + 2;        // 2: the last PV_t of the unit complete
  uint64_t* mk_full = o_final + 2;       // 4: staged mask half h of query tile t landed (2t + h)
  uint64_t* mk_empty = mk_full + 4;      // 4: ... and read by tile t's softmax warps
  uint64_t* un_full = mk_empty + 4;      // 4: unit index published (taken from the counter)
  uint64_t* un_empty = un_full + 4;      // 4: ... and read by every role
  uint64_t* mma_drain = un_empty + 4;    // 1: every MMA of the issuing thread complete (before TMEM is released)
  int* un_slot = reinterpret_cast<int*>(mma_drain + 1);                 // 4 unit indices
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(un_slot + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work units: (batch x query head, pair of 128-row query tiles).  Causal: listed
  // heaviest first (the last row pairs see the most key tiles).  The CTAs are
  // persistent; CTA c takes units c, 2G-1-c, 2G+c, ... of the list (G CTAs),
  // a snake order that evens out the causal work.
  const int BHq = p.B * p.Hq;
  const int units = (p.L + 2 * BM - 1) / (2 * BM);
  const int total = BHq * units;
  auto unit_index = [&](int r) {   // r-th unit of this CTA, or -1
    const int G = gridDim.x, c = blockIdx.x;
    const int k = r * G + ((r & 1) ? G - 1 - c : c);
    return k < total ? k : -1;
  };
  // With a counter (p.sched), the CTAs take units in turn instead: the producer
  // thread takes each index and publishes it through a 4-slot ring, and the MMA
  // thread, the softmax warps and the mask producer read the same sequence.  A
  // wait that gives up (abort) reads whatever the slot holds: a stale unit index
  // or the initial -1, never an out-of-range one.
  const bool dyn = p.sched != nullptr;
  auto take_unit = [&](int r) {   // producer thread
    if (!dyn) return unit_index(r);
    const int sl = r & 3;
    mbar_wait(&un_empty[sl], ((r >> 2) & 1) ^ 1, abort_flag, p.status, status_code(0x1d));
    const unsigned tk = atomicAdd(p.sched, 1u);
    const int k = tk < static_cast<unsigned>(total) ? static_cast<int>(tk) : -1;
    un_slot[sl] = k;
    mbar_arrive(&un_full[sl]);   // release: the slot's value is visible to the waiters
    return k;
  };
  auto read_unit = [&](int r) {   // other roles; the caller then reports the read on un_empty
    if (!dyn) return unit_index(r);
    const int sl = r & 3;
    mbar_wait(&un_full[sl], (r >> 2) & 1, abort_flag, p.status, status_code(0x1e));
    return *reinterpret_cast<volatile int*>(&un_slot[sl]);
  };
  // Key tiles of a unit: tile t (rows rt..rt+127) needs key tiles [a_t, b_t),
  // from lo(rt) to hi(last row before Lb) (padding and band; empty when no row
  // sees a key); the unit loads their union [j0, j1), which is contiguous.
  struct Unit {
    int bh, b, h, bkv, r0, a[2], e[2], j0, j1;
  };
  const bool right_bounded = p.band.right >= 0;
  auto unit_at = [&](int k) {
    Unit u;
    // right-bounded (causal-like): row pairs outer (the last, heaviest pairs of every
    // head first); otherwise heads outer, so the pairs of one head run side by side
    // and share its K/V in L2
    const int pair = right_bounded ? k / BHq : k % units;
    u.bh = right_bounded ? k - pair * BHq : k / units;
    u.b = u.bh / p.Hq;
    u.h = u.bh - u.b * p.Hq;
    u.bkv = u.b * p.Hkv + u.h / p.G;
    u.r0 = (units - 1 - pair) * 2 * BM;
    const BandRows br = band_rows(p.band, u.b, p.L, p.S);
    u.j0 = 0x7fffffff;
    u.j1 = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int rt = u.r0 + t * BM, last = min(rt + BM, br.Lb) - 1;
      const int lo = br.lo(rt), hi = last >= rt ? br.hi(last) : -1;
      u.a[t] = hi >= lo ? lo / BN : 0;
      u.e[t] = hi >= lo ? hi / BN + 1 : 0;
      if (u.e[t] > u.a[t]) {
        u.j0 = min(u.j0, u.a[t]);
        u.j1 = max(u.j1, u.e[t]);
      }
    }
    if (u.j1 == 0) u.j0 = 0;
    return u;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(q_free, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);
      mbar_init(&o_final[t], 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(&mk_full[2 * t + h], 1);
        mbar_init(&mk_empty[2 * t + h], 4);
      }
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&un_full[i], 1);
      mbar_init(&un_empty[i], 9 + (MK == kMaskStaged ? 1 : 0));   // MMA thread, 8 softmax warps, mask producer
      un_slot[i] = -1;
    }
    mbar_init(mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp >= 8) {
    regs_dec<kRegsOther>();
    if (warp == 8 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      int it = 0;       // ring position, continued across units
      int nunits = 0;   // units whose Q tiles were requested (one bar_q phase each)
      for (int r = 0;; ++r) {
        const int k = take_unit(r);
        if (k < 0) break;
        const Unit u = unit_at(k);
        ++nunits;
        // the previous unit's S MMAs have read its Q tiles
        mbar_wait(q_free, (r & 1) ^ 1, abort_flag, p.status, status_code(0x10));
        const int nq = (u.e[0] > u.a[0]) + (u.e[1] > u.a[1]);
        mbar_arrive_expect_tx(bar_q, nq * C::kQBytes);   // no tiles: a plain arrival
        for (int t = 0; t < 2; ++t) {
          if (u.e[t] == u.a[t]) continue;
          for (int c = 0; c < ECH; ++c)
            tma_load_3d(smem + C::kOffQ + t * C::kQBytes + c * kChunkBytes, &tmQ, bar_q, c * 64, u.r0 + t * BM,
                        u.bh);
        }
        // ring order = consumption order: K_j0, then per j: V_j, K_{j+1} (if any)
        auto load = [&](bool is_k, int j) {
          const int s = it % NS;
          mbar_wait(&empty[s], ((it / NS) & 1) ^ 1, abort_flag, p.status, status_code(0x11));
          uint8_t* dst = smem + C::kOffRing + s * C::kItem;
          const int ch = is_k ? ECH : VCH;
          mbar_arrive_expect_tx(&full[s], ch * kChunkBytes);
          for (int c = 0; c < ch; ++c)
            tma_load_3d(dst + c * kChunkBytes, is_k ? &tmK : &tmV, &full[s], c * 64, j * BN, u.bkv);
          ++it;
        };
        if (u.j1 > u.j0) load(true, u.j0);
        for (int j = u.j0; j < u.j1; ++j) {
          load(false, j);
          if (j + 1 < u.j1) load(true, j + 1);
        }
      }
      if (*abort_flag) {   // a wait gave up: let this thread's copies land before the CTA exits
        if (nunits > 0) mbar_drain(bar_q, static_cast<uint32_t>((nunits - 1) & 1));
        mbar_drain_ring(full, NS, it);
      }
    } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
      // The one lane that issues: elected once (lane 0 of the converged warp), so every
      // MMA and commit comes from the same thread, as a commit only covers its own thread's
      // MMAs.  Electing once measured faster than an elect.sync per MMA (C3 forward 0.188
      // -> 0.185 ms), and much faster than testing lane == 0 (0.232 ms).
      const bool lead = elect_one();
      auto leader = [&]() { return lead; };
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);        // Q (K-major) x K (K-major)
      constexpr uint32_t idesc_o = idesc_bf16(BM, C::Ev, 0, 1);     // P (TMEM, K-major) x V (MN-major)
      // Operand descriptors, built once; a K-step, a tile or a ring slot moves only the start address.
      const SmemDesc dq = smem_desc(smem_u32(smem + C::kOffQ), 16, 1024);            // Q, K-major
      const SmemDesc dk = smem_desc(smem_u32(smem + C::kOffRing), 16, 1024);         // K slot 0, K-major
      const SmemDesc dv = smem_desc(smem_u32(smem + C::kOffRing), kChunkBytes, 1024);  // V slot 0, MN-major
      auto issue_s = [&](int t, int slot) {
        const SmemDesc qa = dq + t * C::kQBytes, ka = dk + slot * C::kItem;
#pragma unroll
        for (int kk = 0; kk < C::E / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          if (leader()) umma_ss(tmem + t * BN, qa + off, ka + off, idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const SmemDesc va = dv + slot * C::kItem;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)   // 16 keys = 8 TMEM columns of bf16 pairs per step
          if (leader()) umma_ts(tmem + 256 + t * 128, tmem + t * BN + kk * 8, va + kk * 16 * 128, idesc_o,
                  (acc || kk > 0) ? 1u : 0u);
      };
      int it = 0;               // ring position, continued across units
      uint32_t pc[2] = {0, 0};  // p_full completions consumed per tile
      for (int r = 0;; ++r) {
        const int k = read_unit(r);
        if (dyn && lane == 0) mbar_arrive(&un_empty[r & 3]);
        if (k < 0) break;
        const Unit u = unit_at(k);
        mbar_wait(bar_q, r & 1, abort_flag, p.status, status_code(0x12));
        if (u.j1 == u.j0) {
          if (leader()) umma_commit(q_free);   // nothing to compute; covers the earlier units' MMAs
          continue;
        }
        {
          const int s = it % NS;
          mbar_wait(&full[s], (it / NS) & 1, abort_flag, p.status, status_code(0x13));
          tc_fence_after();
          for (int t = 0; t < 2; ++t) {
            if (u.a[t] != u.j0 || u.e[t] == u.a[t]) continue;
            issue_s(t, s);
            if (leader()) umma_commit(&s_full[t]);
          }
          if (leader()) umma_commit(&empty[s]);
          if (u.j1 - u.j0 == 1 && leader()) umma_commit(q_free);
          ++it;
        }
        for (int j = u.j0; j < u.j1; ++j) {
          const int sv = it % NS;
          mbar_wait(&full[sv], (it / NS) & 1, abort_flag, p.status, status_code(0x14));
          tc_fence_after();
          ++it;
          int sk = -1;
          for (int t = 0; t < 2; ++t) {
            const bool pv = u.a[t] <= j && j < u.e[t];
            if (pv) {
              mbar_wait(&p_full[t], pc[t] & 1, abort_flag, p.status, status_code(0x15));
              ++pc[t];
              tc_fence_after();
              issue_pv(t, sv, j > u.a[t]);
            }
            if (u.a[t] <= j + 1 && j + 1 < u.e[t]) {
              if (sk < 0) {
                sk = it % NS;
                mbar_wait(&full[sk], (it / NS) & 1, abort_flag, p.status, status_code(0x16));
                tc_fence_after();
                ++it;
              }
              issue_s(t, sk);   // overwrites P_t(j) after PV_t(j) in issue order
              if (leader()) umma_commit(&s_full[t]);
            } else if (pv) {
              if (leader()) umma_commit(&o_final[t]);
            }
          }
          if (j + 1 < u.j1 && sk < 0) {   // K_{j+1} is in the ring for the other tile only: release it
            sk = it % NS;
            mbar_wait(&full[sk], (it / NS) & 1, abort_flag, p.status, status_code(0x16));
            ++it;
          }
          if (leader()) umma_commit(&empty[sv]);
          if (sk >= 0 && leader()) umma_commit(&empty[sk]);
          if (j + 2 == u.j1 && leader()) umma_commit(q_free);   // the unit's last S MMAs were just issued
        }
      }
      // every MMA this thread issued is complete before the CTA releases TMEM (after a wait
      // that gave up, some may still be queued; the drain is bounded like every wait)
      if (leader()) umma_commit(mma_drain);
      mbar_drain(mma_drain, 0);
    } else if (MK == kMaskStaged && warp == 10 && lane == 0) {
    // ------------------------------------------------------------ mask producer
      // One buffer in two halves (keys 0-63 and 64-127 of a key tile), filled in the
      // softmax warps' order of use: key tile j of query tile 0, then of tile 1, then
      // j + 1 ...  Each (tile, half) has its own full/empty pair, so a wait never has
      // to tell apart two phases of the same parity; a half is refilled as soon as
      // the previous fill of that half (of either tile) has been read, so the next
      // tile's first half is in flight while the softmax still waits for the second.
      prefetch_tmap(&tmM);
      const long long LS = static_cast<long long>(p.L) * p.S;
      int cnt[2] = {0, 0}, last[2] = {-1, -1};   // fills per tile; tile that last filled half h
      for (int ur = 0;; ++ur) {
        const int k = read_unit(ur);
        if (dyn) mbar_arrive(&un_empty[ur & 3]);
        if (k < 0) break;
        const Unit u = unit_at(k);
        const int slice = static_cast<int>((u.b * p.mask_sb + u.h * p.mask_sh) / LS);
        for (int j = u.j0; j < u.j1; ++j) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int row_first = u.r0 + t * BM;
            if (row_first >= p.L || j < u.a[t] || j >= u.e[t]) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (last[h] >= 0)
                mbar_wait(&mk_empty[2 * last[h] + h], (cnt[last[h]] - 1) & 1, abort_flag, p.status, status_code(0x1b));
              mbar_arrive_expect_tx(&mk_full[2 * t + h], C::kMaskBytes / 2);
#pragma unroll
              for (int q = 2 * h; q < 2 * h + 2; ++q)   // 32-key boxes of this half
                tma_load_3d(smem + C::kOffMask + q * (BM * 128), &tmM, &mk_full[2 * t + h], j * BN + 32 * q, row_first,
                            slice);
              last[h] = t;
            }
            if (j + 1 < u.e[t])   // the tile's next key tile into L2 now, so its fill is an L2 hit
#pragma unroll
              for (int q = 0; q < BN / 32; ++q) tma_prefetch_l2_3d(&tmM, (j + 1) * BN + 32 * q, row_first, slice);
            ++cnt[t];
          }
        }
      }
      if (*abort_flag)   // a wait gave up: let this thread's copies land before the CTA exits
        for (int t = 0; t < 2; ++t)
          if (cnt[t] > 0)
            for (int h = 0; h < 2; ++h) mbar_drain(&mk_full[2 * t + h], static_cast<uint32_t>((cnt[t] - 1) & 1));
    }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;               // query tile
    const int wq = warp & 3;               // TMEM lane quarter
    const int r = wq * 32 + lane;          // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tO = tmem + lane_off + 256 + t * 128;
    // alpha*log2(e), kept > 0 (alpha = 0 becomes the smallest normal float, which
    // gives the same exponentials): then the row max of the raw scores, scaled,
    // is the max of the scaled scores, and x = s*sc - m is one FMA (unmasked path)
    const float sc = fmaxf(p.scale_log2, 1.17549435e-38f);
    uint32_t sc_cnt = 0, oc_cnt = 0;       // s_full / o_final completions consumed
    uint32_t mk_cnt = 0;                   // staged mask tiles of this query tile consumed
    for (int ur = 0;; ++ur) {
      const int k = read_unit(ur);
      if (dyn) {   // every lane has read the slot before it is reported free
        __syncwarp();
        if (lane == 0) mbar_arrive(&un_empty[ur & 3]);
      }
      if (k < 0) break;
      const Unit u = unit_at(k);
      const int row_first = u.r0 + t * BM;   // first row of this tile
      const int row = row_first + r;
      if (row_first >= p.L) continue;
      const int ja = t ? u.a[1] : u.a[0], je = t ? u.e[1] : u.e[0];
      if (je == ja) {   // no row of this tile sees a key: o = 0, lse = -inf
        if (row < p.L) {
          __nv_bfloat16* orow =
              static_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(u.bh) * p.L + row) * C::Ev;
#pragma unroll
          for (int c = 0; c < C::Ev / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[static_cast<size_t>(u.bh) * p.L + row] = kNegInf;
        }
        continue;
      }
      const BandRows br = band_rows(p.band, u.b, p.L, p.S);
      // the tile's rows all see every key of a key tile inside [lo(last row), hi(first row)]
      const int row_last = row_first + BM - 1;
      const bool rows_full = row_last < br.Lb;
      const int full_lo = rows_full ? br.lo(row_last) : 0x7fffffff, full_hi = br.hi(row_first);
      // 256-bit mask loads need 32-byte aligned rows: base aligned and S a multiple of 8
      const bool mask_v8 = (reinterpret_cast<uintptr_t>(p.mask) & 31) == 0 && (p.S & 7) == 0;
      const float* mrow = (p.mask && row < p.L)
                              ? p.mask + u.b * p.mask_sb + u.h * p.mask_sh + static_cast<size_t>(row) * p.S
                              : nullptr;
      float m_run = kNegInf, l_run = 0.f;
      for (int j = ja; j < je; ++j) {
        const int kb = j * BN;
        float x[BN];
        if (MASKED) {   // the TMEM loads below are executed by the whole warp in either branch
          // the mask values of this row's keys, read before the scores land so the
          // loads' latency overlaps the wait; whole 32-byte sectors when the rows
          // are 32-byte aligned (S a multiple of 8), else 16-byte or scalar loads.
          // Rows past L (mrow == nullptr) read nothing.  Staged: the row from shared
          // memory (zero-filled past L and S), then the buffer goes back to the producer.
          if (MK == kMaskStaged) {
            const uint8_t* ms = smem + C::kOffMask + r * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {   // keys 64h .. 64h + 63: two 32-key boxes
              mbar_wait(&mk_full[2 * t + h], mk_cnt & 1, abort_flag, p.status, status_code(0x1c));
#pragma unroll
              for (int q = 2 * h; q < 2 * h + 2; ++q)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const float4 mv = *reinterpret_cast<const float4*>(ms + q * (BM * 128) + ((c ^ (r & 7)) << 4));
                  x[32 * q + 4 * c + 0] = mv.x;
                  x[32 * q + 4 * c + 1] = mv.y;
                  x[32 * q + 4 * c + 2] = mv.z;
                  x[32 * q + 4 * c + 3] = mv.w;
                }
              // the next fill is a TMA (async-proxy) write: order this lane's reads before it
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(&mk_empty[2 * t + h]);
            }
            ++mk_cnt;
          } else if (mask_v8) {
            const float* mtile = mrow + kb;
#pragma unroll
            for (int c = 0; c < BN / 8; ++c) {
              const int key = kb + 8 * c;
              float m8[8];
              if (mrow && key < p.S) {
                asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                             : "=f"(m8[0]), "=f"(m8[1]), "=f"(m8[2]), "=f"(m8[3]), "=f"(m8[4]), "=f"(m8[5]),
                               "=f"(m8[6]), "=f"(m8[7])
                             : "l"(mtile + 8 * c));
              } else {
#pragma unroll
                for (int u8 = 0; u8 < 8; ++u8) m8[u8] = 0.f;
              }
#pragma unroll
              for (int u8 = 0; u8 < 8; ++u8) x[8 * c + u8] = m8[u8];
            }
          } else if ((p.S & 3) == 0) {
#pragma unroll
            for (int c = 0; c < BN / 4; ++c) {
              const int key = kb + 4 * c;
              const float4 mv = mrow && key < p.S ? __ldg(reinterpret_cast<const float4*>(mrow + key))
                                                  : make_float4(0.f, 0.f, 0.f, 0.f);
              x[4 * c + 0] = mv.x;
              x[4 * c + 1] = mv.y;
              x[4 * c + 2] = mv.z;
              x[4 * c + 3] = mv.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < BN; ++i) x[i] = mrow && kb + i < p.S ? __ldg(mrow + kb + i) : 0.f;
          }
          mbar_wait(&s_full[t], sc_cnt & 1, abort_flag, p.status, status_code(0x18));
          ++sc_cnt;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tS + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; i += 2)   // t = s * alpha + mask (natural-log units)
              fma2(x[c * 32 + i], x[c * 32 + i + 1], __uint_as_float(v[i]), __uint_as_float(v[i + 1]), p.scale,
                   p.scale, x[c * 32 + i], x[c * 32 + i + 1]);
          }
        } else {
          mbar_wait(&s_full[t], sc_cnt & 1, abort_flag, p.status, status_code(0x18));
          ++sc_cnt;
          tc_fence_after();
          uint32_t v[BN];
          tmem_ld128(tS, v);
#pragma unroll
          for (int i = 0; i < BN; i += 2)
            x[i] = __uint_as_float(v[i]), x[i + 1] = __uint_as_float(v[i + 1]);   // raw scores
        }
        if (!(kb >= full_lo && kb + BN - 1 <= full_hi)) {   // warp-uniform: the tile crosses a boundary
          // this row sees key kb + i exactly for i in [ilo, ihi]
          const int ilo = br.lo(row) - kb, ihi = row < br.Lb ? br.hi(row) - kb : -1;
#pragma unroll
          for (int i = 0; i < BN; ++i)
            if (i < ilo || i > ihi) x[i] = kNegInf;
        }
        // row max: eight independent chains of three-input maxima
        float mx8[8];
#pragma unroll
        for (int u8 = 0; u8 < 8; ++u8) mx8[u8] = fmaxf(x[u8], x[8 + u8]);
#pragma unroll
        for (int i = 16; i < BN; i += 16)
#pragma unroll
          for (int u8 = 0; u8 < 8; ++u8) mx8[u8] = max3f(mx8[u8], x[i + u8], x[i + 8 + u8]);
        const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7]));
        // to log2 units: raw scores times alpha*log2(e), or the masked t times log2(e)
        const float xs = MASKED ? kLog2e : sc;
        const float m_new = fmaxf(m_run, mx * xs);
        const bool need = m_new > m_run + kRescaleThreshold;
        const float m_use = need ? m_new : m_run;
        const float nm = (m_use == kNegInf) ? 0.f : -m_use;
        const float corr = need ? ex2(m_run + nm) : 1.f;
        // p = exp2(x - m), packed to bf16 pairs; row sum in eight independent chains.  In
        // three passes (all exponents, all exponentials, then sums and packing), which
        // measured 1 % faster than one pass per pair (C3 forward 0.1867 -> 0.1846 ms).
        uint32_t pk[BN / 2];
        float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < BN; i += 2) fma2(x[i], x[i + 1], x[i], x[i + 1], xs, xs, nm, nm);   // x * xs - m
#pragma unroll
        for (int i = 0; i < BN; ++i) x[i] = ex2(x[i]);
#pragma unroll
        for (int i = 0; i < BN; i += 2) {
          const int q4 = (i >> 1) & 3;
          add2(rs8[2 * q4], rs8[2 * q4 + 1], rs8[2 * q4], rs8[2 * q4 + 1], x[i], x[i + 1]);
          pk[i >> 1] = pack_bf16x2(x[i], x[i + 1]);
        }
        const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        l_run = l_run * corr + rs;
        if (DROP) {
          // dropout: the row sum above keeps every weight; P V gets P o keep (1/(1-p) at the end)
#pragma unroll
          for (int g = 0; g < BN / 8; ++g) {
            uint32_t keep[4];
            dropout_keep8(p.drop, static_cast<unsigned>((kb >> 3) + g), static_cast<unsigned>(row),
                          static_cast<unsigned>(u.bh), keep);
#pragma unroll
            for (int c = 0; c < 4; ++c) pk[g * 4 + c] &= keep[c];
          }
        }
        if (j > ja) {
          // O_t holds PV_t(ja..j-1) (complete: the commit after S_t(j) covered it)
          if (__any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int c = 0; c < C::Ev / 32; ++c) {
              uint32_t v[32];
              tmem_ld32(tO + c * 32, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * corr);
              tmem_st32(tO + c * 32, v);
            }
          }
        }
        m_run = m_use;
        {
          // P_t(j) over the first 64 columns of S_t: column c holds keys 2c (low) and 2c+1 (high)
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) w[c] = pk[c];
          tmem_st32(tS, w);
#pragma unroll
          for (int c = 0; c < 32; ++c) w[c] = pk[32 + c];
          tmem_st32(tS + 32, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[t]);
      }
      // ---------------------------------------------------------- epilogue
      // O_t is read out before this warp writes the next unit's P_t, so the
      // next unit's first PV_t (which waits for that P_t) cannot overwrite it early.
      mbar_wait(&o_final[t], oc_cnt & 1, abort_flag, p.status, status_code(0x1a));
      ++oc_cnt;
      tc_fence_after();
      const float inv = (l_run > 0.f) ? p.drop.scale / l_run : 0.f;   // dropout's 1/(1-p) (1 without)
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(u.bh) * p.L + row) * C::Ev;
#pragma unroll
      for (int c = 0; c < C::Ev / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + c * 32, v);
        if (row < p.L) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[q4 * 8 + 0]) * inv, __uint_as_float(v[q4 * 8 + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(v[q4 * 8 + 2]) * inv, __uint_as_float(v[q4 * 8 + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(v[q4 * 8 + 4]) * inv, __uint_as_float(v[q4 * 8 + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(v[q4 * 8 + 6]) * inv, __uint_as_float(v[q4 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + q4 * 8) = w;
          }
        }
      }
      if (row < p.L)
        p.lse[static_cast<size_t>(u.bh) * p.L + row] = (l_run > 0.f) ? (m_run + __log2f(l_run)) * kLn2 : kNegInf;
      tc_fence_before();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int ECH, int VCH, int MK, bool DROP>
cudaError_t run(const FwdParams& p, cudaStream_t st) {
  using C = FwdCfg<ECH, VCH, MK>;
  alignas(64) CUtensorMap tmQ, tmK, tmV;
  if (!encode_tmap_bf16_3d(&tmQ, p.q, C::E, p.L, static_cast<uint64_t>(p.B) * p.Hq, 64, BM) ||
      !encode_tmap_bf16_3d(&tmK, p.k, C::E, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BN) ||
      !encode_tmap_bf16_3d(&tmV, p.v, C::Ev, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BN))
    return cudaErrorInvalidValue;
  alignas(64) CUtensorMap tmM = tmK;   // unused unless the mask is staged
  if (MK == kMaskStaged) {
    // the mask's distinct [L, S] slices: B x mask heads, or the heads alone, or one
    const long long LS = static_cast<long long>(p.L) * p.S;
    const long long slices = p.mask_sb ? static_cast<long long>(p.B) * (p.mask_sb / LS) : (p.mask_sh ? p.Hq : 1);
    if (!encode_tmap_f32_3d(&tmM, p.mask, p.S, p.L, static_cast<uint64_t>(slices), 32, BM, true))
      return cudaErrorInvalidValue;
  }
  auto kern = fwd_tc_kernel<ECH, VCH, MK, DROP>;
  // The register split in the kernel assumes the launch reserves exactly kRegsLaunch per thread.
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kBytes, kRegsLaunch);
  if (e != cudaSuccess) return e;
  const long long units = static_cast<long long>(p.B) * p.Hq * ((p.L + 2 * BM - 1) / (2 * BM));
  const int sms = num_sms();
  const unsigned grid = static_cast<unsigned>(units < sms ? units : sms);   // persistent: one CTA per SM
  kern<<<grid, kThreads, C::kBytes, st>>>(tmQ, tmK, tmV, tmM, p);
  return cudaGetLastError();
}

template <int MK, bool DROP>
cudaError_t launch_widths(const FwdParams& p, cudaStream_t st) {
  const int ech = p.E / 64, vch = p.Ev / 64;
  if (ech == 2 && vch == 2) return run<2, 2, MK, DROP>(p, st);
  if (ech == 1 && vch == 1) return run<1, 1, MK, DROP>(p, st);
  if (ech == 2 && vch == 1) return run<2, 1, MK, DROP>(p, st);
  return run<1, 2, MK, DROP>(p, st);
}

// Launch for one mask mode; the three mask modes are instantiated in separate
// translation units (fwd_tc.cu, fwd_tc_direct.cu, fwd_tc_staged.cu) so they compile in parallel.
template <int MK>
cudaError_t launch_mask_mode(const FwdParams& p, cudaStream_t st) {
  return p.drop.active ? launch_widths<MK, true>(p, st) : launch_widths<MK, false>(p, st);
}

}  // namespace
}  // namespace sdpa_impl
