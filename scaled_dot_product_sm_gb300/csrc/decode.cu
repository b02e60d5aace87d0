// decode.cu - memory-bound split-KV decode forward (bf16) and its merge.
//
// Problem: a few query rows (the Hq/Hkv heads of one grouped-query group,
// times L, usually L = 1) against a long key/value cache.  All the time is
// reading K and V from HBM once.  One CTA owns (batch, KV head, row group of
// up to 8 rows, key split):
//  * a producer warp streams 64-key stages of K and V into shared memory with
//    TMA tensor copies (128-byte swizzle, so the tensor-core operand reads
//    below are free of bank conflicts), NSTAGE stages in flight; with paged
//    caches it looks each stage's blocks up in the page table and copies from
//    the containers (one box per min(block size, 64) keys);
//  * four consumer warps each take 16 keys of a stage and compute the scores
//    of all rows at once as S^T = K Q^T with warp-level bf16 MMAs (rows are the
//    MMA's N = 8 side: the group's 4 query heads share every K/V byte read),
//    keep a running max and sum per row (online softmax in log2 units), and
//    accumulate O^T = V^T P^T;
//  * at the end the four warps' partial states are merged in shared memory
//    and the split's normalised partial output and log2-sum-exp are written.
// A second kernel merges the splits: lse = logsumexp_s(lse_s), o = sum_s
// exp(lse_s - lse) o_s (cuDNN "Attention" page: softmax stats, natural log
// on output, and their split-KV merges), with empty splits (lse_s = -inf)
// contributing nothing and an all-empty row giving o = 0, lse = -inf.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "sdpa.h"

namespace sdpa_impl {

namespace {

using namespace sdpa_ptx;

constexpr int kStageKeys = 64;   // the paged producer's shifts assume 64 = 2^6
constexpr int kRowsPerCta = 8;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int ECH, int VCH, int NSTAGE>
struct DecodeSmem {
  static constexpr int kKBytes = ECH * kStageKeys * 128;   // 64 keys x 64 bf16 per box
  static constexpr int kVBytes = VCH * kStageKeys * 128;
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kBytes = NSTAGE * kStageBytes + 1024 /* alignment */ + 256 /* barriers */;
};

template <int ECH, int VCH, int NSTAGE>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                const __grid_constant__ CUtensorMap tmV,
                                                                DecodeParams dp) {
  using SM = DecodeSmem<ECH, VCH, NSTAGE>;
  constexpr int E = ECH * 64, Ev = VCH * 64;
  constexpr int kKs = E / 16;     // MMA k-steps over E
  constexpr int kMt = Ev / 16;    // MMA m-tiles over Ev
  const FwdParams& p = dp.f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * SM::kStageBytes);
  uint64_t* empty = full + NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + NSTAGE);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int nrg = (p.G * p.L + kRowsPerCta - 1) / kRowsPerCta;
  const int bk = blockIdx.y / nrg, rg = blockIdx.y - bk * nrg;   // bk = b * Hkv + hkv
  const int b = bk / p.Hkv, hk = bk - b * p.Hkv;
  const int rows = p.G * p.L;
  // This split's keys, cut to those the CTA's rows can see (padding and band):
  // lo of the smallest query index .. hi of the largest one below Lb.
  const BandRows br = band_rows(p.band, b, p.L, p.S);
  int imin = p.L, imax = -1;
  for (int r = rg * kRowsPerCta; r < min(rows, (rg + 1) * kRowsPerCta); ++r) {
    const int i = r % p.L;
    imin = min(imin, i);
    imax = max(imax, i);
  }
  imax = min(imax, br.Lb - 1);
  const int k_begin = split * dp.keys_per_split;
  const int k_end = min(p.S, k_begin + dp.keys_per_split);
  const int k_lo = imax >= imin ? max(k_begin, br.lo(imin)) : k_end;
  const int k_hi = imax >= imin ? min(k_end, br.hi(imax) + 1) : k_begin;
  const int k_first = k_begin + (k_lo - k_begin) / kStageKeys * kStageKeys;   // first stage's key
  const int nst = k_hi > k_lo ? (k_hi - k_first + kStageKeys - 1) / kStageKeys : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (!dp.page_k) {
      if (lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        for (int it = 0; it < nst; ++it) {
          const int s = it % NSTAGE;
          mbar_wait(&empty[s], ((it / NSTAGE) & 1) ^ 1, abort_flag, p.status, status_code(0x21));
          uint8_t* st = smem + s * SM::kStageBytes;
          mbar_arrive_expect_tx(&full[s], SM::kStageBytes);
          const int key0 = k_first + it * kStageKeys;
#pragma unroll
          for (int c = 0; c < ECH; ++c) tma_load_3d(st + c * kStageKeys * 128, &tmK, &full[s], c * 64, key0, bk);
#pragma unroll
          for (int c = 0; c < VCH; ++c)
            tma_load_3d(st + SM::kKBytes + c * kStageKeys * 128, &tmV, &full[s], c * 64, key0, bk);
        }
      }
    } else {
      // Paged caches.  A stage's keys come from the container blocks the tables name, one
      // box per min(bs, 64) keys; a box lands on a 1024-byte (8-row) boundary, so the stage's
      // 128-byte swizzle is the same as with one 64-row box.  The warp reads the tables 32
      // boxes at a time (lane l holds box w + l) and lane 0 takes each box's entry by a shuffle.
      // An entry past the table or outside the container becomes block nblk: past the tensor
      // map, so the copy fills zeros (those keys lie past the sequence's length and are masked).
      if (lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
      }
      const int rows_k = min(dp.bs_k, kStageKeys), rows_v = min(dp.bs_v, kStageKeys);
      const int lgr_k = min(dp.lg_k, 6), lgr_v = min(dp.lg_v, 6);   // log2 of rows per box
      const int* tab_k = dp.page_k + static_cast<size_t>(b) * dp.page_stride;
      const int* tab_v = dp.page_v + static_cast<size_t>(b) * dp.page_stride;
      // z coordinate (block * Hkv + head) of box i counted from key k_first
      auto box_z = [&](const int* tab, int i, int lgr, int lg, int nblk) {
        const int blk = (k_first + (i << lgr)) >> lg;
        int page = blk < dp.page_stride ? __ldg(tab + blk) : -1;
        if (page < 0 || page >= nblk) page = nblk;
        return page * p.Hkv + hk;
      };
      int wk = 0, wv = 0;   // first box of the window each lane holds an entry of
      int zk = box_z(tab_k, lane, lgr_k, dp.lg_k, dp.nblk_k), zv = box_z(tab_v, lane, lgr_v, dp.lg_v, dp.nblk_v);
      for (int it = 0; it < nst; ++it) {
        const int s = it % NSTAGE;
        mbar_wait(&empty[s], ((it / NSTAGE) & 1) ^ 1, abort_flag, p.status, status_code(0x21));
        uint8_t* st = smem + s * SM::kStageBytes;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], SM::kStageBytes);
        const int key0 = k_first + it * kStageKeys;
        const int nbk = kStageKeys >> lgr_k, nbv = kStageKeys >> lgr_v;
        for (int sub = 0; sub < nbk; ++sub) {
          const int i = (it << (6 - lgr_k)) + sub;
          if (i >= wk + 32) {
            wk += 32;
            zk = box_z(tab_k, wk + lane, lgr_k, dp.lg_k, dp.nblk_k);
          }
          const int z = __shfl_sync(0xffffffffu, zk, i - wk);
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < ECH; ++c)
              tma_load_3d(st + c * kStageKeys * 128 + sub * rows_k * 128, &tmK, &full[s], c * 64,
                          (key0 + sub * rows_k) & (dp.bs_k - 1), z);
          }
        }
        for (int sub = 0; sub < nbv; ++sub) {
          const int i = (it << (6 - lgr_v)) + sub;
          if (i >= wv + 32) {
            wv += 32;
            zv = box_z(tab_v, wv + lane, lgr_v, dp.lg_v, dp.nblk_v);
          }
          const int z = __shfl_sync(0xffffffffu, zv, i - wv);
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < VCH; ++c)
              tma_load_3d(st + SM::kKBytes + c * kStageKeys * 128 + sub * rows_v * 128, &tmV, &full[s], c * 64,
                          (key0 + sub * rows_v) & (dp.bs_v - 1), z);
          }
        }
      }
    }
    // a wait gave up: let this warp's copies land before the CTA exits
    if (lane == 0 && *abort_flag) mbar_drain_ring(full, NSTAGE, nst);
  } else {
    // ------------------------------------------------------------ consumers
    // Q^T as the MMA's B operand (k = E, n = row): lane holds row n = lane/4,
    // k = 2*(lane%4) + {0,1} and + 8.  Rows past the group are zero.
    const int n = lane >> 2, tq = lane & 3;
    const int row_n = rg * kRowsPerCta + n;
    uint32_t qb[kKs][2];
    {
      const bool ok = row_n < rows;
      const int g = ok ? row_n / p.L : 0, i = ok ? row_n - g * p.L : 0;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          static_cast<const __nv_bfloat16*>(p.q) +
          ((static_cast<size_t>(b) * p.Hq + hk * p.G + g) * p.L + i) * E);
#pragma unroll
      for (int ks = 0; ks < kKs; ++ks) {
        qb[ks][0] = ok ? __ldg(qrow + ks * 8 + tq) : 0u;
        qb[ks][1] = ok ? __ldg(qrow + ks * 8 + 4 + tq) : 0u;
      }
    }
    // query index and mask row of the two rows (columns) this lane owns: cols 2*tq, 2*tq+1
    const float* mrow[2] = {nullptr, nullptr};
    int irow[2] = {p.L, p.L};   // rows past the group: index L, never visible
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r = rg * kRowsPerCta + 2 * tq + t;
      if (r < rows) {
        const int g = r / p.L, i = r - g * p.L;
        irow[t] = i;
        if (p.mask) mrow[t] = p.mask + b * p.mask_sb + (hk * p.G + g) * p.mask_sh + static_cast<size_t>(i) * p.S;
      }
    }
    float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
    float acc[kMt][4];
#pragma unroll
    for (int mt = 0; mt < kMt; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;

    const int kw = warp * 16;   // this warp's 16 keys within a stage
    for (int it = 0; it < nst; ++it) {
      const int s = it % NSTAGE;
      mbar_wait(&full[s], (it / NSTAGE) & 1, abort_flag, p.status, status_code(0x22));
      const uint32_t kbase = smem_u32(smem + s * SM::kStageBytes);
      const uint32_t vbase = kbase + SM::kKBytes;
      // ---- S^T = K Q^T (16 keys x 8 rows)
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int key = kw + (lane & 15);
#pragma unroll
        for (int ks = 0; ks < kKs; ++ks) {
          const int e = ks * 16 + (lane >> 4) * 8;
          const uint32_t addr = kbase + (e >> 6) * (kStageKeys * 128) + key * 128 +
                                ((((e & 63) >> 3) ^ (key & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(addr, a0, a1, a2, a3);
          mma_bf16_16816(c, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        }
      }
      // ---- scale, mask, online softmax per row (column of S^T)
      const int key0 = k_first + it * kStageKeys + kw + n;   // keys of c0/c1; +8 for c2/c3
      float x[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int key = key0 + ((t >> 1) << 3);
        float v = c[t] * p.scale_log2;
        if (key >= k_hi || !br.visible(irow[t & 1], key)) v = kNegInf;
        else if (mrow[t & 1]) v += mrow[t & 1][key] * kLog2e;
        x[t] = v;
      }
      float pr[4];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        float mx = fmaxf(x[t], x[t + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m[t], mx);
        const float msafe = (mnew == kNegInf) ? 0.f : mnew;
        const float corr = ex2(m[t] - msafe);
        pr[t] = ex2(x[t] - msafe);
        pr[t + 2] = ex2(x[t + 2] - msafe);
        float sum = pr[t] + pr[t + 2];
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        l[t] = l[t] * corr + sum;
        m[t] = mnew;
#pragma unroll
        for (int mt = 0; mt < kMt; ++mt) {
          acc[mt][t] *= corr;
          acc[mt][t + 2] *= corr;
        }
      }
      // ---- P^T as the B operand: lane needs P[key 2tq, 2tq+1, +8, +9][row n]
      const uint32_t w01 = pack_bf16x2(pr[0], pr[1]);   // key n,   rows 2tq, 2tq+1
      const uint32_t w23 = pack_bf16x2(pr[2], pr[3]);   // key n+8, rows 2tq, 2tq+1
      const int src = 8 * tq + (n >> 1);
      const uint32_t x01a = __shfl_sync(0xffffffffu, w01, src);
      const uint32_t x01b = __shfl_sync(0xffffffffu, w01, src + 4);
      const uint32_t x23a = __shfl_sync(0xffffffffu, w23, src);
      const uint32_t x23b = __shfl_sync(0xffffffffu, w23, src + 4);
      const uint32_t sel = (n & 1) ? 0x7632u : 0x5410u;
      const uint32_t pb0 = __byte_perm(x01a, x01b, sel);
      const uint32_t pb1 = __byte_perm(x23a, x23b, sel);
      // ---- O^T += V^T P^T
      {
        const int mi = lane >> 3;
        const int key = kw + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int mt = 0; mt < kMt; ++mt) {
          const int ev = mt * 16 + (mi & 1) * 8;
          const uint32_t addr = vbase + (ev >> 6) * (kStageKeys * 128) + key * 128 +
                                ((((ev & 63) >> 3) ^ (key & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(addr, a0, a1, a2, a3);
          mma_bf16_16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // every stage issued has been consumed by this warp; fall through to the merge
    // (lanes with the same tq hold identical m, l; acc rows = Ev index)
    __syncwarp();
    // per-warp row statistics, then (after every consumer warp has left the
    // pipeline) the accumulators in the freed stage memory
    __shared__ float s_m[kConsumerWarps][kRowsPerCta], s_l[kConsumerWarps][kRowsPerCta];
    if (n == 0) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        s_m[warp][2 * tq + t] = m[t];
        s_l[warp][2 * tq + t] = l[t];
      }
    }
    // wait for every consumer warp to leave the pipeline before reusing stage memory
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    float* sacc = reinterpret_cast<float*>(smem);    // [warp][row 8][Ev]
#pragma unroll
    for (int mt = 0; mt < kMt; ++mt) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int ev = mt * 16 + n + ((t >> 1) << 3);
        const int r = 2 * tq + (t & 1);
        sacc[(warp * kRowsPerCta + r) * Ev + ev] = acc[mt][t];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    // combine: thread -> (row r, 8 consecutive ev)
    const int tid = threadIdx.x;
    constexpr int kPerRow = Ev / 8;
    for (int w = tid; w < kRowsPerCta * kPerRow; w += kConsumerWarps * 32) {
      const int r = w / kPerRow, e0 = (w - r * kPerRow) * 8;
      const int grow = rg * kRowsPerCta + r;
      if (grow >= rows) continue;
      float M = kNegInf;
#pragma unroll
      for (int ww = 0; ww < kConsumerWarps; ++ww) M = fmaxf(M, s_m[ww][r]);
      float wsc[kConsumerWarps], lsum = 0.f;
      const float Ms = (M == kNegInf) ? 0.f : M;
#pragma unroll
      for (int ww = 0; ww < kConsumerWarps; ++ww) {
        wsc[ww] = ex2(s_m[ww][r] - Ms);
        lsum += wsc[ww] * s_l[ww][r];
      }
      const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
      const int g = grow / p.L, i = grow - g * p.L;
      const size_t orow = (static_cast<size_t>(b) * p.Hq + hk * p.G + g) * p.L + i;
      float* po = dp.part_o + (orow * dp.nsplit + split) * Ev + e0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float v = 0.f;
#pragma unroll
        for (int ww = 0; ww < kConsumerWarps; ++ww) v += wsc[ww] * sacc[(ww * kRowsPerCta + r) * Ev + e0 + e];
        po[e] = v * inv;
      }
      if (e0 == 0) dp.part_lse[orow * dp.nsplit + split] = (lsum > 0.f) ? M + __log2f(lsum) : kNegInf;
    }
  }
}

// One warp per output row: combine nsplit partial (o_s, lse_s) into o, lse.
template <int Ev>
__global__ void __launch_bounds__(128) decode_merge_kernel(DecodeParams dp) {
  const FwdParams& p = dp.f;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.L;
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* pl = dp.part_lse + row * dp.nsplit;
  float M = kNegInf;
  for (int s = lane; s < dp.nsplit; s += 32) M = fmaxf(M, pl[s]);
  M = warp_max(M);
  constexpr int kPer = Ev / 32;
  float o[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) o[e] = 0.f;
  float W = 0.f;
  if (M != kNegInf) {
    for (int s = 0; s < dp.nsplit; ++s) {
      const float w = ex2(pl[s] - M);
      W += w;
      const float* po = dp.part_o + (row * dp.nsplit + s) * Ev;
#pragma unroll
      for (int e = 0; e < kPer; ++e) o[e] = fmaf(w, po[lane + 32 * e], o[e]);
    }
  }
  const float inv = (W > 0.f) ? 1.f / W : 0.f;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.o) + row * Ev;
#pragma unroll
  for (int e = 0; e < kPer; ++e) out[lane + 32 * e] = __float2bfloat16_rn(o[e] * inv);
  if (lane == 0) p.lse[row] = (W > 0.f) ? (M + __log2f(W)) * kLn2 : kNegInf;
}

template <int ECH, int VCH>
cudaError_t run(const DecodeParams& dp, cudaStream_t st) {
  constexpr int NSTAGE = (ECH + VCH) <= 2 ? 6 : 4;
  using SM = DecodeSmem<ECH, VCH, NSTAGE>;
  const FwdParams& p = dp.f;
  alignas(64) CUtensorMap tmK, tmV;
  if (!dp.page_k) {
    if (!encode_tmap_bf16_3d(&tmK, p.k, ECH * 64, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, kStageKeys))
      return cudaErrorInvalidValue;
    if (!encode_tmap_bf16_3d(&tmV, p.v, VCH * 64, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, kStageKeys))
      return cudaErrorInvalidValue;
  } else {   // containers [nblk, Hkv, bs, E|Ev] as (E|Ev, bs, nblk * Hkv), boxes of min(bs, 64) rows
    if (!encode_tmap_bf16_3d(&tmK, p.k, ECH * 64, dp.bs_k, static_cast<uint64_t>(dp.nblk_k) * p.Hkv, 64,
                             std::min(dp.bs_k, kStageKeys)) ||
        !encode_tmap_bf16_3d(&tmV, p.v, VCH * 64, dp.bs_v, static_cast<uint64_t>(dp.nblk_v) * p.Hkv, 64,
                             std::min(dp.bs_v, kStageKeys)))
      return cudaErrorInvalidValue;
  }
  auto kern = decode_split_kernel<ECH, VCH, NSTAGE>;
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), SM::kBytes, 0);
  if (e != cudaSuccess) return e;
  const int nrg = (p.G * p.L + kRowsPerCta - 1) / kRowsPerCta;
  dim3 grid(dp.nsplit, p.B * p.Hkv * nrg);
  kern<<<grid, kThreads, SM::kBytes, st>>>(tmK, tmV, dp);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.L;
  const unsigned mblocks = static_cast<unsigned>((rows + 3) / 4);
  if (VCH == 1)
    decode_merge_kernel<64><<<mblocks, 128, 0, st>>>(dp);
  else
    decode_merge_kernel<128><<<mblocks, 128, 0, st>>>(dp);
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(int E, int Ev) { return (E == 64 || E == 128) && (Ev == 64 || Ev == 128); }
int decode_rows_per_cta() { return kRowsPerCta; }
int decode_stage_keys() { return kStageKeys; }

cudaError_t launch_decode(const DecodeParams& dp, cudaStream_t st) {
  const int ech = dp.f.E / 64, vch = dp.f.Ev / 64;
  if (ech == 2 && vch == 2) return run<2, 2>(dp, st);
  if (ech == 1 && vch == 1) return run<1, 1>(dp, st);
  if (ech == 2 && vch == 1) return run<2, 1>(dp, st);
  return run<1, 2>(dp, st);
}

// ---------------------------------------------------------------- fixed scratch
// Split partials of sdpa_decode_noalloc, for callers that cannot hand the
// library a workspace.  A file-scope device array: every GPU that loads the
// library holds one copy of SDPA_DECODE_STATIC_SCRATCH_BYTES until the process
// exits.  Host code must not pass g_decode_scratch itself to a kernel (on the
// host that name is only a stand-in); decode_static_scratch() looks up its
// device address once per device, with that device current.
static __device__ __align__(256) unsigned char g_decode_scratch[SDPA_DECODE_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kScratchDevices] = {};
unsigned long long g_scratch_ctx[kScratchDevices] = {};   // context the address belongs to
}  // namespace

cudaError_t decode_static_scratch(void** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  // A cached address is reused only inside the context it was looked up in:
  // after cudaDeviceReset the device's next context loads the array anew.
  const unsigned long long ctx = current_context_id();
  if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = addr;
    g_scratch_ctx[dev] = current_context_id();
  }
  *ptr = g_scratch_addr[dev];
  *bytes = sizeof(g_decode_scratch);
  return cudaSuccess;
}

}  // namespace sdpa_impl
