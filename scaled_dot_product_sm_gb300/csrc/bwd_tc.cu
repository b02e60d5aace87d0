// bwd_tc.cu - bf16 backward on the 5th-generation tensor cores (E = Ev = 128).
//
// The hand-derived backward of the course chapter "Scaled dot-product
// attention (forward and backward)", section 2.3:
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),  D_i = dO_i . O_i,
//   dQ = alpha dS K,  dK = alpha dS^T Q,
// with P rebuilt from the forward's log-sum-exp (P_ij = exp(s_ij - lse_i))
// instead of being stored, as the GPU path of "ScaledDotProductAttentionBackward"
// (apply) and the FlashAttention-2 backward the chapter points to do.
//
// Three launches:
//  1. rowstats: per query row (-lse*log2(e), D) as a float2 (rows padded to a
//     multiple of 64 with (-inf, 0), so a padded or fully masked row has P = 0),
//     and the fp32 dQ accumulator zeroed;
//  2. the main kernel, one CTA per (batch, KV head, 128-key tile).  K and V stay
//     in shared memory; the CTA walks the Hq/Hkv query heads of its group and
//     their 64-row query tiles (last to first, down to the diagonal when causal), so dK and dV
//     are summed over the group inside the CTA (no atomics for them):
//        S^T  = K Q^T          (TMEM, 128 keys x 64 queries)
//        dP^T = V dO^T         (TMEM)
//        P^T  = exp2(S^T alpha log2e + mask log2e - lse log2e),  dS^T = P^T o (dP^T - D)
//        dV  += P^T dO,  dK += dS^T Q     (TMEM accumulators, 128 x 128 each)
//        dQ^T = K^T dS^T       (TMEM, 128 head dims x 64 queries)
//     dQ^T puts the head dimension on the TMEM lanes, so the four drain warps
//     add each query's 128 fp32 values to the global accumulator with fully
//     coalesced reductions (red.global.add.f32, 128 bytes per warp instruction);
//  3. dQ = bf16(accumulator).
// Warp roles (320 threads): warps 0-3 elementwise (thread = key = TMEM lane),
// warps 4-7 dQ drain (thread = head dim = TMEM lane), warp 8 TMA producer,
// warp 9 TMEM allocator and single-thread MMA issuer.  S^T(i+1) and dP^T(i+1)
// are issued as soon as the elementwise warps have read S^T(i) and dP^T(i), so
// the tensor core computes the next scores while the current gradients wait for
// P^T and dS^T.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa_impl {

namespace {

using namespace sdpa_ptx;

constexpr int E = 128, Ev = 128;
constexpr int BKV = 128;       // keys per CTA
constexpr int BQ = 64;         // queries per iteration
constexpr int kThreads = 320;
constexpr int kNSQ = 3;        // query-tile stages (prefetch two tiles ahead)
constexpr float kNegInf = -__builtin_huge_valf();

// shared memory map (bytes; every operand block 1024-aligned)
constexpr int kKBytes = 2 * BKV * 128;                 // K tile: 2 chunks of [128 keys x 64 dims]
constexpr int kQTile = 2 * BQ * 128;                   // Q (or dO) tile: 2 chunks of [64 rows x 64 dims]
constexpr int kStage = 2 * kQTile + 1024;              // Q, dO, rowstats (512 B, padded)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKBytes;
constexpr int kOffStage = kOffV + kKBytes;
constexpr int kOffP = kOffStage + kNSQ * kStage;       // P^T [128 keys x 64 queries] bf16
constexpr int kOffDS = kOffP + BKV * 128;              // dS^T
constexpr int kOffBar = kOffDS + BKV * 128;
constexpr int kSmemBytes = kOffBar + 256 + 1024;

// TMEM columns
constexpr uint32_t kColDK = 0, kColDV = 128, kColS = 256, kColDP = 320, kColDQ = 384;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

struct TcBwdArgs {
  BwdParams p;
  const float2* rowstats;   // [B*Hq][Lpad] (-lse*log2e, D)
  int Lpad;
};

__global__ void __launch_bounds__(256) bwd_rowstats_kernel(TcBwdArgs a) {
  const BwdParams& p = a.p;
  const long long rows = static_cast<long long>(p.B) * p.Hq * a.Lpad;
  const long long gr = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gr >= rows) return;
  const long long bh = gr / a.Lpad;
  const int q = static_cast<int>(gr - bh * a.Lpad);
  float2 st = make_float2(kNegInf, 0.f);
  if (q < p.L) {
    const size_t row = static_cast<size_t>(bh) * p.L + q;
    const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(p.o) + row * Ev;
    const __nv_bfloat16* dO = static_cast<const __nv_bfloat16*>(p.dO) + row * Ev;
    const __nv_bfloat162 a2 = reinterpret_cast<const __nv_bfloat162*>(o)[lane * 2];
    const __nv_bfloat162 b2 = reinterpret_cast<const __nv_bfloat162*>(o)[lane * 2 + 1];
    const __nv_bfloat162 c2 = reinterpret_cast<const __nv_bfloat162*>(dO)[lane * 2];
    const __nv_bfloat162 d2 = reinterpret_cast<const __nv_bfloat162*>(dO)[lane * 2 + 1];
    float s = __low2float(a2) * __low2float(c2);
    s = fmaf(__high2float(a2), __high2float(c2), s);
    s = fmaf(__low2float(b2), __low2float(d2), s);
    s = fmaf(__high2float(b2), __high2float(d2), s);
    s = warp_sum(s);
    const float lse = p.lse[row];
    st = make_float2(lse == kNegInf ? kNegInf : -lse * kLog2e, s);
    float4* acc = reinterpret_cast<float4*>(p.dq_acc + row * E);
    acc[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (lane == 0) const_cast<float2*>(a.rowstats)[gr] = st;
}

__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdParams p) {
  const size_t n8 = static_cast<size_t>(p.B) * p.Hq * p.L * E / 8;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(p.dq_acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(p.dq_acc)[2 * i + 1];
    uint4 w;
    w.x = pack_bf16x2(a.x, a.y);
    w.y = pack_bf16x2(a.z, a.w);
    w.z = pack_bf16x2(b.x, b.y);
    w.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(p.dq)[i] = w;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO, TcBwdArgs a) {
  const BwdParams& p = a.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kv_full = bar;                 // 1
  uint64_t* q_full = bar + 1;              // kNSQ
  uint64_t* q_empty = q_full + kNSQ;       // kNSQ
  uint64_t* s_full = q_empty + kNSQ;       // 1
  uint64_t* s_free = s_full + 1;           // 1
  uint64_t* dp_full = s_free + 1;          // 1
  uint64_t* dp_free = dp_full + 1;         // 1
  uint64_t* p_full = dp_free + 1;          // 1
  uint64_t* p_free = p_full + 1;           // 1
  uint64_t* dq_full = p_free + 1;          // 1
  uint64_t* dq_free = dq_full + 1;         // 1
  uint64_t* kdv_done = dq_free + 1;        // 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(kdv_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bkv = blockIdx.x, b = bkv / p.Hkv, hkv = bkv - b * p.Hkv;
  const int k0 = blockIdx.y * BKV;                       // heaviest (causal) tiles first
  const int nqt = (p.L + BQ - 1) / BQ;
  const int qt_begin = p.causal ? min(k0 / BQ, nqt) : 0;
  const int per_head = nqt - qt_begin;
  const int n = p.G * per_head;                          // iterations
  // Iteration i -> (query tile, head): tiles from the last down to the diagonal,
  // the group's heads innermost.  Every CTA of a KV group starts at the same
  // (last) tile and walks down in step, so the CTAs running at the same time
  // read the same Q/dO tiles and mostly hit in L2.
  auto tile_of = [&](int i, int& qt, int& g) {
    qt = nqt - 1 - i / p.G;
    g = i - (i / p.G) * p.G;
  };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < kNSQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);     // one arrival per elementwise warp
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 4);
    mbar_init(p_full, 4);
    mbar_init(p_free, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);    // one arrival per drain warp
    mbar_init(kdv_done, 1);
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

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n > 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmdO);
      mbar_arrive_expect_tx(kv_full, 2 * kKBytes);
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(smem + kOffK + c * BKV * 128, &tmK, kv_full, c * 64, k0, bkv);
        tma_load_3d(smem + kOffV + c * BKV * 128, &tmV, kv_full, c * 64, k0, bkv);
      }
      for (int i = 0; i < n; ++i) {
        const int s = i % kNSQ;
        int qt, g;
        tile_of(i, qt, g);
        const int bh = b * p.Hq + hkv * p.G + g;
        mbar_wait(&q_empty[s], ((i / kNSQ) & 1) ^ 1, abort_flag, p.status, status_code(0x31));
        uint8_t* st = smem + kOffStage + s * kStage;
        mbar_arrive_expect_tx(&q_full[s], 2 * kQTile + BQ * 8);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(st + c * BQ * 128, &tmQ, &q_full[s], c * 64, qt * BQ, bh);
          tma_load_3d(st + kQTile + c * BQ * 128, &tmdO, &q_full[s], c * 64, qt * BQ, bh);
        }
        bulk_load(st + 2 * kQTile, a.rowstats + static_cast<size_t>(bh) * a.Lpad + qt * BQ, BQ * 8, &q_full[s]);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t id_s = idesc_bf16(BKV, BQ, 0, 0);     // S^T, dP^T: K-major x K-major
      constexpr uint32_t id_kv = idesc_bf16(BKV, E, 0, 1);     // dV, dK: K-major x MN-major
      constexpr uint32_t id_q = idesc_bf16(E, BQ, 1, 1);       // dQ^T: MN-major x MN-major
      const uint32_t kA = smem_u32(smem + kOffK), vA = smem_u32(smem + kOffV);
      const uint32_t pA = smem_u32(smem + kOffP), dsA = smem_u32(smem + kOffDS);
      const uint32_t stage0 = smem_u32(smem + kOffStage);
      mbar_wait(kv_full, 0, abort_flag, p.status, status_code(0x32));
      auto issue_sdp = [&](int i) {
        const int s = i % kNSQ;
        mbar_wait(&q_full[s], (i / kNSQ) & 1, abort_flag, p.status, status_code(0x33));
        tc_fence_after();
        const uint32_t qA = stage0 + s * kStage, doA = qA + kQTile;
        if (i > 0) {
          mbar_wait(s_free, (i - 1) & 1, abort_flag, p.status, status_code(0x34));
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < E / 16; ++kk) {
          umma_ss(tmem + kColS, sdesc_sw128(kA + (kk >> 2) * (BKV * 128) + (kk & 3) * 32, 16, 1024),
                  sdesc_sw128(qA + (kk >> 2) * (BQ * 128) + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
        }
        umma_commit(s_full);
        if (i > 0) {
          mbar_wait(dp_free, (i - 1) & 1, abort_flag, p.status, status_code(0x35));
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < Ev / 16; ++kk) {
          umma_ss(tmem + kColDP, sdesc_sw128(vA + (kk >> 2) * (BKV * 128) + (kk & 3) * 32, 16, 1024),
                  sdesc_sw128(doA + (kk >> 2) * (BQ * 128) + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
        }
        umma_commit(dp_full);
      };
      issue_sdp(0);
      for (int i = 0; i < n; ++i) {
        if (i + 1 < n) issue_sdp(i + 1);
        const int s = i % kNSQ;
        const uint32_t qA = stage0 + s * kStage, doA = qA + kQTile;
        mbar_wait(p_full, i & 1, abort_flag, p.status, status_code(0x36));
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {   // dV += P^T dO ; dK += dS^T Q   (K = queries)
          umma_ss(tmem + kColDV, sdesc_sw128(pA + kk * 32, 16, 1024),
                  sdesc_sw128(doA + kk * 16 * 128, BQ * 128, 1024), id_kv, (i > 0 || kk > 0) ? 1u : 0u);
          umma_ss(tmem + kColDK, sdesc_sw128(dsA + kk * 32, 16, 1024),
                  sdesc_sw128(qA + kk * 16 * 128, BQ * 128, 1024), id_kv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&q_empty[s]);
        if (i > 0) {
          mbar_wait(dq_free, (i - 1) & 1, abort_flag, p.status, status_code(0x37));
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {  // dQ^T = K^T dS^T   (K = keys)
          umma_ss(tmem + kColDQ, sdesc_sw128(kA + kk * 16 * 128, BKV * 128, 1024),
                  sdesc_sw128(dsA + kk * 16 * 128, BQ * 128, 1024), id_q, kk > 0);
        }
        umma_commit(p_free);
        umma_commit(dq_full);
      }
      umma_commit(kdv_done);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ elementwise warps (thread = key)
    const int r = warp * 32 + lane;
    const int key = k0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    uint8_t* prow = smem + kOffP + r * 128;
    uint8_t* dsrow = smem + kOffDS + r * 128;
    for (int i = 0; i < n; ++i) {
      const int s = i % kNSQ;
      int qt, g;
      tile_of(i, qt, g);
      const int h = hkv * p.G + g;
      const int q0 = qt * BQ;
      const float2* rs = reinterpret_cast<const float2*>(smem + kOffStage + s * kStage + 2 * kQTile);
      mbar_wait(&q_full[s], (i / kNSQ) & 1, abort_flag, p.status, status_code(0x38));
      mbar_wait(s_full, i & 1, abort_flag, p.status, status_code(0x39));
      tc_fence_after();
      float x[BQ];
      {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColS, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
        tmem_ld32(tmem + lane_off + kColS + 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[32 + j] = __uint_as_float(v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      const float* mcol = (p.mask && key < p.S)
                              ? p.mask + b * p.mask_sb + h * p.mask_sh + static_cast<size_t>(q0) * p.S + key
                              : nullptr;
      const bool dead_key = key >= p.S;
      const bool diag = p.causal && (k0 + BKV - 1 > q0);
#pragma unroll
      for (int j = 0; j < BQ; ++j) {
        float t = fmaf(x[j], p.scale_log2, rs[j].x);
        if (mcol && q0 + j < p.L) t = fmaf(__ldg(mcol + static_cast<size_t>(j) * p.S), kLog2e, t);
        if (dead_key || (diag && key > q0 + j)) t = kNegInf;
        x[j] = ex2(t);                                   // P^T
      }
      mbar_wait(dp_full, i & 1, abort_flag, p.status, status_code(0x3a));
      tc_fence_after();
      float d[BQ];
      {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColDP, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) d[j] = __uint_as_float(v[j]);
        tmem_ld32(tmem + lane_off + kColDP + 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) d[32 + j] = __uint_as_float(v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_free);
#pragma unroll
      for (int j = 0; j < BQ; ++j) d[j] = x[j] * (d[j] - rs[j].y);   // dS^T
      if (i > 0) mbar_wait(p_free, (i - 1) & 1, abort_flag, p.status, status_code(0x3b));
#pragma unroll
      for (int c = 0; c < BQ / 8; ++c) {
        uint4 w, u;
        w.x = pack_bf16x2(x[8 * c + 0], x[8 * c + 1]);
        w.y = pack_bf16x2(x[8 * c + 2], x[8 * c + 3]);
        w.z = pack_bf16x2(x[8 * c + 4], x[8 * c + 5]);
        w.w = pack_bf16x2(x[8 * c + 6], x[8 * c + 7]);
        u.x = pack_bf16x2(d[8 * c + 0], d[8 * c + 1]);
        u.y = pack_bf16x2(d[8 * c + 2], d[8 * c + 3]);
        u.z = pack_bf16x2(d[8 * c + 4], d[8 * c + 5]);
        u.w = pack_bf16x2(d[8 * c + 6], d[8 * c + 7]);
        const int off = (c ^ (r & 7)) << 4;
        *reinterpret_cast<uint4*>(prow + off) = w;
        *reinterpret_cast<uint4*>(dsrow + off) = u;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ---------------------------------------------------------- dK, dV epilogue
    __nv_bfloat16* dkrow = static_cast<__nv_bfloat16*>(p.dk) + (static_cast<size_t>(bkv) * p.S + key) * E;
    __nv_bfloat16* dvrow = static_cast<__nv_bfloat16*>(p.dv) + (static_cast<size_t>(bkv) * p.S + key) * Ev;
    if (n > 0) {
      mbar_wait(kdv_done, 0, abort_flag, p.status, status_code(0x3c));
      tc_fence_after();
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t col = m == 0 ? kColDK : kColDV;
      const float sc = m == 0 ? p.scale : 1.f;
      __nv_bfloat16* dst = m == 0 ? dkrow : dvrow;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_off + col + c * 32, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
        if (key < p.S) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[u * 8 + 0]) * sc, __uint_as_float(v[u * 8 + 1]) * sc);
            w.y = pack_bf16x2(__uint_as_float(v[u * 8 + 2]) * sc, __uint_as_float(v[u * 8 + 3]) * sc);
            w.z = pack_bf16x2(__uint_as_float(v[u * 8 + 4]) * sc, __uint_as_float(v[u * 8 + 5]) * sc);
            w.w = pack_bf16x2(__uint_as_float(v[u * 8 + 6]) * sc, __uint_as_float(v[u * 8 + 7]) * sc);
            *reinterpret_cast<uint4*>(dst + c * 32 + u * 8) = w;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ drain (thread = head dim)
    const int e = (warp - 4) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 4) * 32) << 16;
    for (int i = 0; i < n; ++i) {
      int qt, g;
      tile_of(i, qt, g);
      const int bh = b * p.Hq + hkv * p.G + g;
      const int q0 = qt * BQ;
      mbar_wait(dq_full, i & 1, abort_flag, p.status, status_code(0x3d));
      tc_fence_after();
      uint32_t v0[32], v1[32];
      tmem_ld32(tmem + lane_off + kColDQ, v0);
      tmem_ld32(tmem + lane_off + kColDQ + 32, v1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      float* dst = p.dq_acc + (static_cast<size_t>(bh) * p.L + q0) * E + e;
      const int nq = min(BQ, p.L - q0);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < nq) red_add_f32(dst + static_cast<size_t>(j) * E, __uint_as_float(v0[j]) * p.scale);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (32 + j < nq) red_add_f32(dst + static_cast<size_t>(32 + j) * E, __uint_as_float(v1[j]) * p.scale);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool bwd_tc_supported(int E_, int Ev_) { return E_ == E && Ev_ == Ev; }

int bwd_tc_row_pad() { return BQ; }

cudaError_t launch_bwd_tc(const BwdParams& p, cudaStream_t st) {
  TcBwdArgs a;
  a.p = p;
  a.Lpad = (p.L + BQ - 1) / BQ * BQ;
  a.rowstats = reinterpret_cast<const float2*>(p.D);
  const long long srows = static_cast<long long>(p.B) * p.Hq * a.Lpad;
  bwd_rowstats_kernel<<<static_cast<unsigned>((srows + 7) / 8), 256, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tmK, tmV, tmQ, tmdO;
  if (!encode_tmap_bf16_3d(&tmK, p.k, E, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BKV) ||
      !encode_tmap_bf16_3d(&tmV, p.v, Ev, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BKV) ||
      !encode_tmap_bf16_3d(&tmQ, p.q, E, p.L, static_cast<uint64_t>(p.B) * p.Hq, 64, BQ) ||
      !encode_tmap_bf16_3d(&tmdO, p.dO, Ev, p.L, static_cast<uint64_t>(p.B) * p.Hq, 64, BQ))
    return cudaErrorInvalidValue;
  if ((e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) !=
      cudaSuccess)
    return e;
  dim3 grid(p.B * p.Hkv, (p.S + BKV - 1) / BKV);
  bwd_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(tmK, tmV, tmQ, tmdO, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t n8 = static_cast<size_t>(p.B) * p.Hq * p.L * E / 8;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n8 + 255) / 256, 152 * 16));
  bwd_dq_convert_kernel<<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sdpa_impl
