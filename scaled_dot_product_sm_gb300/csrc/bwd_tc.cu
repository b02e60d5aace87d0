// bwd_tc.cu - bf16 backward on the 5th-generation tensor cores (E = Ev = 64 or 128).
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
//  1. rowstats: per 64-row query tile, the 64 values -lse*log2(e) followed by
//     the 64 values -D (rows padded to a multiple of 64 with (-inf, 0), so a
//     padded or fully masked row has P = 0), and the fp32 dQ accumulator zeroed;
//  2. the main kernel, one CTA per (batch, KV head, 128-key tile).  K and V stay
//     in shared memory; the CTA walks the Hq/Hkv query heads of its group and
//     their 64-row query tiles (last to first, down to the diagonal when
//     causal), so dK and dV are summed over the group inside the CTA:
//        S^T  = K Q^T                       (TMEM, 128 keys x 64 queries, two buffers)
//        dP^T = V dO^T                      (TMEM)
//        P^T  = exp2(S^T alpha log2e + mask log2e - lse log2e),  dS^T = P^T o (dP^T - D)
//        dV  += P^T dO                      (A operand P^T in TMEM, over the scores it came from)
//        dK  += dS^T Q,  dQ^T = K^T dS^T    (dS^T in shared memory, two buffers; dQ^T in TMEM,
//                                            128 head dims x 64 queries)
//     dQ^T goes from TMEM to the drain warps' registers and is added (without
//     alpha) to the global fp32 accumulator by reductions in L2: for each query
//     a warp adds 32 consecutive floats, one full 128-byte line.  Nothing is
//     staged in shared memory, whose bandwidth the SS MMAs (K and Q, V and dO,
//     K^T and dS^T) already use heavily; the 32 KB saved give the masked
//     variant its third query-tile stage.  At the end the eight elementwise
//     warps write dK (times alpha) and dV as bf16 through the idle query-tile
//     stages, and one thread stores them with TMA;
//  3. dQ = bf16(alpha * accumulator).
// The main kernel and the conversion are programmatic dependent launches: each
// starts while the grid before it finishes, and waits for it (griddepcontrol)
// before touching its results, which hides their launch and set-up.
// Warp roles (512 threads, four warpgroups with a register split):
//   warps 0-7   elementwise (thread = key = TMEM lane; warps w and w+4 share
//               the lane quarter and take query columns 0-31 / 32-63)    152 regs
//   warps 8-11  dQ drain (thread = head dim = TMEM lane)                  136 regs
//   warp  12    TMA producer                                              72 regs
//   warp  13    TMEM allocator and issuer of the gradient MMAs (dV, dK, dQ^T)
//   warp  14    issuer of the score MMAs (S^T, dP^T)
//   warp  15    idle (it completes the fourth warpgroup)
// TMEM (512 columns): dK [0,128), dV [128,256), S^T buffers [256,320) and
// [320,384) (iteration i uses buffer i & 1), dP^T [384,448), dQ^T [448,512).
// Two threads issue MMAs into the one tensor pipe.  The score issuer puts S^T(i)
// in as soon as dV(i-2) has read P^T(i-2) out of the same buffer, which is about
// an iteration before the elementwise warps need it, and dP^T(i) once they have
// read dP^T(i-1); the gradient issuer puts dV(i) in once P^T(i) is stored, then
// dK(i) and dQ^T(i) once dS^T(i) is in shared memory.  The pipe accepts only a
// few MMAs ahead, so with one issuer every barrier it waited on let the pipe
// run dry; with two, one thread's wait does not stop the other's work.  Each
// double buffer has a barrier pair per buffer, so no wait ever has to tell apart
// two phases of one barrier.  dK reads dS^T from shared memory (where dQ^T needs
// it anyway) rather than from a TMEM copy: the 32 columns go to the second S^T
// buffer.  Against one S^T buffer, P^T and dS^T in TMEM and the row statistics
// inside each 1 KB-padded query-tile stage, this layout took the causal E = 128
// backward from 0.636 to 0.610 ms and the non-causal one from 1.240 to 1.172 ms.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace sdpa_impl {

namespace {

using namespace sdpa_ptx;

constexpr int BKV = 128;       // keys per CTA
constexpr int BQ = 64;         // queries per iteration
constexpr int kThreads = 512;
constexpr float kNegInf = -__builtin_huge_valf();

constexpr int kRegsLaunch = 128;
constexpr int kRegsElem = 152, kRegsDrain = 136, kRegsOther = 72;
static_assert(128 * (2 * kRegsElem + kRegsDrain + kRegsOther) <= kThreads * kRegsLaunch, "register split too large");
static_assert(2 * kRegsElem + kRegsDrain + kRegsOther <= 512, "per sub-partition register file exceeded");
constexpr int kHalf = BQ / 2;   // query columns per elementwise warp

// Shared memory map for head width E = Ev (bytes; every operand block 1024-aligned).
// The dQ^T MMA always runs with M = 128: at E = 64 its A rows 64..127 read the
// 64-dim block after K (the start of V), and the drain never reads those rows of
// dQ^T, so they cannot reach the result.
template <int E_, bool MSTAGE>
struct BwdCfg {
  static constexpr int E = E_, Ev = E_;
  static constexpr int ECH = E / 64;                          // 64-element column blocks
  // query-tile stages: three at E = 128 (a fourth misses the 227 KB by 256 bytes), four at
  // E = 64, where they fit easily (C2 backward 0.0706 -> 0.0671 ms, and 0.551 -> 0.492 ms on
  // the GQA causal shape at E = 64, against three stages)
  static constexpr int NSQ = E_ == 64 ? 4 : 3;
  static constexpr int kKBytes = ECH * BKV * 128;             // K tile: ECH blocks of [128 keys x 64 dims]
  static constexpr int kQTile = ECH * BQ * 128;               // Q (or dO) tile: ECH blocks of [64 rows x 64 dims]
  static constexpr int kStage = 2 * kQTile;                   // Q, dO
  static constexpr int kMaskBytes = MSTAGE ? BQ * BKV * 4 : 0;   // additive mask [64 queries x 128 keys] fp32
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKBytes;
  static constexpr int kOffStage = kOffV + kKBytes;
  // dS^T [128 keys x 64 queries] bf16, 128-byte swizzled, two buffers
  static constexpr int NDS = 2;
  static constexpr int kOffDS = kOffStage + NSQ * kStage;
  static constexpr int kOffRS = kOffDS + NDS * BKV * 128;     // row statistics of each stage (512 B)
  static constexpr int kOffMask = kOffRS + NSQ * BQ * 8;      // mask tile (TMA, one iteration ahead)
  static constexpr int kOffBar = kOffMask + kMaskBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static_assert(E == 64 || E == 128, "head width");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

// TMEM columns
constexpr uint32_t kColDK = 0, kColDV = 128, kColS = 256, kColDP = 384, kColDQ = 448;   // S^T: two 64-column buffers
// P^T(i) (bf16 pairs) overwrites the S^T buffer it came from: warp half hf puts its 32 queries'
// 16 columns at hf*32, inside the columns it read, so no other warp's scores are overwritten.
__device__ __forceinline__ uint32_t p_col(int buf, int kk16) {   // column of P^T queries 16*kk16..
  return kColS + buf * 64 + (kk16 >> 1) * 32 + (kk16 & 1) * 8;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void red_add_f32(float* gdst, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(gdst), "f"(v) : "memory");
}

struct TcBwdArgs {
  BwdParams p;
  const float* rowstats;   // per (head, 64-row query tile): 64 x (-lse*log2e), then 64 x (-D)
  int Lpad;
  int mslice_b, mslice_h;  // staged mask: [L, S] slice of (b, h) = b * mslice_b + h * mslice_h
};

template <int E>
__global__ void __launch_bounds__(256) bwd_rowstats_kernel(TcBwdArgs a) {
  // the main kernel may launch as soon as every block of this grid has started
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const BwdParams& p = a.p;
  const long long rows = static_cast<long long>(p.B) * p.Hq * a.Lpad;
  const long long gr = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gr >= rows) return;
  const long long bh = gr / a.Lpad;
  const int q = static_cast<int>(gr - bh * a.Lpad);
  float nl = kNegInf, nd = 0.f;
  if (q < p.L) {
    const size_t row = static_cast<size_t>(bh) * p.L + q;
    const __nv_bfloat162* o =
        reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(p.o) + row * E);
    const __nv_bfloat162* dO =
        reinterpret_cast<const __nv_bfloat162*>(static_cast<const __nv_bfloat16*>(p.dO) + row * E);
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < E / 64; ++u) {   // this lane's E/32 elements, as E/64 bf16 pairs
      const __nv_bfloat162 a2 = o[lane * (E / 64) + u], c2 = dO[lane * (E / 64) + u];
      s = fmaf(__low2float(a2), __low2float(c2), s);
      s = fmaf(__high2float(a2), __high2float(c2), s);
    }
    s = warp_sum(s);
    const float lse = p.lse[row];
    nl = lse == kNegInf ? kNegInf : -lse * kLog2e;
    nd = -s;
    float4* acc = reinterpret_cast<float4*>(p.dq_acc + row * E);
    if (lane < E / 4) acc[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (lane == 0) {
    float* tile = const_cast<float*>(a.rowstats) + (gr - (q & (BQ - 1))) * 2;   // this row's 64-row tile
    tile[q & (BQ - 1)] = nl;
    tile[BQ + (q & (BQ - 1))] = nd;
  }
}

template <int E>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(BwdParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the main kernel's accumulator is complete
  const float sc = p.scale;
  const size_t n8 = static_cast<size_t>(p.B) * p.Hq * p.L * E / 8;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(p.dq_acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(p.dq_acc)[2 * i + 1];
    uint4 w;
    w.x = pack_bf16x2(a.x * sc, a.y * sc);
    w.y = pack_bf16x2(a.z * sc, a.w * sc);
    w.z = pack_bf16x2(b.x * sc, b.y * sc);
    w.w = pack_bf16x2(b.z * sc, b.w * sc);
    reinterpret_cast<uint4*>(p.dq)[i] = w;
  }
}

template <int E_, bool DROP, bool MSTAGE>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmM, const __grid_constant__ CUtensorMap tmdK,
                  const __grid_constant__ CUtensorMap tmdV, TcBwdArgs a) {
  using C = BwdCfg<E_, MSTAGE>;
  constexpr int kNSQ = C::NSQ;
  constexpr int E = C::E, Ev = C::Ev, ECH = C::ECH;
  constexpr int kKBytes = C::kKBytes, kQTile = C::kQTile, kStage = C::kStage;
  constexpr int kOffK = C::kOffK, kOffV = C::kOffV, kOffStage = C::kOffStage, kOffDS = C::kOffDS,
                kOffBar = C::kOffBar;
  const BwdParams& p = a.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* kv_full = bar;                 // 1
  uint64_t* q_full = bar + 1;              // kNSQ
  uint64_t* q_empty = q_full + kNSQ;       // kNSQ
  uint64_t* s_full = q_empty + kNSQ;       // 2: S^T(i) complete in buffer i & 1
  uint64_t* dp_full = s_full + 2;          // 1
  uint64_t* dp_free = dp_full + 1;         // 1
  uint64_t* pt_full = dp_free + 1;         // 2: P^T(i) in buffer i & 1 (one arrival per elementwise warp)
  uint64_t* pt_free = pt_full + 2;         // 2: dV(i) complete (buffer i & 1 free for S^T(i + 2))
  uint64_t* ds_full = pt_free + 2;         // 2: dS^T(i) in shared-memory buffer i % NDS
  uint64_t* ds_free = ds_full + 2;         // 2: dK(i) and dQ^T(i) complete (that buffer free)
  uint64_t* dq_full = ds_free + 2;         // 1
  uint64_t* dq_free = dq_full + 1;         // 1
  uint64_t* kdv_done = dq_free + 1;        // 1
  uint64_t* m_full = kdv_done + 1;         // 1: staged mask tile landed
  uint64_t* m_empty = m_full + 1;          // 1: mask tile read by the elementwise warps
  uint64_t* mma_drain = m_empty + 1;       // 2: every MMA of the score / gradient issuer complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Right-bounded (causal-like) bands: grid (KV groups, key tiles), so the
  // heaviest key tiles of every group start first.  Otherwise every CTA has
  // about the same work and the grid is (key tiles, KV groups): the key-tile
  // CTAs of one group run side by side and share its Q/dO tiles and dQ
  // accumulator rows in L2.
  const bool right_bounded = p.band.right >= 0;
  const int bkv = right_bounded ? blockIdx.x : blockIdx.y, b = bkv / p.Hkv, hkv = bkv - b * p.Hkv;
  const int k0 = (right_bounded ? blockIdx.y : blockIdx.x) * BKV;
  // query tiles that see a key of this tile: rows first_row_reaching(k0) ..
  // last_row_starting_by(last key before Sb) (padding and band)
  const BandRows br = band_rows(p.band, b, p.L, p.S);
  const int klast = min(k0 + BKV, br.Sb) - 1;
  const int i_first = klast >= k0 ? br.first_row_reaching(k0) : 1;
  const int i_last = klast >= k0 ? br.last_row_starting_by(klast) : 0;
  const int qt_lo = i_first / BQ, qt_hi = i_last >= i_first ? i_last / BQ : qt_lo - 1;
  const int per_head = qt_hi - qt_lo + 1;
  const int n = p.G * per_head;                          // iterations
  // Iteration i -> (query tile, head): tiles from the last down to the diagonal,
  // the group's heads innermost.  Every CTA of a KV group starts at the same
  // (last) tile and walks down in step, so the CTAs running at the same time
  // read the same Q/dO tiles and mostly hit in L2.
  struct TileIter {   // (query tile, head) of iteration i, advanced without divisions
    int qt, g, G;
    __device__ void next() {
      if (++g == G) {
        g = 0;
        --qt;
      }
    }
  };
  const TileIter tile0{qt_hi, 0, p.G};

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < kNSQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&pt_full[t], 8);   // one arrival per elementwise warp
      mbar_init(&pt_free[t], 1);
      mbar_init(&ds_full[t], 8);
      mbar_init(&ds_free[t], 1);
    }
    mbar_init(dp_full, 1);
    mbar_init(dp_free, 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);    // one arrival per drain warp
    mbar_init(kdv_done, 1);
    mbar_init(m_full, 1);
    mbar_init(m_empty, 8);
    mbar_init(&mma_drain[0], 1);
    mbar_init(&mma_drain[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Launched behind the row statistics (programmatic dependent launch), so this
  // set-up overlaps their tail: every role reads what that grid writes, so all
  // wait for it here; then the conversion grid may launch.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp >= 12) {
    regs_dec<kRegsOther>();
    if (warp == 12 && lane == 0 && n > 0) {
      // ---------------------------------------------------------- TMA producer
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmdO);
      if (MSTAGE) prefetch_tmap(&tmM);
      mbar_arrive_expect_tx(kv_full, 2 * kKBytes);
      for (int c = 0; c < ECH; ++c) {
        tma_load_3d(smem + kOffK + c * BKV * 128, &tmK, kv_full, c * 64, k0, bkv);
        tma_load_3d(smem + kOffV + c * BKV * 128, &tmV, kv_full, c * 64, k0, bkv);
      }
      TileIter ti = tile0;
      for (int i = 0; i < n; ++i, ti.next()) {
        const int s = i % kNSQ;
        const int qt = ti.qt, g = ti.g;
        const int bh = b * p.Hq + hkv * p.G + g;
        mbar_wait(&q_empty[s], ((i / kNSQ) & 1) ^ 1, abort_flag, p.status, status_code(0x31));
        uint8_t* st = smem + kOffStage + s * kStage;
        mbar_arrive_expect_tx(&q_full[s], 2 * kQTile + BQ * 8);
        for (int c = 0; c < ECH; ++c) {
          tma_load_3d(st + c * BQ * 128, &tmQ, &q_full[s], c * 64, qt * BQ, bh);
          tma_load_3d(st + kQTile + c * BQ * 128, &tmdO, &q_full[s], c * 64, qt * BQ, bh);
        }
        bulk_load(smem + C::kOffRS + s * (BQ * 8), a.rowstats + (static_cast<size_t>(bh) * a.Lpad + qt * BQ) * 2, BQ * 8,
                  &q_full[s]);
        if (MSTAGE) {   // mask rows qt*BQ.., keys k0.. of head (b, h); zero-filled past L and S
          mbar_wait(m_empty, (i & 1) ^ 1, abort_flag, p.status, status_code(0x3e));
          mbar_arrive_expect_tx(m_full, C::kMaskBytes);
          tma_load_3d(smem + C::kOffMask, &tmM, m_full, k0, qt * BQ,
                      b * a.mslice_b + (hkv * p.G + g) * a.mslice_h);
        }
      }
      if (*abort_flag) {   // a wait gave up: let this thread's copies land before the CTA exits
        mbar_drain(kv_full, 0);
        mbar_drain_ring(q_full, kNSQ, n);
        if (MSTAGE) mbar_drain(m_full, static_cast<uint32_t>((n - 1) & 1));
      }
    } else if ((warp == 13 || warp == 14) && lane == 0 && n > 0) {
      // ---------------------------------------------------------- MMA issuers
      constexpr uint32_t id_s = idesc_bf16(BKV, BQ, 0, 0);     // S^T, dP^T: K-major x K-major
      constexpr uint32_t id_kv = idesc_bf16(BKV, E, 0, 1);     // dV, dK: TMEM (K-major) x MN-major
      constexpr uint32_t id_q = idesc_bf16(128, BQ, 1, 1);     // dQ^T: MN-major x MN-major (M = 128 >= E)
      // Operand descriptors, built once; a K-step or a stage moves only the start address.
      const uint32_t stage0 = smem_u32(smem + kOffStage);
      const SmemDesc dK_k = smem_desc(smem_u32(smem + kOffK), 16, 1024);            // K [keys x dims], K-major
      const SmemDesc dV_k = smem_desc(smem_u32(smem + kOffV), 16, 1024);            // V [keys x dims], K-major
      const SmemDesc dK_mn = smem_desc(smem_u32(smem + kOffK), BKV * 128, 1024);    // K^T as MN-major A
      const SmemDesc dDS_mn = smem_desc(smem_u32(smem + kOffDS), BQ * 128, 1024);   // dS^T as MN-major B
      const SmemDesc dDS_k = smem_desc(smem_u32(smem + kOffDS), 16, 1024);          // dS^T as K-major A
      const SmemDesc dQ_k = smem_desc(stage0, 16, 1024);                           // Q/dO stage 0, K-major
      const SmemDesc dQ_mn = smem_desc(stage0, BQ * 128, 1024);                    // Q/dO stage 0, MN-major
      mbar_wait(kv_full, 0, abort_flag, p.status, status_code(0x32));
      auto issue_sdp = [&](int i) {
        const int s = i % kNSQ;
        mbar_wait(&q_full[s], (i / kNSQ) & 1, abort_flag, p.status, status_code(0x33));
        tc_fence_after();
        const SmemDesc q_k = dQ_k + s * kStage, do_k = q_k + kQTile;
        const int sb = i & 1;
        if (i >= 2) {   // dV(i-2) has read P^T(i-2) from this buffer
          mbar_wait(&pt_free[sb], ((i >> 1) - 1) & 1, abort_flag, p.status, status_code(0x34));
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < E / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * (BKV * 128) + (kk & 3) * 32, kb = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
          umma_ss(tmem + kColS + sb * 64, dK_k + ka, q_k + kb, id_s, kk > 0);
        }
        umma_commit(&s_full[sb]);
        if (i > 0) {
          mbar_wait(dp_free, (i - 1) & 1, abort_flag, p.status, status_code(0x35));
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < Ev / 16; ++kk) {
          const uint32_t ka = (kk >> 2) * (BKV * 128) + (kk & 3) * 32, kb = (kk >> 2) * (BQ * 128) + (kk & 3) * 32;
          umma_ss(tmem + kColDP, dV_k + ka, do_k + kb, id_s, kk > 0);
        }
        umma_commit(dp_full);
      };
      if (warp == 14) {
        for (int i = 0; i < n; ++i) issue_sdp(i);   // score MMAs
        // every MMA this thread issued is complete before the CTA releases TMEM (after a
        // wait that gave up, some may still be queued; the drain is bounded like every wait)
        umma_commit(&mma_drain[0]);
        mbar_drain(&mma_drain[0], 0);
      } else {
        for (int i = 0; i < n; ++i) {               // gradient MMAs
          const int s = i % kNSQ;
          const SmemDesc q_mn = dQ_mn + s * kStage, do_mn = q_mn + kQTile;
          const int sb = i & 1, db = i % C::NDS;
          const SmemDesc ds_k = dDS_k + db * (BKV * 128), ds_mn = dDS_mn + db * (BKV * 128);
          // dV += P^T dO as soon as P^T is in TMEM (the elementwise warps are still on dS)
          mbar_wait(&pt_full[sb], (i >> 1) & 1, abort_flag, p.status, status_code(0x36));
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)     // K = queries; 16 queries = 8 TMEM columns
            umma_ts(tmem + kColDV, tmem + p_col(sb, kk), do_mn + kk * 16 * 128, id_kv, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&pt_free[sb]);
          // dK += dS^T Q, dS^T from shared memory (K-major: 128 key rows of 64 queries)
          mbar_wait(&ds_full[db], (i / C::NDS) & 1, abort_flag, p.status, status_code(0x40));
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)
            umma_ss(tmem + kColDK, ds_k + kk * 32, q_mn + kk * 16 * 128, id_kv, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&q_empty[s]);   // Q and dO of the stage are read
          if (i > 0) {
            mbar_wait(dq_free, (i - 1) & 1, abort_flag, p.status, status_code(0x37));
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)    // dQ^T = K^T dS^T   (K = keys)
            umma_ss(tmem + kColDQ, dK_mn + kk * 16 * 128, ds_mn + kk * 16 * 128, id_q, kk > 0);
          umma_commit(&ds_free[db]);
          umma_commit(dq_full);
        }
        umma_commit(kdv_done);
        umma_commit(&mma_drain[1]);   // as for the score issuer
        mbar_drain(&mma_drain[1], 0);
      }
    }
  } else if (warp < 8) {
    regs_inc<kRegsElem>();
    // ------------------------------------------------------------ elementwise warps (thread = key)
    const int wq = warp & 3, hf = warp >> 2;   // TMEM lane quarter, query-column half
    const int r = wq * 32 + lane;
    const int key = k0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    uint8_t* dsrow0 = smem + kOffDS + r * 128;
    const float sc = p.scale_log2;
    // With the staged mask, iteration i's dS^T stores are fenced and handed to the
    // gradient issuer only after iteration i + 1 has read its scores, so the fence finds
    // the stores done instead of waiting for them (masked backward 0.791 -> 0.772 ms; the
    // unmasked ones, whose tensor pipe needs dK and dQ^T promptly, measured slower).
    constexpr bool kDeferDS = MSTAGE;
    int pend = -1;   // iteration whose dS^T stores are not yet fenced and handed over
    auto hand_over = [&]() {
      fence_proxy_async_smem();   // the dS^T stores (generic proxy), then the MMAs (async proxy) read them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (DROP) mbar_arrive(&pt_full[pend & 1]);
        mbar_arrive(&ds_full[pend % C::NDS]);
      }
      pend = -1;
    };
    TileIter ti = tile0;
    for (int i = 0; i < n; ++i, ti.next()) {
      const int s = i % kNSQ;
      const int qt = ti.qt, g = ti.g;
      const int h = hkv * p.G + g;
      const int q0 = qt * BQ;
      const float* rs = reinterpret_cast<const float*>(smem + C::kOffRS + s * (BQ * 8));
      const int qc = q0 + hf * kHalf;          // first query of this warp's columns
      mbar_wait(&q_full[s], (i / kNSQ) & 1, abort_flag, p.status, status_code(0x38));
      // this warp's 32 values -lse*log2e (plus mask*log2e for its key), read before
      // the scores arrive so the loads' latency overlaps the wait
      float nl[kHalf];
#pragma unroll
      for (int c = 0; c < kHalf / 4; ++c) {
        const float4 v4 = reinterpret_cast<const float4*>(rs + hf * kHalf)[c];
        nl[4 * c] = v4.x, nl[4 * c + 1] = v4.y, nl[4 * c + 2] = v4.z, nl[4 * c + 3] = v4.w;
      }
      if (MSTAGE) {   // the staged tile: row = query, 128 keys per row; lanes read consecutive words
        mbar_wait(m_full, i & 1, abort_flag, p.status, status_code(0x3f));
        const float* mt = reinterpret_cast<const float*>(smem + C::kOffMask) + hf * kHalf * BKV + r;
#pragma unroll
        for (int j = 0; j < kHalf; ++j) nl[j] = fmaf(mt[j * BKV], kLog2e, nl[j]);
        // the next fill is a TMA (async-proxy) write: order this lane's reads before it
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(m_empty);
      } else if (p.mask) {
        if (key < p.S) {   // lanes are consecutive keys: each load instruction reads 128 contiguous bytes
          const float* mcol = p.mask + b * p.mask_sb + h * p.mask_sh + static_cast<size_t>(qc) * p.S + key;
#pragma unroll
          for (int j = 0; j < kHalf; ++j)
            if (qc + j < p.L) nl[j] = fmaf(__ldg(mcol + static_cast<size_t>(j) * p.S), kLog2e, nl[j]);
        }
      }
      // dropout: keep bits of this lane's key for the warp's 32 queries (bit jj = query qc + jj).
      // Lane l draws the 32 keys kw..kw+31 of query qc + l (four Philox blocks, the forward's
      // layout), and 32 ballots transpose the bits so that lane j gets key kw + j's column.
      uint32_t col = 0xFFFFFFFFu;
      if (DROP) {
        const unsigned kw = static_cast<unsigned>(k0 + wq * 32), bh = static_cast<unsigned>(b * p.Hq + h);
        uint32_t word = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t k8[4];
          dropout_keep8(p.drop, (kw >> 3) + g, static_cast<unsigned>(qc + lane), bh, k8);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            word |= (k8[c] & 1u) << (8 * g + 2 * c) | ((k8[c] >> 16) & 1u) << (8 * g + 2 * c + 1);
        }
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const uint32_t bal = __ballot_sync(0xffffffffu, (word >> t) & 1u);
          if (t == lane) col = bal;
        }
      }
      const int sb = i & 1, db = i % C::NDS;
      mbar_wait(&s_full[sb], (i >> 1) & 1, abort_flag, p.status, status_code(0x39));
      tc_fence_after();
      float x[kHalf];
      {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColS + sb * 64 + hf * kHalf, v);
#pragma unroll
        for (int j = 0; j < kHalf; ++j) x[j] = __uint_as_float(v[j]);
      }
      if (kDeferDS && pend >= 0) hand_over();
      // t = s alpha log2e + mask log2e - lse log2e
#pragma unroll
      for (int j = 0; j < kHalf; j += 2) fma2(x[j], x[j + 1], x[j], x[j + 1], sc, sc, nl[j], nl[j + 1]);
      // padding and band: the per-element test only where this warp's 32 queries do
      // not all see every key of the tile (a warp-uniform test)
      if (!(qc + kHalf - 1 < br.Lb && br.lo(qc + kHalf - 1) <= k0 && br.hi(qc) >= k0 + BKV - 1)) {
        // query qc + j sees this lane's key exactly for j in [jlo, jhi]:
        // hi(qc + j) >= key, lo(qc + j) <= key and qc + j < Lb, solved for j
        int jlo = 0, jhi = key < br.Sb ? br.Lb - 1 - qc : -1;
        if (br.right >= 0) jlo = key - qc - br.off - br.right;
        if (br.left > 0) jhi = min(jhi, key - qc - br.off + br.left - 1);
#pragma unroll
        for (int j = 0; j < kHalf; ++j)
          if (j < jlo || j > jhi) x[j] = kNegInf;
      }
#pragma unroll
      for (int j = 0; j < kHalf; ++j) x[j] = ex2(x[j]);     // P^T
      // P^T to TMEM now, so dV(i) runs while dS is computed.  (With dropout, P^T and dS^T
      // go together after dS: the early hand-off measured slower there, 1.14 vs 1.07 ms.)
      if (!DROP) {
        uint32_t pp[kHalf / 2];
#pragma unroll
        for (int c = 0; c < kHalf / 2; ++c) pp[c] = pack_bf16x2(x[2 * c], x[2 * c + 1]);
        // over the scores this warp read (its own columns of the buffer)
        tmem_st16(tmem + lane_off + kColS + sb * 64 + hf * kHalf, pp);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pt_full[sb]);
      }
      float nd[kHalf];   // -D of this warp's 32 queries
#pragma unroll
      for (int c = 0; c < kHalf / 4; ++c) {
        const float4 v4 = reinterpret_cast<const float4*>(rs + BQ + hf * kHalf)[c];
        nd[4 * c] = v4.x, nd[4 * c + 1] = v4.y, nd[4 * c + 2] = v4.z, nd[4 * c + 3] = v4.w;
      }
      mbar_wait(dp_full, i & 1, abort_flag, p.status, status_code(0x3a));
      tc_fence_after();
      float d[kHalf];
      {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColDP + hf * kHalf, v);
#pragma unroll
        for (int j = 0; j < kHalf; ++j) d[j] = __uint_as_float(v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dp_free);
      uint32_t pd[kHalf / 2];
      uint32_t pp[DROP ? kHalf / 2 : 1];
      if (DROP) {
        // dropout: dS^T = P^T (dP^T o m - D), dV takes (P o m)^T, m = keep / (1 - p)
#pragma unroll
        for (int j = 0; j < kHalf; ++j) {
          const float mj = ((col >> j) & 1u) ? p.drop.scale : 0.f;
          const float xm = x[j] * mj;
          d[j] = x[j] * fmaf(d[j], mj, nd[j]);
          x[j] = xm;
        }
#pragma unroll
        for (int c = 0; c < kHalf / 2; ++c) pp[c] = pack_bf16x2(x[2 * c], x[2 * c + 1]);
      } else {
#pragma unroll
        for (int j = 0; j < kHalf; j += 2) {                // dS^T = P^T (dP^T - D)
          float t0, t1;
          add2(t0, t1, d[j], d[j + 1], nd[j], nd[j + 1]);
          mul2(d[j], d[j + 1], x[j], x[j + 1], t0, t1);
        }
      }
#pragma unroll
      for (int c = 0; c < kHalf / 2; ++c) pd[c] = pack_bf16x2(d[2 * c], d[2 * c + 1]);
      if (i >= C::NDS) {   // dK and dQ^T of iteration i - NDS have read this dS^T buffer
        mbar_wait(&ds_free[db], ((i / C::NDS) - 1) & 1, abort_flag, p.status, status_code(0x41));
        tc_fence_after();
      }
      if constexpr (DROP) {   // (P o m)^T over this warp's scores, as above
        tmem_st16(tmem + lane_off + kColS + sb * 64 + hf * kHalf, pp);
        tmem_wait_st();
      }
      uint8_t* dsrow = dsrow0 + db * (BKV * 128);
#pragma unroll
      for (int c = 0; c < kHalf / 8; ++c) {
        const int chunk = hf * (kHalf / 8) + c;
        const uint4 u = make_uint4(pd[4 * c], pd[4 * c + 1], pd[4 * c + 2], pd[4 * c + 3]);
        *reinterpret_cast<uint4*>(dsrow + ((chunk ^ (r & 7)) << 4)) = u;
      }
      pend = i;
      if (!kDeferDS) hand_over();
    }
    if (pend >= 0) hand_over();
    // ---------------------------------------------------------- dK, dV epilogue
    // Warps hf = 0 take dK and warps hf = 1 dV, each its 32 keys: scaled, packed to bf16
    // and written as 128-byte-swizzled [128 keys x 64 dims] blocks into the query-tile
    // stages (idle once the last MMA is complete), which one thread then stores with TMA
    // (rows past S are not written).  Stored row by row from registers, each warp
    // instruction wrote 16 bytes into 32 different lines and the epilogue took about 4 us.
    if (n > 0) {
      mbar_wait(kdv_done, 0, abort_flag, p.status, status_code(0x3c));
      tc_fence_after();
    }
    {
      const uint32_t col = hf == 0 ? kColDK : kColDV;
      const float sc2 = hf == 0 ? p.scale : 1.f;
      uint8_t* blk = smem + kOffStage + hf * kKBytes;   // ECH blocks of [128 keys x 64 dims]
#pragma unroll
      for (int c = 0; c < E / 32; ++c) {
        uint32_t v[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_off + col + c * 32, v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(v[u * 8 + 0]) * sc2, __uint_as_float(v[u * 8 + 1]) * sc2);
          w.y = pack_bf16x2(__uint_as_float(v[u * 8 + 2]) * sc2, __uint_as_float(v[u * 8 + 3]) * sc2);
          w.z = pack_bf16x2(__uint_as_float(v[u * 8 + 4]) * sc2, __uint_as_float(v[u * 8 + 5]) * sc2);
          w.w = pack_bf16x2(__uint_as_float(v[u * 8 + 6]) * sc2, __uint_as_float(v[u * 8 + 7]) * sc2);
          const int chunk = (c & 1) * 4 + u;   // 16-byte chunk of this key's 128-byte row in block c / 2
          *reinterpret_cast<uint4*>(blk + (c >> 1) * (BKV * 128) + r * 128 + ((chunk ^ (r & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_smem();   // generic writes, then the TMA (async proxy) reads them
      named_bar_sync(2, 256);     // the eight elementwise warps
      if (warp == 0 && lane == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int cb = 0; cb < ECH; ++cb)
            tma_store_3d(t == 0 ? &tmdK : &tmdV, smem + kOffStage + t * kKBytes + cb * (BKV * 128), cb * 64, k0,
                         bkv);
        bulk_commit_and_wait_read();   // the stages stay in use until the TMA has read them
      }
    }
  } else if (warp < 12) {
    regs_inc<kRegsDrain>();
    // ------------------------------------------------------------ dQ drain (thread = head dim)
    const int e = (warp - 8) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp - 8) * 32) << 16;
    TileIter ti = tile0;
    for (int i = 0; i < n; ++i, ti.next()) {
      const int qt = ti.qt, g = ti.g;
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
      // dQ rows straight from registers: for each query, the 32 lanes of a warp add 32
      // consecutive floats (one 128-byte line) of the fp32 accumulator in L2
      if (e < E) {
        float* dst = p.dq_acc + (static_cast<size_t>(bh) * p.L + q0) * E + e;
        const int nq = min(BQ, p.L - q0);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < nq) red_add_f32(dst + static_cast<size_t>(j) * E, __uint_as_float(v0[j]));
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (32 + j < nq) red_add_f32(dst + static_cast<size_t>(32 + j) * E, __uint_as_float(v1[j]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int E, bool DROP, bool MSTAGE>
cudaError_t run_bwd(const BwdParams& p, cudaStream_t st) {
  using C = BwdCfg<E, MSTAGE>;
  TcBwdArgs a;
  a.p = p;
  a.Lpad = (p.L + BQ - 1) / BQ * BQ;
  a.rowstats = p.D;
  const long long LS = static_cast<long long>(p.L) * p.S;
  a.mslice_b = static_cast<int>(p.mask_sb / LS);
  a.mslice_h = static_cast<int>(p.mask_sh / LS);
  auto kern = bwd_tc_kernel<E, DROP, MSTAGE>;
  // The register split in the main kernel assumes the launch reserves exactly kRegsLaunch per thread.
  cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), C::kSmemBytes, kRegsLaunch);
  if (e != cudaSuccess) return e;
  const long long srows = static_cast<long long>(p.B) * p.Hq * a.Lpad;
  bwd_rowstats_kernel<E><<<static_cast<unsigned>((srows + 7) / 8), 256, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap tmK, tmV, tmQ, tmdO, tmdK, tmdV;
  if (!encode_tmap_bf16_3d(&tmdK, p.dk, E, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BKV) ||
      !encode_tmap_bf16_3d(&tmdV, p.dv, E, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BKV) ||
      !encode_tmap_bf16_3d(&tmK, p.k, E, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BKV) ||
      !encode_tmap_bf16_3d(&tmV, p.v, E, p.S, static_cast<uint64_t>(p.B) * p.Hkv, 64, BKV) ||
      !encode_tmap_bf16_3d(&tmQ, p.q, E, p.L, static_cast<uint64_t>(p.B) * p.Hq, 64, BQ) ||
      !encode_tmap_bf16_3d(&tmdO, p.dO, E, p.L, static_cast<uint64_t>(p.B) * p.Hq, 64, BQ))
    return cudaErrorInvalidValue;
  alignas(64) CUtensorMap tmM = tmK;   // unused unless the mask is staged
  if (MSTAGE) {
    // the mask's distinct [L, S] slices: B x mask heads, or the heads alone, or one
    const long long slices = a.mslice_b ? static_cast<long long>(p.B) * a.mslice_b : (a.mslice_h ? p.Hq : 1);
    if (!encode_tmap_f32_3d(&tmM, p.mask, p.S, p.L, static_cast<uint64_t>(slices), BKV, BQ, false))
      return cudaErrorInvalidValue;
  }
  const unsigned groups = static_cast<unsigned>(p.B * p.Hkv), ktiles = static_cast<unsigned>((p.S + BKV - 1) / BKV);
  const dim3 grid = p.band.right >= 0 ? dim3(groups, ktiles) : dim3(ktiles, groups);
  // programmatic dependent launches: each grid may start while the previous one
  // finishes and waits for it (griddepcontrol.wait) before reading its results
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, kern, tmK, tmV, tmQ, tmdO, tmM, tmdK, tmdV, a)) != cudaSuccess) return e;
  const size_t n8 = static_cast<size_t>(p.B) * p.Hq * p.L * E / 8;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n8 + 255) / 256, 152 * 16));
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(blocks);
  cfg2.blockDim = dim3(256);
  cfg2.stream = st;
  cfg2.attrs = &attr;
  cfg2.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg2, bwd_dq_convert_kernel<E>, p);
}

template <bool DROP, bool MSTAGE>
cudaError_t run_widths(const BwdParams& p, cudaStream_t st) {
  return p.E == 64 ? run_bwd<64, DROP, MSTAGE>(p, st) : run_bwd<128, DROP, MSTAGE>(p, st);
}

}  // namespace

bool bwd_tc_supported(int E_, int Ev_) { return E_ == Ev_ && (E_ == 64 || E_ == 128); }

int bwd_tc_row_pad() { return BQ; }

cudaError_t launch_bwd_tc(const BwdParams& p, cudaStream_t st) {
  // An additive mask (16-byte aligned base, checked at the boundary) is staged
  // through shared memory by TMA when its rows are 16-byte multiples (S a
  // multiple of 4); otherwise the elementwise warps read it directly.
  const bool mstage = p.mask && (p.S & 3) == 0;
  if (p.drop.active) return mstage ? run_widths<true, true>(p, st) : run_widths<true, false>(p, st);
  return mstage ? run_widths<false, true>(p, st) : run_widths<false, false>(p, st);
}

}  // namespace sdpa_impl
