// attn_simt.cu - CUDA-core (FFMA, fp32 arithmetic) attention kernels.
//
// These serve fp32 inputs (no TF32: fp32 products and fp32 accumulation, as an
// fp32 caller expects) and bf16 widths the tensor-core kernels do not take.
// Forward: one CTA per 16 query rows of one (batch, head), key/value tiles of
// 64 staged in shared memory, online softmax in natural-exp units (course
// chapter "Scaled dot-product attention (forward and backward)", sections 2.1
// and 2.2; running max and sum as in the "online softmax" the chapter points
// to).  Backward (section 2.3): D_i = dO_i . O_i first, then a query-parallel
// kernel for dQ and a key-parallel kernel for dK and dV (summed over the query
// heads of a grouped-query group), both recomputing P = exp(s - lse) tile by
// tile and never storing it.  No atomics: results are deterministic.
#include "common.cuh"

namespace sdpa_impl {

namespace {

constexpr int kRows = 16;   // query rows per forward / dQ CTA (4 per warp)
constexpr int kKT = 64;     // keys per staged tile
constexpr int kKeys = 16;   // keys per dK/dV CTA (4 per warp)
constexpr int kQT = 64;     // query rows per staged tile in the dK/dV kernel
constexpr int kMaxC = 4;    // output columns per lane: 4 * 32 = 128 = max width
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ float neg_inf() { return kNegInf; }

template <typename T>
__global__ void __launch_bounds__(128) fwd_simt_kernel(FwdParams p) {
  extern __shared__ float smem[];
  const int E = p.E, Ev = p.Ev, S = p.S, L = p.L;
  const int KS = E + 1, VS = Ev;
  float* sQ = smem;                     // [kRows][E]
  float* sK = sQ + kRows * E;           // [kKT][E+1]
  float* sV = sK + kKT * KS;            // [kKT][Ev]
  float* sP = sV + kKT * VS;            // [kRows][kKT]
  const int bh = blockIdx.y, b = bh / p.Hq, h = bh % p.Hq, hk = h / p.G;
  const int i0 = blockIdx.x * kRows;
  const T* q = static_cast<const T*>(p.q) + static_cast<size_t>(bh) * L * E;
  const T* k = static_cast<const T*>(p.k) + static_cast<size_t>(b * p.Hkv + hk) * S * E;
  const T* v = static_cast<const T*>(p.v) + static_cast<size_t>(b * p.Hkv + hk) * S * Ev;
  const float* mask = p.mask ? p.mask + b * p.mask_sb + h * p.mask_sh : nullptr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int x = tid; x < kRows * E; x += blockDim.x) {
    const int r = x / E, e = x - r * E, i = i0 + r;
    sQ[x] = (i < L) ? to_f(q[static_cast<size_t>(i) * E + e]) : 0.f;
  }
  float m[4], l[4], acc[4][kMaxC];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    m[rr] = neg_inf();
    l[rr] = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) acc[rr][c] = 0.f;
  }
  // keys any row of this block can see: lo(first row) .. hi(last row before Lb)
  const BandRows br = band_rows(p.band, b, L, S);
  const int ilast = min(i0 + kRows, br.Lb) - 1;
  const int kbeg = ilast >= i0 ? br.lo(i0) / kKT * kKT : 0;
  const int kend = ilast >= i0 ? br.hi(ilast) + 1 : 0;

  for (int j0 = kbeg; j0 < kend; j0 += kKT) {
    __syncthreads();
    for (int x = tid; x < kKT * E; x += blockDim.x) {
      const int jj = x / E, e = x - jj * E, j = j0 + jj;
      sK[jj * KS + e] = (j < S) ? to_f(k[static_cast<size_t>(j) * E + e]) : 0.f;
    }
    for (int x = tid; x < kKT * Ev; x += blockDim.x) {
      const int jj = x / Ev, e = x - jj * Ev, j = j0 + jj;
      sV[jj * VS + e] = (j < S) ? to_f(v[static_cast<size_t>(j) * Ev + e]) : 0.f;
    }
    __syncthreads();
    const int nk = min(kKT, S - j0);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr, i = i0 + r;
      float x[2];
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int jj = lane + 32 * t, j = j0 + jj;
        float s = 0.f;
        for (int e = 0; e < E; ++e) s = fmaf(sQ[r * E + e], sK[jj * KS + e], s);
        s *= p.scale;
        if (j >= S || !br.visible(i, j)) s = neg_inf();
        else if (mask && i < L) s += mask[static_cast<size_t>(i) * S + j];
        x[t] = s;
      }
      const float mnew = fmaxf(m[rr], warp_max(fmaxf(x[0], x[1])));
      const float msafe = (mnew == neg_inf()) ? 0.f : mnew;
      const float corr = expf(m[rr] - msafe);
      const float p0 = expf(x[0] - msafe), p1 = expf(x[1] - msafe);
      l[rr] = l[rr] * corr + warp_sum(p0 + p1);
      m[rr] = mnew;
      float d0 = 1.f, d1 = 1.f;   // dropout keep flags: P o keep feeds P V (the row sum keeps every weight)
      if (p.drop.active) {
        d0 = dropout_m1(p.drop, i, j0 + lane, bh) != 0.f ? 1.f : 0.f;
        d1 = dropout_m1(p.drop, i, j0 + lane + 32, bh) != 0.f ? 1.f : 0.f;
      }
      sP[r * kKT + lane] = p0 * d0;
      sP[r * kKT + lane + 32] = p1 * d1;
#pragma unroll
      for (int c = 0; c < kMaxC; ++c) acc[rr][c] *= corr;
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr;
      for (int jj = 0; jj < nk; ++jj) {
        const float pj = sP[r * kKT + jj];
#pragma unroll
        for (int c = 0; c < kMaxC; ++c) {
          const int col = lane + 32 * c;
          if (col < Ev) acc[rr][c] = fmaf(pj, sV[jj * VS + col], acc[rr][c]);
        }
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int i = i0 + warp * 4 + rr;
    if (i >= L) continue;
    const float inv = (l[rr] > 0.f) ? p.drop.scale / l[rr] : 0.f;   // 1/(1-p) applied once
    T* o = static_cast<T*>(p.o) + (static_cast<size_t>(bh) * L + i) * Ev;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      const int col = lane + 32 * c;
      if (col < Ev) o[col] = from_f<T>(acc[rr][c] * inv);
    }
    if (lane == 0) p.lse[static_cast<size_t>(bh) * L + i] = (l[rr] > 0.f) ? m[rr] + logf(l[rr]) : neg_inf();
  }
}

// D_i = sum_e dO_ie * O_ie (fp32), one warp per row.
template <typename T>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(BwdParams p) {
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.L;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* o = static_cast<const T*>(p.o) + row * p.Ev;
  const T* dO = static_cast<const T*>(p.dO) + row * p.Ev;
  float s = 0.f;
  for (int e = lane; e < p.Ev; e += 32) s = fmaf(to_f(o[e]), to_f(dO[e]), s);
  s = warp_sum(s);
  if (lane == 0) p.D[row] = s;
}

// dQ_i = alpha * sum_j P_ij (dP_ij - D_i) k_j, query-parallel.
template <typename T>
__global__ void __launch_bounds__(128) bwd_dq_simt_kernel(BwdParams p) {
  extern __shared__ float smem[];
  const int E = p.E, Ev = p.Ev, S = p.S, L = p.L;
  const int KS = E + 1, VS = Ev + 1;
  float* sQ = smem;                     // [kRows][E]
  float* sDO = sQ + kRows * E;          // [kRows][Ev]
  float* sK = sDO + kRows * Ev;         // [kKT][E+1]
  float* sV = sK + kKT * KS;            // [kKT][Ev+1]
  float* sP = sV + kKT * VS;            // [kRows][kKT]  (dS values)
  const int bh = blockIdx.y, b = bh / p.Hq, h = bh % p.Hq, hk = h / p.G;
  const int i0 = blockIdx.x * kRows;
  const T* q = static_cast<const T*>(p.q) + static_cast<size_t>(bh) * L * E;
  const T* dO = static_cast<const T*>(p.dO) + static_cast<size_t>(bh) * L * Ev;
  const T* k = static_cast<const T*>(p.k) + static_cast<size_t>(b * p.Hkv + hk) * S * E;
  const T* v = static_cast<const T*>(p.v) + static_cast<size_t>(b * p.Hkv + hk) * S * Ev;
  const float* mask = p.mask ? p.mask + b * p.mask_sb + h * p.mask_sh : nullptr;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int x = tid; x < kRows * E; x += blockDim.x) {
    const int r = x / E, e = x - r * E, i = i0 + r;
    sQ[x] = (i < L) ? to_f(q[static_cast<size_t>(i) * E + e]) : 0.f;
  }
  for (int x = tid; x < kRows * Ev; x += blockDim.x) {
    const int r = x / Ev, e = x - r * Ev, i = i0 + r;
    sDO[x] = (i < L) ? to_f(dO[static_cast<size_t>(i) * Ev + e]) : 0.f;
  }
  float lse[4], Dv[4], acc[4][kMaxC];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int i = i0 + warp * 4 + rr;
    lse[rr] = (i < L) ? p.lse[static_cast<size_t>(bh) * L + i] : neg_inf();
    Dv[rr] = (i < L) ? p.D[static_cast<size_t>(bh) * L + i] : 0.f;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) acc[rr][c] = 0.f;
  }
  const BandRows br = band_rows(p.band, b, L, S);
  const int ilast = min(i0 + kRows, br.Lb) - 1;
  const int kbeg = ilast >= i0 ? br.lo(i0) / kKT * kKT : 0;
  const int kend = ilast >= i0 ? br.hi(ilast) + 1 : 0;
  for (int j0 = kbeg; j0 < kend; j0 += kKT) {
    __syncthreads();
    for (int x = tid; x < kKT * E; x += blockDim.x) {
      const int jj = x / E, e = x - jj * E, j = j0 + jj;
      sK[jj * KS + e] = (j < S) ? to_f(k[static_cast<size_t>(j) * E + e]) : 0.f;
    }
    for (int x = tid; x < kKT * Ev; x += blockDim.x) {
      const int jj = x / Ev, e = x - jj * Ev, j = j0 + jj;
      sV[jj * VS + e] = (j < S) ? to_f(v[static_cast<size_t>(j) * Ev + e]) : 0.f;
    }
    __syncthreads();
    const int nk = min(kKT, S - j0);
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr, i = i0 + r;
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int jj = lane + 32 * t, j = j0 + jj;
        float ds = 0.f;
        if (j < S && br.visible(i, j) && lse[rr] != neg_inf()) {
          float s = 0.f, dp = 0.f;
          for (int e = 0; e < E; ++e) s = fmaf(sQ[r * E + e], sK[jj * KS + e], s);
          for (int e = 0; e < Ev; ++e) dp = fmaf(sDO[r * Ev + e], sV[jj * VS + e], dp);
          s *= p.scale;
          if (mask) s += mask[static_cast<size_t>(i) * S + j];
          const float pij = expf(s - lse[rr]);
          if (p.drop.active) dp *= dropout_m1(p.drop, i, j, bh);   // dP o m
          ds = pij * (dp - Dv[rr]);
        }
        sP[r * kKT + jj] = ds;
      }
    }
    __syncwarp();
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = warp * 4 + rr;
      for (int jj = 0; jj < nk; ++jj) {
        const float d = sP[r * kKT + jj];
#pragma unroll
        for (int c = 0; c < kMaxC; ++c) {
          const int col = lane + 32 * c;
          if (col < E) acc[rr][c] = fmaf(d, sK[jj * KS + col], acc[rr][c]);
        }
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int i = i0 + warp * 4 + rr;
    if (i >= L) continue;
    T* dq = static_cast<T*>(p.dq) + (static_cast<size_t>(bh) * L + i) * E;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      const int col = lane + 32 * c;
      if (col < E) dq[col] = from_f<T>(acc[rr][c] * p.scale);
    }
  }
}

// dV_j = sum_{h in group} sum_i P_ij dO_i ; dK_j = alpha sum_h sum_i dS_ij q_i, key-parallel.
template <typename T>
__global__ void __launch_bounds__(128) bwd_dkdv_simt_kernel(BwdParams p) {
  extern __shared__ float smem[];
  const int E = p.E, Ev = p.Ev, S = p.S, L = p.L;
  const int QS = E + 1, OS = Ev + 1;
  float* sK = smem;                      // [kKeys][E]
  float* sV = sK + kKeys * E;            // [kKeys][Ev]
  float* sQ = sV + kKeys * Ev;           // [kQT][E+1]
  float* sDO = sQ + kQT * QS;            // [kQT][Ev+1]
  float* sL = sDO + kQT * OS;            // [kQT]
  float* sD = sL + kQT;                  // [kQT]
  float* sP = sD + kQT;                  // [kKeys][kQT]
  float* sS = sP + kKeys * kQT;          // [kKeys][kQT]
  const int bk = blockIdx.y, b = bk / p.Hkv, hk = bk % p.Hkv;
  const int j0 = blockIdx.x * kKeys;
  const T* k = static_cast<const T*>(p.k) + static_cast<size_t>(bk) * S * E;
  const T* v = static_cast<const T*>(p.v) + static_cast<size_t>(bk) * S * Ev;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int x = tid; x < kKeys * E; x += blockDim.x) {
    const int r = x / E, e = x - r * E, j = j0 + r;
    sK[x] = (j < S) ? to_f(k[static_cast<size_t>(j) * E + e]) : 0.f;
  }
  for (int x = tid; x < kKeys * Ev; x += blockDim.x) {
    const int r = x / Ev, e = x - r * Ev, j = j0 + r;
    sV[x] = (j < S) ? to_f(v[static_cast<size_t>(j) * Ev + e]) : 0.f;
  }
  float dk[4][kMaxC], dv[4][kMaxC];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr)
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) dk[rr][c] = dv[rr][c] = 0.f;

  // rows that see a key of this block: from the first row reaching j0 to the
  // last row whose range starts by the block's last key (before Sb)
  const BandRows br = band_rows(p.band, b, L, S);
  const int jlast = min(j0 + kKeys, br.Sb) - 1;
  const int ibeg = jlast >= j0 ? br.first_row_reaching(j0) / kQT * kQT : L;
  const int iend = jlast >= j0 ? br.last_row_starting_by(jlast) + 1 : 0;
  for (int g = 0; g < p.G; ++g) {
    const int h = hk * p.G + g, bh = b * p.Hq + h;
    const T* q = static_cast<const T*>(p.q) + static_cast<size_t>(bh) * L * E;
    const T* dO = static_cast<const T*>(p.dO) + static_cast<size_t>(bh) * L * Ev;
    const float* mask = p.mask ? p.mask + b * p.mask_sb + h * p.mask_sh : nullptr;
    for (int it0 = ibeg; it0 < iend; it0 += kQT) {
      __syncthreads();
      for (int x = tid; x < kQT * E; x += blockDim.x) {
        const int r = x / E, e = x - r * E, i = it0 + r;
        sQ[r * QS + e] = (i < L) ? to_f(q[static_cast<size_t>(i) * E + e]) : 0.f;
      }
      for (int x = tid; x < kQT * Ev; x += blockDim.x) {
        const int r = x / Ev, e = x - r * Ev, i = it0 + r;
        sDO[r * OS + e] = (i < L) ? to_f(dO[static_cast<size_t>(i) * Ev + e]) : 0.f;
      }
      for (int r = tid; r < kQT; r += blockDim.x) {
        const int i = it0 + r;
        sL[r] = (i < L) ? p.lse[static_cast<size_t>(bh) * L + i] : neg_inf();
        sD[r] = (i < L) ? p.D[static_cast<size_t>(bh) * L + i] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int kk = warp * 4 + rr, j = j0 + kk;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int r = lane + 32 * t, i = it0 + r;
          float pij = 0.f, ds = 0.f;
          if (j < S && i < L && br.visible(i, j) && sL[r] != neg_inf()) {
            float s = 0.f, dp = 0.f;
            for (int e = 0; e < E; ++e) s = fmaf(sQ[r * QS + e], sK[kk * E + e], s);
            for (int e = 0; e < Ev; ++e) dp = fmaf(sDO[r * OS + e], sV[kk * Ev + e], dp);
            s *= p.scale;
            if (mask) s += mask[static_cast<size_t>(i) * S + j];
            pij = expf(s - sL[r]);
            if (p.drop.active) {   // dV takes P o m, dS takes (dP o m - D)
              const float mij = dropout_m1(p.drop, i, j, b * p.Hq + h);
              dp *= mij;
              ds = pij * (dp - sD[r]);
              pij *= mij;
            } else {
              ds = pij * (dp - sD[r]);
            }
          }
          sP[kk * kQT + r] = pij;
          sS[kk * kQT + r] = ds;
        }
      }
      __syncwarp();
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int kk = warp * 4 + rr;
        for (int r = 0; r < kQT; ++r) {
          const float pij = sP[kk * kQT + r], ds = sS[kk * kQT + r];
#pragma unroll
          for (int c = 0; c < kMaxC; ++c) {
            const int col = lane + 32 * c;
            if (col < Ev) dv[rr][c] = fmaf(pij, sDO[r * OS + col], dv[rr][c]);
            if (col < E) dk[rr][c] = fmaf(ds, sQ[r * QS + col], dk[rr][c]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int j = j0 + warp * 4 + rr;
    if (j >= S) continue;
    T* dkp = static_cast<T*>(p.dk) + (static_cast<size_t>(bk) * S + j) * E;
    T* dvp = static_cast<T*>(p.dv) + (static_cast<size_t>(bk) * S + j) * Ev;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c) {
      const int col = lane + 32 * c;
      if (col < E) dkp[col] = from_f<T>(dk[rr][c] * p.scale);
      if (col < Ev) dvp[col] = from_f<T>(dv[rr][c]);
    }
  }
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

template <typename T>
cudaError_t fwd_simt(const FwdParams& p, cudaStream_t st) {
  const size_t smem = sizeof(float) * (kRows * p.E + kKT * (p.E + 1) + kKT * p.Ev + kRows * kKT);
  cudaError_t e = set_smem(fwd_simt_kernel<T>, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((p.L + kRows - 1) / kRows, p.B * p.Hq);
  fwd_simt_kernel<T><<<grid, 128, smem, st>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t bwd_simt(const BwdParams& p, cudaStream_t st) {
  const size_t smem_dq = sizeof(float) * (kRows * p.E + kRows * p.Ev + kKT * (p.E + 1) + kKT * (p.Ev + 1) +
                                          kRows * kKT);
  cudaError_t e = set_smem(bwd_dq_simt_kernel<T>, smem_dq);
  if (e != cudaSuccess) return e;
  dim3 gq((p.L + kRows - 1) / kRows, p.B * p.Hq);
  bwd_dq_simt_kernel<T><<<gq, 128, smem_dq, st>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t smem_kv = sizeof(float) * (kKeys * p.E + kKeys * p.Ev + kQT * (p.E + 1) + kQT * (p.Ev + 1) +
                                          2 * kQT + 2 * kKeys * kQT);
  if ((e = set_smem(bwd_dkdv_simt_kernel<T>, smem_kv)) != cudaSuccess) return e;
  dim3 gk((p.S + kKeys - 1) / kKeys, p.B * p.Hkv);
  bwd_dkdv_simt_kernel<T><<<gk, 128, smem_kv, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdParams& p, int is_bf16, cudaStream_t st) {
  return is_bf16 ? fwd_simt<__nv_bfloat16>(p, st) : fwd_simt<float>(p, st);
}

cudaError_t launch_bwd_preprocess(const BwdParams& p, int is_bf16, cudaStream_t st) {
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.L;
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  if (is_bf16)
    bwd_preprocess_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(p);
  else
    bwd_preprocess_kernel<float><<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const BwdParams& p, int is_bf16, cudaStream_t st) {
  return is_bf16 ? bwd_simt<__nv_bfloat16>(p, st) : bwd_simt<float>(p, st);
}

}  // namespace sdpa_impl
