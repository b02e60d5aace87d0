// common.cuh - parameter blocks and small device helpers shared by the kernels.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sdpa_impl {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status codes written by bounded waits: low byte = sdpa_status value
// (4 = timeout), next byte = which wait gave up (for diagnosis).
constexpr unsigned kStatusTimeout = 4u;
__host__ __device__ constexpr unsigned status_code(unsigned where) { return kStatusTimeout | (where << 8); }

// Padding and diagonal band of a call ("Attention" (cuDNN): Configurable
// Options, Padding mask and Diagonal masking options).  For batch b the actual
// lengths are Lb = seq_len_q[b] and Sb = seq_len_kv[b] (clamped to [0, L] and
// [0, S]; L and S without length arrays).  Row i < Lb sees the keys lo(i)..hi(i):
//   diagonal d(i) = i (top-left) or i + Sb - Lb (bottom-right),
//   hi(i) = min(Sb - 1, d(i) + right) with a right bound (0 = causal), else Sb - 1,
//   lo(i) = max(0, d(i) - left + 1) with a left bound, else 0;
// rows i >= Lb see nothing.  The host clamps both bounds to L + S, so the
// arithmetic below stays within int.
struct Band {
  const int* seqlen_q;   // device [B] or nullptr
  const int* seqlen_kv;  // device [B] or nullptr
  int bottom_right;      // 1: the diagonal is aligned at the bottom-right
  int right;             // < 0: no right bound
  int left;              // <= 0: no left bound
  __host__ __device__ bool restricts() const { return seqlen_q || seqlen_kv || right >= 0 || left > 0; }
};

// A Band resolved for one batch.  lo and hi are non-decreasing in i.
struct BandRows {
  int Lb, Sb, off, right, left;
  __device__ __forceinline__ int hi(int i) const { return right >= 0 ? min(Sb - 1, i + off + right) : Sb - 1; }
  __device__ __forceinline__ int lo(int i) const { return left > 0 ? max(0, i + off - left + 1) : 0; }
  __device__ __forceinline__ bool visible(int i, int j) const { return i < Lb && j >= lo(i) && j <= hi(i); }
  // first row whose range reaches key j (hi(i) >= j), for j < Sb
  __device__ __forceinline__ int first_row_reaching(int j) const { return right >= 0 ? max(0, j - off - right) : 0; }
  // last row whose range starts at or before key j (lo(i) <= j), capped at Lb - 1
  __device__ __forceinline__ int last_row_starting_by(int j) const {
    return left > 0 ? min(Lb - 1, j - off + left - 1) : Lb - 1;
  }
};

__device__ __forceinline__ BandRows band_rows(const Band& bd, int b, int L, int S) {
  BandRows r;
  r.Lb = bd.seqlen_q ? min(max(__ldg(bd.seqlen_q + b), 0), L) : L;
  r.Sb = bd.seqlen_kv ? min(max(__ldg(bd.seqlen_kv + b), 0), S) : S;
  r.off = bd.bottom_right ? r.Sb - r.Lb : 0;
  r.right = bd.right;
  r.left = bd.left;
  return r;
}

// Attention dropout ("Scaled dot-product attention (forward and backward)",
// section 2.5: one uniform per weight, keep where u >= p, kept weights scaled by
// 1/(1-p), the backward replaying the mask; "Attention" (cuDNN), Philox RNG
// dropout with a seed and an offset).  Weight (b, h, i, j) takes its uniform from
// Philox4x32-10 with key (seed mod 2^32, seed / 2^32) and counter (j / 8, i,
// b * Hq + h, offset): the four 32-bit words give eight 16-bit uniforms, word
// t / 2, bits 16 * (t % 2) .. for key j = 8 * (j / 8) + t.  keep iff u16 >=
// thr16 = ceil(p * 2^16) (thr16 = 65536 drops everything).
struct DropoutParams {
  int active;            // 0: no dropout
  unsigned thr16;        // 0 .. 65536
  float scale;           // 1 / (1 - p)
  unsigned seed_lo, seed_hi, offset;
};

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC 2011): each round multiplies counter words 0
// and 2 by fixed odd multipliers, mixes the high product halves with words 1 and
// 3 and the key, and advances the key by two Weyl constants.
__device__ __forceinline__ void philox4x32_10(unsigned c0, unsigned c1, unsigned c2, unsigned c3, unsigned k0,
                                              unsigned k1, uint32_t (&w)[4]) {
  constexpr unsigned kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
  constexpr unsigned kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one 32 x 32 -> 64-bit multiply gives both halves of each product
    const unsigned long long p0 = static_cast<unsigned long long>(c0) * kM0;
    const unsigned long long p1 = static_cast<unsigned long long>(c2) * kM1;
    const unsigned hi0 = static_cast<unsigned>(p0 >> 32), lo0 = static_cast<unsigned>(p0);
    const unsigned hi1 = static_cast<unsigned>(p1 >> 32), lo1 = static_cast<unsigned>(p1);
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
    k0 += kW0;
    k1 += kW1;
  }
  w[0] = c0;
  w[1] = c1;
  w[2] = c2;
  w[3] = c3;
}

// keep flags of the 8 keys 8g .. 8g+7 of query i, head bh, as 4 words of two
// 16-bit lanes (0xFFFF = keep): word c covers keys 8g + 2c (low) and 8g + 2c + 1.
__device__ __forceinline__ void dropout_keep8(const DropoutParams& d, unsigned g, unsigned i, unsigned bh,
                                              uint32_t (&keep)[4]) {
  uint32_t w[4];
  philox4x32_10(g, i, bh, d.offset, d.seed_lo, d.seed_hi, w);
  const unsigned thr = d.thr16 > 0xFFFFu ? 0u : d.thr16 * 0x10001u;
#pragma unroll
  for (int c = 0; c < 4; ++c) keep[c] = d.thr16 > 0xFFFFu ? 0u : __vcmpgeu2(w[c], thr);
}

// dropout multiplier m = keep / (1 - p) of one weight (query i, key j, head bh)
__device__ __forceinline__ float dropout_m1(const DropoutParams& d, unsigned i, unsigned j, unsigned bh) {
  uint32_t w[4];
  philox4x32_10(j >> 3, i, bh, d.offset, d.seed_lo, d.seed_hi, w);
  const unsigned t = j & 7u;
  const unsigned u = (w[t >> 1] >> (16 * (t & 1u))) & 0xFFFFu;
  return (d.thr16 <= 0xFFFFu && u >= d.thr16) ? d.scale : 0.f;
}

// Forward problem (prefill and decode).  Strides are in elements.
struct FwdParams {
  const void* q;
  const void* k;
  const void* v;
  const float* mask;     // nullptr or [mask_b, mask_h, L, S]
  void* o;
  float* lse;
  int B, Hq, Hkv, L, S, E, Ev, G;
  long long mask_sb;     // element stride of the mask's batch index (0 when broadcast)
  long long mask_sh;     // element stride of the mask's head index (0 when broadcast)
  float scale;           // alpha
  float scale_log2;      // alpha * log2(e)
  Band band;             // padding and diagonal band (top-left causal = right bound 0)
  DropoutParams drop;
  unsigned* status;
  // tensor-core prefill: nullptr = every CTA walks a fixed list of work units; else a
  // zeroed device counter from which the CTAs take units in turn (uneven work: padding)
  unsigned* sched = nullptr;
};

struct BwdParams {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dO;
  const float* lse;
  const float* mask;
  float* D;              // [B, Hq, L] fp32 workspace
  float* dq_acc;         // [B, Hq, L, E] fp32 workspace (bf16 tensor-core path) or nullptr
  void* dq;
  void* dk;
  void* dv;
  int B, Hq, Hkv, L, S, E, Ev, G;
  long long mask_sb, mask_sh;
  float scale, scale_log2;
  Band band;
  DropoutParams drop;
  unsigned* status;
};

struct DecodeParams {
  FwdParams f;
  float* part_o;         // [B*Hq*L, nsplit, Ev] fp32: normalised partial outputs
  float* part_lse;       // [B*Hq*L, nsplit]     fp32: partial log2-sum-exp (log2 units)
  int nsplit;
  int keys_per_split;    // multiple of the decode stage
  // Paged caches (f.k / f.v are then containers [nblk, Hkv, bs, E|Ev]); page_k == nullptr: dense.
  // Key s of batch b is row s % bs of block page[b * page_stride + s / bs].
  const int* page_k;
  const int* page_v;
  int page_stride;       // entries per table row (>= ceil(S / bs))
  int bs_k, bs_v;        // keys per block, powers of two >= 8
  int lg_k, lg_v;        // log2 of bs_k, bs_v
  int nblk_k, nblk_v;    // blocks in the containers
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Pack two floats into a bf16x2 word (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- host launchers
cudaError_t launch_fwd_simt(const FwdParams& p, int is_bf16, cudaStream_t st);
cudaError_t launch_bwd_simt(const BwdParams& p, int is_bf16, cudaStream_t st);
cudaError_t launch_bwd_preprocess(const BwdParams& p, int is_bf16, cudaStream_t st);
cudaError_t launch_fwd_tc(const FwdParams& p, cudaStream_t st);
cudaError_t launch_bwd_tc(const BwdParams& p, cudaStream_t st);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t st);
bool fwd_tc_supported(int E, int Ev);
bool bwd_tc_supported(int E, int Ev);
int bwd_tc_row_pad();   // query rows of the tensor-core backward's row-statistics padding
bool decode_supported(int E, int Ev);
int decode_rows_per_cta();
int decode_stage_keys();
// Device address and size of the fixed decode scratch on the current device
// (looked up on first use per device, and again when the device's context has
// been replaced, e.g. after cudaDeviceReset).
cudaError_t decode_static_scratch(void** ptr, size_t* bytes);
// Unique id (cuCtxGetId) of the calling thread's current CUDA context, 0 if no
// context is current.  A device symbol's address belongs to one context: after
// cudaDeviceReset the next context loads the module again, possibly elsewhere,
// so cached symbol addresses are keyed on this id.
unsigned long long current_context_id();
// Once per kernel and CUDA context: checks that the kernel is compiled for
// `regs` registers per thread (0: no check; warp-specialised kernels split
// exactly that many with setmaxnreg) and opts it in to `smem_bytes` of dynamic
// shared memory.  cudaFuncGetAttributes and cudaFuncSetAttribute cost
// microseconds of host time each; later launches in the same context skip them.
cudaError_t prepare_kernel(const void* kernel, int smem_bytes, int regs);

// Tensor-map encoder obtained from the driver at run time (no libcuda link).
bool encode_tmap_bf16_3d(void* tmap /* CUtensorMap* */, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint32_t box0, uint32_t box1);
// The same for a dense fp32 [d2][d1][d0] array; d0 * 4 must be a multiple of 16.
// Without swizzle the box's rows (box0 * 4 bytes) land back to back in shared
// memory; with the 128-byte swizzle box0 must be 32 (one 128-byte row) and the
// 16-byte chunk c of row y lands at chunk c ^ (y % 8).
bool encode_tmap_f32_3d(void* tmap /* CUtensorMap* */, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                        uint32_t box0, uint32_t box1, bool swizzle128);
int num_sms();

}  // namespace sdpa_impl
