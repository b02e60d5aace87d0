// api.cu - the C ABI declared in include/sdpa.h: argument checks, workspace
// sizing, routing to the kernels, tensor-map encoding and the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "sdpa.h"

namespace sdpa_impl {

// Written by kernels whose bounded waits give up (see ptx.cuh); read and cleared
// by sdpa_last_device_status().
__device__ unsigned g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_status_ptr[kMaxDevices] = {};
unsigned long long g_status_ctx[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

// cuCtxGetCurrent / cuCtxGetId through the runtime's driver entry points (no libcuda link).
std::once_flag g_ctx_fn_once;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

}  // namespace

unsigned long long current_context_id() {
  std::call_once(g_ctx_fn_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx || g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

namespace {
std::mutex g_prep_mu;
struct Prepared {
  const void* kernel;
  unsigned long long ctx;
  int smem;
};
Prepared g_prepared[256];
int g_nprepared = 0;
}  // namespace

cudaError_t prepare_kernel(const void* kernel, int smem_bytes, int regs) {
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(g_prep_mu);
  if (ctx != 0)
    for (int i = 0; i < g_nprepared; ++i)
      if (g_prepared[i].kernel == kernel && g_prepared[i].ctx == ctx && g_prepared[i].smem == smem_bytes)
        return cudaSuccess;
  if (regs > 0) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != regs) return cudaErrorInvalidConfiguration;
  }
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  const unsigned long long now = current_context_id();   // the calls above make a context current
  if (now != 0 && g_nprepared < 256) g_prepared[g_nprepared++] = Prepared{kernel, now, smem_bytes};
  return cudaSuccess;
}

namespace {

unsigned* status_ptr() {
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  // cudaGetSymbolAddress makes the runtime's context current if none is, so
  // the id is read after it on a first lookup
  const unsigned long long ctx = current_context_id();
  if (!g_status_ptr[d] || ctx == 0 || ctx != g_status_ctx[d]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[d] = static_cast<unsigned*>(ptr);
    g_status_ctx[d] = current_context_id();
  }
  return g_status_ptr[d];
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Checked {
  int B, Hq, Hkv, L, S, E, Ev, G;
  bool bf16;
  long long mask_sb, mask_sh;
};

// Shape checks shared by every entry point; mirrors the argument checks of the
// "ScaledDotProductAttentionBackward" page (matching batch dims, q/k widths,
// k/v lengths) plus the grouped-query rule Hq % Hkv == 0.
sdpa_status check_shape(const sdpa_shape* s, int enable_gqa, bool has_mask, Checked* c) {
  if (!s) return SDPA_ERR_INVALID_ARG;
  if (s->B <= 0 || s->Hq <= 0 || s->Hkv <= 0 || s->L <= 0 || s->S <= 0 || s->E <= 0 || s->Ev <= 0)
    return SDPA_ERR_INVALID_ARG;
  if (s->dtype != SDPA_F32 && s->dtype != SDPA_BF16) return SDPA_ERR_INVALID_ARG;
  if (s->Hq % s->Hkv != 0) return SDPA_ERR_INVALID_ARG;
  if (s->Hq != s->Hkv && !enable_gqa) return SDPA_ERR_INVALID_ARG;
  if (has_mask) {
    if (!(s->mask_b == 1 || s->mask_b == s->B) || !(s->mask_h == 1 || s->mask_h == s->Hq))
      return SDPA_ERR_INVALID_ARG;
  }
  // sizes the kernels index with 32-bit row counters and grid dimensions; each
  // dimension is bounded before any product of them is formed
  if (s->B > INT_MAX || s->Hq > INT_MAX || s->Hkv > INT_MAX || s->L > INT_MAX / 2 || s->S > INT_MAX / 2)
    return SDPA_ERR_UNSUPPORTED;
  if (s->E > 128 || s->Ev > 128) return SDPA_ERR_UNSUPPORTED;
  if (s->B * s->Hq > INT_MAX || s->B * s->Hkv > 65535 * 64) return SDPA_ERR_UNSUPPORTED;
  // element counts of every tensor and workspace stay below 2^56, so no byte count wraps
  {
    const double kMaxElems = 72057594037927936.0;   // 2^56
    const double rows_q = static_cast<double>(s->B) * static_cast<double>(s->Hq) * static_cast<double>(s->L);
    const double rows_kv = static_cast<double>(s->B) * static_cast<double>(s->Hkv) * static_cast<double>(s->S);
    const double mask_elems =
        has_mask ? static_cast<double>(s->mask_b) * s->mask_h * static_cast<double>(s->L) * static_cast<double>(s->S)
                 : 0.0;
    if (rows_q * 128.0 > kMaxElems || rows_kv * 128.0 > kMaxElems || mask_elems > kMaxElems)
      return SDPA_ERR_UNSUPPORTED;
  }
  if (s->dtype == SDPA_BF16 && (s->E % 8 != 0 || s->Ev % 8 != 0)) return SDPA_ERR_UNSUPPORTED;
  c->B = static_cast<int>(s->B);
  c->Hq = static_cast<int>(s->Hq);
  c->Hkv = static_cast<int>(s->Hkv);
  c->L = static_cast<int>(s->L);
  c->S = static_cast<int>(s->S);
  c->E = static_cast<int>(s->E);
  c->Ev = static_cast<int>(s->Ev);
  c->G = c->Hq / c->Hkv;
  c->bf16 = s->dtype == SDPA_BF16;
  const long long LS = s->L * s->S;
  c->mask_sh = (has_mask && s->mask_h != 1) ? LS : 0;
  c->mask_sb = (has_mask && s->mask_b != 1) ? LS * s->mask_h : 0;
  return SDPA_OK;
}

sdpa_status check_scale(double scale, int E, float* alpha) {
  if (std::isnan(scale)) {
    *alpha = static_cast<float>(1.0 / std::sqrt(static_cast<double>(E)));
    return SDPA_OK;
  }
  if (std::isinf(scale) || scale < 0.0) return SDPA_ERR_INVALID_ARG;
  *alpha = static_cast<float>(scale);
  return SDPA_OK;
}

sdpa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SDPA_OK : SDPA_ERR_CUDA; }

// Failure-path self-test: one thread waits on an mbarrier nothing arrives at; the
// bounded wait gives up after its limit, records a timeout in the status word and
// the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sdpa_ptx::mbar_init(&bar, 1);
    abort_flag = 0;
    sdpa_ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) sdpa_ptx::mbar_wait(&bar, 0, &abort_flag, status, status_code(0x7f));
}

// Tensor-core prefill workspace: the unit counter of padded calls (one word, padded).
constexpr size_t kFwdSchedBytes = 256;

// The band of the plain entry points: no padding, top-left, causal = right bound 0.
Band plain_band(int is_causal) { return Band{nullptr, nullptr, 0, is_causal ? 0 : -1, 0}; }

DropoutParams no_dropout() { return DropoutParams{0, 0u, 1.f, 0u, 0u, 0u}; }

// Dropout of sdpa_options: p in [0, 1) and an offset below 2^32 (INVALID_ARG
// otherwise: the offset fills one 32-bit counter word); p = 0 is no dropout.
sdpa_status dropout_from_options(const sdpa_options* o, DropoutParams* d) {
  *d = no_dropout();
  if (!o) return SDPA_OK;
  const double pr = o->dropout_p;
  if (!(pr >= 0.0 && pr < 1.0)) return SDPA_ERR_INVALID_ARG;
  if (pr == 0.0) return SDPA_OK;
  if (o->dropout_offset > 0xFFFFFFFFull) return SDPA_ERR_INVALID_ARG;
  d->active = 1;
  d->thr16 = static_cast<unsigned>(std::ceil(pr * 65536.0));
  d->scale = static_cast<float>(1.0 / (1.0 - pr));
  d->seed_lo = static_cast<unsigned>(o->dropout_seed & 0xFFFFFFFFull);
  d->seed_hi = static_cast<unsigned>(o->dropout_seed >> 32);
  d->offset = static_cast<unsigned>(o->dropout_offset);
  return SDPA_OK;
}

// Checks sdpa_options and turns them into a Band (NULL options = no padding, no band).
sdpa_status band_from_options(const sdpa_options* o, const Checked& c, Band* band) {
  *band = plain_band(0);
  if (!o) return SDPA_OK;
  if (o->diagonal_alignment != SDPA_TOP_LEFT && o->diagonal_alignment != SDPA_BOTTOM_RIGHT)
    return SDPA_ERR_INVALID_ARG;
  if ((o->seq_len_q && (reinterpret_cast<uintptr_t>(o->seq_len_q) & 3)) ||
      (o->seq_len_kv && (reinterpret_cast<uintptr_t>(o->seq_len_kv) & 3)))
    return SDPA_ERR_INVALID_ARG;
  const long long cap = static_cast<long long>(c.L) + c.S;   // a bound this wide no longer restricts
  band->seqlen_q = o->seq_len_q;
  band->seqlen_kv = o->seq_len_kv;
  band->bottom_right = o->diagonal_alignment == SDPA_BOTTOM_RIGHT ? 1 : 0;
  band->right = o->right_bound < 0 ? -1 : static_cast<int>(std::min<long long>(o->right_bound, cap));
  band->left = o->left_bound <= 0 ? 0 : static_cast<int>(std::min<long long>(o->left_bound, cap));
  return SDPA_OK;
}

void fill_fwd(FwdParams& p, const Checked& c, const void* q, const void* k, const void* v, const float* mask,
              float alpha, const Band& band, void* o, float* lse) {
  p.q = q;
  p.k = k;
  p.v = v;
  p.mask = mask;
  p.o = o;
  p.lse = lse;
  p.B = c.B;
  p.Hq = c.Hq;
  p.Hkv = c.Hkv;
  p.L = c.L;
  p.S = c.S;
  p.E = c.E;
  p.Ev = c.Ev;
  p.G = c.G;
  p.mask_sb = c.mask_sb;
  p.mask_sh = c.mask_sh;
  p.scale = alpha;
  p.scale_log2 = alpha * kLog2e;
  p.band = band;
  p.drop = no_dropout();
  p.status = status_ptr();
}

// Split count: at least two waves of (SMs x 2 resident CTAs) and, among up to
// twice that count, the one whose last wave is fullest.
int auto_splits(const Checked& c) {
  const int stage = decode_stage_keys();
  const long long units =
      static_cast<long long>(c.B) * c.Hkv * ((c.G * c.L + decode_rows_per_cta() - 1) / decode_rows_per_cta());
  const long long slots = static_cast<long long>(num_sms()) * 2;
  const int max_splits = (c.S + stage - 1) / stage;
  int lo = static_cast<int>((2 * slots + units - 1) / units);
  lo = std::max(1, std::min(lo, max_splits));
  int best = lo;
  double best_eff = -1.0;
  for (int n = lo; n <= std::min(2 * lo, max_splits); ++n) {
    const long long ctas = units * n;
    const long long waves = (ctas + slots - 1) / slots;
    const double eff = static_cast<double>(ctas) / static_cast<double>(waves * slots);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = n;
    }
  }
  return best;
}

// Normalises a split count so every split but the last covers a whole number of stages.
void split_layout(const Checked& c, int want, int* nsplit, int* kps) {
  const int stage = decode_stage_keys();
  const int max_splits = (c.S + stage - 1) / stage;
  want = std::max(1, std::min(want, max_splits));
  int per = (c.S + want - 1) / want;
  per = (per + stage - 1) / stage * stage;
  *kps = per;
  *nsplit = (c.S + per - 1) / per;
}

size_t decode_ws(const Checked& c, int nsplit) {
  const size_t rows = static_cast<size_t>(c.B) * c.Hq * c.L;
  return round_up(rows * nsplit * c.Ev * sizeof(float), 256) + round_up(rows * nsplit * sizeof(float), 256);
}

bool routes_to_decode(const Checked& c) { return c.bf16 && c.L == 1 && decode_supported(c.E, c.Ev); }

bool bwd_uses_tc(const Checked& c) { return c.bf16 && bwd_tc_supported(c.E, c.Ev); }

// Tensor-core backward: per-row (-lse*log2e, D) float2 rows padded per head to a
// multiple of the query tile, then the fp32 dQ accumulator.  CUDA-core backward:
// D only.
size_t bwd_stats_bytes(const Checked& c) {
  if (!bwd_uses_tc(c)) return round_up(static_cast<size_t>(c.B) * c.Hq * c.L * sizeof(float), 256);
  const size_t pad = static_cast<size_t>(bwd_tc_row_pad());
  const size_t lpad = (static_cast<size_t>(c.L) + pad - 1) / pad * pad;
  return round_up(static_cast<size_t>(c.B) * c.Hq * lpad * 2 * sizeof(float), 256);
}

size_t bwd_ws(const Checked& c) {
  size_t bytes = bwd_stats_bytes(c);
  if (bwd_uses_tc(c)) bytes += round_up(static_cast<size_t>(c.B) * c.Hq * c.L * c.E * sizeof(float), 256);
  return bytes;
}

sdpa_status run_decode(const Checked& c, const Band& band, const void* q, const void* k, const void* v,
                       const float* mask, float alpha, int num_splits, void* o, float* lse, void* ws,
                       size_t ws_bytes, cudaStream_t st, const sdpa_paged_kv* paged = nullptr) {
  int nsplit, kps;
  split_layout(c, num_splits > 0 ? num_splits : auto_splits(c), &nsplit, &kps);
  if (c.B * c.Hkv * ((c.G * c.L + decode_rows_per_cta() - 1) / decode_rows_per_cta()) > 65535)
    return SDPA_ERR_UNSUPPORTED;
  const size_t need = decode_ws(c, nsplit);
  if (!ws || ws_bytes < need || !aligned16(ws)) return SDPA_ERR_INVALID_ARG;
  DecodeParams dp;
  fill_fwd(dp.f, c, q, k, v, mask, alpha, band, o, lse);
  const size_t rows = static_cast<size_t>(c.B) * c.Hq * c.L;
  dp.part_o = static_cast<float*>(ws);
  dp.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) +
                                         round_up(rows * nsplit * c.Ev * sizeof(float), 256));
  dp.nsplit = nsplit;
  dp.keys_per_split = kps;
  dp.page_k = paged ? paged->page_table_k : nullptr;
  dp.page_v = paged ? paged->page_table_v : nullptr;
  dp.page_stride = paged ? paged->max_blocks : 0;
  dp.bs_k = paged ? paged->block_size_k : 0;
  dp.bs_v = paged ? paged->block_size_v : 0;
  dp.lg_k = dp.bs_k ? __builtin_ctz(static_cast<unsigned>(dp.bs_k)) : 0;
  dp.lg_v = dp.bs_v ? __builtin_ctz(static_cast<unsigned>(dp.bs_v)) : 0;
  dp.nblk_k = paged ? static_cast<int>(paged->num_blocks_k) : 0;
  dp.nblk_v = paged ? static_cast<int>(paged->num_blocks_v) : 0;
  return from_cuda(launch_decode(dp, st));
}

}  // namespace

int num_sms() {
  const int d = current_device();
  if (d < 0) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 148;
    g_sms[d] = n;
  }
  return g_sms[d];
}

namespace {
// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
bool encode_3d(void* tmap, CUtensorMapDataType dt, const void* base, const cuuint64_t (&dims)[3],
               const cuuint64_t (&strides)[2], uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode_tried) {
      g_encode_tried = true;
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
              cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  if (!g_encode) return false;
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(static_cast<CUtensorMap*>(tmap), dt, 3, const_cast<void*>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace

bool encode_tmap_bf16_3d(void* tmap, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                         uint32_t box1) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  return encode_3d(tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box0, box1,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

bool encode_tmap_f32_3d(void* tmap, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0,
                        uint32_t box1, bool swizzle128) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
  return encode_3d(tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box0, box1,
                   swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace sdpa_impl

using namespace sdpa_impl;

namespace sdpa_impl {
namespace {

sdpa_status check_io(const Checked& c, const void* q, const void* k, const void* v, const float* mask, void* o,
                     float* lse) {
  (void)c;
  if (!q || !k || !v || !o || !lse) return SDPA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (mask && !aligned16(mask)))
    return SDPA_ERR_INVALID_ARG;
  return SDPA_OK;
}

sdpa_status forward_impl(const sdpa_shape* shape, const sdpa_options* opts, int is_causal, const void* q,
                         const void* k, const void* v, const float* mask, double scale, int enable_gqa, void* o,
                         float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  Checked c;
  sdpa_status s = check_shape(shape, enable_gqa, mask != nullptr, &c);
  if (s != SDPA_OK) return s;
  float alpha;
  if ((s = check_scale(scale, c.E, &alpha)) != SDPA_OK) return s;
  if ((s = check_io(c, q, k, v, mask, o, lse)) != SDPA_OK) return s;
  Band band = plain_band(is_causal);
  if (opts && (s = band_from_options(opts, c, &band)) != SDPA_OK) return s;
  DropoutParams drop;
  if ((s = dropout_from_options(opts, &drop)) != SDPA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (routes_to_decode(c) && !drop.active)   // dropout is a training-time forward: the prefill kernels
    return run_decode(c, band, q, k, v, mask, alpha, 0, o, lse, workspace, workspace_bytes, st);
  FwdParams p;
  fill_fwd(p, c, q, k, v, mask, alpha, band, o, lse);
  p.drop = drop;
  if (c.bf16 && fwd_tc_supported(c.E, c.Ev)) {
    if ((c.L + 255) / 256 > 65535) return SDPA_ERR_UNSUPPORTED;
    // Padding lengths make the work units uneven: with the workspace the query
    // reports, the CTAs take units from a counter in it instead of a fixed list.
    if ((band.seqlen_q || band.seqlen_kv) && workspace && workspace_bytes >= kFwdSchedBytes &&
        aligned16(workspace)) {
      p.sched = static_cast<unsigned*>(workspace);
      const cudaError_t e = cudaMemsetAsync(p.sched, 0, sizeof(unsigned), st);
      if (e != cudaSuccess) return from_cuda(e);
    }
    return from_cuda(launch_fwd_tc(p, st));
  }
  if ((c.L + 15) / 16 > 65535 || static_cast<long long>(c.B) * c.Hq > 65535) return SDPA_ERR_UNSUPPORTED;
  return from_cuda(launch_fwd_simt(p, c.bf16 ? 1 : 0, st));
}

// A paged cache description: both tables present and 4-byte aligned, block sizes powers of
// two >= 8, tables wide enough for S keys, container indices within int.
sdpa_status check_paged(const sdpa_paged_kv* pg, const Checked& c) {
  if (!pg || !pg->page_table_k || !pg->page_table_v) return SDPA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(pg->page_table_k) & 3) || (reinterpret_cast<uintptr_t>(pg->page_table_v) & 3))
    return SDPA_ERR_INVALID_ARG;
  for (int bs : {pg->block_size_k, pg->block_size_v})
    if (bs < 8 || bs > (1 << 20) || (bs & (bs - 1))) return SDPA_ERR_INVALID_ARG;
  const long long need_k = (static_cast<long long>(c.S) + pg->block_size_k - 1) / pg->block_size_k;
  const long long need_v = (static_cast<long long>(c.S) + pg->block_size_v - 1) / pg->block_size_v;
  if (pg->max_blocks < need_k || pg->max_blocks < need_v) return SDPA_ERR_INVALID_ARG;
  for (long long nb : {pg->num_blocks_k, pg->num_blocks_v})
    if (nb < 1 || nb > INT_MAX || (nb + 1) * c.Hkv > INT_MAX) return SDPA_ERR_INVALID_ARG;
  return SDPA_OK;
}

sdpa_status decode_impl(const sdpa_shape* shape, const sdpa_options* opts, const void* q, const void* k,
                        const void* v, const float* mask, double scale, int enable_gqa, int num_splits, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, bool static_scratch, void* stream,
                        const sdpa_paged_kv* paged = nullptr) {
  Checked c;
  sdpa_status s = check_shape(shape, enable_gqa, mask != nullptr, &c);
  if (s != SDPA_OK) return s;
  float alpha;
  if ((s = check_scale(scale, c.E, &alpha)) != SDPA_OK) return s;
  if (num_splits < 0) return SDPA_ERR_INVALID_ARG;
  if ((s = check_io(c, q, k, v, mask, o, lse)) != SDPA_OK) return s;
  Band band = plain_band(0);
  if (opts && (s = band_from_options(opts, c, &band)) != SDPA_OK) return s;
  if (opts && opts->dropout_p != 0.0) return SDPA_ERR_INVALID_ARG;   // no dropout in the decode
  if (paged && (s = check_paged(paged, c)) != SDPA_OK) return s;
  if (!c.bf16 || !decode_supported(c.E, c.Ev)) return SDPA_ERR_UNSUPPORTED;
  const int want = num_splits > 0 ? num_splits : auto_splits(c);
  if (static_scratch) {
    int nsplit, kps;
    split_layout(c, want, &nsplit, &kps);
    if (decode_ws(c, nsplit) > SDPA_DECODE_STATIC_SCRATCH_BYTES) return SDPA_ERR_UNSUPPORTED;
    size_t cap = 0;
    if (decode_static_scratch(&workspace, &cap) != cudaSuccess) return SDPA_ERR_CUDA;
    workspace_bytes = cap;
  }
  return run_decode(c, band, q, k, v, mask, alpha, want, o, lse, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream), paged);
}

sdpa_status backward_impl(const sdpa_shape* shape, const sdpa_options* opts, int is_causal, const void* q,
                          const void* k, const void* v, const void* o, const void* dO, const float* lse,
                          const float* mask, double scale, int enable_gqa, void* dq, void* dk, void* dv,
                          void* workspace, size_t workspace_bytes, void* stream) {
  Checked c;
  sdpa_status s = check_shape(shape, enable_gqa, mask != nullptr, &c);
  if (s != SDPA_OK) return s;
  float alpha;
  if ((s = check_scale(scale, c.E, &alpha)) != SDPA_OK) return s;
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return SDPA_ERR_INVALID_ARG;
  if (mask && !aligned16(mask)) return SDPA_ERR_INVALID_ARG;
  Band band = plain_band(is_causal);
  if (opts && (s = band_from_options(opts, c, &band)) != SDPA_OK) return s;
  DropoutParams drop;
  if ((s = dropout_from_options(opts, &drop)) != SDPA_OK) return s;
  const size_t need = bwd_ws(c);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return SDPA_ERR_INVALID_ARG;
  BwdParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.dO = dO;
  p.lse = lse;
  p.mask = mask;
  p.D = static_cast<float*>(workspace);
  p.dq_acc = bwd_uses_tc(c) ? reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_stats_bytes(c))
                            : nullptr;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = c.B;
  p.Hq = c.Hq;
  p.Hkv = c.Hkv;
  p.L = c.L;
  p.S = c.S;
  p.E = c.E;
  p.Ev = c.Ev;
  p.G = c.G;
  p.mask_sb = c.mask_sb;
  p.mask_sh = c.mask_sh;
  p.scale = alpha;
  p.scale_log2 = alpha * kLog2e;
  p.band = band;
  p.drop = drop;
  p.status = status_ptr();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.dq_acc) {
    if (c.B * c.Hkv > 65535 * 64 || (c.S + 127) / 128 > 65535) return SDPA_ERR_UNSUPPORTED;
    return from_cuda(launch_bwd_tc(p, st));
  }
  cudaError_t e = launch_bwd_preprocess(p, c.bf16 ? 1 : 0, st);
  if (e != cudaSuccess) return SDPA_ERR_CUDA;
  if ((c.L + 15) / 16 > 65535 || (c.S + 15) / 16 > 65535 || static_cast<long long>(c.B) * c.Hq > 65535)
    return SDPA_ERR_UNSUPPORTED;
  return from_cuda(launch_bwd_simt(p, c.bf16 ? 1 : 0, st));
}

}  // namespace
}  // namespace sdpa_impl

extern "C" {

sdpa_status sdpa_forward(const sdpa_shape* shape, const void* q, const void* k, const void* v,
                         const float* mask_or_null, double scale, int is_causal, int enable_gqa, void* o,
                         float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return forward_impl(shape, nullptr, is_causal, q, k, v, mask_or_null, scale, enable_gqa, o, lse, workspace,
                      workspace_bytes, stream);
}

sdpa_status sdpa_forward_opts(const sdpa_shape* shape, const sdpa_options* options, const void* q, const void* k,
                              const void* v, const float* mask_or_null, double scale, int enable_gqa, void* o,
                              float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!options) return SDPA_ERR_INVALID_ARG;
  return forward_impl(shape, options, 0, q, k, v, mask_or_null, scale, enable_gqa, o, lse, workspace,
                      workspace_bytes, stream);
}

size_t sdpa_forward_workspace_bytes(const sdpa_shape* shape) {
  Checked c;
  if (check_shape(shape, 1, false, &c) != SDPA_OK) return 0;
  if (!routes_to_decode(c)) return c.bf16 && fwd_tc_supported(c.E, c.Ev) ? kFwdSchedBytes : 0;
  int nsplit, kps;
  split_layout(c, auto_splits(c), &nsplit, &kps);
  return decode_ws(c, nsplit);
}

sdpa_status sdpa_decode(const sdpa_shape* shape, const void* q, const void* k, const void* v,
                        const float* mask_or_null, double scale, int enable_gqa, int num_splits, void* o,
                        float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(shape, nullptr, q, k, v, mask_or_null, scale, enable_gqa, num_splits, o, lse, workspace,
                     workspace_bytes, false, stream);
}

sdpa_status sdpa_decode_opts(const sdpa_shape* shape, const sdpa_options* options, const void* q, const void* k,
                             const void* v, const float* mask_or_null, double scale, int enable_gqa,
                             int num_splits, void* o, float* lse, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (!options) return SDPA_ERR_INVALID_ARG;
  return decode_impl(shape, options, q, k, v, mask_or_null, scale, enable_gqa, num_splits, o, lse, workspace,
                     workspace_bytes, false, stream);
}

sdpa_status sdpa_decode_paged(const sdpa_shape* shape, const sdpa_options* options, const sdpa_paged_kv* paged,
                              const void* q, const void* k_container, const void* v_container,
                              const float* mask_or_null, double scale, int enable_gqa, int num_splits, void* o,
                              float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!paged) return SDPA_ERR_INVALID_ARG;
  return decode_impl(shape, options, q, k_container, v_container, mask_or_null, scale, enable_gqa, num_splits, o,
                     lse, workspace, workspace_bytes, false, stream, paged);
}

sdpa_status sdpa_decode_noalloc(const sdpa_shape* shape, const void* q, const void* k, const void* v,
                                const float* mask_or_null, double scale, int enable_gqa, int num_splits, void* o,
                                float* lse, void* stream) {
  return decode_impl(shape, nullptr, q, k, v, mask_or_null, scale, enable_gqa, num_splits, o, lse, nullptr, 0,
                     true, stream);
}

size_t sdpa_decode_workspace_bytes(const sdpa_shape* shape, int num_splits) {
  Checked c;
  if (check_shape(shape, 1, false, &c) != SDPA_OK || num_splits < 0) return 0;
  int nsplit, kps;
  split_layout(c, num_splits > 0 ? num_splits : auto_splits(c), &nsplit, &kps);
  return decode_ws(c, nsplit);
}

int sdpa_decode_num_splits(const sdpa_shape* shape) {
  Checked c;
  if (check_shape(shape, 1, false, &c) != SDPA_OK) return 0;
  int nsplit, kps;
  split_layout(c, auto_splits(c), &nsplit, &kps);
  return nsplit;
}

sdpa_status sdpa_backward(const sdpa_shape* shape, const void* q, const void* k, const void* v, const void* o,
                          const void* dO, const float* lse, const float* mask_or_null, double scale,
                          int is_causal, int enable_gqa, void* dq, void* dk, void* dv, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return backward_impl(shape, nullptr, is_causal, q, k, v, o, dO, lse, mask_or_null, scale, enable_gqa, dq, dk, dv,
                       workspace, workspace_bytes, stream);
}

sdpa_status sdpa_backward_opts(const sdpa_shape* shape, const sdpa_options* options, const void* q, const void* k,
                               const void* v, const void* o, const void* dO, const float* lse,
                               const float* mask_or_null, double scale, int enable_gqa, void* dq, void* dk,
                               void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (!options) return SDPA_ERR_INVALID_ARG;
  return backward_impl(shape, options, 0, q, k, v, o, dO, lse, mask_or_null, scale, enable_gqa, dq, dk, dv,
                       workspace, workspace_bytes, stream);
}

size_t sdpa_backward_workspace_bytes(const sdpa_shape* shape) {
  Checked c;
  if (check_shape(shape, 1, false, &c) != SDPA_OK) return 0;
  return bwd_ws(c);
}

const char* sdpa_status_string(sdpa_status status) {
  switch (status) {
    case SDPA_OK: return "ok";
    case SDPA_ERR_INVALID_ARG: return "invalid argument";
    case SDPA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case SDPA_ERR_CUDA: return "CUDA error";
    case SDPA_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

sdpa_status sdpa_selftest_wait_timeout(void* stream) {
  unsigned* status = status_ptr();
  if (!status) return SDPA_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return from_cuda(cudaGetLastError());
}

sdpa_status sdpa_last_device_status(void* stream) {
  // Ordered after the work already on `stream` and synchronising only that
  // stream: no other stream or host thread of the device waits for it.
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* word = status_ptr();
  if (!word) return SDPA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return SDPA_ERR_CUDA;
  if (v != 0) {
    if (cudaMemsetAsync(word, 0, sizeof(v), st) != cudaSuccess || cudaStreamSynchronize(st) != cudaSuccess)
      return SDPA_ERR_CUDA;
    return static_cast<sdpa_status>(v & 0xffu);
  }
  return SDPA_OK;
}

}  // extern "C"
