/*
 * sdpa.h - C ABI of a GB300 (sm_103a) scaled dot-product attention library.
 *
 * The library computes  O = softmax(alpha * Q K^T + mask) V  (forward, with a
 * per-row log-sum-exp), its hand-derived backward (dQ, dK, dV), and a
 * split-KV decode for a single query row.  Definitions follow the course
 * chapter "Scaled dot-product attention (forward and backward)" (sections 2.1
 * to 2.3: scores, masked softmax, output, and the backward dV = P^T dO,
 * dP = dO V^T, dS = P o (dP - D), D = rowsum(dO o O), dQ = alpha dS K,
 * dK = alpha dS^T Q), the "ScaledDotProductAttentionBackward" API page
 * (additive mask, engine-side causal j <= i, argument checks), the
 * "Understanding PyTorch Scaled Dot-Product Attention" post (section 3: causal
 * = tril(diagonal=0); section 4: grouped-query heads by repeat_interleave) and
 * the cuDNN "Attention" page (stats = max + ln(sum exp(s - max)), fp32,
 * natural log; split-KV merges of such statistics).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layout    Every tensor is dense, row-major "BHSD":
 *              q [B, Hq, L, E]    k [B, Hkv, S, E]    v [B, Hkv, S, Ev]
 *              o [B, Hq, L, Ev]   dO like o           lse [B, Hq, L] (fp32)
 *              dq like q          dk like k           dv like v
 *              mask [mask_b, mask_h, L, S] fp32 with mask_b in {1, B} and
 *              mask_h in {1, Hq}; a size-1 dimension broadcasts.
 *  Pointers  All tensor and workspace pointers are DEVICE pointers on the
 *            current CUDA device, 16-byte aligned.  The caller owns every
 *            buffer; the library never allocates or frees device memory and
 *            never synchronises the stream: work is enqueued on `stream`
 *            (0 = legacy default stream) and the call returns.
 *  dtype     q, k, v, o, dO, dq, dk, dv share one dtype (SDPA_F32 or
 *            SDPA_BF16).  mask and lse are always fp32.  Accumulation and all
 *            softmax statistics are fp32 in every path.
 *  scale     alpha.  Pass a NaN to select the default 1/sqrt(E).  It scales
 *            Q K^T only, never the mask.  Negative or infinite -> INVALID_ARG.
 *  mask      Additive: -inf blocks a (query, key) pair, finite values are
 *            added to the scaled score.  NULL = no mask.
 *  causal    is_causal != 0 blocks key j for query i when j > i (top-left
 *            aligned, for any L and S).  Combines with a mask.  The *_opts
 *            entry points take padding lengths, a diagonal alignment and band
 *            bounds instead (sdpa_options below).
 *  GQA       Query head h reads KV head h / (Hq / Hkv).  Hq != Hkv requires
 *            enable_gqa != 0 and Hq % Hkv == 0.  dk and dv are summed over
 *            the Hq / Hkv query heads that share a KV head.
 *  Empty rows  A query row whose every key is blocked gets o = 0,
 *            lse = -inf, dq = 0, and adds nothing to dk, dv.
 *  Errors    Functions never throw.  Argument errors are detected on the host
 *            before anything is enqueued.  A kernel launch failure returns
 *            SDPA_ERR_CUDA.  Kernels never trap: a device-side pipeline wait
 *            that exceeds its time limit records SDPA_ERR_TIMEOUT in a device
 *            status word, read by sdpa_last_device_status().
 *
 * Supported sizes: B, Hq, Hkv, L, S >= 1.  fp32: 1 <= E, Ev <= 128.  bf16:
 * E and Ev multiples of 8, at most 128 (the tensor-core prefill and backward
 * take E, Ev in {64, 128}; other bf16 widths run on the CUDA-core kernels).
 * Extents: B, Hq, Hkv <= 2^31 - 1, B * Hq <= 2^31 - 1, L, S <= 2^30 - 1,
 * B * Hkv <= 4,194,240, B * Hq * L and B * Hkv * S at most 2^49 rows, and
 * at most 2^56 mask elements (each extent is bounded before any product is
 * formed, so no size computation wraps).  Anything else ->
 * SDPA_ERR_UNSUPPORTED.
 */
#ifndef SDPA_GB300_H
#define SDPA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SDPA_OK = 0,
  SDPA_ERR_INVALID_ARG = 1,   /* bad pointer, shape, scale or workspace size */
  SDPA_ERR_UNSUPPORTED = 2,   /* valid but outside the supported sizes/dtypes */
  SDPA_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  SDPA_ERR_TIMEOUT = 4        /* a device-side wait gave up (see below) */
} sdpa_status;

typedef enum { SDPA_F32 = 0, SDPA_BF16 = 1 } sdpa_dtype;

/* Problem sizes.  mask_b / mask_h are the mask's first two extents (1 or B,
 * 1 or Hq); ignored when the mask pointer is NULL. */
typedef struct {
  int64_t B, Hq, Hkv, L, S, E, Ev;
  int32_t dtype;               /* sdpa_dtype */
  int32_t mask_b, mask_h;
} sdpa_shape;

/* Forward: o = softmax(scale * q k^T + mask + causal) v and
 * lse[b,h,i] = max_j t_ij + ln(sum_j exp(t_ij - max_j t_ij)), t = the masked
 * scaled scores (course chapter sections 2.1-2.2; cuDNN "Attention",
 * Scaled Dot Product Attention, stats).  lse is always written.
 * A bf16 call with L == 1 (E, Ev in {64, 128}) runs the split-KV decode (same
 * contract as sdpa_decode with num_splits = 0) and needs the workspace
 * reported by sdpa_forward_workspace_bytes; every other call needs none
 * (workspace may then be NULL with workspace_bytes = 0).  A bf16 prefill call
 * on the tensor cores (E, Ev in {64, 128}) with padding lengths
 * (sdpa_forward_opts) uses the workspace when it is given (at least
 * sdpa_forward_workspace_bytes, 16-byte aligned): the call zeroes a counter in
 * it on the stream and the kernel's CTAs take work units from it in turn,
 * which evens out sequences of unequal length; without it the units follow a
 * fixed order.  Both give the same results. */
sdpa_status sdpa_forward(const sdpa_shape* shape,
                         const void* q, const void* k, const void* v,
                         const float* mask_or_null, double scale,
                         int is_causal, int enable_gqa,
                         void* o, float* lse,
                         void* workspace, size_t workspace_bytes,
                         void* stream /* cudaStream_t */);

/* Device workspace bytes sdpa_forward uses for `shape`: the decode path's
 * partials when it routes there, 256 bytes (a unit counter) for a bf16 prefill
 * on the tensor cores, 0 otherwise. */
size_t sdpa_forward_workspace_bytes(const sdpa_shape* shape);

/* Backward of sum(o * dO) (course chapter section 2.3): writes dq [B,Hq,L,E],
 * dk [B,Hkv,S,E], dv [B,Hkv,S,Ev].  o and lse must be the forward's outputs for
 * the same inputs and flags; P is recomputed from q, k and lse, never stored.
 * D_i = dO_i . o_i is computed in fp32 first.  dq, dk, dv are fully
 * overwritten.  Needs sdpa_backward_workspace_bytes(shape) bytes of device
 * workspace (fp32 D, and for bf16 an fp32 dQ accumulator). */
sdpa_status sdpa_backward(const sdpa_shape* shape,
                          const void* q, const void* k, const void* v,
                          const void* o, const void* dO, const float* lse,
                          const float* mask_or_null, double scale,
                          int is_causal, int enable_gqa,
                          void* dq, void* dk, void* dv,
                          void* workspace, size_t workspace_bytes,
                          void* stream /* cudaStream_t */);

size_t sdpa_backward_workspace_bytes(const sdpa_shape* shape);

/* Split-KV decode forward (bf16, any L but typically L == 1): the S keys of
 * each (batch, KV head) are cut into num_splits contiguous ranges; one pass
 * per range reads its keys and values once for all Hq/Hkv query heads of the
 * group and writes a partial (o_s, lse_s) to the workspace; a merge pass
 * combines them: lse = logsumexp_s(lse_s) (empty ranges have lse_s = -inf),
 * o = sum_s exp(lse_s - lse) o_s (cuDNN "Attention": log-sum-exp statistics
 * and their split-KV merges).  num_splits = 0 picks a count from the GPU's SM
 * count.  The result equals the plain forward up to fp32 rounding for every
 * split count.  No causal flag here (top-left causal would leave one key for
 * L == 1); sdpa_decode_opts takes padding lengths (e.g. each sequence's cache
 * length) and a bottom-right band. */
sdpa_status sdpa_decode(const sdpa_shape* shape,
                        const void* q, const void* k, const void* v,
                        const float* mask_or_null, double scale, int enable_gqa,
                        int num_splits,
                        void* o, float* lse,
                        void* workspace, size_t workspace_bytes,
                        void* stream /* cudaStream_t */);

/* Workspace bytes for sdpa_decode with this split count (0 = automatic). */
size_t sdpa_decode_workspace_bytes(const sdpa_shape* shape, int num_splits);

/* The split count sdpa_decode uses for num_splits = 0 on the current device. */
int sdpa_decode_num_splits(const sdpa_shape* shape);

/* Size of the fixed device scratch behind sdpa_decode_noalloc: 8 MiB. */
#define SDPA_DECODE_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

/* sdpa_decode without a workspace, for callers that cannot allocate device
 * memory.  (The pages describe no such entry point: it exists for callers of
 * this library, not for the method.)  Typical callers: an operator plugin
 * inside another runtime that is handed its input and output tensors but no
 * scratch, or a serving loop whose device memory is planned once at start-up
 * and which may not call cudaMalloc afterwards (cudaMalloc can synchronise the
 * device and fragments a fixed budget).
 *
 * Same arguments, result and errors as sdpa_decode, minus the workspace.  The
 * split partials live in one file-scope device array of
 * SDPA_DECODE_STATIC_SCRATCH_BYTES that every GPU which loads the library holds
 * until the process exits.  A call needs B*Hq*L*num_splits*(Ev+1)*4 bytes of it
 * (the two parts each rounded up to 256 bytes); a call that needs more returns
 * SDPA_ERR_UNSUPPORTED before anything is enqueued.  Neither the library nor
 * this call allocates or frees device memory.
 *
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  The address is kept per device and context: after the
 * device's context is replaced (cudaDeviceReset), the next call looks it up
 * again, and that call too should come before any capture.  Every call uses the same array and leaves its partials
 * there; each call overwrites all of the scratch it reads, so nothing needs
 * clearing between calls.  Calls whose work overlaps on the GPU (other streams,
 * other host threads) race on the array and corrupt each other's results:
 * issue them in order on one stream. */
sdpa_status sdpa_decode_noalloc(const sdpa_shape* shape,
                                const void* q, const void* k, const void* v,
                                const float* mask_or_null, double scale, int enable_gqa,
                                int num_splits,
                                void* o, float* lse,
                                void* stream /* cudaStream_t */);

/* Padding and diagonal-band options of the *_opts entry points (cuDNN
 * "Attention": Configurable Options, Padding mask and Diagonal masking
 * options; Scaled Dot Product Attention, Args seq_len_q, seq_len_kv,
 * diagonal_alignment, diagonal_band_left_bound, diagonal_band_right_bound).
 *
 *  seq_len_q, seq_len_kv  NULL, or DEVICE arrays of B int32 (4-byte aligned)
 *            holding each batch's actual query / key-value length; values are
 *            clamped to [0, L] and [0, S].  Query rows i >= seq_len_q[b] are
 *            padding: o = 0, lse = -inf, dq = 0, and they add nothing to dk,
 *            dv.  Keys j >= seq_len_kv[b] are masked (dk = dv = 0 there).  A
 *            batch of length 0 is skipped this way.  NULL = full length.
 *  diagonal_alignment  SDPA_TOP_LEFT: row i's diagonal is column i.
 *            SDPA_BOTTOM_RIGHT: column i + Skv_b - Sq_b, with the actual
 *            lengths of batch b (prefix-LM and decode diagonals).
 *  right_bound  < 0: none.  >= 0: columns beyond diagonal + right_bound are
 *            masked (0 = causal about the aligned diagonal).
 *  left_bound   <= 0: none.  >= 1: columns at or before diagonal - left_bound
 *            are masked (a sliding window of left_bound keys ending at the
 *            diagonal).
 * All of it applies together with the additive mask; a row left without keys
 * follows the empty-row rule above.
 *
 *  dropout_p, dropout_seed, dropout_offset  Attention dropout of the prefill
 *            forward and backward ("Scaled dot-product attention (forward and
 *            backward)", section 2.5; cuDNN "Attention", Philox RNG dropout):
 *            o = (P o m) v with m = keep / (1 - p), one uniform per weight,
 *            keep where u >= p; the backward replays m (dV = (P o m)^T dO,
 *            dP = (dO v^T) o m).  lse stays the statistics of P before dropout.
 *            Weight (b, h, i, j) takes its uniform from Philox4x32-10 with key
 *            (dropout_seed mod 2^32, dropout_seed / 2^32) and counter (j / 8, i,
 *            b * Hq + h, dropout_offset): 16-bit chunk j % 8 of the 128-bit
 *            output (word (j % 8) / 2, bits 16 * (j % 2)), kept iff
 *            >= ceil(p * 65536).  p = 0: no dropout; p outside [0, 1), or
 *            dropout_offset >= 2^32 with p != 0 -> INVALID_ARG.  The decode
 *            entry points take no dropout (dropout_p != 0 -> INVALID_ARG).
 *
 * The backward must get the forward's options.  Other values of
 * diagonal_alignment, or misaligned length pointers, -> INVALID_ARG. */
typedef enum { SDPA_TOP_LEFT = 0, SDPA_BOTTOM_RIGHT = 1 } sdpa_diag_alignment;

typedef struct {
  const int32_t* seq_len_q;
  const int32_t* seq_len_kv;
  int32_t diagonal_alignment;  /* sdpa_diag_alignment */
  int32_t right_bound;
  int32_t left_bound;
  double dropout_p;
  uint64_t dropout_seed;
  uint64_t dropout_offset;
} sdpa_options;

/* sdpa_forward, sdpa_backward and sdpa_decode with sdpa_options in place of
 * is_causal (is_causal != 0 equals {NULL, NULL, SDPA_TOP_LEFT, 0, 0}).  Same
 * arguments, workspaces, routing and errors otherwise; options must not be
 * NULL (INVALID_ARG).  The lengths are read on the device, so the work skipped
 * for padding is decided by the kernels. */
sdpa_status sdpa_forward_opts(const sdpa_shape* shape, const sdpa_options* options,
                              const void* q, const void* k, const void* v,
                              const float* mask_or_null, double scale, int enable_gqa,
                              void* o, float* lse,
                              void* workspace, size_t workspace_bytes,
                              void* stream /* cudaStream_t */);

sdpa_status sdpa_backward_opts(const sdpa_shape* shape, const sdpa_options* options,
                               const void* q, const void* k, const void* v,
                               const void* o, const void* dO, const float* lse,
                               const float* mask_or_null, double scale, int enable_gqa,
                               void* dq, void* dk, void* dv,
                               void* workspace, size_t workspace_bytes,
                               void* stream /* cudaStream_t */);

sdpa_status sdpa_decode_opts(const sdpa_shape* shape, const sdpa_options* options,
                             const void* q, const void* k, const void* v,
                             const float* mask_or_null, double scale, int enable_gqa,
                             int num_splits,
                             void* o, float* lse,
                             void* workspace, size_t workspace_bytes,
                             void* stream /* cudaStream_t */);

/* Paged K/V caches of sdpa_decode_paged (cuDNN "Attention": Configurable
 * Options, Paged attention; Tensors, Page Table K / V).  k and v are then
 * containers of fixed-size key blocks, k [num_blocks_k, Hkv, block_size_k, E]
 * and v [num_blocks_v, Hkv, block_size_v, Ev] (bf16, dense, 16-byte aligned),
 * and key s of batch b is
 *     k_cache[b, h, s, :] = k[page_table_k[b * max_blocks + s / block_size_k], h, s % block_size_k, :]
 * (likewise v).  page_table_k / page_table_v: DEVICE int32 arrays of
 * B * max_blocks entries, 4-byte aligned (they may be the same array).
 * block_size_k / block_size_v: powers of two, at least 8.  max_blocks: the
 * tables' row length, at least ceil(S / block_size) for both.  An entry that
 * is negative or >= num_blocks reads zeros (use it for blocks past a
 * sequence's length, which seq_len_kv masks anyway).  Bad fields -> INVALID_ARG. */
typedef struct {
  const int32_t* page_table_k;
  const int32_t* page_table_v;
  int32_t block_size_k;
  int32_t block_size_v;
  int32_t max_blocks;
  int64_t num_blocks_k;
  int64_t num_blocks_v;
} sdpa_paged_kv;

/* sdpa_decode_opts over paged K/V caches.  shape->S is the longest cache (the
 * logical key length); options may be NULL and usually give seq_len_kv, each
 * sequence's cache length.  Same workspace, results and errors as
 * sdpa_decode. */
sdpa_status sdpa_decode_paged(const sdpa_shape* shape, const sdpa_options* options, const sdpa_paged_kv* paged,
                              const void* q, const void* k_container, const void* v_container,
                              const float* mask_or_null, double scale, int enable_gqa,
                              int num_splits,
                              void* o, float* lse,
                              void* workspace, size_t workspace_bytes,
                              void* stream /* cudaStream_t */);

/* Static, NUL-terminated description of a status code. */
const char* sdpa_status_string(sdpa_status status);

/* Failure-path self-test: launches, on `stream`, one CTA whose thread waits on an
 * mbarrier that nothing ever arrives at.  The wait is bounded like every wait in
 * the kernels: it gives up after its limit (about a second), records
 * SDPA_ERR_TIMEOUT in the device status word and the kernel returns normally, so
 * the context stays usable.  Returns the launch's status; the caller then reads
 * sdpa_last_device_status() (SDPA_ERR_TIMEOUT once, then SDPA_OK). */
sdpa_status sdpa_selftest_wait_timeout(void* stream /* cudaStream_t */);

/* Reads and clears the current device's status word that kernels set when a
 * bounded device-side wait gives up.  Returns SDPA_OK when no kernel has timed
 * out since the last call.  The read is enqueued on `stream` (a cudaStream_t;
 * NULL is the default stream) after the work already there, and only that
 * stream is synchronised: pass the stream the library's calls ran on.  Calls
 * still running on other streams are not waited for, so their timeouts show
 * on a later read.  A host-blocking call: keep it off the hot path (tests,
 * after an error). */
sdpa_status sdpa_last_device_status(void* stream /* cudaStream_t */);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_GB300_H */
