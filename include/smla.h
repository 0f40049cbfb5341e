/* smla — sparse top-k MLA attention for one GB300 (sm_103a). C ABI.
 *
 * What is computed (DeepSeek-V4-style sparse MLA; pages: sglang PR "[SM12x] Drop the
 * 64-head TP pad on the DSv4 MLA prefill path", Problem — H query heads share a single
 * latent KV row per cached token (num_kv_heads = 1), prefill is many query rows and
 * compute-bound, decode is few rows and KV-bandwidth-bound; flashinfer PR "add topk=256
 * prefill-dsv4 dispatch", Description — the launch is parameterised by num_heads, topk,
 * page_block_size = 64, topk_extra and extra_page_block_size; flashinfer PR "explain
 * sparse-MLA decode dispatch misses; add config query API", merged-body Summary and
 * Compatibility — -1 marks a masked slot, index and out_lse tensors may be row-strided,
 * T = 0 returns without work; sglang PR Correctness — an attention-sink logit per head):
 *
 *   for every query token t (sequence s = token_seq[t]) and head h < H:
 *     J      = valid entries of t's main index row, plus valid entries of its extra row
 *     x_j    = sm_scale * <q[t,h,0:576], K_j[0:576]>
 *     m      = max(x_j, sink[h]);  Z = sum_j e^(x_j - m);  D = Z + e^(sink[h] - m)
 *     out[t,h,0:512] = sum_j e^(x_j - m) * K_j[0:512] / D        (V = first 512 channels)
 *     lse[t,h]       = m + ln Z            (natural log; the sink is not included)
 *   With no sink the sink terms vanish. If J is empty: out = 0 and lse = -inf.
 *
 * Validity of entry j of token t in a set: j < topk (and j < topk_length[t] when given),
 * i = indices[t*idx_stride + j] satisfies 0 <= i < seq_lens[s], i/64 < bt_stride, and
 * p = block_table[s*bt_stride + i/64] satisfies 0 <= p < num_pages. Invalid entries are
 * never read. token_seq[t] outside [0, num_seqs) gives token t an empty J.
 * Cache row of logical position i: cache + p*page_stride_bytes + (i%64)*row_stride_bytes.
 *
 * Row formats (d_qk = 576 = 512 latent + 64 rope, d_v = 512):
 *   SMLA_KV_BF16          576 x bf16 (1152 bytes).
 *   SMLA_KV_FP8_E4M3_S128 656 bytes: [512 x OCP E4M3FN][4 x fp32 scale, one per 128
 *                         latent channels][64 x bf16 rope]; K[c] = e4m3[c]*scale[c/128].
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library keeps no
 *     reference after the call returns and allocates no device memory.
 *   - Work is enqueued on `stream` only; no call synchronises the device or the stream.
 *   - Argument errors are returned before anything is launched; nothing aborts, throws
 *     or traps. A launch failure returns SMLA_ERR_CUDA.
 *   - The GPU path is the only path: there is no CPU fallback.
 *   - Calls are thread-safe except smla_set_crossover / smla_load_crossover, which
 *     replace the process-global dispatch table and must not race with smla_forward.
 */
#ifndef SMLA_H
#define SMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMLA_D_QK 576
#define SMLA_D_V 512
#define SMLA_PAGE_SIZE 64
#define SMLA_MAX_HEADS 128

typedef struct CUstream_st* smla_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  SMLA_OK = 0,
  SMLA_ERR_INVALID = 1,     /* malformed arguments (null pointer, bad stride, misalignment) */
  SMLA_ERR_UNSUPPORTED = 2, /* well-formed but outside the envelope (smla_supported says why) */
  SMLA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than smla_workspace_size() */
  SMLA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  SMLA_ERR_DEVICE = 5       /* a kernel gave up on a bounded wait (see smla_device_error) */
} smla_status;

typedef enum { SMLA_KV_BF16 = 0, SMLA_KV_FP8_E4M3_S128 = 1 } smla_kv_format;

/* One paged latent cache plus the index set that reads it (the main set, or the
 * "extra" set of the dual-cache layout, flashinfer PR "add topk=256 prefill-dsv4
 * dispatch", Description: topk_extra / extra_page_block_size). */
typedef struct {
  const void* cache;          /* device; page 0 row 0; 16-byte aligned */
  int32_t format;             /* smla_kv_format */
  int64_t row_stride_bytes;   /* >= row bytes (1152 / 656), multiple of 16; padded rows allowed */
  int64_t page_stride_bytes;  /* >= 64 * row_stride_bytes, multiple of 16 */
  int32_t page_size;          /* must be 64 (checked: a wrong page size must not run) */
  int32_t num_pages;          /* physical pages in `cache` (bounds for block_table entries); <= 2^25 */
  const int32_t* block_table; /* device [num_seqs, bt_stride]: logical page -> physical page */
  int32_t bt_stride;          /* >= 1 */
  const int32_t* seq_lens;    /* device [num_seqs]: valid positions per sequence */
  const int32_t* indices;     /* device [T, idx_stride] logical positions; < 0 = masked */
  int64_t idx_stride;         /* elements, >= topk (row-strided views allowed) */
  int32_t topk;               /* >= 1 entries per token (any width; not only multiples of 64) */
  const int32_t* topk_length; /* device [T] valid width per token, or NULL for topk */
} smla_kv_set;

typedef struct {
  int32_t T;        /* query tokens (0 = nothing to do) */
  int32_t H;        /* heads, 1..128 (no padding: any value runs natively) */
  int32_t d_qk;     /* must be 576 */
  int32_t d_v;      /* must be 512 */
  int32_t num_seqs; /* rows of block_table / seq_lens (both sets) */
  const void* q;    /* device bf16 [T, H, 576]; element (t,h,c) at q[t*q_stride_t + h*q_stride_h + c] */
  int64_t q_stride_t, q_stride_h; /* elements, multiples of 8; q 16-byte aligned */
  const int32_t* token_seq;       /* device [T]: sequence id of each query token */
  smla_kv_set main;
  const smla_kv_set* extra;       /* host pointer to the second set, or NULL */
  const float* sink;              /* device fp32 [H] per-head logits, or NULL */
  float sm_scale;                 /* multiplies q.K; the sink is NOT scaled */
  void* out;                      /* device bf16 [T, H, 512], element at out[t*out_stride_t + h*out_stride_h + c] */
  int64_t out_stride_t, out_stride_h; /* elements, multiples of 8; out 16-byte aligned */
  float* lse;                     /* device fp32 [T, H] at lse[t*lse_stride_t + h], or NULL */
  int64_t lse_stride_t;           /* elements, >= H when lse != NULL */
  void* workspace;                /* device scratch for smla_decode / smla_forward, 256-byte aligned */
  size_t workspace_bytes;
} smla_params;

/* Envelope query (flashinfer PR "explain sparse-MLA decode dispatch misses; add config
 * query API": name which parameter missed and what is accepted). Returns 1 if `p`
 * describes a supported problem, else 0 and writes a NUL-terminated reason naming the
 * field and the accepted values into why[0..why_len) (why may be NULL). Reads only
 * host-side fields; never touches device memory. */
int smla_supported(const smla_params* p, char* why, size_t why_len);

/* Device scratch bytes smla_decode needs for `p` (split-K partial outputs and
 * log-sum-exps); smla_forward needs the same. 0 when the problem needs none. The value
 * depends only on T, H, the top-k widths and the GPU's SM count. */
size_t smla_workspace_size(const smla_params* p);

/* Prefill schedule: one CTA per (token, head group) streams the token's whole index
 * list through the tensor cores and writes out/lse directly. Correct for any T >= 1.
 * Uses no workspace. (sglang PR Problem: prefill, many query rows, compute-bound.) */
smla_status smla_prefill(const smla_params* p, smla_stream_t stream);

/* Decode schedule: the index list of each (token, head group) is split across CTAs
 * (split-K); partial outputs go to `workspace` and a combine kernel merges them by their
 * log-sum-exps, then applies the sink. Correct for any T >= 1.
 * Requires workspace_bytes >= smla_workspace_size(p). (sglang PR Problem: decode, few
 * rows, KV-bandwidth-bound; flashinfer PR "explain ..." merged body: decode split-K.) */
smla_status smla_decode(const smla_params* p, smla_stream_t stream);

/* smla_decode without a caller-provided workspace. None of the cited sources has a
 * counterpart: this entry point exists for callers that cannot allocate device memory themselves (a plugin behind a
 * fixed C interface that passes only the problem tensors, or a runtime whose device memory
 * is wholly owned by its own pool). It ignores p->workspace / p->workspace_bytes and keeps
 * the split-K partials in a 32 MiB array inside the library, which every GPU that loads
 * libsmla holds until the process exits; it calls no allocator. Problems whose
 * smla_workspace_size() exceeds 32 MiB are rejected with SMLA_ERR_WORKSPACE before any
 * launch. The first call on a device looks up that array's device address (with the
 * device current); make that first call before any stream capture. All calls on a device
 * share the one array: calls that overlap on the GPU (unordered streams) race, so order
 * them. Results equal smla_decode's. */
smla_status smla_decode_static(const smla_params* p, smla_stream_t stream);

/* Cache writer: packs n new latent rows into a paged cache (the step that fills the cache
 * this library reads; the pages' benchmark packs its KV with such a quantiser before every
 * measurement: flashinfer PR "add topk=256 prefill-dsv4 dispatch", conversation, GB10
 * benchmark "Method" paragraph).
 *   kv        device [n, kv_stride] rows of 576 values (512 latent + 64 rope), bf16
 *             (kv_dtype = SMLA_IN_BF16) or fp32 (SMLA_IN_F32); 16-byte aligned, kv_stride
 *             in elements, kv_stride * element size a multiple of 16.
 *   slots     device int64 [n]: physical row of each new token, page * 64 + row in page;
 *             a slot < 0 or >= num_pages * 64 skips that row (nothing is written).
 *   cache     device bytes laid out as smla_kv_set describes (row/page strides, num_pages).
 *   format    SMLA_KV_BF16: every channel rounded to bf16 (nearest, ties to even; a bf16
 *             input is copied). SMLA_KV_FP8_E4M3_S128: per 128 latent channels
 *             scale = amax / 448 in fp32 (1 for an all-zero block), code = E4M3FN of the fp32
 *             quotient x / scale rounded to nearest even and saturated to +-448; rope
 *             rounded to bf16. The reading of the pages is ours: they give no arithmetic.
 * Inputs are expected to be finite. Rows written by two entries with the same slot race.
 * Argument errors return before any launch; enqueued on `stream` only. */
typedef enum { SMLA_IN_BF16 = 0, SMLA_IN_F32 = 1 } smla_in_dtype;
smla_status smla_quantize_kv(const void* kv, int32_t kv_dtype, int64_t kv_stride, int32_t n,
                             const int64_t* slots, void* cache, int32_t format,
                             int64_t row_stride_bytes, int64_t page_stride_bytes, int32_t num_pages,
                             smla_stream_t stream);

/* Calibrated dispatch (flashinfer PR "explain ..." merged body, Dispatch: crossover —
 * decode serves T <= decode_max_tokens for the configuration, prefill serves the rest).
 * Routes to smla_decode when T <= smla_decode_max_tokens(H, topk total, main format),
 * else to smla_prefill. Both routes compute the same result. */
smla_status smla_forward(const smla_params* p, smla_stream_t stream);

/* The crossover threshold currently in force for (H, total top-k width, main format):
 * the calibrated table entry nearest in (H, topk) if a table is loaded, else the
 * built-in analytical default. */
int32_t smla_decode_max_tokens(int32_t H, int32_t topk_total, int32_t format);

/* Replace the process-global crossover table with n entries (H, topk_total, format,
 * decode_max_tokens) given as 4*n host int32 values; n = 0 clears it. */
smla_status smla_set_crossover(const int32_t* entries, int32_t n);

/* Load a crossover table written by the calibration script: a JSON file holding
 * {"version": 1, "entries": [[H, topk_total, format, decode_max_tokens], ...]}. An
 * unknown version is treated as absent (the table is cleared, SMLA_ERR_UNSUPPORTED). */
smla_status smla_load_crossover(const char* json_path);

/* Human-readable name of a status. Never NULL. */
const char* smla_status_string(smla_status s);

/* Text of the last CUDA failure seen by a call on this host thread (the CUDA error name and
 * the step that failed), or "" if none. The pointer stays valid until the next call. */
const char* smla_last_error(void);

/* Reads and clears the device-side error word that kernels set when a bounded wait
 * gives up (0 = none). Synchronous: waits for the device. */
smla_status smla_device_error(int32_t* code);

/* Measurement hook: when both are non-NULL cudaEvent_t handles, the next calls record
 * `start` just before and `stop` just after the dominant kernel's launch on the call's
 * stream. Pass NULLs to disable. Process-global; meant for benchmarks. */
smla_status smla_set_timing_events(void* start_event, void* stop_event);

/* ABI self-check for foreign-language bindings: sizeof(smla_params) for which = 0,
 * sizeof(smla_kv_set) for which = 1, else 0. */
size_t smla_struct_size(int32_t which);

/* Library version, (major << 16) | minor. */
int32_t smla_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SMLA_H */
