/* Reference (oracle) for sparse top-k MLA attention — TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU implementation of what the CUDA library computes. Only the
 * tests, the package's smoke check and the benchmark's CPU-baseline leg may load it;
 * the product path never does. It shares no code, header or constant with the CUDA
 * library.
 *
 * Definition followed (DSv4 sparse MLA, pages: sglang PR "[SM12x] Drop the 64-head TP
 * pad on the DSv4 MLA prefill path", Problem section — all query heads share one latent
 * KV row per cached token; flashinfer PR "add topk=256 prefill-dsv4 dispatch",
 * Description — per-token index list of width topk over 64-token pages, plus an optional
 * second "extra" cache and index list; the same page's Correctness section of the sglang
 * PR — every (token, head) is computed independently; the attention sink is a per-head
 * logit checked against num_heads):
 *
 *   J(t)   = multiset of valid main entries and valid extra entries of token t
 *   x_j    = sm_scale * sum_c q[t,h,c] * K_j[c]             (c < 576)
 *   m      = max({x_j} U {sigma_h})      (sigma_h only when a sink is given)
 *   Z      = sum_j exp(x_j - m),   D = Z + exp(sigma_h - m)  (D = Z without sink)
 *   O[t,h] = sum_j exp(x_j - m) * V_j / D,   V_j = K_j[0:512]
 *   LSE    = m + log Z   (natural log; the sink is NOT included)
 *   J empty: O = 0, LSE = -inf.
 *
 * An entry idx[t, j] is valid iff j < topk (and j < topk_length[t] when given),
 * 0 <= idx < seq_lens[s], the page idx/64 is inside the block table row, and the
 * physical page block_table[s][idx/64] lies in [0, num_pages). s = token_seq[t] must lie
 * in [0, num_seqs); otherwise the token has no valid entries. Row r of physical page p
 * starts at byte p*page_stride + r*row_stride.
 *
 * Row formats: bf16 — 576 x bf16. fp8 — [512 x e4m3 (OCP E4M3FN)][4 x fp32 scale, one per
 * 128 latent channels][64 x bf16 rope]; K[c] = e4m3(byte c) * scale[c/128] for c < 512,
 * K[c] = bf16 rope for c >= 512; dequantisation is exact in fp64.
 */
#ifndef SMLA_ORACLE_H
#define SMLA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  const uint8_t* cache;       /* host bytes */
  int32_t fmt;                /* 0 = bf16 rows, 1 = fp8 rows */
  int64_t row_stride;         /* bytes */
  int64_t page_stride;        /* bytes */
  int32_t num_pages;
  const int32_t* block_table; /* [num_seqs, bt_stride] */
  int32_t bt_stride;
  const int32_t* seq_lens;    /* [num_seqs] */
  const int32_t* indices;     /* [T, idx_stride] */
  int64_t idx_stride;
  int32_t topk;
  const int32_t* topk_length; /* [T] or NULL */
} oracle_kvset;

typedef struct {
  int32_t T, H, num_seqs;
  const uint16_t* q;          /* bf16 bits, element (t,h,c) at q[t*q_stride_t + h*q_stride_h + c] */
  int64_t q_stride_t, q_stride_h;
  const int32_t* token_seq;   /* [T] */
  oracle_kvset main;
  const oracle_kvset* extra;  /* NULL when absent */
  const float* sink;          /* [H] logits or NULL */
  float sm_scale;
} oracle_problem;

/* Computes tokens tokens[0..n) (all T tokens when tokens == NULL, n ignored).
 * O: [n, H, 512] fp64, lse: [n, H] fp64. Returns 0, or -1 on a malformed problem. */
int oracle_attention(const oracle_problem* p, const int32_t* tokens, int32_t n, double* O,
                     double* lse, int32_t nthreads);

/* Cache writer: packs n rows of 576 values (x_dtype 0 = bf16 bits, 1 = fp32; row i at
 * element offset i*x_stride) into row bytes of format fmt (0 bf16: 1152 B, 1 fp8: 656 B),
 * written contiguously to out [n, row_bytes]. fp8 reading: per 128 latent channels
 * scale = fl32(amax/448) (1 if amax = 0), code = nearest E4M3FN to fl32(x/scale), ties to
 * even, saturating at 448; rope and bf16 rows: nearest bf16, ties to even.
 * Returns 0, or -1 on malformed arguments. */
int oracle_pack_rows(const void* x, int32_t x_dtype, int64_t x_stride, int32_t n, int32_t fmt, uint8_t* out);

/* Exact value of one OCP E4M3FN code (NaN for S.1111.111). */
double oracle_e4m3_value(uint8_t code);
/* Exact value of one bfloat16 bit pattern. */
double oracle_bf16_value(uint16_t bits);
/* Number of threads the oracle uses for a given request (0 = all hardware threads). */
int32_t oracle_threads(int32_t requested);

#ifdef __cplusplus
}
#endif
#endif
