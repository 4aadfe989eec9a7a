/*
 * oracle.h -- slow, plain fp64 CPU oracle for the paged INT8 group-64 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The product path (the CUDA
 * library under quantized_paged_kv_cache_gb300/) never links, imports or calls
 * it, and shares no code, header, table or helper with it.
 *
 * What is computed (sources are the NInfer README pages):
 *   - INT8 group-64 KV storage: int8 codes with one scale per 64-channel group
 *     ("NInfer" README, capability list: "BF16 and INT8 group-64 KV cache";
 *     "NInfer-3090" README, "Choosing a KV format", int8 row).
 *   - kv_cache_append, the Op that owns KV quantization and stores values from
 *     the bf16 source directly ("NInfer-3090" README, introduction and
 *     "RotorQuant KV (rk8v4)").
 *   - Paged decode / MTP-verify attention that re-reads the whole cache each
 *     step ("NInfer-3090" README, "Choosing a KV format"; "Decode after the
 *     small-T kernels": a verify round covers draft+1 token columns).
 * The pages leave the quantizer's rounding rule, the scale type and the mask
 * among the T verify columns open; the readings taken here are:
 *   s = fp32(absmax / 127) (s = 1 when absmax = 0),
 *   q = clamp(round_half_even(fp32(x / s)), -127, 127),
 *   query column t of T sees keys 0 .. ctx_len - T + t (ctx_len counts the T
 *   new tokens, whose K/V are already in the cache).
 *
 * Pool layout (one contiguous chunk per (page, kv-head)):
 *   Kc[P][D] int8 | Ks[P][D/64] fp32 | Vc[P][D] int8 | Vs[P][D/64] fp32
 *   pool = [num_pages][num_kv_heads][chunk]
 * Tensors given to the oracle are host arrays; bf16 values are passed as their
 * raw uint16 bit patterns.
 *
 * The rk8v4 format (second section below) follows the same plan with its own
 * layout and readings.
 *
 * Parity status: every function here is pinned by tests in tests/test_oracle_*.py
 * against library routines, closed forms, invariants and hand-derived golden
 * cases (see the test files for which pin covers which function).
 */
#ifndef NK_ORACLE_H
#define NK_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exact widening of a bf16 bit pattern. */
double oracle_bf16_to_double(uint16_t bits);
/* Round a double to the nearest bf16, ties to even (overflow -> inf). */
uint16_t oracle_double_to_bf16(double x);
/* Round an array of doubles to bf16 bit patterns. */
void oracle_round_bf16(const double* x, size_t n, uint16_t* out);

/* Quantize one group of n bf16 values (n = 64 in the cache). Writes n int8
 * codes to q and returns the fp32 scale. */
float oracle_quantize_group(const uint16_t* x, int n, int8_t* q);

/* Bytes of one (page, kv-head) chunk and of the whole pool. */
size_t oracle_chunk_bytes(int page_size, int head_dim);
size_t oracle_pool_bytes(int num_pages, int page_size, int num_kv_heads, int head_dim);

/* kv_cache_append: quantize k/v rows [total_new][Hkv][D] (bf16 bits), laid out
 * sequence after sequence as given by cu_new[B+1], and write them at positions
 * start_pos[b] + j through block_table[b][max_pages]. Returns 0, or the number
 * of (token) units skipped because a position or page id was out of range. */
int oracle_kv_append(uint8_t* pool, int num_pages, int page_size, int num_kv_heads, int head_dim,
                     const int32_t* block_table, int max_pages, const int32_t* start_pos,
                     const int32_t* cu_new, int B, const uint16_t* k, const uint16_t* v);

/* Attention of one query row (b, t, q-head i) over the visible keys whose
 * position lies in [key_begin, key_end) (clipped to the causal limit).
 * Writes the normalized output o[D] (fp64) and the natural-log LSE of the
 * scaled scores. An empty range gives o = 0 and lse = -inf.
 * Returns 0, or nonzero on out-of-range data. */
int oracle_attention_row(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                         int head_dim, const int32_t* block_table, int max_pages,
                         const int32_t* ctx_lens, int B, int T, int num_q_heads,
                         const uint16_t* q, double sm_scale, int b, int t, int i,
                         int key_begin, int key_end, double* o, double* lse);

/* Full attention for every row: out[B][T][Hq][D] fp64 and lse[B][T][Hq]
 * (lse may be NULL). Returns 0 or the number of rows with bad data. */
int oracle_paged_attention(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                           int head_dim, const int32_t* block_table, int max_pages,
                           const int32_t* ctx_lens, int B, int T, int num_q_heads,
                           const uint16_t* q, double sm_scale, double* out, double* lse);

/* Log-sum-exp merge of S partial results: part_o[S][R][D] (normalized, fp32),
 * part_lse[S][R] (fp32, -inf for an empty split). out[R][D] fp64. */
void oracle_combine(const float* part_o, const float* part_lse, int S, int R, int D, double* out);

/* ---------------------------------------------------------------------------
 * rk8v4 ("NInfer-3090" README, "RotorQuant KV (rk8v4)"): keys rotated by the
 * 64-point Hadamard transform and stored as INT8 group-64 codes; values not
 * rotated, stored as signed 4-bit codes (15 levels), two per byte, one scale
 * per 32 channels; every scale fp16 (the section's 26,112 bytes per token on
 * the 27B model: 16 attention layers x 4 kv-heads x 408 bytes). Readings taken
 * where the section is silent:
 *   rotation R = H64 / 8 per 64-channel group (Sylvester order,
 *     H[i][j] = (-1)^popcount(i & j); orthonormal and its own inverse), so
 *     q . k = (R q) . (R k);
 *   at append R k is taken as its plain definition: every output is the
 *     exact sum of the 64 signed inputs divided by 8, rounded once to fp32
 *     (round to nearest, ties to even; past the fp32 range it is infinite);
 *     inputs are finite bf16 values;
 *   key scale  s = RN_fp16(absmax(R k) / 127), value scale s = RN_fp16(absmax(v) / 7);
 *     s = 1 when it rounds to 0 (absmax = 0 or below the fp16 range), and
 *     s = 65504 when it rounds past the fp16 maximum;
 *   codes q = clamp(round_half_even(fp32(x / s)), -127, 127) for keys and
 *     [-7, 7] for values; byte j of a value group holds element 2j in its low
 *     nibble and 2j + 1 in its high nibble (two's complement);
 *   attention rotates each query row by R (fp64 here) and scores it against
 *     the dequantized rotated keys; values are dequantized as q * s.
 * Pool layout (one contiguous chunk per (page, kv-head)):
 *   Kc[P][D] int8 | Ks[P][D/64] fp16 | Vc[P][D/2] uint8 | Vs[P][D/32] fp16
 * ------------------------------------------------------------------------- */

/* Round a double to the nearest fp16, ties to even (overflow -> inf); the bits. */
uint16_t oracle_double_to_f16(double x);
/* Exact widening of an fp16 bit pattern. */
double oracle_f16_to_double(uint16_t bits);
/* R x of one 64-channel group of bf16 values: RN_fp32 of the exact H64 x / 8. */
void oracle_rk_rotate64(const uint16_t* x, float* y);
/* Key group: 64 rotated fp32 values -> 64 codes; returns the fp16 scale bits. */
uint16_t oracle_rk_quantize_k(const float* y, int8_t* q);
/* Value group: 32 bf16 values -> 16 packed bytes; returns the fp16 scale bits. */
uint16_t oracle_rk_quantize_v(const uint16_t* x, uint8_t* packed);

size_t oracle_rk_chunk_bytes(int page_size, int head_dim);
size_t oracle_rk_pool_bytes(int num_pages, int page_size, int num_kv_heads, int head_dim);

/* kv_cache_append into an rk8v4 pool; arguments and result as oracle_kv_append. */
int oracle_rk_append(uint8_t* pool, int num_pages, int page_size, int num_kv_heads, int head_dim,
                     const int32_t* block_table, int max_pages, const int32_t* start_pos,
                     const int32_t* cu_new, int B, const uint16_t* k, const uint16_t* v);

/* Attention over an rk8v4 pool; arguments and results as oracle_attention_row
 * and oracle_paged_attention. */
int oracle_rk_attention_row(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                            int head_dim, const int32_t* block_table, int max_pages,
                            const int32_t* ctx_lens, int B, int T, int num_q_heads,
                            const uint16_t* q, double sm_scale, int b, int t, int i,
                            int key_begin, int key_end, double* o, double* lse);
int oracle_rk_paged_attention(const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                              int head_dim, const int32_t* block_table, int max_pages,
                              const int32_t* ctx_lens, int B, int T, int num_q_heads,
                              const uint16_t* q, double sm_scale, double* out, double* lse);

/* ---------------------------------------------------------------------------
 * The pages' own INT8 layout ("NInfer-3090" README, "Choosing a KV format":
 * int8 at 33,792 bytes per token on the 27B model = 16 layers x 4 kv-heads x
 * (2 x 256 codes + 2 x 4 two-byte scales)): INT8 group-64 codes for K and V
 * with fp16 scales, no rotation. Readings: s = RN_fp16(absmax / 127), 1 when
 * that is 0 and 65504 past the fp16 maximum (as rk8v4's keys);
 * q = clamp(round_half_even(fp32(x / s)), -127, 127).
 * Chunk per (page, kv-head): Kc[P][D] int8 | Ks[P][D/64] fp16 | Vc[P][D] int8 | Vs[P][D/64] fp16
 *
 * And the unquantized baseline the same table lists (bf16, 65,536 bytes per
 * token): chunk per (page, kv-head) K[P][D] bf16 | V[P][D] bf16.
 * ------------------------------------------------------------------------- */

/* One group of 64 bf16 values -> 64 codes; returns the fp16 scale bits. */
uint16_t oracle_i8h_quantize_group(const uint16_t* x, int8_t* q);
size_t oracle_i8h_chunk_bytes(int page_size, int head_dim);
size_t oracle_bf16kv_chunk_bytes(int page_size, int head_dim);

/* kv_cache_append into a pool of the given format (1 = INT8 with fp16
 * scales, 2 = bf16); arguments and result as oracle_kv_append. */
int oracle_fmt_append(int fmt, uint8_t* pool, int num_pages, int page_size, int num_kv_heads, int head_dim,
                      const int32_t* block_table, int max_pages, const int32_t* start_pos,
                      const int32_t* cu_new, int B, const uint16_t* k, const uint16_t* v);

/* Attention over a pool of the given format (1 or 2); arguments and results
 * as oracle_paged_attention. */
int oracle_fmt_paged_attention(int fmt, const uint8_t* pool, int num_pages, int page_size, int num_kv_heads,
                               int head_dim, const int32_t* block_table, int max_pages,
                               const int32_t* ctx_lens, int B, int T, int num_q_heads,
                               const uint16_t* q, double sm_scale, double* out, double* lse);

/* Threads the oracle's parallel loops use. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
