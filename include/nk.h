/*
 * nk.h -- C ABI of the paged INT8 group-64 KV cache for one GB300 (sm_103a).
 *
 * Three operations, all enqueued on a caller-supplied CUDA stream:
 *   nk_kv_append          quantize new bf16 K/V rows into 64-channel int8 groups
 *                         and scatter them into pages ("NInfer-3090" README,
 *                         introduction: the kv_cache_append Op owns KV
 *                         quantization; "RotorQuant KV (rk8v4)": values are
 *                         stored from the represented bf16 source directly;
 *                         "NInfer" README, capability list: INT8 group-64 KV).
 *   nk_paged_decode_attn  GQA decode / small-T verify attention over the paged
 *                         cache, dequantizing inside the kernel, split over
 *                         pages and merged by a log-sum-exp combine
 *                         ("NInfer-3090" README, "Choosing a KV format":
 *                         attention re-reads the whole cache every step;
 *                         "Decode after the small-T kernels": a verify round
 *                         covers draft+1 token columns per sequence).
 *   nk_attn_combine       the log-sum-exp merge of split partial results, on
 *                         its own.
 * and two conveniences the pages have no counterpart for: nk_decode_step (a
 * step's append and attention in one call) and nk_paged_decode_attn_noalloc
 * (the attention with library-owned scratch).
 *
 * Every kernel is launched with programmatic stream serialization: it may
 * become resident while the previous kernel of the stream is still running,
 * and waits for it before touching memory that kernel could have written, so
 * the order of the stream is kept (calls can also be captured in a CUDA
 * graph).
 *
 * Conventions for every entry point
 *   - Pointers named *_dev are device pointers; everything else is host.
 *   - bf16 tensors are raw 16-bit bf16 bit patterns in device memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   - The library allocates no memory and never synchronizes (except
 *     nk_decode_step_host, the host-memory step, which waits for its stream).
 *     All buffers (pool, tables, Q, outputs, workspace, status word) belong
 *     to the caller.
 *   - Host-checkable argument errors return an NK_ERR_* code before anything
 *     is launched. Errors in device-resident data (a page id outside the
 *     pool, a position beyond the block table, ctx_len < T or > max_ctx) are
 *     reported by OR-ing NK_DEVFLAG_* bits into *status_dev (when it is not
 *     NULL); the affected unit is skipped and its output left unspecified.
 *     Nothing traps. A launch failure returns NK_ERR_CUDA.
 *
 * Quantization (one (token, kv-head, 64-channel group) at a time; the pages
 * name the format but not the rule, and this is the rule implemented):
 *   a = max |x|;  s = fp32(a / 127) (IEEE division), s = 1 when a = 0;
 *   q = clamp(round_half_even(fp32(x / s)), -127, 127).
 *
 * KV pool layout (one contiguous chunk per (page, kv-head), all offsets
 * multiples of 16 bytes):
 *   chunk = Kc[P][D] int8 | Ks[P][D/64] fp32 | Vc[P][D] int8 | Vs[P][D/64] fp32
 *   pool  = chunk[num_pages][num_kv_heads]
 * Position n of sequence b lives in page block_table[b][n / P], slot n % P.
 * At P = 64, D = 256 a chunk is 34,816 bytes (544 bytes per token and head).
 *
 * Attention semantics: Q is [B][T][Hq][D] bf16. ctx_len[b] counts every
 * token of sequence b including its T query tokens, whose K/V must already be
 * appended. Query column t (0-based) sees keys 0 .. ctx_len[b] - T + t; q-head
 * i reads kv-head i / (Hq / Hkv). Scores are sm_scale * q.k; the softmax and
 * LSE use natural exponentials. Output O is [B][T][Hq][D] bf16 (round to
 * nearest even).
 */
#ifndef NK_H
#define NK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NK_OK = 0,
  NK_ERR_NULL = 1,        /* a required pointer is NULL */
  NK_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
  NK_ERR_UNSUPPORTED = 3, /* a size the library has no kernel for */
  NK_ERR_WORKSPACE = 4,   /* the workspace is too small */
  NK_ERR_CUDA = 5,        /* a CUDA call failed (launch or attribute) */
  NK_ERR_DEVICE_DATA = 6, /* used by callers to report a nonzero status word */
  NK_ERR_TIMEOUT = 7      /* used by callers to report NK_DEVFLAG_TIMEOUT */
} nk_status;

/* Bits OR-ed into *status_dev by the kernels. */
#define NK_DEVFLAG_BAD_PAGE 0x1u    /* block-table entry outside [0, num_pages) */
#define NK_DEVFLAG_BAD_POS 0x2u     /* append position outside the block table */
#define NK_DEVFLAG_BAD_CTX 0x4u     /* ctx_len < T, > max_ctx or > table capacity */
#define NK_DEVFLAG_TIMEOUT 0x8u     /* a bounded wait on an async copy gave up */
#define NK_DEVFLAG_RANGE 0x10u      /* attention: an output is not finite (a true fp32
                                       overflow; the tensor-core kernels scale their fp16
                                       operands by powers of two, so no finite bf16 input
                                       leaves their range); rk8v4 append: a group scale
                                       saturated at the fp16 maximum, or a non-finite value */

/* Limits of the library. */
#define NK_GROUP 64      /* channels per quantization group */
#define NK_MAX_T 16      /* query tokens per sequence (decode + MTP verify) */
#define NK_MAX_HEAD_DIM 256

/* A KV pool: `base_dev` points at num_pages * num_kv_heads chunks laid out
 * as above (16-byte aligned; 1024-byte alignment is recommended). */
typedef struct nk_kv_pool {
  void* base_dev;
  int32_t num_pages;
  int32_t page_size;    /* P: multiple of 16, 16..256 */
  int32_t num_kv_heads; /* Hkv >= 1 */
  int32_t head_dim;     /* D: 64, 128 or 256 */
} nk_kv_pool;

/* Bytes of one (page, kv-head) chunk, and of a whole pool. 0 for bad sizes.
 * The pages size the INT8 cache per token ("NInfer-3090" README, "Choosing a
 * KV format": 33,792 bytes per token on the 27B model, 16 attention layers x 4
 * kv-heads x (2 x 256 codes + 2 x 4 two-byte scales)); this layout stores the
 * same codes with four-byte scales, 544 bytes per (token, kv-head) at D = 256
 * (2 x D codes + 2 x D/64 scales), and pads nothing. */
size_t nk_kv_chunk_bytes(int32_t page_size, int32_t head_dim);
size_t nk_kv_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim);

/*
 * nk_kv_append -- quantize and scatter new K/V rows.
 *   block_table_dev  int32 [B][max_pages_per_seq] physical page ids. Every
 *                    page a new position falls in must already be assigned.
 *   start_pos_dev    int32 [B]: position of sequence b's first new row.
 *   cu_new_dev       int32 [B+1]: new rows of sequence b are rows
 *                    cu_new[b] .. cu_new[b+1]-1 of k/v (cu_new[0] = 0,
 *                    cu_new[B] = total_new).
 *   k_dev, v_dev     bf16 [total_new][Hkv][D].
 * Writes codes and scales of every (row, kv-head) into the pool. Rows whose
 * position or page id is out of range are skipped and flagged. Two new rows
 * that map to the same slot race (undefined which one wins). Returns
 * NK_ERR_SHAPE when total_new * Hkv * D / 32 reaches 2^31.
 */
int nk_kv_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                 const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                 const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream);

/*
 * Work split of nk_paged_decode_attn (the pages describe no split; attention
 * re-reads the whole cache every step -- "NInfer-3090" README, "Choosing a KV
 * format" -- so the cache of one step is cut into page ranges that run in
 * parallel, flash-decoding style). The flat list of (sequence, kv-head, page)
 * items is cut into `num_splits` near-equal contiguous ranges, one per CTA;
 * each (CTA, (sequence, kv-head)) overlap produces one partial result, so
 * there are at most num_splits + B*Hkv - 1 partials. A "split" is one such CTA
 * range. num_splits <= 0 (the num_ctas argument of the calls below) picks the
 * default: a multiple of the device's SM count (of Hkv for one sequence),
 * capped by the number of items. Host arithmetic only; returns >= 1.
 * nk_decode_default_ctas is the same function under its earlier name.
 */
int32_t nk_decode_default_splits(int32_t B, int32_t num_kv_heads, int32_t max_ctx, int32_t page_size);
int32_t nk_decode_default_ctas(int32_t B, int32_t num_kv_heads, int32_t max_ctx, int32_t page_size);

/*
 * Workspace bytes nk_paged_decode_attn needs for this shape and split count
 * (num_splits <= 0: room for the default). The workspace is the pair of
 * split-partial arrays, back to back:
 *   part_o   fp32 [S][T*G][D]  at byte 0 (each partial normalized by its own
 *                              softmax sum),
 *   part_lse fp32 [S][T*G]     right after part_o (natural-log LSE of the
 *                              partial's scaled scores, -inf when empty),
 * with S = num_splits + B*Hkv partial slots and G = Hq / Hkv; the row of
 * query column t, q-head h*G + g is t*G + g. They are what nk_attn_combine
 * merges. The total is rounded up to 256 bytes. 0 for bad sizes.
 */
size_t nk_decode_workspace_bytes(int32_t B, int32_t T, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t num_splits);

/*
 * nk_paged_decode_attn -- split-KV GQA attention over the paged cache.
 *   q_dev          bf16 [B][T][Hq][D]
 *   ctx_lens_dev   int32 [B], each in [T, max_ctx]
 *   max_ctx        host-side upper bound of ctx_lens (sizes the work split)
 *   num_ctas       <= 0 for the default
 *   workspace_dev  nk_decode_workspace_bytes(...) bytes, 256-byte aligned;
 *                  scratch, contents on entry do not matter
 *   out_dev        bf16 [B][T][Hq][D]
 * Runs the split kernel (tensor-core path) and then the combine on `stream`.
 * T is 1 .. NK_MAX_T. When the G*T query rows of a kv-head do not fit one
 * split kernel -- more than 32 rows at head_dim 256 with 64-key pages, more
 * than 48 otherwise -- the columns run as consecutive chunks (at most 24
 * and 48 rows respectively), each a split kernel and a combine over the same
 * pages with its own causal limits. The workspace size for T covers every
 * chunk. A page too large for two stages of the kernels' shared-memory ring
 * (256-key pages at head_dim 256) returns NK_ERR_UNSUPPORTED before anything
 * is launched; nk_paged_decode_attn_simt takes pages of any size.
 * On the tcgen05 shapes, when a CTA may run more than 512 pages of one
 * kv-head (a caller-chosen split much coarser than the default, or under the
 * default split one sequence beyond about 1.2 million keys), the split
 * kernel runs an instance that folds its fp32 accumulators every 128 pages
 * (about 2% slower), so that coarse splits keep the accuracy of fine ones.
 * The mma.sync shapes (every other tensor-core shape, and the last chunk of
 * a chunked verify when it has too few rows for tcgen05) have no such
 * instance, and their error grows with the keys one CTA runs: a num_ctas
 * that could give one of their CTAs more than 262,144 keys of one kv-head
 * (4,096 pages of 64 keys) returns NK_ERR_UNSUPPORTED before anything is
 * launched. The default split reaches that only beyond about 10 million
 * keys per sequence; nk_paged_decode_attn_simt has no such limit.
 */
int nk_paged_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                         int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                         int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                         void* workspace_dev, size_t workspace_bytes, void* out_dev, int32_t* status_dev,
                         void* stream);

/*
 * nk_decode_step -- one decode (or verify) step: nk_kv_append of the step's
 * new rows followed by nk_paged_decode_attn, on `stream`, with the arguments
 * of those two calls (the block table is shared; B sequences in both). All
 * arguments of both are checked before anything is launched; the result is
 * bit-identical to the two calls in sequence. The attention's split kernel
 * reads the context lengths, block-table entries and Q while the append is
 * still running (the append writes only pool pages) and waits for it before
 * its first page load. The pages define the append and the attention; this
 * pairing of them has no counterpart there.
 */
int nk_decode_step(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                   const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t total_new, const void* k_dev,
                   const void* v_dev, const void* q_dev, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                   int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas, void* workspace_dev,
                   size_t workspace_bytes, void* out_dev, int32_t* status_dev, void* stream);

/*
 * nk_decode_step_host -- nk_decode_step from host memory, end to end: the
 * step's inputs are read from one host buffer in_host laid out by
 * nk_step_host_layout (pinned memory makes the transfer asynchronous),
 * copied in one transfer into the caller's device staging buffer staging_dev
 * (the same layout; 16-byte aligned), the step runs on `stream` exactly as
 * nk_decode_step with those device copies, and the B*T*num_q_heads*head_dim
 * bf16 output rows (written to out_dev) are copied to out_host, the status
 * word *status_dev (when both it and status_host are given) to *status_host.
 * The call then waits for the stream: this is the one entry point that
 * synchronizes. Arguments and checks as nk_decode_step; NK_ERR_NULL for a
 * missing in_host, staging_dev or out_host; a failed copy or wait returns
 * NK_ERR_CUDA. The pages have no counterpart; it is the step a serving loop
 * makes when its inputs live on the host.
 */
int nk_decode_step_host(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                        int32_t B, int32_t total_new, int32_t T, int32_t num_q_heads, float sm_scale,
                        int32_t max_ctx, int32_t num_ctas, const void* in_host, void* staging_dev,
                        void* workspace_dev, size_t workspace_bytes, void* out_dev, void* out_host,
                        int32_t* status_dev, int32_t* status_host, void* stream);

/* Layout of nk_decode_step_host's input buffer (host and device alike):
 * offsets[0] new K rows [total_new][num_kv_heads][head_dim] bf16,
 * offsets[1] new V rows (same), offsets[2] Q [B][T][num_q_heads][head_dim]
 * bf16, offsets[3] start_pos [B] int32, offsets[4] cu_new [B + 1] int32,
 * offsets[5] ctx_lens [B] int32; each region starts at a multiple of 256
 * bytes. Returns the total size in bytes (0 for an invalid shape). */
size_t nk_step_host_layout(int32_t B, int32_t total_new, int32_t T, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, size_t offsets[6]);

/* Same contract and result, computed by the fp32 CUDA-core kernel that the
 * tensor-core path is measured against. */
int nk_paged_decode_attn_simt(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                              int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                              int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                              void* workspace_dev, size_t workspace_bytes, void* out_dev,
                              int32_t* status_dev, void* stream);

/*
 * rk8v4 -- the "RotorQuant KV (rk8v4)" format of the "NInfer-3090" README:
 * keys rotated by R = H64 / 8 (64-point Sylvester Hadamard per 64-channel
 * group; R is orthonormal and its own inverse) and stored as INT8 group-64
 * codes; values stored unrotated as signed 4-bit codes (15 levels, -7..7),
 * two per byte, one scale per 32 channels; every scale fp16 (26,112 bytes
 * per token on the page's 27B model). Chunk per (page, kv-head):
 *   Kc[P][D] int8 | Ks[P][D/64] fp16 | Vc[P][D/2] uint8 | Vs[P][D/32] fp16
 * with channel 2j of a value row in the low nibble of byte j and 2j + 1 in
 * the high one; pool = [num_pages][num_kv_heads][chunk]. The same nk_kv_pool
 * struct describes an rk8v4 pool; its storage is sized with
 * nk_rk8v4_pool_bytes and only the nk_rk8v4_* calls may touch it.
 * Quantization (the readings where the page is silent):
 *   keys:   y = R k = RN_fp32(H64 k / 8): the exact sum of the 64 signed
 *           inputs, divided by 8 and rounded once to fp32 (ties to even);
 *           s = RN_fp16(max|y| / 127); q = clamp(rne(fp32(y / s)), -127, 127);
 *   values: s = RN_fp16(max|v| / 7);    q = clamp(rne(fp32(v / s)), -7, 7);
 *   a scale that rounds to 0 is stored as 1 (the codes are then 0); one past
 *   the fp16 maximum is stored as 65504 and sets NK_DEVFLAG_RANGE.
 */
size_t nk_rk8v4_chunk_bytes(int32_t page_size, int32_t head_dim);
size_t nk_rk8v4_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim);

/* kv_cache_append into an rk8v4 pool: arguments, checks, device flags,
 * ordering and ownership exactly as nk_kv_append. */
int nk_rk8v4_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                    const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                    const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream);

/* Split-KV decode / verify attention over an rk8v4 pool: arguments, checks,
 * workspace (nk_decode_workspace_bytes), causal mask, output and device
 * flags exactly as nk_paged_decode_attn. Each query row is rotated by R
 * inside the kernel and scored against the stored rotated keys
 * (q . k = (R q) . (R k)); values are dequantized as code * scale. Head dim
 * 128 or 256 with up to 32 query rows (G * T) per kv-head: tensor cores (the
 * rotated row as fp16 hi + lo against the INT8 key codes; the 4-bit value
 * codes widened exactly; a wider verify runs as column chunks of up to 32
 * rows). Other shapes: an fp32 CUDA-core kernel with G = Hq / Hkv <= 8 and
 * column chunks of 8. */
int nk_rk8v4_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                         int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                         int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas, void* workspace_dev,
                         size_t workspace_bytes, void* out_dev, int32_t* status_dev, void* stream);

/*
 * The pages' own INT8 layout and the unquantized bf16 baseline ("NInfer-3090"
 * README, "Choosing a KV format": int8 at 33,792 and bf16 at 65,536 bytes per
 * token on the 27B model, 16 attention layers x 4 kv-heads x 256 channels).
 * Chunks per (page, kv-head), pool = [num_pages][num_kv_heads][chunk]:
 *   int8 with fp16 scales (i8f16):
 *     Kc[P][D] int8 | Ks[P][D/64] fp16 | Vc[P][D] int8 | Vs[P][D/64] fp16
 *     (528 bytes per (token, kv-head) at D = 256: the page's 33,792 per token);
 *   bf16 (bf16kv): K[P][D] bf16 | V[P][D] bf16 (the page's 65,536 per token).
 * i8f16 quantization (the rule of the rk8v4 keys, without the rotation):
 *   s = RN_fp16(max|x| / 127), 1 when that is 0, 65504 past the fp16 maximum
 *   (NK_DEVFLAG_RANGE); q = clamp(round_half_even(fp32(x / s)), -127, 127).
 * bf16kv stores the rows as they are. The nk_kv_pool struct describes these
 * pools too; size them with their own *_pool_bytes, and only the calls of a
 * format may touch its pool.
 */
size_t nk_i8f16_chunk_bytes(int32_t page_size, int32_t head_dim);
size_t nk_i8f16_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim);
size_t nk_bf16kv_chunk_bytes(int32_t page_size, int32_t head_dim);
size_t nk_bf16kv_pool_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim);

/* kv_cache_append into an i8f16 or a bf16kv pool: arguments, checks, device
 * flags, ordering and ownership exactly as nk_kv_append. */
int nk_i8f16_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                    const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                    const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream);
int nk_bf16kv_append(const nk_kv_pool* pool, const int32_t* block_table_dev, int32_t max_pages_per_seq,
                     const int32_t* start_pos_dev, const int32_t* cu_new_dev, int32_t B, int32_t total_new,
                     const void* k_dev, const void* v_dev, int32_t* status_dev, void* stream);

/* Split-KV decode / verify attention over an i8f16 or a bf16kv pool:
 * arguments, checks, workspace (nk_decode_workspace_bytes), column chunks,
 * causal mask, output and device flags exactly as nk_paged_decode_attn, on the
 * same tensor-core kernels (i8f16: the tcgen05 and mma.sync kernels with fp16
 * scales). nk_bf16kv_decode_attn returns NK_ERR_UNSUPPORTED: its
 * kernel path (mma.sync with bf16 operands) is held back after a GPU fault at
 * the C1 decode size whose cause is not yet found. */
int nk_i8f16_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                         int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                         int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas, void* workspace_dev,
                         size_t workspace_bytes, void* out_dev, int32_t* status_dev, void* stream);
int nk_bf16kv_decode_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                          int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                          int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                          void* workspace_dev, size_t workspace_bytes, void* out_dev, int32_t* status_dev,
                          void* stream);

/*
 * nk_paged_decode_attn_noalloc -- nk_paged_decode_attn for callers that
 * cannot allocate device memory (the pages have no counterpart of this entry
 * point). Some callers cannot call cudaMalloc or pass a scratch buffer: hosts
 * that own a fixed device-memory budget and forbid allocation after start,
 * or code that must not risk the device synchronization an allocation can
 * bring. This variant keeps the split partials in a fixed array of
 * NK_NOALLOC_MAX_WORKSPACE bytes inside the library's device memory (held on
 * every GPU that loads the library, until the process exits) and calls no
 * allocator. The caller still provides q, the pool, the tables, out and the
 * optional status word; the arguments mean what they mean for
 * nk_paged_decode_attn.
 *   - The first call on a device looks up the array's device address once
 *     (cudaGetSymbolAddress) and keeps it until the process exits; make that
 *     first call before any stream capture. A call with B = 0 does only this
 *     set-up (nothing is launched, and the other arguments are not read), so
 *     it serves as the warm-up. Do not use the entry point on a device across
 *     a cudaDeviceReset of that device.
 *   - Returns NK_ERR_WORKSPACE when nk_decode_workspace_bytes() for this shape
 *     and CTA count exceeds NK_NOALLOC_MAX_WORKSPACE.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (no part of it needs to start at zero). Calls whose kernels
 *     overlap on the GPU race on it: serialize them (one stream, or events).
 */
#define NK_NOALLOC_MAX_WORKSPACE (8u << 20)
int nk_paged_decode_attn_noalloc(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                                 int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                                 int32_t num_q_heads, float sm_scale, int32_t max_ctx, int32_t num_ctas,
                                 void* out_dev, int32_t* status_dev, void* stream);

/*
 * nk_paged_prefill_attn -- chunked-prefill attention over the paged INT8
 * group-64 cache ("NInfer-4090" README, "What this fork changes": the INT8
 * attention prefill on the append shape, with causal key-block tiles; prefill
 * runs in chunks, "NInfer-3090" README, "Capabilities"). The T tokens of one
 * chunk per sequence -- T = 1,024 in the pages' chunked prefill, any T >= 1 --
 * attend to the cache exactly as nk_paged_decode_attn defines it: ctx_len[b]
 * counts the chunk's tokens, whose K/V the chunk's nk_kv_append already
 * stored, and token t sees keys 0 .. ctx_len[b] - T + t.
 *   q_dev    bf16 [B][T][Hq][D];  out_dev bf16 [B][T][Hq][D]
 * No workspace and no split: each CTA takes 128 query rows of one (sequence,
 * kv-head) over every key they see (mma.sync tensor cores; P a multiple of 16
 * whose page fits twice in shared memory). Checks, device flags, ordering and
 * ownership as nk_paged_decode_attn; NK_ERR_SHAPE when G * T or the grid
 * reaches 2^31.
 */
int nk_paged_prefill_attn(const nk_kv_pool* pool, const void* q_dev, const int32_t* block_table_dev,
                          int32_t max_pages_per_seq, const int32_t* ctx_lens_dev, int32_t B, int32_t T,
                          int32_t num_q_heads, float sm_scale, int32_t max_ctx, void* out_dev, int32_t* status_dev,
                          void* stream);

/*
 * nk_attn_combine -- log-sum-exp merge of S partial results. The pages give
 * attention over the whole cache ("NInfer-3090" README, "Choosing a KV
 * format") but no split or merge; this is the exact re-join of a softmax
 * computed over disjoint key ranges: with l_s the softmax sum of range s,
 * sum_s l_s O_s / sum_s l_s is the attention over the union, and
 * lse_s = m_s + ln l_s carries l_s up to a common factor.
 *   part_o_dev    fp32 [S][R][D]: each partial normalized by its own softmax sum
 *   part_lse_dev  fp32 [S][R]: natural-log LSE of the partial's scaled scores,
 *                 -inf for a partial that saw no key (weight 0)
 *   out_dev       bf16 [R][D] = sum_s w_s * O_s / sum_s w_s, w_s = exp(lse_s - max lse)
 * A row whose partials are all empty is written as zeros.
 */
int nk_attn_combine(const float* part_o_dev, const float* part_lse_dev, int32_t num_splits, int32_t rows,
                    int32_t head_dim, void* out_dev, void* stream);

/* Static string for an nk_status code. */
const char* nk_status_string(int code);

/* Library version as major*10000 + minor*100 + patch. */
int nk_version(void);

/*
 * nk_test_inject_copy_stall -- failure injection for tests of the bounded
 * waits (the pages have no counterpart; nothing here faults or traps). While
 * withheld_page >= 0, every tensor-core decode and prefill launched
 * afterwards by this process (nk_paged_decode_attn, nk_decode_step, the
 * no-alloc variant, the other formats' decodes, nk_paged_prefill_attn) never
 * issues the page copies of its CTA page numbers >= withheld_page, and bounds
 * each of its waits by wait_cycles SM clock cycles (0 keeps the default of
 * about 2 s). A wait for a withheld page runs out, sets NK_DEVFLAG_TIMEOUT in
 * the status word, and the kernel runs on without blocking, issues nothing
 * more, lets the copies and tensor-core work it did issue complete, and
 * returns; the outputs of the call are then unspecified and the device stays
 * usable. withheld_page < 0 switches it off. Process-wide, not thread-safe
 * against concurrent decode calls; for tests only.
 */
void nk_test_inject_copy_stall(int32_t withheld_page, uint64_t wait_cycles);

#ifdef __cplusplus
}
#endif
#endif /* NK_H */
