/*
 * pkv.h -- C ABI of libpkv: paged-KV decode attention for GB300 (sm_103a).
 *
 * The library implements the decode-step hot path of a small Llama-3.2-1B
 * serving engine as described in the samir-vllm README summary
 * ("从零用 C++ 和 CUDA 实现 Llama 3.2 1B 推理引擎:6 小时视频与 85 页手写笔记",
 * section "目前已完成的功能", features done so far):
 *   - a shared BF16 KV page pool; each physical page holds K and V of 16
 *     tokens; every (sequence, layer) reaches its pages through a block table;
 *     the number of requests does not grow the pool;
 *   - decode appends one new token per sequence at its absolute RoPE position;
 *   - paged decode attention: each query head streams its sequence's cached
 *     pages with an FP32 online softmax, without gathering a contiguous prefix
 *     and without storing attention scores;
 * plus, from the same page's section "当前范围" (current scope), pages that are
 * allocated lazily and returned when a request finishes.
 *
 * Geometry supported by the kernels (Llama-3.2-1B attention): 32 query heads,
 * 8 KV heads (grouped-query attention, group 4, query head h reads KV head
 * h / 4), head_dim 64, 16 tokens per page.
 *
 * Memory layout (a reading: the pages fix no in-page layout):
 *   pool slab   : num_pages pages, page p at  slab + p * PKV_PAGE_BYTES;
 *   one page    : [2: K then V][8 KV heads][16 slots][64 dims] BF16 (32 KiB);
 *                 the K tile of (page, head) is one contiguous 2 KiB run, its
 *                 V tile another 2 KiB run 16 KiB further on;
 *   block table : int32 [B][max_blocks] per layer; entry j of row b is the
 *                 physical page holding tokens 16j .. 16j+15 of sequence b;
 *                 unused entries are -1;
 *   q, out      : BF16 [B][32][64];  k_new, v_new : BF16 [B][8][64];
 *   seq_lens    : int32 [B], the length AFTER this step's append (the new
 *                 token sits at position seq_len - 1 and attends to itself);
 *   pos         : int32 [B], the absolute position of the appended token.
 * BF16 values travel as uint16_t bit patterns.
 *
 * Ownership: the caller owns every device buffer (slab, q, k_new, v_new,
 * tables, lengths, workspace, out, error flag); the library owns only the
 * host-side pkv_pool object (free list and bookkeeping) and never frees the
 * slab.  Kernel launches are asynchronous on the caller's stream
 * (cudaStream_t passed as void*, NULL = legacy default stream).
 *
 * Errors: every entry point returns a status code synchronously after host
 * checks (PKV_OK = 0, negative on error; nothing is launched on error).
 * Faults the host cannot see (a block-table entry outside the pool, a length
 * beyond the table) are caught by the kernels' own bounds checks: the unit is
 * skipped, its outputs are written as zeros, and a bit is OR-ed into the
 * caller's int32 device error flag; kernels never trap.  Read it with
 * pkv_check_device_error().
 *
 * Thread safety: a pkv_pool is not thread-safe; calls on distinct pools are.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- constants */
#define PKV_PAGE_SIZE 16
#define PKV_NUM_Q_HEADS 32
#define PKV_NUM_KV_HEADS 8
#define PKV_HEAD_DIM 64
#define PKV_PAGE_BYTES (2 * PKV_NUM_KV_HEADS * PKV_PAGE_SIZE * PKV_HEAD_DIM * 2) /* 32768 */

/* status codes */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1)         /* null pointer, size or shape out of range */
#define PKV_ERR_OUT_OF_PAGES (-2)        /* allocation larger than the free list (nothing taken) */
#define PKV_ERR_DOUBLE_FREE (-3)         /* freeing a page that is not allocated */
#define PKV_ERR_CUDA (-4)                /* a CUDA runtime / launch error */
#define PKV_ERR_DEVICE_BOUNDS (-5)       /* the device error flag was set */
#define PKV_ERR_BUDGET_EXCEEDS_POOL (-6) /* a request larger than the whole pool */
#define PKV_ERR_UNSUPPORTED (-7)         /* geometry other than 32/8/64/16 */
#define PKV_ERR_WORKSPACE_TOO_SMALL (-8)

/* device error-flag bits (OR-ed by kernels into the caller's int32 flag) */
#define PKV_DEVERR_PAGE_RANGE 0x1  /* a block-table entry outside [0, num_pages) */
#define PKV_DEVERR_LENGTH 0x2      /* seq_len < 1, seq_len > max_blocks*16, or pos out of range */
#define PKV_DEVERR_TIMEOUT 0x4     /* a bounded wait on a copy barrier gave up */

/* decode kernel variants (pkv_decode_attention_variant) */
#define PKV_DECODE_DEFAULT 0 /* the fastest measured variant */
#define PKV_DECODE_SIMT 1    /* CUDA-core FP32 dot products and warp-shuffle reductions */
#define PKV_DECODE_MMA 2     /* warp-level BF16 tensor-core MMA for the 16-token page tiles */

typedef struct pkv_pool pkv_pool; /* opaque, host side */

/* ------------------------------------------------------------------- pool */

/* Create the host-side manager of a caller-owned device slab.
 * Source: samir-vllm README summary, "目前已完成的功能" (shared BF16 KV page
 * pool of 16-token pages) and "从零构建大模型推理引擎" section 5.1 (preallocate
 * one large buffer and manage it by offsets).
 *   dev_slab     device pointer, at least 16-byte aligned (checked; cudaMalloc
 *                and torch give 256), never freed by the library
 *   slab_bytes   size; num_pages = slab_bytes / PKV_PAGE_BYTES (>= 1)
 *   page_size, num_kv_heads, head_dim  must be 16, 8, 64 (else PKV_ERR_UNSUPPORTED)
 *   seed         seeds the shuffle of the free list, so pages handed out are
 *                scattered through the slab reproducibly
 *   out          receives the pool object
 * Host only: no CUDA call is made. */
int pkv_pool_create(void *dev_slab, size_t slab_bytes, int page_size, int num_kv_heads, int head_dim,
                    uint64_t seed, pkv_pool **out);

/* KV storage formats of a pool */
#define PKV_KV_BF16 0
#define PKV_KV_FP8 1 /* FP8 E4M3 codes + one FP32 scale per (token, KV head) row */
#define PKV_PAGE_BYTES_FP8 (2 * PKV_NUM_KV_HEADS * PKV_PAGE_SIZE * (PKV_HEAD_DIM + 4)) /* 17408 */

/* As pkv_pool_create, for a pool of FP8 pages ("从零构建大模型推理引擎：KV缓存、算子融合与量化优化实战",
 * section 5.1:
 * keep the KV cache in low precision and dequantize before attention; the scheme
 * is this library's reading).  A page is 17408 bytes: 8 units of 2176 bytes, one
 * per KV head, each the K codes [16 slots][64 dims], the V codes (1024 bytes: slots
 * 2p and 2p+1 share line p of 128 bytes, in which dims 8c..8c+7 of both form 16-byte
 * chunk c -- byte 2 (dim % 8) + slot % 2 -- stored at chunk position c XOR (2p mod 8))
 * and the row scales [2 (K,V)][16] FP32; codes are E4M3 without infinities (largest
 * 448), one byte each.  One (page, KV head) is one contiguous copy.  A row of 64 values x is stored
 * as scale = amax|x| / 448 (FP32; 1 for an all-zero row) and codes
 * E4M3_rne_satfinite(x / scale) (FP32 division); x is the BF16 value the BF16 path
 * would store (the rotated key, or the value).  Every entry point below accepts
 * an FP8 pool: appends and prefills quantize, attention dequantizes (codes are
 * exact in FP16; K scales multiply the scores, V scales the softmax weights).
 * The SIMT decode variant is not provided for FP8 (PKV_ERR_UNSUPPORTED). */
int pkv_pool_create_fp8(void *dev_slab, size_t slab_bytes, uint64_t seed, pkv_pool **out);

/* The pool's KV format (PKV_KV_BF16 or PKV_KV_FP8), or a negative status. */
int pkv_pool_kv_format(const pkv_pool *pool);

/* Destroy the host object (never touches the slab).  NULL is accepted. */
int pkv_pool_destroy(pkv_pool *pool);

/* Take n pages, all or nothing (samir-vllm README summary, "当前范围": pages are
 * allocated lazily, on demand).  ids_out receives n int32 page ids.
 * PKV_ERR_OUT_OF_PAGES if fewer than n are free (nothing is taken). */
int pkv_pool_alloc(pkv_pool *pool, int n, int32_t *ids_out);

/* Return n pages (same section: pages come back when a request finishes or
 * stops early).  All ids are checked first: an id outside the pool is
 * PKV_ERR_INVALID_ARG, an id not currently allocated (or repeated in the call)
 * is PKV_ERR_DOUBLE_FREE; on error nothing is freed. */
int pkv_pool_free(pkv_pool *pool, int n, const int32_t *ids);

/* Report the slab's K base, V base (= K base + 16 KiB; FP8 pools: head 0's V
 * codes, K base + 1 KiB, with the heads' units 2176 bytes apart), page stride in
 * bytes (32768; FP8 pools 17408), page count and free-page count.  Any output
 * pointer may be NULL. */
int pkv_pool_info(const pkv_pool *pool, void **k_base, void **v_base, int64_t *page_stride_bytes,
                  int *num_pages, int *num_free);

/* Build block tables for `layers` layers and B sequences on the host (samir-
 * vllm README summary, "目前已完成的功能": block tables per sequence and layer).
 * For every (layer l, sequence b) it takes ceil(seq_lens[b]/16) pages from the
 * free list and writes them to bt_host[l][b][0..], padding with -1 up to
 * max_blocks.  All or nothing: PKV_ERR_OUT_OF_PAGES if the total does not fit,
 * PKV_ERR_INVALID_ARG if a length is negative or needs more than max_blocks
 * pages.  A length of 0 takes no pages.  Host only. */
int pkv_block_tables_build(pkv_pool *pool, int layers, int B, const int32_t *seq_lens, int max_blocks,
                           int32_t *bt_host);

/* ------------------------------------------------------------------- RoPE */

/* Bytes of the rotary-embedding table of pkv_rope_table_init: max_pos x half_dim
 * entries of 4 floats (16 bytes); 0 for max_pos < 1 or half_dim other than 32. */
size_t pkv_rope_table_bytes(int max_pos, int half_dim);

/* Fill a device table of rotary-embedding factors ("从零构建大模型推理引擎" section 4.1:
 * rotary embedding injects the absolute position; the samir-vllm page's RoPE item).
 * Entry (p, i) holds c = cos(p * theta^(-2i/(2*half_dim))) and s = sin(...), computed
 * on the host in FP64, each as two FP32 parts: {c_hi, s_hi, c_lo, s_lo} with c_hi the
 * FP32 nearest c and c_lo the FP32 nearest c - c_hi (about 48 bits together).  The
 * kernels rotate with both parts and error-free products, so a rotated value rounds to
 * the BF16 nearest the exact rotation even where its two products nearly cancel.  The
 * pairing is rotate-half: dimension i turns with dimension i + half_dim.
 *   theta      base (500000 for Llama 3.2); half_dim must be 32
 *   max_pos    rows; positions 0 .. max_pos-1 (2048 for the engine's context)
 *   dev_cos_sin device buffer of pkv_rope_table_bytes(max_pos, half_dim) bytes
 *              (max_pos * half_dim * 4 floats), 16-byte aligned
 * Copies synchronously with respect to the host (the stream is synchronised). */
int pkv_rope_table_init(double theta, int max_pos, int half_dim, float *dev_cos_sin, void *cuda_stream);

/* ----------------------------------------------------------------- append */

/* Fused RoPE + page-slot append for one layer (samir-vllm README summary,
 * "目前已完成的功能": decode appends one token at its absolute RoPE position).
 * For every sequence b with p = pos_dev[b]: rotate k_new[b][g] to position p
 * (FP32 arithmetic on the table's factors, rounded to BF16 to nearest even)
 * and store it, with v_new[b][g] unrotated, into page bt_dev[b][p/16], slot
 * p%16, for the 8 KV heads g.  If q is not NULL, the 32 query heads of q[b]
 * are rotated in place by the same factors.
 *   bt_dev     this layer's table [B][max_blocks]
 *   rope_table from pkv_rope_table_init with max_pos rows
 *   dev_err_flag int32 device flag (may be NULL: errors are then only skipped)
 * Device checks: pos outside [0, min(max_pos, 16*max_blocks)) or a page id
 * outside the pool sets the flag and skips that sequence. */
int pkv_append_rope(const pkv_pool *pool, const uint16_t *k_new, const uint16_t *v_new, uint16_t *q,
                    const int32_t *bt_dev, int max_blocks, const int32_t *pos_dev, int B,
                    const float *rope_table, int max_pos, int32_t *dev_err_flag, void *cuda_stream);

/* ---------------------------------------------------------------- decode */

/* Bytes of device workspace pkv_decode_attention (and pkv_decode_step) needs for
 * B sequences, a table width of max_blocks and pages_per_chunk pages per work
 * unit: per-(sequence, KV head) merge counters [B][8] int32, then the chunk
 * partials (m, l) [B][32][chunks] and o [B][32][chunks][64] FP32, chunks =
 * ceil(max_blocks / pages_per_chunk), each region 256-byte aligned.  0 for
 * arguments below 1. */
size_t pkv_decode_workspace_bytes(int B, int max_blocks, int pages_per_chunk);

/* Paged decode attention for one layer (samir-vllm README summary, "目前已完成
 * 的功能": each query head streams its sequence's cached pages with an FP32
 * online softmax and accumulates weighted V, no contiguous gather, no stored
 * scores; "从零构建大模型推理引擎" section 3.2: scores q.k / sqrt(head_dim), the
 * maximum subtracted before the exponential).
 * For each sequence b and query head h (KV head h/4):
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . K_t) V_t,  t < seq_lens[b],
 * K_t, V_t read from page bt_dev[b][t/16], slot t%16.  The result is rounded to
 * BF16 (nearest even).
 * Work split: a sequence's pages are cut into chunks of pages_per_chunk pages
 * (1..128); one CTA handles one (sequence, KV head, chunk) and serves all 4
 * query heads of the group from a single read of each page; chunk partials
 * (running max, sum, unnormalised output in FP32) are merged by log-sum-exp in
 * chunk order, inside the same launch: the CTA that finishes a (sequence, KV
 * head) last merges it.
 * The chunking depends only on each sequence's own length and pages_per_chunk,
 * never on B, so a sequence's result is bit-identical alone or in any batch.
 *   workspace  device buffer of at least pkv_decode_workspace_bytes(...) bytes,
 *              16-byte aligned (may be NULL when every sequence fits one chunk,
 *              i.e. max_blocks <= pages_per_chunk).  Its counter region (the
 *              first B*8 int32) must be zero before the FIRST call -- e.g. one
 *              cudaMemset after allocating; every call leaves it zero again.
 *              Calls sharing a workspace must not overlap on the GPU.
 *   scale      1/sqrt(64) = 0.125 for the engine
 * Launch: programmatic dependent launch.  Before its dependency wait a CTA reads
 * only seq_lens, bt_dev and the cached pages holding no position at or beyond
 * seq_len - 2; q, the two last positions' pages and every output come after it.
 * So the kernel immediately before this call on the stream may write q (e.g. a
 * projection) and positions seq_len - 1 and seq_len - 2 (the append of this step,
 * pkv_append_rope at pos = seq_len - 1, or of the previous step), but must not
 * write seq_lens, bt_dev or any earlier position of these sequences' pages.  A
 * pkv_prefill_append on the same pool makes the next decode launch on the pool go
 * without programmatic dependent launch.
 * Device checks: seq_len outside [1, 16*max_blocks] or a page id outside the
 * pool sets the flag; the affected (sequence, head) outputs are zeros. */
int pkv_decode_attention(const pkv_pool *pool, const uint16_t *q, const int32_t *bt_dev, int max_blocks,
                         const int32_t *seq_lens_dev, int B, float scale, int pages_per_chunk,
                         void *workspace, size_t workspace_bytes, uint16_t *out, int32_t *dev_err_flag,
                         void *cuda_stream);

/* The two-kernel form of pkv_decode_attention (option bit of
 * pkv_decode_attention_variant): the split kernel writes every chunk's partial to
 * the workspace and a second small kernel merges them by log-sum-exp.  Launched
 * without programmatic dependent launch; the workspace needs no initialisation
 * (its counter region is not used).  Results are bit-identical to the default
 * form's: the merge does the same arithmetic in the same chunk order. */
#define PKV_DECODE_SPLIT_MERGE 0x80000

/* As pkv_decode_attention, with the page policy chosen explicitly in the low byte
 * of `variant` (PKV_DECODE_DEFAULT, PKV_DECODE_SIMT or PKV_DECODE_MMA), OR-ed with
 * launch options: PKV_STEP_NO_PDL, PKV_STEP_RING(n), PKV_STEP_SORTED and
 * PKV_STEP_TEST_EXPIRE_WAIT as for pkv_decode_step, or PKV_DECODE_SPLIT_MERGE alone
 * (the two-kernel form; no other option with it).  None of the options changes a
 * result bit.  Unknown bits: PKV_ERR_INVALID_ARG. */
int pkv_decode_attention_variant(const pkv_pool *pool, const uint16_t *q, const int32_t *bt_dev,
                                 int max_blocks, const int32_t *seq_lens_dev, int B, float scale,
                                 int pages_per_chunk, void *workspace, size_t workspace_bytes, uint16_t *out,
                                 int32_t *dev_err_flag, void *cuda_stream, int variant);

/* -------------------------------------------------------------- scheduler */

/* Request scheduler over a page pool (samir-vllm README summary, "当前范围"):
 * admission by page budget -- a request reserves prompt + allowed_new - 1 tokens,
 * rounded up to 16-token pages in each layer, as credits separate from physical
 * pages; allowed_new is capped so that prefix stays within the context -- FIFO
 * waiting, rejection of budgets larger than the whole pool, lazy page allocation,
 * pages and credits returned on finish or early stop, no preemption.  Continuous
 * batching admits whenever credits allow; static batching admits the next group
 * only after the current one has finished ("构建": --static / --continuous).
 * Host only (no CUDA call).  The scheduler assumes it owns the pool's pages that
 * are free when it is created (their number is the credit total); every page it
 * hands out belongs to exactly one (request, layer).  Not thread-safe. */
typedef struct pkv_sched pkv_sched;

#define PKV_SCHED_CONTINUOUS 0
#define PKV_SCHED_STATIC 1

typedef struct pkv_sched_stats {
    int64_t pool_pages;           /* pages in the pool */
    int64_t peak_active;          /* most requests active at once */
    int64_t max_decode_batch;     /* largest decode batch */
    int64_t peak_allocated_pages; /* most physical pages held at once */
    int64_t admission_waits;      /* admission rounds in which the FIFO head had to wait for credits */
    int64_t final_free_pages;     /* pages free in the pool now */
    int64_t submitted, admitted, finished, rejected;
    int64_t active, waiting, allocated_pages, free_credits; /* current state */
} pkv_sched_stats;

/* layers: layers per request (16); max_blocks: table width (128); max_context:
 * context cap in tokens (2048, at most 16*max_blocks); max_batch: decode batch cap;
 * mode: PKV_SCHED_CONTINUOUS or PKV_SCHED_STATIC. */
int pkv_sched_create(pkv_pool *pool, int layers, int max_blocks, int max_context, int max_batch, int mode,
                     pkv_sched **out);
/* Frees the pages of requests still active. */
int pkv_sched_destroy(pkv_sched *sched);
/* Queue a request.  PKV_ERR_BUDGET_EXCEEDS_POOL if its budget exceeds every credit
 * (it could never run); PKV_ERR_INVALID_ARG for prompt < 1, prompt > max_context,
 * max_new < 1 or a duplicate id. */
int pkv_sched_submit(pkv_sched *sched, int64_t id, int prompt_tokens, int max_new_tokens);
/* Admit waiting requests in FIFO order while credits and the batch cap allow (at
 * most max_n).  For each: its id, prompt length and block-table rows
 * bt_rows_out[i][layers][max_blocks] holding the pages of its prompt (allocated
 * now), for the caller's prefill.  *n_out = number admitted.  The credits are the
 * pool's free pages when the scheduler was created; if pages were taken from the
 * pool outside the scheduler since, a head whose prompt pages are not all free keeps
 * waiting (counted in admission_waits) and nothing of it is allocated. */
int pkv_sched_admit(pkv_sched *sched, int max_n, int64_t *ids_out, int32_t *prompt_lens_out, int32_t *bt_rows_out,
                    int *n_out);
/* Next decode step: retire requests whose last step has run, then append one token
 * to every active request (taking a new page per layer when it crosses a page
 * boundary) and return the batch: ids_out[B], seq_lens_out[B] (lengths after the
 * append) and bt_out[layers][B][max_blocks].  max_b bounds B.  PKV_ERR_OUT_OF_PAGES
 * only if pages were taken from the pool outside the scheduler: then no request
 * advances (pages already taken for this step stay with their requests) and the
 * call can be repeated once pages are back. */
int pkv_sched_decode_batch(pkv_sched *sched, int max_b, int64_t *ids_out, int32_t *seq_lens_out, int32_t *bt_out,
                           int *B_out);
/* Early stop (e.g. an end-of-sequence token): free the request's pages and credits
 * now, or drop it from the queue. */
int pkv_sched_finish(pkv_sched *sched, int64_t id);
int pkv_sched_get_stats(const pkv_sched *sched, pkv_sched_stats *out);

/* ------------------------------------------------------------ prefill fill */

/* Write T consecutive tokens of ONE sequence into its pages, for `layers` layers:
 * token t goes to position start_pos + t, its key rotated to that position exactly
 * as pkv_append_rope rotates the decode token (samir-vllm README summary, "目前已完成
 * 的功能": prefill fills the prompt's pages; decode appends at the absolute RoPE
 * position).  k, v: [layers][T][8][64] BF16; bt_rows: device [layers][max_blocks]
 * (this sequence's table in every layer).  Device checks: a position beyond the
 * table or max_pos, or a page id outside the pool, sets the flag and skips it.
 * The next pkv_decode_step / pkv_decode_attention launch on this pool goes without
 * programmatic dependent launch, because it may read these pages. */
int pkv_prefill_append(const pkv_pool *pool, const uint16_t *k, const uint16_t *v, const int32_t *bt_rows,
                       int max_blocks, int layers, int start_pos, int T, const float *rope_table, int max_pos,
                       int32_t *dev_err_flag, void *cuda_stream);

/* ------------------------------------------------------ fused decode step */

/* option bits for pkv_decode_step (and pkv_decode_attention_variant) */
#define PKV_STEP_NO_PDL 0x100 /* launch without programmatic dependent launch */
#define PKV_STEP_GRID 0x200   /* one CTA per (sequence, KV head, chunk): the only schedule, accepted for clarity */
/* TMA ring depth per warp, 2..4 stages (0 = library default: 3 for pages_per_chunk
 * >= 64, else 2).  A stage is 4 KiB for BF16 pages, one 2176-byte unit for FP8 pages.
 * Fewer stages mean less shared memory per CTA and more CTAs resident per SM. */
#define PKV_STEP_RING(n) ((n) << 12)
#define PKV_STEP_RING_MASK 0xf000
/* Dispatch the work units largest first (page count, then sequence, chunk, KV head)
 * instead of in (KV head, sequence, chunk) order.  The block scheduler places CTAs in
 * index order wherever there is room, so the largest units start first and small ones
 * fill the gaps, which balances the SMs when a ragged batch fits in one wave.  Which
 * CTA computes which unit is all that changes: results are identical.  B <= 1024
 * (PKV_ERR_INVALID_ARG beyond). */
#define PKV_STEP_SORTED 0x20000
/* Testing aid for the bounded waits: the first wait for a page copy in every work unit
 * of sequence 0 gives up without polling, as a wait that ran out of its iteration
 * limit does.  The unit then waits (bounded) for its copies in flight -- they are
 * copies of valid pages, so they land -- sets PKV_DEVERR_TIMEOUT in the error flag and
 * finishes: sequence 0's outputs are undefined, every other sequence's are computed as
 * usual, and the merge counters are left at zero.  No copy stalls and nothing faults. */
#define PKV_STEP_TEST_EXPIRE_WAIT 0x40000

/* Bytes of device workspace pkv_decode_step needs: pkv_decode_workspace_bytes. */
size_t pkv_decode_step_workspace_bytes(int B, int max_blocks, int pages_per_chunk);

/* One layer of the decode step in ONE kernel launch: pkv_append_rope with
 * pos = seq_lens - 1 (q rotated in place, the new key rotated and stored with its
 * value into page bt_dev[b][pos/16], slot pos%16) followed by
 * pkv_decode_attention -- the two steps the samir-vllm README summary lists in
 * "目前已完成的功能" (append at the absolute RoPE position; paged decode
 * attention with an FP32 online softmax).  Results are bit-identical to the two
 * separate calls with the same variant and pages_per_chunk.
 *   k_new, v_new [B][8][64] BF16; q [B][32][64] BF16, required, rotated in place;
 *   rope_table / max_pos as for pkv_append_rope (seq_lens[b] <= max_pos);
 *   workspace  >= pkv_decode_step_workspace_bytes(...) bytes, 16-byte aligned.
 *              Its counter region must be zero before the FIRST call (e.g. one
 *              cudaMemset after allocating); every call leaves it zero again.
 *              Calls sharing a workspace must not overlap on the GPU.
 *   options    PKV_DECODE_DEFAULT / _SIMT / _MMA, optionally | PKV_STEP_NO_PDL,
 *              PKV_STEP_RING(n), PKV_STEP_SORTED, PKV_STEP_TEST_EXPIRE_WAIT.
 *              None of them changes a result bit.
 * Launch: programmatic dependent launch (unless PKV_STEP_NO_PDL), with the
 * contract of pkv_decode_attention: before its dependency wait a CTA reads only
 * seq_lens, bt_dev and the cached pages holding no position at or beyond
 * seq_len - 2, and it lets the next launch begin only after its own wait.  So the
 * previous step of the same layer may be the immediately preceding kernel (a
 * one-layer model: it wrote position seq_len - 2), but that kernel must not write
 * seq_lens, bt_dev or earlier positions.  The first decode launch on a pool after
 * a pkv_prefill_append on it goes without programmatic dependent launch.
 * Device checks as pkv_decode_attention, plus seq_len > max_pos.
 * FP8 pools: the same single launch (a ring stage is one 2176-byte unit): the new
 * token's rotated key row and value row are quantized as pkv_append_rope quantizes
 * them, and results are bit-identical to the separate calls.  The SIMT variant
 * returns PKV_ERR_UNSUPPORTED. */
int pkv_decode_step(const pkv_pool *pool, const uint16_t *k_new, const uint16_t *v_new, uint16_t *q,
                    const int32_t *bt_dev, int max_blocks, const int32_t *seq_lens_dev, int B,
                    const float *rope_table, int max_pos, float scale, int pages_per_chunk, void *workspace,
                    size_t workspace_bytes, uint16_t *out, int32_t *dev_err_flag, void *cuda_stream, int options);

/* Every layer of one decode step: pkv_decode_step for layer l = 0 .. layers-1, in
 * that order, on the one stream.  The pages put each layer of the model after the
 * previous one; in the samir-vllm README summary the decode loop runs the layers in
 * turn, and this call keeps that order.  It exists so that a host loop issues one call
 * per step instead of one per layer (the per-call host work is the same as
 * pkv_decode_step's, done here in native code).
 *   Layer l's arguments are the given base pointers plus l times a layer stride, in
 *   elements: k_new and v_new + l * kv_layer_stride (BF16 elements), q and out +
 *   l * q_layer_stride (BF16 elements), bt_dev + l * bt_layer_stride (int32
 *   entries).  A stride of 0 reuses the same array for every layer.  seq_lens_dev,
 *   rope_table, workspace, dev_err_flag, options and the stream are shared by all
 *   layers; the layers run one after another, so sharing the workspace is allowed.
 *   Layouts, ownership, validation and device checks are pkv_decode_step's.
 * Errors: layers < 1 or a negative stride -> PKV_ERR_INVALID_ARG before anything is
 * launched.  Otherwise the first failing layer's status is returned and no later
 * layer is launched.  Earlier layers have then been launched and run. */
int pkv_decode_step_layers(const pkv_pool *pool, int layers, const uint16_t *k_new, const uint16_t *v_new,
                           uint16_t *q, const int32_t *bt_dev, int max_blocks, const int32_t *seq_lens_dev, int B,
                           const float *rope_table, int max_pos, float scale, int pages_per_chunk, void *workspace,
                           size_t workspace_bytes, uint16_t *out, int32_t *dev_err_flag, void *cuda_stream,
                           int options, int64_t kv_layer_stride, int64_t q_layer_stride, int64_t bt_layer_stride);

/* Size of the library's static scratch used by pkv_decode_attention_noalloc. */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB */

/* pkv_decode_attention without a workspace argument and without any allocation.
 * The pages have no counterpart: this entry point exists for callers that cannot
 * call cudaMalloc -- a plugin inside an engine that owns the whole device-memory
 * budget and gives its plugins no workspace, a latency-critical loop that must
 * not call cudaMalloc/cudaFree (they can synchronise the device), or a C caller
 * with no device allocator of its own.  The chunk partials go to a static
 * device array of PKV_NOALLOC_SCRATCH_BYTES inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   Arguments, layouts and results are those of pkv_decode_attention; it runs the
 *   two-kernel form (PKV_DECODE_SPLIT_MERGE), whose results are bit-identical to
 *   the default form's.  The caller still passes every input and the output.
 *   Limit: a problem whose pkv_decode_workspace_bytes(B, max_blocks,
 *   pages_per_chunk) exceeds PKV_NOALLOC_SCRATCH_BYTES is rejected with
 *   PKV_ERR_WORKSPACE_TOO_SMALL before anything is launched (for example batch
 *   256 at 128 table entries fits with pages_per_chunk 16: 17.3 MB).
 *   No cudaMalloc, cudaFree or allocating library routine is called.
 *   The first call on a device looks up the array's device address with that
 *   device current (cudaGetSymbolAddress); make that first call before any
 *   stream capture begins.
 *   All calls share the one array and it keeps the last call's contents; nothing
 *   in it needs to start at zero.  Calls whose work overlaps on the GPU (other
 *   streams, concurrent graph replays) race on it: serialise them. */
int pkv_decode_attention_noalloc(const pkv_pool *pool, const uint16_t *q, const int32_t *bt_dev, int max_blocks,
                                 const int32_t *seq_lens_dev, int B, float scale, int pages_per_chunk,
                                 uint16_t *out, int32_t *dev_err_flag, void *cuda_stream);

/* ------------------------------------------------------------------ misc */

/* Synchronise the stream, read the device error flag into *host_flag (may be
 * NULL) and return PKV_ERR_DEVICE_BOUNDS if any bit is set, else PKV_OK. */
int pkv_check_device_error(const int32_t *dev_err_flag, int32_t *host_flag, void *cuda_stream);

/* Human-readable name of a status code (static storage). */
const char *pkv_status_string(int status);

/* Library version string, e.g. "pkv 0.1 sm_103a". */
const char *pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
