/*
 * pkv.h -- C ABI of libpkv, paged-KV grouped-query attention for GB300 (sm_103a).
 *
 * The calls follow the contract of the source listings this library restates:
 *   "nx_f32_attn_paged.nx source"     paged append + attend, caller contract
 *   "nx_f32_gqa_attention.nx source"  GQA head grouping, layouts, self-test
 *   "nx_f32_llama_v4b.nx source"      batched multi-sequence decode step
 *   "nx_paged_kv_gate.nx source"      pool KAT, EQUIV, FORK + COW, REWIND gate
 *
 * Step order (caller contract in the header comment of "nx_f32_attn_paged.nx
 * source", and the Stack section of "nx_f32_llama_v4b.nx source"):
 *   pkv_ensure_append[_batch]   once per step, before layer 0
 *   pkv_attn_with_paged / pkv_attn_batch   once per layer: append + attend
 *   pkv_advance[_batch]         once per step, after the last layer
 *
 * Conventions
 *   - All float data are IEEE f32, row-major.  Q and out are [rows, n_heads*head_dim];
 *     K_new and V_new are [rows, n_kv_heads*head_dim] ("nx_f32_gqa_attention.nx
 *     source", header).  Query head h reads kv head h / (n_heads / n_kv_heads).
 *   - Device pointers are CUDA device addresses, 16-byte aligned when head_dim
 *     is a multiple of 4 (vector access) and 4-byte aligned otherwise; host
 *     pointers are plain host memory.  The caller owns every pointer it
 *     passes; the library never frees them.
 *   - A stream argument is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  A pool binds one stream: every device operation on the pool and
 *     its sequences (copy-on-append copies, page-table uploads, append, attend)
 *     is issued on it, in call order.
 *   - Every call returns a status (or NULL / -1 for constructors and ids) and
 *     validates its arguments before it changes any state.  pkv_last_error()
 *     describes the last failure of the calling thread.
 *   - Host metadata calls are synchronous on the host; device work is
 *     asynchronous on the pool stream.  A pool and its sequences must be used
 *     from one host thread at a time.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  1..3 carry the meaning of the NX_F32_AP_* codes at the top of
 * "nx_f32_attn_paged.nx source" (bad dim, bad GQA grouping, sequence /
 * storage failure); the rest are this library's. */
enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_BAD_DIM = 1,       /* a size <= 0, or a shape the kernels do not take */
    PKV_ERR_BAD_GQA = 2,       /* n_heads is not a multiple of n_kv_heads         */
    PKV_ERR_SEQ = 3,           /* NULL / dead sequence, or rows not ensured        */
    PKV_ERR_EXHAUSTED = 4,     /* the pool has too few free blocks                 */
    PKV_ERR_CAPACITY = 5,      /* len + n exceeds the sequence's max_tokens        */
    PKV_ERR_ARG = 6,           /* any other bad argument (NULL, alignment, dup)    */
    PKV_ERR_CUDA = 7,          /* a CUDA call failed                               */
    PKV_ERR_DEVICE_BOUNDS = 8, /* a kernel met a block id or page index out of range
                                  and skipped that access                          */
    PKV_ERR_DEVICE_TIMEOUT = 9 /* a kernel's bounded wait ran out; the tile it was
                                  working on was not written                       */
};

/* Bits of a device error word (the kernels OR them in; the sync calls below
 * read, clear and map them to PKV_ERR_DEVICE_BOUNDS / PKV_ERR_DEVICE_TIMEOUT). */
#define PKV_DEVERR_BOUNDS 1u
#define PKV_DEVERR_TIMEOUT 2u

typedef struct pkv_pool pkv_pool;
typedef struct pkv_seq pkv_seq;
typedef void *pkv_stream_t; /* cudaStream_t */

/* pkv_pool_new flags */
#define PKV_POOL_HOST_ONLY 1u /* metadata only: no device memory, no device work */
/* bf16 storage (no counterpart on the pages, which store f32): every K/V row
 * is rounded to the nearest bfloat16 (ties to even) when it is written and
 * widened to f32 when it is read; all arithmetic stays f32.  Halves the pool's
 * bytes and the decode traffic.  Needs an even kv_dim.  The fused append
 * (pkv_set_fused_append) rounds the new rows the same way; the contiguous
 * twin stays f32. */
#define PKV_POOL_BF16 2u
/* fp8 e4m3 storage (no counterpart on the pages): every K/V row is stored as
 * e4m3(x / scale) -- nearest, ties to even, saturated to +-448 -- and read as
 * that value times scale; scale is a power of two (pkv_pool_set_kv_scale,
 * default 1), so the read values are exact in f32 (and, times a tile's
 * power of two, in the tensor-core kernel's f16) and only the storage
 * rounding differs from f32.  Quarters the pool's bytes.  Needs kv_dim
 * % 4 == 0 (% 16 with head_dim 128).  As for bf16, the fused append rounds
 * the new rows the same way, and the contiguous twin stays f32. */
#define PKV_POOL_FP8 4u

/* ---------------------------------------------------------------- pool ---- */

/* Create a refcounted block pool ("nx_paged_kv_gate.nx source", KAT section:
 * pool_new(n_blocks, n_layers, kv_dim)).  Device layout of each of the K and V
 * pools: [n_blocks][n_layers][block_size][kv_dim] elements, f32 (or bf16 with
 * PKV_POOL_BF16, fp8 e4m3 with PKV_POOL_FP8); a block holds block_size
 * consecutive token rows of every layer.  k_pool_dev / v_pool_dev: caller-owned 16-byte-aligned device buffers
 * of that size (both non-NULL), or both NULL to let the library allocate them.  max_seqs bounds the live sequences; max_blocks_per_seq bounds
 * one page table.  The free list is a LIFO stack whose first pops are 0,1,2,...
 * Returns NULL on failure (bad sizes, out of memory).  With PKV_POOL_HOST_ONLY
 * the pool keeps metadata only and the device pointers / stream are ignored. */
PKV_API pkv_pool *pkv_pool_new(int32_t n_blocks, int32_t n_layers, int32_t kv_dim, int32_t block_size,
                       void *k_pool_dev, void *v_pool_dev, int32_t max_seqs,
                       int32_t max_blocks_per_seq, pkv_stream_t stream, uint32_t flags);

/* Release the pool, every sequence still alive in it, and library-owned memory.
 * Waits for the pool stream first. */
PKV_API void pkv_pool_free(pkv_pool *pool);

/* Rebind the pool stream.  The caller orders the old stream's work before the
 * new stream's (e.g. by synchronising).  Returns PKV_OK or PKV_ERR_ARG. */
PKV_API int pkv_pool_set_stream(pkv_pool *pool, pkv_stream_t stream);

/* Device base addresses of the K and V pools (NULL for a host-only pool);
 * f32, bf16 or fp8 elements as the pool was created. */
PKV_API void *pkv_pool_k_data(const pkv_pool *pool);
PKV_API void *pkv_pool_v_data(const pkv_pool *pool);

/* Scale of an fp8 pool (no counterpart on the pages): stored element =
 * e4m3(x / scale), read value = element * scale.  A power of two in
 * [2^-20, 2^20]; settable only while every block is free.  PKV_ERR_ARG for a
 * pool that is not fp8, a bad scale, or blocks in use. */
PKV_API int pkv_pool_set_kv_scale(pkv_pool *pool, float scale);

/* Number of blocks on the free list, or -1 for NULL. */
PKV_API int32_t pkv_pool_free_blocks(const pkv_pool *pool);

/* Work list of the pool's last attend call (diagnostics and measurement; no
 * counterpart on the pages).  Writes min(cap, PKV_WORK_FIELDS) values into
 * the caller's host array `out`; returns PKV_OK, or PKV_ERR_ARG for a NULL
 * pool or array or a negative cap:
 *   [0] split-K decode units, [1] tensor-core prefill tiles, [2] shared-prefix
 *   tiles, [3] merge items, [4] visible (query, key) pairs of the prefill rows,
 *   [5] (query, key) pairs of the shared-prefix pass, [6] 1 if the call ran
 *   with the fused append, [7] operand images (64-key tile x kv heads) the
 *   call took from the image cache, [8] operand images it built, [9] keys per
 *   split of the shared-prefix pass (0 without one), [10] CTAs of the
 *   tensor-core prefill launch (see pkv_set_prefill_pairing). */
#define PKV_WORK_FIELDS 11
PKV_API int pkv_pool_last_work(const pkv_pool *pool, int64_t *out, int32_t cap);

/* Operand-image cache (no counterpart on the pages; off by default).  The
 * tensor-core launches read every 64-key tile they attend as an image of
 * f16 pieces (the tile's values times a power of two, split into two f16
 * planes; n_kv_heads x 64 KiB per tile, head_dim 128), which a split pass
 * builds from the pool.  With the cache on, images of tiles whose
 * pages have not been written since are kept across calls in up to
 * max_bytes of device memory (least recently used first out) instead of
 * being rebuilt: a chunked prefill then splits each key tile once rather
 * than once per later chunk, and the pages of a shared prefix once rather
 * than once per decode step.  A tile is identified by its layer, its length
 * and the pages holding it with their write generations; the library bumps a
 * page's generation whenever it writes the page (append, copy-on-append,
 * allocation).  Writes into caller-owned pool storage that bypass the
 * library are not seen: call this function again after them, which forgets
 * every cached image.  A call that needs more tiles than the cache holds
 * builds its images as without the cache.  max_bytes = 0 turns the cache off
 * and frees it.  Returns PKV_OK; PKV_ERR_ARG for a NULL or host-only pool or a
 * negative size; PKV_ERR_CUDA if the buffer cannot be allocated (the cache is
 * then off). */
PKV_API int pkv_pool_set_image_cache(pkv_pool *pool, int64_t max_bytes);

/* Allocate one block: its id (refcount 1), or -1 when the pool is exhausted
 * ("nx_paged_kv_gate.nx source", KAT section: ids 0,1,2 then -1). */
PKV_API int64_t pkv_alloc_block(pkv_pool *pool);

/* Drop one reference; at zero the id returns to the free list and is the next
 * one handed out (KAT section: a freed id recycles).  PKV_ERR_ARG for an id
 * out of range or not allocated. */
PKV_API int pkv_unref_block(pkv_pool *pool, int64_t id);

/* Refcount of a block (0 when free), or -1 for an id out of range
 * ("nx_paged_kv_gate.nx source", FORK section reads pool.refcnt[id]). */
PKV_API int32_t pkv_refcnt(const pkv_pool *pool, int64_t id);

/* ------------------------------------------------------------ sequences ---- */

/* New empty sequence with room for max_tokens tokens ("nx_paged_kv_gate.nx
 * source", EQUIV section: seq_new(pool, 64)).  NULL if max_tokens <= 0, if
 * ceil(max_tokens / block_size) > max_blocks_per_seq, or if max_seqs are live. */
PKV_API pkv_seq *pkv_seq_new(pkv_pool *pool, int32_t max_tokens);

/* Fork: a new sequence sharing every block of the parent (refcount + 1 each)
 * with the same length ("nx_paged_kv_gate.nx source", FORK section).  Writes
 * into a shared block are preceded by a private copy (copy-on-append, see
 * pkv_ensure_append).  NULL on failure. */
PKV_API pkv_seq *pkv_seq_fork(pkv_seq *parent);

/* Release a sequence: unreference its blocks, last block first. */
PKV_API int pkv_seq_free(pkv_seq *seq);

/* Speculative-decode rewind ("nx_paged_kv_gate.nx source", REWIND section):
 * len := new_len, blocks with index >= ceil(new_len / block_size) are
 * unreferenced (last first).  PKV_ERR_ARG unless 0 <= new_len <= len. */
PKV_API int pkv_seq_truncate(pkv_seq *seq, int32_t new_len);

/* pkv_seq_truncate for M sequences of one pool: new_len is a host array of M
 * lengths; all are validated (PKV_ERR_ARG, duplicates included) before any
 * sequence changes, then applied in batch order. */
PKV_API int pkv_seq_truncate_batch(pkv_seq *const *seqs, int32_t M, const int32_t *new_len);

/* Current length (tokens already committed by pkv_advance), or -1 for NULL. */
PKV_API int32_t pkv_seq_len(const pkv_seq *seq);

/* Copy up to cap page-table entries (block ids, in position order) to out (host).
 * Returns the number of entries the table holds, or -1 for NULL seq. */
PKV_API int32_t pkv_seq_page_table(const pkv_seq *seq, int32_t *out, int32_t cap);

/* Pool slot of the sequence's page-table row on the device (0..max_seqs-1), or -1. */
PKV_API int32_t pkv_seq_slot(const pkv_seq *seq);

/* Make positions [len, len+n) writable, once per step before layer 0
 * ("nx_f32_attn_paged.nx source", caller contract; "nx_f32_llama_v4b.nx
 * source", Stack section).  Shared blocks among those the rows fall in are
 * first copied to fresh private blocks (copy-on-append; the copy of every
 * layer's K and V rows is issued on the pool stream at once), then missing
 * tail blocks are allocated, both in ascending block index.  All-or-nothing:
 * PKV_ERR_CAPACITY if len+n > max_tokens, PKV_ERR_EXHAUSTED if the pool has
 * too few free blocks -- nothing changes in either case.  PKV_ERR_ARG if n <= 0. */
PKV_API int pkv_ensure_append(pkv_seq *seq, int32_t n);

/* pkv_ensure_append for M sequences, all-or-nothing over the whole batch;
 * n is a host array of M counts.  Duplicate sequences -> PKV_ERR_ARG. */
PKV_API int pkv_ensure_append_batch(pkv_seq *const *seqs, int32_t M, const int32_t *n);

/* Commit n appended tokens, once per step after the last layer
 * ("nx_f32_attn_paged.nx source", caller contract).  PKV_ERR_SEQ if no block
 * covers the new length, PKV_ERR_CAPACITY past max_tokens, PKV_ERR_ARG if n <= 0. */
PKV_API int pkv_advance(pkv_seq *seq, int32_t n);

/* pkv_advance for M sequences (validated as a whole, then applied). */
PKV_API int pkv_advance_batch(pkv_seq *const *seqs, int32_t M, const int32_t *n);

/* ------------------------------------------------------------ per layer ---- */

/* Append only: write n_tokens rows of K_new / V_new (device, [n_tokens, kv_dim])
 * at positions len..len+n_tokens-1 of layer `layer` through the page table
 * (the append step of "nx_f32_attn_paged.nx source": blocks pre-ensured).
 * PKV_ERR_SEQ if those rows are not in existing private blocks. */
PKV_API int pkv_append_layer(pkv_seq *seq, int32_t layer, const float *K_new, const float *V_new,
                     int32_t n_tokens);

/* Append + attend for one sequence and one layer (nx_f32_attn_with_paged,
 * "nx_f32_attn_paged.nx source"): append n_tokens rows, then for every query
 * row i and head h attend over total_k = len + n_tokens keys with
 * q_pos = total_k - n_tokens + i (causal != 0: keys j <= q_pos; causal == 0:
 * all keys), scores scale * <Q, K>, softmax, weighted sum of V rows.
 * Q, out: device [n_tokens, n_heads*head_dim]; K_new, V_new: device
 * [n_tokens, n_kv_heads*head_dim]; n_kv_heads*head_dim must equal the pool's
 * kv_dim, head_dim <= 256.  Checks, in order: sizes <= 0 -> PKV_ERR_BAD_DIM;
 * grouping -> PKV_ERR_BAD_GQA; NULL seq or rows not ensured -> PKV_ERR_SEQ.
 * Range: the kernels sum p * V in f32 with p taken relative to a running
 * maximum (each p at most 256), so results are finite while 256 x (visible
 * keys) x max|V| < 3.4e38: max|V| up to about 1e30 for a million keys. */
PKV_API int pkv_attn_with_paged(const float *Q, const float *K_new, const float *V_new,
                        int32_t n_tokens, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                        pkv_seq *seq, int32_t layer, int32_t causal, float scale, float *out);

/* Batched append + attend for M sequences of one pool (the per-row attention
 * loop of "nx_f32_llama_v4b.nx source", Block section, as one launch set):
 * row r owns n_q[r] consecutive rows of Q / K_new / V_new / out, in batch
 * order.  n_q[r] = 1 for decode rows; n_q[r] > 1 is a chunked-prefill row
 * (offset-causal).  n_q is a host array.  Each row's result equals the M = 1
 * call on that row bit for bit, except rows of a shared-prefix group (see
 * pkv_set_cascade), which agree with it within f32 rounding.  Errors as
 * pkv_attn_with_paged; duplicate sequences -> PKV_ERR_ARG. */
PKV_API int pkv_attn_batch(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q,
                   const float *K_new, const float *V_new, int32_t n_heads, int32_t n_kv_heads,
                   int32_t head_dim, int32_t layer, int32_t causal, float scale, float *out);

/* pkv_attn_batch with rotary position embedding on append ("nx_f32_llama_v4b.nx
 * source", Block section, RoPE step: each row's position is its sequence's
 * length, the build-cs / apply-cs-neox pair applied to every query head and
 * every new key head before the attend call).  Row t of batch row r sits at
 * position p = len(r) + t; for every head and i < head_dim/2 the pair
 * (x[i], x[i + head_dim/2]) turns by the angle p * rope_base^(-2i/head_dim):
 *   x'[i] = x[i] cos - x[i+h/2] sin,  x'[i+h/2] = x[i] sin + x[i+h/2] cos,
 * with cos and sin of the angle computed in double precision and rounded to
 * f32, and each product and sum rounded to f32 (no fused multiply-add).  The rotated keys go into the pool (V is not rotated); the rotated
 * queries are library scratch; the caller's Q and K_new are left unchanged.
 * rope_base must be > 0 (PKV_ERR_ARG) and head_dim even (PKV_ERR_BAD_DIM);
 * the pages pass the base as an integer (rope_log_base).  Calls with RoPE keep
 * the separate append launch (no fused append). */
PKV_API int pkv_attn_batch_rope(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q,
                        const float *K_new, const float *V_new, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, int32_t layer, int32_t causal,
                        float scale, double rope_base, float *out);

/* pkv_attn_batch taking HOST buffers for Q, K_new, V_new and out; returns
 * when out is filled, with the same result as pkv_attn_batch.  When Q and out
 * are page-locked host memory the device can address (cudaHostAlloc /
 * cudaMallocHost, or registered, under unified addressing; 16-byte aligned
 * when head_dim % 4 == 0), the kernels read Q and write out in host memory
 * directly, so those transfers overlap the attention work; K_new and V_new
 * are copied to device staging first.  Other host memory is copied to device
 * staging before the launches and back after them. */
PKV_API int pkv_attn_batch_host(pkv_seq *const *seqs, int32_t M, const int32_t *n_q, const float *Q_host,
                        const float *K_new_host, const float *V_new_host, int32_t n_heads,
                        int32_t n_kv_heads, int32_t head_dim, int32_t layer, int32_t causal,
                        float scale, float *out_host);

/* Contiguous twin (nx_f32_attn_with_cache, the reference side of the EQUIV
 * gate in "nx_paged_kv_gate.nx source"): the same kernels over a contiguous
 * history.  Kc, Vc: device [total_k, n_kv_heads*head_dim], already holding the
 * n_q new rows at the end; Q, out: device [n_q, n_heads*head_dim].  For the
 * same history it returns the paged path's output bit for bit.  Its scratch
 * (work list, split-K partials and, when the row takes the tensor-core kernel
 * (n_q >= 32, head_dim 128), the operand images of its keys: 64 KiB per
 * 64-key tile and kv head) comes from a stream-ordered memory pool and is
 * released on the stream after the launches; PKV_ERR_CUDA if it cannot be
 * allocated.  Failures the kernels find on the device are read by
 * pkv_contiguous_sync_error. */
PKV_API int pkv_attn_contiguous(const float *Q, const float *Kc, const float *Vc, int32_t n_q,
                        int32_t total_k, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                        int32_t causal, float scale, float *out, pkv_stream_t stream);

/* No counterpart in the paper: an addition of this library.
 * pkv_attn_contiguous for callers that cannot let a library allocate device
 * memory -- a serving engine that has reserved its whole device-memory budget
 * (a further cudaMalloc would fail or break its accounting), code running
 * inside an allocator or memory-pressure callback (allocating again would
 * re-enter that allocator), and latency-critical loops where cudaMalloc /
 * cudaFree may synchronise the device.  Same arguments, kernels and result as
 * pkv_attn_contiguous, but it calls no cudaMalloc, cudaFree or other
 * allocating routine: its scratch (work list, split-K partials and, for a row
 * that takes the tensor-core kernel, the operand images of its keys, 64 KiB per
 * 64-key tile and kv head) is one static device array of
 * PKV_NOALLOC_SCRATCH_BYTES, held by every GPU that loads the library until the
 * process exits.  The caller still passes the inputs and the output.  When a
 * tensor-core row's images do not fit in the array beside the rest, the row
 * goes to the split-K decode kernels instead (the same attention within f32
 * rounding, not the same bits as pkv_attn_contiguous).  Requests whose scratch
 * would still exceed the array are rejected with PKV_ERR_CAPACITY before any
 * work is enqueued (pkv_last_error() names the sizes).
 * The first call on a device does a one-time set-up with that device current:
 * it looks up the array's device address and clears the array's error word
 * (waiting for the device to finish the clear); make that first call before
 * any stream capture.  Every call shares the array and finds the previous
 * call's contents in it: calls whose GPU work overlaps (different streams, or
 * threads without ordering between their streams) race; calls on one stream
 * are ordered.  Failures the kernels find on the device (PKV_DEVERR_*)
 * gather in the array's error word until pkv_contiguous_sync_error reads
 * them. */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)
PKV_API int pkv_attn_contiguous_noalloc(const float *Q, const float *Kc, const float *Vc,
                                        int32_t n_q, int32_t total_k, int32_t n_heads,
                                        int32_t n_kv_heads, int32_t head_dim, int32_t causal,
                                        float scale, float *out, pkv_stream_t stream);

/* ---------------------------------------------------------- diagnostics ---- */

/* Wait for the pool stream, then return and clear the pool's device error
 * word (the fail-fast return codes of "nx_f32_attn_paged.nx source", applied
 * to failures found on the device after a call has returned): PKV_OK;
 * PKV_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out (the tile it was
 * working on left its output unwritten); PKV_ERR_DEVICE_BOUNDS if a kernel
 * met a block id or page index out of range and skipped that access; or
 * PKV_ERR_CUDA.  When both happened the timeout is reported and
 * pkv_last_error() names both. */
PKV_API int pkv_sync_error(pkv_pool *pool);

/* The same for the contiguous entry points, which have no pool: wait for
 * `stream`, then read and clear the current device's error words of
 * pkv_attn_contiguous and pkv_attn_contiguous_noalloc (each word gathers the
 * bits of every call on that device since it was last read).  Returns
 * PKV_OK, PKV_ERR_DEVICE_TIMEOUT, PKV_ERR_DEVICE_BOUNDS or PKV_ERR_CUDA as
 * pkv_sync_error does. */
PKV_API int pkv_contiguous_sync_error(pkv_stream_t stream);

/* Tests of the status mapping (no counterpart on the pages): OR `bits`
 * (PKV_DEVERR_*) into a device error word with a host-to-device copy, as a
 * kernel that met the condition would, so that the sync calls can be checked
 * without making any kernel fail.  which = PKV_ERRWORD_POOL: the pool's word
 * (waits for the pool stream first); PKV_ERRWORD_CONTIGUOUS /
 * PKV_ERRWORD_NOALLOC: the current device's word of pkv_attn_contiguous /
 * pkv_attn_contiguous_noalloc (pool ignored; the first use on a device sets
 * the word up as the first call of that entry point would).  Returns PKV_OK,
 * PKV_ERR_ARG (NULL or host-only pool, unknown `which`, bits outside
 * PKV_DEVERR_*) or PKV_ERR_CUDA. */
#define PKV_ERRWORD_POOL 0
#define PKV_ERRWORD_CONTIGUOUS 1
#define PKV_ERRWORD_NOALLOC 2
PKV_API int pkv_debug_or_error_bits(pkv_pool *pool, int32_t which, uint32_t bits);

/* Upload pending page-table changes now (they are otherwise uploaded by the
 * next device call on the pool). */
PKV_API int pkv_pool_flush(pkv_pool *pool);

/* Keys per split-K work unit of the decode kernels on f32 pools (default 1024,
 * a multiple of 32 in [32, 65536]); units on bf16 / fp8 pools take 2x / 4x as
 * many keys (the same bytes of K/V), at most 65536.  Tensor-core prefill rows
 * split every 16 x keys.  Process-wide; every call uses the value current at
 * the call, so results stay bit-exact between calls made under one setting. */
PKV_API int pkv_set_split_keys(int32_t keys);
PKV_API int32_t pkv_get_split_keys(void);

/* Fused append (default on).  The per-layer step appends the new K/V rows
 * into their pages and then attends over the sequence ("nx_f32_attn_paged.nx
 * source", header comment and step 1 of nx_f32_attn_with_paged).  With
 * fusion on, a decode call -- no row takes the tensor-core prefill path,
 * head_dim 128, group size 1, 2 or 4 (8 too on an fp8 pool), no RoPE -- whose
 * pending page-table changes all lie in pages that hold only this call's new
 * positions (fresh pages; not a copy-on-append tail, a fork or a truncate)
 * runs as the decode kernel alone: it reads the new rows from K_new / V_new
 * (rounded to the pool element as the append rounds them, on bf16 / fp8
 * pools), stores them into the pool and enters the new pages into the device
 * page table, with no separate append launch.  Every other call takes the
 * unfused path.  Results, pool contents and page tables are bit-identical
 * either way.  on != 0 enables; process-wide. */
PKV_API int pkv_set_fused_append(int32_t on);
PKV_API int32_t pkv_get_fused_append(void);

/* Shared-prefix (cascade) decode (default on).  Forks share their prefix
 * pages by reference ("nx_paged_kv_gate.nx source", FORK section: the fork
 * holds the parent's pages and each shared page's refcount reads 2).  When
 * a batch holds 16 or more consecutive rows with one query each whose first
 * 2048 or more keys lie in the same whole pages (head_dim 128, group size 1,
 * 2, 4 or 8), those keys are attended once for the whole run by a tensor-core
 * pass over the stacked queries, and each row's remaining keys by the decode
 * kernel; the two parts are combined by the log-sum-exp merge.  The result is
 * the same attention within f32 rounding (the split boundaries differ from
 * the non-cascade path, so it is not bit-identical to it).  on != 0 enables;
 * process-wide. */
PKV_API int pkv_set_cascade(int32_t on);
PKV_API int32_t pkv_get_cascade(void);

/* Placement of the tensor-core prefill tiles (no counterpart on the pages).
 * A CTA of the tensor-core kernel runs two tiles of 128 query rows of one row
 * and key split side by side, sharing every K/V tile.  mode 0: one tile per
 * CTA; 1: neighbouring tiles in pairs; 2 (default): pairs, with the last
 * pairs of the launch split into one-tile CTAs where a cost model says the
 * launch then ends sooner on the device's SMs (paged calls; the contiguous
 * entry points use mode 1 there).  The shared-prefix pass pairs its tiles in
 * every mode (its split size is chosen for pairs).  Each tile's arithmetic is
 * the same whatever its CTA holds, so results are bit-identical in every
 * mode.  Returns PKV_OK, or PKV_ERR_ARG for a mode outside 0-2;
 * process-wide. */
PKV_API int pkv_set_prefill_pairing(int32_t mode);
PKV_API int32_t pkv_get_prefill_pairing(void);

/* Kernel launch accounting.  pkv_launch_count: kernels launched by the library
 * so far (all kinds).  When profiling is on, every launch is bracketed by CUDA
 * events on its stream; pkv_profile_read synchronises those events and
 * returns, for kernel kind `kind` (see PKV_KERNEL_*), the summed device time in
 * ms and the number of launches since the last reset. */
enum pkv_kernel_kind {
    PKV_KERNEL_APPEND = 0,
    PKV_KERNEL_DECODE = 1,
    PKV_KERNEL_MERGE = 2,
    PKV_KERNEL_PREFILL = 3,
    PKV_KERNEL_COPY = 4,
    PKV_KERNEL_PAGETABLE = 5,
    PKV_KERNEL_SPLIT = 6,  /* operand images for the tensor-core launches */
    PKV_KERNEL_KINDS = 7
};
PKV_API int64_t pkv_launch_count(void);
PKV_API int pkv_profile_enable(int32_t on);
PKV_API int pkv_profile_reset(void);
PKV_API int pkv_profile_read(int32_t kind, double *ms, int64_t *launches);

/* Measured issue rate of tcgen05.mma kind::tf32 (a diagnostic for the
 * roofline of the tensor-core kernels; no counterpart on the pages).  On the current
 * device, one CTA per SM has one thread issue `iters` MMAs of M = 128, N =
 * n_cols, K = 8 back to back into one accumulator (A from tensor memory when
 * a_in_tmem != 0, else from shared memory; B from shared memory; zero
 * operands).  Writes the SM clocks per MMA (SM 0's CTA) and the GPU's TF32
 * rate in TFLOP/s (2 * 128 * n_cols * 8 flops per MMA, over the launch's
 * CUDA-event time).  n_cols 64, 128 or 256; iters a multiple of 16 in
 * [16, 1048576].  Synchronous; allocates a few bytes of device memory.
 * PKV_ERR_ARG, PKV_ERR_CUDA, or PKV_ERR_DEVICE_TIMEOUT if the bounded wait for
 * the MMAs ran out. */
PKV_API int pkv_probe_tf32_mma(int32_t n_cols, int32_t a_in_tmem, int32_t iters, double *clk_per_mma,
                               double *tflops);

/* The same for tcgen05.mma kind::f16 (f16 A and B, f32 accumulator), the
 * instruction of the tensor-core prefill kernel: K = 16 per MMA, rate over
 * 2 * 128 * n_cols * 16 flops per MMA.  Arguments, errors and side effects as
 * pkv_probe_tf32_mma. */
PKV_API int pkv_probe_f16_mma(int32_t n_cols, int32_t a_in_tmem, int32_t iters, double *clk_per_mma,
                              double *tflops);

/* Description of the calling thread's last failure ("" if none). */
PKV_API const char *pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
