/*
 * pkv.h -- C ABI of libpkv: paged KV-cache append and single-query decode
 * attention on NVIDIA GB300 (sm_103a).
 *
 * The method (blog pages on the paged KV cache, cited by title and section):
 *   "Build a Paged KV Cache in Pure Python"
 *     Step 1  a block holds the keys and values of block_size consecutive
 *             token positions, for every head of one layer;
 *     Step 2  blocks come from a shared, pre-allocated pool;
 *     Step 3  PagedKVCache.append: the token at position pos goes to row
 *             pos % block_size of the sequence's (pos // block_size)-th block;
 *             retrieve: a sequence's tokens are its blocks read in list order;
 *     Step 4  scaled_dot_product_attention: scores = scale * q.k_t over the
 *             sequence, max-subtracted softmax, weighted sum of v_t; an empty
 *             cache gives zeros;
 *     Step 5  a decode step appends the new token, then attends (the token
 *             attends to itself).
 *   "Building a Streaming Sliding-Window Attention Engine in Pure Python"
 *     Step 3  sliding_window_attention: with window w, attend over positions
 *             [max(0, T - w), T) of a length-T context.
 *
 * Conventions shared by every entry point
 *   - Pointers named *_cache, q, k, v, out, block_tables, context_lens,
 *     positions and slot_mapping are DEVICE pointers on the current CUDA
 *     device; the caller owns them.  Data pointers must be 16-byte aligned.
 *     A decode's q, k_new, v_new and out may also be device-side addresses
 *     of pinned host memory (pkv_device_address): the kernels then read or
 *     write them there, over the host link.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work on it and returns without synchronising, except
 *     where stated.
 *   - Return value: PKV_OK or a pkv_status code.  Arguments are checked on
 *     the host before anything is launched; a failed check launches nothing.
 *   - The K/V pool is HEAD-MAJOR: [num_blocks][num_kv_heads][block_size]
 *     [head_dim], row-major.  One (block, kv head) tile is one contiguous run
 *     of block_size * head_dim elements.  The pages store a block as
 *     (block_size, num_heads, head_dim); the head-major order is a storage
 *     choice that does not change what is computed.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_dtype {
  PKV_FLOAT32 = 0,
  PKV_FLOAT16 = 1,
  PKV_BFLOAT16 = 2,
  PKV_FP8_E4M3 = 3, /* pools only: E4M3 codes + one float32 scale per (token, kv head)
                       row; see pkv_append_fp8.  q, out, k_new, v_new are then fp16. */
  PKV_INT8 = 4      /* pools only: int8 codes + one float32 scale per row; see
                       pkv_append_int8.  q and out are then fp16. */
} pkv_dtype;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = 1,        /* a required pointer is NULL                          */
  PKV_ERR_SHAPE = 2,       /* a size is negative or sizes are inconsistent         */
  PKV_ERR_DTYPE = 3,       /* unknown dtype code                                  */
  PKV_ERR_UNSUPPORTED = 4, /* valid, not implemented (head_dim, block_size, ...)  */
  PKV_ERR_ALIGNMENT = 5,   /* a data pointer is not 16-byte aligned              */
  PKV_ERR_CUDA = 6,        /* a CUDA runtime call or a kernel launch failed       */
  PKV_ERR_NOMEM = 7,       /* the split-K workspace could not be allocated        */
  PKV_ERR_SCRATCH = 8,     /* pkv_decode_noalloc: the problem needs more split-K
                              scratch than its fixed buffer holds                */
  PKV_ERR_RANGE = 9        /* pkv_validate_indices: an index is out of range      */
} pkv_status;

/* Shape of one layer's K (or V) pool. */
typedef struct pkv_cache_layout {
  int64_t num_blocks;   /* NB: blocks in the pool                                  */
  int32_t num_kv_heads; /* Hkv                                                     */
  int32_t block_size;   /* bs: tokens per block; a multiple of 16, at most 256     */
  int32_t head_dim;     /* D: 64 or 128                                            */
  int32_t dtype;        /* pkv_dtype of the pool, and of q, k, v and out           */
} pkv_cache_layout;

/*
 * pkv_device_address -- the address through which this library's kernels
 *   reach `p`: p itself for device or managed memory, the mapped device-side
 *   address for pinned host memory.  Pageable or unknown host memory:
 *   PKV_ERR_UNSUPPORTED and *device_address = NULL.  Host-only: launches
 *   nothing and does not synchronise.  Not an operation of the pages: a
 *   decode's q, k_new, v_new and out may be such addresses of pinned host
 *   memory, read or written by the kernels over the host link (DecodeStep
 *   reads a step's queries and new rows that way).
 */
int pkv_device_address(const void* p, void** device_address);

/*
 * pkv_stage_copy -- copy `bytes` from src to dst with a kernel on `stream`.
 *   Not an operation of the pages: it moves a decode step's staged inputs
 *   from pinned host memory to the device and its output back.  Either side
 *   may be device memory, managed memory or pinned host memory (the kernel
 *   uses its device-side address); on a host whose pinned memory the GPU
 *   reaches over a coherent link this finishes small transfers well before a
 *   copy-engine copy.  Both addresses 16-byte aligned; any byte count.
 *   Pageable or unknown host memory: PKV_ERR_UNSUPPORTED (nothing launched).
 *   The ranges must not overlap.  Asynchronous, like every call here.
 */
int pkv_stage_copy(void* dst, const void* src, int64_t bytes, void* stream);

/*
 * pkv_slot_mapping -- slot of each sequence's new token.
 *   ("Build a Paged KV Cache in Pure Python", Step 3, PagedKVCache.append)
 *   slot_mapping[b] = block_tables[b][pos / bs] * bs + pos % bs, pos =
 *   positions[b].  A negative position, a position at or beyond
 *   max_blocks_per_seq * bs, or a negative block id gives -1 ("no write"
 *   for pkv_append).
 *   block_tables  [num_seqs][max_blocks_per_seq] int32, device
 *   positions     [num_seqs] int64, device
 *   slot_mapping  [num_seqs] int64, device, written
 */
int pkv_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                     const int64_t* positions, int32_t block_size, int64_t* slot_mapping,
                     void* stream);

/*
 * pkv_append -- write each new token's key and value into its cache slot.
 *   ("Build a Paged KV Cache in Pure Python", Step 3, PagedKVCache.append:
 *   keys[offset] = key_vec in the token's physical block)
 *   k, v          [num_tokens][num_kv_heads][head_dim], layout->dtype
 *   slot_mapping  [num_tokens] int64: token i goes to block slot / bs, row
 *                 slot % bs; a negative slot skips the token; a slot at or
 *                 beyond num_blocks * bs is skipped as well (nothing is written
 *                 out of bounds).
 *   k_cache, v_cache  head-major pools described by *layout, updated in place.
 *   The copy is bit-exact.  Two tokens mapped to the same slot race (the
 *   result is one of the two rows, unspecified which).
 */
int pkv_append(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens,
               void* k_cache, void* v_cache, const pkv_cache_layout* layout, void* stream);

/*
 * pkv_decode -- single-query attention of every (sequence, query head) over
 * its paged context.
 *   ("Build a Paged KV Cache in Pure Python", Step 4; "Building a Streaming
 *   Sliding-Window Attention Engine in Pure Python", Step 3)
 *   For sequence b with L = context_lens[b], lo = max(0, L - window) when
 *   window > 0, else 0, and query head h reading kv head h / (Hq / Hkv):
 *     s_t   = scale * sum_d q[b][h][d] * K[b, t][d]      for t in [lo, L)
 *     out[b][h][:] = sum_t softmax(s)_t * V[b, t][:]     (zeros when L == lo)
 *   where K[b, t] is row t % bs of kv head h/G in block block_tables[b][t / bs].
 *   q    [num_seqs][num_q_heads][head_dim], layout->dtype
 *   block_tables [num_seqs][max_blocks_per_seq] int32; entries past a
 *                sequence's last block are never read.
 *   context_lens [num_seqs] int32, the length including the token appended
 *                this step.
 *   out  [num_seqs][num_q_heads][head_dim], layout->dtype, written.
 *   Arithmetic: products and sums in fp32 (tensor-core MMA for fp16/bf16),
 *   online softmax in fp32, output rounded to nearest-even into the dtype.
 *   In-kernel errors never trap: a block id outside [0, num_blocks) or a
 *   context length outside [0, max_blocks_per_seq * bs] makes that
 *   sequence's output rows NaN.
 *   Long contexts are split across CTAs (flash-decoding); the partial
 *   results go to a workspace the library allocates (cudaMalloc) per
 *   (device, stream) on first use and replaces with a larger one when a
 *   larger problem arrives; outgrown buffers stay allocated (queued work or a
 *   captured CUDA graph may still use them) until pkv_release_workspaces.
 *   Issue the largest call once before capturing a CUDA graph, so that no
 *   allocation happens during capture.  Calls on one stream share that
 *   stream's workspace and are ordered by the stream; calls on different
 *   streams never share one.
 */
int pkv_decode(const void* q, int32_t num_seqs, int32_t num_q_heads,
               const void* k_cache, const void* v_cache, const pkv_cache_layout* layout,
               const int32_t* block_tables, int32_t max_blocks_per_seq,
               const int32_t* context_lens, int32_t window, float scale, void* out,
               void* stream);

/*
 * pkv_decode_split -- pkv_decode with an explicit context split.
 *   tokens_per_split: a positive multiple of 16 up to 65536 (each CTA handles
 *   at most that many tokens of one sequence; larger: PKV_ERR_UNSUPPORTED),
 *   or 0 to let the library choose (exactly what pkv_decode does).  The result is the same up to fp32 rounding
 *   order for every choice.
 */
int pkv_decode_split(const void* q, int32_t num_seqs, int32_t num_q_heads,
                     const void* k_cache, const void* v_cache, const pkv_cache_layout* layout,
                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                     const int32_t* context_lens, int32_t window, float scale, void* out,
                     int32_t tokens_per_split, void* stream);

/*
 * pkv_append_decode -- one decode step in one launch: pkv_append of every
 * sequence's new token, then pkv_decode, fused.
 *   ("Build a Paged KV Cache in Pure Python", Step 5: append the new token,
 *   then attend, so it attends to itself.)
 *   The new token of sequence b sits at position L - 1, L = context_lens[b]
 *   (the length after the append): its K and V rows, k_new[b][h][:] and
 *   v_new[b][h][:] ([num_seqs][num_kv_heads][head_dim], layout->dtype), are
 *   written to row (L-1) % bs of block block_tables[b][(L-1) / bs] and used
 *   for that position.  Sequences with L == 0 have no new token.  The pools and
 *   the output end up bit-identical to pkv_slot_mapping(positions = L - 1) +
 *   pkv_append + pkv_decode_split with the same tokens_per_split.
 *   Precondition: no other sequence of the call reads the block that receives
 *   a sequence's new token (true whenever the block holding a sequence's
 *   last position is private to it); otherwise use the separate calls.
 */
int pkv_append_decode(const void* q, const void* k_new, const void* v_new, int32_t num_seqs,
                      int32_t num_q_heads, void* k_cache, void* v_cache,
                      const pkv_cache_layout* layout, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t window,
                      float scale, void* out, int32_t tokens_per_split, void* stream);

/* Options of pkv_decode_ex. */
typedef struct pkv_decode_options {
  int32_t window;           /* <= 0: no window                                        */
  int32_t num_sinks;        /* with window > 0, positions [0, num_sinks) are attended
                               as well (attention sinks); 0: plain window             */
  int32_t tokens_per_split; /* a multiple of 16 up to 65536, or 0 for the library plan */
  const void* k_new;        /* both non-NULL: fused append of position L-1, as in    */
  const void* v_new;        /* pkv_append_decode; both NULL: decode only             */
  const float* k_scale;     /* 8-bit pools: [NB][Hkv][bs] row scales, 16-byte aligned; */
  const float* v_scale;     /* NULL otherwise                                         */
} pkv_decode_options;

/*
 * pkv_prefill -- append a chunk of new tokens per sequence and compute their
 * attention (chunked prefill over a paged cache).
 *   ("Building a Streaming Sliding-Window Attention Engine in Pure Python",
 *   Step 3, prefill_attention: query i attends key j when j <= i and, with a
 *   window, i - j < window; softmax per query row.)
 *   The chunks are packed: sequence b owns tokens cu_q[b] .. cu_q[b+1]-1
 *   (cu_q [num_seqs + 1] int32, device; n_b = cu_q[b+1] - cu_q[b] <= max_chunk).
 *   q    [T][num_q_heads][head_dim], k, v [T][num_kv_heads][head_dim] (T =
 *        cu_q[num_seqs]), layout->dtype (fp16 or bf16)
 *   context_lens [num_seqs]: L_b, the length after the chunk; the chunk sits at
 *        positions L_b - n_b .. L_b - 1, the tokens before it are in the pools.
 *   First the chunk's K/V rows are written to their slots (block_tables as in
 *   pkv_decode); then the query at position p attends positions j <= p (and
 *   p - j < window when window > 0) of the pools, which hold the prefix and
 *   the chunk.  With window > 0 and num_sinks > 0 the positions j <
 *   num_sinks (j <= p) are attended as well, as in pkv_decode_ex ("...
 *   Sliding-Window Attention Engine", Extending: attention sinks); num_sinks
 *   is ignored without a window and must not be negative.
 *   out [T][num_q_heads][head_dim].
 *   Limits: head_dim 64 or 128; num_seqs <= 65534.  The P.V product runs in
 *   fp16: with a bf16 cache, a V value beyond the fp16 range (|v| > 65504)
 *   makes the rows of the work items that read it non-finite (inf or NaN).
 *   Uses the stream's workspace (as pkv_decode's split-K) for the order of
 *   its work items, 4 bytes per (sequence, token chunk); may return
 *   PKV_ERR_NOMEM when that has to grow.
 *   In-kernel errors (bad block id, L_b < n_b) make the rows of the affected
 *   work item NaN: up to 256 (token, query head) rows of one sequence and kv
 *   head.
 */
int pkv_prefill(const void* q, const void* k, const void* v, const int32_t* cu_q,
                int32_t num_seqs, int32_t num_q_heads, int32_t max_chunk, void* k_cache,
                void* v_cache, const pkv_cache_layout* layout, const int32_t* block_tables,
                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t window,
                int32_t num_sinks, float scale, void* out, void* stream);

/*
 * pkv_append_fp8 -- quantise each new token's K and V rows into FP8 pools.
 *   ("Building a Memory-Compressed Attention Engine with KV Caching",
 *   Extending, item 2: INT8 or FP8 quantisation of the cached keys and
 *   values cuts the cache's memory traffic.)
 *   k, v        [num_tokens][num_kv_heads][head_dim], dtype in_dtype (fp32, fp16
 *               or bf16)
 *   slot_mapping as in pkv_append (negative or out-of-pool slots are skipped)
 *   k_cache, v_cache  E4M3 code pools [NB][Hkv][bs][D] (layout->dtype ==
 *               PKV_FP8_E4M3), k_scale, v_scale [NB][Hkv][bs] float32.
 *   Each (token, kv head) row is quantised on its own: scale = absmax / 448,
 *   code_d = E4M3(x_d * (448 / absmax)) rounded to nearest even, saturating;
 *   an all-zero row gets scale 1.  The stored value is code * scale.  Division
 *   and product are single IEEE float32 operations, so the codes are exactly
 *   reproducible.  head_dim 64 or 128.
 */
int pkv_append_fp8(const void* k, const void* v, int32_t in_dtype, const int64_t* slot_mapping,
                   int64_t num_tokens, void* k_cache, void* v_cache, float* k_scale,
                   float* v_scale, const pkv_cache_layout* layout, void* stream);

/*
 * pkv_append_int8 -- quantise each new token's K and V rows into INT8 pools.
 *   (Same passage as pkv_append_fp8: INT8 or FP8 quantisation of the cached
 *   keys and values.)
 *   Arguments as pkv_append_fp8, with int8 code pools (layout->dtype ==
 *   PKV_INT8).  Each (token, kv head) row is quantised on its own: scale =
 *   absmax / 127, code_d = x_d * (127 / absmax) rounded to the nearest
 *   integer, ties to even, clamped to [-127, 127] (-128 is never written; a
 *   NaN product gives 0); an all-zero row gets scale 1.  The stored value is
 *   code * scale; single IEEE float32 division and product, so the codes are
 *   exactly reproducible.  head_dim 64 or 128 (decode: 128).
 */
int pkv_append_int8(const void* k, const void* v, int32_t in_dtype, const int64_t* slot_mapping,
                    int64_t num_tokens, void* k_cache, void* v_cache, float* k_scale,
                    float* v_scale, const pkv_cache_layout* layout, void* stream);

/*
 * pkv_decode_ex -- pkv_decode with every option.
 *   ("Building a Streaming Sliding-Window Attention Engine in Pure Python",
 *   Step 3 for the window and the StreamingLLM item of its "Extending" list
 *   for the sinks: the first tokens are kept regardless of the window.)
 *   With window w > 0 and num_sinks s > 0 a length-L context attends the
 *   positions [0, min(s, lo)) and [lo, L), lo = max(0, L - w).  The other
 *   arguments, the errors and the workspace are those of pkv_decode; k_cache
 *   and v_cache are written only with the fused append.
 *   8-bit pools (layout->dtype == PKV_FP8_E4M3 or PKV_INT8, head_dim 128):
 *   the attended values are code * row scale; q and out are fp16; k_scale and
 *   v_scale are required; the fused append is not available for them
 *   (PKV_ERR_UNSUPPORTED).
 */
int pkv_decode_ex(const void* q, int32_t num_seqs, int32_t num_q_heads, void* k_cache,
                  void* v_cache, const pkv_cache_layout* layout, const int32_t* block_tables,
                  int32_t max_blocks_per_seq, const int32_t* context_lens, float scale, void* out,
                  const pkv_decode_options* options, void* stream);

/*
 * pkv_decode_plan -- the split pkv_decode_ex would use (host only, no GPU
 * work).  num_sms: streaming multiprocessors to plan for (<= 0: query the
 * current device).  Writes the tokens per split and the number of splits
 * the grid provides for the longest possible context.
 */
int pkv_decode_plan(int32_t num_seqs, int32_t num_q_heads, const pkv_cache_layout* layout,
                    int32_t max_blocks_per_seq, int32_t window, int32_t num_sinks,
                    int32_t tokens_per_split, int32_t num_sms, int32_t* tokens_per_split_out,
                    int32_t* num_splits_out);

/*
 * pkv_decode_noalloc -- pkv_decode for callers that cannot allocate device
 * memory.  (The pages have no counterpart: it is a deployment variant.)
 *   Same arguments, same result and same split plan as pkv_decode.  Where
 *   pkv_decode asks cudaMalloc for its split-K workspace, this entry point
 *   uses a fixed buffer of PKV_NOALLOC_SCRATCH_BYTES (32 MiB) that is part of
 *   the library image: every GPU that loads libpkv holds it until the process
 *   exits.  It never calls cudaMalloc, cudaFree or any allocating routine, so
 *   it suits callers that have handed all free HBM to their own pool (a
 *   serving engine that reserves memory for its KV blocks up front leaves a
 *   library nothing to allocate from) and callers that cannot afford the
 *   device-wide synchronisation cudaMalloc / cudaFree may bring in a hot
 *   loop.
 *   Limit: B * Hq * num_splits * (head_dim * 4 + 8) bytes must fit in the
 *   buffer (num_splits from pkv_decode_plan; a problem that needs no split
 *   uses no scratch); otherwise PKV_ERR_SCRATCH and nothing is launched.
 *   8-bit pools (FP8, INT8) need row scales this call does not take:
 *   PKV_ERR_UNSUPPORTED (pkv_decode_noalloc_ex takes them).
 *   Set-up: the first call on each device looks up the buffer's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is kept until
 *   pkv_release_workspaces; after a device reset (cudaDeviceReset reloads
 *   the library's device image) call pkv_release_workspaces before the next
 *   pkv_decode_noalloc, so that it looks the buffer up again.
 *   Sharing: every call on every stream of a device uses the same buffer,
 *   which keeps the last call's partial results.  Nothing in it needs to start
 *   at zero (each call writes every partial it reads), but calls that overlap
 *   on the GPU race on it: order them (one stream, or events).
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int pkv_decode_noalloc(const void* q, int32_t num_seqs, int32_t num_q_heads,
                       const void* k_cache, const void* v_cache, const pkv_cache_layout* layout,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t window, float scale, void* out,
                       void* stream);

/*
 * pkv_decode_noalloc_ex -- pkv_decode_ex (window, attention sinks, tokens
 * per split, fused append rows, 8-bit pools with their row scales) with the
 * fixed scratch buffer of pkv_decode_noalloc instead of an allocated
 * workspace: the arguments and results of pkv_decode_ex, the limit, set-up
 * and sharing rules of pkv_decode_noalloc (PKV_ERR_SCRATCH beyond the
 * buffer).
 */
int pkv_decode_noalloc_ex(const void* q, int32_t num_seqs, int32_t num_q_heads, void* k_cache,
                          void* v_cache, const pkv_cache_layout* layout,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* context_lens, float scale, void* out,
                          const pkv_decode_options* options, void* stream);

/*
 * pkv_validate_indices -- debug aid, not part of the hot path: range-check
 * the indices that the other calls trust.
 *   The pages check capacity where an index is made: the allocator of "Build
 *   a Paged KV Cache in Pure Python" (Step 2) raises MemoryError when the pool
 *   cannot supply a block, and the cache manager of "Building a Streaming
 *   Sliding-Window Attention Engine in Pure Python" (Step 2) asserts that an
 *   append fits.  The kernels here cannot raise: a bad block id is skipped and
 *   the sequence's output is NaN, a slot past the pool is skipped.  This call
 *   finds such indices before they reach a kernel.
 *   block_tables [num_seqs][max_blocks_per_seq] int32, context_lens [num_seqs]
 *   int32 and slot_mapping [num_slots] int64 (NULL when num_slots == 0) are
 *   copied to the host on `stream`; the call then WAITS for the stream.  It
 *   checks, in this order:
 *     1 context_lens[b] in [0, max_blocks_per_seq * block_size];
 *     2 block_tables[b][j] in [0, num_blocks) for every block the context
 *       uses, j < ceil(context_lens[b] / block_size) (later entries are never
 *       read and may hold anything);
 *     3 slot_mapping[i] < num_blocks * block_size (negative = skipped);
 *     4 no two tokens share a slot (the order of their writes is undefined).
 *   Returns PKV_OK, or PKV_ERR_RANGE with the first failure in `error` (if
 *   not NULL): what = the check's number above, row / col = the index
 *   (b, j) or (i, earlier i'), value = the offending entry.  NULL arrays
 *   with non-zero sizes: PKV_ERR_NULL; negative sizes or block_size < 1:
 *   PKV_ERR_SHAPE; a failed copy: PKV_ERR_CUDA.
 */
typedef struct pkv_index_error {
  int32_t what;  /* 0 = none, else the number of the failed check */
  int64_t row, col, value;
} pkv_index_error;
int pkv_validate_indices(const int32_t* block_tables, int32_t num_seqs,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         const int64_t* slot_mapping, int64_t num_slots, int64_t num_blocks,
                         int32_t block_size, void* stream, pkv_index_error* error);

/* Human-readable name of a pkv_status code (static storage). */
const char* pkv_status_string(int status);

/*
 * pkv_release_workspaces -- free every split-K workspace the library holds,
 * outgrown ones included, and forget the device addresses of the fixed
 * scratch buffer of pkv_decode_noalloc (looked up again on the next call).
 * Synchronises the device; call it only when no pkv_decode is in flight and
 * no captured graph that contains one will run again.
 */
int pkv_release_workspaces(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
