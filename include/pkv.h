/*
 * pkv.h -- C ABI of libpkv: one model step of paged-KV attention for
 * continuous batching, on NVIDIA GB300 (sm_103a).
 *
 * Sources (pages on continuous batching; no code is taken from them):
 *   [LB]  Lucebox, "Continuous batching: Qwen3.8-27B at 301 tok/s across five
 *         clients, up to 1.97x llama.cpp"
 *   [T15] "Tutorial 15: Continuous Batching and Scheduling"
 *   [MX]  mlxcel manual, "Continuous batching"
 *
 * One step, in stream order on the caller's stream:
 *   1. pkv_plan_lower (host) turns the scheduler's step plan -- which slots
 *      advance by how many rows, prompt chunks first, decode rows after --
 *      into one packed token axis with segment metadata, growing each slot's
 *      block table from the shared free pool ([LB] §Packing unequal prompt
 *      chunks together; §Paged KV and paged attention).
 *   2. pkv_plan_work (host) splits the step's attention into work items.
 *   3. pkv_cache_write appends each new row's key and value to the pool.
 *   4. pkv_attention computes grouped-query attention for every packed row,
 *      causal inside prompt chunks, reading the pool through block tables.
 *
 * Conventions for every call:
 *   - bf16 tensors are passed as `void*`/`const void*` to 16-bit storage
 *     (IEEE bfloat16 bit patterns). All device tensors are row-major and
 *     contiguous, with the shapes given per argument.
 *   - The caller owns every buffer. The library allocates no device memory
 *     and never synchronises, except pkv_check_device_status.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). Arguments are validated on the host before any
 *     launch; a call that returns an error has launched nothing.
 *   - Index errors only visible on the device (a block ID outside the pool, a
 *     slot mapping past the pool, metadata that disagrees with the work list)
 *     never fault: the kernel skips the access and ORs a PKV_DEV_* bit into
 *     `device_status` (if non-NULL). Read it with pkv_check_device_status.
 *   - Supported shapes: head_dim 64 or 128; block_size 16, 32 or 64;
 *     num_q_heads a multiple of num_kv_heads with group size 1..16.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pkv_stream_t; /* identical to cudaStream_t */

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,          /* a pointer, size or shape is wrong */
    PKV_ERR_OUT_OF_RANGE = 2,         /* an index (slot, position, block) is outside its table */
    PKV_ERR_UNSUPPORTED = 3,          /* a valid shape this build has no kernel for */
    PKV_ERR_WORKSPACE_TOO_SMALL = 4,  /* a caller buffer is smaller than required */
    PKV_ERR_CUDA = 5,                 /* a CUDA runtime call failed */
    PKV_ERR_DEVICE_TIMEOUT = 6,       /* a kernel's bounded wait gave up (device_status) */
    PKV_ERR_NO_BLOCKS = 7,            /* the pool cannot satisfy a reservation */
    PKV_ERR_DEVICE_INDEX = 8          /* a kernel met an invalid index and skipped it */
} pkv_status;

/* Bits a kernel ORs into *device_status. */
#define PKV_DEV_BAD_SLOT_MAPPING 0x1u /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEV_BAD_BLOCK 0x2u        /* block-table entry outside [0, num_blocks) */
#define PKV_DEV_BAD_SEGMENT 0x4u      /* segment metadata disagrees with the work list */
#define PKV_DEV_TIMEOUT 0x8u          /* a bounded mbarrier wait expired */

/* Static text for a status code. */
const char *pkv_status_string(pkv_status status);

/* Library version as major*10000 + minor*100 + patch. */
int32_t pkv_version(void);

/* ------------------------------------------------------------------------
 * Block pool (host side). [LB] §Paged KV and paged attention: KV is divided
 * into fixed-size physical blocks shared by all sequences; each sequence owns
 * a block table mapping logical positions to physical blocks; finished
 * requests return their blocks, which a new request may take without moving
 * anyone else. [LB] §Admission and step planning are different decisions:
 * admission reserves KV capacity atomically. [LB] §Keeping track of each
 * request: each admitted request gets a stable sequence slot.
 *
 * The free list is a stack: released blocks go on top and are handed out
 * first. All calls are host-only, not thread-safe, and never touch a GPU.
 *
 * Blocks are reference counted ([MX] §Paged KV cache and prefix sharing: one
 * refcount + copy-on-write block pool). A request whose prompt starts with
 * another sequence's tokens adopts that sequence's blocks by reference
 * (pkv_pool_adopt) instead of prefilling them; a block held by several
 * tables is copied only when one of them first appends into it
 * (pkv_plan_lower records the copy; pkv_pool_take_copies hands it to the
 * caller, who runs pkv_copy_blocks before the step's cache write). A prompt
 * prefix cache is a slot that adopts a finished request's prefix and is
 * released to evict it.
 * ---------------------------------------------------------------------- */
typedef struct pkv_pool pkv_pool;

typedef struct pkv_pool_stats {
    int64_t num_blocks;     /* blocks in the pool */
    int32_t block_size;     /* tokens per block */
    int32_t max_slots;      /* sequence slots */
    int64_t free_blocks;    /* on the free stack */
    int64_t owned_blocks;   /* distinct blocks held by live slots (free + owned = available) */
    int32_t live_slots;     /* slots currently admitted */
    int64_t live_tokens;    /* sum of live slots' lengths */
    int64_t shared_blocks;  /* blocks held by more than one slot */
} pkv_pool_stats;

/*
 * Create a pool of `num_blocks` blocks of `block_size` tokens for
 * `max_slots` slots of at most `max_blocks_per_slot` blocks each.
 * `free_order` (nullable) gives the initial free stack, top LAST, as
 * `free_order_len` distinct block IDs; blocks not listed start out
 * unavailable. NULL means all blocks, block 0 on top.
 * Returns NULL on invalid arguments or allocation failure.
 */
pkv_pool *pkv_pool_create(int64_t num_blocks, int32_t block_size, int32_t max_slots,
                          int32_t max_blocks_per_slot, const int32_t *free_order,
                          int64_t free_order_len);
void pkv_pool_destroy(pkv_pool *pool);

/*
 * Admit a request into free slot `slot`: reserve ceil(reserve_tokens /
 * block_size) blocks off the free stack, all or nothing, as the first
 * entries of the slot's block table. The slot's length starts at 0.
 * Errors: PKV_ERR_OUT_OF_RANGE (bad slot or too many blocks for one slot),
 * PKV_ERR_INVALID_ARG (slot already live), PKV_ERR_NO_BLOCKS (not enough free
 * blocks; nothing is taken).
 */
pkv_status pkv_pool_admit(pkv_pool *pool, int32_t slot, int64_t reserve_tokens);

/*
 * Admit into `slot` with the given physical blocks (in logical order), each
 * of which must be on the free stack. All or nothing.
 */
pkv_status pkv_pool_admit_blocks(pkv_pool *pool, int32_t slot, const int32_t *blocks,
                                 int32_t num);

/*
 * Retire `slot`: each of its blocks loses one reference; blocks no other
 * table holds go back on the free stack (the slot's first such block on
 * top), and the slot becomes free. Other slots are untouched.
 * Errors: PKV_ERR_OUT_OF_RANGE, PKV_ERR_INVALID_ARG (slot not live).
 */
pkv_status pkv_pool_release(pkv_pool *pool, int32_t slot);

/*
 * Admit `slot` by adopting the first `num_tokens` tokens of live slot
 * `donor_slot`: the slot's table starts with the donor's first
 * ceil(num_tokens / block_size) blocks (one more reference each) and its
 * length is num_tokens, so those positions are never prefilled again. Fresh
 * blocks are reserved after them, all or nothing, up to
 * ceil(reserve_tokens / block_size) blocks in all. A partly filled last
 * shared block is copied on the slot's first append (pkv_plan_lower).
 * Errors: PKV_ERR_OUT_OF_RANGE, PKV_ERR_INVALID_ARG (slot live, donor not
 * live, same slot, num_tokens beyond the donor's length), PKV_ERR_NO_BLOCKS.
 */
pkv_status pkv_pool_adopt(pkv_pool *pool, int32_t slot, int32_t donor_slot, int64_t num_tokens,
                          int64_t reserve_tokens);

/* Tables currently holding `block` (0 if free), or -1 for a bad block ID. */
int32_t pkv_pool_block_refs(const pkv_pool *pool, int32_t block);

/*
 * Hand over the copy-on-write copies recorded by pkv_plan_lower since the
 * last call: `pairs` receives 2 * num_pairs int32 (source block, destination
 * block); the list is then cleared. With too little `capacity` (in pairs)
 * nothing is cleared and *num_pairs says how many there are
 * (PKV_ERR_WORKSPACE_TOO_SMALL). The copies must run (pkv_copy_blocks, same
 * stream) before the step's cache write.
 */
pkv_status pkv_pool_take_copies(pkv_pool *pool, int32_t *pairs, int64_t capacity,
                                int64_t *num_pairs);

/* Current length (tokens appended) of a live slot, or -1. */
int64_t pkv_pool_slot_length(const pkv_pool *pool, int32_t slot);

/* Blocks currently in the slot's table, or -1. */
int32_t pkv_pool_slot_blocks(const pkv_pool *pool, int32_t slot);

/* Counters in the spirit of [MX] §Paged KV cache and prefix sharing (block
 * size, allocated/free blocks). */
pkv_status pkv_pool_get_stats(const pkv_pool *pool, pkv_pool_stats *stats);

/*
 * Copy the block tables, int32 [max_slots][max_blocks_per_slot] with -1 in
 * unused entries, to host memory `out` of `capacity` entries.
 */
pkv_status pkv_pool_copy_block_tables(const pkv_pool *pool, int32_t *out, int64_t capacity);

/* ------------------------------------------------------------------------
 * Step-plan lowering (host side).
 * [LB] §One scheduler, model-specific execution: the engine lowers the
 * selected prompt chunks and decode rows into its backend's layout.
 * [LB] §Packing unequal prompt chunks together: one token axis, no padding,
 * segment metadata saying where each chunk ends and which slot owns it.
 * [LB] §Chunked prefill is a slot phase: each chunk appends to its slot's KV.
 * ---------------------------------------------------------------------- */
typedef struct pkv_segment {
    int32_t slot;       /* live slot whose sequence advances */
    int32_t num_tokens; /* new rows this step (1 for a decode row; a chunk otherwise) */
} pkv_segment;

/*
 * Lower a step plan (segments in packed order). For segment s with n rows
 * in slot c of current length len: rows take positions len .. len+n-1, the
 * slot's length becomes len+n, and blocks are taken off the free stack when
 * a position opens a block the table does not have yet (all or nothing for
 * the whole plan). A segment whose first append falls in a block that
 * another table also holds gets a fresh copy of that block first (recorded
 * for pkv_pool_take_copies). Host outputs:
 *   cu_seqlens_q  int32 [num_segments+1]  row offsets of each segment
 *   seq_slot      int32 [num_segments]    row-to-slot map
 *   context_lens  int32 [max_slots]       every slot's length after the step (0 if free)
 *   slot_mapping  int64 [capacity]        pool row of each new row:
 *                 table[c][p / block_size] * block_size + p % block_size
 *   total_q       number of packed rows written to slot_mapping
 * Errors: PKV_ERR_INVALID_ARG (slot not live, duplicate slot, negative n),
 * PKV_ERR_OUT_OF_RANGE (slot beyond max_blocks_per_slot),
 * PKV_ERR_WORKSPACE_TOO_SMALL (slot_mapping capacity), PKV_ERR_NO_BLOCKS.
 * On error nothing changes.
 */
pkv_status pkv_plan_lower(pkv_pool *pool, const pkv_segment *plan, int32_t num_segments,
                          int32_t *cu_seqlens_q, int32_t *seq_slot, int32_t *context_lens,
                          int64_t *slot_mapping, int64_t slot_mapping_capacity,
                          int64_t *total_q);

/* ------------------------------------------------------------------------
 * Attention work list (host side).
 * Segments of up to 16 / (num_q_heads / num_kv_heads) rows — decode rows,
 * and short runs of causal rows such as speculative-verification rows — go to
 * the split-KV decode kernel: the segment's keys are cut into fixed spans of
 * PKV_SPLIT_KEYS (the cut depends only on that segment's context, so a row's
 * result does not depend on what else is in the batch); a merge kernel
 * combines each row's spans in order.
 * Segments with several rows (prompt chunks) go to the tensor-core chunk
 * kernel, in tiles of 128 / (num_q_heads / num_kv_heads) query rows; with
 * head_dim 128 one item is a pair of consecutive tiles run by two SMs
 * together. The pages leave this split open; it is this library's design.
 *
 * Item words: decode (segment, slot, key span, first partial or -1; the
 * partial of span s, row i is first + s * rows + i); prefill (segment, slot,
 * first query tile, tiles in the item: 1 or 2); merge, one per row of a
 * multi-span segment (segment, slot, spans | row << 16 | (rows - 1) << 24,
 * first partial of the row); scratch, one per prompt-chunk segment
 * (segment, slot, first scratch block, blocks = ceil(context / block_size)),
 * used only by pkv_attention_q8.
 * ---------------------------------------------------------------------- */
#define PKV_SPLIT_KEYS 256
#define PKV_WORK_WORDS_PER_ITEM 4

typedef struct pkv_work_info {
    int32_t num_decode_items;  /* (segment, key span) items */
    int32_t num_prefill_items; /* (segment, query tile or tile pair) items */
    int32_t num_combine_items; /* (segment row) merge items: rows of decode segments with more than one span */
    int32_t num_partials;      /* span results kept in the workspace */
    int64_t work_words;        /* int32 words of the item array: decode, prefill, then merge items */
    uint64_t workspace_bytes;  /* device workspace pkv_attention needs (may be 0) */
    int32_t decode_rows_max;   /* most rows in a segment of the decode path (0: none) */
    int32_t num_scratch_items; /* (segment) items of the 8-bit pool's chunk path, one per chunk segment */
    int64_t scratch_blocks;    /* bf16 scratch blocks those items widen the chunks' histories into */
    uint64_t workspace_bytes_q8; /* device workspace pkv_attention_q8 needs (may be 0) */
    int32_t num_long_combine_items; /* the first merge items, whose rows have more than 64 spans */
} pkv_work_info;

/*
 * Build the item array for a step from HOST copies of the step metadata
 * (the same values later passed to pkv_attention on the device).
 * Validates: cu_seqlens_q starts at 0 and never decreases; seq_slot in
 * [0, max_slots) with no slot twice; every segment's rows <= its context
 * length <= max_blocks_per_slot * block_size; supported head shape.
 * `work` receives info->work_words int32 values; if `work_capacity` is too
 * small (or `work` is NULL) the call fills `info` and returns
 * PKV_ERR_WORKSPACE_TOO_SMALL, so it can size the array first.
 */
pkv_status pkv_plan_work(const int32_t *cu_seqlens_q, int32_t num_seqs,
                         const int32_t *seq_slot, const int32_t *context_lens,
                         int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t *work, int64_t work_capacity, pkv_work_info *info);

/* ------------------------------------------------------------------------
 * Device calls.
 * ---------------------------------------------------------------------- */

/*
 * Append new keys and values to the pool.
 * [LB] §Chunked prefill is a slot phase: each selected chunk (and each
 * decode row) appends directly to its slot's paged KV. [LB] §Paged KV and
 * paged attention: the pool is fixed-size blocks addressed through tables.
 *
 *   k_new, v_new  bf16 [num_tokens][num_kv_heads][head_dim]   device
 *   slot_mapping  int64 [num_tokens]  pool row per token; < 0 = skip   device
 *   k_pool, v_pool bf16 [num_blocks][num_kv_heads][block_size][head_dim] device
 * For token t with s = slot_mapping[t] >= 0, for every kv head h:
 *   k_pool[s / block_size][h][s % block_size][:] = k_new[t][h][:]  (same for v)
 * A bit-exact copy. Entries >= num_blocks * block_size are skipped and set
 * PKV_DEV_BAD_SLOT_MAPPING. Two tokens naming one row race (undefined which
 * wins); pkv_plan_lower never produces that. num_tokens == 0 launches nothing.
 */
pkv_status pkv_cache_write(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                           int64_t num_tokens, void *k_pool, void *v_pool, int64_t num_blocks,
                           int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                           uint32_t *device_status, pkv_stream_t stream);

/*
 * Paged grouped-query attention over one packed step.
 * [LB] §Paged KV and paged attention: attention reads each sequence's cached
 * history by following its block table in logical order, directly over the
 * shared pool. [LB] §Packing unequal prompt chunks together: per-query
 * causal positions and block-table metadata let prompt and decode rows share
 * one call. [LB] §Keeping track of each request: outputs follow the explicit
 * row-to-slot map, so slot reuse moves no other sequence's state.
 * [MX] §Paged KV cache and prefix sharing: a native block-table kernel in
 * place of a gather.
 *
 * Device inputs:
 *   q             bf16 [total_q][num_q_heads][head_dim]
 *   cu_seqlens_q  int32 [num_seqs+1]   packed row offsets per segment
 *   seq_slot      int32 [num_seqs]     slot of each segment
 *   context_lens  int32 [max_slots]    per-slot length INCLUDING this step's rows
 *   block_tables  int32 [max_slots][max_blocks_per_slot]
 *   k_pool, v_pool bf16 [num_blocks][num_kv_heads][block_size][head_dim]
 *   work          int32 [info->work_words]  pkv_plan_work's array, copied to the device
 * Host inputs: info (from pkv_plan_work for the same metadata), shapes,
 *   scale (<= 0 selects 1/sqrt(head_dim)).
 * Output: out bf16 [total_q][num_q_heads][head_dim], in packed row order.
 *
 * Row i of segment s (n rows, slot c, L = context_lens[c]) sits at position
 * p = L - n + i and attends keys 0..p of slot c; q head h reads kv head
 * h / (num_q_heads / num_kv_heads). Softmax in fp32 with fp32 accumulation,
 * output rounded to bf16 (nearest even). Results are deterministic and do
 * not depend on the other segments in the step or on their order.
 * `workspace` (device, >= info->workspace_bytes, 256-byte aligned) holds the
 * key-span partial results between the decode kernel and the merge kernel,
 * then the decode kernel's task counter (the last 256 bytes); it needs no
 * initialisation: on steps with more decode tasks than three per warp the
 * call zeroes the counter on `stream` (cudaMemsetAsync) before the decode
 * kernel. Calls that share a workspace must not overlap on the GPU. The pool must already hold this step's rows (pkv_cache_write
 * first, same stream). The kernels are launched with programmatic dependent
 * launch, so they may start while the previous kernel in the stream drains.
 * The decode and chunk kernels read the step metadata, q and the cached
 * history at once and wait for that previous kernel only before reading the
 * 16-key sub-tiles (decode) or 128-key tiles (chunk) that hold this step's
 * new rows. So the previous kernel must not signal dependents before the
 * data it leaves for this call is complete: pkv_cache_write signals only
 * after every kernel before it has finished, and a kernel that does not use
 * programmatic dependent launch signals at its end. When a step has both prompt
 * chunks and decode rows, the decode kernels run on a stream the library owns
 * (one per device), forked from `stream` at the call and joined back into it
 * before the call returns: work enqueued on `stream` afterwards still starts
 * only after all of this call's kernels.
 */
pkv_status pkv_attention(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs,
                         int64_t total_q, const int32_t *seq_slot, const int32_t *context_lens,
                         const int32_t *block_tables, int32_t max_slots,
                         int32_t max_blocks_per_slot, int32_t block_size, const void *k_pool,
                         const void *v_pool, int64_t num_blocks, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, float scale, const int32_t *work,
                         const pkv_work_info *info, void *out, void *workspace,
                         uint64_t workspace_bytes, uint32_t *device_status, pkv_stream_t stream);

/*
 * pkv_attention without a caller-provided workspace. The pages have no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory (a process whose device memory is all reserved up front in
 * its own arena, or a serving loop that may not allocate between steps).
 *
 * Same arguments and results as pkv_attention, minus `workspace` and
 * `workspace_bytes`: the span partials live in a file-scope device array of
 * PKV_NO_ALLOC_SCRATCH_BYTES bytes that every GPU loading the library holds
 * until the process exits. The call allocates nothing.
 *   - A step whose info->workspace_bytes exceeds PKV_NO_ALLOC_SCRATCH_BYTES
 *     is rejected with PKV_ERR_WORKSPACE_TOO_SMALL before any GPU work.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture. PKV_ERR_CUDA if the lookup fails.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; nothing in it needs to start at zero. Calls that overlap on the
 *     GPU (other streams, other host threads) race on it: serialise them.
 */
#define PKV_NO_ALLOC_SCRATCH_BYTES (32u << 20)

pkv_status pkv_attention_no_alloc(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs,
                                  int64_t total_q, const int32_t *seq_slot,
                                  const int32_t *context_lens, const int32_t *block_tables,
                                  int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size,
                                  const void *k_pool, const void *v_pool, int64_t num_blocks,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  float scale, const int32_t *work, const pkv_work_info *info,
                                  void *out, uint32_t *device_status, pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * 8-bit block-scaled KV pool.
 * [LB] §Qwen3.8-27B DFlash2 on the R9700 (vs llama.cpp) and §DeepSeek V4
 * Flash on Strix Halo and two GPUs: the pages serve from 8-bit and 4-bit KV
 * caches but do not define the formats. This library's 8-bit format: each
 * pool row (token, kv head) is cut into groups of 32 consecutive values; a
 * group keeps one power-of-two scale d -- the smallest power of two at or
 * above amax / 127 (amax = max |x| over the group, the quotient in float32),
 * at least 2^-126, 0 when amax is 0 -- stored as a bfloat16 (exact), and 32
 * int8 codes round_half_even(x / d) clamped to [-127, 127]. A code stands
 * for code * d, which is always a bfloat16 number.
 *
 *   k_codes, v_codes   int8 [num_blocks][num_kv_heads][block_size][head_dim]
 *   k_scales, v_scales bf16 [num_blocks][num_kv_heads][block_size][head_dim / 32]
 * A row costs head_dim + head_dim / 16 bytes instead of 2 * head_dim.
 * ---------------------------------------------------------------------- */

/*
 * pkv_cache_write for an 8-bit pool: quantise each new row's key and value
 * (bf16 [num_tokens][num_kv_heads][head_dim], device) into the pool row
 * slot_mapping[t] (< 0: skip). Bit-exact with the format's definition. Same
 * validation, device-status bits and stream behaviour as pkv_cache_write;
 * all pool pointers 16-byte aligned.
 */
pkv_status pkv_cache_write_q8(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                              int64_t num_tokens, int8_t *k_codes, void *k_scales, int8_t *v_codes,
                              void *v_scales, int64_t num_blocks, int32_t block_size,
                              int32_t num_kv_heads, int32_t head_dim, uint32_t *device_status,
                              pkv_stream_t stream);

/*
 * Copy-on-write copies ([MX] §Paged KV cache and prefix sharing): for each
 * (source, destination) pair of `pairs` (device, int32 [num_pairs][2], from
 * pkv_pool_take_copies), copy the whole source block over the destination
 * block in each of the `num_arrays` (1 to 4) pool arrays: arrays[a] (device,
 * 16-byte aligned) holds num_blocks blocks of block_bytes[a] bytes (a
 * multiple of 16) each -- a bf16 pool's K and V, or an 8-bit pool's codes
 * and scales. `arrays` and `block_bytes` are host arrays. A pair naming a
 * block outside the pool (or the same block twice) is skipped and sets
 * PKV_DEV_BAD_BLOCK. Run before the step's cache write, on its stream.
 */
pkv_status pkv_copy_blocks(const int32_t *pairs, int64_t num_pairs, void *const *arrays,
                           const int64_t *block_bytes, int32_t num_arrays, int64_t num_blocks,
                           uint32_t *device_status, pkv_stream_t stream);

/*
 * pkv_attention over an 8-bit pool: attention over the values the codes
 * stand for (code * scale), with the same arguments, results and ordering
 * rules as pkv_attention, except:
 *   - the pool is the four arrays above;
 *   - `workspace` must hold info->workspace_bytes_q8 bytes (256-byte
 *     aligned): the span partials, then, when the step has prompt chunks, a
 *     bf16 scratch pool of info->scratch_blocks blocks for K and for V and a
 *     scratch block table [max_slots][max_blocks_per_slot]. The chunk
 *     segments' histories are widened there (code * scale rounded to bf16)
 *     before the tensor-core chunk kernel reads them; decode rows read the
 *     codes directly.
 * `info` must come from pkv_plan_work for the same shapes (its
 * workspace_bytes_q8 is checked against them: PKV_ERR_INVALID_ARG otherwise).
 */
pkv_status pkv_attention_q8(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs,
                            int64_t total_q, const int32_t *seq_slot, const int32_t *context_lens,
                            const int32_t *block_tables, int32_t max_slots,
                            int32_t max_blocks_per_slot, int32_t block_size, const int8_t *k_codes,
                            const void *k_scales, const int8_t *v_codes, const void *v_scales,
                            int64_t num_blocks, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, float scale, const int32_t *work,
                            const pkv_work_info *info, void *out, void *workspace,
                            uint64_t workspace_bytes, uint32_t *device_status, pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * 4-bit block-scaled KV pool (head_dim 128). The same sources (Lucebox,
 * §DeepSeek V4 Flash on Strix Halo and two GPUs: 4-bit KV) and the same rule
 * as the 8-bit format with 7 in place of 127: per group of 32 values a
 * power-of-two scale d, the smallest at or above amax / 7 (at least 2^-126,
 * 0 when amax is 0), stored as a bfloat16, and codes round_half_even(x / d)
 * clamped to [-7, 7], stored as 4-bit two's complement nibbles, two per byte,
 * the even value in the low nibble. Every code * d is a bfloat16 number.
 *
 *   k_codes, v_codes   uint8 [num_blocks][num_kv_heads][block_size][head_dim / 2]
 *   k_scales, v_scales bf16 [num_blocks][num_kv_heads][block_size][head_dim / 32]
 * A row costs head_dim / 2 + head_dim / 16 bytes (72 at head_dim 128, against
 * 256 for bf16).
 * ---------------------------------------------------------------------- */

/*
 * pkv_cache_write_q8 for a 4-bit pool: same arguments, results (bit-exact
 * with the format) and errors; PKV_ERR_UNSUPPORTED unless head_dim is 128.
 */
pkv_status pkv_cache_write_q4(const void *k_new, const void *v_new, const int64_t *slot_mapping,
                              int64_t num_tokens, uint8_t *k_codes, void *k_scales, uint8_t *v_codes,
                              void *v_scales, int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim, uint32_t *device_status, pkv_stream_t stream);

/*
 * pkv_attention_q8 over a 4-bit pool: attention over code * scale, with the
 * same arguments, workspace (info->workspace_bytes_q8), results and ordering
 * rules; PKV_ERR_UNSUPPORTED unless head_dim is 128. Decode rows read the
 * nibbles directly; prompt chunks read their histories widened to bf16.
 */
pkv_status pkv_attention_q4(const void *q, const int32_t *cu_seqlens_q, int32_t num_seqs, int64_t total_q,
                            const int32_t *seq_slot, const int32_t *context_lens, const int32_t *block_tables,
                            int32_t max_slots, int32_t max_blocks_per_slot, int32_t block_size,
                            const uint8_t *k_codes, const void *k_scales, const uint8_t *v_codes,
                            const void *v_scales, int64_t num_blocks, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, float scale, const int32_t *work, const pkv_work_info *info,
                            void *out, void *workspace, uint64_t workspace_bytes, uint32_t *device_status,
                            pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * Host-staged step: a whole step from host memory in one call.
 * [LB] §One scheduler, model-specific execution: the engine hands the lowered
 * step to its backend in one go. The pages give no host/device protocol; this
 * one is the library's design: every per-step input sits in one caller-owned
 * host staging buffer at offsets fixed by pkv_stage_layout_init, so a step is
 * one host-to-device copy, the cache write, the attention call and one
 * device-to-host copy of the output (or, with PKV_STEP_IN_PLACE, the output
 * written by the kernels straight into host memory), all on `stream`.
 * ---------------------------------------------------------------------- */
typedef struct pkv_stage_layout {
    /* shapes the layout was made for */
    int64_t total_q;
    int32_t num_seqs, max_slots, max_blocks_per_slot, num_q_heads, num_kv_heads, head_dim;
    /* byte offsets into the staging buffers (each a multiple of 256) */
    uint64_t q;            /* bf16 [total_q][num_q_heads][head_dim] */
    uint64_t k_new;        /* bf16 [total_q][num_kv_heads][head_dim] */
    uint64_t v_new;        /* bf16 [total_q][num_kv_heads][head_dim] */
    uint64_t slot_mapping; /* int64 [total_q] */
    uint64_t cu_seqlens_q; /* int32 [num_seqs + 1] */
    uint64_t seq_slot;     /* int32 [num_seqs] */
    uint64_t context_lens; /* int32 [max_slots] */
    uint64_t block_tables; /* int32 [max_slots][max_blocks_per_slot] */
    uint64_t work;         /* int32 work list, written by pkv_step; runs to the end of the buffer */
} pkv_stage_layout;

/*
 * Fill `layout` for a step of these shapes. The caller writes the step's
 * inputs (as pkv_plan_lower and its own model produce them) at the offsets;
 * a staging buffer needs `layout->work` bytes plus room for the work list.
 * PKV_ERR_INVALID_ARG for a negative or zero shape or a size overflow.
 */
pkv_status pkv_stage_layout_init(pkv_stage_layout *layout, int64_t total_q, int32_t num_seqs,
                                 int32_t max_slots, int32_t max_blocks_per_slot,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim);

/*
 * Run one step from the host staging buffer `host_stage` (host memory laid
 * out by `layout`; page-locked for the copies to be asynchronous):
 *   1. plan the work list on the host from the staged cu_seqlens_q, seq_slot
 *      and context_lens, writing it into host_stage at layout->work (the
 *      room left there, (host_stage_bytes - layout->work) / 4 words, bounds it);
 *   2. one cudaMemcpyAsync of host_stage[0, layout->work + work bytes) to
 *      `device_stage` (device, 256-byte aligned, at least that many bytes);
 *   3. pkv_cache_write of the staged k_new / v_new / slot_mapping;
 *   4. pkv_attention over the staged q and metadata into `out` (device,
 *      bf16 [total_q][num_q_heads][head_dim]), with `workspace` as there;
 *   5. if `out_host` is not NULL, one cudaMemcpyAsync of `out` to it.
 * Nothing synchronises: the caller waits on `stream` before reading
 * out_host or writing host_stage again. `info_out` (nullable) receives the
 * step's work info, also on PKV_ERR_WORKSPACE_TOO_SMALL, so a caller can grow
 * `workspace` or the staging buffers and call again. The staged
 * cu_seqlens_q must end at layout->total_q. Any error from steps 1-2 returns
 * before anything is enqueued; an error from steps 3-5 is returned as
 * soon as it happens, with the earlier steps already enqueued.
 *
 * `options` (bit flags, 0 for none):
 *   PKV_STEP_IN_PLACE — the step skips the copy out when the device can
 *   address out_host (page-locked memory under unified addressing, as
 *   cudaPointerGetAttributes reports it): its output rows are written straight
 *   into out_host as the kernels produce them, and `out` is left untouched
 *   (the head_dim 128 chunk kernel then stages its rows in shared memory so
 *   that every store carries whole 256-byte rows over the host link). A step
 *   without prompt chunks whose staged bytes (inputs and work list) are at
 *   most PKV_STEP_IN_PLACE_MAX_BYTES also skips the copy in when the device
 *   can address host_stage: the kernels read the staged inputs from
 *   host_stage in place and device_stage is left untouched (with out_host
 *   NULL such a step writes `out`). For small steps each copy costs more in
 *   latency than its bytes; reading in place over the host link costs a few
 *   dependent accesses instead. Without device addresses for the buffers the
 *   step runs the copies as above.
 */
#define PKV_STEP_IN_PLACE 1u
#define PKV_STEP_IN_PLACE_MAX_BYTES (1u << 20)
pkv_status pkv_step(const pkv_stage_layout *layout, void *host_stage, uint64_t host_stage_bytes,
                    void *device_stage, uint64_t device_stage_bytes, void *k_pool, void *v_pool,
                    int64_t num_blocks, int32_t block_size, float scale, void *workspace,
                    uint64_t workspace_bytes, void *out, void *out_host, uint32_t *device_status,
                    pkv_stream_t stream, pkv_work_info *info_out, uint32_t options);

/*
 * Synchronise `stream`, read *device_status (device memory), clear it, and
 * map it to a status: PKV_OK if zero; PKV_ERR_DEVICE_TIMEOUT if the timeout
 * bit is set; otherwise PKV_ERR_DEVICE_INDEX. `bits_out` (nullable, host)
 * receives the raw bits. The only call that blocks the host.
 */
pkv_status pkv_check_device_status(uint32_t *device_status, pkv_stream_t stream,
                                   uint32_t *bits_out);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
