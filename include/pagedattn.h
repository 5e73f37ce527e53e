/*
 * pagedattn.h - C ABI of libpagedattn: attention over a paged KV cache for one flat ragged
 * continuous-batching step, on one NVIDIA GB300 (sm_103a).
 *
 * The operation follows "P3: native paged-KV continuous-batching sampler"
 * (code/docs/P3_ENGINE.md), Design / paged.py and Design / engine.py:
 *   - per-layer K and V pools shaped [num_blocks, block_size, Hkv, D];
 *   - an int32 block table [B, max_blocks] per step ("the argument a kernel takes");
 *   - a copy-free append: new K/V rows scatter into (block, offset) through a slot mapping;
 *   - one flat ragged step mixes decode rows and chunked-prefill segments
 *     (cu_seqlens_q, ctx_lens), with the GQA map kv_head = q_head / (Hq / Hkv);
 *   - a kernel contract with a fixed KV split per context length and no atomics, so that a
 *     sequence's output bits do not depend on what else is in the batch.
 * and "Finish RL Training Faster: Bitwise-Consistent, High-Performance, Agent-Driven",
 * section 2 (batch independence, phase consistency: a token gets the same bits in prefill
 * and in decode) and 4.2 (decode goes through the prefill read path).
 *
 * Conventions for every function below:
 *   - Every function returns a pa_status (PA_OK == 0) unless stated otherwise. Arguments are
 *     validated on the host before anything is launched; a failed check launches nothing.
 *   - "host" pointers are ordinary CPU memory; "device" pointers are CUDA global memory on
 *     the current device. The caller owns all buffers; the library never frees them and the
 *     step calls (paged_kv_write, paged_attention_step) allocate no memory.
 *   - bf16 tensors are passed as void* holding IEEE bfloat16 values, row-major, dense.
 *   - Kernels never trap. Device-side range checks (a block id outside the pool, a slot
 *     outside the pool) skip the access and OR a PA_DEVERR_* bit into *err_flag when the
 *     caller passes a device int32 (may be NULL). Every device wait is bounded; a wait that
 *     runs out sets PA_DEVERR_TIMEOUT and the kernel returns.
 *   - Streams: pa_stream_t is cudaStream_t (struct CUstream_st*); NULL is the legacy stream.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t;

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,       /* null pointer, negative size, inconsistent metadata */
    PA_ERR_SHAPE = 2,         /* head_dim / group / block_size this build does not support */
    PA_ERR_BOUNDS = 3,        /* block id, slot or position outside the pool or the table */
    PA_ERR_OOM = 4,           /* pool exhausted; the allocator changed nothing */
    PA_ERR_READONLY = 5,      /* a write would land in a block with refcount > 1 */
    PA_ERR_DOUBLE_FREE = 6,   /* free of a block whose refcount is already 0 */
    PA_ERR_INCONSISTENT = 7,  /* allocator books do not balance */
    PA_ERR_WORKSPACE = 8,     /* workspace smaller than pa_workspace_bytes() */
    PA_ERR_CUDA = 9,          /* a CUDA runtime call failed: pa_last_cuda_error() */
    PA_ERR_STATE = 10         /* unknown or duplicate sequence id */
} pa_status;

/* Bits OR-ed into the optional device error word by the kernels. */
#define PA_DEVERR_BLOCK   1   /* a block-table entry outside [0, num_blocks) was read */
#define PA_DEVERR_SLOT    2   /* a slot outside [0, num_blocks * block_size) was written */
#define PA_DEVERR_TIMEOUT 4   /* a bounded device wait ran out */
#define PA_DEVERR_META    8   /* a work item inconsistent with cu_seqlens_q / ctx_lens / limits */

/* Fixed KV split: keys [s * PA_SPLIT_TOKENS, (s + 1) * PA_SPLIT_TOKENS) form split s of every
 * sequence. It depends on nothing but the key position, which keeps the numerics of a row
 * independent of the batch ("fixed KV split per context length", P3 page Design / paged.py).
 * The size was tuned once on GB300 (2048 beat 1024 on every measured workload: fewer split
 * folds per prefill tile and fewer, longer decode items) and is frozen: changing it changes
 * the bits of every row longer than one split. */
#define PA_SPLIT_TOKENS 2048
/* Keys per tile of the shared tile routine; tiles are aligned to multiples of this. */
#define PA_TILE_KEYS 128
/* Persistent attention grid: min(n_items, PA_PLAN_CTAS) CTAs, one per SM of a GB300, and the
 * same number of item lists in a plan (CTA c walks list c). A device with fewer SMs runs the
 * surplus CTAs as SMs free up: the same results, later. */
#define PA_PLAN_CTAS 152

/* Geometry of one layer's pool. Supported: head_dim in {64, 128}; group = Hq / Hkv in
 * {1, 2, 4, 8, 16}; block_size a power of two in [8, 128]. */
typedef struct pa_shape {
    int32_t num_q_heads;    /* Hq */
    int32_t num_kv_heads;   /* Hkv; divides Hq */
    int32_t head_dim;       /* D */
    int32_t block_size;     /* tokens per block */
    int32_t num_blocks;     /* blocks in each of the K and V pools */
} pa_shape;

/* One unit of attention work: query rows [q_start, q_start + n_q) of sequence `seq`, one KV
 * head, one KV split. Produced by pa_plan_step on the host; copied to the device by the
 * caller and passed to paged_attention_step. The items form min(n, PA_PLAN_CTAS) lists, n the
 * real items: list c starts at item c and continues through `next`, and CTA c of the kernel
 * walks it. An item with n_q == 0 is padding: a CTA that meets one (as its first item, or
 * through `next`) has no more work, without error. Padding follows every real item. A caller
 * that captures a step in a CUDA graph pads every plan at its end to one fixed item count
 * (pa_plan_max_items for its limits) and rewrites the device buffers in place before each
 * replay: the CTAs past the real plan's lists then start at padding. A plan built by other
 * means must put every real item on exactly one list: an item on no list is not computed, and
 * one on two lists is computed twice (to the same values). */
typedef struct pa_work_item {
    int32_t seq;        /* index into cu_seqlens_q / ctx_lens / block_table rows */
    int32_t q_start;    /* first query row (token index into q and out) */
    int32_t n_q;        /* query rows, 1 .. 128 / group */
    int32_t kv_head;    /* KV head */
    int32_t split;      /* first KV split index */
    int32_t n_tiles;    /* key tiles of PA_TILE_KEYS the item reads (a cost estimate) */
    int32_t n_splits;   /* consecutive splits from `split` the item covers (0 counts as 1) */
    int32_t next;       /* index of the next item of this item's list; <= 0 ends the list. A
                         * successor has a higher index (an item that breaks this, or points
                         * past n_items, ends its list and raises PA_DEVERR_META) */
    int32_t kind;       /* PA_ITEM_PLAIN, PA_ITEM_GROUP or PA_ITEM_RESUME (see below) */
    int32_t tile0;      /* GROUP / RESUME: the shared key tiles [0, tile0) of split 0 */
} pa_work_item;

/* Item kinds. A PLAIN item is as described above. Prefix sharing (pa_plan_step_shared) adds
 * two: a GROUP item holds the decode rows of n_q consecutive sequences seq .. seq + n_q - 1
 * (one query row each, at tokens q_start .. q_start + n_q - 1) whose block tables agree on the
 * blocks of key tiles [0, tile0); it reads those shared tiles once, through seq's table, for
 * all of its rows, and saves each row's softmax state (accumulator, maximum, sum) to the row's
 * split-0 workspace slot. A RESUME item, later on the same list, continues one of those rows
 * over its own keys [tile0 * PA_TILE_KEYS, end of split 0) from the saved state. Every row runs
 * the same instruction sequence as without sharing (a tensor-core output element depends only
 * on its own row of A and column of B, and the state carried across is exact), so the output
 * bits are those of PLAIN items. */
#define PA_ITEM_PLAIN 0
#define PA_ITEM_GROUP 1
#define PA_ITEM_RESUME 2

/* ---------------------------------------------------------------- library ---------- */

/* ABI version of this header (returns the integer, not a status). */
int32_t pa_abi_version(void);

/* Human-readable name of a pa_status (static string; never NULL). */
const char* pa_status_string(int32_t status);

/* The cudaError_t of the most recent failed CUDA call on this host thread (0 if none). */
int32_t pa_last_cuda_error(void);

/* Streaming multiprocessors of the current device, in *n (host). */
int32_t pa_device_sm_count(int32_t* n);

/* ------------------------------------------------- host block allocator ------------ */
/* "P3: native paged-KV continuous-batching sampler", Design / paged.py: BlockAllocator is a
 * LIFO free list with refcounts; free on refcount 0 raises; check_consistent proves
 * free + referenced == total with no duplicates. PagedKVCache: ensure_capacity is
 * all-or-nothing; a block with refcount > 1 is read-only for everyone, owner included.
 * Design / engine.py: prefix sharing adopts the leading FULL blocks of a running sequence.
 * Exhaustion is a typed error, never truncation ("Optional paged KV cache (vLLM-style) - v1
 * design", Design: alloc throws PagedPoolExhausted).
 * The free stack starts so that the first allocation returns block 0; a freed block is the
 * next one handed out. Sequence ids are any non-negative int32. Not thread-safe. */
typedef struct pa_allocator pa_allocator;

/* Creates an allocator over num_blocks blocks of block_size tokens; *out owns it. */
int32_t pa_alloc_create(int32_t num_blocks, int32_t block_size, pa_allocator** out);
/* Destroys it (NULL is ignored). Returns PA_OK. */
int32_t pa_alloc_destroy(pa_allocator* a);
/* Pops one block (refcount 1) into *block; PA_ERR_OOM when none is free. */
int32_t pa_alloc_block(pa_allocator* a, int32_t* block);
/* Adds a reference to a live block; PA_ERR_STATE if it is free, PA_ERR_BOUNDS if out of range. */
int32_t pa_alloc_incref(pa_allocator* a, int32_t block);
/* Drops a reference; the block returns to the free list at 0. PA_ERR_DOUBLE_FREE at 0. */
int32_t pa_alloc_free_block(pa_allocator* a, int32_t block);
/* Creates the table of `seq` covering n_tokens tokens. With share_src >= 0, its first
 * n_shared blocks are the leading blocks of share_src's table (they must be full blocks of
 * the source, n_shared * block_size <= n_tokens), each gaining a reference. All or nothing:
 * PA_ERR_OOM / PA_ERR_STATE / PA_ERR_INVALID leave every table and refcount unchanged. */
int32_t pa_alloc_admit(pa_allocator* a, int32_t seq, int32_t n_tokens, int32_t share_src,
                       int32_t n_shared);
/* Grows seq's table to cover n_tokens; all or nothing (PA_ERR_OOM changes nothing). */
int32_t pa_alloc_ensure_capacity(pa_allocator* a, int32_t seq, int32_t n_tokens);
/* Releases every block of seq's table and forgets seq. */
int32_t pa_alloc_free_seq(pa_allocator* a, int32_t seq);
/* Rollback ("Optional paged KV cache (vLLM-style) - v1 design", Design: trim(n) rewinds the
 * offset and frees the now-unoccupied tail blocks; stale bytes past the offset are never
 * read). Keeps the ceil(n_tokens / block_size) leading blocks of seq and releases the rest,
 * last block first (a block shared with another table only loses this table's reference).
 * PA_ERR_BOUNDS if n_tokens needs more blocks than the table holds; nothing changes then. */
int32_t pa_alloc_trim(pa_allocator* a, int32_t seq, int32_t n_tokens);

/* Copy-on-write fork (same page, "Block-level CoW prefix sharing": refcounted block tables,
 * fork on divergent write). dst (a new id) gets every block of src, the partial last block
 * included; every block's refcount goes up by one. */
int32_t pa_alloc_fork(pa_allocator* a, int32_t src, int32_t dst);

/* Before seq writes positions [start, start + n): every block holding one of them that is
 * referenced by more than one table is replaced, in table order, by a fresh block, and the
 * (old, new) pairs are returned in pairs[2 * k], pairs[2 * k + 1] (host, up to max_pairs
 * pairs, count in *n_pairs). The caller copies each old block to its new block on the device
 * (paged_copy_blocks) before the write. All or nothing: PA_ERR_OOM if the pool cannot supply
 * every replacement, PA_ERR_INVALID if max_pairs is too small, PA_ERR_BOUNDS past the table;
 * nothing changes then. */
int32_t pa_alloc_cow(pa_allocator* a, int32_t seq, int32_t start, int32_t n, int32_t* pairs,
                     int32_t max_pairs, int32_t* n_pairs);

/* PA_OK if free + referenced == total, the free list has no duplicates and every refcount
 * equals the references held by live tables; PA_ERR_INCONSISTENT otherwise. */
int32_t pa_alloc_check_consistent(const pa_allocator* a);
/* Free blocks (returns the count, not a status; -1 on NULL). */
int32_t pa_alloc_num_free(const pa_allocator* a);
/* Refcount of a block (returns the count; -1 when out of range). */
int32_t pa_alloc_refcount(const pa_allocator* a, int32_t block);
/* Copies seq's table into out[0 .. cap) (host), the table length into *n. */
int32_t pa_alloc_table(const pa_allocator* a, int32_t seq, int32_t* out, int32_t cap, int32_t* n);
/* Slots of positions start .. start+n-1 of seq (host out[n]); PA_ERR_READONLY if any lands in
 * a block with refcount > 1, PA_ERR_BOUNDS beyond the table. Writes nothing on error. */
int32_t pa_alloc_slots(const pa_allocator* a, int32_t seq, int32_t start, int32_t n,
                       int32_t* out);
/* Builds one step's host metadata from the allocator: sequence i of the step is seqs[i] with
 * ctx_lens[i] tokens after the step, n_new[i] of them new (written this step). Outputs
 * (host, caller-owned): cu_seqlens_q[B+1], slot_mapping[sum n_new], block_table[B*max_blocks]
 * (row-major, -1 padded). Capacity must already cover ctx_lens (PA_ERR_BOUNDS otherwise);
 * PA_ERR_READONLY if a new token would land in a shared block. Writes nothing on error. */
int32_t pa_alloc_build_step(const pa_allocator* a, const int32_t* seqs, const int32_t* ctx_lens,
                            const int32_t* n_new, int32_t B, int32_t* cu_seqlens_q,
                            int32_t* slot_mapping, int32_t* block_table, int32_t max_blocks);

/* ------------------------------------------------------- host step metadata -------- */

/* ------------------------------------------------------------ host step scheduler --- */
/* "P3: native paged-KV continuous-batching sampler", Design / engine.py (Scheduler,
 * Admit/evict, Prefix sharing). The scheduler owns a block allocator and turns requests
 * (prompt length, tokens to generate, optional prefix leader) into flat ragged steps:
 *   - a step schedules n_new = min(remaining, chunk, budget) per sequence, remaining being
 *     tokens not yet in the cache; decodes (remaining 1) come first, then the other running
 *     sequences, each in admission order, then waiting sequences are admitted in FIFO order
 *     while budget remains (admission reserves blocks for the whole current token list and
 *     stops at the first request that does not fit or defers);
 *   - when a running sequence cannot grow, the youngest running sequence not yet scheduled in
 *     the step is preempted by recompute (blocks freed, num_computed = 0, back to the head of
 *     the waiting queue); with no such sequence the one being scheduled sits the step out;
 *   - a request with a leader shares (prompt - 1) / block_size leading full blocks of the
 *     leader once the leader has computed them (read-only, refcounted), defers while the
 *     leader waits or computes, is admitted without sharing once the leader has finished, and
 *     recomputes its own tokens from the first unshared position (its last prompt token
 *     always);
 *   - after a step, pa_sched_commit adds each sequence's n_new to its cache; a sequence whose
 *     cache reaches its token count samples one token: after max_new samples it finishes and
 *     its blocks are freed (the last sampled token is never written), else it gains a token.
 * Sequence ids are any non-negative int32. Not thread-safe. */
typedef struct pa_scheduler pa_scheduler;

int32_t pa_sched_create(int32_t num_blocks, int32_t block_size, int32_t chunk, int32_t budget,
                        pa_scheduler** out);
int32_t pa_sched_destroy(pa_scheduler* s);
/* The scheduler's allocator (owned by the scheduler; tables, slots, build_step, checks). */
pa_allocator* pa_sched_allocator(pa_scheduler* s);
/* Queues a request: prompt_len >= 1 tokens, max_new >= 1 tokens to sample, leader = a
 * sequence id whose prompt it shares, or -1. PA_ERR_STATE if seq was added before. */
int32_t pa_sched_add(pa_scheduler* s, int32_t seq, int32_t prompt_len, int32_t max_new,
                     int32_t leader);
/* Schedules one step (host out): for i < *n_out, sequence seqs[i] computes n_new[i] tokens
 * ending at context ctx_lens[i], in step order. cap must be at least the number of waiting
 * plus running sequences. Feed the result to pa_alloc_build_step on pa_sched_allocator(s).
 * PA_ERR_STATE if the previous step was not committed. */
int32_t pa_sched_step(pa_scheduler* s, int32_t* seqs, int32_t* n_new, int32_t* ctx_lens,
                      int32_t cap, int32_t* n_out);
/* Applies the pending step; the sequences that finished go to finished[] (host). */
int32_t pa_sched_commit(pa_scheduler* s, int32_t* finished, int32_t cap, int32_t* n_finished);
int32_t pa_sched_counts(const pa_scheduler* s, int32_t* n_waiting, int32_t* n_running,
                        int64_t* preemptions);
/* Token count, tokens in the cache and samples taken so far of one sequence. */
int32_t pa_sched_seq(const pa_scheduler* s, int32_t seq, int32_t* n_tokens,
                     int32_t* num_computed, int32_t* generated);

/* Slot mapping from explicit host tables (P3 page, Design / paged.py: copy-free append).
 * Token i of sequence s sits at position p = ctx_lens[s] - n_q(s) + i, where
 * n_q(s) = cu_seqlens_q[s+1] - cu_seqlens_q[s]; its slot is
 * block_table[s*max_blocks + p/block_size] * block_size + p % block_size.
 * Validates: cu_seqlens_q[0] == 0 and non-decreasing; 0 <= n_q(s) <= ctx_lens[s];
 * ceil(ctx/block_size) <= max_blocks; table entries covering ctx in [0, num_blocks).
 * Output slot_mapping[T] (host), T = cu_seqlens_q[B]. Writes nothing on error. */
int32_t pa_compute_slots(const pa_shape* shape, const int32_t* block_table, int32_t B,
                         int32_t max_blocks, const int32_t* cu_seqlens_q,
                         const int32_t* ctx_lens, int32_t* slot_mapping);

/* Upper bound on the work items pa_plan_step produces for B sequences, T query rows and no
 * context longer than max_ctx. Returns the count (0 on bad arguments). */
int64_t pa_plan_max_items(const pa_shape* shape, int32_t B, int32_t T, int32_t max_ctx);

/* Splits the step into work items (host in, host out). Query rows of a sequence are cut
 * into tiles of 128 / group rows. A sequence with one query row (a decode) gives one item per
 * (KV head, KV split its row reaches), so a long context is spread over many CTAs and its
 * splits are folded by the split-combine kernel. A sequence with more query rows (a prefill
 * chunk) gives one item per (tile, KV head) that covers every split the tile's last row
 * reaches; the kernel folds those splits itself, in the same ascending order and arithmetic,
 * so a row's bits are the same either way. paged_attention_step relies on this rule (an item
 * that breaks it is flagged PA_DEVERR_META and skipped). Balance: the items, taken by
 * decreasing n_tiles (ties in generation order), are dealt longest-processing-time first to
 * G = min(n, PA_PLAN_CTAS) lists, each to the list of least total cost so far (cost of an
 * item: n_tiles + 1; ties go to the lower list). The output holds the first item of every
 * list (list c at index c), then the second item of every list that has one, in list order,
 * and so on, with `next` linking each list. Everything is a pure function of the metadata.
 * Validates the metadata like pa_compute_slots (minus the table). PA_ERR_INVALID if
 * max_items is too small. */
int32_t pa_plan_step(const pa_shape* shape, int32_t B, const int32_t* cu_seqlens_q,
                     const int32_t* ctx_lens, pa_work_item* items, int32_t max_items,
                     int32_t* n_items);

/* pa_plan_step with prefix sharing (same output for steps without it): runs of consecutive
 * decode sequences (one query row each, at most 128 / group of them) whose block tables
 * [B, max_blocks] agree on the blocks of at least two leading key tiles become GROUP and
 * RESUME items (see pa_work_item) for every KV head, their splits past 0 PLAIN items. The
 * shared tiles are whole tiles of split 0 below every member's last key (at most
 * PA_SPLIT_TOKENS / PA_TILE_KEYS - 1 of them), so that each RESUME item has keys of its own. A
 * group's items (GROUP, then its RESUMEs) are dealt to one list as a unit; the balance rule is
 * otherwise that of pa_plan_step. Since a group's items share one list, such a plan can have
 * fewer lists than min(items, PA_PLAN_CTAS); its padding items (n_q == 0) then take indices
 * lists .. PA_PLAN_CTAS - 1, before the lists' second items, and *n_items counts them. A plan
 * with such items needs the workspace even when no
 * context exceeds PA_SPLIT_TOKENS (pa_workspace_bytes(shape, T, max_ctx) bytes; without one
 * its GROUP and RESUME items are flagged PA_DEVERR_META and skipped). At most
 * pa_plan_max_items_shared items. */
int64_t pa_plan_max_items_shared(const pa_shape* shape, int32_t B, int32_t T, int32_t max_ctx);
int32_t pa_plan_step_shared(const pa_shape* shape, int32_t B, const int32_t* cu_seqlens_q,
                            const int32_t* ctx_lens, const int32_t* block_table,
                            int32_t max_blocks, pa_work_item* items, int32_t max_items,
                            int32_t* n_items);

/* Bytes of fp32 workspace paged_attention_step needs for T query rows and contexts up to
 * max_ctx: split partials (acc[D], m, l) for every (row, split, q head). Sized by limits, not
 * by the load, so one buffer serves every step under the same limits. */
size_t pa_workspace_bytes(const pa_shape* shape, int32_t T, int32_t max_ctx);

/* Copies a validated host block table [B * max_blocks] to device memory `dev` on `stream`
 * (an ordinary async copy; pinned host memory makes it asynchronous). Entries must be -1 or
 * in [0, num_blocks): PA_ERR_BOUNDS otherwise, and nothing is copied. */
int32_t pa_upload_block_table(const pa_shape* shape, const int32_t* host, int32_t* dev,
                              int32_t B, int32_t max_blocks, pa_stream_t stream);

/* ------------------------------------------------------------- device step --------- */

/* KV-write scatter (P3 page, Design / paged.py: "write scatters into (block, offset) in
 * place"). For t in [0, T): if slot_mapping[t] >= 0, copies k_new[t] (Hkv*D bf16) to
 * k_pool[slot] and v_new[t] to v_pool[slot], where the pools are viewed as
 * [num_blocks*block_size, Hkv, D]. Bytes are copied unchanged (16-byte vector stores).
 * Device: k_new, v_new [T, Hkv, D] bf16; slot_mapping [T] int32; k_pool, v_pool
 * [num_blocks, block_size, Hkv, D] bf16; err_flag optional. A slot >= num_blocks*block_size
 * is skipped and sets PA_DEVERR_SLOT. T == 0 launches nothing. */
int32_t paged_kv_write(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                       int32_t T, void* k_pool, void* v_pool, const pa_shape* shape,
                       int32_t* err_flag, pa_stream_t stream);

/* Copy-on-write block copies (pairs from pa_alloc_cow, uploaded by the caller): for k in
 * [0, n_pairs), the K and V of block pairs[2k] are copied unchanged to block pairs[2k + 1].
 * Device: pairs [2 * n_pairs] int32; k_pool, v_pool as for paged_kv_write. A pair with an id
 * outside [0, num_blocks) or equal ids is skipped and sets PA_DEVERR_BLOCK. n_pairs == 0
 * launches nothing. Order it before the step's paged_kv_write on the same stream. */
int32_t paged_copy_blocks(const int32_t* pairs, int32_t n_pairs, void* k_pool, void* v_pool,
                          const pa_shape* shape, int32_t* err_flag, pa_stream_t stream);

/* Attention for one flat ragged step over an already-written pool (call paged_kv_write
 * first: ctx_lens count this step's tokens, P3 page "write new K/V, return [T, H, D]").
 * For every query row t of sequence s at position p = ctx_lens[s] - n_q(s) + (t - cu[s]) and
 * every q head h: out[t, h] = sum_{j <= p} softmax_j(q[t,h] . K_s[j, h/g] / sqrt(D)) V_s[j, h/g],
 * where K_s, V_s are s's keys in table order. Arithmetic: bf16 tensor-core products with fp32
 * accumulation, fp32 online softmax per fixed KV split, splits combined in ascending order,
 * result rounded to bf16 (nearest even). Every row, decode or prefill, runs the same tile
 * routine, so its bits depend only on its own query, keys and position.
 * Launches: the attention kernel, then (when max_ctx > PA_SPLIT_TOKENS) the split-combine
 * kernel, which finishes the decode rows whose context spans several splits (a prefill tile's
 * item folds its splits itself, in the same order and arithmetic), both as programmatic
 * dependent launches: each may start while the previous kernel
 * on the stream drains, and waits for that kernel to complete before it reads anything, so
 * stream order is kept for every input.
 * Device inputs: q [T, Hq, D] bf16; k_pool, v_pool [num_blocks, block_size, Hkv, D] bf16;
 * block_table [B, max_blocks] int32; cu_seqlens_q [B+1], ctx_lens [B] int32 (the same values
 * given to pa_plan_step); items [n_items] from pa_plan_step; workspace of ws_bytes >=
 * pa_workspace_bytes(shape, T, max_ctx) with max_ctx >= every ctx_lens[s], 16-byte aligned
 * (partials are stored and read as vectors; it may be NULL when max_ctx <= PA_SPLIT_TOKENS).
 * Device output: out [T, Hq, D] bf16 (rows not covered by items are not written).
 * Host checks: pointers, shape support, workspace size (PA_ERR_WORKSPACE) and alignment
 * (PA_ERR_INVALID); T == 0 or n_items == 0 launches nothing. */
int32_t paged_attention_step(const void* q, const void* k_pool, const void* v_pool,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                             int32_t B, int32_t T, int32_t max_ctx,
                             const pa_work_item* items, int32_t n_items,
                             void* workspace, size_t ws_bytes, void* out,
                             const pa_shape* shape, int32_t* err_flag, pa_stream_t stream);

/* Test of the bounded-wait error path (no counterpart on the pages: a diagnostic of this
 * library). The same call as paged_attention_step, except that the softmax role of every CTA
 * first waits, for at most never_ns nanoseconds (1 .. 10^9), on a barrier that nothing ever
 * completes. That wait runs out, the CTA's roles leave their loops exactly as after any other
 * wait that runs out (each drains its own copies and MMAs, with its usual bounded waits, and
 * TMEM is freed), PA_DEVERR_TIMEOUT is ORed into *err_flag, and the kernel returns; the
 * outputs of the step are then undefined, but the device stays usable for the next call. It
 * faults nothing and hangs nothing. PA_ERR_INVALID for never_ns outside that range. */
int32_t paged_attention_step_wait_test(const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_table, int32_t max_blocks,
                                       const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                       int32_t B, int32_t T, int32_t max_ctx,
                                       const pa_work_item* items, int32_t n_items,
                                       void* workspace, size_t ws_bytes, void* out,
                                       const pa_shape* shape, int32_t* err_flag,
                                       uint64_t never_ns, pa_stream_t stream);

/* ------------------------------------------------------------------ step pipeline
 * A stream of steps under fixed limits, run end to end from host buffers (no counterpart on
 * the pages: the serving loop around "P3: native paged-KV continuous-batching sampler",
 * Design / engine.py, one flat ragged step per engine step). Two slots take alternate steps;
 * each owns device metadata, q / k_new / v_new / out buffers, a workspace, pinned host
 * metadata, and a CUDA graph of its KV write (paged_kv_write, or paged_kv_write_fp8) and
 * attention (paged_attention_step, or its fp8 form) captured once at creation. A submission
 * plans the step on the host (pa_plan_step_shared, so that samples sharing a prompt's blocks
 * read them once, and pa_compute_slots, into the slot's pinned metadata), then queues the
 * uploads of the metadata and of the caller's q / k_new / v_new on one stream, the graph on a
 * second (after the uploads, and after the previous step's kernels), and the read of the
 * output into the caller's buffer on a third. One step's host
 * work and copies so overlap the kernels of the step before it; the kernels run in
 * submission order. Not thread-safe; one pipeline per device and host thread. */
typedef struct pa_pipeline pa_pipeline;

/* Creates a pipeline for steps of exactly B sequences and T query rows, tables of at most
 * max_blocks columns and contexts up to max_ctx, over device pools k_pool / v_pool (bf16, or
 * float8_e4m3fn codes with fp8 != 0 and the per-tensor scales k_scale, v_scale). Allocates its
 * buffers (cudaMalloc, cudaMallocHost) and captures its graphs on the current device; the
 * caller keeps the pools alive until pa_pipeline_destroy. *out owns the pipeline. */
int32_t pa_pipeline_create(const pa_shape* shape, int32_t B, int32_t T, int32_t max_blocks,
                           int32_t max_ctx, void* k_pool, void* v_pool, int32_t fp8,
                           float k_scale, float v_scale, pa_pipeline** out);
/* Waits for the pipeline's outstanding steps and frees everything it allocated (NULL ignored). */
int32_t pa_pipeline_destroy(pa_pipeline* p);
/* Bytes of metadata a submission uploads (the plan padded to pa_plan_max_items_shared,
 * cu_seqlens_q, ctx_lens, the table at max_blocks columns and the slots), or -1 for NULL. */
int64_t pa_pipeline_meta_bytes(const pa_pipeline* p);
/* Queues one step. Host inputs: cu_seqlens_q [B+1] (cu[B] == T), ctx_lens [B] (each <=
 * max_ctx), block_table [B * table_cols] row-major (table_cols <= max_blocks); h_q [T, Hq, D],
 * h_k_new / h_v_new [T, Hkv, D] bf16 and h_out [T, Hq, D] bf16, host memory (pinned memory
 * makes the copies asynchronous). Validates everything before queueing anything (PA_ERR_*
 * as pa_plan_step and pa_compute_slots). *slot receives the slot (0 or 1) the step went to.
 * The caller leaves the step's host buffers alone until pa_pipeline_wait(p, slot) returns, and
 * waits for a slot before submitting two more steps (a submission into a busy slot first
 * waits for that slot's previous step). */
int32_t pa_pipeline_submit(pa_pipeline* p, const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                           const int32_t* block_table, int32_t table_cols, const void* h_q,
                           const void* h_k_new, const void* h_v_new, void* h_out,
                           int32_t* slot);
/* Blocks until the step last submitted into slot has its output in its h_out. */
int32_t pa_pipeline_wait(pa_pipeline* p, int32_t slot);
/* Waits for outstanding steps, then ORs the device error words of both slots into *err. */
int32_t pa_pipeline_device_error(pa_pipeline* p, int32_t* err);

/* ------------------------------------------------------------------ FP8 KV cache
 * K and V stored as float8_e4m3fn codes (1 byte each) with one scale per tensor ("P3: native
 * paged-KV continuous-batching sampler", Review, kv_dtype item: dequantised on read; unscaled
 * e4m3 is lossy, so per-tensor scales. "Finish RL Training Faster: Bitwise-Consistent, ...",
 * 4.2: FP8 storage, one shared write path, one read path for prefill and decode).
 * Pools: uint8 [num_blocks, block_size, Hkv, D], the same geometry as the bf16 pools. The
 * value a code stands for is code_value * scale; the caller chooses the scales (for example
 * amax / 448 of what it writes) and passes the same ones to every write and read of a pool.
 *
 * Write: code = e4m3(x / scale) for each element, the division in fp32 with IEEE rounding,
 * then rounding to the nearest e4m3 value (ties to even) with finite values beyond 448
 * saturating to +-448. Arguments as paged_kv_write, plus k_scale, v_scale (finite, > 0; else
 * PA_ERR_INVALID). Hkv * D must be a multiple of 16. */
int32_t paged_kv_write_fp8(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                           int32_t T, void* k_pool, void* v_pool, float k_scale, float v_scale,
                           const pa_shape* shape, int32_t* err_flag, pa_stream_t stream);

/* Read: paged_attention_step over fp8 pools (head_dim 128 only, else PA_ERR_SHAPE). Every row
 * runs the same tile routine as on a bf16 cache, with f16 operands: the codes are expanded to
 * f16 exactly in shared memory, Q is rounded to f16 (saturating at +-65504) and P is rounded
 * to f16. The K scale multiplies the softmax constant; out = bf16(O * (rcp(l) * v_scale)).
 * Bit identity across batch mixes and between prefill and decode holds within the fp8 path.
 * Arguments, items, workspace and errors as paged_attention_step, plus k_scale, v_scale. */
int32_t paged_attention_step_fp8(const void* q, const void* k_pool, const void* v_pool,
                                 const int32_t* block_table, int32_t max_blocks,
                                 const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                 int32_t B, int32_t T, int32_t max_ctx,
                                 const pa_work_item* items, int32_t n_items, float k_scale,
                                 float v_scale, void* workspace, size_t ws_bytes, void* out,
                                 const pa_shape* shape, int32_t* err_flag, pa_stream_t stream);

/* Allocation-free variant of paged_attention_step (no counterpart on the pages: it is a
 * deployment convenience of this library). Same arguments, meaning and result as
 * paged_attention_step, minus the workspace: the split partials go to a fixed device array of
 * PA_STATIC_SCRATCH_BYTES that the library itself holds on every GPU that loads it, until the
 * process exits. It is meant for callers that cannot allocate device memory when they run a
 * step: a serving process that reserves all GPU memory at start-up and allows no later
 * cudaMalloc, a plug-in that only receives tensors from its host framework, or a loop that
 * cannot afford cudaMalloc's implicit synchronisation. It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *   - Limit: a step whose partials need more than PA_STATIC_SCRATCH_BYTES (see
 *     pa_workspace_bytes(shape, T, max_ctx); steps with max_ctx <= PA_SPLIT_TOKENS need none)
 *     returns PA_ERR_WORKSPACE and launches nothing.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current); make that first call before any stream capture.
 *   - Every call on a device shares the one array, and it keeps whatever the last call left
 *     there. Nothing in it needs to start at zero for a plan from pa_plan_step (or one that
 *     meets the list rules of pa_work_item): every partial the combine reads is then written
 *     earlier in the same call. A plan that leaves out an item of a multi-split decode row
 *     gives an undefined result for that row, which may fold stale partials of an earlier
 *     call, another caller's included. Calls whose kernels overlap on the GPU (different
 *     streams, no ordering between them) race on the array: order them on one stream or with
 *     events. */
#define PA_STATIC_SCRATCH_BYTES (32u << 20)
int32_t paged_attention_step_static_scratch(const void* q, const void* k_pool, const void* v_pool,
                                            const int32_t* block_table, int32_t max_blocks,
                                            const int32_t* cu_seqlens_q, const int32_t* ctx_lens,
                                            int32_t B, int32_t T, int32_t max_ctx,
                                            const pa_work_item* items, int32_t n_items, void* out,
                                            const pa_shape* shape, int32_t* err_flag,
                                            pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
