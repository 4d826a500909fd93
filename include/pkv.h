/*
 * pkv.h -- C ABI of the GB300 (sm_103a) block-paged KV attention library.
 *
 * The operations are those of a vLLM-style block-paged KV cache as the page
 * "paged-cache.md" (mlx-node docs) describes it: each request keeps its keys and
 * values in fixed-size blocks of a per-layer pool (LayerKVPool row of the type
 * table), reached through a per-request block table, and requests that share a
 * prompt prefix point at the same refcounted blocks.  The page "perf.md"
 * (mlx-node docs, paged knob table) names the three steps on the hot path: the
 * graph-native K/V write into pool slots (MLX_PAGED_NATIVE_KV_WRITE), the paged
 * decode that reads the pages through the table, split into partitions whose
 * softmax partials a reducer merges (MLX_PAGED_GRAPH_DECODE_GATHER and the
 * partition-rule paragraphs), and a prefill chunk attending a paged prefix
 * (gather_kv_for_prefill_chunk).
 *
 * Conventions (the plainest reading where the pages are silent):
 *   - pool layout [num_blocks][num_kv_heads][block_size][head_dim], row major,
 *     element type pkv_dtype; the K and V pools share the shape;
 *   - slot = block_id * block_size + offset;  a negative slot is skipped;
 *   - block tables: int32 [batch][max_blocks_per_seq]; entry j of row r is the
 *     physical block of the row's positions j*block_size .. +block_size-1;
 *     -1 is the null sentinel of expired sliding blocks (never read);
 *   - seq_lens[r] counts every token of row r including those appended this
 *     step; the decode query of row r sits at position seq_lens[r] - 1;
 *   - grouped-query attention: q head h reads kv head h / (Hq / Hkv);
 *   - window W > 0: a query at absolute position p attends positions
 *     max(0, p - W + 1) .. p; W = 0 is full attention;
 *   - an empty key range (seq_len 0) yields an all-zero output row;
 *   - softmax scores are scale * (q . k); accumulation is fp32.
 *
 * Ownership and errors.  Every pointer named "device" is device memory owned
 * by the caller; the library allocates no device memory.  All calls are
 * asynchronous on the caller's stream.  Arguments are checked on the host
 * before anything is launched and a bad one returns PKV_ERR_INVALID_ARG (a
 * combination that is not built returns PKV_ERR_UNSUPPORTED) with nothing
 * enqueued.  Faults that only the device can see (an out-of-pool block id, a
 * slot past the pool, a length past the table) never trap: the element is
 * skipped or masked and a bit is OR-ed into *dev_status (device int32, may be
 * NULL), see PKV_DEV_*.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,
    PKV_ERR_UNSUPPORTED = 2,
    PKV_ERR_CUDA = 3,
    PKV_ERR_WORKSPACE = 4,
    PKV_ERR_OUT_OF_BLOCKS = 5 /* block allocator: the pool (at its maximum) cannot hold the request */
} pkv_status;

/*
 * Element type of a pool.  PKV_FP8_E4M3: the FP8 KV cache with per-layer
 * scales of "perf.md" (quantisation scheme table, FP8 KV cache row).  Each
 * element is one E4M3 code c ("FP8 Formats for Deep Learning", E4M3: bias 7,
 * 3 mantissa bits, max 448, S.1111.111 = NaN) holding e4m3(c) * scale, with
 * pool.k_scale for the K pool and pool.v_scale for the V pool.  Queries,
 * outputs and appended rows of an FP8 pool are bf16.  An FP8 pool has
 * block_size 16 and head_dim 64, 128 or 256; its (block, kv head) tiles are
 * 16 * head_dim bytes in the operand order of the m16n8k16 tensor-core
 * product (so each thread's operands are 16 consecutive bytes):
 *   K byte of (token t, dim d):  (d/64)*1024 + (t/8)*512 + ((t%8)*4 + c)*16 + ((d%64)/16)*4 + j
 *       with k = d%16, c = (k%8)/2, j = k%2 + 2*(k/8);
 *   V byte of (token t, dim d):  (d/32)*512 + ((d%8)*4 + c)*16 + ((d%32)/8)*4 + j
 *       with c = (t%8)/2, j = t%2 + 2*(t/8).
 */
typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
#define PKV_DEV_BAD_BLOCK 1  /* a table entry inside a row's key range is < 0 or >= num_blocks:
                                that block is treated as fully masked */
#define PKV_DEV_BAD_SLOT 2   /* an append slot >= num_blocks * block_size: token skipped */
#define PKV_DEV_BAD_LEN 4    /* seq_len < 0, > max_blocks_per_seq * block_size or > max_seq_len,
                                or a prefill chunk longer than its row: the row is clamped */
#define PKV_DEV_BAD_PREFIX 8 /* a row of a shared-prefix group does not hold the group's
                                prefix blocks, or is shorter than the prefix */
#define PKV_DEV_TIMEOUT 16   /* a pipeline wait gave up after its time limit; the outputs of
                                that call are not valid */
#define PKV_DEV_Q_RANGE 32   /* FP8 pools: a query element's magnitude is past 65504, the f16
                                range the FP8 path computes q . k in; outputs not valid */

/* One layer's K/V block pool (device pointers, 16-byte aligned). */
typedef struct {
    void *k;
    void *v;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    pkv_dtype dtype;
    float k_scale;  /* PKV_FP8_E4M3 only (finite, > 0): the layer's K and V scales */
    float v_scale;
} pkv_pool;

/*
 * Shared-prefix descriptor ("paged-cache.md": requests share refcounted blocks
 * for a common prompt prefix).  Rows of one group hold the same physical
 * blocks in their first prefix_blocks[group] table entries; the decode reads
 * those blocks once for all rows of the group.  pkv_prefix_groups_host derives
 * the device arrays from the block tables.
 */
typedef struct {
    int32_t num_groups;            /* host: number of groups (0 = none) */
    int32_t max_group_rows;        /* host: upper bound on the rows of any group */
    int32_t max_prefix_blocks;     /* host: upper bound on prefix_blocks[] */
    const int32_t *group_of_row;   /* device int32 [batch]: group of each row, -1 = none */
    const int32_t *prefix_blocks;  /* device int32 [num_groups]: shared leading blocks */
} pkv_prefix_desc;

/*
 * Append ("perf.md", paged knob table, MLX_PAGED_NATIVE_KV_WRITE: new K/V rows
 * are written into their pool slots).  For token t with slot s >= 0:
 *   pool.k[s / bs][h][s % bs][:] = k_new[t][h][:]   for every kv head h (same for v).
 * k_new, v_new: device [num_tokens][num_kv_heads][head_dim] of pool.dtype (bf16
 * for an FP8 pool).  slot_mapping: device int32 [num_tokens].  Bit-exact copy;
 * into an FP8 pool each element x is stored as the E4M3 code nearest to the
 * float32 quotient x / scale (ties to the even code, magnitudes past 448
 * saturate to +-448), at its byte of the tile.  Two tokens naming one slot
 * race (the caller must not do that).
 */
pkv_status paged_kv_append(const pkv_pool *pool, const int32_t *slot_mapping, int32_t num_tokens,
                           const void *k_new, const void *v_new, int32_t *dev_status,
                           pkv_stream_t stream);

/*
 * Bytes of device workspace paged_decode_attention needs for these sizes on the
 * current device (the split plan depends on its SM count).  prefix may be NULL.
 * The size does not depend on the pool's dtype: f32, bf16 and FP8 pools of
 * the same sizes take the same workspace (the plan's partial slots per row do
 * not change with the dtype; only how many CTAs share a prefix group's rows
 * does).  Returns 0 for invalid sizes.
 */
size_t paged_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t max_seq_len,
                                   int32_t window, const pkv_prefix_desc *prefix);

/*
 * Batched paged decode attention ("perf.md", MLX_PAGED_GRAPH_DECODE_GATHER and
 * the partition-rule paragraphs; "paged-cache.md", Gemma4 coordinator section
 * for sliding groups).  For every row r and q head h:
 *   out[r][h][:] = softmax_p(scale * q[r][h] . K_p) . V_p
 * over the positions p of row r in its key range (see the conventions above),
 * K_p/V_p read through block_tables from kv head h / (Hq / Hkv).
 *   q, out:        device [batch][num_q_heads][head_dim], pool.dtype (bf16 for FP8)
 *   block_tables:  device int32 [batch][max_blocks_per_seq]
 *   seq_lens:      device int32 [batch]
 *   max_seq_len:   host upper bound on seq_lens (sizes the split plan)
 *   workspace:     device, >= paged_decode_workspace_size(...) bytes, 256-byte aligned
 *   prefix:        NULL, or a shared-prefix descriptor (window must be 0)
 * Split-KV: each row's key range is cut into fixed-size runs of blocks; every
 * run yields fp32 (max, sum, weighted values) partials that a second kernel
 * merges.  The cut depends only on the sizes and the SM count, so a call is
 * bit-reproducible.  Built: f32, bf16 and FP8; block_size 16 for bf16 and FP8
 * (any block_size <= 64 for f32); head_dim 64, 128, 256; Hq / Hkv <= 16.  FP8
 * pools: q . k is computed with q converted to f16 (exact for bf16 values of
 * magnitude 2^-14 .. 65504; smaller ones round to f16 subnormals, larger ones
 * set PKV_DEV_Q_RANGE) against the exact code values, the scales applied in
 * fp32; probabilities enter P.V as f16.
 */
pkv_status paged_decode_attention(const void *q, int32_t num_q_heads, const pkv_pool *pool,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *seq_lens, int32_t batch, int32_t max_seq_len,
                                  int32_t window, float scale, void *out, void *workspace,
                                  size_t ws_bytes, const pkv_prefix_desc *prefix,
                                  int32_t *dev_status, pkv_stream_t stream);

/*
 * Fused decode over several groups of a model's layers ("paged-cache.md",
 * Gemma4 grouped-coordinator passage: full-attention and sliding-window groups
 * keep pools and block tables of their own and advance together; "perf.md",
 * paged knob table: a sliding group's decode reads from its first live block).
 * Each group is one paged_decode_attention call (prefix = NULL) over the same
 * batch and q heads: its own q, out, pool, tables, lengths, window and scale.
 * All groups run in one split launch and one merge launch, so a small group
 * (a sliding window) fills the gaps of a large one instead of running after
 * it.  The groups' pools must share dtype (bf16 or FP8; f32 returns
 * PKV_ERR_UNSUPPORTED), head_dim, block_size and num_kv_heads, else
 * PKV_ERR_INVALID_ARG.  Every group's output equals, bit for bit, that of its
 * own paged_decode_attention call.
 *   groups:    host array of n_groups (1 .. PKV_MAX_DECODE_GROUPS) descriptors
 *   workspace: device, >= paged_decode_groups_workspace_size(...) bytes,
 *              256-byte aligned
 */
#define PKV_MAX_DECODE_GROUPS 4

typedef struct {
    const void *q;                /* device [batch][num_q_heads][head_dim] */
    void *out;                    /* device [batch][num_q_heads][head_dim] */
    pkv_pool pool;                /* the group's pool (by value) */
    const int32_t *block_tables;  /* device int32 [batch][max_blocks_per_seq] */
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;      /* device int32 [batch] */
    int32_t max_seq_len;          /* host bound on seq_lens */
    int32_t window;               /* 0 = full attention */
    float scale;
} pkv_decode_group;

/* Bytes of workspace for paged_decode_attention_groups (0 for invalid sizes). */
size_t paged_decode_groups_workspace_size(const pkv_decode_group *groups, int32_t n_groups,
                                          int32_t batch, int32_t num_q_heads);

pkv_status paged_decode_attention_groups(const pkv_decode_group *groups, int32_t n_groups,
                                         int32_t batch, int32_t num_q_heads, void *workspace,
                                         size_t ws_bytes, int32_t *dev_status,
                                         pkv_stream_t stream);

/*
 * Allocation-free decode.  The pages have no counterpart: this entry point
 * exists for callers that cannot allocate device memory where they call the
 * library (a plug-in inside a framework that owns all device memory, a serving
 * loop that bans cudaMalloc on its hot path) and so have no workspace to pass.
 * It is paged_decode_attention with its scratch taken from a fixed array in
 * the library's device image, PKV_NO_ALLOC_SCRATCH_BYTES long, which every GPU
 * that loads the library holds until the process exits.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 *     routine.
 *   - The scratch is that of the CURRENT device: make the device that holds
 *     the pools and buffers current (cudaSetDevice) before the call.  The
 *     first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and keeps it for the life of the process; make
 *     that first call before any stream capture.  After cudaDeviceReset the
 *     kept address is stale: do not call this entry point on that device
 *     again in the same process.
 *   - Sizes whose workspace (paged_decode_workspace_size) exceeds
 *     PKV_NO_ALLOC_SCRATCH_BYTES return PKV_ERR_WORKSPACE, nothing enqueued.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind (nothing in it has to start at zero).  Calls that overlap on the
 *     GPU (different streams, or different host threads without ordering)
 *     race on it: order them.
 * Arguments, results and the other errors are those of paged_decode_attention.
 */
#define PKV_NO_ALLOC_SCRATCH_BYTES (16u << 20)

pkv_status paged_decode_attention_no_alloc(const void *q, int32_t num_q_heads,
                                           const pkv_pool *pool, const int32_t *block_tables,
                                           int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                           int32_t batch, int32_t max_seq_len, int32_t window,
                                           float scale, void *out, const pkv_prefix_desc *prefix,
                                           int32_t *dev_status, pkv_stream_t stream);

/* Bytes of device workspace paged_prefill_chunk_attention needs on the
 * current device (0: none).  Two schedules use one, both for bf16 and FP8
 * pools (the size covers either dtype; f32 pools need less):
 *   - short chunks (every C_r <= 128 / (Hq / Hkv), a speculative-verify step,
 *     say) on grids too small to fill the GPU: their key ranges are cut into
 *     runs whose fp32 partials a second kernel merges;
 *   - longer chunks with more (row, kv head, 256-row query tile pair) items
 *     than SMs: one persistent CTA per SM takes an equal share of the items'
 *     64-key tiles (computed on the device from the actual lengths by a
 *     one-CTA plan kernel); an item cut by a CTA boundary is computed in
 *     pieces whose fp32 partials a merge kernel combines.
 * Both cuts depend only on the sizes, the lengths and the SM count, so a call
 * is bit-reproducible. */
size_t paged_prefill_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size, int32_t max_q_len,
                                    int32_t max_seq_len, int32_t window);

/*
 * Chunked prefill against a paged prefix ("perf.md", gather_kv_for_prefill_chunk:
 * a prefill chunk attends the cached prefix through the pages; "paged-cache.md",
 * chunked prefill whose boundaries change the reduction order but not the
 * result).  Row r owns the packed queries cu_q_lens[r] .. cu_q_lens[r+1]-1
 * (C_r of them); its chunk's K/V must already be in the pool (paged_kv_append).
 * Query i of row r sits at p = seq_lens[r] - C_r + i and attends the positions
 * max(0, p - W + 1) .. p (W = 0: 0 .. p), i.e. the whole prefix and the chunk
 * causally.
 *   q, out:      device [cu_q_lens[batch]][num_q_heads][head_dim], pool.dtype
 *                (bf16 for FP8)
 *   cu_q_lens:   device int32 [batch + 1], non-decreasing, cu_q_lens[0] = 0
 *   max_q_len:   host upper bound on C_r;  max_seq_len: host bound on seq_lens
 *   workspace:   device, >= paged_prefill_workspace_size(...) bytes, 256-byte
 *                aligned (NULL when that size is 0)
 * Built: bf16 and FP8, block_size 16, head_dim 128, Hq / Hkv <= 16 (tcgen05 tensor
 * cores, fp32 accumulation in tensor memory; for bf16 pools probabilities
 * enter the P.V product as bf16 hi + lo terms); f32 pools run a CUDA-core
 * kernel.  bf16
 * chunks with max_q_len * (Hq / Hkv) <= 16 (a speculative-verify step) run on
 * the split-KV decode kernel instead, one M-row per (query, head) pair, for
 * head_dim 64, 128 or 256.  FP8 pools: the tensor-core kernel widens the E4M3
 * tiles to f16 in shared memory and multiplies f16 x f16 (the query converted
 * to f16, PKV_DEV_Q_RANGE past 65504), P as one f16 term (2^-11 relative, as
 * in the FP8 decode).
 */
pkv_status paged_prefill_chunk_attention(const void *q, const int32_t *cu_q_lens,
                                         int32_t num_q_heads, const pkv_pool *pool,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *seq_lens, int32_t batch, int32_t max_q_len,
                                         int32_t max_seq_len, int32_t window, float scale,
                                         void *out, void *workspace, size_t ws_bytes,
                                         int32_t *dev_status, pkv_stream_t stream);

/* Static text for a status code. */
const char *pkv_status_string(pkv_status status);

/*
 * Host helper: slot of each (row, position) pair, slot = table[row][pos / bs] * bs
 * + pos % bs.  Pairs whose table entry is missing (-1, past the table, or past
 * the pool) get -1 and make the call return PKV_ERR_INVALID_ARG after filling
 * every slot.  All arrays are host memory.
 */
pkv_status pkv_slot_mapping_host(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 int32_t batch, int32_t num_blocks, const int32_t *rows,
                                 const int32_t *positions, int32_t n, int32_t block_size,
                                 int32_t *slots_out);

/*
 * Host helper, a debug check of a slot mapping before an append: every slot
 * >= 0 of slots[0 .. n-1] lies inside the pool (< num_blocks * block_size)
 * and no two tokens name the same slot.  Two tokens written to one slot would
 * leave whichever store lands last, a race that breaks the run-to-run
 * determinism the mlx-bun notes require of the batched kernels (section
 * "Risks": no atomics, deterministic).  The append itself does not look for
 * repeats.  Returns PKV_OK, or PKV_ERR_INVALID_ARG with *first_bad (may be
 * NULL) the index of the first token at fault in order (for a repeat, the later
 * token of the pair); *first_bad is -1 when the arguments themselves are
 * invalid or nothing is wrong.  Host arrays; allocates host scratch.
 */
pkv_status pkv_slot_mapping_check_host(const int32_t *slots, int32_t n, int32_t num_blocks,
                                       int32_t block_size, int32_t *first_bad);

/*
 * Host helper: shared-prefix groups read off the block tables (host arrays).
 * Rows whose first entry is the same physical block form a group when there
 * are at least two of them; the group's prefix is the longest run of leading
 * entries common to all its rows, cut to blocks that are full in every row
 * (prefix_blocks * block_size <= seq_len: only full blocks are shared).  Groups
 * are numbered by their lowest row.  Writes group_of_row[batch] (-1 = none) and
 * prefix_blocks[0 .. num_groups-1] (capacity batch); returns num_groups, or -1
 * on invalid arguments.
 */
int32_t pkv_prefix_groups_host(const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *seq_lens, int32_t batch, int32_t block_size,
                               int32_t *group_of_row, int32_t *prefix_blocks);

/*
 * Diagnostic: force the decode split size to this many blocks per split
 * (0 = the automatic plan).  Process-wide; for tests of split invariance, in
 * the spirit of the pages' partition-override knob ("perf.md",
 * MLX_PAGED_GROUPED_D512_STRIPES).  Returns the previous value.
 */
int32_t pkv_set_decode_split_blocks(int32_t blocks_per_split);

/*
 * Diagnostic fail-closed drill for the device-side wait timeout (the pages
 * require the paged path to fail closed rather than degrade silently:
 * "paged-cache.md", fail-closed gates of the grouped coordinator;
 * "perf.md", paged knob table, MLX_PAGED_NATIVE_KV_WRITE row, where batched
 * decode hard-errors instead of falling back).  Process-wide, for the
 * launches that follow (bf16 and FP8 decode, tensor-core prefill):
 *   wait_limit_ns: limit of each pipeline data wait, 0 = the default
 *                  (2 s); values above the default are cut to it;
 *   flags:         0, or PKV_DRILL_WITHHOLD_FIRST_LOAD: every pipeline
 *                  leaves its first load unissued, so that the wait for it
 *                  runs out after wait_limit_ns.
 * A wait that runs out sets PKV_DEV_TIMEOUT in the status word; the CTA then
 * waits (with the 2 s default limit) for every copy it did issue to land
 * and for its tensor-core products to finish, and exits.  The call's output
 * is then undefined.  pkv_set_wait_drill(0, 0) restores normal operation.
 * Returns PKV_ERR_INVALID_ARG for unknown flags.
 */
#define PKV_DRILL_WITHHOLD_FIRST_LOAD 1u
pkv_status pkv_set_wait_drill(uint64_t wait_limit_ns, uint32_t flags);

/* Number of splits per row and blocks per split the automatic plan picks for
 * these sizes on the current device (diagnostic; -1 on invalid sizes). */
int32_t pkv_decode_plan(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int32_t max_seq_len, int32_t window,
                        int32_t *blocks_per_split_out);

/*
 * Diagnostic kernel timing and launch counting (no counterpart on the pages:
 * measurement plumbing).  Kernel kinds: */
typedef enum {
    PKV_KERNEL_APPEND = 0,
    PKV_KERNEL_DECODE_PREFIX = 1, /* shared-prefix read-once decode */
    PKV_KERNEL_DECODE_SPLIT = 2,  /* per-row split-KV decode */
    PKV_KERNEL_DECODE_COMBINE = 3,
    PKV_KERNEL_PREFILL = 4,
    PKV_KERNEL_KINDS = 5
} pkv_kernel_kind;

/* Bit k of kind_mask enables timing of kernel kind k: each such launch is
 * bracketed by two CUDA events recorded on its stream (the events are host
 * objects; no device memory is allocated).  Resets the accumulated records.
 * Up to 65536 launches are recorded.  Not for use inside stream capture. */
pkv_status pkv_profile_enable(uint32_t kind_mask);

/* Changes which kinds are timed without resetting the records: timing only
 * some launches (one in N, say) keeps the events, which end the overlap of a
 * launch with its neighbours, off the other launches. */
pkv_status pkv_profile_mask(uint32_t kind_mask);

/* Launches recorded for a kind and their summed device time in milliseconds.
 * Waits for the recorded events. */
pkv_status pkv_profile_read(int32_t kind, int64_t *launches, double *total_ms);

/* The device times (milliseconds) of the recorded launches of a kind, in
 * launch order: up to `cap` of them go to ms_out (host array), *launches
 * receives how many were recorded in all.  Waits for the recorded events. */
pkv_status pkv_profile_times(int32_t kind, float *ms_out, int64_t cap, int64_t *launches);

/* Number of kernels this process has launched through the library. */
int64_t pkv_launch_count(void);

/* Library version string. */
const char *pkv_version(void);

/* ========================================================================
 * Host block allocator ("paged-cache.md": the BlockAllocator row of the
 * component table - per-block refcounts, LRU eviction, a prefix-hash table for
 * reuse across requests; the PagedKVCacheAdapter per-request lifecycle; the
 * grow-on-demand rule of the pool-sizing passage; a block enters the prefix
 * table only once it is full).  Host memory only, single-threaded (callers serialise).  It
 * hands out block ids of the caller's device pools; when it grows, the caller
 * grows the pools to pkv_allocator_stats' num_blocks before using new ids.
 *
 * Block identity: a full block's hash is FNV-1a (64-bit) over the
 * little-endian bytes of its parent's hash (0 for the first block), its
 * block_size token ids (int32) and one 64-bit extra key (0 for text-only
 * blocks; image digests and similar go there), so a block's identity carries
 * its whole prefix.  Equal hashes are taken as equal blocks.
 *
 * Block states: free (lowest id handed out first); in use (refcount = the
 * requests whose table holds it); cache-only (published, refcount 0, on an LRU
 * list ordered by release time).  A reservation that needs k new blocks when
 * fewer than k are free:
 *   - if free + cache-only blocks cannot cover k and the pool is below its
 *     maximum, the pool grows once first, to
 *       min(max_blocks, max(2 * current, current + (k - free)));
 *   - then cache-only blocks are evicted, least recently released first
 *     (they leave the prefix table);
 *   - if k blocks are still not there, PKV_ERR_OUT_OF_BLOCKS and nothing
 *     changes.
 * ======================================================================== */
typedef struct pkv_allocator pkv_allocator;

/* block_size tokens per block; the pool starts at initial_blocks and grows up
 * to max_blocks (initial_blocks <= max_blocks).  NULL on invalid sizes. */
pkv_allocator *pkv_allocator_create(int32_t block_size, int32_t initial_blocks,
                                    int32_t max_blocks);
void pkv_allocator_destroy(pkv_allocator *a);

/* A new request (reset_for_new_request): its id, >= 0, with an empty table. */
int32_t pkv_allocator_begin(pkv_allocator *a);

/* find_cached_prefix: for a fresh request with prompt tokens[0..n_tokens),
 * walk the prompt's full blocks in order, hashing each on its parent, and take
 * every block found in the prefix table until the first miss (refcount + 1; a
 * cache-only block leaves the LRU).  extra_keys: NULL, or one key per full
 * block.  *cached_tokens = the tokens covered (a multiple of block_size). */
pkv_status pkv_allocator_find_cached_prefix(pkv_allocator *a, int32_t req,
                                            const int32_t *tokens, int32_t n_tokens,
                                            const uint64_t *extra_keys,
                                            int32_t *cached_tokens);

/* allocate_suffix_blocks: extend the request's table with new blocks until it
 * covers n_tokens tokens (grow / evict as above).  PKV_ERR_OUT_OF_BLOCKS
 * leaves the table as it was. */
pkv_status pkv_allocator_reserve(pkv_allocator *a, int32_t req, int32_t n_tokens);

/* record_tokens + register_full_blocks_for_reuse: tokens[0..n_tokens) are the
 * request's tokens so far (n_tokens <= its table's capacity).  Each full block
 * of the table not yet published is hashed and published, unless the prefix
 * table already holds that hash under another block (this block then stays
 * private to the request).  extra_keys as above. */
pkv_status pkv_allocator_publish(pkv_allocator *a, int32_t req, const int32_t *tokens,
                                 int32_t n_tokens, const uint64_t *extra_keys);

/* Sliding-window groups ("paged-cache.md", Gemma4 row and coordinator
 * passage: expired sliding blocks are replaced by a null sentinel): every
 * block of the table that lies wholly before first_live_token loses the
 * request's reference (as in release) and its table entry becomes -1, the
 * sentinel the decode never reads.  Table positions are kept (absolute). */
pkv_status pkv_allocator_expire(pkv_allocator *a, int32_t req, int32_t first_live_token);

/* release_request: every block of the table loses a reference; a published
 * block at refcount 0 becomes cache-only (LRU tail), an unpublished one free.
 * The id is retired. */
pkv_status pkv_allocator_release(pkv_allocator *a, int32_t req);

/* The request's block table: min(cap, n) ids into out (host), n into *n_blocks. */
pkv_status pkv_allocator_table(const pkv_allocator *a, int32_t req, int32_t *out, int32_t cap,
                               int32_t *n_blocks);

/* Refcount of one block (-1 for an id outside the pool). */
int32_t pkv_allocator_refcount(const pkv_allocator *a, int32_t block);

/* Pool counters: current block count, free, cache-only, grows so far. */
pkv_status pkv_allocator_stats(const pkv_allocator *a, int32_t *num_blocks, int32_t *free_blocks,
                               int32_t *cached_blocks, int32_t *grows);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
