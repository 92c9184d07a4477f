/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-attention library.
 *
 * PagedAttention keeps each sequence's KV cache in fixed-size physical blocks
 * and reaches them through a per-sequence block table that maps logical block
 * i to a physical block anywhere in the pool ("PagedAttention: memetakan blok
 * KV logis ke memori fisik tidak kontigu", section "Urutan logis dipisahkan
 * dari penempatan fisik"; "Apa itu PagedAttention?", section "Cara kerja
 * PagedAttention: Blok halaman non-kontigu").  The attention kernel follows
 * the block table before it loads K and V (nalar.dev, section "Kernel
 * attention harus mengikuti block table"); the attention equation itself is
 * unchanged (same page, opening section).
 *
 * Conventions for every call
 * --------------------------
 *  - Return value: PA_OK (0) or a PA_ERR_* code; pa_last_error_string()
 *    gives the message of the last failing call on the calling thread.
 *  - Tensors are caller-owned DEVICE pointers (unless a parameter says host).
 *    The library never allocates device memory in an op call and keeps no
 *    pointer after it returns.
 *  - Ops are asynchronous on the given stream (a cudaStream_t; NULL = the
 *    legacy default stream).  The status covers argument checks and launch
 *    errors only; device-side errors (an out-of-range block id, a pipeline
 *    wait that ran out) are recorded in a device error word read by
 *    pa_device_error().
 *  - dtype: PA_BF16 (bfloat16) or PA_F32 (float32) for q, K/V caches and
 *    outputs.  Accumulation is always fp32.
 *  - Cache layout (both K and V): [num_blocks][Hkv][block_size][head_dim],
 *    contiguous, so one (block, KV head) is block_size*head_dim contiguous
 *    elements.  Pool base pointers must be 16-byte aligned.
 *  - GQA: query head h reads KV head h / (Hq / Hkv).
 *  - Supported shapes: head_dim 64 or 128; Hq/Hkv in {1, 2, 4, 8};
 *    block_size a power of two in [8, 128].
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pa_stream_t; /* same type as cudaStream_t */

enum {
    PA_OK = 0,
    PA_ERR_INVALID = 1,     /* bad argument, shape or (validate mode) metadata */
    PA_ERR_OOM = 2,         /* block manager: not enough free blocks or host memory */
    PA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    PA_ERR_UNSUPPORTED = 4, /* valid request this build has no kernel for */
    PA_ERR_DEVICE = 5       /* pa_device_error found a device-side error */
};

enum { PA_BF16 = 0, PA_F32 = 1 };

/* device error word bits (pa_device_error) */
enum {
    PA_DEVERR_BAD_BLOCK = 1, /* a block-table entry was outside [0, num_blocks) */
    PA_DEVERR_TIMEOUT = 2    /* a bounded pipeline wait ran out; output invalid */
};

/* Message of the last failing call on this thread ("" if none). */
const char *pa_last_error_string(void);

/* Library ABI version (incremented on any signature change). */
int pa_version(void);

/*
 * Validate mode (off by default).  When on, every op first copies its
 * metadata (slot_mapping, block_table, context_lens, copy pairs) to the host
 * and checks it: slots and block ids inside the pool, no duplicate slots in
 * one reshape call, copy pairs disjoint, context lengths in (0, table
 * capacity].  It synchronizes the stream, so it is for debugging and tests.
 */
int pa_set_validate(int on);

/*
 * Read (and, if clear != 0, reset) the device error word of the current
 * device.  Synchronizes the stream.  *bits receives PA_DEVERR_* bits.
 * Returns PA_ERR_DEVICE if any bit was set, else PA_OK.
 */
int pa_device_error(int *bits, int clear, pa_stream_t stream);

/*
 * pa_reshape_and_cache -- store the new tokens' K and V into their slots.
 * Only the new token's K/V is computed and stored; earlier tokens are read
 * back from the cache ("KV Cache dan PagedAttention: Apa Fungsinya dan
 * Mengapa Itu Penting", section "Apa itu KV Cache?").
 *   k_new, v_new  [T][Hkv][head_dim]               (dtype)
 *   k_cache, v_cache  pool as above, written in place
 *   slot_mapping  int64 [T]: slot = physical_block * block_size + offset;
 *                 a negative slot is padding and is skipped
 * Effect: k_cache[slot/bs][h][slot%bs][:] = k_new[t][h][:] (same for V), bit
 * exact.  Duplicate slots in one call are a caller error (undefined which
 * token wins; PA_ERR_INVALID in validate mode).
 */
int pa_reshape_and_cache(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t T, int64_t num_blocks, int Hkv,
                         int block_size, int head_dim, int dtype, pa_stream_t stream);

/*
 * pa_copy_blocks -- copy-on-write support: for each pair (src, dst), physical
 * block dst of BOTH caches becomes a byte copy of block src ("Apa itu
 * PagedAttention?", section "Cara kerja PagedAttention", item 3; nalar.dev,
 * section "Sharing blok dapat menghindari duplikasi state KV").
 *   pairs  int64 [n][2] device array of (src, dst) block ids
 * No dst may equal any src or another dst in the same call (PA_ERR_INVALID in
 * validate mode).  Bit exact.
 */
int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int64_t n,
                   int64_t num_blocks, int Hkv, int block_size, int head_dim, int dtype,
                   pa_stream_t stream);

/*
 * pa_swap_blocks -- move whole blocks between two pools of the same shape,
 * e.g. swap a sequence's blocks out to pinned host memory and back: when the
 * device pool is full, small pages go to the CPU instead of whole sequences
 * ("KV Cache and PagedAttention: Why Your LLM Server Slows Down", section
 * "How PagedAttention fixes this", fine-grained eviction).
 * For each pair (src, dst): block dst of the destination pools becomes a byte
 * copy of block src of the source pools, K and V.  Each pool (and the pairs
 * array) may be device memory or pinned host memory (reached through its
 * mapped device alias); pageable host memory is rejected.
 *   pairs  int64 [n][2] (src block in the source pool, dst block in the
 *          destination pool); destinations must be distinct (validate mode).
 * Bit exact; asynchronous on the stream like every op.
 */
int pa_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                   const int64_t *pairs, int64_t n, int64_t src_num_blocks,
                   int64_t dst_num_blocks, int Hkv, int block_size, int head_dim, int dtype,
                   pa_stream_t stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs: the
 * per-item partial counts (4 bytes per (sequence, query head), padded to a
 * multiple of 256 bytes) and the fp32 partials (max, sum and weighted values)
 * of up to partitions-of-the-table-capacity + 1 segments per (sequence,
 * query head).  Non-zero for every B > 0 (0 for B = 0).  partition_tokens as
 * for pa_decode (0 = library default).  PA_ERR_INVALID on bad sizes or when
 * the size does not fit in size_t.
 */
int pa_decode_workspace_size(int B, int Hq, int head_dim, int max_blocks_per_seq,
                             int block_size, int partition_tokens, size_t *bytes);

/* kernels pa_decode can launch (pa_decode_kernel_for) */
enum { PA_DECODE_PERSISTENT = 1, PA_DECODE_GRID = 2 };

/*
 * pa_decode_kernel_for -- which kernel pa_decode launches for a batch of these
 * sizes on the current device.  The choice depends on the sizes only (never
 * on context lengths or device data), so one batch shape always runs the
 * same kernel:
 *   PA_DECODE_PERSISTENT  one persistent grid (2 CTAs of 4 warps per SM) that
 *                         splits the batch's (sequence, KV head, 16-token
 *                         tile) units evenly over its warps;
 *   PA_DECODE_GRID        one CTA per (sequence, KV head, partition), then a
 *                         merge kernel; chosen when B * Hkv * (partitions of
 *                         the table capacity) is at most 1.75 times the
 *                         persistent grid's warp count (little work), and for
 *                         B > 4096.
 * Both meet the same error bound; their results may differ in the last bits
 * (another order of the partial sums).  Arguments as for pa_decode;
 * *kernel receives PA_DECODE_PERSISTENT or PA_DECODE_GRID.  PA_ERR_INVALID
 * on bad sizes, PA_ERR_CUDA without a current device.
 */
int pa_decode_kernel_for(int B, int Hkv, int max_blocks_per_seq, int block_size,
                         int partition_tokens, int *kernel);

/* per-tile math of the persistent decode kernel (pa_decode_tile_for) */
enum { PA_DECODE_TILE_CUDA_CORE = 1, PA_DECODE_TILE_TENSOR_CORE = 2 };

/*
 * pa_decode_tile_for -- how the persistent decode kernel computes a tile of
 * one (sequence, KV head) for these shapes (the grid kernel always uses the
 * CUDA-core tile):
 *   PA_DECODE_TILE_TENSOR_CORE  bf16 with groups of 4 or 8 query heads per KV
 *       head (and num_blocks * Hkv * block_size < 2^31): 16-token tiles by
 *       2D tensor copies (128-byte swizzle); scores and the weighted sum of
 *       values by warp-level bf16 tensor-core MMAs with fp32 accumulation
 *       (the group's heads are the N = 8 columns; softmax weights enter as a
 *       bf16 hi + lo pair);
 *   PA_DECODE_TILE_CUDA_CORE    every other case: packed fp32 FMAs and warp
 *       shuffles.
 * Both meet the same error bound.  PA_ERR_INVALID on bad shapes.
 */
int pa_decode_tile_for(int Hq, int Hkv, int head_dim, int block_size, int64_t num_blocks,
                       int dtype, int *tile);

/*
 * pa_decode -- paged decode attention: one query token per sequence.
 * For sequence b with context length L = context_lens[b] (the newest token,
 * already stored by pa_reshape_and_cache, included) and query head h:
 *   o[b][h] = sum_{j<L} exp(s_j - max s) V_b[j][h/g] / sum_j exp(s_j - max s),
 *   s_j = scale * (q[b][h] . K_b[j][h/g])
 * where token j of sequence b lives in physical block
 * block_table[b][j / block_size] at offset j % block_size.  The sum over j
 * is split into partitions of partition_tokens tokens whose partial
 * (max, sum, weighted values) are merged by log-sum-exp when L exceeds one
 * partition.  The result depends only on the logical token order, never on
 * where blocks sit in the pool (bit-identical under any placement).
 *   out, q        [B][Hq][head_dim]                    (dtype)
 *   block_table   int32 [B][max_blocks_per_seq]
 *   context_lens  int32 [B], each in [1, max_blocks_per_seq*block_size]
 *   partition_tokens  0 = default (512), or a positive multiple of both 32
 *                 and block_size
 *   workspace     device buffer of at least pa_decode_workspace_size bytes,
 *                 16-byte aligned; its contents on entry do not matter (every
 *                 partial and per-item count is written before it is read)
 *                 and it holds scratch afterwards.  Calls that may overlap on
 *                 the GPU need separate workspaces.
 * Launches: the decode grid (persistent or grid kernel, pa_decode_kernel_for)
 * and a kernel that merges the partials of items split across warps or
 * partitions.  Each is launched as a programmatic dependent of the kernel
 * before it in the stream: it may start while that kernel drains, and waits
 * for that kernel to complete before it reads any input.
 */
int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, int max_blocks_per_seq, const int32_t *context_lens,
              int B, int Hq, int Hkv, int head_dim, int block_size, int64_t num_blocks,
              float scale, int partition_tokens, void *workspace, size_t workspace_bytes,
              int dtype, pa_stream_t stream);

/*
 * pa_decode_contiguous -- the decode of pa_decode over a plain contiguous
 * cache, for measuring what paging costs: each sequence reserves max_len
 * slots up front, the reservation that paging replaces ("Apa itu
 * PagedAttention?", section "Masalah fragmentasi memori KV Cache
 * konvensional"), so no block table is read and no address depends on a
 * table entry.  Following the block table is the cost paging adds
 * ("PagedAttention: memetakan blok KV logis ke memori fisik tidak kontigu",
 * section "Kernel attention harus mengikuti block table").  The kernel is
 * pa_decode's persistent kernel with the same tiles and split; only the
 * address of a tile differs.
 *   k, v   [B][Hkv][max_len][head_dim] device arrays (dtype); token j of
 *          sequence b, KV head h at row (b * Hkv + h) * max_len + j
 *   max_len  a positive multiple of 32; context_lens[b] in [1, max_len]
 *   workspace  at least pa_decode_contiguous_workspace_size bytes
 * Other arguments and the result as for pa_decode.  At most 4096 sequences
 * (PA_ERR_UNSUPPORTED beyond).
 */
int pa_decode_contiguous_workspace_size(int B, int Hq, int head_dim, int max_len,
                                        int partition_tokens, size_t *bytes);
int pa_decode_contiguous(void *out, const void *q, const void *k, const void *v,
                         const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                         int max_len, float scale, int partition_tokens, void *workspace,
                         size_t workspace_bytes, int dtype, pa_stream_t stream);

/*
 * pa_decode_shared -- pa_decode for a batch in which groups of sequences share
 * the physical blocks of a common prefix: a system prompt, or the history of
 * parallel-sampling branches forked from one parent.  A shared block is one
 * physical copy that serves every sequence referencing it ("PagedAttention:
 * memetakan blok KV logis ke memori fisik tidak kontigu", section "Sharing
 * blok dapat menghindari duplikasi state KV"; "Apa itu PagedAttention?",
 * section "Cara kerja PagedAttention", item 3).  Here the shared part is also
 * READ once per (group, KV head): a prefix kernel streams the group's shared
 * blocks once through shared memory and computes the attention partials
 * (max, sum, weighted values) of every member's query heads against them on
 * tensor cores; the decode then covers each member's private tokens only and
 * merges the two parts by log-sum-exp.
 * Same arguments and result as pa_decode (within the same error bound: the
 * sums are taken in another order, so the bits may differ from pa_decode's),
 * plus the groups:
 *   shared_len    int32 [B] device: tokens at the start of sequence b covered by
 *                 its group's shared blocks; a positive multiple of block_size
 *                 below context_lens[b] for a member, 0 for a sequence in no
 *                 group.  All members of a group have the same value and the
 *                 same first shared_len / block_size block-table entries (the
 *                 first member's row is read for the shared blocks).
 *   group_start   int32 [G+1] device: the members of group g are
 *                 group_seqs[group_start[g] .. group_start[g+1]).
 *   group_seqs    int32 [num_members] device: batch rows of the members; a
 *                 sequence belongs to at most one group.
 *   G, num_members, max_group_size, max_shared_len: host ints bounding the
 *                 arrays (max_group_size >= every group's size,
 *                 max_shared_len >= every shared_len).
 *   workspace     at least pa_decode_shared_workspace_size bytes.
 * Validate mode checks every rule above.  Calls that cannot take the shared
 * path (fp32, batches that pa_decode_kernel_for sends to the grid kernel,
 * pools of 2^31 rows or more) decode every sequence whole, which gives the
 * same result.  Launches (each a programmatic dependent of the one before):
 * block sizes 8..64: the decode grid, the tcgen05 prefix kernel (it reads none
 * of the decode's results: the decode grid releases it at its start, so its
 * CTAs take the SMs the decode leaves, and it waits for that grid only before
 * exiting), the merge (released at the prefix kernel's start; it waits for
 * that kernel before it reads anything); other block sizes: the warp-level
 * prefix kernel, the decode grid, the merge.
 * Outside validate mode, a member whose own shared_len is not a positive
 * multiple of block_size below its context length is decoded whole and
 * PA_DEVERR_BAD_BLOCK is recorded; members that disagree with their group's
 * first member (another shared_len or other shared blocks) give undefined
 * output (PA_DEVERR_BAD_BLOCK is recorded for a differing shared_len; other
 * blocks are only caught by validate mode).
 */
int pa_decode_shared_workspace_size(int B, int Hq, int head_dim, int max_blocks_per_seq,
                                    int block_size, int partition_tokens, int max_shared_len,
                                    size_t *bytes);
int pa_decode_shared(void *out, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, int max_blocks_per_seq,
                     const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                     int block_size, int64_t num_blocks, float scale, int partition_tokens,
                     const int32_t *shared_len, const int32_t *group_start,
                     const int32_t *group_seqs, int G, int num_members, int max_group_size,
                     int max_shared_len, void *workspace, size_t workspace_bytes, int dtype,
                     pa_stream_t stream);

/*
 * pa_decode_shared_forks -- pa_decode_shared for a batch that also holds
 * forked children ("Apa itu PagedAttention?", section "Cara kerja
 * PagedAttention", item 3: a forked branch shares its parent's blocks until
 * it writes; "PagedAttention: memetakan blok KV logis ke memori fisik tidak
 * kontigu", section "Sharing blok dapat menghindari duplikasi state KV").
 * A child shares with its parent not only the group's prefix but every
 * block before its fork point; here those blocks are read once for both:
 * the parent's K/V tiles over [shared_len, fork_len) also serve the child's
 * query heads (bf16, groups of 4 query heads: the tensor-core tile's spare
 * columns), and the child's own reads start at its fork point.
 * Same arguments and result as pa_decode_shared (within the same error
 * bound), plus:
 *   fork_parent   int32 [B] device: for a child, the batch row of its parent,
 *                 else -1.  A parent is no child itself and has one child.
 *   fork_len      int32 [B] device: for a child, the tokens whose blocks it
 *                 shares with its parent: a positive multiple of block_size
 *                 in [shared_len, both context lengths), the two table rows
 *                 equal before it.  Ignored for other rows.
 *   workspace     at least pa_decode_shared_forks_workspace_size bytes.
 * Validate mode checks every rule above.  Outside it, a child whose fork
 * does not meet them (or the second child of one parent) reads its whole
 * range itself and PA_DEVERR_BAD_BLOCK is recorded; rows that agree on the
 * numbers but not on the blocks give undefined output.  Other shapes (fp32,
 * groups of 1, 2 or 8 heads, the grid kernel) read every range themselves,
 * with the same result.  Launches as pa_decode_shared.  Measured on a fork
 * step of 320 sequences (64 children, ~256 private tokens each): 11 % fewer
 * DRAM reads than pa_decode_shared but 3.4 us slower per call (the fork
 * tile's per-tile masking and wider partial rows cost more than the reads).
 */
int pa_decode_shared_forks_workspace_size(int B, int Hq, int head_dim, int max_blocks_per_seq,
                                          int block_size, int partition_tokens,
                                          int max_shared_len, size_t *bytes);
int pa_decode_shared_forks(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                           int block_size, int64_t num_blocks, float scale, int partition_tokens,
                           const int32_t *shared_len, const int32_t *group_start,
                           const int32_t *group_seqs, int G, int num_members, int max_group_size,
                           int max_shared_len, const int32_t *fork_parent,
                           const int32_t *fork_len, void *workspace, size_t workspace_bytes,
                           int dtype, pa_stream_t stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory (for example a plug-in whose host program owns all device memory
 * through its own pool, or a latency-critical loop where cudaMalloc, which
 * may synchronize the device, is not allowed).  The pages have no
 * counterpart to this entry point; it only changes where the split-KV
 * workspace comes from.
 * Same arguments and result as pa_decode, without workspace: the library
 * uses a fixed device array of pa_decode_noalloc_capacity() bytes (16 MiB)
 * that every GPU loading the library holds until the process exits.  A
 * batch whose pa_decode_workspace_size exceeds it is rejected with
 * PA_ERR_INVALID.  The first call on a device (with that device current)
 * looks up the array's device address; make it before any stream capture.
 * All calls on a device share the array: calls that overlap on the GPU race
 * and must be serialized by the caller.  Nothing is allocated, no
 * cudaMalloc/cudaFree is called.
 */
size_t pa_decode_noalloc_capacity(void);
int pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_table, int max_blocks_per_seq,
                      const int32_t *context_lens, int B, int Hq, int Hkv, int head_dim,
                      int block_size, int64_t num_blocks, float scale, int partition_tokens,
                      int dtype, pa_stream_t stream);

/*
 * pa_check_wait_timeout -- diagnostic of the device-side failure path: one
 * warp waits, with the same bounded wait (about 2 s) the pipelined kernels
 * use on their copies and hand-offs, on an mbarrier that nothing completes.
 * The wait runs out, PA_DEVERR_TIMEOUT is recorded in the device error word
 * and the kernel returns: nothing faults and the context stays usable.
 * Asynchronous on `stream`; read the outcome with pa_device_error().
 */
int pa_check_wait_timeout(pa_stream_t stream);

/*
 * pa_prefill_chunk -- chunked prefill over paged context ("Melihat Lebih
 * Dalam vLLM v0.7", section "Blueprint Arsitektur 3: Chunked Prefill": a long
 * prompt is cut into chunks of e.g. 512 tokens and run next to decode).
 * Request r has n_r = query_start[r+1]-query_start[r] new query tokens whose
 * K/V are already in the cache; its context length is L_r = context_lens[r]
 * (prior tokens plus the chunk), so new token i sits at absolute position
 * P_r + i with P_r = L_r - n_r and attends to positions 0..P_r+i (causal).
 *   out, q        [query_start[R]][Hq][head_dim]       (bf16 only)
 *   query_start   int32 [R+1] prefix sum of new-token counts
 *   context_lens  int32 [R]
 *   max_query_len host int >= every n_r (sizes the grid)
 */
int pa_prefill_chunk(void *out, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, int max_blocks_per_seq,
                     const int32_t *query_start, const int32_t *context_lens, int R,
                     int max_query_len, int Hq, int Hkv, int head_dim, int block_size,
                     int64_t num_blocks, float scale, int dtype, pa_stream_t stream);

/* kernels pa_prefill_chunk can launch (pa_prefill_kernel_for) */
enum { PA_PREFILL_PERSISTENT_GRID = 1, PA_PREFILL_ITEM_GRID = 2, PA_PREFILL_SIMPLE = 3 };

/*
 * pa_prefill_kernel_for -- which kernel pa_prefill_chunk launches for these
 * sizes (sizes only, never device data; no device needed).  A work item is
 * (request, 256 query rows, KV head).
 *   PA_PREFILL_PERSISTENT_GRID  one CTA per SM (at most one per item), each
 *                               running a list of items dealt longest first
 *                               to the least-loaded CTA; batches of at most
 *                               256 (request, 256-row) pairs and 512 items;
 *   PA_PREFILL_ITEM_GRID        one CTA per item, longest first (larger
 *                               batches);
 *                               both: blocks of 8..64 tokens, tables of at
 *                               most 1024 blocks, fewer than 2^31 pool rows
 *                               of (block, KV head, slot);
 *   PA_PREFILL_SIMPLE           one CTA of 128 threads per 128 rows (every
 *                               other supported size, e.g. 128-token blocks).
 * All three meet the same error bound.  Arguments as for pa_prefill_chunk;
 * *kernel receives the choice.  PA_ERR_INVALID / PA_ERR_UNSUPPORTED as
 * pa_prefill_chunk would return for the sizes.
 */
int pa_prefill_kernel_for(int R, int max_query_len, int Hq, int Hkv, int head_dim,
                          int block_size, int64_t num_blocks, int max_blocks_per_seq,
                          int *kernel);

/* ------------------------------------------------------------------------
 * Host block manager (opaque handle; C++ behind the C ABI).
 *
 * Free list, per-block reference counts, sequences as lists of physical
 * blocks, fork (prefix sharing), append with copy-on-write.  A new block is
 * taken only when a sequence crosses a block boundary ("Melihat Lebih Dalam
 * vLLM v0.7", section "Blueprint Arsitektur 2", item "Alokasi On-Demand");
 * shared blocks stay shared while unchanged and the branch that writes into a
 * shared, partly filled last block gets a copy first (copy-on-write).  A full
 * shared block needs no copy.  Sharing is explicit (fork), never by content.
 *
 * Free-list order: a stack; initially 0..num_blocks-1, or a Fisher-Yates
 * shuffle driven by SplitMix64(seed) when seed != 0; allocation takes the next
 * block of that order and freed blocks are reused first.
 * Every failing call leaves the manager unchanged.  Not thread safe.
 * ---------------------------------------------------------------------- */
typedef struct pa_bm pa_bm;

int pa_bm_create(int64_t num_blocks, int block_size, uint64_t seed, pa_bm **out);
void pa_bm_destroy(pa_bm *bm);

/* New sequence seq holding n_tokens prompt tokens; slots (host int64
 * [n_tokens], may be NULL) receives their slots.  PA_ERR_INVALID if seq
 * exists, PA_ERR_OOM if too few free blocks. */
int pa_bm_add_seq(pa_bm *bm, int64_t seq, int64_t n_tokens, int64_t *slots);

/* child shares all of parent's blocks (refcount + 1 each). */
int pa_bm_fork(pa_bm *bm, int64_t parent, int64_t child);

/* One new token for seq: *slot receives its slot; (*cow_src, *cow_dst) the
 * block copy to run before writing it, or (-1, -1). */
int pa_bm_append(pa_bm *bm, int64_t seq, int64_t *slot, int64_t *cow_src, int64_t *cow_dst);

/* n new tokens (host int64 slots[n]); at most one copy-on-write pair (only
 * the first new token can hit a shared block). */
int pa_bm_append_n(pa_bm *bm, int64_t seq, int64_t n, int64_t *slots, int64_t *cow_src,
                   int64_t *cow_dst);

/* Drop seq; blocks whose refcount reaches 0 return to the free list. */
int pa_bm_free_seq(pa_bm *bm, int64_t seq);

/* Host int32 out[n][max_blocks]: the block table rows of seqs[0..n), padded
 * with 0.  PA_ERR_INVALID if a sequence is unknown or has more blocks. */
int pa_bm_block_table(const pa_bm *bm, const int64_t *seqs, int n, int32_t *out,
                      int max_blocks);

int pa_bm_seq_len(const pa_bm *bm, int64_t seq, int64_t *len);
/* Physical blocks of seq in logical order: out[cap], *n = number of blocks. */
int pa_bm_seq_blocks(const pa_bm *bm, int64_t seq, int32_t *out, int64_t cap, int64_t *n);
int pa_bm_refcount(const pa_bm *bm, int64_t block, int *refcount);
int64_t pa_bm_num_free(const pa_bm *bm);

/*
 * Host fault injection, for tests of the failure path: from now on the k-th
 * point at which a block-manager call may allocate host memory (k = 0: the
 * next one) fails as if memory had run out; the call returns PA_ERR_OOM and
 * leaves the manager unchanged.  One failure per arming; k < 0 disarms.
 * Process-wide, not thread safe; never armed unless a caller arms it.
 */
void pa_bm_inject_alloc_failure(int64_t k);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
