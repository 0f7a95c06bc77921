/*
 * pkv.h -- C ABI of libpkv: a paged KV cache for one GPU (sm_103a).
 *
 * The method, as the pages on paged KV caches describe it:
 *   "04 - Hacia PagedAttention (vista previa)", section "La idea de PagedAttention":
 *     1. the KV cache is cut into fixed-size blocks of B_block tokens (B_block = 16);
 *     2. every sequence keeps a block table: logical block i -> physical block X;
 *     3. to extend a sequence by one token, write into its last block if it has room,
 *        otherwise take a new physical block and extend the table;
 *     4. freeing a sequence returns its blocks to a free list;
 *     5. the attention kernel takes the block table as an argument and gathers internally.
 *   "PagedAttention e continuous batching", section "01 - Conceito":
 *     paragraph 3  blocks live anywhere in the pool; the allocator hands a sequence a new
 *                  block when it outgrows its last one, without moving anything;
 *     paragraph 6  identical prompt prefixes share read-only blocks; copy-on-write gives a
 *                  diverging branch a new block; reference counts return blocks to the pool;
 *     paragraph 7  admission reasons in countable blocks and refuses early, clearly;
 *     paragraph 8  block metrics: free/used blocks, allocation failures, tail waste,
 *                  prefix hits, preemptions.
 *
 * Two halves:
 *   - device calls (kv append, paged decode attention -- optionally with the step's append
 *     fused in --, chunked-prefill attention, block copy, the upload of a step's metadata):
 *     asynchronous on the caller's CUDA stream, no host synchronisation, no allocation; every
 *     device pointer is owned by the caller;
 *   - a host block manager (pure C, no CUDA): free list, block tables, reference counts,
 *     prefix sharing, copy-on-write decisions, admission in blocks, checkpoint / resume.
 *
 * Memory layout (the pages fix none; this library's reading):
 *   pool (K or V) = [n_layers][num_blocks][n_kv_heads][block_size][head_dim] elements,
 *   row-major, so layer l starts at pool + l * num_blocks * n_kv_heads * block_size * head_dim
 *   and one physical block id names the same 16 token positions in every layer (one block
 *   table serves all layers, as the 1 MiB all-layer block of "01 - Conceito" paragraph 3).
 *   slot of a token = physical block * block_size + (position mod block_size).
 *   q, out   = [n_seqs][n_q_heads][head_dim]; query head h reads KV head h / (n_q / n_kv).
 *   k, v     = [n_tokens][n_kv_heads][head_dim] (the new rows to append).
 *   block_tables = int32 [n_seqs][max_blocks_per_seq]; context_lens = int32 [n_seqs].
 *
 * One GPU per call: the pools, q, out and workspaces of a call live in the memory of the device
 * current at the call. The library caches per-device facts (the device addresses of its status
 * word and scratch array, the multiprocessor count, TMA tensor maps) for the life of the process:
 * calling cudaDeviceReset, or otherwise tearing down a device's primary context, while the library
 * is loaded is not supported (the cached addresses would then be stale).
 *
 * Status: every call returns PKV_OK (0) or one PKV_ERR_* code; pkv_status_str names it.
 * Argument errors are caught on the host before anything is launched. Values that live on
 * the device (table entries, context lengths, slots, copy pairs) are range-checked inside
 * the kernels: a bad one is skipped and recorded in a device status word that
 * pkv_get_device_status reads and clears; no kernel traps.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- types ------------------------------------------------------------------------- */

typedef enum { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2 } pkv_dtype;

enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, unknown id      */
    PKV_ERR_UNSUPPORTED = 2, /* shape outside the compiled set (see pkv_cache_desc)        */
    PKV_ERR_NO_BLOCKS = 3,   /* not enough free blocks: admission refused / append OOM      */
    PKV_ERR_BAD_STATE = 4,   /* internal inconsistency detected (never expected)            */
    PKV_ERR_CUDA = 5         /* a CUDA runtime call failed (launch, attribute, copy)         */
};

/* Device status bits, set by kernels that skipped a bad device-side value. */
enum {
    PKV_DEV_BAD_BLOCK_ID = 1u,    /* block table entry outside [0, num_blocks)               */
    PKV_DEV_BAD_CONTEXT_LEN = 2u, /* context length < 0 or > max_blocks_per_seq*block_size  */
    PKV_DEV_BAD_SLOT = 4u,        /* slot >= num_blocks*block_size                           */
    PKV_DEV_BAD_PAIR = 8u,        /* copy pair id outside [0, num_blocks)                    */
    PKV_DEV_WAIT_TIMEOUT = 16u,   /* a bounded wait on an asynchronous copy gave up          */
    PKV_DEV_BAD_QUERY_RANGE = 32u /* prefill: query_start / chunk length inconsistent         */
};

/*
 * Shape of one paged cache. Supported: block_size == 16; head_dim in {64, 128, 256};
 * n_q_heads == G * n_kv_heads with G in {1, 2, 4, 8}; dtype in pkv_dtype; all counts >= 1.
 * Anything else returns PKV_ERR_UNSUPPORTED (or PKV_ERR_INVALID_ARG for non-positive counts).
 */
typedef struct {
    int32_t dtype;      /* pkv_dtype                                  */
    int32_t n_layers;
    int32_t num_blocks; /* physical blocks in the pool (every layer) */
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t block_size; /* tokens per block; must be 16               */
} pkv_cache_desc;

/* ---- descriptors and sizes --------------------------------------------------------- */

const char* pkv_status_str(int status);

/* PKV_OK if the descriptor is supported, else the error code the device calls would return. */
int pkv_validate_desc(const pkv_cache_desc* desc);

/*
 * KV bytes one token occupies across all layers: 2 (K and V) * n_layers * n_kv_heads *
 * head_dim * element bytes ("Paged Attention em Large Language Models LLMs", section
 * "Configurando as Constantes": 524,288 bytes for 32 x 32 x 128 in fp16). 0 if desc is invalid.
 */
uint64_t pkv_bytes_per_token(const pkv_cache_desc* desc);

/* Bytes of one pool (K or V) over all layers: n_layers*num_blocks*n_kv*block_size*head_dim*e. */
uint64_t pkv_pool_bytes(const pkv_cache_desc* desc);

/*
 * Split-K geometry of paged decode attention (an interface helper; the pages describe no kernel)
 * for n_seqs sequences whose tables have max_blocks_per_seq columns, on a device with sm_count
 * multiprocessors that each hold ctas_per_sm CTAs of the decode kernel at once. A long context is
 * cut into partitions of *blocks_per_partition table entries, each computed by its own CTA and
 * merged in the same launch; *n_partitions = ceil(max_blocks_per_seq / *blocks_per_partition);
 * *workspace_bytes receives the scratch those partials need (0 when *n_partitions is 1). With
 * pairs = n_seqs * n_kv_heads and slots = sm_count * ctas_per_sm:
 *   - one wave: if pairs < slots, parts = slots / pairs fills at least 3/4 of the slots and the
 *     partitions ceil(max_blocks_per_seq / parts) are long (>= 64 entries; fp16 / bf16 pools,
 *     whose kernel streams its table entries), that is the partition: the grid is one wave;
 *   - otherwise 64 entries, halved (down to 4) while pairs * n_partitions < 4 * sm_count.
 * The decode calls use exactly this geometry with the current device's facts
 * (pkv_decode_ctas_per_sm). Host-only arithmetic: needs no GPU. Output pointers may be NULL.
 * PKV_ERR_INVALID_ARG when a count is not positive; descriptor errors as pkv_validate_desc.
 */
int pkv_decode_split_geometry(const pkv_cache_desc* desc, int32_t n_seqs, int32_t max_blocks_per_seq,
                              int32_t sm_count, int32_t ctas_per_sm, int32_t* blocks_per_partition,
                              int32_t* n_partitions, size_t* workspace_bytes);

/*
 * The current device's facts behind that geometry for pools of this descriptor: its multiprocessor
 * count and how many CTAs of the decode kernel the descriptor selects one multiprocessor holds at
 * once (the CUDA occupancy calculator: shared memory, registers, threads). Read once per device and
 * kernel, then cached. Output pointers may be NULL. PKV_ERR_CUDA without a usable device.
 */
int pkv_decode_ctas_per_sm(const pkv_cache_desc* desc, int32_t* ctas_per_sm, int32_t* sm_count);

/*
 * Scratch bytes pkv_paged_decode_attention needs on the current device for n_seqs sequences whose
 * tables have max_blocks_per_seq columns: split-K partial results plus one 8-byte arrival counter
 * per (sequence, KV head); 0 when no split is needed -- and also when the descriptor or a count is
 * invalid or no CUDA device can be queried. Equals pkv_decode_split_geometry's *workspace_bytes
 * with the current device's pkv_decode_ctas_per_sm.
 */
size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t n_seqs, int32_t max_blocks_per_seq);

/* ---- device calls ------------------------------------------------------------------ */

/*
 * Append the K/V rows of n_tokens new tokens of one layer into the pools
 * ("La idea de PagedAttention", step 3; the slot comes from the block manager).
 *   k, v          device, [n_tokens][n_kv_heads][head_dim] of desc->dtype, 16-byte aligned
 *   slot_mapping  device int64 [n_tokens]; slot < 0 marks padding and is skipped;
 *                 slot >= num_blocks*block_size is skipped and sets PKV_DEV_BAD_SLOT
 *   k_pool, v_pool device, whole pools (all layers), 16-byte aligned
 * Bit-exact byte copies. n_tokens == 0 is a no-op. Slots must be distinct (else the
 * surviving row is unspecified).
 */
int pkv_kv_append(const pkv_cache_desc* desc, int32_t layer, const void* k, const void* v,
                  const int64_t* slot_mapping, int32_t n_tokens, void* k_pool, void* v_pool,
                  void* stream);

/*
 * Paged decode attention for one layer: one query token per sequence attends to the
 * first context_lens[s] logical positions of its own cache, gathered through its block
 * table ("La idea de PagedAttention", step 5). For query head h and KV head g = h / G:
 *   out[s][h] = sum_j softmax_j(scale * q[s][h] . K_j) V_j,  j < context_lens[s],
 * K_j, V_j being row (block_tables[s][j / 16], g, j mod 16) of layer `layer`. Paging changes
 * only where rows live, so this equals dense attention over the same rows ("Lo que deberias
 * llevarte de la Fase 22 sobre la Fase 27", item 2). Accumulation is fp32; out is rounded
 * to desc->dtype (round to nearest even). context_lens[s] == 0 gives a zero row.
 *   q, out        device [n_seqs][n_q_heads][head_dim] of desc->dtype, 16-byte aligned
 *   k_pool, v_pool device, whole pools (all layers), 16-byte aligned
 *   block_tables  device int32 [n_seqs][max_blocks_per_seq]; only the first
 *                 ceil(context_lens[s]/16) entries of row s are read
 *   context_lens  device int32 [n_seqs], 0 <= len <= max_blocks_per_seq*16 (a larger one
 *                 is clamped and sets PKV_DEV_BAD_CONTEXT_LEN)
 *   workspace     device, >= pkv_decode_workspace_bytes(...) bytes, 16-byte aligned
 *                 (may be NULL when that is 0); contents need no initialisation (the split-K
 *                 arrival counters kept there carry a per-call tag, so leftovers of earlier
 *                 calls of any shape read as zero). Calls that overlap on the GPU must not
 *                 share one workspace.
 * Rows outside the valid positions (tails of last blocks, unreferenced blocks) are never
 * used: NaN there cannot reach the output. A table entry outside [0, num_blocks) is
 * skipped (its rows count as masked) and sets PKV_DEV_BAD_BLOCK_ID. fp16 / bf16 pools of
 * 2^31 rows per layer or more (num_blocks * n_kv_heads * 16; the tensor copies' row
 * coordinates are 32-bit) return PKV_ERR_UNSUPPORTED, launching nothing.
 */
int pkv_paged_decode_attention(const pkv_cache_desc* desc, int32_t layer, const void* q,
                               const void* k_pool, const void* v_pool, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t n_seqs,
                               float scale, void* out, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * One decode step of one layer in a single kernel: pkv_kv_append of one new token per sequence
 * followed by pkv_paged_decode_attention. The token of sequence s sits at logical position
 * context_lens[s] - 1 ("La idea de PagedAttention", step 3: written into the last block, which
 * the block manager has already reserved -- pkv_mgr_append_slot's slot), so its slot follows
 * from the table: block_tables[s][(len-1)/16] * 16 + (len-1) % 16. The rows
 * k_new[s][g], v_new[s][g] (device, [n_seqs][n_kv_heads][head_dim] of desc->dtype, 16-byte
 * aligned) are written there in layer `layer` of the pools, then the sequence attends to its
 * first context_lens[s] positions, the new one included. Results (pools and out) are
 * bit-identical to the two separate calls. Other arguments, layout and errors as
 * pkv_paged_decode_attention; k_pool / v_pool are written. Sequences with context_lens[s] == 0
 * append nothing. Copy-on-write block copies for this step must already have run.
 */
int pkv_paged_decode_append_attention(const pkv_cache_desc* desc, int32_t layer, const void* q,
                                      const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t n_seqs, float scale, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * pkv_paged_decode_append_attention with launch flags. PKV_DECODE_OVERLAP_PREVIOUS launches the
 * kernel as a programmatic dependent of the previous kernel on `stream` (fp16 / bf16 storage; the
 * flag has no effect for fp32): it may start while that kernel is finishing; before the previous
 * kernel completes it may read q, k_new, v_new, the tables, the lengths and layer `layer` of the
 * pools and write the new rows into their slots of layer `layer`; it writes the workspace, out
 * and the status word only after. Set it only when the previous kernel on the stream writes none
 * of those inputs and reads none of those new rows' slots -- in a decode step, the call for the
 * previous layer with the same tables, lengths and workspace (its own out, k_new / v_new rows and
 * pool layer are distinct), or a prefill attention of the same layer over other sequences (a
 * decoding sequence appends into its own last block, which no other sequence reads). Unknown flag
 * bits: PKV_ERR_INVALID_ARG. Results are bit-identical to pkv_paged_decode_append_attention.
 */
#define PKV_DECODE_OVERLAP_PREVIOUS 1u
int pkv_paged_decode_append_attention_ex(const pkv_cache_desc* desc, int32_t layer, const void* q,
                                         const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t n_seqs, float scale, void* out,
                                         void* workspace, size_t workspace_bytes, uint32_t flags, void* stream);

/*
 * Decode attention over a dense, contiguous KV cache: the pre-allocated (batch, heads, maximum
 * length, head_dim) cache that "04 - Hacia PagedAttention (vista previa)" starts from ("Lo que
 * funciona en la Fase 22"), read by the same kernels as pkv_paged_decode_attention with the block
 * table replaced by the identity walk (logical block i of a sequence is its i-th 16-row chunk).
 * It exists to price the table walk: paging changes where rows live, not the result ("Lo que
 * deberias llevarte de la Fase 22 sobre la Fase 27", item 2), at the cost of a constant factor
 * (items 2-3). For query head h and KV head g = h / G:
 *   out[s][h] = sum_j softmax_j(scale * q[s][h] . K[s][g][j]) V[s][g][j],  j < context_lens[s].
 *   k_cache, v_cache device [n_layers][n_seqs][n_kv_heads][max_seq_len][head_dim] of desc->dtype,
 *                 16-byte aligned (desc->num_blocks is not used)
 *   max_seq_len   positions reserved per sequence: a positive multiple of 16
 *   context_lens  device int32 [n_seqs], 0 <= len <= max_seq_len (larger: clamped, and
 *                 PKV_DEV_BAD_CONTEXT_LEN is set)
 *   q, out, scale as pkv_paged_decode_attention
 *   workspace     as pkv_paged_decode_attention with max_blocks_per_seq = max_seq_len / 16
 *   flags         0 or PKV_DECODE_OVERLAP_PREVIOUS (as pkv_paged_decode_append_attention_ex)
 * Equal, bit for bit, to pkv_paged_decode_attention over a pool holding the same rows in the same
 * logical order. Rows past context_lens[s] are never used. PKV_ERR_UNSUPPORTED when
 * n_seqs * n_kv_heads * max_seq_len reaches 2^31 rows.
 */
int pkv_dense_decode_attention(const pkv_cache_desc* desc, int32_t layer, const void* q, const void* k_cache,
                               const void* v_cache, int32_t max_seq_len, const int32_t* context_lens,
                               int32_t n_seqs, float scale, void* out, void* workspace, size_t workspace_bytes,
                               uint32_t flags, void* stream);

/* Size of the fixed scratch array used by pkv_paged_decode_attention_static (16 MiB). */
#define PKV_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * pkv_paged_decode_attention without a workspace argument, for callers that cannot allocate
 * device memory when they run attention (code inside a stream capture, a serving loop that
 * forbids allocation after start-up, an embedding host with a fixed memory budget). The pages
 * have no counterpart: this is an interface convenience, not part of the method.
 * Same arguments, layout, result and errors as pkv_paged_decode_attention minus workspace and
 * workspace_bytes. The split-K partial results go to a scratch array of
 * PKV_STATIC_SCRATCH_BYTES compiled into the library; every GPU that loads the library holds
 * it until the process exits. The call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *   - Returns PKV_ERR_UNSUPPORTED, launching nothing, when the call would need more than
 *     PKV_STATIC_SCRATCH_BYTES (when pkv_decode_workspace_bytes(desc, n_seqs,
 *     max_blocks_per_seq) exceeds it); use pkv_paged_decode_attention with your own workspace.
 *   - The first call on each device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call before any stream
 *     capture begins.
 *   - All calls share the one array and it keeps the last call's contents. No call reads an
 *     earlier call's partial results (each is written before it is merged), and the split-K
 *     arrival counters kept there carry a per-call tag, so leftovers of earlier calls of any
 *     shape read as zero: nothing needs clearing. Calls that overlap on the GPU -- on
 *     different streams, or from several host threads -- race on it: serialise them.
 */
int pkv_paged_decode_attention_static(const pkv_cache_desc* desc, int32_t layer, const void* q,
                                      const void* k_pool, const void* v_pool, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t n_seqs,
                                      float scale, void* out, void* stream);

/*
 * Paged prefill (or chunked prefill) attention for one layer: a chunk of new query tokens per
 * sequence attends causally to the sequence's cache through its block table ("PagedAttention e
 * continuous batching", "01 - Conceito", paragraph 5: a long prompt is processed in slices that
 * share steps with decoding; "La idea de PagedAttention", step 5: the kernel gathers the rows).
 * The chunk's K/V rows must already be appended (pkv_kv_append). With c = context_lens[s] and
 * n_s = query_start[s+1] - query_start[s], chunk token i of sequence s sits at position
 * p = c - n_s + i and, for query head h and KV head g = h / G,
 *   out[t][h] = sum_{j <= p} softmax_j(scale * q[t][h] . K_j) V_j,   t = query_start[s] + i,
 * K_j, V_j being row (block_tables[s][j / 16], g, j mod 16) of layer `layer`: dense causal
 * attention over the gathered rows. A whole prompt is the chunk n_s == c. fp32 accumulation; out
 * rounded to desc->dtype.
 *   q, out        device [n_tokens][n_q_heads][head_dim] of desc->dtype, 16-byte aligned; the
 *                 chunk tokens of all sequences packed in order (sequence s owns rows
 *                 query_start[s] .. query_start[s+1]-1, in position order); rows owned by no
 *                 sequence are left unwritten
 *   k_pool, v_pool device, whole pools (all layers), 16-byte aligned
 *   block_tables  device int32 [n_seqs][max_blocks_per_seq]; the first ceil(c/16) entries are read
 *   context_lens  device int32 [n_seqs]: tokens in the cache after the chunk, n_s <= c <=
 *                 max_blocks_per_seq*16
 *   query_start   device int32 [n_seqs + 1], non-decreasing, query_start[0] >= 0,
 *                 query_start[n_seqs] <= n_tokens
 *   max_query_len host: the largest n_s (sizes the grid), 0 <= max_query_len <= n_tokens
 * A sequence whose device-side values break these rules (n_s < 0, n_s > max_query_len, n_s > c,
 * c too large, query_start outside [0, n_tokens]) is skipped, its rows left unwritten, and sets
 * PKV_DEV_BAD_QUERY_RANGE. A table entry outside [0, num_blocks) is skipped (its keys count as
 * masked) and sets PKV_DEV_BAD_BLOCK_ID. Rows past a query's position or past the context are
 * never used: NaN there cannot reach the output. No workspace; nothing is allocated.
 * fp16 / bf16 run on the tensor cores; fp32 on the CUDA cores (the precision mode). For one GPU:
 * k_pool and v_pool must be device memory of the current device, because the tensor copies read
 * them directly; the first fp16 / bf16 call on a pool layer checks this before building its copy
 * descriptors (cached afterwards by address) and returns PKV_ERR_INVALID_ARG for host memory or
 * another GPU's memory, launching nothing. The same holds for the fp16 / bf16 decode calls.
 * fp16 / bf16 pools of 2^31 rows per layer or more (num_blocks * n_kv_heads * 16) return
 * PKV_ERR_UNSUPPORTED, launching nothing (the tensor copies' row coordinates are 32-bit).
 */
int pkv_paged_prefill_attention(const pkv_cache_desc* desc, int32_t layer, const void* q,
                                const void* k_pool, const void* v_pool, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens,
                                const int32_t* query_start, int32_t n_seqs, int32_t n_tokens,
                                int32_t max_query_len, float scale, void* out, void* stream);

/*
 * pkv_paged_prefill_attention with launch flags. PKV_PREFILL_OVERLAP_PREVIOUS launches the kernel
 * as a programmatic dependent of the previous kernel on `stream` (fp16 / bf16 storage; no effect
 * for fp32): it may start while that kernel is finishing and read q, the tables, the lengths,
 * query_start and layer `layer` of the pools before the previous kernel completes; it writes out
 * and the status word only after, so the call completes after the previous kernel. Set it only
 * when the previous kernel on the stream writes none of those inputs -- in a chunked-prefill step
 * that appends the chunk's rows of every layer before the first attention launch, the attention
 * launch of the previous layer, or the previous layer's decode call over other sequences. Unknown
 * flag bits: PKV_ERR_INVALID_ARG. Results are bit-identical to pkv_paged_prefill_attention.
 */
#define PKV_PREFILL_OVERLAP_PREVIOUS 1u
int pkv_paged_prefill_attention_ex(const pkv_cache_desc* desc, int32_t layer, const void* q, const void* k_pool,
                                   const void* v_pool, const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* query_start, int32_t n_seqs,
                                   int32_t n_tokens, int32_t max_query_len, float scale, void* out, uint32_t flags,
                                   void* stream);

/*
 * Scheduling helper for chunked prefill (the pages slice long prompts into chunks, "01 -
 * Conceito", paragraph 5, but fix no chunk size): *tokens receives how many new tokens of one
 * sequence fill exactly one wave of pkv_paged_prefill_attention's grid on the current device:
 * the CTAs the GPU holds at once (SMs x CTAs per SM; at head_dim 256, whose CTAs work in pairs, no
 * more than twice the pairs the cluster scheduler can place at once) x tokens per CTA (128 / G query
 * rows; 32 / G for fp32) / n_kv_heads.
 * A chunk of a whole number of waves leaves no SM idle through a partly filled last wave (head_dim
 * 256 on a GB300: 1,216 tokens; chunks of 2,432 run 12 % faster per launch than chunks of 2,048).
 * PKV_ERR_CUDA without a usable device; descriptor errors as pkv_validate_desc.
 */
int pkv_prefill_wave_tokens(const pkv_cache_desc* desc, int32_t* tokens);

/*
 * Copy-on-write block copies ("01 - Conceito", paragraph 6): for each pair (src, dst) in
 * pairs (device int32 [n_pairs][2]) copy physical block src onto dst in K and V, all layers.
 * Bit-exact. The dst ids must be distinct and disjoint from the src ids (else the result is
 * unspecified). An id outside [0, num_blocks) skips its pair and sets PKV_DEV_BAD_PAIR.
 */
int pkv_copy_blocks(const pkv_cache_desc* desc, void* k_pool, void* v_pool, const int32_t* pairs,
                    int32_t n_pairs, void* stream);

/*
 * Upload one step's metadata -- the packed block tables, context lengths, slots, query starts
 * and copy pairs that the host block manager wrote ("La idea de PagedAttention", steps 2 and 5:
 * the kernel takes the block table as an argument) -- from host to device memory with a kernel
 * whose threads read the host buffer directly over the host link.
 *   dst       device memory of the current device, 16-byte aligned, `bytes` long
 *   src_host  page-locked host memory visible to the device (cudaHostAlloc / cudaMallocHost, or
 *             registered), 16-byte aligned; the caller keeps it unchanged until the upload has
 *             run on `stream` (record an event after this call)
 *   bytes     a multiple of 4, at most 1 GiB; 0 is a no-op
 * Bit-exact. Unlike a copy-engine copy, the upload does not queue behind bulk host-to-device
 * copies that other streams have in flight: a step's kernels wait only for their own metadata
 * while the next step's rows stream in beside them. Pageable, device-invisible or misaligned
 * memory and a dst on another device return PKV_ERR_INVALID_ARG before anything is launched.
 */
int pkv_upload_metadata(void* dst, const void* src_host, size_t bytes, void* stream);

/*
 * Synchronise `stream`, then read and clear this library's device status word on the
 * current device (PKV_DEV_* bits, 0 if every device-side value was in range). For tests
 * and debugging; the only call here that blocks the host.
 */
int pkv_get_device_status(void* stream, uint32_t* flags);

/*
 * Measurement helper (the pages have no counterpart): read every byte of buf once, as a plain
 * coalesced stream, and XOR-fold its 32-bit words into *fold. Timing this call over a buffer much
 * larger than the L2 cache gives the read-only HBM bandwidth of the device, the ceiling of a kernel
 * that only reads (paged decode attention writes a few bytes per kilobyte it reads).
 *   buf    device, 16-byte aligned, `bytes` long (a multiple of 16)
 *   fold   device uint32, 4-byte aligned; XORed with the fold of buf's words (set it to 0 first to
 *          read the fold itself: the XOR of every little-endian 32-bit word of buf)
 * Asynchronous on `stream`. PKV_ERR_INVALID_ARG for a misaligned or NULL pointer or a size that is
 * not a multiple of 16; bytes == 0 is a no-op.
 */
int pkv_hbm_read_probe(const void* buf, size_t bytes, uint32_t* fold, void* stream);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t pkv_launch_count(void);

/*
 * Self-test of the bounded waits every kernel here uses on its asynchronous copies: launches one
 * CTA that waits on an mbarrier nothing will ever complete. The wait gives up after its limit
 * (about one second), records PKV_DEV_WAIT_TIMEOUT in the device status word (read it with
 * pkv_get_device_status) and the kernel returns normally, leaving the context usable. No fault,
 * trap or hang is involved. Asynchronous on `stream`; PKV_ERR_CUDA if the launch fails.
 */
int pkv_selftest_wait_timeout(void* stream);

/* ---- host block manager ------------------------------------------------------------ */

typedef struct pkv_mgr pkv_mgr;

typedef struct {
    int64_t free_blocks;
    int64_t used_blocks;
    int64_t n_seqs;
    int64_t alloc_failures;  /* refused admissions + appends that found no free block     */
    int64_t tail_waste_rows; /* sum over sequences of 16*n_blocks - context length          */
    int64_t prefix_hits;     /* blocks obtained by fork (shared) instead of allocation     */
    int64_t cow_copies;      /* copy-on-write pairs emitted                                 */
    int64_t append_oom;      /* appends refused for lack of blocks (a preemption signal)   */
} pkv_stats;

/*
 * Create a manager over num_blocks physical blocks of block_size (16) tokens.
 * initial_free_order (host, num_blocks ids, a permutation of 0..num_blocks-1) fixes the
 * free list's initial order; NULL means 0, 1, ..., num_blocks-1. Returns NULL on bad
 * arguments or allocation failure. The free list is FIFO: allocation takes the front,
 * release appends to the back, a freed sequence releases its blocks in logical order.
 */
pkv_mgr* pkv_mgr_create(int32_t num_blocks, int32_t block_size, const int32_t* initial_free_order);

/* Deep copy (checkpoint of the bookkeeping); NULL on allocation failure. */
pkv_mgr* pkv_mgr_clone(const pkv_mgr* mgr);

void pkv_mgr_destroy(pkv_mgr* mgr);

/*
 * Every manager call below is transactional: on any error the manager's state is unchanged
 * (only the failure counters of pkv_stats move).
 *
 * Admit sequence seq_id with n_prompt_tokens tokens ("01 - Conceito", paragraph 7): it needs
 * ceil(n_prompt/16) + ceil(reserve_tokens/16) free blocks, else PKV_ERR_NO_BLOCKS; only the
 * prompt blocks are taken (reserve_tokens is headroom, not a reservation). slots_out (host,
 * n_prompt_tokens entries, may be NULL) receives each prompt token's slot.
 * PKV_ERR_INVALID_ARG if seq_id exists or a count is negative.
 */
int pkv_mgr_add_seq(pkv_mgr* mgr, int64_t seq_id, int32_t n_prompt_tokens, int32_t reserve_tokens,
                    int64_t* slots_out);

/*
 * child starts as a copy of parent's table and context; every block gains a reference
 * (prefix sharing, "01 - Conceito" paragraph 6). PKV_ERR_INVALID_ARG if parent is unknown,
 * child exists, or they are equal.
 */
int pkv_mgr_fork(pkv_mgr* mgr, int64_t parent, int64_t child);

/*
 * Reserve the slot of one new token of seq_id ("La idea de PagedAttention", step 3):
 *   last block full (or none): take a fresh block;
 *   last block partially filled and referenced only by seq_id: write in place;
 *   last block partially filled and shared: copy on write -- take a fresh block, report
 *     (*cow_src, *cow_dst) for pkv_copy_blocks, drop one reference of the old block.
 * *cow_src = *cow_dst = -1 when no copy is needed. PKV_ERR_NO_BLOCKS when a block is needed
 * and none is free (counted in append_oom). Copy before append before attention.
 */
int pkv_mgr_append_slot(pkv_mgr* mgr, int64_t seq_id, int64_t* slot, int32_t* cow_src, int32_t* cow_dst);

/*
 * Extend sequence seq_id by n_tokens new tokens at once (one chunk of a chunked prefill, "01 -
 * Conceito", paragraph 5), all or nothing. slots_out (n_tokens entries, may be NULL when
 * n_tokens == 0) receives the slots of positions ctx .. ctx+n_tokens-1. The result equals
 * n_tokens successive pkv_mgr_append_slot calls: only the first token can copy a shared,
 * partially filled last block (that pair in *cow_src / *cow_dst, else -1; run it through
 * pkv_copy_blocks before the appends), then fresh blocks are taken in order. If the pool cannot
 * hold all n_tokens, nothing changes, alloc_failures and append_oom each grow by one and
 * PKV_ERR_NO_BLOCKS is returned. n_tokens == 0 is a no-op.
 */
int pkv_mgr_extend(pkv_mgr* mgr, int64_t seq_id, int32_t n_tokens, int64_t* slots_out, int32_t* cow_src,
                   int32_t* cow_dst);

/*
 * Append one token to each of seq_ids[0..n) in order. slots_out[n] receives the slots,
 * cow_pairs_out[2*n] the (src, dst) pairs that were emitted, *n_cow their count, *n_done the
 * number of sequences served. Stops at the first failing sequence and returns its status;
 * the sequences before it stay appended (each single append is transactional).
 */
int pkv_mgr_append_batch(pkv_mgr* mgr, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                         int32_t* cow_pairs_out, int32_t* n_cow, int32_t* n_done);

/*
 * Release seq_id ("La idea de PagedAttention", step 4): each block loses one reference and
 * returns to the back of the free list when none is left. PKV_ERR_INVALID_ARG if unknown
 * (double free).
 */
int pkv_mgr_free_seq(pkv_mgr* mgr, int64_t seq_id);

/* Copy seq_id's table into out[cap]; *n_blocks and *ctx_len receive its size and length.
 * PKV_ERR_INVALID_ARG if unknown or cap < n_blocks (nothing written then). */
int pkv_mgr_block_table(const pkv_mgr* mgr, int64_t seq_id, int32_t* out, int32_t cap, int32_t* n_blocks,
                        int32_t* ctx_len);

/*
 * Pack the tables of seq_ids[0..n) into tables_out[n][max_blocks] (unused entries = -1) and
 * their lengths into lens_out[n]: the host image of the device arguments of
 * pkv_paged_decode_attention. PKV_ERR_INVALID_ARG if an id is unknown or a table is wider
 * than max_blocks.
 */
int pkv_mgr_pack_tables(const pkv_mgr* mgr, const int64_t* seq_ids, int32_t n, int32_t max_blocks,
                        int32_t* tables_out, int32_t* lens_out);

int pkv_mgr_stats(const pkv_mgr* mgr, pkv_stats* out);

/* Reference count of a block, or -1 if the id is out of range. */
int32_t pkv_mgr_refcount(const pkv_mgr* mgr, int32_t block);

/* Copy up to cap free-list entries, front first, into out; returns the free-list length. */
int32_t pkv_mgr_free_list(const pkv_mgr* mgr, int32_t* out, int32_t cap);

/*
 * Fault injection for tests: the (after_n_allocs + 1)-th block allocation attempted from
 * now on fails as if the pool were empty (once); a negative value disables it. Used to
 * check that multi-block operations roll back completely.
 */
int pkv_mgr_inject_alloc_failure(pkv_mgr* mgr, int32_t after_n_allocs);

/*
 * Checkpoint / resume of the host manager (the pages have no counterpart; the device pools are
 * caller-owned tensors and are saved by the caller). The image is a little-endian byte string:
 * "PKVM", version 1, num_blocks, block_size, the free list front first, the four event counters
 * of pkv_stats, then every sequence in ascending id order (id, context length, block count,
 * table), then an FNV-1a 64 checksum of everything before it. Reference counts are not stored:
 * a block's count is the number of tables that hold it. The fault-injection setting is not saved.
 *
 * pkv_mgr_save_bytes: the size of the image of the current state (0 if mgr is NULL).
 * pkv_mgr_save: write it into buf (host, cap bytes); *written receives its size.
 *   PKV_ERR_INVALID_ARG if an argument is NULL or cap is too small (nothing written).
 * pkv_mgr_load: a new manager whose state equals the saved one (same tables, lengths, free-list
 *   order, reference counts and counters; every later operation gives the same results as on the
 *   saved manager), or NULL if the image is malformed: wrong magic, version, size or checksum, an
 *   id out of range, a block both free and referenced or neither, a table whose length does not
 *   match its context, a repeated sequence id.
 */
size_t pkv_mgr_save_bytes(const pkv_mgr* mgr);
int pkv_mgr_save(const pkv_mgr* mgr, void* buf, size_t cap, size_t* written);
pkv_mgr* pkv_mgr_load(const void* buf, size_t len);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
