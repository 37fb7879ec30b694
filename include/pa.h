/*
 * pa.h - C ABI of a paged-KV-cache attention library for NVIDIA GB300 (sm_103a).
 *
 * The KV cache is split into fixed-size physical blocks of `block_size` tokens;
 * a request's logical blocks map to physical blocks through its Block Table,
 * so its KV need not be contiguous ("2.1 PagedAttention", §2-§3).  Attention
 * kernels translate each logical token t into (physical_block_number =
 * table[t / block_size], physical_block_offset = t % block_size) (§5).
 *
 * Conventions for every call below
 * --------------------------------
 * - Cache layout: k_cache and v_cache are separate tensors, each
 *   [num_blocks][block_size][kv_heads][head_dim], row-major, contiguous.
 * - Block tables: int32 [num_seqs][max_blocks_per_seq], row-major; entries
 *   past a request's last logical block are never read (any value).
 * - Element types: PA_FP16 or PA_BF16 for q/k/v/out (inputs and outputs in the
 *   same type); accumulation and softmax are fp32.
 * - head_dim in {64, 128}; block_size in {4, 8, 16, 32};
 *   q_heads % kv_heads == 0 and q_heads / kv_heads <= 16.  Query head h reads
 *   KV head h / (q_heads / kv_heads) (contiguous GQA groups).
 * - Device calls: every pointer is device memory owned by the caller; the
 *   library allocates no device memory and keeps no pointer after returning.
 *   Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream).  All device pointers must be 16-byte aligned.
 * - Ordering: kernels are launched with programmatic dependent launch.  A
 *   kernel of this library may start its set-up while the kernel before it on
 *   the same stream is finishing, and reads only q, block tables, q_start and
 *   context lengths during that set-up; caches, scratch and outputs are read
 *   or written only once the previous kernel has completed.  So those four
 *   inputs must be ready when the call is enqueued (they are if whatever writes
 *   them was enqueued earlier on the stream without allowing early launch of
 *   its successor, as plain kernels and copies do).
 * - Errors: every call returns a pa_status.  Argument errors are caught on the
 *   host before anything is launched.  Data errors that only the device can
 *   see (a block id outside [0, num_blocks), a slot past the pool, a context
 *   length past the table, a wait that timed out) never fault or trap: the
 *   kernel records the first such code in a per-device error word, skips the
 *   offending access, and finishes; read it with pa_get_device_error().
 *   Nothing aborts, nothing throws.
 * - Thread safety: device calls may be made from any host thread.  A pa_alloc
 *   handle is single-threaded.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = -1,        /* bad argument (shape, pointer, id, range)        */
  PA_ERR_NO_FREE_BLOCKS = -2, /* pool exhausted; allocator state unchanged      */
  PA_ERR_DTYPE = -3,          /* unsupported element type                       */
  PA_ERR_CUDA = -4,           /* a CUDA runtime/driver call failed              */
  PA_ERR_DEVICE_CHECK = -5,   /* pa_get_device_error found a recorded error     */
  PA_ERR_SHARED_BLOCK = -6,   /* append into a shared partial block: cow first  */
  PA_ERR_WORKSPACE = -7,      /* workspace missing or smaller than required     */
  PA_ERR_HOST_MEMORY = -8     /* a host allocation failed; nothing changed      */
} pa_status;

typedef enum { PA_FP16 = 0, PA_BF16 = 1 } pa_dtype;

/* Device error codes recorded by kernels (first one wins). */
enum {
  PA_DEVERR_NONE = 0,
  PA_DEVERR_BLOCK_ID = 1,     /* block-table entry or copy pair outside [0, num_blocks) */
  PA_DEVERR_CONTEXT_LEN = 2,  /* context length < 0 or > max_blocks_per_seq*block_size */
  PA_DEVERR_SLOT = 3,         /* slot_mapping entry >= num_blocks*block_size            */
  PA_DEVERR_TIMEOUT = 4,      /* a bounded wait on a shared-memory barrier expired      */
  PA_DEVERR_QUERY_RANGE = 5   /* bad q_start / chunk length in chunked prefill          */
};

typedef struct CUstream_st* pa_stream; /* identical to cudaStream_t */

/* Human-readable name of a pa_status value (static string). */
const char* pa_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int pa_version(void);

/* Number of kernels this library has launched in this process. */
uint64_t pa_launch_count(void);

/* ----------------------------------------------------------------------------
 * pa_reshape_and_cache - scatter new tokens' K/V into their slots.
 *
 * "2.1 PagedAttention" §3: each new token fills the next free slot of its
 * request's current block; the forward pass writes the KV into the blocks the
 * allocator handed out ("Khám phá vLLM … phần 2", prefix caching).  For token
 * i with slot s = slot_mapping[i] >= 0:
 *     k_cache[s / block_size][s % block_size][:][:] = k[i][:][:]   (same for v)
 * A negative slot marks a padding token and is skipped.  The copy is
 * bit-exact.
 *   k, v          [num_tokens][kv_heads][head_dim], contiguous
 *   slot_mapping  int32 [num_tokens]; slots must be distinct
 *   k_cache,v_cache  the pool (see conventions)
 * num_tokens == 0 is a no-op.  A slot >= num_blocks*block_size records
 * PA_DEVERR_SLOT and is skipped.
 * ------------------------------------------------------------------------- */
int pa_reshape_and_cache(const void* k, const void* v, const int32_t* slot_mapping, int num_tokens,
                         void* k_cache, void* v_cache, int num_blocks, int block_size, int kv_heads,
                         int head_dim, pa_dtype dtype, pa_stream stream);

/* ----------------------------------------------------------------------------
 * pa_copy_blocks - the device half of Copy-on-Write.
 *
 * "2.1 PagedAttention" §6: before a request writes a block other requests
 * share, the block is copied to a private block and the request's table
 * entry is repointed (the allocator's pa_alloc_cow does the bookkeeping).
 * For each pair p: block pairs[2p+1] (dst) of k_cache and v_cache becomes a
 * bit-exact copy of block pairs[2p] (src).
 *   pairs  int32 [num_pairs][2] (src, dst), DEVICE memory.  A dst must not
 *          repeat nor be the src of another pair (otherwise the result is
 *          unspecified).  Ids outside [0, num_blocks) record
 *          PA_DEVERR_BLOCK_ID and the pair is skipped.
 * num_pairs == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                   int block_size, int kv_heads, int head_dim, pa_dtype dtype, pa_stream stream);

/* ----------------------------------------------------------------------------
 * pa_swap_blocks - the device half of preemption by swapping.
 *
 * "2.1 PagedAttention" §7: when the GPU pool runs short, a request's blocks
 * are copied to a pool in CPU memory and its GPU blocks are released; later
 * they are copied back into fresh GPU blocks (pa_alloc_swap_out /
 * pa_alloc_swap_in do the bookkeeping and produce the pairs).  For each pair
 * p: block pairs[2p+1] of (dst_k, dst_v) becomes a bit-exact copy of block
 * pairs[2p] of (src_k, src_v).  Both pools have the KV-cache layout
 * [num_*_blocks][block_size][kv_heads][head_dim].
 *   src_*, dst_*  device memory or PAGE-LOCKED host memory (cudaHostAlloc /
 *          cudaHostRegister, mapped); the kernel reads and writes host memory
 *          directly over the CPU-GPU link.  Pageable host memory is rejected
 *          with PA_ERR_INVALID.  All four 16-byte aligned.
 *   pairs  int32 [num_pairs][2] (src, dst), device or page-locked host
 *          memory.  dst ids must not repeat.  A src id outside
 *          [0, num_src_blocks) or a dst id outside [0, num_dst_blocks)
 *          records PA_DEVERR_BLOCK_ID and the pair is skipped.
 * The call is asynchronous on stream; host buffers must stay alive and
 * untouched until it completes.  num_pairs == 0 is a no-op.
 * ------------------------------------------------------------------------- */
int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int32_t* pairs,
                   int num_pairs, int num_src_blocks, int num_dst_blocks, int block_size, int kv_heads,
                   int head_dim, pa_dtype dtype, pa_stream stream);

/* ----------------------------------------------------------------------------
 * Paged decode attention (one query token per request).
 *
 * "2.1 PagedAttention" §3 and §5: the kernel reads the request's whole KV
 * history from scattered physical blocks through its Block Table.  For
 * request r and query head h (g = h / (q_heads / kv_heads)):
 *     s_t = scale * <q[r][h], K_r[t][g]>           for t < context_lens[r]
 *     out[r][h] = sum_t softmax(s)_t * V_r[t][g]
 * context_lens[r] counts every token of the request, including the one this
 * step wrote with pa_reshape_and_cache.  A zero context gives a zero row.
 *
 * The context is processed in partitions of `split_tokens` tokens (0 = the
 * library's choice).  pa_decode_split_tokens returns the partition size a
 * call with these arguments uses, or PA_ERR_INVALID if split_tokens is not
 * allowed.  A request with one
 * partition is written straight to `out`; a request with more keeps per
 * partition the unnormalised output o_c, the reference maximum m_c its
 * exponents were taken against (the running maximum, or up to 8 below it in
 * log2 units) and the sum l_c, and pa_lse_merge combines them:
 * M = max_c m_c,  out = sum_c e^(m_c-M) o_c / sum_c e^(m_c-M) l_c.
 *
 *   q             [num_seqs][q_heads][head_dim]
 *   out           [num_seqs][q_heads][head_dim]
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]
 *   context_lens  int32 [num_seqs], each in [0, max_blocks_per_seq*block_size]
 *   split_tokens  0, or a multiple of max(16, block_size) no larger than
 *                 256*block_size
 *   workspace     device scratch of at least pa_decode_workspace_size(...)
 *                 bytes (may be NULL when that size is 0).  Owned by the
 *                 caller; its contents need no initialisation.
 * pa_decode = pa_decode_partial followed by pa_lse_merge on the same stream.
 * ------------------------------------------------------------------------- */
int pa_decode_split_tokens(int max_blocks_per_seq, int block_size, int split_tokens);

size_t pa_decode_workspace_size(int num_seqs, int q_heads, int head_dim, int max_blocks_per_seq,
                                int block_size, int split_tokens);

int pa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_heads,
              int kv_heads, int head_dim, int block_size, int num_blocks, float scale,
              int split_tokens, void* workspace, size_t workspace_bytes, void* out, pa_dtype dtype,
              pa_stream stream);

/* First half of pa_decode: per-partition partials (or the final row for
 * requests with a single partition). Same arguments as pa_decode. */
int pa_decode_partial(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs, int q_heads, int kv_heads,
                      int head_dim, int block_size, int num_blocks, float scale, int split_tokens,
                      void* workspace, size_t workspace_bytes, void* out, pa_dtype dtype,
                      pa_stream stream);

/* Second half of pa_decode: log-sum-exp merge of the partials of every request
 * with more than one partition.  Arguments must match the pa_decode_partial
 * call whose workspace it reads. */
int pa_lse_merge(const void* workspace, size_t workspace_bytes, const int32_t* context_lens,
                 int num_seqs, int q_heads, int head_dim, int max_blocks_per_seq, int block_size,
                 int split_tokens, void* out, pa_dtype dtype, pa_stream stream);

/* ----------------------------------------------------------------------------
 * pa_verify_decode - the attention of the verify step of speculative decoding.
 *
 * "Khám phá vLLM … phần 2", speculative decoding: a proposer drafts k tokens
 * and the large model checks them in ONE forward pass over the context plus
 * the drafts, which yields k+1 distributions.  Its attention is decode with
 * q_len = k+1 queries per request: the drafts' K/V are written first (with
 * pa_reshape_and_cache, into slots the allocator appended), so
 * context_lens[r] = L counts them, and query i (0 <= i < q_len) of request r
 * attends tokens [0, L - (q_len-1-i)) - causal inside the draft.  A query
 * that sees no token gives a zero row.  All q_len*group query rows of a KV
 * head share every K/V tile read, so the pass costs the KV bytes of one
 * decode step.
 *   q, out        [num_seqs][q_len][q_heads][head_dim]
 *   q_len         >= 1, with (q_heads / kv_heads) * q_len <= 32
 *   split_tokens  as pa_decode; 0 = the library's choice, which for q_len > 1
 *                 and contexts up to 8192 tokens is 768 (longer than decode's:
 *                 each partition's partials and merge rows grow with q_len)
 *   workspace     at least pa_verify_workspace_size(...) bytes
 * Everything else as pa_decode (which is the q_len = 1 case).
 * pa_verify_split_tokens returns the partition size such a call uses, or
 * PA_ERR_INVALID.
 * ------------------------------------------------------------------------- */
int pa_verify_split_tokens(int max_blocks_per_seq, int block_size, int q_len, int split_tokens);

size_t pa_verify_workspace_size(int num_seqs, int q_len, int q_heads, int head_dim, int max_blocks_per_seq,
                                int block_size, int split_tokens);

int pa_verify_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_len, int q_heads,
                     int kv_heads, int head_dim, int block_size, int num_blocks, float scale, int split_tokens,
                     void* workspace, size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream);

/* ----------------------------------------------------------------------------
 * pa_verify_decode_tc - the same verify attention on the tensor cores.
 *
 * The computation of pa_verify_decode ("Khám phá vLLM … phần 2",
 * speculative decoding: query i of request r attends tokens
 * [0, context_lens[r] - (q_len-1-i))), read as what it also is: a chunked
 * prefill of a q_len-token chunk at the end of the context.  The
 * (query, group head) rows of one (request, KV head) - at most 128 - are one
 * work unit of a tcgen05 kernel (tensor memory, TMA gathers) that walks the
 * whole context in 128-key tiles; no workspace, no merge.  A unit's gather
 * cost does not depend on its row count, so this form pays when the rows are
 * many (k = 7 drafts x 4 group heads = 32) and the batch gives every SM units.
 *   q, out        [num_seqs][q_len][q_heads][head_dim], as pa_verify_decode
 *   q_len         >= 1, with (q_heads / kv_heads) * q_len <= 128
 *   block_size    8, 16 or 32 (the gather's boxes hold 8-row swizzle atoms)
 *   max_ctas      0: one CTA per unit; > 0: that many CTAs, each taking units
 *                 b, b + max_ctas, ... (one CTA per SM fits)
 * With one CTA per unit, units of at most 32 rows are spread over all four
 * tensor-memory lane quarters (each takes a quarter of every key tile; the
 * four partial results are merged exactly); a capped grid keeps them in one.
 * Results equal pa_verify_decode's within the attention tolerance (the sums
 * are taken in another order); a query that sees no token gives a zero row.
 * Errors as pa_chunked_prefill.
 * ------------------------------------------------------------------------- */
int pa_verify_decode_tc(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_len, int q_heads,
                        int kv_heads, int head_dim, int block_size, int num_blocks, float scale, int max_ctas,
                        void* out, pa_dtype dtype, pa_stream stream);

/* ----------------------------------------------------------------------------
 * Contiguous virtual KV, vAttention style ("vAttention 完全拆解") - the
 * competing design, built as a comparison baseline for the paged kernels.
 *
 * Each K and V tensor of each layer is ONE contiguous virtual range
 * [num_slots][max_len][kv_heads][head_dim]; request slot s starts at
 * s*max_len*kv_heads*head_dim*2 bytes, token t of the slot is row
 * s*max_len + t, and no Block Table exists.  Physical pages (CUDA virtual
 * memory: cuMemCreate / cuMemMap / cuMemSetAccess) are mapped into a slot
 * only when pa_vkv_step sees its length reach them:
 *  - pages for n tokens: ceil(roundup(n, 16) * kv_heads*head_dim*2 /
 *    page_bytes) in every one of the 2*num_layers sub-tensors (the attention
 *    kernel reads whole 16-token tiles, so the rounded length is mapped);
 *  - pa_vkv_free_slot keeps the slot's pages mapped; pa_vkv_alloc_slot hands
 *    out the free slot holding the most pages (lowest id on ties), whose
 *    pages the new request reuses;
 *  - a step that needs more than max_pages mapped pages in total unmaps whole
 *    inactive slots (lowest id first, after cudaDeviceSynchronize) and fails
 *    with PA_ERR_NO_FREE_BLOCKS, changing nothing, if even that is not enough.
 * page_bytes = 0 takes the driver's minimum granularity (2 MiB on current
 * GPUs); max_len * kv_heads*head_dim*2 must be a multiple of page_bytes and
 * max_len a multiple of 16.  PA_VKV_DRY_RUN keeps only the bookkeeping (no
 * memory, no GPU needed; page_bytes must then be given).
 * Kernels only ever touch rows below a slot's mapped bound: pa_vkv_decode and
 * pa_vkv_reshape_and_cache check every access against the device copy of the
 * per-slot mapped token counts, which pa_vkv_step updates in stream order.
 * ------------------------------------------------------------------------- */
typedef struct pa_vkv pa_vkv;
#define PA_VKV_DRY_RUN 1

typedef struct {
  int64_t page_bytes;
  int64_t slot_pages;        /* virtual pages per slot per sub-tensor          */
  int64_t pages_mapped;      /* over all sub-tensors                           */
  int64_t pages_pooled;      /* created, currently unmapped                    */
  int64_t pages_created;     /* cuMemCreate calls                              */
  int64_t map_calls;         /* page mappings made (one per page per tensor)   */
  int64_t unmap_calls;
  int64_t bytes_reserved;    /* virtual address space                          */
  int64_t bytes_committed;   /* pages_mapped * page_bytes                      */
  int64_t last_step_map_ns;  /* host time the last pa_vkv_step spent mapping   */
  int64_t total_map_ns;
  int64_t active_slots;
  int64_t step_failures;     /* pa_vkv_step calls refused for want of pages   */
  int64_t bytes_used;        /* K/V bytes of the last step's tokens; tail
                                waste = bytes_committed - bytes_used        */
} pa_vkv_stats;

int pa_vkv_granularity(size_t* out);
int pa_vkv_create(int num_slots, int max_len, int num_layers, int kv_heads, int head_dim, pa_dtype dtype,
                  size_t page_bytes, int64_t max_pages, int flags, pa_vkv** out);
/* Synchronises the device, unmaps and releases every page, frees the range. */
void pa_vkv_destroy(pa_vkv* v);
int pa_vkv_alloc_slot(pa_vkv* v, int* slot_out);
int pa_vkv_free_slot(pa_vkv* v, int slot);
/* lens: HOST int32 [num_slots], the length every slot reaches this iteration
 * (0 for inactive slots).  Maps what is missing, then copies the per-slot
 * mapped token counts to the device on `stream`. */
int pa_vkv_step(pa_vkv* v, const int32_t* lens, pa_stream stream);
/* Base of layer `layer`'s K (is_v = 0) or V tensor; NULL in dry-run mode. */
int pa_vkv_tensor(const pa_vkv* v, int layer, int is_v, void** out);
/* Tokens of each slot backed by mapped pages: into host_out [num_slots] (may
 * be NULL); *device_out (may be NULL) = the device copy the kernels read. */
int pa_vkv_slot_tokens(const pa_vkv* v, int32_t* host_out, const int32_t** device_out);
int pa_vkv_slot_pages(const pa_vkv* v, int slot);
int pa_vkv_get_stats(const pa_vkv* v, pa_vkv_stats* out);

/* Decode over a contiguous [num_slots][max_len][kv_heads][head_dim] cache:
 * request r reads slot slot_ids[r] (device int32 [num_seqs]; NULL: slot r),
 * tokens [0, context_lens[r]).  slot_tokens (device int32 [num_slots], may be
 * NULL = all max_len rows exist) bounds the rows each slot has backed by
 * memory: a context past it records PA_DEVERR_CONTEXT_LEN and its tokens past
 * the bound count as absent; a bad slot id records PA_DEVERR_BLOCK_ID and
 * gives a zero row.  Same math, partitions (pa_decode_split_tokens(max_len/16,
 * 16, split_tokens)) and workspace (pa_decode_workspace_size(num_seqs,
 * q_heads, head_dim, max_len/16, 16, split_tokens)) as pa_decode with 16-token
 * blocks, whose result it equals bit for bit on the same K/V. */
int pa_decode_contiguous(const void* q, const void* k_cache, const void* v_cache, int num_slots, int max_len,
                         const int32_t* slot_ids, const int32_t* slot_tokens, const int32_t* context_lens,
                         int num_seqs, int q_heads, int kv_heads, int head_dim, float scale, int split_tokens,
                         void* workspace, size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream);
/* reshape_and_cache into a contiguous cache: token i to row
 * slot_ids[i]*max_len + positions[i] (slot < 0: padding, skipped); a
 * position outside [0, bound) - bound = slot_tokens[slot] or max_len - records
 * PA_DEVERR_SLOT and is skipped. */
int pa_reshape_and_cache_slots(const void* k, const void* v, const int32_t* slot_ids, const int32_t* positions,
                               int num_tokens, void* k_cache, void* v_cache, int num_slots, int max_len,
                               const int32_t* slot_tokens, int kv_heads, int head_dim, pa_dtype dtype,
                               pa_stream stream);
/* The two calls above on layer `layer` of a manager, with its mapped bounds. */
int pa_vkv_decode(const pa_vkv* v, int layer, const void* q, const int32_t* slot_ids, const int32_t* context_lens,
                  int num_seqs, int q_heads, float scale, int split_tokens, void* workspace, size_t workspace_bytes,
                  void* out, pa_stream stream);
int pa_vkv_reshape_and_cache(const pa_vkv* v, int layer, const void* k, const void* vv, const int32_t* slot_ids,
                             const int32_t* positions, int num_tokens, pa_stream stream);

/* ----------------------------------------------------------------------------
 * pa_decode_shared_prefix - decode for a batch whose requests all start with
 * the same physical blocks (a shared prompt prefix).
 *
 * "2.1 PagedAttention" §6: with paging, many Block Tables point at the same
 * physical blocks of a common prefix.  Instead of reading those blocks once per
 * request, this call attends the prefix once for every request's queries:
 * rows (request, query head of the group) x prefix keys are dense tiles for the
 * 5th-generation tensor cores, split into key ranges (512 tokens), each
 * producing a log-sum-exp partial; each request's own suffix (tokens
 * prefix_len .. context_lens[r]-1) runs through the paged decode kernel into
 * further partials; the merge combines them.  The result equals pa_decode
 * with the full tables, up to floating-point rounding.
 *   prefix_blocks  int32 [prefix_len / block_size], DEVICE memory: the shared
 *                  physical blocks in logical order.  Every row of
 *                  block_tables must begin with them (checked on the device:
 *                  a mismatch records PA_DEVERR_BLOCK_ID).
 *   prefix_len     host int, > 0, a multiple of block_size, <= every
 *                  context_lens[r] (a shorter context records
 *                  PA_DEVERR_CONTEXT_LEN).  pa_alloc_common_prefix gives the
 *                  number of shared full blocks of a set of sequences.
 *   workspace      at least pa_decode_shared_prefix_workspace_size(...) bytes.
 *   prefix_stream  NULL (or == stream): all three passes run on `stream`.
 *                  Otherwise the prefix pass runs on prefix_stream, with NO
 *                  dependency on `stream`, concurrently with the suffix pass
 *                  (the prefix pass is tensor-core work on a few SMs, the
 *                  suffix pass HBM-bound on the rest); the merge on `stream`
 *                  waits for it.  The caller orders prefix_stream after every
 *                  write of q, prefix_blocks and the prefix's K/V, and after
 *                  every earlier use of the workspace.  In this mode the
 *                  prefix key ranges grow (512 x 2^k tokens) until the prefix
 *                  pass needs at most a quarter of the SMs.
 * Other arguments as pa_decode.  With 4-token blocks this is pa_decode (on
 * `stream`).
 * ------------------------------------------------------------------------- */
size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int q_heads, int head_dim, int max_blocks_per_seq,
                                              int block_size, int prefix_len, int split_tokens);

/* The partition size pa_decode_shared_prefix uses for the suffixes: split_tokens
 * if it is > 0, else about a quarter of the suffix bound
 * (max_blocks_per_seq * block_size - prefix_len), at least 128 tokens and at
 * most pa_decode_split_tokens(max_blocks_per_seq, block_size, 0).  Negative:
 * a pa_status error for invalid arguments. */
int pa_decode_shared_prefix_split_tokens(int max_blocks_per_seq, int block_size, int prefix_len, int split_tokens);

int pa_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache, const int32_t* prefix_blocks,
                            int prefix_len, const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int q_heads, int kv_heads, int head_dim,
                            int block_size, int num_blocks, float scale, int split_tokens, void* workspace,
                            size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream,
                            pa_stream prefix_stream);

/* ----------------------------------------------------------------------------
 * pa_chunked_prefill - a chunk of prompt tokens per request attends its paged
 * history plus itself, causally.
 *
 * "Khám phá vLLM … phần 2", chunked prefill: a long prompt is prefilled a
 * bounded number of tokens per engine step; the chunk's K/V are written to the
 * cache first (pa_reshape_and_cache) and its queries attend everything before
 * them.  Request r's queries are rows q_start[r] .. q_start[r+1]-1 of q;
 * context_lens[r] includes the chunk, so the chunk starts at absolute
 * position p0 = context_lens[r] - chunk and query i sees keys 0 .. p0 + i.
 *   q, out        [total_q][q_heads][head_dim]
 *   q_start       int32 [num_reqs + 1], non-decreasing, q_start[num_reqs] <= total_q
 *   max_q_len     host-side upper bound of any chunk length (sizes the grid)
 *   max_ctas      with blocks of >= 8 tokens the work is cut into units of
 *                 256 (query, group head) rows of one (request, KV head);
 *                 at most max_ctas CTAs (one per SM) loop over them.  <= 0:
 *                 one CTA per unit.  A caller that runs decode concurrently
 *                 on another stream can leave the remaining SMs to it (decode
 *                 is bound by HBM, not by SM count).  Ignored for 4-token
 *                 blocks.
 * A chunk longer than max_q_len or a context shorter than its chunk records
 * PA_DEVERR_QUERY_RANGE and that request is skipped.
 * ------------------------------------------------------------------------- */
int pa_chunked_prefill(const void* q, const int32_t* q_start, const int32_t* context_lens,
                       const void* k_cache, const void* v_cache, const int32_t* block_tables,
                       int max_blocks_per_seq, int num_reqs, int total_q, int max_q_len, int max_ctas,
                       int q_heads, int kv_heads, int head_dim, int block_size, int num_blocks,
                       float scale, void* out, pa_dtype dtype, pa_stream stream);

/* ----------------------------------------------------------------------------
 * pa_decode_noalloc - pa_decode without a caller-provided workspace.
 *
 * The pages have no counterpart to this call: it only repackages pa_decode
 * for callers that cannot allocate device memory for the decode scratch - a
 * plugin inside a host framework that has already reserved the GPU's memory
 * for its own pool and offers the plugin no allocator, or a latency-critical
 * loop where cudaMalloc/cudaFree (which can synchronise the device) are not
 * acceptable.  The caller still passes all inputs and outputs (same meaning
 * as pa_decode); the split-K partials go to a scratch array held by the
 * library: a file-scope device array of PA_DECODE_NOALLOC_SCRATCH_BYTES
 * (16 MiB) that every GPU loading the library keeps until the process exits.
 * The call allocates nothing.
 *
 * - Size limit: if the scratch this call needs (pa_decode_workspace_size with
 *   the same arguments) exceeds PA_DECODE_NOALLOC_SCRATCH_BYTES it returns
 *   PA_ERR_WORKSPACE and launches nothing; use pa_decode with your own
 *   workspace then.  Requests that fit one partition need no scratch.
 * - Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is looked up again when the
 *   device's current context changes (after cudaDeviceReset the library's
 *   device code is loaded anew and the array may move); the first call after
 *   such a reset should also come before any capture.
 * - Sharing: all calls share the one array, which keeps the last call's
 *   contents.  Nothing in it has to start at zero (every partial the merge
 *   reads is written earlier in the same call).  Calls that overlap on the
 *   GPU (two streams, or two host threads launching at once) race on the
 *   array and corrupt each other's results: serialise them.
 * ------------------------------------------------------------------------- */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_heads,
                      int kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                      int split_tokens, void* out, pa_dtype dtype, pa_stream stream);

/* Read and clear the calling device's error word.  Synchronises `stream`.
 * *host_code receives the PA_DEVERR_* code (0 = none).  Returns
 * PA_ERR_DEVICE_CHECK if a code was recorded, PA_OK otherwise. */
int pa_get_device_error(int32_t* host_code, pa_stream stream);

/* Self-test of the bounded waits: launches one thread that waits on a
 * shared-memory barrier phase nothing completes, with a limit of wait_ms
 * (1..2000) instead of the kernels' 2 s.  The wait gives up, records
 * PA_DEVERR_TIMEOUT in the error word and the kernel finishes normally, as
 * any kernel of the library does when one of its waits expires; the context
 * stays usable.  Asynchronous on `stream`; PA_ERR_INVALID for wait_ms out of
 * range. */
int pa_selftest_wait_timeout(int wait_ms, pa_stream stream);

/* ============================================================================
 * Host block allocator ("2.1 PagedAttention" §9.1-§9.3, §3, §6).
 *
 * A pool of num_blocks physical blocks with a reference count each and a free
 * queue kept as a doubly linked list (O(1) pop from the head, O(1) removal
 * from the middle).  Sequences own Block Tables that grow a block at a time,
 * only when the last block is full.  Tables may share blocks (refcount =
 * number of tables holding the block); a sequence about to write a shared
 * block copies it first (pa_alloc_cow).  Freeing a sequence releases its
 * blocks in reverse order; blocks whose count reaches zero go to the HEAD of
 * the free queue in that order, so a request's last block is reused first.
 * Freed blocks keep their contents (no clearing).
 *
 * Every call is all-or-nothing: on error the state is unchanged.  Handles are
 * single-threaded.  Sequence ids are any non-negative int.
 * ========================================================================== */
typedef struct pa_alloc pa_alloc;

typedef struct {
  int64_t num_blocks;
  int64_t num_free;
  int64_t num_used;        /* blocks with refcount > 0                        */
  int64_t num_shared;      /* blocks with refcount > 1                        */
  int64_t num_seqs;
  int64_t cow_copies;      /* pa_alloc_cow calls that produced a copy          */
  int64_t alloc_failures;  /* calls that returned PA_ERR_NO_FREE_BLOCKS        */
  int64_t waste_slots;     /* sum over sequences of unused slots in the last block */
} pa_alloc_stats;

/* initial_free_order: NULL for ascending ids, else a permutation of
 * 0..num_blocks-1 giving the initial free-queue order (head first). */
int pa_alloc_create(int num_blocks, int block_size, const int32_t* initial_free_order, pa_alloc** out);
void pa_alloc_destroy(pa_alloc* a);

int pa_alloc_add_seq(pa_alloc* a, int seq_id);

/* Give the next n_tokens tokens of seq_id their slots (slots_out[i] =
 * block*block_size + offset), taking new blocks from the head of the free
 * queue only as the last block fills.  PA_ERR_NO_FREE_BLOCKS if the pool
 * cannot cover them; PA_ERR_SHARED_BLOCK if the partially filled last block is
 * shared (call pa_alloc_cow first).  slots_out may be NULL. */
int pa_alloc_append_slots(pa_alloc* a, int seq_id, int n_tokens, int32_t* slots_out);

/* dst_seq (empty) starts with the first n_tokens tokens of src_seq: its table
 * points at src's first ceil(n_tokens/block_size) blocks, each refcount +1. */
int pa_alloc_share(pa_alloc* a, int dst_seq, int src_seq, int n_tokens);

/* Make seq_id's logical block private.  If its refcount is 1, src_dst_out =
 * {b, b} and nothing changes.  Otherwise a fresh block n is taken from the
 * free queue, the table entry becomes n, b's refcount drops by one, and
 * src_dst_out = {b, n}: the caller must then run pa_copy_blocks on (b, n). */
int pa_alloc_cow(pa_alloc* a, int seq_id, int logical_block, int32_t* src_dst_out);

int pa_alloc_free_seq(pa_alloc* a, int seq_id);

/* Copy seq_id's Block Table into out[0..cap); *n_out = its length.
 * PA_ERR_INVALID if cap is too small (nothing written). */
int pa_alloc_block_table(const pa_alloc* a, int seq_id, int32_t* out, int cap, int* n_out);

/* Fill a padded batch table: out is [n][max_blocks_per_seq], row i = table of
 * seq_ids[i] padded with -1; lens_out[i] = its token count (may be NULL). */
int pa_alloc_build_tables(const pa_alloc* a, const int* seq_ids, int n, int32_t* out,
                          int max_blocks_per_seq, int32_t* lens_out);

/* Number of leading FULL blocks that all of seq_ids[0..n) hold in common (same
 * physical ids, in order): the shared prefix pa_decode_shared_prefix can use. */
int pa_alloc_common_prefix(const pa_alloc* a, const int* seq_ids, int n, int* n_blocks_out);
int pa_alloc_seq_len(const pa_alloc* a, int seq_id, int64_t* n_tokens_out);
int pa_alloc_num_free(const pa_alloc* a);
/* Refcount of block_id, or PA_ERR_INVALID if it is out of range. */
int pa_alloc_ref(const pa_alloc* a, int block_id);
/* Free-queue snapshot head to tail into out[0..cap); returns the number
 * written, or PA_ERR_INVALID if cap < the queue length. */
int pa_alloc_free_list(const pa_alloc* a, int32_t* out, int cap);
int pa_alloc_get_stats(const pa_alloc* a, pa_alloc_stats* out);

/* ----------------------------------------------------------------------------
 * Automatic prefix caching ("Khám phá vLLM … phần 2", prefix caching;
 * "2.1 PagedAttention" §9.2-§9.3).  Off until pa_alloc_enable_prefix_caching.
 *
 * Only FULL blocks are cached.  Block i of a sequence has the chained hash
 * h_i = pa_block_hash(h_{i-1}, its block_size token ids), with the sequence's
 * salt as h_{-1}; the allocator keeps a map hash -> block.
 *  - pa_alloc_add_seq_cached: a new sequence whose table starts with the
 *    longest run of cached blocks matching its prompt's full blocks, looked up
 *    in order up to the first miss, at most floor((n_tokens-1)/block_size)
 *    blocks (at least one prompt token is left to compute).  Hit blocks get
 *    refcount +1 and, if they were free, leave the free queue.
 *    *n_cached_out = tokens covered (a multiple of block_size).
 *  - pa_alloc_append_tokens: pa_alloc_append_slots for tokens whose ids are
 *    known; each block they fill is registered (hash -> block) unless that
 *    hash is already cached.  After pa_alloc_append_slots (ids unknown) a
 *    sequence registers nothing more.
 *  - Freeing: blocks whose count reaches zero go to the HEAD of the free queue
 *    if they carry no hash (as above) and to the TAIL if they do, in release
 *    order, so cached blocks are evicted oldest-released first and a
 *    request's first block last.
 *  - A cached block loses its hash only when the free queue hands it out
 *    again (new block, CoW copy); its map entry is removed then.
 *  - pa_alloc_share continues the hash chain into dst only when the shared
 *    part ends on a full, hashed block.
 * ------------------------------------------------------------------------- */
typedef struct {
  int64_t lookup_blocks;  /* prompt blocks looked up by pa_alloc_add_seq_cached */
  int64_t hit_blocks;     /* ... of which were found                          */
  int64_t evictions;      /* cached blocks handed out again (hash dropped)     */
  int64_t cached_blocks;  /* entries in the hash map now                       */
} pa_prefix_cache_stats;

/* 64-bit FNV-1a over parent (8 bytes, little-endian) followed by the n token
 * ids (4 bytes each, little-endian, two's complement). */
uint64_t pa_block_hash(uint64_t parent, const int32_t* tokens, int n);
int pa_alloc_enable_prefix_caching(pa_alloc* a);
/* seq_id must be new; tokens may be NULL when n_tokens == 0; n_cached_out may
 * be NULL.  With caching off this is pa_alloc_add_seq and *n_cached_out = 0. */
int pa_alloc_add_seq_cached(pa_alloc* a, int seq_id, const int32_t* tokens, int n_tokens, uint64_t salt,
                            int* n_cached_out);
/* Errors as pa_alloc_append_slots; tokens may be NULL when n_tokens == 0. */
int pa_alloc_append_tokens(pa_alloc* a, int seq_id, const int32_t* tokens, int n_tokens, int32_t* slots_out);
/* *is_cached_out = 1 and *hash_out = its hash if block_id is in the map, else 0. */
int pa_alloc_block_hash(const pa_alloc* a, int block_id, uint64_t* hash_out, int* is_cached_out);
int pa_alloc_get_prefix_cache_stats(const pa_alloc* a, pa_prefix_cache_stats* out);

/* ----------------------------------------------------------------------------
 * Preemption by swapping ("2.1 PagedAttention" §7).  Off until
 * pa_alloc_enable_swap gives the size of the CPU swap pool (its own free
 * queue of ids 0..num_cpu_blocks-1, handed out from the head).
 *  - pa_alloc_swap_out: the sequence's table moves to swap blocks taken from
 *    the swap pool's head, one per GPU block in logical order; its GPU blocks
 *    are released exactly as pa_alloc_free_seq releases them (a block another
 *    sequence shares stays with that sequence; a cached block keeps its
 *    hash).  pairs_out[i] = (gpu block, swap block) for logical block i: run
 *    pa_swap_blocks(gpu pool -> swap pool) on them BEFORE anything writes the
 *    released GPU blocks.
 *  - pa_alloc_swap_in: the sequence gets new GPU blocks from the free queue
 *    (as appends do); pairs_out[i] = (swap block, gpu block); its swap blocks
 *    return to the swap pool's head, its last block first.  Run
 *    pa_swap_blocks(swap pool -> gpu pool) before the sequence is read.
 *  - While swapped out a sequence can only be swapped in, freed (its swap
 *    blocks return to the swap pool's head) or queried; append, share, CoW,
 *    table building and common-prefix calls on it return PA_ERR_INVALID.
 *    Its block table then lists swap-pool ids.
 * cap is the capacity of pairs_out in pairs; *n_out (may be NULL) = the number
 * of pairs needed, also when cap is too small (PA_ERR_INVALID).  A shortage of
 * swap blocks (swap_out) or GPU blocks (swap_in) returns PA_ERR_NO_FREE_BLOCKS
 * and changes nothing.
 * ------------------------------------------------------------------------- */
int pa_alloc_enable_swap(pa_alloc* a, int num_cpu_blocks);

/* ----------------------------------------------------------------------------
 * Checkpoint and resume of the host allocator: its whole state (free queue
 * order, refcounts, every sequence's Block Table, token count and hashing
 * state, the prefix cache, the swap pool and the counters) as a flat list of
 * int64 words.
 *
 * pa_alloc_export writes the words to out[0..cap) and their number to
 * *n_out; with out = NULL and cap = 0 it only reports the number.  Returns
 * PA_ERR_INVALID if cap is smaller than needed (nothing is written then).
 * Equal states give equal words (sequences and cached hashes are written in
 * key order).
 *
 * pa_alloc_import builds a new allocator (owned by the caller, freed with
 * pa_alloc_destroy) from such words.  It validates every count, id and range
 * and the state's consistency (refcounts equal the tables holding each block,
 * the free queue holds exactly the unheld blocks, the cache holds exactly
 * the hashed blocks under their hashes); malformed words give PA_ERR_INVALID
 * and no allocator.  An imported
 * allocator behaves as the exported one for every later call.
 *
 * Layout (version 1): magic 0x504b5641, version, num_blocks, block_size,
 * caching, num_cpu_blocks, cow_copies, alloc_failures, lookup_blocks,
 * hit_blocks, evictions; n_free and the free queue head to tail; ref[],
 * has_hash[] and hash[] of every block; n_cached and (hash, block) pairs;
 * n_cpu_free and the swap pool's free queue; n_seqs and per sequence (by id):
 * id, num_tokens, salt, parent hash, hashable, swapped, n_blocks, blocks,
 * n_pending, pending token ids.
 * ------------------------------------------------------------------------- */
int pa_alloc_export(const pa_alloc* a, int64_t* out, int64_t cap, int64_t* n_out);
int pa_alloc_import(const int64_t* words, int64_t n, pa_alloc** out);
int pa_alloc_num_free_cpu(const pa_alloc* a);
/* 1 if seq_id is swapped out, 0 if resident, PA_ERR_INVALID if unknown. */
int pa_alloc_is_swapped(const pa_alloc* a, int seq_id);
int pa_alloc_swap_out(pa_alloc* a, int seq_id, int32_t* pairs_out, int cap, int* n_out);
int pa_alloc_swap_in(pa_alloc* a, int seq_id, int32_t* pairs_out, int cap, int* n_out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
