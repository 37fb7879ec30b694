// Internal interfaces between the library's translation units (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "pa.h"

namespace pa {

// Counts kernel launches (pa_launch_count).
void note_launch(int n = 1);

// Launch with programmatic stream serialisation (programmatic dependent
// launch): the kernel may start while the previous kernel on the stream is
// finishing; it synchronises with griddepcontrol.wait before touching memory
// that kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e == cudaSuccess) note_launch();
  return e;
}

struct DecodeParams {
  const void* q;
  const int32_t* tables;
  const int32_t* lens;
  void* out;
  float* part_o;   // [num_seqs][q_heads][max_splits][head_dim]
  float* part_m;   // [num_seqs][q_heads][max_splits], log2 units
  float* part_l;   // [num_seqs][q_heads][max_splits]
  int* err;
  int maxblk, num_seqs, q_heads, kv_heads, group, num_blocks, block_size, split_tokens, max_splits;
  int tab_entries;  // block-table entries per partition: split_tokens / block_size
  float scale_log2;
  // Shared-prefix mode: attend only tokens [tok_begin, context_len) (the
  // request's own suffix), always write partials, to slots slot_base + c, and
  // check that each table starts with the prefix blocks.
  int tok_begin, slot_base, always_partial;
  const int32_t* prefix_blocks;
  int prefix_nblk;
  int grid_splits;  // partitions the grid covers (normal mode: max_splits)
  // Queries per request (1 = decode; k+1 = speculative verify).  Query i of
  // request r is row r*q_len + i of q / out / the partials and sees tokens
  // [0, context_len - (q_len-1-i)).
  int q_len;
  // Contiguous mode (launch_decode_contig): the cache is [num_slots][contig_len]
  // rows; request r reads slot slot_ids[r] (r if null); slot_tokens (may be
  // null) bounds the rows of each slot that are backed by memory.
  const int32_t* slot_ids;
  const int32_t* slot_tokens;
  int num_slots, contig_len;
};

struct MergeParams {
  const float* part_o;
  const float* part_m;
  const float* part_l;
  const int32_t* lens;
  void* out;
  int num_seqs, q_heads, max_splits, split_tokens, cap;
  // shared-prefix mode: extra_slots partials precede the suffix partitions of
  // [tok_begin, context_len); every row is merged (even a single slot)
  int tok_begin, extra_slots, always;
  int q_len;  // queries per request: row / (q_heads * q_len) is the request
};

struct PrefillParams {
  const void* q;
  const int32_t* q_start;
  const int32_t* lens;
  const int32_t* tables;
  void* out;
  int* err;
  int maxblk, num_reqs, total_q, max_q_len, q_heads, kv_heads, group, num_blocks, block_size;
  float scale_log2;
  // Shared-prefix mode (tcgen05 kernel only; causal == 0): one virtual request
  // whose total_q "queries" are the decode queries of a batch, all seeing keys
  // [0, prefix_len) of the prefix table (`tables`, one row); grid.z splits the
  // keys into ranges of key_split; each range writes an unnormalised partial
  // (o, m in log2 units, l) to slot blockIdx.z of the decode workspace.
  int causal;
  int prefix_len, key_split, max_splits;
  // tcgen05 path: CTAs launched (each takes work units b, b + gridDim.x, ...);
  // <= 0 launches one CTA per unit
  int max_ctas;
  // > 0 (one-tile kernel, causal): every request has fixed_q_len queries, rows
  // r*fixed_q_len.. of q and out (q_start unused), and a context shorter than
  // that leaves the first queries without keys (zero rows): the speculative
  // verify
  int fixed_q_len;
  float* part_o;
  float* part_m;
  float* part_l;
};

// Workspace carve-up for decode partials.
struct DecodeWorkspace {
  size_t o_off, m_off, l_off, bytes;
};
DecodeWorkspace decode_workspace_layout(int num_seqs, int q_heads, int head_dim, int max_splits);

// Launchers (return cudaSuccess or the launch error).  `bsub` is the TMA box
// height min(block_size, 16); the tensor maps describe k_cache / v_cache as
// 4-D {64, head_dim/64, kv_heads, num_blocks*block_size} with boxes
// {64, 1, 1, bsub} and the 128-byte swizzle.
cudaError_t launch_decode_partial(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                  int head_dim, int bsub, pa_dtype dt, cudaStream_t stream);
cudaError_t launch_lse_merge(const MergeParams& p, int head_dim, pa_dtype dt, cudaStream_t stream);
cudaError_t launch_decode_contig(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                 int head_dim, pa_dtype dt, cudaStream_t stream);
cudaError_t launch_chunked_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                                   int head_dim, int bsub, pa_dtype dt, cudaStream_t stream);
// tcgen05/TMEM kernel for blocks of >= 8 tokens (bsub >= 8): chunked prefill
// (p.causal = 1) and the shared-prefix pass of a decode batch (p.causal = 0,
// partials).  Two 128-row Q tiles per CTA, 128-key K/V tiles, P kept in TMEM.
cudaError_t launch_wait_timeout(int* err, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_attn_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p, int head_dim,
                           int bsub, pa_dtype dt, cudaStream_t stream);
// SMs of the current device (cached per device; 0 if the query fails).
int num_sms();
// Grid of a grid-stride copy kernel: enough 256-thread CTAs for `total`
// vectors, at most 16 per SM of the current device.
inline unsigned copy_grid(int64_t total) {
  const int64_t cap = 16 * (int64_t)(num_sms() > 0 ? num_sms() : 1);
  const int64_t want = (total + 255) / 256;
  return (unsigned)(want < cap ? want : cap);
}
// tcgen05 kernel with one 128-row tile per (request, KV head) work unit and
// Q, P in tensor memory (causal with fixed_q_len: the speculative verify).
cudaError_t launch_attn_tile(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                             int head_dim, int bsub, pa_dtype dt, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const void* k, const void* v, const int32_t* slots, int num_tokens,
                                     void* k_cache, void* v_cache, int64_t num_slots, int row_bytes, int* err,
                                     cudaStream_t stream);
// pointers as the kernel dereferences them (host pools through their mapped
// device addresses); block_bytes = one block of K (or V)
cudaError_t launch_reshape_and_cache_slots(const void* k, const void* v, const int32_t* slot_ids,
                                           const int32_t* positions, int num_tokens, void* k_cache, void* v_cache,
                                           int num_slots, int contig_len, const int32_t* slot_tokens, int row_bytes,
                                           int* err, cudaStream_t stream);
cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int32_t* pairs,
                               int num_pairs, int num_src, int num_dst, int64_t block_bytes, int* err,
                               cudaStream_t stream);
cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                               int num_blocks, int64_t block_bytes, int* err, cudaStream_t stream);

}  // namespace pa
