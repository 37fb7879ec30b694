// C ABI of the paged-KV library: argument checks, TMA descriptor cache,
// per-device error word, and the launches (see include/pa.h for the contract).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "pa_internal.h"

namespace pa {

namespace {

std::atomic<uint64_t> g_launches{0};

// Per-device error word: kernels record the first data error here.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
// Automatic partition size: shorter partitions balance the grid better,
// longer ones write fewer partials for the merge.  Measured on GB300: 384 tokens
// is best for contexts up to 8K (batch-64 Llama-8B-style decode), 512 beyond
// (128K-token contexts, where 256 doubles the merge traffic).
constexpr int kAutoSplitShort = 384;
constexpr int kAutoSplitLong = 512;
constexpr int64_t kShortContext = 8192;
// Verify (q_len > 1): each partition writes q_len x the partials of decode and
// the merge has q_len x the rows, so longer partitions pay off.  Measured on
// GB300 (batch 64, contexts 512..4096, k = 3 / 7 drafts, step time in us):
// 256: 108.6 / 143.6, 384: 103.6 / 135.9, 512: 111.4 / 130.7,
// 768: 100.8 / 128.6, 1024: 100.6 / 152.7, 2048: 153.1 / 157.5.
constexpr int kAutoSplitVerify = 768;

std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return -1;
  return d;
}

// Device address of the error word on the current device (set up once).
int* device_error_ptr() {
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[d]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[d] = static_cast<int*>(p);
  }
  return g_err_ptr[d];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// Small cache of KV tensor maps keyed by (pointer, shape, dtype, device).
struct MapKey {
  const void* ptr;
  int64_t rows;
  int kv_heads, head_dim, bsub, dtype, dev;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && kv_heads == o.kv_heads && head_dim == o.head_dim &&
           bsub == o.bsub && dtype == o.dtype && dev == o.dev;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  uint64_t stamp;
  bool used;
};
constexpr int kMapCache = 32;
MapEntry g_maps[kMapCache];
uint64_t g_stamp = 0;

// 4-D view of a cache tensor: {64, head_dim/64, kv_heads, num_blocks*block_size}
// elements, boxes {64, 1, 1, bsub}, 128-byte swizzle.
bool kv_map(const void* base, int num_blocks, int block_size, int kv_heads, int head_dim, pa_dtype dt,
            CUtensorMap* out) {
  const int bsub = block_size < 16 ? block_size : 16;
  const int64_t rows = (int64_t)num_blocks * block_size;
  MapKey key{base, rows, kv_heads, head_dim, bsub, (int)dt, current_device()};
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& e : g_maps)
      if (e.used && e.key == key) {
        e.stamp = ++g_stamp;
        *out = e.map;
        return true;
      }
  }
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)(head_dim / 64), (cuuint64_t)kv_heads, (cuuint64_t)rows};
  cuuint64_t strides[3] = {128, (cuuint64_t)head_dim * 2, (cuuint64_t)kv_heads * head_dim * 2};
  cuuint32_t box[4] = {64, 1, 1, (cuuint32_t)bsub};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMap m;
  CUresult rc = enc(&m, dt == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (rc != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  MapEntry* victim = &g_maps[0];
  for (auto& e : g_maps) {
    if (!e.used) {
      victim = &e;
      break;
    }
    if (e.stamp < victim->stamp) victim = &e;
  }
  victim->key = key;
  victim->map = m;
  victim->stamp = ++g_stamp;
  victim->used = true;
  *out = m;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_kv_shape(int num_blocks, int block_size, int kv_heads, int head_dim, pa_dtype dt) {
  if (dt != PA_FP16 && dt != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_INVALID;
  if (block_size != 4 && block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_INVALID;
  if (kv_heads <= 0 || kv_heads > 1024 || num_blocks <= 0) return PA_ERR_INVALID;
  // row coordinates (one past the pool included) must fit the TMA's int32
  if (((int64_t)num_blocks + 1) * block_size > INT32_MAX) return PA_ERR_INVALID;
  return PA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// The address a kernel dereferences for p: device or managed memory as is,
// page-locked host memory through its mapped device address; nullptr for
// pageable host memory (or anything CUDA does not know).
const void* device_view(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      return at.devicePointer;
    default:
      return nullptr;
  }
}

struct DecodeSetup {
  int split, max_splits;
  DecodeWorkspace ws;
};

int decode_setup(int num_seqs, int q_heads, int head_dim, int max_blocks_per_seq, int block_size, int split_tokens,
                 DecodeSetup* s) {
  const int split = pa_decode_split_tokens(max_blocks_per_seq, block_size, split_tokens);
  if (split <= 0) return PA_ERR_INVALID;
  const int64_t cap = (int64_t)max_blocks_per_seq * block_size;
  if (cap > INT32_MAX) return PA_ERR_INVALID;
  s->split = split;
  s->max_splits = (int)((cap + split - 1) / split);
  if (s->max_splits < 1) s->max_splits = 1;
  s->ws = s->max_splits > 1 ? decode_workspace_layout(num_seqs, q_heads, head_dim, s->max_splits)
                            : DecodeWorkspace{0, 0, 0, 0};
  return PA_OK;
}

// Shared-prefix decode: the prefix is cut into key ranges of kPrefixKeySplit
// (one partial slot each), the suffix into decode partitions after them.  The
// workspace is laid out for this split; a concurrent prefix pass uses longer
// ranges (fewer slots) in the same layout.
constexpr int kPrefixKeySplit = 512;

int sm_count() {
  static int cached[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 0;
  if (!cached[d]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    cached[d] = n;
  }
  return cached[d];
}

// Key range of a prefix pass that runs beside the suffix pass: 512 x 2^k
// tokens, the smallest whose units (pairs of 128-row tiles x KV heads x
// ranges) fit in a quarter of the SMs: the suffix pass is bound by the bytes
// each SM keeps in flight, so the SMs it keeps matter more than how soon the
// prefix pass ends.  Measured on GB300 (256 requests, 2048-token prefix, 32/8
// heads), shared-prefix call: 512-token ranges (128 CTAs) 73.1 us, 1024 (64
// CTAs) 65.5 us, 2048 (32 CTAs) 62.0 us.
int concurrent_key_split(int num_seqs, int group, int kv_heads, int prefix_len) {
  const int64_t row_pairs = ((int64_t)num_seqs * group + 255) / 256;
  const int64_t quarter = sm_count() / 4;
  int ks = kPrefixKeySplit;
  while (ks < prefix_len && row_pairs * kv_heads * ((prefix_len + ks - 1) / ks) > quarter) ks *= 2;
  return ks;
}

// One event per device marks the end of a concurrent prefix pass.
cudaEvent_t prefix_done_event() {
  static cudaEvent_t ev[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!ev[d] && cudaEventCreateWithFlags(&ev[d], cudaEventDisableTiming) != cudaSuccess) return nullptr;
  return ev[d];
}

constexpr int kSuffixSplitMin = 128;  // a multiple of every supported block size

struct SharedPrefixSetup {
  int split, prefix_splits, suffix_splits, max_splits;
  DecodeWorkspace ws;
};

int shared_prefix_setup(int num_seqs, int q_heads, int head_dim, int max_blocks_per_seq, int block_size,
                        int prefix_len, int split_tokens, SharedPrefixSetup* s) {
  if (num_seqs < 0 || q_heads <= 0 || head_dim <= 0) return PA_ERR_INVALID;
  int split = pa_decode_split_tokens(max_blocks_per_seq, block_size, split_tokens);
  if (split <= 0) return PA_ERR_INVALID;
  const int64_t cap = (int64_t)max_blocks_per_seq * block_size;
  if (cap > INT32_MAX || prefix_len <= 0 || prefix_len > cap || prefix_len % block_size != 0) return PA_ERR_INVALID;
  if (split_tokens == 0) {
    // automatic: suffixes are short next to the contexts the decode default
    // is tuned for, so cut them into partitions of about a quarter of their
    // bound (at least kSuffixSplitMin tokens) for more CTAs per KV byte.
    // Measured on GB300 (256 requests, suffixes of 16..512 tokens): 128-token
    // partitions 80.9 us per step, 256: 82.2 us, 384: 84.2 us.
    const int64_t quarter = ((cap - prefix_len) / 4 + block_size - 1) / block_size * block_size;
    const int64_t want = quarter < kSuffixSplitMin ? kSuffixSplitMin : quarter;
    if (want < split) split = (int)want;
  }
  s->split = split;
  s->prefix_splits = (prefix_len + kPrefixKeySplit - 1) / kPrefixKeySplit;
  const int64_t suffix = cap - prefix_len;
  s->suffix_splits = (int)((suffix + split - 1) / split);
  if (s->suffix_splits < 1) s->suffix_splits = 1;
  s->max_splits = s->prefix_splits + s->suffix_splits;
  s->ws = decode_workspace_layout(num_seqs, q_heads, head_dim, s->max_splits);
  return PA_OK;
}

}  // namespace

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

int num_sms() { return sm_count(); }

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID";
    case PA_ERR_NO_FREE_BLOCKS: return "PA_ERR_NO_FREE_BLOCKS";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE_CHECK: return "PA_ERR_DEVICE_CHECK";
    case PA_ERR_SHARED_BLOCK: return "PA_ERR_SHARED_BLOCK";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_HOST_MEMORY: return "PA_ERR_HOST_MEMORY";
    default: return "PA_UNKNOWN_STATUS";
  }
}

int pa_version(void) { return 100; }

uint64_t pa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int pa_reshape_and_cache(const void* k, const void* v, const int32_t* slot_mapping, int num_tokens, void* k_cache,
                         void* v_cache, int num_blocks, int block_size, int kv_heads, int head_dim, pa_dtype dtype,
                         pa_stream stream) {
  int st = check_kv_shape(num_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_INVALID;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  return cuda_status(launch_reshape_and_cache(k, v, slot_mapping, num_tokens, k_cache, v_cache,
                                              (int64_t)num_blocks * block_size, kv_heads * head_dim * 2, err,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks, int block_size,
                   int kv_heads, int head_dim, pa_dtype dtype, pa_stream stream) {
  int st = check_kv_shape(num_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_pairs < 0) return PA_ERR_INVALID;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !pairs || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  return cuda_status(launch_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_blocks,
                                        (int64_t)block_size * kv_heads * head_dim * 2, err,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int pa_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int32_t* pairs,
                   int num_pairs, int num_src_blocks, int num_dst_blocks, int block_size, int kv_heads, int head_dim,
                   pa_dtype dtype, pa_stream stream) {
  int st = check_kv_shape(num_src_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  st = check_kv_shape(num_dst_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_pairs < 0) return PA_ERR_INVALID;
  if (num_pairs == 0) return PA_OK;
  if (!src_k || !src_v || !dst_k || !dst_v || !pairs) return PA_ERR_INVALID;
  if (!aligned16(src_k) || !aligned16(src_v) || !aligned16(dst_k) || !aligned16(dst_v)) return PA_ERR_INVALID;
  const void* sk = device_view(src_k);
  const void* sv = device_view(src_v);
  void* dk = const_cast<void*>(device_view(dst_k));
  void* dv = const_cast<void*>(device_view(dst_v));
  const int32_t* pr = static_cast<const int32_t*>(device_view(pairs));
  if (!sk || !sv || !dk || !dv || !pr) return PA_ERR_INVALID;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  return cuda_status(launch_swap_blocks(sk, sv, dk, dv, pr, num_pairs, num_src_blocks, num_dst_blocks,
                                        (int64_t)block_size * kv_heads * head_dim * 2, err,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int pa_decode_split_tokens(int max_blocks_per_seq, int block_size, int split_tokens) {
  if (max_blocks_per_seq <= 0 || block_size <= 0) return PA_ERR_INVALID;
  const int unit = block_size > 16 ? block_size : 16;
  const int64_t cap = (int64_t)max_blocks_per_seq * block_size;
  int s = split_tokens != 0 ? split_tokens : (cap <= kShortContext ? kAutoSplitShort : kAutoSplitLong);
  if (s <= 0 || s % unit != 0 || s > 256 * block_size) return PA_ERR_INVALID;
  return s;
}

size_t pa_decode_workspace_size(int num_seqs, int q_heads, int head_dim, int max_blocks_per_seq, int block_size,
                                int split_tokens) {
  if (num_seqs < 0 || q_heads <= 0 || head_dim <= 0) return 0;
  DecodeSetup s;
  if (decode_setup(num_seqs, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens, &s) != PA_OK) return 0;
  return s.ws.bytes;
}

namespace {

// The partition pass of decode (q_len = 1) and of the speculative verify
// (q_len = k+1 queries per request, rows r*q_len + i).
int decode_partial_impl(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_len, int q_heads,
                        int kv_heads, int head_dim, int block_size, int num_blocks, float scale, int split_tokens,
                        void* workspace, size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream) {
  int st = check_kv_shape(num_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || q_heads <= 0 || q_heads % kv_heads != 0 || q_heads / kv_heads > 16)
    return PA_ERR_INVALID;
  if (q_len < 1 || (q_heads / kv_heads) * q_len > 32) return PA_ERR_INVALID;
  if (max_blocks_per_seq <= 0 || !std::isfinite(scale)) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_INVALID;
  DecodeSetup s;
  st = decode_setup(num_seqs * q_len, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens, &s);
  if (st != PA_OK) return st;
  if (s.ws.bytes > 0 && (!workspace || workspace_bytes < s.ws.bytes || !aligned16(workspace)))
    return PA_ERR_WORKSPACE;
  if ((int64_t)s.max_splits * kv_heads > (int64_t)INT32_MAX) return PA_ERR_INVALID;
  CUtensorMap km, vm;
  if (!kv_map(k_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &km) ||
      !kv_map(v_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &vm))
    return PA_ERR_CUDA;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  DecodeParams p{};
  p.q = q;
  p.tables = block_tables;
  p.lens = context_lens;
  p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_o = s.ws.bytes ? reinterpret_cast<float*>(ws + s.ws.o_off) : nullptr;
  p.part_m = s.ws.bytes ? reinterpret_cast<float*>(ws + s.ws.m_off) : nullptr;
  p.part_l = s.ws.bytes ? reinterpret_cast<float*>(ws + s.ws.l_off) : nullptr;
  p.err = err;
  p.maxblk = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.q_heads = q_heads;
  p.kv_heads = kv_heads;
  p.group = q_heads / kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.split_tokens = s.split;
  p.max_splits = s.max_splits;
  p.grid_splits = s.max_splits;
  p.tab_entries = s.split / block_size;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_len = q_len;
  const int bsub = block_size < 16 ? block_size : 16;
  return cuda_status(
      launch_decode_partial(km, vm, p, head_dim, bsub, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

int lse_merge_impl(const void* workspace, size_t workspace_bytes, const int32_t* context_lens, int num_seqs,
                   int q_len, int q_heads, int head_dim, int max_blocks_per_seq, int block_size, int split_tokens,
                   void* out, pa_dtype dtype, pa_stream stream) {
  if (dtype != PA_FP16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_INVALID;
  if (num_seqs < 0 || q_heads <= 0 || q_len < 1) return PA_ERR_INVALID;
  // the merge kernels number their (request, query, head) rows in int32
  if ((int64_t)num_seqs * q_len * q_heads > (int64_t)INT32_MAX - 8) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  DecodeSetup s;
  int st = decode_setup(num_seqs * q_len, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens, &s);
  if (st != PA_OK) return st;
  if (s.ws.bytes == 0) return PA_OK;  // a single partition: pa_decode_partial wrote `out`
  if (!workspace || workspace_bytes < s.ws.bytes || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  if (!context_lens || !out || !aligned16(out)) return PA_ERR_INVALID;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  MergeParams p{};
  p.part_o = reinterpret_cast<const float*>(ws + s.ws.o_off);
  p.part_m = reinterpret_cast<const float*>(ws + s.ws.m_off);
  p.part_l = reinterpret_cast<const float*>(ws + s.ws.l_off);
  p.lens = context_lens;
  p.out = out;
  p.num_seqs = num_seqs;
  p.q_heads = q_heads;
  p.max_splits = s.max_splits;
  p.split_tokens = s.split;
  p.cap = max_blocks_per_seq * block_size;
  p.q_len = q_len;
  return cuda_status(launch_lse_merge(p, head_dim, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

int pa_decode_partial(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_heads, int kv_heads,
                      int head_dim, int block_size, int num_blocks, float scale, int split_tokens, void* workspace,
                      size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream) {
  return decode_partial_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, 1,
                             q_heads, kv_heads, head_dim, block_size, num_blocks, scale, split_tokens, workspace,
                             workspace_bytes, out, dtype, stream);
}

int pa_lse_merge(const void* workspace, size_t workspace_bytes, const int32_t* context_lens, int num_seqs,
                 int q_heads, int head_dim, int max_blocks_per_seq, int block_size, int split_tokens, void* out,
                 pa_dtype dtype, pa_stream stream) {
  return lse_merge_impl(workspace, workspace_bytes, context_lens, num_seqs, 1, q_heads, head_dim,
                        max_blocks_per_seq, block_size, split_tokens, out, dtype, stream);
}

int pa_decode_contiguous(const void* q, const void* k_cache, const void* v_cache, int num_slots, int max_len,
                         const int32_t* slot_ids, const int32_t* slot_tokens, const int32_t* context_lens,
                         int num_seqs, int q_heads, int kv_heads, int head_dim, float scale, int split_tokens,
                         void* workspace, size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream) {
  if (num_slots <= 0 || max_len <= 0 || max_len % 16 != 0 || (int64_t)num_slots * max_len > INT32_MAX - 16)
    return PA_ERR_INVALID;
  const int maxblk = max_len / 16;
  int st = check_kv_shape(num_slots * maxblk, 16, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || q_heads <= 0 || q_heads % kv_heads != 0 || q_heads / kv_heads > 16)
    return PA_ERR_INVALID;
  if (!std::isfinite(scale)) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !context_lens || !out) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_INVALID;
  DecodeSetup s;
  st = decode_setup(num_seqs, q_heads, head_dim, maxblk, 16, split_tokens, &s);
  if (st != PA_OK) return st;
  if (s.ws.bytes > 0 && (!workspace || workspace_bytes < s.ws.bytes || !aligned16(workspace)))
    return PA_ERR_WORKSPACE;
  CUtensorMap km, vm;
  if (!kv_map(k_cache, num_slots * maxblk, 16, kv_heads, head_dim, dtype, &km) ||
      !kv_map(v_cache, num_slots * maxblk, 16, kv_heads, head_dim, dtype, &vm))
    return PA_ERR_CUDA;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  DecodeParams p{};
  p.q = q;
  p.lens = context_lens;
  p.out = out;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_o = s.ws.bytes ? reinterpret_cast<float*>(ws + s.ws.o_off) : nullptr;
  p.part_m = s.ws.bytes ? reinterpret_cast<float*>(ws + s.ws.m_off) : nullptr;
  p.part_l = s.ws.bytes ? reinterpret_cast<float*>(ws + s.ws.l_off) : nullptr;
  p.err = err;
  p.maxblk = maxblk;
  p.num_seqs = num_seqs;
  p.q_heads = q_heads;
  p.kv_heads = kv_heads;
  p.group = q_heads / kv_heads;
  p.num_blocks = num_slots * maxblk;
  p.block_size = 16;
  p.split_tokens = s.split;
  p.max_splits = s.max_splits;
  p.grid_splits = s.max_splits;
  p.tab_entries = 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_len = 1;
  p.slot_ids = slot_ids;
  p.slot_tokens = slot_tokens;
  p.num_slots = num_slots;
  p.contig_len = max_len;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  st = cuda_status(launch_decode_contig(km, vm, p, head_dim, dtype, cs));
  if (st != PA_OK) return st;
  return lse_merge_impl(workspace, workspace_bytes, context_lens, num_seqs, 1, q_heads, head_dim, maxblk, 16,
                        split_tokens, out, dtype, stream);
}

int pa_reshape_and_cache_slots(const void* k, const void* v, const int32_t* slot_ids, const int32_t* positions,
                               int num_tokens, void* k_cache, void* v_cache, int num_slots, int max_len,
                               const int32_t* slot_tokens, int kv_heads, int head_dim, pa_dtype dtype,
                               pa_stream stream) {
  if (num_slots <= 0 || max_len <= 0 || max_len % 16 != 0 || (int64_t)num_slots * max_len > INT32_MAX - 16)
    return PA_ERR_INVALID;
  int st = check_kv_shape(num_slots * (max_len / 16), 16, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_INVALID;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_ids || !positions || !k_cache || !v_cache) return PA_ERR_INVALID;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  return cuda_status(launch_reshape_and_cache_slots(k, v, slot_ids, positions, num_tokens, k_cache, v_cache,
                                                    num_slots, max_len, slot_tokens, kv_heads * head_dim * 2, err,
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

int pa_verify_split_tokens(int max_blocks_per_seq, int block_size, int q_len, int split_tokens) {
  if (q_len < 1) return PA_ERR_INVALID;
  if (split_tokens == 0 && q_len > 1 && max_blocks_per_seq > 0 && block_size > 0 &&
      (int64_t)max_blocks_per_seq * block_size <= kShortContext)
    split_tokens = kAutoSplitVerify;
  return pa_decode_split_tokens(max_blocks_per_seq, block_size, split_tokens);
}

size_t pa_verify_workspace_size(int num_seqs, int q_len, int q_heads, int head_dim, int max_blocks_per_seq,
                                int block_size, int split_tokens) {
  if (num_seqs < 0 || q_len < 1 || q_heads <= 0 || head_dim <= 0) return 0;
  if ((int64_t)num_seqs * q_len > INT32_MAX) return 0;
  split_tokens = pa_verify_split_tokens(max_blocks_per_seq, block_size, q_len, split_tokens);
  if (split_tokens < 0) return 0;
  DecodeSetup s;
  if (decode_setup(num_seqs * q_len, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens, &s) != PA_OK)
    return 0;
  return s.ws.bytes;
}

int pa_verify_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_len, int q_heads,
                     int kv_heads, int head_dim, int block_size, int num_blocks, float scale, int split_tokens,
                     void* workspace, size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream) {
  if (q_len < 1 || (int64_t)num_seqs * q_len > INT32_MAX / 64) return PA_ERR_INVALID;
  split_tokens = pa_verify_split_tokens(max_blocks_per_seq, block_size, q_len, split_tokens);
  if (split_tokens < 0) return split_tokens;
  int st = decode_partial_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, q_len,
                               q_heads, kv_heads, head_dim, block_size, num_blocks, scale, split_tokens, workspace,
                               workspace_bytes, out, dtype, stream);
  if (st != PA_OK) return st;
  return lse_merge_impl(workspace, workspace_bytes, context_lens, num_seqs, q_len, q_heads, head_dim,
                        max_blocks_per_seq, block_size, split_tokens, out, dtype, stream);
}

int pa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_heads, int kv_heads,
              int head_dim, int block_size, int num_blocks, float scale, int split_tokens, void* workspace,
              size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream) {
  int st = pa_decode_partial(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, q_heads,
                             kv_heads, head_dim, block_size, num_blocks, scale, split_tokens, workspace,
                             workspace_bytes, out, dtype, stream);
  if (st != PA_OK) return st;
  return pa_lse_merge(workspace, workspace_bytes, context_lens, num_seqs, q_heads, head_dim, max_blocks_per_seq,
                      block_size, split_tokens, out, dtype, stream);
}

int pa_chunked_prefill(const void* q, const int32_t* q_start, const int32_t* context_lens, const void* k_cache,
                       const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq, int num_reqs,
                       int total_q, int max_q_len, int max_ctas, int q_heads, int kv_heads, int head_dim,
                       int block_size, int num_blocks, float scale, void* out, pa_dtype dtype, pa_stream stream) {
  int st = check_kv_shape(num_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_reqs < 0 || num_reqs > 65535 || total_q < 0 || max_q_len < 0 || q_heads <= 0 ||
      q_heads % kv_heads != 0 || kv_heads > 65535 || max_blocks_per_seq <= 0 || !std::isfinite(scale))
    return PA_ERR_INVALID;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_INVALID;
  if (num_reqs == 0 || max_q_len == 0 || total_q == 0) return PA_OK;
  if ((int64_t)max_q_len * (q_heads / kv_heads) > (int64_t)INT32_MAX / 2) return PA_ERR_INVALID;
  if (!q || !q_start || !context_lens || !k_cache || !v_cache || !block_tables || !out) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_INVALID;
  CUtensorMap km, vm;
  if (!kv_map(k_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &km) ||
      !kv_map(v_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &vm))
    return PA_ERR_CUDA;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  PrefillParams p{};
  p.q = q;
  p.q_start = q_start;
  p.lens = context_lens;
  p.tables = block_tables;
  p.out = out;
  p.err = err;
  p.maxblk = max_blocks_per_seq;
  p.num_reqs = num_reqs;
  p.total_q = total_q;
  p.max_q_len = max_q_len;
  p.q_heads = q_heads;
  p.kv_heads = kv_heads;
  p.group = q_heads / kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = 1;
  p.max_ctas = max_ctas;
  const int bsub = block_size < 16 ? block_size : 16;
  cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  // blocks of >= 8 tokens: 5th-generation tensor cores (tcgen05 + TMEM);
  // 4-token blocks: warp-level MMA kernel
  if (bsub >= 8) return cuda_status(launch_attn_tc(km, vm, p, head_dim, bsub, dtype, st_));
  return cuda_status(launch_chunked_prefill(km, vm, p, head_dim, bsub, dtype, st_));
}

int pa_verify_decode_tc(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int q_len, int q_heads,
                        int kv_heads, int head_dim, int block_size, int num_blocks, float scale, int max_ctas,
                        void* out, pa_dtype dtype, pa_stream stream) {
  int st = check_kv_shape(num_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (block_size < 8 || num_seqs < 0 || num_seqs > 65535 || q_len < 1 || q_heads <= 0 || q_heads % kv_heads != 0 ||
      (q_heads / kv_heads) * q_len > 128 || max_blocks_per_seq <= 0 || !std::isfinite(scale))
    return PA_ERR_INVALID;
  if ((int64_t)max_blocks_per_seq * block_size > INT32_MAX) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_INVALID;
  CUtensorMap km, vm;
  if (!kv_map(k_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &km) ||
      !kv_map(v_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &vm))
    return PA_ERR_CUDA;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  PrefillParams p{};
  p.q = q;
  p.lens = context_lens;
  p.tables = block_tables;
  p.out = out;
  p.err = err;
  p.maxblk = max_blocks_per_seq;
  p.num_reqs = num_seqs;
  p.total_q = num_seqs * q_len;
  p.max_q_len = q_len;
  p.fixed_q_len = q_len;
  p.q_heads = q_heads;
  p.kv_heads = kv_heads;
  p.group = q_heads / kv_heads;
  p.num_blocks = num_blocks;
  p.block_size = block_size;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = 1;
  p.max_ctas = max_ctas;
  return cuda_status(launch_attn_tile(km, vm, p, head_dim, block_size < 16 ? block_size : 16, dtype,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int q_heads, int head_dim, int max_blocks_per_seq,
                                              int block_size, int prefix_len, int split_tokens) {
  if (block_size < 8)  // 4-token blocks: plain pa_decode is used
    return pa_decode_workspace_size(num_seqs, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens);
  SharedPrefixSetup s;
  if (shared_prefix_setup(num_seqs, q_heads, head_dim, max_blocks_per_seq, block_size, prefix_len, split_tokens,
                          &s) != PA_OK)
    return 0;
  return s.ws.bytes;
}

int pa_decode_shared_prefix_split_tokens(int max_blocks_per_seq, int block_size, int prefix_len, int split_tokens) {
  if (block_size < 8) return pa_decode_split_tokens(max_blocks_per_seq, block_size, split_tokens);
  SharedPrefixSetup s;
  const int st = shared_prefix_setup(1, 1, 64, max_blocks_per_seq, block_size, prefix_len, split_tokens, &s);
  return st != PA_OK ? st : s.split;
}

int pa_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache, const int32_t* prefix_blocks,
                            int prefix_len, const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int q_heads, int kv_heads, int head_dim,
                            int block_size, int num_blocks, float scale, int split_tokens, void* workspace,
                            size_t workspace_bytes, void* out, pa_dtype dtype, pa_stream stream,
                            pa_stream prefix_stream) {
  int st = check_kv_shape(num_blocks, block_size, kv_heads, head_dim, dtype);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535 || q_heads <= 0 || q_heads % kv_heads != 0 || q_heads / kv_heads > 16)
    return PA_ERR_INVALID;
  if (max_blocks_per_seq <= 0 || !std::isfinite(scale)) return PA_ERR_INVALID;
  if (prefix_len <= 0 || prefix_len % block_size != 0 || prefix_len > (int64_t)max_blocks_per_seq * block_size)
    return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (block_size < 8)  // no tensor-core prefix pass for 4-token blocks: same result through pa_decode
    return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, q_heads, kv_heads,
                     head_dim, block_size, num_blocks, scale, split_tokens, workspace, workspace_bytes, out, dtype,
                     stream);
  if (!q || !k_cache || !v_cache || !prefix_blocks || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_ERR_INVALID;
  SharedPrefixSetup s;
  st = shared_prefix_setup(num_seqs, q_heads, head_dim, max_blocks_per_seq, block_size, prefix_len, split_tokens, &s);
  if (st != PA_OK) return st;
  if (!workspace || workspace_bytes < s.ws.bytes || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  CUtensorMap km, vm;
  if (!kv_map(k_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &km) ||
      !kv_map(v_cache, num_blocks, block_size, kv_heads, head_dim, dtype, &vm))
    return PA_ERR_CUDA;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* po = reinterpret_cast<float*>(ws + s.ws.o_off);
  float* pm = reinterpret_cast<float*>(ws + s.ws.m_off);
  float* pl = reinterpret_cast<float*>(ws + s.ws.l_off);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int bsub = block_size < 16 ? block_size : 16;
  const int G = q_heads / kv_heads;
  const float sl2 = scale * 1.4426950408889634f;
  const bool concurrent = prefix_stream != nullptr && prefix_stream != stream;
  cudaEvent_t done = nullptr;
  if (concurrent && !(done = prefix_done_event())) return PA_ERR_CUDA;
  const int key_split = concurrent ? concurrent_key_split(num_seqs, G, kv_heads, prefix_len) : kPrefixKeySplit;
  const int prefix_splits = (prefix_len + key_split - 1) / key_split;  // <= s.prefix_splits

  // 1. the shared prefix, once for every request's queries (tensor cores)
  PrefillParams pp{};
  pp.q = q;
  pp.tables = prefix_blocks;
  pp.err = err;
  pp.maxblk = prefix_len / block_size;
  pp.num_reqs = 1;
  pp.total_q = num_seqs;
  pp.max_q_len = num_seqs;
  pp.q_heads = q_heads;
  pp.kv_heads = kv_heads;
  pp.group = G;
  pp.num_blocks = num_blocks;
  pp.block_size = block_size;
  pp.scale_log2 = sl2;
  pp.causal = 0;
  pp.prefix_len = prefix_len;
  pp.key_split = key_split;
  pp.max_splits = s.max_splits;
  pp.part_o = po;
  pp.part_m = pm;
  pp.part_l = pl;
  if (concurrent) {
    cudaStream_t ps = reinterpret_cast<cudaStream_t>(prefix_stream);
    st = cuda_status(launch_attn_tc(km, vm, pp, head_dim, bsub, dtype, ps));
    if (st == PA_OK) st = cuda_status(cudaEventRecord(done, ps));
  } else {
    st = cuda_status(launch_attn_tc(km, vm, pp, head_dim, bsub, dtype, cs));
  }
  if (st != PA_OK) return st;

  // 2. each request's own suffix (paged decode, partials after the prefix's)
  DecodeParams dp{};
  dp.q = q;
  dp.tables = block_tables;
  dp.lens = context_lens;
  dp.out = out;
  dp.part_o = po;
  dp.part_m = pm;
  dp.part_l = pl;
  dp.err = err;
  dp.maxblk = max_blocks_per_seq;
  dp.num_seqs = num_seqs;
  dp.q_heads = q_heads;
  dp.kv_heads = kv_heads;
  dp.group = G;
  dp.num_blocks = num_blocks;
  dp.block_size = block_size;
  dp.split_tokens = s.split;
  dp.max_splits = s.max_splits;
  dp.grid_splits = s.suffix_splits;
  dp.tab_entries = s.split / block_size;
  dp.scale_log2 = sl2;
  dp.tok_begin = prefix_len;
  dp.slot_base = prefix_splits;
  dp.always_partial = 1;
  dp.prefix_blocks = prefix_blocks;
  dp.prefix_nblk = prefix_len / block_size;
  dp.q_len = 1;
  st = cuda_status(launch_decode_partial(km, vm, dp, head_dim, bsub, dtype, cs));
  if (st != PA_OK) return st;

  // 3. log-sum-exp merge of prefix and suffix partials
  MergeParams mp{};
  mp.part_o = po;
  mp.part_m = pm;
  mp.part_l = pl;
  mp.lens = context_lens;
  mp.out = out;
  mp.num_seqs = num_seqs;
  mp.q_heads = q_heads;
  mp.max_splits = s.max_splits;
  mp.split_tokens = s.split;
  mp.cap = max_blocks_per_seq * block_size;
  mp.tok_begin = prefix_len;
  mp.extra_slots = prefix_splits;
  mp.always = 1;
  mp.q_len = 1;
  if (concurrent && cudaStreamWaitEvent(cs, done, 0) != cudaSuccess) return PA_ERR_CUDA;
  return cuda_status(launch_lse_merge(mp, head_dim, dtype, cs));
}

int pa_selftest_wait_timeout(int wait_ms, pa_stream stream) {
  if (wait_ms < 1 || wait_ms > 2000) return PA_ERR_INVALID;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  return cuda_status(launch_wait_timeout(err, (uint64_t)wait_ms * 1000000ull, reinterpret_cast<cudaStream_t>(stream)));
}

int pa_get_device_error(int32_t* host_code, pa_stream stream) {
  if (!host_code) return PA_ERR_INVALID;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  *host_code = v;
  return v ? PA_ERR_DEVICE_CHECK : PA_OK;
}

}  // extern "C"
