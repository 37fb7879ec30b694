// pa_decode_noalloc: paged decode for callers that cannot allocate device
// memory for the decode scratch.
//
// Who needs it: a plugin running inside a host framework that has already
// reserved the GPU's memory for its own pool and gives the plugin no allocator,
// and latency-critical loops in which cudaMalloc/cudaFree (which can
// synchronise the device) are not acceptable.  Such callers still pass their
// inputs and outputs; only the split-K partials move into a scratch array that
// the library itself holds.
//
// The array is a file-scope __device__ variable of PA_DECODE_NOALLOC_SCRATCH_BYTES:
// every GPU that loads the library holds it until the process exits.  Host
// code must not pass the array's name to a kernel (on the host it is only a
// stand-in symbol); the device address is looked up with cudaGetSymbolAddress,
// with that device current, on the first call there, and again whenever the
// device's current context is not the one the address was taken in (after
// cudaDeviceReset, or once the primary context was released and created anew,
// the module is loaded again and the array may sit at another address).
#include <mutex>

#include "pa_internal.h"

namespace {

constexpr size_t kScratchBytes = PA_DECODE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // id of the context each address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context; 0 if there is none yet
// or the driver cannot say (then the address is looked up on every call).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<CtxGetCurrentFn>(fn)
               : nullptr;
  }();
  static CtxGetIdFn get_id = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    return cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess
               ? reinterpret_cast<CtxGetIdFn>(fn)
               : nullptr;
  }();
  CUcontext c = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] && ctx != 0 && ctx == g_scratch_ctx[dev]) return g_scratch_ptr[dev];
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
  g_scratch_ptr[dev] = p;
  g_scratch_ctx[dev] = current_context_id();  // the lookup made the device's context current
  return p;
}

}  // namespace

extern "C" int pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                                 int num_seqs, int q_heads, int kv_heads, int head_dim, int block_size,
                                 int num_blocks, float scale, int split_tokens, void* out, pa_dtype dtype,
                                 pa_stream stream) {
  // Scratch this call needs: exactly what pa_decode would ask the caller for
  // (0 when every request fits one partition, or when the arguments are
  // invalid - pa_decode then reports the argument error).
  const size_t need =
      pa_decode_workspace_size(num_seqs, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens);
  if (need > kScratchBytes) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    scratch = scratch_on_current_device();
    if (!scratch) return PA_ERR_CUDA;
  }
  return pa_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs, q_heads,
                   kv_heads, head_dim, block_size, num_blocks, scale, split_tokens, scratch,
                   need > 0 ? kScratchBytes : 0, out, dtype, stream);
}
