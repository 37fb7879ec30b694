// vAttention-style KV memory manager: contiguous virtual KV tensors whose
// physical pages are mapped on demand with the CUDA virtual memory API.
//
// "vAttention 完全拆解": each K and V tensor of each layer is one virtual range
// [num_slots][max_len][kv_heads][head_dim]; slot s starts at s*max_len*row
// bytes.  Pages of page_bytes are created (cuMemCreate), mapped into a slot's
// range (cuMemMap + cuMemSetAccess) only when a step's lengths reach them,
// kept mapped when the slot's request finishes (a later request on the slot
// reuses them), and unmapped only when a step cannot be covered otherwise:
// then whole inactive slots give their pages back, after the device has been
// synchronised so that no kernel still reads them.  Unmapped pages stay in a
// pool of handles for reuse; they are released at destroy.
//
// The bookkeeping is a model of its own (no shared code with the oracle):
//   pages_for(n)  = ceil(roundup(n, 16) * row / page_bytes)   per sub-tensor
//   alloc_slot    = the free slot holding the most pages, lowest id on ties
//   step          = all or nothing
// With PA_VKV_DRY_RUN nothing is reserved, created or mapped; the same
// bookkeeping runs, so host logic is testable without a GPU.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <chrono>
#include <cstdint>
#include <cstring>
#include <memory>
#include <vector>

#include "pa.h"
#include "pa_guard.h"
#include "pa_internal.h"

namespace {

struct Driver {
  PFN_cuMemGetAllocationGranularity_v10020 granularity = nullptr;
  PFN_cuMemAddressReserve_v10020 reserve = nullptr;
  PFN_cuMemAddressFree_v10020 addr_free = nullptr;
  PFN_cuMemCreate_v10020 create = nullptr;
  PFN_cuMemRelease_v10020 release = nullptr;
  PFN_cuMemMap_v10020 map = nullptr;
  PFN_cuMemUnmap_v10020 unmap = nullptr;
  PFN_cuMemSetAccess_v10020 set_access = nullptr;
  bool ok = false;
};

template <typename F>
bool entry(const char* name, F* out) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &fn, 10020, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return false;
  *out = reinterpret_cast<F>(fn);
  return true;
}

const Driver& driver() {
  static Driver d = [] {
    Driver x;
    x.ok = entry("cuMemGetAllocationGranularity", &x.granularity) && entry("cuMemAddressReserve", &x.reserve) &&
           entry("cuMemAddressFree", &x.addr_free) && entry("cuMemCreate", &x.create) &&
           entry("cuMemRelease", &x.release) && entry("cuMemMap", &x.map) && entry("cuMemUnmap", &x.unmap) &&
           entry("cuMemSetAccess", &x.set_access);
    return x;
  }();
  return d;
}

CUmemAllocationProp page_prop(int device) {
  CUmemAllocationProp prop;
  std::memset(&prop, 0, sizeof(prop));
  prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
  prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
  prop.location.id = device;
  return prop;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

struct pa_vkv {
  int B = 0, L = 0, layers = 0, kv_heads = 0, head_dim = 0, tensors = 0;
  pa_dtype dtype = PA_BF16;
  int64_t row = 0;    // bytes per token of one sub-tensor
  int64_t G = 0;      // page bytes
  int64_t slot_pages = 0;
  int64_t max_pages = 0;
  bool dry = false;
  int device = 0;
  CUdeviceptr base = 0;  // tensors * B * L * row bytes of virtual addresses
  int64_t tensor_bytes = 0;
  std::vector<int> mapped;   // pages mapped per slot (the same in every sub-tensor)
  std::vector<char> active;
  // handles[(t * B + s) * slot_pages + k]: page k of slot s in sub-tensor t
  std::vector<CUmemGenericAllocationHandle> handles;
  std::vector<CUmemGenericAllocationHandle> pool;  // created, unmapped
  int64_t created = 0, map_calls = 0, unmap_calls = 0;
  int64_t step_failures = 0;  // pa_vkv_step calls refused for want of pages
  std::vector<int32_t> held;  // per slot: tokens of the last successful step (0 once the slot is freed)
  int64_t last_map_ns = 0, total_map_ns = 0;
  int32_t* d_slot_tokens = nullptr;
  std::vector<int32_t> h_slot_tokens;

  int64_t pages_for(int64_t n) const {
    if (n <= 0) return 0;
    return cdiv(cdiv(n, 16) * 16 * row, G);
  }
  int64_t in_use() const {
    int64_t s = 0;
    for (int m : mapped) s += m;
    return s * tensors;
  }
  int32_t slot_tokens(int s) const {
    const int64_t t = (int64_t)mapped[s] * G / row;
    return (int32_t)(t < L ? t : L);
  }
  CUdeviceptr page_addr(int t, int s, int64_t k) const {
    return base + (CUdeviceptr)(t * tensor_bytes + (int64_t)s * L * row + k * G);
  }
};

namespace {

// Unmap every page of slot s (device already synchronised by the caller).
int unmap_slot(pa_vkv* v, int s) {
  const Driver& d = driver();
  for (int t = 0; t < v->tensors; ++t)
    for (int64_t k = 0; k < v->mapped[s]; ++k) {
      if (!v->dry) {
        if (d.unmap(v->page_addr(t, s, k), (size_t)v->G) != CUDA_SUCCESS) return PA_ERR_CUDA;
        CUmemGenericAllocationHandle& h = v->handles[((int64_t)t * v->B + s) * v->slot_pages + k];
        v->pool.push_back(h);
        h = 0;
      }
      ++v->unmap_calls;
    }
  v->mapped[s] = 0;
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_vkv_granularity(size_t* out) {
  if (!out) return PA_ERR_INVALID;
  const Driver& d = driver();
  if (!d.ok) return PA_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  CUmemAllocationProp prop = page_prop(dev);
  size_t g = 0;
  if (d.granularity(&g, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM) != CUDA_SUCCESS || g == 0) return PA_ERR_CUDA;
  *out = g;
  return PA_OK;
}

int pa_vkv_create(int num_slots, int max_len, int num_layers, int kv_heads, int head_dim, pa_dtype dtype,
                  size_t page_bytes, int64_t max_pages, int flags, pa_vkv** out) {
  return pa_guarded([&]() -> int {
    if (!out) return PA_ERR_INVALID;
    *out = nullptr;
    if (dtype != PA_FP16 && dtype != PA_BF16) return PA_ERR_DTYPE;
    if (num_slots <= 0 || max_len <= 0 || max_len % 16 != 0 || num_layers <= 0 || kv_heads <= 0 ||
        (head_dim != 64 && head_dim != 128) || max_pages < 0 || (flags & ~PA_VKV_DRY_RUN))
      return PA_ERR_INVALID;
    const bool dry = (flags & PA_VKV_DRY_RUN) != 0;
    if (page_bytes == 0) {
      if (dry) return PA_ERR_INVALID;
      int st = pa_vkv_granularity(&page_bytes);
      if (st != PA_OK) return st;
    }
    const int64_t row = (int64_t)kv_heads * head_dim * 2;
    const int64_t slot_bytes = (int64_t)max_len * row;
    // slots must start on page boundaries, and row coordinates must fit TMA's int32
    if (slot_bytes % (int64_t)page_bytes != 0) return PA_ERR_INVALID;
    if ((int64_t)num_slots * max_len + 16 > INT32_MAX) return PA_ERR_INVALID;
    std::unique_ptr<pa_vkv> v(new pa_vkv);
    v->B = num_slots;
    v->L = max_len;
    v->layers = num_layers;
    v->kv_heads = kv_heads;
    v->head_dim = head_dim;
    v->dtype = dtype;
    v->tensors = 2 * num_layers;
    v->row = row;
    v->G = (int64_t)page_bytes;
    v->slot_pages = slot_bytes / v->G;
    v->max_pages = max_pages;
    v->dry = dry;
    v->tensor_bytes = (int64_t)num_slots * slot_bytes;
    v->mapped.assign(num_slots, 0);
    v->active.assign(num_slots, 0);
    v->held.assign(num_slots, 0);
    v->h_slot_tokens.assign(num_slots, 0);
    if (!dry) {
      const Driver& d = driver();
      if (!d.ok || cudaGetDevice(&v->device) != cudaSuccess) return PA_ERR_CUDA;
      v->handles.assign((size_t)v->tensors * num_slots * v->slot_pages, 0);  // host memory before any CUDA resource
      if (d.reserve(&v->base, (size_t)(v->tensors * v->tensor_bytes), (size_t)v->G, 0, 0) != CUDA_SUCCESS)
        return PA_ERR_CUDA;
      if (cudaMalloc(&v->d_slot_tokens, sizeof(int32_t) * num_slots) != cudaSuccess ||
          cudaMemset(v->d_slot_tokens, 0, sizeof(int32_t) * num_slots) != cudaSuccess) {
        cudaGetLastError();
        d.addr_free(v->base, (size_t)(v->tensors * v->tensor_bytes));
        if (v->d_slot_tokens) cudaFree(v->d_slot_tokens);
        return PA_ERR_CUDA;
      }
    }
    *out = v.release();
    return PA_OK;
  });
}

void pa_vkv_destroy(pa_vkv* v) {
  if (!v) return;
  if (!v->dry) {
    const Driver& d = driver();
    cudaDeviceSynchronize();  // no kernel may still read a page released below
    for (int s = 0; s < v->B; ++s) unmap_slot(v, s);
    for (auto h : v->pool) d.release(h);
    d.addr_free(v->base, (size_t)(v->tensors * v->tensor_bytes));
    cudaFree(v->d_slot_tokens);
  }
  delete v;
}

int pa_vkv_alloc_slot(pa_vkv* v, int* slot_out) {
  if (!v || !slot_out) return PA_ERR_INVALID;
  int best = -1;
  for (int s = 0; s < v->B; ++s)
    if (!v->active[s] && (best < 0 || v->mapped[s] > v->mapped[best])) best = s;
  if (best < 0) return PA_ERR_NO_FREE_BLOCKS;
  v->active[best] = 1;
  *slot_out = best;
  return PA_OK;
}

int pa_vkv_free_slot(pa_vkv* v, int slot) {
  if (!v || slot < 0 || slot >= v->B || !v->active[slot]) return PA_ERR_INVALID;
  v->active[slot] = 0;  // its pages stay mapped for the slot's next request
  v->held[slot] = 0;    // but its tokens no longer count as used
  return PA_OK;
}

int pa_vkv_step(pa_vkv* v, const int32_t* lens, pa_stream stream) {
  return pa_guarded([&]() -> int {
    if (!v || !lens) return PA_ERR_INVALID;
    std::vector<int64_t> need(v->B);
    int64_t extra = 0;
    for (int s = 0; s < v->B; ++s) {
      const int32_t n = lens[s];
      if (n < 0 || n > v->L || (n > 0 && !v->active[s])) return PA_ERR_INVALID;
      need[s] = v->pages_for(n);
      if (need[s] > v->mapped[s]) extra += (need[s] - v->mapped[s]) * v->tensors;
    }
    int64_t short_by = extra - (v->max_pages - v->in_use());
    if (short_by > 0) {
      int64_t reclaimable = 0;
      for (int s = 0; s < v->B; ++s)
        if (!v->active[s]) reclaimable += (int64_t)v->mapped[s] * v->tensors;
      if (reclaimable < short_by) {
        ++v->step_failures;
        return PA_ERR_NO_FREE_BLOCKS;
      }
      std::vector<int> donors;
      for (int s = 0; s < v->B && short_by > 0; ++s) {
        if (v->active[s] || v->mapped[s] == 0) continue;
        short_by -= (int64_t)v->mapped[s] * v->tensors;
        donors.push_back(s);
      }
      if (!v->dry) {
        // every kernel launched so far has finished; the device copy of the
        // bounds drops to zero for the donors (a blocking copy) before their
        // pages go, so no later kernel can reach an unmapped row
        if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
        for (int s : donors) v->h_slot_tokens[s] = 0;
        if (cudaMemcpy(v->d_slot_tokens, v->h_slot_tokens.data(), sizeof(int32_t) * v->B, cudaMemcpyHostToDevice) !=
            cudaSuccess)
          return PA_ERR_CUDA;
      }
      for (int s : donors) {
        const int st = unmap_slot(v, s);
        if (st != PA_OK) return st;
      }
    }
    const auto t0 = std::chrono::steady_clock::now();
    if (!v->dry && extra > 0) {
      const Driver& d = driver();
      // take every page first (pool, then new handles) so that a failed
      // creation leaves the mappings as they were
      std::vector<CUmemGenericAllocationHandle> got;
      got.reserve((size_t)extra);
      v->pool.reserve(v->pool.size() + (size_t)extra);  // the pages go back there if a creation fails
      CUmemAllocationProp prop = page_prop(v->device);
      while ((int64_t)got.size() < extra) {
        if (!v->pool.empty()) {
          got.push_back(v->pool.back());
          v->pool.pop_back();
          continue;
        }
        CUmemGenericAllocationHandle h = 0;
        if (d.create(&h, (size_t)v->G, &prop, 0) != CUDA_SUCCESS) {
          for (auto x : got) v->pool.push_back(x);
          ++v->step_failures;
          return PA_ERR_NO_FREE_BLOCKS;
        }
        ++v->created;
        got.push_back(h);
      }
      CUmemAccessDesc acc;
      std::memset(&acc, 0, sizeof(acc));
      acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
      acc.location.id = v->device;
      acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
      size_t gi = 0;
      for (int s = 0; s < v->B; ++s)
        for (int64_t k = v->mapped[s]; k < need[s]; ++k)
          for (int t = 0; t < v->tensors; ++t) {
            const CUdeviceptr a = v->page_addr(t, s, k);
            const CUmemGenericAllocationHandle h = got[gi++];
            if (d.map(a, (size_t)v->G, 0, h, 0) != CUDA_SUCCESS ||
                d.set_access(a, (size_t)v->G, &acc, 1) != CUDA_SUCCESS)
              return PA_ERR_CUDA;
            v->handles[((int64_t)t * v->B + s) * v->slot_pages + k] = h;
          }
    }
    for (int s = 0; s < v->B; ++s)
      if (need[s] > v->mapped[s]) {
        v->map_calls += (need[s] - v->mapped[s]) * v->tensors;
        v->mapped[s] = (int)need[s];
      }
    v->last_map_ns =
        std::chrono::duration_cast<std::chrono::nanoseconds>(std::chrono::steady_clock::now() - t0).count();
    for (int s = 0; s < v->B; ++s) v->held[s] = lens[s];  // nonzero only on active slots (checked above)
    v->total_map_ns += v->last_map_ns;
    bool changed = false;
    for (int s = 0; s < v->B; ++s) {
      const int32_t t = v->slot_tokens(s);
      changed |= t != v->h_slot_tokens[s];
      v->h_slot_tokens[s] = t;
    }
    if (!v->dry && changed &&
        cudaMemcpyAsync(v->d_slot_tokens, v->h_slot_tokens.data(), sizeof(int32_t) * v->B, cudaMemcpyHostToDevice,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
      return PA_ERR_CUDA;
    return PA_OK;
  });
}

int pa_vkv_tensor(const pa_vkv* v, int layer, int is_v, void** out) {
  if (!v || !out || layer < 0 || layer >= v->layers) return PA_ERR_INVALID;
  *out = v->dry ? nullptr : reinterpret_cast<void*>(v->base + (CUdeviceptr)((2 * layer + (is_v ? 1 : 0)) *
                                                                            v->tensor_bytes));
  return PA_OK;
}

int pa_vkv_slot_tokens(const pa_vkv* v, int32_t* host_out, const int32_t** device_out) {
  if (!v) return PA_ERR_INVALID;
  if (host_out)
    for (int s = 0; s < v->B; ++s) host_out[s] = v->slot_tokens(s);
  if (device_out) *device_out = v->d_slot_tokens;
  return PA_OK;
}

int pa_vkv_slot_pages(const pa_vkv* v, int slot) {
  if (!v || slot < 0 || slot >= v->B) return PA_ERR_INVALID;
  return v->mapped[slot];
}

int pa_vkv_get_stats(const pa_vkv* v, pa_vkv_stats* out) {
  if (!v || !out) return PA_ERR_INVALID;
  pa_vkv_stats st{};
  st.page_bytes = v->G;
  st.slot_pages = v->slot_pages;
  st.pages_mapped = v->in_use();
  st.pages_pooled = (int64_t)v->pool.size();
  st.pages_created = v->created;
  st.map_calls = v->map_calls;
  st.unmap_calls = v->unmap_calls;
  st.bytes_reserved = v->tensors * v->tensor_bytes;
  st.bytes_committed = v->in_use() * v->G;
  st.last_step_map_ns = v->last_map_ns;
  st.total_map_ns = v->total_map_ns;
  int64_t act = 0;
  for (char a : v->active) act += a ? 1 : 0;
  st.active_slots = act;
  st.step_failures = v->step_failures;
  int64_t tokens = 0;
  for (int s = 0; s < v->B; ++s) tokens += v->active[s] ? v->held[s] : 0;
  st.bytes_used = tokens * v->row * v->tensors;
  *out = st;
  return PA_OK;
}

int pa_vkv_decode(const pa_vkv* v, int layer, const void* q, const int32_t* slot_ids, const int32_t* context_lens,
                  int num_seqs, int q_heads, float scale, int split_tokens, void* workspace, size_t workspace_bytes,
                  void* out, pa_stream stream) {
  if (!v || v->dry || layer < 0 || layer >= v->layers) return PA_ERR_INVALID;
  void* k = nullptr;
  void* vv = nullptr;
  pa_vkv_tensor(v, layer, 0, &k);
  pa_vkv_tensor(v, layer, 1, &vv);
  return pa_decode_contiguous(q, k, vv, v->B, v->L, slot_ids, v->d_slot_tokens, context_lens, num_seqs, q_heads,
                              v->kv_heads, v->head_dim, scale, split_tokens, workspace, workspace_bytes, out,
                              v->dtype, stream);
}

int pa_vkv_reshape_and_cache(const pa_vkv* v, int layer, const void* k, const void* vv, const int32_t* slot_ids,
                             const int32_t* positions, int num_tokens, pa_stream stream) {
  if (!v || v->dry || layer < 0 || layer >= v->layers) return PA_ERR_INVALID;
  void* kc = nullptr;
  void* vc = nullptr;
  pa_vkv_tensor(v, layer, 0, &kc);
  pa_vkv_tensor(v, layer, 1, &vc);
  return pa_reshape_and_cache_slots(k, vv, slot_ids, positions, num_tokens, kc, vc, v->B, v->L, v->d_slot_tokens,
                                    v->kv_heads, v->head_dim, v->dtype, stream);
}

}  // extern "C"
