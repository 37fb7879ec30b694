// KV-cache writes for sm_103a: reshape_and_cache (scatter new tokens into
// their slots) and copy_blocks (the device half of Copy-on-Write).
//
// Both are pure data movement bound by HBM bandwidth.  With the cache layout
// [num_blocks][block_size][kv_heads][head_dim], one token's K for all KV heads
// is one contiguous row of kv_heads*head_dim elements in the source and in its
// slot, so reshape_and_cache is a row gather/scatter of 16-byte vectors, and a
// whole physical block is one contiguous span that copy_blocks moves with
// 16-byte vectors.  Both copy bits, never values, so they are bit-exact.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Grid-stride over (token, 16-byte vector of the token's row).
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             const int32_t* __restrict__ slots, uint4* __restrict__ k_cache,
                             uint4* __restrict__ v_cache, int num_tokens, int row_vecs, int64_t num_slots,
                             int* err) {
  griddep_wait();  // k/v/slots and the cache may come from the kernel before this one
  griddep_launch_dependents();
  const int64_t total = (int64_t)num_tokens * row_vecs;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = i / row_vecs;
    const int64_t j = i - tok * row_vecs;
    const int32_t s = __ldg(slots + tok);
    if (s < 0) continue;  // padding token
    if (s >= num_slots) {
      if (j == 0) record_error(err, PA_DEVERR_SLOT);
      continue;
    }
    const uint4 kv = ld_stream(k + i);
    const uint4 vv = ld_stream(v + i);
    k_cache[(int64_t)s * row_vecs + j] = kv;
    v_cache[(int64_t)s * row_vecs + j] = vv;
  }
}

// reshape_and_cache into a contiguous [num_slots][contig_len] cache: token i
// goes to row slot_ids[i]*contig_len + positions[i].  A negative slot marks
// padding; a position outside [0, bound) - bound = slot_tokens[slot], the rows
// of the slot backed by memory, or contig_len - records PA_DEVERR_SLOT and the
// token is skipped, so no write ever reaches an unmapped page.
__global__ void __launch_bounds__(256)
    reshape_and_cache_slots_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                   const int32_t* __restrict__ slot_ids, const int32_t* __restrict__ positions,
                                   uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, int num_tokens,
                                   int row_vecs, int num_slots, int contig_len,
                                   const int32_t* __restrict__ slot_tokens, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  const int64_t total = (int64_t)num_tokens * row_vecs;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = i / row_vecs;
    const int64_t j = i - tok * row_vecs;
    const int32_t s = __ldg(slot_ids + tok);
    if (s < 0) continue;  // padding token
    const int32_t pos = __ldg(positions + tok);
    const int bound = s < num_slots ? (slot_tokens ? min(__ldg(slot_tokens + s), contig_len) : contig_len) : 0;
    if (s >= num_slots || pos < 0 || pos >= bound) {
      if (j == 0) record_error(err, PA_DEVERR_SLOT);
      continue;
    }
    const int64_t row = (int64_t)s * contig_len + pos;
    const uint4 kv = ld_stream(k + i);
    const uint4 vv = ld_stream(v + i);
    k_cache[row * row_vecs + j] = kv;
    v_cache[row * row_vecs + j] = vv;
  }
}

// blockIdx.y strides over pairs; x threads over the block's 16-byte vectors.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ pairs,
                       int num_pairs, int64_t block_vecs, int num_blocks, int* err) {
  griddep_wait();
  griddep_launch_dependents();
  for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
    const int src = __ldg(pairs + 2 * pi), dst = __ldg(pairs + 2 * pi + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, PA_DEVERR_BLOCK_ID);
      continue;
    }
    const uint4* ks = k_cache + (int64_t)src * block_vecs;
    const uint4* vs = v_cache + (int64_t)src * block_vecs;
    uint4* kd = k_cache + (int64_t)dst * block_vecs;
    uint4* vd = v_cache + (int64_t)dst * block_vecs;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < block_vecs;
         i += (int64_t)gridDim.x * blockDim.x) {
      const uint4 a = ks[i];
      const uint4 b = vs[i];
      kd[i] = a;
      vd[i] = b;
    }
  }
}

// Swap step of preemption: block dst of one pool becomes a copy of block src
// of another; either pool may be page-locked host memory read or written
// directly by the kernel (over NVLink-C2C on Grace-Blackwell).  Four 16-byte
// vectors per thread are loaded before any is stored, to keep enough
// requests in flight across the host link.
__global__ void __launch_bounds__(256)
    swap_blocks_kernel(const uint4* __restrict__ sk, const uint4* __restrict__ sv, uint4* __restrict__ dk,
                       uint4* __restrict__ dv, const int32_t* __restrict__ pairs, int num_pairs, int64_t block_vecs,
                       int num_src, int num_dst, int* err) {
  constexpr int U = 4;
  griddep_wait();
  griddep_launch_dependents();
  for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
    const int src = pairs[2 * pi], dst = pairs[2 * pi + 1];
    if (src < 0 || src >= num_src || dst < 0 || dst >= num_dst) {
      if (threadIdx.x == 0 && blockIdx.x == 0) record_error(err, PA_DEVERR_BLOCK_ID);
      continue;
    }
    const uint4* ks = sk + (int64_t)src * block_vecs;
    const uint4* vs = sv + (int64_t)src * block_vecs;
    uint4* kd = dk + (int64_t)dst * block_vecs;
    uint4* vd = dv + (int64_t)dst * block_vecs;
    for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x * U + threadIdx.x; i0 < block_vecs;
         i0 += (int64_t)gridDim.x * blockDim.x * U) {
      uint4 a[U], b[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + (int64_t)u * blockDim.x;
        if (i < block_vecs) {
          a[u] = ks[i];
          b[u] = vs[i];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + (int64_t)u * blockDim.x;
        if (i < block_vecs) {
          kd[i] = a[u];
          vd[i] = b[u];
        }
      }
    }
  }
}

// Self-test of the bounded wait every kernel of the library uses: one
// thread waits on an mbarrier phase that no arrival completes.  The wait
// gives up after limit_ns, records PA_DEVERR_TIMEOUT and the kernel returns
// normally, so the context stays usable.
__global__ void __launch_bounds__(32) wait_timeout_kernel(int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  if (!mbar_wait_for(smem_u32(&bar), 0, limit_ns)) record_error(err, PA_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout(int* err, uint64_t limit_ns, cudaStream_t stream) {
  return launch_pdl(wait_timeout_kernel, dim3(1), dim3(32), 0, stream, err, limit_ns);
}

cudaError_t launch_swap_blocks(const void* src_k, const void* src_v, void* dst_k, void* dst_v, const int32_t* pairs,
                               int num_pairs, int num_src, int num_dst, int64_t block_bytes, int* err,
                               cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t block_vecs = block_bytes / 16;
  int64_t bx = (block_vecs + 1023) / 1024;
  if (bx > 8) bx = 8;
  const int by = num_pairs < 65535 ? num_pairs : 65535;
  return launch_pdl(swap_blocks_kernel, dim3((unsigned)bx, by), dim3(256), 0, stream,
                    static_cast<const uint4*>(src_k), static_cast<const uint4*>(src_v), static_cast<uint4*>(dst_k),
                    static_cast<uint4*>(dst_v), pairs, num_pairs, block_vecs, num_src, num_dst, err);
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, const int32_t* slots, int num_tokens,
                                     void* k_cache, void* v_cache, int64_t num_slots, int row_bytes, int* err,
                                     cudaStream_t stream) {
  const int row_vecs = row_bytes / 16;
  const int64_t total = (int64_t)num_tokens * row_vecs;
  if (total == 0) return cudaSuccess;
  return launch_pdl(reshape_and_cache_kernel, dim3(copy_grid(total)), dim3(256), 0, stream,
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, static_cast<uint4*>(k_cache),
                    static_cast<uint4*>(v_cache), num_tokens, row_vecs, num_slots, err);
}

cudaError_t launch_reshape_and_cache_slots(const void* k, const void* v, const int32_t* slot_ids,
                                           const int32_t* positions, int num_tokens, void* k_cache, void* v_cache,
                                           int num_slots, int contig_len, const int32_t* slot_tokens, int row_bytes,
                                           int* err, cudaStream_t stream) {
  const int row_vecs = row_bytes / 16;
  const int64_t total = (int64_t)num_tokens * row_vecs;
  if (total == 0) return cudaSuccess;
  return launch_pdl(reshape_and_cache_slots_kernel, dim3(copy_grid(total)), dim3(256), 0, stream,
                    static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_ids, positions,
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_tokens, row_vecs, num_slots,
                    contig_len, slot_tokens, err);
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs, int num_blocks,
                               int64_t block_bytes, int* err, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int64_t block_vecs = block_bytes / 16;
  int64_t bx = (block_vecs + 255) / 256;
  if (bx > 8) bx = 8;
  const int by = num_pairs < 65535 ? num_pairs : 65535;
  return launch_pdl(copy_blocks_kernel, dim3((unsigned)bx, by), dim3(256), 0, stream, static_cast<uint4*>(k_cache),
                    static_cast<uint4*>(v_cache), pairs, num_pairs, block_vecs, num_blocks, err);
}

}  // namespace pa
