// Chunked-prefill attention over a paged KV cache for sm_103a.
//
// A CTA owns 64 query rows of one (request, KV head); a row is one (query,
// head-of-the-GQA-group) pair, rows ordered query-major, so the whole group
// shares every K/V tile.  Query i of a chunk that starts at absolute position
// p0 sees keys 0 .. p0+i.  The CTA walks keys in tiles of 64 tokens up to the
// last key any of its rows can see.
//
// Warp roles: one producer warp gathers each 64-token K/V tile from its
// physical blocks with TMA (one box per block per 64-element half of
// head_dim) into a ring of STAGES stages; four consumer warps (16 rows each)
// compute S = Q K^T and O += P V with mma.m16n8k16 (fp32 accumulate) and an
// online softmax per row.  Full/empty mbarriers order the ring; every wait is
// bounded and records PA_DEVERR_TIMEOUT instead of hanging.
#include <float.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kPrefillConsumers = 4;
constexpr int kPrefillStages = 3;
constexpr int kKeyTile = 64;
constexpr int kTableChunk = 512;  // block-table entries staged in shared memory at a time

__device__ __forceinline__ uint8_t* align1024p(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, int BSUB, typename T, int CW, int STAGES>
struct PrefillSmem {
  using Tile = KvTile<D, BSUB, kKeyTile>;
  static constexpr int STAGE_BYTES = 2 * Tile::BYTES;
  static constexpr int FULL_OFF = STAGES * STAGE_BYTES;
  static constexpr int EMPTY_OFF = FULL_OFF + STAGES * 8;
  static constexpr int ZERO_OFF = EMPTY_OFF + STAGES * 8;  // consumers' "stale rows zeroed" barrier
  static constexpr int TAB_OFF = ZERO_OFF + 8;
  static constexpr int BYTES = TAB_OFF + kTableChunk * 4 + 1024;
};

template <int D, int BSUB, typename T, int CW, int STAGES>
__global__ void __launch_bounds__((CW + 1) * 32)
    chunked_prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           const PrefillParams p) {
  using L = PrefillSmem<D, BSUB, T, CW, STAGES>;
  using Tile = typename L::Tile;
  constexpr int KSTEPS = D / 16;
  constexpr int DT8 = D / 8;  // 8-wide n-tiles of the output
  constexpr int ROWS = CW * 16;
  constexpr int LOADS = Tile::NH * 2;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024p(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::FULL_OFF);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L::EMPTY_OFF);
  uint64_t* zbar = reinterpret_cast<uint64_t*>(smem + L::ZERO_OFF);
  int32_t* tab = reinterpret_cast<int32_t*>(smem + L::TAB_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.z, h = blockIdx.y;
  const int row0 = blockIdx.x * ROWS;
  const int G = p.group;

  // request geometry (uniform across the CTA)
  const int qs = __ldg(p.q_start + r), qe = __ldg(p.q_start + r + 1);
  const int chunk = qe - qs;
  const int ctx = __ldg(p.lens + r);
  const int p0 = ctx - chunk;
  if (qs < 0 || qe < qs || qe > p.total_q || chunk > p.max_q_len || p0 < 0 || ctx > p.maxblk * p.block_size) {
    griddep_wait();
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) record_error(p.err, PA_DEVERR_QUERY_RANGE);
    return;
  }
  const int rows = chunk * G;
  if (row0 >= rows) {
    griddep_wait();
    return;
  }
  const int last_row = min(row0 + ROWS, rows) - 1;
  const int kmax = p0 + last_row / G + 1;  // keys [0, kmax) are visible to some row
  const int ntiles = (kmax + kKeyTile - 1) / kKeyTile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), CW);
    }
    mbar_init(smem_u32(zbar), CW);
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == CW) {
    // ------------------------------------------------------------ producer
    const int32_t* trow = p.tables + (size_t)r * p.maxblk;
    const int need_blocks = (kmax + p.block_size - 1) / p.block_size;
    int chunk_base = -kTableChunk;
    const uint64_t pol = policy_evict_last();  // K/V tiles are re-read by the other row tiles
    griddep_wait();  // the cache (this step's reshape_and_cache) comes from the kernel before
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % STAGES;
      if (j >= STAGES && !mbar_wait(smem_u32(&empty[s]), ((j / STAGES) - 1) & 1)) {
        if (lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
        return;
      }
      const int ts = j * kKeyTile;
      const int nvalid = min(kKeyTile, kmax - ts);
      const int nsub = (nvalid + BSUB - 1) / BSUB;
      const int lb_first = ts / p.block_size;
      const int lb_last = (ts + nvalid - 1) / p.block_size;
      if (lb_last >= chunk_base + kTableChunk) {
        chunk_base = lb_first;
        __syncwarp();
        for (int i = lane; i < kTableChunk && chunk_base + i < need_blocks; i += 32) {
          int b = __ldg(trow + chunk_base + i);
          if (b < 0 || b >= p.num_blocks) {
            record_error(p.err, PA_DEVERR_BLOCK_ID);
            b = p.num_blocks;  // rows past the tensor map: TMA zero-fills
          }
          tab[i] = b;
        }
        __syncwarp();
      }
      const uint32_t bar = smem_u32(&full[s]);
      const uint32_t kdst = smem_u32(smem + s * L::STAGE_BYTES);
      if (lane == 0) mbar_arrive_expect_tx(bar, nsub * LOADS * Tile::BOX_BYTES);
      __syncwarp();
      for (int i = lane; i < nsub * LOADS; i += 32) {
        const int sub = i / LOADS, rem = i % LOADS;
        const int isv = rem / Tile::NH, hf = rem % Tile::NH;
        const int tok = ts + sub * BSUB;
        const int b = tab[tok / p.block_size - chunk_base];
        const int row = b * p.block_size + tok % p.block_size;
        tma_load_4d_hint(kdst + isv * Tile::BYTES + Tile::box(hf, sub), isv ? &vmap : &kmap, bar, 0, hf, h, row,
                         pol);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ra = row0 + warp * 16 + (lane >> 2);
  const int rb = ra + 8;
  const int qia = ra / G, qib = rb / G;
  const int lima = ra < rows ? p0 + qia : -1;  // last visible key of the row
  const int limb = rb < rows ? p0 + qib : -1;

  // Q A-fragments: rows ra/rb, d = 16ks + 2(lane%4) (+8)
  uint32_t qa[KSTEPS][4];
  {
    const T* q = reinterpret_cast<const T*>(p.q);
    const T* qra = q + ((size_t)(qs + qia) * p.q_heads + h * G + ra % G) * D;
    const T* qrb = q + ((size_t)(qs + qib) * p.q_heads + h * G + rb % G) * D;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      const int d = ks * 16 + 2 * (lane & 3);
      qa[ks][0] = ra < rows ? __ldg(reinterpret_cast<const uint32_t*>(qra + d)) : 0u;
      qa[ks][1] = rb < rows ? __ldg(reinterpret_cast<const uint32_t*>(qrb + d)) : 0u;
      qa[ks][2] = ra < rows ? __ldg(reinterpret_cast<const uint32_t*>(qra + d + 8)) : 0u;
      qa[ks][3] = rb < rows ? __ldg(reinterpret_cast<const uint32_t*>(qrb + d + 8)) : 0u;
    }
  }

  griddep_wait();  // before writing `out` (and reading tiles of this step's cache)
  float acc[DT8][4];
#pragma unroll
  for (int i = 0; i < DT8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
  const float sl2 = p.scale_log2;
  const int mi = lane >> 3, rr = lane & 7;

  for (int j = 0; j < ntiles; ++j) {
    const int s = j % STAGES;
    if (!mbar_wait(smem_u32(&full[s]), (j / STAGES) & 1)) {
      if (lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
      return;
    }
    const int ts = j * kKeyTile;
    const int nvalid = min(kKeyTile, kmax - ts);
    uint8_t* kt = smem + s * L::STAGE_BYTES;
    uint8_t* vt = kt + Tile::BYTES;
    if (nvalid < kKeyTile) {
      // Only the last tile is partial.  Keys past the last visible one: the
      // consumers zero their V rows (a share each), then meet on zbar, so
      // that p = 0 never multiplies stale NaN/Inf.
      const int nz = (kKeyTile - nvalid) * Tile::NH * 8;
      for (int i = warp * 32 + lane; i < nz; i += CW * 32) {
        const int row = nvalid + i / (Tile::NH * 8);
        const int rem = i % (Tile::NH * 8);
        *reinterpret_cast<uint4*>(vt + Tile::line(rem >> 3, row) + ((rem & 7) << 4)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(zbar));
      if (!mbar_wait(smem_u32(zbar), 0)) {
        if (lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
        return;
      }
    }
    const uint32_t kts = smem_u32(kt), vts = smem_u32(vt);

    // S = Q K^T over 64 keys: 8 n-tiles of 8 keys
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; nt += 2) {
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        uint32_t b[4];
        ldmatrix_x4(b, kts + Tile::offset(8 * (nt + (mi >> 1)) + rr, 2 * ks + (mi & 1)));
        mma_16816<T>(sc[nt], qa[ks], b[0], b[1]);
        mma_16816<T>(sc[nt + 1], qa[ks], b[2], b[3]);
      }
    }

    // causal mask + online softmax (rows ra: elements 0,1; rb: elements 2,3)
    float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int key = ts + nt * 8 + 2 * (lane & 3);
      sc[nt][0] = key <= lima ? sc[nt][0] * sl2 : -INFINITY;
      sc[nt][1] = key + 1 <= lima ? sc[nt][1] * sl2 : -INFINITY;
      sc[nt][2] = key <= limb ? sc[nt][2] * sl2 : -INFINITY;
      sc[nt][3] = key + 1 <= limb ? sc[nt][3] * sl2 : -INFINITY;
      mxa = fmaxf(mxa, fmaxf(sc[nt][0], sc[nt][1]));
      mxb = fmaxf(mxb, fmaxf(sc[nt][2], sc[nt][3]));
    }
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
    const float mna = fmaxf(ma, mxa), mnb = fmaxf(mb, mxb);
    const float ua = mna == -INFINITY ? 0.f : mna;  // fully masked so far: keep everything at 0
    const float ub = mnb == -INFINITY ? 0.f : mnb;
    const float ala = exp2f(ma - ua), alb = exp2f(mb - ub);
    ma = mna;
    mb = mnb;
    // P rounded to the input type for the P.V MMA; the denominators sum the
    // same rounded values, so each output row is an exact convex combination
    float suma = 0.f, sumb = 0.f;
    uint32_t pka[8], pkb[8];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      pka[nt] = Elem<T>::pack(exp2f(sc[nt][0] - ua), exp2f(sc[nt][1] - ua));
      pkb[nt] = Elem<T>::pack(exp2f(sc[nt][2] - ub), exp2f(sc[nt][3] - ub));
      suma += Elem<T>::sum2(pka[nt]);
      sumb += Elem<T>::sum2(pkb[nt]);
    }
    la = la * ala + suma;
    lb = lb * alb + sumb;
#pragma unroll
    for (int i = 0; i < DT8; ++i) {
      acc[i][0] *= ala;
      acc[i][1] *= ala;
      acc[i][2] *= alb;
      acc[i][3] *= alb;
    }

    // O += P V: 4 k-steps of 16 keys; P from the S accumulators in registers
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint32_t pa[4] = {pka[2 * kk], pkb[2 * kk], pka[2 * kk + 1], pkb[2 * kk + 1]};
#pragma unroll
      for (int nd = 0; nd < DT8; nd += 2) {
        uint32_t b[4];
        ldmatrix_x4_trans(b, vts + Tile::offset(16 * kk + rr + 8 * (mi & 1), nd + (mi >> 1)));
        mma_16816<T>(acc[nd], pa, b[0], b[1]);
        mma_16816<T>(acc[nd + 1], pa, b[2], b[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
  }

  la += __shfl_xor_sync(0xffffffffu, la, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  lb += __shfl_xor_sync(0xffffffffu, lb, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  T* out = reinterpret_cast<T*>(p.out);
  if (ra < rows) {
    const float inv = la > 0.f ? 1.f / la : 0.f;
    T* o = out + ((size_t)(qs + qia) * p.q_heads + h * G + ra % G) * D + 2 * (lane & 3);
#pragma unroll
    for (int nd = 0; nd < DT8; ++nd)
      *reinterpret_cast<uint32_t*>(o + nd * 8) = Elem<T>::pack(acc[nd][0] * inv, acc[nd][1] * inv);
  }
  if (rb < rows) {
    const float inv = lb > 0.f ? 1.f / lb : 0.f;
    T* o = out + ((size_t)(qs + qib) * p.q_heads + h * G + rb % G) * D + 2 * (lane & 3);
#pragma unroll
    for (int nd = 0; nd < DT8; ++nd)
      *reinterpret_cast<uint32_t*>(o + nd * 8) = Elem<T>::pack(acc[nd][2] * inv, acc[nd][3] * inv);
  }
}

template <int D, int BSUB, typename T>
cudaError_t launch_prefill_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                             cudaStream_t stream) {
  constexpr int CW = kPrefillConsumers, S = kPrefillStages;
  using L = PrefillSmem<D, BSUB, T, CW, S>;
  auto kern = chunked_prefill_kernel<D, BSUB, T, CW, S>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int row_tiles = (p.max_q_len * p.group + CW * 16 - 1) / (CW * 16);
  dim3 grid(row_tiles, p.kv_heads, p.num_reqs);
  return launch_pdl(kern, grid, dim3((CW + 1) * 32), L::BYTES, stream, kmap, vmap, p);
}

template <int D, typename T>
cudaError_t launch_prefill_bs(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p, int bsub,
                              cudaStream_t stream) {
  switch (bsub) {
    case 4: return launch_prefill_t<D, 4, T>(kmap, vmap, p, stream);
    case 8: return launch_prefill_t<D, 8, T>(kmap, vmap, p, stream);
    case 16: return launch_prefill_t<D, 16, T>(kmap, vmap, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_chunked_prefill(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                                   int head_dim, int bsub, pa_dtype dt, cudaStream_t stream) {
  if (head_dim == 128) {
    return dt == PA_BF16 ? launch_prefill_bs<128, __nv_bfloat16>(kmap, vmap, p, bsub, stream)
                         : launch_prefill_bs<128, __half>(kmap, vmap, p, bsub, stream);
  }
  if (head_dim == 64) {
    return dt == PA_BF16 ? launch_prefill_bs<64, __nv_bfloat16>(kmap, vmap, p, bsub, stream)
                         : launch_prefill_bs<64, __half>(kmap, vmap, p, bsub, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
