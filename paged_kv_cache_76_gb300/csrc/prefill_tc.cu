// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05 with
// tensor memory), sm_103a, for block_size >= 8.
//
// A CTA owns 128 rows of one (request, KV head); a row is one (query,
// head-of-the-GQA-group) pair, rows ordered query-major, so the whole group
// shares every K/V tile.  Query i of a chunk that starts at absolute position
// p0 sees keys 0 .. p0+i.  Keys are walked in tiles of 128.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: gathers each 128-key K and V tile from its
//               physical blocks (one 128-byte-swizzled box per block and
//               64-element half of head_dim) into a 2-stage ring.
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               S buffers (M=128, N=128, K=16 per instruction), so the tensor
//               core computes S_{j+1} while the softmax works on S_j; then
//               O += P_j V_j, accumulated in TMEM across all tiles.
//   warps 2..5  softmax: thread = TMEM lane = tile row.  Loads its whole S row
//               from TMEM (four loads, one wait), applies the causal limit,
//               and writes P = 2^(s*scale*log2e - m) as bf16/fp16 into the K
//               slot of the stage (K_j is dead once S_j is done).  m is a
//               running maximum that is only raised when the row's maximum
//               exceeds it by more than 2^8 (then O in TMEM and the row sum
//               are rescaled); the final O / sum uses the same m, so this is
//               exact and O is rarely touched by the softmax warps.
// Shared-memory operands use the canonical 128-byte-swizzled layouts: Q, K and
// P K-major (8-row atoms, 1024-byte stride), V MN-major (head_dim contiguous;
// its two 64-element halves 16 KB apart).  All mbarrier waits are bounded.
#include <float.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kTcRows = 128;   // M: rows per CTA
constexpr int kTcKeys = 128;   // keys per stage (N of S, K of P.V)
constexpr int kTcTableChunk = 512;
constexpr int kTcStages = 2;
constexpr int kTcThreads = 192;
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ uint8_t* align1024t(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, int BSUB>
struct TcSmem {
  using Tile = KvTile<D, BSUB, kTcKeys>;  // K or V: D/64 halves x 128 rows x 128 B, rows contiguous
  static constexpr int NH = D / 64;
  static constexpr int QHALF = kTcRows * 128;
  static constexpr int Q_OFF = 0;
  static constexpr int STAGE_OFF = Q_OFF + NH * QHALF;
  // a stage is [K, later overwritten by P | V]; P is 128 rows x 128 keys
  // (two 64-key halves of 16 KB), which is more than K when head_dim is 64
  static constexpr int P_HALF = kTcRows * 128;
  static constexpr int KP_BYTES = Tile::BYTES > 2 * P_HALF ? Tile::BYTES : 2 * P_HALF;
  static constexpr int STAGE_BYTES = KP_BYTES + Tile::BYTES;
  static constexpr int BAR_OFF = STAGE_OFF + kTcStages * STAGE_BYTES;
  static constexpr int NBARS = 18;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int TAB_OFF = SLOT_OFF + 16;
  static constexpr int BYTES = TAB_OFF + kTcTableChunk * 4 + 1024;
  static_assert(BSUB * 128 >= 1024, "tcgen05 path needs blocks of at least 8 tokens");
};

// barrier indices
enum : int {
  B_KFULL = 0, B_VFULL = 3, B_KVEMPTY = 6, B_SFULL = 9, B_SEMPTY = 11, B_PFULL = 13, B_OFULL = 15, B_QFULL = 16,
  B_MMADONE = 17
};

template <int D, int BSUB, typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
    chunked_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                              const PrefillParams p) {
  using L = TcSmem<D, BSUB>;
  using Tile = typename L::Tile;
  constexpr int NH = L::NH;
  constexpr int KSTEPS = D / 16;        // S = Q K^T, K dimension = head_dim
  constexpr int PSTEPS = kTcKeys / 16;  // O = P V,   K dimension = keys
  constexpr int LOADS = NH * 2;
  constexpr uint32_t S_COL = 0;              // S buffers: columns [0,128) and [128,256)
  constexpr uint32_t O_COL = 2 * kTcKeys;    // O accumulator: columns [256, 256+D)
  constexpr uint32_t IDESC_S = idesc_f16<T>(kTcRows, kTcKeys, false);
  constexpr uint32_t IDESC_O = idesc_f16<T>(kTcRows, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024t(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::SLOT_OFF);
  int32_t* tab = reinterpret_cast<int32_t*>(smem + L::TAB_OFF);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int row0 = blockIdx.x * kTcRows;
  const int G = p.group;

  // geometry (uniform across the CTA); only immutable inputs are read.
  // Causal mode: request r = blockIdx.z, its chunk starts at absolute position
  // p0, row (query i, head g) sees keys 0 .. p0+i.  Shared-prefix mode: one
  // virtual request of total_q queries (the decode batch), keys
  // [k0, kend) = split blockIdx.z of the prefix, all visible to every row.
  int r, qs, chunk, p0, k0, kend;
  if (p.causal) {
    r = blockIdx.z;
    qs = __ldg(p.q_start + r);
    const int qe = __ldg(p.q_start + r + 1);
    chunk = qe - qs;
    const int ctx = __ldg(p.lens + r);
    p0 = ctx - chunk;
    if (qs < 0 || qe < qs || qe > p.total_q || chunk > p.max_q_len || p0 < 0 || ctx > p.maxblk * p.block_size) {
      griddep_wait();
      if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) record_error(p.err, PA_DEVERR_QUERY_RANGE);
      return;
    }
    k0 = 0;
    const int last_row = min(row0 + kTcRows, chunk * G) - 1;
    kend = p0 + last_row / G + 1;  // keys [0, kend) are visible to some row
  } else {
    r = 0;
    qs = 0;
    chunk = p.total_q;
    p0 = 0;
    k0 = blockIdx.z * p.key_split;
    kend = min(k0 + p.key_split, p.prefix_len);
  }
  const int rows = chunk * G;
  if (row0 >= rows || k0 >= kend) {
    griddep_wait();
    return;
  }
  const int ntiles = (kend - k0 + kTcKeys - 1) / kTcKeys;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_KVEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SEMPTY + i), 4);
      mbar_init(bar(B_PFULL + i), 4);
    }
    mbar_init(bar(B_OFULL), 1);
    mbar_init(bar(B_QFULL), 4);
    mbar_init(bar(B_MMADONE), 1);
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    const int32_t* trow = p.tables + (size_t)r * p.maxblk;
    const int need_blocks = (kend + p.block_size - 1) / p.block_size;
    const uint64_t pol = policy_evict_last();  // K/V tiles are re-read by the other row tiles
    int chunk_base = -kTcTableChunk;
    int issued = 0;
    bool failed = false;
    griddep_wait();  // the cache (this step's reshape_and_cache) comes from the kernel before
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kTcStages;
      if (j >= kTcStages && !mbar_wait(bar(B_KVEMPTY + s), ((j / kTcStages) - 1) & 1)) {
        failed = true;
        break;
      }
      const int ts = k0 + j * kTcKeys;
      const int nvalid = min(kTcKeys, kend - ts);
      const int nsub = (nvalid + BSUB - 1) / BSUB;
      const int lb_first = ts / p.block_size;
      const int lb_last = (ts + nvalid - 1) / p.block_size;
      if (lb_last >= chunk_base + kTcTableChunk) {
        chunk_base = lb_first;
        __syncwarp();
        for (int i = lane; i < kTcTableChunk && chunk_base + i < need_blocks; i += 32) {
          int b = __ldg(trow + chunk_base + i);
          if (b < 0 || b >= p.num_blocks) {
            record_error(p.err, PA_DEVERR_BLOCK_ID);
            b = p.num_blocks;  // rows past the tensor map: TMA zero-fills
          }
          tab[i] = b;
        }
        __syncwarp();
      }
      const uint32_t kdst = smem_u32(smem + L::STAGE_OFF + s * L::STAGE_BYTES);
      const uint32_t vdst = kdst + L::KP_BYTES;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(B_KFULL + s), nsub * NH * Tile::BOX_BYTES);
        mbar_arrive_expect_tx(bar(B_VFULL + s), nsub * NH * Tile::BOX_BYTES);
      }
      __syncwarp();
      for (int i = lane; i < nsub * LOADS; i += 32) {
        const int sub = i / LOADS, rem = i % LOADS;
        const int isv = rem / NH, hf = rem % NH;
        const int tok = ts + sub * BSUB;
        const int b = tab[tok / p.block_size - chunk_base];
        const int row = b * p.block_size + tok % p.block_size;
        tma_load_4d_hint((isv ? vdst : kdst) + Tile::box(hf, sub), isv ? &vmap : &kmap,
                         bar((isv ? B_VFULL : B_KFULL) + s), 0, hf, h, row, pol);
      }
      issued = j + 1;
    }
    if (failed && lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
    // loads still in flight land before the CTA can exit (bounded)
    for (int j = issued - kTcStages < 0 ? 0 : issued - kTcStages; j < issued; ++j) {
      mbar_wait(bar(B_KFULL + j % kTcStages), (j / kTcStages) & 1);
      mbar_wait(bar(B_VFULL + j % kTcStages), (j / kTcStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(bar(B_QFULL), 0);
      const uint32_t qa = smem_u32(smem + L::Q_OFF);
      auto issue_pv = [&](int i) -> bool {
        const int b = i & 1, s = i % kTcStages;
        if (!mbar_wait(bar(B_PFULL + b), (i >> 1) & 1)) return false;
        if (!mbar_wait(bar(B_VFULL + s), (i / kTcStages) & 1)) return false;
        tc_fence_after();
        const uint32_t pbase = smem_u32(smem + L::STAGE_OFF + s * L::STAGE_BYTES);  // P sits in the K slot
        const uint32_t vbase = pbase + L::KP_BYTES;
#pragma unroll
        for (int kk = 0; kk < PSTEPS; ++kk) {
          // A = P[128 rows x keys 16kk..16kk+15], K-major: half kk/4, 32 bytes per k-step
          const uint64_t ad = smem_desc_sw128(pbase + (kk >> 2) * L::P_HALF + (kk & 3) * 32, 16, 1024);
          // B = V[keys 16kk.. x head_dim], MN-major: 16 rows = two 8-row atoms; halves Tile::HALF apart
          const uint64_t bd = smem_desc_sw128(vbase + kk * 2048, Tile::HALF, 1024);
          tc_mma_f16(tmem + O_COL, ad, bd, IDESC_O, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(B_OFULL));
        tc_commit(bar(B_KVEMPTY + s));
        return true;
      };
      int j = 0;
      for (; ok && j < ntiles; ++j) {
        const int s = j % kTcStages, b = j & 1;
        if (!mbar_wait(bar(B_KFULL + s), (j / kTcStages) & 1)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bar(B_SEMPTY + b), ((j >> 1) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kbase = smem_u32(smem + L::STAGE_OFF + s * L::STAGE_BYTES);
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const uint64_t ad = smem_desc_sw128(qa + (ks >> 2) * L::QHALF + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kbase + (ks >> 2) * Tile::HALF + (ks & 3) * 32, 16, 1024);
          tc_mma_f16(tmem + S_COL + b * kTcKeys, ad, bd, IDESC_S, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(B_SFULL + b));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && ntiles > 0) ok = issue_pv(ntiles - 1);
      if (!ok) record_error(p.err, PA_DEVERR_TIMEOUT);
      tc_commit(bar(B_MMADONE));
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int quarter = warp & 3;            // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;     // tile row == TMEM lane
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int grow = row0 + row;
    const bool valid = grow < rows;
    const int qi = grow / G, g = grow % G;
    const int lim = !valid ? -1 : (p.causal ? p0 + qi : kend - 1);  // last key this row may see
    // Q row -> shared memory (K-major, 128-byte swizzle); padding rows are zero
    {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.q) +
                                                        ((size_t)(qs + qi) * p.q_heads + h * G + g) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 x = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + L::Q_OFF + (c >> 3) * L::QHALF + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = x;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QFULL));
    }
    griddep_wait();  // before writing `out`

    float m = -INFINITY, l = 0.f;  // running (possibly stale) max in log2 units, row sum
    const float sl2 = p.scale_log2;
    constexpr float kRescale = 8.f;   // raise m only when a row max exceeds it by 2^8
    const uint32_t ocol = tmem + lane_addr + O_COL;
    bool ok = true;

    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1, s = j % kTcStages;
      if (!mbar_wait(bar(B_SFULL + b), (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const int ts = k0 + j * kTcKeys;
      // every row of this warp sees every key of the tile: no mask needed
      const bool all_full = __all_sync(0xffffffffu, ts + kTcKeys - 1 <= lim);
      const uint32_t scol = tmem + lane_addr + S_COL + b * kTcKeys;
      float sv[kTcKeys];
#pragma unroll
      for (int c = 0; c < kTcKeys / 32; ++c) tmem_ld32(scol + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SEMPTY + b));  // S buffer free: S_{j+2} may go there

      float mraw = -INFINITY;  // row max of the raw scores this row may see
      if (all_full) {
#pragma unroll
        for (int e = 0; e < kTcKeys; ++e) mraw = fmaxf(mraw, sv[e]);
      } else {
        const int nvis = lim - ts + 1;  // keys ts .. ts+nvis-1 are visible (nvis may be <= 0)
#pragma unroll
        for (int e = 0; e < kTcKeys; ++e) {
          sv[e] = e < nvis ? sv[e] : -INFINITY;
          mraw = fmaxf(mraw, sv[e]);
        }
      }
      const float mx = mraw * sl2;  // scale > 0 keeps the order

      const bool raise = mx > m + kRescale;  // also true for the first finite max (m = -inf)
      if (__any_sync(0xffffffffu, raise && m != -INFINITY) && j > 0) {
        // O holds sum_{i<j} P_i V_i relative to the old m: rescale it in TMEM
        // once the tensor core has finished with tile j-1 (warp-collective)
        if (!mbar_wait(bar(B_OFULL), (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const float a = (raise && m != -INFINITY) ? exp2f(m - mx) : 1.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tmem_ld32(ocol + 32 * c, ov);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] *= a;
          tmem_st32(ocol + 32 * c, ov);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      if (raise) {
        l = (m == -INFINITY) ? 0.f : l * exp2f(m - mx);
        m = mx;
      }
      const float neg_m = m == -INFINITY ? 0.f : -m;  // fully masked so far: all P are 0
      // P = 2^(s*scale*log2e - m) into the K slot of this stage
      uint8_t* pbase = smem + L::STAGE_OFF + s * L::STAGE_BYTES;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < kTcKeys / 16; ++c) {
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float p0v = exp2f(fmaf(sv[16 * c + e], sl2, neg_m));
          const float p1v = exp2f(fmaf(sv[16 * c + e + 1], sl2, neg_m));
          sum += p0v + p1v;
          pk[e >> 1] = Elem<T>::pack(p0v, p1v);
        }
        // keys 16c..16c+15 = two 16-byte chunks of 8 keys in the 64-key half c/4
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int chunk16 = (c & 3) * 2 + q;
          *reinterpret_cast<uint4*>(pbase + (c >> 2) * L::P_HALF + row * 128 + ((chunk16 ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      l += sum;
      const int nvalid = min(kTcKeys, kend - ts);
      if (nvalid < kTcKeys) {
        // last tile: keys past kend were loaded from stale slots (or not at
        // all); zero their V rows so that p = 0 never meets NaN/Inf
        if (!mbar_wait(bar(B_VFULL + s), (j / kTcStages) & 1)) { ok = false; break; }
        if (row >= nvalid) {
          uint8_t* vrow = pbase + L::KP_BYTES + row * 128;
#pragma unroll
          for (int hf = 0; hf < NH; ++hf)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vrow + hf * Tile::HALF + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();  // P (and zeroed V rows) before the tensor core reads them
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + b));
    }
    if (ok && ntiles > 0) ok = mbar_wait(bar(B_OFULL), (ntiles - 1) & 1);
    if (!ok) {
      if (lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
    } else if (p.causal) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                            ((size_t)(qs + qi) * p.q_heads + h * G + g) * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tmem_ld32(ocol + 32 * c, ov);  // warp-collective: every lane loads, valid rows store
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[4 * c + q] = make_uint4(Elem<T>::pack(ov[8 * q] * inv, ov[8 * q + 1] * inv),
                                        Elem<T>::pack(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv),
                                        Elem<T>::pack(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv),
                                        Elem<T>::pack(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv));
        }
      }
      tc_fence_before();
    } else {
      // shared-prefix partial of this key range: unnormalised o, m, l
      tc_fence_after();
      const size_t prow = ((size_t)qi * p.q_heads + h * G + g) * p.max_splits + blockIdx.z;
      float4* po = reinterpret_cast<float4*>(p.part_o + prow * D);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tmem_ld32(ocol + 32 * c, ov);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int q = 0; q < 8; ++q) po[8 * c + q] = make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
        }
      }
      if (valid) {
        p.part_m[prow] = m;
        p.part_l[prow] = l;
      }
      tc_fence_before();
    }
  }

  // ------------------------------------------------------------------ teardown
  if (warp == 1 && lane == 0) mbar_wait(bar(B_MMADONE), 0);  // no tcgen05 op still running (bounded)
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int BSUB, typename T>
cudaError_t launch_tc_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                        cudaStream_t stream) {
  using L = TcSmem<D, BSUB>;
  auto kern = chunked_prefill_tc_kernel<D, BSUB, T>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int row_tiles = (p.max_q_len * p.group + kTcRows - 1) / kTcRows;
  const int zdim = p.causal ? p.num_reqs : (p.prefix_len + p.key_split - 1) / p.key_split;
  dim3 grid(row_tiles, p.kv_heads, zdim);
  return launch_pdl(kern, grid, dim3(kTcThreads), L::BYTES, stream, kmap, vmap, p);
}

template <int D, typename T>
cudaError_t launch_tc_bs(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p, int bsub,
                         cudaStream_t stream) {
  switch (bsub) {
    case 8: return launch_tc_t<D, 8, T>(kmap, vmap, p, stream);
    case 16: return launch_tc_t<D, 16, T>(kmap, vmap, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_chunked_prefill_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                                      int head_dim, int bsub, pa_dtype dt, cudaStream_t stream) {
  if (head_dim == 128) {
    return dt == PA_BF16 ? launch_tc_bs<128, __nv_bfloat16>(kmap, vmap, p, bsub, stream)
                         : launch_tc_bs<128, __half>(kmap, vmap, p, bsub, stream);
  }
  if (head_dim == 64) {
    return dt == PA_BF16 ? launch_tc_bs<64, __nv_bfloat16>(kmap, vmap, p, bsub, stream)
                         : launch_tc_bs<64, __half>(kmap, vmap, p, bsub, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
