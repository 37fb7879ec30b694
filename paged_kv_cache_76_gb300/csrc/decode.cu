// Paged decode attention for sm_103a: context-split partial kernel and the
// log-sum-exp merge.
//
// Work decomposition.  One warp owns one (request r, KV head h, partition c)
// unit and walks the partition's tokens in tiles of 16 (one bs=16 block, or
// 16/bs blocks for smaller blocks), in logical order.  A CTA holds WARPS
// consecutive units of one request (for 8 KV heads and 4 warps: four heads of
// one partition), so neighbouring heads of the same physical block are read
// by the same CTA at about the same time.  Each warp has its own ring of
// STAGES shared-memory stages fed by TMA (cp.async.bulk.tensor) behind a
// per-warp copy of the partition's Block Table slice: the warp issues the
// loads of tile j+STAGES as soon as it has consumed tile j, so up to STAGES
// tiles per warp are in flight while it computes.  Measured on GB300: 4 warps
// x 2 stages (~65 KB of shared memory, 3 CTAs and 12 streaming warps per SM)
// beats deeper rings with fewer resident CTAs - shorter CTA lifetimes leave a
// smaller tail when the grid drains.
//
// Math per tile (GQA: the whole query-head group shares every K/V tile):
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]       mma.m16n8k16, D/16 k-steps
//   online softmax per head column (reference max in log2 units, raised only
//   when a score passes it by more than 8, and the running sum)
//   P^T -> bf16/fp16, transposed in registers with movmatrix into the B
//   fragment of   O^T[D x 8] += V^T[D x 16 tok] . P^T[16 x 8]   (D/16 m-tiles)
// Tokens past the context are masked to -inf in S and their V rows are zeroed
// in shared memory, so stale data in a partially filled block (NaN included)
// never reaches the output.  All reduction orders depend only on logical
// positions, so relabelling physical blocks gives bitwise-identical results.
//
// Speculative verify (q_len = k+1 queries per request): the n-tile columns are
// the group's heads of each query, column n = i*group + head, up to 32
// columns.  Up to 16 columns one warp holds them (NT = 1 or 2); 17..32
// columns are split over two warps that share the unit's TMA ring (the first
// issues the loads, an "empty" barrier per stage counts both warps out before
// the stage is refilled), which keeps every warp at NT = 2 and 168 registers.
// Column n stops at token ctx - (q_len-1-i) (causal within the draft); a
// column with no visible token in a partition keeps m = -inf, l = 0, o = 0,
// which the merge weighs by zero.  Per column the arithmetic is the same
// whatever the split, so each query's result equals decode over its visible
// prefix bit for bit.
//
// Contiguous mode (CONTIG): the cache is one [slots][max_len][Hkv][D] tensor
// (a vAttention-style virtual tensor, or plain memory) and request r reads
// slot slot_ids[r]: token t is row slot*max_len + t, one 16-row TMA box per
// tile, no Block Table.  Only tokens below the slot's mapped bound
// (slot_tokens[slot], a multiple of 16) are ever loaded; a context past it
// records PA_DEVERR_CONTEXT_LEN and the rest counts as empty.
#include <cuda_pipeline.h>
#include <float.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 2;
constexpr int kMaxTableEntries = 256;  // per warp: split_tokens / block_size <= 256

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// One ring of STAGES K+V tiles per unit; a unit is one warp, or CW > 1 warps
// that split the unit's query columns (NT*8 each) and share its tiles.
template <int D, int BSUB, int NT, typename T, int WARPS, int STAGES, int CW>
struct DecodeSmem {
  using Tile = KvTile<D, BSUB, 16>;
  static constexpr int UNITS = WARPS / CW;
  static constexpr int NBARS = CW > 1 ? 2 * STAGES : STAGES;  // full (+ empty) per stage
  static constexpr int STAGE_BYTES = 2 * Tile::BYTES;  // K tile then V tile
  static constexpr int WARP_BYTES = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = UNITS * WARP_BYTES;
  static constexpr int TAB_OFF = BAR_OFF + UNITS * NBARS * 8;
  // dynamic bytes for `entries` table entries per unit, + alignment slack
  static constexpr int bytes(int entries) { return TAB_OFF + UNITS * entries * 4 + 1024; }
  static constexpr int MAX_BYTES = TAB_OFF + UNITS * kMaxTableEntries * 4 + 1024;
};

template <int D, int BSUB, int NT, typename T, int WARPS, int STAGES, bool CONTIG, int CW>
__global__ void __launch_bounds__(WARPS * 32)
    decode_partial_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          const DecodeParams p) {
  using L = DecodeSmem<D, BSUB, NT, T, WARPS, STAGES, CW>;
  using Tile = typename L::Tile;
  constexpr bool PAIR = CW > 1;  // several warps per unit
  constexpr int KSTEPS = D / 16;
  constexpr int LOADS = Tile::NH * 2;  // TMA boxes per sub-block: halves x {K, V}

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CW > 1: warps CW*k .. CW*k+CW-1 share unit k's ring; the first issues the
  // loads, warp CW*k+i takes query columns [i*NT*8, (i+1)*NT*8)
  const int uw = warp / CW;
  const int half = warp % CW;
  const bool issuer = half == 0;
  const int col0 = half * NT * 8;
  uint8_t* wbase = smem + uw * L::WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF) + uw * L::NBARS;
  uint64_t* empty = bars + STAGES;  // CW > 1 only: every warp of the unit has consumed the stage
  int32_t* tab = reinterpret_cast<int32_t*>(smem + L::TAB_OFF) + uw * p.tab_entries;

  if (lane == 0 && issuer) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      if constexpr (PAIR) mbar_init(smem_u32(&empty[s]), CW);
    }
    fence_mbar_init();
  }
  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  __syncthreads();  // the only CTA-wide barrier; warps are independent below
  griddep_launch_dependents();

  const int r = blockIdx.y;
  const int u = blockIdx.x * L::UNITS + uw;
  const int h = u % p.kv_heads;
  const int c = u / p.kv_heads;
  const int cap = p.maxblk * p.block_size;
  int ctx = __ldg(p.lens + r);
  // tokens [tok_begin, ctx) are this kernel's (tok_begin > 0: the suffix
  // after a shared prefix attended elsewhere)
  bool bad_len = ctx < p.tok_begin || ctx > cap;
  ctx = ctx < p.tok_begin ? p.tok_begin : (ctx > cap ? cap : ctx);
  // contiguous mode: the slot and the tokens it has backed by memory
  int slot = 0, mapped = cap;
  bool bad_slot = false;
  if constexpr (CONTIG) {
    slot = p.slot_ids ? __ldg(p.slot_ids + r) : r;
    if (slot < 0 || slot >= p.num_slots) {
      bad_slot = true;
      mapped = 0;
    } else if (p.slot_tokens) {
      mapped = min(cap, __ldg(p.slot_tokens + slot) & ~15);
    }
    if (ctx > mapped && !bad_slot) bad_len = true;
  }
  const int nsplit = (ctx - p.tok_begin + p.split_tokens - 1) / p.split_tokens;
  const bool active = c < (nsplit > 0 ? nsplit : (p.always_partial ? 0 : 1));
  const int G = p.group;
  const int NC = G * p.q_len;  // columns: (query i, head) pairs, i-major
  const int qh0 = h * G;
  const int tok0 = p.tok_begin + c * p.split_tokens;
  const int tok1 = min(tok0 + p.split_tokens, ctx);
  const int load_end = min(tok1, mapped);  // == tok1 unless a contiguous slot is short of memory
  const int ntiles = active && load_end > tok0 ? (load_end - tok0 + 15) >> 4 : 0;
  const int blk0 = tok0 / p.block_size;

  // Set-up that reads only this call's immutable inputs (block table slice,
  // q) overlaps the previous kernel's tail; the cache is read after
  // griddep_wait().
  bool bad_id = bad_slot;
  uint32_t qf[NT][KSTEPS][2];
  if (ntiles > 0) {
    // Block Table slice of this partition; an out-of-range id is replaced by
    // num_blocks, whose rows lie past the tensor map: TMA then zero-fills.
    if (!CONTIG && issuer) {
      const int nblk = (tok1 - 1) / p.block_size - blk0 + 1;
      const int32_t* trow = p.tables + (size_t)r * p.maxblk + blk0;
      for (int i = lane; i < nblk; i += 32) {
        int b = __ldg(trow + i);
        if (b < 0 || b >= p.num_blocks) {
          bad_id = true;
          b = p.num_blocks;
        }
        tab[i] = b;
      }
    }
    // Q^T as the B operand of S^T = K Q^T: lane holds column (lane/4) of each
    // 8-column n-tile, elements d = 16ks + 2(lane%4) + {0,1} and +8.
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = col0 + nt * 8 + (lane >> 2);
      const int qi = n < NC ? n / G : 0;
      const T* qb = reinterpret_cast<const T*>(p.q) +
                    ((size_t)(r * p.q_len + qi) * p.q_heads + qh0 + (n - qi * G)) * D;
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int d = ks * 16 + 2 * (lane & 3);
        if (n < NC) {
          qf[nt][ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qb + d));
          qf[nt][ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qb + d + 8));
        } else {
          qf[nt][ks][0] = 0u;
          qf[nt][ks][1] = 0u;
        }
      }
    }
  }
  // shared-prefix mode: each table must start with the prefix blocks
  if (!CONTIG && issuer && p.prefix_blocks && c == 0 && h == 0) {
    const int32_t* trow0 = p.tables + (size_t)r * p.maxblk;
    for (int i = lane; i < p.prefix_nblk; i += 32)
      if (__ldg(trow0 + i) != __ldg(p.prefix_blocks + i)) bad_id = true;
  }
  griddep_wait();
  if (bad_len && lane == 0) record_error(p.err, PA_DEVERR_CONTEXT_LEN);
  if (bad_id) record_error(p.err, PA_DEVERR_BLOCK_ID);
  if (!active) return;

  T* out = reinterpret_cast<T*>(p.out);
  // row of column n in q / out / the partials
  auto row_of = [&](int n) {
    const int qi = n / G;
    return (size_t)(r * p.q_len + qi) * p.q_heads + qh0 + (n - qi * G);
  };
  if (ctx == 0) {  // this warp's columns get zero rows
    const int ncw = max(0, min(NC - col0, NT * 8));
    for (int i = lane; i < ncw * D; i += 32) out[row_of(col0 + i / D) * D + i % D] = Elem<T>::from(0.f);
    return;
  }
  __syncwarp();

  const uint64_t pol = policy_evict_first();
  auto issue = [&](int j) {
    const int s = j % STAGES;
    const int ts = tok0 + 16 * j;
    const int nvalid = min(16, load_end - ts);
    const int nsub = (nvalid + BSUB - 1) / BSUB;
    const uint32_t bar = smem_u32(&bars[s]);
    const uint32_t kdst = smem_u32(wbase + s * L::STAGE_BYTES);
    fence_proxy_async_smem();  // earlier generic reads/writes of this stage before the async writes
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, nsub * LOADS * Tile::BOX_BYTES);
    __syncwarp();
    if (lane < nsub * LOADS) {
      const int sub = lane / LOADS;
      const int rem = lane % LOADS;
      const int isv = rem / Tile::NH;
      const int hf = rem % Tile::NH;
      const int tok = ts + sub * BSUB;
      int row;
      if constexpr (CONTIG) {
        row = slot * p.contig_len + tok;
      } else {
        const int b = tab[tok / p.block_size - blk0];
        row = b * p.block_size + tok % p.block_size;
      }
      tma_load_4d_hint(kdst + isv * Tile::BYTES + Tile::box(hf, sub), isv ? &vmap : &kmap, bar, 0, hf, h, row,
                       pol);
    }
  };

  float m[NT][2], lp[NT][2];
  float acc[NT][KSTEPS][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    lp[nt][0] = lp[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) acc[nt][mt][0] = acc[nt][mt][1] = acc[nt][mt][2] = acc[nt][mt][3] = 0.f;
  }

  const int npro = ntiles < STAGES ? ntiles : STAGES;
  if (issuer)
    for (int j = 0; j < npro; ++j) issue(j);

  const float sl2 = p.scale_log2;
  const int mi = lane >> 3, rr = lane & 7;
  const int r0 = lane >> 2;
  // last visible token + 1 of this lane's two columns per n-tile (tok1 for
  // decode, where every column sees the whole partition)
  int lim[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = col0 + nt * 8 + 2 * (lane & 3) + e;
      const int qi = n < NC ? n / G : p.q_len - 1;
      lim[nt][e] = min(load_end, ctx - (p.q_len - 1 - qi));
    }
  bool failed = false;
  int j = 0;
  for (; j < ntiles; ++j) {
    const int s = j % STAGES;
    if (!mbar_wait(smem_u32(&bars[s]), (j / STAGES) & 1)) {
      failed = true;
      break;
    }
    const int ts = tok0 + 16 * j;
    const int nvalid = min(16, load_end - ts);
    uint8_t* kt = wbase + s * L::STAGE_BYTES;
    uint8_t* vt = kt + Tile::BYTES;
    if (nvalid < 16) {
      // rows past the context: zero V so that p = 0 never meets stale NaN/Inf
      const int nz = (16 - nvalid) * Tile::NH * 8;
      for (int i = lane; i < nz; i += 32) {
        const int row = nvalid + i / (Tile::NH * 8);
        const int rem = i % (Tile::NH * 8);
        *reinterpret_cast<uint4*>(vt + Tile::line(rem >> 3, row) + ((rem & 7) << 4)) = make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    const uint32_t kts = smem_u32(kt), vts = smem_u32(vt);

    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      uint32_t a[4];
      ldmatrix_x4(a, kts + Tile::offset(rr + 8 * (mi & 1), 2 * ks + (mi >> 1)));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816<T>(sacc[nt], a, qf[nt][ks][0], qf[nt][ks][1]);
    }

    uint32_t pb0[NT], pb1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int t0 = ts + r0;
      const float s0 = t0 < lim[nt][0] ? sacc[nt][0] * sl2 : -INFINITY;
      const float s1 = t0 < lim[nt][1] ? sacc[nt][1] * sl2 : -INFINITY;
      const float s2 = t0 + 8 < lim[nt][0] ? sacc[nt][2] * sl2 : -INFINITY;
      const float s3 = t0 + 8 < lim[nt][1] ? sacc[nt][3] * sl2 : -INFINITY;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      // m is the reference the column's exponents are taken against.  It is
      // raised (to the tile's maximum) only when a score exceeds it by more
      // than 8 (log2 units), so p stays below 2^8 and most tiles skip the
      // rescale of o and l; o, l and m stay consistent, so out and the merge
      // are unchanged up to rounding.  Each column decides from its own
      // scores alone (the vote only skips work when no column moves), so a
      // column's bits do not depend on its neighbours.  A column that has
      // seen no token yet keeps m = -inf: exponents then use 0 as reference,
      // so every p is exactly 0.
      const bool up0 = mx0 > m[nt][0] + 8.f, up1 = mx1 > m[nt][1] + 8.f;
      if (__any_sync(0xffffffffu, up0 || up1)) {
        const float al0 = up0 ? exp2f(m[nt][0] - mx0) : 1.f;
        const float al1 = up1 ? exp2f(m[nt][1] - mx1) : 1.f;
        m[nt][0] = up0 ? mx0 : m[nt][0];
        m[nt][1] = up1 ? mx1 : m[nt][1];
        lp[nt][0] *= al0;
        lp[nt][1] *= al1;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          acc[nt][mt][0] *= al0;
          acc[nt][mt][1] *= al1;
          acc[nt][mt][2] *= al0;
          acc[nt][mt][3] *= al1;
        }
      }
      const float mb0 = m[nt][0] == -INFINITY ? 0.f : m[nt][0];
      const float mb1 = m[nt][1] == -INFINITY ? 0.f : m[nt][1];
      const float p0 = exp2f(s0 - mb0), p1 = exp2f(s1 - mb1);
      const float p2 = exp2f(s2 - mb0), p3 = exp2f(s3 - mb1);
      // P is rounded to the input type for the P.V MMA; the denominator sums
      // the same rounded values, so the output is an exact convex combination
      const uint32_t pk01 = Elem<T>::pack(p0, p1), pk23 = Elem<T>::pack(p2, p3);
      lp[nt][0] += Elem<T>::lo(pk01) + Elem<T>::lo(pk23);
      lp[nt][1] += Elem<T>::hi(pk01) + Elem<T>::hi(pk23);
      pb0[nt] = movmatrix_trans(pk01);
      pb1[nt] = movmatrix_trans(pk23);
    }

#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      uint32_t a[4];
      ldmatrix_x4_trans(a, vts + Tile::offset(rr + 8 * (mi >> 1), 2 * mt + (mi & 1)));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816<T>(acc[nt][mt], a, pb0[nt], pb1[nt]);
    }
    __syncwarp();
    if constexpr (PAIR) {
      // the stage is refilled once both warps of the pair are done with it
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      if (issuer && j + STAGES < ntiles) {
        if (!mbar_wait(smem_u32(&empty[s]), (j / STAGES) & 1)) {
          failed = true;
          break;
        }
        issue(j + STAGES);
      }
    } else {
      if (j + STAGES < ntiles) issue(j + STAGES);
    }
  }

  if (failed) {
    if (lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
    // the issuing warp drains its loads still in flight (bounded) before leaving
    if (issuer)
      for (int k = j + 1; k < ntiles && k < j + STAGES; ++k)
        mbar_wait(smem_u32(&bars[k % STAGES]), (k / STAGES) & 1);
    return;
  }

  // finish the per-head sums across the 8 lanes holding each column
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = lp[nt][e];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      lp[nt][e] = l;
    }

  if (nsplit == 1 && !p.always_partial) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int n = col0 + nt * 8 + 2 * (lane & 3) + e;
        if (n < NC) {
          const float inv = lp[nt][e] > 0.f ? 1.f / lp[nt][e] : 0.f;
          T* o = out + row_of(n) * D;
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            o[mt * 16 + r0] = Elem<T>::from(acc[nt][mt][e] * inv);
            o[mt * 16 + r0 + 8] = Elem<T>::from(acc[nt][mt][2 + e] * inv);
          }
        }
      }
  } else {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int n = col0 + nt * 8 + 2 * (lane & 3) + e;
        if (n < NC) {
          const size_t row = row_of(n);
          const int slot = p.slot_base + c;
          float* po = p.part_o + (row * p.max_splits + slot) * D;
#pragma unroll
          for (int mt = 0; mt < KSTEPS; ++mt) {
            po[mt * 16 + r0] = acc[nt][mt][e];
            po[mt * 16 + r0 + 8] = acc[nt][mt][2 + e];
          }
          if (r0 == 0) {
            p.part_m[row * p.max_splits + slot] = m[nt][e];
            p.part_l[row * p.max_splits + slot] = lp[nt][e];
          }
        }
      }
  }
}

// One CTA of 4 warps per (request, query head): combine the partitions of
// requests that have more than one.  M = max_c m_c; w_c = 2^(m_c - M);
// out = sum_c w_c o_c / sum_c w_c l_c.  Warp w takes partitions w, w+4, ...;
// the four partial sums are added in warp order, so the result depends only on
// logical positions.
template <int D, typename T>
__global__ void __launch_bounds__(128) lse_merge_kernel(const MergeParams p) {
  constexpr int V = D / 32;
  constexpr int NW = 4;
  __shared__ float s_max[NW];
  __shared__ float s_den[NW];
  __shared__ __align__(16) float s_acc[NW][D];
  griddep_wait();  // the partials come from the kernel before this one
  griddep_launch_dependents();
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (row >= p.num_seqs * p.q_len * p.q_heads) return;
  const int r = row / (p.q_heads * p.q_len);
  int ctx = __ldg(p.lens + r);
  ctx = ctx < p.tok_begin ? p.tok_begin : (ctx > p.cap ? p.cap : ctx);
  const int nsplit = p.extra_slots + (ctx - p.tok_begin + p.split_tokens - 1) / p.split_tokens;
  if (nsplit <= 1 && !p.always) return;  // pa_decode_partial wrote this row directly
  const float* pm = p.part_m + (size_t)row * p.max_splits;
  const float* pl = p.part_l + (size_t)row * p.max_splits;
  const float* po = p.part_o + (size_t)row * p.max_splits * D + lane * V;

  float M = -INFINITY;
  for (int c = threadIdx.x; c < nsplit; c += NW * 32) M = fmaxf(M, pm[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_max[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(s_max[0], s_max[1]), fmaxf(s_max[2], s_max[3]));

  float a[V];
#pragma unroll
  for (int i = 0; i < V; ++i) a[i] = 0.f;
  float den = 0.f;
#pragma unroll 4
  for (int c = warp; c < nsplit; c += NW) {
    const float w = pm[c] == -INFINITY ? 0.f : exp2f(pm[c] - M);  // a partition the row sees nothing of
    den += w * pl[c];
    if constexpr (V == 4) {
      const float4 x = *reinterpret_cast<const float4*>(po + (size_t)c * D);
      a[0] += w * x.x;
      a[1] += w * x.y;
      a[2] += w * x.z;
      a[3] += w * x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(po + (size_t)c * D);
      a[0] += w * x.x;
      a[1] += w * x.y;
    }
  }
#pragma unroll
  for (int i = 0; i < V; ++i) s_acc[warp][lane * V + i] = a[i];
  if (lane == 0) s_den[warp] = den;
  __syncthreads();
  const float dsum = ((s_den[0] + s_den[1]) + s_den[2]) + s_den[3];
  const float inv = dsum > 0.f ? 1.f / dsum : 0.f;
  T* o = reinterpret_cast<T*>(p.out) + (size_t)row * D;
  for (int d = threadIdx.x; d < D; d += NW * 32)
    o[d] = Elem<T>::from((((s_acc[0][d] + s_acc[1][d]) + s_acc[2][d]) + s_acc[3][d]) * inv);
}

// The same merge with one warp per row, for at most 32 partitions: lane c
// holds m_c and l_c, each lane owns D/32 output dims, and the o partials are
// loaded eight partitions at a time ahead of the sums, so a row costs about
// one round trip to L2.  Partitions are added in order (deterministic).
template <int D, typename T>
__global__ void __launch_bounds__(256) lse_merge_warp_kernel(const MergeParams p) {
  constexpr int V = D / 32;
  constexpr int CH = 8;  // o partials in flight per lane
  griddep_wait();        // the partials come from the kernel before this one
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= p.num_seqs * p.q_len * p.q_heads) return;
  const int r = row / (p.q_heads * p.q_len);
  int ctx = __ldg(p.lens + r);
  ctx = ctx < p.tok_begin ? p.tok_begin : (ctx > p.cap ? p.cap : ctx);
  const int nsplit = p.extra_slots + (ctx - p.tok_begin + p.split_tokens - 1) / p.split_tokens;
  if (nsplit <= 1 && !p.always) return;  // pa_decode_partial wrote this row directly
  const float* pm = p.part_m + (size_t)row * p.max_splits;
  const float* pl = p.part_l + (size_t)row * p.max_splits;
  const float* po = p.part_o + (size_t)row * p.max_splits * D + lane * V;
  const float mc = lane < nsplit ? pm[lane] : -INFINITY;
  const float lc = lane < nsplit ? pl[lane] : 0.f;
  float x[CH][V];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    if (c < nsplit) {
      if constexpr (V == 4) {
        const float4 v = *reinterpret_cast<const float4*>(po + (size_t)c * D);
        x[c][0] = v.x, x[c][1] = v.y, x[c][2] = v.z, x[c][3] = v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(po + (size_t)c * D);
        x[c][0] = v.x, x[c][1] = v.y;
      }
    }
  }
  float M = mc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w = lane < nsplit && mc != -INFINITY ? exp2f(mc - M) : 0.f;
  float den = w * lc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  float a[V];
#pragma unroll
  for (int i = 0; i < V; ++i) a[i] = 0.f;
  for (int c0 = 0; c0 < nsplit; c0 += CH) {
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const float wc = __shfl_sync(0xffffffffu, w, (c0 + c) & 31);
      if (c0 + c < nsplit) {
#pragma unroll
        for (int i = 0; i < V; ++i) a[i] += wc * x[c][i];
      }
    }
    // next chunk of o partials
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int cc = c0 + CH + c;
      if (cc < nsplit) {
        if constexpr (V == 4) {
          const float4 v = *reinterpret_cast<const float4*>(po + (size_t)cc * D);
          x[c][0] = v.x, x[c][1] = v.y, x[c][2] = v.z, x[c][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(po + (size_t)cc * D);
          x[c][0] = v.x, x[c][1] = v.y;
        }
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  T* o = reinterpret_cast<T*>(p.out) + (size_t)row * D + lane * V;
  if constexpr (V == 4) {
    *reinterpret_cast<uint2*>(o) = make_uint2(Elem<T>::pack(a[0] * inv, a[1] * inv), Elem<T>::pack(a[2] * inv, a[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(o) = Elem<T>::pack(a[0] * inv, a[1] * inv);
  }
}

template <int D, int BSUB, int NT, typename T, bool CONTIG = false, int CW = 1>
cudaError_t launch_decode_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                            cudaStream_t stream) {
  constexpr int W = kDecodeWarps, S = kDecodeStages;
  using L = DecodeSmem<D, BSUB, NT, T, W, S, CW>;
  auto kern = decode_partial_kernel<D, BSUB, NT, T, W, S, CONTIG, CW>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::MAX_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int units = p.grid_splits * p.kv_heads;
  dim3 grid((units + L::UNITS - 1) / L::UNITS, p.num_seqs);
  return launch_pdl(kern, grid, dim3(W * 32), L::bytes(CONTIG ? 0 : p.tab_entries), stream, kmap, vmap, p);
}

template <int D, typename T>
cudaError_t launch_decode_contig_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                   cudaStream_t stream) {
  if (p.group * p.q_len <= 8) return launch_decode_t<D, 16, 1, T, true>(kmap, vmap, p, stream);
  if (p.group * p.q_len <= 16) return launch_decode_t<D, 16, 2, T, true>(kmap, vmap, p, stream);
  return cudaErrorInvalidValue;
}

template <int D, int BSUB, typename T>
cudaError_t launch_decode_nt(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                             cudaStream_t stream) {
  const int cols = p.group * p.q_len;
  if (cols <= 8) return launch_decode_t<D, BSUB, 1, T>(kmap, vmap, p, stream);
  if (cols <= 16) return launch_decode_t<D, BSUB, 2, T>(kmap, vmap, p, stream);
  // 17..32 columns: two warps per unit, 16 columns each, sharing its tiles.
  // Measured on GB300 (k = 7 drafts, 32 columns, spec_verify_decode shape):
  // one warp with 32 columns (255 registers, spills) 152.6 us per step; two
  // warps x 16 columns 140.5 us (4 stages: 141.4); four warps x 8 columns
  // (4 stages, 93 registers, 5 CTAs per SM) 148.7 us - each warp re-reads
  // the K/V tile from shared memory for its own columns.
  if (cols <= 32) return launch_decode_t<D, BSUB, 2, T, false, 2>(kmap, vmap, p, stream);
  return cudaErrorInvalidValue;
}

template <int D, typename T>
cudaError_t launch_decode_bs(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p, int bsub,
                             cudaStream_t stream) {
  switch (bsub) {
    case 4: return launch_decode_nt<D, 4, T>(kmap, vmap, p, stream);
    case 8: return launch_decode_nt<D, 8, T>(kmap, vmap, p, stream);
    case 16: return launch_decode_nt<D, 16, T>(kmap, vmap, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_partial(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                  int head_dim, int bsub, pa_dtype dt, cudaStream_t stream) {
  if (head_dim == 128) {
    return dt == PA_BF16 ? launch_decode_bs<128, __nv_bfloat16>(kmap, vmap, p, bsub, stream)
                         : launch_decode_bs<128, __half>(kmap, vmap, p, bsub, stream);
  }
  if (head_dim == 64) {
    return dt == PA_BF16 ? launch_decode_bs<64, __nv_bfloat16>(kmap, vmap, p, bsub, stream)
                         : launch_decode_bs<64, __half>(kmap, vmap, p, bsub, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_contig(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                                 int head_dim, pa_dtype dt, cudaStream_t stream) {
  if (head_dim == 128)
    return dt == PA_BF16 ? launch_decode_contig_t<128, __nv_bfloat16>(kmap, vmap, p, stream)
                         : launch_decode_contig_t<128, __half>(kmap, vmap, p, stream);
  if (head_dim == 64)
    return dt == PA_BF16 ? launch_decode_contig_t<64, __nv_bfloat16>(kmap, vmap, p, stream)
                         : launch_decode_contig_t<64, __half>(kmap, vmap, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_lse_merge(const MergeParams& p, int head_dim, pa_dtype dt, cudaStream_t stream) {
  if (p.max_splits <= 32) {  // one warp per row
    const dim3 grid((p.num_seqs * p.q_len * p.q_heads + 7) / 8), block(256);
    if (head_dim == 128)
      return dt == PA_BF16 ? launch_pdl(lse_merge_warp_kernel<128, __nv_bfloat16>, grid, block, 0, stream, p)
                           : launch_pdl(lse_merge_warp_kernel<128, __half>, grid, block, 0, stream, p);
    if (head_dim == 64)
      return dt == PA_BF16 ? launch_pdl(lse_merge_warp_kernel<64, __nv_bfloat16>, grid, block, 0, stream, p)
                           : launch_pdl(lse_merge_warp_kernel<64, __half>, grid, block, 0, stream, p);
    return cudaErrorInvalidValue;
  }
  const dim3 grid(p.num_seqs * p.q_len * p.q_heads), block(128);
  if (head_dim == 128)
    return dt == PA_BF16 ? launch_pdl(lse_merge_kernel<128, __nv_bfloat16>, grid, block, 0, stream, p)
                         : launch_pdl(lse_merge_kernel<128, __half>, grid, block, 0, stream, p);
  if (head_dim == 64)
    return dt == PA_BF16 ? launch_pdl(lse_merge_kernel<64, __nv_bfloat16>, grid, block, 0, stream, p)
                         : launch_pdl(lse_merge_kernel<64, __half>, grid, block, 0, stream, p);
  return cudaErrorInvalidValue;
}

DecodeWorkspace decode_workspace_layout(int num_seqs, int q_heads, int head_dim, int max_splits) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  DecodeWorkspace w{};
  const size_t rows = (size_t)num_seqs * q_heads * max_splits;
  w.o_off = 0;
  w.m_off = al(rows * head_dim * sizeof(float));
  w.l_off = w.m_off + al(rows * sizeof(float));
  w.bytes = w.l_off + al(rows * sizeof(float));
  return w;
}

}  // namespace pa
