// Paged attention of many query rows on the 5th-generation tensor cores
// (tcgen05 + tensor memory), sm_103a, for blocks of >= 8 tokens: chunked
// prefill (causal) and the shared-prefix pass of a decode batch (partials).
//
// A CTA owns two tiles of 128 rows (A and B) of one (request, KV head); a row
// is one (query, head of the GQA group) pair, so the whole group shares every
// K/V tile, and each 64-key K/V tile gathered from the paged cache serves 256
// rows.
//
// Tensor memory (512 columns, one CTA per SM):
//
//   S_x buffer b  [(2x + b) * 64, +64)   S = Q_x K^T of key tiles j = b mod 2 (fp32);
//                                        P_x(j) over its first 32 columns (two per column)
//   O_A, O_B      [256, 384), [384, 512) fp32 accumulators, 128 rows x D
//
// Design points, each measured on GB300:
//  * Two S buffers per Q tile break the chain S_x(j) -> softmax -> P.V_x(j)
//    -> S_x(j+1): S_x(j) overwrites only P_x(j-2), so it is issued while the
//    softmax still works on tile j-1.  Two of them fit beside both O
//    accumulators only at 64 keys per tile, where an SS MMA is bound by its
//    6 KB of shared-memory operand reads (2/3 rate); the kernel still gains,
//    because the 128-key form spent most of each tile waiting on its chain.
//  * P stays in tensor memory: the softmax writes P (bf16/fp16) over the
//    first half of its S columns and O += P V reads A from TMEM, so P never
//    crosses shared memory.
//  * The softmax warps never issue MMAs and do not meet per tile: each warp
//    waits for its S buffer on its own and signals its part of P on an
//    mbarrier, so no warp waits for another's MMA issue.
//  * The softmax holds its S row in registers (one TMEM round trip per tile).
//
// Warp roles (384 threads = 12 warps, so that each thread may hold 168
// registers):
//   warps 0,1   MMA issuers, one warp per Q tile x (one elected lane issues,
//               with warp-uniform descriptors): per key tile j,
//                 S_x(j) = Q_x K_j^T into buffer j % 2, once P.V_x(j-2) has
//                 completed (the tcgen05 ordering guarantee covers only MMAs
//                 into the same accumulator), then
//                 O_x += P_x(j-1) V_{j-1}, once the tile's four softmax warps
//                 have written P_x(j-1).
//               The two issuers wait only on their own tile; the tensor pipe
//               interleaves their MMAs.
//   warp 2      TMA producer of K, warp 3 of V; separate 4-stage rings, so a
//               K slot frees as soon as both S MMAs have read it.
//   warps 4..7  softmax of tile A, warps 8..11 of tile B: thread = TMEM lane
//               = row.  It loads its S row, takes the row maximum, writes
//               P = 2^(s*scale*log2e - m) into TMEM and sums it.  The running
//               maximum m is raised only when a row maximum exceeds it by
//               more than 2^8 (O is then rescaled in TMEM, once P.V_x(j-1)
//               has completed); the final O / sum uses the same m, so this is
//               exact.
// Q and K are K-major and V is MN-major in the canonical 128-byte-swizzled
// shared-memory layouts.  Every mbarrier wait is bounded.
#include <float.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kRows = 128;  // rows per Q tile (M of every MMA)
constexpr int kKeys = 64;   // keys per K/V tile (N of S, K of P.V)
// 4 K and 4 V stages of 64-key tiles (head_dim 128: Q 64 KB + K 64 KB + V 64
// KB of shared memory); 5 of either measured slower.
constexpr int kKStages = 4;
constexpr int kVStages = 4;
constexpr int kMmaWarp = 0;  // warps 0, 1: MMA issuers of Q tiles A, B (warp 0 owns TMEM)
constexpr unsigned kAll = 0xffffffffu;
constexpr int kKWarp = 2;
constexpr int kVWarp = 3;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kThreads = 32 * 12;
constexpr uint32_t kTmem = 512;

__device__ __forceinline__ uint8_t* align1024_tc(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, int BSUB>
struct TcSmem {
  using Tile = KvTile<D, BSUB, kKeys>;  // D/64 halves x 128 rows x 128 B
  static constexpr int NH = D / 64;
  static constexpr int QHALF = kRows * 128;
  static constexpr int QTILE = NH * QHALF;
  static constexpr int Q_OFF = 0;  // Q_A, Q_B
  static constexpr int K_OFF = Q_OFF + 2 * QTILE;
  static constexpr int V_OFF = K_OFF + kKStages * Tile::BYTES;
  static constexpr int BAR_OFF = V_OFF + kVStages * Tile::BYTES;
  static constexpr int NBARS = 2 * kKStages + 2 * kVStages + 15;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = SLOT_OFF + 16 + 1024;
  static_assert(BSUB * 128 >= 1024, "needs blocks of at least 8 tokens (one 8-row swizzle atom per box)");
  static_assert(BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert((kKeys / BSUB) * NH <= 32, "the V producer issues one box per lane");
};

// barrier indices
constexpr int B_KFULL = 0;                     // [kKStages] the K producer warp arrives (+ TMA bytes)
constexpr int B_KEMPTY = B_KFULL + kKStages;   // [kKStages] one tcgen05.commit per issuer after S_x(j)
constexpr int B_VFULL = B_KEMPTY + kKStages;   // [kVStages] the V producer warp arrives (+ TMA bytes)
constexpr int B_VEMPTY = B_VFULL + kVStages;   // [kVStages] one tcgen05.commit per issuer after P.V_x(j)
constexpr int B_SFULL = B_VEMPTY + kVStages;   // [2 Q tiles][2 S buffers] S_x(j) written (commit)
constexpr int B_PFULL = B_SFULL + 4;           // [2 Q tiles][2 S buffers] P_x(j) in TMEM (four softmax warps)
constexpr int B_OFULL = B_PFULL + 4;           // [2 Q tiles][2 S buffers] P.V_x(j) complete (commit)
constexpr int B_QFULL = B_OFULL + 4;            // [2] Q_x of the next work unit in smem (four softmax warps)
constexpr int B_MMADONE = B_QFULL + 2;
static_assert(B_MMADONE + 1 == 2 * kKStages + 2 * kVStages + 15, "barrier count");

// One work unit: a tile of 2 x 128 rows of one (request, KV head) for the
// causal prefill, or of one (prefix key range, KV head) for the shared-prefix
// pass.  Units are numbered z-major, then row tile in reverse, then head: the
// last row tiles of a causal chunk see the most keys, so dispatch in index
// order starts the longest units of every head first.
struct TcUnit {
  int z, h, row0, r, qs, chunk, p0, k0, kend, rows, ntiles;
};

// Geometry of unit u from immutable inputs only.  false: the request's
// q_start/context_lens are inconsistent (the unit is skipped).
__device__ __forceinline__ bool tc_unit(const PrefillParams& p, int u, int row_tiles, TcUnit& w) {
  const int per_z = row_tiles * p.kv_heads;
  w.z = u / per_z;
  const int rem = u - w.z * per_z;
  const int rt = rem / p.kv_heads;
  w.h = rem - rt * p.kv_heads;
  w.row0 = (row_tiles - 1 - rt) * 2 * kRows;
  w.ntiles = 0;
  const int G = p.group;
  if (p.causal) {
    // request r = z, chunk at absolute position p0, row (query i, head g)
    // sees keys 0 .. p0+i
    w.r = w.z;
    w.qs = __ldg(p.q_start + w.r);
    const int qe = __ldg(p.q_start + w.r + 1);
    w.chunk = qe - w.qs;
    const int ctx = __ldg(p.lens + w.r);
    w.p0 = ctx - w.chunk;
    if (w.qs < 0 || qe < w.qs || qe > p.total_q || w.chunk > p.max_q_len || w.p0 < 0 ||
        ctx > p.maxblk * p.block_size)
      return false;
    w.k0 = 0;
    w.rows = w.chunk * G;
    if (w.row0 >= w.rows) return true;
    const int last_row = min(w.row0 + 2 * kRows, w.rows) - 1;
    w.kend = w.p0 + last_row / G + 1;
  } else {
    // one virtual request of total_q queries (the decode batch); keys
    // [k0, kend) = split z of the prefix, visible to every row
    w.r = 0;
    w.qs = 0;
    w.chunk = p.total_q;
    w.p0 = 0;
    w.k0 = w.z * p.key_split;
    w.kend = min(w.k0 + p.key_split, p.prefix_len);
    w.rows = w.chunk * G;
    if (w.row0 >= w.rows || w.k0 >= w.kend) return true;
  }
  w.ntiles = (w.kend - w.k0 + kKeys - 1) / kKeys;
  return true;
}

template <int D, int BSUB, typename T>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const PrefillParams p) {
  using L = TcSmem<D, BSUB>;
  using Tile = typename L::Tile;
  constexpr int NH = D / 64;
  constexpr int KSTEPS = D / 16;      // S = Q K^T: K dimension = head_dim
  constexpr int PSTEPS = kKeys / 16;  // O = P V:   K dimension = keys
  constexpr int SUBS = kKeys / BSUB;  // boxes per half per tile
  constexpr uint32_t S_COL = 0;       // S_x buffer b at (2x + b) * kKeys; P_x(j) in the first kKeys/2 of its buffer
  constexpr uint32_t O_COL = 4 * kKeys;
  constexpr uint32_t IDESC_S = idesc_f16<T>(kRows, kKeys, false);
  constexpr uint32_t IDESC_O = idesc_f16<T>(kRows, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024_tc(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::SLOT_OFF);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  // CTA b (linear block index) takes units b, b + nctas, ...
  const int row_tiles = (p.max_q_len * G + 2 * kRows - 1) / (2 * kRows);
  const int nunits = row_tiles * p.kv_heads * (p.causal ? p.num_reqs : (p.prefix_len + p.key_split - 1) / p.key_split);
  const int cta0 = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int nctas = gridDim.x * gridDim.y * gridDim.z;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 2);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VEMPTY + i), 2);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_PFULL + i), 4);
      mbar_init(bar(B_OFULL + i), 1);
    }
    mbar_init(bar(B_QFULL), 4);
    mbar_init(bar(B_QFULL + 1), 4);
    mbar_init(bar(B_MMADONE), 2);  // the two MMA issuers' last commits
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmem);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == kKWarp || warp == kVWarp) {
    // ---------------------------------------------------------------- producers
    const int isv = warp == kVWarp;  // 0: K, 1: V
    const int my_sub = lane / NH, hf = lane % NH;  // one box per lane: subs [0, SUBS) x halves
    const bool has_box = lane < SUBS * NH;
    const CUtensorMap* map = isv ? &vmap : &kmap;
    const int full0 = isv ? B_VFULL : B_KFULL, empty0 = isv ? B_VEMPTY : B_KEMPTY;
    const uint32_t base = smem_u32(smem + (isv ? L::V_OFF : L::K_OFF));
    const uint64_t pol = policy_evict_last();  // K/V tiles are re-read by the other row tiles
    const int nst = isv ? kVStages : kKStages;
    int gt = 0;  // K/V tiles issued by this CTA (ring position and phase)
    bool failed = false;
    griddep_wait();  // the cache (this step's reshape_and_cache) comes from the kernel before
    for (int u = cta0; u < nunits && !failed; u += nctas) {
      TcUnit w;
      if (!tc_unit(p, u, row_tiles, w) || w.ntiles <= 0) continue;
      const int32_t* trow = p.tables + (size_t)w.r * p.maxblk;
      for (int j = 0; j < w.ntiles; ++j, ++gt) {
        const int s = gt % nst;
        if (gt >= nst && !mbar_wait(bar(empty0 + s), ((gt / nst) - 1) & 1)) {
          failed = true;
          break;
        }
        const int ts = w.k0 + j * kKeys;
        const int nvalid = min(kKeys, w.kend - ts);
        const int nsub = (nvalid + BSUB - 1) / BSUB;
        if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), nsub * NH * Tile::BOX_BYTES);
        __syncwarp();
        if (has_box && my_sub < nsub) {
          const int tok = ts + my_sub * BSUB;
          int b = __ldg(trow + tok / p.block_size);
          if (b < 0 || b >= p.num_blocks) {
            record_error(p.err, PA_DEVERR_BLOCK_ID);
            b = p.num_blocks;  // rows past the tensor map: TMA zero-fills
          }
          tma_load_4d_hint(base + s * Tile::BYTES + Tile::box(hf, my_sub), map, bar(full0 + s), 0, hf, w.h,
                           b * p.block_size + tok % p.block_size, pol);
        }
      }
    }
    if (failed && lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
    for (int t = gt - nst < 0 ? 0 : gt - nst; t < gt; ++t)  // loads in flight land before exit (bounded)
      mbar_wait(bar(full0 + t % nst), (t / nst) & 1);
  } else if (warp < kKWarp) {
    // ---------------------------------------------------------------- MMA issuers
    // One warp per Q tile: warp 0 issues tile A's MMAs, warp 1 tile B's.
    // tcgen05.mma issue blocks while the tensor pipe is busy, so a single
    // issuer serialises its waits behind the other tile's MMAs; two issuers
    // wait only on their own tile, and the pipe interleaves their work.  The
    // whole warp runs the loop (its waits are voted, so control flow stays
    // warp-uniform) and one elected lane issues each MMA and commit, with
    // descriptors that are warp-uniform values.
    {
      const int x = warp;
      bool ok = true;
      const uint32_t kbase = smem_u32(smem + L::K_OFF);
      const uint32_t qa = smem_u32(smem + L::Q_OFF + x * L::QTILE);
      const uint32_t sd = tmem + S_COL + 2 * x * kKeys;
      const uint32_t vbase = smem_u32(smem + L::V_OFF);
      const uint32_t od0 = tmem + O_COL + x * D;
      int gt = 0, nu = 0;  // key tiles and units processed by this CTA
      // O_x += P_x(t) V_t once the four softmax warps have written P_x(t)
      // (jt: the tile's index in its unit; its first P.V overwrites O_x)
      auto issue_pv = [&](int t, int jt) -> bool {
        const int pb = t & 1, vst = t % kVStages;
        if (!__all_sync(kAll, mbar_wait(bar(B_PFULL + 2 * x + pb), (t >> 1) & 1) &&
                                  mbar_wait(bar(B_VFULL + vst), (t / kVStages) & 1)))
          return false;
        tc_fence_after();
        const uint32_t vb = vbase + vst * Tile::BYTES;
#pragma unroll
        for (int kk = 0; kk < PSTEPS; ++kk) {
          // A = P_x[128 rows x keys 16kk..16kk+15] in TMEM (8 columns); B = V rows 16kk.., MN-major
          const uint64_t bd = smem_desc_sw128(vb + kk * 2048, Tile::HALF, 1024);
          tc_mma_f16_ts_warp(od0, sd + pb * kKeys + kk * 8, bd, IDESC_O, (jt > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit_warp(bar(B_OFULL + 2 * x + pb));
        tc_commit_warp(bar(B_VEMPTY + vst));  // this issuer is done with V_t
        return true;
      };
      for (int u = cta0; ok && u < nunits; u += nctas) {
        TcUnit w;
        if (!tc_unit(p, u, row_tiles, w)) {
          if (x == 0) {
            griddep_wait();
            if (lane == 0) record_error(p.err, PA_DEVERR_QUERY_RANGE);
          }
          continue;
        }
        if (w.ntiles <= 0) continue;
        // Q_x of this unit is in smem; the softmax warps have also finished
        // the previous unit (its last P.V completed and O_x was read out).
        if (!__all_sync(kAll, mbar_wait(bar(B_QFULL + x), nu & 1))) { ok = false; break; }
        // Tile B starts half a key tile behind tile A (once P_A(0) is being
        // written), so that the two softmaxes alternate instead of overlapping.
        if (x == 1 && nu == 0 && !__all_sync(kAll, mbar_wait(bar(B_PFULL), 0))) { ok = false; break; }
        ++nu;
        for (int j = 0; ok && j < w.ntiles; ++j, ++gt) {
          const int sk = gt % kKStages, b = gt & 1;
          // S_x(j) = Q_x K_j^T into buffer b.  It overwrites P_x(j-2): wait for P.V_x(j-2).
          if (!__all_sync(kAll, mbar_wait(bar(B_KFULL + sk), (gt / kKStages) & 1))) { ok = false; break; }
          if (gt >= 2 && !__all_sync(kAll, mbar_wait(bar(B_OFULL + 2 * x + b), ((gt - 2) >> 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb = kbase + sk * Tile::BYTES;
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            const uint64_t ad = smem_desc_sw128(qa + (ks >> 2) * L::QHALF + (ks & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(kb + (ks >> 2) * Tile::HALF + (ks & 3) * 32, 16, 1024);
            tc_mma_f16_warp(sd + b * kKeys, ad, bd, IDESC_S, ks > 0 ? 1u : 0u);
          }
          tc_commit_warp(bar(B_SFULL + 2 * x + b));
          tc_commit_warp(bar(B_KEMPTY + sk));  // this issuer is done with K_j
          // P.V of the previous tile, behind S(j) so that S(j) does not wait for it
          if (j > 0 && !issue_pv(gt - 1, j - 1)) {
            ok = false;
            break;
          }
        }
        if (ok && !issue_pv(gt - 1, w.ntiles - 1)) ok = false;  // the unit's last P.V
      }
      if (!ok && lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
      tc_commit_warp(bar(B_MMADONE));
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int x = (warp - kSoftmaxWarp0) >> 2;  // Q tile: 0 = A (warps 4..7), 1 = B (warps 8..11)
    const int quarter = warp & 3;                // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;         // row within the tile == TMEM lane
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    constexpr float kRescale = 8.f;
    const uint32_t scol0 = tmem + lane_addr + S_COL + 2 * x * kKeys;
    const uint32_t ocol = tmem + lane_addr + O_COL + x * D;
    uint8_t* qt = smem + L::Q_OFF + x * L::QTILE;
    bool ok = true;
    int gt = 0;  // key tiles processed by this CTA
    for (int u = cta0; ok && u < nunits; u += nctas) {
      TcUnit w;
      if (!tc_unit(p, u, row_tiles, w) || w.ntiles <= 0) continue;
      const int grow = w.row0 + x * kRows + row;
      const bool valid = grow < w.rows;
      const int qi = grow / G, g = grow % G;
      const int lim = !valid ? -1 : (p.causal ? w.p0 + qi : w.kend - 1);  // last key this row may see
      {
        // Q row -> shared memory (K-major, 128-byte swizzle); padding rows are
        // zero.  The previous unit's S MMAs have completed (its last P.V did).
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.q) +
                                                          ((size_t)(w.qs + qi) * p.q_heads + w.h * G + g) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(qt + (c >> 3) * L::QHALF + row * 128 + (((c & 7) ^ (row & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_QFULL + x));
      }
      griddep_wait();  // before writing outputs (a no-op after the first unit)

      float m = -INFINITY, l = 0.f;  // running (possibly stale) max in log2 units, row sum
      for (int j = 0; j < w.ntiles; ++j, ++gt) {
        const int sb = gt & 1;  // S buffer of this tile
        const uint32_t scol = scol0 + sb * kKeys;
        // each warp waits on its own (S is double-buffered: no group meeting per tile)
        if (!__all_sync(kAll, mbar_wait(bar(B_SFULL + 2 * x + sb), (gt >> 1) & 1))) { ok = false; break; }
        tc_fence_after();
        const int ts = w.k0 + j * kKeys;
        const int nvis = lim - ts + 1;  // keys of this tile the row may see (<= 0: none)
        const bool all_full = __all_sync(0xffffffffu, nvis >= kKeys);

        // the whole S row in registers: one TMEM round trip
        float sv[kKeys];
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c) tmem_ld32(scol + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
        tmem_wait_ld();
        if (!all_full) {
#pragma unroll
          for (int e = 0; e < kKeys; ++e) sv[e] = e < nvis ? sv[e] : -INFINITY;
        }
        // row maximum: four independent chains of three-input max
        float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;
#pragma unroll
        for (int e = 0; e < kKeys; e += 8) {
          ma = fmax3(ma, sv[e], sv[e + 1]);
          mb = fmax3(mb, sv[e + 2], sv[e + 3]);
          mc = fmax3(mc, sv[e + 4], sv[e + 5]);
          md = fmax3(md, sv[e + 6], sv[e + 7]);
        }
        const float mx = fmax3(ma, mb, fmaxf(mc, md)) * sl2;
        const bool raise = mx > m + kRescale;  // also the first finite max (m = -inf)
        // O and l are rescaled by 2^(m_old - m_new) when the maximum is raised
        const float alpha = (raise && m != -INFINITY) ? ex2_approx(m - mx) : 1.f;
        const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
        if (raise) {
          l = (m == -INFINITY) ? 0.f : l * alpha;
          m = mx;
        }
        const float neg_m = m == -INFINITY ? 0.f : -m;

        // P = 2^(s*sl2 - m) (masked keys hold -inf: p = 0), written over the
        // first kKeys/2 columns of this tile's S buffer, 32 keys at a time;
        // the sum runs in four packed-pair chains
        float sx[4] = {0.f, 0.f, 0.f, 0.f}, sy[4] = {0.f, 0.f, 0.f, 0.f};
        const int nvalid = min(kKeys, w.kend - ts);
        bool vok = true;
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float a0, a1;
            ffma2(a0, a1, sv[32 * c + e], sv[32 * c + e + 1], sl2, sl2, neg_m, neg_m);
            const float p0v = ex2_approx(a0), p1v = ex2_approx(a1);
            const int k = (e >> 1) & 3;
            fadd2(sx[k], sy[k], sx[k], sy[k], p0v, p1v);
            pk[e >> 1] = Elem<T>::pack(p0v, p1v);
          }
          tmem_st16u(scol + 16 * c, pk);  // keys 32c..32c+31 -> columns 16c..16c+15
        }
        if (rescale) {
          // rescale O_x in TMEM before P.V_x(j) starts (warp-collective),
          // once P.V_x(j-1) has completed (S_x(j) waited only for
          // P.V_x(j-2)); a rescale needs a finite reference, so j >= 1
          if (!mbar_wait(bar(B_OFULL + 2 * x + ((gt - 1) & 1)), ((gt - 1) >> 1) & 1)) vok = false;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            float ov[16];
            tmem_ld16(ocol + 16 * c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] *= alpha;
            tmem_st16u(ocol + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(ov));
          }
        }
        if (nvalid < kKeys) {
          // last key tile: keys past kend came from stale slots (or were
          // not loaded); zero their V rows so that p = 0 never meets
          // NaN/Inf.  Both Q tiles' softmax warps write the same zeros
          // (either P.V may run first); each P.V starts only after its own
          // group's.
          const int s = gt % kVStages;
          if (!mbar_wait(bar(B_VFULL + s), (gt / kVStages) & 1)) {
            vok = false;
          } else if (row >= nvalid && row < kKeys) {
            uint8_t* vrow = smem + L::V_OFF + s * Tile::BYTES + row * 128;
#pragma unroll
            for (int hf = 0; hf < NH; ++hf)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vrow + hf * Tile::HALF + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        // P_x(j), any rescale of O_x and any V rows past the keys are this
        // warp's share of what the Q tile's MMA warp waits for before
        // P.V_x(j); one barrier per (Q tile, S buffer), so that arrivals for
        // tile j+1 never land in tile j's phase
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + 2 * x + sb));
        if (!vok) ok = false;
        l += ((sx[0] + sy[0]) + (sx[1] + sy[1])) + ((sx[2] + sy[2]) + (sx[3] + sy[3]));
        if (!ok) break;
      }
      const bool ofull = ok && mbar_wait(bar(B_OFULL + 2 * x + ((gt - 1) & 1)), ((gt - 1) >> 1) & 1);  // the unit's last P.V_x
      ok = bar_red_and(1 + x, 128, ofull);
      if (!ok) break;
      tc_fence_after();
      if (p.causal) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                              ((size_t)(w.qs + qi) * p.q_heads + w.h * G + g) * D);
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
      } else {
        // shared-prefix partial of this key range: unnormalised o, m, l
        const size_t pr = ((size_t)qi * p.q_heads + w.h * G + g) * p.max_splits + w.z;
        float4* po = reinterpret_cast<float4*>(p.part_o + pr * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tmem_ld32(ocol + 32 * c, ov);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              po[8 * c + q] = make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
          }
        }
        if (valid) {
          p.part_m[pr] = m;
          p.part_l[pr] = l;
        }
      }
      tc_fence_before();  // O_x read out before the next unit's P.V overwrites it
    }
    if (lane == 0 && !ok) record_error(p.err, PA_DEVERR_TIMEOUT);
  }

  // ------------------------------------------------------------------ teardown
  if (warp == kMmaWarp && lane == 0) mbar_wait(bar(B_MMADONE), 0);  // both issuers' tcgen05 ops done (bounded)
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmem);
  }
}

template <int D, int BSUB, typename T>
cudaError_t launch_tc_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                         cudaStream_t stream) {
  using L = TcSmem<D, BSUB>;
  auto kern = attn_tc_kernel<D, BSUB, T>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int row_tiles = (p.max_q_len * p.group + 2 * kRows - 1) / (2 * kRows);
  const int zdim = p.causal ? p.num_reqs : (p.prefix_len + p.key_split - 1) / p.key_split;
  const long long nunits = (long long)row_tiles * p.kv_heads * zdim;
  if (nunits <= 0) return cudaSuccess;
  if (nunits > INT32_MAX) return cudaErrorInvalidValue;
  // one CTA per unit: a (row tile, head, request) grid, whose linear order is
  // the unit order; capped: a 1-D grid of max_ctas persistent CTAs
  const dim3 grid = p.max_ctas > 0 && p.max_ctas < nunits ? dim3(p.max_ctas) : dim3(row_tiles, p.kv_heads, zdim);
  return launch_pdl(kern, grid, dim3(kThreads), L::BYTES, stream, kmap, vmap, p);
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

cudaError_t launch_attn_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p, int head_dim,
                            int bsub, pa_dtype dt, cudaStream_t stream) {
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
