// Paged attention of up to 128 query rows per (request, KV head) on the
// 5th-generation tensor cores (tcgen05 + tensor memory), sm_103a, for blocks
// of >= 8 tokens.  Its use here is the speculative verify: the k+1 queries of
// a request times the heads of a GQA group (at most 128 rows) attend the
// request's context causally (query i sees tokens [0, L - k + i)), which is a
// chunked prefill of a k+1-token chunk.  A work unit is one (request, KV head)
// and walks 128-key K/V tiles gathered from the paged cache by TMA; it needs
// one TMA box per 16 tokens and half of a head dimension, whatever its row
// count, so a 32-row unit costs the gather no more than a 128-row one.
//
// Everything the MMAs touch besides K and V lives in tensor memory (512
// columns per CTA, one CTA per SM):
//
//   O   [0, D)                 fp32 accumulator, 128 rows x D
//   S0  [D, D + 128)           S = Q K^T of even key tiles (fp32)
//   S1  [D + 128, D + 256)     S of odd key tiles
//   Q   [D + 256, + D/2)       the unit's queries, two elements per column (A of S)
//   P   [.., + 64)             probabilities of one key tile, two per column (A of P.V)
//
// Because Q and P have columns of their own, S of key tile j+2 can be issued
// as soon as the softmax has read S(j) out of its buffer: it never waits for
// P.V(j).
//
// Warp roles (384 threads = 12 warps):
//   warps 0..7  softmax: warp w reads TMEM lanes 32*(w%4).. (thread = row) and
//               owns keys [64*(w/4), +64) of every key tile (half of P) and
//               dims [D/2*(w/4), +D/2) of O and Q.  Each thread loads its
//               whole S row (the row maximum needs all 128 scores), writes
//               P = 2^(s*scale*log2e - m) for its 64 keys into TMEM, and sums
//               them.  The running maximum m is raised only when a row
//               maximum exceeds it by more than 2^8 (O is then rescaled in
//               TMEM, all D columns by the warp of the low key half, before
//               either half of the tile's P.V, each of which adds to every
//               column, can start); the final O / sum uses the same m, so
//               this is exact.
//               A warp whose 32 rows are all past the unit's rows skips the
//               arithmetic and only keeps the barrier phases.  The next
//               unit's Q rows are staged in shared memory by cp.async.
//   (spread)    units of at most 32 rows (a verify of k+1 <= 32 / group
//               queries): every lane quarter holds a copy of the same rows
//               (Q is written four times; S costs the MMA the same), and
//               quarter q takes keys [32q, +32) of every tile: each thread
//               loads 32 scores instead of 128 and computes 16
//               probabilities instead of 64.  P stays zero outside the
//               quarter's window, so O of quarter q sums its keys only, with
//               its own running maximum; the epilogue merges the four
//               partial results (O = sum 2^(m_q - M) O_q / sum 2^(m_q - M)
//               l_q) through shared memory (V stages 0 and 1, idle by then:
//               the spread form runs one unit per CTA).  The first half of
//               P.V takes the low 16 keys of every window.
//   warp 8      issues S(j) = Q K_j^T into S(j % 2) (A from TMEM); owns TMEM
//   warp 9      issues O += P(j) V_j (A from TMEM), in two 64-key halves
//   warps 10,11 TMA producers of K (3-stage ring) and V (3 stages)
// (One thread issues a tcgen05.mma per ~100 clk here, so S and P.V have an
// issuing thread each.)  K is K-major and V MN-major in the canonical
// 128-byte-swizzled shared-memory layouts that the TMA boxes write.  Every
// mbarrier wait is bounded.
#include <float.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kRows = 128;  // rows per unit (M of every MMA)
constexpr int kKeys = 128;      // keys per K/V tile (N of S, K of P.V)
constexpr int kKStages = 3;
constexpr int kVStages = 3;
constexpr unsigned kAll = 0xffffffffu;
constexpr int kSoftmaxWarps = 8;
constexpr int kSWarp = 8;    // issues S = Q K^T; owns the TMEM allocation
constexpr int kPvWarp = 9;   // issues O += P V
constexpr int kKWarp = 10;   // TMA producer of K
constexpr int kVWarp = 11;   // TMA producer of V
constexpr int kThreads = 32 * 12;
constexpr uint32_t kTmem = 512;

__device__ __forceinline__ uint8_t* align1024_tc(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int D, int BSUB, bool SPREAD>
struct TcSmem {
  using Tile = KvTile<D, BSUB, kKeys>;  // D/64 halves x 128 rows x 128 B
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + kKStages * Tile::BYTES;
  // staged Q rows of the next unit; spread: two [32 rows][D] fp32 partial outputs
  static constexpr int Q_OFF = V_OFF + kVStages * Tile::BYTES;
  // row sums: [2 key halves][128 rows]; spread: maxima [4][32] and sums [4][2][32]
  static constexpr int L_OFF = Q_OFF + kRows * D * 2;
  static constexpr int BAR_OFF = L_OFF + (SPREAD ? 3 : 2) * kRows * 4;
  static constexpr int NBARS = 4 * 3 + 2 + 2 + 6;
  static constexpr int SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = SLOT_OFF + 16 + 1024;
  static_assert(BSUB * 128 >= 1024, "needs blocks of at least 8 tokens (one 8-row swizzle atom per box)");
  static_assert(BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert((kKeys / BSUB) * (D / 64) <= 32, "a producer warp issues one box per lane");
};

// barrier indices
constexpr int B_KFULL = 0;                    // [kKStages] K producer arrival (+ TMA bytes)
constexpr int B_KEMPTY = B_KFULL + kKStages;  // [kKStages] commit after S(j)
constexpr int B_VFULL = B_KEMPTY + kKStages;  // [kVStages] V producer arrival (+ TMA bytes)
constexpr int B_VEMPTY = B_VFULL + kVStages;  // [kVStages] commit after P.V(j)
constexpr int B_SFULL = B_VEMPTY + kVStages;  // [2] S buffer written (commit)
constexpr int B_SFREE = B_SFULL + 2;          // [2] S buffer read out (8 softmax warps)
constexpr int B_PLO = B_SFREE + 2;            // low key half of P in TMEM (4 warps; V rows past the keys zeroed, O rescaled)
constexpr int B_PHI = B_PLO + 1;              // high key half of P (4 warps)
constexpr int B_PVDONE = B_PHI + 1;           // P.V(j) complete (commit)
constexpr int B_QFULL = B_PVDONE + 1;         // the unit's Q in TMEM (8 warps)
constexpr int B_OFREE = B_QFULL + 1;          // the unit's O read out (8 warps)
constexpr int B_MMADONE = B_OFREE + 1;        // every MMA of the CTA complete (commit)
static_assert(B_MMADONE + 1 == 4 * 3 + 2 + 2 + 6, "barrier count");

// One work unit: the rows of one (request, KV head), at most 128: query i of
// the request's fixed_q_len queries times head g of the group, row i*G + g
// (rows past 128 of a larger request would be further units; the ABI limits
// q_len * group to 128).  Units are numbered request-major, then head.
struct TcUnit {
  int z, h, row0, r, qs, chunk, p0, k0, kend, rows, ntiles;
};

// Geometry of unit u from immutable inputs only: row (query i, head g) sees
// keys 0 .. p0 + i, p0 = context - q_len (negative for a context shorter
// than q_len: its first queries see no key).  false: the request's context
// length is out of range (the unit is skipped).
__device__ __forceinline__ bool tc_unit(const PrefillParams& p, int u, int row_tiles, TcUnit& w) {
  const int per_z = row_tiles * p.kv_heads;
  w.z = u / per_z;
  const int rem = u - w.z * per_z;
  w.h = rem / row_tiles;
  w.row0 = (row_tiles - 1 - (rem - w.h * row_tiles)) * kRows;
  w.ntiles = 0;
  const int G = p.group;
  w.r = w.z;
  w.qs = w.r * p.fixed_q_len;
  w.chunk = p.fixed_q_len;
  const int ctx = __ldg(p.lens + w.r);
  w.p0 = ctx - w.chunk;
  if (ctx < 0 || ctx > p.maxblk * p.block_size) return false;
  w.k0 = 0;
  w.rows = w.chunk * G;
  if (w.row0 >= w.rows) return true;
  const int last_row = min(w.row0 + kRows, w.rows) - 1;
  w.kend = w.p0 + last_row / G + 1;
  if (w.kend <= 0) return true;  // no row sees a key (ntiles = 0)
  w.ntiles = (w.kend - w.k0 + kKeys - 1) / kKeys;
  return true;
}

template <int D, int BSUB, typename T, bool SPREAD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tile_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const PrefillParams p) {
  using L = TcSmem<D, BSUB, SPREAD>;
  using Tile = typename L::Tile;
  constexpr int NH = D / 64;
  constexpr int KSTEPS = D / 16;      // S = Q K^T: K dimension = head_dim
  constexpr int SUBS = kKeys / BSUB;  // boxes per half per tile
  constexpr int DH = D / 2;           // dims of O (and Q) per softmax warp
  constexpr uint32_t O_COL = 0;
  constexpr uint32_t S_COL = D;                  // S0, S1: kKeys columns each
  constexpr uint32_t Q_COL = D + 2 * kKeys;      // D/2 columns
  constexpr uint32_t P_COL = Q_COL + D / 2;      // kKeys/2 columns
  static_assert(P_COL + kKeys / 2 <= kTmem, "tensor memory columns");
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
  const int row_tiles = (p.max_q_len * G + kRows - 1) / kRows;
  const int nunits = row_tiles * p.kv_heads * p.num_reqs;
  const int cta0 = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int nctas = gridDim.x * gridDim.y * gridDim.z;
  // the spread form keeps its epilogue's partial outputs in V stages that
  // the next unit's loads would overwrite: it takes one unit per CTA (the
  // host launches it so)
  if (SPREAD && nctas < nunits) {
    if (threadIdx.x == 0) record_error(p.err, PA_DEVERR_QUERY_RANGE);
    return;
  }

  // the first unit >= u (in this CTA's stride) that has key tiles, or nunits
  auto next_unit = [&](int u, TcUnit& w, bool report) -> int {
    for (; u < nunits; u += nctas) {
      if (!tc_unit(p, u, row_tiles, w)) {
        if (report) {
          griddep_wait();
          if (lane == 0) record_error(p.err, PA_DEVERR_QUERY_RANGE);
        }
        continue;
      }
      if (w.ntiles > 0) return u;
    }
    return nunits;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KEMPTY + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VEMPTY + i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_SFULL + b), 1);
      mbar_init(bar(B_SFREE + b), kSoftmaxWarps);
    }
    mbar_init(bar(B_PLO), kSoftmaxWarps / 2);
    mbar_init(bar(B_PHI), kSoftmaxWarps / 2);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_QFULL), kSoftmaxWarps);
    mbar_init(bar(B_OFREE), kSoftmaxWarps);
    mbar_init(bar(B_MMADONE), 2);  // both issuers' last commits
    fence_mbar_init();
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }
  if (warp == kSWarp) {
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
    const uint64_t pol = policy_evict_first();  // a unit's K/V is read once: streamed
    const int nst = isv ? kVStages : kKStages;
    int gt = 0;  // K/V tiles issued by this CTA (ring position and phase)
    bool failed = false;
    griddep_wait();  // the cache (this step's reshape_and_cache) comes from the kernel before
    TcUnit w;
    for (int u = next_unit(cta0, w, false); u < nunits && !failed; u = next_unit(u + nctas, w, false)) {
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
  } else if (warp == kSWarp) {
    // ---------------------------------------------------------------- S issuer
    // S(gs) = Q K(gs)^T into buffer gs % 2, up to two key tiles ahead of the
    // softmax: the buffer is free once the softmax has read S(gs - 2); a
    // unit's first S needs the unit's Q in TMEM.  (An MMA issue costs its
    // thread about 100 clk, so S and P.V have an issuing warp each.)  The
    // whole warp runs the loop with voted waits and one elected lane issues
    // (warp-uniform descriptors).
    {
      bool ok = true;
      const uint32_t kbase = smem_u32(smem + L::K_OFF);
      int gs = 0, ns = 0;  // key tiles and units of this CTA's stream
      TcUnit w;
      for (int u = next_unit(cta0, w, true); ok && u < nunits; u = next_unit(u + nctas, w, true), ++ns) {
        if (!__all_sync(kAll, mbar_wait(bar(B_QFULL), ns & 1))) { ok = false; break; }
        for (int j = 0; j < w.ntiles; ++j, ++gs) {
          const int b = gs & 1, sk = gs % kKStages;
          if (!__all_sync(kAll, (gs < 2 || mbar_wait(bar(B_SFREE + b), ((gs - 2) >> 1) & 1)) &&
                                    mbar_wait(bar(B_KFULL + sk), (gs / kKStages) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb = kbase + sk * Tile::BYTES;
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            const uint64_t bd = smem_desc_sw128(kb + (ks >> 2) * Tile::HALF + (ks & 3) * 32, 16, 1024);
            tc_mma_f16_ts_warp(tmem + S_COL + b * kKeys, tmem + Q_COL + ks * 8, bd, IDESC_S, ks > 0 ? 1u : 0u);
          }
          tc_commit_warp(bar(B_SFULL + b));
          tc_commit_warp(bar(B_KEMPTY + sk));  // K(gs) read
        }
      }
      if (!ok && lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
      tc_commit_warp(bar(B_MMADONE));
    }
  } else if (warp == kPvWarp) {
    // ---------------------------------------------------------------- P.V issuer
    // O += P(gp) V(gp) in two 64-key halves, each once its half of P is in
    // TMEM; the unit's first P.V overwrites O, which the previous unit's
    // epilogue must have read out.  Warp-converged like the S issuer.
    {
      bool ok = true;
      const uint32_t vbase = smem_u32(smem + L::V_OFF);
      int gp = 0, np = 0;  // key tiles and units of this CTA's stream
      TcUnit w;
      for (int u = next_unit(cta0, w, false); ok && u < nunits; u = next_unit(u + nctas, w, false), ++np) {
        if (np > 0 && !__all_sync(kAll, mbar_wait(bar(B_OFREE), (np - 1) & 1))) { ok = false; break; }
        for (int j = 0; j < w.ntiles; ++j, ++gp) {
          const int sv = gp % kVStages;
          const uint32_t vb = vbase + sv * Tile::BYTES;
          if (!__all_sync(kAll, mbar_wait(bar(B_VFULL + sv), (gp / kVStages) & 1))) { ok = false; break; }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if (!__all_sync(kAll, mbar_wait(bar(hh ? B_PHI : B_PLO), gp & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              // A = P[128 rows x keys 16kk..16kk+15] in TMEM (8 columns); B = V rows 16kk.., MN-major.
              // Half hh: keys 64hh.. (spread: the 16-key steps of key half hh of every window)
              const int kk = SPREAD ? 2 * k4 + hh : hh * 4 + k4;
              const uint64_t bd = smem_desc_sw128(vb + kk * 2048, Tile::HALF, 1024);
              tc_mma_f16_ts_warp(tmem + O_COL, tmem + P_COL + kk * 8, bd, IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
            }
          }
          if (!ok) break;
          tc_commit_warp(bar(B_PVDONE));
          tc_commit_warp(bar(B_VEMPTY + sv));  // V(gp) read
        }
      }
      if (!ok && lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
      tc_commit_warp(bar(B_MMADONE));
    }
  } else if (warp < kSoftmaxWarps) {
    // ---------------------------------------------------------------- softmax
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int kh = warp >> 2;      // key half of P (of the quarter's window when spread), dim half of O and Q
    // the unit row this thread owns: its TMEM lane, or (spread) the same 32
    // rows in every lane quarter
    const int row = SPREAD ? lane : quarter * 32 + lane;
    const int vrow = quarter * 32 + lane;  // V row this thread zeroes past the keys
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    constexpr float kRescale = 8.f;
    // S columns the warp reads: the whole tile, or (spread) its quarter's 32-key window
    constexpr int KS = SPREAD ? 32 : kKeys;
    const int s_key0 = SPREAD ? 32 * quarter : 0;
    // keys of P the warp writes, two per TMEM column
    constexpr int KP = SPREAD ? 16 : kKeys / 2;
    const int p_key0 = SPREAD ? 32 * quarter + 16 * kh : 64 * kh;
    const uint32_t qst = smem_u32(smem + L::Q_OFF) + row * (D * 2);  // this row's staged Q (not spread)
    float* lsum = reinterpret_cast<float*>(smem + L::L_OFF);
    uint4 qreg[SPREAD ? DH / 8 : 1];  // spread: this thread's half of its Q row for the next unit

    // this thread's half of its Q row for unit w: into registers (spread), or
    // into shared memory by cp.async (16-byte chunks, XOR-swizzled by row);
    // rows past the unit are zero
    auto stage_q = [&](const TcUnit& w) {
      const int grow = w.row0 + row;
      const bool valid = grow < w.rows;
      const int qi = grow / G, g = grow % G;
      const char* src = reinterpret_cast<const char*>(p.q) +
                        (valid ? ((size_t)(w.qs + qi) * p.q_heads + w.h * G + g) * D * sizeof(T) : 0);
      if constexpr (SPREAD) {
#pragma unroll
        for (int c = 0; c < DH / 8; ++c)
          qreg[c] = valid ? __ldg(reinterpret_cast<const uint4*>(src) + kh * (DH / 8) + c) : make_uint4(0, 0, 0, 0);
      } else {
#pragma unroll
        for (int c = kh * (D / 16); c < (kh + 1) * (D / 16); ++c)
          cp_async16(qst + ((c ^ (row & 7)) << 4), src + c * 16, valid ? 16u : 0u);
        cp_async_commit();
      }
    };
    // the staged half row -> Q columns of TMEM (two elements per column)
    auto q_to_tmem = [&]() {
      if constexpr (!SPREAD) cp_async_wait_all();
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 x;
          if constexpr (SPREAD) {
            x = qreg[cc * 4 + i];
          } else {
            const int c = kh * (D / 16) + cc * 4 + i;
            x = *reinterpret_cast<const uint4*>(smem + L::Q_OFF + row * (D * 2) + ((c ^ (row & 7)) << 4));
          }
          v[4 * i] = x.x, v[4 * i + 1] = x.y, v[4 * i + 2] = x.z, v[4 * i + 3] = x.w;
        }
        tmem_st16u(tl + Q_COL + kh * (D / 4) + cc * 16, v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QFULL));
    };

    if constexpr (SPREAD) {
      // P columns of the other quarters' windows stay zero in this lane
      // quarter for the whole kernel.  Column c holds keys of window c / 16
      // and key half (c / 8) % 2: exactly one warp ever writes it.
      const uint32_t zero8[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        if (qq != quarter) tmem_st8u(tl + P_COL + 16 * qq + 8 * kh, zero8);
      tmem_wait_st();  // fenced before this warp's first arrival on a P barrier
    }

    // units whose rows see no key at all (a verify request shorter than its
    // queries) are skipped by every role; their rows are written as zeros here
    // (spread: by the first lane quarter)
    {
      TcUnit z;
      for (int uz = cta0; uz < nunits; uz += nctas) {
        if (!tc_unit(p, uz, row_tiles, z) || z.ntiles > 0 || z.row0 >= z.rows) continue;
        griddep_wait();
        const int grow = z.row0 + row;
        if (grow < z.rows && (!SPREAD || quarter == 0)) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                                ((size_t)(z.qs + grow / G) * p.q_heads + z.h * G + grow % G) * D + kh * DH);
#pragma unroll
          for (int c = 0; c < DH / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
      }
    }

    bool ok = true;
    int gt = 0;  // key tiles processed by this CTA
    TcUnit w, wn;
    int u = next_unit(cta0, w, false);
    int un = nunits;
    if (u < nunits) {
      stage_q(w);
      q_to_tmem();
      un = next_unit(u + nctas, wn, false);
      if (un < nunits) stage_q(wn);  // in flight during this unit
    }
    while (ok && u < nunits) {
      griddep_wait();  // before writing outputs (a no-op after the first unit)
      const int grow = w.row0 + row;
      const bool valid = grow < w.rows;
      const int qi = grow / G, g = grow % G;
      const int lim = !valid ? -1 : w.p0 + qi;  // last key this row may see
      const bool wvalid = __any_sync(kAll, valid);  // else: only keep the barrier phases
      float m = -INFINITY, l = 0.f;  // running (possibly stale) max in log2 units, sum of this warp's keys
      for (int j = 0; j < w.ntiles; ++j, ++gt) {
        const int b = gt & 1;
        ok = __all_sync(kAll, mbar_wait(bar(B_SFULL + b), (gt >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        const int ts = w.k0 + j * kKeys;
        const int nvis = lim - ts + 1 - s_key0;  // keys of this warp's S window the row may see (<= 0: none)
        // rows past the unit (whose output is never read) do not force the masking pass
        const bool all_full = __all_sync(kAll, nvis >= KS || !valid);

        // the warp's S window in registers (one TMEM round trip); then the
        // buffer may take S(gt + 2)
        auto max32 = [](const float* x) {
          float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;  // four chains of 3-input max
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            ma = fmax3(ma, x[e], x[e + 1]);
            mb = fmax3(mb, x[e + 2], x[e + 3]);
            mc = fmax3(mc, x[e + 4], x[e + 5]);
            md = fmax3(md, x[e + 6], x[e + 7]);
          }
          return fmax3(ma, mb, fmaxf(mc, md));
        };
        auto max64 = [](const float* x) {
          float ma = -INFINITY, mb = -INFINITY, mc = -INFINITY, md = -INFINITY;
#pragma unroll
          for (int e = 0; e < 64; e += 8) {
            ma = fmax3(ma, x[e], x[e + 1]);
            mb = fmax3(mb, x[e + 2], x[e + 3]);
            mc = fmax3(mc, x[e + 4], x[e + 5]);
            md = fmax3(md, x[e + 6], x[e + 7]);
          }
          return fmax3(ma, mb, fmaxf(mc, md));
        };
        float sv[KS];
#pragma unroll
        for (int c = 0; c < KS / 32; ++c)
          tmem_ld32(tl + S_COL + b * kKeys + s_key0 + 32 * c, *reinterpret_cast<float(*)[32]>(&sv[32 * c]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SFREE + b));
        if (j == w.ntiles - 1 && un < nunits) q_to_tmem();  // the unit's last S done: the next unit's Q
        const int nvalid = min(kKeys, w.kend - ts);
        if (!wvalid) {
          // rows all past the unit: no P (its rows of O are never read), but
          // the zeroing of V rows past the keys is this warp's share
          if (kh == 0 && nvalid < kKeys) {
            const int s = gt % kVStages;
            ok = __all_sync(kAll, mbar_wait(bar(B_VFULL + s), (gt / kVStages) & 1));
            if (!ok) break;
            if (vrow >= nvalid) {
              uint8_t* vt = smem + L::V_OFF + s * Tile::BYTES;
#pragma unroll
              for (int hf = 0; hf < NH; ++hf)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  *reinterpret_cast<uint4*>(vt + Tile::line(hf, vrow) + c * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          // P(gt)'s barrier counts one arrival per warp and tile: like every
          // warp, arrive for gt only once P.V(gt - 1) is complete, so that no
          // arrival lands in the previous tile's phase
          if (gt > 0) {
            ok = __all_sync(kAll, mbar_wait(bar(B_PVDONE), (gt - 1) & 1));
            if (!ok) break;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kh ? B_PHI : B_PLO));
          continue;
        }

        if (!all_full) {
#pragma unroll
          for (int e = 0; e < KS; ++e) sv[e] = e < nvis ? sv[e] : -INFINITY;
        }
        float mraw;
        if constexpr (SPREAD) mraw = max32(sv);
        else mraw = fmaxf(max64(sv), max64(sv + 64));
        const float mx = mraw * sl2;
        const bool raise = mx > m + kRescale;  // also the first finite max (m = -inf)
        // O and l are rescaled by 2^(m_old - m_new) when the maximum is raised
        const float alpha = (raise && m != -INFINITY) ? ex2_approx(m - mx) : 1.f;
        const bool rescale = __any_sync(kAll, alpha != 1.f);
        if (raise) {
          l = (m == -INFINITY) ? 0.f : l * alpha;
          m = mx;
        }
        const float neg_m = m == -INFINITY ? 0.f : -m;

        // P = 2^(s*sl2 - m) for this warp's keys (masked keys hold -inf:
        // p = 0); the sum runs in four packed-pair chains
        float sx[4] = {0.f, 0.f, 0.f, 0.f}, sy[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[KP / 2];
#pragma unroll
        for (int e = 0; e < KP; e += 2) {
          float a0, a1;
          // selects with constant indices (a runtime index would put sv in local memory)
          const float s0 = kh ? sv[KP + e] : sv[e], s1 = kh ? sv[KP + e + 1] : sv[e + 1];
          ffma2(a0, a1, s0, s1, sl2, sl2, neg_m, neg_m);
          const float p0v = ex2_approx(a0), p1v = ex2_approx(a1);
          const int k = (e >> 1) & 3;
          fadd2(sx[k], sy[k], sx[k], sy[k], p0v, p1v);
          pk[e >> 1] = Elem<T>::pack(p0v, p1v);
        }
        // P(gt) overwrites P(gt - 1) and a rescale touches O: both once
        // P.V(gt - 1) has completed
        if (gt > 0) {
          ok = __all_sync(kAll, mbar_wait(bar(B_PVDONE), (gt - 1) & 1));
          if (!ok) break;
          tc_fence_after();
        }
        if (kh == 0 && rescale) {
          // all of the row's O, by the warp whose half of P the first half
          // of P.V(gt) waits for: each half of P.V adds to every column of O
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            float ov[16];
            tmem_ld16(tl + O_COL + 16 * c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] *= alpha;
            tmem_st16u(tl + O_COL + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(ov));
          }
        }
        if (kh == 0 && nvalid < kKeys) {
          // last key tile: keys past kend came from stale slots (or were not
          // loaded); zero their V rows so that p = 0 never meets NaN/Inf
          const int s = gt % kVStages;
          ok = __all_sync(kAll, mbar_wait(bar(B_VFULL + s), (gt / kVStages) & 1));
          if (!ok) break;
          if (vrow >= nvalid) {
            uint8_t* vt = smem + L::V_OFF + s * Tile::BYTES;
#pragma unroll
            for (int hf = 0; hf < NH; ++hf)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vt + Tile::line(hf, vrow) + c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        if constexpr (SPREAD) {
          tmem_st8u(tl + P_COL + p_key0 / 2, pk);
        } else {
          tmem_st16u(tl + P_COL + p_key0 / 2, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
          tmem_st16u(tl + P_COL + p_key0 / 2 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kh ? B_PHI : B_PLO));
        l += ((sx[0] + sy[0]) + (sx[1] + sy[1])) + ((sx[2] + sy[2]) + (sx[3] + sy[3]));
      }
      // epilogue: the unit's last P.V has completed
      if (ok) ok = __all_sync(kAll, mbar_wait(bar(B_PVDONE), (gt - 1) & 1));
      tc_fence_after();
      if constexpr (SPREAD) {
        // The four lane quarters hold partial results of the same rows over
        // disjoint keys, each relative to its own running maximum m_q:
        //   O = sum_q 2^(m_q - M) O_q / sum_q 2^(m_q - M) l_q,  M = max_q m_q.
        // Every warp puts its half of O_q (fp32) and its (m_q, l) into shared
        // memory (the partial outputs in V stages 0 and 1, idle by now: a
        // spread CTA has one unit and loads no further tile); after one AND
        // vote of all 8 warps, which every exit of the unit passes through,
        // the 256 threads merge and write 32 rows x D: thread t takes row
        // t / 8 and the 16-byte chunks t % 8, t % 8 + 8, ... of it (8 threads
        // per row: conflict-free shared-memory reads, 64-byte runs of output).
        float* mq = lsum;           // [4 quarters][32 rows] running maxima
        float* lq = lsum + 4 * 32;  // [4 quarters][2 key halves][32 rows] sums
        if (kh == 0) mq[quarter * 32 + lane] = m;
        lq[(quarter * 2 + kh) * 32 + lane] = l;
        // 16-byte chunk ch of row r of quarter qq's partial, XOR-swizzled by row
        auto part = [&](int qq, int r, int ch) {
          return reinterpret_cast<float4*>(smem + L::V_OFF + qq * (32 * D * 4) + r * (D * 4)) + (ch ^ (r & 7));
        };
        if (ok) {
#pragma unroll
          for (int c = 0; c < DH / 32; ++c) {
            float ov[32];
            tmem_ld32(tl + O_COL + kh * DH + 32 * c, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *part(quarter, lane, kh * (DH / 4) + 8 * c + i) =
                  make_float4(ov[4 * i], ov[4 * i + 1], ov[4 * i + 2], ov[4 * i + 3]);
          }
        }
        if (!bar_red_and(5, 32 * kSoftmaxWarps, ok)) {
          ok = false;
          break;
        }
        const int t = threadIdx.x;  // 0..255: the softmax warps
        const int r = t >> 3, c0 = t & 7;
        if (w.row0 + r < w.rows) {
          float f[4], mmax = -INFINITY, lt = 0.f;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) mmax = fmaxf(mmax, mq[qq * 32 + r]);
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const float mv = mq[qq * 32 + r];
            f[qq] = mv == -INFINITY ? 0.f : ex2_approx(mv - mmax);
            lt += f[qq] * (lq[(qq * 2) * 32 + r] + lq[(qq * 2 + 1) * 32 + r]);
          }
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
          const int rr = w.row0 + r;
          T* orow = reinterpret_cast<T*>(p.out) + ((size_t)(w.qs + rr / G) * p.q_heads + w.h * G + rr % G) * D;
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            const int ch = c0 + 8 * i;  // 16-byte chunk of the fp32 row = 4 output elements
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const float4 x = *part(qq, r, ch);
              a.x += f[qq] * x.x, a.y += f[qq] * x.y, a.z += f[qq] * x.z, a.w += f[qq] * x.w;
            }
            *reinterpret_cast<uint2*>(orow + 4 * ch) =
                make_uint2(Elem<T>::pack(a.x * inv, a.y * inv), Elem<T>::pack(a.z * inv, a.w * inv));
          }
        }
      } else {
        // the row's sum over both key halves is added in key-half order; the
        // two warps of this lane quarter meet twice (written, then read).  The
        // first meeting is an AND vote that every exit of the unit passes
        // through, so that a warp that gave up on a wait never leaves its
        // partner at a barrier.
        lsum[kh * kRows + row] = l;
        if (!bar_red_and(1 + quarter, 64, ok)) {
          ok = false;
          break;
        }
        const float lt = lsum[row] + lsum[kRows + row];
        asm volatile("bar.sync %0, %1;\n" ::"r"(1 + quarter), "r"(64) : "memory");
        if (wvalid) {
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<T*>(p.out) +
                                                ((size_t)(w.qs + qi) * p.q_heads + w.h * G + g) * D + kh * DH);
#pragma unroll
          for (int c = 0; c < DH / 32; ++c) {
            float ov[32];
            tmem_ld32(tl + O_COL + kh * DH + 32 * c, ov);  // warp-collective: every lane loads, valid rows store
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
        }
      }
      tc_fence_before();  // O read out before the next unit's first P.V overwrites it
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OFREE));
      u = un;
      w = wn;
      if (u < nunits) {
        un = next_unit(u + nctas, wn, false);
        if (un < nunits) stage_q(wn);
      }
    }
    if (!ok && lane == 0) record_error(p.err, PA_DEVERR_TIMEOUT);
    if constexpr (!SPREAD) cp_async_wait_all();  // no staging copy still in flight at exit
  }

  // ------------------------------------------------------------------ teardown
  if (warp == kSWarp && lane == 0) mbar_wait(bar(B_MMADONE), 0);  // every MMA of the CTA done (bounded)
  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmem);
  }
}

template <int D, int BSUB, typename T, bool SPREAD>
cudaError_t launch_tc_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p,
                         cudaStream_t stream) {
  using L = TcSmem<D, BSUB, SPREAD>;
  auto kern = attn_tile_kernel<D, BSUB, T, SPREAD>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // every request has fixed_q_len queries, and their rows fit one unit
  if (p.fixed_q_len <= 0 || p.max_q_len != p.fixed_q_len || p.fixed_q_len * p.group > kRows)
    return cudaErrorInvalidValue;
  const int row_tiles = (p.max_q_len * p.group + kRows - 1) / kRows;
  const int zdim = p.num_reqs;
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
  // units of at most 32 rows, one per CTA: the rows are copied into every
  // lane quarter and the softmax of a key tile is spread over all 8 softmax
  // warps
  const bool spread = p.fixed_q_len > 0 && p.fixed_q_len * p.group <= 32 &&
                      (p.max_ctas <= 0 || (long long)p.max_ctas >= (long long)p.kv_heads * p.num_reqs);
  switch (bsub) {
    case 8: return spread ? launch_tc_t<D, 8, T, true>(kmap, vmap, p, stream)
                          : launch_tc_t<D, 8, T, false>(kmap, vmap, p, stream);
    case 16: return spread ? launch_tc_t<D, 16, T, true>(kmap, vmap, p, stream)
                           : launch_tc_t<D, 16, T, false>(kmap, vmap, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attn_tile(const CUtensorMap& kmap, const CUtensorMap& vmap, const PrefillParams& p, int head_dim,
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
