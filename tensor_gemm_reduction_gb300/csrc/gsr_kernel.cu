// gsr_kernel.cu -- the shard-reduction GEMM kernel for GB300 (sm_103a).
//
// One persistent, warp-specialised kernel serves all three modes of the fused
// projection (vLLM PR #53053 summary "Extend GEMM-RS to GEMM-AR",
// implementation breakdown step 1 and key source snippets: one kernel, RS and
// AR differing only in where the reduced rows go; PR #54151 "[Kimi-K3] AG-GEMM
// for Sequence Parallelism", Purpose: GEMM over gathered activation shards):
//
//   warp 0      TMA producer (the whole warp walks the schedule; one elected
//               lane issues each copy): for each work unit, walks its k-blocks; in AR/RS
//               mode a k-block belongs to one K-shard and is fetched through
//               that shard's descriptors (X_r, W_r) straight from the shard's
//               own allocation; in AG mode the unit's M-shard descriptor A_r
//               and the single W descriptor are used. No operand is copied or
//               padded: rows or columns past a shard's extent are zero-filled
//               by the TMA unit.
//   warp 1      MMA issuer: the whole warp walks the schedule with warp-uniform
//               values and one elected lane issues tcgen05.mma (kind::f16, bf16
//               in, fp32 accumulate) into a TMEM accumulator. In AR/RS mode the
//               accumulator runs across every shard's k-blocks, so the
//               cross-shard sum happens inside the tensor-core accumulator.
//               Two accumulators (2 x BN TMEM columns) let the epilogue of one
//               tile overlap the main loop of the next.
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, bf16 round-to-nearest-
//               even, 16-byte stores routed to Y (AR), to the owning shard's
//               Y_s (RS: global row m goes to shard m / rps), or to the shard's
//               row range of Y (AG). With split-K, each piece writes an fp32
//               partial tile to the workspace and bumps a per-tile counter; the
//               last piece to arrive sums the pieces in ascending piece order
//               (independent of arrival order) and stores, then resets the
//               counter to zero, so no flag reset or entry barrier is needed
//               between calls (PR #53053 summary, motivation).
//
// Every wait is bounded by %globaltimer; on expiry the kernel records a
// timeout code in the workspace status word, lets its in-flight copies and
// MMAs land, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "gsr_device.cuh"
#include "gsr_params.h"

namespace gsr {
namespace {

// ------------------------------------------------------------ scheduling

struct Unit {
  int tile;       // output tile index (also the split-K counter index)
  int piece;      // which piece of the tile's k range (k order)
  int npieces;    // pieces the tile is cut into (1 = whole tile)
  int slot0;      // partial slot of the tile's piece 0 (pieces are consecutive)
  int n0;         // first output column of the tile
  int m0;         // first row of THIS CTA's 128 rows in its A operand: AR/RS
                  // global, AG local to the CTA's shard
  int shard;      // AG: M-shard of this CTA's rows (-1: the idle half of an odd
                  // last pair tile, which reads zeros and stores nothing); with
                  // 64-row granules, of its first 64 rows (see next_granule)
  int kb_begin;   // k-blocks [kb_begin, kb_end) of this piece
  int kb_end;
};

// AG: the shard and first shard row of row granule g (granules are numbered
// over all shards, each inside one shard); shard -1 past the last row. Called
// by whole warps (`mt_begins` holds shard_mt_begin[lane]).
__device__ __forceinline__ void locate_granule(const Params& p, int mt_begins, int g, int& shard,
                                               int& m0) {
  if (g >= p.ag_halves) {
    shard = -1;
    m0 = 0;
    return;
  }
  int r = 0;
  while (r + 1 < p.R && __shfl_sync(0xffffffffu, mt_begins, r + 1) <= g) ++r;
  shard = r;
  m0 = (g - __shfl_sync(0xffffffffu, mt_begins, r)) * p.ag_gran;
}

// AG with 64-row granules: the granule after (shard, m0), i.e. the second half
// of a CTA's 128 rows, derived where it is used rather than carried in every
// unit (registers). Called by whole warps.
__device__ __forceinline__ void next_granule(const Params& p, int mt_begins, int shard, int m0,
                                             int& shard_b, int& m0b) {
  if (shard < 0) {
    shard_b = -1;
    m0b = 0;
    return;
  }
  const int g = __shfl_sync(0xffffffffu, mt_begins, shard) + m0 / p.ag_gran + 1;
  locate_granule(p, mt_begins, g, shard_b, m0b);
}

// Position of the tile in the output (raster order) and its shard. Called by
// whole warps: `mt_begins` holds shard_mt_begin[lane] in each lane (AG), read
// with shuffles rather than dynamically indexed kernel-parameter loads, which
// are slow on the set-up path of every unit.
template <int BN, int CG>
__device__ __forceinline__ void place_tile(const Params& p, Unit& t, uint32_t rank, int mt_begins) {
  // Raster: groups of group_m m-tiles; inside a group the m index runs fastest,
  // so CTAs working at the same time share W (B) panels and A rows in L2. With
  // group_n > 0 the roles swap: groups of group_n n-tiles, n fastest inside, so
  // a group's W panels serve every wave of the group.
  int mt, nt;
  if (p.group_n > 0) {
    const int span = p.group_n * p.m_tiles;
    const int g = t.tile / span;
    const int first_n = g * p.group_n;
    const int gn = min(p.n_tiles - first_n, p.group_n);
    const int in_g = t.tile - g * span;
    nt = first_n + in_g % gn;
    mt = in_g / gn;
  } else {
    const int span = p.group_m * p.n_tiles;
    const int g = t.tile / span;
    const int first_m = g * p.group_m;
    const int gm = min(p.m_tiles - first_m, p.group_m);
    const int in_g = t.tile - g * span;
    mt = first_m + in_g % gm;
    nt = in_g / gm;
  }
  t.n0 = nt * BN;
  // This CTA's 128 rows: half-tile h. AG rows come in granules numbered over
  // all shards, each inside one shard: one 128-row granule per CTA tile, or
  // two 64-row granules (where shards are multiples of 64 but not of 128 rows,
  // e.g. 448) that may come from neighbouring shards. Either way the halves of
  // a pair tile may too, and no rows are wasted on shard boundaries.
  const int h = mt * CG + static_cast<int>(rank);
  if (p.mode == kModeAG) {
    locate_granule(p, mt_begins, p.ag_gran == BM ? h : 2 * h, t.shard, t.m0);
  } else {
    t.shard = 0;
    t.m0 = h * BM;
  }
}

// Per-worker walk over the schedule; every role of a CTA walks it identically.
// Stream-K positions are 32-bit: the host keeps (sk_iters + 1) * (G + 1) below
// 2^32 (64-bit divisions cost about a microsecond on the set-up path).
struct Sched {
  int w;              // this worker (CTA, or CTA pair)
  int G;              // workers
  int next;           // uniform: next unit; stream-K: next whole tile
  uint32_t it;        // stream-K: next k-block of this worker's range
  uint32_t it_end;
  int mt_begins;      // AG: shard_mt_begin[lane] (lanes 0..kMaxShards)
};

template <int CG>
__device__ __forceinline__ Sched sched_begin(const Params& p) {
  Sched s;
  s.w = static_cast<int>(blockIdx.x) / CG;
  s.G = static_cast<int>(gridDim.x) / CG;
  s.next = s.w;
  if (p.sched == kSchedSplitTail) {
    // One piece of the tail for each of the first (tail tiles x splits) workers.
    const int pieces = (p.tiles - p.dp_tiles) * p.splits;
    s.it = s.w < pieces ? static_cast<uint32_t>(s.w) : 0u;
    s.it_end = s.w < pieces ? s.it + 1u : 0u;
  } else {
    const uint32_t I = static_cast<uint32_t>(p.sk_iters), G = static_cast<uint32_t>(s.G);
    s.it = static_cast<uint32_t>(s.w) * I / G;
    s.it_end = static_cast<uint32_t>(s.w + 1) * I / G;
  }
  const int lane = static_cast<int>(threadIdx.x) & 31;
  s.mt_begins = p.shard_mt_begin[lane <= kMaxShards ? lane : kMaxShards];
  return s;
}

// The worker whose stream-K range holds k-block `it` (ranges are
// [w*I/G, (w+1)*I/G), every one non-empty because I >= G).
__device__ __forceinline__ int sk_worker_of(uint32_t it, uint32_t I, uint32_t G) {
  return static_cast<int>(((it + 1) * G + I - 1) / I) - 1;
}

template <int BN, int CG>
__device__ __forceinline__ bool sched_next(const Params& p, Sched& s, Unit& t, uint32_t rank) {
  if (p.sched == kSchedUniform) {
    if (s.next >= p.units) return false;
    const int u = s.next;
    s.next += s.G;
    t.tile = u / p.splits;
    t.piece = u - t.tile * p.splits;
    t.npieces = p.splits;
    t.slot0 = t.tile * p.splits;
    t.kb_begin = t.piece * p.kb_total / p.splits;
    t.kb_end = (t.piece + 1) * p.kb_total / p.splits;
    place_tile<BN, CG>(p, t, rank, s.mt_begins);
    return true;
  }
  if (p.sched == kSchedSplitTail && s.it < s.it_end) {
    // This worker's piece of the tail, first: piece u / tail of tile
    // dp + u % tail, so the workers holding piece j of the tail tiles run side
    // by side over the same k-blocks and share those tiles' A rows and W
    // columns in L2 (stream-K's ranges start anywhere and share little).
    const int tail = p.tiles - p.dp_tiles, u = static_cast<int>(s.it);
    s.it = s.it_end;
    const int tt = u % tail;
    t.tile = p.dp_tiles + tt;
    t.piece = u / tail;
    t.npieces = p.splits;
    t.slot0 = tt * p.splits;
    t.kb_begin = t.piece * p.kb_total / p.splits;
    t.kb_end = (t.piece + 1) * p.kb_total / p.splits;
    place_tile<BN, CG>(p, t, rank, s.mt_begins);
    return true;
  }
  // By default the stream-K range comes first: the pieces that need summing
  // finish early, and their sums overlap the main loops of the whole tiles that
  // follow instead of trailing at the end of the kernel.
  if (s.it >= s.it_end || (p.sk_last && s.next < p.dp_tiles)) {
    if (s.next >= p.dp_tiles) return false;
    t.tile = s.next;                   // a whole tile
    s.next += s.G;
    t.piece = 0;
    t.npieces = 1;
    t.slot0 = 0;
    t.kb_begin = 0;
    t.kb_end = p.kb_total;
    place_tile<BN, CG>(p, t, rank, s.mt_begins);
    return true;
  }
  // the next piece of this worker's stream-K range
  const uint32_t kt = static_cast<uint32_t>(p.kb_total);
  const uint32_t I = static_cast<uint32_t>(p.sk_iters), G = static_cast<uint32_t>(s.G);
  const uint32_t sk_tile = s.it / kt;
  const uint32_t k_lo = s.it - sk_tile * kt;
  const uint32_t k_hi = min(kt, k_lo + (s.it_end - s.it));
  s.it += k_hi - k_lo;
  const int first_w = sk_worker_of(sk_tile * kt, I, G);
  const int last_w = sk_worker_of((sk_tile + 1) * kt - 1, I, G);
  t.tile = p.dp_tiles + static_cast<int>(sk_tile);
  t.piece = s.w - first_w;
  t.npieces = last_w - first_w + 1;
  // Along the stream-K range each new piece starts a new tile, a new worker's
  // range, or both, so (tile + worker) numbers the pieces without collisions.
  t.slot0 = static_cast<int>(sk_tile) + first_w;
  t.kb_begin = static_cast<int>(k_lo);
  t.kb_end = static_cast<int>(k_hi);
  place_tile<BN, CG>(p, t, rank, s.mt_begins);
  return true;
}

// MMA N of a tile: the full BN, or the ragged tail rounded up to 16 columns.
template <int BN>
__device__ __forceinline__ uint32_t tile_mma_n(const Params& p, const Unit& t) {
  return static_cast<uint32_t>(min(BN, (p.N - t.n0 + 15) & ~15));
}

// ------------------------------------------------------------ shared layout

// TMEM columns of the two accumulators: a power of two (an allocation rule),
// each accumulator at half of it (192-column tiles use 2 x 256 columns).
template <int BN>
__host__ __device__ constexpr uint32_t tmem_cols() { return BN <= 64 ? 128 : BN <= 128 ? 256 : 512; }
template <int BN>
__host__ __device__ constexpr uint32_t acc_stride() { return tmem_cols<BN>() / 2; }

template <int BN, int STAGES, int CG>
struct Layout {
  static constexpr uint32_t kABytes = BM * BK * 2;            // this CTA's rows of A
  // This CTA's columns of B: all of them, or its half of a pair's (with two
  // pairs in a cluster, each pair loads half of that half and multicasts it).
  static constexpr uint32_t kBBytes = (BN / (CG == 1 ? 1 : 2)) * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTiles = STAGES * kStageBytes;
  // barriers: full[S], empty[S], tmem_full[2], tmem_empty[2], drain
  static constexpr uint32_t kNumBars = 2 * STAGES + 5;
  static constexpr uint32_t kBarBytes = kNumBars * 8;
  static constexpr uint32_t kMiscBytes = 64;
  static constexpr size_t kSmem = 1024 + kTiles + kBarBytes + kMiscBytes;
  static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0, "tiles must stay 1024-aligned");
};

// ------------------------------------------------------------ roles

// The producer's L2 policies, schedule and first unit, taken at kernel entry
// before the CTA's own set-up (barriers, TMEM, cluster sync): their kernel-
// parameter reads and the prefetch of the first unit's descriptors, cold after
// a launch, overlap that set-up instead of delaying the first copy. Called by
// the whole producer warp.
template <int BN, int CG>
struct ProducerEntry {
  uint64_t pol_a, pol_b;
  Sched sch;
  Unit t;
  bool have;
  __device__ void init(const Params& p, uint32_t rank) {
    pol_a = make_l2_policy(p.policy_a);
    pol_b = make_l2_policy(p.policy_b);
    sch = sched_begin<CG>(p);
    have = sched_next<BN, CG>(p, sch, t, rank);
    if (!have) return;
    if (p.mode == kModeAG) {
      prefetch_tensormap(&p.tmap_a[t.shard >= 0 ? t.shard : p.ag_pad_shard]);
      prefetch_tensormap(&p.tmap_b[0]);
    } else {
      int r = 0;
      while (p.shard_kb_begin[r + 1] <= t.kb_begin) ++r;
      prefetch_tensormap(&p.tmap_a[r]);
      prefetch_tensormap(&p.tmap_b[r]);
    }
  }
};

template <int BN, int STAGES, int CG>
__device__ void run_producer(const Params& p, uint32_t tiles_base, uint32_t bars, uint32_t rank,
                             ProducerEntry<BN, CG>& entry, const Ctl& ctl) {
  using L = Layout<BN, STAGES, CG>;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES;
  // The descriptors of the other shards are prefetched once the first k-block
  // is on its way (the first copies fetch their own): the first loads leave
  // about a microsecond earlier.
  auto prefetch_descriptors = [&]() {
    if (p.mode == kModeAG) {
      for (int r = 0; r < p.R; ++r)   // empty shards have no descriptor
        if (p.shard_rows[r] > 0) prefetch_tensormap(&p.tmap_a[r]);
      prefetch_tensormap(&p.tmap_b[0]);
    } else {
      for (int r = 0; r < p.R; ++r) {
        prefetch_tensormap(&p.tmap_a[r]);
        prefetch_tensormap(&p.tmap_b[r]);
      }
    }
  };
  const uint64_t pol_a = entry.pol_a;
  const uint64_t pol_b = entry.pol_b;
  // AR/RS: the shard table in the warp's lanes (lane r holds shard r's first
  // k-block, lanes past R the k-block count), read with shuffles, so the
  // k-block loop loads nothing from the kernel's parameter space: a
  // dynamically indexed parameter load per k-block cost about 60 ns of the
  // loop's issue time (traced: about 320 ns per k-block before, which bound
  // tiles narrower than 256 columns).
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const int begins = p.shard_kb_begin[lane <= kMaxShards ? lane : kMaxShards];
  // With a pair, every copy completes on the leader's full barrier: the
  // barriers' addresses as seen from this CTA, mapped once.
  // With two pairs in a cluster (CG = 4) the pairs are ranks {0, 1} and {2, 3}.
  const uint32_t lead_full0 = CG == 1 ? full0 : map_shared_to_rank(full0, rank & ~1u);
  uint32_t issued = 0;
  uint32_t slot = 0, slot_parity = 1;   // ring slot of the next load; its free-wait parity
  uint32_t arrived = 0;   // AG with arrival flags: shards seen ready (bit r)
  bool ok = true;
  Sched& sch = entry.sch;
  Unit t = entry.t;
  for (bool have = entry.have; ok && have; have = sched_next<BN, CG>(p, sch, t, rank)) {
    const bool a_two = p.mode == kModeAG && p.ag_gran != BM;   // two 64-row boxes
    int shard_b = t.shard, m0b = t.m0;
    if (a_two) next_granule(p, sch.mt_begins, t.shard, t.m0, shard_b, m0b);
    // AG with arrival flags: every shard this CTA's rows come from must be in.
    for (int j = 0; ok && j < 2; ++j) {
      const int sh = j ? shard_b : t.shard;
      if (p.ready != nullptr && sh >= 0 && !(arrived & (1u << sh))) {
        const bool here = wait_flag(p.ready + sh, p.epoch, ctl, (kRoleProducer << 8) | 3);
        __syncwarp();
        if (!here) ok = false;
        else arrived |= 1u << sh;
      }
    }
    if (!ok) break;
    // This CTA's rows of A, and its columns of B: with a CTA pair the MMA's N
    // columns are split in halves between the two CTAs.
    // The idle half of an odd last pair tile reads rows past the end of a
    // non-empty shard: the TMA unit fills them with zeros.
    const int a_shard = t.shard >= 0 ? t.shard : p.ag_pad_shard;
    const int a_row = t.shard >= 0 ? t.m0 : p.shard_rows[p.ag_pad_shard];
    const int a_shard_b = shard_b >= 0 ? shard_b : p.ag_pad_shard;
    const int a_row_b = shard_b >= 0 ? m0b : p.shard_rows[p.ag_pad_shard];
    // CG = 4: this CTA's columns of B (its pair half) are loaded as two
    // quarter boxes, one by each pair, and multicast to the CTA at the same
    // place in both pairs; quarter p lands BN/4 rows into the half.
    const int b_row = CG <= 2 ? t.n0 + static_cast<int>(rank * (tile_mma_n<BN>(p, t) / CG))
                              : t.n0 + static_cast<int>((rank & 1u) * (tile_mma_n<BN>(p, t) / 2)) +
                                    static_cast<int>(rank >> 1) * (BN / 4);
    // AR/RS: shard r holds k-blocks [r_begin, r_end). The search stops at a
    // shard whose range holds kb_begin (< the k-block count, and every shard
    // has at least one k-block).
    int r = 0, r_begin = 0, r_end = 0;
    if (p.mode != kModeAG) {
      r_end = __shfl_sync(0xffffffffu, begins, 1);
      while (r_end <= t.kb_begin) r_end = __shfl_sync(0xffffffffu, begins, ++r + 1);
      r_begin = __shfl_sync(0xffffffffu, begins, r);
    }
    // The k-block loop, in two compiled forms so that the usual one (one box of
    // A rows) carries no test for the second box: this loop alone feeds the
    // tensor pipe, and every instruction added to it per k-block costs.
    auto stream_kblocks = [&](auto two_boxes) {
      constexpr bool kTwo = decltype(two_boxes)::value;
      for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
        const uint32_t stage = slot;
        const bool free_slot = wait_bounded(empty0 + 8 * stage, slot_parity, ctl, (kRoleProducer << 8) | 1);
        __syncwarp();
        if (!free_slot) {
          ok = false;
          break;
        }
        const uint32_t full = full0 + 8 * stage;
        const uint32_t sa = tiles_base + stage * L::kABytes;
        const uint32_t sb = tiles_base + STAGES * L::kABytes + stage * L::kBBytes;
        const CUtensorMap* ma;
        const CUtensorMap* ma_b = nullptr;   // the second 64-row box's shard
        const CUtensorMap* mb;
        int kx;
        if (p.mode == kModeAG) {
          ma = &p.tmap_a[a_shard];
          if constexpr (kTwo) ma_b = &p.tmap_a[a_shard_b];
          mb = &p.tmap_b[0];
          kx = kb * BK;
        } else {
          while (r_end <= kb) {
            r_begin = r_end;
            r_end = __shfl_sync(0xffffffffu, begins, ++r + 1);
          }
          ma = &p.tmap_a[r];
          mb = &p.tmap_b[r];
          kx = (kb - r_begin) * BK;
        }
        // With 64-row AG granules the A tile is two boxes of 64 rows (8 KB each,
        // a whole number of 128-byte swizzle atoms, so the layout is that of one
        // 128-row box).
        constexpr uint32_t kHalfA = L::kABytes / 2;
        if constexpr (CG == 1) {
          mbar_arrive_expect_tx(full, L::kStageBytes);
          tma_load_2d_hint(sa, ma, full, kx, a_row, pol_a);
          if constexpr (kTwo) tma_load_2d_hint(sa + kHalfA, ma_b, full, kx, a_row_b, pol_a);
          tma_load_2d_hint(sb, mb, full, kx, b_row, pol_b);
        } else {
          // Both CTAs' bytes are counted on the leader's full barrier, which the
          // leader alone arms (for the pair's bytes). The expect_tx and the
          // copies go out under one elected lane: an election per instruction
          // measured as issue time on this loop.
          const uint32_t lead_full = lead_full0 + 8 * stage;
          const bool leader = (rank & 1u) == 0;
          if constexpr (CG == 4) {
            // The pair's bytes (its A rows and both halves of its B columns,
            // whichever pair loaded them) complete on its leader's barrier.
            if (leader) mbar_arrive_expect_tx(full, 2 * L::kStageBytes);
            tma_load_2d_pair(sa, ma, lead_full, kx, a_row, pol_a);
            if constexpr (kTwo) tma_load_2d_pair(sa + kHalfA, ma_b, lead_full, kx, a_row_b, pol_a);
            const uint16_t both = static_cast<uint16_t>((1u << (rank & 1u)) | (4u << (rank & 1u)));
            tma_load_2d_pair_multicast(sb + (rank >> 1) * (L::kBBytes / 2), mb, lead_full, kx, b_row,
                                       both, pol_b);
          } else if constexpr (kTwo) {
            if (leader) mbar_arrive_expect_tx(full, CG * L::kStageBytes);
            tma_load_2d_pair(sa, ma, lead_full, kx, a_row, pol_a);
            tma_load_2d_pair(sa + kHalfA, ma_b, lead_full, kx, a_row_b, pol_a);
            tma_load_2d_pair(sb, mb, lead_full, kx, b_row, pol_b);
          } else {
            stage_copies_pair(leader ? 1u : 0u, full, CG * L::kStageBytes, lead_full, sa, ma,
                              a_row, sb, mb, b_row, kx, pol_a, pol_b);
          }
        }
        if (++issued == 1) prefetch_descriptors();
        if (++slot == STAGES) {
          slot = 0;
          slot_parity ^= 1u;
        }
      }
    };
    if (a_two)
      stream_kblocks(std::true_type{});
    else
      stream_kblocks(std::false_type{});
  }
  if (!ok && (CG == 1 || (rank & 1u) == 0)) {
    // Let every copy already issued land before the CTA's shared memory goes
    // away (with a pair, the leader's barriers count the peer's copies too).
    const uint32_t first = issued > STAGES ? issued - STAGES : 0;
    for (uint32_t i = first; i < issued; ++i)
      wait_drain(full0 + 8 * (i % STAGES), (i / STAGES) & 1u, 100000000ull);
  }
}

template <int BN, int STAGES, int CG>
__device__ void run_mma(const Params& p, uint32_t tiles_base, uint32_t bars, uint32_t tmem_base,
                        uint32_t rank, const Ctl& ctl) {
  using L = Layout<BN, STAGES, CG>;
  const uint32_t full0 = bars, tfull0 = bars + 16 * STAGES, tempty0 = tfull0 + 16;
  const uint32_t empty0 = bars + 8 * STAGES, drain = tempty0 + 16;
  // Only a pair's leader issues its MMAs (rank 0, or 0 and 2 with two pairs).
  // A stage is freed in every CTA its copies wrote: both CTAs of the pair, or
  // all four with two pairs (each CTA's empty barrier then counts both
  // leaders' commits). The accumulator is the pair's.
  constexpr uint16_t kFreeMask = CG == 4 ? 0xF : 0x3;
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (rank & ~1u));
  uint32_t stage = 0, phase = 0, local = 0;   // next ring slot and its fill phase
  bool ok = true, issued_any = false;
  Sched sch = sched_begin<CG>(p);
  // The next unit is placed while the current one's first k-block runs on the
  // tensor pipe, so the walk's arithmetic stays off the gap between units.
  Unit t, tn;
  bool have = sched_next<BN, CG>(p, sch, t, rank);
  for (; ok && have; ++local) {
    bool have_next = false, looked_ahead = false;
    const uint32_t acc = local & 1u;
    const uint32_t acc_parity = ((local >> 1) & 1u) ^ 1u;
    const bool free_acc = wait_bounded(tempty0 + 8 * acc, acc_parity, ctl, (kRoleMma << 8) | 1);
    __syncwarp();
    if (!free_acc) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + acc * acc_stride<BN>();
    const uint32_t idesc = make_idesc(BM * (CG == 1 ? 1 : 2), tile_mma_n<BN>(p, t));
    // The next slot's barrier is tested (without blocking) before this slot's
    // MMAs are issued, so the test overlaps the tensor pipe's work instead of
    // sitting between the MMAs of two consecutive k-blocks. The slot's bytes
    // were written by TMA and read by the MMAs, both in the async proxy; the
    // barrier's completion orders them.
    bool ready = mbar_test_wait(full0 + 8 * stage, phase);
    for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
      if (!ready) {
        const bool got = wait_bounded(full0 + 8 * stage, phase, ctl, (kRoleMma << 8) | 2);
        __syncwarp();
        if (!got) {
          ok = false;
          break;
        }
      }
      const uint32_t cur = stage;
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
      ready = kb + 1 < t.kb_end && mbar_test_wait(full0 + 8 * stage, phase);
      const uint64_t a_desc = smem_desc_sw128(tiles_base + cur * L::kABytes);
      const uint64_t b_desc = smem_desc_sw128(tiles_base + STAGES * L::kABytes + cur * L::kBBytes);
      if constexpr (CG == 1) {
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          // advance 16 elements (32 bytes) along K inside the swizzled 128-byte rows
          const uint32_t accumulate = (kb > t.kb_begin || k > 0) ? 1u : 0u;
          mma_bf16_ss(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, accumulate);
        }
      } else {
        // The k-block's four K=16 steps under one election (one per MMA
        // measured as issue time on this loop).
        mma4_bf16_pair(d_tmem, a_desc, b_desc, idesc, kb > t.kb_begin ? 1u : 0u);
      }
      issued_any = true;
      if constexpr (CG == 1)
        mma_commit(empty0 + 8 * cur);
      else
        mma_commit_pair(empty0 + 8 * cur, kFreeMask);   // frees the slot in every CTA it fed
      if (!looked_ahead) {
        have_next = sched_next<BN, CG>(p, sch, tn, rank);
        looked_ahead = true;
      }
    }
    if (!ok) break;
    if constexpr (CG == 1)
      mma_commit(tfull0 + 8 * acc);
    else
      mma_commit_pair(tfull0 + 8 * acc, pair_mask);   // both CTAs' epilogues may read
    if (!looked_ahead) have_next = sched_next<BN, CG>(p, sch, tn, rank);
    t = tn;
    have = have_next;
  }
  if (!ok && issued_any) {
    // Every MMA issued so far must finish before the TMEM is released.
    if constexpr (CG == 1)
      mma_commit(drain);
    else
      mma_commit_pair(drain, static_cast<uint16_t>(1u << rank));
    wait_drain(drain, 0, 100000000ull);
  }
}

__device__ __forceinline__ void store_row_chunk(uint16_t* row_ptr, int col_in_tile, int n_valid,
                                                const uint32_t (&v)[32], bool row_ok) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = col_in_tile + 8 * j;
    if (row_ok && c < n_valid) {
      uint4 w;
      w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
      w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
      w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
      w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
      *reinterpret_cast<uint4*>(row_ptr + c) = w;
    }
  }
}

template <int BN, int STAGES, int CG>
__device__ void run_epilogue(const Params& p, uint32_t bars, uint32_t tmem_base, uint32_t rank,
                             volatile int* last_flag, const Ctl& ctl) {
  const uint32_t tfull0 = bars + 16 * STAGES, tempty0 = tfull0 + 16;
  const int et = static_cast<int>(threadIdx.x) - 64;          // 0..127
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const int quad = (static_cast<int>(threadIdx.x) >> 5) & 3;  // TMEM lanes this warp may read
  const int row_in_tile = quad * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
  uint32_t local = 0;
  Sched sch = sched_begin<CG>(p);
  Unit t;
  for (; sched_next<BN, CG>(p, sch, t, rank); ++local) {
    const uint32_t acc = local & 1u;
    const uint32_t acc_parity = (local >> 1) & 1u;
    bool ok = wait_bounded(tfull0 + 8 * acc, acc_parity, ctl, (kRoleEpilogue << 8) | 1);
    if (!epilogue_bar_and(ok)) break;  // all 128 threads leave together
    tc_fence_after_sync();

    const uint32_t taddr = tmem_base + lane_addr + acc * acc_stride<BN>();
    const int n_valid = min(BN, p.N - t.n0);
    const int chunks = (n_valid + 31) >> 5;
    const int m0 = t.m0;   // this CTA's first row

    // Where this thread's output row goes (with replicated outputs: the same
    // offset in every one of the R buffers).
    bool row_ok;
    uint16_t* row_ptr;
    size_t rep_off = 0;
    if (p.mode == kModeAG) {
      // With 64-row granules, rows 64..127 of the tile are the second granule's.
      int shard_b = t.shard, m0b = t.m0;
      if (p.ag_gran != BM) next_granule(p, sch.mt_begins, t.shard, t.m0, shard_b, m0b);
      const bool second = p.ag_gran != BM && row_in_tile >= 64;
      const int shard = second ? shard_b : t.shard;
      const int sh = shard >= 0 ? shard : 0;
      const int lr = second ? m0b + (row_in_tile - 64) : m0 + row_in_tile;
      row_ok = shard >= 0 && lr < p.shard_rows[sh];
      row_ptr = p.y + (static_cast<size_t>(p.shard_row_begin[sh]) + lr) * p.N + t.n0;
    } else {
      const int gr = m0 + row_in_tile;
      row_ok = gr < p.M;
      if (p.mode == kModeRS) {
        const int s = row_ok ? gr / p.rps : 0;
        row_ptr = p.y_r[s] + static_cast<size_t>(gr - s * p.rps) * p.N + t.n0;
      } else if (p.mode == kModeARRep) {
        rep_off = static_cast<size_t>(gr) * p.N + t.n0;
        row_ptr = p.y_r[0] + rep_off;
      } else {
        row_ptr = p.y + static_cast<size_t>(gr) * p.N + t.n0;
      }
    }
    auto emit = [&](int col, const uint32_t (&v)[32]) {
      if (p.mode == kModeARRep) {
        for (int i = 0; i < p.R; ++i) store_row_chunk(p.y_r[i] + rep_off, col, n_valid, v, row_ok);
      } else {
        store_row_chunk(row_ptr, col, n_valid, v, row_ok);
      }
    };

    // Hands the accumulator back to the MMA issuer (the leader's barrier with a
    // pair): one arrival per warp once its TMEM reads are complete.
    auto release_accumulator = [&]() {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 1)
          mbar_arrive(tempty0 + 8 * acc);
        else
          mbar_arrive_cluster(map_shared_to_rank(tempty0 + 8 * acc, rank & ~1u));
      }
    };

    // A CTA half with no valid row (the second half of a pair tile past M, or
    // the idle half of an odd AG pair) stores nothing and, with a cut tile,
    // skips the partial/counter protocol: every piece of this half is idle
    // alike, and its counter stays at zero.
    const bool idle = p.mode == kModeAG ? t.shard < 0 : t.m0 >= p.M;
    if (idle) {
      release_accumulator();
      continue;
    }

    if (t.npieces == 1) {
      // Two 32-column TMEM loads per wait halve the load round trips.
      for (int c = 0; c < chunks; c += 2) {
        uint32_t v[32], u[32];
        tmem_ld_32cols(taddr + 32 * c, v);
        if (c + 1 < chunks) tmem_ld_32cols(taddr + 32 * (c + 1), u);
        tmem_ld_wait2(v, u);
        emit(32 * c, v);
        if (c + 1 < chunks) emit(32 * (c + 1), u);
      }
      release_accumulator();
      continue;
    }

    // Split tile. A piece that finds every other piece already published is
    // the last: it keeps its own accumulator in TMEM and writes no partial.
    // Otherwise it publishes its fp32 partial (slot layout [column group of
    // 4][row][4], so a warp's float4 stores are contiguous), fences, and bumps
    // the tile's counter; the piece that brings the counter to npieces - 1 is
    // the last. The last piece sums all pieces in k order and stores the tile.
    // A piece that publishes hands its accumulator back as soon as it has read
    // it (before the fence and the counter round trips: the MMA issuer may need
    // it for the unit after next); if it then turns out to be the last, it reads
    // its own partial back from its slot. A CTA pair keeps one slot and one
    // counter per half.
    const int half = t.tile * CG + static_cast<int>(rank);
    const uint32_t others = static_cast<uint32_t>(t.npieces - 1);
    if (et == 0) *last_flag = (ld_relaxed_gpu(&p.counters[half]) == others) ? 1 : 0;
    epilogue_bar_sync();
    bool last = *last_flag != 0;
    bool own_in_tmem = true;
    if (!last) {
      float* slot = p.partials +
                    (static_cast<size_t>(t.slot0 + t.piece) * CG + rank) * (BM * BN);
      for (int c = 0; c < chunks; ++c) {
        uint32_t v[32];
        tmem_ld_32cols(taddr + 32 * c, v);
        tmem_ld_wait(v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float4 f = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                 __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          __stcg(reinterpret_cast<float4*>(slot) + (8 * c + j) * BM + row_in_tile, f);
        }
      }
      release_accumulator();
      own_in_tmem = false;
      __threadfence();
      epilogue_bar_sync();
      if (et == 0) *last_flag = (atomicAdd(&p.counters[half], 1u) == others) ? 1 : 0;
      epilogue_bar_sync();
      last = *last_flag != 0;
    }
    if (last) {
      __threadfence();
      // The tile's pieces sit in consecutive slots from slot0, in k order. Each
      // step reads 64 columns of one piece (its own from TMEM, another's from
      // its slot: 16 independent float4 loads in flight per thread).
      const float4* base = reinterpret_cast<const float4*>(p.partials);
      const size_t slot_f4 = static_cast<size_t>(BM) * BN / 4;
      auto load_piece = [&](int s, int c, float (&d)[64]) {
        if (s == t.piece && own_in_tmem) {
          uint32_t v[32], u[32];
          tmem_ld_32cols(taddr + 32 * c, v);
          if (c + 1 < chunks) tmem_ld_32cols(taddr + 32 * (c + 1), u);
          tmem_ld_wait2(v, u);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            d[j] = __uint_as_float(v[j]);
            d[32 + j] = __uint_as_float(u[j]);
          }
        } else {
          const float4* src = base + ((static_cast<size_t>(t.slot0) + s) * CG + rank) * slot_f4;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            // chunk c covers column groups 8c .. 8c+15 over two chunks
            const float4 f = __ldcg(src + (8 * c + j) * BM + row_in_tile);
            d[4 * j] = f.x; d[4 * j + 1] = f.y; d[4 * j + 2] = f.z; d[4 * j + 3] = f.w;
          }
        }
      };
      for (int c = 0; c < chunks; c += 2) {
        float a[64], b[64];
        load_piece(0, c, a);
        for (int s = 1; s < t.npieces; ++s) {
          load_piece(s, c, b);
#pragma unroll
          for (int j = 0; j < 64; ++j) a[j] += b[j];
        }
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(a[j]);
        emit(32 * c, v);
        if (c + 1 < chunks) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(a[32 + j]);
          emit(32 * (c + 1), v);
        }
      }
      if (et == 0) atomicExch(&p.counters[half], 0u);  // ready for the next call
    }
    if (own_in_tmem) release_accumulator();  // the TMEM accumulator is free for the next tile
  }
}

// ------------------------------------------------------------ kernel

template <int BN, int STAGES, int CG>
__global__ void __launch_bounds__(kThreads, 1) gsr_gemm_kernel(const __grid_constant__ Params p) {
  using L = Layout<BN, STAGES, CG>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t tiles_base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (tiles_base - raw);
  const uint32_t bars = tiles_base + L::kTiles;
  uint8_t* misc = base_ptr + L::kTiles + L::kBarBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(misc + 8);

  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const uint32_t rank = (CG == 1) ? 0u : cluster_rank();
  ProducerEntry<BN, CG> entry;
  if (warp == 0) entry.init(p, rank);

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bars + 8 * i, 1);                 // full: the (leader's) expect_tx + TMA bytes
      mbar_init(bars + 8 * (STAGES + i), CG == 4 ? 2 : 1);   // empty: each feeding leader's commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 16 * STAGES + 8 * i, 1);               // tmem_full: MMA commit
      mbar_init(bars + 16 * STAGES + 16 + 8 * i, CG == 1 ? 4 : 8);   // tmem_empty: one per epilogue warp of the pair
    }
    mbar_init(bars + 16 * STAGES + 32, 1);  // drain
    *abort_flag = 0;
    *last_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (CG == 1) {
      tmem_alloc(smem_u32(tmem_slot), tmem_cols<BN>());
      tmem_relinquish();
    } else {
      tmem_alloc_pair(smem_u32(tmem_slot), tmem_cols<BN>());
      tmem_relinquish_pair();
    }
  }
  tc_fence_before_sync();
  if constexpr (CG == 1)
    __syncthreads();
  else
    cluster_barrier();   // the peer's barriers exist before anyone signals them
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  // Programmatic dependent launch: everything above (barriers, TMEM, cluster
  // sync) may overlap the tail of the previous kernel in the stream; nothing
  // below touches global memory before that kernel has completed and its
  // writes are visible. A kernel launched after this one may likewise start
  // its own set-up now; it waits for this grid the same way.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  Ctl ctl{abort_flag, p.status, p.timeout_ns};
  if (warp == 0) {
    run_producer<BN, STAGES, CG>(p, tiles_base, bars, rank, entry, ctl);   // whole warp, elected issue
    __syncwarp();
  } else if (warp == 1) {
    // The whole warp walks the MMA loop (its values stay warp-uniform); one
    // elected lane issues each MMA and commit.
    if ((rank & 1u) == 0) run_mma<BN, STAGES, CG>(p, tiles_base, bars, tmem_base, rank, ctl);
    __syncwarp();
  } else {
    run_epilogue<BN, STAGES, CG>(p, bars, tmem_base, rank, last_flag, ctl);
  }

  tc_fence_before_sync();
  if constexpr (CG == 1)
    __syncthreads();
  else
    cluster_barrier();   // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after_sync();
    if constexpr (CG == 1)
      tmem_dealloc(tmem_base, tmem_cols<BN>());
    else
      tmem_dealloc_pair(tmem_base, tmem_cols<BN>());
  }
}

// Ring depths: each instance fills 192-224 KB of shared memory.
template <int BN, int CG> struct Stages;
template <> struct Stages<256, 1> { static constexpr int value = 4; };   // 48 KB stages
template <> struct Stages<128, 1> { static constexpr int value = 6; };   // 32 KB
template <> struct Stages<256, 2> { static constexpr int value = 7; };   // 32 KB per CTA
template <> struct Stages<128, 2> { static constexpr int value = 8; };   // 24 KB per CTA
template <> struct Stages<192, 2> { static constexpr int value = 8; };   // 28 KB per CTA
// Two CTA pairs per cluster (B multicast between the pairs): the same stages.
template <> struct Stages<256, 4> { static constexpr int value = 7; };
template <> struct Stages<128, 4> { static constexpr int value = 8; };
template <> struct Stages<192, 4> { static constexpr int value = 8; };

template <int BN, int CG>
using KernelLayout = Layout<BN, Stages<BN, CG>::value, CG>;

template <int BN, int CG>
cudaError_t set_smem_limit() {
  return cudaFuncSetAttribute(gsr_gemm_kernel<BN, Stages<BN, CG>::value, CG>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(KernelLayout<BN, CG>::kSmem));
}

template <int BN, int CG>
cudaError_t launch_instance(const Params& p, int ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  // May start while the previous kernel in the stream finishes (the kernel
  // waits for it with griddepcontrol.wait before touching global memory).
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (CG >= 2) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = CG;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = KernelLayout<BN, CG>::kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, gsr_gemm_kernel<BN, Stages<BN, CG>::value, CG>, p);
}

}  // namespace

size_t kernel_smem_bytes(int block_n, int cta_group) {
  if (cta_group >= 2)
    return block_n == 256   ? KernelLayout<256, 2>::kSmem
           : block_n == 192 ? KernelLayout<192, 2>::kSmem
                            : KernelLayout<128, 2>::kSmem;
  return block_n == 256 ? KernelLayout<256, 1>::kSmem : KernelLayout<128, 1>::kSmem;
}

cudaError_t prepare_kernels(int device, int* pair_clusters, int* quad_clusters) {
  (void)device;  // the caller has made `device` current
  cudaError_t e = set_smem_limit<256, 1>();
  if (e == cudaSuccess) e = set_smem_limit<128, 1>();
  if (e == cudaSuccess) e = set_smem_limit<256, 2>();
  if (e == cudaSuccess) e = set_smem_limit<128, 2>();
  if (e == cudaSuccess) e = set_smem_limit<192, 2>();
  if (e == cudaSuccess) e = set_smem_limit<256, 4>();
  if (e == cudaSuccess) e = set_smem_limit<128, 4>();
  if (e == cudaSuccess) e = set_smem_limit<192, 4>();
  if (e != cudaSuccess) return e;
  {
    // How many clusters of two CTA pairs can be resident at once.
    cudaLaunchConfig_t cfg4 = {};
    cudaLaunchAttribute attr4[1];
    attr4[0].id = cudaLaunchAttributeClusterDimension;
    attr4[0].val.clusterDim.x = 4;
    attr4[0].val.clusterDim.y = 1;
    attr4[0].val.clusterDim.z = 1;
    cfg4.gridDim = dim3(4, 1, 1);
    cfg4.blockDim = dim3(kThreads, 1, 1);
    cfg4.dynamicSmemBytes = KernelLayout<256, 4>::kSmem;
    cfg4.attrs = attr4;
    cfg4.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(quad_clusters, gsr_gemm_kernel<256, Stages<256, 4>::value, 4>,
                                       &cfg4);
    if (e != cudaSuccess) return e;
  }
  // How many CTA pairs can be resident at once (SMs pair up inside a GPC).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = KernelLayout<256, 2>::kSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(pair_clusters,
                                        gsr_gemm_kernel<256, Stages<256, 2>::value, 2>, &cfg);
}

cudaError_t launch_gemm(const Params& p, int block_n, int cta_group, int ctas, cudaStream_t stream) {
  if (cta_group == 4)
    return block_n == 256   ? launch_instance<256, 4>(p, ctas, stream)
           : block_n == 192 ? launch_instance<192, 4>(p, ctas, stream)
                            : launch_instance<128, 4>(p, ctas, stream);
  if (cta_group == 2)
    return block_n == 256   ? launch_instance<256, 2>(p, ctas, stream)
           : block_n == 192 ? launch_instance<192, 2>(p, ctas, stream)
                            : launch_instance<128, 2>(p, ctas, stream);
  return block_n == 256 ? launch_instance<256, 1>(p, ctas, stream)
                        : launch_instance<128, 1>(p, ctas, stream);
}

}  // namespace gsr
