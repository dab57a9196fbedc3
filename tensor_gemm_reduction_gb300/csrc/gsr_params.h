// gsr_params.h -- launch parameters of the shard-reduction GEMM kernel
// (internal to the library; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gsr {

constexpr int kMaxShards = 16;
constexpr int BM = 128;          // output tile rows = tcgen05 MMA M (cta_group::1)
constexpr int BK = 64;           // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kEpilogueThreads = 128;

// kModeARRep: the AR sum written whole into each of R output buffers.
enum Mode : int { kModeAR = 0, kModeRS = 1, kModeAG = 2, kModeARRep = 3 };

// Work schedules. Uniform: unit u = tile * splits + piece, dealt round-robin.
// Stream-K: tiles [0, dp_tiles) are dealt whole, round-robin; the k-blocks of
// the remaining tiles, in tile order, are cut into one contiguous range per
// worker (a CTA, or a CTA pair), and a tile cut by a worker boundary is
// summed by the last of its pieces to finish, in k order.
// Small (small-M kernel): one CTA pair per tile of W rows over the whole K
// range, tiles dealt round-robin to the pairs.
enum Sched : int { kSchedUniform = 0, kSchedStreamK = 1, kSchedSmall = 2, kSchedSplitTail = 3 };

// L2 eviction priority requested for an operand's TMA loads.
enum Policy : int { kPolicyNormal = 0, kPolicyEvictFirst = 1, kPolicyEvictLast = 2 };

// Status word codes written by the kernel (workspace offset 0). 0 = OK.
// A timed-out wait stores kStatusTimeout | (role << 8) | site.
constexpr uint32_t kStatusTimeout = 0x54000000u;

// Workspace layout (bytes): [0, 256) header (status word at 0);
// [256, 256 + 4*counter_slots) per-tile arrival counters, rounded up to 256;
// then fp32 split-K partial tiles of BM x BN each.
constexpr size_t kWsHeader = 256;

struct Params {  // 128-byte aligned through its CUtensorMap members
  // Per-shard TMA descriptors. AR/RS: tmap_a[r] = X_r (box 64 x 128),
  // tmap_b[r] = W_r (box 64 x BN). AG: tmap_a[r] = A_r, tmap_b[0] = W.
  CUtensorMap tmap_a[kMaxShards];
  CUtensorMap tmap_b[kMaxShards];

  uint16_t* y;                  // AR, AG: output rows x N (bf16 bits)
  uint16_t* y_r[kMaxShards];    // RS: shard outputs, rps x N each; AR replicated:
                                // R outputs, M x N each
  const uint32_t* ready;        // AG with arrival flags: ready[r] reaches epoch when
                                // shard r's rows are in memory (NULL: no waiting)
  uint32_t epoch;
  uint32_t* status;             // workspace status word
  uint32_t* counters;           // workspace per-tile arrival counters
  float* partials;              // workspace split-K partial tiles
  uint64_t timeout_ns;          // limit of every bounded wait

  int mode;
  int R;
  int M;                        // AR/RS: rows; AG: sum of M_r
  int N;
  int m_tiles;                  // AR/RS: ceil(M/(BM*CG)); AG: ceil(halves/CG)
  int n_tiles;                  // ceil(N/BN)
  int tiles;                    // m_tiles * n_tiles
  int kb_total;                 // k-blocks per tile (AR/RS: sum_r ceil(K_r/BK)); the
                                // small-M kernel: stages of small_kz k-blocks
  int splits;                   // uniform schedule: pieces per tile (1 = none)
  int units;                    // uniform schedule: tiles * splits
  int sched;                    // kSchedUniform, kSchedStreamK or kSchedSplitTail
  int dp_tiles;                 // stream-K: tiles [0, dp_tiles) run whole, round-robin
  long long sk_iters;           // stream-K: k-blocks of tiles [dp_tiles, tiles)
  int sk_last;                  // stream-K: walk the whole tiles first, the range last
  int group_m;                  // raster group height, in m-tiles (1 = n fastest)
  int group_n;                  // > 0: raster groups of group_n n-tiles instead, n fastest
  int policy_a;                 // L2 policy of A-operand loads (kPolicy*)
  int policy_b;                 // L2 policy of B-operand loads (kPolicy*)
  int rps;                      // RS: rows per shard = ceil(M/R)
  int shard_kb_begin[kMaxShards + 1];  // AR/RS: first k-block (small-M: stage) of shard r
  int shard_mt_begin[kMaxShards + 1];  // AG: first row granule of shard r
  int ag_halves;                // AG: row granules over all shards
  int ag_gran;                  // AG: rows per granule, 128 (one per CTA tile) or 64
                                // (two per CTA tile, possibly from two shards)
  int ag_pad_shard;             // AG: a non-empty shard, read out of range (zeros)
                                // by the idle half of an odd last pair tile
  int shard_row_begin[kMaxShards + 1]; // AG: first output row of shard r
  int shard_rows[kMaxShards];          // AG: M_r
  int m_pad;                    // small-M kernel: activation rows rounded up to 16;
                                // 0 for the main kernel
  int stages;                   // small-M kernel: depth of the shared-memory ring
  int tile_rows;                // small-M kernel: W rows per tile (the pair MMA's N:
                                // a multiple of 16, at most kSmallMaxTileN)
  int small_kz;                 // small-M kernel: k-blocks per copy (1: 2-D copies;
                                // 2..4: 3-D copies of that many k-blocks)
};

// ---------------------------------------------------------------- small M
// The small-M kernel (M <= kSmallMaxM, AR/RS) runs one CTA pair (a cluster of
// two) per tile of tile_rows rows of W (output columns; a multiple of 16, at
// most kSmallMaxTileN) over the whole K range, with every activation row in
// the tile: tcgen05.mma.cta_group::2 with the activation rows as the MMA's M
// (each CTA holds h = ceil(M / 2) rows rounded up to 8: an MMA of 128 rows,
// 64 per CTA, when h <= 64, else of 256, 128 per CTA) and the tile's W rows
// as its N (each CTA holds half of them). A ring stage holds kz consecutive
// k-blocks of each operand (one copy each: kz = 1 is a 2-D box, kz = 2..4
// a 3-D box over a {64, rows, K_r / 64} view of the shard, whose last stage
// may run past the shard's k-blocks into zero fill). Its shared memory, from a
// 1024-aligned base: the X ring, the W ring, the mbarriers and a few words.
// Host and device share this layout.
constexpr int kSmallMaxM = 256;
constexpr int kSmallMaxTileN = 256;
constexpr int kSmallEpiWarps = 4;                 // one per TMEM lane quarter
constexpr int kSmallThreads = 64 + 32 * kSmallEpiWarps;  // warp 0 TMA, warp 1 MMA, the rest epilogue
constexpr int kSmallMaxStages = 32;
constexpr uint32_t kSmallSmemLimit = 232448;     // 227 KB per CTA

struct SmallLayout {
  uint32_t mma_m;        // 128 (x_rows <= 64) or 256
  uint32_t x_rows;       // h: activation rows per CTA, a multiple of 8 (rank r holds rows r*h ..
                         // r*h + h); the X box height
  uint32_t kz;           // k-blocks per stage
  uint32_t x_bytes, w_bytes;    // one k-block of X, of W
  uint32_t x_stage, w_stage;    // one stage: kz k-blocks
  uint32_t stages;
  uint32_t w_off, bars_off, misc_off, total;  // total includes 1024 of alignment slack
  uint32_t acc_cols;     // TMEM columns one accumulator uses
  uint32_t acc_stride;   // columns between the two accumulators
  uint32_t tmem_cols;    // allocated: a power of two, at least 32
};

__host__ __device__ inline SmallLayout small_layout(int M, int tile_rows, int stages, int kz) {
  SmallLayout L;
  // The rows are split evenly over the pair, so that both CTAs stream the same
  // bytes; the MMA reads mma_m / 2 rows from each, of which rows past h are
  // stale shared memory (TMEM lanes that are never stored) and rows past M
  // are zero-filled by the copy (or, when a CTA has none, never loaded).
  const int half = (M + 1) / 2;
  L.x_rows = static_cast<uint32_t>(half <= 8 ? 8 : (half + 7) / 8 * 8);   // whole 8-row swizzle atoms
  L.mma_m = L.x_rows <= 64 ? 128u : 256u;
  L.x_bytes = L.x_rows * BK * 2;
  L.w_bytes = static_cast<uint32_t>(tile_rows / 2) * BK * 2;
  L.kz = static_cast<uint32_t>(kz);
  L.x_stage = L.kz * L.x_bytes;
  L.w_stage = L.kz * L.w_bytes;
  L.stages = static_cast<uint32_t>(stages);
  L.w_off = L.stages * L.x_stage;
  // The MMA reads mma_m / 2 rows from an X k-block: the last one's read runs
  // past the X ring into the W ring (or, if that is shorter, into padding).
  uint32_t end = L.w_off + L.stages * L.w_stage;
  const uint32_t x_read_end = L.w_off - L.x_bytes + L.mma_m / 2 * BK * 2;
  if (x_read_end > end) end = x_read_end;
  L.bars_off = end;
  L.misc_off = L.bars_off + (2 * L.stages + 5) * 8;   // full, empty, tfull[2], tempty[2], drain
  L.total = 1024 + L.misc_off + 16;
  L.acc_cols = L.mma_m == 256 ? static_cast<uint32_t>(tile_rows) : static_cast<uint32_t>(tile_rows / 2);
  L.acc_stride = (L.acc_cols + 31) / 32 * 32;
  uint32_t cols = 32;
  while (cols < 2 * L.acc_stride) cols *= 2;
  L.tmem_cols = cols;
  return L;
}

// Deepest ring that fits the shared-memory limit.
__host__ __device__ inline int small_stages(int M, int tile_rows, int kz) {
  int s = kSmallMaxStages;
  while (s > 2 && small_layout(M, tile_rows, s, kz).total > kSmallSmemLimit) --s;
  return s;
}

// ---------------------------------------------------------------- packed gather
// P[g, t*H .. (t+1)*H) = S[r][t][g - row_begin[r], :] for output rows g <
// rows_out, g in shard r's rows [row_begin[r], row_begin[r+1]).
constexpr int kMaxPackStates = 16;
constexpr int64_t kPackPieceMax = 16384;     // bytes per bulk copy

struct PackParams {
  const uint16_t* src[kMaxShards * kMaxPackStates];  // src[r*T + t]: M_r x H, row-major
  int64_t row_begin[kMaxShards + 1];                  // entries past R: the sum of M_r
  uint16_t* dst;                                      // rows_out x T*H, row-major
  uint32_t* status;                                   // workspace status word
  uint64_t timeout_ns;
  int64_t rows_out;
  int64_t seg_bytes;                                  // H * 2: one state row
  int R, T;
  int pieces_per_seg;                                 // ceil(seg_bytes / kPackPieceMax)
};

// Host-side launcher (defined with the kernel).
// cta_group 1: one CTA per 128-row tile; 2: a CTA pair (cluster of two) per
// 256-row tile; 4: two CTA pairs (a cluster of four) on two 256-row tiles of
// the same columns, sharing each copy of B. block_n is 128, 192 (pairs) or
// 256. `ctas` counts CTAs (a multiple of the cluster size).
cudaError_t launch_gemm(const Params& p, int block_n, int cta_group, int ctas, cudaStream_t stream);
// Sets shared-memory limits and reports how many CTA pairs, and how many
// clusters of two CTA pairs, can be resident.
cudaError_t prepare_kernels(int device, int* pair_clusters, int* quad_clusters);
size_t kernel_smem_bytes(int block_n, int cta_group);
// The small-M kernel (gsr_small.cu): `ctas` is even (CTA pairs).
cudaError_t launch_small(const Params& p, int ctas, cudaStream_t stream);
cudaError_t prepare_small_kernel();
// The packed gather (gsr_pack.cu): one warp per CTA.
cudaError_t launch_pack(const PackParams& p, int ctas, cudaStream_t stream);
cudaError_t prepare_pack_kernel();

}  // namespace gsr
