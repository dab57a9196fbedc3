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
// K-pair (small-M kernel): each output tile is computed by the two CTAs of a
// cluster, each over half of the k-blocks, and the two halves are added in
// distributed shared memory.
enum Sched : int { kSchedUniform = 0, kSchedStreamK = 1, kSchedKPair = 2, kSchedSplitTail = 3 };

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
  int kb_total;                 // k-blocks per tile (AR/RS: sum_r ceil(K_r/BK))
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
  int shard_kb_begin[kMaxShards + 1];  // AR/RS: first k-block of shard r
  int shard_mt_begin[kMaxShards + 1];  // AG: first row granule of shard r
  int ag_halves;                // AG: row granules over all shards
  int ag_gran;                  // AG: rows per granule, 128 (one per CTA tile) or 64
                                // (two per CTA tile, possibly from two shards)
  int ag_pad_shard;             // AG: a non-empty shard, read out of range (zeros)
                                // by the idle half of an odd last pair tile
  int shard_row_begin[kMaxShards + 1]; // AG: first output row of shard r
  int shard_rows[kMaxShards];          // AG: M_r
  int m_pad;                    // small-M kernel: activation rows rounded up to 16
                                // (the MMA's N); 0 for the main kernel
  int stages;                   // small-M kernel: depth of the shared-memory ring
  int tile_rows;                // small-M kernel: W rows per tile (a multiple of 8,
                                // at most kSmallTileN; TMEM lanes past it unused)
};

// ---------------------------------------------------------------- small M
// The small-M kernel (M <= kSmallMaxM, AR/RS) swaps the operands: a tile is
// up to kSmallTileN rows of W (output columns, the MMA's M, always 128: rows
// past the tile are stale shared memory whose TMEM lanes are never stored)
// against all m_pad activation rows (the MMA's N). Its shared memory, from a 1024-aligned base:
// the W ring, the X ring, the staging area that receives the peer CTA's
// partial for the output rows this CTA finishes (and, once read, the bf16
// transposes of the finished rows), the mbarriers and a few words. Host and device share
// this layout.
constexpr int kSmallTileN = 128;
constexpr int kSmallMaxM = 256;
constexpr int kSmallEpiWarps = 8;            // two per TMEM lane quarter
constexpr int kSmallEpiThreads = 32 * kSmallEpiWarps;
constexpr int kSmallThreads = 64 + kSmallEpiThreads;  // warp 0 TMA, warp 1 MMA, the rest epilogue
constexpr int kGranule = 16;                 // output rows per exchange granule
constexpr int kSmallMaxStages = 16;
constexpr uint32_t kSmallSmemLimit = 232448; // 227 KB per CTA

struct SmallLayout {
  uint32_t w_bytes, x_bytes, stages;
  uint32_t x_off, staging_off, bars_off, misc_off, total;  // total includes 1024 of alignment slack
  uint32_t tmem_cols, acc_stride;
};

__host__ __device__ inline uint32_t small_owned_granules(int m_pad) {
  return static_cast<uint32_t>((m_pad / kGranule + 1) / 2);
}

__host__ __device__ inline SmallLayout small_layout(int m_pad, int stages) {
  SmallLayout L;
  L.w_bytes = kSmallTileN * BK * 2;
  L.x_bytes = static_cast<uint32_t>(m_pad) * BK * 2;
  L.stages = static_cast<uint32_t>(stages);
  L.x_off = L.stages * L.w_bytes;
  L.staging_off = L.x_off + L.stages * L.x_bytes;
  L.bars_off = L.staging_off + small_owned_granules(m_pad) * kGranule * kSmallTileN * 4;
  L.misc_off = L.bars_off + (2 * L.stages + 7) * 8;
  L.total = 1024 + L.misc_off + 16;
  uint32_t cols = 32;
  while (cols < 2u * static_cast<uint32_t>(m_pad)) cols *= 2;
  L.tmem_cols = cols;
  L.acc_stride = cols / 2;
  return L;
}

// Deepest ring that fits the shared-memory limit for m_pad activation rows.
__host__ __device__ inline int small_stages(int m_pad) {
  int s = kSmallMaxStages;
  while (s > 2 && small_layout(m_pad, s).total > kSmallSmemLimit) --s;
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
// The small-M kernel (gsr_small.cu): `ctas` is even (clusters of two).
cudaError_t launch_small(const Params& p, int ctas, cudaStream_t stream);
cudaError_t prepare_small_kernel();
// The packed gather (gsr_pack.cu): one warp per CTA.
cudaError_t launch_pack(const PackParams& p, int ctas, cudaStream_t stream);
cudaError_t prepare_pack_kernel();

}  // namespace gsr
