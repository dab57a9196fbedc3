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
enum Sched : int { kSchedUniform = 0, kSchedStreamK = 1 };

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
  int sched;                    // kSchedUniform or kSchedStreamK
  int dp_tiles;                 // stream-K: tiles [0, dp_tiles) run whole, round-robin
  long long sk_iters;           // stream-K: k-blocks of tiles [dp_tiles, tiles)
  int sk_last;                  // stream-K: walk the whole tiles first, the range last
  int group_m;                  // raster group height, in m-tiles (1 = n fastest)
  int policy_a;                 // L2 policy of A-operand loads (kPolicy*)
  int policy_b;                 // L2 policy of B-operand loads (kPolicy*)
  int rps;                      // RS: rows per shard = ceil(M/R)
  int shard_kb_begin[kMaxShards + 1];  // AR/RS: first k-block of shard r
  int shard_mt_begin[kMaxShards + 1];  // AG: first 128-row half-tile of shard r
  int ag_halves;                // AG: 128-row half-tiles over all shards
  int ag_pad_shard;             // AG: a non-empty shard, read out of range (zeros)
                                // by the idle half of an odd last pair tile
  int shard_row_begin[kMaxShards + 1]; // AG: first output row of shard r
  int shard_rows[kMaxShards];          // AG: M_r
};

// Host-side launcher (defined with the kernel).
// cta_group 1: one CTA per 128-row tile; 2: a CTA pair (cluster of two) per
// 256-row tile. block_n is 128 or 256. `ctas` counts CTAs (even for pairs).
cudaError_t launch_gemm(const Params& p, int block_n, int cta_group, int ctas, cudaStream_t stream);
// Sets shared-memory limits and reports how many CTA pairs can be resident.
cudaError_t prepare_kernels(int device, int* pair_clusters);
size_t kernel_smem_bytes(int block_n, int cta_group);

}  // namespace gsr
