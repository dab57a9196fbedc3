// gsr_api.cu -- host side of the C ABI declared in include/gsr.h: plans,
// argument validation, kernel configuration, per-shard TMA descriptors and the
// launch. Nothing here allocates device memory.
//
// The plan mirrors the pages' init_gemm_rs_ar(max_M, N, all_reduce) singleton
// and its can_run/should_run checks (vLLM PR #53053 summary, model.py and
// call sites): shape checks happen once per call on the host, before any
// launch, and failures come back as status codes instead of exceptions that a
// caller must catch to fall back.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "gsr.h"
#include "gsr_params.h"

using gsr::BK;
using gsr::BM;
using gsr::kMaxShards;

struct gemm_shard_plan {
  int device;
  int sm_count;
  int64_t max_M, max_N, max_K;
  int max_R;
  int opt_split;       // 0 = heuristic
  int opt_block_n;     // 0 = heuristic
  int opt_max_ctas;    // 0 = one per SM
  int opt_raster_m;    // 0 = heuristic
  int opt_raster_n;    // 0 = raster by m-tile groups
  int opt_l2_hints;    // 0 = heuristic
  int opt_cta_group;   // 0 = heuristic
  int opt_schedule;    // 0 = heuristic, 1 = uniform, 2 = stream-K over the last one or two
                       // waves, 3/4 = stream-K over a partial last wave (its range first /
                       // last), 5 = split tail (GSR_OPT_SCHEDULE in gsr.h)
  int opt_small;       // 0 = heuristic, 1 = never use the small-M kernel, 2 = always when it applies
  int opt_small_rows;  // small-M kernel: W rows per tile (0 = heuristic)
  int opt_small_kz;    // small-M kernel: k-blocks per copy (0 = heuristic)
  int64_t l2_bytes;    // the device's L2 size
  int pair_clusters;   // CTA pairs that can be resident at once
  int quad_clusters;   // clusters of two CTA pairs that can be resident at once
  uint64_t timeout_ns;
};

namespace {

thread_local std::string g_last_error;

gsr_status fail(gsr_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

gsr_status ok() { return GSR_OK; }

gsr_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GSR_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so that the
// library itself has no link-time dependency on the driver library.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// cuStreamWriteValue32: a stream memory operation that writes a word without
// running a kernel.
typedef CUresult (*WriteValueFn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
WriteValueFn g_write_value = nullptr;
std::once_flag g_write_value_once;

WriteValueFn write_value_fn() {
  std::call_once(g_write_value_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_write_value = reinterpret_cast<WriteValueFn>(fn);
  });
  return g_write_value;
}

// Restores the caller's current device on scope exit.
struct DeviceScope {
  int prev = -1;
  bool switched = false;
  cudaError_t err = cudaSuccess;
  explicit DeviceScope(int dev) {
    err = cudaGetDevice(&prev);
    if (err == cudaSuccess && prev != dev) {
      err = cudaSetDevice(dev);
      switched = (err == cudaSuccess);
    }
  }
  ~DeviceScope() {
    if (switched) cudaSetDevice(prev);
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Most output tiles any call under the plan can have: block_n = 128, and in AG
// mode up to one extra partial m-tile per shard.
int64_t plan_max_tiles(const gemm_shard_plan* P) {
  // Per-shard rounding adds at most one m-tile per shard, and CTA-pair tiles
  // (two counters each) at most one more.
  return (cdiv(P->max_M, BM) + 2 * P->max_R) * cdiv(P->max_N, 128);
}

// The counter region has a fixed size per plan, so the partials of one call
// never overlap the counters of another.
size_t counters_bytes(const gemm_shard_plan* P) {
  return round256(4 * static_cast<size_t>(plan_max_tiles(P)));
}

struct Config {
  int block_n = 256;
  int cta_group = 1;
  int sched = gsr::kSchedUniform;
  int splits = 1;
  int64_t m_tiles = 0, n_tiles = 0, tiles = 0, kb_total = 0, units = 0;
  int64_t dp_tiles = 0, sk_iters = 0, slots = 0;   // slots: fp32 partial tiles per CTA half
  int sk_last = 0;
  int ctas = 0;
  int group_m = 1;
  int group_n = 0;
  int policy_a = gsr::kPolicyNormal;
  int policy_b = gsr::kPolicyNormal;
  size_t ws_bytes = 0;
  int small = 0;      // the small-M kernel (a CTA pair per tile of W rows)
  int m_pad = 0;      // small-M: activation rows rounded up to 16
  int stages = 0;     // small-M: ring depth
  int x_rows = 0;     // small-M: activation rows per CTA copy (the X box height)
  int kz = 1;         // small-M: k-blocks per copy (3-D boxes when > 1)
};


// Kernel configuration: a function of the shape (rows, N, per-shard sizes, R)
// and the device, never of the mode, so AR and RS on the same inputs run the
// same tiles, the same pieces and the same summation order (bit-identical rows).
// Three steps: the small-M kernel if it applies (small_m_config), else the main
// kernel's tile shape (choose_config itself) and its work schedule
// (uniform_schedule or tail_schedule).

// AG row granule: 128 rows (one per CTA tile), or 64 rows (two per CTA tile,
// possibly from neighbouring shards) when that needs fewer CTA tiles, i.e.
// when shards are multiples of 64 but not of 128 rows (448-row shards: 28
// CTA tiles of rows for 8 shards instead of 32). A function of the shard
// sizes only.
int ag_granule(int R, const int64_t* M_r) {
  int64_t g128 = 0, g64 = 0;
  for (int r = 0; r < R; ++r) {
    g128 += cdiv(M_r[r], 128);
    g64 += cdiv(M_r[r], 64);
  }
  return cdiv(g64, 2) < g128 ? 64 : 128;
}

// Small M (AR/RS, a decode-like batch of at most 256 rows): streaming W is
// the whole cost, so the small-M kernel runs every activation row against
// tiles of W rows, one CTA pair per tile over the whole K range. The tile
// height (the pair MMA's N) is the smallest multiple of 16 (up to 256) that
// covers N with every pair in the fewest waves, so that all SMs stream W
// (N = 7168 on 76 pairs: 96 rows, 75 tiles). Returns false when the kernel
// does not apply (or an option forces the main kernel).
bool small_m_config(const gemm_shard_plan* P, int mode, int64_t M, int64_t N, int R,
                    const int64_t* sizes, Config& c) {
  if (mode == gsr::kModeAG || M < 1 || M > gsr::kSmallMaxM || P->opt_small == 1) return false;
  int64_t kb = 0;
  for (int r = 0; r < R; ++r) kb += cdiv(sizes[r], BK);
  const bool forced = P->opt_split || P->opt_block_n || P->opt_cta_group || P->opt_schedule;
  if (kb < 1 || (P->opt_small != 2 && forced)) return false;
  c.small = 1;
  c.m_pad = static_cast<int>(std::max<int64_t>(16, cdiv(M, 16) * 16));
  const int cap = P->opt_max_ctas ? std::min(P->opt_max_ctas, P->sm_count) : P->sm_count;
  const int64_t clusters = std::max(cap / 2, 1);
  int64_t rows = P->opt_small_rows;
  if (!rows) {
    const int64_t waves = cdiv(N, gsr::kSmallMaxTileN * clusters);
    rows = std::min<int64_t>(gsr::kSmallMaxTileN, cdiv(cdiv(N, waves * clusters), 16) * 16);
  }
  c.block_n = static_cast<int>(rows);
  c.cta_group = 2;
  c.sched = gsr::kSchedSmall;
  c.splits = 1;
  // k-blocks per copy: the largest of 4, 3, 2, 1 (at most the option) that
  // leaves a ring of at least four stages in shared memory, where no shard
  // has a ragged k-block (a 3-D view of a shard would read the next row where
  // a 2-D box reads zeros). A shard's last copy may run past its k-blocks:
  // those are zero-filled (no memory read) and add nothing.
  c.kz = 1;
  bool whole = true;
  for (int r = 0; r < R; ++r) whole = whole && sizes[r] % BK == 0;
  for (int kz = P->opt_small_kz ? P->opt_small_kz : 4; whole && kz > 1 && c.kz == 1; --kz) {
    const int st = gsr::small_stages(static_cast<int>(M), c.block_n, kz);
    if (st >= 4 &&
        gsr::small_layout(static_cast<int>(M), c.block_n, st, kz).total <= gsr::kSmallSmemLimit)
      c.kz = kz;
  }
  // The kernel walks stages of kz k-blocks: kb_total counts them.
  kb = 0;
  for (int r = 0; r < R; ++r) kb += cdiv(cdiv(sizes[r], BK), c.kz);
  c.stages = gsr::small_stages(static_cast<int>(M), c.block_n, c.kz);
  c.x_rows = static_cast<int>(
      gsr::small_layout(static_cast<int>(M), c.block_n, c.stages, c.kz).x_rows);
  c.kb_total = kb;
  c.m_tiles = 1;
  c.n_tiles = cdiv(N, rows);
  c.tiles = c.n_tiles;
  c.units = c.tiles;
  c.ctas = static_cast<int>(2 * std::min<int64_t>(c.tiles, clusters));
  // Every cluster reads all of X and a disjoint slice of W.
  const int hints = P->opt_l2_hints;
  c.policy_a = (hints == 0 || hints == 2) ? gsr::kPolicyEvictLast
               : hints == 3               ? gsr::kPolicyEvictFirst
                                          : gsr::kPolicyNormal;
  c.policy_b = (hints == 0 || hints == 2) ? gsr::kPolicyEvictFirst
               : hints == 3               ? gsr::kPolicyEvictLast
                                          : gsr::kPolicyNormal;
  c.ws_bytes = gsr::kWsHeader + counters_bytes(P);
  return true;
}

// Uniform schedule: every tile cut into the same number of pieces, dealt
// round-robin (the default with fewer single-CTA tiles than SMs).
void uniform_schedule(const gemm_shard_plan* P, int64_t workers, Config& c) {
  c.sched = gsr::kSchedUniform;
  if (P->opt_split) {
    c.splits = static_cast<int>(std::min<int64_t>(P->opt_split, c.kb_total));
  } else if (c.tiles >= workers) {
    c.splits = 1;
  } else {
    int64_t sp = workers / std::max<int64_t>(c.tiles, 1);
    sp = std::min<int64_t>(sp, std::max<int64_t>(c.kb_total / 4, 1));
    c.splits = static_cast<int>(std::max<int64_t>(std::min<int64_t>(sp, 16), 1));
  }
  c.units = c.tiles * c.splits;
  c.dp_tiles = 0;
  c.sk_iters = 0;
  c.slots = c.splits > 1 ? c.units : 0;
  c.ctas = static_cast<int>(c.cta_group * std::min<int64_t>(c.units, workers));
}

// Whole tiles for every full wave, and for the partial last wave one of:
//  - a split tail, when it is at most half a wave and its pieces keep at least
//    60 % of the workers busy: each of its tiles cut into the same 2 or 3
//    k-pieces, one per worker, so the workers holding the same
//    piece of neighbouring tiles read the same k-blocks together (stream-K's
//    ranges start anywhere, share little in L2, and leave some workers with
//    two cut pieces). AR M = 1000, N = 7168: 36 tail tiles x 2 pieces on 76
//    pairs;
//  - whole tiles, when it is mostly full (at least 70 % of the workers:
//    sharing it out saves under 30 % of a tile, less than the cut tiles'
//    pieces cost; measured at 76, 89 and 95 % (AG MLA M = 3584, AR M = 4096,
//    AG KDA M = 3072) 2.3, 2.5 and 4 % faster; at 63 % stream-K still won by
//    1-2 %, at 53 % by 0.7 %), when there is too little to
//    share out, or too much for the kernel's 32-bit stream-K arithmetic
//    ((sk_iters + 1) * (workers + 1) must stay below 2^32);
//  - otherwise stream-K: its k-blocks cut evenly over every worker (schedule 2
//    shares out the last one or two waves instead).
void tail_schedule(const gemm_shard_plan* P, int64_t workers, Config& c) {
  const int64_t full = c.tiles / workers, rem = c.tiles % workers;
  c.splits = 1;
  c.units = c.tiles;
  c.sk_last = 0;
  const int64_t tail_split = rem ? std::min<int64_t>({3, workers / rem, c.kb_total}) : 0;
  const bool split_tail =
      rem != 0 && (P->opt_schedule == 5 ||
                   (P->opt_schedule == 0 && tail_split >= 2 && rem * tail_split * 10 >= workers * 6));
  if (split_tail) {
    c.sched = gsr::kSchedSplitTail;
    c.splits = static_cast<int>(std::max<int64_t>(tail_split, 1));
    c.dp_tiles = full * workers;
    c.sk_iters = 0;
    c.slots = rem * c.splits;
    c.ctas = static_cast<int>(c.cta_group * workers);
    return;
  }
  c.sched = gsr::kSchedStreamK;
  int64_t dp = c.tiles;
  if (rem != 0) {
    if (P->opt_schedule == 2)
      dp = full >= 2 ? (full - 1) * workers : 0;    // the last one or two waves
    else                                            // 0, 3, 4
      dp = full * workers;                          // only the partial last wave
  }
  int64_t sk_iters = (c.tiles - dp) * c.kb_total;
  const bool nearly_full = P->opt_schedule == 0 && rem * 10 >= workers * 7;
  if (nearly_full || (sk_iters > 0 && sk_iters < 4 * workers) ||
      (sk_iters + 1) * (workers + 1) >= (int64_t(1) << 32)) {
    dp = c.tiles;
    sk_iters = 0;
  }
  c.dp_tiles = dp;
  c.sk_iters = sk_iters;
  c.sk_last = P->opt_schedule == 4 ? 1 : 0;
  c.slots = sk_iters > 0 ? (c.tiles - dp) + workers - 1 : 0;
  c.ctas = static_cast<int>(c.cta_group *
                            (sk_iters > 0 ? workers : std::min<int64_t>(c.tiles, workers)));
}

Config choose_config(const gemm_shard_plan* P, int mode, int64_t M, int64_t N, int64_t K_ag, int R,
                     const int64_t* sizes) {
  Config c;
  if (small_m_config(P, mode, M, N, R, sizes, c)) return c;
  c.block_n = P->opt_block_n ? P->opt_block_n : (N <= 128 ? 128 : 256);
  // Tile rows: 128 per CTA; a CTA pair (cta_group 2) covers 256. AG tiles never
  // cross a shard.
  // AG counts 128-row half-tiles per shard; a pair tile takes two consecutive
  // half-tiles, which may belong to neighbouring shards.
  auto count_m_tiles = [&](int64_t cg) {
    int64_t halves = 0;
    if (mode == gsr::kModeAG) {
      const int gran = ag_granule(R, sizes);
      for (int r = 0; r < R; ++r) halves += cdiv(sizes[r], gran);
      halves = cdiv(halves, BM / gran);
    } else {
      halves = cdiv(M, BM);
    }
    return cdiv(halves, cg);
  };
  int64_t rows = 0;
  if (mode == gsr::kModeAG) {
    c.kb_total = cdiv(K_ag, BK);
    for (int r = 0; r < R; ++r) rows += sizes[r];
  } else {
    for (int r = 0; r < R; ++r) c.kb_total += cdiv(sizes[r], BK);
    rows = M;
  }
  c.n_tiles = cdiv(N, c.block_n);
  const int64_t mt1 = count_m_tiles(1), mt2 = count_m_tiles(2);
  const int cap = P->opt_max_ctas ? std::min(P->opt_max_ctas, P->sm_count) : P->sm_count;
  // One 128-row tile of rows (M <= 128, decode-like): single CTAs with
  // 128-column tiles, cut into uniform pieces, measured fastest (every CTA
  // streams its slice of W; no pair half sits idle).
  const bool one_row_tile = mt1 == 1 && mt1 * c.n_tiles < P->sm_count;
  if (one_row_tile && !P->opt_block_n && !P->opt_cta_group) {
    c.block_n = 128;
    c.n_tiles = cdiv(N, c.block_n);
  }

  // CTA pairs halve each SM's bytes of B per flop and deepen the smem ring; they
  // run when there are at least as many single-CTA tiles as SMs and 256-row
  // tiles waste no more rows than 128-row tiles do (only an odd number of
  // 128-row halves leaves one half idle).
  const bool pairs_fit = P->pair_clusters > 0 && cap >= 2;
  // With fewer single-CTA tiles than SMs (small M) the kernel streams W at HBM
  // bandwidth: CTA pairs cut into a few uniform pieces measured fastest there
  // (fewer partial tiles to sum than stream-K's pieces of every tile).
  const bool small = mt1 * c.n_tiles < P->sm_count;
  if (P->opt_cta_group) {
    const bool quads_fit = P->quad_clusters > 0 && cap >= 4;
    c.cta_group = (P->opt_cta_group == 4 && quads_fit)   ? 4
                  : (P->opt_cta_group >= 2 && pairs_fit) ? 2
                                                         : 1;
  } else if (small) {
    c.cta_group = pairs_fit && c.block_n == 256 && !one_row_tile ? 2 : 1;
  } else {
    const double eff1 = static_cast<double>(rows) / (mt1 * BM);
    const double eff2 = static_cast<double>(rows) / (mt2 * 2 * BM);
    c.cta_group = (pairs_fit && eff2 >= 0.9 * eff1) ? 2 : 1;   // pairs measured 10-20 % faster
  }
  // 192-column tiles exist for CTA pairs only.
  if (c.block_n == 192 && c.cta_group == 1) {
    c.block_n = 256;
    c.n_tiles = cdiv(N, c.block_n);
  }
  c.m_tiles = c.cta_group == 4 ? count_m_tiles(4) : c.cta_group == 2 ? mt2 : mt1;
  c.tiles = c.m_tiles * c.n_tiles;
  const int64_t workers =
      c.cta_group == 4   ? std::min<int64_t>(cap / 4, P->quad_clusters)
      : c.cta_group == 2 ? std::min<int64_t>(cap / 2, P->pair_clusters)
                         : static_cast<int64_t>(cap);
  // 192-column pair tiles where 256 leaves a narrow last column of tiles (N a
  // multiple of 192 but not of 256, like N = 3648 = 19 x 192) and 192 fills at
  // most four whole waves, so no tile is cut. Measured at AG N = 3648 against
  // 256-column tiles: M = 2048 (two waves) 4 %, M = 3072 (three) 2 % and
  // M = 4096 (four) 4 % faster; at eight waves (M = 8192) within 1 %, and at
  // large M 192-column tiles are slower.
  if (!P->opt_block_n && c.cta_group == 2 && c.block_n == 256 && N % 256 != 0 && N % 192 == 0) {
    const int64_t t192 = c.m_tiles * (N / 192);
    if (workers > 0 && t192 % workers == 0 && t192 / workers <= 4) {
      c.block_n = 192;
      c.n_tiles = N / 192;
      c.tiles = t192;
    }
  }

  if (P->opt_split || P->opt_schedule == 1 || (P->opt_schedule == 0 && small))
    uniform_schedule(P, workers, c);
  else
    tail_schedule(P, workers, c);
  c.ctas = std::max(c.ctas, c.cta_group);

  // Raster: groups of group_m m-tiles, m fastest inside a group, so a wave of
  // concurrent CTAs covers about group_m x (#workers / group_m) tiles and reads
  // that many A row-blocks and W column-blocks once each from HBM. Eight
  // m-tiles keep a wave's working set smallest (about 8 + 76 / 8 blocks of
  // 3.7 MB at K = 7168): measured at M = 32768, the fewest HBM reads (AG 3.1 GB
  // per launch, against 3.3 GB at 16, 4.2 GB at 4, 5.6 GB at 32) and the most
  // throughput at the power limit.
  c.group_m = P->opt_raster_m ? P->opt_raster_m : 8;
  c.group_n = P->opt_raster_n;
  switch (P->opt_l2_hints) {
    case 0: {
      // A evict-last and B evict-first where both operands fit in L2 at once
      // (mid M: a few waves re-read each tile of A and of W). Measured with an
      // L2 flush before each launch: AG N = 3648, M = 2048..4096, 2-5 %
      // faster; AR o_proj M = 1000 3 %; AG N = 6288 M = 2048 unchanged.
      // Where they do not fit, the hints kept A lines that the raster order
      // does not reuse soon: 5-7 % slower at M = 32768, mixed in between.
      int64_t K = K_ag;
      if (mode != gsr::kModeAG) {
        K = 0;
        for (int r = 0; r < R; ++r) K += sizes[r];
      }
      const bool fits = 2 * (rows + N) * K <= P->l2_bytes;
      c.policy_a = fits ? gsr::kPolicyEvictLast : gsr::kPolicyNormal;
      c.policy_b = fits ? gsr::kPolicyEvictFirst : gsr::kPolicyNormal;
      break;
    }
    case 2:
      c.policy_a = gsr::kPolicyEvictLast;
      c.policy_b = gsr::kPolicyEvictFirst;
      break;
    case 3:
      c.policy_a = gsr::kPolicyEvictFirst;
      c.policy_b = gsr::kPolicyEvictLast;
      break;
    default:
      c.policy_a = gsr::kPolicyNormal;
      c.policy_b = gsr::kPolicyNormal;
      break;
  }
  size_t bytes = gsr::kWsHeader + counters_bytes(P);
  bytes += static_cast<size_t>(c.slots) * c.cta_group * BM * c.block_n * sizeof(float);
  c.ws_bytes = bytes;
  return c;
}

// The same rows viewed as {64 columns, rows, cols / 64 k-blocks} (cols a
// multiple of 64), with a box of kz k-blocks: one copy lands kz consecutive
// 128B-swizzled tiles of box_rows rows, one after the other.
CUresult encode_kmajor_3d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows,
                          int kz) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(BK), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(cols / BK)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2, static_cast<cuuint64_t>(BK) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(kz)};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_kmajor(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// GSR_LOG_CONFIG (set and not "0"): every call that passes validation writes
// its configuration to stderr, one line, before the launch. Read once.
bool log_config_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GSR_LOG_CONFIG");
    return v != nullptr && v[0] != '\0' && std::strcmp(v, "0") != 0;
  }();
  return on;
}

void log_config(const char* mode, int64_t M, int64_t N, int R, const Config& c) {
  if (!log_config_enabled()) return;
  const char* sched = c.small                            ? "small_m"
                      : c.sched == gsr::kSchedSplitTail ? "split_tail"
                      : c.sched == gsr::kSchedStreamK   ? "stream_k"
                                                        : "uniform";
  std::fprintf(stderr,
               "gsr: %s M=%lld N=%lld R=%d kernel=%s block_n=%d cta_group=%d schedule=%s "
               "split=%d tiles=%lld dp_tiles=%lld sk_iters=%lld ctas=%d workspace=%zu\n",
               mode, (long long)M, (long long)N, R, c.small ? "small" : "main", c.block_n,
               c.cta_group, sched, c.splits, (long long)c.tiles, (long long)c.dp_tiles,
               (long long)c.sk_iters, c.ctas, c.ws_bytes);
}

gsr_status check_plan(const gemm_shard_plan* P) {
  if (!P) return fail(GSR_ERR_INVALID_VALUE, "plan is NULL");
  return ok();
}

gsr_status check_ws(const Config& c, const void* ws, size_t ws_bytes) {
  if (!ws) return fail(GSR_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(GSR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < c.ws_bytes)
    return fail(GSR_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", ws_bytes,
                c.ws_bytes);
  return ok();
}

void fill_common(gsr::Params& p, const gemm_shard_plan* P, const Config& c, int mode, int R,
                 int64_t M, int64_t N, void* ws) {
  p.mode = mode;
  p.R = R;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.m_tiles = static_cast<int>(c.m_tiles);
  p.n_tiles = static_cast<int>(c.n_tiles);
  p.tiles = static_cast<int>(c.tiles);
  p.kb_total = static_cast<int>(c.kb_total);
  p.splits = c.splits;
  p.units = static_cast<int>(c.units);
  p.sched = c.sched;
  p.dp_tiles = static_cast<int>(c.dp_tiles);
  p.sk_iters = c.sk_iters;
  p.sk_last = c.sk_last;
  p.group_m = c.group_m;
  p.group_n = c.group_n;
  p.policy_a = c.policy_a;
  p.policy_b = c.policy_b;
  p.m_pad = c.m_pad;
  p.stages = c.stages;
  p.tile_rows = c.small ? c.block_n : 0;
  p.small_kz = c.kz;
  p.ag_gran = BM;   // AG sets its own
  p.timeout_ns = P->timeout_ns;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.status = reinterpret_cast<uint32_t*>(w);
  p.counters = reinterpret_cast<uint32_t*>(w + gsr::kWsHeader);
  p.partials = reinterpret_cast<float*>(w + gsr::kWsHeader + counters_bytes(P));
}

gsr_status launch(const gemm_shard_plan* P, const gsr::Params& p, const Config& c,
                  gsr_stream_t stream) {
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: arguments are valid, nothing launched");
  DeviceScope scope(P->device);
  if (scope.err != cudaSuccess) return cuda_fail(scope.err, "selecting the plan's device");
  cudaError_t e = c.small ? gsr::launch_small(p, c.ctas, reinterpret_cast<cudaStream_t>(stream))
                          : gsr::launch_gemm(p, c.block_n, c.cta_group, c.ctas,
                                             reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return ok();
}

// Shared validation of the K-sharded (AR/RS) argument lists.
gsr_status check_ksharded(const gemm_shard_plan* P, int64_t M, int64_t N, int R, const int64_t* K_r,
                          const void* const* X_r, const void* const* W_r) {
  if (M < 0) return fail(GSR_ERR_INVALID_VALUE, "M must be >= 0 (got %lld)", (long long)M);
  if (M > P->max_M)
    return fail(GSR_ERR_INVALID_VALUE, "M=%lld exceeds the plan's max_M=%lld", (long long)M,
                (long long)P->max_M);
  if (N < 8 || N % 8)
    return fail(GSR_ERR_INVALID_VALUE, "N must be a positive multiple of 8 (got %lld)", (long long)N);
  if (N > P->max_N)
    return fail(GSR_ERR_INVALID_VALUE, "N=%lld exceeds the plan's max_N=%lld", (long long)N,
                (long long)P->max_N);
  if (R < 1 || R > P->max_R)
    return fail(GSR_ERR_INVALID_VALUE, "R=%d outside 1..%d", R, P->max_R);
  if (!K_r || !X_r || !W_r)
    return fail(GSR_ERR_INVALID_VALUE, "K_r, X_r and W_r must not be NULL");
  int64_t K = 0;
  for (int r = 0; r < R; ++r) {
    if (K_r[r] < 8 || K_r[r] % 8)
      return fail(GSR_ERR_INVALID_VALUE, "K_r[%d]=%lld must be a positive multiple of 8", r,
                  (long long)K_r[r]);
    // With M == 0 the activation shards have no rows and may be NULL.
    if ((M > 0 && !X_r[r]) || !W_r[r])
      return fail(GSR_ERR_INVALID_VALUE, "shard %d has a NULL operand pointer", r);
    if (!aligned16(X_r[r]) || !aligned16(W_r[r]))
      return fail(GSR_ERR_INVALID_VALUE, "shard %d operand is not 16-byte aligned", r);
    K += K_r[r];
  }
  if (K > P->max_K)
    return fail(GSR_ERR_INVALID_VALUE, "sum of K_r = %lld exceeds the plan's max_K=%lld",
                (long long)K, (long long)P->max_K);
  return ok();
}

gsr_status run_ksharded(const gemm_shard_plan* P, int mode, int64_t M, int64_t N, int R,
                        const int64_t* K_r, const void* const* X_r, const void* const* W_r,
                        void* Y, void* const* Y_r, void* ws, size_t ws_bytes,
                        gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  s = check_ksharded(P, M, N, R, K_r, X_r, W_r);
  if (s) return s;
  // Outputs may be NULL only when there is no row to write (M == 0).
  if (mode == gsr::kModeAR) {
    if ((M > 0 && !Y) || !aligned16(Y))
      return fail(GSR_ERR_INVALID_VALUE, "Y must be non-NULL and 16-byte aligned");
  } else {
    if (!Y_r) return fail(GSR_ERR_INVALID_VALUE, "Y_r must not be NULL");
    for (int r = 0; r < R; ++r)
      if ((M > 0 && !Y_r[r]) || !aligned16(Y_r[r]))
        return fail(GSR_ERR_INVALID_VALUE, "Y_r[%d] must be non-NULL and 16-byte aligned", r);
  }
  // Replicated AR is AR with another epilogue: the same configuration.
  const Config c = choose_config(P, mode == gsr::kModeARRep ? gsr::kModeAR : mode, M, N, 0, R, K_r);
  s = check_ws(c, ws, ws_bytes);
  if (s) return s;
  if (M == 0) return ok();
  log_config(mode == gsr::kModeAR ? "ar" : mode == gsr::kModeRS ? "rs" : "ar_replicated", M, N, R, c);
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: arguments are valid, nothing launched");
  if (!encode_fn()) return fail(GSR_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is unavailable");

  gsr::Params p;
  std::memset(&p, 0, sizeof p);
  fill_common(p, P, c, mode, R, M, N, ws);
  int kb = 0;
  for (int r = 0; r < R; ++r) {
    p.shard_kb_begin[r] = kb;
    // The small-M kernel counts stages of kz k-blocks (kz = 1 elsewhere).
    kb += static_cast<int>(cdiv(cdiv(K_r[r], BK), c.kz));
    // A small-M CTA loads up to x_rows activation rows at once, kz k-blocks a copy.
    CUresult cr = c.kz > 1 ? encode_kmajor_3d(&p.tmap_a[r], X_r[r], M, K_r[r], c.x_rows, c.kz)
                           : encode_kmajor(&p.tmap_a[r], X_r[r], M, K_r[r], c.small ? c.x_rows : BM);
    if (cr != CUDA_SUCCESS) return fail(GSR_ERR_CUDA, "encoding X_r[%d] descriptor failed (%d)", r, (int)cr);
    cr = c.kz > 1 ? encode_kmajor_3d(&p.tmap_b[r], W_r[r], N, K_r[r], c.block_n / 2, c.kz)
                  : encode_kmajor(&p.tmap_b[r], W_r[r], N, K_r[r], c.block_n / c.cta_group);
    if (cr != CUDA_SUCCESS) return fail(GSR_ERR_CUDA, "encoding W_r[%d] descriptor failed (%d)", r, (int)cr);
  }
  for (int r = R; r <= kMaxShards; ++r) p.shard_kb_begin[r] = kb;
  if (mode == gsr::kModeAR) {
    p.y = static_cast<uint16_t*>(Y);
  } else {
    p.rps = static_cast<int>(cdiv(M, R));
    for (int r = 0; r < R; ++r) p.y_r[r] = static_cast<uint16_t*>(Y_r[r]);
  }
  if (mode == gsr::kModeARRep) p.mode = gsr::kModeARRep;
  return launch(P, p, c, stream);
}

}  // namespace

extern "C" {

const char* gsr_last_error_string(void) { return g_last_error.c_str(); }

static gsr_status check_maxima(gemm_shard_plan** out, int64_t max_M, int64_t max_N, int64_t max_K,
                               int max_R) {
  if (!out) return fail(GSR_ERR_INVALID_VALUE, "out is NULL");
  *out = nullptr;
  if (max_M < 1 || max_N < 8 || max_K < 8 || max_N % 8 || max_K % 8)
    return fail(GSR_ERR_INVALID_VALUE,
                "maxima must be >= 1 (max_M) or positive multiples of 8 (max_N, max_K)");
  if (max_M > INT32_MAX - BM || max_N > INT32_MAX - 256 || max_K > INT32_MAX - BK)
    return fail(GSR_ERR_INVALID_VALUE, "maxima must stay below 2^31");
  if (max_R < 1 || max_R > kMaxShards)
    return fail(GSR_ERR_INVALID_VALUE, "max_R=%d outside 1..%d", max_R, kMaxShards);
  // The kernels count tiles and pieces (up to 16 per tile) in 32-bit integers.
  const int64_t tiles = (cdiv(max_M, BM) + 2 * max_R) * cdiv(max_N, 128);
  if (tiles > INT32_MAX / 16)
    return fail(GSR_ERR_INVALID_VALUE,
                "max_M x max_N gives %lld output tiles of 128 x 128; at most %d are supported",
                (long long)tiles, INT32_MAX / 16);
  return ok();
}

static gemm_shard_plan* new_plan(int device, int sm_count, int64_t max_M, int64_t max_N,
                                 int64_t max_K, int max_R) {
  gemm_shard_plan* P = new gemm_shard_plan();
  P->device = device;
  P->sm_count = sm_count;
  P->max_M = max_M;
  P->max_N = max_N;
  P->max_K = max_K;
  P->max_R = max_R;
  P->opt_split = 0;
  P->opt_block_n = 0;
  P->opt_max_ctas = 0;
  P->opt_raster_m = 0;
  P->opt_raster_n = 0;
  P->opt_l2_hints = 0;
  P->opt_cta_group = 0;
  P->opt_schedule = 0;
  P->opt_small = 0;
  P->opt_small_rows = 0;
  P->opt_small_kz = 0;
  P->l2_bytes = int64_t(126) << 20;  // host plans: a GB300's L2
  P->pair_clusters = sm_count / 2;   // host plans: every SM pairs up
  P->quad_clusters = sm_count / 4;
  P->timeout_ns = 2000000000ull;
  return P;
}

gsr_status gemm_shard_plan_create_host(gemm_shard_plan** out, int sm_count, int64_t max_M,
                                       int64_t max_N, int64_t max_K, int max_R) {
  gsr_status s = check_maxima(out, max_M, max_N, max_K, max_R);
  if (s) return s;
  if (sm_count < 1) return fail(GSR_ERR_INVALID_VALUE, "sm_count must be >= 1");
  *out = new_plan(-1, sm_count, max_M, max_N, max_K, max_R);
  return ok();
}

gsr_status gemm_shard_plan_create(gemm_shard_plan** out, int device, int64_t max_M, int64_t max_N,
                                  int64_t max_K, int max_R) {
  gsr_status s = check_maxima(out, max_M, max_N, max_K, max_R);
  if (s) return s;
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess) return fail(GSR_ERR_UNSUPPORTED, "no usable CUDA device: %s", cudaGetErrorString(e));
  if (device < 0 || device >= count)
    return fail(GSR_ERR_INVALID_VALUE, "device %d outside 0..%d", device, count - 1);
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3)
    return fail(GSR_ERR_UNSUPPORTED, "device %d is compute capability %d.%d; this library is built for sm_103a",
                device, prop.major, prop.minor);
  if (!encode_fn()) return fail(GSR_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is unavailable");
  int pair_clusters = 0, quad_clusters = 0;
  {
    DeviceScope scope(device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cudaSetDevice");
    const size_t need = std::max(gsr::kernel_smem_bytes(256, 1), gsr::kernel_smem_bytes(256, 2));
    if (static_cast<size_t>(prop.sharedMemPerBlockOptin) < need)
      return fail(GSR_ERR_UNSUPPORTED, "device allows %zu bytes of shared memory per block; %zu needed",
                  static_cast<size_t>(prop.sharedMemPerBlockOptin), need);
    e = gsr::prepare_kernels(device, &pair_clusters, &quad_clusters);
    if (e == cudaSuccess) e = gsr::prepare_small_kernel();
    if (e == cudaSuccess) e = gsr::prepare_pack_kernel();
    if (e != cudaSuccess) return cuda_fail(e, "configuring the kernels");
  }
  *out = new_plan(device, prop.multiProcessorCount, max_M, max_N, max_K, max_R);
  (*out)->l2_bytes = prop.l2CacheSize;
  (*out)->pair_clusters = pair_clusters;
  (*out)->quad_clusters = quad_clusters;
  return ok();
}

gsr_status gemm_shard_plan_destroy(gemm_shard_plan* plan) {
  delete plan;
  return ok();
}

gsr_status gemm_shard_plan_set_option(gemm_shard_plan* plan, gsr_option option, int64_t value) {
  gsr_status s = check_plan(plan);
  if (s) return s;
  switch (option) {
    case GSR_OPT_SPLIT_K:
      if (value < 0 || value > 16) return fail(GSR_ERR_INVALID_VALUE, "split must be 0..16");
      plan->opt_split = static_cast<int>(value);
      return ok();
    case GSR_OPT_BLOCK_N:
      if (value != 0 && value != 128 && value != 192 && value != 256)
        return fail(GSR_ERR_INVALID_VALUE, "block_n must be 0, 128, 192 or 256");
      plan->opt_block_n = static_cast<int>(value);
      return ok();
    case GSR_OPT_TIMEOUT_NS:
      if (value < 0) return fail(GSR_ERR_INVALID_VALUE, "timeout must be >= 0");
      plan->timeout_ns = value ? static_cast<uint64_t>(value) : 2000000000ull;
      return ok();
    case GSR_OPT_MAX_CTAS:
      if (value < 0 || value > INT32_MAX) return fail(GSR_ERR_INVALID_VALUE, "max_ctas must be >= 0");
      plan->opt_max_ctas = static_cast<int>(value);
      return ok();
    case GSR_OPT_RASTER_M:
      if (value < 0 || value > 64) return fail(GSR_ERR_INVALID_VALUE, "raster_m must be 0..64");
      plan->opt_raster_m = static_cast<int>(value);
      return ok();
    case GSR_OPT_RASTER_N:
      if (value < 0 || value > 64) return fail(GSR_ERR_INVALID_VALUE, "raster_n must be 0..64");
      plan->opt_raster_n = static_cast<int>(value);
      return ok();
    case GSR_OPT_L2_HINTS:
      if (value < 0 || value > 3) return fail(GSR_ERR_INVALID_VALUE, "l2_hints must be 0..3");
      plan->opt_l2_hints = static_cast<int>(value);
      return ok();
    case GSR_OPT_CTA_GROUP:
      if (value < 0 || value > 4 || value == 3)
        return fail(GSR_ERR_INVALID_VALUE, "cta_group must be 0, 1, 2 or 4");
      plan->opt_cta_group = static_cast<int>(value);
      return ok();
    case GSR_OPT_SCHEDULE:
      if (value < 0 || value > 5) return fail(GSR_ERR_INVALID_VALUE, "schedule must be 0..5");
      plan->opt_schedule = static_cast<int>(value);
      return ok();
    case GSR_OPT_SMALL_M:
      if (value < 0 || value > 2) return fail(GSR_ERR_INVALID_VALUE, "small_m must be 0..2");
      plan->opt_small = static_cast<int>(value);
      return ok();
    case GSR_OPT_SMALL_KBLOCKS:
      if (value < 0 || value > 4)
        return fail(GSR_ERR_INVALID_VALUE, "small_kblocks must be 0..4");
      plan->opt_small_kz = static_cast<int>(value);
      return ok();
    case GSR_OPT_SMALL_TILE_ROWS:
      if (value < 0 || value > gsr::kSmallMaxTileN || value % 16)
        return fail(GSR_ERR_INVALID_VALUE, "small_tile_rows must be 0 or a multiple of 16 up to %d",
                    gsr::kSmallMaxTileN);
      plan->opt_small_rows = static_cast<int>(value);
      return ok();
  }
  return fail(GSR_ERR_INVALID_VALUE, "unknown option %d", static_cast<int>(option));
}

size_t gemm_shard_workspace_size(const gemm_shard_plan* P) {
  if (!P) return 0;
  // Worst case over every shape within the plan: most tiles at block_n = 128
  // (AG adds up to one partial m-tile per shard), and split-K partials for the
  // heuristic (pieces only while tiles < SMs, so at most one slot per SM) or
  // for a forced split on every tile.
  const int64_t max_tiles = plan_max_tiles(P);
  size_t bytes = gsr::kWsHeader + counters_bytes(P);
  const size_t slot = static_cast<size_t>(BM) * 256 * sizeof(float);
  if (P->opt_split > 1) {
    bytes += static_cast<size_t>(max_tiles) * P->opt_split * slot;
  } else if (P->opt_schedule == 1) {
    // uniform heuristic: pieces only while tiles < workers, one slot per CTA
    bytes += static_cast<size_t>(P->sm_count) * slot;
  } else {
    // stream-K: fewer than two waves of tiles are cut, plus one piece per
    // worker boundary: under three slots per CTA
    bytes += static_cast<size_t>(3) * P->sm_count * slot;
  }
  return bytes;
}

gsr_status gemm_shard_workspace_init(const gemm_shard_plan* P, void* ws, size_t ws_bytes,
                                     gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  if (!ws) return fail(GSR_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(GSR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  const size_t zero_bytes = gsr::kWsHeader + counters_bytes(P);
  if (ws_bytes < zero_bytes)
    return fail(GSR_ERR_WORKSPACE, "workspace too small: %zu bytes given, at least %zu needed",
                ws_bytes, zero_bytes);
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: nothing to initialise");
  DeviceScope scope(P->device);
  if (scope.err != cudaSuccess) return cuda_fail(scope.err, "selecting the plan's device");
  cudaError_t e = cudaMemsetAsync(ws, 0, zero_bytes, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return ok();
}

gsr_status gemm_ar(const gemm_shard_plan* plan, int64_t M, int64_t N, int R, const int64_t* K_r,
                   const void* const* X_r, const void* const* W_r, void* Y, void* ws,
                   size_t ws_bytes, gsr_stream_t stream) {
  return run_ksharded(plan, gsr::kModeAR, M, N, R, K_r, X_r, W_r, Y, nullptr, ws, ws_bytes, stream);
}

gsr_status gemm_ar_replicated(const gemm_shard_plan* plan, int64_t M, int64_t N, int R,
                              const int64_t* K_r, const void* const* X_r, const void* const* W_r,
                              void* const* Y_r, void* ws, size_t ws_bytes, gsr_stream_t stream) {
  return run_ksharded(plan, gsr::kModeARRep, M, N, R, K_r, X_r, W_r, nullptr, Y_r, ws, ws_bytes,
                      stream);
}

gsr_status gemm_rs(const gemm_shard_plan* plan, int64_t M, int64_t N, int R, const int64_t* K_r,
                   const void* const* X_r, const void* const* W_r, void* const* Y_r, void* ws,
                   size_t ws_bytes, gsr_stream_t stream) {
  return run_ksharded(plan, gsr::kModeRS, M, N, R, K_r, X_r, W_r, nullptr, Y_r, ws, ws_bytes,
                      stream);
}

static gsr_status run_ag(const gemm_shard_plan* P, int64_t N, int64_t K, int R, const int64_t* M_r,
                         const void* const* A_r, const void* W, void* Y, const uint32_t* ready,
                         uint32_t epoch, void* ws, size_t ws_bytes, gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  if (N < 8 || N % 8)
    return fail(GSR_ERR_INVALID_VALUE, "N must be a positive multiple of 8 (got %lld)", (long long)N);
  if (N > P->max_N)
    return fail(GSR_ERR_INVALID_VALUE, "N=%lld exceeds the plan's max_N=%lld", (long long)N,
                (long long)P->max_N);
  if (K < 8 || K % 8)
    return fail(GSR_ERR_INVALID_VALUE, "K must be a positive multiple of 8 (got %lld)", (long long)K);
  if (K > P->max_K)
    return fail(GSR_ERR_INVALID_VALUE, "K=%lld exceeds the plan's max_K=%lld", (long long)K,
                (long long)P->max_K);
  if (R < 1 || R > P->max_R) return fail(GSR_ERR_INVALID_VALUE, "R=%d outside 1..%d", R, P->max_R);
  if (!M_r || !A_r) return fail(GSR_ERR_INVALID_VALUE, "M_r and A_r must not be NULL");
  if (!W || !aligned16(W)) return fail(GSR_ERR_INVALID_VALUE, "W must be non-NULL and 16-byte aligned");
  int64_t M = 0;
  for (int r = 0; r < R; ++r) {
    if (M_r[r] < 0) return fail(GSR_ERR_INVALID_VALUE, "M_r[%d] must be >= 0", r);
    if (M_r[r] > 0 && (!A_r[r] || !aligned16(A_r[r])))
      return fail(GSR_ERR_INVALID_VALUE, "A_r[%d] must be non-NULL and 16-byte aligned", r);
    M += M_r[r];
  }
  if ((M > 0 && !Y) || !aligned16(Y))
    return fail(GSR_ERR_INVALID_VALUE, "Y must be non-NULL and 16-byte aligned");
  if (M > P->max_M)
    return fail(GSR_ERR_INVALID_VALUE, "sum of M_r = %lld exceeds the plan's max_M=%lld",
                (long long)M, (long long)P->max_M);
  const Config c = choose_config(P, gsr::kModeAG, M, N, K, R, M_r);
  s = check_ws(c, ws, ws_bytes);
  if (s) return s;
  if (M == 0) return ok();
  log_config(ready ? "ag_flagged" : "ag", M, N, R, c);
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: arguments are valid, nothing launched");
  if (!encode_fn()) return fail(GSR_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is unavailable");

  gsr::Params p;
  std::memset(&p, 0, sizeof p);
  fill_common(p, P, c, gsr::kModeAG, R, M, N, ws);
  int mt = 0, row = 0;
  p.ag_pad_shard = -1;
  p.ag_gran = ag_granule(R, M_r);
  for (int r = 0; r < R; ++r) {
    p.shard_mt_begin[r] = mt;        // in row granules, each inside one shard
    p.shard_row_begin[r] = row;
    p.shard_rows[r] = static_cast<int>(M_r[r]);
    mt += static_cast<int>(cdiv(M_r[r], p.ag_gran));
    row += static_cast<int>(M_r[r]);
    if (M_r[r] > 0 && p.ag_pad_shard < 0) p.ag_pad_shard = r;
    if (M_r[r] > 0) {
      CUresult cr = encode_kmajor(&p.tmap_a[r], A_r[r], M_r[r], K, p.ag_gran);
      if (cr != CUDA_SUCCESS) return fail(GSR_ERR_CUDA, "encoding A_r[%d] descriptor failed (%d)", r, (int)cr);
    }
  }
  for (int r = R; r <= kMaxShards; ++r) {
    p.shard_mt_begin[r] = mt;
    p.shard_row_begin[r] = row;
  }
  p.ag_halves = mt;
  CUresult cr = encode_kmajor(&p.tmap_b[0], W, N, K, c.block_n / c.cta_group);
  if (cr != CUDA_SUCCESS) return fail(GSR_ERR_CUDA, "encoding the W descriptor failed (%d)", (int)cr);
  p.y = static_cast<uint16_t*>(Y);
  p.ready = ready;
  p.epoch = epoch;
  return launch(P, p, c, stream);
}

gsr_status gemm_ag(const gemm_shard_plan* P, int64_t N, int64_t K, int R, const int64_t* M_r,
                   const void* const* A_r, const void* W, void* Y, void* ws, size_t ws_bytes,
                   gsr_stream_t stream) {
  return run_ag(P, N, K, R, M_r, A_r, W, Y, nullptr, 0, ws, ws_bytes, stream);
}

gsr_status gemm_ag_flagged(const gemm_shard_plan* P, int64_t N, int64_t K, int R,
                           const int64_t* M_r, const void* const* A_r, const void* W, void* Y,
                           const uint32_t* ready, uint32_t epoch, void* ws, size_t ws_bytes,
                           gsr_stream_t stream) {
  if (!ready || (reinterpret_cast<uintptr_t>(ready) & 3u))
    return fail(GSR_ERR_INVALID_VALUE, "ready must be a non-NULL, 4-byte aligned device array");
  return run_ag(P, N, K, R, M_r, A_r, W, Y, ready, epoch, ws, ws_bytes, stream);
}

gsr_status gemm_shard_signal(const gemm_shard_plan* P, uint32_t* flag, uint32_t value,
                             gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  if (!flag || (reinterpret_cast<uintptr_t>(flag) & 3u))
    return fail(GSR_ERR_INVALID_VALUE, "flag must be a non-NULL, 4-byte aligned device word");
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: nothing to signal");
  WriteValueFn fn = write_value_fn();
  if (!fn) return fail(GSR_ERR_UNSUPPORTED, "cuStreamWriteValue32 is unavailable");
  DeviceScope scope(P->device);
  if (scope.err != cudaSuccess) return cuda_fail(scope.err, "selecting the plan's device");
  // CU_STREAM_WRITE_VALUE_DEFAULT (0): the write is preceded by a system-wide
  // memory fence, so data written by earlier work on the stream is visible first.
  CUresult r = fn(reinterpret_cast<CUstream>(stream), reinterpret_cast<CUdeviceptr>(flag), value, 0);
  if (r != CUDA_SUCCESS) return fail(GSR_ERR_CUDA, "cuStreamWriteValue32 failed (%d)", (int)r);
  return ok();
}

gsr_status gemm_shard_pack_gather(const gemm_shard_plan* P, int R, const int64_t* M_r, int T,
                                  int64_t H, const void* const* S, int64_t rows_out, void* Pout,
                                  void* ws, size_t ws_bytes, gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  if (R < 1 || R > P->max_R) return fail(GSR_ERR_INVALID_VALUE, "R=%d outside 1..%d", R, P->max_R);
  if (T < 1 || T > gsr::kMaxPackStates)
    return fail(GSR_ERR_INVALID_VALUE, "T=%d outside 1..%d", T, gsr::kMaxPackStates);
  if (H < 8 || H % 8)
    return fail(GSR_ERR_INVALID_VALUE, "H must be a positive multiple of 8 (got %lld)", (long long)H);
  if (!M_r || !S) return fail(GSR_ERR_INVALID_VALUE, "M_r and S must not be NULL");
  int64_t total = 0;
  for (int r = 0; r < R; ++r) {
    if (M_r[r] < 0) return fail(GSR_ERR_INVALID_VALUE, "M_r[%d] must be >= 0", r);
    total += M_r[r];
  }
  if (rows_out < 0 || rows_out > total)
    return fail(GSR_ERR_INVALID_VALUE, "rows_out=%lld outside 0..%lld (the sum of M_r)",
                (long long)rows_out, (long long)total);
  // States of shards that hold a kept row must be valid; the rest are not read.
  int64_t begin = 0;
  for (int r = 0; r < R; ++r) {
    if (begin < rows_out && M_r[r] > 0) {
      for (int t = 0; t < T; ++t)
        if (!S[r * T + t] || !aligned16(S[r * T + t]))
          return fail(GSR_ERR_INVALID_VALUE, "S[%d] (shard %d, state %d) must be non-NULL and 16-byte aligned",
                      r * T + t, r, t);
    }
    begin += M_r[r];
  }
  if (rows_out > 0 && (!Pout || !aligned16(Pout)))
    return fail(GSR_ERR_INVALID_VALUE, "P must be non-NULL and 16-byte aligned");
  if (!ws) return fail(GSR_ERR_WORKSPACE, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(GSR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < gsr::kWsHeader)
    return fail(GSR_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", ws_bytes,
                gsr::kWsHeader);
  if (rows_out == 0) return ok();
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: arguments are valid, nothing launched");

  gsr::PackParams p;
  std::memset(&p, 0, sizeof p);
  int64_t row = 0;
  for (int r = 0; r < R; ++r) {
    p.row_begin[r] = row;
    row += M_r[r];
    for (int t = 0; t < T; ++t) p.src[r * T + t] = static_cast<const uint16_t*>(S[r * T + t]);
  }
  for (int r = R; r <= kMaxShards; ++r) p.row_begin[r] = row;
  p.dst = static_cast<uint16_t*>(Pout);
  p.status = static_cast<uint32_t*>(ws);
  p.timeout_ns = P->timeout_ns;
  p.rows_out = rows_out;
  p.seg_bytes = H * 2;
  p.R = R;
  p.T = T;
  p.pieces_per_seg = static_cast<int>(cdiv(p.seg_bytes, gsr::kPackPieceMax));
  const int64_t pieces = rows_out * T * p.pieces_per_seg;
  const int ctas = static_cast<int>(std::min<int64_t>(P->sm_count, pieces));
  DeviceScope scope(P->device);
  if (scope.err != cudaSuccess) return cuda_fail(scope.err, "selecting the plan's device");
  cudaError_t e = gsr::launch_pack(p, ctas, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return ok();
}

}  // extern "C"

namespace {
// Reads the status word at `word_addr` after synchronising the stream, clears
// it if it is set, and turns it into GSR_OK or GSR_ERR_TIMEOUT.
gsr_status read_and_clear_status(int device, void* word_addr, cudaStream_t st) {
  DeviceScope scope(device);
  if (scope.err != cudaSuccess) return cuda_fail(scope.err, "selecting the plan's device");
  uint32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, word_addr, sizeof word, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (word == 0) return ok();
  e = cudaMemsetAsync(word_addr, 0, sizeof word, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  return fail(GSR_ERR_TIMEOUT, "in-kernel wait ran out (code 0x%08x: role %u, site %u)", word,
              (word >> 8) & 0xFFu, word & 0xFFu);
}
}  // namespace

extern "C" {

gsr_status gemm_shard_check_status(const gemm_shard_plan* P, void* ws, gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  if (!ws) return fail(GSR_ERR_WORKSPACE, "workspace is NULL");
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: no device status to read");
  return read_and_clear_status(P->device, ws, reinterpret_cast<cudaStream_t>(stream));
}

gsr_status gemm_shard_describe(const gemm_shard_plan* P, int mode, int64_t M, int64_t N, int64_t K,
                               int R, const int64_t* sizes, gsr_config* out) {
  gsr_status s = check_plan(P);
  if (s) return s;
  if (!out) return fail(GSR_ERR_INVALID_VALUE, "out is NULL");
  if (mode < 0 || mode > 2) return fail(GSR_ERR_INVALID_VALUE, "mode must be 0, 1 or 2");
  if (R < 1 || R > kMaxShards || !sizes) return fail(GSR_ERR_INVALID_VALUE, "bad R or sizes");
  if (N < 8 || N % 8) return fail(GSR_ERR_INVALID_VALUE, "N must be a positive multiple of 8");
  if (mode == gsr::kModeAG) {
    if (K < 8 || K % 8) return fail(GSR_ERR_INVALID_VALUE, "K must be a positive multiple of 8");
    for (int r = 0; r < R; ++r)
      if (sizes[r] < 0) return fail(GSR_ERR_INVALID_VALUE, "M_r[%d] must be >= 0", r);
  } else {
    if (M < 0) return fail(GSR_ERR_INVALID_VALUE, "M must be >= 0");
    for (int r = 0; r < R; ++r)
      if (sizes[r] < 8 || sizes[r] % 8)
        return fail(GSR_ERR_INVALID_VALUE, "K_r[%d] must be a positive multiple of 8", r);
  }
  const Config c = choose_config(P, mode, M, N, K, R, sizes);
  out->block_n = c.block_n;
  out->cta_group = c.cta_group;
  out->schedule = c.small                               ? 3
                  : c.sched == gsr::kSchedSplitTail ? 4
                  : c.sched == gsr::kSchedStreamK   ? 2
                                                    : 1;
  out->split = c.splits;
  out->tiles = c.tiles;
  out->dp_tiles = (c.sched == gsr::kSchedStreamK || c.sched == gsr::kSchedSplitTail) ? c.dp_tiles : c.tiles;
  out->sk_iters = c.sk_iters;
  out->ctas = c.ctas;
  out->workspace_bytes = c.ws_bytes;
  out->kblocks = c.small ? c.kz : 1;
  out->l2_hints = c.policy_a == gsr::kPolicyEvictLast    ? 2
                  : c.policy_a == gsr::kPolicyEvictFirst ? 3
                                                         : 1;
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// AR without any device allocation.
//
// Some callers cannot allocate device memory at all, not even once: an
// inference engine that claims all free HBM for its KV cache at start-up and
// afterwards hands a kernel nothing but its inputs and outputs, or a caller on
// a latency-critical path where cudaMalloc's implicit device synchronisation
// is not acceptable. gemm_ar_noalloc serves them from a scratch array that is
// part of the library's device image: it exists on every GPU that loads the
// library, from load until process exit, and is never allocated by a call.

namespace {
constexpr size_t kBuiltinScratchBytes = size_t(24) << 20;  // 24 MiB
constexpr int kScratchDevices = 64;
}  // namespace

static __device__ __align__(256) unsigned char gsr_builtin_scratch[kBuiltinScratchBytes];

namespace {
// The context a cached address belongs to, through the driver's entry points
// (the library links no driver library). A cudaDeviceReset, or any other end
// of the device's primary context, unloads the library image; the next context
// loads it again, possibly at another address.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_fns_once;

// The current context's unique id; false if there is none on this thread or
// the driver does not offer the query.
bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_fns_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  CUcontext ctx = nullptr;
  if (!g_ctx_current || !g_ctx_id || g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchSlot {
  void* addr = nullptr;
  unsigned long long ctx_id = 0;
};
std::mutex g_scratch_mutex;
ScratchSlot g_scratch[kScratchDevices];

// Device address of the scratch array on `device` (which must be current),
// looked up once per device and context. Host code cannot use the array's
// name as an address: on the host it names a shadow object, not device memory.
gsr_status builtin_scratch_address(int device, void** out) {
  if (device < 0 || device >= kScratchDevices)
    return fail(GSR_ERR_UNSUPPORTED, "device ordinal %d has no built-in scratch slot", device);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchSlot& slot = g_scratch[device];
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  if (!slot.addr || !have_id || id != slot.ctx_id) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, gsr_builtin_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "looking up the built-in scratch address");
    slot.addr = p;
    // The lookup makes the device's primary context current on this thread.
    slot.ctx_id = current_context_id(&id) ? id : 0;
  }
  *out = slot.addr;
  return ok();
}
}  // namespace

extern "C" gsr_status gemm_ar_noalloc(const gemm_shard_plan* P, int64_t M, int64_t N, int R,
                                      const int64_t* K_r, const void* const* X_r,
                                      const void* const* W_r, void* Y, gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  s = check_ksharded(P, M, N, R, K_r, X_r, W_r);
  if (s) return s;
  // The plan's own configuration when its scratch fits; otherwise the uniform
  // schedule, whose split pieces need at most one 128 KiB slot per SM.
  // A schedule or split the caller forced through a plan option is kept (the
  // call is then rejected if it does not fit), since another schedule would
  // change the summation order.
  gemm_shard_plan fitted = *P;
  if (choose_config(P, gsr::kModeAR, M, N, 0, R, K_r).ws_bytes > kBuiltinScratchBytes &&
      P->opt_split == 0 && P->opt_schedule == 0)
    fitted.opt_schedule = 1;
  const Config c = choose_config(&fitted, gsr::kModeAR, M, N, 0, R, K_r);
  if (c.ws_bytes > kBuiltinScratchBytes)
    return fail(GSR_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch but the built-in scratch of gemm_ar_noalloc "
                "holds %zu; use gemm_ar with a workspace of gemm_shard_workspace_size bytes",
                c.ws_bytes, kBuiltinScratchBytes);
  P = &fitted;
  if (M == 0) return ok();
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: arguments are valid, nothing launched");
  DeviceScope scope(P->device);
  if (scope.err != cudaSuccess) return cuda_fail(scope.err, "selecting the plan's device");
  void* scratch = nullptr;
  s = builtin_scratch_address(P->device, &scratch);
  if (s) return s;
  // The array keeps whatever the previous call left; the status word and the
  // split-K arrival counters must start at zero.
  cudaError_t e = cudaMemsetAsync(scratch, 0, gsr::kWsHeader + counters_bytes(P),
                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "clearing the built-in scratch");
  return run_ksharded(P, gsr::kModeAR, M, N, R, K_r, X_r, W_r, Y, nullptr, scratch,
                      kBuiltinScratchBytes, stream);
}

extern "C" gsr_status gemm_ar_noalloc_check_status(const gemm_shard_plan* P, gsr_stream_t stream) {
  gsr_status s = check_plan(P);
  if (s) return s;
  if (P->device < 0) return fail(GSR_ERR_UNSUPPORTED, "host plan: no device status to read");
  DeviceScope scope(P->device);
  if (scope.err != cudaSuccess) return cuda_fail(scope.err, "selecting the plan's device");
  void* scratch = nullptr;
  s = builtin_scratch_address(P->device, &scratch);
  if (s) return s;
  return read_and_clear_status(P->device, scratch, reinterpret_cast<cudaStream_t>(stream));
}
