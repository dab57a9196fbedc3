// gsr_kernel.cu -- the shard-reduction GEMM kernel for GB300 (sm_103a).
//
// One persistent, warp-specialised kernel serves all three modes of the fused
// projection (vLLM PR #53053 summary "Extend GEMM-RS to GEMM-AR",
// implementation breakdown step 1 and key source snippets: one kernel, RS and
// AR differing only in where the reduced rows go; PR #54151 "[Kimi-K3] AG-GEMM
// for Sequence Parallelism", Purpose: GEMM over gathered activation shards):
//
//   warp 0      TMA producer: for each work unit, walks its k-blocks; in AR/RS
//               mode a k-block belongs to one K-shard and is fetched through
//               that shard's descriptors (X_r, W_r) straight from the shard's
//               own allocation; in AG mode the unit's M-shard descriptor A_r
//               and the single W descriptor are used. No operand is copied or
//               padded: rows or columns past a shard's extent are zero-filled
//               by the TMA unit.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (kind::f16, bf16 in,
//               fp32 accumulate) into a TMEM accumulator. In AR/RS mode the
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

#include "gsr_params.h"

namespace gsr {
namespace {

// ------------------------------------------------------------------ PTX glue

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// 2-D tiled TMA load into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major bf16, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Each thread of the warp reads 32 consecutive fp32 columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// Wait for this thread's tcgen05.ld results; the registers are tied to the wait so
// that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// Named barrier over the 128 epilogue threads.
__device__ __forceinline__ void epilogue_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpilogueThreads) : "memory");
}

// Named barrier over the epilogue threads that also ANDs a predicate.
__device__ __forceinline__ bool epilogue_bar_and(bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(v)), "n"(kEpilogueThreads)
      : "memory");
  return out != 0;
}

// ------------------------------------------------------------ descriptors

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 64 elements (128 B), 8-row groups 1024 B apart.
// Fields: start address >> 4 in bits 0-13; leading byte offset (unused for
// swizzled K-major, set to 1) in 16-29; stride byte offset 1024 >> 4 in
// 32-45; descriptor version 1 in 46-47; base offset 0 (tiles are 1024-byte
// aligned); swizzle mode 2 (128-byte) in 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16: D fp32 (bits 4-5 = 1), A bf16 (7-9 = 1),
// B bf16 (10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in 17-22,
// M >> 4 in 24-28.
__device__ __forceinline__ uint32_t make_idesc(uint32_t mma_m, uint32_t mma_n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((mma_n >> 3) << 17) | ((mma_m >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<uint32_t*>(&h);
}

// ------------------------------------------------------------ bounded waits

struct Ctl {
  volatile int* abort;    // shared: set by the first role whose wait runs out
  uint32_t* status;       // global: workspace status word
  uint64_t timeout_ns;
};

// Role ids stored in the timeout code.
enum : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3 };

__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Ctl& c,
                                          uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 31u) == 0) {
      if (*c.abort) return false;
      if (global_timer_ns() - t0 > c.timeout_ns) {
        *c.abort = 1;
        atomicCAS(c.status, 0u, kStatusTimeout | site);
        return false;
      }
    }
  }
}

// Used only on the way out after an abort: wait for copies or MMAs already
// issued, ignoring the abort flag, for at most limit_ns.
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ------------------------------------------------------------ scheduling

struct Unit {
  int tile;       // output tile index (also the split-K counter index)
  int split;      // piece of the tile's k range
  int n0;         // first output column
  int m0;         // first row in the A operand: AR/RS global, AG local to shard
  int shard;      // AG: M-shard of the tile
  int kb_begin;   // k-blocks [kb_begin, kb_end) of this piece
  int kb_end;
};

template <int BN>
__device__ __forceinline__ Unit decode_unit(const Params& p, int u) {
  Unit t;
  t.tile = u / p.splits;
  t.split = u - t.tile * p.splits;
  // Raster: groups of group_m m-tiles; inside a group the m index runs fastest,
  // so CTAs working at the same time share W (B) panels and A rows in L2.
  const int span = p.group_m * p.n_tiles;
  const int g = t.tile / span;
  const int first_m = g * p.group_m;
  const int gm = min(p.m_tiles - first_m, p.group_m);
  const int in_g = t.tile - g * span;
  const int mt = first_m + in_g % gm;
  const int nt = in_g / gm;
  t.n0 = nt * BN;
  if (p.mode == kModeAG) {
    int r = 0;
    while (r + 1 < p.R && p.shard_mt_begin[r + 1] <= mt) ++r;
    t.shard = r;
    t.m0 = (mt - p.shard_mt_begin[r]) * BM;
  } else {
    t.shard = 0;
    t.m0 = mt * BM;
  }
  t.kb_begin = static_cast<int>((static_cast<long long>(t.split) * p.kb_total) / p.splits);
  t.kb_end = static_cast<int>((static_cast<long long>(t.split + 1) * p.kb_total) / p.splits);
  return t;
}

// ------------------------------------------------------------ shared layout

template <int BN, int STAGES>
struct Layout {
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBBytes = BN * BK * 2;
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

template <int BN, int STAGES>
__device__ void run_producer(const Params& p, uint32_t tiles_base, uint32_t bars, const Ctl& ctl) {
  using L = Layout<BN, STAGES>;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES;
  if (p.mode == kModeAG) {
    for (int r = 0; r < p.R; ++r)
      if (p.shard_rows[r] > 0) prefetch_tensormap(&p.tmap_a[r]);
    prefetch_tensormap(&p.tmap_b[0]);
  } else {
    for (int r = 0; r < p.R; ++r) {
      prefetch_tensormap(&p.tmap_a[r]);
      prefetch_tensormap(&p.tmap_b[r]);
    }
  }
  uint32_t issued = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
    const Unit t = decode_unit<BN>(p, u);
    int r = 0;
    if (p.mode != kModeAG)
      while (p.shard_kb_begin[r + 1] <= t.kb_begin) ++r;
    for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
      const uint32_t stage = issued % STAGES;
      const uint32_t parity = ((issued / STAGES) & 1u) ^ 1u;
      if (!wait_bounded(empty0 + 8 * stage, parity, ctl, (kRoleProducer << 8) | 1)) {
        ok = false;
        break;
      }
      const uint32_t full = full0 + 8 * stage;
      const uint32_t sa = tiles_base + stage * L::kABytes;
      const uint32_t sb = tiles_base + STAGES * L::kABytes + stage * L::kBBytes;
      mbar_arrive_expect_tx(full, L::kStageBytes);
      if (p.mode == kModeAG) {
        tma_load_2d(sa, &p.tmap_a[t.shard], full, kb * BK, t.m0);
        tma_load_2d(sb, &p.tmap_b[0], full, kb * BK, t.n0);
      } else {
        while (p.shard_kb_begin[r + 1] <= kb) ++r;
        const int kx = (kb - p.shard_kb_begin[r]) * BK;
        tma_load_2d(sa, &p.tmap_a[r], full, kx, t.m0);
        tma_load_2d(sb, &p.tmap_b[r], full, kx, t.n0);
      }
      ++issued;
    }
  }
  if (!ok) {
    // Let every copy already issued land before the CTA's shared memory goes away.
    const uint32_t first = issued > STAGES ? issued - STAGES : 0;
    for (uint32_t i = first; i < issued; ++i)
      wait_drain(full0 + 8 * (i % STAGES), (i / STAGES) & 1u, 100000000ull);
  }
}

template <int BN, int STAGES>
__device__ void run_mma(const Params& p, uint32_t tiles_base, uint32_t bars, uint32_t tmem_base,
                        const Ctl& ctl) {
  using L = Layout<BN, STAGES>;
  const uint32_t full0 = bars, tfull0 = bars + 16 * STAGES, tempty0 = tfull0 + 16;
  const uint32_t empty0 = bars + 8 * STAGES, drain = tempty0 + 16;
  uint32_t consumed = 0, local = 0;
  bool ok = true, issued_any = false;
  for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, ++local) {
    const Unit t = decode_unit<BN>(p, u);
    const uint32_t acc = local & 1u;
    const uint32_t acc_parity = ((local >> 1) & 1u) ^ 1u;
    if (!wait_bounded(tempty0 + 8 * acc, acc_parity, ctl, (kRoleMma << 8) | 1)) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + acc * BN;
    const int n_left = p.N - t.n0;
    const uint32_t mma_n = static_cast<uint32_t>(min(BN, (n_left + 15) & ~15));
    const uint32_t idesc = make_idesc(BM, mma_n);
    for (int kb = t.kb_begin; kb < t.kb_end; ++kb) {
      const uint32_t stage = consumed % STAGES;
      const uint32_t parity = (consumed / STAGES) & 1u;
      if (!wait_bounded(full0 + 8 * stage, parity, ctl, (kRoleMma << 8) | 2)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint64_t a_desc = smem_desc_sw128(tiles_base + stage * L::kABytes);
      const uint64_t b_desc = smem_desc_sw128(tiles_base + STAGES * L::kABytes + stage * L::kBBytes);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        // advance 16 elements (32 bytes) along K inside the swizzled 128-byte rows
        mma_bf16_ss(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc,
                    (kb > t.kb_begin || k > 0) ? 1u : 0u);
      }
      issued_any = true;
      mma_commit(empty0 + 8 * stage);
      ++consumed;
    }
    if (!ok) break;
    mma_commit(tfull0 + 8 * acc);
  }
  if (!ok && issued_any) {
    // Every MMA issued so far must finish before the TMEM is released.
    mma_commit(drain);
    wait_drain(drain, 0, 100000000ull);
  }
}

template <int BN>
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

template <int BN, int STAGES>
__device__ void run_epilogue(const Params& p, uint32_t bars, uint32_t tmem_base,
                             volatile int* last_flag, const Ctl& ctl) {
  const uint32_t tfull0 = bars + 16 * STAGES, tempty0 = tfull0 + 16;
  const int et = static_cast<int>(threadIdx.x) - 64;          // 0..127
  const int quad = (static_cast<int>(threadIdx.x) >> 5) & 3;  // TMEM lanes this warp may read
  const int row_in_tile = quad * 32 + (static_cast<int>(threadIdx.x) & 31);
  const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
  uint32_t local = 0;
  for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++local) {
    const Unit t = decode_unit<BN>(p, u);
    const uint32_t acc = local & 1u;
    const uint32_t acc_parity = (local >> 1) & 1u;
    bool ok = wait_bounded(tfull0 + 8 * acc, acc_parity, ctl, (kRoleEpilogue << 8) | 1);
    if (!epilogue_bar_and(ok)) break;  // all 128 threads leave together
    tc_fence_after_sync();

    const uint32_t taddr = tmem_base + lane_addr + acc * BN;
    const int n_valid = min(BN, p.N - t.n0);
    const int chunks = (n_valid + 31) >> 5;

    // Where this thread's output row goes.
    bool row_ok;
    uint16_t* row_ptr;
    if (p.mode == kModeAG) {
      const int lr = t.m0 + row_in_tile;
      row_ok = lr < p.shard_rows[t.shard];
      row_ptr = p.y + (static_cast<size_t>(p.shard_row_begin[t.shard]) + lr) * p.N + t.n0;
    } else {
      const int gr = t.m0 + row_in_tile;
      row_ok = gr < p.M;
      if (p.mode == kModeRS) {
        const int s = row_ok ? gr / p.rps : 0;
        row_ptr = p.y_r[s] + static_cast<size_t>(gr - s * p.rps) * p.N + t.n0;
      } else {
        row_ptr = p.y + static_cast<size_t>(gr) * p.N + t.n0;
      }
    }

    if (p.splits == 1) {
      for (int c = 0; c < chunks; ++c) {
        uint32_t v[32];
        tmem_ld_32cols(taddr + 32 * c, v);
        tmem_ld_wait(v);
        store_row_chunk<BN>(row_ptr, 32 * c, n_valid, v, row_ok);
      }
      tc_fence_before_sync();
      mbar_arrive(tempty0 + 8 * acc);
      continue;
    }

    // Split-K: publish this piece's fp32 partial tile. Layout inside a slot:
    // [column group of 4][row][4], so a warp's float4 stores are contiguous.
    float* slot = p.partials + static_cast<size_t>(u) * (BM * BN);
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
    tc_fence_before_sync();
    mbar_arrive(tempty0 + 8 * acc);  // the accumulator is free for the next tile
    __threadfence();
    epilogue_bar_sync();
    if (et == 0) {
      const uint32_t before = atomicAdd(&p.counters[t.tile], 1u);
      *last_flag = (before == static_cast<uint32_t>(p.splits - 1)) ? 1 : 0;
    }
    epilogue_bar_sync();
    if (*last_flag) {
      __threadfence();
      const float4* piece0 =
          reinterpret_cast<const float4*>(p.partials + static_cast<size_t>(t.tile) * p.splits * (BM * BN));
      for (int c = 0; c < chunks; ++c) {
        float a[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 f = __ldcg(piece0 + (8 * c + j) * BM + row_in_tile);
          a[4 * j] = f.x; a[4 * j + 1] = f.y; a[4 * j + 2] = f.z; a[4 * j + 3] = f.w;
        }
        for (int s = 1; s < p.splits; ++s) {
          const float4* piece = piece0 + static_cast<size_t>(s) * (BM * BN / 4);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f = __ldcg(piece + (8 * c + j) * BM + row_in_tile);
            a[4 * j] += f.x; a[4 * j + 1] += f.y; a[4 * j + 2] += f.z; a[4 * j + 3] += f.w;
          }
        }
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(a[j]);
        store_row_chunk<BN>(row_ptr, 32 * c, n_valid, v, row_ok);
      }
      if (et == 0) atomicExch(&p.counters[t.tile], 0u);  // ready for the next call
    }
  }
}

// ------------------------------------------------------------ kernel

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1) gsr_gemm_kernel(const __grid_constant__ Params p) {
  using L = Layout<BN, STAGES>;
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bars + 8 * i, 1);                 // full: producer's expect_tx + TMA bytes
      mbar_init(bars + 8 * (STAGES + i), 1);      // empty: one MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 16 * STAGES + 8 * i, 1);                      // tmem_full: MMA commit
      mbar_init(bars + 16 * STAGES + 16 + 8 * i, kEpilogueThreads);  // tmem_empty
    }
    mbar_init(bars + 16 * STAGES + 32, 1);  // drain
    *abort_flag = 0;
    *last_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 2 * BN);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  Ctl ctl{abort_flag, p.status, p.timeout_ns};
  if (warp == 0) {
    if (lane == 0) run_producer<BN, STAGES>(p, tiles_base, bars, ctl);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) run_mma<BN, STAGES>(p, tiles_base, bars, tmem_base, ctl);
    __syncwarp();
  } else {
    run_epilogue<BN, STAGES>(p, bars, tmem_base, last_flag, ctl);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 2 * BN);
  }
}

constexpr int kStages256 = 4;
constexpr int kStages128 = 6;

}  // namespace

size_t kernel_smem_bytes(int block_n) {
  return block_n == 256 ? Layout<256, kStages256>::kSmem : Layout<128, kStages128>::kSmem;
}

cudaError_t prepare_kernels(int device) {
  (void)device;  // the caller has made `device` current
  cudaError_t e = cudaFuncSetAttribute(gsr_gemm_kernel<256, kStages256>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Layout<256, kStages256>::kSmem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gsr_gemm_kernel<128, kStages128>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(Layout<128, kStages128>::kSmem));
}

cudaError_t launch_gemm(const Params& p, int block_n, int ctas, cudaStream_t stream) {
  if (block_n == 256) {
    gsr_gemm_kernel<256, kStages256>
        <<<ctas, kThreads, Layout<256, kStages256>::kSmem, stream>>>(p);
  } else {
    gsr_gemm_kernel<128, kStages128>
        <<<ctas, kThreads, Layout<128, kStages128>::kSmem, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace gsr
