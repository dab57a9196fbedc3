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

// The producer helpers (expect_tx, TMA loads, descriptor prefetch) are called
// by a whole converged warp with warp-uniform operands; one elected lane acts.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
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

// Non-blocking test of the same phase condition.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// 2-D tiled TMA load into this CTA's shared memory, completing on `bar`, with
// an L2 cache policy (from createpolicy) attached.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int x, int y, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t make_l2_policy(int kind) {
  uint64_t pol;
  if (kind == kPolicyEvictLast)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  else if (kind == kPolicyEvictFirst)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e prefetch.tensormap [%0];\n\t}" ::"l"(reinterpret_cast<uint64_t>(map))
      : "memory");
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
// Called by a whole converged warp with warp-uniform operands; one elected
// lane issues the MMA (the MMA and commit helpers below all work this way).
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op the elected lane issued so far is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
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

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait for two batches of tcgen05.ld results at once.
__device__ __forceinline__ void tmem_ld_wait2(uint32_t (&v)[32], uint32_t (&u)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
  asm volatile(""
               : "+r"(u[0]), "+r"(u[1]), "+r"(u[2]), "+r"(u[3]), "+r"(u[4]), "+r"(u[5]),
                 "+r"(u[6]), "+r"(u[7]), "+r"(u[8]), "+r"(u[9]), "+r"(u[10]), "+r"(u[11]),
                 "+r"(u[12]), "+r"(u[13]), "+r"(u[14]), "+r"(u[15]), "+r"(u[16]), "+r"(u[17]),
                 "+r"(u[18]), "+r"(u[19]), "+r"(u[20]), "+r"(u[21]), "+r"(u[22]), "+r"(u[23]),
                 "+r"(u[24]), "+r"(u[25]), "+r"(u[26]), "+r"(u[27]), "+r"(u[28]), "+r"(u[29]),
                 "+r"(u[30]), "+r"(u[31])
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

// ------------------------------------------------------------ CTA-pair glue
// A CTA pair is a cluster of two CTAs (ranks 0 and 1); rank 0 issues the
// pair's MMAs (cta_group::2), each CTA holds half of A (rows) and half of B
// (columns of the output) in its own shared memory and TMEM.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared-memory address `addr` of this CTA, as seen in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}

__device__ __forceinline__ void cluster_barrier() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (possibly the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D (256 rows split over the pair's TMEM) (+)= A (pair halves) * B (pair halves)^T.
__device__ __forceinline__ void mma_bf16_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at offset `bar` in every CTA of `mask` when all
// tcgen05 ops the elected lane issued so far are done.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(mask)
      : "memory");
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

// Limits grow along the dependency chain (producer x1, MMA x2, epilogue x3),
// so when something upstream never arrives the wait closest to the cause runs
// out first and its site is the one recorded.
__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, const Ctl& c,
                                               uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  const uint64_t limit = c.timeout_ns * (site >> 8);
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 31u) == 0) {
      if (*c.abort) return false;
      if (global_timer_ns() - t0 > limit) {
        *c.abort = 1;
        atomicCAS(c.status, 0u, kStatusTimeout | site);
        return false;
      }
    }
  }
}

// The common case (the phase already complete) costs one try_wait and no call.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Ctl& c,
                                             uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bounded_slow(bar, parity, c, site);
}

// Wait until the arrival word `flag` reaches `epoch` (wrap-around compare),
// bounded like every other wait. The word is written by another agent (a copy
// stream's memory operation), so it is read with acquire semantics at GPU scope,
// and the async proxy is fenced before TMA reads the data it guards.
__device__ __noinline__ bool wait_flag(const uint32_t* flag, uint32_t epoch, const Ctl& c,
                                       uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t spin = 0;; ++spin) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (static_cast<int32_t>(v - epoch) >= 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if (*c.abort) return false;
    if (global_timer_ns() - t0 > c.timeout_ns) {
      *c.abort = 1;
      atomicCAS(c.status, 0u, kStatusTimeout | site);
      return false;
    }
    __nanosleep(spin < 64 ? 32 : 256);
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
  int piece;      // which piece of the tile's k range (k order)
  int npieces;    // pieces the tile is cut into (1 = whole tile)
  int slot0;      // partial slot of the tile's piece 0 (pieces are consecutive)
  int n0;         // first output column of the tile
  int m0;         // first row of THIS CTA's 128 rows in its A operand: AR/RS
                  // global, AG local to the CTA's shard
  int shard;      // AG: M-shard of this CTA's rows (-1: the idle half of an odd
                  // last pair tile, which reads zeros and stores nothing)
  int kb_begin;   // k-blocks [kb_begin, kb_end) of this piece
  int kb_end;
};

// Position of the tile in the output (raster order) and its shard.
template <int BN, int CG>
__device__ __forceinline__ void place_tile(const Params& p, Unit& t, uint32_t rank) {
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
  // This CTA's 128 rows: half-tile h. AG half-tiles are numbered over all
  // shards, each inside one shard, so the two halves of a pair tile may come
  // from neighbouring shards and no rows are wasted on shard boundaries.
  const int h = mt * CG + static_cast<int>(rank);
  if (p.mode == kModeAG) {
    if (h >= p.ag_halves) {
      t.shard = -1;
      t.m0 = 0;
    } else {
      int r = 0;
      while (r + 1 < p.R && p.shard_mt_begin[r + 1] <= h) ++r;
      t.shard = r;
      t.m0 = (h - p.shard_mt_begin[r]) * BM;
    }
  } else {
    t.shard = 0;
    t.m0 = h * BM;
  }
}

// Per-worker walk over the schedule; every role of a CTA walks it identically.
struct Sched {
  int w;              // this worker (CTA, or CTA pair)
  int G;              // workers
  int next;           // uniform: next unit; stream-K: next whole tile
  long long it;       // stream-K: next k-block of this worker's range
  long long it_end;
};

template <int CG>
__device__ __forceinline__ Sched sched_begin(const Params& p) {
  Sched s;
  s.w = static_cast<int>(blockIdx.x) / CG;
  s.G = static_cast<int>(gridDim.x) / CG;
  s.next = s.w;
  s.it = (static_cast<long long>(s.w) * p.sk_iters) / s.G;
  s.it_end = (static_cast<long long>(s.w + 1) * p.sk_iters) / s.G;
  return s;
}

// The worker whose stream-K range holds k-block `it` (ranges are
// [w*I/G, (w+1)*I/G), every one non-empty because I >= G).
__device__ __forceinline__ int sk_worker_of(long long it, long long I, int G) {
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
    t.kb_begin = static_cast<int>((static_cast<long long>(t.piece) * p.kb_total) / p.splits);
    t.kb_end = static_cast<int>((static_cast<long long>(t.piece + 1) * p.kb_total) / p.splits);
    place_tile<BN, CG>(p, t, rank);
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
    place_tile<BN, CG>(p, t, rank);
    return true;
  }
  // the next piece of this worker's stream-K range
  const long long kt = p.kb_total;
  const int sk_tile = static_cast<int>(s.it / kt);
  const int k_lo = static_cast<int>(s.it - sk_tile * kt);
  const int k_hi = static_cast<int>(min(kt, k_lo + (s.it_end - s.it)));
  s.it += k_hi - k_lo;
  const int first_w = sk_worker_of(sk_tile * kt, p.sk_iters, s.G);
  const int last_w = sk_worker_of((sk_tile + 1) * kt - 1, p.sk_iters, s.G);
  t.tile = p.dp_tiles + sk_tile;
  t.piece = s.w - first_w;
  t.npieces = last_w - first_w + 1;
  // Along the stream-K range each new piece starts a new tile, a new worker's
  // range, or both, so (tile + worker) numbers the pieces without collisions.
  t.slot0 = sk_tile + first_w;
  t.kb_begin = k_lo;
  t.kb_end = k_hi;
  place_tile<BN, CG>(p, t, rank);
  return true;
}

// MMA N of a tile: the full BN, or the ragged tail rounded up to 16 columns.
template <int BN>
__device__ __forceinline__ uint32_t tile_mma_n(const Params& p, const Unit& t) {
  return static_cast<uint32_t>(min(BN, (p.N - t.n0 + 15) & ~15));
}

// ------------------------------------------------------------ shared layout

template <int BN, int STAGES, int CG>
struct Layout {
  static constexpr uint32_t kABytes = BM * BK * 2;            // this CTA's rows of A
  static constexpr uint32_t kBBytes = (BN / CG) * BK * 2;     // this CTA's columns of B
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

template <int BN, int STAGES, int CG>
__device__ void run_producer(const Params& p, uint32_t tiles_base, uint32_t bars, uint32_t rank,
                             const Ctl& ctl) {
  using L = Layout<BN, STAGES, CG>;
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
  const uint64_t pol_a = make_l2_policy(p.policy_a);
  const uint64_t pol_b = make_l2_policy(p.policy_b);
  uint32_t issued = 0;
  uint32_t slot = 0, slot_parity = 1;   // ring slot of the next load; its free-wait parity
  uint32_t arrived = 0;   // AG with arrival flags: shards seen ready (bit r)
  bool ok = true;
  Sched sch = sched_begin<CG>(p);
  Unit t;
  while (ok && sched_next<BN, CG>(p, sch, t, rank)) {
    if (p.ready != nullptr && t.shard >= 0 && !(arrived & (1u << t.shard))) {
      const bool here = wait_flag(p.ready + t.shard, p.epoch, ctl, (kRoleProducer << 8) | 3);
      __syncwarp();
      if (!here) {
        ok = false;
        break;
      }
      arrived |= 1u << t.shard;
    }
    // This CTA's rows of A, and its columns of B: with a CTA pair the MMA's N
    // columns are split in halves between the two CTAs.
    // The idle half of an odd last pair tile reads rows past the end of a
    // non-empty shard: the TMA unit fills them with zeros.
    const int a_shard = t.shard >= 0 ? t.shard : p.ag_pad_shard;
    const int a_row = t.shard >= 0 ? t.m0 : p.shard_rows[p.ag_pad_shard];
    const int b_row = t.n0 + static_cast<int>(rank * (tile_mma_n<BN>(p, t) / CG));
    int r = 0;
    if (p.mode != kModeAG)
      while (p.shard_kb_begin[r + 1] <= t.kb_begin) ++r;
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
      const CUtensorMap* mb;
      int kx;
      if (p.mode == kModeAG) {
        ma = &p.tmap_a[a_shard];
        mb = &p.tmap_b[0];
        kx = kb * BK;
      } else {
        while (p.shard_kb_begin[r + 1] <= kb) ++r;
        ma = &p.tmap_a[r];
        mb = &p.tmap_b[r];
        kx = (kb - p.shard_kb_begin[r]) * BK;
      }
      if constexpr (CG == 1) {
        mbar_arrive_expect_tx(full, L::kStageBytes);
        tma_load_2d_hint(sa, ma, full, kx, a_row, pol_a);
        tma_load_2d_hint(sb, mb, full, kx, b_row, pol_b);
      } else {
        // Both CTAs' bytes are counted on the leader's full barrier, which the
        // leader alone arms (for the pair's bytes).
        if (rank == 0) mbar_arrive_expect_tx(full, CG * L::kStageBytes);
        const uint32_t lead_full = map_shared_to_rank(full, 0);
        tma_load_2d_pair(sa, ma, lead_full, kx, a_row, pol_a);
        tma_load_2d_pair(sb, mb, lead_full, kx, b_row, pol_b);
      }
      ++issued;
      if (++slot == STAGES) {
        slot = 0;
        slot_parity ^= 1u;
      }
    }
  }
  if (!ok && (CG == 1 || rank == 0)) {
    // Let every copy already issued land before the CTA's shared memory goes
    // away (with a pair, the leader's barriers count the peer's copies too).
    const uint32_t first = issued > STAGES ? issued - STAGES : 0;
    for (uint32_t i = first; i < issued; ++i)
      wait_drain(full0 + 8 * (i % STAGES), (i / STAGES) & 1u, 100000000ull);
  }
}

template <int BN, int STAGES, int CG>
__device__ void run_mma(const Params& p, uint32_t tiles_base, uint32_t bars, uint32_t tmem_base,
                        const Ctl& ctl) {
  using L = Layout<BN, STAGES, CG>;
  const uint32_t full0 = bars, tfull0 = bars + 16 * STAGES, tempty0 = tfull0 + 16;
  const uint32_t empty0 = bars + 8 * STAGES, drain = tempty0 + 16;
  const uint32_t rank = 0;   // only the leader issues MMAs; tile k ranges do not depend on rank
  uint32_t stage = 0, phase = 0, local = 0;   // next ring slot and its fill phase
  bool ok = true, issued_any = false;
  Sched sch = sched_begin<CG>(p);
  Unit t;
  for (; ok && sched_next<BN, CG>(p, sch, t, rank); ++local) {
    const uint32_t acc = local & 1u;
    const uint32_t acc_parity = ((local >> 1) & 1u) ^ 1u;
    const bool free_acc = wait_bounded(tempty0 + 8 * acc, acc_parity, ctl, (kRoleMma << 8) | 1);
    __syncwarp();
    if (!free_acc) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + acc * BN;
    const uint32_t idesc = make_idesc(BM * CG, tile_mma_n<BN>(p, t));
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
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        // advance 16 elements (32 bytes) along K inside the swizzled 128-byte rows
        const uint32_t accumulate = (kb > t.kb_begin || k > 0) ? 1u : 0u;
        if constexpr (CG == 1)
          mma_bf16_ss(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, accumulate);
        else
          mma_bf16_ss_pair(d_tmem, a_desc + 2 * k, b_desc + 2 * k, idesc, accumulate);
      }
      issued_any = true;
      if constexpr (CG == 1)
        mma_commit(empty0 + 8 * cur);
      else
        mma_commit_pair(empty0 + 8 * cur, 0x3);     // frees the slot in both CTAs
    }
    if (!ok) break;
    if constexpr (CG == 1)
      mma_commit(tfull0 + 8 * acc);
    else
      mma_commit_pair(tfull0 + 8 * acc, 0x3);       // both CTAs' epilogues may read
  }
  if (!ok && issued_any) {
    // Every MMA issued so far must finish before the TMEM is released.
    if constexpr (CG == 1)
      mma_commit(drain);
    else
      mma_commit_pair(drain, 0x1);
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

    const uint32_t taddr = tmem_base + lane_addr + acc * BN;
    const int n_valid = min(BN, p.N - t.n0);
    const int chunks = (n_valid + 31) >> 5;
    const int m0 = t.m0;   // this CTA's first row

    // Where this thread's output row goes (with replicated outputs: the same
    // offset in every one of the R buffers).
    bool row_ok;
    uint16_t* row_ptr;
    size_t rep_off = 0;
    if (p.mode == kModeAG) {
      const int sh = t.shard >= 0 ? t.shard : 0;
      const int lr = m0 + row_in_tile;
      row_ok = t.shard >= 0 && lr < p.shard_rows[sh];
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
          mbar_arrive_cluster(map_shared_to_rank(tempty0 + 8 * acc, 0));
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
    // the last. The last piece sums all pieces in k order (its own from TMEM)
    // and stores the tile. A CTA pair keeps one slot and one counter per half.
    const int half = t.tile * CG + static_cast<int>(rank);
    const uint32_t others = static_cast<uint32_t>(t.npieces - 1);
    if (et == 0) *last_flag = (ld_relaxed_gpu(&p.counters[half]) == others) ? 1 : 0;
    epilogue_bar_sync();
    bool last = *last_flag != 0;
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
        if (s == t.piece) {
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
    release_accumulator();  // the TMEM accumulator is free for the next tile
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(bars + 8 * i, 1);                 // full: the (leader's) expect_tx + TMA bytes
      mbar_init(bars + 8 * (STAGES + i), 1);      // empty: one MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 16 * STAGES + 8 * i, 1);               // tmem_full: MMA commit
      mbar_init(bars + 16 * STAGES + 16 + 8 * i, 4 * CG);     // tmem_empty: one per epilogue warp
    }
    mbar_init(bars + 16 * STAGES + 32, 1);  // drain
    *abort_flag = 0;
    *last_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    if constexpr (CG == 1) {
      tmem_alloc(smem_u32(tmem_slot), 2 * BN);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(smem_u32(tmem_slot), 2 * BN);
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
    run_producer<BN, STAGES, CG>(p, tiles_base, bars, rank, ctl);   // whole warp, elected issue
    __syncwarp();
  } else if (warp == 1) {
    // The whole warp walks the MMA loop (its values stay warp-uniform); one
    // elected lane issues each MMA and commit.
    if (rank == 0) run_mma<BN, STAGES, CG>(p, tiles_base, bars, tmem_base, ctl);
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
      tmem_dealloc(tmem_base, 2 * BN);
    else
      tmem_dealloc_pair(tmem_base, 2 * BN);
  }
}

// Ring depths: each instance fills 192-224 KB of shared memory.
template <int BN, int CG> struct Stages;
template <> struct Stages<256, 1> { static constexpr int value = 4; };   // 48 KB stages
template <> struct Stages<128, 1> { static constexpr int value = 6; };   // 32 KB
template <> struct Stages<256, 2> { static constexpr int value = 7; };   // 32 KB per CTA
template <> struct Stages<128, 2> { static constexpr int value = 8; };   // 24 KB per CTA

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
  if (CG == 2) {
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
  if (cta_group == 2)
    return block_n == 256 ? KernelLayout<256, 2>::kSmem : KernelLayout<128, 2>::kSmem;
  return block_n == 256 ? KernelLayout<256, 1>::kSmem : KernelLayout<128, 1>::kSmem;
}

cudaError_t prepare_kernels(int device, int* pair_clusters) {
  (void)device;  // the caller has made `device` current
  cudaError_t e = set_smem_limit<256, 1>();
  if (e == cudaSuccess) e = set_smem_limit<128, 1>();
  if (e == cudaSuccess) e = set_smem_limit<256, 2>();
  if (e == cudaSuccess) e = set_smem_limit<128, 2>();
  if (e != cudaSuccess) return e;
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
  if (cta_group == 2)
    return block_n == 256 ? launch_instance<256, 2>(p, ctas, stream)
                          : launch_instance<128, 2>(p, ctas, stream);
  return block_n == 256 ? launch_instance<256, 1>(p, ctas, stream)
                        : launch_instance<128, 1>(p, ctas, stream);
}

}  // namespace gsr
