// gsr_small.cu -- the small-M kernel of the shard-reduction GEMM (AR and RS
// modes, M <= 256 activation rows: decode-like batches) for GB300 (sm_103a).
//
// It computes the same sum as the main kernel, Y = sum_r X_r W_r^T over the
// K-shards (vLLM PR #53053 summary "Extend GEMM-RS to GEMM-AR", key source
// snippets: each rank's partial torch.mm(x, weight.T), reduced across ranks),
// for the shapes where the work is streaming W from HBM: with few activation
// rows, W (N x K) is the only large operand.
//
// One CTA pair (a cluster of two) owns a tile of tile_rows rows of W (output
// columns) over the whole K range (every shard's k-blocks, in shard order),
// against every activation row: tcgen05.mma.cta_group::2 with the activation
// rows as the MMA's M and the tile's W rows as its N, so the pair streams a
// disjoint slice of W and nothing is reduced between CTAs. Each CTA holds
// half of the tile's W rows and h = ceil(M / 2) activation rows (rounded up
// to 8; rank r holds rows r*h .. r*h + h, so both stream the same bytes):
// - h <= 64: the MMA's M is 128, 64 rows per CTA. The accumulator of a CTA
//   holds its 64 rows twice over in TMEM: lanes 0-63 the tile's first
//   tile_rows/2 columns, lanes 64-127 the others (columns 0 .. tile_rows/2).
// - h > 64: the MMA's M is 256, 128 rows per CTA, lane i = row i of the
//   CTA's half, every column of the tile.
// The MMA's rows past h read stale shared memory into TMEM lanes that are
// never stored; a CTA whose rows are all past M loads no activations.
// The MMA is always the same size for a given M: each output element is the
// same chain of fp32 additions over k (k-blocks in shard order, four K = 16
// steps each) whatever the tile height, so every tile height gives the same
// bits, and RS rows equal AR rows.
//
// A ring stage holds kz consecutive k-blocks of each operand, one copy each
// (kz > 1: a 3-D box over a {64, rows, K_r / 64} view of the shard; a
// shard's last stage may run past its k-blocks, which the copy zero-fills and
// the MMAs add as zeros). The stream runs at a roughly fixed number of stages
// per unit time per SM, whatever their size: 48-row W boxes of one k-block
// streamed W at 2.2 TB/s, of two k-blocks at 3.6 TB/s.
//
// Both CTAs' copies of a stage complete on the leader's (rank 0's) barrier;
// the leader issues the MMAs and its commits free the slot in both CTAs. The
// epilogue of each CTA reads its own rows from TMEM and stores each thread's
// columns of its row as 16-byte vectors (no exchange, no transpose).
//
// Roles (192 threads): warp 0 TMA producer, warp 1 MMA issuer (leader only),
// warps 2..5 epilogue, one per quarter of the TMEM lanes. Every wait is
// bounded by %globaltimer like the main kernel's.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gsr_device.cuh"
#include "gsr_params.h"

namespace gsr {
namespace {

// Named barrier 2: warp 1 (which allocates the TMEM) and the epilogue warps.
__device__ __forceinline__ void tmem_handoff_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(32 + 32 * kSmallEpiWarps) : "memory");
}

// Named barrier 3: warp 1 (which creates the mbarriers) and the producer.
__device__ __forceinline__ void barriers_ready_arrive() {
  asm volatile("bar.arrive 3, 64;" ::: "memory");
}
__device__ __forceinline__ void barriers_ready_sync() {
  asm volatile("bar.sync 3, 64;" ::: "memory");
}

// Barrier offsets of the small kernel (bytes from the barrier base).
struct SmallBars {
  uint32_t full0, empty0, tfull0, tempty0, drain;
  __device__ explicit SmallBars(uint32_t bars, uint32_t stages)
      : full0(bars),
        empty0(bars + 8 * stages),
        tfull0(bars + 16 * stages),
        tempty0(bars + 16 * stages + 16),
        drain(bars + 16 * stages + 32) {}
};

// Walks the k-blocks of this pair's tiles, in order: each tile over the whole
// K range. The whole producer warp runs it with warp-uniform values; lane r
// holds shard r's first k-block (`begins`), read with a shuffle, so the loop
// issues no load from the kernel's parameter space (dynamically indexed
// parameter loads measured several hundred ns each and throttled the TMA
// stream when made per k-block).
static_assert(kMaxShards + 1 <= 32, "the shard table must fit in the lanes of a warp");

// `kb` counts stages (kz k-blocks each; one k-block when kz = 1).
struct KCursor {
  int n0, n_step, kb, kb_end, kz, shard, shard_begin, next_begin;
  __device__ void start(int begins, int stages_per_tile, int tile_rows, int kblocks) {
    n0 = static_cast<int>(blockIdx.x) / 2 * tile_rows;
    n_step = static_cast<int>(gridDim.x) / 2 * tile_rows;
    kb = 0;
    kb_end = stages_per_tile;
    kz = kblocks;
    seek(begins, 0);
  }
  __device__ __forceinline__ void seek(int begins, int from) {
    shard = from;
    next_begin = __shfl_sync(0xffffffffu, begins, shard + 1);
    while (next_begin <= kb) next_begin = __shfl_sync(0xffffffffu, begins, ++shard + 1);
    shard_begin = __shfl_sync(0xffffffffu, begins, shard);
  }
  // The stage's first k-block within its shard (the 3-D box's z), and its column (2-D).
  __device__ __forceinline__ int kz_index() const { return (kb - shard_begin) * kz; }
  __device__ __forceinline__ int kx() const { return (kb - shard_begin) * BK; }
  __device__ __forceinline__ void advance(int begins) {
    if (++kb == kb_end) {
      kb = 0;
      n0 += n_step;
      seek(begins, 0);
    } else if (next_begin <= kb) {
      seek(begins, shard);
    }
  }
};

// Number of tiles this pair walks.
__device__ __forceinline__ int small_tiles_of_pair(const Params& p) {
  const int c = static_cast<int>(blockIdx.x) / 2, step = static_cast<int>(gridDim.x) / 2;
  return c < p.n_tiles ? (p.n_tiles - 1 - c) / step + 1 : 0;
}

// The producer's kernel-parameter reads and its walk's starting point. Taken
// at kernel entry, before the CTA's own set-up, so that the first reads of the
// parameters and of the first shard's descriptors (cold after a launch) overlap
// that set-up instead of delaying the first copy.
struct ProducerStart {
  uint64_t pol_x, pol_w;
  uint32_t stage_tx;
  int total, begins, x_row, w_row_off;
  bool load_x;
  KCursor kc;
  // Called by the whole producer warp.
  __device__ void init(const Params& p, const SmallLayout& L, uint32_t rank) {
    pol_x = make_l2_policy(p.policy_a);
    pol_w = make_l2_policy(p.policy_b);
    x_row = static_cast<int>(rank * L.x_rows);
    load_x = x_row < p.M;
    w_row_off = static_cast<int>(rank) * (p.tile_rows / 2);
    // The leader's barrier counts both CTAs' copies: two W halves, the
    // leader's activation rows and, if it has any, the peer's.
    stage_tx = 2 * L.w_stage + L.x_stage * (static_cast<int>(L.x_rows) < p.M ? 2u : 1u);
    // shard_kb_begin[0..kMaxShards] in lanes 0..16 (kMaxShards + 1 <= 32)
    const int lane = static_cast<int>(threadIdx.x) & 31;
    begins = p.shard_kb_begin[lane <= kMaxShards ? lane : kMaxShards];
    total = p.kb_total * small_tiles_of_pair(p);
    kc.start(begins, p.kb_total, p.tile_rows, p.small_kz);
    prefetch_tensormap(&p.tmap_b[kc.shard]);
    if (load_x) prefetch_tensormap(&p.tmap_a[kc.shard]);
  }
};

__device__ void small_producer(const Params& p, const SmallLayout& L, uint32_t base,
                               const SmallBars& b, ProducerStart& st, uint32_t rank,
                               const Ctl& ctl) {
  const uint64_t pol_x = st.pol_x, pol_w = st.pol_w;
  const uint32_t stage_tx = st.stage_tx;
  const int total = st.total, begins = st.begins, x_row = st.x_row, w_row_off = st.w_row_off;
  const bool load_x = st.load_x;
  const uint32_t arm = rank == 0 ? 1u : 0u;
  // This loop alone feeds the tensor pipe: its critical path is kept short
  // (slot and parity advance incrementally; no division or search per k-block).
  KCursor& kc = st.kc;
  uint32_t slot = 0, slot_parity = 1, issued = 0;
  bool ok = true;
  for (int i = 0; i < total; ++i) {
    // Slot `slot` is free once the pair's MMAs of stage i - stages are done.
    const bool free_slot = wait_bounded(b.empty0 + 8 * slot, slot_parity, ctl, (kRoleProducer << 8) | 1);
    __syncwarp();
    if (!free_slot) {
      ok = false;
      break;
    }
    const uint32_t full = b.full0 + 8 * slot;
    const uint32_t lead_full = map_shared_to_rank(full, 0);
    const uint32_t xs = base + slot * L.x_stage, ws = base + L.w_off + slot * L.w_stage;
    // W rows past N and activation rows past M are zero-filled.
    if (L.kz == 1) {
      if (load_x)
        stage_copies_pair(arm, full, stage_tx, lead_full, xs, &p.tmap_a[kc.shard], x_row, ws,
                          &p.tmap_b[kc.shard], kc.n0 + w_row_off, kc.kx(), pol_x, pol_w);
      else
        tma_load_2d_pair(ws, &p.tmap_b[kc.shard], lead_full, kc.kx(), kc.n0 + w_row_off, pol_w);
    } else {
      if (load_x)
        stage_copies_pair_3d(arm, full, stage_tx, lead_full, xs, &p.tmap_a[kc.shard], x_row, ws,
                             &p.tmap_b[kc.shard], kc.n0 + w_row_off, kc.kz_index(), pol_x, pol_w);
      else
        tma_load_3d_pair(ws, &p.tmap_b[kc.shard], lead_full, kc.n0 + w_row_off, kc.kz_index(), pol_w);
    }
    kc.advance(begins);
    if (++issued == 1) {
      // The other shards' descriptors, once the first copies are on their way.
      for (int r = 0; r < p.R; ++r) {
        if (load_x) prefetch_tensormap(&p.tmap_a[r]);
        prefetch_tensormap(&p.tmap_b[r]);
      }
    }
    if (++slot == L.stages) {
      slot = 0;
      slot_parity ^= 1u;
    }
  }
  if (ok) {
    // The leader's commits for the last ring's worth of stages land here
    // too; nothing else waits for them, and they must land before this CTA
    // leaves (its exit barrier does not order them).
    const uint32_t first = issued > L.stages ? issued - L.stages : 0;
    for (uint32_t i = first; i < issued && ok; ++i) {
      ok = wait_bounded(b.empty0 + 8 * (i % L.stages), (i / L.stages) & 1u, ctl, (kRoleProducer << 8) | 2);
      __syncwarp();
    }
  } else {
    // Let the copies already issued land before the shared memory goes away
    // (they complete on the leader's barrier; this CTA cannot see them, so it
    // waits for the pair's MMAs to have freed the slots, or gives up).
    const uint32_t first = issued > L.stages ? issued - L.stages : 0;
    for (uint32_t i = first; i < issued; ++i)
      wait_drain(b.empty0 + 8 * (i % L.stages), (i / L.stages) & 1u, 100000000ull);
  }
}

// The pair's MMAs (rank 0 only).
__device__ void small_mma(const Params& p, const SmallLayout& L, uint32_t base, const SmallBars& b,
                          uint32_t tmem_base, const Ctl& ctl) {
  const uint32_t idesc = make_idesc(L.mma_m, static_cast<uint32_t>(p.tile_rows));
  uint32_t stage = 0, phase = 0, local = 0;
  bool ok = true, issued_any = false;
  for (int tile = static_cast<int>(blockIdx.x) / 2; ok && tile < p.n_tiles;
       tile += static_cast<int>(gridDim.x) / 2, ++local) {
    const uint32_t acc = local & 1u;
    const uint32_t acc_parity = ((local >> 1) & 1u) ^ 1u;
    const bool free_acc = wait_bounded(b.tempty0 + 8 * acc, acc_parity, ctl, (kRoleMma << 8) | 1);
    __syncwarp();
    if (!free_acc) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + acc * L.acc_stride;
    for (int kb = 0; kb < p.kb_total; ++kb) {   // stages of kz k-blocks
      const bool got = wait_bounded(b.full0 + 8 * stage, phase, ctl, (kRoleMma << 8) | 2);
      __syncwarp();
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint32_t xs = base + stage * L.x_stage, ws = base + L.w_off + stage * L.w_stage;
      for (uint32_t j = 0; j < L.kz; ++j)
        mma4_bf16_pair(d_tmem, smem_desc_sw128(xs + j * L.x_bytes),
                       smem_desc_sw128(ws + j * L.w_bytes), idesc, (kb > 0 || j > 0) ? 1u : 0u);
      issued_any = true;
      mma_commit_pair(b.empty0 + 8 * stage, 0x3);   // frees the slot in both CTAs
      if (++stage == L.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    mma_commit_pair(b.tfull0 + 8 * acc, 0x3);       // both CTAs' epilogues may read
  }
  if (!ok && issued_any) {
    mma_commit_pair(b.drain, 0x1);
    wait_drain(b.drain, 0, 100000000ull);
  }
}

// Row m of the output (routed by mode). The parameters it needs are read when
// the epilogue starts: the first read of a parameter's line comes from memory,
// and at the end of the stream it would delay the stores by a round trip.
struct OutRows {
  uint16_t* y;
  int mode, rps, N;
  __device__ explicit OutRows(const Params& p) : y(p.y), mode(p.mode), rps(p.rps), N(p.N) {
    // Make these reads (and those of both lines of y_r) happen now.
    asm volatile("" ::"l"(y), "r"(mode), "r"(rps), "r"(N), "l"(p.y_r[0]),
                 "l"(p.y_r[kMaxShards - 1]));
  }
  __device__ __forceinline__ uint16_t* row(const Params& p, int m, int rep) const {
    if (mode == kModeRS) {
      const int s = m / rps;
      return p.y_r[s] + static_cast<size_t>(m - s * rps) * N;
    }
    if (mode == kModeARRep) return p.y_r[rep] + static_cast<size_t>(m) * N;
    return y + static_cast<size_t>(m) * N;
  }
};

__device__ void small_epilogue(const Params& p, const SmallLayout& L, const SmallBars& b,
                               uint32_t tmem_base, uint32_t rank, const Ctl& ctl) {
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const int quad = (static_cast<int>(threadIdx.x) >> 5) & 3;  // TMEM lanes this warp may read
  const int idx = quad * 32 + lane;                            // this thread's TMEM lane
  const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
  const int half = p.tile_rows / 2;
  // This thread's row among the CTA's activation rows, its output row and its
  // columns within the tile (see the layouts at the top of the file).
  const int a_row = L.mma_m == 256 ? idx : (idx & 63);
  const int row = static_cast<int>(rank * L.x_rows) + a_row;
  const int col0 = L.mma_m == 256 ? 0 : (idx >> 6) * half;
  const int ncols = static_cast<int>(L.acc_cols);
  const OutRows out(p);
  const bool live = a_row < static_cast<int>(L.x_rows) && row < p.M;
  const int reps = p.mode == kModeARRep ? p.R : 1;
  const uint32_t lead_tempty = map_shared_to_rank(b.tempty0, 0);
  const int step = static_cast<int>(gridDim.x) / 2;
  uint32_t local = 0;
  for (int tile = static_cast<int>(blockIdx.x) / 2; tile < p.n_tiles; tile += step, ++local) {
    const uint32_t acc = local & 1u;
    const bool ok = wait_bounded(b.tfull0 + 8 * acc, (local >> 1) & 1u, ctl, (kRoleEpilogue << 8) | 1);
    if (!epilogue_bar_and<32 * kSmallEpiWarps>(ok)) break;
    tc_fence_after_sync();
    const uint32_t taddr = tmem_base + lane_addr + acc * L.acc_stride;
    const int n_base = tile * p.tile_rows + col0;
    for (int c = 0; c < ncols; c += 16) {
      // 16 columns per TMEM load; an 8-column load for a ragged last chunk
      // (never past the accumulator's columns).
      uint32_t v[16];
      const int cnt = ncols - c >= 16 ? 16 : 8;
      if (cnt == 16)
        tmem_ld_16cols_wait(taddr + c, v);
      else
        tmem_ld_8cols_wait(taddr + c, *reinterpret_cast<uint32_t(*)[8]>(&v[0]));
      if (live) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int n = n_base + c + 8 * j;
          if (8 * j < cnt && n < out.N) {
            uint4 w;
            w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
            w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
            w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
            w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
            for (int rep = 0; rep < reps; ++rep)
              *reinterpret_cast<uint4*>(out.row(p, row, rep) + n) = w;
          }
        }
      }
    }
    // The accumulator goes back to the leader's MMA issuer, which waits for it
    // only before a tile two further on (none after the last two tiles: no
    // arrive that nothing waits for, so the exit barrier need not order it).
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0 && tile + 2 * step < p.n_tiles) mbar_arrive_cluster(lead_tempty + 8 * acc);
  }
}

__global__ void __launch_bounds__(kSmallThreads, 1) gsr_small_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const SmallLayout L = small_layout(p.M, p.tile_rows, p.stages, p.small_kz);
  const SmallBars b(base + L.bars_off, L.stages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L.misc_off + 4);
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const uint32_t rank = cluster_rank();
  // Warp 0's (the producer's) set-up first; see ProducerStart.
  ProducerStart start;
  if (warp == 0) start.init(p, L, rank);

  // Thread 32 (warp 1) creates the barriers and publishes them to the peer
  // with its (releasing) arrival on the cluster barrier, and to this CTA's
  // producer through named barrier 3. The other warps arrive without a
  // release: the producer's arrival would otherwise wait for its cold
  // descriptor prefetches (measured 1.6 us). Each role waits for the peer's
  // barriers only before its first access to the peer; the leader's producer,
  // which starts the stream, waits after its loop. The TMEM allocation
  // (collective over the pair) comes after the arrival, off the producers'
  // path: the MMA issuer and the epilogue get its address through named
  // barrier 2.
  if (threadIdx.x == 32) {
    for (uint32_t i = 0; i < L.stages; ++i) {
      mbar_init(b.full0 + 8 * i, 1);    // the leader's expect_tx + both CTAs' bytes
      mbar_init(b.empty0 + 8 * i, 1);   // one MMA commit (the leader's, in both CTAs)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b.tfull0 + 8 * i, 1);                     // MMA commit
      mbar_init(b.tempty0 + 8 * i, 2 * kSmallEpiWarps);   // every epilogue warp of the pair
    }
    mbar_init(b.drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    __syncwarp();
    cluster_arrive();
    barriers_ready_arrive();
  } else if (warp == 0) {
    barriers_ready_sync();
    cluster_arrive_relaxed();
  } else {
    cluster_arrive_relaxed();
  }

  // Programmatic dependent launch, as in the main kernel: nothing above
  // touches global memory.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  Ctl ctl{abort_flag, p.status, p.timeout_ns};
  uint32_t tmem_base = 0;
  if (warp == 0) {
    if (rank != 0) cluster_wait();
    small_producer(p, L, base, b, start, rank, ctl);
    __syncwarp();
    if (rank == 0) cluster_wait();
  } else if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), L.tmem_cols);
    tmem_relinquish_pair();
    tc_fence_before_sync();
    tmem_handoff_sync();
    tc_fence_after_sync();
    tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    cluster_wait();
    if (rank == 0) small_mma(p, L, base, b, tmem_base, ctl);
    __syncwarp();
  } else {
    tmem_handoff_sync();
    tc_fence_after_sync();
    tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
    cluster_wait();
    small_epilogue(p, L, b, tmem_base, rank, ctl);
  }

  // No CTA leaves while its peer may still write or signal it. On the normal
  // path every copy, commit and arrive a CTA receives is one it waits for (the
  // producers drain the last commits; no accumulator hand-back follows the
  // last two tiles), so the barrier needs no release, which would wait for
  // the output stores.
  tc_fence_before_sync();
  cluster_barrier_relaxed();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, L.tmem_cols);
  }
  // After a timed-out wait: the peer may have sent what this CTA stopped
  // waiting for. Having passed the barrier, the peer has issued all of it;
  // the CTA stays resident until it has surely landed.
  if (threadIdx.x == 0 && *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 20000ull) __nanosleep(1000);
  }
}

}  // namespace

cudaError_t prepare_small_kernel() {
  return cudaFuncSetAttribute(gsr_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmallSmemLimit));
}

cudaError_t launch_small(const Params& p, int ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kSmallThreads, 1, 1);
  cfg.dynamicSmemBytes = small_layout(p.M, p.tile_rows, p.stages, p.small_kz).total;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gsr_small_kernel, p);
}

}  // namespace gsr
