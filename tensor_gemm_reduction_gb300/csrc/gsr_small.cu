// gsr_small.cu -- the small-M kernel of the shard-reduction GEMM (AR and RS
// modes, M <= 256 activation rows: decode-like batches) for GB300 (sm_103a).
//
// It computes the same sum as the main kernel, Y = sum_r X_r W_r^T over the
// K-shards (vLLM PR #53053 summary "Extend GEMM-RS to GEMM-AR", key source
// snippets: each rank's partial torch.mm(x, weight.T), reduced across ranks),
// for the shapes where the work is streaming W from HBM: with few activation
// rows, W (N x K) is the only large operand.
//
// Operands are swapped so that no tensor-core row is wasted on a short batch:
// a tile is tile_rows rows of W (output columns; the MMA's M) against all m_pad
// activation rows (M rounded up to 16; the MMA's N), Y^T[n, m] accumulated in
// TMEM with TMEM lane = output column and TMEM column = output row. The MMA is
// always 128 rows tall; with tile_rows < 128 (a multiple of 8, chosen so that
// N spreads over every pair of SMs) the rows past the tile read stale shared
// memory into TMEM lanes that are never stored.
//
// Each tile belongs to a cluster of two CTAs. CTA rank k accumulates the
// k-blocks of its half of the K range (over every shard's k-blocks, in shard
// order), so both stream disjoint halves of the tile's W rows. The two fp32
// halves are then added in distributed shared memory instead of through global
// memory: the output rows are cut into 16-row granules, the first half of the
// granules is finished by rank 0 and the rest by rank 1, and each CTA writes
// the granules its peer finishes straight into the peer's shared memory with
// asynchronous stores (st.async) whose bytes complete the peer's mbarrier,
// which the peer armed with the byte count it expects. The owner adds the
// peer's half to its own (one fp32 addition per output, commutative, so the
// result does not depend on which CTA adds), rounds to bf16 (round to nearest
// even) and transposes each 32 x 32 block through shared memory so that the
// global stores are 16-byte vectors, four per 64-byte row segment (a thread
// holds one output column; storing its 2-byte values row by row measured an
// order of magnitude slower). RS routes output row m to
// shard m / rps; the configuration depends only on the shape, so RS rows equal
// AR rows bit for bit.
//
// Roles (320 threads): warp 0 TMA producer, warp 1 MMA issuer, warps 2..9
// epilogue, two per quarter of the TMEM lanes (a warp reads only the lanes of
// its own quarter), taking alternate 32-row chunks of the output rows: the
// epilogue is latency-bound inside each warp, so two warps per quarter halve
// it. Every wait is bounded by %globaltimer like the main kernel's.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gsr_device.cuh"
#include "gsr_params.h"

namespace gsr {
namespace {

// Barrier offsets of the small kernel (bytes from the barrier base).
struct SmallBars {
  uint32_t full0, empty0, tfull0, tempty0, staged, drained, drain;
  __device__ explicit SmallBars(uint32_t bars, uint32_t stages)
      : full0(bars),
        empty0(bars + 8 * stages),
        tfull0(bars + 16 * stages),
        tempty0(bars + 16 * stages + 16),
        staged(bars + 16 * stages + 32),
        drained(bars + 16 * stages + 40),
        drain(bars + 16 * stages + 48) {}
};

// The k-blocks of CTA `rank` of the pair: the first or the second half.
__device__ __forceinline__ void kpair_range(const Params& p, uint32_t rank, int& lo, int& hi) {
  const int half = p.kb_total / 2;
  lo = rank ? half : 0;
  hi = rank ? p.kb_total : half;
}

// Walks the k-blocks this CTA loads, in order: its tiles in turn, each over
// this CTA's half of the K range. The whole producer warp runs it with
// warp-uniform values; lane r holds shard r's first k-block (`begins`), read
// with a shuffle, so the loop issues no load from the kernel's parameter space
// (dynamically indexed parameter loads measured several hundred ns each and
// throttled the TMA stream when made per k-block).
static_assert(kMaxShards + 1 <= 32, "the shard table must fit in the lanes of a warp");

struct KCursor {
  int n0, n_step, kb, shard, shard_begin, next_begin;
  __device__ void start(int begins, int kb_lo, int tile_rows) {
    n0 = static_cast<int>(blockIdx.x) / 2 * tile_rows;
    n_step = static_cast<int>(gridDim.x) / 2 * tile_rows;
    kb = kb_lo;
    seek(begins, 0);
  }
  __device__ __forceinline__ void seek(int begins, int from) {
    shard = from;
    next_begin = __shfl_sync(0xffffffffu, begins, shard + 1);
    while (next_begin <= kb) next_begin = __shfl_sync(0xffffffffu, begins, ++shard + 1);
    shard_begin = __shfl_sync(0xffffffffu, begins, shard);
  }
  __device__ __forceinline__ int kx() const { return (kb - shard_begin) * BK; }
  __device__ __forceinline__ void advance(int begins, int kb_lo, int kb_hi) {
    if (++kb == kb_hi) {
      kb = kb_lo;
      n0 += n_step;
      seek(begins, 0);
    } else if (next_begin <= kb) {
      seek(begins, shard);
    }
  }
};

// Number of tiles this cluster walks.
__device__ __forceinline__ int small_tiles_of_cluster(const Params& p) {
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
  int kb_lo, kb_hi, total, begins;
  KCursor kc;
  // Called by the whole producer warp.
  __device__ void init(const Params& p, const SmallLayout& L, uint32_t rank) {
    pol_x = make_l2_policy(p.policy_a);
    pol_w = make_l2_policy(p.policy_b);
    // A slot's barrier counts both tiles: tile_rows rows of W and m_pad rows of X.
    stage_tx = static_cast<uint32_t>(p.tile_rows) * BK * 2 + L.x_bytes;
    // shard_kb_begin[0..kMaxShards] in lanes 0..16 (kMaxShards + 1 <= 32)
    const int lane = static_cast<int>(threadIdx.x) & 31;
    begins = p.shard_kb_begin[lane <= kMaxShards ? lane : kMaxShards];
    kpair_range(p, rank, kb_lo, kb_hi);
    total = (kb_hi - kb_lo) * small_tiles_of_cluster(p);
    kc.start(begins, kb_lo, p.tile_rows);
    prefetch_tensormap(&p.tmap_b[kc.shard]);
    prefetch_tensormap(&p.tmap_a[kc.shard]);
  }
};

__device__ void small_producer(const Params& p, const SmallLayout& L, uint32_t base,
                               const SmallBars& b, ProducerStart& st, const Ctl& ctl) {
  const uint64_t pol_x = st.pol_x, pol_w = st.pol_w;
  const uint32_t stage_tx = st.stage_tx;
  const int kb_lo = st.kb_lo, kb_hi = st.kb_hi, total = st.total, begins = st.begins;
  KCursor& kc = st.kc;
  // This loop alone feeds the tensor pipe and shares its scheduler with a
  // waiting warp: its critical path is kept short (slot and parity advance
  // incrementally; no division or search per k-block). Each added operation
  // per k-block measured as lost HBM bandwidth.
  uint32_t slot = 0, slot_parity = 1, issued = 0;
  bool ok = true;
  for (int i = 0; i < total; ++i) {
    // Slot `slot` is free once the MMAs of k-block i - stages are done.
    const bool free_slot = wait_bounded(b.empty0 + 8 * slot, slot_parity, ctl, (kRoleProducer << 8) | 1);
    __syncwarp();
    if (!free_slot) {
      ok = false;
      break;
    }
    const uint32_t full = b.full0 + 8 * slot;
    mbar_arrive_expect_tx(full, stage_tx);
    // W rows past N and activation rows past M (up to m_pad) are zero-filled.
    tma_load_2d_hint(base + slot * L.w_bytes, &p.tmap_b[kc.shard], full, kc.kx(), kc.n0, pol_w);
    tma_load_2d_hint(base + L.x_off + slot * L.x_bytes, &p.tmap_a[kc.shard], full, kc.kx(), 0, pol_x);
    kc.advance(begins, kb_lo, kb_hi);
    if (++issued == 1) {
      // The other shards' descriptors, once the first copies are on their way.
      for (int r = 0; r < p.R; ++r) {
        prefetch_tensormap(&p.tmap_a[r]);
        prefetch_tensormap(&p.tmap_b[r]);
      }
    }
    if (++slot == L.stages) {
      slot = 0;
      slot_parity ^= 1u;
    }
  }
  if (!ok) {
    // Let the copies already issued land before the shared memory goes away.
    const uint32_t first = issued > L.stages ? issued - L.stages : 0;
    for (uint32_t i = first; i < issued; ++i)
      wait_drain(b.full0 + 8 * (i % L.stages), (i / L.stages) & 1u, 100000000ull);
  }
}

__device__ void small_mma(const Params& p, const SmallLayout& L, uint32_t base, const SmallBars& b,
                          uint32_t tmem_base, uint32_t rank, const Ctl& ctl) {
  int kb_lo, kb_hi;
  kpair_range(p, rank, kb_lo, kb_hi);
  const uint32_t idesc = make_idesc(kSmallTileN, static_cast<uint32_t>(p.m_pad));
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
    for (int kb = kb_lo; kb < kb_hi; ++kb) {
      const bool got = wait_bounded(b.full0 + 8 * stage, phase, ctl, (kRoleMma << 8) | 2);
      __syncwarp();
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const uint64_t w_desc = smem_desc_sw128(base + stage * L.w_bytes);
      const uint64_t x_desc = smem_desc_sw128(base + L.x_off + stage * L.x_bytes);
#pragma unroll
      for (int k = 0; k < BK / 16; ++k)
        mma_bf16_ss(d_tmem, w_desc + 2 * k, x_desc + 2 * k, idesc,
                    (kb > kb_lo || k > 0) ? 1u : 0u);
      issued_any = true;
      mma_commit(b.empty0 + 8 * stage);
      if (++stage == L.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    mma_commit(b.tfull0 + 8 * acc);
  }
  if (!ok && issued_any) {
    mma_commit(b.drain);
    wait_drain(b.drain, 0, 100000000ull);
  }
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
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

// Up to two consecutive granules (32 TMEM columns) of this thread's lane.
__device__ __forceinline__ void load_granules(uint32_t taddr, int count, uint32_t (&v)[32]) {
  if (count == 2) {
    tmem_ld_32cols(taddr, v);
    tmem_ld_wait(v);
  } else {
    tmem_ld_16cols_wait(taddr, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
  }
}

__device__ void small_epilogue(const Params& p, const SmallLayout& L, uint32_t base,
                               uint8_t* base_ptr, const SmallBars& b, uint32_t tmem_base,
                               uint32_t rank, const Ctl& ctl) {
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const int ew = (static_cast<int>(threadIdx.x) >> 5) - 2;     // epilogue warp 0..7
  const int quad = (static_cast<int>(threadIdx.x) >> 5) & 3;  // TMEM lanes this warp may read
  const int first = 2 * (ew >> 2);   // this warp's first granule pair: chunks alternate
  const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
  const int granules = p.m_pad / kGranule;
  const int g_split = static_cast<int>(small_owned_granules(p.m_pad));  // rank 0 owns [0, g_split)
  const int own_lo = rank ? g_split : 0, own_hi = rank ? granules : g_split;
  const int peer_lo = rank ? 0 : g_split, peer_hi = rank ? g_split : granules;
  const uint32_t peer = rank ^ 1u;
  // Staging: [granule of the owner's range][column group of 4][TMEM lane][4] fp32.
  const uint32_t peer_staging = map_shared_to_rank(base + L.staging_off, peer);
  const float4* my_staging = reinterpret_cast<const float4*>(base_ptr + L.staging_off);
  const uint32_t peer_staged = map_shared_to_rank(b.staged, peer);
  const uint32_t peer_drained = map_shared_to_rank(b.drained, peer);
  const int col_lane = quad * 32 + lane;   // this thread's TMEM lane = column in the tile
  const int reps = p.mode == kModeARRep ? p.R : 1;
  // A quarter of TMEM lanes wholly past the tile (96-row tiles: lanes 96..127)
  // holds no output: its warps only take part in the handshakes.
  const bool live = quad * 32 < p.tile_rows;
  const OutRows out(p);
  const int m_rows = p.M;
  // Bytes the peer sends this CTA per tile (its complete_tx on `staged`): 16
  // fp32 per owned granule for every TMEM lane of a live quarter.
  const uint32_t rx_bytes = static_cast<uint32_t>((own_hi - own_lo) * ((p.tile_rows + 31) / 32) *
                                                  32 * kGranule * 4);
  uint32_t local = 0;
  const int step = static_cast<int>(gridDim.x) / 2;
  for (int tile = static_cast<int>(blockIdx.x) / 2; tile < p.n_tiles; tile += step, ++local) {
    const uint32_t acc = local & 1u;
    // One arrive per tile, with the bytes to expect; the staged wait of the
    // previous tile (same warp) has seen the previous phase complete.
    if (ew == 0) mbar_arrive_expect_tx(b.staged, rx_bytes);
    bool ok = wait_bounded(b.tfull0 + 8 * acc, (local >> 1) & 1u, ctl, (kRoleEpilogue << 8) | 1);
    if (!epilogue_bar_and<kSmallEpiThreads>(ok)) break;
    tc_fence_after_sync();
    const uint32_t taddr = tmem_base + lane_addr + acc * L.acc_stride;
    const int n0 = tile * p.tile_rows;
    const int n_end = min(n0 + p.tile_rows, p.N);   // TMEM lanes past the tile are not output

    // 1. The granules the peer finishes go into the peer's staging area, once
    //    the peer has consumed what this CTA sent for the previous tile. The
    //    stores are asynchronous and counted on the peer's staged barrier.
    if (local > 0) {
      ok = wait_bounded_cluster(b.drained, (local - 1) & 1u, ctl, (kRoleEpilogue << 8) | 2);
      if (!epilogue_bar_and<kSmallEpiThreads>(ok)) break;
    }
    for (int g = peer_lo + first; live && g < peer_hi; g += 4) {
      const int cnt = min(2, peer_hi - g);
      uint32_t v[32];
      load_granules(taddr + g * kGranule, cnt, v);
      const uint32_t dst = peer_staging + ((g - peer_lo) * 4 * kSmallTileN + col_lane) * 16;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4)
        if (c4 < 4 * cnt)
          st_async_v4(dst + c4 * kSmallTileN * 16, v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2],
                      v[4 * c4 + 3], peer_staged);
    }

    // 2. This CTA's granules: its own half plus the peer's, rounded to bf16,
    //    transposed and stored. The transpose goes back into the part of the
    //    staging area this warp has just read (its 32 lanes of the granules'
    //    column groups, 512 bytes each, 2048 bytes apart): 8 rows of 32 bf16
    //    columns per block, so no separate buffer is needed.
    ok = wait_bounded_cluster(b.staged, local & 1u, ctl, (kRoleEpilogue << 8) | 3);
    if (!epilogue_bar_and<kSmallEpiThreads>(ok)) break;
    for (int g = own_lo + first; live && g < own_hi; g += 4) {
      const int cnt = min(2, own_hi - g);
      uint32_t v[32];
      load_granules(taddr + g * kGranule, cnt, v);
      const float4* src = my_staging + (g - own_lo) * 4 * kSmallTileN + col_lane;
      uint8_t* const blocks = base_ptr + L.staging_off +
                              static_cast<size_t>((g - own_lo) * 4 * kSmallTileN + quad * 32) * 16;
      float4 f[8];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4)
        if (c4 < 4 * cnt) f[c4] = src[c4 * kSmallTileN];
      __syncwarp();   // every lane has read its staging before the blocks are overwritten
      // rows 16g .. 16g + 16 cnt of this warp's 32 columns: row r at block r / 8
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        if (c4 >= 4 * cnt) break;
        const float a[4] = {f[c4].x, f[c4].y, f[c4].z, f[c4].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 4 * c4 + j;
          reinterpret_cast<uint16_t*>(blocks + (r >> 3) * (kSmallTileN * 16) + (r & 7) * 64)[lane] =
              bf16_bits(__uint_as_float(v[r]) + a[j]);
        }
      }
      __syncwarp();
      // 16-byte vectors: 8 rows x 4 parts of 8 columns per instruction
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int vi = lane + 32 * t;
        const int row = vi >> 2, part = vi & 3;
        const int m = g * kGranule + row;
        const int n = n0 + quad * 32 + part * 8;
        if (row < kGranule * cnt && m < m_rows && n < n_end) {
          const uint4 val = *reinterpret_cast<const uint4*>(blocks + t * (kSmallTileN * 16) +
                                                            (row & 7) * 64 + part * 16);
          for (int rep = 0; rep < reps; ++rep)
            *reinterpret_cast<uint4*>(out.row(p, m, rep) + n) = val;
        }
      }
      __syncwarp();
    }
    if (tile + step < p.n_tiles) {
      // This CTA's staging may be written again (the peer waits for it only
      // before a next tile; after the last one, no handshake and no wait for
      // the stores above).
      mbar_arrive_cluster(peer_drained);
    }

    // 3. The TMEM accumulator goes back to the MMA issuer.
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(b.tempty0 + 8 * acc);
  }
}

__global__ void __launch_bounds__(kSmallThreads, 1) gsr_small_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const SmallLayout L = small_layout(p.m_pad, p.stages);
  const SmallBars b(base + L.bars_off, L.stages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + L.misc_off + 4);
  const int warp = static_cast<int>(threadIdx.x) >> 5;
  const uint32_t rank = cluster_rank();
  // Warp 0's (the producer's) set-up first; see ProducerStart.
  ProducerStart start;
  if (warp == 0) start.init(p, L, rank);

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < L.stages; ++i) {
      mbar_init(b.full0 + 8 * i, 1);    // expect_tx + the W and X bytes of a k-block
      mbar_init(b.empty0 + 8 * i, 1);   // one MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b.tfull0 + 8 * i, 1);                  // MMA commit
      mbar_init(b.tempty0 + 8 * i, kSmallEpiWarps);    // one per epilogue warp
    }
    mbar_init(b.staged, 1);    // one expect_tx arrive per tile; the peer's bytes complete it
    mbar_init(b.drained, kSmallEpiThreads);
    mbar_init(b.drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), L.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // Only the epilogue touches the peer CTA (its staging area and barriers), so
  // only the epilogue waits here for the peer's barriers to exist; the
  // producer and the MMA issuer start at once and wait after their loops.
  cluster_arrive();

  // Programmatic dependent launch, as in the main kernel: nothing above
  // touches global memory.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  Ctl ctl{abort_flag, p.status, p.timeout_ns};
  if (warp == 0) {
    small_producer(p, L, base, b, start, ctl);
    __syncwarp();
    cluster_wait();
  } else if (warp == 1) {
    small_mma(p, L, base, b, tmem_base, rank, ctl);
    __syncwarp();
    cluster_wait();
  } else {
    cluster_wait();
    small_epilogue(p, L, base, base_ptr, b, tmem_base, rank, ctl);
  }

  // No CTA leaves while its peer may still write or signal it. On the normal
  // path every write and arrive a CTA receives is one it waits for (the
  // peer's staged bytes, and the drained arrive before a next tile; none
  // follows the last tile), so the barrier needs no release, which would
  // wait for the output stores.
  tc_fence_before_sync();
  cluster_barrier_relaxed();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, L.tmem_cols);
  }
  // After a timed-out wait that is no longer so: the peer may have sent what
  // this CTA stopped waiting for. Having passed the barrier, the peer has
  // issued all of it; the CTA stays resident until it has surely landed.
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
  cfg.dynamicSmemBytes = small_layout(p.m_pad, p.stages).total;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gsr_small_kernel, p);
}

}  // namespace gsr
