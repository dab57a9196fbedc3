// gsr_pack.cu -- the packed gather of per-shard states for GB300 (sm_103a).
//
// The pages' sequence-parallel change (vLLM PR #51070 summary, "Kimi K3 SP:
// pack the per-layer all-gathers into one", implementation steps 2-3 and the
// model.py snippet) stops gathering each auxiliary hidden state on its own:
// every rank concatenates its hidden state and its auxiliary states along the
// last dimension, one all-gather stacks the ranks' packed rows, and the result
// is cut to the token count before padding; splitting it by the hidden size
// gives the gathered states back. Here the R ranks are R sets of buffers on one
// GPU, and the concatenation, the gather and the cut are one pass of copies:
//
//   P[g, t*H : (t+1)*H] = S[r][t][g - row_begin[r], :]   for g < rows_out,
//
// with g in shard r's rows [row_begin[r], row_begin[r+1]). Every state is read
// once and P written once; the split-back states are strided views of P.
//
// The work is HBM-bound (no arithmetic), so the copy runs on the TMA engine
// with few SM instructions: each CTA owns a contiguous range of P, cut into
// pieces of at most 16 KB (one state row, or part of one), and one warp streams
// them through a ring of shared-memory buffers: a bulk load global -> shared
// completing on an mbarrier, then, a fixed number of pieces later, a bulk store
// shared -> global in a bulk group. Loads run kLead pieces ahead of stores; a
// buffer is reloaded only after the bulk store that read it has finished
// reading (cp.async.bulk.wait_group.read). Every wait is bounded like the GEMM
// kernels'.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gsr_device.cuh"
#include "gsr_params.h"

namespace gsr {
namespace {

constexpr int kPackBufs = 12;                       // ring of 16 KB buffers: 192 KB
constexpr int kPackLead = 8;                        // loads in flight ahead of stores
constexpr int kPackStoreSlack = kPackBufs - kPackLead - 1;   // store groups that may still read

// The helpers below are issued by one thread (lane 0): a thread's bulk groups
// are its own, so the stores, their commits and the waits on them must all come
// from the same thread.
__device__ __forceinline__ void arm_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile(
      "cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(dst)),
      "r"(src), "r"(bytes)
      : "memory");
}

// Wait until at most kPackStoreSlack bulk-store groups may still read shared memory.
__device__ __forceinline__ void bulk_wait_read_slack() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPackStoreSlack) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Shard table in shared memory: the state pointers and the shards' first
// output rows (read per piece; dynamically indexed kernel-parameter loads are
// slow on this loop's critical path).
struct PackTables {
  const uint8_t* src[kMaxShards * kMaxPackStates];
  int64_t row_begin[kMaxShards + 1];
};

// Walks pieces in the order of P: output row g, state t, piece k of the row's
// state segment. Advances without division.
struct PieceCursor {
  int64_t g;        // output row
  int t, k, r;      // state, piece within the segment, shard of row g
  // The shard of row g; bounded by R because the cursors step one row past
  // the last kept row (after their last piece) and rows_out may equal the sum
  // of M_r.
  __device__ void locate_shard(const PackTables& tb, int R) {
    while (r + 1 < R && g >= tb.row_begin[r + 1]) ++r;
  }
  __device__ const uint8_t* src(const PackTables& tb, const PackParams& p) const {
    return tb.src[r * p.T + t] + (g - tb.row_begin[r]) * p.seg_bytes +
           static_cast<int64_t>(k) * kPackPieceMax;
  }
  __device__ uint32_t bytes(const PackParams& p) const {
    const int64_t left = p.seg_bytes - static_cast<int64_t>(k) * kPackPieceMax;
    return static_cast<uint32_t>(left < kPackPieceMax ? left : kPackPieceMax);
  }
  __device__ void advance(const PackTables& tb, const PackParams& p) {
    if (++k == p.pieces_per_seg) {
      k = 0;
      if (++t == p.T) {
        t = 0;
        ++g;
        locate_shard(tb, p.R);
      }
    }
  }
};

__global__ void __launch_bounds__(32, 1) gsr_pack_kernel(const __grid_constant__ PackParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t bars = base + kPackBufs * kPackPieceMax;
  uint8_t* misc = base_ptr + kPackBufs * kPackPieceMax + kPackBufs * 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc);
  PackTables& tb = *reinterpret_cast<PackTables*>(misc + 16);
  const int lane = static_cast<int>(threadIdx.x);
  if (lane == 0) {
    for (int i = 0; i < kPackBufs; ++i) mbar_init(bars + 8 * i, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  for (int i = lane; i < p.R * p.T; i += 32) tb.src[i] = reinterpret_cast<const uint8_t*>(p.src[i]);
  for (int i = lane; i <= kMaxShards; i += 32) tb.row_begin[i] = p.row_begin[i];
  __syncwarp();
  // Programmatic dependent launch: the states may be written by the previous
  // kernel in the stream.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (lane != 0) return;

  // This CTA's pieces [q0, q1) of the whole sequence (contiguous in P).
  const int64_t pieces = p.rows_out * p.T * p.pieces_per_seg;
  const int64_t q0 = pieces * blockIdx.x / gridDim.x;
  const int64_t q1 = pieces * (blockIdx.x + 1) / gridDim.x;
  const int n = static_cast<int>(q1 - q0);
  PieceCursor lc, sc;   // the load and the store cursors
  {
    const int64_t seg = q0 / p.pieces_per_seg;
    lc.k = static_cast<int>(q0 - seg * p.pieces_per_seg);
    lc.g = seg / p.T;
    lc.t = static_cast<int>(seg - lc.g * p.T);
    lc.r = 0;
    lc.locate_shard(tb, p.R);
    sc = lc;
  }
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.dst) + q0 / p.pieces_per_seg * p.seg_bytes +
                 static_cast<int64_t>(lc.k) * kPackPieceMax;
  const uint64_t pol = make_l2_policy(kPolicyEvictFirst);
  Ctl ctl{abort_flag, p.status, p.timeout_ns};
  uint32_t lb = 0, sb = 0, s_parity = 0;   // load buffer, store buffer, its fill parity
  int loads = 0;
  bool ok = true;
  for (int i = 0; i < n + kPackLead; ++i) {
    if (i < n) {
      // Buffer lb last held piece i - kPackBufs, whose store was issued
      // kPackBufs - kPackLead iterations ago.
      if (i >= kPackBufs) bulk_wait_read_slack();
      const uint32_t bytes = lc.bytes(p);
      arm_tx(bars + 8 * lb, bytes);
      bulk_load(base + lb * kPackPieceMax, lc.src(tb, p), bytes, bars + 8 * lb, pol);
      lc.advance(tb, p);
      ++loads;
      if (++lb == kPackBufs) lb = 0;
    }
    if (i >= kPackLead) {
      if (!wait_bounded(bars + 8 * sb, s_parity, ctl, (kRoleProducer << 8) | 4)) {
        ok = false;
        break;
      }
      const uint32_t bytes = sc.bytes(p);
      bulk_store(dst, base + sb * kPackPieceMax, bytes);
      dst += bytes;
      sc.advance(tb, p);
      if (++sb == kPackBufs) {
        sb = 0;
        s_parity ^= 1u;
      }
    }
  }
  // Stores must finish reading shared memory (and land) before the CTA exits;
  // after a timeout, loads already issued must land too.
  bulk_wait_all();
  if (!ok) {
    const int first = loads > kPackBufs ? loads - kPackBufs : 0;
    for (int i = first; i < loads; ++i)
      wait_drain(bars + 8 * (i % kPackBufs), (i / kPackBufs) & 1u, 100000000ull);
  }
}

constexpr uint32_t kPackSmem = 1024 + kPackBufs * kPackPieceMax + kPackBufs * 8 + 16 +
                               static_cast<uint32_t>(sizeof(PackTables));

}  // namespace

cudaError_t prepare_pack_kernel() {
  return cudaFuncSetAttribute(gsr_pack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kPackSmem));
}

cudaError_t launch_pack(const PackParams& p, int ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.dynamicSmemBytes = kPackSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gsr_pack_kernel, p);
}

}  // namespace gsr
