/*
 * gsr.h -- C ABI of the GB300 (sm_103a) shard-reduction GEMM.
 *
 * A BF16 linear projection whose cross-shard reduction is fused into the GEMM,
 * stated for one GPU: the R "ranks" of a tensor-parallel group are R shard
 * buffers in this GPU's memory, and one kernel launch reads them all in place.
 *
 *   gemm_ar  Y   = sum_r X_r . W_r^T                (all-reduce over K-shards)
 *   gemm_rs  Y_s = rows [s*rps, min(M,(s+1)*rps)) of sum_r X_r . W_r^T
 *                  with rps = ceil(M / R)           (reduce-scatter by rows)
 *   gemm_ag  Y   = concat_r(A_r) . W^T              (all-gather of M-shards)
 *   gemm_ar_replicated  the AR sum written into each of R output buffers
 *
 * Sources of the definitions: vLLM PR #53053 summary ("Extend GEMM-RS to
 * GEMM-AR"), implementation breakdown step 1 (one kernel serves RS and AR;
 * AR accepts any M with no padding or input copy; flags handled inside the
 * kernel) and the test's `_reference` (torch.mm(x, weight.T) per rank, then
 * dist.all_reduce, or dist.reduce_scatter_single over rows padded to
 * ceil(M/R)*R); vLLM PR #54151 "[Kimi-K3] AG-GEMM for Sequence Parallelism",
 * Purpose (GEMM over the gathered activation shards).
 *
 * Conventions shared by every call
 *   - Element type: bf16 in and out; products accumulate in fp32; the output
 *     is rounded once, to nearest even.
 *   - Layout: dense row-major, leading dimension = last dimension. Every GEMM
 *     operand is K-major like an nn.Linear weight: X_r is M x K_r, W_r is
 *     N x K_r, A_r is M_r x K, W is N x K. Outputs are rows x N.
 *   - Alignment: every pointer 16-byte aligned; N and every K_r (AR/RS) or K
 *     (AG) a multiple of 8, so that each row starts on a 16-byte boundary.
 *   - Ownership: the caller owns every device buffer (shards, outputs,
 *     workspace) and the stream. The library owns only the plan, a host
 *     object; it allocates no device memory. Host pointer arrays are read
 *     during the call only.
 *   - Streams: calls are stream-ordered and asynchronous. Nothing synchronises
 *     except gemm_shard_check_status. One workspace must not be used by two
 *     calls that may run at the same time.
 *   - Graphs: gemm_ar, gemm_rs and gemm_ag may be recorded in a CUDA graph
 *     (stream capture). A call's tensor maps and kernel parameters are built
 *     on the host when the call is made, so the graph holds that call's
 *     pointers and shapes, and a replay reads the buffers' current contents.
 *     The workspace's split-K counters are back at zero after every launch,
 *     so replays need no re-initialisation. gemm_shard_check_status
 *     synchronises and cannot be captured.
 *   - Errors: argument errors are detected before any launch and return
 *     GSR_ERR_INVALID_VALUE / GSR_ERR_WORKSPACE without touching the GPU. A
 *     failed launch returns GSR_ERR_CUDA. Every wait inside the kernel is
 *     bounded; a wait that runs out records GSR_ERR_TIMEOUT in the workspace
 *     status word, the kernel returns cleanly, and gemm_shard_check_status
 *     reports it. The library never aborts the process and never traps.
 *     gsr_last_error_string() describes the last failure on this thread.
 *   - Logging: with the environment variable GSR_LOG_CONFIG set (to anything
 *     but "0") when the library is first used, every GEMM call that passes
 *     validation and has rows to compute writes one line to stderr before its
 *     launch: the mode, the shape and the kernel configuration it chose (the
 *     fields of gsr_config). Nothing is logged otherwise.
 */
#ifndef GSR_H
#define GSR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *gsr_stream_t;

typedef struct gemm_shard_plan gemm_shard_plan;

typedef enum {
    GSR_OK = 0,
    GSR_ERR_INVALID_VALUE = 1, /* bad pointer, shape, alignment or option      */
    GSR_ERR_UNSUPPORTED = 2,   /* device is not a GB300-class sm_103 part      */
    GSR_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small   */
    GSR_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed         */
    GSR_ERR_TIMEOUT = 5        /* a bounded in-kernel wait ran out             */
} gsr_status;

/* Largest number of shards (ranks) one call accepts; the pages' gating allows
 * tensor-parallel sizes 2..16 (PR #53053 summary, model.py gating chain). */
#define GSR_MAX_SHARDS 16

/* Plan options (gemm_shard_plan_set_option). 0 restores the default. */
typedef enum {
    GSR_OPT_SPLIT_K = 1,    /* pieces per output tile: 0 = heuristic, 1..16 forced */
    GSR_OPT_BLOCK_N = 2,    /* output tile width: 0 = heuristic, 128, 192 (CTA
                               pairs only; 256 otherwise) or 256              */
    GSR_OPT_TIMEOUT_NS = 3, /* limit of every in-kernel wait, ns (default 2e9)      */
    GSR_OPT_MAX_CTAS = 4,   /* cap on persistent CTAs: 0 = one per SM               */
    GSR_OPT_RASTER_M = 5,   /* m-tiles per raster group (m runs fastest inside a
                               group): 0 = heuristic, 1..64                         */
    GSR_OPT_L2_HINTS = 6,   /* TMA L2 eviction hints: 0 = heuristic (main kernel:
                               2 where both operands together fit in the L2,
                               else none; small-M kernel: 2), 1 = none,
                               2 = A evict-last / B evict-first,
                               3 = A evict-first / B evict-last                     */
    GSR_OPT_CTA_GROUP = 7,  /* CTAs per MMA tile: 0 = heuristic, 1 = one CTA per
                               128-row tile, 2 = a CTA pair per 256-row tile,
                               4 = two CTA pairs per cluster on two 256-row
                               tiles of the same columns, each copy of a B tile
                               loaded once and multicast to both pairs        */
    GSR_OPT_SCHEDULE = 8,   /* work schedule: 0 = heuristic (uniform while there
                               are fewer single-CTA tiles than SMs; else whole
                               tiles for the full waves and, for a partial last
                               wave, a split tail (5) when it is at most half a
                               wave and its pieces keep at least 60 % of the
                               workers busy, whole tiles when at least 70 % of
                               the workers have one, stream-K (3) otherwise),
                               1 = uniform (every tile cut
                               into the same number of pieces), 2 = stream-K
                               over the last one or two waves, 3 = stream-K
                               over the partial last wave, each worker's
                               stream-K range before its whole tiles, 4 = as 3
                               with the whole tiles first, 5 = split tail: each
                               tile of the partial last wave cut into the same
                               k-pieces (2 or 3, one per worker, at most as many
                               pieces as workers), walked before the whole
                               tiles                                             */
    GSR_OPT_SMALL_M = 9,    /* the small-M kernel (AR/RS, M <= 256): 0 = heuristic
                               (used when M <= 256 and no other option above
                               forces a configuration), 1 = never, 2 = whenever
                               M <= 256. It streams W in tiles of rows
                               (GSR_OPT_SMALL_TILE_ROWS, at most 256), one CTA
                               pair per tile over the whole K range, against
                               all M rows at once (the activation rows are the
                               pair MMA's M, the tile's rows its N); it needs
                               no workspace beyond the status word               */
    GSR_OPT_SMALL_TILE_ROWS = 10, /* W rows per tile of the small-M kernel: 0 =
                               heuristic (the fewest rows, in multiples of 16 up
                               to 256, that spread N over every SM pair in the
                               fewest waves), else a multiple of 16 in 16..256   */
    GSR_OPT_RASTER_N = 11,  /* main kernel: n-tiles per raster group, n running
                               fastest inside a group (0 = off: GSR_OPT_RASTER_M
                               applies), 1..64                                   */
    GSR_OPT_SMALL_KBLOCKS = 12 /* small-M kernel: k-blocks of 64 per copy: 0 =
                               heuristic (the largest of 4, 3, 2 that leaves a
                               ring of four stages, where every K_r is a
                               multiple of 64; else 1), else 1..4: at most that
                               many, by the same rule                            */
} gsr_option;

/*
 * Create a plan for device `device` (a CUDA ordinal). The plan records the
 * device's SM count and shared-memory limit and the largest shapes it will
 * accept: max_M rows (AR/RS: M; AG: sum of M_r), max_N output columns, max_K
 * reduction length (AR/RS: sum of K_r; AG: K) and max_R shards. It mirrors the
 * pages' init_gemm_rs_ar(max_M, N, all_reduce) singleton (PR #53053 summary,
 * model.py), minus the mode, which here is chosen per call.
 * Returns GSR_ERR_UNSUPPORTED (and no plan) on anything but a compute
 * capability 10.3 device or when no CUDA driver is present;
 * GSR_ERR_INVALID_VALUE when out is NULL, a maximum is < 1, max_N or max_K is
 * not a multiple of 8, max_R is outside 1..GSR_MAX_SHARDS, or the maxima give
 * 2^27 or more output tiles of 128 x 128 (an output of about 2.2e12 elements,
 * far past any device's memory; the kernels count tiles and their pieces in
 * 32-bit integers).
 */
gsr_status gemm_shard_plan_create(gemm_shard_plan **out, int device, int64_t max_M,
                                  int64_t max_N, int64_t max_K, int max_R);

/*
 * Create a plan bound to no device, for a machine without a GPU: it describes
 * a device with `sm_count` SMs. Calls made with it check their arguments and
 * workspace exactly as on a device, then return GSR_ERR_UNSUPPORTED instead of
 * launching (no device pointer is touched). It takes a GB300's L2 size (126
 * MiB) where the configuration depends on it. gemm_shard_describe and
 * gemm_shard_workspace_size work as for a device plan. Errors as
 * gemm_shard_plan_create, plus GSR_ERR_INVALID_VALUE for sm_count < 1.
 */
gsr_status gemm_shard_plan_create_host(gemm_shard_plan **out, int sm_count, int64_t max_M,
                                       int64_t max_N, int64_t max_K, int max_R);

/* Destroy a plan (NULL is accepted). Outstanding calls are unaffected. */
gsr_status gemm_shard_plan_destroy(gemm_shard_plan *plan);

/* Set an option (see gsr_option). Options change the kernel configuration of
 * later calls only; they never change which elements are computed. */
gsr_status gemm_shard_plan_set_option(gemm_shard_plan *plan, gsr_option option,
                                      int64_t value);

/*
 * Bytes of workspace that every call under this plan (at any shape within its
 * maxima, with its current options) needs. Always > 0: the workspace holds a
 * status word, per-tile split-K arrival counters and fp32 split-K partials.
 * Returns 0 for a NULL plan.
 */
size_t gemm_shard_workspace_size(const gemm_shard_plan *plan);

/*
 * Zero the workspace's status word and counters (stream-ordered memset). Do
 * this once after allocating it, and again after a GSR_ERR_TIMEOUT. Kernels
 * leave the counters at zero when they finish, so no reset is needed between
 * calls. ws must be 256-byte aligned and at least gemm_shard_workspace_size
 * bytes.
 */
gsr_status gemm_shard_workspace_init(const gemm_shard_plan *plan, void *ws,
                                     size_t ws_bytes, gsr_stream_t stream);

/*
 * AR: Y = sum_{r<R} X_r . W_r^T.
 *   M      rows of every X_r and of Y; 0 returns GSR_OK with no launch
 *   N      rows of every W_r and columns of Y (multiple of 8)
 *   R      number of shards, 1..plan max_R
 *   K_r    host array of R shard widths, each >= 8 and a multiple of 8
 *   X_r    host array of R device pointers, X_r[r] is M x K_r[r] bf16 (may be
 *          NULL when M == 0; so may Y)
 *   W_r    host array of R device pointers, W_r[r] is N x K_r[r] bf16
 *   Y      device pointer, M x N bf16; rows [0, M) are written, nothing else
 *   ws     workspace of ws_bytes bytes (gemm_shard_workspace_size)
 * Shards are read in place from their own allocations; no input is copied or
 * padded. The sum over shards is accumulated in fp32 in a fixed order (shards
 * ascending, k ascending within a shard, split-K pieces ascending), so results
 * are deterministic and identical to the rows gemm_rs writes.
 */
gsr_status gemm_ar(const gemm_shard_plan *plan, int64_t M, int64_t N, int R,
                   const int64_t *K_r, const void *const *X_r, const void *const *W_r,
                   void *Y, void *ws, size_t ws_bytes, gsr_stream_t stream);

/*
 * RS: the AR sum, scattered by rows. With rps = ceil(M / R), shard s receives
 * global rows [s*rps, min(M, (s+1)*rps)) as rows [0, count_s) of Y_r[s];
 * Y_r[s] must hold rps rows of N bf16. Rows of Y_r[s] at or past count_s
 * (the reference's zero-padding rows) are not written. Arguments otherwise as
 * gemm_ar. Every written element is bit-identical to the same element of
 * gemm_ar on the same inputs.
 */
gsr_status gemm_rs(const gemm_shard_plan *plan, int64_t M, int64_t N, int R,
                   const int64_t *K_r, const void *const *X_r, const void *const *W_r,
                   void *const *Y_r, void *ws, size_t ws_bytes, gsr_stream_t stream);

/*
 * AR with replicated outputs: the AR sum written whole into each of R output
 * buffers, Y_r[r] = sum_q X_q . W_q^T for every r. This is the one-GPU
 * statement of an all-reduce whose result every rank holds: the GEMM-AR page
 * reduces each row once and multicasts it to all ranks (PR #53053 summary,
 * implementation breakdown step 1, and key source snippets: AR mode takes
 * local_M = partial_uc.shape[0] // num_ranks and stores through
 * multimem_st_16B). Here the reduced tile is rounded once and stored R times
 * from the same epilogue. Y_r[r] must each hold M x N bf16. Every written
 * element is bit-identical to gemm_ar's on the same inputs. Arguments otherwise
 * as gemm_ar.
 */
gsr_status gemm_ar_replicated(const gemm_shard_plan *plan, int64_t M, int64_t N, int R,
                              const int64_t *K_r, const void *const *X_r,
                              const void *const *W_r, void *const *Y_r, void *ws,
                              size_t ws_bytes, gsr_stream_t stream);

/*
 * AG: Y = concat_r(A_r) . W^T.
 *   N      rows of W and columns of Y (multiple of 8)
 *   K      columns of every A_r and of W (multiple of 8)
 *   R      number of shards, 1..plan max_R
 *   M_r    host array of R row counts (>= 0; a shard of 0 rows is skipped)
 *   A_r    host array of R device pointers, A_r[r] is M_r[r] x K bf16 (ignored
 *          when M_r[r] == 0)
 *   W      device pointer, N x K bf16
 *   Y      device pointer, (sum M_r) x N bf16; shard r's rows start at
 *          sum_{q<r} M_q. A sum of 0 returns GSR_OK with no launch (Y may then
 *          be NULL).
 */
gsr_status gemm_ag(const gemm_shard_plan *plan, int64_t N, int64_t K, int R,
                   const int64_t *M_r, const void *const *A_r, const void *W, void *Y,
                   void *ws, size_t ws_bytes, gsr_stream_t stream);

/*
 * AG whose shards may still be arriving when the call starts: the single-kernel
 * AG-GEMM with in-kernel waiting that the AG-GEMM page names as future work
 * ("[Kimi-K3] AG-GEMM for Sequence Parallelism", Component breakdown, closing
 * remark). Before the kernel reads any row of A_r it waits until the device
 * word ready[r] reaches `epoch` (compared with wrap-around: (int32)(ready[r] -
 * epoch) >= 0), so the copies that bring the shards in (a copy stream, in shard
 * order) overlap the GEMM on the shards already present. Pass a new epoch per
 * call instead of resetting the flags.
 *   ready  device array of R uint32 words, 4-byte aligned; written by another
 *          agent, typically gemm_shard_signal on the copy stream
 * The wait is bounded by the plan's timeout (GSR_OPT_TIMEOUT_NS): if a flag
 * never arrives the kernel records GSR_ERR_TIMEOUT in the workspace status
 * word, lets its in-flight copies land, frees its resources and returns;
 * gemm_shard_check_status reports it and the workspace must be re-initialised.
 * Y is then incomplete. Arguments otherwise as gemm_ag.
 */
gsr_status gemm_ag_flagged(const gemm_shard_plan *plan, int64_t N, int64_t K, int R,
                           const int64_t *M_r, const void *const *A_r, const void *W, void *Y,
                           const uint32_t *ready, uint32_t epoch, void *ws, size_t ws_bytes,
                           gsr_stream_t stream);

/*
 * Enqueue on `stream` a write of `value` to the device word `flag`, after all
 * earlier work on the stream and behind a system-wide memory fence. It is a
 * stream memory operation (cuStreamWriteValue32): it runs no kernel, so it can
 * signal a kernel that occupies every SM, such as gemm_ag_flagged.
 * GSR_ERR_INVALID_VALUE for a NULL or misaligned flag; GSR_ERR_UNSUPPORTED on
 * a host plan or a driver without stream memory operations.
 */
gsr_status gemm_shard_signal(const gemm_shard_plan *plan, uint32_t *flag, uint32_t value,
                             gsr_stream_t stream);

/*
 * AR exactly as gemm_ar, for callers that cannot allocate device memory: there
 * is no workspace argument. (The pages have no counterpart; this entry point
 * exists for callers such as an inference engine that claims all free HBM for
 * its KV cache at start-up, or code on a latency-critical path where
 * cudaMalloc's implicit synchronisation is not acceptable.)
 *
 * Its scratch (status word, split-K counters and partials) is one fixed array
 * of 24 MiB in device global memory, part of the library image: every GPU that
 * loads the library holds it until the process exits. Nothing is allocated or
 * freed by the call.
 *   - When the plan's configuration for a shape needs more than 24 MiB of
 *     scratch, the call runs the uniform schedule instead (the same results
 *     within rounding; split pieces then need at most one 128 KiB slot per
 *     SM), unless the plan forces a split (GSR_OPT_SPLIT_K) or a schedule
 *     (GSR_OPT_SCHEDULE): a forced configuration is never replaced, and one
 *     that does not fit is rejected with GSR_ERR_WORKSPACE before anything is
 *     launched; use gemm_ar with a workspace for it. The uniform schedule
 *     always fits when 4 bytes x (ceil(max_M/128) + 2 max_R) x ceil(max_N/128)
 *     counters plus 128 KiB per SM stay under 24 MiB (on a 152-SM GB300:
 *     plans of up to about a million output tiles). Where the configuration
 *     is the plan's own (gemm_shard_describe reports it), the result is
 *     bit-identical to gemm_ar's.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) and keeps it for that device's context; make
 *     that first call before any stream capture begins. The lookup is
 *     repeated only when the device's context has changed (after a
 *     cudaDeviceReset, the library image and its array are loaded again) or
 *     on a thread where no context is current yet.
 *   - Every call on a device shares the one array and starts by clearing its
 *     status word and counters (a stream-ordered memset). Calls that may
 *     overlap on the GPU (different streams, or different host threads without
 *     ordering) race on it and must not be issued.
 *   - A bounded in-kernel wait that runs out leaves its code in the array's
 *     status word: gemm_ar_noalloc_check_status reads it. The next call
 *     clears it, so read it before the next call.
 * Arguments, validation and results are those of gemm_ar.
 */
gsr_status gemm_ar_noalloc(const gemm_shard_plan *plan, int64_t M, int64_t N, int R,
                           const int64_t *K_r, const void *const *X_r,
                           const void *const *W_r, void *Y, gsr_stream_t stream);

/*
 * gemm_shard_check_status for gemm_ar_noalloc: synchronise `stream`, read the
 * built-in scratch's status word on the plan's device, clear it and return
 * GSR_OK or GSR_ERR_TIMEOUT (the code of the first wait that ran out is in
 * gsr_last_error_string). It reports on the last gemm_ar_noalloc call on that
 * device, whichever plan made it. (The pages have no counterpart.)
 * GSR_ERR_INVALID_VALUE for a NULL plan, GSR_ERR_UNSUPPORTED on a host plan,
 * GSR_ERR_CUDA if the copy fails.
 */
gsr_status gemm_ar_noalloc_check_status(const gemm_shard_plan *plan, gsr_stream_t stream);

/*
 * Packed gather of per-shard states (the pages' "Kimi K3 SP: pack the per-layer
 * all-gathers into one", PR #51070 summary, implementation steps 2-3 and its
 * model.py snippet: each rank concatenates its hidden state and auxiliary
 * states along the last dimension, one all-gather stacks the ranks' packed
 * rows, and the result keeps the first full_num_tokens rows; splitting it by
 * the hidden size gives the gathered states back). Here the ranks are R sets of
 * buffers on this GPU and the whole thing is one pass of copies:
 *     P[g, t*H : (t+1)*H] = S[r*T + t][g - row_begin_r, :]      for g < rows_out,
 * where row_begin_r = M_0 + ... + M_{r-1} and g lies in [row_begin_r,
 * row_begin_r + M_r). Bits are copied unchanged (bf16 in, bf16 out).
 *   R         shards, 1..the plan's max_R
 *   M_r       host array of R row counts (>= 0; the sequence-parallel shards)
 *   T         states per shard, 1..16 (the hidden state, then the aux states)
 *   H         columns of every state (the hidden size), a positive multiple of 8
 *   S         host array of R*T device pointers, S[r*T + t] = shard r's state t,
 *             M_r x H row-major bf16, 16-byte aligned; read in place. A shard
 *             with no kept row (all of its rows at or past rows_out) is not
 *             read and its pointers may be NULL.
 *   rows_out  rows kept (full_num_tokens), 0..sum of M_r
 *   P         device output, rows_out x (T*H) row-major bf16, 16-byte aligned,
 *             caller-owned; every element is written, nothing else is. The
 *             split-back state t is the strided view P[:, t*H : (t+1)*H].
 *   ws        the plan's workspace (only its status word is used; a bounded
 *             wait that runs out is reported by gemm_shard_check_status)
 * Errors: GSR_ERR_INVALID_VALUE for the shapes and pointers above,
 * GSR_ERR_WORKSPACE for a NULL, misaligned or too small workspace,
 * GSR_ERR_UNSUPPORTED on a host plan (after validation), GSR_ERR_CUDA when the
 * launch fails. rows_out == 0 returns GSR_OK with no launch. Stream-ordered.
 */
gsr_status gemm_shard_pack_gather(const gemm_shard_plan *plan, int R, const int64_t *M_r, int T,
                                  int64_t H, const void *const *S, int64_t rows_out, void *P,
                                  void *ws, size_t ws_bytes, gsr_stream_t stream);

/*
 * Synchronise `stream`, read the workspace status word, clear it and return
 * GSR_OK or GSR_ERR_TIMEOUT (the code of the first wait that ran out is
 * available through gsr_last_error_string). After a timeout, re-run
 * gemm_shard_workspace_init before the next call.
 */
gsr_status gemm_shard_check_status(const gemm_shard_plan *plan, void *ws,
                                   gsr_stream_t stream);

/* Text of the last error on the calling thread ("" if none). Never NULL. */
const char *gsr_last_error_string(void);

/* Kernel configuration of a call, as gemm_shard_describe reports it. */
typedef struct {
    int block_n;            /* output tile width: 128, 192 or 256 (the small-M
                               kernel: W rows per tile, a multiple of 16 <= 256)  */
    int cta_group;          /* 1: a CTA per 128-row tile; 2: a CTA pair per 256 rows */
    int schedule;           /* 1 = uniform pieces, 2 = stream-K hybrid, 3 = the
                               small-M kernel (one CTA pair per tile of block_n
                               W rows over the whole K range, split = 1),
                               4 = split tail (split = pieces per tail tile)      */
    int split;              /* uniform schedule: pieces per tile                    */
    int64_t tiles;          /* output tiles                                         */
    int64_t dp_tiles;       /* stream-K: tiles run whole                            */
    int64_t sk_iters;       /* stream-K: k-blocks shared out over the workers       */
    int ctas;               /* persistent CTAs launched                             */
    size_t workspace_bytes; /* workspace this call needs                           */
    int kblocks;            /* small-M kernel: k-blocks of 64 per copy (1 to 4);
                               1 for the main kernel                              */
    int l2_hints;           /* the TMA L2 hints taken: 1 = none, 2 = A evict-last /
                               B evict-first, 3 = A evict-first / B evict-last    */
} gsr_config;

/* The kernel configuration the plan chooses for a call, for logging and tests:
 * mode 0 = AR, 1 = RS, 2 = AG. AR/RS use M (>= 0) and sizes = K_r (positive
 * multiples of 8; K is ignored); AG uses K (a positive multiple of 8) and
 * sizes = M_r (>= 0; M is ignored). The plan's maxima are not checked. The
 * configuration depends on the shape, the device and the plan's options, never
 * on the mode, except that AG counts tiles per shard. GSR_ERR_INVALID_VALUE
 * for a NULL plan, out or sizes, a mode outside 0..2, R outside 1..16 or a
 * size that breaks the rules above. */
gsr_status gemm_shard_describe(const gemm_shard_plan *plan, int mode, int64_t M,
                               int64_t N, int64_t K, int R, const int64_t *sizes,
                               gsr_config *out);

#ifdef __cplusplus
}
#endif

#endif /* GSR_H */
