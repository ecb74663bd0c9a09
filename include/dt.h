/*
 * dt.h -- collectives among P logical ranks that share one GPU.
 *
 * The operation set is the ThreadGroup collective set of the DTorch developer
 * guide page "集合通信组件" (collective communication component): §2.1 lists
 * the ThreadGroup methods (AllReduce, AllGatherIntoTensor, AllGather with
 * uneven shards, ReduceScatterTensor, AllToAll, Barrier) and §2.3 describes
 * ThreadGroupSameDeviceBackend, the backend used when every rank of the group
 * lives on the same GPU.  On top of that set come the fused gradient-bucket
 * all-reduce with 1/P scaling of "异步融合 AllReduce 流水线优化" (MindSpore
 * hyper-parallel issue #120, AllReduceParamGroup) and the notify/wait barrier
 * of "Barrier：仅信号（Signals Only）" (PyPTO distributed tutorial).
 *
 * Group-wide calls.  One call carries every rank's buffer (rank ==
 * DT_ALL_RANKS, pointer arrays with P entries) and runs as one kernel that
 * reads all P rank buffers directly from HBM.
 *
 * Rank-local calls.  As in DTorch, where every rank is a host thread that
 * calls ThreadGroup with its own tensor, each of P threads may call with
 * rank = its rank (0..P-1), one-entry pointer arrays and its own stream.  The
 * ranks meet on the host the way the MemoryTensorStore of §3.4 does (mutex,
 * condition variable, CUDA events): each rank records a ready event on its
 * stream, the last rank to arrive makes its stream wait on the others' ready
 * events and launches the one group-wide kernel, and every other rank's
 * stream waits on that launch's done event, so results are valid in each
 * rank's own stream order.  All ranks of a round must make the same call
 * (same collective, sizes, dtype, op, flags; AllGather's rows are each
 * rank's own) or every rank gets DT_ERR_INVALID.  A rank whose partners do
 * not all arrive within the group's time limit gets DT_ERR_TIMEOUT and the
 * group is poisoned until dt_group_reset.  Ranks of one group must not mix
 * rank-local and group-wide calls within a round.  dt_bucket_allreduce is
 * group-wide only.
 *
 * Conventions shared by every entry point:
 *   Streams   `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *             default stream).  A call enqueues its work on `stream` and
 *             returns without waiting for the GPU, like a collective in
 *             synchronous mode on the PyTorch page "通信与互联（05）" §四.2:
 *             results are valid in stream order.  Inputs must be produced in
 *             stream order, or the caller makes `stream` wait on an event.
 *   Buffers   Device pointers.  The caller owns them and keeps them alive
 *             until `stream` has passed the call (§五.5 of the same page).
 *             The group owns only its signal window, error word and bucket
 *             plan scratch.  dt_group_create allocates them; the plan scratch
 *             grows only when a bucket plan outgrows it or when every plan
 *             slot is pinned by a CUDA graph (see "CUDA graphs" below).
 *   Alignment Any alignment is accepted.  When every pointer and size is a
 *             multiple of 16 bytes the kernels move 16-byte vectors; otherwise
 *             they fall back to element-wise access with identical results.
 *   Errors    Argument errors are reported before anything is enqueued.  A
 *             device-side wait that runs out of time records DT_ERR_TIMEOUT
 *             in the group's error word; that code is returned by the next
 *             call on the group (and by dt_group_check), and the group then
 *             refuses work until dt_group_reset.  No call throws.
 *   Numerics  fp32 and bf16 reduce in fp32 registers, combining ranks in
 *             ascending rank order (rank 0 first, as the same-device
 *             AllReduce adds ranks 1..P-1 onto rank 0's tensor in order); bf16
 *             is rounded once, to nearest even, at the store; AVG divides the
 *             fp32 sum by P with IEEE division; int32 sums wrap modulo 2^32;
 *             MAX/MIN select an input element (a NaN wins; on equal values
 *             the lower rank's element is kept).
 */
#ifndef DT_H
#define DT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dt_group *dt_group_t;
typedef struct dt_work *dt_work_t;

typedef enum {
    DT_OK = 0,
    DT_ERR_INVALID = 1,      /* bad argument; nothing was enqueued */
    DT_ERR_UNSUPPORTED = 2,  /* legal request the library does not support (AVG on int32, ...) */
    DT_ERR_CUDA = 3,         /* a CUDA runtime call failed */
    DT_ERR_TIMEOUT = 4,      /* a device-side wait ran out of time (see dt_group_check) */
    DT_ERR_OOM = 5,          /* the group could not allocate its own state */
    DT_ERR_POISONED = 6,     /* an earlier timeout left the group unusable until reset */
    DT_ERR_TOO_LARGE = 7,    /* request exceeds the fixed scratch of dt_bucket_allreduce_static */
    DT_NOT_READY = 8         /* dt_work_query: the work has not finished yet (not an error) */
} dt_status;

typedef enum { DT_F32 = 0, DT_BF16 = 1, DT_I32 = 2 } dt_dtype;

/* ReduceOpType of the ThreadGroup interface: kSum, kAvg, kMax, kMin.
 * DT_SUM_STEPWISE is the literal `result += DestGet(rank)` of the same-device
 * AllReduce ("集合通信组件" §2.3): ranks added in ascending order with every
 * add rounded to the element type, so bf16 rounds after each rank instead of
 * once at the end; for fp32 and int32 it equals DT_SUM. */
typedef enum { DT_SUM = 0, DT_AVG = 1, DT_MAX = 2, DT_MIN = 3, DT_SUM_STEPWISE = 4 } dt_redop;

#define DT_MAX_RANKS 16
#define DT_ALL_RANKS (-1)
/* Flag: every out[] entry names the same buffer; the result is written once.
 * The same-device AllReduce hands all ranks one shared result tensor. */
#define DT_SHARED_OUTPUT 0x1u
/* Default bucket cap: DDP's bucket_cap_mb = 25, read as 25 MiB. */
#define DT_DEFAULT_BUCKET_CAP_BYTES ((size_t)25 << 20)

/* Environment switches, read once per process:
 *   DT_TIMEOUT_MS  limit of every device wait and host rendezvous, in ms
 *                  (default 2000; read by dt_group_create)
 *   DT_LOG=1       every kernel launch and bucket plan is printed to stderr
 *   DT_PDL=0       kernels are launched without programmatic dependent launch
 *   DT_DEBUG=1     every launch is followed by a synchronisation of its stream
 *                  (not while the stream is being captured), so a kernel that
 *                  fails is reported by the call that launched it */

/* ------------------------------------------------------------------ groups */

/* Create a group of world_size (1..DT_MAX_RANKS) logical ranks on CUDA device
 * cuda_device.  Allocates the P x P int32 signal window, the error word and
 * two 1 MiB bucket-plan slots on that device; later calls allocate nothing
 * except a bucket all-reduce whose plan needs a larger or an extra slot.
 * The device-side wait limit is read from the environment variable
 * DT_TIMEOUT_MS (default 2000).  Like the TensorStore constructor, which
 * starts all participants from one state, the window starts at zero.
 * Returns DT_ERR_INVALID for a bad size or NULL out, DT_ERR_CUDA / DT_ERR_OOM
 * on a failed CUDA call (nothing is leaked). */
dt_status dt_group_create(int world_size, int cuda_device, dt_group_t *out);

/* Wait for the group's outstanding work, then free everything it owns. */
dt_status dt_group_destroy(dt_group_t g);

/* TensorStore::Reset analogue: zero the signal window and the error word on
 * `stream`, wait for that stream, clear the poisoned state and restart the
 * barrier generation at 0.  Blocks the calling thread. */
dt_status dt_group_reset(dt_group_t g, void *stream);

/* Report the first device-side error recorded so far without synchronising:
 * DT_OK, or the recorded code (the group is poisoned from then on).
 * rank/peer/generation of the failed wait are returned when the pointers are
 * not NULL. */
dt_status dt_group_check(dt_group_t g);
dt_status dt_group_error_detail(dt_group_t g, int *rank, int *peer, int *generation);

/* Number of ranks; number of barrier launches issued on the host since
 * create/reset (a barrier captured in a CUDA graph counts once, however
 * often the graph replays; the device-side generations live in the window). */
int dt_group_size(dt_group_t g);
int64_t dt_group_generation(dt_group_t g);

/* Change the device-side wait limit of later calls (milliseconds, >= 1). */
dt_status dt_group_set_timeout_ms(dt_group_t g, uint32_t timeout_ms);

const char *dt_status_string(dt_status st);

/* Kernels this library has launched in this process (all groups). */
uint64_t dt_launch_count(void);

/* CUDA graphs: group-wide calls may be captured in a stream capture.  Every
 * collective passes its rank pointers in the kernel's parameter block, and the
 * barrier keeps each rank's generation on the device, so replays advance the
 * window as eager calls would.  Make one eager call of each collective before
 * capturing it (the first call sets kernel attributes and caches launch
 * shapes).  A bucket all-reduce can be captured only after an eager call with
 * the same gradients, counts, dtype, op and cap (building a plan may allocate;
 * otherwise the call returns DT_ERR_UNSUPPORTED).  The captured call pins that
 * plan in the group: later bucket calls with other arguments use other plan
 * slots, so the graph keeps replaying against its own plan.  The group must
 * outlive every graph that holds its calls.  Rank-local calls meet on the host
 * and are not meant for capture. */

/* ------------------------------------------------------------- collectives */

/* AllReduce (P -> R): "集合通信组件" §2.1 AllReduce(input, reduceOpType) and
 * the three-phase same-device AllReduce of §2.3.
 *   in[r]   rank r's `count` elements of `dtype` (P entries)
 *   out[q]  rank q's result, `count` elements (P entries); out[q] may equal
 *           in[q] (in place).  With DT_SHARED_OUTPUT all out[] are one buffer
 *           written once; it may not overlap any input.
 * out[q][i] = scale( in[0][i] op in[1][i] op ... op in[P-1][i] ), scale = 1/P
 * for DT_AVG.  DT_AVG on DT_I32 -> DT_ERR_UNSUPPORTED. */
dt_status dt_allreduce(dt_group_t g, int rank, const void *const *in, void *const *out,
                       size_t count, int dtype, int op, unsigned flags, void *stream);

/* ReduceScatter (P -> S(0)): "集合通信组件" §2.1 ReduceScatterTensor.
 *   in[r]   rank r's P * recv_count elements: shard s is elements
 *           [s * recv_count, (s + 1) * recv_count) (dim 0 split evenly)
 *   out[r]  recv_count elements: the reduction over all ranks of shard r.
 * Outputs may not overlap inputs. */
dt_status dt_reduce_scatter(dt_group_t g, int rank, const void *const *in, void *const *out,
                            size_t recv_count, int dtype, int op, void *stream);

/* AllGather (S(0) -> R): "集合通信组件" §2.1 AllGatherIntoTensor (equal
 * shards, rows == NULL: every rank has rows_equal rows) and AllGather with
 * uneven shards (rows[r] rows on rank r).  In a rank-local call rows must be
 * NULL and rows_equal is the calling rank's own row count.  Rows are row_bytes bytes; rank r's
 * rows land at row offset rows[0] + ... + rows[r-1] of every out[q], which
 * holds the sum of all rows.  With DT_SHARED_OUTPUT every out[] is one buffer
 * written once.  Byte copies: any element type. */
dt_status dt_all_gather(dt_group_t g, int rank, const void *const *in, void *const *out,
                        const size_t *rows, size_t rows_equal, size_t row_bytes,
                        unsigned flags, void *stream);

/* AllToAll (S -> S, split and concatenated along dim 0): "集合通信组件"
 * §2.1 AllToAll.  in[i] is P chunks of chunk_bytes; chunk j of rank i goes
 * to rank j, which stacks what it receives in ascending source rank:
 *   out[j][i * chunk_bytes + k] = in[i][j * chunk_bytes + k]. */
dt_status dt_all_to_all(dt_group_t g, int rank, const void *const *in, void *const *out,
                        size_t chunk_bytes, void *stream);

/* ReplicateToShard (R -> S): "集合通信组件" §2.1 ReplicateToShard(input,
 * shardIdx) and the R -> S entry of the §2.5 placement matrix.  Every rank
 * holds the whole tensor (rows rows of row_bytes bytes, rows a multiple of
 * P); rank r keeps row block shard_idx[r] (NULL: block r) of the P equal
 * blocks: out[r] = in[r][shard_idx[r] * rows/P, (shard_idx[r] + 1) * rows/P).
 * Byte copies.  Rank-local: shard_idx points at the calling rank's own index
 * (NULL: its rank).  The sub-split coordinate of the page (nested meshes) is
 * not modelled. */
dt_status dt_replicate_to_shard(dt_group_t g, int rank, const void *const *in, void *const *out,
                                const int *shard_idx, size_t rows, size_t row_bytes, void *stream);

/* AllGatherIntoVec (S -> R, kept apart): "集合通信组件" §2.1
 * AllGatherIntoVec: every rank receives every rank's shard as a tensor of
 * its own.  out has P * P entries; out[q * P + r] (rows[r] rows, or
 * rows_equal when rows is NULL, of row_bytes bytes) receives rank r's shard
 * on rank q.  Rank-local: out has the calling rank's P entries, rows must be
 * NULL and rows_equal is the rank's own row count. */
dt_status dt_all_gather_into_vec(dt_group_t g, int rank, const void *const *in, void *const *out,
                                 const size_t *rows, size_t rows_equal, size_t row_bytes,
                                 void *stream);

/* AllToAll(srcDim, destDim) (S(src_dim) -> S(dest_dim)): "集合通信组件"
 * §2.1 AllToAll(input, srcDim, destDim) on 2-D tensors of R x C elements of
 * elem_bytes bytes (row-major).  Rank i splits its tensor along dest_dim into
 * P equal parts (h x w: R/P x C or R x C/P); part j goes to rank j, which
 * concatenates the parts it receives along src_dim in ascending source rank:
 * out[j] is (P h) x w for src_dim 0 and h x (P w) for src_dim 1.
 * (0, 0) is dt_all_to_all with chunk_bytes = R/P * C * elem_bytes. */
dt_status dt_all_to_all_2d(dt_group_t g, int rank, const void *const *in, void *const *out,
                           size_t R, size_t C, size_t elem_bytes, int src_dim, int dest_dim,
                           void *stream);

/* Fused gradient-bucket all-reduce: "异步融合 AllReduce 流水线优化"
 * (AllReduceParamGroup.issue_async_allreduce / wait_and_apply_grads: SUM
 * all-reduce of the fused gradient buffer, each gradient view then divided by
 * the replicate world size for AVG) with the bucketing of "通信与互联（05）"
 * §六.5 (DDP gathers gradients into bucket_cap_mb = 25 MB buckets).
 *   grads[t * P + p]  rank p's gradient t, counts[t] elements, updated in place
 *   dtype             DT_BF16 or DT_F32;  op  DT_SUM or DT_AVG
 *   bucket_cap_bytes  0 -> DT_DEFAULT_BUCKET_CAP_BYTES
 * Tensors are grouped in order into buckets (dt_bucket_plan); each bucket is
 * one kernel that reads and writes the gradients in place through a chunk
 * table (no flatten copy), and one signal-window barrier (the notify / wait
 * of dt_barrier, one generation each) runs between consecutive buckets: in an
 * extra last block of the earlier bucket's kernel, which waits until that
 * bucket's other blocks have finished.  The next bucket's kernel stores
 * nothing before that whole kernel has completed (its first blocks load
 * their first gradients while it drains: tensors no kernel of the call has
 * written yet).  The plan table is staged through the group's scratch; at
 * most one bucket call per group may be in flight. */
dt_status dt_bucket_allreduce(dt_group_t g, void *const *grads, const size_t *counts,
                              size_t n_tensors, int dtype, int op, size_t bucket_cap_bytes,
                              void *stream);

/* The bucket plan used above, on the host only (no GPU needed): greedy in the
 * given order, a bucket closes when the next tensor would take it past
 * cap_bytes, a tensor larger than the cap gets a bucket of its own.
 * bucket_of[t] receives tensor t's bucket; *n_buckets the bucket count. */
dt_status dt_bucket_plan(const size_t *counts, size_t n_tensors, size_t elem_bytes,
                         size_t cap_bytes, size_t *bucket_of, size_t *n_buckets);

/* Signal-window barrier: "Barrier：仅信号（Signals Only）".  The group keeps
 * an int32 window win[P][P] in HBM (row r of rank q's window is win[q][r]).
 * The g-th barrier (1-based generation, bumped by every call) is one kernel
 * in which each rank is one warp: rank r adds 1 (AtomicAdd) to win[q][r] of
 * every peer q != r, then waits until win[r][s] >= g (Ge) for every s != r.
 * Afterwards win[r][s] == g for s != r and win[r][r] == 0.  Stream order
 * orders the data around the barrier kernel, so its adds and polls are
 * relaxed GPU-scope atomics and loads.  Each wait gives up after the group's
 * time limit and records DT_ERR_TIMEOUT. */
dt_status dt_barrier(dt_group_t g, int rank, void *stream);

/* Allocation-free fused bucket all-reduce.  The pages have no counterpart:
 * this entry point exists for callers that cannot let a library allocate
 * device memory -- applications that own all device memory through their own
 * pool (a library's cudaMalloc escapes their accounting and can fail once the
 * pool has taken the device) and code on a latency-critical path that must
 * not stall other streams (cudaMalloc and cudaFree can synchronise the whole
 * device).  Such callers cannot create a dt_group.
 *   world_size        P (1..DT_MAX_RANKS); no group is needed
 *   grads, counts, n_tensors, dtype, op, bucket_cap_bytes, stream
 *                     as dt_bucket_allreduce; the results are identical
 * The tensor and pointer tables live in one fixed 1 MiB device array inside
 * this library (every GPU that loads the library holds it until the process
 * exits) and are staged from a fixed host array: the call allocates nothing.
 * Tables that do not fit (n_tensors * (P * 8 + 24) bytes plus 4 bytes per
 * thread block of every bucket: one block per 2048 bf16 or 1024 fp32
 * elements of each tensor, at most 16 per resident block slot, so about 40
 * full 25 MiB buckets) or more than 4096 buckets return DT_ERR_TOO_LARGE before anything
 * is enqueued.  Every call shares the array and leaves its contents behind;
 * calls that overlap on the GPU (unordered streams) race on it, calls on one
 * stream do not.  A call whose tables differ from the last ones copied to
 * this device copies them with a pageable cudaMemcpyAsync, which CUDA may
 * finish only after the work already queued on `stream`, so such a call can
 * block the host until then; a call that repeats the previous call's
 * gradients, counts, dtype, cap and ranks on the same device finds its
 * tables there and neither copies nor waits.  A call on a stream that is
 * being captured returns DT_ERR_UNSUPPORTED and enqueues nothing (a captured
 * copy would read the host array at replay time, after later calls have
 * rewritten it).  No signal barrier runs between buckets (there is no group
 * window); stream order orders them.  The first call on each device looks up
 * the array's device address with that device current.  The current CUDA
 * device must be the gradients'. */
dt_status dt_bucket_allreduce_static(int world_size, void *const *grads, const size_t *counts,
                                     size_t n_tensors, int dtype, int op,
                                     size_t bucket_cap_bytes, void *stream);

/* ----------------------------------------------------------- async work */

/* Asynchronous collectives, after the async mode of "通信与互联（05）" §四.3
 * (async_op=True): the collective runs on the backend's own stream, which
 * first waits for the caller's stream (syncStream), and the caller gets a
 * Work whose end event it waits on later; §五.5's rule holds: buffers of an
 * unfinished work are neither read nor written on any stream.
 *   dt_async_begin  makes the group's communication stream wait for the work
 *                   already on `stream` and returns that communication stream
 *                   in *comm_stream: pass it to the dt_* calls of the scope
 *                   (any collective, any number); one scope per group at a
 *                   time, opened and closed by one thread
 *   dt_async_end    closes the scope and returns a work handle whose end
 *                   event covers everything enqueued in the scope
 *   dt_work_wait    makes `stream` wait for the work (no host blocking)
 *   dt_work_query   DT_OK when the work has finished, DT_NOT_READY if not
 *   dt_work_free    returns the handle to its group (after waiting or
 *                   querying; freeing does not cancel the work)
 * Groups on different communication streams (for example the shard and
 * replicate groups of an HSDP mesh) run their works concurrently. */
dt_status dt_async_begin(dt_group_t g, void *stream, void **comm_stream);
dt_status dt_async_end(dt_group_t g, dt_work_t *work);
dt_status dt_work_wait(dt_work_t work, void *stream);
dt_status dt_work_query(dt_work_t work);
dt_status dt_work_free(dt_work_t work);

/* ------------------------------------------------------------- test hooks */

/* Copy the P x P window to host_out (row-major, win[q][r] at q * P + r) after
 * the work already on `stream`; blocks the calling thread. */
dt_status dt_debug_read_window(dt_group_t g, int32_t *host_out, void *stream);

/* The ordering example of the barrier page (built-in reveal): one kernel,
 * one block per rank; rank r copies in[r] to stage[r], passes the barrier,
 * then copies stage[(r + 1) % P] to out[r].  Each buffer holds `bytes`. */
dt_status dt_debug_ring_after_barrier(dt_group_t g, const void *const *in,
                                      void *const *stage, void *const *out, size_t bytes,
                                      void *stream);

/* Failure injection for tests: run one barrier kernel whose waits expect the
 * generation current + extra (extra >= 1), which no rank will reach, with a
 * wait limit of timeout_ms.  The waits give up, DT_ERR_TIMEOUT is recorded
 * in the error word and the kernel returns; the GPU stays usable. */
dt_status dt_debug_barrier_expect(dt_group_t g, int extra, uint32_t timeout_ms, void *stream);

/* ------------------------------------------------------------- tracing */

/* Per-block timeline of the library's kernels, recorded only by a library
 * built with DT_TIMELINE=1 in the environment (elsewhere both calls return
 * DT_ERR_UNSUPPORTED).  The pages trace collectives with profiler timelines
 * ("通信与互联（05）" §六: the communication kernels of each stream on their
 * own row); this records, for every thread block of every kernel launched
 * after dt_timeline_start, when it started, when it passed its wait on the
 * previous kernel (the bucket barrier block: when its barrier completed) and
 * when it ended, in %globaltimer nanoseconds.
 *   dt_timeline_start  (re)allocates room for max_records on the current
 *                      device and empties it; the last one wins
 *   dt_timeline_read   waits for the device, copies up to max_records records
 *                      to host memory and sets *n_records; records past the
 *                      room are dropped and counted in *n_records */
#define DT_TL_REDUCE 1          /* AllReduce / ReduceScatter, vector kernel */
#define DT_TL_REDUCE_SHIFT 2    /* the same, inputs at their own offsets */
#define DT_TL_COPY_BULK 3       /* AllGather / AllToAll, TMA bulk copies */
#define DT_TL_COPY_VEC 4        /* small copies */
#define DT_TL_COPY_SHIFT 5      /* copies at other offsets */
#define DT_TL_COPY_2D 6         /* AllToAll along other dims */
#define DT_TL_BUCKET 7          /* bucket all-reduce, data block */
#define DT_TL_BUCKET_BARRIER 8  /* bucket all-reduce, the barrier block after a bucket */
#define DT_TL_BARRIER 9         /* signal-window barrier kernel */
#define DT_TL_MARK 10           /* dt_timeline_mark: block = the caller's tag */
typedef struct {
    uint64_t grid;       /* the launch's %gridid */
    uint32_t kind;       /* DT_TL_* */
    uint32_t block;      /* blockIdx.x + gridDim.x * blockIdx.y */
    uint32_t sm;         /* %smid */
    uint32_t pad;
    uint64_t t_start, t_waited, t_end;
} dt_timeline_record;
dt_status dt_timeline_start(size_t max_records);
dt_status dt_timeline_read(dt_timeline_record *out, size_t max_records, size_t *n_records);
/* A mark on the timeline at this point of `stream`: a one-thread kernel
 * records DT_TL_MARK with block = tag, so a caller can bracket its own work
 * (a GEMM, a copy) and compare it with the collectives' blocks. */
dt_status dt_timeline_mark(void *stream, uint32_t tag);

/* ------------------------------------------------------- build flavours */

/* Which instrumented flavour this library is (a bit set; 0 = the default
 * build).  Each flavour is chosen by a variable in the environment of the
 * build and compiled into its own objects.
 *   DT_BUILD_NVTX      every entry point opens an NVTX range (DT_NVTX=1)
 *   DT_BUILD_TIMELINE  the kernel timeline above is recorded (DT_TIMELINE=1)
 *   DT_BUILD_BOUNDS    bounds-checked kernels (DT_BOUNDS=1): every global
 *                      load and store of the data kernels is checked against
 *                      the extent of its buffer as the call's arguments give
 *                      it.  An access outside is skipped and DT_ERR_INVALID
 *                      is recorded in the group's error word, with
 *                      dt_group_error_detail giving rank = the kernel
 *                      (DT_BOUNDS_* below), peer = the buffer (reductions:
 *                      input r as r, output q as 16 + q; copies: source
 *                      segment s as s, destination q as 256 + q; bucket
 *                      kernel: the tensor's index in its bucket) and
 *                      generation = the low 31 bits of the byte offset from
 *                      the buffer's start.  dt_bucket_allreduce_static
 *                      has no error word: its out-of-bounds accesses are only
 *                      skipped.  The checks cost time: for testing only.
 *                      DT_BOUNDS_TRIM=<bytes> in the environment of a
 *                      program using this flavour records every destination
 *                      extent that many bytes short (a self-test of the
 *                      checker: the stores it skips lie inside the buffers). */
#define DT_BUILD_NVTX 1u
#define DT_BUILD_TIMELINE 2u
#define DT_BUILD_BOUNDS 4u
#define DT_BOUNDS_REDUCE 1       /* AllReduce / ReduceScatter */
#define DT_BOUNDS_REDUCE_SHIFT 2 /* the same, inputs at their own offsets */
#define DT_BOUNDS_COPY_BULK 3
#define DT_BOUNDS_COPY_VEC 4
#define DT_BOUNDS_COPY_EDGE 5
#define DT_BOUNDS_COPY_SHIFT 6
#define DT_BOUNDS_COPY_2D 7
#define DT_BOUNDS_BUCKET 8
uint32_t dt_build_flags(void);

#ifdef __cplusplus
}
#endif

#endif /* DT_H */
