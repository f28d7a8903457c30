/*
 * ar.h -- C ABI of the GB300 gradient all-reduce library (libar_gb300.so).
 *
 * The operation (primer ch. 4, "Collective communication: algorithms, cost and
 * the library that runs them", §4.1, table of collectives): N ranks each hold
 * a buffer of `count` elements; after the all-reduce every rank holds the
 * element-wise sum of all N buffers. Scaling ML Systems ("Collective
 * communication", the ring all-reduce algorithm box) states the same input and
 * output: rank i starts with G_i, every rank ends with G = G_0 + ... + G_{N-1}.
 *
 * Here the N ranks are virtual: their buffers all live in the memory of one
 * GPU, and a "send" is the receiving rank's kernel reading the sender's
 * buffer. There is no inter-GPU traffic and no communication library.
 *
 * Conventions for every call:
 *  - Pointers named `bufs`, `outs`, `workspace`, `tensors`, `bucket` are
 *    DEVICE pointers owned by the caller; arrays of them (`void* const*`) are
 *    HOST arrays of length n_ranks (or n_ranks * n_tensors). Device buffers
 *    must be 16-byte aligned and must not overlap one another, except that
 *    outs[r] may equal bufs[r] (in place).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Calls that take a stream only enqueue work and return without
 *    synchronising; completion is observed by the caller through the stream
 *    (Scaling ML Systems, "Collective communication": initiation of a
 *    collective is non-blocking, returning does not mean completion).
 *  - Errors are returned as ar_status, never printed and never fatal.
 *    Argument checks happen before any work is enqueued; a call that returns
 *    an error has enqueued nothing. AR_ECUDA reports a CUDA error at launch.
 *  - No call allocates device memory, and no call synchronises the device,
 *    except ar_execute_host (which waits for its own copies) and
 *    ar_device_status (which reads a status word). The first executing call
 *    on each device pins one 4-byte host word, the host-visible copy of the
 *    device's status word (see "status" below); nothing else is allocated.
 *  - The library never reads environment variables.
 */
#ifndef AR_GB300_H
#define AR_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define AR_MAX_RANKS 64          /* largest N the kernels accept */
#define AR_MAX_BUCKET_TENSORS 32 /* tensors in one bucket call */

typedef enum {
  AR_OK = 0,
  AR_EINVAL = 1,        /* bad argument: see each call */
  AR_EUNSUPPORTED = 2,  /* valid request the library does not implement */
  AR_ENOMEM = 3,        /* host allocation failed */
  AR_ECUDA = 4,         /* a CUDA runtime call failed */
  AR_ETIMEOUT = 5       /* a device-side bounded wait ran out (sticky) */
} ar_status;

typedef enum { AR_F32 = 0, AR_BF16 = 1 } ar_dtype;

/* Algorithms (primer §4.2 ring, §4.3 Rabenseifner, §4.4 hierarchical and
 * in-network reduction). AR_RING, AR_RABENSEIFNER and AR_HIER run the
 * schedule step by step: one kernel per dependent step, each step reading
 * and writing the rank buffers as the schedule's sends and receives do.
 * AR_FUSED computes the same result in a single pass over HBM: every element
 * of every rank is read once and written once, the traffic of a rank that
 * sends its buffer once and receives the sum once (primer §4.4, "In-network
 * reduction"). */
typedef enum {
  AR_RING = 0,
  AR_RABENSEIFNER = 1,
  AR_HIER = 2,
  AR_FUSED = 3,
  AR_AUTO = 4,
  AR_RECDOUBLING = 5, /* recursive doubling (primer §4.3, "Trees", Fig. 4.5):
                         log2 N steps; in step k ranks i and i xor 2^(k-1)
                         exchange whole buffers and both add. N a power of two.
                         Its sum is the balanced tree of AR_ORDER_TREE. */
  AR_DBTREE = 6,      /* double binary tree (primer §4.3, Fig. 4.6): tree 1 is
                         root 0 over the in-order binary tree of ranks 1..N-1
                         (rank r with lowest set bit b >= 2 has children
                         r - b/2 and r + b/2, the right offset halved until the
                         child is below N); tree 2 is its mirror, r -> N-1-r.
                         Tree t carries half t of the buffer ([0, floor(L/2))
                         and the rest): a reduce up the tree, level by level,
                         inner nodes folding (own + first child) + second
                         child in ascending rank order, then a broadcast down.
                         About 2 log2 N steps. */
  AR_TORUS = 7        /* dimension-ordered all-reduce on a torus (Scaling ML
                         Systems, "Collective communication", torus section):
                         ar_desc.torus_dims = {X, Y, Z} with X*Y*Z = N, rank
                         (x, y, z) = x + X*(y + Y*z); a ring all-reduce along
                         every X line, then every Y line, then every Z line,
                         each over the whole buffer; partial sums stay fp32
                         between dimensions. 2(X-1) + 2(Y-1) + 2(Z-1) steps. */
} ar_algo;
/* AR_AUTO: ar_plan picks the algorithm with ar_select under this GPU's own
 * fabric (virtual ranks in one HBM: every step costs AR_DEVICE_ALPHA_S plus
 * its HBM bytes at AR_DEVICE_BW, both measured on GB300) and records the
 * choice in the plan's descriptor (ar_plan_desc). With one shared memory the
 * single pass always moves the fewest bytes in the fewest steps, so AR_AUTO
 * resolves to AR_FUSED. */
#define AR_DEVICE_ALPHA_S 1.5e-6 /* per dependent kernel launch, graph-replayed */
#define AR_DEVICE_BW 6.0e12      /* bytes/s of algorithmic HBM traffic */
#define AR_DEVICE_CTA_STEP_S 0.28e-6 /* per step of a plan run whole in one
                                        CTA (ar_stats.launches == 1 with more
                                        than one step) with its buffers copied
                                        to shared memory (8 bytes per element
                                        and rank fit in 160 KiB): a block
                                        barrier and the step's shared-memory
                                        accesses, measured on GB300 (device
                                        time: 16-rank ring at 1 KiB 13.2 us
                                        for 30 steps, Rabenseifner 7.2 us for
                                        8; the rest is the launch and the
                                        copies in and out) */
#define AR_DEVICE_CTA_STEP_MEM_S 0.75e-6 /* the same for a one-CTA plan whose
                                            buffers stay in memory: a block
                                            barrier and the step's round trip
                                            to the L2 */

/* Per-element summation order of AR_FUSED. (For AR_REDUCE_SCATTER,
 * AR_ORDER_RING is the order of its ring, which folds chunk c from rank c+1:
 * ((g_{c+1} + g_{c+2}) + ...) + g_c.) Floating-point addition is not
 * associative, so the order is part of the result (Scaling ML Systems,
 * "Collective communication": bitwise identity across algorithms is not
 * guaranteed). Each order reproduces one schedule bit for bit:
 *  AR_ORDER_RING: element of chunk c: ((g_c + g_{c+1}) + ...) + g_{c-1}, the
 *                 order of AR_RING (rank i sends chunk (i - s) mod N at
 *                 reduce-scatter step s, primer §4.2).
 *  AR_ORDER_RANK: ((g_0 + g_1) + ...) + g_{N-1}.
 *  AR_ORDER_TREE: balanced binary tree over ranks in index order, the order
 *                 of AR_RABENSEIFNER (N a power of two).
 *  AR_ORDER_HIER: the order of AR_HIER with group_size G: inside each group
 *                 a fold from local rank k+1 for slice k, then the group
 *                 partials folded from group j for sub-chunk j.          */
typedef enum { AR_ORDER_RING = 0, AR_ORDER_RANK = 1, AR_ORDER_TREE = 2, AR_ORDER_HIER = 3 } ar_order;

/* Which collective (primer §4.1, table of collectives; the all-reduce is a
 * reduce-scatter followed by an all-gather).
 *  AR_ALLREDUCE:      every rank ends with the sum of all N buffers.
 *  AR_REDUCE_SCATTER: rank r ends with chunk r of the sum, in chunk r's range
 *                     [floor(r*count/N), floor((r+1)*count/N)) of its output
 *                     buffer; the other elements of that buffer are left
 *                     unspecified (the step executor keeps partial sums there).
 *  AR_ALLGATHER:      rank r contributes chunk r of its input buffer (its other
 *                     elements are ignored); every rank ends with all N chunks.
 *                     Values are copied; `scale` is ignored.
 * Buffers keep the all-reduce's shape: count elements per rank. The
 * reduce-scatter and all-gather run as AR_RING (N-1 steps, rank i sending
 * chunk (i-1-s) resp. (i-s) mod N at step s, so that rank i owns chunk i) or
 * AR_FUSED (orders RING, RANK or TREE for the reduce-scatter); the other
 * algorithms return AR_EUNSUPPORTED. */
typedef enum { AR_ALLREDUCE = 0, AR_REDUCE_SCATTER = 1, AR_ALLGATHER = 2 } ar_collective;

/* Which kernel runs the single pass (AR_FUSED all-reduce and
 * ar_bucket_allreduce). Both compute the same result, bit for bit; they differ
 * in how bytes move between HBM and the SM.
 *  AR_KERNEL_AUTO:  the library's choice, the faster one measured: the
 *                   register pipeline for the all-reduce and reduce-scatter
 *                   (at every SM budget measured); for the all-gather, bulk
 *                   copies when a rank's buffer holds at least 96 MiB
 *                   (16 x 192 MiB fp32: 0.93 of HBM against 0.90), the
 *                   register pipeline below (64 x 4 MiB: 0.79 against 0.56).
 *  AR_KERNEL_LOADS: persistent register pipeline, 2 CTAs per SM; each thread
 *                   keeps a batch of 16-byte loads in flight.
 *  AR_KERNEL_BULK:  bulk copies (TMA) through shared memory.
 *                   All-reduce: one CTA per SM; a producer warp stages every
 *                   rank's slice of a tile in shared memory through a ring of
 *                   mbarrier-guarded stages; consumer warps fold from shared
 *                   memory and the result leaves through bulk stores; N <= 24
 *                   (the stages must fit in shared memory).
 *                   All-gather: each tile of a chunk is bulk-loaded once from
 *                   its owner and bulk-stored to the N ranks; any N.
 *                   The reduce-scatter has no bulk variant. Unsupported
 *                   requests make ar_plan return AR_EUNSUPPORTED. The waits are
 *                   bounded: a wait that runs out sets the device status word
 *                   (ar_device_status) instead of hanging.
 * The step executors (AR_RING, AR_RABENSEIFNER, AR_HIER) ignore it. */
typedef enum { AR_KERNEL_AUTO = 0, AR_KERNEL_LOADS = 1, AR_KERNEL_BULK = 2 } ar_kernel;

typedef struct {
  int n_ranks;     /* N, 1..AR_MAX_RANKS */
  size_t count;    /* elements per rank buffer, >= 0 */
  ar_dtype dtype;  /* element type of the rank buffers */
  ar_algo algo;
  int group_size;  /* AR_HIER, AR_ORDER_HIER: G >= 1 with N % G == 0; else ignored */
  ar_order order;  /* AR_FUSED only */
  float scale;     /* multiplies the complete fp32 sum once (1.0f = plain sum) */
  ar_collective collective; /* AR_ALLREDUCE (0) unless set */
  int sm_budget;   /* at most this many SMs' worth of CTAs per kernel (0 = all SMs).
                      A collective that overlaps computation takes only part of
                      the GPU, as a NCCL channel takes one SM (primer §4.5).
                      A budget of B launches the CTAs B SMs hold (2 B for the
                      single pass), which the scheduler spreads one per SM; the
                      single pass then loads the next tile while it stores
                      this one (all orders but the hierarchical). Results do
                      not depend on it. */
  ar_kernel kernel; /* AR_KERNEL_AUTO (0) unless set */
  int torus_dims[3]; /* AR_TORUS: {X, Y, Z}, a 0 counting as 1, product N
                        (AR_EINVAL otherwise); ignored by the others */
} ar_desc;

/* Accounting of one ar_execute (primer §4.2 and §4.3 cost formulas). */
typedef struct {
  int steps;                   /* dependent steps: 2(N-1) ring, 2 log2 N
                                  Rabenseifner, 2(G-1)+2(M-1) hierarchical,
                                  1 fused */
  int launches;                /* kernels one ar_execute launches: 1 for a
                                  step plan whose every step moves at most
                                  2048 elements (its whole schedule runs in
                                  one CTA, a block barrier between steps,
                                  with the same results; when 8 bytes per
                                  element and rank fit in 160 KiB and every
                                  buffer is 4-byte aligned with count times
                                  the element size a multiple of 4, the
                                  buffers are copied to shared memory, every
                                  step runs there and the results are
                                  written back). ar_bind keeps such a plan's
                                  launch parameters and ar_execute_bound
                                  launches it directly. */
  size_t bytes_sent_per_rank;  /* largest per-rank send volume of the
                                  schedule, in bytes of the payload type */
  size_t hbm_bytes;            /* algorithmic HBM bytes of one ar_execute:
                                  every element read or written counted once
                                  per access, at its storage width. An
                                  out-of-place all-gather by steps also
                                  writes every rank's own chunk to its output:
                                  count elements more, written by the first
                                  step as it sends them (a plan run in one
                                  CTA copies them first, reading them too);
                                  these bytes are not included */
  size_t workspace_bytes;      /* device workspace ar_execute needs (0 = none) */
} ar_stats;
/* With one rank the schedule is empty (all fields 0 but workspace_bytes);
 * ar_execute then only copies to `outs` and applies `scale`, if needed. */

typedef struct ar_plan ar_plan_t;

/* Validate `desc` and build the schedule's step tables on the host (no GPU
 * call). Errors (AR_EINVAL): desc or out NULL; n_ranks outside
 * 1..AR_MAX_RANKS; unknown dtype/algo/order; AR_RABENSEIFNER or
 * AR_ORDER_TREE with N not a power of two (primer §4.3: Rabenseifner needs a
 * power-of-two N); AR_HIER or AR_ORDER_HIER with group_size < 1 or N % group_size != 0;
 * scale not finite. AR_ENOMEM if the host tables cannot be allocated. On
 * success *out owns the tables until ar_plan_destroy. */
ar_status ar_plan(const ar_desc* desc, ar_plan_t** out);

/* Fill *stats for the plan. AR_EINVAL if either pointer is NULL. */
ar_status ar_plan_stats(const ar_plan_t* plan, ar_stats* stats);

/* Copy the plan's descriptor into *desc. */
ar_status ar_plan_desc(const ar_plan_t* plan, ar_desc* desc);

/* Enqueue the all-reduce on `stream`.
 *  bufs[r]:   rank r's input buffer (count elements of dtype), device.
 *  outs:      NULL for in place (results overwrite bufs), or outs[r] = rank
 *             r's output buffer (may equal bufs[r]).
 *  workspace: device scratch of ar_stats.workspace_bytes bytes, 16-byte
 *             aligned (fp32 partial sums of the bf16 step executors), or NULL
 *             when that size is 0. Its contents on entry do not matter.
 * Every rank ends with bitwise identical results. Errors (AR_EINVAL): NULL
 * plan or bufs; a NULL or misaligned buffer; overlapping buffers; workspace
 * NULL or misaligned when one is needed. count == 0 enqueues nothing.
 * AR_ETIMEOUT, enqueuing nothing, while the current device's status word
 * records a device-side wait that ran out (sticky: see ar_plan_query). */
ar_status ar_execute(const ar_plan_t* plan, void* const* bufs, void* const* outs, void* workspace,
                     void* stream);

/* The same all-reduce from and to HOST memory; returns when the results are
 * in host memory (host_out[r] may equal host_in[r]).
 *  - AR_FUSED plans whose host buffers are page-locked and device-accessible
 *    (pinned memory on a unified-address system such as Grace-Blackwell):
 *    the single pass reads host_in and writes host_out directly over the
 *    host link; dev_bufs are not touched.
 *  - Other AR_FUSED plans: the buffers are cut into slabs; each slab is copied
 *    to dev_bufs, reduced, and copied back, with the copies of neighbouring
 *    slabs in both directions overlapping the reduction.
 *  - Step plans: copy host_in to dev_bufs, run the plan in place, copy back.
 * dev_bufs and workspace are caller-owned device memory as in ar_execute. */
ar_status ar_execute_host(const ar_plan_t* plan, const void* const* host_in, void* const* host_out,
                          void* const* dev_bufs, void* workspace, void* stream);

/* Size in bytes of the library's own device workspace used by
 * ar_execute_noalloc. */
#define AR_STATIC_WORKSPACE_BYTES (64u << 20)

/* ar_execute for callers that cannot allocate device memory. None of the
 * source pages describes such a call.
 *
 * Who needs it: callers whose device memory is owned by another allocator (a
 * framework's caching pool, or a fixed budget handed out by a host
 * application) and who may not call cudaMalloc themselves, and callers on
 * latency-sensitive paths where cudaMalloc could implicitly synchronise the
 * device. Such callers cannot provide the workspace that ar_execute asks for
 * (ar_stats.workspace_bytes; only the bf16 step-by-step plans need one).
 *
 * What it does: exactly what ar_execute(plan, bufs, outs, workspace, stream)
 * does, with the workspace taken from a fixed array of
 * AR_STATIC_WORKSPACE_BYTES bytes inside the library's device memory (every
 * GPU that loads the library holds that array until the process exits). It
 * calls no cudaMalloc, cudaFree or other device-allocating routine (like
 * every executing call, the first one on a device pins the 4-byte host status
 * word). The caller still passes the input and output buffers.
 *
 * Limits and rules:
 *  - A plan whose ar_stats.workspace_bytes exceeds AR_STATIC_WORKSPACE_BYTES
 *    is rejected with AR_EINVAL before anything is enqueued (use ar_execute
 *    with your own workspace for it). Plans that need no workspace run as
 *    with ar_execute.
 *  - The first call on each device that needs the array looks up its
 *    device address there. With lazy module loading (the CUDA default) that
 *    lookup is also the moment the library's module is loaded on the device,
 *    which reserves the AR_STATIC_WORKSPACE_BYTES array in device memory; and
 *    the first executing call on a device pins the 4-byte host status word.
 *    Either can synchronise, and on a device whose memory another pool has
 *    already taken, the module load can fail (AR_ECUDA). So make one warm-up
 *    call per device at start-up, with a plan that needs the workspace,
 *    before any pool takes the device's memory and before any stream capture
 *    begins.
 *  - All calls share the one array, and it keeps whatever the previous call
 *    left in it. That is harmless: the kernels write every workspace word
 *    before they read it within the same call, so nothing has to start at
 *    zero. But two calls that overlap on the GPU (for example on two streams
 *    at once) race on the array and give wrong results: order them on one
 *    stream or with events.
 * Other arguments and errors as ar_execute. */
ar_status ar_execute_noalloc(const ar_plan_t* plan, void* const* bufs, void* const* outs, void* stream);

/* ---------------------------------------------------------------- persistent collectives
 * A plan bound to its buffers (Scaling ML Systems, "Collective communication":
 * persistent, pre-registered collectives amortise the set-up of a collective
 * that is issued again and again on the same buffers, as DDP does every
 * step). ar_bind validates the buffers once. For a step-by-step plan it
 * records every launch of one ar_execute(plan, bufs, outs, workspace) into a
 * CUDA graph, which ar_execute_bound replays with one host call: 2(N-1) ring
 * steps cost one graph launch on the host instead of 2(N-1) kernel launches.
 * A single-pass (AR_FUSED) plan, and a step plan that runs whole in one CTA
 * (ar_stats.launches == 1), are one kernel, launched directly without the
 * argument checks (the one-CTA plan's launch parameters are built here,
 * once). The results are those of ar_execute, bit for bit. */
typedef struct ar_bound ar_bound_t;

/* Bind `plan` to its buffers (arguments and errors as ar_execute; nothing is
 * launched). The plan may be destroyed afterwards; the buffers must stay
 * allocated, at the same addresses, until ar_bound_destroy. The graph belongs
 * to the device current at this call. count == 0 makes no CUDA call. Errors:
 * AR_EINVAL (as ar_execute, or NULL out), AR_ENOMEM, AR_ECUDA (a CUDA call
 * failed while recording; nothing is left behind). Recording a step plan
 * creates CUDA graph objects (driver-managed); no device buffer is
 * allocated (a one-CTA plan keeps its launch parameters, about 29 KB, in
 * host memory). */
ar_status ar_bind(const ar_plan_t* plan, void* const* bufs, void* const* outs, void* workspace,
                  ar_bound_t** out);

/* Enqueue the bound all-reduce on `stream` (asynchronous, as ar_execute).
 * AR_EINVAL: NULL bound, or a current device other than the one at ar_bind.
 * Calls on one bound collective that overlap on the GPU (two streams at once)
 * race on its buffers, as ar_execute calls would. */
ar_status ar_execute_bound(const ar_bound_t* bound, void* stream);

void ar_bound_destroy(ar_bound_t* bound);

void ar_plan_destroy(ar_plan_t* plan);

/* ---------------------------------------------------------------- cost model
 * The primer's alpha-beta model (§4.3: T = alpha * dependent steps + bytes /
 * B) evaluated as the AI Infra Book's round model (ch. 7, §7.1.2 and §7.2.1:
 * rounds run one after another, transfers inside a round in parallel on
 * their own links, T = sum over rounds of (alpha + max over the round's
 * transfers of bytes / B_link)), over the plan's own step tables. */
typedef struct {
  double alpha;          /* seconds per dependent step (round) */
  double bw_local;       /* bytes/s of a rank's link to a rank in the same server */
  double bw_net;         /* bytes/s of a rank's link to a rank in another server */
  int ranks_per_server;  /* r and r' share a server iff r/ranks_per_server ==
                            r'/ranks_per_server; 0 = all ranks in one server */
  int in_network;        /* 1: switches reduce in flight, so AR_FUSED runs as
                            in-network reduction: one round in which every rank
                            sends its buffer once and receives the result once
                            (primer §4.4) */
  int shared_memory;     /* 1: all ranks share one memory of bandwidth bw_local
                            (virtual ranks on one GPU): every kernel launch of
                            the plan costs alpha, every step of a plan run
                            whole in one CTA AR_DEVICE_CTA_STEP_S (buffers on
                            chip) or AR_DEVICE_CTA_STEP_MEM_S, and the
                            plan's algorithmic memory bytes cost
                            bytes / bw_local */
} ar_fabric;

/* Predicted seconds of one ar_execute of `plan` on `fabric`. Transfer bytes
 * are the payload as stored (fp32 partial sums 4 bytes, bf16 values 2).
 * AR_EINVAL: NULL pointers, alpha < 0, a bandwidth <= 0 or not finite.
 * AR_EUNSUPPORTED: an AR_FUSED plan on a fabric that neither reduces in the
 * network nor shares memory. */
ar_status ar_plan_predict(const ar_plan_t* plan, const ar_fabric* fabric, double* seconds);

/* The algorithm with the smallest predicted time for `desc` on `fabric`
 * among AR_FUSED (in-network or shared memory), AR_RING, AR_RABENSEIFNER and
 * AR_RECDOUBLING (N a power of two), AR_DBTREE, and AR_HIER with
 * group_size = ranks_per_server (when that divides N and lies strictly
 * between 1 and N), in that order, an earlier one winning a tie; only
 * AR_FUSED and AR_RING for a reduce-scatter or all-gather. AR_TORUS is never
 * chosen (the fabric does not describe a torus). desc->algo is ignored.
 * Writes the choice to *algo (and its group size to *group_size if not NULL)
 * and its predicted time to *seconds (if not NULL). The choice NCCL makes per
 * call from its tables (primer §4.5), here from the model. */
ar_status ar_select(const ar_desc* desc, const ar_fabric* fabric, ar_algo* algo, int* group_size,
                    double* seconds);

/* Introspection of a step plan's schedule (host only). For step `step`
 * (0 <= step < ar_stats.steps), writes *op (0 = reduce: the receiver adds,
 * 1 = copy: the receiver overwrites) and *n_xfers, and, if xfers is not NULL,
 * up to max_xfers rows of 4 int64 values {src rank, dst rank, first element,
 * end element}: rank dst receives elements [first, end) from rank src. Empty
 * transfers (chunks with no elements) are omitted. An exchange (recursive
 * doubling) is two rows, one per direction; a tree node receiving from two
 * children in one step is two rows. AR_EINVAL for a NULL
 * plan/op/n_xfers, an AR_FUSED plan, or step out of range. */
ar_status ar_plan_transfers(const ar_plan_t* plan, int step, int* op, int* n_xfers, int64_t* xfers,
                            int max_xfers);

/* ---------------------------------------------------------------- buckets
 * DDP bucket fusion (Scaling ML Systems, "Collective communication", section
 * "Bucket fusion"): gradients are grouped into buckets of a capped byte size,
 * filled in the reverse of the parameters' forward order, one all-reduce per
 * bucket.
 *
 * Tensors are numbered 0..n_tensors-1 in FORWARD order. A bucket always holds
 * a contiguous range of tensor ids [t_begin, t_end); inside the bucket they
 * are packed in DESCENDING id order (the order backward produces them), so
 * tensor t sits at packed offset sum(counts[u] for t < u < t_end).           */

/* Assign tensors to buckets. counts[t] = elements of tensor t (forward
 * order), elem_bytes = bytes per gradient element, cap_bytes = bucket cap.
 * Filling starts at the last tensor; a bucket closes when the next tensor
 * would take it over cap_bytes; a tensor larger than the cap gets its own
 * bucket. Outputs: bucket_of_tensor[t] (bucket 0 fills first) and
 * *n_buckets. Host only. AR_EINVAL: NULL pointers, n_tensors < 1,
 * elem_bytes == 0. */
ar_status ar_bucket_plan(const size_t* counts, int n_tensors, size_t elem_bytes, size_t cap_bytes,
                         int* bucket_of_tensor, int* n_buckets);

/* Pack bucket [t_begin, t_end): bucket[r][packed offset of t + e] =
 * fp32(tensors[r * n_tensors + t][e]) for every rank r (bf16 widened
 * exactly). bucket[r] has room for the bucket's element total. */
ar_status ar_bucket_pack(int n_ranks, const void* const* tensors, const size_t* counts, int n_tensors,
                         int t_begin, int t_end, ar_dtype in_dtype, void* const* bucket, void* stream);

/* Unpack bucket [t_begin, t_end): tensors[r * n_tensors + t][e] =
 * round(scale * bucket[r][packed offset of t + e]) in out_dtype (bf16:
 * round to nearest even, once). */
ar_status ar_bucket_unpack(int n_ranks, const void* const* bucket, float scale, ar_dtype out_dtype,
                           void* const* tensors, const size_t* counts, int n_tensors, int t_begin,
                           int t_end, void* stream);

/* Pack + ring all-reduce + unpack of bucket [t_begin, t_end) in ONE pass with
 * no pack buffer: every element of every rank's tensors is read once and the
 * scaled, rounded result written once to every rank. The sum of packed
 * element e runs in ring order over the packed bucket (chunk boundaries at
 * floor(c * bucket_count / N)), so the result is bit-identical to
 * ar_bucket_pack + AR_RING (fp32) + ar_bucket_unpack. dtype is the tensors'
 * type. In place. sm_budget and kernel as in ar_desc (0 = all SMs, automatic
 * kernel); AR_KERNEL_BULK with N > 24 returns AR_EUNSUPPORTED. */
ar_status ar_bucket_allreduce(int n_ranks, void* const* tensors, const size_t* counts, int n_tensors,
                              int t_begin, int t_end, ar_dtype dtype, float scale, int sm_budget,
                              ar_kernel kernel, void* stream);

/* ---------------------------------------------------------------- compression
 * Blockwise INT8 gradient compression with error feedback (Scaling ML
 * Systems, "Collective communication", the section on gradient compression:
 * "Quantization: reducing precision" gives the INT8 scale max|g| / 127 and the
 * codes round(g / scale); "Blockwise quantization for gradient communication"
 * gives one scale per block of b elements and a message of d one-byte codes
 * plus 4 bytes of fp32 scale per block; "Error feedback and residual
 * accumulation" gives x = g + e, transmit C(x), keep e' = x - C(x)).
 *
 * Arithmetic, per rank and block k = [k*block, min((k+1)*block, count)) (the
 * last block may be short), every operation one IEEE fp32 operation rounded to
 * nearest even:
 *   x = g + e (x = g without error feedback; bf16 g widened exactly)
 *   s = max|x| / 127
 *   q = the nearest integer to x / s, ties to even, clamped to [-127, 127];
 *       q = 0 for every element of a block whose s is 0
 *   d = q * s (the value the receiver reconstructs)
 *   e' = x - d
 * The page writes round() without a tie rule; ties to even (the IEEE default)
 * is this library's reading. The reduction sums the N ranks' d in rank order,
 * ((d_0 + d_1) + ...) + d_{N-1}, multiplies by `scale` once and rounds once to
 * the output type (bf16: nearest even); no partial sum is re-quantised (the
 * page's interfaces that fuse quantisation and reduction).
 *
 * Layout: rank r's codes are `count` int8 values (codes[r][e] for element e),
 * its scales ceil(count / block) fp32 values (scales[r][k] for block k), its
 * residuals `count` fp32 values. block is a power of two from
 * AR_COMPRESS_MIN_BLOCK to AR_COMPRESS_MAX_BLOCK (the page's typical sizes are
 * 64 and 128). count == 0 enqueues nothing. Buffers follow the conventions at
 * the top of this file (caller-owned device memory, 16-byte aligned, no
 * overlaps unless stated). */
#define AR_COMPRESS_MIN_BLOCK 16
#define AR_COMPRESS_MAX_BLOCK 1024

/* Sizes of one rank's message for `count` elements: *n_scales = ceil(count /
 * block) and *message_bytes = count + 4 * ceil(count / block), the page's d +
 * 4d/b (either output may be NULL). Host only. AR_EINVAL: block not a power of
 * two in [AR_COMPRESS_MIN_BLOCK, AR_COMPRESS_MAX_BLOCK]. */
ar_status ar_compress_sizes(size_t count, int block, size_t* n_scales, size_t* message_bytes);

/* Compress every rank's gradient into its message (the sending side).
 *  grads[r]:     count elements of dtype (AR_F32 or AR_BF16), read only.
 *  residuals:    NULL for no error feedback, or residuals[r] = rank r's fp32
 *                residual e (count values): read as e, overwritten with e'.
 *  codes[r]:     count int8 codes, written.
 *  scales[r]:    ceil(count / block) fp32 scales, written.
 * AR_EINVAL: n_ranks outside 1..AR_MAX_RANKS; a bad block or dtype; a NULL
 * array; a NULL or misaligned pointer; overlapping buffers. */
ar_status ar_compress(int n_ranks, size_t count, int block, ar_dtype dtype, const void* const* grads,
                      void* const* residuals, void* const* codes, void* const* scales, void* stream);

/* Sum the N ranks' messages (the receiving side): every outs[r] (count
 * elements of out_dtype) is written with round(scale * sum over ranks in rank
 * order of codes[r'][e] * scales[r'][e / block]). codes and scales as written
 * by ar_compress. AR_EINVAL as ar_compress, and for a non-finite scale. */
ar_status ar_compressed_reduce(int n_ranks, size_t count, int block, const void* const* codes,
                               const void* const* scales, float scale, ar_dtype out_dtype, void* const* outs,
                               void* stream);

/* ar_compress followed by ar_compressed_reduce in one pass, without message
 * buffers: every element of every rank is read once (with its residual) and
 * the result written once to every rank; with error feedback each residual is
 * read and rewritten once. The results (outputs and residuals) are
 * bit-identical to the two calls. outs: NULL for in place (results overwrite
 * grads), else outs[r] may equal grads[r]. Output dtype = dtype.
 * AR_EINVAL as ar_compress, and for a non-finite scale. */
ar_status ar_compressed_allreduce(int n_ranks, size_t count, int block, ar_dtype dtype, const void* const* grads,
                                  void* const* residuals, float scale, void* const* outs, void* stream);

/* ---------------------------------------------------------------- status */

/* Every device-side wait in the library is bounded. One that runs out (for
 * example an mbarrier wait of a bulk-copy kernel) sets the device's sticky
 * status word, both in device memory and in a host-visible copy (page-locked
 * mapped host memory). The error surfaces after the call that enqueued the
 * work has returned, since initiation is non-blocking (Scaling ML Systems,
 * "Collective communication"). From then on the executing calls
 * (ar_execute, ar_execute_host, ar_execute_noalloc, ar_bind,
 * ar_execute_bound, ar_bucket_allreduce) on that device return AR_ETIMEOUT
 * and enqueue nothing, until ar_device_status(1) clears the word. */

/* Read (and clear, if clear != 0) the calling device's sticky status word.
 * Synchronises the device. Returns AR_OK or AR_ETIMEOUT (or AR_ECUDA). */
ar_status ar_device_status(int clear);

/* The plan's asynchronous error, without synchronising and without any CUDA
 * call: AR_ETIMEOUT if the host-visible status word of the device that last
 * executed `plan` (ar_execute, ar_execute_host, ar_execute_noalloc or
 * ar_bind) records a wait that ran out, else AR_OK (also for a plan never
 * executed). A kernel still running has not reported yet: after the stream
 * has drained, the answer covers all of the plan's work. Does not clear the
 * word. AR_EINVAL if plan is NULL. */
ar_status ar_plan_query(const ar_plan_t* plan);

/* Failure-path self-test: launches one thread that waits, with a bound of
 * `polls` polls, on an mbarrier that nothing will ever complete. The wait gives
 * up, sets the device status word and the kernel returns; a following
 * ar_device_status reports AR_ETIMEOUT. This exercises the same bounded wait
 * that the bulk-copy kernels use, without any fault and without a hang. */
ar_status ar_selftest_wait_timeout(unsigned int polls, void* stream);

/* Self-test of the compression's block scale (Scaling ML Systems, "Blockwise
 * quantization": the scale is max|x| / 127, here an fp32 quotient rounded to
 * nearest). The kernels compute it without a division, by a product with the
 * rounded reciprocal of 127 and an FMA correction. This call compares that
 * computation with the IEEE division for every non-negative float bit pattern
 * (2^31 of them: zero, subnormals, normals, +inf and NaNs, where both give a
 * NaN) on the current device, and writes the number of differing results to
 * *mismatches (0 when the method is exact). Synchronises the device.
 * AR_EINVAL if mismatches is NULL; AR_ECUDA on a CUDA error. */
ar_status ar_selftest_scale_quotient(unsigned long long* mismatches);

/* Human-readable name of a status code (static string). */
const char* ar_status_string(ar_status status);

/* Library version, for the binding's load check. */
int ar_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AR_GB300_H */
