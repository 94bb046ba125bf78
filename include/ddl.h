/*
 * ddl.h -- C ABI of libddl: the synchronous-SGD gradient all-reduce of P
 * logical data-parallel workers whose gradient buffers all live in the HBM of
 * one GPU (GB300, sm_103a).
 *
 * What the operation is (sources cited by page title and section):
 *  - Data-parallel training adds one step to every iteration: the workers'
 *    gradients are averaged with an all-reduce collective ("索尼发布新的方法，
 *    在ImageNet数据集上224秒内成功训练了ResNet-50", section "2大方法解决不稳定
 *    问题"; Baidu ring-allreduce write-up, final page, section "总结").
 *  - Three schedules: the ring all-reduce, a chunked reduce-scatter then an
 *    all-gather (Baidu write-up, "总结", after Patarasuk & Yuan 2009); the
 *    multi-ring pattern of "[论文解读] PowerAI DDL" (abstract, "提出的方法"),
 *    k rings over different rank orders; and the 2D-torus all-reduce of the
 *    Sony page, section "2D-Torus All-reduce", Fig. 1 and Fig. 2: on an X x Y
 *    grid, a horizontal reduce-scatter, a vertical all-reduce and a
 *    horizontal all-gather.
 *  - FP16 gradient communication (Sony page, section "训练设置").
 *  - Buckets in reverse-layer order, so the all-reduce of the output layers
 *    starts while back-propagation still runs (Baidu write-up, opening
 *    paragraphs of its final page).
 *
 * Result contract: after ddl_allreduce every rank buffer holds, bit for bit,
 * what the schedule computes when run send-by-send with IEEE binary32 adds in
 * its own order (fp16 mode: binary16 on every hop, binary32 adds, the owner's
 * last add kept in binary32, multiplied by the scale, rounded once).  The
 * rules that fix that order (chunk split, ring direction, multi-ring orders,
 * torus layout, bucket packing) are stated at each call below.
 *
 * Conventions for every call:
 *  - No call aborts or throws; each returns a ddl_status_t.  Argument errors
 *    are found before any work is queued and leave no side effects.
 *  - "stream" is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  GPU work is queued on it asynchronously; calls return after
 *    enqueue.
 *  - A plan binds to the CUDA device that is current at its first GPU call;
 *    later GPU calls must be made with that device current.
 *  - A plan is not thread-safe: do not call into one plan from two host
 *    threads at once, and do not queue two all-reduces of one plan that may
 *    run concurrently on the GPU over the same buffers.
 *  - Failure testing: with the environment variable
 *    DDL_INJECT_ALLOC_FAILURE=1, the upload of a plan's device tables fails
 *    as if the device were out of memory (DDL_ERR_OOM, nothing queued); the
 *    plan uploads them at its next call once the variable is unset.
 */
#ifndef DDL_H_
#define DDL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DDL_OK = 0,
  DDL_ERR_INVALID_ARG = 1,  /* bad argument; nothing was queued */
  DDL_ERR_UNSUPPORTED = 2,  /* valid request this library does not build (e.g. P > 256) */
  DDL_ERR_OOM = 3,          /* host or device allocation of plan tables failed */
  DDL_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
  DDL_ERR_DEVICE_CHECK = 5  /* a kernel's own check failed (see ddl_plan_check) */
} ddl_status_t;

typedef enum {
  DDL_FP32 = 0, /* binary32 storage and arithmetic */
  DDL_FP16 = 1  /* binary16 storage and hops, binary32 adds */
} ddl_dtype_t;

typedef enum { DDL_RING = 0, DDL_MULTIRING = 1, DDL_TORUS = 2 } ddl_topo_kind_t;

/* kind = DDL_RING: k, X, Y ignored.
 * kind = DDL_MULTIRING: k rings, 1 <= k <= phi(P); ring j uses the rank order
 *   pi_j(t) = t * s_j mod P, s_j the j-th smallest integer in [1, P) coprime
 *   to P (s_0 = 1 when P = 1).
 * kind = DDL_TORUS: X * Y == P; rank r sits at column x = r mod X, row
 *   y = r / X; rows are the horizontal rings, columns the vertical ones. */
typedef struct {
  int32_t kind;
  int32_t k;
  int32_t X;
  int32_t Y;
} ddl_topology_t;

typedef enum {
  DDL_MODE_FUSED = 0,     /* one HBM pass per bucket, schedule order (bit-exact) */
  DDL_MODE_STEPWISE = 1,  /* one kernel per communication step (bit-exact; slow) */
  DDL_MODE_RANKORDER = 2  /* one HBM pass, ranks added in order 0..P-1 with no
                             intermediate binary16 rounding; accurate to the
                             fp64 sum within 1e-6 (fp32) / 2e-3 (fp16)
                             normwise, but not the schedule's bits */
} ddl_mode_t;

typedef enum {
  DDL_KERNEL_AUTO = 0,  /* the library's choice (the same as DDL_KERNEL_LDG for ddl_allreduce;
                           see ddl_allreduce_host and the bucket scheduler for the others) */
  DDL_KERNEL_LDG = 1,   /* the column passes with 16-byte loads and stores: the register pass,
                           and for small buffers the small-item and shared-memory latency passes
                           (ddl_plan_kernel_name reports which one a plan takes) */
  /* 2 is not used (a staged pass with bulk stores, removed: it was slower
     than the register pass at every P measured) */
  DDL_KERNEL_BULK_LOAD = 3, /* bulk async loads of all ranks' tiles into shared memory, stores
                               from registers (the zero-copy host pass's kernel) */
  /* 4 is not used (2D tensor-map loads from a slab, removed: slower than
     the register pass at every P measured) */
  DDL_KERNEL_CHUNKED = 5    /* bulk async loads of the register pass's tiles (up to 8 KB per
                               rank) into shared memory, 2 ranks per stage in fold order,
                               the fold kept in registers across an item's stages, stores
                               from registers (the overlap side stream's kernel for buckets of full-size
                               8 KB work items; smaller ones take the library's own choice) */
} ddl_kernel_t;

typedef struct ddl_plan* ddl_plan_t;

/* Creates a plan for P rank buffers of N elements each: the averaging step
 * of synchronous data-parallel SGD, in which every worker holds a full copy
 * of the gradient and all of them end with the same mean (Baidu
 * ring-allreduce write-up, final page, opening paragraphs and "总结"; Sony
 * page, "2大方法解决不稳定问题").  topo picks the schedule: the ring
 * (Baidu write-up, "总结"), the multi-ring ("[论文解读] PowerAI DDL",
 * ABSTRACT and "提出的方法") or the 2D torus (Sony page, "2D-Torus
 * All-reduce", Fig. 1 and Fig. 2); dtype DDL_FP16 is the half-precision
 * gradient communication of the Sony page, "训练设置".
 *  P: 1..256.  N: >= 1 elements per rank.
 *  bucket_bytes: 0 = the whole buffer is one bucket; otherwise buckets of at
 *    least this many bytes, taken from the highest addresses down (bucket 0 =
 *    output layers, issued first).  Without a layer list (see
 *    ddl_plan_set_layers) bucket b covers elements
 *    [max(0, N - (b+1)*B), N - b*B), B = bucket_bytes / element size.
 *  Inside a bucket of n elements, a split into m parts gives part i
 *  n/m + (i < n%m) elements starting at i*(n/m) + min(i, n%m); the ring uses
 *  m = P chunks, the multi-ring k slices of P chunks, the torus X row chunks
 *  of Y sub-chunks.
 * Host-only: allocates the plan and builds its tables; touches no GPU.
 * On success *out owns the plan (free with ddl_plan_destroy). */
ddl_status_t ddl_plan_create(int P, size_t N, ddl_dtype_t dtype, ddl_topology_t topo,
                             size_t bucket_bytes, ddl_plan_t* out);

/* Optional: the gradient's tensors, numel_fwd_order[0..n_tensors-1] in
 * forward (input-to-output) order at increasing addresses; they must sum to
 * N.  Buckets are then packed greedily from the last tensor backwards, a
 * bucket closing once it holds >= bucket_bytes; the remainder is the last
 * bucket.  The array is copied.  Host-only. */
ddl_status_t ddl_plan_set_layers(ddl_plan_t plan, int n_tensors, const size_t* numel_fwd_order);

/* Makes the plan an n-dimensional torus: dims[0..ndims-1] (1 <= ndims <= 4,
 * each >= 1, product == P), rank r at coordinates x_k = (r / (D_0...D_{k-1}))
 * mod D_k (dim 0 varies fastest).  The schedule generalises the 2D-torus of
 * "索尼发布新的方法，在ImageNet数据集上224秒内成功训练了ResNet-50"
 * ("2D-Torus All-reduce", Fig. 1) to the several-level rings with which
 * "[论文解读] PowerAI DDL" ("提出的方法") adapts to a machine's topology:
 * reduce-scatter along dims 0..d-2, each line of D_k ranks working on the
 * range it has reduced so far (a rank at x_k keeps part (x_k + 1) mod D_k),
 * all-reduce along dim d-1 (scale applied at its owner), then all-gather
 * along dims d-2..0.  Element results are d nested left folds, innermost over
 * dim 0.  Trailing dims of size 1 are dropped; dims {X, Y} give exactly the
 * DDL_TORUS result and dims {P} the ring's.  Host-only. */
ddl_status_t ddl_plan_set_torus_dims(ddl_plan_t plan, int ndims, const int* dims);

/* Selects the mode (default DDL_MODE_FUSED).  DDL_MODE_FUSED and
 * DDL_MODE_STEPWISE give the bits of the schedule run send by send (the ring
 * of the Baidu write-up, "总结"; the torus of the Sony page, "2D-Torus
 * All-reduce"; fp16 hops of its "训练设置"): the first in one HBM pass, the
 * second with one kernel per communication step.  DDL_MODE_RANKORDER adds
 * the ranks in plain order 0..P-1, which the pages do not describe; it is
 * the reordered fast mode, accurate to the binary64 sum within 1e-6 (fp32)
 * or 2e-3 (fp16) normwise and within the error bound of a P-term binary32
 * sum element by element.  Host-only. */
ddl_status_t ddl_plan_set_mode(ddl_plan_t plan, ddl_mode_t mode);

/* Selects the fused kernel variant (default DDL_KERNEL_AUTO; values 2 and 4
 * return DDL_ERR_INVALID_ARG).  Results are identical for every variant.
 * Host-only. */
ddl_status_t ddl_plan_set_kernel(ddl_plan_t plan, ddl_kernel_t kernel);

/* All-reduces every bucket, in place, in issue order (fused and rank-order
 * modes: one launch covering every bucket's work, bucket 0's first).
 *  rank_bufs: host array of P device pointers, rank r's N elements (binary32,
 *    or binary16 for DDL_FP16).  The buffers must be distinct and must not
 *    overlap; the caller owns them and keeps them valid until the queued work
 *    has finished.  Pointers that are not 16-byte aligned are accepted and
 *    take a slower element-wise path; results do not change.
 *  scale: binary32 factor applied once per element (1/P gives the mean).
 * The first call on a device uploads the plan's tables (device memory owned
 * by the plan) and creates its side stream and events.
 * Stream order is kept.  The launch is a programmatic dependent of the kernel
 * before it on `stream`: its CTAs may start and read the plan's tables while
 * that kernel drains, but touch no rank buffer until every earlier kernel on
 * the stream has finished and its writes are visible. */
ddl_status_t ddl_allreduce(ddl_plan_t plan, void* const* rank_bufs, float scale, void* stream);

/* All-reduce followed by the synchronous-SGD update, in the same HBM pass.
 * Every iteration of synchronous data-parallel SGD runs forward, backward,
 * the gradient all-reduce and the update (Baidu write-up, opening paragraph);
 * the pages' own large-batch optimizer (LARS, on the Sony page, "训练设置")
 * lost its formula, so this is momentum SGD.  After the all-reduce of
 * grad_bufs (exactly as ddl_allreduce computes it, schedule order, scale),
 * with g the averaged gradient as stored (binary16 for DDL_FP16), every rank
 * r updates its own binary32 copies, element by element:
 *   d = g + weight_decay * p;  v = momentum * v + d;  p = p - lr * v
 * each product and sum rounded to binary32 on its own (no fused
 * multiply-add).  This saves the update's second read of the gradient, and
 * all of the gradient's write-back when keep_grads == 0 (grad_bufs are then
 * left as they were, not averaged).
 *  param_bufs: P device arrays of N binary32 parameters, one per rank.
 *  mom_bufs: P device arrays of N binary32 momenta; NULL only with
 *    momentum == 0 (then v = d).
 * All 2P or 3P buffers (with the gradients) must be distinct and
 * non-overlapping.  Fused and rank-order modes of 1-, 2-level schedules (ring,
 * multi-ring, 2D torus) with P <= 128; other plans return
 * DDL_ERR_UNSUPPORTED. */
ddl_status_t ddl_allreduce_sgd(ddl_plan_t plan, void* const* grad_bufs, float* const* param_bufs,
                               float* const* mom_bufs, float scale, float lr, float momentum, float weight_decay,
                               int keep_grads, void* stream);

/* ddl_allreduce for rank buffers laid out in one slab: rank r's N elements
 * start at base + r * rank_stride_bytes (rank_stride_bytes >= N * element
 * size when P > 1; the slab is caller-owned device memory).  The same call,
 * with the P pointers computed from the slab. */
ddl_status_t ddl_allreduce_slab(ddl_plan_t plan, void* base, size_t rank_stride_bytes, float scale, void* stream);

/* All-reduces bucket b only (0 <= b < ddl_plan_num_buckets). */
ddl_status_t ddl_allreduce_bucket(ddl_plan_t plan, int bucket, void* const* rank_bufs, float scale,
                                  void* stream);

/* End-to-end form for gradients held in host memory; the host buffers are
 * updated in place.
 *  host_bufs: P host pointers, N elements each.  They must stay valid until
 *    the stream reaches the end of the queued work.
 *  dev_bufs: P device buffers as for ddl_allreduce (caller-owned staging):
 *    the call copies the host buffers in, all-reduces, and copies the results
 *    back, pipelined over element ranges on the plan's own copy-in, compute
 *    and copy-out streams (joined to `stream` at both ends).  Page-locked
 *    host memory is needed for the copies to overlap.
 *  dev_bufs == NULL: no staging.  The fused pass reads and writes the host
 *    buffers directly over the host link.  They must be memory the GPU can
 *    reach: page-locked (cudaHostAlloc / cudaHostRegister), managed, or
 *    pageable on systems with coherent GPU access to pageable memory; other
 *    memory returns DDL_ERR_INVALID_ARG.  Not available in stepwise mode
 *    (DDL_ERR_UNSUPPORTED).  With DDL_KERNEL_AUTO, P <= 64, and 16-byte
 *    aligned page-locked buffers (not the n-D torus), the pass is the
 *    bulk-load staged pass over a second set of work items sized for it:
 *    its whole-tile copies move more over the host link.  The first such
 *    call builds and uploads those items (an allocation); later calls reuse
 *    them until the plan changes.  Results are the same bits either way. */
ddl_status_t ddl_allreduce_host(ddl_plan_t plan, void* const* host_bufs, void* const* dev_bufs, float scale,
                                void* stream);

/* Overlap with back-propagation: the all-reduce of the output layers'
 * gradients starts while the earlier layers' are still being computed
 * (Baidu write-up, final page, opening paragraphs).  ddl_overlap_begin
 * records the buffers and scale; each ddl_bucket_ready(b, stream) marks
 * bucket b's gradients complete at the current point of `stream` (an event),
 * after which the plan's side stream all-reduces bucket b; ddl_overlap_end
 * makes `stream` wait for every bucket issued so far, then all-reduces on
 * `stream` every bucket that was never signalled, so every bucket is reduced
 * once per begin/end pair.  Each bucket is signalled at most once per
 * begin/end pair (a second signal returns DDL_ERR_INVALID_ARG); bucket 0
 * (output layers) is normally signalled first. */
ddl_status_t ddl_overlap_begin(ddl_plan_t plan, void* const* rank_bufs, float scale, void* stream);
ddl_status_t ddl_bucket_ready(ddl_plan_t plan, int bucket, void* stream);
ddl_status_t ddl_overlap_end(ddl_plan_t plan, void* stream);

/* Allocation-free form of ddl_allreduce, with no plan.  The web pages have no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc -- a framework whose device memory all belongs to its own pool,
 * a training loop that must not take cudaMalloc's implicit device
 * synchronisation, or a deployment that fixes its memory footprint at
 * start-up.  The arguments mean what they mean for ddl_plan_create,
 * ddl_plan_set_layers (n_tensors = 0: no layer list) and ddl_allreduce
 * (topo.kind DDL_RING, DDL_MULTIRING or DDL_TORUS); the mode is
 * DDL_MODE_FUSED and the results are bit-identical to a plan's, whose table
 * code it runs.
 *  - The fused kernel's work tables live in one static 1 MiB device array
 *    inside this library (every GPU that loads it holds the array until the
 *    process exits) instead of plan-owned device memory.  Problems whose
 *    tables need more than that (about 60,000 tiles of 8 KB per rank, i.e.
 *    roughly 480 MB per rank) return DDL_ERR_UNSUPPORTED before any work.
 *  - No cudaMalloc, cudaFree or other allocating call, and no host heap use.
 *    The tables are written into a static host buffer and copied into the
 *    array with cudaMemcpyAsync on `stream`, ordered before the kernel; the
 *    call returns once the runtime holds its own copy of the host buffer.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the array, which keeps the last call's tables; each call
 *    rewrites what it uses and clears the kernel error word (read it with
 *    ddl_noalloc_check).  Calls whose GPU work overlaps (other streams, other
 *    host threads) race on the array and must be ordered by the caller.  Host
 *    threads are serialised inside. */
ddl_status_t ddl_allreduce_noalloc(int P, size_t N, ddl_dtype_t dtype, ddl_topology_t topo, size_t bucket_bytes,
                                   int n_tensors, const size_t* numel_fwd_order, void* const* rank_bufs,
                                   float scale, void* stream);

/* Reads the kernel error word that the last ddl_allreduce_noalloc on the
 * current device left in the static array, without allocating: waits for
 * `stream` (the stream of that call), copies the word into a static host
 * word, and returns DDL_ERR_DEVICE_CHECK if the kernel found a bad table
 * entry (the word is then cleared), DDL_OK otherwise or when no
 * allocation-free call has run on this device.  The web pages have no
 * counterpart. */
ddl_status_t ddl_noalloc_check(void* stream);

/* Bucket table: *n buckets; bucket b covers elements [*begin, *end). */
ddl_status_t ddl_plan_num_buckets(ddl_plan_t plan, int* n);
ddl_status_t ddl_plan_bucket_range(ddl_plan_t plan, int bucket, size_t* begin, size_t* end);

/* What the schedule would move between workers: the total number of
 * elements sent over all messages (2(P-1)N for every schedule, so each
 * worker sends and receives 2(P-1)/P of the gradient: the Baidu write-up's
 * "each GPU sends and receives about 2.4 GB" for a 1.2 GB gradient, final
 * page, opening paragraphs) and the number of sequential communication steps
 * (ring and multi-ring 2(P-1), torus 2(X-1)+2(Y-1), per bucket; the torus's
 * fewer steps are the point of the Sony page's "2D-Torus All-reduce").
 * Host-only. */
ddl_status_t ddl_plan_traffic(ddl_plan_t plan, uint64_t* elems_moved_total, uint64_t* steps);

/* alpha-beta cost of the schedule on a cluster of P real workers, each with
 * links_per_worker (>= 1) network links.  In every communication step all
 * workers send at once; a worker's message of concurrent ring j travels on
 * its link j mod links_per_worker, messages sharing a link one after another;
 * the step costs alpha_s (latency) plus beta_s_per_byte times the bytes of
 * the busiest link of any worker; the all-reduce costs the sum over its steps
 * and buckets.  Ring and torus send one message per worker per step:
 * 2(P-1)(alpha + (n/P)e beta) and 2(X-1)(alpha + (n/X)e beta) +
 * 2(Y-1)(alpha + (n/(XY))e beta), for any link count.  A k-ring multi-ring
 * sends k messages of about n/(kP) elements per worker per step: with one
 * link it costs what the ring costs (plus the ragged splits), with k links
 * its bandwidth term shrinks k-fold.  This is the latency / bandwidth
 * trade-off that "[论文解读] PowerAI DDL" (ABSTRACT) names for its multi-ring
 * pattern; one link per worker compares the three schedules on equal
 * hardware.  The Baidu write-up's example (a 1.2 GB gradient, about 6 GB/s
 * InfiniBand, about 400 ms per iteration; final page, opening paragraphs) is
 * the ring in this model with alpha = 0.  Host-only.  alpha_s,
 * beta_s_per_byte >= 0; DDL_ERR_INVALID_ARG otherwise. */
ddl_status_t ddl_plan_cost(ddl_plan_t plan, double alpha_s, double beta_s_per_byte, int links_per_worker,
                           double* seconds);

/* Introspection: the fold order of element i as the plan's tables hold it:
 * order[0..P-1] = ranks in the order they are added, *inner = group length
 * (X for the torus, else P), *groups = Y for the torus, else 1.  Host-only. */
ddl_status_t ddl_plan_fold_order(ddl_plan_t plan, size_t i, int32_t* order, int32_t* inner, int32_t* groups);

/* Number of kernels this plan has launched since it was created. */
ddl_status_t ddl_plan_launches(ddl_plan_t plan, uint64_t* n);

/* Introspection: the kernel that ddl_allreduce launches for this plan, in its
 * current mode and kernel choice, when every rank buffer is 16-byte aligned:
 * "fold_ldg_kernel" (the register pass), "fold_small_kernel" (small items of
 * one unrounded fold group), "fold_lat_kernel" or "fold_lat_kernel (one
 * group)" (small items of P >= 16 ranks staged in shared memory),
 * "fold_nd_kernel", "fold_nd_h2_kernel" or "fold_lat_nd_kernel" (n-D torus),
 * "fold_bulk_kernel", "fold_chunked_kernel" (staged choices), or "step_kernel"
 * (stepwise mode).  *name points to a static string.  Host-only; the one rule
 * that depends on the device (how many latency-pass CTAs fit at once, for a
 * single fold group) assumes a GB300's 152 SMs when no device is present. */
ddl_status_t ddl_plan_kernel_name(ddl_plan_t plan, const char** name);

/* Waits for the plan's device work and reads its kernels' error word:
 * DDL_ERR_DEVICE_CHECK if a kernel found a bad table entry or a bounded wait
 * ran out (the word is then cleared), DDL_OK otherwise. */
ddl_status_t ddl_plan_check(ddl_plan_t plan);

/* Self-test of the bounded waits in the staged kernels: queues one CTA that
 * waits on an mbarrier nothing arrives at, gives up after limit_us
 * microseconds (1..1,000,000) and records the timeout in the plan's error
 * word, as a staged pass whose copies never completed would.  The next
 * ddl_plan_check then returns DDL_ERR_DEVICE_CHECK and clears the word; the
 * CUDA context stays usable.  The pages have no counterpart: this checks the
 * library's own failure path without faulting or hanging the GPU. */
ddl_status_t ddl_selftest_wait_timeout(ddl_plan_t plan, uint32_t limit_us, void* stream);

/* A static string for a status code. */
const char* ddl_status_string(ddl_status_t status);

/* Frees the plan, its device tables, side stream and events.  Waits for the
 * plan's side stream first.  NULL is accepted. */
ddl_status_t ddl_plan_destroy(ddl_plan_t plan);

#ifdef __cplusplus
}
#endif

#endif /* DDL_H_ */
