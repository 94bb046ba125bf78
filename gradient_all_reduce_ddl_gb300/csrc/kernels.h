// kernels.h -- launch records of the all-reduce kernels (internal).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace ddl {

// Error word bits written by kernels (read back by ddl_plan_check).
enum : uint32_t {
  kErrBadItem = 1u,      // a work item points outside the segment table
  kErrBadOrder = 2u,     // a segment's group shape does not cover P ranks
  kErrWaitTimeout = 4u,  // a bounded wait on an mbarrier ran out
  kErrBadXfer = 8u       // a message names a rank outside 0..P-1
};

// Segment s's rank order is orders[s*P .. s*P + P); the fold shape (inner,
// groups) is the same for every segment of a plan, so kernels read neither
// the segment records nor more than one table entry before their data.
struct FoldParams {
  const Item* items;
  const Segment* segs;  // not read by the kernels (kept for the tables' owner)
  const uint8_t* orders;
  uint32_t* err;
  uint32_t item0;      // first item of this launch
  uint32_t n_segs;
  uint32_t n_orders;
  int32_t P;
  float scale;
  int32_t round_hops;  // binary16 storage: round every intermediate result
  int32_t vector_ok;   // every rank pointer is 16-byte aligned
  uint32_t n_items;    // items in this launch (persistent kernels)
  uint32_t tile_bytes; // bytes per rank of the largest item
  int32_t nlev;        // n-D torus: fold levels (0 = two-level fold: inner, groups)
  uint16_t lev[kMaxDims];  // level sizes, innermost first (the torus dims)
  int32_t top;         // highest level of size > 1 (its last add is the final one)
  int32_t inner;       // two-level fold: group length (P for ring / multi-ring, X for the torus)
  int32_t groups;      // number of groups (1, or Y for the torus)
  void* bufs[kMaxP];   // rank r's buffer
};

// Fused all-reduce + momentum SGD (rank pointers of three buffer sets).
constexpr int kMaxPSgd = 128;
struct SgdParams {
  const Item* items;
  const Segment* segs;  // not read by the kernel
  const uint8_t* orders;
  uint32_t* err;
  uint32_t item0;
  uint32_t n_segs;
  uint32_t n_orders;
  int32_t P;
  int32_t inner, groups;  // the plan's two-level fold shape
  float scale, lr, mu, wd;
  int32_t round_hops;
  int32_t vector_ok;   // every buffer 16-byte aligned
  int32_t keep_grads;  // store the all-reduced gradient back
  int32_t has_mom;     // momentum buffers given (else v = d)
  uint32_t tile_bytes; // gradient bytes per rank of the largest item
  void* grads[kMaxPSgd];
  float* params[kMaxPSgd];
  float* moms[kMaxPSgd];
};

cudaError_t launch_sgd(const SgdParams& p, uint32_t n_items, bool f16, cudaStream_t stream);

struct StepParams {
  const Xfer* xfers;
  uint32_t* err;
  uint32_t xfer0;
  int32_t P;
  float scale;
  int32_t vector_ok;
  void* bufs[kMaxP];
};

// Variants of the fused pass: the register pass, the bulk-load staged pass
// (all ranks of a tile per stage), the rank-chunked staged pass.
enum FoldVariant : int { kVarLdg = 1, kVarBulkLoad = 3, kVarChunked = 4 };

// The pass a fused launch of n_items work items takes.  launch_fold launches
// exactly this choice; it depends on the plan's shape, the buffers' alignment
// (p.vector_ok), the variant and, for a single fold group, on how many CTAs of
// the latency pass fit on the device at once.
enum FoldPass : int {
  kPassRegister = 0,   // fold_ldg_kernel
  kPassSmallItem,      // fold_small_kernel: one unrounded group, small items
  kPassLatency,        // fold_lat_kernel, several groups
  kPassLatencySingle,  // fold_lat_kernel, one group
  kPassNdRegister,     // fold_nd_kernel, fold_nd_h2_kernel (binary16 hops)
  kPassNdLatency,      // fold_lat_nd_kernel
  kPassBulkLoad,       // fold_bulk_kernel
  kPassChunked         // fold_chunked_kernel
};
FoldPass fold_pass(const FoldParams& p, uint32_t n_items, bool f16, int variant);
// The kernel's name (a static string); packed_hops: binary16 storage with
// rounded hops.
const char* fold_pass_kernel(FoldPass pass, bool packed_hops);

// early_launch: launch the register passes as programmatic dependents of the
// kernel before them on the stream (they read only the plan's tables before
// griddepcontrol.wait, so their prologue overlaps that kernel's tail).
cudaError_t launch_fold(const FoldParams& p, uint32_t n_items, bool f16, int variant, cudaStream_t stream,
                        bool early_launch = false);
cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t stream);
// early_launch: as for launch_fold (the step kernel reads only its message
// table before griddepcontrol.wait).
cudaError_t launch_step(const StepParams& p, uint32_t n_xfers, uint64_t max_len, bool f16, cudaStream_t stream,
                        bool early_launch = false);

}  // namespace ddl
