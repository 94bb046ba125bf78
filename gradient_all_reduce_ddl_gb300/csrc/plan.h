// plan.h -- host-side tables of an all-reduce plan, and the records the
// kernels read.  Host code only builds them; no CUDA calls here.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

namespace ddl {

constexpr int kMaxP = 256;          // rank orders are stored as bytes
#ifndef DDL_TILE_BYTES
#define DDL_TILE_BYTES 8192
#endif
constexpr int kTileBytes = DDL_TILE_BYTES;  // bytes per rank in one fused work item (<= 8192)

// One contiguous run of elements whose fold order is the same.  The ranks are
// added in the order orders[order_off .. order_off+P), as `groups` groups of
// `inner` consecutive ranks: each group is left-folded, then the group totals
// are left-folded.  Ring and multi-ring: groups = 1.  Torus: inner = X
// (a row, from column c on), groups = Y (rows from row d on).
struct Segment {
  uint32_t order_off;
  uint16_t inner;
  uint16_t groups;
};

// One CTA's work in the fused pass: elements [begin, begin + len) of segment
// `seg`.  Items never cross a segment edge or a kTileBytes-aligned boundary.
struct Item {
  uint64_t begin;
  uint32_t len;
  uint32_t seg;
};

// One message of one communication step (stepwise mode).
enum XferOp : uint32_t {
  kAddHop = 0,    // dst += src; the result travels again (rounded to storage)
  kAddFinal = 1,  // dst = (src + dst) * scale; the owner's last add
  kCopy = 2,      // dst = src (all-gather)
  kScaleOnly = 3  // dst = dst * scale (a ring of one: the owner has no add)
};

struct Xfer {
  uint64_t lo;
  uint64_t len;
  uint16_t src;
  uint16_t dst;
  uint32_t op;
};

struct Step {
  uint32_t xfer_begin, xfer_end;
  uint64_t max_len;
};

struct Bucket {
  uint64_t lo, hi;
  uint32_t item_begin, item_end;  // fused / rank-order items
  uint32_t step_begin, step_end;  // stepwise steps
};

enum Topo : int32_t { kRing = 0, kMultiRing = 1, kTorus = 2, kTorusND = 3 };
constexpr int kMaxDims = 4;  // n-D torus: dims 0 (fastest in the rank number) .. 3
enum Mode : int32_t { kFused = 0, kStepwise = 1, kRankOrder = 2 };

struct Spec {
  int P = 0;
  uint64_t N = 0;
  int esize = 4;      // 4 (binary32) or 2 (binary16)
  int topo = kRing;
  int k = 1, X = 0, Y = 0;
  uint64_t bucket_bytes = 0;
  std::vector<uint64_t> layers;
  int mode = kFused;
  uint32_t tile_bytes = kTileBytes;  // bytes per rank in one work item
  std::vector<int> dims;             // n-D torus sizes (trailing 1s dropped)
};

// Work-item size of the shared-memory-staged pass: P ranks' tiles of one
// pipeline stage fill about 64 KB, between 256 B and kTileBytes per rank.
uint32_t bulk_tile_bytes(int P);

// Plans of at least this many ranks fold small buffers in the latency pass
// (all P ranks' columns of a work item staged in shared memory at once).
#ifndef DDL_LAT_MIN_P
#define DDL_LAT_MIN_P 16
#endif
constexpr int kLatMinP = DDL_LAT_MIN_P;
// With binary16 storage and rounded hops the register pass's per-rank chain
// is longer, and the latency pass already wins from 8 ranks (P = 8 fp16 torus
// at 16,384 elements: 2.80 against 2.25 us per all-reduce in graph replay;
// at 262,144: 6.32 against 3.51 us).
constexpr int kLatMinPHops = 8;

// Work-item size of the register, small-item and latency passes: kTileBytes,
// or smaller, down to `floor` bytes, when a rank's buffer is too small to give
// every SM of a large GPU (2 x 152 items) work at that size.
uint32_t ldg_tile_bytes(uint64_t bytes_per_rank, uint32_t floor);

// That floor for a plan: 256 bytes where small buffers take the latency pass
// (P >= kLatMinP, or P >= kLatMinPHops with binary16 hops on a two-level
// fold) or the small-item pass (a single fold group with no
// intermediate rounding: rank order, and the binary32 ring, multi-ring and
// one-row torus), whose time falls with the bytes one CTA stages; 1 KB where
// they take the register pass, whose fixed costs per CTA then dominate.
// Y: the torus's rows (ignored for other schedules).
uint32_t fused_tile_floor(int P, int topo, int Y, int esize, int mode);

struct Tables {
  std::vector<Bucket> buckets;
  std::vector<Segment> segs;
  std::vector<uint8_t> orders;
  std::vector<Item> items;
  std::vector<Xfer> xfers;
  std::vector<Step> steps;
  uint64_t moved = 0;   // elements sent over all messages
  uint64_t nsteps = 0;  // sequential communication steps
};

// What fixes the fused tables, as plain values that own no memory (the
// allocation-free entry point builds one without touching the heap).
struct Shape {
  int P = 0;
  uint64_t N = 0;
  int esize = 4;
  int topo = kRing;
  int k = 1, X = 0, Y = 0;
  uint64_t bucket_bytes = 0;
  const uint64_t* layers = nullptr;  // tensor sizes in forward order, or null
  uint64_t n_layers = 0;
  int mode = kFused;
  uint32_t tile_bytes = kTileBytes;
  int ndims = 0;
  int dims[kMaxDims] = {0, 0, 0, 0};
};

Shape shape_of(const Spec& s);

// Receives the fused (or rank-order) tables in table order: for every bucket
// (highest addresses first) its segments, and after each segment its work
// items.  A false return stops the walk.
struct FusedSink {
  virtual bool bucket(uint64_t lo, uint64_t hi) = 0;
  virtual bool segment(const int* order, int P, int inner, int groups) = 0;
  virtual bool item(uint64_t begin, uint32_t len) = 0;
  virtual bool bucket_end() { return true; }

 protected:
  ~FusedSink() = default;
};

// Walks the fused tables of s into the sink; uses no heap memory.  Returns
// false if the sink stopped the walk.  Items never cross a segment edge or a
// tile_bytes-aligned boundary.
bool emit_fused(const Shape& s, FusedSink* sink);

// nullptr if the shape is valid, else a static reason.  *unsupported is set
// when the request is valid in principle but outside what this library
// builds.  Uses no heap memory.
const char* check_shape(const Shape& s, bool* unsupported);

// Returns "" if the spec is valid, else a reason (check_shape on the spec).
std::string validate(const Spec& s, bool* unsupported);

// The multi-ring multipliers s_0..s_{k-1} (the j-th smallest integers in
// [1, P) coprime to P; s_0 = 1 when P = 1) into out[0..k-1]; false if fewer
// than k exist.  No heap memory.
bool ring_multipliers_into(int P, int k, int* out);
bool ring_multipliers(int P, int k, std::vector<int>* out);

// Builds buckets, the fused (or rank-order) segment and item tables, and the
// step/message tables (steps only listed when with_steps).  Returns false on
// allocation failure.
bool build_tables(const Spec& s, bool with_steps, Tables* t);

// alpha-beta time of the schedule on P workers with `links` network links
// each: every step costs alpha plus beta times the bytes of the busiest
// (worker, link) pair, the message of concurrent ring j going on link
// j mod links.  False on allocation failure.
bool schedule_cost(const Spec& s, double alpha, double beta, int links, double* seconds);

// Fold order of element i from the built tables.
bool fold_order_of(const Spec& s, const Tables& t, uint64_t i, int32_t* order, int32_t* inner, int32_t* groups);

}  // namespace ddl
