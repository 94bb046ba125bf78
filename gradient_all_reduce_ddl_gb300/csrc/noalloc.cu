// noalloc.cu -- ddl_allreduce_noalloc: the fused all-reduce for callers that
// must not allocate memory.
//
// The fused pass normally reads its work tables (work items, fold-order
// segments, rank orders, an error word) from device memory that a plan
// allocates with cudaMalloc.  Some callers cannot do that: a framework whose
// device memory all belongs to its own pool and that forbids allocations
// outside it, a training loop that must never hit cudaMalloc's implicit
// device synchronisation, or a deployment that fixes its memory footprint at
// start-up and allows no dynamic allocation afterwards.  This entry point has
// the plan code's own table walk (plan.cpp, emit_fused) write the same tables
// into a static host buffer, copies them into a file-scope static device
// array (kScratchBytes, held by every GPU that loads this library until the
// process exits), and launches the same fused kernel on the caller's
// buffers.  It calls no cudaMalloc, cudaFree or other allocating routine,
// and uses no heap memory on the host.
//
// Every call shares the one device array, which keeps the last call's
// tables; each call rewrites the tables it uses and clears the error word.
// Calls whose GPU work overlaps (different streams, or different host
// threads) race on that array and must be ordered by the caller.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "ddl.h"
#include "kernels.h"
#include "plan.h"

namespace {

constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB of tables
constexpr size_t kHeaderBytes = 256;                // error word, then padding
constexpr int kMaxDevices = 64;

static_assert(std::is_same<size_t, uint64_t>::value, "layer sizes are passed through as uint64_t");

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Host staging copy of the tables (no heap); guarded by g_mu together with
// the per-device addresses and the error word read back by ddl_noalloc_check.
alignas(256) static unsigned char g_stage[kScratchBytes];
static void* g_dev_scratch[kMaxDevices];
static uint32_t g_err_host;
static std::mutex g_mu;

// Where the tables sit in the array: the error word, the work items, the
// segments, then P rank bytes per segment (16-byte aligned).
struct Layout {
  uint64_t items_off, segs_off, orders_off, used;
};

Layout layout_of(uint64_t n_items, uint64_t n_segs, int P) {
  Layout l;
  l.items_off = kHeaderBytes;
  l.segs_off = l.items_off + n_items * sizeof(ddl::Item);
  l.orders_off = (l.segs_off + n_segs * sizeof(ddl::Segment) + 15) & ~uint64_t(15);
  l.used = l.orders_off + n_segs * (uint64_t)P;
  return l;
}

// First pass: counts the tables and stops the walk as soon as they no
// longer fit the array.
struct CountSink final : ddl::FusedSink {
  int P;
  uint64_t n_items = 0, n_segs = 0;
  bool fits = true;
  explicit CountSink(int p) : P(p) {}
  bool bucket(uint64_t, uint64_t) override { return true; }
  bool segment(const int*, int, int, int) override {
    ++n_segs;
    return fits = layout_of(n_items, n_segs, P).used <= kScratchBytes;
  }
  bool item(uint64_t, uint32_t) override {
    ++n_items;
    return fits = layout_of(n_items, n_segs, P).used <= kScratchBytes;
  }
};

// Second pass: writes the tables into the host staging buffer.
struct StageSink final : ddl::FusedSink {
  ddl::Item* items;
  ddl::Segment* segs;
  uint8_t* orders;
  uint64_t cap_items, cap_segs;
  uint64_t n_items = 0, n_segs = 0;
  bool bucket(uint64_t, uint64_t) override { return true; }
  bool segment(const int* order, int P, int inner, int groups) override {
    if (n_segs >= cap_segs) return false;
    segs[n_segs].order_off = (uint32_t)(n_segs * (uint64_t)P);
    segs[n_segs].inner = (uint16_t)inner;
    segs[n_segs].groups = (uint16_t)groups;
    for (int t = 0; t < P; ++t) orders[n_segs * (uint64_t)P + t] = (uint8_t)order[t];
    ++n_segs;
    return true;
  }
  bool item(uint64_t begin, uint32_t len) override {
    if (n_items >= cap_items || n_segs == 0) return false;
    items[n_items++] = ddl::Item{begin, len, (uint32_t)(n_segs - 1)};
    return true;
  }
};

ddl_status_t check_rank_bufs(const ddl::Shape& sh, void* const* bufs, int device, bool* aligned) {
  if (!bufs) return DDL_ERR_INVALID_ARG;
  uintptr_t a[ddl::kMaxP];
  bool al = true;
  for (int r = 0; r < sh.P; ++r) {
    if (!bufs[r]) return DDL_ERR_INVALID_ARG;
    a[r] = reinterpret_cast<uintptr_t>(bufs[r]);
    al = al && (a[r] % 16 == 0);
  }
  // insertion sort (P <= 256), then adjacent ranges must not overlap
  for (int i = 1; i < sh.P; ++i)
    for (int j = i; j > 0 && a[j - 1] > a[j]; --j) {
      const uintptr_t t = a[j];
      a[j] = a[j - 1];
      a[j - 1] = t;
    }
  const uint64_t bytes = sh.N * (uint64_t)sh.esize;
  for (int r = 0; r + 1 < sh.P; ++r)
    if (a[r] + bytes > a[r + 1] || a[r] + bytes < a[r]) return DDL_ERR_INVALID_ARG;
  for (int r = 0; r < sh.P; ++r) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, bufs[r]) != cudaSuccess) {
      cudaGetLastError();
      return DDL_ERR_INVALID_ARG;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return DDL_ERR_INVALID_ARG;
    if (at.type == cudaMemoryTypeDevice && at.device != device) return DDL_ERR_INVALID_ARG;
  }
  *aligned = al;
  return DDL_OK;
}

// The array's device address on the current device, looked up once per
// device with that device current (caller holds g_mu).
ddl_status_t scratch_of(int dev, unsigned char** out) {
  if (!g_dev_scratch[dev]) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_scratch);
    if (e != cudaSuccess || !addr) {
      cudaGetLastError();
      return DDL_ERR_CUDA;
    }
    g_dev_scratch[dev] = addr;
  }
  *out = static_cast<unsigned char*>(g_dev_scratch[dev]);
  return DDL_OK;
}

ddl_status_t current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  return DDL_OK;
}

}  // namespace

extern "C" ddl_status_t ddl_allreduce_noalloc(int P, size_t N, ddl_dtype_t dtype, ddl_topology_t topo,
                                              size_t bucket_bytes, int n_tensors, const size_t* numel_fwd_order,
                                              void* const* rank_bufs, float scale, void* stream) {
  // the plan's shape, as ddl_plan_create and ddl_plan_set_layers build it
  if (topo.kind != DDL_RING && topo.kind != DDL_MULTIRING && topo.kind != DDL_TORUS) return DDL_ERR_INVALID_ARG;
  if (n_tensors < 0 || (n_tensors > 0 && !numel_fwd_order)) return DDL_ERR_INVALID_ARG;
  ddl::Shape sh;
  sh.P = P;
  sh.N = N;
  sh.esize = dtype == DDL_FP32 ? 4 : (dtype == DDL_FP16 ? 2 : 0);
  sh.topo = topo.kind;
  sh.k = topo.kind == DDL_MULTIRING ? topo.k : 1;
  sh.X = topo.kind == DDL_TORUS ? topo.X : 0;
  sh.Y = topo.kind == DDL_TORUS ? topo.Y : 0;
  sh.bucket_bytes = bucket_bytes;
  sh.layers = n_tensors > 0 ? numel_fwd_order : nullptr;
  sh.n_layers = (uint64_t)n_tensors;
  sh.mode = ddl::kFused;
  bool unsupported = false;
  if (ddl::check_shape(sh, &unsupported)) return unsupported ? DDL_ERR_UNSUPPORTED : DDL_ERR_INVALID_ARG;
  // N * esize <= 2^40 here
  sh.tile_bytes = ddl::ldg_tile_bytes(sh.N * (uint64_t)sh.esize,
                                      ddl::fused_tile_floor(sh.P, sh.topo, sh.Y, sh.esize, sh.mode));

  // sizes first: a problem whose tables exceed the static array is refused
  // before anything is touched (the count stops at the first table that
  // does not fit)
  CountSink count(P);
  if (!ddl::emit_fused(sh, &count) || !count.fits) return DDL_ERR_UNSUPPORTED;
  const Layout lay = layout_of(count.n_items, count.n_segs, P);

  int dev = -1;
  ddl_status_t st = current_device(&dev);
  if (st != DDL_OK) return st;
  bool aligned = false;
  st = check_rank_bufs(sh, rank_bufs, dev, &aligned);
  if (st != DDL_OK) return st;

  std::lock_guard<std::mutex> lock(g_mu);
  // set-up, once per device, with that device current
  unsigned char* dscr = nullptr;
  st = scratch_of(dev, &dscr);
  if (st != DDL_OK) return st;

  std::memset(g_stage, 0, kHeaderBytes);  // error word starts at zero
  StageSink stage;
  stage.items = reinterpret_cast<ddl::Item*>(g_stage + lay.items_off);
  stage.segs = reinterpret_cast<ddl::Segment*>(g_stage + lay.segs_off);
  stage.orders = g_stage + lay.orders_off;
  stage.cap_items = count.n_items;
  stage.cap_segs = count.n_segs;
  if (!ddl::emit_fused(sh, &stage) || stage.n_items != count.n_items || stage.n_segs != count.n_segs)
    return DDL_ERR_UNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // pageable source: the call returns once the runtime holds its own copy of
  // g_stage, so the next call may overwrite it; the copy into the array is
  // ordered on s before the kernel
  cudaError_t e = cudaMemcpyAsync(dscr, g_stage, lay.used, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  ddl::FoldParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.items = reinterpret_cast<const ddl::Item*>(dscr + lay.items_off);
  fp.segs = reinterpret_cast<const ddl::Segment*>(dscr + lay.segs_off);
  fp.orders = dscr + lay.orders_off;
  fp.err = reinterpret_cast<uint32_t*>(dscr);
  fp.item0 = 0;
  fp.n_segs = (uint32_t)count.n_segs;
  fp.n_orders = (uint32_t)(count.n_segs * (uint64_t)P);
  fp.P = P;
  fp.inner = topo.kind == DDL_TORUS ? topo.X : P;  // the plan's fold shape
  fp.groups = topo.kind == DDL_TORUS ? topo.Y : 1;
  fp.scale = scale;
  fp.round_hops = sh.esize == 2 ? 1 : 0;
  fp.vector_ok = aligned ? 1 : 0;
  fp.n_items = (uint32_t)count.n_items;
  fp.tile_bytes = sh.tile_bytes;
  for (int r = 0; r < P; ++r) fp.bufs[r] = rank_bufs[r];
  e = ddl::launch_fold(fp, (uint32_t)count.n_items, sh.esize == 2, ddl::kVarLdg, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  return DDL_OK;
}

extern "C" ddl_status_t ddl_noalloc_check(void* stream) {
  int dev = -1;
  ddl_status_t st = current_device(&dev);
  if (st != DDL_OK) return st;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_dev_scratch[dev]) return DDL_OK;  // no allocation-free call on this device yet
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  g_err_host = 0;
  cudaError_t e = cudaMemcpyAsync(&g_err_host, g_dev_scratch[dev], sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  if (g_err_host == 0) return DDL_OK;
  e = cudaMemsetAsync(g_dev_scratch[dev], 0, sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  return DDL_ERR_DEVICE_CHECK;
}
