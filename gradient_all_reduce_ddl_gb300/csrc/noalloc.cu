// noalloc.cu -- ddl_allreduce_noalloc: the fused all-reduce for callers that
// must not allocate memory.
//
// The fused pass normally reads its work tables (work items, fold-order
// segments, rank orders, an error word) from device memory that a plan
// allocates with cudaMalloc.  Some callers cannot do that: a framework whose
// device memory all belongs to its own pool and that forbids allocations
// outside it, a training loop that must never hit cudaMalloc's implicit
// device synchronisation, or a deployment that fixes its memory footprint at
// start-up and allows no dynamic allocation afterwards.  This entry point
// builds the same tables in a static host buffer, copies them into a
// file-scope static device array (kScratchBytes, held by every GPU that loads
// this library until the process exits), and launches the same fused kernel
// on the caller's buffers.  It calls no cudaMalloc, cudaFree or other
// allocating routine, and uses no heap memory on the host.
//
// Every call shares the one device array, which keeps the last call's
// tables; each call rewrites the tables it uses and clears the error word.
// Calls whose GPU work overlaps (different streams, or different host
// threads) race on that array and must be ordered by the caller.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "ddl.h"
#include "kernels.h"
#include "plan.h"

namespace {

constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB of tables
constexpr size_t kHeaderBytes = 256;                // error word, then padding
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Host staging copy of the tables (no heap); guarded by g_mu together with
// the per-device addresses.
alignas(256) static unsigned char g_stage[kScratchBytes];
static void* g_dev_scratch[kMaxDevices];
static std::mutex g_mu;

inline uint64_t part_len(uint64_t n, uint64_t m, uint64_t i) { return n / m + (i < n % m ? 1 : 0); }
inline uint64_t part_lo(uint64_t n, uint64_t m, uint64_t i) { return i * (n / m) + (i < n % m ? i : n % m); }

int gcd_int(int a, int b) {
  while (b) {
    const int r = a % b;
    a = b;
    b = r;
  }
  return a;
}

// Writes the tables into three fixed regions, or only counts them when the
// region pointers are null.  Returns false if a region would overflow.
struct Emitter {
  ddl::Item* items;
  ddl::Segment* segs;
  uint8_t* orders;
  uint64_t cap_items, cap_segs, cap_orders;
  uint64_t n_items = 0, n_segs = 0, n_orders = 0;
  uint64_t tile = 0;
  bool ok = true;

  void segment(uint64_t lo, uint64_t len, const int* order, int P, int inner, int groups) {
    if (len == 0 || !ok) return;
    if (n_segs + 1 > cap_segs || n_orders + (uint64_t)P > cap_orders) {
      ok = false;
      return;
    }
    if (segs) {
      segs[n_segs].order_off = (uint32_t)n_orders;
      segs[n_segs].inner = (uint16_t)inner;
      segs[n_segs].groups = (uint16_t)groups;
      for (int t = 0; t < P; ++t) orders[n_orders + t] = (uint8_t)order[t];
    }
    for (uint64_t a = lo, end = lo + len; a < end;) {
      const uint64_t next = (a / tile + 1) * tile < end ? (a / tile + 1) * tile : end;
      if (n_items + 1 > cap_items) {
        ok = false;
        return;
      }
      if (items) items[n_items] = ddl::Item{a, (uint32_t)(next - a), (uint32_t)n_segs};
      ++n_items;
      a = next;
    }
    ++n_segs;
    n_orders += (uint64_t)P;
  }
};

struct Problem {
  int P;
  uint64_t N;
  int esize;
  ddl_topology_t topo;
  uint64_t bucket_bytes;
  int n_tensors;
  const size_t* layers;
  int mult[ddl::kMaxP];  // multi-ring multipliers
};

void emit_bucket(const Problem& pr, uint64_t lo, uint64_t hi, Emitter* em) {
  int order[ddl::kMaxP];
  const int P = pr.P;
  const uint64_t n = hi - lo;
  if (pr.topo.kind == DDL_TORUS) {
    const int X = pr.topo.X, Y = pr.topo.Y;
    for (int c = 0; c < X; ++c) {
      const uint64_t clo = lo + part_lo(n, X, c), cn = part_len(n, X, c);
      for (int d = 0; d < Y; ++d) {
        for (int g = 0; g < Y; ++g)
          for (int h = 0; h < X; ++h) order[g * X + h] = ((d + g) % Y) * X + (c + h) % X;
        em->segment(clo + part_lo(cn, Y, d), part_len(cn, Y, d), order, P, X, Y);
      }
    }
    return;
  }
  const int k = pr.topo.kind == DDL_MULTIRING ? pr.topo.k : 1;
  for (int j = 0; j < k; ++j) {
    const uint64_t slo = lo + part_lo(n, k, j), sn = part_len(n, k, j);
    for (int c = 0; c < P; ++c) {
      for (int t = 0; t < P; ++t) order[t] = (int)((int64_t)((c + t) % P) * pr.mult[j] % P);
      em->segment(slo + part_lo(sn, P, c), part_len(sn, P, c), order, P, P, 1);
    }
  }
}

// Buckets from the highest addresses down, as ddl_plan_create documents.
void emit_all(const Problem& pr, Emitter* em) {
  if (pr.bucket_bytes == 0) {
    emit_bucket(pr, 0, pr.N, em);
    return;
  }
  if (pr.n_tensors == 0) {
    const uint64_t per = pr.bucket_bytes / (uint64_t)pr.esize;
    for (uint64_t hi = pr.N; hi > 0 && em->ok;) {
      const uint64_t lo = hi > per ? hi - per : 0;
      emit_bucket(pr, lo, hi, em);
      hi = lo;
    }
    return;
  }
  uint64_t top = pr.N, cursor = pr.N, bytes = 0;
  for (int i = pr.n_tensors; i-- > 0 && em->ok;) {
    cursor -= pr.layers[i];
    bytes += (uint64_t)pr.layers[i] * (uint64_t)pr.esize;
    if (bytes >= pr.bucket_bytes) {
      emit_bucket(pr, cursor, top, em);
      top = cursor;
      bytes = 0;
    }
  }
  if (top > 0 && em->ok) emit_bucket(pr, 0, top, em);
}

ddl_status_t check_problem(Problem* pr) {
  if (pr->P < 1 || pr->N < 1 || pr->esize == 0) return DDL_ERR_INVALID_ARG;
  if (pr->P > ddl::kMaxP) return DDL_ERR_UNSUPPORTED;
  if (pr->N * (uint64_t)pr->esize > (1ull << 40)) return DDL_ERR_UNSUPPORTED;
  if (pr->bucket_bytes != 0 && pr->bucket_bytes < (uint64_t)pr->esize) return DDL_ERR_INVALID_ARG;
  const ddl_topology_t& t = pr->topo;
  if (t.kind == DDL_TORUS) {
    if (t.X < 1 || t.Y < 1 || (int64_t)t.X * t.Y != pr->P) return DDL_ERR_INVALID_ARG;
  } else if (t.kind == DDL_MULTIRING) {
    if (t.k < 1) return DDL_ERR_INVALID_ARG;
    int found = 0;
    if (pr->P == 1) {
      pr->mult[found++] = 1;
    } else {
      for (int c = 1; c < pr->P && found < t.k; ++c)
        if (gcd_int(c, pr->P) == 1) pr->mult[found++] = c;
    }
    if (found < t.k) return DDL_ERR_UNSUPPORTED;
  } else if (t.kind == DDL_RING) {
    pr->mult[0] = 1;
  } else {
    return DDL_ERR_INVALID_ARG;
  }
  if (pr->n_tensors < 0 || (pr->n_tensors > 0 && !pr->layers)) return DDL_ERR_INVALID_ARG;
  if (pr->n_tensors > 0) {
    uint64_t sum = 0;
    for (int i = 0; i < pr->n_tensors; ++i) {
      if (pr->layers[i] == 0) return DDL_ERR_INVALID_ARG;
      sum += pr->layers[i];
    }
    if (sum != pr->N) return DDL_ERR_INVALID_ARG;
  }
  return DDL_OK;
}

ddl_status_t check_rank_bufs(const Problem& pr, void* const* bufs, int device, bool* aligned) {
  if (!bufs) return DDL_ERR_INVALID_ARG;
  uintptr_t a[ddl::kMaxP];
  bool al = true;
  for (int r = 0; r < pr.P; ++r) {
    if (!bufs[r]) return DDL_ERR_INVALID_ARG;
    a[r] = reinterpret_cast<uintptr_t>(bufs[r]);
    al = al && (a[r] % 16 == 0);
  }
  // insertion sort (P <= 256), then adjacent ranges must not overlap
  for (int i = 1; i < pr.P; ++i)
    for (int j = i; j > 0 && a[j - 1] > a[j]; --j) {
      const uintptr_t t = a[j];
      a[j] = a[j - 1];
      a[j - 1] = t;
    }
  const uint64_t bytes = pr.N * (uint64_t)pr.esize;
  for (int r = 0; r + 1 < pr.P; ++r)
    if (a[r] + bytes > a[r + 1] || a[r] + bytes < a[r]) return DDL_ERR_INVALID_ARG;
  for (int r = 0; r < pr.P; ++r) {
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

}  // namespace

extern "C" ddl_status_t ddl_allreduce_noalloc(int P, size_t N, ddl_dtype_t dtype, ddl_topology_t topo,
                                              size_t bucket_bytes, int n_tensors, const size_t* numel_fwd_order,
                                              void* const* rank_bufs, float scale, void* stream) {
  Problem pr;
  pr.P = P;
  pr.N = N;
  pr.esize = dtype == DDL_FP32 ? 4 : (dtype == DDL_FP16 ? 2 : 0);
  pr.topo = topo;
  pr.bucket_bytes = bucket_bytes;
  pr.n_tensors = n_tensors;
  pr.layers = numel_fwd_order;
  ddl_status_t st = check_problem(&pr);
  if (st != DDL_OK) return st;

  // sizes first: a problem whose tables exceed the static array is refused
  // before anything is touched
  Emitter count{nullptr, nullptr, nullptr, ~0ull, ~0ull, ~0ull};
  count.tile = (uint64_t)ddl::kTileBytes / (uint64_t)pr.esize;
  emit_all(pr, &count);
  const uint64_t items_off = kHeaderBytes;
  const uint64_t segs_off = items_off + count.n_items * sizeof(ddl::Item);
  const uint64_t orders_off = (segs_off + count.n_segs * sizeof(ddl::Segment) + 15) & ~uint64_t(15);
  const uint64_t used = orders_off + count.n_orders;
  if (used > kScratchBytes || count.n_items > 0xFFFFFFFFull) return DDL_ERR_UNSUPPORTED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  bool aligned = false;
  st = check_rank_bufs(pr, rank_bufs, dev, &aligned);
  if (st != DDL_OK) return st;

  std::lock_guard<std::mutex> lock(g_mu);
  // set-up, once per device, with that device current
  if (!g_dev_scratch[dev]) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_scratch);
    if (e != cudaSuccess || !addr) {
      cudaGetLastError();
      return DDL_ERR_CUDA;
    }
    g_dev_scratch[dev] = addr;
  }
  unsigned char* dscr = static_cast<unsigned char*>(g_dev_scratch[dev]);

  std::memset(g_stage, 0, kHeaderBytes);  // error word starts at zero
  Emitter em{reinterpret_cast<ddl::Item*>(g_stage + items_off), reinterpret_cast<ddl::Segment*>(g_stage + segs_off),
             g_stage + orders_off, count.n_items, count.n_segs, count.n_orders};
  em.tile = count.tile;
  emit_all(pr, &em);
  if (!em.ok) return DDL_ERR_UNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // pageable source: the call returns once g_stage has been consumed
  cudaError_t e = cudaMemcpyAsync(dscr, g_stage, used, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  ddl::FoldParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.items = reinterpret_cast<const ddl::Item*>(dscr + items_off);
  fp.segs = reinterpret_cast<const ddl::Segment*>(dscr + segs_off);
  fp.orders = dscr + orders_off;
  fp.err = reinterpret_cast<uint32_t*>(dscr);
  fp.item0 = 0;
  fp.n_segs = (uint32_t)em.n_segs;
  fp.n_orders = (uint32_t)em.n_orders;
  fp.P = P;
  fp.inner = topo.kind == DDL_TORUS ? topo.X : P;  // the plan's fold shape
  fp.groups = topo.kind == DDL_TORUS ? topo.Y : 1;
  fp.scale = scale;
  fp.round_hops = pr.esize == 2 ? 1 : 0;
  fp.vector_ok = aligned ? 1 : 0;
  for (int r = 0; r < P; ++r) fp.bufs[r] = rank_bufs[r];
  e = ddl::launch_fold(fp, (uint32_t)em.n_items, pr.esize == 2, ddl::kVarLdg, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DDL_ERR_CUDA;
  }
  return DDL_OK;
}
