// ddl_api.cu -- the C ABI declared in include/ddl.h.
//
// A plan holds the host tables (plan.cpp), their device copies, the side
// stream and the per-bucket events.  Every entry point validates its
// arguments before queueing anything, maps CUDA failures to DDL_ERR_CUDA, and
// never throws across the ABI.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "ddl.h"
#include "kernels.h"
#include "plan.h"

struct ddl_plan {
  ddl::Spec spec;
  ddl::Tables tab;
  int kernel = DDL_KERNEL_AUTO;
  // device side
  int device = -1;
  bool dev_current = false;  // device tables match tab
  ddl::Item* d_items = nullptr;
  ddl::Segment* d_segs = nullptr;
  uint8_t* d_orders = nullptr;
  ddl::Xfer* d_xfers = nullptr;
  uint32_t* d_err = nullptr;
  cudaStream_t side = nullptr;
  std::vector<cudaEvent_t> ev_ready;
  cudaEvent_t ev_done = nullptr;
  uint64_t launches = 0;
  // overlap with back-propagation
  bool ov_active = false;
  std::vector<void*> ov_bufs;
  float ov_scale = 1.f;
  std::vector<char> ov_issued;
  // last rank-pointer set that passed the device-pointer check
  std::vector<void*> checked;
  bool checked_aligned = false;
  // last parameter / momentum pointer set that passed the checks
  std::vector<void*> checked_sgd;
  bool checked_sgd_aligned = false;
  // host-buffer pipeline: copy-in, compute and copy-out streams, events
  cudaStream_t hs[3] = {nullptr, nullptr, nullptr};
  std::vector<cudaEvent_t> hev;
  // the zero-copy pass's own work items (staged-size tiles), built on first use
  ddl_plan* zc = nullptr;
};

namespace {

using ddl::Spec;

void drop_zero_copy(ddl_plan* p);

ddl_status_t rebuild(ddl_plan* p) {
  drop_zero_copy(p);
  ddl::Tables t;
  if (!ddl::build_tables(p->spec, p->spec.mode == ddl::kStepwise, &t)) return DDL_ERR_OOM;
  if (t.items.size() > 0xFFFFFFFFull || t.xfers.size() > 0xFFFFFFFFull) return DDL_ERR_UNSUPPORTED;
  p->tab = std::move(t);
  p->dev_current = false;
  return DDL_OK;
}

void free_device_tables(ddl_plan* p) {
  cudaFree(p->d_items);
  cudaFree(p->d_segs);
  cudaFree(p->d_orders);
  cudaFree(p->d_xfers);
  p->d_items = nullptr;
  p->d_segs = nullptr;
  p->d_orders = nullptr;
  p->d_xfers = nullptr;
}

// The zero-copy helper shares its parent's device and error word; it owns
// only its tables and per-bucket events.
void drop_zero_copy(ddl_plan* p) {
  ddl_plan* z = p->zc;
  if (!z) return;
  p->zc = nullptr;
  free_device_tables(z);
  for (cudaEvent_t ev : z->ev_ready) cudaEventDestroy(ev);
  delete z;
}

// Host-side fault injection for the failure tests: with the environment
// variable DDL_INJECT_ALLOC_FAILURE=1, uploading a plan's tables fails as if
// the device were out of memory (no GPU call is made for it).
bool alloc_failure_injected() {
  const char* v = std::getenv("DDL_INJECT_ALLOC_FAILURE");
  return v && v[0] == '1' && v[1] == '\0';
}

template <typename T>
cudaError_t upload(T** dst, const std::vector<T>& v) {
  if (v.empty()) return cudaSuccess;
  if (alloc_failure_injected()) return cudaErrorMemoryAllocation;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dst), v.size() * sizeof(T));
  if (e != cudaSuccess) return e;
  return cudaMemcpy(*dst, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice);
}

ddl_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DDL_OK;
  cudaGetLastError();  // clear a non-sticky error so later calls start clean
  return e == cudaErrorMemoryAllocation ? DDL_ERR_OOM : DDL_ERR_CUDA;
}

// The plan's two-level fold shape: ring, multi-ring and rank order fold one
// group of P; the torus folds Y groups of X.
void fold_shape(const Spec& s, int32_t* inner, int32_t* groups) {
  if (s.mode != ddl::kRankOrder && s.topo == ddl::kTorus) {
    *inner = s.X;
    *groups = s.Y;
  } else if (s.mode != ddl::kRankOrder && s.topo == ddl::kTorusND) {
    *inner = s.dims[0];
    *groups = s.P / s.dims[0];
  } else {
    *inner = s.P;
    *groups = 1;
  }
}

// n-D torus plans fold through the level cascade (nlev > 0); others use the
// two-level shape.
void set_levels(const ddl_plan* p, ddl::FoldParams* fp) {
  fold_shape(p->spec, &fp->inner, &fp->groups);
  if (p->spec.topo != ddl::kTorusND || p->spec.mode == ddl::kRankOrder) return;
  fp->nlev = (int32_t)p->spec.dims.size();
  fp->top = -1;
  for (int l = 0; l < fp->nlev; ++l) {
    fp->lev[l] = (uint16_t)p->spec.dims[l];
    if (p->spec.dims[l] > 1) fp->top = l;
  }
}

// Work-item size for the plan's kernel: the n-D pass covers 8 KB (fp32) or
// 4 KB (fp16) per rank per CTA; the staged passes fill ~64 KB per stage.
uint32_t choose_tile(const Spec& s, int kernel) {
  const uint32_t ldg =
      ddl::ldg_tile_bytes(s.N * (uint64_t)s.esize, ddl::fused_tile_floor(s.P, s.topo, s.Y, s.esize, s.mode));
  if (s.topo == ddl::kTorusND) {
    // the n-D pass's columns per thread: two, except fp16 without rounded hops
    const uint32_t cap = (s.esize == 2 && s.mode != ddl::kFused) ? 4096u : 8192u;
    return ldg < cap ? ldg : cap;
  }
  if (kernel == DDL_KERNEL_BULK_LOAD) return ddl::bulk_tile_bytes(s.P);
  return ldg;
}

// Binds the plan to the current device and makes its device tables current.
ddl_status_t ensure_device(ddl_plan* p) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (p->device >= 0 && p->device != dev) return DDL_ERR_INVALID_ARG;
  if (p->device < 0) {
    p->device = dev;
    e = cudaMalloc(reinterpret_cast<void**>(&p->d_err), sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->ev_done, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (!p->dev_current) {
    free_device_tables(p);
    e = upload(&p->d_items, p->tab.items);
    if (e == cudaSuccess) e = upload(&p->d_segs, p->tab.segs);
    if (e == cudaSuccess) e = upload(&p->d_orders, p->tab.orders);
    if (e == cudaSuccess) e = upload(&p->d_xfers, p->tab.xfers);
    if (e != cudaSuccess) {
      free_device_tables(p);
      return cuda_status(e);
    }
    const size_t nb = p->tab.buckets.size();
    while (p->ev_ready.size() < nb) {
      cudaEvent_t ev;
      e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_status(e);
      p->ev_ready.push_back(ev);
    }
    p->dev_current = true;
  }
  return DDL_OK;
}

// Checks the P rank pointers: non-null, distinct, non-overlapping, and (once
// per new pointer set) device-accessible memory.  *aligned = all 16-byte aligned.
ddl_status_t check_bufs(ddl_plan* p, void* const* bufs, bool device_check, bool* aligned) {
  if (!bufs) return DDL_ERR_INVALID_ARG;
  const int P = p->spec.P;
  const uint64_t bytes = p->spec.N * (uint64_t)p->spec.esize;
  std::vector<uintptr_t> a(P);
  bool al = true;
  for (int r = 0; r < P; ++r) {
    if (!bufs[r]) return DDL_ERR_INVALID_ARG;
    a[r] = reinterpret_cast<uintptr_t>(bufs[r]);
    al = al && (a[r] % 16 == 0);
  }
  std::sort(a.begin(), a.end());
  for (int r = 0; r + 1 < P; ++r)
    if (a[r] + bytes > a[r + 1] || a[r] + bytes < a[r]) return DDL_ERR_INVALID_ARG;
  *aligned = al;
  if (!device_check) return DDL_OK;
  if (p->checked.size() == (size_t)P && std::equal(p->checked.begin(), p->checked.end(), bufs)) return DDL_OK;
  for (int r = 0; r < P; ++r) {
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, bufs[r]);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return DDL_ERR_INVALID_ARG;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return DDL_ERR_INVALID_ARG;
    if (at.type == cudaMemoryTypeDevice && at.device != p->device) return DDL_ERR_INVALID_ARG;
  }
  p->checked.assign(bufs, bufs + P);
  return DDL_OK;
}

// The launch record of the fused pass over items [ia, ib), and the variant it
// runs (the plan's kernel choice, or force_variant; the staged passes need
// 16-byte aligned buffers, else the register pass runs its element-wise path,
// with the same results).
int fold_params(const ddl_plan* p, uint32_t ia, uint32_t ib, void* const* bufs, bool aligned, float scale,
                int force_variant, ddl::FoldParams* fp) {
  const bool f16 = p->spec.esize == 2;
  std::memset(fp, 0, sizeof(*fp));
  fp->items = p->d_items;
  fp->segs = p->d_segs;
  fp->orders = p->d_orders;
  fp->err = p->d_err;
  fp->item0 = ia;
  fp->n_segs = (uint32_t)p->tab.segs.size();
  fp->n_orders = (uint32_t)p->tab.orders.size();
  fp->P = p->spec.P;
  fp->scale = scale;
  fp->round_hops = (f16 && p->spec.mode == ddl::kFused) ? 1 : 0;
  fp->vector_ok = aligned ? 1 : 0;
  for (int r = 0; r < p->spec.P; ++r) fp->bufs[r] = bufs ? bufs[r] : nullptr;
  fp->n_items = ib - ia;
  fp->tile_bytes = p->spec.tile_bytes;
  set_levels(p, fp);
  int variant = ddl::kVarLdg;
  if (aligned && p->kernel == DDL_KERNEL_BULK_LOAD) variant = ddl::kVarBulkLoad;
  if (aligned && p->kernel == DDL_KERNEL_CHUNKED) variant = ddl::kVarChunked;
  if (aligned && force_variant) variant = force_variant;
  return variant;
}

// Fused pass over items [ia, ib): a whole bucket, or a tile-aligned element range of one.
// early: launch as a programmatic dependent of the kernel before it on s (only
// where nothing but that kernel orders the launch: no event waits, no copies).
ddl_status_t run_items(ddl_plan* p, uint32_t ia, uint32_t ib, void* const* bufs, bool aligned, float scale,
                       cudaStream_t s, bool early = false, int force_variant = 0) {
  if (ib <= ia) return DDL_OK;
  ddl::FoldParams fp;
  const int variant = fold_params(p, ia, ib, bufs, aligned, scale, force_variant, &fp);
  const cudaError_t e = ddl::launch_fold(fp, ib - ia, p->spec.esize == 2, variant, s, early);
  if (e != cudaSuccess) return cuda_status(e);
  ++p->launches;
  return DDL_OK;
}

// An NVTX range per bucket, so a timeline shows which bucket each launch
// reduced (costs nothing measurable without a tool attached).
struct BucketRange {
  BucketRange(int b, const ddl::Bucket& bk) {
    char name[96];
    std::snprintf(name, sizeof(name), "ddl bucket %d [%llu, %llu)", b, (unsigned long long)bk.lo,
                  (unsigned long long)bk.hi);
    nvtxRangePushA(name);
  }
  ~BucketRange() { nvtxRangePop(); }
};

ddl_status_t run_bucket(ddl_plan* p, int b, void* const* bufs, bool aligned, float scale, cudaStream_t s,
                        bool early = false, int force_variant = 0) {
  const ddl::Bucket& bk = p->tab.buckets[b];
  const BucketRange range(b, bk);
  const bool f16 = p->spec.esize == 2;
  if (p->spec.mode == ddl::kStepwise) {
    ddl::StepParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.xfers = p->d_xfers;
    sp.err = p->d_err;
    sp.P = p->spec.P;
    sp.scale = scale;
    sp.vector_ok = aligned ? 1 : 0;
    for (int r = 0; r < p->spec.P; ++r) sp.bufs[r] = bufs[r];
    for (uint32_t st = bk.step_begin; st < bk.step_end; ++st) {
      const ddl::Step& step = p->tab.steps[st];
      sp.xfer0 = step.xfer_begin;
      // every step after the first follows this bucket's previous step on s
      const cudaError_t e =
          ddl::launch_step(sp, step.xfer_end - step.xfer_begin, step.max_len, f16, s, early || st > bk.step_begin);
      if (e != cudaSuccess) return cuda_status(e);
      ++p->launches;
    }
    return DDL_OK;
  }
  return run_items(p, bk.item_begin, bk.item_end, bufs, aligned, scale, s, early, force_variant);
}

// First item of bucket b that starts at or after element x.
uint32_t item_at(const ddl_plan* p, const ddl::Bucket& bk, uint64_t x) {
  auto first = p->tab.items.begin() + bk.item_begin, last = p->tab.items.begin() + bk.item_end;
  return (uint32_t)(std::lower_bound(first, last, x,
                                     [](const ddl::Item& it, uint64_t v) { return it.begin < v; }) -
                    p->tab.items.begin());
}

ddl_status_t prepare(ddl_plan* p, void* const* bufs, bool* aligned) {
  if (!p || !bufs) return DDL_ERR_INVALID_ARG;
  // repeated call with the pointer set that passed every check last time
  if (p->dev_current && p->checked.size() == (size_t)p->spec.P &&
      std::memcmp(p->checked.data(), bufs, sizeof(void*) * (size_t)p->spec.P) == 0) {
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev == p->device) {
      *aligned = p->checked_aligned;
      return DDL_OK;
    }
  }
  bool al = false;
  ddl_status_t st = check_bufs(p, bufs, false, &al);
  if (st != DDL_OK) return st;
  st = ensure_device(p);
  if (st != DDL_OK) return st;
  st = check_bufs(p, bufs, true, &al);
  if (st != DDL_OK) return st;
  *aligned = al;
  p->checked_aligned = al;
  return DDL_OK;
}

}  // namespace

extern "C" {

ddl_status_t ddl_plan_create(int P, size_t N, ddl_dtype_t dtype, ddl_topology_t topo, size_t bucket_bytes,
                             ddl_plan_t* out) {
  if (!out) return DDL_ERR_INVALID_ARG;
  *out = nullptr;
  Spec s;
  s.P = P;
  s.N = N;
  s.esize = dtype == DDL_FP16 ? 2 : (dtype == DDL_FP32 ? 4 : 0);
  s.topo = topo.kind;
  s.k = topo.kind == DDL_MULTIRING ? topo.k : 1;
  s.X = topo.kind == DDL_TORUS ? topo.X : 0;
  s.Y = topo.kind == DDL_TORUS ? topo.Y : 0;
  s.bucket_bytes = bucket_bytes;
  s.tile_bytes = choose_tile(s, DDL_KERNEL_AUTO);
  bool unsupported = false;
  const std::string why = ddl::validate(s, &unsupported);
  if (!why.empty()) return unsupported ? DDL_ERR_UNSUPPORTED : DDL_ERR_INVALID_ARG;
  ddl_plan* p = new (std::nothrow) ddl_plan();
  if (!p) return DDL_ERR_OOM;
  p->spec = s;
  const ddl_status_t st = rebuild(p);
  if (st != DDL_OK) {
    delete p;
    return st;
  }
  *out = p;
  return DDL_OK;
}

ddl_status_t ddl_plan_set_layers(ddl_plan_t p, int n_tensors, const size_t* numel) {
  if (!p || n_tensors < 0 || (n_tensors > 0 && !numel) || p->ov_active) return DDL_ERR_INVALID_ARG;
  Spec s = p->spec;
  s.layers.assign(numel, numel + n_tensors);
  bool unsupported = false;
  const std::string why = ddl::validate(s, &unsupported);
  if (!why.empty()) return unsupported ? DDL_ERR_UNSUPPORTED : DDL_ERR_INVALID_ARG;
  const Spec old = p->spec;
  p->spec = s;
  const ddl_status_t st = rebuild(p);
  if (st != DDL_OK) p->spec = old;
  return st;
}

ddl_status_t ddl_plan_set_mode(ddl_plan_t p, ddl_mode_t mode) {
  if (!p || p->ov_active || mode < DDL_MODE_FUSED || mode > DDL_MODE_RANKORDER) return DDL_ERR_INVALID_ARG;
  if ((int)mode == p->spec.mode) return DDL_OK;
  const Spec old = p->spec;
  p->spec.mode = (int)mode;
  p->spec.tile_bytes = choose_tile(p->spec, p->kernel);  // the floor follows the fold shape
  const ddl_status_t st = rebuild(p);
  if (st != DDL_OK) {
    p->spec = old;
    rebuild(p);
  }
  return st;
}

ddl_status_t ddl_plan_set_torus_dims(ddl_plan_t p, int ndims, const int* dims) {
  if (!p || p->ov_active || ndims < 1 || ndims > ddl::kMaxDims || !dims) return DDL_ERR_INVALID_ARG;
  Spec s = p->spec;
  s.topo = ddl::kTorusND;
  s.dims.assign(dims, dims + ndims);
  while (s.dims.size() > 1 && s.dims.back() == 1) s.dims.pop_back();  // no steps along them
  s.k = 1;
  s.X = s.Y = 0;
  s.tile_bytes = choose_tile(s, p->kernel);
  bool unsupported = false;
  const std::string why = ddl::validate(s, &unsupported);
  if (!why.empty()) return unsupported ? DDL_ERR_UNSUPPORTED : DDL_ERR_INVALID_ARG;
  const Spec old = p->spec;
  p->spec = s;
  const ddl_status_t st = rebuild(p);
  if (st != DDL_OK) {
    p->spec = old;
    rebuild(p);
  }
  return st;
}

ddl_status_t ddl_plan_set_kernel(ddl_plan_t p, ddl_kernel_t k) {
  if (!p || p->ov_active) return DDL_ERR_INVALID_ARG;
  if (k != DDL_KERNEL_AUTO && k != DDL_KERNEL_LDG && k != DDL_KERNEL_BULK_LOAD && k != DDL_KERNEL_CHUNKED)
    return DDL_ERR_INVALID_ARG;
  const uint32_t tile = choose_tile(p->spec, (int)k);
  if (tile != p->spec.tile_bytes) {
    const Spec old = p->spec;
    p->spec.tile_bytes = tile;
    const ddl_status_t st = rebuild(p);
    if (st != DDL_OK) {
      p->spec = old;
      rebuild(p);
      return st;
    }
  }
  p->kernel = (int)k;
  return DDL_OK;
}

ddl_status_t ddl_allreduce(ddl_plan_t p, void* const* bufs, float scale, void* stream) {
  bool aligned = false;
  ddl_status_t st = prepare(p, bufs, &aligned);
  if (st != DDL_OK) return st;
  if (p->ov_active) return DDL_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->spec.mode != ddl::kStepwise && p->tab.buckets.size() > 1) {
    // every bucket back to back: one launch over all work items (stored
    // bucket by bucket, so bucket 0's CTAs still start first)
    nvtxRangePushA("ddl all buckets");
    st = run_items(p, 0, (uint32_t)p->tab.items.size(), bufs, aligned, scale, s, true);
    nvtxRangePop();
    return st;
  }
  for (int b = 0; b < (int)p->tab.buckets.size(); ++b) {
    st = run_bucket(p, b, bufs, aligned, scale, s, true);
    if (st != DDL_OK) return st;
  }
  return DDL_OK;
}

ddl_status_t ddl_allreduce_sgd(ddl_plan_t p, void* const* grad_bufs, float* const* param_bufs, float* const* mom_bufs,
                               float scale, float lr, float momentum, float weight_decay, int keep_grads,
                               void* stream) {
  if (!p || !param_bufs) return DDL_ERR_INVALID_ARG;
  if (p->spec.mode == ddl::kStepwise || p->spec.topo == ddl::kTorusND || p->spec.P > ddl::kMaxPSgd)
    return DDL_ERR_UNSUPPORTED;
  if (!mom_bufs && momentum != 0.0f) return DDL_ERR_INVALID_ARG;
  if (p->ov_active) return DDL_ERR_INVALID_ARG;
  const int P = p->spec.P;
  bool aligned = false;
  ddl_status_t st = prepare(p, grad_bufs, &aligned);
  if (st != DDL_OK) return st;
  // parameters and momenta: distinct binary32 device arrays that overlap
  // neither each other nor the gradients (the check is cached per full set)
  std::vector<void*> cur(grad_bufs, grad_bufs + P);
  cur.insert(cur.end(), param_bufs, param_bufs + P);
  if (mom_bufs) cur.insert(cur.end(), mom_bufs, mom_bufs + P);
  if (p->checked_sgd != cur) {
    const uint64_t gbytes = p->spec.N * (uint64_t)p->spec.esize, fbytes = p->spec.N * 4ull;
    std::vector<std::pair<uintptr_t, uint64_t>> all;
    for (int r = 0; r < P; ++r) all.push_back({reinterpret_cast<uintptr_t>(grad_bufs[r]), gbytes});
    bool al = true;
    for (size_t i = (size_t)P; i < cur.size(); ++i) {
      void* q = cur[i];
      if (!q) return DDL_ERR_INVALID_ARG;
      all.push_back({reinterpret_cast<uintptr_t>(q), fbytes});
      al = al && (reinterpret_cast<uintptr_t>(q) % 16 == 0);
      cudaPointerAttributes at;
      if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
        cudaGetLastError();
        return DDL_ERR_INVALID_ARG;
      }
      if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return DDL_ERR_INVALID_ARG;
    }
    std::sort(all.begin(), all.end());
    for (size_t i = 0; i + 1 < all.size(); ++i)
      if (all[i].first + all[i].second > all[i + 1].first) return DDL_ERR_INVALID_ARG;
    p->checked_sgd = cur;
    p->checked_sgd_aligned = al;
  }
  ddl::SgdParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.items = p->d_items;
  sp.segs = p->d_segs;
  sp.orders = p->d_orders;
  sp.err = p->d_err;
  sp.n_segs = (uint32_t)p->tab.segs.size();
  sp.n_orders = (uint32_t)p->tab.orders.size();
  sp.P = P;
  fold_shape(p->spec, &sp.inner, &sp.groups);
  sp.scale = scale;
  sp.lr = lr;
  sp.mu = momentum;
  sp.wd = weight_decay;
  sp.round_hops = (p->spec.esize == 2 && p->spec.mode == ddl::kFused) ? 1 : 0;
  sp.vector_ok = (aligned && p->checked_sgd_aligned) ? 1 : 0;
  sp.keep_grads = keep_grads ? 1 : 0;
  sp.has_mom = mom_bufs ? 1 : 0;
  sp.tile_bytes = p->spec.tile_bytes;
  for (int r = 0; r < P; ++r) {
    sp.grads[r] = grad_bufs[r];
    sp.params[r] = param_bufs[r];
    sp.moms[r] = mom_bufs ? mom_bufs[r] : nullptr;
  }
  // every bucket in one launch (items are stored bucket by bucket)
  sp.item0 = 0;
  const cudaError_t e =
      ddl::launch_sgd(sp, (uint32_t)p->tab.items.size(), p->spec.esize == 2, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  ++p->launches;
  return DDL_OK;
}

ddl_status_t ddl_allreduce_slab(ddl_plan_t p, void* base, size_t stride, float scale, void* stream) {
  if (!p || !base || p->ov_active) return DDL_ERR_INVALID_ARG;
  const int P = p->spec.P;
  const uint64_t row = p->spec.N * (uint64_t)p->spec.esize;
  if (P > 1 && stride < row) return DDL_ERR_INVALID_ARG;
  std::vector<void*> bufs(P);
  for (int r = 0; r < P; ++r) bufs[r] = static_cast<char*>(base) + (size_t)r * stride;
  return ddl_allreduce(p, bufs.data(), scale, stream);
}

ddl_status_t ddl_allreduce_bucket(ddl_plan_t p, int bucket, void* const* bufs, float scale, void* stream) {
  if (!p || bucket < 0 || bucket >= (int)p->tab.buckets.size()) return DDL_ERR_INVALID_ARG;
  bool aligned = false;
  const ddl_status_t st = prepare(p, bufs, &aligned);
  if (st != DDL_OK) return st;
  return run_bucket(p, bucket, bufs, aligned, scale, static_cast<cudaStream_t>(stream));
}

// Zero-copy form: the fused pass works on host buffers that the GPU can
// reach directly (page-locked, managed, or pageable where the system gives
// the GPU coherent access to it).
// The zero-copy pass's plan: the same schedule with staged-size work items
// for the bulk-load pass, built on the first zero-copy call; it shares the
// parent's device and error word.
static ddl_status_t zero_copy_plan(ddl_plan* p, ddl_plan** out) {
  if (!p->zc) {
    ddl_plan* z = new (std::nothrow) ddl_plan;
    if (!z) return DDL_ERR_OOM;
    z->spec = p->spec;
    z->spec.tile_bytes = choose_tile(p->spec, DDL_KERNEL_BULK_LOAD);
    z->kernel = DDL_KERNEL_BULK_LOAD;
    z->device = p->device;
    z->d_err = p->d_err;
    p->zc = z;
    ddl_status_t st = rebuild(z);
    if (st == DDL_OK) st = ensure_device(z);
    if (st != DDL_OK) {
      drop_zero_copy(p);
      return st;
    }
  }
  *out = p->zc;
  return DDL_OK;
}

static ddl_status_t allreduce_in_host_memory(ddl_plan* p, void* const* host_bufs, float scale, cudaStream_t s) {
  bool al = false;
  ddl_status_t st = check_bufs(p, host_bufs, false, &al);
  if (st != DDL_OK) return st;
  st = ensure_device(p);
  if (st != DDL_OK) return st;
  int pageable = 0;
  cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, p->device);
  bool locked = true;  // every buffer page-locked (mapped like device memory)
  for (int r = 0; r < p->spec.P; ++r) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, host_bufs[r]) != cudaSuccess) {
      cudaGetLastError();
      return DDL_ERR_INVALID_ARG;
    }
    const bool reach = at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged ||
                       (at.type == cudaMemoryTypeUnregistered && pageable);
    if (!reach) return DDL_ERR_INVALID_ARG;
    locked = locked && at.type == cudaMemoryTypeHost;
  }
  if (p->spec.mode == ddl::kStepwise) return DDL_ERR_UNSUPPORTED;
  // With the default kernel choice, aligned page-locked buffers take the
  // bulk-load pass: its cp.async.bulk copies of whole tiles move more over the
  // host link than the register pass's 16-byte loads.  (Up to P = 64, where
  // its shared-memory ring still holds 1 KB per rank; the n-D torus keeps its
  // cascade pass; managed and pageable memory keep the register pass.)
  if (al && locked && p->kernel == DDL_KERNEL_AUTO && p->spec.mode == ddl::kFused &&
      p->spec.topo != ddl::kTorusND && p->spec.P <= 64) {
    ddl_plan* z = nullptr;
    st = zero_copy_plan(p, &z);
    if (st != DDL_OK) return st;
    const uint64_t before = z->launches;
    for (int b = 0; b < (int)z->tab.buckets.size() && st == DDL_OK; ++b) st = run_bucket(z, b, host_bufs, al, scale, s);
    p->launches += z->launches - before;
    return st;
  }
  for (int b = 0; b < (int)p->tab.buckets.size(); ++b) {
    st = run_bucket(p, b, host_bufs, al, scale, s);
    if (st != DDL_OK) return st;
  }
  return DDL_OK;
}

ddl_status_t ddl_allreduce_host(ddl_plan_t p, void* const* host_bufs, void* const* dev_bufs, float scale,
                                void* stream) {
  if (!p || !host_bufs) return DDL_ERR_INVALID_ARG;
  for (int r = 0; r < p->spec.P; ++r)
    if (!host_bufs[r]) return DDL_ERR_INVALID_ARG;
  if (p->ov_active) return DDL_ERR_INVALID_ARG;
  if (!dev_bufs) return allreduce_in_host_memory(p, host_bufs, scale, static_cast<cudaStream_t>(stream));
  bool aligned = false;
  ddl_status_t st = prepare(p, dev_bufs, &aligned);
  if (st != DDL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t es = (size_t)p->spec.esize;
  const int P = p->spec.P;
  auto copy_all = [&](uint64_t lo, uint64_t hi, cudaMemcpyKind kind, cudaStream_t cs) -> cudaError_t {
    for (int r = 0; r < P; ++r) {
      char* h = static_cast<char*>(host_bufs[r]) + lo * es;
      char* d = static_cast<char*>(dev_bufs[r]) + lo * es;
      const cudaError_t e = kind == cudaMemcpyHostToDevice ? cudaMemcpyAsync(d, h, (hi - lo) * es, kind, cs)
                                                           : cudaMemcpyAsync(h, d, (hi - lo) * es, kind, cs);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  };
  if (p->spec.mode == ddl::kStepwise) {
    // whole buckets move through the steps: copy in, reduce, copy out
    cudaError_t e = copy_all(0, p->spec.N, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e);
    for (int b = 0; b < (int)p->tab.buckets.size(); ++b) {
      st = run_bucket(p, b, dev_bufs, aligned, scale, s);
      if (st != DDL_OK) return st;
    }
    e = copy_all(0, p->spec.N, cudaMemcpyDeviceToHost, s);
    return cuda_status(e);
  }
  // Every output element depends only on the same element of every rank, so
  // the copy-in, the fused pass and the copy-out pipeline over element ranges
  // (tile-aligned, so each range is a run of whole work items) on three
  // streams: copy-in of range i+1 and copy-out of range i-1 overlap the pass
  // over range i, and the two copy directions overlap each other.
  // Eight ranges: more of them queue more copies than the streams retire in
  // step (32 ranges of the 4x4 ResNet-50 gradient took 13.6 ms, 8 took 11.6).
#ifndef DDL_HOST_RANGES
#define DDL_HOST_RANGES 8
#endif
  constexpr int kMaxRanges = DDL_HOST_RANGES;
  const uint64_t tile = (uint64_t)p->spec.tile_bytes / es;
  uint64_t R = (p->spec.N + kMaxRanges - 1) / kMaxRanges;
  R = ((R + tile - 1) / tile) * tile;
  const uint64_t min_r = ((uint64_t)(1u << 20) / es + tile - 1) / tile * tile;  // >= 1 MiB per rank
  if (R < min_r) R = min_r;
  cudaError_t e = cudaSuccess;
  if (!p->hs[0])
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&p->hs[i], cudaStreamNonBlocking);
  const size_t need = 1 + 3 * (size_t)(kMaxRanges + p->tab.buckets.size());
  while (e == cudaSuccess && p->hev.size() < need) {
    cudaEvent_t ev;
    e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e == cudaSuccess) p->hev.push_back(ev);
  }
  if (e != cudaSuccess) return cuda_status(e);
  cudaStream_t sin = p->hs[0], scomp = p->hs[1], sout = p->hs[2];
  size_t evi = 0;
  cudaEvent_t start = p->hev[evi++];
  e = cudaEventRecord(start, s);
  for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(p->hs[i], start, 0);
  if (e != cudaSuccess) return cuda_status(e);
  // buckets run from the highest addresses down; ranges ascend inside each
  for (int b = 0; b < (int)p->tab.buckets.size(); ++b) {
    const ddl::Bucket& bk = p->tab.buckets[b];
    for (uint64_t lo = bk.lo; lo < bk.hi;) {
      uint64_t hi = (lo / R + 1) * R;
      if (hi > bk.hi) hi = bk.hi;
      cudaEvent_t ein = p->hev[evi++], ecomp = p->hev[evi++];
      e = copy_all(lo, hi, cudaMemcpyHostToDevice, sin);
      if (e == cudaSuccess) e = cudaEventRecord(ein, sin);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(scomp, ein, 0);
      if (e != cudaSuccess) return cuda_status(e);
      st = run_items(p, item_at(p, bk, lo), item_at(p, bk, hi), dev_bufs, aligned, scale, scomp);
      if (st != DDL_OK) return st;
      e = cudaEventRecord(ecomp, scomp);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(sout, ecomp, 0);
      if (e == cudaSuccess) e = copy_all(lo, hi, cudaMemcpyDeviceToHost, sout);
      if (e != cudaSuccess) return cuda_status(e);
      lo = hi;
    }
  }
  cudaEvent_t done = p->hev[evi++];
  e = cudaEventRecord(done, sout);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, done, 0);
  return cuda_status(e);
}

ddl_status_t ddl_overlap_begin(ddl_plan_t p, void* const* bufs, float scale, void* stream) {
  (void)stream;
  bool aligned = false;
  if (p && p->ov_active) return DDL_ERR_INVALID_ARG;
  const ddl_status_t st = prepare(p, bufs, &aligned);
  if (st != DDL_OK) return st;
  p->ov_bufs.assign(bufs, bufs + p->spec.P);
  p->ov_scale = scale;
  p->ov_issued.assign(p->tab.buckets.size(), 0);
  p->ov_active = true;
  return DDL_OK;
}

ddl_status_t ddl_bucket_ready(ddl_plan_t p, int bucket, void* stream) {
  if (!p || !p->ov_active || bucket < 0 || bucket >= (int)p->tab.buckets.size() || p->ov_issued[bucket])
    return DDL_ERR_INVALID_ARG;
  bool aligned = false;
  ddl_status_t st = prepare(p, p->ov_bufs.data(), &aligned);
  if (st != DDL_OK) return st;
  cudaError_t e = cudaEventRecord(p->ev_ready[bucket], static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->side, p->ev_ready[bucket], 0);
  if (e != cudaSuccess) return cuda_status(e);
  p->ov_issued[bucket] = 1;
  // With the library's kernel choice and full-size (8 KB) work items the side
  // stream runs the rank-chunked staged pass: a persistent grid of two CTAs
  // per SM that streams the bucket's work items, instead of one CTA per item.
  // Sharing the GPU with the producer's kernels, it measured faster than the
  // register pass (ResNet-101 multi-ring, 7 buckets: 9.24 ms overlapped
  // against 9.47 ms sequential, where the register pass took 10.08 ms).
  // Smaller items (small buckets) take the library's own pass choice: the
  // staged pass's persistent grid and pipeline cost several microseconds per
  // bucket there (4x4 torus, 8 buckets of 32 KB per rank: 54.5 against the
  // plain all-reduce's 3.7 us).  Same results either way.
  const bool staged = p->kernel == DDL_KERNEL_AUTO && p->spec.topo != ddl::kTorusND &&
                      p->spec.tile_bytes == (uint32_t)ddl::kTileBytes;
  return run_bucket(p, bucket, p->ov_bufs.data(), aligned, p->ov_scale, p->side, false,
                    staged ? ddl::kVarChunked : 0);
}

ddl_status_t ddl_overlap_end(ddl_plan_t p, void* stream) {
  if (!p || !p->ov_active) return DDL_ERR_INVALID_ARG;
  p->ov_active = false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaEventRecord(p->ev_done, p->side);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p->ev_done, 0);
  if (e != cudaSuccess) return cuda_status(e);
  // buckets never signalled: all-reduced here, on `stream`, after everything
  // queued on it so far (one launch over each run of consecutive buckets)
  bool aligned = false;
  ddl_status_t st = prepare(p, p->ov_bufs.data(), &aligned);
  if (st != DDL_OK) return st;
  const int nb = (int)p->tab.buckets.size();
  for (int b = 0; b < nb;) {
    if (p->ov_issued[b]) {
      ++b;
      continue;
    }
    int c = b;
    while (c < nb && !p->ov_issued[c]) ++c;
    if (p->spec.mode == ddl::kStepwise) {
      for (int q = b; q < c && st == DDL_OK; ++q) st = run_bucket(p, q, p->ov_bufs.data(), aligned, p->ov_scale, s);
    } else {
      st = run_items(p, p->tab.buckets[b].item_begin, p->tab.buckets[c - 1].item_end, p->ov_bufs.data(), aligned,
                     p->ov_scale, s);
    }
    if (st != DDL_OK) return st;
    b = c;
  }
  return DDL_OK;
}

ddl_status_t ddl_plan_num_buckets(ddl_plan_t p, int* n) {
  if (!p || !n) return DDL_ERR_INVALID_ARG;
  *n = (int)p->tab.buckets.size();
  return DDL_OK;
}

ddl_status_t ddl_plan_bucket_range(ddl_plan_t p, int b, size_t* begin, size_t* end) {
  if (!p || !begin || !end || b < 0 || b >= (int)p->tab.buckets.size()) return DDL_ERR_INVALID_ARG;
  *begin = p->tab.buckets[b].lo;
  *end = p->tab.buckets[b].hi;
  return DDL_OK;
}

ddl_status_t ddl_plan_traffic(ddl_plan_t p, uint64_t* moved, uint64_t* steps) {
  if (!p || !moved || !steps) return DDL_ERR_INVALID_ARG;
  *moved = p->tab.moved;
  *steps = p->tab.nsteps;
  return DDL_OK;
}

ddl_status_t ddl_plan_cost(ddl_plan_t p, double alpha_s, double beta_s_per_byte, int links_per_worker,
                           double* seconds) {
  if (!p || !seconds || !(alpha_s >= 0.0) || !(beta_s_per_byte >= 0.0) || links_per_worker < 1)
    return DDL_ERR_INVALID_ARG;
  // the step tables of the schedule, whatever the plan's own mode
  ddl::Spec s = p->spec;
  s.mode = ddl::kStepwise;
  return ddl::schedule_cost(s, alpha_s, beta_s_per_byte, links_per_worker, seconds) ? DDL_OK : DDL_ERR_OOM;
}

ddl_status_t ddl_plan_fold_order(ddl_plan_t p, size_t i, int32_t* order, int32_t* inner, int32_t* groups) {
  if (!p || !order || !inner || !groups) return DDL_ERR_INVALID_ARG;
  if (p->spec.mode == ddl::kStepwise) return DDL_ERR_UNSUPPORTED;
  return ddl::fold_order_of(p->spec, p->tab, i, order, inner, groups) ? DDL_OK : DDL_ERR_INVALID_ARG;
}

ddl_status_t ddl_plan_launches(ddl_plan_t p, uint64_t* n) {
  if (!p || !n) return DDL_ERR_INVALID_ARG;
  *n = p->launches;
  return DDL_OK;
}

ddl_status_t ddl_plan_kernel_name(ddl_plan_t p, const char** name) {
  if (!p || !name) return DDL_ERR_INVALID_ARG;
  if (p->spec.mode == ddl::kStepwise) {
    *name = "step_kernel";
    return DDL_OK;
  }
  // the launch ddl_allreduce makes: one over all of the plan's work items
  const uint32_t n = (uint32_t)p->tab.items.size();
  ddl::FoldParams fp;
  const int variant = fold_params(p, 0, n, nullptr, true, 1.0f, 0, &fp);
  *name = ddl::fold_pass_kernel(ddl::fold_pass(fp, n, p->spec.esize == 2, variant), fp.round_hops != 0);
  return DDL_OK;
}

ddl_status_t ddl_plan_check(ddl_plan_t p) {
  if (!p) return DDL_ERR_INVALID_ARG;
  if (p->device < 0) return DDL_OK;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e);
  uint32_t w = 0;
  e = cudaMemcpy(&w, p->d_err, sizeof(w), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  if (w == 0) return DDL_OK;
  cudaMemset(p->d_err, 0, sizeof(uint32_t));
  return DDL_ERR_DEVICE_CHECK;
}

ddl_status_t ddl_selftest_wait_timeout(ddl_plan_t p, uint32_t limit_us, void* stream) {
  if (!p || limit_us == 0 || limit_us > 1000000) return DDL_ERR_INVALID_ARG;
  const ddl_status_t st = ensure_device(p);
  if (st != DDL_OK) return st;
  const cudaError_t e =
      ddl::launch_wait_timeout_selftest(p->d_err, (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

const char* ddl_status_string(ddl_status_t s) {
  switch (s) {
    case DDL_OK: return "DDL_OK";
    case DDL_ERR_INVALID_ARG: return "DDL_ERR_INVALID_ARG: invalid argument";
    case DDL_ERR_UNSUPPORTED: return "DDL_ERR_UNSUPPORTED: request outside what the library builds";
    case DDL_ERR_OOM: return "DDL_ERR_OOM: allocation failed";
    case DDL_ERR_CUDA: return "DDL_ERR_CUDA: a CUDA call or kernel launch failed";
    case DDL_ERR_DEVICE_CHECK: return "DDL_ERR_DEVICE_CHECK: a kernel's own check failed";
  }
  return "unknown ddl_status_t";
}

ddl_status_t ddl_plan_destroy(ddl_plan_t p) {
  if (!p) return DDL_OK;
  if (p->device >= 0) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    if (p->side) cudaStreamSynchronize(p->side);
    drop_zero_copy(p);
    free_device_tables(p);
    cudaFree(p->d_err);
    for (int i = 0; i < 3; ++i)
      if (p->hs[i]) {
        cudaStreamSynchronize(p->hs[i]);
        cudaStreamDestroy(p->hs[i]);
      }
    for (cudaEvent_t ev : p->hev) cudaEventDestroy(ev);
    for (cudaEvent_t ev : p->ev_ready) cudaEventDestroy(ev);
    if (p->ev_done) cudaEventDestroy(p->ev_done);
    if (p->side) cudaStreamDestroy(p->side);
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
  }
  delete p;
  return DDL_OK;
}

}  // extern "C"
