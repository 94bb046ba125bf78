// fold_kernels.cu -- the fused all-reduce pass.
//
// One CTA takes one work item: a run of elements that all share one fold
// order (one chunk of one bucket; for the torus one sub-chunk of one row
// chunk).  Each thread owns whole 16-byte columns: it loads the column from
// all P ranks, adds them in the schedule's order in registers, multiplies by
// the scale once, and stores the result to all P ranks.  That is the whole
// reduce-scatter + scale + all-gather of a chunk (ring: Baidu write-up,
// "总结"; torus: Sony page, "2D-Torus All-reduce"; fp16 hops: Sony page,
// "训练设置") in one read and one write of every rank element.
//
// The order of the adds is exactly the step-by-step schedule's: groups of
// `inner` ranks are left-folded, then the group totals are left-folded.  With
// binary16 storage every intermediate result is rounded to binary16 (it would
// travel on the next hop) except the very last add, which stays binary32, is
// scaled, and is rounded once.  Adds and the multiply use the _rn intrinsics
// so the compiler cannot contract or reorder them.
#include <cuda_fp16.h>

#include "kernels.h"

namespace ddl {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float round_h(float x) { return __half2float(__float2half_rn(x)); }

// 16 bytes -> binary32 lanes (4 for fp32, 8 for fp16; widening is exact)
template <bool F16>
__device__ __forceinline__ void unpack(const uint4 r, float* f) {
  if constexpr (F16) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xFFFFu)));
      f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
    }
  } else {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
}

template <bool F16>
__device__ __forceinline__ uint4 pack(const float* f) {
  uint4 r;
  if constexpr (F16) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __half_as_ushort(__float2half_rn(f[2 * i]));
      const uint32_t hi = __half_as_ushort(__float2half_rn(f[2 * i + 1]));
      w[i] = lo | (hi << 16);
    }
    r = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    r = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
  return r;
}

// Uniform control of fold position t (same for every lane of the CTA).
struct Ctl {
  bool group_start;  // first rank of a group: the group value starts here
  bool group_end;    // last rank of a group: fold the group total into the outer value
  bool first_group;
  bool round_in;     // round the inner add's result to binary16
  bool round_out;    // round the outer add's result to binary16
};

__device__ __forceinline__ Ctl ctl_at(int t, int h, int g, int inner, int groups, int P, bool rh) {
  Ctl c;
  const bool last = (t == P - 1);
  c.group_start = (h == 0);
  c.group_end = (h == inner - 1);
  c.first_group = (g == 0);
  c.round_in = rh && !(last && groups == 1);
  c.round_out = rh && !last;
  return c;
}

template <int NL>
__device__ __forceinline__ void fold_lanes(float* in, float* out, const float* v, const Ctl& c) {
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    float a = v[l];
    if (!c.group_start) {
      a = __fadd_rn(in[l], a);
      if (c.round_in) a = round_h(a);
    }
    in[l] = a;
    if (c.group_end) {
      float o = a;
      if (!c.first_group) {
        o = __fadd_rn(out[l], a);
        if (c.round_out) o = round_h(o);
      }
      out[l] = o;
    }
  }
}

template <bool F16>
__device__ __forceinline__ float load_elem(const char* base, uint64_t e) {
  if constexpr (F16) {
    return __half2float(__ushort_as_half(__ldcs(reinterpret_cast<const unsigned short*>(base) + e)));
  } else {
    return __ldcs(reinterpret_cast<const float*>(base) + e);
  }
}

template <bool F16>
__device__ __forceinline__ void store_elem(char* base, uint64_t e, float v) {
  if constexpr (F16) {
    __stcs(reinterpret_cast<unsigned short*>(base) + e, __half_as_ushort(__float2half_rn(v)));
  } else {
    __stcs(reinterpret_cast<float*>(base) + e, v);
  }
}

// Element-wise path: segment edges that cut a 16-byte column, and buffers
// that are not 16-byte aligned.
template <bool F16>
__device__ void fold_scalar(char* const* ptr, uint64_t e, int P, int inner, int groups, bool rh, float scale) {
  float in = 0.f, out = 0.f;
  int h = 0, g = 0;
  for (int t = 0; t < P; ++t) {
    const float v = load_elem<F16>(ptr[t], e);
    const Ctl c = ctl_at(t, h, g, inner, groups, P, rh);
    fold_lanes<1>(&in, &out, &v, c);
    if (++h == inner) {
      h = 0;
      ++g;
    }
  }
  const float r = __fmul_rn(out, scale);
  for (int t = 0; t < P; ++t) store_elem<F16>(ptr[t], e, r);
}

// Prologue shared by the fused kernels: fetch the item, check it, and lay out
// the rank pointers in fold order in shared memory.  Returns false if the
// item is unusable (the error word is then set).
__device__ __forceinline__ bool load_item(const FoldParams& p, char** s_ptr, Item* s_item, Segment* s_seg,
                                          int* s_ok) {
  if (threadIdx.x == 0) {
    const Item it = p.items[p.item0 + blockIdx.x];
    int ok = it.seg < p.n_segs;
    Segment sg{0, 1, 1};
    if (ok) {
      sg = p.segs[it.seg];
      ok = (int)sg.inner * (int)sg.groups == p.P && sg.order_off + (uint32_t)p.P <= p.n_orders;
      if (!ok) atomicOr(p.err, kErrBadOrder);
    } else {
      atomicOr(p.err, kErrBadItem);
    }
    *s_item = it;
    *s_seg = sg;
    *s_ok = ok;
  }
  __syncthreads();
  if (!*s_ok) return false;
  for (int t = threadIdx.x; t < p.P; t += blockDim.x) {
    const unsigned r = p.orders[s_seg->order_off + t];
    s_ptr[t] = static_cast<char*>(p.bufs[r < (unsigned)p.P ? r : 0]);
  }
  __syncthreads();
  return true;
}

// ---------------------------------------------------------------------------
// Variant 1: register pass.  V columns per thread, B ranks' loads in flight.
// ---------------------------------------------------------------------------
template <bool F16, int V, int B>
__global__ void __launch_bounds__(kThreads, 2) fold_ldg_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = F16 ? 8 : 4;  // elements per 16-byte column
  __shared__ char* s_ptr[kMaxP];
  __shared__ Item s_item;
  __shared__ Segment s_seg;
  __shared__ int s_ok;
  if (!load_item(p, s_ptr, &s_item, &s_seg, &s_ok)) return;

  const int P = p.P, inner = s_seg.inner, groups = s_seg.groups;
  const bool rh = F16 && p.round_hops;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;

  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads)
      fold_scalar<F16>(s_ptr, e, P, inner, groups, rh, p.scale);
    return;
  }

  uint64_t col[V];
  bool live[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    col[u] = vb + threadIdx.x + (uint64_t)u * kThreads;
    live[u] = col[u] < ve;
  }
  float in[V][L], out[V][L];
  int h = 0, g = 0;
  for (int t0 = 0; t0 < P; t0 += B) {
    uint4 raw[B][V];
#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (t0 + j < P) {
        const uint4* base = reinterpret_cast<const uint4*>(s_ptr[t0 + j]);
#pragma unroll
        for (int u = 0; u < V; ++u) raw[j][u] = live[u] ? __ldcs(base + col[u]) : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (t0 + j < P) {
        const Ctl c = ctl_at(t0 + j, h, g, inner, groups, P, rh);
#pragma unroll
        for (int u = 0; u < V; ++u) {
          float f[L];
          unpack<F16>(raw[j][u], f);
          fold_lanes<L>(in[u], out[u], f, c);
        }
        if (++h == inner) {
          h = 0;
          ++g;
        }
      }
    }
  }
  uint4 res[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    float r[L];
#pragma unroll
    for (int l = 0; l < L; ++l) r[l] = __fmul_rn(out[u][l], p.scale);
    res[u] = pack<F16>(r);
  }
  for (int t = 0; t < P; ++t) {
    uint4* base = reinterpret_cast<uint4*>(s_ptr[t]);
#pragma unroll
    for (int u = 0; u < V; ++u)
      if (live[u]) __stcs(base + col[u], res[u]);
  }
  // the few elements of a cut column at either end of the item
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    fold_scalar<F16>(s_ptr, e, P, inner, groups, rh, p.scale);
  }
}

template <bool F16>
cudaError_t launch_ldg(const FoldParams& p, uint32_t n_items, cudaStream_t stream) {
  fold_ldg_kernel<F16, 2, 8><<<n_items, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fold(const FoldParams& p, uint32_t n_items, bool f16, int variant, cudaStream_t stream) {
  if (n_items == 0) return cudaSuccess;
  (void)variant;
  return f16 ? launch_ldg<true>(p, n_items, stream) : launch_ldg<false>(p, n_items, stream);
}

}  // namespace ddl
