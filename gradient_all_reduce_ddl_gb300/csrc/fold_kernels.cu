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

#include <atomic>
#include <type_traits>

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

// Packed binary16 hop adds.  For binary16 a and b, fl16(fl32(a + b)) equals
// the correctly rounded fl16(a + b): binary32 carries 24 >= 2*11 + 2
// significand bits, the bound under which double rounding of a sum is
// innocuous (S. A. Figueroa, "When is double rounding innocuous?", SIGNUM
// Newsletter 30(3), 1995), and every binary16 sum is inside binary32's
// exponent range.  So a hop add whose result is rounded to binary16 is one
// add.rn.f16x2 per two lanes, bit for bit the same as widen + add + round.
__device__ __forceinline__ uint32_t hadd2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One fold position that is not the last (every add rounded to binary16), on
// a 16-byte column of binary16 pairs.
__device__ __forceinline__ void fold_h2(uint32_t* in, uint32_t* out, const uint4 v, const Ctl& c) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t a = w[i];
    if (!c.group_start) a = hadd2_rn(in[i], a);
    in[i] = a;
    if (c.group_end) out[i] = c.first_group ? a : hadd2_rn(out[i], a);
  }
}

__device__ __forceinline__ void widen_h2(const uint32_t* h, float* f) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __half2float(__ushort_as_half((unsigned short)(h[i] & 0xFFFFu)));
    f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(h[i] >> 16)));
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

// The element-wise fold at element e: rank position t's buffer is at(t).  Its
// loads go out eight positions at a time, so an element costs P/8 dependent
// round trips rather than P (the fold, its order and its roundings are those
// of the column passes).  Returns the folded value before the scale.
template <bool F16, class At>
__device__ __forceinline__ float fold_elem(At at, uint64_t e, int P, int inner, int groups, bool rh) {
  float in = 0.f, out = 0.f;
  int h = 0, g = 0;
  for (int t0 = 0; t0 < P; t0 += 8) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (t0 + j < P) v[j] = load_elem<F16>(at(t0 + j), e);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (t0 + j < P) {
        const Ctl c = ctl_at(t0 + j, h, g, inner, groups, P, rh);
        fold_lanes<1>(&in, &out, &v[j], c);
        if (++h == inner) {
          h = 0;
          ++g;
        }
      }
    }
  }
  return out;
}

// Element-wise path: segment edges that cut a 16-byte column, and buffers
// that are not 16-byte aligned.  Kept out of line: inlined, its batched loads
// took registers from the column passes around it and slowed their small
// buffers (P = 16 ring at 16K elements 2.45 against 2.26 us per all-reduce).
template <bool F16>
__device__ __noinline__ void fold_scalar(char* const* ptr, uint64_t e, int P, int inner, int groups, bool rh,
                                         float scale) {
  const float r = __fmul_rn(fold_elem<F16>([ptr](int t) { return ptr[t]; }, e, P, inner, groups, rh), scale);
  for (int t = 0; t < P; ++t) store_elem<F16>(ptr[t], e, r);
}

// Programmatic dependent launch.  The register passes let the next kernel on
// the stream start as soon as all of their CTAs are running, and wait for the
// kernel before them (completed, its writes visible) only after reading the
// plan's tables, which no kernel writes.  Both are no-ops in a launch that
// did not ask for it.
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Prologue shared by the fused kernels: every thread reads the item (one
// broadcast load), P threads read its rank order and lay the rank pointers out
// in fold order in shared memory; one barrier.  Returns false (after setting
// the error word) if the item points outside the tables.
__device__ __forceinline__ bool load_item(const FoldParams& p, char** s_ptr, Item* item) {
  *item = p.items[p.item0 + blockIdx.x];
  const uint64_t off = (uint64_t)item->seg * (uint64_t)p.P;
  const bool ok = item->seg < p.n_segs && off + (uint64_t)p.P <= p.n_orders;
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadItem);
    return false;
  }
  for (int t = threadIdx.x; t < p.P; t += blockDim.x) {
    const unsigned r = p.orders[off + t];
    s_ptr[t] = static_cast<char*>(p.bufs[r < (unsigned)p.P ? r : 0]);
  }
  __syncthreads();
  return true;
}

// ---------------------------------------------------------------------------
// The register pass.  V columns per thread, B ranks' loads in flight,
// sized for MINB CTAs per SM.  V * kThreads columns must cover the largest
// item (V * 4 KB per rank); the launcher picks V from the plan's item size.
// ---------------------------------------------------------------------------
#ifndef DDL_LDG_F32_B
#define DDL_LDG_F32_B 8
#endif
#ifndef DDL_LDG_F16_B
#define DDL_LDG_F16_B 8
#endif
#ifndef DDL_LDG_MINB
#define DDL_LDG_MINB 2
#endif

// H2: binary16 with rounded hops; every position but the last folds packed
// pairs (fold_h2), the last one widens and takes its final add in binary32.
template <bool F16, bool H2, int V, int B, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) fold_ldg_kernel(const __grid_constant__ FoldParams p) {
  static_assert(F16 || !H2, "packed hops are binary16 only");
  constexpr int L = F16 ? 8 : 4;  // elements per 16-byte column
  __shared__ char* s_ptr[kMaxP];
  Item s_item;
  griddep_launch_dependents();
  if (!load_item(p, s_ptr, &s_item)) return;
  griddep_wait();

  const int P = p.P, inner = p.inner, groups = p.groups;
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
  uint32_t hin[V][4] = {}, hout[V][4] = {};  // packed accumulators (H2)
  uint4 xl[V];  // the last position's values (H2: folded after the loop)
  Ctl cl = {};
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
        if constexpr (H2) {
          if (t0 + j < P - 1) {
#pragma unroll
            for (int u = 0; u < V; ++u) fold_h2(hin[u], hout[u], raw[j][u], c);
          } else {
#pragma unroll
            for (int u = 0; u < V; ++u) xl[u] = raw[j][u];
            cl = c;
          }
        } else {
#pragma unroll
          for (int u = 0; u < V; ++u) {
            float f[L];
            unpack<F16>(raw[j][u], f);
            fold_lanes<L>(in[u], out[u], f, c);
          }
        }
        if (++h == inner) {
          h = 0;
          ++g;
        }
      }
    }
  }
  if constexpr (H2) {  // the last position: widen, its final add stays binary32
#pragma unroll
    for (int u = 0; u < V; ++u) {
      widen_h2(hin[u], in[u]);
      widen_h2(hout[u], out[u]);
      float f[L];
      unpack<F16>(xl[u], f);
      fold_lanes<L>(in[u], out[u], f, cl);
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

// ---------------------------------------------------------------------------
// Small-item pass: small buffers (items of at most 4 KB per rank) whose fold
// is one group with no intermediate rounding -- the binary32 ring and
// multi-ring, and every rank-order plan.  The fold is then the plain left fold
// x_0 + x_1 + ... + x_{P-1} in the item's order, so each thread takes one
// 16-byte column and adds the ranks one by one as it loads them.  Such
// buffers are latency-bound (a few warps per SM, nothing to hide instruction
// latency behind), and this is the shortest chain of dependent instructions
// from the loads to the stores: the 2 MB ring takes 1.64 us per all-reduce in
// graph replay here against 1.84 us in the general register pass, whose
// per-position fold logic (groups, hop rounding) sits on that chain.
// ---------------------------------------------------------------------------
template <bool F16>
__global__ void __launch_bounds__(kThreads) fold_small_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = F16 ? 8 : 4;  // elements per 16-byte column
  __shared__ char* s_ptr[kMaxP];
  Item s_item;
  griddep_launch_dependents();
  if (!load_item(p, s_ptr, &s_item)) return;
  griddep_wait();

  const int P = p.P;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;
  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads)
      fold_scalar<F16>(s_ptr, e, P, P, 1, false, p.scale);
    return;
  }
  const uint64_t c = vb + threadIdx.x;
  if (c < ve) {
    // ranks in batches of four: a batch's loads are all issued before its
    // adds (a rank-by-rank loop, load then add, measured 2.25 us here)
    float acc[L];
    uint4 raw[4];
    for (int t0 = 0; t0 < P; t0 += 4) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (t0 + j < P) raw[j] = __ldcs(reinterpret_cast<const uint4*>(s_ptr[t0 + j]) + c);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (t0 + j < P) {
          float f[L];
          unpack<F16>(raw[j], f);
#pragma unroll
          for (int l = 0; l < L; ++l) acc[l] = (t0 + j == 0) ? f[l] : __fadd_rn(acc[l], f[l]);
        }
      }
    }
#pragma unroll
    for (int l = 0; l < L; ++l) acc[l] = __fmul_rn(acc[l], p.scale);
    const uint4 res = pack<F16>(acc);
    for (int t = 0; t < P; ++t) __stcs(reinterpret_cast<uint4*>(s_ptr[t]) + c, res);
  }
  // the few elements of a cut column at either end of the item
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    fold_scalar<F16>(s_ptr, e, P, P, 1, false, p.scale);
  }
}

// ---------------------------------------------------------------------------
// Latency pass: small items of two-level folds (ring, multi-ring, 2D torus;
// any dtype and rounding) whose P tiles fit in shared memory.  The register
// pass folds P ranks in batches of 8, one global round trip per batch, which
// dominates when a buffer is too small to keep the GPU busy.  Here the CTA
// loads all P ranks' columns of its item into shared memory at once (one
// round trip, every thread issuing loads), folds each row group of the
// schedule in parallel (thread per group and column), folds the group totals
// (thread per column), and stores the result to every rank from shared
// memory, all threads at once.  The adds, their order and their roundings are
// exactly those of the register pass: a group is the left fold of its inner
// ranks, each add rounded to binary16 where a hop would carry it; the group
// totals are left-folded, every add rounded but the final one.  A single
// group (SINGLE: the ring and multi-ring folds, and rank order) has no totals
// to fold: its fold, scaled, is the result, one barrier earlier (per
// all-reduce in graph replay, P = 64 multi-ring at 4K / 16K elements per rank:
// 3.07 / 4.51 us, against 3.28 / 4.72 us through the totals phase).
// Shared memory: P x tile bytes of data (fold position t at t * tile), then
// the binary32 group totals, then one 16-byte result per column.  The totals
// are 16-byte slices of 4 lanes: slice q of group g sits in row g * L/4 + q,
// one 16-byte column per thread, so a warp's threads touch consecutive 16
// bytes.  Stored one binary32 lane at a time, L lanes apart, they conflicted
// 4- to 8-way in the shared-memory banks (8x4 fp16 torus at 4K / 16K / 64K
// elements: 3.29 / 5.33 / 5.75 us then, 3.08 / 4.73 / 5.21 us now).
// ---------------------------------------------------------------------------
__host__ __device__ constexpr uint32_t lat_smem_bytes(uint32_t P, uint32_t groups, uint32_t tile, uint32_t lanes) {
  return P * tile + groups * (tile / 16u) * lanes * 4u + (tile / 16u) * 16u;
}

template <bool F16, bool SINGLE>
__global__ void __launch_bounds__(kThreads) fold_lat_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = F16 ? 8 : 4;  // elements per 16-byte column
  extern __shared__ __align__(16) unsigned char s_lat[];
  __shared__ char* s_ptr[kMaxP];
  Item s_item;
  griddep_launch_dependents();
  if (!load_item(p, s_ptr, &s_item)) return;
  griddep_wait();

  const int P = p.P, inner = p.inner, groups = p.groups;
  const bool rh = F16 && p.round_hops;
  const uint32_t T = p.tile_bytes;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;
  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads)
      fold_scalar<F16>(s_ptr, e, P, inner, groups, rh, p.scale);
    return;
  }
  const uint32_t ncols = (uint32_t)(ve - vb);  // <= T / 16
  // the group totals' 4-lane slices: row g * L/4 + q, CT columns per row
  const uint32_t CT = T / 16u;
  float4* s_tot = reinterpret_cast<float4*>(s_lat + (size_t)P * T);
  uint4* s_res = reinterpret_cast<uint4*>(s_lat + (size_t)P * T + (size_t)groups * CT * L * 4u);

  // every fold position's columns, all loads in flight together
  for (uint32_t i = threadIdx.x; i < (uint32_t)P * ncols; i += kThreads) {
    const uint32_t t = i / ncols, c = i % ncols;
    *reinterpret_cast<uint4*>(s_lat + (size_t)t * T + c * 16u) =
        __ldcs(reinterpret_cast<const uint4*>(s_ptr[t]) + vb + c);
  }
  __syncthreads();

  // each row group of each column: the left fold of its inner positions
  for (uint32_t i = threadIdx.x; i < (uint32_t)groups * ncols; i += kThreads) {
    const int g = (int)(i / ncols);
    const uint32_t c = i % ncols;
    float a[L];
    for (int h = 0; h < inner; ++h) {
      const int t = g * inner + h;
      float f[L];
      unpack<F16>(*reinterpret_cast<const uint4*>(s_lat + (size_t)t * T + c * 16u), f);
      if (h == 0) {
#pragma unroll
        for (int l = 0; l < L; ++l) a[l] = f[l];
      } else {
        // rounded where the sum travels again: every inner add but the final
        // add of a single-group fold
        const bool round = rh && !(t == P - 1 && groups == 1);
#pragma unroll
        for (int l = 0; l < L; ++l) {
          const float v = __fadd_rn(a[l], f[l]);
          a[l] = round ? round_h(v) : v;
        }
      }
    }
    if constexpr (SINGLE) {  // one group: its fold is the result
#pragma unroll
      for (int l = 0; l < L; ++l) a[l] = __fmul_rn(a[l], p.scale);
      s_res[c] = pack<F16>(a);
    } else {
#pragma unroll
      for (int q = 0; q < L / 4; ++q)
        s_tot[((size_t)g * (L / 4) + q) * CT + c] = make_float4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
    }
  }
  __syncthreads();

  // each column: the left fold of its group totals, scaled, in storage form
  if constexpr (!SINGLE) {
    for (uint32_t c = threadIdx.x; c < ncols; c += kThreads) {
      float o[L];
#pragma unroll
      for (int q = 0; q < L / 4; ++q) {
        const float4 v = s_tot[(size_t)q * CT + c];
        o[4 * q] = v.x, o[4 * q + 1] = v.y, o[4 * q + 2] = v.z, o[4 * q + 3] = v.w;
      }
      for (int g = 1; g < groups; ++g) {
        const bool round = rh && g != groups - 1;  // the last group's add is the final one
        float t[L];
#pragma unroll
        for (int q = 0; q < L / 4; ++q) {
          const float4 v = s_tot[((size_t)g * (L / 4) + q) * CT + c];
          t[4 * q] = v.x, t[4 * q + 1] = v.y, t[4 * q + 2] = v.z, t[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int l = 0; l < L; ++l) {
          const float v = __fadd_rn(o[l], t[l]);
          o[l] = round ? round_h(v) : v;
        }
      }
#pragma unroll
      for (int l = 0; l < L; ++l) o[l] = __fmul_rn(o[l], p.scale);
      s_res[c] = pack<F16>(o);
    }
    __syncthreads();
  }
  // the result to every rank, all threads at once
  for (uint32_t i = threadIdx.x; i < (uint32_t)P * ncols; i += kThreads) {
    const uint32_t t = i / ncols, c = i % ncols;
    __stcs(reinterpret_cast<uint4*>(s_ptr[t]) + vb + c, s_res[c]);
  }
  // the few elements of a cut column at either end of the item
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    fold_scalar<F16>(s_ptr, e, P, inner, groups, rh, p.scale);
  }
}

// ---------------------------------------------------------------------------
// n-D torus register pass: the fold is d nested left folds (innermost over
// dim 0 from chunk c_0, then dim 1, ...).  A cascade of one accumulator per
// level follows the ranks in fold order: a finished group of level l is added
// into level l+1.  Every add is rounded to binary16 where a hop would carry
// it, except the final add (the last one at the highest level of size > 1).
// fp32 takes two columns per thread (items up to 8 KB per rank); fp16, whose
// 4 levels x 8 lanes of accumulators fill the registers, takes one (4 KB).
// ---------------------------------------------------------------------------
// One accumulator per level (levels written out, so every index is a
// compile-time constant and the accumulators live in registers); NL lanes.
template <int NL>
struct Cascade {
  float a0[NL], a1[NL], a2[NL], a3[NL];
  int c0 = 0, c1 = 0, c2 = 0, c3 = 0;

  // cur into level acc (first of its group: copy; else add, rounded unless final)
  __device__ __forceinline__ static void add(float* acc, const float* cur, bool first, bool round) {
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      if (first) {
        acc[l] = cur[l];
      } else {
        const float s = __fadd_rn(acc[l], cur[l]);
        acc[l] = round ? round_h(s) : s;
      }
    }
  }
  // one value at fold position t (last = t is the final position); returns
  // after the first level whose group is still open
  __device__ __forceinline__ void push(const float* v, bool last, const FoldParams& p, bool rh) {
    add(a0, v, c0 == 0, rh && !(last && p.top == 0));
    if (++c0 < (int)p.lev[0]) return;
    c0 = 0;
    if (p.nlev < 2) return;
    add(a1, a0, c1 == 0, rh && !(last && p.top == 1));
    if (++c1 < (int)p.lev[1]) return;
    c1 = 0;
    if (p.nlev < 3) return;
    add(a2, a1, c2 == 0, rh && !(last && p.top == 2));
    if (++c2 < (int)p.lev[2]) return;
    c2 = 0;
    if (p.nlev < 4) return;
    add(a3, a2, c3 == 0, rh && !(last && p.top == 3));
    if (++c3 < (int)p.lev[3]) return;
    c3 = 0;
  }
  // the outermost level's value
  __device__ __forceinline__ void result(float* out, int nlev) const {
#pragma unroll
    for (int l = 0; l < NL; ++l) out[l] = nlev == 1 ? a0[l] : nlev == 2 ? a1[l] : nlev == 3 ? a2[l] : a3[l];
  }
};

// The same cascade on binary16 pairs with rounded hops, for V columns (one
// set of group counters: every column of a thread follows the same order).
// Every position but the last adds packed (hadd2_rn, the rounded binary32 add
// bit for bit).  At the last position every group closes: the adds below
// level `top` are rounded as before, and the add at level `top` is the final
// one, taken in binary32; levels above `top` have size 1.
// NL: the plan's number of levels (a compile-time count, so unused levels
// take no registers).
template <int V, int NL>
struct CascadeH2 {
  uint32_t a0[V][4], a1[V][4], a2[V][4], a3[V][4];
  int c0 = 0, c1 = 0, c2 = 0, c3 = 0;

  __device__ __forceinline__ static void add(uint32_t (*acc)[4], const uint32_t (*cur)[4], bool first) {
#pragma unroll
    for (int u = 0; u < V; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[u][i] = first ? cur[u][i] : hadd2_rn(acc[u][i], cur[u][i]);
  }
  // a position before the last
  __device__ __forceinline__ void push(const uint32_t (*v)[4], const FoldParams& p) {
    add(a0, v, c0 == 0);
    if (++c0 < (int)p.lev[0]) return;
    c0 = 0;
    if constexpr (NL >= 2) {
      add(a1, a0, c1 == 0);
      if (++c1 < (int)p.lev[1]) return;
      c1 = 0;
    }
    if constexpr (NL >= 3) {
      add(a2, a1, c2 == 0);
      if (++c2 < (int)p.lev[2]) return;
      c2 = 0;
    }
    if constexpr (NL >= 4) {
      add(a3, a2, c3 == 0);
      if (++c3 < (int)p.lev[3]) return;
      c3 = 0;
    }
  }
  // the top level's add: binary32, unrounded
  __device__ __forceinline__ static void at_top(const uint32_t (*acc)[4], bool first, const uint32_t (*x)[4],
                                                float (*out)[8]) {
#pragma unroll
    for (int u = 0; u < V; ++u) {
      widen_h2(x[u], out[u]);
      if (first) continue;
      float a[8];
      widen_h2(acc[u], a);
#pragma unroll
      for (int l = 0; l < 8; ++l) out[u][l] = __fadd_rn(a[l], out[u][l]);
    }
  }
  // the last position's values; writes the fold's binary32 results
  // (top < NL: the highest level of size > 1, or -1 if there is none)
  __device__ __forceinline__ void last(uint32_t (*x)[4], const FoldParams& p, float (*out)[8]) const {
    const int top = p.top;
    if (top < 0) {
#pragma unroll
      for (int u = 0; u < V; ++u) widen_h2(x[u], out[u]);
      return;
    }
    // below the top x = acc + x, rounded, unless x opens the group
    if (top == 0) return at_top(a0, c0 == 0, x, out);
    if (c0 != 0) add(x, a0, false);
    if constexpr (NL >= 2) {
      if (top == 1) return at_top(a1, c1 == 0, x, out);
      if (c1 != 0) add(x, a1, false);
    }
    if constexpr (NL >= 3) {
      if (top == 2) return at_top(a2, c2 == 0, x, out);
      if (c2 != 0) add(x, a2, false);
    }
    if constexpr (NL >= 4) at_top(a3, c3 == 0, x, out);
  }
};

template <bool F16>
__device__ __noinline__ void fold_nd_scalar(const FoldParams& p, char* const* ptr, uint64_t e, bool rh) {
  Cascade<1> cs;
  for (int t0 = 0; t0 < p.P; t0 += 8) {  // loads eight positions at a time
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (t0 + j < p.P) v[j] = load_elem<F16>(ptr[t0 + j], e);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (t0 + j < p.P) cs.push(&v[j], t0 + j == p.P - 1, p, rh);
  }
  float fin;
  cs.result(&fin, p.nlev);
  const float r = __fmul_rn(fin, p.scale);
  for (int t = 0; t < p.P; ++t) store_elem<F16>(ptr[t], e, r);
}

template <bool F16, int V, int B>
__global__ void __launch_bounds__(kThreads, 2) fold_nd_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = F16 ? 8 : 4;
  __shared__ char* s_ptr[kMaxP];
  Item s_item;
  griddep_launch_dependents();
  if (!load_item(p, s_ptr, &s_item)) return;
  griddep_wait();
  const int P = p.P;
  const bool rh = F16 && p.round_hops;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;

  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads) fold_nd_scalar<F16>(p, s_ptr, e, rh);
    return;
  }
  if (ve - vb > (uint64_t)V * kThreads) {  // V columns per thread cover the largest item
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadItem);
    return;
  }
  uint64_t col[V];
  bool live[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    col[u] = vb + threadIdx.x + (uint64_t)u * kThreads;
    live[u] = col[u] < ve;
  }
  Cascade<L> cs[V];
  for (int t0 = 0; t0 < P; t0 += B) {
    uint4 raw[B][V];
#pragma unroll
    for (int j = 0; j < B; ++j)
      if (t0 + j < P) {
#pragma unroll
        for (int u = 0; u < V; ++u)
          raw[j][u] = live[u] ? __ldcs(reinterpret_cast<const uint4*>(s_ptr[t0 + j]) + col[u]) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (t0 + j < P) {
#pragma unroll
        for (int u = 0; u < V; ++u) {
          float f[L];
          unpack<F16>(raw[j][u], f);
          cs[u].push(f, t0 + j == P - 1, p, rh);
        }
      }
    }
  }
  uint4 res[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    float r[L];
    cs[u].result(r, p.nlev);
#pragma unroll
    for (int l = 0; l < L; ++l) r[l] = __fmul_rn(r[l], p.scale);
    res[u] = pack<F16>(r);
  }
  for (int t = 0; t < P; ++t) {
#pragma unroll
    for (int u = 0; u < V; ++u)
      if (live[u]) __stcs(reinterpret_cast<uint4*>(s_ptr[t]) + col[u], res[u]);
  }
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    fold_nd_scalar<F16>(p, s_ptr, e, rh);
  }
}

#ifndef DDL_ND_H2_B1
#define DDL_ND_H2_B1 8  // one or two levels
#endif
#ifndef DDL_ND_H2_B3
#define DDL_ND_H2_B3 7
#endif
#ifndef DDL_ND_H2_B4
#define DDL_ND_H2_B4 6
#endif

// binary16 with rounded hops: the packed cascade of NL levels; V columns per
// thread, B ranks' loads in flight
template <int V, int B, int NL>
__global__ void __launch_bounds__(kThreads, 2) fold_nd_h2_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = 8;
  __shared__ char* s_ptr[kMaxP];
  Item s_item;
  griddep_launch_dependents();
  if (!load_item(p, s_ptr, &s_item)) return;
  griddep_wait();
  const int P = p.P;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;

  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads) fold_nd_scalar<true>(p, s_ptr, e, true);
    return;
  }
  if (ve - vb > (uint64_t)V * kThreads) {  // V columns per thread cover the largest item
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadItem);
    return;
  }
  uint64_t col[V];
  bool live[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    col[u] = vb + threadIdx.x + (uint64_t)u * kThreads;
    live[u] = col[u] < ve;
  }
  CascadeH2<V, NL> cs;
  uint32_t xl[V][4];  // the last position's values
  for (int t0 = 0; t0 < P; t0 += B) {
    uint4 raw[B][V];
#pragma unroll
    for (int j = 0; j < B; ++j)
      if (t0 + j < P) {
#pragma unroll
        for (int u = 0; u < V; ++u)
          raw[j][u] = live[u] ? __ldcs(reinterpret_cast<const uint4*>(s_ptr[t0 + j]) + col[u]) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int j = 0; j < B; ++j) {
      if (t0 + j < P) {
        uint32_t w[V][4];
#pragma unroll
        for (int u = 0; u < V; ++u) {
          w[u][0] = raw[j][u].x;
          w[u][1] = raw[j][u].y;
          w[u][2] = raw[j][u].z;
          w[u][3] = raw[j][u].w;
        }
        if (t0 + j < P - 1) {
          cs.push(w, p);
        } else {
#pragma unroll
          for (int u = 0; u < V; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i) xl[u][i] = w[u][i];
        }
      }
    }
  }
  float fin[V][L];
  cs.last(xl, p, fin);
  uint4 res[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
#pragma unroll
    for (int l = 0; l < L; ++l) fin[u][l] = __fmul_rn(fin[u][l], p.scale);
    res[u] = pack<true>(fin[u]);
  }
  for (int t = 0; t < P; ++t) {
#pragma unroll
    for (int u = 0; u < V; ++u)
      if (live[u]) __stcs(reinterpret_cast<uint4*>(s_ptr[t]) + col[u], res[u]);
  }
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    fold_nd_scalar<true>(p, s_ptr, e, true);
  }
}

// ---------------------------------------------------------------------------
// Latency pass of the n-D torus: small items (at most 4 KB per rank) of n-D
// plans with at least 32 ranks whose P tiles fit in shared memory.  As the
// two-level latency pass above, the CTA loads all P ranks' columns of its item
// into shared memory at once, then folds the d levels of the n-D schedule:
// level 0 groups lev[0] consecutive fold positions, level l groups lev[l]
// totals of level l-1.  All groups of a level are folded at once, a thread per
// group and column, and a group's total goes into the shared-memory slot of
// its first member, which no other group reads (totals below the top are
// binary16 values where hops are rounded, so they keep their storage form).
// Every add is rounded to binary16 where a hop would carry it -- all but the
// final add, the last one at the highest level of size > 1 -- as in the n-D
// register pass.  The result is stored to every rank from shared memory.
// (The two-level plans keep their own pass: with totals kept in binary32 and a
// fixed two-step fold it measured 0.2-0.35 us faster on them.)
// Shared memory: P x tile bytes (fold position t at t * tile), then one
// 16-byte result per column.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr uint32_t lat_nd_smem_bytes(uint32_t P, uint32_t tile) {
  return P * tile + (tile / 16u) * 16u;
}

template <bool F16>
__global__ void __launch_bounds__(kThreads) fold_lat_nd_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = F16 ? 8 : 4;  // elements per 16-byte column
  extern __shared__ __align__(16) unsigned char s_lat[];
  __shared__ char* s_ptr[kMaxP];
  Item s_item;
  griddep_launch_dependents();
  if (!load_item(p, s_ptr, &s_item)) return;
  griddep_wait();

  const int P = p.P, nlev = p.nlev, top = p.top;
  const bool rh = F16 && p.round_hops;
  const uint32_t T = p.tile_bytes;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;
  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads) fold_nd_scalar<F16>(p, s_ptr, e, rh);
    return;
  }
  const uint32_t ncols = (uint32_t)(ve - vb);  // <= T / 16
  uint4* s_res = reinterpret_cast<uint4*>(s_lat + (size_t)P * T);

  // every fold position's columns, all loads in flight together
  for (uint32_t i = threadIdx.x; i < (uint32_t)P * ncols; i += kThreads) {
    const uint32_t t = i / ncols, c = i % ncols;
    *reinterpret_cast<uint4*>(s_lat + (size_t)t * T + c * 16u) =
        __ldcs(reinterpret_cast<const uint4*>(s_ptr[t]) + vb + c);
  }
  __syncthreads();

  // the levels, innermost first; members of a level-l group sit `stride`
  // slots apart
  int stride = 1;
  for (int l = 0; l < nlev; ++l) {
    const int D = (int)p.lev[l];
    if (D > 1) {
      const uint32_t ng = (uint32_t)(P / (stride * D));  // one group at the top level
      for (uint32_t i = threadIdx.x; i < ng * ncols; i += kThreads) {
        const uint32_t g = i / ncols, c = i % ncols;
        const size_t first = (size_t)g * (size_t)D * (size_t)stride;
        float a[L];
        unpack<F16>(*reinterpret_cast<const uint4*>(s_lat + first * T + c * 16u), a);
        for (int m = 1; m < D; ++m) {
          float f[L];
          unpack<F16>(*reinterpret_cast<const uint4*>(s_lat + (first + (size_t)m * stride) * T + c * 16u), f);
          const bool round = rh && !(l == top && m == D - 1);
#pragma unroll
          for (int q = 0; q < L; ++q) {
            const float v = __fadd_rn(a[q], f[q]);
            a[q] = round ? round_h(v) : v;
          }
        }
        if (l == top) {  // the final value: scaled, in storage form
#pragma unroll
          for (int q = 0; q < L; ++q) a[q] = __fmul_rn(a[q], p.scale);
          s_res[c] = pack<F16>(a);
        } else {         // a total below the top: exact in storage form
          *reinterpret_cast<uint4*>(s_lat + first * T + c * 16u) = pack<F16>(a);
        }
      }
      __syncthreads();
    }
    stride *= D;
  }

  // the result to every rank, all threads at once
  for (uint32_t i = threadIdx.x; i < (uint32_t)P * ncols; i += kThreads) {
    const uint32_t t = i / ncols, c = i % ncols;
    __stcs(reinterpret_cast<uint4*>(s_ptr[t]) + vb + c, s_res[c]);
  }
  // the few elements of a cut column at either end of the item
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    fold_nd_scalar<F16>(p, s_ptr, e, rh);
  }
}

// ---------------------------------------------------------------------------
// The bulk-load pass: shared-memory staged, with bulk asynchronous loads,
// warp-specialised.
//
// Persistent CTAs (one per SM) of 1 producer warp + 8 consumer warps walk
// their work items through a ring of kStages stages in shared memory.  The
// producer waits until the consumers have released a stage (its "empty"
// mbarrier), publishes the next item's bounds and fold order, arms the
// stage's "full" mbarrier with the byte count, and issues one cp.async.bulk
// per rank (global -> shared).  Consumers wait on "full", fold their columns
// from shared memory in the schedule's order, and release the stage.  The
// result goes back from registers, one 16-byte store per rank.  The producer
// never joins a consumer barrier, so its table reads stay off the consumers'
// path.  Every
// wait is bounded: a wait that runs out sets kErrWaitTimeout and the warp
// leaves its loop; the CTA then drains its own copies (bounded) and returns.
// ---------------------------------------------------------------------------

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kBulkThreads = kConsumers + 32;
constexpr int kStages = 3;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait before giving up

struct BulkMeta {
  uint64_t eb, ee;   // item elements [eb, ee)
  uint64_t vb, ve;   // 16-byte columns [vb, ve) staged through shared memory
  uint32_t inner, groups;
  uint32_t ok, order_off;
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for the phase with the given parity to complete: gives up
// after limit_ns of wall time (or 2^28 polls) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 28); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u && global_ns() - t0 > limit_ns) break;
  }
  return false;
}

// Exercises the bounded wait's give-up path: one CTA waits on an mbarrier
// that nothing arrives at, with a short limit, and records the timeout in
// the error word exactly as the staged kernels do.
__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) atomicOr(err, kErrWaitTimeout);
}

__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared memory: stages x P x tile | stages x kMaxP order | meta | barriers
__host__ __device__ constexpr uint32_t bulk_smem_bytes(uint32_t P, uint32_t tile) {
  return (uint32_t)kStages * P * tile + (uint32_t)kStages * kMaxP +
         (uint32_t)(kStages * sizeof(BulkMeta)) + (uint32_t)(2 * kStages * sizeof(uint64_t)) + 16u;
}

// Out of line, as fold_scalar: inlined, its batched loads raised the staged
// passes' registers (rank-chunked 80 to 94), which share the SMs with the
// producer's kernels on the overlap side stream.
template <bool F16>
__device__ __noinline__ void fold_scalar_ordered(const FoldParams& p, const uint8_t* order, uint64_t e, int inner, int groups,
                                    bool rh) {
  const auto at = [&p, order](int t) { return static_cast<const char*>(p.bufs[order[t]]); };
  const float r = __fmul_rn(fold_elem<F16>(at, e, p.P, inner, groups, rh), p.scale);
  for (int t = 0; t < p.P; ++t) store_elem<F16>(static_cast<char*>(p.bufs[order[t]]), e, r);
}

template <bool F16>
__global__ void __launch_bounds__(kBulkThreads, 1) fold_bulk_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = F16 ? 8 : 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t P = (uint32_t)p.P, T = p.tile_bytes;
  unsigned char* stage = smem;
  uint8_t* s_order = smem + (uint32_t)kStages * P * T;
  BulkMeta* s_meta = reinterpret_cast<BulkMeta*>(s_order + kStages * kMaxP);
  uint64_t* full = reinterpret_cast<uint64_t*>(s_meta + kStages);
  uint64_t* empty = full + kStages;

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  const uint32_t my_n = p.n_items > blockIdx.x ? (p.n_items - 1u - blockIdx.x) / gridDim.x + 1u : 0u;
  const bool rh = F16 && p.round_hops;

  if (tid == 0) {
    for (int k = 0; k < kStages; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  uint32_t issued = 0, consumed = 0;  // items this thread's role got through
  bool timed_out = false;

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    for (uint32_t s = 0; s < my_n; ++s) {
      const uint32_t k = s % kStages;
      if (s >= (uint32_t)kStages && !mbar_wait(&empty[k], ((s / kStages) - 1u) & 1u)) {
        timed_out = true;
        break;
      }
      if (lane == 0) {
        const Item item = p.items[p.item0 + blockIdx.x + s * gridDim.x];
        BulkMeta m;
        m.eb = item.begin;
        m.ee = item.begin + item.len;
        m.vb = (m.eb + L - 1) / L;
        m.ve = m.ee / L;
        if (m.ve < m.vb) m.ve = m.vb;
        m.order_off = item.seg * P;
        m.ok = item.seg < p.n_segs && (uint64_t)item.seg * P + P <= p.n_orders;
        m.inner = (uint32_t)p.inner;
        m.groups = (uint32_t)p.groups;
        if (!m.ok) atomicOr(p.err, kErrBadItem);
        s_meta[k] = m;
      }
      __syncwarp();
      const BulkMeta m = s_meta[k];
      if (m.ok)
        for (uint32_t t = lane; t < P; t += 32) {
          const uint32_t r = p.orders[m.order_off + t];
          s_order[k * kMaxP + t] = (uint8_t)(r < P ? r : 0);
        }
      const uint32_t bytes = m.ok ? (uint32_t)(m.ve - m.vb) * 16u : 0u;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[k], bytes * P);  // release: meta and order are published
      __syncwarp();
      if (bytes)
        for (uint32_t r = lane; r < P; r += 32)
          bulk_load(stage + ((size_t)k * P + r) * T, static_cast<const char*>(p.bufs[r]) + m.vb * 16u, bytes,
                    &full[k]);
      issued = s + 1;
    }
    if (timed_out && lane == 0) atomicOr(p.err, kErrWaitTimeout);
  } else {
    // ---------------- consumer warps ----------------
    for (uint32_t s = 0; s < my_n; ++s) {
      const uint32_t k = s % kStages;
      if (!mbar_wait(&full[k], (s / kStages) & 1u)) {
        timed_out = true;
        break;
      }
      const BulkMeta m = s_meta[k];
      const uint8_t* ord = s_order + k * kMaxP;
      const uint32_t ncols = (uint32_t)(m.ve - m.vb);
      if (m.ok) {
        const unsigned char* st = stage + (size_t)k * P * T;
        for (uint32_t c = tid; c < ncols; c += kConsumers) {
          float in[L], out[L];
          int h = 0, g = 0;
          for (uint32_t t0 = 0; t0 < P; t0 += 8) {
            uint4 raw[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (t0 + q < P) raw[q] = *reinterpret_cast<const uint4*>(st + (size_t)ord[t0 + q] * T + c * 16u);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (t0 + q < P) {
                float f[L];
                unpack<F16>(raw[q], f);
                const Ctl ctl = ctl_at((int)(t0 + q), h, g, (int)m.inner, (int)m.groups, (int)P, rh);
                fold_lanes<L>(in, out, f, ctl);
                if (++h == (int)m.inner) {
                  h = 0;
                  ++g;
                }
              }
            }
          }
          float r[L];
#pragma unroll
          for (int l = 0; l < L; ++l) r[l] = __fmul_rn(out[l], p.scale);
          const uint4 res = pack<F16>(r);
          for (uint32_t t = 0; t < P; ++t) __stcs(reinterpret_cast<uint4*>(p.bufs[t]) + m.vb + c, res);
        }
        // elements of a column cut by the item's ends: straight from global
        const uint64_t nh = (m.ve > m.vb) ? m.vb * L - m.eb : m.ee - m.eb;
        const uint64_t nt = (m.ve > m.vb) ? m.ee - m.ve * L : 0;
        if (tid < nh + nt) {
          const uint64_t e = tid < nh ? m.eb + tid : m.ve * L + (tid - nh);
          fold_scalar_ordered<F16>(p, ord, e, (int)m.inner, (int)m.groups, rh);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[k]);  // this warp is done with stage k
      consumed = s + 1;
    }
    if (timed_out && lane == 0) atomicOr(p.err, kErrWaitTimeout);
  }

  // Both roles leave their loops (every wait is bounded).  Publish how far the
  // producer got, then let loads that nobody consumed land before exit.
  __shared__ uint32_t s_issued, s_consumed;
  if (warp == kConsumerWarps && lane == 0) s_issued = issued;
  if (tid == 0) s_consumed = consumed;
  __syncthreads();
  if (tid == 0)
    for (uint32_t q = s_consumed; q < s_issued; ++q) mbar_wait(&full[q % kStages], (q / kStages) & 1u);
}

// ---------------------------------------------------------------------------
// The rank-chunked pass: staged through shared memory in rank chunks.  The
// bulk-load pass above holds all P ranks of a tile in one stage, so at large P a
// stage carries little per rank and few consumers have work.  Here a stage
// holds kChunk ranks (in fold order) of a whole register-pass tile (up to
// 8 KB per rank): the producer warp streams an item's ranks through the
// stage ring chunk by chunk with one cp.async.bulk per rank, and each of
// the 256 consumer threads keeps its two 16-byte columns' fold in registers
// across the item's chunks, then scales and stores the result to every rank
// from registers.  Every wait is bounded as in the bulk-load pass.  Two
// ranks per stage, three stages and two CTAs per SM measured fastest (8 ranks
// per stage and one CTA: 0.92 of the copy peak at P = 16; deeper rings were
// slower too).
// ---------------------------------------------------------------------------
#ifndef DDL_CHUNK_RANKS
#define DDL_CHUNK_RANKS 2
#endif
#ifndef DDL_CHUNK_MINB
#define DDL_CHUNK_MINB 2
#endif
#ifndef DDL_CHUNK_STAGES
#define DDL_CHUNK_STAGES 3
#endif
constexpr int kChunk = DDL_CHUNK_RANKS;  // ranks per stage
constexpr int kCStages = DDL_CHUNK_STAGES;  // depth of the stage ring

struct ChunkMeta {
  uint64_t eb, ee, vb, ve;  // item elements [eb, ee); staged columns [vb, ve)
  uint32_t t0, nr;          // this stage's fold positions [t0, t0 + nr)
  uint32_t ok, last;        // table entry valid; last chunk of the item
};

// stages x kChunk x tile | stages x kMaxP order | stages meta | barriers
__host__ __device__ constexpr uint32_t chunked_smem_bytes(uint32_t tile) {
  return (uint32_t)kCStages * kChunk * tile + (uint32_t)kCStages * kMaxP + (uint32_t)(kCStages * sizeof(ChunkMeta)) +
         (uint32_t)(2 * kCStages * sizeof(uint64_t)) + 16u;
}

template <bool F16>
__global__ void __launch_bounds__(kBulkThreads, DDL_CHUNK_MINB) fold_chunked_kernel(const __grid_constant__ FoldParams p) {
  constexpr int L = F16 ? 8 : 4;
  constexpr int V = 2;  // columns per consumer thread: 2 x 256 x 16 B = 8 KB
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t P = (uint32_t)p.P, T = p.tile_bytes;
  unsigned char* stage = smem;
  uint8_t* s_order = smem + (uint32_t)kCStages * kChunk * T;
  ChunkMeta* s_meta = reinterpret_cast<ChunkMeta*>(s_order + kCStages * kMaxP);
  uint64_t* full = reinterpret_cast<uint64_t*>(s_meta + kCStages);
  uint64_t* empty = full + kCStages;

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  const uint32_t my_n = p.n_items > blockIdx.x ? (p.n_items - 1u - blockIdx.x) / gridDim.x + 1u : 0u;
  const uint32_t nq = (P + kChunk - 1) / kChunk;  // chunks per item
  const uint32_t n_stages = my_n * nq;
  const bool rh = F16 && p.round_hops;

  if (tid == 0) {
    for (int k = 0; k < kCStages; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  uint32_t issued = 0, consumed = 0;  // stages this thread's role got through
  bool timed_out = false;

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ----------------
    for (uint32_t u = 0; u < n_stages; ++u) {
      const uint32_t k = u % kCStages, s = u / nq, q = u % nq;
      if (u >= (uint32_t)kCStages && !mbar_wait(&empty[k], ((u / kCStages) - 1u) & 1u)) {
        timed_out = true;
        break;
      }
      if (lane == 0) {
        const Item item = p.items[p.item0 + blockIdx.x + s * gridDim.x];
        ChunkMeta m;
        m.eb = item.begin;
        m.ee = item.begin + item.len;
        m.vb = (m.eb + L - 1) / L;
        m.ve = m.ee / L;
        if (m.ve < m.vb) m.ve = m.vb;
        m.t0 = q * kChunk;
        m.nr = P - m.t0 < (uint32_t)kChunk ? P - m.t0 : (uint32_t)kChunk;
        m.last = q + 1 == nq;
        m.ok = item.seg < p.n_segs && (uint64_t)item.seg * P + P <= p.n_orders &&
               (m.ve - m.vb) * 16u <= (uint64_t)T;
        if (!m.ok) atomicOr(p.err, kErrBadItem);
        s_meta[k] = m;
      }
      __syncwarp();
      const ChunkMeta m = s_meta[k];
      const uint32_t seg = p.items[p.item0 + blockIdx.x + s * gridDim.x].seg;
      if (m.ok)
        for (uint32_t t = lane; t < P; t += 32) {
          const uint32_t r = p.orders[(uint64_t)seg * P + t];
          s_order[k * kMaxP + t] = (uint8_t)(r < P ? r : 0);
        }
      const uint32_t bytes = m.ok ? (uint32_t)(m.ve - m.vb) * 16u : 0u;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[k], bytes * m.nr);  // release: meta and order are published
      __syncwarp();
      if (bytes && lane < m.nr) {
        const uint32_t r = s_order[k * kMaxP + m.t0 + lane];
        bulk_load(stage + ((size_t)k * kChunk + lane) * T, static_cast<const char*>(p.bufs[r]) + m.vb * 16u, bytes,
                  &full[k]);
      }
      issued = u + 1;
    }
    if (timed_out && lane == 0) atomicOr(p.err, kErrWaitTimeout);
  } else {
    // ---------------- consumer warps ----------------
    float in[V][L], out[V][L];
    uint32_t hin[V][4] = {}, hout[V][4] = {};  // packed binary16 accumulators (rounded hops)
    int h = 0, g = 0;
    for (uint32_t u = 0; u < n_stages; ++u) {
      const uint32_t k = u % kCStages;
      if (!mbar_wait(&full[k], (u / kCStages) & 1u)) {
        timed_out = true;
        break;
      }
      const ChunkMeta m = s_meta[k];
      const uint32_t ncols = (uint32_t)(m.ve - m.vb);
      const int inner = p.inner, groups = p.groups;
      if (m.t0 == 0) h = g = 0;
      if (m.ok) {
        const unsigned char* st = stage + (size_t)k * kChunk * T;
        for (uint32_t j = 0; j < m.nr; ++j) {
          const int t = (int)(m.t0 + j);
          const Ctl c = ctl_at(t, h, g, inner, groups, (int)P, rh);
#pragma unroll
          for (int v = 0; v < V; ++v) {
            const uint32_t col = tid + (uint32_t)v * kConsumers;
            if (col >= ncols) continue;
            const uint4 raw = *reinterpret_cast<const uint4*>(st + (size_t)j * T + col * 16u);
            if constexpr (F16) {
              if (rh && t < (int)P - 1) {
                fold_h2(hin[v], hout[v], raw, c);
                continue;
              }
              if (rh) {  // the last position: its final add stays binary32
                widen_h2(hin[v], in[v]);
                widen_h2(hout[v], out[v]);
              }
            }
            float f[L];
            unpack<F16>(raw, f);
            fold_lanes<L>(in[v], out[v], f, c);
          }
          if (++h == inner) {
            h = 0;
            ++g;
          }
        }
      }
      if (m.ok && m.last) {  // before releasing the stage: the edge path reads its order
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const uint32_t col = tid + (uint32_t)v * kConsumers;
          if (col >= ncols) continue;
          float r[L];
#pragma unroll
          for (int l = 0; l < L; ++l) r[l] = __fmul_rn(out[v][l], p.scale);
          const uint4 res = pack<F16>(r);
          for (uint32_t t = 0; t < P; ++t) __stcs(reinterpret_cast<uint4*>(p.bufs[t]) + m.vb + col, res);
        }
        // elements of a column cut by the item's ends: straight from global
        const uint64_t nh = (m.ve > m.vb) ? m.vb * L - m.eb : m.ee - m.eb;
        const uint64_t nt = (m.ve > m.vb) ? m.ee - m.ve * L : 0;
        if (tid < nh + nt) {
          const uint64_t e = tid < nh ? m.eb + tid : m.ve * L + (tid - nh);
          fold_scalar_ordered<F16>(p, s_order + k * kMaxP, e, inner, groups, rh);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[k]);  // this warp is done with stage k
      consumed = u + 1;
    }
    if (timed_out && lane == 0) atomicOr(p.err, kErrWaitTimeout);
  }

  // Both roles leave their loops (every wait is bounded).  Publish how far the
  // producer got, then let loads that nobody consumed land before exit.
  __shared__ uint32_t s_issued, s_consumed;
  if (warp == kConsumerWarps && lane == 0) s_issued = issued;
  if (tid == 0) s_consumed = consumed;
  __syncthreads();
  if (tid == 0)
    for (uint32_t q = s_consumed; q < s_issued; ++q) mbar_wait(&full[q % kCStages], (q / kCStages) & 1u);
}

template <bool F16>
cudaError_t launch_bulk(const FoldParams& p, uint32_t n_items, cudaStream_t stream) {
  const uint32_t smem = bulk_smem_bytes((uint32_t)p.P, p.tile_bytes);
  int dev = 0, sms = 0, max_smem = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (smem > (uint32_t)max_smem || p.tile_bytes % 16 != 0 || p.tile_bytes == 0) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(fold_bulk_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const uint32_t grid = n_items < (uint32_t)sms ? n_items : (uint32_t)sms;
  fold_bulk_kernel<F16><<<grid, kBulkThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_chunked(const FoldParams& p, uint32_t n_items, cudaStream_t stream) {
  const uint32_t smem = chunked_smem_bytes(p.tile_bytes);
  int dev = 0, sms = 0, max_smem = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  // two 16-byte columns per consumer thread cover a tile of at most 8 KB
  if (smem > (uint32_t)max_smem || p.tile_bytes % 16 != 0 || p.tile_bytes == 0 ||
      p.tile_bytes > 2u * (uint32_t)kConsumers * 16u)
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(fold_chunked_kernel<F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const uint32_t cap = (uint32_t)sms * DDL_CHUNK_MINB;
  const uint32_t grid = n_items < cap ? n_items : cap;
  fold_chunked_kernel<F16><<<grid, kBulkThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// One CTA of kThreads per work item, optionally as a programmatic dependent.
cudaError_t launch_items(void (*kernel)(FoldParams), const FoldParams& p, uint32_t n_items, cudaStream_t stream,
                         bool early, uint32_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// The latency pass takes small items (at most 4 KB per rank) of plans with at
// least kLatMinP ranks (plan.h) whose shared-memory footprint stays within
// kLatMaxSmem.  Measured per all-reduce in graph replay at 16,384 elements per
// rank: P = 32 (8x4 fp16 torus) 5.33 us against 7.18 us in the register pass
// (1 KB items), P = 64 (4-ring multi-ring, fp32) 4.72 against 8.62 us; with
// 256-byte items, P = 16 ring 2.27 against 2.88 us (small-item pass) and 4x4
// torus 2.33 against 3.17 us (register pass).  Below 16 it is mixed (P = 8:
// fp16 torus 2.26 against 2.87 us, fp32 torus at 65,536 elements 2.67 against
// 2.46 us) and at P = 4 it loses (ring 2.05 against 1.64 us).
constexpr uint32_t kLatMaxSmem = 96u * 1024u;

// The n-D latency pass's conditions: aligned buffers, items of at most 4 KB
// per rank, P >= kLatMinP, levels that cover the P ranks, the tiles within
// kLatMaxSmem.
bool lat_nd_applies(const FoldParams& p) {
  if (!p.vector_ok || p.tile_bytes > (uint32_t)kThreads * 16u || p.P < kLatMinP) return false;
  if (p.nlev < 1 || p.nlev > kMaxDims || p.top < 0 || p.top >= p.nlev) return false;
  int64_t prod = 1;
  for (int l = 0; l < p.nlev; ++l) prod *= p.lev[l];
  return prod == p.P && lat_nd_smem_bytes((uint32_t)p.P, p.tile_bytes) <= kLatMaxSmem;
}

// The current device's SM count, looked up once per device (GB300's 152 if the
// query fails).  Threads may launch at once: the cache is atomic.
uint32_t sm_count() {
  static std::atomic<int> sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      return 152;
    }
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return (uint32_t)n;
}

// CTAs of the latency pass that fit on the GPU at once with `smem` bytes of
// dynamic shared memory each (plus the 2 KB rank-pointer table, and 1 KB the
// hardware keeps per CTA; at most 8 CTAs of kThreads per SM).
uint32_t lat_wave(uint32_t smem) {
  const uint32_t per_sm_bytes = 228u * 1024u;
  uint32_t per_sm = per_sm_bytes / (smem + 3u * 1024u);
  if (per_sm > 8u) per_sm = 8u;
  if (per_sm < 1u) per_sm = 1u;
  return per_sm * sm_count();
}

// The opt-in above 48 KB of shared memory, once per kernel and device (the
// attribute call is idempotent, so two threads that race here both succeed).
cudaError_t lat_smem_opt_in(void (*kernel)(FoldParams), std::atomic<bool>* ready) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kLatMaxSmem);
    if (e != cudaSuccess) return e;
    ready[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

template <bool F16>
cudaError_t launch_lat_nd(const FoldParams& p, uint32_t n_items, cudaStream_t stream, bool early) {
  static std::atomic<bool> ready[64];
  const cudaError_t e = lat_smem_opt_in(fold_lat_nd_kernel<F16>, ready);
  if (e != cudaSuccess) return e;
  return launch_items(fold_lat_nd_kernel<F16>, p, n_items, stream, early, lat_nd_smem_bytes((uint32_t)p.P, p.tile_bytes));
}

template <bool F16>
cudaError_t launch_lat(const FoldParams& p, uint32_t n_items, cudaStream_t stream, bool early, uint32_t smem) {
  static std::atomic<bool> ready[2][64];
  const bool single = p.groups == 1;
  void (*const kernel)(FoldParams) = single ? fold_lat_kernel<F16, true> : fold_lat_kernel<F16, false>;
  const cudaError_t e = lat_smem_opt_in(kernel, ready[single ? 1 : 0]);
  if (e != cudaSuccess) return e;
  return launch_items(kernel, p, n_items, stream, early, smem);
}

template <bool F16>
cudaError_t launch_ldg(const FoldParams& p, uint32_t n_items, cudaStream_t stream, bool early) {
  // two 16-byte columns per thread cover kTileBytes per rank; a larger item
  // is refused (the element-wise path, taken for unaligned buffers, covers
  // any item)
  if (p.vector_ok && p.tile_bytes > (uint32_t)kTileBytes) return cudaErrorInvalidValue;
  // 4 KB items (buffers of 1.2 to 2.5 MB per rank, L2-resident): one column
  // per thread keeps every thread busy, and the smaller register set fits
  // three CTAs per SM (four with packed binary16 hops).  Per all-reduce in
  // graph replay: 4x4 torus at 524,288 elements 10.07 against 8.86 us, 8x4
  // fp16 torus at 1,048,576 elements 23.78 against 19.04 us.  With 1 KB items
  // it measured slower (P = 8 torus at 65,536 elements 2.46 against 3.08 us).
  if (p.tile_bytes == (uint32_t)kThreads * 16u) {
    if constexpr (F16) {
      if (p.round_hops) return launch_items(fold_ldg_kernel<true, true, 1, 8, 4>, p, n_items, stream, early);
      return launch_items(fold_ldg_kernel<true, false, 1, 8, 3>, p, n_items, stream, early);
    } else {
      return launch_items(fold_ldg_kernel<false, false, 1, 8, 3>, p, n_items, stream, early);
    }
  }
  if constexpr (F16) {
    if (p.round_hops)
      return launch_items(fold_ldg_kernel<true, true, 2, DDL_LDG_F16_B, DDL_LDG_MINB>, p, n_items, stream, early);
    return launch_items(fold_ldg_kernel<true, false, 2, DDL_LDG_F16_B, DDL_LDG_MINB>, p, n_items, stream, early);
  } else {
    return launch_items(fold_ldg_kernel<false, false, 2, DDL_LDG_F32_B, DDL_LDG_MINB>, p, n_items, stream, early);
  }
}

// The n-D torus's level-cascade register pass: two columns per thread (items
// up to 8 KB); fp16 with rounded hops folds packed pairs, fp16 without them
// (unused by the plans) one column (4 KB).
cudaError_t launch_nd(const FoldParams& p, uint32_t n_items, bool f16, cudaStream_t stream, bool early) {
  // 2 and 4 KB items: one column per thread, as in the 2-level pass (4x4x4
  // torus at 262,144 elements 34.1 against 27.0 us, 4x4x2 fp16 torus at
  // 1,048,576 elements 24.0 against 19.4 us per all-reduce in graph replay)
  if (p.tile_bytes >= 2048u && p.tile_bytes <= (uint32_t)kThreads * 16u) {
    if (f16 && p.round_hops) {
      if (p.nlev < 1 || p.nlev > 4) return cudaErrorInvalidValue;
      void (*const h1[4])(FoldParams) = {fold_nd_h2_kernel<1, DDL_ND_H2_B1, 1>, fold_nd_h2_kernel<1, DDL_ND_H2_B1, 2>,
                                         fold_nd_h2_kernel<1, DDL_ND_H2_B3, 3>, fold_nd_h2_kernel<1, DDL_ND_H2_B4, 4>};
      return launch_items(h1[p.nlev - 1], p, n_items, stream, early);
    }
    return launch_items(f16 ? fold_nd_kernel<true, 1, 8> : fold_nd_kernel<false, 1, 8>, p, n_items, stream, early);
  }
  if (f16 && p.round_hops) {
    if (p.nlev < 1 || p.nlev > 4) return cudaErrorInvalidValue;
    void (*const h2[4])(FoldParams) = {fold_nd_h2_kernel<2, DDL_ND_H2_B1, 1>, fold_nd_h2_kernel<2, DDL_ND_H2_B1, 2>,
                                       fold_nd_h2_kernel<2, DDL_ND_H2_B3, 3>, fold_nd_h2_kernel<2, DDL_ND_H2_B4, 4>};
    return launch_items(h2[p.nlev - 1], p, n_items, stream, early);
  }
  if (f16) return launch_items(fold_nd_kernel<true, 1, 8>, p, n_items, stream, early);
  return launch_items(fold_nd_kernel<false, 2, 8>, p, n_items, stream, early);
}

uint32_t lat_smem_of(const FoldParams& p, bool f16) {
  return lat_smem_bytes((uint32_t)p.P, (uint32_t)p.groups, p.tile_bytes, f16 ? 8u : 4u);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint32_t* err, uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

FoldPass fold_pass(const FoldParams& p, uint32_t n_items, bool f16, int variant) {
  if (p.nlev > 0)  // n-D torus: small items of many ranks take its latency pass
    return variant == kVarLdg && lat_nd_applies(p) ? kPassNdLatency : kPassNdRegister;
  if (variant == kVarBulkLoad) return kPassBulkLoad;
  if (variant == kVarChunked) return kPassChunked;
  // small items of many ranks: the latency pass, within the limits where it
  // measured fastest (per all-reduce in graph replay):
  // - several fold groups, or binary16 hops: items of at most 2 KB per rank;
  //   with 4 KB items two of its CTAs fit on an SM and the register pass wins
  //   (4x4 torus at 524,288 elements: 16.6 against 10.0 us; P = 16 fp16 ring
  //   at 1,048,576: 16.9 against 10.0 us; 8x4 fp16 torus at 524,288, 2 KB
  //   items: 18.0 against 18.9 us);
  // - a single unrounded group: items within one wave of its CTAs, else the
  //   small-item pass's occupancy wins (P = 64 multi-ring, 3 latency CTAs per
  //   SM with 1 KB items: 409 items 16.6 against 18.4 us, 646 items 26.0
  //   against 20.5 us); and below 32 ranks items of at most 512 bytes, where
  //   the small-item pass's chain of P / 4 round trips is short (P = 16 ring
  //   at 262,144 elements, 2 KB items: 7.05 against 5.74 us).
  const bool unrounded = !f16 || !p.round_hops;
  const bool single = unrounded && p.groups == 1 && p.inner == p.P;
  const bool small_items = p.tile_bytes <= (uint32_t)kThreads * 16u;
  const int lat_min_p = f16 && p.round_hops ? kLatMinPHops : kLatMinP;
  if (p.vector_ok && small_items && p.P >= lat_min_p && p.groups >= 1 && p.inner >= 1 &&
      (int64_t)p.inner * p.groups == p.P) {
    const uint32_t smem = lat_smem_of(p, f16);
    bool take = smem <= kLatMaxSmem;
    if (!single) take = take && p.tile_bytes <= 2048u;
    if (single) take = take && n_items <= lat_wave(smem) && (p.P >= 32 || p.tile_bytes <= 512u);
    if (take) return p.groups == 1 ? kPassLatencySingle : kPassLatency;
  }
  // small items of a single unrounded group: the small-item pass (one column
  // per thread covers up to kThreads * 16 bytes per rank)
  if (single && small_items) return kPassSmallItem;
  return kPassRegister;
}

const char* fold_pass_kernel(FoldPass pass, bool packed_hops) {
  switch (pass) {
    case kPassRegister: return "fold_ldg_kernel";
    case kPassSmallItem: return "fold_small_kernel";
    case kPassLatency: return "fold_lat_kernel";
    case kPassLatencySingle: return "fold_lat_kernel (one group)";
    case kPassNdRegister: return packed_hops ? "fold_nd_h2_kernel" : "fold_nd_kernel";
    case kPassNdLatency: return "fold_lat_nd_kernel";
    case kPassBulkLoad: return "fold_bulk_kernel";
    case kPassChunked: return "fold_chunked_kernel";
  }
  return "unknown";
}

cudaError_t launch_fold(const FoldParams& p, uint32_t n_items, bool f16, int variant, cudaStream_t stream,
                        bool early_launch) {
  if (n_items == 0) return cudaSuccess;
  switch (fold_pass(p, n_items, f16, variant)) {
    case kPassNdLatency:
      return f16 ? launch_lat_nd<true>(p, n_items, stream, early_launch)
                 : launch_lat_nd<false>(p, n_items, stream, early_launch);
    case kPassNdRegister:
      return launch_nd(p, n_items, f16, stream, early_launch);
    case kPassBulkLoad:
      return f16 ? launch_bulk<true>(p, n_items, stream) : launch_bulk<false>(p, n_items, stream);
    case kPassChunked:
      return f16 ? launch_chunked<true>(p, n_items, stream) : launch_chunked<false>(p, n_items, stream);
    case kPassLatency:
    case kPassLatencySingle:
      return f16 ? launch_lat<true>(p, n_items, stream, early_launch, lat_smem_of(p, true))
                 : launch_lat<false>(p, n_items, stream, early_launch, lat_smem_of(p, false));
    case kPassSmallItem:
      return launch_items(f16 ? fold_small_kernel<true> : fold_small_kernel<false>, p, n_items, stream, early_launch);
    case kPassRegister:
      break;
  }
  return f16 ? launch_ldg<true>(p, n_items, stream, early_launch) : launch_ldg<false>(p, n_items, stream, early_launch);
}

}  // namespace ddl
