// sgd_kernels.cu -- the fused all-reduce followed by the momentum-SGD update.
//
// Synchronous data-parallel SGD runs forward, backward, the gradient
// all-reduce, then the update, every iteration (Baidu write-up, opening
// paragraph; "索尼发布新的方法...ResNet-50", section "2大方法解决不稳定问题").
// This pass folds each column of the P gradient buffers in the schedule's
// order exactly as the fused all-reduce does, rounds the scaled mean to the
// gradient's storage type, and then -- still in registers -- applies
//   d = g + wd * p;   v = mu * v + d;   p = p - lr * v
// to every rank's binary32 parameter and momentum copy, each operation
// rounded on its own (_rn intrinsics: no fused multiply-add).  The gradient is
// read once and, if asked, written once; the unfused sequence would read it
// again for the update.
#include <cuda_fp16.h>

#include <atomic>

#include "kernels.h"

namespace ddl {
namespace {

constexpr int kThreads = 256;
constexpr int kV = 2;  // 16-byte gradient columns per thread
constexpr int kB = 8;  // ranks' loads in flight
#ifndef DDL_SGD_F16_UB
#define DDL_SGD_F16_UB 1  // fp16: ranks whose parameters and momenta are loaded at once
#endif

__device__ __forceinline__ float round_h(float x) { return __half2float(__float2half_rn(x)); }

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
  if constexpr (F16) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = (uint32_t)__half_as_ushort(__float2half_rn(f[2 * i])) |
             ((uint32_t)__half_as_ushort(__float2half_rn(f[2 * i + 1])) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
}

// fold one rank's lanes into (in, out): groups of `inner` left-folded, then
// the group totals; every add rounded to binary16 where a hop carries it,
// except the last add of the fold
template <int NL>
__device__ __forceinline__ void fold_step(float* in, float* out, const float* v, int t, int h, int g, int inner,
                                          int groups, int P, bool rh) {
  const bool last = (t == P - 1), gs = (h == 0), ge = (h == inner - 1), fg = (g == 0);
  const bool rin = rh && !(last && groups == 1), rout = rh && !last;
#pragma unroll
  for (int l = 0; l < NL; ++l) {
    float a = v[l];
    if (!gs) {
      a = __fadd_rn(in[l], a);
      if (rin) a = round_h(a);
    }
    in[l] = a;
    if (ge) {
      float o = a;
      if (!fg) {
        o = __fadd_rn(out[l], a);
        if (rout) o = round_h(o);
      }
      out[l] = o;
    }
  }
}

// A fold position before the last with binary16 hops: every add is rounded to
// binary16, and fl16(fl32(a + b)) is the correctly rounded binary16 sum
// (binary32 has 24 >= 2*11 + 2 significand bits: Figueroa, "When is double
// rounding innocuous?", 1995), so one packed add.rn.f16x2 does two lanes.
__device__ __forceinline__ uint32_t hadd2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void fold_step_h2(uint32_t* in, uint32_t* out, const uint4 v, int h, int g, int inner) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t a = w[i];
    if (h != 0) a = hadd2_rn(in[i], a);
    in[i] = a;
    if (h == inner - 1) out[i] = g == 0 ? a : hadd2_rn(out[i], a);
  }
}

__device__ __forceinline__ void widen_h2(const uint32_t* hv, float* f) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __half2float(__ushort_as_half((unsigned short)(hv[i] & 0xFFFFu)));
    f[2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(hv[i] >> 16)));
  }
}

// the update of one element of one rank; returns the new parameter, writes v
__device__ __forceinline__ float sgd_one(float g, float pv, float* mv, const SgdParams& p) {
  const float d = __fadd_rn(g, __fmul_rn(p.wd, pv));
  const float v = p.has_mom ? __fadd_rn(__fmul_rn(p.mu, *mv), d) : d;
  *mv = v;
  return __fsub_rn(pv, __fmul_rn(p.lr, v));
}

template <bool F16>
__device__ void sgd_scalar(const SgdParams& p, char* const* gp, float* const* pp, float* const* mp, uint64_t e,
                           int inner, int groups, bool rh) {
  float in = 0.f, out = 0.f;
  int h = 0, g = 0;
  for (int t = 0; t < p.P; ++t) {
    const float v = F16 ? __half2float(__ushort_as_half(reinterpret_cast<const unsigned short*>(gp[t])[e]))
                        : reinterpret_cast<const float*>(gp[t])[e];
    fold_step<1>(&in, &out, &v, t, h, g, inner, groups, p.P, rh);
    if (++h == inner) {
      h = 0;
      ++g;
    }
  }
  float gm = __fmul_rn(out, p.scale);
  if (F16) gm = round_h(gm);  // the update reads the gradient as stored
  for (int t = 0; t < p.P; ++t) {
    if (p.keep_grads) {
      if (F16) reinterpret_cast<unsigned short*>(gp[t])[e] = __half_as_ushort(__float2half_rn(gm));
      else reinterpret_cast<float*>(gp[t])[e] = gm;
    }
    float m = p.has_mom ? mp[t][e] : 0.f;
    pp[t][e] = sgd_one(gm, pp[t][e], &m, p);
    if (p.has_mom) mp[t][e] = m;
  }
}

// H2: binary16 with rounded hops, folded as packed pairs up to the last position
template <bool F16, bool H2>
__global__ void __launch_bounds__(kThreads, 2) fold_sgd_kernel(const __grid_constant__ SgdParams p) {
  static_assert(F16 || !H2, "packed hops are binary16 only");
  constexpr int L = F16 ? 8 : 4;  // gradient elements per 16-byte column
  constexpr int Q = L / 4;        // 16-byte binary32 vectors per column of parameters
  __shared__ char* s_g[kMaxPSgd];
  __shared__ float* s_p[kMaxPSgd];
  __shared__ float* s_m[kMaxPSgd];
  // a programmatic dependent of the kernel before it (see launch_sgd): tables
  // first, then wait for that kernel before touching gradients or parameters
  asm volatile("griddepcontrol.launch_dependents;");
  const Item s_item = p.items[p.item0 + blockIdx.x];  // one broadcast load
  const uint64_t off = (uint64_t)s_item.seg * (uint64_t)p.P;
  if (!(s_item.seg < p.n_segs && off + (uint64_t)p.P <= p.n_orders)) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadItem);
    return;
  }
  for (int t = threadIdx.x; t < p.P; t += kThreads) {
    unsigned r = p.orders[off + t];
    r = r < (unsigned)p.P ? r : 0;
    s_g[t] = static_cast<char*>(p.grads[r]);
    s_p[t] = p.params[r];
    s_m[t] = p.moms[r];
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int P = p.P, inner = p.inner, groups = p.groups;
  const bool rh = F16 && p.round_hops;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;
  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads) sgd_scalar<F16>(p, s_g, s_p, s_m, e, inner, groups, rh);
    return;
  }
  uint64_t col[kV];
  bool live[kV];
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    col[u] = vb + threadIdx.x + (uint64_t)u * kThreads;
    live[u] = col[u] < ve;
  }
  float in[kV][L], out[kV][L];
  uint32_t hin[kV][4] = {}, hout[kV][4] = {};  // packed accumulators (H2)
  int h = 0, g = 0;
  for (int t0 = 0; t0 < P; t0 += kB) {
    uint4 raw[kB][kV];
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (t0 + j < P) {
#pragma unroll
        for (int u = 0; u < kV; ++u)
          raw[j][u] = live[u] ? __ldcs(reinterpret_cast<const uint4*>(s_g[t0 + j]) + col[u]) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (t0 + j < P) {
#pragma unroll
        for (int u = 0; u < kV; ++u) {
          if constexpr (H2) {
            if (t0 + j < P - 1) {
              fold_step_h2(hin[u], hout[u], raw[j][u], h, g, inner);
              continue;
            }
            widen_h2(hin[u], in[u]);  // the last position: its final add stays binary32
            widen_h2(hout[u], out[u]);
          }
          float f[L];
          unpack<F16>(raw[j][u], f);
          fold_step<L>(in[u], out[u], f, t0 + j, h, g, inner, groups, P, rh);
        }
        if (++h == inner) {
          h = 0;
          ++g;
        }
      }
  }
  float gm[kV][L];
  uint4 res[kV];
#pragma unroll
  for (int u = 0; u < kV; ++u) {
#pragma unroll
    for (int l = 0; l < L; ++l) gm[u][l] = __fmul_rn(out[u][l], p.scale);
    res[u] = pack<F16>(gm[u]);
    if (F16) unpack<F16>(res[u], gm[u]);  // the update reads the gradient as stored
  }
  // the update: parameter and momentum loads of kUB ranks in flight at once
  constexpr int kUB = F16 ? DDL_SGD_F16_UB : 4;  // fp16 columns carry twice the parameters
  for (int t0 = 0; t0 < P; t0 += kUB) {
    float4 pw[kUB][kV][Q], mw[kUB][kV][Q];
#pragma unroll
    for (int j = 0; j < kUB; ++j)
#pragma unroll
      for (int u = 0; u < kV; ++u)
        if (t0 + j < P && live[u]) {
          const float4* pv = reinterpret_cast<const float4*>(s_p[t0 + j]) + col[u] * Q;
          const float4* mv = reinterpret_cast<const float4*>(s_m[t0 + j]) + col[u] * Q;
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            pw[j][u][q] = __ldcs(pv + q);
            mw[j][u][q] = p.has_mom ? __ldcs(mv + q) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
    for (int j = 0; j < kUB; ++j)
#pragma unroll
      for (int u = 0; u < kV; ++u)
        if (t0 + j < P && live[u]) {
          if (p.keep_grads) __stcs(reinterpret_cast<uint4*>(s_g[t0 + j]) + col[u], res[u]);
          float4* pv = reinterpret_cast<float4*>(s_p[t0 + j]) + col[u] * Q;
          float4* mv = reinterpret_cast<float4*>(s_m[t0 + j]) + col[u] * Q;
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            float* pe = reinterpret_cast<float*>(&pw[j][u][q]);
            float* me = reinterpret_cast<float*>(&mw[j][u][q]);
#pragma unroll
            for (int l = 0; l < 4; ++l) pe[l] = sgd_one(gm[u][q * 4 + l], pe[l], &me[l], p);
            __stcs(pv + q, pw[j][u][q]);
            if (p.has_mom) __stcs(mv + q, mw[j][u][q]);
          }
        }
  }
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    sgd_scalar<F16>(p, s_g, s_p, s_m, e, inner, groups, rh);
  }
}

// ---------------------------------------------------------------------------
// The staged pass for small items.  With a small buffer the register pass
// above is a chain of dependent round trips per CTA: the fold's batches of
// ranks, then the update's parameter and momentum loads, rank after rank.
// Here the CTA loads every rank's gradient tile, parameter and momentum
// columns of its item into shared memory at once (one round trip, all threads
// issuing loads), folds each row group of the schedule (a thread per group and
// column), folds the group totals (a thread per column) -- or, for a single
// group, takes its fold as the result -- and then updates every rank's
// parameters and momenta from shared memory, all threads at once.  The adds,
// their order and roundings, the scale, the storage rounding of the gradient
// and the update (sgd_one) are those of the register pass.
// Shared memory: P x tile gradient bytes, P x tile x (4 / esize) parameter and
// as many momentum bytes, the group totals and the result in binary32 as
// 16-byte slices (row g * Q + q, a column per 16 bytes), the result in storage
// form (16 bytes per column).
// ---------------------------------------------------------------------------
__host__ __device__ constexpr uint32_t sgd_lat_smem_bytes(uint32_t P, uint32_t groups, uint32_t tile, uint32_t q) {
  return P * tile + 2u * P * tile * q + groups * tile * q + tile * q + tile;
}

template <bool F16, bool SINGLE>
__global__ void __launch_bounds__(kThreads) fold_sgd_lat_kernel(const __grid_constant__ SgdParams p) {
  constexpr int L = F16 ? 8 : 4;  // gradient elements per 16-byte column
  constexpr int Q = L / 4;        // 16-byte binary32 vectors per column of parameters
  extern __shared__ __align__(16) unsigned char s_sgd[];
  __shared__ char* s_g[kMaxPSgd];
  __shared__ float* s_p[kMaxPSgd];
  __shared__ float* s_m[kMaxPSgd];
  asm volatile("griddepcontrol.launch_dependents;");
  const Item s_item = p.items[p.item0 + blockIdx.x];
  const uint64_t off = (uint64_t)s_item.seg * (uint64_t)p.P;
  if (!(s_item.seg < p.n_segs && off + (uint64_t)p.P <= p.n_orders)) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadItem);
    return;
  }
  for (int t = threadIdx.x; t < p.P; t += kThreads) {
    unsigned r = p.orders[off + t];
    r = r < (unsigned)p.P ? r : 0;
    s_g[t] = static_cast<char*>(p.grads[r]);
    s_p[t] = p.params[r];
    s_m[t] = p.moms[r];
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int P = p.P, inner = p.inner, groups = p.groups;
  const bool rh = F16 && p.round_hops;
  const uint32_t T = p.tile_bytes, CT = T / 16u;
  const uint64_t eb = s_item.begin, ee = eb + s_item.len;
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;
  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads) sgd_scalar<F16>(p, s_g, s_p, s_m, e, inner, groups, rh);
    return;
  }
  const uint32_t ncols = (uint32_t)(ve - vb);  // <= T / 16
  unsigned char* s_grad = s_sgd;
  float4* s_par = reinterpret_cast<float4*>(s_sgd + (size_t)P * T);
  float4* s_mom = s_par + (size_t)P * CT * Q;
  float4* s_tot = s_mom + (size_t)P * CT * Q;
  float4* s_res = s_tot + (size_t)groups * CT * Q;
  uint4* s_st = reinterpret_cast<uint4*>(s_res + (size_t)CT * Q);

  // every rank's gradient column, parameters and momenta, all loads in flight
  for (uint32_t i = threadIdx.x; i < (uint32_t)P * ncols; i += kThreads) {
    const uint32_t t = i / ncols, c = i % ncols;
    *reinterpret_cast<uint4*>(s_grad + (size_t)t * T + c * 16u) =
        __ldcs(reinterpret_cast<const uint4*>(s_g[t]) + vb + c);
    const float4* pv = reinterpret_cast<const float4*>(s_p[t]) + (vb + c) * Q;
    const float4* mv = reinterpret_cast<const float4*>(s_m[t]) + (vb + c) * Q;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      s_par[((size_t)t * CT + c) * Q + q] = __ldcs(pv + q);
      if (p.has_mom) s_mom[((size_t)t * CT + c) * Q + q] = __ldcs(mv + q);
    }
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
      unpack<F16>(*reinterpret_cast<const uint4*>(s_grad + (size_t)t * T + c * 16u), f);
      if (h == 0) {
#pragma unroll
        for (int l = 0; l < L; ++l) a[l] = f[l];
      } else {
        const bool round = rh && !(t == P - 1 && groups == 1);  // the final add of one group is not
#pragma unroll
        for (int l = 0; l < L; ++l) {
          const float v = __fadd_rn(a[l], f[l]);
          a[l] = round ? round_h(v) : v;
        }
      }
    }
    if constexpr (SINGLE) {  // one group: its fold, scaled, is the gradient
#pragma unroll
      for (int l = 0; l < L; ++l) a[l] = __fmul_rn(a[l], p.scale);
      const uint4 st = pack<F16>(a);
      if (F16) unpack<F16>(st, a);  // the update reads the gradient as stored
      s_st[c] = st;
#pragma unroll
      for (int q = 0; q < Q; ++q) s_res[(size_t)q * CT + c] = make_float4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
    } else {
#pragma unroll
      for (int q = 0; q < Q; ++q)
        s_tot[((size_t)g * Q + q) * CT + c] = make_float4(a[4 * q], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
    }
  }
  __syncthreads();

  if constexpr (!SINGLE) {  // each column: the left fold of its group totals
    for (uint32_t c = threadIdx.x; c < ncols; c += kThreads) {
      float o[L];
#pragma unroll
      for (int q = 0; q < Q; ++q) {
        const float4 v = s_tot[(size_t)q * CT + c];
        o[4 * q] = v.x, o[4 * q + 1] = v.y, o[4 * q + 2] = v.z, o[4 * q + 3] = v.w;
      }
      for (int g = 1; g < groups; ++g) {
        const bool round = rh && g != groups - 1;  // the last group's add is the final one
        float t4[L];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const float4 v = s_tot[((size_t)g * Q + q) * CT + c];
          t4[4 * q] = v.x, t4[4 * q + 1] = v.y, t4[4 * q + 2] = v.z, t4[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int l = 0; l < L; ++l) {
          const float v = __fadd_rn(o[l], t4[l]);
          o[l] = round ? round_h(v) : v;
        }
      }
#pragma unroll
      for (int l = 0; l < L; ++l) o[l] = __fmul_rn(o[l], p.scale);
      const uint4 st = pack<F16>(o);
      if (F16) unpack<F16>(st, o);
      s_st[c] = st;
#pragma unroll
      for (int q = 0; q < Q; ++q) s_res[(size_t)q * CT + c] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
    __syncthreads();
  }

  // the update of every rank's parameters and momenta, and the gradient stores
  for (uint32_t i = threadIdx.x; i < (uint32_t)P * ncols * Q; i += kThreads) {
    const uint32_t t = i / (ncols * Q), r = i % (ncols * Q), c = r / Q, q = r % Q;
    const float4 g4 = s_res[(size_t)q * CT + c];
    float4 pw = s_par[((size_t)t * CT + c) * Q + q];
    float4 mw = p.has_mom ? s_mom[((size_t)t * CT + c) * Q + q] : make_float4(0.f, 0.f, 0.f, 0.f);
    const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
    float* pe = reinterpret_cast<float*>(&pw);
    float* me = reinterpret_cast<float*>(&mw);
#pragma unroll
    for (int l = 0; l < 4; ++l) pe[l] = sgd_one(gv[l], pe[l], &me[l], p);
    __stcs(reinterpret_cast<float4*>(s_p[t]) + (vb + c) * Q + q, pw);
    if (p.has_mom) __stcs(reinterpret_cast<float4*>(s_m[t]) + (vb + c) * Q + q, mw);
    if (p.keep_grads && q == 0) __stcs(reinterpret_cast<uint4*>(s_g[t]) + vb + c, s_st[c]);
  }
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    sgd_scalar<F16>(p, s_g, s_p, s_m, e, inner, groups, rh);
  }
}

#ifndef DDL_SGD_LAT_MAX_TILE
#define DDL_SGD_LAT_MAX_TILE 1024
#endif
constexpr uint32_t kSgdLatMaxSmem = 96u * 1024u;

// The opt-in above 48 KB of shared memory, once per kernel and device.
cudaError_t sgd_smem_opt_in(void (*kernel)(SgdParams), std::atomic<bool>* ready) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!ready[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSgdLatMaxSmem);
    if (e != cudaSuccess) return e;
    ready[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

}  // namespace

// One CTA per work item, launched as a programmatic dependent of the kernel
// before it on the stream: its table prologue overlaps that kernel's tail.
// Small items (up to DDL_SGD_LAT_MAX_TILE bytes per rank) whose ranks'
// gradients, parameters and momenta fit in 96 KB of shared memory take the
// staged pass.
cudaError_t launch_sgd(const SgdParams& p, uint32_t n_items, bool f16, cudaStream_t stream) {
  if (n_items == 0) return cudaSuccess;
  uint32_t smem = 0;
  void (*kernel)(SgdParams) = nullptr;
  if (p.vector_ok && p.tile_bytes <= (uint32_t)DDL_SGD_LAT_MAX_TILE && p.tile_bytes % 16u == 0 && p.groups >= 1 &&
      p.inner >= 1 && (int64_t)p.inner * p.groups == p.P) {
    smem = sgd_lat_smem_bytes((uint32_t)p.P, (uint32_t)p.groups, p.tile_bytes, f16 ? 2u : 1u);
    if (smem <= kSgdLatMaxSmem) {
      static std::atomic<bool> ready[2][2][64];
      const bool single = p.groups == 1;
      kernel = f16 ? (single ? fold_sgd_lat_kernel<true, true> : fold_sgd_lat_kernel<true, false>)
                   : (single ? fold_sgd_lat_kernel<false, true> : fold_sgd_lat_kernel<false, false>);
      const cudaError_t e = sgd_smem_opt_in(kernel, ready[f16 ? 1 : 0][single ? 1 : 0]);
      if (e != cudaSuccess) return e;
    }
  }
  if (!kernel) {
    smem = 0;
    kernel = f16 && p.round_hops ? fold_sgd_kernel<true, true>
             : f16               ? fold_sgd_kernel<true, false>
                                 : fold_sgd_kernel<false, false>;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace ddl
