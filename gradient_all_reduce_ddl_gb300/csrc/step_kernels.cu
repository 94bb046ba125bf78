// step_kernels.cu -- the step-by-step schedule, one kernel per communication
// step (DDL_MODE_STEPWISE).
//
// Each launch carries every message of one step of the ring, multi-ring or
// torus schedule (Baidu write-up "总结"; "[论文解读] PowerAI DDL";
// Sony page "2D-Torus All-reduce"): the receiver adds the sender's chunk into
// its own copy (reduce-scatter) or overwrites it (all-gather).  The values are
// stored in the buffers' own type after every step, so binary16 rounding at
// every hop is inherent; the owner's last add is scaled before it is stored.
// Within one step no message reads a range another message writes, so all of
// a step's messages run concurrently in place.  This mode moves about
// 5(P-1)N elements through HBM instead of the fused pass's 2PN; it exists to
// show what fusing the steps saves and as a second GPU witness of the
// schedule's result.
#include <cuda_fp16.h>

#include "kernels.h"

namespace ddl {
namespace {

constexpr int kThreads = 256;

template <bool F16>
__device__ __forceinline__ float ld1(const char* b, uint64_t e) {
  if constexpr (F16) return __half2float(__ushort_as_half(reinterpret_cast<const unsigned short*>(b)[e]));
  else return reinterpret_cast<const float*>(b)[e];
}
template <bool F16>
__device__ __forceinline__ void st1(char* b, uint64_t e, float v) {
  if constexpr (F16) reinterpret_cast<unsigned short*>(b)[e] = __half_as_ushort(__float2half_rn(v));
  else reinterpret_cast<float*>(b)[e] = v;
}

template <bool F16>
__device__ __forceinline__ void op_elem(const Xfer& x, const char* src, char* dst, uint64_t e, float scale) {
  if (x.op == kCopy) {
    if constexpr (F16) reinterpret_cast<unsigned short*>(dst)[e] = reinterpret_cast<const unsigned short*>(src)[e];
    else reinterpret_cast<float*>(dst)[e] = reinterpret_cast<const float*>(src)[e];
    return;
  }
  const float d = ld1<F16>(dst, e);
  float v;
  if (x.op == kScaleOnly) {
    v = __fmul_rn(d, scale);
  } else {
    v = __fadd_rn(ld1<F16>(src, e), d);
    if (x.op == kAddFinal) v = __fmul_rn(v, scale);
  }
  st1<F16>(dst, e, v);
}

// One 16-byte column of a message: the receiver's value dr and the sender's sr
// (loaded by the caller) give the value the receiver stores.
template <bool F16>
__device__ __forceinline__ uint4 op_vec(const Xfer& x, const uint4 dr, const uint4 sr, float scale) {
  if (x.op == kCopy) return sr;
  const uint32_t dw[4] = {dr.x, dr.y, dr.z, dr.w}, sw[4] = {sr.x, sr.y, sr.z, sr.w};
  uint32_t ow[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (F16) {
      uint32_t o = 0;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float d = __half2float(__ushort_as_half((unsigned short)(dw[i] >> (16 * half))));
        const float s = __half2float(__ushort_as_half((unsigned short)(sw[i] >> (16 * half))));
        float v = (x.op == kScaleOnly) ? __fmul_rn(d, scale) : __fadd_rn(s, d);
        if (x.op == kAddFinal) v = __fmul_rn(v, scale);
        o |= (uint32_t)__half_as_ushort(__float2half_rn(v)) << (16 * half);
      }
      ow[i] = o;
    } else {
      const float d = __uint_as_float(dw[i]), s = __uint_as_float(sw[i]);
      float v = (x.op == kScaleOnly) ? __fmul_rn(d, scale) : __fadd_rn(s, d);
      if (x.op == kAddFinal) v = __fmul_rn(v, scale);
      ow[i] = __float_as_uint(v);
    }
  }
  return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// grid.x: tiles of kTileBytes over the step's longest message; grid.y: message.
// Launched as a programmatic dependent of the step before it: a CTA reads its
// message from the plan's table, then waits for that step (finished, writes
// visible) before touching a buffer.
template <bool F16>
__global__ void __launch_bounds__(kThreads) step_kernel(const __grid_constant__ StepParams p) {
  constexpr int L = F16 ? 8 : 4;
  constexpr uint64_t kTile = (uint64_t)kTileBytes / (F16 ? 2 : 4);
  asm volatile("griddepcontrol.launch_dependents;");
  const Xfer x = p.xfers[p.xfer0 + blockIdx.y];
  const uint64_t off = (uint64_t)blockIdx.x * kTile;
  if (off >= x.len) return;
  if (x.src >= p.P || x.dst >= p.P) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrBadXfer);
    return;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const char* src = static_cast<const char*>(p.bufs[x.src]);
  char* dst = static_cast<char*>(p.bufs[x.dst]);
  const uint64_t eb = x.lo + off, ee = x.lo + (x.len < off + kTile ? x.len : off + kTile);
  const uint64_t vb = (eb + L - 1) / L, ve = ee / L;
  if (!p.vector_ok || vb >= ve) {
    for (uint64_t e = eb + threadIdx.x; e < ee; e += kThreads) op_elem<F16>(x, src, dst, e, p.scale);
    return;
  }
  // two columns per thread per round: all four loads issued before any store
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  const bool need_dst = x.op != kCopy, need_src = x.op != kScaleOnly;
  for (uint64_t c0 = vb + threadIdx.x; c0 < ve; c0 += 2 * kThreads) {
    const uint64_t c1 = c0 + kThreads;
    const bool two = c1 < ve;
    const uint4 z = make_uint4(0, 0, 0, 0);
    const uint4 d0 = need_dst ? d4[c0] : z, s0 = need_src ? s4[c0] : z;
    const uint4 d1 = (two && need_dst) ? d4[c1] : z, s1 = (two && need_src) ? s4[c1] : z;
    d4[c0] = op_vec<F16>(x, d0, need_src ? s0 : d0, p.scale);
    if (two) d4[c1] = op_vec<F16>(x, d1, need_src ? s1 : d1, p.scale);
  }
  const uint64_t nh = vb * L - eb, nt = ee - ve * L;
  if (threadIdx.x < nh + nt) {
    const uint64_t e = threadIdx.x < nh ? eb + threadIdx.x : ve * L + (threadIdx.x - nh);
    op_elem<F16>(x, src, dst, e, p.scale);
  }
}

}  // namespace

cudaError_t launch_step(const StepParams& p, uint32_t n_xfers, uint64_t max_len, bool f16, cudaStream_t stream,
                        bool early_launch) {
  if (n_xfers == 0 || max_len == 0) return cudaSuccess;
  const uint64_t tile = (uint64_t)kTileBytes / (f16 ? 2 : 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((max_len + tile - 1) / tile), n_xfers);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early_launch ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, f16 ? step_kernel<true> : step_kernel<false>, p);
}

}  // namespace ddl
