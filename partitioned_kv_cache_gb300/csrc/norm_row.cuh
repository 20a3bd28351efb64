// norm_row.cuh -- one AdaRMSNorm row by one warp (device code).
//
// "Reflex: Real-Time VLA Control through Streaming Inference", §III "Core
// formulas", Eq. (2) and §V "Key implementation": y = x * rsqrt(mean(x^2) +
// eps) * gamma, with the mean of squares accumulated in fp32.  The row is
// read and written as 16-byte vectors of eight bf16; lane l takes vectors
// l, l + 32, ...  and the lanes' partial sums meet by shuffles.  Both the
// standalone norm kernel and the attention launch that runs norm rows beside
// its key loop use this routine, so their outputs are the same bits.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace rx {

__device__ __forceinline__ void norm_unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t norm_pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float norm_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint4 norm_scale8(const uint4& xv, float r, const float4& g0, const float4& g1) {
  float f[8];
  norm_unpack8(xv, f);
  return make_uint4(norm_pack2(f[0] * r * g0.x, f[1] * r * g0.y), norm_pack2(f[2] * r * g0.z, f[3] * r * g0.w),
                    norm_pack2(f[4] * r * g1.x, f[5] * r * g1.y), norm_pack2(f[6] * r * g1.z, f[7] * r * g1.w));
}

// One row of nv = d/8 vectors; every lane of the warp calls it.  MAXV > 0:
// the row (nv <= 32 * MAXV) and its gamma slice are loaded together into
// registers, one round trip; MAXV = 0: any width, the row read twice (the
// second pass mostly from L1).  Both sum a lane's squares in the same order
// (vector by vector, element by element), so the result does not depend on
// which form ran.
template <int MAXV>
__device__ __forceinline__ void adarmsnorm_row(const uint4* __restrict__ xr, const float* __restrict__ gamma,
                                               int nv, float inv_d, float eps, uint4* __restrict__ yr, int lane) {
  if constexpr (MAXV > 0) {
    uint4 xv[MAXV];
    float4 g0[MAXV], g1[MAXV];
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int v = lane + 32 * u;
      if (v < nv) {
        xv[u] = xr[v];
        g0[u] = *reinterpret_cast<const float4*>(gamma + 8 * v);
        g1[u] = *reinterpret_cast<const float4*>(gamma + 8 * v + 4);
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      if (lane + 32 * u < nv) {
        float f[8];
        norm_unpack8(xv[u], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
      }
    }
    const float r = rsqrtf(norm_warp_sum(ss) * inv_d + eps);
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int v = lane + 32 * u;
      if (v < nv) yr[v] = norm_scale8(xv[u], r, g0[u], g1[u]);
    }
  } else {
    float ss = 0.f;
    for (int v = lane; v < nv; v += 32) {
      float f[8];
      norm_unpack8(xr[v], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
    const float r = rsqrtf(norm_warp_sum(ss) * inv_d + eps);
    for (int v = lane; v < nv; v += 32) {
      const float4 g0 = *reinterpret_cast<const float4*>(gamma + 8 * v);
      const float4 g1 = *reinterpret_cast<const float4*>(gamma + 8 * v + 4);
      yr[v] = norm_scale8(xr[v], r, g0, g1);
    }
  }
}

}  // namespace rx
