// adarmsnorm.cu -- AdaRMSNorm and its conditioning gate.
//
// "Reflex: Real-Time VLA Control through Streaming Inference", §III "Core
// formulas", Eq. (2):
//   AdaRMSNorm(x, c) = x / RMS(x) * gamma(c),  gamma(c) = 1 + MLP(c),
//   RMS(x) = sqrt(mean_i x_i^2 + eps)
// with c = [sinusoidal t_k; robot state s_t].  The mean of squares is taken in
// FP32 (the page's remedy for bf16 underflow); the MLP is
// Linear(cond -> hidden) -> SiLU -> Linear(hidden -> d) ("Model components"),
// run here with bf16 weights and fp32 arithmetic.
//
// gamma depends only on (t_k, s_t) and the site's weights, never on x, so one
// launch computes every (weight set, conditioning vector) pair of a tick up
// front; the norm itself is one warp per row with 16-byte bf16 vectors.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "rx_internal.h"
#include "sm103_ptx.cuh"

namespace rx {
namespace {

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per row.  MAXV = 16-byte vectors per lane kept in registers
// (d <= 256 * MAXV); MAXV = 0 selects the two-pass path for wider rows.
template <int MAXV>
__global__ void __launch_bounds__(256) adarmsnorm_kernel(const uint4* __restrict__ x,
                                                         const float* __restrict__ gamma,
                                                         int rows, int d, float eps,
                                                         uint4* __restrict__ y) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;
  if (row >= rows) return;
  const int nv = d >> 3;
  const uint4* xr = x + row * nv;
  uint4* yr = y + row * nv;
  const float inv_d = 1.0f / static_cast<float>(d);
  if constexpr (MAXV > 0) {
    // The row and its gamma slice are loaded together, so the gamma read is
    // not a second round trip after the reduction.
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
        unpack8(xv[u], f);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
      }
    }
    const float r = rsqrtf(warp_sum(ss) * inv_d + eps);
#pragma unroll
    for (int u = 0; u < MAXV; ++u) {
      const int v = lane + 32 * u;
      if (v < nv) {
        float f[8];
        unpack8(xv[u], f);
        yr[v] = make_uint4(pack2(f[0] * r * g0[u].x, f[1] * r * g0[u].y),
                           pack2(f[2] * r * g0[u].z, f[3] * r * g0[u].w),
                           pack2(f[4] * r * g1[u].x, f[5] * r * g1[u].y),
                           pack2(f[6] * r * g1[u].z, f[7] * r * g1[u].w));
      }
    }
  } else {
    float ss = 0.f;
    for (int v = lane; v < nv; v += 32) {
      float f[8];
      unpack8(xr[v], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
    const float r = rsqrtf(warp_sum(ss) * inv_d + eps);
    for (int v = lane; v < nv; v += 32) {
      float f[8];
      unpack8(xr[v], f);
      const float4 g0 = *reinterpret_cast<const float4*>(gamma + 8 * v);
      const float4 g1 = *reinterpret_cast<const float4*>(gamma + 8 * v + 4);
      yr[v] = make_uint4(pack2(f[0] * r * g0.x, f[1] * r * g0.y),
                         pack2(f[2] * r * g0.z, f[3] * r * g0.w),
                         pack2(f[4] * r * g1.x, f[5] * r * g1.y),
                         pack2(f[6] * r * g1.z, f[7] * r * g1.w));
    }
  }
}

constexpr int kGammaRows = 64;   // output rows of gamma per CTA

// grid (ceil(d / 64), n_sets), 256 threads.  Shared: c [n_cond][cond_dim] and
// the hidden activations h [n_cond][hidden].  Every CTA of a weight set
// recomputes h; W1 (hidden x cond_dim) is small and stays in L2.
__global__ void __launch_bounds__(256) ada_gamma_kernel(
    const float* __restrict__ t, const float* __restrict__ state, int n_cond, int emb_dim,
    int state_dim, const __nv_bfloat16* __restrict__ W1, const __nv_bfloat16* __restrict__ b1,
    int hidden, const __nv_bfloat16* __restrict__ W2, const __nv_bfloat16* __restrict__ b2,
    int d, float* __restrict__ gamma) {
  extern __shared__ float sh[];
  grid_dependency_wait();
  grid_launch_dependents();
  const int cond_dim = emb_dim + state_dim;
  float* c = sh;                        // [n_cond][cond_dim]
  float* h = sh + ((n_cond * cond_dim + 3) & ~3);   // [n_cond][hidden], 16-byte aligned
  const int set = blockIdx.y;
  const int half = emb_dim / 2;

  // c_k = [sin(t_k w_j), cos(t_k w_j), state_k],  w_j = 10000^(-j/half)
  for (int idx = threadIdx.x; idx < n_cond * cond_dim; idx += blockDim.x) {
    const int k = idx / cond_dim, j = idx - k * cond_dim;
    float v;
    if (j < emb_dim) {
      const int jj = j < half ? j : j - half;
      const float w = powf(10000.0f, -static_cast<float>(jj) / static_cast<float>(half));
      v = j < half ? sinf(t[k] * w) : cosf(t[k] * w);
    } else {
      v = state[k * state_dim + (j - emb_dim)];
    }
    c[idx] = v;
  }
  __syncthreads();

  // h_k = SiLU(W1 c_k + b1)
  const __nv_bfloat16* W1s = W1 + static_cast<size_t>(set) * hidden * cond_dim;
  const __nv_bfloat16* b1s = b1 + static_cast<size_t>(set) * hidden;
  for (int j = threadIdx.x; j < hidden; j += blockDim.x) {
    float acc[kMaxCond];
#pragma unroll
    for (int k = 0; k < kMaxCond; ++k) acc[k] = 0.f;
    const __nv_bfloat16* wr = W1s + static_cast<size_t>(j) * cond_dim;
    int e0 = 0;
    if ((cond_dim & 7) == 0 && (reinterpret_cast<uintptr_t>(W1s) & 15) == 0) {
      // 16-byte rows: 8 weights per load, four loads in flight
      const uint4* w4 = reinterpret_cast<const uint4*>(wr);
      for (; e0 + 32 <= cond_dim; e0 += 32) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = w4[e0 / 8 + u];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float w[8];
          unpack8(v[u], w);
#pragma unroll
          for (int x = 0; x < 8; ++x)
#pragma unroll
            for (int k = 0; k < kMaxCond; ++k)
              if (k < n_cond) acc[k] = fmaf(w[x], c[k * cond_dim + e0 + 8 * u + x], acc[k]);
        }
      }
    }
    for (int e = e0; e < cond_dim; ++e) {
      const float w = __bfloat162float(wr[e]);
#pragma unroll
      for (int k = 0; k < kMaxCond; ++k)
        if (k < n_cond) acc[k] = fmaf(w, c[k * cond_dim + e], acc[k]);
    }
    const float bias = __bfloat162float(b1s[j]);
#pragma unroll
    for (int k = 0; k < kMaxCond; ++k) {
      if (k < n_cond) {
        const float z = acc[k] + bias;
        h[k * hidden + j] = z / (1.0f + expf(-z));
      }
    }
  }
  __syncthreads();

  // gamma_k[i] = 1 + W2[i] . h_k + b2[i].  Four threads per output row; thread
  // q of a row takes hidden columns {16t + 4q .. 16t + 4q + 3}, so the four
  // threads of a row read 64 contiguous bytes of h (shared by the warp's 8
  // rows: one conflict-free wavefront) and 32 contiguous bytes of W2.
  const int q = threadIdx.x & 3;
  const int i = blockIdx.x * kGammaRows + (threadIdx.x >> 2);
  const __nv_bfloat16* W2s = W2 + static_cast<size_t>(set) * d * hidden;
  const __nv_bfloat16* b2s = b2 + static_cast<size_t>(set) * d;
  float acc[kMaxCond];
#pragma unroll
  for (int k = 0; k < kMaxCond; ++k) acc[k] = 0.f;
  const int ir = i < d ? i : d - 1;   // rows past d compute a duplicate and are not stored
  const uint2* wr = reinterpret_cast<const uint2*>(W2s + static_cast<size_t>(ir) * hidden);
#pragma unroll 8
  for (int t = 0; t < hidden / 16; ++t) {
    const int j = 16 * t + 4 * q;
    const uint2 wv = wr[j >> 2];
    const float w0 = __uint_as_float(wv.x << 16), w1 = __uint_as_float(wv.x & 0xFFFF0000u);
    const float w2 = __uint_as_float(wv.y << 16), w3 = __uint_as_float(wv.y & 0xFFFF0000u);
#pragma unroll
    for (int k = 0; k < kMaxCond; ++k) {
      if (k < n_cond) {
        const float4 hv = *reinterpret_cast<const float4*>(h + k * hidden + j);
        acc[k] = fmaf(w0, hv.x, fmaf(w1, hv.y, fmaf(w2, hv.z, fmaf(w3, hv.w, acc[k]))));
      }
    }
  }
  const float bias = __bfloat162float(b2s[ir]);
#pragma unroll
  for (int k = 0; k < kMaxCond; ++k) {
    if (k < n_cond) {
      float v = acc[k];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      if (q == 0 && i < d) gamma[(static_cast<size_t>(set) * n_cond + k) * d + i] = 1.0f + v + bias;
    }
  }
}

}  // namespace

cudaError_t launch_adarmsnorm(const __nv_bfloat16* x, const float* gamma, int rows, int d,
                              float eps, __nv_bfloat16* y, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const unsigned int blocks = static_cast<unsigned int>((rows + 7) / 8);
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* yv = reinterpret_cast<uint4*>(y);
  cudaError_t e;
  if (d <= 256)
    e = launch_k(adarmsnorm_kernel<1>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv);
  else if (d <= 512)
    e = launch_k(adarmsnorm_kernel<2>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv);
  else if (d <= 1024)
    e = launch_k(adarmsnorm_kernel<4>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv);
  else if (d <= 2048)
    e = launch_k(adarmsnorm_kernel<8>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv);
  else
    e = launch_k(adarmsnorm_kernel<0>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_ada_gamma(const float* t, const float* state, int n_cond, int emb_dim,
                             int state_dim, const __nv_bfloat16* W1, const __nv_bfloat16* b1,
                             int hidden, const __nv_bfloat16* W2, const __nv_bfloat16* b2, int d,
                             int n_sets, float* gamma, cudaStream_t s) {
  const size_t c_floats = (static_cast<size_t>(n_cond) * (emb_dim + state_dim) + 3) & ~size_t(3);
  const size_t smem = (c_floats + static_cast<size_t>(n_cond) * hidden) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(ada_gamma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid((d + kGammaRows - 1) / kGammaRows, n_sets);
  const cudaError_t e = launch_k(ada_gamma_kernel, grid, dim3(256), smem, s, t, state, n_cond,
                                 emb_dim, state_dim, W1, b1, hidden, W2, b2, d, gamma);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rx
