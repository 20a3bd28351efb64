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
// front, with its second layer on the tensor cores; the norm itself is one
// warp per row with 16-byte bf16 vectors.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "norm_row.cuh"
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

// SM count of device `dev`, queried once per device.
cudaError_t device_sm_count(int dev, int* out) {
  static std::atomic<int> cache[64];
  const bool cached = dev >= 0 && dev < 64;
  if (cached && (*out = cache[dev].load(std::memory_order_relaxed)) > 0) return cudaSuccess;
  const cudaError_t e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && cached) cache[dev].store(*out, std::memory_order_relaxed);
  return e;
}

// One warp per row (adarmsnorm_row).  MAXV = 16-byte vectors per lane kept
// in registers (d <= 256 * MAXV); MAXV = 0 selects the two-pass path for
// wider rows.
template <int MAXV>
__global__ void __launch_bounds__(256) adarmsnorm_kernel(const uint4* __restrict__ x,
                                                         const float* __restrict__ gamma,
                                                         int rows, int d, float eps,
                                                         uint4* __restrict__ y, int prefetch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + warp;
  const int nv = d >> 3;
  // A launch that fits on the GPU at once fetches its rows and gamma towards
  // L2 while the previous kernel finishes (a hint: safe before the dependency
  // wait), so the loads below do not pay the DRAM latency inside the launch
  // chain.  Larger launches skip it: their later CTAs start long after the
  // wait, and the extra requests only cost bandwidth.
  if (prefetch) {
    if (lane == 0 && row < rows) bulk_prefetch_l2(x + row * nv, static_cast<uint32_t>(d) * 2u);
    if (threadIdx.x == 32 * 7 + 1) bulk_prefetch_l2(gamma, static_cast<uint32_t>(d) * 4u);
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (row >= rows) return;
  adarmsnorm_row<MAXV>(x + row * nv, gamma, nv, 1.0f / static_cast<float>(d), eps, y + row * nv, lane);
}

// ---------------------------------------------------------------- gamma MLP
// The first layer and the SiLU run on the CUDA cores in fp32 (each CTA
// recomputes h for its weight set: 16K multiply-adds per vector).  The second
// layer runs on the tensor cores: per weight set, W2 [d x hidden] times H^T,
// where the rows of H are the hidden activations of the conditioning vectors.
// One CTA computes 128 rows of W2 against every vector (tcgen05 M = 128,
// N = 32, K = hidden).  h enters the MMA as two bf16 rows per vector,
// hi = bf16(h) and lo = bf16(h - hi), so the product keeps ~16 bits of h with
// an fp32 accumulator: rows 0..15 of the B operand are the hi parts, rows
// 16..31 the lo parts, and gamma = 1 + D[:, k] + D[:, 16 + k] + b2.  W2 streams through a
// four-slot ring of 64-column blocks (16 KB, 128-byte swizzle) by TMA; the
// blocks beyond the ring are prefetched into L2 at the start, so that their
// loads, which wait for the ring, come from L2.
constexpr int kGM = 128;                 // W2 rows per CTA (MMA M)
constexpr int kGN = 32;                  // B rows: 16 hi + 16 lo (MMA N)
constexpr int kGSlots = 4;               // W2 K-block ring
constexpr int kGBlock = kGM * 128;       // one 64-column block of W2 rows: 16 KB
constexpr int kGHBlock = kGN * 128;      // one 64-column block of H: 4 KB
constexpr int kGThreads = 256;

struct GammaArgs {
  CUtensorMap tm_w2;   // (hidden, d, n_sets, 1) bf16, box (64, 128, 1, 1), 128-byte swizzle
  const float* t;
  const float* state;
  const __nv_bfloat16* W1;
  const __nv_bfloat16* b1;
  const __nv_bfloat16* b2;
  float* gamma;
  int n_cond, emb_dim, state_dim, hidden, d;
};

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// h of hidden unit j for vector k -> rows k (hi) and 16 + k (lo) of the H
// operand tile, in the swizzled K-major layout (row n of 64-column block kb:
// 128 bytes at n * 128, 16-byte chunk q at position q ^ (n & 7)).
__device__ __forceinline__ void store_h(uint32_t sH, int j, int k, float hv) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(hv);
  const __nv_bfloat16 lo = __float2bfloat16_rn(hv - __bfloat162float(hi));
  const uint32_t col = sH + (j >> 6) * kGHBlock + (j & 7) * 2;
  const int q = (j & 63) >> 3;
  const int n_hi = k, n_lo = 16 + k;
  st_shared_u16(col + n_hi * 128 + ((q ^ (n_hi & 7)) << 4), *reinterpret_cast<const uint16_t*>(&hi));
  st_shared_u16(col + n_lo * 128 + ((q ^ (n_lo & 7)) << 4), *reinterpret_cast<const uint16_t*>(&lo));
}

// Shared layout (1024-byte aligned base): ring [kGSlots][16 KB] | H [hidden/64][4 KB]
// | c [n_cond][c_stride] fp32 | barriers full[kGSlots], empty[kGSlots], done | TMEM slot.
__global__ void __launch_bounds__(kGThreads, 1) ada_gamma_kernel(const __grid_constant__ GammaArgs a) {
  extern __shared__ uint8_t gsm_raw[];
  const uint32_t raw = smem_u32(gsm_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = gsm_raw + (base - raw);
  const int nkb = (a.hidden + 63) / 64;
  const int cond_dim = a.emb_dim + a.state_dim;
  const int c_stride = (cond_dim + 3) & ~3;
  const uint32_t sRing = base;
  const uint32_t sH = base + kGSlots * kGBlock;
  float* c = reinterpret_cast<float*>(gbase + kGSlots * kGBlock + nkb * kGHBlock);
  const uint32_t off_bar = (kGSlots * kGBlock + nkb * kGHBlock + a.n_cond * c_stride * 4 + 7) & ~7;
  const uint32_t sBar = base + off_bar;
  auto FULL = [&](int i) { return sBar + 8u * i; };
  auto EMPTY = [&](int i) { return sBar + 8u * (kGSlots + i); };
  const uint32_t DONE = sBar + 8u * (2 * kGSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + off_bar + 8 * (2 * kGSlots + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + off_bar + 8 * (2 * kGSlots + 1) + 4);
  const int tile = blockIdx.x, set = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGSlots; ++i) {
      mbar_init(FULL(i), 1);
      mbar_init(EMPTY(i), 1);
    }
    mbar_init(DONE, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&a.tm_w2);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dependency_wait();
  grid_launch_dependents();

  // The small inputs are requested before W2: the 1 MB per set of W2 fills
  // the DRAM queues for microseconds, and anything requested behind it waits
  // that long.  This thread's first kPreRows rows of W1 and b1, its output
  // row's b2 and its share of t and state go first; the common shapes
  // (hidden <= 512, cond width <= 32, n_cond * cond width <= 512) need no
  // other load before the MMAs.
  constexpr int kPreRows = 2;
  const __nv_bfloat16* W1s = a.W1 + static_cast<size_t>(set) * a.hidden * cond_dim;
  const __nv_bfloat16* b1s = a.b1 + static_cast<size_t>(set) * a.hidden;
  const bool w1_fast = (cond_dim & 7) == 0 && cond_dim <= 32 && (reinterpret_cast<uintptr_t>(W1s) & 15) == 0;
  // (kept as raw bf16 until used: converting at the load would wait for it)
  uint4 w1v[kPreRows][4];
  __nv_bfloat16 b1v[kPreRows];
  const int i_out = tile * kGM + (warp & 3) * 32 + lane;   // this thread's output row (epilogue)
  const __nv_bfloat16 b2v = a.b2[static_cast<size_t>(set) * a.d + (i_out < a.d ? i_out : a.d - 1)];
#pragma unroll
  for (int r = 0; r < kPreRows; ++r) {
    const int j = threadIdx.x + r * kGThreads;
    b1v[r] = __float2bfloat16_rn(0.f);
    if (w1_fast && j < a.hidden) {
      const uint4* src = reinterpret_cast<const uint4*>(W1s + static_cast<size_t>(j) * cond_dim);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (8 * u < cond_dim) w1v[r][u] = __ldg(src + u);
      b1v[r] = b1s[j];
    }
  }

  // c_k = [sin(t_k w_j), cos(t_k w_j), state_k],  w_j = 10000^(-j/half):
  // element idx of c reads t[k] (embedding) or one state value.
  constexpr int kPreC = 2;
  float cin[kPreC];
#pragma unroll
  for (int r = 0; r < kPreC; ++r) {
    const int idx = threadIdx.x + r * kGThreads;
    cin[r] = 0.f;
    if (idx < a.n_cond * cond_dim) {
      const int k = idx / cond_dim, j = idx - k * cond_dim;
      cin[r] = j < a.emb_dim ? a.t[k] : a.state[k * a.state_dim + (j - a.emb_dim)];
    }
  }
  __syncthreads();   // every small load is out before W2 is requested
  // W2 blocks 0..kGSlots-1 go out first, the rest to L2; h is computed while
  // they land.
  int issued = 0;
  if (threadIdx.x == 0) {
    for (; issued < kGSlots && issued < nkb; ++issued) {
      mbar_arrive_expect_tx(FULL(issued), kGBlock);
      tma_load_4d(sRing + issued * kGBlock, &a.tm_w2, issued * 64, tile * kGM, set, 0, FULL(issued));
    }
    for (int b = kGSlots; b < nkb; ++b) tma_prefetch_l2_4d(&a.tm_w2, b * 64, tile * kGM, set, 0);
  }

  const int half = a.emb_dim / 2;
  auto c_elem = [&](int idx, float in) {
    const int k = idx / cond_dim, j = idx - k * cond_dim;
    float v = in;
    if (j < a.emb_dim) {
      const int jj = j < half ? j : j - half;
      const float w = powf(10000.0f, -static_cast<float>(jj) / static_cast<float>(half));
      v = j < half ? sinf(in * w) : cosf(in * w);
    }
    c[k * c_stride + j] = v;
  };
#pragma unroll
  for (int r = 0; r < kPreC; ++r)
    if (threadIdx.x + r * kGThreads < a.n_cond * cond_dim) c_elem(threadIdx.x + r * kGThreads, cin[r]);
  for (int idx = threadIdx.x + kPreC * kGThreads; idx < a.n_cond * cond_dim; idx += blockDim.x) {
    const int k = idx / cond_dim, j = idx - k * cond_dim;
    c_elem(idx, j < a.emb_dim ? a.t[k] : a.state[k * a.state_dim + (j - a.emb_dim)]);
  }
  // H starts as zeros: unused vectors, and columns past hidden in the last block.
  for (int o = threadIdx.x * 16; o < nkb * kGHBlock; o += blockDim.x * 16)
    st_shared_v4(sH + o, 0u, 0u, 0u, 0u);
  __syncthreads();

  // h_k = SiLU(W1 c_k + b1) in fp32, stored as hi / lo bf16 rows of H.
  int j_rest = 0;   // first row not covered by the preloaded ones
  if (w1_fast) {
#pragma unroll
    for (int r = 0; r < kPreRows; ++r) {
      const int j = threadIdx.x + r * kGThreads;
      if (j < a.hidden) {
        float acc[kMaxCond];
#pragma unroll
        for (int k = 0; k < kMaxCond; ++k) acc[k] = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (8 * u < cond_dim) {
            float w[8];
            unpack8(w1v[r][u], w);
#pragma unroll
            for (int k = 0; k < kMaxCond; ++k) {
              if (k < a.n_cond) {
                const float4 c0 = *reinterpret_cast<const float4*>(c + k * c_stride + 8 * u);
                const float4 c1 = *reinterpret_cast<const float4*>(c + k * c_stride + 8 * u + 4);
                acc[k] = fmaf(w[0], c0.x, fmaf(w[1], c0.y, fmaf(w[2], c0.z, fmaf(w[3], c0.w, acc[k]))));
                acc[k] = fmaf(w[4], c1.x, fmaf(w[5], c1.y, fmaf(w[6], c1.z, fmaf(w[7], c1.w, acc[k]))));
              }
            }
          }
        }
#pragma unroll
        for (int k = 0; k < kMaxCond; ++k) {
          if (k < a.n_cond) {
            const float z = acc[k] + __bfloat162float(b1v[r]);
            store_h(sH, j, k, __fdividef(z, 1.0f + __expf(-z)));
          }
        }
      }
    }
    j_rest = kPreRows * kGThreads;
  }
  for (int j = j_rest + threadIdx.x; j < a.hidden; j += blockDim.x) {   // wider shapes
    float acc[kMaxCond];
#pragma unroll
    for (int k = 0; k < kMaxCond; ++k) acc[k] = 0.f;
    const __nv_bfloat16* wr = W1s + static_cast<size_t>(j) * cond_dim;
    for (int e = 0; e < cond_dim; ++e) {
      const float w = __bfloat162float(wr[e]);
#pragma unroll
      for (int k = 0; k < kMaxCond; ++k)
        if (k < a.n_cond) acc[k] = fmaf(w, c[k * c_stride + e], acc[k]);
    }
    const float bias = __bfloat162float(b1s[j]);
#pragma unroll
    for (int k = 0; k < kMaxCond; ++k) {
      if (k < a.n_cond) {
        const float z = acc[k] + bias;
        store_h(sH, j, k, __fdividef(z, 1.0f + __expf(-z)));
      }
    }
  }
  fence_proxy_async_smem();   // H (generic-proxy stores) -> tensor-core reads
  __syncthreads();

  if (threadIdx.x == 0) {
    // D = W2_tile . H^T over the hidden blocks; block kb + kGSlots reuses the
    // slot once the MMAs of block kb have read it.
    constexpr uint32_t idesc = idesc_bf16_f32(kGM, kGN, false, false);
    bool ok = true;
    int kb = 0;
    for (; kb < nkb; ++kb) {
      const int slot = kb % kGSlots;
      const uint32_t ph = static_cast<uint32_t>(kb / kGSlots) & 1u;
      if (!mbar_wait(FULL(slot), ph, abort_flag)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = sdesc_sw128(sRing + slot * kGBlock + kk * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(sH + kb * kGHBlock + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(EMPTY(slot));
      if (kb + kGSlots < nkb) {
        if (!mbar_wait(EMPTY(slot), ph, abort_flag)) { ok = false; ++kb; break; }
        mbar_arrive_expect_tx(FULL(slot), kGBlock);
        tma_load_4d(sRing + slot * kGBlock, &a.tm_w2, (kb + kGSlots) * 64, tile * kGM, set, 0, FULL(slot));
        ++issued;
      }
    }
    umma_commit(DONE);   // every MMA issued above has completed when DONE fires
    if (!ok) {
      // every copy issued must land before the CTA exits
      volatile int no_abort = 0;
      for (int b = kb; b < issued; ++b) mbar_wait(FULL(b % kGSlots), static_cast<uint32_t>(b / kGSlots) & 1u, &no_abort);
    }
  }
  __syncwarp();
  volatile int no_abort = 0;
  mbar_wait(DONE, 0, &no_abort);
  tc_fence_after();

  // Epilogue: warps w and w + 4 hold rows 32(w % 4) .. +31 of the tile (TMEM
  // lane quarter w % 4) and store vectors [0, 8) and [8, 16) respectively.
  float v[32];
  tmem_ld32(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16), v);
  const int i = i_out;
  if (i < a.d) {
    const bool failed = *abort_flag != 0;
    const float bias = __bfloat162float(b2v);
    float* gi = a.gamma + static_cast<size_t>(set) * a.n_cond * a.d + i;
    const float nan = __int_as_float(0x7fc00000);
    if (warp < 4) {
#pragma unroll
      for (int k = 0; k < kMaxCond / 2; ++k)
        if (k < a.n_cond) gi[static_cast<size_t>(k) * a.d] = failed ? nan : 1.0f + v[k] + v[16 + k] + bias;
    } else {
#pragma unroll
      for (int k = kMaxCond / 2; k < kMaxCond; ++k)
        if (k < a.n_cond) gi[static_cast<size_t>(k) * a.d] = failed ? nan : 1.0f + v[k] + v[16 + k] + bias;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 32);
}

}  // namespace

cudaError_t launch_adarmsnorm(const __nv_bfloat16* x, const float* gamma, int rows, int d,
                              float eps, __nv_bfloat16* y, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const unsigned int blocks = static_cast<unsigned int>((rows + 7) / 8);
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* yv = reinterpret_cast<uint4*>(y);
  cudaError_t e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = device_sm_count(dev, &sms)) != cudaSuccess) return e;
  const int pf = blocks <= static_cast<unsigned int>(sms) ? 1 : 0;
  if (d <= 256)
    e = launch_k(adarmsnorm_kernel<1>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv, pf);
  else if (d <= 512)
    e = launch_k(adarmsnorm_kernel<2>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv, pf);
  else if (d <= 1024)
    e = launch_k(adarmsnorm_kernel<4>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv, pf);
  else if (d <= 2048)
    e = launch_k(adarmsnorm_kernel<8>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv, pf);
  else
    e = launch_k(adarmsnorm_kernel<0>, dim3(blocks), dim3(256), 0, s, xv, gamma, rows, d, eps, yv, pf);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_ada_gamma(const float* t, const float* state, int n_cond, int emb_dim,
                             int state_dim, const __nv_bfloat16* W1, const __nv_bfloat16* b1,
                             int hidden, const __nv_bfloat16* W2, const __nv_bfloat16* b2, int d,
                             int n_sets, float* gamma, cudaStream_t s) {
  GammaArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t dims[4] = {static_cast<uint64_t>(hidden), static_cast<uint64_t>(d),
                            static_cast<uint64_t>(n_sets), 1};
  const uint64_t strides[3] = {static_cast<uint64_t>(hidden) * 2, static_cast<uint64_t>(d) * hidden * 2,
                               static_cast<uint64_t>(n_sets) * d * hidden * 2};
  const uint32_t box[4] = {64u, static_cast<uint32_t>(kGM), 1u, 1u};
  if (!encode_tmap_4d(&a.tm_w2, W2, dims, strides, box)) return cudaErrorInvalidValue;
  a.t = t;
  a.state = state;
  a.W1 = W1;
  a.b1 = b1;
  a.b2 = b2;
  a.gamma = gamma;
  a.n_cond = n_cond;
  a.emb_dim = emb_dim;
  a.state_dim = state_dim;
  a.hidden = hidden;
  a.d = d;
  const int nkb = (hidden + 63) / 64;
  const size_t c_bytes = static_cast<size_t>(n_cond) * ((emb_dim + state_dim + 3) & ~3) * 4;
  const size_t smem = 1024 + static_cast<size_t>(kGSlots) * kGBlock + static_cast<size_t>(nkb) * kGHBlock +
                      ((c_bytes + 7) & ~size_t(7)) + 8 * (2 * kGSlots + 1) + 16;
  if (smem > 232448) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(ada_gamma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const dim3 grid((d + kGM - 1) / kGM, n_sets);
  e = launch_k(ada_gamma_kernel, grid, dim3(kGThreads), smem, s, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rx
