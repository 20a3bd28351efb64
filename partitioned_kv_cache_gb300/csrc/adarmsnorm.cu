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
// The first layer and the SiLU run on the CUDA cores in fp32, shared out over
// the cluster of the weight set's row tiles (each CTA computes 1/8 of h and
// copies it into its peers' shared memory).  The second
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
  int cluster;         // CTAs of one weight set (row tiles) that share the first layer
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
  // No early release of the next kernel (griddepcontrol.launch_dependents):
  // as with the ring append, an attention chain released early behind a
  // launch that holds the SMs' shared memory ran ~1 us slower per launch.
  grid_dependency_wait();

  // The first layer is shared out over the cluster of the weight set's row
  // tiles: CTA `crank` of `csize` computes the 64-unit blocks kb of h with
  // kb % csize == crank and copies each into its peers' H operand, so each
  // CTA computes 1/csize of the layer instead of all of it.  Within a block,
  // thread t takes unit kb * 64 + (t % 64) and the vectors k = t / 64 + 4i.
  const int crank = a.cluster > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int csize = a.cluster;
  // Peers write into this CTA's shared memory below; the matching wait
  // (before those writes) guarantees every CTA of the cluster has started.
  if (csize > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const int ju = threadIdx.x & 63, kq = threadIdx.x >> 6;
  const __nv_bfloat16* W1s = a.W1 + static_cast<size_t>(set) * a.hidden * cond_dim;
  const __nv_bfloat16* b1s = a.b1 + static_cast<size_t>(set) * a.hidden;
  const bool w1_fast = (cond_dim & 7) == 0 && cond_dim <= 32 && (reinterpret_cast<uintptr_t>(W1s) & 15) == 0;

  // The small inputs are requested before W2: the 1 MB per set of W2 fills
  // the DRAM queues for microseconds, and anything requested behind it waits
  // that long.  This thread's row of W1 in its first block, its b1, its
  // output row's b2 go first, and W2 is requested once thread 0's have
  // arrived.
  // (kept as raw bf16 until used: converting at the load would wait for it)
  uint4 w1v[4];
  const int j0 = crank * 64 + ju;                           // this thread's unit in its first block
  const bool have0 = crank < nkb && j0 < a.hidden;
  __nv_bfloat16 b1v = __float2bfloat16_rn(0.f);
  if (w1_fast && have0) {
    const uint4* src = reinterpret_cast<const uint4*>(W1s + static_cast<size_t>(j0) * cond_dim);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (8 * u < cond_dim) w1v[u] = __ldg(src + u);
    b1v = b1s[j0];
  }
  const int i_out = tile * kGM + (warp & 3) * 32 + lane;   // this thread's output row (epilogue)
  const __nv_bfloat16 b2v = a.b2[static_cast<size_t>(set) * a.d + (i_out < a.d ? i_out : a.d - 1)];
  // The conditioning inputs of this thread's first element of c: a time
  // (embedding pairs) and a state value.
  const int half = a.emb_dim / 2;
  const float t_in = threadIdx.x < a.n_cond * half ? a.t[threadIdx.x / half] : 0.f;
  const float s_in = threadIdx.x < a.n_cond * a.state_dim ? a.state[threadIdx.x] : 0.f;
  __syncthreads();   // every small load is out before W2 is requested
  // W2 blocks 0..kGSlots-1 go out first, the rest to L2; h is computed while
  // they land.
  int issued = 0;
  if (threadIdx.x == 0) {
    if (w1_fast && have0) {
      uint32_t dep = __bfloat16_as_ushort(b2v) ^ __bfloat16_as_ushort(b1v) ^ __float_as_uint(t_in) ^
                     __float_as_uint(s_in);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (8 * u < cond_dim) dep ^= w1v[u].x ^ w1v[u].w;
      asm volatile("" ::"r"(dep));
    }
    for (; issued < kGSlots && issued < nkb; ++issued) {
      mbar_arrive_expect_tx(FULL(issued), kGBlock);
      tma_load_4d(sRing + issued * kGBlock, &a.tm_w2, issued * 64, tile * kGM, set, 0, FULL(issued));
    }
    for (int b = kGSlots; b < nkb; ++b) tma_prefetch_l2_4d(&a.tm_w2, b * 64, tile * kGM, set, 0);
  }

  // c_k = [sin(t_k w_j), cos(t_k w_j), state_k],  w_j = 10000^(-j/half):
  // one sincos per (vector, frequency), the state copied.
  for (int idx = threadIdx.x; idx < a.n_cond * half; idx += blockDim.x) {
    const int k = idx / half, jj = idx - k * half;
    const float w = powf(10000.0f, -static_cast<float>(jj) / static_cast<float>(half));
    float sv, cv;
    sincosf((idx == threadIdx.x ? t_in : a.t[k]) * w, &sv, &cv);
    c[k * c_stride + jj] = sv;
    c[k * c_stride + half + jj] = cv;
  }
  for (int idx = threadIdx.x; idx < a.n_cond * a.state_dim; idx += blockDim.x) {
    const int k = idx / a.state_dim, e = idx - k * a.state_dim;
    c[k * c_stride + a.emb_dim + e] = idx == threadIdx.x ? s_in : a.state[idx];
  }
  // This CTA's blocks of H start as zeros: unused vectors, and columns past
  // hidden in the last block.  Blocks owned by a peer are written whole by it.
  for (int kb = crank; kb < nkb; kb += csize) st_shared_v4(sH + kb * kGHBlock + threadIdx.x * 16, 0u, 0u, 0u, 0u);
  __syncthreads();

  // h_k = SiLU(W1 c_k + b1) in fp32, stored as hi / lo bf16 rows of H.
  for (int kb = crank; kb < nkb; kb += csize) {
    const int j = kb * 64 + ju;
    if (j >= a.hidden) continue;
    float acc[kMaxCond / 4];
#pragma unroll
    for (int i = 0; i < kMaxCond / 4; ++i) acc[i] = 0.f;
    if (w1_fast) {
      uint4 wv[4];
      if (kb == crank) {
#pragma unroll
        for (int u = 0; u < 4; ++u) wv[u] = w1v[u];
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(W1s + static_cast<size_t>(j) * cond_dim);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (8 * u < cond_dim) wv[u] = __ldg(src + u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (8 * u < cond_dim) {
          float w[8];
          unpack8(wv[u], w);
#pragma unroll
          for (int i = 0; i < kMaxCond / 4; ++i) {
            const int k = kq + 4 * i;
            if (k < a.n_cond) {
              const float4 c0 = *reinterpret_cast<const float4*>(c + k * c_stride + 8 * u);
              const float4 c1 = *reinterpret_cast<const float4*>(c + k * c_stride + 8 * u + 4);
              acc[i] = fmaf(w[0], c0.x, fmaf(w[1], c0.y, fmaf(w[2], c0.z, fmaf(w[3], c0.w, acc[i]))));
              acc[i] = fmaf(w[4], c1.x, fmaf(w[5], c1.y, fmaf(w[6], c1.z, fmaf(w[7], c1.w, acc[i]))));
            }
          }
        }
      }
    } else {   // wider or unaligned first layers
      const __nv_bfloat16* wr = W1s + static_cast<size_t>(j) * cond_dim;
      for (int e = 0; e < cond_dim; ++e) {
        const float w = __bfloat162float(wr[e]);
#pragma unroll
        for (int i = 0; i < kMaxCond / 4; ++i) {
          const int k = kq + 4 * i;
          if (k < a.n_cond) acc[i] = fmaf(w, c[k * c_stride + e], acc[i]);
        }
      }
    }
    const float bias = __bfloat162float(w1_fast && kb == crank ? b1v : b1s[j]);
#pragma unroll
    for (int i = 0; i < kMaxCond / 4; ++i) {
      const int k = kq + 4 * i;
      if (k < a.n_cond) {
        const float z = acc[i] + bias;
        store_h(sH, j, k, __fdividef(z, 1.0f + __expf(-z)));
      }
    }
  }
  if (csize > 1) {
    // The rows of each own block that hold vectors (hi rows k < n_cond and
    // lo rows 16 + k, 128 bytes each; one 16-byte chunk per thread) go to
    // the same place in every peer's H.  A peer's other rows feed only
    // columns of the product that are never read.  Then one cluster barrier:
    // after it every CTA holds all of H, and no peer writes into this CTA's
    // shared memory any more.
    __syncthreads();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");   // every peer has started
    const int n_rows = 2 * a.n_cond;
    const int row = threadIdx.x >> 3;                       // 0..31
    const bool used = threadIdx.x < 8 * 32 && (row < a.n_cond || (row >= 16 && row < 16 + a.n_cond));
    for (int kb = crank; kb < nkb && used && n_rows > 0; kb += csize) {
      const uint32_t src = sH + kb * kGHBlock + threadIdx.x * 16;
      uint32_t v0, v1, v2, v3;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3) : "r"(src));
      for (int pr = 0; pr < csize; ++pr) {
        if (pr == crank) continue;
        uint32_t dst;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(src), "r"(pr));
        asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v0), "r"(v1), "r"(v2),
                     "r"(v3)
                     : "memory");
      }
    }
    asm volatile("fence.proxy.async;" ::: "memory");   // this thread's H stores -> tensor-core reads
    cluster_sync_all();
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
  // The row tiles of one weight set share the first layer as one cluster of
  // up to 8 CTAs (the largest of 8, 4, 2 that divides the tile count).
  const int tiles = (d + kGM - 1) / kGM;
  a.cluster = tiles % 8 == 0 ? 8 : tiles % 4 == 0 ? 4 : tiles % 2 == 0 ? 2 : 1;
  const dim3 grid(tiles, n_sets);
  if (a.cluster == 1) {
    e = launch_k(ada_gamma_kernel, grid, dim3(kGThreads), smem, s, a);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = a.cluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, ada_gamma_kernel, a);
    count_launch();
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rx
