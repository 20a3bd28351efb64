// partitioned_attn.cu -- split-KV partitioned attention on tcgen05 (sm_103a).
//
// "Reflex: Real-Time VLA Control through Streaming Inference", §III "Core
// formulas", Eq. (1): suffix queries attend with one softmax over
// [K_pin; K_slide(t); K_dyn(k)] and the matching values.  Proposition A.1:
// the result does not depend on how the key set is partitioned or ordered.
//
// Design (one CTA = 128 query rows x one slice of the key sequence):
//   * All Hq/Hkv heads of the suffix tokens that share one K/V head form the
//     rows of a 128-row tile (row r = token r/G, head g*G + r%G), so every K/V
//     tile feeds a dense M=128 contraction -- with MQA (Hkv = 1) all 8 heads x
//     51 tokens share the same keys.
//   * The key sequence is walked region by region (pinned, window, dynamic) in
//     64-key tiles loaded by TMA straight from where each region lives; the
//     window is read in physical slot order, which Proposition A.1 permits.
//     Keys past a region's length are masked.
//   * S = Q K^T and O += P V run on tcgen05 with both accumulators in TMEM
//     (O: D columns; S: two 64-column buffers).  One thread per row does the
//     online softmax in the exp2 domain; O is rescaled in TMEM only when the
//     running maximum grows by more than 2^8 (otherwise the stale maximum is
//     kept: exact after the final division by the row sum).
//   * The key sequence is split across CTAs (gridDim.y).  Each split writes an
//     fp32 partial (O, m, l); a merge kernel combines them with the global
//     maximum.  With a single split the CTA writes the bf16 output directly.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator and
// MMA issuer, warps 2..5 = softmax and epilogue (TMEM lane quarter = warp % 4).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "rx_internal.h"
#include "sm103_ptx.cuh"

namespace rx {
namespace {

constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

template <int D>
struct Layout {
  static constexpr int KB = D / 64;                 // 64-column blocks of the head dim
  static constexpr int Q_BLOCK = kBM * 128;         // one 64-column block of Q: 128 rows x 128 B
  static constexpr int KV_BLOCK = kBN * 128;        // one 64-column block of a K/V tile
  static constexpr int Q_BYTES = KB * Q_BLOCK;
  static constexpr int KV_BYTES = KB * KV_BLOCK;
  static constexpr int P_BYTES = kBM * kBN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;     // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int NUM_BARS = 12;
  static constexpr int OFF_MISC = OFF_BAR + 16 * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;        // slack for 1024-byte alignment
  static constexpr int TMEM_COLS = (D + 2 * kBN) <= 256 ? 256 : 512;
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Barrier indices.
enum : int { B_Q = 0, B_KF = 1, B_VF = 3, B_SF = 5, B_PF = 7, B_PV = 9, B_DRAIN = 11 };

struct AttnParams {
  CUtensorMap tm_q;      // 4-D (D, G, Hkv, S), box (64, G, 1, 128/G)
  CUtensorMap tm_k[3];   // 4-D (D, Hkv, keys, layers), box (64, 1, 64, 1): pin, window, dyn
  CUtensorMap tm_v[3];
  __nv_bfloat16* out;    // [S][Hq][D]
  float* part_o;         // [Hkv][splits][rows_pad][D]
  float2* part_ml;       // [Hkv][splits][rows_pad]
  const DevState* st;
  int* err;
  int layer;
  int P, F;
  int n_priv;            // dynamic keys
  int Hq, G;
  int rows;              // S * G
  int rows_pad;
  int n_splits;
  float scale_log2;      // log2(e) / sqrt(D)
};

struct TileInfo {
  int region;   // 0 pinned, 1 window, 2 dynamic
  int key0;     // first key of the tile within its region
  int nvalid;   // keys of the tile inside the region (1..64)
};

__device__ __forceinline__ TileInfo tile_at(int t, int nt_pin, int nt_win, int P, int win_len,
                                            int n_priv) {
  TileInfo ti;
  if (t < nt_pin) {
    ti.region = 0;
    ti.key0 = t * kBN;
    ti.nvalid = min(kBN, P - ti.key0);
  } else if (t < nt_pin + nt_win) {
    ti.region = 1;
    ti.key0 = (t - nt_pin) * kBN;
    ti.nvalid = min(kBN, win_len - ti.key0);
  } else {
    ti.region = 2;
    ti.key0 = (t - nt_pin - nt_win) * kBN;
    ti.nvalid = min(kBN, n_priv - ti.key0);
  }
  return ti;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// All lanes wait on the barrier, then agree: the warp proceeds only if every
// lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using Lay = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + Lay::OFF_Q;
  const uint32_t sK = base + Lay::OFF_K;
  const uint32_t sV = base + Lay::OFF_V;
  const uint32_t sP = base + Lay::OFF_P;
  const uint32_t sBar = base + Lay::OFF_BAR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Lay::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Lay::OFF_MISC + 4);
  auto BAR = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mt = blockIdx.x;
  const int split = blockIdx.y;
  const int g = blockIdx.z;

  // Key tiles of this split.  The window length comes from the device-side
  // ring state written by the append kernel earlier in stream order.
  const int valid = *reinterpret_cast<const volatile int*>(&p.st->valid);
  const int win_len = valid * p.F;
  const int nt_pin = (p.P + kBN - 1) / kBN;
  const int nt_win = (win_len + kBN - 1) / kBN;
  const int nt_dyn = (p.n_priv + kBN - 1) / kBN;
  const int T = nt_pin + nt_win + nt_dyn;
  const int t0 = static_cast<int>(static_cast<long long>(split) * T / p.n_splits);
  const int t1 = static_cast<int>(static_cast<long long>(split + 1) * T / p.n_splits);
  const int n = t1 - t0;

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_Q), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_KF + i), 1);
      mbar_init(BAR(B_VF + i), 1);
      mbar_init(BAR(B_SF + i), 1);
      mbar_init(BAR(B_PF + i), 128);
      mbar_init(BAR(B_PV + i), 1);
    }
    mbar_init(BAR(B_DRAIN), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    for (int r = 0; r < 3; ++r) {
      tma_prefetch_desc(&p.tm_k[r]);
      tma_prefetch_desc(&p.tm_v[r]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem;                               // columns [0, D)
  const uint32_t tS = tmem + static_cast<uint32_t>(D);    // two buffers of 64 columns

  const int qtok = kBM / p.G;   // query tokens per tile

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(BAR(B_Q), Lay::Q_BYTES);
      for (int kb = 0; kb < Lay::KB; ++kb)
        tma_load_4d(sQ + kb * Lay::Q_BLOCK, &p.tm_q, kb * 64, 0, g, mt * qtok, BAR(B_Q));
      for (int j = 0; j < n; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(BAR(B_PV + st), ((j - 2) >> 1) & 1, abort_flag)) break;
        const TileInfo ti = tile_at(t0 + j, nt_pin, nt_win, p.P, win_len, p.n_priv);
        const int lay = ti.region == 2 ? 0 : p.layer;
        mbar_arrive_expect_tx(BAR(B_KF + st), Lay::KV_BYTES);
        for (int kb = 0; kb < Lay::KB; ++kb)
          tma_load_4d(sK + st * Lay::KV_BYTES + kb * Lay::KV_BLOCK, &p.tm_k[ti.region], kb * 64,
                      g, ti.key0, lay, BAR(B_KF + st));
        mbar_arrive_expect_tx(BAR(B_VF + st), Lay::KV_BYTES);
        for (int kb = 0; kb < Lay::KB; ++kb)
          tma_load_4d(sV + st * Lay::KV_BYTES + kb * Lay::KV_BLOCK, &p.tm_v[ti.region], kb * 64,
                      g, ti.key0, lay, BAR(B_VF + st));
        issued = j + 1;
      }
      // Every copy issued must land before the CTA exits, even after an abort.
      volatile int no_abort = 0;
      mbar_wait(BAR(B_Q), 0, &no_abort);
      for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j) {
        mbar_wait(BAR(B_KF + (j & 1)), (j >> 1) & 1, &no_abort);
        mbar_wait(BAR(B_VF + (j & 1)), (j >> 1) & 1, &no_abort);
      }
    }
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, false, true);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(BAR(B_KF + st), (j >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kb = kk >> 2, ko = (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sQ + kb * Lay::Q_BLOCK + ko, 16, 1024);
          const uint64_t b = sdesc_sw128(sK + st * Lay::KV_BYTES + kb * Lay::KV_BLOCK + ko, 16, 1024);
          umma_bf16(tS + st * kBN, a, b, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(BAR(B_SF + st));
        return true;
      };
      bool ok = mbar_wait(BAR(B_Q), 0, abort_flag) && issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) break;
        const int st = j & 1;
        if (!mbar_wait(BAR(B_PF + st), (j >> 1) & 1, abort_flag)) break;
        if (!mbar_wait(BAR(B_VF + st), (j >> 1) & 1, abort_flag)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // A = P (K-major, 128 x 64 keys); B = V tile, MN-major: D runs along
          // the 128-byte rows, 64-column blocks Lay::KV_BLOCK apart (LBO),
          // 8-key groups 1024 B apart (SBO).
          const uint64_t a = sdesc_sw128(sP + st * Lay::P_BYTES + kk * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sV + st * Lay::KV_BYTES + kk * 16 * 128, Lay::KV_BLOCK, 1024);
          umma_bf16(tO, a, b, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(BAR(B_PV + st));
      }
      // No tensor-core work may be in flight when TMEM is released.
      umma_commit(BAR(B_DRAIN));
      volatile int no_abort = 0;
      mbar_wait(BAR(B_DRAIN), 0, &no_abort);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int R = mt * kBM + row;                      // row within this K/V head
    const bool row_valid = R < p.rows;
    const size_t part_idx = (static_cast<size_t>(g) * p.n_splits + split) * p.rows_pad + R;
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = n > 0;
    for (int j = 0; ok && j < n; ++j) {
      const int st = j & 1;
      if (!warp_wait(BAR(B_SF + st), (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float s[kBN];
      tmem_ld32(tS + st * kBN + lane_off, s);
      tmem_ld32(tS + st * kBN + 32 + lane_off, s + 32);
      const TileInfo ti = tile_at(t0 + j, nt_pin, nt_win, p.P, win_len, p.n_priv);
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        s[c] = c < ti.nvalid ? s[c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + kRescaleThreshold;
      float fac = 1.f;
      if (need) {
        fac = exp2f(m_used - m_new);   // 0 when nothing was accumulated yet
        l *= fac;
        m_used = m_new;
      }
      if (__any_sync(0xffffffffu, need && j > 0)) {
        // O holds P_{j-1} V_{j-1}: wait for that product, then rescale in TMEM.
        if (!warp_wait(BAR(B_PV + ((j - 1) & 1)), ((j - 1) >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + c + lane_off, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= fac;
          tmem_st32(tO + c + lane_off, o);
        }
      }
      const float mb = m_used == -INFINITY ? 0.f : m_used;
      uint32_t pk[kBN / 2];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kBN / 2; ++c) {
        const float a = exp2f(s[2 * c] - mb);
        const float b = exp2f(s[2 * c + 1] - mb);
        rs += a + b;
        pk[c] = pack_bf16x2(a, b);
      }
      l += rs;
      // P buffer `st` was last read by P_{j-2} V_{j-2}.
      if (j >= 2 && !warp_wait(BAR(B_PV + st), ((j - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
      const uint32_t prow = sP + st * Lay::P_BYTES + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(prow + ((c ^ (row & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(BAR(B_PF + st));
    }
    if (ok) ok = warp_wait(BAR(B_PV + ((n - 1) & 1)), ((n - 1) >> 1) & 1, abort_flag);
    if (ok) {
      tc_fence_after();
      if (p.n_splits == 1) {
        const int tok = R / p.G;
        const int h = g * p.G + R % p.G;
        __nv_bfloat16* dst = p.out + (static_cast<size_t>(tok) * p.Hq + h) * D;
        const float inv = 1.f / l;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + c + lane_off, o);
          if (row_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                 pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                 pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                 pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
          }
        }
      } else {
        float* dst = p.part_o + part_idx * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + c + lane_off, o);
          if (row_valid) {
            float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          }
        }
        if (row_valid) p.part_ml[part_idx] = make_float2(m_used, l);
      }
    } else if (n == 0 && row_valid && p.n_splits > 1) {
      p.part_ml[part_idx] = make_float2(-INFINITY, 0.f);   // empty split: merge skips it
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Lay::TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err, kErrAttnTimeout);
}

// Combine the splits of every row: m = max m_s, l = sum 2^(m_s - m) l_s,
// out = sum 2^(m_s - m) O_s / l.  One warp per row, D/32 columns per lane.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const float* __restrict__ part_o,
                                                         const float2* __restrict__ part_ml,
                                                         __nv_bfloat16* __restrict__ out,
                                                         int rows, int rows_pad, int n_splits,
                                                         int Hq, int G) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = blockIdx.x * 8 + warp;
  const int g = blockIdx.y;
  if (R >= rows) return;
  const size_t head_base = static_cast<size_t>(g) * n_splits * rows_pad;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) {
    const float2 v = part_ml[head_base + static_cast<size_t>(s) * rows_pad + R];
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  float acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const size_t idx = head_base + static_cast<size_t>(s) * rows_pad + R;
    const float2 v = part_ml[idx];
    if (!(v.y > 0.f)) continue;
    const float w = exp2f(v.x - M);
    lsum += w * v.y;
    const float* o = part_o + idx * D + lane * E;
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float2 x = *reinterpret_cast<const float2*>(o + i);
      acc[i] += w * x.x;
      acc[i + 1] += w * x.y;
    }
  }
  const float inv = 1.f / lsum;
  const int tok = R / G, h = g * G + R % G;
  __nv_bfloat16* dst = out + (static_cast<size_t>(tok) * Hq + h) * D + lane * E;
#pragma unroll
  for (int i = 0; i < E; i += 2)
    *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
}

template <int D>
cudaError_t launch_one(const AttnParams& prm, int m_tiles, int Hkv, cudaStream_t s) {
  using Lay = Layout<D>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Lay::ALLOC);
  });
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(m_tiles, prm.n_splits, Hkv);
  attn_kernel<D><<<grid, kThreads, Lay::ALLOC, s>>>(prm);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || prm.n_splits == 1) return e;
  dim3 mgrid((prm.rows + 7) / 8, Hkv);
  attn_merge_kernel<D><<<mgrid, 256, 0, s>>>(prm.part_o, prm.part_ml, prm.out, prm.rows,
                                              prm.rows_pad, prm.n_splits, prm.Hq, prm.G);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_partitioned_attention(const AttnLaunch& a, const AttnRequest* reqs, int nreq,
                                         cudaStream_t s, int* used_splits) {
  const int G = a.Hq / a.Hkv;
  for (int r = 0; r < nreq; ++r) {
    const AttnRequest& q = reqs[r];
    AttnParams prm;
    memset(&prm, 0, sizeof(prm));
    // Q: (D, G, Hkv, S) so that one box of (64, G, 1, 128/G) is a 128-row tile.
    {
      const uint64_t dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(G),
                                static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(q.n_tok)};
      const uint64_t strides[3] = {static_cast<uint64_t>(a.D) * 2,
                                   static_cast<uint64_t>(G) * a.D * 2,
                                   static_cast<uint64_t>(a.Hq) * a.D * 2};
      const uint32_t box[4] = {64u, static_cast<uint32_t>(G), 1u, static_cast<uint32_t>(kBM / G)};
      if (!encode_tmap_4d(&prm.tm_q, q.q, dims, strides, box)) return cudaErrorInvalidValue;
    }
    prm.tm_k[0] = *a.tm_pin_k;
    prm.tm_v[0] = *a.tm_pin_v;
    prm.tm_k[1] = *a.tm_slide_k;
    prm.tm_v[1] = *a.tm_slide_v;
    if (q.n_priv > 0) {
      const uint64_t dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hkv),
                                static_cast<uint64_t>(q.n_priv), 1};
      const uint64_t strides[3] = {static_cast<uint64_t>(a.D) * 2,
                                   static_cast<uint64_t>(a.Hkv) * a.D * 2,
                                   static_cast<uint64_t>(q.n_priv) * a.Hkv * a.D * 2};
      const uint32_t box[4] = {64u, 1u, static_cast<uint32_t>(kBN), 1u};
      if (!encode_tmap_4d(&prm.tm_k[2], q.k_priv, dims, strides, box)) return cudaErrorInvalidValue;
      if (!encode_tmap_4d(&prm.tm_v[2], q.v_priv, dims, strides, box)) return cudaErrorInvalidValue;
    } else {
      prm.tm_k[2] = *a.tm_pin_k;   // never read: no dynamic tiles
      prm.tm_v[2] = *a.tm_pin_v;
    }
    prm.out = static_cast<__nv_bfloat16*>(q.out);
    prm.part_o = a.part_o;
    prm.part_ml = a.part_ml;
    prm.st = a.st;
    prm.err = a.err;
    prm.layer = a.layer;
    prm.P = a.P;
    prm.F = a.F;
    prm.n_priv = q.n_priv;
    prm.Hq = a.Hq;
    prm.G = G;
    prm.rows = q.n_tok * G;
    const int m_tiles = (prm.rows + kBM - 1) / kBM;
    prm.rows_pad = m_tiles * kBM;
    prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
    // Split the key sequence so that the grid fills the GPU once.
    const int t_max = (a.P + kBN - 1) / kBN + (a.N * a.F + kBN - 1) / kBN + (q.n_priv + kBN - 1) / kBN;
    int splits = a.forced_splits > 0 ? a.forced_splits : a.num_sms / (m_tiles * a.Hkv);
    splits = splits < 1 ? 1 : splits;
    splits = splits > t_max ? t_max : splits;
    splits = splits > a.max_splits ? a.max_splits : splits;
    prm.n_splits = splits;
    if (used_splits) *used_splits = splits;
    cudaError_t e;
    switch (a.D) {
      case 64: e = launch_one<64>(prm, m_tiles, a.Hkv, s); break;
      case 128: e = launch_one<128>(prm, m_tiles, a.Hkv, s); break;
      case 256: e = launch_one<256>(prm, m_tiles, a.Hkv, s); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace rx
