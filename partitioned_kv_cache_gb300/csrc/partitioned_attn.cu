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
  static constexpr int Q_BYTES = KB * Q_BLOCK;
  static constexpr int P_BYTES = kBM * kBN * 2;
  // K/V stream through a ring of 8 KB pieces.  A K tile is KB pieces (one per
  // 64-column block: 64 keys x 128 B); a V tile is KB pieces of VK keys each
  // (all D columns: KB blocks of VK keys x 128 B).  Each piece is released as
  // soon as the MMAs that read it complete.
  static constexpr int PIECE = 8192;
  static constexpr int NS = 16;                     // ring slots
  static constexpr int VK = v_piece_keys(D);        // keys per V piece
  static constexpr int PIECES_PER_TILE = 2 * KB;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;
  static constexpr int OFF_P = OFF_RING + NS * PIECE;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 64 * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;        // slack for 1024-byte alignment
  static constexpr int TMEM_COLS = (D + 2 * kBN) <= 256 ? 256 : 512;
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(KB * VK * 128 == PIECE, "a V piece fills one ring slot");
};

// Barrier indices: Q, ring full[NS], ring empty[NS], S full[2], P full[2],
// PV done[2], drain.
enum : int { B_Q = 0, B_FULL = 1, B_EMPTY = 17, B_SF = 33, B_PF = 35, B_PV = 37, B_DRAIN = 39 };

struct AttnParams {
  CUtensorMap tm_q;      // 4-D (D, G, Hkv, S), box (64, G, 1, 128/G)
  CUtensorMap tm_k[3];   // 4-D (D, Hkv, keys, layers), box (64, 1, 64, 1): pin, window, dyn
  CUtensorMap tm_v[3];
  __nv_bfloat16* out;    // [S][Hq][D]
  float* part_o;         // [Hkv][splits][D][rows_pad] (column-major per split)
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
  const uint32_t sRing = base + Lay::OFF_RING;
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
    for (int i = 0; i < Lay::NS; ++i) {
      mbar_init(BAR(B_FULL + i), 1);
      mbar_init(BAR(B_EMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
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
      int issued = 0;   // pieces issued
      mbar_arrive_expect_tx(BAR(B_Q), Lay::Q_BYTES);
      for (int kb = 0; kb < Lay::KB; ++kb)
        tma_load_4d(sQ + kb * Lay::Q_BLOCK, &p.tm_q, kb * 64, 0, g, mt * qtok, BAR(B_Q));
      bool ok = true;
      for (int j = 0; ok && j < n; ++j) {
        const TileInfo ti = tile_at(t0 + j, nt_pin, nt_win, p.P, win_len, p.n_priv);
        const int lay = ti.region == 2 ? 0 : p.layer;
        for (int q = 0; q < Lay::PIECES_PER_TILE; ++q) {
          const int pc = issued;
          const int slot = pc % Lay::NS;
          if (pc >= Lay::NS && !mbar_wait(BAR(B_EMPTY + slot), ((pc / Lay::NS) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t dst = sRing + slot * Lay::PIECE;
          mbar_arrive_expect_tx(BAR(B_FULL + slot), Lay::PIECE);
          if (q < Lay::KB) {   // K columns [64q, 64q+64) of 64 keys
            tma_load_4d(dst, &p.tm_k[ti.region], q * 64, g, ti.key0, lay, BAR(B_FULL + slot));
          } else {             // V keys [VK*vb, VK*vb + VK), all columns
            const int vb = q - Lay::KB;
            for (int db = 0; db < Lay::KB; ++db)
              tma_load_4d(dst + db * Lay::VK * 128, &p.tm_v[ti.region], db * 64, g,
                          ti.key0 + vb * Lay::VK, lay, BAR(B_FULL + slot));
          }
          issued = pc + 1;
        }
      }
      // Every copy issued must land before the CTA exits, even after an abort.
      volatile int no_abort = 0;
      mbar_wait(BAR(B_Q), 0, &no_abort);
      for (int pc = issued - Lay::NS < 0 ? 0 : issued - Lay::NS; pc < issued; ++pc)
        mbar_wait(BAR(B_FULL + pc % Lay::NS), (pc / Lay::NS) & 1, &no_abort);
    }
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, false, true);
      // S_j = Q K_j^T: K piece kb holds columns [64kb, 64kb+64) of the tile's
      // 64 keys; four K=16 steps per piece.
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        for (int kb = 0; kb < Lay::KB; ++kb) {
          const int pc = j * Lay::PIECES_PER_TILE + kb;
          const int slot = pc % Lay::NS;
          if (!mbar_wait(BAR(B_FULL + slot), (pc / Lay::NS) & 1, abort_flag)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = sdesc_sw128(sQ + kb * Lay::Q_BLOCK + kk * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(sRing + slot * Lay::PIECE + kk * 32, 16, 1024);
            umma_bf16(tS + st * kBN, a, b, kIdescS, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(BAR(B_EMPTY + slot));
        }
        umma_commit(BAR(B_SF + st));
        return true;
      };
      bool ok = mbar_wait(BAR(B_Q), 0, abort_flag) && issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !issue_s(j + 1)) break;
        const int st = j & 1;
        if (!mbar_wait(BAR(B_PF + st), (j >> 1) & 1, abort_flag)) break;
        // O += P_j V_j: V piece vb holds keys [VK vb, VK vb + VK) with D along the
        // 128-byte rows (MN-major): 64-column blocks VK*128 B apart (LBO), 8-key
        // groups 1024 B apart (SBO).  P (K-major) advances 32 B per 16 keys.
        for (int vb = 0; ok && vb < Lay::KB; ++vb) {
          const int pc = j * Lay::PIECES_PER_TILE + Lay::KB + vb;
          const int slot = pc % Lay::NS;
          if (!mbar_wait(BAR(B_FULL + slot), (pc / Lay::NS) & 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < Lay::VK / 16; ++kk) {
            const int k16 = vb * (Lay::VK / 16) + kk;   // 16-key step within the tile
            const uint64_t a = sdesc_sw128(sP + st * Lay::P_BYTES + k16 * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(sRing + slot * Lay::PIECE + kk * 16 * 128, Lay::VK * 128, 1024);
            umma_bf16(tO, a, b, kIdescO, (j > 0 || k16 > 0) ? 1u : 0u);
          }
          umma_commit(BAR(B_EMPTY + slot));
        }
        if (!ok) break;
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
        // Partial O is stored column-major per split ([D][rows_pad]): for each
        // column the 32 lanes of a warp write 32 consecutive rows (128 B).
        float* dst = p.part_o + (static_cast<size_t>(g) * p.n_splits + split) * p.rows_pad * D + R;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float o[32];
          tmem_ld32(tO + c + lane_off, o);
          if (row_valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[static_cast<size_t>(c + i) * p.rows_pad] = o[i];
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
// out = sum 2^(m_s - m) O_s / l.  One warp = 32 consecutive rows x 32
// columns: lane r owns row r, reads its (m, l) per split (coalesced across
// lanes) and, per split, 32 columns of the column-major partial (each load a
// coalesced 128-byte row run), all independent of one another.
template <int D>
__global__ void __launch_bounds__(32) attn_merge_kernel(const float* __restrict__ part_o,
                                                        const float2* __restrict__ part_ml,
                                                        __nv_bfloat16* __restrict__ out,
                                                        int rows, int rows_pad, int n_splits,
                                                        int Hq, int G) {
  const int lane = threadIdx.x;
  const int R = blockIdx.x * 32 + lane;
  const int c0 = blockIdx.y * 32;
  const int g = blockIdx.z;
  const bool valid = R < rows;
  const size_t head = static_cast<size_t>(g) * n_splits;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) {
    const float2 v = valid ? part_ml[(head + s) * rows_pad + R] : make_float2(-INFINITY, 0.f);
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const float2 v = valid ? part_ml[(head + s) * rows_pad + R] : make_float2(-INFINITY, 0.f);
    const float w = v.y > 0.f ? exp2f(v.x - M) : 0.f;
    lsum += w * v.y;
    if (w != 0.f) {
      const float* o = part_o + (head + s) * rows_pad * D + static_cast<size_t>(c0) * rows_pad + R;
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] += w * o[static_cast<size_t>(i) * rows_pad];
    }
  }
  if (!valid) return;
  const float inv = 1.f / lsum;
  const int tok = R / G, h = g * G + R % G;
  uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(tok) * Hq + h) * D + c0);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    dst[i] = make_uint4(pack_bf16x2(acc[8 * i] * inv, acc[8 * i + 1] * inv),
                        pack_bf16x2(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv),
                        pack_bf16x2(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv),
                        pack_bf16x2(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv));
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
  dim3 mgrid((prm.rows + 31) / 32, D / 32, Hkv);
  attn_merge_kernel<D><<<mgrid, 32, 0, s>>>(prm.part_o, prm.part_ml, prm.out, prm.rows,
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
      const uint32_t vbox[4] = {64u, 1u, static_cast<uint32_t>(v_piece_keys(a.D)), 1u};
      if (!encode_tmap_4d(&prm.tm_k[2], q.k_priv, dims, strides, box)) return cudaErrorInvalidValue;
      if (!encode_tmap_4d(&prm.tm_v[2], q.v_priv, dims, strides, vbox)) return cudaErrorInvalidValue;
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
