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
//     64-key tiles read straight from where each region lives; the window is
//     read in physical slot order, which Proposition A.1 permits.  Keys past a
//     region's length are masked.  The store keeps its regions pre-tiled in
//     the operand layout, so a K or V tile is one contiguous bulk copy; the
//     caller's dynamic K/V (and any untiled region) come in by TMA boxes that
//     produce the same layout.  K and V tiles stream through a ring of slots;
//     a K slot is released once Q K^T has read it, a V slot once P V has.
//   * S = Q K^T and O += P V run on tcgen05 with both accumulators in TMEM
//     (O: D columns; S: two 64-column buffers).  One thread per row does the
//     online softmax in the exp2 domain; O is rescaled in TMEM only when the
//     running maximum grows by more than 2^8 (otherwise the stale maximum is
//     kept: exact after the final division by the row sum).
//   * The key sequence is split across CTAs (gridDim.y).  When the splits of an
//     M-tile form one thread-block cluster (up to kMaxClusterSplits), each CTA
//     parks its normalised partial O / l (bf16, in 16-column halves of 4 KB)
//     and its fp32 (m, l) in its own shared memory, then pushes every half
//     with one bulk copy to the cluster CTA that owns those columns; owners
//     read all splits' (m, l) through distributed shared memory and finish
//     their columns of the bf16 output: no partials leave the chip and no
//     second kernel runs.  Beyond that size each split writes an fp32 partial
//     to global memory and a merge kernel combines them.  With a single split
//     the CTA writes the bf16 output directly.
//
// Warp roles (224 threads): warp 0 = copy producer, warp 1 = TMEM allocator and
// Q K^T issuer, warp 6 = P V issuer, warps 2..5 = softmax and epilogue (TMEM
// lane quarter = warp % 4).  The two MMA streams are issued by different warps
// so that queueing Q K^T of the next tile behind the tensor pipe never delays
// P V of the current one.
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

constexpr int kThreads = 224;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr int kTilesPerSplit = 3;            // target key tiles per split (on-chip merge)
constexpr int kMaxClusterSplits = 16;        // splits merged on chip through a cluster

template <int D>
struct Layout {
  static constexpr int KB = D / 64;                 // 64-column blocks of the head dim
  static constexpr int Q_BLOCK = kBM * 128;         // one 64-column block of Q: 128 rows x 128 B
  static constexpr int Q_BYTES = KB * Q_BLOCK;
  static constexpr int P_BYTES = kBM * kBN * 2;
  static constexpr int TILE = static_cast<int>(tile_bytes(D));   // one K or V tile: [KB][64][128 B]
  static constexpr int NS = (128 * 1024) / TILE;    // ring slots (4 at D = 256)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;
  static constexpr int OFF_P = OFF_RING + NS * TILE;
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_MISC = OFF_BAR + 64 * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;        // slack for 1024-byte alignment
  static constexpr int TMEM_COLS = (D + 2 * kBN) <= 256 ? 256 : 512;
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(NS >= 4 && NS <= 16, "ring depth");
};

// Barrier indices: Q, ring full[NS], ring empty[NS], S full[2], P full[2],
// PV done[2], drain.
enum : int { B_Q = 0, B_FULL = 1, B_EMPTY = 17, B_SF = 33, B_PF = 35, B_PV = 37, B_DRAIN = 39, B_RECV = 40 };

// One group of query rows: the action suffix, or a dense batch of language
// streams.  Its M-tiles occupy workspace rows [row_base, row_base + m_tiles*128).
struct SegParams {
  CUtensorMap tm_q;      // 4-D (D, G, Hkv, tokens), box (64, G, 1, 128/G)
  CUtensorMap tm_kp;     // private keys: 4-D (D, Hkv, n_priv, 1), box (64, 1, 64, 1)
  CUtensorMap tm_vp;
  __nv_bfloat16* out;    // [tokens][Hq][D]
  const int* tail_len;   // stream mask: keys held by each stream's tail (device)
  int n_priv;            // private keys
  int rows;              // tokens * G
  int row_base;
  int m_tiles;
  int tok_per_stream;    // stream mask: query tokens per stream
  int tail_cap;          // stream mask: private keys per stream; 0 = no mask
  int state_tokens;      // block-causal: tokens below see private keys [0, state_tokens) only
};

struct AttnParams {
  SegParams seg[2];
  CUtensorMap tm_k[2];   // pin, window when not pre-tiled: (D, Hkv, keys, layers), box (64, 1, 64, 1)
  CUtensorMap tm_v[2];
  const uint8_t* k_tiles[2];   // pre-tiled pin / window of (layer, head 0); null = tensor map
  const uint8_t* v_tiles[2];
  long long head_stride[2];    // bytes between heads of a tiled region
  float* part_o;         // [Hkv][splits][D][rows_pad] (column-major per split)
  float2* part_ml;       // [Hkv][splits][rows_pad]
  const DevState* st;
  int* err;
  int layer;
  int P, F, N, slots;    // pinned tokens; window: tokens per frame, frames, frame slots
  int Hq, G;
  int rows_pad;          // workspace rows of all segments
  int n_splits;
  int fused;             // 1: the splits of an M-tile form a cluster and merge on chip
  float scale_log2;      // log2(e) / sqrt(D)
};

struct TileInfo {
  int region;   // 0 pinned, 1 window, 2 dynamic
  int key0;     // first key of the tile among the region's keys (masks, stream windows)
  int phys0;    // first stored token of the tile (where it is read from)
  int nvalid;   // keys of the tile inside the region (1..64)
};

// Window tiles skip the spare slot's tiles [hole0, hole0 + hole_n) once the
// ring is full (hole_n = 0 otherwise).
__device__ __forceinline__ TileInfo tile_at(int t, int nt_pin, int nt_win, int P, int win_len,
                                            int n_priv, int hole0, int hole_n) {
  TileInfo ti;
  if (t < nt_pin) {
    ti.region = 0;
    ti.key0 = t * kBN;
    ti.phys0 = ti.key0;
    ti.nvalid = min(kBN, P - ti.key0);
  } else if (t < nt_pin + nt_win) {
    const int tw = t - nt_pin;
    ti.region = 1;
    ti.key0 = tw * kBN;
    ti.phys0 = (tw < hole0 ? tw : tw + hole_n) * kBN;
    ti.nvalid = min(kBN, win_len - ti.key0);
  } else {
    ti.region = 2;
    ti.key0 = (t - nt_pin - nt_win) * kBN;
    ti.phys0 = ti.key0;
    ti.nvalid = min(kBN, n_priv - ti.key0);
  }
  return ti;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One contiguous global -> shared copy, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Park this thread's row of the split's normalised partial O / l (bf16) and
// (m, l) in shared memory for the cluster merge.  Layout at `os`: [D/16
// halves][8 column pairs][128 rows] of bf16x2, so a half is one contiguous
// 4 KB block (one bulk copy) and a warp's 4-byte stores cover 128 contiguous
// bytes; (m, l) follow at os + D*256.  With have_o == false the row is zeros
// (an empty split, l = 0).  Warp-collective (TMEM loads).
template <int D>
__device__ __forceinline__ void park_partial(uint32_t os, uint32_t t_row, int row, float m, float l,
                                             bool have_o) {
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
  for (int c = 0; c < D; c += 32) {
    float o[32];
    if (have_o) {
      tmem_ld32(t_row + c, o);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0.f;
    }
#pragma unroll
    for (int pr = 0; pr < 16; ++pr) {
      const int col = c + 2 * pr;   // columns col, col+1
      const uint32_t a = os + (col / 16) * 4096 + ((col % 16) / 2) * 512 + row * 4;
      asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(pack_bf16x2(o[2 * pr] * inv, o[2 * pr + 1] * inv))
                   : "memory");
    }
  }
  const uint32_t mla = os + D * 256 + row * 8;
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(mla), "f"(m), "f"(l) : "memory");
  fence_proxy_async_smem();   // the halves leave through the copy engine (async proxy)
}

// Push `bytes` of this CTA's shared memory to shared memory of a cluster
// peer (addresses from dsmem_map), completion counted on the peer's mbarrier.
__device__ __forceinline__ void bulk_push(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                          uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(bar_cluster)
      : "memory");
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
  const int si = static_cast<int>(blockIdx.x) < p.seg[0].m_tiles ? 0 : 1;
  const SegParams& sg = p.seg[si];
  const int mt = blockIdx.x - (si ? p.seg[0].m_tiles : 0);   // M-tile within the segment
  const int split = blockIdx.y;
  const int g = blockIdx.z;

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
    mbar_init(BAR(B_DRAIN), 2);   // one commit from each MMA issuer
    mbar_init(BAR(B_RECV), 1);    // cluster merge: partial halves pushed to this CTA
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Lay::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {   // prefetch only the descriptors this CTA uses
    tma_prefetch_desc(&sg.tm_q);
    for (int r = 0; r < 2; ++r) {
      if (p.k_tiles[r]) continue;
      tma_prefetch_desc(&p.tm_k[r]);
      tma_prefetch_desc(&p.tm_v[r]);
    }
    if (sg.n_priv > 0) {
      tma_prefetch_desc(&sg.tm_kp);
      tma_prefetch_desc(&sg.tm_vp);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Everything above touched only shared memory, TMEM and the parameters; from
  // here on the kernel reads inputs an earlier kernel may have written.
  grid_dependency_wait();
  grid_launch_dependents();
  // Key tiles of this split.  The window comes from the device-side ring state
  // published by the append kernel (one 64-bit word: a consistent snapshot
  // even while a push on another stream is publishing).
  int head = 0, valid = 0;
  load_ring_state(p.st, &head, &valid);
  asm volatile("fence.acq_rel.gpu;" ::: "memory");   // frame data before the snapshot
  // With a spare slot and a full ring the window is every slot but `head`.
  const bool hole = p.slots > p.N && valid == p.N;
  const int win_len = hole ? (p.slots - 1) * p.F : valid * p.F;
  const int hole0 = hole ? head * p.F / kBN : 0;
  const int hole_n = hole ? p.F / kBN : 0;
  const int nt_pin = (p.P + kBN - 1) / kBN;
  const int nt_win = (win_len + kBN - 1) / kBN;
  const int nt_dyn = (sg.n_priv + kBN - 1) / kBN;
  const int T = nt_pin + nt_win + nt_dyn;
  const int t0 = static_cast<int>(static_cast<long long>(split) * T / p.n_splits);
  const int t1 = static_cast<int>(static_cast<long long>(split + 1) * T / p.n_splits);
  const int n = t1 - t0;

  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem;                               // columns [0, D)
  const uint32_t tS = tmem + static_cast<uint32_t>(D);    // two buffers of 64 columns

  const int qtok = kBM / p.G;   // query tokens per tile

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    // Ring order: K_0, V_0, K_1, V_1, ...; item i uses slot i % NS.
    if (lane == 0) {
      int issued = 0;
      mbar_arrive_expect_tx(BAR(B_Q), Lay::Q_BYTES);
      for (int kb = 0; kb < Lay::KB; ++kb)
        tma_load_4d(sQ + kb * Lay::Q_BLOCK, &sg.tm_q, kb * 64, 0, g, mt * qtok, BAR(B_Q));
      for (int j = 0; j < n && issued >= 0; ++j) {
        const TileInfo ti = tile_at(t0 + j, nt_pin, nt_win, p.P, win_len, sg.n_priv, hole0, hole_n);
        const int lay = ti.region == 2 ? 0 : p.layer;
        for (int kv = 0; kv < 2; ++kv) {
          const int it = issued;
          const int slot = it % Lay::NS;
          if (it >= Lay::NS && !mbar_wait(BAR(B_EMPTY + slot), ((it / Lay::NS) - 1) & 1, abort_flag)) {
            issued = -issued - 1;   // stop; remember how many were issued
            break;
          }
          const uint32_t dst = sRing + slot * Lay::TILE;
          mbar_arrive_expect_tx(BAR(B_FULL + slot), Lay::TILE);
          const uint8_t* tiles = ti.region < 2 ? (kv ? p.v_tiles[ti.region] : p.k_tiles[ti.region]) : nullptr;
          if (tiles) {
            bulk_load(dst, tiles + g * p.head_stride[ti.region] + static_cast<long long>(ti.phys0 / kBN) * Lay::TILE,
                      Lay::TILE, BAR(B_FULL + slot));
          } else {
            const CUtensorMap* tm = ti.region == 2 ? (kv ? &sg.tm_vp : &sg.tm_kp)
                                                   : (kv ? &p.tm_v[ti.region] : &p.tm_k[ti.region]);
            for (int kb = 0; kb < Lay::KB; ++kb)
              tma_load_4d(dst + kb * 8192, tm, kb * 64, g, ti.phys0, lay, BAR(B_FULL + slot));
          }
          issued = it + 1;
        }
      }
      if (issued < 0) issued = -issued - 1;
      // Every copy issued must land before the CTA exits, even after an abort.
      volatile int no_abort = 0;
      mbar_wait(BAR(B_Q), 0, &no_abort);
      for (int it = issued - Lay::NS < 0 ? 0 : issued - Lay::NS; it < issued; ++it)
        mbar_wait(BAR(B_FULL + it % Lay::NS), (it / Lay::NS) & 1, &no_abort);
    }
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
      bool ok = mbar_wait(BAR(B_Q), 0, abort_flag);
      for (int j = 0; ok && j < n; ++j) {
        const int st = j & 1;
        // S buffer st last held S_{j-2}; the softmax is done with it once it
        // has published P_{j-2}.
        if (j >= 2 && !mbar_wait(BAR(B_PF + st), ((j - 2) >> 1) & 1, abort_flag)) break;
        const int it = 2 * j;
        const int slot = it % Lay::NS;
        if (!mbar_wait(BAR(B_FULL + slot), (it / Lay::NS) & 1, abort_flag)) break;
        tc_fence_after();
        // S_j = Q K_j^T (both K-major): column block kb of the K tile sits at
        // kb * 8 KB; four K=16 steps of 32 B within each 128-byte row.
        const uint32_t kt = sRing + slot * Lay::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t kb = kk >> 2, ko = (kk & 3) * 32;
          const uint64_t a = sdesc_sw128(sQ + kb * Lay::Q_BLOCK + ko, 16, 1024);
          const uint64_t b = sdesc_sw128(kt + kb * 8192 + ko, 16, 1024);
          umma_bf16(tS + st * kBN, a, b, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(BAR(B_EMPTY + slot));
        umma_commit(BAR(B_SF + st));
      }
      // No tensor-core work may be in flight when TMEM is released.
      umma_commit(BAR(B_DRAIN));
      volatile int no_abort = 0;
      mbar_wait(BAR(B_DRAIN), 0, &no_abort);
    }
  } else if (n > 0 && warp == 6) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBM, D, false, true);
      for (int j = 0; j < n; ++j) {
        const int st = j & 1;
        if (!mbar_wait(BAR(B_PF + st), (j >> 1) & 1, abort_flag)) break;
        const int it = 2 * j + 1;
        const int slot = it % Lay::NS;
        if (!mbar_wait(BAR(B_FULL + slot), (it / Lay::NS) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t vt = sRing + slot * Lay::TILE;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // A = P (K-major, 128 x 64 keys); B = V tile read MN-major: D runs
          // along the 128-byte rows, 64-column blocks 8 KB apart (LBO), 8-key
          // groups 1 KB apart (SBO), 16 keys = 2 KB per K step.
          const uint64_t a = sdesc_sw128(sP + st * Lay::P_BYTES + kk * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(vt + kk * 16 * 128, 8192, 1024);
          umma_bf16(tO, a, b, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(BAR(B_EMPTY + slot));
        umma_commit(BAR(B_PV + st));
      }
      umma_commit(BAR(B_DRAIN));
      volatile int no_abort = 0;
      mbar_wait(BAR(B_DRAIN), 0, &no_abort);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int Rs = mt * kBM + row;                     // row within the segment
    const bool row_valid = Rs < sg.rows;
    const int R = sg.row_base + Rs;                    // row within the workspace
    const size_t part_idx = (static_cast<size_t>(g) * p.n_splits + split) * p.rows_pad + R;
    // Private-key window of this row: its stream's tail (stream mask) or the
    // state block's own keys (block-causal suffix); [0, n_priv) otherwise.
    int lo = 0, hi = sg.n_priv;
    if (sg.tail_cap > 0) {
      lo = hi = 0;
      if (row_valid) {
        const int b = (Rs / p.G) / sg.tok_per_stream;
        lo = b * sg.tail_cap;
        hi = lo + min(max(sg.tail_len[b], 0), sg.tail_cap);
      }
    }
    if (sg.state_tokens > 0 && Rs / p.G < sg.state_tokens) hi = min(hi, sg.state_tokens);
    const bool priv_masked = sg.tail_cap > 0 || sg.state_tokens > 0;
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
      const TileInfo ti = tile_at(t0 + j, nt_pin, nt_win, p.P, win_len, sg.n_priv, hole0, hole_n);
      if (ti.region == 2 && priv_masked) {   // private keys outside this row's window
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          const int key = ti.key0 + c;
          if (c >= ti.nvalid || key < lo || key >= hi) s[c] = -INFINITY;
        }
      } else if (ti.nvalid < kBN) {   // ragged tile: keys past the region are not keys
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c >= ti.nvalid) s[c] = -INFINITY;
      }
      // Row maximum of the raw scores (the scale is positive), as a tree.
      float t32[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) t32[c] = fmaxf(s[c], s[c + 32]);
#pragma unroll
      for (int w = 16; w > 0; w >>= 1)
#pragma unroll
        for (int c = 0; c < w; ++c) t32[c] = fmaxf(t32[c], t32[c + w]);
      const float mx = t32[0] * p.scale_log2;
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
      // p = 2^(s * scale - m): one FMA feeds each exponential.
      const float nmb = m_used == -INFINITY ? 0.f : -m_used;
      uint32_t pk[kBN / 2];
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kBN / 2; ++c) {
        const float a = exp2f(fmaf(s[2 * c], p.scale_log2, nmb));
        const float b = exp2f(fmaf(s[2 * c + 1], p.scale_log2, nmb));
        rs[c & 3] += a + b;
        pk[c] = pack_bf16x2(a, b);
      }
      l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
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
        const int tok = Rs / p.G;
        const int h = g * p.G + Rs % p.G;
        __nv_bfloat16* dst = sg.out + (static_cast<size_t>(tok) * p.Hq + h) * D;
        const float inv = l > 0.f ? 1.f / l : 0.f;   // a row with no key at all gets zeros
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
      } else if (p.fused) {
        park_partial<D>(base + Lay::OFF_Q, tO + lane_off, row, m_used, l, true);
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
    } else if (p.fused) {
      // empty (or abandoned) split: zeros with l = 0 contribute nothing
      park_partial<D>(base + Lay::OFF_Q, tO + lane_off, row, -INFINITY, 0.f, false);
    } else if (n == 0 && row_valid && p.n_splits > 1) {
      p.part_ml[part_idx] = make_float2(-INFINITY, 0.f);   // empty split: merge skips it
    }
  }

  if (p.fused) {
    // ---------------------------------------------------------- cluster merge
    // Each CTA owns the 16-column halves rank, rank + C, ... of the output.
    // After barrier 1 every CTA pushes each of its parked halves (4 KB) into
    // the owner's receive slot [local half][source rank]; the owner combines
    // them from its own shared memory.  All threads of all CTAs of the
    // cluster pass both barriers, whatever path they took above.
    const int C = p.n_splits;
    const uint32_t rank = cluster_ctarank();
    const int owned = (D / 16 - static_cast<int>(rank) + C - 1) / C;
    const uint32_t os_local = base + Lay::OFF_Q;
    const uint32_t recv_local = os_local + D * 256 + 1024;
    if (threadIdx.x == 0) mbar_arrive_expect_tx(BAR(B_RECV), owned * C * 4096);
    __syncwarp();
    cluster_sync_all();
    if (threadIdx.x == 0) {
      for (int half = 0; half < D / 16; ++half) {
        const uint32_t owner = static_cast<uint32_t>(half % C);
        const uint32_t slot = static_cast<uint32_t>((half / C) * C) + rank;
        bulk_push(dsmem_map(recv_local + slot * 4096, owner), os_local + half * 4096, 4096,
                  dsmem_map(BAR(B_RECV), owner));
      }
    }
    if (warp >= 2 && warp <= 5) {
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      const int Rs = mt * kBM + row;
      const uint32_t ml_local = os_local + D * 256 + row * 8;
      float ms[kMaxClusterSplits], ws[kMaxClusterSplits];
      float M = -INFINITY;
#pragma unroll
      for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
        ws[s2] = 0.f;
        ms[s2] = -INFINITY;
        if (s2 < C) {
          const float2 v = dsmem_ld_f32x2(dsmem_map(ml_local, s2));
          if (v.y > 0.f) {
            ms[s2] = v.x;
            ws[s2] = v.y;
            M = fmaxf(M, v.x);
          }
        }
      }
      // Weight of split s: 2^(m_s - M) l_s / L (the parked partials are O_s / l_s).
      float L = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
        const float w = ws[s2] > 0.f ? exp2f(ms[s2] - M) * ws[s2] : 0.f;
        L += w;
        ws[s2] = w;
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;   // a row with no key at all gets zeros
#pragma unroll
      for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) ws[s2] *= inv;
      const bool row_valid = Rs < sg.rows;
      const int tok = Rs / p.G, h = g * p.G + Rs % p.G;
      const bool got = warp_wait(BAR(B_RECV), 0, abort_flag);
      for (int k = 0; got && k < owned; ++k) {
        const int half = static_cast<int>(rank) + k * C;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
          if (s2 < C) {
            const uint32_t src = recv_local + (k * C + s2) * 4096 + row * 4;
#pragma unroll
            for (int pr = 0; pr < 8; ++pr) {
              uint32_t v;
              asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(src + pr * 512) : "memory");
              acc[2 * pr] = fmaf(ws[s2], __uint_as_float(v << 16), acc[2 * pr]);
              acc[2 * pr + 1] = fmaf(ws[s2], __uint_as_float(v & 0xFFFF0000u), acc[2 * pr + 1]);
            }
          }
        }
        if (row_valid) {
          uint4* d4 = reinterpret_cast<uint4*>(sg.out + (static_cast<size_t>(tok) * p.Hq + h) * D + half * 16);
          d4[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                             pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
          d4[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                             pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
        }
      }
    }
    // Every push into this CTA must land before it leaves barrier 2 (an
    // abandoned wait above still drains here, bounded).
    if (threadIdx.x == 0) {
      volatile int no_abort = 0;
      mbar_wait(BAR(B_RECV), 0, &no_abort);
    }
    __syncwarp();
    cluster_sync_all();   // peers may still read this CTA's shared memory until here
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Lay::TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err, kErrAttnTimeout);
}

// Combine the splits of every row: m = max m_s, l = sum 2^(m_s - m) l_s,
// out = sum 2^(m_s - m) O_s / l.  A block covers 32 consecutive workspace rows
// (of one segment) x 32 columns; lane r owns row r.  The four warps take every fourth split, so up
// to eight splits' loads are in flight per lane (two per warp, unrolled), each
// a coalesced 128-byte run of the column-major partial; the warps' sums meet
// in shared memory.
template <int D>
__global__ void __launch_bounds__(128) attn_merge_kernel(const float* __restrict__ part_o,
                                                         const float2* __restrict__ part_ml,
                                                         __nv_bfloat16* out0, int rows0,
                                                         __nv_bfloat16* out1, int rows1,
                                                         int row_base1, int rows_pad, int n_splits,
                                                         int Hq, int G) {
  __shared__ float red[3][32][33];
  __shared__ float red_l[3][32];
  grid_dependency_wait();
  grid_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = blockIdx.x * 32 + lane;               // workspace row
  const int si = static_cast<int>(blockIdx.x) * 32 < row_base1 ? 0 : 1;   // blocks never straddle
  const int base = si ? row_base1 : 0;
  const int rows = si ? rows1 : rows0;
  __nv_bfloat16* out = si ? out1 : out0;
  if (static_cast<int>(blockIdx.x) * 32 - base >= rows) return;   // padding only
  const int Rs = R - base;
  const int c0 = blockIdx.y * 32;
  const int g = blockIdx.z;
  const bool valid = Rs < rows;
  const int Rc = valid ? R : base + rows - 1;   // keep loads on written rows
  const size_t head = static_cast<size_t>(g) * n_splits;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) {
    const float2 v = part_ml[(head + s) * rows_pad + Rc];
    if (v.y > 0.f) M = fmaxf(M, v.x);
  }
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  float lsum = 0.f;
  const size_t col_off = static_cast<size_t>(c0) * rows_pad + Rc;
#pragma unroll 2
  for (int s = warp; s < n_splits; s += 4) {
    const float2 v = part_ml[(head + s) * rows_pad + Rc];
    const bool live = v.y > 0.f;
    const float w = live ? exp2f(v.x - M) : 0.f;
    lsum += w * v.y;
    const float* o = part_o + (head + s) * rows_pad * D + col_off;
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = o[static_cast<size_t>(i) * rows_pad];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] += live ? w * x[i] : 0.f;
  }
  if (warp > 0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) red[warp - 1][i][lane] = acc[i];
    red_l[warp - 1][lane] = lsum;
  }
  __syncthreads();
  if (warp > 0 || !valid) return;
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] += red[0][i][lane] + red[1][i][lane] + red[2][i][lane];
  lsum += red_l[0][lane] + red_l[1][lane] + red_l[2][lane];
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;   // a row with no key at all gets zeros
  const int tok = Rs / G, h = g * G + Rs % G;
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
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(m_tiles, prm.n_splits, Hkv);
  cudaError_t e;
  if (prm.fused) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Lay::ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = prm.n_splits;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, attn_kernel<D>, prm);
    count_launch();
  } else {
    e = launch_k(attn_kernel<D>, grid, dim3(kThreads), Lay::ALLOC, s, prm);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || prm.n_splits == 1 || prm.fused) return e;
  dim3 mgrid(prm.rows_pad / 32, D / 32, Hkv);
  e = launch_k(attn_merge_kernel<D>, mgrid, dim3(128), 0, s, static_cast<const float*>(prm.part_o),
               static_cast<const float2*>(prm.part_ml), prm.seg[0].out, prm.seg[0].rows,
               prm.seg[1].out, prm.seg[1].rows, prm.seg[1].row_base, prm.rows_pad, prm.n_splits,
               prm.Hq, prm.G);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Largest cluster of attention CTAs (one per SM) the device can co-schedule,
// capped at kMaxClusterSplits; 1 if clusters are unavailable.
template <int D>
int max_cluster_splits() {
  static int cached = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (cached >= 0) return cached;
  cached = 1;
  cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<D>::ALLOC);
  cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  for (int c = kMaxClusterSplits; c >= 2; c /= 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, c, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Layout<D>::ALLOC;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = c;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_kernel<D>, &cfg) == cudaSuccess && n >= 1) {
      cached = c;
      break;
    }
  }
  cudaGetLastError();
  return cached;
}

}  // namespace

cudaError_t launch_partitioned_attention(const AttnLaunch& a, const AttnSegment* segs, int nseg,
                                         cudaStream_t s, int* used_splits) {
  if (nseg < 1 || nseg > 2) return cudaErrorInvalidValue;
  const int G = a.Hq / a.Hkv;
  AttnParams prm;
  memset(&prm, 0, sizeof(prm));
  int m_total = 0, t_max = 0;
  const int t_shared = (a.P + kBN - 1) / kBN + (a.N * a.F + kBN - 1) / kBN;
  for (int i = 0; i < nseg; ++i) {
    const AttnSegment& q = segs[i];
    SegParams& sp = prm.seg[i];
    // Q: (D, G, Hkv, tokens) so that one box of (64, G, 1, 128/G) is a 128-row tile.
    const uint64_t qdims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(G),
                               static_cast<uint64_t>(a.Hkv), static_cast<uint64_t>(q.tokens)};
    const uint64_t qstrides[3] = {static_cast<uint64_t>(a.D) * 2, static_cast<uint64_t>(G) * a.D * 2,
                                  static_cast<uint64_t>(a.Hq) * a.D * 2};
    const uint32_t qbox[4] = {64u, static_cast<uint32_t>(G), 1u, static_cast<uint32_t>(kBM / G)};
    if (!encode_tmap_4d(&sp.tm_q, q.q, qdims, qstrides, qbox)) return cudaErrorInvalidValue;
    if (q.n_priv > 0) {
      const uint64_t dims[4] = {static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.Hkv),
                                static_cast<uint64_t>(q.n_priv), 1};
      const uint64_t strides[3] = {static_cast<uint64_t>(a.D) * 2,
                                   static_cast<uint64_t>(a.Hkv) * a.D * 2,
                                   static_cast<uint64_t>(q.n_priv) * a.Hkv * a.D * 2};
      const uint32_t box[4] = {64u, 1u, static_cast<uint32_t>(kBN), 1u};
      if (!encode_tmap_4d(&sp.tm_kp, q.k_priv, dims, strides, box)) return cudaErrorInvalidValue;
      if (!encode_tmap_4d(&sp.tm_vp, q.v_priv, dims, strides, box)) return cudaErrorInvalidValue;
    }
    sp.out = static_cast<__nv_bfloat16*>(q.out);
    sp.tail_len = q.tail_len;
    sp.n_priv = q.n_priv;
    sp.rows = q.tokens * G;
    sp.m_tiles = (sp.rows + kBM - 1) / kBM;
    sp.row_base = m_total * kBM;
    sp.tok_per_stream = q.tok_per_stream > 0 ? q.tok_per_stream : 1;
    sp.tail_cap = q.tail_cap;
    sp.state_tokens = q.state_tokens;
    m_total += sp.m_tiles;
    const int t = t_shared + (q.n_priv + kBN - 1) / kBN;
    t_max = t > t_max ? t : t_max;
  }
  if (nseg == 1) prm.seg[1].row_base = m_total * kBM;   // no second segment
  if (!a.pin_k_tiles) {
    prm.tm_k[0] = *a.tm_pin_k;
    prm.tm_v[0] = *a.tm_pin_v;
  }
  if (!a.win_k_tiles) {
    prm.tm_k[1] = *a.tm_slide_k;
    prm.tm_v[1] = *a.tm_slide_v;
  }
  prm.k_tiles[0] = static_cast<const uint8_t*>(a.pin_k_tiles);
  prm.v_tiles[0] = static_cast<const uint8_t*>(a.pin_v_tiles);
  prm.k_tiles[1] = static_cast<const uint8_t*>(a.win_k_tiles);
  prm.v_tiles[1] = static_cast<const uint8_t*>(a.win_v_tiles);
  prm.head_stride[0] = a.pin_head_stride;
  prm.head_stride[1] = a.win_head_stride;
  prm.part_o = a.part_o;
  prm.part_ml = a.part_ml;
  prm.st = a.st;
  prm.err = a.err;
  prm.layer = a.layer;
  prm.P = a.P;
  prm.F = a.F;
  prm.N = a.N;
  prm.slots = a.slots > 0 ? a.slots : a.N;
  prm.Hq = a.Hq;
  prm.G = G;
  prm.rows_pad = m_total * kBM;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a.D)));
  // Split the key sequence: about kTilesPerSplit 64-key tiles per CTA (the
  // per-CTA set-up, Q load and partial write amortise over them), at most one
  // wave of CTAs.
  const int wave = a.num_sms / (m_total * a.Hkv);
  int splits = a.forced_splits > 0 ? a.forced_splits : (t_max + kTilesPerSplit - 1) / kTilesPerSplit;
  if (a.forced_splits <= 0 && splits > wave) splits = wave;
  splits = splits < 1 ? 1 : splits;
  splits = splits > t_max ? t_max : splits;
  int cmax = 1;
  switch (a.D) {
    case 64: cmax = max_cluster_splits<64>(); break;
    case 128: cmax = max_cluster_splits<128>(); break;
    case 256: cmax = max_cluster_splits<256>(); break;
    default: return cudaErrorInvalidValue;
  }
  // Prefer an on-chip (cluster) merge: cap the automatic split count there.
  if (a.forced_splits <= 0 && splits > cmax && cmax >= 2) splits = cmax;
  const bool fused = splits >= 2 && splits <= cmax;
  if (!fused) splits = splits > a.max_splits ? a.max_splits : splits;
  splits = splits < 1 ? 1 : splits;
  prm.n_splits = splits;
  prm.fused = fused ? 1 : 0;
  if (used_splits) *used_splits = splits;
  switch (a.D) {
    case 64: return launch_one<64>(prm, m_total, a.Hkv, s);
    case 128: return launch_one<128>(prm, m_total, a.Hkv, s);
    case 256: return launch_one<256>(prm, m_total, a.Hkv, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rx
