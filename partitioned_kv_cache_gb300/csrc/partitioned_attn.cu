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
//     Short key loops use one ring with K and V alternating; longer ones (the
//     deeper build) keep K and V in separate rings, each filled by its own
//     producer lane, so that a K load never waits for the P V that frees a
//     V slot.
//   * S = Q K^T and O += P V run on tcgen05 with both accumulators in TMEM
//     (O: D columns; S: two 64-column buffers).  One thread per row does the
//     online softmax in the exp2 domain and writes P (bf16) back to TMEM (two
//     32-column buffers), where P V reads its A operand: P never touches
//     shared memory.  O is rescaled in TMEM only when the running maximum
//     grows by more than 2^8 (otherwise the stale maximum is kept: exact after
//     the final division by the row sum).
//   * The key sequence is split across CTAs (gridDim.y).  Every split writes
//     its normalised partial O / l (bf16) and fp32 (m, l) to an exchange area
//     in L2.  When the splits of an M-tile form one thread-block cluster (up
//     to kMaxClusterSplits), the cluster passes one barrier and each CTA then
//     combines a block of rows from all C partials and writes the bf16
//     output: no second kernel runs.  Beyond that size a combine kernel reads
//     the same exchange area.  With a single split the CTA writes the bf16
//     output directly.
//   * The output columns of a (tile, split) may be shared by dparts CTAs: each
//     computes S in full but loads only its D/dparts columns of V, so its key
//     loop moves fewer bytes and its partial is dparts times smaller.
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

#include "norm_row.cuh"
#include "partition.h"
#include "rx_internal.h"
#include "sm103_ptx.cuh"

namespace rx {
namespace {

constexpr int kThreads = 224;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// Shared memory for the K/V ring, in two sizes (separate builds of the
// kernel, each also built per merge shape; see attn_kernel's CM): 128 KB for
// key loops of at most kShallowTiles tiles per CTA, which have nothing to
// gain from a deeper ring and run faster with the smaller allocation, and
// 160 KB for longer loops, which prefetch one tile deeper and split it into
// a K ring (3/5 of it) and a V ring.
constexpr int kRingShallowKB = 128;
constexpr int kRingDeepKB = 160;
constexpr int kShallowTiles = 4;
constexpr int kMergeWide = 32;               // build tags: see attn_kernel's CM
constexpr int kNoClusterMerge = 0;

template <int D, int RING_KB>
struct Layout {
  static constexpr int KB = D / 64;                 // 64-column blocks of the head dim
  static constexpr int Q_BLOCK = kBM * 128;         // one 64-column block of Q: 128 rows x 128 B
  static constexpr int Q_BYTES = KB * Q_BLOCK;
  static constexpr int TILE = static_cast<int>(tile_bytes(D));   // one K or V tile: [KB][64][128 B]
  static constexpr bool SPLIT = RING_KB > kRingShallowKB;   // separate K and V rings
  static constexpr int RING = RING_KB * 1024;
  static constexpr int NS_FIT = RING / TILE;
  static constexpr int NS = NS_FIT > 16 ? 16 : NS_FIT;     // single ring: slots (4 at D = 256)
  static constexpr int NK_FIT = (RING * 3 / 5) / TILE;
  static constexpr int NK = NK_FIT > 16 ? 16 : NK_FIT;     // split: K slots (3 at D = 256)
  static constexpr int V_BYTES = RING - NK * TILE;          // split: V ring, cut at run time into
                                                            // slots of one CTA's V columns
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + Q_BYTES;          // the single ring, or the K ring
  static constexpr int OFF_VRING = OFF_RING + NK * TILE;    // split: the V ring
  static constexpr int OFF_BAR = OFF_RING + (SPLIT ? RING : NS * TILE);
  static constexpr int OFF_MISC = OFF_BAR + 80 * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr int ALLOC = BYTES + 1024;        // slack for 1024-byte alignment
  static constexpr int TMEM_COLS = (D + 3 * kBN) <= 256 ? 256 : 512;   // O, S x 2, P x 2
  static_assert(ALLOC <= 232448, "shared memory budget");
  static_assert(SPLIT ? (NK >= 2 && V_BYTES >= 2 * TILE) : (NS >= 4), "ring depth");
};

// Barrier indices: Q, ring full / empty [16] (the single ring, or the K ring),
// V ring full / empty [16], S full[2], P full[2], PV done[2], drain.
enum : int {
  B_Q = 0, B_FULL = 1, B_EMPTY = 17, B_VFULL = 33, B_VEMPTY = 49, B_SF = 65, B_PF = 67, B_PV = 69,
  B_DRAIN = 71
};

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

// An AdaRMSNorm job run by the launch's softmax warps (NormJob, device form).
struct NormParams {
  const uint4* x;
  const float* gamma;
  uint4* y;
  int rows;
  int nv;        // 16-byte vectors per row (d / 8)
  float inv_d;
  float eps;
};

struct AttnParams {
  SegParams seg[2];
  NormParams norm[kMaxNormJobs];
  int n_norm_rows;       // rows of all norm jobs (0: none)
  CUtensorMap tm_k[2];   // pin, window when not pre-tiled: (D, Hkv, keys, layers), box (64, 1, 64, 1)
  CUtensorMap tm_v[2];
  const uint8_t* k_tiles[2];   // pre-tiled pin / window of (layer, head 0); null = tensor map
  const uint8_t* v_tiles[2];
  long long head_stride[2];    // bytes between heads of a tiled region
  void* xchg;            // split partials: see the split merge in attn_kernel
  const DevState* st;
  int* err;
  int layer;
  int P, F, N, slots;    // pinned tokens; window: tokens per frame, frames, frame slots
  int Hq, G;
  int rows_pad;          // workspace rows of all segments
  int n_splits;
  int dparts;            // output columns split over dparts CTAs (each computes S in full)
  int fused;             // 1: the splits of an M-tile form a cluster and merge on chip
  int inject_tx;         // test aid: extra bytes CTA 0 expects on its first K tile
  int prefetch_l2;       // L2 prefetch before the dependency wait: Q and the split's first
                         // prefetch_l2 key tiles (0: none)
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

// O += P V with P (the A operand) read from tensor memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
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

// All lanes wait on the barrier, then agree: the warp proceeds only if every
// lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  const bool ok = mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Exchange area of the split partials, per (tile, head, column share) unit
// u = blockIdx.z * gridDim.x + blockIdx.x: O [splits][D/dparts/8 pieces][128
// rows] of 16 bytes for every unit, then (m, l) [splits][128] for every unit.
__device__ __forceinline__ uint4* xchg_o(const AttnParams& p, int DV, int split) {
  const size_t u = static_cast<size_t>(blockIdx.z) * gridDim.x + blockIdx.x;
  return reinterpret_cast<uint4*>(p.xchg) + (u * p.n_splits + split) * (DV / 8) * kBM;
}
__device__ __forceinline__ float2* xchg_ml(const AttnParams& p, int DV, int split) {
  const size_t u = static_cast<size_t>(blockIdx.z) * gridDim.x + blockIdx.x;
  return reinterpret_cast<float2*>(reinterpret_cast<uint4*>(p.xchg) +
                                   static_cast<size_t>(gridDim.x) * gridDim.z * p.n_splits * (DV / 8) * kBM) +
         (u * p.n_splits + split) * kBM;
}

// The cluster merge's last step: rows [r0, r0 + nr) of the tile from the C
// partial slots of the cluster.  An item is PP adjacent 16-byte pieces of one
// row; items go rows fastest (a warp's loads of one split are consecutive
// 16-byte rows).  Each thread takes U items per pass and loads the CM >= C
// partial pieces and (m, l) of each together (splits >= C re-read split C-1
// and weigh 0), U * CM * PP pieces in flight.  The weight of split s is
// 2^(m_s - M) l_s / sum, as the partials are O_s / l_s.
template <int D, int U, int CM, int PP = 1>
__device__ __forceinline__ void cluster_combine(const uint4* xo, const float2* xml, int C, int kPieces, int r0,
                                                int nr, int mt, const SegParams& sg, int Hq, int G, int g,
                                                int dcol) {
  const int items = nr * (kPieces / PP);
  for (int base = threadIdx.x; base < items; base += kThreads * U) {
    uint4 pv[U][PP][CM];
    float2 ml[U][CM];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int item = min(base + q * kThreads, items - 1);   // past the end: re-read, not stored
      const int i = item % nr, k = item / nr * PP;
      const uint4* src = xo + static_cast<size_t>(k) * kBM + r0 + i;
#pragma unroll
      for (int s2 = 0; s2 < CM; ++s2) {
        const int sc = min(s2, C - 1);
#pragma unroll
        for (int pp = 0; pp < PP; ++pp)
          pv[q][pp][s2] = __ldcg(src + static_cast<size_t>(sc) * kPieces * kBM + pp * kBM);
        ml[q][s2] = __ldcg(xml + sc * kBM + r0 + i);
      }
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int item = base + q * kThreads;
      const int i = item % nr, k = item / nr * PP;
      const int Rs = mt * kBM + r0 + i;
      if (item >= items || Rs >= sg.rows) continue;
      float M = -INFINITY;
#pragma unroll
      for (int s2 = 0; s2 < CM; ++s2)
        if (s2 < C && ml[q][s2].y > 0.f) M = fmaxf(M, ml[q][s2].x);
      float w[CM];
      float L = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < CM; ++s2) {
        w[s2] = s2 < C && ml[q][s2].y > 0.f ? exp2f(ml[q][s2].x - M) * ml[q][s2].y : 0.f;
        L += w[s2];
      }
      const float invL = L > 0.f ? 1.f / L : 0.f;   // a row with no key at all gets zeros
      const int tok = Rs / G, h = g * G + Rs % G;
#pragma unroll
      for (int pp = 0; pp < PP; ++pp) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < CM; ++s2) {
          const float ws = w[s2] * invL;
          const uint32_t vv[4] = {pv[q][pp][s2].x, pv[q][pp][s2].y, pv[q][pp][s2].z, pv[q][pp][s2].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = fmaf(ws, __uint_as_float(vv[e] << 16), acc[2 * e]);
            acc[2 * e + 1] = fmaf(ws, __uint_as_float(vv[e] & 0xFFFF0000u), acc[2 * e + 1]);
          }
        }
        *reinterpret_cast<uint4*>(sg.out + (static_cast<size_t>(tok) * Hq + h) * D + dcol + (k + pp) * 8) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                       pack_bf16x2(acc[6], acc[7]));
      }
    }
  }
}

// Norm rows of the launch's jobs, in job order, are shared out over the
// grid's CTAs and, within a CTA, over its four softmax warps: row r goes to
// CTA r mod nCTA, warp (r / nCTA) mod 4.  (The warp's first row: r = cta +
// nCTA * sw.)
__device__ __forceinline__ int first_norm_row(int sw) {
  const int ncta = static_cast<int>(gridDim.x * gridDim.y * gridDim.z);
  const int cta = static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
  return cta + ncta * sw;
}

// The norm rows of softmax warp sw (0..3) of this CTA.  They run after the
// dependency wait, while the warp would otherwise wait for its first score
// tile (the producer has issued Q and the first key tile by then).
__device__ __noinline__ void run_norm_rows(const AttnParams& p, int sw, int lane) {
  const int ncta = static_cast<int>(gridDim.x * gridDim.y * gridDim.z);
  for (int r = first_norm_row(sw); r < p.n_norm_rows; r += 4 * ncta) {
    const int j = r < p.norm[0].rows ? 0 : 1;
    const NormParams& nj = p.norm[j];
    const size_t row = static_cast<size_t>(j ? r - p.norm[0].rows : r);
    if (nj.nv <= 128)
      adarmsnorm_row<4>(nj.x + row * nj.nv, nj.gamma, nj.nv, nj.inv_d, nj.eps, nj.y + row * nj.nv, lane);
    else
      adarmsnorm_row<0>(nj.x + row * nj.nv, nj.gamma, nj.nv, nj.inv_d, nj.eps, nj.y + row * nj.nv, lane);
  }
}

// CM: the most splits a launch of this build may merge in a cluster
// (kMaxClusterSplits, or a small count whose combine keeps several rows'
// loads in flight per thread), or kMergeWide: up to kMaxClusterSplits splits
// whose rows hold more (row, piece) items than the CTA has threads, taken two
// pieces per thread so that one pass finishes them; or kNoClusterMerge, for
// launches whose splits are merged by attn_combine_kernel.
template <int D, int RING_KB, int CM = kMaxClusterSplits>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  using Lay = Layout<D, RING_KB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + Lay::OFF_Q;
  const uint32_t sRing = base + Lay::OFF_RING;
  const uint32_t sVring = base + Lay::OFF_VRING;
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
  const int g = blockIdx.z / p.dparts;                 // K/V head
  const int DV = D / p.dparts;                         // output columns of this CTA
  const int dcol = (blockIdx.z % p.dparts) * DV;       // first output column

  if (threadIdx.x == 0) {
    mbar_init(BAR(B_Q), 1);
    for (int i = 0; i < 16; ++i) {
      mbar_init(BAR(B_FULL + i), 1);
      mbar_init(BAR(B_EMPTY + i), 1);
      mbar_init(BAR(B_VFULL + i), 1);
      mbar_init(BAR(B_VEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_SF + i), 1);
      mbar_init(BAR(B_PF + i), 128);
      mbar_init(BAR(B_PV + i), 1);
    }
    mbar_init(BAR(B_DRAIN), 2);   // one commit from each MMA issuer
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
    if (p.prefetch_l2) {
      // A store larger than L2 sends every key tile from DRAM, and the
      // caller's Q usually too.  Ask for this CTA's Q tile and its split's
      // first K and V tile to be fetched into L2 now, while the previous
      // kernel drains.  A prefetch is a hint with no effect on what any load
      // returns, so it may run before the dependency wait; the ring state is
      // not read here (it may still be changing), and the first tile is the
      // one of a full window, clamped inside the regions.
      for (int kb = 0; kb < Lay::KB; ++kb) tma_prefetch_l2_4d(&sg.tm_q, kb * 64, 0, g, mt * (kBM / p.G));
      const bool spare = p.slots > p.N;
      const int wl = (spare ? p.slots - 1 : p.N) * p.F;
      const int np = (p.P + kBN - 1) / kBN, nw = (wl + kBN - 1) / kBN, nd = (sg.n_priv + kBN - 1) / kBN;
      const int T = np + nw + nd;
      const int tf = static_cast<int>(static_cast<unsigned>(split * T) / static_cast<unsigned>(p.n_splits));
      const int tl = static_cast<int>(static_cast<unsigned>((split + 1) * T) / static_cast<unsigned>(p.n_splits));
      for (int t = tf; t < tl && t < tf + p.prefetch_l2; ++t) {
        const TileInfo ti = tile_at(t, np, nw, p.P, wl, sg.n_priv, 0, 0);
        const uint8_t* kt = ti.region < 2 ? p.k_tiles[ti.region] : nullptr;
        const uint8_t* vt = ti.region < 2 ? p.v_tiles[ti.region] : nullptr;
        if (kt && vt) {
          const long long off = g * p.head_stride[ti.region] + static_cast<long long>(ti.phys0 / kBN) * Lay::TILE;
          bulk_prefetch_l2(kt + off, static_cast<uint32_t>(Lay::TILE));
          bulk_prefetch_l2(vt + off + dcol * 128, static_cast<uint32_t>(DV) * 128u);
        } else if (ti.region == 2) {
          for (int kb = 0; kb < Lay::KB; ++kb) tma_prefetch_l2_4d(&sg.tm_kp, kb * 64, g, ti.phys0, 0);
          for (int kb = dcol / 64; kb < (dcol + DV) / 64; ++kb) tma_prefetch_l2_4d(&sg.tm_vp, kb * 64, g, ti.phys0, 0);
        }
      }
    }
  }
  // Norm rows of this CTA's softmax warps: fetch the first row and its gamma
  // into L2 while the previous kernel drains (a hint, safe before the wait).
  if (p.n_norm_rows > 0 && warp >= 2 && warp <= 5 && lane == 0) {
    const int r = first_norm_row(warp - 2);
    if (r < p.n_norm_rows) {
      const int j = r < p.norm[0].rows ? 0 : 1;
      const NormParams& nj = p.norm[j];
      const size_t row = static_cast<size_t>(j ? r - p.norm[0].rows : r);
      bulk_prefetch_l2(nj.x + row * nj.nv, static_cast<uint32_t>(nj.nv) * 16u);
      bulk_prefetch_l2(nj.gamma, static_cast<uint32_t>(nj.nv) * 32u);
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
  // even while a push on another stream is publishing).  Pushes in stream
  // order completed before the dependency wait above; only a cache with a
  // spare slot takes pushes concurrently, and there the frame data must be
  // ordered after the snapshot.
  // One thread per CTA reads the word (every CTA of the grid reads the same
  // line) and hands it to the others through shared memory.
  volatile int* ring_word = reinterpret_cast<volatile int*>(gbase + Lay::OFF_MISC + 8);
  if (threadIdx.x == 0) {
    int h = 0, v = 0;
    load_ring_state(p.st, &h, &v);
    if (p.slots > p.N) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    ring_word[0] = h;
    ring_word[1] = v;
  }
  __syncthreads();
  const int head = ring_word[0], valid = ring_word[1];
  // With a spare slot and a full ring the window is every slot but `head`.
  const bool hole = p.slots > p.N && valid == p.N;
  const int win_len = hole ? (p.slots - 1) * p.F : valid * p.F;
  const int hole0 = hole ? head * p.F / kBN : 0;
  const int hole_n = hole ? p.F / kBN : 0;
  const int nt_pin = (p.P + kBN - 1) / kBN;
  const int nt_win = (win_len + kBN - 1) / kBN;
  const int nt_dyn = (sg.n_priv + kBN - 1) / kBN;
  const int T = nt_pin + nt_win + nt_dyn;
  const int t0 = static_cast<int>(static_cast<unsigned>(split * T) / static_cast<unsigned>(p.n_splits));
  const int t1 = static_cast<int>(static_cast<unsigned>((split + 1) * T) / static_cast<unsigned>(p.n_splits));
  const int n = t1 - t0;

  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem;                               // columns [0, D)
  const uint32_t tS = tmem + static_cast<uint32_t>(D);    // two buffers of 64 columns
  const uint32_t tP = tS + 2 * kBN;                       // two P buffers of 32 columns (bf16 pairs)

  const int qtok = kBM / p.G;   // query tokens per tile
  const int ns = Lay::NS;                                    // single ring: slots
  const uint32_t vtile = static_cast<uint32_t>(DV) * 128;      // split: one V slot
  const int nv_fit = Lay::SPLIT ? static_cast<int>(Lay::V_BYTES / vtile) : 2;
  const int nv = nv_fit > 16 ? 16 : nv_fit;                  // split: V slots
  // The softmax thread's final row state, for the cluster merge.
  float fin_m = -INFINITY, fin_l = 0.f;
  bool fin_have = false;

  // One K (kv = 0) or V (kv = 1) tile into shared memory at dst, counted on
  // bar, which expects `extra` bytes more than the tile (a test aid: they
  // never arrive, so the waits on bar run out).
  auto issue_tile = [&](const TileInfo& ti, int kv, uint32_t dst, uint32_t bar, uint32_t extra) {
    // K: all D/64 column blocks; V: only the blocks of this CTA's columns.
    const int kb0 = kv ? dcol / 64 : 0;
    const int nkb = kv ? DV / 64 : Lay::KB;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nkb * 8192) + extra);
    const uint8_t* tiles = ti.region < 2 ? (kv ? p.v_tiles[ti.region] : p.k_tiles[ti.region]) : nullptr;
    if (tiles) {
      bulk_load(dst, tiles + g * p.head_stride[ti.region] + static_cast<long long>(ti.phys0 / kBN) * Lay::TILE +
                         kb0 * 8192,
                static_cast<uint32_t>(nkb * 8192), bar);
    } else {
      const int lay = ti.region == 2 ? 0 : p.layer;
      const CUtensorMap* tm = ti.region == 2 ? (kv ? &sg.tm_vp : &sg.tm_kp)
                                             : (kv ? &p.tm_v[ti.region] : &p.tm_k[ti.region]);
      for (int kb = 0; kb < nkb; ++kb)
        tma_load_4d(dst + kb * 8192, tm, (kb0 + kb) * 64, g, ti.phys0, lay, bar);
    }
  };

  if (n > 0 && warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues Q first.  Single ring: lane 0 then issues K_0, V_0, K_1,
    // V_1, ...; item i uses slot i % ns.  Split rings: lane 0 issues K_j into
    // K slot j % NK and lane 1 V_j into V slot j % nv, independently.
    const int kv_lane = Lay::SPLIT ? lane : 0;   // split: 0 = K, 1 = V
    if (lane == 0 || (Lay::SPLIT && lane == 1)) {
      const int rs = Lay::SPLIT ? (kv_lane ? nv : Lay::NK) : ns;
      const int bfull = kv_lane ? B_VFULL : B_FULL, bempty = kv_lane ? B_VEMPTY : B_EMPTY;
      const uint32_t rbase = kv_lane ? sVring : sRing;
      const uint32_t rstride = kv_lane ? vtile : static_cast<uint32_t>(Lay::TILE);
      const int per_tile = Lay::SPLIT ? 1 : 2;   // items per key tile in this lane's ring
      if (lane == 0) {
        mbar_arrive_expect_tx(BAR(B_Q), Lay::Q_BYTES);
        for (int kb = 0; kb < Lay::KB; ++kb)
          tma_load_4d(sQ + kb * Lay::Q_BLOCK, &sg.tm_q, kb * 64, 0, g, mt * qtok, BAR(B_Q));
      }
      int issued = 0;
      int slot = 0, rnd = 0;   // issued % rs and issued / rs, kept without dividing
      bool stop = false;
      for (int j = 0; j < n && !stop; ++j) {
        const TileInfo ti = tile_at(t0 + j, nt_pin, nt_win, p.P, win_len, sg.n_priv, hole0, hole_n);
        for (int k = 0; k < per_tile; ++k) {
          if (rnd > 0 && !mbar_wait(BAR(bempty + slot), (rnd - 1) & 1, abort_flag)) {
            stop = true;
            break;
          }
          const bool first_k = issued == 0 && lane == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
          issue_tile(ti, Lay::SPLIT ? kv_lane : k, rbase + slot * rstride, BAR(bfull + slot),
                     first_k ? static_cast<uint32_t>(p.inject_tx) : 0u);
          ++issued;
          if (++slot == rs) {
            slot = 0;
            ++rnd;
          }
        }
      }
      // Every copy issued must land before the CTA exits, even after an abort.
      volatile int no_abort = 0;
      if (lane == 0) mbar_wait(BAR(B_Q), 0, &no_abort);
      for (int it = issued - rs < 0 ? 0 : issued - rs; it < issued; ++it)
        mbar_wait(BAR(bfull + it % rs), (it / rs) & 1, &no_abort);
    }
  } else if (n > 0 && warp == 1) {
    // ------------------------------------------------------------ Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false, false);
      bool ok = mbar_wait(BAR(B_Q), 0, abort_flag);
      // K_j: item 2j of the single ring, or item j of the K ring
      constexpr int kStep = Lay::SPLIT ? 1 : 2;
      constexpr int kSlots = Lay::SPLIT ? Lay::NK : Lay::NS;
      int slot = 0, rnd = 0;
      for (int j = 0; ok && j < n; ++j) {
        const int st = j & 1;
        // S buffer st last held S_{j-2}; the softmax is done with it once it
        // has published P_{j-2}.
        if (j >= 2 && !mbar_wait(BAR(B_PF + st), ((j - 2) >> 1) & 1, abort_flag)) break;
        if (!mbar_wait(BAR(B_FULL + slot), rnd & 1, abort_flag)) break;
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
        if ((slot += kStep) >= kSlots) {
          slot -= kSlots;
          ++rnd;
        }
      }
      // No tensor-core work may be in flight when TMEM is released.
      umma_commit(BAR(B_DRAIN));
      volatile int no_abort = 0;
      mbar_wait(BAR(B_DRAIN), 0, &no_abort);
    }
  } else if (n > 0 && warp == 6) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      const uint32_t kIdescO = idesc_bf16_f32(kBM, DV, false, true);
      // V_j: item 2j + 1 of the single ring, or item j of the V ring
      const int vStep = Lay::SPLIT ? 1 : 2;
      const int vSlots = Lay::SPLIT ? nv : ns;
      const int bvfull = Lay::SPLIT ? B_VFULL : B_FULL, bvempty = Lay::SPLIT ? B_VEMPTY : B_EMPTY;
      const uint32_t vbase = Lay::SPLIT ? sVring : sRing;
      const uint32_t vstride = Lay::SPLIT ? vtile : static_cast<uint32_t>(Lay::TILE);
      int slot = Lay::SPLIT ? 0 : 1, rnd = 0;
      for (int j = 0; j < n; ++j) {
        const int st = j & 1;
        if (!mbar_wait(BAR(B_PF + st), (j >> 1) & 1, abort_flag)) break;
        if (!mbar_wait(BAR(bvfull + slot), rnd & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t vt = vbase + slot * vstride;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // A = P (K-major, 128 x 64 keys); B = V tile read MN-major: D runs
          // along the 128-byte rows, 64-column blocks 8 KB apart (LBO), 8-key
          // groups 1 KB apart (SBO), 16 keys = 2 KB per K step.
          const uint64_t b = sdesc_sw128(vt + kk * 16 * 128, 8192, 1024);
          umma_bf16_ts(tO, tP + st * (kBN / 2) + kk * 8, b, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(BAR(bvempty + slot));
        umma_commit(BAR(B_PV + st));
        if ((slot += vStep) >= vSlots) {
          slot -= vSlots;
          ++rnd;
        }
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
    if (p.n_norm_rows > 0 && warp <= 5) run_norm_rows(p, warp - 2, lane);
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
        for (int c = 0; c < DV; c += 32) {
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
      tmem_st32(tP + st * (kBN / 2) + lane_off, reinterpret_cast<const float*>(pk));
      tc_fence_before();
      mbar_arrive(BAR(B_PF + st));
    }
    if (ok) ok = warp_wait(BAR(B_PV + ((n - 1) & 1)), ((n - 1) >> 1) & 1, abort_flag);
    if (ok) {
      tc_fence_after();
      if (p.n_splits == 1) {
        const int tok = Rs / p.G;
        const int h = g * p.G + Rs % p.G;
        __nv_bfloat16* dst = sg.out + (static_cast<size_t>(tok) * p.Hq + h) * D + dcol;
        const float inv = l > 0.f ? 1.f / l : 0.f;   // a row with no key at all gets zeros
#pragma unroll 1
        for (int c = 0; c < DV; c += 64) {   // 64 columns per TMEM load: half the round trips
          float o[64];
          tmem_ld64(tO + c + lane_off, o);
          if (row_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_uint4(pack_bf16x2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                 pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                 pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                 pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
          }
        }
      } else if (p.fused) {
        fin_m = m_used;   // O stays in TMEM until the merge
        fin_l = l;
        fin_have = true;
      } else {
        // More splits than a cluster: this row's partial goes to the exchange
        // area in the layout of the cluster merge below, and
        // attn_combine_kernel combines the splits after the grid.
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4* dst = xchg_o(p, DV, split) + row;
#pragma unroll 1
        for (int c = 0; c < DV; c += 64) {   // 64 columns per TMEM load: half the round trips
          float o[64];
          tmem_ld64(tO + c + lane_off, o);
          if (row_valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[static_cast<size_t>(c / 8 + q) * kBM] =
                  make_uint4(pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                             pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                             pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                             pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
          }
        }
        if (row_valid) xchg_ml(p, DV, split)[row] = make_float2(m_used, l);
      }
    } else if (!p.fused && p.n_splits > 1 && row_valid) {
      // A split without keys (or one that gave up): zeros and l = 0, which
      // the combine skips.
      uint4* dst = xchg_o(p, DV, split) + row;
      for (int c = 0; c < DV / 8; ++c) dst[static_cast<size_t>(c) * kBM] = make_uint4(0u, 0u, 0u, 0u);
      xchg_ml(p, DV, split)[row] = make_float2(-INFINITY, 0.f);
    }
  }

  if constexpr (CM != kNoClusterMerge) if (p.fused) {
    // ---------------------------------------------------------- cluster merge
    // The C splits of this (tile, head, column share) exchange their partials
    // through L2: each softmax thread writes its row's normalised partial
    // O / l (bf16) and (m, l) to this split's slot of the exchange area, one
    // cluster barrier, then cluster CTA o combines rows [o*per, (o+1)*per) of
    // the C slots and writes the bf16 output.  Exchange layout per cluster:
    // O [C][D/8 / dparts pieces][128 rows] of 16 bytes (a warp's store is 512
    // contiguous bytes), then (m, l) [C][128].  All threads of all CTAs of
    // the cluster pass the barrier, whatever path they took above.
    const int kPieces = DV / 8;      // 16-byte pieces of a row
    const int C = p.n_splits;
    const int rank = static_cast<int>(cluster_ctarank());
    const size_t cid = static_cast<size_t>(blockIdx.z) * gridDim.x + blockIdx.x;
    uint4* xo = reinterpret_cast<uint4*>(p.xchg) + cid * C * kPieces * kBM;
    float2* xml = reinterpret_cast<float2*>(reinterpret_cast<uint4*>(p.xchg) +
                                            static_cast<size_t>(gridDim.x) * gridDim.z * C * kPieces * kBM) +
                  cid * C * kBM;
    if (warp >= 2 && warp <= 5) {
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
      const bool valid = mt * kBM + row < sg.rows;   // padding rows are never read
      const float inv = fin_l > 0.f ? 1.f / fin_l : 0.f;
      uint4* dst = xo + static_cast<size_t>(rank) * kPieces * kBM + row;
#pragma unroll 1
      for (int c = 0; c < DV; c += 64) {   // 64 columns per TMEM load: half the round trips
        float o[64];
        if (fin_have) {   // warp-uniform: the TMEM load is warp-collective
          tmem_ld64(tO + c + lane_off, o);
        } else {
#pragma unroll
          for (int e = 0; e < 64; ++e) o[e] = 0.f;
        }
        if (valid) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[static_cast<size_t>(c / 8 + q) * kBM] =
                make_uint4(pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                           pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                           pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                           pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
        }
      }
      if (valid) xml[rank * kBM + row] = make_float2(fin_have ? fin_m : -INFINITY, fin_have ? fin_l : 0.f);
    }
    __syncwarp();
    cluster_sync_all();   // release / acquire: the slots are visible to the whole cluster
    if constexpr (CM == kMergeWide) {
      const int per = (kBM + C - 1) / C;
      const int r0 = rank * per;
      const int nr = max(0, min(per, kBM - r0));
      cluster_combine<D, 1, kMaxClusterSplits, 2>(xo, xml, C, kPieces, r0, nr, mt, sg, p.Hq, p.G, g, dcol);
    } else if constexpr (CM < kMaxClusterSplits) {
      // The build for clusters of at most CM splits: each CTA finishes many
      // rows, so a thread takes several items per pass.
      const int per = (kBM + C - 1) / C;
      const int r0 = rank * per;
      const int nr = max(0, min(per, kBM - r0));
      // Two pieces of a row per item (one (m, l) load for both), and enough
      // items per thread that the 64, 32 or 22 rows x 32 pieces of a
      // cluster of 2, 4 or 6-8 splits at D = 256 take one pass.
      constexpr int kU = CM == 2 ? 5 : CM == 4 ? 3 : 2;
      cluster_combine<D, kU, CM, 2>(xo, xml, C, kPieces, r0, nr, mt, sg, p.Hq, p.G, g, dcol);
    } else
    // Every thread of the CTA finishes at most one (piece k, row i) item per
    // pass, rows fastest (a warp's loads of one split are consecutive 16-byte
    // rows).  The C partial pieces and the C (m, l) of the row are loaded
    // together (splits >= C re-read split C-1 and weigh 0); the weight of
    // split s is 2^(m_s - M) l_s / sum, as the partials are O_s / l_s.
    {
      const int per = (kBM + C - 1) / C;
      const int r0 = rank * per;
      const int nr = max(0, min(per, kBM - r0));            // rows this CTA finishes
      for (int item = threadIdx.x; item < nr * kPieces; item += kThreads) {
        const int i = item % nr, k = item / nr;
        const int Rs = mt * kBM + r0 + i;
        if (Rs >= sg.rows) continue;
        const uint4* src = xo + static_cast<size_t>(k) * kBM + r0 + i;
        uint4 pv[kMaxClusterSplits];
        float2 ml[kMaxClusterSplits];
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
          const int sc = min(s2, C - 1);
          pv[s2] = __ldcg(src + static_cast<size_t>(sc) * kPieces * kBM);
          ml[s2] = __ldcg(xml + sc * kBM + r0 + i);
        }
        float M = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
          if (s2 < C && ml[s2].y > 0.f) M = fmaxf(M, ml[s2].x);
        float w[kMaxClusterSplits];
        float L = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
          w[s2] = s2 < C && ml[s2].y > 0.f ? exp2f(ml[s2].x - M) * ml[s2].y : 0.f;
          L += w[s2];
        }
        const float invL = L > 0.f ? 1.f / L : 0.f;   // a row with no key at all gets zeros
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
          const float ws = w[s2] * invL;
          const uint32_t vv[4] = {pv[s2].x, pv[s2].y, pv[s2].z, pv[s2].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = fmaf(ws, __uint_as_float(vv[e] << 16), acc[2 * e]);
            acc[2 * e + 1] = fmaf(ws, __uint_as_float(vv[e] & 0xFFFF0000u), acc[2 * e + 1]);
          }
        }
        const int tok = Rs / p.G, h = g * p.G + Rs % p.G;
        *reinterpret_cast<uint4*>(sg.out + (static_cast<size_t>(tok) * p.Hq + h) * D + dcol + k * 8) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, Lay::TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) atomicOr(p.err, kErrAttnTimeout);
}

// Combine the splits of every row when they do not form a cluster (more than
// kMaxClusterSplits of them), over the exchange area the attention grid
// wrote, with the weighting of the in-kernel merge: out = sum_s w_s O_s / l_s
// divided by sum_s w_s, where w_s = 2^(m_s - M) l_s.  A lane pair owns one
// (row, 16-byte piece): lane 2r + h takes the splits s = h, h + 2, ...  A
// warp covers 16 consecutive rows of one piece, so its load of one split
// pair is two runs of 256 contiguous bytes.  A CTA covers 16 rows x 8
// pieces (its 8 warps, one piece each), so the rows' (m, l) are fetched from
// L2 once per CTA and served to the other warps from L1.  Grid: (M-tiles of
// all segments x 8 row groups, pieces / 8, Hkv x dparts), 256 threads.  Each
// lane loads up to kCombineChunk of its splits at a time, so up to 28 splits
// are in flight per (row, piece).  More splits run with a running maximum.  The
// pair's (M, L, sums) meet by one shuffle.  Compiled with a register cap
// rather than a thread bound: 128 registers either way, but c4's call took
// 11.93 us with the bound, 11.76 us with a cap of 128 and 11.61 us with 132
// or 136 (A/Bs on one GB300).  A cap that lets it use more (140 and up)
// keeps a second combine CTA off each SM and was slower (12.0 us).  A lane
// loads up to 14 splits at a time: the 27 splits of c4's partition in one
// pass (11.75 -> 11.61 us per call against 16 at a time).
constexpr int kCombineChunk = 14;

template <int D>
__global__ void __maxnreg__(136) attn_combine_kernel(const uint4* __restrict__ xchg,
                                                           __nv_bfloat16* out0, int rows0, int m_tiles0,
                                                           __nv_bfloat16* out1, int rows1, int n_splits,
                                                           int dparts, int Hq, int G) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int DV = D / dparts;
  const int kPieces = DV / 8;
  const int mt_all = blockIdx.x >> 3;                      // M-tile among all segments
  const int m_total = gridDim.x >> 3;
  const int si = mt_all < m_tiles0 ? 0 : 1;
  const int mt = mt_all - (si ? m_tiles0 : 0);
  const int rows = si ? rows1 : rows0;
  __nv_bfloat16* out = si ? out1 : out0;
  const int lane = threadIdx.x & 31;
  const int half = lane & 1;
  const int i = (blockIdx.x & 7) * 16 + (lane >> 1);      // row within the tile
  const int k = blockIdx.y * 8 + (threadIdx.x >> 5);       // piece
  const int Rs = mt * kBM + i;
  const bool live_row = Rs < rows;   // padding rows were never written: their loads stay in the tile
  const int C = n_splits;
  const size_t cid = static_cast<size_t>(blockIdx.z) * m_total + mt_all;
  const uint4* src = xchg + cid * C * kPieces * kBM + static_cast<size_t>(k) * kBM + i;
  const float2* ml_src = reinterpret_cast<const float2*>(xchg + static_cast<size_t>(m_total) * gridDim.z * C *
                                                                    kPieces * kBM) +
                         cid * C * kBM + i;
  float M = -INFINITY, L = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int s0 = half; s0 < C; s0 += 2 * kCombineChunk) {
    uint4 pv[kCombineChunk];
    float2 ml[kCombineChunk];
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u) {   // this lane's splits s0, s0 + 2, ...
      const int s = s0 + 2 * u;
      const bool use = live_row && s < C;
      pv[u] = use ? __ldcg(src + static_cast<size_t>(s) * kPieces * kBM) : make_uint4(0u, 0u, 0u, 0u);
      ml[u] = use ? ml_src[static_cast<size_t>(s) * kBM] : make_float2(-INFINITY, 0.f);   // L1: 8 warps read it
    }
    float mc = -INFINITY;
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u)
      if (ml[u].y > 0.f) mc = fmaxf(mc, ml[u].x);
    if (mc == -INFINITY) continue;   // none of these splits saw a key
    const float Mn = fmaxf(M, mc);
    const float sc = exp2f(M - Mn);  // 0 before the first live split
    L *= sc;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= sc;
#pragma unroll
    for (int u = 0; u < kCombineChunk; ++u) {
      const float w = ml[u].y > 0.f ? exp2f(ml[u].x - Mn) * ml[u].y : 0.f;
      L += w;
      const uint32_t vv[4] = {pv[u].x, pv[u].y, pv[u].z, pv[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[2 * e] = fmaf(w, __uint_as_float(vv[e] << 16), acc[2 * e]);
        acc[2 * e + 1] = fmaf(w, __uint_as_float(vv[e] & 0xFFFF0000u), acc[2 * e + 1]);
      }
    }
    M = Mn;
  }
  // The lane pair's halves: rescale both to the larger maximum and add.
  const float Mo = __shfl_xor_sync(0xffffffffu, M, 1);
  const float Mt = fmaxf(M, Mo);
  const float f = M == -INFINITY ? 0.f : exp2f(M - Mt);
  L *= f;
  L += __shfl_xor_sync(0xffffffffu, L, 1);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    acc[e] *= f;
    acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], 1);
  }
  if (half || !live_row) return;
  const float inv = L > 0.f ? 1.f / L : 0.f;   // a row with no key at all gets zeros
  const int g = blockIdx.z / dparts, dcol = (blockIdx.z % dparts) * DV;
  const int tok = Rs / G, h = g * G + Rs % G;
  *reinterpret_cast<uint4*>(out + (static_cast<size_t>(tok) * Hq + h) * D + dcol + k * 8) =
      make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                 pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
}

template <int D, int RING_KB, int CM = kMaxClusterSplits>
cudaError_t launch_one(const AttnParams& prm, int m_tiles, int Hkv, cudaStream_t s) {
  using Lay = Layout<D, RING_KB>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_kernel<D, RING_KB, CM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    Lay::ALLOC);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(attn_kernel<D, RING_KB, CM>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess) return attr_err;
  dim3 grid(m_tiles, prm.n_splits, Hkv * prm.dparts);
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
    e = cudaLaunchKernelEx(&cfg, attn_kernel<D, RING_KB, CM>, prm);
    count_launch();
  } else {
    e = launch_k(attn_kernel<D, RING_KB, CM>, grid, dim3(kThreads), Lay::ALLOC, s, prm);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || prm.n_splits == 1 || prm.fused) return e;
  dim3 cgrid(m_tiles * 8, D / prm.dparts / 64, Hkv * prm.dparts);
  e = launch_k(attn_combine_kernel<D>, cgrid, dim3(256), 0, s, static_cast<const uint4*>(prm.xchg),
               prm.seg[0].out, prm.seg[0].rows, prm.seg[0].m_tiles, prm.seg[1].out, prm.seg[1].rows,
               prm.n_splits, prm.dparts, prm.Hq, prm.G);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The build for head dimension D: the 128 KB ring for short key loops, else
// the 160 KB ring; with the merge for clusters of at most cm splits, or the
// two-pieces-per-thread merge (cm = kMergeWide).
template <int D>
cudaError_t launch_d(const AttnParams& prm, int m_tiles, int Hkv, cudaStream_t s, bool deep, int cm) {
  if (!deep)
    return cm == kMergeWide ? launch_one<D, kRingShallowKB, kMergeWide>(prm, m_tiles, Hkv, s)
                            : launch_one<D, kRingShallowKB>(prm, m_tiles, Hkv, s);
  switch (cm) {
    case kNoClusterMerge: return launch_one<D, kRingDeepKB, kNoClusterMerge>(prm, m_tiles, Hkv, s);
    case kMergeWide: return launch_one<D, kRingDeepKB, kMergeWide>(prm, m_tiles, Hkv, s);
    case 2: return launch_one<D, kRingDeepKB, 2>(prm, m_tiles, Hkv, s);
    case 4: return launch_one<D, kRingDeepKB, 4>(prm, m_tiles, Hkv, s);
    case 8: return launch_one<D, kRingDeepKB, 8>(prm, m_tiles, Hkv, s);
    default: return launch_one<D, kRingDeepKB>(prm, m_tiles, Hkv, s);
  }
}

// How many clusters of c attention CTAs (one per SM) the device can hold at
// once, for c = 1..kMaxClusterSplits (index c); 0 where clusters of that size
// cannot be scheduled.  Clusters live within one GPC, so this is not simply
// SMs / c.  Queried once per head dimension.
template <int D, int RING_KB>
const int* cluster_capacity() {
  static int cap[kMaxClusterSplits + 1];
  static bool done = false;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (done) return cap;
  cudaFuncSetAttribute(attn_kernel<D, RING_KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       Layout<D, RING_KB>::ALLOC);
  cudaFuncSetAttribute(attn_kernel<D, RING_KB>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  cap[0] = 0;
  for (int c = 1; c <= kMaxClusterSplits; ++c) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, c, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Layout<D, RING_KB>::ALLOC;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = c;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    cap[c] = cudaOccupancyMaxActiveClusters(&n, attn_kernel<D, RING_KB>, &cfg) == cudaSuccess ? n : 0;
  }
  cudaGetLastError();
  done = true;
  return cap;
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
  if (a.n_norms < 0 || a.n_norms > kMaxNormJobs) return cudaErrorInvalidValue;
  for (int i = 0; i < a.n_norms; ++i) {
    const NormJob& nj = a.norms[i];
    NormParams& np = prm.norm[i];
    np.x = static_cast<const uint4*>(nj.x);
    np.gamma = nj.gamma;
    np.y = static_cast<uint4*>(nj.y);
    np.rows = nj.rows;
    np.nv = nj.d / 8;
    np.inv_d = 1.0f / static_cast<float>(nj.d);
    np.eps = nj.eps;
    prm.n_norm_rows += nj.rows;
  }
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
  prm.xchg = a.xchg;
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
  // Partition (partition.h): `splits` slices of the key sequence times
  // `dparts` shares of the output columns per (tile, head), from the
  // device's cluster capacity.
  const int* cap = nullptr;
  switch (a.D) {
    case 64: cap = cluster_capacity<64, kRingDeepKB>(); break;   // the larger build: capacity it fits
    case 128: cap = cluster_capacity<128, kRingDeepKB>(); break;
    case 256: cap = cluster_capacity<256, kRingDeepKB>(); break;
    default: return cudaErrorInvalidValue;
  }
  const int units = m_total * a.Hkv;
  PartitionChoice pc;
  if (!choose_partition({t_max, units, a.D, a.num_sms, a.max_splits, a.forced_splits, a.forced_dparts, cap}, &pc))
    return cudaErrorInvalidValue;
  const int splits = pc.splits, dparts = pc.dparts;
  const bool fused = pc.fused;
  const bool deep = (t_max + splits - 1) / splits > kShallowTiles;
  // Long key loops merged by small clusters (many query tiles) get a build
  // whose merge keeps several rows' loads in flight per thread.
  // Clusters whose CTAs each finish more (row, piece) items than they have
  // threads get the build that takes two pieces per thread.
  const int merge_items = (kBM + splits - 1) / splits * (a.D / dparts / 8);
  const int cm = !fused ? (splits > 1 ? kNoClusterMerge : kMaxClusterSplits)
                 : deep && splits <= 2 ? 2 : deep && splits <= 4 ? 4 : deep && splits <= 8 ? 8
                 : merge_items > kThreads ? kMergeWide : kMaxClusterSplits;
  prm.n_splits = splits;
  prm.dparts = dparts;
  prm.inject_tx = a.inject_tx;
  prm.prefetch_l2 = a.prefetch_l2;
  prm.fused = fused ? 1 : 0;
  if (used_splits) *used_splits = splits;
  switch (a.D) {
    case 64: return launch_d<64>(prm, m_total, a.Hkv, s, deep, cm);
    case 128: return launch_d<128>(prm, m_total, a.Hkv, s, deep, cm);
    case 256: return launch_d<256>(prm, m_total, a.Hkv, s, deep, cm);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rx
