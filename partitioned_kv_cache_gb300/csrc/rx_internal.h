// rx_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace rx {

// Device-side ring state of one cache.  Lives in the cache's allocation and
// is advanced by the append kernel itself, so captured graphs replay it.
struct DevState {
  // head (slot the next push writes) and valid (frames held, <= N) are one
  // 64-bit word: the append publishes both with a single store and readers
  // load both with a single load.
  int head;
  int valid;
  long long pushes;
  unsigned int append_arrivals;   // CTAs of the running append that finished
  int err;         // error bits set by kernels (see kErr*)
  int pad[2];
};

__device__ __forceinline__ void load_ring_state(const DevState* st, int* head, int* valid) {
  const unsigned long long hv = *reinterpret_cast<const volatile unsigned long long*>(st);
  *head = static_cast<int>(hv & 0xFFFFFFFFull);
  *valid = static_cast<int>(hv >> 32);
}
__device__ __forceinline__ void publish_ring_state(DevState* st, int head, int valid) {
  *reinterpret_cast<volatile unsigned long long*>(st) =
      static_cast<unsigned long long>(static_cast<unsigned int>(head)) |
      (static_cast<unsigned long long>(static_cast<unsigned int>(valid)) << 32);
}

constexpr int kErrAttnTimeout = 1;    // attention kernel: a bounded wait gave up
constexpr int kErrBatchTimeout = 2;   // batched attention: a bounded wait gave up
constexpr int kErrAppendTimeout = 4;  // ring append: a bounded wait gave up

constexpr int kMaxCond = 16;          // rx_ada_gamma: conditioning vectors per call
constexpr int kMaxHidden = 2048;      // rx_ada_gamma: hidden width

// Count of kernel launches made by the library (for benchmark accounting).
void count_launch(int n = 1);

// Whether kernels are launched with programmatic stream serialization (the
// next kernel may start its prologue while the previous one drains).  On by
// default; RX_PDL=0 in the environment turns it off.
bool pdl_enabled();

// Launch `k` on `s`, with programmatic stream serialization when enabled.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
  count_launch();
  return e;
}

// Set the message rx_last_error() returns on this thread.
void set_last_error(const char* where, const char* msg);

// ---- tiled store layout -----------------------------------------------------
// The pinned region and the window of every (layer, K/V head) are stored as
// tiles of 64 tokens, each tile already in the shared-memory layout the
// attention kernel's tensor-core operands use: [D/64 column blocks][64 tokens]
// [128 bytes], the eight 16-byte chunks of a 128-byte row permuted by
// chunk ^ (token & 7) (the 128-byte swizzle).  A tile is then one contiguous
// 128*D-byte bulk copy.  Region layout: [L][Hkv][tiles][tile bytes].
constexpr int kTileTok = 64;
__host__ __device__ constexpr long long tile_bytes(int D) { return 128LL * D; }
__host__ __device__ constexpr int tiles_for(long long tokens) {
  return static_cast<int>((tokens + kTileTok - 1) / kTileTok);
}

// Pack tokens [tok0, tok0 + n) of one region for all layers and heads from
// the user layout src [L][n][Hkv][D] into the tiled layout (T tiles per
// (layer, head)).  When `st` is non-null this is a ring append: tok0 is
// head * F read on the device, and the last CTA advances {head, valid}.
cudaError_t launch_pack_tiles(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                              int L, int n, int Hkv, int D, int T, int tok0, DevState* st,
                              int F, int N, int slots, int num_sms, cudaStream_t s);

// Append one token per active stream at tail_len[b] (bounded by tail_cap).
cudaError_t launch_tail_append(void* k_tail, void* v_tail, int* tail_len, const void* k_new,
                               const void* v_new, const int* active, int B, int tail_cap,
                               int Hkv, int D, int* overflow, cudaStream_t s);

// Inverse of the packing for one layer and token range (test aid):
// dst [n][Hkv][D] <- tiles.
cudaError_t launch_unpack_tiles(const void* k_tiles, const void* v_tiles, void* k_dst, void* v_dst,
                                int layer, int tok0, int n, int Hkv, int D, int T, cudaStream_t s);

// ---- AdaRMSNorm ------------------------------------------------------------
cudaError_t launch_adarmsnorm(const __nv_bfloat16* x, const float* gamma, int rows, int d,
                              float eps, __nv_bfloat16* y, cudaStream_t s);
cudaError_t launch_ada_gamma(const float* t, const float* state, int n_cond, int emb_dim,
                             int state_dim, const __nv_bfloat16* W1, const __nv_bfloat16* b1,
                             int hidden, const __nv_bfloat16* W2, const __nv_bfloat16* b2,
                             int d, int n_sets, float* gamma, cudaStream_t s);

// ---- partitioned attention -------------------------------------------------
constexpr int kBM = 128;   // query rows per CTA (one tcgen05 M=128 tile)
constexpr int kBN = 64;    // keys per KV tile

// An AdaRMSNorm job (y = x * rsqrt(mean x^2 + eps) * gamma over `rows` rows
// of width d) that an attention launch runs beside its key loop.
struct NormJob {
  const void* x;        // bf16 [rows][d]
  const float* gamma;   // fp32 [d]
  void* y;              // bf16 [rows][d]
  int rows;
  int d;                // multiple of 8
  float eps;
};
constexpr int kMaxNormJobs = 2;

struct AttnLaunch {
  // Shared regions (pinned, window) of one layer.  Each is either pre-tiled
  // (pointers below non-null: bulk copies) or read through its tensor map.
  const CUtensorMap* tm_pin_k;
  const CUtensorMap* tm_pin_v;
  const CUtensorMap* tm_slide_k;
  const CUtensorMap* tm_slide_v;
  const void* pin_k_tiles;      // tiles of (layer, head 0); nullptr = tensor map
  const void* pin_v_tiles;
  const void* win_k_tiles;
  const void* win_v_tiles;
  long long pin_head_stride;    // bytes between K/V heads of the tiled regions
  long long win_head_stride;
  int layer, P, F, N, D, Hq, Hkv;
  int slots;          // frame slots of the window: N, or N + 1 with a spare slot
  const DevState* st;
  int* err;
  void* xchg;         // workspace for the split partials (attention grid <-> merge):
                      // Hkv * splits * tiles*128 * (2*D + 8*dparts) bytes
  int max_splits;     // capacity of the workspace in splits (at dparts <= 4)
  int forced_splits;  // 0 = automatic
  int forced_dparts;  // output-column split: 0 = automatic, else 1, 2 or 4
  int num_sms;
  int inject_tx;      // test aid: extra bytes CTA 0 expects on its first K tile (0 = none)
  const NormJob* norms = nullptr;   // up to kMaxNormJobs norm jobs run in the same launch
  int n_norms = 0;
  int prefetch_l2 = 0;  // > 0: the store is larger than L2 can keep; each CTA asks for
                        // its Q tile and its split's first prefetch_l2 key tiles to be
                        // fetched into L2 while the previous kernel drains
};

// One group of query rows attending over [pinned; window; private keys].
// Rows are (token, head-in-group) pairs: row r = token r / G, head g*G + r % G.
struct AttnSegment {
  const void* q;          // bf16 [tokens][Hq][D]
  const void* k_priv;     // bf16 [n_priv][Hkv][D] (may be null if n_priv == 0)
  const void* v_priv;
  void* out;              // bf16 [tokens][Hq][D]
  int tokens;             // query tokens
  int n_priv;             // private keys
  // Stream mask (language batches): token t belongs to stream t / tok_per_stream
  // and sees private key j only if j / tail_cap is its stream and
  // j % tail_cap < tail_len[stream].  tail_cap = 0 disables the mask.
  const int* tail_len;
  int tok_per_stream;
  int tail_cap;
  // Block-causal suffix: tokens t < state_tokens see only private keys
  // [0, state_tokens).  0 disables it.
  int state_tokens;
};

// Launch the attention kernel over one or two segments (plus the split merge
// when more than one split is used).  Both segments read the same shared K/V.
cudaError_t launch_partitioned_attention(const AttnLaunch& a, const AttnSegment* segs, int nseg,
                                         cudaStream_t s, int* used_splits);

// Tensor-map encoding through the driver entry point (no -lcuda link).
bool encode_tmap_4d(CUtensorMap* tm, const void* base, const uint64_t dims[4],
                    const uint64_t strides_bytes[3], const uint32_t box[4]);

}  // namespace rx
