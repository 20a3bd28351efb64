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
  int head;        // slot the next push writes
  int valid;       // frames held, min(pushes, N)
  long long pushes;
  unsigned int append_arrivals;   // CTAs of the running append that finished
  int err;         // error bits set by kernels (see kErr*)
  int pad[2];
};

constexpr int kErrAttnTimeout = 1;    // attention kernel: a bounded wait gave up
constexpr int kErrBatchTimeout = 2;   // batched attention: a bounded wait gave up

constexpr int kMaxCond = 16;          // rx_ada_gamma: conditioning vectors per call
constexpr int kMaxHidden = 2048;      // rx_ada_gamma: hidden width

// Count of kernel launches made by the library (for benchmark accounting).
void count_launch(int n = 1);

// Set the message rx_last_error() returns on this thread.
void set_last_error(const char* where, const char* msg);

// ---- ring append ---------------------------------------------------------
cudaError_t launch_ring_append(const void* k_src, const void* v_src, void* k_slide,
                               void* v_slide, DevState* st, int L, int N,
                               long long frame_bytes, int num_sms, cudaStream_t s);

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

// Keys per V piece of the attention kernel's load ring: one 8 KB piece holds
// all D columns of this many keys.  The V tensor maps use it as box height.
__host__ __device__ constexpr int v_piece_keys(int D) { return 16 * (256 / D); }

// One M-tile of queries: `rows` rows starting at row `row0` of a request.
// Row r of a request is (token r / G, head g*G + r % G).
struct TileDesc {
  int req;        // request index (selects q / private-key maps and out)
  int row0;       // first row of the tile within the request
};

constexpr int kMaxReq = 40;   // requests per batched launch (tensor maps in params)

struct AttnLaunch {
  // Shared regions (pinned, window) of one layer.
  const CUtensorMap* tm_pin_k;
  const CUtensorMap* tm_pin_v;
  const CUtensorMap* tm_slide_k;
  const CUtensorMap* tm_slide_v;
  int layer, P, F, N, D, Hq, Hkv;
  const DevState* st;
  int* err;
  float* part_o;      // workspace: [Hkv][splits][tiles*128][D] fp32
  float2* part_ml;    // workspace: [Hkv][splits][tiles*128]
  int max_splits;     // capacity of the workspace in splits
  int forced_splits;  // 0 = automatic
  int num_sms;
};

struct AttnRequest {
  const void* q;      // bf16 [n_tok][Hq][D]
  const void* k_priv; // bf16 [n_priv][Hkv][D] (may be null if n_priv == 0)
  const void* v_priv;
  void* out;          // bf16 [n_tok][Hq][D]
  int n_tok;
  int n_priv;
};

// Encode the tensor maps of every request and launch the attention kernel
// (plus the split merge when more than one split is used).
cudaError_t launch_partitioned_attention(const AttnLaunch& a, const AttnRequest* reqs,
                                         int nreq, cudaStream_t s, int* used_splits);

// Tensor-map encoding through the driver entry point (no -lcuda link).
bool encode_tmap_4d(CUtensorMap* tm, const void* base, const uint64_t dims[4],
                    const uint64_t strides_bytes[3], const uint32_t box[4]);

}  // namespace rx
