// rx_api.cu -- host side of the C ABI declared in include/rx.h.
//
// The store object ("Reflex: Real-Time VLA Control through Streaming
// Inference", §V "Key implementation": a statically preallocated,
// zero-initialised ring buffer with a write pointer) owns one device
// allocation holding, for K and V, the pinned region (P_cap tokens) and the
// window (N frames x F tokens) of every (layer, head) in the tiled layout of
// rx_internal.h, the device-side ring state and the split-KV workspace of the
// attention kernel.  Every entry point validates its
// arguments on the host, returns an rx_status and never throws.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "rx.h"
#include "partition.h"
#include "rx_internal.h"

namespace {

thread_local std::string g_last_error;
std::atomic<long long> g_launches{0};

rx_status fail(rx_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

rx_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RX_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

namespace rx {

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("RX_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

void set_last_error(const char* where, const char* msg) {
  g_last_error = std::string(where) + ": " + msg;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_tmap_4d(CUtensorMap* tm, const void* base, const uint64_t dims[4],
                    const uint64_t strides_bytes[3], const uint32_t box[4]) {
  EncodeTiledFn f = encode_tiled();
  if (!f) return false;
  cuuint64_t gd[4], gs[3];
  cuuint32_t bx[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < 4; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i < 3; ++i) gs[i] = strides_bytes[i];
  const CUresult r =
      f(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gd, gs, bx, es,
        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace rx

struct rx_cache {
  rx_config cfg{};
  int device = 0;
  int num_sms = 0;
  void* mem = nullptr;
  size_t mem_bytes = 0;
  __nv_bfloat16* k_pin = nullptr;
  __nv_bfloat16* v_pin = nullptr;
  __nv_bfloat16* k_win = nullptr;
  __nv_bfloat16* v_win = nullptr;
  rx::DevState* dstate = nullptr;
  void* xchg = nullptr;
  int max_splits = 0;
  int T_pin = 0;         // tiles of the pinned region per (layer, head), >= 1
  int T_win = 0;         // tiles of the window per (layer, head)
  int slots = 0;         // frame slots of the window: N, or N + 1 with a spare slot
  cudaEvent_t consumer_done = nullptr;   // rx_push_frame_async ordering: consumer work so far
  cudaEvent_t push_done = nullptr;       // ... and the previous asynchronous push
  long long async_pushes = 0;
  int P = 0;             // pinned tokens currently held
  long long host_pushes = 0;
  int forced_splits = 0;
  int forced_dparts = 0;
  int inject_tx = 0;   // rx_debug_inject_timeout: applies to the next attention launch
  int prefetch_l2 = 0; // key tiles an attention CTA asks to be fetched into L2 before its
                       // dependency wait: 1 when the K/V store is larger than half the
                       // device's L2 (its tiles come from DRAM), else 0
};

#define RX_GUARD_BEGIN try {
#define RX_GUARD_END                                              \
  }                                                               \
  catch (const std::bad_alloc&) {                                 \
    return fail(RX_ERR_ARG, "host allocation failed");            \
  }                                                               \
  catch (...) {                                                   \
    return fail(RX_ERR_ARG, "unexpected host exception");         \
  }

extern "C" {

const char* rx_status_str(int s) {
  switch (s) {
    case RX_OK: return "RX_OK";
    case RX_ERR_ARG: return "RX_ERR_ARG";
    case RX_ERR_LAYER: return "RX_ERR_LAYER";
    case RX_ERR_CAPACITY: return "RX_ERR_CAPACITY";
    case RX_ERR_CUDA: return "RX_ERR_CUDA";
    case RX_ERR_TIMEOUT: return "RX_ERR_TIMEOUT";
    case RX_ERR_UNSUPPORTED: return "RX_ERR_UNSUPPORTED";
    case RX_ERR_STATE: return "RX_ERR_STATE";
    default: return "RX_ERR_UNKNOWN";
  }
}

const char* rx_last_error(void) { return g_last_error.c_str(); }

long long rx_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

rx_status rx_cache_create(const rx_config* cfg, rx_cache_t* out) {
  RX_GUARD_BEGIN
  if (!cfg || !out) return fail(RX_ERR_ARG, "rx_cache_create: null argument");
  *out = nullptr;
  const rx_config& c = *cfg;
  if (c.L < 1 || c.Hq < 1 || c.Hkv < 1 || c.N < 1 || c.F < 1 || c.S_cap < 1 || c.P_cap < 0 ||
      c.tail_cap < 0 || c.max_req < 0)
    return fail(RX_ERR_ARG, "rx_cache_create: sizes out of range");
  if (c.Hq % c.Hkv) return fail(RX_ERR_ARG, "rx_cache_create: Hq must be a multiple of Hkv");
  if (c.spare_slot != 0 && c.spare_slot != 1) return fail(RX_ERR_ARG, "rx_cache_create: spare_slot must be 0 or 1");
  if (c.spare_slot && c.F % rx::kTileTok)
    return fail(RX_ERR_UNSUPPORTED, "rx_cache_create: a spare slot needs F %% 64 == 0 (F = %d)", c.F);
  const int G = c.Hq / c.Hkv;
  if (!pow2(G) || G > rx::kBM)
    return fail(RX_ERR_UNSUPPORTED, "rx_cache_create: Hq/Hkv = %d must be a power of two <= 128", G);
  if (c.D != 64 && c.D != 128 && c.D != 256)
    return fail(RX_ERR_UNSUPPORTED, "rx_cache_create: head dim %d not in {64, 128, 256}", c.D);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(RX_ERR_UNSUPPORTED, "rx_cache_create: device is sm_%d%d, the kernels are built for sm_103a",
                prop.major, prop.minor);

  rx_cache* h = new rx_cache();
  h->cfg = c;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  h->max_splits = h->num_sms < 64 ? h->num_sms : 64;
  h->T_pin = rx::tiles_for(c.P_cap > 0 ? c.P_cap : 1);
  h->slots = c.N + c.spare_slot;
  h->T_win = rx::tiles_for(static_cast<long long>(h->slots) * c.F);

  const size_t tile = static_cast<size_t>(rx::tile_bytes(c.D));
  const size_t pin_b = round_up(static_cast<size_t>(c.L) * c.Hkv * h->T_pin * tile, 256);
  const size_t win_b = round_up(static_cast<size_t>(c.L) * c.Hkv * h->T_win * tile, 256);
  // Workspace rows: the action suffix plus a language batch (rx_attend_batch).
  const size_t rows_pad = round_up(static_cast<size_t>(c.S_cap) * G, rx::kBM) +
                          round_up(static_cast<size_t>(c.max_req) * G, rx::kBM);
  // Split partials: per row and split, D bf16 values and dparts (m, l) pairs.
  const size_t part_rows = static_cast<size_t>(c.Hkv) * h->max_splits * rows_pad;
  const size_t xchg_b = round_up(part_rows * (2 * static_cast<size_t>(c.D) + 8 * 4), 256);
  const size_t st_b = 256;
  h->mem_bytes = 2 * pin_b + 2 * win_b + st_b + xchg_b;
  int l2 = 0;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) l2 = 0;
  cudaGetLastError();
  h->prefetch_l2 = l2 > 0 && 2 * (pin_b + win_b) > static_cast<size_t>(l2) / 2 ? 1 : 0;
  e = cudaMalloc(&h->mem, h->mem_bytes);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "rx_cache_create: cudaMalloc");
  }
  e = cudaMemset(h->mem, 0, h->mem_bytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->mem);
    delete h;
    return cuda_fail(e, "rx_cache_create: cudaMemset");
  }
  char* p = static_cast<char*>(h->mem);
  h->k_pin = reinterpret_cast<__nv_bfloat16*>(p); p += pin_b;
  h->v_pin = reinterpret_cast<__nv_bfloat16*>(p); p += pin_b;
  h->k_win = reinterpret_cast<__nv_bfloat16*>(p); p += win_b;
  h->v_win = reinterpret_cast<__nv_bfloat16*>(p); p += win_b;
  h->dstate = reinterpret_cast<rx::DevState*>(p); p += st_b;
  h->xchg = p;
  if (c.spare_slot) {
    e = cudaEventCreateWithFlags(&h->consumer_done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h->push_done, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      cudaFree(h->mem);
      delete h;
      return cuda_fail(e, "rx_cache_create: cudaEventCreate");
    }
  }
  *out = h;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_cache_destroy(rx_cache_t h) {
  RX_GUARD_BEGIN
  if (!h) return RX_OK;
  cudaError_t e = cudaDeviceSynchronize();
  if (h->consumer_done) cudaEventDestroy(h->consumer_done);
  if (h->push_done) cudaEventDestroy(h->push_done);
  cudaError_t e2 = cudaFree(h->mem);
  delete h;
  if (e != cudaSuccess) return cuda_fail(e, "rx_cache_destroy: synchronize");
  if (e2 != cudaSuccess) return cuda_fail(e2, "rx_cache_destroy: cudaFree");
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_pin_prefix(rx_cache_t h, const void* k, const void* v, int P, void* stream) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_pin_prefix: null cache");
  const rx_config& c = h->cfg;
  if (P < 0) return fail(RX_ERR_ARG, "rx_pin_prefix: P < 0");
  if (P > c.P_cap) return fail(RX_ERR_CAPACITY, "rx_pin_prefix: P = %d > P_cap = %d", P, c.P_cap);
  if (P > 0 && (!k || !v)) return fail(RX_ERR_ARG, "rx_pin_prefix: null K/V");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (P > 0) {
    // The prefix is packed into the tiled layout on the device.  Host (or
    // misaligned) sources are staged through a temporary device buffer: a
    // one-time set-up copy.
    const size_t bytes = static_cast<size_t>(c.L) * P * c.Hkv * c.D * 2;
    cudaPointerAttributes ak{}, av{};
    const bool dev_k = cudaPointerGetAttributes(&ak, k) == cudaSuccess && ak.devicePointer != nullptr &&
                       ak.type != cudaMemoryTypeHost && aligned16(k);
    const bool dev_v = cudaPointerGetAttributes(&av, v) == cudaSuccess && av.devicePointer != nullptr &&
                       av.type != cudaMemoryTypeHost && aligned16(v);
    cudaGetLastError();   // clear a lookup error for unregistered host memory
    void* tmp = nullptr;
    const void* sk = k;
    const void* sv = v;
    cudaError_t e = cudaSuccess;
    if (!dev_k || !dev_v) {
      e = cudaMalloc(&tmp, 2 * bytes);
      if (e == cudaSuccess) e = cudaMemcpyAsync(tmp, k, bytes, cudaMemcpyDefault, s);
      if (e == cudaSuccess) e = cudaMemcpyAsync(static_cast<char*>(tmp) + bytes, v, bytes, cudaMemcpyDefault, s);
      sk = tmp;
      sv = static_cast<char*>(tmp) + bytes;
    }
    if (e == cudaSuccess)
      e = rx::launch_pack_tiles(sk, sv, h->k_pin, h->v_pin, c.L, P, c.Hkv, c.D, h->T_pin, 0, nullptr,
                                0, 0, 0, h->num_sms, s);
    if (tmp) {
      const cudaError_t e2 = cudaStreamSynchronize(s);
      cudaFree(tmp);
      if (e == cudaSuccess) e = e2;
    }
    if (e != cudaSuccess) return cuda_fail(e, "rx_pin_prefix: copy");
  }
  h->P = P;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_push_frame(rx_cache_t h, const void* k, const void* v, int* evicted, void* stream) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_push_frame: null cache");
  if (!k || !v) return fail(RX_ERR_ARG, "rx_push_frame: null K/V");
  if (!aligned16(k) || !aligned16(v)) return fail(RX_ERR_ARG, "rx_push_frame: K/V not 16-byte aligned");
  const rx_config& c = h->cfg;
  cudaError_t e = rx::launch_pack_tiles(k, v, h->k_win, h->v_win, c.L, c.F, c.Hkv, c.D, h->T_win, 0,
                                        h->dstate, c.F, c.N, h->slots, h->num_sms,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rx_push_frame: launch");
  if (evicted) *evicted = h->host_pushes >= c.N ? 1 : 0;
  h->host_pushes += 1;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_push_frame_async(rx_cache_t h, const void* k, const void* v, int* evicted,
                              void* producer_stream, void* consumer_stream) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_push_frame_async: null cache");
  if (!h->cfg.spare_slot) return fail(RX_ERR_STATE, "rx_push_frame_async: the cache has no spare slot");
  if (!k || !v) return fail(RX_ERR_ARG, "rx_push_frame_async: null K/V");
  if (!aligned16(k) || !aligned16(v)) return fail(RX_ERR_ARG, "rx_push_frame_async: K/V not 16-byte aligned");
  const rx_config& c = h->cfg;
  cudaStream_t ps = static_cast<cudaStream_t>(producer_stream);
  cudaStream_t cs = static_cast<cudaStream_t>(consumer_stream);
  // This push overwrites the slot the previous push evicted.  Windows that
  // contain it were published before the previous push; work enqueued on the
  // consumer stream from now on waits for the previous push, so only work
  // already enqueued may still read the slot: the producer waits for that.
  cudaError_t e = cudaEventRecord(h->consumer_done, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ps, h->consumer_done, 0);
  if (e == cudaSuccess && h->async_pushes > 0) e = cudaStreamWaitEvent(cs, h->push_done, 0);
  if (e == cudaSuccess)
    e = rx::launch_pack_tiles(k, v, h->k_win, h->v_win, c.L, c.F, c.Hkv, c.D, h->T_win, 0, h->dstate,
                              c.F, c.N, h->slots, h->num_sms, ps);
  if (e == cudaSuccess) e = cudaEventRecord(h->push_done, ps);
  if (e != cudaSuccess) return cuda_fail(e, "rx_push_frame_async");
  if (evicted) *evicted = h->host_pushes >= c.N ? 1 : 0;
  h->host_pushes += 1;
  h->async_pushes += 1;
  return RX_OK;
  RX_GUARD_END
}

static rx::AttnLaunch make_launch(rx_cache_t h, int layer) {
  rx::AttnLaunch a;
  a.tm_pin_k = a.tm_pin_v = a.tm_slide_k = a.tm_slide_v = nullptr;   // regions are tiled
  const long long tile = rx::tile_bytes(h->cfg.D);
  a.pin_head_stride = h->T_pin * tile;
  a.win_head_stride = h->T_win * tile;
  const long long pin_layer = static_cast<long long>(layer) * h->cfg.Hkv * a.pin_head_stride;
  const long long win_layer = static_cast<long long>(layer) * h->cfg.Hkv * a.win_head_stride;
  a.pin_k_tiles = reinterpret_cast<const char*>(h->k_pin) + pin_layer;
  a.pin_v_tiles = reinterpret_cast<const char*>(h->v_pin) + pin_layer;
  a.win_k_tiles = reinterpret_cast<const char*>(h->k_win) + win_layer;
  a.win_v_tiles = reinterpret_cast<const char*>(h->v_win) + win_layer;
  a.layer = layer;
  a.P = h->P;
  a.F = h->cfg.F;
  a.N = h->cfg.N;
  a.slots = h->slots;
  a.D = h->cfg.D;
  a.Hq = h->cfg.Hq;
  a.Hkv = h->cfg.Hkv;
  a.st = h->dstate;
  a.err = &h->dstate->err;
  a.xchg = h->xchg;
  a.max_splits = h->max_splits;
  a.forced_splits = h->forced_splits;
  a.forced_dparts = h->forced_dparts;
  a.num_sms = h->num_sms;
  a.inject_tx = h->inject_tx;
  h->inject_tx = 0;
  a.prefetch_l2 = h->prefetch_l2;
  return a;
}

// Checks the norm jobs an attention launch runs beside its key loop and
// copies them into `jobs`.  The same conditions as rx_adarmsnorm, plus: no
// job's output may overlap another job's input or output.
static rx_status check_norms(const char* where, const rx_norm_rows* norms, int n_norms,
                             rx::NormJob* jobs) {
  if (n_norms < 0 || n_norms > RX_MAX_NORM_JOBS)
    return fail(RX_ERR_ARG, "%s: n_norms = %d not in [0, %d]", where, n_norms, RX_MAX_NORM_JOBS);
  if (n_norms > 0 && !norms) return fail(RX_ERR_ARG, "%s: null norm jobs", where);
  long long total = 0;
  for (int i = 0; i < n_norms; ++i) {
    const rx_norm_rows& n = norms[i];
    if (n.rows < 0) return fail(RX_ERR_ARG, "%s: norm job %d: rows < 0", where, i);
    if (n.d < 8 || (n.d & 7)) return fail(RX_ERR_ARG, "%s: norm job %d: d = %d must be a positive multiple of 8", where, i, n.d);
    if (!(n.eps >= 0.f)) return fail(RX_ERR_ARG, "%s: norm job %d: eps must be >= 0", where, i);
    if (n.rows > 0) {
      if (!n.x || !n.gamma || !n.y) return fail(RX_ERR_ARG, "%s: norm job %d: null pointer", where, i);
      if (!aligned16(n.x) || !aligned16(n.y) || !aligned16(n.gamma))
        return fail(RX_ERR_ARG, "%s: norm job %d: pointers must be 16-byte aligned", where, i);
    }
    total += n.rows;
    jobs[i] = rx::NormJob{n.x, n.gamma, n.y, n.rows, n.d, n.eps};
  }
  if (total > (1LL << 30)) return fail(RX_ERR_ARG, "%s: too many norm rows", where);
  // y of every job against x and y of every job (byte ranges).
  for (int i = 0; i < n_norms; ++i) {
    if (jobs[i].rows == 0) continue;
    const char* y0 = static_cast<const char*>(jobs[i].y);
    const char* y1 = y0 + static_cast<size_t>(jobs[i].rows) * jobs[i].d * 2;
    for (int j = 0; j < n_norms; ++j) {
      if (jobs[j].rows == 0) continue;
      const size_t b = static_cast<size_t>(jobs[j].rows) * jobs[j].d * 2;
      const char* x0 = static_cast<const char*>(jobs[j].x);
      if (y0 < x0 + b && x0 < y1) return fail(RX_ERR_ARG, "%s: norm job %d's y overlaps job %d's x", where, i, j);
      const char* z0 = static_cast<const char*>(jobs[j].y);
      if (j != i && y0 < z0 + b && z0 < y1)
        return fail(RX_ERR_ARG, "%s: norm jobs %d and %d write overlapping rows", where, i, j);
    }
  }
  return RX_OK;
}

// A buffer of the attention the norm jobs of the same launch run beside.
struct Span {
  const void* p;
  long long bytes;
};

static bool spans_overlap(const void* a, long long an, const void* b, long long bn) {
  if (!a || !b || an <= 0 || bn <= 0) return false;
  const char* a0 = static_cast<const char*>(a);
  const char* b0 = static_cast<const char*>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

// The norm jobs run concurrently with the attention of the same launch: no
// job may write bytes the attention reads or writes, and no job may read
// bytes the attention writes.
static rx_status check_norms_beside(const char* where, const rx::NormJob* jobs, int n_norms,
                                    const Span* att_in, int n_in, const Span* att_out, int n_out) {
  for (int i = 0; i < n_norms; ++i) {
    const rx::NormJob& j = jobs[i];
    if (j.rows == 0) continue;
    const long long b = static_cast<long long>(j.rows) * j.d * 2;
    for (int k = 0; k < n_in; ++k)
      if (spans_overlap(j.y, b, att_in[k].p, att_in[k].bytes))
        return fail(RX_ERR_ARG, "%s: norm job %d's y overlaps an input of the attention", where, i);
    for (int k = 0; k < n_out; ++k)
      if (spans_overlap(j.y, b, att_out[k].p, att_out[k].bytes) ||
          spans_overlap(j.x, b, att_out[k].p, att_out[k].bytes) ||
          spans_overlap(j.gamma, static_cast<long long>(j.d) * 4, att_out[k].p, att_out[k].bytes))
        return fail(RX_ERR_ARG, "%s: norm job %d overlaps the attention's output", where, i);
  }
  return RX_OK;
}

static rx_status attend_suffix_impl(const char* where, rx_cache_t h, int layer, const void* q,
                                    const void* k_dyn, const void* v_dyn, int S, void* out,
                                    const rx_norm_rows* norms, int n_norms, void* stream) {
  if (!h) return fail(RX_ERR_ARG, "%s: null cache", where);
  const rx_config& c = h->cfg;
  if (layer < 0 || layer >= c.L) return fail(RX_ERR_LAYER, "%s: layer %d not in [0, %d)", where, layer, c.L);
  if (S < 1) return fail(RX_ERR_ARG, "%s: S < 1", where);
  if (S > c.S_cap) return fail(RX_ERR_CAPACITY, "%s: S = %d > S_cap = %d", where, S, c.S_cap);
  if (!q || !k_dyn || !v_dyn || !out) return fail(RX_ERR_ARG, "%s: null pointer", where);
  if (!aligned16(q) || !aligned16(k_dyn) || !aligned16(v_dyn) || !aligned16(out))
    return fail(RX_ERR_ARG, "%s: pointers must be 16-byte aligned", where);
  rx::NormJob jobs[rx::kMaxNormJobs];
  rx_status ns = check_norms(where, norms, n_norms, jobs);
  if (ns != RX_OK) return ns;
  const long long qb = static_cast<long long>(S) * c.Hq * c.D * 2, kb = static_cast<long long>(S) * c.Hkv * c.D * 2;
  const Span in[3] = {{q, qb}, {k_dyn, kb}, {v_dyn, kb}};
  const Span outs[1] = {{out, qb}};
  ns = check_norms_beside(where, jobs, n_norms, in, 3, outs, 1);
  if (ns != RX_OK) return ns;
  rx::AttnLaunch a = make_launch(h, layer);
  a.norms = jobs;
  a.n_norms = n_norms;
  rx::AttnSegment seg{q, k_dyn, v_dyn, out, S, S, nullptr, 1, 0, 0};
  cudaError_t e = rx::launch_partitioned_attention(a, &seg, 1, static_cast<cudaStream_t>(stream), nullptr);
  if (e != cudaSuccess)
    return fail(RX_ERR_CUDA, "%s: launch: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return RX_OK;
}

rx_status rx_attend_suffix_norms(rx_cache_t h, int layer, const void* q, const void* k_dyn,
                                 const void* v_dyn, int S, void* out, const rx_norm_rows* norms,
                                 int n_norms, void* stream) {
  RX_GUARD_BEGIN
  return attend_suffix_impl("rx_attend_suffix_norms", h, layer, q, k_dyn, v_dyn, S, out, norms, n_norms,
                            stream);
  RX_GUARD_END
}

rx_status rx_attend_suffix(rx_cache_t h, int layer, const void* q, const void* k_dyn,
                           const void* v_dyn, int S, void* out, void* stream) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_attend_suffix: null cache");
  const rx_config& c = h->cfg;
  if (layer < 0 || layer >= c.L) return fail(RX_ERR_LAYER, "rx_attend_suffix: layer %d not in [0, %d)", layer, c.L);
  if (S < 1) return fail(RX_ERR_ARG, "rx_attend_suffix: S < 1");
  if (S > c.S_cap) return fail(RX_ERR_CAPACITY, "rx_attend_suffix: S = %d > S_cap = %d", S, c.S_cap);
  if (!q || !k_dyn || !v_dyn || !out) return fail(RX_ERR_ARG, "rx_attend_suffix: null pointer");
  if (!aligned16(q) || !aligned16(k_dyn) || !aligned16(v_dyn) || !aligned16(out))
    return fail(RX_ERR_ARG, "rx_attend_suffix: pointers must be 16-byte aligned");
  const rx::AttnLaunch a = make_launch(h, layer);
  rx::AttnSegment seg{q, k_dyn, v_dyn, out, S, S, nullptr, 1, 0, 0};
  cudaError_t e = rx::launch_partitioned_attention(a, &seg, 1, static_cast<cudaStream_t>(stream), nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "rx_attend_suffix: launch");
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_attend_suffix_block_causal(rx_cache_t h, int layer, const void* q, const void* k_dyn,
                                        const void* v_dyn, int S, int n_state, void* out,
                                        void* stream) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_attend_suffix_block_causal: null cache");
  const rx_config& c = h->cfg;
  if (layer < 0 || layer >= c.L)
    return fail(RX_ERR_LAYER, "rx_attend_suffix_block_causal: layer %d not in [0, %d)", layer, c.L);
  if (S < 1) return fail(RX_ERR_ARG, "rx_attend_suffix_block_causal: S < 1");
  if (S > c.S_cap) return fail(RX_ERR_CAPACITY, "rx_attend_suffix_block_causal: S = %d > S_cap = %d", S, c.S_cap);
  if (n_state < 0 || n_state > S) return fail(RX_ERR_ARG, "rx_attend_suffix_block_causal: n_state = %d not in [0, S]", n_state);
  if (!q || !k_dyn || !v_dyn || !out) return fail(RX_ERR_ARG, "rx_attend_suffix_block_causal: null pointer");
  if (!aligned16(q) || !aligned16(k_dyn) || !aligned16(v_dyn) || !aligned16(out))
    return fail(RX_ERR_ARG, "rx_attend_suffix_block_causal: pointers must be 16-byte aligned");
  const rx::AttnLaunch a = make_launch(h, layer);
  // n_state == S: every token is in the state block, which sees all S keys: plain Eq. 1.
  rx::AttnSegment seg{q, k_dyn, v_dyn, out, S, S, nullptr, 1, 0, n_state < S ? n_state : 0};
  cudaError_t e = rx::launch_partitioned_attention(a, &seg, 1, static_cast<cudaStream_t>(stream), nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "rx_attend_suffix_block_causal: launch");
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_tail_append(void* k_tail, void* v_tail, int* tail_len, const void* k_new,
                         const void* v_new, const int* active, int B, int tail_cap, int Hkv, int D,
                         int* overflow, void* stream) {
  RX_GUARD_BEGIN
  if (B < 0 || tail_cap < 1 || Hkv < 1 || D < 1 || (static_cast<long long>(Hkv) * D) % 8)
    return fail(RX_ERR_ARG, "rx_tail_append: sizes out of range (Hkv*D must be a multiple of 8)");
  if (B == 0) return RX_OK;
  if (!k_tail || !v_tail || !tail_len || !k_new || !v_new)
    return fail(RX_ERR_ARG, "rx_tail_append: null pointer");
  if (!aligned16(k_tail) || !aligned16(v_tail) || !aligned16(k_new) || !aligned16(v_new) ||
      (reinterpret_cast<uintptr_t>(tail_len) & 3) || (reinterpret_cast<uintptr_t>(active) & 3) ||
      (reinterpret_cast<uintptr_t>(overflow) & 3))
    return fail(RX_ERR_ARG, "rx_tail_append: misaligned pointer");
  cudaError_t e = rx::launch_tail_append(k_tail, v_tail, tail_len, k_new, v_new, active, B, tail_cap,
                                         Hkv, D, overflow, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rx_tail_append: launch");
  return RX_OK;
  RX_GUARD_END
}

namespace {
// Snapshot layout: [SnapHeader, 256 B][pinned K | pinned V | window K | window V | DevState].
struct SnapHeader {
  char magic[8];
  rx_config cfg;
  int P;
  long long host_pushes;
  long long body_bytes;
};
static_assert(sizeof(SnapHeader) <= 256, "snapshot header");
constexpr long long kSnapHeader = 256;

// Writes a snapshot's header: the values travel as the kernel's argument, so
// nothing on the host has to outlive the call (the same holds under stream
// capture).
__global__ void snapshot_header_kernel(const __grid_constant__ SnapHeader hd, SnapHeader* dst) {
  if (threadIdx.x == 0) *dst = hd;
}

long long snapshot_body(rx_cache_t h) {
  return reinterpret_cast<const char*>(h->dstate) + sizeof(rx::DevState) -
         reinterpret_cast<const char*>(h->k_pin);
}
}  // namespace

rx_status rx_snapshot_bytes(rx_cache_t h, long long* bytes) {
  RX_GUARD_BEGIN
  if (!h || !bytes) return fail(RX_ERR_ARG, "rx_snapshot_bytes: null argument");
  *bytes = kSnapHeader + snapshot_body(h);
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_snapshot(rx_cache_t h, void* dst, void* stream) {
  RX_GUARD_BEGIN
  if (!h || !dst) return fail(RX_ERR_ARG, "rx_snapshot: null argument");
  if (!aligned16(dst)) return fail(RX_ERR_ARG, "rx_snapshot: dst must be 16-byte aligned");
  SnapHeader hd;
  memset(&hd, 0, sizeof(hd));
  memcpy(hd.magic, "RXSNAP01", 8);
  hd.cfg = h->cfg;
  hd.P = h->P;
  hd.host_pushes = h->host_pushes;
  hd.body_bytes = snapshot_body(h);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  snapshot_header_kernel<<<1, 32, 0, s>>>(hd, static_cast<SnapHeader*>(dst));
  rx::count_launch();
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(static_cast<char*>(dst) + kSnapHeader, h->k_pin, hd.body_bytes,
                        cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "rx_snapshot: copy");
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_restore(rx_cache_t h, const void* src, void* stream) {
  RX_GUARD_BEGIN
  if (!h || !src) return fail(RX_ERR_ARG, "rx_restore: null argument");
  if (!aligned16(src)) return fail(RX_ERR_ARG, "rx_restore: src must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SnapHeader hd;
  cudaError_t e = cudaMemcpyAsync(&hd, src, sizeof(hd), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "rx_restore: reading the header");
  if (memcmp(hd.magic, "RXSNAP01", 8) != 0 || memcmp(&hd.cfg, &h->cfg, sizeof(rx_config)) != 0 ||
      hd.body_bytes != snapshot_body(h))
    return fail(RX_ERR_ARG, "rx_restore: not a snapshot of a cache with this configuration");
  e = cudaMemcpyAsync(h->k_pin, static_cast<const char*>(src) + kSnapHeader, hd.body_bytes,
                      cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return cuda_fail(e, "rx_restore: copy");
  h->P = hd.P;
  h->host_pushes = hd.host_pushes;
  return RX_OK;
  RX_GUARD_END
}

static rx_status attend_batch_impl(rx_cache_t h, int layer, const void* q_act, const void* k_dyn,
                                   const void* v_dyn, int S, void* out_act, const rx_stream_batch* lang,
                                   const rx_norm_rows* norms, int n_norms, void* stream);

rx_status rx_attend_batch(rx_cache_t h, int layer, const void* q_act, const void* k_dyn,
                          const void* v_dyn, int S, void* out_act, const rx_stream_batch* lang,
                          void* stream) {
  RX_GUARD_BEGIN
  return attend_batch_impl(h, layer, q_act, k_dyn, v_dyn, S, out_act, lang, nullptr, 0, stream);
  RX_GUARD_END
}

rx_status rx_attend_batch_norms(rx_cache_t h, int layer, const void* q_act, const void* k_dyn,
                                const void* v_dyn, int S, void* out_act, const rx_stream_batch* lang,
                                const rx_norm_rows* norms, int n_norms, void* stream) {
  RX_GUARD_BEGIN
  return attend_batch_impl(h, layer, q_act, k_dyn, v_dyn, S, out_act, lang, norms, n_norms, stream);
  RX_GUARD_END
}

static rx_status attend_batch_impl(rx_cache_t h, int layer, const void* q_act, const void* k_dyn,
                                   const void* v_dyn, int S, void* out_act, const rx_stream_batch* lang,
                                   const rx_norm_rows* norms, int n_norms, void* stream) {
  if (!h) return fail(RX_ERR_ARG, "rx_attend_batch: null cache");
  const rx_config& c = h->cfg;
  if (layer < 0 || layer >= c.L) return fail(RX_ERR_LAYER, "rx_attend_batch: layer %d not in [0, %d)", layer, c.L);
  if (S < 0) return fail(RX_ERR_ARG, "rx_attend_batch: S < 0");
  if (S > c.S_cap) return fail(RX_ERR_CAPACITY, "rx_attend_batch: S = %d > S_cap = %d", S, c.S_cap);
  rx::AttnSegment segs[2];
  int nseg = 0;
  if (S > 0) {
    if (!q_act || !k_dyn || !v_dyn || !out_act) return fail(RX_ERR_ARG, "rx_attend_batch: null action pointer");
    if (!aligned16(q_act) || !aligned16(k_dyn) || !aligned16(v_dyn) || !aligned16(out_act))
      return fail(RX_ERR_ARG, "rx_attend_batch: action pointers must be 16-byte aligned");
    segs[nseg++] = rx::AttnSegment{q_act, k_dyn, v_dyn, out_act, S, S, nullptr, 1, 0, 0};
  }
  if (lang && lang->B > 0) {
    const rx_stream_batch& b = *lang;
    if (b.T < 1) return fail(RX_ERR_ARG, "rx_attend_batch: T < 1");
    if (static_cast<long long>(b.B) * b.T > c.max_req)
      return fail(RX_ERR_CAPACITY, "rx_attend_batch: B*T = %lld > max_req = %d",
                  static_cast<long long>(b.B) * b.T, c.max_req);
    if (c.tail_cap < 1) return fail(RX_ERR_CAPACITY, "rx_attend_batch: the cache has tail_cap = 0");
    if (!b.q || !b.k_tail || !b.v_tail || !b.tail_len || !b.out)
      return fail(RX_ERR_ARG, "rx_attend_batch: null language pointer");
    if (!aligned16(b.q) || !aligned16(b.k_tail) || !aligned16(b.v_tail) || !aligned16(b.out) ||
        (reinterpret_cast<uintptr_t>(b.tail_len) & 3))
      return fail(RX_ERR_ARG, "rx_attend_batch: language pointers misaligned");
    segs[nseg++] = rx::AttnSegment{b.q, b.k_tail, b.v_tail, b.out, b.B * b.T, b.B * c.tail_cap,
                                   b.tail_len, b.T, c.tail_cap, 0};
  }
  rx::NormJob jobs[rx::kMaxNormJobs];
  rx_status ns = check_norms("rx_attend_batch", norms, n_norms, jobs);
  if (ns != RX_OK) return ns;
  {
    Span in[7] = {};
    Span outs[2] = {};
    int n_in = 0, n_out = 0;
    if (S > 0) {
      const long long qb = static_cast<long long>(S) * c.Hq * c.D * 2;
      const long long kb = static_cast<long long>(S) * c.Hkv * c.D * 2;
      in[n_in++] = {q_act, qb};
      in[n_in++] = {k_dyn, kb};
      in[n_in++] = {v_dyn, kb};
      outs[n_out++] = {out_act, qb};
    }
    if (lang && lang->B > 0) {
      const rx_stream_batch& b = *lang;
      const long long qb = static_cast<long long>(b.B) * b.T * c.Hq * c.D * 2;
      const long long tb = static_cast<long long>(b.B) * c.tail_cap * c.Hkv * c.D * 2;
      in[n_in++] = {b.q, qb};
      in[n_in++] = {b.k_tail, tb};
      in[n_in++] = {b.v_tail, tb};
      in[n_in++] = {b.tail_len, static_cast<long long>(b.B) * 4};
      outs[n_out++] = {b.out, qb};
    }
    ns = check_norms_beside("rx_attend_batch", jobs, n_norms, in, n_in, outs, n_out);
    if (ns != RX_OK) return ns;
  }
  int norm_rows = 0;
  for (int i = 0; i < n_norms; ++i) norm_rows += jobs[i].rows;
  if (nseg == 0) {
    // No attention: the norm jobs alone, as rx_adarmsnorm launches.
    for (int i = 0; i < n_norms; ++i) {
      if (jobs[i].rows == 0) continue;
      const cudaError_t e = rx::launch_adarmsnorm(static_cast<const __nv_bfloat16*>(jobs[i].x), jobs[i].gamma,
                                                  jobs[i].rows, jobs[i].d, jobs[i].eps,
                                                  static_cast<__nv_bfloat16*>(jobs[i].y),
                                                  static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_fail(e, "rx_attend_batch: norm launch");
    }
    return RX_OK;
  }
  rx::AttnLaunch a = make_launch(h, layer);
  a.norms = jobs;
  a.n_norms = norm_rows > 0 ? n_norms : 0;
  cudaError_t e = rx::launch_partitioned_attention(a, segs, nseg, static_cast<cudaStream_t>(stream), nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "rx_attend_batch: launch");
  return RX_OK;
}

rx_status rx_ada_gamma(const float* t, const float* state, int n_cond, int emb_dim, int state_dim,
                       const void* W1, const void* b1, int hidden, const void* W2, const void* b2,
                       int d, int n_sets, float* gamma, void* stream) {
  RX_GUARD_BEGIN
  if (n_cond < 1 || n_cond > rx::kMaxCond)
    return fail(RX_ERR_ARG, "rx_ada_gamma: n_cond = %d not in [1, %d]", n_cond, rx::kMaxCond);
  if (emb_dim < 0 || (emb_dim & 1) || state_dim < 0 || emb_dim + state_dim < 1)
    return fail(RX_ERR_ARG, "rx_ada_gamma: emb_dim must be even, widths >= 0, cond width >= 1");
  if (hidden < 16 || hidden > rx::kMaxHidden || (hidden & 15))
    return fail(RX_ERR_ARG, "rx_ada_gamma: hidden = %d must be a multiple of 16 in [16, %d]", hidden, rx::kMaxHidden);
  if (d < 8 || (d & 7)) return fail(RX_ERR_ARG, "rx_ada_gamma: d = %d must be a positive multiple of 8", d);
  if (n_sets < 1) return fail(RX_ERR_ARG, "rx_ada_gamma: n_sets < 1");
  if (!t || (state_dim > 0 && !state) || !W1 || !b1 || !W2 || !b2 || !gamma)
    return fail(RX_ERR_ARG, "rx_ada_gamma: null pointer");
  if (!aligned16(W2) || (reinterpret_cast<uintptr_t>(W1) & 1) || (reinterpret_cast<uintptr_t>(b1) & 1) ||
      (reinterpret_cast<uintptr_t>(b2) & 1) || (reinterpret_cast<uintptr_t>(gamma) & 3) ||
      (reinterpret_cast<uintptr_t>(t) & 3) || (reinterpret_cast<uintptr_t>(state) & 3))
    return fail(RX_ERR_ARG, "rx_ada_gamma: misaligned pointer");
  cudaError_t e = rx::launch_ada_gamma(t, state, n_cond, emb_dim, state_dim,
                                       static_cast<const __nv_bfloat16*>(W1),
                                       static_cast<const __nv_bfloat16*>(b1), hidden,
                                       static_cast<const __nv_bfloat16*>(W2),
                                       static_cast<const __nv_bfloat16*>(b2), d, n_sets, gamma,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rx_ada_gamma: launch");
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_adarmsnorm(const void* x, const float* gamma, int rows, int d, float eps, void* y,
                        void* stream) {
  RX_GUARD_BEGIN
  if (rows < 0) return fail(RX_ERR_ARG, "rx_adarmsnorm: rows < 0");
  if (d < 8 || (d & 7)) return fail(RX_ERR_ARG, "rx_adarmsnorm: d = %d must be a positive multiple of 8", d);
  if (!(eps >= 0.f)) return fail(RX_ERR_ARG, "rx_adarmsnorm: eps must be >= 0");
  if (rows == 0) return RX_OK;
  if (!x || !gamma || !y) return fail(RX_ERR_ARG, "rx_adarmsnorm: null pointer");
  if (!aligned16(x) || !aligned16(y) || !aligned16(gamma))
    return fail(RX_ERR_ARG, "rx_adarmsnorm: pointers must be 16-byte aligned");
  if (x == y) return fail(RX_ERR_ARG, "rx_adarmsnorm: y may not alias x");
  cudaError_t e = rx::launch_adarmsnorm(static_cast<const __nv_bfloat16*>(x), gamma, rows, d, eps,
                                        static_cast<__nv_bfloat16*>(y),
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "rx_adarmsnorm: launch");
  return RX_OK;
  RX_GUARD_END
}

static rx_status read_state(rx_cache_t h, rx::DevState* ds, cudaStream_t s) {
  cudaError_t e = cudaMemcpyAsync(ds, h->dstate, sizeof(*ds), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading device ring state");
  return RX_OK;
}

rx_status rx_get_state(rx_cache_t h, int* head, int* valid, long long* pushes, void* stream) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_get_state: null cache");
  rx::DevState ds;
  rx_status r = read_state(h, &ds, static_cast<cudaStream_t>(stream));
  if (r != RX_OK) return r;
  if (head) *head = ds.head;
  if (valid) *valid = ds.valid;
  if (pushes) *pushes = ds.pushes;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_debug_window(rx_cache_t h, int* slots, int* valid, void* stream) {
  RX_GUARD_BEGIN
  if (!h || !slots || !valid) return fail(RX_ERR_ARG, "rx_debug_window: null argument");
  rx::DevState ds;
  rx_status r = read_state(h, &ds, static_cast<cudaStream_t>(stream));
  if (r != RX_OK) return r;
  const int ns = h->slots;
  const int oldest = ((ds.head - ds.valid) % ns + ns) % ns;
  for (int i = 0; i < ds.valid; ++i) slots[i] = (oldest + i) % ns;
  *valid = ds.valid;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_export_window(rx_cache_t h, int layer, void* k_out, void* v_out, void* stream) {
  RX_GUARD_BEGIN
  if (!h || !k_out || !v_out) return fail(RX_ERR_ARG, "rx_export_window: null argument");
  const rx_config& c = h->cfg;
  if (layer < 0 || layer >= c.L) return fail(RX_ERR_LAYER, "rx_export_window: layer %d", layer);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int slots[4096];
  if (c.N > 4096) return fail(RX_ERR_UNSUPPORTED, "rx_export_window: N > 4096");
  int valid = 0;
  rx_status r = rx_debug_window(h, slots, &valid, stream);
  if (r != RX_OK) return r;
  const size_t fb = static_cast<size_t>(c.F) * c.Hkv * c.D * 2;
  for (int i = 0; i < valid; ++i) {
    cudaError_t e = rx::launch_unpack_tiles(h->k_win, h->v_win, static_cast<char*>(k_out) + i * fb,
                                            static_cast<char*>(v_out) + i * fb, layer, slots[i] * c.F,
                                            c.F, c.Hkv, c.D, h->T_win, s);
    if (e != cudaSuccess) return cuda_fail(e, "rx_export_window: copy");
  }
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_check_device_error(rx_cache_t h, int* code, void* stream) {
  RX_GUARD_BEGIN
  if (!h || !code) return fail(RX_ERR_ARG, "rx_check_device_error: null argument");
  rx::DevState ds;
  rx_status r = read_state(h, &ds, static_cast<cudaStream_t>(stream));
  if (r != RX_OK) return r;
  *code = ds.err;
  if (ds.err) {
    cudaError_t e = cudaMemsetAsync(&h->dstate->err, 0, sizeof(int), static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "rx_check_device_error: clear");
  }
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_set_attn_splits(rx_cache_t h, int splits) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_set_attn_splits: null cache");
  if (splits < 0 || splits > h->max_splits)
    return fail(RX_ERR_ARG, "rx_set_attn_splits: %d not in [0, %d]", splits, h->max_splits);
  h->forced_splits = splits;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_debug_inject_timeout(rx_cache_t h, int bytes) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_debug_inject_timeout: null cache");
  if (bytes < 0 || bytes > (1 << 20) || (bytes & 15))
    return fail(RX_ERR_ARG, "rx_debug_inject_timeout: %d not a multiple of 16 in [0, 2^20]", bytes);
  h->inject_tx = bytes;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_debug_choose_partition(int t_max, int units, int D, int num_sms, int max_splits,
                                    int forced_splits, int forced_dparts, const int* cluster_capacity,
                                    int* splits, int* dparts, int* fused) {
  RX_GUARD_BEGIN
  if (!cluster_capacity || !splits || !dparts || !fused)
    return fail(RX_ERR_ARG, "rx_debug_choose_partition: null pointer");
  if (t_max < 1 || units < 1 || num_sms < 1 || max_splits < 1 || forced_splits < 0 || forced_dparts < 0 ||
      t_max > (1 << 24) || units > (1 << 24) || num_sms > (1 << 16) || max_splits > (1 << 16) ||
      forced_splits > (1 << 16))
    return fail(RX_ERR_ARG, "rx_debug_choose_partition: sizes out of range");
  if (D != 64 && D != 128 && D != 256) return fail(RX_ERR_ARG, "rx_debug_choose_partition: D = %d", D);
  rx::PartitionChoice pc;
  if (!rx::choose_partition({t_max, units, D, num_sms, max_splits, forced_splits, forced_dparts, cluster_capacity},
                            &pc))
    return fail(RX_ERR_ARG, "rx_debug_choose_partition: column split %d does not fit D = %d", forced_dparts, D);
  *splits = pc.splits;
  *dparts = pc.dparts;
  *fused = pc.fused ? 1 : 0;
  return RX_OK;
  RX_GUARD_END
}

rx_status rx_set_attn_dparts(rx_cache_t h, int dparts) {
  RX_GUARD_BEGIN
  if (!h) return fail(RX_ERR_ARG, "rx_set_attn_dparts: null cache");
  if (!(dparts == 0 || dparts == 1 || dparts == 2 || dparts == 4) || (dparts > 0 && h->cfg.D / dparts < 64))
    return fail(RX_ERR_ARG, "rx_set_attn_dparts: %d not 0, or 1/2/4 with D/dparts >= 64 (D = %d)", dparts,
                h->cfg.D);
  h->forced_dparts = dparts;
  return RX_OK;
  RX_GUARD_END
}

}  // extern "C"
