// attend_static.cu -- partitioned attention that allocates no memory.
//
// Some callers cannot call cudaMalloc at all: a real-time control loop where
// an allocation would synchronise the device and stall the loop, an embedded
// runtime that reserved its whole memory budget up front, or a plugin living
// inside a host framework that owns the device allocator.  They cannot create
// an rx_cache (that allocates the store and the workspace), so this file gives
// them one entry point that runs the same split-KV attention kernel over K/V
// regions they already hold, with the kernel's scratch (split partials and a
// small state block) placed in a fixed file-scope device array instead of an
// allocation.  The array is part of the library image: every GPU that loads
// librx.so holds it until the process exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "rx.h"
#include "rx_internal.h"
#include "sm103_ptx.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;   // 8 MiB, see RX_STATIC_SCRATCH_BYTES
constexpr size_t kStateBytes = 256;                 // DevState block at the start
constexpr int kMaxDevices = 128;

static_assert(kScratchBytes == RX_STATIC_SCRATCH_BYTES, "header and library disagree");

// The scratch.  In host code this name is only a stand-in for the symbol, not
// a device address: never pass it to a kernel; use the address from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Writes the state block the attention kernel reads: the window is one run of
// W tokens (valid = W frames of one token, head 0), and the error word is
// cleared.  The values travel as kernel arguments, so nothing on the host has
// to outlive the call.  It waits for the stream's previous kernel, which may
// be an earlier call still reading the block.
__global__ void static_state_kernel(rx::DevState* st, int W) {
  rx::grid_dependency_wait();
  rx::grid_launch_dependents();
  if (threadIdx.x == 0) {
    st->head = 0;
    st->valid = W;
    st->pushes = 0;
    st->append_arrivals = 0;
    st->err = 0;
  }
}

rx_status reject(rx_status s, const char* msg) {
  rx::set_last_error("rx_attend_regions_static", msg);
  return s;
}

}  // namespace

extern "C" rx_status rx_attend_regions_static(const void* q, int S, int Hq, int Hkv, int D,
                                              const void* k_pin, const void* v_pin, int P,
                                              const void* k_win, const void* v_win, int W,
                                              const void* k_dyn, const void* v_dyn, int n_dyn,
                                              void* out, void* stream) {
  try {
    if (S < 1 || Hq < 1 || Hkv < 1 || P < 0 || W < 0 || n_dyn < 0 || P + W + n_dyn < 1)
      return reject(RX_ERR_ARG, "sizes out of range");
    if (Hq % Hkv) return reject(RX_ERR_ARG, "Hq must be a multiple of Hkv");
    const int G = Hq / Hkv;
    if ((G & (G - 1)) != 0 || G > rx::kBM) return reject(RX_ERR_UNSUPPORTED, "Hq/Hkv must be a power of two <= 128");
    if (D != 64 && D != 128 && D != 256) return reject(RX_ERR_UNSUPPORTED, "head dim not in {64, 128, 256}");
    if (!q || !out || (P && (!k_pin || !v_pin)) || (W && (!k_win || !v_win)) ||
        (n_dyn && (!k_dyn || !v_dyn)))
      return reject(RX_ERR_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(out) || (P && (!aligned16(k_pin) || !aligned16(v_pin))) ||
        (W && (!aligned16(k_win) || !aligned16(v_win))) ||
        (n_dyn && (!aligned16(k_dyn) || !aligned16(v_dyn))))
      return reject(RX_ERR_ARG, "pointers must be 16-byte aligned");

    const size_t rows_pad = (static_cast<size_t>(S) * G + rx::kBM - 1) / rx::kBM * rx::kBM;
    // Split partials: per row and split, D bf16 values and up to 4 (m, l) pairs.
    const size_t per_split = static_cast<size_t>(Hkv) * rows_pad * (static_cast<size_t>(D) * 2 + 32);
    const size_t fit = (kScratchBytes - kStateBytes) / per_split;
    if (fit < 1) return reject(RX_ERR_CAPACITY, "Hkv * S * Hq/Hkv query rows exceed the 8 MiB static scratch");

    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return reject(RX_ERR_CUDA, cudaGetErrorString(e));
    if (major != 10 || minor != 3) return reject(RX_ERR_UNSUPPORTED, "the kernels are built for sm_103a");
    if (dev >= kMaxDevices) return reject(RX_ERR_UNSUPPORTED, "device index too large");
    void* base = nullptr;
    e = scratch_address(dev, &base);
    if (e != cudaSuccess) return reject(RX_ERR_CUDA, cudaGetErrorString(e));

    // Scratch layout: [DevState | split partials].
    char* sb = static_cast<char*>(base);
    rx::DevState* st = reinterpret_cast<rx::DevState*>(sb);
    const size_t use_splits = fit < 64 ? fit : 64;

    // The kernel reads the window length as valid * F from the state block;
    // here the window is one run of W tokens (F = 1).  Every call rewrites the
    // block on its stream, clearing the error word.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = rx::launch_k(static_state_kernel, dim3(1), dim3(32), 0, s, st, W);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return reject(RX_ERR_CUDA, cudaGetErrorString(e));

    // Tensor maps over the caller's regions: (D, Hkv, tokens, 1).  An empty
    // region gets a one-token map on another valid buffer; it is never read.
    const void* any = n_dyn ? k_dyn : (W ? k_win : k_pin);
    CUtensorMap tm[4];
    const uint64_t tok = static_cast<uint64_t>(Hkv) * D * 2;
    const void* bases[4] = {P ? k_pin : any, P ? v_pin : any, W ? k_win : any, W ? v_win : any};
    const int ntok[4] = {P ? P : 1, P ? P : 1, W ? W : 1, W ? W : 1};
    for (int i = 0; i < 4; ++i) {
      const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv),
                                static_cast<uint64_t>(ntok[i]), 1};
      const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2, tok, ntok[i] * tok};
      const uint32_t box[4] = {64u, 1u, static_cast<uint32_t>(rx::kBN), 1u};
      if (!rx::encode_tmap_4d(&tm[i], bases[i], dims, strides, box))
        return reject(RX_ERR_CUDA, "tensor-map encoding failed");
    }
    rx::AttnLaunch a;
    a.pin_k_tiles = a.pin_v_tiles = a.win_k_tiles = a.win_v_tiles = nullptr;   // caller layout: TMA
    a.pin_head_stride = a.win_head_stride = 0;
    a.tm_pin_k = &tm[0];
    a.tm_pin_v = &tm[1];
    a.tm_slide_k = &tm[2];
    a.tm_slide_v = &tm[3];
    a.layer = 0;
    a.P = P;
    a.F = 1;
    a.N = W;
    a.slots = W;
    a.D = D;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.st = st;
    a.err = &st->err;
    a.xchg = sb + kStateBytes;
    a.max_splits = static_cast<int>(use_splits);
    a.forced_splits = 0;
    a.forced_dparts = 0;
    a.inject_tx = 0;
    a.num_sms = sms;
    rx::AttnSegment seg{q, k_dyn, v_dyn, out, S, n_dyn, nullptr, 1, 0, 0};
    e = rx::launch_partitioned_attention(a, &seg, 1, s, nullptr);
    if (e != cudaSuccess) return reject(RX_ERR_CUDA, cudaGetErrorString(e));
    return RX_OK;
  } catch (...) {
    return reject(RX_ERR_ARG, "unexpected host exception");
  }
}
