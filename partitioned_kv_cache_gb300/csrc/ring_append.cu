// ring_append.cu -- O(1) FIFO append of one observation frame into every
// layer's sliding window, and the tiled store layout it writes.
//
// "Reflex: Real-Time VLA Control through Streaming Inference", §III "System
// architecture": each tick enqueues the newest frame and evicts the oldest;
// §V "Key implementation": add_new_prefix() adds the new tokens and reports
// evictions, evict_source_prefix() drops the oldest frame from all layers.
//
// The window of (layer l, K/V head g) holds N frame slots of F tokens (N + 1
// with a spare slot); slot s covers window tokens [s*F, s*F + F).  A push
// writes the frame into slot `head` of every layer -- overwriting the oldest
// frame once the window is full, which is the eviction (with a spare slot the
// overwritten slot is the one evicted by the previous push, already outside
// every published window) -- and advances head <- (head+1) mod slots,
// valid <- min(valid+1, N).  Nothing else moves.  The state update is done on
// the device by the last CTA to finish, so a captured CUDA graph replays
// pushes correctly.
//
// Tokens are stored in the tiled layout described in rx_internal.h (tiles of
// 64 tokens, 128-byte rows, chunk ^ (token & 7) swizzle), so that the
// attention kernel moves a whole tile with one bulk copy.  The same packing
// serves the one-time pinned-prefix copy.
//
// When whole tiles are written (F, or the start token, a multiple of 64) the
// tensor-memory-access unit does the re-layout: one CTA per destination tile
// loads the source tokens as 128-byte-swizzled boxes, which is exactly the
// tile layout, and stores the tile back with one bulk copy.  Otherwise a
// thread per 16-byte chunk computes the tiled offset.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "rx_internal.h"
#include "sm103_ptx.cuh"

namespace rx {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;   // 16-byte chunks per thread per tensor

// Byte offset of 16-byte chunk c of token tok of (layer l, head g).
__device__ __forceinline__ long long tiled_offset(int l, int g, int Hkv, int T, int D, int tok,
                                                  int c) {
  const int t = tok >> 6, r = tok & 63, kb = c >> 3, cb = c & 7;
  return ((static_cast<long long>(l) * Hkv + g) * T + t) * tile_bytes(D) + kb * 8192LL + r * 128 +
         ((cb ^ (r & 7)) << 4);
}

// Neither packing kernel lets the next kernel launch early (no
// griddepcontrol.launch_dependents: the next kernel is released when this
// grid completes).  Measured on GB300 with a tick of the long-history stack:
// when a push released the attention chain after it early, the attention
// launches of the whole tick took ~1 us longer each (2.41 against 2.20 ms
// a tick); the chain's CTAs are launched while the push's CTAs still hold
// the SMs' shared memory.
__global__ void __launch_bounds__(kThreads) pack_tiles_kernel(
    const uint4* __restrict__ k_src, const uint4* __restrict__ v_src, uint8_t* __restrict__ k_dst,
    uint8_t* __restrict__ v_dst, int L, int n, int Hkv, int D, int T, int tok0, DevState* st,
    int F, int N, int slots) {
  grid_dependency_wait();
  // A ring append reads the state before any CTA can update it (the update
  // waits for every CTA to arrive).
  int head = 0, valid = 0;
  if (st) load_ring_state(st, &head, &valid);
  const int base_tok = st ? head * F : tok0;
  const int cpt = D >> 3;   // 16-byte chunks per token and head
  const long long total = static_cast<long long>(L) * n * Hkv * cpt;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += stride * kVecPerThread) {
    uint4 kv[kVecPerThread], vv[kVecPerThread];
    long long idx[kVecPerThread];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      idx[u] = i + u * stride;
      if (idx[u] < total) {
        kv[u] = k_src[idx[u]];
        vv[u] = v_src[idx[u]];
      }
    }
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      if (idx[u] < total) {
        long long rest = idx[u];
        const int c = static_cast<int>(rest % cpt);
        rest /= cpt;
        const int g = static_cast<int>(rest % Hkv);
        rest /= Hkv;
        const int f = static_cast<int>(rest % n);
        const int l = static_cast<int>(rest / n);
        const long long off = tiled_offset(l, g, Hkv, T, D, base_tok + f, c);
        *reinterpret_cast<uint4*>(k_dst + off) = kv[u];
        *reinterpret_cast<uint4*>(v_dst + off) = vv[u];
      }
    }
  }
  if (!st) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int prev = atomicAdd(&st->append_arrivals, 1u);
    if (prev == gridDim.x - 1) {
      // Every CTA fenced its frame writes before arriving: publish.
      __threadfence();
      publish_ring_state(st, head + 1 == slots ? 0 : head + 1, valid < N ? valid + 1 : N);
      st->pushes += 1;
      st->append_arrivals = 0;
      __threadfence();
    }
  }
}

// One CTA per stream: append k_new[b] / v_new[b] at position tail_len[b].
__global__ void __launch_bounds__(64) tail_append_kernel(
    uint4* __restrict__ k_tail, uint4* __restrict__ v_tail, int* __restrict__ tail_len,
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, const int* __restrict__ active,
    int tail_cap, int vecs, int* overflow) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  if (active && active[b] == 0) return;
  const int len = tail_len[b];   // every thread reads it before thread 0 advances it
  if (len < 0 || len >= tail_cap) {
    if (threadIdx.x == 0 && overflow) atomicOr(overflow, 1);
    return;
  }
  const long long dst = (static_cast<long long>(b) * tail_cap + len) * vecs;
  for (int i = threadIdx.x; i < vecs; i += blockDim.x) {
    k_tail[dst + i] = k_new[static_cast<long long>(b) * vecs + i];
    v_tail[dst + i] = v_new[static_cast<long long>(b) * vecs + i];
  }
  __syncthreads();
  if (threadIdx.x == 0) tail_len[b] = len + 1;
}

__global__ void __launch_bounds__(kThreads) unpack_tiles_kernel(
    const uint8_t* __restrict__ k_tiles, const uint8_t* __restrict__ v_tiles, uint4* __restrict__ k_dst,
    uint4* __restrict__ v_dst, int layer, int tok0, int n, int Hkv, int D, int T) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int cpt = D >> 3;
  const long long total = static_cast<long long>(n) * Hkv * cpt;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * kThreads) {
    long long rest = i;
    const int c = static_cast<int>(rest % cpt);
    rest /= cpt;
    const int g = static_cast<int>(rest % Hkv);
    const int f = static_cast<int>(rest / Hkv);
    const long long off = tiled_offset(layer, g, Hkv, T, D, tok0 + f, c);
    k_dst[i] = *reinterpret_cast<const uint4*>(k_tiles + off);
    v_dst[i] = *reinterpret_cast<const uint4*>(v_tiles + off);
  }
}

// One CTA per destination tile: blockIdx.x = source tile (64 tokens),
// blockIdx.y = layer * Hkv + head, blockIdx.z = K (0) or V (1).
struct PackTma {
  CUtensorMap tm[2];    // sources (D, Hkv, n, L), box (64, 1, 64, 1), 128-byte swizzle
  uint8_t* dst[2];      // tiled regions
  DevState* st;         // ring append when non-null
  int Hkv, D, T, tok0, F, N, slots;
};

// The last of the grid's CTAs to arrive publishes the advanced state.  acq_rel:
// each CTA's read of the old state is ordered before its arrival, and the
// publisher's stores after every arrival.
__device__ __forceinline__ void arrive_and_publish(DevState* st, unsigned int total, int head,
                                                   int valid, int N, int slots) {
  unsigned int prev;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
               : "=r"(prev)
               : "l"(&st->append_arrivals)
               : "memory");
  if (prev == total - 1) {
    publish_ring_state(st, head + 1 == slots ? 0 : head + 1, valid < N ? valid + 1 : N);
    st->pushes += 1;
    st->append_arrivals = 0;
    __threadfence();
  }
}

__global__ void __launch_bounds__(32) pack_tiles_tma_kernel(const __grid_constant__ PackTma a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;   // swizzle atoms are 1 KB
  const uint32_t bar = base + static_cast<uint32_t>(tile_bytes(a.D));
  const int l = blockIdx.y / a.Hkv, g = blockIdx.y % a.Hkv, kv = blockIdx.z;
  // The source tile is fetched towards L2 while the previous kernel finishes
  // (a hint: safe before the dependency wait), so the boxes below come from
  // L2 rather than DRAM.
  if (threadIdx.x == 0)
    for (int kb = 0; kb < a.D / 64; ++kb) tma_prefetch_l2_4d(&a.tm[kv], kb * 64, g, blockIdx.x * kTileTok, l);
  grid_dependency_wait();   // no early release of the next kernel (see pack_tiles_kernel)
  if (threadIdx.x != 0) return;
  const uint32_t bytes = static_cast<uint32_t>(tile_bytes(a.D));
  // The source boxes do not depend on the ring state: issue them first and
  // read the state while they are in flight.
  mbar_init(bar, 1);
  fence_barrier_init();
  mbar_arrive_expect_tx(bar, bytes);
  for (int kb = 0; kb < a.D / 64; ++kb)
    tma_load_4d(base + kb * 8192, &a.tm[kv], kb * 64, g, blockIdx.x * kTileTok, l, bar);
  int head = 0, valid = 0;
  if (a.st) load_ring_state(a.st, &head, &valid);
  const bool spare = a.slots > a.N;
  const unsigned int total = gridDim.x * gridDim.y * gridDim.z;
  if (a.st && !spare) {
    // Without a spare slot every reader of the state and of the slot is
    // ordered after this kernel's completion, which makes the tile visible:
    // the publish only has to wait until every CTA has read the old state.
    arrive_and_publish(a.st, total, head, valid, a.N, a.slots);
  }
  const int base_tok = a.st ? head * a.F : a.tok0;   // a multiple of 64 (host-checked)
  volatile int gave_up = 0;
  const bool ok = mbar_wait(bar, 0, &gave_up);
  if (ok) {
    uint8_t* dst = a.dst[kv] + ((static_cast<long long>(l) * a.Hkv + g) * a.T + base_tok / kTileTok + blockIdx.x) * bytes;
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(base), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (spare) {
      // Spare-slot ring: attention may run concurrently and reads the state
      // as soon as it is published, so the tile must be written first.
      asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
    } else {
      // Only the shared-memory source must be read before this CTA exits.
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
  } else {
    // the copy may still land in shared memory: wait for it (bounded) before exiting
    volatile int no_abort = 0;
    mbar_wait(bar, 0, &no_abort);
    if (a.st) atomicOr(&a.st->err, kErrAppendTimeout);
  }
  if (a.st && spare) {
    __threadfence();
    arrive_and_publish(a.st, total, head, valid, a.N, a.slots);
  }
}

}  // namespace

cudaError_t launch_pack_tiles(const void* k_src, const void* v_src, void* k_dst, void* v_dst,
                              int L, int n, int Hkv, int D, int T, int tok0, DevState* st, int F,
                              int N, int slots, int num_sms, cudaStream_t s) {
  // Whole destination tiles: the TMA path.
  const bool whole = st ? (F % kTileTok == 0) : (tok0 % kTileTok == 0);
  if (whole && n > 0) {
    PackTma a;
    memset(&a, 0, sizeof(a));
    const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv), static_cast<uint64_t>(n),
                              static_cast<uint64_t>(L)};
    const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Hkv) * D * 2,
                                 static_cast<uint64_t>(n) * Hkv * D * 2};
    const uint32_t box[4] = {64u, 1u, static_cast<uint32_t>(kTileTok), 1u};
    if (encode_tmap_4d(&a.tm[0], k_src, dims, strides, box) && encode_tmap_4d(&a.tm[1], v_src, dims, strides, box)) {
      a.dst[0] = static_cast<uint8_t*>(k_dst);
      a.dst[1] = static_cast<uint8_t*>(v_dst);
      a.st = st;
      a.Hkv = Hkv;
      a.D = D;
      a.T = T;
      a.tok0 = tok0;
      a.F = F;
      a.N = N;
      a.slots = slots;
      const size_t smem = static_cast<size_t>(tile_bytes(D)) + 1024 + 16;
      const dim3 grid(static_cast<unsigned int>((n + kTileTok - 1) / kTileTok), static_cast<unsigned int>(L * Hkv), 2);
      const cudaError_t e = launch_k(pack_tiles_tma_kernel, grid, dim3(32), smem, s, a);
      return e != cudaSuccess ? e : cudaGetLastError();
    }
  }
  const long long total = static_cast<long long>(L) * n * Hkv * (D >> 3);
  long long blocks = (total + static_cast<long long>(kThreads) * kVecPerThread - 1) /
                     (static_cast<long long>(kThreads) * kVecPerThread);
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const cudaError_t e = launch_k(pack_tiles_kernel, dim3(static_cast<unsigned int>(blocks)),
                                 dim3(kThreads), 0, s, static_cast<const uint4*>(k_src),
                                 static_cast<const uint4*>(v_src), static_cast<uint8_t*>(k_dst),
                                 static_cast<uint8_t*>(v_dst), L, n, Hkv, D, T, tok0, st, F, N, slots);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_tail_append(void* k_tail, void* v_tail, int* tail_len, const void* k_new,
                               const void* v_new, const int* active, int B, int tail_cap, int Hkv,
                               int D, int* overflow, cudaStream_t s) {
  if (B == 0) return cudaSuccess;
  const int vecs = Hkv * D / 8;
  const cudaError_t e = launch_k(tail_append_kernel, dim3(B), dim3(64), 0, s,
                                 static_cast<uint4*>(k_tail), static_cast<uint4*>(v_tail), tail_len,
                                 static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
                                 active, tail_cap, vecs, overflow);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_unpack_tiles(const void* k_tiles, const void* v_tiles, void* k_dst, void* v_dst,
                                int layer, int tok0, int n, int Hkv, int D, int T, cudaStream_t s) {
  const long long total = static_cast<long long>(n) * Hkv * (D >> 3);
  long long blocks = (total + kThreads - 1) / kThreads;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  const cudaError_t e = launch_k(unpack_tiles_kernel, dim3(static_cast<unsigned int>(blocks)),
                                 dim3(kThreads), 0, s, static_cast<const uint8_t*>(k_tiles),
                                 static_cast<const uint8_t*>(v_tiles), static_cast<uint4*>(k_dst),
                                 static_cast<uint4*>(v_dst), layer, tok0, n, Hkv, D, T);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rx
