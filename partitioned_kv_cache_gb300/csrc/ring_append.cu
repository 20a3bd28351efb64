// ring_append.cu -- O(1) FIFO append of one observation frame into every
// layer's sliding window.
//
// "Reflex: Real-Time VLA Control through Streaming Inference", §III "System
// architecture": each tick enqueues the newest frame and evicts the oldest;
// §V "Key implementation": add_new_prefix() adds the new tokens and reports
// evictions, evict_source_prefix() drops the oldest frame from all layers.
//
// The window of layer l is N frame slots [l][slot][F][Hkv][D].  A push copies
// the frame into slot `head` of every layer -- overwriting the oldest frame
// once the window is full, which is the eviction -- and advances
// head <- (head+1) mod N, valid <- min(valid+1, N).  Nothing else moves.
// The state update is done on the device by the last CTA to finish, so a
// captured CUDA graph replays pushes correctly.
#include <cuda_runtime.h>

#include <cstdint>

#include "rx_internal.h"

namespace rx {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;   // 16-byte vectors per thread per tensor

__global__ void __launch_bounds__(kThreads) ring_append_kernel(
    const uint4* __restrict__ k_src, const uint4* __restrict__ v_src, uint4* __restrict__ k_win,
    uint4* __restrict__ v_win, DevState* st, int L, int N, long long frame_vecs) {
  // Every CTA reads head before any CTA can update it (the update waits for
  // all CTAs to arrive).
  const int head = *reinterpret_cast<volatile int*>(&st->head);
  const long long total = static_cast<long long>(L) * frame_vecs;
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i < total; i += stride * kVecPerThread) {
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
        const long long l = idx[u] / frame_vecs;
        const long long off = idx[u] - l * frame_vecs;
        const long long dst = (l * N + head) * frame_vecs + off;
        k_win[dst] = kv[u];
        v_win[dst] = vv[u];
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int prev = atomicAdd(&st->append_arrivals, 1u);
    if (prev == gridDim.x - 1) {
      st->head = head + 1 == N ? 0 : head + 1;
      st->valid = st->valid < N ? st->valid + 1 : N;
      st->pushes += 1;
      st->append_arrivals = 0;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_ring_append(const void* k_src, const void* v_src, void* k_win, void* v_win,
                               DevState* st, int L, int N, long long frame_bytes, int num_sms,
                               cudaStream_t s) {
  const long long frame_vecs = frame_bytes / 16;
  const long long total = static_cast<long long>(L) * frame_vecs;
  long long blocks = (total + static_cast<long long>(kThreads) * kVecPerThread - 1) /
                     (static_cast<long long>(kThreads) * kVecPerThread);
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  ring_append_kernel<<<static_cast<unsigned int>(blocks), kThreads, 0, s>>>(
      static_cast<const uint4*>(k_src), static_cast<const uint4*>(v_src),
      static_cast<uint4*>(k_win), static_cast<uint4*>(v_win), st, L, N, frame_vecs);
  count_launch();
  return cudaGetLastError();
}

}  // namespace rx
