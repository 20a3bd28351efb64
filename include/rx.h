/*
 * rx.h -- C ABI of the GB300 partitioned KV cache and attention library
 * (librx.so, built for sm_103a).
 *
 * What it computes
 * ----------------
 * Streaming inference for flow-matching vision-language-action policies as
 * described in "Reflex: Real-Time VLA Control through Streaming Inference":
 *
 *  - §III "System architecture": the attention context is split into a
 *    pinned instruction prefix (computed once), a sliding history holding a
 *    FIFO of N observation frames (each tick enqueues the newest frame and
 *    evicts the oldest) and a dynamic flow-state suffix recomputed at every
 *    denoising step.
 *  - §III "Core formulas", Eq. (1): the suffix queries attend with one softmax
 *    over the concatenation [K_pin; K_slide(t); K_dyn(k)] (values likewise);
 *    Proposition A.1: the result equals full-batch attention.
 *  - §III "Core formulas", Eq. (2): AdaRMSNorm(x, c) = x / RMS(x) * gamma(c),
 *    gamma(c) = 1 + MLP(c), RMS with an FP32 mean of squares.
 *  - §V "Key implementation": a statically preallocated, zero-initialised
 *    ring buffer with a write pointer; add_new_prefix() reports evictions.
 *
 * "OxyGen: Unified KV Cache Management for Vision-Language-Action Models under
 * Multi-Task Parallelism", §"Core method": several requests read one
 * read-only prefill cache while each keeps its own appended KV
 * (rx_attend_batch).
 *
 * Conventions
 * -----------
 *  - Every function returns an rx_status: 0 on success, negative on error.
 *    No C++ exception crosses this boundary.  rx_last_error() gives a
 *    thread-local message for the last failure on the calling thread.
 *  - "bf16" buffers hold IEEE bfloat16 values, row-major in the stated shape,
 *    densely packed.  Unless stated otherwise a pointer is DEVICE memory
 *    owned by the caller, 16-byte aligned; the library only reads inputs
 *    and writes outputs during the call's stream work and keeps no pointer
 *    to them afterwards.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls enqueue work and return without synchronising, except
 *    where stated.  Work for one cache must stay in stream order: the cache
 *    owns one workspace and one device-side {head, valid} state.
 *  - Shapes: L layers, Hq query heads, Hkv key/value heads (Hq = G*Hkv, G a
 *    power of two <= 128; query head h reads key/value head h / G), head
 *    dimension D in {64, 128, 256}.
 */
#ifndef RX_H
#define RX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rx_status {
  RX_OK = 0,
  RX_ERR_ARG = -1,         /* null/misaligned pointer, bad shape or size    */
  RX_ERR_LAYER = -2,       /* layer index outside [0, L)                    */
  RX_ERR_CAPACITY = -3,    /* P > P_cap, S > S_cap, tail > tail_cap, ...    */
  RX_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed             */
  RX_ERR_TIMEOUT = -5,     /* a bounded device-side wait gave up            */
  RX_ERR_UNSUPPORTED = -6, /* shape the kernels do not handle (D, G, GPU)   */
  RX_ERR_STATE = -7        /* call made in an invalid state                 */
} rx_status;

/* Opaque store: owns the pinned and sliding regions of every layer, the
 * device-side ring state and the attention workspace, all in one device
 * allocation made by rx_cache_create. */
typedef struct rx_cache* rx_cache_t;

typedef struct rx_config {
  int L;        /* layers                                                   */
  int Hq;       /* query heads                                              */
  int Hkv;      /* key/value heads                                          */
  int D;        /* head dimension: 64, 128 or 256                           */
  int P_cap;    /* pinned-prefix capacity, tokens (>= 0)                    */
  int N;        /* frames in the sliding window (>= 1)                      */
  int F;        /* tokens per frame (>= 1)                                  */
  int S_cap;    /* most query tokens of one attention call (>= 1)           */
  int tail_cap; /* private tail capacity of a language stream (>= 0)        */
  int max_req;  /* most language query tokens (B*T) of one rx_attend_batch  */
  int spare_slot; /* 1: keep one spare frame slot (N+1 slots) so that pushes
                     can run concurrently with attention (rx_push_frame_async);
                     requires F % 64 == 0.  0: N slots.                      */
} rx_config;

/* Allocate and zero every region ("Reflex ...", §V: the ring buffer is
 * allocated once at model load with torch.zeros and a write pointer of 0).
 * Device = the current CUDA device.  Synchronous.  On success *out owns the
 * allocation until rx_cache_destroy.  Errors: RX_ERR_ARG (bad config),
 * RX_ERR_UNSUPPORTED (D, G, or a GPU without sm_103a tcgen05), RX_ERR_CUDA. */
rx_status rx_cache_create(const rx_config* cfg, rx_cache_t* out);

/* Free everything the cache owns.  Synchronises the device first.  NULL is a
 * no-op.  Errors: RX_ERR_CUDA (the synchronisation or the free failed). */
rx_status rx_cache_destroy(rx_cache_t cache);

/* Copy the instruction prefix into the pinned region ("Reflex ...", §III
 * Eq. 1 where-clause: K_pin, V_pin are computed once at t = 0 and pinned).
 * k, v: bf16 [L][P][Hkv][D], host or device memory (copied with
 * cudaMemcpyDefault, stream-ordered).  0 <= P <= P_cap.  Re-pinning replaces
 * the prefix.  Errors: RX_ERR_ARG, RX_ERR_CAPACITY, RX_ERR_CUDA. */
rx_status rx_pin_prefix(rx_cache_t cache, const void* k, const void* v, int P,
                        void* stream);

/* Ring append ("Reflex ...", §III "System architecture", sliding history;
 * §V add_new_prefix / evict_source_prefix): for every layer write one frame's
 * K/V into the slot at the device-side head, then head <- (head+1) mod N and
 * valid <- min(valid+1, N).  Only the new frame is moved: O(L*F*Hkv*D) bytes,
 * independent of N.  k, v: bf16 [L][F][Hkv][D], device memory.
 * evicted (host, nullable): 1 if this push overwrote the oldest frame, else 0,
 * from the host's count of pushes made through this function.
 * Errors: RX_ERR_ARG, RX_ERR_CUDA. */
rx_status rx_push_frame(rx_cache_t cache, const void* k, const void* v,
                        int* evicted, void* stream);

/* Ring append on a producer stream, concurrent with attention on a consumer
 * stream ("Reflex ...", §III "System architecture": Thread A encodes frames
 * into the ring buffer while Thread B reads the latest tokens and denoises).
 * Needs a cache created with spare_slot = 1.  The frame is written into the
 * spare slot, which no published window contains; the last CTA then
 * publishes {head, valid} in one 64-bit store, so an attention kernel reads
 * either the previous window or the new one, never a mix.  Ordering, by CUDA
 * events (no device spinning): producer_stream first waits for all work
 * already enqueued on consumer_stream, and consumer_stream waits for the
 * previous asynchronous push.  So every attention enqueued after this call sees
 * the window after the previous push or after this one, and the slot this push
 * overwrites can only be read by work that the producer waited for.  The push
 * runs concurrently with consumer work enqueued after the call.
 * Errors: RX_ERR_STATE (cache without a spare slot), RX_ERR_ARG, RX_ERR_CUDA. */
rx_status rx_push_frame_async(rx_cache_t cache, const void* k, const void* v,
                              int* evicted, void* producer_stream,
                              void* consumer_stream);

/* Partitioned attention for one layer ("Reflex ...", §III Eq. 1): for every
 * suffix token s and query head h,
 *   out[s][h] = softmax_j( q[s][h] . K_j / sqrt(D) ) V_j
 * over all keys j of [pinned P; the window's valid*F frame tokens; k_dyn S],
 * key/value head h / G.  No mask.  The window is read in place in physical
 * slot order (softmax is order-invariant, Proposition A.1).
 * q: bf16 [S][Hq][D]; k_dyn, v_dyn: bf16 [S][Hkv][D]; out: bf16 [S][Hq][D];
 * 1 <= S <= S_cap.  fp32 accumulation and softmax; out rounded once to bf16.
 * Errors: RX_ERR_ARG, RX_ERR_LAYER, RX_ERR_CAPACITY, RX_ERR_CUDA. */
rx_status rx_attend_suffix(rx_cache_t cache, int layer, const void* q,
                           const void* k_dyn, const void* v_dyn, int S,
                           void* out, void* stream);

/* Block-causal variant of rx_attend_suffix (the other plain reading of the
 * attention-mask figure of "Reflex ...", §III "System architecture"): the
 * first n_state suffix tokens (the state block) attend over the cached
 * regions and only the state block's own dynamic keys, k_dyn[0, n_state);
 * the remaining (action) tokens attend over every key.  n_state = 0 is
 * rx_attend_suffix.  0 <= n_state <= S.  Errors as rx_attend_suffix. */
rx_status rx_attend_suffix_block_causal(rx_cache_t cache, int layer, const void* q,
                                        const void* k_dyn, const void* v_dyn, int S,
                                        int n_state, void* out, void* stream);

/* A dense batch of language streams sharing the cache: B streams of T query
 * tokens each, every stream with its own appended keys (its private tail). */
typedef struct rx_stream_batch {
  const void* q;        /* bf16 [B][T][Hq][D]                                   */
  const void* k_tail;   /* bf16 [B][tail_cap][Hkv][D]: stream b's appended keys */
  const void* v_tail;   /* bf16 [B][tail_cap][Hkv][D]                           */
  const int* tail_len;  /* DEVICE int32 [B]: keys held by each tail, clamped to
                           [0, tail_cap] by the kernel (read on the device, so a
                           captured graph follows tails that grow)             */
  void* out;            /* bf16 [B][T][Hq][D]                                   */
  int B;                /* streams, >= 0                                        */
  int T;                /* query tokens per stream, >= 1                        */
} rx_stream_batch;

/* Shared-cache multi-request attention in ONE launch ("OxyGen ...",
 * §"Core method": one read-only prefill cache serves the action expert across
 * its denoising steps while language streams, stacked along a batch
 * dimension, each append their own KV).  The action suffix attends over
 * [pinned; window; its k_dyn] exactly as rx_attend_suffix; stream b attends
 * over [pinned; window; its first tail_len[b] tail keys] and nothing another
 * stream appended.  Both groups share every K/V tile of the cache in the same
 * launch.
 * Action: q_act [S][Hq][D], k_dyn/v_dyn [S][Hkv][D], out_act [S][Hq][D];
 * S = 0 (pointers may be NULL) for no action suffix; S <= S_cap.
 * lang: may be NULL (or B = 0) for no language streams; B*T <= max_req and
 * the cache's tail_cap >= 1.  A stream whose tail is empty and whose cache
 * regions hold no key gets zeros.
 * Errors: RX_ERR_ARG, RX_ERR_LAYER, RX_ERR_CAPACITY, RX_ERR_CUDA. */
rx_status rx_attend_batch(rx_cache_t cache, int layer, const void* q_act,
                          const void* k_dyn, const void* v_dyn, int S,
                          void* out_act, const rx_stream_batch* lang,
                          void* stream);

/* One AdaRMSNorm ("Reflex ...", §III Eq. (2); §V forward) over `rows` rows
 * of width d, for an attention call to run in the same launch:
 *   y = x * rsqrt(mean(x^2) + eps) * gamma, mean of squares in fp32.
 * x, y: bf16 [rows][d] device memory; gamma: fp32 [d]; d % 8 == 0; rows >= 0;
 * all 16-byte aligned.  y may not overlap x or another job's x or y. */
typedef struct rx_norm_rows {
  const void* x;
  const float* gamma;
  void* y;
  int rows;
  int d;
  float eps;
} rx_norm_rows;
#define RX_MAX_NORM_JOBS 2

/* rx_attend_suffix and up to RX_MAX_NORM_JOBS AdaRMSNorm jobs in ONE launch,
 * the FP32-variance AdaRMSNorm fused in beside the partitioned attention
 * ("Reflex ...", §III "Model components": AdaRMSNorm before the attention and
 * before the MLP of every layer).  The attention output
 * is that of rx_attend_suffix and every y is bit for bit that of
 * rx_adarmsnorm on the same arguments.  The norm rows run on the attention
 * CTAs' softmax warps while those wait for their first score tile.  The jobs
 * must not read what the attention call writes or write what it reads (the
 * launch runs both at once): a job whose y overlaps q, k_dyn, v_dyn or out,
 * or whose x or gamma overlaps out, is refused with RX_ERR_ARG.  n_norms = 0
 * is rx_attend_suffix.
 * Errors: those of rx_attend_suffix and rx_adarmsnorm (RX_ERR_ARG for a bad
 * job). */
rx_status rx_attend_suffix_norms(rx_cache_t cache, int layer, const void* q,
                                 const void* k_dyn, const void* v_dyn, int S,
                                 void* out, const rx_norm_rows* norms,
                                 int n_norms, void* stream);

/* rx_attend_batch with norm jobs in the same launch, as
 * rx_attend_suffix_norms (no job may write the action's or the language
 * streams' inputs, tails or tail lengths, nor read or write their outputs).
 * With neither an action suffix nor language streams, the jobs run as
 * rx_adarmsnorm launches.  Errors: those of rx_attend_batch and
 * rx_adarmsnorm (RX_ERR_ARG for a bad or overlapping job). */
rx_status rx_attend_batch_norms(rx_cache_t cache, int layer, const void* q_act,
                                const void* k_dyn, const void* v_dyn, int S,
                                void* out_act, const rx_stream_batch* lang,
                                const rx_norm_rows* norms, int n_norms,
                                void* stream);

/* Append one token to each active language stream's private tail (cross-frame
 * continuous batching, "OxyGen ...", §"Core method": a stream's KV cache grows
 * by one entry per decoded token and the stream resumes across frames).
 * For every b < B with active[b] != 0 (or every b when active is NULL):
 *   if tail_len[b] < tail_cap: k_tail[b][tail_len[b]] = k_new[b],
 *                              v_tail[b][tail_len[b]] = v_new[b], tail_len[b] += 1
 *   else: the token is dropped and bit 0 of *overflow is set (a full stream
 *         must be retired; a host scheduler resets tail_len[b] = 0 to reuse it).
 * k_tail, v_tail: bf16 [B][tail_cap][Hkv][D]; k_new, v_new: bf16 [B][Hkv][D];
 * tail_len: DEVICE int32 [B] (read and advanced on the device, so a captured
 * graph keeps appending); active: DEVICE int32 [B] or NULL; overflow: DEVICE
 * int32 or NULL.  Hkv*D % 8 == 0.  Errors: RX_ERR_ARG, RX_ERR_CUDA. */
rx_status rx_tail_append(void* k_tail, void* v_tail, int* tail_len, const void* k_new,
                         const void* v_new, const int* active, int B, int tail_cap,
                         int Hkv, int D, int* overflow, void* stream);

/* Ring-state snapshot / restore (execution-state capsules as in the FlashRT
 * summary page: snapshot and restore of the named static buffers).  A
 * snapshot holds the pinned prefix, the window, the device-side ring state
 * and the host-side counters; restoring it and then pushing the same frames
 * reproduces every later output bit for bit.
 * rx_snapshot_bytes: size of a snapshot of this cache.
 * rx_snapshot: dst is caller-owned DEVICE memory of that size; the copy is
 *   enqueued on `stream` after the work already there.
 * rx_restore: src must hold a snapshot of a cache with the same rx_config;
 *   synchronises `stream` to validate it, then enqueues the copies.
 * Errors: RX_ERR_ARG (null, or a snapshot of another configuration),
 * RX_ERR_CUDA. */
rx_status rx_snapshot_bytes(rx_cache_t cache, long long* bytes);
rx_status rx_snapshot(rx_cache_t cache, void* dst, void* stream);
rx_status rx_restore(rx_cache_t cache, const void* src, void* stream);

/* Gamma of AdaRMSNorm ("Reflex ...", §III Eq. 2 and "Model components"):
 * for every weight set i and conditioning vector k
 *   c_k      = [sin(t_k w_0..), cos(t_k w_0..), state_k]   (emb_dim + state_dim)
 *   w_j      = 10000^(-j / (emb_dim/2)),  j < emb_dim/2
 *   gamma[i][k] = 1 + W2_i SiLU(W1_i c_k + b1_i) + b2_i
 * t: fp32 [n_cond]; state: fp32 [n_cond][state_dim];
 * W1: bf16 [n_sets][hidden][emb_dim+state_dim]; b1: bf16 [n_sets][hidden];
 * W2: bf16 [n_sets][d][hidden]; b2: bf16 [n_sets][d];
 * gamma: fp32 [n_sets][n_cond][d] (output).  bf16 weights, fp32 arithmetic;
 * the second layer runs on the tensor cores with SiLU(...) split into two
 * bf16 parts (~16 bits kept) and an fp32 accumulator.  W2 must be 16-byte
 * aligned.  A device-side timeout (a copy that never lands) writes NaN into
 * the affected outputs.
 * Limits: 1 <= n_cond <= 16, emb_dim even, hidden % 16 == 0 and <= 2048,
 * d % 8 == 0; RX_ERR_CUDA if the conditioning vectors and H do not fit in
 * shared memory (emb_dim + state_dim of several hundred with hidden 2048).
 * Errors: RX_ERR_ARG, RX_ERR_CUDA. */
rx_status rx_ada_gamma(const float* t, const float* state, int n_cond,
                       int emb_dim, int state_dim, const void* W1,
                       const void* b1, int hidden, const void* W2,
                       const void* b2, int d, int n_sets, float* gamma,
                       void* stream);

/* AdaRMSNorm ("Reflex ...", §III Eq. 2; §V forward): for each row
 *   y = x * rsqrt(mean(x^2) + eps) * gamma
 * with the mean of squares accumulated in fp32.  x, y: bf16 [rows][d];
 * gamma: fp32 [d]; d % 8 == 0; rows >= 0 (0 is a no-op).  y may not alias x.
 * Errors: RX_ERR_ARG, RX_ERR_CUDA. */
rx_status rx_adarmsnorm(const void* x, const float* gamma, int rows, int d,
                        float eps, void* y, void* stream);

/* Read the device-side ring state (synchronises `stream`): head = slot the
 * next push writes, valid = frames held, pushes = pushes applied on the
 * device (advances under CUDA-graph replay too).  Any pointer may be NULL.
 * Errors: RX_ERR_ARG (null cache), RX_ERR_CUDA. */
rx_status rx_get_state(rx_cache_t cache, int* head, int* valid,
                       long long* pushes, void* stream);

/* Test aid: the window's physical slots in logical order, oldest first
 * (slots: host int[N], the first *valid entries are filled).  Reads the
 * device state (synchronises `stream`).  Errors: RX_ERR_ARG (null argument),
 * RX_ERR_CUDA. */
rx_status rx_debug_window(rx_cache_t cache, int* slots, int* valid,
                          void* stream);

/* Test aid: copy one layer's window in logical order (oldest frame first)
 * into k_out, v_out: device bf16 [valid*F][Hkv][D].  Reads the device state
 * (synchronises `stream`), then enqueues the copies.  Errors: RX_ERR_ARG
 * (null argument), RX_ERR_LAYER, RX_ERR_UNSUPPORTED (N > 4096), RX_ERR_CUDA. */
rx_status rx_export_window(rx_cache_t cache, int layer, void* k_out,
                           void* v_out, void* stream);

/* Device-side error word of the cache (bit flags set by kernels whose bounded
 * waits gave up).  Synchronises `stream`; *code = 0 means no error.  The word
 * is cleared by this call. */
rx_status rx_check_device_error(rx_cache_t cache, int* code, void* stream);

/* Test aid for the bounded waits: the next attention launch of this cache
 * has its first CTA expect `bytes` more on its first K tile's barrier than
 * the copy delivers.  That barrier never completes, the CTA's waits give up
 * after their time limit (2 s), the kernel unwinds (waiting, bounded, for its
 * own copies and tensor-core work) and sets bit 1 of the error word, which
 * rx_check_device_error reports; that launch's output is undefined.  Later
 * launches are unaffected.  bytes: a multiple of 16 in [0, 2^20]; 0 cancels.
 * Errors: RX_ERR_ARG. */
rx_status rx_debug_inject_timeout(rx_cache_t cache, int bytes);

/* Test aid: the partition an attention launch chooses, computed on the host
 * from the given device figures.  Proposition A.1 of "Reflex: Real-Time VLA
 * Control through Streaming Inference" (§III "Core formulas") lets the key
 * sequence be cut into slices merged afterwards.  A launch runs `units` =
 * (128-row query tiles x K/V heads).  Each is cut into *splits key slices
 * times *dparts output-column shares.  *fused = 1 when the splits of a unit
 * form one thread-block cluster and merge on chip, 0 when a second kernel
 * merges them (or *splits = 1).  Inputs: t_max = key tiles (64 keys) of the
 * longest query segment; D = 64, 128 or 256; num_sms; max_splits = splits
 * the cache's workspace holds; forced_splits / forced_dparts = 0 for the
 * automatic choice (as rx_set_attn_splits / rx_set_attn_dparts);
 * cluster_capacity = host array of 17 ints, entry c = clusters of c CTAs the
 * device holds at once (entry 0 unused).  Touches no device.
 * Errors: RX_ERR_ARG (a size below 1 or above 2^24 (t_max, units) or 2^16
 * (num_sms, max_splits, forced_splits), a null pointer, or a column split
 * that is not 1, 2 or 4 or leaves a share narrower than 64 columns). */
rx_status rx_debug_choose_partition(int t_max, int units, int D, int num_sms, int max_splits,
                                    int forced_splits, int forced_dparts, const int* cluster_capacity,
                                    int* splits, int* dparts, int* fused);

/* Number of split-KV partitions for attention launches of this cache
 * (0 = chosen from the SM count, the default).  A tuning knob: results are
 * the same for every value up to rounding order.  Errors: RX_ERR_ARG (null
 * cache, or splits outside [0, the workspace's capacity]). */
rx_status rx_set_attn_splits(rx_cache_t cache, int splits);

/* Number of CTAs that share the output columns of one (query tile, split):
 * each computes the scores in full but the value product, and the partial it
 * merges, for D/dparts columns only.  1, 2 or 4 with D/dparts >= 64, or 0 =
 * chosen from the SM count (the default).  A tuning knob: results are the
 * same for every value up to rounding order.  Errors: RX_ERR_ARG. */
rx_status rx_set_attn_dparts(rx_cache_t cache, int dparts);

/* Kernel launches made by the library in this process (all entry points,
 * all caches).  For accounting in benchmarks.  Cannot fail. */
long long rx_launch_count(void);

const char* rx_status_str(int status);
const char* rx_last_error(void);

/* ------------------------------------------------------------------------
 * Allocation-free attention.  (The pages have no counterpart: this entry
 * point exists for callers, not for the method.)
 *
 * For callers that cannot call cudaMalloc -- a real-time control loop where
 * an allocation would synchronise the device and stall it, an embedded runtime
 * that reserved its whole memory budget up front, a plugin inside a framework
 * that owns the device allocator -- and therefore cannot create an rx_cache.
 * It computes the same attention as rx_attend_suffix, with the same kernels,
 * over K/V regions the caller already holds:
 *   out[s][h] = softmax_j(q[s][h] . K_j / sqrt(D)) V_j over the keys of
 *   [k_pin (P tokens); k_win (W tokens); k_dyn (n_dyn tokens)].
 * q, out: bf16 [S][Hq][D]; k_pin/v_pin [P][Hkv][D]; k_win/v_win [W][Hkv][D];
 * k_dyn/v_dyn [n_dyn][Hkv][D]; all device memory, 16-byte aligned; a region of
 * 0 tokens may pass NULL.  Nothing is allocated: the kernel's scratch (split
 * partials and a small state block) lives in one fixed device array of
 * RX_STATIC_SCRATCH_BYTES that every GPU loading this library holds until
 * the process exits.  Limit: Hkv * ceil(S*Hq/Hkv / 128) * 128 *
 * (2*D + 32) bytes must fit in that array (about 15 000 query rows at D = 256);
 * larger calls return RX_ERR_CAPACITY.  The first call on each device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  Every call shares
 * the one array and rewrites it, so calls that overlap on the GPU (different
 * streams, or several host threads) race: serialise them.  A device-side wait
 * that gives up is recorded in the array and is not reported by this call.
 * Errors: RX_ERR_ARG, RX_ERR_CAPACITY, RX_ERR_UNSUPPORTED, RX_ERR_CUDA. */
#define RX_STATIC_SCRATCH_BYTES (8u << 20)
rx_status rx_attend_regions_static(const void* q, int S, int Hq, int Hkv, int D,
                                   const void* k_pin, const void* v_pin, int P,
                                   const void* k_win, const void* v_win, int W,
                                   const void* k_dyn, const void* v_dyn,
                                   int n_dyn, void* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RX_H */
