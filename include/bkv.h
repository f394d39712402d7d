/*
 * bkv.h - C ABI of the BeaconKV periodic KV-cache eviction step on one GPU.
 *
 * Method source: the page "BeaconKV：用历史查询代表保护长推理的远程回看" (reading
 * notes on "BeaconKV: Key-Value Cache Compression Guided by Beacon Queries for
 * Efficient Large Reasoning Model Inference"), cited as "BeaconKV reading
 * notes" with its section and equation; buffer sizes 32 -> 16 and the 16+16
 * split also appear in the rcap.io summary of the same paper.
 *
 * For every (sequence, layer, KV head) - a "unit" - an eviction
 *   1. rotates each query head's beacon queries to the current step t and its
 *      recent queries to their own positions (notes §2.3, Q_obs equation);
 *   2. scores every cached key by softmax attention from those rows, max-pooled
 *      over rows and over the query heads of the GQA group (§2.1 eqs. 4-5,
 *      §2.3 eq. 7);
 *   3. keeps the prefix, the recent window and the top-k scores up to the
 *      budget, in slot order (§2.3 eq. 8);
 *   4. compacts K and V in place to slots [0, budget);
 *   5. compresses each query head's beacons + recents to fps_keep beacons by
 *      farthest-point sampling (§2.2 Algorithm 1, eq. 9, Algorithm 2).
 *
 * Conventions shared by every call
 *   - bf16 tensors are IEEE bfloat16, little-endian, contiguous, 16-byte
 *     aligned device memory.
 *   - Every call that launches work enqueues it on the handle's stream and
 *     returns without waiting. Argument and state errors are found on the
 *     host before anything is enqueued; they return a code and change nothing.
 *   - Errors found on the device (non-finite inputs) are latched in a status
 *     word in the workspace; bkv_sync returns and clears it.
 *   - Nothing aborts, traps or throws across this boundary.
 *   - The caller owns every pointer it passes (workspace, q_pre, K, V, kept).
 *     They must stay valid until the enqueued work completes. The library
 *     allocates no device memory; on the host it allocates the handle and,
 *     while profiling is on, a pool of CUDA events.
 *   - A handle is used from one host thread at a time.
 */
#ifndef BKV_H
#define BKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bkv_ctx* bkv_handle;

typedef enum bkv_status {
  BKV_OK = 0,
  BKV_ERR_INVALID_ARG = 1, /* null or misaligned pointer, size out of range */
  BKV_ERR_STATE = 2,       /* step out of order, cache_len not the tracked length */
  BKV_ERR_WORKSPACE = 3,   /* workspace smaller than bkv_workspace_bytes() or misaligned */
  BKV_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  BKV_ERR_NONFINITE = 5,   /* a query or key held Inf/NaN (latched on the device) */
  BKV_ERR_TIMEOUT = 6,     /* a bounded device-side wait ran out (latched on the device) */
  BKV_ERR_UNSUPPORTED = 7, /* shape the kernels do not implement (d != 128, too many rows) */
  BKV_ERR_INTERNAL = 8     /* an internal consistency check failed */
} bkv_status;

/* Keep each eviction's Score[j] in the workspace for bkv_get_scores. */
#define BKV_FLAG_KEEP_SCORES 1
/* Order-free compaction, a relaxation of eq. 8's Sort (notes §2.3): the same
 * keep set, but kept slots below the budget stay where they are and the
 * dropped slots below the budget (ascending) take the kept slots at or above
 * the budget (ascending), so at most cache_len - budget rows move instead of
 * every row after the first dropped slot. Slots [0, budget) then hold the
 * kept tokens out of position order; the appended slots [budget, cache_len)
 * stay in position order, which the next eviction's recent window and causal
 * mask rely on, so bkv_evict requires recent <= cache_len - budget. */
#define BKV_FLAG_ORDER_FREE 2
/* Mean pooling: Score[j] = the mean over all G * (beacons + recents)
 * observation rows of their attention weight on slot j (0 where a recent row
 * cannot see j), instead of the max (notes §2.1 eq. 6, the aggregation Table 2
 * compares with max pooling over queries and heads). */
#define BKV_FLAG_MEAN_POOL 4

typedef struct bkv_config {
  int32_t heads;      /* query heads per layer, H                                   */
  int32_t kv_heads;   /* KV heads per layer, Hkv; H % Hkv == 0, G = H / Hkv         */
  int32_t d;          /* head dimension; only 128 is implemented                    */
  int32_t budget;     /* B_KV^min: slots each eviction keeps (notes §2.3 eq. 8)     */
  int32_t period;     /* slots appended between evictions; the caller evicts at
                         cache_len = budget + period (notes §2.1, Figure 5)         */
  int32_t prefix;     /* n_prefix: leading slots always kept                        */
  int32_t recent;     /* trailing slots always kept (the recent KV window)          */
  int32_t fps_cap;    /* B_Q^max of eq. 9; 1 <= fps_cap <= 32                       */
  int32_t fps_keep;   /* B_Q^min = n_beacon of eq. 9; 0 <= fps_keep < fps_cap.
                         The recent-query ring holds n_rq = fps_cap - fps_keep.    */
  int32_t layers;     /* 1..128                                                     */
  int32_t batch;      /* sequences                                                  */
  int32_t max_cache;  /* slot capacity of each K/V tensor; > budget                 */
  double rope_theta;  /* RoPE base; inv_freq_i = theta^(-2i/d), rotate-half pairs   */
  int32_t flags;      /* BKV_FLAG_* bits                                            */
} bkv_config;

typedef struct bkv_stats {
  uint64_t evictions;      /* bkv_evict calls completed on the host side              */
  uint64_t fps_calls;      /* FPS launches (each covers every query head)             */
  uint64_t rows_moved;     /* K/V rows copied by compaction, summed over units (device) */
  int32_t beacons;         /* current beacons per query head                          */
  int32_t recents;         /* current recent queries per query head                   */
  int32_t cache_len;       /* cache length the library expects at the next evict      */
  int64_t last_step;       /* step of the last bkv_append_queries, -1 before the first */
} bkv_stats;

/* Bytes of device workspace a handle with this config needs (>= 256-B aligned
 * base required). Holds per query head the beacon buffer (fps_cap x d bf16),
 * the recent ring (n_rq x d bf16) and the last FPS trace, a RoPE table, the
 * status word and, with BKV_FLAG_KEEP_SCORES, layers*batch*kv_heads*max_cache
 * fp32 scores. Errors: BKV_ERR_INVALID_ARG for a null pointer or an invalid
 * config, BKV_ERR_UNSUPPORTED for d != 128 or fps_cap > 32. */
bkv_status bkv_workspace_bytes(const bkv_config* cfg, size_t* bytes);

/* Creates a handle over a caller-allocated workspace (device pointer) and a
 * CUDA stream (cudaStream_t, may be NULL for the legacy default stream).
 * Enqueues the zeroing of the library state. The stream starts with an empty
 * cache and no query state. */
bkv_status bkv_create(const bkv_config* cfg, void* workspace, size_t workspace_bytes,
                      void* cuda_stream, bkv_handle* out);

/* Makes later calls enqueue on another stream. The caller orders the two
 * streams (the library records no event). */
bkv_status bkv_set_stream(bkv_handle h, void* cuda_stream);

/* One decode step: pushes each query head's pre-RoPE query of step `step`
 * into its recent ring; when the ring already holds n_rq queries its oldest
 * moves to the end of the beacon buffer, and when that buffer reaches fps_cap
 * it is compressed to fps_keep rows by farthest-point sampling (notes §2.2,
 * eq. 9). The caller appends the step's key and value to cache slot
 * cache_len itself; the library counts that slot.
 *   q_pre: device bf16 [layers][batch][heads][d].
 *   step:  absolute position of this token; the first call may use any
 *          step >= 0, every later one must be the previous step + 1
 *          (BKV_ERR_STATE otherwise). The counted cache length may not exceed
 *          max_cache (BKV_ERR_STATE: evict first). */
bkv_status bkv_append_queries(bkv_handle h, const void* q_pre, int64_t step);

/* The eviction step at time t = step (notes §2.3 eqs. 7-8, Algorithm 2).
 *   K, V:  host arrays of `layers` device pointers; each points to a bf16
 *          [batch][kv_heads][max_cache][d] cache whose slots [0, cache_len)
 *          hold post-RoPE keys / values in position order.
 *   cache_len: must equal the length the library counted (budget after the
 *          previous eviction plus one per append since), with
 *          budget < cache_len <= max_cache; BKV_ERR_STATE otherwise.
 *   step:  must equal the step of the last bkv_append_queries.
 *   kept:  device int32 [layers][batch][kv_heads][budget]; receives I_final,
 *          ascending slot indices into the pre-eviction cache. With
 *          BKV_FLAG_ORDER_FREE it receives the layout instead: kept[i] is the
 *          pre-eviction slot whose row now sits in slot i (the same set, not
 *          ascending).
 * On completion slots [0, budget) of every unit hold K[kept] / V[kept];
 * slots [budget, cache_len) are left with unspecified contents. Then every
 * query head's beacons become FPS(beacons + recents, fps_keep) and its recent
 * ring is emptied. Units with more than 256 observation rows are scored in
 * row chunks of at most 256 (same result); BKV_ERR_UNSUPPORTED if
 * G * (beacons + recents) > 2048;
 * BKV_ERR_INVALID_ARG with BKV_FLAG_ORDER_FREE if recent > cache_len - budget. */
bkv_status bkv_evict(bkv_handle h, void* const* K, void* const* V, int32_t cache_len,
                     int64_t step, int32_t* kept);

/* Prefill (notes §2.2: at prefill the first representatives are sampled from
 * the input queries). Sets every query head's observation state from the
 * prompt's pre-RoPE queries: the last min(n_rq, P) become the recent queries
 * at their own positions, and the beacons are FPS (Algorithm 1) of the earlier
 * ones, fps_keep of them (all when fewer), in candidate order. The caller
 * writes the prompt's keys and values to cache slots [0, P) itself; when
 * P > budget, bkv_evict(K, V, P, first_step + P - 1, kept) then evicts the
 * prompt down to the budget, and decoding continues with bkv_append_queries
 * at step first_step + P.
 *   q_prompt:   device bf16 [P][layers][batch][heads][d], 16-B aligned.
 *   P:          1 <= P <= max_cache.
 *   first_step: position of the first prompt token, >= 0.
 *   trace_out:  optional device int32 [layers][batch][heads][min(fps_keep, N)]
 *               receiving each head's picks (indices into its N = P - recents
 *               older queries) in pick order; NULL to skip. The int8 trace of
 *               bkv_get_fps_trace is not updated.
 * Needs a handle with no queries appended yet (BKV_ERR_STATE otherwise);
 * BKV_ERR_UNSUPPORTED if P - min(n_rq, P) exceeds what one CTA's shared
 * memory holds (about 20K older queries). */
bkv_status bkv_prefill(bkv_handle h, const void* q_prompt, int32_t P, int64_t first_step,
                       int32_t* trace_out);

/* Future-query coverage (notes §3.2, Figure 6): for every query head and each
 * of n_future pre-RoPE queries, the largest cosine between that query and the
 * head's current observation set - its beacons and recent queries, the rows
 * the next bkv_evict would score. Call it before bkv_evict (which replaces
 * the set) with the queries of the steps that follow. The cosine is the FPS
 * arithmetic: exact dot products rounded once to fp64, IEEE fp64 division and
 * square root, 0 for a zero vector; -inf where a head's set is empty.
 *   q_future: device bf16 [n_future][layers][batch][heads][d], 16-B aligned.
 *   out:      device double [layers][batch][heads][n_future], 8-B aligned.
 * Asynchronous on the handle's stream; BKV_ERR_INVALID_ARG for null or
 * misaligned pointers or n_future < 1. */
bkv_status bkv_coverage(bkv_handle h, const void* q_future, int32_t n_future, double* out);

/* Waits for the handle's stream, then returns and clears the latched device
 * status (BKV_OK when no device error was seen), or BKV_ERR_CUDA. */
bkv_status bkv_sync(bkv_handle h);

/* Copies the pick order of the last FPS call of every query head into host
 * memory: int8 [layers][batch][heads][fps_keep], indices into that call's
 * candidate list (beacons oldest first, then recents oldest first), -1 where
 * fewer than fps_keep candidates existed. Synchronizes the stream.
 * n: bytes available at host_out. */
bkv_status bkv_get_fps_trace(bkv_handle h, int8_t* host_out, size_t n);

/* Copies the last eviction's Score[j] into host memory: fp32
 * [layers][batch][kv_heads][max_cache], entries j >= cache_len unspecified.
 * Needs BKV_FLAG_KEEP_SCORES (BKV_ERR_STATE otherwise). Synchronizes.
 * n: floats available at host_out. */
bkv_status bkv_get_scores(bkv_handle h, float* host_out, size_t n);

/* Copies one query head's current beacons (rows [0, beacons)) and recent
 * ring (slot s holds the query of the step tau with tau % n_rq == s) into
 * host memory: bf16 [fps_cap + n_rq][d]. Synchronizes. Debug and tests. */
bkv_status bkv_get_head_state(bkv_handle h, int32_t layer, int32_t seq, int32_t head,
                              uint16_t* host_out, size_t n);

/* Per-kernel device time, from CUDA events the library records on its stream
 * around each of its launches while profiling is on. Index with BKV_K_*. */
enum { BKV_K_APPEND = 0, BKV_K_ROPE = 1, BKV_K_SCORE = 2 /* score, keep set and compaction */,
       BKV_K_FPS = 3, BKV_K_COVERAGE = 4, BKV_K_PREFILL = 5, BKV_K_COUNT = 6 };
typedef struct bkv_kernel_times {
  double ms[BKV_K_COUNT];          /* summed launch durations, milliseconds */
  uint64_t launches[BKV_K_COUNT];  /* launches summed */
} bkv_kernel_times;

/* enable != 0: start recording (and zero the sums); 0: stop recording.
 * Events come from a host-side pool the handle owns; no device memory. */
bkv_status bkv_profile(bkv_handle h, int32_t enable);

/* Synchronizes the stream and returns the sums since profiling was enabled. */
bkv_status bkv_profile_read(bkv_handle h, bkv_kernel_times* out);

/* Score + keep-set selection of one eviction without a handle or workspace.
 * The BeaconKV paper has no counterpart: this is a deployment variant of the
 * scoring step of bkv_evict for callers that cannot allocate device memory -
 * code running from a fixed, pre-sized memory arena, runtimes that forbid
 * cudaMalloc after start-up because it can synchronize the device, plugins
 * that may only use the buffers their host passes in. It allocates nothing:
 * its one scratch buffer, the RoPE cos/sin table of the eviction step
 * (16,896 bytes), is a file-scope __device__ array that every GPU loading the
 * library holds until the process exits.
 *   cfg:      as bkv_create. BKV_FLAG_MEAN_POOL selects mean pooling as in
 *             bkv_evict; BKV_FLAG_KEEP_SCORES and BKV_FLAG_ORDER_FREE have no
 *             effect (no scores are kept, nothing is compacted).
 *   bq:       device bf16 [layers][batch][heads][fps_cap][d]; rows [0, beacons)
 *             of each query head are its pre-RoPE beacons, oldest first.
 *   rq:       device bf16 [layers][batch][heads][fps_cap - fps_keep][d]; the
 *             recent queries of steps step - recents + 1 .. step, the query of
 *             step tau in slot tau % (fps_cap - fps_keep).
 *   beacons:  0 <= beacons < fps_cap; recents: 0 <= recents <= fps_cap - fps_keep
 *             and at most 32 (BKV_ERR_UNSUPPORTED beyond: the scratch holds
 *             1 + 32 table rows); beacons + recents >= 1.
 *   K, cache_len, step, kept: as bkv_evict, but cache_len is only checked
 *             against budget < cache_len <= max_cache. Nothing else is written:
 *             no compaction, no FPS, no state.
 *   status:   optional device uint32 (4-byte aligned, caller-owned). The call
 *             sets it to 0, then the kernel latches the first device-side
 *             error: BKV_ERR_TIMEOUT (a bounded wait ran out; kept is then
 *             partly unwritten and must not be used), BKV_ERR_NONFINITE (a
 *             score was NaN, e.g. from a non-finite key). NULL: such errors go
 *             unreported, and a timeout cannot be told from success.
 *   cuda_stream: where the work is enqueued.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. The address is kept for later calls, so do not
 * call this entry point on a device after resetting it (cudaDeviceReset).
 * Every call rewrites the whole table before using it; calls whose work
 * overlaps on the GPU share the array and race, so order them. Host checks
 * return BKV_ERR_INVALID_ARG / BKV_ERR_UNSUPPORTED / BKV_ERR_CUDA and
 * enqueue nothing. */
bkv_status bkv_score_select_noalloc(const bkv_config* cfg, const void* bq, const void* rq,
                                    int32_t beacons, int32_t recents, void* const* K,
                                    int32_t cache_len, int64_t step, int32_t* kept,
                                    uint32_t* status, void* cuda_stream);

/* Self-test of the bounded device-side waits every kernel uses (the timeout
 * latch and the abort of the other waiting warps): enqueues on the handle's
 * stream a kernel whose four warps wait up to wait_cycles SM clock cycles
 * (1 .. 2e9; the kernels' own limit is 2e9, about a second) on a barrier that
 * nothing completes. The next bkv_sync then returns BKV_ERR_TIMEOUT and
 * clears it; the stream, the handle and its state stay usable. Nothing else
 * is touched. BKV_ERR_INVALID_ARG for a limit out of range. */
bkv_status bkv_selftest_wait(bkv_handle h, int64_t wait_cycles);

/* Counters and bookkeeping; synchronizes to read the device counter. */
bkv_status bkv_get_stats(bkv_handle h, bkv_stats* out);

/* Frees the handle (not the workspace). Enqueued work must be complete. */
void bkv_destroy(bkv_handle h);

/* Static string naming a status code. */
const char* bkv_status_str(bkv_status s);

#ifdef __cplusplus
}
#endif

#endif /* BKV_H */
