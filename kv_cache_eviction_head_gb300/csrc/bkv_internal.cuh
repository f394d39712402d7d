// Internal declarations shared by the host API and the kernels of libbkv.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bkv.h"

namespace bkv {

constexpr int kD = 128;             // head dimension the kernels implement
constexpr int kMaxLayers = 128;     // per-layer K/V pointers travel in the launch parameters
constexpr int kMaxObsRows = 2048;   // observation rows per unit (G * (beacons + recents)), in chunks of <= 256
constexpr int kMaxFpsCap = 32;      // one warp lane per FPS candidate
constexpr int kRopePairs = kD / 2;

// Device-side error latch: the first error code wins.
__device__ __forceinline__ void latch(uint32_t* status, uint32_t code) {
  if (status) atomicCAS(status, 0u, code);
}

// Bounds-checked build (compiled with -DBKV_CHECKED, libbkv_checked.so): every
// computed slot, row and offset the kernels index with is tested against its
// buffer before use; a failed test latches BKV_ERR_INTERNAL and the access is
// skipped, so a bad index shows up as a status code instead of a fault. In the
// regular build the test compiles away and the condition is not evaluated.
#ifdef BKV_CHECKED
__device__ __forceinline__ bool checked_in_range(bool ok, uint32_t* status) {
  if (!ok) latch(status, BKV_ERR_INTERNAL);
  return ok;
}
#define BKV_IN_RANGE(cond, status) (::bkv::checked_in_range((cond), (status)))
#else
#define BKV_IN_RANGE(cond, status) true
#endif

// ---------------------------------------------------------------------------
// append: push one query per query head into its recent ring
struct AppendParams {
  const uint4* q;           // [heads_total][d] bf16 as 16 uint4 per row
  uint4* bq;                // [heads_total][fps_cap][d]
  uint4* rq;                // [heads_total][n_rq][d]
  int64_t heads_total;
  int fps_cap, n_rq;
  int slot;                 // ring slot of this step (step % n_rq)
  int spill;                // 1: the ring is full; its oldest row moves to bq[nb] first
  int nb;                   // beacons before this push
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);

// RoPE cos/sin table: row 0 is the eviction step t, row 1 + k the k-th oldest recent
struct RopeParams {
  float2* tab;              // [rows][kRopePairs] (cos, sin)
  int64_t t;
  int nr;                   // recent rows; rows = 1 + nr
  double theta;
};
cudaError_t launch_rope_table(const RopeParams& p, cudaStream_t s);

// ---------------------------------------------------------------------------
// farthest-point sampling of every query head's candidate set
struct FpsParams {
  uint4* bq;                // [heads_total][fps_cap][d]; rows [0, nb) are candidates, output too
  const uint4* rq;          // [heads_total][n_rq][d]; nr recents follow the beacons
  int8_t* trace;            // [heads_total][m]
  uint32_t* status;
  int64_t heads_total;
  int fps_cap, n_rq;
  int nb, nr;               // candidates: nb beacons then nr recents (N = nb + nr <= 64)
  int ring_first;           // ring slot of the oldest recent
  int m;                    // rows kept (fps_keep)
};
cudaError_t launch_fps(const FpsParams& p, cudaStream_t s);

// ---------------------------------------------------------------------------
// future-query coverage of each head's observation set (diagnostic)
struct CoverageParams {
  const uint4* bq;        // [heads_total][fps_cap][d]; rows [0, nb) are beacons
  const uint4* rq;        // [heads_total][n_rq][d]; nr recents from ring_first
  const uint4* q_future;  // [n_future][heads_total][d]
  double* out;            // [heads_total][n_future]
  int64_t heads_total;
  int fps_cap, n_rq, nb, nr, ring_first, n_future;
};
cudaError_t launch_coverage(const CoverageParams& p, cudaStream_t s);

// ---------------------------------------------------------------------------
// prefill: initial beacons (FPS over the prompt's older queries) and recent ring
struct PrefillParams {
  const uint4* q;         // [P][heads_total][d] prompt queries, pre-RoPE
  uint4* bq;              // [heads_total][fps_cap][d]
  uint4* rq;              // [heads_total][n_rq][d]
  int32_t* trace;         // optional [heads_total][m] picks in pick order
  uint32_t* status;
  int64_t heads_total;
  int64_t first_step;     // position of prompt query 0
  int P, N, m, nr;        // prompt length, FPS candidates, beacons kept, recents
  int fps_cap, n_rq;
};
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t s);
size_t prefill_smem_bytes(int N);

// ---------------------------------------------------------------------------
// score + keep-set selection: persistent CTAs over the units
struct ScoreParams {
  CUtensorMap kmap[kMaxLayers];  // per layer: K as 2-D [batch*kv_heads*max_cache][d] bf16
  const uint4* bq;          // [layers][batch][heads][fps_cap][d]
  const uint4* rq;          // [layers][batch][heads][n_rq][d]
  const float2* rope;       // [1 + nr][kRopePairs]
  int32_t* kept;            // [units][budget]
  float* scores;            // [units][max_cache] or null
  uint32_t* status;
  int batch, kv_heads, group, fps_cap, n_rq;
  int nb, nr, ring_first;
  int L, budget, prefix, recent, max_cache;
  int units;
  // in-place compaction of the kept rows (null pointers / compact = 0: none)
  __nv_bfloat16* Kc[kMaxLayers];
  __nv_bfloat16* Vc[kMaxLayers];
  unsigned long long* rows_moved;
  int compact;  // 0: score and keep set only; 1: compact in slot order (eq. 8);
                // 2: order-free (holes below the budget filled from the kept tail)
  int pool_mean;  // 1: Score[j] = mean over the observation rows of W[., j] (Table 2)
};
cudaError_t launch_score_select(const ScoreParams& p, cudaStream_t s);
// Four warps wait `limit` cycles on a barrier nothing completes (see bkv_selftest_wait).
cudaError_t launch_wait_selftest(uint32_t* status, long long limit, cudaStream_t s);
// Dynamic shared memory the score kernel needs (huge when the shape does not fit).
size_t score_smem_bytes(int R, int L, int nr, int budget, int compact);
// Fills p.kmap for K[0..layers) (host; no device allocation). False on failure.
bool encode_kmaps(ScoreParams& p, const void* const* K, int layers, int batch, int kv_heads,
                  int max_cache);

}  // namespace bkv
