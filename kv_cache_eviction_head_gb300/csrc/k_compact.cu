// In-place K/V compaction, one CTA per unit (BeaconKV reading notes, §2.3
// eq. 8: K_hat = K[:, I_final, :], V_hat = V[:, I_final, :]).
//
// kept = I_final is strictly increasing with kept[i] >= i, so rows below the
// first evicted slot stay where they are and every later row moves down. The
// CTA walks the destination rows in increasing chunks of kChunk rows: it loads
// the whole chunk's sources into registers, passes a barrier, then stores.
// This is race-free in place:
//   * a chunk's sources are all >= its first destination, so the chunk's own
//     stores can only clobber sources that were already loaded (barrier);
//   * later chunks read slots >= their first destination, beyond every slot
//     an earlier chunk wrote;
//   * the barrier of chunk c + 1 follows every load of chunk c, so no store of
//     chunk c + 1 can overtake a load of chunk c.
#include "bkv_internal.cuh"

namespace bkv {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 64;                         // destination rows per step
constexpr int kVecPerRow = kD * 2 / 16;            // 16 uint4 per bf16 row
constexpr int kPer = kChunk * kVecPerRow / kThreads;  // uint4 per thread per tensor

}  // namespace

__global__ void __launch_bounds__(kThreads) compact_kernel(const __grid_constant__ CompactParams P) {
  __shared__ int first_moved;
  __shared__ int kept_s[kChunk];
  const int tid = threadIdx.x;
  const int u = blockIdx.x;
  const int kvh = u % P.kv_heads;
  const int seq = (u / P.kv_heads) % P.batch;
  const int layer = u / (P.kv_heads * P.batch);
  const size_t base = (size_t)(seq * P.kv_heads + kvh) * P.max_cache * kVecPerRow;
  uint4* K = reinterpret_cast<uint4*>(P.K[layer]) + base;
  uint4* V = reinterpret_cast<uint4*>(P.V[layer]) + base;
  const int32_t* kept = P.kept + (size_t)u * P.budget;

  // The keep set must be strictly increasing slots below L; anything else
  // (for instance a selection that latched an error and wrote nothing) is
  // reported and the unit is left untouched.
  if (tid == 0) first_moved = P.budget;
  __syncthreads();
  bool bad = false;
  for (int i = tid; i < P.budget; i += kThreads) {
    const int k = kept[i];
    bad |= k < i || k >= P.L || (i > 0 && kept[i - 1] >= k);
    if (k != i) atomicMin(&first_moved, i);
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) latch(P.status, BKV_ERR_INTERNAL);
    return;
  }
  const int i0 = first_moved;

  for (int c = i0; c < P.budget; c += kChunk) {
    if (tid < kChunk) kept_s[tid] = c + tid < P.budget ? kept[c + tid] : 0;
    __syncthreads();
    uint4 kv[kPer], vv[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int idx = tid + q * kThreads;
      const int r = idx / kVecPerRow, part = idx % kVecPerRow;
      if (c + r < P.budget) {
        const size_t src = (size_t)kept_s[r] * kVecPerRow + part;
        kv[q] = K[src];
        vv[q] = V[src];
      }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int idx = tid + q * kThreads;
      const int r = idx / kVecPerRow, part = idx % kVecPerRow;
      if (c + r < P.budget) {
        const size_t dst = (size_t)(c + r) * kVecPerRow + part;
        K[dst] = kv[q];
        V[dst] = vv[q];
      }
    }
  }
  if (tid == 0 && P.rows_moved) atomicAdd(P.rows_moved, (unsigned long long)(P.budget - i0));
}

cudaError_t launch_compact(const CompactParams& p, cudaStream_t s) {
  compact_kernel<<<p.units, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
