// bkv_score_select_noalloc: the eviction's score + keep-set selection for
// callers that cannot allocate device memory.
//
// Some callers run where no allocator is available or allowed: code that
// executes inside a pre-sized static memory arena, a runtime that forbids
// cudaMalloc after start-up (allocation can synchronize the device and break
// latency guarantees), or a plugin that may only touch the buffers its host
// hands it. Such callers cannot provide the workspace that bkv_create needs.
// This entry point keeps the only scratch the score kernel uses - the table of
// RoPE cosines and sines for the eviction step and the recent positions - in
// a file-scope __device__ array instead, so a call needs nothing but the
// caller's inputs and outputs.
//
// Every GPU that loads the library holds the array (kScratchBytes below) until
// the process exits. All calls on a device share it and each call overwrites
// it completely before use, so nothing has to start zeroed; calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on
// it and must be ordered by the caller. The array's device address is looked
// up once per device and kept; a device reset (cudaDeviceReset) may move it,
// so a process that resets a device must not call this entry point on that
// device again.
//
// Device-side failures (a bounded wait that ran out, a non-finite score) are
// latched into the caller's optional status word, which the call zeroes
// first; without one they go unreported.
#include <mutex>

#include "bkv_internal.cuh"

namespace {

constexpr int kMaxRecents = 32;  // largest recent-query count a call may pass
constexpr int kScratchRows = 1 + kMaxRecents;
constexpr size_t kScratchBytes = (size_t)kScratchRows * bkv::kRopePairs * sizeof(float2);  // 16,896

static __device__ __align__(256) float2 g_rope_scratch[kScratchRows * bkv::kRopePairs];
static_assert(sizeof(g_rope_scratch) == kScratchBytes, "scratch size");

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float2* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once
// per device (host code cannot use the symbol itself as a device pointer).
cudaError_t scratch_for_current_device(float2** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_rope_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float2*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" bkv_status bkv_score_select_noalloc(const bkv_config* c, const void* bq, const void* rq,
                                               int32_t beacons, int32_t recents, void* const* K,
                                               int32_t cache_len, int64_t step, int32_t* kept,
                                               uint32_t* status, void* cuda_stream) {
  if (!c || !bq || !rq || !K || !kept) return BKV_ERR_INVALID_ARG;
  if (c->flags & ~(BKV_FLAG_KEEP_SCORES | BKV_FLAG_ORDER_FREE | BKV_FLAG_MEAN_POOL)) return BKV_ERR_INVALID_ARG;
  if (c->heads <= 0 || c->kv_heads <= 0 || c->heads % c->kv_heads != 0 || c->budget <= 0 ||
      c->prefix < 0 || c->recent < 0 || (int64_t)c->prefix + c->recent > c->budget ||
      c->fps_cap <= 0 || c->fps_keep < 0 || c->fps_keep >= c->fps_cap || c->layers <= 0 ||
      c->batch <= 0 || c->max_cache <= c->budget || !(c->rope_theta > 0.0))
    return BKV_ERR_INVALID_ARG;
  if (c->d != bkv::kD || c->fps_cap > bkv::kMaxFpsCap || c->layers > bkv::kMaxLayers)
    return BKV_ERR_UNSUPPORTED;
  const int n_rq = c->fps_cap - c->fps_keep;
  if (beacons < 0 || beacons >= c->fps_cap || recents < 0 || recents > n_rq || beacons + recents == 0)
    return BKV_ERR_INVALID_ARG;  // no observation row: nothing to score with
  if (recents > kMaxRecents) return BKV_ERR_UNSUPPORTED;  // scratch holds 1 + 32 RoPE rows
  if (!aligned(bq, 16) || !aligned(rq, 16) || !aligned(kept, 4) || !aligned(status, 4)) return BKV_ERR_INVALID_ARG;
  for (int l = 0; l < c->layers; ++l)
    if (!K[l] || !aligned(K[l], 16)) return BKV_ERR_INVALID_ARG;
  if (cache_len <= c->budget || cache_len > c->max_cache || step < recents - 1)
    return BKV_ERR_INVALID_ARG;
  const int64_t units = (int64_t)c->layers * c->batch * c->kv_heads;
  const int group = c->heads / c->kv_heads;
  const int R = group * (beacons + recents);
  if (units > 0x7FFFFFFF || R > bkv::kMaxObsRows || cache_len > 8192 ||
      bkv::score_smem_bytes(R, cache_len, recents, c->budget, 0) > 227 * 1024)
    return BKV_ERR_UNSUPPORTED;

  float2* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return BKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return BKV_ERR_CUDA;

  bkv::RopeParams rp{};
  rp.tab = scratch;
  rp.t = step;
  rp.nr = recents;
  rp.theta = c->rope_theta;
  if (bkv::launch_rope_table(rp, s) != cudaSuccess) return BKV_ERR_CUDA;

  bkv::ScoreParams sp{};
  sp.bq = static_cast<const uint4*>(bq);
  sp.rq = static_cast<const uint4*>(rq);
  sp.rope = scratch;
  if (!bkv::encode_kmaps(sp, K, c->layers, c->batch, c->kv_heads, c->max_cache)) return BKV_ERR_CUDA;
  sp.kept = kept;
  sp.scores = nullptr;
  sp.status = status;  // may be null: device errors then go unreported
  sp.batch = c->batch;
  sp.kv_heads = c->kv_heads;
  sp.group = group;
  sp.fps_cap = c->fps_cap;
  sp.n_rq = n_rq;
  sp.nb = beacons;
  sp.nr = recents;
  sp.ring_first = (int)((((step - recents + 1) % n_rq) + n_rq) % n_rq);
  sp.L = cache_len;
  sp.budget = c->budget;
  sp.prefix = c->prefix;
  sp.recent = c->recent;
  sp.max_cache = c->max_cache;
  sp.units = (int)units;
  sp.compact = 0;  // score and keep set only
  sp.pool_mean = (c->flags & BKV_FLAG_MEAN_POOL) ? 1 : 0;
  if (bkv::launch_score_select(sp, s) != cudaSuccess) return BKV_ERR_CUDA;
  return BKV_OK;
}
