// Host side of the C ABI declared in include/bkv.h: argument validation, the
// per-handle step bookkeeping, workspace layout and the launch sequence.
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "bkv_internal.cuh"

namespace {

// NVTX range over one API call, named after it, for timeline tools (Nsight
// Systems, ncu --nvtx); without an attached tool a push/pop is a no-op check.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr size_t kAlign = 256;
constexpr size_t kMaxSmem = 227 * 1024;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t status = 0, rows_moved = 0, rope = 0, bq = 0, rq = 0, trace = 0, scores = 0, total = 0;
};

bool mul_ok(size_t a, size_t b, size_t& out) {
  if (a != 0 && b > SIZE_MAX / a) return false;
  out = a * b;
  return true;
}

bkv_status check_config(const bkv_config* c) {
  if (!c) return BKV_ERR_INVALID_ARG;
  if (c->heads <= 0 || c->kv_heads <= 0 || c->heads % c->kv_heads != 0) return BKV_ERR_INVALID_ARG;
  if (c->d <= 0 || c->budget <= 0 || c->period <= 0 || c->prefix < 0 || c->recent < 0)
    return BKV_ERR_INVALID_ARG;
  if ((int64_t)c->prefix + c->recent > c->budget) return BKV_ERR_INVALID_ARG;
  if (c->fps_cap <= 0 || c->fps_keep < 0 || c->fps_keep >= c->fps_cap) return BKV_ERR_INVALID_ARG;
  if (c->layers <= 0 || c->batch <= 0 || c->max_cache <= c->budget) return BKV_ERR_INVALID_ARG;
  if (!(c->rope_theta > 0.0)) return BKV_ERR_INVALID_ARG;
  if (c->flags & ~(BKV_FLAG_KEEP_SCORES | BKV_FLAG_ORDER_FREE | BKV_FLAG_MEAN_POOL)) return BKV_ERR_INVALID_ARG;
  if (c->d != bkv::kD || c->fps_cap > bkv::kMaxFpsCap || c->layers > bkv::kMaxLayers)
    return BKV_ERR_UNSUPPORTED;
  const int64_t units = (int64_t)c->layers * c->batch * c->kv_heads;
  if (units > 0x7FFFFFFF) return BKV_ERR_UNSUPPORTED;  // one CTA per unit in a 1-D grid
  return BKV_OK;
}

bool make_layout(const bkv_config& c, Layout& L) {
  const size_t heads_total = (size_t)c.layers * c.batch * c.heads;
  const size_t units = (size_t)c.layers * c.batch * c.kv_heads;
  const size_t n_rq = (size_t)(c.fps_cap - c.fps_keep);
  const size_t row = (size_t)c.d * 2;
  size_t off = 0, sz;
  L.status = off;
  L.rows_moved = off + 8;
  off += kAlign;
  L.rope = off;
  off += align_up((1 + n_rq) * bkv::kRopePairs * sizeof(float2));
  L.bq = off;
  if (!mul_ok(heads_total, (size_t)c.fps_cap * row, sz)) return false;
  off += align_up(sz);
  L.rq = off;
  if (!mul_ok(heads_total, n_rq * row, sz)) return false;
  off += align_up(sz);
  L.trace = off;
  if (!mul_ok(heads_total, (size_t)c.fps_keep, sz)) return false;
  off += align_up(sz);
  L.scores = off;
  if (c.flags & BKV_FLAG_KEEP_SCORES) {
    if (!mul_ok(units, (size_t)c.max_cache * 4, sz)) return false;
    off += align_up(sz);
  }
  L.total = off;
  return true;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

struct bkv_ctx {
  bkv_config cfg;
  cudaStream_t stream;
  char* ws;
  size_t ws_bytes;
  Layout lay;
  int64_t heads_total, units;
  int group, n_rq;
  int nb = 0, nr = 0;           // beacons and recents per query head
  int64_t last_step = -1;
  int64_t cache_len = 0;        // tracked length of the caller's cache
  uint64_t evictions = 0, fps_calls = 0;

  // profiling: event pairs recorded around launches, folded into sums on read
  struct Mark {
    int kernel;
    cudaEvent_t start, stop;
  };
  bool prof = false;
  std::vector<Mark> marks;
  std::vector<cudaEvent_t> pool;
  double prof_ms[BKV_K_COUNT] = {};
  uint64_t prof_n[BKV_K_COUNT] = {};

  cudaEvent_t take_event() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
  // Runs `launch` between two recorded events when profiling is on.
  template <class F>
  cudaError_t timed(int kernel, cudaStream_t on, F launch) {
    if (!prof) return launch();
    cudaEvent_t a = take_event(), b = take_event();
    if (!a || !b) {  // keep whichever event was made for later use
      if (a) pool.push_back(a);
      if (b) pool.push_back(b);
      return cudaErrorMemoryAllocation;
    }
    cudaEventRecord(a, on);
    const cudaError_t e = launch();
    cudaEventRecord(b, on);
    marks.push_back({kernel, a, b});
    return e;
  }
  template <class F>
  cudaError_t timed(int kernel, F launch) {
    return timed(kernel, stream, launch);
  }
  ~bkv_ctx() {
    for (auto& m : marks) {
      cudaEventDestroy(m.start);
      cudaEventDestroy(m.stop);
    }
    for (auto e : pool) cudaEventDestroy(e);
  }

  uint32_t* status() { return reinterpret_cast<uint32_t*>(ws + lay.status); }
  unsigned long long* rows_moved() { return reinterpret_cast<unsigned long long*>(ws + lay.rows_moved); }
  float2* rope() { return reinterpret_cast<float2*>(ws + lay.rope); }
  uint4* bq() { return reinterpret_cast<uint4*>(ws + lay.bq); }
  uint4* rq() { return reinterpret_cast<uint4*>(ws + lay.rq); }
  int8_t* trace() { return reinterpret_cast<int8_t*>(ws + lay.trace); }
  float* scores() {
    return (cfg.flags & BKV_FLAG_KEEP_SCORES) ? reinterpret_cast<float*>(ws + lay.scores) : nullptr;
  }
  int ring_slot(int64_t step) const { return (int)(((step % n_rq) + n_rq) % n_rq); }
};

static bkv_status launch_fps_all(bkv_handle h, int nb, int nr, int ring_first, cudaStream_t on) {
  bkv::FpsParams f{};
  f.bq = h->bq();
  f.rq = h->rq();
  f.trace = h->trace();
  f.status = h->status();
  f.heads_total = h->heads_total;
  f.fps_cap = h->cfg.fps_cap;
  f.n_rq = h->n_rq;
  f.nb = nb;
  f.nr = nr;
  f.ring_first = ring_first;
  f.m = h->cfg.fps_keep;
  if (h->timed(BKV_K_FPS, on, [&] { return bkv::launch_fps(f, on); }) != cudaSuccess)
    return BKV_ERR_CUDA;
  h->fps_calls++;
  return BKV_OK;
}

extern "C" {

bkv_status bkv_workspace_bytes(const bkv_config* cfg, size_t* bytes) {
  if (!bytes) return BKV_ERR_INVALID_ARG;
  const bkv_status st = check_config(cfg);
  if (st != BKV_OK) return st;
  Layout L;
  if (!make_layout(*cfg, L)) return BKV_ERR_INVALID_ARG;
  *bytes = L.total;
  return BKV_OK;
}

bkv_status bkv_create(const bkv_config* cfg, void* workspace, size_t workspace_bytes,
                      void* cuda_stream, bkv_handle* out) {
  if (!out) return BKV_ERR_INVALID_ARG;
  *out = nullptr;
  const bkv_status st = check_config(cfg);
  if (st != BKV_OK) return st;
  Layout L;
  if (!make_layout(*cfg, L)) return BKV_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, kAlign) || workspace_bytes < L.total) return BKV_ERR_WORKSPACE;
  bkv_ctx* h = new (std::nothrow) bkv_ctx();
  if (!h) return BKV_ERR_INTERNAL;
  h->cfg = *cfg;
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  h->ws = static_cast<char*>(workspace);
  h->ws_bytes = workspace_bytes;
  h->lay = L;
  h->heads_total = (int64_t)cfg->layers * cfg->batch * cfg->heads;
  h->units = (int64_t)cfg->layers * cfg->batch * cfg->kv_heads;
  h->group = cfg->heads / cfg->kv_heads;
  h->n_rq = cfg->fps_cap - cfg->fps_keep;
  if (cudaMemsetAsync(h->ws, 0, L.total, h->stream) != cudaSuccess) {
    delete h;
    return BKV_ERR_CUDA;
  }
  *out = h;
  return BKV_OK;
}

bkv_status bkv_set_stream(bkv_handle h, void* cuda_stream) {
  if (!h) return BKV_ERR_INVALID_ARG;
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  return BKV_OK;
}

bkv_status bkv_append_queries(bkv_handle h, const void* q_pre, int64_t step) {
  NvtxRange nvtx("bkv_append_queries");
  if (!h || !q_pre || !aligned(q_pre, 16) || step < 0) return BKV_ERR_INVALID_ARG;
  if (h->last_step >= 0 && step != h->last_step + 1) return BKV_ERR_STATE;
  if (h->cache_len + 1 > h->cfg.max_cache) return BKV_ERR_STATE;
  const bool spill = h->nr == h->n_rq;
  bkv::AppendParams a{};
  a.q = static_cast<const uint4*>(q_pre);
  a.bq = h->bq();
  a.rq = h->rq();
  a.heads_total = h->heads_total;
  a.fps_cap = h->cfg.fps_cap;
  a.n_rq = h->n_rq;
  a.slot = h->ring_slot(step);
  a.spill = spill ? 1 : 0;
  a.nb = h->nb;
  if (h->timed(BKV_K_APPEND, [&] { return bkv::launch_append(a, h->stream); }) != cudaSuccess)
    return BKV_ERR_CUDA;
  if (spill) h->nb++;
  else h->nr++;
  h->last_step = step;
  h->cache_len++;
  if (h->nb >= h->cfg.fps_cap) {  // eq. 9: compress a full beacon buffer
    const bkv_status st = launch_fps_all(h, h->nb, 0, 0, h->stream);
    if (st != BKV_OK) return st;
    h->nb = h->cfg.fps_keep;
  }
  return BKV_OK;
}

bkv_status bkv_evict(bkv_handle h, void* const* K, void* const* V, int32_t cache_len, int64_t step,
                     int32_t* kept) {
  NvtxRange nvtx("bkv_evict");
  if (!h || !K || !V || !kept || !aligned(kept, 4)) return BKV_ERR_INVALID_ARG;
  const bkv_config& c = h->cfg;
  for (int l = 0; l < c.layers; ++l)
    if (!K[l] || !V[l] || !aligned(K[l], 16) || !aligned(V[l], 16)) return BKV_ERR_INVALID_ARG;
  if (h->last_step < 0 || step != h->last_step) return BKV_ERR_STATE;
  if (cache_len != h->cache_len || cache_len <= c.budget || cache_len > c.max_cache)
    return BKV_ERR_STATE;
  const bool order_free = (c.flags & BKV_FLAG_ORDER_FREE) != 0;
  if (order_free && c.recent > cache_len - c.budget) return BKV_ERR_INVALID_ARG;
  const int compact = order_free ? 2 : 1;
  const int R = h->group * (h->nb + h->nr);
  if (R > bkv::kMaxObsRows || cache_len > 8192) return BKV_ERR_UNSUPPORTED;
  if (bkv::score_smem_bytes(R, cache_len, h->nr, c.budget, compact) > kMaxSmem) return BKV_ERR_UNSUPPORTED;

  const int ring_first = h->ring_slot(step - h->nr + 1);
  bkv::RopeParams rp{};
  rp.tab = h->rope();
  rp.t = step;
  rp.nr = h->nr;
  rp.theta = c.rope_theta;
  if (h->timed(BKV_K_ROPE, [&] { return bkv::launch_rope_table(rp, h->stream); }) != cudaSuccess)
    return BKV_ERR_CUDA;

  bkv::ScoreParams sp{};
  sp.bq = h->bq();
  sp.rq = h->rq();
  sp.rope = h->rope();
  if (!bkv::encode_kmaps(sp, K, c.layers, c.batch, c.kv_heads, c.max_cache)) return BKV_ERR_CUDA;
  sp.kept = kept;
  sp.scores = h->scores();
  sp.status = h->status();
  sp.batch = c.batch;
  sp.kv_heads = c.kv_heads;
  sp.group = h->group;
  sp.fps_cap = c.fps_cap;
  sp.n_rq = h->n_rq;
  sp.nb = h->nb;
  sp.nr = h->nr;
  sp.ring_first = ring_first;
  sp.L = cache_len;
  sp.budget = c.budget;
  sp.prefix = c.prefix;
  sp.recent = c.recent;
  sp.max_cache = c.max_cache;
  sp.units = (int)h->units;
  for (int l = 0; l < c.layers; ++l) {
    sp.Kc[l] = static_cast<__nv_bfloat16*>(K[l]);
    sp.Vc[l] = static_cast<__nv_bfloat16*>(V[l]);
  }
  sp.rows_moved = h->rows_moved();
  sp.compact = compact;
  sp.pool_mean = (c.flags & BKV_FLAG_MEAN_POOL) ? 1 : 0;
  if (h->timed(BKV_K_SCORE, [&] { return bkv::launch_score_select(sp, h->stream); }) != cudaSuccess)
    return BKV_ERR_CUDA;

  // Algorithm 2: the next period starts from FPS(beacons + recents)
  {
    const bkv_status st = launch_fps_all(h, h->nb, h->nr, ring_first, h->stream);
    if (st != BKV_OK) return st;
  }
  const int n = h->nb + h->nr;
  h->nb = n > c.fps_keep ? c.fps_keep : n;
  h->nr = 0;
  h->cache_len = c.budget;
  h->evictions++;
  return BKV_OK;
}

bkv_status bkv_prefill(bkv_handle h, const void* q_prompt, int32_t P, int64_t first_step,
                       int32_t* trace_out) {
  NvtxRange nvtx("bkv_prefill");
  if (!h || !q_prompt || !aligned(q_prompt, 16) || (trace_out && !aligned(trace_out, 4)) || first_step < 0)
    return BKV_ERR_INVALID_ARG;
  const bkv_config& c = h->cfg;
  if (P < 1 || P > c.max_cache) return BKV_ERR_INVALID_ARG;
  if (h->last_step >= 0 || h->nb != 0 || h->nr != 0 || h->cache_len != 0) return BKV_ERR_STATE;
  const int nr = P < h->n_rq ? P : h->n_rq;
  const int N = P - nr;
  const int m = N < c.fps_keep ? N : c.fps_keep;
  if (bkv::prefill_smem_bytes(N > 0 ? N : 1) > kMaxSmem) return BKV_ERR_UNSUPPORTED;
  bkv::PrefillParams p{};
  p.q = static_cast<const uint4*>(q_prompt);
  p.bq = h->bq();
  p.rq = h->rq();
  p.trace = trace_out;
  p.status = h->status();
  p.heads_total = h->heads_total;
  p.first_step = first_step;
  p.P = P;
  p.N = N;
  p.m = m;
  p.nr = nr;
  p.fps_cap = c.fps_cap;
  p.n_rq = h->n_rq;
  if (h->timed(BKV_K_PREFILL, [&] { return bkv::launch_prefill(p, h->stream); }) != cudaSuccess)
    return BKV_ERR_CUDA;
  h->nb = m;
  h->nr = nr;
  h->last_step = first_step + P - 1;
  h->cache_len = P;
  return BKV_OK;
}

bkv_status bkv_coverage(bkv_handle h, const void* q_future, int32_t n_future, double* out) {
  NvtxRange nvtx("bkv_coverage");
  if (!h || !q_future || !out || n_future < 1 || !aligned(q_future, 16) || !aligned(out, 8))
    return BKV_ERR_INVALID_ARG;
  bkv::CoverageParams p{};
  p.bq = h->bq();
  p.rq = h->rq();
  p.q_future = static_cast<const uint4*>(q_future);
  p.out = out;
  p.heads_total = h->heads_total;
  p.fps_cap = h->cfg.fps_cap;
  p.n_rq = h->n_rq;
  p.nb = h->nb;
  p.nr = h->nr;
  p.ring_first = h->nr > 0 ? h->ring_slot(h->last_step - h->nr + 1) : 0;
  p.n_future = n_future;
  if (h->timed(BKV_K_COVERAGE, [&] { return bkv::launch_coverage(p, h->stream); }) != cudaSuccess)
    return BKV_ERR_CUDA;
  return BKV_OK;
}

bkv_status bkv_selftest_wait(bkv_handle h, int64_t wait_cycles) {
  NvtxRange nvtx("bkv_selftest_wait");
  if (!h || wait_cycles < 1 || wait_cycles > 2000000000LL) return BKV_ERR_INVALID_ARG;
  if (bkv::launch_wait_selftest(h->status(), (long long)wait_cycles, h->stream) != cudaSuccess)
    return BKV_ERR_CUDA;
  return BKV_OK;
}

bkv_status bkv_sync(bkv_handle h) {
  NvtxRange nvtx("bkv_sync");
  if (!h) return BKV_ERR_INVALID_ARG;
  uint32_t code = 0;
  if (cudaMemcpyAsync(&code, h->status(), sizeof(code), cudaMemcpyDeviceToHost, h->stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(h->stream) != cudaSuccess)
    return BKV_ERR_CUDA;
  if (code != 0) {
    if (cudaMemsetAsync(h->status(), 0, sizeof(uint32_t), h->stream) != cudaSuccess ||
        cudaStreamSynchronize(h->stream) != cudaSuccess)
      return BKV_ERR_CUDA;
    return static_cast<bkv_status>(code);
  }
  return BKV_OK;
}

bkv_status bkv_get_fps_trace(bkv_handle h, int8_t* host_out, size_t n) {
  if (!h || !host_out) return BKV_ERR_INVALID_ARG;
  const size_t need = (size_t)h->heads_total * h->cfg.fps_keep;
  if (n < need) return BKV_ERR_INVALID_ARG;
  if (need == 0) return BKV_OK;
  if (cudaMemcpyAsync(host_out, h->trace(), need, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess ||
      cudaStreamSynchronize(h->stream) != cudaSuccess)
    return BKV_ERR_CUDA;
  return BKV_OK;
}

bkv_status bkv_get_scores(bkv_handle h, float* host_out, size_t n) {
  if (!h || !host_out) return BKV_ERR_INVALID_ARG;
  if (!(h->cfg.flags & BKV_FLAG_KEEP_SCORES)) return BKV_ERR_STATE;
  const size_t need = (size_t)h->units * h->cfg.max_cache;
  if (n < need) return BKV_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(host_out, h->scores(), need * 4, cudaMemcpyDeviceToHost, h->stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(h->stream) != cudaSuccess)
    return BKV_ERR_CUDA;
  return BKV_OK;
}

bkv_status bkv_get_head_state(bkv_handle h, int32_t layer, int32_t seq, int32_t head,
                              uint16_t* host_out, size_t n) {
  if (!h || !host_out) return BKV_ERR_INVALID_ARG;
  const bkv_config& c = h->cfg;
  if (layer < 0 || layer >= c.layers || seq < 0 || seq >= c.batch || head < 0 || head >= c.heads)
    return BKV_ERR_INVALID_ARG;
  const size_t rows = (size_t)c.fps_cap + h->n_rq;
  if (n < rows * c.d) return BKV_ERR_INVALID_ARG;
  const int64_t hid = ((int64_t)layer * c.batch + seq) * c.heads + head;
  const size_t rb = (size_t)c.d * 2;
  if (cudaMemcpyAsync(host_out, h->bq() + hid * c.fps_cap * 16, c.fps_cap * rb,
                      cudaMemcpyDeviceToHost, h->stream) != cudaSuccess ||
      cudaMemcpyAsync(host_out + (size_t)c.fps_cap * c.d, h->rq() + hid * h->n_rq * 16,
                      h->n_rq * rb, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess ||
      cudaStreamSynchronize(h->stream) != cudaSuccess)
    return BKV_ERR_CUDA;
  return BKV_OK;
}

bkv_status bkv_get_stats(bkv_handle h, bkv_stats* out) {
  if (!h || !out) return BKV_ERR_INVALID_ARG;
  unsigned long long moved = 0;
  if (cudaMemcpyAsync(&moved, h->rows_moved(), sizeof(moved), cudaMemcpyDeviceToHost, h->stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(h->stream) != cudaSuccess)
    return BKV_ERR_CUDA;
  out->evictions = h->evictions;
  out->fps_calls = h->fps_calls;
  out->rows_moved = moved;
  out->beacons = h->nb;
  out->recents = h->nr;
  out->cache_len = (int32_t)h->cache_len;
  out->last_step = h->last_step;
  return BKV_OK;
}

bkv_status bkv_profile(bkv_handle h, int32_t enable) {
  if (!h) return BKV_ERR_INVALID_ARG;
  if (enable) {
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return BKV_ERR_CUDA;
    for (auto& m : h->marks) {
      h->pool.push_back(m.start);
      h->pool.push_back(m.stop);
    }
    h->marks.clear();
    for (int k = 0; k < BKV_K_COUNT; ++k) {
      h->prof_ms[k] = 0.0;
      h->prof_n[k] = 0;
    }
  }
  h->prof = enable != 0;
  return BKV_OK;
}

bkv_status bkv_profile_read(bkv_handle h, bkv_kernel_times* out) {
  if (!h || !out) return BKV_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return BKV_ERR_CUDA;
  for (auto& m : h->marks) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, m.start, m.stop) != cudaSuccess) return BKV_ERR_CUDA;
    h->prof_ms[m.kernel] += ms;
    h->prof_n[m.kernel] += 1;
    h->pool.push_back(m.start);
    h->pool.push_back(m.stop);
  }
  h->marks.clear();
  for (int k = 0; k < BKV_K_COUNT; ++k) {
    out->ms[k] = h->prof_ms[k];
    out->launches[k] = h->prof_n[k];
  }
  return BKV_OK;
}

void bkv_destroy(bkv_handle h) { delete h; }

const char* bkv_status_str(bkv_status s) {
  switch (s) {
    case BKV_OK: return "BKV_OK";
    case BKV_ERR_INVALID_ARG: return "BKV_ERR_INVALID_ARG";
    case BKV_ERR_STATE: return "BKV_ERR_STATE";
    case BKV_ERR_WORKSPACE: return "BKV_ERR_WORKSPACE";
    case BKV_ERR_CUDA: return "BKV_ERR_CUDA";
    case BKV_ERR_NONFINITE: return "BKV_ERR_NONFINITE";
    case BKV_ERR_TIMEOUT: return "BKV_ERR_TIMEOUT";
    case BKV_ERR_UNSUPPORTED: return "BKV_ERR_UNSUPPORTED";
    case BKV_ERR_INTERNAL: return "BKV_ERR_INTERNAL";
  }
  return "BKV_ERR_UNKNOWN";
}

}  // extern "C"
