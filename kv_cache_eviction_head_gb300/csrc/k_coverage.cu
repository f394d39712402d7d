// Future-query coverage of the observation set (BeaconKV reading notes §3.2,
// Figure 6): for a query head and each of N future pre-RoPE queries q, the
// largest cosine between q and any row of the head's current observation set
// (its beacons, then its recent queries - what the next eviction scores).
// The cosine is FPS's exact arithmetic: G = the exact dot product rounded once
// to float64, cos = G_qo / sqrt(G_qq G_oo) in IEEE float64, 0 for a zero
// vector; an empty set gives -inf. One warp per (head, 32 future queries).
//
// Dot products of rows whose exponents span <= 20 binades run on pre-decoded
// integers: row r is stored as v_rk = (-1)^s sig_k 2^(e_k - emin_r) (< 2^28 in
// magnitude), so sum_k v_ok v_fk is exact in 64 bits (128 products < 2^56)
// and the float64 value is that integer rounded once and scaled by
// 2^(emin_o + emin_f). Wider rows take the 544-bit accumulator.
#include <cmath>

#include "bkv_internal.cuh"
#include "exact_dot.cuh"

namespace bkv {

namespace {

constexpr int kObsMax = 64;   // beacons (< fps_cap <= 32) + recents (<= 32)
constexpr int kFutChunk = 32;  // future queries per warp, one per lane

struct CovSmem {
  int v_obs[kObsMax][kD];       // decoded observation rows (row-major: broadcast reads)
  int v_fut[kD][kFutChunk];     // decoded future rows, transposed (lane-contiguous reads)
  double g_obs[kObsMax];        // exact G_oo
  int emin_obs[kObsMax];
  int wide_obs[kObsMax];
};

// Decodes one bf16 row into scaled integers; returns emin, sets wide and the
// exact squared norm. v(k) receives the k-th value.
template <class Store>
__device__ void decode_row(const uint4* row, int& emin_out, int& wide_out, double& g_out, Store v) {
  int emin = 0x7FFFFFFF, emax = -0x7FFFFFFF;
  for (int k = 0; k < kD; ++k) {
    int sig, e, neg, nf;
    decode_bf16(elem(row, k), sig, e, neg, nf);
    if (sig != 0 && !nf) {
      emin = min(emin, e);
      emax = max(emax, e);
    }
  }
  if (emin == 0x7FFFFFFF) emin = emax = 0;
  const bool wide = emax - emin > 20;
  long long acc = 0;
  for (int k = 0; k < kD; ++k) {
    int sig, e, neg, nf;
    decode_bf16(elem(row, k), sig, e, neg, nf);
    int x = 0;
    if (!wide && sig != 0 && !nf) x = sig << (e - emin);
    x = neg ? -x : x;
    v(k, x);
    acc += (long long)x * x;
  }
  emin_out = emin;
  wide_out = wide;
  g_out = wide ? exact_dot_wide(row, row) : (acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(2 * emin)));
}

__global__ void __launch_bounds__(32) coverage_kernel(CoverageParams P) {
  extern __shared__ __align__(16) unsigned char cov_smem[];
  CovSmem& sm = *reinterpret_cast<CovSmem*>(cov_smem);
  const int lane = threadIdx.x;
  const int64_t head = blockIdx.x;
  const int f0 = blockIdx.y * kFutChunk, f = f0 + lane;
  const int nb = P.nb, n = P.nb + P.nr;
  const uint4* bq = P.bq + head * P.fps_cap * 16;
  const uint4* rq = P.rq + head * P.n_rq * 16;
  auto obs_row = [&](int i) -> const uint4* {
    return i < nb ? bq + i * 16 : rq + ((P.ring_first + i - nb) % P.n_rq) * 16;
  };
  for (int r = lane; r < n; r += 32) {
    int e, w;
    double g;
    decode_row(obs_row(r), e, w, g, [&](int k, int x) { sm.v_obs[r][k] = x; });
    sm.emin_obs[r] = e;
    sm.wide_obs[r] = w;
    sm.g_obs[r] = g;
  }
  const bool live = f < P.n_future;
  const uint4* frow = P.q_future + ((int64_t)(live ? f : 0) * P.heads_total + head) * 16;
  int emin_f = 0, wide_f = 0;
  double g_f = 0.0;
  decode_row(frow, emin_f, wide_f, g_f, [&](int k, int x) { sm.v_fut[k][lane] = x; });
  __syncwarp();

  double best = -INFINITY;
  for (int o = 0; o < n; ++o) {
    double g;
    if (!wide_f && !sm.wide_obs[o]) {
      long long acc = 0;
#pragma unroll 8
      for (int k = 0; k < kD; ++k) acc += (long long)sm.v_obs[o][k] * sm.v_fut[k][lane];
      g = acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(emin_f + sm.emin_obs[o]));
    } else {
      g = exact_dot_wide(frow, obs_row(o));
    }
    const double goo = sm.g_obs[o];
    const double c = (g_f == 0.0 || goo == 0.0) ? 0.0 : __ddiv_rn(g, __dsqrt_rn(__dmul_rn(g_f, goo)));
    best = c > best ? c : best;
  }
  if (live) P.out[head * P.n_future + f] = best;
}

}  // namespace

size_t coverage_smem_bytes() { return sizeof(CovSmem); }

cudaError_t launch_coverage(const CoverageParams& p, cudaStream_t s) {
  if (p.heads_total <= 0 || p.n_future <= 0) return cudaSuccess;
  if (p.nb + p.nr > kObsMax) return cudaErrorInvalidValue;
  static_assert(sizeof(CovSmem) <= 227 * 1024, "coverage shared memory");
  cudaError_t e = cudaFuncSetAttribute(coverage_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sizeof(CovSmem));
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)p.heads_total, (unsigned)((p.n_future + kFutChunk - 1) / kFutChunk));
  coverage_kernel<<<grid, 32, sizeof(CovSmem), s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
