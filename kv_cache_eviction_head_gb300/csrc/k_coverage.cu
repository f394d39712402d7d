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
//
// The float64 division and square root run only where they can decide the
// maximum: each pair first gets c32 = float(acc) phi_f phi_o with the row
// factors phi_r = 2^emin_r / sqrt(G_rr) rounded to float32, within
// 5 x 2^-24 (< 3.1e-7 with the float64 value's own rounding) of the exact
// cosine. A lane keeps its two largest c32; if the runner-up is more than
// 2 kCovErr below, the float64 cosine of the leader alone is the maximum,
// otherwise every pair's float64 cosine is computed. Pairs with a wide row
// are always computed in float64.
#include <cmath>

#include "bkv_internal.cuh"
#include "exact_dot.cuh"

namespace bkv {

namespace {

constexpr int kObsMax = 64;     // beacons (< fps_cap <= 32) + recents (<= 32)
constexpr int kFutChunk = 32;   // future queries per warp, one per lane
constexpr float kCovErr = 1e-6f;  // |c32 - cos64| bound used by the filter

// Shared memory for n observation rows.
struct CovSmem {
  int (*v_fut)[kFutChunk];  // [kD][32] decoded future rows, transposed (lane-contiguous reads)
  int (*v_obs)[kD];         // [n][kD] decoded observation rows (row-major: broadcast reads)
  double* g_obs;            // [n] exact G_oo
  float* phi_obs;           // [n] 2^emin / sqrt(G_oo) in float32 (0 for a zero row)
  int* emin_obs;            // [n]
  int* wide_obs;            // [n]
};

__host__ __device__ inline size_t cov_smem_bytes(int n) {
  return (size_t)kD * kFutChunk * 4 + (size_t)n * (kD * 4 + 8 + 4 + 4 + 4) + 16;
}

__device__ inline CovSmem cov_carve(unsigned char* base, int n) {
  CovSmem s;
  size_t off = 0;
  s.v_fut = reinterpret_cast<int(*)[kFutChunk]>(base + off);
  off += (size_t)kD * kFutChunk * 4;
  s.v_obs = reinterpret_cast<int(*)[kD]>(base + off);
  off += (size_t)n * kD * 4;
  s.g_obs = reinterpret_cast<double*>(base + off);
  off += (size_t)n * 8;
  s.phi_obs = reinterpret_cast<float*>(base + off);
  off += (size_t)n * 4;
  s.emin_obs = reinterpret_cast<int*>(base + off);
  off += (size_t)n * 4;
  s.wide_obs = reinterpret_cast<int*>(base + off);
  return s;
}

// float32 factor 2^emin / sqrt(G) of a non-wide row (0 for a zero row)
__device__ __forceinline__ float row_phi(int emin, double g) {
  return g == 0.0 ? 0.f : __double2float_rn(__ddiv_rn(pow2(emin), __dsqrt_rn(g)));
}

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
  const int lane = threadIdx.x;
  const int64_t head = blockIdx.x;
  const int f0 = blockIdx.y * kFutChunk, f = f0 + lane;
  const int nb = P.nb, n = P.nb + P.nr;
  CovSmem sm = cov_carve(cov_smem, n);
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
    sm.phi_obs[r] = w ? 0.f : row_phi(e, g);
  }
  const bool live = f < P.n_future;
  const uint4* frow = P.q_future + ((int64_t)(live ? f : 0) * P.heads_total + head) * 16;
  int emin_f = 0, wide_f = 0;
  double g_f = 0.0;
  decode_row(frow, emin_f, wide_f, g_f, [&](int k, int x) { sm.v_fut[k][lane] = x; });
  const float phi_f = wide_f ? 0.f : row_phi(emin_f, g_f);
  __syncwarp();

  auto int_dot = [&](int o) -> long long {
    long long acc = 0;
#pragma unroll 8
    for (int k = 0; k < kD; ++k) acc += (long long)sm.v_obs[o][k] * sm.v_fut[k][lane];
    return acc;
  };
  // the float64 cosine of the reference arithmetic; acc is the integer dot when neither row is wide
  auto cos64 = [&](int o, long long acc) -> double {
    double g;
    if (!wide_f && !sm.wide_obs[o])
      g = acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(emin_f + sm.emin_obs[o]));
    else
      g = exact_dot_wide(frow, obs_row(o));
    const double goo = sm.g_obs[o];
    return (g_f == 0.0 || goo == 0.0) ? 0.0 : __ddiv_rn(g, __dsqrt_rn(__dmul_rn(g_f, goo)));
  };

  // pass over the rows: float32 cosines, their two largest, float64 for wide pairs
  const float neg_inf32 = __int_as_float(0xff800000u);
  float m1 = neg_inf32, m2 = neg_inf32;
  int o1 = -1;
  double best = -INFINITY;
  for (int o = 0; o < n; ++o) {
    if (!wide_f && !sm.wide_obs[o]) {
      const float c = __fmul_rn(__fmul_rn(__ll2float_rn(int_dot(o)), phi_f), sm.phi_obs[o]);
      if (o1 < 0 || c > m1) {
        m2 = m1;
        m1 = c;
        o1 = o;
      } else if (c > m2) {
        m2 = c;
      }
    } else {
      const double c = cos64(o, 0);
      best = c > best ? c : best;
    }
  }
  if (o1 >= 0) {
    if (m2 >= m1 - 2.0f * kCovErr) {
      // close call: every pair in float64
      for (int o = 0; o < n; ++o) {
        if (wide_f || sm.wide_obs[o]) continue;
        const double c = cos64(o, int_dot(o));
        best = c > best ? c : best;
      }
    } else {
      const double c = cos64(o1, int_dot(o1));
      best = c > best ? c : best;
    }
  }
  if (live) P.out[head * P.n_future + f] = best;
}

}  // namespace

cudaError_t launch_coverage(const CoverageParams& p, cudaStream_t s) {
  if (p.heads_total <= 0 || p.n_future <= 0) return cudaSuccess;
  const int n = p.nb + p.nr;
  if (n > kObsMax) return cudaErrorInvalidValue;
  const size_t smem = cov_smem_bytes(n);
  static_assert(kD * kFutChunk * 4 + kObsMax * (kD * 4 + 20) + 16 <= 227 * 1024, "coverage shared memory");
  cudaError_t e = cudaFuncSetAttribute(coverage_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)cov_smem_bytes(kObsMax));
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)p.heads_total, (unsigned)((p.n_future + kFutChunk - 1) / kFutChunk));
  coverage_kernel<<<grid, 32, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
