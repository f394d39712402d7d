// Prefill: each query head's initial observation state from the prompt
// (BeaconKV reading notes §2.2: at prefill the first representatives are
// sampled from the input queries). Of the P prompt queries, the last
// nr = min(n_rq, P) go to the recent ring at their own positions and the
// beacons are FPS (Algorithm 1) of the N = P - nr older ones, keeping
// m = min(fps_keep, N). One CTA per head: 512 threads with the candidates'
// rows resident in shared memory when they fit (N up to ~750), else 128
// threads reading them from global memory on every pass.
//
// FPS over N candidates (up to thousands) in O(N d m) instead of the O(N^2 d)
// of a Gram matrix:
//   * every candidate becomes a float32 unit vector u_j = (x_j 2^s_j) / ||.||
//     (power-of-two scaling as in the FPS kernel, then rsqrtf); each warp
//     takes one candidate at a time, lane l holding dimensions 4l..4l+3;
//   * the mean cosine a_i = (1/N) sum_j cos(x_i, x_j) = u_i . mbar with
//     mbar = (1/N) sum_j u_j, each lane's share summed in float32 with a
//     compensation term (Kahan), the warps' partials merged in float64, then
//     rounded to float32 (the compensated sum errs by <= 2^-23 sum |u_jk|,
//     i.e. < 3e-8 per component after the division by N, < 3.4e-7 on a_i);
//   * every pick round refreshes S_j = max(S_j, u_j . u_r) in one pass.
// With the rows resident, each row is stored once more as y_j = x_j 2^s_j in
// bf16 (exact: a power-of-two scaling, apart from components more than ~126
// binades below the row's largest, which round in the bf16 subnormal range,
// < 2^-126 each against a largest component >= 1), and the passes give each
// thread whole candidates: c_j = (y_j . v) / ||y_j|| with the float32 dot in
// four partial sums of 32 products (gamma_35 = 2.1e-6 relative to
// ||y_j|| ||v||), so |c32 - cos| <= 4e-6 for v a computed unit vector and
// |a32 - a64| <= 4.5e-6 plus the reference's summation error, within the same
// filter bounds.
// Error bounds (relative to unit vectors, so absolute on cosines): u_j carries
// <= 5.7e-7 per component (norm: 4 FMAs and a 5-level tree, gamma_9; rsqrtf
// 2 ulp; one multiply), a float32 dot adds gamma_9; so |c32 - cos| <= 2e-6 and
// |a32 - a64| <= 2.5e-6 plus the float64 reference's own summation error
// (<= N 2^-53). The filters use kCosErr = 2e-5 and kMeanErr = 2.5e-5: a pick
// is final when the float32 minimum beats every other candidate by twice the
// bound; otherwise the exact float64 values of the close candidates (exact dot
// products rounded once, IEEE division and square root, a_i summed left to
// right) decide, ties to the lowest index.
#include <climits>

#include "bkv_internal.cuh"
#include "exact_dot.cuh"

namespace bkv {

namespace {

constexpr int kMaxWarps = 16;
constexpr int kRowStride = kD * 2 + 16;  // bytes per resident row: 16-byte reads of 8 consecutive rows hit distinct banks
constexpr int kBatch = 8;                // candidates per warp whose row loads are in flight together
constexpr float kCosErr = 2e-5f;
constexpr float kMeanErr = 2.5e-5f;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, off));
  return v;
}

// Shared memory for N candidates.
struct PfSmem {
  float* inv;       // [N] 1 / ||x_j 2^s_j||
  float* S;         // [N] mean cosine, then the running max cosine to the picks
  uint8_t* E;       // [N] largest biased exponent of the row (sets s_j)
  uint8_t* flag;    // [N] bit 0: picked
  double* mpart;    // [warps][kD] per-warp sums of unit vectors
  float* mvec;      // [kD] mean unit vector, float32
  float* up;        // [kD] unit vector of the latest pick
  double* xv;       // [warps][32] exact values, one chunk per warp
  double* bestv;    // [warps]
  int* besti;       // [warps]
  uint32_t* red;    // [warps] reduction scratch
  unsigned char* rows;  // resident: [N][kRowStride] scaled rows, bf16
  int* picks;       // [32]
  int* cntw;        // [warps] close candidates per warp
  int* lastw;       // [warps] the largest of them
};

__host__ __device__ inline size_t pf_smem_bytes(int N, bool resident) {
  size_t b = resident ? (size_t)N * kRowStride : 0;
  b += (size_t)N * 10;
  b = (b + 15) / 16 * 16;
  return b + (size_t)kMaxWarps * kD * 8 + kD * 4 * 2 + kMaxWarps * 32 * 8 + kMaxWarps * 8 + kMaxWarps * 4 +
         kMaxWarps * 4 + 32 * 4 + 2 * kMaxWarps * 4 + 64;
}

__device__ inline PfSmem pf_carve(unsigned char* base, int N, bool resident) {
  PfSmem s;
  size_t off = 0;
  s.rows = base;
  if (resident) off += (size_t)N * kRowStride;
  s.inv = reinterpret_cast<float*>(base + off);
  off += (size_t)N * 4;
  s.S = reinterpret_cast<float*>(base + off);
  off += (size_t)N * 4;
  s.E = base + off;
  off += N;
  s.flag = base + off;
  off += N;
  off = (off + 15) / 16 * 16;
  s.mpart = reinterpret_cast<double*>(base + off);
  off += (size_t)kMaxWarps * kD * 8;
  s.xv = reinterpret_cast<double*>(base + off);
  off += (size_t)kMaxWarps * 32 * 8;
  s.bestv = reinterpret_cast<double*>(base + off);
  off += kMaxWarps * 8;
  s.mvec = reinterpret_cast<float*>(base + off);
  off += kD * 4;
  s.up = reinterpret_cast<float*>(base + off);
  off += kD * 4;
  s.besti = reinterpret_cast<int*>(base + off);
  off += kMaxWarps * 4;
  s.red = reinterpret_cast<uint32_t*>(base + off);
  off += kMaxWarps * 4;
  s.picks = reinterpret_cast<int*>(base + off);
  off += 32 * 4;
  s.cntw = reinterpret_cast<int*>(base + off);
  off += kMaxWarps * 4;
  s.lastw = reinterpret_cast<int*>(base + off);
  return s;
}

// exponent range and wideness of a bf16 row (for the exact dot products)
__device__ void row_meta(const uint4* row, int& emin_out, bool& wide_out) {
  int emin = INT_MAX, emax = INT_MIN;
  for (int k = 0; k < kD; ++k) {
    int sig, e, neg, nf;
    decode_bf16(elem(row, k), sig, e, neg, nf);
    if (sig != 0 && !nf) {
      emin = min(emin, e);
      emax = max(emax, e);
    }
  }
  if (emin == INT_MAX) emin = emax = 0;
  emin_out = emin;
  wide_out = emax - emin > 20;
}

// the float64 cosine of the reference arithmetic; gii = exact G_ii
__device__ double cos64_rows(const uint4* ri, int ei, bool wi, double gii, const uint4* rj) {
  int ej;
  bool wj;
  row_meta(rj, ej, wj);
  const double gjj = exact_dot(rj, rj, ej, ej, wj);
  if (gii == 0.0 || gjj == 0.0) return 0.0;
  const double g = exact_dot(ri, rj, ei, ej, wi || wj);
  return __ddiv_rn(g, __dsqrt_rn(__dmul_rn(gii, gjj)));
}

// The resident variant's per-candidate dot: y_j (scaled bf16 row in shared
// memory) with a float32 vector v, four partial sums of 32 products.
__device__ __forceinline__ float resident_dot(const unsigned char* yrow, const float* v) {
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < kD / 8; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(yrow + c * 16);
    const float4 v0 = *reinterpret_cast<const float4*>(v + 8 * c);
    const float4 v1 = *reinterpret_cast<const float4*>(v + 8 * c + 4);
    a0 = __ffma2_rn(make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u)),
                    make_float2(v0.x, v0.y), a0);
    a1 = __ffma2_rn(make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u)),
                    make_float2(v0.z, v0.w), a1);
    a0 = __ffma2_rn(make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u)),
                    make_float2(v1.x, v1.y), a0);
    a1 = __ffma2_rn(make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u)),
                    make_float2(v1.z, v1.w), a1);
  }
  return __fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y));
}

template <int kThreads, bool kResident>
__global__ void __launch_bounds__(kThreads) prefill_kernel(PrefillParams P) {
  constexpr int kWarps = kThreads / 32;
  static_assert(kWarps <= kMaxWarps, "shared-memory plan");
  extern __shared__ __align__(16) unsigned char pf_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t head = blockIdx.x;
  const int N = P.N, m = P.m;
  PfSmem sm = pf_carve(pf_smem, N, kResident);
  auto row = [&](int j) -> const uint4* { return P.q + ((int64_t)j * P.heads_total + head) * 16; };
  uint4* bq = P.bq + head * P.fps_cap * 16;
  uint4* rq = P.rq + head * P.n_rq * 16;

  // ---- recent ring: prompt query P - nr + k at position first_step + P - nr + k
  for (int idx = tid; idx < P.nr * 16; idx += kThreads) {
    const int k = idx >> 4, part = idx & 15;
    const int64_t tau = P.first_step + P.P - P.nr + k;
    const int slot = (int)(((tau % P.n_rq) + P.n_rq) % P.n_rq);
    rq[slot * 16 + part] = row(P.P - P.nr + k)[part];
  }
  if (N <= 0 || m <= 0) return;  // uniform: no beacons to sample
  if (N <= m) {                   // every older query is kept in order
    for (int idx = tid; idx < N * 16; idx += kThreads) bq[idx] = row(idx >> 4)[idx & 15];
    if (P.trace)
      for (int k = tid; k < m; k += kThreads) P.trace[head * m + k] = k < N ? k : -1;
    return;
  }

  // The lane's 8 bytes (four components) of the rows of candidates j0,
  // j0 + kWarps, ..., issued together: one memory latency per batch.
  auto fetch = [&](int j0, uint2 (&w)[kBatch]) {
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int j = j0 + b * kWarps;
      if (kResident)
        w[b] = j < N ? *reinterpret_cast<const uint2*>(sm.rows + (size_t)j * kRowStride + lane * 8) : make_uint2(0u, 0u);
      else
        w[b] = j < N ? __ldg(reinterpret_cast<const uint2*>(row(j)) + lane) : make_uint2(0u, 0u);
    }
  };
  // lane's four components of a row as float32 (the bf16 values), and their largest biased exponent
  auto split4 = [&](uint2 w, float (&y)[4], uint32_t& emax) {
    const uint32_t h[4] = {w.x & 0xFFFFu, w.x >> 16, w.y & 0xFFFFu, w.y >> 16};
    emax = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      emax = max(emax, (h[i] >> 7) & 0xFFu);
      y[i] = __uint_as_float(h[i] << 16);
    }
  };
  // unit vector components of candidate j from its fetched bytes
  auto unit4 = [&](int j, uint2 w, float (&u)[4]) {
    float y[4];
    uint32_t e;
    split4(w, y, e);
    const float scale = __int_as_float(max(254 - (int)sm.E[j], 1) << 23);
    const float iv = sm.inv[j];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __fmul_rn(__fmul_rn(y[i], scale), iv);
  };

  if (kResident) {
    // ---- phase 0: the candidates' rows into shared memory, 8 loads in flight per thread
    for (int i0 = tid; i0 < N * 16; i0 += kThreads * 8) {
      uint4 v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int i = i0 + b * kThreads;
        if (i < N * 16) v[b] = __ldg(row(i >> 4) + (i & 15));
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int i = i0 + b * kThreads;
        if (i < N * 16) *reinterpret_cast<uint4*>(sm.rows + (size_t)(i >> 4) * kRowStride + (i & 15) * 16) = v[b];
      }
    }
    __syncthreads();
  }

  // ---- phase A: scaling, norms, flags, sum of unit vectors (resident rows
  // are rewritten scaled by 2^s_j)
  // compensated float32 sums (Kahan): float64 adds are scarce on this part
  float msum[4] = {0.f, 0.f, 0.f, 0.f}, mcomp[4] = {0.f, 0.f, 0.f, 0.f};
  bool bad = false;
  for (int j0 = warp; j0 < N; j0 += kWarps * kBatch) {
    uint2 wb[kBatch];
    fetch(j0, wb);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int j = j0 + b * kWarps;
      if (j >= N) break;  // uniform across the warp
      float y[4];
      uint32_t e;
      split4(wb[b], y, e);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) e = max(e, __shfl_xor_sync(kFull, e, off));
      bad |= e == 0xFFu;
      const float scale = __int_as_float(max(254 - (int)e, 1) << 23);
#pragma unroll
      for (int i = 0; i < 4; ++i) y[i] = __fmul_rn(y[i], scale);
      if (kResident) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]), hi = __floats2bfloat162_rn(y[2], y[3]);
        *reinterpret_cast<uint2*>(sm.rows + (size_t)j * kRowStride + lane * 8) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
      }
      float n2 = __fmul_rn(y[0], y[0]);
      n2 = __fmaf_rn(y[1], y[1], n2);
      n2 = __fmaf_rn(y[2], y[2], n2);
      n2 = __fmaf_rn(y[3], y[3], n2);
      n2 = warp_sum(n2);
      const float iv = n2 > 0.f ? rsqrtf(n2) : 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x = __fsub_rn(__fmul_rn(y[i], iv), mcomp[i]);
        const float t = __fadd_rn(msum[i], x);
        mcomp[i] = __fsub_rn(__fsub_rn(t, msum[i]), x);
        msum[i] = t;
      }
      if (lane == 0) {
        sm.inv[j] = iv;
        sm.E[j] = (uint8_t)e;
        sm.flag[j] = 0;
      }
    }
  }
  if (__syncthreads_or(bad) && tid == 0) latch(P.status, BKV_ERR_NONFINITE);
#pragma unroll
  for (int i = 0; i < 4; ++i) sm.mpart[warp * kD + 4 * lane + i] = (double)msum[i] - (double)mcomp[i];
  __syncthreads();
  if (tid < kD) {
    double s = 0.0;
    for (int w = 0; w < kWarps; ++w) s = __dadd_rn(s, sm.mpart[w * kD + tid]);
    sm.mvec[tid] = __double2float_rn(__ddiv_rn(s, (double)N));
  }
  __syncthreads();

  // ---- phase B: mean cosines a_j = u_j . mbar
  if (kResident) {
    for (int j = tid; j < N; j += kThreads)
      sm.S[j] = __fmul_rn(resident_dot(sm.rows + (size_t)j * kRowStride, sm.mvec), sm.inv[j]);
  } else {
    for (int j0 = warp; j0 < N; j0 += kWarps * kBatch) {
      uint2 wb[kBatch];
      fetch(j0, wb);
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int j = j0 + b * kWarps;
        if (j >= N) break;
        float u[4];
        unit4(j, wb[b], u);
        float a = __fmul_rn(u[0], sm.mvec[4 * lane]);
#pragma unroll
        for (int i = 1; i < 4; ++i) a = __fmaf_rn(u[i], sm.mvec[4 * lane + i], a);
        a = warp_sum(a);
        if (lane == 0) sm.S[j] = a;
      }
    }
  }
  __syncthreads();

  // ---- filtered argmin over the unpicked candidates; exact values decide close calls
  // kind 0: mean cosine of candidate i; kind 1: running max cosine over picks[0, k)
  auto choose = [&](float err, int kind, int k) -> int {
    uint32_t key = 0xFFFFFFFFu;
    for (int j = tid; j < N; j += kThreads)
      if (!(sm.flag[j] & 1)) key = min(key, fkey(sm.S[j]));
    key = __reduce_min_sync(kFull, key);
    if (lane == 0) sm.red[warp] = key;
    __syncthreads();
    uint32_t all = sm.red[0];
    for (int w = 1; w < kWarps; ++w) all = min(all, sm.red[w]);
    const float lim = unkey(all) + 2.0f * err;
    // close candidates: each warp publishes its count and its largest one,
    // so one barrier gives every thread the total (and, if it is 1, the pick)
    int cnt = 0, last = -1;
    for (int j = tid; j < N; j += kThreads)
      if (!(sm.flag[j] & 1) && sm.S[j] <= lim) {
        ++cnt;
        last = j;
      }
    const int wcnt = (int)__reduce_add_sync(kFull, (uint32_t)cnt);
    const int wlast = __reduce_max_sync(kFull, last);
    if (lane == 0) {
      sm.cntw[warp] = wcnt;
      sm.lastw[warp] = wlast;
    }
    __syncthreads();
    int total = 0, only = -1;
    for (int w = 0; w < kWarps; ++w) {
      total += sm.cntw[w];
      if (sm.cntw[w] == 1) only = sm.lastw[w];
    }
    int pick;
    if (total == 1) {
      pick = only;
    } else {
      // each warp evaluates the close candidates of its residue class exactly
      double bv = 0.0;
      int bi = -1;
      for (int i = warp; i < N; i += kWarps) {
        if ((sm.flag[i] & 1) || !(sm.S[i] <= lim)) continue;  // uniform across the warp
        const uint4* ri = row(i);
        int ei;
        bool wi;
        row_meta(ri, ei, wi);
        const double gii = exact_dot(ri, ri, ei, ei, wi);
        double v;
        if (kind == 0) {
          double acc = 0.0;  // sum_j cos64(i, j), left to right in j
          for (int j0 = 0; j0 < N; j0 += 32) {
            const int j = j0 + lane;
            if (j < N) sm.xv[warp * 32 + lane] = cos64_rows(ri, ei, wi, gii, row(j));
            __syncwarp();
            if (lane == 0)
              for (int q = 0; q < 32 && j0 + q < N; ++q) acc = __dadd_rn(acc, sm.xv[warp * 32 + q]);
            __syncwarp();
          }
          v = __ddiv_rn(__shfl_sync(kFull, acc, 0), (double)N);
        } else {
          double mx = -__longlong_as_double(0x7ff0000000000000LL);
          for (int q = lane; q < k; q += 32) {
            const double c = cos64_rows(ri, ei, wi, gii, row(sm.picks[q]));
            mx = c > mx ? c : mx;
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const double o = __shfl_xor_sync(kFull, mx, off);
            mx = o > mx ? o : mx;
          }
          v = mx;
        }
        if (bi < 0 || v < bv) {  // i ascends within the warp: ties keep the lower index
          bv = v;
          bi = i;
        }
      }
      if (lane == 0) {
        sm.bestv[warp] = bv;
        sm.besti[warp] = bi;
      }
      __syncthreads();
      pick = -1;
      double pv = 0.0;
      for (int w = 0; w < kWarps; ++w) {
        const int i = sm.besti[w];
        if (i < 0) continue;
        const double v = sm.bestv[w];
        if (pick < 0 || v < pv || (v == pv && i < pick)) {
          pick = i;
          pv = v;
        }
      }
      if (pick < 0) pick = 0;  // only with NaN inputs, which are latched
    }
    return pick;
  };

  // ---- Algorithm 1
  for (int k = 0; k < m; ++k) {
    const int r = choose(k == 0 ? kMeanErr : kCosErr, k == 0 ? 0 : 1, k);
    if (tid == 0) {
      sm.picks[k] = r;
      sm.flag[r] |= 1;
    }
    if (warp == 0) {
      float u[4];
      if (kResident) {  // the stored row is already scaled: u = y_r / ||y_r||
        float y[4];
        uint32_t e;
        split4(*reinterpret_cast<const uint2*>(sm.rows + (size_t)r * kRowStride + lane * 8), y, e);
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = __fmul_rn(y[i], sm.inv[r]);
      } else {
        unit4(r, __ldg(reinterpret_cast<const uint2*>(row(r)) + lane), u);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sm.up[4 * lane + i] = u[i];
    }
    __syncthreads();
    if (k + 1 < m && kResident) {
      for (int j = tid; j < N; j += kThreads) {
        const float c = __fmul_rn(resident_dot(sm.rows + (size_t)j * kRowStride, sm.up), sm.inv[j]);
        sm.S[j] = k == 0 ? c : fmaxf(sm.S[j], c);
      }
      __syncthreads();
    } else if (k + 1 < m) {
      for (int j0 = warp; j0 < N; j0 += kWarps * kBatch) {
        uint2 wb[kBatch];
        fetch(j0, wb);
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          const int j = j0 + b * kWarps;
          if (j >= N) break;
          float u[4];
          unit4(j, wb[b], u);
          float c = __fmul_rn(u[0], sm.up[4 * lane]);
#pragma unroll
          for (int i = 1; i < 4; ++i) c = __fmaf_rn(u[i], sm.up[4 * lane + i], c);
          c = warp_sum(c);
          if (lane == 0) sm.S[j] = k == 0 ? c : fmaxf(sm.S[j], c);
        }
      }
      __syncthreads();
    }
  }

  // ---- beacons: the picked rows in candidate order; the trace in pick order
  if (P.trace)
    for (int k = tid; k < m; k += kThreads) P.trace[head * m + k] = sm.picks[k];
  for (int idx = tid; idx < m * 16; idx += kThreads) {
    const int k = idx >> 4;
    // the k-th smallest pick
    int v = 0;
    for (int q = 0; q < m; ++q) {
      int rank = 0;
      for (int q2 = 0; q2 < m; ++q2) rank += sm.picks[q2] < sm.picks[q];
      if (rank == k) v = sm.picks[q];
    }
    bq[idx] = row(v)[idx & 15];
  }
}

}  // namespace

size_t prefill_smem_bytes(int N) { return pf_smem_bytes(N, false); }

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t s) {
  if (p.heads_total <= 0) return cudaSuccess;
  const int n = p.N > 0 ? p.N : 1;
  const size_t cap = 227 * 1024;
  const bool resident = pf_smem_bytes(n, true) <= cap;
  const size_t smem = pf_smem_bytes(n, resident);
  if (smem > cap) return cudaErrorInvalidValue;
  cudaError_t e;
  if (resident) {
    e = cudaFuncSetAttribute(prefill_kernel<512, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<512, true><<<(unsigned)p.heads_total, 512, smem, s>>>(p);
  } else {
    e = cudaFuncSetAttribute(prefill_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_kernel<128, false><<<(unsigned)p.heads_total, 128, smem, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace bkv
