// Farthest-point sampling of pre-RoPE queries, one CTA per query head.
//
// BeaconKV reading notes, §2.2, Algorithm 1 (and eq. 9 / Algorithm 2 for when
// it runs): with cos the cosine similarity of two candidates,
//   a_i = (1/N) sum_j cos(q_i, q_j),  p = argmin_i a_i,  I = {p},  S_j = cos(q_j, q_p);
//   repeat r = argmin_{j not in I} S_j,  I += {r},  S_j = max(S_j, cos(q_j, q_r))
// until |I| = m. Ties go to the lowest index. The kept rows are written back
// in candidate order (oldest first) and the pick order is the trace.
//
// The reference arithmetic is float64: G_ij is the exact dot product of the
// two bf16 vectors rounded once to float64, cos_ij = G_ij / sqrt(G_ii G_jj)
// with IEEE float64 multiply, square root and divide (0 if either vector is
// zero), a_i is summed left to right in j order and then divided by N. Every
// pick this kernel makes is the pick that arithmetic makes, bit for bit, but
// float64 runs only where it can change the answer:
//   * the Gram matrix is first formed in float32 from the bf16 rows scaled by a
//     power of two (exact), with four interleaved partial sums; products of
//     bf16 values are exact in float32, so the Gram error is at most
//     gamma_33 * ||x_i|| ||x_j|| (plus < 2^-142 from products that underflow)
//     and the float32 cosine c_ij is within kCosErr = 2e-5 of the float64
//     cosine (the derived bound is 4.7e-6);
//   * a decision (argmin of the mean cosine, argmin of the running max) is
//     final when the float32 minimum beats every other candidate by more than
//     twice its error bound - then the float64 values order the same way;
//   * otherwise the float64 values of the close candidates are computed
//     exactly as defined above and compared, ties going to the lowest index.
// The exact G_ij uses 64-bit integer arithmetic on the bf16 significands when
// both vectors' exponents span <= 20 binades (128 products then sum below
// 2^63), otherwise a 544-bit fixed-point accumulator over the whole bf16
// product range; either way it is rounded once to nearest even.
#include <climits>

#include "bkv_internal.cuh"

namespace bkv {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxCand = 64;          // beacons (< fps_cap <= 32) + recents (<= 32)
constexpr int kYStride = kD + 4;      // float row stride (528 B): LDS.128 rows hit distinct banks
constexpr float kCosErr = 2e-5f;      // |c32 - cos64| bound used by the filters
constexpr float kMeanErr = 2.5e-5f;   // |a32 - a64| bound (kCosErr + summation error, N <= 64)

// Dynamic shared memory for n candidates.
struct FpsSmem {
  uint4* x;        // [n][16]   bf16 rows
  float* y;        // [n][kYStride] rows scaled by 2^-(emax+8), exact in float32
  float* c;        // [n][n+1]  float32 cosines
  double* diag;    // [n]       exact G_ii rounded to float64
  int* emin;       // [n]       smallest exponent of a nonzero component
  int* emax;       // [n]
  int* flags;      // [n]       bit 0: wide (exponent span > 20), bit 1: y not exact
  int* picks;      // [32]      pick order
  int* keep_src;   // [32]
  int* cand;       // [kMaxCand] fallback candidate list
  double* v64;     // [kMaxCand] fallback values
  int n;
  __device__ float& Y(int i, int k) { return y[i * kYStride + k]; }
  __device__ float& C(int i, int j) { return c[i * (n + 1) + j]; }
};

__host__ __device__ inline size_t fps_smem_bytes(int n) {
  return (size_t)n * 256 + (size_t)n * kYStride * 4 + (((size_t)n * (n + 1) * 4 + 15) / 16) * 16 +
         (size_t)n * 8 + (size_t)n * 12 + 64 * 4 + (size_t)kMaxCand * 4 + (size_t)kMaxCand * 8 + 64;
}

__device__ inline FpsSmem carve(unsigned char* base, int n) {
  FpsSmem s;
  s.n = n;
  size_t off = 0;
  s.x = reinterpret_cast<uint4*>(base);
  off += (size_t)n * 256;
  s.y = reinterpret_cast<float*>(base + off);
  off += (size_t)n * kYStride * 4;
  s.c = reinterpret_cast<float*>(base + off);
  off += (((size_t)n * (n + 1) * 4 + 15) / 16) * 16;
  s.diag = reinterpret_cast<double*>(base + off);
  off += (size_t)n * 8;
  s.v64 = reinterpret_cast<double*>(base + off);
  off += (size_t)kMaxCand * 8;
  s.emin = reinterpret_cast<int*>(base + off);
  s.emax = s.emin + n;
  s.flags = s.emax + n;
  s.picks = s.flags + n;
  s.keep_src = s.picks + 32;
  s.cand = s.keep_src + 32;
  return s;
}

// bf16 = (-1)^neg * sig * 2^exp with an integer significand sig < 256.
__device__ __forceinline__ void decode_bf16(uint32_t bits, int& sig, int& exp, int& neg,
                                            int& nonfinite) {
  const int e = (int)((bits >> 7) & 0xFFu);
  const int f = (int)(bits & 0x7Fu);
  neg = (int)((bits >> 15) & 1u);
  nonfinite = e == 0xFF;
  if (e == 0) {
    sig = f;
    exp = -133;
  } else {
    sig = 0x80 | f;
    exp = e - 134;
  }
}

__device__ __forceinline__ double pow2(int e) {  // exact 2^e for -1022 <= e <= 1023
  return __longlong_as_double((long long)(e + 1023) << 52);
}

__device__ __forceinline__ uint32_t elem(const uint4* row, int k) {
  const uint32_t w = reinterpret_cast<const uint32_t*>(row)[k >> 1];
  return (k & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Exact sum of the 128 products of two bf16 vectors, rounded once to nearest
// even float64. Product magnitudes are sig_a*sig_b < 2^16 at binary exponents
// in [-266, 240]; a fixed-point integer with unit 2^-266 and 17 limbs of 32 bits
// holds every partial sum exactly. Limbs are accumulated as signed 64-bit
// values (each gets at most 256 additions below 2^32) and carried once.
__device__ __noinline__ double exact_dot_wide(const uint4* xa, const uint4* xb) {
  long long acc[17];
#pragma unroll
  for (int i = 0; i < 17; ++i) acc[i] = 0;
  for (int k = 0; k < kD; ++k) {
    int sa, ea, na, fa, sb, eb, nbv, fb;
    decode_bf16(elem(xa, k), sa, ea, na, fa);
    decode_bf16(elem(xb, k), sb, eb, nbv, fb);
    if (sa == 0 || sb == 0 || fa || fb) continue;
    const int pos = ea + eb + 266;
    const int li = pos >> 5, sh = pos & 31;
    const unsigned long long v = (unsigned long long)(uint32_t)(sa * sb) << sh;
    const long long lo = (long long)(v & 0xFFFFFFFFull), hi = (long long)(v >> 32);
    if (na ^ nbv) {
      acc[li] -= lo;
      acc[li + 1] -= hi;
    } else {
      acc[li] += lo;
      acc[li + 1] += hi;
    }
  }
  unsigned long long limb[17];
  long long carry = 0;
  for (int i = 0; i < 17; ++i) {
    const long long x = acc[i] + carry;
    limb[i] = (unsigned long long)x & 0xFFFFFFFFull;
    carry = x >> 32;
  }
  bool negative = false;
  if (carry < 0) {  // redo on the negated sum to get the magnitude
    negative = true;
    carry = 0;
    for (int i = 0; i < 17; ++i) {
      const long long x = -acc[i] + carry;
      limb[i] = (unsigned long long)x & 0xFFFFFFFFull;
      carry = x >> 32;
    }
  }
  int h = 16;
  while (h >= 0 && limb[h] == 0) --h;
  if (h < 0) return 0.0;
  const int nlz = __clz((int)(uint32_t)limb[h]);
  const unsigned long long l1 = h >= 1 ? limb[h - 1] : 0ull;
  const unsigned long long l2 = h >= 2 ? limb[h - 2] : 0ull;
  unsigned long long w = (limb[h] << 32) | l1;
  bool sticky;
  if (nlz) {
    w = (w << nlz) | (l2 >> (32 - nlz));
    sticky = ((l2 << nlz) & 0xFFFFFFFFull) != 0;
  } else {
    sticky = l2 != 0;
  }
  for (int i = 0; i < h - 2; ++i) sticky |= limb[i] != 0;
  unsigned long long mant = w >> 11;
  const bool round_bit = (w >> 10) & 1ull;
  sticky |= (w & 0x3FFull) != 0;
  int e = 32 * h + 31 - nlz - 52 - 266;  // binary exponent of mant's last bit
  if (round_bit && (sticky || (mant & 1ull))) ++mant;
  if (mant == (1ull << 53)) {
    mant >>= 1;
    ++e;
  }
  const double r = __dmul_rn(__ull2double_rn(mant), pow2(e));
  return negative ? -r : r;
}

// Exact dot product of rows i and j of the candidate set, rounded once to float64.
__device__ double exact_dot(FpsSmem& sm, int i, int j) {
  if ((sm.flags[i] | sm.flags[j]) & 1) return exact_dot_wide(sm.x + i * 16, sm.x + j * 16);
  const int ei = sm.emin[i], ej = sm.emin[j];
  long long acc = 0;
  for (int k = 0; k < kD; ++k) {
    int sa, ea, na, fa, sb, eb, nbv, fb;
    decode_bf16(elem(sm.x + i * 16, k), sa, ea, na, fa);
    decode_bf16(elem(sm.x + j * 16, k), sb, eb, nbv, fb);
    if (sa == 0 || sb == 0 || fa || fb) continue;
    const long long p = (long long)(sa << (ea - ei)) * (long long)(sb << (eb - ej));
    acc += (na ^ nbv) ? -p : p;
  }
  return acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(ei + ej));
}

// The float64 cosine of the reference arithmetic.
__device__ double cos64(FpsSmem& sm, int i, int j) {
  const double gii = sm.diag[i], gjj = sm.diag[j];
  if (gii == 0.0 || gjj == 0.0) return 0.0;
  return __ddiv_rn(exact_dot(sm, i, j), __dsqrt_rn(__dmul_rn(gii, gjj)));
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
  return v;
}

__device__ __forceinline__ double warp_max64(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double o = __shfl_xor_sync(0xFFFFFFFFu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

// Decides argmin over the candidates whose float32 values v0 (index lane) and
// v1 (index lane + 32) are valid, with error bound err. Exact float64 values
// for close candidates come from exact(j), evaluated cooperatively by the
// warp: exact(j, lane) returns lane's share, combined with `combine`.
// Returns the winning index (same on every lane).
template <class Exact>
__device__ int filtered_argmin(FpsSmem& sm, float v0, float v1, bool ok0, bool ok1, float err,
                               Exact exact) {
  const int lane = threadIdx.x & 31;
  const float inf = __int_as_float(0x7f800000);
  const float m = warp_min(fminf(ok0 ? v0 : inf, ok1 ? v1 : inf));
  const float lim = m + 2.0f * err;
  const unsigned b0 = __ballot_sync(0xFFFFFFFFu, ok0 && v0 <= lim);
  const unsigned b1 = __ballot_sync(0xFFFFFFFFu, ok1 && v1 <= lim);
  const int nc = __popc(b0) + __popc(b1);
  if (nc == 1) return b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
  if (nc == 0) {  // only with NaN values (already latched as non-finite): lowest valid index
    const unsigned o0 = __ballot_sync(0xFFFFFFFFu, ok0), o1 = __ballot_sync(0xFFFFFFFFu, ok1);
    return o0 ? __ffs(o0) - 1 : (o1 ? 32 + __ffs(o1) - 1 : 0);
  }
  // close call: list the candidates in index order, then compare float64 values
  if (ok0 && v0 <= lim) sm.cand[__popc(b0 & ((1u << lane) - 1u))] = lane;
  if (ok1 && v1 <= lim) sm.cand[__popc(b0) + __popc(b1 & ((1u << lane) - 1u))] = lane + 32;
  __syncwarp();
  int best = -1;
  double bv = 0.0;
  for (int q = 0; q < nc; ++q) {
    const int j = sm.cand[q];
    const double v = exact(j);  // warp-cooperative, same value on every lane
    if (best < 0 || v < bv) {
      best = j;
      bv = v;
    }
  }
  __syncwarp();
  return best;
}

__global__ void __launch_bounds__(kThreads) fps_kernel(FpsParams P) {
  extern __shared__ __align__(16) unsigned char fps_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t head = blockIdx.x;
  const int nb = P.nb, n = P.nb + P.nr, m = P.m;
  if (m == 0) return;  // nothing is kept and there is no trace
  FpsSmem sm = carve(fps_smem, n);
  uint4* bq = P.bq + head * P.fps_cap * 16;
  const uint4* rq = P.rq + head * P.n_rq * 16;

  // candidates: beacons (oldest first), then recents (oldest first)
  for (int idx = tid; idx < n * 16; idx += kThreads) {
    const int r = idx >> 4, part = idx & 15;
    const uint4* src = r < nb ? bq + r * 16 : rq + ((P.ring_first + r - nb) % P.n_rq) * 16;
    sm.x[idx] = src[part];
  }
  __syncthreads();

  int8_t* trace = P.trace + head * m;
  if (n <= m) {  // nothing to sample: keep every candidate in order
    for (int idx = tid; idx < n * 16; idx += kThreads) bq[idx] = sm.x[idx];
    for (int k = tid; k < m; k += kThreads) trace[k] = k < n ? (int8_t)k : (int8_t)-1;
    return;
  }

  // per row: exponent range, scaled float32 copy, exact diagonal (4 threads per row)
  for (int r0 = 0; r0 < n; r0 += kThreads / 4) {
    const int r = r0 + (tid >> 2), q = tid & 3;
    int emin = INT_MAX, emax = INT_MIN, bad = 0;
    if (r < n) {
      for (int k = q * 32; k < q * 32 + 32; ++k) {
        int sig, e, neg, nf;
        decode_bf16(elem(sm.x + r * 16, k), sig, e, neg, nf);
        bad |= nf;
        if (sig != 0 && !nf) {
          emin = min(emin, e);
          emax = max(emax, e);
        }
      }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      emin = min(emin, __shfl_xor_sync(0xFFFFFFFFu, emin, off));
      emax = max(emax, __shfl_xor_sync(0xFFFFFFFFu, emax, off));
      bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, off);
    }
    const bool zero_row = emin == INT_MAX;
    if (zero_row) emin = emax = 0;
    const bool wide = (emax - emin) > 20;
    const bool inexact = (emax - emin) > 110;  // scaled float32 copy could underflow
    long long acc = 0;
    if (r < n) {
      if (bad && q == 0) latch(P.status, BKV_ERR_NONFINITE);
      for (int k = q * 32; k < q * 32 + 32; ++k) {
        int sig, e, neg, nf;
        decode_bf16(elem(sm.x + r * 16, k), sig, e, neg, nf);
        float yv = 0.f;
        if (sig != 0 && !nf) {
          // sig * 2^(e - emax - 8), exact: the power of two is a normal float32 here
          if (!inexact) yv = (float)sig * __int_as_float((e - emax - 8 + 127) << 23);
          if (!wide) acc += (long long)(sig << (e - emin)) * (long long)(sig << (e - emin));
        }
        sm.Y(r, k) = neg ? -yv : yv;
      }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
    if (r < n && q == 0) {
      sm.emin[r] = emin;
      sm.emax[r] = emax;
      sm.flags[r] = (wide ? 1 : 0) | (inexact ? 2 : 0);
      if (!wide) sm.diag[r] = acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(2 * emin));
    }
  }
  __syncthreads();
  for (int r = tid; r < n; r += kThreads)  // wide rows: exact diagonal by the long accumulator
    if (sm.flags[r] & 1) sm.diag[r] = exact_dot_wide(sm.x + r * 16, sm.x + r * 16);
  __syncthreads();

  // float32 Gram: warp item = 8 rows x 32 columns; lane = column, rows broadcast
  const int rblocks = (n + 7) / 8, cgroups = (n + 31) / 32;
  for (int item = warp; item < rblocks * cgroups; item += kThreads / 32) {
    const int i0 = (item % rblocks) * 8, j = (item / rblocks) * 32 + lane;
    float s[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a) s[a][0] = s[a][1] = s[a][2] = s[a][3] = 0.f;
    const float* yj = &sm.Y(j < n ? j : 0, 0);
#pragma unroll 2
    for (int k = 0; k < kD; k += 4) {
      const float4 b = *reinterpret_cast<const float4*>(yj + k);
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const int i = i0 + a < n ? i0 + a : 0;
        const float4 av = *reinterpret_cast<const float4*>(&sm.Y(i, k));
        s[a][0] = __fmaf_rn(av.x, b.x, s[a][0]);
        s[a][1] = __fmaf_rn(av.y, b.y, s[a][1]);
        s[a][2] = __fmaf_rn(av.z, b.z, s[a][2]);
        s[a][3] = __fmaf_rn(av.w, b.w, s[a][3]);
      }
    }
    if (j < n) {
#pragma unroll
      for (int a = 0; a < 8; ++a)
        if (i0 + a < n) sm.C(i0 + a, j) = __fadd_rn(__fadd_rn(s[a][0], s[a][1]), __fadd_rn(s[a][2], s[a][3]));
    }
  }
  __syncthreads();

  // float32 cosines, in place (each entry is read and rewritten by one thread);
  // rows whose scaled copy is not exact take the float64 value
  float* inv = reinterpret_cast<float*>(sm.v64);  // 1 / sqrt(G32_ii), reusing the fallback buffer
  for (int i = tid; i < n; i += kThreads) inv[i] = sm.C(i, i) > 0.f ? rsqrtf(sm.C(i, i)) : 0.f;
  __syncthreads();
  for (int i = warp; i < n; i += kThreads / 32) {
    for (int j = lane; j < n; j += 32) {
      float v;
      if ((sm.flags[i] | sm.flags[j]) & 2) v = __double2float_rn(cos64(sm, i, j));
      else v = __fmul_rn(__fmul_rn(sm.C(i, j), inv[i]), inv[j]);
      sm.C(i, j) = v;
    }
  }
  __syncthreads();

  if (warp == 0) {
    const int i0 = lane, i1 = lane + 32;
    const bool live0 = i0 < n, live1 = i1 < n;
    float a0 = 0.f, a1 = 0.f;
    if (live0) {
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = __fadd_rn(acc, sm.C(i0, j));
      a0 = __fdiv_rn(acc, (float)n);
    }
    if (live1) {
      float acc = 0.f;
      for (int j = 0; j < n; ++j) acc = __fadd_rn(acc, sm.C(i1, j));
      a1 = __fdiv_rn(acc, (float)n);
    }
    // exact mean cosine of candidate i: lanes evaluate cos64(i, j) for their j,
    // lane 0 sums them left to right
    auto mean64 = [&](int i) -> double {
      for (int j = lane; j < n; j += 32) sm.v64[j] = cos64(sm, i, j);
      __syncwarp();
      double acc = 0.0;
      for (int j = 0; j < n; ++j) acc = __dadd_rn(acc, sm.v64[j]);
      __syncwarp();
      return __ddiv_rn(acc, (double)n);
    };
    const int p0 = filtered_argmin(sm, a0, a1, live0, live1, kMeanErr, mean64);
    if (lane == 0) sm.picks[0] = p0;
    bool ch0 = i0 == p0, ch1 = i1 == p0;
    float S0 = live0 ? sm.C(i0, p0) : 0.f, S1 = live1 ? sm.C(i1, p0) : 0.f;
    for (int k = 1; k < m; ++k) {
      // exact running maximum of candidate j over the picks so far
      auto smax64 = [&](int j) -> double {
        double v = -__longlong_as_double(0x7ff0000000000000LL);
        for (int q = lane; q < k; q += 32) {
          const double c = cos64(sm, j, sm.picks[q]);
          v = c > v ? c : v;
        }
        return warp_max64(v);
      };
      __syncwarp();
      const int r = filtered_argmin(sm, S0, S1, live0 && !ch0, live1 && !ch1, kCosErr, smax64);
      if (i0 == r) ch0 = true;
      if (i1 == r) ch1 = true;
      if (live0) S0 = fmaxf(S0, sm.C(i0, r));
      if (live1) S1 = fmaxf(S1, sm.C(i1, r));
      if (lane == 0) sm.picks[k] = r;
    }
    __syncwarp();
    for (int k = lane; k < m; k += 32) trace[k] = (int8_t)sm.picks[k];
    const unsigned m0 = __ballot_sync(0xFFFFFFFFu, ch0), m1 = __ballot_sync(0xFFFFFFFFu, ch1);
    const unsigned lt = (1u << lane) - 1u;
    if (ch0) sm.keep_src[__popc(m0 & lt)] = i0;
    if (ch1) sm.keep_src[__popc(m0) + __popc(m1 & lt)] = i1;
  }
  __syncthreads();

  for (int idx = tid; idx < m * 16; idx += kThreads) bq[idx] = sm.x[sm.keep_src[idx >> 4] * 16 + (idx & 15)];
}

}  // namespace

cudaError_t launch_fps(const FpsParams& p, cudaStream_t s) {
  const int n = p.nb + p.nr;
  if (p.heads_total <= 0 || p.m == 0) return cudaSuccess;
  if (n > kMaxCand || n <= 0) return n <= 0 ? cudaSuccess : cudaErrorInvalidValue;
  const size_t smem = fps_smem_bytes(n);
  static size_t configured = 48 * 1024;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(fps_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  fps_kernel<<<(unsigned)p.heads_total, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
