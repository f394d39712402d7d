// Farthest-point sampling of pre-RoPE queries, one CTA per query head.
//
// BeaconKV reading notes, §2.2, Algorithm 1 (and eq. 9 / Algorithm 2 for when
// it runs): with cos the cosine similarity of two candidates,
//   a_i = (1/N) sum_j cos(q_i, q_j),  p = argmin_i a_i,  I = {p},  S_j = cos(q_j, q_p);
//   repeat r = argmin_{j not in I} S_j,  I += {r},  S_j = max(S_j, cos(q_j, q_r))
// until |I| = m. Ties go to the lowest index. The kept rows are written back
// in candidate order (oldest first) and the pick order is the trace.
//
// Every decision is taken on float64 values that are bit-identical to a plain
// float64 evaluation of the same formulas:
//   * G_ij, the dot product of two bf16 vectors, is computed EXACTLY and then
//     rounded once to float64 - with 64-bit integer arithmetic on the bf16
//     significands when both vectors' exponents span <= 20 binades (the sum of
//     128 products then stays below 2^63), otherwise with a 544-bit fixed-point
//     accumulator over the whole bf16 product range;
//   * cos_ij = G_ij / sqrt(G_ii * G_jj) with correctly rounded IEEE float64
//     multiply, square root and divide (0 if either vector is zero);
//   * a_i is summed left to right in j order, then divided by N.
#include <climits>

#include "bkv_internal.cuh"

namespace bkv {

namespace {

constexpr int kThreads = 128;
constexpr int kMaxCand = 64;      // beacons (< fps_cap <= 32) + recents (<= 32)
constexpr int kAStride = kD + 1;  // int32 row stride: row i, column k lands in bank (i + k) % 32

// Dynamic shared memory for n candidates:
//   x[n][16] uint4 (bf16 rows) | a[n][129] int32 | g[n][n+1] double (Gram, then cosines)
//   | diag[n] double | ebase[n] int | wide[n] int | keep_src[32] int
struct FpsSmem {
  uint4* x;
  int32_t* a;
  double* g;
  double* diag;
  int* ebase;
  int* wide;
  int* keep_src;
  int n;
  __device__ double& G(int i, int j) { return g[i * (n + 1) + j]; }
  __device__ int32_t& A(int i, int k) { return a[i * kAStride + k]; }
};

__host__ __device__ inline size_t fps_smem_bytes(int n) {
  size_t off = (size_t)n * 256;
  off += ((size_t)n * kAStride * 4 + 15) / 16 * 16;
  off += (size_t)n * (n + 1) * 8;
  off += (size_t)n * 8;
  off += (size_t)n * 8 + 32 * 4;
  return off;
}

__device__ inline FpsSmem carve(unsigned char* base, int n) {
  FpsSmem s;
  s.n = n;
  size_t off = 0;
  s.x = reinterpret_cast<uint4*>(base);
  off += (size_t)n * 256;
  s.a = reinterpret_cast<int32_t*>(base + off);
  off += ((size_t)n * kAStride * 4 + 15) / 16 * 16;
  s.g = reinterpret_cast<double*>(base + off);
  off += (size_t)n * (n + 1) * 8;
  s.diag = reinterpret_cast<double*>(base + off);
  off += (size_t)n * 8;
  s.ebase = reinterpret_cast<int*>(base + off);
  s.wide = s.ebase + n;
  s.keep_src = s.wide + n;
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

// Lexicographic (value, index) minimum over the lanes where `valid` holds.
__device__ __forceinline__ int warp_argmin(double v, int idx, bool valid) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double ov = __shfl_xor_sync(0xFFFFFFFFu, v, off);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, idx, off);
    const bool ovalid = __shfl_xor_sync(0xFFFFFFFFu, (int)valid, off) != 0;
    const bool take = ovalid && (!valid || ov < v || (ov == v && oi < idx));
    if (take) {
      v = ov;
      idx = oi;
      valid = true;
    }
  }
  return idx;
}

// Upper-triangle pair number -> (i, j), i <= j < n.
__device__ __forceinline__ void tri_pair(int p, int n, int& i, int& j) {
  i = 0;
  while (p >= n - i) {
    p -= n - i;
    ++i;
  }
  j = i + p;
}

__global__ void __launch_bounds__(kThreads) fps_kernel(FpsParams P) {
  extern __shared__ __align__(16) unsigned char fps_smem[];
  const int tid = threadIdx.x;
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

  // integer significands on a per-row common exponent (4 threads per row)
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
    if (r < n) {
      if (emin == INT_MAX) emin = emax = 0;  // zero row
      const int wide = (emax - emin) > 20;
      if (bad && q == 0) latch(P.status, BKV_ERR_NONFINITE);
      for (int k = q * 32; k < q * 32 + 32; ++k) {
        int sig, e, neg, nf;
        decode_bf16(elem(sm.x + r * 16, k), sig, e, neg, nf);
        int v = 0;
        if (!wide && sig != 0 && !nf) v = sig << (e - emin);
        sm.A(r, k) = neg ? -v : v;
      }
      if (q == 0) {
        sm.ebase[r] = emin;
        sm.wide[r] = wide;
      }
    }
  }
  __syncthreads();

  // exact Gram over the upper triangle
  const int npairs = n * (n + 1) / 2;
  for (int p = tid; p < npairs; p += kThreads) {
    int i, j;
    tri_pair(p, n, i, j);
    double gv;
    if (!sm.wide[i] && !sm.wide[j]) {
      const int32_t* ai = &sm.A(i, 0);
      const int32_t* aj = &sm.A(j, 0);
      long long acc = 0;
#pragma unroll 8
      for (int k = 0; k < kD; ++k) acc += (long long)ai[k] * (long long)aj[k];
      gv = acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(sm.ebase[i] + sm.ebase[j]));
    } else {
      gv = exact_dot_wide(sm.x + i * 16, sm.x + j * 16);
    }
    sm.G(i, j) = gv;
    sm.G(j, i) = gv;
    if (i == j) sm.diag[i] = gv;
  }
  __syncthreads();

  // cosines, in place of the Gram
  for (int p = tid; p < npairs; p += kThreads) {
    int i, j;
    tri_pair(p, n, i, j);
    const double gii = sm.diag[i], gjj = sm.diag[j];
    double cv = 0.0;
    if (gii != 0.0 && gjj != 0.0) cv = __ddiv_rn(sm.G(i, j), __dsqrt_rn(__dmul_rn(gii, gjj)));
    if (cv != cv) latch(P.status, BKV_ERR_NONFINITE);
    sm.G(i, j) = cv;
    sm.G(j, i) = cv;
  }
  __syncthreads();

  // mean cosine, start point and greedy picks; lane i owns candidates i and i + 32
  if (tid < 32) {
    const int i0 = tid, i1 = tid + 32;
    const bool live0 = i0 < n, live1 = i1 < n;
    double a0 = 0.0, a1 = 0.0;
    if (live0) {
      double acc = 0.0;
      for (int j = 0; j < n; ++j) acc = __dadd_rn(acc, sm.G(i0, j));
      a0 = __ddiv_rn(acc, (double)n);
    }
    if (live1) {
      double acc = 0.0;
      for (int j = 0; j < n; ++j) acc = __dadd_rn(acc, sm.G(i1, j));
      a1 = __ddiv_rn(acc, (double)n);
    }
    // local lexicographic minimum of the lane's two candidates (i0 < i1)
    const bool take1 = live1 && (!live0 || a1 < a0);
    const int p0 = warp_argmin(take1 ? a1 : a0, take1 ? i1 : i0, live0 || live1);
    bool ch0 = i0 == p0, ch1 = i1 == p0;
    double S0 = live0 ? sm.G(i0, p0) : 0.0, S1 = live1 ? sm.G(i1, p0) : 0.0;
    if (tid == 0) trace[0] = (int8_t)p0;
    for (int k = 1; k < m; ++k) {
      const bool v0 = live0 && !ch0, v1 = live1 && !ch1;
      const bool t1 = v1 && (!v0 || S1 < S0);
      const int r = warp_argmin(t1 ? S1 : S0, t1 ? i1 : i0, v0 || v1);
      if (i0 == r) ch0 = true;
      if (i1 == r) ch1 = true;
      if (live0) {
        const double cr = sm.G(i0, r);
        S0 = cr > S0 ? cr : S0;
      }
      if (live1) {
        const double cr = sm.G(i1, r);
        S1 = cr > S1 ? cr : S1;
      }
      if (tid == 0) trace[k] = (int8_t)r;
    }
    const unsigned m0 = __ballot_sync(0xFFFFFFFFu, ch0), m1 = __ballot_sync(0xFFFFFFFFu, ch1);
    const unsigned lt = (1u << tid) - 1u;
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
