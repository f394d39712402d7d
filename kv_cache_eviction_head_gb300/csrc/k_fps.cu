// Farthest-point sampling of pre-RoPE queries, one warp per query head.
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
//   * rows are kept in shared memory as bf16. A batch of rows whose every
//     8-component piece is zero or has its largest magnitude in
//     [2^-40, 2^21) is kept as loaded: each nonzero row's largest component
//     then lies in that range, products stay below 2^44 and sums below 2^51,
//     and the at most 255 products or partial sums flushed below 2^-126 move
//     G_ij by less than 2^-118, under 2^-38 of ||y_i|| ||y_j|| >= 2^-80. Any other row is scaled
//     by a power of two that brings its largest component into [1, 4), or
//     above 2^-7 for a row of bf16 subnormals (exact, apart from components
//     more than 126 binades below the largest, which round to the bf16
//     subnormal grid with an error below 2^-134). Cosines do not depend on
//     the scale; when every row is held as loaded, the kept rows are written
//     back from shared memory;
//   * up to 32 candidates (one 32-row block per head): the Gram comes from the
//     tensor cores. The warps of a persistent CTA write their heads' rows into
//     one 128 x 128 bf16 operand; each warp multiplies it by its own 32 rows
//     (tcgen05.mma, M = 128, N = 32, fp32 accumulators in its 32 of the CTA's
//     128 TMEM columns) and reads rows 32 w.. of the result, its head's Gram,
//     one row per lane. The products are exact; the accumulation order
//     and rounding are the hardware's, so the bound used assumes only fp32
//     precision at each of the 127 additions with any rounding direction:
//     |G32 - G| <= 127 * 2^-23 * sum_k |y_ik y_jk| <= 1.52e-5 ||y_i|| ||y_j||
//     (products of bf16 subnormals, if flushed, add below 2^-100 relative). A
//     probe of 128 x 128 x 128 Grams (normal, near-duplicate, wide-exponent,
//     cancelling and two-scale rows) measured at most 10.8 * 2^-24 of
//     sum_k |y_ik y_jk|, a twentieth of the bound;
//   * up to 64 candidates: the float32 Gram entry is two interleaved sums
//     (even and odd k) of 64 bf16 products each (exact, or below 2^-149 off
//     where a product underflows), added once, so its error is at most
//     gamma_64 * ||y_i|| ||y_j|| (3.8e-6 relative) plus < 2^-123 from the
//     subnormal roundings, against ||y_i|| >= 2^-7 for every nonzero scaled
//     row (2^-40 for one held as loaded);
//   * c_ij = (G32_ij * r_i) * r_j with r_i = rsqrtf(G32_ii) (2 ulp, on a
//     diagonal within 1.52e-5 relative) is then within 3.2e-5 of the float64
//     cosine (8.5e-6 for the float32 Gram); the filters use kCosErr = 4e-5;
//   * the mean a_i in float32 (any summation order, N <= 64) is within
//     3.2e-5 + 63 * 2^-24 of the float64 mean; the filters use kMeanErr;
//   * a decision (argmin of the mean cosine, argmin of the running max) is
//     final when the float32 minimum beats every other candidate by more than
//     twice its error bound - then the float64 values order the same way;
//   * otherwise the float64 values of the close candidates are computed
//     exactly as defined above and compared, ties going to the lowest index;
//     a candidate's running maximum is taken over the picks whose float32
//     cosine lies within twice the bound of its float32 maximum only (every
//     other pick's float64 cosine is below that maximum's).
// The exact G_ij uses 64-bit integer arithmetic on the bf16 significands when
// both vectors' exponents span <= 20 binades (128 products then sum below
// 2^63), otherwise a 544-bit fixed-point accumulator over the whole bf16
// product range; either way it is rounded once to nearest even, and a whole
// warp evaluates one dot product (four elements per lane, exact 64-bit sums
// added across the warp) where a decision waits on it. The per-row data the
// exact path needs (exponent range, exact G_ii) is made when a close call
// first needs the row.
#include <atomic>
#include <climits>

#include "bkv_internal.cuh"
#include "exact_dot.cuh"
#include "score_common.cuh"  // mbarrier, TMEM and tcgen05 wrappers

namespace bkv {

namespace {

// one warp per head; up to 32 candidates four heads share one tensor-core Gram
template <int NH>
constexpr int kHeadsPerCta = NH == 1 ? 4 : 2;
constexpr int kMaxCand = 64;          // beacons (< fps_cap <= 32) + recents (<= 32)
constexpr int kYStride = kD + 8;      // bf16 row stride (272 bytes): 16-byte aligned rows, and LDS.64 of 8 consecutive rows hit distinct banks
constexpr float kCosErr = 4e-5f;      // |c32 - cos64| bound used by the filters
constexpr float kMeanErr = 4.5e-5f;   // |a32 - a64| bound used by the filters
constexpr int kGramCols = 128;        // TMEM columns of the tensor-core Gram (4 heads x 32)
constexpr uint32_t kRawHi = 148u << 7;  // bf16 magnitude bits of 2^21
constexpr uint32_t kRawLo = 87u << 7;   // bf16 magnitude bits of 2^-40
constexpr float kInfF = __builtin_huge_valf();

// Per-warp shared memory for NT = 32 * NH candidate slots.
template <int NH>
struct WarpSmem {
  static constexpr int NT = 32 * NH;
  // NH == 1: the rows live in the CTA's tensor-core operand instead
  static constexpr size_t kY = NH == 1 ? 0 : (((size_t)NT * kYStride * 2 + 15) / 16) * 16;
  static constexpr size_t kC = (((size_t)NT * (NT + 1) * 4 + 15) / 16) * 16;
  static constexpr size_t kMisc = (size_t)NT * 8 * 2 + (size_t)NT * 4 * 5 + 64 * 4;
  static constexpr size_t kBytes = ((kY + kC + kMisc) + 15) / 16 * 16;

  __nv_bfloat16* y;  // [NT][kYStride] rows as loaded or scaled by a power of two, bf16 (see the header)
  float* c;       // [NT][NT + 1]   Gram, then cosines
  double* diag;   // [NT] exact G_ii rounded to float64 (close calls only)
  double* v64;    // [NT] exact values of a close call
  float* inv;     // [NT] rsqrt of the float32 diagonal
  int* emin;      // [NT] smallest exponent of a nonzero component
  int* emax;      // [NT]
  int* wide;      // [NT] exponent span > 20
  int* cand;      // [NT] close-call candidates
  int* picks;     // [32] pick order
  int* keep_src;  // [32]

  __device__ WarpSmem(unsigned char* base) {
    y = reinterpret_cast<__nv_bfloat16*>(base);
    c = reinterpret_cast<float*>(base + kY);
    unsigned char* m = base + kY + kC;
    diag = reinterpret_cast<double*>(m);
    v64 = diag + NT;
    inv = reinterpret_cast<float*>(v64 + NT);
    emin = reinterpret_cast<int*>(inv + NT);
    emax = emin + NT;
    wide = emax + NT;
    cand = wide + NT;
    picks = cand + NT;
    keep_src = picks + 32;
  }
  __device__ float& C(int i, int j) { return c[i * (NT + 1) + j]; }
};

__device__ __forceinline__ double warp_max64(double v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double o = __shfl_xor_sync(kFull, v, off);
    v = o > v ? o : v;
  }
  return v;
}

// Order-preserving map of float32 to uint32 (for a single-instruction warp min).
__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unkey(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Decides argmin over the candidates whose float32 values v0 (index lane) and
// v1 (index lane + 32) are valid, with error bound err. Exact float64 values
// for close candidates come from exact(j), evaluated cooperatively by the
// warp (same value on every lane). Returns the winning index on every lane.
template <class Exact>
__device__ __forceinline__ int filtered_argmin(int* cand, float v0, float v1, bool ok0, bool ok1, float err, Exact exact) {
  const int lane = threadIdx.x & 31;
  const uint32_t k = min(ok0 ? fkey(v0) : 0xFFFFFFFFu, ok1 ? fkey(v1) : 0xFFFFFFFFu);
  const float m = unkey(__reduce_min_sync(kFull, k));
  const float lim = m + 2.0f * err;
  const unsigned b0 = __ballot_sync(kFull, ok0 && v0 <= lim);
  const unsigned b1 = __ballot_sync(kFull, ok1 && v1 <= lim);
  const int nc = __popc(b0) + __popc(b1);
  if (nc == 1) return b0 ? __ffs(b0) - 1 : 32 + __ffs(b1) - 1;
  if (nc == 0) {  // only with NaN values (already latched as non-finite): lowest valid index
    const unsigned o0 = __ballot_sync(kFull, ok0), o1 = __ballot_sync(kFull, ok1);
    return o0 ? __ffs(o0) - 1 : (o1 ? 32 + __ffs(o1) - 1 : 0);
  }
  // close call: list the candidates in index order, then compare float64 values
  if (ok0 && v0 <= lim) cand[__popc(b0 & ((1u << lane) - 1u))] = lane;
  if (ok1 && v1 <= lim) cand[__popc(b0) + __popc(b1 & ((1u << lane) - 1u))] = lane + 32;
  __syncwarp();
  int best = -1;
  double bv = 0.0;
  for (int q = 0; q < nc; ++q) {
    const int j = cand[q];
    const double v = exact(j);
    if (best < 0 || v < bv) {
      best = j;
      bv = v;
    }
  }
  __syncwarp();
  return best;
}

// Dynamic shared memory of one CTA (NH == 1: the 1024-aligned 128 x 128 bf16
// operand of the Gram, then the warps' blocks).
template <int NH>
constexpr size_t fps_cta_smem() {
  return (NH == 1 ? 1024 + (size_t)kTileBytes : 0) + WarpSmem<NH>::kBytes * kHeadsPerCta<NH>;
}

template <int NH>
__global__ void __launch_bounds__(32 * kHeadsPerCta<NH>, NH == 1 ? 4 : 8) fps_kernel(FpsParams P) {
  using W = WarpSmem<NH>;
  constexpr int NT = W::NT;
  extern __shared__ __align__(16) unsigned char fps_smem[];
  __shared__ uint64_t gram_bar[4];  // NH == 1: one per warp, its Gram product is done
  __shared__ uint32_t gram_tmem;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = P.nb, n = P.nb + P.nr, m = P.m;
  unsigned char* opnd = fps_smem;  // NH == 1: the Gram's operand, rows 32 * warp + r
  unsigned char* wbase = fps_smem;
  if constexpr (NH == 1) {
    opnd = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(fps_smem) + 1023) & ~(uintptr_t)1023);
    wbase = opnd + kTileBytes;
  }
  W sm(wbase + (size_t)warp * W::kBytes);
  // NH == 1 with sampling: persistent CTAs of four warps; each warp takes a
  // head at a time and multiplies the CTA's 128-row operand by its own 32
  // rows into its own 32 TMEM columns, so the warps never wait on each other
  const bool tc = NH == 1 && n > m;  // the same for the whole launch
  if (tc) {
    if (warp == 0) tmem_alloc(&gram_tmem, kGramCols);
    if (threadIdx.x == 0) {
      for (int w = 0; w < 4; ++w) mbar_init(&gram_bar[w], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  const uint32_t tmem = tc ? gram_tmem : 0u;
  uint32_t gph = 0u;  // parity of this warp's Gram barrier
  const int64_t stride = (int64_t)gridDim.x * kHeadsPerCta<NH>;
  for (int64_t head = (int64_t)blockIdx.x * kHeadsPerCta<NH> + warp; head < P.heads_total; head += stride) {
  uint4* bq = P.bq + head * P.fps_cap * 16;
  const uint4* rq = P.rq + head * P.n_rq * 16;
  // candidates: beacons (oldest first), then recents (oldest first)
  auto row = [&](int i) -> const uint4* {
    return i < nb ? bq + i * 16 : rq + ((P.ring_first + i - nb) % P.n_rq) * 16;
  };
  int8_t* trace = P.trace + head * m;
  bool raw_rows = n > m;  // every candidate row sits in shared memory exactly as loaded

  if (n > m) {
    // ---- rows -> bf16 in shared memory, as loaded or each scaled so its
    // largest component lies in [1, 4)
    // lanes 0-15 take one row, lanes 16-31 the next; padding rows are zero.
    // A batch of rows is loaded before any is processed: all 32 rows at once
    // for up to 32 candidates (one memory latency per head), 16 at a time for
    // up to 64; the rows were prefetched into L2 during the warp's previous head.
    constexpr int kLoadBatch = NH == 1 ? 16 : 8;
    bool bad = false;
    const int part = lane & 15;
#pragma unroll 1
    for (int r0 = 0; r0 < NT; r0 += 2 * kLoadBatch) {
      uint4 vb[kLoadBatch];
#pragma unroll
      for (int bi = 0; bi < kLoadBatch; ++bi) {
        const int r = r0 + 2 * bi + (lane >> 4);
        vb[bi] = r < n ? __ldg(row(r) + part) : make_uint4(0, 0, 0, 0);
      }
      // a batch whose every 8-component piece is zero or has its largest
      // magnitude in [2^-40, 2^21) is kept as loaded (then every row's
      // largest component lies there too)
      bool in_range = true;
#pragma unroll
      for (int bi = 0; bi < kLoadBatch; ++bi) {
        uint32_t mx = 0;
        const uint32_t w[4] = {vb[bi].x, vb[bi].y, vb[bi].z, vb[bi].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t x = w[q] & 0x7FFF7FFFu;  // bf16 magnitudes order as integers
          mx = max(mx, max(x & 0xFFFFu, x >> 16));
        }
        in_range &= mx < kRawHi && (mx >= kRawLo || mx == 0u);
      }
      const bool raw = __all_sync(kFull, in_range);
      raw_rows &= raw;
#pragma unroll
      for (int bi = 0; bi < kLoadBatch; ++bi) {
        const int r = r0 + 2 * bi + (lane >> 4);
        const uint32_t w[4] = {vb[bi].x, vb[bi].y, vb[bi].z, vb[bi].w};
        uint32_t o[4] = {w[0], w[1], w[2], w[3]};
        if (!raw) {
          uint32_t e = 0;
#pragma unroll
          for (int q = 0; q < 4; ++q) e = max(e, max((w[q] >> 7) & 0xFFu, (w[q] >> 23) & 0xFFu));
#pragma unroll
          for (int off = 1; off < 16; off <<= 1) e = max(e, __shfl_xor_sync(kFull, e, off));
          bad |= e == 0xFFu;
          const float scale = __int_as_float(max(254 - (int)e, 1) << 23);  // 2^(127 - e)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = __fmul_rn(__uint_as_float(w[q] << 16), scale);
            const float hi = __fmul_rn(__uint_as_float(w[q] & 0xFFFF0000u), scale);
            o[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
          }
        }
        if constexpr (NH == 1)  // SWIZZLE_128B K-major: 64-column slabs of 128-byte rows
          *reinterpret_cast<uint4*>(opnd + (part >> 3) * kSlabBytes + (32 * warp + r) * 128 +
                                    (((part & 7) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        else
          *reinterpret_cast<uint4*>(sm.y + r * kYStride + part * 8) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    if (__any_sync(kFull, bad) && lane == 0) latch(P.status, BKV_ERR_NONFINITE);
    // this warp's next head: its candidate rows into L2 while this one computes
    if (lane == 0 && head + stride < P.heads_total) {
      if (nb > 0) bulk_prefetch_l2(P.bq + (head + stride) * P.fps_cap * 16, (uint32_t)nb * (kD * 2));
      bulk_prefetch_l2(P.rq + (head + stride) * P.n_rq * 16, (uint32_t)P.n_rq * (kD * 2));
    }
    __syncwarp();

    // ---- tensor-core Gram (NH == 1): this warp's 32 rows against the CTA's
    // 128-row operand, D = Y_cta Y_w^T into columns 32 w; the rows 32 w.. of D
    // are this head's Gram (the other rows, from the other warps' heads, are
    // not read)
    float gr[32];  // NH == 1: row `lane` of this head's Gram
    if constexpr (NH == 1) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();  // this warp's reads of its columns (previous head) are complete
      __syncwarp();
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = smem_u32(opnd), b0 = a0 + (uint32_t)(32 * warp * 128);
        const uint32_t id = idesc_bf16(128, 32);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kSlabBytes + (uint32_t)(kk & 3) * 32;
          umma_bf16(tmem + (uint32_t)(32 * warp), sw128_desc(a0 + off), sw128_desc(b0 + off), id, kk ? 1u : 0u);
        }
        umma_commit(&gram_bar[warp]);
      }
      // bounded wait: a product that never completes latches BKV_ERR_TIMEOUT
      bool done = mbar_test(&gram_bar[warp], gph);
      const long long t0 = clock64();
      while (!done && clock64() - t0 < kWaitCycles) done = mbar_test(&gram_bar[warp], gph);
      if (!__all_sync(kFull, done) && lane == 0) latch(P.status, BKV_ERR_TIMEOUT);
      gph ^= 1u;
      tc_fence_after();
      tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(32 * warp), gr);
      tmem_wait_ld();
    }

    // ---- float32 Gram (NH == 2), 32 x 32 tiles; lane (I, J) = (lane & 7, lane >> 3)
    // owns rows I + 8a (a < 4) and columns J + 4b (b < 8) of a tile, so each
    // LDS.128 touches 8 (or 4) consecutive rows: distinct banks
    const int I = lane & 7, J = lane >> 3;
#pragma unroll 1
    for (int tile = 0; tile < (NH == 1 ? 0 : 3); ++tile) {
      const int ti = tile == 2 ? 1 : 0, tj = tile == 0 ? 0 : 1;
      const __nv_bfloat16* ya = sm.y + (ti * 32 + I) * kYStride;
      const __nv_bfloat16* yb = sm.y + (tj * 32 + J) * kYStride;
      // bf16 pair (k, k + 1) in one word -> float2 (exact)
      auto pair = [](uint32_t w) { return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)); };
      float2 s[4][8];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) s[a][b] = make_float2(0.f, 0.f);
#pragma unroll 2
      for (int k = 0; k < kD; k += 4) {
        uint2 av[4], bv[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) av[a] = *reinterpret_cast<const uint2*>(ya + 8 * a * kYStride + k);
#pragma unroll
        for (int b = 0; b < 8; ++b) bv[b] = *reinterpret_cast<const uint2*>(yb + 4 * b * kYStride + k);
        float2 b01[8], b23[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          b01[b] = pair(bv[b].x);
          b23[b] = pair(bv[b].y);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float2 a01 = pair(av[a].x), a23 = pair(av[a].y);
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            // (even k, odd k) partial sums of the same entry
            s[a][b] = __ffma2_rn(a01, b01[b], s[a][b]);
            s[a][b] = __ffma2_rn(a23, b23[b], s[a][b]);
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          const int i = ti * 32 + I + 8 * a, j = tj * 32 + J + 4 * b;
          const float g = __fadd_rn(s[a][b].x, s[a][b].y);
          sm.C(i, j) = g;
          if (ti != tj) sm.C(j, i) = g;  // exact products: the transposed sum is the same
        }
    }
    __syncwarp();

    // ---- cosines, row i by lane i (and i + 32), with the row sums for the means
    float a[NH];
    if constexpr (NH == 1) {
      // the diagonal entry of this lane's row, by selects in inline PTX: the
      // same chain in C++ is recognised as gr[lane] and moves the row to
      // local memory, a round trip that stalled every head
      float gd = 0.f;
#pragma unroll
      for (int q = 0; q < 32; ++q)
        asm("{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %2, %3;\n\tselp.f32 %0, %1, %0, p;\n\t}"
            : "+f"(gd)
            : "f"(gr[q]), "r"(q), "r"(lane));
      const float ri = gd > 0.f ? rsqrtf(gd) : 0.f;
      float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float v = __fmul_rn(__fmul_rn(gr[j], ri), __shfl_sync(kFull, ri, j));
        sm.C(lane, j) = v;
        if (j < n) {
          if (j & 1) acc1 = __fadd_rn(acc1, v);
          else acc0 = __fadd_rn(acc0, v);
        }
      }
      a[0] = __fdiv_rn(__fadd_rn(acc0, acc1), (float)n);
    } else {
    for (int i = lane; i < NT; i += 32) {
      const float g = sm.C(i, i);
      sm.inv[i] = g > 0.f ? rsqrtf(g) : 0.f;
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const int i = lane + 32 * h;
      float acc0 = 0.f, acc1 = 0.f;
      if (i < n) {
        const float ri = sm.inv[i];
        for (int j = 0; j < n; ++j) {
          const float v = __fmul_rn(__fmul_rn(sm.C(i, j), ri), sm.inv[j]);
          sm.C(i, j) = v;
          if (j & 1) acc1 = __fadd_rn(acc1, v);
          else acc0 = __fadd_rn(acc0, v);
        }
      }
      a[h] = __fdiv_rn(__fadd_rn(acc0, acc1), (float)n);
    }
    }
    __syncwarp();

    // ---- exact path: per-row data (exponent range, exact G_ii) made when a
    // close call first needs the row; bit r of `ready` marks row r
    unsigned long long ready = 0ull;  // the same on every lane
    auto ensure = [&](int r) {
      if ((ready >> r) & 1ull) return;
      const uint4* x = row(r);
      int emin = INT_MAX, emax = INT_MIN;
#pragma unroll
      for (int q = 0; q < kD / 32; ++q) {
        int sig, e, neg, nf;
        decode_bf16(elem(x, lane + 32 * q), sig, e, neg, nf);
        if (sig != 0 && !nf) {
          emin = min(emin, e);
          emax = max(emax, e);
        }
      }
      emin = __reduce_min_sync(kFull, emin);
      emax = __reduce_max_sync(kFull, emax);
      if (emin == INT_MAX) emin = emax = 0;
      const bool wide = emax - emin > 20;
      const double d = exact_dot_warp(x, x, emin, emin, wide);
      if (lane == 0) {
        sm.emin[r] = emin;
        sm.emax[r] = emax;
        sm.wide[r] = wide;
        sm.diag[r] = d;
      }
      __syncwarp();
      ready |= 1ull << r;
    };
    // the float64 cosine of the reference arithmetic; cos64 by one lane (rows
    // ready), cos64w by the whole warp
    auto cos64 = [&](int i, int j) -> double {
      const double gii = sm.diag[i], gjj = sm.diag[j];
      if (gii == 0.0 || gjj == 0.0) return 0.0;
      const double g = exact_dot(row(i), row(j), sm.emin[i], sm.emin[j], sm.wide[i] | sm.wide[j]);
      return __ddiv_rn(g, __dsqrt_rn(__dmul_rn(gii, gjj)));
    };
    auto cos64w = [&](int i, int j) -> double {
      ensure(i);
      ensure(j);
      const double gii = sm.diag[i], gjj = sm.diag[j];
      if (gii == 0.0 || gjj == 0.0) return 0.0;
      const double g = exact_dot_warp(row(i), row(j), sm.emin[i], sm.emin[j], sm.wide[i] | sm.wide[j]);
      return __ddiv_rn(g, __dsqrt_rn(__dmul_rn(gii, gjj)));
    };

    // ---- Algorithm 1
    const int i0 = lane, i1 = lane + 32;
    const bool live0 = i0 < n, live1 = NH > 1 && i1 < n;
    // exact mean cosine of candidate i: lanes evaluate cos64(i, j) for their j,
    // every lane sums them left to right
    auto mean64 = [&](int i) -> double {
      for (int r = 0; r < n; ++r) ensure(r);
      for (int j = lane; j < n; j += 32) sm.v64[j] = cos64(i, j);
      __syncwarp();
      double acc = 0.0;
      for (int j = 0; j < n; ++j) acc = __dadd_rn(acc, sm.v64[j]);
      __syncwarp();
      return __ddiv_rn(acc, (double)n);
    };
    const int p0 = filtered_argmin(sm.cand, a[0], NH > 1 ? a[NH - 1] : 0.f, live0, live1, kMeanErr, mean64);
    if (lane == 0) sm.picks[0] = p0;
    bool ch0 = i0 == p0, ch1 = i1 == p0;
    float S0 = live0 ? sm.C(i0, p0) : 0.f, S1 = live1 ? sm.C(i1, p0) : 0.f;
    for (int k = 1; k < m; ++k) {
      // exact running maximum of candidate j over the picks so far: only the
      // picks whose float32 cosine lies within twice the bound of the float32
      // maximum can hold it (every other one is below that pick's float64 value)
      auto smax64 = [&](int j) -> double {
        float c32 = -kInfF;
        for (int q = lane; q < k; q += 32) c32 = fmaxf(c32, sm.C(j, sm.picks[q]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c32 = fmaxf(c32, __shfl_xor_sync(kFull, c32, off));
        const float lim = c32 - 2.0f * kCosErr;
        double v = -__longlong_as_double(0x7ff0000000000000LL);
        for (int q0 = 0; q0 < k; q0 += 32) {
          const int q = q0 + lane;
          unsigned near = __ballot_sync(kFull, q < k && !(sm.C(j, sm.picks[q]) < lim));
          while (near) {
            const int qq = q0 + __ffs(near) - 1;
            near &= near - 1;
            const double c = cos64w(j, sm.picks[qq]);
            v = c > v ? c : v;
          }
        }
        return v;
      };
      __syncwarp();
      const int r = filtered_argmin(sm.cand, S0, S1, live0 && !ch0, live1 && !ch1, kCosErr, smax64);
      if (i0 == r) ch0 = true;
      if (i1 == r) ch1 = true;
      if (live0) S0 = fmaxf(S0, sm.C(i0, r));
      if (live1) S1 = fmaxf(S1, sm.C(i1, r));
      if (lane == 0) sm.picks[k] = r;
    }
    __syncwarp();
    for (int k = lane; k < m; k += 32)
      if (BKV_IN_RANGE(sm.picks[k] >= 0 && sm.picks[k] < n, P.status)) trace[k] = (int8_t)sm.picks[k];
    const unsigned m0 = __ballot_sync(kFull, ch0), m1 = __ballot_sync(kFull, ch1);
    const unsigned lt = (1u << lane) - 1u;
    if (ch0) sm.keep_src[__popc(m0 & lt)] = i0;
    if (ch1) sm.keep_src[__popc(m0) + __popc(m1 & lt)] = i1;
  } else {
    // nothing to sample: every candidate is kept in order
    for (int k = lane; k < m; k += 32) trace[k] = k < n ? (int8_t)k : (int8_t)-1;
    if (lane < n) sm.keep_src[lane] = lane;
  }
  __syncwarp();

  {
    // ---- kept rows back into the beacon buffer (m <= 31 rows of 16 uint4).
    // Rows held in shared memory as loaded are copied from there; otherwise
    // every source row is read again and staged before any is overwritten:
    // NH == 1 in this warp's operand rows (its product is done; the other
    // warps' products only read them into rows of D nobody reads), NH == 2 in
    // the cosines
    const int kept = n < m ? n : m;
    if (raw_rows) {
#pragma unroll 4
      for (int q = 0; q < 16; ++q) {
        const int idx = lane + 32 * q, src = sm.keep_src[idx >> 4], part = idx & 15;
        if (idx < kept * 16 && BKV_IN_RANGE(src >= 0 && src < n, P.status)) {
          if constexpr (NH == 1)
            bq[idx] = *reinterpret_cast<const uint4*>(opnd + (part >> 3) * kSlabBytes + (32 * warp + src) * 128 +
                                                      (((part & 7) ^ (src & 7)) << 4));
          else
            bq[idx] = *reinterpret_cast<const uint4*>(sm.y + src * kYStride + part * 8);
        }
      }
    } else {
      auto stage = [&](int idx) -> uint4* {
        if constexpr (NH == 1)
          return reinterpret_cast<uint4*>(opnd + (idx >> 8) * kSlabBytes + 32 * warp * 128) + (idx & 255);
        else
          return reinterpret_cast<uint4*>(sm.c) + idx;
      };
#pragma unroll 4
      for (int q = 0; q < 16; ++q) {
        const int idx = lane + 32 * q;
        if (idx < kept * 16 && BKV_IN_RANGE(sm.keep_src[idx >> 4] >= 0 && sm.keep_src[idx >> 4] < n, P.status))
          *stage(idx) = row(sm.keep_src[idx >> 4])[idx & 15];
      }
      __syncwarp();
#pragma unroll 4
      for (int q = 0; q < 16; ++q) {
        const int idx = lane + 32 * q;
        if (idx < kept * 16) bq[idx] = *stage(idx);
      }
    }
  }
  __syncwarp();  // the next head reuses this warp's rows and cosines
  }
  if (tc) {  // every warp is done reading the Gram: free its columns
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(gram_tmem, kGramCols);
  }
}

template <int NH>
cudaError_t launch_nh(const FpsParams& p, cudaStream_t s) {
  const size_t smem = fps_cta_smem<NH>();
  static std::atomic<unsigned long long> configured{0};  // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(fps_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  int64_t blocks = (p.heads_total + kHeadsPerCta<NH> - 1) / kHeadsPerCta<NH>;
  if (NH == 1 && p.nb + p.nr > p.m) {  // persistent: four CTAs per SM (their TMEM columns fill the SM's 512)
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    blocks = blocks < 4LL * sms ? blocks : 4LL * sms;
  }
  fps_kernel<NH><<<(unsigned)blocks, 32 * kHeadsPerCta<NH>, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fps(const FpsParams& p, cudaStream_t s) {
  const int n = p.nb + p.nr;
  if (p.heads_total <= 0 || p.m == 0 || n <= 0) return cudaSuccess;
  if (n > kMaxCand || p.m > 31) return cudaErrorInvalidValue;
  return n <= 32 ? launch_nh<1>(p, s) : launch_nh<2>(p, s);
}

}  // namespace bkv
