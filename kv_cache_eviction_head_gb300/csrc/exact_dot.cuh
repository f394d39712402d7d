// Exact dot products of bf16 vectors, rounded once to float64: the
// arithmetic that makes FPS picks and coverage values bit-reproducible
// (BeaconKV reading notes §2.2: cosine similarity of pre-RoPE queries).
// Used by the FPS and coverage kernels; internal linkage in each unit.
#pragma once

#include <cstdint>

#include "bkv_internal.cuh"

namespace bkv {
namespace {

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

// Exact dot product of two bf16 rows, rounded once to float64; emin_* are the
// rows' smallest nonzero exponents (used when neither row is wide).
__device__ double exact_dot(const uint4* xi, const uint4* xj, int emin_i, int emin_j, bool wide) {
  if (wide) return exact_dot_wide(xi, xj);
  long long acc = 0;
  for (int k = 0; k < kD; ++k) {
    int sa, ea, na, fa, sb, eb, nbv, fb;
    decode_bf16(elem(xi, k), sa, ea, na, fa);
    decode_bf16(elem(xj, k), sb, eb, nbv, fb);
    if (sa == 0 || sb == 0 || fa || fb) continue;
    const long long p = (long long)(sa << (ea - emin_i)) * (long long)(sb << (eb - emin_j));
    acc += (na ^ nbv) ? -p : p;
  }
  return acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(emin_i + emin_j));
}

// exact_dot evaluated by a whole warp on one pair of rows (every lane passes
// the same arguments and gets the same result): lane l takes elements
// l, l + 32, l + 64, l + 96, and the exact 64-bit integer partial sums are
// added exactly across the warp before the one rounding, so the value is
// exact_dot's, bit for bit. Wide pairs take exact_dot_wide on every lane.
__device__ double exact_dot_warp(const uint4* xi, const uint4* xj, int emin_i, int emin_j, bool wide) {
  if (wide) return exact_dot_wide(xi, xj);
  const int lane = threadIdx.x & 31;
  long long acc = 0;
#pragma unroll
  for (int q = 0; q < kD / 32; ++q) {
    const int k = lane + 32 * q;
    int sa, ea, na, fa, sb, eb, nbv, fb;
    decode_bf16(elem(xi, k), sa, ea, na, fa);
    decode_bf16(elem(xj, k), sb, eb, nbv, fb);
    if (sa == 0 || sb == 0 || fa || fb) continue;
    const long long p = (long long)(sa << (ea - emin_i)) * (long long)(sb << (eb - emin_j));
    acc += (na ^ nbv) ? -p : p;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  return acc == 0 ? 0.0 : __dmul_rn(__ll2double_rn(acc), pow2(emin_i + emin_j));
}

}  // namespace
}  // namespace bkv
