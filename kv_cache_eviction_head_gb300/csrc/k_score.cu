// Fused observation-row RoPE, attention scoring and keep-set selection,
// one CTA per unit (sequence, layer, KV head).
//
// BeaconKV reading notes:
//   §2.3, Q_obs equation: beacons are rotated to the eviction step t, recent
//         queries keep their own positions tau;
//   §2.1 eq. 4: w_{r,j} = exp(q_r.k_j/sqrt d) / sum_{l accessible} exp(q_r.k_l/sqrt d),
//         where a recent row at tau reaches the keys at positions <= tau;
//   §2.3 eq. 7: Score[j] = max over every query head of the group and every
//         observation row of w_{r,j};
//   §2.3 eq. 8: I_final = Sort(prefix + recent window + TopK(Score, k_sel)).
//
// Score[j] = exp(max_r (l_rj - lse_r)), lse_r the row's log-sum-exp: the max of
// the weights is the exp of the max of the log-weights. Two passes over the
// unit's keys, both on bf16 tensor-core tiles with fp32 accumulation: pass 1
// keeps an online (max, sum) per observation row, pass 2 recomputes the logits
// and max-reduces l - lse down each key's column. The second pass re-reads the
// unit's K slice right after the first, so it is served from L2.
//
// Selection drops the D = L - budget lowest-scoring candidates among slots
// [prefix, L - recent); among equal scores the higher slot is dropped first,
// so the lower slot wins a tie. A 4 x 8-bit radix select over the fp32 score
// bits (scores are >= 0, so the bit patterns order like the values) finds the
// D-th smallest score, then block scans place the kept slots in order.
#include "bkv_internal.cuh"

namespace bkv {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileKeys = 128;                // keys per K tile
constexpr int kRowBytes = kD * 2;             // 256 bytes per bf16 row
constexpr int kTileBytes = kTileKeys * kRowBytes;
constexpr float kLog2e = 1.4426950408889634f;

// 16-byte chunk c of row r lives at chunk (c ^ (r & 7)): the 8 rows that one
// ldmatrix phase reads then sit in 8 different bank groups.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * kRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// Exclusive block-wide prefix sum; every thread also receives the total.
__device__ __forceinline__ int block_scan(int v, int* wsum, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int s = wsum[w];
    if (w < warp) base += s;
    tot += s;
  }
  __syncthreads();
  total = tot;
  return base + incl - v;
}

struct UnitGeom {
  int layer, seq, kvh;
};

__device__ __forceinline__ UnitGeom unit_geom(int u, int batch, int kv_heads) {
  UnitGeom g;
  g.kvh = u % kv_heads;
  g.seq = (u / kv_heads) % batch;
  g.layer = u / (kv_heads * batch);
  return g;
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 2) score_select_kernel(const __grid_constant__ ScoreParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  const float kNegInf = __int_as_float(0xff800000u);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int u = blockIdx.x;
  const UnitGeom ug = unit_geom(u, P.batch, P.kv_heads);
  const int per_head = P.nb + P.nr;
  const int R = P.group * per_head;
  const int Rp = (R + 15) & ~15;
  const int L = P.L;
  const int ntiles = (L + kTileKeys - 1) / kTileKeys;
  const int Lp = ntiles * kTileKeys;

  unsigned char* qs = smem;                                  // [Rp][256 B]
  unsigned char* ks = qs + Rp * kRowBytes;                   // [2][128][256 B]
  float* sc = reinterpret_cast<float*>(ks + 2 * kTileBytes); // [Lp]
  float* lse = sc + Lp;                                      // [Rp] (log2 units)
  int* lim = reinterpret_cast<int*>(lse + Rp);               // [Rp] exclusive key bound
  int* wsum = lim + Rp;                                      // [kWarps]
  unsigned* hist = reinterpret_cast<unsigned*>(wsum + kWarps);  // [256]
  int* sel = reinterpret_cast<int*>(hist + 256);             // [4]

  const __nv_bfloat16* kbase =
      P.K[ug.layer] + ((size_t)(ug.seq * P.kv_heads + ug.kvh) * P.max_cache) * kD;
  const int64_t head0 = ((int64_t)ug.layer * P.batch + ug.seq) * (P.kv_heads * P.group) +
                        (int64_t)ug.kvh * P.group;

  // ---- K tile loader: sequence index s covers pass 1 (s < ntiles) then pass 2
  auto load_tile = [&](int s) {
    const int kt = s % ntiles;
    const uint32_t dst0 = smem_u32(ks + (s & 1) * kTileBytes);
#pragma unroll
    for (int it = 0; it < (kTileKeys * 16) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int row = idx >> 4, ch = idx & 15;
      const int key = kt * kTileKeys + row;
      const bool ok = key < L;
      const __nv_bfloat16* src = kbase + (size_t)(ok ? key : 0) * kD + ch * 8;
      cp_async16(dst0 + swz(row, ch), src, ok ? 16 : 0);
    }
    cp_async_commit();
  };
  load_tile(0);

  // ---- observation rows: RoPE in fp32 from the fp64-derived table, rounded to bf16
  for (int idx = tid; idx < Rp * 8; idx += kThreads) {
    const int r = idx >> 3, part = idx & 7;
    uint4 lo_out = make_uint4(0, 0, 0, 0), hi_out = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int gi = r / per_head, w = r % per_head;
      const int64_t hq = head0 + gi;
      const uint4* src;
      int prow;
      if (w < P.nb) {
        src = P.bq + (hq * P.fps_cap + w) * 16;
        prow = 0;
      } else {
        const int k = w - P.nb;
        src = P.rq + (hq * P.n_rq + (P.ring_first + k) % P.n_rq) * 16;
        prow = 1 + k;
      }
      const uint4 xl = src[part], xh = src[part + 8];
      const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&xl);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&xh);
      __nv_bfloat162* lo2 = reinterpret_cast<__nv_bfloat162*>(&lo_out);
      __nv_bfloat162* ho2 = reinterpret_cast<__nv_bfloat162*>(&hi_out);
      const float2* cs = P.rope + prow * kRopePairs + part * 8;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = __bfloat1622float2(l2[e]), b = __bfloat1622float2(h2[e]);
        const float2 c0 = cs[2 * e], c1 = cs[2 * e + 1];
        lo2[e] = __floats2bfloat162_rn(a.x * c0.x - b.x * c0.y, a.y * c1.x - b.y * c1.y);
        ho2[e] = __floats2bfloat162_rn(b.x * c0.x + a.x * c0.y, b.y * c1.x + a.y * c1.y);
      }
    }
    *reinterpret_cast<uint4*>(qs + swz(r, part)) = lo_out;
    *reinterpret_cast<uint4*>(qs + swz(r, part + 8)) = hi_out;
  }
  for (int r = tid; r < Rp; r += kThreads) {
    int bound = 0;
    if (r < R) {
      const int w = r % per_head;
      bound = w < P.nb ? L : L - P.nr + (w - P.nb) + 1;
    }
    lim[r] = bound;
  }

  const float qk_scale = kLog2e * rsqrtf((float)kD);  // logits in log2 units
  const int mtiles = Rp / 16;
  const int g = lane >> 2, c2 = (lane & 3) * 2;

  // pass-1 running statistics: up to 2 m-tiles per warp, rows g and g + 8
  float run_m[2][2], run_z[2][2];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      run_m[a][b] = kNegInf;
      run_z[a][b] = 0.f;
    }

  for (int s = 0; s < 2 * ntiles; ++s) {
    if (s + 1 < 2 * ntiles) {
      load_tile(s + 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t kb = smem_u32(ks + (s & 1) * kTileBytes);
    const uint32_t qb = smem_u32(qs);
    const int kt = s % ntiles;

    if (s < ntiles) {
      // ---------------- pass 1: warp owns m-tiles warp, warp + 8
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int mt = warp + mi * kWarps;
        if (mt >= mtiles) break;
        const int r0 = mt * 16 + g, r1 = r0 + 8;
        const int lim0 = lim[r0], lim1 = lim[r1];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float acc[8][4];
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            uint32_t a[4];
            ldsm_x4(qb + swz(mt * 16 + (lane & 15), kk * 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
              const int key = half * 64 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
              uint32_t b0, b1, b2, b3;
              ldsm_x4(kb + swz(key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
              mma_bf16(acc[np * 2], a, b0, b1);
              mma_bf16(acc[np * 2 + 1], a, b2, b3);
            }
          }
          const int jb = kt * kTileKeys + half * 64 + c2;
          float tm0 = kNegInf, tm1 = kNegInf;
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = jb + i * 8 + e;
              acc[i][e] = j < lim0 ? acc[i][e] * qk_scale : kNegInf;
              acc[i][2 + e] = j < lim1 ? acc[i][2 + e] * qk_scale : kNegInf;
              tm0 = fmaxf(tm0, acc[i][e]);
              tm1 = fmaxf(tm1, acc[i][2 + e]);
            }
          float nm0 = fmaxf(run_m[mi][0], tm0), nm1 = fmaxf(run_m[mi][1], tm1);
          float z0 = nm0 == kNegInf ? 0.f : run_z[mi][0] * fast_exp2(run_m[mi][0] - nm0);
          float z1 = nm1 == kNegInf ? 0.f : run_z[mi][1] * fast_exp2(run_m[mi][1] - nm1);
          if (nm0 != kNegInf) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
              for (int e = 0; e < 2; ++e) z0 += fast_exp2(acc[i][e] - nm0);
          }
          if (nm1 != kNegInf) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
              for (int e = 0; e < 2; ++e) z1 += fast_exp2(acc[i][2 + e] - nm1);
          }
          run_m[mi][0] = nm0;
          run_m[mi][1] = nm1;
          run_z[mi][0] = z0;
          run_z[mi][1] = z1;
        }
      }
      if (s == ntiles - 1) {
        // combine the four lanes that share each row, then lse = m + log2(z)
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          const int mt = warp + mi * kWarps;
          if (mt >= mtiles) break;
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            float mm = run_m[mi][hr], zz = run_z[mi][hr];
#pragma unroll
            for (int off = 1; off < 4; off <<= 1) {
              const float om = __shfl_xor_sync(0xFFFFFFFFu, mm, off);
              const float oz = __shfl_xor_sync(0xFFFFFFFFu, zz, off);
              const float nm = fmaxf(mm, om);
              if (nm != kNegInf) {
                zz = (mm == kNegInf ? 0.f : zz * fast_exp2(mm - nm)) +
                     (om == kNegInf ? 0.f : oz * fast_exp2(om - nm));
              }
              mm = nm;
            }
            if ((lane & 3) == 0) lse[mt * 16 + g + hr * 8] = zz > 0.f ? mm + fast_log2(zz) : kNegInf;
          }
        }
      }
    } else {
      // ---------------- pass 2: warp owns keys [warp * 16, warp * 16 + 16) of the tile
      float cm[2][2] = {{kNegInf, kNegInf}, {kNegInf, kNegInf}};
      for (int mt = 0; mt < mtiles; ++mt) {
        float acc[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t a[4];
          ldsm_x4(qb + swz(mt * 16 + (lane & 15), kk * 2 + (lane >> 4)), a[0], a[1], a[2], a[3]);
          const int key = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz(key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_bf16(acc[0], a, b0, b1);
          mma_bf16(acc[1], a, b2, b3);
        }
        const int r0 = mt * 16 + g, r1 = r0 + 8;
        const int lim0 = lim[r0], lim1 = lim[r1];
        const float l0 = lse[r0], l1 = lse[r1];
        const int jb = kt * kTileKeys + warp * 16 + c2;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = jb + i * 8 + e;
            if (j < lim0) cm[i][e] = fmaxf(cm[i][e], acc[i][e] * qk_scale - l0);
            if (j < lim1) cm[i][e] = fmaxf(cm[i][e], acc[i][2 + e] * qk_scale - l1);
          }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = cm[i][e];
          v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 16));
          cm[i][e] = v;
        }
      if (lane < 4) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = kt * kTileKeys + warp * 16 + i * 8 + c2 + e;
            sc[j] = cm[i][e] == kNegInf ? 0.f : fast_exp2(cm[i][e]);
          }
      }
    }
    __syncthreads();
  }

  // ---------------- keep-set selection over the scores in shared memory
  const int c0 = P.prefix < L ? P.prefix : L;
  const int c1 = L - P.recent > c0 ? L - P.recent : c0;
  const int D = L - P.budget;  // candidates to drop, 1 <= D <= c1 - c0

  bool bad = false;
  for (int j = tid; j < L; j += kThreads) bad |= sc[j] != sc[j];
  if (__syncthreads_or(bad) && tid == 0) latch(P.status, BKV_ERR_NONFINITE);

  uint32_t want = 0, mask = 0;
  int k = D;
  for (int shift = 24; shift >= 0; shift -= 8) {
    hist[tid] = 0;
    __syncthreads();
    for (int j = c0 + tid; j < c1; j += kThreads) {
      const uint32_t key = __float_as_uint(sc[j]);
      if ((key & mask) == want) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      int cnt = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) cnt += (int)hist[lane * 8 + b];
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
      }
      const int excl = incl - cnt;
      if (excl < k && k <= incl) {
        int cum = excl;
        for (int b = 0; b < 8; ++b) {
          const int hb = (int)hist[lane * 8 + b];
          if (cum + hb >= k) {
            sel[0] = lane * 8 + b;
            sel[1] = k - cum;
            sel[2] = hb;
            break;
          }
          cum += hb;
        }
      }
    }
    __syncthreads();
    want |= (uint32_t)sel[0] << shift;
    mask |= 0xFFu << shift;
    k = sel[1];
    __syncthreads();
  }
  const uint32_t T = want;      // the D-th smallest score bits
  const int n_eq = sel[2];      // candidates whose score equals T
  const int keep_eq = n_eq - k; // the lowest-slot keep_eq of them stay

  const int chunk = (L + kThreads - 1) / kThreads;  // <= 32 (L <= 8192)
  const int j0 = min(tid * chunk, L), j1 = min(j0 + chunk, L);
  int my_eq = 0;
  for (int j = j0; j < j1; ++j)
    if (j >= c0 && j < c1 && __float_as_uint(sc[j]) == T) ++my_eq;
  int dummy;
  int eq_rank = block_scan(my_eq, wsum, dummy);
  uint32_t keepbits = 0;
  int my_keep = 0;
  for (int j = j0; j < j1; ++j) {
    bool keep = true;
    if (j >= c0 && j < c1) {
      const uint32_t key = __float_as_uint(sc[j]);
      if (key < T) keep = false;
      else if (key == T) keep = eq_rank++ < keep_eq;
    }
    if (keep) {
      keepbits |= 1u << (j - j0);
      ++my_keep;
    }
  }
  int total;
  int dst = block_scan(my_keep, wsum, total);
  if (total != P.budget) {
    if (tid == 0) latch(P.status, BKV_ERR_INTERNAL);
  } else {
    int32_t* out = P.kept + (size_t)u * P.budget;
    for (int j = j0; j < j1; ++j)
      if (keepbits >> (j - j0) & 1u) out[dst++] = j;
  }
  if (P.scores) {
    float* so = P.scores + (size_t)u * P.max_cache;
    for (int j = tid; j < L; j += kThreads) so[j] = sc[j];
  }
}

size_t score_smem_bytes(int R, int L) {
  const int Rp = (R + 15) & ~15;
  const int Lp = (L + kTileKeys - 1) / kTileKeys * kTileKeys;
  return (size_t)Rp * kRowBytes + 2 * (size_t)kTileBytes + (size_t)Lp * 4 + (size_t)Rp * 8 +
         kWarps * 4 + 256 * 4 + 16;
}

cudaError_t launch_score_select(const ScoreParams& p, cudaStream_t s) {
  const size_t smem = score_smem_bytes(p.group * (p.nb + p.nr), p.L);
  static size_t configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(score_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  score_select_kernel<<<p.units, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
