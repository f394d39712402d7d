// Fused observation-row RoPE, attention scoring and keep-set selection on the
// fifth-generation tensor cores (tcgen05, TMEM accumulators, TMA loads).
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
// Score[j] = exp(max_r (l_rj - lse_r)), lse_r the row's log-sum-exp (the max of
// the weights is the exp of the max of the log-weights). Per unit (sequence,
// layer, KV head) the K slice streams through shared memory twice: pass 1
// keeps an online (max, sum) per observation row, pass 2 recomputes the
// logits and takes each key's max of l - lse. The second read of the slice
// follows the first at once and is served from L2.
//
// Precision: the rotated observation rows are split into bf16 hi + lo parts
// (residual below 2^-17 relative); both parts multiply the bf16 keys on the
// tensor cores into one fp32 accumulator, so a logit's error stays far below
// the 2e-3 score tolerance even for large logits.
//
// Structure: one persistent CTA per SM walks the units; its warps specialise.
//   warp 0   TMA producer: two 128-row x 64-column SWIZZLE_128B boxes per
//            128-key tile into a ring of shared-memory stages;
//   warp 1   TMEM owner and single-thread MMA issuer:
//              pass 1  D[row][key] = Q . K_tile^T   (M = 128 rows, N = 128 keys)
//              pass 2  D[key][row] = K_tile . Q^T   (M = 128 keys, N = rows)
//            so each epilogue thread owns one TMEM lane (a row in pass 1, a
//            key in pass 2) and reduces along its own registers only;
//   warp 2   builds the next unit's rotated rows while the tensor cores finish
//            the current unit;
//   warp 3   selects the keep set of a finished unit from its scores;
//   warps 4-7  epilogue: TMEM -> registers, online log-sum-exp in pass 1,
//            max-pooling in pass 2, scores to shared memory.
// Every cross-warp wait is a bounded wait on an mbarrier; on expiry the kernel
// latches BKV_ERR_TIMEOUT, every role stops at its next wait, outstanding
// copies are drained and the TMEM is freed before the CTA exits.
//
// Selection drops the D = L - budget lowest-scoring candidates among slots
// [prefix, L - recent); among equal scores the higher slot is dropped first,
// so the lower slot wins a tie. A 4 x 8-bit radix select over the fp32 score
// bits (scores are >= 0, so the bit patterns order like the values) finds the
// D-th smallest score, then a scan places the kept slots in order.
#include "bkv_internal.cuh"

namespace bkv {

namespace {

constexpr int kThreads = 256;
constexpr int kTileKeys = 128;
constexpr int kSlabBytes = kTileKeys * 128;   // 128 rows x 64 bf16: one SWIZZLE_128B box
constexpr int kTileBytes = 2 * kSlabBytes;    // 32 KB per 128-key tile
constexpr int kEpiThreads = 128;              // warps 4-7
constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s: far beyond any legitimate wait
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

struct Ctl {
  volatile int abort;  // raised by the first role whose wait ran out
  uint32_t tmem_base;
};

// Bounded wait for the phase with the given parity. Returns false (after
// latching the timeout and raising the abort flag) if it never completes, or
// as soon as another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, Ctl* ctl, uint32_t* status) {
  if (mbar_test(b, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(b, parity)) {
    if (ctl->abort) return false;
    if (clock64() - t0 > kWaitCycles) {
      latch(status, BKV_ERR_TIMEOUT);
      ctl->abort = 1;
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// 32 TMEM lanes x 32 consecutive 32-bit columns: thread t of the warp reads
// lane (lane base of its warp quarter) + t into 32 registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand in the canonical
// SWIZZLE_128B layout: 8-row groups of 128-byte rows, 1024 bytes apart (SBO);
// descriptor version 1; layout type 2 = SWIZZLE_128B. Moving along K inside
// the 128-byte swizzle atom advances the start address by 32 bytes per 16
// bf16 elements.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
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

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// Keep set of one unit from its scores sc[0, L), written ascending to out.
// One warp. Returns false if the kept count came out wrong (never expected).
__device__ bool select_keep(const float* sc, int L, int prefix, int recent, int budget, int32_t* out,
                            unsigned* hist) {
  const int lane = threadIdx.x & 31;
  const int c0 = prefix < L ? prefix : L;
  const int c1 = L - recent > c0 ? L - recent : c0;
  uint32_t want = 0, mask = 0;
  int k = L - budget;  // rank (1-based) of the threshold among the candidates
  int n_eq = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = lane; b < 256; b += 32) hist[b] = 0;
    __syncwarp();
    for (int j = c0 + lane; j < c1; j += 32) {
      const uint32_t key = __float_as_uint(sc[j]);
      if ((key & mask) == want) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncwarp();
    int cnt = 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) cnt += (int)hist[lane * 8 + b];
    const int incl = warp_incl_scan(cnt, lane);
    const int excl = incl - cnt;
    const unsigned hit = __ballot_sync(kFull, excl < k && k <= incl);
    const int src = hit ? __ffs(hit) - 1 : 0;
    int digit = 0, kk = k, hb_sel = 0;
    if (lane == src) {
      int cum = excl;
      for (int b = 0; b < 8; ++b) {
        const int hb = (int)hist[lane * 8 + b];
        if (cum + hb >= k) {
          digit = lane * 8 + b;
          kk = k - cum;
          hb_sel = hb;
          break;
        }
        cum += hb;
      }
    }
    digit = __shfl_sync(kFull, digit, src);
    k = __shfl_sync(kFull, kk, src);
    n_eq = __shfl_sync(kFull, hb_sel, src);
    want |= (uint32_t)digit << shift;
    mask |= 0xFFu << shift;
    __syncwarp();
  }
  const uint32_t T = want;
  const int keep_eq = n_eq - k;  // the lowest-slot keep_eq candidates equal to T stay
  // lanes take contiguous slot ranges so the scans preserve slot order
  const int chunk = (L + 31) / 32;
  const int j0 = min(lane * chunk, L), j1 = min(j0 + chunk, L);
  int my_eq = 0;
  for (int j = j0; j < j1; ++j)
    if (j >= c0 && j < c1 && __float_as_uint(sc[j]) == T) ++my_eq;
  int eq_rank = warp_incl_scan(my_eq, lane) - my_eq;
  const int eq_start = eq_rank;
  int my_keep = 0;
  for (int j = j0; j < j1; ++j) {
    bool keep = true;
    if (j >= c0 && j < c1) {
      const uint32_t key = __float_as_uint(sc[j]);
      if (key < T) keep = false;
      else if (key == T) keep = eq_rank++ < keep_eq;
    }
    my_keep += keep;
  }
  const int incl = warp_incl_scan(my_keep, lane);
  const int total = __shfl_sync(kFull, incl, 31);
  if (total != budget) return false;
  int dst = incl - my_keep;
  eq_rank = eq_start;
  for (int j = j0; j < j1; ++j) {
    bool keep = true;
    if (j >= c0 && j < c1) {
      const uint32_t key = __float_as_uint(sc[j]);
      if (key < T) keep = false;
      else if (key == T) keep = eq_rank++ < keep_eq;
    }
    if (keep) out[dst++] = j;
  }
  return true;
}

struct Layout {
  int R, Rp16, mtiles, qrows;  // rows, rows rounded to 16, M tiles of 128 rows, rows allocated
  int ntiles, Lp, stages, bufcols;
  size_t q_hi, q_lo, kst, sc, lse, lim, bars, misc, total;
};

__host__ __device__ inline Layout make_layout(int R, int L) {
  Layout s;
  s.R = R;
  s.Rp16 = (R + 15) & ~15;
  s.mtiles = R > 128 ? 2 : 1;
  s.qrows = s.Rp16 > 128 ? s.Rp16 : 128;  // a second M tile covers rows [Rp16 - 128, Rp16)
  s.ntiles = (L + kTileKeys - 1) / kTileKeys;
  s.Lp = s.ntiles * kTileKeys;
  s.bufcols = (s.mtiles > 1 || s.Rp16 > 128) ? 256 : 128;
  const size_t qbytes = ((size_t)s.qrows * 256 + 1023) / 1024 * 1024;  // two 128-byte slabs per row
  size_t off = 0;
  s.q_hi = off;
  off += qbytes;
  s.q_lo = off;
  off += qbytes;
  s.kst = off;  // 1024-aligned
  const size_t tail = 2 * (size_t)s.Lp * 4 + (size_t)s.qrows * 8 + 64 * 8 + 2048;
  const size_t cap = 227 * 1024 - 1024;  // 1 KB kept for aligning the dynamic base
  const long long room = (long long)cap - (long long)off - (long long)tail;
  const int st = room > 0 ? (int)(room / kTileBytes) : 0;
  s.stages = st > 4 ? 4 : st;
  off += (size_t)s.stages * kTileBytes;
  s.sc = off;
  off += 2 * (size_t)s.Lp * 4;
  s.lse = off;
  off += (size_t)s.qrows * 4;
  s.lim = off;
  off += (size_t)s.qrows * 4;
  s.bars = (off + 7) & ~(size_t)7;
  off = s.bars + 64 * 8;
  s.misc = off;
  off += 2048;
  s.total = off + 1024;
  return s;
}

__device__ __forceinline__ void unit_geom(int u, int batch, int kv_heads, int& layer, int& seq, int& kvh) {
  kvh = u % kv_heads;
  seq = (u / kv_heads) % batch;
  layer = u / (kv_heads * batch);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1) score_select_kernel(const __grid_constant__ ScoreParams P) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_head = P.nb + P.nr;
  const Layout lay = make_layout(P.group * per_head, P.L);
  const int R = lay.R, L = P.L, T = lay.ntiles, S = lay.stages;

  unsigned char* q_hi = smem + lay.q_hi;
  unsigned char* q_lo = smem + lay.q_lo;
  unsigned char* kst = smem + lay.kst;
  float* sc = reinterpret_cast<float*>(smem + lay.sc);    // [2][Lp]
  float* lse = reinterpret_cast<float*>(smem + lay.lse);  // [qrows], log2 units
  int* lim = reinterpret_cast<int*>(smem + lay.lim);      // [qrows], exclusive key bound per row
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* kfull = bars;        // [4]
  uint64_t* kempty = bars + 4;   // [4]
  uint64_t* tfull = bars + 8;    // [2]
  uint64_t* tempty = bars + 10;  // [2]
  uint64_t* qready = bars + 12;
  uint64_t* qfree = bars + 13;
  uint64_t* sready = bars + 14;  // [2]
  uint64_t* sfree = bars + 16;   // [2]
  uint64_t* lsebar = bars + 18;
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + lay.misc);
  unsigned* hist = reinterpret_cast<unsigned*>(smem + lay.misc + 64);  // [256]

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiThreads);
      mbar_init(&sready[i], kEpiThreads);
      mbar_init(&sfree[i], 32);
    }
    mbar_init(qready, 32);
    mbar_init(qfree, 1);
    mbar_init(lsebar, kEpiThreads);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // zero both row buffers once: padding rows stay zero for the whole launch
  for (int i = tid; i < (int)(2 * (lay.q_lo - lay.q_hi) / 16); i += kThreads)
    reinterpret_cast<uint4*>(q_hi)[i] = make_uint4(0, 0, 0, 0);
  for (int r = tid; r < lay.qrows; r += kThreads) {
    int bound = 0;
    if (r < R) {
      const int w = r % per_head;
      bound = w < P.nb ? L : L - P.nr + (w - P.nb) + 1;
    }
    lim[r] = bound;
  }
  const uint32_t ncols = 2 * (uint32_t)lay.bufcols;
  if (warp == 1) tmem_alloc(&ctl->tmem_base, ncols);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int mine = P.units > (int)blockIdx.x ? (P.units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      long long g = 0;
      bool ok = true;
      for (int it = 0; it < mine && ok; ++it) {
        int layer, seq, kvh;
        unit_geom(blockIdx.x + it * gridDim.x, P.batch, P.kv_heads, layer, seq, kvh);
        const int row0 = (seq * P.kv_heads + kvh) * P.max_cache;
        for (int s = 0; s < 2 * T; ++s, ++g) {
          const int st = (int)(g % S);
          if (g >= S && !mbar_wait(&kempty[st], (uint32_t)(((g / S) + 1) & 1), ctl, P.status)) {
            ok = false;
            break;
          }
          const int kt = s % T;
          mbar_expect_tx(&kfull[st], kTileBytes);
          const uint32_t dst = smem_u32(kst + (size_t)st * kTileBytes);
          tma_load_2d(dst, &P.kmap[layer], 0, row0 + kt * kTileKeys, &kfull[st]);
          tma_load_2d(dst + kSlabBytes, &P.kmap[layer], 64, row0 + kt * kTileKeys, &kfull[st]);
        }
      }
      // drain: every load issued has landed before the CTA may exit
      for (int st = 0; st < S && st < g; ++st) {
        const long long last = g - 1 - ((g - 1 - st) % S);
        const long long t0 = clock64();
        while (!mbar_test(&kfull[st], (uint32_t)((last / S) & 1)) && clock64() - t0 < kWaitCycles) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      long long g = 0;
      bool ok = true;
      const uint32_t qh = smem_u32(q_hi), ql = smem_u32(q_lo);
      const uint32_t slab_q = (uint32_t)lay.qrows * 128;  // bytes of one 64-column slab of the rows
      const uint32_t id1 = idesc_bf16(128, 128), id2 = idesc_bf16(128, lay.Rp16);
      for (int it = 0; it < mine && ok; ++it) {
        ok = mbar_wait(qready, (uint32_t)(it & 1), ctl, P.status);
        for (int s = 0; s < 2 * T && ok; ++s, ++g) {
          const int st = (int)(g % S), b = (int)(g & 1);
          ok = mbar_wait(&kfull[st], (uint32_t)((g / S) & 1), ctl, P.status);
          if (ok && g >= 2) ok = mbar_wait(&tempty[b], (uint32_t)(((g >> 1) + 1) & 1), ctl, P.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kb = smem_u32(kst + (size_t)st * kTileBytes);
          const uint32_t d = tmem + (uint32_t)(b * lay.bufcols);
          if (s < T) {
            for (int mt = 0; mt < lay.mtiles; ++mt) {
#pragma unroll
              for (int part = 0; part < 2; ++part) {
                const uint32_t qbase = (part ? ql : qh) + (uint32_t)(mt ? lay.Rp16 - 128 : 0) * 128;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint32_t off = (uint32_t)(kk & 3) * 32;
                  const uint64_t a = sw128_desc(qbase + (uint32_t)(kk >> 2) * slab_q + off);
                  const uint64_t bd = sw128_desc(kb + (uint32_t)(kk >> 2) * kSlabBytes + off);
                  umma_bf16(d + (uint32_t)mt * 128, a, bd, id1, (part | kk) ? 1u : 0u);
                }
              }
            }
          } else {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              const uint32_t qbase = part ? ql : qh;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (uint32_t)(kk & 3) * 32;
                const uint64_t a = sw128_desc(kb + (uint32_t)(kk >> 2) * kSlabBytes + off);
                const uint64_t bd = sw128_desc(qbase + (uint32_t)(kk >> 2) * slab_q + off);
                umma_bf16(d, a, bd, id2, (part | kk) ? 1u : 0u);
              }
            }
          }
          umma_commit(&kempty[st]);
          umma_commit(&tfull[b]);
        }
        if (ok) umma_commit(qfree);  // arrives when every MMA that read this unit's rows is done
      }
      // after an abort, let the MMAs already issued finish before the TMEM is freed
      if (!ok && g > 0) {
        const long long t0 = clock64();
        while (!mbar_test(&tfull[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1)) &&
               clock64() - t0 < kWaitCycles) {
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ row builder
    const float qk_scale = kLog2e * rsqrtf((float)kD);  // rows carry 1/sqrt(d) and log2(e)
    const uint32_t slab_q = (uint32_t)lay.qrows * 128;
    for (int it = 0; it < mine; ++it) {
      if (it > 0) {  // the previous unit's MMAs must be done with the row buffers
        const bool ok = __all_sync(kFull, mbar_wait(qfree, (uint32_t)((it - 1) & 1), ctl, P.status));
        if (!ok) break;
      }
      int layer, seq, kvh;
      unit_geom(blockIdx.x + it * gridDim.x, P.batch, P.kv_heads, layer, seq, kvh);
      const int64_t head0 =
          ((int64_t)layer * P.batch + seq) * (P.kv_heads * P.group) + (int64_t)kvh * P.group;
      for (int idx = lane; idx < R * 8; idx += 32) {
        const int r = idx >> 3, part = idx & 7;
        const int gi = r / per_head, w = r % per_head;
        const int64_t hq = head0 + gi;
        const uint4* src;
        int prow;
        if (w < P.nb) {
          src = P.bq + (hq * P.fps_cap + w) * 16;
          prow = 0;
        } else {
          const int kq = w - P.nb;
          src = P.rq + (hq * P.n_rq + (P.ring_first + kq) % P.n_rq) * 16;
          prow = 1 + kq;
        }
        const uint4 xl = src[part], xh = src[part + 8];
        const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&xl);
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&xh);
        uint4 o[4];  // slab 0 hi, slab 1 hi, slab 0 lo, slab 1 lo
        __nv_bfloat162* o0 = reinterpret_cast<__nv_bfloat162*>(&o[0]);
        __nv_bfloat162* o1 = reinterpret_cast<__nv_bfloat162*>(&o[1]);
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o[2]);
        __nv_bfloat162* o3 = reinterpret_cast<__nv_bfloat162*>(&o[3]);
        const float2* cs = P.rope + prow * kRopePairs + part * 8;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = __bfloat1622float2(l2[e]), bb = __bfloat1622float2(h2[e]);
          const float2 c0 = cs[2 * e], c1 = cs[2 * e + 1];
          const float2 vl =
              make_float2((a.x * c0.x - bb.x * c0.y) * qk_scale, (a.y * c1.x - bb.y * c1.y) * qk_scale);
          const float2 vh =
              make_float2((bb.x * c0.x + a.x * c0.y) * qk_scale, (bb.y * c1.x + a.y * c1.y) * qk_scale);
          o0[e] = __float22bfloat162_rn(vl);
          o1[e] = __float22bfloat162_rn(vh);
          const float2 fl = __bfloat1622float2(o0[e]), fh = __bfloat1622float2(o1[e]);
          o2[e] = __floats2bfloat162_rn(vl.x - fl.x, vl.y - fl.y);
          o3[e] = __floats2bfloat162_rn(vh.x - fh.x, vh.y - fh.y);
        }
        const uint32_t inrow = (uint32_t)r * 128 + (uint32_t)((part ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(q_hi + inrow) = o[0];
        *reinterpret_cast<uint4*>(q_hi + slab_q + inrow) = o[1];
        *reinterpret_cast<uint4*>(q_lo + inrow) = o[2];
        *reinterpret_cast<uint4*>(q_lo + slab_q + inrow) = o[3];
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(qready);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ keep-set selector
    for (int it = 0; it < mine; ++it) {
      const int b = it & 1;
      const bool ok = __all_sync(kFull, mbar_wait(&sready[b], (uint32_t)((it >> 1) & 1), ctl, P.status));
      if (!ok) break;
      const int u = blockIdx.x + it * gridDim.x;
      const float* s_u = sc + (size_t)b * lay.Lp;
      bool bad = false;
      for (int j = lane; j < L; j += 32) bad |= s_u[j] != s_u[j];
      if (__any_sync(kFull, bad) && lane == 0) latch(P.status, BKV_ERR_NONFINITE);
      if (!select_keep(s_u, L, P.prefix, P.recent, P.budget, P.kept + (size_t)u * P.budget, hist) && lane == 0)
        latch(P.status, BKV_ERR_INTERNAL);
      if (P.scores) {
        float* so = P.scores + (size_t)u * P.max_cache;
        for (int j = lane; j < L; j += 32) so[j] = s_u[j];
      }
      __syncwarp();
      mbar_arrive(&sfree[b]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = tid - 128, q = warp - 4;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const float neg_inf = __int_as_float(0xff800000u);
    long long g = 0;
    bool ok = true;
    for (int it = 0; it < mine && ok; ++it) {
      const int b_sc = it & 1;
      float* s_u = sc + (size_t)b_sc * lay.Lp;
      float run_m[2] = {neg_inf, neg_inf}, run_z[2] = {0.f, 0.f};
      for (int s = 0; s < 2 * T; ++s, ++g) {
        const int b = (int)(g & 1);
        ok = __all_sync(kFull, mbar_wait(&tfull[b], (uint32_t)((g >> 1) & 1), ctl, P.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t col0 = tmem + lane_base + (uint32_t)(b * lay.bufcols);
        const int kt = s % T;
        if (s < T) {
          // pass 1: this thread owns observation row et (and et + 128 with a second M tile)
          for (int mt = 0; mt < lay.mtiles; ++mt) {
            const int row = mt ? lay.Rp16 - 128 + et : et;
            if (mt && row < 128) continue;  // the second tile overlaps the first on these lanes
            const int bound = lim[row] - kt * kTileKeys;  // keys [0, bound) are visible
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              float v[32];
              tmem_ld32(col0 + (uint32_t)(mt * 128 + h * 32), v);
              tmem_wait_ld();
              if (bound < (h + 1) * 32) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (h * 32 + e >= bound) v[e] = neg_inf;
              }
              float tm = v[0];
#pragma unroll
              for (int e = 1; e < 32; ++e) tm = fmaxf(tm, v[e]);
              const float nm = fmaxf(run_m[mt], tm);
              if (nm != neg_inf) {
                float z = run_m[mt] == neg_inf ? 0.f : run_z[mt] * fast_exp2(run_m[mt] - nm);
#pragma unroll
                for (int e = 0; e < 32; ++e) z += fast_exp2(v[e] - nm);
                run_z[mt] = z;
                run_m[mt] = nm;
              }
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[b]);
          if (s == T - 1) {
            for (int mt = 0; mt < lay.mtiles; ++mt) {
              const int row = mt ? lay.Rp16 - 128 + et : et;
              if (mt && row < 128) continue;
              lse[row] = run_z[mt] > 0.f ? run_m[mt] + fast_log2(run_z[mt]) : neg_inf;
            }
            mbar_arrive(lsebar);  // every row's lse is needed by every key in pass 2
            ok = __all_sync(kFull, mbar_wait(lsebar, (uint32_t)(it & 1), ctl, P.status));
            // this unit's scores go to sc[b_sc]: the selector must be done with unit it - 2
            if (ok && it >= 2)
              ok = __all_sync(kFull, mbar_wait(&sfree[b_sc], (uint32_t)(((it >> 1) + 1) & 1), ctl, P.status));
            if (!ok) break;
          }
        } else {
          // pass 2: this thread owns key j of the tile; columns are observation rows
          const int j = kt * kTileKeys + et;
          const bool masked_tile = (kt + 1) * kTileKeys > L - P.nr + 1;
          float mx = neg_inf;
          for (int c = 0; c < lay.Rp16; c += 32) {
            float v[32];
            tmem_ld32(col0 + (uint32_t)c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int r = c + e;
              if (r < R && (!masked_tile || j < lim[r])) mx = fmaxf(mx, v[e] - lse[r]);
            }
          }
          tc_fence_before();
          mbar_arrive(&tempty[b]);
          if (j < L) s_u[j] = mx == neg_inf ? 0.f : fast_exp2(mx);
          if (s == 2 * T - 1) mbar_arrive(&sready[b_sc]);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

size_t score_smem_bytes(int R, int L) {
  const Layout s = make_layout(R, L);
  return s.stages >= 2 ? s.total : (size_t)1 << 30;  // under two stages: not supported
}

bool encode_kmaps(ScoreParams& p, const void* const* K, int layers, int batch, int kv_heads,
                  int max_cache) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult qres;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qres) !=
            cudaSuccess ||
        qres != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t rows = (cuuint64_t)batch * kv_heads * max_cache;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kTileKeys};
  const cuuint32_t estr[2] = {1, 1};
  for (int l = 0; l < layers; ++l) {
    const CUresult r = encode(&p.kmap[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(K[l]),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
  }
  return true;
}

cudaError_t launch_score_select(const ScoreParams& p, cudaStream_t s) {
  const size_t smem = score_smem_bytes(p.group * (p.nb + p.nr), p.L);
  static size_t configured = 0;
  if (smem > configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(score_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  }
  const int grid = p.units < sms ? p.units : sms;
  score_select_kernel<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
