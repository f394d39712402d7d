// Device helpers shared by the score kernels: warp-role constants, bounded
// mbarrier waits, L2 cache policies, TMA and bulk copies, tcgen05 (TMEM, MMA)
// wrappers and the 64-bit key networks of the keep-set selection.
#pragma once

#include "bkv_internal.cuh"

namespace bkv {
namespace {

constexpr int kThreads = 384;
constexpr int kTileKeys = 128;
constexpr int kSlabBytes = kTileKeys * 128;   // 128 rows x 64 bf16: one SWIZZLE_128B box
constexpr int kTileBytes = 2 * kSlabBytes;    // 32 KB per 128-key tile
constexpr int kEpiThreads = 128;              // one epilogue warpgroup (warps 4-7 or 8-11)
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
// latching the timeout and raising the abort flag) if it does not complete
// within `limit` cycles, or as soon as another role has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, Ctl* ctl, uint32_t* status,
                                          long long limit = kWaitCycles) {
  if (mbar_test(b, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(b, parity)) {
    if (ctl->abort) return false;
    if (clock64() - t0 > limit) {
      latch(status, BKV_ERR_TIMEOUT);
      ctl->abort = 1;
      return false;
    }
  }
  return true;
}

// ------------------------------------------------------------------ L2 policies
// Cache-eviction priorities for the .L2::cache_hint operand of TMA and bulk
// copies: evict_last for lines a kernel reads again soon, evict_first for
// lines it streams through once.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Non-tensor bulk copies: global -> shared with an mbarrier, shared -> global
// in bulk groups.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
               ::"l"(dst), "r"(src), "r"(bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

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

// ------------------------------------------------------------------ observation rows
// Builds R rotated observation rows (BeaconKV reading notes §2.3: beacons
// rotated to the eviction step, recent queries to their own positions), each
// scaled by log2(e)/sqrt(d) and split into bf16 hi + lo, in the SWIZZLE_128B
// K-major layout of two 64-column slabs (slab_q bytes apart). rowinfo[r].x is
// the row's offset in uint4 units from bq_head (bit 30 set: from rq_head), or
// -1 for a zero padding row; rowinfo[r].y its RoPE table row. Thread t of n
// builds the 16-byte items t, t + n, ...
__device__ __forceinline__ void build_obs_rows(unsigned char* q_hi, unsigned char* q_lo, uint32_t slab_q, int R,
                                               const int2* rowinfo, const uint4* bq_head, const uint4* rq_head,
                                               const float2* rope, float qk_scale, int t, int n) {
  constexpr int kBatch = 4;  // items per thread with loads in flight together
  for (int base = 0; base < R * 8; base += n * kBatch) {
    uint4 xl[kBatch], xh[kBatch];
    int prow[kBatch];
#pragma unroll
    for (int bi = 0; bi < kBatch; ++bi) {
      const int idx = base + t + n * bi;
      xl[bi] = xh[bi] = make_uint4(0, 0, 0, 0);
      prow[bi] = 0;
      if (idx < R * 8) {
        const int2 info = rowinfo[idx >> 3];
        prow[bi] = info.y;
        if (info.x >= 0) {
          const uint4* src = ((info.x & (1 << 30)) ? rq_head : bq_head) + (info.x & ~(1 << 30));
          xl[bi] = src[idx & 7];
          xh[bi] = src[(idx & 7) + 8];
        }
      }
    }
#pragma unroll
    for (int bi = 0; bi < kBatch; ++bi) {
      const int idx = base + t + n * bi;
      if (idx >= R * 8) break;
      const int r = idx >> 3, part = idx & 7;
      const __nv_bfloat162* l2 = reinterpret_cast<const __nv_bfloat162*>(&xl[bi]);
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&xh[bi]);
      uint4 o[4];  // slab 0 hi, slab 1 hi, slab 0 lo, slab 1 lo
      __nv_bfloat162* o0 = reinterpret_cast<__nv_bfloat162*>(&o[0]);
      __nv_bfloat162* o1 = reinterpret_cast<__nv_bfloat162*>(&o[1]);
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o[2]);
      __nv_bfloat162* o3 = reinterpret_cast<__nv_bfloat162*>(&o[3]);
      const float2* cs = rope + prow[bi] * kRopePairs + part * 8;  // shared by all units: L1-resident
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = __bfloat1622float2(l2[e]), bb = __bfloat1622float2(h2[e]);
        const float2 c0 = __ldg(cs + 2 * e), c1 = __ldg(cs + 2 * e + 1);
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
  }
}

// Per-row tables of a row chunk: the exclusive key bound of each row (a recent
// row at position tau reaches keys <= tau; 0 masks padding rows) and each
// row's source (rowinfo as build_obs_rows reads it). Rows rl of the chunk are
// rows r = r0 + rl of the unit, R of them (rows64 / qrows entries written).
__device__ __forceinline__ void fill_row_tables(int* lim, int2* rowinfo, int r0, int R, int Rtot, int rows64,
                                                int qrows, int nb, int nr, int L, int fps_cap, int n_rq,
                                                int ring_first, int t, int n) {
  const int per_head = nb + nr;
  for (int rl = t; rl < rows64; rl += n) {
    const int r = r0 + rl;
    int bound = 0;
    if (rl < R && r < Rtot) {
      const int w = r % per_head;
      bound = w < nb ? L : L - nr + (w - nb) + 1;
    }
    lim[rl] = bound;
  }
  for (int rl = t; rl < qrows; rl += n) {
    const int r = r0 + rl;
    if (rl >= R || r >= Rtot) {
      rowinfo[rl] = make_int2(-1, 0);
      continue;
    }
    const int gi = r / per_head, w = r % per_head;
    if (w < nb) {
      rowinfo[rl] = make_int2((gi * fps_cap + w) * 16, 0);
    } else {
      const int kq = w - nb;
      rowinfo[rl] = make_int2(((gi * n_rq + (ring_first + kq) % n_rq) * 16) | (1 << 30), 1 + kq);
    }
  }
}

// ------------------------------------------------------------------ selection keys
// Candidate keys (score bits << 32 | ~slot): scores are >= 0, so the fp32 bit
// patterns order like the values, and among equal scores the higher slot has
// the smaller key (drops first).
constexpr int kList = 8;
typedef unsigned long long u64;
constexpr u64 kNoKey = ~0ull;

__device__ __forceinline__ void cswap(u64& a, u64& b) {
  const u64 lo = a < b ? a : b, hi = a < b ? b : a;
  a = lo;
  b = hi;
}
__device__ __forceinline__ void sort8(u64 (&k)[8]) {
  cswap(k[0], k[1]); cswap(k[2], k[3]); cswap(k[4], k[5]); cswap(k[6], k[7]);
  cswap(k[0], k[2]); cswap(k[1], k[3]); cswap(k[4], k[6]); cswap(k[5], k[7]);
  cswap(k[1], k[2]); cswap(k[5], k[6]);
  cswap(k[0], k[4]); cswap(k[1], k[5]); cswap(k[2], k[6]); cswap(k[3], k[7]);
  cswap(k[2], k[4]); cswap(k[3], k[5]);
  cswap(k[1], k[2]); cswap(k[3], k[4]); cswap(k[5], k[6]);
}
// list <- the 8 smallest of list and k, both sorted ascending
__device__ __forceinline__ void merge8(u64 (&list)[8], const u64 (&k)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) list[i] = list[i] < k[7 - i] ? list[i] : k[7 - i];  // bitonic
#pragma unroll
  for (int dd = 4; dd > 0; dd >>= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((i & dd) == 0) cswap(list[i], list[i + dd]);
}

__device__ __forceinline__ void unit_geom(int u, int batch, int kv_heads, int& layer, int& seq, int& kvh) {
  kvh = u % kv_heads;
  seq = (u / kv_heads) % batch;
  layer = u / (kv_heads * batch);
}


}  // namespace
}  // namespace bkv
