// Decode-step query push and the per-eviction RoPE table.
//
// Push (BeaconKV reading notes, §2.2 eq. 9 and Algorithm 2): each query head
// keeps its recent queries in a ring of n_rq slots indexed by step % n_rq. When
// the ring is full, the slot about to be overwritten holds the oldest recent
// query, which moves to the end of the beacon buffer first. FPS of a full
// beacon buffer is a separate launch (k_fps.cu).
#include "bkv_internal.cuh"

namespace bkv {

// One thread per 16-byte chunk: 16 threads per query head row.
__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t head = gid >> 4;
  const int part = (int)(gid & 15);
  if (head >= p.heads_total) return;
  uint4* ring = p.rq + (head * p.n_rq + p.slot) * 16 + part;
  if (p.spill) p.bq[(head * p.fps_cap + p.nb) * 16 + part] = *ring;
  *ring = p.q[head * 16 + part];
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
  const int64_t threads = p.heads_total * 16;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  append_kernel<<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// Row r of the table holds, for pair i < d/2, (cos, sin) of pos_r * theta^(-2i/d):
// pos_0 = t (beacons are rotated to the eviction step), pos_{1+k} = t - nr + 1 + k
// (the k-th oldest recent query keeps its own position). Angles and their
// sines/cosines are evaluated in fp64 once per eviction, then rounded to fp32.
__global__ void rope_table_kernel(RopeParams p) {
  const int row = blockIdx.x;
  const int i = threadIdx.x;
  if (i >= kRopePairs) return;
  const int64_t pos = row == 0 ? p.t : p.t - p.nr + row;
  const double inv_freq = pow(p.theta, -2.0 * (double)i / (double)kD);
  const double ang = (double)pos * inv_freq;
  double sn, cs;
  sincos(ang, &sn, &cs);
  p.tab[row * kRopePairs + i] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(const RopeParams& p, cudaStream_t s) {
  rope_table_kernel<<<1 + p.nr, kRopePairs, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace bkv
