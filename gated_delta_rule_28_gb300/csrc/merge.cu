// Ordered merge of affine segment summaries (sm_103a).
//
// S_init_0 = h0 (or 0), S_init_{s+1} = M_s S_init_s + S_ext_s, all fp32
// (apply_kda_state_summary on the hyper-parallel "Diff Coverage" page, which
// keeps the communicated state in fp32 with autocast off; SANA
// distributed_scan.py _exclusive_prefix_compose). One CTA per (batch row and
// head, 32 state columns); the K x K transfer of each segment is staged in
// shared memory and applied with fp32 FMA.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int BV = 32;
constexpr int NTH = 256;
constexpr int MP = GDN_DK + 1;
constexpr int VP = BV + 1;

__global__ void __launch_bounds__(NTH) merge_kernel(MergeArgs a) {
  extern __shared__ float smem[];
  float *sM = smem;              // [128][MP]
  float *sS = sM + GDN_DK * MP;  // [128][VP]
  const int tid = threadIdx.x;
  const int col0 = blockIdx.x * BV;
  const int64_t bh = blockIdx.y;
  const int64_t KV = (int64_t)GDN_DK * GDN_DV;

  for (int idx = tid; idx < GDN_DK * BV; idx += NTH) {
    const int d = idx / BV, c = idx % BV;
    sS[d * VP + c] = a.h0 ? a.h0[bh * KV + d * GDN_DV + col0 + c] : 0.f;
  }
  __syncthreads();
  int m0, n0;
  tile_origin<128, BV, 4, 4>(tid, m0, n0);
  for (int s = 0; s < a.nseg; ++s) {
    const int64_t slot = bh * a.nseg + s;
    for (int idx = tid; idx < GDN_DK * BV; idx += NTH) {
      const int d = idx / BV, c = idx % BV;
      a.S_init[slot * KV + d * GDN_DV + col0 + c] = sS[d * VP + c];
    }
    const float *Ms = a.M + slot * GDN_DK * GDN_DK;
    for (int idx = tid; idx < GDN_DK * GDN_DK; idx += NTH) sM[(idx >> 7) * MP + (idx & 127)] = Ms[idx];
    __syncthreads();
    float acc[4][4];
    zero_acc(acc);
    auto fa = [&](int m, int kk) { return sM[m * MP + kk]; };
    auto fb = [&](int kk, int nn) { return sS[kk * VP + nn]; };
    mm_acc<128, BV, GDN_DK, 4, 4>(fa, fb, acc, tid);
    __syncthreads();
    const float *Es = a.S_ext + slot * KV;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y)
        sS[(m0 + x) * VP + n0 + y] = acc[x][y] + Es[(m0 + x) * GDN_DV + col0 + n0 + y];
    __syncthreads();
  }
  if (a.ht) {
    for (int idx = tid; idx < GDN_DK * BV; idx += NTH) {
      const int d = idx / BV, c = idx % BV;
      a.ht[bh * KV + d * GDN_DV + col0 + c] = sS[d * VP + c];
    }
  }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t st) {
  const size_t bytes = (size_t)(GDN_DK * MP + GDN_DK * VP) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)bytes);
  if (e != cudaSuccess) return e;
  merge_kernel<<<dim3(GDN_DV / BV, a.BH), NTH, bytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
