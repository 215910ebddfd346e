// Ordered merge of affine segment summaries (sm_103a).
//
// S_init_0 = h0 (or 0), S_init_{s+1} = M_s S_init_s + S_ext_s, all fp32
// (apply_kda_state_summary on the hyper-parallel "Diff Coverage" page, which
// keeps the communicated state in fp32 with autocast off; SANA
// distributed_scan.py _exclusive_prefix_compose). The adjoint (backward) merge walks the
// segments from the last to the first with the transposed maps: dS_exit_{nseg-1} = dht,
// dS_entry_s = M_s^T dS_exit_s + dS_ext_s, dS_exit_{s-1} = dS_entry_s
// (_CPAllGatherMerge.backward in SANA's distributed_scan.py).
//
// The columns of the state are independent, so one CTA owns one (batch row and
// head, 8 state columns) and walks the segments in order; its 128 threads own
// one state row each. Per segment the only dependent work is the 128 x 8 x 128
// product M_s S; the transfer maps (64 KB each) are copied two segments ahead into
// three shared-memory buffers (cp.async) while the current one is applied, and the
// local terms one segment ahead into registers. M is kept
// row-major with the 16-byte chunks of row m XOR-swizzled by m mod 32, so the 16-byte
// reads of a quarter warp (eight rows, the same columns) hit eight distinct bank groups;
// the state slice is read by all threads alike (broadcast).
#include "common.cuh"
#include "kernels.h"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tile;

constexpr int BV = 8;      // state columns per CTA
constexpr int NTH = 128;   // one thread per state row
constexpr int M_FLOATS = GDN_DK * GDN_DK;
constexpr int MSTAGES = 3;  // transfer-map buffers
constexpr size_t SMEM_BYTES = (MSTAGES * M_FLOATS + 2 * GDN_DK * BV) * sizeof(float);

// float offset of M[m][4 c4] in the swizzled buffer (c4: 16-byte chunk, 32 per row)
__device__ __forceinline__ int msw(int m, int c4) { return m * GDN_DK + ((c4 ^ (m & 31)) << 2); }

__global__ void __launch_bounds__(NTH) merge_kernel(MergeArgs a) {
  extern __shared__ __align__(16) float smem[];
  float *sM = smem;                        // MSTAGES transfer maps
  float *sS = smem + MSTAGES * M_FLOATS;   // two state slices [128][8]
  const int m = threadIdx.x;
  const int col0 = blockIdx.x * BV;
  const int64_t bh = blockIdx.y;
  const int64_t KV = (int64_t)GDN_DK * GDN_DV;
  const uint32_t sMa = static_cast<uint32_t>(__cvta_generic_to_shared(sM));

  const bool adj = a.adjoint != 0;
  // segment visited at step i (forward order, or reverse for the adjoint)
  auto seg_at = [&](int i) { return adj ? a.nseg - 1 - i : i; };
  auto fetch_M = [&](int i) {  // every thread copies one row: 32 chunks of 16 bytes
    const float *Ms = a.M + (bh * a.nseg + seg_at(i)) * M_FLOATS + (int64_t)m * GDN_DK;
    const uint32_t dst = sMa + (uint32_t)((i % MSTAGES) * M_FLOATS) * 4u;
#pragma unroll 8
    for (int c4 = 0; c4 < 32; ++c4) cp_async16(dst + (uint32_t)msw(m, c4) * 4u, Ms + 4 * c4, 16u);
    cp_async_commit();
  };

  float cur[BV];
  {
    const float *src = a.h0 ? a.h0 + bh * KV + (int64_t)m * GDN_DV + col0 : nullptr;
#pragma unroll
    for (int j = 0; j < BV; ++j) cur[j] = src ? src[j] : 0.f;
  }
#pragma unroll
  for (int j = 0; j < BV; ++j) sS[m * BV + j] = cur[j];
  // the local term of the segment visited at step i (row m, this CTA's columns)
  auto ext_at = [&](int i, float4 &e0, float4 &e1) {
    const float4 *es = reinterpret_cast<const float4 *>(
        a.S_ext + (bh * a.nseg + seg_at(i)) * KV + (int64_t)m * GDN_DV + col0);
    e0 = es[0];
    e1 = es[1];
  };
  float4 e0 = make_float4(0.f, 0.f, 0.f, 0.f), e1 = e0;
  if (a.nseg > 0) {
    fetch_M(0);
    ext_at(0, e0, e1);
  }
  if (a.nseg > 1) fetch_M(1);
  for (int s = 0; s < a.nseg; ++s) {
    const int64_t slot = bh * a.nseg + seg_at(s);
    // this segment's entry state; the next segment's local term, meanwhile
    float4 *dst = reinterpret_cast<float4 *>(a.S_init + slot * KV + (int64_t)m * GDN_DV + col0);
    dst[0] = make_float4(cur[0], cur[1], cur[2], cur[3]);
    dst[1] = make_float4(cur[4], cur[5], cur[6], cur[7]);
    float4 n0 = e0, n1 = e1;
    if (s + 1 < a.nseg) ext_at(s + 1, n0, n1);
    // M_s has landed (M_{s+1} may still be in flight)
    if (s + 1 < a.nseg) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();  // M_s and the state slice are visible; every read of M_{s-1} is done
    if (s + 2 < a.nseg) fetch_M(s + 2);  // into the buffer M_{s-1} held
    const float *Mb = sM + (s % MSTAGES) * M_FLOATS;
    const float *Sb = sS + (s & 1) * GDN_DK * BV;
    float acc[BV];
#pragma unroll
    for (int j = 0; j < BV; ++j) acc[j] = 0.f;
#pragma unroll 4
    for (int c4 = 0; c4 < 32; ++c4) {
      float mk[4];
      if (!adj) {  // row m of M
        const float4 mv = *reinterpret_cast<const float4 *>(Mb + msw(m, c4));
        mk[0] = mv.x; mk[1] = mv.y; mk[2] = mv.z; mk[3] = mv.w;
      } else {  // row m of M^T: column m of M (a warp reads 32 consecutive columns of one row)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mk[kk] = Mb[msw(4 * c4 + kk, m >> 2) + (m & 3)];
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 s0 = *reinterpret_cast<const float4 *>(Sb + (4 * c4 + kk) * BV);
        const float4 s1 = *reinterpret_cast<const float4 *>(Sb + (4 * c4 + kk) * BV + 4);
        acc[0] = fmaf(mk[kk], s0.x, acc[0]);
        acc[1] = fmaf(mk[kk], s0.y, acc[1]);
        acc[2] = fmaf(mk[kk], s0.z, acc[2]);
        acc[3] = fmaf(mk[kk], s0.w, acc[3]);
        acc[4] = fmaf(mk[kk], s1.x, acc[4]);
        acc[5] = fmaf(mk[kk], s1.y, acc[5]);
        acc[6] = fmaf(mk[kk], s1.z, acc[6]);
        acc[7] = fmaf(mk[kk], s1.w, acc[7]);
      }
    }
    cur[0] = acc[0] + e0.x;
    cur[1] = acc[1] + e0.y;
    cur[2] = acc[2] + e0.z;
    cur[3] = acc[3] + e0.w;
    cur[4] = acc[4] + e1.x;
    cur[5] = acc[5] + e1.y;
    cur[6] = acc[6] + e1.z;
    cur[7] = acc[7] + e1.w;
    e0 = n0;
    e1 = n1;
    float *Sn = sS + ((s + 1) & 1) * GDN_DK * BV;
#pragma unroll
    for (int j = 0; j < BV; ++j) Sn[m * BV + j] = cur[j];
  }
  if (a.ht) {
    float4 *dst = reinterpret_cast<float4 *>(a.ht + bh * KV + (int64_t)m * GDN_DV + col0);
    dst[0] = make_float4(cur[0], cur[1], cur[2], cur[3]);
    dst[1] = make_float4(cur[4], cur[5], cur[6], cur[7]);
  }
  cp_async_wait<0>();
}

}  // namespace

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  merge_kernel<<<dim3(GDN_DV / BV, a.BH), NTH, SMEM_BYTES, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
