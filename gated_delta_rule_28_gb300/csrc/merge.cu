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
// head, 8 state columns) and walks the segments in order; its 256 threads own one
// state row and half of its contraction each (the two halves added through shared
// memory). Per segment the only dependent work is the 128 x 8 x 128 product M_s S. The
// transfer maps (64 KB each) arrive two segments ahead in three shared-memory buffers
// (four TMA boxes of 32 columns each, on one mbarrier per buffer) while the current one is
// applied, and the local terms one segment ahead into registers. A box holds its 128 rows
// of 128 bytes with the 16-byte chunks of row r XOR-swizzled by r mod 8, so the 16-byte
// reads of a quarter warp (eight rows, the same columns) and the 4-byte reads of a warp (32
// columns of one row) are free of bank conflicts; the state slice is read by all threads
// alike (broadcast).
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tile;
using namespace tc;

constexpr int BV = 8;      // state columns per CTA
constexpr int NTH = 256;   // two threads per state row (halves of the contraction)
constexpr int M_FLOATS = GDN_DK * GDN_DK;
constexpr int MSTAGES = 3;  // transfer-map buffers
constexpr size_t SMEM_BYTES = (MSTAGES * M_FLOATS + 3 * GDN_DK * BV) * sizeof(float) + 64 + 1024;
constexpr uint32_t WAIT_LIMIT = 1u << 22;

// float offset of M[m][4 c4] in a buffer: box c4 / 8 (16 KB each), row m (128 bytes), chunk
// (c4 mod 8) XOR (m mod 8)
__device__ __forceinline__ int msw(int m, int c4) { return (c4 >> 3) * 4096 + m * 32 + (((c4 & 7) ^ (m & 7)) << 2); }

struct MergeMaps {
  TmaMap m;  // every transfer map: [BH * nseg * 128 rows][128] fp32, 32 x 128 boxes
};

__global__ void __launch_bounds__(NTH) merge_kernel(MergeArgs a, const __grid_constant__ MergeMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  float *smem = reinterpret_cast<float *>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  float *sM = smem;                        // MSTAGES transfer maps
  float *sS = smem + MSTAGES * M_FLOATS;   // two state slices [128][8]
  float *sP = sS + 2 * GDN_DK * BV;        // the second half's partial products [128][8]
  uint64_t *bar = reinterpret_cast<uint64_t *>(sP + GDN_DK * BV);  // one per buffer
  const int m = threadIdx.x & (GDN_DK - 1), half = threadIdx.x >> 7;
  const int col0 = blockIdx.x * BV;
  const int64_t bh = blockIdx.y;
  const int64_t KV = (int64_t)GDN_DK * GDN_DV;
  const uint32_t sMa = smem_u32(sM);
  const int warp = threadIdx.x >> 5;

  const bool adj = a.adjoint != 0;
  // segment visited at step i (forward order, or reverse for the adjoint)
  auto seg_at = [&](int i) { return adj ? a.nseg - 1 - i : i; };
  int issued = 0;  // maps requested so far (warp 0)
  auto fetch_M = [&](int i) {  // warp 0: the four boxes of the map of step i
    const int st = i % MSTAGES;
    const uint32_t dst = sMa + (uint32_t)(st * M_FLOATS) * 4u;
    const int y = (int)((bh * a.nseg + seg_at(i)) * GDN_DK);
    mbar_expect_tx_w(&bar[st], M_FLOATS * 4);
#pragma unroll
    for (int b = 0; b < 4; ++b) tma_load_2d_w(dst + b * 16384, &maps.m, 32 * b, y, &bar[st]);
    issued = i + 1;
  };
  if (threadIdx.x == 0) {
    for (int st = 0; st < MSTAGES; ++st) mbar_init(&bar[st], 1);
    mbar_fence_init();
  }
  __syncthreads();

  float cur[BV];
  {
    const float *src = a.h0 ? a.h0 + bh * KV + (int64_t)m * GDN_DV + col0 : nullptr;
#pragma unroll
    for (int j = 0; j < BV; ++j) cur[j] = src ? src[j] : 0.f;
  }
  if (!half)
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
    if (warp == 0) fetch_M(0);
    ext_at(0, e0, e1);
  }
  if (a.nseg > 1 && warp == 0) fetch_M(1);
  bool late = false;
  for (int s = 0; s < a.nseg; ++s) {
    const int64_t slot = bh * a.nseg + seg_at(s);
    // this segment's entry state; the next segment's local term, meanwhile
    float4 n0 = e0, n1 = e1;
    if (!half) {
      float4 *dst = reinterpret_cast<float4 *>(a.S_init + slot * KV + (int64_t)m * GDN_DV + col0);
      dst[0] = make_float4(cur[0], cur[1], cur[2], cur[3]);
      dst[1] = make_float4(cur[4], cur[5], cur[6], cur[7]);
      if (s + 1 < a.nseg) ext_at(s + 1, n0, n1);
    }
    // M_s has landed (M_{s+1} may still be in flight)
    if (!mbar_wait(&bar[s % MSTAGES], (uint32_t)((s / MSTAGES) & 1), WAIT_LIMIT)) late = true;
    fence_proxy_async();  // this thread's reads of M_{s-1}, before its buffer's next copy
    if (__syncthreads_or(late)) {  // M_s and the state slice are visible; M_{s-1} is read
      late = true;
      break;
    }
    if (s + 2 < a.nseg && warp == 0) fetch_M(s + 2);  // into the buffer M_{s-1} held
    const float *Mb = sM + (s % MSTAGES) * M_FLOATS;
    const float *Sb = sS + (s & 1) * GDN_DK * BV;
    float acc[BV];
#pragma unroll
    for (int j = 0; j < BV; ++j) acc[j] = 0.f;
#pragma unroll 4
    for (int c4 = 16 * half; c4 < 16 * half + 16; ++c4) {
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
    if (half)
#pragma unroll
      for (int j = 0; j < BV; ++j) sP[m * BV + j] = acc[j];
    __syncthreads();  // the second half's partial products are in place
    if (!half) {
      const float e[BV] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
      float *Sn = sS + ((s + 1) & 1) * GDN_DK * BV;
#pragma unroll
      for (int j = 0; j < BV; ++j) {
        cur[j] = (acc[j] + sP[m * BV + j]) + e[j];
        Sn[m * BV + j] = cur[j];
      }
      e0 = n0;
      e1 = n1;
    }
  }
  if (late) {  // a map did not arrive: report, let the copies in flight land, leave
    if (threadIdx.x == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    if (warp == 0)
      for (int i = 0; i < issued; ++i) mbar_wait(&bar[i % MSTAGES], (uint32_t)((i / MSTAGES) & 1), WAIT_LIMIT);
    return;
  }
  if (a.ht && !half) {
    float4 *dst = reinterpret_cast<float4 *>(a.ht + bh * KV + (int64_t)m * GDN_DV + col0);
    dst[0] = make_float4(cur[0], cur[1], cur[2], cur[3]);
    dst[1] = make_float4(cur[4], cur[5], cur[6], cur[7]);
  }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (a.nseg < 1) return cudaErrorInvalidValue;
  const uint64_t rows = (uint64_t)a.BH * a.nseg * GDN_DK;  // every map's rows (32-bit TMA rows)
  if (rows > (uint64_t)INT32_MAX) return cudaErrorInvalidValue;
  MergeMaps maps;
  e = make_tmap_f32_32x128(&maps.m, a.M, rows);
  if (e != cudaSuccess) return e;
  merge_kernel<<<dim3(GDN_DV / BV, a.BH), NTH, SMEM_BYTES, st>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace gdn
