// Dense per-token transition scan (SANA, distributed_scan.py page: cp_frame_gdn_scan and
// its local scan), fp32 on the FMA pipes (the page runs it in fp32), state width D = 32 or 64:
//
//   KV state, right multiply:  S[t] = S[t-1] W_kv[t] + U_kv[t]
//   Z state, left multiply:    s[t] = W_z[t] s[t-1] + u_z[t]
//
// truncate_to_active: positions t >= active leave both states unchanged (the page sets W = I,
// U = 0 there), so their outputs repeat the state of position active-1.
//
// A long sequence is split into segments that run on different SMs (the page's ranks, here
// the SMs of one GPU): a summary pass runs every segment from the zero state and the identity
// map (its final state h and transition product M: M_kv = W_kv[a] ... W_kv[b-1], M_z =
// W_z[b-1] ... W_z[a]); the merge composes them in order (S_init_{j+1} = S_init_j M_kv_j +
// h_kv_j, s_init_{j+1} = M_z_j s_init_j + h_z_j, the page's exclusive prefix composition);
// the scan pass re-runs every segment from its entry state and writes every position's
// state. The page adds S_init W_cum[t] to the zero-start states instead of re-running; by
// the recurrence's linearity the two are the same numbers up to rounding.
//
// One CTA (256 threads) walks the positions of one segment. Each position's W_kv, U_kv, W_z
// and u_z (3 D^2 + D floats) arrive by bulk copies STAGES positions ahead, completing on one
// mbarrier per stage. The KV state (and the summary's KV map) is kept transposed in shared
// memory, double-buffered by position, so that a thread's 4 x 4 (D = 64) or 2 x 2 (D = 32)
// output tile reads one vector of the state and one of W per step of the contraction; the
// Z state's matrix-vector product takes 256 / D threads per row and a shuffle reduction.
// Every mbarrier wait is bounded; a wait that runs out stops the CTA after its copies land
// and raises the device flag.
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace gdn {
namespace {
using namespace tc;

constexpr int FS_NTH = 256;
constexpr uint32_t FS_WAIT_LIMIT = 1u << 22;

template <int D>
struct FsShape {
  static constexpr int TM = D == 64 ? 4 : 2;         // output rows per thread
  static constexpr int TN = D == 64 ? 4 : 2;         // output columns per thread
  static constexpr int GN = D / TN;                  // threads along the columns
  static constexpr int P = D + 4;                    // padded row of a transposed tile
  static constexpr int POS = 3 * D * D + D;          // floats of one position: W_kv, U_kv, W_z, u_z
  static constexpr int TPR = FS_NTH / D;             // threads per row of the Z product
  static constexpr int KPT = D / TPR;                // Z contraction length per thread
  static_assert((D / TM) * (D / TN) == FS_NTH, "tile grid covers the CTA");
};

template <int D, bool SUMMARY, int STAGES>
constexpr int fs_smem_bytes() {
  using S = FsShape<D>;
  return 4 * (STAGES * S::POS + 2 * D * S::P + (SUMMARY ? 2 * D * S::P + 2 * D * D : 0) + 2 * D) + 8 * STAGES + 16;
}

template <int N>
struct Vec;
template <>
struct Vec<4> {
  static __device__ __forceinline__ void ld(const float *p, float *v) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
  }
  static __device__ __forceinline__ void st(float *p, const float *v) {
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<2> {
  static __device__ __forceinline__ void ld(const float *p, float *v) {
    const float2 x = *reinterpret_cast<const float2 *>(p);
    v[0] = x.x, v[1] = x.y;
  }
  static __device__ __forceinline__ void st(float *p, const float *v) {
    *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
  }
};

// acc[r][c] = sum_k At[k][i0 + r] B[k][j0 + c]  (At: transposed left factor, row stride P)
template <int D>
__device__ __forceinline__ void prod_right(const float *At, const float *B, int i0, int j0,
                                           float (&acc)[FsShape<D>::TM][FsShape<D>::TN]) {
  using S = FsShape<D>;
#pragma unroll 4
  for (int k = 0; k < D; ++k) {
    float a[S::TM], b[S::TN];
    Vec<S::TM>::ld(At + k * S::P + i0, a);
    Vec<S::TN>::ld(B + k * D + j0, b);
#pragma unroll
    for (int r = 0; r < S::TM; ++r)
#pragma unroll
      for (int c = 0; c < S::TN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}
// acc[r][c] = sum_k A[i0 + r][k] B[k][j0 + c]  (A row-major, row stride D)
template <int D>
__device__ __forceinline__ void prod_left(const float *A, const float *B, int i0, int j0,
                                          float (&acc)[FsShape<D>::TM][FsShape<D>::TN]) {
  using S = FsShape<D>;
#pragma unroll 4
  for (int k = 0; k < D; ++k) {
    float a[S::TM], b[S::TN];
#pragma unroll
    for (int r = 0; r < S::TM; ++r) a[r] = A[(i0 + r) * D + k];
    Vec<S::TN>::ld(B + k * D + j0, b);
#pragma unroll
    for (int r = 0; r < S::TM; ++r)
#pragma unroll
      for (int c = 0; c < S::TN; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
  }
}
// z_out[row] = sum_k A[row][k] z[k] + u[row]: TPR threads per row, reduced by shuffles
template <int D>
__device__ __forceinline__ void matvec(const float *A, const float *z, const float *u, float *z_out, int tid) {
  using S = FsShape<D>;
  const int row = tid / S::TPR, part = tid % S::TPR;
  float sum = 0.f;
#pragma unroll
  for (int kk = 0; kk < S::KPT; ++kk) {
    const int k = part * S::KPT + kk;
    sum = fmaf(A[row * D + k], z[k], sum);
  }
#pragma unroll
  for (int off = S::TPR / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (part == 0) z_out[row] = sum + (u ? u[row] : 0.f);
}

template <int D, bool SUMMARY, int STAGES>
__global__ void __launch_bounds__(FS_NTH, 1) frame_scan_kernel(FrameScanArgs a) {
  using S = FsShape<D>;
  extern __shared__ __align__(16) float smf[];
  float *pos = smf;                                        // STAGES positions
  float *St = pos + STAGES * S::POS;                       // 2 x transposed KV state
  float *Mt = St + 2 * D * S::P;                           // summary: 2 x transposed KV map
  float *Mz = Mt + (SUMMARY ? 2 * D * S::P : 0);           // summary: 2 x Z map (row-major)
  float *zs = Mz + (SUMMARY ? 2 * D * D : 0);              // 2 x Z state
  uint64_t *bar = reinterpret_cast<uint64_t *>(reinterpret_cast<uintptr_t>(zs + 2 * D + 3) & ~uintptr_t(7));

  const int tid = threadIdx.x, warp = tid >> 5;
  const int bh = blockIdx.y, seg = blockIdx.x;
  const int64_t T = a.T;
  const int64_t t0 = (int64_t)seg * a.seg_len, t1 = min(t0 + a.seg_len, T);
  const int64_t tact = a.active > 0 ? min(t1, (int64_t)a.active) : t1;  // [t0, tact) update
  const int i0 = (tid / S::GN) * S::TM, j0 = (tid % S::GN) * S::TN;
  const int64_t slot = (int64_t)bh * a.nseg + seg;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  // entry state: the segment's merged entry state, the caller's initial state, or zero (and
  // the identity maps of the summary)
  const float *S_in = nullptr, *z_in = nullptr;
  if (!SUMMARY) {
    if (a.S_init) {
      S_in = a.S_init + slot * D * D;
      z_in = a.z_init + slot * D;
    } else {
      S_in = a.S0 ? a.S0 + (int64_t)bh * D * D : nullptr;
      z_in = a.z0 ? a.z0 + (int64_t)bh * D : nullptr;
    }
  }
  for (int e = tid; e < D * D; e += FS_NTH) {
    const int i = e / D, j = e % D;
    St[j * S::P + i] = S_in ? S_in[e] : 0.f;
    if (SUMMARY) {
      Mt[j * S::P + i] = i == j ? 1.f : 0.f;
      Mz[e] = i == j ? 1.f : 0.f;
    }
  }
  for (int e = tid; e < D; e += FS_NTH) zs[e] = z_in ? z_in[e] : 0.f;
  __syncthreads();

  const float *gW = a.W_kv + (int64_t)bh * T * D * D, *gU = a.U_kv + (int64_t)bh * T * D * D;
  const float *gWz = a.W_z + (int64_t)bh * T * D * D, *gu = a.u_z + (int64_t)bh * T * D;
  int64_t last_issued = -1;
  auto issue = [&](int64_t t) {  // warp 0: position t into its stage
    const int s = (int)((t - t0) % STAGES);
    float *dst = pos + s * S::POS;
    mbar_expect_tx_w(&bar[s], S::POS * 4);
    bulk_load_w(smem_u32(dst), gW + t * D * D, D * D * 4, &bar[s]);
    bulk_load_w(smem_u32(dst + D * D), gU + t * D * D, D * D * 4, &bar[s]);
    bulk_load_w(smem_u32(dst + 2 * D * D), gWz + t * D * D, D * D * 4, &bar[s]);
    bulk_load_w(smem_u32(dst + 3 * D * D), gu + t * D, D * 4, &bar[s]);
    last_issued = t;
  };
  if (warp == 0)
    for (int s = 0; s < STAGES && t0 + s < tact; ++s) issue(t0 + s);

  int cur = 0;  // buffer of the current state
  bool bad = false;
  float *gS = a.S_all ? a.S_all + (int64_t)bh * T * D * D : nullptr;
  float *gz = a.z_all ? a.z_all + (int64_t)bh * T * D : nullptr;
  for (int64_t t = t0; t < t1; ++t) {
    float sv[S::TM][S::TN];
    if (t < tact) {
      const int s = (int)((t - t0) % STAGES);
      if (!mbar_wait(&bar[s], (uint32_t)(((t - t0) / STAGES) & 1), FS_WAIT_LIMIT)) bad = true;
      const float *W = pos + s * S::POS, *U = W + D * D, *Wz = W + 2 * D * D, *u = W + 3 * D * D;
      // KV: S W + U
#pragma unroll
      for (int r = 0; r < S::TM; ++r) Vec<S::TN>::ld(U + (i0 + r) * D + j0, sv[r]);
      prod_right<D>(St + cur * D * S::P, W, i0, j0, sv);
      float *Sn = St + (cur ^ 1) * D * S::P;
#pragma unroll
      for (int c = 0; c < S::TN; ++c) {
        float col[S::TM];
#pragma unroll
        for (int r = 0; r < S::TM; ++r) col[r] = sv[r][c];
        Vec<S::TM>::st(Sn + (j0 + c) * S::P + i0, col);
      }
      // Z: W_z s + u
      matvec<D>(Wz, zs + cur * D, u, zs + (cur ^ 1) * D, tid);
      if (SUMMARY) {
        // KV map M W; Z map W_z M_z
        float mv[S::TM][S::TN] = {};
        prod_right<D>(Mt + cur * D * S::P, W, i0, j0, mv);
        float *Mn = Mt + (cur ^ 1) * D * S::P;
#pragma unroll
        for (int c = 0; c < S::TN; ++c) {
          float col[S::TM];
#pragma unroll
          for (int r = 0; r < S::TM; ++r) col[r] = mv[r][c];
          Vec<S::TM>::st(Mn + (j0 + c) * S::P + i0, col);
        }
        float zv[S::TM][S::TN] = {};
        prod_left<D>(Wz, Mz + cur * D * D, i0, j0, zv);
#pragma unroll
        for (int r = 0; r < S::TM; ++r) Vec<S::TN>::st(Mz + (cur ^ 1) * D * D + (i0 + r) * D + j0, zv[r]);
      }
      cur ^= 1;
    } else if (!SUMMARY) {  // a held position: the state of position active-1
#pragma unroll
      for (int r = 0; r < S::TM; ++r)
#pragma unroll
        for (int c = 0; c < S::TN; ++c) sv[r][c] = St[cur * D * S::P + (j0 + c) * S::P + i0 + r];
    }
    if (!SUMMARY && gS) {
      float *dst = gS + t * D * D;
#pragma unroll
      for (int r = 0; r < S::TM; ++r) Vec<S::TN>::st(dst + (i0 + r) * D + j0, sv[r]);
    }
    if (__syncthreads_or(bad)) {  // every thread is done with the position's buffers
      bad = true;
      break;
    }
    if (!SUMMARY && gz && tid < D) gz[t * D + tid] = zs[cur * D + tid];
    if (warp == 0 && t + STAGES < tact) issue(t + STAGES);
  }

  if (bad) {
    if (warp == 0 && last_issued >= 0)  // copies in flight land before the CTA leaves
      for (int64_t t = max(t0, last_issued - STAGES + 1); t <= last_issued; ++t)
        mbar_wait(&bar[(t - t0) % STAGES], (uint32_t)(((t - t0) / STAGES) & 1), FS_WAIT_LIMIT);
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    return;
  }
  if (SUMMARY) {
    float *h = a.h_kv + slot * D * D, *M = a.M_kv + slot * D * D, *Mzo = a.M_z + slot * D * D;
    for (int e = tid; e < D * D; e += FS_NTH) {
      const int i = e / D, j = e % D;
      h[e] = St[cur * D * S::P + j * S::P + i];
      M[e] = Mt[cur * D * S::P + j * S::P + i];
      Mzo[e] = Mz[cur * D * D + e];
    }
    for (int e = tid; e < D; e += FS_NTH) a.h_z[slot * D + e] = zs[cur * D + e];
  } else if (seg == a.nseg - 1) {  // the terminal state (the state of position active-1)
    for (int e = tid; e < D * D; e += FS_NTH)
      if (a.S_last) a.S_last[(int64_t)bh * D * D + e] = St[cur * D * S::P + (e % D) * S::P + e / D];
    for (int e = tid; e < D; e += FS_NTH)
      if (a.z_last) a.z_last[(int64_t)bh * D + e] = zs[cur * D + e];
  }
}

// Entry state of every segment: S_init_0 = S0 (or 0), S_init_{j+1} = S_init_j M_kv_j + h_kv_j,
// s_init_{j+1} = M_z_j s_init_j + h_z_j. One CTA per sequence.
template <int D>
__global__ void __launch_bounds__(FS_NTH, 1) frame_merge_kernel(FrameScanArgs a) {
  using S = FsShape<D>;
  extern __shared__ __align__(16) float smf[];
  float *St = smf;                   // 2 x transposed KV state
  float *M = St + 2 * D * S::P;      // M_kv_j (row-major)
  float *Mz = M + D * D;             // M_z_j
  float *zs = Mz + D * D;            // 2 x Z state
  const int tid = threadIdx.x, bh = blockIdx.x;
  const int i0 = (tid / S::GN) * S::TM, j0 = (tid % S::GN) * S::TN;
  for (int e = tid; e < D * D; e += FS_NTH) {
    const int i = e / D, j = e % D;
    St[j * S::P + i] = a.S0 ? a.S0[(int64_t)bh * D * D + e] : 0.f;
  }
  for (int e = tid; e < D; e += FS_NTH) zs[e] = a.z0 ? a.z0[(int64_t)bh * D + e] : 0.f;
  int cur = 0;
  for (int j = 0; j < a.nseg; ++j) {
    const int64_t slot = (int64_t)bh * a.nseg + j;
    __syncthreads();
    for (int e = tid; e < D * D; e += FS_NTH) {
      a.S_init[slot * D * D + e] = St[cur * D * S::P + (e % D) * S::P + e / D];
      M[e] = a.M_kv[slot * D * D + e];
      Mz[e] = a.M_z[slot * D * D + e];
    }
    for (int e = tid; e < D; e += FS_NTH) a.z_init[slot * D + e] = zs[cur * D + e];
    __syncthreads();
    if (j + 1 == a.nseg) break;
    float sv[S::TM][S::TN];
#pragma unroll
    for (int r = 0; r < S::TM; ++r) Vec<S::TN>::ld(a.h_kv + slot * D * D + (i0 + r) * D + j0, sv[r]);
    prod_right<D>(St + cur * D * S::P, M, i0, j0, sv);
    float *Sn = St + (cur ^ 1) * D * S::P;
#pragma unroll
    for (int c = 0; c < S::TN; ++c) {
      float col[S::TM];
#pragma unroll
      for (int r = 0; r < S::TM; ++r) col[r] = sv[r][c];
      Vec<S::TM>::st(Sn + (j0 + c) * S::P + i0, col);
    }
    matvec<D>(Mz, zs + cur * D, a.h_z + slot * D, zs + (cur ^ 1) * D, tid);
    cur ^= 1;
  }
}

// ---- one pass with the KV rows split over CTAs -----------------------------------------------
// The rows of the KV state are independent (S[t][i, :] = S[t-1][i, :] W_kv[t] + U_kv[t][i, :]),
// so R rows of one sequence (or segment) go to one CTA, and D / R such CTAs walk the same
// positions, each reading the whole W_kv[t] (L2 serves the repeats). In a CTA of 256 threads,
// KQ = 256 / D groups split the contraction over k (thread = one column of one group, its R
// rows in registers); the groups' partial sums meet in shared memory, where all threads add
// them, two outputs each. The Z state takes a CTA of its own.
template <int D, int R, int STAGES>
__device__ __forceinline__ void frame_kv_rows(const FrameScanArgs &a) {
  constexpr int STG = D * D + R * D;  // floats of one stage: W_kv[t], U_kv[t] rows r0 .. r0+R-1
  constexpr int KQ = FS_NTH / D, KL = D / KQ;  // contraction groups, k per group
  constexpr int OPT = R * D / FS_NTH;          // outputs per thread in the sum
  static_assert(OPT >= 1 && OPT * FS_NTH == R * D, "whole outputs per thread");
  extern __shared__ __align__(16) float smf[];
  float *pos = smf;
  float *St = pos + STAGES * STG;  // 2 x [D][R]: St[k][r] = S[r0 + r][k]
  float *Part = St + 2 * D * R;    // [KQ][R][D] partial sums
  uint64_t *bar = reinterpret_cast<uint64_t *>(Part + KQ * R * D);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int j = tid % D, kq = tid / D;
  const int r0 = blockIdx.x * R, seg = blockIdx.y, bh = blockIdx.z;
  const int64_t T = a.T;
  const int64_t t0 = (int64_t)seg * a.seg_len, t1 = min(t0 + a.seg_len, T);
  const int64_t tact = a.active > 0 ? min(t1, (int64_t)a.active) : t1;
  const int64_t slot = (int64_t)bh * a.nseg + seg;
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  const float *S_in = a.S_init ? a.S_init + slot * D * D : a.S0 ? a.S0 + (int64_t)bh * D * D : nullptr;
  for (int e = tid; e < R * D; e += FS_NTH) {
    const int r = e / D, c = e % D;
    St[c * R + r] = S_in ? S_in[(r0 + r) * D + c] : 0.f;
  }
  __syncthreads();
  const float *gW = a.W_kv + (int64_t)bh * T * D * D, *gU = a.U_kv + (int64_t)bh * T * D * D;
  int64_t last_issued = -1;
  auto issue = [&](int64_t t) {  // warp 0
    const int s = (int)((t - t0) % STAGES);
    float *dst = pos + s * STG;
    mbar_expect_tx_w(&bar[s], STG * 4);
    bulk_load_w(smem_u32(dst), gW + t * D * D, D * D * 4, &bar[s]);
    bulk_load_w(smem_u32(dst + D * D), gU + t * D * D + r0 * D, R * D * 4, &bar[s]);
    last_issued = t;
  };
  if (warp == 0)
    for (int s = 0; s < STAGES && t0 + s < tact; ++s) issue(t0 + s);
  int cur = 0;
  bool bad = false;
  float *gS = a.S_all + (int64_t)bh * T * D * D;
  for (int64_t t = t0; t < t1; ++t) {
    float *Sn = St + (cur ^ 1) * D * R;
    const float *Sc = St + cur * D * R;
    if (t < tact) {
      const int s = (int)((t - t0) % STAGES);
      if (!mbar_wait(&bar[s], (uint32_t)(((t - t0) / STAGES) & 1), FS_WAIT_LIMIT)) bad = true;
      const float *W = pos + s * STG, *U = W + D * D;
      float acc[R];
#pragma unroll
      for (int r = 0; r < R; ++r) acc[r] = kq == 0 ? U[r * D + j] : 0.f;
#pragma unroll
      for (int kk = 0; kk < KL; ++kk) {
        const int k = kq * KL + kk;
        const float w = W[k * D + j];
        float sk[R];
#pragma unroll
        for (int q = 0; q < R / 4; ++q) Vec<4>::ld(Sc + k * R + 4 * q, sk + 4 * q);
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] = fmaf(sk[r], w, acc[r]);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) Part[(kq * R + r) * D + j] = acc[r];
      __syncthreads();
#pragma unroll
      for (int o = 0; o < OPT; ++o) {
        const int e = tid + o * FS_NTH, r = e / D, c = e % D;
        float v = 0.f;
#pragma unroll
        for (int g = 0; g < KQ; ++g) v += Part[(g * R + r) * D + c];
        Sn[c * R + r] = v;
        gS[t * D * D + (r0 + r) * D + c] = v;
      }
      cur ^= 1;
    } else {
#pragma unroll
      for (int o = 0; o < OPT; ++o) {
        const int e = tid + o * FS_NTH, r = e / D, c = e % D;
        gS[t * D * D + (r0 + r) * D + c] = Sc[c * R + r];
      }
    }
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
    if (warp == 0 && t + STAGES < tact) issue(t + STAGES);
  }
  if (bad) {
    if (warp == 0 && last_issued >= 0)
      for (int64_t t = max(t0, last_issued - STAGES + 1); t <= last_issued; ++t)
        mbar_wait(&bar[(t - t0) % STAGES], (uint32_t)(((t - t0) / STAGES) & 1), FS_WAIT_LIMIT);
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    return;
  }
  if (seg == a.nseg - 1 && a.S_last)
    for (int e = tid; e < R * D; e += FS_NTH) {
      const int r = e / D, c = e % D;
      a.S_last[(int64_t)bh * D * D + (r0 + r) * D + c] = St[cur * D * R + c * R + r];
    }
}

// The Z state of one sequence (or segment): s[t] = W_z[t] s[t-1] + u_z[t], 256 threads; in each
// of D / 16 passes a warp takes two rows, 16 lanes per row, one float4 of the row per lane
// (a warp reads 512 contiguous bytes: no bank conflict), and sums with shuffles.
template <int D, int STAGES>
__device__ __forceinline__ void frame_z(const FrameScanArgs &a) {
  constexpr int STG = D * D + D;  // W_z[t], u_z[t]
  constexpr int LPR = D / 4;      // lanes per row: one float4 each
  constexpr int RPP = FS_NTH / LPR;  // rows per pass
  extern __shared__ __align__(16) float smf[];
  float *pos = smf;
  float *zs = pos + STAGES * STG;  // 2 x [D]
  uint64_t *bar = reinterpret_cast<uint64_t *>(zs + 2 * D);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int seg = blockIdx.y, bh = blockIdx.z;
  const int64_t T = a.T;
  const int64_t t0 = (int64_t)seg * a.seg_len, t1 = min(t0 + a.seg_len, T);
  const int64_t tact = a.active > 0 ? min(t1, (int64_t)a.active) : t1;
  const int64_t slot = (int64_t)bh * a.nseg + seg;
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bar[s], 1);
    mbar_fence_init();
  }
  const float *z_in = a.z_init ? a.z_init + slot * D : a.z0 ? a.z0 + (int64_t)bh * D : nullptr;
  if (tid < D) zs[tid] = z_in ? z_in[tid] : 0.f;
  __syncthreads();
  const float *gW = a.W_z + (int64_t)bh * T * D * D, *gu = a.u_z + (int64_t)bh * T * D;
  int64_t last_issued = -1;
  auto issue = [&](int64_t t) {
    const int s = (int)((t - t0) % STAGES);
    float *dst = pos + s * STG;
    mbar_expect_tx_w(&bar[s], STG * 4);
    bulk_load_w(smem_u32(dst), gW + t * D * D, D * D * 4, &bar[s]);
    bulk_load_w(smem_u32(dst + D * D), gu + t * D, D * 4, &bar[s]);
    last_issued = t;
  };
  if (warp == 0)
    for (int s = 0; s < STAGES && t0 + s < tact; ++s) issue(t0 + s);
  int cur = 0;
  bool bad = false;
  float *gz = a.z_all + (int64_t)bh * T * D;
  const int lr = tid / LPR, q = tid % LPR;  // row within the pass, float4 index within the row
  for (int64_t t = t0; t < t1; ++t) {
    if (t < tact) {
      const int s = (int)((t - t0) % STAGES);
      if (!mbar_wait(&bar[s], (uint32_t)(((t - t0) / STAGES) & 1), FS_WAIT_LIMIT)) bad = true;
      const float *W = pos + s * STG, *u = W + D * D;
      float zq[4];
      Vec<4>::ld(zs + cur * D + 4 * q, zq);
#pragma unroll
      for (int p = 0; p < D / RPP; ++p) {
        const int row = p * RPP + lr;
        float w[4];
        Vec<4>::ld(W + row * D + 4 * q, w);
        float sum = w[0] * zq[0];
        sum = fmaf(w[1], zq[1], sum);
        sum = fmaf(w[2], zq[2], sum);
        sum = fmaf(w[3], zq[3], sum);
#pragma unroll
        for (int off = LPR / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (q == 0) zs[(cur ^ 1) * D + row] = sum + u[row];
      }
      cur ^= 1;
    }
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
    if (tid < D) gz[t * D + tid] = zs[cur * D + tid];
    if (warp == 0 && t + STAGES < tact) issue(t + STAGES);
  }
  if (bad) {
    if (warp == 0 && last_issued >= 0)
      for (int64_t t = max(t0, last_issued - STAGES + 1); t <= last_issued; ++t)
        mbar_wait(&bar[(t - t0) % STAGES], (uint32_t)(((t - t0) / STAGES) & 1), FS_WAIT_LIMIT);
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    return;
  }
  if (seg == a.nseg - 1 && a.z_last && tid < D) a.z_last[(int64_t)bh * D + tid] = zs[cur * D + tid];
}

// One grid for both states: blocks 0 .. D/R-1 of every sequence (or segment) take KV rows,
// block D/R its Z state, so that the two run side by side.
template <int D, int R, int KS, int ZS>
__global__ void __launch_bounds__(FS_NTH, 1) frame_rows_kernel(FrameScanArgs a) {
  if (blockIdx.x < D / R) frame_kv_rows<D, R, KS>(a);
  else frame_z<D, ZS>(a);
}

template <int D>
cudaError_t launch_rows(const FrameScanArgs &a, cudaStream_t st) {
  constexpr int R = 8, KS = 4, ZS = 4;
  constexpr int ksmem = 4 * (KS * (D * D + R * D) + 2 * D * R + (FS_NTH / D) * R * D) + 8 * KS;
  constexpr int zsmem = 4 * (ZS * (D * D + D) + 2 * D) + 8 * ZS;
  constexpr int smem = ksmem > zsmem ? ksmem : zsmem;
  static_assert(smem <= 232448, "shared memory");
  auto kern = frame_rows_kernel<D, R, KS, ZS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(D / R + 1, a.nseg, a.BH), FS_NTH, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D, bool SUMMARY, int STAGES>
cudaError_t launch_scan(const FrameScanArgs &a, dim3 grid, cudaStream_t st) {
  constexpr int smem = fs_smem_bytes<D, SUMMARY, STAGES>();
  auto kern = frame_scan_kernel<D, SUMMARY, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, FS_NTH, smem, st>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_all(const FrameScanArgs &a0, cudaStream_t st) {
  FrameScanArgs a = a0;
  if (a.nseg > 1) {
    cudaError_t e = launch_scan<D, true, 2>(a, dim3(a.nseg, a.BH), st);
    if (e != cudaSuccess) return e;
    constexpr int msmem = 4 * (2 * D * FsShape<D>::P + 2 * D * D + 2 * D);
    e = cudaFuncSetAttribute(frame_merge_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, msmem);
    if (e != cudaSuccess) return e;
    frame_merge_kernel<D><<<a.BH, FS_NTH, msmem, st>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  } else {
    a.S_init = nullptr;
    a.z_init = nullptr;
  }
  return launch_rows<D>(a, st);
}

}  // namespace

static_assert(fs_smem_bytes<64, true, 2>() <= 232448 && fs_smem_bytes<64, false, 3>() <= 232448,
              "shared memory");

cudaError_t launch_frame_scan(const FrameScanArgs &a, cudaStream_t st) {
  return a.D == 64 ? launch_all<64>(a, st) : launch_all<32>(a, st);
}

}  // namespace gdn
