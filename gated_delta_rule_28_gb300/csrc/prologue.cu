// Input maps around the chunk kernels (sm_103a): the KDA adapter's in-kernel
// options ("Diff Coverage" page, _prepare_kda: use_qk_l2norm_in_kernel with
// epsilon 1e-6 and use_beta_sigmoid_in_kernel; the backward finalize takes
// q_rstd / k_rstd and a fused beta-sigmoid backward).
//
//   prologue (before the forward and the backward):
//     q, k <- x / sqrt(sum_d x_d^2 + 1e-6)   per (token, head) row of 128
//     beta <- 1 / (1 + exp(-beta))
//   epilogue (after the backward, in place on its outputs):
//     dx    <- rstd (dxn - xn <xn, dxn>),  rstd = 1 / sqrt(sum_d x_d^2 + 1e-6)
//     dbeta <- dbeta s (1 - s),  s = sigmoid(beta)
//
// Memory-bound elementwise work: half a warp per row, each lane eight consecutive
// elements (one 16-byte bf16 or two 16-byte fp32 vectors), the row sum by shuffles
// inside the half warp; a warp takes eight rows per pass (four in the backward's
// map, which reads two tensors per row) and issues all of their loads before the
// first sum, so that 64 bytes per lane (bf16) are in flight;
// grid-stride over the passes with a grid of whole waves of the SMs. The norm is
// computed in fp32 from the stored inputs (the backward recomputes it from the raw
// rows rather than reading a saved rstd).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int PRO_THREADS = 256;
constexpr float L2_EPS = 1e-6f;
constexpr int RPW = 8;      // rows per warp and pass: two half warps x 4
constexpr int RPW_BWD = 4;  // the same for the backward's map (two inputs per row: fewer registers)

// eight consecutive elements of a row (16-byte aligned: rows are 128 elements)
template <typename T>
struct Vec8;
template <>
struct Vec8<float> {
  __device__ static void load(const float *p, float (&x)[8]) {
    const float4 v0 = *reinterpret_cast<const float4 *>(p), v1 = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w; x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
  }
  __device__ static void store(float *p, const float (&x)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(x[4], x[5], x[6], x[7]);
  }
};
template <>
struct Vec8<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(__nv_bfloat16 *p, const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// sum over the 16 lanes of a half warp
__device__ __forceinline__ float half_sum(float s) {
#pragma unroll
  for (int off = 8; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

__device__ __forceinline__ float sigmoidf(float x) { return 1.f / (1.f + __expf(-x)); }

template <typename T>
__global__ void __launch_bounds__(PRO_THREADS) prologue_kernel(InputMapArgs a) {
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int64_t warps = (int64_t)gridDim.x * (PRO_THREADS / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (PRO_THREADS / 32) + (threadIdx.x >> 5);
  const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k);
  T *qn = static_cast<T *>(a.qn), *kn = static_cast<T *>(a.kn);
  if (a.l2norm) {
    const int64_t nrows = 2 * a.rows;  // rows of q, then rows of k
    for (int64_t b = w0; b * RPW < nrows; b += warps) {
      float x[4][8];
      bool on[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // every load of the pass first
        const int64_t r = b * RPW + 2 * u + half;
        const bool isq = r < a.rows;
        on[u] = r < nrows && !(isq && !q);  // (half-warp uniform)
        if (on[u]) Vec8<T>::load((isq ? q : k) + (isq ? r : r - a.rows) * GDN_DK + 8 * hl, x[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = on[u] ? fmaf(x[u][i], x[u][i], ss) : 0.f;
        const float rstd = rsqrtf(half_sum(ss) + L2_EPS);
        if (on[u]) {
          const int64_t r = b * RPW + 2 * u + half;
          const bool isq = r < a.rows;
#pragma unroll
          for (int i = 0; i < 8; ++i) x[u][i] *= rstd;
          Vec8<T>::store((isq ? qn : kn) + (isq ? r : r - a.rows) * GDN_DK + 8 * hl, x[u]);
        }
      }
    }
  }
  if (a.beta_sigmoid) {
    const T *beta = static_cast<const T *>(a.beta);
    T *beff = static_cast<T *>(a.beta_eff);
    const int64_t threads = (int64_t)gridDim.x * PRO_THREADS;
    for (int64_t r = (int64_t)blockIdx.x * PRO_THREADS + threadIdx.x; r < a.rows; r += threads)
      beff[r] = from_f32<T>(sigmoidf(to_f32(beta[r])));
  }
}

template <typename T>
__global__ void __launch_bounds__(PRO_THREADS) epilogue_bwd_kernel(InputMapArgs a) {
  const int lane = threadIdx.x & 31, half = lane >> 4, hl = lane & 15;
  const int64_t warps = (int64_t)gridDim.x * (PRO_THREADS / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (PRO_THREADS / 32) + (threadIdx.x >> 5);
  const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k);
  T *dq = static_cast<T *>(a.dq), *dk = static_cast<T *>(a.dk);
  if (a.l2norm) {
    const int64_t nrows = 2 * a.rows;
    for (int64_t b = w0; b * RPW_BWD < nrows; b += warps) {
      float x[RPW_BWD / 2][8], d[RPW_BWD / 2][8];
      bool on[RPW_BWD / 2];
#pragma unroll
      for (int u = 0; u < RPW_BWD / 2; ++u) {  // every load of the pass first
        const int64_t r = b * RPW_BWD + 2 * u + half;
        const bool isq = r < a.rows;
        on[u] = r < nrows;  // (half-warp uniform)
        if (on[u]) {
          const int64_t off = (isq ? r : r - a.rows) * GDN_DK + 8 * hl;
          Vec8<T>::load((isq ? q : k) + off, x[u]);
          Vec8<T>::load((isq ? dq : dk) + off, d[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < RPW_BWD / 2; ++u) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = on[u] ? fmaf(x[u][i], x[u][i], ss) : 0.f;
        const float rstd = rsqrtf(half_sum(ss) + L2_EPS);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[u][i] *= rstd;  // xn
        float dt = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) dt = on[u] ? fmaf(x[u][i], d[u][i], dt) : 0.f;
        const float dot = half_sum(dt);
        if (on[u]) {
          const int64_t r = b * RPW_BWD + 2 * u + half;
          const bool isq = r < a.rows;
#pragma unroll
          for (int i = 0; i < 8; ++i) d[u][i] = rstd * (d[u][i] - x[u][i] * dot);
          Vec8<T>::store((isq ? dq : dk) + (isq ? r : r - a.rows) * GDN_DK + 8 * hl, d[u]);
        }
      }
    }
  }
  if (a.beta_sigmoid) {
    const T *beta = static_cast<const T *>(a.beta);
    T *db = static_cast<T *>(a.dbeta);
    const int64_t threads = (int64_t)gridDim.x * PRO_THREADS;
    for (int64_t r = (int64_t)blockIdx.x * PRO_THREADS + threadIdx.x; r < a.rows; r += threads) {
      const float s = sigmoidf(to_f32(beta[r]));
      db[r] = from_f32<T>(to_f32(db[r]) * s * (1.f - s));
    }
  }
}

template <typename T>
cudaError_t launch_pair(const InputMapArgs &a, bool bwd, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // eight resident CTAs of 8 warps per SM, capped by the work (eight rows per warp and pass)
  const int rpw = bwd ? RPW_BWD : RPW;
  const int64_t passes = (2 * a.rows + rpw - 1) / rpw;
  const int64_t need = (passes + PRO_THREADS / 32 - 1) / (PRO_THREADS / 32);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sms * 8));
  if (bwd)
    epilogue_bwd_kernel<T><<<grid, PRO_THREADS, 0, st>>>(a);
  else
    prologue_kernel<T><<<grid, PRO_THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_input_maps(const InputMapArgs &a, bool bf16, bool backward, cudaStream_t st) {
  return bf16 ? launch_pair<__nv_bfloat16>(a, backward, st) : launch_pair<float>(a, backward, st);
}

}  // namespace gdn
