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
// Memory-bound elementwise work: one warp per row, each lane four consecutive
// elements (one 8-byte bf16 or 16-byte fp32 vector), the row sum by warp
// shuffles; grid-stride over rows with a grid of whole waves of the SMs. The
// norm is computed in fp32 from the stored inputs (the backward recomputes it
// from the raw rows rather than reading a saved rstd).
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int PRO_THREADS = 256;
constexpr float L2_EPS = 1e-6f;

template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
  using type = float4;
  __device__ static void load(const float *p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  __device__ static void store(float *p, const float (&x)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};
template <>
struct Vec4<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16 *p, float (&x)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  }
  __device__ static void store(__nv_bfloat16 *p, const float (&x)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(x[2], x[3]);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t *>(&a);
    v.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = v;
  }
};

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
  for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

__device__ __forceinline__ float sigmoidf(float x) { return 1.f / (1.f + __expf(-x)); }

template <typename T>
__global__ void __launch_bounds__(PRO_THREADS) prologue_kernel(InputMapArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (PRO_THREADS / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (PRO_THREADS / 32) + (threadIdx.x >> 5);
  const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k);
  T *qn = static_cast<T *>(a.qn), *kn = static_cast<T *>(a.kn);
  if (a.l2norm) {
    for (int64_t r = w0; r < 2 * a.rows; r += warps) {  // rows of q, then rows of k
      const bool isq = r < a.rows;
      if (isq && !q) continue;
      const int64_t off = (isq ? r : r - a.rows) * GDN_DK + 4 * lane;
      float x[4];
      Vec4<T>::load((isq ? q : k) + off, x);
      const float rstd = rsqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]) + L2_EPS);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] *= rstd;
      Vec4<T>::store((isq ? qn : kn) + off, x);
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
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (PRO_THREADS / 32);
  const int64_t w0 = (int64_t)blockIdx.x * (PRO_THREADS / 32) + (threadIdx.x >> 5);
  const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k);
  T *dq = static_cast<T *>(a.dq), *dk = static_cast<T *>(a.dk);
  if (a.l2norm) {
    for (int64_t r = w0; r < 2 * a.rows; r += warps) {
      const bool isq = r < a.rows;
      const int64_t off = (isq ? r : r - a.rows) * GDN_DK + 4 * lane;
      float x[4], d[4];
      Vec4<T>::load((isq ? q : k) + off, x);
      Vec4<T>::load((isq ? dq : dk) + off, d);
      const float rstd = rsqrtf(warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]) + L2_EPS);
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] *= rstd;  // xn
      const float dot = warp_sum(x[0] * d[0] + x[1] * d[1] + x[2] * d[2] + x[3] * d[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) d[i] = rstd * (d[i] - x[i] * dot);
      Vec4<T>::store((isq ? dq : dk) + off, d);
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
  // four resident CTAs of 8 warps per SM, capped by the work (one warp per row)
  const int64_t need = (2 * a.rows + PRO_THREADS / 32 - 1) / (PRO_THREADS / 32);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(need, (int64_t)sms * 4));
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
