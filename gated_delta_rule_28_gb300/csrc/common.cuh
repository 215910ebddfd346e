// Shared device helpers for the gated-delta-rule kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define GDN_CHUNK 64
#define GDN_DK 128
#define GDN_DV 128

namespace gdn {

// Error word raised by kernels that meet inconsistent device metadata or a
// bounded wait that ran out; read and cleared by gdn_device_status().
enum : int { kDevOk = 0, kDevCheck = 1, kDevTimeout = 2 };

__device__ __forceinline__ void raise_device_flag(int* flag, int code) {
  if (flag) atomicMax(flag, code);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Decay base: exp(x) for natural gates, 2^x for base-2 gates (IEEE-accurate
// library calls; the fast paths use their own approximations).
__device__ __forceinline__ float gate_pow(float x, bool exp2_base) {
  return exp2_base ? exp2f(x) : expf(x);
}

// Token range of one independent run (a batch row, a packed document, or a
// segment of a batch row) in flattened rows of the [rows, H, D] layout.
struct RunRange {
  int64_t r0, r1;     // first and one-past-last flattened row
  int64_t chunk0;     // index of the run's first chunk in the h_chunks layout
};

}  // namespace gdn

namespace gdn {

// Register-tiled product over shared-memory operands for a 256-thread CTA:
// acc[i][j] += sum_kk fa(m0 + i, kk) * fb(kk, n0 + j), where the thread owns
// rows m0 .. m0+TM-1 and columns n0 .. n0+TN-1 of an M x N output.
template <int M, int N, int KD, int TM, int TN, class FA, class FB>
__device__ __forceinline__ void mm_acc(FA fa, FB fb, float (&acc)[TM][TN], int tid) {
  static_assert((M / TM) * (N / TN) == 256, "tile grid must cover 256 threads");
  const int tx = tid % (N / TN), ty = tid / (N / TN);
  const int m0 = ty * TM, n0 = tx * TN;
#pragma unroll 4
  for (int kk = 0; kk < KD; ++kk) {
    float av[TM], bv[TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) av[i] = fa(m0 + i, kk);
#pragma unroll
    for (int j = 0; j < TN; ++j) bv[j] = fb(kk, n0 + j);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
}

// Warp-level tf32 tensor-core product over fp32 shared-memory operands (mma.sync
// m16n8k8, fp32 accumulation): the warp's 16 x (8 NT) block of an output at rows
// r0 .. r0+15 and columns c0 .. c0+8NT-1, acc[j] holding the fragment of columns
// c0+8j .. +7 (thread: rows r0 + lane/4 (+8), columns 2(lane%4) (+1)), accumulated over
// KD (a multiple of 8) steps of fa(m, kk) fb(kk, n). The operands are rounded to tf32.
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
template <int KD, int NT, class FA, class FB>
__device__ __forceinline__ void mma_tf32_acc(FA fa, FB fb, float (&acc)[NT][4], int r0, int c0, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int k0 = 0; k0 < KD; k0 += 8) {
    const uint32_t a0 = to_tf32(fa(r0 + g, k0 + t)), a1 = to_tf32(fa(r0 + g + 8, k0 + t));
    const uint32_t a2 = to_tf32(fa(r0 + g, k0 + t + 4)), a3 = to_tf32(fa(r0 + g + 8, k0 + t + 4));
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const uint32_t b0 = to_tf32(fb(k0 + t, c0 + 8 * j + g)), b1 = to_tf32(fb(k0 + t + 4, c0 + 8 * j + g));
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+f"(acc[j][0]), "+f"(acc[j][1]), "+f"(acc[j][2]), "+f"(acc[j][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}
// store such a fragment block into a row-major shared-memory matrix (row stride ld floats)
template <int NT>
__device__ __forceinline__ void mma_frag_store(float *dst, int ld, const float (&acc)[NT][4], int r0, int c0, int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int c = c0 + 8 * j + 2 * t;
    dst[(r0 + g) * ld + c] = acc[j][0];
    dst[(r0 + g) * ld + c + 1] = acc[j][1];
    dst[(r0 + g + 8) * ld + c] = acc[j][2];
    dst[(r0 + g + 8) * ld + c + 1] = acc[j][3];
  }
}

template <int M, int N, int TM, int TN>
__device__ __forceinline__ void tile_origin(int tid, int& m0, int& n0) {
  m0 = (tid / (N / TN)) * TM;
  n0 = (tid % (N / TN)) * TN;
}

template <int TM, int TN>
__device__ __forceinline__ void zero_acc(float (&acc)[TM][TN]) {
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
}

}  // namespace gdn
