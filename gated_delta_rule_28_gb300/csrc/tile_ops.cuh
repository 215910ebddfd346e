// Shared-memory tile helpers of the tensor-core chunk kernels (sm_103a):
// cp.async staging, bf16 packing, the 128-byte-swizzled K-major tile layout,
// 16x16 transposes with ldmatrix/stmatrix, and the blocked fp32 solve
// X = (I + L)^-1 of a strictly-lower 64x64 L (16x16 diagonal blocks by
// elimination, off-diagonal block levels with tf32 mma.sync).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {
namespace tile {
namespace {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// decay factor base^x: base 2 (E2) or e, chosen at compile time
template <bool E2>
__device__ __forceinline__ float gexp(float x) { return E2 ? exp2f(x) : __expf(x); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&t);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}
__device__ __forceinline__ uint4 pack8(const float *f) {
  uint4 u;
  u.x = pack_bf16(f[0], f[1]);
  u.y = pack_bf16(f[2], f[3]);
  u.z = pack_bf16(f[4], f[5]);
  u.w = pack_bf16(f[6], f[7]);
  return u;
}
__device__ __forceinline__ void unpack8(uint4 u, float *f) {
  const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y), c = unpack_bf16(u.z), d = unpack_bf16(u.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y; f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}
// byte offset of 16-byte chunk c8 of row `row` in a 128-byte-row swizzled tile
__device__ __forceinline__ uint32_t chunk_off(int row, int c8) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + (((c8 ^ row) & 7) << 4));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// --- blocked 64x64 fp32 matrices for the solve ------------------------------------------
__device__ __forceinline__ int blk(int bi, int bj) { return bi * (bi + 1) / 2 + bj; }
__device__ __forceinline__ int bsw(int r, int c) { return r * 16 + (c ^ (((r >> 1) & 3) << 2)); }

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// acc (16x16 as two 16x8 tiles) += A (16x16) B (16x16), tf32 inputs, fp32 accumulate
__device__ __forceinline__ void mm16_tf32(const float *A, const float *B, float (&acc)[2][4], int lane) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int kk = 0; kk < 16; kk += 8) {
    const uint32_t a0 = to_tf32(A[bsw(g, kk + t)]), a1 = to_tf32(A[bsw(g + 8, kk + t)]);
    const uint32_t a2 = to_tf32(A[bsw(g, kk + t + 4)]), a3 = to_tf32(A[bsw(g + 8, kk + t + 4)]);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint32_t b0 = to_tf32(B[bsw(kk + t, nt * 8 + g)]);
      const uint32_t b1 = to_tf32(B[bsw(kk + t + 4, nt * 8 + g)]);
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
          "{%0,%1,%2,%3};"
          : "+f"(acc[nt][0]), "+f"(acc[nt][1]), "+f"(acc[nt][2]), "+f"(acc[nt][3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
  }
}
__device__ __forceinline__ void acc_store(float *C, const float (&acc)[2][4], int lane, float sign) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    C[bsw(g, nt * 8 + 2 * t)] = sign * acc[nt][0];
    C[bsw(g, nt * 8 + 2 * t + 1)] = sign * acc[nt][1];
    C[bsw(g + 8, nt * 8 + 2 * t)] = sign * acc[nt][2];
    C[bsw(g + 8, nt * 8 + 2 * t + 1)] = sign * acc[nt][3];
  }
}

__device__ __forceinline__ void solve_group_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// X = (I + L)^-1 from the lower 16x16 blocks of a strictly-lower L; called by
// warps 0..3 only (named barrier 1).
__device__ void solve_blocks(const float *L, float *X, float *T, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  {  // diagonal block `warp`: fp32 row elimination, rows 2k + half of column c per thread
    const int b = warp, c = lane & 15, half = lane >> 4;
    const float *Lb = L + blk(b, b) * 256;
    float x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = (2 * k + half == c) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 15; ++j) {  // row j is final: remove L[r][j] row_j from rows r > j
      const float xj = __shfl_sync(0xffffffffu, x[j >> 1], c + 16 * (j & 1));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int r = 2 * k + half;
        if (2 * k + 1 > j && r > j) x[k] = fmaf(-Lb[bsw(r, j)], xj, x[k]);
      }
    }
    float *Xb = X + blk(b, b) * 256;
#pragma unroll
    for (int k = 0; k < 8; ++k) Xb[bsw(2 * k + half, c)] = x[k];
  }
  solve_group_sync();
  // 32x32 halves: X_10 = -X_11 L_10 X_00 and X_32 = -X_33 L_32 X_22 (warps 0, 1)
  if (warp < 2) {
    const int b0 = 2 * warp, b1 = b0 + 1;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    mm16_tf32(L + blk(b1, b0) * 256, X + blk(b0, b0) * 256, acc, lane);
    float *Tw = T + warp * 256;
    acc_store(Tw, acc, lane, 1.f);
    __syncwarp();
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    mm16_tf32(X + blk(b1, b1) * 256, Tw, acc2, lane);
    acc_store(X + blk(b1, b0) * 256, acc2, lane, -1.f);
  }
  solve_group_sync();
  // lower-left 32x32: Tb = L_bt X_top, then X_bt = -X_bot Tb (one 16x16 block per warp)
  {
    const int r = 2 + (warp >> 1), cc = warp & 1;  // block (r, cc), r in {2,3}, cc in {0,1}
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int kb = cc; kb < 2; ++kb) mm16_tf32(L + blk(r, kb) * 256, X + blk(kb, cc) * 256, acc, lane);
    acc_store(T + warp * 256, acc, lane, 1.f);  // T block (r, cc), in warp order
  }
  solve_group_sync();
  {
    const int r = 2 + (warp >> 1), cc = warp & 1;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int kb = 2; kb <= r; ++kb)  // X_bot rows r, columns kb; T rows kb (warp 2*(kb-2)+cc)
      mm16_tf32(X + blk(r, kb) * 256, T + (2 * (kb - 2) + cc) * 256, acc, lane);
    acc_store(X + blk(r, cc) * 256, acc, lane, -1.f);
  }
  solve_group_sync();
}

}  // namespace
}  // namespace tile
}  // namespace gdn
