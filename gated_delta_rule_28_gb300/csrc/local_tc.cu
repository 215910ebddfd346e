// Local gradients of the chunked backward on bf16 tensor cores, scalar gate (sm_103a).
//
// One CTA of 8 warps per (chunk, head) computes dq, dk, dv, dbeta and dg of its chunk from
// the chunk's inputs, its entry state h, the gradient dh of its exit state and the gradient
// dN of v_new (the recompute's and the reverse recurrence's outputs, bf16 tiles in this
// kernel's shared-memory layout, fetched with bulk copies) -- the finalize stage of the backward
// (the KDA adapter's chunk_kda_bwd_finalize on the "Diff Coverage" page; the GDN adapter's
// chunk_gated_delta_rule_bwd contract). With gamma_i = b^(G_i), lambda_i = b^(G_last - G_i),
// Gamma_ij = b^(G_i - G_j) and X = (I + L)^-1 (the forward's A slot):
//
//   forward recompute   W = V - diag(gamma) K h,  N = X diag(beta) W           (v_new)
//   dZ = X^T dN:        dv = diag(beta) dZ,  dbeta += rowsum(dZ (.) W),  dY = -diag(beta) dZ
//   dX = (dN W^T) diag(beta) (lower part),  dL = -X^T (dX X^T) (strictly lower),
//                       dbeta += rowsum(dL (.) P),  dS_k = diag(beta) dL (.) Gamma
//   dA_qk = scale dO N^T (lower incl.),  dS_q = dA_qk (.) Gamma
//   dq = diag(gamma) scale dO h^T + dS_q K
//   dk = diag(gamma) dY h^T + diag(lambda) N dh^T + dS_k K + dS_k^T K + dS_q^T Q
//   dG_i from every exponential (gamma, lambda, Gamma, b^(G_last)); dg = reverse cumsum of dG
//
// with P = K K^T (.) Gamma (strictly lower). Every contraction is a bf16 mma.sync
// (m16n8k16, fp32 accumulation) whose operands come from 128-byte-swizzled shared-memory
// tiles through ldmatrix (transposed where the product needs it); dq and dk accumulate in
// registers over the phases; per-row reductions go through warp shuffles and one-writer
// slots summed in a fixed order, so the result does not depend on thread timing.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tc;
using namespace tile;

constexpr int NTH = 256;
// shared memory (bytes from a 1024-aligned base); tiles are bf16, 128-byte swizzled rows,
// columns in 64-wide K-blocks of rows x 128 bytes
constexpr int O_K = 0;            // K      [64 x 128]
constexpr int O_Q = 16384;        // Q      [64 x 128]
constexpr int O_H = 32768;        // h      [128 keys x 128 values]
constexpr int O_DO = 65536;       // dO     [64 x 128]
constexpr int O_DH = 81920;       // dh     [128 x 128]
constexpr int O_X = 114688;       // X      [64 x 64]
constexpr int O_XB = 122880;      // X diag(beta) [64 x 64], later dX
constexpr int O_W = 131072;       // V, then W = V - gamma K h, later T1 = dX X^T [64 x 64]
constexpr int O_DN = 147456;      // dN [64 x 128], later dS_k and dS_q [64 x 64] each
constexpr int O_N = 163840;       // N = v_new [64 x 128]
constexpr int O_DY = 180224;      // dY [64 x 128]
constexpr int O_SMALL = 196608;
constexpr int SMEM_BYTES = O_SMALL + 4096 + 1024;

struct __align__(16) Small {
  float G[64], gam[64], lam[64], beta[64];
  float part[6][64];   // per-row partial sums, one writer each: [column half][row] x 3
  float gl[8];         // per-warp partials of the G_last terms
  uint64_t ldbar;      // the chunk's tile copies
};
// TMA maps over q, k, v, dO ([token rows][H * 128] bf16, 64 x 64 boxes)
struct LocalMaps {
  TmaMap q, k, v, dO;
};
constexpr uint32_t WAIT_LIMIT = 1u << 22;
static_assert(sizeof(Small) <= 4096, "small state");

struct Tl {
  uint32_t base;  // shared-memory address
  int rows;       // rows of the stored tile
};
// address of 16-byte chunk c8 (column 8 c8) of `row`
__device__ __forceinline__ uint32_t toff(Tl t, int row, int c8) {
  return t.base + (uint32_t)((c8 >> 3) * t.rows * 128) + chunk_off(row, c8 & 7);
}
__device__ __forceinline__ float ldt(const uint8_t *sm, uint32_t sb, Tl t, int row, int col) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + (toff(t, row, col >> 3) - sb) + (col & 7) * 2));
}
// columns col, col + 1 (col even: the same 16-byte chunk) of `row`
__device__ __forceinline__ float2 ldt2(const uint8_t *sm, uint32_t sb, Tl t, int row, int col) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(sm + (toff(t, row, col >> 3) - sb) + (col & 7) * 2));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc[NT][4] += A[m0 .. m0+15][k] B[k][n0 .. n0+8 NT-1] over k in [0, 16 KS), one warp.
// A stored as (m, k) rows (at = false) or as (k, m) rows (at = true); B stored as (n, k) rows
// (bt = false) or as (k, n) rows (bt = true). NT even.
template <int KS, int NT>
__device__ __forceinline__ void wmma(float (&acc)[NT][4], Tl A, bool at, int m0, Tl B, bool bt, int n0, int lane) {
  const int q = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t af[4];
    if (!at)
      ldsm_x4(toff(A, m0 + (lane & 15), 2 * ks + (lane >> 4)), af);
    else
      ldsm_x4_trans(toff(A, 16 * ks + r8 + 8 * (q >> 1), (m0 >> 3) + (q & 1)), af);
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      const int nc = n0 + 16 * np;
      uint32_t x[4];
      if (!bt) {
        ldsm_x4(toff(B, nc + (lane & 15), 2 * ks + (lane >> 4)), x);
        mma16816(acc[2 * np], af, x[0], x[2]);
        mma16816(acc[2 * np + 1], af, x[1], x[3]);
      } else {
        ldsm_x4_trans(toff(B, 16 * ks + r8 + 8 * (q & 1), (nc >> 3) + (q >> 1)), x);
        mma16816(acc[2 * np], af, x[0], x[1]);
        mma16816(acc[2 * np + 1], af, x[2], x[3]);
      }
    }
  }
}
template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
}
// store a fragment block (rows m0 + g (+8), columns n0 + 8 j + 2 t (+1)) into a bf16 tile
template <int NT, class F>
__device__ __forceinline__ void put(uint8_t *sm, uint32_t sb, Tl T, const float (&acc)[NT][4], int m0, int n0,
                                    int lane, F f) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = m0 + g + 8 * hr, c = n0 + 8 * j + 2 * t;
      *reinterpret_cast<uint32_t *>(sm + (toff(T, r, c >> 3) - sb) + (c & 7) * 2) =
          pack_bf16(f(r, c, acc[j][2 * hr]), f(r, c + 1, acc[j][2 * hr + 1]));
    }
}
// sum over the four lanes of a fragment row (lanes 4 g .. 4 g + 3)
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

template <bool E2>
__global__ void __launch_bounds__(NTH, 1) local_tc_kernel(BwdArgs a, const __grid_constant__ LocalMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Small &sv = *reinterpret_cast<Small *>(sm + O_SMALL);
  const uint32_t sb = smem_u32(sm);
  const Tl tK{sb + O_K, 64}, tQ{sb + O_Q, 64}, tH{sb + O_H, 128}, tDO{sb + O_DO, 64}, tDH{sb + O_DH, 128};
  const Tl tX{sb + O_X, 64}, tXB{sb + O_XB, 64}, tW{sb + O_W, 64}, tDN{sb + O_DN, 64}, tN{sb + O_N, 64};
  const Tl tDY{sb + O_DY, 64}, tDX{sb + O_XB, 64}, tT1{sb + O_W, 64}, tSK{sb + O_DN, 64}, tSQ{sb + O_DN + 8192, 64};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = a.H, h = blockIdx.y;
  const int g = lane >> 2, t4 = lane & 3;
  const int64_t zc = blockIdx.x;
  const float lnb = E2 ? 0.69314718055994530942f : 1.f;
  const float scale = a.scale;
  const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
  __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(a.dq);
  __nv_bfloat16 *dk = static_cast<__nv_bfloat16 *>(a.dk);
  __nv_bfloat16 *dv = static_cast<__nv_bfloat16 *>(a.dv);
  __nv_bfloat16 *dbeta = static_cast<__nv_bfloat16 *>(a.dbeta);

  // ---- the chunk ----------------------------------------------------------------------
  int64_t c0, slot;
  int n;
  if (a.cu) {
    const int seq = a.chunk_indices[2 * zc], cc = a.chunk_indices[2 * zc + 1];
    bool ok = seq >= 0 && seq < a.num_seqs && cc >= 0;
    c0 = 0;
    n = 0;
    if (ok) {
      c0 = a.cu[seq] + (int64_t)cc * GDN_CHUNK;
      ok = c0 < a.cu[seq + 1] && a.cu[seq + 1] <= a.T;
      n = ok ? (int)min((int64_t)GDN_CHUNK, (int64_t)a.cu[seq + 1] - c0) : 0;
    }
    if (!ok) {
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      return;
    }
    slot = zc * H + h;
  } else {
    const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
    const int b = (int)(zc / NT), cc = (int)(zc % NT);
    c0 = (int64_t)b * a.T + (int64_t)cc * GDN_CHUNK;
    n = min(GDN_CHUNK, a.T - cc * GDN_CHUNK);
    slot = ((int64_t)b * H + h) * NT + cc;
  }
  auto row_of = [&](int i) { return (c0 + i) * H + h; };

  if (tid == 0) {
    mbar_init(&sv.ldbar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // ---- loads: the gate, beta and X (rows past the end: identity) into registers first, so
  // that they do not queue behind the tiles; then the tiles (below) ----------------------------
  float G_t = 0.f, beta_t = 0.f;
  if (tid < 64) {
    G_t = a.g_cumsum[row_of(min(tid, n - 1))];
    if (tid < n) beta_t = __bfloat162float(beta[row_of(tid)]);
  }
  float4 xr[2][2];  // X row x >> 3, columns 8 (x & 7) .. +7, for x = tid, tid + 256
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int x = tid + u * NTH, r = x >> 3, c8 = x & 7;
    const float4 *src = reinterpret_cast<const float4 *>(a.A + row_of(r < n ? r : 0) * GDN_CHUNK + 8 * c8);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) xr[u][hh] = r < n ? __ldg(src + hh) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // the tiles: q, k, v, dO as two 64 x 64 TMA boxes each (rows past the chunk's end hold the
  // tensor's next rows, zeroed below), h, dh and dN (already in this layout) as bulk copies
  if (warp == 0) {
    uint64_t *bar = &sv.ldbar;
    const int y = (int)c0, x0 = h * GDN_DK;
    mbar_expect_tx_w(bar, 4 * 16384 + 2 * 32768 + 16384);
    tma_load_2d_w(sb + O_K, &maps.k, x0, y, bar);
    tma_load_2d_w(sb + O_K + 8192, &maps.k, x0 + 64, y, bar);
    tma_load_2d_w(sb + O_Q, &maps.q, x0, y, bar);
    tma_load_2d_w(sb + O_Q + 8192, &maps.q, x0 + 64, y, bar);
    tma_load_2d_w(sb + O_W, &maps.v, x0, y, bar);
    tma_load_2d_w(sb + O_W + 8192, &maps.v, x0 + 64, y, bar);
    tma_load_2d_w(sb + O_DO, &maps.dO, x0, y, bar);
    tma_load_2d_w(sb + O_DO + 8192, &maps.dO, x0 + 64, y, bar);
    bulk_load_w(sb + O_H, a.h_tiles + slot * STATE_TILE, 32768, bar);
    bulk_load_w(sb + O_DH, a.dh_tiles + slot * STATE_TILE, 32768, bar);
    bulk_load_w(sb + O_DN, a.dv_tiles + slot * DV_TILE, 16384, bar);
  }
  if (tid < 64) {
    sv.G[tid] = G_t;
    sv.beta[tid] = beta_t;
    sv.gam[tid] = gexp<E2>(G_t);
  }
  __syncthreads();  // beta and the gate of every row are in place
  if (tid < 64) sv.lam[tid] = gexp<E2>(sv.G[63] - sv.G[tid]);
  // X (rows i, columns j; identity outside the chunk) and X diag(beta)
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int x = tid + u * NTH, r = x >> 3, c8 = x & 7;
    const float raw[8] = {xr[u][0].x, xr[u][0].y, xr[u][0].z, xr[u][0].w,
                          xr[u][1].x, xr[u][1].y, xr[u][1].z, xr[u][1].w};
    float xv[8], xb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = 8 * c8 + e;
      xv[e] = (r < n && j < n) ? raw[e] : (r == j ? 1.f : 0.f);
      xb[e] = xv[e] * sv.beta[j];
    }
    *reinterpret_cast<uint4 *>(sm + (toff(tX, r, c8) - sb)) = pack8(xv);
    *reinterpret_cast<uint4 *>(sm + (toff(tXB, r, c8) - sb)) = pack8(xb);
  }
  const bool late = !mbar_wait(&sv.ldbar, 0, WAIT_LIMIT);
  if (__syncthreads_or(late)) {  // the tiles did not arrive: report, let the copies land, leave
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    mbar_wait(&sv.ldbar, 0, WAIT_LIMIT);
    return;
  }
  // rows past the chunk's end are zero in K, Q, V, dO (the boxes hold the tensor's next rows)
  // and dN (the tile holds whatever the reverse recurrence computed there); <dh, h> over the
  // whole state for the gradient of the last gate
  if (n < 64)
    for (int x = tid; x < (64 - n) * 16; x += NTH) {
      const int r = n + x / 16, c16 = x % 16;
      const uint4 z = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4 *>(sm + (toff(tK, r, c16) - sb)) = z;
      *reinterpret_cast<uint4 *>(sm + (toff(tQ, r, c16) - sb)) = z;
      *reinterpret_cast<uint4 *>(sm + (toff(tW, r, c16) - sb)) = z;
      *reinterpret_cast<uint4 *>(sm + (toff(tDO, r, c16) - sb)) = z;
      *reinterpret_cast<uint4 *>(sm + (toff(tDN, r, c16) - sb)) = z;
    }
  {
    float hdh = 0.f;
    for (int x = tid; x < 2048; x += NTH) {  // the same swizzle in both tiles: element-wise
      float hv[8], dv8[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + O_H + 16 * x), hv);
      unpack8(*reinterpret_cast<const uint4 *>(sm + O_DH + 16 * x), dv8);
#pragma unroll
      for (int e = 0; e < 8; ++e) hdh = fmaf(hv[e], dv8[e], hdh);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) hdh += __shfl_xor_sync(0xffffffffu, hdh, off);
    if (lane == 0) sv.gl[warp] = hdh;
  }
  __syncthreads();

  // warp tile of the 64 x 128 products: rows m0 .. +15, columns n0 .. +63
  const int m0 = 16 * (warp & 3), n0 = 64 * (warp >> 2), hw = warp >> 2;
  float dqa[8][4], dka[8][4];
  zero(dqa);
  zero(dka);
  // per-row partial sums (rows m0 + g, m0 + g + 8): dbeta, dG, and the G_last terms
  float pb[2] = {0.f, 0.f}, pg[2] = {0.f, 0.f}, plast = 0.f;
  auto tile_val = [&](Tl T, int r, int c) { return ldt(sm, sb, T, r, c); };
  auto tile_val2 = [&](Tl T, int r, int c) { return ldt2(sm, sb, T, r, c); };

  // ---- 1. W = V - diag(gamma) K h (in place of V) ----------------------------------------
  {
    float acc[8][4];
    zero(acc);
    wmma<8, 8>(acc, tK, false, m0, tH, true, n0, lane);
    // each element of V is read and rewritten by the one thread that owns its fragment
    put<8>(sm, sb, tW, acc, m0, n0, lane, [&](int r, int c, float y) { return tile_val(tW, r, c) - sv.gam[r] * y; });
  }
  __syncthreads();
  // ---- 2. N = X diag(beta) W --------------------------------------------------------------
  {
    float acc[8][4];
    zero(acc);
    wmma<4, 8>(acc, tXB, false, m0, tW, true, n0, lane);
    put<8>(sm, sb, tN, acc, m0, n0, lane, [](int, int, float y) { return y; });
  }
  // ---- 3. dZ = X^T dN: dv = beta dZ, dbeta += rowsum(dZ W), dY = -beta dZ ---------------------
  {
    float acc[8][4];
    zero(acc);
    wmma<4, 8>(acc, tX, true, m0, tDN, true, n0, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = m0 + g + 8 * hr, c = n0 + 8 * j + 2 * t4;
        const float2 w2 = tile_val2(tW, r, c);
        pb[hr] = fmaf(acc[j][2 * hr], w2.x, pb[hr]);
        pb[hr] = fmaf(acc[j][2 * hr + 1], w2.y, pb[hr]);
        if (r < n) {
          const float bt = sv.beta[r];
          *reinterpret_cast<uint32_t *>(dv + row_of(r) * GDN_DV + c) = pack_bf16(bt * acc[j][2 * hr], bt * acc[j][2 * hr + 1]);
        }
      }
    put<8>(sm, sb, tDY, acc, m0, n0, lane, [&](int r, int, float z) { return -sv.beta[r] * z; });
  }
  __syncthreads();  // N, dY complete; W still in use below
  // ---- 4. dX = (dN W^T) diag(beta), lower blocks (upper blocks zero) --------------------------
  for (int b = warp; b < 16; b += 8) {
    const int bi = b >> 2, bj = b & 3;
    float acc[2][4];
    zero(acc);
    if (bj <= bi) wmma<8, 2>(acc, tDN, false, 16 * bi, tW, false, 16 * bj, lane);
    put<2>(sm, sb, tDX, acc, 16 * bi, 16 * bj, lane, [&](int, int c, float y) { return y * sv.beta[c]; });
  }
  __syncthreads();  // dX complete; W and dN are free (T1, dS_k, dS_q take their place)
  // ---- 5. dA_qk = scale dO N^T (lower incl.), A_qk = Q K^T (.) Gamma: dS_q, and the dG terms of
  //         the intra-chunk gate come with the products below --------------------------------
  for (int b = warp; b < 16; b += 8) {
    const int bi = b >> 2, bj = b & 3;
    float acc[2][4];
    zero(acc);
    if (bj <= bi) wmma<8, 2>(acc, tDO, false, 16 * bi, tN, false, 16 * bj, lane);
    put<2>(sm, sb, tSQ, acc, 16 * bi, 16 * bj, lane, [&](int r, int c, float y) {
      return c <= r ? scale * y * gexp<E2>(sv.G[r] - sv.G[c]) : 0.f;
    });
  }
  // T1 = dX X^T (full)
  for (int b = warp; b < 16; b += 8) {
    const int bi = b >> 2, bj = b & 3;
    float acc[2][4];
    zero(acc);
    wmma<4, 2>(acc, tDX, false, 16 * bi, tX, false, 16 * bj, lane);
    put<2>(sm, sb, tT1, acc, 16 * bi, 16 * bj, lane, [](int, int, float y) { return y; });
  }
  // ---- 6. dQg = scale dO h^T: dq += gamma dQg, dG += lnb gamma rowsum(dQg Q) ------------------
  {
    float acc[8][4];
    zero(acc);
    wmma<8, 8>(acc, tDO, false, m0, tH, false, n0, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = m0 + g + 8 * hr, c = n0 + 8 * j + 2 * t4;
        const float gm = sv.gam[r];
        const float2 q2 = tile_val2(tQ, r, c);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float d = scale * acc[j][2 * hr + e];
          dqa[j][2 * hr + e] = gm * d;
          pg[hr] = fmaf(lnb * gm * d, e ? q2.y : q2.x, pg[hr]);
        }
      }
  }
  // ---- 7. dKl = N dh^T: dk += lambda dKl, dG -= lnb lambda rowsum(dKl K), G_last term ---------
  {
    float acc[8][4];
    zero(acc);
    wmma<8, 8>(acc, tN, false, m0, tDH, false, n0, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = m0 + g + 8 * hr, c = n0 + 8 * j + 2 * t4;
        const float la = sv.lam[r];
        const float2 k2 = tile_val2(tK, r, c);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float d = la * acc[j][2 * hr + e];
          dka[j][2 * hr + e] = d;
          const float w = lnb * d * (e ? k2.y : k2.x);
          pg[hr] -= w;
          plast += w;
        }
      }
  }
  // ---- 8. dKg = dY h^T: dk += gamma dKg, dG += lnb gamma rowsum(dKg K) -------------------------
  {
    float acc[8][4];
    zero(acc);
    wmma<8, 8>(acc, tDY, false, m0, tH, false, n0, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = m0 + g + 8 * hr, c = n0 + 8 * j + 2 * t4;
        const float gm = sv.gam[r];
        const float2 k2 = tile_val2(tK, r, c);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float d = gm * acc[j][2 * hr + e];
          dka[j][2 * hr + e] += d;
          pg[hr] = fmaf(lnb * d, e ? k2.y : k2.x, pg[hr]);
        }
      }
  }
  __syncthreads();  // T1 and dS_q complete
  // ---- 9. dL = -X^T T1 (strictly lower); P = K K^T (.) Gamma: dbeta += rowsum(dL P),
  //         dS_k = diag(beta) dL (.) Gamma ---------------------------------------------------------
  for (int b = warp; b < 16; b += 8) {
    const int bi = b >> 2, bj = b & 3;
    float acc[2][4], pk[2][4];
    zero(acc);
    zero(pk);
    if (bj <= bi) {
      wmma<4, 2>(acc, tX, true, 16 * bi, tT1, true, 16 * bj, lane);
      wmma<8, 2>(pk, tK, false, 16 * bi, tK, false, 16 * bj, lane);
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = 16 * bi + g + 8 * hr, c = 16 * bj + 8 * j + 2 * t4 + e;
          const float gam = c < r ? gexp<E2>(sv.G[r] - sv.G[c]) : 0.f;
          const float dl = -acc[j][2 * hr + e];
          rs[hr] = fmaf(dl, pk[j][2 * hr + e] * gam, rs[hr]);
          acc[j][2 * hr + e] = sv.beta[r] * dl * gam;  // dS_k
        }
    put<2>(sm, sb, tSK, acc, 16 * bi, 16 * bj, lane, [](int, int, float y) { return y; });
    // dbeta from dL: the quad's lanes, then one writer per (column block, row): slots 2 .. 5
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const float s = quad_sum(rs[hr]);
      if (t4 == 0) sv.part[2 + bj][16 * bi + g + 8 * hr] = s;
    }
  }
  __syncthreads();  // dS_k complete
  // ---- 10. dq += dS_q K; dk += dS_k K + dS_k^T K + dS_q^T Q, with the dG terms of Gamma ---------
  {
    float acc[8][4];
#pragma unroll 1
    for (int which = 0; which < 4; ++which) {
      zero(acc);
      const Tl M = which < 2 ? tSK : tSQ;
      const bool tr = which == 1 || which == 3;
      wmma<4, 8>(acc, which == 2 ? tSQ : M, tr, m0, which == 3 ? tQ : tK, true, n0, lane);
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = m0 + g + 8 * hr, c = n0 + 8 * j + 2 * t4;
          const float2 o2 = tile_val2(which == 2 ? tQ : tK, r, c);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float d = acc[j][2 * hr + e];
            const float w = lnb * d * (e ? o2.y : o2.x);
            if (which == 2) {
              dqa[j][2 * hr + e] += d;
              pg[hr] += w;
            } else {
              dka[j][2 * hr + e] += d;
              pg[hr] += (which == 0) ? w : -w;
            }
          }
        }
    }
  }
  // ---- write dq, dk; per-row reductions -----------------------------------------------------
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int r = m0 + g + 8 * hr, c = n0 + 8 * j + 2 * t4;
      if (r < n) {
        *reinterpret_cast<uint32_t *>(dq + row_of(r) * GDN_DK + c) = pack_bf16(dqa[j][2 * hr], dqa[j][2 * hr + 1]);
        *reinterpret_cast<uint32_t *>(dk + row_of(r) * GDN_DK + c) = pack_bf16(dka[j][2 * hr], dka[j][2 * hr + 1]);
      }
    }
  // dbeta from dZ: one writer per (column half, row), slots 0 and 1
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const float b1 = quad_sum(pb[hr]);
    pg[hr] = quad_sum(pg[hr]);
    if (t4 == 0) sv.part[hw][m0 + g + 8 * hr] = b1;
  }
  // dG per column half goes through slots 0 and 1 once dbeta has been summed
  plast = quad_sum(plast);
  plast += __shfl_xor_sync(0xffffffffu, plast, 4);
  plast += __shfl_xor_sync(0xffffffffu, plast, 8);
  plast += __shfl_xor_sync(0xffffffffu, plast, 16);
  __syncthreads();  // dbeta partials of every warp are in place; gl holds <dh, h> per warp
  float dbeta_row = 0.f;
  if (tid < 64) dbeta_row = sv.part[0][tid] + sv.part[1][tid] + sv.part[2][tid] + sv.part[3][tid] +
                            sv.part[4][tid] + sv.part[5][tid];
  float hdh_all = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) hdh_all += sv.gl[w];
  __syncthreads();  // the slots are reused for dG below
  if (t4 == 0) {
    sv.part[hw][m0 + g] = pg[0];
    sv.part[hw][m0 + g + 8] = pg[1];
  }
  if (lane == 0) sv.gl[warp] = plast;
  if (tid < 64 && tid < n) dbeta[row_of(tid)] = __float2bfloat16_rn(dbeta_row);
  __syncthreads();
  if (warp == 0) {  // the reverse cumulative sum over the chunk's rows, two rows per lane
    float extra = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) extra += sv.gl[w];
    extra += lnb * gexp<E2>(sv.G[63]) * hdh_all;
    const int i0 = 2 * lane, i1 = i0 + 1;
    const float x0 = i0 < n ? sv.part[0][i0] + sv.part[1][i0] + (i0 == n - 1 ? extra : 0.f) : 0.f;
    const float x1 = i1 < n ? sv.part[0][i1] + sv.part[1][i1] + (i1 == n - 1 ? extra : 0.f) : 0.f;
    float incl = x0 + x1;  // then: the sum over the rows of this lane and every later lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_down_sync(0xffffffffu, incl, off);
      if (lane + off < 32) incl += y;
    }
    float later = __shfl_down_sync(0xffffffffu, incl, 1);
    if (lane == 31) later = 0.f;
    const float run1 = x1 + later;
    if (i1 < n) a.dg[row_of(i1)] = run1;
    if (i0 < n) a.dg[row_of(i0)] = x0 + run1;
  }
}

}  // namespace

cudaError_t launch_bwd_local_tc(const BwdArgs &a, cudaStream_t st) {
  auto kern = a.use_exp2 ? local_tc_kernel<true> : local_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int64_t nch = a.cu ? a.num_chunks : (int64_t)a.B * ((a.T + GDN_CHUNK - 1) / GDN_CHUNK);
  if (nch == 0) return cudaSuccess;
  const uint64_t rows = a.cu ? (uint64_t)a.T : (uint64_t)a.B * a.T;  // token rows (32-bit TMA rows)
  if (rows > (uint64_t)INT32_MAX) return cudaErrorInvalidValue;
  const uint64_t pitch = (uint64_t)a.H * GDN_DK * 2;
  LocalMaps maps;
  e = make_tmap_bf16(&maps.q, a.q, (uint64_t)a.H * GDN_DK, rows, pitch);
  if (e == cudaSuccess) e = make_tmap_bf16(&maps.k, a.k, (uint64_t)a.H * GDN_DK, rows, pitch);
  if (e == cudaSuccess) e = make_tmap_bf16(&maps.v, a.v, (uint64_t)a.H * GDN_DV, rows, (uint64_t)a.H * GDN_DV * 2);
  if (e == cudaSuccess) e = make_tmap_bf16(&maps.dO, a.dO, (uint64_t)a.H * GDN_DV, rows, (uint64_t)a.H * GDN_DV * 2);
  if (e != cudaSuccess) return e;
  kern<<<dim3((unsigned)nch, a.H), NTH, SMEM_BYTES, st>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace gdn
