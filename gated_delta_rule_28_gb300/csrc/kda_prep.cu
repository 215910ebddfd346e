// Per-key (KDA) preparation of every 64-token chunk, for all chunks and heads at
// once (bf16 inputs, sm_103a): everything of the chunk algorithm that does not
// depend on the state (the KDA adapter's chunk_kda_fwd_prepare stage on the
// "Diff Coverage" page; the per-key gate of "state_summary.py"
// kda_split_state_summary_kernel, where the decay is applied per key channel):
//
//   G     = in-chunk cumulative log-gate, per key channel
//   Gamma_ij,d = b^(G_id - G_jd)                         (b = 2 or e)
//   L     = strictly-lower(diag(beta) (K K^T (.) Gamma)),  X = (I + L)^-1
//   A_qk  = lower-incl(Q K^T (.) Gamma)
//   w     = X diag(beta) (K (.) b^G),  u = X diag(beta) V
//   and the operands K (.) b^(G_last - G), Q (.) b^G, b^(G_last) of the state recurrence.
//
// The gated Gram matrices run on bf16 tensor cores (mma.sync) through one
// reference row per chunk (r = 32, the middle): with e_id = b^(G_id - G_rd),
//   (K K^T (.) Gamma)_ij = sum_d (k_id e_id) (k_jd / e_jd),
// and the same for Q K^T; K (.) b^G = (K (.) e) Diag(b^(G_r)), so w is formed from
// the same tile, and K (.) b^(G_last - G) = (K / e) Diag(b^(G_last - G_r)). Every
// element then costs one exponential and one reciprocal. A chunk in which some
// |G_id - G_rd| exceeds 100 (in base 2) would leave the range of fp32 and bf16;
// it is computed term by term instead, with one exponential per (i, j, d) for the
// Gram matrices and direct exponentials for the factors, exactly for any gate range.
//
// The outputs go to one blob per (chunk, head), in the 128-byte-swizzled
// layout the chain kernel's operands take in shared memory (kernels.h, kda::).
// Persistent CTAs of 8 warps, two per SM (about 100 KB of shared memory each):
// every global load of an item (K, Q, V by cp.async, the gate column of each
// thread) is issued at once, and one CTA's loads overlap the other's compute.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tc;
using namespace tile;
using namespace kda;

constexpr int NTH = 256;
constexpr int REF = 32;   // reference row of the Gram factorisation
constexpr int GS = 132;   // row stride (floats) of G: 16-byte aligned, rows shift by 4 banks
// shared memory map (bytes from a 1024-aligned base); swizzled bf16 tiles hold 64 rows as
// two K-blocks of 64 columns (8 KB apart)
constexpr int OFF_G = 0;                // G fp32 [64][GS]; once the factors exist: L, X, T
constexpr int OFF_K = OFF_G + 34816;    // K, then K e (Gram A and B of w), or K b^G (exact)
constexpr int OFF_Q = OFF_K + 16384;    // Q, then Q e (Gram A), then X diag(beta) in bf16
constexpr int OFF_V = OFF_Q + 16384;    // V (B of u)
constexpr int OFF_KB = OFF_V + 16384;   // K / e (Gram B); exact chunks: L while G is in use
constexpr int OFF_SMALL = OFF_KB + 16384;
constexpr int SMEM_BYTES = OFF_SMALL + 2048 + 1024;
constexpr int L_FLOATS = 10 * 256, X_FLOATS = 10 * 256;  // lower 16x16 blocks (blk / bsw)
constexpr int OFF_AQS = OFF_G + 24576;  // A_qk staged for its bulk copy, after L, X and T
static_assert(64 * GS * 4 <= 34816 && (L_FLOATS + X_FLOATS + 4 * 256) * 4 <= 24576 && 24576 + 8192 <= 34816,
              "G region: G; then L, X, T and the staged A_qk; then the staged u");

// largest |exponent| (base 2) a factor may take on the tensor-core path
constexpr float EXP_LIMIT = 100.f;

struct __align__(16) Small {
  uint64_t ldbar;  // the item's tile copies
  uint64_t pad;
  float beta[64];
  float part[128];
  float eref[128];  // b^(G_r) per key channel
  float elr[128];   // b^(G_last - G_r) per key channel
};
static_assert(sizeof(Small) <= 2048, "small state");

template <bool E2>
__device__ __forceinline__ float expo_to_base2(float x) { return E2 ? x : x * 1.4426950408889634f; }
// b^x with one special-function instruction (PTX ex2.approx.ftz: relative error near
// 2^-22, results below 2^-126 flush to zero) -- ample for factors rounded to bf16
template <bool E2>
__device__ __forceinline__ float fexp(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(expo_to_base2<E2>(x)));
  return y;
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of the 8 columns c0 .. c0+7 of `row` in a swizzled 64-row tile
__device__ __forceinline__ uint32_t tile_off(int row, int c0) {
  return (uint32_t)((c0 >> 6) * 8192) + chunk_off(row, (c0 & 63) >> 3);
}
__device__ __forceinline__ void load_g8(const float *sG, int i, int c0, float (&g)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(sG + i * GS + c0);
  const float4 b = *reinterpret_cast<const float4 *>(sG + i * GS + c0 + 4);
  g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w; g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
}

// TMA maps over k, q, v ([token rows][H * 128] bf16, 64 x 64 boxes); q and v only when given
struct PrepMaps {
  TmaMap k, q, v;
};
constexpr uint32_t WAIT_LIMIT = 1u << 22;

template <bool E2>
__global__ void __launch_bounds__(NTH, 2) kda_prep_kernel(KdaPrepArgs a, int64_t items,
                                                          const __grid_constant__ PrepMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float *sG = reinterpret_cast<float *>(sm + OFF_G);
  float *sL = sG;  // once the factors are formed
  float *sX = sG + L_FLOATS;
  float *sT = sX + X_FLOATS;
  Small &sv = *reinterpret_cast<Small *>(sm + OFF_SMALL);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = a.H;
  const void *v = a.v;
  const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
  const float scale = a.scale;
  const bool has_q = a.q != nullptr;
  const int gq = lane >> 2, t4 = lane & 3;

  auto locate = [&](int64_t it, int64_t &r0, int &n) -> bool {
    const int64_t slot = it / H;
    int64_t r1;
    if (a.cu) {
      const int seq = a.chunk_indices[2 * slot], cc = a.chunk_indices[2 * slot + 1];
      if (!(seq >= 0 && seq < a.num_seqs && cc >= 0)) return false;
      r0 = (int64_t)a.cu[seq] + (int64_t)cc * GDN_CHUNK;
      r1 = a.cu[seq + 1];
      if (!(r0 >= 0 && r0 < r1 && r1 <= a.T)) return false;
    } else {
      const int64_t b = slot / NT, c = slot % NT;
      r0 = b * a.T + c * GDN_CHUNK;
      r1 = b * a.T + a.T;
    }
    n = (int)min((int64_t)GDN_CHUNK, r1 - r0);
    return true;
  };

  // the chain kernel launched after this one may be scheduled as SMs free up (it waits for
  // this grid's completion before it reads a blob)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint32_t ldphase = 0;
  if (tid == 0) {
    mbar_init(&sv.ldbar, 1);
    mbar_fence_init();
  }
  if (!v)  // no v: the V tile is zero for every item (u = 0)
    for (int x = tid; x < 1024; x += NTH) *reinterpret_cast<uint4 *>(sm + OFF_V + 16 * x) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    int64_t r0 = 0;
    int n = 0;
    if (!locate(it, r0, n)) {  // uniform: every thread read the same chunk index
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      continue;
    }
    const int h = (int)(it % H);
    uint8_t *blob = a.blob + (size_t)it * BLOB_BYTES;
    auto grow = [&](int i) { return ((r0 + i) * H + h) * (int64_t)GDN_DK; };  // token row, 128 wide

    // ---- every load at once: K, Q, V tiles (two 64 x 64 TMA boxes each; rows past the end
    // hold the tensor's next rows and are zeroed below), the gate column, beta ----
    if (warp == 0) {
      const int y = (int)r0, x0 = h * GDN_DK;
      mbar_expect_tx_w(&sv.ldbar, 16384u * (1u + (has_q ? 1u : 0u) + (v ? 1u : 0u)));
      tma_load_2d_w(sb + OFF_K, &maps.k, x0, y, &sv.ldbar);
      tma_load_2d_w(sb + OFF_K + 8192, &maps.k, x0 + 64, y, &sv.ldbar);
      if (has_q) {
        tma_load_2d_w(sb + OFF_Q, &maps.q, x0, y, &sv.ldbar);
        tma_load_2d_w(sb + OFF_Q + 8192, &maps.q, x0 + 64, y, &sv.ldbar);
      }
      if (v) {  // (no v: the V tile stays zero, u = 0)
        tma_load_2d_w(sb + OFF_V, &maps.v, x0, y, &sv.ldbar);
        tma_load_2d_w(sb + OFF_V + 8192, &maps.v, x0 + 64, y, &sv.ldbar);
      }
    }
    if (tid < 64) sv.beta[tid] = tid < n ? __bfloat162float(beta[(r0 + tid) * H + h]) : 0.f;
    const int d = tid & 127, half = tid >> 7;
    // gate element (row i, this thread's key channel): a scalar gate serves every channel
    const int64_t gstride = a.scalar_gate ? (int64_t)H : (int64_t)H * GDN_DK;
    const int64_t g0 = a.scalar_gate ? r0 * H + h : grow(0) + d;
    auto gidx = [&](int i) { return g0 + i * gstride; };
    float gcol[32];
    if (a.g_cum_in) {
      const float *gp = a.g_cum_in + g0;
#pragma unroll
      for (int j = 0; j < 32; ++j) gcol[j] = gp[min(32 * half + j, n - 1) * gstride];
    } else {
      const float *gp = a.g + g0;
#pragma unroll
      for (int j = 0; j < 32; ++j) gcol[j] = 32 * half + j < n ? gp[(32 * half + j) * gstride] : 0.f;
#pragma unroll
      for (int j = 1; j < 32; ++j) gcol[j] += gcol[j - 1];
      if (half == 0) sv.part[d] = gcol[31];
    }
    __syncthreads();
    if (!a.g_cum_in && half == 1) {
      const float base = sv.part[d];
#pragma unroll
      for (int j = 0; j < 32; ++j) gcol[j] += base;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) sG[(32 * half + j) * GS + d] = gcol[j];
    if (a.g_cumsum && !a.g_cum_in && (!a.scalar_gate || d == 0)) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (32 * half + j < n) a.g_cumsum[gidx(32 * half + j)] = gcol[j];
    }
    if (half == 1) {  // this thread holds rows 32..63 of its channel: G_r and G_last
      const float gr = gcol[0], gl = gcol[31];
      sv.eref[d] = gexp<E2>(gr);
      sv.elr[d] = gexp<E2>(gl - gr);
      reinterpret_cast<float *>(blob + BLOB_EL)[d] = gexp<E2>(gl);
    }
    __syncthreads();
    // range of the factors around the reference row
    bool out_of_range;
    {
      float lo = gcol[0], hi = gcol[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) {
        lo = fminf(lo, gcol[j]);
        hi = fmaxf(hi, gcol[j]);
      }
      const float gr = sG[REF * GS + d];
      out_of_range = fmaxf(expo_to_base2<E2>(hi - gr), expo_to_base2<E2>(gr - lo)) > EXP_LIMIT;
    }
    const bool exact = __syncthreads_or(out_of_range);
    const bool late = !mbar_wait(&sv.ldbar, ldphase, WAIT_LIMIT);
    ldphase ^= 1u;
    if (__syncthreads_or(late)) {  // the tiles did not arrive: report, let the copies land, stop
      if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
      mbar_wait(&sv.ldbar, ldphase ^ 1u, WAIT_LIMIT);
      break;
    }
    if (n < 64) {  // rows past the chunk's end: zero K, Q, V
      for (int x = tid; x < (64 - n) * 16; x += NTH) {
        const int r = n + x / 16, c16 = x % 16;
        const uint32_t o = (c16 >> 3) * 8192 + chunk_off(r, c16 & 7);
        const uint4 z = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(sm + OFF_K + o) = z;
        *reinterpret_cast<uint4 *>(sm + OFF_Q + o) = z;
        *reinterpret_cast<uint4 *>(sm + OFF_V + o) = z;
      }
      __syncthreads();
    }

    if (exact) {  // Gram matrices term by term while K, Q and G are intact: L -> the Kb region
      float *sLx = reinterpret_cast<float *>(sm + OFF_KB);
      for (int p = tid; p < 64 * 64; p += NTH) {
        const int i = p >> 6, j = p & 63;
        if ((j >> 4) > (i >> 4)) continue;  // blocks right of the diagonal are never read
        float sk = 0.f, sq = 0.f;
        if (j <= i && i < n) {
          for (int c0 = 0; c0 < GDN_DK; c0 += 8) {
            float ki[8], kj[8], qi[8], gi[8], gj[8];
            unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_K + tile_off(i, c0)), ki);
            unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_K + tile_off(j, c0)), kj);
            unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_Q + tile_off(i, c0)), qi);
            load_g8(sG, i, c0, gi);
            load_g8(sG, j, c0, gj);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float gam = gexp<E2>(gi[e] - gj[e]);
              sk = fmaf(ki[e] * kj[e], gam, sk);
              sq = fmaf(qi[e] * kj[e], gam, sq);
            }
          }
        }
        sLx[blk(i >> 4, j >> 4) * 256 + bsw(i & 15, j & 15)] = j < i ? sv.beta[i] * sk : 0.f;
        if (has_q)
          *reinterpret_cast<__nv_bfloat16 *>(blob + BLOB_AQ + chunk_off(i, j >> 3) + (j & 7) * 2) =
              __float2bfloat16_rn(j <= i ? scale * sq : 0.f);
      }
      __syncthreads();
    }

    // ---- factors (8 channels of one token row per step) ----
    for (int x = tid; x < 1024; x += NTH) {
      const int i = x >> 4, c0 = (x & 15) * 8;
      const uint32_t to = tile_off(i, c0);
      float kv[8], qv[8], gv[8], o1[8], o4[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_K + to), kv);
      unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_Q + to), qv);
      load_g8(sG, i, c0, gv);
      if (!exact) {
        float gr[8], o2[8], o3[8], er[8], el[8];
        load_g8(sG, REF, c0, gr);
        {
          const float4 *pe = reinterpret_cast<const float4 *>(sv.eref + c0);
          const float4 *pl = reinterpret_cast<const float4 *>(sv.elr + c0);
          const float4 e0 = pe[0], e1 = pe[1], l0 = pl[0], l1 = pl[1];
          er[0] = e0.x; er[1] = e0.y; er[2] = e0.z; er[3] = e0.w; er[4] = e1.x; er[5] = e1.y; er[6] = e1.z; er[7] = e1.w;
          el[0] = l0.x; el[1] = l0.y; el[2] = l0.z; el[3] = l0.w; el[4] = l1.x; el[5] = l1.y; el[6] = l1.z; el[7] = l1.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float ef = fexp<E2>(gv[e] - gr[e]);
          const float rf = fexp<E2>(gr[e] - gv[e]);
          o1[e] = kv[e] * ef;                      // K e      (Gram A; B of w)
          o2[e] = qv[e] * ef;                      // Q e      (Gram A)
          o3[e] = kv[e] * rf;                      // K / e    (Gram B)
          o4[e] = o3[e] * el[e];                   // K b^(Gl - G)
          qv[e] = scale * o2[e] * er[e];           // scale Q b^G
        }
        *reinterpret_cast<uint4 *>(sm + OFF_KB + to) = pack8(o3);
        *reinterpret_cast<uint4 *>(sm + OFF_Q + to) = pack8(o2);
      } else {
        float gl[8];
        load_g8(sG, 63, c0, gl);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float eg = gexp<E2>(gv[e]);
          o1[e] = kv[e] * eg;                      // K b^G (B of w; no column factor)
          o4[e] = kv[e] * gexp<E2>(gl[e] - gv[e]); // K b^(Gl - G)
          qv[e] = scale * qv[e] * eg;              // scale Q b^G
        }
      }
      *reinterpret_cast<uint4 *>(sm + OFF_K + to) = pack8(o1);
      const uint32_t co = chunk_off(i, (c0 & 63) >> 3);
      *reinterpret_cast<uint4 *>(blob + BLOB_KL + (c0 >> 6) * 8192 + co) = pack8(o4);
      if (has_q) *reinterpret_cast<uint4 *>(blob + BLOB_WQ + (c0 >> 6) * 16384 + 8192 + co) = pack8(qv);
    }
    __syncthreads();  // G is dead from here on: its region takes L, X and T

    if (!exact) {
      // ---- L and A_qk: the 10 lower 16x16 blocks of each; warp w takes blocks w, w+8, w+16 ----
      for (int jb = warp; jb < 20; jb += 8) {
        const int which = jb >= 10, bidx = jb - 10 * which;  // 0: L from K e, 1: A_qk from Q e
        const int bi = bidx < 1 ? 0 : bidx < 3 ? 1 : bidx < 6 ? 2 : 3;
        const int bj = bidx - bi * (bi + 1) / 2;
        if (which && !has_q) continue;
        const uint32_t abase = sb + (which ? OFF_Q : OFF_K);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int c8 = (2 * ks + (lane >> 4)) & 7;
          uint32_t af[4], bfr[4];
          ldsm_x4(abase + (ks >> 2) * 8192 + chunk_off(16 * bi + (lane & 15), c8), af);
          ldsm_x4(sb + OFF_KB + (ks >> 2) * 8192 + chunk_off(16 * bj + (lane & 15), c8), bfr);
          mma16816(acc[0], af, bfr[0], bfr[2]);
          mma16816(acc[1], af, bfr[1], bfr[3]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int rr = gq + 8 * hr, c = nt * 8 + 2 * t4;
            const int i = 16 * bi + rr, j = 16 * bj + c;
            if (which == 0) {
              const float bt = sv.beta[i];
              float2 val;
              val.x = j < i ? bt * acc[nt][2 * hr] : 0.f;
              val.y = j + 1 < i ? bt * acc[nt][2 * hr + 1] : 0.f;
              *reinterpret_cast<float2 *>(&sL[blk(bi, bj) * 256 + bsw(rr, c)]) = val;
            } else {  // A_qk staged in G's free tail, copied out below
              *reinterpret_cast<uint32_t *>(sm + OFF_AQS + chunk_off(i, j >> 3) + (j & 7) * 2) =
                  pack_bf16(j <= i ? scale * acc[nt][2 * hr] : 0.f, j + 1 <= i ? scale * acc[nt][2 * hr + 1] : 0.f);
            }
          }
      }
    } else {
      const float *sLx = reinterpret_cast<const float *>(sm + OFF_KB);
      for (int x = tid; x < L_FLOATS; x += NTH) sL[x] = sLx[x];
    }
    if (has_q) {  // A_qk right of each row's diagonal block is zero
      uint8_t *aq = exact ? blob + BLOB_AQ : sm + OFF_AQS;
      for (int x = tid; x < 64 * 8; x += NTH) {
        const int i = x >> 3, c8 = x & 7;
        if (c8 >= 2 * ((i >> 4) + 1)) *reinterpret_cast<uint4 *>(aq + chunk_off(i, c8)) = make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async();  // the staged A_qk, to the bulk copy
    __syncthreads();
    if (warp == 0 && has_q && !exact) bulk_store_w(blob + BLOB_AQ, sb + OFF_AQS, 8192);

    // ---- X = (I + L)^-1 (warps 0..3) ----
    if (warp < 4) solve_blocks(sL, sX, sT, tid);
    __syncthreads();
    // X diag(beta) in bf16 (A of w and u, into the Q tile) and the fp32 X as the A output
    {
      const int i = tid >> 2, cq = (tid & 3) * 16, bi = i >> 4;
      float vals[16];
#pragma unroll
      for (int c4 = 0; c4 < 16; c4 += 4) {
        const int c = cq + c4, cb = c >> 4;
        const float4 x4 = cb <= bi ? *reinterpret_cast<const float4 *>(&sX[blk(bi, cb) * 256 + bsw(i & 15, c & 15)])
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        vals[c4] = x4.x;
        vals[c4 + 1] = x4.y;
        vals[c4 + 2] = x4.z;
        vals[c4 + 3] = x4.w;
      }
      if (a.A && i < n) {
        float4 *Ad = reinterpret_cast<float4 *>(a.A + ((r0 + i) * H + h) * GDN_CHUNK + cq);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          Ad[c4] = make_float4(vals[4 * c4], vals[4 * c4 + 1], vals[4 * c4 + 2], vals[4 * c4 + 3]);
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) vals[c] *= sv.beta[cq + c];
      *reinterpret_cast<uint4 *>(sm + OFF_Q + chunk_off(i, cq >> 3)) = pack8(vals);
      *reinterpret_cast<uint4 *>(sm + OFF_Q + chunk_off(i, (cq >> 3) + 1)) = pack8(vals + 8);
    }
    __syncthreads();

    // ---- w = X diag(beta) (K e) Diag(b^G_r), u = X diag(beta) V: warp -> 16 rows, 64 columns ----
    {
      const int mt = warp & 3, n0 = (warp >> 2) * 64;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t bbase = sb + (which ? OFF_V : OFF_K);
        float acc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t af[4];
          ldsm_x4(sb + OFF_Q + chunk_off(16 * mt + (lane & 15), (2 * ks + (lane >> 4)) & 7), af);
#pragma unroll
          for (int np = 0; np < 4; ++np) {  // pairs of 8-column tiles
            const int nc = n0 + 16 * np;
            uint32_t x[4];
            const int m = lane >> 3, rr = lane & 7;
            ldsm_x4_trans(bbase + (nc >> 6) * 8192 + chunk_off(16 * ks + rr + 8 * (m & 1), ((nc & 63) >> 3) + (m >> 1)), x);
            mma16816(acc[2 * np], af, x[0], x[1]);
            mma16816(acc[2 * np + 1], af, x[2], x[3]);
          }
        }
        // staged as two 64-column blocks of 64 rows: u in G's region (L, X and T are dead), w in
        // K / e's (the Gram's right operand), copied out below
        uint8_t *dst = sm + (which ? OFF_G : OFF_KB);
        const uint32_t kstride = 8192u;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int c = n0 + 8 * nt + 2 * t4;
          const bool unit = which || exact;
          const float f0 = unit ? 1.f : sv.eref[c], f1 = unit ? 1.f : sv.eref[c + 1];
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int i = 16 * mt + gq + 8 * hr;
            *reinterpret_cast<uint32_t *>(dst + (c >> 6) * kstride + chunk_off(i, (c & 63) >> 3) + (c & 7) * 2) =
                pack_bf16(acc[nt][2 * hr] * f0, acc[nt][2 * hr + 1] * f1);
          }
        }
      }
    }
    fence_proxy_async();  // the staged w and u, to the bulk copies
    __syncthreads();
    if (warp == 0) {
      bulk_store_w(blob + BLOB_WQ, sb + OFF_KB, 8192);  // w: rows 0..63 of each 128-row K-block
      bulk_store_w(blob + BLOB_WQ + 16384, sb + OFF_KB + 8192, 8192);
      bulk_store_w(blob + BLOB_U, sb + OFF_G, 16384);
      bulk_store_wait_read_w();
    }
    fence_proxy_async();  // this item's reads of K, Q, V, before the next item's copies
    __syncthreads();  // shared memory is rewritten by the next item
  }
  if (warp == 0) bulk_store_wait_w();  // the blobs have reached global memory
}

}  // namespace

cudaError_t launch_kda_prep(const KdaPrepArgs &a, int slots, cudaStream_t st) {
  if (slots <= 0) return cudaSuccess;
  const int64_t items = (int64_t)slots * a.H;
  auto kern = a.use_exp2 ? kda_prep_kernel<true> : kda_prep_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NTH, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
  const uint64_t rows = a.cu ? (uint64_t)a.T : (uint64_t)(slots / NT) * a.T;  // token rows
  if (rows > (uint64_t)INT32_MAX) return cudaErrorInvalidValue;  // 32-bit TMA rows
  const uint64_t pitch = (uint64_t)a.H * GDN_DK * 2;
  PrepMaps maps{};
  e = make_tmap_bf16(&maps.k, a.k, (uint64_t)a.H * GDN_DK, rows, pitch);
  if (e == cudaSuccess && a.q) e = make_tmap_bf16(&maps.q, a.q, (uint64_t)a.H * GDN_DK, rows, pitch);
  if (e == cudaSuccess && a.v) e = make_tmap_bf16(&maps.v, a.v, (uint64_t)a.H * GDN_DV, rows, (uint64_t)a.H * GDN_DV * 2);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(items, (int64_t)std::max(1, sms * std::max(1, per_sm)));
  kern<<<(unsigned)grid, NTH, SMEM_BYTES, st>>>(a, items, maps);
  return cudaGetLastError();
}

}  // namespace gdn
