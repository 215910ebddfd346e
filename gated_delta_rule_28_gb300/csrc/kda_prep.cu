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
// The gated Gram matrices run on bf16 tensor cores (mma.sync) through a
// factorisation of Gamma by 16-row blocks: for rows i of block bi and the
// reference row r = 16 bi, (K K^T (.) Gamma)_ij = sum_d (k_id b^(G_id - G_rd))
// (k_jd b^(G_rd - G_jd)). For j < r (blocks left of the diagonal) both factors
// are at most 1 for decaying gates, so nothing overflows; inside the diagonal
// block the column factor grows with the decay over at most 15 tokens. A row
// block whose factors would leave the range that fp32 and bf16 represent
// (exponent above 100 in base 2) is computed term by term with one
// exponential per (i, j, d) instead, exactly for any gate range.
//
// The outputs go to one blob per (chunk, head), in the 128-byte-swizzled
// layout the chain kernel's operands take in shared memory (kernels.h, kda::).
// Persistent CTAs of 8 warps, two per SM (about 108 KB of shared memory each).
#include <algorithm>

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
// shared memory map (bytes from a 1024-aligned base)
constexpr int OFF_G = 0;                 // G, fp32 [64][128]
constexpr int OFF_V = OFF_G + 32768;     // V, bf16 K-major swizzled (2 K-blocks of 64 columns)
constexpr int OFF_KA = OFF_V + 16384;    // K b^(G - G_ref) (Gram A), later K b^G (B of w)
constexpr int OFF_QA = OFF_KA + 16384;   // Q b^(G - G_ref) (Gram A), later X diag(beta) in bf16
constexpr int OFF_KB = OFF_QA + 16384;   // K b^(G_ref - G) of the current row block, later X, T
constexpr int OFF_L = OFF_KB + 16384;    // L in 16x16 fp32 blocks (blk / bsw of tile_ops)
constexpr int OFF_SMALL = OFF_L + 10240;
constexpr int SMEM_BYTES = OFF_SMALL + 1024 + 1024;
static_assert(10240 + 4096 <= 16384, "X and T fit in the Kb region");

// largest exponent (base 2) a factor may take on the tensor-core path
constexpr float EXP_LIMIT = 100.f;

struct Small {
  float beta[64];
  float part[128];
  int flags;  // bit bi: row block bi takes the exact path
};

template <bool E2>
__device__ __forceinline__ float expo_to_base2(float x) { return E2 ? x : x * 1.4426950408889634f; }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 8 bf16 of a global row (zeros when the row is not valid)
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, bool valid, float (&x)[8]) {
  if (valid) {
    unpack8(*reinterpret_cast<const uint4 *>(p), x);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
  }
}

template <bool E2>
__global__ void __launch_bounds__(NTH, 2) kda_prep_kernel(KdaPrepArgs a, int64_t items) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float *sG = reinterpret_cast<float *>(sm + OFF_G);
  float *sL = reinterpret_cast<float *>(sm + OFF_L);
  Small &sv = *reinterpret_cast<Small *>(sm + OFF_SMALL);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = a.H;
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
  const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
  const float scale = a.scale;

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
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    int64_t r0 = 0;
    int n = 0;
    const bool ok = locate(it, r0, n);
    if (!ok) {  // uniform: every thread read the same chunk index
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      continue;
    }
    const int h = (int)(it % H);
    uint8_t *blob = a.blob + (size_t)it * BLOB_BYTES;
    auto grow = [&](int i) { return ((r0 + i) * H + h) * (int64_t)GDN_DK; };  // row start, 128 wide

    // ---- loads: V by cp.async (zero past the end), the gate column of this thread, beta ----
    for (int x = tid; x < 1024; x += NTH) {
      const int r = x >> 4, c16 = x & 15;
      const bool valid = r < n;
      const __nv_bfloat16 *src = v + ((r0 + (valid ? r : 0)) * H + h) * GDN_DV + c16 * 8;
      cp_async16(sb + OFF_V + (c16 >> 3) * 8192 + chunk_off(r, c16 & 7), src, valid ? 16u : 0u);
    }
    cp_async_commit();
    if (tid < 64) sv.beta[tid] = tid < n ? __bfloat162float(beta[(r0 + tid) * H + h]) : 0.f;
    if (tid == 0) sv.flags = 0;
    const int d = tid & 127, half = tid >> 7;
    float gcol[32];
    // gate element of row i for this thread's key channel (a scalar gate serves every channel)
    auto gidx = [&](int i) { return a.scalar_gate ? (r0 + i) * H + h : grow(i) + d; };
    if (a.g_cum_in) {
#pragma unroll
      for (int j = 0; j < 32; ++j) gcol[j] = a.g_cum_in[gidx(min(32 * half + j, n - 1))];
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) gcol[j] = 32 * half + j < n ? a.g[gidx(32 * half + j)] : 0.f;
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
    for (int j = 0; j < 32; ++j) sG[(32 * half + j) * GDN_DK + d] = gcol[j];
    if (a.g_cumsum && !a.g_cum_in && (!a.scalar_gate || d == 0)) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (32 * half + j < n) a.g_cumsum[gidx(32 * half + j)] = gcol[j];
    }
    __syncthreads();
    if (tid < GDN_DK) reinterpret_cast<float *>(blob + BLOB_EL)[tid] = gexp<E2>(sG[63 * GDN_DK + tid]);

    // ---- pass A (8 keys of one row per step): Q b^G, K b^(Gl - G) to the blob; the Gram
    // A operands K b^(G - G_ref), Q b^(G - G_ref) with G_ref the row block's first row ----
    {
      int over = 0;
      for (int x = tid; x < 1024; x += NTH) {
        const int i = x >> 4, c0 = (x & 15) * 8;
        float kv[8], qv[8], gv[8], gl[8], gr[8];
        load8(k + grow(i) + c0, i < n, kv);
        load8(q ? q + grow(i) + c0 : nullptr, i < n && q, qv);
        const int r = i & ~15;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          gv[e] = sG[i * GDN_DK + c0 + e];
          gl[e] = sG[63 * GDN_DK + c0 + e];
          gr[e] = sG[r * GDN_DK + c0 + e];
        }
        float o1[8], o2[8], o3[8], o4[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float eg = gexp<E2>(gv[e]);
          o1[e] = scale * qv[e] * eg;                 // Q b^G (scaled)
          o2[e] = kv[e] * gexp<E2>(gl[e] - gv[e]);    // K b^(Gl - G)
          const float xr = gv[e] - gr[e];
          over |= fabsf(expo_to_base2<E2>(xr)) > EXP_LIMIT;
          const float er = gexp<E2>(xr);
          o3[e] = kv[e] * er;                         // K b^(G - G_ref)
          o4[e] = qv[e] * er;                         // Q b^(G - G_ref)
        }
        const uint32_t co = chunk_off(i, (c0 & 63) >> 3);
        if (!a.no_q) *reinterpret_cast<uint4 *>(blob + BLOB_WQ + (c0 >> 6) * 16384 + 8192 + co) = pack8(o1);
        *reinterpret_cast<uint4 *>(blob + BLOB_KL + (c0 >> 6) * 8192 + co) = pack8(o2);
        *reinterpret_cast<uint4 *>(sm + OFF_KA + (c0 >> 6) * 8192 + co) = pack8(o3);
        *reinterpret_cast<uint4 *>(sm + OFF_QA + (c0 >> 6) * 8192 + co) = pack8(o4);
        if (over) atomicOr(&sv.flags, 1 << (i >> 4));
        over = 0;
      }
    }

    // ---- gated Gram matrices, one row block at a time ----
    for (int bi = 0; bi < 4; ++bi) {
      const int r = 16 * bi, ncol = 16 * bi + 16;
      // column operand K b^(G_ref - G) for rows j < ncol
      for (int x = tid; x < ncol * 16; x += NTH) {
        const int j = x >> 4, c0 = (x & 15) * 8;
        float kv[8], o[8];
        load8(k + grow(j) + c0, j < n, kv);
        int over = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float xr = sG[r * GDN_DK + c0 + e] - sG[j * GDN_DK + c0 + e];
          over |= fabsf(expo_to_base2<E2>(xr)) > EXP_LIMIT;
          o[e] = kv[e] * gexp<E2>(xr);
        }
        *reinterpret_cast<uint4 *>(sm + OFF_KB + (c0 >> 6) * 8192 + chunk_off(j, (c0 & 63) >> 3)) = pack8(o);
        if (over) atomicOr(&sv.flags, 1 << bi);
      }
      __syncthreads();
      const bool exact = (sv.flags >> bi) & 1;
      if (!exact) {
        // warp 2 bj + which: block (bi, bj) of L (which 0) or of A_qk (which 1)
        const int which = warp & 1, bj = warp >> 1;
        if (bj <= bi && !(which == 1 && a.no_q)) {
          const uint32_t abase = sb + (which ? OFF_QA : OFF_KA);
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int c8 = (2 * ks + (lane >> 4)) & 7;
            uint32_t af[4], bfr[4];
            ldsm_x4(abase + (ks >> 2) * 8192 + chunk_off(r + (lane & 15), c8), af);
            ldsm_x4(sb + OFF_KB + (ks >> 2) * 8192 + chunk_off(16 * bj + (lane & 15), c8), bfr);
            mma16816(acc[0], af, bfr[0], bfr[2]);
            mma16816(acc[1], af, bfr[1], bfr[3]);
          }
          const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int rr = gq + 8 * hr, c = nt * 8 + 2 * t4;
              const int i = r + rr, j = 16 * bj + c;
              float2 val;
              if (which == 0) {
                const float bt = sv.beta[i];
                val.x = j < i ? bt * acc[nt][2 * hr] : 0.f;
                val.y = j + 1 < i ? bt * acc[nt][2 * hr + 1] : 0.f;
                *reinterpret_cast<float2 *>(&sL[blk(bi, bj) * 256 + bsw(rr, c)]) = val;
              } else {
                val.x = j <= i ? scale * acc[nt][2 * hr] : 0.f;
                val.y = j + 1 <= i ? scale * acc[nt][2 * hr + 1] : 0.f;
                *reinterpret_cast<uint32_t *>(blob + BLOB_AQ + chunk_off(i, j >> 3) + (j & 7) * 2) =
                    pack_bf16(val.x, val.y);
              }
            }
        }
      } else {
        // exact: one exponential per (i, j, d), rows of block bi against columns j <= i
        for (int p = tid; p < 16 * ncol; p += NTH) {
          const int i = r + p / ncol, j = p % ncol;
          float sk = 0.f, sq = 0.f;
          if (j <= i && i < n) {
            for (int c0 = 0; c0 < GDN_DK; c0 += 8) {
              float ki[8], kj[8], qi[8];
              load8(k + grow(i) + c0, true, ki);
              load8(k + grow(j) + c0, true, kj);
              load8(q ? q + grow(i) + c0 : nullptr, q != nullptr, qi);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float gam = gexp<E2>(sG[i * GDN_DK + c0 + e] - sG[j * GDN_DK + c0 + e]);
                sk = fmaf(ki[e] * kj[e], gam, sk);
                sq = fmaf(qi[e] * kj[e], gam, sq);
              }
            }
          }
          const int bj = j >> 4;
          sL[blk(bi, bj) * 256 + bsw(i - r, j & 15)] = j < i ? sv.beta[i] * sk : 0.f;
          if (!a.no_q) {
            const float val = j <= i ? scale * sq : 0.f;
            *reinterpret_cast<__nv_bfloat16 *>(blob + BLOB_AQ + chunk_off(i, j >> 3) + (j & 7) * 2) =
                __float2bfloat16_rn(val);
          }
        }
      }
      // A_qk right of the diagonal block is zero
      if (!a.no_q)
        for (int x = tid; x < 16 * (64 - ncol) / 8; x += NTH) {
          const int per = (64 - ncol) / 8, i = r + x / per, c8 = ncol / 8 + x % per;
          *reinterpret_cast<uint4 *>(blob + BLOB_AQ + chunk_off(i, c8)) = make_uint4(0, 0, 0, 0);
        }
      __syncthreads();  // the next row block rewrites the column operand
    }

    // ---- X = (I + L)^-1 (warps 0..3), meanwhile K b^G as the B operand of w (warps 4..7) ----
    float *sX = reinterpret_cast<float *>(sm + OFF_KB);
    float *sT = sX + 10 * 256;
    if (warp < 4) {
      solve_blocks(sL, sX, sT, tid);
    } else {
      for (int x = tid - 128; x < 1024; x += 128) {
        const int i = x >> 4, c0 = (x & 15) * 8;
        float kv[8], o[8];
        load8(k + grow(i) + c0, i < n, kv);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = kv[e] * gexp<E2>(sG[i * GDN_DK + c0 + e]);
        *reinterpret_cast<uint4 *>(sm + OFF_KA + (c0 >> 6) * 8192 + chunk_off(i, (c0 & 63) >> 3)) = pack8(o);
      }
    }
    __syncthreads();
    // X diag(beta) in bf16 (A of w and u); the fp32 X as the A output
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
      *reinterpret_cast<uint4 *>(sm + OFF_QA + chunk_off(i, cq >> 3)) = pack8(vals);
      *reinterpret_cast<uint4 *>(sm + OFF_QA + chunk_off(i, (cq >> 3) + 1)) = pack8(vals + 8);
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- w = X diag(beta) (K b^G), u = X diag(beta) V: warp -> 16 rows, 64 columns ----
    {
      const int mt = warp & 3, n0 = (warp >> 2) * 64;
      const int gq = lane >> 2, t4 = lane & 3;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t bbase = sb + (which ? OFF_V : OFF_KA);
        float acc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t af[4];
          ldsm_x4(sb + OFF_QA + chunk_off(16 * mt + (lane & 15), (2 * ks + (lane >> 4)) & 7), af);
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
        uint8_t *dst = blob + (which ? BLOB_U : BLOB_WQ);
        const uint32_t kstride = which ? 8192u : 16384u;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int i = 16 * mt + gq + 8 * hr, c = n0 + 8 * nt + 2 * t4;
            *reinterpret_cast<uint32_t *>(dst + (c >> 6) * kstride + chunk_off(i, (c & 63) >> 3) + (c & 7) * 2) =
                pack_bf16(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
          }
      }
    }
    __syncthreads();  // shared memory is rewritten by the next item
  }
  cp_async_wait<0>();
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
  const int64_t grid = std::min<int64_t>(items, (int64_t)std::max(1, sms * std::max(1, per_sm)));
  kern<<<(unsigned)grid, NTH, SMEM_BYTES, st>>>(a, items);
  return cudaGetLastError();
}

}  // namespace gdn
