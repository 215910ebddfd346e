// UT transform of every 64-token chunk, for all chunks and heads at once
// (bf16 keys, scalar gate, sm_103a).
//
// Per chunk (the UT/WY transform; GDN Ascend C adapter forward, steps
// chunk_local_cumsum / chunk_scaled_dot_kkt / solve_tril):
//   G = cumsum(g) inside the chunk
//   L = strictly-lower(diag(beta) (K K^T (.) Gamma)),  Gamma_ij = base^(G_i - G_j)
//   X = (I + L)^-1
// X has no dependence on the state, so it is computed here for every chunk
// in parallel (persistent CTAs of 4 warps walking the (chunk, head) items; K K^T
// on bf16 mma.sync, the solve in fp32 shared memory) and written in bf16 for the tensor-core
// state kernel, scaled by its columns as the pair [X diag(beta); X diag(beta base^G)], so
// that the state kernel only multiplies by it; with a table of the chunk's per-token gate
// factors (GateTabRow: G, base^G, base^(G_last - G), beta base^G,
// beta, and the two factors of the gate between 16-token blocks).
// The fp32 X (the A output of the forward) and the cumulative gate are
// written here when asked for.
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

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Persistent: each CTA walks the (chunk, head) items with a stride of the grid (eight CTAs per
// SM: one key buffer each, 27 KB of shared memory), prefetching the next item's gate and beta
// into registers.
// TMA map over the X pairs: [slots * H * 128 rows][64] bf16, 64 x 64 boxes
struct UtMaps {
  TmaMap x;
};

template <bool E2>
__global__ void __launch_bounds__(128, 8) ut_kernel(UtArgs a, int64_t items, const __grid_constant__ UtMaps maps) {
  __shared__ __align__(1024) uint8_t kbuf[1][16384];  // keys (64 rows x 2 K-blocks, swizzled);
                                                      // after K K^T it holds L's blocks
  __shared__ __align__(16) float XB[10 * 256];
  // the solve's scratch: the last 6 KB of the key buffer, which L (10 blocks, 10 KB) leaves free
  float *TB = reinterpret_cast<float *>(kbuf[0] + 10 * 256 * 4);
  __shared__ __align__(16) float sg[64];
  __shared__ __align__(16) float sG[64];
  __shared__ __align__(16) float sbeta[64];
  __shared__ __align__(16) float sBEG[64];              // beta base^G (column factor of X diag(b e^G))
  // the block-factorised gate (rows F_EA, F_EB1..) while L is formed, in the solve's scratch
  float *sEA = TB;
  float(*sEB)[64] = reinterpret_cast<float(*)[64]>(TB + 64);

  // the state kernel launched after this one may be scheduled as SMs free up (it waits for
  // this grid's completion before it reads anything written here)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = a.H;
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
  const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
  const float *gsrc = a.g_cum_in ? a.g_cum_in : a.g;
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;

  // Item it = slot * H + h covers rows [r0, r0 + n) of head h. Each item is located once,
  // one iteration ahead, in 32-bit arithmetic (the launch checks that items < 2^31).
  struct Loc {
    int64_t r0, slot;
    int n, h;
    bool live, ok;  // live: it < items; ok: a valid chunk (a corrupt packed index is not)
  };
  auto locate = [&](int64_t it) -> Loc {
    Loc L{0, 0, 0, 0, it < items, false};
    if (!L.live) return L;
    const uint32_t u = (uint32_t)it, slot = u / (uint32_t)H;
    L.slot = slot;
    L.h = (int)(u - slot * (uint32_t)H);
    int64_t r1;
    if (a.cu) {
      const int seq = a.chunk_indices[2 * slot], cc = a.chunk_indices[2 * slot + 1];
      if (!(seq >= 0 && seq < a.num_seqs && cc >= 0)) return L;
      L.r0 = (int64_t)a.cu[seq] + (int64_t)cc * GDN_CHUNK;
      r1 = a.cu[seq + 1];
      if (!(L.r0 >= 0 && L.r0 < r1 && r1 <= a.T)) return L;
    } else {
      const uint32_t b = slot / (uint32_t)NT, c = slot - b * (uint32_t)NT;
      L.r0 = (int64_t)b * a.T + (int64_t)c * GDN_CHUNK;
      r1 = (int64_t)b * a.T + a.T;
    }
    L.n = (int)min((int64_t)GDN_CHUNK, r1 - L.r0);
    L.ok = true;
    return L;
  };
  auto load_keys = [&](const Loc &L, int buf) {  // zero past the chunk end
    if (L.live && L.ok) {
      const uint32_t kt = smem_u32(kbuf[buf]);
#pragma unroll
      for (int x = tid; x < 1024; x += 128) {
        const int r = x >> 4, f16 = x & 15;
        const bool valid = r < L.n;
        const __nv_bfloat16 *src = k + ((L.r0 + (valid ? r : 0)) * H + L.h) * GDN_DK + f16 * 8;
        cp_async16(kt + (f16 >> 3) * 8192 + chunk_off(r, f16 & 7), src, valid ? 16u : 0u);
      }
    }
    cp_async_commit();
  };

  // gate and beta of an item into registers, one item ahead (rows past the end: no gate
  // increment, beta 0)
  auto load_gb = [&](const Loc &L, float &gv, float &bv) {
    gv = 0.f;
    bv = 0.f;
    if (tid < 64 && L.live && L.ok && tid < L.n) {
      gv = gsrc[(L.r0 + tid) * H + L.h];
      bv = __bfloat162float(beta[(L.r0 + tid) * H + L.h]);
    }
  };
  const int buf = 0;
  float ng, nb;
  Loc cur = locate(blockIdx.x);
  load_gb(cur, ng, nb);
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    load_keys(cur, buf);
    const Loc nxt = locate(it + gridDim.x);  // while the keys arrive
    const bool ok = cur.ok;
    const int64_t r0 = cur.r0, slot = cur.slot;
    const int n = cur.n, h = cur.h;
    if (tid < 64) {
      sg[tid] = ng;
      sbeta[tid] = nb;
    }
    cp_async_wait<0>();
    __syncthreads();
    load_gb(nxt, ng, nb);
    cur = nxt;
    if (!ok) {
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      continue;  // uniform: every thread saw the same chunk index
    }
    if (a.g_cum_in) {
      if (tid < 64) sG[tid] = sg[min(tid, n - 1)];
    } else if (warp == 0) {
      const float x0 = sg[2 * lane], x1 = sg[2 * lane + 1], pair = x0 + x1;
      float incl = pair;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const float ex = incl - pair;
      sG[2 * lane] = ex + x0;
      sG[2 * lane + 1] = ex + pair;
    }

    // K K^T blocks (bi, bj), bj <= bi, in blk() order; warp w takes blocks w, w+4, w+8
    const uint32_t kt = smem_u32(kbuf[buf]);
    float acc[3][2][4];
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      const int bidx = warp + 4 * u;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[u][nt][e] = 0.f;
      if (bidx >= 10) continue;
      const int bi = bidx < 1 ? 0 : bidx < 3 ? 1 : bidx < 6 ? 2 : 3;
      const int bj = bidx - bi * (bi + 1) / 2;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // 16 features per step
        const int c8 = (2 * ks + (lane >> 4)) & 7;
        const uint32_t kb = kt + (ks >> 2) * 8192;
        uint32_t af[4], bf[4];
        ldsm_x4(kb + chunk_off(16 * bi + (lane & 15), c8), af);
        ldsm_x4(kb + chunk_off(16 * bj + (lane & 15), c8), bf);
        mma_bf16_16816(acc[u][0], af, bf[0], bf[2]);
        mma_bf16_16816(acc[u][1], af, bf[1], bf[3]);
      }
    }
    __syncthreads();  // the keys are consumed (their buffer now takes L); sG is complete
    // base^(G_t - G_{16 b(t)}) and base^(G_{16 b} - G_s) for s < 16 b: for t > s in
    // different blocks the gate is their product (each factor at most 1 for decaying gates)
    if (tid < 64) sEA[tid] = gexp<E2>(sG[tid] - sG[tid & ~15]);
    for (int e = tid; e < 192; e += 128) {
      const int bb = 1 + (e >> 6), s2 = e & 63;
      sEB[bb - 1][s2] = s2 < 16 * bb ? gexp<E2>(sG[16 * bb] - sG[s2]) : 0.f;
    }
    if (tid < 64) sBEG[tid] = sbeta[tid] * gexp<E2>(sG[tid]);
    __syncthreads();
    float *LB = reinterpret_cast<float *>(kbuf[buf]);
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      const int bidx = warp + 4 * u;
      if (bidx >= 10) continue;
      const int bi = bidx < 1 ? 0 : bidx < 3 ? 1 : bidx < 6 ? 2 : 3;
      const int bj = bidx - bi * (bi + 1) / 2;
      const int g = lane >> 2, t = lane & 3;
      float *Lb = LB + blk(bi, bj) * 256;
      // this thread's rows g, g+8 and columns nt*8 + 2t + {0, 1}
      const float bi_[2] = {sbeta[16 * bi + g], sbeta[16 * bi + g + 8]};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int r = g + 8 * hr, c = nt * 8 + 2 * t;
          const int i = 16 * bi + r, j = 16 * bj + c;
          float2 val;
          if (bi > bj) {  // off-diagonal block: factorised gate, no exponential
            const float fa = bi_[hr] * sEA[i];
            const float2 eb = *reinterpret_cast<const float2 *>(&sEB[bi - 1][j]);
            val.x = fa * acc[u][nt][2 * hr] * eb.x;
            val.y = fa * acc[u][nt][2 * hr + 1] * eb.y;
          } else {  // diagonal block: strictly lower part
            val.x = i > j ? bi_[hr] * acc[u][nt][2 * hr] * gexp<E2>(sG[i] - sG[j]) : 0.f;
            val.y = i > j + 1 ? bi_[hr] * acc[u][nt][2 * hr + 1] * gexp<E2>(sG[i] - sG[j + 1]) : 0.f;
          }
          *reinterpret_cast<float2 *>(&Lb[bsw(r, c)]) = val;  // c even: c, c+1 adjacent after the swizzle
        }
      }
    }
    __syncthreads();
    solve_blocks(LB, XB, TB, tid);

    // X rows: thread -> row tid/2, columns 32 (tid&1) .. +32
    {
      const int row = tid >> 1, half = tid & 1, bi = row >> 4;
      float vals[32];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int cb = 2 * half + q;
#pragma unroll
        for (int c4 = 0; c4 < 16; c4 += 4) {  // aligned groups of 4 stay contiguous under bsw
          const float4 x = cb <= bi ? *reinterpret_cast<const float4 *>(&XB[blk(bi, cb) * 256 + bsw(row & 15, c4)])
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
          vals[16 * q + c4] = x.x;
          vals[16 * q + c4 + 1] = x.y;
          vals[16 * q + c4 + 2] = x.z;
          vals[16 * q + c4 + 3] = x.w;
        }
      }
      if (a.A && row < n) {
        float4 *Ad = reinterpret_cast<float4 *>(a.A + ((r0 + row) * H + h) * GDN_CHUNK + 32 * half);
#pragma unroll
        for (int q = 0; q < 8; ++q) Ad[q] = make_float4(vals[4 * q], vals[4 * q + 1], vals[4 * q + 2], vals[4 * q + 3]);
      }
      // the pair [X diag(beta); X diag(beta base^G)] in bf16, 128 rows per chunk and head, staged
      // in the key buffer (free after the solve) as two 64-row boxes in the 128-byte-swizzled
      // layout, then written by two TMA stores
      uint8_t *stage = kbuf[buf];
      float sc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) sc[j] = vals[j] * sbeta[32 * half + j];
#pragma unroll
      for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4 *>(stage + chunk_off(row, 4 * half + q)) = pack8(sc + 8 * q);
#pragma unroll
      for (int j = 0; j < 32; ++j) sc[j] = vals[j] * sBEG[32 * half + j];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(stage + 8192 + chunk_off(row, 4 * half + q)) = pack8(sc + 8 * q);
    }
    fence_proxy_async();  // the staged pair, to the TMA unit
    __syncthreads();
    if (warp == 0) {
      const int y = (int)((slot * H + h) * 2 * GDN_CHUNK);
      tma_store_2d_w(&maps.x, 0, y, smem_u32(kbuf[buf]));
      tma_store_2d_w(&maps.x, 0, y + GDN_CHUNK, smem_u32(kbuf[buf]) + 8192);
    }
    if (a.g_cumsum && !a.g_cum_in && tid < n) a.g_cumsum[(r0 + tid) * H + h] = sG[tid];
    if (tid < 64) {  // per-token gate factors for the state kernels (rows of GateTabRow)
      float *tab = a.ftab + (slot * H + h) * F_TAB;
      const float G = sG[tid], eg = gexp<E2>(G), bt = sbeta[tid];
      tab[F_G * 64 + tid] = G;
      tab[F_EG * 64 + tid] = eg;
      tab[F_EGL * 64 + tid] = gexp<E2>(sG[63] - G);
      tab[F_BEG * 64 + tid] = bt * eg;
      tab[F_BETA * 64 + tid] = bt;
      tab[F_EA * 64 + tid] = gexp<E2>(G - sG[tid & ~15]);  // recomputed: the solve reused their space
#pragma unroll
      for (int bb = 1; bb <= 3; ++bb) tab[(F_EB1 + bb - 1) * 64 + tid] = tid < 16 * bb ? gexp<E2>(sG[16 * bb] - G) : 0.f;
    }
    if (warp == 0) bulk_store_wait_read_w();  // the key buffer takes the next item's keys
    __syncthreads();  // sG, sbeta and the X blocks are rewritten by the next item
  }
  cp_async_wait<0>();
  if (warp == 0) bulk_store_wait_w();  // the X pairs have reached global memory
}

// The backward's X pair and gate tables from the forward's A slot (X, fp32) instead of a
// second UT transform: the same values the UT kernel forms, bit for bit (X rows past the
// chunk's end are identity rows there, so those pair rows are zero). One CTA per item.
template <bool E2>
__global__ void __launch_bounds__(256) ut_pair_kernel(UtArgs a, const float *__restrict__ A) {
  __shared__ __align__(16) float sG[64], sbeta[64], sBEG[64], sEA[64], sEB[3][64];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, H = a.H;
  const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
  const uint32_t u = blockIdx.x, slot = u / (uint32_t)H;
  const int h = (int)(u - slot * (uint32_t)H);
  int64_t r0, r1;
  if (a.cu) {
    const int seq = a.chunk_indices[2 * slot], cc = a.chunk_indices[2 * slot + 1];
    const bool ok = seq >= 0 && seq < a.num_seqs && cc >= 0 && (r0 = (int64_t)a.cu[seq] + (int64_t)cc * GDN_CHUNK,
                                                                r1 = a.cu[seq + 1], r0 >= 0 && r0 < r1 && r1 <= a.T);
    if (!ok) {
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      return;
    }
  } else {
    const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
    const uint32_t b = slot / (uint32_t)NT, c = slot - b * (uint32_t)NT;
    r0 = (int64_t)b * a.T + (int64_t)c * GDN_CHUNK;
    r1 = (int64_t)b * a.T + a.T;
  }
  const int n = (int)min((int64_t)GDN_CHUNK, r1 - r0);
  // this thread's X values (rows r and r + 32, columns 8 c .. 8 c + 7), issued before the gate
  // and beta loads so that the two wait together
  const int r = tid >> 3, c = tid & 7;
  float4 xv[2][2];
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2) {
    const int rr = r + 32 * k2;
    const float4 *src = reinterpret_cast<const float4 *>(A + ((r0 + min(rr, n - 1)) * H + h) * GDN_CHUNK + 8 * c);
    xv[k2][0] = rr < n ? __ldg(src) : make_float4(0.f, 0.f, 0.f, 0.f);
    xv[k2][1] = rr < n ? __ldg(src + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (tid < 64) {
    sG[tid] = a.g_cum_in[(r0 + min(tid, n - 1)) * H + h];
    sbeta[tid] = tid < n ? __bfloat162float(beta[(r0 + tid) * H + h]) : 0.f;
  }
  __syncthreads();
  if (tid < 64) {
    sEA[tid] = gexp<E2>(sG[tid] - sG[tid & ~15]);
    sBEG[tid] = sbeta[tid] * gexp<E2>(sG[tid]);
  }
  if (tid < 192) {
    const int bb = 1 + (tid >> 6), s2 = tid & 63;
    sEB[bb - 1][s2] = s2 < 16 * bb ? gexp<E2>(sG[16 * bb] - sG[s2]) : 0.f;
  }
  __syncthreads();
  // pair rows r and r + 32 (and 64 + those), columns 8 c .. 8 c + 7: 128-byte rows per 8 lanes
  __nv_bfloat16 *xw = a.xw + (int64_t)u * 2 * GDN_CHUNK * GDN_CHUNK;
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2) {
    const int rr = r + 32 * k2;
    const float x[8] = {xv[k2][0].x, xv[k2][0].y, xv[k2][0].z, xv[k2][0].w,
                        xv[k2][1].x, xv[k2][1].y, xv[k2][1].z, xv[k2][1].w};
    float s0[8], s1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      s0[e] = x[e] * sbeta[8 * c + e];
      s1[e] = x[e] * sBEG[8 * c + e];
    }
    *reinterpret_cast<uint4 *>(xw + rr * GDN_CHUNK + 8 * c) = pack8(s0);
    *reinterpret_cast<uint4 *>(xw + (GDN_CHUNK + rr) * GDN_CHUNK + 8 * c) = pack8(s1);
  }
  if (tid < 64) {  // the gate table, as the UT kernel writes it
    float *tab = a.ftab + (int64_t)u * F_TAB;
    const float G = sG[tid], eg = gexp<E2>(G), bt = sbeta[tid];
    tab[F_G * 64 + tid] = G;
    tab[F_EG * 64 + tid] = eg;
    tab[F_EGL * 64 + tid] = gexp<E2>(sG[63] - G);
    tab[F_BEG * 64 + tid] = bt * eg;
    tab[F_BETA * 64 + tid] = bt;
    tab[F_EA * 64 + tid] = sEA[tid];
    tab[F_EB1 * 64 + tid] = sEB[0][tid];
    tab[F_EB2 * 64 + tid] = sEB[1][tid];
    tab[F_EB3 * 64 + tid] = sEB[2][tid];
  }
}

}  // namespace

cudaError_t launch_ut_pair(const UtArgs &a, const float *A, int slots, cudaStream_t st) {
  if (slots <= 0) return cudaSuccess;
  const int64_t items = (int64_t)slots * a.H;
  if (items > INT32_MAX || !a.g_cum_in) return cudaErrorInvalidValue;
  auto kern = a.use_exp2 ? ut_pair_kernel<true> : ut_pair_kernel<false>;
  kern<<<(unsigned)items, 256, 0, st>>>(a, A);
  return cudaGetLastError();
}

cudaError_t launch_ut(const UtArgs &a, int slots, cudaStream_t st) {
  if (slots <= 0) return cudaSuccess;
  const int64_t items = (int64_t)slots * a.H;
  auto kern = a.use_exp2 ? ut_kernel<true> : ut_kernel<false>;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, 0);
  if (e != cudaSuccess) return e;
  // the kernel locates items in 32 bits, and the X pairs' TMA rows are 32-bit coordinates
  if (items > INT32_MAX / (2 * GDN_CHUNK)) return cudaErrorInvalidValue;
  UtMaps maps;
  e = make_tmap_bf16(&maps.x, a.xw, GDN_CHUNK, (uint64_t)items * 2 * GDN_CHUNK, GDN_CHUNK * 2);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(items, (int64_t)std::max(1, sms * std::max(1, per_sm)));
  kern<<<(unsigned)grid, 128, 0, st>>>(a, items, maps);
  return cudaGetLastError();
}

}  // namespace gdn
