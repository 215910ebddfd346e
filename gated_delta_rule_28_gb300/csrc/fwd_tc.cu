// Tensor-core (tcgen05) chunk forward for bf16 inputs, scalar gate (sm_103a).
//
// One CTA owns one independent run (batch row, packed document or segment)
// of one head and 64 of the 128 state columns; the state slice h (128 x 64,
// fp32) lives in registers (thread = key row, 32 columns), its bf16 copy in
// shared memory is the operand of the state contraction. Per 64-token chunk
// the CTA takes the chunk algorithm's steps (north star; GDN Ascend C adapter
// forward; chunk_fwd_h / chunk_kda_fwd_finalize of the KDA adapter), with
// every dense contraction on the tensor core (bf16 operands from shared
// memory, fp32 accumulators in tensor memory) and M = 128 throughout:
//
//   P1   S = [K; Q] K^T                          -> L = strictly-lower(beta S (.) Gamma),
//                                                   A_qk = lower-incl(S_qk (.) Gamma)
//   SIMT X = (I + L)^-1 (fp32, 16x16 blocks: diagonal blocks by forward
//        substitution, then the off-diagonal block levels)
//   P3a  [X; A_qk] X            -> A_qk X
//   P3b  [X; A_qk X] [beta Kg | beta V]  -> [w | u ; A_qk w | A_qk u]   (Kg = K (.) e^G)
//   P4   [-w; Qg - A_qk w] h   accumulated onto [u; A_qk u]  -> [v_new ; o / scale]
//        (o = scale (Qg h + A_qk v_new) = scale ((Qg - A_qk w) h + A_qk u))
//   P5   (K (.) e^(G_last - G))^T v_new          -> h <- e^(G_last) h + P5
//
// Loads of chunk c+1 (cp.async, zero-filled past the run end) overlap the
// work on chunk c. All mbarrier waits are bounded; a wait that runs out sets
// the device flag and the CTA leaves after releasing its tensor memory.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace gdn {
namespace {
using namespace tc;

constexpr int TBV = 64;    // state columns per CTA
constexpr int TNT = 256;   // threads per CTA
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t T_S = 0;   // 64 columns: S, then A_qk X, then P5
constexpr uint32_t T_W = 64;  // 192 columns: P3b; P4 accumulates into [T_W+128, T_W+192)

// shared memory map (bytes from a 1024-aligned base)
constexpr int SZ_KQ = 2 * 128 * 128;  // two K-blocks of 128 rows ([K; Q]) x 128 B
constexpr int SZ_V = 64 * TBV * 2;    // value slice, plain [token][column]
constexpr int OFF_KQ = 0;             // 2 stages
constexpr int OFF_V = OFF_KQ + 2 * SZ_KQ;
constexpr int OFF_AOP = OFF_V + 2 * SZ_V;     // [X; A_qk | A_qk X]  128 x 64
constexpr int OFF_AT = OFF_AOP + 16384;       // X^T                  64 x 64
constexpr int OFF_B3 = OFF_AT + 8192;         // [beta Kg | beta V]^T 192 x 64
constexpr int OFF_WQ = OFF_B3 + 24576;        // [-w; Qg - A_qk w]    2 x 128 x 64
constexpr int OFF_KL = OFF_WQ + 32768;        // kgl^T                128 x 64
constexpr int OFF_HT = OFF_KL + 16384;        // h^T                  2 x 64 x 64
constexpr int OFF_VN = OFF_HT + 16384;        // v_new^T              64 x 64
constexpr int OFF_SMALL = OFF_VN + 8192;
constexpr int SMEM_BYTES = OFF_SMALL + 2048 + 1024;
// fp32 solve buffers alias [OFF_WQ, OFF_WQ + 49152) (free while solving)
constexpr int LS = 65;
constexpr int OFF_L = OFF_WQ;
constexpr int OFF_X = OFF_L + 64 * LS * 4;
constexpr int OFF_T = OFF_X + 64 * LS * 4;
static_assert(OFF_T + 3 * 256 * 4 <= OFF_WQ + 49152, "solve buffers overflow");
static_assert(SMEM_BYTES <= 232448, "shared memory");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// base-e or base-2 decay factor of a (difference of) cumulative log-gate(s)
__device__ __forceinline__ float gexp(float x, bool e2) { return e2 ? exp2f(x) : __expf(x); }

__device__ __forceinline__ void st_bf16(uint8_t *base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
}
__device__ __forceinline__ float ld_bf16(const uint8_t *base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}

// X = (I + L)^-1 for a 64x64 strictly-lower L (stride LS), 256 threads.
__device__ void solve64(const float *L, float *X, float *T, int tid) {
  if (tid < 64) {  // diagonal 16x16 blocks, one column per thread
    const int b = tid >> 4, c = tid & 15, base = b * 16;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < 16; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) acc = fmaf(L[(base + r) * LS + base + j], x[j], acc);
      if (r > c) x[r] = -acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) X[(base + r) * LS + base + c] = x[r];
  }
  for (int e = tid; e < 64 * 64; e += TNT) {
    const int i = e >> 6, j = e & 63;
    if ((i >> 4) < (j >> 4)) X[i * LS + j] = 0.f;
  }
  __syncthreads();
  for (int dist = 1; dist <= 3; ++dist) {
    const int nblk = 4 - dist;
    for (int e = tid; e < nblk * 256; e += TNT) {
      const int bi = dist + e / 256, bj = bi - dist, r = (e & 255) >> 4, c = e & 15;
      float acc = 0.f;
      for (int kb = bj; kb < bi; ++kb)
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          acc = fmaf(L[(bi * 16 + r) * LS + kb * 16 + kk], X[(kb * 16 + kk) * LS + bj * 16 + c], acc);
      T[e] = acc;
    }
    __syncthreads();
    for (int e = tid; e < nblk * 256; e += TNT) {
      const int bi = dist + e / 256, bj = bi - dist, r = (e & 255) >> 4, c = e & 15;
      const int eb = e & ~255;
      float acc = 0.f;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        acc = fmaf(X[(bi * 16 + r) * LS + bi * 16 + kk], T[eb + kk * 16 + c], acc);
      X[(bi * 16 + r) * LS + bj * 16 + c] = -acc;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(TNT, 1) tc_fwd_kernel(SimtFwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  float *sG = reinterpret_cast<float *>(sm + OFF_SMALL);  // [2][64] raw g, then cumulative
  float *sBeta = sG + 128;                                // [2][64]
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_SMALL + 1024);
  uint32_t *tbase_p = reinterpret_cast<uint32_t *>(sm + OFF_SMALL + 1040);
  float *sL = reinterpret_cast<float *>(sm + OFF_L);
  float *sX = reinterpret_cast<float *>(sm + OFF_X);
  float *sT = reinterpret_cast<float *>(sm + OFF_T);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H, h = blockIdx.y, z = blockIdx.z;
  const int col0 = blockIdx.x * TBV;
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
  const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o);

  // ---- the run -------------------------------------------------------------
  int64_t r0, r1, chunk_base = 0;
  int b = 0, s = 0, state_idx;
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
  if (a.cu) {
    r0 = a.cu[z];
    r1 = a.cu[z + 1];
    bool ok = r0 >= 0 && r1 > r0 && r1 <= a.T;
    if (ok) {
      for (int m = 0; m < z; ++m) chunk_base += (a.cu[m + 1] - a.cu[m] + GDN_CHUNK - 1) / GDN_CHUNK;
      ok = chunk_base + (r1 - r0 + GDN_CHUNK - 1) / GDN_CHUNK <= a.num_chunks;
    }
    if (!ok) {
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      return;
    }
    state_idx = z;
  } else if (a.nseg > 0) {
    b = z / a.nseg;
    s = z % a.nseg;
    r0 = (int64_t)b * a.T + (int64_t)s * a.seg_len;
    r1 = min(r0 + a.seg_len, (int64_t)b * a.T + a.T);
    chunk_base = (int64_t)s * a.seg_len / GDN_CHUNK;
    state_idx = b;
  } else {
    b = z;
    r0 = (int64_t)b * a.T;
    r1 = r0 + a.T;
    state_idx = b;
  }
  const int64_t nchunks = (r1 - r0 + GDN_CHUNK - 1) / GDN_CHUNK;

  // ---- tensor memory and barrier ---------------------------------------------
  if (warp == 0) {
    tmem_alloc(tbase_p, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tbase_p;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const int row = tid & 127;   // TMEM lane / key row owned by this thread
  const int half = tid >> 7;   // column half owned by this thread
  uint32_t phase = 0;
  bool bad = false;

  // ---- initial state ------------------------------------------------------------
  float hreg[32];
  {
    const float *src = nullptr;
    if (a.h0) {
      const int64_t slot = a.nseg > 0 ? (((int64_t)b * H + h) * a.nseg + s) : ((int64_t)state_idx * H + h);
      src = a.h0 + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV + col0 + half * 32;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) hreg[j] = src ? src[j] : 0.f;
  }

  auto write_ht_bf16 = [&]() {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int c = half * 32 + j;
      st_bf16(sm, OFF_HT + (row >> 6) * 8192 + sw128_offset(c, row & 63), hreg[j]);
    }
  };
  write_ht_bf16();

  auto issue_loads = [&](int64_t ci, int stage) {
    const int64_t c0 = r0 + ci * GDN_CHUNK;
    const int n = (int)min((int64_t)GDN_CHUNK, r1 - c0);
    const uint32_t kq = smem_u32(sm + OFF_KQ + stage * SZ_KQ);
    const uint32_t vb = smem_u32(sm + OFF_V + stage * SZ_V);
    for (int x = tid; x < 2048 + 512; x += TNT) {
      if (x < 2048) {
        const int which = x >> 10, rem = x & 1023, r = rem >> 4, f16 = rem & 15;
        const bool valid = r < n;
        const __nv_bfloat16 *src = (which ? q : k) + ((c0 + (valid ? r : 0)) * H + h) * GDN_DK + f16 * 8;
        const int rr = r + which * 64, kb = f16 >> 3, c8 = f16 & 7;
        const uint32_t dst = kq + kb * 16384 + (rr >> 3) * 1024 + (rr & 7) * 128 + ((c8 ^ (rr & 7)) << 4);
        cp_async16(dst, src, valid ? 16u : 0u);
      } else {
        const int rem = x - 2048, r = rem >> 3, c8 = rem & 7;
        const bool valid = r < n;
        const __nv_bfloat16 *src = v + ((c0 + (valid ? r : 0)) * H + h) * GDN_DV + col0 + c8 * 8;
        cp_async16(vb + r * 128 + c8 * 16, src, valid ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  // gate and beta of one chunk, one row per thread (tid < 64)
  auto load_gb = [&](int64_t ci, float &gv, float &bv) {
    const int64_t c0 = r0 + ci * GDN_CHUNK;
    const int n = (int)min((int64_t)GDN_CHUNK, r1 - c0);
    gv = 0.f;
    bv = 0.f;
    if (tid < n) {
      gv = a.g[(c0 + tid) * H + h];
      bv = __bfloat162float(beta[(c0 + tid) * H + h]);
    }
  };

  auto mma_wait = [&]() {
    if (!mbar_wait(bar, phase & 1, WAIT_LIMIT)) bad = true;
    ++phase;
    fence_after_sync();
  };

  if (nchunks > 0) {
    issue_loads(0, 0);
    float gv, bv;
    load_gb(0, gv, bv);
    if (tid < 64) {
      sG[tid] = gv;
      sBeta[tid] = bv;
    }
  }

  const float scale = a.scale;
  const bool e2 = a.use_exp2 != 0;
  const bool lead = blockIdx.x == 0;
  for (int64_t ci = 0; ci < nchunks && !bad; ++ci) {
    const int stage = (int)(ci & 1);
    const int64_t c0 = r0 + ci * GDN_CHUNK;
    const int n = (int)min((int64_t)GDN_CHUNK, r1 - c0);
    uint8_t *kq = sm + OFF_KQ + stage * SZ_KQ;
    const uint8_t *vs = sm + OFF_V + stage * SZ_V;
    float *G = sG + stage * 64;
    float *Bt = sBeta + stage * 64;

    // entry state of this chunk
    if (a.h_chunks) {
      const int64_t slot = a.cu ? (chunk_base + ci) * H + h : ((int64_t)b * H + h) * NT + chunk_base + ci;
      float *dst = a.h_chunks + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV + col0 + half * 32;
#pragma unroll
      for (int j = 0; j < 32; ++j) dst[j] = hreg[j];
    }

    cp_async_wait_all();
    fence_proxy_async();
    __syncthreads();
    float g_next = 0.f, b_next = 0.f;
    if (ci + 1 < nchunks) {
      issue_loads(ci + 1, stage ^ 1);
      load_gb(ci + 1, g_next, b_next);
    }

    // P1: S = [K; Q] K^T
    if (tid == 0) {
      fence_after_sync();
      const uint32_t kqa = smem_u32(kq);
      mma_tiles(tmem + T_S, kqa, 16384, kqa, 16384, 128, idesc_bf16(128, 64), false);
      mma_commit(bar);
    }
    // cumulative gate (rows past the end carry g = 0, so G stays flat there)
    if (warp == 0) {
      const int lane = tid;
      const float x0 = G[2 * lane], x1 = G[2 * lane + 1];
      const float pair = x0 + x1;
      float incl = pair;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const float ex = incl - pair;
      G[2 * lane] = ex + x0;
      G[2 * lane + 1] = ex + pair;
    }
    __syncthreads();
    if (lead && a.g_cumsum && tid < n) a.g_cumsum[(c0 + tid) * H + h] = G[tid];
    const float Gl = G[63];
    mma_wait();

    // gated Gram rows: L (fp32, for the solve) and A_qk (bf16 operand rows 64..127)
    {
      float sv[32];
      float t16[16];
      tmem_ld16(tmem + lane_base + T_S + half * 32, t16);
#pragma unroll
      for (int j = 0; j < 16; ++j) sv[j] = t16[j];
      tmem_ld16(tmem + lane_base + T_S + half * 32 + 16, t16);
#pragma unroll
      for (int j = 0; j < 16; ++j) sv[16 + j] = t16[j];
      tmem_ld_wait();
      if (row < 64) {
        const int i = row;
        const float bi = Bt[i], gi = G[i];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = half * 32 + jj;
          sL[i * LS + j] = j < i ? bi * sv[jj] * gexp(gi - G[j], e2) : 0.f;
        }
      } else {
        const int i = row - 64;
        const float gi = G[i];
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = half * 32 + jj;
          st_bf16(sm, OFF_AOP + sw128_offset(64 + i, j), j <= i ? sv[jj] * gexp(gi - G[j], e2) : 0.f);
        }
      }
    }
    fence_before_sync();
    __syncthreads();

    solve64(sL, sX, sT, tid);

    // X into the operand tiles (and the optional fp32 A slot)
    for (int e = tid; e < 64 * 64; e += TNT) {
      const int i = e >> 6, j = e & 63;
      const float x = sX[i * LS + j];
      st_bf16(sm, OFF_AOP + sw128_offset(i, j), x);
      st_bf16(sm, OFF_AT + sw128_offset(j, i), x);
      if (lead && a.A && i < n) a.A[((c0 + i) * H + h) * GDN_CHUNK + j] = x;
    }
    __syncthreads();  // solve buffers are dead from here

    // [beta Kg | beta V]^T and kgl^T, 8 tokens per item (one 16-byte chunk)
    for (int e = tid; e < (192 + 128) * 8; e += TNT) {
      const int f = e >> 3, j0 = (e & 7) * 8;
      alignas(16) __nv_bfloat16 pk[8];
      if (f < 128) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int j = j0 + t;
          const float kv = ld_bf16(kq, (f >> 6) * 16384 + sw128_offset(j, f & 63));
          pk[t] = __float2bfloat16_rn(Bt[j] * kv * gexp(G[j], e2));
        }
        *reinterpret_cast<uint4 *>(sm + OFF_B3 + sw128_offset(f, j0)) = *reinterpret_cast<uint4 *>(pk);
      } else if (f < 192) {
        const int cc = f - 128;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int j = j0 + t;
          const float vv = ld_bf16(vs, j * 128 + cc * 2);
          pk[t] = __float2bfloat16_rn(Bt[j] * vv);
        }
        *reinterpret_cast<uint4 *>(sm + OFF_B3 + sw128_offset(f, j0)) = *reinterpret_cast<uint4 *>(pk);
      } else {
        const int d = f - 192;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int j = j0 + t;
          const float kv = ld_bf16(kq, (d >> 6) * 16384 + sw128_offset(j, d & 63));
          pk[t] = __float2bfloat16_rn(kv * gexp(Gl - G[j], e2));
        }
        *reinterpret_cast<uint4 *>(sm + OFF_KL + sw128_offset(d, j0)) = *reinterpret_cast<uint4 *>(pk);
      }
    }
    fence_proxy_async();
    __syncthreads();

    // P3a: [X; A_qk] X  -> rows 64..127 hold A_qk X
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_S, smem_u32(sm + OFF_AOP), 16384, smem_u32(sm + OFF_AT), 8192, 64,
                idesc_bf16(128, 64), false);
      mma_commit(bar);
    }
    mma_wait();
    if ((warp & 3) >= 2) {  // lanes 64..127
      float t16[16];
      const int i = row - 64;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tmem_ld16(tmem + lane_base + T_S + half * 32 + part * 16, t16);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          st_bf16(sm, OFF_AOP + sw128_offset(64 + i, half * 32 + part * 16 + jj), t16[jj]);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();

    // P3b: [X; A_qk X] [beta Kg | beta V]
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_W, smem_u32(sm + OFF_AOP), 16384, smem_u32(sm + OFF_B3), 24576, 64,
                idesc_bf16(128, 192), false);
      mma_commit(bar);
    }
    mma_wait();
    // operand of P4: rows 0..63 = -w, rows 64..127 = Qg - A_qk w
    {
      float t16[16];
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        const int dcol = half * 64 + part * 16;
        tmem_ld16(tmem + lane_base + T_W + dcol, t16);
        tmem_ld_wait();
        if (row < 64) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int d = dcol + jj;
            st_bf16(sm, OFF_WQ + (d >> 6) * 16384 + sw128_offset(row, d & 63), -t16[jj]);
          }
        } else {
          const int i = row - 64;
          const float eg = gexp(G[i], e2);
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int d = dcol + jj;
            const float qv = ld_bf16(kq, (d >> 6) * 16384 + sw128_offset(64 + i, d & 63));
            st_bf16(sm, OFF_WQ + (d >> 6) * 16384 + sw128_offset(row, d & 63), qv * eg - t16[jj]);
          }
        }
      }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();

    // P4: [v_new; o/scale] = [u; A_qk u] + [-w; q'] h
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_W + 128, smem_u32(sm + OFF_WQ), 16384, smem_u32(sm + OFF_HT), 8192, 128,
                idesc_bf16(128, 64), true);
      mma_commit(bar);
    }
    mma_wait();
    {
      float t16[16];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        const int cb = half * 32 + part * 16;
        tmem_ld16(tmem + lane_base + T_W + 128 + cb, t16);
        tmem_ld_wait();
        if (row < 64) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) st_bf16(sm, OFF_VN + sw128_offset(cb + jj, row), t16[jj]);
        } else if (row - 64 < n) {
          alignas(16) __nv_bfloat16 pk[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) pk[jj] = __float2bfloat16_rn(scale * t16[jj]);
          uint4 *dst = reinterpret_cast<uint4 *>(o + ((c0 + row - 64) * H + h) * GDN_DV + col0 + cb);
          dst[0] = reinterpret_cast<uint4 *>(pk)[0];
          dst[1] = reinterpret_cast<uint4 *>(pk)[1];
        }
      }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();

    // P5: kgl^T v_new
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_S, smem_u32(sm + OFF_KL), 16384, smem_u32(sm + OFF_VN), 8192, 64,
                idesc_bf16(128, 64), false);
      mma_commit(bar);
    }
    mma_wait();
    {
      const float el = gexp(Gl, e2);
      float t16[16];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tmem_ld16(tmem + lane_base + T_S + half * 32 + part * 16, t16);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) hreg[part * 16 + jj] = fmaf(el, hreg[part * 16 + jj], t16[jj]);
      }
    }
    write_ht_bf16();
    if (tid < 64) {
      sG[(stage ^ 1) * 64 + tid] = g_next;
      sBeta[(stage ^ 1) * 64 + tid] = b_next;
    }
    fence_proxy_async();
    fence_before_sync();
    if (__syncthreads_or(bad)) bad = true;
  }

  if (bad) {
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    cp_async_wait_all();
    mbar_wait(bar, phase & 1, WAIT_LIMIT);  // let an MMA still in flight finish
  } else {
    float *dst = nullptr;
    if (a.ht && (a.nseg == 0 || s == a.nseg - 1))
      dst = a.ht + ((int64_t)state_idx * H + h) * GDN_DK * GDN_DV;
    if (dst) {
      float *p = dst + (int64_t)row * GDN_DV + col0 + half * 32;
#pragma unroll
      for (int j = 0; j < 32; ++j) p[j] = hreg[j];
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int tc_fwd_bv() { return TBV; }

cudaError_t launch_tc_fwd(const SimtFwdArgs &a, dim3 grid, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  tc_fwd_kernel<<<grid, TNT, SMEM_BYTES, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
