// Tensor-core (tcgen05) chunk forward for bf16 inputs, scalar gate (sm_103a).
//
// One CTA (512 threads) owns one independent run (batch row, packed document
// or segment) of one head and 64 of the 128 state columns. The state slice h
// (128 x 64, fp32) lives in registers: thread = key row (its tensor-memory
// lane) and 16 columns. Per 64-token chunk the CTA takes the steps of the
// chunk algorithm (north star; GDN Ascend C adapter forward; chunk_fwd_h and
// chunk_kda_fwd_finalize of the KDA adapter) with every dense contraction on
// the tensor core (bf16 operands in shared memory, fp32 accumulators in
// tensor memory, M = 128):
//
//   P1   S = [K; Q] K^T                   -> L = strictly-lower(beta S (.) Gamma),
//                                            A_qk = lower-incl(S_qk (.) Gamma)
//   X = (I + L)^-1: 16x16 diagonal blocks by fp32 forward substitution, the
//        off-diagonal block levels with tf32 mma.sync
//   P3a  [X; A_qk] X                      -> A_qk X
//   P3b  [X; A_qk X] [beta e^G K | beta V] -> [w | u ; A_qk w | A_qk u]
//   P4   [-w; e^G Q - A_qk w] h accumulated onto [u; A_qk u] -> [v_new ; o / scale]
//   P5   (e^(G_last - G) K)^T v_new       -> h <- e^(G_last) h + P5
//
// Every operand tile is K-major with the 128-byte swizzle; the transposed
// tiles (X^T, [beta e^G K | beta V]^T, (e^(G_last-G) K)^T, v_new^T, h^T) are
// made with ldmatrix.trans / stmatrix, scaling per token on the way, and all
// other operands are written with 16-byte stores. Loads of chunk c+1 (cp.async,
// zero-filled past the run end) and its P1 overlap the work on chunk c. Every
// mbarrier wait is bounded; a wait that runs out sets the device flag and the
// CTA leaves after its MMAs have drained and its tensor memory is released.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tc;
using namespace tile;

constexpr int TBV = 64;   // state columns per CTA
constexpr int NTH = 512;  // threads per CTA
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S0 = 0;    // 2 x 64 columns: S (per chunk parity), then A_qk X
constexpr uint32_t T_W = 128;   // 192 columns: P3b; P4 accumulates into [T_W+128, T_W+192)
constexpr uint32_t T_P5 = 320;  // 64 columns

// shared memory map (bytes from a 1024-aligned base); every tile K-major, 128 B rows
constexpr int SZ_KQ = 32768;                     // [K; Q]: 2 K-blocks x 128 rows
constexpr int SZ_V = 8192;                       // V slice: 64 rows
constexpr int OFF_KQ = 0;                        // 2 stages
constexpr int OFF_V = OFF_KQ + 2 * SZ_KQ;        // 2 stages
constexpr int OFF_AOP = OFF_V + 2 * SZ_V;        // [X; A_qk | A_qk X]     128 rows, K = 64
constexpr int OFF_XT = OFF_AOP + 16384;          // X^T                    64 rows, K = 64
constexpr int OFF_B3 = OFF_XT + 8192;            // [b e^G K | b V]^T      192 rows, K = 64
constexpr int OFF_KL = OFF_B3 + 24576;           // (e^(Gl-G) K)^T         128 rows, K = 64
constexpr int OFF_WQ = OFF_KL + 16384;           // [-w; q']               2 K-blocks x 128 rows
constexpr int OFF_HT = OFF_WQ + 32768;           // h^T                    2 K-blocks x 64 rows
constexpr int OFF_VN = OFF_HT + 16384;           // v_new^T                64 rows, K = 64
constexpr int OFF_SMALL = OFF_VN + 8192;
constexpr int SMALL_BYTES = 17408;
constexpr int SMEM_BYTES = OFF_SMALL + SMALL_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
// aliases: the solve's fp32 blocks live in WQ (free until WQ is formed); the
// row-major staging of v_new and h (for their transposes) lives in B3 (free
// after P3b)
constexpr int OFF_LB = OFF_WQ;               // 10 lower 16x16 fp32 blocks of L
constexpr int OFF_XB = OFF_WQ + 10 * 1024;   // 10 blocks of X
constexpr int OFF_TB = OFF_WQ + 20 * 1024;   // 4 scratch blocks (one per solve warp)
static_assert(24 * 1024 <= 32768, "solve buffers");
constexpr int OFF_STG = OFF_B3;              // staging: v_new 64 rows (8 KB), h 128 rows (16 KB)
static_assert(16384 <= 24576, "staging");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct TcState {
  float G[2][64], eG[2][64], eGL[2][64], bEG[2][64];  // per chunk parity
  // e^(G_i - G_r(i)) with r(i) the first row of i's 16-row block, and
  // e^(G_16b - G_j) for j < 16b: the Gram gate of an off-diagonal block is their
  // product (both factors <= 1, no overflow for any gate strength)
  float eA[2][64], eB[2][4][64];
  // gate of the four diagonal 16x16 blocks: base^(G_{16b+r} - G_{16b+j}) for j <= r, else 0
  alignas(16) float gd[2][4][16][20];  // rows padded to 20: conflict-free float4 reads
  float g[2][64];                                     // raw gate per load stage
  float braw[2][64];                                  // raw beta per load stage
  float beta[2][64];
  float EL[2];
  uint64_t bar_s[2], bar_m;
  uint32_t tmem;
};
static_assert(sizeof(TcState) <= SMALL_BYTES, "small state");

template <bool E2>
__global__ void __launch_bounds__(NTH, 1) tc_fwd_kernel(SimtFwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  TcState &st = *reinterpret_cast<TcState *>(sm + OFF_SMALL);
  float *LB = reinterpret_cast<float *>(sm + OFF_LB);
  float *XB = reinterpret_cast<float *>(sm + OFF_XB);
  float *TB = reinterpret_cast<float *>(sm + OFF_TB);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3;         // tensor-memory lane quarter of this warp
  const int cg = warp >> 2;        // column group: 16 of 64 columns
  const int row = q4 * 32 + lane;  // tensor-memory lane = matrix row
  const int H = a.H, h = blockIdx.y, z = blockIdx.z;
  const int col0 = blockIdx.x * TBV;
  const float scale = a.scale;
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
  const __nv_bfloat16 *beta = static_cast<const __nv_bfloat16 *>(a.beta);
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o);

  // ---- the run -------------------------------------------------------------------
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
  const int64_t nch = (r1 - r0 + GDN_CHUNK - 1) / GDN_CHUNK;
  auto chunk_rows = [&](int64_t c) { return (int)min((int64_t)GDN_CHUNK, r1 - (r0 + c * GDN_CHUNK)); };

  // ---- tensor memory, barriers -----------------------------------------------------
  if (warp == 0) {
    tmem_alloc(&st.tmem, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&st.bar_s[0], 1);
    mbar_init(&st.bar_s[1], 1);
    mbar_init(&st.bar_m, 1);
    mbar_fence_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = st.tmem;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);  // this warp's lane quarter
  uint32_t ph_s0 = 0, ph_s1 = 0, ph_m = 0;
  bool bad = false;
  auto wait_bar = [&](uint64_t *bar, uint32_t &ph) {
    if (!mbar_wait(bar, ph & 1, WAIT_LIMIT)) bad = true;
    ++ph;
    fence_after_sync();
  };
  // one MMA group issued by thread 0 and waited for by every thread
  auto mma_sync_wait = [&]() {
    if (tid == 0) mma_commit(&st.bar_m);
    wait_bar(&st.bar_m, ph_m);
  };

  // ---- loads -----------------------------------------------------------------------
  auto issue_loads = [&](int64_t c) {
    const int stage = (int)(c & 1);
    const int64_t c0 = r0 + c * GDN_CHUNK;
    const int n = chunk_rows(c);
    const uint32_t kq = sb + OFF_KQ + stage * SZ_KQ;
    const uint32_t vb = sb + OFF_V + stage * SZ_V;
#pragma unroll
    for (int x = tid; x < 2048 + 512; x += NTH) {
      if (x < 2048) {
        const int which = x >> 10, r = (x >> 4) & 63, f16 = x & 15;
        const bool valid = r < n;
        const __nv_bfloat16 *src = (which ? q : k) + ((c0 + (valid ? r : 0)) * H + h) * GDN_DK + f16 * 8;
        cp_async16(kq + (f16 >> 3) * 16384 + chunk_off(r + which * 64, f16 & 7), src, valid ? 16u : 0u);
      } else {
        const int r = (x - 2048) >> 3, c8 = x & 7;
        const bool valid = r < n;
        const __nv_bfloat16 *src = v + ((c0 + (valid ? r : 0)) * H + h) * GDN_DV + col0 + c8 * 8;
        cp_async16(vb + chunk_off(r, c8), src, valid ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  // gate and beta rows of chunk c (threads < 64; zero past the run end), loaded
  // into registers well before they are stored for chunk_factors
  const float *gsrc = a.g_cum_in ? a.g_cum_in : a.g;
  auto load_gb = [&](int64_t c) -> float2 {
    float2 gb = make_float2(0.f, 0.f);
    if (tid < 64 && c < nch) {
      const int64_t c0 = r0 + c * GDN_CHUNK;
      if (tid < chunk_rows(c)) {
        gb.x = gsrc[(c0 + tid) * H + h];
        gb.y = __bfloat162float(beta[(c0 + tid) * H + h]);
      }
    }
    return gb;
  };
  auto store_gb = [&](int64_t c, float2 gb) {
    if (tid < 64) {
      st.g[c & 1][tid] = gb.x;
      st.braw[c & 1][tid] = gb.y;
    }
  };
  // cumulative gate and per-token factors of chunk c once its loads landed
  // Run by warps 4..15 only (named barrier 2), so that warps 0..3 can go on with
  // the solve; the results are read after the next CTA-wide barrier.
  auto chunk_factors = [&](int64_t c) {
    if (warp < 4) return;
    const int par = (int)(c & 1);
    const int n = chunk_rows(c);
    const int t = tid - 128;  // 0..383
    if (a.g_cum_in) {  // saved cumulative gate; rows past the end repeat the last one
      if (t < 64) st.G[par][t] = st.g[par][min(t, n - 1)];
    } else if (warp == 4) {
      const float x0 = st.g[par][2 * lane], x1 = st.g[par][2 * lane + 1];
      const float pair = x0 + x1;
      float incl = pair;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const float ex = incl - pair;
      st.G[par][2 * lane] = ex + x0;
      st.G[par][2 * lane + 1] = ex + pair;
    }
    if (t < 64) st.beta[par][t] = st.braw[par][t];
    asm volatile("bar.sync 2, 384;" ::: "memory");
    if (t < 64) {
      const float G = st.G[par][t], Gl = st.G[par][63];
      st.eG[par][t] = gexp<E2>(G);
      st.eGL[par][t] = gexp<E2>(Gl - G);
      st.bEG[par][t] = st.beta[par][t] * gexp<E2>(G);
      st.eA[par][t] = gexp<E2>(G - st.G[par][t & ~15]);
#pragma unroll
      for (int bb = 1; bb < 4; ++bb)
        st.eB[par][bb][t] = t < 16 * bb ? gexp<E2>(st.G[par][16 * bb] - G) : 0.f;
      if (t == 0) st.EL[par] = gexp<E2>(Gl);
      if (a.g_cumsum && blockIdx.x == 0 && t < n) a.g_cumsum[(r0 + c * GDN_CHUNK + t) * H + h] = G;
    }
    for (int e = t; e < 4 * 256; e += NTH - 128) {  // diagonal-block gates
      const int bb = e >> 8, r = (e >> 4) & 15, j = e & 15;
      st.gd[par][bb][r][j] = j <= r ? gexp<E2>(st.G[par][16 * bb + r] - st.G[par][16 * bb + j]) : 0.f;
    }
  };
  auto issue_p1 = [&](int64_t c) {  // S = [K; Q] K^T
    if (tid == 0) {
      fence_after_sync();
      const uint32_t kq = sb + OFF_KQ + (int)(c & 1) * SZ_KQ;
      mma_tiles(tmem + T_S0 + 64 * (uint32_t)(c & 1), kq, 16384, kq, 16384, 128, idesc_bf16(128, 64), false);
      mma_commit(&st.bar_s[c & 1]);
    }
  };

  // ---- state ------------------------------------------------------------------------
  float hreg[16];
  {
    const float *src = nullptr;
    if (a.h0) {
      const int64_t slot = a.nseg > 0 ? (((int64_t)b * H + h) * a.nseg + s) : ((int64_t)state_idx * H + h);
      src = a.h0 + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV + col0 + cg * 16;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) hreg[j] = src ? src[j] : 0.f;
  }
  // h^T operand: h row-major through the staging tile, then 16x16 transposes
  auto write_h_operand = [&]() {
    uint8_t *stg = sm + OFF_STG;
    *reinterpret_cast<uint4 *>(stg + chunk_off(row, cg * 2)) = pack8(hreg);
    *reinterpret_cast<uint4 *>(stg + chunk_off(row, cg * 2 + 1)) = pack8(hreg + 8);
    __syncthreads();
    for (int jb = warp; jb < 32; jb += NTH / 32) {  // 8 key blocks x 4 column blocks
      const int rb = jb >> 2, cb = jb & 3;
      trans16(TransJob{sb + OFF_STG, rb * 16, cb * 2, sb + OFF_HT + (rb >> 2) * 8192, cb * 16}, nullptr, lane);
    }
  };

  // ---- prologue -----------------------------------------------------------------------
  if (nch > 0) {
    issue_loads(0);
    store_gb(0, load_gb(0));
    store_gb(1, load_gb(1));
    cp_async_wait<0>();
    fence_proxy_async();
    __syncthreads();
    issue_p1(0);
    chunk_factors(0);
    if (nch > 1) issue_loads(1);
  }
  write_h_operand();
  fence_proxy_async();
  __syncthreads();

  const bool lead = blockIdx.x == 0;
  for (int64_t c = 0; c < nch && !bad; ++c) {
    const int par = (int)(c & 1);
    const int64_t c0 = r0 + c * GDN_CHUNK;
    const int n = chunk_rows(c);
    const uint32_t kq = sb + OFF_KQ + par * SZ_KQ;
    const uint32_t vs = sb + OFF_V + par * SZ_V;
    const float *G = st.G[par];
    const float2 gb_pf = load_gb(c + 2);  // gate and beta rows of chunk c+2, stored at the end

    if (a.h_chunks) {  // entry state of chunk c
      const int64_t slot = a.cu ? (chunk_base + c) * H + h : ((int64_t)b * H + h) * NT + chunk_base + c;
      float4 *dst = reinterpret_cast<float4 *>(a.h_chunks + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV +
                                               col0 + cg * 16);
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4)
        dst[g4] = make_float4(hreg[g4 * 4], hreg[g4 * 4 + 1], hreg[g4 * 4 + 2], hreg[g4 * 4 + 3]);
    }

    // ---- gated Gram rows: L (fp32 blocks) and A_qk (operand rows 64..127) --------------
    if (par) wait_bar(&st.bar_s[1], ph_s1); else wait_bar(&st.bar_s[0], ph_s0);
    {
      float sv[16];
      tmem_ld16(tl + T_S0 + 64 * par + cg * 16, sv);
      tmem_ld_wait();
      if (row < 64) {
        const int i = row, bi = i >> 4;
        if (bi >= cg) {
          const float bt = st.beta[par][i], gi = G[i];
          float vals[16];
          if (cg < bi) {  // off-diagonal block: factorised gate
            const float fa = bt * st.eA[par][i];
            const float *fb = st.eB[par][bi] + cg * 16;
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) vals[jj] = fa * sv[jj] * fb[jj];
          } else {  // diagonal block: tabulated gate, strictly lower part
            float gdr[16];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              *reinterpret_cast<float4 *>(gdr + 4 * k4) = reinterpret_cast<const float4 *>(st.gd[par][bi][i & 15])[k4];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) vals[jj] = jj < (i & 15) ? bt * sv[jj] * gdr[jj] : 0.f;
          }
          float *Lrow = LB + blk(bi, cg) * 256;
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4)
            *reinterpret_cast<float4 *>(Lrow + bsw(i & 15, g4 * 4)) =
                make_float4(vals[g4 * 4], vals[g4 * 4 + 1], vals[g4 * 4 + 2], vals[g4 * 4 + 3]);
        }
      } else {
        const int i = row - 64, bi = i >> 4;
        const float gi = G[i];
        float vals[16];
        if (cg < bi) {
          const float fa = st.eA[par][i];
          const float *fb = st.eB[par][bi] + cg * 16;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) vals[jj] = fa * sv[jj] * fb[jj];
        } else if (cg == bi) {  // diagonal block: tabulated gate (zero above the diagonal)
          float gdr[16];
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            *reinterpret_cast<float4 *>(gdr + 4 * k4) = reinterpret_cast<const float4 *>(st.gd[par][bi][i & 15])[k4];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) vals[jj] = sv[jj] * gdr[jj];
        } else {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) vals[jj] = 0.f;
        }
        *reinterpret_cast<uint4 *>(sm + OFF_AOP + chunk_off(row, cg * 2)) = pack8(vals);
        *reinterpret_cast<uint4 *>(sm + OFF_AOP + chunk_off(row, cg * 2 + 1)) = pack8(vals + 8);
      }
    }
    fence_before_sync();
    __syncthreads();
    // ---- next chunk: loads landed -> its factors and P1 (overlaps this chunk) ------------
    if (c + 1 < nch) {
      cp_async_wait<0>();
      fence_proxy_async();
      __syncthreads();
      issue_p1(c + 1);
      chunk_factors(c + 1);
    }

    // ---- X = (I + L)^-1 on warps 0..3; K and V transposes on warps 4..15 meanwhile -------
    if (warp < 4) {
      solve_blocks(LB, XB, TB, tid);
    } else {
      for (int jb = warp - 4; jb < 32 + 16; jb += NTH / 32 - 4) {
        if (jb < 32) {  // K: 4 token blocks x 8 feature blocks -> B3 rows 0..127 and KL
          const int rb = jb >> 3, fb = jb & 7;
          const uint32_t src = kq + (fb >> 2) * 16384;
          const int cc = (fb & 3) * 2;
          trans16(TransJob{src, rb * 16, cc, sb + OFF_B3, fb * 16}, st.bEG[par], lane);
          trans16(TransJob{src, rb * 16, cc, sb + OFF_KL, fb * 16}, st.eGL[par], lane);
        } else {  // V: 4 token blocks x 4 column blocks -> B3 rows 128..191
          const int t = jb - 32, rb = t >> 2, cb = t & 3;
          trans16(TransJob{vs, rb * 16, cb * 2, sb + OFF_B3, 128 + cb * 16}, st.beta[par], lane);
        }
      }
    }
    __syncthreads();
    if (row < 64) {  // X into operand rows 0..63 (and the optional fp32 A slot)
      const int i = row, bi = i >> 4;
      float vals[16];
      if (bi >= cg) {
        const float *Xr = XB + blk(bi, cg) * 256;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          const float4 t = *reinterpret_cast<const float4 *>(Xr + bsw(i & 15, g4 * 4));
          vals[g4 * 4] = t.x;
          vals[g4 * 4 + 1] = t.y;
          vals[g4 * 4 + 2] = t.z;
          vals[g4 * 4 + 3] = t.w;
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) vals[jj] = 0.f;
      }
      *reinterpret_cast<uint4 *>(sm + OFF_AOP + chunk_off(i, cg * 2)) = pack8(vals);
      *reinterpret_cast<uint4 *>(sm + OFF_AOP + chunk_off(i, cg * 2 + 1)) = pack8(vals + 8);
      if (a.A && lead && i < n) {
        float4 *Ad = reinterpret_cast<float4 *>(a.A + ((c0 + i) * H + h) * GDN_CHUNK + cg * 16);
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4)
          Ad[g4] = make_float4(vals[g4 * 4], vals[g4 * 4 + 1], vals[g4 * 4 + 2], vals[g4 * 4 + 3]);
      }
    }
    __syncthreads();
    if (warp < 16) {  // X^T: 4 x 4 blocks of the 64x64 X
      const int rb = warp >> 2, cb = warp & 3;
      trans16(TransJob{sb + OFF_AOP, rb * 16, cb * 2, sb + OFF_XT, cb * 16}, nullptr, lane);
    }
    fence_proxy_async();
    __syncthreads();

    // ---- P3a: [X; A_qk] X -> rows 64..127 hold A_qk X -------------------------------------
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_S0 + 64 * par, sb + OFF_AOP, 16384, sb + OFF_XT, 8192, 64, idesc_bf16(128, 64), false);
    }
    mma_sync_wait();
    if (row >= 64) {
      float sv[16];
      tmem_ld16(tl + T_S0 + 64 * par + cg * 16, sv);
      tmem_ld_wait();
      *reinterpret_cast<uint4 *>(sm + OFF_AOP + chunk_off(row, cg * 2)) = pack8(sv);
      *reinterpret_cast<uint4 *>(sm + OFF_AOP + chunk_off(row, cg * 2 + 1)) = pack8(sv + 8);
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    // ---- P3b: [X; A_qk X] [b e^G K | b V] ----------------------------------------------------
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_W, sb + OFF_AOP, 16384, sb + OFF_B3, 24576, 64, idesc_bf16(128, 192), false);
    }
    mma_sync_wait();
    // ---- operand of P4: rows 0..63 = -w, rows 64..127 = e^G Q - A_qk w ----------------------
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const int d0 = cg * 32 + part * 16;  // 16 key columns
      float sv[16];
      tmem_ld16(tl + T_W + d0, sv);
      tmem_ld_wait();
      const int kb = d0 >> 6, ch = (d0 & 63) >> 3;
      float vals[16];
      if (row < 64) {
#pragma unroll
        for (int t = 0; t < 16; ++t) vals[t] = -sv[t];
      } else {
        const float eg = st.eG[par][row - 64];
        float qf[16];
        const uint8_t *qrow = sm + OFF_KQ + par * SZ_KQ + kb * 16384;
        unpack8(*reinterpret_cast<const uint4 *>(qrow + chunk_off(row, ch)), qf);
        unpack8(*reinterpret_cast<const uint4 *>(qrow + chunk_off(row, ch + 1)), qf + 8);
#pragma unroll
        for (int t = 0; t < 16; ++t) vals[t] = fmaf(qf[t], eg, -sv[t]);
      }
      uint8_t *dst = sm + OFF_WQ + kb * 16384;
      *reinterpret_cast<uint4 *>(dst + chunk_off(row, ch)) = pack8(vals);
      *reinterpret_cast<uint4 *>(dst + chunk_off(row, ch + 1)) = pack8(vals + 8);
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    if (c + 2 < nch) issue_loads(c + 2);  // chunk c's stage is free from here
    // ---- P4: [v_new; o/scale] = [u; A_qk u] + [-w; q'] h ---------------------------------------
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_W + 128, sb + OFF_WQ, 16384, sb + OFF_HT, 8192, 128, idesc_bf16(128, 64), true);
    }
    mma_sync_wait();
    {
      float sv[16];
      tmem_ld16(tl + T_W + 128 + cg * 16, sv);
      tmem_ld_wait();
      if (row < 64) {  // v_new row-major into the staging tile
        *reinterpret_cast<uint4 *>(sm + OFF_STG + chunk_off(row, cg * 2)) = pack8(sv);
        *reinterpret_cast<uint4 *>(sm + OFF_STG + chunk_off(row, cg * 2 + 1)) = pack8(sv + 8);
      } else if (o && row - 64 < n) {
#pragma unroll
        for (int t = 0; t < 16; ++t) sv[t] *= scale;
        uint4 *dst = reinterpret_cast<uint4 *>(o + ((c0 + row - 64) * H + h) * GDN_DV + col0 + cg * 16);
        dst[0] = pack8(sv);
        dst[1] = pack8(sv + 8);
      }
    }
    __syncthreads();
    if (warp < 16) {  // v_new^T: 4 x 4 blocks
      const int rb = warp >> 2, cb = warp & 3;
      trans16(TransJob{sb + OFF_STG, rb * 16, cb * 2, sb + OFF_VN, cb * 16}, nullptr, lane);
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    // ---- P5: (e^(Gl-G) K)^T v_new --------------------------------------------------------------
    if (tid == 0) {
      fence_after_sync();
      mma_tiles(tmem + T_P5, sb + OFF_KL, 16384, sb + OFF_VN, 8192, 64, idesc_bf16(128, 64), false);
    }
    mma_sync_wait();
    {
      float sv[16];
      tmem_ld16(tl + T_P5 + cg * 16, sv);
      tmem_ld_wait();
      const float el = st.EL[par];
#pragma unroll
      for (int t = 0; t < 16; ++t) hreg[t] = fmaf(el, hreg[t], sv[t]);
    }
    fence_before_sync();
    __syncthreads();  // the staging tile (v_new) has been consumed
    write_h_operand();
    store_gb(c + 2, gb_pf);
    fence_proxy_async();
    if (__syncthreads_or(bad)) bad = true;
  }

  if (bad) {
    if (tid == 0) {
      raise_device_flag(a.dev_flag, kDevTimeout);
      mma_commit(&st.bar_m);  // arrives once every MMA issued so far has finished
    }
    cp_async_wait<0>();
    mbar_wait(&st.bar_m, ph_m & 1, WAIT_LIMIT);
  } else if (a.ht && (a.nseg == 0 || s == a.nseg - 1)) {
    float4 *dst = reinterpret_cast<float4 *>(a.ht + ((int64_t)state_idx * H + h) * GDN_DK * GDN_DV +
                                             (int64_t)row * GDN_DV + col0 + cg * 16);
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4)
      dst[g4] = make_float4(hreg[g4 * 4], hreg[g4 * 4 + 1], hreg[g4 * 4 + 2], hreg[g4 * 4 + 3]);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int tc_fwd_bv() { return TBV; }

cudaError_t launch_tc_fwd(const SimtFwdArgs &a, dim3 grid, cudaStream_t st) {
  auto kern = a.use_exp2 ? tc_fwd_kernel<true> : tc_fwd_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, NTH, SMEM_BYTES, st>>>(a);
  return cudaGetLastError();
}

}  // namespace gdn
