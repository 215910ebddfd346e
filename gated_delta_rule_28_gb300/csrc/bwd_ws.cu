// Tensor-core (tcgen05) reverse state recurrence of the backward (dhu) for bf16
// inputs, scalar gate (sm_103a), overlapped with the preparation of the
// previous chunk.
//
// For every run and head, from the last chunk to the first (the reverse loop of
// the hyper-parallel "Diff Coverage" page's kda_state_grad_ext_kernel; KDA
// adapter backward, stage bwd_dhu), with dh the gradient of the chunk's exit
// state:
//
//   dv_new = kgl dh + scale A_qk^T dO                 kgl = K (.) base^(G_last - G)
//   dh    <- base^(G_last) dh + scale (Q (.) base^G)^T dO - w^T dv_new
//                                                      w   = X diag(beta base^G) K
//
// One CTA (512 threads) owns one run of one head and 64 of the 128 value
// columns; dh lives in fp32 registers of the chain warps 0..7, which run
//   D1   [kgl; -] dh            accumulated onto  scale A_qk^T dO   -> dv_new
//   D2   -w^T dv_new            accumulated onto  scale Qg^T dO     -> dh update
// while the producer warps 8..15 prepare the previous chunk: A_qk^T (from
// [Q; K] Q^T and the gate) and the three h-independent products scale A_qk^T dO,
// scale Qg^T dO = Q^T (diag(scale base^G) dO) and w^T (= K^T (X diag(beta base^G))^T),
// with Q, K and dO read in place as MN-major operands. The chain warps form that chunk's
// operands kgl and w^T (from tensor memory) in the parts of their round where they would wait. X diag(beta base^G) and the
// per-token gate factors come from the UT transform kernel.
// Loads are TMA copies completing on mbarriers.
// It writes dh of every chunk (the exit-state gradient) and dv_new for the
// local-gradient kernel -- bf16 tiles in that kernel's layout, bulk-copied from
// the MMA operand tiles (fp32 rows when no tiles are asked for) -- and dh of the
// first chunk's entry as dh0.
// Every mbarrier wait is bounded; a wait that runs out sets the device flag
// and the CTA drains its MMAs, frees its tensor memory and leaves.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tc;
using namespace tile;

constexpr int TBV = 64;   // value columns per CTA
constexpr int NTH = 512;  // 256 chain + 256 producer threads
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S = 0;     // 2 x 64: [Q; K] Q^T per parity (rows 64..127 = K Q^T)
constexpr uint32_t T_I1 = 128;  // 2 x 64: rows 0..63 = scale A_qk^T dO, then dv_new
constexpr uint32_t T_I2 = 256;  // 2 x 64: scale Qg^T dO, then the dh increment
constexpr uint32_t T_WT = 384;  // 64: w^T (keys x tokens)

// shared memory (bytes from a 1024-aligned base); K-major tiles, 128 B rows
constexpr int SZ_STAGE = 32768;               // [Q; K]: 2 K-blocks x 128 rows
constexpr int OFF_ST = 0;                     // 2 stages
constexpr int OFF_X0 = OFF_ST + 2 * SZ_STAGE; // X diag(beta base^G) of even-order chunks (64 rows)
constexpr int OFF_X1 = OFF_X0 + 8192;
constexpr int OFF_DO = OFF_X1 + 8192;         // dO slice per order parity: 64 token rows (MN-major B)
constexpr int OFF_DOS = OFF_DO + 2 * 8192;    // diag(scale base^G) dO: 64 token rows (MN-major B)
constexpr int OFF_AQT = OFF_DOS + 8192;       // A_qk^T rows 0..63 (rows 64..127 of the operand: kgl's,
                                              // whose output rows are not read)
constexpr int OFF_KGL = OFF_AQT + 8192;       // kgl, 2 K-blocks of 64 rows
constexpr int OFF_WT = OFF_KGL + 16384;       // w^T, 128 rows
constexpr int OFF_DHT = OFF_WT + 16384;       // dh: 128 key rows (MN-major B of D1)
constexpr int OFF_DVT = OFF_DHT + 16384;      // dv_new: 64 token rows (MN-major B of D2)
constexpr int OFF_SMALL = OFF_DVT + 8192;
constexpr int SMALL_BYTES = 6144;
// gates of the four diagonal 16x16 blocks, gdn[b][x][y] = base^(G_{16b+x} - G_{16b+y}) for
// x >= y (else 0) at b * GD_B + x * 16 + y; block stride 272 against bank conflicts
constexpr int GD_B = GD_BLOCK;
constexpr int OFF_GD = OFF_SMALL + SMALL_BYTES;
constexpr int SMEM_BYTES = OFF_GD + 4 * GD_B * 4 + 1024;
// The MN-major K^T operand of w^T (the second stage's K rows: two 64-key groups 16 KB apart, 64
// token rows) stays below the small state under either assignment of its descriptor's two
// stride fields (groups 16 KB apart and K rows in 1 KB atoms, or the reverse).
static_assert(OFF_ST + SZ_STAGE + 8192 + 16384 + 8 * 1024 <= OFF_SMALL &&
                  OFF_ST + SZ_STAGE + 8192 + 1024 + 7 * 16384 + 1024 <= OFF_SMALL,
              "MN-major K^T operand extent");
static_assert(SMEM_BYTES <= 232448, "shared memory");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct BwState {
  alignas(16) float tab[2][F_ROWS][64];  // gate factor table per order parity
  float seg[2][64];                 // scale base^G
  float EL[2];
  uint64_t bar_p1, bar_p3, bar_d1, bar_d2, bar_x0, bar_x1;
  uint64_t bar_ld[2], bar_do[2];  // TMA loads per order parity: Q, K, X, factors; dO
  uint32_t tmem;
};
static_assert(sizeof(BwState) <= SMALL_BYTES, "small state");

__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void prod_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }

// TMA maps: q, k, dO over [rows, H*128] and X over [slots*H*64, 64], 64 x 64 boxes
struct BwdMaps {
  TmaMap q, k, dO, x;
};

template <bool E2>
__global__ void __launch_bounds__(NTH, 1) tc_dhu_kernel(BwdArgs a, const __grid_constant__ BwdMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base by pointer arithmetic on the shared array, so that the compiler keeps
  // the shared address space (shared-memory instructions, not generic ones)
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  BwState &st = *reinterpret_cast<BwState *>(sm + OFF_SMALL);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp >= 8;
  const int q4 = warp & 3, hc = (warp >> 2) & 1, row = q4 * 32 + lane;
  const int H = a.H, h = blockIdx.y, z = blockIdx.z;
  const int col0 = blockIdx.x * TBV;
  const float scale = a.scale;

  // ---- the run: chunk slots as the forward (X workspace: xbase + c; states: slot()) ----
  int64_t r0, r1, chunk_base = 0, xbase;
  int b = 0, sg = 0;
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
    xbase = chunk_base;
  } else if (a.nseg > 0) {  // segment sg of batch row b
    b = z / a.nseg;
    sg = z % a.nseg;
    r0 = (int64_t)b * a.T + (int64_t)sg * a.seg_len;
    r1 = min(r0 + a.seg_len, (int64_t)b * a.T + a.T);
    chunk_base = (int64_t)sg * a.seg_len / GDN_CHUNK;
    xbase = (int64_t)b * NT + chunk_base;
  } else {
    b = z;
    r0 = (int64_t)b * a.T;
    r1 = r0 + a.T;
    xbase = (int64_t)b * NT;
  }
  // dht / dh0 state of the run: [N, H, K, V], or [B, H, nseg, K, V] for segments
  const int64_t state_off =
      (a.nseg > 0 ? ((int64_t)b * H + h) * a.nseg + sg : (int64_t)z * H + h) * GDN_DK * GDN_DV;
  const int64_t nch = (r1 - r0 + GDN_CHUNK - 1) / GDN_CHUNK;
  auto chunk_rows = [&](int64_t c) { return (int)min((int64_t)GDN_CHUNK, r1 - (r0 + c * GDN_CHUNK)); };
  auto state_slot = [&](int64_t c) -> int64_t {
    return a.cu ? (chunk_base + c) * H + h : ((int64_t)b * H + h) * NT + chunk_base + c;
  };
  // order index m = nch - 1 - c: the reverse loop visits m = 0, 1, ...
  auto chunk_of = [&](int64_t m) { return nch - 1 - m; };

  // ---- tensor memory, barriers -------------------------------------------------------
  if (warp == 0) {
    tmem_alloc(&st.tmem, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&st.bar_p1, 1);
    mbar_init(&st.bar_p3, 1);
    mbar_init(&st.bar_d1, 1);
    mbar_init(&st.bar_d2, 1);
    mbar_init(&st.bar_x0, 1);
    mbar_init(&st.bar_x1, 1);
    mbar_init(&st.bar_ld[0], 1);
    mbar_init(&st.bar_ld[1], 1);
    mbar_init(&st.bar_do[0], 1);
    mbar_init(&st.bar_do[1], 1);
    mbar_fence_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = st.tmem;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
  bool bad = false;
  auto wait_par = [&](uint64_t *bar, int64_t phase) {
    if (!mbar_wait(bar, (uint32_t)(phase & 1), WAIT_LIMIT)) bad = true;
    fence_after_sync();
  };

  // ---- producer: loads (TMA, issued by one thread: ptid 32, warp 9 lane 0) --------------
  // Rows past the run end are loaded as they are (the next run's tokens, or zeros past
  // the tensor); the gating and the factor scale (scale base^G) are zeroed there, and
  // beta = 0 removes them from w.
  const int ptid = tid - 256;
  const bool loader = warp == 9;  // TMA loads, issued warp-collectively (tc.cuh)
  int64_t last_ld[2] = {-1, -1}, last_do[2] = {-1, -1};  // loader: newest order index per barrier
  auto issue_qkx = [&](int64_t m) {  // Q, K, X and the gate table of order index m
    const int64_t c = chunk_of(m);
    const int s2 = (int)(m & 1);
    const uint32_t stg = sb + OFF_ST + s2 * SZ_STAGE;
    const uint32_t xt = sb + (s2 ? OFF_X1 : OFF_X0);
    const int y = (int)(r0 + c * GDN_CHUNK);
    const int64_t xs = (xbase + c) * H + h;
    uint64_t *bar = &st.bar_ld[s2];
    mbar_expect_tx_w(bar, 5 * 8192 + F_ROWS * GDN_CHUNK * 4);
    tma_load_2d_w(stg, &maps.q, h * GDN_DK, y, bar);  // rows 0..63: Q
    tma_load_2d_w(stg + 16384, &maps.q, h * GDN_DK + 64, y, bar);
    tma_load_2d_w(stg + 8192, &maps.k, h * GDN_DK, y, bar);  // rows 64..127: K
    tma_load_2d_w(stg + 16384 + 8192, &maps.k, h * GDN_DK + 64, y, bar);
    tma_load_2d_w(xt, &maps.x, 0, (int)(xs * 2 * GDN_CHUNK + GDN_CHUNK), bar);  // X diag(b e^G)
    bulk_load_w(smem_u32(&st.tab[s2][0][0]), a.ftab + xs * F_TAB, F_ROWS * GDN_CHUNK * 4, bar);
    last_ld[s2] = m;
  };
  auto issue_do = [&](int64_t m) {  // the CTA's 64 columns of dO
    const int64_t c = chunk_of(m);
    const int s2 = (int)(m & 1);
    mbar_expect_tx_w(&st.bar_do[s2], 8192);
    tma_load_2d_w(sb + OFF_DO + s2 * 8192, &maps.dO, h * GDN_DV + col0, (int)(r0 + c * GDN_CHUNK), &st.bar_do[s2]);
    last_do[s2] = m;
  };

  // ---- producer: one chunk (order index pm) ------------------------------------------------
  auto produce = [&](int64_t pm) {
    const int ps = (int)(pm & 1);
    const uint32_t stg = sb + OFF_ST + ps * SZ_STAGE;
    const float(&tab)[F_ROWS][64] = st.tab[ps];
    const int n = chunk_rows(chunk_of(pm));
    if (loader && pm + 1 < nch) {  // the other buffers were last read by chunk pm - 1's products
      issue_qkx(pm + 1);
      issue_do(pm + 1);
    }
    wait_par(&st.bar_ld[ps], pm >> 1);  // Q, K, X and factors of this chunk have landed
    if (ptid == 0) st.EL[ps] = tab[F_EG][63];
    if (warp == 8) {  // P1: [Q; K] Q^T (rows 64..127 = K Q^T), issued warp-collectively
      fence_after_sync();
      mma_tiles_w(tmem + T_S + 64 * ps, stg, 16384, stg, 16384, 128, idesc_bf16(128, 64), false);
      mma_commit_w(&st.bar_p1);
    }
    __syncwarp();
    if (ptid < 64) st.seg[ps][ptid] = ptid < n ? scale * tab[F_EG][ptid] : 0.f;
    prod_sync();
    {  // diagonal-block gate table, spread over all producer threads (read after the next barrier)
      float *gdn = reinterpret_cast<float *>(sm + OFF_GD);
      for (int e = ptid; e < 1024; e += 256) {
        const int b = e >> 8, x = (e >> 4) & 15, y = e & 15;
        const float v = gexp<E2>(tab[F_G][16 * b + x] - tab[F_G][16 * b + y]);
        gdn[b * GD_B + x * 16 + y] = x >= y ? v : 0.f;
      }
    }
    // diag(scale base^G) dO (zero past the chunk end): the right operand of Qg^T dO
    wait_par(&st.bar_do[ps], pm >> 1);  // dO of this chunk
    {
      const int r = ptid >> 2;
      const uint8_t *src = sm + OFF_DO + ps * 8192;
      const float f = st.seg[ps][r];
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        const int c16 = 2 * (ptid & 3) + q2;
        float x[8];
        unpack8(*reinterpret_cast<const uint4 *>(src + chunk_off(r, c16)), x);
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= f;
        *reinterpret_cast<uint4 *>(sm + OFF_DOS + chunk_off(r, c16)) = pack8(x);
      }
    }
    prod_sync();  // the gate table is complete
    // gating of K Q^T (rows 64..127 of S): A_qk^T[s][t] = scale (k_s . q_t) base^(G_t - G_s),
    // s <= t < n; gate factors from tables as in the forward, formed while P1 may still run.
    float gf[32];
    if (q4 >= 2) {
      const int s = row - 64, bs = s >> 4;
      const float *gd = reinterpret_cast<const float *>(sm + OFF_GD) + bs * GD_B + (s & 15);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int t = 32 * hc + j, bt = t >> 4;
        const float off = tab[F_EA][t] * tab[F_EB1 + (bt > 0 ? bt - 1 : 0)][s], dg = gd[(t & 15) * 16];
        const float f = bt > bs ? off : (bt == bs ? dg : 0.f);
        gf[j] = t < n ? scale * f : 0.f;
      }
    }
    wait_par(&st.bar_p1, pm);
    if (q4 >= 2) {
      const int s = row - 64;
      float sv[32];
      tmem_ld16(tl + T_S + 64 * ps + 32 * hc, *reinterpret_cast<float(*)[16]>(sv));
      tmem_ld16(tl + T_S + 64 * ps + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(sv + 16));
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) sv[j] *= gf[j];
      uint8_t *dst = sm + OFF_AQT;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8)
        *reinterpret_cast<uint4 *>(dst + chunk_off(s, 4 * hc + q8)) = pack8(sv + 8 * q8);
    }
    fence_proxy_async();
    fence_before_sync();
    prod_sync();
    if (warp == 8) {  // the h-independent products
      fence_after_sync();
      const uint32_t xt = sb + (ps ? OFF_X1 : OFF_X0);
      // scale A_qk^T dO  (rows 64..127 of the operand are not used); dO read as an MN-major B
      mma_ops_w(tmem + T_I1 + 64 * ps, kmaj(sb + OFF_AQT, 8192), mnmaj(sb + OFF_DO + ps * 8192, 0), 64,
                idesc_bf16(128, 64, false, false, true), false);
      // scale Qg^T dO = Q^T (diag(scale base^G) dO): the stage's Q rows read as an MN-major A
      mma_ops_w(tmem + T_I2 + 64 * ps, mnmaj(stg, 16384), mnmaj(sb + OFF_DOS, 0), 64,
                idesc_bf16(128, 64, false, true, true), false);
      // w^T = K^T (X diag(beta base^G))^T: the stage's K rows read as an MN-major A
      mma_ops_w(tmem + T_WT, mnmaj(stg + 8192, 16384), kmaj(xt, 0), 64, idesc_bf16(128, 64, false, true, false), false);
      mma_commit_w(&st.bar_p3);
    }
    __syncwarp();
    fence_proxy_async();
    fence_before_sync();
  };

  // ---- chain ----------------------------------------------------------------------------
  // the operands of chunk pm's D1 and D2 that come from the producer's work, written by the
  // chain warps while the chain of chunk pm - 1 waits or idles (the producer bounds a round):
  // kgl rows (K rows scaled by base^(G_last - G); the lanes of tokens 64..127 of the stage) and
  // w^T rows (keys, from tensor memory once the producer's products are done)
  auto write_kgl = [&](int64_t pm) {  // warps of lanes 64..127 only
    const int ps = (int)(pm & 1);
    wait_par(&st.bar_ld[ps], pm >> 1);
    const int t = row - 64;
    const float egl = st.tab[ps][F_EGL][t];
    const uint8_t *krow = sm + OFF_ST + ps * SZ_STAGE + hc * 16384;
    uint8_t *dst = sm + OFF_KGL + hc * 8192;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4 *>(krow + chunk_off(row, c8)), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] *= egl;
      *reinterpret_cast<uint4 *>(dst + chunk_off(t, c8)) = pack8(f);
    }
  };
  auto write_wt = [&](int64_t pm) {
    wait_par(&st.bar_p3, pm);
    uint8_t *dst = sm + OFF_WT;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      float sv[16];
      tmem_ld16(tl + T_WT + 32 * hc + 16 * part, sv);
      tmem_ld_wait();
      *reinterpret_cast<uint4 *>(dst + chunk_off(row, 4 * hc + 2 * part)) = pack8(sv);
      *reinterpret_cast<uint4 *>(dst + chunk_off(row, 4 * hc + 2 * part + 1)) = pack8(sv + 8);
    }
  };
  float dh[32];
  if (!producer) {
    const float *src = a.dht ? a.dht + state_off + (int64_t)row * GDN_DV + col0 + 32 * hc : nullptr;
#pragma unroll
    for (int j = 0; j < 32; ++j) dh[j] = src ? src[j] : 0.f;
  }
  auto write_dht = [&]() {  // dh (MN-major B operand of D1): key `row`, columns 32*hc .. +32
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8)
      *reinterpret_cast<uint4 *>(sm + OFF_DHT + chunk_off(row, 4 * hc + q8)) = pack8(dh + 8 * q8);
  };
  auto chain = [&](int64_t m) {
    const int cs = (int)(m & 1);
    const int64_t c = chunk_of(m);
    const int64_t c0 = r0 + c * GDN_CHUNK;
    const int n = chunk_rows(c);
    uint8_t *dvt = a.dv_tiles ? reinterpret_cast<uint8_t *>(a.dv_tiles + state_slot(c) * DV_TILE) + (col0 >> 6) * 8192
                              : nullptr;
    if (a.dh_tiles) {  // gradient of this chunk's exit state: D1's dh operand is that bf16 tile
      if (warp == 0)
        bulk_store_w(reinterpret_cast<uint8_t *>(a.dh_tiles + state_slot(c) * STATE_TILE) + (col0 >> 6) * 16384,
                     sb + OFF_DHT, 16384);
    } else {  // fp32
      float4 *dst = reinterpret_cast<float4 *>(a.dh_chunks + state_slot(c) * GDN_DK * GDN_DV +
                                               (int64_t)row * GDN_DV + col0 + 32 * hc);
#pragma unroll
      for (int g4 = 0; g4 < 8; ++g4) dst[g4] = make_float4(dh[4 * g4], dh[4 * g4 + 1], dh[4 * g4 + 2], dh[4 * g4 + 3]);
    }
    if (warp == 0) {  // D1: dv_new = kgl dh + scale A_qk^T dO
      fence_after_sync();
      mma_ops_w(tmem + T_I1 + 64 * cs, kmaj(sb + OFF_KGL, 8192), mnmaj(sb + OFF_DHT, 0), 128,
                idesc_bf16(128, 64, false, false, true), true);
      mma_commit_w(&st.bar_d1);
    }
    __syncwarp();
    wait_par(&st.bar_d1, m);
    if (q4 < 2) {  // dv_new rows: fp32 to the workspace, bf16 into D2's operand
      const bool valid = row < n;
      float4 *gdst = reinterpret_cast<float4 *>(a.dvnew + ((c0 + (valid ? row : 0)) * H + h) * GDN_DV + col0 + 32 * hc);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float dv[16];
        tmem_ld16(tl + T_I1 + 64 * cs + 32 * hc + 16 * part, dv);
        tmem_ld_wait();
        if (!dvt && valid) {  // (the bf16 tile is D2's operand, stored below as it stands)
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4)
            gdst[4 * part + g4] = make_float4(dv[4 * g4], dv[4 * g4 + 1], dv[4 * g4 + 2], dv[4 * g4 + 3]);
        }
        *reinterpret_cast<uint4 *>(sm + OFF_DVT + chunk_off(row, 4 * hc + 2 * part)) = pack8(dv);
        *reinterpret_cast<uint4 *>(sm + OFF_DVT + chunk_off(row, 4 * hc + 2 * part + 1)) = pack8(dv + 8);
      }
    } else if (m + 1 < nch) {  // D1 has read kgl: the next chunk's, meanwhile
      write_kgl(m + 1);
    }
    fence_proxy_async();
    fence_before_sync();
    if (warp == 0 && a.dh_tiles) bulk_store_wait_read_w();  // the dh tile is rewritten below
    chain_sync();
    if (warp == 0) {  // D2: dh increment = scale Qg^T dO - w^T dv_new
      fence_after_sync();
      if (dvt)  // dv_new as a bf16 tile (rows past the end hold values the local kernel never uses)
        bulk_store_w(dvt, sb + OFF_DVT, 8192);
      mma_ops_w(tmem + T_I2 + 64 * cs, kmaj(sb + OFF_WT, 16384), mnmaj(sb + OFF_DVT, 0), 64,
                idesc_bf16(128, 64, true, false, true), true);
      mma_commit_w(&st.bar_d2);
    }
    __syncwarp();
    wait_par(&st.bar_d2, m);
    {
      const float el = st.EL[cs];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float inc[16];
        tmem_ld16(tl + T_I2 + 64 * cs + 32 * hc + 16 * part, inc);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) dh[16 * part + j] = fmaf(el, dh[16 * part + j], inc[j]);
      }
      write_dht();
    }
    if (m + 1 < nch) write_wt(m + 1);  // D2 has read w^T: the next chunk's
    if (warp == 0 && dvt) bulk_store_wait_read_w();  // the dv_new tile is rewritten next round
    fence_proxy_async();
    fence_before_sync();
  };

  // ---- prologue and rounds ------------------------------------------------------------------
  if (loader && nch > 0) {
    issue_qkx(0);
    issue_do(0);
  }
  if (!producer) {
    write_dht();
    fence_proxy_async();
  }
  __syncthreads();
  // round m: the chain runs order index m while the producer prepares m+1
  for (int64_t m = -1; m < nch; ++m) {
    if (producer) {
      if (m + 1 < nch) produce(m + 1);
    } else if (m >= 0) {
      chain(m);
    } else if (nch > 0) {  // chunk 0's kgl and w^T
      if (q4 >= 2) write_kgl(0);
      write_wt(0);
      fence_proxy_async();
      fence_before_sync();
    }
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
  }

  if (bad) {
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    // each issuing warp's elected lane: arrives once every MMA it issued has finished
    if (warp == 0) mma_commit_w(&st.bar_x0);
    if (warp == 8) mma_commit_w(&st.bar_x1);
    if (warp == 0) mbar_wait(&st.bar_x0, 0, WAIT_LIMIT);
    if (warp == 8) mbar_wait(&st.bar_x1, 0, WAIT_LIMIT);
    if (loader) {  // copies still in flight land before the CTA leaves
      for (int s2 = 0; s2 < 2; ++s2)
        if (last_ld[s2] >= 0) mbar_wait(&st.bar_ld[s2], (uint32_t)((last_ld[s2] >> 1) & 1), WAIT_LIMIT);
      for (int s2 = 0; s2 < 2; ++s2)
        if (last_do[s2] >= 0) mbar_wait(&st.bar_do[s2], (uint32_t)((last_do[s2] >> 1) & 1), WAIT_LIMIT);
    }
  } else if (!producer && a.dh0) {
    float4 *dst = reinterpret_cast<float4 *>(a.dh0 + state_off + (int64_t)row * GDN_DV + col0 + 32 * hc);
#pragma unroll
    for (int g4 = 0; g4 < 8; ++g4) dst[g4] = make_float4(dh[4 * g4], dh[4 * g4 + 1], dh[4 * g4 + 2], dh[4 * g4 + 3]);
  }
  if (warp == 0) bulk_store_wait_w();  // the tiles' bulk stores have completed
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_tc_dhu(const BwdArgs &a, int runs, cudaStream_t st) {
  const uint64_t rows = a.cu ? (uint64_t)a.T : (uint64_t)a.B * a.T;
  const uint64_t slots = a.cu ? (uint64_t)a.num_chunks : (uint64_t)a.B * ((a.T + GDN_CHUNK - 1) / GDN_CHUNK);
  const uint64_t pitch = (uint64_t)a.H * GDN_DK * 2;
  BwdMaps maps;
  cudaError_t e = make_tmap_bf16(&maps.q, a.q, (uint64_t)a.H * GDN_DK, rows, pitch);
  if (e == cudaSuccess) e = make_tmap_bf16(&maps.k, a.k, (uint64_t)a.H * GDN_DK, rows, pitch);
  if (e == cudaSuccess) e = make_tmap_bf16(&maps.dO, a.dO, (uint64_t)a.H * GDN_DV, rows, (uint64_t)a.H * GDN_DV * 2);
  if (e == cudaSuccess) e = make_tmap_bf16(&maps.x, a.xw, GDN_CHUNK, slots * a.H * 2 * GDN_CHUNK, GDN_CHUNK * 2);
  if (e != cudaSuccess) return e;
  auto kern = a.use_exp2 ? tc_dhu_kernel<true> : tc_dhu_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<dim3(GDN_DV / TBV, a.H, runs), NTH, SMEM_BYTES, st>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace gdn
