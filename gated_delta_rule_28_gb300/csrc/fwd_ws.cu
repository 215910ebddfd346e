// Tensor-core (tcgen05) chunk forward for bf16 inputs, scalar gate (sm_103a),
// state recurrence overlapped with the preparation of the next chunk.
//
// One CTA (512 threads) owns one independent run (batch row, packed document
// or segment) of one head and 64 of the 128 state columns; the UT transform
// kernel supplies X = (I + L)^-1 of every chunk already scaled by its columns,
// as the pair [X diag(b); X diag(b e^G)] in bf16. Per chunk (GDN Ascend C adapter
// forward, chunk_fwd_h and the output step):
//
//   producer warps 8..15, chunk c+1 (no dependence on the state):
//     P1   S = Q K^T                           -> A_qk = lower-incl(Q K^T (.) Gamma)
//     P3   [X diag(b); X diag(b e^G)] [K | V]  -> w = X diag(b e^G) K,  u = X diag(b) V
//          w rows of the operand [w; Q] of P4 (Q is loaded into it)
//   chain warps 0..7, chunk c (the state h lives in their registers, fp32):
//     P4   [w; Q] h                            -> v_new = u - w h,  Q h
//     P5   K^T (e^(G_last - G) v_new)          -> h <- e^(G_last) h + P5
//     PO   A_qk v_new                          -> o = scale (e^G (Q h) + A_qk v_new)
//
// The two warp groups meet once per chunk (a CTA barrier); every buffer one group
// writes while the other reads is double-buffered by chunk parity (K, read by P5 one
// round later, by three).
// Loads are TMA copies (tensor tiles with the 128-byte swizzle, and bulk copies
// of the chunk's gate factors) completing on mbarriers. No operand is
// transposed: the token-major tiles (K, V, v_new, h by key) enter the MMAs as
// MN-major operands, and every row the threads write is a run of 16-byte stores.
// Every mbarrier wait is bounded; a wait that runs out sets the device flag and
// the CTA drains its MMAs, frees its tensor memory and leaves.
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tc;
using namespace tile;

constexpr int TBV = 64;   // state columns per CTA
constexpr int NTH = 512;  // threads per CTA: 256 chain + 256 producer
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_S = 0;     // 64: P1 (rows 0..63 = Q K^T)
constexpr uint32_t T_PO = 64;   // 64: PO (rows 64..127 = A_qk v_new)
constexpr uint32_t T_WW = 128;  // 128: P3w rows 64..127 = w
constexpr uint32_t T_U = 256;   // 2 x 64: P3u rows 0..63 = u, per chunk parity
constexpr uint32_t T_D4 = 384;  // 64: P4 rows 0..63 = w h, rows 64..127 = Q h
constexpr uint32_t T_P5 = 448;  // 64: P5

// shared memory map (bytes from a 1024-aligned base); tiles of 128-byte rows, swizzled.
// Token-major tiles (Q, K, V as loaded, v_new, h) serve as K- or MN-major operands as they
// are. P1 and PO use 128-row A operands whose rows 64..127 (P1) or 0..63 (PO) are not
// needed: they read whatever follows (precedes) the tile, and land in unread rows of D.
constexpr int OFF_WQ = 0;                     // [w; Q] per chunk parity: 2 K-blocks x 128 rows
constexpr int OFF_K = OFF_WQ + 2 * 32768;     // K, three chunks in flight: 2 K-blocks x 64 rows
constexpr int OFF_XX = OFF_K + 3 * 16384;     // [X diag(b); X diag(b e^G)] per parity: 128 rows
constexpr int OFF_V = OFF_XX + 2 * 16384;     // V slice per parity: 64 rows
constexpr int OFF_HT = OFF_V + 2 * 8192;      // h: 128 key rows (MN-major B of P4)
constexpr int OFF_VN = OFF_HT + 16384;        // v_new: 64 token rows (MN-major B of PO)
constexpr int OFF_VNL = OFF_VN + 8192;        // e^(Gl - G) v_new (MN-major B of P5)
constexpr int OFF_AQ = OFF_VNL + 8192;        // A_qk per parity: 64 rows (PO's rows 0..63: the 8 KB before)
constexpr int OFF_SMALL = OFF_AQ + 2 * 8192;
constexpr int SMALL_BYTES = 6144;
constexpr int SMEM_BYTES = OFF_SMALL + SMALL_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
// The MN-major K operand (two 64-key groups 8 KB apart, 64 token rows) stays below the small
// state under either assignment of its descriptor's two stride fields: groups 8 KB apart and
// K rows in 1 KB atoms, or the reverse. The other MN-major operands have one group.
static_assert(OFF_K + 2 * 16384 + 8192 + 8 * 1024 <= OFF_XX &&
                  OFF_K + 2 * 16384 + 1024 + 7 * 8192 + 1024 <= OFF_SMALL,
              "MN-major K operand extent");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct WsState {
  alignas(16) float tab[2][F_ROWS][64];  // refilled with chunk c+2 while the chain runs chunk c
  float EGL[2][64];                 // base^(G_last - G) per chunk parity, for the chain
  float EG[2][64];                  // base^G per chunk parity, for the chain
  float EL[2];                      // base^(G_last) per chunk parity, for the chain
  uint64_t bar_p1, bar_p3, bar_p4, bar_p5, bar_po, bar_d0, bar_d1, bar_d2;
  uint64_t bar_ld[2];  // TMA loads per chunk parity: K, the X pair, V, gate factors
  uint64_t bar_q[2];   // TMA loads per chunk parity: Q (issued once P4 has read the buffer)
  uint32_t tmem;
};
static_assert(sizeof(WsState) <= SMALL_BYTES, "small state");

__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// TMA maps: q, k, v over [rows, H*128]; the X pair over [slots*H*128, 64]; 64 x 64 boxes
struct FwdMaps {
  TmaMap q, k, v, x;
};

template <bool E2>
__global__ void __launch_bounds__(NTH, 1) tc_fwd_ws_kernel(SimtFwdArgs a, const __grid_constant__ FwdMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base by pointer arithmetic on the shared array, so that the compiler keeps
  // the shared address space (shared-memory instructions, not generic ones)
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  WsState &st = *reinterpret_cast<WsState *>(sm + OFF_SMALL);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool producer = warp >= 8;
  const int q4 = warp & 3;         // tensor-memory lane quarter of this warp
  const int hc = (warp >> 2) & 1;  // column half (32 of 64) inside the warp group
  const int row = q4 * 32 + lane;  // tensor-memory lane = matrix row
  const int H = a.H, h = blockIdx.y, z = blockIdx.z;
  const int col0 = blockIdx.x * TBV;
  const float scale = a.scale;
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.o);

  // ---- the run -------------------------------------------------------------------
  // xbase: global chunk index of the run's first chunk (X workspace slot / H);
  // h_chunks slots: [B, H, NT] for BSND, [chunks, H] for packed documents
  int64_t r0, r1, chunk_base = 0, xbase;
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
    xbase = chunk_base;
  } else if (a.nseg > 0) {
    b = z / a.nseg;
    s = z % a.nseg;
    r0 = (int64_t)b * a.T + (int64_t)s * a.seg_len;
    r1 = min(r0 + a.seg_len, (int64_t)b * a.T + a.T);
    chunk_base = (int64_t)s * a.seg_len / GDN_CHUNK;
    state_idx = b;
    xbase = (int64_t)b * NT + chunk_base;
  } else {
    b = z;
    r0 = (int64_t)b * a.T;
    r1 = r0 + a.T;
    state_idx = b;
    xbase = (int64_t)b * NT;
  }
  const int64_t nch = (r1 - r0 + GDN_CHUNK - 1) / GDN_CHUNK;
  auto chunk_rows = [&](int64_t c) { return (int)min((int64_t)GDN_CHUNK, r1 - (r0 + c * GDN_CHUNK)); };

  // ---- tensor memory, barriers -----------------------------------------------------
  if (warp == 0) {
    tmem_alloc(&st.tmem, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&st.bar_p1, 1);
    mbar_init(&st.bar_p3, 1);
    mbar_init(&st.bar_p4, 1);
    mbar_init(&st.bar_p5, 1);
    mbar_init(&st.bar_po, 1);
    mbar_init(&st.bar_d0, 1);
    mbar_init(&st.bar_d1, 1);
    mbar_init(&st.bar_d2, 1);
    mbar_init(&st.bar_q[0], 1);
    mbar_init(&st.bar_q[1], 1);
    mbar_init(&st.bar_ld[0], 1);
    mbar_init(&st.bar_ld[1], 1);
    mbar_fence_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // the X pair and the gate tables come from the kernel launched before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem = st.tmem;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);  // this warp's lane quarter
  bool bad = false;
  auto wait_par = [&](uint64_t *bar, int64_t phase) {
    if (!mbar_wait(bar, (uint32_t)(phase & 1), WAIT_LIMIT)) bad = true;
    fence_after_sync();
  };
  auto wq_at = [&](int64_t c) { return sb + OFF_WQ + (uint32_t)(c & 1) * 32768u; };
  auto k_at = [&](int64_t c) { return sb + OFF_K + (uint32_t)(c % 3) * 16384u; };
  auto xx_at = [&](int64_t c) { return sb + OFF_XX + (uint32_t)(c & 1) * 16384u; };
  auto v_at = [&](int64_t c) { return sb + OFF_V + (uint32_t)(c & 1) * 8192u; };

  // ---- producer: loads (TMA, issued by warp 9) ------------------------------------------
  // Every TMA copy and tcgen05 MMA is issued warp-collectively (one elected lane of a
  // warp-uniform call, tc.cuh): warp 9 the loads and P1, warp 10 P3, warp 0 the chain's
  // MMAs and its Q loads.
  // Rows past the run end are loaded as they are (the next run's tokens, or zeros past
  // the tensor): they only meet beta = 0 (zero columns of both X's), a causal mask, or rows
  // of o that are not stored.
  const int ptid = tid - 256;
  const bool loader = warp == 9;
  const bool issuer = warp == 10;  // producer MMAs: P3 by warp 10, P1 by warp 9
  int64_t last_ld[2] = {-1, -1};   // loader: newest chunk per barrier
  auto issue_loads = [&](int64_t c) {  // K, the X pair, V and the gate factors of chunk c
    const int s2 = (int)(c & 1);
    const int y = (int)(r0 + c * GDN_CHUNK);
    const int64_t xs = (xbase + c) * H + h;
    uint64_t *bar = &st.bar_ld[s2];
    mbar_expect_tx_w(bar, 5 * 8192 + F_ROWS * GDN_CHUNK * 4);
    tma_load_2d_w(k_at(c), &maps.k, h * GDN_DK, y, bar);
    tma_load_2d_w(k_at(c) + 8192, &maps.k, h * GDN_DK + 64, y, bar);
    tma_load_2d_w(xx_at(c), &maps.x, 0, (int)(xs * 2 * GDN_CHUNK), bar);
    tma_load_2d_w(xx_at(c) + 8192, &maps.x, 0, (int)(xs * 2 * GDN_CHUNK + GDN_CHUNK), bar);
    tma_load_2d_w(v_at(c), &maps.v, h * GDN_DV + col0, y, bar);
    bulk_load_w(smem_u32(&st.tab[s2][0][0]), a.ftab + xs * F_TAB, F_ROWS * GDN_CHUNK * 4, bar);
    last_ld[s2] = c;
  };
  // Q of chunk c into rows 64..127 of [w; Q] of parity c&1, by the chain's warp 0 (the
  // buffer held chunk c-2, whose P4 it waits for)
  int64_t last_q[2] = {-1, -1};
  auto issue_q = [&](int64_t c) {
    const int s2 = (int)(c & 1);
    const int y = (int)(r0 + c * GDN_CHUNK);
    mbar_expect_tx_w(&st.bar_q[s2], 2 * 8192);
    tma_load_2d_w(wq_at(c) + 8192, &maps.q, h * GDN_DK, y, &st.bar_q[s2]);
    tma_load_2d_w(wq_at(c) + 16384 + 8192, &maps.q, h * GDN_DK + 64, y, &st.bar_q[s2]);
    last_q[s2] = c;
  };

  // ---- producer: one chunk -------------------------------------------------------------
  // warps 8, 9, 12, 13 (lane quarters 0, 1): gating of Q K^T; warps 10, 11, 14, 15
  // (quarters 2, 3): the w rows of the P4 operand.
  auto produce = [&](int64_t pc) {
    const int ps = (int)(pc & 1);
    const float(&tab)[F_ROWS][64] = st.tab[ps];
    // buffers of chunk pc+1 (they held chunk pc-1, and K chunk pc-2: finished, P4 included)
    if (loader && pc + 1 < nch) issue_loads(pc + 1);
    wait_par(&st.bar_ld[ps], pc >> 1);  // K, X's, V and factors of chunk pc have landed
    if (issuer) {
      // P3: [X diag(b); X diag(b e^G)] [K | V] -> rows 64..127 of the K product = w,
      // rows 0..63 of the V product = u (K and V token-major, read as MN-major B)
      mma_ops_w(tmem + T_WW, kmaj(xx_at(pc), 0), mnmaj(k_at(pc), 8192), 64, idesc_bf16(128, 128, false, false, true),
              false);
      mma_ops_w(tmem + T_U + 64 * ps, kmaj(xx_at(pc), 0), mnmaj(v_at(pc), 0), 64,
              idesc_bf16(128, 64, false, false, true), false);
      mma_commit_w(&st.bar_p3);
    }
    __syncwarp();  // the issuing warp reconverges before any of its lanes polls a barrier
    if (q4 < 2) {
      const int t = row;
      if (ptid == 0) st.EL[ps] = tab[F_EG][63];
      if (hc == 0) {
        st.EGL[ps][t] = tab[F_EGL][t];
        st.EG[ps][t] = tab[F_EG][t];
      }
      if (warp == 9) {
        // P1: S = Q K^T, once Q has landed (A rows 64..127: the next 64 rows of shared
        // memory, unread output rows)
        wait_par(&st.bar_q[ps], pc >> 1);
        mma_ops_w(tmem + T_S, kmaj(wq_at(pc) + 8192, 16384), kmaj(k_at(pc), 8192), 128, idesc_bf16(128, 64), false);
        mma_commit_w(&st.bar_p1);
      }
      // gating of Q K^T (rows 0..63 of S) -> A_qk, lower triangle including the diagonal.
      // Gate factors of this thread's 32 key tokens s, formed while P1 runs: between
      // 16-token blocks from the tables, EA[t] EB_{b(t)}[s] (no exponential); inside the
      // diagonal block base^(G_t - G_s), 16 exponentials in the two warps whose key tokens
      // hold their rows' diagonal blocks (8: rows 0..31, keys 0..31; 13: rows 32..63, keys
      // 32..63).
      float gf[32];
      {
        const int bt = t >> 4;
        const float ea = tab[F_EA][t];
        const float *eb = tab[F_EB1 + (bt > 0 ? bt - 1 : 0)];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int sj = 32 * hc + j;
          gf[j] = (sj >> 4) < bt ? ea * eb[sj] : 0.f;
        }
        if (q4 == hc) {
          const float gt = tab[F_G][t];
          const int hi = bt & 1, r = t & 15;  // the diagonal block is keys 32 hc + 16 hi + 0..15
          const float *gs = &tab[F_G][32 * hc + 16 * hi];
          float e[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) e[jj] = jj <= r ? gexp<E2>(gt - gs[jj]) : 0.f;
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            if (hi == 0) gf[jj] = e[jj];
            else gf[16 + jj] = e[jj];
          }
        }
      }
      wait_par(&st.bar_p1, pc);
      {
        float sv[32];
        tmem_ld16(tl + T_S + 32 * hc, *reinterpret_cast<float(*)[16]>(sv));
        tmem_ld16(tl + T_S + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(sv + 16));
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) sv[j] *= gf[j];
        uint8_t *dst = sm + OFF_AQ + ps * 8192;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8)
          *reinterpret_cast<uint4 *>(dst + chunk_off(t, 4 * hc + q8)) = pack8(sv + 8 * q8);
      }
    } else {
      // rows 0..63 of the P4 operand [w; Q] of chunk pc (keys 64*hc .. +64), once P3 is done
      uint8_t *wq = sm + OFF_WQ + ps * 32768 + hc * 16384;
      wait_par(&st.bar_p3, pc);
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        float sv[16];
        tmem_ld16(tl + T_WW + 64 * hc + 16 * part, sv);
        tmem_ld_wait();
        *reinterpret_cast<uint4 *>(wq + chunk_off(row - 64, 2 * part)) = pack8(sv);
        *reinterpret_cast<uint4 *>(wq + chunk_off(row - 64, 2 * part + 1)) = pack8(sv + 8);
      }
    }
    fence_proxy_async();
    fence_before_sync();
  };

  // ---- chain: state and one chunk ----------------------------------------------------------
  float hreg[32];
  if (!producer) {
    const float *src = nullptr;
    if (a.h0) {
      const int64_t slot = a.nseg > 0 ? (((int64_t)b * H + h) * a.nseg + s) : ((int64_t)state_idx * H + h);
      src = a.h0 + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV + col0 + 32 * hc;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) hreg[j] = src ? src[j] : 0.f;
  }
  // h in bf16 (MN-major B operand of P4): this thread's key `row`, columns 32*hc .. +32
  auto write_ht = [&]() {
    uint8_t *hrow = sm + OFF_HT;
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8)
      *reinterpret_cast<uint4 *>(hrow + chunk_off(row, 4 * hc + q8)) = pack8(hreg + 8 * q8);
  };
  auto chain = [&](int64_t c) {
    const int par = (int)(c & 1);
    const int64_t c0 = r0 + c * GDN_CHUNK;
    const int n = chunk_rows(c);
    if (a.h_chunks || a.h_tiles) {  // entry state of chunk c
      const int64_t slot = a.cu ? (chunk_base + c) * H + h : ((int64_t)b * H + h) * NT + chunk_base + c;
      if (a.h_chunks) {
        float4 *dst = reinterpret_cast<float4 *>(a.h_chunks + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV +
                                                 col0 + 32 * hc);
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4)
          dst[g4] = make_float4(hreg[g4 * 4], hreg[g4 * 4 + 1], hreg[g4 * 4 + 2], hreg[g4 * 4 + 3]);
      }
      if (a.h_tiles) {  // key `row`, values col0 + 32 hc .. +31: four 16-byte chunks of the tile
        uint8_t *tb = reinterpret_cast<uint8_t *>(a.h_tiles + slot * STATE_TILE) + (col0 >> 6) * 16384;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8)
          *reinterpret_cast<uint4 *>(tb + chunk_off(row, 4 * hc + q8)) = pack8(hreg + 8 * q8);
      }
    }
    if (warp == 0) {  // P4: [w; Q] h
      fence_after_sync();
      mma_ops_w(tmem + T_D4, kmaj(wq_at(c), 16384), mnmaj(sb + OFF_HT, 0), 128,
              idesc_bf16(128, 64, false, false, true), false);
      mma_commit_w(&st.bar_p4);
    }
    __syncwarp();  // the issuing warp reconverges before any of its lanes polls a barrier
    wait_par(&st.bar_p4, c);
    if (warp == 0 && c + 2 < nch) issue_q(c + 2);  // P4 has read Q of chunk c
    if (q4 < 2) {  // v_new = u - w h (token row), and e^(Gl - G) v_new
      const float egl = st.EGL[par][row];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float wh[16], u[16];
        tmem_ld16(tl + T_D4 + 32 * hc + 16 * part, wh);
        tmem_ld16(tl + T_U + 64 * par + 32 * hc + 16 * part, u);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) u[j] -= wh[j];
        *reinterpret_cast<uint4 *>(sm + OFF_VN + chunk_off(row, 4 * hc + 2 * part)) = pack8(u);
        *reinterpret_cast<uint4 *>(sm + OFF_VN + chunk_off(row, 4 * hc + 2 * part + 1)) = pack8(u + 8);
#pragma unroll
        for (int j = 0; j < 16; ++j) u[j] *= egl;
        *reinterpret_cast<uint4 *>(sm + OFF_VNL + chunk_off(row, 4 * hc + 2 * part)) = pack8(u);
        *reinterpret_cast<uint4 *>(sm + OFF_VNL + chunk_off(row, 4 * hc + 2 * part + 1)) = pack8(u + 8);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    chain_sync();
    if (warp == 0) {  // the intra-chunk output term (the output is the longer path), then
                      // P5: K^T (e^(Gl-G) v_new), K read as MN-major A
      fence_after_sync();
      mma_ops_w(tmem + T_PO, kmaj(sb + OFF_AQ + par * 8192 - 8192, 0), mnmaj(sb + OFF_VN, 0), 64,
                idesc_bf16(128, 64, false, false, true), false);
      mma_commit_w(&st.bar_po);
      mma_ops_w(tmem + T_P5, mnmaj(k_at(c), 8192), mnmaj(sb + OFF_VNL, 0), 64, idesc_bf16(128, 64, false, true, true),
                false);
      mma_commit_w(&st.bar_p5);
    }
    __syncwarp();  // the issuing warp reconverges before any of its lanes polls a barrier
    wait_par(&st.bar_p5, c);
    {
      const float el = st.EL[par];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float p5[16];
        tmem_ld16(tl + T_P5 + 32 * hc + 16 * part, p5);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) hreg[16 * part + j] = fmaf(el, hreg[16 * part + j], p5[j]);
      }
      write_ht();
      fence_proxy_async();  // h for the next P4 (the output below goes to global memory)
      if (q4 >= 2) {  // o = scale (base^G Q h + A_qk v_new); the whole warp loads (collective)
        wait_par(&st.bar_po, c);
        const float eg = st.EG[par][row - 64];
        const bool st_row = o && row - 64 < n;
        uint4 *dst = reinterpret_cast<uint4 *>(o + ((c0 + (st_row ? row - 64 : 0)) * H + h) * GDN_DV + col0 + 32 * hc);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float ov[16], av[16];
          tmem_ld16(tl + T_D4 + 32 * hc + 16 * part, ov);
          tmem_ld16(tl + T_PO + 32 * hc + 16 * part, av);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) ov[j] = scale * fmaf(eg, ov[j], av[j]);
          if (st_row) {
            dst[2 * part] = pack8(ov);
            dst[2 * part + 1] = pack8(ov + 8);
          }
        }
      }
    }
    fence_before_sync();
  };

  // ---- prologue --------------------------------------------------------------------------
  if (loader && nch > 0) issue_loads(0);
  if (warp == 0) {
    if (nch > 0) issue_q(0);
    if (nch > 1) issue_q(1);
  }
  if (!producer) {
    write_ht();
    fence_proxy_async();
  }
  __syncthreads();

  // round c: the chain runs chunk c while the producer prepares chunk c+1
  for (int64_t c = -1; c < nch; ++c) {
    if (producer) {
      if (c + 1 < nch) produce(c + 1);
    } else if (c >= 0) {
      chain(c);
    }
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
  }

  if (bad) {
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    // each issuing warp's elected lane: arrives once every MMA it issued has finished
    if (warp == 0) mma_commit_w(&st.bar_d0);
    if (issuer) mma_commit_w(&st.bar_d1);
    if (warp == 9) mma_commit_w(&st.bar_d2);
    if (warp == 0) mbar_wait(&st.bar_d0, 0, WAIT_LIMIT);
    if (issuer) mbar_wait(&st.bar_d1, 0, WAIT_LIMIT);
    if (warp == 9) mbar_wait(&st.bar_d2, 0, WAIT_LIMIT);
    if (warp == 0)  // Q copies still in flight land before the CTA leaves
      for (int s2 = 0; s2 < 2; ++s2)
        if (last_q[s2] >= 0) mbar_wait(&st.bar_q[s2], (uint32_t)((last_q[s2] >> 1) & 1), WAIT_LIMIT);
    if (loader) {  // copies still in flight land before the CTA leaves
      for (int s2 = 0; s2 < 2; ++s2)
        if (last_ld[s2] >= 0) mbar_wait(&st.bar_ld[s2], (uint32_t)((last_ld[s2] >> 1) & 1), WAIT_LIMIT);
    }
  } else if (!producer && a.ht && (a.nseg == 0 || s == a.nseg - 1)) {
    float4 *dst = reinterpret_cast<float4 *>(a.ht + ((int64_t)state_idx * H + h) * GDN_DK * GDN_DV +
                                             (int64_t)row * GDN_DV + col0 + 32 * hc);
#pragma unroll
    for (int g4 = 0; g4 < 8; ++g4)
      dst[g4] = make_float4(hreg[g4 * 4], hreg[g4 * 4 + 1], hreg[g4 * 4 + 2], hreg[g4 * 4 + 3]);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int tc_fwd_ws_bv() { return TBV; }

cudaError_t launch_tc_fwd_ws(const SimtFwdArgs &a, dim3 grid, cudaStream_t st) {
  const uint64_t rows = a.cu ? (uint64_t)a.T : (uint64_t)a.B * a.T;
  const uint64_t slots = a.cu ? (uint64_t)a.num_chunks : (uint64_t)a.B * ((a.T + GDN_CHUNK - 1) / GDN_CHUNK);
  const uint64_t pitch = (uint64_t)a.H * GDN_DK * 2;
  FwdMaps maps;
  memset(&maps, 0, sizeof(maps));
  cudaError_t e = cudaSuccess;
  if (rows > 0) {  // an empty sequence loads nothing (the kernel only writes ht = h0)
    e = make_tmap_bf16(&maps.q, a.q, (uint64_t)a.H * GDN_DK, rows, pitch);
    if (e == cudaSuccess) e = make_tmap_bf16(&maps.k, a.k, (uint64_t)a.H * GDN_DK, rows, pitch);
    if (e == cudaSuccess) e = make_tmap_bf16(&maps.v, a.v, (uint64_t)a.H * GDN_DV, rows, (uint64_t)a.H * GDN_DV * 2);
    if (e == cudaSuccess) e = make_tmap_bf16(&maps.x, a.xw, GDN_CHUNK, slots * a.H * 2 * GDN_CHUNK, GDN_CHUNK * 2);
  }
  if (e != cudaSuccess) return e;
  auto kern = a.use_exp2 ? tc_fwd_ws_kernel<true> : tc_fwd_ws_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the CTAs may start (tensor memory, barriers, h0) while
  // the UT transform kernel before them in the stream finishes; they wait for it before
  // their first load
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NTH);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, maps);
}

}  // namespace gdn
