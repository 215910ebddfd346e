// Tensor-core (tcgen05) chunk forward for bf16 inputs, scalar gate (sm_103a),
// state recurrence overlapped with the preparation of the next chunk.
//
// One CTA (512 threads) owns one independent run (batch row, packed document
// or segment) of one head and 64 of the 128 state columns; X = (I + L)^-1 of
// every chunk comes precomputed in bf16 (UT transform kernel). Per chunk
// (north star; GDN Ascend C adapter forward, chunk_fwd_h and the output step):
//
//   producer warps 8..15, chunk c+1 (no dependence on the state):
//     P1   S = [Q; K] K^T                      -> A_qk = lower-incl(Q K^T (.) Gamma)
//     P3b  X [b e^G K | b V]                   -> w = X diag(b e^G) K,  u = X diag(b) V
//          operand [w; e^G Q] for P4
//   chain warps 0..7, chunk c (the state h lives in their registers, fp32):
//     P4   [w; e^G Q] h                        -> v_new = u - w h,  q' h
//     P5   (e^(G_last - G) K)^T v_new          -> h <- e^(G_last) h + P5
//     PO   A_qk v_new added onto q' h          -> o = scale (q' h + A_qk v_new)
//
// The two warp groups meet once per chunk (a CTA barrier); inside a chunk the
// producer waits for P4 of the chain before it overwrites the P4 operand.
// Loads are TMA copies (tensor tiles with the 128-byte swizzle, and one bulk copy
// of the chunk's gate factors) completing on mbarriers.
// Operands are K-major tiles with the 128-byte swizzle; the state-side
// transposes (v_new^T, h^T) are written column-wise straight from the tensor
// memory loads, the key and value transposes of the producer with
// ldmatrix.trans / stmatrix. Every mbarrier wait is bounded; a wait that runs
// out sets the device flag and the CTA drains its MMAs, frees its tensor
// memory and leaves.
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
constexpr uint32_t T_S = 0;     // 2 x 64: P1 per chunk parity (rows 0..63 = Q K^T)
constexpr uint32_t T_WW = 128;  // 128: P3b rows 0..63 = w
constexpr uint32_t T_U = 256;   // 2 x 64: P3b rows 0..63 = u, per chunk parity
constexpr uint32_t T_D4 = 384;  // 64: P4 rows 0..63 = w h, rows 64..127 = q' h (+ A_qk v_new)
constexpr uint32_t T_P5 = 448;  // 64: P5

// shared memory map (bytes from a 1024-aligned base); every tile K-major, 128 B rows.
// The P3b operand is a 128-row tile whose rows 64..127 are not used: each X tile
// is placed in front of a buffer that no copy writes while P3b runs (B3, KL),
// and the A_qk tiles behind v_new^T for the same reason.
constexpr int SZ_STAGE = 32768;                // [Q; K]: 2 K-blocks x 128 rows
constexpr int OFF_ST = 0;                      // 2 stages
constexpr int OFF_V = OFF_ST + 2 * SZ_STAGE;   // V slice, 64 rows (one buffer)
constexpr int OFF_X0 = OFF_V + 8192;           // X of even chunks              64 rows
constexpr int OFF_B3 = OFF_X0 + 8192;          // [b e^G K | b V]^T            192 rows
constexpr int OFF_X1 = OFF_B3 + 24576;         // X of odd chunks               64 rows
constexpr int OFF_KL = OFF_X1 + 8192;          // (e^(Gl-G) K)^T                2 x 128 rows
constexpr int OFF_WQ = OFF_KL + 2 * 16384;     // [w; e^G Q]                    2 K-blocks x 128 rows
constexpr int OFF_HT = OFF_WQ + 32768;         // h^T                           2 K-blocks x 64 rows
constexpr int OFF_VN = OFF_HT + 16384;         // v_new^T                       64 rows
constexpr int OFF_AQ = OFF_VN + 8192;          // A_qk                          2 x 64 rows
constexpr int OFF_SMALL = OFF_AQ + 2 * 8192;
constexpr int SMALL_BYTES = 5120;
// gates inside the four diagonal 16x16 blocks of one chunk (the F_GD part of its gate
// table, one buffer: refilled for chunk c+1 once the gating of chunk c has read it)
constexpr int GD_B = GD_BLOCK;
constexpr int OFF_GD = OFF_SMALL + SMALL_BYTES;
constexpr int SMEM_BYTES = OFF_GD + 4 * GD_B * 4 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct WsState {
  alignas(16) float tab[2][F_ROWS][64];  // refilled with chunk c+2 while the chain runs chunk c
  float EL[2];                      // base^(G_last) per chunk parity, for the chain
  uint64_t bar_p1, bar_p3, bar_p4, bar_p5, bar_po, bar_d0, bar_d1;
  uint64_t bar_ld[2], bar_v, bar_gd;  // TMA loads: stage parity (K, Q, X, factors), V, diagonal gates
  uint32_t tmem;
};
static_assert(sizeof(WsState) <= SMALL_BYTES, "small state");

__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ void prod_sync() { asm volatile("bar.sync 2, 256;" ::: "memory"); }
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
  const __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t *>(&b);
}

// TMA maps: q, k, v over [rows, H*128] and X over [slots*H*64, 64], 64 x 64 boxes
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
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(a.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(a.v);
  const __nv_bfloat16 *xw = a.xw;
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
    mbar_init(&st.bar_ld[0], 1);
    mbar_init(&st.bar_ld[1], 1);
    mbar_init(&st.bar_v, 1);
    mbar_init(&st.bar_gd, 1);
    mbar_fence_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = st.tmem;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);  // this warp's lane quarter
  bool bad = false;
  auto wait_par = [&](uint64_t *bar, int64_t phase) {
    if (!mbar_wait(bar, (uint32_t)(phase & 1), WAIT_LIMIT)) bad = true;
    fence_after_sync();
  };

  // ---- producer: loads (TMA, issued by one thread: ptid 32, warp 9 lane 0) --------------
  // Rows past the run end are loaded as they are (the next run's tokens, or zeros past
  // the tensor): they only meet beta = 0, a causal mask, or rows of o that are not stored.
  const int ptid = tid - 256;
  const bool loader = ptid == 32;
  int64_t last_ld[2] = {-1, -1}, last_v = -1;  // loader: newest chunk per barrier
  auto issue_kqx = [&](int64_t c) {  // K, Q, X and the gate factors of chunk c (buffers of parity c&1)
    const int s2 = (int)(c & 1);
    const uint32_t stg = sb + OFF_ST + s2 * SZ_STAGE;
    const uint32_t xt = sb + (s2 ? OFF_X1 : OFF_X0);
    const int y = (int)(r0 + c * GDN_CHUNK);
    const int64_t xs = (xbase + c) * H + h;
    uint64_t *bar = &st.bar_ld[s2];
    mbar_expect_tx(bar, 5 * 8192 + F_ROWS * GDN_CHUNK * 4);
    tma_load_2d(stg, &maps.q, h * GDN_DK, y, bar);  // rows 0..63: Q
    tma_load_2d(stg + 16384, &maps.q, h * GDN_DK + 64, y, bar);
    tma_load_2d(stg + 8192, &maps.k, h * GDN_DK, y, bar);  // rows 64..127: K
    tma_load_2d(stg + 16384 + 8192, &maps.k, h * GDN_DK + 64, y, bar);
    tma_load_2d(xt, &maps.x, 0, (int)(xs * GDN_CHUNK), bar);
    bulk_load(smem_u32(&st.tab[s2][0][0]), a.ftab + xs * F_TAB, F_ROWS * GDN_CHUNK * 4, bar);
    last_ld[s2] = c;
  };
  int64_t last_gd = -1;
  auto issue_gd = [&](int64_t c) {  // gates inside the diagonal blocks of chunk c
    mbar_expect_tx(&st.bar_gd, 4 * GD_B * 4);
    bulk_load(sb + OFF_GD, a.ftab + ((xbase + c) * H + h) * F_TAB + F_GD, 4 * GD_B * 4, &st.bar_gd);
    last_gd = c;
  };
  auto issue_v = [&](int64_t c) {  // the CTA's 64 columns of V of chunk c
    mbar_expect_tx(&st.bar_v, 8192);
    tma_load_2d(sb + OFF_V, &maps.v, h * GDN_DV + col0, (int)(r0 + c * GDN_CHUNK), &st.bar_v);
    last_v = c;
  };

  // ---- producer: one chunk -------------------------------------------------------------
  auto produce = [&](int64_t pc, int64_t c_chain) {
    const int ps = (int)(pc & 1);
    const uint32_t stg = sb + OFF_ST + ps * SZ_STAGE;
    const float(&tab)[F_ROWS][64] = st.tab[ps];
    // buffers of chunk pc+1 (they held chunk pc-1, finished in the previous round)
    if (loader && pc + 1 < nch) issue_kqx(pc + 1);
    wait_par(&st.bar_ld[ps], pc >> 1);  // K, Q, X and factors of chunk pc have landed
    if (ptid == 0) {  // P1: S = [Q; K] K^T (rows 0..63 = Q K^T)
      st.EL[ps] = tab[F_EG][63];
      fence_after_sync();
      mma_tiles(tmem + T_S + 64 * ps, stg, 16384, stg + 8192, 16384, 128, idesc_bf16(128, 64), false);
      mma_commit(&st.bar_p1);
    }
    __syncwarp();  // the issuing warp reconverges before any of its lanes polls a barrier
    // transposes, loads first: K -> B3 rows 0..127 (b e^G) and KL (e^(Gl-G)); V -> B3 rows 128..191 (b)
    {
      const int pw = warp - 8;
      uint32_t xk[4][4], xv[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int jb = pw + 8 * i, rb = jb >> 3, fb = jb & 7;
        trans16_load(stg + (fb >> 2) * 16384, 64 + rb * 16, (fb & 3) * 2, lane, xk[i]);  // K rows
      }
      wait_par(&st.bar_v, pc);  // V of chunk pc
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = pw + 8 * i, rb = t >> 2, cb = t & 3;
        trans16_load(sb + OFF_V, rb * 16, cb * 2, lane, xv[i]);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = pw + 8 * i, rb = t >> 2, cb = t & 3;
        trans16_store(sb + OFF_B3, 128 + cb * 16, rb * 16, xv[i], tab[F_BETA], lane);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int jb = pw + 8 * i, rb = jb >> 3, fb = jb & 7;
        trans16_store(sb + OFF_B3, fb * 16, rb * 16, xk[i], tab[F_BEG], lane);
        trans16_store(sb + OFF_KL + ps * 16384, fb * 16, rb * 16, xk[i], tab[F_EGL], lane);
      }
    }
    prod_sync();  // V consumed (the next chunk's is loaded after the P3b issue)
    // gating of Q K^T (rows 0..63 of S) -> A_qk, lower triangle including the diagonal.
    // Gate factors of this thread's 32 key tokens s, all read from tables (no exponential
    // here): between 16-token blocks EA[t] EB_{b(t)}[s], inside the diagonal block the UT
    // kernel's table (in OFF_GD). They do not depend on S, so they are formed while P1 may
    // still run.
    wait_par(&st.bar_gd, pc);  // diagonal-block gates of chunk pc
    float gf[32];
    if (q4 < 2) {
      const int t = row, bt = t >> 4;
      const float ea = tab[F_EA][t];
      const float *eb = tab[F_EB1 + (bt > 0 ? bt - 1 : 0)];
      const float *gd = reinterpret_cast<const float *>(sm + OFF_GD) + bt * GD_B + (t & 15);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int sj = 32 * hc + j, bs = sj >> 4;
        const float off = ea * eb[sj], dg = gd[(sj & 15) * 16];
        gf[j] = bs < bt ? off : (bs == bt ? dg : 0.f);
      }
    }
    wait_par(&st.bar_p1, pc);
    if (q4 < 2) {
      const int t = row;
      float sv[32];
      tmem_ld16(tl + T_S + 64 * ps + 32 * hc, *reinterpret_cast<float(*)[16]>(sv));
      tmem_ld16(tl + T_S + 64 * ps + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(sv + 16));
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) sv[j] *= gf[j];
      uint8_t *dst = sm + OFF_AQ + ps * 8192;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8)
        *reinterpret_cast<uint4 *>(dst + chunk_off(t, 4 * hc + q8)) = pack8(sv + 8 * q8);
    }
    fence_proxy_async();
    fence_before_sync();
    prod_sync();
    if (loader && pc + 1 < nch) issue_gd(pc + 1);  // the gating has read this chunk's
    if (ptid == 0) {  // P3b: w and u
      fence_after_sync();
      const uint32_t xt = sb + (ps ? OFF_X1 : OFF_X0);
      mma_tiles(tmem + T_WW, xt, 8192, sb + OFF_B3, 24576, 64, idesc_bf16(128, 128), false);
      mma_tiles(tmem + T_U + 64 * ps, xt, 8192, sb + OFF_B3 + 16384, 24576, 64, idesc_bf16(128, 64), false);
      mma_commit(&st.bar_p3);
    }
    __syncwarp();  // the issuing warp reconverges before any of its lanes polls a barrier
    if (loader && pc + 1 < nch) issue_v(pc + 1);  // V consumed by the transposes
    // operand of P4: rows 64..127 = e^G Q once the chain's P4 has read the previous one,
    // rows 0..63 = w once P3b is done (keys 64*hc .. +64 per thread)
    uint8_t *wq = sm + OFF_WQ + hc * 16384;
    if (c_chain >= 0) wait_par(&st.bar_p4, c_chain);
    if (q4 >= 2) {
      const float eg = tab[F_EG][row - 64];
      const uint8_t *qrow = sm + OFF_ST + ps * SZ_STAGE + hc * 16384;  // Q: stage rows 0..63
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4 *>(qrow + chunk_off(row - 64, c8)), f);
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] *= eg;
        *reinterpret_cast<uint4 *>(wq + chunk_off(row, c8)) = pack8(f);
      }
    }
    wait_par(&st.bar_p3, pc);
    if (q4 < 2) {
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        float sv[16];
        tmem_ld16(tl + T_WW + 64 * hc + 16 * part, sv);
        tmem_ld_wait();
        *reinterpret_cast<uint4 *>(wq + chunk_off(row, 2 * part)) = pack8(sv);
        *reinterpret_cast<uint4 *>(wq + chunk_off(row, 2 * part + 1)) = pack8(sv + 8);
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
  // h^T (B operand of P4): this thread's key `row`, columns 32*hc .. +32
  auto write_ht = [&]() {
    const uint32_t hbase = sb + OFF_HT + (row >> 6) * 8192 + (row & 7) * 2;
    const int kc = (row & 63) >> 3;
#pragma unroll
    for (int j = 0; j < 32; ++j) sts_u16(hbase + chunk_off(32 * hc + j, kc), bf16_bits(hreg[j]));
  };
  auto chain = [&](int64_t c) {
    const int par = (int)(c & 1);
    const int64_t c0 = r0 + c * GDN_CHUNK;
    const int n = chunk_rows(c);
    if (a.h_chunks) {  // entry state of chunk c
      const int64_t slot = a.cu ? (chunk_base + c) * H + h : ((int64_t)b * H + h) * NT + chunk_base + c;
      float4 *dst = reinterpret_cast<float4 *>(a.h_chunks + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV +
                                               col0 + 32 * hc);
#pragma unroll
      for (int g4 = 0; g4 < 8; ++g4)
        dst[g4] = make_float4(hreg[g4 * 4], hreg[g4 * 4 + 1], hreg[g4 * 4 + 2], hreg[g4 * 4 + 3]);
    }
    if (tid == 0) {  // P4: [w; e^G Q] h
      fence_after_sync();
      mma_tiles(tmem + T_D4, sb + OFF_WQ, 16384, sb + OFF_HT, 8192, 128, idesc_bf16(128, 64), false);
      mma_commit(&st.bar_p4);
    }
    __syncwarp();  // the issuing warp reconverges before any of its lanes polls a barrier
    wait_par(&st.bar_p4, c);
    if (q4 < 2) {  // v_new = u - w h  ->  v_new^T (column writes)
      const uint32_t base = sb + OFF_VN + (row & 7) * 2;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float wh[16], u[16];
        tmem_ld16(tl + T_D4 + 32 * hc + 16 * part, wh);
        tmem_ld16(tl + T_U + 64 * par + 32 * hc + 16 * part, u);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          sts_u16(base + chunk_off(32 * hc + 16 * part + j, row >> 3), bf16_bits(u[j] - wh[j]));
      }
    }
    fence_proxy_async();
    fence_before_sync();
    chain_sync();
    if (tid == 0) {  // P5, then the intra-chunk output term
      fence_after_sync();
      mma_tiles(tmem + T_P5, sb + OFF_KL + par * 16384, 16384, sb + OFF_VN, 8192, 64, idesc_bf16(128, 64), false);
      mma_commit(&st.bar_p5);
      mma_tiles(tmem + T_D4, sb + OFF_AQ + par * 8192 - 8192, 16384, sb + OFF_VN, 8192, 64, idesc_bf16(128, 64), true);
      mma_commit(&st.bar_po);
    }
    __syncwarp();  // the issuing warp reconverges before any of its lanes polls a barrier
    wait_par(&st.bar_p5, c);
    {
      const float el = st.EL[par];
      const uint32_t hbase = sb + OFF_HT + (row >> 6) * 8192 + (row & 7) * 2;
      const int kc = (row & 63) >> 3;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float p5[16];
        tmem_ld16(tl + T_P5 + 32 * hc + 16 * part, p5);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float &hv = hreg[16 * part + j];
          hv = fmaf(el, hv, p5[j]);
          sts_u16(hbase + chunk_off(32 * hc + 16 * part + j, kc), bf16_bits(hv));
        }
      }
      if (q4 >= 2) {  // o = scale (q' h + A_qk v_new); the whole warp loads (collective)
        wait_par(&st.bar_po, c);
        const bool st_row = o && row - 64 < n;
        uint4 *dst = reinterpret_cast<uint4 *>(o + ((c0 + (st_row ? row - 64 : 0)) * H + h) * GDN_DV + col0 + 32 * hc);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float ov[16];
          tmem_ld16(tl + T_D4 + 32 * hc + 16 * part, ov);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) ov[j] *= scale;
          if (st_row) {
            dst[2 * part] = pack8(ov);
            dst[2 * part + 1] = pack8(ov + 8);
          }
        }
      }
    }
    fence_proxy_async();
    fence_before_sync();
  };

  // ---- prologue --------------------------------------------------------------------------
  if (loader && nch > 0) {
    issue_kqx(0);
    issue_v(0);
    issue_gd(0);
  }
  if (!producer) {
    write_ht();
    fence_proxy_async();
  }
  __syncthreads();

  // round c: the chain runs chunk c while the producer prepares chunk c+1
  for (int64_t c = -1; c < nch; ++c) {
    if (producer) {
      if (c + 1 < nch) produce(c + 1, c);
    } else if (c >= 0) {
      chain(c);
    }
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
  }

  if (bad) {
    if (tid == 0) {
      raise_device_flag(a.dev_flag, kDevTimeout);
      mma_commit(&st.bar_d0);  // arrives once every MMA this thread issued has finished
    }
    if (tid == 256) mma_commit(&st.bar_d1);
    if (tid == 0) mbar_wait(&st.bar_d0, 0, WAIT_LIMIT);
    if (tid == 256) mbar_wait(&st.bar_d1, 0, WAIT_LIMIT);
    if (loader) {  // copies still in flight land before the CTA leaves
      for (int s2 = 0; s2 < 2; ++s2)
        if (last_ld[s2] >= 0) mbar_wait(&st.bar_ld[s2], (uint32_t)((last_ld[s2] >> 1) & 1), WAIT_LIMIT);
      if (last_v >= 0) mbar_wait(&st.bar_v, (uint32_t)(last_v & 1), WAIT_LIMIT);
      if (last_gd >= 0) mbar_wait(&st.bar_gd, (uint32_t)(last_gd & 1), WAIT_LIMIT);
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
    if (e == cudaSuccess) e = make_tmap_bf16(&maps.x, a.xw, GDN_CHUNK, slots * a.H * GDN_CHUNK, GDN_CHUNK * 2);
  }
  if (e != cudaSuccess) return e;
  auto kern = a.use_exp2 ? tc_fwd_ws_kernel<true> : tc_fwd_ws_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, NTH, SMEM_BYTES, st>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace gdn
