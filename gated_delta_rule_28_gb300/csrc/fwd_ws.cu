// Tensor-core (tcgen05) chunk forward for bf16 inputs, scalar gate (sm_103a):
// the state recurrence, with the preparation of the next chunk and the output
// of the current one interleaved on the tensor pipe.
//
// One CTA (512 threads) owns one independent run (batch row, packed document
// or segment) of one head and 64 of the 128 state columns; the UT transform
// kernel supplies X = (I + L)^-1 of every chunk already scaled by its columns,
// as the pair [X diag(b); X diag(b e^G)] in bf16. Per chunk (GDN Ascend C adapter
// forward, chunk_fwd_h and the output step):
//
//     P1   S = Q K^T                           -> A_qk = lower-incl(Q K^T (.) Gamma)
//     P3   [X diag(b); X diag(b e^G)] [K | V]  -> w = X diag(b e^G) K,  u = X diag(b) V
//     P4   [w; Q] h                            -> v_new = u - w h,  Q h
//     P5   K^T (e^(G_last - G) v_new)          -> h <- e^(G_last) h + P5
//     PO   A_qk v_new                          -> o = scale (e^G (Q h) + A_qk v_new)
//
// Only P4 -> v_new -> P5 -> h is a dependence chain from one chunk to the next;
// the tensor pipe runs one MMA group at a time, so one warp issues every MMA in
// the order P4(c), P3(c+1), P5(c), PO(c), P1(c+1): the next chunk's preparation
// fills the pipe while the chain converts v_new and h, and the output term runs
// while the chain waits for its next state. The warps are split by role and meet
// only on mbarriers (no CTA barrier per chunk):
//   warps 0..7   the state h in fp32 registers (thread = key row, 32 columns):
//                v_new (lane quarters 0, 1: token rows), Q h and the output
//                (quarters 2, 3), the update of h and its bf16 copy
//   warps 8, 9, 12, 13   the gating of Q K^T into A_qk
//   warp 10      the MMAs and the tensor copies of K, the X pair, V and the gate table
//   warps 11, 14, 15     w from tensor memory into the rows of the P4 operand [w; Q]
// The issuer waits on five barriers per chunk: "ready for P4" (h, w and the read of
// the previous Q h), the loads of chunk c+1, v_new, "ready for PO" (A_qk and the read of
// the previous output term) and Q of chunk c+1. Buffers are double- or triple-buffered so
// that every wait is for the event it names and no mbarrier runs two phases ahead of a
// thread that waits on it.
// Loads are TMA copies (tensor tiles with the 128-byte swizzle, and bulk copies of
// the gate table). No operand is transposed: the token-major tiles (K, V, v_new, h
// by key) enter the MMAs as MN-major operands. Every mbarrier wait is bounded; a
// wait that runs out raises the CTA's abort word, the others give up within a few
// hundred polls, and the CTA drains its MMAs and copies, frees its tensor memory
// and leaves with the device flag set.
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
constexpr int NTH = 512;  // 8 chain warps + 8 preparation warps
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
constexpr int OFF_K = OFF_WQ + 2 * 32768;     // K per chunk mod 3: 2 K-blocks x 64 rows
constexpr int OFF_XX = OFF_K + 3 * 16384;     // [X diag(b); X diag(b e^G)] per parity: 128 rows
constexpr int OFF_V = OFF_XX + 2 * 16384;     // V slice per parity: 64 rows
constexpr int OFF_HT = OFF_V + 2 * 8192;      // h: 128 key rows (MN-major B of P4)
constexpr int OFF_VN = OFF_HT + 16384;        // v_new: 64 token rows (MN-major B of PO)
constexpr int OFF_VNL = OFF_VN + 8192;        // e^(Gl - G) v_new (MN-major B of P5)
constexpr int OFF_AQ = OFF_VNL + 8192;        // A_qk per parity: 64 rows (PO's rows 0..63: the 8 KB before)
constexpr int OFF_TAB = OFF_AQ + 2 * 8192;    // gate table per chunk mod 3 (F_TAB floats)
constexpr int OFF_SMALL = OFF_TAB + 3 * F_TAB * 4;
constexpr int SMALL_BYTES = 512;
constexpr int SMEM_BYTES = OFF_SMALL + SMALL_BYTES + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert((F_TAB * 4) % 16 == 0 && OFF_TAB % 16 == 0, "bulk copy alignment");
// The MN-major K operand (two 64-key groups 8 KB apart, 64 token rows) stays inside shared
// memory under either assignment of its descriptor's two stride fields: groups 8 KB apart
// and K rows in 1 KB atoms, or the reverse. The other MN-major operands have one group.
static_assert(OFF_K + 2 * 16384 + 8192 + 8 * 1024 <= OFF_XX &&
                  OFF_K + 2 * 16384 + 1024 + 7 * 8192 + 1024 <= OFF_SMALL,
              "MN-major K operand extent");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct WsState {
  // MMA completions (tcgen05.commit by the issuing warp)
  uint64_t p1, p3, p4, p5, po, d0;
  // hand-offs to the issuer: ready for P4(c) = h(c) (8 chain warps) + w(c) (3) + Q h of
  // c-1 read (4 output warps); v_new(c) (4); ready for PO(c) = A_qk(c) (4 gating warps) +
  // output of c-1 read (4 output warps)
  uint64_t rdy4, vn, rdyo;
  uint64_t ld[3];  // TMA loads per chunk mod 3: K, the X pair, V and the gate table
  uint64_t q[2];   // TMA loads per chunk parity: Q (issued once P4 has read the buffer)
  uint32_t tmem;
  int abort;       // raised by a wait that ran out; the other waits then give up
};
static_assert(sizeof(WsState) <= SMALL_BYTES, "small state");

// TMA maps: q, k, v over [rows, H*128]; the X pair over [slots*H*128, 64]; 64 x 64 boxes
struct FwdMaps {
  TmaMap q, k, v, x;
};

// Polls until the phase of `parity` has completed; false once `limit` polls ran out or
// (checked every 256 polls) the CTA's abort word is set.
__device__ __forceinline__ bool poll(uint64_t *bar, uint32_t parity, const volatile int *abort) {
#pragma unroll 1
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort) return false;
  }
  return false;
}

template <bool E2>
__global__ void __launch_bounds__(NTH, 1) tc_fwd_ws_kernel(SimtFwdArgs a, const __grid_constant__ FwdMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned base by pointer arithmetic on the shared array, so that the compiler keeps
  // the shared address space (shared-memory instructions, not generic ones)
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  WsState &st = *reinterpret_cast<WsState *>(sm + OFF_SMALL);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool chain_warp = warp < 8;
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
  const int nch = (int)((r1 - r0 + GDN_CHUNK - 1) / GDN_CHUNK);
  auto chunk_rows = [&](int c) { return (int)min((int64_t)GDN_CHUNK, r1 - (r0 + (int64_t)c * GDN_CHUNK)); };

  // ---- tensor memory, barriers -----------------------------------------------------
  if (warp == 0) {
    tmem_alloc(&st.tmem, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&st.p1, 1);
    mbar_init(&st.p3, 1);
    mbar_init(&st.p4, 1);
    mbar_init(&st.p5, 1);
    mbar_init(&st.po, 1);
    mbar_init(&st.d0, 1);
    mbar_init(&st.rdy4, 15);
    mbar_init(&st.vn, 4);
    mbar_init(&st.rdyo, 8);
    for (int i = 0; i < 3; ++i) mbar_init(&st.ld[i], 1);
    mbar_init(&st.q[0], 1);
    mbar_init(&st.q[1], 1);
    st.abort = 0;
    mbar_fence_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // the X pair and the gate tables come from the kernel launched before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem = st.tmem;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);  // this warp's lane quarter
  volatile int *abort_word = &st.abort;
  bool bad = false;
  // warp-uniform bounded wait for the completion of phase `phase` (its parity)
  auto wt = [&](uint64_t *bar, int phase) -> bool {
    bool ok = poll(bar, (uint32_t)(phase & 1), abort_word);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      bad = true;
      *abort_word = 1;
    }
    fence_after_sync();
    return ok;
  };
  // one arrival per warp, after the warp's shared-memory writes (made visible to the tensor
  // core) and tensor-memory reads
  auto arrive_w = [&](uint64_t *bar) {
    fence_proxy_async();
    fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  };
  auto wq_at = [&](int c) { return sb + OFF_WQ + (uint32_t)(c & 1) * 32768u; };
  auto k_at = [&](int c) { return sb + OFF_K + (uint32_t)(c % 3) * 16384u; };
  auto xx_at = [&](int c) { return sb + OFF_XX + (uint32_t)(c & 1) * 16384u; };
  auto v_at = [&](int c) { return sb + OFF_V + (uint32_t)(c & 1) * 8192u; };
  auto tab_at = [&](int c) { return reinterpret_cast<const float(*)[64]>(sm + OFF_TAB + (c % 3) * (F_TAB * 4)); };

  int last_ld[3] = {-1, -1, -1};  // issuer: newest chunk loaded per buffer
  int last_q[2] = {-1, -1};       // chain warp 0: newest Q load per parity
  float hreg[32];                     // chain warps: the state (key `row`, 32 columns)
  // Q of chunk c into rows 64..127 of [w; Q] of parity c&1, by chain warp 0 once P4 of
  // chunk c-2 (the last reader of the buffer) has completed
  auto issue_q = [&](int c) {
    const int s2 = c & 1;
    const int y = (int)(r0 + (int64_t)c * GDN_CHUNK);
    mbar_expect_tx_w(&st.q[s2], 2 * 8192);
    tma_load_2d_w(wq_at(c) + 8192, &maps.q, h * GDN_DK, y, &st.q[s2]);
    tma_load_2d_w(wq_at(c) + 16384 + 8192, &maps.q, h * GDN_DK + 64, y, &st.q[s2]);
    last_q[s2] = c;
  };

  if (warp == 10) {
    // ---- MMA issue and loads -------------------------------------------------------------
    // Every TMA copy and tcgen05 MMA is issued warp-collectively (one elected lane of a
    // warp-uniform call, tc.cuh). Rows past the run end are loaded as they are (the next
    // run's tokens, or zeros past the tensor): they only meet beta = 0 (zero columns of
    // both X's), a causal mask, or rows of o that are not stored.
    auto issue_loads = [&](int c) {  // K, the X pair, V and the gate table of chunk c
      const int sl = c % 3;
      const int y = (int)(r0 + (int64_t)c * GDN_CHUNK);
      const int64_t xs = (xbase + c) * H + h;
      uint64_t *bar = &st.ld[sl];
      mbar_expect_tx_w(bar, 5 * 8192 + F_TAB * 4);
      tma_load_2d_w(k_at(c), &maps.k, h * GDN_DK, y, bar);
      tma_load_2d_w(k_at(c) + 8192, &maps.k, h * GDN_DK + 64, y, bar);
      tma_load_2d_w(xx_at(c), &maps.x, 0, (int)(xs * 2 * GDN_CHUNK), bar);
      tma_load_2d_w(xx_at(c) + 8192, &maps.x, 0, (int)(xs * 2 * GDN_CHUNK + GDN_CHUNK), bar);
      tma_load_2d_w(v_at(c), &maps.v, h * GDN_DV + col0, y, bar);
      bulk_load_w(sb + OFF_TAB + (uint32_t)sl * (F_TAB * 4), a.ftab + xs * F_TAB, F_TAB * 4, bar);
      last_ld[sl] = c;
    };
    // P3: [X diag(b); X diag(b e^G)] [K | V] -> rows 64..127 of the K product = w, rows
    // 0..63 of the V product = u (K and V token-major, read as MN-major B)
    auto p3 = [&](int c) {
      mma_grp_w(tmem + T_WW, kmaj(xx_at(c), 0), mnmaj(k_at(c), 8192), 64, idesc_bf16(128, 128, false, false, true),
                false);
      mma_grp_w(tmem + T_U + 64 * (uint32_t)(c & 1), kmaj(xx_at(c), 0), mnmaj(v_at(c), 0), 64,
                idesc_bf16(128, 64, false, false, true), false);
      mma_commit_w(&st.p3);
    };
    // P1: S = Q K^T (A rows 64..127: the next 64 rows of shared memory, unread output rows)
    auto p1 = [&](int c) {
      mma_grp_w(tmem + T_S, kmaj(wq_at(c) + 8192, 16384), kmaj(k_at(c), 8192), 128, idesc_bf16(128, 64), false);
      mma_commit_w(&st.p1);
    };
    do {
      if (nch > 0) issue_loads(0);
      if (nch > 1) issue_loads(1);
      if (nch == 0) break;
      if (!wt(&st.ld[0], 0)) break;
      p3(0);
      if (!wt(&st.q[0], 0)) break;
      p1(0);
      for (int c = 0; c < nch; ++c) {
        const int par = c & 1;
        // P4(c): h(c), w(c) written, Q h of c-1 read; Q(c) landed (waited for P1(c))
        if (!wt(&st.rdy4, c)) break;
        mma_grp_w(tmem + T_D4, kmaj(wq_at(c), 16384), mnmaj(sb + OFF_HT, 0), 128,
                  idesc_bf16(128, 64, false, false, true), false);
        mma_commit_w(&st.p4);
        // loads of chunk c+2: its X / V buffers held chunk c (P3(c) came before P5(c-1), done
        // before h(c)); its K buffer and gate table chunk c-1 (P5(c-1) done; every warp read
        // its factors of c-1 before h(c) or A_qk(c-1))
        if (c + 2 < nch) issue_loads(c + 2);
        // P3(c+1): its loads landed; w(c) and u(c-1) have left tensor memory
        if (c + 1 < nch) {
          if (!wt(&st.ld[(c + 1) % 3], ((c + 1) / 3) & 1)) break;
          p3(c + 1);
        }
        // P5(c): K^T (e^(Gl-G) v_new), K read as MN-major A
        if (!wt(&st.vn, c)) break;
        mma_grp_w(tmem + T_P5, mnmaj(k_at(c), 8192), mnmaj(sb + OFF_VNL, 0), 64, idesc_bf16(128, 64, false, true, true),
                  false);
        mma_commit_w(&st.p5);
        // PO(c): A_qk(c) written; the output of c-1 has read its accumulator
        if (!wt(&st.rdyo, c)) break;
        mma_grp_w(tmem + T_PO, kmaj(sb + OFF_AQ + par * 8192 - 8192, 0), mnmaj(sb + OFF_VN, 0), 64,
                  idesc_bf16(128, 64, false, false, true), false);
        mma_commit_w(&st.po);
        // P1(c+1): Q(c+1) landed; A_qk(c) has left tensor memory
        if (c + 1 < nch) {
          if (!wt(&st.q[(c + 1) & 1], (c + 1) >> 1)) break;
          p1(c + 1);
        }
      }
    } while (false);
  } else if (warp == 11 || warp == 14 || warp == 15) {
    // ---- w rows of the P4 operand -----------------------------------------------------------
    // rows 0..63 of [w; Q] of chunk c = P3 rows 64..127: warp 14 rows 64..95, all 128 keys;
    // warps 11, 15 rows 96..127, keys 0..63 / 64..127
    const int kb0 = warp == 15 ? 1 : 0, kb1 = warp == 14 ? 2 : kb0 + 1;
    for (int c = 0; c < nch; ++c) {
      if (!wt(&st.p3, c)) break;
      uint8_t *wq = sm + OFF_WQ + (c & 1) * 32768;
      for (int kb = kb0; kb < kb1; ++kb) {
#pragma unroll
        for (int part = 0; part < 4; ++part) {
          float sv[16];
          tmem_ld16(tl + T_WW + 64 * kb + 16 * part, sv);
          tmem_ld_wait();
          *reinterpret_cast<uint4 *>(wq + kb * 16384 + chunk_off(row - 64, 2 * part)) = pack8(sv);
          *reinterpret_cast<uint4 *>(wq + kb * 16384 + chunk_off(row - 64, 2 * part + 1)) = pack8(sv + 8);
        }
      }
      arrive_w(&st.rdy4);
    }
  } else if (!chain_warp) {
    // ---- gating of Q K^T (rows 0..63 of S) -> A_qk, lower triangle with the diagonal ----------
    // Gate factors of this thread's 32 key tokens s, formed before P1 completes: between
    // 16-token blocks from the tables, EA[t] EB_{b(t)}[s] (no exponential); inside the
    // diagonal block base^(G_t - G_s), 16 exponentials in the two warps whose key tokens
    // hold their rows' diagonal blocks (8: rows 0..31, keys 0..31; 13: rows 32..63, keys
    // 32..63).
    const int t = row;
    for (int c = 0; c < nch; ++c) {
      if (!wt(&st.ld[c % 3], (c / 3) & 1)) break;
      const float(*tab)[64] = tab_at(c);
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
      if (!wt(&st.p1, c)) break;
      float sv[32];
      tmem_ld16(tl + T_S + 32 * hc, *reinterpret_cast<float(*)[16]>(sv));
      tmem_ld16(tl + T_S + 32 * hc + 16, *reinterpret_cast<float(*)[16]>(sv + 16));
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) sv[j] *= gf[j];
      uint8_t *dst = sm + OFF_AQ + (c & 1) * 8192;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) *reinterpret_cast<uint4 *>(dst + chunk_off(t, 4 * hc + q8)) = pack8(sv + 8 * q8);
      arrive_w(&st.rdyo);
    }
  } else {
    // ---- chain: the state, v_new, Q h, the output ------------------------------------------------
    const float *src = nullptr;
    if (a.h0) {
      const int64_t slot = a.nseg > 0 ? (((int64_t)b * H + h) * a.nseg + s) : ((int64_t)state_idx * H + h);
      src = a.h0 + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV + col0 + 32 * hc;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) hreg[j] = src ? src[j] : 0.f;
    // h in bf16 (MN-major B operand of P4): this thread's key `row`, columns 32*hc .. +32
    auto write_ht = [&]() {
      uint8_t *hrow = sm + OFF_HT;
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8)
        *reinterpret_cast<uint4 *>(hrow + chunk_off(row, 4 * hc + q8)) = pack8(hreg + 8 * q8);
    };
    if (warp == 0) {
      if (nch > 0) issue_q(0);
      if (nch > 1) issue_q(1);
    }
    write_ht();
    arrive_w(&st.rdy4);  // h(0)
    if (q4 >= 2) {       // no Q h and no output before chunk 0
      arrive_w(&st.rdy4);
      arrive_w(&st.rdyo);
    }
    for (int c = 0; c < nch; ++c) {
      const int par = c & 1;
      const int64_t c0 = r0 + (int64_t)c * GDN_CHUNK;
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
      // this thread's gate factors of chunk c, read before h(c+1) is handed over (after which
      // the table's buffer may be refilled)
      if (!wt(&st.ld[c % 3], (c / 3) & 1)) break;
      const float(*tab)[64] = tab_at(c);
      const float el = tab[F_EG][63];
      const float egl = tab[F_EGL][row & 63];
      const float eg = tab[F_EG][row & 63];
      if (!wt(&st.p4, c)) break;
      if (warp == 0 && c + 2 < nch) issue_q(c + 2);  // P4 has read Q of chunk c
      uint32_t qe[16];  // output rows: base^G Q h in bf16 pairs
      if (q4 < 2) {  // v_new = u - w h (token row), and e^(Gl - G) v_new
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
        arrive_w(&st.vn);
      } else {  // base^G Q h (rows 64..127 of P4), kept for the output
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float qv[16];
          tmem_ld16(tl + T_D4 + 32 * hc + 16 * part, qv);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(eg * qv[2 * j], eg * qv[2 * j + 1]);
            qe[8 * part + j] = *reinterpret_cast<const uint32_t *>(&b2);
          }
        }
        arrive_w(&st.rdy4);
      }
      if (!wt(&st.p5, c)) break;
      {
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float p5[16];
          tmem_ld16(tl + T_P5 + 32 * hc + 16 * part, p5);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) hreg[16 * part + j] = fmaf(el, hreg[16 * part + j], p5[j]);
        }
        write_ht();
        arrive_w(&st.rdy4);
      }
      if (q4 >= 2) {  // o = scale (base^G Q h + A_qk v_new)
        if (!wt(&st.po, c)) break;
        const bool st_row = o && row - 64 < n;
        uint4 *dst = reinterpret_cast<uint4 *>(o + ((c0 + (st_row ? row - 64 : 0)) * H + h) * GDN_DV + col0 + 32 * hc);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          float av[16];
          tmem_ld16(tl + T_PO + 32 * hc + 16 * part, av);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 q2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qe[8 * part + j]));
            av[2 * j] = scale * (q2.x + av[2 * j]);
            av[2 * j + 1] = scale * (q2.y + av[2 * j + 1]);
          }
          if (st_row) {
            dst[2 * part] = pack8(av);
            dst[2 * part + 1] = pack8(av + 8);
          }
        }
        arrive_w(&st.rdyo);
      }
    }
  }

  if (__syncthreads_or(bad)) {
    if (warp == 10) {
      // the elected lane arrives once every MMA it issued has finished; copies in flight land
      mma_commit_w(&st.d0);
      mbar_wait(&st.d0, 0, WAIT_LIMIT);
      for (int sl = 0; sl < 3; ++sl)
        if (last_ld[sl] >= 0) mbar_wait(&st.ld[sl], (uint32_t)((last_ld[sl] / 3) & 1), WAIT_LIMIT);
    }
    if (warp == 0)  // Q copies still in flight land before the CTA leaves
      for (int s2 = 0; s2 < 2; ++s2)
        if (last_q[s2] >= 0) mbar_wait(&st.q[s2], (uint32_t)((last_q[s2] >> 1) & 1), WAIT_LIMIT);
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
  } else if (chain_warp && a.ht && (a.nseg == 0 || s == a.nseg - 1)) {
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
