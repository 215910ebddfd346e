// Per-key (KDA) state recurrence on tensor cores (tcgen05, sm_103a), over the
// per-chunk blobs of the prep kernel (kda_prep.cu). The decay acts per key
// channel, so the state's rows decay by b^(G_last) of their key before the
// rank-one updates ("state_summary.py" kda_split_state_summary_kernel, loop
// body: the state is decayed by the last cumulative gate and updated with v_new
// computed against the undecayed entry state; the KDA adapter's chunk_fwd_h and
// chunk_kda_fwd_finalize stages on the "Diff Coverage" page):
//
//   P4   [w; Q b^G] h          -> v_new = u - w h,  Q b^G h
//   PO   A_qk v_new            -> o = Q b^G h + A_qk v_new   (scale folded in by the prep)
//   P5   (K b^(G_last-G))^T v_new -> h <- Diag(b^(G_last)) h + P5
//
// One CTA (8 chain warps + 1 loader warp) owns one run (batch row, packed
// document or segment) of one head and 64 state columns; the state lives in fp32
// registers of the chain warps (thread = key row, 32 columns). The loader warp
// fetches the next chunk's blob with bulk copies into the other of two buffers
// while the chain works on the current one. The output of chunk c is written
// during step c + 1, by the warps whose tensor-memory lanes hold it (the output
// rows) while the others form v_new, so it is off the state's critical path:
// P4 and PO accumulate into two tensor-memory buffers by chunk parity.
//
// Summary mode runs the same recurrence for the segment summary (combined mode
// of kda_split_state_summary_kernel): column slices 0, 1 carry S_ext (from a
// zero state, with u), slices 2, 3 the transfer map M (from the identity, with
// u = 0, so v_new = -w h), and nothing but the final states is written.
//
// Every mbarrier wait is bounded; a wait that runs out sets the device flag and
// the CTA drains its MMAs and copies, frees its tensor memory and leaves.
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tile_ops.cuh"

namespace gdn {
namespace {
using namespace tc;
using namespace tile;
using namespace kda;

constexpr int TBV = 64;
constexpr int NTH = 288;  // 8 chain warps + the loader
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t T_D4 = 0;    // 2 x 64, per chunk parity: P4 rows 0..63 = w h, rows 64..127 = Q b^G h
constexpr uint32_t T_PO = 128;  // 2 x 64, per chunk parity: PO rows 64..127 = A_qk v_new
constexpr uint32_t T_P5 = 256;  // 64: P5, 128 key rows

// one buffer per chunk parity: the blob's pieces this CTA needs
constexpr int BUF_WQ = 0;       // [w; Q b^G], K-blocks 16 KB apart
constexpr int BUF_KL = 32768;   // K b^(G_last - G), two 64-key groups
constexpr int BUF_U = 49152;    // u, this CTA's 64 columns
constexpr int BUF_AQ = 57344;   // A_qk (PO's A operand starts 8 KB before it: its rows 0..63
                                // are unread output rows)
constexpr int BUF_EL = 65536;   // b^(G_last) per key
constexpr int BUF_BYTES = 66560;
constexpr int OFF_HT = 2 * BUF_BYTES;    // h in bf16: 128 key rows (MN-major B of P4)
constexpr int OFF_VN = OFF_HT + 16384;   // v_new: 64 token rows (MN-major B of PO and P5)
constexpr int OFF_SMALL = OFF_VN + 8192;
constexpr int SMEM_BYTES = OFF_SMALL + 1024 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(BUF_BYTES % 1024 == 0 && BUF_AQ - 8192 >= 0, "tile alignment");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct ChainState {
  uint64_t bar_p4, bar_p5, bar_po, bar_d0;
  uint64_t bar_ld[2];
  uint32_t tmem;
};

__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__global__ void __launch_bounds__(NTH, 1) kda_chain_kernel(KdaChainArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  ChainState &st = *reinterpret_cast<ChainState *>(sm + OFF_SMALL);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool loader = warp == 8;
  const int q4 = warp & 3;         // tensor-memory lane quarter
  const int hc = (warp >> 2) & 1;  // 32-column half of the CTA's 64 columns
  const int row = q4 * 32 + lane;  // tensor-memory lane = key row (P4: token row)
  const int H = a.H, h = blockIdx.y, z = blockIdx.z;
  const int slice = blockIdx.x;
  const bool summ = a.summary != 0;
  const bool mcols = summ && slice >= 2;  // transfer-map columns: identity start, u = 0
  const int col0 = (slice & 1) * TBV;

  // ---- the run ----------------------------------------------------------------
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

  // ---- tensor memory, barriers -------------------------------------------------------
  if (warp == 0) {
    tmem_alloc(&st.tmem, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&st.bar_p4, 1);
    mbar_init(&st.bar_p5, 1);
    mbar_init(&st.bar_po, 1);
    mbar_init(&st.bar_d0, 1);
    mbar_init(&st.bar_ld[0], 1);
    mbar_init(&st.bar_ld[1], 1);
    mbar_fence_init();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // the blobs come from the prep kernel launched before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem = st.tmem;
  const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16);
  bool bad = false;
  auto wait_par = [&](uint64_t *bar, int64_t phase) {
    if (!mbar_wait(bar, (uint32_t)(phase & 1), WAIT_LIMIT)) bad = true;
    fence_after_sync();
  };
  auto buf_at = [&](int64_t c) { return sb + (uint32_t)(c & 1) * BUF_BYTES; };

  // ---- loader: the blob pieces of chunk c into buffer c&1 ---------------------------------
  int64_t last_ld[2] = {-1, -1};
  auto issue_loads = [&](int64_t c) {
    const int par = (int)(c & 1);
    const uint8_t *blob = a.blob + (size_t)((xbase + c) * H + h) * BLOB_BYTES;
    const uint32_t dst = buf_at(c);
    uint64_t *bar = &st.bar_ld[par];
    const bool with_u = !mcols;
    if (!summ) {
      mbar_expect_tx_w(bar, 32768 + 16384 + 8192 + 8192 + 512);
      bulk_load_w(dst + BUF_WQ, blob + BLOB_WQ, 32768, bar);
      bulk_load_w(dst + BUF_AQ, blob + BLOB_AQ, 8192, bar);
    } else {  // w rows only (no Q, no A_qk in the summary)
      mbar_expect_tx_w(bar, 16384 + 16384 + (with_u ? 8192 : 0) + 512);
      bulk_load_w(dst + BUF_WQ, blob + BLOB_WQ, 8192, bar);
      bulk_load_w(dst + BUF_WQ + 16384, blob + BLOB_WQ + 16384, 8192, bar);
    }
    bulk_load_w(dst + BUF_KL, blob + BLOB_KL, 16384, bar);
    if (with_u) bulk_load_w(dst + BUF_U, blob + BLOB_U + (col0 >> 6) * 8192, 8192, bar);
    bulk_load_w(dst + BUF_EL, blob + BLOB_EL, 512, bar);
    last_ld[par] = c;
  };

  // ---- chain: state and one chunk ----------------------------------------------------------
  float hreg[32];
  if (!loader) {
    if (mcols) {
#pragma unroll
      for (int j = 0; j < 32; ++j) hreg[j] = (row == col0 + 32 * hc + j) ? 1.f : 0.f;
    } else {
      const float *src = nullptr;
      if (a.h0 && !summ) {
        const int64_t slot = a.nseg > 0 ? (((int64_t)b * H + h) * a.nseg + s) : ((int64_t)state_idx * H + h);
        src = a.h0 + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV + col0 + 32 * hc;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) hreg[j] = src ? src[j] : 0.f;
    }
  }
  auto write_ht = [&]() {
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8)
      *reinterpret_cast<uint4 *>(sm + OFF_HT + chunk_off(row, 4 * hc + q8)) = pack8(hreg + 8 * q8);
  };
  // o = Q b^G h + A_qk v_new of chunk c (token row - 64), by the warps of lanes 64..127
  auto output = [&](int64_t c) {
    const int par = (int)(c & 1);
    const int64_t c0 = r0 + c * GDN_CHUNK;
    const int n = (int)min((int64_t)GDN_CHUNK, r1 - c0);
    wait_par(&st.bar_po, c);
    const bool st_row = a.o && row - 64 < n;
    uint4 *dst = reinterpret_cast<uint4 *>(a.o + ((c0 + (st_row ? row - 64 : 0)) * H + h) * GDN_DV + col0 + 32 * hc);
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      float ov[16], av[16];
      tmem_ld16(tl + T_D4 + 64 * par + 32 * hc + 16 * part, ov);
      tmem_ld16(tl + T_PO + 64 * par + 32 * hc + 16 * part, av);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) ov[j] += av[j];
      if (st_row) {
        dst[2 * part] = pack8(ov);
        dst[2 * part + 1] = pack8(ov + 8);
      }
    }
  };
  auto chain = [&](int64_t c) {
    const int par = (int)(c & 1);
    const uint32_t buf = buf_at(c);
    uint8_t *bufp = sm + (size_t)par * BUF_BYTES;
    if (a.h_chunks) {  // entry state of chunk c
      const int64_t slot = a.cu ? (chunk_base + c) * H + h : ((int64_t)b * H + h) * NT + chunk_base + c;
      float4 *dst = reinterpret_cast<float4 *>(a.h_chunks + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV +
                                               col0 + 32 * hc);
#pragma unroll
      for (int g4 = 0; g4 < 8; ++g4)
        dst[g4] = make_float4(hreg[g4 * 4], hreg[g4 * 4 + 1], hreg[g4 * 4 + 2], hreg[g4 * 4 + 3]);
    }
    wait_par(&st.bar_ld[par], c >> 1);
    if (warp == 0) {  // P4: [w; Q b^G] h
      mma_ops_w(tmem + T_D4 + 64 * par, kmaj(buf + BUF_WQ, 16384), mnmaj(sb + OFF_HT, 0), 128,
                idesc_bf16(128, 64, false, false, true), false);
      mma_commit_w(&st.bar_p4);
    }
    __syncwarp();
    if (!summ && q4 >= 2 && c > 0) output(c - 1);  // the previous chunk's output, meanwhile
    wait_par(&st.bar_p4, c);
    if (q4 < 2) {  // v_new = u - w h (token row), the whole warp loads tensor memory
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float wh[16], u[16];
        tmem_ld16(tl + T_D4 + 64 * par + 32 * hc + 16 * part, wh);
        tmem_ld_wait();
        if (mcols) {
#pragma unroll
          for (int j = 0; j < 16; ++j) u[j] = 0.f;
        } else {
          unpack8(*reinterpret_cast<const uint4 *>(bufp + BUF_U + chunk_off(row, 4 * hc + 2 * part)), u);
          unpack8(*reinterpret_cast<const uint4 *>(bufp + BUF_U + chunk_off(row, 4 * hc + 2 * part + 1)), u + 8);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) u[j] -= wh[j];
        *reinterpret_cast<uint4 *>(sm + OFF_VN + chunk_off(row, 4 * hc + 2 * part)) = pack8(u);
        *reinterpret_cast<uint4 *>(sm + OFF_VN + chunk_off(row, 4 * hc + 2 * part + 1)) = pack8(u + 8);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    chain_sync();
    if (warp == 0) {
      fence_after_sync();
      // P5 first (the state update waits for it): (K b^(Gl-G))^T v_new, the key tile read
      // as MN-major A; then PO for the output (read during the next step). The commit of
      // the next P4 also covers this PO, so v_new is not rewritten before PO has read it.
      mma_ops_w(tmem + T_P5, mnmaj(buf + BUF_KL, 8192), mnmaj(sb + OFF_VN, 0), 64,
                idesc_bf16(128, 64, false, true, true), false);
      mma_commit_w(&st.bar_p5);
      if (!summ) {  // PO: A_qk v_new (A rows 64..127 = A_qk)
        mma_ops_w(tmem + T_PO + 64 * par, kmaj(buf + BUF_AQ - 8192, 0), mnmaj(sb + OFF_VN, 0), 64,
                  idesc_bf16(128, 64, false, false, true), false);
        mma_commit_w(&st.bar_po);
      }
    }
    __syncwarp();
    wait_par(&st.bar_p5, c);
    const float el = reinterpret_cast<const float *>(bufp + BUF_EL)[row];
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      float p5[16];
      tmem_ld16(tl + T_P5 + 32 * hc + 16 * part, p5);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) hreg[16 * part + j] = fmaf(el, hreg[16 * part + j], p5[j]);
    }
    write_ht();
    fence_proxy_async();
    fence_before_sync();
  };

  // ---- rounds ------------------------------------------------------------------------------
  if (loader && nch > 0) issue_loads(0);
  if (!loader) {
    write_ht();
    fence_proxy_async();
  }
  __syncthreads();
  for (int64_t c = 0; c < nch; ++c) {
    if (loader) {
      if (c + 1 < nch) issue_loads(c + 1);  // the buffer held chunk c-1, finished last round
    } else {
      chain(c);
    }
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
  }
  if (!bad && !summ && nch > 0 && !loader && q4 >= 2) {  // the last chunk's output
    output(nch - 1);
  }
  if (__syncthreads_or(bad)) bad = true;

  if (bad) {
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    if (warp == 0) mma_commit_w(&st.bar_d0);  // arrives once every MMA warp 0 issued is done
    if (warp == 0) mbar_wait(&st.bar_d0, 0, WAIT_LIMIT);
    if (loader)  // copies still in flight land before the CTA leaves
      for (int p2 = 0; p2 < 2; ++p2)
        if (last_ld[p2] >= 0) mbar_wait(&st.bar_ld[p2], (uint32_t)((last_ld[p2] >> 1) & 1), WAIT_LIMIT);
  } else if (!loader) {
    float *dst = nullptr;
    if (summ) {
      const int64_t sl = ((int64_t)b * H + h) * a.nseg + s;
      dst = mcols ? a.M + sl * GDN_DK * GDN_DK : a.S_ext + sl * GDN_DK * GDN_DV;
    } else if (a.ht && (a.nseg == 0 || s == a.nseg - 1)) {
      dst = a.ht + ((int64_t)state_idx * H + h) * GDN_DK * GDN_DV;
    }
    if (dst) {
      float4 *d4 = reinterpret_cast<float4 *>(dst + (int64_t)row * GDN_DV + col0 + 32 * hc);
#pragma unroll
      for (int g4 = 0; g4 < 8; ++g4)
        d4[g4] = make_float4(hreg[g4 * 4], hreg[g4 * 4 + 1], hreg[g4 * 4 + 2], hreg[g4 * 4 + 3]);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_kda_chain(const KdaChainArgs &a, dim3 grid, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(kda_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: set-up overlaps the end of the prep kernel
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
  return cudaLaunchKernelEx(&cfg, kda_chain_kernel, a);
}

}  // namespace gdn
