// Per-key (KDA) reverse state recurrence on tensor cores (tcgen05, sm_103a), over the
// per-chunk blobs of the prep kernel (kda_prep.cu) recomputed for the backward. Per chunk,
// from the last to the first (the reverse loop of "state_summary.py"
// kda_state_grad_ext_kernel; the KDA adapter's bwd_dhu stage on the "Diff Coverage" page):
//
//   dv_new_c = (K b^(G_last - G)) dh_{c+1} + scale A_qk^T dO_c
//   dh_c     = Diag(b^(G_last)) dh_{c+1} + (scale Q b^G)^T dO_c - w_c^T dv_new_c
//
// where dh_{c+1} is the gradient of chunk c's exit state. Every operand is in the blob:
// K b^(G_last - G) (token rows), scale A_qk, [w; scale Q b^G], b^(G_last); dO comes by a
// TMA tile copy. It writes what the per-key local-gradient kernel reads: the exit-state
// gradient of every chunk (fp32) and dv_new (fp32), and returns dh_0.
//
// One CTA (8 state warps + 1 loader warp) owns one run (batch row, packed document or
// segment) of one head and 64 state columns; dh lives in fp32 registers (thread = key row,
// 32 columns) and in bf16 in shared memory as the MN-major B operand of the first product.
// The loader fetches the next chunk's blob pieces and dO tile into the other of two buffers.
// Tokens past the run end are zeroed in the dO tile (they would otherwise reach dv_new and
// dh through A_qk^T dO and (Q b^G)^T dO). Every mbarrier wait is bounded; a wait that runs
// out sets the device flag and the CTA drains its MMAs and copies and leaves.
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
constexpr int NTH = 288;  // 8 state warps + the loader
constexpr uint32_t TMEM_COLS = 128;
constexpr uint32_t T_DV = 0;   // 64: dv_new, token rows 0..63
constexpr uint32_t T_DH = 64;  // 64: the state-gradient product, key rows

// one buffer per round parity
constexpr int BUF_WQ = 0;       // [w; scale Q b^G], K-blocks 16 KB apart
constexpr int BUF_KL = 32768;   // K b^(G_last - G), two 64-key groups 8 KB apart
constexpr int BUF_AQ = 49152;   // scale A_qk (rows t, columns s)
constexpr int BUF_DO = 57344;   // dO, 64 tokens x this CTA's 64 columns
constexpr int BUF_EL = 65536;   // b^(G_last) per key
constexpr int BUF_BYTES = 66560;
constexpr int OFF_DH = 2 * BUF_BYTES;   // dh in bf16: 128 key rows (MN-major B)
constexpr int OFF_DV = OFF_DH + 16384;  // dv_new in bf16: 64 token rows (MN-major B)
constexpr int OFF_SMALL = OFF_DV + 8192;
constexpr int SMEM_BYTES = OFF_SMALL + 1024 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
// 128-row operands whose rows 64..127 are not needed read the bytes after their 64 rows:
// the KL tile's second key group (KL as a K-major A), the dO tile (A_qk^T as an MN-major A)
static_assert(BUF_KL + 8192 + 8192 <= BUF_BYTES && BUF_AQ + 8192 + 8192 <= BUF_BYTES, "operand extents");

constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct DhuState {
  uint64_t bar_dv, bar_dh, bar_d0;
  uint64_t bar_ld[2];
  uint32_t tmem;
};

__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

struct DhuMaps {
  TmaMap dO;
};

__global__ void __launch_bounds__(NTH, 1) kda_dhu_kernel(BwdArgs a, const __grid_constant__ DhuMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  DhuState &st = *reinterpret_cast<DhuState *>(sm + OFF_SMALL);
  const uint32_t sb = smem_u32(sm);

  const int tid = threadIdx.x, warp = tid >> 5;
  const bool loader = warp == 8;
  const int q4 = warp & 3, hc = (warp >> 2) & 1;
  const int row = q4 * 32 + (tid & 31);
  const int H = a.H, h = blockIdx.y, z = blockIdx.z;
  const int col0 = blockIdx.x * TBV;
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;

  // ---- the run ----------------------------------------------------------------------
  int64_t r0, r1, chunk_base = 0, xbase;
  int b = 0, s = 0, state_idx;
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
  // the run's dht / dh0 state, [N, H, K, V] or [B, H, nseg, K, V] for segments
  const int64_t soff =
      (a.nseg > 0 ? ((int64_t)b * H + h) * a.nseg + s : (int64_t)state_idx * H + h) * GDN_DK * GDN_DV;

  if (warp == 0) {
    tmem_alloc(&st.tmem, TMEM_COLS);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&st.bar_dv, 1);
    mbar_init(&st.bar_dh, 1);
    mbar_init(&st.bar_d0, 1);
    mbar_init(&st.bar_ld[0], 1);
    mbar_init(&st.bar_ld[1], 1);
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

  // ---- loader: round p takes chunk nch-1-p, into buffer p&1 ---------------------------------
  int64_t last_ld[2] = {-1, -1};
  auto issue_loads = [&](int64_t p) {
    const int64_t c = nch - 1 - p;
    const int par = (int)(p & 1);
    const uint8_t *blob = a.blob + (size_t)((xbase + c) * H + h) * BLOB_BYTES;
    const uint32_t dst = sb + (uint32_t)par * BUF_BYTES;
    uint64_t *bar = &st.bar_ld[par];
    mbar_expect_tx_w(bar, 32768 + 16384 + 8192 + 8192 + 512);
    bulk_load_w(dst + BUF_WQ, blob + BLOB_WQ, 32768, bar);
    bulk_load_w(dst + BUF_KL, blob + BLOB_KL, 16384, bar);
    bulk_load_w(dst + BUF_AQ, blob + BLOB_AQ, 8192, bar);
    bulk_load_w(dst + BUF_EL, blob + BLOB_EL, 512, bar);
    tma_load_2d_w(dst + BUF_DO, &maps.dO, h * GDN_DV + col0, (int)(r0 + c * GDN_CHUNK), bar);
    last_ld[par] = p;
  };

  // ---- state warps -----------------------------------------------------------------------
  float dh[32];
  if (!loader) {
    const float *src = a.dht ? a.dht + soff + (int64_t)row * GDN_DV + col0 + 32 * hc : nullptr;
#pragma unroll
    for (int j = 0; j < 32; ++j) dh[j] = src ? src[j] : 0.f;
  }
  auto write_dh = [&]() {  // bf16 copy: key `row`, columns 32 hc .. +31
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8)
      *reinterpret_cast<uint4 *>(sm + OFF_DH + chunk_off(row, 4 * hc + q8)) = pack8(dh + 8 * q8);
  };
  auto round = [&](int64_t p) {
    const int64_t c = nch - 1 - p;
    const int par = (int)(p & 1);
    const uint32_t buf = sb + (uint32_t)par * BUF_BYTES;
    uint8_t *bufp = sm + (size_t)par * BUF_BYTES;
    const int64_t c0 = r0 + c * GDN_CHUNK;
    const int n = (int)min((int64_t)GDN_CHUNK, r1 - c0);
    {  // gradient of this chunk's exit state
      const int64_t slot = a.cu ? (chunk_base + c) * H + h : ((int64_t)b * H + h) * NT + chunk_base + c;
      float4 *dst = reinterpret_cast<float4 *>(a.dh_chunks + slot * GDN_DK * GDN_DV + (int64_t)row * GDN_DV +
                                               col0 + 32 * hc);
#pragma unroll
      for (int g4 = 0; g4 < 8; ++g4) dst[g4] = make_float4(dh[g4 * 4], dh[g4 * 4 + 1], dh[g4 * 4 + 2], dh[g4 * 4 + 3]);
    }
    wait_par(&st.bar_ld[par], p >> 1);
    if (n < GDN_CHUNK) {  // dO rows past the run end: zero
      const int ltid = tid;  // 0 .. 255
      for (int e = ltid; e < (GDN_CHUNK - n) * 8; e += 256) {
        const int r = n + e / 8, c8 = e % 8;
        *reinterpret_cast<uint4 *>(bufp + BUF_DO + chunk_off(r, c8)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    chain_sync();
    if (warp == 0) {  // dv_new = KL dh + A_qk^T dO
      fence_after_sync();
      mma_ops_w(tmem + T_DV, kmaj(buf + BUF_KL, 8192), mnmaj(sb + OFF_DH, 0), 128,
                idesc_bf16(128, 64, false, false, true), false);
      mma_ops_w(tmem + T_DV, mnmaj(buf + BUF_AQ, 8192), mnmaj(buf + BUF_DO, 0), 64,
                idesc_bf16(128, 64, false, true, true), true);
      mma_commit_w(&st.bar_dv);
    }
    __syncwarp();
    if (q4 < 2) {  // token rows: dv_new to the workspace (fp32) and in bf16 for the next product
      wait_par(&st.bar_dv, p);
      const bool st_row = row < n;
      float *dvo = a.dvnew + ((c0 + (st_row ? row : 0)) * H + h) * GDN_DV + col0 + 32 * hc;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        float v[16];
        tmem_ld16(tl + T_DV + 32 * hc + 16 * part, v);
        tmem_ld_wait();
        if (st_row) {
          float4 *d4 = reinterpret_cast<float4 *>(dvo + 16 * part);
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) d4[g4] = make_float4(v[4 * g4], v[4 * g4 + 1], v[4 * g4 + 2], v[4 * g4 + 3]);
        }
        *reinterpret_cast<uint4 *>(sm + OFF_DV + chunk_off(row, 4 * hc + 2 * part)) = pack8(v);
        *reinterpret_cast<uint4 *>(sm + OFF_DV + chunk_off(row, 4 * hc + 2 * part + 1)) = pack8(v + 8);
      }
    }
    fence_proxy_async();
    fence_before_sync();
    chain_sync();
    if (warp == 0) {  // (scale Q b^G)^T dO - w^T dv_new, key rows
      fence_after_sync();
      mma_ops_w(tmem + T_DH, mnmaj(buf + BUF_WQ + 8192, 16384), mnmaj(buf + BUF_DO, 0), 64,
                idesc_bf16(128, 64, false, true, true), false);
      mma_ops_w(tmem + T_DH, mnmaj(buf + BUF_WQ, 16384), mnmaj(sb + OFF_DV, 0), 64,
                idesc_bf16(128, 64, true, true, true), true);
      mma_commit_w(&st.bar_dh);
    }
    __syncwarp();
    wait_par(&st.bar_dh, p);
    const float el = reinterpret_cast<const float *>(bufp + BUF_EL)[row];
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      float d[16];
      tmem_ld16(tl + T_DH + 32 * hc + 16 * part, d);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) dh[16 * part + j] = fmaf(el, dh[16 * part + j], d[j]);
    }
    write_dh();
    fence_proxy_async();
    fence_before_sync();
  };

  // ---- rounds ------------------------------------------------------------------------------
  // the blobs come from the prep kernel launched before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (loader && nch > 0) issue_loads(0);
  if (!loader) {
    write_dh();
    fence_proxy_async();
  }
  __syncthreads();
  for (int64_t p = 0; p < nch; ++p) {
    if (loader) {
      if (p + 1 < nch) issue_loads(p + 1);  // the buffer held round p-1, finished
    } else {
      round(p);
    }
    if (__syncthreads_or(bad)) {
      bad = true;
      break;
    }
  }
  if (bad) {
    if (tid == 0) raise_device_flag(a.dev_flag, kDevTimeout);
    if (warp == 0) mma_commit_w(&st.bar_d0);  // arrives once every MMA warp 0 issued is done
    if (warp == 0) mbar_wait(&st.bar_d0, 0, WAIT_LIMIT);
    if (loader)  // copies still in flight land before the CTA leaves
      for (int p2 = 0; p2 < 2; ++p2)
        if (last_ld[p2] >= 0) mbar_wait(&st.bar_ld[p2], (uint32_t)((last_ld[p2] >> 1) & 1), WAIT_LIMIT);
  } else if (!loader && a.dh0) {
    float4 *d4 = reinterpret_cast<float4 *>(a.dh0 + soff + (int64_t)row * GDN_DV + col0 + 32 * hc);
#pragma unroll
    for (int g4 = 0; g4 < 8; ++g4) d4[g4] = make_float4(dh[g4 * 4], dh[g4 * 4 + 1], dh[g4 * 4 + 2], dh[g4 * 4 + 3]);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

cudaError_t launch_kda_dhu(const BwdArgs &a, int runs, cudaStream_t st) {
  const uint64_t rows = a.cu ? (uint64_t)a.T : (uint64_t)a.B * a.T;
  DhuMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (rows == 0) return cudaSuccess;
  cudaError_t e = make_tmap_bf16(&maps.dO, a.dO, (uint64_t)a.H * GDN_DV, rows, (uint64_t)a.H * GDN_DV * 2);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kda_dhu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kda_dhu_kernel<<<dim3(GDN_DV / TBV, a.H, runs), NTH, SMEM_BYTES, st>>>(a, maps);
  return cudaGetLastError();
}

}  // namespace gdn
