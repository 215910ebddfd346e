// Internal launcher interface between the C ABI (gdn_api.cu) and the kernel
// translation units. Not installed; not part of the public header.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn.h"

namespace gdn {

// Opaque storage of a TMA tensor map (the driver's CUtensorMap: 128 bytes, 64-byte aligned).
struct alignas(64) TmaMap {
  unsigned char bytes[128];
};
// Map over a row-major bf16 matrix [rows][cols] (row pitch row_bytes) read in
// 64 x 64 boxes with the 128-byte swizzle; zero fill outside the matrix.
cudaError_t make_tmap_bf16(TmaMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes);
// Map over a row-major fp32 matrix [rows][128] read in 32-column x 128-row boxes with the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r mod 8) of the row's 128 bytes)
cudaError_t make_tmap_f32_32x128(TmaMap *map, const void *base, uint64_t rows);

// Rows of the per-chunk gate factor table written by the UT transform kernel
// (64 floats each, one per token t of the chunk, b(t) = t / 16 its 16-token block):
//   F_G    G_t (cumulative gate)            F_EG   base^G_t
//   F_EGL  base^(G_last - G_t)              F_BEG  beta_t base^G_t        F_BETA beta_t
//   F_EA   base^(G_t - G_{16 b(t)})         F_EB1 + b - 1  base^(G_{16 b} - G_t) for t < 16 b, else 0
// so that for tokens t > s in different blocks base^(G_t - G_s) = EA[t] EB_{b(t)}[s], a
// product of two factors that are both at most 1 for decaying gates.
enum GateTabRow { F_G = 0, F_EG, F_EGL, F_BEG, F_BETA, F_EA, F_EB1, F_EB2, F_EB3, F_ROWS };
constexpr int F_TAB = F_ROWS * 64;  // floats per chunk and head
// block stride (floats) of a shared-memory table of the gates inside the four diagonal
// 16x16 blocks; 272 keeps column-wise reads free of bank conflicts
constexpr int GD_BLOCK = 272;

// Arguments of the fp32 SIMT chunk kernel (forward, correction run, segment
// summary and the backward's state recompute share it).
struct SimtFwdArgs {
  const void *q, *k, *v;
  const float *g;
  const void *beta;
  const float *h0;   // [N,H,K,V]; segment mode [B,H,nseg,K,V]
  void *o;           // nullable
  float *ht;         // nullable
  float *g_cumsum;   // nullable
  float *A;          // nullable, [rows,H,64]
  float *h_chunks;   // nullable entry states
  float *S_ext, *M;  // summary mode outputs
  int B, T, H;
  float scale;
  int use_exp2;
  const int32_t *cu;  // packed offsets (device) or nullptr
  int num_seqs;
  int num_chunks;     // packed: chunk slots of h_chunks (bounds check)
  int seg_len, nseg;  // segment runs when nseg > 0
  int summary;        // 1: columns [0,V) from v with zero start, [V,V+K) transfer from I
  const float *g_cum_in;  // nullable: read the cumulative gate instead of summing g
  const float *A_in;      // nullable: read X = (I + L)^-1 instead of solving
  const __nv_bfloat16 *xw;  // tensor-core path: [X diag(b); X diag(b e^G)] of every chunk, [slots, H, 128, 64] bf16
  const float *ftab;        // tensor-core path: gate factor table of every chunk, [slots, H, F_TAB]
  // nullable: the entry state of every chunk in bf16, as the backward's local kernel reads it:
  // per (chunk slot, head) a [128 keys x 128 values] tile of two 64-column K-blocks (16 KB
  // each, 128-byte rows swizzled by key), slots as h_chunks
  __nv_bfloat16 *h_tiles;
  int *dev_flag;
};
// elements of one state tile (h_tiles, dh_tiles) and of one dv_new tile (dv_tiles)
constexpr int STATE_TILE = 128 * 128;
constexpr int DV_TILE = 64 * 128;

cudaError_t launch_simt_fwd(const SimtFwdArgs &a, bool per_key, bool bf16, dim3 grid,
                            cudaStream_t st);
int simt_fwd_bv();  // value columns per CTA

// UT transform of every chunk (bf16 keys, scalar gate): X = (I + L)^-1 in bf16
// as the pair [X diag(beta); X diag(beta base^G)] into xw [slots, H, 128, 64];
// optionally the fp32 X (A) and the cumulative gate.
struct UtArgs {
  const void *k;
  const float *g;         // raw gate, or
  const float *g_cum_in;  // the saved cumulative gate (nullable)
  const void *beta;
  __nv_bfloat16 *xw;
  float *ftab;      // per chunk and head: the gate factor table (F_TAB floats, GateTabRow)
  float *A;         // nullable, [rows, H, 64]
  float *g_cumsum;  // nullable
  int T, H;
  int use_exp2;
  const int32_t *cu, *chunk_indices;  // packed documents, or nullptr
  int num_seqs;
  int *dev_flag;
};
cudaError_t launch_ut(const UtArgs &a, int slots, cudaStream_t st);
// The same X pair and gate tables from a saved X (the forward's A slot, fp32 [rows, H, 64]) and
// the saved cumulative gate (a.g_cum_in): the backward's recompute, without a second solve
cudaError_t launch_ut_pair(const UtArgs &a, const float *A, int slots, cudaStream_t st);

// tcgen05 chunk forward with the state recurrence overlapped with the next
// chunk's preparation; reads X from a.xw (launch_ut first)
cudaError_t launch_tc_fwd_ws(const SimtFwdArgs &a, dim3 grid, cudaStream_t st);
int tc_fwd_ws_bv();

// Ordered merge of segment summaries. adjoint = 0: S_init_0 = h0, S_init_{s+1} = M_s S_init_s
// + S_ext_s, ht the state after the last segment. adjoint = 1 (the backward): the gradient
// runs from the last segment to the first through M^T: S_init receives every segment's exit
// gradient (dS_exit_{nseg-1} = h0 = dht), S_ext holds the backward summaries, ht receives dh0.
struct MergeArgs {
  const float *S_ext, *M, *h0;
  float *S_init, *ht;
  int BH, nseg;
  int adjoint;
  int *dev_flag;
};
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t st);

// Dense per-token transition scan (frame_scan.cu). Inputs [BH, T, D, D] (u_z [BH, T, D]);
// nseg = 1: one pass per sequence from S0 / z0; nseg > 1: summary, merge and seeded scan
// over segments of seg_len positions, with h_kv, M_kv, M_z, S_init [BH, nseg, D, D] and
// h_z, z_init [BH, nseg, D] in the workspace.
struct FrameScanArgs {
  const float *W_kv, *U_kv, *W_z, *u_z;
  const float *S0, *z0;                 // nullable initial states
  float *S_all, *z_all, *S_last, *z_last;
  float *h_kv, *M_kv, *h_z, *M_z, *S_init, *z_init;
  int BH, D, active, nseg;
  int64_t T, seg_len;
  int *dev_flag;
};
cudaError_t launch_frame_scan(const FrameScanArgs &a, cudaStream_t st);

// Backward: reverse state recurrence (dhu) and local gradients.
struct BwdArgs {
  const void *q, *k, *v, *beta, *dO;
  const float *g_cumsum, *A, *dht;
  void *dq, *dk, *dv, *dbeta;
  float *dg, *dh0;
  const float *h_chunks;  // workspace: entry state of every chunk
  float *dh_chunks;       // workspace: gradient of every chunk's exit state
  float *dvnew;           // workspace: [rows,H,V] gradient of v_new
  const __nv_bfloat16 *xw;  // tensor-core path: the X pair of every chunk (UT transform kernel)
  const float *ftab;        // tensor-core path: gate factor table of every chunk
  int B, T, H;
  float scale;
  int use_exp2;
  const int32_t *cu;
  const int32_t *chunk_indices;
  int num_seqs, num_chunks;
  int seg_len, nseg;  // segment runs when nseg > 0: dht / dh0 are [B, H, nseg, K, V]
  // bf16 tensor-core backward: the states, exit-state gradients and dv_new as bf16 tiles in
  // the local kernel's shared-memory layout (per chunk slot and head: h and dh [128 x 128] as two
  // 64-column K-blocks, dv_new [64 tokens x 128] likewise), replacing h_chunks, dh_chunks, dvnew
  const __nv_bfloat16 *h_tiles;
  __nv_bfloat16 *dh_tiles, *dv_tiles;
  // bf16 per-key backward: the prep kernel's blobs of every chunk (kda:: layout)
  const uint8_t *blob;
  int *dev_flag;
};
cudaError_t launch_bwd_dhu(const BwdArgs &a, bool per_key, bool bf16, cudaStream_t st);
cudaError_t launch_bwd_local(const BwdArgs &a, bool per_key, bool bf16, cudaStream_t st);
// local gradients on bf16 tensor cores (mma.sync), bf16 inputs with a scalar gate
cudaError_t launch_bwd_local_tc(const BwdArgs &a, cudaStream_t st);
// tcgen05 reverse state recurrence (bf16, scalar gate); needs a.xw / a.ftab
cudaError_t launch_tc_dhu(const BwdArgs &a, int runs, cudaStream_t st);
// tcgen05 reverse state recurrence (bf16, per-key gate) over the prep blobs; needs a.blob
cudaError_t launch_kda_dhu(const BwdArgs &a, int runs, cudaStream_t st);

// ---- per-key (KDA) tensor-core path ----------------------------------------------------
// The prep kernel writes, for every (chunk, head), one blob of bf16 tiles already in the
// 128-byte-swizzled shared-memory layout of the chain kernel's operands, so that the chain
// kernel fetches each with one bulk copy (G = in-chunk cumulative per-key gate, b the base):
namespace kda {
constexpr int BLOB_WQ = 0;      // [w; scale Q b^G] (128 rows x 128 keys, K-major: two K-blocks
                                //  16 KB apart, each the 64 w rows then the 64 Q rows)
constexpr int BLOB_KL = 32768;  // K b^(G_last - G): 64 token rows, two 64-key groups 8 KB apart
constexpr int BLOB_U = 49152;   // u = X diag(beta) V: 64 token rows, two 64-column halves
constexpr int BLOB_AQ = 65536;  // scale A_qk: 64 x 64, K-major
constexpr int BLOB_EL = 73728;  // b^(G_last) per key, fp32 [128]
constexpr int BLOB_BYTES = 74240;
}  // namespace kda

struct KdaPrepArgs {
  const void *q, *k, *v, *beta;  // bf16
  const float *g;                // raw per-key gate [rows, H, K], or
  const float *g_cum_in;         // the saved cumulative gate (nullable)
  uint8_t *blob;                 // [slots * H][BLOB_BYTES]
  float *g_cumsum, *A;           // nullable outputs
  int T, H;
  float scale;
  int use_exp2;
  const int32_t *cu, *chunk_indices;  // packed documents, or nullptr
  int num_seqs;
  int no_q;         // 1: q is not given (segment summary): the Q tile and A_qk are not written
  int scalar_gate;  // 1: g is one gate per (token, head), the same for every key channel
  int *dev_flag;
};
cudaError_t launch_kda_prep(const KdaPrepArgs &a, int slots, cudaStream_t st);

// Chain kernel over the blobs: the state recurrence and the output (forward, correction
// run), or the segment summary's [V | I] recurrence (summary = 1: grid x = 4 column slices).
struct KdaChainArgs {
  const uint8_t *blob;
  const float *h0;  // [N,H,K,V]; segment mode [B,H,nseg,K,V]
  __nv_bfloat16 *o;
  float *ht, *h_chunks;
  float *S_ext, *M;  // summary mode outputs
  int B, T, H;
  const int32_t *cu;
  int num_seqs, num_chunks;
  int seg_len, nseg;
  int summary;
  int *dev_flag;
};
cudaError_t launch_kda_chain(const KdaChainArgs &a, dim3 grid, cudaStream_t st);

// The optional input maps (q, k L2 norm; beta sigmoid) before the chunk kernels, and their
// chain rules after the backward (in place on dq, dk, dbeta).
struct InputMapArgs {
  const void *q, *k, *beta;  // raw inputs (q may be null: maps k only)
  void *qn, *kn, *beta_eff;  // prologue outputs
  void *dq, *dk, *dbeta;     // epilogue: gradients w.r.t. the mapped inputs, replaced in place
  int64_t rows;              // (token, head) rows
  int l2norm, beta_sigmoid;
};
cudaError_t launch_input_maps(const InputMapArgs &a, bool bf16, bool backward, cudaStream_t st);

// One CTA waits, with the kernels' bounded wait and `polls` polls, on an mbarrier that
// nothing arrives on, then raises the timeout flag (self-test of the wait path).
cudaError_t launch_wait_selftest(uint32_t polls, int *flag, cudaStream_t st);

}  // namespace gdn

namespace gdn {
// Records `msg` for gdn_last_error() in the calling thread and returns `st`.
gdn_status set_error(gdn_status st, const char *msg);
}  // namespace gdn
