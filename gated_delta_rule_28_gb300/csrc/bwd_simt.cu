// fp32 SIMT backward of the chunked gated delta rule (sm_103a).
//
// Three stages, as the pages' backward is staged (KDA adapter backward on the
// hyper-parallel "Diff Coverage" page: bwd_prepare -> bwd_dhu -> bwd_finalize;
// the GDN adapter's chunk_gated_delta_rule_bwd consumes q, k, v, g_cumsum,
// beta, A and dO):
//  1. entry state h_c of every chunk, recomputed by the forward chunk kernel
//     from the saved g_cumsum and A (launched by the API, not here);
//  2. dhu: the reverse state recurrence, per (run, head, 32 state columns),
//        dv_new_c = kgl_c dh_{c+1} + scale A_qk^T dO_c
//        dh_c     = Diag(base^G_last) dh_{c+1} + scale Qg^T dO_c - w_c^T dv_new_c
//     (the reverse loop of state_summary.py kda_state_grad_ext_kernel), with
//     w_c^T dv_new = Kg^T beta (X^T dv_new); it stores dh_{c+1} per chunk and
//     dv_new, and returns dh_0;
//  3. local: per (chunk, head), with the whole value width, the adjoint of the
//     chunk's UT transform, gates and Gram matrices, giving dq, dk, dv, dbeta
//     and dg (reverse in-chunk cumulative sum: the gradient of the raw gate).
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int NTH = 256;
constexpr int KP = GDN_DK + 1;
constexpr int CP = GDN_CHUNK + 1;

// ---------------------------------------------------------------------------
// run / chunk bookkeeping shared by both kernels
struct Run {
  int64_t r0, r1, chunk_base;
  int state_idx, b, s;
  bool ok;
};

__device__ Run run_of(const BwdArgs &a, int z) {
  Run r{};
  r.ok = true;
  if (a.cu) {
    r.r0 = a.cu[z];
    r.r1 = a.cu[z + 1];
    r.ok = r.r0 >= 0 && r.r1 > r.r0 && r.r1 <= a.T;
    r.chunk_base = 0;
    if (r.ok) {
      for (int m = 0; m < z; ++m) r.chunk_base += (a.cu[m + 1] - a.cu[m] + GDN_CHUNK - 1) / GDN_CHUNK;
      r.ok = r.chunk_base + (r.r1 - r.r0 + GDN_CHUNK - 1) / GDN_CHUNK <= a.num_chunks;
    }
    r.state_idx = z;
    r.b = 0;
  } else if (a.nseg > 0) {  // segment s of batch row b
    r.b = z / a.nseg;
    r.s = z % a.nseg;
    r.r0 = (int64_t)r.b * a.T + (int64_t)r.s * a.seg_len;
    r.r1 = min(r.r0 + a.seg_len, (int64_t)r.b * a.T + a.T);
    r.chunk_base = (int64_t)r.s * a.seg_len / GDN_CHUNK;
    r.state_idx = r.b;
  } else {
    r.b = z;
    r.r0 = (int64_t)z * a.T;
    r.r1 = r.r0 + a.T;
    r.chunk_base = 0;
    r.state_idx = z;
  }
  return r;
}

__device__ __forceinline__ int64_t chunk_slot(const BwdArgs &a, const Run &r, int64_t ci, int h) {
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
  return a.cu ? (r.chunk_base + ci) * a.H + h : ((int64_t)r.b * a.H + h) * NT + r.chunk_base + ci;
}

// element offset of the run's dht / dh0 state: [N, H, K, V], or [B, H, nseg, K, V] for segments
__device__ __forceinline__ int64_t state_off(const BwdArgs &a, const Run &r, int h) {
  const int64_t slot = a.nseg > 0 ? ((int64_t)r.b * a.H + h) * a.nseg + r.s : (int64_t)r.state_idx * a.H + h;
  return slot * GDN_DK * GDN_DV;
}

// ---------------------------------------------------------------------------
// dhu: reverse state recurrence
constexpr int DBV = 32;
constexpr int DVP = DBV + 1;

template <bool PER_KEY>
constexpr size_t dhu_smem_floats() {
  return 3 * 64 * KP + (PER_KEY ? 64 * KP : 3 * 64) + 2 * 64 * CP + 128 * DVP + 3 * 64 * DVP + 64 + 128;
}

template <typename T, bool PER_KEY>
__global__ void __launch_bounds__(NTH) dhu_kernel(BwdArgs a) {
  extern __shared__ float smem[];
  float *sKl = smem;                        // K (.) base^(G_last - G)
  float *sQg = sKl + 64 * KP;               // scale Q (.) base^G
  float *sKg = sQg + 64 * KP;               // K (.) base^G
  float *sG = sKg + 64 * KP;                // cumulative gate (scalar gate: + e^G, e^(Gl-G))
  float *sX = sG + (PER_KEY ? 64 * KP : 3 * 64);
  float *sAqk = sX + 64 * CP;
  float *sDH = sAqk + 64 * CP;              // [128][DVP]
  float *sDO = sDH + 128 * DVP;             // [64][DVP]
  float *sDD = sDO + 64 * DVP;              // dv_new slice
  float *sDY = sDD + 64 * DVP;              // -beta X^T dv_new
  float *sBeta = sDY + 64 * DVP;
  float *sEL = sBeta + 64;

  const int tid = threadIdx.x, H = a.H, h = blockIdx.y, z = blockIdx.z;
  const int col0 = blockIdx.x * DBV;
  const bool e2 = a.use_exp2 != 0;
  const T *q = static_cast<const T *>(a.q);
  const T *k = static_cast<const T *>(a.k);
  const T *beta = static_cast<const T *>(a.beta);
  const T *dO = static_cast<const T *>(a.dO);
  const Run run = run_of(a, z);
  if (!run.ok) {
    if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
    return;
  }
  const int64_t KV = (int64_t)GDN_DK * GDN_DV;
  for (int idx = tid; idx < 128 * DBV; idx += NTH) {
    const int d = idx / DBV, c = idx % DBV;
    sDH[d * DVP + c] = a.dht ? a.dht[state_off(a, run, h) + d * GDN_DV + col0 + c] : 0.f;
  }
  __syncthreads();
  const int64_t nchunks = (run.r1 - run.r0 + GDN_CHUNK - 1) / GDN_CHUNK;
  for (int64_t ci = nchunks - 1; ci >= 0; --ci) {
    const int64_t c0 = run.r0 + ci * GDN_CHUNK;
    const int n = (int)min((int64_t)GDN_CHUNK, run.r1 - c0);
    {  // gradient of this chunk's exit state
      float *dst = a.dh_chunks + chunk_slot(a, run, ci, h) * KV;
      for (int idx = tid; idx < 128 * DBV; idx += NTH) {
        const int d = idx / DBV, c = idx % DBV;
        dst[d * GDN_DV + col0 + c] = sDH[d * DVP + c];
      }
    }
    for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
      const int i = idx >> 7, d = idx & 127;
      float kv = 0.f, qv = 0.f, gv = 0.f;
      if (i < n) {
        const int64_t off = ((c0 + i) * H + h) * GDN_DK + d;
        kv = to_f32(k[off]);
        qv = to_f32(q[off]);
        if (PER_KEY) gv = a.g_cumsum[off];
      }
      sKl[i * KP + d] = kv;
      sQg[i * KP + d] = qv;
      if (PER_KEY) sG[i * KP + d] = gv;
    }
    for (int idx = tid; idx < 64 * DBV; idx += NTH) {
      const int i = idx / DBV, c = idx % DBV;
      sDO[i * DVP + c] = i < n ? to_f32(dO[((c0 + i) * H + h) * GDN_DV + col0 + c]) : 0.f;
    }
    for (int idx = tid; idx < 64 * 64; idx += NTH) {
      const int i = idx >> 6, j = idx & 63;
      sX[i * CP + j] = (i < n && j < n) ? a.A[((c0 + i) * H + h) * GDN_CHUNK + j] : (i == j ? 1.f : 0.f);
    }
    if (tid < 64) {
      sBeta[tid] = tid < n ? to_f32(beta[(c0 + tid) * H + h]) : 0.f;
      if (!PER_KEY) sG[tid] = a.g_cumsum[(c0 + min(tid, n - 1)) * H + h];
    }
    __syncthreads();
    if (PER_KEY) {  // rows past the end hold the last valid cumulative gate
      for (int idx = tid; idx < (64 - n) * GDN_DK; idx += NTH) {
        const int i = n + idx / GDN_DK, d = idx % GDN_DK;
        sG[i * KP + d] = sG[(n - 1) * KP + d];
      }
      __syncthreads();
    }
    // A_qk = lower-incl(Q K^T (.) Gamma)
    {
      int m0, n0;
      tile_origin<64, 64, 4, 4>(tid, m0, n0);
      float acc[4][4];
      zero_acc(acc);
      if (n0 <= m0 + 3) {
        if (PER_KEY) {
          for (int d = 0; d < GDN_DK; ++d) {
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                if (n0 + y > m0 + x) continue;
                acc[x][y] = fmaf(sQg[(m0 + x) * KP + d] * sKl[(n0 + y) * KP + d],
                                 gate_pow(sG[(m0 + x) * KP + d] - sG[(n0 + y) * KP + d], e2), acc[x][y]);
              }
          }
        } else {
          auto fq = [&](int m, int kk) { return sQg[m * KP + kk]; };
          auto fkt = [&](int kk, int nn) { return sKl[nn * KP + kk]; };
          mm_acc<64, 64, GDN_DK, 4, 4>(fq, fkt, acc, tid);
#pragma unroll
          for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) acc[x][y] *= gate_pow(sG[m0 + x] - sG[n0 + y], e2);
        }
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) sAqk[(m0 + x) * CP + n0 + y] = (n0 + y <= m0 + x) ? acc[x][y] : 0.f;
    }
    if (!PER_KEY && tid < 64) {  // per-token gate factors (scalar gate)
      sG[64 + tid] = gate_pow(sG[tid], e2);
      sG[128 + tid] = gate_pow(sG[63] - sG[tid], e2);
    }
    __syncthreads();
    for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
      const int i = idx >> 7, d = idx & 127;
      const float Gi = PER_KEY ? sG[i * KP + d] : sG[i];
      const float Gl = PER_KEY ? sG[63 * KP + d] : sG[63];
      const float kk = sKl[i * KP + d];
      const float eg = PER_KEY ? gate_pow(Gi, e2) : sG[64 + i];
      const float egl = PER_KEY ? gate_pow(Gl - Gi, e2) : sG[128 + i];
      sKg[i * KP + d] = kk * eg;
      sQg[i * KP + d] *= a.scale * eg;
      sKl[i * KP + d] = kk * egl;
    }
    if (tid < GDN_DK) sEL[tid] = gate_pow(PER_KEY ? sG[63 * KP + tid] : sG[63], e2);
    __syncthreads();
    // dv_new = kgl dh + scale A_qk^T dO
    {
      float acc[2][4];
      zero_acc(acc);
      auto fa = [&](int m, int kk) { return sKl[m * KP + kk]; };
      auto fb = [&](int kk, int nn) { return sDH[kk * DVP + nn]; };
      mm_acc<64, DBV, GDN_DK, 2, 4>(fa, fb, acc, tid);
      float acc2[2][4];
      zero_acc(acc2);
      auto fa2 = [&](int m, int kk) { return sAqk[kk * CP + m]; };
      auto fb2 = [&](int kk, int nn) { return sDO[kk * DVP + nn]; };
      mm_acc<64, DBV, GDN_CHUNK, 2, 4>(fa2, fb2, acc2, tid);
      int m0, n0;
      tile_origin<64, DBV, 2, 4>(tid, m0, n0);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const float val = acc[x][y] + a.scale * acc2[x][y];
          sDD[(m0 + x) * DVP + n0 + y] = val;
          if (m0 + x < n) a.dvnew[((c0 + m0 + x) * H + h) * GDN_DV + col0 + n0 + y] = val;
        }
    }
    __syncthreads();
    // dY = -beta (X^T dv_new)
    {
      float acc[2][4];
      zero_acc(acc);
      auto fa = [&](int m, int kk) { return sX[kk * CP + m]; };
      auto fb = [&](int kk, int nn) { return sDD[kk * DVP + nn]; };
      mm_acc<64, DBV, GDN_CHUNK, 2, 4>(fa, fb, acc, tid);
      int m0, n0;
      tile_origin<64, DBV, 2, 4>(tid, m0, n0);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) sDY[(m0 + x) * DVP + n0 + y] = -sBeta[m0 + x] * acc[x][y];
    }
    __syncthreads();
    // dh <- Diag(base^G_last) dh + Qg^T dO + Kg^T dY
    {
      float acc[4][4];
      zero_acc(acc);
      auto fa = [&](int m, int kk) { return sQg[kk * KP + m]; };
      auto fb = [&](int kk, int nn) { return sDO[kk * DVP + nn]; };
      mm_acc<128, DBV, GDN_CHUNK, 4, 4>(fa, fb, acc, tid);
      auto fa2 = [&](int m, int kk) { return sKg[kk * KP + m]; };
      auto fb2 = [&](int kk, int nn) { return sDY[kk * DVP + nn]; };
      mm_acc<128, DBV, GDN_CHUNK, 4, 4>(fa2, fb2, acc, tid);
      int m0, n0;
      tile_origin<128, DBV, 4, 4>(tid, m0, n0);
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          float &dh = sDH[(m0 + x) * DVP + n0 + y];
          dh = fmaf(sEL[m0 + x], dh, acc[x][y]);
        }
    }
    __syncthreads();
  }
  if (a.dh0) {
    for (int idx = tid; idx < 128 * DBV; idx += NTH) {
      const int d = idx / DBV, c = idx % DBV;
      a.dh0[state_off(a, run, h) + d * GDN_DV + col0 + c] = sDH[d * DVP + c];
    }
  }
}

// ---------------------------------------------------------------------------
// 16-byte global loads (every operand row and the slices within it start on 16 bytes):
// 8 bf16 or 4 fp32 values per load. The local kernel issues all of a phase's loads before
// its first shared-memory store, so that one memory round trip covers the phase.
__device__ __forceinline__ uint4 ld16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
template <typename T>
__device__ __forceinline__ float lane16(const uint4 &u, int e) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  if constexpr (std::is_same<T, float>::value) {
    return __uint_as_float(w[e]);
  } else {
    const uint32_t x = w[e >> 1];
    return __uint_as_float((e & 1) ? (x & 0xffff0000u) : (x << 16));
  }
}

// ---------------------------------------------------------------------------
// local gradients, one CTA per (chunk, head), the value width in 8 slices
constexpr int LBV = 16;

// Row strides (floats) of the local kernel's shared-memory matrices, and its value-slice
// width. The FMA path (fp32 inputs) pads rows by one float. The tensor-core path (bf16
// inputs, per-key gate; a scalar gate with bf16 inputs runs on local_tc) reads mma
// fragments, lane (g, t) at row g and column t (or transposed), so its strides are 4 mod 32:
// the row-major fragment reads then hit 32 distinct banks, the transposed ones at most two
// lanes per bank. It also keeps a region of xtra floats after A_qk's, so that A_qk's region
// with it, and it with X's, each hold one 64 x 128 operand tile while A_qk's or X's
// contents are not in use.
template <typename T, bool PER_KEY>
struct LocalStrides {
  static constexpr bool tc = !std::is_same<T, float>::value;
  static_assert(!tc || PER_KEY, "bf16 inputs with a scalar gate run on local_tc");
  static constexpr int kp = tc ? GDN_DK + 4 : GDN_DK + 1;
  static constexpr int cp = tc ? GDN_CHUNK + 4 : GDN_CHUNK + 1;
  static constexpr int lbv = LBV;
  static constexpr int lvp = tc ? lbv + 4 : lbv + 1;
  static constexpr int xtra = tc ? 64 * kp - 64 * cp + 128 : 0;
};

template <typename T, bool PER_KEY>
constexpr size_t local_smem_floats() {
  // K, Q, (G), P, Aqk, (extra), X, slice buffers, beta, dbeta, EL, dGLh, dGlast, dGrow, ...
  using S = LocalStrides<T, PER_KEY>;
  return 2 * 64 * S::kp + (PER_KEY ? 64 * S::kp : 3 * 64) + 3 * 64 * S::cp + S::xtra +
         (2 * 128 * S::lvp + 6 * 64 * S::lvp) + 64 + 64 + 128 + 128 + 128 + 64 + 3 * 64 + 8 * 128 + 8;
}

template <typename T, bool PER_KEY>
__global__ void __launch_bounds__(NTH, 1) local_kernel(BwdArgs a) {
  // this kernel's strides and slice width (hide the namespace-scope ones)
  using LS = LocalStrides<T, PER_KEY>;
  constexpr int KP = LS::kp, CP = LS::cp, LBV = LS::lbv, LVP = LS::lvp;
  extern __shared__ float smem[];
  float *sK = smem;
  float *sQ = sK + 64 * KP;
  float *sG = sQ + 64 * KP;  // cumulative gate (scalar gate: + e^G, e^(Gl-G))
  float *sP = sG + (PER_KEY ? 64 * KP : 3 * 64);  // gated K K^T (strict lower), later dP (.) Gamma
  float *sAqk = sP + 64 * CP;   // dA_qk (.) Gamma (after the value pass)
  float *sX = sAqk + 64 * CP + LS::xtra;
  float *sSl = sX + 64 * CP;    // slice region
  // tensor-core path: 64 x 128 operand tiles over A_qk's region and the extra floats (the
  // Gram's right operand, then K (.) b^G during the value pass), and over the extra floats
  // and X's region (the Gram adjoints' right operands, once X is no longer read)
  float *sWideA = sAqk, *sWideB = sAqk + 64 * CP;
  float *sHs = sSl;                  // [128][LVP] h slice
  float *sDHs = sHs + 128 * LVP;     // [128][LVP] dh_{c+1} slice
  float *sVs = sDHs + 128 * LVP;     // [64][LVP]
  float *sDOs = sVs + 64 * LVP;
  float *sDDs = sDOs + 64 * LVP;     // dv_new slice
  float *sZs = sDDs + 64 * LVP;      // beta (V - Kg h)
  float *sDels = sZs + 64 * LVP;     // v_new slice
  float *sDYs = sDels + 64 * LVP;    // -beta X^T dv_new
  float *sBeta = sSl + 2 * 128 * LVP + 6 * 64 * LVP;
  float *sDBeta = sBeta + 64;
  float *sEL = sDBeta + 64;
  float *sDGLh = sEL + 128;   // sum_c dh_{c+1} (.) h per key channel
  float *sDGlast = sDGLh + 128;
  float *sDGrow = sDGlast + 128;
  // partial sums, each slot with one writer and summed in a fixed order, so that the
  // gradients do not depend on the order threads arrive in (no shared-memory atomics)
  float *sDBpart = sDGrow + 64;      // [3][64]: dbeta from the two column halves, and from dL
  float *sGlPart = sDBpart + 3 * 64;  // [8 warps][128]: dG_last per key channel
  float *sRowX = sGlPart + 8 * 128;   // [4 warps]: the G_last term of the scalar gate

  const int tid = threadIdx.x, H = a.H, h = blockIdx.y;
  const int64_t zc = blockIdx.x;
  const bool e2 = a.use_exp2 != 0;
  const float lnb = e2 ? 0.69314718055994530942f : 1.f;
  const T *q = static_cast<const T *>(a.q);
  const T *k = static_cast<const T *>(a.k);
  const T *v = static_cast<const T *>(a.v);
  const T *beta = static_cast<const T *>(a.beta);
  const T *dO = static_cast<const T *>(a.dO);
  T *dq = static_cast<T *>(a.dq);
  T *dk = static_cast<T *>(a.dk);
  T *dv = static_cast<T *>(a.dv);
  T *dbeta = static_cast<T *>(a.dbeta);

  // ---- locate the chunk --------------------------------------------------
  int64_t c0, slot;
  int n;
  if (a.cu) {
    const int seq = a.chunk_indices[2 * zc], cc = a.chunk_indices[2 * zc + 1];
    bool ok = seq >= 0 && seq < a.num_seqs && cc >= 0;
    if (ok) {
      c0 = a.cu[seq] + (int64_t)cc * GDN_CHUNK;
      ok = c0 < a.cu[seq + 1] && a.cu[seq + 1] <= a.T;
      n = ok ? (int)min((int64_t)GDN_CHUNK, (int64_t)a.cu[seq + 1] - c0) : 0;
    }
    if (!ok) {
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      return;
    }
    slot = zc * H + h;
  } else {
    const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
    const int b = (int)(zc / NT), cc = (int)(zc % NT);
    c0 = (int64_t)b * a.T + (int64_t)cc * GDN_CHUNK;
    n = min(GDN_CHUNK, a.T - cc * GDN_CHUNK);
    slot = ((int64_t)b * H + h) * NT + cc;
  }
  const int64_t KV = (int64_t)GDN_DK * GDN_DV;
  const float *hc = a.h_chunks + slot * KV;
  const float *dhc = a.dh_chunks + slot * KV;

  // ---- chunk operands (16-byte loads, all issued before the first store) ---------
  float bet = 0.f, gsc = 0.f;  // beta and (scalar gate) the cumulative gate of token tid
  {
    constexpr int EV = 16 / sizeof(T);               // q, k values per load
    constexpr int NV = 64 * GDN_DK / EV / NTH;        // loads per thread and operand
    constexpr int NG = PER_KEY ? 64 * GDN_DK / 4 / NTH : 1;
    uint4 kr[NV], qr[NV], gr[NG], xr[64 * GDN_CHUNK / 4 / NTH];
    const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int r = 0; r < NV; ++r) {
      const int idx = tid + r * NTH, i = idx / (GDN_DK / EV), d0 = idx % (GDN_DK / EV) * EV;
      const int64_t off = ((c0 + i) * H + h) * GDN_DK + d0;
      kr[r] = i < n ? ld16(k + off) : z4;
      qr[r] = i < n ? ld16(q + off) : z4;
    }
    if (PER_KEY) {
#pragma unroll
      for (int r = 0; r < NG; ++r) {
        const int idx = tid + r * NTH, i = idx / (GDN_DK / 4), d0 = idx % (GDN_DK / 4) * 4;
        gr[r] = i < n ? ld16(a.g_cumsum + ((c0 + i) * H + h) * GDN_DK + d0) : z4;
      }
    }
#pragma unroll
    for (int r = 0; r < 64 * GDN_CHUNK / 4 / NTH; ++r) {
      const int idx = tid + r * NTH, i = idx / (GDN_CHUNK / 4), j0 = idx % (GDN_CHUNK / 4) * 4;
      xr[r] = i < n ? ld16(a.A + ((c0 + i) * H + h) * GDN_CHUNK + j0) : z4;
    }
    if (tid < 64) {
      if (tid < n) bet = to_f32(beta[(c0 + tid) * H + h]);
      if (!PER_KEY) gsc = a.g_cumsum[(c0 + min(tid, n - 1)) * H + h];
    }
#pragma unroll
    for (int r = 0; r < NV; ++r) {
      const int idx = tid + r * NTH, i = idx / (GDN_DK / EV), d0 = idx % (GDN_DK / EV) * EV;
#pragma unroll
      for (int e = 0; e < EV; ++e) {
        sK[i * KP + d0 + e] = lane16<T>(kr[r], e);
        sQ[i * KP + d0 + e] = lane16<T>(qr[r], e);
      }
    }
    if (PER_KEY) {
#pragma unroll
      for (int r = 0; r < NG; ++r) {
        const int idx = tid + r * NTH, i = idx / (GDN_DK / 4), d0 = idx % (GDN_DK / 4) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) sG[i * KP + d0 + e] = lane16<float>(gr[r], e);
      }
    }
#pragma unroll
    for (int r = 0; r < 64 * GDN_CHUNK / 4 / NTH; ++r) {
      const int idx = tid + r * NTH, i = idx / (GDN_CHUNK / 4), j0 = idx % (GDN_CHUNK / 4) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + e;
        sX[i * CP + j] = (i < n && j < n) ? lane16<float>(xr[r], e) : (i == j ? 1.f : 0.f);
      }
    }
  }
  if (tid < 64) {
    sBeta[tid] = bet;
    sDBeta[tid] = 0.f;
    sDGrow[tid] = 0.f;
    sDBpart[tid] = sDBpart[64 + tid] = sDBpart[128 + tid] = 0.f;
    if (!PER_KEY) sG[tid] = gsc;
  }
  if (tid < 128) {
    sDGLh[tid] = 0.f;
    sDGlast[tid] = 0.f;
  }
  __syncthreads();
  if (PER_KEY) {
    for (int idx = tid; idx < (64 - n) * GDN_DK; idx += NTH) {
      const int i = n + idx / GDN_DK, d = idx % GDN_DK;
      sG[i * KP + d] = sG[(n - 1) * KP + d];
    }
    __syncthreads();
  }
  auto Gv = [&](int i, int d) { return PER_KEY ? sG[i * KP + d] : sG[i]; };
  if (tid < GDN_DK) sEL[tid] = gate_pow(Gv(63, tid), e2);
  if (!PER_KEY && tid >= 128 && tid < 192) {  // per-token gate factors (scalar gate)
    const int i = tid - 128;
    sG[64 + i] = gate_pow(sG[i], e2);
    sG[128 + i] = gate_pow(sG[63] - sG[i], e2);
  }
  // e^G and e^(G_last - G) of token i, key channel d
  auto EG = [&](int i, int d) { return PER_KEY ? gate_pow(sG[i * KP + d], e2) : sG[64 + i]; };
  auto EGL = [&](int i, int d) {
    return PER_KEY ? gate_pow(sG[63 * KP + d] - sG[i * KP + d], e2) : sG[128 + i];
  };

  // bf16 inputs: the chunk's dense contractions run on tf32 tensor cores (mma.sync), each warp
  // owning rows 16 (warp % 4) .. +15 and a quarter-width column block of an output; fp32
  // inputs keep the FMA path, whose error bound is tighter than tf32 rounding
  constexpr bool TC = !std::is_same<T, float>::value;
  const int wr0 = 16 * ((tid >> 5) & 3), lane = tid & 31;
  const int wc128 = 64 * (tid >> 7), wc64 = 32 * (tid >> 7);
  const int fg = lane >> 2, ft = lane & 3;  // this thread's fragment row / column pair

  // per-key gate on the tensor-core path: with one reference row r per chunk and
  // e_id = b^(G_id - G_rd), every gated product is a plain product of pre-scaled operands,
  //   sum_j M_ij x_jd b^(G_id - G_jd) = e_id sum_j M_ij (x_jd / e_jd),
  // each scaled operand formed once in shared memory; valid while every |G_id - G_rd| stays
  // within 100 in base 2 (the factors stay inside the fp32 range); a chunk beyond that takes
  // the term-by-term loops, exact for any gate range
  constexpr int REFR = 32;
  const float l2b = e2 ? 1.f : 1.4426950408889634f;
  bool fast = false;
  if constexpr (TC && PER_KEY) {
    const int d = tid & 127, r0 = 32 * (tid >> 7);
    const float gr = sG[REFR * KP + d];
    float span = 0.f;
    for (int i = r0; i < r0 + 32; ++i) span = fmaxf(span, fabsf(sG[i * KP + d] - gr));
    fast = !__syncthreads_or(!(span * l2b <= 100.f));
  }
  // b^x with one special-function instruction (PTX ex2.approx.ftz, relative error near 2^-22)
  auto bx = [&](float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * l2b));
    return y;
  };

  // ---- gated Gram matrix P = strictly-lower(K K^T (.) Gamma) ----------------------
  // (the gated Q K^T of the forward is not needed: dA_qk is formed from dO and v_new)
  {
    int m0, n0;
    tile_origin<64, 64, 4, 4>(tid, m0, n0);
    float accP[4][4];
    zero_acc(accP);
    bool in_tiles = true;
    {
      if constexpr (TC) {
        if (fast) {  // (K (.) e)(K / e)^T on tensor cores, fragments straight into sP
          float *tA = sSl, *tB = sWideA;  // [64][KP] each: K (.) e and K / e
          for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
            const int i = idx >> 7, d = idx & 127;
            const float kv = sK[i * KP + d], x = sG[i * KP + d] - sG[REFR * KP + d];
            tA[i * KP + d] = kv * bx(x);
            tB[i * KP + d] = kv * bx(-x);
          }
          __syncthreads();
          float fP[4][4];
          zero_acc(fP);
          auto fa = [&](int m, int kk) { return tA[m * KP + kk]; };
          auto fb = [&](int kk, int nn) { return tB[nn * KP + kk]; };
          mma_tf32_acc<GDN_DK, 4>(fa, fb, fP, wr0, wc64, lane);
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = wr0 + fg + 8 * (e >> 1), c = wc64 + 8 * j + 2 * ft + (e & 1);
              sP[i * CP + c] = c < i ? fP[j][e] : 0.f;
            }
          in_tiles = false;
        }
      }
      if (in_tiles && n0 <= m0 + 3) {
        if (PER_KEY) {
          for (int d = 0; d < GDN_DK; ++d) {
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                if (n0 + y > m0 + x) continue;
                const float gam = gate_pow(sG[(m0 + x) * KP + d] - sG[(n0 + y) * KP + d], e2);
                accP[x][y] = fmaf(sK[(m0 + x) * KP + d] * sK[(n0 + y) * KP + d], gam, accP[x][y]);
              }
          }
        } else {
          auto fk = [&](int m, int kk) { return sK[m * KP + kk]; };
          auto fkt = [&](int kk, int nn) { return sK[nn * KP + kk]; };
          mm_acc<64, 64, GDN_DK, 4, 4>(fk, fkt, accP, tid);
#pragma unroll
          for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) accP[x][y] *= gate_pow(sG[m0 + x] - sG[n0 + y], e2);
        }
      }
    }
    if (in_tiles) {
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int i = m0 + x, j = n0 + y;
          sP[i * CP + j] = j < i ? accP[x][y] : 0.f;
        }
    }
  }
  __syncthreads();
  if constexpr (TC) {  // K (.) b^G, the left operand of the value pass's state product
    for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
      const int i = idx >> 7, d = idx & 127;
      sWideA[i * KP + d] = sK[i * KP + d] * bx(sG[i * KP + d]);
    }
    // (the first slice's barrier orders these stores before the product reads them)
  }

  // ---- pass over value slices: accumulate the value contractions -----------
  // register tiles: 64x64 (4x4 per thread) and 64x128 (4x8 per thread)
  int pm0, pn0, gm0, gn0;
  tile_origin<64, 64, 4, 4>(tid, pm0, pn0);
  tile_origin<64, 128, 4, 8>(tid, gm0, gn0);
  float aX[4][4], aQk[4][4], aQg[4][8], aKg[4][8], aKl[4][8];
  zero_acc(aX);
  zero_acc(aQk);
  zero_acc(aQg);
  zero_acc(aKg);
  zero_acc(aKl);
  // tensor-core path: the five value contractions below accumulate as fragments, moved into
  // the thread tiles above after the pass
  float fQg[8][4], fKg[8][4], fKl[8][4], fX[4][4], fQk[4][4];
  zero_acc(fQg);
  zero_acc(fKg);
  zero_acc(fKl);
  zero_acc(fX);
  zero_acc(fQk);
  for (int vs = 0; vs < GDN_DV; vs += LBV) {
    {  // the slice: h, dh (128 x LBV), v, dO, dv_new (64 x LBV), 16-byte loads issued together
      constexpr int EV = 16 / sizeof(T);
      constexpr int NH = 128 * LBV / 4, NVv = 64 * LBV / EV, ND = 64 * LBV / 4;
      constexpr int RH = (NH + NTH - 1) / NTH, RV = (NVv + NTH - 1) / NTH, RD = (ND + NTH - 1) / NTH;
      uint4 hr[RH], dhr[RH], vr[RV], dor[RV], ddr[RD];
      const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        const int idx = tid + r * NTH, d = idx / (LBV / 4), cc = idx % (LBV / 4) * 4;
        if (idx < NH) {
          hr[r] = ld16(hc + d * GDN_DV + vs + cc);
          dhr[r] = ld16(dhc + d * GDN_DV + vs + cc);
        }
      }
#pragma unroll
      for (int r = 0; r < RV; ++r) {
        const int idx = tid + r * NTH, i = idx / (LBV / EV), cc = idx % (LBV / EV) * EV;
        const int64_t off = ((c0 + i) * H + h) * GDN_DV + vs + cc;
        vr[r] = (idx < NVv && i < n) ? ld16(v + off) : z4;
        dor[r] = (idx < NVv && i < n) ? ld16(dO + off) : z4;
      }
#pragma unroll
      for (int r = 0; r < RD; ++r) {
        const int idx = tid + r * NTH, i = idx / (LBV / 4), cc = idx % (LBV / 4) * 4;
        ddr[r] = (idx < ND && i < n) ? ld16(a.dvnew + ((c0 + i) * H + h) * GDN_DV + vs + cc) : z4;
      }
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        const int idx = tid + r * NTH, d = idx / (LBV / 4), cc = idx % (LBV / 4) * 4;
        if (idx < NH) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sHs[d * LVP + cc + e] = lane16<float>(hr[r], e);
            sDHs[d * LVP + cc + e] = lane16<float>(dhr[r], e);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RV; ++r) {
        const int idx = tid + r * NTH, i = idx / (LBV / EV), cc = idx % (LBV / EV) * EV;
        if (idx < NVv) {
#pragma unroll
          for (int e = 0; e < EV; ++e) {
            sVs[i * LVP + cc + e] = lane16<T>(vr[r], e);
            sDOs[i * LVP + cc + e] = lane16<T>(dor[r], e);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < RD; ++r) {
        const int idx = tid + r * NTH, i = idx / (LBV / 4), cc = idx % (LBV / 4) * 4;
        if (idx < ND) {
#pragma unroll
          for (int e = 0; e < 4; ++e) sDDs[i * LVP + cc + e] = lane16<float>(ddr[r], e);
        }
      }
    }
    __syncthreads();
    // Z = beta (V - (K (.) base^G) h) ; also keep V - Y for dbeta
    if constexpr (TC) {  // the 64 x LBV product on tensor cores, LBV/16 tiles per warp
      constexpr int NZ = LBV / 16;
      const int zr0 = 16 * ((tid >> 5) & 3), zc0 = (LBV / 2) * (tid >> 7);
      float fz[NZ][4];
      zero_acc(fz);
      auto fkg = [&](int m, int kk) { return sWideA[m * KP + kk]; };
      auto fhs = [&](int kk, int nn) { return sHs[kk * LVP + nn]; };
      mma_tf32_acc<GDN_DK, NZ>(fkg, fhs, fz, zr0, zc0, lane);
#pragma unroll
      for (int j = 0; j < NZ; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = zr0 + fg + 8 * (e >> 1), c = zc0 + 8 * j + 2 * ft + (e & 1);
          const float r = sVs[i * LVP + c] - fz[j][e];
          sZs[i * LVP + c] = sBeta[i] * r;
          sVs[i * LVP + c] = r;  // V - Y
        }
    } else if (tid < 64 * LBV / 4) {
      const int i = tid / (LBV / 4), c4 = (tid % (LBV / 4)) * 4;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int d = 0; d < GDN_DK; ++d) {
        const float kg = sK[i * KP + d] * EG(i, d);
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[y] = fmaf(kg, sHs[d * LVP + c4 + y], acc[y]);
      }
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const float r = sVs[i * LVP + c4 + y] - acc[y];
        sZs[i * LVP + c4 + y] = sBeta[i] * r;
        sVs[i * LVP + c4 + y] = r;  // V - Y
      }
    }
    __syncthreads();
    // v_new = X Z ; dZ = X^T dv_new
    if constexpr (TC) {  // both 64 x LBV products on tensor cores, LBV/16 tiles per warp
      constexpr int NZ = LBV / 16;
      const int zr0 = 16 * ((tid >> 5) & 3), zc0 = (LBV / 2) * (tid >> 7);
      float fv[NZ][4], fd[NZ][4];
      zero_acc(fv);
      zero_acc(fd);
      auto fx = [&](int m, int kk) { return sX[m * CP + kk]; };
      auto fxt = [&](int m, int kk) { return sX[kk * CP + m]; };
      auto fzs = [&](int kk, int nn) { return sZs[kk * LVP + nn]; };
      auto fdd = [&](int kk, int nn) { return sDDs[kk * LVP + nn]; };
      mma_tf32_acc<GDN_CHUNK, NZ>(fx, fzs, fv, zr0, zc0, lane);
      mma_tf32_acc<GDN_CHUNK, NZ>(fxt, fdd, fd, zr0, zc0, lane);
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {  // rows zr0 + fg and zr0 + fg + 8
        const int i = zr0 + fg + 8 * hr;
        float db = 0.f;
#pragma unroll
        for (int j = 0; j < NZ; ++j)
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int e = 2 * hr + cc, c = zc0 + 8 * j + 2 * ft + cc;
            sDels[i * LVP + c] = fv[j][e];
            db = fmaf(fd[j][e], sVs[i * LVP + c], db);
            sDYs[i * LVP + c] = -sBeta[i] * fd[j][e];
            if (i < n) dv[((c0 + i) * H + h) * GDN_DV + vs + c] = from_f32<T>(sBeta[i] * fd[j][e]);
          }
        // the row's four lanes, then one writer per (column half, row)
        db += __shfl_xor_sync(0xffffffffu, db, 1);
        db += __shfl_xor_sync(0xffffffffu, db, 2);
        if (ft == 0) sDBpart[64 * (tid >> 7) + i] += db;
      }
    } else if (tid < 64 * LBV / 4) {
      const int i = tid / (LBV / 4), c4 = (tid % (LBV / 4)) * 4;
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < GDN_CHUNK; ++j) {
        const float x = sX[i * CP + j], xt = sX[j * CP + i];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          acc[y] = fmaf(x, sZs[j * LVP + c4 + y], acc[y]);
          acc2[y] = fmaf(xt, sDDs[j * LVP + c4 + y], acc2[y]);
        }
      }
      float db = 0.f;
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        sDels[i * LVP + c4 + y] = acc[y];
        db = fmaf(acc2[y], sVs[i * LVP + c4 + y], db);
        sDYs[i * LVP + c4 + y] = -sBeta[i] * acc2[y];
        if (i < n) dv[((c0 + i) * H + h) * GDN_DV + vs + c4 + y] = from_f32<T>(sBeta[i] * acc2[y]);
      }
      // the row's LBV/4 consecutive lanes, then one writer per row
#pragma unroll
      for (int off = 1; off < LBV / 4; off <<= 1) db += __shfl_xor_sync(0xffffffffu, db, off);
      if (c4 == 0) sDBpart[i] += db;
    }
    if (tid < GDN_DK) {
      float acc = 0.f;
      for (int c = 0; c < LBV; ++c) acc = fmaf(sDHs[tid * LVP + c], sHs[tid * LVP + c], acc);
      sDGLh[tid] += acc;
    }
    __syncthreads();
    // dX += dv_new Z^T ; dA_qk += scale dO v_new^T ; dQg += dO h^T ; dKg += dY h^T ;
    // dkgl += v_new dh^T
    {
      auto fdd = [&](int m, int kk) { return sDDs[m * LVP + kk]; };
      auto fz = [&](int kk, int nn) { return sZs[nn * LVP + kk]; };
      auto fo = [&](int m, int kk) { return sDOs[m * LVP + kk]; };
      auto fdl = [&](int kk, int nn) { return sDels[nn * LVP + kk]; };
      auto fy = [&](int m, int kk) { return sDYs[m * LVP + kk]; };
      auto fd = [&](int m, int kk) { return sDels[m * LVP + kk]; };
      auto fh = [&](int kk, int nn) { return sHs[nn * LVP + kk]; };
      auto fdh = [&](int kk, int nn) { return sDHs[nn * LVP + kk]; };
      if constexpr (TC) {
        mma_tf32_acc<LBV, 4>(fdd, fz, fX, wr0, wc64, lane);
        mma_tf32_acc<LBV, 4>(fo, fdl, fQk, wr0, wc64, lane);
        mma_tf32_acc<LBV, 8>(fo, fh, fQg, wr0, wc128, lane);
        mma_tf32_acc<LBV, 8>(fy, fh, fKg, wr0, wc128, lane);
        mma_tf32_acc<LBV, 8>(fd, fdh, fKl, wr0, wc128, lane);
      } else {
        mm_acc<64, 64, LBV, 4, 4>(fdd, fz, aX, tid);
        mm_acc<64, 64, LBV, 4, 4>(fo, fdl, aQk, tid);
        mm_acc<64, 128, LBV, 4, 8>(fo, fh, aQg, tid);
        mm_acc<64, 128, LBV, 4, 8>(fy, fh, aKg, tid);
        mm_acc<64, 128, LBV, 4, 8>(fd, fdh, aKl, tid);
      }
    }
    __syncthreads();
  }

  if constexpr (TC) {  // tensor-core fragments -> the thread tiles, through the slice region
    constexpr int LD = GDN_DK + 4;
    float *st = sSl;  // [64][LD], free after the pass
    auto to_tiles = [&](auto &frag, auto &tile, int c0, int tm0, int tn0) {
      mma_frag_store(st, LD, frag, wr0, c0, lane);
      __syncthreads();
      constexpr int TMv = sizeof(tile) / sizeof(tile[0]);
      constexpr int TNv = sizeof(tile[0]) / sizeof(float);
#pragma unroll
      for (int x = 0; x < TMv; ++x)
#pragma unroll
        for (int y = 0; y < TNv; ++y) tile[x][y] = st[(tm0 + x) * LD + tn0 + y];
      __syncthreads();
    };
    to_tiles(fX, aX, wc64, pm0, pn0);
    to_tiles(fQk, aQk, wc64, pm0, pn0);
    to_tiles(fQg, aQg, wc128, gm0, gn0);
    to_tiles(fKg, aKg, wc128, gm0, gn0);
    to_tiles(fKl, aKl, wc128, gm0, gn0);
  }

  // ---- dL = -X^T dX X^T ; dbeta ; dP ------------------------------------------
  float *sDX = sSl;              // [64][CP]
  float *sT1 = sSl + 64 * CP;    // [64][CP]
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      sDX[(pm0 + x) * CP + pn0 + y] = aX[x][y];
      // dA_qk is used only on the causal part; fold the output scale in now
      aQk[x][y] = (pn0 + y <= pm0 + x) ? a.scale * aQk[x][y] : 0.f;
    }
  __syncthreads();
  {
    auto fa = [&](int m, int kk) { return sDX[m * CP + kk]; };
    auto fb = [&](int kk, int nn) { return sX[nn * CP + kk]; };
    if constexpr (TC) {  // dX X^T on tensor cores, fragments straight into sT1
      float fr[4][4];
      zero_acc(fr);
      mma_tf32_acc<GDN_CHUNK, 4>(fa, fb, fr, wr0, wc64, lane);
      mma_frag_store(sT1, CP, fr, wr0, wc64, lane);
    } else {
      float acc[4][4];
      zero_acc(acc);
      mm_acc<64, 64, GDN_CHUNK, 4, 4>(fa, fb, acc, tid);  // dX X^T
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) sT1[(pm0 + x) * CP + pn0 + y] = acc[x][y];
    }
  }
  __syncthreads();
  {
    float acc[4][4];
    zero_acc(acc);
    auto fa = [&](int m, int kk) { return sX[kk * CP + m]; };
    auto fb = [&](int kk, int nn) { return sT1[kk * CP + nn]; };
    if constexpr (TC) {  // X^T (dX X^T) on tensor cores, into the thread tile through sDX (free)
      float fr[4][4];
      zero_acc(fr);
      mma_tf32_acc<GDN_CHUNK, 4>(fa, fb, fr, wr0, wc64, lane);
      mma_frag_store(sDX, CP, fr, wr0, wc64, lane);
      __syncthreads();
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = sDX[(pm0 + x) * CP + pn0 + y];
    } else {
      mm_acc<64, 64, GDN_CHUNK, 4, 4>(fa, fb, acc, tid);  // X^T (dX X^T)
    }
    float rows[4] = {0.f, 0.f, 0.f, 0.f};
    float dPv[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int i = pm0 + x, j = pn0 + y;
        const float dL = j < i ? -acc[x][y] : 0.f;
        rows[x] = fmaf(dL, sP[i * CP + j], rows[x]);
        dPv[x][y] = sBeta[i] * dL;
      }
    // the 16 lanes of a row block (consecutive threads), then one writer per row
#pragma unroll
    for (int x = 0; x < 4; ++x) {
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) rows[x] += __shfl_xor_sync(0xffffffffu, rows[x], off);
      if ((tid & 15) == 0) sDBpart[128 + pm0 + x] = rows[x];
    }
    __syncthreads();  // every read of sP (the gated Gram) is done
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int i = pm0 + x, j = pn0 + y;
        float mP = dPv[x][y], mQ = aQk[x][y];
        if (!PER_KEY) {
          const float gam = j <= i ? gate_pow(sG[i] - sG[j], e2) : 0.f;
          mP *= gam;
          mQ *= gam;
        }
        sP[i * CP + j] = mP;
        sAqk[i * CP + j] = mQ;
      }
  }
  __syncthreads();

  // ---- fold everything into dq, dk, dG ------------------------------------------
  float rdq[4][8], rdk[4][8], rdG[4][8];
  float colGl[8];
#pragma unroll
  for (int y = 0; y < 8; ++y) colGl[y] = 0.f;
#pragma unroll
  for (int x = 0; x < 4; ++x)
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      const int i = gm0 + x, d = gn0 + y;
      const float eg = TC ? bx(sG[i * KP + d]) : EG(i, d);
      const float egl = TC ? bx(sG[63 * KP + d] - sG[i * KP + d]) : EGL(i, d);
      const float kk = sK[i * KP + d], qq = sQ[i * KP + d];
      const float dQg = a.scale * aQg[x][y];
      rdq[x][y] = dQg * eg;
      rdk[x][y] = aKg[x][y] * eg + aKl[x][y] * egl;
      rdG[x][y] = lnb * (dQg * qq * eg + aKg[x][y] * kk * eg - aKl[x][y] * kk * egl);
      colGl[y] = fmaf(aKl[x][y] * kk, egl, colGl[y]);
    }
  // threads t and t + 16 of a warp share the columns, then one slot per (warp, column)
#pragma unroll
  for (int y = 0; y < 8; ++y) {
    colGl[y] += __shfl_xor_sync(0xffffffffu, colGl[y], 16);
    if (lane < 16) sGlPart[(tid >> 5) * 128 + gn0 + y] = colGl[y];
  }
  // Gram adjoints, one at a time: (dP K), (dAqk K), (dP^T K), (dAqk^T Q), with Gamma (in
  // this order the tensor-core path forms its right operands K / e, K (.) e, Q (.) e once each)
#pragma unroll 1
  for (int step = 0; step < 4; ++step) {
    const int which = step == 1 ? 2 : step == 2 ? 1 : step;
    const float *Mx = which < 2 ? sP : sAqk;
    const bool tr = which == 1 || which == 3;  // use M^T
    const float *Op = which == 3 ? sQ : sK;
    float t[4][8];
    zero_acc(t);
    // term by term, one gate factor per (i, j, d): exact for any gate range
    auto by_terms = [&]() {
      for (int j = 0; j < GDN_CHUNK; ++j) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int i = gm0 + x;
          const float m = tr ? Mx[j * CP + i] : Mx[i * CP + j];
          if (m == 0.f) continue;
#pragma unroll
          for (int y = 0; y < 8; ++y) {
            const int d = gn0 + y;
            float w = m * Op[j * KP + d];
            if (PER_KEY)
              w *= tr ? gate_pow(sG[j * KP + d] - sG[i * KP + d], e2)
                      : gate_pow(sG[i * KP + d] - sG[j * KP + d], e2);
            t[x][y] += w;
          }
        }
      }
    };
    if constexpr (TC) {
      if (fast) {
        // (M or M^T)(Op (.) e^-+1) on tf32 tensor cores, then the row factor e^+-1 of (i, d)
        constexpr int LD = GDN_DK + 4;
        float *st = sSl;
        float *tB = sWideB;  // [64][KP], the right operand (X's region is free by now)
        if (step != 1) {
          for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
            const int j = idx >> 7, d = idx & 127;
            const float x = sG[j * KP + d] - sG[REFR * KP + d];
            tB[j * KP + d] = Op[j * KP + d] * bx(tr ? x : -x);
          }
          __syncthreads();
        }
        float fr[8][4];
        zero_acc(fr);
        auto fm = [&](int m, int kk) { return tr ? Mx[kk * CP + m] : Mx[m * CP + kk]; };
        auto fop = [&](int kk, int nn) { return tB[kk * KP + nn]; };
        mma_tf32_acc<GDN_CHUNK, 8>(fm, fop, fr, wr0, wc128, lane);
        mma_frag_store(st, LD, fr, wr0, wc128, lane);
        __syncthreads();
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 8; ++y) {
            const int i = gm0 + x, d = gn0 + y;
            const float xi = sG[i * KP + d] - sG[REFR * KP + d];
            t[x][y] = st[i * LD + d] * bx(tr ? -xi : xi);
          }
        __syncthreads();
      } else {
        by_terms();
      }
    } else {
      by_terms();
    }
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) {
        const int i = gm0 + x, d = gn0 + y;
        const float kk = sK[i * KP + d], qq = sQ[i * KP + d];
        if (which == 0) {
          rdk[x][y] += t[x][y];
          rdG[x][y] += lnb * kk * t[x][y];
        } else if (which == 1) {
          rdk[x][y] += t[x][y];
          rdG[x][y] -= lnb * kk * t[x][y];
        } else if (which == 2) {
          rdq[x][y] += t[x][y];
          rdG[x][y] += lnb * qq * t[x][y];
        } else {
          rdk[x][y] += t[x][y];
          rdG[x][y] -= lnb * kk * t[x][y];
        }
      }
  }
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int i = gm0 + x;
    if (i >= n) continue;
#pragma unroll
    for (int y = 0; y < 8; ++y) {
      const int64_t off = ((c0 + i) * H + h) * GDN_DK + gn0 + y;
      dq[off] = from_f32<T>(rdq[x][y]);
      dk[off] = from_f32<T>(rdk[x][y]);
    }
  }
  __syncthreads();  // the dG_last slots are complete; sQ is free for the gate gradient
  if (tid < GDN_DK) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) acc += sGlPart[w * 128 + tid];
    sDGlast[tid] = acc;
  }
  if (tid < 64) sDBeta[tid] = sDBpart[tid] + sDBpart[64 + tid] + sDBpart[128 + tid];
  __syncthreads();
  // ---- gate gradient: add G_last terms, reverse cumulative sum ---------------
  if (PER_KEY) {
    float *sDG = sQ;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 8; ++y) sDG[(gm0 + x) * KP + gn0 + y] = rdG[x][y];
    __syncthreads();
    if (tid < GDN_DK) {
      const int d = tid;
      const float extra = lnb * (sDGlast[d] + sEL[d] * sDGLh[d]);
      float run = 0.f;
      for (int i = n - 1; i >= 0; --i) {
        run += sDG[i * KP + d] + (i == n - 1 ? extra : 0.f);
        a.dg[((c0 + i) * H + h) * GDN_DK + d] = run;
      }
    }
  } else {
    // the 16 lanes of a row block, then one writer per row
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      float sr = 0.f;
#pragma unroll
      for (int y = 0; y < 8; ++y) sr += rdG[x][y];
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) sr += __shfl_xor_sync(0xffffffffu, sr, off);
      if ((tid & 15) == 0) sDGrow[gm0 + x] = sr;
    }
    if (tid < GDN_DK) {  // the G_last term, summed over the key channels warp by warp
      float xg = lnb * (sDGlast[tid] + sEL[tid] * sDGLh[tid]);
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) xg += __shfl_xor_sync(0xffffffffu, xg, off);
      if (lane == 0) sRowX[tid >> 5] = xg;
    }
    __syncthreads();
    if (tid == 0) {
      float run = 0.f;
      const float extra = sRowX[0] + sRowX[1] + sRowX[2] + sRowX[3];
      for (int i = n - 1; i >= 0; --i) {
        run += sDGrow[i] + (i == n - 1 ? extra : 0.f);
        a.dg[(c0 + i) * H + h] = run;
      }
    }
  }
  if (tid < n) dbeta[(c0 + tid) * H + h] = from_f32<T>(sDBeta[tid]);
}

template <typename T, bool PK>
cudaError_t dhu_one(const BwdArgs &a, cudaStream_t st) {
  const size_t bytes = dhu_smem_floats<PK>() * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(dhu_kernel<T, PK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const int runs = a.cu ? a.num_seqs : (a.nseg > 0 ? a.B * a.nseg : a.B);
  dhu_kernel<T, PK><<<dim3(GDN_DV / DBV, a.H, runs), NTH, bytes, st>>>(a);
  return cudaGetLastError();
}

template <typename T, bool PK>
cudaError_t local_one(const BwdArgs &a, cudaStream_t st) {
  const size_t bytes = local_smem_floats<T, PK>() * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(local_kernel<T, PK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  const int64_t nch = a.cu ? a.num_chunks : (int64_t)a.B * ((a.T + GDN_CHUNK - 1) / GDN_CHUNK);
  if (nch == 0) return cudaSuccess;
  local_kernel<T, PK><<<dim3((unsigned)nch, a.H), NTH, bytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dhu(const BwdArgs &a, bool per_key, bool bf16, cudaStream_t st) {
  if (bf16) return per_key ? dhu_one<__nv_bfloat16, true>(a, st) : dhu_one<__nv_bfloat16, false>(a, st);
  return per_key ? dhu_one<float, true>(a, st) : dhu_one<float, false>(a, st);
}

cudaError_t launch_bwd_local(const BwdArgs &a, bool per_key, bool bf16, cudaStream_t st) {
  if (bf16) {  // a scalar gate with bf16 inputs runs on local_tc (launch_bwd_local_tc)
    if (!per_key) return cudaErrorNotSupported;
    return local_one<__nv_bfloat16, true>(a, st);
  }
  return per_key ? local_one<float, true>(a, st) : local_one<float, false>(a, st);
}

}  // namespace gdn
