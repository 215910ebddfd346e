// fp32 SIMT chunk kernel for the gated delta rule (sm_103a).
//
// One CTA owns one independent run (a batch row, a packed document or a
// segment) of one head and one 32-column slice of the state, and walks the
// run's 64-token chunks in order. Per chunk it takes the steps of the chunk
// algorithm ("state_summary.py" kda_split_state_summary_kernel
// loop body; chunk_fwd_h / chunk_kda_fwd_finalize stages of the KDA adapter):
//   G   = in-chunk cumulative log-gate
//   L   = strictly-lower(diag(beta) (K K^T (.) Gamma)),  X = (I + L)^-1
//   v_new = X (beta (.) (V - (K (.) base^G) h))     ( = u - w h )
//   o   = scale ((Q (.) base^G) h + A_qk v_new)
//   h  <- Diag(base^G_last) h + (K (.) base^(G_last - G))^T v_new
// Everything is fp32 in shared memory with register-tiled FMA products; the
// per-key gate Gamma_ijd = base^(G_id - G_jd) is evaluated term by term, so
// this path is exact up to fp32 rounding for any gate range. It serves fp32
// inputs, the segment summary (the same recurrence on [V | I] columns), and
// the backward's recompute of chunk entry states.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int BV = 32;            // state columns per CTA
constexpr int NTH = 256;          // threads per CTA
constexpr int KP = GDN_DK + 1;    // padded row stride of [64][128] tiles
constexpr int CP = GDN_CHUNK + 1; // padded row stride of [64][64] tiles
constexpr int VP = BV + 1;        // padded row stride of [*][32] tiles

template <bool PER_KEY>
constexpr size_t smem_floats() {
  return 3 * 64 * KP + (PER_KEY ? 64 * KP : 3 * 64) + 2 * 64 * CP + 128 * VP + 3 * 64 * VP + 64 +
         128;
}

template <typename T, bool PER_KEY>
__global__ void __launch_bounds__(NTH) simt_chunk_kernel(SimtFwdArgs a) {
  extern __shared__ float smem[];
  float *sK = smem;                                // K, later K (.) base^(G_last - G)
  float *sQ = sK + 64 * KP;                        // Q, later scale Q (.) base^G
  float *sKg = sQ + 64 * KP;                       // L during the solve, then K (.) base^G
  float *sG = sKg + 64 * KP;                       // cumulative gate [64][KP], or [64] + e^G + e^(Gl-G)
  float *sX = sG + (PER_KEY ? 64 * KP : 3 * 64);   // X = (I + L)^-1
  float *sAqk = sX + 64 * CP;                      // gated causal Q K^T
  float *sH = sAqk + 64 * CP;                      // state slice [128][VP]
  float *sV = sH + 128 * VP;                       // value slice
  float *sZ = sV + 64 * VP;                        // beta (V - Kg h)
  float *sD = sZ + 64 * VP;                        // v_new slice
  float *sBeta = sD + 64 * VP;                     // [64]
  float *sEL = sBeta + 64;                         // base^G_last per key channel [128]

  const int tid = threadIdx.x;
  const int H = a.H;
  const int h = blockIdx.y;
  const int z = blockIdx.z;
  const int col0 = blockIdx.x * BV;
  const bool e2 = a.use_exp2 != 0;
  const bool summ = a.summary != 0;
  const T *q = static_cast<const T *>(a.q);
  const T *k = static_cast<const T *>(a.k);
  const T *v = static_cast<const T *>(a.v);
  const T *beta = static_cast<const T *>(a.beta);
  T *o = static_cast<T *>(a.o);

  // ---- the run this CTA owns -------------------------------------------
  int64_t r0, r1, chunk_base = 0;
  int b = 0, s = 0, state_idx;
  const int NT = (a.T + GDN_CHUNK - 1) / GDN_CHUNK;
  if (a.cu) {
    r0 = a.cu[z];
    r1 = a.cu[z + 1];
    if (r0 < 0 || r1 <= r0 || r1 > a.T) {
      if (tid == 0) raise_device_flag(a.dev_flag, kDevCheck);
      return;
    }
    for (int m = 0; m < z; ++m) chunk_base += (a.cu[m + 1] - a.cu[m] + GDN_CHUNK - 1) / GDN_CHUNK;
    if (chunk_base + (r1 - r0 + GDN_CHUNK - 1) / GDN_CHUNK > a.num_chunks) {
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

  // ---- entry state -----------------------------------------------------
  for (int idx = tid; idx < 128 * BV; idx += NTH) {
    const int d = idx / BV, c = idx % BV, col = col0 + c;
    float val = 0.f;
    if (summ) {
      val = (col >= GDN_DV && d == col - GDN_DV) ? 1.f : 0.f;
    } else if (a.h0) {
      const int64_t base = a.nseg > 0 ? (((int64_t)b * H + h) * a.nseg + s)
                                      : ((int64_t)state_idx * H + h);
      val = a.h0[base * GDN_DK * GDN_DV + d * GDN_DV + col];
    }
    sH[d * VP + c] = val;
  }
  __syncthreads();

  int64_t ci = 0;
  for (int64_t c0 = r0; c0 < r1; c0 += GDN_CHUNK, ++ci) {
    const int n = (int)min((int64_t)GDN_CHUNK, r1 - c0);

    // entry state of this chunk
    if (a.h_chunks) {
      int64_t slot;
      if (a.cu)
        slot = (chunk_base + ci) * H + h;
      else
        slot = ((int64_t)b * H + h) * NT + chunk_base + ci;
      float *dst = a.h_chunks + slot * GDN_DK * GDN_DV;
      for (int idx = tid; idx < 128 * BV; idx += NTH) {
        const int d = idx / BV, c = idx % BV;
        dst[d * GDN_DV + col0 + c] = sH[d * VP + c];
      }
    }

    // ---- loads ----------------------------------------------------------
    for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
      const int i = idx >> 7, d = idx & 127;
      float kv = 0.f, qv = 0.f;
      if (i < n) {
        const int64_t off = ((c0 + i) * H + h) * GDN_DK + d;
        kv = to_f32(k[off]);
        if (!summ) qv = to_f32(q[off]);
      }
      sK[i * KP + d] = kv;
      sQ[i * KP + d] = qv;
    }
    for (int idx = tid; idx < 64 * BV; idx += NTH) {
      const int i = idx / BV, c = idx % BV, col = col0 + c;
      float vv = 0.f;
      if (i < n && col < GDN_DV) vv = to_f32(v[((c0 + i) * H + h) * GDN_DV + col]);
      sV[i * VP + c] = vv;
    }
    if (tid < 64) sBeta[tid] = tid < n ? to_f32(beta[(c0 + tid) * H + h]) : 0.f;
    if (a.g_cum_in) {  // saved cumulative gate; rows past the end repeat the last one
      if (PER_KEY) {
        for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
          const int i = idx >> 7, d = idx & 127;
          sG[i * KP + d] = a.g_cum_in[((c0 + min(i, n - 1)) * H + h) * GDN_DK + d];
        }
      } else if (tid < 64) {
        sG[tid] = a.g_cum_in[(c0 + min(tid, n - 1)) * H + h];
      }
    } else if (PER_KEY) {
      if (tid < GDN_DK) {
        float run = 0.f;
        for (int i = 0; i < GDN_CHUNK; ++i) {
          if (i < n) run += a.g[((c0 + i) * H + h) * GDN_DK + tid];
          sG[i * KP + tid] = run;
        }
      }
    } else if (tid < 32) {
      const int i0 = 2 * tid, i1 = 2 * tid + 1;
      const float x0 = i0 < n ? a.g[(c0 + i0) * H + h] : 0.f;
      const float x1 = i1 < n ? a.g[(c0 + i1) * H + h] : 0.f;
      const float pair = x0 + x1;
      float incl = pair;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (tid >= off) incl += y;
      }
      const float excl = incl - pair;
      sG[i0] = excl + x0;
      sG[i1] = excl + pair;
    }
    __syncthreads();

    const bool lead = blockIdx.x == 0 && !summ;
    if (lead && a.g_cumsum) {
      if (PER_KEY) {
        for (int idx = tid; idx < n * GDN_DK; idx += NTH)
          a.g_cumsum[((c0 + (idx >> 7)) * H + h) * GDN_DK + (idx & 127)] =
              sG[(idx >> 7) * KP + (idx & 127)];
      } else if (tid < n) {
        a.g_cumsum[(c0 + tid) * H + h] = sG[tid];
      }
    }

    // ---- gated Gram matrices: L (into sKg) and A_qk ----------------------
    {
      int m0, n0;
      tile_origin<64, 64, 4, 4>(tid, m0, n0);
      float accP[4][4], accQ[4][4];
      zero_acc(accP);
      zero_acc(accQ);
      if (n0 <= m0 + 3) {  // tiles wholly above the diagonal stay zero
        if (PER_KEY) {
          for (int d = 0; d < GDN_DK; ++d) {
            float ki[4], qi[4], gi[4], kj[4], gj[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              ki[t] = sK[(m0 + t) * KP + d];
              qi[t] = sQ[(m0 + t) * KP + d];
              gi[t] = sG[(m0 + t) * KP + d];
              kj[t] = sK[(n0 + t) * KP + d];
              gj[t] = sG[(n0 + t) * KP + d];
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
              for (int y = 0; y < 4; ++y) {
                if (n0 + y > m0 + x) continue;
                const float gam = gate_pow(gi[x] - gj[y], e2);
                accP[x][y] = fmaf(ki[x] * kj[y], gam, accP[x][y]);
                accQ[x][y] = fmaf(qi[x] * kj[y], gam, accQ[x][y]);
              }
          }
        } else {
          auto fk = [&](int m, int kk) { return sK[m * KP + kk]; };
          auto fq = [&](int m, int kk) { return sQ[m * KP + kk]; };
          auto fkt = [&](int kk, int nn) { return sK[nn * KP + kk]; };
          mm_acc<64, 64, GDN_DK, 4, 4>(fk, fkt, accP, tid);
          if (!summ) mm_acc<64, 64, GDN_DK, 4, 4>(fq, fkt, accQ, tid);
#pragma unroll
          for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
              const float gam = gate_pow(sG[m0 + x] - sG[n0 + y], e2);
              accP[x][y] *= gam;
              accQ[x][y] *= gam;
            }
        }
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int i = m0 + x, j = n0 + y;
          sKg[i * CP + j] = j < i ? sBeta[i] * accP[x][y] : 0.f;
          sAqk[i * CP + j] = j <= i ? accQ[x][y] : 0.f;
        }
    }
    __syncthreads();

    if (!PER_KEY && tid >= 64 && tid < 128) {  // per-token gate factors (scalar gate)
      const int i = tid - 64;
      sG[64 + i] = gate_pow(sG[i], e2);
      sG[128 + i] = gate_pow(sG[63] - sG[i], e2);
    }
    // ---- X = (I + L)^-1 by forward substitution, one column per thread ---
    if (a.A_in) {
      for (int idx = tid; idx < 64 * 64; idx += NTH) {
        const int i = idx >> 6, j = idx & 63;
        sX[i * CP + j] = (i < n && j < n) ? a.A_in[((c0 + i) * H + h) * GDN_CHUNK + j]
                                          : (i == j ? 1.f : 0.f);
      }
    } else if (tid < GDN_CHUNK) {
      const int c = tid;
      for (int i = 0; i < c; ++i) sX[i * CP + c] = 0.f;
      sX[c * CP + c] = 1.f;
      for (int i = c + 1; i < GDN_CHUNK; ++i) {
        float acc = 0.f;
        for (int j = c; j < i; ++j) acc = fmaf(sKg[i * CP + j], sX[j * CP + c], acc);
        sX[i * CP + c] = -acc;
      }
    }
    __syncthreads();
    if (lead && a.A) {
      for (int idx = tid; idx < n * GDN_CHUNK; idx += NTH) {
        const int i = idx >> 6, j = idx & 63;
        a.A[((c0 + i) * H + h) * GDN_CHUNK + j] = sX[i * CP + j];
      }
    }

    // ---- gate the operands ----------------------------------------------
    for (int idx = tid; idx < 64 * GDN_DK; idx += NTH) {
      const int i = idx >> 7, d = idx & 127;
      const float Gi = PER_KEY ? sG[i * KP + d] : sG[i];
      const float Gl = PER_KEY ? sG[63 * KP + d] : sG[63];
      const float kk = sK[i * KP + d];
      const float eg = PER_KEY ? gate_pow(Gi, e2) : sG[64 + i];
      const float egl = PER_KEY ? gate_pow(Gl - Gi, e2) : sG[128 + i];
      sKg[i * KP + d] = kk * eg;
      sQ[i * KP + d] *= a.scale * eg;
      sK[i * KP + d] = kk * egl;
    }
    if (tid < GDN_DK) sEL[tid] = gate_pow(PER_KEY ? sG[63 * KP + tid] : sG[63], e2);
    __syncthreads();

    // ---- Z = beta (V - Kg h) ----------------------------------------------
    {
      float acc[2][4];
      zero_acc(acc);
      auto fa = [&](int m, int kk) { return sKg[m * KP + kk]; };
      auto fb = [&](int kk, int nn) { return sH[kk * VP + nn]; };
      mm_acc<64, BV, GDN_DK, 2, 4>(fa, fb, acc, tid);
      int m0, n0;
      tile_origin<64, BV, 2, 4>(tid, m0, n0);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y)
          sZ[(m0 + x) * VP + n0 + y] = sBeta[m0 + x] * (sV[(m0 + x) * VP + n0 + y] - acc[x][y]);
    }
    __syncthreads();
    // ---- v_new = X Z -------------------------------------------------------
    {
      float acc[2][4];
      zero_acc(acc);
      auto fa = [&](int m, int kk) { return sX[m * CP + kk]; };
      auto fb = [&](int kk, int nn) { return sZ[kk * VP + nn]; };
      mm_acc<64, BV, GDN_CHUNK, 2, 4>(fa, fb, acc, tid);
      int m0, n0;
      tile_origin<64, BV, 2, 4>(tid, m0, n0);
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) sD[(m0 + x) * VP + n0 + y] = acc[x][y];
    }
    __syncthreads();
    // ---- output and state update --------------------------------------------
    if (!summ && o) {
      float acc[2][4];
      zero_acc(acc);
      auto fq = [&](int m, int kk) { return sQ[m * KP + kk]; };
      auto fh = [&](int kk, int nn) { return sH[kk * VP + nn]; };
      mm_acc<64, BV, GDN_DK, 2, 4>(fq, fh, acc, tid);
      auto fa = [&](int m, int kk) { return sAqk[m * CP + kk]; };
      auto fd = [&](int kk, int nn) { return sD[kk * VP + nn]; };
      float acc2[2][4];
      zero_acc(acc2);
      mm_acc<64, BV, GDN_CHUNK, 2, 4>(fa, fd, acc2, tid);
      int m0, n0;
      tile_origin<64, BV, 2, 4>(tid, m0, n0);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        if (m0 + x >= n) continue;
        T *dst = o + ((c0 + m0 + x) * H + h) * GDN_DV + col0 + n0;
#pragma unroll
        for (int y = 0; y < 4; ++y) dst[y] = from_f32<T>(acc[x][y] + a.scale * acc2[x][y]);
      }
    }
    {
      float acc[4][4];
      zero_acc(acc);
      auto fa = [&](int m, int kk) { return sK[kk * KP + m]; };  // (K (.) base^(Gl-G))^T
      auto fb = [&](int kk, int nn) { return sD[kk * VP + nn]; };
      mm_acc<128, BV, GDN_CHUNK, 4, 4>(fa, fb, acc, tid);
      int m0, n0;
      tile_origin<128, BV, 4, 4>(tid, m0, n0);
      __syncthreads();  // every read of sH above is done
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          float &hv = sH[(m0 + x) * VP + n0 + y];
          hv = fmaf(sEL[m0 + x], hv, acc[x][y]);
        }
    }
    __syncthreads();
  }

  // ---- final state -------------------------------------------------------
  float *dst = nullptr;
  int ld = GDN_DV, cshift = 0;
  if (summ) {
    const int64_t sl = ((int64_t)b * H + h) * a.nseg + s;
    if (col0 >= GDN_DV) {
      dst = a.M + sl * GDN_DK * GDN_DK;
      ld = GDN_DK;
      cshift = GDN_DV;
    } else {
      dst = a.S_ext + sl * GDN_DK * GDN_DV;
    }
  } else if (a.ht && (a.nseg == 0 || s == a.nseg - 1)) {
    dst = a.ht + ((int64_t)state_idx * H + h) * GDN_DK * GDN_DV;
  }
  if (dst) {
    for (int idx = tid; idx < 128 * BV; idx += NTH) {
      const int d = idx / BV, c = idx % BV;
      dst[d * ld + col0 - cshift + c] = sH[d * VP + c];
    }
  }
}

template <typename T, bool PK>
cudaError_t launch_one(const SimtFwdArgs &a, dim3 grid, cudaStream_t st) {
  const size_t bytes = smem_floats<PK>() * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(simt_chunk_kernel<T, PK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  simt_chunk_kernel<T, PK><<<grid, NTH, bytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

int simt_fwd_bv() { return BV; }

cudaError_t launch_simt_fwd(const SimtFwdArgs &a, bool per_key, bool bf16, dim3 grid,
                            cudaStream_t st) {
  if (bf16)
    return per_key ? launch_one<__nv_bfloat16, true>(a, grid, st)
                   : launch_one<__nv_bfloat16, false>(a, grid, st);
  return per_key ? launch_one<float, true>(a, grid, st) : launch_one<float, false>(a, grid, st);
}

}  // namespace gdn
