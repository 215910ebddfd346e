// C ABI of the chunked gated-delta-rule library: validation, workspace
// layout and dispatch to the sm_103a kernels. See include/gdn.h for the
// contract of every entry point.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/gdn.h"
#include "common.cuh"
#include "kernels.h"

namespace {

thread_local std::string g_last_error;

// Device-side error word (see gdn_device_status); one per device that loads
// the library, written by kernels with atomicMax.
__device__ int g_dev_flag;

gdn_status fail(gdn_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
gdn_status fail(gdn_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

gdn_status ok() {
  g_last_error.clear();
  return GDN_OK;
}

gdn_status cuda_fail(cudaError_t e, const char *what) {
  return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// sm_103 check, cached per device ordinal.
gdn_status check_device(int *dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static int cached[64];  // 0 unknown, 1 ok, 2 bad
  if (dev < 64 && cached[dev] == 1) {
    *dev_out = dev;
    return GDN_OK;
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    if (dev < 64) cached[dev] = 2;
    return fail(GDN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, major, minor);
  }
  if (dev < 64) cached[dev] = 1;
  *dev_out = dev;
  return GDN_OK;
}

int *device_flag_ptr() {
  int *p = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_dev_flag) != cudaSuccess) return nullptr;
  return p;
}

int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Validation shared by the entry points (no device work).
gdn_status check_problem(const gdn_problem *p, bool allow_segments) {
  if (!p) return fail(GDN_ERR_INVALID_ARGUMENT, "problem is NULL");
  if (p->layout != GDN_LAYOUT_BSND && p->layout != GDN_LAYOUT_TND)
    return fail(GDN_ERR_INVALID_ARGUMENT, "layout must be BSND (0) or TND (1), got %d", p->layout);
  if (p->gate_kind != GDN_GATE_SCALAR && p->gate_kind != GDN_GATE_PER_KEY)
    return fail(GDN_ERR_INVALID_ARGUMENT, "gate_kind must be 0 or 1, got %d", p->gate_kind);
  if (p->dtype != GDN_DTYPE_F32 && p->dtype != GDN_DTYPE_BF16)
    return fail(GDN_ERR_INVALID_ARGUMENT, "dtype must be F32 (0) or BF16 (1), got %d", p->dtype);
  if (p->use_exp2 != 0 && p->use_exp2 != 1)
    return fail(GDN_ERR_INVALID_ARGUMENT, "use_exp2 must be 0 or 1");
  if (p->use_qk_l2norm != 0 && p->use_qk_l2norm != 1)
    return fail(GDN_ERR_INVALID_ARGUMENT, "use_qk_l2norm must be 0 or 1");
  if (p->use_beta_sigmoid != 0 && p->use_beta_sigmoid != 1)
    return fail(GDN_ERR_INVALID_ARGUMENT, "use_beta_sigmoid must be 0 or 1");
  if (p->B < 1 || p->H < 1 || p->T < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "need B >= 1, H >= 1, T >= 0 (got B=%d H=%d T=%d)", p->B,
                p->H, p->T);
  if (p->K != GDN_DK || p->V != GDN_DV)
    return fail(GDN_ERR_UNSUPPORTED, "K and V must be 128 (got K=%d V=%d)", p->K, p->V);
  if (p->chunk_size != GDN_CHUNK)
    return fail(GDN_ERR_UNSUPPORTED, "chunk_size must be 64, got %d", p->chunk_size);
  if (!std::isfinite(p->scale))
    return fail(GDN_ERR_INVALID_ARGUMENT, "scale must be finite");
  if ((int64_t)p->B * p->T * p->H * GDN_DK >= (int64_t)1 << 40)
    return fail(GDN_ERR_INVALID_ARGUMENT, "problem too large");
  if (p->layout == GDN_LAYOUT_TND) {
    if (p->B != 1)
      return fail(GDN_ERR_INVALID_ARGUMENT, "packed TND layout requires physical batch size one (B=%d)", p->B);
    if (!p->cu_seqlens || p->num_seqs < 1)
      return fail(GDN_ERR_INVALID_ARGUMENT, "packed TND layout requires cu_seqlens and num_seqs >= 1");
    if (!p->chunk_indices || p->num_chunks < p->num_seqs)
      return fail(GDN_ERR_INVALID_ARGUMENT,
                  "packed TND layout requires chunk_indices with num_chunks >= num_seqs");
    if (p->T < p->num_seqs)
      return fail(GDN_ERR_INVALID_ARGUMENT, "T=%d packed tokens cannot hold %d documents", p->T,
                  p->num_seqs);
    if (!aligned16(p->cu_seqlens) || !aligned16(p->chunk_indices))
      return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens and chunk_indices must be 16-byte aligned");
    if (p->segment_len != 0)
      return fail(GDN_ERR_UNSUPPORTED, "segment_len applies to the BSND layout only");
  } else if (p->cu_seqlens) {
    return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens given with the BSND layout");
  }
  if (p->segment_len != 0) {
    if (!allow_segments) return fail(GDN_ERR_UNSUPPORTED, "segment_len must be 0 here");
    if (p->segment_len < 0 || p->segment_len % GDN_CHUNK != 0)
      return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len must be a positive multiple of 64, got %d",
                  p->segment_len);
  }
  return GDN_OK;
}

#define REQUIRE_PTR(ptr, name)                                                         \
  do {                                                                                 \
    if (!(ptr)) return fail(GDN_ERR_INVALID_ARGUMENT, "%s must not be NULL", name);    \
    if (!aligned16(ptr)) return fail(GDN_ERR_INVALID_ARGUMENT, "%s must be 16-byte aligned", name); \
  } while (0)
#define OPTIONAL_PTR(ptr, name)                                                        \
  do {                                                                                 \
    if ((ptr) && !aligned16(ptr))                                                      \
      return fail(GDN_ERR_INVALID_ARGUMENT, "%s must be 16-byte aligned", name);       \
  } while (0)

float eff_scale(const gdn_problem *p) {
  return p->scale == 0.f ? 1.0f / std::sqrt((float)p->K) : p->scale;
}

// bf16 inputs with one gate per head run on the tensor-core kernels; fp32
// inputs and per-key gates run on the fp32 SIMT kernel. (The input maps run
// before either, so the choice is made on the mapped problem.)
bool use_tensor_cores(const gdn_problem *p) {
  return p->dtype == GDN_DTYPE_BF16 && p->gate_kind == GDN_GATE_SCALAR;
}

// bf16 inputs with one gate per key channel run on the per-key tensor-core path (prep
// kernel + chain kernel over the per-chunk blobs)
bool use_kda_tc(const gdn_problem *p) {
  return p->dtype == GDN_DTYPE_BF16 && p->gate_kind == GDN_GATE_PER_KEY;
}
int64_t n_chunk_slots(const gdn_problem *p);
size_t align256(size_t x);
size_t blob_bytes(const gdn_problem *p) {
  return align256((size_t)n_chunk_slots(p) * p->H * gdn::kda::BLOB_BYTES);
}
// bf16 summaries (either gate kind) run on the tensor-core prep + chain kernels
size_t summary_blob_bytes(const gdn_problem *p) {
  return p->dtype == GDN_DTYPE_BF16 ? blob_bytes(p) : 0;
}
gdn::KdaPrepArgs kda_prep_args(const gdn_problem *p, const void *q, const void *k, const void *v,
                               const float *g, const float *g_cum_in, const void *beta, void *blob,
                               float *g_cumsum, float *A, float scale, int *flag) {
  gdn::KdaPrepArgs r{};
  r.q = q;
  r.k = k;
  r.v = v;
  r.beta = beta;
  r.g = g;
  r.g_cum_in = g_cum_in;
  r.blob = static_cast<uint8_t *>(blob);
  r.g_cumsum = g_cumsum;
  r.A = A;
  r.T = p->T;
  r.H = p->H;
  r.scale = scale;
  r.use_exp2 = p->use_exp2;
  const bool packed = p->layout == GDN_LAYOUT_TND;
  r.cu = packed ? p->cu_seqlens : nullptr;
  r.chunk_indices = packed ? p->chunk_indices : nullptr;
  r.num_seqs = p->num_seqs;
  r.no_q = q == nullptr;
  r.scalar_gate = p->gate_kind == GDN_GATE_SCALAR;
  r.dev_flag = flag;
  return r;
}
gdn::KdaChainArgs kda_chain_args(const gdn::SimtFwdArgs &a, const void *blob) {
  gdn::KdaChainArgs c{};
  c.blob = static_cast<const uint8_t *>(blob);
  c.h0 = a.h0;
  c.o = static_cast<__nv_bfloat16 *>(a.o);
  c.ht = a.ht;
  c.h_chunks = a.h_chunks;
  c.S_ext = a.S_ext;
  c.M = a.M;
  c.B = a.B;
  c.T = a.T;
  c.H = a.H;
  c.cu = a.cu;
  c.num_seqs = a.num_seqs;
  c.num_chunks = a.num_chunks;
  c.seg_len = a.seg_len;
  c.nseg = a.nseg;
  c.summary = a.summary;
  c.dev_flag = a.dev_flag;
  return c;
}

// ---- input maps: L2 norm of q and k, sigmoid of beta ----------------------------------
int64_t token_rows(const gdn_problem *p) {
  return p->layout == GDN_LAYOUT_TND ? (int64_t)p->T : (int64_t)p->B * p->T;
}
size_t elt_bytes(const gdn_problem *p) { return p->dtype == GDN_DTYPE_BF16 ? 2 : 4; }
size_t align256(size_t x);
// workspace of the mapped inputs: [q_n][k_n] (L2 norm), then [beta_eff] (sigmoid)
size_t map_part_bytes(const gdn_problem *p) {
  const size_t rows = (size_t)token_rows(p) * p->H;
  size_t b = 0;
  if (p->use_qk_l2norm) b += 2 * align256(rows * GDN_DK * elt_bytes(p));
  if (p->use_beta_sigmoid) b += align256(rows * elt_bytes(p));
  return b;
}
// the problem the chunk kernels see once the maps have run
gdn_problem mapped_problem(const gdn_problem *p) {
  gdn_problem m = *p;
  m.use_qk_l2norm = 0;
  m.use_beta_sigmoid = 0;
  return m;
}
// Runs the prologue into `ws` and points q, k, beta at the mapped copies (q may be null).
cudaError_t run_input_maps(const gdn_problem *p, const void **q, const void **k, const void **beta,
                           void *ws, cudaStream_t s) {
  const size_t rows = (size_t)token_rows(p) * p->H;
  char *w = static_cast<char *>(ws);
  gdn::InputMapArgs m{};
  m.q = *q;
  m.k = *k;
  m.beta = *beta;
  m.rows = (int64_t)rows;
  m.l2norm = p->use_qk_l2norm;
  m.beta_sigmoid = p->use_beta_sigmoid;
  if (p->use_qk_l2norm) {
    m.qn = w;
    m.kn = w + align256(rows * GDN_DK * elt_bytes(p));
    w += 2 * align256(rows * GDN_DK * elt_bytes(p));
  }
  if (p->use_beta_sigmoid) m.beta_eff = w;
  cudaError_t e = gdn::launch_input_maps(m, p->dtype == GDN_DTYPE_BF16, false, s);
  if (e != cudaSuccess) return e;
  if (p->use_qk_l2norm) {
    if (*q) *q = m.qn;
    *k = m.kn;
  }
  if (p->use_beta_sigmoid) *beta = m.beta_eff;
  return cudaSuccess;
}

int64_t n_chunk_slots(const gdn_problem *p) {
  return p->layout == GDN_LAYOUT_TND ? (int64_t)p->num_chunks : (int64_t)p->B * div_up(p->T, GDN_CHUNK);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// bf16 X = (I + L)^-1 of every chunk and head, then the chunks' gate factor
// tables (tensor-core path only)
size_t x_part_bytes(const gdn_problem *p) {
  return align256((size_t)n_chunk_slots(p) * p->H * 2 * GDN_CHUNK * GDN_CHUNK * 2);
}
size_t x_ws_bytes(const gdn_problem *p) {
  if (use_kda_tc(p)) return blob_bytes(p);
  if (!use_tensor_cores(p)) return 0;
  return x_part_bytes(p) + align256((size_t)n_chunk_slots(p) * p->H * gdn::F_TAB * sizeof(float));
}

gdn::UtArgs ut_args(const gdn_problem *p, const void *k, const float *g, const float *g_cum_in,
                    const void *beta, void *xw, float *A, float *g_cumsum, int *flag) {
  gdn::UtArgs u{};
  u.k = k;
  u.g = g;
  u.g_cum_in = g_cum_in;
  u.beta = beta;
  u.xw = static_cast<__nv_bfloat16 *>(xw);
  u.ftab = reinterpret_cast<float *>(static_cast<char *>(xw) + x_part_bytes(p));
  u.A = A;
  u.g_cumsum = g_cumsum;
  u.T = p->T;
  u.H = p->H;
  u.use_exp2 = p->use_exp2;
  const bool packed = p->layout == GDN_LAYOUT_TND;
  u.cu = packed ? p->cu_seqlens : nullptr;
  u.chunk_indices = packed ? p->chunk_indices : nullptr;
  u.num_seqs = p->num_seqs;
  u.dev_flag = flag;
  return u;
}

struct BwdWs {
  size_t h_chunks, dh_chunks, dvnew, xw, total;
};

// Backward workspace: entry states, exit-state gradients, dv_new, then the forward's. The bf16
// scalar-gate path keeps the first three as bf16 tiles in its local kernel's layout (32 KB, 32 KB
// and 16 KB per chunk and head); the other paths as fp32 arrays.
BwdWs bwd_ws_layout(const gdn_problem *p) {
  BwdWs w{};
  const size_t slots = (size_t)n_chunk_slots(p) * p->H;
  const size_t rows = (size_t)p->B * p->T;
  const bool tiles = use_tensor_cores(p);
  const size_t state = tiles ? (size_t)gdn::STATE_TILE * 2 : (size_t)GDN_DK * GDN_DV * sizeof(float);
  const size_t dv = tiles ? slots * gdn::DV_TILE * 2 : rows * p->H * GDN_DV * sizeof(float);
  w.h_chunks = 0;
  w.dh_chunks = align256(slots * state);
  w.dvnew = w.dh_chunks + align256(slots * state);
  w.xw = w.dvnew + align256(dv);
  w.total = w.xw + x_ws_bytes(p);
  return w;
}

}  // namespace

extern "C" {

const char *gdn_last_error(void) { return g_last_error.c_str(); }

gdn_status gdn_device_status(void *stream) {
  int dev;
  gdn_status st = check_device(&dev);
  if (st != GDN_OK) return st;
  int *flag = device_flag_ptr();
  if (!flag) return fail(GDN_ERR_CUDA, "device flag unavailable");
  int host = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&host, flag, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device flag");
  if (host == gdn::kDevOk) return ok();
  const int zero = 0;
  e = cudaMemcpyAsync(flag, &zero, sizeof(int), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device flag");
  if (host == gdn::kDevTimeout) return fail(GDN_ERR_TIMEOUT, "a bounded device-side wait ran out");
  return fail(GDN_ERR_DEVICE_CHECK, "a kernel found inconsistent device metadata (code %d)", host);
}

gdn_status gdn_selftest_wait_timeout(uint32_t polls, void *stream) {
  if (polls < 1 || polls > GDN_SELFTEST_MAX_POLLS)
    return fail(GDN_ERR_INVALID_ARGUMENT, "polls must be in [1, %u], got %u", (unsigned)GDN_SELFTEST_MAX_POLLS,
                polls);
  int dev;
  gdn_status st = check_device(&dev);
  if (st != GDN_OK) return st;
  int *flag = device_flag_ptr();
  if (!flag) return fail(GDN_ERR_CUDA, "device flag unavailable");
  cudaError_t e = gdn::launch_wait_selftest(polls, flag, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
  return ok();
}

gdn_status gdn_prepare_varlen(const int32_t *cu, int32_t n_seq_plus_1, int64_t total_tokens,
                              int32_t *chunk_indices, int32_t *num_chunks) {
  if (!cu || !num_chunks) return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens and num_chunks must not be NULL");
  if (n_seq_plus_1 < 2)
    return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens needs at least two offsets, got %d", n_seq_plus_1);
  if (cu[0] != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens must start at zero, got %d", cu[0]);
  if ((int64_t)cu[n_seq_plus_1 - 1] != total_tokens)
    return fail(GDN_ERR_INVALID_ARGUMENT, "cu_seqlens must end at the packed token count %lld, got %d",
                (long long)total_tokens, cu[n_seq_plus_1 - 1]);
  int64_t count = 0;
  for (int i = 0; i + 1 < n_seq_plus_1; ++i) {
    if (cu[i] >= cu[i + 1])
      return fail(GDN_ERR_INVALID_ARGUMENT,
                  "cu_seqlens must strictly increase (offsets %d and %d at %d)", cu[i], cu[i + 1], i);
    count += div_up(cu[i + 1] - cu[i], GDN_CHUNK);
  }
  if (count > INT32_MAX) return fail(GDN_ERR_INVALID_ARGUMENT, "too many chunks");
  if (chunk_indices) {
    if (*num_chunks < count)
      return fail(GDN_ERR_INVALID_ARGUMENT, "chunk_indices capacity %d < %lld chunks", *num_chunks,
                  (long long)count);
    int64_t w = 0;
    for (int i = 0; i + 1 < n_seq_plus_1; ++i)
      for (int64_t c = 0; c < div_up(cu[i + 1] - cu[i], GDN_CHUNK); ++c) {
        chunk_indices[2 * w] = i;
        chunk_indices[2 * w + 1] = (int32_t)c;
        ++w;
      }
  }
  *num_chunks = (int32_t)count;
  return ok();
}

gdn_status gdn_chunk_fwd_workspace(const gdn_problem *p, size_t *bytes) {
  gdn_status st = check_problem(p, true);
  if (st != GDN_OK) return st;
  if (!bytes) return fail(GDN_ERR_INVALID_ARGUMENT, "bytes must not be NULL");
  const gdn_problem m = mapped_problem(p);
  *bytes = map_part_bytes(p) + x_ws_bytes(&m);
  return ok();
}

gdn_status gdn_chunk_fwd(const gdn_problem *pin, const void *q, const void *k, const void *v,
                         const float *g, const void *beta, const float *h0, void *o, float *ht,
                         float *g_cumsum, float *A, float *h_chunks, void *ws, size_t ws_bytes,
                         void *stream) {
  gdn_status st = check_problem(pin, true);
  if (st != GDN_OK) return st;
  const gdn_problem mp = mapped_problem(pin);
  const gdn_problem *p = &mp;
  if (p->T > 0) {  // an empty sequence has no token tensors (they may be NULL)
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(g, "g");
    REQUIRE_PTR(beta, "beta");
    REQUIRE_PTR(o, "o");
  }
  OPTIONAL_PTR(h0, "h0");
  OPTIONAL_PTR(ht, "ht");
  OPTIONAL_PTR(g_cumsum, "g_cumsum");
  OPTIONAL_PTR(A, "A");
  OPTIONAL_PTR(h_chunks, "h_chunks");
  const size_t maps = map_part_bytes(pin);
  const size_t need = maps + x_ws_bytes(p);
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(GDN_ERR_WORKSPACE, "forward workspace needs %zu bytes, got %zu", need,
                ws ? ws_bytes : (size_t)0);
  if (ws && !aligned16(ws)) return fail(GDN_ERR_INVALID_ARGUMENT, "ws must be 16-byte aligned");
  if (p->segment_len > 0 && !h0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len > 0 needs h0 = S_init [B,H,nseg,K,V]");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (maps > 0 && p->T > 0) {  // normalised q, k and effective beta into the workspace
    cudaError_t e = run_input_maps(pin, &q, &k, &beta, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "input map launch");
  }
  ws = static_cast<char *>(ws) + maps;

  gdn::SimtFwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.h0 = h0;
  a.o = o;
  a.ht = ht;
  a.g_cumsum = g_cumsum;
  a.A = A;
  a.h_chunks = h_chunks;
  a.B = p->B;
  a.T = p->T;
  a.H = p->H;
  a.scale = eff_scale(p);
  a.use_exp2 = p->use_exp2;
  a.cu = p->layout == GDN_LAYOUT_TND ? p->cu_seqlens : nullptr;
  a.num_seqs = p->num_seqs;
  a.num_chunks = p->num_chunks;
  a.seg_len = p->segment_len;
  a.nseg = p->segment_len > 0 ? (int)div_up(p->T, p->segment_len) : 0;
  a.dev_flag = device_flag_ptr();
  const int runs = a.cu ? p->num_seqs : (a.nseg > 0 ? p->B * a.nseg : p->B);
  if (a.nseg > 0 && p->T == 0) return ok();
  cudaError_t e;
  if (use_kda_tc(p)) {
    const gdn::KdaPrepArgs pa = kda_prep_args(p, q, k, v, g, nullptr, beta, ws, g_cumsum, A, a.scale, a.dev_flag);
    if ((e = gdn::launch_kda_prep(pa, (int)n_chunk_slots(p), s)) != cudaSuccess) return cuda_fail(e, "KDA prep launch");
    e = gdn::launch_kda_chain(kda_chain_args(a, ws), dim3(2, p->H, runs), s);
  } else if (use_tensor_cores(p)) {
    const gdn::UtArgs u = ut_args(p, k, g, nullptr, beta, ws, A, g_cumsum, a.dev_flag);
    if ((e = gdn::launch_ut(u, (int)n_chunk_slots(p), s)) != cudaSuccess) return cuda_fail(e, "UT transform launch");
    a.xw = u.xw;
    a.ftab = u.ftab;
    e = gdn::launch_tc_fwd_ws(a, dim3(GDN_DV / gdn::tc_fwd_ws_bv(), p->H, runs), s);
  } else {
    const dim3 grid(GDN_DV / gdn::simt_fwd_bv(), p->H, runs);
    e = gdn::launch_simt_fwd(a, p->gate_kind == GDN_GATE_PER_KEY, p->dtype == GDN_DTYPE_BF16, grid, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "chunk forward launch");
  return ok();
}

gdn_status gdn_chunk_bwd_workspace(const gdn_problem *p, size_t *bytes) {
  gdn_status st = check_problem(p, true);
  if (st != GDN_OK) return st;
  if (!bytes) return fail(GDN_ERR_INVALID_ARGUMENT, "bytes must not be NULL");
  const gdn_problem m = mapped_problem(p);
  *bytes = map_part_bytes(p) + bwd_ws_layout(&m).total;
  return ok();
}

gdn_status gdn_chunk_bwd(const gdn_problem *pin, const void *q, const void *k, const void *v,
                         const float *g_cumsum, const void *beta, const float *A, const void *dO,
                         const float *h0, const float *dht, void *dq, void *dk, void *dv, float *dg,
                         void *dbeta, float *dh0, void *ws, size_t ws_bytes, void *stream) {
  gdn_status st = check_problem(pin, true);
  if (st != GDN_OK) return st;
  const gdn_problem mp = mapped_problem(pin);
  const gdn_problem *p = &mp;
  const size_t maps = map_part_bytes(pin);
  const void *q_raw = q, *k_raw = k, *beta_raw = beta;
  const int nseg = p->segment_len > 0 ? (int)div_up(p->T, p->segment_len) : 0;
  if (nseg > 0 && !h0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len > 0 needs h0 = S_init [B,H,nseg,K,V]");
  if (p->T > 0) {
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(g_cumsum, "g_cumsum");
    REQUIRE_PTR(beta, "beta");
    REQUIRE_PTR(A, "A");
    REQUIRE_PTR(dO, "dO");
    REQUIRE_PTR(dq, "dq");
    REQUIRE_PTR(dk, "dk");
    REQUIRE_PTR(dv, "dv");
    REQUIRE_PTR(dg, "dg");
    REQUIRE_PTR(dbeta, "dbeta");
  }
  OPTIONAL_PTR(h0, "h0");
  OPTIONAL_PTR(dht, "dht");
  OPTIONAL_PTR(dh0, "dh0");
  const BwdWs L = bwd_ws_layout(p);
  if (maps + L.total > 0 && (!ws || ws_bytes < maps + L.total))
    return fail(GDN_ERR_WORKSPACE, "backward workspace needs %zu bytes, got %zu", maps + L.total,
                ws ? ws_bytes : (size_t)0);
  if (ws && !aligned16(ws)) return fail(GDN_ERR_INVALID_ARGUMENT, "ws must be 16-byte aligned");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool pk = p->gate_kind == GDN_GATE_PER_KEY, bf = p->dtype == GDN_DTYPE_BF16;
  if (maps > 0 && p->T > 0) {  // the forward's mapped inputs, recomputed into the workspace
    cudaError_t e = run_input_maps(pin, &q, &k, &beta, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "input map launch");
  }
  char *w = static_cast<char *>(ws) + maps;
  float *hch = reinterpret_cast<float *>(w + L.h_chunks);
  float *dhch = reinterpret_cast<float *>(w + L.dh_chunks);
  float *dvn = reinterpret_cast<float *>(w + L.dvnew);
  void *xw = w + L.xw;
  const bool packed = p->layout == GDN_LAYOUT_TND;
  const int runs = packed ? p->num_seqs : (nseg > 0 ? p->B * nseg : p->B);
  int *flag = device_flag_ptr();

  if (p->T == 0) {  // nothing but the state: dh0 = dht (no segments at all in segment mode)
    if (dh0 && nseg == 0 && p->segment_len == 0) {
      const size_t bytes = (size_t)runs * p->H * GDN_DK * GDN_DV * sizeof(float);
      cudaError_t e = dht ? cudaMemcpyAsync(dh0, dht, bytes, cudaMemcpyDeviceToDevice, s)
                          : cudaMemsetAsync(dh0, 0, bytes, s);
      if (e != cudaSuccess) return cuda_fail(e, "dh0 pass-through");
    }
    return ok();
  }

  // 1. entry state of every chunk, from the saved cumulative gate and A
  const bool tiles = use_tensor_cores(p);
  gdn::SimtFwdArgs f{};
  f.q = q;
  f.k = k;
  f.v = v;
  f.g = g_cumsum;
  f.beta = beta;
  f.h0 = h0;
  f.h_chunks = tiles ? nullptr : hch;
  f.h_tiles = tiles ? reinterpret_cast<__nv_bfloat16 *>(hch) : nullptr;
  f.B = p->B;
  f.T = p->T;
  f.H = p->H;
  f.scale = eff_scale(p);
  f.use_exp2 = p->use_exp2;
  f.cu = packed ? p->cu_seqlens : nullptr;
  f.num_seqs = p->num_seqs;
  f.num_chunks = p->num_chunks;
  f.seg_len = p->segment_len;
  f.nseg = nseg;
  f.g_cum_in = g_cumsum;
  f.A_in = A;
  f.dev_flag = flag;
  cudaError_t e;
  if (use_kda_tc(p)) {  // blobs recomputed from the saved cumulative gate, then the chain
    const gdn::KdaPrepArgs pa = kda_prep_args(p, q, k, v, nullptr, g_cumsum, beta, xw, nullptr, nullptr,
                                              f.scale, flag);
    if ((e = gdn::launch_kda_prep(pa, (int)n_chunk_slots(p), s)) != cudaSuccess) return cuda_fail(e, "KDA prep launch");
    e = gdn::launch_kda_chain(kda_chain_args(f, xw), dim3(2, p->H, runs), s);
  } else if (use_tensor_cores(p)) {  // the X pair and gate tables from the saved A and cumulative gate
    const gdn::UtArgs u = ut_args(p, k, nullptr, g_cumsum, beta, xw, nullptr, nullptr, flag);
    if ((e = gdn::launch_ut_pair(u, A, (int)n_chunk_slots(p), s)) != cudaSuccess) return cuda_fail(e, "X pair launch");
    f.xw = u.xw;
    f.ftab = u.ftab;
    e = gdn::launch_tc_fwd_ws(f, dim3(GDN_DV / gdn::tc_fwd_ws_bv(), p->H, runs), s);
  } else {
    e = gdn::launch_simt_fwd(f, pk, bf, dim3(GDN_DV / gdn::simt_fwd_bv(), p->H, runs), s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward state recompute launch");

  gdn::BwdArgs b{};
  b.q = q;
  b.k = k;
  b.v = v;
  b.beta = beta;
  b.dO = dO;
  b.g_cumsum = g_cumsum;
  b.A = A;
  b.dht = dht;
  b.dq = dq;
  b.dk = dk;
  b.dv = dv;
  b.dbeta = dbeta;
  b.dg = dg;
  b.dh0 = dh0;
  b.h_chunks = hch;
  b.dh_chunks = dhch;
  b.dvnew = dvn;
  if (tiles) {
    b.h_tiles = reinterpret_cast<const __nv_bfloat16 *>(hch);
    b.dh_tiles = reinterpret_cast<__nv_bfloat16 *>(dhch);
    b.dv_tiles = reinterpret_cast<__nv_bfloat16 *>(dvn);
  }
  b.B = p->B;
  b.T = p->T;
  b.H = p->H;
  b.scale = eff_scale(p);
  b.use_exp2 = p->use_exp2;
  b.cu = packed ? p->cu_seqlens : nullptr;
  b.chunk_indices = packed ? p->chunk_indices : nullptr;
  b.num_seqs = p->num_seqs;
  b.num_chunks = p->num_chunks;
  b.seg_len = p->segment_len;
  b.nseg = nseg;
  b.dev_flag = flag;
  // 2. reverse state recurrence
  if (use_tensor_cores(p)) {
    b.xw = f.xw;
    b.ftab = f.ftab;
    e = gdn::launch_tc_dhu(b, runs, s);
  } else if (use_kda_tc(p)) {
    b.blob = static_cast<const uint8_t *>(xw);
    e = gdn::launch_kda_dhu(b, runs, s);
  } else {
    e = gdn::launch_bwd_dhu(b, pk, bf, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "dhu launch");
  // 3. local gradients
  e = use_tensor_cores(p) ? gdn::launch_bwd_local_tc(b, s) : gdn::launch_bwd_local(b, pk, bf, s);
  if (e != cudaSuccess) return cuda_fail(e, "local gradient launch");
  // 4. chain rules of the input maps, in place: gradients w.r.t. the raw q, k and beta
  if (maps > 0) {
    gdn::InputMapArgs m{};
    m.q = q_raw;
    m.k = k_raw;
    m.beta = beta_raw;
    m.dq = dq;
    m.dk = dk;
    m.dbeta = dbeta;
    m.rows = token_rows(p) * p->H;
    m.l2norm = pin->use_qk_l2norm;
    m.beta_sigmoid = pin->use_beta_sigmoid;
    if ((e = gdn::launch_input_maps(m, bf, true, s)) != cudaSuccess) return cuda_fail(e, "input map backward launch");
  }
  return ok();
}

gdn_status kda_segment_summary_workspace(const gdn_problem *p, int32_t segment_len, size_t *bytes) {
  gdn_status st = check_problem(p, true);
  if (st != GDN_OK) return st;
  if (!bytes) return fail(GDN_ERR_INVALID_ARGUMENT, "bytes must not be NULL");
  if (segment_len <= 0 || segment_len % GDN_CHUNK != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len must be a positive multiple of 64, got %d",
                segment_len);
  const gdn_problem m = mapped_problem(p);
  *bytes = map_part_bytes(p) + summary_blob_bytes(&m);
  return ok();
}

gdn_status kda_segment_summary(const gdn_problem *pin, const void *k, const void *v, const float *g,
                               const void *beta, int32_t segment_len, float *S_ext, float *M,
                               void *ws, size_t ws_bytes, void *stream) {
  gdn_status st = check_problem(pin, true);
  if (st != GDN_OK) return st;
  const gdn_problem mp = mapped_problem(pin);
  const gdn_problem *p = &mp;
  if (p->layout != GDN_LAYOUT_BSND)
    return fail(GDN_ERR_UNSUPPORTED, "segment summaries take the BSND layout");
  if (segment_len <= 0 || segment_len % GDN_CHUNK != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len must be a positive multiple of 64, got %d",
                segment_len);
  REQUIRE_PTR(k, "k");
  REQUIRE_PTR(v, "v");
  REQUIRE_PTR(g, "g");
  REQUIRE_PTR(beta, "beta");
  REQUIRE_PTR(S_ext, "S_ext");
  REQUIRE_PTR(M, "M");
  const size_t maps = map_part_bytes(pin);
  const size_t need = maps + summary_blob_bytes(p);
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(GDN_ERR_WORKSPACE, "segment summary workspace needs %zu bytes, got %zu", need,
                ws ? ws_bytes : (size_t)0);
  if (ws && !aligned16(ws)) return fail(GDN_ERR_INVALID_ARGUMENT, "ws must be 16-byte aligned");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  if (p->T == 0) return ok();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (maps > 0) {  // normalised k and effective beta (q is not needed)
    const void *qnull = nullptr;
    cudaError_t e = run_input_maps(pin, &qnull, &k, &beta, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "input map launch");
  }
  gdn::SimtFwdArgs a{};
  a.q = k;  // unused in summary mode
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.S_ext = S_ext;
  a.M = M;
  a.B = p->B;
  a.T = p->T;
  a.H = p->H;
  a.scale = 1.f;
  a.use_exp2 = p->use_exp2;
  a.seg_len = segment_len;
  a.nseg = (int)div_up(p->T, segment_len);
  a.summary = 1;
  a.dev_flag = device_flag_ptr();
  cudaError_t e;
  if (summary_blob_bytes(p) > 0) {  // bf16: prep (no q) + chain on [V | I] columns
    void *blob = static_cast<char *>(ws) + maps;
    const gdn::KdaPrepArgs pa = kda_prep_args(p, nullptr, k, v, g, nullptr, beta, blob, nullptr, nullptr, 1.f,
                                              a.dev_flag);
    if ((e = gdn::launch_kda_prep(pa, (int)n_chunk_slots(p), s)) != cudaSuccess) return cuda_fail(e, "KDA prep launch");
    e = gdn::launch_kda_chain(kda_chain_args(a, blob), dim3(4, p->H, p->B * a.nseg), s);
  } else {
    const dim3 grid((GDN_DV + GDN_DK) / gdn::simt_fwd_bv(), p->H, p->B * a.nseg);
    e = gdn::launch_simt_fwd(a, p->gate_kind == GDN_GATE_PER_KEY, false, grid, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "segment summary launch");
  return ok();
}

gdn_status kda_segment_summary_bwd_workspace(const gdn_problem *p, int32_t segment_len, size_t *bytes) {
  if (!p) return fail(GDN_ERR_INVALID_ARGUMENT, "problem is NULL");
  if (segment_len <= 0 || segment_len % GDN_CHUNK != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len must be a positive multiple of 64, got %d",
                segment_len);
  gdn_problem sp = *p;
  sp.segment_len = segment_len;
  return gdn_chunk_bwd_workspace(&sp, bytes);
}

gdn_status kda_segment_summary_bwd(const gdn_problem *pin, const void *q, const void *k,
                                   const float *g_cumsum, const void *beta, const float *A,
                                   const void *dO, int32_t segment_len, float *dS_ext, void *ws,
                                   size_t ws_bytes, void *stream) {
  gdn_status st = check_problem(pin, true);
  if (st != GDN_OK) return st;
  if (pin->layout != GDN_LAYOUT_BSND)
    return fail(GDN_ERR_UNSUPPORTED, "segment summaries take the BSND layout");
  if (segment_len <= 0 || segment_len % GDN_CHUNK != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len must be a positive multiple of 64, got %d",
                segment_len);
  gdn_problem sp = mapped_problem(pin);
  sp.segment_len = segment_len;
  const gdn_problem *p = &sp;
  REQUIRE_PTR(q, "q");
  REQUIRE_PTR(k, "k");
  REQUIRE_PTR(g_cumsum, "g_cumsum");
  REQUIRE_PTR(beta, "beta");
  REQUIRE_PTR(A, "A");
  REQUIRE_PTR(dO, "dO");
  REQUIRE_PTR(dS_ext, "dS_ext");
  const size_t maps = map_part_bytes(pin);
  const BwdWs L = bwd_ws_layout(p);
  if (!ws || ws_bytes < maps + L.total)
    return fail(GDN_ERR_WORKSPACE, "backward segment summary workspace needs %zu bytes, got %zu",
                maps + L.total, ws ? ws_bytes : (size_t)0);
  if (!aligned16(ws)) return fail(GDN_ERR_INVALID_ARGUMENT, "ws must be 16-byte aligned");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  if (p->T == 0) return ok();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (maps > 0) {  // the forward's mapped q, k and beta
    cudaError_t e = run_input_maps(pin, &q, &k, &beta, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "input map launch");
  }
  char *w = static_cast<char *>(ws) + maps;
  const int nseg = (int)div_up(p->T, segment_len);
  gdn::BwdArgs b{};
  b.q = q;
  b.k = k;
  b.beta = beta;
  b.dO = dO;
  b.g_cumsum = g_cumsum;
  b.A = A;
  b.dht = nullptr;  // every segment's reverse pass starts from a zero gradient at its exit
  b.dh0 = dS_ext;
  b.dh_chunks = reinterpret_cast<float *>(w + L.dh_chunks);
  b.dvnew = reinterpret_cast<float *>(w + L.dvnew);
  if (use_tensor_cores(p)) {  // the workspace holds bf16 tiles on this path
    b.dh_tiles = reinterpret_cast<__nv_bfloat16 *>(w + L.dh_chunks);
    b.dv_tiles = reinterpret_cast<__nv_bfloat16 *>(w + L.dvnew);
  }
  b.B = p->B;
  b.T = p->T;
  b.H = p->H;
  b.scale = eff_scale(p);
  b.use_exp2 = p->use_exp2;
  b.seg_len = segment_len;
  b.nseg = nseg;
  b.dev_flag = device_flag_ptr();
  cudaError_t e;
  if (use_tensor_cores(p)) {
    const gdn::UtArgs u = ut_args(p, k, nullptr, g_cumsum, beta, w + L.xw, nullptr, nullptr, b.dev_flag);
    if ((e = gdn::launch_ut_pair(u, A, (int)n_chunk_slots(p), s)) != cudaSuccess) return cuda_fail(e, "X pair launch");
    b.xw = u.xw;
    b.ftab = u.ftab;
    e = gdn::launch_tc_dhu(b, p->B * nseg, s);
  } else if (use_kda_tc(p)) {  // the prep's blobs (no v: the reverse recurrence does not read u)
    const gdn::KdaPrepArgs pa = kda_prep_args(p, q, k, nullptr, nullptr, g_cumsum, beta, w + L.xw, nullptr, nullptr,
                                              b.scale, b.dev_flag);
    if ((e = gdn::launch_kda_prep(pa, (int)n_chunk_slots(p), s)) != cudaSuccess) return cuda_fail(e, "KDA prep launch");
    b.blob = reinterpret_cast<const uint8_t *>(w + L.xw);
    e = gdn::launch_kda_dhu(b, p->B * nseg, s);
  } else {
    e = gdn::launch_bwd_dhu(b, p->gate_kind == GDN_GATE_PER_KEY, p->dtype == GDN_DTYPE_BF16, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "backward segment summary launch");
  return ok();
}

gdn_status kda_segment_merge_bwd(const gdn_problem *p, const float *dS_ext, const float *M,
                                 int32_t nseg, const float *dht, float *dS_exit, float *dh0,
                                 void *stream) {
  gdn_status st = check_problem(p, true);
  if (st != GDN_OK) return st;
  if (p->layout != GDN_LAYOUT_BSND)
    return fail(GDN_ERR_UNSUPPORTED, "segment merge takes the BSND layout");
  if (nseg < 1) return fail(GDN_ERR_INVALID_ARGUMENT, "nseg must be >= 1, got %d", nseg);
  REQUIRE_PTR(dS_ext, "dS_ext");
  REQUIRE_PTR(M, "M");
  REQUIRE_PTR(dS_exit, "dS_exit");
  OPTIONAL_PTR(dht, "dht");
  OPTIONAL_PTR(dh0, "dh0");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  gdn::MergeArgs a{dS_ext, M, dht, dS_exit, dh0, p->B * p->H, nseg, 1, device_flag_ptr()};
  cudaError_t e = gdn::launch_merge(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "adjoint segment merge launch");
  return ok();
}

gdn_status kda_segment_merge(const gdn_problem *p, const float *S_ext, const float *M,
                             int32_t nseg, const float *h0, float *S_init, float *ht,
                             void *stream) {
  gdn_status st = check_problem(p, true);
  if (st != GDN_OK) return st;
  if (p->layout != GDN_LAYOUT_BSND)
    return fail(GDN_ERR_UNSUPPORTED, "segment merge takes the BSND layout");
  if (nseg < 1) return fail(GDN_ERR_INVALID_ARGUMENT, "nseg must be >= 1, got %d", nseg);
  REQUIRE_PTR(S_ext, "S_ext");
  REQUIRE_PTR(M, "M");
  REQUIRE_PTR(S_init, "S_init");
  OPTIONAL_PTR(h0, "h0");
  OPTIONAL_PTR(ht, "ht");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  gdn::MergeArgs a{S_ext, M, h0, S_init, ht, p->B * p->H, nseg, 0, device_flag_ptr()};
  cudaError_t e = gdn::launch_merge(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "segment merge launch");
  return ok();
}

namespace {
// the problem of a one-call split forward: `p` with its segment length, checked
gdn_status split_problem(const gdn_problem *p, int32_t segment_len, gdn_problem *sp) {
  if (!p) return fail(GDN_ERR_INVALID_ARGUMENT, "problem is NULL");
  if (segment_len <= 0 || segment_len % GDN_CHUNK != 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len must be a positive multiple of 64, got %d",
                segment_len);
  *sp = *p;
  sp->segment_len = segment_len;
  gdn_status st = check_problem(sp, true);
  if (st != GDN_OK) return st;
  const gdn_problem m = mapped_problem(sp);
  if (m.layout != GDN_LAYOUT_BSND || !use_kda_tc(&m))
    return fail(GDN_ERR_UNSUPPORTED,
                "the one-call split forward takes bf16 inputs with a per-key gate in the BSND layout");
  return GDN_OK;
}
}  // namespace

gdn_status gdn_chunk_fwd_split_workspace(const gdn_problem *p, int32_t segment_len, size_t *bytes) {
  gdn_problem sp;
  gdn_status st = split_problem(p, segment_len, &sp);
  if (st != GDN_OK) return st;
  if (!bytes) return fail(GDN_ERR_INVALID_ARGUMENT, "bytes must not be NULL");
  const gdn_problem m = mapped_problem(&sp);
  *bytes = map_part_bytes(&sp) + blob_bytes(&m);
  return ok();
}

gdn_status gdn_chunk_fwd_split(const gdn_problem *pin, const void *q, const void *k, const void *v,
                               const float *g, const void *beta, const float *h0, int32_t segment_len,
                               void *o, float *ht, float *S_ext, float *M, float *S_init,
                               float *g_cumsum, float *A, float *h_chunks, void *ws, size_t ws_bytes,
                               void *stream) {
  gdn_problem sp;
  gdn_status st = split_problem(pin, segment_len, &sp);
  if (st != GDN_OK) return st;
  const gdn_problem mp = mapped_problem(&sp);
  const gdn_problem *p = &mp;
  if (p->T > 0) {
    REQUIRE_PTR(q, "q");
    REQUIRE_PTR(k, "k");
    REQUIRE_PTR(v, "v");
    REQUIRE_PTR(g, "g");
    REQUIRE_PTR(beta, "beta");
    REQUIRE_PTR(o, "o");
  }
  REQUIRE_PTR(S_ext, "S_ext");
  REQUIRE_PTR(M, "M");
  REQUIRE_PTR(S_init, "S_init");
  OPTIONAL_PTR(h0, "h0");
  OPTIONAL_PTR(ht, "ht");
  OPTIONAL_PTR(g_cumsum, "g_cumsum");
  OPTIONAL_PTR(A, "A");
  OPTIONAL_PTR(h_chunks, "h_chunks");
  const size_t maps = map_part_bytes(&sp);
  const size_t need = maps + blob_bytes(p);
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(GDN_ERR_WORKSPACE, "split forward workspace needs %zu bytes, got %zu", need,
                ws ? ws_bytes : (size_t)0);
  if (ws && !aligned16(ws)) return fail(GDN_ERR_INVALID_ARGUMENT, "ws must be 16-byte aligned");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  if (p->T == 0) return ok();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (maps > 0) {
    cudaError_t e = run_input_maps(&sp, &q, &k, &beta, ws, s);
    if (e != cudaSuccess) return cuda_fail(e, "input map launch");
  }
  void *blob = static_cast<char *>(ws) + maps;
  const int nseg = (int)div_up(p->T, segment_len);
  int *flag = device_flag_ptr();
  // 1. every chunk's operands, once for both passes (the summary reads w, u and the decays;
  //    the corrected run also the query-side operands)
  const gdn::KdaPrepArgs pa = kda_prep_args(p, q, k, v, g, nullptr, beta, blob, g_cumsum, A, eff_scale(p), flag);
  cudaError_t e = gdn::launch_kda_prep(pa, (int)n_chunk_slots(p), s);
  if (e != cudaSuccess) return cuda_fail(e, "KDA prep launch");
  // 2. segment summaries on [V | I] columns, as kda_segment_summary
  gdn::SimtFwdArgs a{};
  a.B = p->B;
  a.T = p->T;
  a.H = p->H;
  a.scale = eff_scale(p);
  a.use_exp2 = p->use_exp2;
  a.seg_len = segment_len;
  a.nseg = nseg;
  a.dev_flag = flag;
  a.S_ext = S_ext;
  a.M = M;
  a.summary = 1;
  if ((e = gdn::launch_kda_chain(kda_chain_args(a, blob), dim3(4, p->H, p->B * nseg), s)) != cudaSuccess)
    return cuda_fail(e, "segment summary launch");
  // 3. ordered merge from h0, as kda_segment_merge (the final state comes from step 4)
  gdn::MergeArgs ma{S_ext, M, h0, S_init, nullptr, p->B * p->H, nseg, 0, flag};
  if ((e = gdn::launch_merge(ma, s)) != cudaSuccess) return cuda_fail(e, "segment merge launch");
  // 4. every segment from its merged entry state, as gdn_chunk_fwd with segment_len
  a.S_ext = nullptr;
  a.M = nullptr;
  a.summary = 0;
  a.h0 = S_init;
  a.o = o;
  a.ht = ht;
  a.h_chunks = h_chunks;
  if ((e = gdn::launch_kda_chain(kda_chain_args(a, blob), dim3(2, p->H, p->B * nseg), s)) != cudaSuccess)
    return cuda_fail(e, "chunk forward launch");
  return ok();
}

namespace {
gdn_status check_frame(const frame_scan_problem *p, int *nseg) {
  if (!p) return fail(GDN_ERR_INVALID_ARGUMENT, "problem is NULL");
  if (p->BH < 1 || p->T < 1 || p->BH > 65535)
    return fail(GDN_ERR_INVALID_ARGUMENT, "need 1 <= BH <= 65535 and T >= 1 (got BH=%d T=%d)", p->BH, p->T);
  if (p->D != 32 && p->D != 64) return fail(GDN_ERR_UNSUPPORTED, "D must be 32 or 64, got %d", p->D);
  if (p->active < 0 || p->active > p->T)
    return fail(GDN_ERR_INVALID_ARGUMENT, "active must be 0 or in [1, T=%d], got %d", p->T, p->active);
  if (p->segment_len < 0)
    return fail(GDN_ERR_INVALID_ARGUMENT, "segment_len must be >= 0, got %d", p->segment_len);
  if ((int64_t)p->BH * p->T * p->D * p->D >= (int64_t)1 << 40)
    return fail(GDN_ERR_INVALID_ARGUMENT, "problem too large");
  *nseg = p->segment_len > 0 ? (int)(((int64_t)p->T + p->segment_len - 1) / p->segment_len) : 1;
  if ((int64_t)*nseg > 65535) return fail(GDN_ERR_INVALID_ARGUMENT, "more than 65535 segments");
  return GDN_OK;
}
size_t frame_ws_bytes(const frame_scan_problem *p, int nseg) {
  if (nseg <= 1) return 0;
  return (size_t)p->BH * nseg * (4 * (size_t)p->D * p->D + 2 * (size_t)p->D) * sizeof(float);
}
}  // namespace

gdn_status frame_scan_workspace(const frame_scan_problem *p, size_t *bytes) {
  int nseg = 1;
  gdn_status st = check_frame(p, &nseg);
  if (st != GDN_OK) return st;
  if (!bytes) return fail(GDN_ERR_INVALID_ARGUMENT, "bytes must not be NULL");
  *bytes = frame_ws_bytes(p, nseg);
  return ok();
}

gdn_status frame_scan_fwd(const frame_scan_problem *p, const float *W_kv, const float *U_kv,
                          const float *W_z, const float *u_z, const float *S0_kv,
                          const float *s0_z, float *S_kv_all, float *s_z_all, float *S_kv_last,
                          float *s_z_last, void *ws, size_t ws_bytes, void *stream) {
  int nseg = 1;
  gdn_status st = check_frame(p, &nseg);
  if (st != GDN_OK) return st;
  REQUIRE_PTR(W_kv, "W_kv");
  REQUIRE_PTR(U_kv, "U_kv");
  REQUIRE_PTR(W_z, "W_z");
  REQUIRE_PTR(u_z, "u_z");
  REQUIRE_PTR(S_kv_all, "S_kv_all");
  REQUIRE_PTR(s_z_all, "s_z_all");
  OPTIONAL_PTR(S0_kv, "S0_kv");
  OPTIONAL_PTR(s0_z, "s0_z");
  OPTIONAL_PTR(S_kv_last, "S_kv_last");
  OPTIONAL_PTR(s_z_last, "s_z_last");
  const size_t need = frame_ws_bytes(p, nseg);
  if (need > 0 && (!ws || ws_bytes < need))
    return fail(GDN_ERR_WORKSPACE, "frame scan workspace needs %zu bytes, got %zu", need, ws_bytes);
  if (need > 0) OPTIONAL_PTR(ws, "workspace");
  int dev;
  if ((st = check_device(&dev)) != GDN_OK) return st;
  gdn::FrameScanArgs a;
  memset(&a, 0, sizeof(a));
  a.W_kv = W_kv;
  a.U_kv = U_kv;
  a.W_z = W_z;
  a.u_z = u_z;
  a.S0 = S0_kv;
  a.z0 = s0_z;
  a.S_all = S_kv_all;
  a.z_all = s_z_all;
  a.S_last = S_kv_last;
  a.z_last = s_z_last;
  a.BH = p->BH;
  a.D = p->D;
  a.active = p->active;
  a.nseg = nseg;
  a.T = p->T;
  a.seg_len = nseg > 1 ? p->segment_len : p->T;
  a.dev_flag = device_flag_ptr();
  if (nseg > 1) {
    float *w = static_cast<float *>(ws);
    const size_t DD = (size_t)p->BH * nseg * p->D * p->D, Dn = (size_t)p->BH * nseg * p->D;
    a.h_kv = w;
    a.M_kv = w + DD;
    a.M_z = w + 2 * DD;
    a.S_init = w + 3 * DD;
    a.h_z = w + 4 * DD;
    a.z_init = w + 4 * DD + Dn;
  }
  cudaError_t e = gdn::launch_frame_scan(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "frame scan launch");
  return ok();
}

}  // extern "C"

namespace gdn {
gdn_status set_error(gdn_status st, const char *msg) {
  g_last_error = msg ? msg : "";
  return st;
}
}  // namespace gdn
