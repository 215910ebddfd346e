/*
 * gdn.h -- C ABI of the GB300 (sm_103a) chunked gated-delta-rule scan.
 *
 * The operation (the gated delta rule, restated):
 *   S_t = (I - beta_t k_t k_t^T) Diag(a_t) S_{t-1} + beta_t k_t v_t^T,
 *   o_t = scale * S_t^T q_t,
 *   a_t = exp(g_t) (use_exp2 = 0) or 2^(g_t) (use_exp2 = 1),
 * with one log-gate per (token, head) (GDN, "gate_kind" SCALAR) or one per
 * (token, head, key channel) (KDA, PER_KEY), computed in 64-token chunks:
 * in-chunk cumulative log-gate, UT/WY transform A = (I + L)^-1, w, u, an fp32
 * inter-chunk state recurrence and the intra-chunk output. The argument list
 * follows the call contract of chunk_gated_delta_rule_fwd / _bwd in the GDN
 * Ascend C adapter ("Diff Coverage" page of hyper-parallel, _AscendCGDN):
 * q/k/v/g/beta, BSND or packed TND layout with cu_seqlens and chunk_indices,
 * chunk 64, state [K, V] (state_v_first = False), optional initial and final
 * state.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership: the caller allocates every input, output and workspace buffer.
 *   The library never allocates or frees memory, never synchronises a
 *   stream (gdn_device_status excepted) and launches only on `stream`.
 * Pointers: "device" pointers are CUDA device (or managed) memory of the
 *   current device; "host" pointers are ordinary host memory. Every device
 *   pointer must be 16-byte aligned; row strides are implied by the shapes
 *   (all tensors contiguous, row-major).
 * Layouts: BSND = [B, T, H, D]; TND = packed [T, H, D] (B must be 1) with
 *   document offsets. q, k are [.., H, K]; v, o, dO are [.., H, V]; beta is
 *   [.., H]; g is [.., H] (SCALAR) or [.., H, K] (PER_KEY). States are fp32
 *   [N, H, K, V] with N = B (BSND) or num_seqs (TND).
 * Element types: q, k, v, beta, o, dq, dk, dv, dbeta use `dtype` (fp32 or
 *   bf16); g, g_cumsum, A, states, dg are always fp32.
 * Errors: every argument is validated before any launch. On failure the
 *   call returns a nonzero gdn_status, launches nothing and leaves a message
 *   for gdn_last_error(). A failed launch returns GDN_ERR_CUDA. Kernels that
 *   detect an inconsistent input on the device (for example non-increasing
 *   device cu_seqlens) skip the affected work and raise a device flag that
 *   gdn_device_status() reports as GDN_ERR_DEVICE_CHECK.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARGUMENT = 1, /* contract violation (bad shape, null pointer, offsets) */
    GDN_ERR_UNSUPPORTED = 2,      /* valid but not provided (K or V != 128, chunk != 64, no sm_103 device) */
    GDN_ERR_WORKSPACE = 3,        /* workspace missing or smaller than the query returned */
    GDN_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    GDN_ERR_TIMEOUT = 5,          /* a bounded device-side wait ran out */
    GDN_ERR_DEVICE_CHECK = 6      /* a kernel found inconsistent device-side metadata */
} gdn_status;

enum { GDN_LAYOUT_BSND = 0, GDN_LAYOUT_TND = 1 };
enum { GDN_GATE_SCALAR = 0, GDN_GATE_PER_KEY = 1 };
enum { GDN_DTYPE_F32 = 0, GDN_DTYPE_BF16 = 1 };

/* Problem description shared by the entry points.
 *   B, T, H, K, V : batch, tokens per batch row (TND: total packed tokens),
 *                   heads, key width, value width. K = V = 128.
 *   layout        : GDN_LAYOUT_BSND or GDN_LAYOUT_TND.
 *   gate_kind     : GDN_GATE_SCALAR (GDN) or GDN_GATE_PER_KEY (KDA).
 *   dtype         : element type of q, k, v, beta and the token outputs.
 *   use_exp2      : 0 -> a = exp(g); 1 -> a = 2^g (the KDA stages use base 2).
 *   scale         : output scale; 0 selects K^-1/2 (the adapters' default).
 *   chunk_size    : must be 64 (the fused backends require chunk_size=64).
 *   use_qk_l2norm : q and k are raw; a prologue kernel normalises them,
 *                   x / sqrt(sum x^2 + 1e-6) per (token, head) row, into the
 *                   workspace before the chunk kernels (the KDA adapter's
 *                   use_qk_l2norm_in_kernel, epsilon 1e-6). The backward then
 *                   returns dq, dk w.r.t. the raw q, k.
 *   cu_seqlens    : TND only: device int32 [num_seqs + 1] document offsets,
 *                   validated beforehand with gdn_prepare_varlen.
 *   num_seqs      : TND only: number of documents.
 *   chunk_indices : TND only: device int32 [2 * num_chunks] (document, chunk)
 *                   pairs produced by gdn_prepare_varlen.
 *   num_chunks    : TND only: total chunks (sum of ceil(len / 64)).
 *   segment_len   : BSND only, 0 or a multiple of 64. When nonzero,
 *                   gdn_chunk_fwd treats every segment of segment_len tokens
 *                   as an independent run whose entry state is read from
 *                   h0 laid out [B, H, nseg, K, V] (the S_init produced by
 *                   kda_segment_merge): the correction run of the segment
 *                   split. ht then receives each batch row's final state.
 *   use_beta_sigmoid : beta is raw; the prologue maps it to 1 / (1 + exp(-beta))
 *                   (the KDA adapter's use_beta_sigmoid_in_kernel). The
 *                   backward then returns dbeta w.r.t. the raw beta.
 */
typedef struct gdn_problem {
    int32_t B, T, H, K, V;
    int32_t layout;
    int32_t gate_kind;
    int32_t dtype;
    int32_t use_exp2;
    float scale;
    int32_t chunk_size;
    int32_t use_qk_l2norm;
    const int32_t *cu_seqlens;
    int32_t num_seqs;
    const int32_t *chunk_indices;
    int32_t num_chunks;
    int32_t segment_len;
    int32_t use_beta_sigmoid;
} gdn_problem;

/* Thread-local text of the last failure in this thread ("" after success). */
const char *gdn_last_error(void);

/* Reads and clears the device-side error flag: synchronises `stream`.
 * Returns GDN_OK, GDN_ERR_DEVICE_CHECK or GDN_ERR_TIMEOUT. */
gdn_status gdn_device_status(void *stream);

/* Self-test of the bounded device-side waits (a diagnostic; the pages' kernels
 * have no counterpart). Every wait of the library's tensor-core kernels polls
 * its barrier a bounded number of times; when the budget runs out the kernel
 * raises the device flag, finishes or waits out its copies in flight, frees its
 * tensor memory and returns. This call launches one CTA on `stream` that waits
 * in that same way, with `polls` polls (1 .. GDN_SELFTEST_MAX_POLLS), on a
 * barrier that nothing arrives on, so the wait always runs out: afterwards
 * gdn_device_status() returns GDN_ERR_TIMEOUT (and clears the flag). Nothing
 * is left in flight and the context stays usable. Returns GDN_OK once the
 * kernel is launched, GDN_ERR_INVALID_ARGUMENT for a budget out of range. */
#define GDN_SELFTEST_MAX_POLLS (1u << 20)
gdn_status gdn_selftest_wait_timeout(uint32_t polls, void *stream);

/* Packed-sequence metadata (host only, no device work).
 * Defined by _packed_offsets / _packed_metadata of the Ascend C adapters
 * ("Diff Coverage" page): offsets must have at least two entries, start at
 * 0, end at total_tokens and strictly increase; else
 * GDN_ERR_INVALID_ARGUMENT. chunk_indices receives, for every document n in
 * order and every chunk c < ceil(len_n / 64), the pair (n, c).
 *   cu_seqlens_host   : host int32 [n_seq_plus_1], read only.
 *   chunk_indices_host: host int32 [2 * capacity] output, or NULL to only
 *                       count; capacity is *num_chunks on entry when
 *                       non-NULL (GDN_ERR_INVALID_ARGUMENT if too small).
 *   num_chunks        : out, number of chunks. */
gdn_status gdn_prepare_varlen(const int32_t *cu_seqlens_host, int32_t n_seq_plus_1,
                              int64_t total_tokens, int32_t *chunk_indices_host,
                              int32_t *num_chunks);

/* Workspace bytes gdn_chunk_fwd needs for `p` (0 is a valid answer). */
gdn_status gdn_chunk_fwd_workspace(const gdn_problem *p, size_t *bytes);

/* Chunked forward (the GDN forward's ten-slot contract, slots that are
 * enabled here: o, final_state, g_cumsum, A, h). All pointers device.
 *   q, k, v, g, beta : inputs (read only).
 *   h0       : nullable fp32 [N, H, K, V] initial state; with segment_len > 0
 *              it is [B, H, nseg, K, V] (entry state of every segment).
 *   o        : output, layout of v, element type `dtype`.
 *   ht       : nullable fp32 [N, H, K, V] final state.
 *   g_cumsum : nullable fp32, shape of g: in-chunk cumulative log-gate,
 *              restarting at every chunk and document start.
 *   A        : nullable fp32 [.., H, 64]: row i of the chunk's
 *              (I + L)^-1, L = strictly-lower(diag(beta)(K K^T (.) Gamma));
 *              beta is not folded in (the separate "beta_eff" slot).
 *   h_chunks : nullable fp32 entry state of every chunk:
 *              BSND [B, H, ceil(T/64), K, V]; TND [num_chunks, H, K, V] in
 *              chunk_indices order.
 *   ws, ws_bytes : workspace of at least gdn_chunk_fwd_workspace bytes.
 *   stream   : cudaStream_t (NULL = legacy default stream). */
gdn_status gdn_chunk_fwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                         const float *g, const void *beta, const float *h0, void *o, float *ht,
                         float *g_cumsum, float *A, float *h_chunks, void *ws, size_t ws_bytes,
                         void *stream);

/* Workspace bytes gdn_chunk_bwd needs for `p`. */
gdn_status gdn_chunk_bwd_workspace(const gdn_problem *p, size_t *bytes);

/* Chunked backward (the GDN backward's contract: inputs q, k, v, the saved
 * g_cumsum, beta and A, the output gradient and scale; first five result
 * slots dq, dk, dv, dbeta, dg). All pointers device.
 *   q, k, v, beta : forward inputs.
 *   g_cumsum, A   : the forward's saved slots (fp32). The local gradients, and
 *                   the state recompute of a scalar gate, take X from A (no
 *                   second solve), so A must be the forward's own, for the
 *                   same k, beta and g.
 *   dO            : output gradient, layout of v.
 *   h0            : nullable fp32 [N, H, K, V] initial state of the forward.
 *   dht           : nullable fp32 [N, H, K, V] gradient of the final state.
 *   dq, dk, dv, dbeta : outputs, element type `dtype`.
 *   dg            : fp32, shape of g: gradient w.r.t. the raw per-token
 *                   gate (not its cumulative sum).
 *   dh0           : nullable fp32 [N, H, K, V] gradient of h0.
 *   ws, ws_bytes  : workspace of at least gdn_chunk_bwd_workspace bytes.
 * With segment_len > 0 (BSND) this is the corrected backward of the segment
 * split: h0 is the S_init of every segment [B, H, nseg, K, V] (required), dht
 * the gradient at every segment's exit [B, H, nseg, K, V] (kda_segment_merge_bwd),
 * and dh0 receives the gradient at every segment's entry [B, H, nseg, K, V].
 * With use_qk_l2norm / use_beta_sigmoid the inputs are
 * the raw q, k, beta of the forward (A and g_cumsum its saved slots), and dq,
 * dk, dbeta are w.r.t. those raw inputs: the prologue recomputes the mapped
 * inputs into the workspace and an epilogue kernel applies the chain rules of
 * the maps to the outputs in place. */
gdn_status gdn_chunk_bwd(const gdn_problem *p, const void *q, const void *k, const void *v,
                         const float *g_cumsum, const void *beta, const float *A,
                         const void *dO, const float *h0, const float *dht, void *dq, void *dk,
                         void *dv, float *dg, void *dbeta, float *dh0, void *ws,
                         size_t ws_bytes, void *stream);

/* Backward without a caller workspace (the adapters this library follows have
 * no counterpart; this is a convenience of this library).
 * For callers that cannot allocate device memory: runtimes that plan every
 * device buffer at start-up and forbid allocation afterwards, and plugin
 * hosts that hand a library only its input and output buffers. Arguments,
 * outputs and numerics are those of gdn_chunk_bwd; the scratch lives in one
 * array of GDN_NOALLOC_SCRATCH_BYTES (64 MiB) of device memory inside the
 * library, which every GPU that loads the library holds until the process
 * exits. Nothing here allocates or frees memory.
 *   - Problems whose backward workspace (gdn_chunk_bwd_workspace) exceeds
 *     GDN_NOALLOC_SCRATCH_BYTES are rejected with GDN_ERR_WORKSPACE and a
 *     message giving both sizes, before any device work.
 *   - Every call looks up the array's device address on the current device
 *     (cudaGetSymbolAddress); nothing is cached between calls, so the address
 *     stays valid across a device reset. The first call on a device also
 *     loads the library's device code there; make it before any stream
 *     capture.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents; the backward writes every scratch element it reads in
 *     the same call, so no clearing is needed. Calls whose work overlaps on
 *     the GPU (other streams, other host threads) race on the array: order
 *     them, for example on one stream. */
#define GDN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
gdn_status gdn_chunk_bwd_noalloc(const gdn_problem *p, const void *q, const void *k,
                                 const void *v, const float *g_cumsum, const void *beta,
                                 const float *A, const void *dO, const float *h0,
                                 const float *dht, void *dq, void *dk, void *dv, float *dg,
                                 void *dbeta, float *dh0, void *stream);

/* Affine segment summary (state_summary.py kda_split_state_summary_kernel,
 * combined mode): for every batch row b, head h and segment s of
 * segment_len tokens (BSND, segment_len a multiple of 64; the last segment
 * may be shorter), the local state from a zero start and the transfer map
 * from the identity, so that  S_exit = M S_entry + S_ext.  q is not needed.
 *   k, v, g, beta : device inputs (g_cumsum is computed internally).
 *   S_ext         : device fp32 [B, H, nseg, K, V].
 *   M             : device fp32 [B, H, nseg, K, K].
 *   ws, ws_bytes  : workspace of at least kda_segment_summary_workspace bytes
 *                   (may be NULL when that is 0). */
gdn_status kda_segment_summary_workspace(const gdn_problem *p, int32_t segment_len,
                                         size_t *bytes);
gdn_status kda_segment_summary(const gdn_problem *p, const void *k, const void *v,
                               const float *g, const void *beta, int32_t segment_len,
                               float *S_ext, float *M, void *ws, size_t ws_bytes, void *stream);

/* Backward segment summary (state_summary.py kda_state_grad_ext_kernel): for
 * every batch row b, head h and segment s of segment_len tokens (BSND), the
 * gradient of the segment's entry state from the segment's own outputs alone,
 * i.e. the reverse recurrence dv_new = kgl dh + scale A_qk^T dO,
 * dh <- Diag(b^(G_last)) dh + scale Qg^T dO - w^T dv_new run over the segment
 * from a zero gradient at its exit. It needs no forward state, so every segment
 * runs at once. The gradient flows across segments through the forward summary's
 * transfer maps transposed (kda_segment_merge_bwd).
 *   q, k, g_cumsum, beta, A, dO : as for gdn_chunk_bwd (v is not needed).
 *   dS_ext        : device fp32 [B, H, nseg, K, V].
 *   ws, ws_bytes  : at least kda_segment_summary_bwd_workspace bytes. */
gdn_status kda_segment_summary_bwd_workspace(const gdn_problem *p, int32_t segment_len,
                                             size_t *bytes);
gdn_status kda_segment_summary_bwd(const gdn_problem *p, const void *q, const void *k,
                                   const float *g_cumsum, const void *beta, const float *A,
                                   const void *dO, int32_t segment_len, float *dS_ext, void *ws,
                                   size_t ws_bytes, void *stream);

/* Adjoint of the ordered merge (SANA distributed_scan.py,
 * _CPAllGatherMerge.backward; the "Diff Coverage" page's state-summary apply
 * helpers, backward): from the last segment to the first, in fp32,
 *   dS_exit_{nseg-1} = dht (or 0),  dS_entry_s = M_s^T dS_exit_s + dS_ext_s,
 *   dS_exit_{s-1} = dS_entry_s.
 *   dS_ext, M : device fp32 [B, H, nseg, K, V] (kda_segment_summary_bwd) and
 *               [B, H, nseg, K, K] (kda_segment_summary).
 *   dht       : nullable device fp32 [B, H, K, V].
 *   dS_exit   : device fp32 [B, H, nseg, K, V], the gradient at every segment's
 *               exit (the dht of gdn_chunk_bwd in segment mode).
 *   dh0       : nullable device fp32 [B, H, K, V], the gradient of the initial
 *               state (dS_entry_0). */
gdn_status kda_segment_merge_bwd(const gdn_problem *p, const float *dS_ext, const float *M,
                                 int32_t nseg, const float *dht, float *dS_exit, float *dh0,
                                 void *stream);

/* Ordered merge of segment summaries (apply_kda_state_summary on the
 * "Diff Coverage" page; _exclusive_prefix_compose in SANA's
 * distributed_scan.py): S_init_0 = h0 (or 0), S_init_{s+1} = M_s S_init_s
 * + S_ext_s, in fp32.
 *   S_ext, M : device fp32 [B, H, nseg, K, V] and [B, H, nseg, K, K].
 *   h0       : nullable device fp32 [B, H, K, V].
 *   S_init   : device fp32 [B, H, nseg, K, V], entry state of every segment.
 *   ht       : nullable device fp32 [B, H, K, V], the state after the last
 *              segment. */
gdn_status kda_segment_merge(const gdn_problem *p, const float *S_ext, const float *M,
                             int32_t nseg, const float *h0, float *S_init, float *ht,
                             void *stream);

/* The whole split forward in one call, for bf16 inputs with a per-key gate in
 * the BSND layout: the segment summaries (as kda_segment_summary), their ordered
 * merge from h0 (as kda_segment_merge) and the corrected run of every segment from
 * its merged entry state (as gdn_chunk_fwd with segment_len) -- the split of the
 * long-context forward over the SMs on the state_summary.py and "Diff Coverage"
 * pages (kda_split_state_summary_kernel, apply_kda_state_summary, the KDA state
 * CP's forward). The chunk preparation (gated Gram matrices, the UT solve, w, u and
 * the scaled operands) runs once and serves both passes, where the three calls run
 * it twice; every output equals theirs bit for bit. All pointers device.
 *   q, k, v, g, beta, o, g_cumsum, A, h_chunks : as for gdn_chunk_fwd
 *                   (h_chunks in the BSND layout; g_cumsum, A, h_chunks nullable).
 *   h0            : nullable fp32 [B, H, K, V], the state before the first segment.
 *   segment_len   : a positive multiple of 64 (the last segment may be shorter).
 *   ht            : nullable fp32 [B, H, K, V], the state after the last segment.
 *   S_ext, M      : fp32 [B, H, nseg, K, V] and [B, H, nseg, K, K], the summaries.
 *   S_init        : fp32 [B, H, nseg, K, V], the entry state of every segment.
 *   ws, ws_bytes  : at least gdn_chunk_fwd_split_workspace bytes.
 * Other dtypes, gate kinds and layouts return GDN_ERR_UNSUPPORTED (use the three
 * calls); p->segment_len is ignored (the argument sets it). */
gdn_status gdn_chunk_fwd_split_workspace(const gdn_problem *p, int32_t segment_len, size_t *bytes);
gdn_status gdn_chunk_fwd_split(const gdn_problem *p, const void *q, const void *k, const void *v,
                               const float *g, const void *beta, const float *h0,
                               int32_t segment_len, void *o, float *ht, float *S_ext, float *M,
                               float *S_init, float *g_cumsum, float *A, float *h_chunks, void *ws,
                               size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Dense per-token transition scan (SANA, distributed_scan.py page:
 * cp_frame_gdn_scan and its local scan). For each of BH independent sequences of
 * T positions, with D x D transitions, in fp32:
 *   KV state, right multiply:  S_kv[t] = S_kv[t-1] W_kv[t] + U_kv[t]
 *   Z state, left multiply:    s_z[t]  = W_z[t] s_z[t-1] + u_z[t]
 * from S_kv[-1] = S0_kv (or 0) and s_z[-1] = s0_z (or 0). With active > 0 (the
 * page's truncate_to_active), positions t >= active leave both states unchanged
 * (the page sets W = I and U = 0 there): their outputs repeat the state of
 * position active-1, which is also the terminal state.
 * With segment_len > 0 a sequence runs as ceil(T / segment_len) segments on
 * different SMs: each segment's final state from zero and transition product
 * (M_kv = W_kv[a] ... W_kv[b-1], M_z = W_z[b-1] ... W_z[a]), their ordered
 * composition into every segment's entry state (S_init_{j+1} = S_init_j M_kv_j
 * + h_kv_j, s_init_{j+1} = M_z_j s_init_j + h_z_j, the page's exclusive prefix
 * composition), then every segment from its entry state: the page's context-
 * parallel scan, with its ranks as the SMs of one GPU.
 *   BH, T, D     : sequences (at most 65535), positions, state width (D = 32
 *                  or 64).
 *   active       : 0 (every position) or 1 <= active <= T.
 *   segment_len  : 0 (one pass per sequence) or >= 1.                         */
typedef struct frame_scan_problem {
    int32_t BH;
    int32_t T;
    int32_t D;
    int32_t active;
    int32_t segment_len;
} frame_scan_problem;

/* Workspace bytes of frame_scan_fwd: 0 for one pass, else
 * BH * nseg * (4 D^2 + 2 D) * 4 (the segments' summaries and entry states). */
gdn_status frame_scan_workspace(const frame_scan_problem *p, size_t *bytes);

/*   W_kv, U_kv, W_z : device fp32 [BH, T, D, D], row-major D x D per position.
 *   u_z             : device fp32 [BH, T, D].
 *   S0_kv, s0_z     : nullable device fp32 [BH, D, D], [BH, D] initial states.
 *   S_kv_all, s_z_all : device fp32 [BH, T, D, D], [BH, T, D]: every position's
 *                   state (outputs).
 *   S_kv_last, s_z_last : nullable device fp32 [BH, D, D], [BH, D]: the
 *                   terminal states (position active-1, or T-1).
 *   workspace       : device, frame_scan_workspace() bytes (may be NULL when 0).
 * Errors: GDN_ERR_INVALID_ARGUMENT (shapes, null or unaligned pointers, active
 * or segment_len out of range), GDN_ERR_UNSUPPORTED (D not 32 or 64),
 * GDN_ERR_WORKSPACE, GDN_ERR_CUDA. A bounded wait that runs out raises the
 * device flag (GDN_ERR_TIMEOUT from gdn_device_status). */
gdn_status frame_scan_fwd(const frame_scan_problem *p, const float *W_kv, const float *U_kv,
                          const float *W_z, const float *u_z, const float *S0_kv,
                          const float *s0_z, float *S_kv_all, float *s_z_all, float *S_kv_last,
                          float *s_z_last, void *workspace, size_t workspace_bytes,
                          void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
