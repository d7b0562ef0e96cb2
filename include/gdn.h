/*
 * gdn.h -- C ABI of the GB300-native Gated DeltaNet (GDN) causal core.
 *
 * The library (libgdn.so, built for sm_103a) runs every step of the core in
 * its own CUDA kernels.  It never allocates device memory: every buffer,
 * including scratch ("workspace") space, is owned by the caller, and its size
 * is reported by gdn_workspace_size().  Every entry point is asynchronous on
 * the caller's stream (passed as a cudaStream_t cast to void*; NULL = the
 * legacy default stream); only argument validation runs on the host.  Errors
 * are returned as gdn_status codes; nothing is printed and nothing traps.
 *
 * Sources, by page title and section:
 *   [P1] "[6/8] feat(models): port Qwen3.5 / Qwen3-Next GDN to the head-sharded
 *        layer": "What" (grouped value heads, flat q/k/v layout),
 *        "Summary of an earlier run" (grouped-value accumulation of q/k grads).
 *   [P2] prime-rl #3860: "Summary" (shared GatedDeltaNet and
 *        ZeroCenteredRMSNorm; causal_conv1d with cu_seqlens; chunk op called
 *        with initial_state=None, output_final_state=False).
 *   [P3] "[main] feat(moe): Support gated delta net for Qwen3-Next (1/4)":
 *        "GDN args" (conv kernel 4, head dims 128, 16 k-heads, 32 v-heads),
 *        --apply-layernorm-1p (zero-centred norm), review comment on A_log.
 *
 * What the core computes (per packed token t of sequence n, v-head h, k-head
 * kh = h / (h_v/h_k)):
 *   conv:  xc = silu(sum_j w[c,j] x[t-3+j, c])    (zero / conv cache before
 *          the sequence start)                                   [P2][P3]
 *   l2:    q^ = q/sqrt(|q|^2+l2_eps) * d_k^-1/2,  k^ = k/sqrt(|k|^2+l2_eps)
 *   gates: g = -exp(A_log[h]) softplus(a + dt_bias[h]),  beta = sigmoid(b) [P3]
 *   rule:  S_t = exp(g_t) S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T,
 *          o_t = S_t q^_t,  S in fp32 [d_v x d_k]
 *   norm:  y = o / sqrt(mean(o^2) + norm_eps) * (1 + w) * gate(z),
 *          gate = silu (default) or sigmoid (dims.gate)          [P2][P3]
 *
 * Layouts (row-major, packed over tokens; T = total tokens, N = sequences,
 * C = 2*h_k*d_k + h_v*d_v conv channels, G = h_v/h_k):
 *   x, dx          [T, C]  io dtype; channels flat [q (h_k*d_k) | k (h_k*d_k) |
 *                  v (h_v*d_v)] (dims.layout = GDN_LAYOUT_FLAT, [P1] "What":
 *                  HF's flat layout) or group-major: for each k-head kh in
 *                  order, [q_kh | k_kh | v_{kh*G} .. v_{kh*G+G-1}], d channels
 *                  each (GDN_LAYOUT_GROUP, [P1] "What": q/k/v and the conv in
 *                  group-major layout).  conv_w, conv_state and their
 *                  gradients follow x's channel order.
 *   qkv, dqkv      [T, C]  fp32, always the flat order (conv+SiLU+L2 output,
 *                  an intermediate between the conv and the chunk entry points)
 *   a, b, da, db   [T, h_v] io dtype
 *   z, o, y, dz    [T, h_v, d_v] io dtype
 *   conv_w         [C, 4] fp32; tap 3 multiplies the current token
 *   conv_state     [N, C, 3] io dtype; [..., m] = input at position start-3+m
 *                  (gradients of conv states: fp32)
 *   A_log, dt_bias [h_v] fp32;  norm_w [d_v] fp32 (shared by all heads)
 *   states         [N, h_v, d_v, d_k] fp32
 *   cu_seqlens     int32 [N+1], cu[0] = 0, non-decreasing, cu[N] = T.  Entry
 *                  points that take it want the device copy AND a host copy
 *                  (validated on the host; the device copy is re-checked by
 *                  the first kernel, which sets the workspace status word).
 * All device pointers must be 16-byte aligned.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size, bad cu_seqlens */
    GDN_ERR_UNSUPPORTED = 2,   /* dims outside what this build implements            */
    GDN_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required         */
    GDN_ERR_CUDA = 4,          /* a CUDA launch or copy failed                       */
    GDN_ERR_DEVICE_TIMEOUT = 5,/* a bounded device wait gave up (status word)        */
    GDN_ERR_DEVICE_CHECK = 6   /* a device-side argument check failed (status word)  */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Problem dimensions.  This build supports d_k = d_v = 128, conv_k = 4,
 * chunk = 64, h_v % h_k == 0, io_dtype F32 or BF16, total_tokens < 2^31 and
 * (64-token chunks) * h_v * 128 < 2^31 (GDN_ERR_UNSUPPORTED otherwise). */
typedef struct {
    int32_t num_seqs;      /* N (the decode batch for gdn_recurrent_step)   */
    int64_t total_tokens;  /* T (= N for gdn_recurrent_step)                */
    int32_t h_k, h_v;      /* k-heads and v-heads; each k-head serves h_v/h_k */
    int32_t d_k, d_v;      /* head dims                                     */
    int32_t conv_k;        /* conv taps                                     */
    int32_t chunk;         /* chunk length of the WY form                   */
    int32_t io_dtype;      /* gdn_dtype of the activations                  */
    float l2_eps;          /* eps inside the q/k L2 norm (1e-6 typical)      */
    float norm_eps;        /* eps inside the gated RMSNorm (1e-6 typical)    */
    int32_t qkv_tf32;      /* 0 or 1, see below                               */
    int32_t gate;          /* gdn_gate: output gate of the gated norm         */
    int32_t layout;        /* gdn_layout: q/k/v channel order of x            */
} gdn_dims;

/* Output gate of the zero-centred gated RMSNorm ([P2] "Summary": the shared
 * GatedDeltaNet takes output_gate_type; Qwen3.5 uses silu, Qwen3.8 sigmoid). */
typedef enum { GDN_GATE_SILU = 0, GDN_GATE_SIGMOID = 1 } gdn_gate;

/* Channel order of x / dx / conv_w / conv states (see Layouts above). */
typedef enum { GDN_LAYOUT_FLAT = 0, GDN_LAYOUT_GROUP = 1 } gdn_layout;

/* qkv_tf32 = 1: the conv output qkv carries tf32 values (fp32 storage, 10
 * fraction bits).  gdn_conv1d_silu then rounds its output to nearest tf32, and
 * gdn_chunk_fwd / gdn_chunk_bwd, whose tensor-core products read q, k and v
 * at tf32 precision in any case, use the tiles as loaded instead of rounding
 * each one again; only their few elementwise uses of q, k, v (gate-gradient
 * dot products) see the rounded values.  With 1, the qkv passed to the chunk
 * entry points must be tf32 values (as gdn_conv1d_silu writes them): other
 * values reach the tensor cores truncated.  qkv_tf32 = 0: qkv is exact fp32
 * and rounded where the tensor cores read it.  Other entry points ignore it. */

/* Workspace kinds for gdn_workspace_size(). */
enum {
    GDN_WS_FWD = 0,        /* saved-for-backward buffer of gdn_chunk_fwd       */
    GDN_WS_BWD = 1,        /* scratch of gdn_chunk_bwd                          */
    GDN_WS_CONV_BWD = 2,   /* scratch of gdn_conv1d_silu_bwd                    */
    GDN_WS_NORM_BWD = 3    /* scratch of gdn_gated_rmsnorm_bwd                  */
};

/* Bytes of workspace `kind` needs for these dims and sequence lengths.
 * cu_seqlens_host may be NULL for GDN_WS_NORM_BWD. */
gdn_status gdn_workspace_size(const gdn_dims* dims, const int32_t* cu_seqlens_host, int kind,
                              size_t* bytes);

/* Causal depthwise conv1d (K = 4) + SiLU over all C channels, then per
 * (token, k-head) L2 normalisation of q (times d_k^-1/2) and k.  [P2] "Summary"
 * (causal_conv1d with cu_seqlens), [P3] "GDN args".  The conv restarts at every
 * sequence start from conv_state_in (NULL = zeros).  conv_state_out (nullable)
 * receives the last 3 inputs of each sequence (from conv_state_in where the
 * sequence is shorter than 3); it may alias conv_state_in.
 * Out: qkv_out [T, C] fp32. */
gdn_status gdn_conv1d_silu(const gdn_dims* dims, const int32_t* cu_seqlens,
                           const int32_t* cu_seqlens_host, const void* x, const float* conv_w,
                           const void* conv_state_in, float* qkv_out, void* conv_state_out,
                           void* stream);

/* Backward of gdn_conv1d_silu: given dqkv [T, C] fp32 (gradient of its qkv
 * output) and, if not NULL, dconv_state_out_grad [N, C, 3] fp32 (gradient of
 * its conv_state_out: a sequence split across calls hands the gradient of the
 * next call's conv_state_in back here), writes dx [T, C] (io dtype), dconv_w
 * [C, 4] fp32 and, if not NULL, dconv_state_in_out [N, C, 3] fp32, the
 * gradient of conv_state_in.  Recomputes the conv from x.  Scratch:
 * GDN_WS_CONV_BWD. */
gdn_status gdn_conv1d_silu_bwd(const gdn_dims* dims, const int32_t* cu_seqlens,
                               const int32_t* cu_seqlens_host, const void* x,
                               const float* conv_w, const void* conv_state_in, const float* dqkv,
                               const float* dconv_state_out_grad, void* dx_out,
                               float* dconv_w_out, float* dconv_state_in_out, void* ws,
                               size_t ws_bytes, void* stream);

/* Gated delta rule over packed varlen sequences in the chunked WY form
 * (chunk 64), with the gates computed from a, b, A_log, dt_bias, grouped value
 * heads read in place (no repeated q/k, [P1] "What"), and, when z != NULL, the
 * zero-centred gated RMSNorm fused into the output ([P2], [P3]).
 *   qkv: output of gdn_conv1d_silu.  initial_state: NULL = zeros.
 *   o_out (nullable when z != NULL), y_out (required when z != NULL),
 *   final_state_out (nullable; [P2] output_final_state).
 *   fwd_ws: GDN_WS_FWD bytes; holds what gdn_chunk_bwd reads back, so keep it
 *   unchanged until the backward has run. */
gdn_status gdn_chunk_fwd(const gdn_dims* dims, const int32_t* cu_seqlens,
                         const int32_t* cu_seqlens_host, const float* qkv, const void* a,
                         const void* b, const float* A_log, const float* dt_bias,
                         const float* initial_state, const void* z, const float* norm_w,
                         void* o_out, void* y_out, float* final_state_out, void* fwd_ws,
                         size_t fwd_ws_bytes, void* stream);

/* Backward of gdn_chunk_fwd (same inputs, same z/norm_w choice, the fwd_ws it
 * wrote).  dy: gradient of y (z != NULL) or of o (z == NULL), io dtype.
 * dfinal_state: nullable.  Writes dqkv_out [T, C] fp32 (gradients of q^, k^
 * summed over the v-heads of each group, [P1] "Summary of an earlier run", and
 * of v), da/db (io), and when not NULL dA_log/ddt_bias [h_v] fp32, dz (io),
 * dnorm_w [d_v] fp32, dinitial_state fp32.  All reductions run in a fixed
 * order: results are bitwise reproducible.  Scratch: GDN_WS_BWD. */
gdn_status gdn_chunk_bwd(const gdn_dims* dims, const int32_t* cu_seqlens,
                         const int32_t* cu_seqlens_host, const float* qkv, const void* a,
                         const void* b, const float* A_log, const float* dt_bias,
                         const float* initial_state, const void* z, const float* norm_w,
                         const void* fwd_ws, size_t fwd_ws_bytes, const void* dy,
                         const float* dfinal_state, float* dqkv_out, void* da_out, void* db_out,
                         float* dA_log_out, float* ddt_bias_out, void* dz_out,
                         float* dnorm_w_out, float* dinitial_state_out, void* bwd_ws,
                         size_t bwd_ws_bytes, void* stream);

/* Zero-centred gated RMSNorm, standalone ([P2] ZeroCenteredRMSNorm, [P3]
 * --apply-layernorm-1p): y = o * rsqrt(mean(o^2) + eps) * (1 + w) * gate(z)
 * per (token, v-head) over d_v.  rstd_out [T, h_v] fp32 is nullable. */
gdn_status gdn_gated_rmsnorm(const gdn_dims* dims, const void* o, const void* z,
                             const float* norm_w, void* y_out, float* rstd_out, void* stream);

/* Backward of gdn_gated_rmsnorm: do_out, dz_out (io dtype), dnorm_w_out [d_v]
 * fp32 (deterministic two-level sum).  Scratch: GDN_WS_NORM_BWD. */
gdn_status gdn_gated_rmsnorm_bwd(const gdn_dims* dims, const void* o, const void* z,
                                 const float* norm_w, const void* dy, void* do_out, void* dz_out,
                                 float* dnorm_w_out, void* ws, size_t ws_bytes, void* stream);

/* Allocation-free variant of gdn_gated_rmsnorm_bwd, for callers that cannot
 * hand the library a workspace: code running inside a serving runtime that
 * owns all device memory through its own pool and forbids new device
 * allocations after start-up, plugins that hold no allocator handle, and
 * loops that must not call cudaMalloc/cudaFree because cudaFree synchronises
 * the whole device.  Same inputs and outputs as gdn_gated_rmsnorm_bwd (the
 * caller still owns o, z, norm_w, dy, do_out, dz_out, dnorm_w_out); the
 * dnorm_w partial sums go to a 4 MiB array built into the library instead of
 * `ws`.  The pages have no counterpart of this entry point.
 *  - Size limit: total_tokens * h_v <= GDN_NOALLOC_NORM_BWD_MAX_ROWS, else
 *    GDN_ERR_WORKSPACE with nothing launched.
 *  - It calls no cudaMalloc / cudaFree and no allocating routine.
 *  - The first call in a device's CUDA context looks up the array's device
 *    address (cudaGetSymbolAddress, with that device current) and caches it
 *    under the context's unique ID; a context rebuilt later (cudaDeviceReset,
 *    or the primary context released and retained again) looks it up anew.
 *    Make that first call before any stream capture.
 *  - Every call on a device shares the one array: calls that overlap on the
 *    GPU (other streams, other host threads) race on it -- serialise them.
 *    The array keeps the last call's contents; every partial a call reads it
 *    first writes itself, so nothing needs clearing between calls. */
#define GDN_NOALLOC_NORM_BWD_MAX_ROWS 524288
gdn_status gdn_gated_rmsnorm_bwd_noalloc(const gdn_dims* dims, const void* o, const void* z,
                                         const float* norm_w, const void* dy, void* do_out,
                                         void* dz_out, float* dnorm_w_out, void* stream);

/* One recurrent decode step for a batch of num_seqs independent sequences
 * (total_tokens must equal num_seqs): updates conv_state [N, C, 3] and state
 * [N, h_v, d_v, d_k] (fp32) in place and writes y_t [N, h_v, d_v] and, if not
 * NULL, o_t.  x_t [N, C], a_t, b_t [N, h_v], z_t [N, h_v, d_v] in io dtype.
 * Equal to the last token of gdn_conv1d_silu + gdn_chunk_fwd run on the whole
 * sequence. */
gdn_status gdn_recurrent_step(const gdn_dims* dims, const void* x_t, const float* conv_w,
                              void* conv_state, const void* a_t, const void* b_t,
                              const float* A_log, const float* dt_bias, const void* z_t,
                              const float* norm_w, float* state, void* o_t, void* y_t,
                              void* stream);

/* Reads the device status word at the start of a GDN_WS_FWD / GDN_WS_BWD /
 * GDN_WS_CONV_BWD workspace (0 = OK, else a gdn_status) and clears it.
 * Synchronises `stream`.
 * GDN_ERR_DEVICE_TIMEOUT means a kernel gave up a bounded wait (about 2^24
 * polls) on a copy or a tensor-core product and returned early: that call's
 * outputs are invalid, and because a copy it had requested may still have
 * been in flight when it left, treat outputs of later launches on the same
 * device as untrusted until the CUDA context has been rebuilt. */
gdn_status gdn_read_status(void* ws, int32_t* code, void* stream);

/* Self-test of that failure path, safe to run on a healthy GPU: one CTA
 * allocates tensor memory, waits on an mbarrier with at most poll_limit polls
 * (1 .. 2^24), frees the tensor memory and returns.  arrive = 0: nothing ever
 * completes the barrier (no copy, product or arrive is pending on it), so the
 * wait gives up and GDN_ERR_DEVICE_TIMEOUT lands in the status word at the
 * start of `ws` (>= 4 bytes, 16-byte aligned; read it with gdn_read_status).
 * arrive = 1: the CTA arrives on the barrier first, the wait succeeds and the
 * status word is left as it was.  Nothing is in flight when the kernel
 * returns, so, unlike a real timeout, the device stays trustworthy. */
gdn_status gdn_selftest_bounded_wait(void* ws, size_t ws_bytes, int32_t poll_limit,
                                     int32_t arrive, void* stream);

/* Kernel launches the library has made in this process, over all entry points. */
int64_t gdn_launch_count(void);

/* Per-kernel timing, off by default.  While on (on != 0) every kernel launch
 * is bracketed by a pair of CUDA events recorded on that launch's stream. */
gdn_status gdn_profile_enable(int32_t on);

/* Waits for the timed launches recorded so far and writes one text line per
 * kernel name, "<name> <launches> <total_ms>\n", into buf (NUL-terminated);
 * then forgets them.  GDN_ERR_INVALID_ARG if buf is too small. */
gdn_status gdn_profile_report(char* buf, size_t buf_bytes);

/* Human-readable name of a status code (static storage). */
const char* gdn_status_string(gdn_status status);

/* ABI version of this header (major * 100 + minor); the major number changes
 * whenever a struct or a signature changes (2.00: gdn_dims.qkv_tf32; 3.00:
 * gdn_dims.gate and .layout, the conv backward's dconv_state_out_grad), the
 * minor number when an entry point is added. */
#define GDN_ABI_VERSION 300
int32_t gdn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
