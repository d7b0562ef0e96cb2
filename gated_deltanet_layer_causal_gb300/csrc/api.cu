// C ABI of the GDN library (declared in include/gdn.h): argument validation on
// the host, workspace carving, and kernel launches on the caller's stream.
// Nothing here allocates device memory, prints, or synchronises (except
// gdn_read_status, which by definition reads a device word back).
#include <cuda_runtime.h>

#include <cstring>

#include "../../include/gdn.h"
#include "common.cuh"
#include "kernels.h"

using namespace gdn;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_dims(const gdn_dims* d) {
    if (d == nullptr) return GDN_ERR_INVALID_ARG;
    if (d->num_seqs < 0 || d->total_tokens < 0 || d->h_k <= 0 || d->h_v <= 0)
        return GDN_ERR_INVALID_ARG;
    if (d->h_v % d->h_k != 0) return GDN_ERR_INVALID_ARG;
    if (d->d_k != kD || d->d_v != kD || d->conv_k != kConvK || d->chunk != kChunk)
        return GDN_ERR_UNSUPPORTED;
    if (d->io_dtype != GDN_F32 && d->io_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
    if (d->total_tokens >= (int64_t)1 << 31) return GDN_ERR_UNSUPPORTED;
    if (!(d->l2_eps >= 0.f) || !(d->norm_eps >= 0.f)) return GDN_ERR_INVALID_ARG;
    if (d->qkv_tf32 != 0 && d->qkv_tf32 != 1) return GDN_ERR_INVALID_ARG;
    if (d->gate != GDN_GATE_SILU && d->gate != GDN_GATE_SIGMOID) return GDN_ERR_INVALID_ARG;
    if (d->layout != GDN_LAYOUT_FLAT && d->layout != GDN_LAYOUT_GROUP) return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

// Validates the host copy of cu_seqlens and counts the 64-token chunks.
gdn_status check_cu(const gdn_dims* d, const int32_t* cu, int* nt) {
    if (cu == nullptr) return GDN_ERR_INVALID_ARG;
    if (cu[0] != 0 || (int64_t)cu[d->num_seqs] != d->total_tokens) return GDN_ERR_INVALID_ARG;
    int64_t chunks = 0;
    for (int n = 0; n < d->num_seqs; n++) {
        int64_t L = (int64_t)cu[n + 1] - cu[n];
        if (L < 0) return GDN_ERR_INVALID_ARG;
        chunks += (L + kChunk - 1) / kChunk;
    }
    // chunk-start state rows (chunk, head, row) are tensor-map coordinates: int32
    if (chunks * d->h_v * kD >= (int64_t)1 << 31) return GDN_ERR_UNSUPPORTED;
    *nt = (int)chunks;
    return GDN_OK;
}

int channels(const gdn_dims* d) { return (2 * d->h_k + d->h_v) * kD; }

ConvArgs conv_args(const gdn_dims* d, const int32_t* cu, const void* x, const float* conv_w,
                   const void* cs_in) {
    ConvArgs a{};
    a.bf16 = d->io_dtype == GDN_BF16;
    a.group_major = d->layout == GDN_LAYOUT_GROUP;
    a.N = d->num_seqs;
    a.C = channels(d);
    a.hk = d->h_k;
    a.hv = d->h_v;
    a.T = d->total_tokens;
    a.cu = cu;
    a.x = x;
    a.w = conv_w;
    a.cs_in = cs_in;
    a.l2_eps = d->l2_eps;
    a.q_scale = 1.f / sqrtf((float)kD);
    return a;
}

// ---------------------------------------------------------------- workspace carving
struct Carver {
    char* base;
    size_t off = 0;
    template <class T> T* take(size_t count) {
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off = align_up(off + count * sizeof(T));
        return p;
    }
};

FwdSaved carve_fwd(void* ws, const gdn_dims* d, int NT, size_t* bytes) {
    Carver c{static_cast<char*>(ws)};
    const size_t T = (size_t)d->total_tokens, H = (size_t)d->h_v;
    FwdSaved s;
    s.status = c.take<int32_t>(kAlign / 4);
    s.chunks = c.take<ChunkInfo>((size_t)NT);
    s.seq_chunk = c.take<int32_t>((size_t)d->num_seqs + 1);
    s.T = d->total_tokens;
    s.qkv_tf32 = d->qkv_tf32;
    s.gam = c.take<float>(T * H);
    s.beta = c.take<float>(T * H);
    s.W = c.take<float>(T * H * kD);
    s.U = c.take<float>(T * H * kD);
    s.S0 = c.take<float>((size_t)NT * H * kD * kD);
    s.Tm = c.take<float>((size_t)NT * H * 2 * 64 * 64);
    s.o = c.take<float>(T * H * kD);
    s.rstd = c.take<float>(T * H);
    *bytes = c.off;
    return s;
}

BwdScratch carve_bwd(void* ws, const gdn_dims* d, int NT, int32_t** status, size_t* bytes) {
    Carver c{static_cast<char*>(ws)};
    const size_t T = (size_t)d->total_tokens, H = (size_t)d->h_v;
    BwdScratch s;
    *status = c.take<int32_t>(kAlign / 4);
    s.status = *status;
    s.dO = c.take<float>(T * H * kD);
    s.dU = c.take<float>(T * H * kD);
    s.dQv = c.take<float>(T * (size_t)d->h_k * kD);    // per k-head (state-facing groups)
    s.dKv = c.take<float>(T * (size_t)d->h_k * kD);
    s.dQv2 = c.take<float>(T * (size_t)d->h_k * kD);   // per k-head (the P / dP groups)
    s.dKv2 = c.take<float>(T * (size_t)d->h_k * kD);
    s.dKv3 = c.take<float>(T * H * kD);
    s.dUl = s.dKv3;   // dU_local until the WY kernel writes its dK part there
    s.dW = c.take<float>(T * H * kD);
    s.dS = c.take<float>((size_t)NT * H * kD * kD);
    s.dgam = c.take<float>(T * H);
    s.dgam2 = c.take<float>(T * H);
    s.dgs = c.take<float>(T * H);
    s.dp_next = c.take<int32_t>(kAlign / 4);
    // dnorm_w partials [NT*H][kD], gate partials [NT*H][2], column-sum stage [512][kD]
    s.nw_part = c.take<float>((size_t)NT * H * kD + (size_t)NT * H * 2 + 512 * kD);
    *bytes = c.off;
    return s;
}

size_t conv_bwd_bytes(const gdn_dims* d) {
    return kAlign + align_up((size_t)conv_bwd_parts(d->total_tokens) * channels(d) * kConvK *
                             sizeof(float));
}

size_t norm_bwd_bytes(const gdn_dims* d) {
    int64_t rows = d->total_tokens * d->h_v;
    return align_up((size_t)norm_bwd_parts(rows) * kD * sizeof(float));
}

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

#define GDN_TRY(expr)                        \
    do {                                     \
        gdn_status _s = (expr);              \
        if (_s != GDN_OK) return _s;         \
    } while (0)

#define GDN_NEED(cond)                                     \
    do {                                                   \
        if (!(cond)) return GDN_ERR_INVALID_ARG;           \
    } while (0)

}  // namespace

extern "C" {

int32_t gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT";
        case GDN_ERR_DEVICE_CHECK: return "GDN_ERR_DEVICE_CHECK";
    }
    return "GDN_ERR_UNKNOWN";
}

gdn_status gdn_workspace_size(const gdn_dims* dims, const int32_t* cu_host, int kind,
                              size_t* bytes) {
    GDN_TRY(check_dims(dims));
    GDN_NEED(bytes != nullptr);
    if (kind == GDN_WS_NORM_BWD) {
        *bytes = norm_bwd_bytes(dims);
        return GDN_OK;
    }
    int NT = 0;
    GDN_TRY(check_cu(dims, cu_host, &NT));
    int32_t* st;
    switch (kind) {
        case GDN_WS_FWD: carve_fwd(nullptr, dims, NT, bytes); return GDN_OK;
        case GDN_WS_BWD: carve_bwd(nullptr, dims, NT, &st, bytes); return GDN_OK;
        case GDN_WS_CONV_BWD: *bytes = conv_bwd_bytes(dims); return GDN_OK;
    }
    return GDN_ERR_INVALID_ARG;
}

gdn_status gdn_conv1d_silu(const gdn_dims* dims, const int32_t* cu, const int32_t* cu_host,
                           const void* x, const float* conv_w, const void* cs_in, float* qkv,
                           void* cs_out, void* stream) {
    GDN_TRY(check_dims(dims));
    int NT;
    GDN_TRY(check_cu(dims, cu_host, &NT));
    GDN_NEED(cu && aligned16(x) && x && conv_w && aligned16(conv_w) && qkv && aligned16(qkv));
    GDN_NEED(!cs_in || aligned16(cs_in));
    if (dims->num_seqs == 0) return GDN_OK;
    ConvArgs a = conv_args(dims, cu, x, conv_w, cs_in);
    a.qkv = qkv;
    a.cs_out = cs_out;
    a.round_tf32 = dims->qkv_tf32 != 0;
    return cuda_status(launch_conv_fwd(a, (cudaStream_t)stream));
}

gdn_status gdn_conv1d_silu_bwd(const gdn_dims* dims, const int32_t* cu, const int32_t* cu_host,
                               const void* x, const float* conv_w, const void* cs_in,
                               const float* dqkv, const float* dcs_out, void* dx, float* dconv_w,
                               float* dcs, void* ws, size_t ws_bytes, void* stream) {
    GDN_TRY(check_dims(dims));
    int NT;
    GDN_TRY(check_cu(dims, cu_host, &NT));
    GDN_NEED(cu && x && aligned16(x) && conv_w && aligned16(conv_w) && dqkv && aligned16(dqkv));
    GDN_NEED(dx && aligned16(dx) && dconv_w && (!cs_in || aligned16(cs_in)));
    if (ws == nullptr || ws_bytes < conv_bwd_bytes(dims)) return GDN_ERR_WORKSPACE;
    if (dims->num_seqs == 0) return GDN_OK;
    ConvArgs a = conv_args(dims, cu, x, conv_w, cs_in);
    a.dqkv = dqkv;
    a.dcs_out = dcs_out;
    a.dx = dx;
    a.dw = dconv_w;
    a.wpart = reinterpret_cast<float*>(static_cast<char*>(ws) + kAlign);
    a.dcs = dcs;
    return cuda_status(launch_conv_bwd(a, (cudaStream_t)stream));
}

static gdn_status fill_chunk_args(ChunkArgs& a, const gdn_dims* dims, int NT, const int32_t* cu,
                                  const float* qkv, const void* av, const void* bv,
                                  const float* A_log, const float* dt_bias, const float* S_init,
                                  const void* z, const float* norm_w) {
    GDN_NEED(cu && qkv && aligned16(qkv) && av && bv && A_log && dt_bias);
    GDN_NEED(!S_init || aligned16(S_init));
    GDN_NEED(!z || (aligned16(z) && norm_w && aligned16(norm_w)));
    a.bf16 = dims->io_dtype == GDN_BF16;
    a.N = dims->num_seqs;
    a.NT = NT;
    a.hk = dims->h_k;
    a.hv = dims->h_v;
    a.T = dims->total_tokens;
    a.cu = cu;
    a.qkv = qkv;
    a.a = av;
    a.b = bv;
    a.A_log = A_log;
    a.dt_bias = dt_bias;
    a.S_init = S_init;
    a.z = z;
    a.norm_w = norm_w;
    a.norm_eps = dims->norm_eps;
    a.gate = dims->gate;
    return GDN_OK;
}

gdn_status gdn_chunk_fwd(const gdn_dims* dims, const int32_t* cu, const int32_t* cu_host,
                         const float* qkv, const void* av, const void* bv, const float* A_log,
                         const float* dt_bias, const float* S_init, const void* z,
                         const float* norm_w, void* o_out, void* y_out, float* S_final,
                         void* fwd_ws, size_t fwd_ws_bytes, void* stream) {
    GDN_TRY(check_dims(dims));
    int NT;
    GDN_TRY(check_cu(dims, cu_host, &NT));
    ChunkArgs a{};
    GDN_TRY(fill_chunk_args(a, dims, NT, cu, qkv, av, bv, A_log, dt_bias, S_init, z, norm_w));
    GDN_NEED(!o_out || aligned16(o_out));
    GDN_NEED(z ? (y_out && aligned16(y_out)) : (o_out != nullptr));
    GDN_NEED(!S_final || aligned16(S_final));
    size_t need;
    carve_fwd(nullptr, dims, NT, &need);
    if (fwd_ws == nullptr || fwd_ws_bytes < need || !aligned16(fwd_ws)) return GDN_ERR_WORKSPACE;
    if (dims->num_seqs == 0) return GDN_OK;
    a.sv = carve_fwd(fwd_ws, dims, NT, &need);
    a.o_out = o_out;
    a.y_out = y_out;
    a.S_final = S_final;
    cudaStream_t st = (cudaStream_t)stream;
    GDN_TRY(cuda_status(launch_plan(cu, a.N, a.T, NT, a.sv, st)));
    return cuda_status(launch_chunk_fwd(a, st));
}

gdn_status gdn_chunk_bwd(const gdn_dims* dims, const int32_t* cu, const int32_t* cu_host,
                         const float* qkv, const void* av, const void* bv, const float* A_log,
                         const float* dt_bias, const float* S_init, const void* z,
                         const float* norm_w, const void* fwd_ws, size_t fwd_ws_bytes,
                         const void* dy, const float* dS_final, float* dqkv, void* da, void* db,
                         float* dA_log, float* ddt_bias, void* dz, float* dnorm_w, float* dS_init,
                         void* bwd_ws, size_t bwd_ws_bytes, void* stream) {
    GDN_TRY(check_dims(dims));
    int NT;
    GDN_TRY(check_cu(dims, cu_host, &NT));
    ChunkArgs a{};
    GDN_TRY(fill_chunk_args(a, dims, NT, cu, qkv, av, bv, A_log, dt_bias, S_init, z, norm_w));
    GDN_NEED(dy && aligned16(dy) && dqkv && aligned16(dqkv) && da && db);
    GDN_NEED(!z || (dz && aligned16(dz) && dnorm_w));
    GDN_NEED(!dS_final || aligned16(dS_final));
    GDN_NEED(!dS_init || aligned16(dS_init));
    size_t need_f, need_b;
    carve_fwd(nullptr, dims, NT, &need_f);
    int32_t* status;
    carve_bwd(nullptr, dims, NT, &status, &need_b);
    if (fwd_ws == nullptr || fwd_ws_bytes < need_f) return GDN_ERR_WORKSPACE;
    if (bwd_ws == nullptr || bwd_ws_bytes < need_b || !aligned16(bwd_ws)) return GDN_ERR_WORKSPACE;
    if (dims->num_seqs == 0) return GDN_OK;
    a.sv = carve_fwd(const_cast<void*>(fwd_ws), dims, NT, &need_f);
    BwdScratch w = carve_bwd(bwd_ws, dims, NT, &status, &need_b);
    a.dy = dy;
    a.dS_final = dS_final;
    a.dqkv = dqkv;
    a.da = da;
    a.db = db;
    a.dA_log = dA_log;
    a.ddt_bias = ddt_bias;
    a.dz = dz;
    a.dnorm_w = dnorm_w;
    a.dS_init = dS_init;
    cudaStream_t st = (cudaStream_t)stream;
    cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    return cuda_status(launch_chunk_bwd(a, w, st));
}

gdn_status gdn_gated_rmsnorm(const gdn_dims* dims, const void* o, const void* z,
                             const float* norm_w, void* y, float* rstd, void* stream) {
    GDN_TRY(check_dims(dims));
    GDN_NEED(o && aligned16(o) && z && aligned16(z) && norm_w && aligned16(norm_w) && y &&
             aligned16(y));
    NormArgs a{};
    a.bf16 = dims->io_dtype == GDN_BF16;
    a.gate = dims->gate;
    a.rows = dims->total_tokens * dims->h_v;
    a.o = o;
    a.z = z;
    a.w = norm_w;
    a.eps = dims->norm_eps;
    a.y = y;
    a.rstd = rstd;
    return cuda_status(launch_norm_fwd(a, (cudaStream_t)stream));
}

gdn_status gdn_gated_rmsnorm_bwd(const gdn_dims* dims, const void* o, const void* z,
                                 const float* norm_w, const void* dy, void* d_o, void* dz,
                                 float* dnorm_w, void* ws, size_t ws_bytes, void* stream) {
    GDN_TRY(check_dims(dims));
    GDN_NEED(o && aligned16(o) && z && aligned16(z) && norm_w && aligned16(norm_w));
    GDN_NEED(dy && aligned16(dy) && d_o && aligned16(d_o) && dz && aligned16(dz) && dnorm_w);
    if (ws == nullptr || ws_bytes < norm_bwd_bytes(dims) || !aligned16(ws))
        return GDN_ERR_WORKSPACE;
    NormArgs a{};
    a.bf16 = dims->io_dtype == GDN_BF16;
    a.gate = dims->gate;
    a.rows = dims->total_tokens * dims->h_v;
    a.o = o;
    a.z = z;
    a.w = norm_w;
    a.eps = dims->norm_eps;
    a.dy = dy;
    a.d_o = d_o;
    a.dz = dz;
    a.dw = dnorm_w;
    a.part = static_cast<float*>(ws);
    return cuda_status(launch_norm_bwd(a, (cudaStream_t)stream));
}

gdn_status gdn_gated_rmsnorm_bwd_noalloc(const gdn_dims* dims, const void* o, const void* z,
                                         const float* norm_w, const void* dy, void* d_o,
                                         void* dz, float* dnorm_w, void* stream) {
    GDN_TRY(check_dims(dims));
    GDN_NEED(o && aligned16(o) && z && aligned16(z) && norm_w && aligned16(norm_w));
    GDN_NEED(dy && aligned16(dy) && d_o && aligned16(d_o) && dz && aligned16(dz) && dnorm_w);
    if (dims->total_tokens * dims->h_v > (int64_t)norm_bwd_noalloc_max_rows())
        return GDN_ERR_WORKSPACE;
    NormArgs a{};
    a.bf16 = dims->io_dtype == GDN_BF16;
    a.gate = dims->gate;
    a.rows = dims->total_tokens * dims->h_v;
    a.o = o;
    a.z = z;
    a.w = norm_w;
    a.eps = dims->norm_eps;
    a.dy = dy;
    a.d_o = d_o;
    a.dz = dz;
    a.dw = dnorm_w;
    return cuda_status(launch_norm_bwd_noalloc(a, (cudaStream_t)stream));
}

gdn_status gdn_recurrent_step(const gdn_dims* dims, const void* x_t, const float* conv_w,
                              void* conv_state, const void* a_t, const void* b_t,
                              const float* A_log, const float* dt_bias, const void* z_t,
                              const float* norm_w, float* state, void* o_t, void* y_t,
                              void* stream) {
    GDN_TRY(check_dims(dims));
    GDN_NEED(dims->total_tokens == dims->num_seqs);
    GDN_NEED(dims->h_v / dims->h_k <= 8);
    GDN_NEED(x_t && aligned16(x_t) && conv_w && conv_state && a_t && b_t && A_log && dt_bias);
    GDN_NEED(z_t && aligned16(z_t) && norm_w && aligned16(norm_w) && state && aligned16(state));
    GDN_NEED(y_t && aligned16(y_t) && (!o_t || aligned16(o_t)));
    StepArgs a{};
    a.bf16 = dims->io_dtype == GDN_BF16;
    a.gate = dims->gate;
    a.group_major = dims->layout == GDN_LAYOUT_GROUP;
    a.N = dims->num_seqs;
    a.hk = dims->h_k;
    a.hv = dims->h_v;
    a.C = channels(dims);
    a.x = x_t;
    a.w = conv_w;
    a.cs = conv_state;
    a.a = a_t;
    a.b = b_t;
    a.A_log = A_log;
    a.dt_bias = dt_bias;
    a.z = z_t;
    a.norm_w = norm_w;
    a.S = state;
    a.o = o_t;
    a.y = y_t;
    a.l2_eps = dims->l2_eps;
    a.q_scale = 1.f / sqrtf((float)kD);
    a.norm_eps = dims->norm_eps;
    return cuda_status(launch_step(a, (cudaStream_t)stream));
}

gdn_status gdn_read_status(void* ws, int32_t* code, void* stream) {
    GDN_NEED(ws && code);
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemcpyAsync(code, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return GDN_ERR_CUDA;
    return GDN_OK;
}

}  // extern "C"
