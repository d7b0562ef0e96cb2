// Zero-centred gated RMSNorm (standalone forward / backward) and the recurrent
// single-token decode step.
//
// Norm: prime-rl #3860 "Summary" (ZeroCenteredRMSNorm shared by the GDN
// layers; the output gate silu or sigmoid), "[main] feat(moe): Support gated
// delta net for Qwen3-Next (1/4)" (--apply-layernorm-1p): y = o rsqrt(mean(o^2)
// + eps) (1 + w) gate(z) per (token, v-head) over d_v = 128.  HBM-bound: one warp per row, 4 columns per
// lane, warp-shuffle reductions; the weight gradient is summed per CTA and then
// across CTAs in a fixed order (bitwise reproducible).
//
// Decode step: one token of the same core for a batch of independent
// sequences -- conv-cache update, conv + SiLU, L2 norms, gates, the rank-1
// state update S <- e^g S + beta (v - e^g S k) k^T, o = S q, and the norm.
// HBM-bound on the fp32 state, which is read once and written once.
#include <cuda.h>

#include <mutex>

#include "../../include/gdn.h"
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace gdn {

constexpr int kNormWarps = 8;
constexpr int kNormRowsPerCta = 64;

template <class IO>
__global__ void __launch_bounds__(kNormWarps * 32)
norm_fwd_kernel(const IO* __restrict__ o, const IO* __restrict__ z, const float* __restrict__ w,
                float eps, int gate, int64_t rows, IO* __restrict__ y, float* rstd) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float4 w4 = ld4(w + lane * 4);
    for (int64_t r = (int64_t)blockIdx.x * kNormWarps + warp; r < rows;
         r += (int64_t)gridDim.x * kNormWarps) {
        const int64_t off = r * kD + lane * 4;
        float4 o4 = ld4(o + off), z4 = ld4(z + off);
        float ss = warp_sum(o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w);
        float rs = rsqrtf(ss * (1.f / kD) + eps);
        st4(y + off, gated_norm4(o4, rs, w4, z4, gate));
        if (rstd && lane == 0) rstd[r] = rs;
    }
}

template <class IO>
__global__ void __launch_bounds__(kNormWarps * 32)
norm_bwd_kernel(const IO* __restrict__ o, const IO* __restrict__ z, const float* __restrict__ w,
                const IO* __restrict__ dy, float eps, int gate, int64_t rows,
                IO* __restrict__ d_o, IO* __restrict__ dz, float* __restrict__ part) {
    __shared__ float4 red[kNormWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float4 w4 = ld4(w + lane * 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t r0 = (int64_t)blockIdx.x * kNormRowsPerCta;
    const int64_t r1 = min(r0 + kNormRowsPerCta, rows);
    for (int64_t r = r0 + warp; r < r1; r += kNormWarps) {
        const int64_t off = r * kD + lane * 4;
        NormRowGrad gr =
            norm_row_bwd(ld4(o + off), ld4(z + off), ld4(dy + off), w4, eps, acc, gate);
        st4(d_o + off, gr.d_o);
        st4(dz + off, gr.dz);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float4 s = red[0][lane];
        for (int i = 1; i < kNormWarps; i++) {
            s.x += red[i][lane].x; s.y += red[i][lane].y;
            s.z += red[i][lane].z; s.w += red[i][lane].w;
        }
        st4(part + (int64_t)blockIdx.x * kD + lane * 4, s);
    }
}

// out[i] = sum_p part[p][i] in order p = 0, 1, ...  (one thread per column)
__global__ void colsum_kernel(const float* __restrict__ part, int64_t nparts, int cols,
                              float* __restrict__ out) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= cols) return;
    float acc = 0.f;
    for (int64_t p = 0; p < nparts; p++) acc += part[p * cols + i];
    out[i] = acc;
}

int norm_bwd_parts(int64_t rows) { return (int)((rows + kNormRowsPerCta - 1) / kNormRowsPerCta); }

template <class IO>
static cudaError_t norm_fwd_t(const NormArgs& a, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    int64_t blocks = (a.rows + kNormWarps - 1) / kNormWarps;
    if (blocks > 152 * 16) blocks = 152 * 16;
    GDN_PROF("norm_fwd", st);
    norm_fwd_kernel<IO><<<(unsigned)blocks, kNormWarps * 32, 0, st>>>(
        (const IO*)a.o, (const IO*)a.z, a.w, a.eps, a.gate, a.rows, (IO*)a.y, a.rstd);
    return cudaGetLastError();
}
cudaError_t launch_norm_fwd(const NormArgs& a, cudaStream_t st) {
    return a.bf16 ? norm_fwd_t<__nv_bfloat16>(a, st) : norm_fwd_t<float>(a, st);
}

template <class IO>
static cudaError_t norm_bwd_t(const NormArgs& a, cudaStream_t st) {
    int parts = norm_bwd_parts(a.rows);
    if (parts == 0) {
        cudaMemsetAsync(a.dw, 0, sizeof(float) * kD, st);
        return cudaGetLastError();
    }
    {
        GDN_PROF("norm_bwd", st);
        norm_bwd_kernel<IO><<<parts, kNormWarps * 32, 0, st>>>(
            (const IO*)a.o, (const IO*)a.z, a.w, (const IO*)a.dy, a.eps, a.gate, a.rows,
            (IO*)a.d_o, (IO*)a.dz, a.part);
    }
    {
        GDN_PROF("norm_w_reduce", st);
        colsum_kernel<<<1, kD, 0, st>>>(a.part, parts, kD, a.dw);
    }
    return cudaGetLastError();
}
cudaError_t launch_norm_bwd(const NormArgs& a, cudaStream_t st) {
    return a.bf16 ? norm_bwd_t<__nv_bfloat16>(a, st) : norm_bwd_t<float>(a, st);
}

// ------------------------------------------------------------------ allocation-free backward
// Scratch of gdn_gated_rmsnorm_bwd_noalloc: the dnorm_w partial sums (one row of
// kD floats per CTA of kNormRowsPerCta rows) live in this file-scope array
// instead of a caller workspace.  Every device that loads the library holds it
// (4 MiB) until the process exits.
constexpr int kNoAllocParts = 8192;
static __device__ __align__(256) float g_norm_bwd_scratch[kNoAllocParts * kD];

static_assert(kNoAllocParts * kNormRowsPerCta == GDN_NOALLOC_NORM_BWD_MAX_ROWS,
              "the header's row limit is the array's capacity");
int norm_bwd_noalloc_max_rows() { return kNoAllocParts * kNormRowsPerCta; }

namespace {
constexpr int kMaxDevices = 64;

// The array's device address belongs to the CUDA context that loaded this
// module: after a context is destroyed and rebuilt (cudaDeviceReset, or the
// primary context released and retained again) the module is loaded afresh
// and the array may sit elsewhere.  So the cached address is keyed on the
// context's process-unique ID, read through the driver entry points (looked
// up once through the runtime; the library links no driver library).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
struct CtxQuery {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};
const CtxQuery& ctx_query() {
    static const CtxQuery q = [] {
        CtxQuery r;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult st;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &st) == cudaSuccess &&
            st == cudaDriverEntryPointSuccess)
            r.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &st) ==
                cudaSuccess &&
            st == cudaDriverEntryPointSuccess)
            r.get_id = reinterpret_cast<CtxGetIdFn>(p);
        return r;
    }();
    return q;
}
// ID of the calling thread's current context; false if there is none or the
// driver cannot tell.
bool current_ctx_id(unsigned long long* id) {
    const CtxQuery& q = ctx_query();
    CUcontext ctx = nullptr;
    if (q.get_current == nullptr || q.get_id == nullptr) return false;
    if (q.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return q.get_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchAddr {
    unsigned long long ctx_id = 0;
    bool valid = false;
    float* addr = nullptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_dev[kMaxDevices];   // per device: the context it was read in
}  // namespace

// Device address of g_norm_bwd_scratch in the current device's context.  Host
// code only sees a host-side stand-in for the array, so the address is looked
// up (cudaGetSymbolAddress, with that device current) the first time a context
// uses it and cached under the context's ID; a rebuilt context looks it up
// again.  Without the driver's context query it is looked up on every call.
static cudaError_t norm_bwd_noalloc_scratch(float** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchAddr& slot = g_scratch_dev[dev];
    unsigned long long id = 0;
    if (slot.valid && current_ctx_id(&id) && id == slot.ctx_id) {
        *out = slot.addr;
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_norm_bwd_scratch);   // makes the context current if needed
    if (e != cudaSuccess) return e;
    slot.valid = current_ctx_id(&id);
    slot.ctx_id = id;
    slot.addr = static_cast<float*>(p);
    *out = slot.addr;
    return cudaSuccess;
}

cudaError_t launch_norm_bwd_noalloc(const NormArgs& a, cudaStream_t st) {
    if (a.rows > (int64_t)norm_bwd_noalloc_max_rows()) return cudaErrorInvalidValue;
    NormArgs b = a;
    cudaError_t e = norm_bwd_noalloc_scratch(&b.part);
    if (e != cudaSuccess) return e;
    // each CTA writes its whole partial row before the column sum reads it,
    // so the array's previous contents never matter
    return launch_norm_bwd(b, st);
}

// ------------------------------------------------------------------ decode step
// grid (hk, N), 256 threads: one CTA owns k-head kh of sequence n and the G
// v-heads that read it, so the conv cache of all its channels is updated in
// place by exactly one CTA.
constexpr int kMaxGroup = 8;

template <class IO>
__global__ void __launch_bounds__(256)
step_kernel(const IO* __restrict__ x, const float* __restrict__ w, IO* cs,
            const IO* __restrict__ av, const IO* __restrict__ bv, const float* __restrict__ A_log,
            const float* __restrict__ dt_bias, const IO* __restrict__ z,
            const float* __restrict__ norm_w, float* __restrict__ S, IO* o_out, IO* y_out,
            int hk, int hv, float l2_eps, float q_scale, float norm_eps, int gate,
            bool group_major) {
    __shared__ float q[kD], k[kD], v[kMaxGroup][kD], o[kMaxGroup][kD];
    __shared__ float gdec[kMaxGroup], gbeta[kMaxGroup];
    const int kh = blockIdx.x, n = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int G = hv / hk, C = (2 * hk + hv) * kD;
    // conv + SiLU over this CTA's (2 + G) * 128 channels; cache shifts left.
    // Channel of x / conv_w / the cache: flat [q | k | v], or group-major (the
    // group's q, k and v heads contiguous), which is this loop's own order.
    for (int i = tid; i < (2 + G) * kD; i += 256) {
        int c = group_major ? kh * (2 + G) * kD + i
              : i < kD ? kh * kD + i
              : i < 2 * kD ? hk * kD + kh * kD + (i - kD)
                           : 2 * hk * kD + kh * G * kD + (i - 2 * kD);
        IO* cc = cs + ((int64_t)n * C + c) * (kConvK - 1);
        float h3 = to_f(cc[0]), h2 = to_f(cc[1]), h1 = to_f(cc[2]);
        float cur = to_f(x[(int64_t)n * C + c]);
        const float* wc = w + (int64_t)c * kConvK;
        float pre = wc[0] * h3 + wc[1] * h2 + wc[2] * h1 + wc[3] * cur;
        float xc = siluf_(pre);
        cc[0] = from_f<IO>(h2);
        cc[1] = from_f<IO>(h1);
        cc[2] = x[(int64_t)n * C + c];
        if (i < kD) q[i] = xc;
        else if (i < 2 * kD) k[i - kD] = xc;
        else v[(i - 2 * kD) / kD][(i - 2 * kD) % kD] = xc;
    }
    if (tid < G) {
        int h = kh * G + tid;
        gdec[tid] = expf(-expf(A_log[h]) * softplusf_(to_f(av[(int64_t)n * hv + h]) + dt_bias[h]));
        gbeta[tid] = sigmoidf_(to_f(bv[(int64_t)n * hv + h]));
    }
    __syncthreads();
    if (warp < 2) {  // L2 norms: warp 0 -> q (scaled), warp 1 -> k
        float* vec = warp == 0 ? q : k;
        float4 a4 = ld4(vec + lane * 4);
        float ss = warp_sum(a4.x * a4.x + a4.y * a4.y + a4.z * a4.z + a4.w * a4.w);
        float r = rsqrtf(ss + l2_eps) * (warp == 0 ? q_scale : 1.f);
        a4.x *= r; a4.y *= r; a4.z *= r; a4.w *= r;
        st4(vec + lane * 4, a4);
    }
    __syncthreads();
    const float4 q4 = ld4(q + lane * 4), k4 = ld4(k + lane * 4);
    const float kq = warp_sum(q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w);
    // rank-1 update, one state row per warp iteration
    for (int row = warp; row < G * kD; row += 8) {
        const int j = row / kD, a = row % kD, h = kh * G + j;
        float* Sr = S + (((int64_t)n * hv + h) * kD + a) * kD + lane * 4;
        float4 s4 = ld4(Sr);
        float sk = warp_sum(s4.x * k4.x + s4.y * k4.y + s4.z * k4.z + s4.w * k4.w);
        float sq = warp_sum(s4.x * q4.x + s4.y * q4.y + s4.z * q4.z + s4.w * q4.w);
        const float dec = gdec[j];
        const float delta = gbeta[j] * (v[j][a] - dec * sk);
        s4.x = dec * s4.x + delta * k4.x;
        s4.y = dec * s4.y + delta * k4.y;
        s4.z = dec * s4.z + delta * k4.z;
        s4.w = dec * s4.w + delta * k4.w;
        st4(Sr, s4);
        if (lane == 0) o[j][a] = dec * sq + delta * kq;
    }
    __syncthreads();
    // gated RMSNorm per v-head
    const float4 w4 = ld4(norm_w + lane * 4);
    for (int j = warp; j < G; j += 8) {
        const int h = kh * G + j;
        const int64_t off = ((int64_t)n * hv + h) * kD + lane * 4;
        float4 o4 = ld4(&o[j][lane * 4]);
        if (o_out) st4(o_out + off, o4);
        float ss = warp_sum(o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w);
        float rs = rsqrtf(ss * (1.f / kD) + norm_eps);
        st4(y_out + off, gated_norm4(o4, rs, w4, ld4(z + off), gate));
    }
}

template <class IO>
static cudaError_t step_t(const StepArgs& a, cudaStream_t st) {
    if (a.N == 0) return cudaSuccess;
    GDN_PROF("recurrent_step", st);
    step_kernel<IO><<<dim3(a.hk, a.N), 256, 0, st>>>(
        (const IO*)a.x, a.w, (IO*)a.cs, (const IO*)a.a, (const IO*)a.b, a.A_log, a.dt_bias,
        (const IO*)a.z, a.norm_w, a.S, (IO*)a.o, (IO*)a.y, a.hk, a.hv, a.l2_eps, a.q_scale,
        a.norm_eps, a.gate, a.group_major);
    return cudaGetLastError();
}
cudaError_t launch_step(const StepArgs& a, cudaStream_t st) {
    return a.bf16 ? step_t<__nv_bfloat16>(a, st) : step_t<float>(a, st);
}

}  // namespace gdn
