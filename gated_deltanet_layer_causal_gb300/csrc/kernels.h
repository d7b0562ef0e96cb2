// Internal launch interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

struct ChunkInfo;

// Raise a kernel's dynamic shared-memory limit on the current device.  The
// attribute belongs to the device's context, so it is set before every launch
// that needs more than 48 KB (a host-only call of about a microsecond): right
// on every device a process drives, after a context is rebuilt, and from any
// host thread.
template <class K>
inline cudaError_t smem_attr(K* kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

struct ConvArgs {
    bool bf16;
    bool group_major;      // channel layout of x, conv_w, the conv cache and dx
    int N, C, hk, hv;
    int64_t T;
    const int32_t* cu;
    const void* x;
    const float* w;
    const void* cs_in;
    float l2_eps, q_scale;
    // forward
    float* qkv;
    void* cs_out;
    bool round_tf32;   // qkv rounded to nearest tf32
    // backward
    const float* dqkv;
    void* dx;
    float* dw;
    float* wpart;   // [conv_bwd_parts(T), C, 4] scratch
    float* dcs;             // gradient of cs_in [N, C, 3] (nullable)
    const float* dcs_out;   // gradient of cs_out [N, C, 3] (nullable)
};
cudaError_t launch_conv_fwd(const ConvArgs& a, cudaStream_t st);
cudaError_t launch_conv_bwd(const ConvArgs& a, cudaStream_t st);
int conv_bwd_parts(int64_t T);

// Saved-for-backward layout of the chunk forward (all fp32 unless noted).
struct FwdSaved {
    int32_t* status;       // device status word
    ChunkInfo* chunks;     // [NT]
    int32_t* seq_chunk;    // [N+1] first chunk of each sequence
    int64_t T;             // total tokens
    int32_t qkv_tf32;      // qkv holds tf32 values: q / k / v tiles are not rounded again
    float* gam;            // [Hv, T] in-chunk cumulative gate (head-major)
    float* beta;           // [Hv, T]
    float* W;              // [T, Hv, d]
    float* U;              // [T, Hv, d]  (U~ from prep, then U)
    float* S0;             // [NT, Hv, d_v, d_k] chunk-start state, row-major, rounded to tf32
    float* Tm;             // [NT * Hv][2][64 * 64] (I + A)^-1 per chunk: K-major T, K-major T^T
    float* o;              // [T, Hv, d] core output (before the norm)
    float* rstd;           // [T, Hv] norm rstd
};

// Tensor maps of the row tensors the chunk kernels load as 64 x 128 tiles
// (3-D: {128 columns, heads, tokens}, 64 x 32 boxes).  The K-major maps use the
// 128-byte swizzle with 16-byte atoms; the *_mn maps the 128-byte swizzle with
// 32-byte atoms, the layout in which the tensor core reads a tile whose rows
// (tokens) are the contraction dimension -- an MN-major operand.
constexpr int kTileCols = 128;
struct TileMaps {
    CUtensorMap q, k, v;   // q / k / v channels of the conv output [T, C]
    CUtensorMap W, U, o;   // [T, Hv, d]
    CUtensorMap dO, dU, dW;
    CUtensorMap dQv, dKv, dUl;
    CUtensorMap dv;        // v channels of the conv-output gradient [T, C]
    CUtensorMap q_mn, k_mn, v_mn, U_mn, W_mn, dO_mn, dU_mn, dW_mn;
    // the chunk-start states as rows (chunk Hv + head) 128 + a of 128 columns b:
    // K-major (rows a; the output kernel) and MN-major (the state-facing kernel)
    CUtensorMap S0, S0_mn;
    // the gradients of the chunk-end states (same rows), and dU_local MN-major
    CUtensorMap dS, dS_mn, dUl_mn;
};
cudaError_t make_rows_map(CUtensorMap* m, const float* base, int heads, int64_t T,
                          int64_t token_stride, bool mn_major = false);

struct ChunkArgs {
    bool bf16;
    int N, NT, hk, hv;
    int64_t T;
    const int32_t* cu;
    const float* qkv;
    const void *a, *b;
    const float *A_log, *dt_bias;
    const float* S_init;
    const void* z;
    const float* norm_w;
    float norm_eps;
    int gate;              // output gate of the fused norm: kGateSilu / kGateSigmoid
    // forward outputs
    void* o_out;
    void* y_out;
    float* S_final;
    FwdSaved sv;
    // backward
    const void* dy;
    const float* dS_final;
    float* dqkv;
    void *da, *db;
    float *dA_log, *ddt_bias;
    void* dz;
    float* dnorm_w;
    float* dS_init;
};

struct BwdScratch {
    int32_t* status; // device status word of the backward workspace
    float* dO;       // [T, Hv, d]
    float* dU;       // [T, Hv, d]
    float* dS;       // [NT, Hv, d_v, d_k] gradient of the state at each chunk end, row-major,
                     // rounded to tf32
    float* dUl;      // [T, Hv, d] dU_local (the local kernel's part of dU); shares dKv3's
                     // memory, which the WY kernel writes only after the state pass
    float* dQv;      // [T, Hk, d] per k-head dq^, state-facing part (summed over its v-heads)
    float* dKv;      // [T, Hk, d] per k-head dk^, state-facing part (summed over its v-heads)
    float* dQv2;     // [T, Hk, d] per k-head dq^, P / dP part (summed over its v-heads)
    float* dKv2;     // [T, Hk, d] per k-head dk^, P / dP part (summed over its v-heads)
    float* dKv3;     // [T, Hk, d] per k-head dk^, WY part (summed over its v-heads); the
                     // [T, Hv, d] dU_local before (dUl, allocated at that size)
    float* dW;       // [T, Hv, d]
    float* dgam;     // [T, Hv] partial dgamma from the state-facing terms
    float* dgam2;    // [T, Hv] the P / dP kernel's dgam terms (it runs beside the state pass)
    float* dgs;      // [T, Hv] dg (per token)
    int32_t* dp_next;  // tile counter of the P / dP kernel (zeroed before its launch)
    float* nw_part;  // [NT * Hv, d] dnorm_w partials
};

cudaError_t launch_plan(const int32_t* cu, int N, int64_t T, int NT, FwdSaved sv, cudaStream_t st);
cudaError_t launch_chunk_fwd(const ChunkArgs& a, cudaStream_t st);
cudaError_t launch_chunk_bwd(const ChunkArgs& a, const BwdScratch& w, cudaStream_t st);

struct NormArgs {
    bool bf16;
    int gate;       // kGateSilu / kGateSigmoid
    int64_t rows;   // T * Hv
    const void *o, *z;
    const float* w;
    float eps;
    void* y;
    float* rstd;
    const void* dy;
    void *d_o, *dz;
    float* dw;
    float* part;    // [norm_bwd_parts(rows), d]
};
cudaError_t launch_norm_fwd(const NormArgs& a, cudaStream_t st);
cudaError_t launch_norm_bwd(const NormArgs& a, cudaStream_t st);
int norm_bwd_parts(int64_t rows);
cudaError_t launch_norm_bwd_noalloc(const NormArgs& a, cudaStream_t st);
int norm_bwd_noalloc_max_rows();

struct StepArgs {
    bool bf16;
    int gate;              // kGateSilu / kGateSigmoid
    bool group_major;      // channel layout of x, conv_w and the conv cache
    int N, hk, hv, C;
    const void* x;
    const float* w;
    void* cs;
    const void *a, *b;
    const float *A_log, *dt_bias;
    const void* z;
    const float* norm_w;
    float* S;
    void *o, *y;
    float l2_eps, q_scale, norm_eps;
};
cudaError_t launch_step(const StepArgs& a, cudaStream_t st);

}  // namespace gdn
