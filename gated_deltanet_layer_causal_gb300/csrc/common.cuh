// Shared device helpers of the GDN CUDA library: dtype conversion, math,
// warp reductions, asynchronous copies, tf32 rounding, the gated-norm row
// backward and the unit lower-triangular inverse.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kD = 128;      // d_k = d_v
constexpr int kChunk = 64;   // chunk length of the WY form
constexpr int kConvK = 4;    // conv taps

// ----------------------------------------------------------------- dtypes
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <class T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// 4 consecutive elements (16 B for fp32, 8 B for bf16) as a float4
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&u.x);
    __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&u.y);
    float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}
// The same 4 elements as loaded, converted later by cvt4: a load whose value is
// first used long after it is issued stays in flight meanwhile.
__device__ __forceinline__ float4 ld4_raw(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ uint2 ld4_raw(const __nv_bfloat16* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ float4 cvt4(float4 v) { return v; }
__device__ __forceinline__ float4 cvt4(uint2 u) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
template <class T> using raw4_t = decltype(ld4_raw(static_cast<const T*>(nullptr)));
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&lo);
    u.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(p) = u;
}

// ----------------------------------------------------------------- math
// The hardware exponential and reciprocal (a few ulp): the kernels that apply
// these gates run few warps per SM, where the full-precision reciprocal's
// dependent refinement steps are exposed latency.  Below x = -87 the result is
// 0 where the true value is under 2^-125.
__device__ __forceinline__ float sigmoidf_(float x) { return __fdividef(1.f, 1.f + __expf(-x)); }
__device__ __forceinline__ float siluf_(float x) { return x * sigmoidf_(x); }

// Output gate of the gated norm (prime-rl #3860 "Summary": GatedDeltaNet takes
// an output_gate_type, "silu" for Qwen3.5, "sigmoid" for Qwen3.8): gate 0 =
// silu(z), gate 1 = sigmoid(z); and its derivative.
constexpr int kGateSilu = 0, kGateSigmoid = 1;
__device__ __forceinline__ float out_gate(float z, int gate) {
    const float s = sigmoidf_(z);
    return gate == kGateSigmoid ? s : z * s;
}
__device__ __forceinline__ float out_gate_grad(float z, int gate) {
    const float s = sigmoidf_(z);
    return gate == kGateSigmoid ? s * (1.f - s) : s * (1.f + z * (1.f - s));
}
// y = o rs (1 + w) gate(z) for four columns
__device__ __forceinline__ float4 gated_norm4(float4 o4, float rs, float4 w4, float4 z4, int gate) {
    return make_float4(o4.x * rs * (1.f + w4.x) * out_gate(z4.x, gate),
                       o4.y * rs * (1.f + w4.y) * out_gate(z4.y, gate),
                       o4.z * rs * (1.f + w4.z) * out_gate(z4.z, gate),
                       o4.w * rs * (1.f + w4.w) * out_gate(z4.w, gate));
}
// softplus with torch's linear branch above 20
__device__ __forceinline__ float softplusf_(float x) { return x > 20.f ? x : log1pf(expf(x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ----------------------------------------------------------------- async copies
// 16-byte global->shared copy that bypasses L1; with pred false it writes 16
// zero bytes and reads nothing (src must still be a valid address).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = pred ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
// 4-byte variant (through L1) for rows that start at an arbitrary element.
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, bool pred) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = pred ? 4 : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
// 8-byte variant (through L1), e.g. four bf16 elements.
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem) : "memory");
}
// Four consecutive elements of type T (16 B fp32, 8 B bf16).
__device__ __forceinline__ void cp_async_row4(float* smem, const float* g) {
    cp_async16(smem, g, true);
}
__device__ __forceinline__ void cp_async_row4(__nv_bfloat16* smem, const __nv_bfloat16* g) {
    cp_async8(smem, g);
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------- tensor cores
// Round to the nearest tf32 value, ties away from zero, on the bit pattern:
// fp32 keeps sign and exponent, tf32 the top 10 of the 23 fraction bits, so
// adding half a tf32 unit (bit 12) to the magnitude bits and clearing the low
// 13 bits rounds the magnitude half-up -- ties away from zero, for either sign.
// Finite values round exactly as cvt.rna.tf32.f32 does (an overflow carries
// into the exponent, as it must); two integer operations, at ALU rate.
__device__ __forceinline__ uint32_t f2tf32(float x) {
    return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u;
}
// Four values rounded to nearest tf32, kept as fp32.
__device__ __forceinline__ float4 tf32_round(float4 v) {
    return make_float4(__uint_as_float(f2tf32(v.x)), __uint_as_float(f2tf32(v.y)),
                       __uint_as_float(f2tf32(v.z)), __uint_as_float(f2tf32(v.w)));
}

// Backward of one gated-RMSNorm row held by a warp (4 columns per lane):
//   n = o rs, dn = dy (1+w) gate(z): do = rs (dn - n mean(dn n)),
//   dz = dy n (1+w) gate'(z), dw += dy n gate(z).
struct NormRowGrad {
    float4 d_o, dz;
};
__device__ __forceinline__ NormRowGrad norm_row_bwd(float4 o4, float4 z4, float4 dy4, float4 w4,
                                                    float eps, float4& dw_acc, int gate) {
    float ss = warp_sum(o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w);
    float rs = rsqrtf(ss * (1.f / kD) + eps);
    float o[4] = {o4.x, o4.y, o4.z, o4.w}, z[4] = {z4.x, z4.y, z4.z, z4.w};
    float dy[4] = {dy4.x, dy4.y, dy4.z, dy4.w}, w[4] = {w4.x, w4.y, w4.z, w4.w};
    float nn[4], dn[4], sz[4], dsz[4], m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        sz[i] = out_gate(z[i], gate);
        dsz[i] = out_gate_grad(z[i], gate);
        nn[i] = o[i] * rs;
        dn[i] = dy[i] * (1.f + w[i]) * sz[i];
        m += dn[i] * nn[i];
    }
    m = warp_sum(m) * (1.f / kD);
    float od[4], zd[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        od[i] = rs * (dn[i] - nn[i] * m);
        zd[i] = dy[i] * nn[i] * (1.f + w[i]) * dsz[i];
    }
    dw_acc.x += dy[0] * nn[0] * sz[0];
    dw_acc.y += dy[1] * nn[1] * sz[1];
    dw_acc.z += dy[2] * nn[2] * sz[2];
    dw_acc.w += dy[3] * nn[3] * sz[3];
    return {make_float4(od[0], od[1], od[2], od[3]), make_float4(zd[0], zd[1], zd[2], zd[3])};
}

// T = (I + A)^-1 for strictly lower A [64][lda] (unit lower-triangular
// inverse), 256 threads; lda and ldt multiples of 4, As and Ts 16-byte aligned.
// Blocked: the four 16 x 16 diagonal blocks by forward substitution
// (T_ij = -sum_{m=j}^{i-1} A_im T_mj, one thread per column), then two merge
// levels of the block formula
//   [[L11, 0], [L21, L22]]^-1 = [[T11, 0], [-T22 L21 T11, T22]]
// (16 -> 32, then 32 -> 64) as small products on the CUDA cores.  Every sum
// runs over m in ascending order.  The substitution is right-looking (each new
// T_mj is added into the partial sums of the rows below at once), so its
// dependent chain is one multiply-add per row; the products run m-outermost with
// each thread's rows of the left factor read four at a time (broadcast float4)
// and each value of the right factor read once for all its rows, the zeros of
// the triangular factors included in the sums.  X is 32 x 32 scratch.
__device__ __forceinline__ void tril_inverse64(const float* As, int lda, float* Ts, int ldt,
                                               float* X) {
    const int tid = threadIdx.x;
    for (int e = tid; e < kChunk * kChunk; e += 256) Ts[(e >> 6) * ldt + (e & 63)] = 0.f;
    __syncthreads();
    if (tid < kChunk) {   // diagonal blocks: thread = column c, solved in registers
        const int c = tid, b0 = c & ~15, cl = c & 15;
        float x[16], acc[16];
#pragma unroll
        for (int i = 0; i < 16; i++) acc[i] = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m++) {
            x[m] = m == cl ? 1.f : (m > cl ? -acc[m] : 0.f);
#pragma unroll
            for (int i = m + 1; i < 16; i++) acc[i] += As[(b0 + i) * lda + b0 + m] * x[m];
        }
#pragma unroll
        for (int i = 0; i < 16; i++) Ts[(b0 + i) * ldt + c] = x[i];
    }
    __syncthreads();
    // 16 -> 32: for the pairs (0,1) and (2,3) of 16-blocks, X = L21 T11, T21 = -T22 X;
    // thread: rows i and i + 8 of pair p, column jj
    {
        const int p = tid >> 7, e = tid & 127;
        const int r0 = 32 * p, r1 = r0 + 16, i = e >> 4, jj = e & 15;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 l0 = *reinterpret_cast<const float4*>(As + (r1 + i) * lda + r0 + m);
            const float4 l1 = *reinterpret_cast<const float4*>(As + (r1 + i + 8) * lda + r0 + m);
            const float t0 = Ts[(r0 + m) * ldt + r0 + jj], t1 = Ts[(r0 + m + 1) * ldt + r0 + jj];
            const float t2 = Ts[(r0 + m + 2) * ldt + r0 + jj], t3 = Ts[(r0 + m + 3) * ldt + r0 + jj];
            a0 += l0.x * t0; a0 += l0.y * t1; a0 += l0.z * t2; a0 += l0.w * t3;
            a1 += l1.x * t0; a1 += l1.y * t1; a1 += l1.z * t2; a1 += l1.w * t3;
        }
        X[p * 256 + i * 16 + jj] = a0;
        X[p * 256 + (i + 8) * 16 + jj] = a1;
        __syncthreads();
        a0 = 0.f;
        a1 = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
            const float4 l0 = *reinterpret_cast<const float4*>(Ts + (r1 + i) * ldt + r1 + m);
            const float4 l1 = *reinterpret_cast<const float4*>(Ts + (r1 + i + 8) * ldt + r1 + m);
            const float x0 = X[p * 256 + m * 16 + jj], x1 = X[p * 256 + (m + 1) * 16 + jj];
            const float x2 = X[p * 256 + (m + 2) * 16 + jj], x3 = X[p * 256 + (m + 3) * 16 + jj];
            a0 += l0.x * x0; a0 += l0.y * x1; a0 += l0.z * x2; a0 += l0.w * x3;
            a1 += l1.x * x0; a1 += l1.y * x1; a1 += l1.z * x2; a1 += l1.w * x3;
        }
        Ts[(r1 + i) * ldt + r0 + jj] = -a0;
        Ts[(r1 + i + 8) * ldt + r0 + jj] = -a1;
    }
    __syncthreads();
    // 32 -> 64: X = L21 T11 (32 x 32), T21 = -T22 X; thread: rows i0 + 8 q, column jj
    {
        const int jj = tid & 31, i0 = tid >> 5;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 32; m += 4) {
            float t[4];
#pragma unroll
            for (int u = 0; u < 4; u++) t[u] = Ts[(m + u) * ldt + jj];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 l = *reinterpret_cast<const float4*>(As + (32 + i0 + 8 * q) * lda + m);
                a[q] += l.x * t[0]; a[q] += l.y * t[1]; a[q] += l.z * t[2]; a[q] += l.w * t[3];
            }
        }
#pragma unroll
        for (int q = 0; q < 4; q++) X[(i0 + 8 * q) * 32 + jj] = a[q];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < 4; q++) a[q] = 0.f;
#pragma unroll
        for (int m = 0; m < 32; m += 4) {
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; u++) x[u] = X[(m + u) * 32 + jj];
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 l = *reinterpret_cast<const float4*>(Ts + (32 + i0 + 8 * q) * ldt + 32 + m);
                a[q] += l.x * x[0]; a[q] += l.y * x[1]; a[q] += l.z * x[2]; a[q] += l.w * x[3];
            }
        }
#pragma unroll
        for (int q = 0; q < 4; q++) Ts[(32 + i0 + 8 * q) * ldt + jj] = -a[q];
    }
    __syncthreads();
}

// Varlen plan entry of one chunk: first token, length, sequence, chunk within sequence.
struct ChunkInfo {
    int32_t start, len, seq, idx;
};

}  // namespace gdn
