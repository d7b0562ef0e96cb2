// Forward of the gated delta rule in the chunked WY form (chunk 64), with the
// gates, grouped value heads and the fused zero-centred gated RMSNorm.
//
// Per chunk (tokens i = 0..L-1, in-chunk cumulative gate gam_i):
//   A_ij = beta_i exp(gam_i - gam_j) k_i.k_j (j < i);  T = (I + A)^-1
//   W = T diag(beta e^gam) K ;  U~ = T diag(beta) V          (prep, parallel)
//   U = U~ - W S0^T ;  S_end = e^{gam_L} S0 + U^T diag(e^{gam_L-gam}) K
//                                                            (state, sequential)
//   O = diag(e^gam) Q S0^T + (Q K^T (.) exp(gam_i-gam_j) (.) [i>=j]) U
//   y = O rsqrt(mean(O^2)+eps) (1+w) silu(z)                 (out, parallel)
// which unrolls S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
// o_t = S_t q_t exactly.  Sources: "[6/8] feat(models): port Qwen3.5 / Qwen3-Next
// GDN to the head-sharded layer" ("What": grouped value heads, native GVA);
// prime-rl #3860 "Summary" (chunk op with cu_seqlens / initial_state /
// output_final_state; ZeroCenteredRMSNorm); "[main] feat(moe): Support gated
// delta net for Qwen3-Next (1/4)" (A_log review comment: decay rate exp(A_log)).
//
// All products run on the tensor cores (tf32 operands, fp32 accumulation); the
// state stays fp32 in registers across the whole sequence.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace gdn {

// ------------------------------------------------------------------ varlen plan
// One CTA: chunk counts per sequence, exclusive scan, chunk table.  Checks the
// device copy of cu_seqlens against what the host planned (NT chunks, cu[N] =
// T); on mismatch it sets the status word and plans zero chunks.
__global__ void plan_kernel(const int32_t* __restrict__ cu, int N, int64_t T, int NT,
                            ChunkInfo* __restrict__ chunks, int32_t* __restrict__ seq_chunk,
                            int32_t* status) {
    __shared__ int32_t part[1024];
    __shared__ int bad;
    const int tid = threadIdx.x, nth = blockDim.x;
    const int per = (N + nth - 1) / nth;
    const int n0 = min(N, tid * per), n1 = min(N, n0 + per);
    if (tid == 0) bad = (cu[0] != 0 || (int64_t)cu[N] != T) ? 1 : 0;
    __syncthreads();
    int cnt = 0;
    for (int n = n0; n < n1; n++) {
        int L = cu[n + 1] - cu[n];
        if (L < 0) atomicOr(&bad, 1);
        else cnt += (L + kChunk - 1) / kChunk;
    }
    part[tid] = cnt;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int i = 0; i < nth; i++) { int c = part[i]; part[i] = run; run += c; }
        if (run != NT) bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) *status = 6;  // GDN_ERR_DEVICE_CHECK
        for (int n = tid; n <= N; n += nth) seq_chunk[n] = 0;
        for (int i = tid; i < NT; i += nth) chunks[i] = ChunkInfo{0, 0, 0, 0};
        return;
    }
    int off = part[tid];
    for (int n = n0; n < n1; n++) {
        seq_chunk[n] = off;
        int s = cu[n], L = cu[n + 1] - s;
        for (int j = 0; j * kChunk < L; j++)
            chunks[off + j] = ChunkInfo{s + j * kChunk, min(kChunk, L - j * kChunk), n, j};
        off += (L + kChunk - 1) / kChunk;
    }
    if (tid == nth - 1) seq_chunk[N] = NT;
}

// ------------------------------------------------------------------ prep
// grid (NT, Hv), 256 threads.  Gates, in-chunk cumsum, A, T, W, U~.
constexpr int kLdK = 132, kLdV = 136, kLdA = 68;
constexpr size_t kPrepSmem = sizeof(float) * (64 * kLdK + 64 * kLdV + 2 * 64 * kLdA + 3 * 64);

template <class IO>
__global__ void __launch_bounds__(256, 2)
prep_kernel(const float* __restrict__ qkv, const IO* __restrict__ av, const IO* __restrict__ bv,
            const float* __restrict__ A_log, const float* __restrict__ dt_bias, int hk, int hv,
            FwdSaved sv) {
    extern __shared__ float sm[];
    float* Ks = sm;
    float* Vs = Ks + 64 * kLdK;
    float* As = Vs + 64 * kLdV;
    float* Ts = As + 64 * kLdA;
    float* gam = Ts + 64 * kLdA;
    float* bet = gam + 64;
    float* be = bet + 64;
    const ChunkInfo ci = sv.chunks[blockIdx.x];
    if (ci.len == 0) return;
    const int h = blockIdx.y, kh = h / (hv / hk), tid = threadIdx.x;
    const int C = (2 * hk + hv) * kD;
    const float* kbase = qkv + (int64_t)hk * kD + kh * kD;
    const float* vbase = qkv + (int64_t)2 * hk * kD + h * kD;
    for (int idx = tid; idx < 64 * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
        if (r < ci.len) {
            int64_t row = (int64_t)(ci.start + r) * C;
            kk = ld4(kbase + row + c4);
            vv = ld4(vbase + row + c4);
        }
        st4(Ks + r * kLdK + c4, kk);
        st4(Vs + r * kLdV + c4, vv);
    }
    if (tid < 64) {
        float g = 0.f, b = 0.f;
        if (tid < ci.len) {
            int64_t t = ci.start + tid;
            g = -expf(A_log[h]) * softplusf_(to_f(av[t * hv + h]) + dt_bias[h]);
            b = sigmoidf_(to_f(bv[t * hv + h]));
        }
        gam[tid] = g;
        bet[tid] = b;
    }
    __syncthreads();
    if (tid < 32) warp_cumsum64(gam);
    __syncthreads();
    if (tid < 64) {
        be[tid] = bet[tid] * expf(gam[tid]);
        if (tid < ci.len) {
            int64_t t = ci.start + tid;
            sv.gam[t * hv + h] = gam[tid];
            sv.beta[t * hv + h] = bet[tid];
        }
    }
    {
        using TL = Tile<64, 64, 8>;
        typename TL::Acc acc;
        tile_zero<64, 64, 8>(acc);
        tile_mma<64, 64, kD, 8>(acc, [&](int r, int k) { return Ks[r * kLdK + k]; },
                                [&](int k, int c) { return Ks[c * kLdK + k]; });
        tile_each<64, 64, 8>(acc, [&](int r, int c, float& v) {
            As[r * kLdA + c] = (c < r) ? bet[r] * expf(gam[r] - gam[c]) * v : 0.f;
        });
    }
    __syncthreads();
    tril_inverse64(As, kLdA, Ts, kLdA);
    __syncthreads();
    using TW = Tile<64, kD, 8>;
    typename TW::Acc acc;
    tile_zero<64, kD, 8>(acc);
    tile_mma<64, kD, 64, 8>(acc, [&](int r, int k) { return Ts[r * kLdA + k]; },
                            [&](int k, int c) { return be[k] * Ks[k * kLdK + c]; });
    tile_each2<64, kD, 8>(acc, [&](int r, int c, float& v0, float& v1) {
        if (r < ci.len)
            *reinterpret_cast<float2*>(sv.W + ((int64_t)(ci.start + r) * hv + h) * kD + c) =
                make_float2(v0, v1);
    });
    tile_zero<64, kD, 8>(acc);
    tile_mma<64, kD, 64, 8>(acc, [&](int r, int k) { return Ts[r * kLdA + k]; },
                            [&](int k, int c) { return bet[k] * Vs[k * kLdV + c]; });
    tile_each2<64, kD, 8>(acc, [&](int r, int c, float& v0, float& v1) {
        if (r < ci.len)
            *reinterpret_cast<float2*>(sv.U + ((int64_t)(ci.start + r) * hv + h) * kD + c) =
                make_float2(v0, v1);
    });
}

// ------------------------------------------------------------------ state pass
// grid (d_v / kSlice, Hv, N), 128 threads.  Rows a of S evolve independently
// (k, beta, g are shared by all rows), so each CTA carries a 32-row slice of
// the fp32 state -- kept transposed, S^T[b][a], in the MMA accumulators --
// through all chunks of its sequence.
constexpr int kSlice = 32;
constexpr int kLdS = kSlice + 8;   // 40: conflict-free as a K-major operand
constexpr size_t kStateSmem =
    sizeof(float) * (64 * kLdK + 64 * kLdV + 64 * kLdS + kD * kLdS + 2 * 64);

__global__ void __launch_bounds__(128)
state_fwd_kernel(const float* __restrict__ qkv, int hk, int hv, const float* S_init,
                 float* S_final, FwdSaved sv) {
    extern __shared__ float sm[];
    float* Ws = sm;                    // [64][kLdK]
    float* Ks = Ws + 64 * kLdK;        // [64][kLdV]
    float* Us = Ks + 64 * kLdV;        // [64][kLdS]
    float* St = Us + 64 * kLdS;        // [128][kLdS]  S^T slice
    float* gam = St + kD * kLdS;       // [64]
    float* fk = gam + 64;              // [64] exp(gam_L - gam_i)
    const int sl = blockIdx.x, h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
    const int a0 = sl * kSlice, kh = h / (hv / hk);
    const int C = (2 * hk + hv) * kD;
    using TS = Tile<kD, kSlice, 4>;    // S^T: rows b (d_k), cols a (slice)
    using TU = Tile<64, kSlice, 4>;
    typename TS::Acc sacc;
    const int64_t sbase = ((int64_t)n * hv + h) * kD * kD;
    tile_each<kD, kSlice, 4>(sacc, [&](int b, int a, float& v) {
        v = S_init ? S_init[sbase + (int64_t)(a0 + a) * kD + b] : 0.f;
        St[b * kLdS + a] = v;
    });
    const int c0 = sv.seq_chunk[n], c1 = sv.seq_chunk[n + 1];
    for (int ci = c0; ci < c1; ci++) {
        const ChunkInfo info = sv.chunks[ci];
        const int L = info.len;
        __syncthreads();
        for (int idx = tid; idx < 64 * 32; idx += 128) {
            int r = idx >> 5, c4 = (idx & 31) * 4;
            float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = w4;
            if (r < L) {
                int64_t t = info.start + r;
                w4 = ld4(sv.W + (t * hv + h) * kD + c4);
                k4 = ld4(qkv + t * C + (int64_t)hk * kD + kh * kD + c4);
            }
            st4(Ws + r * kLdK + c4, w4);
            st4(Ks + r * kLdV + c4, k4);
        }
        for (int idx = tid; idx < 64 * kSlice / 4; idx += 128) {
            int r = idx / (kSlice / 4), c4 = (idx % (kSlice / 4)) * 4;
            float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < L) u4 = ld4(sv.U + ((int64_t)(info.start + r) * hv + h) * kD + a0 + c4);
            st4(Us + r * kLdS + c4, u4);
        }
        if (tid < 64) gam[tid] = tid < L ? sv.gam[(int64_t)(info.start + tid) * hv + h] : 0.f;
        // state at the chunk start, for the output and the backward
        const int64_t obase = ((int64_t)ci * hv + h) * kD * kD;
        tile_each2<kD, kSlice, 4>(sacc, [&](int b, int a, float& v0, float& v1) {
            sv.S0[obase + (int64_t)(a0 + a) * kD + b] = v0;
            sv.S0[obase + (int64_t)(a0 + a + 1) * kD + b] = v1;
        });
        __syncthreads();
        if (tid < 64) fk[tid] = tid < L ? expf(gam[L - 1] - gam[tid]) : 0.f;
        // U = U~ - W S^T   (64 x slice)
        typename TU::Acc uacc;
        tile_zero<64, kSlice, 4>(uacc);
        tile_mma<64, kSlice, kD, 4>(uacc, [&](int i, int b) { return Ws[i * kLdK + b]; },
                                    [&](int b, int a) { return St[b * kLdS + a]; });
        __syncthreads();
        tile_each<64, kSlice, 4>(uacc, [&](int i, int a, float& v) {
            float u = i < L ? Us[i * kLdS + a] - v : 0.f;
            Us[i * kLdS + a] = u;
            if (i < L) sv.U[((int64_t)(info.start + i) * hv + h) * kD + a0 + a] = u;
        });
        __syncthreads();
        // S^T = e^{gam_L} S^T + (diag(fk) K)^T U
        const float dl = expf(gam[L - 1]);
        tile_each<kD, kSlice, 4>(sacc, [&](int, int, float& v) { v *= dl; });
        tile_mma<kD, kSlice, 64, 4>(sacc, [&](int b, int i) { return fk[i] * Ks[i * kLdV + b]; },
                                    [&](int i, int a) { return Us[i * kLdS + a]; });
        tile_each<kD, kSlice, 4>(sacc, [&](int b, int a, float& v) { St[b * kLdS + a] = v; });
    }
    if (S_final)
        tile_each<kD, kSlice, 4>(sacc, [&](int b, int a, float& v) {
            S_final[sbase + (int64_t)(a0 + a) * kD + b] = v;
        });
}

// ------------------------------------------------------------------ output + norm
// grid (NT, Hv), 256 threads.
constexpr size_t kOutSmem =
    sizeof(float) * (64 * kLdK * 2 + 64 * kLdV + kD * kLdK + 64 * kLdA + 2 * 64);

template <class IO>
__global__ void __launch_bounds__(256)
out_fwd_kernel(const float* __restrict__ qkv, int hk, int hv, const IO* z,
               const float* norm_w, float norm_eps, IO* o_out, IO* y_out, FwdSaved sv) {
    extern __shared__ float sm[];
    float* Qs = sm;                    // [64][kLdK]   (later O)
    float* Ks = Qs + 64 * kLdK;        // [64][kLdK]
    float* Us = Ks + 64 * kLdK;        // [64][kLdV]
    float* Ss = Us + 64 * kLdV;        // [128][kLdK]  S0[a][b]
    float* Ps = Ss + kD * kLdK;        // [64][kLdA]
    float* gam = Ps + 64 * kLdA;
    float* eg = gam + 64;
    const ChunkInfo ci = sv.chunks[blockIdx.x];
    if (ci.len == 0) return;
    const int h = blockIdx.y, kh = h / (hv / hk), tid = threadIdx.x, L = ci.len;
    const int C = (2 * hk + hv) * kD;
    for (int idx = tid; idx < 64 * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = q4, u4 = q4;
        if (r < L) {
            int64_t t = ci.start + r;
            q4 = ld4(qkv + t * C + kh * kD + c4);
            k4 = ld4(qkv + t * C + (int64_t)hk * kD + kh * kD + c4);
            u4 = ld4(sv.U + (t * hv + h) * kD + c4);
        }
        st4(Qs + r * kLdK + c4, q4);
        st4(Ks + r * kLdK + c4, k4);
        st4(Us + r * kLdV + c4, u4);
    }
    const float* S0 = sv.S0 + ((int64_t)blockIdx.x * hv + h) * kD * kD;
    for (int idx = tid; idx < kD * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        st4(Ss + r * kLdK + c4, ld4(S0 + r * kD + c4));
    }
    if (tid < 64) {  // padding rows continue the last gate value (g = 0)
        float g = sv.gam[(int64_t)(ci.start + min(tid, L - 1)) * hv + h];
        gam[tid] = g;
        eg[tid] = tid < L ? expf(g) : 0.f;
    }
    __syncthreads();
    {
        using TL = Tile<64, 64, 8>;
        typename TL::Acc acc;
        tile_zero<64, 64, 8>(acc);
        tile_mma<64, 64, kD, 8>(acc, [&](int r, int k) { return Qs[r * kLdK + k]; },
                                [&](int k, int c) { return Ks[c * kLdK + k]; });
        tile_each<64, 64, 8>(acc, [&](int r, int c, float& v) {
            Ps[r * kLdA + c] = (c <= r) ? v * expf(gam[r] - gam[c]) : 0.f;
        });
    }
    __syncthreads();
    using TO = Tile<64, kD, 8>;
    typename TO::Acc acc;
    tile_zero<64, kD, 8>(acc);
    tile_mma<64, kD, 64, 8>(acc, [&](int r, int k) { return Ps[r * kLdA + k]; },
                            [&](int k, int c) { return Us[k * kLdV + c]; });
    tile_mma<64, kD, kD, 8>(acc, [&](int r, int k) { return eg[r] * Qs[r * kLdK + k]; },
                            [&](int k, int c) { return Ss[c * kLdK + k]; });
    __syncthreads();
    float* Os = Qs;
    tile_each2<64, kD, 8>(acc, [&](int r, int c, float& v0, float& v1) {
        *reinterpret_cast<float2*>(Os + r * kLdK + c) = make_float2(v0, v1);
    });
    __syncthreads();
    // gated RMSNorm, one warp per row, lane = 4 columns
    const int lane = tid & 31, warp = tid >> 5;
    float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (z) w4 = ld4(norm_w + lane * 4);
    for (int r = warp; r < L; r += 8) {
        const int64_t t = ci.start + r;
        const int64_t off = (t * hv + h) * kD + lane * 4;
        float4 o4 = ld4(Os + r * kLdK + lane * 4);
        st4(sv.o + off, o4);
        if (o_out) st4(o_out + off, o4);
        if (z) {
            float ss = warp_sum(o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w);
            float rs = rsqrtf(ss * (1.f / kD) + norm_eps);
            float4 z4 = ld4(z + off), y4;
            y4.x = o4.x * rs * (1.f + w4.x) * siluf_(z4.x);
            y4.y = o4.y * rs * (1.f + w4.y) * siluf_(z4.y);
            y4.z = o4.z * rs * (1.f + w4.z) * siluf_(z4.z);
            y4.w = o4.w * rs * (1.f + w4.w) * siluf_(z4.w);
            st4(y_out + off, y4);
            if (lane == 0) sv.rstd[t * hv + h] = rs;
        }
    }
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_plan(const int32_t* cu, int N, int64_t T, int NT, FwdSaved sv, cudaStream_t st) {
    cudaMemsetAsync(sv.status, 0, sizeof(int32_t), st);
    GDN_PROF("plan", st);
    plan_kernel<<<1, 1024, 0, st>>>(cu, N, T, NT, sv.chunks, sv.seq_chunk, sv.status);
    return cudaGetLastError();
}

template <class IO>
static cudaError_t chunk_fwd_t(const ChunkArgs& a, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(prep_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPrepSmem);
        cudaFuncSetAttribute(state_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStateSmem);
        cudaFuncSetAttribute(out_fwd_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kOutSmem);
        attr = true;
    }
    if (a.NT > 0) {
        GDN_PROF("chunk_prep", st);
        prep_kernel<IO><<<dim3(a.NT, a.hv), 256, kPrepSmem, st>>>(
            a.qkv, (const IO*)a.a, (const IO*)a.b, a.A_log, a.dt_bias, a.hk, a.hv, a.sv);
    }
    if (a.N > 0) {
        GDN_PROF("chunk_state_fwd", st);
        state_fwd_kernel<<<dim3(kD / kSlice, a.hv, a.N), 128, kStateSmem, st>>>(
            a.qkv, a.hk, a.hv, a.S_init, a.S_final, a.sv);
    }
    if (a.NT > 0) {
        GDN_PROF("chunk_out_fwd", st);
        out_fwd_kernel<IO><<<dim3(a.NT, a.hv), 256, kOutSmem, st>>>(
            a.qkv, a.hk, a.hv, (const IO*)a.z, a.norm_w, a.norm_eps, (IO*)a.o_out,
            (IO*)a.y_out, a.sv);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_fwd(const ChunkArgs& a, cudaStream_t st) {
    return a.bf16 ? chunk_fwd_t<__nv_bfloat16>(a, st) : chunk_fwd_t<float>(a, st);
}

}  // namespace gdn
