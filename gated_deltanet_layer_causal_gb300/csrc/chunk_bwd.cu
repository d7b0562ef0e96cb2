// Backward of the chunked gated delta rule (and of the fused gated RMSNorm).
//
// Per chunk, with P = (Q K^T) (.) Gam (.) [i>=j] (Gam_ij = e^{gam_i - gam_j}),
// K~ = diag(e^{gam_L - gam}) K, Q~ = diag(e^gam) Q, and dS the gradient of the
// state at the chunk END:
//   dU  = P^T dO + K~ dS^T                                   (local + state)
//   dS0 = e^{gam_L} dS + Q~^T dO - W^T dU   (on S^T; the reverse state pass)
//   dQ  = Q~-part: diag(e^gam) dO S0  +  (dO U^T (.) Gam (.) M) K
//   dK  = (dO U^T (.) Gam (.) M)^T Q + diag(e^{gam_L-gam}) U dS
//         + diag(beta e^gam) T^T dW + dKK K + dKK^T K
//   dW  = -dU S0 ;  dV = diag(beta) T^T dU
//   dA  = -T^T (dW (D_be K)^T + dU (D_b V)^T) T^T  (strictly lower part)
//   dKK = dA (.) beta_i Gam_ij ;  dbeta, dgam from every place beta and gam
//   enter; dg = reverse in-chunk cumsum of dgam; da, db through the gates.
// The q/k gradients of the v-heads that share a k-head are summed in a fixed
// order ("[6/8] feat(models): port Qwen3.5 / Qwen3-Next GDN to the head-sharded
// layer", "Summary of an earlier run": the grouped-value accumulation decides
// bitwise results), so the whole backward is run-to-run reproducible.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace gdn {

constexpr int kL4 = 132, kL8 = 136, kM4 = 68, kM8 = 72;

__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// gam with padding rows continuing the last valid value (keeps Gam finite)
__device__ __forceinline__ void load_gam(float* gam, const float* src, const ChunkInfo& ci,
                                         int hv, int h) {
    const int tid = threadIdx.x;
    if (tid < 64) gam[tid] = src[(int64_t)(ci.start + min(tid, ci.len - 1)) * hv + h];
}

// ------------------------------------------------------------------ B1: local
// grid (NT, Hv), 256 threads.  Gated-norm backward (dO, dz, dnorm_w partials)
// and dU_local = P^T dO.
constexpr size_t kB1Smem = sizeof(float) * (2 * 64 * kL4 + 64 * kL8 + 64 * kM8 + 64);

template <class IO>
__global__ void __launch_bounds__(256)
bwd_local_kernel(const float* __restrict__ qkv, int hk, int hv, const IO* z, const float* norm_w,
                 float norm_eps, const IO* __restrict__ dy, IO* dz, FwdSaved sv, BwdScratch w) {
    extern __shared__ float sm[];
    float* Qs = sm;
    float* Ks = Qs + 64 * kL4;
    float* dOs = Ks + 64 * kL4;
    float* Ps = dOs + 64 * kL8;
    float* gam = Ps + 64 * kM8;
    const ChunkInfo ci = sv.chunks[blockIdx.x];
    if (ci.len == 0) return;
    const int h = blockIdx.y, kh = h / (hv / hk), tid = threadIdx.x, L = ci.len;
    const int lane = tid & 31, warp = tid >> 5;
    const int C = (2 * hk + hv) * kD;
    for (int idx = tid; idx < 64 * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 q4 = zero4(), k4 = zero4();
        if (r < L) {
            int64_t t = ci.start + r;
            q4 = ld4(qkv + t * C + kh * kD + c4);
            k4 = ld4(qkv + t * C + (int64_t)hk * kD + kh * kD + c4);
        }
        st4(Qs + r * kL4 + c4, q4);
        st4(Ks + r * kL4 + c4, k4);
    }
    load_gam(gam, sv.gam, ci, hv, h);
    // norm backward, one warp per row
    float4 wacc = zero4();
    const float4 w4 = z ? ld4(norm_w + lane * 4) : zero4();
    for (int r = warp; r < 64; r += 8) {
        float4 d4 = zero4();
        if (r < L) {
            const int64_t off = ((int64_t)(ci.start + r) * hv + h) * kD + lane * 4;
            if (z) {
                NormRowGrad gr = norm_row_bwd(ld4(sv.o + off), ld4(z + off), ld4(dy + off), w4,
                                              norm_eps, wacc);
                d4 = gr.d_o;
                st4(dz + off, gr.dz);
            } else {
                d4 = ld4(dy + off);
            }
            st4(w.dO + off, d4);
        }
        st4(dOs + r * kL8 + lane * 4, d4);
    }
    if (z) {
        __shared__ float4 red[8][32];
        red[warp][lane] = wacc;
        __syncthreads();
        if (warp == 0) {
            float4 s = red[0][lane];
            for (int i = 1; i < 8; i++) {
                s.x += red[i][lane].x; s.y += red[i][lane].y;
                s.z += red[i][lane].z; s.w += red[i][lane].w;
            }
            st4(w.nw_part + ((int64_t)blockIdx.x * hv + h) * kD + lane * 4, s);
        }
    }
    __syncthreads();
    {
        typename Tile<64, 64, 8>::Acc acc;
        tile_zero<64, 64, 8>(acc);
        tile_mma<64, 64, kD, 8>(acc, [&](int r, int k) { return Qs[r * kL4 + k]; },
                                [&](int k, int c) { return Ks[c * kL4 + k]; });
        tile_each<64, 64, 8>(acc, [&](int r, int c, float& v) {
            Ps[r * kM8 + c] = (c <= r) ? v * expf(gam[r] - gam[c]) : 0.f;
        });
    }
    __syncthreads();
    typename Tile<64, kD, 8>::Acc acc;
    tile_zero<64, kD, 8>(acc);
    tile_mma<64, kD, 64, 8>(acc, [&](int j, int i) { return Ps[i * kM8 + j]; },
                            [&](int i, int a) { return dOs[i * kL8 + a]; });
    tile_each2<64, kD, 8>(acc, [&](int r, int c, float& v0, float& v1) {
        if (r < L)
            *reinterpret_cast<float2*>(w.dU + ((int64_t)(ci.start + r) * hv + h) * kD + c) =
                make_float2(v0, v1);
    });
}

// ------------------------------------------------------------------ B2: reverse state pass
// grid (d_v / 32, Hv, N), 128 threads.  Carries a 32-row slice of dS (as
// dS^T[b][a] in the accumulators) from the last chunk of the sequence to the
// first; stores dS at every chunk end and completes dU.
constexpr int kSl = 32, kLdS = kSl + 8;
constexpr size_t kB2Smem = sizeof(float) * (2 * 64 * kL8 + 2 * 64 * kLdS + kD * kLdS + 3 * 64);

__global__ void __launch_bounds__(128)
bwd_state_kernel(const float* __restrict__ qkv, int hk, int hv, const float* dS_final,
                 float* dS_init, FwdSaved sv, BwdScratch w) {
    extern __shared__ float sm[];
    float* X1 = sm;                    // K, then Q
    float* X2 = X1 + 64 * kL8;         // W
    float* dOs = X2 + 64 * kL8;        // [64][kLdS]
    float* dUs = dOs + 64 * kLdS;      // [64][kLdS]
    float* dSt = dUs + 64 * kLdS;      // [128][kLdS]
    float* gam = dSt + kD * kLdS;
    float* fk = gam + 64;
    float* eg = fk + 64;
    const int sl = blockIdx.x, h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
    const int a0 = sl * kSl, kh = h / (hv / hk);
    const int C = (2 * hk + hv) * kD;
    const int64_t sbase = ((int64_t)n * hv + h) * kD * kD;
    typename Tile<kD, kSl, 4>::Acc sacc;
    tile_each<kD, kSl, 4>(sacc, [&](int b, int a, float& v) {
        v = dS_final ? dS_final[sbase + (int64_t)(a0 + a) * kD + b] : 0.f;
        dSt[b * kLdS + a] = v;
    });
    const int c0 = sv.seq_chunk[n], c1 = sv.seq_chunk[n + 1];
    for (int ci = c1 - 1; ci >= c0; ci--) {
        const ChunkInfo info = sv.chunks[ci];
        const int L = info.len;
        __syncthreads();
        for (int idx = tid; idx < 64 * 32; idx += 128) {
            int r = idx >> 5, c4 = (idx & 31) * 4;
            float4 k4 = zero4(), w4 = zero4();
            if (r < L) {
                int64_t t = info.start + r;
                k4 = ld4(qkv + t * C + (int64_t)hk * kD + kh * kD + c4);
                w4 = ld4(sv.W + (t * hv + h) * kD + c4);
            }
            st4(X1 + r * kL8 + c4, k4);
            st4(X2 + r * kL8 + c4, w4);
        }
        for (int idx = tid; idx < 64 * kSl / 4; idx += 128) {
            int r = idx / (kSl / 4), c4 = (idx % (kSl / 4)) * 4;
            float4 o4 = zero4(), u4 = zero4();
            if (r < L) {
                int64_t off = ((int64_t)(info.start + r) * hv + h) * kD + a0 + c4;
                o4 = ld4(w.dO + off);
                u4 = ld4(w.dU + off);
            }
            st4(dOs + r * kLdS + c4, o4);
            st4(dUs + r * kLdS + c4, u4);
        }
        load_gam(gam, sv.gam, info, hv, h);
        // gradient of the state at this chunk's end
        const int64_t obase = ((int64_t)ci * hv + h) * kD * kD;
        tile_each2<kD, kSl, 4>(sacc, [&](int b, int a, float& v0, float& v1) {
            w.dS[obase + (int64_t)(a0 + a) * kD + b] = v0;
            w.dS[obase + (int64_t)(a0 + a + 1) * kD + b] = v1;
        });
        __syncthreads();
        if (tid < 64) {
            fk[tid] = tid < L ? expf(gam[L - 1] - gam[tid]) : 0.f;
            eg[tid] = tid < L ? expf(gam[tid]) : 0.f;
        }
        __syncthreads();
        // dU = dU_local + K~ dS^T  (64 x slice)
        typename Tile<64, kSl, 4>::Acc uacc;
        tile_zero<64, kSl, 4>(uacc);
        tile_mma<64, kSl, kD, 4>(uacc, [&](int i, int b) { return fk[i] * X1[i * kL8 + b]; },
                                 [&](int b, int a) { return dSt[b * kLdS + a]; });
        __syncthreads();   // X1 (K) no longer read: load Q over it
        for (int idx = tid; idx < 64 * 32; idx += 128) {
            int r = idx >> 5, c4 = (idx & 31) * 4;
            float4 q4 = zero4();
            if (r < L) q4 = ld4(qkv + (int64_t)(info.start + r) * C + kh * kD + c4);
            st4(X1 + r * kL8 + c4, q4);
        }
        tile_each<64, kSl, 4>(uacc, [&](int i, int a, float& v) {
            float u = i < L ? dUs[i * kLdS + a] + v : 0.f;
            dUs[i * kLdS + a] = u;
            if (i < L) w.dU[((int64_t)(info.start + i) * hv + h) * kD + a0 + a] = u;
        });
        __syncthreads();
        // dS^T = e^{gam_L} dS^T + Q~^T dO - W^T dU
        const float dl = expf(gam[L - 1]);
        tile_each<kD, kSl, 4>(sacc, [&](int, int, float& v) { v *= dl; });
        tile_mma<kD, kSl, 64, 4>(sacc, [&](int b, int i) { return eg[i] * X1[i * kL8 + b]; },
                                 [&](int i, int a) { return dOs[i * kLdS + a]; });
        tile_mma<kD, kSl, 64, 4>(sacc, [&](int b, int i) { return -X2[i * kL8 + b]; },
                                 [&](int i, int a) { return dUs[i * kLdS + a]; });
        tile_each<kD, kSl, 4>(sacc, [&](int b, int a, float& v) { dSt[b * kLdS + a] = v; });
    }
    if (dS_init)
        tile_each<kD, kSl, 4>(sacc, [&](int b, int a, float& v) {
            dS_init[sbase + (int64_t)(a0 + a) * kD + b] = v;
        });
}

// ------------------------------------------------------------------ B3a: state-facing terms
// grid (NT, Hv), 256 threads.
//   X = dO S0 -> dQ partial e^gam X, dgam_i += e^{gam_i} X_i . Q_i
//   dW = -dU S0
//   dK~ = U dS -> dK partial fk dK~, dgam_j -= Z_j, dgam_L += sum Z + e^{gam_L}<dS, S0>
constexpr size_t kB3aSmem = sizeof(float) * (kD * kL8 + 2 * 64 * kL4 + 3 * 64 + 2 * 64 + 8);

__global__ void __launch_bounds__(256)
bwd_sfacing_kernel(const float* __restrict__ qkv, int hk, int hv, FwdSaved sv, BwdScratch w) {
    extern __shared__ float sm[];
    float* Ss = sm;                    // [128][kL8]  S0, then dS
    float* A1 = Ss + kD * kL8;         // [64][kL4]   dO, then U
    float* A2 = A1 + 64 * kL4;         // [64][kL4]   dU
    float* gam = A2 + 64 * kL4;
    float* eg = gam + 64;
    float* fk = eg + 64;
    float* part = fk + 64;             // [2][64]
    float* red = part + 128;           // [8]
    const ChunkInfo ci = sv.chunks[blockIdx.x];
    if (ci.len == 0) return;
    const int h = blockIdx.y, kh = h / (hv / hk), tid = threadIdx.x, L = ci.len;
    const int C = (2 * hk + hv) * kD;
    const int64_t sb = ((int64_t)blockIdx.x * hv + h) * kD * kD;
    for (int idx = tid; idx < kD * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        st4(Ss + r * kL8 + c4, ld4(sv.S0 + sb + r * kD + c4));
    }
    for (int idx = tid; idx < 64 * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 o4 = zero4(), u4 = zero4();
        if (r < L) {
            int64_t off = ((int64_t)(ci.start + r) * hv + h) * kD + c4;
            o4 = ld4(w.dO + off);
            u4 = ld4(w.dU + off);
        }
        st4(A1 + r * kL4 + c4, o4);
        st4(A2 + r * kL4 + c4, u4);
    }
    load_gam(gam, sv.gam, ci, hv, h);
    __syncthreads();
    if (tid < 64) {
        eg[tid] = tid < L ? expf(gam[tid]) : 0.f;
        fk[tid] = tid < L ? expf(gam[L - 1] - gam[tid]) : 0.f;
    }
    __syncthreads();
    float dg_row[2] = {0.f, 0.f};   // this thread's share of dgam (rows tid, tid-64 unused)
    typename Tile<64, kD, 8>::Acc acc;
    // X = dO S0
    tile_zero<64, kD, 8>(acc);
    tile_mma<64, kD, kD, 8>(acc, [&](int i, int a) { return A1[i * kL4 + a]; },
                            [&](int a, int b) { return Ss[a * kL8 + b]; });
    tile_each2<64, kD, 8>(acc, [&](int i, int b, float& v0, float& v1) {
        if (i < L)
            *reinterpret_cast<float2*>(w.dQv + ((int64_t)(ci.start + i) * hv + h) * kD + b) =
                make_float2(eg[i] * v0, eg[i] * v1);
    });
    tile_rowpart<64, kD, 8>(acc, [&](int i, int b, float v) {
        return i < L ? eg[i] * v * qkv[(int64_t)(ci.start + i) * C + kh * kD + b] : 0.f;
    }, part);
    __syncthreads();
    if (tid < 64) dg_row[0] = part[tid] + part[64 + tid];
    // dW = -dU S0
    tile_zero<64, kD, 8>(acc);
    tile_mma<64, kD, kD, 8>(acc, [&](int i, int a) { return A2[i * kL4 + a]; },
                            [&](int a, int b) { return Ss[a * kL8 + b]; });
    tile_each2<64, kD, 8>(acc, [&](int i, int b, float& v0, float& v1) {
        if (i < L)
            *reinterpret_cast<float2*>(w.dW + ((int64_t)(ci.start + i) * hv + h) * kD + b) =
                make_float2(-v0, -v1);
    });
    __syncthreads();
    // swap in dS (and take <dS, S0> on the way) and U
    float dot = 0.f;
    const float* dSg = w.dS + sb;
    for (int idx = tid; idx < kD * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 s4 = ld4(Ss + r * kL8 + c4), d4 = ld4(dSg + r * kD + c4);
        dot += s4.x * d4.x + s4.y * d4.y + s4.z * d4.z + s4.w * d4.w;
        st4(Ss + r * kL8 + c4, d4);
    }
    for (int idx = tid; idx < 64 * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 u4 = zero4();
        if (r < L) u4 = ld4(sv.U + ((int64_t)(ci.start + r) * hv + h) * kD + c4);
        st4(A1 + r * kL4 + c4, u4);
    }
    dot = warp_sum(dot);
    if ((tid & 31) == 0) red[tid >> 5] = dot;
    __syncthreads();
    // dK~ = U dS
    tile_zero<64, kD, 8>(acc);
    tile_mma<64, kD, kD, 8>(acc, [&](int j, int a) { return A1[j * kL4 + a]; },
                            [&](int a, int b) { return Ss[a * kL8 + b]; });
    tile_each2<64, kD, 8>(acc, [&](int j, int b, float& v0, float& v1) {
        if (j < L)
            *reinterpret_cast<float2*>(w.dKv + ((int64_t)(ci.start + j) * hv + h) * kD + b) =
                make_float2(fk[j] * v0, fk[j] * v1);
    });
    tile_rowpart<64, kD, 8>(acc, [&](int j, int b, float v) {
        return j < L ? fk[j] * v * qkv[(int64_t)(ci.start + j) * C + (int64_t)hk * kD + kh * kD + b]
                     : 0.f;
    }, part);
    __syncthreads();
    if (tid < 64) {
        float z = part[tid] + part[64 + tid];   // Z_j
        dg_row[1] = -z;
        part[tid] = z;                          // reuse for the sum over j
    }
    __syncthreads();
    if (tid < 64 && tid < L) {
        float g = dg_row[0] + dg_row[1];
        if (tid == L - 1) {
            float zs = 0.f, dd = 0.f;
            for (int j = 0; j < 64; j++) zs += part[j];
            for (int i = 0; i < 8; i++) dd += red[i];
            g += zs + expf(gam[L - 1]) * dd;
        }
        w.dgam[(int64_t)(ci.start + tid) * hv + h] = g;
    }
}

// ------------------------------------------------------------------ B3b: chunk-local terms
// grid (NT, Hv), 256 threads.  Finishes dQ, dK (per v-head), dV, dbeta, dgam,
// then dg, da, db and the per-chunk dA_log / ddt_bias partials.
constexpr size_t kB3bSmem =
    sizeof(float) * (4 * 64 * kL8 + 3 * 64 * kM4 + 64 * kM8 + 8 * 64 + 2 * 64 + 4 * 64 + 16);

template <class IO>
__global__ void __launch_bounds__(256, 1)
bwd_local2_kernel(const float* __restrict__ qkv, const IO* __restrict__ av,
                  const IO* __restrict__ bv, const float* __restrict__ A_log,
                  const float* __restrict__ dt_bias, int hk, int hv, float* __restrict__ dqkv,
                  IO* __restrict__ da, IO* __restrict__ db, float* __restrict__ gate_part,
                  FwdSaved sv, BwdScratch w) {
    extern __shared__ float sm[];
    float* B0 = sm;                    // Q, then V      [64][kL8]
    float* B1 = B0 + 64 * kL8;         // K              [64][kL8]
    float* B2 = B1 + 64 * kL8;         // dO, then dW    [64][kL8]
    float* B3 = B2 + 64 * kL8;         // U, then dU     [64][kL8]
    float* M0 = B3 + 64 * kL8;         // GamKK          [64][kM4]
    float* M1 = M0 + 64 * kM4;         // dPm, then T    [64][kM4]
    float* M2 = M1 + 64 * kM4;         // A, dT, dKK     [64][kM4]
    float* M3 = M2 + 64 * kM4;         // Y              [64][kM8]
    float* gam = M3 + 64 * kM8;
    float* eg = gam + 64;
    float* bet = eg + 64;
    float* be = bet + 64;
    float* dgs = be + 64;              // dgam accumulated here
    float* dbs = dgs + 64;             // dbeta accumulated here
    float* rk = dbs + 64;              // scratch row values
    float* sc = rk + 64;               // scratch
    float* rpart = sc + 64;            // [2][64]
    float* cpart = rpart + 128;        // [4][64]
    float* red = cpart + 256;          // [16]
    const ChunkInfo ci = sv.chunks[blockIdx.x];
    if (ci.len == 0) return;
    const int h = blockIdx.y, kh = h / (hv / hk), tid = threadIdx.x, L = ci.len;
    const int C = (2 * hk + hv) * kD;
    auto tok = [&](int i) { return (int64_t)(ci.start + i); };
    auto vrow = [&](int i) { return (tok(i) * hv + h) * kD; };
    // ---- phase 1: Q, K, dO, U
    for (int idx = tid; idx < 64 * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 q4 = zero4(), k4 = zero4(), o4 = zero4(), u4 = zero4();
        if (r < L) {
            q4 = ld4(qkv + tok(r) * C + kh * kD + c4);
            k4 = ld4(qkv + tok(r) * C + (int64_t)hk * kD + kh * kD + c4);
            o4 = ld4(w.dO + vrow(r) + c4);
            u4 = ld4(sv.U + vrow(r) + c4);
        }
        st4(B0 + r * kL8 + c4, q4);
        st4(B1 + r * kL8 + c4, k4);
        st4(B2 + r * kL8 + c4, o4);
        st4(B3 + r * kL8 + c4, u4);
    }
    load_gam(gam, sv.gam, ci, hv, h);
    if (tid < 64) {
        float b = tid < L ? sv.beta[tok(tid) * hv + h] : 0.f;
        bet[tid] = b;
        dgs[tid] = 0.f;
        dbs[tid] = 0.f;
    }
    __syncthreads();
    if (tid < 64) {
        eg[tid] = tid < L ? expf(gam[tid]) : 0.f;
        be[tid] = bet[tid] * eg[tid];
    }
    {
        typename Tile<64, 64, 8>::Acc qk, dou;
        tile_zero<64, 64, 8>(qk);
        tile_zero<64, 64, 8>(dou);
        tile_mma<64, 64, kD, 8>(qk, [&](int i, int b) { return B0[i * kL8 + b]; },
                                [&](int b, int j) { return B1[j * kL8 + b]; });
        tile_mma<64, 64, kD, 8>(dou, [&](int i, int a) { return B2[i * kL8 + a]; },
                                [&](int a, int j) { return B3[j * kL8 + a]; });
        // dPm = dOU (.) Gam (.) M ; R = dPm (.) QK  (dgam_i += sum_j R, dgam_j -= sum_i R)
        tile_each<64, 64, 8>(dou, [&](int i, int j, float& v) {
            float gm = (j <= i) ? expf(gam[i] - gam[j]) : 0.f;
            v *= gm;
            M1[i * kM4 + j] = v;
        });
        // elementwise R into dou (fragments of qk and dou align)
        {
            using TL = Tile<64, 64, 8>;
#pragma unroll
            for (int a = 0; a < TL::MPW; a++)
#pragma unroll
                for (int b = 0; b < TL::NPW; b++)
#pragma unroll
                    for (int e = 0; e < 4; e++) dou[a][b][e] *= qk[a][b][e];
        }
        tile_rowpart<64, 64, 8>(dou, [&](int, int, float v) { return v; }, rpart);
        tile_colpart<64, 64, 8>(dou, [&](int, int, float v) { return v; }, cpart);
    }
    __syncthreads();
    if (tid < 64)
        dgs[tid] += (rpart[tid] + rpart[64 + tid]) -
                    (cpart[tid] + cpart[64 + tid] + cpart[128 + tid] + cpart[192 + tid]);
    typename Tile<64, kD, 8>::Acc dk;
    tile_zero<64, kD, 8>(dk);
    {
        typename Tile<64, kD, 8>::Acc dq;
        tile_zero<64, kD, 8>(dq);
        tile_mma<64, kD, 64, 8>(dq, [&](int i, int j) { return M1[i * kM4 + j]; },
                                [&](int j, int b) { return B1[j * kL8 + b]; });
        tile_each2<64, kD, 8>(dq, [&](int i, int b, float& v0, float& v1) {
            if (i < L) {
                float2* p = reinterpret_cast<float2*>(w.dQv + vrow(i) + b);
                float2 o = *p;
                *p = make_float2(o.x + v0, o.y + v1);
            }
        });
        tile_mma<64, kD, 64, 8>(dk, [&](int j, int i) { return M1[i * kM4 + j]; },
                                [&](int i, int b) { return B0[i * kL8 + b]; });
    }
    __syncthreads();
    // ---- phase 2: V, dW, dU (K stays)
    for (int idx = tid; idx < 64 * 32; idx += 256) {
        int r = idx >> 5, c4 = (idx & 31) * 4;
        float4 v4 = zero4(), w4 = zero4(), u4 = zero4();
        if (r < L) {
            v4 = ld4(qkv + tok(r) * C + (int64_t)2 * hk * kD + h * kD + c4);
            w4 = ld4(w.dW + vrow(r) + c4);
            u4 = ld4(w.dU + vrow(r) + c4);
        }
        st4(B0 + r * kL8 + c4, v4);
        st4(B2 + r * kL8 + c4, w4);
        st4(B3 + r * kL8 + c4, u4);
    }
    {
        typename Tile<64, 64, 8>::Acc kk;
        tile_zero<64, 64, 8>(kk);
        tile_mma<64, 64, kD, 8>(kk, [&](int i, int b) { return B1[i * kL8 + b]; },
                                [&](int b, int j) { return B1[j * kL8 + b]; });
        tile_each<64, 64, 8>(kk, [&](int i, int j, float& v) {
            float gkk = (j < i) ? expf(gam[i] - gam[j]) * v : 0.f;
            M0[i * kM4 + j] = gkk;
            M2[i * kM4 + j] = bet[i] * gkk;
        });
    }
    __syncthreads();
    tril_inverse64(M2, kM4, M1, kM4);
    __syncthreads();
    {   // dT = dW (D_be K)^T + dU (D_b V)^T
        typename Tile<64, 64, 8>::Acc dt;
        tile_zero<64, 64, 8>(dt);
        tile_mma<64, 64, kD, 8>(dt, [&](int i, int b) { return B2[i * kL8 + b]; },
                                [&](int b, int j) { return be[j] * B1[j * kL8 + b]; });
        tile_mma<64, 64, kD, 8>(dt, [&](int i, int a) { return B3[i * kL8 + a]; },
                                [&](int a, int j) { return bet[j] * B0[j * kL8 + a]; });
        tile_each<64, 64, 8>(dt, [&](int i, int j, float& v) { M2[i * kM4 + j] = v; });
    }
    {   // T^T dW: dK += D_be (.), dbeta_j += e^gam_j r_j, dgam_j += be_j r_j
        typename Tile<64, kD, 8>::Acc x;
        tile_zero<64, kD, 8>(x);
        tile_mma<64, kD, 64, 8>(x, [&](int j, int i) { return M1[i * kM4 + j]; },
                                [&](int i, int b) { return B2[i * kL8 + b]; });
        tile_rowpart<64, kD, 8>(x, [&](int j, int b, float v) { return v * B1[j * kL8 + b]; },
                                rpart);
        using TW = Tile<64, kD, 8>;
        const int lane = tid & 31, g = lane >> 2;
        const int m0 = TW::m0();
#pragma unroll
        for (int a = 0; a < TW::MPW; a++)
#pragma unroll
            for (int b = 0; b < TW::NPW; b++)
#pragma unroll
                for (int e = 0; e < 4; e++) dk[a][b][e] += be[m0 + a * 16 + g + (e >> 1) * 8] * x[a][b][e];
    }
    __syncthreads();
    if (tid < 64) {
        float r = rpart[tid] + rpart[64 + tid];
        dbs[tid] += eg[tid] * r;
        dgs[tid] += be[tid] * r;
    }
    {   // T^T dU: dV = D_b (.), dbeta_j += sum_a (.) V
        typename Tile<64, kD, 8>::Acc x;
        tile_zero<64, kD, 8>(x);
        tile_mma<64, kD, 64, 8>(x, [&](int j, int i) { return M1[i * kM4 + j]; },
                                [&](int i, int a) { return B3[i * kL8 + a]; });
        tile_each2<64, kD, 8>(x, [&](int j, int a, float& v0, float& v1) {
            if (j < L)
                *reinterpret_cast<float2*>(dqkv + tok(j) * C + (int64_t)2 * hk * kD + h * kD + a) =
                    make_float2(bet[j] * v0, bet[j] * v1);
        });
        tile_rowpart<64, kD, 8>(x, [&](int j, int a, float v) { return v * B0[j * kL8 + a]; },
                                rpart);
    }
    __syncthreads();
    if (tid < 64) dbs[tid] += rpart[tid] + rpart[64 + tid];
    {   // Y = dT T^T
        typename Tile<64, 64, 8>::Acc y;
        tile_zero<64, 64, 8>(y);
        tile_mma<64, 64, 64, 8>(y, [&](int i, int j) { return M2[i * kM4 + j]; },
                                [&](int j, int m) { return M1[m * kM4 + j]; });
        tile_each<64, 64, 8>(y, [&](int i, int m, float& v) { M3[i * kM8 + m] = v; });
    }
    __syncthreads();
    {   // dA = -T^T Y (strictly lower) ; dKK = dA beta_j Gam ; dbeta, dgam
        typename Tile<64, 64, 8>::Acc x;
        tile_zero<64, 64, 8>(x);
        tile_mma<64, 64, 64, 8>(x, [&](int j, int i) { return M1[i * kM4 + j]; },
                                [&](int i, int m) { return M3[i * kM8 + m]; });
        tile_each<64, 64, 8>(x, [&](int j, int m, float& v) {
            float dA = (m < j) ? -v : 0.f;
            v = dA * M0[j * kM4 + m];       // dA (.) GamKK
            M2[j * kM4 + m] = (m < j) ? dA * bet[j] * expf(gam[j] - gam[m]) : 0.f;
        });
        tile_rowpart<64, 64, 8>(x, [&](int, int, float v) { return v; }, rpart);
        tile_colpart<64, 64, 8>(x, [&](int j, int, float v) { return bet[j] * v; }, cpart);
    }
    __syncthreads();
    if (tid < 64) {
        float r = rpart[tid] + rpart[64 + tid];
        dbs[tid] += r;
        dgs[tid] += bet[tid] * r -
                    (cpart[tid] + cpart[64 + tid] + cpart[128 + tid] + cpart[192 + tid]);
    }
    // dK += dKK K + dKK^T K
    tile_mma<64, kD, 64, 8>(dk, [&](int j, int m) { return M2[j * kM4 + m]; },
                            [&](int m, int b) { return B1[m * kL8 + b]; });
    tile_mma<64, kD, 64, 8>(dk, [&](int j, int m) { return M2[m * kM4 + j]; },
                            [&](int m, int b) { return B1[m * kL8 + b]; });
    tile_each2<64, kD, 8>(dk, [&](int j, int b, float& v0, float& v1) {
        if (j < L) {
            float2* p = reinterpret_cast<float2*>(w.dKv + vrow(j) + b);
            float2 o = *p;
            *p = make_float2(o.x + v0, o.y + v1);
        }
    });
    __syncthreads();
    // ---- phase 3: dg = reverse cumsum of dgam; gates
    if (tid < 64) sc[tid] = tid < L ? dgs[tid] + w.dgam[tok(tid) * hv + h] : 0.f;
    __syncthreads();
    if (tid < 32) {
        // reverse inclusive scan over 64 values, two per lane
        const int lane = tid;
        float a = sc[63 - 2 * lane], b = sc[62 - 2 * lane], s = a + b;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float u = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += u;
        }
        float ex = s - (a + b);
        rk[63 - 2 * lane] = ex + a;
        rk[62 - 2 * lane] = ex + a + b;
    }
    __syncthreads();
    float gterm = 0.f, dterm = 0.f;
    if (tid < L) {
        const float dg = rk[tid];
        const float Aexp = expf(A_log[h]);
        const float xa = to_f(av[tok(tid) * hv + h]) + dt_bias[h];
        const float gval = -Aexp * softplusf_(xa);
        const float dav = dg * (-Aexp) * sigmoidf_(xa);
        const float bb = bet[tid];
        da[tok(tid) * hv + h] = from_f<IO>(dav);
        db[tok(tid) * hv + h] = from_f<IO>(dbs[tid] * bb * (1.f - bb));
        w.dgs[tok(tid) * hv + h] = dg;
        gterm = dg * gval;
        dterm = dav;
    }
    if (tid < 64) {
        gterm = warp_sum(gterm);
        dterm = warp_sum(dterm);
        if ((tid & 31) == 0) { red[tid >> 5] = gterm; red[2 + (tid >> 5)] = dterm; }
    }
    __syncthreads();
    if (tid == 0) {
        gate_part[((int64_t)blockIdx.x * hv + h) * 2 + 0] = red[0] + red[1];
        gate_part[((int64_t)blockIdx.x * hv + h) * 2 + 1] = red[2] + red[3];
    }
}

// ------------------------------------------------------------------ B4: GVA sum
// dqkv q/k channels of k-head kh = sum over its G v-heads in order j = 0..G-1.
__global__ void gva_sum_kernel(const float* __restrict__ dQv, const float* __restrict__ dKv,
                               int64_t T, int hk, int hv, float* __restrict__ dqkv) {
    const int G = hv / hk, C = (2 * hk + hv) * kD;
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // over T * hk * 32
    if (idx >= T * hk * 32) return;
    const int c4 = (int)(idx % 32) * 4;
    const int kh = (int)(idx / 32 % hk);
    const int64_t t = idx / 32 / hk;
    float4 q = zero4(), k = zero4();
    for (int j = 0; j < G; j++) {
        const int64_t off = (t * hv + kh * G + j) * kD + c4;
        float4 a = ld4(dQv + off), b = ld4(dKv + off);
        q.x += a.x; q.y += a.y; q.z += a.z; q.w += a.w;
        k.x += b.x; k.y += b.y; k.z += b.z; k.w += b.w;
    }
    st4(dqkv + t * C + kh * kD + c4, q);
    st4(dqkv + t * C + (int64_t)hk * kD + kh * kD + c4, k);
}

// dA_log[h] = sum over chunks of part[c][h][0]; ddt_bias[h] likewise [1]; fixed order.
__global__ void gate_reduce_kernel(const float* __restrict__ part, int NT, int hv, float* dA_log,
                                   float* ddt_bias) {
    int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= hv) return;
    float a = 0.f, b = 0.f;
    for (int c = 0; c < NT; c++) {
        a += part[((int64_t)c * hv + h) * 2 + 0];
        b += part[((int64_t)c * hv + h) * 2 + 1];
    }
    if (dA_log) dA_log[h] = a;
    if (ddt_bias) ddt_bias[h] = b;
}

__global__ void colsum2_kernel(const float* __restrict__ part, int64_t nparts, int cols,
                               float* __restrict__ out) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= cols) return;
    float acc = 0.f;
    for (int64_t p = 0; p < nparts; p++) acc += part[p * cols + i];
    out[i] = acc;
}

// ------------------------------------------------------------------ launcher
template <class IO>
static cudaError_t chunk_bwd_t(const ChunkArgs& a, const BwdScratch& w, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(bwd_local_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kB1Smem);
        cudaFuncSetAttribute(bwd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kB2Smem);
        cudaFuncSetAttribute(bwd_sfacing_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kB3aSmem);
        cudaFuncSetAttribute(bwd_local2_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kB3bSmem);
        attr = true;
    }
    float* gate_part = w.nw_part + (size_t)a.NT * a.hv * kD;
    if (a.NT > 0) {
        GDN_PROF("chunk_bwd_local", st);
        bwd_local_kernel<IO><<<dim3(a.NT, a.hv), 256, kB1Smem, st>>>(
            a.qkv, a.hk, a.hv, (const IO*)a.z, a.norm_w, a.norm_eps, (const IO*)a.dy,
            (IO*)a.dz, a.sv, w);
    }
    if (a.N > 0) {
        GDN_PROF("chunk_bwd_state", st);
        bwd_state_kernel<<<dim3(kD / kSl, a.hv, a.N), 128, kB2Smem, st>>>(
            a.qkv, a.hk, a.hv, a.dS_final, a.dS_init, a.sv, w);
    }
    if (a.NT > 0) {
        {
            GDN_PROF("chunk_bwd_sfacing", st);
            bwd_sfacing_kernel<<<dim3(a.NT, a.hv), 256, kB3aSmem, st>>>(a.qkv, a.hk, a.hv, a.sv,
                                                                          w);
        }
        GDN_PROF("chunk_bwd_wy", st);
        bwd_local2_kernel<IO><<<dim3(a.NT, a.hv), 256, kB3bSmem, st>>>(
            a.qkv, (const IO*)a.a, (const IO*)a.b, a.A_log, a.dt_bias, a.hk, a.hv, a.dqkv,
            (IO*)a.da, (IO*)a.db, gate_part, a.sv, w);
    }
    if (a.T > 0) {
        int64_t n = a.T * a.hk * 32;
        GDN_PROF("gva_sum", st);
        gva_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w.dQv, w.dKv, a.T, a.hk,
                                                                    a.hv, a.dqkv);
    }
    if (a.dA_log || a.ddt_bias) {
        if (a.NT > 0) {
            GDN_PROF("gate_reduce", st);
            gate_reduce_kernel<<<(a.hv + 127) / 128, 128, 0, st>>>(gate_part, a.NT, a.hv,
                                                                   a.dA_log, a.ddt_bias);
        } else {
            if (a.dA_log) cudaMemsetAsync(a.dA_log, 0, sizeof(float) * a.hv, st);
            if (a.ddt_bias) cudaMemsetAsync(a.ddt_bias, 0, sizeof(float) * a.hv, st);
        }
    }
    if (a.z && a.dnorm_w) {
        if (a.NT > 0) {
            GDN_PROF("norm_w_reduce", st);
            colsum2_kernel<<<1, kD, 0, st>>>(w.nw_part, (int64_t)a.NT * a.hv, kD, a.dnorm_w);
        } else
            cudaMemsetAsync(a.dnorm_w, 0, sizeof(float) * kD, st);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_bwd(const ChunkArgs& a, const BwdScratch& w, cudaStream_t st) {
    return a.bf16 ? chunk_bwd_t<__nv_bfloat16>(a, w, st) : chunk_bwd_t<float>(a, w, st);
}

}  // namespace gdn
