// Causal depthwise conv1d (4 taps) + SiLU + per-head L2 norm of q and k, and
// its backward.  x may hold the q / k / v channels flat or group-major; the
// output qkv is always flat.
//
// prime-rl #3860 "Summary": the layer runs causal_conv1d over the q/k/v mix with
// cu_seqlens (the conv restarts at every sequence start); "[main] feat(moe):
// Support gated delta net for Qwen3-Next (1/4)", "GDN args": conv kernel 4,
// head dims 128.  L2 normalisation of q and k per (token, k-head), q scaled by
// d_k^-1/2.
//
// HBM-bound.  One warp walks a run of consecutive tokens of one 128-channel
// head; each lane owns 4 channels (one 16-B fp32 / 8-B bf16 vector), keeps the
// previous three inputs in registers (each input row is read once), and the
// per-head sum of squares is a warp shuffle reduction.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace gdn {

constexpr int kConvWarps = 8;
constexpr int kConvRun = 64;   // tokens per warp
// backward: four-token steps each lane holds in its copy ring (two CTAs of
// eight warps per SM fit either way)
template <class T>
constexpr int conv_ring() { return sizeof(T) == 2 ? 4 : 3; }
constexpr int kConvFwdRing = 4;   // forward: the same, input rows only

template <class T>
constexpr size_t conv_fwd_smem() {
    return (size_t)kConvFwdRing * 4 * kConvWarps * 32 * 4 * sizeof(T);
}

// Backward shared memory: per lane a ring of conv_ring steps, each four rows of
// the incoming gradient (float4) and four new input rows (4 x T); reused for
// the dw reduction at the end.
template <class T>
constexpr size_t conv_bwd_smem() {
    return (size_t)conv_ring<T>() * 4 * kConvWarps * 32 * (sizeof(float4) + 4 * sizeof(T));
}

__device__ __forceinline__ int seq_of(const int32_t* cu, int N, int64_t t) {
    // last n with cu[n] <= t (sequences may be empty)
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Raw conv input at position p of sequence n (start s): x, else the conv cache, else 0.
template <class T>
__device__ __forceinline__ float4 conv_in(const T* x, const T* cs, int64_t p, int64_t s, int n,
                                          int C, int c) {
    if (p >= s) return ld4(x + p * C + c);
    int64_t m = (kConvK - 1) + (p - s);
    if (cs == nullptr || m < 0) return make_float4(0.f, 0.f, 0.f, 0.f);
    const T* b = cs + ((int64_t)n * C + c) * (kConvK - 1) + m;
    return make_float4(to_f(b[0]), to_f(b[kConvK - 1]), to_f(b[2 * (kConvK - 1)]),
                       to_f(b[3 * (kConvK - 1)]));
}

__device__ __forceinline__ float conv4(const float (&w)[kConvK], float a3, float a2, float a1,
                                       float a0) {
    // w[3] multiplies the current token (a0), w[0] the token three back
    return w[0] * a3 + w[1] * a2 + w[2] * a1 + w[3] * a0;
}

// Where x's 128-channel block `blk` goes in the conv output qkv (always the
// flat [q (h_k heads) | k (h_k) | v (h_v)] order the chunk kernels read) and
// its role: 0 = q, 1 = k, 2 = v.  Flat x: the same block.  Group-major x
// ("[6/8] feat(models): port Qwen3.5 / Qwen3-Next GDN to the head-sharded
// layer", "What": q/k/v and the conv in group-major layout): block
// kh (2 + G) + r holds q (r = 0), k (r = 1) or v-head kh G + r - 2 of k-head
// group kh, so a group's channels are contiguous.  conv_w and the conv cache
// follow x's channel order.
struct ConvBlock {
    int out, role;
};
__device__ __forceinline__ ConvBlock conv_block(int blk, int hk, int G, bool group_major) {
    if (!group_major) return ConvBlock{blk, blk < hk ? 0 : blk < 2 * hk ? 1 : 2};
    const int kh = blk / (2 + G), r = blk % (2 + G);
    return r == 0 ? ConvBlock{kh, 0}
         : r == 1 ? ConvBlock{hk + kh, 1}
                  : ConvBlock{2 * hk + kh * G + r - 2, 2};
}

// Gradient reaching input x[t] of sequence n ([s, e)) through conv_state_out,
// which copies the sequence's last three inputs: dcso [N, C, 3] (nullable).
__device__ __forceinline__ void add_state_out_grad(float4& o, const float* dcso, int n, int C,
                                                   int c, int64_t t, int64_t e) {
    if (dcso == nullptr || t < e - (kConvK - 1)) return;
    const float* g = dcso + ((int64_t)n * C + c) * (kConvK - 1) + (t - (e - (kConvK - 1)));
    o.x += g[0];
    o.y += g[kConvK - 1];
    o.z += g[2 * (kConvK - 1)];
    o.w += g[3 * (kConvK - 1)];
}

template <class T>
__global__ void __launch_bounds__(kConvWarps * 32)
conv_fwd_kernel(const T* __restrict__ x, const float* __restrict__ w, const T* cs_in,
                const int32_t* __restrict__ cu, int N, int64_t Ttot, int C, int hk, int G,
                bool group_major, float l2_eps, float q_scale, bool rnd, float* __restrict__ out) {
    extern __shared__ __align__(16) unsigned char conv_fwd_smem_raw[];
    T* ring = reinterpret_cast<T*>(conv_fwd_smem_raw);   // [ring][4][threads][4]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = blockIdx.y;
    const int c = grp * kD + lane * 4;   // channel of x, conv_w, the cache
    const ConvBlock cb = conv_block(grp, hk, G, group_major);
    const int oc = cb.out * kD + lane * 4;   // channel of qkv
    const int64_t t0 = ((int64_t)blockIdx.x * kConvWarps + warp) * kConvRun;
    if (t0 >= Ttot) return;
    const int64_t t1 = min(t0 + (int64_t)kConvRun, Ttot);
    const bool norm = cb.role < 2;
    const float scale = cb.role == 0 ? q_scale : 1.f;
    float wr[4][kConvK];
#pragma unroll
    for (int ch = 0; ch < 4; ch++)
#pragma unroll
        for (int j = 0; j < kConvK; j++) wr[ch][j] = w[(c + ch) * kConvK + j];

    int n = seq_of(cu, N, t0);
    int64_t s = cu[n], e = cu[n + 1];
    float4 h1 = conv_in(x, cs_in, t0 - 1, s, n, C, c);
    float4 h2 = conv_in(x, cs_in, t0 - 2, s, n, C, c);
    float4 h3 = conv_in(x, cs_in, t0 - 3, s, n, C, c);
    int64_t t = t0;
    if (t1 <= e) {
        // the whole run lies in one sequence: four tokens per step with
        // independent reductions; each lane copies its own input rows
        // kConvFwdRing-1 steps ahead into its ring slots (cp.async)
        constexpr int kThr = kConvWarps * 32;
        const int tid = threadIdx.x, nsteps = (int)((t1 - t0) / 4);
        auto issue = [&](int i) {
            if (i < nsteps) {
#pragma unroll
                for (int u = 0; u < 4; u++)
                    cp_async_row4(&ring[(((i % kConvFwdRing) * 4 + u) * kThr + tid) * 4],
                                  x + (t0 + 4 * (int64_t)i + u) * C + c);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int i = 0; i < kConvFwdRing - 1; i++) issue(i);
        for (int i = 0; i < nsteps; i++, t += 4) {
            issue(i + kConvFwdRing - 1);   // the slot step i-1 used
            cp_async_wait<kConvFwdRing - 1>();
            float4 xs[4], o[4];
#pragma unroll
            for (int u = 0; u < 4; u++)
                xs[u] = ld4(&ring[(((i % kConvFwdRing) * 4 + u) * kThr + tid) * 4]);
            const float4 hw[7] = {h3, h2, h1, xs[0], xs[1], xs[2], xs[3]};   // x[t-3 .. t+3]
#pragma unroll
            for (int u = 0; u < 4; u++) {
                o[u].x = siluf_(conv4(wr[0], hw[u].x, hw[u + 1].x, hw[u + 2].x, hw[u + 3].x));
                o[u].y = siluf_(conv4(wr[1], hw[u].y, hw[u + 1].y, hw[u + 2].y, hw[u + 3].y));
                o[u].z = siluf_(conv4(wr[2], hw[u].z, hw[u + 1].z, hw[u + 2].z, hw[u + 3].z));
                o[u].w = siluf_(conv4(wr[3], hw[u].w, hw[u + 1].w, hw[u + 2].w, hw[u + 3].w));
            }
            if (norm) {
                float ss[4];
#pragma unroll
                for (int u = 0; u < 4; u++)
                    ss[u] = o[u].x * o[u].x + o[u].y * o[u].y + o[u].z * o[u].z + o[u].w * o[u].w;
#pragma unroll
                for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
                    for (int u = 0; u < 4; u++) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], m);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const float r = rsqrtf(ss[u] + l2_eps) * scale;
                    o[u].x *= r; o[u].y *= r; o[u].z *= r; o[u].w *= r;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; u++) st4(out + (t + u) * C + oc, rnd ? tf32_round(o[u]) : o[u]);
            h3 = xs[1]; h2 = xs[2]; h1 = xs[3];
        }
        cp_async_wait<0>();
    }
    for (; t < t1; t++) {
        if (t >= e) {  // next (non-empty) sequence starts at t
            while (cu[n + 1] <= t) n++;
            s = cu[n];
            e = cu[n + 1];
            h1 = conv_in(x, cs_in, t - 1, s, n, C, c);
            h2 = conv_in(x, cs_in, t - 2, s, n, C, c);
            h3 = conv_in(x, cs_in, t - 3, s, n, C, c);
        }
        const float4 cur = ld4(x + t * C + c);
        float4 o;
        o.x = siluf_(conv4(wr[0], h3.x, h2.x, h1.x, cur.x));
        o.y = siluf_(conv4(wr[1], h3.y, h2.y, h1.y, cur.y));
        o.z = siluf_(conv4(wr[2], h3.z, h2.z, h1.z, cur.z));
        o.w = siluf_(conv4(wr[3], h3.w, h2.w, h1.w, cur.w));
        if (norm) {
            float ss = warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
            float r = rsqrtf(ss + l2_eps) * scale;
            o.x *= r; o.y *= r; o.z *= r; o.w *= r;
        }
        st4(out + t * C + oc, rnd ? tf32_round(o) : o);
        h3 = h2; h2 = h1; h1 = cur;
    }
}

// conv_state_out[n, c, m] = input at position end-3+m (from the cache when the
// sequence is shorter than 3).  Reads all three before writing (alias-safe).
template <class T>
__global__ void conv_state_kernel(const T* __restrict__ x, const T* cs_in,
                                  const int32_t* __restrict__ cu, int N, int C, T* cs_out) {
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)N * C) return;
    int n = (int)(idx / C), c = (int)(idx % C);
    int64_t s = cu[n], e = cu[n + 1];
    float v[kConvK - 1];
#pragma unroll
    for (int m = 0; m < kConvK - 1; m++) {
        int64_t p = e - (kConvK - 1) + m;
        if (p >= s) v[m] = to_f(x[p * C + c]);
        else {
            int64_t mm = (kConvK - 1) + (p - s);
            v[m] = (cs_in != nullptr && mm >= 0) ? to_f(cs_in[idx * (kConvK - 1) + mm]) : 0.f;
        }
    }
#pragma unroll
    for (int m = 0; m < kConvK - 1; m++) cs_out[idx * (kConvK - 1) + m] = from_f<T>(v[m]);
}

// ------------------------------------------------------------------ backward

// Gradient at the conv output pre-activation of token t (backward through SiLU
// and, for q / k channels, the L2 norm and the q scale), given the conv inputs
// a0 = x[t], a1 = x[t-1], a2 = x[t-2], a3 = x[t-3] and the incoming gradient g4.
__device__ __forceinline__ float4 conv_dpre_w(float4 a0, float4 a1, float4 a2, float4 a3,
                                              float4 g4, const float (&w)[4][kConvK], bool norm,
                                              float scale, float l2_eps) {
    float p[4] = {conv4(w[0], a3.x, a2.x, a1.x, a0.x), conv4(w[1], a3.y, a2.y, a1.y, a0.y),
                  conv4(w[2], a3.z, a2.z, a1.z, a0.z), conv4(w[3], a3.w, a2.w, a1.w, a0.w)};
    float gd[4] = {g4.x, g4.y, g4.z, g4.w};
    float xc[4], sg[4];
#pragma unroll
    for (int i = 0; i < 4; i++) { sg[i] = sigmoidf_(p[i]); xc[i] = p[i] * sg[i]; }
    if (norm) {
        // with u = xc r, r = (|xc|^2 + eps)^-1/2 and du = scale g:
        //   d xc = r (du - u (u . du)),  u . du = r scale (xc . g),
        // so |xc|^2 and xc . g come from one (two-value) warp reduction
        float ss = xc[0] * xc[0] + xc[1] * xc[1] + xc[2] * xc[2] + xc[3] * xc[3];
        float xg = xc[0] * gd[0] + xc[1] * gd[1] + xc[2] * gd[2] + xc[3] * gd[3];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, m);
            xg += __shfl_xor_sync(0xffffffffu, xg, m);
        }
        const float r = rsqrtf(ss + l2_eps);
        const float rs = r * scale, c = r * r * xg;
#pragma unroll
        for (int i = 0; i < 4; i++) gd[i] = rs * (gd[i] - xc[i] * c);
    }
    float4 o;
    o.x = gd[0] * sg[0] * (1.f + p[0] * (1.f - sg[0]));
    o.y = gd[1] * sg[1] * (1.f + p[1] * (1.f - sg[1]));
    o.z = gd[2] * sg[2] * (1.f + p[2] * (1.f - sg[2]));
    o.w = gd[3] * sg[3] * (1.f + p[3] * (1.f - sg[3]));
    return o;
}

// dpre at token t for this lane's 4 channels (x channel c, qkv channel oc):
// recompute conv + SiLU (+ L2) and chain the incoming gradient dqkv through L2
// and SiLU.
template <class T>
__device__ __forceinline__ float4 conv_dpre(const T* x, const T* cs, const float* dq, int64_t t,
                                            int64_t s, int n, int C, int c, int oc,
                                            const float (&w)[4][kConvK], bool norm, float scale,
                                            float l2_eps) {
    return conv_dpre_w(ld4(x + t * C + c), conv_in(x, cs, t - 1, s, n, C, c),
                       conv_in(x, cs, t - 2, s, n, C, c), conv_in(x, cs, t - 3, s, n, C, c),
                       ld4(dq + t * C + oc), w, norm, scale, l2_eps);
}

__device__ __forceinline__ float f4(const float4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Gradient of the conv cache of sequence n (length L), written at its first
// token: cache position m (input s - 3 + m) feeds tokens s .. s + 2 - m through
// taps 0 .. 2 - m, and, for a sequence shorter than 3, conv_state_out copies
// cache positions L .. 2, so their share of dcso comes back here too.
__device__ __forceinline__ void conv_cache_grad(float* dcs, const float* dcso, int n, int C, int c,
                                                int64_t L, const float (&wr)[4][kConvK],
                                                float4 d0, float4 d1, float4 d2) {
#pragma unroll
    for (int ch = 0; ch < 4; ch++) {
        float* o3 = dcs + ((int64_t)n * C + c + ch) * (kConvK - 1);
        float g[3] = {wr[ch][0] * f4(d0, ch),
                      wr[ch][0] * f4(d1, ch) + wr[ch][1] * f4(d0, ch),
                      wr[ch][0] * f4(d2, ch) + wr[ch][1] * f4(d1, ch) + wr[ch][2] * f4(d0, ch)};
        if (dcso != nullptr)
            for (int j = (int)L; j < kConvK - 1; j++)
                g[j] += dcso[((int64_t)n * C + c + ch) * (kConvK - 1) + j - L];
        o3[0] = g[0];
        o3[1] = g[1];
        o3[2] = g[2];
    }
}

// The conv-cache gradient before the backward kernel writes it: zero, except
// for an empty sequence, whose conv_state_out is its conv_state_in.
__global__ void conv_cache_grad_init_kernel(const int32_t* __restrict__ cu, int N, int C,
                                            const float* __restrict__ dcso, float* __restrict__ dcs) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)N * C) return;
    const int n = (int)(idx / C);
    const bool empty = cu[n + 1] == cu[n];
#pragma unroll
    for (int m = 0; m < kConvK - 1; m++)
        dcs[idx * (kConvK - 1) + m] = empty && dcso != nullptr ? dcso[idx * (kConvK - 1) + m] : 0.f;
}

// One warp per run of tokens (walked backwards), lane = 4 channels.
// dx[t] = sum_j w[j] dpre[t+3-j] within the sequence; dw partials per CTA
// (fixed-order sum over the CTA's warps) go to wpart[blockIdx.x][c][j].
template <class T>
__global__ void __launch_bounds__(kConvWarps * 32, 2)
conv_bwd_kernel(const T* __restrict__ x, const float* __restrict__ w, const T* cs_in,
                const float* __restrict__ dqkv, const int32_t* __restrict__ cu, int N,
                int64_t Ttot, int C, int hk, int G, bool group_major, float l2_eps,
                float q_scale, T* __restrict__ dx, float* __restrict__ wpart, float* dcs,
                const float* __restrict__ dcso) {
    extern __shared__ __align__(16) unsigned char conv_smem[];
    constexpr int kThr = kConvWarps * 32;
    float4* dq_ring = reinterpret_cast<float4*>(conv_smem);                   // [ring][4][kThr]
    constexpr int kConvRing = conv_ring<T>();
    T* x_ring = reinterpret_cast<T*>(conv_smem + kConvRing * 4 * kThr * sizeof(float4));   // [ring][4][kThr][4]
    auto red = reinterpret_cast<float (*)[kD][kConvK]>(conv_smem);            // [warp][kD][kConvK]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int grp = blockIdx.y;
    const int c = grp * kD + lane * 4;   // channel of x, conv_w, dx, the cache
    const ConvBlock cb = conv_block(grp, hk, G, group_major);
    const int oc = cb.out * kD + lane * 4;   // channel of dqkv
    const bool norm = cb.role < 2;
    const float scale = cb.role == 0 ? q_scale : 1.f;
    float wr[4][kConvK];
#pragma unroll
    for (int ch = 0; ch < 4; ch++)
#pragma unroll
        for (int j = 0; j < kConvK; j++) wr[ch][j] = w[(c + ch) * kConvK + j];
    float dw[4][kConvK];
#pragma unroll
    for (int ch = 0; ch < 4; ch++)
#pragma unroll
        for (int j = 0; j < kConvK; j++) dw[ch][j] = 0.f;

    const int64_t t0 = ((int64_t)blockIdx.x * kConvWarps + warp) * kConvRun;
    if (t0 < Ttot) {
        const int64_t t1 = min(t0 + (int64_t)kConvRun, Ttot);
        int n = seq_of(cu, N, t1 - 1);
        int64_t s = cu[n], e = cu[n + 1];
        const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
        // window of dpre at t+1, t+2, t+3 (zero past the sequence end)
        float4 d1 = (t1 < e) ? conv_dpre(x, cs_in, dqkv, t1, s, n, C, c, oc, wr, norm, scale, l2_eps) : z4;
        float4 d2 = (t1 + 1 < e) ? conv_dpre(x, cs_in, dqkv, t1 + 1, s, n, C, c, oc, wr, norm, scale, l2_eps) : z4;
        float4 d3 = (t1 + 2 < e) ? conv_dpre(x, cs_in, dqkv, t1 + 2, s, n, C, c, oc, wr, norm, scale, l2_eps) : z4;
        if (s <= t0 && (t1 - t0) % 4 == 0) {
            // the whole run lies in one sequence: four tokens per step, whose
            // dpre chains are independent.  Step i covers tokens tb..tb-3
            // (tb = t1-1-4i) and the inputs xr[k] = x[tb - 6 + k]: xr[4..6]
            // carried from the step before, xr[0..3] new.  Each lane copies its
            // own gradient rows and new input rows kConvRing-1 steps ahead into
            // its ring slots (cp.async), so loads stay in flight while it
            // computes; rows before the sequence start come from the cache.
            const int nsteps = (int)((t1 - t0) / 4);
            const int tid = threadIdx.x;
            auto issue = [&](int i) {
                if (i < nsteps) {
                    const int slot = i % kConvRing;
                    const int64_t tb = t1 - 1 - 4 * (int64_t)i;
#pragma unroll
                    for (int u = 0; u < 4; u++)
                        cp_async16(&dq_ring[(slot * 4 + u) * kThr + tid], dqkv + (tb - u) * C + oc, true);
#pragma unroll
                    for (int k = 0; k < 4; k++)
                        if (tb - 6 + k >= s)
                            cp_async_row4(&x_ring[((slot * 4 + k) * kThr + tid) * 4], x + (tb - 6 + k) * C + c);
                }
                cp_async_commit();
            };
            float4 xr[7];
#pragma unroll
            for (int k = 4; k < 7; k++) xr[k] = ld4(x + (t1 - 7 + k) * C + c);
#pragma unroll
            for (int i = 0; i < kConvRing - 1; i++) issue(i);
            for (int i = 0; i < nsteps; i++) {
                const int64_t tb = t1 - 1 - 4 * (int64_t)i;
                issue(i + kConvRing - 1);   // the slot step i-1 used
                cp_async_wait<kConvRing - 1>();
                const int slot = i % kConvRing;
                float4 gq[4], dd[4];
#pragma unroll
                for (int u = 0; u < 4; u++) gq[u] = dq_ring[(slot * 4 + u) * kThr + tid];
#pragma unroll
                for (int k = 0; k < 4; k++)
                    xr[k] = (tb - 6 + k >= s) ? ld4(&x_ring[((slot * 4 + k) * kThr + tid) * 4])
                                              : conv_in(x, cs_in, tb - 6 + k, s, n, C, c);
#pragma unroll
                for (int u = 0; u < 4; u++)
                    dd[u] = conv_dpre_w(xr[6 - u], xr[5 - u], xr[4 - u], xr[3 - u], gq[u], wr, norm,
                                        scale, l2_eps);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const int64_t t = tb - u;
                    const float4 d0 = dd[u];
                    float4 o;
                    o.x = wr[0][3] * d0.x + wr[0][2] * d1.x + wr[0][1] * d2.x + wr[0][0] * d3.x;
                    o.y = wr[1][3] * d0.y + wr[1][2] * d1.y + wr[1][1] * d2.y + wr[1][0] * d3.y;
                    o.z = wr[2][3] * d0.z + wr[2][2] * d1.z + wr[2][1] * d2.z + wr[2][0] * d3.z;
                    o.w = wr[3][3] * d0.w + wr[3][2] * d1.w + wr[3][1] * d2.w + wr[3][0] * d3.w;
                    add_state_out_grad(o, dcso, n, C, c, t, e);
                    st4(dx + t * C + c, o);
#pragma unroll
                    for (int j = 0; j < kConvK; j++)
#pragma unroll
                        for (int ch = 0; ch < 4; ch++) dw[ch][j] += f4(d0, ch) * f4(xr[3 - u + j], ch);
                    if (t == s && dcs != nullptr) conv_cache_grad(dcs, dcso, n, C, c, e - s, wr, d0, d1, d2);
                    d3 = d2; d2 = d1; d1 = d0;
                }
                xr[4] = xr[0]; xr[5] = xr[1]; xr[6] = xr[2];
            }
            cp_async_wait<0>();
        } else {
            // walking backwards: a register window holds x[t], x[t-1], x[t-2], x[t-3];
            // each step loads one new x row and the next dq row ahead of use
            float4 xw0 = conv_in(x, cs_in, t1 - 1, s, n, C, c);
            float4 xw1 = conv_in(x, cs_in, t1 - 2, s, n, C, c);
            float4 xw2 = conv_in(x, cs_in, t1 - 3, s, n, C, c);
            float4 xw3 = conv_in(x, cs_in, t1 - 4, s, n, C, c);
            float4 g = ld4(dqkv + (t1 - 1) * C + oc);
            for (int64_t t = t1 - 1; t >= t0; t--) {
                if (t < s) {  // crossed into the previous (non-empty) sequence
                    while (cu[n] > t) n--;
                    s = cu[n];
                    e = cu[n + 1];
                    d1 = d2 = d3 = z4;
                    xw0 = conv_in(x, cs_in, t, s, n, C, c);
                    xw1 = conv_in(x, cs_in, t - 1, s, n, C, c);
                    xw2 = conv_in(x, cs_in, t - 2, s, n, C, c);
                    xw3 = conv_in(x, cs_in, t - 3, s, n, C, c);
                }
                const float4 xn = conv_in(x, cs_in, t - 4, s, n, C, c);   // for step t - 1
                const float4 gn = t > t0 ? ld4(dqkv + (t - 1) * C + oc) : z4;
                const float4 d0 = conv_dpre_w(xw0, xw1, xw2, xw3, g, wr, norm, scale, l2_eps);
                float4 o;
                o.x = wr[0][3] * d0.x + wr[0][2] * d1.x + wr[0][1] * d2.x + wr[0][0] * d3.x;
                o.y = wr[1][3] * d0.y + wr[1][2] * d1.y + wr[1][1] * d2.y + wr[1][0] * d3.y;
                o.z = wr[2][3] * d0.z + wr[2][2] * d1.z + wr[2][1] * d2.z + wr[2][0] * d3.z;
                o.w = wr[3][3] * d0.w + wr[3][2] * d1.w + wr[3][1] * d2.w + wr[3][0] * d3.w;
                add_state_out_grad(o, dcso, n, C, c, t, e);
                st4(dx + t * C + c, o);
                const float4 xin[kConvK] = {xw3, xw2, xw1, xw0};   // x[t - 3 + j]
    #pragma unroll
                for (int j = 0; j < kConvK; j++)
    #pragma unroll
                    for (int ch = 0; ch < 4; ch++) dw[ch][j] += f4(d0, ch) * f4(xin[j], ch);
                if (t == s && dcs != nullptr) conv_cache_grad(dcs, dcso, n, C, c, e - s, wr, d0, d1, d2);
                d3 = d2; d2 = d1; d1 = d0;
                xw0 = xw1; xw1 = xw2; xw2 = xw3; xw3 = xn;
                g = gn;
            }
        }
    }
    __syncthreads();   // every warp is done with its ring
#pragma unroll
    for (int ch = 0; ch < 4; ch++)
#pragma unroll
        for (int j = 0; j < kConvK; j++) red[warp][lane * 4 + ch][j] = dw[ch][j];
    __syncthreads();
    for (int i = threadIdx.x; i < kD * kConvK; i += blockDim.x) {
        float acc = 0.f;
        for (int wi = 0; wi < kConvWarps; wi++) acc += red[wi][i / kConvK][i % kConvK];
        wpart[((int64_t)blockIdx.x * C + grp * kD) * kConvK + i] = acc;
    }
}

// dconv_w[c, j] = sum over CTA rows of wpart (fixed order).
__global__ void conv_dw_reduce_kernel(const float* __restrict__ wpart, int nparts, int C,
                                      float* __restrict__ dw) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= C * kConvK) return;
    float acc = 0.f;
    for (int p = 0; p < nparts; p++) acc += wpart[(int64_t)p * C * kConvK + i];
    dw[i] = acc;
}

// ------------------------------------------------------------------ launchers
template <class T>
cudaError_t launch_conv_fwd_t(const ConvArgs& a, cudaStream_t st) {
    if (a.T > 0) {
        dim3 grid((unsigned)((a.T + kConvWarps * kConvRun - 1) / (kConvWarps * kConvRun)),
                  (unsigned)(a.C / kD));
        const cudaError_t e = smem_attr(conv_fwd_kernel<T>, conv_fwd_smem<T>());
        if (e != cudaSuccess) return e;
        GDN_PROF("conv_fwd", st);
        conv_fwd_kernel<T><<<grid, kConvWarps * 32, conv_fwd_smem<T>(), st>>>(
            (const T*)a.x, a.w, (const T*)a.cs_in, a.cu, a.N, a.T, a.C, a.hk, a.hv / a.hk,
            a.group_major, a.l2_eps, a.q_scale, a.round_tf32, a.qkv);
    }
    if (a.cs_out != nullptr && a.N > 0) {
        int64_t n = (int64_t)a.N * a.C;
        GDN_PROF("conv_state", st);
        conv_state_kernel<T><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
            (const T*)a.x, (const T*)a.cs_in, a.cu, a.N, a.C, (T*)a.cs_out);
    }
    return cudaGetLastError();
}

cudaError_t launch_conv_fwd(const ConvArgs& a, cudaStream_t st) {
    return a.bf16 ? launch_conv_fwd_t<__nv_bfloat16>(a, st) : launch_conv_fwd_t<float>(a, st);
}

int conv_bwd_parts(int64_t T) {
    return (int)((T + kConvWarps * kConvRun - 1) / (kConvWarps * kConvRun));
}

template <class T>
cudaError_t launch_conv_bwd_t(const ConvArgs& a, cudaStream_t st) {
    int parts = conv_bwd_parts(a.T);
    if (a.dcs != nullptr && a.N > 0) {
        const int64_t n = (int64_t)a.N * a.C;
        GDN_PROF("conv_cache_grad_init", st);
        conv_cache_grad_init_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(a.cu, a.N, a.C,
                                                                                 a.dcs_out, a.dcs);
    }
    if (parts > 0) {
        dim3 grid((unsigned)parts, (unsigned)(a.C / kD));
        static_assert(conv_bwd_smem<float>() >= sizeof(float) * kConvWarps * kD * kConvK &&
                          conv_bwd_smem<__nv_bfloat16>() >= sizeof(float) * kConvWarps * kD * kConvK,
                      "the ring holds the dw reduction");
        const cudaError_t e = smem_attr(conv_bwd_kernel<T>, conv_bwd_smem<T>());
        if (e != cudaSuccess) return e;
        {
            GDN_PROF("conv_bwd", st);
            conv_bwd_kernel<T><<<grid, kConvWarps * 32, conv_bwd_smem<T>(), st>>>(
                (const T*)a.x, a.w, (const T*)a.cs_in, a.dqkv, a.cu, a.N, a.T, a.C, a.hk,
                a.hv / a.hk, a.group_major, a.l2_eps, a.q_scale, (T*)a.dx, a.wpart, a.dcs,
                a.dcs_out);
        }
        {
            GDN_PROF("conv_dw_reduce", st);
            conv_dw_reduce_kernel<<<(a.C * kConvK + 255) / 256, 256, 0, st>>>(a.wpart, parts,
                                                                              a.C, a.dw);
        }
    } else {
        cudaMemsetAsync(a.dw, 0, sizeof(float) * (size_t)a.C * kConvK, st);
    }
    return cudaGetLastError();
}

cudaError_t launch_conv_bwd(const ConvArgs& a, cudaStream_t st) {
    return a.bf16 ? launch_conv_bwd_t<__nv_bfloat16>(a, st) : launch_conv_bwd_t<float>(a, st);
}

}  // namespace gdn
