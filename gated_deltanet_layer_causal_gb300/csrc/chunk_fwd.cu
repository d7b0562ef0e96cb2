// Forward of the gated delta rule in the chunked WY form (chunk 64), with the
// gates, grouped value heads and the fused zero-centred gated RMSNorm.
//
// Per chunk (tokens i = 0..L-1, in-chunk cumulative gate gam_i):
//   A_ij = beta_i exp(gam_i - gam_j) k_i.k_j (j < i);  T = (I + A)^-1
//   W = T diag(beta e^gam) K ;  U~ = T diag(beta) V          (prep, parallel)
//   U = U~ - W S0^T ;  S_end = e^{gam_L} S0 + U^T diag(e^{gam_L-gam}) K
//                                                            (state, sequential)
//   O = diag(e^gam) Q S0^T + (Q K^T (.) exp(gam_i-gam_j) (.) [i>=j]) U
//   y = O rsqrt(mean(O^2)+eps) (1+w) gate(z)                 (out, parallel)
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
#include "umma.cuh"

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

// ------------------------------------------------------------------ gates
// grid (NT, ceil(Hv / 8)), 256 threads: one warp per (chunk, v-head), two tokens
// per lane.  g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b); gam = the
// in-chunk inclusive cumsum of g (a warp scan), stored head-major with beta.
template <class IO>
__global__ void __launch_bounds__(256)
gates_kernel(const IO* __restrict__ av, const IO* __restrict__ bv, const float* __restrict__ A_log,
             const float* __restrict__ dt_bias, int hv, FwdSaved sv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * 8 + warp;
    const ChunkInfo ci = sv.chunks[blockIdx.x];
    if (h >= hv || ci.len == 0) return;
    const int L = ci.len;
    const float Aexp = expf(A_log[h]), db = dt_bias[h];
    float g[2], b[2];
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int j = 2 * lane + e;
        g[e] = b[e] = 0.f;
        if (j < L) {
            const int64_t t = ci.start + j;
            g[e] = -Aexp * softplusf_(to_f(av[t * hv + h]) + db);
            b[e] = sigmoidf_(to_f(bv[t * hv + h]));
        }
    }
    float s = g[0] + g[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += u;
    }
    const float ex = s - (g[0] + g[1]);
    const float gam[2] = {ex + g[0], ex + g[0] + g[1]};
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int j = 2 * lane + e;
        if (j < L) {
            sv.gam[(int64_t)h * sv.T + ci.start + j] = gam[e];
            sv.beta[(int64_t)h * sv.T + ci.start + j] = b[e];
        }
    }
}

// ------------------------------------------------------------------ prep
// Persistent: one CTA per SM walks the (chunk, head) tiles t = blockIdx.x,
// + gridDim.x, ... (chunk = t % NT, head = t / NT).  Per tile, tcgen05, with
// the gates from gates_kernel:
//   D1 = K K^T (64 x 64)  ->  A = beta_i e^{gam_i-gam_j} D1 (j < i)
//   T  = (I + A)^-1        (forward substitution on the CUDA cores; saved)
//   W = (T diag(beta e^gam)) K,  U~ = (T diag(beta)) V      (M=64, N=128, K=64 each)
// K arrives twice through the TMA, as a K-major tile for K K^T and as an
// MN-major tile for W (contracted over tokens), V once, MN-major; the gate
// scalings go into the two A tiles, so no tile is transposed.  W and U~ are
// staged over the A / T scratch, so the next tile's K and V are requested as
// soon as the second products are done; its chunk entry and gates are loaded
// into registers meanwhile.  Tensor memory allocated once.
constexpr int kLdK = 132, kLdA = 68;
constexpr int kPrepFloats = 3 * 64 * 128 + 2 * 64 * kLdA + 2 * 64 * 64;
constexpr size_t kPrepSmem = sizeof(float) * (kPrepFloats + 3 * 64 + 16) + 64 + 1024;

__global__ void __launch_bounds__(256, 1)
prep_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, int NT, FwdSaved sv) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* Ks = sm;                    // [64][128] swizzled K-major K
    float* Km = Ks + 64 * 128;         // [64 (j)][128 (c)] MN-major K
    float* Vm = Km + 64 * 128;         // [64 (j)][128 (a)] MN-major V
    float* As = Vm + 64 * 128;         // [64][kLdA] row-major A
    float* Tr = As + 64 * kLdA;        // [64][kLdA] row-major T
    float* Tk = Tr + 64 * kLdA;        // [64][64] K-major T diag(beta e^gam)
    float* Tv = Tk + 64 * 64;          // [64][64] K-major T diag(beta)
    float* Wst = As;                   // [64][128] swizzled W, over A and T (1 KB-aligned)
    float* Ust = Tk;                   // [64][128] swizzled U~, over Tk and Tv (1 KB-aligned)
    float* gam = Tv + 64 * 64;
    float* bet = gam + 64;
    float* be = bet + 64;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(be + 64 + 16);   // MMA
    uint64_t* mA = mbar + 1;           // K, K (MN-major), V
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mA + 1);
    static_assert(2 * 64 * kLdA >= 64 * 128 && (3 * 64 * 128 * 4) % 1024 == 0 &&
                      ((3 * 64 * 128 + 2 * 64 * kLdA) * 4) % 1024 == 0,
                  "staging tiles fit the A / T scratch and are 1 KB-aligned");
    const int tid = threadIdx.x, warp = tid >> 5;
    const int ntiles = NT * hv;
    int t = blockIdx.x;
    if (t >= ntiles) return;
    ChunkInfo ci = sv.chunks[t % NT];
    if (ci.len == 0) return;   // the device check of cu_seqlens failed: every chunk is empty
    auto issue = [&](const ChunkInfo& c, int tile) {   // one thread
        const int h = tile / NT, kh = h / (hv / hk);
        umma::mbar_expect_tx(mA, 3 * 64 * 128 * 4);
        umma::tma_rows(Ks, 64, &maps.k, kh, c.start, mA);
        umma::tma_rows(Km, 64, &maps.k_mn, kh, c.start, mA);
        umma::tma_rows(Vm, 64, &maps.v_mn, h, c.start, mA);
    };
    // padding rows continue the last gam (g = 0), beta = 0
    auto gates_of = [&](const ChunkInfo& c, int tile, float& gm, float& bt) {
        const int h = tile / NT;
        gm = tid < 64 ? sv.gam[(int64_t)h * sv.T + c.start + min(tid, c.len - 1)] : 0.f;
        bt = tid < c.len ? sv.beta[(int64_t)h * sv.T + c.start + tid] : 0.f;
    };
    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::mbar_init(mA, 1);
        issue(ci, t);
    }
    float g_cur = 0.f, b_cur = 0.f;
    gates_of(ci, t, g_cur, b_cur);
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tD1 = tmem, tD2 = tmem + 256;
    const int half = warp >> 2;
    bool ok = true;
    for (int it = 0;; it++) {
        const int h = t / NT, L = ci.len;
        const int tn = t + (int)gridDim.x;
        const ChunkInfo cn = tn < ntiles ? sv.chunks[tn % NT] : ci;
        if (tid < 64) {
            gam[tid] = g_cur;
            bet[tid] = b_cur;
            be[tid] = b_cur * expf(g_cur);
        }
        if (tid == 0) umma::bulk_wait_read();   // the last tile's stores have read W / U~
        ok = __syncthreads_and(umma::mbar_wait(mA, it & 1));   // K, V; gates visible
        if (!ok) break;
        if (L < 64) {   // tail rows belong to the next sequence
            umma::zero_tail_rows(Ks, 64, 0, L);
            umma::zero_tail_rows(Km, 64, 0, L);
            umma::zero_tail_rows(Vm, 64, 0, L);
            __syncthreads();
        }
        if (!sv.qkv_tf32) umma::tf32r_inplace(Ks, 3 * 64 * 128);   // K (both layouts), V
        umma::fence_smem_to_async();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tD1, umma::swt(Ks, 64), umma::swt(Ks, 64), 64, 64, 128, false);
            umma::commit(mbar);
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 0));
        umma::fence_after_sync();
        if (!ok) break;
        {   // A = beta_i e^{gam_i - gam_j} D1 (j < i); 32 columns per warp, all lanes
            float v[16];
            umma::tmem_ld_m64<4>(umma::tmem_at(tD1, half * 32), v);
            const int rl = umma::frag_row_lo(), cf = umma::frag_col();
#pragma unroll
            for (int hr = 0; hr < 2; hr++) {
                const int r = rl + 8 * hr;
                const float br = bet[r], gr = gam[r];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int j = half * 32 + 8 * k + cf;
                    *reinterpret_cast<float2*>(As + r * kLdA + j) = make_float2(
                        j < r ? br * expf(gr - gam[j]) * v[4 * k + 2 * hr] : 0.f,
                        j + 1 < r ? br * expf(gr - gam[j + 1]) * v[4 * k + 2 * hr + 1] : 0.f);
                }
            }
        }
        __syncthreads();
        const bool next = tn < ntiles && cn.len > 0;   // the entry has arrived by now
        float g_next = 0.f, b_next = 0.f;
        if (next) gates_of(cn, tn, g_next, b_next);
        tril_inverse64(As, kLdA, Tr, kLdA, Tk);   // Tk doubles as scratch
        __syncthreads();
        for (int idx = tid; idx < 64 * 16; idx += 256) {   // T diag(.) -> K-major rows i
            const int r = idx >> 4, c = (idx & 15) * 4;
            const float4 t4 = *reinterpret_cast<const float4*>(Tr + r * kLdA + c);
            *reinterpret_cast<float4*>(Tk + umma::kidx(r, c, 64)) = umma::tf32r(
                make_float4(t4.x * be[c], t4.y * be[c + 1], t4.z * be[c + 2], t4.w * be[c + 3]));
            *reinterpret_cast<float4*>(Tv + umma::kidx(r, c, 64)) = umma::tf32r(
                make_float4(t4.x * bet[c], t4.y * bet[c + 1], t4.z * bet[c + 2], t4.w * bet[c + 3]));
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tD2, umma::kmaj(Tk, 64), umma::mnt(Km), 64, 128, 64, false);
            umma::mma(tD2 + 128, umma::kmaj(Tv, 64), umma::mnt(Vm), 64, 128, 64, false);
            umma::commit(mbar);
        }
        {   // T for the backward, as K-major rows i and as K-major rows j (T^T), rounded
            float* Tg = sv.Tm + ((int64_t)(t % NT) * hv + h) * 2 * 64 * 64;
            for (int idx = tid; idx < 64 * 16; idx += 256) {
                const int r = idx & 63, c4 = idx >> 6;
                st4(Tg + umma::kidx(r, 4 * c4, 64),
                    umma::tf32r(*reinterpret_cast<const float4*>(Tr + r * kLdA + 4 * c4)));
                st4(Tg + 64 * 64 + umma::kidx(r, 4 * c4, 64),
                    umma::tf32r(make_float4(Tr[(4 * c4) * kLdA + r], Tr[(4 * c4 + 1) * kLdA + r],
                                            Tr[(4 * c4 + 2) * kLdA + r], Tr[(4 * c4 + 3) * kLdA + r])));
            }
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 1));
        umma::fence_after_sync();
        if (!ok) break;
        if (next && tid == 0) issue(cn, tn);   // K, K (MN-major) and V consumed
        // warp half 0 -> W (columns 0..127), half 1 -> U~ (128..255), staged as
        // swizzled tiles over the A / T scratch and stored whole
        {
            float* Sw = half == 0 ? Wst : Ust;
            float v[32];
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 64) {
                umma::tmem_ld64_m64(umma::tmem_at(tD2, half * 128 + c0), v);
                if (half == 0)   // W is only ever a tensor-core operand: stored rounded
#pragma unroll
                    for (int k = 0; k < 32; k++) v[k] = umma::tf32r(v[k]);
                umma::frag_to_sw(Sw, v, c0, 1.f, 1.f);
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        if (L == 64) {
            if (tid == 0) {
                umma::tma_store_rows(&maps.W, h, ci.start, Wst);
                umma::tma_store_rows(&maps.U, h, ci.start, Ust);
                umma::bulk_commit();
            }
        } else {
            const int64_t off = ((int64_t)ci.start * hv + h) * kD;
            umma::store_rows_sw(sv.W + off, (int64_t)hv * kD, Wst, L);
            umma::store_rows_sw(sv.U + off, (int64_t)hv * kD, Ust, L);
            __syncthreads();
        }
        if (!next) break;
        g_cur = g_next;
        b_cur = b_next;
        ci = cn;
        t = tn;
    }
    if (tid == 0) umma::bulk_wait_read();
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 512);
    if (!ok && tid == 0) atomicExch(sv.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ state pass
// grid (3, Hv, N), 256 threads, one CTA per SM.  Rows a of S evolve
// independently (k, beta, g are shared by all rows), so each CTA carries a
// slice of rows of the fp32 state -- kept transposed, S^T[b][a], in the MMA
// accumulators -- through all chunks of its sequence: rows 0-47, 48-95 and
// 96-127, so that 3 * Hv CTAs occupy most SMs.  The next chunk's W, K and U~
// slice arrive through the TMA into the other half of a double buffer while
// the current chunk is computed.  A tf32-rounded copy of the state slice, St,
// is held in exactly the layout of its slice of the chunk-start state tile
// (K-major rows a): it feeds the tensor cores without conversion and leaves as
// one bulk copy per chunk.
constexpr int kSliceMax = 48;
struct StateStage {                // one chunk's operands (a multiple of 1 KB)
    float W[64 * 128];             // swizzled, arrives rounded
    float K[64 * 128];             // swizzled
    float U[64 * 64];              // U~ columns a0 .. a0 + 63: two swizzled 64 x 32 boxes
    float gam[256];                // 64 used
};
constexpr int kStageFloats = (int)(sizeof(StateStage) / sizeof(float));
static_assert(sizeof(StateStage) % 1024 == 0, "stage alignment");
constexpr size_t kStateSmem =
    sizeof(float) * (2 * kStageFloats + kSliceMax * kD + kSliceMax * 64 + 64 * 8) + 2 * 8 +
    1024;

template <int SW>
__device__ __forceinline__ void state_fwd_slice(const TileMaps& maps, int hk, int hv, int a0,
                                                const float* S_init, float* S_final,
                                                const FwdSaved& sv, float* sm) {
    StateStage* stage = reinterpret_cast<StateStage*>(sm);
    float* St = sm + 2 * kStageFloats;      // [SW (a)][128 (b)] K-major, rounded
    float* Ub = St + kSliceMax * kD;        // [SW (a)][64 (i)] K-major: fk_i U[i][a], rounded
    // (the ldmatrix pair loads of an odd n-block count read up to 8 rows past St
    // and Ub: the padding keeps them inside shared memory)
    uint64_t* mb = reinterpret_cast<uint64_t*>(Ub + kSliceMax * 64 + 64 * 8);   // [2]
    const int h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
    const int kh = h / (hv / hk);
    constexpr int NB = (SW + 31) / 32;      // U~ boxes of 32 columns
    using TS = Tile<kD, SW, 8>;    // S^T: rows b (d_k), cols a (slice)
    using TU = Tile<64, SW, 8>;
    typename TS::Acc sacc;
    const int64_t sbase = ((int64_t)n * hv + h) * kD * kD;
    if (tid == 0) {
        umma::mbar_init(&mb[0], 1);
        umma::mbar_init(&mb[1], 1);
    }
    tile_each2<kD, SW, 8>(sacc, [&](int b, int a, float& v0, float& v1) {
        v0 = S_init ? S_init[sbase + (int64_t)(a0 + a) * kD + b] : 0.f;
        v1 = S_init ? S_init[sbase + (int64_t)(a0 + a + 1) * kD + b] : 0.f;
        St[umma::kidx(a, b, kD)] = umma::tf32r(v0);
        St[umma::kidx(a + 1, b, kD)] = umma::tf32r(v1);
    });
    umma::fence_smem_to_async();
    __syncthreads();   // barriers initialised, St written
    const int c0 = sv.seq_chunk[n], c1 = sv.seq_chunk[n + 1];
    auto issue = [&](int s, const ChunkInfo& info) {   // tiles: one thread; gates: 64
        if (tid == 0) {
            umma::mbar_expect_tx(&mb[s], (2 * 64 * 128 + NB * 64 * 32) * 4);
            umma::tma_rows(stage[s].W, 64, &maps.W, h, info.start, &mb[s]);
            umma::tma_rows(stage[s].K, 64, &maps.k, kh, info.start, &mb[s]);
#pragma unroll
            for (int bx = 0; bx < NB; bx++)
                umma::tma_box(stage[s].U + bx * 64 * 32, &maps.U, a0 + 32 * bx, h, info.start,
                              &mb[s]);
        }
        if (tid < 64)   // gate rows start at any token: 4-byte copies
            cp_async4(stage[s].gam + tid,
                      sv.gam + (int64_t)h * sv.T + info.start + min(tid, info.len - 1),
                      tid < info.len);
        cp_async_commit();
    };
    if (c0 < c1) issue(0, sv.chunks[c0]);
    bool ok = true;
    const int lane = tid & 31, rg = TU::m0() + (lane >> 2);   // this thread's U rows rg, rg + 8
    for (int ci = c0; ci < c1 && ok; ci++) {
        const int s = (ci - c0) & 1;
        StateStage& cur = stage[s];
        const ChunkInfo info = sv.chunks[ci];
        const int L = info.len;
        if (ci + 1 < c1) {
            issue(s ^ 1, sv.chunks[ci + 1]);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        // chunk-start state in the layout with rows b (exact), from the accumulators
        const int64_t obase = ((int64_t)ci * hv + h) * kD * kD;
        tile_each2<kD, SW, 8>(sacc, [&](int b, int a, float& v0, float& v1) {
            *reinterpret_cast<float2*>(sv.S0b + obase + umma::kidx(b, a0 + a, kD)) =
                make_float2(v0, v1);
        });
        ok = __syncthreads_and(umma::mbar_wait(&mb[s], ((ci - c0) >> 1) & 1));
        if (!ok) break;
        if (tid == 0) {   // ... and with rows a (rounded; an MMA operand only): St whole
            umma::bulk_store(sv.S0 + obase + (int64_t)a0 * kD, St, SW * kD * 4);
            umma::bulk_commit();
        }
        const float gL = cur.gam[L - 1];
        const float f0 = rg < L ? expf(gL - cur.gam[rg]) : 0.f;
        const float f1 = rg + 8 < L ? expf(gL - cur.gam[rg + 8]) : 0.f;
        // U = U~ - W S^T   (64 x slice)
        typename TU::Acc uacc;
        tile_zero<64, SW, 8>(uacc);
        tile_mma_frag<64, SW, kD, 8>(
            uacc,
            [&](int r0, int k0, uint32_t(&f)[4]) {
                ldsm_a(f, r0, k0, [&](int r, int c) { return cur.W + umma::swz(r, c, 64); });
            },
            [&](int k0, int n0, uint32_t(&f)[4]) {
                ldsm_b2(f, k0, n0, [&](int nn, int k) { return St + umma::kidx(nn, k, kD); });
            });
        tile_each2<64, SW, 8>(uacc, [&](int i, int a, float& v0, float& v1) {
            float u0 = 0.f, u1 = 0.f;
            if (i < L) {
                const float2 ut = *reinterpret_cast<const float2*>(cur.U + umma::swz(i, a, 64));
                u0 = ut.x - v0;
                u1 = ut.y - v1;
                // stored rounded: later kernels use U only as a tensor-core operand
                *reinterpret_cast<float2*>(sv.U + ((int64_t)(info.start + i) * hv + h) * kD +
                                           a0 + a) = make_float2(umma::tf32r(u0), umma::tf32r(u1));
            }
            const float f = i == rg ? f0 : f1;
            Ub[umma::kidx(a, i, 64)] = umma::tf32r(f * u0);
            Ub[umma::kidx(a + 1, i, 64)] = umma::tf32r(f * u1);
        });
        __syncthreads();   // Ub complete
        // S^T = e^{gam_L} S^T + K^T (diag(fk) U)
        const float dl = expf(gL);
        tile_each<kD, SW, 8>(sacc, [&](int, int, float& v) { v *= dl; });
        tile_mma_frag<kD, SW, 64, 8>(
            sacc,
            [&](int r0, int k0, uint32_t(&f)[4]) {   // A(b, i) = K[i][b]: element loads
                const int g = lane >> 2, t = lane & 3;
                f[0] = f2tf32(cur.K[umma::swz(k0 + t, r0 + g, 64)]);
                f[1] = f2tf32(cur.K[umma::swz(k0 + t, r0 + g + 8, 64)]);
                f[2] = f2tf32(cur.K[umma::swz(k0 + t + 4, r0 + g, 64)]);
                f[3] = f2tf32(cur.K[umma::swz(k0 + t + 4, r0 + g + 8, 64)]);
            },
            [&](int k0, int n0, uint32_t(&f)[4]) {
                ldsm_b2(f, k0, n0, [&](int nn, int k) { return Ub + umma::kidx(nn, k, 64); });
            });
        if (tid == 0) umma::bulk_wait_read();   // the chunk-start copy has read St
        __syncthreads();   // reads of cur, St and Ub are done
        tile_each2<kD, SW, 8>(sacc, [&](int b, int a, float& v0, float& v1) {
            St[umma::kidx(a, b, kD)] = umma::tf32r(v0);
            St[umma::kidx(a + 1, b, kD)] = umma::tf32r(v1);
        });
        umma::fence_smem_to_async();   // St -> the next chunk's bulk copy
    }
    if (!ok) {
        if (tid == 0) atomicExch(sv.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
        return;
    }
    if (S_final)
        tile_each<kD, SW, 8>(sacc, [&](int b, int a, float& v) {
            S_final[sbase + (int64_t)(a0 + a) * kD + b] = v;
        });
}

__global__ void __launch_bounds__(256, 1)
state_fwd_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, const float* S_init,
                 float* S_final, FwdSaved sv) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    if (blockIdx.x < 2)
        state_fwd_slice<48>(maps, hk, hv, 48 * (int)blockIdx.x, S_init, S_final, sv, sm);
    else
        state_fwd_slice<32>(maps, hk, hv, 96, S_init, S_final, sv, sm);
}

// ------------------------------------------------------------------ output + norm
// Persistent: one CTA per SM walks the (chunk, head) tiles t = blockIdx.x,
// + gridDim.x, ... (chunk = t % NT, head = t / NT).  Per tile, tcgen05:
//   D1 = Q K^T (64 x 64),  D3 = Q S0^T (64 x 128)       -- issued together
//   P  = D1 (.) e^{gam_i - gam_j} (.) [i >= j]          -- staged K-major
//   D2 = P U (64 x 128)
//   O  = D2 + e^{gam_i} D3 ; y = O rsqrt(mean(O^2)+eps) (1+w) gate(z)
// Shared memory: Q, K swizzled 32 KB each and U MN-major 32 KB (TMA; U is the
// B operand of P U, contracted over tokens, so it is read as loaded), S0
// (K-major rows a) 64 KB (one bulk copy), P 16 KB, the z rows 33 KB.  The next
// tile's Q, K and S0 are requested as soon as D1 and D3 are done, its U and z
// rows once this tile's O (staged over U) has been stored; its chunk entry and
// gate values are loaded into registers meanwhile.  Tensor memory: 320 fp32
// columns, allocated once.
constexpr int kOutFloats = 64 * 128 * 2 + 128 * 128 + 64 * 128 + 64 * 64 + 64 * kLdK;
constexpr size_t kOutSmem = sizeof(float) * (kOutFloats + 64 * 2 + 2 * 64 + 16) + 64 + 1024;

template <class IO>
__global__ void __launch_bounds__(256, 1)
out_fwd_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, int NT, const IO* z,
               const float* norm_w, float norm_eps, int gate, IO* o_out, IO* y_out, FwdSaved sv) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* Qs = sm;                    // [64][128] swizzled
    float* Ks = Qs + 64 * 128;         // [64][128] swizzled
    float* Ss = Ks + 64 * 128;         // [128 (a)][128 (b)] K-major
    float* Us = Ss + 128 * 128;        // [64 (j)][128 (a)] MN-major U; then O, swizzled
    float* Ps = Us + 64 * 128;         // [64 (i)][64 (j)] K-major
    char* Zs = reinterpret_cast<char*>(Ps + 64 * 64);   // z rows, kZPitch bytes apart
    float* gam = Ps + 64 * 64 + 64 * kLdK;
    float* eg = gam + 64;
    float* ssq = eg + 64;              // [2][64] partial sums of squares
    uint64_t* mbar = reinterpret_cast<uint64_t*>(ssq + 2 * 64 + 16);   // MMA
    uint64_t* mA = mbar + 1;           // Q, K, S0
    uint64_t* mU = mA + 1;             // U
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mU + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = NT * hv;
    int t = blockIdx.x;
    if (t >= ntiles) return;
    ChunkInfo ci = sv.chunks[t % NT];
    if (ci.len == 0) return;   // the device check of cu_seqlens failed: every chunk is empty
    constexpr int kZPitch = kD * (int)sizeof(IO) + 16;    // bytes; conflict-free row reads
    auto issue_a = [&](const ChunkInfo& c, int tile) {   // one thread
        const int h = tile / NT, kh = h / (hv / hk);
        umma::mbar_expect_tx(mA, 2 * 64 * 128 * 4 + 128 * 128 * 4);
        umma::tma_rows(Qs, 64, &maps.q, kh, c.start, mA);
        umma::tma_rows(Ks, 64, &maps.k, kh, c.start, mA);
        umma::bulk_load(Ss, sv.S0 + ((int64_t)(tile % NT) * hv + h) * kD * kD, 128 * 128 * 4, mA);
    };
    auto issue_u = [&](const ChunkInfo& c, int tile) {   // one thread
        umma::mbar_expect_tx(mU, 64 * 128 * 4);
        umma::tma_rows(Us, 64, &maps.U_mn, tile / NT, c.start, mU);
    };
    auto issue_z = [&](const ChunkInfo& c, int tile) {   // all threads, one cp.async group
        if (z) {
            constexpr int kPieces = kD * (int)sizeof(IO) / 16;
            const int h = tile / NT;
            for (int idx = tid; idx < 64 * kPieces; idx += 256) {
                const int r = idx / kPieces, p = idx % kPieces;
                const int64_t tr = (int64_t)c.start + min(r, c.len - 1);
                cp_async16(Zs + r * kZPitch + p * 16,
                           reinterpret_cast<const char*>(z + (tr * hv + h) * kD) + p * 16, r < c.len);
            }
        }
        cp_async_commit();
    };
    // padding rows continue the last gate value (g = 0)
    auto gam_of = [&](const ChunkInfo& c, int tile) {
        return tid < 64 ? sv.gam[(int64_t)(tile / NT) * sv.T + c.start + min(tid, c.len - 1)] : 0.f;
    };
    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::mbar_init(mA, 1);
        umma::mbar_init(mU, 1);
        issue_a(ci, t);
        issue_u(ci, t);
    }
    issue_z(ci, t);
    float g_cur = gam_of(ci, t);
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tD1 = tmem, tD3 = tmem + 64, tD2 = tmem + 192;
    const int win = warp & 3, half = warp >> 2;
    const int i = win * 16 + lane;     // row held by lanes 0..15 (M = 64 layout)
    const float4 w4 = z ? ld4(norm_w + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    bool ok = true;
    for (int it = 0;; it++) {
        const int h = t / NT, L = ci.len;
        const int tn = t + (int)gridDim.x;
        const ChunkInfo cn = tn < ntiles ? sv.chunks[tn % NT] : ci;
        if (tid < 64) {
            gam[tid] = g_cur;
            eg[tid] = tid < L ? expf(g_cur) : 0.f;
        }
        ok = __syncthreads_and(umma::mbar_wait(mA, it & 1));   // Q, K, S0; gam visible
        if (!ok) break;
        if (L < 64) {   // tail rows belong to the next sequence
            umma::zero_tail_rows(Qs, 64, 0, L);
            umma::zero_tail_rows(Ks, 64, 0, L);
            __syncthreads();
        }
        if (!sv.qkv_tf32) umma::tf32r_inplace(Qs, 64 * 128 * 2);   // Q, K (S0 and U arrive rounded)
        umma::fence_smem_to_async();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tD1, umma::swt(Qs, 64), umma::swt(Ks, 64), 64, 64, 128, false);
            umma::mma(tD3, umma::swt(Qs, 64), umma::kmaj(Ss, 128), 64, 128, 128, false);
            umma::commit(mbar);
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 0));
        umma::fence_after_sync();
        if (!ok) break;
        const bool next = tn < ntiles && cn.len > 0;
        if (next && tid == 0) issue_a(cn, tn);   // Q, K, S0 consumed
        const float g_next = next ? gam_of(cn, tn) : 0.f;
        {   // P = D1 (.) Gam (.) M  -> K-major rows i; 32 columns per warp, all lanes
            float v[16];
            umma::tmem_ld_m64<4>(umma::tmem_at(tD1, half * 32), v);
            const int rl = umma::frag_row_lo(), cf = umma::frag_col();
#pragma unroll
            for (int hr = 0; hr < 2; hr++) {
                const int r = rl + 8 * hr;
                const float gr = gam[r];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int j = half * 32 + 8 * k + cf;
                    const float p0 = j <= r ? v[4 * k + 2 * hr] * expf(gr - gam[j]) : 0.f;
                    const float p1 = j + 1 <= r ? v[4 * k + 2 * hr + 1] * expf(gr - gam[j + 1]) : 0.f;
                    *reinterpret_cast<float2*>(Ps + umma::kidx(r, j, 64)) =
                        make_float2(umma::tf32r(p0), umma::tf32r(p1));
                }
            }
        }
        ok = umma::mbar_wait(mU, it & 1);   // U
        if (ok && L < 64) umma::zero_tail_rows(Us, 64, 0, L);   // each thread: its own pieces
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        ok = __syncthreads_and(ok);
        umma::fence_after_sync();
        if (!ok) break;
        if (tid == 0) {
            umma::mma(tD2, umma::kmaj(Ps, 64), umma::mnt(Us), 64, 128, 64, false);
            umma::commit(mbar);
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 1));
        umma::fence_after_sync();
        if (!ok) break;
        // O = D2 + e^{gam_i} D3, staged as a swizzled tile over U (consumed);
        // the norm and the stores then run row by row on all lanes, one warp
        // per row, fully coalesced
        float* Or = Us;
        {
            float ss = 0.f;
            for (int cc = 0; cc < 64; cc += 16) {
                float v2[16], v3[16];
                umma::tmem_ld16(umma::tmem_at(tD2, half * 64 + cc), v2);
                umma::tmem_ld16(umma::tmem_at(tD3, half * 64 + cc), v3);
                if (lane < 16) {
#pragma unroll
                    for (int u = 0; u < 16; u += 4) {
                        float4 x;
                        x.x = v2[u] + eg[i] * v3[u];
                        x.y = v2[u + 1] + eg[i] * v3[u + 1];
                        x.z = v2[u + 2] + eg[i] * v3[u + 2];
                        x.w = v2[u + 3] + eg[i] * v3[u + 3];
                        ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
                        *reinterpret_cast<float4*>(Or + umma::swz(i, half * 64 + cc + u, 64)) = x;
                    }
                }
            }
            if (lane < 16) ssq[half * 64 + i] = ss;
        }
        cp_async_wait<0>();   // z rows
        umma::fence_before_sync();
        __syncthreads();
        for (int r = warp; r < L; r += 8) {
            const int64_t tok = ci.start + r;
            const int64_t off = (tok * hv + h) * kD + lane * 4;
            const float4 o4 = *reinterpret_cast<const float4*>(Or + umma::swz(r, lane * 4, 64));
            st4(sv.o + off, o4);
            if (o_out) st4(o_out + off, o4);
            if (z) {
                const float rs = rsqrtf((ssq[r] + ssq[64 + r]) * (1.f / kD) + norm_eps);
                const float4 z4 = ld4(reinterpret_cast<const IO*>(Zs + r * kZPitch) + lane * 4);
                st4(y_out + off, gated_norm4(o4, rs, w4, z4, gate));
                if (lane == 0) sv.rstd[tok * hv + h] = rs;
            }
        }
        umma::fence_smem_to_async();   // O staging -> the next U load
        __syncthreads();               // O, z and the sums of squares are read
        if (!next) break;
        if (tid == 0) issue_u(cn, tn);
        issue_z(cn, tn);
        g_cur = g_next;
        ci = cn;
        t = tn;
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 512);
    if (!ok && tid == 0) atomicExch(sv.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
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
    {
        cudaError_t e = smem_attr(prep_kernel, kPrepSmem);
        if (e == cudaSuccess) e = smem_attr(state_fwd_kernel, kStateSmem);
        if (e == cudaSuccess) e = smem_attr(out_fwd_kernel<IO>, kOutSmem);
        if (e != cudaSuccess) return e;
    }
    TileMaps maps{};
    if (a.NT > 0) {
        {
            GDN_PROF("gates", st);
            gates_kernel<IO><<<dim3(a.NT, (a.hv + 7) / 8), 256, 0, st>>>(
                (const IO*)a.a, (const IO*)a.b, a.A_log, a.dt_bias, a.hv, a.sv);
        }
        const int64_t C = (int64_t)(2 * a.hk + a.hv) * kD;
        cudaError_t e = make_rows_map(&maps.q, a.qkv, a.hk, a.T, C);
        if (e == cudaSuccess) e = make_rows_map(&maps.k, a.qkv + (int64_t)a.hk * kD, a.hk, a.T, C);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.v, a.qkv + (int64_t)2 * a.hk * kD, a.hv, a.T, C);
        if (e == cudaSuccess) e = make_rows_map(&maps.U, a.sv.U, a.hv, a.T, (int64_t)a.hv * kD);
        if (e == cudaSuccess) e = make_rows_map(&maps.W, a.sv.W, a.hv, a.T, (int64_t)a.hv * kD);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.U_mn, a.sv.U, a.hv, a.T, (int64_t)a.hv * kD, true);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.k_mn, a.qkv + (int64_t)a.hk * kD, a.hk, a.T, C, true);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.v_mn, a.qkv + (int64_t)2 * a.hk * kD, a.hv, a.T, C, true);
        if (e != cudaSuccess) return e;
        int dev = 0, nsm = 0;
        e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        GDN_PROF("chunk_prep", st);
        prep_kernel<<<min(a.NT * a.hv, nsm), 256, kPrepSmem, st>>>(maps, a.hk, a.hv, a.NT, a.sv);
    }
    if (a.N > 0) {
        GDN_PROF("chunk_state_fwd", st);
        state_fwd_kernel<<<dim3(3, a.hv, a.N), 256, kStateSmem, st>>>(
            maps, a.hk, a.hv, a.S_init, a.S_final, a.sv);
    }
    if (a.NT > 0) {
        int dev = 0, nsm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        const int ntiles = a.NT * a.hv;
        GDN_PROF("chunk_out_fwd", st);
        out_fwd_kernel<IO><<<min(ntiles, nsm), 256, kOutSmem, st>>>(
            maps, a.hk, a.hv, a.NT, (const IO*)a.z, a.norm_w, a.norm_eps, a.gate, (IO*)a.o_out,
            (IO*)a.y_out, a.sv);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_fwd(const ChunkArgs& a, cudaStream_t st) {
    return a.bf16 ? chunk_fwd_t<__nv_bfloat16>(a, st) : chunk_fwd_t<float>(a, st);
}

}  // namespace gdn
