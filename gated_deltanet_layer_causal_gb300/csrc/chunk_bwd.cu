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
#include "umma.cuh"


namespace gdn {


__device__ __forceinline__ float4 zero4() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// ------------------------------------------------------------------ B0: gated-norm backward
// rows = T * Hv rows of d_v = 128, one warp per row, 64 rows per CTA (many CTAs
// per SM: a streaming pass).  dO is stored fp32 and tf32-rounded (it is only
// ever a tensor-core operand), dz in the I/O dtype, one dnorm_w partial row per
// CTA.  Without z there is no norm: dO = dy.
constexpr int kNormRows = 64;
template <class IO>
__global__ void __launch_bounds__(256)
chunk_norm_bwd_kernel(const float* __restrict__ o, const IO* __restrict__ z,
                      const float* __restrict__ norm_w, float norm_eps, int gate,
                      const IO* __restrict__ dy, int64_t rows, float* __restrict__ dO,
                      IO* __restrict__ dz, float* __restrict__ part) {
    __shared__ float4 red[8][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float4 w4 = z ? ld4(norm_w + lane * 4) : zero4();
    float4 acc = zero4();
    const int64_t r0 = (int64_t)blockIdx.x * kNormRows, r1 = min(r0 + kNormRows, rows);
    for (int64_t r = r0 + warp; r < r1; r += 8) {
        const int64_t off = r * kD + lane * 4;
        const float4 dy4 = ld4(dy + off);
        float4 d4 = dy4;
        if (z) {
            const NormRowGrad gr =
                norm_row_bwd(ld4(o + off), ld4(z + off), dy4, w4, norm_eps, acc, gate);
            d4 = gr.d_o;
            st4(dz + off, gr.dz);
        }
        st4(dO + off, umma::tf32r(d4));
    }
    if (!z) return;
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float4 s = red[0][lane];
        for (int i = 1; i < 8; i++) {
            s.x += red[i][lane].x; s.y += red[i][lane].y;
            s.z += red[i][lane].z; s.w += red[i][lane].w;
        }
        st4(part + (int64_t)blockIdx.x * kD + lane * 4, s);
    }
}

// ------------------------------------------------------------------ B1: local
// grid NT * Hk (block = chunk * Hk + k-head), 256 threads, tcgen05: a CTA takes
// the G = Hv / Hk v-heads that share the k-head's q and k, one after another.
//   D1 = K Q^T (64 x 64, once)
//   per v-head h:  P^T_h[j][i] = D1[j][i] e^{gam_h,i - gam_h,j} [i >= j]
//                  dU_local_h = P^T_h dO_h     (64 x 128)
// Shared memory: Q, K swizzled and one v-head's dO MN-major, 32 KB each (TMA; dO
// is the B operand of P^T dO, contracted over tokens, so it is read as loaded,
// and has its own barrier: K Q^T and P^T do not wait for it; the next v-head's is
// requested once the current product is done).  P^T (16 KB) takes the K space
// once K Q^T is done, dU_local is staged in the Q space and stored whole.  About
// 97 KB: two CTAs per SM.  Tensor memory: 192 fp32 columns (256 allocated).
constexpr int kB1Floats = 64 * 128 * 3;
constexpr size_t kB1Smem = sizeof(float) * (kB1Floats + 64 + 16) + 64 + 1024;

__global__ void __launch_bounds__(256, 2)
bwd_local_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, FwdSaved sv,
                 BwdScratch w) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* Qs = sm;                    // [64][128] swizzled; then dU_local staged
    float* Ks = Qs + 64 * 128;         // [64][128] swizzled
    float* dOs = Ks + 64 * 128;        // [64 (i)][128 (a)] MN-major dO (arrives rounded)
    float* PT = Ks;                    // [64 (j)][64 (i)] K-major, after K Q^T
    float* gam = dOs + 64 * 128;
    uint64_t* mbar = reinterpret_cast<uint64_t*>(gam + 64 + 16);
    uint64_t* mbl = mbar + 1;          // Q, K
    uint64_t* mbo = mbl + 1;           // dO of one v-head
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbo + 1);
    // the P / dP kernel, launched after this one, claims its work from this counter
    if (blockIdx.x == 0 && threadIdx.x == 0) *w.dp_next = 0;
    const ChunkInfo ci = sv.chunks[blockIdx.x / hk];
    if (ci.len == 0) return;
    const int kh = blockIdx.x % hk, G = hv / hk, tid = threadIdx.x, L = ci.len;
    const int warp = tid >> 5;
    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::mbar_init(mbl, 1);
        umma::mbar_init(mbo, 1);
        umma::mbar_expect_tx(mbl, 2 * 64 * 128 * 4);
        umma::tma_rows(Qs, 64, &maps.q, kh, ci.start, mbl);
        umma::tma_rows(Ks, 64, &maps.k, kh, ci.start, mbl);
        umma::mbar_expect_tx(mbo, 64 * 128 * 4);
        umma::tma_rows(dOs, 64, &maps.dO_mn, kh * G, ci.start, mbo);
    }
    // gate values of a v-head, loaded a v-head before they are used
    auto gam_of = [&](int h) {
        float g = 0.f;
        if (tid < 64) g = sv.gam[(int64_t)h * sv.T + ci.start + min(tid, L - 1)];
        return g;
    };
    float g_cur = gam_of(kh * G);
    if (warp == 0) umma::tmem_alloc(tslot, 256);
    __syncthreads();
    bool ok = __syncthreads_and(umma::mbar_wait(mbl, 0));
    if (L < 64) {   // tail rows belong to the next sequence
        umma::zero_tail_rows(Qs, 64, 0, L);
        umma::zero_tail_rows(Ks, 64, 0, L);
        __syncthreads();
    }
    if (!sv.qkv_tf32) umma::tf32r_inplace(Qs, 2 * 64 * 128);
    umma::fence_smem_to_async();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tD1 = tmem, tD2 = tmem + 64;
    if (ok && tid == 0) {
        umma::mma(tD1, umma::swt(Ks, 64), umma::swt(Qs, 64), 64, 64, 128, false);
        umma::commit(mbar);
    }
    ok = __syncthreads_and(ok && umma::mbar_wait(mbar, 0));
    umma::fence_after_sync();
    const int half = warp >> 2;
    const int rl = umma::frag_row_lo(), cf = umma::frag_col();
    float d1[16];   // this thread's fragment of K Q^T, for every v-head
    if (ok) umma::tmem_ld_m64<4>(umma::tmem_at(tD1, half * 32), d1);
    for (int jh = 0; jh < G && ok; jh++) {
        const int h = kh * G + jh;
        const float g_next = jh + 1 < G ? gam_of(h + 1) : 0.f;
        if (tid < 64) gam[tid] = g_cur;
        __syncthreads();   // gam visible; the last v-head's P^T read by its product
        {   // P^T[j][i], 32 columns per warp, all lanes
#pragma unroll
            for (int hr = 0; hr < 2; hr++) {
                const int jr = rl + 8 * hr;
                const float gj = gam[jr];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int i = half * 32 + 8 * k + cf, q = 4 * k + 2 * hr;
                    const float p0 = i >= jr ? d1[q] * expf(gam[i] - gj) : 0.f;
                    const float p1 = i + 1 >= jr ? d1[q + 1] * expf(gam[i + 1] - gj) : 0.f;
                    *reinterpret_cast<float2*>(PT + umma::kidx(jr, i, 64)) =
                        make_float2(umma::tf32r(p0), umma::tf32r(p1));
                }
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        ok = __syncthreads_and(umma::mbar_wait(mbo, jh & 1));
        if (!ok) break;
        if (L < 64) {
            umma::zero_tail_rows(dOs, 64, 0, L);
            umma::fence_smem_to_async();
            __syncthreads();
        }
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tD2, umma::kmaj(PT, 64), umma::mnt(dOs), 64, 128, 64, false);
            umma::commit(mbar);
            umma::bulk_wait_read();   // the last v-head's dU_local store has read the Q space
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, (jh + 1) & 1));
        umma::fence_after_sync();
        if (!ok) break;
        if (tid == 0 && jh + 1 < G) {   // dO consumed: the next v-head's
            umma::mbar_expect_tx(mbo, 64 * 128 * 4);
            umma::tma_rows(dOs, 64, &maps.dO_mn, h + 1, ci.start, mbo);
        }
        {   // dU_local staged as a swizzled tile in the Q space, stored whole
            float v[32];
            umma::tmem_ld64_m64(umma::tmem_at(tD2, half * 64), v);
            umma::frag_to_sw(Qs, v, half * 64, 1.f, 1.f);
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        if (L == 64) {
            if (tid == 0) {
                umma::tma_store_rows(&maps.dUl, h, ci.start, Qs);
                umma::bulk_commit();
            }
        } else {
            umma::store_rows_sw(w.dUl + ((int64_t)ci.start * hv + h) * kD, (int64_t)hv * kD, Qs, L);
        }
        g_cur = g_next;
    }
    if (tid == 0) umma::bulk_wait_read();
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 256);
    if (!ok && tid == 0) atomicExch(w.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ B2: reverse state pass
// One CTA per (slice, head, sequence), 320 threads, tcgen05, one CTA per SM (the
// first CTAs of the combined launch below).  Carries rows a0 .. a0 + 63
// (a0 = 64 slice) of dS, the gradient of the state S [d_v x d_k], from the last
// chunk of the sequence to the first.  With dS the gradient at a chunk's end
// and fk_i = e^{gam_L - gam_i} (0 past the chunk), per chunk:
//   D1 = K dS^T                                 (M = 64 tokens, N = 64, K = 128)
//   dU = dU_local + diag(fk) D1                 -> global (rounded)
//   dS_start^T = e^{gam_L} dS^T + B'^T + W^T Ub,   Ub = -diag(fk) D1,
//   B'^T = Q^T diag(e^gam) dO - W^T dU_local    (M = 128, N = 64, K = 64 tokens)
// B' does not depend on dS: it is issued ahead into the chunk's accumulator, so
// the chain per chunk is D1, the Ub epilogue, one 8-instruction product W^T Ub
// and the update.  dS lives in registers as the transposed accumulator (thread
// b holds rows a0 .. a0 + 63 of column b) and is stored at every chunk end as
// its tf32 copy (D1's B operand), row-major, by one tensor store.
// Roles, coupled by mbarriers (one phase per chunk, or per use of a buffer; a
// barrier whose next phase could complete before a waiter has seen the current
// one is split per buffer, so a parity wait never takes one phase for another):
//  - scaling warps (0-3): scale the dO slice by e^gam, negate the dU_local
//    slice, zero both past the chunk; round Q and K when they are not tf32;
//    then the chunk's dU rows (D1 read from tensor memory, dU_local one chunk
//    ahead in registers);
//  - state warps (4-7): the Ub epilogue (D1 read, "Ub ready"), the update
//    ("accumulator read", "dS ready", the dS store);
//  - chain thread (warp 8): D1 once dS and K are ready, then W^T Ub once Ub and
//    B' are; refills K (two buffers, once D1 is done) and W (once W^T Ub is
//    done), prefetching both into L2 a chunk earlier;
//  - product thread (warp 9): B' once Q, dO, dU_local are scaled and the
//    accumulator is free; then refills Q, dO, dU_local.
// dU_local arrives from its own buffer, so dU is written without a hazard.
// Shared memory: dS copy 32 KB, K (K-major) 2 x 32 KB, W (MN-major) 32 KB, Q
// (MN-major) 32 KB, dO and dU_local slices and Ub (MN-major, 64 x 64) 16 KB
// each.  Tensor memory: two accumulators (M = 128, 64 columns) and D1 (M = 64,
// 64 columns).
constexpr int kSl = 64;
constexpr int kStateThreadsB = 320;
constexpr int kB2Floats = 5 * 64 * 128 + 3 * 64 * 64;
constexpr int kB2Bars = 16;
constexpr size_t kB2Smem = sizeof(float) * kB2Floats + kB2Bars * 8 + 8 + 1024;

__device__ __forceinline__ void bwd_state_cta(const TileMaps& maps, int sl, int h, int n, int hk,
                                              int hv, const float* dS_final, float* dS_init,
                                              const FwdSaved& sv, const BwdScratch& w) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* dSt = sm;                   // [64 (a)][128 (b)] swizzled K-major: dS, rounded
    float* Kk0 = dSt + 64 * 128;       // [2][64 (i)][128 (b)] swizzled K-major K
    float* Wm = Kk0 + 2 * 64 * 128;    // [64 (i)][128 (b)] MN-major W (arrives rounded)
    float* Qm = Wm + 64 * 128;         // [64 (i)][128 (b)] MN-major Q
    float* dOs = Qm + 64 * 128;        // [64 (i)][64 (a)] MN-major dO slice (arrives rounded)
    float* dUs = dOs + 64 * 64;        // [64 (i)][64 (a)] MN-major dU_local slice
    float* Ub = dUs + 64 * 64;         // [64 (i)][64 (a)] MN-major -diag(fk) D1, rounded
    uint64_t* mA = reinterpret_cast<uint64_t*>(Ub + 64 * 64);   // Q, dO, dU_local loaded
    uint64_t* mK = mA + 1;             // [2] K loaded, per buffer
    uint64_t* mW = mK + 2;             // W loaded
    uint64_t* bSc = mW + 1;            // Q, dO, dU_local scaled (scaling warps)
    uint64_t* bK = bSc + 1;            // K ready (scaling warps)
    uint64_t* mPb = bK + 1;            // [2] B'^T done, per accumulator (commit)
    uint64_t* mD1 = mPb + 2;           // D1 done (commit)
    uint64_t* bU = mD1 + 1;            // Ub written (state warps)
    uint64_t* mC = bU + 1;             // W^T Ub done (commit)
    uint64_t* bS = mC + 1;             // dS copy written (state warps)
    uint64_t* fA = bS + 1;             // [2] accumulator read (state warps)
    uint64_t* dR = fA + 2;             // D1 read by the scaling warps
    uint32_t* tslot = reinterpret_cast<uint32_t*>(dR + 1);
    auto Kk = [&](int it) { return Kk0 + (it & 1) * 64 * 128; };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int a0 = sl * kSl, kh = h / (hv / hk);
    const int64_t sbase = ((int64_t)n * hv + h) * kD * kD;
    const int c0 = sv.seq_chunk[n], c1 = sv.seq_chunk[n + 1], nc = c1 - c0;
    // iteration it works on chunk c1 - 1 - it
    if (tid == 0) {
        umma::mbar_init(mA, 1);
        umma::mbar_init(&mK[0], 1);
        umma::mbar_init(&mK[1], 1);
        umma::mbar_init(mW, 1);
        umma::mbar_init(bSc, 128);
        umma::mbar_init(bK, 128);
        umma::mbar_init(&mPb[0], 1);
        umma::mbar_init(&mPb[1], 1);
        umma::mbar_init(mD1, 1);
        umma::mbar_init(bU, 128);
        umma::mbar_init(mC, 1);
        umma::mbar_init(bS, 128);
        umma::mbar_init(&fA[0], 128);
        umma::mbar_init(&fA[1], 128);
        umma::mbar_init(dR, 128);
    }
    if (warp == 0) umma::tmem_alloc(tslot, 256);
    umma::fence_before_sync();
    __syncthreads();   // barriers initialised, tensor memory allocated
    umma::fence_after_sync();
    const uint32_t tmem = *tslot, tD1 = tmem + 128;
    auto tAcc = [&](int it) { return tmem + 64u * (uint32_t)(it & 1); };
    auto start_of = [&](int it) { return sv.chunks[c1 - 1 - it].start; };
    bool ok = true;
    if (warp < 4) {
        // ---------------------------------------------------------- scaling warps
        // Per iteration it: K ready (the chain's next D1 waits for it), then the
        // dU rows of chunk it (once D1 is done), then the dO / dU_local slices of
        // chunk it + 1 (B' runs a chunk ahead).  A chunk's gate values and dU_local
        // rows are read two iterations ahead and the exponentials taken at use: a
        // load used at once would wait on memory shared with the P / dP tiles.
        // Slices: thread t scales the 16-byte pieces t + 128 q (rows (t / 8 + 16 q) % 64).
        // dU rows: D1 fragment rows rl, rl + 8, columns 8 k + cf, + 1.
        const int r0 = tid >> 3;
        const int rl = umma::frag_row_lo(), cf = umma::frag_col();
        struct Rows {
            float g[4];            // gam of the slice rows r0 + 16 u
            float glo, ghi, gL;    // gam of the dU rows and of the chunk's last token
            int len, start;
            float ul[32];          // dU_local of the dU rows (0 past the chunk)
        };
        auto load = [&](int it, Rows& r) {
            r.len = r.start = 0;
            r.glo = r.ghi = r.gL = 0.f;
#pragma unroll
            for (int u = 0; u < 4; u++) r.g[u] = 0.f;
#pragma unroll
            for (int x = 0; x < 32; x++) r.ul[x] = 0.f;
            if (it >= nc) return;
            const ChunkInfo info = sv.chunks[c1 - 1 - it];
            const float* g = sv.gam + (int64_t)h * sv.T + info.start;
            r.len = info.len;
            r.start = info.start;
#pragma unroll
            for (int u = 0; u < 4; u++) r.g[u] = g[min(r0 + 16 * u, info.len - 1)];
            r.glo = g[min(rl, info.len - 1)];
            r.ghi = g[min(rl + 8, info.len - 1)];
            r.gL = g[info.len - 1];
#pragma unroll
            for (int hr = 0; hr < 2; hr++) {
                const int i = rl + 8 * hr;
                if (i >= info.len) continue;
                const float* src = w.dUl + ((int64_t)(info.start + i) * hv + h) * kD + a0 + cf;
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const float2 v = *reinterpret_cast<const float2*>(src + 8 * k);
                    r.ul[4 * k + 2 * hr] = v.x;
                    r.ul[4 * k + 2 * hr + 1] = v.y;
                }
            }
        };
        // the dO / dU_local slices of chunk it: e^gam dO and -dU_local, zero past the
        // chunk, rounded; Q rounded when it is not tf32
        auto scale_a = [&](int it, const Rows& r) {
            bool got = umma::mbar_wait(mA, it & 1);
            if (got) {
                float4* o4 = reinterpret_cast<float4*>(dOs);
                float4* u4 = reinterpret_cast<float4*>(dUs);
#pragma unroll
                for (int q = 0; q < 8; q++) {
                    const bool in = r0 + 16 * (q & 3) < r.len;
                    const float e = in ? expf(r.g[q & 3]) : 0.f;
                    const float m = in ? -1.f : 0.f;
                    const float4 ov = o4[tid + 128 * q], uv = u4[tid + 128 * q];
                    o4[tid + 128 * q] = umma::tf32r(make_float4(e * ov.x, e * ov.y, e * ov.z, e * ov.w));
                    u4[tid + 128 * q] = umma::tf32r(make_float4(m * uv.x, m * uv.y, m * uv.z, m * uv.w));
                }
                if (!sv.qkv_tf32) umma::tf32r_inplace<128>(Qm, 64 * 128);
            }
            umma::fence_smem_to_async();
            umma::mbar_arrive(bSc);
            return got;
        };
        Rows cur, nxt;   // chunks it and it + 1
        load(0, cur);
        load(1, nxt);
        if (nc > 0) ok = scale_a(0, cur);
        for (int it = 0; it < nc && ok; it++) {
            if (!sv.qkv_tf32) {   // K rounded in place ("K ready"; else the chain waits the load)
                ok = umma::mbar_wait(&mK[it & 1], (it >> 1) & 1);
                if (ok) umma::tf32r_inplace<128>(Kk(it), 64 * 128);
                umma::fence_smem_to_async();
                umma::mbar_arrive(bK);
            }
            // dU = dU_local + diag(fk) D1 for the rows inside the chunk (rounded: only
            // ever a tensor-core operand later).  "D1 read" lets the next D1 go.
            ok = __all_sync(0xffffffffu, ok && umma::mbar_wait(mD1, it & 1));   // warp-uniform
            umma::fence_after_sync();
            if (ok) {
                float d1[32];
                umma::tmem_ld64_m64(umma::tmem_at(tD1, 0), d1);
#pragma unroll
                for (int hr = 0; hr < 2; hr++) {
                    const int i = rl + 8 * hr;
                    if (i >= cur.len) continue;
                    const float f = expf(cur.gL - (hr ? cur.ghi : cur.glo));
                    float* dst = w.dU + ((int64_t)(cur.start + i) * hv + h) * kD + a0 + cf;
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        *reinterpret_cast<float2*>(dst + 8 * k) = make_float2(
                            umma::tf32r(cur.ul[4 * k + 2 * hr] + f * d1[4 * k + 2 * hr]),
                            umma::tf32r(cur.ul[4 * k + 2 * hr + 1] + f * d1[4 * k + 2 * hr + 1]));
                }
            }
            umma::fence_before_sync();
            umma::mbar_arrive(dR);
            if (ok && it + 1 < nc) ok = scale_a(it + 1, nxt);
            cur = nxt;
            load(it + 2, nxt);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------- state warps
        const int q = warp - 4, bp = 32 * q + lane, sid = tid - 128;
        const int rl = umma::frag_row_lo(), cf = umma::frag_col();
        float s[64];   // s[j] = dS[a0 + j][bp]
#pragma unroll
        for (int j = 0; j < 64; j++)
            s[j] = dS_final ? dS_final[sbase + (int64_t)(a0 + j) * kD + bp] : 0.f;
        // dS into its copy (rounded), "dS ready", then the copy out as the gradient
        // at the end of chunk c (one tensor store: row-major, rounded)
        auto put = [&](int c) {
            if (sid == 0) umma::bulk_wait_read();   // the last store has read the copy
            umma::named_sync(2, 128);
#pragma unroll
            for (int j = 0; j < 64; j++) dSt[umma::swz(j, bp, 64)] = umma::tf32r(s[j]);
            umma::fence_smem_to_async();
            umma::mbar_arrive(bS);
            umma::named_sync(2, 128);
            if (sid == 0) {
                umma::tma_store_rows(&maps.dS, 0, (c * hv + h) * kD + a0, dSt);
                umma::bulk_commit();
            }
            __syncwarp();   // converged again before the warp-wide tensor-memory loads
        };
        // gate values of iteration it: fk of rows rl, rl + 8 and e^{gam_L}
        auto gates = [&](int it, float& f_lo, float& f_hi, float& dl, int& len, int& start) {
            f_lo = f_hi = dl = 0.f;
            len = start = 0;
            if (it >= nc) return;
            const ChunkInfo info = sv.chunks[c1 - 1 - it];
            const float* g = sv.gam + (int64_t)h * sv.T + info.start;
            const float gL = g[info.len - 1];
            f_lo = rl < info.len ? expf(gL - g[rl]) : 0.f;
            f_hi = rl + 8 < info.len ? expf(gL - g[rl + 8]) : 0.f;
            dl = expf(gL);
            len = info.len;
            start = info.start;
        };
        float f_lo, f_hi, dl, f_lo_n, f_hi_n, dl_n;
        int len, start, len_n, start_n;
        gates(0, f_lo, f_hi, dl, len, start);
        if (nc > 0) put(c1 - 1);
        for (int it = 0; it < nc && ok; it++) {
            gates(it + 1, f_lo_n, f_hi_n, dl_n, len_n, start_n);
            ok = __all_sync(0xffffffffu, umma::mbar_wait(mD1, it & 1));   // warp-uniform
            umma::fence_after_sync();
            if (!ok) break;
            float d1[32];   // D1 rows rl, rl + 8, columns 8 k + cf, + 1
            umma::tmem_ld64_m64(umma::tmem_at(tD1, 0), d1);
#pragma unroll
            for (int k = 0; k < 8; k++) {   // Ub = -diag(fk) D1, rounded
                const int a = 8 * k + cf;
                *reinterpret_cast<float2*>(Ub + umma::swz_mn(rl, a, 64)) =
                    make_float2(umma::tf32r(-f_lo * d1[4 * k]), umma::tf32r(-f_lo * d1[4 * k + 1]));
                *reinterpret_cast<float2*>(Ub + umma::swz_mn(rl + 8, a, 64)) =
                    make_float2(umma::tf32r(-f_hi * d1[4 * k + 2]), umma::tf32r(-f_hi * d1[4 * k + 3]));
            }

            umma::fence_smem_to_async();
            umma::fence_before_sync();
            umma::mbar_arrive(bU);
            ok = __all_sync(0xffffffffu, umma::mbar_wait(mC, it & 1));   // warp-uniform
            umma::fence_after_sync();
            if (!ok) break;
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {   // dS <- e^{gam_L} dS + B' + W^T Ub
                float v[32];
                umma::tmem_ld32(umma::tmem_at(tAcc(it), cc), v);
#pragma unroll
                for (int u = 0; u < 32; u++) s[cc + u] = dl * s[cc + u] + v[u];
            }
            umma::fence_before_sync();
            umma::mbar_arrive(&fA[it & 1]);   // the accumulator is read
            if (it + 1 < nc) put(c1 - 2 - it);
            f_lo = f_lo_n;
            f_hi = f_hi_n;
            dl = dl_n;
            len = len_n;
            start = start_n;
        }
        if (sid == 0) umma::bulk_wait_read();
        if (ok && dS_init)
#pragma unroll
            for (int j = 0; j < 64; j++) dS_init[sbase + (int64_t)(a0 + j) * kD + bp] = s[j];
    } else if (tid == 256) {
        // ---------------------------------------------------------- chain thread
        // K of chunk it + 2 is requested once D1 of chunk it is done (two buffers);
        // W of chunk it once the W^T Ub product one back is done (one buffer: its
        // first reader, B', runs well before the second); both prefetched into L2
        // earlier (memory is shared with the P / dP tiles)
        auto issue_k = [&](int it) {
            umma::mbar_expect_tx(&mK[it & 1], 64 * 128 * 4);
            umma::tma_rows(Kk(it), 64, &maps.k, kh, start_of(it), &mK[it & 1]);
        };
        auto issue_w = [&](int it) {
            umma::mbar_expect_tx(mW, 64 * 128 * 4);
            umma::tma_rows(Wm, 64, &maps.W_mn, h, start_of(it), mW);
        };
        if (nc > 0) {
            issue_k(0);
            issue_w(0);
        }
        if (nc > 1) {
            issue_k(1);
            umma::tma_prefetch_rows(&maps.W_mn, h, start_of(1));
        }
        if (nc > 2) umma::tma_prefetch_rows(&maps.k, kh, start_of(2));
        for (int it = 0; it < nc && ok; it++) {
            ok = umma::mbar_wait(bS, it & 1);   // dS at this chunk's end: W^T Ub one back is done
            if (ok && it >= 1) issue_w(it);
            if (ok && it + 2 < nc) umma::tma_prefetch_rows(&maps.W_mn, h, start_of(it + 2));
            if (ok && it + 3 < nc) umma::tma_prefetch_rows(&maps.k, kh, start_of(it + 3));
            ok = ok && (sv.qkv_tf32 ? umma::mbar_wait(&mK[it & 1], (it >> 1) & 1)
                                    : umma::mbar_wait(bK, it & 1));
            if (it >= 1) ok = ok && umma::mbar_wait(dR, (it - 1) & 1);   // D1 one back read
            umma::fence_after_sync();
            if (!ok) break;
            umma::mma(tD1, umma::swt(Kk(it), 64), umma::swt(dSt, 64), 64, 64, 128, false);
            umma::commit(mD1);
            ok = umma::mbar_wait(mD1, it & 1);   // D1 done: its K buffer is free
            if (ok && it + 2 < nc) issue_k(it + 2);
            ok = ok && umma::mbar_wait(bU, it & 1);   // Ub written
            ok = ok && umma::mbar_wait(&mPb[it & 1], (it >> 1) & 1) && umma::mbar_wait(mW, it & 1);
            umma::fence_after_sync();
            if (!ok) break;
            umma::mma(tAcc(it), umma::mnt(Wm), umma::mnt(Ub, 64), 128, 64, 64, true);
            umma::commit(mC);
        }
    } else if (tid == 288) {
        // ---------------------------------------------------------- product thread
        auto issue_a = [&](int it) {
            const int st = start_of(it);
            umma::mbar_expect_tx(mA, (64 * 128 + 2 * 64 * 64) * 4);
            umma::tma_rows(Qm, 64, &maps.q_mn, kh, st, mA);
            umma::tma_box(dOs, &maps.dO_mn, a0, h, st, mA);
            umma::tma_box(dOs + 64 * 32, &maps.dO_mn, a0 + 32, h, st, mA);
            umma::tma_box(dUs, &maps.dUl_mn, a0, h, st, mA);
            umma::tma_box(dUs + 64 * 32, &maps.dUl_mn, a0 + 32, h, st, mA);
        };
        // Q, dO, dU_local of chunk it + 2 prefetched into L2 at iteration it
        auto prefetch_a = [&](int it) {
            const int st = start_of(it);
            umma::tma_prefetch_rows(&maps.q_mn, kh, st);
            umma::tma_prefetch_box(&maps.dO_mn, a0, h, st);
            umma::tma_prefetch_box(&maps.dO_mn, a0 + 32, h, st);
            umma::tma_prefetch_box(&maps.dUl_mn, a0, h, st);
            umma::tma_prefetch_box(&maps.dUl_mn, a0 + 32, h, st);
        };
        if (nc > 0) issue_a(0);
        if (nc > 1) prefetch_a(1);
        for (int it = 0; it < nc && ok; it++) {
            if (it + 2 < nc) prefetch_a(it + 2);
            ok = umma::mbar_wait(bSc, it & 1) && umma::mbar_wait(mW, it & 1);
            // accumulator it & 1: the state warps have read it (two chunks back)
            if (it >= 2) ok = ok && umma::mbar_wait(&fA[it & 1], ((it / 2) - 1) & 1);
            umma::fence_after_sync();
            if (!ok) break;
            umma::mma(tAcc(it), umma::mnt(Qm), umma::mnt(dOs, 64), 128, 64, 64, false);
            umma::mma(tAcc(it), umma::mnt(Wm), umma::mnt(dUs, 64), 128, 64, 64, true);
            umma::commit(&mPb[it & 1]);
            ok = umma::mbar_wait(&mPb[it & 1], (it >> 1) & 1);   // Q, dO, dU_local consumed
            if (ok && it + 1 < nc) issue_a(it + 1);
        }
    }
    umma::fence_before_sync();
    ok = __syncthreads_and(ok);
    if (warp == 0) umma::tmem_free(tmem, 256);
    if (!ok && tid == 0) atomicExch(w.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ B3a: state-facing terms
// Persistent: one CTA per SM walks (chunk, k-head) groups g = blockIdx.x,
// + gridDim.x, ... (chunk = g / Hk, k-head = g % Hk), each as the tiles of its
// G = Hv / Hk v-heads in turn.  Per tile, tcgen05:
//   [X; Y] = [dO; dU] S0     (one M=128, N=128, K=128 MMA; X = dO S0, Y = dU S0)
//   dK~    = U dS            (M=64, N=128, K=128)
// then dW = -Y, and the dgam terms
//   dgam_i += e^{gam_i} X_i . Q_i,  dgam_j -= Z_j = fk_j dK~_j . K_j,
//   dgam_{L-1} += sum_j Z_j + e^{gam_L} <dS, S0>;
// the dQ part e^gam X and the dK part fk dK~ are added, v-head by v-head in
// order, into tensor-memory sums and written once per k-head at the group's last
// v-head (the q / k gradient of a k-head is the sum over its v-heads: a third
// of the bytes at G = 3, written here and read by the GVA sum).
// Shared memory: [dO; dU] 64 KB and U 32 KB swizzled, S0 64 KB MN-major (rows a,
// the contraction dimension of [dO; dU] S0; all by TMA), dS^T 64 KB K-major
// rows b (one bulk copy).  dS^T is free once the
// products are done and takes the next tile's at once; the other tiles hold
// this tile's Q, K and staged outputs until its stores have read them.
// Tensor memory: the products' 256 fp32 columns and the two sums' 256, once.
constexpr int kSfFloats = 128 * 128 * 3 + 64 * 128;
constexpr size_t kB3aSmem = sizeof(float) * (kSfFloats + 64 * 3 + 2 * 128 + 16) + 64 + 1024;

__global__ void __launch_bounds__(256, 1)
bwd_sfacing_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, int NT, FwdSaved sv,
                   BwdScratch w) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* A1 = sm;                      // [128][128] swizzled: rows 0-63 dO, 64-127 dU
    float* S0m = A1 + 128 * 128;         // [128 (a)][128 (b)] MN-major (arrives rounded)
    float* DSm = S0m + 128 * 128;        // [128 (a)][128 (b)] MN-major dS (arrives rounded)
    float* A2 = DSm + 128 * 128;         // [64][128] swizzled: U
    float* eg = A2 + 64 * 128;
    float* fk = eg + 64;
    float* gam = fk + 64;
    float* rpart = gam + 64;             // [2][128]
    float* red = rpart + 2 * 128;        // [16]
    uint64_t* mbar = reinterpret_cast<uint64_t*>(red + 16);   // MMA
    uint64_t* mS = mbar + 1;             // [dO; dU], U, S0^T
    uint64_t* mD = mS + 1;               // dS^T
    uint64_t* mQ = mD + 1;               // Q, K (dgam dot products)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mQ + 1);
    // the products' operands are consumed after the first wait: Q and K come into
    // the S0 space; the outputs are staged as swizzled tiles in the consumed
    // operand space and stored whole: dQ part and dW over [dO; dU], dK part over U
    float* Qr = S0m;                     // [64][128] swizzled
    float* Kr = S0m + 64 * 128;          // [64][128] swizzled
    float* SQ = A1;                      // [64][128] swizzled
    float* SW = A1 + 64 * 128;           // [64][128] swizzled
    float* SK = A2;                      // [64][128] swizzled
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = hv / hk, ngroups = NT * hk;
    // a CTA walks (chunk, k-head) groups g = blockIdx.x, + gridDim.x, ..., each as
    // its G v-head tiles t = chunk H_v + k-head G + j in turn
    auto first_tile = [&](int g) { return (g / hk) * hv + (g % hk) * G; };
    if ((int)blockIdx.x >= ngroups) return;
    int t = first_tile(blockIdx.x);
    ChunkInfo ci = sv.chunks[t / hv];
    if (ci.len == 0) return;   // the device check of cu_seqlens failed: every chunk is empty
    auto issue_main = [&](const ChunkInfo& c, int tile) {   // one thread
        const int h = tile % hv;
        umma::mbar_expect_tx(mS, 3 * 64 * 128 * 4 + 128 * 128 * 4);
        umma::tma_rows(A1, 128, &maps.dO, h, c.start, mS);
        umma::tma_rows(A1 + 64 * 32, 128, &maps.dU, h, c.start, mS);
        umma::tma_rows(A2, 64, &maps.U, h, c.start, mS);
        const int s0row = ((tile / hv) * hv + h) * kD;   // S0 tile rows a = 0 .. 127
        umma::tma_rows(S0m, 128, &maps.S0_mn, 0, s0row, mS);
        umma::tma_rows(S0m + 64 * 32, 128, &maps.S0_mn, 0, s0row + 64, mS);
    };
    auto issue_ds = [&](int tile) {   // one thread
        const int row = ((tile / hv) * hv + tile % hv) * kD;   // dS tile rows a = 0 .. 127
        umma::mbar_expect_tx(mD, 128 * 128 * 4);
        umma::tma_rows(DSm, 128, &maps.dS_mn, 0, row, mD);
        umma::tma_rows(DSm + 64 * 32, 128, &maps.dS_mn, 0, row + 64, mD);
    };
    auto gam_of = [&](const ChunkInfo& c, int tile) {
        return tid < 64 ? sv.gam[(int64_t)(tile % hv) * sv.T + c.start + min(tid, c.len - 1)] : 0.f;
    };
    if (tid == 0) {
        for (int k = 0; k < 4; k++) umma::mbar_init(&mbar[k], 1);
        issue_main(ci, t);
        issue_ds(t);
    }
    float g_cur = gam_of(ci, t);
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    // the group's dQ and dK parts, summed over its v-heads in order: dQ in the
    // layout of the X rows (lanes 0-63), dK in that of the M = 64 product
    const uint32_t tQacc = tmem + 256, tKacc = tmem + 384;
    const int half = warp >> 2, win = warp & 3;
    const int c0 = half * 64;
    bool ok = true;
    for (int it = 0;; it++) {
        const int h = t % hv, kh = h / G, L = ci.len, jh = h % G;
        const bool first = jh == 0, last = jh == G - 1;
        const int gnext = (t / hv) * hk + kh + (int)gridDim.x;   // the next group
        const int tn = last ? (gnext < ngroups ? first_tile(gnext) : -1) : t + 1;
        const ChunkInfo cn = tn < 0 ? ci : (last ? sv.chunks[tn / hv] : ci);
        if (tid < 64) gam[tid] = g_cur;
        ok = umma::mbar_wait(mS, it & 1);
        ok = __syncthreads_and(ok && umma::mbar_wait(mD, it & 1));   // gam visible
        if (!ok) break;
        if (L < 64) {   // tail rows belong to the next sequence
            umma::zero_tail_rows(A1, 128, 0, L);
            umma::zero_tail_rows(A1, 128, 64, L);
            umma::zero_tail_rows(A2, 64, 0, L);
        }
        {   // <dS, S0> over the staged tiles (same layout)
            float dot = 0.f;
            for (int i = tid; i < 128 * 128; i += 256) dot += S0m[i] * DSm[i];
            dot = warp_sum(dot);
            if (lane == 0) red[warp] = dot;
        }
        umma::fence_smem_to_async();
        __syncthreads();   // (dO, dU, U, S0 and dS arrive rounded)
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tmem, umma::swt(A1, 128), umma::mnt(S0m, 128), 128, 128, 128, false);
            umma::mma(tmem + 128, umma::swt(A2, 64), umma::mnt(DSm, 128), 64, 128, 128, false);
            umma::commit(mbar);
        }
        if (tid < 64) {
            eg[tid] = tid < L ? expf(gam[tid]) : 0.f;
            fk[tid] = tid < L ? expf(gam[L - 1] - gam[tid]) : 0.f;
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, it & 1));
        umma::fence_after_sync();
        if (!ok) break;
        const bool next = tn >= 0 && cn.len > 0;
        if (tid == 0) {
            umma::mbar_expect_tx(mQ, 2 * 64 * 128 * 4);
            umma::tma_rows(Qr, 64, &maps.q, kh, ci.start, mQ);
            umma::tma_rows(Kr, 64, &maps.k, kh, ci.start, mQ);
            if (next) issue_ds(tn);   // dS^T consumed by the product and the dot product
        }
        const float g_next = next ? gam_of(cn, tn) : 0.f;
        ok = __syncthreads_and(umma::mbar_wait(mQ, it & 1));
        if (!ok) break;
        // D1: rows 0..127 in lanes 0..127
        {
            const int r = win * 32 + lane;
            float part = 0.f;
            for (int cc = 0; cc < 64; cc += 16) {
                float v[16];
                umma::tmem_ld16(umma::tmem_at(tmem, c0 + cc), v);
                if (r < 64) {
                    const float e = eg[r];
                    float a[16];
                    if (first) {
#pragma unroll
                        for (int u = 0; u < 16; u++) a[u] = 0.f;
                    } else {
                        umma::tmem_ld16(umma::tmem_at(tQacc, c0 + cc), a);
                    }
#pragma unroll
                    for (int u = 0; u < 16; u += 4) {
                        const float4 q4 = *reinterpret_cast<const float4*>(
                            Qr + umma::swz(r, c0 + cc + u, 64));
                        part += v[u] * q4.x + v[u + 1] * q4.y + v[u + 2] * q4.z + v[u + 3] * q4.w;
                        a[u] += e * v[u];
                        a[u + 1] += e * v[u + 1];
                        a[u + 2] += e * v[u + 2];
                        a[u + 3] += e * v[u + 3];
                        if (last)
                            *reinterpret_cast<float4*>(SQ + umma::swz(r, c0 + cc + u, 64)) =
                                make_float4(a[u], a[u + 1], a[u + 2], a[u + 3]);
                    }
                    if (!last) umma::tmem_st16(umma::tmem_at(tQacc, c0 + cc), a);
                } else {
#pragma unroll
                    for (int u = 0; u < 16; u += 4)   // dW: a tensor-core operand only, rounded
                        *reinterpret_cast<float4*>(SW + umma::swz(r - 64, c0 + cc + u, 64)) =
                            umma::tf32r(make_float4(-v[u], -v[u + 1], -v[u + 2], -v[u + 3]));
                }
            }
            if (r < 64) rpart[half * 128 + r] = r < L ? eg[r] * part : 0.f;
        }
        // D2 (M = 64): rows rl and rl + 8 of this thread's fragment
        {
            float v[32];
            umma::tmem_ld64_m64(umma::tmem_at(tmem + 128, c0), v);
            const int rl = umma::frag_row_lo(), rh = rl + 8;
            float pl = 0.f, ph = 0.f;
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int c = c0 + 8 * k + 2 * (lane & 3);
                const float2 kl = *reinterpret_cast<const float2*>(Kr + umma::swz(rl, c, 64));
                const float2 kh2 = *reinterpret_cast<const float2*>(Kr + umma::swz(rh, c, 64));
                pl += v[4 * k] * kl.x + v[4 * k + 1] * kl.y;
                ph += v[4 * k + 2] * kh2.x + v[4 * k + 3] * kh2.y;
            }
            pl += __shfl_xor_sync(0xffffffffu, pl, 1);
            pl += __shfl_xor_sync(0xffffffffu, pl, 2);
            ph += __shfl_xor_sync(0xffffffffu, ph, 1);
            ph += __shfl_xor_sync(0xffffffffu, ph, 2);
            {   // the dK part fk dK~ into the group's sum; staged at the last v-head
                float a[32];
                if (first) {
#pragma unroll
                    for (int u = 0; u < 32; u++) a[u] = 0.f;
                } else {
                    umma::tmem_ld64_m64(umma::tmem_at(tKacc, c0), a);
                }
                const float fl = fk[rl], fh = fk[rh];
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    a[4 * k] += fl * v[4 * k];
                    a[4 * k + 1] += fl * v[4 * k + 1];
                    a[4 * k + 2] += fh * v[4 * k + 2];
                    a[4 * k + 3] += fh * v[4 * k + 3];
                }
                if (last) umma::frag_to_sw(SK, a, c0, 1.f, 1.f);
                else umma::tmem_st64_m64(umma::tmem_at(tKacc, c0), a);
            }
            if ((lane & 3) == 0) {
                rpart[half * 128 + 64 + rl] = rl < L ? fk[rl] * pl : 0.f;
                rpart[half * 128 + 64 + rh] = rh < L ? fk[rh] * ph : 0.f;
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        // dW per v-head; the dQ, dK parts once per k-head, at its last v-head
        if (L == 64) {
            if (tid == 0) {
                umma::tma_store_rows(&maps.dW, h, ci.start, SW);
                if (last) {
                    umma::tma_store_rows(&maps.dQv, kh, ci.start, SQ);
                    umma::tma_store_rows(&maps.dKv, kh, ci.start, SK);
                }
                umma::bulk_commit();
            }
        } else {
            const int64_t off = ((int64_t)ci.start * hv + h) * kD, st = (int64_t)hv * kD;
            umma::store_rows_sw(w.dW + off, st, SW, L);
            if (last) {
                const int64_t ok2 = ((int64_t)ci.start * hk + kh) * kD, sk = (int64_t)hk * kD;
                umma::store_rows_sw(w.dQv + ok2, sk, SQ, L);
                umma::store_rows_sw(w.dKv + ok2, sk, SK, L);
            }
        }
        if (tid < 64 && tid < L) {
            float g = (rpart[tid] + rpart[128 + tid]) - (rpart[64 + tid] + rpart[192 + tid]);
            if (tid == L - 1) {
                float zs = 0.f, dd = 0.f;
                for (int j = 0; j < L; j++) zs += rpart[64 + j] + rpart[192 + j];
                for (int i = 0; i < 8; i++) dd += red[i];
                g += zs + expf(gam[L - 1]) * dd;
            }
            w.dgam[(int64_t)(ci.start + tid) * hv + h] = g;
        }
        __syncthreads();   // staged tiles, Q / K, sums: read (or handed to the stores)
        if (!next) break;
        if (tid == 0) {
            umma::bulk_wait_read();   // the tile stores have read [dO; dU] and U space
            issue_main(cn, tn);
        }
        g_cur = g_next;
        ci = cn;
        t = tn;
    }
    if (tid == 0) umma::bulk_wait_read();   // the tile stores have read shared memory
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 512);
    if (!ok && tid == 0) atomicExch(w.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ B3b: P / dP terms
// Persistent: up to one CTA per SM (the last CTAs of the combined launch
// below), each claiming (chunk, k-head) groups from a counter (chunk = NT - 1 -
// g / H_k, k-head = g % H_k: last chunk first, like the reverse state pass
// running beside them), so CTAs that start late -- on the SMs the reverse state
// pass holds -- simply take fewer groups.  A group is the G = H_v / H_k v-heads
// that share the k-head's q and k, handled one after another.  Per group, tcgen05:
//   D_qk = Q K^T                                         (once: q, k are shared)
//   per v-head h:  D_dou = dO_h U_h^T;  dPm_h = D_dou (.) Gam_h (.) [i>=j];
//                  R = dPm_h (.) D_qk:  dgam_h,i += sum_j R_ij, dgam_h,j -= sum_i R_ij
//   dPs = sum_h dPm_h (fp32, in registers; rounded once)
//   D_dq = dPs K,  D_dk = dPs^T Q                        (64 x 128 each, once)
// -- the group's whole dQ / dK share from these terms, written once per k-head
// (sum_h dPm_h K = (sum_h dPm_h) K because K is the same for every h).  Shared
// memory: Q, K swizzled and MN-major (the latter the B operands of the products
// over tokens), 32 KB each; one v-head's dO, U swizzled, 32 KB each; dPs in both
// orientations 16 KB each.  The next group's swizzled Q, K are requested once
// D_qk is done, its MN-major ones once D_dq / D_dk are; the next v-head's dO, U
// (of this group or the next) once the current D_dou is done.  D_dq and D_dk go
// from tensor memory straight to global memory while the next group's first
// products run.  Tensor memory: D_dq / D_dk in columns 0-255, D_qk and D_dou in
// 256-383 (512 allocated), once.
constexpr int kDpFloats = 6 * 64 * 128 + 2 * 64 * 64;
constexpr size_t kDpSmem = sizeof(float) * (kDpFloats + 4 * 64 + 2 * 64 + 64) + 6 * 8 + 16 + 1024;

__device__ __forceinline__ void bwd_dp_cta(const TileMaps& maps, int hk, int hv, int NT,
                                           const FwdSaved& sv, const BwdScratch& w) {
    // 256 threads (warps 0-7) take part; the launch's other warps leave at once
    if (threadIdx.x >= 256) return;
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* Qs = sm;                    // [64][128] swizzled
    float* Ks = Qs + 64 * 128;         // [64][128] swizzled
    float* dOs = Ks + 64 * 128;        // [64][128] swizzled   (arrives rounded)
    float* Us = dOs + 64 * 128;        // [64][128] swizzled   (arrives rounded)
    float* Qm = Us + 64 * 128;         // [64 (i)][128] MN-major
    float* Km = Qm + 64 * 128;         // [64 (j)][128] MN-major
    float* dPR = Km + 64 * 128;        // [64 (i)][64 (j)] K-major
    float* dPC = dPR + 64 * 64;        // [64 (j)][64 (i)] K-major
    float* colp = dPC + 64 * 64;       // [4 row windows][64] column sums of R
    float* rpart = colp + 4 * 64;      // [2][64] row sums of R
    float* gam = rpart + 2 * 64;
    uint64_t* mQ = reinterpret_cast<uint64_t*>(gam + 64);   // swizzled Q, K
    uint64_t* mB = mQ + 1;             // MN-major Q, K
    uint64_t* mO = mB + 1;             // dO, U of one v-head
    uint64_t* mM = mO + 1;             // MMA (G + 2 commits per group)
    int32_t* claim = reinterpret_cast<int32_t*>(mM + 1);   // [3] claimed groups, slot gi % 3
    uint32_t* tslot = reinterpret_cast<uint32_t*>(claim + 3);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = hv / hk, ngroups = NT * hk;
    auto entry = [&](int g) { return sv.chunks[NT - 1 - g / hk]; };
    auto issue_q = [&](const ChunkInfo& c, int g) {   // one thread
        const int kh = g % hk;
        umma::mbar_expect_tx(mQ, 2 * 64 * 128 * 4);
        umma::tma_rows(Qs, 64, &maps.q, kh, c.start, mQ);
        umma::tma_rows(Ks, 64, &maps.k, kh, c.start, mQ);
    };
    auto issue_b = [&](const ChunkInfo& c, int g) {   // one thread
        const int kh = g % hk;
        umma::mbar_expect_tx(mB, 2 * 64 * 128 * 4);
        umma::tma_rows(Qm, 64, &maps.q_mn, kh, c.start, mB);
        umma::tma_rows(Km, 64, &maps.k_mn, kh, c.start, mB);
    };
    auto issue_o = [&](const ChunkInfo& c, int h) {   // one thread
        umma::mbar_expect_tx(mO, 2 * 64 * 128 * 4);
        umma::tma_rows(dOs, 64, &maps.dO, h, c.start, mO);
        umma::tma_rows(Us, 64, &maps.U, h, c.start, mO);
    };
    if (tid == 0) {
        umma::mbar_init(mQ, 1);
        umma::mbar_init(mB, 1);
        umma::mbar_init(mO, 1);
        umma::mbar_init(mM, 1);
        const int g0 = atomicAdd(w.dp_next, 1);
        claim[0] = g0;
        claim[1] = atomicAdd(w.dp_next, 1);
        if (g0 < ngroups) {
            const ChunkInfo c0 = entry(g0);
            if (c0.len > 0) {
                issue_q(c0, g0);
                issue_b(c0, g0);
                issue_o(c0, (g0 % hk) * G);
            }
        }
    }
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    umma::named_sync(1, 256);
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tDQ = tmem, tDK = tmem + 128, tQK = tmem + 256, tDOU = tmem + 320;
    const int win = warp & 3, half = warp >> 2;
    const int rl = umma::frag_row_lo(), cf = umma::frag_col();
    // D_dq, D_dk rows rl, rl + 8 (those inside the chunk) of the group at token
    // `start`, k-head khp, straight from tensor memory to the per-k-head partials
    auto put_group = [&](int64_t start, int khp, int Lp) {
        const int64_t o_lo = ((start + rl) * hk + khp) * kD;
        const int64_t o_hi = o_lo + (int64_t)8 * hk * kD;
        auto put = [&](float* dst, uint32_t tcol) {
            float v[32];
            umma::tmem_ld64_m64(umma::tmem_at(tcol, half * 64), v);
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const int c = half * 64 + 8 * k + cf;
                if (rl < Lp)
                    *reinterpret_cast<float2*>(dst + o_lo + c) = make_float2(v[4 * k], v[4 * k + 1]);
                if (rl + 8 < Lp)
                    *reinterpret_cast<float2*>(dst + o_hi + c) = make_float2(v[4 * k + 2], v[4 * k + 3]);
            }
        };
        put(w.dQv2, tDQ);
        put(w.dKv2, tDK);
    };
    // Groups are claimed two ahead (the claim for group iteration gi + 2 is made
    // during iteration gi), so a group's chunk entry is loaded an iteration before
    // its operands are requested; a v-head's gate values are loaded a v-head
    // before they are used.
    int g = claim[0], gn = claim[1];
    ChunkInfo ci = g < ngroups ? entry(g) : ChunkInfo{0, 0, 0, 0};
    ChunkInfo cn = gn < ngroups ? entry(gn) : ci;
    float g_cur = 0.f;
    if (tid < 64 && g < ngroups) g_cur = sv.gam[(int64_t)((g % hk) * G) * sv.T + ci.start + min(tid, ci.len - 1)];
    bool ok = true;
    int64_t p_start = -1;   // the previous group, whose D_dq / D_dk are still to go out
    int p_kh = 0, p_L = 0;
    uint32_t nm = 0;        // MMA commits waited so far (mM parity)
    uint32_t no = 0;        // v-head loads waited so far (mO parity)
    for (int gi = 0; g < ngroups; gi++) {
        const int kh = g % hk, L = ci.len;
        if (L == 0) break;   // the device check of cu_seqlens failed: every chunk is empty
        ok = umma::named_sync_and(1, 256, umma::mbar_wait(mQ, gi & 1));   // Q, K
        if (!ok) break;
        if (L < 64) {   // tail rows belong to the next sequence
            umma::zero_tail_rows<256>(Qs, 64, 0, L);
            umma::zero_tail_rows<256>(Ks, 64, 0, L);
            umma::named_sync(1, 256);
        }
        if (!sv.qkv_tf32) umma::tf32r_inplace<256>(Qs, 2 * 64 * 128);   // Q, K
        umma::fence_smem_to_async();
        umma::named_sync(1, 256);
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tQK, umma::swt(Qs, 64), umma::swt(Ks, 64), 64, 64, 128, false);
            umma::commit(mM);
            claim[(gi + 2) % 3] = atomicAdd(w.dp_next, 1);   // the group after the next
        }
        if (p_start >= 0) put_group(p_start, p_kh, p_L);   // while D_qk runs
        umma::fence_before_sync();   // (those tensor-memory reads)
        ok = umma::named_sync_and(1, 256, umma::mbar_wait(mM, nm & 1));   // the claim is visible too
        nm++;
        umma::fence_after_sync();
        if (!ok) break;
        const int g2 = claim[(gi + 2) % 3];
        ChunkInfo c2 = cn;   // used an iteration later
        if (g2 < ngroups) c2 = entry(g2);
        const bool next = gn < ngroups && cn.len > 0;
        if (tid == 0 && next) issue_q(cn, gn);   // the swizzled Q, K are consumed
        float qk[16];
        umma::tmem_ld_m64<4>(umma::tmem_at(tQK, half * 32), qk);
        float ps[16];   // sum over the group's v-heads of dPm, this thread's fragment
#pragma unroll
        for (int q = 0; q < 16; q++) ps[q] = 0.f;
        for (int j = 0; j < G && ok; j++) {
            const int h = kh * G + j;
            // the next v-head's gate values (this group's, else the next group's first)
            float g_next = 0.f;
            if (tid < 64) {
                if (j + 1 < G)
                    g_next = sv.gam[(int64_t)(h + 1) * sv.T + ci.start + min(tid, L - 1)];
                else if (next)
                    g_next = sv.gam[(int64_t)((gn % hk) * G) * sv.T + cn.start + min(tid, cn.len - 1)];
            }
            if (tid < 64) gam[tid] = g_cur;
            ok = umma::named_sync_and(1, 256, umma::mbar_wait(mO, no & 1));   // dO, U; gam visible
            no++;
            if (!ok) break;
            if (L < 64) {
                umma::zero_tail_rows<256>(dOs, 64, 0, L);
                umma::zero_tail_rows<256>(Us, 64, 0, L);
                umma::fence_smem_to_async();
                umma::named_sync(1, 256);
            }
            umma::fence_after_sync();
            if (tid == 0) {
                umma::mma(tDOU, umma::swt(dOs, 64), umma::swt(Us, 64), 64, 64, 128, false);
                umma::commit(mM);
            }
            // while the product runs: the decay factors e^{gam_r - gam_j} [j <= r] of
            // this thread's fragment
            float dec[16];
#pragma unroll
            for (int hr = 0; hr < 2; hr++) {
                const int r = rl + 8 * hr;
                const float gr = gam[r];
#pragma unroll
                for (int k = 0; k < 4; k++)
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int jj = half * 32 + 8 * k + cf + e;
                        dec[4 * k + 2 * hr + e] = jj <= r ? expf(gr - gam[jj]) : 0.f;
                    }
            }
            ok = umma::named_sync_and(1, 256, umma::mbar_wait(mM, nm & 1));
            nm++;
            umma::fence_after_sync();
            if (!ok) break;
            if (tid == 0) {   // dO, U consumed: the next v-head's
                if (j + 1 < G) issue_o(ci, h + 1);
                else if (next) issue_o(cn, (gn % hk) * G);
            }
            {   // dPm_h, R row / column sums by shuffles; dPm_h into the group sum
                float du[16];
                umma::tmem_ld_m64<4>(umma::tmem_at(tDOU, half * 32), du);
                float rs[2] = {0.f, 0.f}, cs[4][2];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    cs[k][0] = cs[k][1] = 0.f;
#pragma unroll
                    for (int hr = 0; hr < 2; hr++)
#pragma unroll
                        for (int e = 0; e < 2; e++) {
                            const int q = 4 * k + 2 * hr + e;
                            const float x = du[q] * dec[q];
                            const float R = x * qk[q];
                            rs[hr] += R;
                            cs[k][e] += R;
                            ps[q] += x;
                        }
                }
                rs[0] = umma::row_quad_sum(rs[0]);
                rs[1] = umma::row_quad_sum(rs[1]);
                if ((lane & 3) == 0) {
                    rpart[half * 64 + rl] = rs[0];
                    rpart[half * 64 + rl + 8] = rs[1];
                }
#pragma unroll
                for (int k = 0; k < 4; k++)
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const float c = umma::col_oct_sum(cs[k][e]);
                        if (lane < 4) colp[win * 64 + half * 32 + 8 * k + 2 * lane + e] = c;
                    }
            }
            umma::fence_before_sync();
            umma::named_sync(1, 256);   // R sums written; D_dou read
            if (tid < 64 && tid < L) {   // dgam from R: row sums minus column sums (fixed order)
                const float cs = (colp[tid] + colp[64 + tid]) + (colp[128 + tid] + colp[192 + tid]);
                w.dgam2[(int64_t)(ci.start + tid) * hv + h] = (rpart[tid] + rpart[64 + tid]) - cs;
            }
            umma::named_sync(1, 256);   // R sums read before the next v-head's
            g_cur = g_next;
        }
        if (!ok) break;
        {   // dPs rounded, in both orientations
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int jj = half * 32 + 8 * k + cf;
#pragma unroll
                for (int hr = 0; hr < 2; hr++) {
                    const int r = rl + 8 * hr;
                    const float d0 = umma::tf32r(ps[4 * k + 2 * hr]), d1 = umma::tf32r(ps[4 * k + 2 * hr + 1]);
                    dPC[umma::kidx(jj, r, 64)] = d0;
                    dPC[umma::kidx(jj + 1, r, 64)] = d1;
                    *reinterpret_cast<float2*>(dPR + umma::kidx(r, jj, 64)) = make_float2(d0, d1);
                }
            }
        }
        umma::fence_smem_to_async();
        ok = umma::named_sync_and(1, 256, umma::mbar_wait(mB, gi & 1));   // MN-major Q, K
        if (!ok) break;
        if (L < 64) {
            umma::zero_tail_rows<256>(Qm, 64, 0, L);
            umma::zero_tail_rows<256>(Km, 64, 0, L);
            umma::named_sync(1, 256);
        }
        if (!sv.qkv_tf32) umma::tf32r_inplace<256>(Qm, 2 * 64 * 128);
        umma::fence_smem_to_async();
        umma::named_sync(1, 256);
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tDQ, umma::kmaj(dPR, 64), umma::mnt(Km), 64, 128, 64, false);
            umma::mma(tDK, umma::kmaj(dPC, 64), umma::mnt(Qm), 64, 128, 64, false);
            umma::commit(mM);
        }
        ok = umma::named_sync_and(1, 256, umma::mbar_wait(mM, nm & 1));
        nm++;
        umma::fence_after_sync();
        if (!ok) break;
        if (tid == 0 && next) issue_b(cn, gn);   // the MN-major operands are consumed
        p_start = ci.start;   // D_dq, D_dk go out at the next group's first product
        p_kh = kh;
        p_L = L;
        umma::fence_before_sync();
        umma::named_sync(1, 256);   // tensor memory read before the next group's products reuse it
        g = gn;
        gn = g2;
        ci = cn;
        cn = c2;
    }
    if (ok && p_start >= 0) put_group(p_start, p_kh, p_L);   // the last group
    umma::fence_before_sync();
    umma::named_sync(1, 256);
    if (warp == 0) umma::tmem_free(tmem, 512);
    if (!ok && tid == 0) atomicExch(w.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ B2 + B3b in one launch
// The reverse state pass holds one CTA per (slice, head, sequence) for its whole
// sequence; for a few long sequences that leaves most SMs free.  One grid of
// 320-thread CTAs: CTAs 0 .. n_state - 1 run the state pass (they come first,
// so they are resident from the start), the rest run the P / dP tiles
// (independent of the state pass, on 256 of the threads) and fill the other
// SMs, then those the state pass frees.  No CTA waits on another.
constexpr size_t kStateDpSmem = kB2Smem > kDpSmem ? kB2Smem : kDpSmem;

__global__ void __launch_bounds__(kStateThreadsB, 1)
bwd_state_dp_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, int NT, int n_state,
                    const float* dS_final, float* dS_init, FwdSaved sv, BwdScratch w) {
    const int b = blockIdx.x;
    if (b < n_state) {
        const int ns = kD / kSl;
        bwd_state_cta(maps, b % ns, (b / ns) % hv, b / (ns * hv), hk, hv, dS_final, dS_init, sv, w);
    } else {
        bwd_dp_cta(maps, hk, hv, NT, sv, w);
    }
}

// ------------------------------------------------------------------ B3c: WY terms and gates
// Persistent: one CTA per SM walks (chunk, k-head) groups g = blockIdx.x,
// + gridDim.x, ... (chunk = g / Hk, k-head = g % Hk), each as the tiles of its
// G = Hv / Hk v-heads in turn (neighbouring SMs hold neighbouring groups of one
// chunk, so the tiles they read come from DRAM once).  Per tile, tcgen05, with T
// saved by the forward:
//   D_kk = K K^T, D_dt1 = dW K^T, D_dt2 = dU V^T          (64 x 64)
//   D_tw = T^T [dW | dU]                                  (64 x 256, one product)
//   dT = D_dt1 diag(beta e^gam) + D_dt2 diag(beta)
//   dV = diag(beta) T^T dU ; dK += diag(beta e^gam) T^T dW
//   dbeta_j += e^{gam_j} (T^T dW)_j . K_j + (T^T dU)_j . V_j ; dgam_j += beta_j e^{gam_j} (..)
//   Y^T = T dT^T ; dA = -T^T Y (strictly lower) ; dKK = dA (.) beta_j Gam
//   dbeta_j += sum_m dA (.) GamKK ; dgam_j += beta_j (..) ; dgam_m -= sum_j beta_j (..)
//   dK += (dKK + dKK^T) K   (one product: the two triangles are disjoint)
// then dg = reverse in-chunk cumsum of the total dgam, and the gate gradients.
// The dK part is summed over the group's v-heads in registers, in order, and
// written once per k-head at the group's last v-head.
// The next tile's operands are requested in two groups as their space frees
// up: dW, dU (K-major) and T^T once dA is formed, dW, dU (MN-major), V and K
// once the last product is done (dK goes to global memory straight from the
// fragments); all of them are prefetched into L2 a tile ahead, and its gate
// inputs are loaded into registers meanwhile.  Tensor memory allocated once.
constexpr int kWyFloats = 4 * 64 * 128 + 256 * 64 + 64 * 64;   // stage-1 operands
constexpr size_t kWySmem = sizeof(float) * (kWyFloats + 10 * 64 + 2 * 64 + 16) + 64 + 1024;

template <class IO>
__global__ void __launch_bounds__(256, 1)
bwd_wy_kernel(const __grid_constant__ TileMaps maps, const IO* __restrict__ av,
              const IO* __restrict__ bv, const float* __restrict__ A_log,
              const float* __restrict__ dt_bias, int hk, int hv, int NT, float* __restrict__ dqkv,
              IO* __restrict__ da, IO* __restrict__ db, float* __restrict__ gate_part, FwdSaved sv,
              BwdScratch w) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    // stage 1: K, V, dW, dU swizzled (TMA)
    float* Ks = sm;                    // [64][128] swizzled
    float* Vs = Ks + 64 * 128;
    float* dWs = Vs + 64 * 128;
    float* dUs = dWs + 64 * 128;
    float* dWm = dUs + 64 * 128;       // [64 (j)][128 (b)] MN-major dW (arrives rounded)
    float* dUm = dWm + 64 * 128;       // [64 (j)][128 (a)] MN-major dU (arrives rounded)
    float* TC = dUm + 64 * 128;        // [64 (j)][64 (i)] K-major T^T
    // stage 2 overlays dW, dU and [dW^T ; dU^T] once the first products are
    // complete; K and V stay for the epilogue's dot products (R later over V)
    float* GKK = dWs;                  // [64][64] K-major Gam (.) KK (strict lower)
    float* DTR = GKK + 64 * 64;        // [64 (i)][64 (j)] K-major dT
    float* TR = DTR + 64 * 64;         // [64 (m)][64 (j)] K-major T
    float* YT = TR + 64 * 64;          // [64 (m)][64 (i)] K-major Y^T
    float* dKS = YT + 64 * 64;         // [64 (j)][64 (m)] K-major dKK + dKK^T (disjoint triangles)
    float* Km = dKS + 2 * 64 * 64;     // [64 (m)][128 (b)] MN-major K (over dU_mn, after stage 1)
    float* Rm = Vs;                    // [64][65] row-major
    float* gam = TC + 64 * 64;
    float* eg = gam + 64;
    float* bet = eg + 64;
    float* be = bet + 64;
    float* dgs = be + 64;
    float* dbs = dgs + 64;
    float* sc = dbs + 64;
    float* rk = sc + 64;
    float* red = rk + 64;              // [64]
    float* rp = red + 64;              // [2][64]
    uint64_t* mbar = reinterpret_cast<uint64_t*>(rp + 128 + 16);   // MMA
    uint64_t* mW = mbar + 1;           // dW, dU (K-major), T^T
    uint64_t* mM = mW + 1;             // dW, dU (MN-major), V
    uint64_t* mK = mM + 1;             // K
    uint64_t* mT = mK + 1;             // stage 2: T, K (MN-major)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mT + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = (2 * hk + hv) * kD;
    const int G = hv / hk, ngroups = NT * hk;
    // a CTA walks (chunk, k-head) groups g = blockIdx.x, + gridDim.x, ..., each as
    // its G v-head tiles t = chunk H_v + k-head G + j in turn; next_tile is the
    // tile after t in that walk (-1: none)
    auto first_tile = [&](int g) { return (g / hk) * hv + (g % hk) * G; };
    auto next_tile = [&](int tt) {
        if (tt < 0) return -1;
        if (tt % G != G - 1) return tt + 1;
        const int gn = (tt / hv) * hk + (tt % hv) / G + (int)gridDim.x;
        return gn < ngroups ? first_tile(gn) : -1;
    };
    if ((int)blockIdx.x >= ngroups) return;
    int t = first_tile(blockIdx.x);
    ChunkInfo ci = sv.chunks[t / hv];
    if (ci.len == 0) return;   // the device check of cu_seqlens failed: every chunk is empty
    auto Tg_of = [&](int tile) {   // T, then T^T, written by the forward
        return sv.Tm + ((int64_t)(tile / hv) * hv + tile % hv) * 2 * 64 * 64;
    };
    auto issue_w = [&](const ChunkInfo& c, int tile) {   // one thread
        const int h = tile % hv;
        umma::mbar_expect_tx(mW, 2 * 64 * 128 * 4 + 64 * 64 * 4);
        umma::tma_rows(dWs, 64, &maps.dW, h, c.start, mW);
        umma::tma_rows(dUs, 64, &maps.dU, h, c.start, mW);
        umma::bulk_load(TC, Tg_of(tile) + 64 * 64, 64 * 64 * 4, mW);
    };
    auto issue_m = [&](const ChunkInfo& c, int tile) {   // one thread
        const int h = tile % hv;
        umma::mbar_expect_tx(mM, 3 * 64 * 128 * 4);
        umma::tma_rows(dWm, 64, &maps.dW_mn, h, c.start, mM);
        umma::tma_rows(dUm, 64, &maps.dU_mn, h, c.start, mM);
        umma::tma_rows(Vs, 64, &maps.v, h, c.start, mM);
    };
    auto issue_k = [&](const ChunkInfo& c, int tile) {   // one thread
        const int kh = tile % hv / (hv / hk);
        umma::mbar_expect_tx(mK, 64 * 128 * 4);
        umma::tma_rows(Ks, 64, &maps.k, kh, c.start, mK);
    };
    // gate inputs of a tile for thread tid < 64: gam, beta, a + dt_bias and the
    // dgam terms of the other kernels (used at the very end)
    // (kept as loaded: the values are first used in the tile's own iteration, so
    // the loads stay in flight meanwhile)
    struct Gates { float g, b; IO a; float dg1, dg2; };
    auto gates_of = [&](const ChunkInfo& c, int tile) {
        Gates q{0.f, 0.f, from_f<IO>(0.f), 0.f, 0.f};
        if (tid < 64) {
            const int h = tile % hv;
            q.g = sv.gam[(int64_t)h * sv.T + c.start + min(tid, c.len - 1)];
            if (tid < c.len) {
                const int64_t tok = c.start + tid;
                q.b = sv.beta[(int64_t)h * sv.T + tok];
                q.a = av[tok * hv + h];
                q.dg1 = w.dgam[tok * hv + h];
                q.dg2 = w.dgam2[tok * hv + h];
            }
        }
        return q;
    };
    if (tid == 0) {
        for (int k = 0; k < 5; k++) umma::mbar_init(&mbar[k], 1);
        issue_w(ci, t);
        issue_m(ci, t);
        issue_k(ci, t);
    }
    Gates gcur = gates_of(ci, t);
    // chunk entries are loaded a tile before they are needed: cn (the next tile's)
    // is at hand at the top of an iteration, c2 (the one after) is requested there
    ChunkInfo cn = next_tile(t) >= 0 ? sv.chunks[next_tile(t) / hv] : ci;
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    // columns: KK 0-63 (later T^T Y), dT1 64-127 and dT2 128-191 (later Y^T, then the
    // 128-column dKK product), T^T [dW | dU] 256-511 (read again at the very end)
    const uint32_t tKK = tmem, tDT1 = tmem + 64, tDT2 = tmem + 128, tX = tmem + 64,
                   tTW = tmem + 256;
    const int win = warp & 3, half = warp >> 2;
    const int rl = umma::frag_row_lo(), cf = umma::frag_col();   // fragment rows rl, rl + 8
    bool ok = true;
    float kacc[32];   // the group's dK part, summed over its v-heads in order (fragment)
    for (int it = 0;; it++) {
        const int h = t % hv, kh = h / G, L = ci.len, chunk = t / hv;
        const bool first = h % G == 0, last = h % G == G - 1;
        const int tn = next_tile(t), t2 = next_tile(tn);
        ChunkInfo c2 = cn;
        if (t2 >= 0) c2 = sv.chunks[t2 / hv];
        auto row = [&](int r) { return (int64_t)ci.start + min(r, L - 1); };
        const float alog = A_log[h], dtb = dt_bias[h];   // first used at the end of the tile
        if (tid == 32 && tn >= 0 && cn.len > 0) {   // the next tile's inputs into L2
            const int hn = tn % hv;
            umma::tma_prefetch_rows(&maps.dW, hn, cn.start);
            umma::tma_prefetch_rows(&maps.dU, hn, cn.start);
            umma::tma_prefetch_rows(&maps.v, hn, cn.start);
            umma::tma_prefetch_rows(&maps.k, hn / (hv / hk), cn.start);
            umma::bulk_prefetch(Tg_of(tn), 2 * 64 * 64 * 4);
        }
        if (tid < 64) {
            gam[tid] = gcur.g;
            bet[tid] = gcur.b;
            dgs[tid] = 0.f;
            dbs[tid] = 0.f;
            eg[tid] = tid < L ? expf(gcur.g) : 0.f;
            be[tid] = gcur.b * (tid < L ? expf(gcur.g) : 0.f);
        }
        ok = umma::mbar_wait(mW, it & 1) && umma::mbar_wait(mM, it & 1);
        ok = __syncthreads_and(ok && umma::mbar_wait(mK, it & 1));   // gates visible
        if (!ok) break;
        if (L < 64) {   // tail rows belong to the next sequence
            umma::zero_tail_rows(Ks, 64, 0, L);
            umma::zero_tail_rows(Vs, 64, 0, L);
            umma::zero_tail_rows(dWs, 64, 0, L);
            umma::zero_tail_rows(dUs, 64, 0, L);
            umma::zero_tail_rows(dWm, 64, 0, L);
            umma::zero_tail_rows(dUm, 64, 0, L);
            __syncthreads();
        }
        if (!sv.qkv_tf32) umma::tf32r_inplace(Ks, 2 * 64 * 128);   // K, V (dW, dU and T^T arrive rounded)
        __syncthreads();
        umma::fence_smem_to_async();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tKK, umma::swt(Ks, 64), umma::swt(Ks, 64), 64, 64, 128, false);
            umma::mma(tDT1, umma::swt(dWs, 64), umma::swt(Ks, 64), 64, 64, 128, false);
            umma::mma(tDT2, umma::swt(dUs, 64), umma::swt(Vs, 64), 64, 64, 128, false);
            // T^T [dW | dU]: the two MN-major tiles are adjacent, one N = 256 product
            umma::mma(tTW, umma::kmaj(TC, 64), umma::mnt(dWm), 64, 256, 64, false);
            umma::commit(mbar);
        }
        // while the products run: the decay factors e^{gam_r - gam_j} [j < r] of this
        // thread's fragment of the 64 x 64 products (Gam (.) KK and dKK use the same pairs)
        float dec[16];
#pragma unroll
        for (int hr = 0; hr < 2; hr++) {
            const int r = rl + 8 * hr;
            const float gr = gam[r];
#pragma unroll
            for (int k = 0; k < 4; k++)
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const int j = half * 32 + 8 * k + cf + e;
                    dec[4 * k + 2 * hr + e] = j < r ? expf(gr - gam[j]) : 0.f;
                }
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 0));
        umma::fence_after_sync();
        if (!ok) break;
        // dW, dU (both layouts) are consumed: fetch T and K as an MN-major tile for stage 2
        if (tid == 0) {
            umma::mbar_expect_tx(mT, 64 * 64 * 4 + 64 * 128 * 4);
            umma::bulk_load(TR, Tg_of(t), 64 * 64 * 4, mT);
            umma::tma_rows(Km, 64, &maps.k_mn, kh, ci.start, mT);
        }
        {
            {   // Gam (.) KK and dT from the 64-column products, 32 columns per warp
                float kk[16], t1[16], t2[16];
                umma::tmem_ld_m64<4>(umma::tmem_at(tKK, half * 32), kk);
                umma::tmem_ld_m64<4>(umma::tmem_at(tDT1, half * 32), t1);
                umma::tmem_ld_m64<4>(umma::tmem_at(tDT2, half * 32), t2);
#pragma unroll
                for (int hr = 0; hr < 2; hr++) {
                    const int r = rl + 8 * hr;
#pragma unroll
                    for (int k = 0; k < 4; k++) {
                        const int j = half * 32 + 8 * k + cf, q = 4 * k + 2 * hr;
                        const float g0 = dec[q] * kk[q];
                        const float g1 = dec[q + 1] * kk[q + 1];
                        const float d0 = t1[q] * be[j] + t2[q] * bet[j];
                        const float d1 = t1[q + 1] * be[j + 1] + t2[q + 1] * bet[j + 1];
                        *reinterpret_cast<float2*>(GKK + umma::kidx(r, j, 64)) = make_float2(g0, g1);
                        *reinterpret_cast<float2*>(DTR + umma::kidx(r, j, 64)) =
                            make_float2(umma::tf32r(d0), umma::tf32r(d1));
                    }
                }
            }
            {   // T^T dW (half 0) and T^T dU (half 1): dV, dbeta / dgam dot products
                float rs[2] = {0.f, 0.f};
                float* dvb = dqkv + (int64_t)2 * hk * kD + h * kD;
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 64) {
                    float v[32];
                    umma::tmem_ld64_m64(umma::tmem_at(tTW, half * 128 + c0), v);
                    const float* X = half == 0 ? Ks : Vs;
#pragma unroll
                    for (int hr = 0; hr < 2; hr++) {
                        const int r = rl + 8 * hr;
#pragma unroll
                        for (int k = 0; k < 8; k++) {
                            const int c = c0 + 8 * k + cf, q = 4 * k + 2 * hr;
                            const float2 x2 = *reinterpret_cast<const float2*>(X + umma::swz(r, c, 64));
                            rs[hr] += v[q] * x2.x + v[q + 1] * x2.y;
                            if (half == 1 && r < L)
                                *reinterpret_cast<float2*>(dvb + row(r) * C + c) =
                                    make_float2(bet[r] * v[q], bet[r] * v[q + 1]);
                        }
                    }
                }
                rs[0] = umma::row_quad_sum(rs[0]);
                rs[1] = umma::row_quad_sum(rs[1]);
                if ((lane & 3) == 0) {
                    rp[half * 64 + rl] = rl < L ? rs[0] : 0.f;
                    rp[half * 64 + rl + 8] = rl + 8 < L ? rs[1] : 0.f;
                }
            }
        }
        __syncthreads();
        if (tid < 64) {
            dbs[tid] += eg[tid] * rp[tid] + rp[64 + tid];
            dgs[tid] += be[tid] * rp[tid];
        }
        const bool next = tn >= 0 && cn.len > 0;
        const Gates gnext = next ? gates_of(cn, tn) : Gates{0.f, 0.f, from_f<IO>(0.f), 0.f, 0.f};
        // stage 2 operands: T arrived as a K-major tile, K as an MN-major tile
        ok = __syncthreads_and(umma::mbar_wait(mT, it & 1));
        if (!ok) break;
        if (L < 64) {
            umma::zero_tail_rows(Km, 64, 0, L);
            __syncthreads();
        }
        if (!sv.qkv_tf32) umma::tf32r_inplace(Km, 64 * 128);
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma_tf32(tX, TR, 64, DTR, 64, 64, 64, 64, false);     // Y^T = T dT^T
            umma::commit(mbar);
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 1));
        umma::fence_after_sync();
        if (!ok) break;
        {   // Y^T, 32 columns per warp, all lanes
            float v[16];
            umma::tmem_ld_m64<4>(umma::tmem_at(tX, half * 32), v);
#pragma unroll
            for (int hr = 0; hr < 2; hr++)
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int c = half * 32 + 8 * k + cf, q = 4 * k + 2 * hr;
                    *reinterpret_cast<float2*>(YT + umma::kidx(rl + 8 * hr, c, 64)) =
                        make_float2(umma::tf32r(v[q]), umma::tf32r(v[q + 1]));
                }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma_tf32(tKK, TC, 64, YT, 64, 64, 64, 64, false);     // T^T Y  (= -dA)
            umma::commit(mbar);
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 0));
        umma::fence_after_sync();
        if (!ok) break;
        float* colp = Rm;                  // [4 row windows][64] column sums of beta_r x
        {   // dA = -(T^T Y) strictly lower; 32 columns per warp, all lanes
            float v[16];
            umma::tmem_ld_m64<4>(umma::tmem_at(tKK, half * 32), v);
            float rs[2] = {0.f, 0.f}, cs[4][2];
#pragma unroll
            for (int k = 0; k < 4; k++) {
                const int m = half * 32 + 8 * k + cf;
                cs[k][0] = cs[k][1] = 0.f;
#pragma unroll
                for (int hr = 0; hr < 2; hr++) {
                    const int r = rl + 8 * hr;
                    const float br = bet[r];
                    const float2 gk = *reinterpret_cast<const float2*>(GKK + umma::kidx(r, m, 64));
#pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const float dA = m + e < r ? -v[4 * k + 2 * hr + e] : 0.f;
                        const float x = dA * (e == 0 ? gk.x : gk.y);
                        rs[hr] += x;
                        cs[k][e] += br * x;
                        // dKK is strictly lower: (r, m) and its mirror are written by the
                        // thread of the lower element only, the diagonal by its own
                        if (m + e < r) {
                            const float dk = umma::tf32r(dA * br * dec[4 * k + 2 * hr + e]);
                            dKS[umma::kidx(r, m + e, 64)] = dk;
                            dKS[umma::kidx(m + e, r, 64)] = dk;
                        } else if (m + e == r) {
                            dKS[umma::kidx(r, r, 64)] = 0.f;
                        }
                    }
                }
            }
            rs[0] = umma::row_quad_sum(rs[0]);
            rs[1] = umma::row_quad_sum(rs[1]);
            if ((lane & 3) == 0) {
                rp[half * 64 + rl] = rs[0];
                rp[half * 64 + rl + 8] = rs[1];
            }
#pragma unroll
            for (int k = 0; k < 4; k++)
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const float c = umma::col_oct_sum(cs[k][e]);
                    if (lane < 4) colp[win * 64 + half * 32 + 8 * k + 2 * lane + e] = c;
                }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            umma::mma(tX, umma::kmaj(dKS, 64), umma::mnt(Km), 64, 128, 64, false);   // (dKK + dKK^T) K
            umma::commit(mbar);
            // Gam (.) KK, dT, T, Y^T and T^T are consumed: the next tile's dW, dU, T^T
            if (next) issue_w(cn, tn);
        }
        if (tid < 64) {
            const float cs = (colp[tid] + colp[64 + tid]) + (colp[128 + tid] + colp[192 + tid]);
            const float rsA = rp[tid] + rp[64 + tid];
            dbs[tid] += rsA;
            dgs[tid] += bet[tid] * rsA - cs;
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 1));
        umma::fence_after_sync();
        if (!ok) break;
        // dKK, K (both layouts) and V (with the column sums over it) are consumed:
        // the next tile's dW, dU (MN-major), V and K
        if (next && tid == 0) {
            issue_m(cn, tn);
            issue_k(cn, tn);
        }
        // dK part = dKK product + diag(beta e^gam) T^T dW into the group's sum; at
        // its last v-head, rows rl, rl + 8 (those inside the chunk) of the k-head's
        // sum straight from the registers
        {
            float vk[32], vw[32];
            umma::tmem_ld64_m64(umma::tmem_at(tX, half * 64), vk);
            umma::tmem_ld64_m64(umma::tmem_at(tTW, half * 64), vw);
            const float bl = be[rl], bh = be[rl + 8];
#pragma unroll
            for (int k = 0; k < 8; k++) {
                const float d0 = vk[4 * k] + bl * vw[4 * k], d1 = vk[4 * k + 1] + bl * vw[4 * k + 1];
                const float d2 = vk[4 * k + 2] + bh * vw[4 * k + 2], d3 = vk[4 * k + 3] + bh * vw[4 * k + 3];
                kacc[4 * k] = first ? d0 : kacc[4 * k] + d0;
                kacc[4 * k + 1] = first ? d1 : kacc[4 * k + 1] + d1;
                kacc[4 * k + 2] = first ? d2 : kacc[4 * k + 2] + d2;
                kacc[4 * k + 3] = first ? d3 : kacc[4 * k + 3] + d3;
            }
            if (last) {
                float* dk_lo = w.dKv3 + ((int64_t)(ci.start + rl) * hk + kh) * kD;
                float* dk_hi = dk_lo + (int64_t)8 * hk * kD;
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    const int c = half * 64 + 8 * k + cf;
                    if (rl < L) *reinterpret_cast<float2*>(dk_lo + c) = make_float2(kacc[4 * k], kacc[4 * k + 1]);
                    if (rl + 8 < L)
                        *reinterpret_cast<float2*>(dk_hi + c) = make_float2(kacc[4 * k + 2], kacc[4 * k + 3]);
                }
            }
        }
        // ---- dg = reverse cumsum of dgam; gates
        if (tid < 64) sc[tid] = tid < L ? dgs[tid] + (gcur.dg1 + gcur.dg2) : 0.f;
        __syncthreads();
        if (tid < 32) {
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
            const int64_t tok = ci.start + tid;
            const float dg = rk[tid];
            const float Aexp = expf(alog);
            const float xa = to_f(gcur.a) + dtb;
            const float gval = -Aexp * softplusf_(xa);
            const float dav = dg * (-Aexp) * sigmoidf_(xa);
            const float bb = bet[tid];
            da[tok * hv + h] = from_f<IO>(dav);
            db[tok * hv + h] = from_f<IO>(dbs[tid] * bb * (1.f - bb));
            w.dgs[tok * hv + h] = dg;
            gterm = dg * gval;
            dterm = dav;
        }
        if (tid < 64) {
            gterm = warp_sum(gterm);
            dterm = warp_sum(dterm);
            if (lane == 0) { red[warp] = gterm; red[2 + warp] = dterm; }
        }
        __syncthreads();
        if (tid == 0) {
            gate_part[((int64_t)chunk * hv + h) * 2 + 0] = red[0] + red[1];
            gate_part[((int64_t)chunk * hv + h) * 2 + 1] = red[2] + red[3];
        }
        __syncthreads();   // gate sums and the tile's scalars are read
        if (!next) break;
        gcur = gnext;
        ci = cn;
        cn = c2;
        t = tn;
    }
    if (tid == 0) umma::bulk_wait_read();
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 512);
    if (!ok && tid == 0) atomicExch(w.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ B4: GVA sum
// dqkv q/k channels of k-head kh = the sum of its state-facing, P / dP and WY
// parts, each already summed over the k-head's G v-heads (fixed order).
__global__ void gva_sum_kernel(const float* __restrict__ dQv, const float* __restrict__ dKv,
                               const float* __restrict__ dQv2, const float* __restrict__ dKv2,
                               const float* __restrict__ dKv3, int64_t T, int hk, int hv,
                               float* __restrict__ dqkv) {
    const int C = (2 * hk + hv) * kD;
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // over T * hk * 32
    if (idx >= T * hk * 32) return;
    const int c4 = (int)(idx % 32) * 4;
    const int kh = (int)(idx / 32 % hk);
    const int64_t t = idx / 32 / hk;
    // every part is per k-head already (summed over its v-heads by its kernel)
    const int64_t okh = (t * hk + kh) * kD + c4;
    const float4 a1 = ld4(dQv + okh), a2 = ld4(dQv2 + okh);
    const float4 b1 = ld4(dKv + okh), b2 = ld4(dKv2 + okh), b3 = ld4(dKv3 + okh);
    const float4 q = make_float4(a1.x + a2.x, a1.y + a2.y, a1.z + a2.z, a1.w + a2.w);
    const float4 k = make_float4(b1.x + b2.x + b3.x, b1.y + b2.y + b3.y, b1.z + b2.z + b3.z,
                                 b1.w + b2.w + b3.w);
    st4(dqkv + t * C + kh * kD + c4, q);
    st4(dqkv + t * C + (int64_t)hk * kD + kh * kD + c4, k);
}

// dA_log[h] = sum over chunks of part[c][h][0]; ddt_bias[h] likewise [1].
// One block per head: thread i sums chunks i, i + kGateThreads, ... in order,
// then a fixed tree over the threads (deterministic).
constexpr int kGateThreads = 256;
__global__ void __launch_bounds__(kGateThreads)
gate_reduce_kernel(const float* __restrict__ part, int NT, int hv, float* dA_log, float* ddt_bias) {
    __shared__ float2 red[kGateThreads];
    const int h = blockIdx.x;
    float a = 0.f, b = 0.f;
    for (int c = threadIdx.x; c < NT; c += kGateThreads) {
        const float2 v = *reinterpret_cast<const float2*>(part + ((int64_t)c * hv + h) * 2);
        a += v.x;
        b += v.y;
    }
    red[threadIdx.x] = make_float2(a, b);
    __syncthreads();
    for (int m = kGateThreads / 2; m > 0; m >>= 1) {
        if (threadIdx.x < m) {
            red[threadIdx.x].x += red[threadIdx.x + m].x;
            red[threadIdx.x].y += red[threadIdx.x + m].y;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (dA_log) dA_log[h] = red[0].x;
        if (ddt_bias) ddt_bias[h] = red[0].y;
    }
}

// Deterministic two-level column sum of part [nparts][kD]: stage 1, block b
// sums rows [b*per, (b+1)*per) in order into tmp[b]; stage 2 sums tmp rows in
// order (8 row groups per column, then the 8 group sums in order).
constexpr int kColsumBlocks = 512;
__global__ void colsum_stage1_kernel(const float* __restrict__ part, int64_t nparts,
                                     float* __restrict__ tmp) {
    const int c = threadIdx.x;   // kD threads
    const int64_t per = (nparts + kColsumBlocks - 1) / kColsumBlocks;
    const int64_t r0 = blockIdx.x * per, r1 = min(nparts, r0 + per);
    float acc = 0.f;
    for (int64_t r = r0; r < r1; r++) acc += part[r * kD + c];
    tmp[blockIdx.x * kD + c] = acc;
}
__global__ void colsum_stage2_kernel(const float* __restrict__ tmp, float* __restrict__ out) {
    __shared__ float red[8][kD];
    const int c = threadIdx.x % kD, g = threadIdx.x / kD;   // 8 * kD threads
    float acc = 0.f;
    for (int r = g; r < kColsumBlocks; r += 8) acc += tmp[r * kD + c];
    red[g][c] = acc;
    __syncthreads();
    if (g == 0) {
        float s = 0.f;
        for (int i = 0; i < 8; i++) s += red[i][c];
        out[c] = s;
    }
}

// ------------------------------------------------------------------ launcher
// Everything on the caller's stream, in order: gated-norm backward, local
// backward, the reverse state pass with the P / dP groups beside it (one
// launch), state-facing terms, WY terms and gates, the GVA sum, then the
// deterministic reductions of the per-head gate sums and the norm weight.

template <class IO>
static cudaError_t chunk_bwd_t(const ChunkArgs& a, const BwdScratch& w, cudaStream_t st) {
    int nsm = 0;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = smem_attr(bwd_local_kernel, kB1Smem);
        if (e == cudaSuccess) e = smem_attr(bwd_state_dp_kernel, kStateDpSmem);
        if (e == cudaSuccess) e = smem_attr(bwd_sfacing_kernel, kB3aSmem);
        if (e == cudaSuccess) e = smem_attr(bwd_wy_kernel<IO>, kWySmem);
        if (e != cudaSuccess) return e;
    }
    float* gate_part = w.nw_part + (size_t)a.NT * a.hv * kD;
    TileMaps maps{};
    if (a.NT > 0) {
        const int64_t C = (int64_t)(2 * a.hk + a.hv) * kD, vs = (int64_t)a.hv * kD;
        cudaError_t e = make_rows_map(&maps.q, a.qkv, a.hk, a.T, C);
        if (e == cudaSuccess) e = make_rows_map(&maps.k, a.qkv + (int64_t)a.hk * kD, a.hk, a.T, C);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.v, a.qkv + (int64_t)2 * a.hk * kD, a.hv, a.T, C);
        if (e == cudaSuccess) e = make_rows_map(&maps.U, a.sv.U, a.hv, a.T, vs);
        if (e == cudaSuccess) e = make_rows_map(&maps.W, a.sv.W, a.hv, a.T, vs);
        if (e == cudaSuccess) e = make_rows_map(&maps.dO, w.dO, a.hv, a.T, vs);
        if (e == cudaSuccess) e = make_rows_map(&maps.dU, w.dU, a.hv, a.T, vs);
        if (e == cudaSuccess) e = make_rows_map(&maps.dW, w.dW, a.hv, a.T, vs);
        if (e == cudaSuccess) e = make_rows_map(&maps.dO_mn, w.dO, a.hv, a.T, vs, true);
        if (e == cudaSuccess) e = make_rows_map(&maps.dU_mn, w.dU, a.hv, a.T, vs, true);
        if (e == cudaSuccess) e = make_rows_map(&maps.dW_mn, w.dW, a.hv, a.T, vs, true);
        if (e == cudaSuccess) e = make_rows_map(&maps.W_mn, a.sv.W, a.hv, a.T, vs, true);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.k_mn, a.qkv + (int64_t)a.hk * kD, a.hk, a.T, C, true);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.q_mn, a.qkv, a.hk, a.T, C, true);
        if (e == cudaSuccess) e = make_rows_map(&maps.dQv, w.dQv, a.hk, a.T, (int64_t)a.hk * kD);
        if (e == cudaSuccess) e = make_rows_map(&maps.dKv, w.dKv, a.hk, a.T, (int64_t)a.hk * kD);
        if (e == cudaSuccess) e = make_rows_map(&maps.dUl, w.dUl, a.hv, a.T, vs);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.dv, a.dqkv + (int64_t)2 * a.hk * kD, a.hv, a.T, C);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.S0_mn, a.sv.S0, 1, (int64_t)a.NT * a.hv * kD, kD, true);
        if (e == cudaSuccess) e = make_rows_map(&maps.dS, w.dS, 1, (int64_t)a.NT * a.hv * kD, kD);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.dS_mn, w.dS, 1, (int64_t)a.NT * a.hv * kD, kD, true);
        if (e == cudaSuccess) e = make_rows_map(&maps.dUl_mn, w.dUl, a.hv, a.T, vs, true);
        if (e != cudaSuccess) return e;
        const int64_t rows = a.T * a.hv;
        {
            GDN_PROF("chunk_norm_bwd", st);
            chunk_norm_bwd_kernel<IO><<<(unsigned)((rows + kNormRows - 1) / kNormRows), 256, 0,
                                        st>>>(a.sv.o, (const IO*)a.z, a.norm_w, a.norm_eps,
                                              a.gate, (const IO*)a.dy, rows, w.dO, (IO*)a.dz,
                                              w.nw_part);
        }
        GDN_PROF("chunk_bwd_local", st);
        bwd_local_kernel<<<a.NT * a.hk, 256, kB1Smem, st>>>(maps, a.hk, a.hv, a.sv, w);
    }
    {
        // the reverse state pass (CTAs 0 .. n_state - 1) and the P / dP tiles
        // (persistent CTAs claiming tiles from a counter) in one grid
        const int n_state = (kD / kSl) * a.hv * a.N;
        const int n_dp = a.NT > 0 ? min(a.NT * a.hk, nsm) : 0;
        if (n_state + n_dp > 0) {
            GDN_PROF("chunk_bwd_state_dp", st);
            bwd_state_dp_kernel<<<(unsigned)(n_state + n_dp), kStateThreadsB, kStateDpSmem, st>>>(
                maps, a.hk, a.hv, a.NT, n_state, a.dS_final, a.dS_init, a.sv, w);
        }
    }
    if (a.NT > 0) {
        {
            GDN_PROF("chunk_bwd_sfacing", st);
            bwd_sfacing_kernel<<<min(a.NT * a.hk, nsm), 256, kB3aSmem, st>>>(maps, a.hk, a.hv,
                                                                               a.NT, a.sv, w);
        }
        GDN_PROF("chunk_bwd_wy", st);
        bwd_wy_kernel<IO><<<min(a.NT * a.hk, nsm), 256, kWySmem, st>>>(
            maps, (const IO*)a.a, (const IO*)a.b, a.A_log, a.dt_bias, a.hk, a.hv, a.NT, a.dqkv,
            (IO*)a.da, (IO*)a.db, gate_part, a.sv, w);
    }
    if (a.T > 0) {
        int64_t n = a.T * a.hk * 32;
        GDN_PROF("gva_sum", st);
        gva_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w.dQv, w.dKv, w.dQv2, w.dKv2, w.dKv3, a.T, a.hk,
                                                                    a.hv, a.dqkv);
    }
    if (a.dA_log || a.ddt_bias) {
        if (a.NT > 0) {
            GDN_PROF("gate_reduce", st);
            gate_reduce_kernel<<<a.hv, kGateThreads, 0, st>>>(gate_part, a.NT, a.hv, a.dA_log,
                                                              a.ddt_bias);
        } else {
            if (a.dA_log) cudaMemsetAsync(a.dA_log, 0, sizeof(float) * a.hv, st);
            if (a.ddt_bias) cudaMemsetAsync(a.ddt_bias, 0, sizeof(float) * a.hv, st);
        }
    }
    if (a.z && a.dnorm_w) {
        if (a.NT > 0) {
            float* tmp = w.nw_part + (size_t)a.NT * a.hv * kD + (size_t)a.NT * a.hv * 2;
            {
                GDN_PROF("norm_w_reduce", st);
                colsum_stage1_kernel<<<kColsumBlocks, kD, 0, st>>>(
                    w.nw_part, (a.T * a.hv + kNormRows - 1) / kNormRows, tmp);
            }
            GDN_PROF("norm_w_reduce2", st);
            colsum_stage2_kernel<<<1, 8 * kD, 0, st>>>(tmp, a.dnorm_w);
        } else
            cudaMemsetAsync(a.dnorm_w, 0, sizeof(float) * kD, st);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_bwd(const ChunkArgs& a, const BwdScratch& w, cudaStream_t st) {
    return a.bf16 ? chunk_bwd_t<__nv_bfloat16>(a, w, st) : chunk_bwd_t<float>(a, w, st);
}

}  // namespace gdn
