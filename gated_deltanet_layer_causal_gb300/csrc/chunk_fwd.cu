// Forward of the gated delta rule in the chunked WY form (chunk 64), with the
// gates, grouped value heads and the fused zero-centred gated RMSNorm.
//
// Per chunk (tokens i = 0..L-1, in-chunk cumulative gate gam_i):
//   A_ij = beta_i exp(gam_i - gam_j) k_i.k_j (j < i);  T = (I + A)^-1
//   W = T diag(beta e^gam) K ;  U~ = T diag(beta) V          (prep, parallel)
//   S_end = e^{gam_L} S0 + U^T diag(e^{gam_L-gam}) K,  U = U~ - W S0^T
//         = e^{gam_L} S0 + S0 M + B                        (state, sequential)
//   U = U~ - W S0^T ;
//   O = diag(e^gam) Q S0^T + (Q K^T (.) exp(gam_i-gam_j) (.) [i>=j]) U
//   y = O rsqrt(mean(O^2)+eps) (1+w) gate(z)             (out, parallel)
// which unrolls S_t = e^{g_t} S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
// o_t = S_t q_t exactly.  Sources: "[6/8] feat(models): port Qwen3.5 / Qwen3-Next
// GDN to the head-sharded layer" ("What": grouped value heads, native GVA);
// prime-rl #3860 "Summary" (chunk op with cu_seqlens / initial_state /
// output_final_state; ZeroCenteredRMSNorm); "[main] feat(moe): Support gated
// delta net for Qwen3-Next (1/4)" (A_log review comment: decay rate exp(A_log)).
//
// All products run on the tcgen05 tensor cores (tf32 operands, fp32
// accumulation); the state stays fp32 in registers across the whole sequence.
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
// + gridDim.x, ... (chunk = t / Hv, head = t % Hv: the v-heads of a chunk run
// side by side, so the q / k tiles they share come from DRAM once).  Per tile, tcgen05, with
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
constexpr int kLdA = 68;
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
    ChunkInfo ci = sv.chunks[t / hv];
    if (ci.len == 0) return;   // the device check of cu_seqlens failed: every chunk is empty
    auto issue = [&](const ChunkInfo& c, int tile) {   // one thread
        const int h = tile % hv, kh = h / (hv / hk);
        umma::mbar_expect_tx(mA, 3 * 64 * 128 * 4);
        umma::tma_rows(Ks, 64, &maps.k, kh, c.start, mA);
        umma::tma_rows(Km, 64, &maps.k_mn, kh, c.start, mA);
        umma::tma_rows(Vm, 64, &maps.v_mn, h, c.start, mA);
    };
    // padding rows continue the last gam (g = 0), beta = 0
    // (predicated loads: the values are first used a tile later)
    auto gates_of = [&](const ChunkInfo& c, int tile, float& gm, float& bt) {
        const int h = tile % hv;
        gm = 0.f;
        bt = 0.f;
        if (tid < 64) gm = sv.gam[(int64_t)h * sv.T + c.start + min(tid, c.len - 1)];
        if (tid < c.len) bt = sv.beta[(int64_t)h * sv.T + c.start + tid];
    };
    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::mbar_init(mA, 1);
        issue(ci, t);
    }
    float g_cur = 0.f, b_cur = 0.f;
    gates_of(ci, t, g_cur, b_cur);
    // chunk entries are loaded a tile before they are needed: cn (the next tile's)
    // is at hand at the top of an iteration, c2 (the one after) is requested there
    ChunkInfo cn = t + (int)gridDim.x < ntiles ? sv.chunks[(t + (int)gridDim.x) / hv] : ci;
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tD1 = tmem, tD2 = tmem + 256;
    const int half = warp >> 2;
    bool ok = true;
    for (int it = 0;; it++) {
        const int h = t % hv, L = ci.len;
        const int tn = t + (int)gridDim.x, t2 = tn + (int)gridDim.x;
        ChunkInfo c2 = cn;
        if (t2 < ntiles) c2 = sv.chunks[t2 / hv];
        if (tid < 64) {
            gam[tid] = g_cur;
            bet[tid] = b_cur;
            be[tid] = b_cur * expf(g_cur);
        }
        float g_next = 0.f, b_next = 0.f;   // the next tile's gates, requested here
        if (tn < ntiles && cn.len > 0) gates_of(cn, tn, g_next, b_next);
        if (tid == 32 && tn < ntiles && cn.len > 0) {   // the next tile's inputs into L2
            const int hn = tn % hv;
            umma::tma_prefetch_rows(&maps.k, hn / (hv / hk), cn.start);
            umma::tma_prefetch_rows(&maps.v_mn, hn, cn.start);
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
        // while the product runs: beta_i e^{gam_i - gam_j} [j < i] of this thread's
        // fragment of the 64 x 64 product
        const int rl = umma::frag_row_lo(), cf = umma::frag_col();
        float dec[16];
#pragma unroll
        for (int hr = 0; hr < 2; hr++) {
            const int r = rl + 8 * hr;
            const float br = bet[r], gr = gam[r];
#pragma unroll
            for (int k = 0; k < 4; k++)
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const int j = half * 32 + 8 * k + cf + e;
                    dec[4 * k + 2 * hr + e] = j < r ? br * expf(gr - gam[j]) : 0.f;
                }
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 0));
        umma::fence_after_sync();
        if (!ok) break;
        {   // A = beta_i e^{gam_i - gam_j} D1 (j < i); 32 columns per warp, all lanes
            float v[16];
            umma::tmem_ld_m64<4>(umma::tmem_at(tD1, half * 32), v);
#pragma unroll
            for (int hr = 0; hr < 2; hr++) {
                const int r = rl + 8 * hr;
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int j = half * 32 + 8 * k + cf, q = 4 * k + 2 * hr;
                    *reinterpret_cast<float2*>(As + r * kLdA + j) =
                        make_float2(dec[q] * v[q], dec[q + 1] * v[q + 1]);
                }
            }
        }
        __syncthreads();
        const bool next = tn < ntiles && cn.len > 0;
        tril_inverse64(As, kLdA, Tr, kLdA, Tk);   // Tk doubles as scratch
        __syncthreads();
        for (int idx = tid; idx < 64 * 16; idx += 256) {   // T diag(.) -> K-major rows i (lane = row)
            const int r = idx & 63, c = (idx >> 6) * 4;
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
            float* Tg = sv.Tm + ((int64_t)(t / hv) * hv + h) * 2 * 64 * 64;
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
        cn = c2;
        t = tn;
    }
    if (tid == 0) umma::bulk_wait_read();
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_free(tmem, 512);
    if (!ok && tid == 0) atomicExch(sv.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ state pass
// grid (2, Hv, N), 448 threads, one CTA per SM: CTA (slice, head, sequence)
// carries rows a0 .. a0 + 63 (a0 = 64 slice) of the fp32 state S [d_v x d_k]
// through the sequence's chunks.  With fk_i = e^{gam_L - gam_i} (0 past the
// chunk's length), a chunk's update S_end = e^{gam_L} S + U^T diag(fk) K with
// U = U~ - W S^T is, transposed,
//   S_end^T = e^{gam_L} S^T + M^T S^T + B^T,   M^T = -(diag(fk) K)^T W  (d_k x d_k),
//                                              B^T = (diag(fk) K)^T U~  (this CTA's columns),
// so one product per chunk waits on the state: M^T S^T (M = 128, N = 64,
// K = 128, tcgen05), with M^T read from tensor memory and S^T from shared
// memory, accumulated onto B^T.  The e^{gam_L} S term is added in fp32: the
// state lives in registers and never passes through tf32 itself.
//
// A tcgen05.mma of these shapes costs about as much to issue as to run, so the
// chain product is one 16-instruction product per chunk, and the products that
// do not depend on the state run ahead of it: M^T in three tensor-memory
// buffers (chunk c's is computed while the chain works on c - 2 and c - 1),
// B^T straight into the chain accumulator of its chunk (two buffers).  Each
// buffer (and each stage) has its own "free" and "ready" barriers, so that the
// phase after the one a thread waits for cannot complete before that thread has
// passed its wait (a parity wait would otherwise take the newer phase for the
// awaited one).
//
// Five roles, coupled only by mbarriers:
//  - product thread (warp 9): once a chunk's K, W, U~ are scaled, issues M^T
//    into its buffer (free once the chain product three chunks back is done)
//    and B^T into the chunk's accumulator (free once the state warps have read
//    the result two chunks back);
//  - scaling warps (0-3): scale K by fk and round U~ in place, walking the
//    tiles in shared-memory order (conflict-free); gate values one chunk ahead;
//  - rounding warps (10-13): once a chunk's M^T is done, round it to nearest
//    tf32 in tensor memory and negate it ("M ready"); one of them requests
//    each chunk's K, W, U~ (TMA, MN-major, two stages, two chunks ahead):
//    chunk c + 2 into chunk c's stage once both products of chunk c are done;
//  - state warps (4-7): thread (warp 4 + q, lane l) holds S[a][b'] for
//    b' = 32 q + l and all 64 rows a; once a chunk's chain product is done they
//    read it (accumulator free), update S and write its tf32 copy (the chain's
//    B operand, "S ready"), which one thread then stores as the next
//    chunk-start state (one tensor store);
//  - chain thread (warp 8): issues a chunk's chain product once M, B^T and S
//    are ready, and commits it to "chain done" and to its M^T buffer's "free".
// U itself is formed by the output kernel, which holds S0 anyway.  Output per
// chunk: the chunk-start state rounded to tf32, row-major [a][b] (the output
// kernel reads it K-major, the backward MN-major, through two tensor maps).
//
// Shared memory: S (rows a, swizzled K-major, 64 x 128) 32 KB and two stages
// of K, W (MN-major, 32 KB each) and the U~ slice (MN-major, 64 x 64, 16 KB).
// Tensor memory: two chain accumulators (M = 128, 64 columns) and three M^T
// tiles (128 columns): all 512 columns.
constexpr int kStFloats = 64 * 128;
constexpr int kStageF = 2 * 64 * 128 + 64 * 64;   // K, W, U~ slice
constexpr int kStateThreads = 448;
constexpr int kStateBars = 19;
constexpr size_t kStateSmem = sizeof(float) * (kStFloats + 2 * kStageF) + kStateBars * 8 + 8 + 1024;


__global__ void __launch_bounds__(kStateThreads, 1)
state_fwd_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, const float* S_init,
                 float* S_final, FwdSaved sv) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* St = sm;                    // [64 (a)][128 (b)] swizzled K-major: S, rounded
    float* stage = St + kStFloats;     // [2] x {K, W: [64 (i)][128] MN-major; U~: [64 (i)][64 (a)]}
    uint64_t* mT = reinterpret_cast<uint64_t*>(stage + 2 * kStageF);   // [2] tiles per stage
    uint64_t* mPm = mT + 2;            // [3] M^T product done, per buffer (commit)
    uint64_t* mPb = mPm + 3;           // [2] B^T product done, per accumulator (commit)
    uint64_t* mC = mPb + 2;            // chain product done (commit)
    uint64_t* bSc = mC + 1;            // [2] chunk scaled, per stage (scaling warps)
    uint64_t* bS = bSc + 2;            // S copy written (state warps)
    uint64_t* bM = bS + 1;             // [3] M^T buffer rounded (rounding warps)
    uint64_t* fM = bM + 3;             // [3] M^T buffer free (chain product commit)
    uint64_t* fA = fM + 3;             // [2] accumulator read (state warps)
    uint32_t* tslot = reinterpret_cast<uint32_t*>(fA + 2);
    auto Km = [&](int st) { return stage + st * kStageF; };
    auto Wm = [&](int st) { return stage + st * kStageF + 64 * 128; };
    auto Um = [&](int st) { return stage + st * kStageF + 2 * 64 * 128; };
    const int sl = blockIdx.x, h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int a0 = 64 * sl, kh = h / (hv / hk);
    const int64_t sbase = ((int64_t)n * hv + h) * kD * kD;
    const int c0 = sv.seq_chunk[n], c1 = sv.seq_chunk[n + 1];
    if (tid == 0) {
        umma::mbar_init(&mT[0], 1);
        umma::mbar_init(&mT[1], 1);
        umma::mbar_init(&mPb[0], 1);
        umma::mbar_init(&mPb[1], 1);
        umma::mbar_init(mC, 1);
        umma::mbar_init(&bSc[0], 128);
        umma::mbar_init(&bSc[1], 128);
        umma::mbar_init(bS, 128);
        for (int b = 0; b < 3; b++) {
            umma::mbar_init(&mPm[b], 1);
            umma::mbar_init(&bM[b], 128);
            umma::mbar_init(&fM[b], 1);
        }
        umma::mbar_init(&fA[0], 128);
        umma::mbar_init(&fA[1], 128);
    }
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    __syncthreads();   // barriers initialised, tensor memory allocated
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    auto tAcc = [&](int it) { return tmem + 64u * (uint32_t)(it & 1); };
    auto tM = [&](int it) { return tmem + 128u + 128u * (uint32_t)(it % 3); };
    bool ok = true;
    if (warp < 4) {
        // ---------------------------------------------------------- scaling warps
        // thread t scales the 16-byte pieces t + 128 q of K (rows (t / 8 + 16 q) % 64,
        // gate rows r = t / 8 + 16 (q % 4)) and rounds pieces t + 128 q of U~
        const int r0 = tid >> 3;
        auto gates = [&](int c, float (&gi)[4], float& gl, int& len) {
            gl = 0.f;
            len = 0;
#pragma unroll
            for (int u = 0; u < 4; u++) gi[u] = 0.f;
            if (c >= c1) return;
            const ChunkInfo info = sv.chunks[c];
            const float* g = sv.gam + (int64_t)h * sv.T + info.start;
#pragma unroll
            for (int u = 0; u < 4; u++) gi[u] = g[min(r0 + 16 * u, info.len - 1)];
            gl = g[info.len - 1];
            len = info.len;
        };
        float gi[4], gl, gi_n[4], gl_n;
        int len, len_n;
        gates(c0, gi, gl, len);
        for (int c = c0; c < c1 && ok; c++) {
            const int it = c - c0, st = it & 1;
            gates(c + 1, gi_n, gl_n, len_n);
            ok = umma::mbar_wait(&mT[st], (it >> 1) & 1);   // chunk c's tiles
            if (ok) {
                float f[4];
#pragma unroll
                for (int u = 0; u < 4; u++) f[u] = r0 + 16 * u < len ? expf(gl - gi[u]) : 0.f;
                float4* kr = reinterpret_cast<float4*>(Km(st));
                float4* ur = reinterpret_cast<float4*>(Um(st));
#pragma unroll
                for (int q0 = 0; q0 < 16; q0 += 8) {
                    float4 kv[8];
#pragma unroll
                    for (int q = 0; q < 8; q++) kv[q] = kr[tid + 128 * (q0 + q)];
#pragma unroll
                    for (int q = 0; q < 8; q++) {
                        const float fq = f[(q0 + q) & 3];
                        kr[tid + 128 * (q0 + q)] = umma::tf32r(
                            make_float4(fq * kv[q].x, fq * kv[q].y, fq * kv[q].z, fq * kv[q].w));
                    }
                }
                float4 uv[8];
#pragma unroll
                for (int q = 0; q < 8; q++) uv[q] = ur[tid + 128 * q];
#pragma unroll
                for (int q = 0; q < 8; q++)   // U~ is stored exact (W arrives rounded)
                    ur[tid + 128 * q] = umma::tf32r(uv[q]);
            }
            umma::fence_smem_to_async();
            umma::mbar_arrive(&bSc[st]);
#pragma unroll
            for (int u = 0; u < 4; u++) gi[u] = gi_n[u];
            gl = gl_n;
            len = len_n;
        }
    } else if (warp >= 10) {
        // ---------------------------------------------------------- rounding warps
        // thread 320 also requests each chunk's K, W, U~ (TMA, MN-major, two
        // stages): chunk c + 2 into chunk c's stage once both its products are done
        auto issue = [&](int c, int start) {
            const int st = (c - c0) & 1;
            umma::mbar_expect_tx(&mT[st], kStageF * 4);
            umma::tma_rows(Km(st), 64, &maps.k_mn, kh, start, &mT[st]);
            umma::tma_rows(Wm(st), 64, &maps.W_mn, h, start, &mT[st]);
            umma::tma_box(Um(st), &maps.U_mn, a0, h, start, &mT[st]);
            umma::tma_box(Um(st) + 64 * 32, &maps.U_mn, a0 + 32, h, start, &mT[st]);
        };
        const bool loader = tid == 320;
        if (loader && c0 < c1) issue(c0, sv.chunks[c0].start);
        if (loader && c0 + 1 < c1) issue(c0 + 1, sv.chunks[c0 + 1].start);
        int start_n = loader && c0 + 2 < c1 ? sv.chunks[c0 + 2].start : 0;   // one chunk ahead
        __syncwarp();   // converged again before the warp-wide tensor-memory accesses
        for (int c = c0; c < c1 && ok; c++) {
            const int it = c - c0;
            const int start = start_n;
            if (loader) start_n = c + 3 < c1 ? sv.chunks[c + 3].start : 0;
            ok = __all_sync(0xffffffffu, umma::mbar_wait(&mPm[it % 3], (it / 3) & 1));   // M^T done
            umma::fence_after_sync();
            if (!ok) break;
#pragma unroll
            for (int cc = 0; cc < 128; cc += 32) {   // M^T = -(accumulator), rounded
                float v[32];
                const uint32_t ta = umma::tmem_at(tM(it), cc);
                umma::tmem_ld32(ta, v);
#pragma unroll
                for (int u = 0; u < 32; u++) v[u] = umma::tf32r(-v[u]);
                umma::tmem_st32(ta, v);
            }
            umma::tmem_wait_st();
            umma::fence_before_sync();
            umma::mbar_arrive(&bM[it % 3]);
            if (loader && c + 2 < c1) {   // B^T of chunk c done too: its stage is free
                ok = umma::mbar_wait(&mPb[it & 1], (it >> 1) & 1);
                if (ok) issue(c + 2, start);
            }
            ok = __all_sync(0xffffffffu, ok);   // (converged again)
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------- state warps
        const int q = warp - 4, bp = 32 * q + lane, sid = tid - 128;
        float s[64];   // s[j] = S[a0 + j][bp]
#pragma unroll
        for (int j = 0; j < 64; j++)
            s[j] = S_init ? S_init[sbase + (int64_t)(a0 + j) * kD + bp] : 0.f;
        // S into St (rounded), "S ready", then St out as chunk c's start state
        // (one tensor store of the 64 rows: row-major, rounded)
        auto put = [&](int c) {
            if (sid == 0) umma::bulk_wait_read();   // the last store has read St
            umma::named_sync(2, 128);
#pragma unroll
            for (int j = 0; j < 64; j++) St[umma::swz(j, bp, 64)] = umma::tf32r(s[j]);
            umma::fence_smem_to_async();
            umma::mbar_arrive(bS);
            if (c >= c1) return;
            umma::named_sync(2, 128);
            if (sid == 0) {
                umma::tma_store_rows(&maps.S0, 0, (c * hv + h) * kD + a0, St);
                umma::bulk_commit();
            }
            __syncwarp();   // converged again before the warp-wide tensor-memory loads
        };
        // gam_L of chunk c, read one chunk ahead into a register
        auto gam_last = [&](int c) {
            if (c >= c1) return 0.f;
            const ChunkInfo info = sv.chunks[c];
            return sv.gam[(int64_t)h * sv.T + info.start + info.len - 1];
        };
        float gL = gam_last(c0);
        if (c0 < c1) put(c0);
        for (int c = c0; c < c1 && ok; c++) {
            const int it = c - c0;
            const float gL_next = gam_last(c + 1);
            ok = __all_sync(0xffffffffu, umma::mbar_wait(mC, it & 1));   // warp-uniform
            umma::fence_after_sync();
            if (!ok) break;
            const float dl = expf(gL);
            gL = gL_next;
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {   // S <- e^{gam_L} S + (B + S M)
                float v[32];
                umma::tmem_ld32(umma::tmem_at(tAcc(it), cc), v);
#pragma unroll
                for (int u = 0; u < 32; u++) s[cc + u] = dl * s[cc + u] + v[u];
            }
            umma::fence_before_sync();
            umma::mbar_arrive(&fA[it & 1]);   // the accumulator is read
            put(c + 1);
        }
        if (sid == 0) umma::bulk_wait_read();
        if (ok && S_final)
#pragma unroll
            for (int j = 0; j < 64; j++) S_final[sbase + (int64_t)(a0 + j) * kD + bp] = s[j];
    } else if (tid == 256) {
        // ---------------------------------------------------------- chain thread
        for (int c = c0; c < c1 && ok; c++) {
            const int it = c - c0;
            ok = umma::mbar_wait(&bM[it % 3], (it / 3) & 1) &&
                 umma::mbar_wait(&mPb[it & 1], (it >> 1) & 1) && umma::mbar_wait(bS, it & 1);
            umma::fence_after_sync();
            if (!ok) break;
            umma::mma_ta(tAcc(it), tM(it), umma::swt(St, 64), 128, 64, 128, true);
            umma::commit(mC);
            umma::commit(&fM[it % 3]);
        }
    } else if (tid == 288) {
        // ---------------------------------------------------------- products
        for (int c = c0; c < c1 && ok; c++) {
            const int it = c - c0, st = it & 1;
            ok = umma::mbar_wait(&bSc[st], (it >> 1) & 1);   // chunk c scaled
            // M^T buffer it % 3: its last chain product (three chunks back) is done
            if (it >= 3) ok = ok && umma::mbar_wait(&fM[it % 3], ((it / 3) - 1) & 1);
            umma::fence_after_sync();
            if (!ok) break;
            umma::mma(tM(it), umma::mnt(Km(st)), umma::mnt(Wm(st)), 128, 128, 64, false);   // -M^T
            umma::commit(&mPm[it % 3]);
            // accumulator it & 1: the state warps have read it (two chunks back)
            if (it >= 2) ok = umma::mbar_wait(&fA[it & 1], ((it / 2) - 1) & 1);
            umma::fence_after_sync();
            if (!ok) break;
            umma::mma(tAcc(it), umma::mnt(Km(st)), umma::mnt(Um(st)), 128, 64, 64, false);  // B^T
            umma::commit(&mPb[it & 1]);
        }
    }
    umma::fence_before_sync();
    ok = __syncthreads_and(ok);
    if (warp == 0) umma::tmem_free(tmem, 512);
    if (!ok && tid == 0) atomicExch(sv.status, 5);   // GDN_ERR_DEVICE_TIMEOUT
}

// ------------------------------------------------------------------ output + norm
// Persistent: one CTA per SM walks the (chunk, head) tiles t = blockIdx.x,
// + gridDim.x, ... (chunk = t / Hv, head = t % Hv: the v-heads of a chunk run
// side by side, so the q / k tiles they share come from DRAM once).  Per tile, tcgen05:
//   [Q; W] [K; S0]^T   one M = 128, N = 192, K = 128 product: rows 0-63 give
//                      D1 = Q K^T (columns 0-63) and D3 = Q S0^T (64-191),
//                      rows 64-127 give DU = W S0^T (columns 64-191)
//   P  = D1 (.) e^{gam_i - gam_j} (.) [i >= j]          -- staged K-major
//   U  = U~ - DU  (rounded; the B operand below, and stored for the backward)
//   D2 = [P; 0] U   (M = 128: rows 0-63 of the accumulator, like D3)
//   O  = D2 + e^{gam_i} D3 ; y = O rsqrt(mean(O^2)+eps) (1+w) gate(z)
// Stacking Q over W and K over S0 makes the three first products one product
// of 16 instructions (a tcgen05.mma of M = 64 costs about as much as one of
// M = 128), and puts P (rows 0-63) and DU (rows 64-127) in different halves of
// the tensor-memory lanes, so the P epilogue (warps 0, 1, 4, 5) and the U
// epilogue (warps 2, 3, 6, 7) run at the same time.
// Shared memory: [Q; W] 64 KB and [K; S0] 96 KB swizzled (TMA into one tile
// each, rows 128 / 192 apart per box), U~ MN-major 32 KB (then U, then O staged,
// swizzled), [P; 0] 32 KB K-major (rows 64-127 zero, written once).  The next
// tile's Q, W, K and S0 are requested as soon as the first product is done, its
// U~ once this tile's O (staged over U) has been stored; all of them are
// prefetched into L2 a tile ahead, and its chunk entry and gate values are
// loaded into registers meanwhile.  While the first product runs, each warp
// requests the z rows of its norm rows (converted only when used) and the P
// warps compute their decay factors.  U goes back in place of U~ by one tensor
// store while P U runs, o by one tensor store from the O staging tile.  Tensor
// memory: 320 fp32 columns (512 allocated), once.
constexpr int kOutFloats = 128 * 128 + 192 * 128 + 64 * 128 + 128 * 64;
constexpr size_t kOutSmem = sizeof(float) * (kOutFloats + 64 * 2 + 2 * 64 + 16) + 32 + 1024;

// Rows 0 .. L-1 of a 64-row MN-major tile to a row-major global tensor, one warp per row.
__device__ __forceinline__ void store_rows_mn(float* dst, int64_t stride, const float* src, int L) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int r = warp; r < L; r += nw)
        *reinterpret_cast<float4*>(dst + r * stride + 4 * lane) =
            *reinterpret_cast<const float4*>(src + umma::swz_mn(r, 4 * lane));
}

template <class IO>
__global__ void __launch_bounds__(256, 1)
out_fwd_kernel(const __grid_constant__ TileMaps maps, int hk, int hv, int NT, const IO* z,
               const float* norm_w, float norm_eps, int gate, IO* o_out, IO* y_out, FwdSaved sv) {
    extern __shared__ float sm_raw[];
    float* sm = umma::align1024(sm_raw);
    float* QW = sm;                    // [4 boxes][128 rows][32]: rows 0-63 Q, 64-127 W (arrives rounded)
    float* KS = QW + 128 * 128;        // [4 boxes][192 rows][32]: rows 0-63 K, 64-191 S0 (rows a)
    float* Us = KS + 192 * 128;        // [64 (j)][128 (a)] MN-major U~, then U; then O, swizzled
    float* P2 = Us + 64 * 128;         // [128 (i)][64 (j)] K-major: P, then zero rows
    float* gam = P2 + 128 * 64;
    float* eg = gam + 64;
    float* ssq = eg + 64;              // [2][64] partial sums of squares
    uint64_t* mbar = reinterpret_cast<uint64_t*>(ssq + 2 * 64 + 16);   // MMA
    uint64_t* mA = mbar + 1;           // Q, W, K, S0
    uint64_t* mU = mA + 1;             // U~
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mU + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ntiles = NT * hv;
    int t = blockIdx.x;
    if (t >= ntiles) return;
    ChunkInfo ci = sv.chunks[t / hv];
    if (ci.len == 0) return;   // the device check of cu_seqlens failed: every chunk is empty
    auto issue_a = [&](const ChunkInfo& c, int tile) {   // one thread
        const int h = tile % hv, kh = h / (hv / hk);
        umma::mbar_expect_tx(mA, (128 * 128 + 192 * 128) * 4);
        umma::tma_rows(QW, 128, &maps.q, kh, c.start, mA);
        umma::tma_rows(QW + 64 * 32, 128, &maps.W, h, c.start, mA);
        umma::tma_rows(KS, 192, &maps.k, kh, c.start, mA);
        const int s0row = ((tile / hv) * hv + h) * kD;   // S0 tile rows a = 0 .. 127
        umma::tma_rows(KS + 64 * 32, 192, &maps.S0, 0, s0row, mA);
        umma::tma_rows(KS + 128 * 32, 192, &maps.S0, 0, s0row + 64, mA);
    };
    auto issue_u = [&](const ChunkInfo& c, int tile) {   // one thread
        umma::mbar_expect_tx(mU, 64 * 128 * 4);
        umma::tma_rows(Us, 64, &maps.U_mn, tile % hv, c.start, mU);
    };
    auto prefetch_in = [&](const ChunkInfo& c, int tile) {   // one thread: what issue_a / issue_u load, into L2
        const int hp = tile % hv, khp = hp / (hv / hk);
        const int s0p = ((tile / hv) * hv + hp) * kD;
        umma::tma_prefetch_rows(&maps.q, khp, c.start);
        umma::tma_prefetch_rows(&maps.k, khp, c.start);
        umma::tma_prefetch_rows(&maps.W, hp, c.start);
        umma::tma_prefetch_rows(&maps.S0, 0, s0p);
        umma::tma_prefetch_rows(&maps.S0, 0, s0p + 64);
        umma::tma_prefetch_rows(&maps.U_mn, hp, c.start);
    };
    // chunk entries are loaded a tile before they are needed: cn (the next tile's)
    // is at hand at the top of an iteration, c2 (the one after) is requested there
    ChunkInfo cn = t + (int)gridDim.x < ntiles ? sv.chunks[(t + (int)gridDim.x) / hv] : ci;
    // padding rows continue the last gate value (g = 0); a predicated load, first
    // used a tile later
    auto gam_of = [&](const ChunkInfo& c, int tile) {
        float g = 0.f;
        if (tid < 64) g = sv.gam[(int64_t)(tile % hv) * sv.T + c.start + min(tid, c.len - 1)];
        return g;
    };
    if (tid == 0) {
        umma::mbar_init(mbar, 1);
        umma::mbar_init(mA, 1);
        umma::mbar_init(mU, 1);
        issue_a(ci, t);
        issue_u(ci, t);
    }
    for (int e = tid; e < 64 * 64; e += 256) P2[64 * 64 + e] = 0.f;   // rows 64-127 of [P; 0]
    float g_cur = gam_of(ci, t);
    if (warp == 0) umma::tmem_alloc(tslot, 512);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tslot;
    const uint32_t tF = tmem, tD2 = tmem + 192;   // first product (192 columns), P U (128)
    const int q4 = warp & 3, half = warp >> 2;
    const int row = 32 * (q4 & 1) + lane;   // this thread's accumulator row within its lane half
    const float4 w4 = z ? ld4(norm_w + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    bool ok = true;
    // issued: this tile's first product was issued at the end of the previous
    // iteration (a whole chunk, operands already tf32), so it runs while that
    // tile's norm and stores do; its gate values are in shared memory then too
    bool issued = false;
    for (int it = 0;; it++) {
        const int h = t % hv, L = ci.len;
        const int tn = t + (int)gridDim.x, t2 = tn + (int)gridDim.x;
        ChunkInfo c2 = cn;
        if (t2 < ntiles) c2 = sv.chunks[t2 / hv];
        if (tid < 64 && !issued) {
            gam[tid] = g_cur;
            eg[tid] = tid < L ? expf(g_cur) : 0.f;
        }
        if (tid == 32 && tn < ntiles && cn.len > 0) prefetch_in(cn, tn);
        float g_next = 0.f;   // the next tile's gate values, requested here
        if (tn < ntiles && cn.len > 0) g_next = gam_of(cn, tn);
        ok = __syncthreads_and(umma::mbar_wait(mA, it & 1));   // Q, W, K, S0; gam visible
        if (!ok) break;
        if (!issued) {
            if (L < 64) {   // tail rows belong to the next sequence
                umma::zero_tail_rows(QW, 128, 0, L);
                umma::zero_tail_rows(QW, 128, 64, L);
                umma::zero_tail_rows(KS, 192, 0, L);
                __syncthreads();
            }
            if (!sv.qkv_tf32) {   // Q and K (W and S0 arrive rounded: rounding them again changes nothing)
                umma::tf32r_inplace(QW, 128 * 128);
                umma::tf32r_inplace(KS, 64 * 128 * 3);
            }
            umma::fence_smem_to_async();
            __syncthreads();
            umma::fence_after_sync();
            if (tid == 0) {
                umma::mma(tF, umma::swt(QW, 128), umma::swt(KS, 192), 128, 192, 128, false);
                umma::commit(mbar);
            }
        }
        // this warp's norm rows r = warp + 8 q: their z values, into registers (used
        // last; rows past the chunk repeat its last row and are not stored)
        raw4_t<IO> zr[8];
        if (z) {
#pragma unroll
            for (int q = 0; q < 8; q++)
                zr[q] = ld4_raw(z + (((int64_t)ci.start + min(warp + 8 * q, L - 1)) * hv + h) * kD + lane * 4);
        }
        // while the product runs, on the warps that form P: the decay factors
        // e^{gam_i - gam_j} [i >= j] of this thread's row of P, by the hardware
        // exponential (a few ulp; P is rounded to tf32 next)
        float dec[32];
        if (q4 < 2) {
            const float gi = gam[row];
#pragma unroll
            for (int k = 0; k < 32; k++) {
                const int j = 32 * half + k;
                dec[k] = j <= row ? __expf(gi - gam[j]) : 0.f;
            }
        }
        ok = __syncthreads_and(umma::mbar_wait(mbar, 0));
        umma::fence_after_sync();
        if (!ok) break;
        const bool next = tn < ntiles && cn.len > 0;
        if (next && tid == 0) issue_a(cn, tn);   // Q, W, K, S0 consumed
        if (q4 < 2) {
            // P = D1 (.) Gam (.) M -> K-major rows i; row i = row, columns j = 32 half .. + 31
            float v[32];
            umma::tmem_ld32(umma::tmem_at(tF, 32 * half), v);
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(P2 + umma::kidx(row, 32 * half + k, 64)) = umma::tf32r(
                    make_float4(v[k] * dec[k], v[k + 1] * dec[k + 1], v[k + 2] * dec[k + 2], v[k + 3] * dec[k + 3]));
        } else {
            // U = U~ - W S0^T in place (rounded), rows past the chunk zero; row i = row,
            // columns a = 64 half .. + 63 (accumulator rows 64-127, columns 64-191)
            ok = __all_sync(0xffffffffu, umma::mbar_wait(mU, it & 1));   // U~ (warp-uniform)
            if (ok) {
                const int i = row;
#pragma unroll
                for (int cc = 0; cc < 64; cc += 32) {
                    float v[32];
                    umma::tmem_ld32(umma::tmem_at(tF, 64 + 64 * half + cc), v);
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        float4* p = reinterpret_cast<float4*>(Us + umma::swz_mn(i, 64 * half + cc + k));
                        const float4 u = *p;
                        *p = i < L ? umma::tf32r(make_float4(u.x - v[k], u.y - v[k + 1], u.z - v[k + 2],
                                                             u.w - v[k + 3]))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        ok = __syncthreads_and(ok);
        umma::fence_after_sync();
        if (!ok) break;
        // U for the backward (only ever a tensor-core operand: stored rounded) while
        // P U runs: a whole chunk by one tensor store in place of U~, a partial one
        // row by row
        if (tid == 0) {
            umma::mma(tD2, umma::kmaj(P2, 64), umma::mnt(Us), 128, 128, 64, false);
            umma::commit(mbar);
            if (L == 64) {
                umma::tma_store_rows(&maps.U_mn, h, ci.start, Us);
                umma::bulk_commit();
            }
        }
        if (L < 64) store_rows_mn(sv.U + ((int64_t)ci.start * hv + h) * kD, (int64_t)hv * kD, Us, L);
        if (tid == 0) umma::bulk_wait_read();   // the U store has read the tile O goes over
        ok = __syncthreads_and(umma::mbar_wait(mbar, 1));   // and the U rows are read
        umma::fence_after_sync();
        if (!ok) break;
        // O = D2 + e^{gam_i} D3 (accumulator rows 0-63: warps 0, 1, 4, 5), staged as a
        // swizzled tile over U (consumed) and stored from there by one tensor store;
        // the norm and the y stores then run row by row on all lanes, one warp per
        // row, fully coalesced
        float* Or = Us;
        if (q4 < 2) {
            const int i = row;
            const float e = eg[i];
            float ss = 0.f;
#pragma unroll
            for (int cc = 0; cc < 64; cc += 32) {
                float v2[32], v3[32];
                umma::tmem_ld32(umma::tmem_at(tD2, 64 * half + cc), v2);
                umma::tmem_ld32(umma::tmem_at(tF, 64 + 64 * half + cc), v3);
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                    float4 x;
                    x.x = v2[k] + e * v3[k];
                    x.y = v2[k + 1] + e * v3[k + 1];
                    x.z = v2[k + 2] + e * v3[k + 2];
                    x.w = v2[k + 3] + e * v3[k + 3];
                    ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
                    *reinterpret_cast<float4*>(Or + umma::swz(i, 64 * half + cc + k, 64)) = x;
                }
            }
            ssq[half * 64 + i] = ss;
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        // the next tile's first product, now that tensor memory is read, when it
        // needs no preparation (a whole chunk with tf32 operands); its gate values
        // go to shared memory (the norm below does not read them)
        const bool early = next && cn.len == 64 && sv.qkv_tf32;
        if (early) {
            if (tid < 64) {
                gam[tid] = g_next;
                eg[tid] = expf(g_next);
            }
            if (tid == 0 && umma::mbar_wait(mA, (it + 1) & 1)) {   // on a timeout the wait at the top fails
                umma::mma(tF, umma::swt(QW, 128), umma::swt(KS, 192), 128, 192, 128, false);
                umma::commit(mbar);
            }
        }
        if (L == 64 && tid == 0) {   // o (fp32, for the backward) by one tensor store
            umma::tma_store_rows(&maps.o, h, ci.start, Or);
            umma::bulk_commit();
        }
        // this warp's eight rows: all reads first, then the math and the stores
        // (independent rows, so their latencies overlap); rows past the chunk are
        // read from the staging tile but not stored
        float4 o4s[8];
        float rss[8];
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int r = warp + 8 * q;
            o4s[q] = *reinterpret_cast<const float4*>(Or + umma::swz(r, lane * 4, 64));
            rss[q] = rsqrtf((ssq[r] + ssq[64 + r]) * (1.f / kD) + norm_eps);
        }
#pragma unroll
        for (int q = 0; q < 8; q++) {
            const int r = warp + 8 * q;
            if (r < L) {
                const int64_t tok = ci.start + r;
                const int64_t off = (tok * hv + h) * kD + lane * 4;
                if (L < 64) st4(sv.o + off, o4s[q]);   // (a whole chunk's went by tensor store)
                if (o_out) st4(o_out + off, o4s[q]);
                if (z) {
                    st4(y_out + off, gated_norm4(o4s[q], rss[q], w4, cvt4(zr[q]), gate));
                    if (lane == 0) sv.rstd[tok * hv + h] = rss[q];
                }
            }
        }
        umma::fence_smem_to_async();   // O staging reads -> the next U~ load
        __syncthreads();               // O and the sums of squares are read
        if (!next) break;
        if (tid == 0) {
            umma::bulk_wait_read();    // the o store has read the staging tile
            issue_u(cn, tn);
        }
        issued = early;
        g_cur = g_next;
        ci = cn;
        cn = c2;
        t = tn;
    }
    if (tid == 0) umma::bulk_wait_read();
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
        if (e == cudaSuccess) e = make_rows_map(&maps.o, a.sv.o, a.hv, a.T, (int64_t)a.hv * kD);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.W_mn, a.sv.W, a.hv, a.T, (int64_t)a.hv * kD, true);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.k_mn, a.qkv + (int64_t)a.hk * kD, a.hk, a.T, C, true);
        if (e == cudaSuccess)
            e = make_rows_map(&maps.v_mn, a.qkv + (int64_t)2 * a.hk * kD, a.hv, a.T, C, true);
        if (e == cudaSuccess) e = make_rows_map(&maps.S0, a.sv.S0, 1, (int64_t)a.NT * a.hv * kD, kD);
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
        state_fwd_kernel<<<dim3(2, a.hv, a.N), kStateThreads, kStateSmem, st>>>(
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
