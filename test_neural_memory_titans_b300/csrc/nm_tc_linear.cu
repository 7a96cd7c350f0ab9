// tcgen05 tensor-core kernel for the linear memory M(x) = M x, d = 128,
// chunk b = 64.
//
// One persistent CTA per (batch, head) unit walks the sequence chunk by
// chunk ("Titans: Imparare a Memorizzare al Tempo di Test", section
// "Addestramento Parallelizzato": chunks of size b, every gradient of a chunk
// taken at the chunk-start weights; sections "Meccanismo di Aggiornamento
// della Memoria" / "Meccanismo di Dimenticanza" for the update, the
// 0h-n0.github.io explainer "メモリ読み出し" for retrieval after the update).
//
// With a_t = 1 - alpha_t and, inside a chunk of n tokens,
//   A_t = prod_{j<=t} a_j,  B_t = prod_{j<=t} beta_j,
//   sigma_t = a_t sigma_{t-1} + eta_t B_t,
//   Gamma_{t,i} = a_t Gamma_{t-1,i} + eta_t u_{t,i},  u_{t,i} = c_i prod_{l=i+1..t} beta_l,
//   gamma_i = Gamma_{n-1,i},  u_i = u_{n-1,i},
// and e_t = 2 (M0 k_t - v_t) (the gradient of ||M k_t - v_t||^2 at M0 is
// e_t k_t^T), the chunk is
//   y_t   = A_t M0 q_t - sigma_t S0 q_t - sum_{i<=t} Gamma_{t,i} (q_t . k_i) e_i
//   M_end = A_{n-1} M0 - sigma_{n-1} S0 - sum_i gamma_i e_i k_i^T
//   S_end = B_{n-1} S0 + sum_i u_i e_i k_i^T.
// Gamma is built column by column with the division-free recursion, so
// beta = 0 and alpha = 1 are exact.
//
// Per CTA (256 threads; thread 0 issues TMA and MMA):
//   TMEM (128 lanes x 512 fp32 columns): M [o][i] in 0..127 and S in 128..255
//     for the whole sequence; per chunk the key forward yhat [t][o] (M=64
//     layout, 256..383), Q K^T [t][i] (M=64, 384..447), M0 q [o][t] (448..511),
//     then S0 q [o][t] (256..319) and sum_i P[t][i] e_i [o][t] (320..383).
//   SMEM: Q and K tiles double-buffered and V single-buffered (TMA, 128-byte
//     swizzle), bf16 copies of M and S (the state as a tensor-core operand),
//     E, -gamma E, u E as [t][o] tiles, P = Gamma (.) Q K^T, Gamma in fp32.
// Per chunk two MMA batches: (1) yhat = K M0^T, Q K^T, M0 Q^T; then e, P and
// the scaled e tiles; (2) S0 Q^T, E^T P^T and the two state updates; then y
// (a [t][o] tile in shared memory, written out by one TMA store) and the next
// chunk's bf16 state.  The fp32 state is rescaled in TMEM
// (M <- A_n M - sigma_n S, S <- B_n S) while batch (1) runs.  The state never
// leaves the chip between chunks; HBM traffic is q, k, v in, y out, the gates,
// and the state once in and once out.
#include <cuda_bf16.h>

#include "nm_internal.h"
#include "tc_common.cuh"

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int BC = 64;
constexpr int NTHREADS = 256;
constexpr uint32_t HALF = BC * 128;   // one 64-column block of a 64-row bf16 tile (8 KB)
constexpr uint32_t TILE = 2 * HALF;   // 64 tokens x 128 features, bf16 (16 KB)
constexpr uint32_t SBLK = 128 * 128;  // one 64-column block of a 128-row tile (16 KB)

constexpr uint32_t OFF_Q = 0;                    // 2 stages
constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;     // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * TILE;
constexpr uint32_t OFF_MH = OFF_V + TILE;        // [128 o][128 i] bf16: two 16 KB column blocks
constexpr uint32_t OFF_SH = OFF_MH + 2 * SBLK;
constexpr uint32_t OFF_E = OFF_SH + 2 * SBLK;    // [64 t][128 o] bf16
constexpr uint32_t OFF_EG = OFF_E + TILE;        // -gamma_t e_t
constexpr uint32_t OFF_EU = OFF_EG + TILE;       // u_t e_t
constexpr uint32_t OFF_P = OFF_EU + TILE;        // [64 t][64 i] bf16
constexpr int GS = 68;                           // padded fp32 row stride of Gamma
constexpr uint32_t OFF_GM = OFF_P + HALF;
constexpr uint32_t OFF_F = OFF_GM + 64 * GS * 4; // gates [2][4][64], A, B, sigma, gamma, u
constexpr uint32_t N_F = 2 * 4 * BC + 5 * BC + 4 * BC + 4;  // + surprise partials [2 halves][e2, k2][64]
                                                             // + the next chunk's A_n, B_n, sigma_n
constexpr uint32_t OFF_BAR = OFF_F + 4 * N_F;
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_EU == OFF_EG + TILE, "a fp32 y tile spans EG and EU");

constexpr uint32_t COL_M = 0, COL_S = 128;
constexpr uint32_t COL_YH = 256, COL_QK = 384, COL_Y1 = 448;  // batch 1
constexpr uint32_t COL_Y2 = 256, COL_PE = 320;                // batch 2
constexpr uint32_t ID_YH = idesc_bf16_f32(64, 128, false, false);
constexpr uint32_t ID_QK = idesc_bf16_f32(64, 64, false, false);
constexpr uint32_t ID_Y = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t ID_PE = idesc_bf16_f32(128, 64, true, false);
constexpr uint32_t ID_UPD = idesc_bf16_f32(128, 128, true, true);
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s

// Shared-memory descriptors (the sw128_desc fields), K-major and MN-major
// with 64-element blocks `lbo` bytes apart.  The start-address field keeps
// bits 4..17 of the address (shared::cta addresses may carry higher bits).
// A k-step adds to the descriptor directly: +2 for 32 bytes (K-major), +128
// for 2048 bytes (16 rows, MN-major).
constexpr uint64_t desc_hi(uint32_t lbo) {
    return (static_cast<uint64_t>(lbo >> 4) << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return desc_hi(16) | ((a >> 4) & 0x3FFFu); }
__device__ __forceinline__ uint64_t mdesc(uint32_t a, uint32_t lbo) { return desc_hi(lbo) | ((a >> 4) & 0x3FFFu); }
constexpr uint64_t KS_K = 2, KS_M = 128;

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}

// 32 bf16 of row r, columns c0..c0+31, of a swizzled tile, as floats.
__device__ __forceinline__ void get_row32(const unsigned char* tile, uint32_t rows, uint32_t r, uint32_t c0, float* v) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 w = ld_shared_v4(base + sw128_offset(r, c0 + 8 * q, rows));
        v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
        v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
        v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
        v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
    }
}

template <typename Tout>
__device__ __forceinline__ void store_y(Tout* p, float x);
template <>
__device__ __forceinline__ void store_y<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ void store_y<float>(float* p, float x) { *p = x; }

// OPT: bit 0 = write the surprise (a.surprise), bit 1 = Huber loss (clip e), bit 2 = the
// gated output o = sigmoid(y) (.) y_attn (a.y_attn), bit 3 = the checkpointing forward of
// the backward pass (every chunk's start state into a.ckpt, y not written); compiled
// variants, so that the plain forward carries none of them.
template <typename Tout, int OPT>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_linear_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap ty, nm_args a,
                     int c_mode) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gates = reinterpret_cast<float*>(sm + OFF_F);  // [2 stages][a, eta, beta, c][64]
    float* sA = gates + 2 * 4 * BC;
    float* sBc = sA + BC;
    float* sSg = sBc + BC;
    float* sGl = sSg + BC;
    float* sU = sGl + BC;
    float* sPart = sU + BC;  // surprise partial sums: [hf][||e||^2 | ||k||^2][64]
    float* sEnd = sPart + 4 * BC;  // A_n, B_n, sigma_n of the chunk (computed during the previous chunk)
    float* Gm = reinterpret_cast<float*>(sm + OFF_GM);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // 0,1: Q|K stages; 2: V; 3: mma
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int qd = warp & 3;   // TMEM lane quadrant
    const int hf = warp >> 2;  // which half of the columns this thread handles
    const long long unit = blockIdx.x;
    const long long T = a.T;
    const long long P = (long long)D * D;
    const int nchunks = (int)((T + BC - 1) / BC);
    const float* alpha = a.alpha + unit * T;
    const float* eta = a.eta + unit * T;
    const float* beta = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    const int orow = 32 * qd + lane;  // row of an M=128 accumulator: output feature o

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
        prefetch_tmap(&ty);
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    auto issue_qk = [&](int chunk, int stage) {
        mbar_arrive_expect_tx(&bars[stage], 2 * TILE);
        const int t0 = chunk * BC;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_load_3d(sm + OFF_Q + stage * TILE + h * HALF, &tq, &bars[stage], h * 64, t0, (int)unit);
            tma_load_3d(sm + OFF_K + stage * TILE + h * HALF, &tk, &bars[stage], h * 64, t0, (int)unit);
        }
    };
    auto issue_v = [&](int chunk) {
        mbar_arrive_expect_tx(&bars[2], TILE);
        const int t0 = chunk * BC;
#pragma unroll
        for (int h = 0; h < 2; ++h) tma_load_3d(sm + OFF_V + h * HALF, &tv, &bars[2], h * 64, t0, (int)unit);
    };
    // A_n, B_n, sigma_n (the products and the sigma recursion of the gate scan,
    // in the scan's order) of the gates staged at `g`
    auto chunk_end = [&](const float* g) {
        float A = 1.f, Bc = 1.f, sg = 0.f;
#pragma unroll 8
        for (int t = 0; t < BC; ++t) {
            const float ga = g[t], ge = g[BC + t], gb = g[2 * BC + t];
            A *= ga;
            Bc *= gb;
            sg = fmaf(ga, sg, ge * Bc);
        }
        sEnd[0] = A;
        sEnd[1] = Bc;
        sEnd[2] = sg;
    };
    if (tid < BC) {  // gates of chunk 0; tokens past T change nothing: a = 1, eta = 0, beta = 1, c = 0
        const long long t = tid;
        float* g = gates;
        const bool ok = t < T;
        const float b = ok ? beta[t] : 1.0f;
        g[tid] = ok ? 1.0f - alpha[t] : 1.0f;
        g[BC + tid] = ok ? eta[t] : 0.0f;
        g[2 * BC + tid] = b;
        g[3 * BC + tid] = ok ? momentum_c(c_mode, b, cc, t) : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)(32 * qd) << 16);  // this warp's lane quadrant
    if (tid == 0 && nchunks > 0) {
        if (!a.skip_first_load) {  // (the test hook leaves chunk 0's tiles unloaded)
            issue_qk(0, 0);
            issue_v(0);
        }
    }
    if (tid == 224) chunk_end(gates);  // (visible after the barrier below)

    // initial state: TMEM fp32 (lane o = row o of M, S) and bf16 operand copies
    {
        float r[32];
        const float* m0 = a.M0 + unit * P + (long long)orow * D;
        const float* s0 = a.S0 + unit * P + (long long)orow * D;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const float* src = which ? s0 : m0;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int c0 = 64 * hf + 32 * j;
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    const float4 w = *reinterpret_cast<const float4*>(src + c0 + q);
                    r[q] = w.x; r[q + 1] = w.y; r[q + 2] = w.z; r[q + 3] = w.w;
                }
                tmem_st32(tl + (which ? COL_S : COL_M) + c0, r);
                put_row32(sm + (which ? OFF_SH : OFF_MH), 128, orow, c0, r);
                if (OPT & 8) {  // chunk 0's start state, for the backward pass
                    float* ck = a.ckpt + unit * nchunks * 2 * P + (which ? P : 0) + (long long)orow * D + c0;
#pragma unroll
                    for (int q = 0; q < 32; q += 4)
                        *reinterpret_cast<float4*>(ck + q) = make_float4(r[q], r[q + 1], r[q + 2], r[q + 3]);
                }
            }
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t aMH = smem_u32(sm + OFF_MH), aSH = smem_u32(sm + OFF_SH), aE = smem_u32(sm + OFF_E);
    const uint32_t aEG = smem_u32(sm + OFF_EG), aEU = smem_u32(sm + OFF_EU), aP = smem_u32(sm + OFF_P);

    bool failed = false;
    uint32_t mma_phase = 0;
    auto mma_wait = [&](bool committed) {  // bounded; uniform over the CTA
        bool ok = true;
        if (committed) {
            ok = mbar_wait(&bars[3], mma_phase, WAIT_NS);
            mma_phase ^= 1u;
        }
        failed = __syncthreads_or(!ok) || failed;
        tc_fence_after();
    };
    auto handoff = [&]() {  // epilogue smem / TMEM writes -> tensor-core reads
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    for (int c = 0; c < nchunks; ++c) {
        const int stage = c & 1;
        const long long t0 = (long long)c * BC;
        const int n = (int)min((long long)BC, T - t0);
        const float* g = gates + stage * 4 * BC;
        const uint32_t aQ = smem_u32(sm + OFF_Q + stage * TILE), aK = smem_u32(sm + OFF_K + stage * TILE);

        // the next chunk's gates: warps 2-3 load them now, raw, and store them after batch 1
        const int gi = tid - 64;
        const bool nxt_valid = gi >= 0 && gi < BC && c + 1 < nchunks && t0 + BC + gi < T;
        float nxt_al = 0.0f, nxt_e = 0.0f, nxt_b = 1.0f, nxt_c = 0.0f;
        if (nxt_valid) {
            const long long t = t0 + BC + gi;
            nxt_al = alpha[t];
            nxt_e = eta[t];
            nxt_b = beta[t];
            if (c_mode == NM_C_PER_TOKEN) nxt_c = cc[t];
        }

        // the gated output: the chunk's y_attn rows into L2 now, for the loads before the y epilogue
        if (OPT & 4) nm_prefetch_attn(a, (unit * T + t0) * D * (long long)sizeof(Tout), (long long)n * D * sizeof(Tout),
                                      tid, NTHREADS);
        // ---- batch 1 (thread 0, as soon as the tiles land): yhat = K M0^T, Q K^T, M0 Q^T;
        //      then the next chunk's Q|K tiles; meanwhile the gate scan
        bool tiles_ok = true;
        if (tid == 0 && !failed) {
            tiles_ok = mbar_wait(&bars[stage], (uint32_t)((c >> 1) & 1), WAIT_NS);
            if (tiles_ok) {
                tc_fence_after();
                const uint64_t dQ = kdesc(aQ), dK = kdesc(aK), dM = kdesc(aMH);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t acc = ks ? 1u : 0u;
                    // k-step ks covers features 16 ks .. 16 ks + 15: column block ks / 4 of each tile
                    const uint64_t kt = (ks >> 2) * (HALF >> 4) + KS_K * (ks & 3);
                    const uint64_t km = (ks >> 2) * (SBLK >> 4) + KS_K * (ks & 3);
                    mma_bf16(tm + COL_YH, dK + kt, dM + km, ID_YH, acc);
                    mma_bf16(tm + COL_QK, dQ + kt, dK + kt, ID_QK, acc);
                    mma_bf16(tm + COL_Y1, dM + km, dQ + kt, ID_Y, acc);
                }
                mma_commit(&bars[3]);
                if (c + 1 < nchunks) issue_qk(c + 1, stage ^ 1);
            }
            // V is read only after batch 1: its wait overlaps the products
            tiles_ok = tiles_ok && mbar_wait(&bars[2], (uint32_t)(c & 1), WAIT_NS);
            bulk_wait_read();  // the previous chunk's y tile (in EG / EU) has been read by its store
        }
        // rescale the fp32 state for this chunk (batch 1 does not touch it) while batch 1
        // runs: M <- A_n M - sigma_n S, S <- B_n S.  Thread 0 is issuing, so warp 4 (the
        // same TMEM lanes) takes warp 0's columns too.
        auto rescale = [&](int h) {
            const float An = sEnd[0], Bn = sEnd[1], sn = sEnd[2];
            float m[32], s[32];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t c0 = 64 * h + 32 * j;
                tmem_ld_n(tl + COL_M + c0, tl + COL_S + c0, m, s);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    m[q] = fmaf(An, m[q], -sn * s[q]);
                    s[q] = Bn * s[q];
                }
                tmem_st_n(tl + COL_M + c0, m);
                tmem_st_n(tl + COL_S + c0, s);
            }
        };
        if (warp != 0) rescale(hf);
        if (warp == 4) rescale(0);
        if (tid >= 160 && tid < 160 + BC) {  // (warps 5 and 6: warp 4 rescales for warp 0)
            // column i of Gamma: Gamma_{t,i} = a_t Gamma_{t-1,i} + eta_t u_{t,i}, zero above the diagonal
            const int i = tid - 160;
            // from row 0 with u = Gamma = 0 and the start injected,
            // u_t = beta_t u_{t-1} + [t = i] c_i: zero above the diagonal, no branch per row;
            // the next four gates are loaded before this group's stores
            const float ci = g[3 * BC + i];
            float u = 0.0f, G = 0.0f;
            const float4* g4 = reinterpret_cast<const float4*>(g);
            float4 va = g4[0], ve = g4[BC / 4], vb = g4[BC / 2];
#pragma unroll
            for (int t4 = 0; t4 < BC / 4; ++t4) {
                const float ga[4] = {va.x, va.y, va.z, va.w}, ge[4] = {ve.x, ve.y, ve.z, ve.w},
                            gb[4] = {vb.x, vb.y, vb.z, vb.w};
                if (t4 + 1 < BC / 4) {
                    va = g4[t4 + 1];
                    ve = g4[BC / 4 + t4 + 1];
                    vb = g4[BC / 2 + t4 + 1];
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int t = 4 * t4 + k;
                    u = fmaf(gb[k], u, t == i ? ci : 0.0f);
                    G = fmaf(ga[k], G, ge[k] * u);
                    Gm[t * GS + i] = G;
                }
            }
            sGl[i] = G;
            sU[i] = u;
        } else if (tid == 224) {
            float A = 1.f, Bc = 1.f, sg = 0.f;
            const float4* g4 = reinterpret_cast<const float4*>(g);
#pragma unroll
            for (int t4 = 0; t4 < BC / 4; ++t4) {
                const float4 va = g4[t4], ve = g4[BC / 4 + t4], vb = g4[BC / 2 + t4];
                const float ga[4] = {va.x, va.y, va.z, va.w}, ge[4] = {ve.x, ve.y, ve.z, ve.w},
                            gb[4] = {vb.x, vb.y, vb.z, vb.w};
                float oa[4], ob[4], os[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    A *= ga[k];
                    Bc *= gb[k];
                    sg = fmaf(ga[k], sg, ge[k] * Bc);
                    oa[k] = A;
                    ob[k] = Bc;
                    os[k] = sg;
                }
                reinterpret_cast<float4*>(sA)[t4] = make_float4(oa[0], oa[1], oa[2], oa[3]);
                reinterpret_cast<float4*>(sBc)[t4] = make_float4(ob[0], ob[1], ob[2], ob[3]);
                reinterpret_cast<float4*>(sSg)[t4] = make_float4(os[0], os[1], os[2], os[3]);
            }
        }
        const bool go1 = !failed && !__syncthreads_or(!tiles_ok);
        if (!go1 && !failed) failed = true;
        mma_wait(go1);
        // ---- e_t = 2 (M0 k_t - v_t) and its gamma / u scaled copies, and
        //      P = Gamma (.) Q K^T.  The M=64 accumulators hold token t in lane
        //      t % 16 of quadrant t / 16; lanes 16..31 take over half of each
        //      row by shuffle: e columns 64 hf + 32 .. (lanes 0..15: 64 hf ..),
        //      P columns 32 hf + 16 .. (lanes 0..15: 32 hf ..)
        {
            float e0[32], e1[32], qk[32];
            tmem_ld_n(tl + COL_YH + 64 * hf, tl + COL_YH + 64 * hf + 32, tl + COL_QK + 32 * hf, e0, e1, qk);
            const bool upper = lane >= 16;
            const int t = 16 * qd + (lane & 15);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const float hi = __shfl_sync(0xffffffffu, e1[q], lane & 15);
                e0[q] = upper ? hi : e0[q];
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float hi = __shfl_sync(0xffffffffu, qk[16 + q], lane & 15);
                qk[q] = upper ? hi : qk[q];
            }
            const bool live = t < n;
            const float gm = -sGl[t], uu = sU[t];
            const uint32_t c0 = 64 * hf + (upper ? 32 : 0);
            float vv[32], o[32];
            get_row32(sm + OFF_V, BC, t, c0, vv);
#pragma unroll
            for (int q = 0; q < 32; ++q) e0[q] = live ? 2.0f * (e0[q] - vv[q]) : 0.0f;
            if (OPT & 2) {  // the Huber loss clips e
#pragma unroll
                for (int q = 0; q < 32; ++q) e0[q] = nm_clip_err(e0[q], a.e_clip);
            }
            if (OPT & 1) {  // partial ||e_t||^2 and ||k_t||^2 over this thread's 32 columns, summed over the row
                float kv[32], e2 = 0.0f, k2 = 0.0f;
                get_row32(sm + OFF_K + stage * TILE, BC, t, c0, kv);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    e2 = fmaf(e0[q], e0[q], e2);
                    k2 = fmaf(kv[q], kv[q], k2);
                }
                e2 += __shfl_xor_sync(0xffffffffu, e2, 16);
                k2 += __shfl_xor_sync(0xffffffffu, k2, 16);
                if (!upper) {
                    sPart[hf * 2 * BC + t] = e2;
                    sPart[hf * 2 * BC + BC + t] = k2;
                }
            }
            put_row32(sm + OFF_E, BC, t, c0, e0);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = gm * e0[q];
            put_row32(sm + OFF_EG, BC, t, c0, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = uu * e0[q];
            put_row32(sm + OFF_EU, BC, t, c0, o);
            const uint32_t p0 = 32 * hf + (upper ? 16 : 0);
            const float* gr = Gm + t * GS + p0;
#pragma unroll
            for (int q = 0; q < 16; q += 4) {
                const float4 gg = *reinterpret_cast<const float4*>(gr + q);
                qk[q] *= gg.x; qk[q + 1] *= gg.y; qk[q + 2] *= gg.z; qk[q + 3] *= gg.w;
            }
            put_row<16>(sm + OFF_P, BC, t, p0, qk);
        }
        if (gi >= 0 && gi < BC && c + 1 < nchunks) {
            float* gn = gates + (stage ^ 1) * 4 * BC;
            gn[gi] = nxt_valid ? 1.0f - nxt_al : 1.0f;
            gn[BC + gi] = nxt_e;
            gn[2 * BC + gi] = nxt_b;
            gn[3 * BC + gi] = !nxt_valid ? 0.0f
                              : c_mode == NM_C_ONE_MINUS_BETA ? 1.0f - nxt_b
                              : c_mode == NM_C_PER_TOKEN ? nxt_c : 1.0f;
        }
        handoff();
        if ((OPT & 1) && hf == 0 && lane < 16) {  // surprise_t = ||e_t|| ||k_t||, token t = 16 qd + lane
            const int t = 16 * qd + lane;
            if (t < n)
                a.surprise[unit * T + t0 + t] = sqrtf(sPart[t] + sPart[2 * BC + t]) *
                                                 sqrtf(sPart[BC + t] + sPart[3 * BC + t]);
        }
        // ---- batch 2: S0 Q^T, E^T P^T, M += (-gamma E)^T K, S += (u E)^T K; the next V tile
        const bool go2 = !failed;
        if (go2 && tid == 0) {
            const uint64_t dQ = kdesc(aQ), dS = kdesc(aSH), dP = kdesc(aP);
            const uint64_t dE = mdesc(aE, HALF), dEG = mdesc(aEG, HALF), dEU = mdesc(aEU, HALF);
            const uint64_t dKm = mdesc(aK, HALF);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t kt = (ks >> 2) * (HALF >> 4) + KS_K * (ks & 3);
                const uint64_t km = (ks >> 2) * (SBLK >> 4) + KS_K * (ks & 3);
                mma_bf16(tm + COL_Y2, dS + km, dQ + kt, ID_Y, ks ? 1u : 0u);
            }
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {  // contraction over 64 tokens: 16 rows per k-step
                mma_bf16(tm + COL_PE, dE + KS_M * ks, dP + KS_K * ks, ID_PE, ks ? 1u : 0u);
                mma_bf16(tm + COL_M, dEG + KS_M * ks, dKm + KS_M * ks, ID_UPD, 1u);
                mma_bf16(tm + COL_S, dEU + KS_M * ks, dKm + KS_M * ks, ID_UPD, 1u);
            }
            mma_commit(&bars[3]);
            if (c + 1 < nchunks) issue_v(c + 1);
        }
        if (tid == 224 && c + 1 < nchunks) chunk_end(gates + (stage ^ 1) * 4 * BC);  // (staged before batch 2)
        // the gated output: y_attn of this thread's output row and 32 tokens, loaded while batch 2 runs
        // (consecutive lanes read consecutive features of a token: coalesced)
        Tout yatt[(OPT & 4) ? 32 : 1];
        if (OPT & 4) {
            const Tout* ya = reinterpret_cast<const Tout*>(a.y_attn) + (unit * T + t0) * D + orow;
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int t = 32 * hf + q;
                yatt[q] = ya[(t < n ? t : 0) * D];  // (rows past T are not stored)
            }
        }
        mma_wait(go2);
        // ---- y_t[o] = A_t (M0 q_t)[o] - sigma_t (S0 q_t)[o] - (E^T P^T)[o][t], tokens 32 hf ..,
        //      into a row-major [64 t][128 o] tile in the EG / EU space (free after batch 2),
        //      written to global memory by one TMA store (rows past T are not written)
        {
            float y1[32], y2[32], pe[32];
            tmem_ld_n(tl + COL_Y1 + 32 * hf, tl + COL_Y2 + 32 * hf, tl + COL_PE + 32 * hf, y1, y2, pe);
            Tout* yt = reinterpret_cast<Tout*>(sm + OFF_EG);
            if (!(OPT & 4)) {
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int t = 32 * hf + q;
                    store_y(yt + t * D + orow, fmaf(sA[t], y1[q], -fmaf(sSg[t], y2[q], pe[q])));
                }
            } else {  // o = sigmoid(y) (.) y_attn with the y_attn loaded above
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int t = 32 * hf + q;
                    const float v = fmaf(sA[t], y1[q], -fmaf(sSg[t], y2[q], pe[q]));
                    store_y(yt + t * D + orow, nm_gate_fast(nm_to_f32(yatt[q]), v));
                }
            }
        }
        // ---- the new state: bf16 operand copies for the next chunk, or the result
        {
            const bool last = c + 1 == nchunks;
            float m[32], s[32];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const uint32_t c0 = 64 * hf + 32 * j;
                tmem_ld_n(tl + COL_M + c0, tl + COL_S + c0, m, s);
                if (!last) {
                    put_row32(sm + OFF_MH, 128, orow, c0, m);
                    put_row32(sm + OFF_SH, 128, orow, c0, s);
                    if (OPT & 8) {  // chunk c + 1's start state, for the backward pass
                        float* mk = a.ckpt + (unit * nchunks + c + 1) * 2 * P + (long long)orow * D + c0;
#pragma unroll
                        for (int q = 0; q < 32; q += 4) {
                            *reinterpret_cast<float4*>(mk + q) = make_float4(m[q], m[q + 1], m[q + 2], m[q + 3]);
                            *reinterpret_cast<float4*>(mk + P + q) = make_float4(s[q], s[q + 1], s[q + 2], s[q + 3]);
                        }
                    }
                } else {
                    float* mt = a.M_T + unit * P + (long long)orow * D + c0;
                    float* st = a.S_T + unit * P + (long long)orow * D + c0;
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        *reinterpret_cast<float4*>(mt + q) = make_float4(m[q], m[q + 1], m[q + 2], m[q + 3]);
                        *reinterpret_cast<float4*>(st + q) = make_float4(s[q], s[q + 1], s[q + 2], s[q + 3]);
                    }
                }
            }
        }
        handoff();
        if (!(OPT & 8) && tid == 0 && !failed) {  // (no y for a checkpointing forward)
            tma_store_3d(&ty, sm + OFF_EG, 0, (int)t0, (int)unit);
            bulk_commit();
        }
    }
    if (tid == 0) bulk_wait_all();
    if (failed) {
        if (tid == 0 && a.status) atomicExch(a.status, NM_ERR_DEVICE_TIMEOUT);
        // let copies and products still in flight land before the CTA leaves
        for (int i = 0; i < 3; ++i) mbar_wait(&bars[i], 0, WAIT_NS / 4);
        mbar_wait(&bars[3], mma_phase, WAIT_NS);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <typename Tout, int OPT>
cudaError_t launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    CUtensorMap tq, tk, tv, ty;
    const long long units = (long long)a.B * a.H;
    if (!make_token_map(&tq, a.q, D, a.T, units) || !make_token_map(&tk, a.k, D, a.T, units) ||
        !make_token_map(&tv, a.v, D, a.T, units) ||
        // without y (a checkpointing forward) the map is made over q, of y's bf16 shape, and never used
        !make_token_store_map(&ty, a.y ? a.y : const_cast<void*>(a.q), D, a.T, units, sizeof(Tout) == 2))
        return cudaErrorInvalidValue;
    auto kern = tc_linear_kernel<Tout, OPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)units, NTHREADS, SMEM_BYTES, s>>>(tq, tk, tv, ty, a, c.c_mode);
    return cudaGetLastError();
}

template <typename Tout>
cudaError_t launch_opt(int opt, const nm_config& c, const nm_args& a, cudaStream_t s) {
    switch (opt) {
        case 0: return launch<Tout, 0>(c, a, s);
        case 1: return launch<Tout, 1>(c, a, s);
        case 2: return launch<Tout, 2>(c, a, s);
        case 3: return launch<Tout, 3>(c, a, s);
        case 4: return launch<Tout, 4>(c, a, s);
        case 5: return launch<Tout, 5>(c, a, s);
        case 6: return launch<Tout, 6>(c, a, s);
        default: return launch<Tout, 7>(c, a, s);
    }
}

}  // namespace

bool nm_tc_linear_supports(const nm_config& c) {
    return c.kind == NM_LINEAR && c.d == D && c.chunk == BC && c.in_dtype == NM_BF16;
}

cudaError_t nm_tc_linear_launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    const int opt = (a.surprise ? 1 : 0) | (a.e_clip < HUGE_VALF ? 2 : 0) | (a.y_attn ? 4 : 0);
    if (a.ckpt) {  // the checkpointing forward: no y, no surprise, no gate; its y map is made over q (bf16)
        if (a.y || a.surprise || a.y_attn) return cudaErrorInvalidValue;
        return opt & 2 ? launch<__nv_bfloat16, 10>(c, a, s) : launch<__nv_bfloat16, 8>(c, a, s);
    }
    return c.out_dtype == NM_BF16 ? launch_opt<__nv_bfloat16>(opt, c, a, s) : launch_opt<float>(opt, c, a, s);
}
