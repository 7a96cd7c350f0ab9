// tcgen05 tensor-core kernel for the linear memory M(x) = M x with d = 64
// and chunks of b = 64 NB tokens (NB = 1, 2 or 4).
//
// Method ("Titans: Imparare a Memorizzare al Tempo di Test", sections
// "Addestramento Parallelizzato", "Meccanismo di Aggiornamento della
// Memoria", "Meccanismo di Dimenticanza"; the 0h-n0.github.io explainer,
// "メモリ読み出し"): every token of a chunk takes its gradient
// e_i k_i^T, e_i = 2 (M0 k_i - v_i), at the chunk-start state (M0, S0), and
//   y_t   = A_t M0 q_t - sigma_t S0 q_t - sum_{i<=t} Gamma_{t,i} (q_t . k_i) e_i,
//   M_end = A_n M0 - sigma_n S0 - sum_i gamma_i e_i k_i^T,
//   S_end = B_n S0 + sum_i u_i e_i k_i^T
// (A, B, sigma, Gamma, gamma, u as in nm_tc_linear.cu, over the whole chunk).
//
// A chunk is processed as NB blocks of 64 tokens.  For a token t of block s
// and a token i of an earlier block, the recursion of Gamma over block s is
// linear in the column's state at the block start, (G_i, U_i) = (Gamma,
// u)_{start(s)-1, i}:  Gamma_{t,i} = p_t G_i + r_t U_i, with
//   p_t = prod_{j=start..t} a_j,  w_t = prod_{j=start..t} beta_j,
//   r_t = a_t r_{t-1} + eta_t w_t   (r_{start-1} = 0).
// So the earlier blocks enter through two d x d accumulators
//   CG = sum_{i<start(s)} G_i e_i k_i^T,   CU = sum_{i<start(s)} U_i e_i k_i^T:
//   y_t = A_t M0 q_t - sigma_t S0 q_t - p_t CG q_t - r_t CU q_t
//         - sum_{i in s, i<=t} Gamma_{t,i} (q_t . k_i) e_i,
// and at the end of block s, with gamma_i, u_i of block s (Gamma, u at its
// last token for its own columns):
//   CG <- p_end CG + r_end CU + sum_{i in s} gamma_i e_i k_i^T,
//   CU <- w_end CU + sum_{i in s} u_i e_i k_i^T.
// After the chunk's last block CG = sum_i gamma_i e_i k_i^T and CU = sum_i
// u_i e_i k_i^T, so M_end = A_n M0 - sigma_n S0 - CG and S_end = B_n S0 + CU.
// The chunk-level A_t, B_t, sigma_t follow from the block-level ones and the
// values at the previous block's end: A_t = A' p_t, B_t = B' w_t,
// sigma_t = sigma' p_t + B' r_t.
//
// Per CTA (one unit, 256 threads; thread 0 issues TMA and MMA):
//   TMEM: CG [o][x] (columns 0..63) and CU (64..127) in the M=64 layout (row r
//     in lane r % 16 + 32 (r / 16)); per block the key forward yhat [t][o] and
//     Q K^T (128..255), then Q [M0 | S0 | CG | CU]^T [t][4 x 64] (128..383) and
//     sum_i P[t][i] e_i [t][o] (384..447).
//   SMEM: Q, K, V tiles double-buffered (TMA, 128-byte swizzle), bf16 copies
//     of M0, S0, CG, CU (one N=256 operand), e, gamma e, u e, P, Gamma, and the
//     chunk-start state in fp32.
#include <cuda_bf16.h>

#include "nm_internal.h"
#include "tc_common.cuh"

namespace {

using namespace tc;

constexpr int D = 64;
constexpr int SB = 64;  // tokens per block
constexpr int NTHREADS = 256;
constexpr uint32_t T64 = 64 * 128;  // [64 rows][64 bf16] swizzled tile (8 KB)
constexpr int GS = 68;              // padded fp32 row stride (Gamma, the fp32 state)

constexpr uint32_t OFF_Q = 0;                      // 2 stages
constexpr uint32_t OFF_K = OFF_Q + 2 * T64;        // 2 stages
constexpr uint32_t OFF_V = OFF_K + 2 * T64;        // 2 stages
constexpr uint32_t OFF_B4 = OFF_V + 2 * T64;       // [M0 | S0 | CG | CU] bf16, each [64 o][64 i]
constexpr uint32_t OFF_E = OFF_B4 + 4 * T64;       // [64 t][64 o] e
constexpr uint32_t OFF_EG = OFF_E + T64;           // gamma_t e_t
constexpr uint32_t OFF_EU = OFF_EG + T64;          // u_t e_t
constexpr uint32_t OFF_P = OFF_EU + T64;           // [64 t][64 i]
constexpr uint32_t OFF_GM = OFF_P + T64;           // fp32 Gamma [64][GS]
constexpr uint32_t OFF_M0F = OFF_GM + 64 * GS * 4; // fp32 chunk-start M [64][GS]
constexpr uint32_t OFF_S0F = OFF_M0F + 64 * GS * 4;
constexpr uint32_t OFF_F = OFF_S0F + 64 * GS * 4;  // gates [2][4][64]; p, w, r, A, sigma, gamma, u [64]
constexpr uint32_t N_F = 2 * 4 * SB + 7 * SB + 4 * SB;  // + surprise partials [2 halves][e2, k2][64]
constexpr uint32_t OFF_BAR = OFF_F + 4 * N_F;
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t COL_CG = 0, COL_CU = 64;
constexpr uint32_t COL_YH = 128, COL_QK = 192;  // batch 1
constexpr uint32_t COL_Y4 = 128, COL_PE = 384;  // batch 2
constexpr uint32_t ID_64 = idesc_bf16_f32(64, 64, false, false);
constexpr uint32_t ID_Y4 = idesc_bf16_f32(64, 256, false, false);
constexpr uint32_t ID_PE = idesc_bf16_f32(64, 64, false, true);
constexpr uint32_t ID_UPD = idesc_bf16_f32(64, 64, true, true);
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s

// Shared-memory descriptors (sw128_desc fields), K-major and MN-major; the
// start-address field keeps bits 4..17 of the address.  A k-step adds +2
// (32 bytes, K-major) or +128 (16 rows, MN-major).
constexpr uint64_t desc_hi(uint32_t lbo) {
    return (static_cast<uint64_t>(lbo >> 4) << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return desc_hi(16) | ((a >> 4) & 0x3FFFu); }
__device__ __forceinline__ uint64_t mdesc(uint32_t a) { return desc_hi(T64) | ((a >> 4) & 0x3FFFu); }
constexpr uint64_t KS_K = 2, KS_M = 128;

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}

__device__ __forceinline__ void get_row32(const unsigned char* tile, uint32_t r, uint32_t c0, float* v) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 w = ld_shared_v4(base + sw128_offset(r, c0 + 8 * q, 64));
        v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
        v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
        v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
        v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
    }
}

template <typename Tout>
__device__ __forceinline__ void store_row32(Tout* p, const float* v);
template <>
__device__ __forceinline__ void store_row32<__nv_bfloat16>(__nv_bfloat16* p, const float* v) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        reinterpret_cast<uint4*>(p)[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                                                    pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}
template <>
__device__ __forceinline__ void store_row32<float>(float* p, const float* v) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(p)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// OPT: bit 0 = write the surprise (a.surprise), bit 1 = Huber loss (clip e); compiled
// variants, so that the plain forward carries neither.
template <int NB, typename Tout, int OPT>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_linear64_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, nm_args a, int c_mode) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gates = reinterpret_cast<float*>(sm + OFF_F);  // [2 stages][a, eta, beta, c][64]
    float* sP = gates + 2 * 4 * SB;                       // block-level p_t
    float* sW = sP + SB;                                  // w_t
    float* sR = sW + SB;                                  // r_t
    float* sA = sR + SB;                                  // chunk-level A_t
    float* sSg = sA + SB;                                 // chunk-level sigma_t
    float* sGl = sSg + SB;                                // gamma_i of the block
    float* sU = sGl + SB;                                 // u_i of the block
    float* sPart = sU + SB;                               // surprise partial sums: [hf][||e||^2 | ||k||^2][64]
    float* Gm = reinterpret_cast<float*>(sm + OFF_GM);
    float* M0f = reinterpret_cast<float*>(sm + OFF_M0F);
    float* S0f = reinterpret_cast<float*>(sm + OFF_S0F);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // 0,1: tile stages; 2: mma
    __shared__ uint32_t s_tmem;
    __shared__ float s_end[3];  // chunk-level A, B, sigma at the block's last token

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int qd = warp & 3;
    const int hf = warp >> 2;
    const long long unit = blockIdx.x;
    const long long T = a.T;
    const long long P = (long long)D * D;
    const int nblocks = (int)((T + SB - 1) / SB);
    const float* alpha = a.alpha + unit * T;
    const float* eta = a.eta + unit * T;
    const float* beta = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    Tout* y = reinterpret_cast<Tout*>(a.y) + unit * T * D;
    const int rr = 16 * qd + (lane & 15);  // row of an M=64 accumulator (lanes 0..15 of the quadrant)
    const bool r64 = lane < 16;
    const int c0 = 32 * hf;                // this thread's 32 columns of a 64-column block

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    auto issue_tiles = [&](int blk, int stage) {
        mbar_arrive_expect_tx(&bars[stage], 3 * T64);
        const int t0 = blk * SB;
        tma_load_3d(sm + OFF_Q + stage * T64, &tq, &bars[stage], 0, t0, (int)unit);
        tma_load_3d(sm + OFF_K + stage * T64, &tk, &bars[stage], 0, t0, (int)unit);
        tma_load_3d(sm + OFF_V + stage * T64, &tv, &bars[stage], 0, t0, (int)unit);
    };
    if (tid < SB) {  // gates of block 0; tokens past T change nothing: a = 1, eta = 0, beta = 1, c = 0
        const long long t = tid;
        const bool ok = t < T;
        const float b = ok ? beta[t] : 1.0f;
        gates[tid] = ok ? 1.0f - alpha[t] : 1.0f;
        gates[SB + tid] = ok ? eta[t] : 0.0f;
        gates[2 * SB + tid] = b;
        gates[3 * SB + tid] = ok ? momentum_c(c_mode, b, cc, t) : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)(32 * qd) << 16);
    if (tid == 0 && nblocks > 0 && !a.skip_first_load) issue_tiles(0, 0);  // (the test hook skips it)

    // the chunk-start state: fp32 and bf16 copies of M0, S0; CG = CU = 0
    {
        const float* m0 = a.M0 + unit * P;
        const float* s0 = a.S0 + unit * P;
        for (int idx = tid; idx < 64 * 16; idx += NTHREADS) {  // 4 consecutive elements each
            const int o = idx >> 4, i4 = (idx & 15) * 4;
            const float4 m = *reinterpret_cast<const float4*>(m0 + o * D + i4);
            const float4 s = *reinterpret_cast<const float4*>(s0 + o * D + i4);
            *reinterpret_cast<float4*>(M0f + o * GS + i4) = m;
            *reinterpret_cast<float4*>(S0f + o * GS + i4) = s;
        }
        __syncthreads();
        if (tid < 64) {  // bf16 rows: M0, S0 from the fp32 copies; CG, CU zero
            float v[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = M0f[tid * GS + 32 * h + q];
                put_row32(sm + OFF_B4, 64, tid, 32 * h, v);
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = S0f[tid * GS + 32 * h + q];
                put_row32(sm + OFF_B4 + T64, 64, tid, 32 * h, v);
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] = 0.0f;
                put_row32(sm + OFF_B4 + 2 * T64, 64, tid, 32 * h, v);
                put_row32(sm + OFF_B4 + 3 * T64, 64, tid, 32 * h, v);
            }
        }
        float z[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) z[q] = 0.0f;
        tmem_st32(tl + COL_CG + c0, z);
        tmem_st32(tl + COL_CU + c0, z);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t aB4 = smem_u32(sm + OFF_B4), aE = smem_u32(sm + OFF_E), aEG = smem_u32(sm + OFF_EG);
    const uint32_t aEU = smem_u32(sm + OFF_EU), aP = smem_u32(sm + OFF_P);

    bool failed = false;
    uint32_t mma_phase = 0;
    auto mma_wait = [&](bool committed) {
        bool ok = true;
        if (committed) {
            ok = mbar_wait(&bars[2], mma_phase, WAIT_NS);
            mma_phase ^= 1u;
        }
        failed = __syncthreads_or(!ok) || failed;
        tc_fence_after();
    };
    auto handoff = [&]() {
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    float carA = 1.0f, carB = 1.0f, carS = 0.0f;  // chunk-level A, B, sigma before the block (thread 224)
    for (int g = 0; g < nblocks; ++g) {
        const int stage = g & 1;
        const int s = g % NB;                       // block within the chunk
        const bool chunk_end = s == NB - 1 || g + 1 == nblocks;
        const long long t0 = (long long)g * SB;
        const int n = (int)min((long long)SB, T - t0);
        // the gated output: this block's y_attn rows into L2 for the epilogue's loads
        if (a.y_attn) nm_prefetch_attn(a, (unit * T + t0) * D * (long long)sizeof(Tout), (long long)n * D * sizeof(Tout),
                                       tid, NTHREADS);
        const float* gt = gates + stage * 4 * SB;
        const uint32_t aQ = smem_u32(sm + OFF_Q + stage * T64), aK = smem_u32(sm + OFF_K + stage * T64);

        // the next block's gates (warps 2-3), stored after batch 1
        const int gi = tid - 64;
        const bool nxt_valid = gi >= 0 && gi < SB && g + 1 < nblocks && t0 + SB + gi < T;
        float nxt_al = 0.0f, nxt_e = 0.0f, nxt_b = 1.0f, nxt_c = 0.0f;
        if (nxt_valid) {
            const long long t = t0 + SB + gi;
            nxt_al = alpha[t];
            nxt_e = eta[t];
            nxt_b = beta[t];
            if (c_mode == NM_C_PER_TOKEN) nxt_c = cc[t];
        }

        // ---- batch 1 (thread 0): yhat = K M0^T, Q K^T; the next block's tiles; meanwhile the scan
        bool tiles_ok = true;
        if (tid == 0 && !failed) {
            tiles_ok = mbar_wait(&bars[stage], (uint32_t)((g >> 1) & 1), WAIT_NS);
            if (tiles_ok) {
                tc_fence_after();
                const uint64_t dQ = kdesc(aQ), dK = kdesc(aK), dM = kdesc(aB4);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t acc = ks ? 1u : 0u;
                    mma_bf16(tm + COL_YH, dK + KS_K * ks, dM + KS_K * ks, ID_64, acc);
                    mma_bf16(tm + COL_QK, dQ + KS_K * ks, dK + KS_K * ks, ID_64, acc);
                }
                mma_commit(&bars[2]);
                if (g + 1 < nblocks) issue_tiles(g + 1, stage ^ 1);
            }
        }
        if (tid >= 128 && tid < 128 + SB) {
            // column i of the block's Gamma (division-free recursion), gamma_i, u_i
            const int i = tid - 128;
            // from row 0 with u = Gamma = 0 and the start injected,
            // u_t = beta_t u_{t-1} + [t = i] c_i: zero above the diagonal, no branch per row;
            // the next four gates are loaded before this group's stores
            const float ci = gt[3 * SB + i];
            float u = 0.0f, G = 0.0f;
            const float4* g4 = reinterpret_cast<const float4*>(gt);
            float4 va = g4[0], ve = g4[SB / 4], vb = g4[SB / 2];
#pragma unroll
            for (int t4 = 0; t4 < SB / 4; ++t4) {
                const float ga[4] = {va.x, va.y, va.z, va.w}, ge[4] = {ve.x, ve.y, ve.z, ve.w},
                            gb[4] = {vb.x, vb.y, vb.z, vb.w};
                if (t4 + 1 < SB / 4) {
                    va = g4[t4 + 1];
                    ve = g4[SB / 4 + t4 + 1];
                    vb = g4[SB / 2 + t4 + 1];
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
            // block-level p, w, r and the chunk-level A, sigma of each token
            if (s == 0) {
                carA = 1.0f;
                carB = 1.0f;
                carS = 0.0f;
            }
            float p = 1.f, w = 1.f, r = 0.f;
            const float4* g4 = reinterpret_cast<const float4*>(gt);
#pragma unroll
            for (int t4 = 0; t4 < SB / 4; ++t4) {
                const float4 va = g4[t4], ve = g4[SB / 4 + t4], vb = g4[SB / 2 + t4];
                const float ga[4] = {va.x, va.y, va.z, va.w}, ge[4] = {ve.x, ve.y, ve.z, ve.w},
                            gb[4] = {vb.x, vb.y, vb.z, vb.w};
                float op[4], ow[4], orr[4], oA[4], oS[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    p *= ga[k];
                    w *= gb[k];
                    r = fmaf(ga[k], r, ge[k] * w);
                    op[k] = p;
                    ow[k] = w;
                    orr[k] = r;
                    oA[k] = carA * p;
                    oS[k] = fmaf(carS, p, carB * r);
                }
                reinterpret_cast<float4*>(sP)[t4] = make_float4(op[0], op[1], op[2], op[3]);
                reinterpret_cast<float4*>(sW)[t4] = make_float4(ow[0], ow[1], ow[2], ow[3]);
                reinterpret_cast<float4*>(sR)[t4] = make_float4(orr[0], orr[1], orr[2], orr[3]);
                reinterpret_cast<float4*>(sA)[t4] = make_float4(oA[0], oA[1], oA[2], oA[3]);
                reinterpret_cast<float4*>(sSg)[t4] = make_float4(oS[0], oS[1], oS[2], oS[3]);
            }
            const float nA = carA * p, nB = carB * w, nS = fmaf(carS, p, carB * r);
            carA = nA;
            carB = nB;
            carS = nS;
            s_end[0] = nA;
            s_end[1] = nB;
            s_end[2] = nS;
        }
        const bool go1 = !failed && !__syncthreads_or(!tiles_ok);
        if (!go1 && !failed) failed = true;
        // carry the earlier blocks over this block: CG <- p_end CG + r_end CU, CU <- w_end CU
        // (TMEM access is warp-wide; lanes 16..31 of a quadrant hold no rows and rewrite what they read)
        {
            const float pe = sP[SB - 1], we = sW[SB - 1], re = sR[SB - 1];
            float cg[32], cu[32];
            tmem_ld32x2(tl + COL_CG + c0, tl + COL_CU + c0, cg, cu);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                cg[q] = fmaf(pe, cg[q], re * cu[q]);
                cu[q] = we * cu[q];
            }
            tmem_st32(tl + COL_CG + c0, cg);
            tmem_st32(tl + COL_CU + c0, cu);
        }
        mma_wait(go1);
        // ---- e_t = 2 (M0 k_t - v_t), gamma_t e_t, u_t e_t; P = Gamma (.) Q K^T (rows t, columns c0 ..)
        {
            float e[32], qk[32];
            tmem_ld32x2(tl + COL_YH + c0, tl + COL_QK + c0, e, qk);
            if (r64) {
                const int t = rr;
                const bool live = t < n;
                float vv[32], o[32];
                get_row32(sm + OFF_V + stage * T64, t, c0, vv);
#pragma unroll
                for (int q = 0; q < 32; ++q) e[q] = live ? 2.0f * (e[q] - vv[q]) : 0.0f;
                if (OPT & 2) {  // the Huber loss clips e
#pragma unroll
                    for (int q = 0; q < 32; ++q) e[q] = nm_clip_err(e[q], a.e_clip);
                }
                if (OPT & 1) {  // partial ||e_t||^2, ||k_t||^2 over this thread's 32 columns
                    float kv[32], e2 = 0.0f, k2 = 0.0f;
                    get_row32(sm + OFF_K + stage * T64, t, c0, kv);
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        e2 = fmaf(e[q], e[q], e2);
                        k2 = fmaf(kv[q], kv[q], k2);
                    }
                    sPart[hf * 2 * SB + t] = e2;
                    sPart[hf * 2 * SB + SB + t] = k2;
                }
                put_row32(sm + OFF_E, 64, t, c0, e);
                const float gm = sGl[t], uu = sU[t];
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = gm * e[q];
                put_row32(sm + OFF_EG, 64, t, c0, o);
#pragma unroll
                for (int q = 0; q < 32; ++q) o[q] = uu * e[q];
                put_row32(sm + OFF_EU, 64, t, c0, o);
                const float* gr = Gm + t * GS + c0;
#pragma unroll
                for (int q = 0; q < 32; q += 4) {
                    const float4 gg = *reinterpret_cast<const float4*>(gr + q);
                    qk[q] *= gg.x; qk[q + 1] *= gg.y; qk[q + 2] *= gg.z; qk[q + 3] *= gg.w;
                }
                put_row32(sm + OFF_P, 64, t, c0, qk);
            }
        }
        if (gi >= 0 && gi < SB && g + 1 < nblocks) {
            float* gn = gates + (stage ^ 1) * 4 * SB;
            gn[gi] = nxt_valid ? 1.0f - nxt_al : 1.0f;
            gn[SB + gi] = nxt_e;
            gn[2 * SB + gi] = nxt_b;
            gn[3 * SB + gi] = !nxt_valid ? 0.0f
                              : c_mode == NM_C_ONE_MINUS_BETA ? 1.0f - nxt_b
                              : c_mode == NM_C_PER_TOKEN ? nxt_c : 1.0f;
        }
        handoff();
        if ((OPT & 1) && hf == 0 && r64 && rr < n)  // surprise_t = ||e_t|| ||k_t|| (gradient at the chunk start)
            a.surprise[unit * T + t0 + rr] = sqrtf(sPart[rr] + sPart[2 * SB + rr]) * sqrtf(sPart[SB + rr] + sPart[3 * SB + rr]);
        // ---- batch 2: Q [M0 | S0 | CG | CU]^T, P E, CG += (gamma E)^T K, CU += (u E)^T K
        const bool go2 = !failed;
        if (go2 && tid == 0) {
            const uint64_t dQ = kdesc(aQ), dB4 = kdesc(aB4), dP = kdesc(aP);
            const uint64_t dE = mdesc(aE), dEG = mdesc(aEG), dEU = mdesc(aEU), dKm = mdesc(aK);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t acc = ks ? 1u : 0u;
                mma_bf16(tm + COL_Y4, dQ + KS_K * ks, dB4 + KS_K * ks, ID_Y4, acc);
                mma_bf16(tm + COL_PE, dP + KS_K * ks, dE + KS_M * ks, ID_PE, acc);
                mma_bf16(tm + COL_CG, dEG + KS_M * ks, dKm + KS_M * ks, ID_UPD, 1u);
                mma_bf16(tm + COL_CU, dEU + KS_M * ks, dKm + KS_M * ks, ID_UPD, 1u);
            }
            mma_commit(&bars[2]);
        }
        mma_wait(go2);
        // ---- y_t = A_t M0 q_t - sigma_t S0 q_t - p_t CG q_t - r_t CU q_t - (P E)_t (rows t, columns c0 ..)
        {
            float y1[32], y2[32], y3[32];
            tmem_ld32x3(tl + COL_Y4 + c0, tl + COL_Y4 + 64 + c0, tl + COL_Y4 + 128 + c0, y1, y2, y3);
            const int t = rr;
            const float At = sA[t], st = sSg[t], pt = sP[t], rt = sR[t];
#pragma unroll
            for (int q = 0; q < 32; ++q) y1[q] = fmaf(At, y1[q], -fmaf(st, y2[q], pt * y3[q]));
            tmem_ld32x2(tl + COL_Y4 + 192 + c0, tl + COL_PE + c0, y2, y3);
#pragma unroll
            for (int q = 0; q < 32; ++q) y1[q] -= fmaf(rt, y2[q], y3[q]);
            if (r64 && t < n) {
                if (a.y_attn) nm_gate_row<32>(a, y + (t0 + t) * D + c0, y1);
                store_row32<Tout>(y + (t0 + t) * D + c0, y1);
            }
        }
        // ---- CG, CU become the next block's operands; at the chunk's end, the new state
        {
            float cg[32], cu[32];
            tmem_ld32x2(tl + COL_CG + c0, tl + COL_CU + c0, cg, cu);
            if (r64) {
                const int o = rr;
                if (!chunk_end) {
                    put_row32(sm + OFF_B4 + 2 * T64, 64, o, c0, cg);
                    put_row32(sm + OFF_B4 + 3 * T64, 64, o, c0, cu);
                } else {
                    // M = A_n M0 - sigma_n S0 - CG,  S = B_n S0 + CU
                    const float An = s_end[0], Bn = s_end[1], sn = s_end[2];
                    float m[32], sv[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        m[q] = fmaf(An, M0f[o * GS + c0 + q], -fmaf(sn, S0f[o * GS + c0 + q], cg[q]));
                        sv[q] = fmaf(Bn, S0f[o * GS + c0 + q], cu[q]);
                    }
                    if (g + 1 == nblocks) {
                        float* mt = a.M_T + unit * P + o * D + c0;
                        float* stp = a.S_T + unit * P + o * D + c0;
#pragma unroll
                        for (int q = 0; q < 32; q += 4) {
                            *reinterpret_cast<float4*>(mt + q) = make_float4(m[q], m[q + 1], m[q + 2], m[q + 3]);
                            *reinterpret_cast<float4*>(stp + q) = make_float4(sv[q], sv[q + 1], sv[q + 2], sv[q + 3]);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 32; q += 4) {
                            *reinterpret_cast<float4*>(M0f + o * GS + c0 + q) = make_float4(m[q], m[q + 1], m[q + 2], m[q + 3]);
                            *reinterpret_cast<float4*>(S0f + o * GS + c0 + q) = make_float4(sv[q], sv[q + 1], sv[q + 2], sv[q + 3]);
                        }
                        put_row32(sm + OFF_B4, 64, o, c0, m);
                        put_row32(sm + OFF_B4 + T64, 64, o, c0, sv);
                        float z[32];
#pragma unroll
                        for (int q = 0; q < 32; ++q) z[q] = 0.0f;
                        put_row32(sm + OFF_B4 + 2 * T64, 64, o, c0, z);
                        put_row32(sm + OFF_B4 + 3 * T64, 64, o, c0, z);
                    }
                }
            }
            if (chunk_end) {  // the next chunk starts with no earlier blocks: CG = CU = 0
                float z[32];
#pragma unroll
                for (int q = 0; q < 32; ++q) z[q] = 0.0f;
                tmem_st32(tl + COL_CG + c0, z);
                tmem_st32(tl + COL_CU + c0, z);
            }
        }
        handoff();
    }
    if (failed) {
        if (tid == 0 && a.status) atomicExch(a.status, NM_ERR_DEVICE_TIMEOUT);
        for (int i = 0; i < 2; ++i) mbar_wait(&bars[i], 0, WAIT_NS / 4);
        mbar_wait(&bars[2], mma_phase, WAIT_NS);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <int NB, typename Tout, int OPT>
cudaError_t launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    const long long units = (long long)a.B * a.H;
    if (!make_token_map(&tq, a.q, D, a.T, units) || !make_token_map(&tk, a.k, D, a.T, units) ||
        !make_token_map(&tv, a.v, D, a.T, units))
        return cudaErrorInvalidValue;
    auto kern = tc_linear64_kernel<NB, Tout, OPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)units, NTHREADS, SMEM_BYTES, s>>>(tq, tk, tv, a, c.c_mode);
    return cudaGetLastError();
}

template <int NB>
cudaError_t launch_nb(const nm_config& c, const nm_args& a, cudaStream_t s) {
    const int opt = (a.surprise ? 1 : 0) | (a.e_clip < HUGE_VALF ? 2 : 0);
    if (c.out_dtype == NM_BF16) {
        switch (opt) {
            case 0: return launch<NB, __nv_bfloat16, 0>(c, a, s);
            case 1: return launch<NB, __nv_bfloat16, 1>(c, a, s);
            case 2: return launch<NB, __nv_bfloat16, 2>(c, a, s);
            default: return launch<NB, __nv_bfloat16, 3>(c, a, s);
        }
    }
    switch (opt) {
        case 0: return launch<NB, float, 0>(c, a, s);
        case 1: return launch<NB, float, 1>(c, a, s);
        case 2: return launch<NB, float, 2>(c, a, s);
        default: return launch<NB, float, 3>(c, a, s);
    }
}

}  // namespace

bool nm_tc_linear64_supports(const nm_config& c) {
    return c.kind == NM_LINEAR && c.d == D && (c.chunk == 64 || c.chunk == 128 || c.chunk == 256) &&
           c.in_dtype == NM_BF16;
}

cudaError_t nm_tc_linear64_launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    if (c.chunk == 64) return launch_nb<1>(c, a, s);
    if (c.chunk == 128) return launch_nb<2>(c, a, s);
    return launch_nb<4>(c, a, s);
}
