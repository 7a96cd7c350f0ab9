// tcgen05 tensor-core kernel for the linear memory, d = 128, chunk b = 64.
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
//   Gamma_{t,i} = c_i sum_{j=i..t} (prod_{l=j+1..t} a_l) eta_j (prod_{l=i+1..j} beta_l),
//   gamma_i = Gamma_{n-1,i},  u_i = c_i prod_{l=i+1..n-1} beta_l,
// and E = 2 (K W0^T - V) (one row per token), the chunk is
//   Y^T   = M0 Q^T diag(A) - S0 Q^T diag(sigma) - E^T (Gamma (.) Q K^T)^T
//   M_end = A_{n-1} M0 - sigma_{n-1} S0 - E^T diag(gamma) K
//   S_end = B_{n-1} S0 + E^T diag(u) K.
// Gamma is built per row by a division-free recursion over i = t, t-1, ..., 0:
//   R <- eta_t;  R <- (prod a) eta_i + beta_{i+1} R;  Gamma_{t,i} = c_i R,
// so beta = 0 and alpha = 1 are exact.
//
// Data placement (one CTA, 4 warps; thread 0 issues TMA and MMA):
//   TMEM (512 columns x 128 lanes, fp32): M [lane o][col i] 0..127,
//     S 128..255, E^T accumulator 256..319, M0 Q^T 320..383, S0 Q^T 384..447,
//     Q K^T (M=64 layout) then E^T P^T 448..511.
//   SMEM: Q, K, V tiles (TMA, 128-byte swizzle, double-buffered), bf16
//     copies of M and S (the state as a tensor-core operand), E^T, -E^T
//     diag(gamma), E^T diag(u), P = Gamma (.) Q K^T, gates and scan values.
// The state never leaves the chip between chunks; HBM traffic is the q, k,
// v tiles in, y out, the gates, and the state once in and once out.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "nm_internal.h"
#include "tc_common.cuh"

namespace {

using namespace tc;

constexpr int D = 128;
constexpr int BC = 64;
constexpr int NTHREADS = 128;
constexpr uint32_t HALF = BC * 128;       // one 64-column block of a 64-row tile
constexpr uint32_t TILE = 2 * HALF;       // 64 tokens x 128 features, bf16
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;
constexpr uint32_t OFF_V = OFF_K + 2 * TILE;
constexpr uint32_t OFF_MH = OFF_V + 2 * TILE;  // [128][128] bf16: two 16 KB blocks
constexpr uint32_t OFF_SH = OFF_MH + 32768;
constexpr uint32_t OFF_ET = OFF_SH + 32768;    // [128][64] bf16
constexpr uint32_t OFF_EG = OFF_ET + 16384;
constexpr uint32_t OFF_EU = OFF_EG + 16384;
constexpr uint32_t OFF_P = OFF_EU + 16384;     // [64][64] bf16
constexpr uint32_t OFF_F = OFF_P + 8192;       // floats
constexpr uint32_t N_FLOATS = 2 * 4 * BC + 5 * BC;
constexpr uint32_t OFF_BAR = OFF_F + 4 * N_FLOATS;
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t COL_M = 0, COL_S = 128, COL_E = 256, COL_Y1 = 320, COL_Y2 = 384, COL_QK = 448;
constexpr uint32_t ID_128x64 = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t ID_64x64 = idesc_bf16_f32(64, 64, false, false);
constexpr uint32_t ID_128x128_BMN = idesc_bf16_f32(128, 128, false, true);
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s

template <typename Tout>
__device__ __forceinline__ void store_y(Tout* p, float x);
template <>
__device__ __forceinline__ void store_y<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ void store_y<float>(float* p, float x) { *p = x; }

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}

template <typename Tout>
__global__ void __launch_bounds__(NTHREADS, 1)
    tc_linear_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, nm_args a, int c_mode) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gates = reinterpret_cast<float*>(sm + OFF_F);  // [2 stages][a, eta, beta, c][64]
    float* sA = gates + 2 * 4 * BC;
    float* sBc = sA + BC;
    float* sSg = sBc + BC;
    float* sGl = sSg + BC;
    float* sU = sGl + BC;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);  // 0,1: tile stages; 2: mma
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const long long unit = blockIdx.x;
    const long long T = a.T;
    const long long P = (long long)D * D;
    const int nchunks = (int)((T + BC - 1) / BC);
    const float* alpha = a.alpha + unit * T;
    const float* eta = a.eta + unit * T;
    const float* beta = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    Tout* y = reinterpret_cast<Tout*>(a.y) + unit * T * D;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s_tmem;
    const uint32_t lb = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quadrant

    auto issue_tiles = [&](int chunk, int stage) {
        mbar_arrive_expect_tx(&bars[stage], 3 * TILE);
        const int t0 = chunk * BC;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            tma_load_3d(sm + OFF_Q + stage * TILE + h * HALF, &tq, &bars[stage], h * 64, t0, (int)unit);
            tma_load_3d(sm + OFF_K + stage * TILE + h * HALF, &tk, &bars[stage], h * 64, t0, (int)unit);
            tma_load_3d(sm + OFF_V + stage * TILE + h * HALF, &tv, &bars[stage], h * 64, t0, (int)unit);
        }
    };
    auto load_gates = [&](int chunk, int stage) {
        if (tid < BC) {
            const long long t = (long long)chunk * BC + tid;
            float* g = gates + stage * 4 * BC;
            if (t < T) {
                const float b = beta[t];
                g[tid] = 1.0f - alpha[t];
                g[BC + tid] = eta[t];
                g[2 * BC + tid] = b;
                g[3 * BC + tid] = momentum_c(c_mode, b, cc, t);
            } else {
                g[tid] = 1.0f;
                g[BC + tid] = 0.0f;
                g[2 * BC + tid] = 0.0f;
                g[3 * BC + tid] = 0.0f;
            }
        }
    };

    if (tid == 0 && nchunks > 0) issue_tiles(0, 0);
    load_gates(0, 0);
    // initial state: TMEM fp32 (lane o = row o of M, S) and bf16 operand copies
    {
        float r[32];
        const float* m0 = a.M0 + unit * P + (long long)tid * D;
        const float* s0 = a.S0 + unit * P + (long long)tid * D;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int q = 0; q < 32; q += 4) {
                float4 w = *reinterpret_cast<const float4*>(m0 + 32 * j + q);
                r[q] = w.x; r[q + 1] = w.y; r[q + 2] = w.z; r[q + 3] = w.w;
            }
            tmem_st32(tm + lb + COL_M + 32 * j, r);
            put_row32(sm + OFF_MH, 128, tid, 32 * j, r);
#pragma unroll
            for (int q = 0; q < 32; q += 4) {
                float4 w = *reinterpret_cast<const float4*>(s0 + 32 * j + q);
                r[q] = w.x; r[q + 1] = w.y; r[q + 2] = w.z; r[q + 3] = w.w;
            }
            tmem_st32(tm + lb + COL_S + 32 * j, r);
            put_row32(sm + OFF_SH, 128, tid, 32 * j, r);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    uint32_t mma_phase = 0;
    bool failed = false;
    int c = 0;
    for (; c < nchunks; ++c) {
        const int stage = c & 1;
        const long long t0 = (long long)c * BC;
        const int n = (int)min((long long)BC, T - t0);
        const float* g = gates + stage * 4 * BC;
        if (c + 1 < nchunks) {
            if (tid == 0) issue_tiles(c + 1, stage ^ 1);
            load_gates(c + 1, stage ^ 1);
        }
        // chunk scan: A, B, sigma (thread 0); gamma, u by the row recursion (thread 32)
        if (tid == 0) {
            float A = 1.f, Bc = 1.f, sg = 0.f;
            for (int t = 0; t < n; ++t) {
                A *= g[t];
                Bc *= g[2 * BC + t];
                sg = fmaf(g[t], sg, g[BC + t] * Bc);
                sA[t] = A;
                sBc[t] = Bc;
                sSg[t] = sg;
            }
        }
        if (tid == 32) {
            float Dp = 1.f, R = g[BC + n - 1], Bp = 1.f;
            sGl[n - 1] = g[3 * BC + n - 1] * R;
            sU[n - 1] = g[3 * BC + n - 1];
            for (int i = n - 2; i >= 0; --i) {
                Dp *= g[i + 1];
                R = fmaf(Dp, g[BC + i], g[2 * BC + i + 1] * R);
                Bp *= g[2 * BC + i + 1];
                sGl[i] = g[3 * BC + i] * R;
                sU[i] = g[3 * BC + i] * Bp;
            }
            for (int i = n; i < BC; ++i) {
                sGl[i] = 0.f;
                sU[i] = 0.f;
            }
        }
        // wait for this chunk's tiles
        bool ok = mbar_wait(&bars[stage], (uint32_t)((c >> 1) & 1), WAIT_NS);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        const uint32_t qa = smem_u32(sm + OFF_Q + stage * TILE);
        const uint32_t ka = smem_u32(sm + OFF_K + stage * TILE);
        if (tid == 0) {
            tc_fence_after();
            const uint32_t mh = smem_u32(sm + OFF_MH), sh = smem_u32(sm + OFF_SH);
#pragma unroll
            for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t acc = (kb | ks) ? 1u : 0u;
                    const uint32_t ko = kb * HALF + ks * 32;      // 64-row tiles
                    const uint32_t mo = kb * 16384 + ks * 32;     // 128-row tiles
                    mma_bf16(tm + COL_E, sw128_desc(mh + mo, 16, 1024), sw128_desc(ka + ko, 16, 1024), ID_128x64, acc);
                    mma_bf16(tm + COL_Y1, sw128_desc(mh + mo, 16, 1024), sw128_desc(qa + ko, 16, 1024), ID_128x64, acc);
                    mma_bf16(tm + COL_Y2, sw128_desc(sh + mo, 16, 1024), sw128_desc(qa + ko, 16, 1024), ID_128x64, acc);
                    mma_bf16(tm + COL_QK, sw128_desc(qa + ko, 16, 1024), sw128_desc(ka + ko, 16, 1024), ID_64x64, acc);
                }
            mma_commit(&bars[2]);
        }
        // rescale the fp32 state for this chunk: M <- A M - sigma S, S <- B S
        {
            const float An = sA[n - 1], Bn = sBc[n - 1], sn = sSg[n - 1];
            float m[32], s[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                tmem_ld32(tm + lb + COL_M + 32 * j, m);
                tmem_ld32(tm + lb + COL_S + 32 * j, s);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    m[q] = fmaf(An, m[q], -sn * s[q]);
                    s[q] = Bn * s[q];
                }
                tmem_st32(tm + lb + COL_M + 32 * j, m);
                tmem_st32(tm + lb + COL_S + 32 * j, s);
            }
        }
        ok = mbar_wait(&bars[2], mma_phase, WAIT_NS);
        mma_phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc_fence_after();
        // errors e_t = 2 (W0 k_t - v_t): lane o holds E^T[o][t]
        {
            const unsigned char* vt = sm + OFF_V + stage * TILE;
            float acc[32], e[32], eg[32], eu[32];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                tmem_ld32(tm + lb + COL_E + 32 * j, acc);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int t = 32 * j + q;
                    const float vv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(vt + sw128_offset(t, tid, BC)));
                    const float ev = t < n ? 2.0f * (acc[q] - vv) : 0.0f;
                    e[q] = ev;
                    eg[q] = -ev * sGl[t];
                    eu[q] = ev * sU[t];
                }
                put_row32(sm + OFF_ET, 128, tid, 32 * j, e);
                put_row32(sm + OFF_EG, 128, tid, 32 * j, eg);
                put_row32(sm + OFF_EU, 128, tid, 32 * j, eu);
            }
        }
        // P = Gamma (.) Q K^T; the M=64 accumulator holds row r at lane (r % 16) + 32 (r / 16)
        {
            float qk0[32], qk1[32];
            tmem_ld32(tm + lb + COL_QK, qk0);
            tmem_ld32(tm + lb + COL_QK + 32, qk1);
            if (lane < 16) {
                const int t = warp * 16 + lane;
                float p[64];
                float Dp = 1.f, R = 0.f;
#pragma unroll
                for (int i = BC - 1; i >= 0; --i) {
                    if (i == t) {
                        R = g[BC + t];
                        Dp = 1.f;
                    } else if (i < t) {
                        Dp *= g[i + 1];
                        R = fmaf(Dp, g[BC + i], g[2 * BC + i + 1] * R);
                    }
                    const float qkv = i < 32 ? qk0[i & 31] : qk1[i & 31];
                    p[i] = (i <= t && t < n) ? g[3 * BC + i] * R * qkv : 0.0f;
                }
                put_row32(sm + OFF_P, BC, t, 0, p);
                put_row32(sm + OFF_P, BC, t, 32, p + 32);
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t et = smem_u32(sm + OFF_ET), eg = smem_u32(sm + OFF_EG), eu = smem_u32(sm + OFF_EU);
            const uint32_t pa = smem_u32(sm + OFF_P);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t acc = ks ? 1u : 0u;
                mma_bf16(tm + COL_QK, sw128_desc(et + ks * 32, 16, 1024), sw128_desc(pa + ks * 32, 16, 1024), ID_128x64, acc);
                mma_bf16(tm + COL_M, sw128_desc(eg + ks * 32, 16, 1024), sw128_desc(ka + ks * 2048, HALF, 1024),
                         ID_128x128_BMN, 1u);
                mma_bf16(tm + COL_S, sw128_desc(eu + ks * 32, 16, 1024), sw128_desc(ka + ks * 2048, HALF, 1024),
                         ID_128x128_BMN, 1u);
            }
            mma_commit(&bars[2]);
        }
        ok = mbar_wait(&bars[2], mma_phase, WAIT_NS);
        mma_phase ^= 1u;
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        tc_fence_after();
        // retrieval: y_t[o] = A_t (M0 q_t)[o] - sigma_t (S0 q_t)[o] - (E^T P^T)[o][t]
        {
            float y1[32], y2[32], y3[32];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                tmem_ld32(tm + lb + COL_Y1 + 32 * j, y1);
                tmem_ld32(tm + lb + COL_Y2 + 32 * j, y2);
                tmem_ld32(tm + lb + COL_QK + 32 * j, y3);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int t = 32 * j + q;
                    if (t < n) store_y(y + (t0 + t) * D + tid, fmaf(sA[t], y1[q], -fmaf(sSg[t], y2[q], y3[q])));
                }
            }
        }
        // state for the next chunk: bf16 operand copies (and the result after the last chunk)
        {
            const bool last = c + 1 == nchunks;
            float m[32], s[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                tmem_ld32(tm + lb + COL_M + 32 * j, m);
                tmem_ld32(tm + lb + COL_S + 32 * j, s);
                if (!last) {
                    put_row32(sm + OFF_MH, 128, tid, 32 * j, m);
                    put_row32(sm + OFF_SH, 128, tid, 32 * j, s);
                } else {
                    float* mt = a.M_T + unit * P + (long long)tid * D + 32 * j;
                    float* st = a.S_T + unit * P + (long long)tid * D + 32 * j;
#pragma unroll
                    for (int q = 0; q < 32; q += 4) {
                        *reinterpret_cast<float4*>(mt + q) = make_float4(m[q], m[q + 1], m[q + 2], m[q + 3]);
                        *reinterpret_cast<float4*>(st + q) = make_float4(s[q], s[q + 1], s[q + 2], s[q + 3]);
                    }
                }
            }
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (failed) {
        if (tid == 0 && a.status) atomicExch(a.status, NM_ERR_DEVICE_TIMEOUT);
        // let copies and products still in flight land before the CTA leaves
        if (c + 1 < nchunks) mbar_wait(&bars[(c & 1) ^ 1], (uint32_t)(((c + 1) >> 1) & 1), WAIT_NS);
        mbar_wait(&bars[2], mma_phase, WAIT_NS);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <typename Tout>
cudaError_t launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    const long long units = (long long)a.B * a.H;
    if (!make_token_map(&tq, a.q, D, a.T, units) || !make_token_map(&tk, a.k, D, a.T, units) ||
        !make_token_map(&tv, a.v, D, a.T, units))
        return cudaErrorInvalidValue;
    auto kern = tc_linear_kernel<Tout>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)units, NTHREADS, SMEM_BYTES, s>>>(tq, tk, tv, a, c.c_mode);
    return cudaGetLastError();
}

}  // namespace

bool nm_tc_linear_supports(const nm_config& c) {
    return c.kind == NM_LINEAR && c.d == D && c.chunk == BC && c.in_dtype == NM_BF16;
}

cudaError_t nm_tc_linear_launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    return c.out_dtype == NM_BF16 ? launch<__nv_bfloat16>(c, a, s) : launch<float>(c, a, s);
}
