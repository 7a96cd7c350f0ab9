// Backward pass of the chunked memory (the linear memory here, the 2-layer
// MLP memory further down): gradients of a loss of the forward's outputs
// (y, M_T, S_T) with respect to every input, for training
// what surrounds the memory ("Titans: Imparare a Memorizzare al Tempo di
// Test", "Addestramento Parallelizzato": the memory's inner loop written with
// matrix products so that the outer loop trains fast).
//
// Forward, per (batch, head) unit and chunk of n tokens with start state
// (Mc, Sc), a_t = 1 - alpha_t, and the scan quantities A_t, B_t, sigma_t,
// Gamma_{t,i}, u_{t,i} (see nm_tc_mlp.cu for their recursions):
//   e_i  = 2 clip(Mc k_i - v_i)                      (gradient at the chunk start)
//   y_t  = A_t Mc q_t - sigma_t Sc q_t - sum_{i<=t} Gamma_{t,i} (k_i . q_t) e_i
//   M_end = A_{n-1} Mc - sigma_{n-1} Sc - sum_i gamma_i e_i k_i^T
//   S_end = B_{n-1} Sc + sum_i u_i e_i k_i^T
// with gamma_i = Gamma_{n-1,i}, u_i = u_{n-1,i}.  Given the adjoints Gy_t of
// y_t and (GM, GS) of (M_end, S_end), reverse-mode differentiation of these
// expressions gives, with Z_{t,i} = Gy_t . e_i and QK_{t,i} = q_t . k_i:
//   lambda_e_i = - sum_{t>=i} Gamma_{t,i} QK_{t,i} Gy_t - gamma_i GM k_i + u_i GS k_i
//   lambda_r_i = 2 [|r_i| inside the clip] lambda_e_i  (r_i = Mc k_i - v_i),  dv_i = -lambda_r_i
//   dk_i = - sum_{t>=i} Gamma_{t,i} Z_{t,i} q_t - gamma_i GM^T e_i + u_i GS^T e_i + Mc^T lambda_r_i
//   dq_t = A_t Mc^T Gy_t - sigma_t Sc^T Gy_t - sum_{i<=t} Gamma_{t,i} Z_{t,i} k_i
//   dMc  = sum_t A_t Gy_t q_t^T + A_{n-1} GM + sum_i lambda_r_i k_i^T
//   dSc  = - sum_t sigma_t Gy_t q_t^T - sigma_{n-1} GM + B_{n-1} GS
// and scalar adjoints of the scan quantities (dL/dA_t = Gy_t . Mc q_t,
// dL/dsigma_t = -Gy_t . Sc q_t, dL/dGamma_{t,i} = -QK_{t,i} Z_{t,i}, plus the
// chunk-end terms <GM, Mc>, -<GM, Sc>, <GS, Sc>, -e_i . GM k_i, e_i . GS k_i),
// which the reverse of the scan recursions turns into gradients of the
// gates.  The chunk-start state's adjoint (dMc, dSc) is the (GM, GS) of the
// chunk before, so chunks are processed from the last to the first; their
// start states come from a forward pass that records them (the fp32 FFMA
// forward kernel with a checkpoint array).
//
// One CTA per unit, every step a block-wide loop over its output elements,
// matrices in a per-unit global workspace (read through L1 / L2).  The
// chunk-sized contractions run either as fp32 FFMA block GEMMs or, on the
// tensor-core path, as tcgen05 kind::tf32 products (operands rounded to tf32,
// fp32 accumulation in TMEM); everything else is the same fp32 code.
#include "nm_internal.h"
#include "tc_common.cuh"

namespace {

constexpr int BW_THREADS = 256;
constexpr int BW_MAX_CHUNK = 256;

struct bwd_args {
    long long T;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* eta;
    const float* beta;
    const float* c;
    const float* ckpt;  // [units][nchunks][2][P] chunk-start (M, S)
    const float* Gy;    // [units][T][d]
    const float* GM;    // [units][P]
    const float* GS;
    float* dq;          // [units][T][d]
    float* dk;
    float* dv;
    float* dalpha;      // [units][T]
    float* deta;
    float* dbeta;
    float* dc;          // [units][T] or NULL
    float* dM0;         // [units][P]
    float* dS0;
    float* ws;          // per-unit workspace
    size_t ws_unit;     // floats per unit
    float e_clip;
    int* status;        // device status word (a timed-out wait of the tensor-core contractions)
};

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}

// Runs store(i, load(i)) for every i in [0, N) over the block, U indices per
// thread at a time, the loads of all U issued before any store: the passes of
// the sweep read and write the same per-unit workspace, so in a plain loop
// each iteration's loads wait for the previous iteration's stores (a round
// trip to L2 per iteration).  The kernels with the register-tiled FFMA
// products take a smaller U, as far as it costs no spills: 2 for the linear
// memory, 1 (a plain loop) for the MLP memory.
template <int U, typename L, typename S>
__device__ __forceinline__ void each(int N, L&& load, S&& store) {
    using V = decltype(load(0));
    for (int i0 = threadIdx.x; i0 < N; i0 += U * BW_THREADS) {
        V v[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int i = i0 + j * BW_THREADS;
            if (i < N) v[j] = load(i);
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int i = i0 + j * BW_THREADS;
            if (i < N) store(i, v[j]);
        }
    }
}
struct F6 {
    float a, b, c, d, e, f;
};
struct F9 {
    float a, b, c, d, e, f, g, h, k;
};

// Sum over the warp, returned to every lane (all 32 lanes must call it).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) v += __shfl_xor_sync(0xffffffffu, v, sh);
    return v;
}

// Sum over the block (every thread passes its partial); the result is returned to all threads.
__device__ float block_sum(float v, float* red) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < BW_THREADS / 32; ++i) s += red[i];
    return s;
}

// ---------------------------------------------------------------- block GEMM (fp32 FFMA)
// C(m, n) = alpha sum_k A(m, k) B(k, n) [+ C(m, n) if accumulate], m < M, n < N, over the whole block.
// A(m, k) = A[m am + k ak], B(k, n) = B[k bk + n bn], C(m, n) = C[m cm + n].  Tiles of 64 x 64 outputs,
// K in steps of 16 staged in shared memory (loaded along whichever dimension is contiguous, so the global
// reads coalesce), 4 x 4 outputs per thread.  Ends with the block synchronised.
constexpr int GM_T = 64, GK_T = 16;
constexpr int GEMM_SMEM_FLOATS = 2 * GM_T * GK_T;

__device__ void block_gemm(int M, int N, int K, const float* A, long long am, long long ak, const float* B,
                           long long bk, long long bn, float* C, long long cm, float alpha, bool accumulate,
                           float* sh) {
    float* As = sh;                 // [GK_T][GM_T]
    float* Bs = sh + GM_T * GK_T;   // [GK_T][GM_T]
    const int tid = threadIdx.x;
    const int tr = tid >> 4, tc = tid & 15;
    for (int m0 = 0; m0 < M; m0 += GM_T) {
        for (int n0 = 0; n0 < N; n0 += GM_T) {
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
            for (int k0 = 0; k0 < K; k0 += GK_T) {
                __syncthreads();
                for (int e = tid; e < GM_T * GK_T; e += BW_THREADS) {
                    int mm, kk;
                    if (ak == 1) { mm = e / GK_T; kk = e % GK_T; } else { kk = e / GM_T; mm = e % GM_T; }
                    const int m = m0 + mm, k = k0 + kk;
                    As[kk * GM_T + mm] = (m < M && k < K) ? A[m * am + k * ak] : 0.f;
                    int nn, kb;
                    if (bn == 1) { kb = e / GM_T; nn = e % GM_T; } else { nn = e / GK_T; kb = e % GK_T; }
                    const int n = n0 + nn, kq = k0 + kb;
                    Bs[kb * GM_T + nn] = (n < N && kq < K) ? B[kq * bk + n * bn] : 0.f;
                }
                __syncthreads();
#pragma unroll
                for (int kk = 0; kk < GK_T; ++kk) {
                    const float4 a4 = *reinterpret_cast<const float4*>(As + kk * GM_T + 4 * tr);
                    const float4 b4 = *reinterpret_cast<const float4*>(Bs + kk * GM_T + 4 * tc);
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = m0 + 4 * tr + i;
                if (m >= M) continue;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = n0 + 4 * tc + j;
                    if (n >= N) continue;
                    float* c = C + m * cm + n;
                    *c = accumulate ? fmaf(alpha, acc[i][j], *c) : alpha * acc[i][j];
                }
            }
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- tensor-core contractions
// C(m, n) = alpha sum_k A(m, k) B(k, n) [+ C(m, n)] as tcgen05.mma kind::tf32
// products, the same contract as block_gemm: per pass up to 256 x 256
// outputs (two M = 128 tiles, N a multiple of 32) in TMEM; K in blocks of 32,
// each staged by all threads into shared memory as tf32 (rounded to nearest)
// in the 128-byte-swizzled K-major layout, double-buffered so that a block is
// staged while the previous one's products run; thread 0 issues the products
// (K = 8 each) and commits them to the stage's mbarrier; the epilogue reads
// the accumulators (row = TMEM lane) and writes C.  Every wait gives up after
// 2 s; the CTA then stops issuing products and reports NM_ERR_DEVICE_TIMEOUT.
constexpr uint32_t TG_ATILE = 128 * 128;               // 128 rows x 32 fp32 k
constexpr uint32_t TG_ASTAGE = 2 * TG_ATILE;           // up to 256 A rows
constexpr uint32_t TG_BSTAGE = 256 * 128;              // up to 256 B rows
constexpr uint32_t TG_SMEM = 2 * (TG_ASTAGE + TG_BSTAGE) + 64 + 1024;  // two stages, barriers, alignment
constexpr uint64_t TG_WAIT_NS = 2000000000ull;
constexpr int TG_U = 4;  // 16-byte chunks per thread whose loads are issued together

// tcgen05 instruction descriptor, kind::tf32: tf32 A and B (format 2), fp32
// accumulator, both K-major, M = 128.
__host__ __device__ constexpr uint32_t tg_idesc(uint32_t N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((128u >> 4) << 24);
}
__device__ __forceinline__ void tg_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ uint32_t tg_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

struct TcCtx {
    uint32_t a_st[2], b_st[2];  // shared addresses of the stages
    uint64_t* bars;             // [2] products of a stage completed
    uint32_t ph[2];             // completions waited per barrier
    uint32_t pending;           // bit s: a commit on bars[s] not waited for
    uint32_t tm;                // TMEM base
    int failed;
};

// Dynamic shared memory, barriers and 512 TMEM columns (every thread calls it).
__device__ void tg_setup(TcCtx& x) {
    extern __shared__ unsigned char tg_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(tg_raw) + 1023) & ~(uintptr_t)1023);
    x.a_st[0] = tc::smem_u32(sm);
    x.a_st[1] = x.a_st[0] + TG_ASTAGE;
    x.b_st[0] = x.a_st[1] + TG_ASTAGE;
    x.b_st[1] = x.b_st[0] + TG_BSTAGE;
    x.bars = reinterpret_cast<uint64_t*>(sm + 2 * (TG_ASTAGE + TG_BSTAGE));
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(x.bars + 2);
    if (threadIdx.x == 0) {
        tc::mbar_init(&x.bars[0], 1);
        tc::mbar_init(&x.bars[1], 1);
        tc::fence_mbar_init();
    }
    if (threadIdx.x < 32) {
        tc::tmem_alloc(s_tmem, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    x.tm = *s_tmem;
    x.ph[0] = x.ph[1] = 0;
    x.pending = 0;
    x.failed = 0;
}

__device__ void tg_teardown(TcCtx& x, int* status) {
    if (x.failed && threadIdx.x == 0 && status) atomicExch(status, NM_ERR_DEVICE_TIMEOUT);
    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) tc::tmem_dealloc(x.tm, 512);
}

// Stages columns k0 .. k0 + 31 of rows 0 .. R - 1 of an operand (element
// (r, k) = p[r sr + k sk], zero for r >= rv or k >= K) into a tile of R
// 128-byte rows, 16-byte chunk kc of row r at r * 128 + ((kc ^ (r % 8)) * 16).
// Consecutive threads take consecutive chunks of a row when k is contiguous,
// consecutive rows otherwise (coalesced loads either way).
__device__ __forceinline__ void tg_stage(uint32_t tile, int R, int rv, const float* p, long long sr, long long sk,
                                         int k0, int K, int tid) {
    const int n = R * 8;
    const bool kfast = sk == 1;
    for (int base = 0; base < n; base += BW_THREADS * TG_U) {
        float v[TG_U][4];
        int rr[TG_U], kc[TG_U];
#pragma unroll
        for (int u = 0; u < TG_U; ++u) {
            const int idx = base + u * BW_THREADS + tid;
            rr[u] = kfast ? idx >> 3 : idx % R;
            kc[u] = kfast ? idx & 7 : idx / R;
            const int k = k0 + 4 * kc[u];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[u][j] = (idx < n && rr[u] < rv && k + j < K) ? p[(long long)rr[u] * sr + (long long)(k + j) * sk] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < TG_U; ++u) {
            const int idx = base + u * BW_THREADS + tid;
            if (idx < n)
                tc::st_shared_v4(tile + (uint32_t)rr[u] * 128u + (((uint32_t)kc[u] ^ ((uint32_t)rr[u] & 7u)) << 4),
                                 tg_tf32(v[u][0]), tg_tf32(v[u][1]), tg_tf32(v[u][2]), tg_tf32(v[u][3]));
        }
    }
}

__device__ __forceinline__ bool tg_wait(TcCtx& x, int st) {
    if (!(x.pending >> st & 1u)) return true;
    const bool ok = tc::mbar_wait(&x.bars[st], x.ph[st] & 1u, TG_WAIT_NS);
    x.ph[st] += 1;
    x.pending &= ~(1u << st);
    return ok;
}

__device__ __noinline__ void tc_gemm(TcCtx& x, int M, int N, int K, const float* A, long long am, long long ak, const float* B,
                        long long bk, long long bn, float* C, long long cm, float alpha, bool accumulate) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int m0 = 0; m0 < M; m0 += 256) {
        const int mr = min(256, M - m0), mt = (mr + 127) >> 7;
        for (int n0 = 0; n0 < N; n0 += 256) {
            const int nr = min(256, N - n0), np = (nr + 31) & ~31;
            const uint32_t idesc = tg_idesc((uint32_t)np);
            bool bad = false;
            int kb = 0;
            for (int k0 = 0; k0 < K && !x.failed; k0 += 32, ++kb) {
                const int st = kb & 1;
                if (!tg_wait(x, st)) bad = true;
                tg_stage(x.a_st[st], 128 * mt, mr, A + (long long)m0 * am, am, ak, k0, K, tid);
                tg_stage(x.b_st[st], np, nr, B + (long long)n0 * bn, bn, bk, k0, K, tid);
                tc::fence_proxy_async();
                if (__syncthreads_or(bad)) {
                    x.failed = 1;
                    break;
                }
                if (tid == 0) {
                    tc::tc_fence_after();
                    for (int m = 0; m < mt; ++m) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tg_mma(x.tm + (uint32_t)(m * np),
                                   tc::sw128_desc(x.a_st[st] + (uint32_t)m * TG_ATILE + kk * 32, 16, 1024),
                                   tc::sw128_desc(x.b_st[st] + kk * 32, 16, 1024), idesc, (k0 > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc::mma_commit(&x.bars[st]);
                }
                x.pending |= 1u << st;
            }
            if (!tg_wait(x, 0)) bad = true;
            if (!tg_wait(x, 1)) bad = true;
            if (__syncthreads_or(bad)) x.failed = 1;
            tc::tc_fence_after();
            if (!x.failed) {
                const int q = warp & 3, hf = warp >> 2, half = np / 2;
                for (int m = 0; m < mt; ++m) {
                    const int gm = m0 + 128 * m + 32 * q + lane;
                    for (int c0 = hf * half; c0 < (hf + 1) * half; c0 += 16) {
                        float v[16];
                        tc::tmem_ld_n(x.tm + ((uint32_t)(32 * q) << 16) + (uint32_t)(m * np + c0), v);
                        if (gm < M) {
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const int gn = n0 + c0 + c;
                                if (gn < N) {
                                    float* cp = C + (long long)gm * cm + gn;
                                    *cp = accumulate ? fmaf(alpha, v[c], *cp) : alpha * v[c];
                                }
                            }
                        }
                    }
                }
            }
            tc::tc_fence_before();
            __syncthreads();
        }
    }
}

template <typename Tin, bool TC>
__global__ void __launch_bounds__(BW_THREADS) bwd_linear_kernel(bwd_args a, int d, int b, int c_mode) {
    __shared__ float s_a[BW_MAX_CHUNK], s_e[BW_MAX_CHUNK], s_b[BW_MAX_CHUNK], s_c[BW_MAX_CHUNK];
    __shared__ float sA[BW_MAX_CHUNK], sB[BW_MAX_CHUNK], sS[BW_MAX_CHUNK];
    __shared__ float s_gam[BW_MAX_CHUNK], s_u[BW_MAX_CHUNK];
    __shared__ float s_gA[BW_MAX_CHUNK], s_gS[BW_MAX_CHUNK], s_hg[BW_MAX_CHUNK], s_hu[BW_MAX_CHUNK];
    __shared__ float s_da[BW_MAX_CHUNK], s_de[BW_MAX_CHUNK], s_db[BW_MAX_CHUNK], s_dc[BW_MAX_CHUNK];
    __shared__ float red[BW_THREADS / 32];
    __shared__ __align__(16) float gsh[GEMM_SMEM_FLOATS];
    TcCtx tcx;
    if constexpr (TC) tg_setup(tcx);
    constexpr int EU = TC ? 4 : 2;  // elementwise passes: indices batched per thread
    // every chunk-sized contraction: tcgen05 tf32 products or fp32 FFMA block GEMMs
    auto gemm_ = [&](int M_, int N_, int K_, const float* A_, long long am_, long long ak_, const float* B_, long long bk_,
                     long long bn_, float* C_, long long cm_, float alpha_, bool acc_, float* sh_) {
        if constexpr (TC) tc_gemm(tcx, M_, N_, K_, A_, am_, ak_, B_, bk_, bn_, C_, cm_, alpha_, acc_);
        else block_gemm(M_, N_, K_, A_, am_, ak_, B_, bk_, bn_, C_, cm_, alpha_, acc_, sh_);
    };

    const long long unit = blockIdx.x;
    const int tid = threadIdx.x;
    const long long T = a.T;
    const int P = d * d;
    const int nch = (int)((T + b - 1) / b);
    const Tin* q = reinterpret_cast<const Tin*>(a.q) + unit * T * d;
    const Tin* k = reinterpret_cast<const Tin*>(a.k) + unit * T * d;
    const Tin* v = reinterpret_cast<const Tin*>(a.v) + unit * T * d;
    const float* al = a.alpha + unit * T;
    const float* et = a.eta + unit * T;
    const float* be = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    const float* Gy_u = a.Gy + unit * T * d;

    float* p_ = a.ws + unit * a.ws_unit;
    auto take = [&](size_t n_) { float* r_ = p_; p_ += n_; return r_; };
    const size_t bd = (size_t)b * d, bb = (size_t)b * b;
    float* GM = take(P);   // [d][d] running adjoint of M (of the current chunk's end state)
    float* GS = take(P);   // [d][d] running adjoint of S
    float* TM = take(P);   // [d][d] the chunk's products for dMc, dSc
    float* TS = take(P);
    float *Kf = take(bd), *Qf = take(bd), *Vf = take(bd), *Gyf = take(bd);  // the chunk's k, q, v, Gy in fp32
    float* E = take(bd);     // e_i
    float* LR = take(bd);    // 2 (Mc k_i - v_i), then lambda_r_i
    float* Mq = take(bd);    // Mc q_t
    float* Sq = take(bd);    // Sc q_t
    float* GMk = take(bd);   // GM k_i
    float* GSk = take(bd);   // GS k_i
    float* GMtE = take(bd);  // GM^T e_i
    float* GStE = take(bd);  // GS^T e_i
    float* DK = take(bd);    // dk accumulator
    float* DQ1 = take(bd);   // Gy_t Mc (as rows: (Mc^T Gy_t)^T)
    float* DQ2 = take(bd);   // Gy_t Sc
    float* LE = take(bd);    // -(Gamma (.) QK)^T Gy, then (Gamma (.) Z) K
    float* SG = take(bd);    // A_t Gy_t, then sigma_t Gy_t
    float *Gam = take(bb), *U = take(bb), *QK = take(bb), *Z = take(bb), *PQ = take(bb), *PZ = take(bb);

    for (int i = tid; i < P; i += BW_THREADS) {
        GM[i] = a.GM[unit * P + i];
        GS[i] = a.GS[unit * P + i];
    }
    for (int c = nch - 1; c >= 0; --c) {
        const long long t0 = (long long)c * b;
        const int n = (int)min((long long)b, T - t0);
        const float* Mc = a.ckpt + (unit * nch + c) * 2 * (long long)P;
        const float* Sc = Mc + P;
        __syncthreads();
        // ---- the chunk's tokens and gates (four iterations' loads issued before their stores)
        for (int i0 = tid; i0 < n * d; i0 += 4 * BW_THREADS) {
            float kv[4], qv[4], vv[4], gv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * BW_THREADS;
                const bool in = i < n * d;
                kv[j] = in ? ld_f(k + t0 * d + i) : 0.f;
                qv[j] = in ? ld_f(q + t0 * d + i) : 0.f;
                vv[j] = in ? ld_f(v + t0 * d + i) : 0.f;
                gv[j] = in ? Gy_u[t0 * d + i] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * BW_THREADS;
                if (i < n * d) {
                    Kf[i] = kv[j];
                    Qf[i] = qv[j];
                    Vf[i] = vv[j];
                    Gyf[i] = gv[j];
                }
            }
        }
        for (int i = tid; i < n; i += BW_THREADS) {
            const float bt = be[t0 + i];
            s_a[i] = 1.0f - al[t0 + i];
            s_e[i] = et[t0 + i];
            s_b[i] = bt;
            s_c[i] = momentum_c(c_mode, bt, cc, t0 + i);
            s_da[i] = 0.f; s_de[i] = 0.f; s_db[i] = 0.f; s_dc[i] = 0.f;
        }
        __syncthreads();
        // ---- the scan: column i of Gamma and u from row 0, the start injected at row i
        for (int i = tid; i < n; i += BW_THREADS) {
            float u = 0.f, G = 0.f;
            for (int t = 0; t < n; ++t) {
                u = fmaf(s_b[t], u, t == i ? s_c[i] : 0.0f);
                G = fmaf(s_a[t], G, s_e[t] * u);
                Gam[t * b + i] = G;
                U[t * b + i] = u;
            }
            s_gam[i] = G;
            s_u[i] = u;
        }
        if (tid == 0) {
            float A = 1.f, Bc = 1.f, sg = 0.f;
            for (int t = 0; t < n; ++t) {
                A *= s_a[t];
                Bc *= s_b[t];
                sg = fmaf(s_a[t], sg, s_e[t] * Bc);
                sA[t] = A; sB[t] = Bc; sS[t] = sg;
            }
        }
        // ---- Mc k_i, Mc q_t, Sc q_t, q_t . k_i  (B(x, o) = Mc[o][x])
        gemm_(n, d, d, Kf, d, 1, Mc, 1, d, LR, d, 1.0f, false, gsh);
        gemm_(n, d, d, Qf, d, 1, Mc, 1, d, Mq, d, 1.0f, false, gsh);
        gemm_(n, d, d, Qf, d, 1, Sc, 1, d, Sq, d, 1.0f, false, gsh);
        gemm_(n, n, d, Qf, d, 1, Kf, 1, d, QK, b, 1.0f, false, gsh);
        // ---- e_i = clip(2 (Mc k_i - v_i)); P_Q = Gamma (.) QK (lower triangle)
        each<EU>(n * d, [&](int idx) { return make_float2(LR[idx], Vf[idx]); },
              [&](int idx, float2 x) {
                  const float r2 = 2.0f * (x.x - x.y);
                  LR[idx] = r2;
                  E[idx] = nm_clip_err(r2, a.e_clip);
              });
        each<EU>(n * n, [&](int idx) { const int t = idx / n, i = idx % n; return make_float2(Gam[t * b + i], QK[t * b + i]); },
              [&](int idx, float2 x) {
                  const int t = idx / n, i = idx % n;
                  PQ[t * b + i] = i <= t ? x.x * x.y : 0.0f;
              });
        __syncthreads();
        // ---- Z = Gy E^T; GM k_i, GS k_i (B(x, o) = G[o][x]); GM^T e_i, GS^T e_i (B(o, x) = G[o][x])
        gemm_(n, n, d, Gyf, d, 1, E, 1, d, Z, b, 1.0f, false, gsh);
        gemm_(n, d, d, Kf, d, 1, GM, 1, d, GMk, d, 1.0f, false, gsh);
        gemm_(n, d, d, Kf, d, 1, GS, 1, d, GSk, d, 1.0f, false, gsh);
        gemm_(n, d, d, E, d, 1, GM, d, 1, GMtE, d, 1.0f, false, gsh);
        gemm_(n, d, d, E, d, 1, GS, d, 1, GStE, d, 1.0f, false, gsh);
        // ---- lambda_e (first part): -(Gamma (.) QK)^T Gy   (A(i, t) = P_Q[t][i])
        gemm_(n, d, n, PQ, 1, b, Gyf, d, 1, LE, d, -1.0f, false, gsh);
        each<EU>(n * n, [&](int idx) { const int t = idx / n, i = idx % n; return make_float2(Z[t * b + i], Gam[t * b + i]); },
              [&](int idx, float2 x) {
                  const int t = idx / n, i = idx % n;
                  const float z = i <= t ? x.x : 0.0f;
                  Z[t * b + i] = z;
                  PZ[t * b + i] = x.y * z;
              });
        // ---- lambda_e = ... - gamma_i GM k_i + u_i GS k_i; lambda_r = 2 [inside the clip] lambda_e; dv = -lambda_r
        each<EU>(n * d, [&](int idx) { return make_float4(LE[idx], GMk[idx], GSk[idx], LR[idx]); },
              [&](int idx, float4 x) {
                  const int i = idx / d;
                  const float le = x.x - s_gam[i] * x.y + s_u[i] * x.z;
                  const float r2 = x.w;
                  const float lr = (r2 <= a.e_clip && r2 >= -a.e_clip) ? 2.0f * le : 0.0f;
                  LR[idx] = lr;
                  a.dv[(unit * T + t0) * d + idx] = -lr;
              });
        __syncthreads();
        // ---- dk = -(Gamma (.) Z)^T Q + lambda_r Mc (...) ; dq parts Gy Mc, Gy Sc, (Gamma (.) Z) K
        gemm_(n, d, n, PZ, 1, b, Qf, d, 1, DK, d, -1.0f, false, gsh);
        gemm_(n, d, d, LR, d, 1, Mc, d, 1, DK, d, 1.0f, true, gsh);
        gemm_(n, d, d, Gyf, d, 1, Mc, d, 1, DQ1, d, 1.0f, false, gsh);
        gemm_(n, d, d, Gyf, d, 1, Sc, d, 1, DQ2, d, 1.0f, false, gsh);
        gemm_(n, d, n, PZ, b, 1, Kf, d, 1, LE, d, 1.0f, false, gsh);
        each<EU>(n * d, [&](int idx) { return F6{DK[idx], GMtE[idx], GStE[idx], DQ1[idx], DQ2[idx], LE[idx]}; },
              [&](int idx, F6 x) {
                  const int i = idx / d;  // also the token t of dq
                  a.dk[(unit * T + t0) * d + idx] = x.a - s_gam[i] * x.b + s_u[i] * x.c;
                  a.dq[(unit * T + t0) * d + idx] = sA[i] * x.d - sS[i] * x.e - x.f;
              });
        // ---- scalar adjoints of A, sigma (per token) and of the chunk-end gamma, u (per column)
        // (four threads per token, each over every fourth feature, summed by shuffles)
        for (int base = 0; base < n; base += BW_THREADS / 4) {
            const int t = base + (tid >> 2), part = tid & 3;
            float ga = 0.f, gs = 0.f, hg = 0.f, hu = 0.f;
            if (t < n) {
                for (int o = part; o < d; o += 4) {
                    ga = fmaf(Gyf[t * d + o], Mq[t * d + o], ga);
                    gs = fmaf(Gyf[t * d + o], Sq[t * d + o], gs);
                    hg = fmaf(E[t * d + o], GMk[t * d + o], hg);
                    hu = fmaf(E[t * d + o], GSk[t * d + o], hu);
                }
            }
#pragma unroll
            for (int sh = 1; sh < 4; sh <<= 1) {
                ga += __shfl_xor_sync(0xffffffffu, ga, sh);
                gs += __shfl_xor_sync(0xffffffffu, gs, sh);
                hg += __shfl_xor_sync(0xffffffffu, hg, sh);
                hu += __shfl_xor_sync(0xffffffffu, hu, sh);
            }
            if (t < n && part == 0) {
                s_gA[t] = ga;
                s_gS[t] = -gs;
                s_hg[t] = -hg;  // dL/dgamma_t (token t as a column i)
                s_hu[t] = hu;   // dL/du_t
            }
        }
        float pmm = 0.f, pms = 0.f, pss = 0.f;
        for (int i = tid; i < P; i += BW_THREADS) {
            pmm = fmaf(GM[i], Mc[i], pmm);
            pms = fmaf(GM[i], Sc[i], pms);
            pss = fmaf(GS[i], Sc[i], pss);
        }
        const float gmm = block_sum(pmm, red);
        const float gms = block_sum(pms, red);
        const float gss = block_sum(pss, red);
        __syncthreads();
        // ---- reverse of the column recursions Gamma_{t,i} = a_t Gamma_{t-1,i} + eta_t u_{t,i},
        //      u_{t,i} = beta_t u_{t-1,i} (+ c_i at t = i)
        // One column i per thread (chunks of at most BW_THREADS tokens).  The adjoints of a_t, eta_t, beta_t
        // gather every column's step-t term: each warp sums its lanes' terms by shuffles and one lane adds them
        // (steps run from the last token down to the warp's first column, the same for all its lanes); the
        // column's values for 8 steps are loaded before those steps are computed.
        {
            const int i = tid, lane = tid & 31, wmin = tid & ~31;
            const bool col = i < n;
            float cG = 0.f, cU = 0.f;  // a_{t+1} gGamma_{t+1}, beta_{t+1} gu_{t+1}
            for (int th = n - 1; th >= wmin; th -= 8) {
                float qk[8], zz[8], gp[8], u0[8], u1[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = th - j;
                    const bool in = col && t >= i;
                    qk[j] = in ? QK[t * b + i] : 0.0f;
                    zz[j] = in ? Z[t * b + i] : 0.0f;
                    gp[j] = in && t > i ? Gam[(t - 1) * b + i] : 0.0f;
                    u0[j] = in ? U[t * b + i] : 0.0f;
                    u1[j] = in && t > i ? U[(t - 1) * b + i] : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = th - j;
                    if (t < wmin) break;  // the same for the whole warp
                    float ta = 0.f, te = 0.f, tb = 0.f;
                    if (col && t >= i) {
                        const float gG = -qk[j] * zz[j] + (t == n - 1 ? s_hg[i] : 0.0f) + cG;
                        const float gu = (t == n - 1 ? s_hu[i] : 0.0f) + s_e[t] * gG + cU;
                        ta = gG * gp[j];
                        te = gG * u0[j];
                        if (t > i) tb = gu * u1[j];
                        else s_dc[i] += gu;
                        cG = s_a[t] * gG;
                        cU = s_b[t] * gu;
                    }
                    ta = warp_sum(ta);
                    te = warp_sum(te);
                    tb = warp_sum(tb);
                    if (lane == 0) {
                        atomicAdd(&s_da[t], ta);
                        atomicAdd(&s_de[t], te);
                        atomicAdd(&s_db[t], tb);
                    }
                }
            }
        }
        // ---- A_t Gy_t as rows, for dMc
        each<EU>(n * d, [&](int idx) { return Gyf[idx]; }, [&](int idx, float g) { SG[idx] = sA[idx / d] * g; });
        __syncthreads();
        // ---- reverse of A_t = a_t A_{t-1}, B_t = beta_t B_{t-1}, sigma_t = a_t sigma_{t-1} + eta_t B_t
        if (tid == 0) {
            float cA = 0.f, cS = 0.f, cB = 0.f;
            for (int t = n - 1; t >= 0; --t) {
                const bool last = t == n - 1;
                const float gA = s_gA[t] + (last ? gmm : 0.0f) + cA;
                const float gS = s_gS[t] + (last ? -gms : 0.0f) + cS;
                const float gB = (last ? gss : 0.0f) + s_e[t] * gS + cB;
                const float Ap = t ? sA[t - 1] : 1.0f, Sp = t ? sS[t - 1] : 0.0f, Bp = t ? sB[t - 1] : 1.0f;
                s_da[t] += gA * Ap + gS * Sp;
                s_de[t] += gS * sB[t];
                s_db[t] += gB * Bp;
                cA = s_a[t] * gA;
                cS = s_a[t] * gS;
                cB = s_b[t] * gB;
            }
        }
        // ---- dMc = sum_t A_t Gy_t q_t^T + sum_i lambda_r_i k_i^T (+ A GM below)   (A(o, t) = SG[t][o])
        gemm_(d, d, n, SG, 1, d, Qf, d, 1, TM, d, 1.0f, false, gsh);
        gemm_(d, d, n, LR, 1, d, Kf, d, 1, TM, d, 1.0f, true, gsh);
        for (int t = tid; t < n; t += BW_THREADS) {
            const long long g = unit * T + t0 + t;
            a.dalpha[g] = -s_da[t];  // a_t = 1 - alpha_t
            a.deta[g] = s_de[t];
            a.dbeta[g] = s_db[t] + (c_mode == NM_C_ONE_MINUS_BETA ? -s_dc[t] : 0.0f);
            if (a.dc) a.dc[g] = s_dc[t];
        }
        each<EU>(n * d, [&](int idx) { return Gyf[idx]; }, [&](int idx, float g) { SG[idx] = sS[idx / d] * g; });
        __syncthreads();
        // ---- dSc = - sum_t sigma_t Gy_t q_t^T (- sigma GM + B GS below)
        gemm_(d, d, n, SG, 1, d, Qf, d, 1, TS, d, -1.0f, false, gsh);
        // ---- the chunk-start state's adjoint becomes the previous chunk's (GM, GS), in place
        const float An = sA[n - 1], Bn = sB[n - 1], Sn = sS[n - 1];
        each<EU>(P, [&](int idx) { return make_float4(GM[idx], GS[idx], TS[idx], TM[idx]); },
              [&](int idx, float4 x) {
                  GS[idx] = x.z - Sn * x.x + Bn * x.y;
                  GM[idx] = x.w + An * x.x;
              });
    }
    __syncthreads();
    for (int i = tid; i < P; i += BW_THREADS) {
        a.dM0[unit * P + i] = GM[i];
        a.dS0[unit * P + i] = GS[i];
    }
    if constexpr (TC) tg_teardown(tcx, a.status);
}

}  // namespace

size_t nm_bwd_linear_ws_floats(int d, int b) {
    return 4 * (size_t)d * d + 17 * (size_t)b * d + 6 * (size_t)b * b;
}

namespace {

// ---------------------------------------------------------------- 2-layer MLP memory
// M(x) = W2 silu(W1 x).  Per chunk, with the chunk-start (W1, S1, W2, S2):
//   z_i = W1 k_i, a_i = silu(z_i), phi_i = silu'(z_i), e_i = clip(2 (W2 a_i - v_i)),
//   p_i = W2^T e_i, delta_i = p_i (.) phi_i,
//   h_t = A_t W1 q_t - sigma_t S1 q_t - sum_{i<=t} Gamma_{t,i} (k_i . q_t) delta_i,  b_t = silu(h_t),
//   y_t = A_t W2 b_t - sigma_t S2 b_t - sum_{i<=t} Gamma_{t,i} (a_i . b_t) e_i,
//   W1_end = A W1 - sigma S1 - sum_i gamma_i delta_i k_i^T,  S1_end = B S1 + sum_i u_i delta_i k_i^T,
//   W2_end = A W2 - sigma S2 - sum_i gamma_i e_i a_i^T,      S2_end = B S2 + sum_i u_i e_i a_i^T.
// Reverse mode, given Gy_t and the end state's adjoints (G1, H1, G2, H2 for W1, S1, W2, S2), with
// Zy_{t,i} = Gy_t . e_i, AA_{t,i} = b_t . a_i, QK_{t,i} = q_t . k_i:
//   db_t = A_t W2^T Gy_t - sigma_t S2^T Gy_t - sum_{i<=t} Gamma Zy a_i;   dh_t = db_t (.) silu'(h_t)
//   Zh_{t,i} = dh_t . delta_i;  dq_t = A_t W1^T dh_t - sigma_t S1^T dh_t - sum_{i<=t} Gamma Zh k_i
//   ddelta_i = - sum_{t>=i} Gamma QK dh_t - gamma_i G1 k_i + u_i H1 k_i
//   dp_i = ddelta_i (.) phi_i;  dz_i = ddelta_i (.) p_i (.) silu''(z_i) + da_i (.) phi_i
//   de_i = - sum_{t>=i} Gamma AA Gy_t - gamma_i G2 a_i + u_i H2 a_i + W2 dp_i
//   dr_i = 2 [inside the clip] de_i,  dv_i = -dr_i
//   da_i = - sum_{t>=i} Gamma Zy b_t - gamma_i G2^T e_i + u_i H2^T e_i + W2^T dr_i
//   dk_i = - sum_{t>=i} Gamma Zh q_t - gamma_i G1^T delta_i + u_i H1^T delta_i + W1^T dz_i
//   dW1 = sum_t A_t dh_t q_t^T + A G1 + sum_i dz_i k_i^T,   dS1 = - sum_t sigma_t dh_t q_t^T - sigma G1 + B H1
//   dW2 = sum_t A_t Gy_t b_t^T + A G2 + sum_i (e_i dp_i^T + dr_i a_i^T),  dS2 = - sum_t sigma_t Gy_t b_t^T - sigma G2 + B H2
// and the scalar adjoints dL/dA_t = Gy_t . W2 b_t + dh_t . W1 q_t, dL/dsigma_t = -(Gy_t . S2 b_t + dh_t . S1 q_t),
// dL/dGamma_{t,i} = -(AA Zy + QK Zh), plus the chunk-end terms, reversed through the scan as for the
// linear memory.  silu''(z) = s (1 - s) (2 + z (1 - 2 s)) with s = sigmoid(z).
__device__ __forceinline__ float sig_f(float z) { return 1.0f / (1.0f + expf(-z)); }

__host__ __device__ inline size_t bwd_mlp_ws_floats(int d, int h, int b) {
    return 8 * (size_t)h * d + 18 * (size_t)b * d + 21 * (size_t)b * h + 10 * (size_t)b * b;
}

template <typename Tin, bool TC>
__global__ void __launch_bounds__(BW_THREADS) bwd_mlp_kernel(bwd_args a, int d, int hd, int b, int c_mode) {
    __shared__ float s_a[BW_MAX_CHUNK], s_e[BW_MAX_CHUNK], s_b[BW_MAX_CHUNK], s_c[BW_MAX_CHUNK];
    __shared__ float sA[BW_MAX_CHUNK], sB[BW_MAX_CHUNK], sS[BW_MAX_CHUNK];
    __shared__ float s_gam[BW_MAX_CHUNK], s_u[BW_MAX_CHUNK];
    __shared__ float s_gA[BW_MAX_CHUNK], s_gS[BW_MAX_CHUNK], s_hg[BW_MAX_CHUNK], s_hu[BW_MAX_CHUNK];
    __shared__ float s_da[BW_MAX_CHUNK], s_de[BW_MAX_CHUNK], s_db[BW_MAX_CHUNK], s_dc[BW_MAX_CHUNK];
    __shared__ float red[BW_THREADS / 32];
    __shared__ __align__(16) float gsh[GEMM_SMEM_FLOATS];
    TcCtx tcx;
    if constexpr (TC) tg_setup(tcx);
    constexpr int EU = TC ? 4 : 1;  // elementwise passes: indices batched per thread
    // every chunk-sized contraction: tcgen05 tf32 products or fp32 FFMA block GEMMs
    auto gemm_ = [&](int M_, int N_, int K_, const float* A_, long long am_, long long ak_, const float* B_, long long bk_,
                     long long bn_, float* C_, long long cm_, float alpha_, bool acc_, float* sh_) {
        if constexpr (TC) tc_gemm(tcx, M_, N_, K_, A_, am_, ak_, B_, bk_, bn_, C_, cm_, alpha_, acc_);
        else block_gemm(M_, N_, K_, A_, am_, ak_, B_, bk_, bn_, C_, cm_, alpha_, acc_, sh_);
    };

    const long long unit = blockIdx.x;
    const int tid = threadIdx.x;
    const long long T = a.T;
    const long long HD = (long long)hd * d;  // size of one weight matrix
    const long long P = 2 * HD;
    const int nch = (int)((T + b - 1) / b);
    const Tin* q = reinterpret_cast<const Tin*>(a.q) + unit * T * d;
    const Tin* k = reinterpret_cast<const Tin*>(a.k) + unit * T * d;
    const Tin* v = reinterpret_cast<const Tin*>(a.v) + unit * T * d;
    const float* al = a.alpha + unit * T;
    const float* et = a.eta + unit * T;
    const float* be = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    const float* Gy_u = a.Gy + unit * T * d;

    float* p_ = a.ws + unit * a.ws_unit;
    auto take = [&](size_t n_) { float* r_ = p_; p_ += n_; return r_; };
    // running adjoints of the end state, in the packed order: [dL/dW1 | dL/dW2] then [dL/dS1 | dL/dS2]
    float* GW1 = take(HD);  // [h][d]
    float* GW2 = take(HD);  // [d][h]
    float* GS1 = take(HD);  // [h][d]
    float* GS2 = take(HD);  // [d][h]
    float *TW1 = take(HD), *TW2 = take(HD), *TS1 = take(HD), *TS2 = take(HD);  // the chunk's products for them
    const size_t bd = (size_t)b * d, bh = (size_t)b * hd, bb = (size_t)b * b;
    float *Kf = take(bd), *Qf = take(bd), *Vf = take(bd), *Gyf = take(bd), *E = take(bd), *R2 = take(bd);
    float *W2b = take(bd), *S2b = take(bd), *G2a = take(bd), *H2a = take(bd), *G1td = take(bd), *H1td = take(bd);
    float *DE = take(bd), *DK = take(bd), *SGy = take(bd), *DHW1 = take(bd), *DHS1 = take(bd), *PZhK = take(bd);
    float *Zs = take(bh), *Ak = take(bh), *PH = take(bh), *PP = take(bh), *DL = take(bh), *PSI = take(bh);
    float *Bt = take(bh), *W1q = take(bh), *S1q = take(bh), *DH = take(bh), *DP = take(bh), *DAk = take(bh);
    float *G1k = take(bh), *H1k = take(bh), *G2te = take(bh), *H2te = take(bh), *DZ = take(bh), *C1 = take(bh);
    float *GyW2 = take(bh), *GyS2 = take(bh), *SGh = take(bh);
    float *Gam = take(bb), *U = take(bb), *QK = take(bb), *AA = take(bb), *Zy = take(bb), *Zh = take(bb);
    float *PQ = take(bb), *PZy = take(bb), *PA = take(bb), *PZh = take(bb);

    for (long long i = tid; i < P; i += BW_THREADS) {
        GW1[i] = a.GM[unit * P + i];
        GS1[i] = a.GS[unit * P + i];
    }

    for (int c = nch - 1; c >= 0; --c) {
        const long long t0 = (long long)c * b;
        const int n = (int)min((long long)b, T - t0);
        const float* W1c = a.ckpt + (unit * nch + c) * 2 * P;  // chunk-start W1 [h][d], W2 [d][h]
        const float* W2c = W1c + HD;
        const float* S1c = W1c + P;
        const float* S2c = S1c + HD;
        __syncthreads();
        for (int i0 = tid; i0 < n * d; i0 += 4 * BW_THREADS) {  // four iterations' loads before their stores
            float kv[4], qv[4], vv[4], gv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * BW_THREADS;
                const bool in = i < n * d;
                kv[j] = in ? ld_f(k + t0 * d + i) : 0.f;
                qv[j] = in ? ld_f(q + t0 * d + i) : 0.f;
                vv[j] = in ? ld_f(v + t0 * d + i) : 0.f;
                gv[j] = in ? Gy_u[t0 * d + i] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * BW_THREADS;
                if (i < n * d) {
                    Kf[i] = kv[j];
                    Qf[i] = qv[j];
                    Vf[i] = vv[j];
                    Gyf[i] = gv[j];
                }
            }
        }
        for (int i = tid; i < n; i += BW_THREADS) {
            const float bt = be[t0 + i];
            s_a[i] = 1.0f - al[t0 + i];
            s_e[i] = et[t0 + i];
            s_b[i] = bt;
            s_c[i] = momentum_c(c_mode, bt, cc, t0 + i);
            s_da[i] = 0.f; s_de[i] = 0.f; s_db[i] = 0.f; s_dc[i] = 0.f;
        }
        __syncthreads();
        for (int i = tid; i < n; i += BW_THREADS) {  // the scan, column by column
            float u = 0.f, G = 0.f;
            for (int t = 0; t < n; ++t) {
                u = fmaf(s_b[t], u, t == i ? s_c[i] : 0.0f);
                G = fmaf(s_a[t], G, s_e[t] * u);
                Gam[t * b + i] = G;
                U[t * b + i] = u;
            }
            s_gam[i] = G;
            s_u[i] = u;
        }
        if (tid == 0) {
            float A = 1.f, Bc = 1.f, sg = 0.f;
            for (int t = 0; t < n; ++t) {
                A *= s_a[t];
                Bc *= s_b[t];
                sg = fmaf(s_a[t], sg, s_e[t] * Bc);
                sA[t] = A; sB[t] = Bc; sS[t] = sg;
            }
        }
        // ---- F1: z = W1 k_i, W1 q_t, S1 q_t (B(x, j) = W1[j][x]); QK
        gemm_(n, hd, d, Kf, d, 1, W1c, 1, d, Zs, hd, 1.0f, false, gsh);
        gemm_(n, hd, d, Qf, d, 1, W1c, 1, d, W1q, hd, 1.0f, false, gsh);
        gemm_(n, hd, d, Qf, d, 1, S1c, 1, d, S1q, hd, 1.0f, false, gsh);
        gemm_(n, n, d, Qf, d, 1, Kf, 1, d, QK, b, 1.0f, false, gsh);
        each<EU>(n * hd, [&](int idx) { return Zs[idx]; },
              [&](int idx, float z) {
                  const float s = sig_f(z);
                  Ak[idx] = z * s;
                  PH[idx] = s * (1.0f + z * (1.0f - s));
              });
        each<EU>(n * n, [&](int idx) { const int t = idx / n, i = idx % n; return make_float2(Gam[t * b + i], QK[t * b + i]); },
              [&](int idx, float2 x) {
                  const int t = idx / n, i = idx % n;
                  PQ[t * b + i] = i <= t ? x.x * x.y : 0.0f;
              });
        __syncthreads();
        // ---- F2: e = clip(2 (W2 a - v))   (B(j, o) = W2[o][j])
        gemm_(n, d, hd, Ak, hd, 1, W2c, 1, hd, R2, d, 1.0f, false, gsh);
        each<EU>(n * d, [&](int idx) { return make_float2(R2[idx], Vf[idx]); },
              [&](int idx, float2 x) {
                  const float r2 = 2.0f * (x.x - x.y);
                  R2[idx] = r2;
                  E[idx] = nm_clip_err(r2, a.e_clip);
              });
        __syncthreads();
        // ---- F3: p = W2^T e (B(o, j) = W2[o][j]), delta = p (.) silu'(z)
        gemm_(n, hd, d, E, d, 1, W2c, hd, 1, PP, hd, 1.0f, false, gsh);
        each<EU>(n * hd, [&](int idx) { return make_float2(PP[idx], PH[idx]); },
              [&](int idx, float2 x) { DL[idx] = x.x * x.y; });
        __syncthreads();
        // ---- F4: h_t = A_t W1 q_t - sigma_t S1 q_t - sum_{i<=t} Gamma QK delta_i; b_t = silu(h_t)
        gemm_(n, hd, n, PQ, b, 1, DL, hd, 1, C1, hd, 1.0f, false, gsh);
        each<EU>(n * hd, [&](int idx) { return make_float3(W1q[idx], S1q[idx], C1[idx]); },
              [&](int idx, float3 x) {
                  const int t = idx / hd;
                  const float hh = sA[t] * x.x - sS[t] * x.y - x.z;
                  const float s = sig_f(hh);
                  Bt[idx] = hh * s;
                  PSI[idx] = s * (1.0f + hh * (1.0f - s));
              });
        __syncthreads();
        // ---- F5: AA = b a^T, Zy = Gy e^T; W2 b_t, S2 b_t
        gemm_(n, n, hd, Bt, hd, 1, Ak, 1, hd, AA, b, 1.0f, false, gsh);
        gemm_(n, n, d, Gyf, d, 1, E, 1, d, Zy, b, 1.0f, false, gsh);
        gemm_(n, d, hd, Bt, hd, 1, W2c, 1, hd, W2b, d, 1.0f, false, gsh);
        gemm_(n, d, hd, Bt, hd, 1, S2c, 1, hd, S2b, d, 1.0f, false, gsh);
        each<EU>(n * n,
              [&](int idx) { const int t = idx / n, i = idx % n; return make_float3(Zy[t * b + i], Gam[t * b + i], AA[t * b + i]); },
              [&](int idx, float3 x) {
                  const int t = idx / n, i = idx % n;
                  const float zy = i <= t ? x.x : 0.0f;
                  Zy[t * b + i] = zy;
                  PZy[t * b + i] = x.y * zy;
                  PA[t * b + i] = i <= t ? x.y * x.z : 0.0f;
              });
        __syncthreads();
        // ---- B2: db_t = A_t W2^T Gy_t - sigma_t S2^T Gy_t - sum_i Gamma Zy a_i;  dh_t = db_t (.) silu'(h_t)
        gemm_(n, hd, d, Gyf, d, 1, W2c, hd, 1, GyW2, hd, 1.0f, false, gsh);
        gemm_(n, hd, d, Gyf, d, 1, S2c, hd, 1, GyS2, hd, 1.0f, false, gsh);
        gemm_(n, hd, n, PZy, b, 1, Ak, hd, 1, C1, hd, 1.0f, false, gsh);
        each<EU>(n * hd, [&](int idx) { return make_float4(GyW2[idx], GyS2[idx], C1[idx], PSI[idx]); },
              [&](int idx, float4 x) {
                  const int t = idx / hd;
                  DH[idx] = (sA[t] * x.x - sS[t] * x.y - x.z) * x.w;
              });
        // ---- B5: the end state's adjoints against the chunk's vectors
        gemm_(n, hd, d, Kf, d, 1, GW1, 1, d, G1k, hd, 1.0f, false, gsh);   // G1 k_i
        gemm_(n, hd, d, Kf, d, 1, GS1, 1, d, H1k, hd, 1.0f, false, gsh);   // H1 k_i
        gemm_(n, hd, d, E, d, 1, GW2, hd, 1, G2te, hd, 1.0f, false, gsh);  // G2^T e_i
        gemm_(n, hd, d, E, d, 1, GS2, hd, 1, H2te, hd, 1.0f, false, gsh);  // H2^T e_i
        gemm_(n, d, hd, Ak, hd, 1, GW2, 1, hd, G2a, d, 1.0f, false, gsh);  // G2 a_i
        gemm_(n, d, hd, Ak, hd, 1, GS2, 1, hd, H2a, d, 1.0f, false, gsh);  // H2 a_i
        gemm_(n, d, hd, DL, hd, 1, GW1, d, 1, G1td, d, 1.0f, false, gsh); // G1^T delta_i
        gemm_(n, d, hd, DL, hd, 1, GS1, d, 1, H1td, d, 1.0f, false, gsh); // H1^T delta_i
        // ---- B3: Zh = dh delta^T; B4: dq
        gemm_(n, n, hd, DH, hd, 1, DL, 1, hd, Zh, b, 1.0f, false, gsh);
        each<EU>(n * n, [&](int idx) { const int t = idx / n, i = idx % n; return make_float2(Zh[t * b + i], Gam[t * b + i]); },
              [&](int idx, float2 x) {
                  const int t = idx / n, i = idx % n;
                  const float zh = i <= t ? x.x : 0.0f;
                  Zh[t * b + i] = zh;
                  PZh[t * b + i] = x.y * zh;
              });
        __syncthreads();
        gemm_(n, d, hd, DH, hd, 1, W1c, d, 1, DHW1, d, 1.0f, false, gsh);
        gemm_(n, d, hd, DH, hd, 1, S1c, d, 1, DHS1, d, 1.0f, false, gsh);
        gemm_(n, d, n, PZh, b, 1, Kf, d, 1, PZhK, d, 1.0f, false, gsh);
        each<EU>(n * d, [&](int idx) { return make_float3(DHW1[idx], DHS1[idx], PZhK[idx]); },
              [&](int idx, float3 x) {
                  const int t = idx / d;
                  a.dq[(unit * T + t0) * d + idx] = sA[t] * x.x - sS[t] * x.y - x.z;
              });
        // ---- B6: ddelta -> dp and the silu'' part of dz; the direct parts of da, de, dk
        gemm_(n, hd, n, PQ, 1, b, DH, hd, 1, C1, hd, -1.0f, false, gsh);    // -sum_t Gamma QK dh_t
        gemm_(n, hd, n, PZy, 1, b, Bt, hd, 1, DAk, hd, -1.0f, false, gsh);  // -sum_t Gamma Zy b_t
        gemm_(n, d, n, PA, 1, b, Gyf, d, 1, DE, d, -1.0f, false, gsh);      // -sum_t Gamma AA Gy_t
        gemm_(n, d, n, PZh, 1, b, Qf, d, 1, DK, d, -1.0f, false, gsh);     // -sum_t Gamma Zh q_t
        each<EU>(n * hd, [&](int idx) { return F9{C1[idx], G1k[idx], H1k[idx], Zs[idx], PH[idx], PP[idx], DAk[idx], G2te[idx], H2te[idx]}; },
              [&](int idx, F9 x) {
                  const int i = idx / hd;
                  const float dd = x.a - s_gam[i] * x.b + s_u[i] * x.c;
                  const float z = x.d, s = sig_f(z);
                  DP[idx] = dd * x.e;
                  DZ[idx] = dd * x.f * (s * (1.0f - s) * (2.0f + z * (1.0f - 2.0f * s)));
                  DAk[idx] = x.g + (-s_gam[i] * x.h + s_u[i] * x.k);
              });
        each<EU>(n * d, [&](int idx) { return F6{DE[idx], G2a[idx], H2a[idx], DK[idx], G1td[idx], H1td[idx]}; },
              [&](int idx, F6 x) {
                  const int i = idx / d;
                  DE[idx] = x.a + (-s_gam[i] * x.b + s_u[i] * x.c);
                  DK[idx] = x.d + (-s_gam[i] * x.e + s_u[i] * x.f);
              });
        __syncthreads();
        // ---- B7: de += W2 dp (B(j, o) = W2[o][j]); dr = 2 [inside the clip] de; dv = -dr
        gemm_(n, d, hd, DP, hd, 1, W2c, 1, hd, DE, d, 1.0f, true, gsh);
        each<EU>(n * d, [&](int idx) { return make_float2(R2[idx], DE[idx]); },
              [&](int idx, float2 x) {
                  const float r2 = x.x;
                  const float dr = (r2 <= a.e_clip && r2 >= -a.e_clip) ? 2.0f * x.y : 0.0f;
                  R2[idx] = dr;
                  a.dv[(unit * T + t0) * d + idx] = -dr;
              });
        __syncthreads();
        // ---- B8: da += W2^T dr (B(o, j) = W2[o][j]); dz += da (.) silu'(z)
        gemm_(n, hd, d, R2, d, 1, W2c, hd, 1, DAk, hd, 1.0f, true, gsh);
        each<EU>(n * hd, [&](int idx) { return make_float3(DAk[idx], PH[idx], DZ[idx]); },
              [&](int idx, float3 x) { DZ[idx] = fmaf(x.x, x.y, x.z); });
        __syncthreads();
        // ---- B9: dk += W1^T dz (B(j, x) = W1[j][x])
        gemm_(n, d, hd, DZ, hd, 1, W1c, d, 1, DK, d, 1.0f, true, gsh);
        each<EU>(n * d, [&](int idx) { return DK[idx]; }, [&](int idx, float x) { a.dk[(unit * T + t0) * d + idx] = x; });
        // ---- B10: scalar adjoints of A, sigma and of the chunk-end gamma, u
        // (four threads per token, each over every fourth feature, summed by shuffles)
        for (int base = 0; base < n; base += BW_THREADS / 4) {
            const int t = base + (tid >> 2), part = tid & 3;
            float ga = 0.f, gs = 0.f, hg = 0.f, hu = 0.f;
            if (t < n) {
                for (int o = part; o < d; o += 4) {
                    ga = fmaf(Gyf[t * d + o], W2b[t * d + o], ga);
                    gs = fmaf(Gyf[t * d + o], S2b[t * d + o], gs);
                    hg = fmaf(E[t * d + o], G2a[t * d + o], hg);
                    hu = fmaf(E[t * d + o], H2a[t * d + o], hu);
                }
                for (int j = part; j < hd; j += 4) {
                    ga = fmaf(DH[t * hd + j], W1q[t * hd + j], ga);
                    gs = fmaf(DH[t * hd + j], S1q[t * hd + j], gs);
                    hg = fmaf(DL[t * hd + j], G1k[t * hd + j], hg);
                    hu = fmaf(DL[t * hd + j], H1k[t * hd + j], hu);
                }
            }
#pragma unroll
            for (int sh = 1; sh < 4; sh <<= 1) {
                ga += __shfl_xor_sync(0xffffffffu, ga, sh);
                gs += __shfl_xor_sync(0xffffffffu, gs, sh);
                hg += __shfl_xor_sync(0xffffffffu, hg, sh);
                hu += __shfl_xor_sync(0xffffffffu, hu, sh);
            }
            if (t < n && part == 0) {
                s_gA[t] = ga;
                s_gS[t] = -gs;
                s_hg[t] = -hg;
                s_hu[t] = hu;
            }
        }
        float pmm = 0.f, pms = 0.f, pss = 0.f;
        for (long long i = tid; i < P; i += BW_THREADS) {
            pmm = fmaf(GW1[i], W1c[i], pmm);   // <G1, W1> + <G2, W2> (W1 | W2 packed)
            pms = fmaf(GW1[i], S1c[i], pms);   // <G1, S1> + <G2, S2>
            pss = fmaf(GS1[i], S1c[i], pss);   // <H1, S1> + <H2, S2>
        }
        const float gmm = block_sum(pmm, red);
        const float gms = block_sum(pms, red);
        const float gss = block_sum(pss, red);
        __syncthreads();
        // One column i per thread; each warp sums its lanes' step-t terms by shuffles and one lane adds them
        // (see the linear memory); the column's values for 8 steps are loaded before those steps are computed.
        {
            const int i = tid, lane = tid & 31, wmin = tid & ~31;
            const bool col = i < n;
            float cG = 0.f, cU = 0.f;
            for (int th = n - 1; th >= wmin; th -= 8) {
                float aa[8], zy[8], qk[8], zh[8], gp[8], u0[8], u1[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = th - j;
                    const bool in = col && t >= i;
                    aa[j] = in ? AA[t * b + i] : 0.0f;
                    zy[j] = in ? Zy[t * b + i] : 0.0f;
                    qk[j] = in ? QK[t * b + i] : 0.0f;
                    zh[j] = in ? Zh[t * b + i] : 0.0f;
                    gp[j] = in && t > i ? Gam[(t - 1) * b + i] : 0.0f;
                    u0[j] = in ? U[t * b + i] : 0.0f;
                    u1[j] = in && t > i ? U[(t - 1) * b + i] : 0.0f;
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int t = th - j;
                    if (t < wmin) break;  // the same for the whole warp
                    float ta = 0.f, te = 0.f, tb = 0.f;
                    if (col && t >= i) {
                        const float gG = -(aa[j] * zy[j] + qk[j] * zh[j]) + (t == n - 1 ? s_hg[i] : 0.0f) + cG;
                        const float gu = (t == n - 1 ? s_hu[i] : 0.0f) + s_e[t] * gG + cU;
                        ta = gG * gp[j];
                        te = gG * u0[j];
                        if (t > i) tb = gu * u1[j];
                        else s_dc[i] += gu;
                        cG = s_a[t] * gG;
                        cU = s_b[t] * gu;
                    }
                    ta = warp_sum(ta);
                    te = warp_sum(te);
                    tb = warp_sum(tb);
                    if (lane == 0) {
                        atomicAdd(&s_da[t], ta);
                        atomicAdd(&s_de[t], te);
                        atomicAdd(&s_db[t], tb);
                    }
                }
            }
        }
        each<EU>(n * hd, [&](int idx) { return DH[idx]; }, [&](int idx, float g) { SGh[idx] = sA[idx / hd] * g; });
        each<EU>(n * d, [&](int idx) { return Gyf[idx]; }, [&](int idx, float g) { SGy[idx] = sA[idx / d] * g; });
        __syncthreads();
        if (tid == 0) {
            float cA = 0.f, cS = 0.f, cB = 0.f;
            for (int t = n - 1; t >= 0; --t) {
                const bool last = t == n - 1;
                const float gA = s_gA[t] + (last ? gmm : 0.0f) + cA;
                const float gS = s_gS[t] + (last ? -gms : 0.0f) + cS;
                const float gB = (last ? gss : 0.0f) + s_e[t] * gS + cB;
                const float Ap = t ? sA[t - 1] : 1.0f, Sp = t ? sS[t - 1] : 0.0f, Bp = t ? sB[t - 1] : 1.0f;
                s_da[t] += gA * Ap + gS * Sp;
                s_de[t] += gS * sB[t];
                s_db[t] += gB * Bp;
                cA = s_a[t] * gA;
                cS = s_a[t] * gS;
                cB = s_b[t] * gB;
            }
        }
        // ---- B11: the chunk's products for the chunk-start state's adjoints
        //      dW1 = sum_t A_t dh_t q_t^T + sum_i dz_i k_i^T; dW2 = sum_t A_t Gy_t b_t^T + sum_i (e_i dp_i^T + dr_i a_i^T)
        gemm_(hd, d, n, SGh, 1, hd, Qf, d, 1, TW1, d, 1.0f, false, gsh);
        gemm_(hd, d, n, DZ, 1, hd, Kf, d, 1, TW1, d, 1.0f, true, gsh);
        gemm_(d, hd, n, SGy, 1, d, Bt, hd, 1, TW2, hd, 1.0f, false, gsh);
        gemm_(d, hd, n, E, 1, d, DP, hd, 1, TW2, hd, 1.0f, true, gsh);
        gemm_(d, hd, n, R2, 1, d, Ak, hd, 1, TW2, hd, 1.0f, true, gsh);
        for (int t = tid; t < n; t += BW_THREADS) {
            const long long g = unit * T + t0 + t;
            a.dalpha[g] = -s_da[t];
            a.deta[g] = s_de[t];
            a.dbeta[g] = s_db[t] + (c_mode == NM_C_ONE_MINUS_BETA ? -s_dc[t] : 0.0f);
            if (a.dc) a.dc[g] = s_dc[t];
        }
        each<EU>(n * hd, [&](int idx) { return DH[idx]; }, [&](int idx, float g) { SGh[idx] = sS[idx / hd] * g; });
        each<EU>(n * d, [&](int idx) { return Gyf[idx]; }, [&](int idx, float g) { SGy[idx] = sS[idx / d] * g; });
        __syncthreads();
        //      dS1 = - sum_t sigma_t dh_t q_t^T, dS2 = - sum_t sigma_t Gy_t b_t^T  (the state terms below)
        gemm_(hd, d, n, SGh, 1, hd, Qf, d, 1, TS1, d, -1.0f, false, gsh);
        gemm_(d, hd, n, SGy, 1, d, Bt, hd, 1, TS2, hd, -1.0f, false, gsh);
        const float An = sA[n - 1], Bn = sB[n - 1], Sn = sS[n - 1];
        for (long long idx = tid; idx < HD; idx += BW_THREADS) {
            const float g1 = GW1[idx], h1 = GS1[idx], g2 = GW2[idx], h2 = GS2[idx];
            GS1[idx] = TS1[idx] - Sn * g1 + Bn * h1;
            GW1[idx] = TW1[idx] + An * g1;
            GS2[idx] = TS2[idx] - Sn * g2 + Bn * h2;
            GW2[idx] = TW2[idx] + An * g2;
        }
    }
    __syncthreads();
    for (long long i = tid; i < P; i += BW_THREADS) {
        a.dM0[unit * P + i] = GW1[i];
        a.dS0[unit * P + i] = GS1[i];
    }
    if constexpr (TC) tg_teardown(tcx, a.status);
}

}  // namespace

size_t nm_bwd_ws_floats(const nm_config& c) {
    return c.kind == NM_LINEAR ? nm_bwd_linear_ws_floats(c.d, c.chunk) : bwd_mlp_ws_floats(c.d, c.hidden, c.chunk);
}

bool nm_bwd_supports(const nm_config& c) {
    const bool common = (c.d == 16 || c.d == 32 || c.d == 64 || c.d == 128) && c.chunk >= 1 &&
                        c.chunk <= BW_MAX_CHUNK && (c.in_dtype == NM_F32 || c.in_dtype == NM_BF16);
    if (c.kind == NM_LINEAR) return common;
    return common && c.kind == NM_MLP2 && nm_layers(c) == 2 && c.hidden > 0 && c.hidden <= 1024 && c.hidden % 32 == 0;
}

namespace {

template <bool TC>
cudaError_t bwd_launch(const nm_config& c, const nm_bwd_call& call, int* status, cudaStream_t s) {
    bwd_args a;
    a.T = call.T;
    a.q = call.q; a.k = call.k; a.v = call.v;
    a.alpha = call.alpha; a.eta = call.eta; a.beta = call.beta; a.c = call.c;
    a.ckpt = call.ckpt;
    a.Gy = call.Gy; a.GM = call.GM; a.GS = call.GS;
    a.dq = call.dq; a.dk = call.dk; a.dv = call.dv;
    a.dalpha = call.dalpha; a.deta = call.deta; a.dbeta = call.dbeta; a.dc = call.dc;
    a.dM0 = call.dM0; a.dS0 = call.dS0;
    a.ws = call.ws;
    a.ws_unit = nm_bwd_ws_floats(c);
    a.e_clip = call.e_clip;
    a.status = status;
    const unsigned units = (unsigned)call.units;
    const unsigned smem = TC ? TG_SMEM : 0;
    auto run = [&](auto kern, auto... args) {
        if (TC) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        kern<<<units, BW_THREADS, smem, s>>>(a, args...);
        return cudaGetLastError();
    };
    if (c.kind == NM_MLP2) {
        if (c.in_dtype == NM_BF16) return run(bwd_mlp_kernel<__nv_bfloat16, TC>, c.d, c.hidden, c.chunk, c.c_mode);
        return run(bwd_mlp_kernel<float, TC>, c.d, c.hidden, c.chunk, c.c_mode);
    }
    if (c.in_dtype == NM_BF16) return run(bwd_linear_kernel<__nv_bfloat16, TC>, c.d, c.chunk, c.c_mode);
    return run(bwd_linear_kernel<float, TC>, c.d, c.chunk, c.c_mode);
}

}  // namespace

// The reverse sweep with fp32 FFMA contractions.
cudaError_t nm_bwd_launch(const nm_config& c, const nm_bwd_call& call, cudaStream_t s) {
    return bwd_launch<false>(c, call, nullptr, s);
}

// The reverse sweep with tensor-core (tcgen05 kind::tf32) contractions; a
// timed-out wait is reported in `status`.
cudaError_t nm_bwd_launch_tc(const nm_config& c, const nm_bwd_call& call, int* status, cudaStream_t s) {
    return bwd_launch<true>(c, call, status, s);
}
