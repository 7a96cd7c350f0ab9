// Backward pass of the chunked linear memory: gradients of a loss of the
// forward's outputs (y, M_T, S_T) with respect to every input, for training
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
// linear kernel with a checkpoint array).
//
// This is an fp32 FFMA kernel: one CTA per unit, every step a block-wide loop
// over its output elements, matrices in a per-unit global workspace (read
// through L1 / L2).
#include "nm_internal.h"

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
};

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
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

template <typename Tin>
__global__ void __launch_bounds__(BW_THREADS) bwd_linear_kernel(bwd_args a, int d, int b, int c_mode) {
    __shared__ float s_a[BW_MAX_CHUNK], s_e[BW_MAX_CHUNK], s_b[BW_MAX_CHUNK], s_c[BW_MAX_CHUNK];
    __shared__ float sA[BW_MAX_CHUNK], sB[BW_MAX_CHUNK], sS[BW_MAX_CHUNK];
    __shared__ float s_gam[BW_MAX_CHUNK], s_u[BW_MAX_CHUNK];
    __shared__ float s_gA[BW_MAX_CHUNK], s_gS[BW_MAX_CHUNK], s_hg[BW_MAX_CHUNK], s_hu[BW_MAX_CHUNK];
    __shared__ float s_da[BW_MAX_CHUNK], s_de[BW_MAX_CHUNK], s_db[BW_MAX_CHUNK], s_dc[BW_MAX_CHUNK];
    __shared__ float red[BW_THREADS / 32];

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

    float* GM = a.ws + unit * a.ws_unit;  // [d][d] running adjoint of M (of the current chunk's end state)
    float* GS = GM + P;                  // [d][d] running adjoint of S
    float* Kf = GS + P;                  // [b][d] the chunk's k, q, v, Gy in fp32
    float* Qf = Kf + (size_t)b * d;
    float* Vf = Qf + (size_t)b * d;
    float* Gyf = Vf + (size_t)b * d;
    float* E = Gyf + (size_t)b * d;      // [b][d] e_i
    float* LR = E + (size_t)b * d;       // [b][d] 2 (Mc k_i - v_i), then lambda_r_i
    float* Mq = LR + (size_t)b * d;      // [b][d] Mc q_t
    float* Sq = Mq + (size_t)b * d;      // [b][d] Sc q_t
    float* GMk = Sq + (size_t)b * d;     // [b][d] GM k_i
    float* GSk = GMk + (size_t)b * d;    // [b][d] GS k_i
    float* GMtE = GSk + (size_t)b * d;   // [b][d] GM^T e_i
    float* GStE = GMtE + (size_t)b * d;  // [b][d] GS^T e_i
    float* Gam = GStE + (size_t)b * d;   // [b][b] Gamma_{t,i}
    float* U = Gam + (size_t)b * b;      // [b][b] u_{t,i}
    float* QK = U + (size_t)b * b;       // [b][b] q_t . k_i
    float* Z = QK + (size_t)b * b;       // [b][b] Gy_t . e_i (i <= t)

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
        // ---- the chunk's tokens and gates
        for (int i = tid; i < n * d; i += BW_THREADS) {
            Kf[i] = ld_f(k + t0 * d + i);
            Qf[i] = ld_f(q + t0 * d + i);
            Vf[i] = ld_f(v + t0 * d + i);
            Gyf[i] = Gy_u[t0 * d + i];
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
        // ---- r_i = Mc k_i - v_i (as 2 r in LR), e_i, Mc q_t, Sc q_t
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, o = idx % d;
            const float* mr = Mc + (size_t)o * d;
            const float* sr = Sc + (size_t)o * d;
            const float* kr = Kf + (size_t)i * d;
            const float* qr = Qf + (size_t)i * d;
            float rk = 0.f, mq = 0.f, sq = 0.f;
            for (int x = 0; x < d; ++x) {
                rk = fmaf(mr[x], kr[x], rk);
                mq = fmaf(mr[x], qr[x], mq);
                sq = fmaf(sr[x], qr[x], sq);
            }
            const float r2 = 2.0f * (rk - Vf[idx]);
            LR[idx] = r2;
            E[idx] = nm_clip_err(r2, a.e_clip);
            Mq[idx] = mq;
            Sq[idx] = sq;
        }
        __syncthreads();
        // ---- QK, Z; GM k_i, GS k_i, GM^T e_i, GS^T e_i
        for (int idx = tid; idx < n * n; idx += BW_THREADS) {
            const int t = idx / n, i = idx % n;
            float qk = 0.f, z = 0.f;
            for (int x = 0; x < d; ++x) {
                qk = fmaf(Qf[t * d + x], Kf[i * d + x], qk);
                z = fmaf(Gyf[t * d + x], E[i * d + x], z);
            }
            QK[t * b + i] = qk;
            Z[t * b + i] = i <= t ? z : 0.0f;
        }
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, o = idx % d;
            float gmk = 0.f, gsk = 0.f, gme = 0.f, gse = 0.f;
            for (int x = 0; x < d; ++x) {
                const float kx = Kf[i * d + x], ex = E[i * d + x];
                gmk = fmaf(GM[o * d + x], kx, gmk);
                gsk = fmaf(GS[o * d + x], kx, gsk);
                gme = fmaf(GM[x * d + o], ex, gme);  // (GM^T e_i)[o]
                gse = fmaf(GS[x * d + o], ex, gse);
            }
            GMk[idx] = gmk;
            GSk[idx] = gsk;
            GMtE[idx] = gme;
            GStE[idx] = gse;
        }
        __syncthreads();
        // ---- lambda_e, lambda_r = 2 [inside the clip] lambda_e, dv = -lambda_r
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, o = idx % d;
            float le = -s_gam[i] * GMk[idx] + s_u[i] * GSk[idx];
            for (int t = i; t < n; ++t) le = fmaf(-Gam[t * b + i] * QK[t * b + i], Gyf[t * d + o], le);
            const float r2 = LR[idx];
            const float lr = (r2 <= a.e_clip && r2 >= -a.e_clip) ? 2.0f * le : 0.0f;
            LR[idx] = lr;
            a.dv[(unit * T + t0) * d + idx] = -lr;
        }
        __syncthreads();
        // ---- dk, dq
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, x = idx % d;
            float g = -s_gam[i] * GMtE[idx] + s_u[i] * GStE[idx];
            for (int t = i; t < n; ++t) g = fmaf(-Gam[t * b + i] * Z[t * b + i], Qf[t * d + x], g);
            for (int o = 0; o < d; ++o) g = fmaf(Mc[o * d + x], LR[i * d + o], g);
            a.dk[(unit * T + t0) * d + idx] = g;
            const int t = i;  // the same index as a token t for dq
            float mg = 0.f, sgy = 0.f;
            for (int o = 0; o < d; ++o) {
                mg = fmaf(Mc[o * d + x], Gyf[t * d + o], mg);
                sgy = fmaf(Sc[o * d + x], Gyf[t * d + o], sgy);
            }
            float dqv = sA[t] * mg - sS[t] * sgy;
            for (int i2 = 0; i2 <= t; ++i2) dqv = fmaf(-Gam[t * b + i2] * Z[t * b + i2], Kf[i2 * d + x], dqv);
            a.dq[(unit * T + t0) * d + idx] = dqv;
        }
        // ---- scalar adjoints of A, sigma (per token) and of the chunk-end gamma, u (per column)
        for (int t = tid; t < n; t += BW_THREADS) {
            float ga = 0.f, gs = 0.f, hg = 0.f, hu = 0.f;
            for (int o = 0; o < d; ++o) {
                ga = fmaf(Gyf[t * d + o], Mq[t * d + o], ga);
                gs = fmaf(Gyf[t * d + o], Sq[t * d + o], gs);
                hg = fmaf(E[t * d + o], GMk[t * d + o], hg);
                hu = fmaf(E[t * d + o], GSk[t * d + o], hu);
            }
            s_gA[t] = ga;
            s_gS[t] = -gs;
            s_hg[t] = -hg;  // dL/dgamma_t (token t as a column i)
            s_hu[t] = hu;   // dL/du_t
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
        for (int i = tid; i < n; i += BW_THREADS) {
            float cG = 0.f, cU = 0.f;  // a_{t+1} gGamma_{t+1}, beta_{t+1} gu_{t+1}
            for (int t = n - 1; t >= i; --t) {
                const float gG = -QK[t * b + i] * Z[t * b + i] + (t == n - 1 ? s_hg[i] : 0.0f) + cG;
                const float gu = (t == n - 1 ? s_hu[i] : 0.0f) + s_e[t] * gG + cU;
                const float Gprev = t > i ? Gam[(t - 1) * b + i] : 0.0f;
                atomicAdd(&s_da[t], gG * Gprev);
                atomicAdd(&s_de[t], gG * U[t * b + i]);
                if (t > i) atomicAdd(&s_db[t], gu * U[(t - 1) * b + i]);
                else atomicAdd(&s_dc[i], gu);
                cG = s_a[t] * gG;
                cU = s_b[t] * gu;
            }
        }
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
        __syncthreads();
        for (int t = tid; t < n; t += BW_THREADS) {
            const long long g = unit * T + t0 + t;
            a.dalpha[g] = -s_da[t];  // a_t = 1 - alpha_t
            a.deta[g] = s_de[t];
            a.dbeta[g] = s_db[t] + (c_mode == NM_C_ONE_MINUS_BETA ? -s_dc[t] : 0.0f);
            if (a.dc) a.dc[g] = s_dc[t];
        }
        // ---- the chunk-start state's adjoint becomes the previous chunk's (GM, GS), in place
        const float An = sA[n - 1], Bn = sB[n - 1], Sn = sS[n - 1];
        for (int idx = tid; idx < P; idx += BW_THREADS) {
            const int o = idx / d, x = idx % d;
            float aq = 0.f, sq = 0.f, lk = 0.f;
            for (int t = 0; t < n; ++t) {
                const float gq = Gyf[t * d + o] * Qf[t * d + x];
                aq = fmaf(sA[t], gq, aq);
                sq = fmaf(sS[t], gq, sq);
                lk = fmaf(LR[t * d + o], Kf[t * d + x], lk);
            }
            const float gm = GM[idx], gs = GS[idx];
            GS[idx] = -sq - Sn * gm + Bn * gs;
            GM[idx] = aq + An * gm + lk;
        }
    }
    __syncthreads();
    for (int i = tid; i < P; i += BW_THREADS) {
        a.dM0[unit * P + i] = GM[i];
        a.dS0[unit * P + i] = GS[i];
    }
}

}  // namespace

size_t nm_bwd_linear_ws_floats(int d, int b) {
    return 2 * (size_t)d * d + 12 * (size_t)b * d + 4 * (size_t)b * b;
}

bool nm_bwd_supports(const nm_config& c) {
    return c.kind == NM_LINEAR && (c.d == 16 || c.d == 32 || c.d == 64 || c.d == 128) && c.chunk >= 1 &&
           c.chunk <= BW_MAX_CHUNK && (c.in_dtype == NM_F32 || c.in_dtype == NM_BF16);
}

cudaError_t nm_bwd_launch(const nm_config& c, const nm_bwd_call& call, cudaStream_t s) {
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
    a.ws_unit = nm_bwd_linear_ws_floats(c.d, c.chunk);
    a.e_clip = call.e_clip;
    const unsigned units = (unsigned)call.units;
    if (c.in_dtype == NM_BF16)
        bwd_linear_kernel<__nv_bfloat16><<<units, BW_THREADS, 0, s>>>(a, c.d, c.chunk, c.c_mode);
    else
        bwd_linear_kernel<float><<<units, BW_THREADS, 0, s>>>(a, c.d, c.chunk, c.c_mode);
    return cudaGetLastError();
}
