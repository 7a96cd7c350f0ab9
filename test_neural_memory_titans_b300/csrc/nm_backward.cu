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
    return 4 * (size_t)h * d + 14 * (size_t)b * d + 17 * (size_t)b * h + 6 * (size_t)b * b;
}

template <typename Tin>
__global__ void __launch_bounds__(BW_THREADS) bwd_mlp_kernel(bwd_args a, int d, int hd, int b, int c_mode) {
    __shared__ float s_a[BW_MAX_CHUNK], s_e[BW_MAX_CHUNK], s_b[BW_MAX_CHUNK], s_c[BW_MAX_CHUNK];
    __shared__ float sA[BW_MAX_CHUNK], sB[BW_MAX_CHUNK], sS[BW_MAX_CHUNK];
    __shared__ float s_gam[BW_MAX_CHUNK], s_u[BW_MAX_CHUNK];
    __shared__ float s_gA[BW_MAX_CHUNK], s_gS[BW_MAX_CHUNK], s_hg[BW_MAX_CHUNK], s_hu[BW_MAX_CHUNK];
    __shared__ float s_da[BW_MAX_CHUNK], s_de[BW_MAX_CHUNK], s_db[BW_MAX_CHUNK], s_dc[BW_MAX_CHUNK];
    __shared__ float red[BW_THREADS / 32];

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

    // running adjoints of the end state, in the packed order: [dL/dW1 | dL/dW2] then [dL/dS1 | dL/dS2]
    float* GW1 = a.ws + unit * a.ws_unit;  // [h][d]
    float* GW2 = GW1 + HD;                 // [d][h]
    float* GS1 = GW2 + HD;                 // [h][d]
    float* GS2 = GS1 + HD;                 // [d][h]
    float* p_ = GS2 + HD;
    auto take = [&](size_t n_) { float* r_ = p_; p_ += n_; return r_; };
    const size_t bd = (size_t)b * d, bh = (size_t)b * hd, bb = (size_t)b * b;
    float *Kf = take(bd), *Qf = take(bd), *Vf = take(bd), *Gyf = take(bd), *E = take(bd), *R2 = take(bd);
    float *W2b = take(bd), *S2b = take(bd), *G2a = take(bd), *H2a = take(bd), *G1td = take(bd), *H1td = take(bd);
    float *DE = take(bd), *DK = take(bd);
    float *Zs = take(bh), *Ak = take(bh), *PH = take(bh), *PP = take(bh), *DL = take(bh), *PSI = take(bh);
    float *Bt = take(bh), *W1q = take(bh), *S1q = take(bh), *DH = take(bh), *DP = take(bh), *DAk = take(bh);
    float *G1k = take(bh), *H1k = take(bh), *G2te = take(bh), *H2te = take(bh), *DZ = take(bh);
    float *Gam = take(bb), *U = take(bb), *QK = take(bb), *AA = take(bb), *Zy = take(bb), *Zh = take(bb);

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
        // ---- F1: z, a(k), silu'(z); W1 q, S1 q; QK
        for (int idx = tid; idx < n * hd; idx += BW_THREADS) {
            const int i = idx / hd, j = idx % hd;
            const float* w1 = W1c + (size_t)j * d;
            const float* s1 = S1c + (size_t)j * d;
            float z = 0.f, wq = 0.f, sq = 0.f;
            for (int x = 0; x < d; ++x) {
                z = fmaf(w1[x], Kf[i * d + x], z);
                wq = fmaf(w1[x], Qf[i * d + x], wq);
                sq = fmaf(s1[x], Qf[i * d + x], sq);
            }
            const float s = sig_f(z);
            Zs[idx] = z;
            Ak[idx] = z * s;
            PH[idx] = s * (1.0f + z * (1.0f - s));
            W1q[idx] = wq;
            S1q[idx] = sq;
        }
        for (int idx = tid; idx < n * n; idx += BW_THREADS) {
            const int t = idx / n, i = idx % n;
            float qk = 0.f;
            for (int x = 0; x < d; ++x) qk = fmaf(Qf[t * d + x], Kf[i * d + x], qk);
            QK[t * b + i] = qk;
        }
        __syncthreads();
        // ---- F2: e = clip(2 (W2 a - v))
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, o = idx % d;
            const float* w2 = W2c + (size_t)o * hd;
            float yh = 0.f;
            for (int j = 0; j < hd; ++j) yh = fmaf(w2[j], Ak[i * hd + j], yh);
            const float r2 = 2.0f * (yh - Vf[idx]);
            R2[idx] = r2;
            E[idx] = nm_clip_err(r2, a.e_clip);
        }
        __syncthreads();
        // ---- F3: p = W2^T e, delta = p (.) silu'(z)
        for (int idx = tid; idx < n * hd; idx += BW_THREADS) {
            const int i = idx / hd, j = idx % hd;
            float p = 0.f;
            for (int o = 0; o < d; ++o) p = fmaf(W2c[(size_t)o * hd + j], E[i * d + o], p);
            PP[idx] = p;
            DL[idx] = p * PH[idx];
        }
        __syncthreads();
        // ---- F4: h_t, b_t = silu(h_t), silu'(h_t)
        for (int idx = tid; idx < n * hd; idx += BW_THREADS) {
            const int t = idx / hd, j = idx % hd;
            float hh = sA[t] * W1q[idx] - sS[t] * S1q[idx];
            for (int i = 0; i <= t; ++i) hh = fmaf(-Gam[t * b + i] * QK[t * b + i], DL[i * hd + j], hh);
            const float s = sig_f(hh);
            Bt[idx] = hh * s;
            PSI[idx] = s * (1.0f + hh * (1.0f - s));
        }
        __syncthreads();
        // ---- F5: AA, Zy; W2 b_t, S2 b_t
        for (int idx = tid; idx < n * n; idx += BW_THREADS) {
            const int t = idx / n, i = idx % n;
            float aa = 0.f, zy = 0.f;
            for (int j = 0; j < hd; ++j) aa = fmaf(Bt[t * hd + j], Ak[i * hd + j], aa);
            for (int o = 0; o < d; ++o) zy = fmaf(Gyf[t * d + o], E[i * d + o], zy);
            AA[t * b + i] = aa;
            Zy[t * b + i] = i <= t ? zy : 0.0f;
        }
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int t = idx / d, o = idx % d;
            const float* w2 = W2c + (size_t)o * hd;
            const float* s2 = S2c + (size_t)o * hd;
            float wb = 0.f, sb = 0.f;
            for (int j = 0; j < hd; ++j) {
                wb = fmaf(w2[j], Bt[t * hd + j], wb);
                sb = fmaf(s2[j], Bt[t * hd + j], sb);
            }
            W2b[idx] = wb;
            S2b[idx] = sb;
        }
        __syncthreads();
        // ---- B2: db_t and dh_t = db_t (.) silu'(h_t)
        for (int idx = tid; idx < n * hd; idx += BW_THREADS) {
            const int t = idx / hd, j = idx % hd;
            float wg = 0.f, sg = 0.f;
            for (int o = 0; o < d; ++o) {
                wg = fmaf(W2c[(size_t)o * hd + j], Gyf[t * d + o], wg);
                sg = fmaf(S2c[(size_t)o * hd + j], Gyf[t * d + o], sg);
            }
            float db = sA[t] * wg - sS[t] * sg;
            for (int i = 0; i <= t; ++i) db = fmaf(-Gam[t * b + i] * Zy[t * b + i], Ak[i * hd + j], db);
            DH[idx] = db * PSI[idx];
        }
        // ---- B5: the end state's adjoints against the chunk's vectors
        for (int idx = tid; idx < n * hd; idx += BW_THREADS) {
            const int i = idx / hd, j = idx % hd;
            float g1k = 0.f, h1k = 0.f, g2e = 0.f, h2e = 0.f;
            for (int x = 0; x < d; ++x) {
                g1k = fmaf(GW1[(size_t)j * d + x], Kf[i * d + x], g1k);
                h1k = fmaf(GS1[(size_t)j * d + x], Kf[i * d + x], h1k);
            }
            for (int o = 0; o < d; ++o) {
                g2e = fmaf(GW2[(size_t)o * hd + j], E[i * d + o], g2e);
                h2e = fmaf(GS2[(size_t)o * hd + j], E[i * d + o], h2e);
            }
            G1k[idx] = g1k; H1k[idx] = h1k; G2te[idx] = g2e; H2te[idx] = h2e;
        }
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, o = idx % d;
            float g2a = 0.f, h2a = 0.f, g1d = 0.f, h1d = 0.f;
            for (int j = 0; j < hd; ++j) {
                g2a = fmaf(GW2[(size_t)o * hd + j], Ak[i * hd + j], g2a);
                h2a = fmaf(GS2[(size_t)o * hd + j], Ak[i * hd + j], h2a);
                g1d = fmaf(GW1[(size_t)j * d + o], DL[i * hd + j], g1d);  // (G1^T delta_i)[x = o]
                h1d = fmaf(GS1[(size_t)j * d + o], DL[i * hd + j], h1d);
            }
            G2a[idx] = g2a; H2a[idx] = h2a; G1td[idx] = g1d; H1td[idx] = h1d;
        }
        __syncthreads();
        // ---- B3: Zh; B4: dq
        for (int idx = tid; idx < n * n; idx += BW_THREADS) {
            const int t = idx / n, i = idx % n;
            float zh = 0.f;
            for (int j = 0; j < hd; ++j) zh = fmaf(DH[t * hd + j], DL[i * hd + j], zh);
            Zh[t * b + i] = i <= t ? zh : 0.0f;
        }
        __syncthreads();
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int t = idx / d, x = idx % d;
            float wd = 0.f, sd = 0.f;
            for (int j = 0; j < hd; ++j) {
                wd = fmaf(W1c[(size_t)j * d + x], DH[t * hd + j], wd);
                sd = fmaf(S1c[(size_t)j * d + x], DH[t * hd + j], sd);
            }
            float g = sA[t] * wd - sS[t] * sd;
            for (int i = 0; i <= t; ++i) g = fmaf(-Gam[t * b + i] * Zh[t * b + i], Kf[i * d + x], g);
            a.dq[(unit * T + t0) * d + idx] = g;
        }
        // ---- B6: ddelta -> dp and the silu'' part of dz; the direct parts of de, da, dk
        for (int idx = tid; idx < n * hd; idx += BW_THREADS) {
            const int i = idx / hd, j = idx % hd;
            float dd = -s_gam[i] * G1k[idx] + s_u[i] * H1k[idx];
            float da = -s_gam[i] * G2te[idx] + s_u[i] * H2te[idx];
            for (int t = i; t < n; ++t) {
                const float gm = Gam[t * b + i];
                dd = fmaf(-gm * QK[t * b + i], DH[t * hd + j], dd);
                da = fmaf(-gm * Zy[t * b + i], Bt[t * hd + j], da);
            }
            const float z = Zs[idx], s = sig_f(z);
            DP[idx] = dd * PH[idx];
            DZ[idx] = dd * PP[idx] * (s * (1.0f - s) * (2.0f + z * (1.0f - 2.0f * s)));
            DAk[idx] = da;
        }
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, o = idx % d;
            float de = -s_gam[i] * G2a[idx] + s_u[i] * H2a[idx];
            float dk = -s_gam[i] * G1td[idx] + s_u[i] * H1td[idx];
            for (int t = i; t < n; ++t) {
                const float gm = Gam[t * b + i];
                de = fmaf(-gm * AA[t * b + i], Gyf[t * d + o], de);
                dk = fmaf(-gm * Zh[t * b + i], Qf[t * d + o], dk);
            }
            DE[idx] = de;
            DK[idx] = dk;
        }
        __syncthreads();
        // ---- B7: de += W2 dp; dr = 2 [inside the clip] de; dv = -dr
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, o = idx % d;
            const float* w2 = W2c + (size_t)o * hd;
            float de = DE[idx];
            for (int j = 0; j < hd; ++j) de = fmaf(w2[j], DP[i * hd + j], de);
            const float r2 = R2[idx];
            const float dr = (r2 <= a.e_clip && r2 >= -a.e_clip) ? 2.0f * de : 0.0f;
            R2[idx] = dr;
            a.dv[(unit * T + t0) * d + idx] = -dr;
        }
        __syncthreads();
        // ---- B8: da += W2^T dr; dz += da (.) silu'(z)
        for (int idx = tid; idx < n * hd; idx += BW_THREADS) {
            const int i = idx / hd, j = idx % hd;
            float da = DAk[idx];
            for (int o = 0; o < d; ++o) da = fmaf(W2c[(size_t)o * hd + j], R2[i * d + o], da);
            DZ[idx] = fmaf(da, PH[idx], DZ[idx]);
        }
        __syncthreads();
        // ---- B9: dk += W1^T dz
        for (int idx = tid; idx < n * d; idx += BW_THREADS) {
            const int i = idx / d, x = idx % d;
            float g = DK[idx];
            for (int j = 0; j < hd; ++j) g = fmaf(W1c[(size_t)j * d + x], DZ[i * hd + j], g);
            a.dk[(unit * T + t0) * d + idx] = g;
        }
        // ---- B10: scalar adjoints of A, sigma and of the chunk-end gamma, u
        for (int t = tid; t < n; t += BW_THREADS) {
            float ga = 0.f, gs = 0.f, hg = 0.f, hu = 0.f;
            for (int o = 0; o < d; ++o) {
                ga = fmaf(Gyf[t * d + o], W2b[t * d + o], ga);
                gs = fmaf(Gyf[t * d + o], S2b[t * d + o], gs);
                hg = fmaf(E[t * d + o], G2a[t * d + o], hg);
                hu = fmaf(E[t * d + o], H2a[t * d + o], hu);
            }
            for (int j = 0; j < hd; ++j) {
                ga = fmaf(DH[t * hd + j], W1q[t * hd + j], ga);
                gs = fmaf(DH[t * hd + j], S1q[t * hd + j], gs);
                hg = fmaf(DL[t * hd + j], G1k[t * hd + j], hg);
                hu = fmaf(DL[t * hd + j], H1k[t * hd + j], hu);
            }
            s_gA[t] = ga;
            s_gS[t] = -gs;
            s_hg[t] = -hg;
            s_hu[t] = hu;
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
        for (int i = tid; i < n; i += BW_THREADS) {
            float cG = 0.f, cU = 0.f;
            for (int t = n - 1; t >= i; --t) {
                const float gG = -(AA[t * b + i] * Zy[t * b + i] + QK[t * b + i] * Zh[t * b + i]) +
                                 (t == n - 1 ? s_hg[i] : 0.0f) + cG;
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
            a.dalpha[g] = -s_da[t];
            a.deta[g] = s_de[t];
            a.dbeta[g] = s_db[t] + (c_mode == NM_C_ONE_MINUS_BETA ? -s_dc[t] : 0.0f);
            if (a.dc) a.dc[g] = s_dc[t];
        }
        // ---- B11: the chunk-start state's adjoints, in place
        const float An = sA[n - 1], Bn = sB[n - 1], Sn = sS[n - 1];
        for (long long idx = tid; idx < HD; idx += BW_THREADS) {  // W1, S1 [h][d]
            const int j = (int)(idx / d), x = (int)(idx % d);
            float aq = 0.f, sq = 0.f, zk = 0.f;
            for (int t = 0; t < n; ++t) {
                const float hq = DH[t * hd + j] * Qf[t * d + x];
                aq = fmaf(sA[t], hq, aq);
                sq = fmaf(sS[t], hq, sq);
                zk = fmaf(DZ[t * hd + j], Kf[t * d + x], zk);
            }
            const float gw = GW1[idx], gs = GS1[idx];
            GS1[idx] = -sq - Sn * gw + Bn * gs;
            GW1[idx] = aq + An * gw + zk;
        }
        for (long long idx = tid; idx < HD; idx += BW_THREADS) {  // W2, S2 [d][h]
            const int o = (int)(idx / hd), j = (int)(idx % hd);
            float ab = 0.f, sb = 0.f, ed = 0.f;
            for (int t = 0; t < n; ++t) {
                const float gb = Gyf[t * d + o] * Bt[t * hd + j];
                ab = fmaf(sA[t], gb, ab);
                sb = fmaf(sS[t], gb, sb);
                ed = fmaf(E[t * d + o], DP[t * hd + j], ed);
                ed = fmaf(R2[t * d + o], Ak[t * hd + j], ed);
            }
            const float gw = GW2[idx], gs = GS2[idx];
            GS2[idx] = -sb - Sn * gw + Bn * gs;
            GW2[idx] = ab + An * gw + ed;
        }
    }
    __syncthreads();
    for (long long i = tid; i < P; i += BW_THREADS) {
        a.dM0[unit * P + i] = GW1[i];
        a.dS0[unit * P + i] = GS1[i];
    }
}

}  // namespace

size_t nm_bwd_linear_ws_floats(int d, int b) {
    return 2 * (size_t)d * d + 12 * (size_t)b * d + 4 * (size_t)b * b;
}

size_t nm_bwd_ws_floats(const nm_config& c) {
    return c.kind == NM_LINEAR ? nm_bwd_linear_ws_floats(c.d, c.chunk) : bwd_mlp_ws_floats(c.d, c.hidden, c.chunk);
}

bool nm_bwd_supports(const nm_config& c) {
    const bool common = (c.d == 16 || c.d == 32 || c.d == 64 || c.d == 128) && c.chunk >= 1 &&
                        c.chunk <= BW_MAX_CHUNK && (c.in_dtype == NM_F32 || c.in_dtype == NM_BF16);
    if (c.kind == NM_LINEAR) return common;
    return common && c.kind == NM_MLP2 && nm_layers(c) == 2 && c.hidden > 0 && c.hidden <= 1024 && c.hidden % 32 == 0;
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
    a.ws_unit = nm_bwd_ws_floats(c);
    a.e_clip = call.e_clip;
    const unsigned units = (unsigned)call.units;
    if (c.kind == NM_MLP2) {
        if (c.in_dtype == NM_BF16)
            bwd_mlp_kernel<__nv_bfloat16><<<units, BW_THREADS, 0, s>>>(a, c.d, c.hidden, c.chunk, c.c_mode);
        else
            bwd_mlp_kernel<float><<<units, BW_THREADS, 0, s>>>(a, c.d, c.hidden, c.chunk, c.c_mode);
    } else if (c.in_dtype == NM_BF16) {
        bwd_linear_kernel<__nv_bfloat16><<<units, BW_THREADS, 0, s>>>(a, c.d, c.chunk, c.c_mode);
    } else {
        bwd_linear_kernel<float><<<units, BW_THREADS, 0, s>>>(a, c.d, c.chunk, c.c_mode);
    }
    return cudaGetLastError();
}
