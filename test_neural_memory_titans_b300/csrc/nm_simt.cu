// fp32 FFMA kernels for the neural-memory forward pass.
//
// These are the precision path (fp32 inputs at 1e-4 parity) and the
// any-shape path.  Both keep one (batch, head) unit per CTA for the whole
// sequence and take every gradient of a chunk at the chunk-start weights
// ("Titans: Imparare a Memorizzare al Tempo di Test", section "Addestramento
// Parallelizzato"); the update and retrieval rules are those of sections
// "Meccanismo di Aggiornamento della Memoria" / "Meccanismo di Dimenticanza"
// and of the 0h-n0.github.io explainer, "メモリ読み出し".
//
//  * Linear memory: the CTA holds M, S and the chunk-start copy W0 in
//    registers, one row per group of R threads.  Each chunk first forms the
//    errors e_t = 2 (W0 k_t - v_t) for all its tokens (they only need W0),
//    then advances S and M token by token with rank-1 updates and reads
//    y_t = M_t q_t.  Exact fp32 recurrence, no b x b matrices.
//
//  * 2-layer MLP memory: the chunked-parallel form.  With a_t = 1 - alpha_t
//    and, inside a chunk, A_t = prod_{j<=t} a_j, B_t = prod_{j<=t} beta_j,
//    sigma_t = a_t sigma_{t-1} + eta_t B_t,
//    u_{t,i} = c_i prod_{j=i+1..t} beta_j,
//    Gamma_{t,i} = a_t Gamma_{t-1,i} + eta_t u_{t,i}  (Gamma_{i-1,i} = 0),
//    the weights after token t are
//        W_t = A_t W0 - sigma_t S0 - sum_{i<=t} Gamma_{t,i} g_i,
//        S_t = B_t S0 + sum_{i<=t} u_{t,i} g_i,
//    so retrieval and the chunk-end state are matrix products of the chunk's
//    keys, queries, errors and backpropagated errors.  Gamma is built by the
//    recursion above (never by dividing cumulative products), so beta = 0 and
//    alpha = 1 are safe.  Intermediates live in a per-unit global workspace.
#include <cuda_bf16.h>

#include "nm_internal.h"

namespace {

template <typename T>
__device__ __forceinline__ float ld_in(const T* p);
template <>
__device__ __forceinline__ float ld_in<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_in<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T>
__device__ __forceinline__ void st_out(T* p, float x);
template <>
__device__ __forceinline__ void st_out<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_out<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float momentum_coef(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float dsilu_f(float z) {
    float s = 1.0f / (1.0f + expf(-z));
    return s * (1.0f + z * (1.0f - s));
}

// ----------------------------------------------------------------- linear

constexpr int LIN_SB = 64;  // tokens staged in shared memory at a time
constexpr int LIN_R = 4;    // threads per memory row

template <int D>
constexpr size_t lin_smem_bytes() {
    return sizeof(float) * (3 * LIN_SB * D + 4 * LIN_SB);
}

template <int D, typename Tin, typename Tout>
__global__ void __launch_bounds__(D * LIN_R) simt_linear_kernel(nm_args a, int chunk, int c_mode) {
    constexpr int R = LIN_R;
    constexpr int NT = D * R;
    constexpr int J = D / R;
    extern __shared__ float smem[];
    float* Ks = smem;               // [LIN_SB][D]
    float* Qs = Ks + LIN_SB * D;    // [LIN_SB][D]
    float* Es = Qs + LIN_SB * D;    // [LIN_SB][D] errors at W0
    float* ga = Es + LIN_SB * D;    // 1 - alpha
    float* ge = ga + LIN_SB;        // eta
    float* gb = ge + LIN_SB;        // beta
    float* gc = gb + LIN_SB;        // c

    const long long unit = blockIdx.x;
    const int tid = threadIdx.x;
    const int r = tid / R;
    const int s = tid % R;
    const long long T = a.T;
    const long long P = (long long)D * D;
    const Tin* q = (const Tin*)a.q + unit * T * D;
    const Tin* k = (const Tin*)a.k + unit * T * D;
    const Tin* v = (const Tin*)a.v + unit * T * D;
    const float* al = a.alpha + unit * T;
    const float* et = a.eta + unit * T;
    const float* be = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    Tout* y = (Tout*)a.y + unit * T * D;

    float M[J], S[J], W0[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        M[j] = a.M0[unit * P + (long long)r * D + j * R + s];
        S[j] = a.S0[unit * P + (long long)r * D + j * R + s];
    }
    for (long long t0 = 0; t0 < T; t0 += chunk) {
        const long long t1 = min(t0 + (long long)chunk, T);
#pragma unroll
        for (int j = 0; j < J; ++j) W0[j] = M[j];
        if (a.ckpt) {  // the chunk-start state, for the backward pass
            float* ck = a.ckpt + (unit * ((T + chunk - 1) / chunk) + t0 / chunk) * 2 * P + (long long)r * D;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                ck[j * R + s] = M[j];
                ck[P + j * R + s] = S[j];
            }
        }
        for (long long sb = t0; sb < t1; sb += LIN_SB) {
            const int n = (int)min((long long)LIN_SB, t1 - sb);
            __syncthreads();
            for (int i = tid; i < n * D; i += NT) {
                Ks[i] = ld_in(k + sb * D + i);
                Qs[i] = ld_in(q + sb * D + i);
            }
            for (int i = tid; i < n; i += NT) {
                ga[i] = 1.0f - al[sb + i];
                ge[i] = et[sb + i];
                gb[i] = be[sb + i];
                gc[i] = momentum_coef(c_mode, be[sb + i], cc, sb + i);
            }
            __syncthreads();
            // e_t = 2 (W0 k_t - v_t): gradient of ||W0 k - v||^2 is e k^T (clipped for the Huber loss)
            for (int t = 0; t < n; ++t) {
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < J; ++j) acc = fmaf(W0[j], Ks[t * D + j * R + s], acc);
#pragma unroll
                for (int o = R / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (s == 0) Es[t * D + r] = nm_clip_err(2.0f * (acc - ld_in(v + (sb + t) * D + r)), a.e_clip);
            }
            __syncthreads();
            if (a.surprise) {  // surprise_t = ||e_t k_t^T||_F = ||e_t|| ||k_t||, one thread per token
                for (int t = tid; t < n; t += NT) {
                    float e2 = 0.f, k2 = 0.f;
                    for (int o0 = 0; o0 < D; ++o0) {
                        const int o = (o0 + t) % D;  // rotated: conflict-free across the warp
                        e2 = fmaf(Es[t * D + o], Es[t * D + o], e2);
                        k2 = fmaf(Ks[t * D + o], Ks[t * D + o], k2);
                    }
                    a.surprise[unit * T + sb + t] = sqrtf(e2) * sqrtf(k2);
                }
            }
            for (int t = 0; t < n; ++t) {
                const float ce = gc[t] * Es[t * D + r];
                const float at = ga[t], eh = ge[t], bt = gb[t];
                float acc = 0.f;
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    const float kv = Ks[t * D + j * R + s];
                    S[j] = fmaf(bt, S[j], ce * kv);          // S = beta S + c e k^T
                    M[j] = fmaf(at, M[j], -eh * S[j]);       // M = (1-alpha) M - eta S
                    acc = fmaf(M[j], Qs[t * D + j * R + s], acc);
                }
#pragma unroll
                for (int o = R / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (s == 0 && a.y) st_out(y + (sb + t) * D + r, nm_gated(a, y + (sb + t) * D + r, acc));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
        a.M_T[unit * P + (long long)r * D + j * R + s] = M[j];
        a.S_T[unit * P + (long long)r * D + j * R + s] = S[j];
    }
}

template <int D, typename Tin, typename Tout>
cudaError_t launch_linear(const nm_config& c, const nm_args& a, cudaStream_t s) {
    constexpr size_t smem = lin_smem_bytes<D>();
    auto kern = simt_linear_kernel<D, Tin, Tout>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(a.B * a.H), D * LIN_R, smem, s>>>(a, c.chunk, c.c_mode);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_linear_d(const nm_config& c, const nm_args& a, cudaStream_t s) {
    switch (c.d) {
        case 16: return launch_linear<16, Tin, Tout>(c, a, s);
        case 32: return launch_linear<32, Tin, Tout>(c, a, s);
        case 64: return launch_linear<64, Tin, Tout>(c, a, s);
        case 128: return launch_linear<128, Tin, Tout>(c, a, s);
        default: return cudaErrorInvalidValue;
    }
}

// ----------------------------------------------------------------- MLP memories

constexpr int MLP_THREADS = 512;
constexpr int MLP_MAX_CHUNK = 256;

// M(x) = W_L silu(W_{L-1} ... silu(W1 x)), L >= 2 (the explainer's
// "ニューラル長期メモリモジュール": an MLP of L_M >= 1 layers; the 2-layer memory is
// L = 2).  The chunked form, layer by layer: every token's gradient is taken at
// the chunk-start weights, g_{l,i} = delta_{l,i} x_{l-1,i}^T with x_0 = k_i
// and delta_L = e_i, so each layer's weights after token t are
// W_l(t) = A_t W_l - sigma_t S_l - sum_{i<=t} Gamma_{t,i} delta_{l,i} x_{l-1,i}^T,
// and retrieval runs the layers in order with
// pre_l(t) = A_t W_l r - sigma_t S_l r - sum_i Gamma_{t,i} (x_{l-1,i} . r) delta_{l,i},
// r the previous layer's retrieval activation (r = q_t for layer 1).

// Every region of the deep kernel's workspace starts on a 16-byte boundary (float4 access).
__host__ __device__ inline size_t round4(size_t n) { return (n + 3) & ~(size_t)3; }
__host__ __device__ inline size_t deep_unit_floats(int d, int h, int b, int L) {
    const size_t P = 2 * (size_t)h * d + (size_t)(L - 2) * h * h;
    return 2 * round4((size_t)b * b) + 2 * round4(b) + 4 * (size_t)b * d + (3 * (size_t)(L - 1) + 2) * (size_t)b * h +
           2 * P;
}
__device__ __forceinline__ long long deep_off(int l, int d, int h) {  // offset of W_l in the packed parameters
    return l == 1 ? 0 : (long long)h * d + (long long)(l - 2) * h * h;
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(MLP_THREADS) simt_deep_kernel(nm_args a, int d, int hd, int L, int chunk,
                                                                int c_mode) {
    __shared__ float sA[MLP_MAX_CHUNK], sB[MLP_MAX_CHUNK], sSg[MLP_MAX_CHUNK];
    __shared__ float sa[MLP_MAX_CHUNK], se[MLP_MAX_CHUNK], sbt[MLP_MAX_CHUNK], sc[MLP_MAX_CHUNK];
    const long long unit = blockIdx.x;
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const long long T = a.T;
    const long long P = 2LL * hd * d + (long long)(L - 2) * hd * hd;
    const int b = chunk;
    const size_t bh = (size_t)b * hd;

    float* ws = (float*)a.scratch + unit * deep_unit_floats(d, hd, b, L);
    float* Gam = ws;                          // [b][b]   Gamma_{t,i}
    float* ub = Gam + round4((size_t)b * b);  // [b]      u_{n-1,i}
    float* gl = ub + round4(b);               // [b]      Gamma_{n-1,i}
    float* Kf = gl + round4(b);               // [b][d]
    float* Qf = Kf + (size_t)b * d;           // [b][d]
    float* Vf = Qf + (size_t)b * d;           // [b][d]
    float* E = Vf + (size_t)b * d;            // [b][d]   e_t (the output layer's delta)
    float* Z = E + (size_t)b * d;             // [L-1][b][h] pre-activations of the keys' forward
    float* X = Z + (L - 1) * bh;              // [L-1][b][h] activations x_l of the keys' forward
    float* Dl = X + (L - 1) * bh;             // [L-1][b][h] delta_l of the hidden layers
    float* R = Dl + (L - 1) * bh;             // [2][b][h]   retrieval activations (ping-pong)
    float* Pm = R + 2 * bh;                   // [b][b]   Gamma (.) inner products of the current layer
    float* Wt = Pm + round4((size_t)b * b);   // [P] the chunk-start weights, each layer transposed to [in][out],
    float* St = Wt + P;                // [P] and the momentum likewise: consecutive threads (consecutive
                                       //     outputs) then read consecutive addresses

    const Tin* q = (const Tin*)a.q + unit * T * d;
    const Tin* k = (const Tin*)a.k + unit * T * d;
    const Tin* v = (const Tin*)a.v + unit * T * d;
    const float* al = a.alpha + unit * T;
    const float* et = a.eta + unit * T;
    const float* be = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    Tout* y = (Tout*)a.y + unit * T * d;
    float* Mw = a.M_T + unit * P;  // the state, updated in place chunk by chunk
    float* Sw = a.S_T + unit * P;
    if (a.M_T != a.M0)
        for (long long i = tid; i < P; i += NT) Mw[i] = a.M0[unit * P + i];
    if (a.S_T != a.S0)
        for (long long i = tid; i < P; i += NT) Sw[i] = a.S0[unit * P + i];
    __syncthreads();

    for (long long t0 = 0; t0 < T; t0 += b) {
        const int n = (int)min((long long)b, T - t0);
        if (a.ckpt) {  // the chunk-start state (W1 .. W_L, then S), for the backward pass
            float* ck = a.ckpt + (unit * ((T + b - 1) / b) + t0 / b) * 2 * P;
            for (long long i = tid; i < P; i += NT) {
                ck[i] = Mw[i];
                ck[P + i] = Sw[i];
            }
        }
        for (int i = tid; i < n * d; i += NT) {
            Kf[i] = ld_in(k + t0 * d + i);
            Qf[i] = ld_in(q + t0 * d + i);
            Vf[i] = ld_in(v + t0 * d + i);
        }
        for (int i = tid; i < n; i += NT) {
            sa[i] = 1.0f - al[t0 + i];
            se[i] = et[t0 + i];
            sbt[i] = be[t0 + i];
            sc[i] = momentum_coef(c_mode, be[t0 + i], cc, t0 + i);
        }
        __syncthreads();
        // decay / momentum scan, one column i of Gamma per thread
        for (int i = tid; i < n; i += NT) {
            float u = sc[i];
            float G = se[i] * u;
            Gam[(size_t)i * b + i] = G;
            for (int t = i + 1; t < n; ++t) {
                u *= sbt[t];
                G = fmaf(sa[t], G, se[t] * u);
                Gam[(size_t)t * b + i] = G;
            }
            ub[i] = u;
            gl[i] = G;
        }
        if (tid == 0) {
            float A = 1.f, Bc = 1.f, sg = 0.f;
            for (int t = 0; t < n; ++t) {
                A *= sa[t];
                Bc *= sbt[t];
                sg = fmaf(sa[t], sg, se[t] * Bc);
                sA[t] = A;
                sB[t] = Bc;
                sSg[t] = sg;
            }
        }
        __syncthreads();
        // the chunk-start W_l and S_l transposed ([out][in] -> [in][out])
        for (int l = 1; l <= L; ++l) {
            const int in = l == 1 ? d : hd, out = l == L ? d : hd;
            const long long o0 = deep_off(l, d, hd);
            for (int idx = tid; idx < out * in; idx += NT) {
                const int j = idx / in, x = idx % in;
                Wt[o0 + (long long)x * out + j] = Mw[o0 + idx];
                St[o0 + (long long)x * out + j] = Sw[o0 + idx];
            }
        }
        __syncthreads();
        // keys' forward at the chunk-start weights: z_l = W_l x_{l-1}, x_l = silu(z_l)
        for (int l = 1; l < L; ++l) {
            const int in = l == 1 ? d : hd;
            const float* xin = l == 1 ? Kf : X + (l - 2) * bh;
            const float* Wtl = Wt + deep_off(l, d, hd);  // [in][h]
            const int h4 = hd / 4;
            for (int idx = tid; idx < n * h4; idx += NT) {  // four consecutive outputs per thread
                const int t = idx / h4, j = 4 * (idx % h4);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int x = 0; x < in; ++x) {
                    const float xv = xin[t * in + x];
                    const float4 w = *reinterpret_cast<const float4*>(Wtl + (long long)x * hd + j);
                    acc.x = fmaf(xv, w.x, acc.x); acc.y = fmaf(xv, w.y, acc.y);
                    acc.z = fmaf(xv, w.z, acc.z); acc.w = fmaf(xv, w.w, acc.w);
                }
                float* zr = Z + (l - 1) * bh + (size_t)t * hd + j;
                float* xr = X + (l - 1) * bh + (size_t)t * hd + j;
                zr[0] = acc.x; zr[1] = acc.y; zr[2] = acc.z; zr[3] = acc.w;
                xr[0] = silu_f(acc.x); xr[1] = silu_f(acc.y); xr[2] = silu_f(acc.z); xr[3] = silu_f(acc.w);
            }
            __syncthreads();
        }
        // e = 2 (W_L x_{L-1} - v), clipped for the Huber loss
        {
            const float* xl = X + (L - 2) * bh;
            const float* WtL = Wt + deep_off(L, d, hd);  // [h][d]
            const int d4 = d / 4;
            for (int idx = tid; idx < n * d4; idx += NT) {  // four consecutive outputs per thread
                const int t = idx / d4, o = 4 * (idx % d4);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j = 0; j < hd; ++j) {
                    const float xv = xl[t * hd + j];
                    const float4 w = *reinterpret_cast<const float4*>(WtL + (long long)j * d + o);
                    acc.x = fmaf(xv, w.x, acc.x); acc.y = fmaf(xv, w.y, acc.y);
                    acc.z = fmaf(xv, w.z, acc.z); acc.w = fmaf(xv, w.w, acc.w);
                }
                const int e0 = t * d + o;
                E[e0] = nm_clip_err(2.0f * (acc.x - Vf[e0]), a.e_clip);
                E[e0 + 1] = nm_clip_err(2.0f * (acc.y - Vf[e0 + 1]), a.e_clip);
                E[e0 + 2] = nm_clip_err(2.0f * (acc.z - Vf[e0 + 2]), a.e_clip);
                E[e0 + 3] = nm_clip_err(2.0f * (acc.w - Vf[e0 + 3]), a.e_clip);
            }
            __syncthreads();
        }
        // backward: delta_l = (W_{l+1}^T delta_{l+1}) (.) silu'(z_l), delta_L = e
        for (int l = L - 1; l >= 1; --l) {
            const int up_n = l + 1 == L ? d : hd;
            const float* up = l + 1 == L ? E : Dl + l * bh;
            const float* Wn = Mw + deep_off(l + 1, d, hd);  // [up_n][h]
            const int h4 = hd / 4;
            for (int idx = tid; idx < n * h4; idx += NT) {  // four consecutive outputs per thread
                const int t = idx / h4, j = 4 * (idx % h4);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int o = 0; o < up_n; ++o) {
                    const float u = up[t * up_n + o];
                    const float4 w = *reinterpret_cast<const float4*>(Wn + (long long)o * hd + j);
                    acc.x = fmaf(u, w.x, acc.x); acc.y = fmaf(u, w.y, acc.y);
                    acc.z = fmaf(u, w.z, acc.z); acc.w = fmaf(u, w.w, acc.w);
                }
                const size_t z0 = (l - 1) * bh + (size_t)t * hd + j;
                Dl[z0] = acc.x * dsilu_f(Z[z0]);
                Dl[z0 + 1] = acc.y * dsilu_f(Z[z0 + 1]);
                Dl[z0 + 2] = acc.z * dsilu_f(Z[z0 + 2]);
                Dl[z0 + 3] = acc.w * dsilu_f(Z[z0 + 3]);
            }
            __syncthreads();
        }
        if (a.surprise) {  // surprise_t = sqrt(sum_l ||delta_{l,t}||^2 ||x_{l-1,t}||^2), one thread per token
            for (int t = tid; t < n; t += NT) {
                float tot = 0.f;
                for (int l = 1; l <= L; ++l) {
                    const int in = l == 1 ? d : hd, out = l == L ? d : hd;
                    const float* xin = l == 1 ? Kf : X + (l - 2) * bh;
                    const float* dl = l == L ? E : Dl + (l - 1) * bh;
                    float x2 = 0.f, d2 = 0.f;
                    for (int x0 = 0; x0 < in; ++x0) {
                        const int x = (x0 + t) % in;  // rotated: conflict-free across the warp
                        x2 = fmaf(xin[t * in + x], xin[t * in + x], x2);
                    }
                    for (int o0 = 0; o0 < out; ++o0) {
                        const int o = (o0 + t) % out;
                        d2 = fmaf(dl[t * out + o], dl[t * out + o], d2);
                    }
                    tot = fmaf(d2, x2, tot);
                }
                a.surprise[unit * T + t0 + t] = sqrtf(tot);
            }
        }
        // retrieval, layer by layer
        const float* r = Qf;  // the previous layer's retrieval activation, [n][in]
        for (int l = 1; l <= L; ++l) {
            const int in = l == 1 ? d : hd, out = l == L ? d : hd;
            const float* xin = l == 1 ? Kf : X + (l - 2) * bh;
            const float* dl = l == L ? E : Dl + (l - 1) * bh;
            for (int idx = tid; idx < n * n; idx += NT) {  // Pm = Gamma (.) (r_t . x_{l-1,i}), lower triangle
                const int t = idx / n, i = idx % n;
                float acc = 0.f;
                if (i <= t) {
                    for (int x = 0; x < in; ++x) acc = fmaf(r[t * in + x], xin[i * in + x], acc);
                    acc *= Gam[(size_t)t * b + i];
                }
                Pm[(size_t)t * b + i] = acc;
            }
            __syncthreads();
            const float* Wtl = Wt + deep_off(l, d, hd);  // [in][out]
            const float* Stl = St + deep_off(l, d, hd);
            float* rn = R + (l & 1) * bh;
            const int o4 = out / 4;
            for (int idx = tid; idx < n * o4; idx += NT) {  // four consecutive outputs per thread
                const int t = idx / o4, j = 4 * (idx % o4);
                float mv[4] = {0.f, 0.f, 0.f, 0.f}, sv[4] = {0.f, 0.f, 0.f, 0.f}, gv[4] = {0.f, 0.f, 0.f, 0.f};
                for (int x = 0; x < in; ++x) {
                    const float rx = r[t * in + x];
                    const float4 w = *reinterpret_cast<const float4*>(Wtl + (long long)x * out + j);
                    const float4 st = *reinterpret_cast<const float4*>(Stl + (long long)x * out + j);
                    mv[0] = fmaf(rx, w.x, mv[0]); mv[1] = fmaf(rx, w.y, mv[1]);
                    mv[2] = fmaf(rx, w.z, mv[2]); mv[3] = fmaf(rx, w.w, mv[3]);
                    sv[0] = fmaf(rx, st.x, sv[0]); sv[1] = fmaf(rx, st.y, sv[1]);
                    sv[2] = fmaf(rx, st.z, sv[2]); sv[3] = fmaf(rx, st.w, sv[3]);
                }
                for (int i = 0; i <= t; ++i) {
                    const float pm = Pm[(size_t)t * b + i];
                    const float4 dv = *reinterpret_cast<const float4*>(dl + (size_t)i * out + j);
                    gv[0] = fmaf(pm, dv.x, gv[0]); gv[1] = fmaf(pm, dv.y, gv[1]);
                    gv[2] = fmaf(pm, dv.z, gv[2]); gv[3] = fmaf(pm, dv.w, gv[3]);
                }
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const float pre = sA[t] * mv[c4] - sSg[t] * sv[c4] - gv[c4];
                    if (l < L) rn[(size_t)t * out + j + c4] = silu_f(pre);
                    else if (a.y) st_out(y + (t0 + t) * d + j + c4, nm_gated(a, y + (t0 + t) * d + j + c4, pre));
                }
            }
            __syncthreads();
            r = rn;
        }
        // chunk-end state, layer by layer: W = A W0 - sigma S0 - sum_i gamma_i g_i, S = B S0 + sum_i u_i g_i
        const float An = sA[n - 1], Bn = sB[n - 1], sn = sSg[n - 1];
        for (int l = 1; l <= L; ++l) {
            const int in = l == 1 ? d : hd, out = l == L ? d : hd;
            const float* xin = l == 1 ? Kf : X + (l - 2) * bh;
            const float* dl = l == L ? E : Dl + (l - 1) * bh;
            float* Wl = Mw + deep_off(l, d, hd);
            float* Sl = Sw + deep_off(l, d, hd);
            const int in4 = in / 4;
            for (int idx = tid; idx < out * in4; idx += NT) {  // four consecutive inputs per thread
                const int j = idx / in4, x = 4 * (idx % in4);
                float gw[4] = {0.f, 0.f, 0.f, 0.f}, gs[4] = {0.f, 0.f, 0.f, 0.f};
                for (int i = 0; i < n; ++i) {
                    const float dj = dl[i * out + j];
                    const float4 xv = *reinterpret_cast<const float4*>(xin + (size_t)i * in + x);
                    const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const float gx = dj * xs[c4];
                        gw[c4] = fmaf(gl[i], gx, gw[c4]);
                        gs[c4] = fmaf(ub[i], gx, gs[c4]);
                    }
                }
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const long long e = (long long)j * in + x + c4;
                    const float w = Wl[e], sv = Sl[e];
                    Wl[e] = An * w - sn * sv - gw[c4];
                    Sl[e] = Bn * sv + gs[c4];
                }
            }
        }
        __syncthreads();
    }
}

template <typename Tin, typename Tout>
cudaError_t launch_deep(const nm_config& c, const nm_args& a, cudaStream_t s) {
    simt_deep_kernel<Tin, Tout><<<(unsigned)(a.B * a.H), MLP_THREADS, 0, s>>>(a, c.d, c.hidden, nm_layers(c), c.chunk,
                                                                            c.c_mode);
    return cudaGetLastError();
}


template <typename Tin>
cudaError_t dispatch_out(const nm_config& c, const nm_args& a, cudaStream_t s) {
    if (c.kind == NM_LINEAR)
        return c.out_dtype == NM_BF16 ? launch_linear_d<Tin, __nv_bfloat16>(c, a, s)
                                      : launch_linear_d<Tin, float>(c, a, s);
    return c.out_dtype == NM_BF16 ? launch_deep<Tin, __nv_bfloat16>(c, a, s) : launch_deep<Tin, float>(c, a, s);
}

}  // namespace

bool nm_simt_supports(const nm_config& c) {
    if (c.chunk < 1 || c.chunk > 256) return false;
    const bool d_ok = c.d == 16 || c.d == 32 || c.d == 64 || c.d == 128;
    if (!d_ok) return false;
    if (c.kind == NM_LINEAR) return true;
    return c.hidden > 0 && c.hidden <= 1024 && c.hidden % 32 == 0;
}

size_t nm_simt_scratch_bytes(const nm_config& c, int B, int H) {
    if (c.kind == NM_LINEAR) return 0;
    return sizeof(float) * deep_unit_floats(c.d, c.hidden, c.chunk, nm_layers(c)) * (size_t)B * (size_t)H;
}

cudaError_t nm_simt_launch(const nm_config& c, const nm_args& a, cudaStream_t s, long long* launches) {
    cudaError_t e = c.in_dtype == NM_BF16 ? dispatch_out<__nv_bfloat16>(c, a, s) : dispatch_out<float>(c, a, s);
    if (e == cudaSuccess) *launches += 1;
    return e;
}
