// tcgen05 tensor-core kernel for deeper MLP memories,
// M(x) = W_L silu(W_{L-1} ... silu(W_1 x)) with L >= 3 layers (the
// 0h-n0.github.io explainer, "ニューラル長期メモリモジュール": an MLP of L_M >= 1
// layers; "メモリ深度の影響": deeper memories lower perplexity).
//
// The chunked form of the 2-layer kernels, layer by layer.  Every token of a
// chunk takes its gradient at the chunk-start weights, so with x_0 = k,
// z_l = W_l x_{l-1}, x_l = silu(z_l), e = 2 (W_L x_{L-1} - v) (clipped for the
// Huber loss), delta_L = e and delta_l = (W_{l+1}^T delta_{l+1}) (.) silu'(z_l),
// layer l's weights after token t of the chunk are
//   W_l(t) = A_t W_l - sigma_t S_l - sum_{i<=t} Gamma_{t,i} delta_{l,i} x_{l-1,i}^T
// (A, sigma, Gamma from the gate scan, as in the linear kernel), retrieval
// runs the layers in order,
//   pre_l(t) = A_t W_l r_t - sigma_t S_l r_t - sum_{i<=t} Gamma_{t,i} (r_t . x_{l-1,i}) delta_{l,i},
// r = q for layer 1 and silu(pre_{l-1}) after it, y_t = pre_L(t), and the
// chunk-end state is
//   W_l <- A_n W_l - sigma_n S_l - sum_i gamma_i delta_{l,i} x_{l-1,i}^T
//   S_l <- B_n S_l + sum_i u_i delta_{l,i} x_{l-1,i}^T.
//
// Design.  One CTA (8 warps) per (batch, head) unit walks the sequence.  The
// fp32 state of a deep memory (2 P floats, 768 KB for 64 -> 256 -> 256 -> 64)
// exceeds one SM's TMEM and shared memory, so it stays in the caller's M_T /
// S_T buffers, updated in place once per chunk, where the L2 (126 MB) holds it
// for every unit at once; the chunk's activations go to a per-unit workspace
// the same way.  Every contraction of a chunk (the keys' forward per layer,
// the output error, the backward per layer, the Gamma-masked inner products,
// the retrieval per layer and the two state updates per layer) is one
// tensor-core GEMM C[M x N] += sum_k A[m][k] B[n][k] with the accumulator in
// TMEM: its operands are read from L2 by all threads in blocks of 32 k,
// scaled where the formula scales them (A_t, -sigma_t, gamma_i, u_i), rounded
// to tf32 (round to nearest) and written into shared memory in the 128-byte
// swizzled K-major layout, double-buffered so that the next block is staged
// while the tensor cores work on the current one; one thread issues
// tcgen05.mma kind::tf32 (M = 128 rows per tile, K = 8 per instruction).
// Transposed operands (W^T in the backward, delta^T and x^T in the updates)
// are the same loads with the strides swapped, so no transposed copy is ever
// stored.  Operands are fp32 rounded once to tf32 (11 significant bits):
// finer than a single bf16 rounding by a factor of 8, which the memory's
// sensitivity to gradient-path rounding needs, at half the bf16 rate and
// without the extra products of a hi/lo split.
//
// Every wait (the MMA completions) gives up after 2 s of %globaltimer; the
// CTA then records NM_ERR_DEVICE_TIMEOUT, issues nothing more, drains with
// bounded waits, frees its TMEM and exits.
#include <cuda_bf16.h>

#include "nm_internal.h"
#include "tc_common.cuh"

namespace {

using namespace tc;

constexpr int NT = 256;            // threads per CTA
constexpr int NTOK = 64;           // token rows of a chunk tile (chunks of at most 64 tokens)
constexpr int GSTR = NTOK + 1;     // padded row stride of Gamma in shared memory
constexpr uint32_t ATILE = 128 * 128;   // one M = 128 tile of 32 fp32 k: 16 KB
constexpr uint32_t BSTAGE = 256 * 128;  // up to 256 B rows of 32 fp32 k: 32 KB
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s

// Instruction descriptor of tcgen05.mma kind::tf32: tf32 A and B (format 2),
// fp32 accumulator, both operands K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((128u >> 4) << 24);
}

// K-major 128-byte-swizzle descriptor of a tile whose rows are 128 bytes (8-row
// groups 1024 bytes apart); a step of 8 tf32 along K adds 32 bytes.
__device__ __forceinline__ uint64_t kdesc(uint32_t saddr) { return sw128_desc(saddr, 16, 1024); }

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// fp32 -> tf32, round to nearest (ties away from zero); the low 13 bits are zero.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float silu_e(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float dsilu_e(float z) {
    const float s = 1.0f / (1.0f + expf(-z));
    return s * (1.0f + z * (1.0f - s));
}

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}

// One GEMM operand: element (r, k) is p[r * sr + k * sk] (fp32 or bf16) times
// rs[r] (if set) times ks[k] (if set) times mul.  Rows r >= rlim are not
// staged (the products in their row or column are never read); k >= klim
// stages as zero (it would add to products that are read).
struct Src {
    const void* p;
    long long sr, sk;
    const float* rs;
    const float* ks;
    float mul;
    int rlim, klim;
    int bf16;
};

__device__ __forceinline__ Src src(const void* p, long long sr, long long sk, int rlim, int klim, int bf16 = 0,
                                   const float* rs = nullptr, const float* ks = nullptr, float mul = 1.0f) {
    Src s;
    s.p = p; s.sr = sr; s.sk = sk; s.rs = rs; s.ks = ks; s.mul = mul; s.rlim = rlim; s.klim = klim; s.bf16 = bf16;
    return s;
}

// One chain of products into one accumulator: sum over K (a multiple of 32)
// of A (mt tiles of 128 rows) times B (N rows).  `fresh` starts the
// accumulator at zero.
struct Seg {
    Src a, b;
    int K;
    uint32_t col;  // TMEM column of M-tile 0's accumulator; tile m at col + m * N
    int fresh;
};

__device__ __forceinline__ float ld_elem(const Src& s, long long off) {
    if (s.bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(s.p)[off]);
    return reinterpret_cast<const float*>(s.p)[off];
}

// Stages columns k0 .. k0 + 31 of rows 0 .. R - 1 of operand s into a tile of
// R 128-byte rows (16-byte chunk kc of row r at r * 128 + ((kc ^ (r % 8)) * 16)),
// as tf32.  Consecutive threads take consecutive 16-byte chunks of a row when
// k is contiguous in memory, consecutive rows otherwise, so that the global
// loads of a warp are coalesced either way.
__device__ __forceinline__ void stage(uint32_t tile, int R, const Src& s, int k0, int tid) {
    const int rows = min(R, s.rlim);
    const int n = rows * 8;
    const bool kfast = s.sk == 1;
    for (int idx = tid; idx < n; idx += NT) {
        int r, kc;
        if (kfast) {
            r = idx >> 3;
            kc = idx & 7;
        } else {
            r = idx % rows;
            kc = idx / rows;
        }
        const int k = k0 + 4 * kc;
        float v[4];
        const long long base = (long long)r * s.sr + (long long)k * s.sk;
        if (kfast && k + 3 < s.klim) {
            if (s.bf16) {
                const uint2 w = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(s.p) + base);
                v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
            } else {
                const float4 w = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(s.p) + base);
                v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = k + j < s.klim ? ld_elem(s, base + (long long)j * s.sk) : 0.0f;
        }
        const float rf = (s.rs ? s.rs[r] : 1.0f) * s.mul;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float f = v[j] * rf;
            if (s.ks) f *= k + j < s.klim ? s.ks[k + j] : 0.0f;
            v[j] = f;
        }
        st_shared_v4(tile + (uint32_t)r * 128u + (((uint32_t)kc ^ ((uint32_t)r & 7u)) << 4), to_tf32(v[0]),
                     to_tf32(v[1]), to_tf32(v[2]), to_tf32(v[3]));
    }
}

// The double-buffered product pipeline of one CTA: two operand stages, one
// mbarrier per stage that the MMA commit of the stage's block arrives on.
struct Pipe {
    uint32_t a_st[2], b_st[2];  // shared-memory addresses of the A and B stages
    uint64_t* bars;             // [2]
    uint32_t ph[2];             // completions of each barrier waited for so far
    uint32_t pending[2];        // a commit on the barrier not yet waited for
    uint32_t tm;                // TMEM base address (lane 0, column 0)
    int failed;                 // a wait gave up: nothing more is issued
};

__device__ __forceinline__ bool pipe_wait(Pipe& p, int st) {
    if (!p.pending[st]) return true;
    const bool ok = mbar_wait(&p.bars[st], p.ph[st] & 1u, WAIT_NS);
    p.ph[st] += 1;
    p.pending[st] = 0;
    return ok;
}

// Runs the products of `nseg` segments (all threads of the CTA), each over
// its K in blocks of 32: block kb is staged into stage kb % 2 once the
// products of block kb - 2 have completed, then thread 0 issues its
// mt x 4 MMAs (K = 8 each) and commits them.  Returns with every product
// complete (or p.failed set).
__device__ void gemm(Pipe& p, const Seg* segs, int nseg, int mt, int N, int tid) {
    if (p.failed) return;
    const uint32_t idesc = idesc_tf32((uint32_t)N);
    int kb = 0;
    bool bad = false;
    for (int s = 0; s < nseg && !p.failed; ++s) {
        const Seg& g = segs[s];
        for (int k0 = 0; k0 < g.K; k0 += 32, ++kb) {
            const int st = kb & 1;
            if (!pipe_wait(p, st)) bad = true;
            stage(p.a_st[st], 128 * mt, g.a, k0, tid);
            stage(p.b_st[st], N, g.b, k0, tid);
            fence_proxy_async();
            if (__syncthreads_or(bad)) {
                p.failed = 1;
                break;
            }
            if (tid == 0) {
                tc_fence_after();
                for (int m = 0; m < mt; ++m) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_tf32(p.tm + g.col + (uint32_t)(m * N), kdesc(p.a_st[st] + m * ATILE + kk * 32),
                                 kdesc(p.b_st[st] + kk * 32), idesc, (g.fresh && k0 == 0 && kk == 0) ? 0u : 1u);
                }
                mma_commit(&p.bars[st]);
            }
            p.pending[st] = 1;
        }
    }
    if (!pipe_wait(p, kb & 1)) bad = true;
    if (!pipe_wait(p, (kb + 1) & 1)) bad = true;
    if (__syncthreads_or(bad)) p.failed = 1;
    tc_fence_after();
}

// Reads an M = 128 x N accumulator (mt tiles, tile m at column col + m N)
// out of TMEM: warp w takes lanes 32 (w % 4) .. + 31 and half w / 4 of the
// columns, 16 at a time, and calls f(row, first column, values[16]) for rows
// below `rows`.
template <typename F>
__device__ __forceinline__ void epilogue(const Pipe& p, uint32_t col, int mt, int N, int rows, int warp, int lane,
                                         F&& f) {
    if (p.failed) return;
    const int q = warp & 3, hf = warp >> 2;
    const int half = N / 2;
    for (int m = 0; m < mt; ++m) {
        const int row = 128 * m + 32 * q + lane;
        for (int c0 = hf * half; c0 < (hf + 1) * half; c0 += 16) {
            float v[16];
            tmem_ld_n(p.tm + ((uint32_t)(32 * q) << 16) + col + (uint32_t)(m * N + c0), v);
            if (row < rows) f(row, c0, v);
        }
    }
}

// The same over two accumulators of one tile (columns col0 and col1), read together.
template <typename F>
__device__ __forceinline__ void epilogue2(const Pipe& p, uint32_t col0, uint32_t col1, int N, int rows, int warp,
                                          int lane, F&& f) {
    if (p.failed) return;
    const int q = warp & 3, hf = warp >> 2;
    const int half = N / 2;
    const int row = 32 * q + lane;
    for (int c0 = hf * half; c0 < (hf + 1) * half; c0 += 16) {
        float v0[16], v1[16];
        const uint32_t base = p.tm + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
        tmem_ld_n(base + col0, base + col1, v0, v1);
        if (row < rows) f(row, c0, v0, v1);
    }
}

// Per-unit workspace, in floats: Z_l, x_l, delta_l for the hidden layers
// ([64][h] each), e ([64][d]), two retrieval activation buffers ([64][h]) and
// the Gamma-masked inner products G ([64][64]).
__host__ __device__ inline size_t deep_ws_floats(int d, int h, int L) {
    return (size_t)NTOK * (3 * (size_t)(L - 1) * h + 2 * (size_t)h + d + NTOK);
}

// Shared-memory bytes of a launch with mt_max M tiles of the hidden width.
__host__ __device__ inline uint32_t deep_smem_bytes(int mt_max) {
    return 2 * (uint32_t)mt_max * ATILE + 2 * BSTAGE + NTOK * GSTR * 4 + 9 * NTOK * 4 + 64 + 1024;
}

template <typename Tout>
__global__ void __launch_bounds__(NT, 1)
    tc_deep_kernel(nm_args a, int d, int hd, int L, int chunk, int c_mode, int mt_max) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t astage = (uint32_t)mt_max * ATILE;
    float* sG = reinterpret_cast<float*>(sm + 2 * astage + 2 * BSTAGE);  // Gamma [t][i], row stride GSTR
    float* ga = sG + NTOK * GSTR;  // 1 - alpha_t
    float* ge = ga + NTOK;         // eta_t
    float* gb = ge + NTOK;         // beta_t
    float* gc = gb + NTOK;         // c_t
    float* sA = gc + NTOK;         // A_t
    float* sB = sA + NTOK;         // B_t
    float* sSg = sB + NTOK;        // sigma_t
    float* gl = sSg + NTOK;        // gamma_i = Gamma_{n-1,i}
    float* ub = gl + NTOK;         // u_i = u_{n-1,i}
    uint64_t* bars = reinterpret_cast<uint64_t*>(ub + NTOK);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2);

    const long long unit = blockIdx.x;
    const long long T = a.T;
    const int h = hd;
    const long long P = 2LL * h * d + (long long)(L - 2) * h * h;
    const int b = chunk;
    const size_t th = (size_t)NTOK * h;

    float* ws = reinterpret_cast<float*>(a.scratch) + (size_t)unit * deep_ws_floats(d, h, L);
    float* Zw = ws;                       // [L-1][64][h]
    float* Xw = Zw + (L - 1) * th;        // [L-1][64][h]
    float* Dw = Xw + (L - 1) * th;        // [L-1][64][h]
    float* Ew = Dw + (L - 1) * th;        // [64][d]
    float* Rw = Ew + (size_t)NTOK * d;    // [2][64][h]
    float* Gw = Rw + 2 * th;              // [64][64]
    auto Z = [&](int l) { return Zw + (size_t)(l - 1) * th; };
    auto X = [&](int l) { return Xw + (size_t)(l - 1) * th; };
    auto Dl = [&](int l) { return l == L ? Ew : Dw + (size_t)(l - 1) * th; };
    auto woff = [&](int l) { return l == 1 ? 0LL : (long long)h * d + (long long)(l - 2) * h * h; };
    auto dim = [&](int l) { return (l == 0 || l == L) ? d : h; };  // width of x_l (x_L: the output)

    const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q) + unit * T * d;
    const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(a.k) + unit * T * d;
    const __nv_bfloat16* vp = reinterpret_cast<const __nv_bfloat16*>(a.v) + unit * T * d;
    const float* al = a.alpha + unit * T;
    const float* et = a.eta + unit * T;
    const float* be = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    Tout* y = reinterpret_cast<Tout*>(a.y) + unit * T * d;
    float* Mw = a.M_T + unit * P;  // the state, updated in place chunk by chunk
    float* Sw = a.S_T + unit * P;

    Pipe p;
    p.bars = bars;
    p.a_st[0] = smem_u32(sm);
    p.a_st[1] = smem_u32(sm + astage);
    p.b_st[0] = smem_u32(sm + 2 * astage);
    p.b_st[1] = smem_u32(sm + 2 * astage + BSTAGE);
    p.ph[0] = p.ph[1] = 0;
    p.pending[0] = p.pending[1] = 0;
    p.failed = 0;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    if (a.M_T != a.M0)
        for (long long i = tid; i < P; i += NT) Mw[i] = a.M0[unit * P + i];
    if (a.S_T != a.S0)
        for (long long i = tid; i < P; i += NT) Sw[i] = a.S0[unit * P + i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    p.tm = *s_tmem;

    // ends an epilogue: its TMEM reads and workspace writes are done before
    // the next products are staged and issued
    auto handoff = [&]() {
        tc_fence_before();
        __syncthreads();
    };

    for (long long t0 = 0; t0 < T && !p.failed; t0 += b) {
        const int n = (int)min((long long)b, T - t0);
        if (tid < n) {
            ga[tid] = 1.0f - al[t0 + tid];
            ge[tid] = et[t0 + tid];
            gb[tid] = be[t0 + tid];
            gc[tid] = momentum_c(c_mode, be[t0 + tid], cc, t0 + tid);
        }
        __syncthreads();
        // gate scan: column i of Gamma per thread (division-free recursion), A, B, sigma by one thread
        if (tid < n) {
            const int i = tid;
            float u = gc[i];
            float G = ge[i] * u;
            sG[i * GSTR + i] = G;
            for (int t = i + 1; t < n; ++t) {
                u *= gb[t];
                G = fmaf(ga[t], G, ge[t] * u);
                sG[t * GSTR + i] = G;
            }
            ub[i] = u;
            gl[i] = G;
        } else if (tid == 128) {
            float A = 1.f, Bc = 1.f, sg = 0.f;
            for (int t = 0; t < n; ++t) {
                A *= ga[t];
                Bc *= gb[t];
                sg = fmaf(ga[t], sg, ge[t] * Bc);
                sA[t] = A;
                sB[t] = Bc;
                sSg[t] = sg;
            }
        }
        __syncthreads();
        const __nv_bfloat16* kc = kp + t0 * d;  // this chunk's keys [t][x]
        const __nv_bfloat16* qc = qp + t0 * d;

        // keys' forward at the chunk-start weights: z_l = W_l x_{l-1}, x_l = silu(z_l)
        for (int l = 1; l < L; ++l) {
            const int in = dim(l - 1);
            Seg s[1];
            s[0].a = src(Mw + woff(l), in, 1, h, in);
            s[0].b = l == 1 ? src(kc, d, 1, n, in, 1) : src(X(l - 1), h, 1, n, in);
            s[0].K = in; s[0].col = 0; s[0].fresh = 1;
            const int mt = (h + 127) / 128;
            gemm(p, s, 1, mt, NTOK, tid);
            float* z = Z(l);
            float* x = X(l);
            epilogue(p, 0, mt, NTOK, h, warp, lane, [&](int j, int c0, const float* v) {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int t = c0 + c;
                    if (t < n) {
                        z[(size_t)t * h + j] = v[c];
                        x[(size_t)t * h + j] = silu_e(v[c]);
                    }
                }
            });
            handoff();
        }
        // e = 2 (W_L x_{L-1} - v), clipped for the Huber loss
        {
            Seg s[1];
            s[0].a = src(Mw + woff(L), h, 1, d, h);
            s[0].b = src(X(L - 1), h, 1, n, h);
            s[0].K = h; s[0].col = 0; s[0].fresh = 1;
            gemm(p, s, 1, 1, NTOK, tid);
            const __nv_bfloat16* vc = vp + t0 * d;
            epilogue(p, 0, 1, NTOK, d, warp, lane, [&](int o, int c0, const float* v) {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int t = c0 + c;
                    if (t < n) Ew[(size_t)t * d + o] = nm_clip_err(2.0f * (v[c] - __bfloat162float(vc[(size_t)t * d + o])), a.e_clip);
                }
            });
            handoff();
        }
        // backward: delta_l = (W_{l+1}^T delta_{l+1}) (.) silu'(z_l)
        for (int l = L - 1; l >= 1; --l) {
            const int up = dim(l + 1);
            Seg s[1];
            s[0].a = src(Mw + woff(l + 1), 1, h, h, up);  // (j, o) -> W_{l+1}[o][j]
            s[0].b = src(Dl(l + 1), up, 1, n, up);
            s[0].K = up; s[0].col = 0; s[0].fresh = 1;
            const int mt = (h + 127) / 128;
            gemm(p, s, 1, mt, NTOK, tid);
            const float* z = Z(l);
            float* dl = Dl(l);
            epilogue(p, 0, mt, NTOK, h, warp, lane, [&](int j, int c0, const float* v) {
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const int t = c0 + c;
                    if (t < n) dl[(size_t)t * h + j] = v[c] * dsilu_e(z[(size_t)t * h + j]);
                }
            });
            handoff();
        }
        // surprise_t = sqrt(sum_l ||delta_{l,t}||^2 ||x_{l-1,t}||^2): one warp per token
        if (a.surprise && !p.failed) {
            for (int t = warp; t < n; t += NT / 32) {
                float tot = 0.f;
                for (int l = 1; l <= L; ++l) {
                    const int in = dim(l - 1), out = dim(l);
                    float x2 = 0.f, d2 = 0.f;
                    for (int x = lane; x < in; x += 32) {
                        const float xv = l == 1 ? __bfloat162float(kc[(size_t)t * d + x]) : X(l - 1)[(size_t)t * h + x];
                        x2 = fmaf(xv, xv, x2);
                    }
                    const float* dl = Dl(l);
                    for (int o = lane; o < out; o += 32) d2 = fmaf(dl[(size_t)t * out + o], dl[(size_t)t * out + o], d2);
#pragma unroll
                    for (int sh = 16; sh > 0; sh >>= 1) {
                        x2 += __shfl_xor_sync(0xffffffffu, x2, sh);
                        d2 += __shfl_xor_sync(0xffffffffu, d2, sh);
                    }
                    tot = fmaf(d2, x2, tot);
                }
                if (lane == 0) a.surprise[unit * T + t0 + t] = sqrtf(tot);
            }
        }
        // retrieval, layer by layer
        for (int l = 1; l <= L && !p.failed; ++l) {
            const int in = dim(l - 1), out = dim(l);
            const void* xin = l == 1 ? (const void*)kc : (const void*)X(l - 1);
            const void* rin = l == 1 ? (const void*)qc : (const void*)(Rw + (size_t)((l - 1) & 1) * th);
            const long long xs = l == 1 ? d : h;
            const int bf = l == 1 ? 1 : 0;
            // G[t][i] = Gamma_{t,i} (r_t . x_{l-1,i}) for i <= t, from P^T[i][t] = x_{l-1,i} . r_t
            {
                Seg s[1];
                s[0].a = src(xin, xs, 1, n, in, bf);
                s[0].b = src(rin, xs, 1, n, in, bf);
                s[0].K = in; s[0].col = 0; s[0].fresh = 1;
                gemm(p, s, 1, 1, NTOK, tid);
                epilogue(p, 0, 1, NTOK, n, warp, lane, [&](int i, int c0, const float* v) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int t = c0 + c;
                        Gw[t * NTOK + i] = (i <= t && t < n) ? sG[t * GSTR + i] * v[c] : 0.0f;
                    }
                });
                handoff();
            }
            // pre_l^T[j][t] = A_t (W_l r_t)_j - sigma_t (S_l r_t)_j - sum_i delta_{l,i,j} G[t][i], one accumulator
            {
                const int mt = (out + 127) / 128;
                Seg s[3];
                s[0].a = src(Mw + woff(l), in, 1, out, in);
                s[0].b = src(rin, xs, 1, n, in, bf, sA);
                s[0].K = in; s[0].col = 0; s[0].fresh = 1;
                s[1].a = src(Sw + woff(l), in, 1, out, in);
                s[1].b = src(rin, xs, 1, n, in, bf, sSg, nullptr, -1.0f);
                s[1].K = in; s[1].col = 0; s[1].fresh = 0;
                s[2].a = src(Dl(l), 1, out, out, n);  // (j, i) -> delta_l[i][j]
                s[2].b = src(Gw, NTOK, 1, n, n, 0, nullptr, nullptr, -1.0f);
                s[2].K = NTOK; s[2].col = 0; s[2].fresh = 0;
                gemm(p, s, 3, mt, NTOK, tid);
                float* rn = Rw + (size_t)(l & 1) * th;
                epilogue(p, 0, mt, NTOK, out, warp, lane, [&](int j, int c0, const float* v) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int t = c0 + c;
                        if (t < n) {
                            if (l < L) {
                                rn[(size_t)t * h + j] = silu_e(v[c]);
                            } else {
                                Tout* yp = y + (t0 + t) * d + j;
                                const float o = nm_gated(a, yp, v[c]);
                                if constexpr (sizeof(Tout) == 2) *yp = __float2bfloat16_rn(o);
                                else *yp = o;
                            }
                        }
                    }
                });
                handoff();
            }
        }
        // chunk-end state, layer by layer, in tiles of 128 rows x up to 256 columns:
        // W_l <- A_n W_l - sigma_n S_l - sum_i gamma_i delta_{l,i} x_{l-1,i}^T, S_l <- B_n S_l + sum_i u_i (same)
        const float An = sA[n - 1], Bn = sB[n - 1], sn = sSg[n - 1];
        for (int l = 1; l <= L && !p.failed; ++l) {
            const int in = dim(l - 1), out = dim(l);
            const void* xin = l == 1 ? (const void*)kc : (const void*)X(l - 1);
            const long long xs = l == 1 ? d : h;
            const int bf = l == 1 ? 1 : 0;
            float* Wl = Mw + woff(l);
            float* Sl = Sw + woff(l);
            for (int m0 = 0; m0 < out; m0 += 128) {
                for (int x0 = 0; x0 < in; x0 += 256) {
                    const int N = min(256, in - x0);
                    Seg s[2];
                    s[0].a = src(Dl(l) + m0, 1, out, out - m0, n, 0, nullptr, gl);  // (j, i) -> gamma_i delta_l[i][m0 + j]
                    s[0].b = l == 1 ? src(kc + x0, 1, xs, N, n, bf) : src(X(l - 1) + x0, 1, xs, N, n, bf);
                    s[0].K = NTOK; s[0].col = 0; s[0].fresh = 1;
                    s[1].a = src(Dl(l) + m0, 1, out, out - m0, n, 0, nullptr, ub);
                    s[1].b = s[0].b;
                    s[1].K = NTOK; s[1].col = 256; s[1].fresh = 1;
                    (void)xin;
                    gemm(p, s, 2, 1, N, tid);
                    epilogue2(p, 0, 256, N, out - m0, warp, lane, [&](int j, int c0, const float* gw, const float* gs) {
                        float* wr = Wl + (size_t)(m0 + j) * in + x0 + c0;
                        float* sr = Sl + (size_t)(m0 + j) * in + x0 + c0;
#pragma unroll
                        for (int c = 0; c < 16; c += 4) {
                            const float4 w = *reinterpret_cast<const float4*>(wr + c);
                            const float4 sv = *reinterpret_cast<const float4*>(sr + c);
                            float4 wn, sn4;
                            wn.x = An * w.x - sn * sv.x - gw[c];
                            wn.y = An * w.y - sn * sv.y - gw[c + 1];
                            wn.z = An * w.z - sn * sv.z - gw[c + 2];
                            wn.w = An * w.w - sn * sv.w - gw[c + 3];
                            sn4.x = Bn * sv.x + gs[c];
                            sn4.y = Bn * sv.y + gs[c + 1];
                            sn4.z = Bn * sv.z + gs[c + 2];
                            sn4.w = Bn * sv.w + gs[c + 3];
                            *reinterpret_cast<float4*>(wr + c) = wn;
                            *reinterpret_cast<float4*>(sr + c) = sn4;
                        }
                    });
                    handoff();
                }
            }
        }
    }
    if (p.failed) {
        if (tid == 0 && a.status) atomicExch(a.status, NM_ERR_DEVICE_TIMEOUT);
        // let products still in flight land before the CTA leaves
        for (int st = 0; st < 2; ++st)
            if (p.pending[st]) mbar_wait(&bars[st], p.ph[st] & 1u, WAIT_NS);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(p.tm, 512);
}

template <typename Tout>
cudaError_t launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    const int mt_max = (c.hidden + 127) / 128;
    const uint32_t smem = deep_smem_bytes(mt_max);
    auto kern = tc_deep_kernel<Tout>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((long long)a.B * a.H), NT, smem, s>>>(a, c.d, c.hidden, nm_layers(c), c.chunk, c.c_mode,
                                                            mt_max);
    return cudaGetLastError();
}

}  // namespace

bool nm_tc_deep_supports(const nm_config& c) {
    return c.kind == NM_MLP2 && nm_layers(c) > 2 && c.in_dtype == NM_BF16 && (c.d == 32 || c.d == 64 || c.d == 128) &&
           c.hidden >= 32 && c.hidden <= 512 && c.hidden % 32 == 0 && c.chunk >= 1 && c.chunk <= NTOK;
}

size_t nm_tc_deep_scratch_bytes(const nm_config& c, int B, int H) {
    return sizeof(float) * deep_ws_floats(c.d, c.hidden, nm_layers(c)) * (size_t)B * (size_t)H;
}

cudaError_t nm_tc_deep_launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    if (!a.scratch || a.scratch_bytes < nm_tc_deep_scratch_bytes(c, a.B, a.H)) return cudaErrorInvalidValue;
    return c.out_dtype == NM_BF16 ? launch<__nv_bfloat16>(c, a, s) : launch<float>(c, a, s);
}
