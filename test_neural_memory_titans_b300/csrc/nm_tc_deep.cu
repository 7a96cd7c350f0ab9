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
// S_T buffers, updated in place once per chunk, where the L2 (126 MB) holds it.
// Every contraction of a chunk (the keys' forward per layer, the output error,
// the backward per layer, the Gamma-masked inner products, the retrieval per
// layer and the two state updates per layer) is one tensor-core GEMM
// C[M x N] += sum_k A[m][k] B[n][k], tcgen05.mma kind::tf32 (M = 128 rows per
// tile, K = 8 per instruction) with the accumulator in TMEM.
//
// Its operands come from a per-unit workspace of operand tiles: tf32 values
// (rounded to nearest) already in the 128-byte-swizzled K-major layout the
// tensor cores read, in blocks of 32 k (a block of R rows is R x 128 bytes).
// Each producer writes its results there in every form a later product
// consumes: the keys' forward epilogue writes x_l as [t][j] (a B operand) and
// as [j][t] (the update's B operand), the backward epilogue delta_l as [t][j]
// and as [j][t] three times (plain, times gamma_t, times u_t), the retrieval
// epilogue r_l three times (plain, times A_t, times -sigma_t), the inner-product
// epilogue -G, and the update epilogue, next to the fp32 state, W_l and S_l as
// [o][i] and W_l as [i][o] for the backward.  A block of a product is then one
// or two bulk copies (cp.async.bulk) into shared memory, issued by a copy
// thread (warp 0) while an MMA thread (warp 1) issues the products: the two
// meet only at the full / empty mbarriers of a ring of 2 to 8 stages, the
// copies run up to ns - 1 blocks ahead, and no thread stages operands.  The
// scalings of the formula (A_t, -sigma_t, gamma_i, u_i) live in those copies,
// so each of retrieval's three chains and each update adds into its
// accumulator directly.  Transposes cost nothing extra: a thread that holds a
// row of an accumulator writes a row of one form and a column of the other.
// fp32 rounded once to tf32 (11 significant bits) is finer than a single
// bf16 rounding by a factor of 8, which the memory's sensitivity to
// gradient-path rounding needs, at half the bf16 rate and without the extra
// products of a hi/lo split.
//
// Every wait (bulk copies, MMA completions) gives up after 2 s of
// %globaltimer; the CTA then records NM_ERR_DEVICE_TIMEOUT, issues nothing
// more, drains what it issued with bounded waits, frees its TMEM and exits.
#include <cuda_bf16.h>

#include "nm_internal.h"
#include "tc_common.cuh"

namespace {

using namespace tc;

constexpr int NT = 256;            // threads per CTA
constexpr int NTOK = 64;           // token rows of a chunk tile (chunks of at most 64 tokens)
constexpr int GSTR = NTOK + 1;     // padded row stride of Gamma in shared memory
constexpr uint32_t ATILE = 128 * 128;   // one M = 128 tile of 32 fp32 k: 16 KB
constexpr uint32_t STAGE_AREA = 196608; // operand stages: 192 KB, cut per GEMM into stages of its block size
constexpr int MAX_STAGES = 8;
constexpr uint32_t EPI_TBUF_BYTES = 36864;                          // 8 warps x 32 x 33 floats, rounded up
constexpr uint32_t EPI_BYTES = EPI_TBUF_BYTES + (NT / 32) * 3 * 4096;  // + three 4 KB block buffers per warp
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

// silu and its derivative with the hardware-tanh sigmoid (relative error about
// 2^-11, the size of the tf32 rounding every result goes through next).
__device__ __forceinline__ float silu_e(float z) { return z * sigmoid_f(z); }
__device__ __forceinline__ float dsilu_e(float z) {
    const float s = sigmoid_f(z);
    return s * (1.0f + z * (1.0f - s));
}

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}


// ---- operand tiles in global memory
// A matrix of R rows and K columns (K a multiple of 32) stored as K / 32
// blocks of R x 32 tf32 values, each block R 128-byte rows with the 16-byte
// chunks of row r permuted by (chunk ^ (r % 8)): the K-major 128-byte swizzle,
// so that any 8-row-aligned run of rows of a block, copied verbatim to a
// 1024-byte-aligned shared-memory address, is a tensor-core operand.
struct Tile {
    float* p;
    int R;
};

// Float offset of element (r, k).
__device__ __forceinline__ uint32_t toff(int R, int r, int k) {
    return (uint32_t)(k >> 5) * (uint32_t)R * 32u + (uint32_t)r * 32u +
           (((((uint32_t)k & 31u) >> 2) ^ ((uint32_t)r & 7u)) << 2) + ((uint32_t)k & 3u);
}

// Per-unit workspace (floats), every region a multiple of 64 floats.
struct Layout {
    size_t tw[NM_MAX_LAYERS + 1], ts[NM_MAX_LAYERS + 1], twt[NM_MAX_LAYERS + 1];  // state tiles per layer
    size_t tk, tkt, tq, tqa, tqs;                                              // this chunk's keys and queries
    size_t tx[NM_MAX_LAYERS], txt[NM_MAX_LAYERS], z[NM_MAX_LAYERS];            // hidden layers 1 .. L-1
    size_t td[NM_MAX_LAYERS + 1], tdt[NM_MAX_LAYERS + 1], tdg[NM_MAX_LAYERS + 1], tdu[NM_MAX_LAYERS + 1];
    size_t tr[NM_MAX_LAYERS], tra[NM_MAX_LAYERS], trs[NM_MAX_LAYERS];
    size_t tg;
    size_t total;
};

__host__ __device__ inline Layout deep_layout(int d, int h, int L) {
    Layout o;
    size_t at = 0;
    auto take = [&](size_t n) { const size_t r = at; at += (n + 63) & ~(size_t)63; return r; };
    for (int l = 1; l <= L; ++l) {
        const size_t in = l == 1 ? d : h, out = l == L ? d : h;
        o.tw[l] = take(out * in);
        o.ts[l] = take(out * in);
        o.twt[l] = l >= 2 ? take(in * out) : 0;
    }
    o.tk = take((size_t)NTOK * d);
    o.tkt = take((size_t)d * NTOK);
    o.tq = take((size_t)NTOK * d);
    o.tqa = take((size_t)NTOK * d);
    o.tqs = take((size_t)NTOK * d);
    for (int l = 1; l < L; ++l) {
        o.tx[l] = take((size_t)NTOK * h);
        o.txt[l] = take((size_t)h * NTOK);
        o.z[l] = take((size_t)NTOK * h);
        o.tr[l] = take((size_t)NTOK * h);
        o.tra[l] = take((size_t)NTOK * h);
        o.trs[l] = take((size_t)NTOK * h);
    }
    for (int l = 1; l <= L; ++l) {  // delta_l (delta_L = e): [t][j] and [j][t] plain, x gamma_t, x u_t
        const size_t w = l == L ? d : h;
        o.td[l] = take((size_t)NTOK * w);
        o.tdt[l] = take(w * NTOK);
        o.tdg[l] = take(w * NTOK);
        o.tdu[l] = take(w * NTOK);
    }
    o.tg = take((size_t)NTOK * NTOK);
    o.total = at;
    return o;
}

// Shared memory: the operand stages, Gamma, the gate vectors, the mbarriers and flags.
constexpr uint32_t MISC_BYTES = 4096;  // producer state, segments, workspace layout
constexpr uint32_t DEEP_SMEM_BYTES = STAGE_AREA + NTOK * GSTR * 4 + 9 * NTOK * 4 + 256 + MISC_BYTES + 1024;
static_assert(DEEP_SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGE_AREA >= EPI_BYTES, "the epilogues' buffers fit in the operand stages");
static_assert(STAGE_AREA >= 2 * (4 * ATILE + 256 * 128), "two stages of the largest one-atom block fit");

// ---- the product pipeline: one thread copies operand blocks and issues the MMAs

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Makes this thread's generic-proxy global writes visible to later bulk copies.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// One chain of products into one accumulator: K (a multiple of 64) of A
// (rows a_row0 .. of tile set a, mt tiles of 128 rows) times B (rows
// b_row0 .. b_row0 + N - 1 of tile set b).  `fresh` starts at zero.
struct Seg {
    const float* a;
    int a_R, a_row0;
    const float* b;
    int b_R, b_row0;
    int K;
    uint32_t col;  // TMEM column of M-tile 0's accumulator; tile m at col + m * N
    int fresh;
};

__device__ __forceinline__ Seg seg(const Tile& a, int a_row0, const Tile& b, int b_row0, int K, uint32_t col,
                                   int fresh) {
    Seg s;
    s.a = a.p; s.a_R = a.R; s.a_row0 = a_row0;
    s.b = b.p; s.b_R = b.R; s.b_row0 = b_row0;
    s.K = K; s.col = col; s.fresh = fresh;
    return s;
}

// What the two producer threads work from, in shared memory: the stage
// area, barriers and TMEM base, the segments of the GEMM being run, and per
// stage the copies issued into it (by the copy thread) and the products that
// read it (by the MMA thread).  Stage s's n-th copy completes phase n of
// full[s], the products that read it phase n of empty[s].
struct Prod {
    uint32_t area, tm;
    uint64_t* full;   // [MAX_STAGES] a stage's copies landed
    uint64_t* empty;  // [MAX_STAGES] the products that read a stage completed
    uint64_t* done;   // all products of a GEMM completed (or a producer gave up)
    int* s_fail;
    int skip;                    // test hook: the call's first GEMM gets no copies (its products' wait expires)
    uint32_t ncopy[MAX_STAGES];  // copies issued into stage s so far (copy thread)
    uint32_t nmma[MAX_STAGES];   // products issued from stage s so far (MMA thread)
    Seg segs[3];
};

struct Pipe {
    uint32_t area;    // shared address of the operand stages
    uint64_t* full;   // [MAX_STAGES] a stage's copies landed
    uint64_t* empty;  // [MAX_STAGES] the products that read a stage completed
    uint64_t* done;   // all products of a GEMM completed (or the producer gave up)
    int* s_fail;
    Prod* prod;       // shared
    uint32_t tm;
    uint32_t ndone;   // GEMMs finished (every thread)
    int failed;
};

// The block geometry of one GEMM.  A block is 64 k (two 32-k swizzle atoms;
// one atom where two such stages would not fit) of A rows (up to mt tiles)
// and N B rows; the blocks cut the stage area into ns = area / block stages
// (at most MAX_STAGES) and block b goes to stage b % ns.
struct Geo {
    uint32_t na, boff, bb, sbytes;
    int lk, ns, total;
};
__device__ __forceinline__ Geo geometry(const Seg* segs, int nseg, int mt, int N) {
    Geo g;
    uint32_t amax = 0;
    for (int s = 0; s < nseg; ++s) amax = max(amax, (uint32_t)min(128 * mt, segs[s].a_R - segs[s].a_row0) * 128u);
    g.bb = (uint32_t)N * 128u;  // one 32-k atom of B (a multiple of 1024: N % 8 == 0)
    g.na = 2u * 2u * (amax + g.bb) <= STAGE_AREA ? 2u : 1u;
    g.lk = g.na == 2u ? 6 : 5;  // log2 of the k per block
    g.total = 0;
    for (int s = 0; s < nseg; ++s) g.total += segs[s].K >> g.lk;
    g.boff = g.na * amax;       // amax is a multiple of 1024 (rows % 8 == 0)
    g.sbytes = g.boff + g.na * g.bb;
    g.ns = (int)min((uint32_t)MAX_STAGES, STAGE_AREA / g.sbytes);
    return g;
}

// The copy thread (warp 0, lane 0): block b's operands into stage b % ns,
// once the products that read the stage's previous block completed (its
// empty barrier), so that the copies run up to ns blocks ahead of the
// products.
__device__ __noinline__ void run_copies(Prod* prod, int nseg, int mt, int N) {
    if (prod->skip) {  // (the test hook: nothing is copied, so the MMA thread's first wait gives up)
        prod->skip = 0;
        return;
    }
    const Seg* segs = prod->segs;
    const Geo geo = geometry(segs, nseg, mt, N);
    bool ok = true;
    for (int b = 0, is = 0, ikb = 0; b < geo.total; ++b) {
        const int st = b % geo.ns;
        const uint32_t n = prod->ncopy[st];
        if (n > 0) {
            ok = mbar_wait(&prod->empty[st], (n - 1u) & 1u, WAIT_NS);
            if (!ok) break;
        }
        const Seg& g = segs[is];
        const int arows = min(128 * mt, g.a_R - g.a_row0);
        const uint32_t ab = (uint32_t)arows * 128u, bb = geo.bb, na = geo.na;
        const uint32_t sa = prod->area + (uint32_t)st * geo.sbytes;
        const float* ga0 = g.a + ((size_t)(na * ikb) * g.a_R + g.a_row0) * 32;
        const float* gb0 = g.b + ((size_t)(na * ikb) * g.b_R + g.b_row0) * 32;
        uint64_t* fb = &prod->full[st];
        mbar_arrive_expect_tx(fb, na * (ab + bb));
        if (na == 1u || (g.a_row0 == 0 && arows == g.a_R)) {  // the atoms of A are one contiguous run
            bulk_g2s(sa, ga0, na * ab, fb);
        } else {
            bulk_g2s(sa, ga0, ab, fb);
            bulk_g2s(sa + ab, ga0 + (size_t)g.a_R * 32, ab, fb);
        }
        if (na == 1u || (g.b_row0 == 0 && N == g.b_R)) {
            bulk_g2s(sa + geo.boff, gb0, na * bb, fb);
        } else {
            bulk_g2s(sa + geo.boff, gb0, bb, fb);
            bulk_g2s(sa + geo.boff + bb, gb0 + (size_t)g.b_R * 32, bb, fb);
        }
        prod->ncopy[st] = n + 1u;
        if (++ikb == (g.K >> geo.lk)) {
            ikb = 0;
            ++is;
        }
    }
    if (!ok) *reinterpret_cast<volatile int*>(prod->s_fail) = 1;
}

// The MMA thread (warp 1, lane 0): waits for each block's copies, issues its
// products (M = 128 per tile, K = 8 each) and commits them to the stage's
// empty barrier; the last commit goes to `done`.  A wait that gives up marks
// the failure and arrives on `done` so that nobody waits longer.
__device__ __noinline__ void run_mmas(Prod* prod, int nseg, int mt, int N) {
    const Seg* segs = prod->segs;
    const Geo geo = geometry(segs, nseg, mt, N);
    const uint32_t idesc = idesc_tf32((uint32_t)N);
    bool ok = true;
    for (int b = 0, cs = 0, ckb = 0; b < geo.total; ++b) {
        const int st = b % geo.ns;
        const uint32_t n = prod->nmma[st];
        ok = mbar_wait(&prod->full[st], n & 1u, WAIT_NS);
        if (!ok) break;
        tc_fence_after();
        const Seg& g = segs[cs];
        const uint32_t ab = (uint32_t)min(128 * mt, g.a_R - g.a_row0) * 128u;
        const uint32_t sa = prod->area + (uint32_t)st * geo.sbytes;
        for (uint32_t hk = 0; hk < geo.na; ++hk) {
            for (int m = 0; m < mt; ++m) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_tf32(prod->tm + g.col + (uint32_t)(m * N), kdesc(sa + hk * ab + (uint32_t)m * ATILE + kk * 32),
                             kdesc(sa + geo.boff + hk * geo.bb + kk * 32), idesc,
                             (g.fresh && ckb == 0 && hk == 0 && kk == 0) ? 0u : 1u);
            }
        }
        mma_commit(&prod->empty[st]);
        prod->nmma[st] = n + 1u;
        if (++ckb == (g.K >> geo.lk)) {
            ckb = 0;
            ++cs;
        }
    }
    if (ok && !*reinterpret_cast<volatile int*>(prod->s_fail)) {
        mma_commit(prod->done);
    } else {
        *reinterpret_cast<volatile int*>(prod->s_fail) = 1;
        mbar_arrive(prod->done);
    }
}

// Every thread: run one GEMM (threads 0 and 32 drive it) and wait for it.  Returns
// false once any wait has given up.
__device__ __forceinline__ bool gemm(Pipe& p, const Seg* segs, int nseg, int mt, int N, int tid) {
    if (p.failed) return false;
    if (tid < 64) {  // the producers' warp-mates wait at a warp barrier, not on the mbarrier: a
                     // try_wait may suspend the whole warp and with it the producer
        if (tid == 0)
            for (int i = 0; i < nseg; ++i) p.prod->segs[i] = segs[i];
        asm volatile("bar.sync 1, 64;" ::: "memory");  // warps 0 and 1: the segments are in place
        if (tid == 0) run_copies(p.prod, nseg, mt, N);
        if (tid == 32) run_mmas(p.prod, nseg, mt, N);
        __syncwarp();
    }
    const bool ok = mbar_wait(p.done, p.ndone & 1u, 2 * WAIT_NS);
    p.ndone += 1;
    if (__syncthreads_or(!ok || *reinterpret_cast<volatile int*>(p.s_fail))) p.failed = 1;
    tc_fence_after();
    return !p.failed;
}

// Visits an M = 128 x N accumulator (mt tiles, tile m at column col + m N,
// N / 2 a multiple of 32) in blocks of 32 rows x 32 columns read from TMEM:
// warp w takes the rows of lanes 32 (w % 4) .. + 31 (its TMEM sub-partition)
// and column half w / 4, and calls f(first row, first column, v) with v this
// lane's row (row first row + lane), for row blocks below `rows` (a multiple
// of 32).
template <typename F>
__device__ __forceinline__ void epi32(const Pipe& p, uint32_t col, int mt, int N, int rows, int warp, F&& f) {
    if (p.failed) return;
    const int q = warp & 3, hf = warp >> 2, half = N / 2;
    for (int m = 0; m < mt; ++m) {
        const int jb = 128 * m + 32 * q;
        if (jb >= rows) continue;  // the same for the whole warp
        for (int c0 = hf * half; c0 < (hf + 1) * half; c0 += 32) {
            float v[32];
            tmem_ld_n(p.tm + ((uint32_t)(32 * q) << 16) + col + (uint32_t)(m * N + c0), v);
            f(jb, c0, v);
        }
    }
}

// The same for two accumulators of one tile (columns col0 and col1), read together.
template <typename F>
__device__ __forceinline__ void epi32x2(const Pipe& p, uint32_t col0, uint32_t col1, int N, int rows, int warp,
                                        F&& f) {
    if (p.failed) return;
    const int q = warp & 3, hf = warp >> 2, half = N / 2;
    const int jb = 32 * q;
    if (jb >= rows) return;
    for (int c0 = hf * half; c0 < (hf + 1) * half; c0 += 32) {
        float v0[32], v1[32];
        const uint32_t base = p.tm + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
        tmem_ld_n(base + col0, base + col1, v0, v1);
        f(jb, c0, v0, v1);
    }
}

// A 32 x 32 block held one row per lane (v) as one column per lane (u, u[r]
// = row r of the block at column `lane`), through 32 x 33 floats of this
// warp's shared memory (conflict-free both ways).
__device__ __forceinline__ void transpose32(float* buf, const float (&v)[32], float (&u)[32], int lane) {
#pragma unroll
    for (int c = 0; c < 32; ++c) buf[lane * 33 + c] = v[c];
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 32; ++r) u[r] = buf[r * 33 + lane];
    __syncwarp();
}

// Block writes of operand tiles.  A 32 x 32 block of a tile (rows r0 ..
// r0 + 31, r0 a multiple of 32, and the 32 k of one block) is one contiguous
// 4 KB piece of global memory: the warp that holds it (lane = k - k0, one
// value per row) writes it into one of three 4 KB buffers of its own in shared
// memory, in the tile's swizzled layout, and lane 0 sends it with one bulk
// copy.  A buffer is reused once at most one later copy is still reading it
// (so two blocks may be open at once).
__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

struct Stager {
    uint32_t base;  // this warp's three 4 KB buffers
    int cnt;        // blocks begun so far
};

__device__ __forceinline__ uint32_t blk_begin(Stager& sg, int lane) {
    const uint32_t buf = sg.base + (uint32_t)(sg.cnt % 3) * 4096u;
    ++sg.cnt;
    if (lane == 0) bulk_wait_read1();
    __syncwarp();
    return buf;
}
// value v of block row i (0..31) at k = k0 + lane
__device__ __forceinline__ void blk_put(uint32_t buf, int i, float v, int lane) {
    st_shared_f32(buf + (uint32_t)i * 128u + ((((uint32_t)lane >> 2) ^ ((uint32_t)i & 7u)) << 4) + ((uint32_t)lane & 3u) * 4u,
                  __uint_as_float(to_tf32(v)));
}
__device__ __forceinline__ void blk_end(uint32_t buf, const Tile& t, int r0, int k0, int lane) {
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) {
        bulk_s2g(t.p + ((size_t)(k0 >> 5) * t.R + r0) * 32, buf, 4096u);
        bulk_commit();
    }
}
// the whole block from one array: v[i] = row r0 + i at k = k0 + lane
__device__ __forceinline__ void put_block(Stager& sg, const Tile& t, int r0, int k0, const float (&v)[32], int lane) {
    const uint32_t buf = blk_begin(sg, lane);
#pragma unroll
    for (int i = 0; i < 32; ++i) blk_put(buf, i, v[i], lane);
    blk_end(buf, t, r0, k0, lane);
}

template <typename Tout>
__global__ void __launch_bounds__(NT, 1)
    tc_deep_kernel(nm_args a, int d, int hd, int L, int chunk, int c_mode) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this warp's 32 x 33 transpose buffer and three 4 KB block buffers, in the
    // operand stages (idle while the epilogues run; 132 KB of the 192 KB)
    float* tbuf = reinterpret_cast<float*>(sm) + warp * 32 * 33;
    Stager sg;
    sg.base = smem_u32(sm) + EPI_TBUF_BYTES + (uint32_t)warp * 3u * 4096u;
    sg.cnt = 0;
    float* sG = reinterpret_cast<float*>(sm + STAGE_AREA);  // Gamma [t][i], row stride GSTR
    float* ga = sG + NTOK * GSTR;  // 1 - alpha_t
    float* ge = ga + NTOK;         // eta_t
    float* gb = ge + NTOK;         // beta_t
    float* gc = gb + NTOK;         // c_t
    float* sA = gc + NTOK;         // A_t
    float* sB = sA + NTOK;         // B_t
    float* sSg = sB + NTOK;        // sigma_t
    float* gl = sSg + NTOK;        // gamma_i = Gamma_{n-1,i}
    float* ub = gl + NTOK;         // u_i = u_{n-1,i}
    uint64_t* bars = reinterpret_cast<uint64_t*>(ub + NTOK);  // full[4], empty[4], done
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * MAX_STAGES + 1);
    int* s_fail = reinterpret_cast<int*>(s_tmem + 1);
    unsigned char* misc = reinterpret_cast<unsigned char*>(bars) + 256;
    Prod* s_prod = reinterpret_cast<Prod*>(misc);
    Layout* s_lo = reinterpret_cast<Layout*>(misc + ((sizeof(Prod) + 15) & ~(size_t)15));

    const long long unit = blockIdx.x;
    const long long T = a.T;
    const int h = hd;
    const long long P = 2LL * h * d + (long long)(L - 2) * h * h;
    const int b = chunk;
    if (tid == 0) *s_lo = deep_layout(d, h, L);
    __syncthreads();
    const volatile Layout& lo = *s_lo;  // read where used (a shared load), not held in registers
    float* ws = reinterpret_cast<float*>(a.scratch) + (size_t)unit * lo.total;
    auto dim = [&](int l) { return (l == 0 || l == L) ? d : h; };  // width of x_l (x_L: the output)
    auto woff = [&](int l) { return l == 1 ? 0LL : (long long)h * d + (long long)(l - 2) * h * h; };
    auto TW = [&](int l) { return Tile{ws + lo.tw[l], dim(l)}; };      // W_l [o][i]
    auto TS = [&](int l) { return Tile{ws + lo.ts[l], dim(l)}; };      // S_l [o][i]
    auto TWt = [&](int l) { return Tile{ws + lo.twt[l], dim(l - 1)}; };  // W_l [i][o], l >= 2
    const Tile TK{ws + lo.tk, NTOK}, TKt{ws + lo.tkt, d};               // k [t][x], [x][t]
    const Tile TQ{ws + lo.tq, NTOK}, TQa{ws + lo.tqa, NTOK}, TQs{ws + lo.tqs, NTOK};  // q, A_t q, -sigma_t q
    auto TX = [&](int l) { return Tile{ws + lo.tx[l], NTOK}; };   // x_l [t][j]
    auto TXt = [&](int l) { return Tile{ws + lo.txt[l], h}; };    // x_l [j][t]
    auto Zp = [&](int l) { return ws + lo.z[l]; };                 // z_l [t][j], fp32
    auto TR = [&](int l) { return Tile{ws + lo.tr[l], NTOK}; };   // r_l [t][j], times A_t, times -sigma_t
    auto TRa = [&](int l) { return Tile{ws + lo.tra[l], NTOK}; };
    auto TRs = [&](int l) { return Tile{ws + lo.trs[l], NTOK}; };
    auto TD = [&](int l) { return Tile{ws + lo.td[l], NTOK}; };   // delta_l [t][j]
    auto TDt = [&](int l) { return Tile{ws + lo.tdt[l], dim(l)}; };  // delta_l [j][t], times gamma_t, times u_t
    auto TDg = [&](int l) { return Tile{ws + lo.tdg[l], dim(l)}; };
    auto TDu = [&](int l) { return Tile{ws + lo.tdu[l], dim(l)}; };
    const Tile TG{ws + lo.tg, NTOK};  // -Gamma_{t,i} (r_t . x_i) [t][i]

    const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q) + unit * T * d;
    const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(a.k) + unit * T * d;
    const __nv_bfloat16* vp = reinterpret_cast<const __nv_bfloat16*>(a.v) + unit * T * d;
    const float* al = a.alpha + unit * T;
    const float* et = a.eta + unit * T;
    const float* be = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    Tout* y = reinterpret_cast<Tout*>(a.y) + unit * T * d;
    float* Mw = a.M_T + unit * P;  // the fp32 state, updated in place chunk by chunk
    float* Sw = a.S_T + unit * P;

    Pipe p;
    p.area = smem_u32(sm);
    p.full = bars;
    p.empty = bars + MAX_STAGES;
    p.done = bars + 2 * MAX_STAGES;
    p.s_fail = s_fail;
    p.prod = s_prod;
    p.ndone = 0;
    p.failed = 0;

    if (tid == 0) {
        for (int i = 0; i < 2 * MAX_STAGES + 1; ++i) mbar_init(&bars[i], 1);
        *s_fail = 0;
        for (int i = 0; i < MAX_STAGES; ++i) s_prod->ncopy[i] = s_prod->nmma[i] = 0;
        s_prod->skip = a.skip_first_load;
        s_prod->area = smem_u32(sm);
        s_prod->full = bars;
        s_prod->empty = bars + MAX_STAGES;
        s_prod->done = bars + 2 * MAX_STAGES;
        s_prod->s_fail = s_fail;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    // the state: fp32 copy into M_T / S_T, and its operand tiles
    for (int l = 1; l <= L; ++l) {
        const int in = dim(l - 1), out = dim(l);
        const Tile tw = TW(l), tsl = TS(l), twt = TWt(l);
        for (int idx = tid; idx < out * in; idx += NT) {
            const int j = idx / in, x = idx - j * in;
            const long long e = woff(l) + idx;
            const float w = a.M0[unit * P + e], sv = a.S0[unit * P + e];
            if (a.M_T != a.M0) Mw[e] = w;
            if (a.S_T != a.S0) Sw[e] = sv;
            tw.p[toff(out, j, x)] = __uint_as_float(to_tf32(w));
            tsl.p[toff(out, j, x)] = __uint_as_float(to_tf32(sv));
            if (l >= 2) twt.p[toff(in, x, j)] = __uint_as_float(to_tf32(w));
        }
    }
    fence_proxy_async_global();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    p.tm = *s_tmem;
    if (tid == 0) s_prod->tm = p.tm;

    // ends an epilogue: its TMEM reads are done, its tile writes visible to the
    // bulk copies of the next products, and its use of the stages (the
    // transposes) ordered before those copies land there
    auto handoff = [&]() {
        if (lane == 0) bulk_wait_all();  // this warp's block copies have landed
        fence_proxy_async_global();
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
    };
    // the same where the block copies just sent are read only in the next chunk (the state's tiles): they
    // need only have read their shared-memory buffers, which the next products' copies reuse; the next
    // chunk's first handoff waits for them to land
    auto handoff_light = [&]() {
        if (lane == 0) bulk_wait_read();
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
    };

    for (long long t0 = 0; t0 < T && !p.failed; t0 += b) {
        const int n = (int)min((long long)b, T - t0);
        if (tid < NTOK) {
            const bool in_chunk = tid < n;
            ga[tid] = in_chunk ? 1.0f - al[t0 + tid] : 0.0f;
            ge[tid] = in_chunk ? et[t0 + tid] : 0.0f;
            gb[tid] = in_chunk ? be[t0 + tid] : 0.0f;
            gc[tid] = in_chunk ? momentum_c(c_mode, be[t0 + tid], cc, t0 + tid) : 0.0f;
            gl[tid] = 0.0f;
            ub[tid] = 0.0f;
            sA[tid] = 0.0f;
            sSg[tid] = 0.0f;
        }
        if (t0 + b < T) {  // the next chunk's q, k, v and gates into L2 (one 128-byte line per thread)
            const long long nb = min((long long)b, T - t0 - b);
            const long long qkv_lines = (nb * d * 2 + 127) / 128, g_lines = (nb * 4 + 127) / 128;
            const long long tot = 3 * qkv_lines + 3 * g_lines;
            for (long long i = tid; i < tot; i += NT) {
                const char* base;
                long long li = i;
                if (li < 3 * qkv_lines) {
                    const int which = (int)(li / qkv_lines);
                    li -= which * qkv_lines;
                    base = reinterpret_cast<const char*>((which == 0 ? qp : which == 1 ? kp : vp) + (t0 + b) * d);
                } else {
                    li -= 3 * qkv_lines;
                    const int which = (int)(li / g_lines);
                    li -= which * g_lines;
                    base = reinterpret_cast<const char*>((which == 0 ? al : which == 1 ? et : be) + t0 + b);
                }
                asm volatile("prefetch.global.L2 [%0];" ::"l"(base + li * 128));
            }
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
        const __nv_bfloat16* kc = kp + t0 * d;  // this chunk's keys and queries [t][x]
        const __nv_bfloat16* qc = qp + t0 * d;
        // their operand tiles (zero past the chunk's end), in 32 x 32 blocks: k as [t][x] and [x][t],
        // q plain, times A_t and times -sigma_t (bf16 values are exact in tf32)
        {
            const int nxb = d / 32;
            for (int blk = warp; blk < 4 * nxb; blk += NT / 32) {
                const bool isq = blk >= 2 * nxb;
                const int bi = isq ? blk - 2 * nxb : blk;
                const int tb = (bi / nxb) * 32, xb = (bi % nxb) * 32;
                const __nv_bfloat16* src = isq ? qc : kc;
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    v[i] = tb + i < n ? __bfloat162float(src[(size_t)(tb + i) * d + xb + lane]) : 0.0f;
                if (!isq) {
                    put_block(sg, TK, tb, xb, v, lane);
                    float u[32];
                    transpose32(tbuf, v, u, lane);
                    put_block(sg, TKt, xb, tb, u, lane);
                } else {
                    put_block(sg, TQ, tb, xb, v, lane);
                    float sc[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) sc[i] = v[i] * sA[tb + i];
                    put_block(sg, TQa, tb, xb, sc, lane);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sc[i] = -v[i] * sSg[tb + i];
                    put_block(sg, TQs, tb, xb, sc, lane);
                }
            }
        }
        handoff();

        // keys' forward at the chunk-start weights: z_l = W_l x_{l-1}, x_l = silu(z_l)
        for (int l = 1; l < L; ++l) {
            const int in = dim(l - 1);
            const int mt = (h + 127) / 128;
            Seg s[1] = {seg(TW(l), 0, l == 1 ? TK : TX(l - 1), 0, in, 0, 1)};
            gemm(p, s, 1, mt, NTOK, tid);
            float* z = Zp(l);
            const Tile tx = TX(l), txt = TXt(l);
            epi32(p, 0, mt, NTOK, h, warp, [&](int jb, int tb, const float (&v)[32]) {
                float xv[32], xu[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {  // lane = feature j = jb + lane, c = token tb + c
                    const int t = tb + c;
                    xv[c] = t < n ? silu_e(v[c]) : 0.0f;
                    if (t < n) z[(size_t)t * h + jb + lane] = v[c];
                }
                put_block(sg, tx, tb, jb, xv, lane);  // x_l [t][j]
                transpose32(tbuf, xv, xu, lane);
                put_block(sg, txt, jb, tb, xu, lane);  // x_l [j][t]
            });
            handoff();
        }
        // e = 2 (W_L x_{L-1} - v), clipped for the Huber loss: delta_L
        {
            Seg s[1] = {seg(TW(L), 0, TX(L - 1), 0, h, 0, 1)};
            gemm(p, s, 1, 1, NTOK, tid);
            const __nv_bfloat16* vc = vp + t0 * d;
            const Tile td = TD(L), tdt = TDt(L), tdg = TDg(L), tdu = TDu(L);
            epi32(p, 0, 1, NTOK, d, warp, [&](int ob, int tb, const float (&v)[32]) {
                float e[32], eu_[32];
                const int o = ob + lane;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int t = tb + c;
                    e[c] = t < n ? nm_clip_err(2.0f * (v[c] - __bfloat162float(vc[(size_t)t * d + o])), a.e_clip) : 0.0f;
                }
                put_block(sg, td, tb, ob, e, lane);  // e [t][o]
                transpose32(tbuf, e, eu_, lane);      // eu_[r] = e of output ob + r at token tb + lane
                put_block(sg, tdt, ob, tb, eu_, lane);
                const float g = gl[tb + lane], u = ub[tb + lane];
                float sc[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) sc[r] = eu_[r] * g;
                put_block(sg, tdg, ob, tb, sc, lane);
#pragma unroll
                for (int r = 0; r < 32; ++r) sc[r] = eu_[r] * u;
                put_block(sg, tdu, ob, tb, sc, lane);
            });
            handoff();
        }
        // backward: delta_l = (W_{l+1}^T delta_{l+1}) (.) silu'(z_l)
        for (int l = L - 1; l >= 1; --l) {
            const int up = dim(l + 1);
            const int mt = (h + 127) / 128;
            Seg s[1] = {seg(TWt(l + 1), 0, TD(l + 1), 0, up, 0, 1)};
            gemm(p, s, 1, mt, NTOK, tid);
            const float* z = Zp(l);
            const Tile td = TD(l), tdt = TDt(l), tdg = TDg(l), tdu = TDu(l);
            epi32(p, 0, mt, NTOK, h, warp, [&](int jb, int tb, const float (&v)[32]) {
                float dl[32], du_[32];
                const int j = jb + lane;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int t = tb + c;
                    dl[c] = t < n ? v[c] * dsilu_e(z[(size_t)t * h + j]) : 0.0f;
                }
                put_block(sg, td, tb, jb, dl, lane);  // delta_l [t][j]
                transpose32(tbuf, dl, du_, lane);
                put_block(sg, tdt, jb, tb, du_, lane);
                const float g = gl[tb + lane], u = ub[tb + lane];
                float sc[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) sc[r] = du_[r] * g;
                put_block(sg, tdg, jb, tb, sc, lane);
#pragma unroll
                for (int r = 0; r < 32; ++r) sc[r] = du_[r] * u;
                put_block(sg, tdu, jb, tb, sc, lane);
            });
            handoff();
        }
        // surprise_t = sqrt(sum_l ||delta_{l,t}||^2 ||x_{l-1,t}||^2): one warp per token, from the
        // [t][.] tiles (the order of a row's values inside a block does not matter to a sum)
        if (a.surprise && !p.failed) {
            for (int t = warp; t < n; t += NT / 32) {
                float tot = 0.f;
                for (int l = 1; l <= L; ++l) {
                    const int in = dim(l - 1), out = dim(l);
                    float x2 = 0.f, d2 = 0.f;
                    for (int x = lane; x < in; x += 32) {
                        const float xv = l == 1 ? __bfloat162float(kc[(size_t)t * d + x])
                                                : TX(l - 1).p[(size_t)(x >> 5) * NTOK * 32 + (size_t)t * 32 + (x & 31)];
                        x2 = fmaf(xv, xv, x2);
                    }
                    const float* dl = TD(l).p;
                    for (int o = lane; o < out; o += 32) {
                        const float dv = dl[(size_t)(o >> 5) * NTOK * 32 + (size_t)t * 32 + (o & 31)];
                        d2 = fmaf(dv, dv, d2);
                    }
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
        // retrieval, layer by layer (r_0 = q)
        for (int l = 1; l <= L && !p.failed; ++l) {
            const int in = dim(l - 1), out = dim(l);
            const Tile xin = l == 1 ? TK : TX(l - 1);
            // -G[t][i] = -Gamma_{t,i} (r_t . x_{l-1,i}) for i <= t, from P^T[i][t] = x_{l-1,i} . r_t
            {
                Seg s[1] = {seg(xin, 0, l == 1 ? TQ : TR(l - 1), 0, in, 0, 1)};
                gemm(p, s, 1, 1, NTOK, tid);
                epi32(p, 0, 1, NTOK, NTOK, warp, [&](int ib, int tb, const float (&v)[32]) {
                    float g[32];
                    const int i = ib + lane;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int t = tb + c;
                        g[c] = (i <= t && t < n) ? -sG[t * GSTR + i] * v[c] : 0.0f;
                    }
                    put_block(sg, TG, tb, ib, g, lane);  // -G [t][i]
                });
                handoff();
            }
            // pre_l^T[j][t] = (W_l (A_t r_t))_j + (S_l (-sigma_t r_t))_j + sum_i delta_{l,i,j} (-G[t][i])
            {
                const int mt = (out + 127) / 128;
                Seg s[3] = {seg(TW(l), 0, l == 1 ? TQa : TRa(l - 1), 0, in, 0, 1),
                            seg(TS(l), 0, l == 1 ? TQs : TRs(l - 1), 0, in, 0, 0),
                            seg(TDt(l), 0, TG, 0, NTOK, 0, 0)};
                gemm(p, s, 3, mt, NTOK, tid);
                const Tile tr = l < L ? TR(l) : TK, tra = l < L ? TRa(l) : TK, trs = l < L ? TRs(l) : TK;
                epi32(p, 0, mt, NTOK, out, warp, [&](int jb, int tb, const float (&v)[32]) {
                    const int j = jb + lane;
                    if (l < L) {
                        float r[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c) r[c] = tb + c < n ? silu_e(v[c]) : 0.0f;
                        put_block(sg, tr, tb, jb, r, lane);  // r_l [t][j]
                        float sc[32];
#pragma unroll
                        for (int c = 0; c < 32; ++c) sc[c] = r[c] * sA[tb + c];
                        put_block(sg, tra, tb, jb, sc, lane);
#pragma unroll
                        for (int c = 0; c < 32; ++c) sc[c] = -r[c] * sSg[tb + c];
                        put_block(sg, trs, tb, jb, sc, lane);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const int t = tb + c;
                            if (t < n) {
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
        // W_l <- A_n W_l - sigma_n S_l - sum_i gamma_i delta_{l,i} x_{l-1,i}^T, S_l <- B_n S_l + sum_i u_i (same),
        // written as fp32 and as the next chunk's operand tiles
        const float An = sA[n - 1], Bn = sB[n - 1], sn = sSg[n - 1];
        for (int l = 1; l <= L && !p.failed; ++l) {
            const int in = dim(l - 1), out = dim(l);
            float* Wl = Mw + woff(l);
            float* Sl = Sw + woff(l);
            const Tile tw = TW(l), tsl = TS(l), twt = TWt(l);
            const Tile xt = l == 1 ? TKt : TXt(l - 1);
            for (int m0 = 0; m0 < out; m0 += 128) {
                for (int x0 = 0; x0 < in; x0 += 256) {
                    const int N = min(256, in - x0);
                    Seg s[2] = {seg(TDg(l), m0, xt, x0, NTOK, 0, 1), seg(TDu(l), m0, xt, x0, NTOK, 256, 1)};
                    gemm(p, s, 2, 1, N, tid);
                    epi32x2(p, 0, 256, N, out - m0, warp, [&](int jb, int cb, const float (&gw)[32], const float (&gs)[32]) {
                        // column-mapped: lane = input x = x0 + cb + lane, r = output row m0 + jb + r
                        float gwu[32], gsu[32];
                        transpose32(tbuf, gw, gwu, lane);
                        transpose32(tbuf, gs, gsu, lane);
                        const int x = x0 + cb + lane, rb = m0 + jb;
                        const uint32_t bw = blk_begin(sg, lane), bs = blk_begin(sg, lane);
#pragma unroll
                        for (int r0 = 0; r0 < 32; r0 += 16) {  // the loads of 16 rows issued before any store
                            float w[16], sv[16];
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                const size_t e = (size_t)(rb + r0 + r) * in + x;
                                w[r] = Wl[e];
                                sv[r] = Sl[e];
                            }
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                const size_t e = (size_t)(rb + r0 + r) * in + x;
                                const float wnew = An * w[r] - sn * sv[r] - gwu[r0 + r];
                                const float snew = Bn * sv[r] + gsu[r0 + r];
                                Wl[e] = wnew;
                                Sl[e] = snew;
                                blk_put(bw, r0 + r, wnew, lane);
                                blk_put(bs, r0 + r, snew, lane);
                                tbuf[(r0 + r) * 33 + lane] = wnew;
                            }
                        }
                        blk_end(bw, tw, rb, x0 + cb, lane);  // W_l, S_l [o][i]
                        blk_end(bs, tsl, rb, x0 + cb, lane);
                        if (l >= 2) {  // W_l [x][o]: back to one row per lane, then one 128-byte row per store
                            __syncwarp();
                            float wv[32];
#pragma unroll
                            for (int c = 0; c < 32; ++c) wv[c] = tbuf[lane * 33 + c];
                            __syncwarp();
                            put_block(sg, twt, x0 + cb, rb, wv, lane);
                        }
                        __syncwarp();
                    });
                    handoff_light();
                }
            }
        }
    }
    if (p.failed) {
        if (tid == 0) {
            if (a.status) atomicExch(a.status, NM_ERR_DEVICE_TIMEOUT);
            // let copies and products still in flight land before the CTA leaves
            for (int st = 0; st < MAX_STAGES; ++st) {
                const uint32_t nc = s_prod->ncopy[st], nm = s_prod->nmma[st];
                if (nc > nm) mbar_wait(&bars[st], nm & 1u, WAIT_NS);                      // a copy not consumed
                if (nm > 0) mbar_wait(&bars[MAX_STAGES + st], (nm - 1u) & 1u, WAIT_NS);  // the last products
            }
        }
    }
    if (lane == 0) bulk_wait_all();  // every block copy has read its buffer and landed before the CTA exits
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(p.tm, 512);
}

template <typename Tout>
cudaError_t launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    auto kern = tc_deep_kernel<Tout>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DEEP_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((long long)a.B * a.H), NT, DEEP_SMEM_BYTES, s>>>(a, c.d, c.hidden, nm_layers(c), c.chunk,
                                                                       c.c_mode);
    return cudaGetLastError();
}

}  // namespace

bool nm_tc_deep_supports(const nm_config& c) {
    return c.kind == NM_MLP2 && nm_layers(c) > 2 && c.in_dtype == NM_BF16 && (c.d == 64 || c.d == 128) &&
           c.hidden >= 64 && c.hidden <= 512 && c.hidden % 64 == 0 && c.chunk >= 1 && c.chunk <= NTOK;
}

size_t nm_tc_deep_scratch_bytes(const nm_config& c, int B, int H) {
    return sizeof(float) * deep_layout(c.d, c.hidden, nm_layers(c)).total * (size_t)B * (size_t)H;
}

cudaError_t nm_tc_deep_launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    if (!a.scratch || a.scratch_bytes < nm_tc_deep_scratch_bytes(c, a.B, a.H)) return cudaErrorInvalidValue;
    return c.out_dtype == NM_BF16 ? launch<__nv_bfloat16>(c, a, s) : launch<float>(c, a, s);
}
