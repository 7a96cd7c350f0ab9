// tcgen05 tensor-core kernel for the 2-layer SiLU MLP memory
// M(x) = W2 silu(W1 x), d = 64, hidden h = 128 * NC, chunk b = 64.
//
// Method ("Titans: Imparare a Memorizzare al Tempo di Test", sections
// "Meccanismo di Aggiornamento della Memoria", "Meccanismo di Dimenticanza",
// "Funzione Obiettivo", "Addestramento Parallelizzato"; the 0h-n0.github.io
// explainer, "ニューラル長期メモリモジュール" and "メモリ読み出し"): inside a chunk
// every token takes its gradient at the chunk-start weights W0, and with
// a_t = 1 - alpha_t,
//   A_t = prod_{j<=t} a_j,  B_t = prod_{j<=t} beta_j,
//   sigma_t = a_t sigma_{t-1} + eta_t B_t,
//   Gamma_{t,i} = a_t Gamma_{t-1,i} + eta_t u_{t,i},  u_{t,i} = c_i prod_{l=i+1..t} beta_l,
// the weights after token t are W_t = A_t W0 - sigma_t S0 - sum_{i<=t} Gamma_{t,i} g_i
// and the momentum S_t = B_t S0 + sum_{i<=t} u_{t,i} g_i.  For this memory
//   z_i = W1 k_i, a(k_i) = silu(z_i), e_i = 2 (W2 a(k_i) - v_i),
//   delta_i = (W2^T e_i) (.) silu'(z_i),  g_i = (delta_i k_i^T, e_i a(k_i)^T),
// so retrieval after token t is
//   h_t = A_t W1 q_t - sigma_t S1 q_t - sum_i Gamma_{t,i} (k_i . q_t) delta_i,
//   y_t = A_t W2 a_t - sigma_t S2 a_t - sum_i Gamma_{t,i} (a(k_i) . a_t) e_i,  a_t = silu(h_t),
// and the chunk-end state is W_end = A_n W0 - sigma_n S0 - sum_i gamma_i g_i,
// S_end = B_n S0 + sum_i u_i g_i with gamma_i = Gamma_{n-1,i}, u_i = u_{n-1,i}.
//
// Work split: a cluster of NC CTAs per (batch, head) unit, CTA r owning the
// hidden units j in [128 r, 128 r + 128): its rows of W1 and S1 and its
// columns of W2 and S2 (kept transposed, [j][o]).  Everything indexed by j is
// local; the two sums over j are exchanged through distributed shared memory:
//   * the key forward W2 a(k_i): each CTA adds its slice's partial sum to the
//     peer's (all-reduce), then both form e_i;
//   * the retrieval y_t: each CTA's partial (its slice of W2 a_t, S2 a_t and
//     of (a(k_i) . a_t)) is reduced onto the CTA that owns those output
//     columns, which writes y.
//
// Per CTA (512 threads, each epilogue thread owning 16 columns of an
// accumulator row; thread 0 issues TMA and MMA):
//   TMEM, 128 lanes x 512 fp32 columns; lane = j for M=128 products, row t at
//   lane (t % 16) + 32 (t / 16) for M=64 products:
//     0..63 W1 [j][x], 64..127 S1 [j][x], 128..191 W2^T [j][o], 192..255 S2^T
//     (the fp32 state, resident for the whole sequence), 256..511 per-chunk
//     accumulators reused phase by phase (see COL_* below).
//   SMEM: the chunk's Q|K tile and V tile (TMA, 128-byte swizzle), bf16
//     copies of the state as tensor-core operands, the chunk's intermediates
//     as bf16 operand tiles, Gamma in fp32, exchange buffers for the peer.
// Per chunk: G1 W1 [q|k], S1 q, Q K^T -> Z, a(k), P1 = Gamma (.) QK^T ->
// G2 partial yhat -> exchange -> E -> G3 W2^T e -> delta -> G4 state update
// and sum_i P1 delta_i -> h, a_t -> G5 W2 a_t | S2 a_t, a_t . a(k_i) -> P2 ->
// G6 P2 E -> y partials -> exchange -> y.  Then the new state becomes the
// next chunk's bf16 operands.
//
// Precision of the gradient path.  Each operand of the products that build
// the gradient and the state update (the chunk-start W1, W2 in the key
// forward and backward, a(k), e, delta and the gamma / u scaled k and e) is
// taken as a hi/lo pair of bf16 tiles, x = hi + lo with lo = bf16(x -
// bf16(x)), and a product A B becomes A_hi B_hi + A_lo B_hi + A_hi B_lo
// (three tensor-core products into one fp32 accumulator; q and k are exact in
// bf16 and need no lo half).  The key forward W2 a(k) splits W2 only: the
// a(k) lo term changes the state by two orders of magnitude less than the
// others in the emulation.  The memory's own dynamics amplify rounding in
// this path: with single bf16 operands, runs of a few thousand tokens leave
// the fp32 tolerance of the state far behind (an fp64 emulation of the
// rounding points put every one of these six operands at about the same
// share).  Retrieval-only products (S1 q, W2 a_t, S2 a_t, the Gamma-weighted
// inner products) keep single bf16 operands.  The lo tiles reuse regions
// that are dead while they live: W1 lo in the a(k) tile (end of the previous
// chunk .. G1), W2 lo and then delta lo in the S1 copy (dead after G1), a(k)
// lo in the q|k tile and e lo in the v tile (the next chunk's tiles load
// after G4), -gamma e lo and u e lo in the W1 copy (dead after G1, rewritten
// after G4), and -gamma k lo, u k lo in their own tiles (room made by
// keeping Gamma in bf16: it only enters the bf16 P tiles).  The W2 / S2
// updates are issued right behind G3 and run while E3 does, so that only the
// W1 / S1 updates stand between delta and retrieval.
#include <cuda_bf16.h>

#include "nm_internal.h"
#include "tc_common.cuh"

namespace {

using namespace tc;

constexpr int D = 64;         // key / value width
constexpr int HS = 128;       // hidden units per CTA
constexpr int BC = 64;        // chunk size
constexpr int CW_DEFAULT = 16;  // columns per thread in the epilogues (512 threads)
constexpr uint32_t T64 = 64 * 128;    // [64 rows][64 bf16] swizzled tile
constexpr uint32_t T128 = 128 * 128;  // [128 rows][64 bf16]

constexpr uint32_t OFF_QK = 0;                // [128][64]: q rows 0..63, k rows 64..127 (TMA)
constexpr uint32_t OFF_V = OFF_QK + T128;     // [64 t][64 o] (TMA)
constexpr uint32_t OFF_W1 = OFF_V + T64;      // [128 j][64 x]  bf16 copy of W1 (this CTA's rows)
constexpr uint32_t OFF_S1 = OFF_W1 + T128;    // [128 j][64 x]
constexpr uint32_t OFF_W2 = OFF_S1 + T128;    // [128 j][64 o]  W2 transposed
constexpr uint32_t OFF_S2 = OFF_W2 + T128;    // [128 j][64 o]  (follows W2: one N=128 operand)
constexpr uint32_t OFF_AK = OFF_S2 + T128;    // [128 j][64 t]  a(k_t)
constexpr uint32_t OFF_DT = OFF_AK + T128;    // [128 j][64 t]  delta_t, later a_t (retrieval)
constexpr uint32_t OFF_KG = OFF_DT + T128;    // [64 t][64 x]   -gamma_t k_t
constexpr uint32_t OFF_KU = OFF_KG + T64;     // [64 t][64 x]   u_t k_t
constexpr uint32_t OFF_E = OFF_KU + T64;      // [64 t][64 o]   e_t
constexpr uint32_t OFF_EG = OFF_E + T64;      // -gamma_t e_t
constexpr uint32_t OFF_EU = OFF_EG + T64;     // u_t e_t
constexpr uint32_t OFF_P = OFF_EU + T64;      // [64 t][64 i]   Gamma (.) inner products
constexpr uint32_t OFF_KLO = OFF_P + T64;     // [2][64 t][64 x] lo halves of -gamma_t k_t, u_t k_t
constexpr int XS = 72;                        // bf16 row stride of the key-forward exchange
constexpr int RB = 40;                        // bf16 row stride of the y exchange
constexpr uint32_t OFF_YX = OFF_KLO + 2 * T64;  // bf16 [64][XS] the peer's partial key forward (E2);
                                                // then the u e lo tile [64 t][64 o] (E3 .. G4)
constexpr int GST = 72;                         // bf16 row stride of Gamma
constexpr uint32_t OFF_GM = OFF_YX + 64 * XS * 2;       // bf16 Gamma [2 stages][64][GST]
constexpr uint32_t OFF_YR = OFF_GM + 2 * 64 * GST * 2;  // bf16 [64][RB] the peer's partial y (own columns)
// lo halves living in regions that are dead meanwhile (see the file header)
constexpr uint32_t OFF_W1LO = OFF_AK;   // [128 j][64 x]  W1 lo: E6 of the previous chunk .. G1
constexpr uint32_t OFF_W2LO = OFF_S1;   // [128 j][64 o]  W2 lo (transposed): E1 .. G3
constexpr uint32_t OFF_AKLO = OFF_QK;   // [128 j][64 t]  a(k) lo: E1 .. G4
constexpr uint32_t OFF_ELO = OFF_V;     // [64 t][64 o]   e lo: E2 .. G3
constexpr uint32_t OFF_EGLO = OFF_W1;   // [64 t][64 o]   -gamma e lo: E2 .. G4
constexpr uint32_t OFF_EULO = OFF_W1 + T64;  // [64 t][64 o]   u e lo: E2 .. G4
constexpr uint32_t OFF_DTLO = OFF_S1;   // [128 j][64 t]  delta lo: E3 .. G4
constexpr uint32_t OFF_F = OFF_YR + 64 * RB * 2;        // gates [2][4][64]; scan [2][A, B, sigma, gamma, u][64]
constexpr uint32_t N_F = 2 * 4 * BC + 2 * 5 * BC;
constexpr uint32_t OFF_SP = OFF_F + 4 * N_F;  // surprise partials (fp32 [64] rows): ||a(k)||^2 [4 quadrants],
constexpr uint32_t N_SP = 18 * BC;             // ||delta||^2 [4 quadrants], ||e||^2 [4 column groups],
                                               // ||k||^2 [4 column groups], the peer's (||a||^2, ||delta||^2)
constexpr uint32_t OFF_BAR = OFF_SP + 4 * N_SP;
constexpr uint32_t SMEM_USED = OFF_BAR + 64;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for the 1024-byte alignment
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(OFF_S2 == OFF_W2 + T128, "W2 and S2 copies form one N=128 operand");
static_assert(OFF_EU == OFF_EG + T64 && OFF_EULO == OFF_EGLO + T64 && OFF_KU == OFF_KG + T64, "paired update operands");
static_assert(OFF_YX % 1024 == 0, "exchange buffer alignment");
// bytes the peer sends per chunk: its whole partial key forward [64 t][64 o], and
// its partial y of this CTA's 32 output columns
constexpr uint32_t XCH_KEY_BYTES = 64 * 64 * 2;
constexpr uint32_t XCH_Y_BYTES = 64 * 32 * 2;
static_assert(OFF_GM % 16 == 0 && (GST * 2) % 16 == 0, "Gamma rows are read 16 bytes at a time");

// TMEM columns
constexpr uint32_t COL_W1 = 0, COL_S1 = 64, COL_W2 = 128, COL_S2 = 192;
static_assert(COL_S1 == COL_W1 + 64 && COL_S2 == COL_W2 + 64, "paired update accumulators");
constexpr uint32_t COL_XA = 256;  // G1: [j][t] W1 q_t (256..319), W1 k_t = z_t (320..383)
constexpr uint32_t COL_Z = 320;
constexpr uint32_t COL_XB = 384;  // G1: [j][t] S1 q_t
constexpr uint32_t COL_QK = 448;  // G1: lanes 0..63 [t][i] q_t . k_i
constexpr uint32_t COL_YH = 320;  // G2: M=64 [t][o] partial W2 a(k_t)
constexpr uint32_t COL_XD = 320;  // G3: [j][t] W2^T e_t
constexpr uint32_t COL_R1 = 320;  // G4: [j][t] sum_i P1[t][i] delta_i
constexpr uint32_t COL_YW = 256;  // G5: M=64 [t][o] W2 a_t (256..319), S2 a_t (320..383)
constexpr uint32_t COL_AA = 384;  // G5: M=64 [t][i] a_t . a(k_i)
constexpr uint32_t COL_PE = 448;  // G6: M=64 [t][o] sum_i P2[t][i] e_i

constexpr uint32_t ID_XA = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t ID_M128N64 = idesc_bf16_f32(128, 64, false, false);
// the W | S updates as one N = 128 product over two adjacent B tiles (T64 apart)
constexpr uint32_t ID_UPD2 = idesc_bf16_f32(128, 128, false, true);
constexpr uint32_t ID_M64N64_TT = idesc_bf16_f32(64, 64, true, true);
constexpr uint32_t ID_M64N192_TT = idesc_bf16_f32(64, 192, true, true);
static_assert(OFF_AK == OFF_S2 + T128 && COL_AA == COL_YW + 128, "N=192 operand and accumulator");
constexpr uint32_t ID_M64N64_BT = idesc_bf16_f32(64, 64, false, true);
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s

// Shared-memory descriptors (the sw128_desc fields) for K-major operands and
// for MN-major operands whose 64-element blocks along M/N are `lbo` bytes
// apart.  The start-address field holds bits 4..17 of the shared address; the
// mask matters: in a cluster launch the shared::cta addresses of this CTA
// carry bits above bit 17, which would otherwise spill into the
// leading-byte-offset field.  Tiles lie below 228 KB of the window, so a
// k-step adds to the descriptor directly without carrying out of the field:
// +2 for 32 bytes (K-major), +128 for 2048 bytes (16 rows, MN-major).
constexpr uint64_t desc_hi(uint32_t lbo) {
    return (static_cast<uint64_t>(lbo >> 4) << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}
__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return desc_hi(16) | ((a >> 4) & 0x3FFFu); }
__device__ __forceinline__ uint64_t mdesc(uint32_t a, uint32_t lbo) { return desc_hi(lbo) | ((a >> 4) & 0x3FFFu); }
constexpr uint64_t KS_K = 2, KS_M = 128;

__device__ __forceinline__ float silu_f(float z) { return z * sigmoid_f(z); }

__device__ __forceinline__ float momentum_c(int mode, float beta, const float* c, long long i) {
    if (mode == NM_C_ONE_MINUS_BETA) return 1.0f - beta;
    if (mode == NM_C_PER_TOKEN) return c[i];
    return 1.0f;
}

// W (16 or 32) bf16 of row r, columns c0..c0+W-1, of a swizzled tile, as floats.
template <int W>
__device__ __forceinline__ void get_row(const unsigned char* tile, uint32_t rows, uint32_t r, uint32_t c0, float* v) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
        const uint4 w = ld_shared_v4(base + sw128_offset(r, c0 + 8 * q, rows));
        v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
        v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
        v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
        v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
    }
}

// W bf16 of a plain row-major row (16-byte aligned), as floats.
template <int W>
__device__ __forceinline__ void get_plain(const __nv_bfloat16* p, float* v) {
    const uint32_t base = smem_u32(p);
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
        const uint4 w = ld_shared_v4(base + 16 * q);
        v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
        v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
        v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
        v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
    }
}

// W consecutive outputs of one row of y.
template <int W>
__device__ __forceinline__ void store_y(__nv_bfloat16* p, const float* v) {
#pragma unroll
    for (int q = 0; q < W / 8; ++q)
        reinterpret_cast<uint4*>(p)[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                                                    pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
}
template <int W>
__device__ __forceinline__ void store_y(float* p, const float* v) {
#pragma unroll
    for (int q = 0; q < W / 4; ++q)
        reinterpret_cast<float4*>(p)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// W values as bf16 into a peer's shared memory (st.async, 16 bytes at a time,
// counted on the peer's mbarrier `bar`) / back to floats.
template <int W>
__device__ __forceinline__ void push_bf16(uint32_t dst, const float* v, uint32_t bar) {
#pragma unroll
    for (int q = 0; q < W / 8; ++q)
        st_async_v4(dst + 16 * q, pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                    pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]), bar);
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
template <int W>
__device__ __forceinline__ void pull_bf16(uint32_t src, float* v) {
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
        const uint4 w = ld_shared_v4(src + 16 * q);
        v[8 * q + 0] = bf16_lo(w.x); v[8 * q + 1] = bf16_hi(w.x);
        v[8 * q + 2] = bf16_lo(w.y); v[8 * q + 3] = bf16_hi(w.y);
        v[8 * q + 4] = bf16_lo(w.z); v[8 * q + 5] = bf16_hi(w.z);
        v[8 * q + 6] = bf16_lo(w.w); v[8 * q + 7] = bf16_hi(w.w);
    }
}

// Sums v[0..15] (one value per lane per column) over the warp's 32 lanes by
// halving exchanges; afterwards lane l holds the total of column
// 8 b4 + 4 b3 + 2 b2 + b1 (b_i = bit i of l), which lanes l and l ^ 1 share.
__device__ __forceinline__ float warp_colsum16(const float (&v)[16], int lane) {
    float w8[8], w4[4], w2[2];
    const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4, h2 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w8[i] = (h16 ? v[8 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, h16 ? v[i] : v[8 + i], 16);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w4[i] = (h8 ? w8[4 + i] : w8[i]) + __shfl_xor_sync(0xffffffffu, h8 ? w8[i] : w8[4 + i], 8);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        w2[i] = (h4 ? w4[2 + i] : w4[i]) + __shfl_xor_sync(0xffffffffu, h4 ? w4[i] : w4[2 + i], 4);
    float w1 = (h2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, h2 ? w2[0] : w2[1], 2);
    return w1 + __shfl_xor_sync(0xffffffffu, w1, 1);
}
__device__ __forceinline__ int colsum16_column(int lane) {
    return 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
}

// SURP: write the surprise (a.surprise); HUB: the Huber loss clips e.  Compiled
// variants, so that the plain forward carries neither.
template <int NC, int CW, typename Tout, bool SURP, bool HUB>
__global__ void __launch_bounds__(128 * (64 / CW), 1)
    tc_mlp_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, nm_args a, int c_mode) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* gates = reinterpret_cast<float*>(sm + OFF_F);  // [2 stages][a, eta, beta, c][64]
    float* scan_out = gates + 2 * 4 * BC;                 // [2 stages][A, B, sigma, gamma, u][64]
    __nv_bfloat16* gamma_all = reinterpret_cast<__nv_bfloat16*>(sm + OFF_GM);  // [2 stages][64][GST]
    // exchange buffers: the peer's partial sums as bf16 (summed here in fp32)
    __nv_bfloat16* Yx = reinterpret_cast<__nv_bfloat16*>(sm + OFF_YX);  // [64][XS]
    __nv_bfloat16* Yr = reinterpret_cast<__nv_bfloat16*>(sm + OFF_YR);  // [64][RB]
    // 0: tiles, 1: mma; the peer's bytes (one phase per chunk each): 2 partial key forward, 3 partial y
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    // per-token surprise partial sums (written only when SURP)
    float* sp_a2 = reinterpret_cast<float*>(sm + OFF_SP);  // [4 qd][64 t] ||a(k_t)||^2 over this CTA's hidden units
    float* sp_d2 = sp_a2 + 4 * BC;                         // [4 qd][64 t] ||delta_t||^2, likewise
    float* sp_e2 = sp_d2 + 4 * BC;                         // [4 hq][64 t] ||e_t||^2 over 16 columns each
    float* sp_k2 = sp_e2 + 4 * BC;                         // [4][64 t]    ||k_t||^2 over 16 columns each
    float* sp_peer = sp_k2 + 4 * BC;                       // [2][64 t]    the peer CTA's ||a||^2, ||delta||^2
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int qd = warp & 3;   // TMEM lane quadrant of this warp
    constexpr int NQ = 64 / CW;  // column groups: threads = 128 * NQ
    const int hq = warp >> 2;    // which CW columns of a 64-column accumulator this thread reads
    const int rank = NC > 1 ? (int)cluster_ctarank() : 0;
    const long long unit = blockIdx.x / NC;
    const long long T = a.T;
    const int hid = HS * NC;
    const long long P = 2LL * hid * D;
    const int nchunks = (int)((T + BC - 1) / BC);
    const float* alpha = a.alpha + unit * T;
    const float* eta = a.eta + unit * T;
    const float* beta = a.beta + unit * T;
    const float* cc = a.c ? a.c + unit * T : nullptr;
    Tout* y = reinterpret_cast<Tout*>(a.y) + unit * T * D;
    const int jr = 32 * qd + lane;           // row of an M=128 accumulator
    const int tr = 16 * qd + lane;           // row of an M=64 accumulator (valid for lane < 16)
    const bool r64 = lane < 16;
    const int j_glob = HS * rank + jr;       // hidden unit of row jr

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
        if (NC > 1 && nchunks > 0) {  // chunk 0's bytes from the peer (the cluster barrier below precedes them)
            mbar_arrive_expect_tx(&bars[2], XCH_KEY_BYTES);
            mbar_arrive_expect_tx(&bars[3], XCH_Y_BYTES);
        }
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 0) {
        tmem_alloc(&s_tmem, 512);
        tmem_relinquish();
    }
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
            } else {  // tokens past T change nothing: a = 1, eta = 0, beta = 1, c = 0
                g[tid] = 1.0f;
                g[BC + tid] = 0.0f;
                g[2 * BC + tid] = 1.0f;
                g[3 * BC + tid] = 0.0f;
            }
        }
    };
    auto issue_tiles = [&](int chunk) {
        mbar_arrive_expect_tx(&bars[0], 3 * T64);
        const int t0 = chunk * BC;
        tma_load_3d(sm + OFF_QK, &tq, &bars[0], 0, t0, (int)unit);
        tma_load_3d(sm + OFF_QK + T64, &tk, &bars[0], 0, t0, (int)unit);
        tma_load_3d(sm + OFF_V, &tv, &bars[0], 0, t0, (int)unit);
    };

    // The scan of one chunk's gates (stage st), one chunk ahead of its use:
    // Gamma column by column (threads 128..191), gamma_i = Gamma_{n-1,i} and
    // u_i = u_{n-1,i}; A, B, sigma by thread 224.  Column i runs the
    // division-free recursion from row 0 with u = Gamma = 0 and the start
    // injected, u_t = beta_t u_{t-1} + [t = i] c_i, Gamma_{t,i} =
    // a_t Gamma_{t-1,i} + eta_t u_t: rows above the diagonal come out exactly
    // zero and no row takes a branch.  The gates of the next four tokens are
    // loaded before a group's stores (shared loads stay behind earlier
    // shared stores).
    auto scan = [&](int st) {
        const float* g = gates + st * 4 * BC;
        float* so = scan_out + st * 5 * BC;
        if (tid >= 128 && tid < 128 + BC) {
            __nv_bfloat16* Gm = gamma_all + st * 64 * GST;
            const int i = tid - 128;
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
                    Gm[t * GST + i] = __float2bfloat16_rn(G);
                }
            }
            so[3 * BC + i] = G;
            so[4 * BC + i] = u;
        } else if (tid == 224) {
            float A = 1.f, Bc = 1.f, sg = 0.f;
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
                reinterpret_cast<float4*>(so)[t4] = make_float4(oa[0], oa[1], oa[2], oa[3]);
                reinterpret_cast<float4*>(so + BC)[t4] = make_float4(ob[0], ob[1], ob[2], ob[3]);
                reinterpret_cast<float4*>(so + 2 * BC)[t4] = make_float4(os[0], os[1], os[2], os[3]);
            }
        }
    };
    load_gates(0, 0);
    __syncthreads();
    scan(0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = s_tmem;
    const uint32_t tl = tm + ((uint32_t)(32 * qd) << 16);  // this warp's lane quadrant
    // The fp32 state m (0..3: W1, S1, W2, S2) from TMEM into its bf16 operand
    // copy in shared memory, or after the last chunk into M_T / S_T.
    auto convert_state = [&](int m, bool last) {
        float w[CW];
        tmem_ld_n(tl + (m == 0 ? COL_W1 : m == 1 ? COL_S1 : m == 2 ? COL_W2 : COL_S2) + CW * hq, w);
        if (!last) {
            put_row<CW>(sm + (m == 0 ? OFF_W1 : m == 1 ? OFF_S1 : m == 2 ? OFF_W2 : OFF_S2), 128, jr, CW * hq, w);
        } else {
            float* dst = (m & 1) ? a.S_T + unit * P : a.M_T + unit * P;
            if (m < 2) {
                float* r = dst + (long long)j_glob * D + CW * hq;
#pragma unroll
                for (int q = 0; q < CW; q += 4)
                    *reinterpret_cast<float4*>(r + q) = make_float4(w[q], w[q + 1], w[q + 2], w[q + 3]);
            } else {
                float* r = dst + (long long)hid * D + j_glob;
#pragma unroll
                for (int q = 0; q < CW; ++q) r[(long long)(CW * hq + q) * hid] = w[q];
            }
        }
    };
    if (tid == 0 && nchunks > 0 && !a.skip_first_load) issue_tiles(0);  // (the test hook skips it)

    // initial state: fp32 into TMEM, bf16 operand copies into shared memory
    {
        const float* m0 = a.M0 + unit * P;
        const float* s0 = a.S0 + unit * P;
        float r[CW];
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const float* src = which ? s0 : m0;
            // W1 (or S1) row j_glob, columns 32 hf .. 32 hf + 31
            const float* w1 = src + (long long)j_glob * D + CW * hq;
#pragma unroll
            for (int q = 0; q < CW; q += 4) {
                const float4 w = *reinterpret_cast<const float4*>(w1 + q);
                r[q] = w.x; r[q + 1] = w.y; r[q + 2] = w.z; r[q + 3] = w.w;
            }
            tmem_st_n(tl + (which ? COL_S1 : COL_W1) + CW * hq, r);
            put_row<CW>(sm + (which ? OFF_S1 : OFF_W1), 128, jr, CW * hq, r);
            if (!which) put_row_lo<CW>(sm + OFF_W1LO, 128, jr, CW * hq, r);
            // W2 (or S2) transposed: [j][o] = W2[o][j_glob], o = 32 hf + q
            const float* w2 = src + (long long)hid * D + j_glob;
#pragma unroll
            for (int q = 0; q < CW; ++q) r[q] = w2[(long long)(CW * hq + q) * hid];
            tmem_st_n(tl + (which ? COL_S2 : COL_W2) + CW * hq, r);
            put_row<CW>(sm + (which ? OFF_S2 : OFF_W2), 128, jr, CW * hq, r);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    if (NC > 1) cluster_sync(); else __syncthreads();
    tc_fence_after();

    const uint32_t aQK = smem_u32(sm + OFF_QK), aW1 = smem_u32(sm + OFF_W1), aS1 = smem_u32(sm + OFF_S1);
    const uint32_t aW2 = smem_u32(sm + OFF_W2), aAK = smem_u32(sm + OFF_AK), aDT = smem_u32(sm + OFF_DT);
    const uint32_t aKG = smem_u32(sm + OFF_KG), aE = smem_u32(sm + OFF_E);
    const uint32_t aEG = smem_u32(sm + OFF_EG), aP = smem_u32(sm + OFF_P);
    const uint32_t aW1lo = smem_u32(sm + OFF_W1LO), aW2lo = smem_u32(sm + OFF_W2LO), aAKlo = smem_u32(sm + OFF_AKLO);
    const uint32_t aElo = smem_u32(sm + OFF_ELO), aEGlo = smem_u32(sm + OFF_EGLO);
    const uint32_t aDTlo = smem_u32(sm + OFF_DTLO), aKGlo = smem_u32(sm + OFF_KLO);
    const int peer = rank ^ 1;

    bool failed = false;
    uint32_t mma_phase = 0;
    // Waits (bounded) for the MMAs committed by thread 0; uniform over the CTA.
    auto mma_wait = [&](bool committed) {
        bool ok = true;
        if (committed) {
            ok = mbar_wait(&bars[1], mma_phase, WAIT_NS);
            mma_phase ^= 1u;
        }
        failed = __syncthreads_or(!ok) || failed;
        tc_fence_after();
    };
    // Every thread: this chunk's bytes from the peer on mbarrier `xb` (bounded
    // wait); then thread 0 expects the next chunk's.  No cluster barrier orders
    // the exchanges: the peer's next stores into a buffer depend on data that
    // this CTA sent after reading it (its next key-forward partial follows its
    // y sum, which needed this CTA's y partial, sent after this CTA read the
    // key-forward buffer; its next y partial follows its e, which needed this
    // CTA's next key-forward partial, sent after this CTA read the y buffer).
    // A CTA whose wait has given up sends nothing more, and the peer then gives
    // up at its next wait.
    auto receive = [&](int xb, uint32_t bytes, int c) {
        bool ok = true;
        if (!failed) ok = mbar_wait_cluster(&bars[xb], (uint32_t)(c & 1), WAIT_NS);
        failed = __syncthreads_or(!ok) || failed;
        if (tid == 0 && !failed && c + 1 < nchunks) mbar_arrive_expect_tx(&bars[xb], bytes);
    };
    auto handoff = [&]() {  // epilogue smem / TMEM writes -> tensor-core reads
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };

    float ds[CW];  // silu'(z) for this thread's row and columns, kept from E1 to E3
    for (int c = 0; c < nchunks; ++c) {
        const int stage = c & 1;
        const long long t0 = (long long)c * BC;
        const int n = (int)min((long long)BC, T - t0);
        // the gated output: this chunk's y_attn rows into L2 for the epilogue's loads
        if (a.y_attn) nm_prefetch_attn(a, (unit * T + t0) * D * (long long)sizeof(Tout), (long long)n * D * sizeof(Tout),
                                       tid, (int)blockDim.x);
        // this chunk's scan (computed during the previous chunk)
        const float* so = scan_out + stage * 5 * BC;
        const float *sA = so, *sBc = so + BC, *sSg = so + 2 * BC, *sGl = so + 3 * BC, *sU = so + 4 * BC;
        const __nv_bfloat16* Gm = gamma_all + stage * 64 * GST;
        // the next chunk's gates: warps 2-3 load them now (raw, so that nothing
        // waits for the loads until they are stored to shared memory after E2)
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

        // ---- G1 (thread 0, as soon as the tiles land): W1 [q|k], S1 q, Q K^T
        bool tiles_ok = true;
        if (tid == 0 && !failed) {
            tiles_ok = mbar_wait(&bars[0], (uint32_t)(c & 1), WAIT_NS);
            if (tiles_ok) {
                tc_fence_after();
                const uint64_t dW1 = kdesc(aW1), dS1 = kdesc(aS1), dQK = kdesc(aQK), dK = kdesc(aQK + T64);
                const uint64_t dW1lo = kdesc(aW1lo);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t acc = ks ? 1u : 0u;
                    mma_bf16(tm + COL_XA, dW1 + KS_K * ks, dQK + KS_K * ks, ID_XA, acc);
                    mma_bf16(tm + COL_Z, dW1lo + KS_K * ks, dK + KS_K * ks, ID_M128N64, 1u);  // z only
                    mma_bf16(tm + COL_XB, dS1 + KS_K * ks, dQK + KS_K * ks, ID_M128N64, acc);
                    mma_bf16(tm + COL_QK, dQK + KS_K * ks, dK + KS_K * ks, ID_M128N64, acc);
                }
                mma_commit(&bars[1]);
            }
        }
        // the tiles (waited for by thread 0) are visible to all after this
        const bool go1 = !failed && !__syncthreads_or(!tiles_ok);
        if (!go1 && !failed) failed = true;
        // -gamma_t k_t and u_t k_t as bf16 operand rows (while G1 runs)
        if (tid < 64 * NQ) {  // row t = tid % 64, columns CW * (tid / 64) ..
            const int t = tid & 63, c0 = CW * (tid >> 6);
            float kv[CW], o1[CW], o2[CW];
            const float gm = -sGl[t], uu = sU[t];
            get_row<CW>(sm + OFF_QK, 128, 64 + t, c0, kv);
#pragma unroll
            for (int q = 0; q < CW; ++q) {
                o1[q] = gm * kv[q];
                o2[q] = uu * kv[q];
            }
            if (SURP) {
                float k2 = 0.0f;
#pragma unroll
                for (int q = 0; q < CW; ++q) k2 = fmaf(kv[q], kv[q], k2);
                sp_k2[(tid >> 6) * BC + t] = k2;
            }
            put_row_hilo<CW>(sm + OFF_KG, sm + OFF_KLO, 64, t, c0, o1);
            put_row_hilo<CW>(sm + OFF_KU, sm + OFF_KLO + T64, 64, t, c0, o2);
        }
        mma_wait(go1);
        // ---- E1: a(k) and silu'(z) from z = W1 k; P1 = Gamma (.) Q K^T
        {
            float z[CW], p[CW];
            if (qd < 2) tmem_ld_n(tl + COL_Z + CW * hq, tl + COL_QK + CW * hq, z, p);
            else tmem_ld_n(tl + COL_Z + CW * hq, z);
#pragma unroll
            for (int q = 0; q < CW; ++q) {
                const float sg = sigmoid_f(z[q]);
                ds[q] = fmaf(z[q] * sg, 1.0f - sg, sg);  // silu'(z) = s + z s (1 - s)
                z[q] *= sg;
            }
            put_row_hilo<CW>(sm + OFF_AK, sm + OFF_AKLO, 128, jr, CW * hq, z);  // (q|k is dead after G1)
            {  // the chunk-start W2 (the state is rescaled only in E2) as the lo tile for G2 and G3
                float w[CW];
                tmem_ld_n(tl + COL_W2 + CW * hq, w);
                put_row_lo<CW>(sm + OFF_W2LO, 128, jr, CW * hq, w);  // the S1 copy is dead after G1
            }
            if (SURP) {  // ||a(k_t)||^2 over this quadrant's 32 hidden units, for columns t of this thread
                float sq[CW];
#pragma unroll
                for (int q = 0; q < CW; ++q) sq[q] = z[q] * z[q];
                const float tot = warp_colsum16(sq, lane);
                if (!(lane & 1)) sp_a2[qd * BC + CW * hq + colsum16_column(lane)] = tot;
            }
            if (qd < 2) {
                float gr[CW];
                get_plain<CW>(Gm + jr * GST + CW * hq, gr);
#pragma unroll
                for (int q = 0; q < CW; ++q) p[q] *= gr[q];
                put_row<CW>(sm + OFF_P, 64, jr, CW * hq, p);
            }
        }
        handoff();
        // ---- G2: partial key forward yhat[t][o] = sum_{j in slice} a(k_t)_j W2[o][j]
        const bool go2 = !failed;
        if (go2 && tid == 0) {
            const uint64_t dAK = mdesc(aAK, T128), dW2 = mdesc(aW2, T128);
            const uint64_t dW2lo = mdesc(aW2lo, T128);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                mma_bf16(tm + COL_YH, dAK + KS_M * ks, dW2 + KS_M * ks, ID_M64N64_TT, ks ? 1u : 0u);
                mma_bf16(tm + COL_YH, dAK + KS_M * ks, dW2lo + KS_M * ks, ID_M64N64_TT, 1u);
            }
            mma_commit(&bars[1]);
        }
        mma_wait(go2);
        // ---- E2: all-reduce of the key forward over the cluster, e = 2 (yhat - v)
        float ev[CW];
        {
            tmem_ld_n(tl + COL_YH + CW * hq, ev);
            if (r64) {
                if (NC > 1 && !failed) {
                    const uint32_t dst = map_to_rank(smem_u32(Yx + tr * XS + CW * hq), (uint32_t)peer);
                    push_bf16<CW>(dst, ev, map_to_rank(smem_u32(&bars[2]), (uint32_t)peer));
                }
                float vv[CW];
                get_row<CW>(sm + OFF_V, 64, tr, CW * hq, vv);
#pragma unroll
                for (int q = 0; q < CW; ++q) ev[q] = 2.0f * (ev[q] - vv[q]);
            }
        }
        // while the peer's partial sums arrive: rescale the fp32 state for this chunk,
        // W <- A_n W - sigma_n S, S <- B_n S (before G4 accumulates into it)
        {
            const float An = sA[BC - 1], Bn = sBc[BC - 1], sn = sSg[BC - 1];
            float w[CW], s[CW];
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const uint32_t cw = (pr ? COL_W2 : COL_W1) + CW * hq, cs = (pr ? COL_S2 : COL_S1) + CW * hq;
                tmem_ld_n(tl + cw, tl + cs, w, s);
#pragma unroll
                for (int q = 0; q < CW; ++q) {
                    w[q] = fmaf(An, w[q], -sn * s[q]);
                    s[q] = Bn * s[q];
                }
                tmem_st_n(tl + cw, w);
                tmem_st_n(tl + cs, s);
            }
        }
        if (NC > 1) receive(2, XCH_KEY_BYTES, c);
        if (r64) {
            if (NC > 1) {
                float px[CW];
                pull_bf16<CW>(smem_u32(Yx + tr * XS + CW * hq), px);
#pragma unroll
                for (int q = 0; q < CW; ++q) ev[q] = fmaf(2.0f, px[q], ev[q]);
            }
            if (HUB) {  // the Huber loss clips e
#pragma unroll
                for (int q = 0; q < CW; ++q) ev[q] = nm_clip_err(ev[q], a.e_clip);
            }
            if (SURP) {
                float e2 = 0.0f;
#pragma unroll
                for (int q = 0; q < CW; ++q) e2 = fmaf(ev[q], ev[q], e2);
                sp_e2[hq * BC + tr] = e2;
            }
            // (e lo lands on this thread's own elements of the v tile, read above)
            put_row_hilo<CW>(sm + OFF_E, sm + OFF_ELO, 64, tr, CW * hq, ev);
            float o1[CW];
            const float gm = -sGl[tr], uu = sU[tr];
#pragma unroll
            for (int q = 0; q < CW; ++q) o1[q] = gm * ev[q];
            put_row_hilo<CW>(sm + OFF_EG, sm + OFF_EGLO, 64, tr, CW * hq, o1);  // (the W1 copy is dead after G1)
#pragma unroll
            for (int q = 0; q < CW; ++q) o1[q] = uu * ev[q];
            put_row_hilo<CW>(sm + OFF_EU, sm + OFF_EULO, 64, tr, CW * hq, o1);
        }
        if (gi >= 0 && gi < BC && c + 1 < nchunks) {
            // tokens past T change nothing: a = 1, eta = 0, beta = 1, c = 0
            float* gn = gates + (stage ^ 1) * 4 * BC;
            gn[gi] = nxt_valid ? 1.0f - nxt_al : 1.0f;
            gn[BC + gi] = nxt_e;
            gn[2 * BC + gi] = nxt_b;
            gn[3 * BC + gi] = !nxt_valid ? 0.0f
                              : c_mode == NM_C_ONE_MINUS_BETA ? 1.0f - nxt_b
                              : c_mode == NM_C_PER_TOKEN ? nxt_c : 1.0f;
        }
        handoff();
        // ---- G3: W2^T e; then the W2 / S2 updates, which complete while E3 runs (the commit of G4
        //      covers them): W2 += (-gamma e)^T a(k), S2 += (u e)^T a(k) into the rescaled state
        const bool go3 = !failed;
        if (go3 && tid == 0) {
            const uint64_t dW2 = kdesc(aW2), dE = kdesc(aE), dW2lo = kdesc(aW2lo), dElo = kdesc(aElo);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma_bf16(tm + COL_XD, dW2 + KS_K * ks, dE + KS_K * ks, ID_M128N64, ks ? 1u : 0u);
                mma_bf16(tm + COL_XD, dW2lo + KS_K * ks, dE + KS_K * ks, ID_M128N64, 1u);
                mma_bf16(tm + COL_XD, dW2 + KS_K * ks, dElo + KS_K * ks, ID_M128N64, 1u);
            }
            mma_commit(&bars[1]);
            // [W2^T | S2^T] += a(k) [-gamma e | u e]: hi x hi, lo x hi, hi x lo
            const uint64_t dAK = kdesc(aAK), dAKlo = kdesc(aAKlo);
            const uint64_t dEGU = mdesc(aEG, T64), dEGUlo = mdesc(aEGlo, T64);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma_bf16(tm + COL_W2, dAK + KS_K * ks, dEGU + KS_M * ks, ID_UPD2, 1u);
                mma_bf16(tm + COL_W2, dAKlo + KS_K * ks, dEGU + KS_M * ks, ID_UPD2, 1u);
                mma_bf16(tm + COL_W2, dAK + KS_K * ks, dEGUlo + KS_M * ks, ID_UPD2, 1u);
            }
        }
        mma_wait(go3);
        // ---- E3: delta = (W2^T e) (.) silu'(z)
        {
            float xd[CW];
            tmem_ld_n(tl + COL_XD + CW * hq, xd);
#pragma unroll
            for (int q = 0; q < CW; ++q) xd[q] *= ds[q];
            put_row_hilo<CW>(sm + OFF_DT, sm + OFF_DTLO, 128, jr, CW * hq, xd);  // (the S1 copy is dead after G1)
            if (SURP) {  // ||delta_t||^2 over this quadrant's 32 hidden units
                float sq[CW];
#pragma unroll
                for (int q = 0; q < CW; ++q) sq[q] = xd[q] * xd[q];
                const float tot = warp_colsum16(sq, lane);
                if (!(lane & 1)) sp_d2[qd * BC + CW * hq + colsum16_column(lane)] = tot;
            }
        }
        handoff();
        // ---- G4: state update and sum_i P1[t][i] delta_i
        const bool go4 = !failed;
        if (go4 && tid == 0) {
            const uint64_t dDT = kdesc(aDT), dP = kdesc(aP);
            const uint64_t dKGU = mdesc(aKG, T64), dDTlo = kdesc(aDTlo), dKGUlo = mdesc(aKGlo, T64);
            // R1 and the W1 / S1 updates (E4 overwrites delta, which they read, with a_t); this
            // commit also covers the W2 / S2 updates issued behind G3
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                mma_bf16(tm + COL_R1, dDT + KS_K * ks, dP + KS_K * ks, ID_M128N64, ks ? 1u : 0u);
                // [W1 | S1] += delta [-gamma k | u k]: hi x hi, lo x hi, hi x lo
                mma_bf16(tm + COL_W1, dDT + KS_K * ks, dKGU + KS_M * ks, ID_UPD2, 1u);
                mma_bf16(tm + COL_W1, dDTlo + KS_K * ks, dKGU + KS_M * ks, ID_UPD2, 1u);
                mma_bf16(tm + COL_W1, dDT + KS_K * ks, dKGUlo + KS_M * ks, ID_UPD2, 1u);
            }
            mma_commit(&bars[1]);
        }
        // while G4 runs: the next chunk's scan (its gates were stored in E2)
        if (c + 1 < nchunks) scan(stage ^ 1);
        mma_wait(go4);
        // every product reading the q|k tile (a(k) lo) and the v tile (e lo) has completed: the next
        // chunk's tiles start loading
        if (tid == 0 && !failed && c + 1 < nchunks) issue_tiles(c + 1);
        // ---- E4: h_t = A_t W1 q_t - sigma_t S1 q_t - sum_i P1[t][i] delta_i, a_t = silu(h_t)
        {
            float xa[CW], xb[CW], r1[CW];
            tmem_ld_n(tl + COL_XA + CW * hq, tl + COL_XB + CW * hq, tl + COL_R1 + CW * hq, xa, xb, r1);
#pragma unroll
            for (int q = 0; q < CW; ++q) {
                const int t = CW * hq + q;
                xa[q] = silu_f(fmaf(sA[t], xa[q], -fmaf(sSg[t], xb[q], r1[q])));
            }
            put_row<CW>(sm + OFF_DT, 128, jr, CW * hq, xa);
        }
        handoff();
        // ---- G5: [W2 a_t | S2 a_t] and a_t . a(k_i), partial over this CTA's slice
        const bool go5 = !failed;
        if (go5 && tid == 0) {
            const uint64_t dAQ = mdesc(aDT, T128), dW2 = mdesc(aW2, T128), dAK = mdesc(aAK, T128);
            // [W2 a_t | S2 a_t | a_t . a(k_i)] in one N=192 product (W2, S2, a(k) copies are consecutive)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
                mma_bf16(tm + COL_YW, dAQ + KS_M * ks, dW2 + KS_M * ks, ID_M64N192_TT, ks ? 1u : 0u);
            mma_commit(&bars[1]);
        }
        // while G5 runs: W1 and S1 (complete since G4) become the next chunk's
        // bf16 operands, or after the last chunk the result
        convert_state(0, c + 1 == nchunks);
        convert_state(1, c + 1 == nchunks);
        mma_wait(go5);
        // ---- E5: P2 = Gamma (.) (a_t . a(k_i))
        {
            float p[CW];
            tmem_ld_n(tl + COL_AA + CW * hq, p);
            if (r64) {
                float gr[CW];
                get_plain<CW>(Gm + tr * GST + CW * hq, gr);
#pragma unroll
                for (int q = 0; q < CW; ++q) p[q] *= gr[q];
                put_row<CW>(sm + OFF_P, 64, tr, CW * hq, p);
            }
        }
        handoff();
        // ---- G6: sum_i P2[t][i] e_i
        const bool go6 = !failed;
        if (go6 && tid == 0) {
            const uint64_t dP = kdesc(aP), dE = mdesc(aE, T64);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(tm + COL_PE, dP + KS_K * ks, dE + KS_M * ks, ID_M64N64_BT, ks ? 1u : 0u);
            mma_commit(&bars[1]);
        }
        mma_wait(go6);
        // ---- E6: partial y, reduced onto the CTA that owns the columns
        {
            float yw[CW], ys[CW], pe[CW];
            tmem_ld_n(tl + COL_YW + CW * hq, tl + COL_YW + 64 + CW * hq, tl + COL_PE + CW * hq, yw, ys, pe);
            const bool own = NC == 1 || (CW * hq) / 32 == rank;
            if (r64) {
                const float At = sA[tr], st = sSg[tr];
#pragma unroll
                for (int q = 0; q < CW; ++q) yw[q] = fmaf(At, yw[q], -fmaf(st, ys[q], pe[q]));
                if (!own && !failed) {
                    const uint32_t dst = map_to_rank(smem_u32(Yr + tr * RB + (CW * hq) % 32), (uint32_t)peer);
                    push_bf16<CW>(dst, yw, map_to_rank(smem_u32(&bars[3]), (uint32_t)peer));
                }
            }
            // while the peer's partial y arrives: W2 and S2 (no longer read by
            // G5) become the next chunk's bf16 operands, or the result
            convert_state(2, c + 1 == nchunks);
            convert_state(3, c + 1 == nchunks);
            if (c + 1 < nchunks) {  // the new W1 as the next G1's lo tile (a(k) is dead: G4 and G5 are done)
                float w[CW];
                tmem_ld_n(tl + COL_W1 + CW * hq, w);
                put_row_lo<CW>(sm + OFF_W1LO, 128, jr, CW * hq, w);
            }
            if (SURP && NC > 1 && rank == 1 && tid < BC) {  // this CTA's ||a||^2, ||delta||^2 to rank 0
                const int t = tid;
                const float a2 = (sp_a2[t] + sp_a2[BC + t]) + (sp_a2[2 * BC + t] + sp_a2[3 * BC + t]);
                const float d2 = (sp_d2[t] + sp_d2[BC + t]) + (sp_d2[2 * BC + t] + sp_d2[3 * BC + t]);
                st_cluster_f32(map_to_rank(smem_u32(sp_peer + t), 0u), a2);
                st_cluster_f32(map_to_rank(smem_u32(sp_peer + BC + t), 0u), d2);
            }
            if (NC > 1) receive(3, XCH_Y_BYTES, c);
            if (SURP && NC > 1) cluster_sync();  // the peer's surprise partials are here
            if (r64 && own && tr < n) {
                if (NC > 1) {
                    float pr[CW];
                    pull_bf16<CW>(smem_u32(Yr + tr * RB + (CW * hq) % 32), pr);
#pragma unroll
                    for (int q = 0; q < CW; ++q) yw[q] += pr[q];
                }
                if (a.y_attn) nm_gate_row<CW>(a, y + (t0 + tr) * D + CW * hq, yw);
                store_y<CW>(y + (t0 + tr) * D + CW * hq, yw);
            }
            if (SURP && rank == 0 && tid < n) {
                // surprise_t = sqrt(||delta_t||^2 ||k_t||^2 + ||e_t||^2 ||a(k_t)||^2) over all hidden units
                const int t = tid;
                float a2 = (sp_a2[t] + sp_a2[BC + t]) + (sp_a2[2 * BC + t] + sp_a2[3 * BC + t]);
                float d2 = (sp_d2[t] + sp_d2[BC + t]) + (sp_d2[2 * BC + t] + sp_d2[3 * BC + t]);
                if (NC > 1) {
                    a2 += sp_peer[t];
                    d2 += sp_peer[BC + t];
                }
                const float e2 = (sp_e2[t] + sp_e2[BC + t]) + (sp_e2[2 * BC + t] + sp_e2[3 * BC + t]);
                const float k2 = (sp_k2[t] + sp_k2[BC + t]) + (sp_k2[2 * BC + t] + sp_k2[3 * BC + t]);
                a.surprise[unit * T + t0 + t] = sqrtf(fmaf(d2, k2, e2 * a2));
            }
        }
        handoff();
    }
    if (failed) {
        if (tid == 0 && a.status) atomicExch(a.status, NM_ERR_DEVICE_TIMEOUT);
        // let copies and products still in flight land before the CTA leaves
        mbar_wait(&bars[0], (uint32_t)(nchunks & 1), WAIT_NS);
        mbar_wait(&bars[1], mma_phase, WAIT_NS);
    }
    tc_fence_before();
    if (NC > 1) cluster_sync(); else __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

template <int NC, int CW, typename Tout, bool SURP, bool HUB>
cudaError_t launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    const long long units = (long long)a.B * a.H;
    if (!make_token_map(&tq, a.q, D, a.T, units) || !make_token_map(&tk, a.k, D, a.T, units) ||
        !make_token_map(&tv, a.v, D, a.T, units))
        return cudaErrorInvalidValue;
    auto kern = tc_mlp_kernel<NC, CW, Tout, SURP, HUB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * NC), 1, 1);
    cfg.blockDim = dim3(128 * (64 / CW), 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = NC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a, c.c_mode);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int NC>
cudaError_t launch_nc(const nm_config& c, const nm_args& a, cudaStream_t s) {
    const bool hub = a.e_clip < HUGE_VALF;
    if (c.out_dtype == NM_BF16) {
        if (a.surprise)
            return hub ? launch<NC, CW_DEFAULT, __nv_bfloat16, true, true>(c, a, s)
                       : launch<NC, CW_DEFAULT, __nv_bfloat16, true, false>(c, a, s);
        return hub ? launch<NC, CW_DEFAULT, __nv_bfloat16, false, true>(c, a, s)
                   : launch<NC, CW_DEFAULT, __nv_bfloat16, false, false>(c, a, s);
    }
    if (a.surprise)
        return hub ? launch<NC, CW_DEFAULT, float, true, true>(c, a, s) : launch<NC, CW_DEFAULT, float, true, false>(c, a, s);
    return hub ? launch<NC, CW_DEFAULT, float, false, true>(c, a, s) : launch<NC, CW_DEFAULT, float, false, false>(c, a, s);
}

}  // namespace

bool nm_tc_mlp_supports(const nm_config& c) {
    return c.kind == NM_MLP2 && c.d == D && (c.hidden == HS || c.hidden == 2 * HS) && c.chunk == BC &&
           c.in_dtype == NM_BF16;
}

cudaError_t nm_tc_mlp_launch(const nm_config& c, const nm_args& a, cudaStream_t s) {
    if (c.hidden == HS) return launch_nc<1>(c, a, s);
    return launch_nc<2>(c, a, s);
}
