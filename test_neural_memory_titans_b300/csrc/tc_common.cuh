// Blackwell (sm_103a) building blocks written as inline PTX: shared-memory
// matrix descriptors, tcgen05 MMA / TMEM access, TMA tile loads and
// mbarriers with bounded waits.  Used by the tensor-core kernels.
//
// Layout facts these helpers rely on (checked on a B300 by a one-CTA test
// kernel against host references): TMA's 128-byte swizzle places element
// (r, c) of a bf16 tile at sw128_offset(r, c, rows); K-major and MN-major
// 128-byte-swizzle descriptors as built by sw128_desc are read as described
// below; an M=64 cta_group::1 accumulator keeps row r in TMEM lane
// (r % 16) + 32 (r / 16), an M=128 accumulator row r in lane r.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tc {

// ------------------------------------------------------------------ basics

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// The two bf16 halves of a packed pair, as floats (exact).
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Byte offset of element (row r, column c) of a bf16 tile stored in the
// 128-byte-swizzle layout that TMA (CU_TENSOR_MAP_SWIZZLE_128B) and the
// tensor-core descriptors use: 64-column blocks of `rows` x 128 B, each row
// 128 B, 16-byte chunk index XOR (row % 8).  The tile base must be 1024-byte
// aligned.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t c, uint32_t rows) {
    const uint32_t blk = c >> 6;
    const uint32_t cc = c & 63u;
    return blk * rows * 128u + (r >> 3) * 1024u + (r & 7u) * 128u + ((((cc >> 3) ^ (r & 7u)) << 4)) + (cc & 7u) * 2u;
}

// Writes 32 fp32 values (columns c0..c0+31 of row r) as bf16 into a
// 128-byte-swizzled tile with `rows` rows.
__device__ __forceinline__ void put_row32(unsigned char* tile, uint32_t rows, uint32_t r, uint32_t c0, const float* v) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t off = sw128_offset(r, c0 + 8 * q, rows);
        st_shared_v4(base + off, pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                     pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
    }
}

// Writes W (16 or 32) fp32 values, columns c0..c0+W-1 of row r (c0 a
// multiple of 8), as bf16 into a 128-byte-swizzled tile with `rows` rows.
template <int W>
__device__ __forceinline__ void put_row(unsigned char* tile, uint32_t rows, uint32_t r, uint32_t c0, const float* v) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
        const uint32_t off = sw128_offset(r, c0 + 8 * q, rows);
        st_shared_v4(base + off, pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                     pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
    }
}

// The part of x that bf16 rounding drops, x - bf16(x) (exact in fp32).  Rounded
// to bf16 in turn it is the "lo" half of a hi/lo pair: hi + lo carries about 16
// significant bits, so a product taken as hi * B + lo * B (two tensor-core
// products into one fp32 accumulator) keeps fp32-like accuracy in the operand
// that was split.
__device__ __forceinline__ float bf16_residual(float x) {
    return x - __bfloat162float(__float2bfloat16_rn(x));
}

// The bf16 pair of (x0, x1) in `hi` and the pair of their residuals
// x - bf16(x) in the return value: one bf16x2 conversion for each pair (the
// rounded values are read back from the packed word by bit operations).
__device__ __forceinline__ uint32_t pack_hi_lo(float x0, float x1, uint32_t& hi) {
    hi = pack_bf16(x0, x1);
    return pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}

// put_row<W> of W values into `hi_tile` and of their residuals (the lo
// halves) into `lo_tile`, at the same row and columns.
template <int W>
__device__ __forceinline__ void put_row_hilo(unsigned char* hi_tile, unsigned char* lo_tile, uint32_t rows, uint32_t r,
                                             uint32_t c0, const float* v) {
    const uint32_t bh = smem_u32(hi_tile), bl = smem_u32(lo_tile);
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) l[p] = pack_hi_lo(v[8 * q + 2 * p], v[8 * q + 2 * p + 1], h[p]);
        const uint32_t off = sw128_offset(r, c0 + 8 * q, rows);
        st_shared_v4(bh + off, h[0], h[1], h[2], h[3]);
        st_shared_v4(bl + off, l[0], l[1], l[2], l[3]);
    }
}

__device__ __forceinline__ void put_row32_hilo(unsigned char* hi_tile, unsigned char* lo_tile, uint32_t rows,
                                               uint32_t r, uint32_t c0, const float* v) {
    put_row_hilo<32>(hi_tile, lo_tile, rows, r, c0, v);
}

// put_row<W> of the residuals x - bf16(x) of W values (the lo halves only).
template <int W>
__device__ __forceinline__ void put_row_lo(unsigned char* tile, uint32_t rows, uint32_t r, uint32_t c0, const float* v) {
    const uint32_t base = smem_u32(tile);
#pragma unroll
    for (int q = 0; q < W / 8; ++q) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) l[p] = pack_hi_lo(v[8 * q + 2 * p], v[8 * q + 2 * p + 1], h[p]);
        st_shared_v4(base + sw128_offset(r, c0 + 8 * q, rows), l[0], l[1], l[2], l[3]);
    }
}

__device__ __forceinline__ void put_row32_lo(unsigned char* tile, uint32_t rows, uint32_t r, uint32_t c0, const float* v) {
    put_row_lo<32>(tile, rows, r, c0, v);
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory at `src` into a cluster peer's at `dst` (`dst` and
// `bar` mapped to the peer), counted on the peer's mbarrier `bar` as
// transaction bytes.  The source must be visible to the async proxy
// (fence_proxy_async by its writers, then a CTA barrier).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// `limit_ns` nanoseconds of wall time and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// try_wait with acquire at cluster scope: for phases completed by the peers'
// st.async stores (whose completion releases at cluster scope).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// sigmoid(z) = (1 + tanh(z / 2)) / 2 with the hardware tanh approximation
// (relative error about 2^-11, below the bf16 rounding its results go
// through): one special-function op per element instead of an exponential
// and a reciprocal.  Epilogues that evaluate silu over a whole tile are
// bound by the special-function issue rate.
__device__ __forceinline__ float tanh_approx(float x) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float sigmoid_f(float z) { return fmaf(0.5f, tanh_approx(0.5f * z), 0.5f); }

// ------------------------------------------------------------------ TMA

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Tiled TMA store of a shared-memory box to global memory (rows or columns
// outside the tensor are not written); completion is tracked by the bulk
// async-group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the shared-memory source of every committed bulk store may be reused.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Waits until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Makes generic-proxy writes to shared memory visible to the async proxy
// (tensor core operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family form:
// start >> 4 in [0,14), leading-byte-offset >> 4 in [16,30), stride-byte-
// offset >> 4 in [32,46), version 1 in [46,48), layout 2 (SWIZZLE_128B) in
// [61,64)).  For K-major operands SBO is the stride between 8-row groups
// (1024 B) and LBO is unused; for MN-major operands LBO is the stride between
// 64-element blocks along M/N and SBO the stride between 8-row groups along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B and an
// fp32 accumulator.  a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
    return (1u << 4)                  // D format: f32
           | (1u << 7)                // A format: bf16
           | (1u << 10)               // B format: bf16
           | ((a_mn ? 1u : 0u) << 15) // A major-ness
           | ((b_mn ? 1u : 0u) << 16) // B major-ness
           | ((N >> 3) << 17)         // N / 8
           | ((M >> 4) << 24);        // M / 16
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every previously issued tcgen05.mma of this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Loads 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane
// per thread) and waits for them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
          "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]),
          "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]),
          "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31])
        : "r"(taddr)
        : "memory");
}

// Loads 32 consecutive fp32 columns at each of 2 TMEM addresses (this warp's
// 32 lanes, one lane per thread) and waits for all of them, in one asm
// statement so that no register is read before the wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t a0, uint32_t a1, float (&r0)[32], float (&r1)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15]), "=f"(r0[16]), "=f"(r0[17]), "=f"(r0[18]), "=f"(r0[19]), "=f"(r0[20]), "=f"(r0[21]), "=f"(r0[22]), "=f"(r0[23]), "=f"(r0[24]), "=f"(r0[25]), "=f"(r0[26]), "=f"(r0[27]), "=f"(r0[28]), "=f"(r0[29]), "=f"(r0[30]), "=f"(r0[31]), "=f"(r1[0]), "=f"(r1[1]), "=f"(r1[2]), "=f"(r1[3]), "=f"(r1[4]), "=f"(r1[5]), "=f"(r1[6]), "=f"(r1[7]), "=f"(r1[8]), "=f"(r1[9]), "=f"(r1[10]), "=f"(r1[11]), "=f"(r1[12]), "=f"(r1[13]), "=f"(r1[14]), "=f"(r1[15]), "=f"(r1[16]), "=f"(r1[17]), "=f"(r1[18]), "=f"(r1[19]), "=f"(r1[20]), "=f"(r1[21]), "=f"(r1[22]), "=f"(r1[23]), "=f"(r1[24]), "=f"(r1[25]), "=f"(r1[26]), "=f"(r1[27]), "=f"(r1[28]), "=f"(r1[29]), "=f"(r1[30]), "=f"(r1[31])
        : "r"(a0), "r"(a1)
        : "memory");
}

// Loads 32 consecutive fp32 columns at each of 3 TMEM addresses (this warp's
// 32 lanes, one lane per thread) and waits for all of them, in one asm
// statement so that no register is read before the wait.
__device__ __forceinline__ void tmem_ld32x3(uint32_t a0, uint32_t a1, uint32_t a2, float (&r0)[32], float (&r1)[32], float (&r2)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%96];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%97];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%98];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15]), "=f"(r0[16]), "=f"(r0[17]), "=f"(r0[18]), "=f"(r0[19]), "=f"(r0[20]), "=f"(r0[21]), "=f"(r0[22]), "=f"(r0[23]), "=f"(r0[24]), "=f"(r0[25]), "=f"(r0[26]), "=f"(r0[27]), "=f"(r0[28]), "=f"(r0[29]), "=f"(r0[30]), "=f"(r0[31]), "=f"(r1[0]), "=f"(r1[1]), "=f"(r1[2]), "=f"(r1[3]), "=f"(r1[4]), "=f"(r1[5]), "=f"(r1[6]), "=f"(r1[7]), "=f"(r1[8]), "=f"(r1[9]), "=f"(r1[10]), "=f"(r1[11]), "=f"(r1[12]), "=f"(r1[13]), "=f"(r1[14]), "=f"(r1[15]), "=f"(r1[16]), "=f"(r1[17]), "=f"(r1[18]), "=f"(r1[19]), "=f"(r1[20]), "=f"(r1[21]), "=f"(r1[22]), "=f"(r1[23]), "=f"(r1[24]), "=f"(r1[25]), "=f"(r1[26]), "=f"(r1[27]), "=f"(r1[28]), "=f"(r1[29]), "=f"(r1[30]), "=f"(r1[31]), "=f"(r2[0]), "=f"(r2[1]), "=f"(r2[2]), "=f"(r2[3]), "=f"(r2[4]), "=f"(r2[5]), "=f"(r2[6]), "=f"(r2[7]), "=f"(r2[8]), "=f"(r2[9]), "=f"(r2[10]), "=f"(r2[11]), "=f"(r2[12]), "=f"(r2[13]), "=f"(r2[14]), "=f"(r2[15]), "=f"(r2[16]), "=f"(r2[17]), "=f"(r2[18]), "=f"(r2[19]), "=f"(r2[20]), "=f"(r2[21]), "=f"(r2[22]), "=f"(r2[23]), "=f"(r2[24]), "=f"(r2[25]), "=f"(r2[26]), "=f"(r2[27]), "=f"(r2[28]), "=f"(r2[29]), "=f"(r2[30]), "=f"(r2[31])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
}


// ---- width-generic TMEM access: 16 or 32 consecutive fp32 columns of this
// warp's 32 lanes (one lane per thread).  tmem_ld_n with several addresses
// issues all loads and waits once, in one asm statement, so that no register
// is read before the wait.
__device__ __forceinline__ void tmem_ld_n(uint32_t a0, float (&r0)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15])
        : "r"(a0)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_n(uint32_t a0, uint32_t a1, float (&r0)[16], float (&r1)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15]), "=f"(r1[0]), "=f"(r1[1]), "=f"(r1[2]), "=f"(r1[3]), "=f"(r1[4]), "=f"(r1[5]), "=f"(r1[6]), "=f"(r1[7]), "=f"(r1[8]), "=f"(r1[9]), "=f"(r1[10]), "=f"(r1[11]), "=f"(r1[12]), "=f"(r1[13]), "=f"(r1[14]), "=f"(r1[15])
        : "r"(a0), "r"(a1)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_n(uint32_t a0, uint32_t a1, uint32_t a2, float (&r0)[16], float (&r1)[16], float (&r2)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%48];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%49];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%50];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15]), "=f"(r1[0]), "=f"(r1[1]), "=f"(r1[2]), "=f"(r1[3]), "=f"(r1[4]), "=f"(r1[5]), "=f"(r1[6]), "=f"(r1[7]), "=f"(r1[8]), "=f"(r1[9]), "=f"(r1[10]), "=f"(r1[11]), "=f"(r1[12]), "=f"(r1[13]), "=f"(r1[14]), "=f"(r1[15]), "=f"(r2[0]), "=f"(r2[1]), "=f"(r2[2]), "=f"(r2[3]), "=f"(r2[4]), "=f"(r2[5]), "=f"(r2[6]), "=f"(r2[7]), "=f"(r2[8]), "=f"(r2[9]), "=f"(r2[10]), "=f"(r2[11]), "=f"(r2[12]), "=f"(r2[13]), "=f"(r2[14]), "=f"(r2[15])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_n(uint32_t a0, float (&r0)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15]), "=f"(r0[16]), "=f"(r0[17]), "=f"(r0[18]), "=f"(r0[19]), "=f"(r0[20]), "=f"(r0[21]), "=f"(r0[22]), "=f"(r0[23]), "=f"(r0[24]), "=f"(r0[25]), "=f"(r0[26]), "=f"(r0[27]), "=f"(r0[28]), "=f"(r0[29]), "=f"(r0[30]), "=f"(r0[31])
        : "r"(a0)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_n(uint32_t a0, uint32_t a1, float (&r0)[32], float (&r1)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15]), "=f"(r0[16]), "=f"(r0[17]), "=f"(r0[18]), "=f"(r0[19]), "=f"(r0[20]), "=f"(r0[21]), "=f"(r0[22]), "=f"(r0[23]), "=f"(r0[24]), "=f"(r0[25]), "=f"(r0[26]), "=f"(r0[27]), "=f"(r0[28]), "=f"(r0[29]), "=f"(r0[30]), "=f"(r0[31]), "=f"(r1[0]), "=f"(r1[1]), "=f"(r1[2]), "=f"(r1[3]), "=f"(r1[4]), "=f"(r1[5]), "=f"(r1[6]), "=f"(r1[7]), "=f"(r1[8]), "=f"(r1[9]), "=f"(r1[10]), "=f"(r1[11]), "=f"(r1[12]), "=f"(r1[13]), "=f"(r1[14]), "=f"(r1[15]), "=f"(r1[16]), "=f"(r1[17]), "=f"(r1[18]), "=f"(r1[19]), "=f"(r1[20]), "=f"(r1[21]), "=f"(r1[22]), "=f"(r1[23]), "=f"(r1[24]), "=f"(r1[25]), "=f"(r1[26]), "=f"(r1[27]), "=f"(r1[28]), "=f"(r1[29]), "=f"(r1[30]), "=f"(r1[31])
        : "r"(a0), "r"(a1)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_n(uint32_t a0, uint32_t a1, uint32_t a2, float (&r0)[32], float (&r1)[32], float (&r2)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%96];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%97];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%98];\n\t"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=f"(r0[0]), "=f"(r0[1]), "=f"(r0[2]), "=f"(r0[3]), "=f"(r0[4]), "=f"(r0[5]), "=f"(r0[6]), "=f"(r0[7]), "=f"(r0[8]), "=f"(r0[9]), "=f"(r0[10]), "=f"(r0[11]), "=f"(r0[12]), "=f"(r0[13]), "=f"(r0[14]), "=f"(r0[15]), "=f"(r0[16]), "=f"(r0[17]), "=f"(r0[18]), "=f"(r0[19]), "=f"(r0[20]), "=f"(r0[21]), "=f"(r0[22]), "=f"(r0[23]), "=f"(r0[24]), "=f"(r0[25]), "=f"(r0[26]), "=f"(r0[27]), "=f"(r0[28]), "=f"(r0[29]), "=f"(r0[30]), "=f"(r0[31]), "=f"(r1[0]), "=f"(r1[1]), "=f"(r1[2]), "=f"(r1[3]), "=f"(r1[4]), "=f"(r1[5]), "=f"(r1[6]), "=f"(r1[7]), "=f"(r1[8]), "=f"(r1[9]), "=f"(r1[10]), "=f"(r1[11]), "=f"(r1[12]), "=f"(r1[13]), "=f"(r1[14]), "=f"(r1[15]), "=f"(r1[16]), "=f"(r1[17]), "=f"(r1[18]), "=f"(r1[19]), "=f"(r1[20]), "=f"(r1[21]), "=f"(r1[22]), "=f"(r1[23]), "=f"(r1[24]), "=f"(r1[25]), "=f"(r1[26]), "=f"(r1[27]), "=f"(r1[28]), "=f"(r1[29]), "=f"(r1[30]), "=f"(r1[31]), "=f"(r2[0]), "=f"(r2[1]), "=f"(r2[2]), "=f"(r2[3]), "=f"(r2[4]), "=f"(r2[5]), "=f"(r2[6]), "=f"(r2[7]), "=f"(r2[8]), "=f"(r2[9]), "=f"(r2[10]), "=f"(r2[11]), "=f"(r2[12]), "=f"(r2[13]), "=f"(r2[14]), "=f"(r2[15]), "=f"(r2[16]), "=f"(r2[17]), "=f"(r2[18]), "=f"(r2[19]), "=f"(r2[20]), "=f"(r2[21]), "=f"(r2[22]), "=f"(r2[23]), "=f"(r2[24]), "=f"(r2[25]), "=f"(r2[26]), "=f"(r2[27]), "=f"(r2[28]), "=f"(r2[29]), "=f"(r2[30]), "=f"(r2[31])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
}
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const float (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
        "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
        "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7]), "f"(r[8]), "f"(r[9]), "f"(r[10]), "f"(r[11]), "f"(r[12]), "f"(r[13]), "f"(r[14]), "f"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const float (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
        "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7]), "f"(r[8]), "f"(r[9]), "f"(r[10]), "f"(r[11]), "f"(r[12]), "f"(r[13]), "f"(r[14]), "f"(r[15]), "f"(r[16]), "f"(r[17]), "f"(r[18]), "f"(r[19]), "f"(r[20]), "f"(r[21]), "f"(r[22]), "f"(r[23]), "f"(r[24]), "f"(r[25]), "f"(r[26]), "f"(r[27]), "f"(r[28]), "f"(r[29]), "f"(r[30]), "f"(r[31])
        : "memory");
}

// Stores 32 consecutive fp32 columns of this warp's 32 TMEM lanes and waits.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
        "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7]), "f"(r[8]),
        "f"(r[9]), "f"(r[10]), "f"(r[11]), "f"(r[12]), "f"(r[13]), "f"(r[14]), "f"(r[15]), "f"(r[16]), "f"(r[17]),
        "f"(r[18]), "f"(r[19]), "f"(r[20]), "f"(r[21]), "f"(r[22]), "f"(r[23]), "f"(r[24]), "f"(r[25]),
        "f"(r[26]), "f"(r[27]), "f"(r[28]), "f"(r[29]), "f"(r[30]), "f"(r[31])
        : "memory");
}

// ------------------------------------------------------------------ clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of every CTA of the cluster: release this CTA's prior memory
// operations (including stores to peers' shared memory) and acquire the
// peers'.  Every thread of the cluster must execute the same sequence of
// cluster_sync calls.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync, for work that does not depend on the peers
// placed between them: cluster_arrive releases, cluster_wait blocks until every
// thread of the cluster has arrived and acquires.  Each thread alternates the
// two, and every thread of the cluster executes the same sequence.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in the shared memory of cluster CTA `rank` that corresponds to the
// local shared-memory address `saddr`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// Non-blocking stores of 16 / 8 bytes into a cluster peer's shared memory
// (`addr` and `bar` both mapped to that peer): on landing, each counts its
// bytes on the peer's mbarrier `bar` as completed transaction bytes, with
// release at cluster scope.  The sender does not wait for them.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(addr),
                 "r"(a), "r"(b), "r"(c), "r"(d), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_b32(uint32_t addr, uint32_t a, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr), "r"(a),
                 "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void st_async_v2(uint32_t addr, uint32_t a, uint32_t b, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "r"(a), "r"(b), "r"(bar)
                 : "memory");
}

// ------------------------------------------------------------------ host: tensor maps

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A [units][T][d] bf16 array viewed as a 3-D tensor, read in boxes of 64
// features x 64 tokens x 1 unit with the 128-byte swizzle.  Tokens past T
// read as zero.  The feature coordinate of every load is a multiple of 64,
// so the 16-byte rule for the innermost coordinate always holds.
inline bool make_token_map(CUtensorMap* m, const void* base, int d, long long T, long long units) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)units};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [units][T][d] array (bf16 or fp32) viewed as a 3-D tensor, written in
// boxes of d features x 64 tokens x 1 unit without swizzle (a plain row-major
// [64][d] shared-memory tile); rows past T are not written.
inline bool make_token_store_map(CUtensorMap* m, void* base, int d, long long T, long long units, bool bf16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t es = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)units};
    cuuint64_t strides[2] = {(cuuint64_t)d * es, (cuuint64_t)T * d * es};
    cuuint32_t box[3] = {(cuuint32_t)d, 64, 1};
    cuuint32_t el[3] = {1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box,
               el, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc
