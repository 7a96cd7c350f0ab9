// Internal declarations shared by the host API (nm_api.cu) and the kernel
// files.  Not part of the public ABI.
#pragma once

#include <math.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "nm.h"

// One forward call's arguments, already validated on the host.
struct nm_args {
    int B, H, T;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* eta;
    const float* beta;
    const float* c;
    const float* M0;
    const float* S0;
    void* y;
    float* M_T;
    float* S_T;
    int* status;      // device status word owned by the handle
    void* scratch;    // device workspace owned by the handle (may be NULL)
    size_t scratch_bytes;
    int skip_first_load;  // test hook: tensor-core kernels skip chunk 0's tile loads
    float e_clip;     // |e| bound: 2 delta for the Huber loss, +inf for the squared loss
    float* surprise;  // [B, H, T] per-token gradient norms, or NULL (not computed)
    const void* y_attn;  // [B, H, T, d] of y's type: when set, the call writes o = sigmoid(y) * y_attn
                         // (the Memory-as-Gate combination) in place of y; NULL for the plain forward
    float* ckpt;         // [B*H][ceil(T / chunk)][2][P] fp32: when set (fp32 FFMA linear kernel, for the
                         // backward pass), every chunk's start state (M, S); y may then be NULL (not written)
};

// The error e = d rho / d r of the loss at the residual r = M(k) - v, given
// 2 r: unchanged for the squared loss (e_clip = +inf), clipped to
// [-2 delta, 2 delta] for the Huber loss.  A NaN passes through unchanged.
__host__ __device__ inline float nm_clip_err(float two_r, float e_clip) {
    return two_r > e_clip ? e_clip : (two_r < -e_clip ? -e_clip : two_r);
}

#ifdef __CUDACC__
__device__ __forceinline__ float nm_to_f32(float x) { return x; }
__device__ __forceinline__ float nm_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// The value a kernel writes at output element p (a pointer into a.y) for the
// memory's retrieval y there: y itself, or with a.y_attn set the
// Memory-as-Gate combination o = sigmoid(y) * y_attn at the same index
// (0h-n0.github.io explainer, "3つのアーキテクチャ変種", MAG; "Titans:
// Imparare a Memorizzare al Tempo di Test", "Varianti dell'Architettura
// Titans", "Memory as Gate (MAG)").  Each element of y_attn is read by the
// thread that writes the same element of o, before it writes it, so o may be
// y_attn itself.
template <typename Tout>
__device__ __forceinline__ float nm_gated(const nm_args& a, const Tout* p, float y) {
    if (!a.y_attn) return y;
    const Tout* ya = reinterpret_cast<const Tout*>(a.y_attn) + (p - reinterpret_cast<const Tout*>(a.y));
    return nm_to_f32(*ya) / (1.0f + expf(-y));
}

// o = sigmoid(y) * y_attn for the tensor-core kernels' epilogues, with the
// fast exponential and division (a few ulp of fp32, far below the bf16
// rounding of their outputs; for y below about -88 the exponential
// overflows and o is 0, the limit).  The fp32 FFMA kernels keep the exact form.
__device__ __forceinline__ float nm_gate_fast(float y_attn, float y) {
    return __fdividef(y_attn, 1.0f + __expf(-y));
}

// The gated output's y_attn bytes [off, off + bytes) into L2, one 128-byte line
// per thread (thread `tid` of `nthreads`): issued at a chunk's start so that the
// epilogue's loads of the chunk's y_attn find them there.  Nothing is read.
__device__ __forceinline__ void nm_prefetch_attn(const nm_args& a, long long off, long long bytes, int tid,
                                                 int nthreads) {
    const char* base = reinterpret_cast<const char*>(a.y_attn) + off;
    for (long long i = tid; i * 128 < bytes; i += nthreads)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(base + i * 128));
}

// W consecutive elements y_attn[idx .. idx + W) as floats, with 16-byte loads
// (idx a multiple of 8 for bf16, of 4 for fp32, and y_attn 16-byte aligned),
// all issued before any is used.
template <int W>
__device__ __forceinline__ void nm_load_row(const __nv_bfloat16* p, float* v) {
#pragma unroll
    for (int i = 0; i < W / 8; ++i) {
        const uint4 w = reinterpret_cast<const uint4*>(p)[i];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
            v[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
        }
    }
}
template <int W>
__device__ __forceinline__ void nm_load_row(const float* p, float* v) {
#pragma unroll
    for (int i = 0; i < W / 4; ++i) {
        const float4 w = reinterpret_cast<const float4*>(p)[i];
        v[4 * i] = w.x; v[4 * i + 1] = w.y; v[4 * i + 2] = w.z; v[4 * i + 3] = w.w;
    }
}

// The Memory-as-Gate combination over W consecutive outputs starting at p
// (a pointer into a.y, its element index a multiple of 8): v <- sigmoid(v) *
// y_attn, the y_attn row loaded first.  Call it only when a.y_attn is set.
template <int W, typename Tout>
__device__ __forceinline__ void nm_gate_row(const nm_args& a, const Tout* p, float* v) {
    float ya[W];
    nm_load_row<W>(reinterpret_cast<const Tout*>(a.y_attn) + (p - reinterpret_cast<const Tout*>(a.y)), ya);
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = nm_gate_fast(ya[i], v[i]);
}
#endif

// nm_forward_host's copy / compute overlap: at most this many unit groups, each
// on a compute stream of its own, and one group per NM_HOST_GROUP_BYTES of q + y.
constexpr int NM_HOST_MAX_GROUPS = 16;
constexpr size_t NM_HOST_GROUP_BYTES = (size_t)16 << 20;

struct nm_handle {
    nm_config cfg;
    int device;
    int path;          // NM_PATH_SIMT or NM_PATH_TC
    int num_sms;
    int* d_status;
    void* workspace;
    size_t workspace_bytes;
    void* stage;       // device staging for nm_forward_host
    size_t stage_bytes;
    void* bwd_ws;      // device workspace of nm_backward (checkpoints, per-unit scratch), grows on demand
    size_t bwd_ws_bytes;
    long long launches;
    int inject_load_skip;  // armed by nm_inject_missing_load, consumed by the next nm_forward
    // nm_forward_host's copy / compute overlap (created on first use): streams for the
    // host->device and device->host copies and one compute stream per group of units
    int pipe_ready;
    cudaStream_t s_in, s_out, s_comp[NM_HOST_MAX_GROUPS];
    cudaEvent_t ev_start, ev_end, ev_in[NM_HOST_MAX_GROUPS], ev_done[NM_HOST_MAX_GROUPS];
};

// The |e| bound of a configuration (see nm_clip_err).
static inline float nm_err_clip(const nm_config& c) {
    return c.loss == NM_LOSS_HUBER ? 2.0f * c.huber_delta : HUGE_VALF;
}

// Depth of an MLP2 memory (a zero `layers` means 2); 1 for the linear memory.
static inline int nm_layers(const nm_config& c) {
    return c.kind == NM_MLP2 ? (c.layers > 2 ? c.layers : 2) : 1;
}

// Parameters per unit.
static inline long long nm_param_count(const nm_config& c) {
    return c.kind == NM_LINEAR ? (long long)c.d * c.d
                               : 2LL * c.hidden * c.d + (long long)(nm_layers(c) - 2) * c.hidden * c.hidden;
}

// ---- backward pass (nm_backward.cu) ----------------------------------------
// One backward call's device pointers, validated on the host.
struct nm_bwd_call {
    long long units, T;
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* eta;
    const float* beta;
    const float* c;
    const float* ckpt;  // chunk-start states from the checkpointing forward
    const float* Gy;
    const float* GM;
    const float* GS;
    float* dq;
    float* dk;
    float* dv;
    float* dalpha;
    float* deta;
    float* dbeta;
    float* dc;
    float* dM0;
    float* dS0;
    float* ws;
    float e_clip;
};
bool nm_bwd_supports(const nm_config& c);
size_t nm_bwd_linear_ws_floats(int d, int b);
size_t nm_bwd_ws_floats(const nm_config& c);  // per-unit scratch of the reverse sweep
cudaError_t nm_bwd_launch(const nm_config& c, const nm_bwd_call& call, cudaStream_t s);

// ---- fp32 FFMA kernels (nm_simt.cu) ----------------------------------------
bool nm_simt_supports(const nm_config& c);
size_t nm_simt_scratch_bytes(const nm_config& c, int B, int H);
cudaError_t nm_simt_launch(const nm_config& c, const nm_args& a, cudaStream_t s, long long* launches);

// ---- tcgen05 tensor-core kernels (nm_tc_*.cu) -----------------------------
bool nm_tc_supports(const nm_config& c);
bool nm_tc_supports_surprise(const nm_config& c);

// Whether the kernel family `path` writes the per-token surprise for `c`.
static inline bool nm_supports_surprise(const nm_config& c, int path) {
    return path == NM_PATH_SIMT || nm_tc_supports_surprise(c);
}
size_t nm_tc_scratch_bytes(const nm_config& c, int B, int H);
cudaError_t nm_tc_launch(const nm_config& c, const nm_args& a, cudaStream_t s, int num_sms, long long* launches);
