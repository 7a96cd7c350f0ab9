// nm_forward_mlp2_noalloc: the 2-layer MLP memory forward for callers that
// cannot allocate device memory.
//
// Some hosts cannot call cudaMalloc at the point where they run the memory
// layer: a framework that has reserved the whole device for its own pool (a
// side allocation would fail or fragment it), or a latency-critical loop that
// cannot afford cudaMalloc's implicit device-wide synchronisation.  They
// still own and pass every input and output buffer; what they cannot provide
// is the per-unit workspace the fp32 FFMA MLP kernel needs for a chunk's
// intermediates (keys' hidden activations, errors, backpropagated errors, the
// b x b decay matrix, the chunk-start weights transposed).  This entry point runs that same kernel with its
// workspace taken from one file-scope device array instead of a handle.
//
// The array is NM_NOALLOC_SCRATCH_BYTES (16 MiB) and lives on every GPU that
// loads this library until the process exits.  Host code must not pass the
// array's name to a kernel: on the host the name is only a stand-in, so every
// call looks the device address up with cudaGetSymbolAddress on the current
// device.  The first call on a device may load the module there; later calls
// are a host-side lookup that allocates nothing.  Looking it up every time
// (rather than caching it) keeps the address right after cudaDeviceReset,
// which rebuilds the context and may place the array elsewhere.
//
// Every call shares the array and it keeps the previous call's contents.  The
// kernel writes every workspace element of a chunk before it reads it, so
// nothing has to start at zero and no clearing is done.  Two calls whose
// kernels overlap on the GPU (different streams, or different host threads on
// the same device) race on the array: callers must order them.
#include "nm_internal.h"

static __device__ __align__(256) unsigned char nm_noalloc_scratch[NM_NOALLOC_SCRATCH_BYTES];

namespace {

// The array's device address on the current device.
int scratch_address(void** out) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, nm_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    *out = p;
    return NM_OK;
}

bool misaligned(const void* p) { return p && ((uintptr_t)p & 15u) != 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || !na || !nb) return false;
    const char* x = (const char*)a;
    const char* y = (const char*)b;
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" int nm_forward_mlp2_noalloc(const nm_config* cfg, int B, int H, int T, const void* q, const void* k,
                                       const void* v, const float* alpha, const float* eta, const float* beta,
                                       const float* c, const float* M0, const float* S0, void* y, float* M_T,
                                       float* S_T, void* stream) {
    if (!cfg) return NM_ERR_ARG;
    if (cfg->kind != NM_MLP2) return NM_ERR_UNSUPPORTED;
    if ((cfg->in_dtype != NM_F32 && cfg->in_dtype != NM_BF16) || (cfg->out_dtype != NM_F32 && cfg->out_dtype != NM_BF16))
        return NM_ERR_ARG;
    if (cfg->c_mode < NM_C_ONE || cfg->c_mode > NM_C_PER_TOKEN) return NM_ERR_ARG;
    if (cfg->path != NM_PATH_AUTO && cfg->path != NM_PATH_SIMT) return NM_ERR_UNSUPPORTED;
    if (cfg->loss != NM_LOSS_L2 && cfg->loss != NM_LOSS_HUBER) return NM_ERR_ARG;
    if (cfg->loss == NM_LOSS_HUBER && !(cfg->huber_delta > 0.0f && cfg->huber_delta <= 3.0e38f)) return NM_ERR_ARG;
    if (cfg->layers != 0 && (cfg->layers < 2 || cfg->layers > NM_MAX_LAYERS)) return NM_ERR_ARG;
    nm_config run = *cfg;
    run.path = NM_PATH_SIMT;
    if (!nm_simt_supports(run)) return NM_ERR_UNSUPPORTED;
    if (B < 0 || H < 0 || T < 0) return NM_ERR_ARG;
    const size_t units = (size_t)B * (size_t)H;
    if (units == 0) return NM_OK;
    if (units > (size_t)0x7fffffff) return NM_ERR_ARG;
    if (nm_simt_scratch_bytes(run, B, H) > (size_t)NM_NOALLOC_SCRATCH_BYTES) return NM_ERR_TOO_LARGE;

    const bool need_c = run.c_mode == NM_C_PER_TOKEN;
    if (!M0 || !S0 || !M_T || !S_T) return NM_ERR_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !eta || !beta || !y)) return NM_ERR_ARG;
    if ((T > 0 && need_c && !c) || (!need_c && c)) return NM_ERR_ARG;
    const void* all[] = {q, k, v, alpha, eta, beta, c, M0, S0, y, M_T, S_T};
    for (const void* p : all)
        if (misaligned(p)) return NM_ERR_ALIGN;
    const size_t tok = units * (size_t)T;
    const size_t in_b = T ? tok * run.d * (run.in_dtype == NM_BF16 ? 2 : 4) : 0;
    const size_t out_b = T ? tok * run.d * (run.out_dtype == NM_BF16 ? 2 : 4) : 0;
    const size_t g_b = T ? tok * sizeof(float) : 0;
    const size_t st_b = units * (size_t)nm_param_count(run) * sizeof(float);
    const void* ins[] = {q, k, v, alpha, eta, beta, c, M0, S0};
    const size_t in_n[] = {in_b, in_b, in_b, g_b, g_b, g_b, need_c ? g_b : 0, st_b, st_b};
    const void* outs[] = {y, M_T, S_T};
    const size_t out_n[] = {out_b, st_b, st_b};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 9; ++i) {
            const bool exact_ok = (o == 1 && i == 7) || (o == 2 && i == 8);
            if (exact_ok && outs[o] == ins[i]) continue;
            if (overlap(outs[o], out_n[o], ins[i], in_n[i])) return NM_ERR_ALIAS;
        }
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlap(outs[o], out_n[o], outs[o2], out_n[o2])) return NM_ERR_ALIAS;
    }

    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        if (M_T != M0 && cudaMemcpyAsync(M_T, M0, st_b, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return NM_ERR_CUDA;
        if (S_T != S0 && cudaMemcpyAsync(S_T, S0, st_b, cudaMemcpyDeviceToDevice, s) != cudaSuccess) return NM_ERR_CUDA;
        return NM_OK;
    }
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc != NM_OK) return rc;

    nm_args a;
    a.B = B; a.H = H; a.T = T;
    a.q = q; a.k = k; a.v = v;
    a.alpha = alpha; a.eta = eta; a.beta = beta; a.c = c;
    a.M0 = M0; a.S0 = S0; a.y = y; a.M_T = M_T; a.S_T = S_T;
    a.status = nullptr;  // the FFMA kernels have no bounded waits to report
    a.scratch = scratch;
    a.scratch_bytes = NM_NOALLOC_SCRATCH_BYTES;
    a.skip_first_load = 0;
    a.e_clip = nm_err_clip(run);
    a.surprise = nullptr;
    a.y_attn = nullptr;
    a.ckpt = nullptr;
    long long launched = 0;
    if (nm_simt_launch(run, a, s, &launched) != cudaSuccess) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    return NM_OK;
}
