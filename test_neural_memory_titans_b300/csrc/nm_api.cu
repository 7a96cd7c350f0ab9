// Host side of the C ABI declared in include/nm.h: argument validation,
// aliasing rules, handle-owned device memory, dispatch to the kernel files.
// No arithmetic of the method happens here.
#include <algorithm>
#include <stdlib.h>
#include <string.h>

#include "nm_internal.h"

// The backward pass's reverse sweep with tensor-core contractions (nm_backward.cu).
cudaError_t nm_bwd_launch_tc(const nm_config& c, const nm_bwd_call& call, int* status, cudaStream_t s);
bool nm_tc_supports_ckpt(const nm_config& c);  // (nm_tc.cu)

namespace {

// Makes `dev` current for the scope and restores the caller's device after.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

bool valid_dtype(int t) { return t == NM_F32 || t == NM_BF16; }
size_t dtype_bytes(int t) { return t == NM_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct Range {
    const char* p;
    size_t n;
};

bool overlaps(Range a, Range b) {
    if (a.n == 0 || b.n == 0 || a.p == nullptr || b.p == nullptr) return false;
    return a.p < b.p + b.n && b.p < a.p + a.n;
}

int check_config(const nm_config* c) {
    if (!c) return NM_ERR_ARG;
    if (c->kind != NM_LINEAR && c->kind != NM_MLP2) return NM_ERR_ARG;
    if (!valid_dtype(c->in_dtype) || !valid_dtype(c->out_dtype)) return NM_ERR_ARG;
    if (c->c_mode < NM_C_ONE || c->c_mode > NM_C_PER_TOKEN) return NM_ERR_ARG;
    if (c->path < NM_PATH_AUTO || c->path > NM_PATH_TC) return NM_ERR_ARG;
    if (c->d <= 0 || c->chunk <= 0) return NM_ERR_ARG;
    if (c->kind == NM_MLP2 && c->hidden <= 0) return NM_ERR_ARG;
    if (c->loss != NM_LOSS_L2 && c->loss != NM_LOSS_HUBER) return NM_ERR_ARG;
    if (c->loss == NM_LOSS_HUBER && !(c->huber_delta > 0.0f && c->huber_delta <= 3.0e38f)) return NM_ERR_ARG;
    if (c->layers != 0 && (c->kind != NM_MLP2 || c->layers < 2 || c->layers > NM_MAX_LAYERS)) return NM_ERR_ARG;
    return NM_OK;
}

int select_path(const nm_config& c) {
    bool tc = nm_tc_supports(c);
    bool simt = nm_simt_supports(c);
    if (c.path == NM_PATH_TC) return tc ? NM_PATH_TC : -1;
    if (c.path == NM_PATH_SIMT) return simt ? NM_PATH_SIMT : -1;
    if (tc) return NM_PATH_TC;
    if (simt) return NM_PATH_SIMT;
    return -1;
}

// Streams and events of nm_forward_host's copy / compute overlap, created once per handle.
int ensure_pipe(nm_handle* h) {
    if (h->pipe_ready) return NM_OK;
    bool ok = cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&h->ev_end, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < NM_HOST_MAX_GROUPS; ++i)
        ok = cudaStreamCreateWithFlags(&h->s_comp[i], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->ev_done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    h->pipe_ready = 1;
    return NM_OK;
}

int ensure_workspace(nm_handle* h, size_t bytes) {
    if (bytes <= h->workspace_bytes) return NM_OK;
    if (h->workspace) {
        if (cudaFree(h->workspace) != cudaSuccess) return NM_ERR_CUDA;
        h->workspace = nullptr;
        h->workspace_bytes = 0;
    }
    if (cudaMalloc(&h->workspace, bytes) != cudaSuccess) {
        cudaGetLastError();
        h->workspace = nullptr;
        return NM_ERR_NOMEM;
    }
    h->workspace_bytes = bytes;
    return NM_OK;
}

}  // namespace

extern "C" {

const char* nm_status_string(int s) {
    switch (s) {
        case NM_OK: return "ok";
        case NM_ERR_ARG: return "invalid argument (null pointer, bad size or bad enum)";
        case NM_ERR_ALIGN: return "pointer not 16-byte aligned";
        case NM_ERR_UNSUPPORTED: return "no kernel built for this (kind, d, hidden, chunk, dtype, path)";
        case NM_ERR_ALIAS: return "output buffer overlaps another buffer (only M_T==M0 and S_T==S0 may alias)";
        case NM_ERR_CUDA: return "CUDA runtime error";
        case NM_ERR_NOMEM: return "allocation failed";
        case NM_ERR_DEVICE_TIMEOUT: return "a bounded on-device wait gave up";
        case NM_ERR_DEVICE_CHECK: return "an on-device consistency check failed";
        case NM_ERR_TOO_LARGE: return "call needs more workspace than the fixed no-alloc array holds";
        default: return "unknown status";
    }
}

int nm_create(const nm_config* cfg, int device, nm_handle_t* out) {
    if (!out) return NM_ERR_ARG;
    int rc = check_config(cfg);
    if (rc != NM_OK) return rc;
    int path = select_path(*cfg);
    if (path < 0) return NM_ERR_UNSUPPORTED;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    if (device < 0 || device >= ndev) return NM_ERR_ARG;
    DeviceGuard g(device);
    if (!g.ok) return NM_ERR_CUDA;
    nm_handle* h = (nm_handle*)calloc(1, sizeof(nm_handle));
    if (!h) return NM_ERR_NOMEM;
    h->cfg = *cfg;
    h->device = device;
    h->path = path;
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        free(h);
        return NM_ERR_CUDA;
    }
    if (cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        free(h);
        return NM_ERR_NOMEM;
    }
    if (cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(h->d_status);
        free(h);
        return NM_ERR_CUDA;
    }
    *out = h;
    return NM_OK;
}

int nm_selected_path(nm_handle_t h) { return h ? h->path : -NM_ERR_ARG; }

int nm_inject_missing_load(nm_handle_t h) {
    if (!h) return NM_ERR_ARG;
    if (h->path != NM_PATH_TC) return NM_ERR_UNSUPPORTED;
    h->inject_load_skip = 1;
    return NM_OK;
}

long long nm_launch_count(nm_handle_t h) { return h ? h->launches : -1; }

namespace {

int forward_impl(nm_handle_t h, int B, int H, int T, const void* q, const void* k, const void* v,
                 const float* alpha, const float* eta, const float* beta, const float* c, const float* M0,
                 const float* S0, void* y, float* M_T, float* S_T, float* surprise, void* stream,
                 const void* y_attn = nullptr) {
    if (!h) return NM_ERR_ARG;
    const nm_config& cfg = h->cfg;
    if (B < 0 || H < 0 || T < 0) return NM_ERR_ARG;
    const long long units = (long long)B * H;
    if (units == 0) return NM_OK;
    if (units > (1LL << 31) - 1 || (long long)T * cfg.d > (1LL << 40)) return NM_ERR_ARG;
    const bool need_c = cfg.c_mode == NM_C_PER_TOKEN;
    if (!M0 || !S0 || !M_T || !S_T) return NM_ERR_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !eta || !beta || !y)) return NM_ERR_ARG;
    if (T > 0 && need_c && !c) return NM_ERR_ARG;
    if (!need_c && c) return NM_ERR_ARG;
    const void* ptrs[] = {q, k, v, alpha, eta, beta, c, M0, S0, y, M_T, S_T, surprise, y_attn};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return NM_ERR_ALIGN;
    if (surprise && !nm_supports_surprise(cfg, h->path)) return NM_ERR_UNSUPPORTED;

    const size_t tok = (size_t)units * (size_t)T;
    const size_t P = (size_t)nm_param_count(cfg);
    const size_t in_b = tok * cfg.d * dtype_bytes(cfg.in_dtype);
    const size_t out_b = tok * cfg.d * dtype_bytes(cfg.out_dtype);
    const size_t gate_b = tok * sizeof(float);
    const size_t st_b = (size_t)units * P * sizeof(float);
    Range in_r[] = {{(const char*)q, T ? in_b : 0},       {(const char*)k, T ? in_b : 0},
                    {(const char*)v, T ? in_b : 0},       {(const char*)alpha, gate_b},
                    {(const char*)eta, gate_b},           {(const char*)beta, gate_b},
                    {(const char*)c, need_c ? gate_b : 0}, {(const char*)M0, st_b},
                    {(const char*)S0, st_b},              {(const char*)y_attn, T ? out_b : 0}};
    Range out_r[] = {{(const char*)y, T ? out_b : 0}, {(const char*)M_T, st_b}, {(const char*)S_T, st_b},
                     {(const char*)surprise, T ? gate_b : 0}};
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 10; ++i) {
            // in-place carry of the state, and the gated output over the attention branch's buffer
            bool exact_ok = (o == 1 && i == 7) || (o == 2 && i == 8) || (o == 0 && i == 9);
            if (exact_ok && out_r[o].p == in_r[i].p) continue;
            if (overlaps(out_r[o], in_r[i])) return NM_ERR_ALIAS;
        }
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlaps(out_r[o], out_r[o2])) return NM_ERR_ALIAS;
    }

    DeviceGuard g(h->device);
    if (!g.ok) return NM_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {
        if (M_T != M0 && cudaMemcpyAsync(M_T, M0, st_b, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return NM_ERR_CUDA;
        if (S_T != S0 && cudaMemcpyAsync(S_T, S0, st_b, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return NM_ERR_CUDA;
        return NM_OK;
    }
    size_t ws = h->path == NM_PATH_TC ? nm_tc_scratch_bytes(cfg, B, H) : nm_simt_scratch_bytes(cfg, B, H);
    int rc = ensure_workspace(h, ws);
    if (rc != NM_OK) return rc;

    nm_args a;
    a.B = B; a.H = H; a.T = T;
    a.q = q; a.k = k; a.v = v;
    a.alpha = alpha; a.eta = eta; a.beta = beta; a.c = c;
    a.M0 = M0; a.S0 = S0; a.y = y; a.M_T = M_T; a.S_T = S_T;
    a.status = h->d_status;
    a.scratch = h->workspace;
    a.scratch_bytes = h->workspace_bytes;
    a.skip_first_load = h->inject_load_skip;
    h->inject_load_skip = 0;
    a.e_clip = nm_err_clip(cfg);
    a.surprise = surprise;
    a.y_attn = y_attn;
    a.ckpt = nullptr;
    cudaError_t e = h->path == NM_PATH_TC ? nm_tc_launch(cfg, a, s, h->num_sms, &h->launches)
                                          : nm_simt_launch(cfg, a, s, &h->launches);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    return NM_OK;
}

}  // namespace

int nm_forward(nm_handle_t h, int B, int H, int T, const void* q, const void* k, const void* v,
               const float* alpha, const float* eta, const float* beta, const float* c,
               const float* M0, const float* S0, void* y, float* M_T, float* S_T, void* stream) {
    return forward_impl(h, B, H, T, q, k, v, alpha, eta, beta, c, M0, S0, y, M_T, S_T, nullptr, stream);
}

int nm_forward_surprise(nm_handle_t h, int B, int H, int T, const void* q, const void* k, const void* v,
                        const float* alpha, const float* eta, const float* beta, const float* c,
                        const float* M0, const float* S0, void* y, float* M_T, float* S_T, float* surprise,
                        void* stream) {
    if (!surprise) return NM_ERR_ARG;
    return forward_impl(h, B, H, T, q, k, v, alpha, eta, beta, c, M0, S0, y, M_T, S_T, surprise, stream);
}

int nm_forward_gated(nm_handle_t h, int B, int H, int T, const void* q, const void* k, const void* v,
                     const float* alpha, const float* eta, const float* beta, const float* c,
                     const float* M0, const float* S0, const void* y_attn, void* o, float* M_T, float* S_T,
                     void* stream) {
    if (T > 0 && !y_attn) return NM_ERR_ARG;
    return forward_impl(h, B, H, T, q, k, v, alpha, eta, beta, c, M0, S0, o, M_T, S_T, nullptr, stream,
                        T > 0 ? y_attn : nullptr);
}

int nm_backward(nm_handle_t h, int B, int H, int T, const void* q, const void* k, const void* v,
                const float* alpha, const float* eta, const float* beta, const float* c, const float* M0,
                const float* S0, const float* Gy, const float* GM, const float* GS, float* dq, float* dk,
                float* dv, float* dalpha, float* deta, float* dbeta, float* dc, float* dM0, float* dS0,
                void* stream) {
    if (!h) return NM_ERR_ARG;
    const nm_config& cfg = h->cfg;
    if (B < 0 || H < 0 || T < 0) return NM_ERR_ARG;
    const long long units = (long long)B * H;
    if (units == 0) return NM_OK;
    if (units > (1LL << 31) - 1 || (long long)T * cfg.d > (1LL << 40)) return NM_ERR_ARG;
    if (!nm_bwd_supports(cfg)) return NM_ERR_UNSUPPORTED;
    const bool need_c = cfg.c_mode == NM_C_PER_TOKEN;
    if (!M0 || !S0 || !GM || !GS || !dM0 || !dS0) return NM_ERR_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !eta || !beta || !Gy || !dq || !dk || !dv || !dalpha || !deta || !dbeta))
        return NM_ERR_ARG;
    if (T > 0 && need_c != (c != nullptr)) return NM_ERR_ARG;
    if (T > 0 && need_c != (dc != nullptr)) return NM_ERR_ARG;
    if (T == 0 && (c || dc)) return NM_ERR_ARG;
    const void* ptrs[] = {q, k, v, alpha, eta, beta, c, M0, S0, Gy, GM, GS, dq, dk, dv, dalpha, deta, dbeta, dc,
                          dM0, dS0};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return NM_ERR_ALIGN;
    const size_t tok = (size_t)units * (size_t)T;
    const size_t P = (size_t)nm_param_count(cfg);
    const size_t in_b = tok * cfg.d * dtype_bytes(cfg.in_dtype), g_b = tok * sizeof(float);
    const size_t tf_b = tok * cfg.d * sizeof(float), st_b = (size_t)units * P * sizeof(float);
    Range in_r[] = {{(const char*)q, T ? in_b : 0}, {(const char*)k, T ? in_b : 0}, {(const char*)v, T ? in_b : 0},
                    {(const char*)alpha, T ? g_b : 0}, {(const char*)eta, T ? g_b : 0},
                    {(const char*)beta, T ? g_b : 0}, {(const char*)c, need_c && T ? g_b : 0},
                    {(const char*)M0, st_b}, {(const char*)S0, st_b}, {(const char*)Gy, T ? tf_b : 0},
                    {(const char*)GM, st_b}, {(const char*)GS, st_b}};
    Range out_r[] = {{(const char*)dq, T ? tf_b : 0}, {(const char*)dk, T ? tf_b : 0},
                     {(const char*)dv, T ? tf_b : 0}, {(const char*)dalpha, T ? g_b : 0},
                     {(const char*)deta, T ? g_b : 0}, {(const char*)dbeta, T ? g_b : 0},
                     {(const char*)dc, need_c && T ? g_b : 0}, {(const char*)dM0, st_b}, {(const char*)dS0, st_b}};
    for (const Range& o : out_r) {
        for (const Range& i : in_r)
            if (overlaps(o, i)) return NM_ERR_ALIAS;
        for (const Range& o2 : out_r)
            if (&o2 != &o && overlaps(o, o2)) return NM_ERR_ALIAS;
    }

    DeviceGuard g(h->device);
    if (!g.ok) return NM_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (T == 0) {  // nothing happens between the inputs and the outputs: the state's adjoints pass through
        if (cudaMemcpyAsync(dM0, GM, st_b, cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(dS0, GS, st_b, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
            return NM_ERR_CUDA;
        return NM_OK;
    }
    // workspace: the chunk-start states of every unit, the forward's final state (not returned), and the
    // reverse sweep's per-unit scratch
    const long long nch = ((long long)T + cfg.chunk - 1) / cfg.chunk;
    auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
    const size_t ck_b = up((size_t)units * nch * 2 * P * sizeof(float));
    const size_t fin_b = up(2 * st_b);
    const size_t sc_b = up((size_t)units * nm_bwd_ws_floats(cfg) * sizeof(float));
    nm_config fc = cfg;
    fc.path = NM_PATH_SIMT;
    // the checkpointing forward: on a tensor-core handle the tcgen05 kernel where one records checkpoints
    // (its states carry the bf16-operand rounding of that path's forward), else the fp32 FFMA kernel
    const bool tc_ckpt = cfg.path == NM_PATH_TC && nm_tc_supports_ckpt(cfg);
    const size_t fw_b = tc_ckpt ? 0 : up(nm_simt_scratch_bytes(fc, B, H));  // the forward kernel's own workspace
    const size_t need = ck_b + fin_b + sc_b + fw_b;
    if (need > h->bwd_ws_bytes) {
        if (h->bwd_ws) cudaFree(h->bwd_ws);
        h->bwd_ws = nullptr;
        h->bwd_ws_bytes = 0;
        if (cudaMalloc(&h->bwd_ws, need) != cudaSuccess) {
            cudaGetLastError();
            return NM_ERR_NOMEM;
        }
        h->bwd_ws_bytes = need;
    }
    char* w = (char*)h->bwd_ws;
    float* ckpt = (float*)w;
    float* fin = (float*)(w + ck_b);
    float* scratch = (float*)(w + ck_b + fin_b);
    void* fw_scratch = fw_b ? (void*)(w + ck_b + fin_b + sc_b) : nullptr;

    // the forward once more, recording each chunk's start state (y is not written)
    nm_args a;
    a.B = B; a.H = H; a.T = T;
    a.q = q; a.k = k; a.v = v;
    a.alpha = alpha; a.eta = eta; a.beta = beta; a.c = c;
    a.M0 = M0; a.S0 = S0; a.y = nullptr; a.M_T = fin; a.S_T = fin + units * P;
    a.status = h->d_status;
    a.scratch = fw_scratch;
    a.scratch_bytes = fw_b;
    a.skip_first_load = 0;
    a.e_clip = nm_err_clip(cfg);
    a.surprise = nullptr;
    a.y_attn = nullptr;
    a.ckpt = ckpt;
    if ((tc_ckpt ? nm_tc_launch(cfg, a, s, h->num_sms, &h->launches) : nm_simt_launch(fc, a, s, &h->launches)) !=
        cudaSuccess) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    nm_bwd_call bc;
    bc.units = units; bc.T = T;
    bc.q = q; bc.k = k; bc.v = v;
    bc.alpha = alpha; bc.eta = eta; bc.beta = beta; bc.c = c;
    bc.ckpt = ckpt;
    bc.Gy = Gy; bc.GM = GM; bc.GS = GS;
    bc.dq = dq; bc.dk = dk; bc.dv = dv;
    bc.dalpha = dalpha; bc.deta = deta; bc.dbeta = dbeta; bc.dc = dc;
    bc.dM0 = dM0; bc.dS0 = dS0;
    bc.ws = scratch;
    bc.e_clip = nm_err_clip(cfg);
    // the reverse sweep's contractions on the tensor cores (tf32) when the handle asked for NM_PATH_TC, else
    // fp32 FFMA (NM_PATH_AUTO: the same speed, since the sweep is bound by its other steps, at fp32 accuracy)
    const cudaError_t be = cfg.path == NM_PATH_TC ? nm_bwd_launch_tc(cfg, bc, h->d_status, s) : nm_bwd_launch(cfg, bc, s);
    if (be != cudaSuccess) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    h->launches += 1;
    return NM_OK;
}

int nm_synchronize(nm_handle_t h) {
    if (!h) return NM_ERR_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return NM_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    int st = 0;
    if (cudaMemcpy(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NM_ERR_CUDA;
    if (st != 0 && cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) return NM_ERR_CUDA;
    return st;
}

int nm_forward_host(nm_handle_t h, int B, int H, int T, const void* q, const void* k, const void* v,
                    const float* alpha, const float* eta, const float* beta, const float* c,
                    const float* M0, const float* S0, void* y, float* M_T, float* S_T, void* stream) {
    if (!h) return NM_ERR_ARG;
    const nm_config& cfg = h->cfg;
    if (B < 0 || H < 0 || T < 0) return NM_ERR_ARG;
    const size_t units = (size_t)B * H;
    if (units == 0) return NM_OK;
    const bool need_c = cfg.c_mode == NM_C_PER_TOKEN;
    if (!M0 || !S0 || !M_T || !S_T) return NM_ERR_ARG;
    if (T > 0 && (!q || !k || !v || !alpha || !eta || !beta || !y)) return NM_ERR_ARG;
    if (T > 0 && need_c && !c) return NM_ERR_ARG;
    if (!need_c && c) return NM_ERR_ARG;
    const size_t tok = units * (size_t)T;
    const size_t P = (size_t)nm_param_count(cfg);
    auto up = [](size_t n) { return (n + 255) & ~(size_t)255; };
    const size_t in_b = tok * cfg.d * dtype_bytes(cfg.in_dtype);
    const size_t out_b = tok * cfg.d * dtype_bytes(cfg.out_dtype);
    const size_t gate_b = tok * sizeof(float);
    const size_t st_b = units * P * sizeof(float);
    const size_t total = 3 * up(in_b) + 4 * up(gate_b) + 4 * up(st_b) + up(out_b);

    DeviceGuard g(h->device);
    if (!g.ok) return NM_ERR_CUDA;
    if (total > h->stage_bytes) {
        if (h->stage) cudaFree(h->stage);
        h->stage = nullptr;
        h->stage_bytes = 0;
        if (cudaMalloc(&h->stage, total) != cudaSuccess) {
            cudaGetLastError();
            return NM_ERR_NOMEM;
        }
        h->stage_bytes = total;
    }
    char* base = (char*)h->stage;
    size_t off = 0;
    auto carve = [&](size_t n) {
        char* p = base + off;
        off += up(n);
        return (void*)p;
    };
    void* dq = carve(in_b);
    void* dk = carve(in_b);
    void* dv = carve(in_b);
    float* da = (float*)carve(gate_b);
    float* de = (float*)carve(gate_b);
    float* db = (float*)carve(gate_b);
    float* dc = (float*)carve(gate_b);
    float* dM0 = (float*)carve(st_b);
    float* dS0 = (float*)carve(st_b);
    float* dMT = (float*)carve(st_b);
    float* dST = (float*)carve(st_b);
    void* dy = carve(out_b);
    cudaStream_t s = (cudaStream_t)stream;
    // Copy / compute overlap: the units are split into groups; group g's inputs go up on one stream, its
    // forward runs on a stream of its own as soon as they have landed (the groups' kernels run side by side,
    // each unit's chain being independent), and its outputs come back on a third stream while later groups'
    // inputs are still being copied.  One group per NM_HOST_GROUP_BYTES of q + y, at least 2 and at most
    // NM_HOST_MAX_GROUPS and the number of units: a group's forward starts once its own inputs are in, so small
    // groups keep the kernels busy behind the copies (and few CTAs in flight at once), while each group costs a
    // dozen copy calls.  Used on the tensor-core path when its kernel needs no workspace (the groups' kernels
    // would share it) and every group's slice of every buffer starts on a 16-byte boundary.
    const size_t by_bytes = (in_b + out_b + NM_HOST_GROUP_BYTES - 1) / NM_HOST_GROUP_BYTES;
    const int groups = (int)std::min<size_t>(std::min<size_t>((size_t)NM_HOST_MAX_GROUPS, units),
                                             std::max<size_t>(2, by_bytes));
    if (h->path == NM_PATH_TC && nm_tc_scratch_bytes(cfg, B, H) == 0 && T > 0 && groups > 1 && (T % 4) == 0 &&
        (P % 4) == 0 && in_b + out_b >= ((size_t)8 << 20)) {
        int prc = ensure_pipe(h);
        if (prc != NM_OK) return prc;
        const size_t in_u = (size_t)T * cfg.d * dtype_bytes(cfg.in_dtype), out_u = (size_t)T * cfg.d * dtype_bytes(cfg.out_dtype);
        const size_t gate_u = (size_t)T * sizeof(float), st_u = P * sizeof(float);
        // the staging buffers carved above, as byte pointers
        char* pq = (char*)dq;
        char* pk = (char*)dk;
        char* pv = (char*)dv;
        char* pa = (char*)da;
        char* pe = (char*)de;
        char* pb = (char*)db;
        char* pc = (char*)dc;
        char* pM0 = (char*)dM0;
        char* pS0 = (char*)dS0;
        char* pMT = (char*)dMT;
        char* pST = (char*)dST;
        char* py = (char*)dy;
        if (cudaEventRecord(h->ev_start, s) != cudaSuccess) return NM_ERR_CUDA;
        // On an error after this point, earlier groups' copies and kernels may still be queued on the
        // handle's streams, reading and writing the caller's host buffers and the staging buffer: wait
        // for all of them before returning, so that nothing outlives the call.
        auto drain = [&](int rc, int used) {
            cudaStreamSynchronize(h->s_in);
            for (int i = 0; i < used; ++i) cudaStreamSynchronize(h->s_comp[i]);
            cudaStreamSynchronize(h->s_out);
            cudaGetLastError();
            return rc;
        };
        if (cudaStreamWaitEvent(h->s_in, h->ev_start, 0) != cudaSuccess) return drain(NM_ERR_CUDA, 0);
        if (cudaStreamWaitEvent(h->s_out, h->ev_start, 0) != cudaSuccess) return drain(NM_ERR_CUDA, 0);
        size_t u0 = 0;
        for (int gi = 0; gi < groups; ++gi) {
            const size_t nu = units / groups + ((size_t)gi < units % groups ? 1 : 0);
            struct Cp { char* dst; const char* src; size_t n; } cin[] = {
                {pq + u0 * in_u, (const char*)q + u0 * in_u, nu * in_u},
                {pk + u0 * in_u, (const char*)k + u0 * in_u, nu * in_u},
                {pv + u0 * in_u, (const char*)v + u0 * in_u, nu * in_u},
                {pa + u0 * gate_u, (const char*)alpha + u0 * gate_u, nu * gate_u},
                {pe + u0 * gate_u, (const char*)eta + u0 * gate_u, nu * gate_u},
                {pb + u0 * gate_u, (const char*)beta + u0 * gate_u, nu * gate_u},
                {pc + u0 * gate_u, need_c ? (const char*)c + u0 * gate_u : nullptr, need_c ? nu * gate_u : 0},
                {pM0 + u0 * st_u, (const char*)M0 + u0 * st_u, nu * st_u},
                {pS0 + u0 * st_u, (const char*)S0 + u0 * st_u, nu * st_u}};
            for (auto& cp : cin)
                if (cp.n && cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyHostToDevice, h->s_in) != cudaSuccess)
                    return drain(NM_ERR_CUDA, gi);
            if (cudaEventRecord(h->ev_in[gi], h->s_in) != cudaSuccess) return drain(NM_ERR_CUDA, gi);
            if (cudaStreamWaitEvent(h->s_comp[gi], h->ev_in[gi], 0) != cudaSuccess) return drain(NM_ERR_CUDA, gi);
            int rc = forward_impl(h, 1, (int)nu, T, pq + u0 * in_u, pk + u0 * in_u, pv + u0 * in_u,
                                  (const float*)(pa + u0 * gate_u), (const float*)(pe + u0 * gate_u),
                                  (const float*)(pb + u0 * gate_u), need_c ? (const float*)(pc + u0 * gate_u) : nullptr,
                                  (const float*)(pM0 + u0 * st_u), (const float*)(pS0 + u0 * st_u), py + u0 * out_u,
                                  (float*)(pMT + u0 * st_u), (float*)(pST + u0 * st_u), nullptr, h->s_comp[gi]);
            if (rc != NM_OK) return drain(rc, gi + 1);
            if (cudaEventRecord(h->ev_done[gi], h->s_comp[gi]) != cudaSuccess) return drain(NM_ERR_CUDA, gi + 1);
            if (cudaStreamWaitEvent(h->s_out, h->ev_done[gi], 0) != cudaSuccess) return drain(NM_ERR_CUDA, gi + 1);
            struct Cp cout_[] = {{(char*)y + u0 * out_u, py + u0 * out_u, nu * out_u},
                                 {(char*)M_T + u0 * st_u, pMT + u0 * st_u, nu * st_u},
                                 {(char*)S_T + u0 * st_u, pST + u0 * st_u, nu * st_u}};
            for (auto& cp : cout_)
                if (cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyDeviceToHost, h->s_out) != cudaSuccess)
                    return drain(NM_ERR_CUDA, gi + 1);
            u0 += nu;
        }
        if (cudaEventRecord(h->ev_end, h->s_out) != cudaSuccess) return drain(NM_ERR_CUDA, groups);
        if (cudaStreamWaitEvent(s, h->ev_end, 0) != cudaSuccess) return drain(NM_ERR_CUDA, groups);
        if (cudaStreamSynchronize(h->s_out) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return NM_ERR_CUDA;
        }
        int st = 0;
        if (cudaMemcpy(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NM_ERR_CUDA;
        if (st != 0) cudaMemset(h->d_status, 0, sizeof(int));
        return st;
    }
    struct Cp { void* dst; const void* src; size_t n; } ins[] = {
        {dq, q, T ? in_b : 0}, {dk, k, T ? in_b : 0}, {dv, v, T ? in_b : 0},
        {da, alpha, T ? gate_b : 0}, {de, eta, T ? gate_b : 0}, {db, beta, T ? gate_b : 0},
        {dc, c, (T && need_c) ? gate_b : 0}, {dM0, M0, st_b}, {dS0, S0, st_b}};
    for (auto& cp : ins)
        if (cp.n && cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return NM_ERR_CUDA;
    int rc = nm_forward(h, B, H, T, T ? dq : nullptr, T ? dk : nullptr, T ? dv : nullptr,
                        T ? da : nullptr, T ? de : nullptr, T ? db : nullptr,
                        (T && need_c) ? dc : nullptr, dM0, dS0, T ? dy : nullptr, dMT, dST, stream);
    if (rc != NM_OK) return rc;
    if (T && cudaMemcpyAsync(y, dy, out_b, cudaMemcpyDeviceToHost, s) != cudaSuccess) return NM_ERR_CUDA;
    if (cudaMemcpyAsync(M_T, dMT, st_b, cudaMemcpyDeviceToHost, s) != cudaSuccess) return NM_ERR_CUDA;
    if (cudaMemcpyAsync(S_T, dST, st_b, cudaMemcpyDeviceToHost, s) != cudaSuccess) return NM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return NM_ERR_CUDA;
    }
    int st = 0;
    if (cudaMemcpy(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NM_ERR_CUDA;
    if (st != 0) cudaMemset(h->d_status, 0, sizeof(int));
    return st;
}

int nm_destroy(nm_handle_t h) {
    if (!h) return NM_OK;
    int rc = NM_OK;
    {
        DeviceGuard g(h->device);
        if (g.ok) {
            if (cudaDeviceSynchronize() != cudaSuccess) {
                cudaGetLastError();
                rc = NM_ERR_CUDA;
            }
            if (h->workspace) cudaFree(h->workspace);
            if (h->stage) cudaFree(h->stage);
            if (h->bwd_ws) cudaFree(h->bwd_ws);
            if (h->pipe_ready) {
                cudaStreamDestroy(h->s_in);
                cudaStreamDestroy(h->s_out);
                cudaEventDestroy(h->ev_start);
                cudaEventDestroy(h->ev_end);
                for (int i = 0; i < NM_HOST_MAX_GROUPS; ++i) {
                    cudaStreamDestroy(h->s_comp[i]);
                    cudaEventDestroy(h->ev_in[i]);
                    cudaEventDestroy(h->ev_done[i]);
                }
            }
            if (h->d_status) cudaFree(h->d_status);
        } else {
            rc = NM_ERR_CUDA;
        }
    }
    free(h);
    return rc;
}

}  // extern "C"
