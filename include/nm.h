/*
 * nm.h - C ABI of the Titans neural long-term memory forward pass (B300, sm_103a).
 *
 * The operation ("Titans: Imparare a Memorizzare al Tempo di Test",
 * lowest.today; sections "Meccanismo di Aggiornamento della Memoria",
 * "Meccanismo di Dimenticanza", "Funzione Obiettivo", "Addestramento
 * Parallelizzato"; and the 0h-n0.github.io Titans explainer, sections
 * "メモリ読み出し", "モメンタム機構", "適応的重み減衰"):
 *
 *   per (batch b, head h), for every chunk of `chunk` consecutive tokens
 *   (the chunk grid starts at token 0 of each call; the last chunk may be
 *   shorter), with W0 the memory at chunk start:
 *       g_t = grad_W || M_W0(k_t) - v_t ||^2          (no 1/2: factor 2 kept;
 *                                                      or the Huber loss, NM_LOSS_HUBER)
 *       S   = beta_t S + c_t g_t                       (momentum over surprise)
 *       M   = (1 - alpha_t) M - eta_t S                (forgetting + step)
 *       y_t = M(q_t)                                   (retrieval after the update)
 *
 *   memory kinds:  NM_LINEAR  M(x) = M x,  M in R^{d x d}, row-major [out][in]
 *                  NM_MLP2    M(x) = W2 silu(W1 x), W1 in R^{hidden x d},
 *                             W2 in R^{d x hidden}, no bias; parameters packed
 *                             as W1 (row-major) followed by W2 (row-major).
 *   P (parameters per unit) = d*d (LINEAR) or 2*hidden*d (MLP2; plus
 *   (layers - 2)*hidden^2 for a deeper MLP2, see nm_config.layers).
 *
 * The library computes this in the chunked-parallel form (matrix products
 * plus a decay / momentum scan inside each chunk), with every unit's state
 * kept on chip by one persistent kernel over the sequence.
 *
 * Threading: a handle may be used from one host thread at a time.
 * All device entry points are asynchronous on the caller's stream.
 */
#ifndef NM_H
#define NM_H

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values of every entry point) ------------------ */
#define NM_OK                  0
#define NM_ERR_ARG             1  /* null pointer, bad size, bad enum          */
#define NM_ERR_ALIGN           2  /* a pointer is not 16-byte aligned          */
#define NM_ERR_UNSUPPORTED     3  /* (kind, d, hidden, chunk, dtype) not built */
#define NM_ERR_ALIAS           4  /* buffers overlap other than M_T==M0, S_T==S0 */
#define NM_ERR_CUDA            5  /* a CUDA runtime call failed                */
#define NM_ERR_NOMEM           6  /* host or device allocation failed          */
#define NM_ERR_DEVICE_TIMEOUT  7  /* a bounded on-device wait gave up          */
#define NM_ERR_DEVICE_CHECK    8  /* an on-device consistency check failed     */
#define NM_ERR_TOO_LARGE       9  /* call needs more than the fixed no-alloc workspace */

/* ---- configuration enums ------------------------------------------------ */
#define NM_LINEAR 0
#define NM_MLP2   1

#define NM_F32  0
#define NM_BF16 1

/* momentum coefficient c_t in S = beta_t S + c_t g_t */
#define NM_C_ONE            0  /* c_t = 1                                   */
#define NM_C_ONE_MINUS_BETA 1  /* c_t = 1 - beta_t (explainer, "モメンタム機構") */
#define NM_C_PER_TOKEN      2  /* c_t read from the `c` array (with eta = 1 and
                                  S negated this is the form of "Meccanismo di
                                  Aggiornamento della Memoria")             */

/* the associative loss (its gradient drives the update):
 *   NM_LOSS_L2     l = ||M(k) - v||^2                   ("Funzione Obiettivo")
 *   NM_LOSS_HUBER  l = sum_o rho(r_o), r = M(k) - v, rho(r) = r^2 for |r| <= delta,
 *                  2 delta |r| - delta^2 beyond: the Huber loss of the YAAD variant
 *                  (0h-n0.github.io explainer, "MIRASフレームワーク", "3つの変種";
 *                  es.news.hada.io, "Modelos basados en MIRAS"), which the pages
 *                  name without formula or threshold.  Element-wise, scaled to equal
 *                  the squared loss inside the threshold, so e = 2 clip(r, -delta, delta)
 *                  replaces e = 2 r.                                              */
#define NM_LOSS_L2    0
#define NM_LOSS_HUBER 1

/* kernel family; AUTO picks the tensor-core path for bf16 inputs when one is
 * built for the shape, else the fp32 FFMA path */
#define NM_PATH_AUTO 0
#define NM_PATH_SIMT 1  /* fp32 FFMA kernels: any supported shape, fp32 or bf16 in */
#define NM_PATH_TC   2  /* tcgen05 tensor-core kernels: bf16 in, fp32 state      */

typedef struct nm_config {
    int kind;       /* NM_LINEAR | NM_MLP2                                    */
    int d;          /* key / value / query width: 16, 32, 64 or 128          */
    int hidden;     /* MLP2 hidden width (multiple of 32, <= 1024); ignored for LINEAR */
    int chunk;      /* chunk size b, 1..256                                   */
    int in_dtype;   /* dtype of q, k, v: NM_F32 | NM_BF16                    */
    int out_dtype;  /* dtype of y: NM_F32 | NM_BF16                          */
    int c_mode;     /* NM_C_ONE | NM_C_ONE_MINUS_BETA | NM_C_PER_TOKEN       */
    int path;       /* NM_PATH_AUTO | NM_PATH_SIMT | NM_PATH_TC              */
    int loss;       /* NM_LOSS_L2 | NM_LOSS_HUBER (a zeroed config means L2)  */
    float huber_delta; /* Huber threshold delta: finite and > 0 for NM_LOSS_HUBER;
                          ignored for NM_LOSS_L2                                 */
    int layers;     /* NM_MLP2 depth L, 2..NM_MAX_LAYERS (0 means 2); must be 0
                       for NM_LINEAR.  L > 2 is the deeper memory
                       W_L silu(W_{L-1} ... silu(W1 x)): W1 hidden x d,
                       W2 .. W_{L-1} hidden x hidden, W_L d x hidden, packed in
                       that order (P = 2 hidden d + (L - 2) hidden^2).  On
                       NM_PATH_TC (tf32 tensor-core kernel) for bf16 inputs,
                       d = 64 or 128, hidden a multiple of 64 up to 512 and
                       chunk <= 64, with a per-unit workspace the handle
                       allocates; every shape on the fp32 FFMA kernels        */
} nm_config;

#define NM_MAX_LAYERS 16

typedef struct nm_handle* nm_handle_t;

/*
 * nm_create - validate `cfg` and bind a handle to CUDA device `device`.
 *   The handle owns: a device status word (bounded waits and on-device checks
 *   report into it), and a device workspace that grows on demand in
 *   nm_forward (so the first call at a larger B*H allocates).
 *   Returns NM_ERR_ARG for null pointers or bad enums, NM_ERR_UNSUPPORTED when
 *   no kernel is built for the shape, NM_ERR_CUDA / NM_ERR_NOMEM on failures.
 *   *out is set only on NM_OK.
 */
int nm_create(const nm_config* cfg, int device, nm_handle_t* out);

/*
 * nm_forward - one forward call over B x H independent units of T tokens.
 *   All pointers are DEVICE pointers on the handle's device, owned by the
 *   caller, contiguous, 16-byte aligned:
 *     q, k, v   [B, H, T, d]  in_dtype
 *     alpha, eta, beta [B, H, T] fp32   (alpha in [0, 1] forgets, eta is the
 *                                        step, beta the momentum decay)
 *     c         [B, H, T] fp32, used only when c_mode == NM_C_PER_TOKEN
 *                                       (must be NULL otherwise)
 *     M0, S0    [B, H, P] fp32  memory and momentum at token 0
 *     y         [B, H, T, d]  out_dtype   (written)
 *     M_T, S_T  [B, H, P] fp32  memory and momentum after token T-1 (written)
 *   M_T == M0 and / or S_T == S0 (exact aliasing) is allowed, for streaming
 *   one long sequence through successive calls; any other overlap between an
 *   output and any buffer returns NM_ERR_ALIAS.
 *   `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   B*H == 0 is a no-op; T == 0 copies M0, S0 into M_T, S_T.
 *   Host-side failures return an error with nothing launched.  Device-side
 *   failures (bounded waits, on-device checks) are recorded in the handle's
 *   status word and returned by nm_synchronize.
 */
int nm_forward(nm_handle_t h, int B, int H, int T,
               const void* q, const void* k, const void* v,
               const float* alpha, const float* eta, const float* beta,
               const float* c, const float* M0, const float* S0,
               void* y, float* M_T, float* S_T, void* stream);

/*
 * nm_forward_surprise - nm_forward that also writes each token's surprise,
 *   the norm of the loss gradient with respect to the memory's parameters
 *   (0h-n0.github.io explainer, "技術的詳細", "Surprise機構"):
 *     surprise [B, H, T] fp32 (DEVICE, caller-owned, 16-byte aligned, written)
 *       = || g_t ||_F over all parameters, with g_t the gradient the update
 *         uses: at the chunk-start weights, of the configured loss.
 *   Linear memory: ||e_t|| ||k_t||; MLP2: sqrt(||delta_t||^2 ||k_t||^2 +
 *   ||e_t||^2 ||silu(W1 k_t)||^2).  Tokens are computed from the same fp32 e
 *   (and delta) as the update, before any rounding to bf16.
 *   Everything else is nm_forward's contract; `surprise` must not overlap any
 *   other buffer (NM_ERR_ALIAS) and must not be NULL (NM_ERR_ARG).
 *   Every kernel family writes it (the tensor-core kernels through a variant
 *   compiled for it, launched only when `surprise` is set).
 */
int nm_forward_surprise(nm_handle_t h, int B, int H, int T,
                        const void* q, const void* k, const void* v,
                        const float* alpha, const float* eta, const float* beta,
                        const float* c, const float* M0, const float* S0,
                        void* y, float* M_T, float* S_T, float* surprise, void* stream);

/*
 * nm_forward_gated - nm_forward with the memory's output combined with an
 *   attention branch's output by the Memory-as-Gate rule (0h-n0.github.io
 *   explainer, "3つのアーキテクチャ変種", MAG: o_t = sigmoid(y_t^mem) (.)
 *   y_t^attn; "Titans: Imparare a Memorizzare al Tempo di Test", "Varianti
 *   dell'Architettura Titans", "Memory as Gate (MAG)": the two branches'
 *   outputs combined by a gate):
 *     y_attn [B, H, T, d] out_dtype (DEVICE, caller-owned, 16-byte aligned,
 *            read): the other branch's output (e.g. sliding-window attention)
 *     o      [B, H, T, d] out_dtype (written) = sigmoid(y) * y_attn element by
 *            element, y the memory's retrieval M_t(q_t) that nm_forward writes
 *   The sigmoid is 1 / (1 + exp(-y)), applied to y in fp32 before the output
 *   is rounded.  y itself is not written.  M_T and S_T are nm_forward's, bit
 *   for bit.  o == y_attn (exact aliasing) is allowed, gating the attention
 *   output in place; any other overlap of y_attn with an output returns
 *   NM_ERR_ALIAS.  y_attn must not be NULL when T > 0 (NM_ERR_ARG).
 *   Everything else is nm_forward's contract.  Every kernel family writes it
 *   from its retrieval epilogue.
 */
int nm_forward_gated(nm_handle_t h, int B, int H, int T,
                     const void* q, const void* k, const void* v,
                     const float* alpha, const float* eta, const float* beta,
                     const float* c, const float* M0, const float* S0,
                     const void* y_attn, void* o, float* M_T, float* S_T, void* stream);

/*
 * nm_backward - gradients of a loss of the forward's outputs with respect to
 *   every input, for training what surrounds the memory ("Titans: Imparare a
 *   Memorizzare al Tempo di Test", "Addestramento Parallelizzato": the inner
 *   loop is written with matrix products so that the outer loop trains
 *   fast).  Given the upstream gradients of L with respect to y, M_T and S_T,
 *   it writes dL/d(every input) of nm_forward on the same inputs:
 *     inputs: q, k, v, alpha, eta, beta, c, M0, S0 as for nm_forward (DEVICE)
 *     Gy      [B, H, T, d] fp32   dL/dy
 *     GM, GS  [B, H, P]    fp32   dL/dM_T, dL/dS_T
 *     outputs (fp32, written): dq, dk, dv [B, H, T, d]; dalpha, deta, dbeta
 *     [B, H, T]; dc [B, H, T] for NM_C_PER_TOKEN (must be NULL otherwise;
 *     with NM_C_ONE_MINUS_BETA the dependence of c on beta is in dbeta);
 *     dM0, dS0 [B, H, P].
 *   Memory kinds: NM_LINEAR and the 2-layer NM_MLP2 (d 16..128, hidden <= 1024
 *   a multiple of 32, chunk <= 256, fp32 or bf16 inputs, either loss); deeper
 *   MLP memories return NM_ERR_UNSUPPORTED.  The gradient is that of
 *   the chunked forward in fp32 arithmetic: the call first runs the forward
 *   once more on the fp32 FFMA kernel (on an NM_PATH_TC handle of the linear
 *   memory with d = 128, chunk 64, the tcgen05 forward kernel, whose states
 *   carry its bf16 operand rounding), recording every chunk's start state in
 *   a handle-owned workspace (B*H*ceil(T/chunk)*2*P floats plus per-unit
 *   scratch; it grows on demand, so a first call at a larger size
 *   allocates), then sweeps the chunks from last to first.  The sweep's
 *   chunk-sized contractions run as fp32 FFMA products, or, on a handle
 *   created with path NM_PATH_TC (bf16 inputs, a shape the forward's
 *   tensor-core kernels take), as tcgen05 tf32 products (fp32 accumulation;
 *   gradients then within the bf16-input tolerances instead of fp32 ones,
 *   and a timed-out product wait is reported by nm_synchronize as
 *   NM_ERR_DEVICE_TIMEOUT).  No output may overlap any input or another
 *   output (NM_ERR_ALIAS).  Asynchronous on `stream`; host-side errors return
 *   with nothing launched.
 */
int nm_backward(nm_handle_t h, int B, int H, int T,
                const void* q, const void* k, const void* v,
                const float* alpha, const float* eta, const float* beta,
                const float* c, const float* M0, const float* S0,
                const float* Gy, const float* GM, const float* GS,
                float* dq, float* dk, float* dv,
                float* dalpha, float* deta, float* dbeta, float* dc,
                float* dM0, float* dS0, void* stream);

/*
 * nm_forward_host - the same operation on HOST buffers (same layouts).
 *   Copies the inputs to the handle's device (into handle-owned buffers that
 *   grow on demand), runs nm_forward on `stream`, copies y, M_T, S_T back and
 *   synchronises the stream before returning.  Pinned host memory gives
 *   asynchronous copies; pageable memory works but is slower.  On the
 *   tensor-core path, when one input tensor plus y hold 8 MiB or more, the
 *   units run in groups (one per 16 MiB of q + y, at least 2, at most 16 and
 *   at most one per unit), each group's forward starting on a stream of its
 *   own as soon as its inputs are in, its outputs copied back while later
 *   groups' inputs are still going up; the results equal nm_forward's bit
 *   for bit, and each group counts as one launch in nm_launch_count.
 *   Returns the first host-side error, or the device status word as
 *   nm_synchronize would.
 */
int nm_forward_host(nm_handle_t h, int B, int H, int T,
                    const void* q, const void* k, const void* v,
                    const float* alpha, const float* eta, const float* beta,
                    const float* c, const float* M0, const float* S0,
                    void* y, float* M_T, float* S_T, void* stream);

/*
 * nm_synchronize - wait for all work on the device, then return and clear
 *   the handle's device status word (NM_OK, NM_ERR_DEVICE_TIMEOUT,
 *   NM_ERR_DEVICE_CHECK) or NM_ERR_CUDA if the device reported an error.
 */
int nm_synchronize(nm_handle_t h);

/*
 * nm_destroy - free everything the handle owns (after synchronising its
 *   device).  NULL is accepted and ignored.
 */
int nm_destroy(nm_handle_t h);

/* nm_status_string - static, never-NULL description of a status code. */
const char* nm_status_string(int status);

/*
 * nm_selected_path - the kernel family nm_forward will use for this handle
 *   (NM_PATH_SIMT or NM_PATH_TC), or a negative status for a bad handle.
 */
int nm_selected_path(nm_handle_t h);

/*
 * nm_launch_count - number of kernels this handle has launched so far
 *   (monotonic; used to count launches inside a timed region).
 */
long long nm_launch_count(nm_handle_t h);

/*
 * nm_inject_missing_load - test hook for the device-side failure detection.
 *   Arms the handle so that its next nm_forward launches the tensor-core
 *   kernel without loading the first chunk's tiles.  The kernel's bounded wait
 *   for those tiles (2 s) then expires; the kernel records
 *   NM_ERR_DEVICE_TIMEOUT in the handle's status word, skips the rest of its
 *   tensor-core work and exits normally, leaving the CUDA context usable.  That
 *   call's outputs are undefined; nm_synchronize returns the status.  The hook
 *   is consumed by that one call.  Not part of the method (the pages have no
 *   counterpart): it exists so that tests can check the timeout path without
 *   faulting a GPU.
 *   Returns NM_ERR_ARG for a NULL handle, NM_ERR_UNSUPPORTED when the handle
 *   uses the fp32 FFMA kernels (they have no waits).
 */
int nm_inject_missing_load(nm_handle_t h);

/*
 * nm_forward_mlp2_noalloc - the MLP2 forward without any allocation.
 *   The paper has no counterpart to this entry point; it exists for callers
 *   that cannot call cudaMalloc when they run the layer: a host that has
 *   reserved the whole device for its own memory pool (a side allocation
 *   would fail or fragment it), or a latency-critical loop that cannot
 *   afford cudaMalloc's implicit device-wide synchronisation.  It needs no
 *   handle (nm_create allocates) and calls no cudaMalloc, cudaFree or
 *   allocating library routine.
 *   Arguments, layouts, aliasing rules and host-side errors are those of
 *   nm_forward, with the configuration passed directly; cfg->kind must be
 *   NM_MLP2 and cfg->path NM_PATH_AUTO or NM_PATH_SIMT (the fp32 FFMA
 *   kernel runs).  The work runs on the CURRENT device, on `stream`.
 *   Workspace: one file-scope device array of NM_NOALLOC_SCRATCH_BYTES,
 *   present on every GPU that loads this library until the process exits.
 *   A call needing more than that (B*H units of
 *   4*(2 r4(b^2) + 2 r4(b) + 4bd + (3L - 1)bh + 2P) bytes each for an L-layer
 *   memory (L = 2 by default), with r4 rounding up to a multiple of 4 and P
 *   the parameter count) returns NM_ERR_TOO_LARGE with nothing launched.  Every call looks up the array's device address on the
 *   current device (cudaGetSymbolAddress); the first call on a device may load
 *   the library's module there, so make that first call before any stream
 *   capture.  The address is not cached, so calls stay correct after
 *   cudaDeviceReset (which may move the array).  Every call shares the array, which keeps
 *   the previous call's contents (the kernel writes each workspace element
 *   before reading it, so nothing needs clearing); calls whose kernels overlap
 *   on the GPU race on it, so the caller must order them.  Bounded-wait
 *   status is not reported (this kernel has no waits).
 */
#define NM_NOALLOC_SCRATCH_BYTES (16u << 20)
int nm_forward_mlp2_noalloc(const nm_config* cfg, int B, int H, int T,
                            const void* q, const void* k, const void* v,
                            const float* alpha, const float* eta, const float* beta,
                            const float* c, const float* M0, const float* S0,
                            void* y, float* M_T, float* S_T, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* NM_H */
