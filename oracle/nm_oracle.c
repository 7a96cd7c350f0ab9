/*
 * Titans neural long-term memory, forward pass: the plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may load this library.  The
 * product path (libnm.so and its Python binding) never calls it and shares no
 * code, header, table or helper with it.
 *
 * Sources (page title, then section):
 *   [IT] "Titans: Imparare a Memorizzare al Tempo di Test" (lowest.today):
 *        "Meccanismo di Aggiornamento della Memoria"  - gradient step and the
 *            momentum ("surprise") recursion, gradient taken at the previous
 *            weights;
 *        "Meccanismo di Dimenticanza"                 - the (1 - alpha_t) decay;
 *        "Funzione Obiettivo"                         - loss ||M(k) - v||^2;
 *        "Addestramento Parallelizzato"               - chunks of size b,
 *            mini-batch gradient descent inside a chunk.
 *   [JA] "論文解説: Titans — 推論時ニューラルメモリ更新による200万トークン超の長期記憶"
 *        (0h-n0.github.io):
 *        "メモリ読み出し"     - retrieval y_t = M_t(q_t);
 *        "モメンタム機構"     - s_t = beta s_{t-1} + (1 - beta) grad;
 *        "適応的重み減衰"     - theta <- (1 - alpha_t) theta - eta_t s_t;
 *        "ニューラル長期メモリモジュール" - the memory is an MLP whose weights
 *            are the storage.
 *
 * What is computed, per (batch, head), in the pages' order and notation:
 *
 *   for every chunk of b consecutive tokens (the grid restarts at t = 0 of
 *   each call; the last chunk may be shorter):
 *       W0 <- M                         (weights at chunk start; [IT] parallel
 *                                        training: every token of a chunk takes
 *                                        its gradient at these weights)
 *       for every token t of the chunk, in order:
 *           g_t = grad_W ||M_W0(k_t) - v_t||^2      (explicit forward+backward)
 *           S   = beta_t S + c_t g_t                 (momentum over surprise)
 *           M   = (1 - alpha_t) M - eta_t S          (forgetting + step)
 *           y_t = M(q_t)                             (retrieval after the update)
 *   M_T = M, S_T = S.
 *
 * The momentum coefficient c_t is ONE (c_t = 1), ONE_MINUS_BETA (c_t = 1 -
 * beta_t, the form of [JA] "モメンタム機構") or PER_TOKEN (c_t read from an
 * array; with eta = 1 and the sign of S flipped this is the form of [IT]).
 *
 * Memories:
 *   LINEAR: M(x) = M x, M in R^{d x d}, row-major [out][in].
 *   MLP2  : M(x) = W2 silu(W1 x), W1 in R^{h x d}, W2 in R^{d x h}, no bias;
 *           parameters packed as W1 (row-major h x d) followed by W2
 *           (row-major d x h).
 *           With `layers` = L > 2 (deeper memories, [JA] "ニューラル長期メモリモジュール":
 *           the memory is an MLP of L_M >= 1 layers; [IT] reports that depth
 *           helps): M(x) = W_L silu(W_{L-1} ... silu(W1 x)), W1 h x d,
 *           W2 .. W_{L-1} h x h, W_L d x h, packed in that order; silu after
 *           every layer but the last.
 *
 * Readings where the pages are silent or disagree:
 *   - the squared norm has no 1/2, so grad = 2 (M(k) - v) ... (kept);
 *   - retrieval uses the weights after token t's update (inclusive);
 *   - gates are one scalar per token per head, shared by every parameter.
 *
 * Two extensions, both optional:
 *   - the Huber loss of the YAAD variant ([JA] "MIRASフレームワーク", "3つの変種";
 *     es.news.hada.io, "Modelos basados en MIRAS"), which the pages name
 *     without a formula or threshold.  Reading: element-wise on the residual
 *     r = M(k) - v, with a caller-given threshold delta, scaled to agree with
 *     ||r||^2 inside it:  rho(r) = r^2 for |r| <= delta, 2 delta |r| - delta^2
 *     beyond, so d rho / d r = 2 clip(r, -delta, delta).  delta = +inf is the
 *     squared loss exactly.
 *   - the surprise of each token ([JA] "技術的詳細", "Surprise機構": the norm of the
 *     loss gradient with respect to the memory's parameters), read as the
 *     Frobenius norm over all parameters of g_t, the gradient the update uses
 *     (at the chunk-start weights).
 *
 * No blocking, no fusion, no reordering: a reader can check each loop against
 * the equations above.  Everything is double precision.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define OR_LINEAR 0
#define OR_MLP2 1

#define OR_C_ONE 0
#define OR_C_ONE_MINUS_BETA 1
#define OR_C_PER_TOKEN 2

#define OR_LOSS_L2 0
#define OR_LOSS_HUBER 1

/* d rho / d r: 2 r (squared loss) or 2 clip(r, -delta, delta) (Huber). */
static double or_dloss(int loss, double delta, double r) {
    if (loss == OR_LOSS_HUBER) {
        if (r > delta) return 2.0 * delta;
        if (r < -delta) return -2.0 * delta;
    }
    return 2.0 * r;
}

static double or_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }
static double or_silu(double z) { return z * or_sigmoid(z); }
/* d/dz [z * sigmoid(z)] = sigmoid(z) + z sigmoid(z) (1 - sigmoid(z)) */
static double or_dsilu(double z) {
    double s = or_sigmoid(z);
    return s * (1.0 + z * (1.0 - s));
}

/* Number of parameters of one memory (layers: MLP depth, >= 2; ignored for LINEAR). */
long oracle_param_count(int kind, int d, int h, int layers) {
    if (kind == OR_LINEAR) return (long)d * d;
    if (kind == OR_MLP2 && layers >= 2) return 2L * h * d + (long)(layers - 2) * h * h;
    return -1;
}

/* y = M_W(x).  work must hold 2h doubles for MLP2. */
void oracle_memory_apply(int kind, int d, int h, int layers, const double* W,
                         const double* x, double* y, double* work) {
    if (kind == OR_LINEAR) {
        for (int o = 0; o < d; ++o) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += W[(long)o * d + i] * x[i];
            y[o] = acc;
        }
        return;
    }
    double* cur = work;       /* h: activation of the current layer */
    double* nxt = work + h;   /* h */
    const double* W1 = W;     /* h x d */
    for (int j = 0; j < h; ++j) {
        double z = 0.0;
        for (int i = 0; i < d; ++i) z += W1[(long)j * d + i] * x[i];
        cur[j] = or_silu(z);
    }
    const double* Wl = W + (long)h * d;
    for (int l = 2; l < layers; ++l) {   /* hidden-to-hidden layers, h x h */
        for (int j = 0; j < h; ++j) {
            double z = 0.0;
            for (int i = 0; i < h; ++i) z += Wl[(long)j * h + i] * cur[i];
            nxt[j] = or_silu(z);
        }
        double* t = cur; cur = nxt; nxt = t;
        Wl += (long)h * h;
    }
    for (int o = 0; o < d; ++o) {        /* last layer W_L, d x h, no activation */
        double acc = 0.0;
        for (int j = 0; j < h; ++j) acc += Wl[(long)o * h + j] * cur[j];
        y[o] = acc;
    }
}

/* The associative loss l(W; k, v) = ||M_W(k) - v||_2^2 ([IT] "Funzione
 * Obiettivo"), or with loss = OR_LOSS_HUBER the sum of rho(r_o) above.
 * work: d + h doubles. */
double oracle_loss(int kind, int d, int h, int layers, int loss, double delta,
                   const double* W, const double* k, const double* v, double* work) {
    double* yhat = work;
    oracle_memory_apply(kind, d, h, layers, W, k, yhat, work + d);
    double acc = 0.0;
    for (int o = 0; o < d; ++o) {
        double r = yhat[o] - v[o];
        if (loss == OR_LOSS_HUBER && fabs(r) > delta)
            acc += 2.0 * delta * fabs(r) - delta * delta;
        else
            acc += r * r;
    }
    return acc;
}

/* g = grad_W l(W; k, v), by an explicit forward and backward pass.
 * work: (2 layers + 2) h + 2d doubles. */
void oracle_grad(int kind, int d, int h, int layers, int loss, double delta,
                 const double* W, const double* k, const double* v, double* g,
                 double* work) {
    if (kind == OR_LINEAR) {
        /* l = sum_o rho((M k - v)[o]),  rho(r) = r^2 for the squared loss
         * dl/dM[o][i] = rho'((M k - v)[o]) k[i]                              */
        double* e = work;
        for (int o = 0; o < d; ++o) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += W[(long)o * d + i] * k[i];
            e[o] = or_dloss(loss, delta, acc - v[o]);
        }
        for (int o = 0; o < d; ++o)
            for (int i = 0; i < d; ++i) g[(long)o * d + i] = e[o] * k[i];
        return;
    }
    const int L = layers;
    /* per hidden layer l = 1 .. L-1: pre-activation z_l and activation a_l (h each) */
    double* z = work;                         /* (L-1) x h */
    double* a = work + (long)(L - 1) * h;     /* (L-1) x h */
    double* da = work + 2L * (L - 1) * h;     /* h: dl/da of the current layer */
    double* dz = da + h;                      /* h: dl/dz of the current layer */
    double* e = dz + h;                       /* d */
    /* offsets of each layer's weights in W (and of its gradient in g) */
    long off[64];
    off[1] = 0;
    off[2] = (long)h * d;
    for (int l = 3; l <= L; ++l) off[l] = off[l - 1] + (long)h * h;
    /* forward: z_1 = W1 k, a_l = silu(z_l), z_l = W_l a_{l-1}, yhat = W_L a_{L-1} */
    for (int l = 1; l < L; ++l) {
        const double* Wl = W + off[l];
        const int in = l == 1 ? d : h;
        const double* x = l == 1 ? k : a + (long)(l - 2) * h;
        for (int j = 0; j < h; ++j) {
            double acc = 0.0;
            for (int i = 0; i < in; ++i) acc += Wl[(long)j * in + i] * x[i];
            z[(long)(l - 1) * h + j] = acc;
            a[(long)(l - 1) * h + j] = or_silu(acc);
        }
    }
    const double* WL = W + off[L];
    const double* aL = a + (long)(L - 2) * h;
    /* dl/dyhat = rho'(yhat - v): 2 (yhat - v) for the squared loss */
    for (int o = 0; o < d; ++o) {
        double acc = 0.0;
        for (int j = 0; j < h; ++j) acc += WL[(long)o * h + j] * aL[j];
        e[o] = or_dloss(loss, delta, acc - v[o]);
    }
    /* dl/dW_L[o][j] = e[o] a_{L-1}[j] */
    for (int o = 0; o < d; ++o)
        for (int j = 0; j < h; ++j) g[off[L] + (long)o * h + j] = e[o] * aL[j];
    /* dl/da_{L-1}[j] = sum_o W_L[o][j] e[o] */
    for (int j = 0; j < h; ++j) {
        double acc = 0.0;
        for (int o = 0; o < d; ++o) acc += WL[(long)o * h + j] * e[o];
        da[j] = acc;
    }
    /* down the hidden layers: dl/dz_l = dl/da_l silu'(z_l); dl/dW_l = dl/dz_l x_{l-1}^T;
     * dl/da_{l-1} = W_l^T dl/dz_l */
    for (int l = L - 1; l >= 1; --l) {
        for (int j = 0; j < h; ++j) dz[j] = da[j] * or_dsilu(z[(long)(l - 1) * h + j]);
        const int in = l == 1 ? d : h;
        const double* x = l == 1 ? k : a + (long)(l - 2) * h;
        for (int j = 0; j < h; ++j)
            for (int i = 0; i < in; ++i) g[off[l] + (long)j * in + i] = dz[j] * x[i];
        if (l > 1) {
            const double* Wl = W + off[l];
            for (int i = 0; i < h; ++i) {
                double acc = 0.0;
                for (int j = 0; j < h; ++j) acc += Wl[(long)j * h + i] * dz[j];
                da[i] = acc;
            }
        }
    }
}

/* One (batch, head) unit.  Pointers are already offset to the unit. */
static void oracle_unit(int kind, int d, int h, int layers, int chunk, int c_mode, int loss,
                        double delta, int T, const double* q, const double* k,
                        const double* v, const double* alpha, const double* eta,
                        const double* beta, const double* c, const double* M0,
                        const double* S0, double* y, double* MT, double* ST,
                        double* surprise) {
    long P = oracle_param_count(kind, d, h, layers);
    double* M = (double*)malloc(sizeof(double) * P);
    double* S = (double*)malloc(sizeof(double) * P);
    double* W0 = (double*)malloc(sizeof(double) * P);
    double* g = (double*)malloc(sizeof(double) * P);
    double* work = (double*)malloc(sizeof(double) * ((2 * (long)layers + 2) * h + 2 * (long)d + 8));
    memcpy(M, M0, sizeof(double) * P);
    memcpy(S, S0, sizeof(double) * P);
    for (int t0 = 0; t0 < T; t0 += chunk) {
        int t1 = t0 + chunk < T ? t0 + chunk : T;
        memcpy(W0, M, sizeof(double) * P); /* chunk-start weights */
        for (int t = t0; t < t1; ++t) {
            oracle_grad(kind, d, h, layers, loss, delta, W0, k + (long)t * d, v + (long)t * d, g, work);
            if (surprise) {
                double n2 = 0.0;
                for (long p = 0; p < P; ++p) n2 += g[p] * g[p];
                surprise[t] = sqrt(n2);
            }
            double ct = 1.0;
            if (c_mode == OR_C_ONE_MINUS_BETA) ct = 1.0 - beta[t];
            else if (c_mode == OR_C_PER_TOKEN) ct = c[t];
            for (long p = 0; p < P; ++p) S[p] = beta[t] * S[p] + ct * g[p];
            for (long p = 0; p < P; ++p) M[p] = (1.0 - alpha[t]) * M[p] - eta[t] * S[p];
            oracle_memory_apply(kind, d, h, layers, M, q + (long)t * d, y + (long)t * d, work);
        }
    }
    memcpy(MT, M, sizeof(double) * P);
    memcpy(ST, S, sizeof(double) * P);
    free(M); free(S); free(W0); free(g); free(work);
}

/*
 * Full forward over B x H independent (batch, head) units.
 *   q, k, v, y : [B, H, T, d]      alpha, eta, beta, c, surprise : [B, H, T]
 *   M0, S0, MT, ST : [B, H, P]     (c may be NULL unless c_mode == PER_TOKEN;
 *                                   surprise may be NULL)
 *   layers: MLP depth L >= 2 (ignored for LINEAR).
 *   loss: OR_LOSS_L2 or OR_LOSS_HUBER with threshold delta > 0.
 * Returns 0, or -1 on a bad argument.  Units run in parallel with OpenMP;
 * each unit's arithmetic is sequential and identical to a one-thread run.
 */
int oracle_forward(int kind, int d, int h, int layers, int chunk, int c_mode, int loss,
                   double delta, int B, int H, int T, const double* q,
                   const double* k, const double* v, const double* alpha,
                   const double* eta, const double* beta, const double* c,
                   const double* M0, const double* S0, double* y, double* MT,
                   double* ST, double* surprise) {
    if ((kind != OR_LINEAR && kind != OR_MLP2) || d <= 0 || chunk <= 0 ||
        B < 0 || H < 0 || T < 0)
        return -1;
    if (loss != OR_LOSS_L2 && !(loss == OR_LOSS_HUBER && delta > 0.0)) return -1;
    if (kind == OR_MLP2 && (h <= 0 || layers < 2 || layers > 63)) return -1;
    if (c_mode == OR_C_PER_TOKEN && c == NULL) return -1;
    long P = oracle_param_count(kind, d, h, layers);
    long units = (long)B * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long u = 0; u < units; ++u) {
        oracle_unit(kind, d, h, layers, chunk, c_mode, loss, delta, T, q + u * T * d,
                    k + u * T * d, v + u * T * d, alpha + u * T, eta + u * T,
                    beta + u * T, c ? c + u * T : NULL, M0 + u * P, S0 + u * P,
                    y + u * T * d, MT + u * P, ST + u * P,
                    surprise ? surprise + u * T : NULL);
    }
    return 0;
}
