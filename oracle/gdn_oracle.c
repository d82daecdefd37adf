/* gdn_oracle.c - reference implementation of the GDN speculative tree-verify
 * step: conv tree step, gated delta-rule tree recurrence, replay-log commit.
 *
 * TEST INFRASTRUCTURE.  This file is the oracle the CUDA library is checked
 * against.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It is deliberately plain: single-threaded loops, double
 * arithmetic, no blocking, no fusion, no reordering beyond what each step's
 * definition states.  Compile with -O2 -ffp-contract=off and no fast-math.
 *
 * Sources, by page title and section:
 *  [P1] lucebox PR #707 "perf(qwen35): fuse the DFlash2 concurrent verify Gated
 *       DeltaNet route" - Optimizations (fused convolution preparation,
 *       read-only mapped recurrence, gate preparation inside the recurrence)
 *       and Validation (persistent state unchanged by verify).
 *  [P2] TensorSharp PR #175 "Feature/support dflash2" - the on-device commit of
 *       the accepted prefix replacing restore-and-re-forward.
 *  [P3] lucebox PR #625 "qwen35: DSpark speculative decoding" - raw-gate GDN:
 *       sigmoid(beta) and softplus(alpha + dt_bias) * A inside the kernel; one
 *       l2_norm over the q|k slab; q/k heads broadcast to value heads.
 *  [P4] lucebox PR #659 "perf(qwen38): various DFlash2 optimizations
 *       concurrency C1-C5" - Summary item 3: replay rows of width 257 at state
 *       size 128 (= k_hat 128 | u 128 | decay 1); transaction preflight.
 *  [P5] llama-cpp-bonsai "llama-cpp-bonsai-gdn-conv.patch" - ssm_conv_concat
 *       kernel: conv input column p is history column p for p < d_conv - 1,
 *       else token p - (d_conv - 1); the sum runs over taps j = 0..3 in order
 *       with tap 3 on the newest column, then SiLU.
 *  [GDN] Yang, Kautz, Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with
 *       Delta Rule" (ICLR 2025): S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,
 *       o_t = S_t q_t.
 *
 * Readings taken where the pages are silent (each is listed with its reason
 * in the design notes): q/k/v channel order q | k | v; value head h uses k-head
 * floor(h / (h_v / h_k)); L2 norm x / sqrt(sum x^2 + 1e-6); softplus linear
 * above 20; replay row = k_hat | u | decay with u = beta (v - decay S_parent k_hat);
 * a node with parent -1 starts from the slot's state and history.
 */
#include "gdn_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define L2_EPS 1e-6

static double silu(double x) { return x / (1.0 + exp(-x)); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

static int conv_channels(const gdn_oracle_dims *dm) {
    return 2 * dm->h_k * dm->d + dm->h_v * dm->d;
}

static int check_dims(const gdn_oracle_dims *dm) {
    if (dm->n_seqs < 0 || dm->n_nodes < 0 || dm->n_slots <= 0 || dm->h_k <= 0 ||
        dm->h_v <= 0 || dm->d <= 0 || dm->d_conv < 2 || dm->h_v % dm->h_k != 0)
        return ORACLE_BAD_DIMS;
    return ORACLE_OK;
}

static int check_offsets(const gdn_oracle_dims *dm, const int *node_off) {
    if (node_off[0] != 0) return ORACLE_BAD_NODE_OFF;
    for (int s = 0; s < dm->n_seqs; ++s)
        if (node_off[s + 1] < node_off[s]) return ORACLE_BAD_NODE_OFF;
    if (node_off[dm->n_seqs] != dm->n_nodes) return ORACLE_BAD_NODE_OFF;
    return ORACLE_OK;
}

/* parents are local indices; a node's parent precedes it (topological order) */
static int check_parents(const int *parents, int n0, int ns) {
    for (int i = 0; i < ns; ++i) {
        int p = parents[n0 + i];
        if (p < -1 || p >= i) return ORACLE_BAD_PARENT;
    }
    return ORACLE_OK;
}

/* ---------------------------------------------------------------- conv ---- */
/* [P1] fused convolution preparation; [P5] column order and tap order.
 * For node t the conv input is the column sequence
 *     P_t = [h_0, ..., h_{K-2}, x(root), ..., x(parent), x(t)]
 * (history oldest first, then the tokens on the root-to-t path).  The conv
 * window is the last K columns of P_t, the commit window the last K-1. */
int gdn_oracle_conv_tree_step(const gdn_oracle_dims *dm, const float *x, long x_stride,
                              const float *conv_w, const float *conv_hist,
                              const int *parents, const int *node_off, const int *slot_map,
                              double *xc, float *win) {
    int rc = check_dims(dm);
    if (rc) return rc;
    if ((rc = check_offsets(dm, node_off))) return rc;
    const int C = conv_channels(dm), K = dm->d_conv;
    const float **col = (const float **)malloc(sizeof(float *) * (size_t)K);
    if (!col) return ORACLE_NOMEM;
    for (int s = 0; s < dm->n_seqs; ++s) {
        const int n0 = node_off[s], ns = node_off[s + 1] - n0, slot = slot_map[s];
        if (slot < 0 || slot >= dm->n_slots) { free(col); return ORACLE_BAD_SLOT; }
        if ((rc = check_parents(parents, n0, ns))) { free(col); return rc; }
        const float *hist = conv_hist + (size_t)slot * (K - 1) * C;
        for (int i = 0; i < ns; ++i) {
            /* col[b] = the column b steps before node i on its path (b = 0: x_i) */
            int cur = i, above = 0;
            col[0] = x + (size_t)(n0 + i) * x_stride;
            for (int b = 1; b < K; ++b) {
                if (cur >= 0) cur = parents[n0 + cur];
                if (cur >= 0) {
                    col[b] = x + (size_t)(n0 + cur) * x_stride;
                } else {
                    col[b] = hist + (size_t)(K - 2 - above) * C;  /* h_{K-2} is the newest */
                    ++above;
                }
            }
            for (int c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int j = 0; j < K; ++j) {       /* window tap j, oldest first */
                    acc += (double)col[K - 1 - j][c] * (double)conv_w[(size_t)c * K + j];
                }
                xc[(size_t)(n0 + i) * C + c] = silu(acc);
                for (int j = 0; j < K - 1; ++j)      /* commit window, oldest first */
                    win[((size_t)(n0 + i) * (K - 1) + j) * C + c] = col[K - 2 - j][c];
            }
        }
    }
    free(col);
    return ORACLE_OK;
}

/* -------------------------------------------------------------- verify ---- */
static void l2_normalise(const float *in, double *out, int d) {
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += (double)in[i] * (double)in[i];
    const double inv = 1.0 / sqrt(ss + L2_EPS);
    for (int i = 0; i < d; ++i) out[i] = (double)in[i] * inv;
}

/* [GDN] recurrence over a tree ([P1] read-only mapped recurrence): every node
 * t, in topological order, starts from its parent's state (the slot's state
 * for a root) and
 *     S'  = decay_t S_parent
 *     u_t = beta_t (v_t - S' k_t)
 *     S_t = S' + u_t k_t^T           (= decay S_p (I - beta k k^T) + beta v k^T)
 *     o_t = q_scale S_t q_t
 * with k, q L2-normalised.  The pool is never written.  The replay row of
 * (t, h) is k_t | u_t | decay_t ([P4] width 2d + 1).
 * S is [d_v][d_k]: row r is value index r, column c key index c. */
int gdn_oracle_tree_verify(const gdn_oracle_dims *dm, const float *xc, const float *ba,
                           long ba_stride, const float *dt_bias, const float *A,
                           const float *ssm, double q_scale, const int *parents,
                           const int *node_off, const int *slot_map,
                           double *o, double *replay) {
    int rc = check_dims(dm);
    if (rc) return rc;
    if ((rc = check_offsets(dm, node_off))) return rc;
    const int C = conv_channels(dm), d = dm->d, Hk = dm->h_k, Hv = dm->h_v;
    const int G = Hv / Hk, R = 2 * d + 1;
    const size_t dd = (size_t)d * d;
    double *qn = (double *)malloc(sizeof(double) * (size_t)d);
    double *kn = (double *)malloc(sizeof(double) * (size_t)d);
    double *u = (double *)malloc(sizeof(double) * (size_t)d);
    double *S0 = (double *)malloc(sizeof(double) * dd);
    if (!qn || !kn || !u || !S0) { free(qn); free(kn); free(u); free(S0); return ORACLE_NOMEM; }
    for (int s = 0; s < dm->n_seqs; ++s) {
        const int n0 = node_off[s], ns = node_off[s + 1] - n0, slot = slot_map[s];
        if (slot < 0 || slot >= dm->n_slots) { rc = ORACLE_BAD_SLOT; goto done; }
        if ((rc = check_parents(parents, n0, ns))) goto done;
        if (ns == 0) continue;
        double *St = (double *)malloc(sizeof(double) * dd * (size_t)ns);
        if (!St) { rc = ORACLE_NOMEM; goto done; }
        for (int h = 0; h < Hv; ++h) {
            const int kh = h / G;                  /* [P3] q/k heads broadcast */
            const float *S0f = ssm + ((size_t)slot * Hv + h) * dd;
            for (int r = 0; r < d; ++r)
                for (int c = 0; c < d; ++c)
                    S0[(size_t)r * d + c] = S0f[(size_t)r * d + c];
            for (int i = 0; i < ns; ++i) {
                const int t = n0 + i, p = parents[t];
                const float *row = xc + (size_t)t * C;
                const float *q = row + (size_t)kh * d;
                const float *k = row + (size_t)Hk * d + (size_t)kh * d;
                const float *v = row + (size_t)2 * Hk * d + (size_t)h * d;
                l2_normalise(q, qn, d);
                l2_normalise(k, kn, d);
                /* [P3] raw gates: beta = sigmoid(b), decay = exp(softplus(a + dt_bias) A) */
                const double b = ba[(size_t)t * ba_stride + h];
                const double a = ba[(size_t)t * ba_stride + Hv + h];
                const double beta = sigmoid(b);
                const double decay = exp(softplus(a + (double)dt_bias[h]) * (double)A[h]);
                const double *Sp = p < 0 ? S0 : St + (size_t)p * dd;
                double *S = St + (size_t)i * dd;
                for (size_t e = 0; e < dd; ++e)
                    S[e] = decay * Sp[e];                              /* S' */
                for (int r = 0; r < d; ++r) {
                    double sk = 0.0;
                    for (int c = 0; c < d; ++c) sk += S[(size_t)r * d + c] * kn[c];
                    u[r] = beta * ((double)v[r] - sk);
                }
                double *orow = o + ((size_t)t * Hv + h) * d;
                for (int r = 0; r < d; ++r)
                    for (int c = 0; c < d; ++c) S[(size_t)r * d + c] += u[r] * kn[c];
                for (int r = 0; r < d; ++r) {
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += S[(size_t)r * d + c] * qn[c];
                    orow[r] = q_scale * acc;
                }
                double *rep = replay + ((size_t)t * Hv + h) * R;
                for (int c = 0; c < d; ++c) rep[c] = kn[c];
                for (int r = 0; r < d; ++r) rep[d + r] = u[r];
                rep[2 * d] = decay;
            }
        }
        free(St);
    }
    rc = ORACLE_OK;
done:
    free(qn); free(kn); free(u); free(S0);
    return rc;
}

/* -------------------------------------------------------------- commit ---- */
/* [P1] replay-log commit after acceptance; [P2] on-device commit of the
 * accepted prefix; [P4] transaction preflight.  All checks run before any
 * write.  For each sequence with accepted node a >= 0, the path root..a is
 * replayed on the slot state of every head, S <- decay_j S + u_j k_j^T in
 * path order, and the slot's conv history becomes a's commit window. */
int gdn_oracle_commit(const gdn_oracle_dims *dm, const int *accepted, const int *parents,
                      const int *node_off, const int *slot_map, const double *replay,
                      const float *win, float *ssm, float *conv_hist) {
    int rc = check_dims(dm);
    if (rc) return rc;
    if ((rc = check_offsets(dm, node_off))) return rc;
    const int C = conv_channels(dm), d = dm->d, Hv = dm->h_v, K = dm->d_conv, R = 2 * d + 1;
    const size_t dd = (size_t)d * d;
    /* preflight */
    for (int s = 0; s < dm->n_seqs; ++s) {
        const int n0 = node_off[s], ns = node_off[s + 1] - n0, a = accepted[s];
        if (a < -1 || a >= ns) return ORACLE_BAD_ACCEPTED;
        if (a < 0) continue;
        const int slot = slot_map[s];
        if (slot < 0 || slot >= dm->n_slots) return ORACLE_BAD_SLOT;
        for (int cur = a; cur >= 0;) {
            const int p = parents[n0 + cur];
            if (p < -1 || p >= cur) return ORACLE_BAD_PARENT;
            cur = p;
        }
        for (int s2 = 0; s2 < s; ++s2)
            if (accepted[s2] >= 0 && slot_map[s2] == slot) return ORACLE_DUP_SLOT;
    }
    /* apply */
    int *path = NULL;
    double *S = (double *)malloc(sizeof(double) * dd);
    if (!S) return ORACLE_NOMEM;
    for (int s = 0; s < dm->n_seqs; ++s) {
        const int n0 = node_off[s], ns = node_off[s + 1] - n0, a = accepted[s];
        if (a < 0) continue;
        const int slot = slot_map[s];
        int *pp = (int *)realloc(path, sizeof(int) * (size_t)(ns > 0 ? ns : 1));
        if (!pp) { free(path); free(S); return ORACLE_NOMEM; }
        path = pp;
        int m = 0;
        for (int cur = a; cur >= 0; cur = parents[n0 + cur]) path[m++] = cur;  /* leaf first */
        for (int h = 0; h < Hv; ++h) {
            float *Sf = ssm + ((size_t)slot * Hv + h) * dd;
            for (size_t e = 0; e < dd; ++e) S[e] = Sf[e];
            for (int step = 0; step < m; ++step) {
                const int j = path[m - 1 - step];           /* root first */
                const double *rep = replay + ((size_t)(n0 + j) * Hv + h) * R;
                const double *kn = rep, *u = rep + d, decay = rep[2 * d];
                for (int r = 0; r < d; ++r)
                    for (int c = 0; c < d; ++c)
                        S[(size_t)r * d + c] = decay * S[(size_t)r * d + c] + u[r] * kn[c];
            }
            for (size_t e = 0; e < dd; ++e) Sf[e] = (float)S[e];
        }
        const int wnode = a;
        const float *w = win + (size_t)(n0 + wnode) * (K - 1) * C;
        float *hst = conv_hist + (size_t)slot * (K - 1) * C;
        memcpy(hst, w, sizeof(float) * (size_t)(K - 1) * C);
    }
    free(path);
    free(S);
    return ORACLE_OK;
}

/* ------------------------------------------------- compact commit windows -- */
/* The commit window of node t, as references instead of copies: the last K-1
 * entries of the column sequence P_t = [h_0 .. h_{K-2}, x(root) .. x(t)]
 * ([P1] the conv tree step also produces the commit window; [P5] column
 * order: history first, oldest first). */
int gdn_oracle_window_refs(const gdn_oracle_dims *dm, const int *parents, const int *node_off,
                           int *refs) {
    int rc = check_dims(dm);
    if (rc) return rc;
    if ((rc = check_offsets(dm, node_off))) return rc;
    const int K = dm->d_conv;
    for (int s = 0; s < dm->n_seqs; ++s) {
        const int n0 = node_off[s], ns = node_off[s + 1] - n0;
        if ((rc = check_parents(parents, n0, ns))) return rc;
        int *cols = (int *)malloc(sizeof(int) * (size_t)(K - 1 + ns + 1));
        int *path = (int *)malloc(sizeof(int) * (size_t)(ns + 1));
        if (!cols || !path) { free(cols); free(path); return ORACLE_NOMEM; }
        for (int i = 0; i < ns; ++i) {
            int m = 0;
            for (int cur = i; cur >= 0; cur = parents[n0 + cur]) path[m++] = cur;   /* t first */
            int len = 0;
            for (int k = 0; k < K - 1; ++k) cols[len++] = -1 - k;                  /* history */
            for (int j = m - 1; j >= 0; --j) cols[len++] = n0 + path[j];          /* root .. t */
            for (int j = 0; j < K - 1; ++j) refs[(size_t)(n0 + i) * (K - 1) + j] = cols[len - (K - 1) + j];
        }
        free(cols);
        free(path);
    }
    return ORACLE_OK;
}

/* The commit with referenced windows: every node's window is gathered from x
 * and the slots' histories as they stand before the commit, then the commit
 * proceeds exactly as gdn_oracle_commit. */
int gdn_oracle_commit_compact(const gdn_oracle_dims *dm, const int *accepted, const int *parents,
                              const int *node_off, const int *slot_map, const double *replay,
                              const float *x, long x_stride, const int *refs, float *ssm,
                              float *conv_hist) {
    int rc = check_dims(dm);
    if (rc) return rc;
    if ((rc = check_offsets(dm, node_off))) return rc;
    const int C = conv_channels(dm), K = dm->d_conv;
    float *win = (float *)malloc(sizeof(float) * (size_t)(dm->n_nodes > 0 ? dm->n_nodes : 1) * (K - 1) * C);
    if (!win) return ORACLE_NOMEM;
    for (int s = 0; s < dm->n_seqs; ++s) {
        /* only the accepted node's window is needed; indices the commit's own
           checks would reject are left for them */
        const int n0 = node_off[s], ns = node_off[s + 1] - n0, slot = slot_map[s], a = accepted[s];
        if (a < 0 || a >= ns || slot < 0 || slot >= dm->n_slots) continue;
        for (int j = 0; j < K - 1; ++j) {
            const int r = refs[(size_t)(n0 + a) * (K - 1) + j];
            float *dst = win + ((size_t)(n0 + a) * (K - 1) + j) * C;
            if (r >= 0 && r < dm->n_nodes)
                memcpy(dst, x + (size_t)r * x_stride, sizeof(float) * (size_t)C);
            else if (r < 0 && -1 - r < K - 1)
                memcpy(dst, conv_hist + ((size_t)slot * (K - 1) + (size_t)(-1 - r)) * C, sizeof(float) * (size_t)C);
            else { free(win); return ORACLE_BAD_NODE_OFF; }
        }
    }
    rc = gdn_oracle_commit(dm, accepted, parents, node_off, slot_map, replay, win, ssm, conv_hist);
    free(win);
    return rc;
}

/* ------------------------------------------------------ gated RMS norm ---- */
/* TensorSharp PR #175, the Qwen 3.5 / Qwen4Exp GDN block: the recurrence's
 * output goes through a gated norm before the scatter; the output gate is a
 * SiLU (gate_mode 0, the existing callers) or a sigmoid (gate_mode 1).  The
 * norm is an RMS norm over the d values of one head with a per-channel weight,
 * then the gate of z multiplies element by element. */
int gdn_oracle_gated_rmsnorm(const gdn_oracle_dims *dm, const float *o, const float *z, long z_stride,
                             const float *w, double eps, int gate_mode, double *y) {
    int rc = check_dims(dm);
    if (rc) return rc;
    if (gate_mode != 0 && gate_mode != 1) return ORACLE_BAD_DIMS;
    const int d = dm->d, Hv = dm->h_v;
    for (int t = 0; t < dm->n_nodes; ++t)
        for (int h = 0; h < Hv; ++h) {
            const float *orow = o + ((size_t)t * Hv + h) * d;
            const float *zrow = z + (size_t)t * z_stride + (size_t)h * d;
            double ss = 0.0;
            for (int i = 0; i < d; ++i) ss += (double)orow[i] * (double)orow[i];
            const double inv = 1.0 / sqrt(ss / d + eps);
            for (int i = 0; i < d; ++i) {
                const double g = gate_mode == 0 ? silu((double)zrow[i]) : sigmoid((double)zrow[i]);
                y[((size_t)t * Hv + h) * d + i] = (double)orow[i] * inv * (double)w[i] * g;
            }
        }
    return ORACLE_OK;
}

/* ---------------------------------------------------------- decode step ---- */
/* TensorSharp PR #175: a step without speculation has nothing to decide later,
 * so its post-window state is committed at once (the caller's "slot -1");
 * lucebox PR #625: ggml_ssm_conv_step (history window + SiLU(conv) + in-place
 * history write-back) and the raw-gate gated delta net in place.  The step is
 * the gated delta rule of [GDN] for one token, state and history updated in
 * the slot. */
int gdn_oracle_decode_step(const gdn_oracle_dims *dm, const float *x, long x_stride, const float *conv_w,
                           float *conv_hist, const float *ba, long ba_stride, const float *dt_bias,
                           const float *A, float *ssm, double q_scale, const int *slot_map, double *xc,
                           double *o) {
    int rc = check_dims(dm);
    if (rc) return rc;
    const int C = conv_channels(dm), K = dm->d_conv, d = dm->d, Hk = dm->h_k, Hv = dm->h_v, G = Hv / Hk;
    const size_t dd = (size_t)d * d;
    for (int s = 0; s < dm->n_seqs; ++s) {
        const int slot = slot_map[s];
        if (slot < 0 || slot >= dm->n_slots) return ORACLE_BAD_SLOT;
        for (int s2 = 0; s2 < s; ++s2)
            if (slot_map[s2] == slot) return ORACLE_DUP_SLOT;
    }
    double *qn = (double *)malloc(sizeof(double) * (size_t)d);
    double *kn = (double *)malloc(sizeof(double) * (size_t)d);
    double *S = (double *)malloc(sizeof(double) * dd);
    if (!qn || !kn || !S) { free(qn); free(kn); free(S); return ORACLE_NOMEM; }
    for (int s = 0; s < dm->n_seqs; ++s) {
        const int slot = slot_map[s];
        float *hist = conv_hist + (size_t)slot * (K - 1) * C;
        const float *xs = x + (size_t)s * x_stride;
        double *xcs = xc + (size_t)s * C;
        /* conv over the column sequence [h_0 .. h_{K-2}, x_s], taps oldest first */
        for (int c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int j = 0; j < K; ++j) {
                const float col = j < K - 1 ? hist[(size_t)j * C + c] : xs[c];
                acc += (double)col * (double)conv_w[(size_t)c * K + j];
            }
            xcs[c] = silu(acc);
        }
        /* the history becomes the last K - 1 columns */
        for (int c = 0; c < C; ++c) {
            for (int j = 0; j < K - 2; ++j) hist[(size_t)j * C + c] = hist[(size_t)(j + 1) * C + c];
            hist[(size_t)(K - 2) * C + c] = xs[c];
        }
        for (int h = 0; h < Hv; ++h) {
            const int kh = h / G;
            const double *q = xcs + (size_t)kh * d, *k = xcs + (size_t)Hk * d + (size_t)kh * d;
            const double *v = xcs + (size_t)2 * Hk * d + (size_t)h * d;
            /* the recurrence reads the conv output at the boundary precision
               (fp32), as the tree path's verify does */
            double sq = 0.0, sk = 0.0;
            for (int c = 0; c < d; ++c) {
                const double qf = (double)(float)q[c], kf = (double)(float)k[c];
                sq += qf * qf;
                sk += kf * kf;
            }
            for (int c = 0; c < d; ++c) {
                qn[c] = (double)(float)q[c] / sqrt(sq + L2_EPS);
                kn[c] = (double)(float)k[c] / sqrt(sk + L2_EPS);
            }
            const double beta = sigmoid((double)ba[(size_t)s * ba_stride + h]);
            const double decay = exp(softplus((double)ba[(size_t)s * ba_stride + Hv + h] + (double)dt_bias[h]) *
                                     (double)A[h]);
            float *Sf = ssm + ((size_t)slot * Hv + h) * dd;
            for (size_t e = 0; e < dd; ++e) S[e] = decay * (double)Sf[e];
            double *orow = o + ((size_t)s * Hv + h) * d;
            for (int r = 0; r < d; ++r) {
                double skr = 0.0;
                for (int c = 0; c < d; ++c) skr += S[(size_t)r * d + c] * kn[c];
                const double u = beta * ((double)(float)v[r] - skr);
                for (int c = 0; c < d; ++c) S[(size_t)r * d + c] += u * kn[c];
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += S[(size_t)r * d + c] * qn[c];
                orow[r] = q_scale * acc;
            }
            for (size_t e = 0; e < dd; ++e) Sf[e] = (float)S[e];
        }
    }
    free(qn); free(kn); free(S);
    return ORACLE_OK;
}
