/* gdn_oracle.h - the oracle's own interface (test infrastructure only).
 *
 * The oracle is a plain, single-threaded C restatement of the GDN speculative
 * tree-verify step.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load it; the library never does, and the two share no
 * source, header, table or helper.
 *
 * Tensors are float32 as they are at the library's boundary; all arithmetic
 * is in double.  Outputs that are computed (xc, o, replay) are returned in
 * double so that a comparison sees the oracle's full precision; outputs that
 * are pure copies (windows, committed history) stay float32 and are exact.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int n_seqs;    /* S: sequences in the batch                          */
    int n_nodes;   /* N: tree nodes of all sequences                     */
    int n_slots;   /* P: slots in the state pools                        */
    int h_k;       /* q/k heads                                          */
    int h_v;       /* value heads, a multiple of h_k                     */
    int d;         /* head width (d_k = d_v = d)                         */
    int d_conv;    /* conv taps                                          */
} gdn_oracle_dims;

enum {
    ORACLE_OK = 0,
    ORACLE_BAD_NODE_OFF = 1,
    ORACLE_BAD_PARENT = 2,
    ORACLE_BAD_SLOT = 3,
    ORACLE_DUP_SLOT = 4,
    ORACLE_BAD_ACCEPTED = 5,
    ORACLE_BAD_DIMS = 6,
    ORACLE_NOMEM = 7
};

/* Depthwise causal conv + SiLU over each sequence's token tree.
 * x [N][x_stride] (first C used), conv_w [C][d_conv], conv_hist [P][d_conv-1][C],
 * parents [N] (local, -1 = root), node_off [S+1], slot_map [S].
 * Out: xc [N][C] (double), win [N][d_conv-1][C] (float, copies). */
int gdn_oracle_conv_tree_step(const gdn_oracle_dims *dm, const float *x, long x_stride,
                              const float *conv_w, const float *conv_hist,
                              const int *parents, const int *node_off, const int *slot_map,
                              double *xc, float *win);

/* Gated delta rule over each sequence's tree, state read from its slot.
 * xc [N][C] (q | k | v), ba [N][ba_stride] (b at [0,h_v), a at [h_v,2h_v)),
 * dt_bias [h_v], A [h_v], ssm [P][h_v][d][d].
 * Out: o [N][h_v][d], replay [N][h_v][2d+1] = k_hat | u | decay (double). */
int gdn_oracle_tree_verify(const gdn_oracle_dims *dm, const float *xc, const float *ba,
                           long ba_stride, const float *dt_bias, const float *A,
                           const float *ssm, double q_scale, const int *parents,
                           const int *node_off, const int *slot_map,
                           double *o, double *replay);

/* Commit the accepted root-to-node path of every sequence (accepted[s] = -1:
 * nothing).  Checks everything first; on any failure returns the code and
 * writes nothing.  replay as produced by gdn_oracle_tree_verify. */
int gdn_oracle_commit(const gdn_oracle_dims *dm, const int *accepted, const int *parents,
                      const int *node_off, const int *slot_map, const double *replay,
                      const float *win, float *ssm, float *conv_hist);

/* Commit-window references.  The commit window of node t is the last
 * d_conv-1 columns of P_t = [h_0, ..., h_{d_conv-2}, x(root), ..., x(t)];
 * refs [N][d_conv-1] names those columns, oldest first: the global node index
 * of an x row (>= 0), or -1 - k for history column h_k of the slot. */
int gdn_oracle_window_refs(const gdn_oracle_dims *dm, const int *parents, const int *node_off,
                           int *refs);

/* gdn_oracle_commit with the window given by references: the window of the
 * accepted node is gathered from the x rows and the slot's history columns
 * (as they are before the commit) that refs names. */
int gdn_oracle_commit_compact(const gdn_oracle_dims *dm, const int *accepted, const int *parents,
                              const int *node_off, const int *slot_map, const double *replay,
                              const float *x, long x_stride, const int *refs, float *ssm,
                              float *conv_hist);

/* Gated RMS norm of the verify output (the output stage after the
 * recurrence): for node t, value head h and i < d,
 *     y[t][h][i] = o[t][h][i] / sqrt(mean_i o[t][h][.]^2 + eps) * w[i] * gate(z[t][h d + i])
 * with gate = SiLU (gate_mode 0) or sigmoid (gate_mode 1).
 * o [N][h_v][d] float, z [N][z_stride] float, w [d] float; y [N][h_v][d] double. */
int gdn_oracle_gated_rmsnorm(const gdn_oracle_dims *dm, const float *o, const float *z, long z_stride,
                             const float *w, double eps, int gate_mode, double *y);

/* Plain decode step: one token per sequence (token s belongs to sequence s),
 * the state and the conv history of its slot advanced in place.  The token
 * is the only node of a one-node tree, accepted at once:
 *     P = [h_0 .. h_{d_conv-2}, x_s],  xc = SiLU(sum_j P[j] w[j]),  h <- last d_conv-1 of P
 *     S <- decay S;  u = beta (v - S k^);  S <- S + u k^T;  o = q_scale S q^
 * x [S][x_stride], ba [S][ba_stride]; ssm, conv_hist in/out; out xc [S][C]
 * (double) and o [S][h_v][d] (double).  Slots must be distinct. */
int gdn_oracle_decode_step(const gdn_oracle_dims *dm, const float *x, long x_stride, const float *conv_w,
                           float *conv_hist, const float *ba, long ba_stride, const float *dt_bias,
                           const float *A, float *ssm, double q_scale, const int *slot_map, double *xc,
                           double *o);

#ifdef __cplusplus
}
#endif
#endif
