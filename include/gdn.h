/* gdn.h - C ABI of the GB300 GDN speculative tree-verify library.
 *
 * One speculative round of a hybrid model's Gated DeltaNet (GDN) layer, for a
 * batch of sequences whose draft tokens form trees:
 *
 *   gdn_conv_tree_step  depthwise causal conv (4 taps) + SiLU over each token
 *                       tree, reading the conv history through a slot map;
 *                       also emits each node's conv commit window.
 *   gdn_tree_verify     gated delta rule over each tree with the gates and the
 *                       q/k L2 norm computed in the kernel; reads the
 *                       recurrent state read-only from its slot and emits the
 *                       attention output and one replay row per node and head.
 *   gdn_chain_verify    the same verify for batches of chains (node i's parent
 *                       is node i - 1), in chunked form.
 *   gdn_commit          once acceptance is known, advances the persistent conv
 *                       and recurrent state of every sequence by its accepted
 *                       root-to-node path, on the device, as one transaction.
 *
 * Sources (page title, section):
 *   lucebox PR #707 "perf(qwen35): fuse the DFlash2 concurrent verify Gated
 *     DeltaNet route" - Optimizations: ssm_conv_tree_step, the read-only
 *     mapped recurrence, gate preparation inside the recurrence; Validation:
 *     persistent state unchanged by verify.
 *   lucebox PR #659 "perf(qwen38): various DFlash2 optimizations concurrency
 *     C1-C5" - Summary item 3 (replay rows of width 257 at state size 128);
 *     test list (padded/permuted slots, transaction preflight); review note on
 *     running the commit on the compute stream.
 *   TensorSharp PR #175 "Feature/support dflash2" - committing the accepted
 *     prefix on the device instead of restore + re-forward; state kept in its
 *     own buffer, read and written as separate in/out.
 *   lucebox PR #625 "qwen35: DSpark speculative decoding" - raw gates
 *     sigmoid(beta) and softplus(alpha + dt_bias) * A applied in the kernel;
 *     one L2 norm over q|k; q/k heads broadcast to the value heads.
 *   llama-cpp-bonsai "llama-cpp-bonsai-gdn-conv.patch" - conv input column
 *     order (history then tokens) and tap/accumulation order.
 *   Yang, Kautz & Hatamizadeh, "Gated Delta Networks" (ICLR 2025) - the
 *     recurrence S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T.
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.  Every pointer argument except `dims` is CUDA device memory on the
 *   current device, owned by the caller (e.g. a torch tensor's data_ptr).  The
 *   library allocates no device memory and keeps no state between calls
 *   (the TMA descriptor of the state pool is encoded on the host per call).
 *   Float tensors are fp32, index tensors int32, all row-major and dense
 *   unless a stride is given.  Pointers to float tensors must be 16-byte
 *   aligned; strides given in floats must be multiples of 4.
 * Shapes.  S = n_seqs, N = n_nodes (all sequences), P = n_slots, d = d_k = d_v
 *   in {16, 32, 64, 128}, H_v a multiple of H_k, G = H_v / H_k, d_conv = 4,
 *   C = 2 H_k d + H_v d conv channels in the order q (H_k d) | k (H_k d) |
 *   v (H_v d).  Sequence s owns nodes node_off[s] .. node_off[s+1]-1
 *   (node_off[0] = 0, node_off[S] = N); N_s = node_off[s+1] - node_off[s]
 *   <= max_seq_nodes <= 64.  parents[n] is the parent's index local to the
 *   sequence, or -1 for a root (which starts from the slot's state and conv
 *   history); a parent precedes its child.  Value head h reads q/k head
 *   floor(h / G).
 * Streams.  All work is enqueued on `stream` (a cudaStream_t; NULL = the
 *   legacy default stream) and is asynchronous.  verify -> (host decides
 *   acceptance) -> commit must be ordered by the caller's stream.  The
 *   library's kernels use programmatic dependent launch: each may start
 *   while the previous kernel on the stream finishes, and waits for it to
 *   complete before touching any buffer the library writes.  They may read
 *   the pure inputs (parents, node_off, slot_map, accepted, win_ref) before
 *   that wait, so a caller that produces those in a kernel on the same stream
 *   must not let that kernel trigger its dependents early
 *   (cudaTriggerProgrammaticLaunchCompletion / griddepcontrol.launch_dependents
 *   before its writes); a plain launch, or a copy, is always safe.
 * Access.  gdn_conv_tree_step and gdn_tree_verify never write the pools
 *   (`conv_hist`, `ssm`).  Only gdn_commit writes them.  No float atomics:
 *   results are bit-for-bit reproducible run to run.
 * Errors.  The return value is a host-side status: GDN_OK or a negative
 *   GDN_ERR_* (nothing was enqueued).  Errors that need the index data are
 *   found on the device and written to `*status` (a device int32 the caller
 *   zeroes; the first error wins).  After a device error the outputs of that
 *   call are unspecified; gdn_commit writes nothing at all (it checks every
 *   sequence before the first write, and also refuses to run when `*status`
 *   is already non-zero on entry, e.g. after a failed verify).  Kernels never
 *   trap; every wait in a kernel is bounded and reports GDN_DEV_TIMEOUT.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t n_seqs;         /* S                                                 */
    int32_t n_nodes;        /* N, tree nodes over all sequences                  */
    int32_t n_slots;        /* P, slots in the conv-history and state pools      */
    int32_t h_k;            /* q/k heads                                         */
    int32_t h_v;            /* value heads (multiple of h_k)                     */
    int32_t d_k;            /* key width   (= d_v, in {16, 32, 64, 128})         */
    int32_t d_v;            /* value width                                       */
    int32_t d_conv;         /* conv taps, must be 4                              */
    int32_t max_seq_nodes;  /* bound on any N_s, 1..64; selects the kernel       */
} gdn_dims;

/* host-side return codes */
enum {
    GDN_OK = 0,
    GDN_ERR_NULL = -1,         /* a required pointer is NULL                      */
    GDN_ERR_DIMS = -2,         /* inconsistent or unsupported dims                */
    GDN_ERR_STRIDE = -3,       /* a stride is smaller than its row or not % 4     */
    GDN_ERR_ALIGN = -4,        /* a float pointer is not 16-byte aligned          */
    GDN_ERR_ALIAS = -5,        /* an output overlaps an input or another output  */
    GDN_ERR_LAUNCH = -6,       /* the CUDA launch failed (cudaGetLastError)       */
    GDN_ERR_TMA = -7,          /* the TMA descriptor of the state pool failed     */
    GDN_ERR_ARG = -8           /* an argument outside its allowed values          */
};

/* device-side codes written to *status */
enum {
    GDN_DEV_BAD_NODE_OFF = 1,  /* node_off not 0..N non-decreasing, or N_s > max  */
    GDN_DEV_BAD_PARENT = 2,    /* parents[n] outside [-1, local index)            */
    GDN_DEV_BAD_SLOT = 3,      /* slot_map[s] outside [0, P)                      */
    GDN_DEV_DUP_SLOT = 4,      /* two committing sequences share a slot           */
    GDN_DEV_BAD_ACCEPTED = 5,  /* accepted[s] outside [-1, N_s)                   */
    GDN_DEV_TIMEOUT = 6,       /* a bounded wait in a kernel ran out              */
    GDN_DEV_BAD_WINDOW = 7     /* a window reference outside [-3, N) (compact)    */
};

/* Conv tree step (lucebox PR #707, Optimizations: fused convolution
 * preparation; conv arithmetic as in llama-cpp-bonsai-gdn-conv.patch).
 * For node t of sequence s, let P_t be the column sequence
 *     h_0, h_1, h_2, x(root), ..., x(parent of t), x(t)
 * with h = conv_hist[slot_map[s]] (h_2 newest).  Then
 *     xc[t][c]     = SiLU( sum_{j=0..3} P_t[-4 + j][c] * conv_w[c][j] )
 * summed in tap order j = 0 (oldest) .. 3 (= x(t)), no bias, and
 *     win[t][j][c] = P_t[-3 + j][c]           j = 0..2 (oldest first)
 * the raw columns that become the slot's history if t is accepted.
 *   x         [N][x_stride] in, first C floats of each row used
 *   conv_w    [C][4]        in
 *   conv_hist [P][3][C]     in (read-only here)
 *   parents   [N], node_off [S+1], slot_map [S]   in
 *   xc        [N][C]        out
 *   win       [N][3][C]     out
 * Device errors: GDN_DEV_BAD_NODE_OFF, GDN_DEV_BAD_PARENT, GDN_DEV_BAD_SLOT. */
int gdn_conv_tree_step(const gdn_dims *dims, const float *x, int64_t x_stride,
                       const float *conv_w, const float *conv_hist,
                       const int32_t *parents, const int32_t *node_off,
                       const int32_t *slot_map, float *xc, float *win,
                       int32_t *status, void *stream);

/* Tree verify (lucebox PR #707, Optimizations: read-only mapped recurrence and
 * gate preparation inside the recurrence; lucebox PR #659, Summary item 3).
 * For node t (topological order) and value head h, with k-head j = h / G:
 *     q = xc[t][j d ..], k = xc[t][H_k d + j d ..], v = xc[t][2 H_k d + h d ..]
 *     q^ = q / sqrt(|q|^2 + 1e-6),  k^ likewise
 *     beta = sigmoid(ba[t][h]),  decay = exp(softplus(ba[t][H_v + h] + dt_bias[h]) * A[h])
 *     S'   = decay * S_parent         (S_parent of a root = ssm[slot_map[s]][h])
 *     u    = beta * (v - S' k^)
 *     S_t  = S' + u k^T               (= decay S_p (I - beta k^ k^T) + beta v k^T)
 *     o[t][h] = q_scale * S_t q^
 *     replay[t][h] = k^ (d) | u (d) | decay (1)
 * S is [d_v][d_k] (row = value index).  ssm is only read.  softplus(x) = x
 * above 20.
 *   xc       [N][C] in (dense)         ba [N][ba_stride] in (b | a; stride >= 2 H_v)
 *   dt_bias  [H_v], A [H_v]  in        ssm [P][H_v][d][d] in (read-only)
 *   o        [N][H_v][d]  out
 *   replay   [N][H_v][replay_stride] out; replay_stride >= 2d + 1 and % 4 == 0
 *            (gdn_replay_row_floats gives the smallest); floats past 2d + 1
 *            in a row are not written
 * Device errors: GDN_DEV_BAD_NODE_OFF, GDN_DEV_BAD_PARENT, GDN_DEV_BAD_SLOT,
 * GDN_DEV_TIMEOUT. */
int gdn_tree_verify(const gdn_dims *dims, const float *xc, const float *ba,
                    int64_t ba_stride, const float *dt_bias, const float *A,
                    const float *ssm, float q_scale, const int32_t *parents,
                    const int32_t *node_off, const int32_t *slot_map, float *o,
                    float *replay, int64_t replay_stride, int32_t *status,
                    void *stream);

/* Chain verify (lucebox PR #707, Scope and fallback: dense chains keep a path
 * of their own; TensorSharp PR #175, change 1: a run of tokens goes through a
 * chunked GDN kernel).  The same operation, arguments, outputs and replay rows
 * as gdn_tree_verify, for batches in which every sequence's nodes form a chain
 * (parents[node_off[s] + i] = i - 1), d = 128 only.  It evaluates the chain in
 * chunks of 16 nodes and carries the state on chip between them, so long
 * chains (up to max_seq_nodes = 64) cost little more per node than short ones.
 * The replay rows feed gdn_commit / gdn_commit_compact unchanged.
 * Host errors: as gdn_tree_verify, and GDN_ERR_DIMS when d != 128.
 * Device errors: GDN_DEV_BAD_NODE_OFF, GDN_DEV_BAD_SLOT, GDN_DEV_BAD_PARENT
 * (a sequence that is not a chain; its outputs are not written),
 * GDN_DEV_TIMEOUT. */
int gdn_chain_verify(const gdn_dims *dims, const float *xc, const float *ba,
                     int64_t ba_stride, const float *dt_bias, const float *A,
                     const float *ssm, float q_scale, const int32_t *parents,
                     const int32_t *node_off, const int32_t *slot_map, float *o,
                     float *replay, int64_t replay_stride, int32_t *status,
                     void *stream);

/* Replay-log commit (lucebox PR #707, Summary; TensorSharp PR #175 on-device
 * commit; lucebox PR #659 transaction preflight and stream ordering).
 * accepted[s] in {-1} U [0, N_s): -1 commits nothing for s.  Otherwise the
 * path root .. accepted[s] is found by walking parents, and for every head h
 *     S <- decay_j S + u_j k^_j^T     for j along the path, root first
 * on ssm[slot_map[s]][h] (k^, u, decay from the replay rows), and
 *     conv_hist[slot_map[s]] <- win[accepted[s]].
 * A preflight checks node_off, accepted, the parent walk and that no two
 * committing sequences share a slot; if any check fails (or *status is
 * already non-zero) nothing is written.
 *   accepted [S] in; parents, node_off, slot_map in; replay, win in (as
 *   produced by verify and conv for this round); ssm, conv_hist in/out.
 * Device errors: GDN_DEV_BAD_NODE_OFF, GDN_DEV_BAD_ACCEPTED,
 * GDN_DEV_BAD_PARENT, GDN_DEV_BAD_SLOT, GDN_DEV_DUP_SLOT. */
int gdn_commit(const gdn_dims *dims, const int32_t *accepted, const int32_t *parents,
               const int32_t *node_off, const int32_t *slot_map, const float *replay,
               int64_t replay_stride, const float *win, float *ssm, float *conv_hist,
               int32_t *status, void *stream);

/* Compact commit windows (lucebox PR #707, Optimizations: the conv tree step
 * also produces the commit window; a window is three columns of the node's
 * column sequence, so it can be named instead of copied).
 * gdn_conv_tree_step_compact computes xc exactly as gdn_conv_tree_step but,
 * instead of the window rows, writes for every node t
 *     win_ref[t][j], j = 0..2 (oldest first)
 * naming column j of t's commit window: a global node index n >= 0 (the
 * window column is x row n) or -1 - k for column h_k of the slot's history.
 * gdn_commit_compact then performs gdn_commit with the accepted node's window
 * gathered through win_ref from x and from the slot's history as it stands
 * before the commit; the caller keeps x (and its stride) unchanged from the
 * conv call to the commit.  This saves the 3 C floats per node that
 * gdn_conv_tree_step writes and the commit reads.
 *   win_ref  [N][3] int32 out (conv) / in (commit); x, x_stride as for conv.
 * Device errors: as the non-compact calls, plus GDN_DEV_BAD_WINDOW (commit:
 * a reference of an accepted node outside [-3, N); nothing is written). */
int gdn_conv_tree_step_compact(const gdn_dims *dims, const float *x, int64_t x_stride,
                               const float *conv_w, const float *conv_hist,
                               const int32_t *parents, const int32_t *node_off,
                               const int32_t *slot_map, float *xc, int32_t *win_ref,
                               int32_t *status, void *stream);

int gdn_commit_compact(const gdn_dims *dims, const int32_t *accepted, const int32_t *parents,
                       const int32_t *node_off, const int32_t *slot_map, const float *replay,
                       int64_t replay_stride, const float *x, int64_t x_stride,
                       const int32_t *win_ref, float *ssm, float *conv_hist, int32_t *status,
                       void *stream);

/* Gated RMS norm, the output stage after the recurrence (TensorSharp PR #175,
 * the Qwen 3.5 / Qwen4Exp GDN block: gated delta net -> gated norm; the output
 * gate is a SiLU, gate_mode 0, or a sigmoid, gate_mode 1).  For node t, value
 * head h and i < d:
 *     y[t][h][i] = o[t][h][i] / sqrt(mean_i(o[t][h][.]^2) + eps) * norm_w[i]
 *                  * gate(z[t][h d + i])
 *   o       [N][H_v][d] in (e.g. gdn_tree_verify's output)
 *   z       [N][z_stride] in, z_stride >= H_v d and % 4 == 0
 *   norm_w  [d] in (one weight vector shared by the heads)
 *   eps     >= 0 (eps = 0 with an all-zero head gives NaN)
 *   y       [N][H_v][d] out (must not overlap the inputs)
 * Host errors: GDN_ERR_ARG for gate_mode outside {0, 1} or eps < 0 / not
 * finite.  No device errors. */
int gdn_gated_rmsnorm(const gdn_dims *dims, const float *o, const float *z, int64_t z_stride,
                      const float *norm_w, float eps, int gate_mode, float *y, void *stream);

/* Plain decode step (TensorSharp PR #175: a step without speculation commits
 * its post-window state at once, the caller's "slot -1"; lucebox PR #625:
 * ggml_ssm_conv_step with in-place history write-back and the raw-gate gated
 * delta net in place).  One token per sequence: dims->n_nodes must equal
 * dims->n_seqs and token s belongs to sequence s.  For each s, with
 * h = conv_hist[slot_map[s]] and the column sequence P = [h_0, h_1, h_2, x_s]:
 *     xc[s][c] = SiLU(sum_{j=0..3} P[j][c] conv_w[c][j]);   h <- [h_1, h_2, x_s]
 * and for every value head h with the gates and normalised q/k of
 * gdn_tree_verify:
 *     S <- decay S;  u = beta (v - S k^);  S <- S + u k^T;  o[s][h] = q_scale S q^
 * on ssm[slot_map[s]][h] in place.  This is gdn_conv_tree_step +
 * gdn_tree_verify + gdn_commit on one-node trees with every node accepted,
 * without the windows and replay rows.
 *   x [S][x_stride] in; conv_w in; conv_hist, ssm in/out; ba [S][ba_stride] in;
 *   dt_bias, A in; slot_map [S] in; xc [S][C] out; o [S][H_v][d] out.
 * Device errors: GDN_DEV_BAD_SLOT, GDN_DEV_DUP_SLOT (two sequences in one
 * slot); on any error (or a non-zero *status on entry) nothing is written. */
int gdn_decode_step(const gdn_dims *dims, const float *x, int64_t x_stride, const float *conv_w,
                    float *conv_hist, const float *ba, int64_t ba_stride, const float *dt_bias,
                    const float *A, float *ssm, float q_scale, const int32_t *slot_map, float *xc,
                    float *o, int32_t *status, void *stream);

/* Test hook for the device timeout path.  The next call that runs a
 * tensor-core verify kernel (gdn_tree_verify with d = 128 and
 * max_seq_nodes <= 16, or gdn_chain_verify) makes one role of its first CTA
 * wait on a barrier that nothing ever completes, for wait_ns (capped at the
 * library's 2 s wait limit); the wait runs out, every role of that CTA drains
 * its copies and tensor-core work and leaves (the chain kernel's other roles
 * each wait out their own limit first, so that call takes about 2 s), and the
 * call reports GDN_DEV_TIMEOUT in *status (its outputs are then unspecified).
 * The hook is consumed by that one call; calls that run another kernel leave
 * it pending.  The paper has no counterpart; it exists so that the bounded-wait
 * path can be tested without a GPU fault. */
void gdn_test_stall_next_verify(uint64_t wait_ns);

/* Name of a host or device status code ("GDN_OK", "GDN_DEV_DUP_SLOT", ...);
 * "unknown" for any other value.  Never NULL. */
const char *gdn_status_str(int code);

/* Smallest replay_stride for widths d_k, d_v: d_k + d_v + 1 rounded up to a
 * multiple of 4 floats (260 at d = 128).  0 for unsupported widths. */
size_t gdn_replay_row_floats(int d_k, int d_v);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H */
