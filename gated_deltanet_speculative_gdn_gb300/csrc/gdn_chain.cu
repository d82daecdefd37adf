// gdn_chain.cu - the chain verify entry point: verify for sequences whose
// draft tokens form a chain (node i's parent is node i - 1), d = 128, in
// chunked form.
//
// lucebox PR #707 "perf(qwen35): fuse the DFlash2 concurrent verify Gated
// DeltaNet route", Scope and fallback: dense chains keep a path of their own;
// TensorSharp PR #175 "Feature/support dflash2", change 1: the recurrence over
// a run of tokens goes through a chunked GDN kernel.  The per-node results are
// the same as the tree verify's (a chain is a tree): o, and replay rows
// k^ | u | decay that the commit applies unchanged.
//
// Method.  The chain is cut into chunks of 16 nodes.  With S the state at the
// start of a chunk, Gamma_t the product of the chunk's decays up to node t and
// gamma_{j->t} the product of those after j up to t,
//     decay_t S_{t-1} k^_t = Gamma_t S k^_t + sum_{j<t} gamma_{j->t} (k^_j . k^_t) u_j
// so the chunk's u solve the unit lower-triangular system
//     (I + diag(beta) CK) u = diag(beta) (v - Gamma a),   a_t = S k^_t,
//     CK[t][j] = gamma_{j->t} k^_j . k^_t  (j < t)
// whose inverse times diag(beta), T, is one 16 x 16 matrix shared by every
// row of the state (the WY / UT form): u_t = sum_j T[t][j] e_j with
// e_j = v_j - Gamma_j a_j.  Then
//     o_t = q_scale (Gamma_t S q^_t + sum_{j<=t} gamma_{j->t} (k^_j . q^_t) u_j)
//     S  <- Gamma_{L-1} S + sum_j gamma_{j->L-1} u_j k^_j^T     (end of chunk)
// The decay products are plain products along the chain (no ratios).  The
// kernel (gdn_chain_tc.cu) keeps the state in tensor memory for the whole
// chain and never writes it back: verify leaves the pool untouched, and the
// commit advances it from the replay rows.
#include "gdn_internal.h"

namespace {
constexpr int D = 128;
}  // namespace

extern "C" int gdn_chain_verify(const gdn_dims *dims, const float *xc, const float *ba, int64_t ba_stride,
                                const float *dt_bias, const float *A, const float *ssm, float q_scale,
                                const int32_t *parents, const int32_t *node_off, const int32_t *slot_map, float *o,
                                float *replay, int64_t replay_stride, int32_t *status, void *stream) {
    int rc = gdn::check_dims(dims);
    if (rc) return rc;
    if (dims->d_k != D) return GDN_ERR_DIMS;
    const int64_t S = dims->n_seqs, N = dims->n_nodes, P = dims->n_slots;
    const int64_t Hv = dims->h_v, C = gdn::conv_channels(dims);
    if (!status) return GDN_ERR_NULL;
    if (S == 0 || N == 0) return GDN_OK;
    if (!xc || !ba || !dt_bias || !A || !ssm || !parents || !node_off || !slot_map || !o || !replay)
        return GDN_ERR_NULL;
    if (ba_stride < 2 * Hv) return GDN_ERR_STRIDE;
    if (replay_stride < 2 * D + 1 || replay_stride % 4 != 0) return GDN_ERR_STRIDE;
    if (!gdn::aligned16(xc) || !gdn::aligned16(ssm) || !gdn::aligned16(o) || !gdn::aligned16(replay))
        return GDN_ERR_ALIGN;
    const gdn::Span outs[] = {{o, size_t(N * Hv * D * 4)},
                              {replay, gdn::strided_bytes(N * Hv, replay_stride, 2 * D + 1)}};
    const gdn::Span ins[] = {{xc, size_t(N * C * 4)},
                             {ba, gdn::strided_bytes(N, ba_stride, 2 * Hv)},
                             {dt_bias, size_t(Hv * 4)},
                             {A, size_t(Hv * 4)},
                             {ssm, size_t(P * Hv * D * D * 4)},
                             {parents, size_t(N * 4)},
                             {node_off, size_t((S + 1) * 4)},
                             {slot_map, size_t(S * 4)},
                             {status, 4}};
    if ((rc = gdn::check_alias(outs, 2, ins, 9))) return rc;

    return gdn::launch_chain_tc(dims, xc, ba, ba_stride, dt_bias, A, ssm, q_scale, parents, node_off, slot_map, o,
                                replay, replay_stride, status, stream);
}
