// gdn_commit.cu - replay-log commit: advance each sequence's persistent conv
// history and recurrent state by its accepted root-to-node path, on the device,
// as one transaction.
//
// lucebox PR #707 "perf(qwen35): fuse the DFlash2 concurrent verify Gated
// DeltaNet route", Summary: persistent state stays read-only during verify and
// the replay-log commit advances it once acceptance is known.  TensorSharp
// PR #175 "Feature/support dflash2": the accepted prefix is committed into the
// live state on the device, replacing restore + re-forward.  lucebox PR #659
// "perf(qwen38): various DFlash2 optimizations concurrency C1-C5": transaction
// preflight; the commit must run on the stream that produced the replay logs.
//
// Two launches on the caller's stream:
//  preflight  one warp per sequence: node range, accepted node, the parent walk
//             (parents held in two registers per lane, walked by shuffles) and
//             slot uniqueness among committing sequences.  Writes *status.
//  apply      one CTA per (value head, sequence); does nothing unless *status
//             is zero.  The path's replay rows are applied in closed form
//                 S = Gamma S0 + sum_j c_j u_j k_j^T,   c_j = prod of decays after j
//             which equals applying S <- decay_j S + u_j k_j^T root first.  The
//             state tile is held in registers (coalesced 128-bit loads and
//             stores), the replay rows are staged in shared memory 16 at a time.
//             The CTA also copies its share of the accepted node's window into
//             the slot's conv history.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace {

constexpr int kApplyThreads = 256;
constexpr int kStage = 16;  // replay rows staged per pass

struct CommitArgs {
    const int32_t *__restrict__ accepted;
    const int32_t *__restrict__ parents;
    const int32_t *__restrict__ node_off;
    const int32_t *__restrict__ slot_map;
    const float *__restrict__ replay;
    int64_t rstride;
    const float *__restrict__ win;
    float *ssm;
    float *hist;
    int32_t *status;
    int S, N, P, Hv, C, max_nodes;
};

__global__ void __launch_bounds__(256) commit_preflight_kernel(const CommitArgs a) {
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= a.S) return;
    const int n0 = a.node_off[s], n1 = a.node_off[s + 1];
    const int acc = a.accepted[s], slot = a.slot_map[s];
    int err = 0;
    if (n0 < 0 || n1 < n0 || n1 > a.N || (s == 0 && n0 != 0) || (s == a.S - 1 && n1 != a.N) ||
        n1 - n0 > a.max_nodes) {
        err = GDN_DEV_BAD_NODE_OFF;
    } else if (acc < -1 || acc >= n1 - n0) {
        err = GDN_DEV_BAD_ACCEPTED;
    } else if (acc >= 0) {
        if (slot < 0 || slot >= a.P) {
            err = GDN_DEV_BAD_SLOT;
        } else {
            const int ns = n1 - n0;  // <= 64
            const int p_lo = lane < ns ? a.parents[n0 + lane] : -1;
            const int p_hi = lane + 32 < ns ? a.parents[n0 + lane + 32] : -1;
            for (int cur = acc; cur >= 0 && !err;) {
                const int p = __shfl_sync(0xffffffffu, cur < 32 ? p_lo : p_hi, cur & 31);
                if (p < -1 || p >= cur) err = GDN_DEV_BAD_PARENT;
                cur = p;
            }
            bool dup = false;
            for (int s2 = lane; s2 < a.S; s2 += 32)
                dup |= (s2 != s && a.accepted[s2] >= 0 && a.slot_map[s2] == slot);
            if (!err && __any_sync(0xffffffffu, dup)) err = GDN_DEV_DUP_SLOT;
        }
    }
    if (err && lane == 0) gdn::record_status(a.status, err);
}

template <int D>
__global__ void __launch_bounds__(kApplyThreads) commit_apply_kernel(const CommitArgs a) {
    constexpr int DV4 = D / 4;
    constexpr int GROUPS = kApplyThreads / DV4;              // row groups
    constexpr int RPT = D / GROUPS > 0 ? D / GROUPS : 1;     // rows per thread
    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
    __shared__ int hdr[4];  // go, first node, path length, slot
    __shared__ int par[gdn::kMaxSeqNodes];
    __shared__ int path[gdn::kMaxSeqNodes];   // root first
    __shared__ float coef[gdn::kMaxSeqNodes];
    __shared__ float gam_s;
    __shared__ __align__(16) float kst[kStage][D];
    __shared__ __align__(16) float ust[kStage][D];

    if (tid == 0) {
        const int st = *reinterpret_cast<volatile int32_t *>(a.status);
        const int acc = a.accepted[s];
        hdr[0] = (st == 0 && acc >= 0);
        hdr[1] = a.node_off[s];
        hdr[2] = acc;  // accepted node for now
        hdr[3] = a.slot_map[s];
    }
    __syncthreads();
    if (!hdr[0]) return;
    const int n0 = hdr[1], acc = hdr[2], slot = hdr[3];
    // the preflight has checked the walk; load the parents up to the accepted node
    for (int i = tid; i <= acc; i += kApplyThreads) par[i] = a.parents[n0 + i];
    __syncthreads();
    if (tid == 0) {
        int m = 0;
        for (int cur = acc; cur >= 0; cur = par[cur]) ++m;
        int k = m;
        for (int cur = acc; cur >= 0; cur = par[cur]) path[--k] = cur;
        hdr[2] = m;
    }
    __syncthreads();
    const int m = hdr[2];
    // decays of the path, then the closed-form coefficients (serial product)
    for (int i = tid; i < m; i += kApplyThreads)
        coef[i] = __ldg(a.replay + ((int64_t(n0) + path[i]) * a.Hv + h) * a.rstride + 2 * D);
    __syncthreads();
    if (tid == 0) {
        float g = 1.0f;
        for (int i = m - 1; i >= 0; --i) {
            const float dec = coef[i];
            coef[i] = g;
            g *= dec;
        }
        gam_s = g;
    }

    // state tile: thread owns float4 column group kc of rows rg + GROUPS * r
    const int kc = tid % DV4, rg = tid / DV4;
    const bool active = rg < D;  // D = 16 leaves some threads idle
    float *sbase = a.ssm + (int64_t(slot) * a.Hv + h) * D * D;
    float4 sv[RPT];
    if (active) {
#pragma unroll
        for (int r = 0; r < RPT; ++r)
            sv[r] = *reinterpret_cast<const float4 *>(sbase + (rg + GROUPS * r) * D + 4 * kc);
    }
    __syncthreads();
    const float gam = gam_s;
    if (active) {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            sv[r].x *= gam; sv[r].y *= gam; sv[r].z *= gam; sv[r].w *= gam;
        }
    }
    for (int base = 0; base < m; base += kStage) {
        const int cnt = min(kStage, m - base);
        for (int idx = tid; idx < cnt * DV4; idx += kApplyThreads) {
            const int j = idx / DV4, c4 = idx - j * DV4;
            const float *row = a.replay + ((int64_t(n0) + path[base + j]) * a.Hv + h) * a.rstride;
            const float cj = coef[base + j];
            *reinterpret_cast<float4 *>(&kst[j][4 * c4]) = __ldg(reinterpret_cast<const float4 *>(row) + c4);
            float4 uv = __ldg(reinterpret_cast<const float4 *>(row + D) + c4);
            uv.x *= cj; uv.y *= cj; uv.z *= cj; uv.w *= cj;
            *reinterpret_cast<float4 *>(&ust[j][4 * c4]) = uv;
        }
        __syncthreads();
        if (active) {
            for (int j = 0; j < cnt; ++j) {
                const float4 kv = *reinterpret_cast<const float4 *>(&kst[j][4 * kc]);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const float uj = ust[j][rg + GROUPS * r];
                    sv[r].x = fmaf(uj, kv.x, sv[r].x);
                    sv[r].y = fmaf(uj, kv.y, sv[r].y);
                    sv[r].z = fmaf(uj, kv.z, sv[r].z);
                    sv[r].w = fmaf(uj, kv.w, sv[r].w);
                }
            }
        }
        __syncthreads();
    }
    if (active) {
#pragma unroll
        for (int r = 0; r < RPT; ++r)
            *reinterpret_cast<float4 *>(sbase + (rg + GROUPS * r) * D + 4 * kc) = sv[r];
    }
    // this head's share of the window copy: conv_hist[slot] <- win[accepted]
    const int64_t total4 = int64_t(3) * a.C / 4;
    const int64_t per = (total4 + a.Hv - 1) / a.Hv;
    const int64_t lo = h * per, hi = min(total4, lo + per);
    const float4 *wsrc = reinterpret_cast<const float4 *>(a.win + (int64_t(n0) + acc) * 3 * a.C);
    float4 *hdst = reinterpret_cast<float4 *>(a.hist + int64_t(slot) * 3 * a.C);
    for (int64_t i = lo + tid; i < hi; i += kApplyThreads) hdst[i] = __ldg(wsrc + i);
}

}  // namespace

extern "C" int gdn_commit(const gdn_dims *dims, const int32_t *accepted, const int32_t *parents,
                          const int32_t *node_off, const int32_t *slot_map, const float *replay,
                          int64_t replay_stride, const float *win, float *ssm, float *conv_hist,
                          int32_t *status, void *stream) {
    int rc = gdn::check_dims(dims);
    if (rc) return rc;
    const int64_t S = dims->n_seqs, N = dims->n_nodes, P = dims->n_slots;
    const int64_t Hv = dims->h_v, D = dims->d_k, C = gdn::conv_channels(dims);
    if (!status) return GDN_ERR_NULL;
    if (S == 0) return GDN_OK;
    if (!accepted || !node_off || !slot_map || !ssm || !conv_hist) return GDN_ERR_NULL;
    if (N > 0 && (!parents || !replay || !win)) return GDN_ERR_NULL;
    if (replay_stride < 2 * D + 1 || replay_stride % 4 != 0) return GDN_ERR_STRIDE;
    if (!gdn::aligned16(ssm) || !gdn::aligned16(conv_hist) || (N > 0 && (!gdn::aligned16(replay) ||
                                                                         !gdn::aligned16(win))))
        return GDN_ERR_ALIGN;
    const gdn::Span outs[] = {{ssm, size_t(P * Hv * D * D * 4)}, {conv_hist, size_t(P * 3 * C * 4)}};
    const gdn::Span ins[] = {{accepted, size_t(S * 4)},
                             {parents, size_t(N * 4)},
                             {node_off, size_t((S + 1) * 4)},
                             {slot_map, size_t(S * 4)},
                             {replay, gdn::strided_bytes(N * Hv, replay_stride, 2 * D + 1)},
                             {win, size_t(N * 3 * C * 4)},
                             {status, 4}};
    if ((rc = gdn::check_alias(outs, 2, ins, 7))) return rc;

    CommitArgs a{accepted, parents, node_off, slot_map, replay, replay_stride, win, ssm, conv_hist, status,
                 int(S), int(N), int(P), int(Hv), int(C), dims->max_seq_nodes};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    commit_preflight_kernel<<<unsigned((S + 7) / 8), 256, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_LAUNCH;
    const dim3 grid{unsigned(Hv), unsigned(S)};
    switch (D) {
        case 16: commit_apply_kernel<16><<<grid, kApplyThreads, 0, st>>>(a); break;
        case 32: commit_apply_kernel<32><<<grid, kApplyThreads, 0, st>>>(a); break;
        case 64: commit_apply_kernel<64><<<grid, kApplyThreads, 0, st>>>(a); break;
        default: commit_apply_kernel<128><<<grid, kApplyThreads, 0, st>>>(a); break;
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}
