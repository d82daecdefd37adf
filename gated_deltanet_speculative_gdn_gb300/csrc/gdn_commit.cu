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
//  apply      CTAs of 32 state rows of one (value head, sequence); do nothing
//             unless *status is zero.  The path's replay rows are applied in
//             closed form
//                 S = Gamma S0 + sum_j c_j u_j k_j^T,   c_j = prod of decays after j
//             which equals applying S <- decay_j S + u_j k_j^T root first.  The
//             state rows are held in registers (coalesced 128-bit loads and
//             stores), the path's replay rows are staged in shared memory, and
//             the CTA also copies its share of the accepted node's window into
//             the slot's conv history.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace {


struct CommitArgs {
    const int32_t *__restrict__ accepted;
    const int32_t *__restrict__ parents;
    const int32_t *__restrict__ node_off;
    const int32_t *__restrict__ slot_map;
    const float *__restrict__ replay;
    int64_t rstride;
    const float *__restrict__ win;      // [N][3][C] windows, or (compact form)
    const int32_t *__restrict__ wref;   // [N][3] window references into x / the history
    const float *__restrict__ x;        // [N][x_stride] tokens (compact form only)
    int64_t x_stride;
    float *ssm;
    float *hist;
    int32_t *status;
    int S, N, P, Hv, C, max_nodes;
};

__global__ void __launch_bounds__(256) commit_preflight_kernel(const CommitArgs a) {
    gdn::grid_dep_launch();
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= a.S) return;
    // the checks that need only the caller's index inputs run before the wait,
    // while the verify launched before this kernel finishes
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
    gdn::grid_dep_wait();  // status; the compact form's window references come from the conv
    if (!err && acc >= 0 && a.wref) {
        for (int j = 0; j < 3; ++j) {
            const int r = a.wref[(int64_t(n0) + acc) * 3 + j];
            if (r < -3 || r >= a.N) err = GDN_DEV_BAD_WINDOW;
        }
    }
    if (err && lane == 0) gdn::record_status(a.status, err);
}

// Apply: a CTA of four warps covers 32 state rows of one (head, sequence);
// warp w owns 8 of them (lane l: row group l / (d/4), float4 column group
// l % (d/4)) and loads them into registers first.  Meanwhile warp 0 walks the
// accepted path (parents two per lane, walked by shuffles), forms the
// closed-form coefficients with a warp scan of the path's decays and leaves
// them in shared memory, and the other warps copy their share of the accepted
// node's window.  The path's replay rows (k^_j and this CTA's slice of u_j)
// are then staged into shared memory together, kBatch entries at a time, so
// the CTA waits for one round trip per batch rather than one per entry, and
// every warp applies them root first from there.
constexpr int kWarpRows = 8;                      // state rows per warp
constexpr int kApplyWarps = 4;
constexpr int kCtaRows = kWarpRows * kApplyWarps; // state rows per CTA
constexpr int kBatch = 16;                        // path entries staged at a time

template <int D>
__global__ void __launch_bounds__(kApplyWarps * 32, 6) commit_apply_kernel(const CommitArgs a) {
    constexpr int DV4 = D / 4;               // float4 chunks per row (<= 32)
    constexpr int RI = 32 / DV4;             // rows one warp instruction covers
    constexpr int NF = kWarpRows / RI;       // float4 per lane
    constexpr int CPH = (D + kCtaRows - 1) / kCtaRows;  // CTAs per head
    constexpr int CR = D < kCtaRows ? D : kCtaRows;     // state rows of a CTA
    static_assert(NF >= 1, "d >= 16");
    __shared__ float4 kst[kBatch][DV4];      // k^_j rows of the batch
    __shared__ float ust[kBatch][CR];        // u_j of the CTA's rows
    __shared__ int nodes[gdn::kMaxSeqNodes]; // path, leaf first
    __shared__ float coef[gdn::kMaxSeqNodes];
    __shared__ float gam_s;
    __shared__ int m_s;

    const int hq = blockIdx.x, s = blockIdx.y;
    const int h = hq / CPH, q = hq % CPH;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned full = 0xffffffffu;
    const int rcta = q * kCtaRows, rbase = rcta + warp * kWarpRows;  // first row of the CTA, the warp
    const bool has_rows = rbase < D;  // d = 16: two warps hold no rows

    // the preflight (earlier on this stream) has checked every index; the range
    // tests here only keep the loads below in bounds
    gdn::grid_dep_launch();
    const int acc = a.accepted[s], n0 = a.node_off[s], n1 = a.node_off[s + 1], slot = a.slot_map[s];
    gdn::grid_dep_wait();  // status, the state pool and the replay rows
    const int st = *reinterpret_cast<volatile int32_t *>(a.status);
    if (!(st == 0 && acc >= 0 && n0 >= 0 && n1 <= a.N && acc < n1 - n0 && acc < gdn::kMaxSeqNodes && slot >= 0 &&
          slot < a.P))
        return;  // the whole CTA: the condition does not depend on the thread

    const int kc = lane % DV4, ro = lane / DV4;
    float *sbase = a.ssm + (int64_t(slot) * a.Hv + h) * D * D;
    float4 sv[NF];
    if (has_rows) {
#pragma unroll
        for (int f = 0; f < NF; ++f)
            sv[f] = *reinterpret_cast<const float4 *>(sbase + (rbase + ro + RI * f) * D + 4 * kc);
    }
    const int64_t rnode = int64_t(a.Hv) * a.rstride;
    const float *rbase_h = a.replay + (int64_t(n0) * a.Hv + h) * a.rstride;  // node 0 of the sequence, head h

    if (warp == 0) {
        // path, leaf first: lane i holds entry i (register lo) and i + 32 (hi)
        const int p_lo = lane <= acc ? a.parents[n0 + lane] : -1;
        const int p_hi = lane + 32 <= acc ? a.parents[n0 + lane + 32] : -1;
        int node_lo = -1, node_hi = -1, m = 0;
        for (int cur = acc; cur >= 0; ++m) {
            if (lane == (m & 31)) {
                if (m < 32) node_lo = cur; else node_hi = cur;
            }
            cur = __shfl_sync(full, cur < 32 ? p_lo : p_hi, cur & 31);
        }
        // coefficient of leaf-first entry i = product of the decays of entries 0..i-1
        const float d_lo = node_lo >= 0 ? __ldg(rbase_h + node_lo * rnode + 2 * D) : 1.0f;
        const float d_hi = node_hi >= 0 ? __ldg(rbase_h + node_hi * rnode + 2 * D) : 1.0f;
        float x_lo = d_lo, x_hi = d_hi;  // inclusive scans
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y_lo = __shfl_up_sync(full, x_lo, o), y_hi = __shfl_up_sync(full, x_hi, o);
            if (lane >= o) {
                x_lo *= y_lo;
                x_hi *= y_hi;
            }
        }
        const float tot_lo = __shfl_sync(full, x_lo, 31);
        float c_lo = __shfl_up_sync(full, x_lo, 1), c_hi = __shfl_up_sync(full, x_hi, 1);
        if (lane == 0) {
            c_lo = 1.0f;
            c_hi = 1.0f;
        }
        c_hi *= tot_lo;
        const float gam = tot_lo * __shfl_sync(full, x_hi, 31);  // all m decays
        if (lane < m) {
            nodes[lane] = node_lo;
            coef[lane] = c_lo;
        }
        if (lane + 32 < m) {
            nodes[lane + 32] = node_hi;
            coef[lane + 32] = c_hi;
        }
        if (lane == 0) {
            gam_s = gam;
            m_s = m;
        }
    } else if (!a.wref) {
        // warps 1-3: their share of the window copy, conv_hist[slot] <- win[accepted]
        const int64_t total4 = int64_t(3) * a.C / 4;
        const int64_t parts = int64_t(a.Hv) * CPH * (kApplyWarps - 1);
        const int64_t per = (total4 + parts - 1) / parts;
        const int64_t lo = ((int64_t(h) * CPH + q) * (kApplyWarps - 1) + warp - 1) * per, hi = min(total4, lo + per);
        const float4 *wsrc = reinterpret_cast<const float4 *>(a.win + (int64_t(n0) + acc) * 3 * a.C);
        float4 *hdst = reinterpret_cast<float4 *>(a.hist + int64_t(slot) * 3 * a.C);
        for (int64_t i = lo + lane; i < hi; i += 32) hdst[i] = __ldg(wsrc + i);
    } else {
        // warps 1-3, compact form: their share of the channel groups of the new
        // history, gathered through the accepted node's references from x rows
        // and the slot's old history; a thread reads all three columns of its
        // channel group before writing any, so in-place reuse of an old column
        // is safe (and no other thread touches that channel group)
        const int64_t total4 = a.C / 4;
        const int64_t parts = int64_t(a.Hv) * CPH * (kApplyWarps - 1);
        const int64_t per = (total4 + parts - 1) / parts;
        const int64_t lo = ((int64_t(h) * CPH + q) * (kApplyWarps - 1) + warp - 1) * per, hi = min(total4, lo + per);
        const int32_t *ref = a.wref + (int64_t(n0) + acc) * 3;
        const int r0 = ref[0], r1 = ref[1], r2 = ref[2];
        float4 *hdst = reinterpret_cast<float4 *>(a.hist + int64_t(slot) * 3 * a.C);
        auto col = [&](int r, int64_t i) -> float4 {
            return r >= 0 ? __ldg(reinterpret_cast<const float4 *>(a.x + int64_t(r) * a.x_stride) + i)
                          : hdst[(-1 - r) * (a.C / 4) + i];
        };
        for (int64_t i = lo + lane; i < hi; i += 32) {
            const float4 v0 = col(r0, i), v1 = col(r1, i), v2 = col(r2, i);
            hdst[i] = v0;
            hdst[a.C / 4 + i] = v1;
            hdst[2 * (a.C / 4) + i] = v2;
        }
    }
    __syncthreads();
    const int m = m_s;
    const float gam = gam_s;
    if (has_rows) {
#pragma unroll
        for (int f = 0; f < NF; ++f) {
            sv[f].x *= gam; sv[f].y *= gam; sv[f].z *= gam; sv[f].w *= gam;
        }
    }
    // root first: leaf-first entries m-1 .. 0, kBatch at a time
    for (int top = m - 1; top >= 0; top -= kBatch) {
        const int nb = min(kBatch, top + 1);  // entries top, top-1, .., top-nb+1 -> slots 0..nb-1
        for (int x = tid; x < nb * DV4; x += kApplyWarps * 32) {
            const int e = x / DV4, c = x % DV4;
            kst[e][c] = __ldg(reinterpret_cast<const float4 *>(rbase_h + nodes[top - e] * rnode) + c);
        }
        for (int x = tid; x < nb * CR / 4; x += kApplyWarps * 32) {
            const int e = x / (CR / 4), c = x % (CR / 4);
            reinterpret_cast<float4 *>(ust[e])[c] =
                __ldg(reinterpret_cast<const float4 *>(rbase_h + nodes[top - e] * rnode + D + rcta) + c);
        }
        __syncthreads();
        if (has_rows) {
            for (int e = 0; e < nb; ++e) {
                const float cj = coef[top - e];
                const float4 kv = kst[e][kc];
#pragma unroll
                for (int f = 0; f < NF; ++f) {
                    // row rbase + ro + RI f
                    const float uj = ust[e][rbase - rcta + ro + RI * f] * cj;
                    sv[f].x = fmaf(uj, kv.x, sv[f].x);
                    sv[f].y = fmaf(uj, kv.y, sv[f].y);
                    sv[f].z = fmaf(uj, kv.z, sv[f].z);
                    sv[f].w = fmaf(uj, kv.w, sv[f].w);
                }
            }
        }
        __syncthreads();  // the batch's staging may be overwritten
    }
    if (has_rows) {
#pragma unroll
        for (int f = 0; f < NF; ++f)
            *reinterpret_cast<float4 *>(sbase + (rbase + ro + RI * f) * D + 4 * kc) = sv[f];
    }
}

int commit_entry(const gdn_dims *dims, const int32_t *accepted, const int32_t *parents, const int32_t *node_off,
                 const int32_t *slot_map, const float *replay, int64_t replay_stride, const float *win,
                 const float *x, int64_t x_stride, const int32_t *wref, float *ssm, float *conv_hist,
                 int32_t *status, void *stream) {
    int rc = gdn::check_dims(dims);
    if (rc) return rc;
    const int64_t S = dims->n_seqs, N = dims->n_nodes, P = dims->n_slots;
    const int64_t Hv = dims->h_v, D = dims->d_k, C = gdn::conv_channels(dims);
    const bool compact = wref != nullptr;
    if (!status) return GDN_ERR_NULL;
    if (S == 0) return GDN_OK;
    if (!accepted || !node_off || !slot_map || !ssm || !conv_hist) return GDN_ERR_NULL;
    if (N > 0 && (!parents || !replay || (compact ? !x : !win))) return GDN_ERR_NULL;
    if (replay_stride < 2 * D + 1 || replay_stride % 4 != 0) return GDN_ERR_STRIDE;
    if (compact && (x_stride < C || x_stride % 4 != 0)) return GDN_ERR_STRIDE;
    if (!gdn::aligned16(ssm) || !gdn::aligned16(conv_hist) ||
        (N > 0 && (!gdn::aligned16(replay) || (compact ? !gdn::aligned16(x) : !gdn::aligned16(win)))))
        return GDN_ERR_ALIGN;
    const gdn::Span outs[] = {{ssm, size_t(P * Hv * D * D * 4)}, {conv_hist, size_t(P * 3 * C * 4)}};
    const gdn::Span ins[] = {{accepted, size_t(S * 4)},
                             {parents, size_t(N * 4)},
                             {node_off, size_t((S + 1) * 4)},
                             {slot_map, size_t(S * 4)},
                             {replay, gdn::strided_bytes(N * Hv, replay_stride, 2 * D + 1)},
                             compact ? gdn::Span{x, gdn::strided_bytes(N, x_stride, C)} : gdn::Span{win, size_t(N * 3 * C * 4)},
                             {wref, compact ? size_t(N * 3 * 4) : 0},
                             {status, 4}};
    if ((rc = gdn::check_alias(outs, 2, ins, 8))) return rc;

    CommitArgs a{accepted, parents, node_off, slot_map, replay, replay_stride, compact ? nullptr : win, wref, x,
                 x_stride, ssm, conv_hist, status, int(S), int(N), int(P), int(Hv), int(C), dims->max_seq_nodes};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (gdn::launch_pdl(commit_preflight_kernel, dim3(unsigned((S + 7) / 8)), dim3(256), 0, st, a) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    // CTAs of 32 state rows: d / 32 per head (one for d = 16)
    const unsigned cph = unsigned((D + kCtaRows - 1) / kCtaRows);
    const dim3 grid{unsigned(Hv) * cph, unsigned(S)};
    cudaError_t e;
    const dim3 block(kApplyWarps * 32);
    switch (D) {
        case 16: e = gdn::launch_pdl(commit_apply_kernel<16>, grid, block, 0, st, a); break;
        case 32: e = gdn::launch_pdl(commit_apply_kernel<32>, grid, block, 0, st, a); break;
        case 64: e = gdn::launch_pdl(commit_apply_kernel<64>, grid, block, 0, st, a); break;
        default: e = gdn::launch_pdl(commit_apply_kernel<128>, grid, block, 0, st, a); break;
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

}  // namespace

extern "C" int gdn_commit(const gdn_dims *dims, const int32_t *accepted, const int32_t *parents,
                          const int32_t *node_off, const int32_t *slot_map, const float *replay,
                          int64_t replay_stride, const float *win, float *ssm, float *conv_hist,
                          int32_t *status, void *stream) {
    if (dims && dims->n_nodes > 0 && !win) return GDN_ERR_NULL;
    return commit_entry(dims, accepted, parents, node_off, slot_map, replay, replay_stride, win, nullptr, 0, nullptr,
                        ssm, conv_hist, status, stream);
}

extern "C" int gdn_commit_compact(const gdn_dims *dims, const int32_t *accepted, const int32_t *parents,
                                  const int32_t *node_off, const int32_t *slot_map, const float *replay,
                                  int64_t replay_stride, const float *x, int64_t x_stride,
                                  const int32_t *win_ref, float *ssm, float *conv_hist, int32_t *status,
                                  void *stream) {
    if (dims && dims->n_nodes > 0 && !win_ref) return GDN_ERR_NULL;
    return commit_entry(dims, accepted, parents, node_off, slot_map, replay, replay_stride, nullptr, x, x_stride,
                        win_ref, ssm, conv_hist, status, stream);
}
