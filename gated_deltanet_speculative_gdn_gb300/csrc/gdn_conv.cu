// gdn_conv.cu - conv tree step: depthwise causal conv (4 taps) + SiLU over each
// sequence's token tree, plus the per-node conv commit windows.
//
// lucebox PR #707 "perf(qwen35): fuse the DFlash2 concurrent verify Gated
// DeltaNet route", Optimizations (fused convolution preparation): one kernel
// reads the slot-mapped conv history, follows the tree parents, applies the
// conv and SiLU and writes the commit window.  Column order and tap order as
// in llama-cpp-bonsai "llama-cpp-bonsai-gdn-conv.patch" (ssm_conv_concat
// kernel): history columns first, taps summed j = 0..3 from the oldest.
//
// Layout: one CTA of four warps per (sequence, block of 128 channels); lane l
// owns channels 4l..4l+3 of the block and warp w takes nodes w, w+4, w+8, ...
// The parent walk of every node (three columns back, into the history above
// the root) is resolved once per CTA in shared memory.  Loads and stores are
// 128-bit and coalesced (512 contiguous bytes per warp); an ancestor's token
// row is read by several warps of the CTA and served from L1/L2.  HBM-bound:
// per node it reads one token row and writes xc (one row) and the window
// (three rows).
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace {

constexpr int kConvThreads = 128;  // 4 warps; 32 lanes x 4 channels = 128 channels per CTA
constexpr int kConvChannels = 128;

struct ConvArgs {
    const float *__restrict__ x;
    int64_t x_stride;
    const float *__restrict__ w;
    const float *__restrict__ hist;
    const int32_t *__restrict__ parents;
    const int32_t *__restrict__ node_off;
    const int32_t *__restrict__ slot_map;
    float *__restrict__ xc;
    float *__restrict__ win;      // [N][3][C] windows (copies), or
    int32_t *__restrict__ wref;   // [N][3] window references (compact form)
    int32_t *status;
    int S, N, P, C, max_nodes;
};

__device__ __forceinline__ float4 silu4(float4 v) {
    return make_float4(gdn::silu_f(v.x), gdn::silu_f(v.y), gdn::silu_f(v.z), gdn::silu_f(v.w));
}

// kCompact: instead of the window rows, each node's window is written as three
// references (oldest first): a global node index (an x row) or -1 - k for
// history column k of the slot; the commit gathers from x and the history.
template <bool kCompact>
__global__ void __launch_bounds__(kConvThreads) conv_tree_step_kernel(const ConvArgs a) {
    const int s = blockIdx.y;
    const int tid = threadIdx.x;
    // hdr: error, first node, node count, slot
    __shared__ int hdr[4];
    __shared__ int par[gdn::kMaxSeqNodes];
    // src[i][b]: the column b + 1 steps before node i: a global node index
    // (>= 0) or -1 - tap for history tap 0..2
    __shared__ int src[gdn::kMaxSeqNodes][3];

    gdn::grid_dep_launch();
    if (tid == 0) {
        const int n0 = a.node_off[s], n1 = a.node_off[s + 1];
        int err = 0;
        if (n0 < 0 || n1 < n0 || n1 > a.N || (s == 0 && n0 != 0) || (s == a.S - 1 && n1 != a.N) ||
            n1 - n0 > a.max_nodes)
            err = GDN_DEV_BAD_NODE_OFF;
        const int slot = a.slot_map[s];
        if (!err && (slot < 0 || slot >= a.P)) err = GDN_DEV_BAD_SLOT;
        hdr[0] = err;
        hdr[1] = n0;
        hdr[2] = n1 - n0;
        hdr[3] = slot;
    }
    __syncthreads();
    // from here on: status, the conv history and the outputs, which the
    // library's other kernels touch
    gdn::grid_dep_wait();
    if (hdr[0]) {
        if (tid == 0) gdn::record_status(a.status, hdr[0]);
        return;
    }
    const int n0 = hdr[1], ns = hdr[2], slot = hdr[3];
    for (int i = tid; i < ns; i += kConvThreads) {
        const int p = a.parents[n0 + i];
        par[i] = p;
        if (p < -1 || p >= i) hdr[0] = GDN_DEV_BAD_PARENT;
    }
    __syncthreads();
    if (hdr[0]) {
        if (tid == 0) gdn::record_status(a.status, hdr[0]);
        return;
    }
    for (int i = tid; i < ns; i += kConvThreads) {
        int cur = i, above = 0;
        for (int b = 0; b < 3; ++b) {
            if (cur >= 0) cur = par[cur];
            if (cur >= 0) {
                src[i][b] = n0 + cur;
            } else {
                src[i][b] = -1 - (2 - above);  // newest history tap first
                ++above;
            }
        }
    }
    __syncthreads();
    if constexpr (kCompact) {
        if (blockIdx.x == 0) {
            for (int i = tid; i < ns; i += kConvThreads) {
                int32_t *r = a.wref + (static_cast<int64_t>(n0) + i) * 3;
                r[0] = src[i][1];
                r[1] = src[i][0];
                r[2] = n0 + i;
            }
        }
    }

    const int lane = tid & 31, warp = tid >> 5;
    const int c4 = blockIdx.x * (kConvChannels / 4) + lane;  // float4 channel group
    if (4 * c4 >= a.C) return;
    const int64_t C = a.C;
    const float4 *w4 = reinterpret_cast<const float4 *>(a.w) + 4 * static_cast<int64_t>(c4);
    const float4 wc0 = __ldg(w4 + 0), wc1 = __ldg(w4 + 1), wc2 = __ldg(w4 + 2), wc3 = __ldg(w4 + 3);
    const float *hbase = a.hist + static_cast<int64_t>(slot) * 3 * C + 4 * c4;
    const float4 h0 = __ldg(reinterpret_cast<const float4 *>(hbase));
    const float4 h1 = __ldg(reinterpret_cast<const float4 *>(hbase + C));
    const float4 h2 = __ldg(reinterpret_cast<const float4 *>(hbase + 2 * C));

    auto column = [&](int sv) -> float4 {
        if (sv >= 0)
            return __ldg(reinterpret_cast<const float4 *>(a.x + static_cast<int64_t>(sv) * a.x_stride + 4 * c4));
        const int tap = -1 - sv;
        return tap == 2 ? h2 : (tap == 1 ? h1 : h0);
    };

    for (int i = warp; i < ns; i += kConvThreads / 32) {
        const int64_t n = n0 + i;
        const float4 c0 = column(n0 + i);     // x(t), newest
        const float4 c1 = column(src[i][0]);
        const float4 c2 = column(src[i][1]);
        const float4 c3 = column(src[i][2]);  // oldest of the window
        // tap j = 0 (oldest, c3) .. 3 (c0), accumulated in that order
        float4 acc;
        acc.x = fmaf(c0.x, wc0.w, fmaf(c1.x, wc0.z, fmaf(c2.x, wc0.y, fmaf(c3.x, wc0.x, 0.0f))));
        acc.y = fmaf(c0.y, wc1.w, fmaf(c1.y, wc1.z, fmaf(c2.y, wc1.y, fmaf(c3.y, wc1.x, 0.0f))));
        acc.z = fmaf(c0.z, wc2.w, fmaf(c1.z, wc2.z, fmaf(c2.z, wc2.y, fmaf(c3.z, wc2.x, 0.0f))));
        acc.w = fmaf(c0.w, wc3.w, fmaf(c1.w, wc3.z, fmaf(c2.w, wc3.y, fmaf(c3.w, wc3.x, 0.0f))));
        *reinterpret_cast<float4 *>(a.xc + n * C + 4 * c4) = silu4(acc);
        if constexpr (!kCompact) {
            float *wrow = a.win + n * 3 * C + 4 * c4;
            // the windows are read back only for the accepted node: stream them past L2
            __stcs(reinterpret_cast<float4 *>(wrow), c2);
            __stcs(reinterpret_cast<float4 *>(wrow + C), c1);
            __stcs(reinterpret_cast<float4 *>(wrow + 2 * C), c0);
        }
    }
}

int conv_entry(const gdn_dims *dims, const float *x, int64_t x_stride, const float *conv_w, const float *conv_hist,
               const int32_t *parents, const int32_t *node_off, const int32_t *slot_map, float *xc, float *win,
               int32_t *wref, int32_t *status, void *stream) {
    int rc = gdn::check_dims(dims);
    if (rc) return rc;
    const int64_t S = dims->n_seqs, N = dims->n_nodes, P = dims->n_slots;
    const int64_t C = gdn::conv_channels(dims);
    const bool compact = wref != nullptr;
    if (!status) return GDN_ERR_NULL;
    if (S == 0 || N == 0) return GDN_OK;
    if (!x || !conv_w || !conv_hist || !parents || !node_off || !slot_map || !xc || (!win && !compact))
        return GDN_ERR_NULL;
    if (x_stride < C || x_stride % 4 != 0) return GDN_ERR_STRIDE;
    if (!gdn::aligned16(x) || !gdn::aligned16(conv_w) || !gdn::aligned16(conv_hist) || !gdn::aligned16(xc) ||
        (!compact && !gdn::aligned16(win)))
        return GDN_ERR_ALIGN;
    const gdn::Span outs[] = {{xc, size_t(N * C * 4)},
                              compact ? gdn::Span{wref, size_t(N * 3 * 4)} : gdn::Span{win, size_t(N * 3 * C * 4)}};
    const gdn::Span ins[] = {{x, gdn::strided_bytes(N, x_stride, C)},
                             {conv_w, size_t(C * 16)},
                             {conv_hist, size_t(P * 3 * C * 4)},
                             {parents, size_t(N * 4)},
                             {node_off, size_t((S + 1) * 4)},
                             {slot_map, size_t(S * 4)},
                             {status, 4}};
    if ((rc = gdn::check_alias(outs, 2, ins, 7))) return rc;

    ConvArgs a{x, x_stride, conv_w, conv_hist, parents, node_off, slot_map, xc, win, wref, status,
               int(S), int(N), int(P), int(C), dims->max_seq_nodes};
    const int c4 = int(C / 4);
    const dim3 grid{unsigned((c4 + kConvChannels / 4 - 1) / (kConvChannels / 4)), unsigned(S)};
    auto k = compact ? conv_tree_step_kernel<true> : conv_tree_step_kernel<false>;
    return gdn::launch_pdl(k, grid, dim3(kConvThreads), 0, static_cast<cudaStream_t>(stream), a) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_LAUNCH;
}

}  // namespace

extern "C" int gdn_conv_tree_step(const gdn_dims *dims, const float *x, int64_t x_stride,
                                  const float *conv_w, const float *conv_hist,
                                  const int32_t *parents, const int32_t *node_off,
                                  const int32_t *slot_map, float *xc, float *win, int32_t *status,
                                  void *stream) {
    if (!win) return GDN_ERR_NULL;
    return conv_entry(dims, x, x_stride, conv_w, conv_hist, parents, node_off, slot_map, xc, win, nullptr, status,
                      stream);
}

extern "C" int gdn_conv_tree_step_compact(const gdn_dims *dims, const float *x, int64_t x_stride,
                                          const float *conv_w, const float *conv_hist,
                                          const int32_t *parents, const int32_t *node_off,
                                          const int32_t *slot_map, float *xc, int32_t *win_ref,
                                          int32_t *status, void *stream) {
    if (!win_ref) return GDN_ERR_NULL;
    return conv_entry(dims, x, x_stride, conv_w, conv_hist, parents, node_off, slot_map, xc, nullptr, win_ref,
                      status, stream);
}
