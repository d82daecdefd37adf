// gdn_decode.cu - plain decode step: one token per sequence, the conv history
// and the recurrent state of its slot advanced in place (no replay rows, no
// deferred commit).
//
// TensorSharp PR #175 "Feature/support dflash2": a step without speculation
// has nothing to decide later, so its post-window state is committed at once
// (the caller's "slot -1"); lucebox PR #625 "qwen35: DSpark speculative
// decoding": ggml_ssm_conv_step (history window + SiLU(conv) + in-place
// history write-back) and the raw-gate gated delta net applied in place.
//
// Three launches on the caller's stream:
//  preflight  warp per sequence: slot in range and not shared by another
//             sequence; writes *status.  The two kernels below do nothing
//             unless *status is zero, so a failed step writes nothing.
//  conv       thread per (sequence, 4 channels): xc = SiLU(conv of the three
//             history columns and the token), history <- last three columns.
//             Each thread reads its channels' history before overwriting it.
//  recur      CTA of four warps per (sequence, value head): q^, k^ (every warp
//             normalises both, 128-bit loads and a warp reduction), gates, then
//             the warps sweep the state rows: a row of d floats spans d/4 lanes
//             (128-bit coalesced loads and stores), S k^ and S q^ are segmented
//             warp reductions, and the row is rewritten in place.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace {

struct DecodeArgs {
    const float *__restrict__ x;
    int64_t x_stride;
    const float *__restrict__ w;
    float *hist;
    const float *__restrict__ ba;
    int64_t ba_stride;
    const float *__restrict__ dt_bias;
    const float *__restrict__ A;
    float *ssm;
    float q_scale;
    const int32_t *__restrict__ slot_map;
    float *xc;
    float *__restrict__ o;
    int32_t *status;
    int S, P, Hk, Hv, C;
};

__global__ void __launch_bounds__(256) decode_preflight_kernel(const DecodeArgs a) {
    gdn::grid_dep_launch();
    gdn::grid_dep_wait();  // status
    const int s = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (s >= a.S) return;
    const int slot = a.slot_map[s];
    int err = 0;
    if (slot < 0 || slot >= a.P) {
        err = GDN_DEV_BAD_SLOT;
    } else {
        bool dup = false;
        for (int s2 = lane; s2 < a.S; s2 += 32) dup |= (s2 != s && a.slot_map[s2] == slot);
        if (__any_sync(0xffffffffu, dup)) err = GDN_DEV_DUP_SLOT;
    }
    if (err && lane == 0) gdn::record_status(a.status, err);
}

constexpr int kConvThreads = 128;

__global__ void __launch_bounds__(kConvThreads) decode_conv_kernel(const DecodeArgs a) {
    gdn::grid_dep_launch();
    const int s = blockIdx.y;
    const int c4 = blockIdx.x * kConvThreads + threadIdx.x;  // float4 channel group
    const int slot = a.slot_map[s];
    gdn::grid_dep_wait();  // status, the history pool
    if (*reinterpret_cast<volatile int32_t *>(a.status) != 0 || slot < 0 || slot >= a.P) return;
    if (4 * c4 >= a.C) return;
    const int64_t C = a.C;
    const float4 *w4 = reinterpret_cast<const float4 *>(a.w) + 4 * int64_t(c4);
    const float4 wc0 = __ldg(w4 + 0), wc1 = __ldg(w4 + 1), wc2 = __ldg(w4 + 2), wc3 = __ldg(w4 + 3);
    float4 *hb = reinterpret_cast<float4 *>(a.hist + int64_t(slot) * 3 * C) + c4;
    const float4 h0 = hb[0], h1 = hb[C / 4], h2 = hb[2 * (C / 4)];
    const float4 xv = __ldg(reinterpret_cast<const float4 *>(a.x + int64_t(s) * a.x_stride) + c4);
    // taps j = 0 (h0, oldest) .. 3 (the token), accumulated in that order
    float4 acc;
    acc.x = fmaf(xv.x, wc0.w, fmaf(h2.x, wc0.z, fmaf(h1.x, wc0.y, fmaf(h0.x, wc0.x, 0.0f))));
    acc.y = fmaf(xv.y, wc1.w, fmaf(h2.y, wc1.z, fmaf(h1.y, wc1.y, fmaf(h0.y, wc1.x, 0.0f))));
    acc.z = fmaf(xv.z, wc2.w, fmaf(h2.z, wc2.z, fmaf(h1.z, wc2.y, fmaf(h0.z, wc2.x, 0.0f))));
    acc.w = fmaf(xv.w, wc3.w, fmaf(h2.w, wc3.z, fmaf(h1.w, wc3.y, fmaf(h0.w, wc3.x, 0.0f))));
    reinterpret_cast<float4 *>(a.xc + int64_t(s) * C)[c4] =
        make_float4(gdn::silu_f(acc.x), gdn::silu_f(acc.y), gdn::silu_f(acc.z), gdn::silu_f(acc.w));
    hb[0] = h1;
    hb[C / 4] = h2;
    hb[2 * (C / 4)] = xv;
}

// sum over the `width` consecutive lanes of each segment (width a power of two)
template <int W>
__device__ __forceinline__ float segment_sum(float v) {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
__global__ void __launch_bounds__(128) decode_recur_kernel(const DecodeArgs a) {
    constexpr int V4 = D / 4;          // lanes per state row
    constexpr int RPI = 32 / V4;       // rows one warp instruction covers
    gdn::grid_dep_launch();
    const int h = blockIdx.x, s = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = a.slot_map[s];
    gdn::grid_dep_wait();  // status, xc from the conv, the state pool
    if (*reinterpret_cast<volatile int32_t *>(a.status) != 0 || slot < 0 || slot >= a.P) return;
    const int64_t C = a.C;
    const int kh = h / (a.Hv / a.Hk);
    const float *xcs = a.xc + int64_t(s) * C;
    const int cl = lane % V4;          // this lane's float4 column group of a row
    const int rl = lane / V4;          // this lane's row within a warp instruction
    // q^ and k^: every warp normalises both (segment sums over the row's lanes)
    const float4 qv = reinterpret_cast<const float4 *>(xcs + kh * D)[cl];
    const float4 kv = reinterpret_cast<const float4 *>(xcs + a.Hk * D + kh * D)[cl];
    float sq = qv.x * qv.x, sk = kv.x * kv.x;
    sq = fmaf(qv.y, qv.y, sq);
    sq = fmaf(qv.z, qv.z, sq);
    sq = fmaf(qv.w, qv.w, sq);
    sk = fmaf(kv.y, kv.y, sk);
    sk = fmaf(kv.z, kv.z, sk);
    sk = fmaf(kv.w, kv.w, sk);
    sq = segment_sum<V4>(sq);
    sk = segment_sum<V4>(sk);
    const float rq = rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
    const float4 qn = make_float4(qv.x * rq, qv.y * rq, qv.z * rq, qv.w * rq);
    const float4 kn = make_float4(kv.x * rk, kv.y * rk, kv.z * rk, kv.w * rk);
    const float beta = gdn::sigmoid_f(__ldg(a.ba + int64_t(s) * a.ba_stride + h));
    const float decay = expf(gdn::softplus_f(__ldg(a.ba + int64_t(s) * a.ba_stride + a.Hv + h) + __ldg(a.dt_bias + h)) *
                             __ldg(a.A + h));
    const float *vrow = xcs + 2 * a.Hk * D + h * D;
    float *Sb = a.ssm + (int64_t(slot) * a.Hv + h) * D * D;
    float *ob = a.o + (int64_t(s) * a.Hv + h) * D;
#pragma unroll 4
    for (int r0 = warp * RPI; r0 < D; r0 += 4 * RPI) {
        const int r = r0 + rl;
        float4 *p = reinterpret_cast<float4 *>(Sb + int64_t(r) * D) + cl;
        float4 sv = *p;
        sv = make_float4(decay * sv.x, decay * sv.y, decay * sv.z, decay * sv.w);  // S' = decay S
        float d1 = gdn::fma4(sv, kn, 0.f);
        d1 = segment_sum<V4>(d1);                                                    // S' k^ (row r)
        const float u = beta * (__ldg(vrow + r) - d1);
        sv = make_float4(fmaf(u, kn.x, sv.x), fmaf(u, kn.y, sv.y), fmaf(u, kn.z, sv.z), fmaf(u, kn.w, sv.w));
        *p = sv;
        float d2 = gdn::fma4(sv, qn, 0.f);
        d2 = segment_sum<V4>(d2);                                                    // S q^ (row r)
        if (cl == 0) ob[r] = a.q_scale * d2;
    }
}

}  // namespace

extern "C" int gdn_decode_step(const gdn_dims *dims, const float *x, int64_t x_stride, const float *conv_w,
                               float *conv_hist, const float *ba, int64_t ba_stride, const float *dt_bias,
                               const float *A, float *ssm, float q_scale, const int32_t *slot_map, float *xc,
                               float *o, int32_t *status, void *stream) {
    int rc = gdn::check_dims(dims);
    if (rc) return rc;
    const int64_t S = dims->n_seqs, P = dims->n_slots, Hv = dims->h_v, D = dims->d_k;
    const int64_t C = gdn::conv_channels(dims);
    if (dims->n_nodes != dims->n_seqs) return GDN_ERR_DIMS;  // one token per sequence
    if (!status) return GDN_ERR_NULL;
    if (S == 0) return GDN_OK;
    if (!x || !conv_w || !conv_hist || !ba || !dt_bias || !A || !ssm || !slot_map || !xc || !o)
        return GDN_ERR_NULL;
    if (x_stride < C || x_stride % 4 != 0 || ba_stride < 2 * Hv) return GDN_ERR_STRIDE;
    if (!gdn::aligned16(x) || !gdn::aligned16(conv_w) || !gdn::aligned16(conv_hist) || !gdn::aligned16(ssm) ||
        !gdn::aligned16(xc) || !gdn::aligned16(o))
        return GDN_ERR_ALIGN;
    const gdn::Span outs[] = {{conv_hist, size_t(P * 3 * C * 4)},
                              {ssm, size_t(P * Hv * D * D * 4)},
                              {xc, size_t(S * C * 4)},
                              {o, size_t(S * Hv * D * 4)}};
    const gdn::Span ins[] = {{x, gdn::strided_bytes(S, x_stride, C)},
                             {conv_w, size_t(C * 16)},
                             {ba, gdn::strided_bytes(S, ba_stride, 2 * Hv)},
                             {dt_bias, size_t(Hv * 4)},
                             {A, size_t(Hv * 4)},
                             {slot_map, size_t(S * 4)},
                             {status, 4}};
    if ((rc = gdn::check_alias(outs, 4, ins, 7))) return rc;

    DecodeArgs a{x, x_stride, conv_w, conv_hist, ba, ba_stride, dt_bias, A, ssm, q_scale, slot_map, xc, o, status,
                 int(S), int(P), dims->h_k, int(Hv), int(C)};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (gdn::launch_pdl(decode_preflight_kernel, dim3(unsigned((S + 7) / 8)), dim3(256), 0, st, a) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const dim3 cgrid{unsigned((C / 4 + kConvThreads - 1) / kConvThreads), unsigned(S)};
    if (gdn::launch_pdl(decode_conv_kernel, cgrid, dim3(kConvThreads), 0, st, a) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const dim3 rgrid{unsigned(Hv), unsigned(S)};
    cudaError_t e;
    switch (D) {
        case 16: e = gdn::launch_pdl(decode_recur_kernel<16>, rgrid, dim3(128), 0, st, a); break;
        case 32: e = gdn::launch_pdl(decode_recur_kernel<32>, rgrid, dim3(128), 0, st, a); break;
        case 64: e = gdn::launch_pdl(decode_recur_kernel<64>, rgrid, dim3(128), 0, st, a); break;
        default: e = gdn::launch_pdl(decode_recur_kernel<128>, rgrid, dim3(128), 0, st, a); break;
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}
