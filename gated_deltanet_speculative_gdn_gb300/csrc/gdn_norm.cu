// gdn_norm.cu - gated RMS norm of the verify output: the output stage that
// follows the gated delta rule in the GDN block.
//
// TensorSharp PR #175 "Feature/support dflash2", the Qwen 3.5 / Qwen4Exp GDN
// block: conv -> gated delta net -> gated norm -> scatter; the output gate is
// a SiLU (gate_mode 0, the existing callers) or a sigmoid (gate_mode 1).
//
// One warp per (node, value head) row of d floats: lane l holds floats
// 4l .. 4l + 3 (128-bit loads of o, z and the weight), the sum of squares is a
// warp reduction, and y = o / sqrt(mean(o^2) + eps) * w * gate(z) is stored
// with 128-bit stores.  HBM-bound: per row it reads o and z and writes y.
#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace {

constexpr int kRowsPerCta = 8;  // one warp per row

struct NormArgs {
    const float *__restrict__ o;
    const float *__restrict__ z;
    int64_t z_stride;
    const float *__restrict__ w;
    float eps;
    int gate_mode;
    float *__restrict__ y;
    int64_t rows;  // N * H_v
    int Hv;
};

template <int D>
__global__ void __launch_bounds__(kRowsPerCta * 32) gated_rmsnorm_kernel(const NormArgs a) {
    constexpr int V4 = D / 4;  // float4 per row, 4 .. 32
    gdn::grid_dep_launch();
    gdn::grid_dep_wait();  // o comes from the verify launched before on this stream
    const int64_t row = int64_t(blockIdx.x) * kRowsPerCta + (threadIdx.x >> 5);
    if (row >= a.rows) return;
    const int lane = threadIdx.x & 31;
    const int64_t t = row / a.Hv;
    const int h = int(row - t * a.Hv);
    float4 ov = make_float4(0.f, 0.f, 0.f, 0.f), zv = ov, wv = ov;
    if (lane < V4) {
        ov = __ldcs(reinterpret_cast<const float4 *>(a.o + row * D) + lane);
        zv = __ldcs(reinterpret_cast<const float4 *>(a.z + t * a.z_stride + int64_t(h) * D) + lane);
        wv = __ldg(reinterpret_cast<const float4 *>(a.w) + lane);
    }
    float ss = ov.x * ov.x;
    ss = fmaf(ov.y, ov.y, ss);
    ss = fmaf(ov.z, ov.z, ss);
    ss = fmaf(ov.w, ov.w, ss);
    ss = gdn::warp_sum(ss);
    const float inv = 1.0f / sqrtf(ss * (1.0f / D) + a.eps);
    if (lane < V4) {
        float4 g;
        if (a.gate_mode == 0) {
            g = make_float4(gdn::silu_f(zv.x), gdn::silu_f(zv.y), gdn::silu_f(zv.z), gdn::silu_f(zv.w));
        } else {
            g = make_float4(gdn::sigmoid_f(zv.x), gdn::sigmoid_f(zv.y), gdn::sigmoid_f(zv.z), gdn::sigmoid_f(zv.w));
        }
        const float4 yv = make_float4(ov.x * inv * wv.x * g.x, ov.y * inv * wv.y * g.y, ov.z * inv * wv.z * g.z,
                                      ov.w * inv * wv.w * g.w);
        __stcs(reinterpret_cast<float4 *>(a.y + row * D) + lane, yv);
    }
}

}  // namespace

extern "C" int gdn_gated_rmsnorm(const gdn_dims *dims, const float *o, const float *z, int64_t z_stride,
                                 const float *norm_w, float eps, int gate_mode, float *y, void *stream) {
    int rc = gdn::check_dims(dims);
    if (rc) return rc;
    const int64_t N = dims->n_nodes, Hv = dims->h_v, D = dims->d_v;
    if (N == 0) return GDN_OK;
    if (!o || !z || !norm_w || !y) return GDN_ERR_NULL;
    if (gate_mode != 0 && gate_mode != 1) return GDN_ERR_ARG;
    if (!(eps >= 0.0f) || !(eps < 3.0e38f)) return GDN_ERR_ARG;
    if (z_stride < Hv * D || z_stride % 4 != 0) return GDN_ERR_STRIDE;
    if (!gdn::aligned16(o) || !gdn::aligned16(z) || !gdn::aligned16(norm_w) || !gdn::aligned16(y))
        return GDN_ERR_ALIGN;
    const gdn::Span outs[] = {{y, size_t(N * Hv * D * 4)}};
    const gdn::Span ins[] = {{o, size_t(N * Hv * D * 4)},
                             {z, gdn::strided_bytes(N, z_stride, Hv * D)},
                             {norm_w, size_t(D * 4)}};
    if ((rc = gdn::check_alias(outs, 1, ins, 3))) return rc;
    NormArgs a{o, z, z_stride, norm_w, eps, gate_mode, y, N * Hv, int(Hv)};
    const dim3 grid(unsigned((N * Hv + kRowsPerCta - 1) / kRowsPerCta)), block(kRowsPerCta * 32);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (D) {
        case 16: e = gdn::launch_pdl(gated_rmsnorm_kernel<16>, grid, block, 0, st, a); break;
        case 32: e = gdn::launch_pdl(gated_rmsnorm_kernel<32>, grid, block, 0, st, a); break;
        case 64: e = gdn::launch_pdl(gated_rmsnorm_kernel<64>, grid, block, 0, st, a); break;
        default: e = gdn::launch_pdl(gated_rmsnorm_kernel<128>, grid, block, 0, st, a); break;
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}
