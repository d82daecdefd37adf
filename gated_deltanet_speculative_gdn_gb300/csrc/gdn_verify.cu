// gdn_verify.cu - tree verify: gated delta rule over each sequence's token tree,
// state read-only from its slot, gates and q/k L2 norm in the kernel, output and
// one replay row per (node, value head).
//
// lucebox PR #707 "perf(qwen35): fuse the DFlash2 concurrent verify Gated
// DeltaNet route", Optimizations: the recurrence reads the state directly from
// the owning slot and writes only the attention output and the replay log (no
// base-state copy, no final state, no per-token states); strided views of the
// stacked beta/alpha projection feed the kernel, which applies sigmoid and
// softplus with bias and scale itself.  lucebox PR #659 "perf(qwen38): various
// DFlash2 optimizations concurrency C1-C5", Summary item 3: replay width 2d+1.
//
// Method.  Rows of the state evolve independently: row i of S_t is
//     S_t[i,:] = Gamma_t S0[i,:] + sum_{j on path(t)} gamma_{j->t} u_j[i] k_j^T
// where Gamma_t is the product of the decays on the root..t path and
// gamma_{j->t} the product of those strictly after j.  So with
//     a_t = S0 k_t,  b_t = S0 q_t                     (one dense contraction)
//     KK[j][t] = k_j . k_t,  KQ[j][t] = k_j . q_t      (Gram terms)
// each node needs only
//     S' k_t = Gamma_t a_t + sum_{j on path(parent)} gamma_{j->t} KK[j][t] u_j
//     u_t    = beta_t (v_t - S' k_t)
//     o_t    = q_scale (Gamma_t b_t + sum_{j on path(t)} gamma_{j->t} KQ[j][t] u_j)
// and no per-node state is ever formed.  The decay products are plain
// products along the path (never ratios), so underflow only ever drops terms
// that are already below the float range.
//
// Mapping (GB300).  One CTA of 128 threads per (sequence, value head).  The
// d x d slot state is staged into shared memory by TMA (128-byte swizzle, so
// that lanes reading 8 consecutive rows hit 8 different banks) while the CTA
// loads and normalises q/k.  Nodes are processed in segments of 16; per
// segment the contraction [S0 | U_prev] x [Gamma k | Gamma q | coefficients]
// (d rows x 32 columns) runs as a register-tiled FFMA product (4 rows x 8
// columns per thread, broadcast column reads), followed by a per-row pass over
// the segment's nodes.  Terms from earlier segments enter the contraction as
// extra K columns (the u rows of earlier nodes), so chains up to 64 nodes keep
// the same dense form.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace {

constexpr int kThreads = 128;
constexpr int kSeg = 16;

template <int D, int NMAX>
struct Layout {
    static constexpr bool kMulti = NMAX > kSeg;
    static constexpr int BK = D + (NMAX - kSeg);  // contraction length (largest segment)
    static constexpr int BS = BK + 4;             // row stride of the column operand
    static constexpr int KS = D + 4;              // row stride of the k^ store
    static constexpr int US = NMAX + 4;           // row stride of the u store
    // float offsets from the 1024-byte aligned base
    static constexpr int S0 = 0;
    static constexpr int BOP = S0 + D * D;
    static constexpr int KH = BOP + 32 * BS;
    static constexpr int R = KH + (kMulti ? NMAX * KS : 0);
    static constexpr int U = R + 32 * D;
    static constexpr int G = U + (kMulti ? D * US : 0);
    static constexpr int CK = G + NMAX * 32;
    static constexpr int CQ = CK + kSeg * kSeg;
    static constexpr int BETA = CQ + kSeg * kSeg;
    static constexpr int DEC = BETA + NMAX;
    static constexpr int GAM = DEC + NMAX;
    static constexpr int PAR = GAM + kSeg;
    static constexpr int BAR = (PAR + NMAX + 1) & ~1;
    static constexpr int FLOATS = BAR + 2;
    static constexpr size_t BYTES = size_t(FLOATS) * 4 + 1024;
};

struct VerifyArgs {
    const float *__restrict__ xc;
    const float *__restrict__ ba;
    int64_t ba_stride;
    const float *__restrict__ dt_bias;
    const float *__restrict__ A;
    float q_scale;
    const int32_t *__restrict__ parents;
    const int32_t *__restrict__ node_off;
    const int32_t *__restrict__ slot_map;
    float *__restrict__ o;
    float *__restrict__ replay;
    int64_t rstride;
    int32_t *status;
    int S, N, P, Hk, Hv, C, max_nodes;
    uint64_t stall_ns;  // test hook: a wait that nothing ends, for this long (0: none)
};

// Row `row`, float4 column group `kc` of the TMA-staged state.  For d >= 32 the
// state arrives as d/32 boxes of [d rows][32 floats] in the 128-byte swizzle:
// 16-byte chunk c of row r sits at chunk c ^ (r & 7).
template <int D>
__device__ __forceinline__ float4 ld_state(const float *s0, int row, int kc) {
    if constexpr (D >= 32) {
        const char *p = reinterpret_cast<const char *>(s0) + (kc >> 3) * (D * 128) + row * 128 +
                        (((kc & 7) ^ (row & 7)) << 4);
        return *reinterpret_cast<const float4 *>(p);
    } else {
        return *reinterpret_cast<const float4 *>(s0 + row * D + 4 * kc);
    }
}

__device__ __forceinline__ float4 scale4(float4 v, float s) {
    return make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
}

template <int D, int NMAX>
__global__ void __launch_bounds__(kThreads, (NMAX > kSeg ? 1 : 2))
    tree_verify_kernel(const __grid_constant__ CUtensorMap tmap, const VerifyArgs a) {
    using L = Layout<D, NMAX>;
    constexpr bool kMulti = L::kMulti;
    constexpr int RT = D >= 32 ? D / 32 : 1;  // rows per lane in the contraction
    constexpr int DV4 = D / 4;
    constexpr int BS = L::BS, KS = L::KS, US = L::US;

    extern __shared__ unsigned char smem_raw[];
    float *sm = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *s0 = sm + L::S0;
    float *bop = sm + L::BOP;                      // [32][BS]: Gamma k^ | Gamma q^ columns + coefficients
    float *khat = kMulti ? sm + L::KH : bop;       // [NMAX][KS] unscaled k^ (single segment: bop rows)
    float *res = sm + L::R;                        // [32][D] contraction result
    float *uall = sm + L::U;                       // [D][US] u of earlier nodes (multi-segment)
    float *gram = sm + L::G;                       // [NMAX][32]
    float *cks = sm + L::CK, *cqs = sm + L::CQ;    // [16][16] in-segment coefficients
    float *beta_s = sm + L::BETA, *dec_s = sm + L::DEC, *gam_s = sm + L::GAM;
    int *par = reinterpret_cast<int *>(sm + L::PAR);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::BAR);
    __shared__ int hdr[4];  // error, first node, node count, slot

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, s = blockIdx.y;
    const int kh = h / (a.Hv / a.Hk);
    gdn::grid_dep_launch();
    gdn::grid_dep_wait();  // xc, the state pool, status

    if (tid == 0) {
        const int n0 = a.node_off[s], n1 = a.node_off[s + 1];
        int err = 0;
        if (n0 < 0 || n1 < n0 || n1 > a.N || (s == 0 && n0 != 0) || (s == a.S - 1 && n1 != a.N) ||
            n1 - n0 > a.max_nodes || n1 - n0 > NMAX)
            err = GDN_DEV_BAD_NODE_OFF;
        const int slot = a.slot_map[s];
        if (!err && (slot < 0 || slot >= a.P)) err = GDN_DEV_BAD_SLOT;
        hdr[0] = err;
        hdr[1] = n0;
        hdr[2] = n1 - n0;
        hdr[3] = slot;
    }
    __syncthreads();
    if (hdr[0] || hdr[2] == 0) {
        if (tid == 0 && hdr[0]) gdn::record_status(a.status, hdr[0]);
        return;
    }
    const int n0 = hdr[1], ns = hdr[2], slot = hdr[3];
    for (int i = tid; i < ns; i += kThreads) {
        const int p = a.parents[n0 + i];
        par[i] = p;
        if (p < -1 || p >= i) hdr[0] = GDN_DEV_BAD_PARENT;
    }
    if (tid == 0) {
        gdn::mbar_init(bar, 1);
        gdn::fence_mbar_init();
    }
    __syncthreads();
    if (hdr[0]) {
        if (tid == 0) gdn::record_status(a.status, hdr[0]);
        return;
    }
    // stage S0 = ssm[slot][h] (d x d) while the first segment's q/k are prepared
    if (tid == 0) {
        gdn::mbar_arrive_expect_tx(bar, D * D * 4);
        const int y = (slot * a.Hv + h) * D;
        if constexpr (D >= 32) {
#pragma unroll
            for (int b = 0; b < D / 32; ++b) gdn::tma_load_2d(s0 + b * D * 32, &tmap, 32 * b, y, bar);
        } else {
            gdn::tma_load_2d(s0, &tmap, 0, y, bar);
        }
    }

    const int64_t C = a.C;
    const int qoff = kh * D, koff = a.Hk * D + kh * D, voff = 2 * a.Hk * D + h * D;
    const float dtb = a.dt_bias[h], Ah = a.A[h];

    for (int g16 = 0; g16 < ns; g16 += kSeg) {
        const int lc = min(kSeg, ns - g16);

        // ---- A: v of this row, gates, normalised q and k ---------------------
        float vreg[kSeg];
#pragma unroll
        for (int t = 0; t < kSeg; ++t)
            vreg[t] = (t < lc && tid < D) ? __ldg(a.xc + (n0 + g16 + t) * C + voff + tid) : 0.0f;
        if (warp == 0 && lane < lc) {
            const int tl = g16 + lane;
            const int64_t n = n0 + tl;
            const float bv = __ldg(a.ba + n * a.ba_stride + h);
            const float av = __ldg(a.ba + n * a.ba_stride + a.Hv + h);
            const float dec = expf(gdn::softplus_f(av + dtb) * Ah);
            beta_s[tl] = gdn::sigmoid_f(bv);
            dec_s[tl] = dec;
            a.replay[(n * a.Hv + h) * a.rstride + 2 * D] = dec;
        }
        {
            // vector vi < lc: k of node vi; lc <= vi < 2 lc: q of node vi - lc
            constexpr int VPW = 2 * kSeg / 4;
            float4 val[VPW];
#pragma unroll
            for (int j = 0; j < VPW; ++j) {
                const int vi = warp + 4 * j;
                val[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (vi < 2 * lc && lane < DV4) {
                    const bool isk = vi < lc;
                    const int t = isk ? vi : vi - lc;
                    val[j] = __ldg(reinterpret_cast<const float4 *>(a.xc + (n0 + g16 + t) * C +
                                                                    (isk ? koff : qoff) + 4 * lane));
                }
            }
#pragma unroll
            for (int j = 0; j < VPW; ++j) {
                const int vi = warp + 4 * j;
                float ss = val[j].x * val[j].x;
                ss = fmaf(val[j].y, val[j].y, ss);
                ss = fmaf(val[j].z, val[j].z, ss);
                ss = fmaf(val[j].w, val[j].w, ss);
                ss = gdn::warp_sum(ss);
                const float inv = rsqrtf(ss + 1e-6f);
                if (vi < 2 * lc && lane < DV4) {
                    const float4 nv = scale4(val[j], inv);
                    if (vi < lc) {
                        const int t = vi;
                        *reinterpret_cast<float4 *>(khat + (g16 + t) * KS + 4 * lane) = nv;
                        *reinterpret_cast<float4 *>(a.replay + ((n0 + g16 + t) * int64_t(a.Hv) + h) * a.rstride +
                                                    4 * lane) = nv;
                    } else {
                        *reinterpret_cast<float4 *>(bop + (kSeg + vi - lc) * BS + 4 * lane) = nv;
                    }
                }
            }
        }
        __syncthreads();

        // ---- B: Gram rows j < g16 + lc against this segment's k^ and q^ -------
        {
            const int e = g16 + lc;
            const int jl = tid & 15, cg = tid >> 4;  // 16 rows x 8 groups of 4 columns
            const float *colp[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = 4 * cg + c;
                colp[c] = col < kSeg ? khat + (g16 + col) * KS : bop + col * BS;
            }
#pragma unroll
            for (int r = 0; r < NMAX / kSeg; ++r) {
                if (16 * r < e) {
                    const int j = jl + 16 * r;
                    const float *krow = khat + j * KS;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int kc = 0; kc < DV4; ++kc) {
                        const float4 kv = *reinterpret_cast<const float4 *>(krow + 4 * kc);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            acc[c] = gdn::fma4(kv, *reinterpret_cast<const float4 *>(colp[c] + 4 * kc), acc[c]);
                    }
                    if (j < e) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) gram[j * 32 + 4 * cg + c] = acc[c];
                    }
                }
            }
        }
        __syncthreads();

        // ---- C: path coefficients and Gamma (one lane per node) ----------------
        if (warp == 0 && lane < kSeg) {
            const int t = lane;
#pragma unroll
            for (int j = 0; j < kSeg; ++j) {
                cks[t * kSeg + j] = 0.f;
                cqs[t * kSeg + j] = 0.f;
            }
            if constexpr (kMulti) {
                for (int j = 0; j < g16; ++j) {
                    bop[t * BS + D + j] = 0.f;
                    bop[(kSeg + t) * BS + D + j] = 0.f;
                }
            }
            float gam = 0.f;
            if (t < lc) {
                const int tl = g16 + t;
                cqs[t * kSeg + t] = gram[tl * 32 + kSeg + t];
                gam = dec_s[tl];
                for (int j = par[tl]; j >= 0; j = par[j]) {
                    const float ck = gam * gram[j * 32 + t];
                    const float cq = gam * gram[j * 32 + kSeg + t];
                    if (j >= g16) {
                        cks[t * kSeg + (j - g16)] = ck;
                        cqs[t * kSeg + (j - g16)] = cq;
                    } else {
                        bop[t * BS + D + j] = ck;
                        bop[(kSeg + t) * BS + D + j] = cq;
                    }
                    gam *= dec_s[j];
                }
            }
            gam_s[t] = gam;
        }
        __syncthreads();

        // ---- C2: column operand = Gamma_t k^_t | Gamma_t q^_t ------------------
        for (int idx = tid; idx < 32 * DV4; idx += kThreads) {
            const int row = idx / DV4, kc = idx - row * DV4;
            const float *srow = row < kSeg ? khat + (g16 + row) * KS : bop + row * BS;
            const float4 v = *reinterpret_cast<const float4 *>(srow + 4 * kc);
            *reinterpret_cast<float4 *>(bop + row * BS + 4 * kc) = scale4(v, gam_s[row & (kSeg - 1)]);
        }
        if (g16 == 0) {
            if (!gdn::mbar_wait_bounded(bar, 0)) hdr[0] = GDN_DEV_TIMEOUT;
        }
        __syncthreads();
        if (hdr[0]) {
            // the state copy never landed: wait once more (bounded) before leaving
            gdn::mbar_wait_bounded(bar, 0);
            if (tid == 0) gdn::record_status(a.status, hdr[0]);
            return;
        }

        // ---- D: [S0 | U_prev] x columns, d rows x 32 columns ------------------
        {
            const int cb = 8 * warp;
            const int rowl = D >= 32 ? lane : (lane & 15);
            float acc[RT][8];
#pragma unroll
            for (int m = 0; m < RT; ++m)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[m][c] = 0.f;
#pragma unroll 2
            for (int kc = 0; kc < DV4; ++kc) {
                float4 av[RT];
#pragma unroll
                for (int m = 0; m < RT; ++m) av[m] = ld_state<D>(s0, rowl + 32 * m, kc);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 bv = *reinterpret_cast<const float4 *>(bop + (cb + c) * BS + 4 * kc);
#pragma unroll
                    for (int m = 0; m < RT; ++m) acc[m][c] = gdn::fma4(av[m], bv, acc[m][c]);
                }
            }
            if constexpr (kMulti) {
                for (int kc = 0; kc < g16 / 4; ++kc) {
                    float4 av[RT];
#pragma unroll
                    for (int m = 0; m < RT; ++m)
                        av[m] = *reinterpret_cast<const float4 *>(uall + (rowl + 32 * m) * US + 4 * kc);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 bv = *reinterpret_cast<const float4 *>(bop + (cb + c) * BS + D + 4 * kc);
#pragma unroll
                        for (int m = 0; m < RT; ++m) acc[m][c] = gdn::fma4(av[m], bv, acc[m][c]);
                    }
                }
            }
            if (D >= 32 || lane < 16) {
#pragma unroll
                for (int m = 0; m < RT; ++m)
#pragma unroll
                    for (int c = 0; c < 8; ++c) res[(cb + c) * D + rowl + 32 * m] = acc[m][c];
            }
        }
        __syncthreads();

        // ---- E: per row, the segment's nodes in order --------------------------
        if (tid < D) {
            float u[kSeg];
#pragma unroll
            for (int t = 0; t < kSeg; ++t) {
                u[t] = 0.f;
                if (t < lc) {
                    const int tl = g16 + t;
                    const int64_t n = n0 + tl;
                    float sk = res[t * D + tid];
#pragma unroll
                    for (int j = 0; j < t; ++j) sk = fmaf(cks[t * kSeg + j], u[j], sk);
                    u[t] = beta_s[tl] * (vreg[t] - sk);
                    float oq = res[(kSeg + t) * D + tid];
#pragma unroll
                    for (int j = 0; j <= t; ++j) oq = fmaf(cqs[t * kSeg + j], u[j], oq);
                    a.o[(n * a.Hv + h) * D + tid] = a.q_scale * oq;
                    a.replay[(n * a.Hv + h) * a.rstride + D + tid] = u[t];
                    if constexpr (kMulti) uall[tid * US + tl] = u[t];
                }
            }
        }
        __syncthreads();
    }
}

// ============================================================================
// Tensor-core variant for d = 128 and trees of at most 16 nodes: a persistent,
// warp-specialised pipeline.
//
// Per (sequence, value head) "item" the contraction
//     D[i][c] = sum_k S0[i][k] B[c][k],   B = [k_0..k_15 | q_0..q_15]   (raw rows)
// is a 128 x 32 x 128 matrix product on tcgen05 with accumulators in tensor
// memory.  Every operand is split as x = hi + lo, hi = x with the low 13
// mantissa bits cleared (a tf32 number) and lo = x - hi (exact in fp32), and
// all four products run as tf32:
//     D = A_hi [B_hi | B_lo] + A_lo [B_hi | B_lo]
// The tensor cores read an fp32 operand as its hi part, so S0 and the raw B
// rows feed the hi operands unchanged and only the lo parts are written out
// (as fp32).  tf32 keeps fp32's exponent range, so the split is exact at any
// scale of the state or of q/k; the lo parts keep 11 bits, which puts the
// product at ~2^-21 of fp32.  A tensor-core instruction costs about the same
// for any N up to 256, so B_hi and B_lo always travel together as N = 64.
// The tensor cores align and truncate when they accumulate, so the large
// A_hi B_hi terms get one short accumulator per K-half and the small terms one
// of their own; the epilogue adds them in fp32, smallest first.
//
// B holds the raw q/k rows, so the products start as soon as they land; the
// epilogue scales column c by 1/|k_c| or 1/|q_c|, which equals S0 k^ up to
// rounding.  The Gram terms of B with itself (k . k, q . k and the norms)
// come from the tensor cores as well: M = N = 64 products of B's rows
// [k | q | k_lo | q_lo] with themselves, so hi x hi, hi x lo, lo x hi and
// lo x lo all appear.
//
// The tree is then solved in closed form.  With Ck[t][j] = gamma_{j->t}
// k^_j . k^_t for j a strict ancestor of t and L = diag(beta) Ck, the node
// updates u_t = beta_t (v_t - Gamma_t a_t - sum_j Ck[t][j] u_j) read
//     (I + L) u = r,   r_t = beta_t (v_t - Gamma_t a_t)
// so u = T r with T = (I + L)^-1, a unit lower-triangular 16 x 16 matrix that
// is the same for all 128 state rows (the UT transform of the chunked delta
// rule, restricted to the tree's ancestor pattern).  Likewise
// o = q_scale (Gamma b + Cq u).  One warp forms T per item; every state row
// then needs two small triangular matrix-vector products (u = T r, then
// o from u) instead of a 16-step serial chain.
//
// Two measured properties of GB300 shape the pipeline.  A thread that issues
// tcgen05.mma waits about 200 cycles per instruction whatever its shape,
// while several issuing warps proceed side by side; so each kind of product
// has an issuer warp of its own.  And a 16 KB S0 chunk arrives some 4 us after
// its TMA load when every SM streams state, so each SM needs well over 100 KB
// of loads in flight; so the lo part of a chunk is written over the chunk
// itself once its A_hi products have read it, and shared memory goes to a
// deep ring of S0 slots.
//
// One CTA per SM walks a list of items.  Warp roles:
//   warp 0       TMA producer, items in order: the item's q/k rows into B
//                buffer v % NB (same layout as the chunks) once the item NB
//                before it is done with that buffer, then S0 as four 16 KB
//                K-chunks ([128 rows][32 floats], 128-byte swizzle = the
//                tensor cores' K-major operand layout) into a ring of NR slots;
//   warps 1-3    MMA issuers, items and chunks in order: the Gram terms once
//                the item's B is split (warp 1); A_hi [B_hi | B_lo] once a
//                chunk lands (warp 2); A_lo [B_hi | B_lo] once the chunk holds
//                its lo part, which frees the slot (warp 3);
//   warps 4-7    team 0 and warps 8-11 team 1, on alternate items: gates, the
//                ancestor decays, norms and path coefficients from the Gram
//                terms, T, and the per-row epilogue reading the accumulators
//                from tensor memory (thread i owns state row i);
//   warps 12-15  splitters, items in order: B's lo rows as soon as the item's
//                q/k rows land, then the lo part of every S0 chunk, in place,
//                as soon as its A_hi products are done.
// With three B buffers for two teams, an item's q/k rows land while the
// previous items still use theirs, and the S0 ring runs ahead of both teams,
// so loads, tensor-core work and CUDA-core work of different items overlap.
namespace wsv {
constexpr int D = 128;
constexpr int kWarps = 16;
constexpr int kThreadsWS = kWarps * 32;
constexpr int kIssueGram = 1, kIssueHi = 2;       // MMA issuer warps (warp 3 issues the A_lo products)
constexpr int kTeam0 = 4;                          // team t: warps 4 + 4t .. 7 + 4t
constexpr int kSplit0 = 12, kSplitThreads = 128;   // splitter warps 12-15
constexpr int kMaxItems = 64;                      // items per CTA
constexpr int NR = 6;                              // S0 ring depth (K-chunks)
constexpr int kPrefetch = 2;                       // items whose state is requested into L2 ahead
constexpr uint32_t kChunk = 128 * 128;             // one S0 K-chunk: 128 rows x 32 fp32
constexpr uint32_t kBChunk = 64 * 128;             // one B K-chunk: rows 0-15 k, 16-31 q, 32-63 their lo
constexpr uint32_t kBTeam = 4 * kBChunk;           // one item's B
constexpr int NB = 3;                              // B buffers, item v in buffer v % NB
constexpr uint32_t kQKBox = 16 * 128;              // 16 rows of k or q, one K-chunk
constexpr uint32_t RAW = 0;
constexpr uint32_t BT = RAW + NR * kChunk;         // per team
constexpr uint32_t kStage = 16 * D * 4;            // one [16 nodes][d] tile
constexpr uint32_t VT = BT + NB * kBTeam;          // per team: the item's v rows
constexpr uint32_t SMALL = VT + 2 * kStage;
// per-team small area (4-byte words), [16][16] matrices:
//   KA + KB = k_t . k_j and QA + QB = q_t . k_j (Gram partial sums from the
//   hi and lo rows, row t); GM = gamma_{j->t} (row t; 1 on the diagonal, 0
//   off the path); LNT = -L transposed (row j holds column j of -L, with
//   L = beta_t Ck); CQT = q_scale Cq transposed (row j holds column j).
//   QQA + QQB = q_t . q_t; gates, parents, Gamma_t / |k_t| (GSK),
//   q_scale Gamma_t / |q_t| (GSQ), 1 / |k_t| (RK), Gamma_t (GAM).
constexpr int T_KA = 0, T_KB = 256, T_QA = 512, T_QB = 768, T_GM = 1024, T_CQT = 1280, T_BETA = 1536,
              T_DEC = 1552, T_GSK = 1568, T_PAR = 1584, T_GSQ = 1600, T_QQA = 1616, T_QQB = 1632,
              T_RK = 1648, T_GAM = 1664, T_LNT = 1680, T_WORDS = 1936;
// mbarriers
constexpr int B_RFULL = 0;                 // NR: S0 chunk landed
constexpr int B_HDONE = B_RFULL + NR;      // NR: the chunk's A_hi products done (1)
constexpr int B_LFULL = B_HDONE + NR;      // NR: its lo part written in place (64)
constexpr int B_REMPTY = B_LFULL + NR;     // NR: the lo part's products done, slot free (1)
constexpr int B_QFULL = B_REMPTY + NR;     // per B buffer: q/k rows landed (1 + bytes)
constexpr int B_BREADY = B_QFULL + NB;     // per B buffer: its lo rows written (128)
constexpr int B_BFREE = B_BREADY + NB;     // per B buffer: the item is done with it (1 from each
                                           // product issuer, 1 from the team)
constexpr int B_GFULL = B_BFREE + NB;      // per team: Gram terms complete (1)
constexpr int B_ACCFULL = B_GFULL + 2;     // per team: accumulators complete (1 from each product issuer)
constexpr int B_ACCEMPTY = B_ACCFULL + 2;  // per team: accumulators read (128)
constexpr int B_VFULL = B_ACCEMPTY + 2;    // per team: the item's v rows landed in its u tile (1 + bytes)
constexpr int B_DRAIN = B_VFULL + 2;       // the issuers' last tensor-core work done (1 from each)
constexpr int B_NEVER = B_DRAIN + 1;       // nothing arrives: the timeout test's wait
constexpr int N_BARS = B_NEVER + 1;
constexpr int W_BARS = 2 * T_WORDS;
constexpr int W_TMEM = W_BARS + 2 * N_BARS;
constexpr int W_ABORT = W_TMEM + 1;
constexpr int W_NV = W_ABORT + 1;
constexpr int W_ERR = W_NV + 1;                    // an index error found during set-up
constexpr int W_LIST = (W_ERR + 4) & ~3;           // kMaxItems x int4 (item, n0, ns, slot), 16-B aligned
constexpr int SMALL_WORDS = W_LIST + 4 * kMaxItems;
constexpr size_t BYTES = SMALL + SMALL_WORDS * 4 + 1024;
static_assert(BYTES <= 227 * 1024, "shared memory");
static_assert((W_BARS % 2) == 0, "mbarriers are 8-byte aligned");
static_assert((T_WORDS % 4) == 0 && (T_GM % 4) == 0 && (T_CQT % 4) == 0, "float4 rows");
// instruction descriptors: fp32 accumulate, tf32 x tf32, K-major operands;
// M = 128, N = 64 for the contraction and M = N = 64 for the Gram terms
constexpr uint32_t IDESC_TF32 = (1u << 4) | (2u << 7) | (2u << 10) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t IDESC_GRAM = (1u << 4) | (2u << 7) | (2u << 10) | ((64u >> 3) << 17) | ((64u >> 4) << 24);
// Team t's accumulators start at column 256 t: K-half kh (chunks 2 kh, 2 kh + 1)
// owns columns 64 kh .. 64 kh + 63, A_hi B_hi in the first 32 and A_hi B_lo in
// the last 32; A_lo B_hi and A_lo B_lo of all four K-chunks sit at 128 and 160.
// The Gram terms G of B's 64 rows with themselves (M = 64: row a of G in lane
// 32 (a / 16) + a % 16) sit at 192.
constexpr uint32_t TMEM_COLS = 512, TEAM_COLS = 256, LHCOL = 128, GCOL = 192;

__device__ __forceinline__ uint32_t sw_off(int row, int k, uint32_t chunk) {
    return uint32_t(k >> 5) * chunk + uint32_t(row) * 128u + ((uint32_t(((k & 31) >> 2) ^ (row & 7))) << 4) +
           uint32_t(k & 3) * 4u;
}
__device__ __forceinline__ void team_sync(int team) {
    asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(128) : "memory");
}
// A wait that gives up at once after any role has timed out (the CTA then
// drains and exits), and otherwise waits at most the library's wait limit.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (*abort_flag) return false;
    if (gdn::mbar_wait_bounded(bar, parity)) return true;
    *abort_flag = 1;
    return false;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gdn::smem_addr(bar)) : "memory");
}
// x - (x with the low 13 mantissa bits cleared), exact
__device__ __forceinline__ float4 lo4(float4 x) {
    return make_float4(x.x - gdn::tf32_hi(x.x), x.y - gdn::tf32_hi(x.y), x.z - gdn::tf32_hi(x.z),
                       x.w - gdn::tf32_hi(x.w));
}
}  // namespace wsv

__global__ void __launch_bounds__(wsv::kThreadsWS, 1)
    tree_verify_ws_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap xmap,
                          const __grid_constant__ CUtensorMap vmap, const VerifyArgs a) {
    using namespace wsv;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sb =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = gdn::smem_addr(sb);
    int *words = reinterpret_cast<int *>(sb + SMALL);
    uint64_t *bars = reinterpret_cast<uint64_t *>(words + W_BARS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(words + W_TMEM);
    volatile int *abort_flag = words + W_ABORT;
    int4 *list = reinterpret_cast<int4 *>(words + W_LIST);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = a.S * a.Hv;
    gdn::grid_dep_launch();

    // ---- set-up: this CTA's valid items, barriers, tensor memory.  It reads
    //      only the caller's index inputs, so it runs before the wait for the
    //      previous kernel; so do L2 requests for the first items' states (a
    //      hint: whatever writes them later still lands in L2). --------------
    if (warp == 0) {
        if (lane == 0) words[W_ERR] = 0;
        __syncwarp();
        int nv = 0;
        for (int k0 = 0; k0 < kMaxItems; k0 += 32) {
            const int it = blockIdx.x + (k0 + lane) * gridDim.x;
            int n0 = 0, ns = 0, slot = 0, err = 0;
            if (k0 + lane < kMaxItems && it < total) {
                const int s = it / a.Hv;
                n0 = a.node_off[s];
                const int n1 = a.node_off[s + 1];
                slot = a.slot_map[s];
                ns = n1 - n0;
                if (n0 < 0 || n1 < n0 || n1 > a.N || (s == 0 && n0 != 0) || (s == a.S - 1 && n1 != a.N) ||
                    ns > a.max_nodes || ns > kSeg)
                    err = GDN_DEV_BAD_NODE_OFF;
                else if (ns > 0 && (slot < 0 || slot >= a.P))
                    err = GDN_DEV_BAD_SLOT;
                if (err) words[W_ERR] = err;  // recorded after the wait
            }
            const bool valid = k0 + lane < kMaxItems && it < total && !err && ns > 0;
            const unsigned m = __ballot_sync(0xffffffffu, valid);
            if (valid) list[nv + __popc(m & ((1u << lane) - 1u))] = make_int4(it, n0, ns, slot);
            nv += __popc(m);
        }
        if (lane == 0) words[W_NV] = nv;
    }
    if (tid == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            uint32_t count = 1;
            if (i >= B_LFULL && i < B_LFULL + NR) count = kSplitThreads;
            if (i >= B_BREADY && i < B_BREADY + NB) count = 128;
            if (i >= B_BFREE && i < B_BFREE + NB) count = 4;
            if (i >= B_ACCEMPTY && i < B_ACCEMPTY + 2) count = 128;
            if (i >= B_ACCFULL && i < B_ACCFULL + 2) count = 2;
            if (i == B_DRAIN) count = 3;
            gdn::mbar_init(bars + i, count);
        }
        gdn::fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 1) {
        gdn::tmem_alloc(tmem_slot, TMEM_COLS);
        gdn::tmem_relinquish();
    }
    gdn::tc_fence_before_sync();
    __syncthreads();
    gdn::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nv = words[W_NV];
    const int nchunks = 4 * nv;
    if (warp == 0 && lane < kPrefetch + 1 && lane < nv) {
        const int4 e = list[lane];
#pragma unroll
        for (int c = 0; c < 4; ++c) gdn::tma_prefetch_2d(&tmap, 32 * c, (e.w * a.Hv + e.x % a.Hv) * D);
    }
    gdn::grid_dep_wait();  // xc, the state pool, status
    if (tid == 0 && words[W_ERR]) gdn::record_status(a.status, words[W_ERR]);

    if (warp == 0) {
        // ---- producer: S0 chunks in order into the ring ----------------------
        if (lane == 0) {
            // the ring holds little more than one item, so the states of the
            // next kPrefetch items are requested into L2 ahead of their loads
            auto prefetch_item = [&](int v) {
                if (v >= nv) return;
                const int4 e = list[v];
#pragma unroll
                for (int c = 0; c < 4; ++c) gdn::tma_prefetch_2d(&tmap, 32 * c, (e.w * a.Hv + e.x % a.Hv) * D);
            };
            int g = 0, qk_issued = 0;
            for (; g < nchunks; ++g) {
                const int r = g % NR;
                const int4 e = list[g >> 2];
                if ((g & 3) == 0) {
                    // the item's q/k rows into its B buffer, once the item NB
                    // before has finished with it (its products and its team)
                    const int v = g >> 2, b = v % NB;
                    if (v >= NB && !wait_or_abort(bars + B_BFREE + b, uint32_t((v / NB - 1) & 1), abort_flag))
                        break;
                    const int kh = (e.x % a.Hv) / (a.Hv / a.Hk);
                    unsigned char *bt = sb + BT + b * kBTeam;
                    uint64_t *qbar = bars + B_QFULL + b;
                    gdn::mbar_arrive_expect_tx(qbar, 8 * kQKBox);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        gdn::tma_load_2d(bt + c * kBChunk, &xmap, a.Hk * D + kh * D + 32 * c, e.y, qbar);
                        gdn::tma_load_2d(bt + c * kBChunk + kQKBox, &xmap, kh * D + 32 * c, e.y, qbar);
                    }
                    ++qk_issued;
                    prefetch_item(v + kPrefetch + 1);
                }
                if (g >= NR && !wait_or_abort(bars + B_REMPTY + r, uint32_t((g / NR - 1) & 1), abort_flag)) break;
                uint64_t *fb = bars + B_RFULL + r;
                gdn::mbar_arrive_expect_tx(fb, kChunk);
                gdn::tma_load_2d(sb + RAW + r * kChunk, &tmap, 32 * (g & 3), (e.w * a.Hv + e.x % a.Hv) * D, fb);
            }
            if (*abort_flag) {
                // copies still in flight land on their own: wait for them (bounded)
                for (int r = 0; r < NR; ++r) {
                    const int last = g - 1 - ((g - 1 - r) % NR + NR) % NR;  // last chunk issued into slot r
                    if (g > 0 && last >= 0) gdn::mbar_wait_bounded(bars + B_RFULL + r, uint32_t((last / NR) & 1));
                }
                for (int b = 0; b < NB; ++b) {
                    const int last = qk_issued - 1 - ((qk_issued - 1 - b) % NB + NB) % NB;  // last item in buffer b
                    if (qk_issued > 0 && last >= 0)
                        gdn::mbar_wait_bounded(bars + B_QFULL + b, uint32_t((last / NB) & 1));
                }
            }
        }
    } else if (warp < kTeam0) {
        // ---- MMA issuers, items and chunks in order.  A thread waits about 200
        //      cycles on each tcgen05.mma it issues, whatever its shape, while
        //      several issuing warps proceed side by side, so the three kinds of
        //      product have a warp each: the Gram terms, A_hi [B_hi | B_lo] (which
        //      frees S0 slots) and A_lo [B_hi | B_lo] (which frees lo slots). -------
        if (lane == 0) {
            bool ok = true;
            for (int v = 0; v < nv && ok; ++v) {
                const int t = v & 1, ut = v >> 1, b = v % NB;
                if (!wait_or_abort(bars + B_BREADY + b, uint32_t((v / NB) & 1), abort_flag)) break;
                if (ut > 0 && !wait_or_abort(bars + B_ACCEMPTY + t, uint32_t((ut - 1) & 1), abort_flag)) break;
                gdn::tc_fence_after_sync();
                const uint32_t dacc = tmem + TEAM_COLS * t;
                const uint32_t bt0 = sbase + BT + b * kBTeam;
                if (warp == kIssueGram) {
                    // Gram terms of B's 64 rows [k | q | k_lo | q_lo] with themselves
                    for (int kt = 0; kt < 4; ++kt) {
                        uint64_t gd = gdn::desc_sw128(bt0 + kt * kBChunk);
                        // a K-step (8 tf32) is 32 bytes: 2 in the descriptors' address field
#pragma unroll 1
                        for (int ks = 0; ks < 4; ++ks, gd += 2)
                            gdn::mma_tf32(dacc + GCOL, gd, gd, IDESC_GRAM, (kt | ks) != 0);
                    }
                    gdn::mma_commit(bars + B_GFULL + t);
                    gdn::mma_commit(bars + B_BFREE + b);
                    continue;
                }
                for (int kb = 0; kb < 4; ++kb) {
                    const int g = 4 * v + kb;
                    uint64_t bst = gdn::desc_sw128(bt0 + kb * kBChunk);  // [B_hi | B_lo], 64 rows
                    const int r = g % NR;
                    const uint32_t par = uint32_t((g / NR) & 1);
                    uint64_t a_op = gdn::desc_sw128(sbase + RAW + r * kChunk);
                    if (warp == kIssueHi) {
                        // the raw chunk (read as A_hi); then the splitters may
                        // overwrite it with its lo part
                        if (!wait_or_abort(bars + B_RFULL + r, par, abort_flag)) {
                            ok = false;
                            break;
                        }
                        gdn::tc_fence_after_sync();
                        const uint32_t dk = dacc + 64u * (kb >> 1);
#pragma unroll 1
                        for (int ks = 0; ks < 4; ++ks, a_op += 2, bst += 2)
                            gdn::mma_tf32(dk, a_op, bst, IDESC_TF32, ((kb & 1) | ks) != 0);
                        gdn::mma_commit(bars + B_HDONE + r);
                    } else {
                        // the same slot once it holds the lo part; then it is free
                        if (!wait_or_abort(bars + B_LFULL + r, par, abort_flag)) {
                            ok = false;
                            break;
                        }
                        gdn::tc_fence_after_sync();
#pragma unroll 1
                        for (int ks = 0; ks < 4; ++ks, a_op += 2, bst += 2)
                            gdn::mma_tf32(dacc + LHCOL, a_op, bst, IDESC_TF32, (kb | ks) != 0);
                        gdn::mma_commit(bars + B_REMPTY + r);
                    }
                }
                if (ok) {
                    gdn::mma_commit(bars + B_ACCFULL + t);
                    gdn::mma_commit(bars + B_BFREE + b);
                }
            }
            // every tensor-core operation of these threads completes before the
            // tensor memory is released
            gdn::mma_commit(bars + B_DRAIN);
            gdn::mbar_wait_bounded(bars + B_DRAIN, 0);
        }
    } else if (warp >= kSplit0) {
        // ---- splitters, items in order: as soon as an item's q/k rows land in
        //      its team's B, the lo rows of B (so that the Gram and product
        //      issuers can start while the team still runs its previous
        //      epilogue); then, once each S0 chunk's A_hi products have read it,
        //      the chunk's lo part in place (elementwise, in the chunk's own
        //      swizzled layout). -------------------------------------------------
        const int st = tid - kSplit0 * 32;
        for (int g = 0; g < nchunks; ++g) {
            const int r = g % NR;
            if ((g & 3) == 0) {
                const int v = g >> 2, b = v % NB;
                if (!wait_or_abort(bars + B_QFULL + b, uint32_t((v / NB) & 1), abort_flag)) break;
                unsigned char *bt = sb + BT + b * kBTeam;
#pragma unroll
                for (int j = 0; j < (4 * 32 * 8) / kSplitThreads; ++j) {
                    const int idx = st + kSplitThreads * j;  // 16-byte unit: K-chunk idx / 256, rows 0-31
                    unsigned char *p = bt + (idx >> 8) * kBChunk + (idx & 255) * 16;
                    const float4 x = *reinterpret_cast<const float4 *>(p);
                    *reinterpret_cast<float4 *>(p + 32 * 128) = lo4(x);
                }
                gdn::fence_proxy_async_smem();
                mbar_arrive(bars + B_BREADY + b);
            }
            if (!wait_or_abort(bars + B_HDONE + r, uint32_t((g / NR) & 1), abort_flag)) break;
            float4 *c = reinterpret_cast<float4 *>(sb + RAW + r * kChunk);
            constexpr int kPer = int(kChunk / 16) / kSplitThreads;  // 16-byte units per thread
#pragma unroll
            for (int b = 0; b < kPer; b += kPer / 2) {
                float4 x[kPer / 2];
#pragma unroll
                for (int j = 0; j < kPer / 2; ++j) x[j] = c[st + kSplitThreads * (b + j)];
#pragma unroll
                for (int j = 0; j < kPer / 2; ++j) c[st + kSplitThreads * (b + j)] = lo4(x[j]);
            }
            gdn::fence_proxy_async_smem();
            mbar_arrive(bars + B_LFULL + r);
        }
    } else {
        // ---- math teams ----------------------------------------------------------
        const int team = (warp - kTeam0) >> 2, tw = warp & 3;  // warp within the team = its TMEM lane quarter
        const int ttid = tw * 32 + lane;                       // 0..127
        const int row = ttid;                                  // tensor-memory lane = state row
        float *tws = reinterpret_cast<float *>(words + team * T_WORDS);
        float *ka = tws + T_KA, *kb = tws + T_KB, *qa = tws + T_QA, *qb = tws + T_QB;
        float *gm = tws + T_GM, *cqt = tws + T_CQT, *lnt = tws + T_LNT;
        float *qqa = tws + T_QQA, *qqb = tws + T_QQB, *beta_s = tws + T_BETA, *dec_s = tws + T_DEC;
        float *gsk = tws + T_GSK, *gsq = tws + T_GSQ, *rk_s = tws + T_RK, *gam_s = tws + T_GAM;
        int *par = reinterpret_cast<int *>(tws + T_PAR);
        // the item's v rows (TMA), read by the epilogue
        float *stg_v = reinterpret_cast<float *>(sb + VT + team * kStage);

        // parents and gate inputs of the team's next item, loaded one item ahead
        int p_nx = -1;
        float bv_nx = 0.f, av_nx = 0.f, dtb_nx = 0.f, ah_nx = 0.f;
        auto prefetch = [&](int v) {
            if (v >= nv) return;
            const int4 e = list[v];
            const int h = e.x % a.Hv, n0 = e.y, lc = e.z;
            p_nx = ttid < lc ? __ldg(a.parents + n0 + ttid) : -1;
            if (tw == 0 && lane < lc) {
                const int64_t n = n0 + lane;
                bv_nx = __ldg(a.ba + n * a.ba_stride + h);
                av_nx = __ldg(a.ba + n * a.ba_stride + a.Hv + h);
                dtb_nx = __ldg(a.dt_bias + h);
                ah_nx = __ldg(a.A + h);
            }
        };
        prefetch(team);
        // the item's q/k rows (in B) and v rows (in the team's v tile) are rows
        // n0 .. n0 + 15; rows past the sequence's last node belong to the next
        // sequence, or are zero-filled past the tensor: they only feed outputs
        // that are never written
        int v_issued = 0;
        // test hook: team 0 of CTA 0 waits on a barrier that nothing completes,
        // so the wait runs out, and every role drains and leaves
        if (a.stall_ns && blockIdx.x == 0 && team == 0 &&
            !gdn::mbar_wait_bounded(bars + B_NEVER, 0, a.stall_ns))
            *abort_flag = 1;

        for (int v = team; v < nv; v += 2) {
            const int ut = v >> 1;
            const int4 e = list[v];
            const int h = e.x % a.Hv, n0 = e.y, lc = e.z;
            const int voff = 2 * a.Hk * D + h * D;
            const int bb = v % NB;
            unsigned char *bt_t = sb + BT + bb * kBTeam;
            int p = p_nx;
            const float bv = bv_nx, av = av_nx, dtb = dtb_nx, Ah = ah_nx;
            // the team's previous epilogue has finished reading the small area
            // and the v tile
            team_sync(team);
            // the item's 16 v rows by TMA into the team's v tile
            if (ttid == 0) {
                uint64_t *vb = bars + B_VFULL + team;
                gdn::mbar_arrive_expect_tx(vb, kSeg * D * 4);
                gdn::tma_load_2d(stg_v, &vmap, voff, n0, vb);
                ++v_issued;
            }

            // ---- A: parents and gates (warp 0 of the team: lane = node) -----------
            if (ttid < kSeg) {
                if (ttid < lc && (p < -1 || p >= ttid)) {
                    gdn::record_status(a.status, GDN_DEV_BAD_PARENT);
                    p = -1;  // outputs of a failed call are unspecified; keep the walks in bounds
                }
                par[ttid] = ttid < lc ? p : -1;
            }
            if (tw == 0 && lane < kSeg) {
                float dec = 1.f, bet = 0.f;
                if (lane < lc) {
                    dec = expf(gdn::softplus_f(av + dtb) * Ah);
                    bet = gdn::sigmoid_f(bv);
                    a.replay[((n0 + lane) * int64_t(a.Hv) + h) * a.rstride + 2 * D] = dec;
                }
                beta_s[lane] = bet;
                dec_s[lane] = dec;
            }
            __syncwarp();
            // ---- the ancestor decays: lane t walks its path and writes row t of
            //      GM, gamma_{j->t} = the decays strictly after j up to t (1 on the
            //      diagonal, 0 off the path), and Gamma_t, all the decays on it.
            //      Products along the path only, so underflow can only drop terms
            //      that are already below the float range. ------------------------
            if (tw == 0 && lane < kSeg) {
                float4 *g4 = reinterpret_cast<float4 *>(gm + lane * kSeg);
#pragma unroll
                for (int j4 = 0; j4 < kSeg / 4; ++j4) g4[j4] = make_float4(0.f, 0.f, 0.f, 0.f);
                float g = 0.f;
                if (lane < lc) {
                    gm[lane * kSeg + lane] = 1.f;
                    g = 1.f;
                    for (int cur = lane;;) {
                        g *= dec_s[cur];
                        cur = par[cur];
                        if (cur < 0) break;
                        gm[lane * kSeg + cur] = g;
                    }
                }
                gam_s[lane] = g;
            }

            // ---- B: Gram terms from tensor memory.  Warp tw holds G rows 16 tw ..
            //      16 tw + 15 (k, q, k_lo, q_lo of the nodes) in lanes 0..15, columns
            //      [k | q | k_lo | q_lo]: a row against column j plus column 32 + j is
            //      its dot product with all of k_j. ----------------------------------
            // warp-uniform: tcgen05.ld is warp-collective.  The Gram terms
            // complete after the splitters wrote B's lo rows, so B is in place
            const bool gready =
                __all_sync(0xffffffffu, wait_or_abort(bars + B_GFULL + team, uint32_t(ut & 1), abort_flag));
            const bool staged = gready;
            if (gready) {
                gdn::tc_fence_after_sync();
                const uint32_t grow = tmem + TEAM_COLS * team + GCOL + (uint32_t(tw * 32) << 16);
                float d0[32], d1[32];
                gdn::tmem_ld32(grow, d0);
                gdn::tmem_ld32(grow + 32u, d1);
                if (lane < kSeg) {
                    float *dst = (tw == 0 ? ka : tw == 1 ? qa : tw == 2 ? kb : qb) + lane * kSeg;
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const int j = 4 * j4;
                        *reinterpret_cast<float4 *>(dst + j) =
                            make_float4(d0[j] + d1[j], d0[j + 1] + d1[j + 1], d0[j + 2] + d1[j + 2], d0[j + 3] + d1[j + 3]);
                    }
                    if (tw & 1) {
                        // q_t . q_t: columns 16 + t and 48 + t (no dynamic register index)
                        float qq = 0.f;
#pragma unroll
                        for (int b = 0; b < kSeg; ++b)
                            if (b == lane) qq = d0[kSeg + b] + d1[kSeg + b];
                        (tw == 1 ? qqa : qqb)[lane] = qq;
                    }
                }
            }
            team_sync(team);  // Gram terms, parents, decays and GM are in

            // ---- C: path coefficients, two entries (t, j) per thread.
            //      L[t][j] = beta_t gamma_{j->t} k^_j . k^_t (j a strict ancestor of t),
            //      CQ[t][j] = q_scale gamma_{j->t} k^_j . q^_t (j on the path of t,
            //      t included; stored transposed), column factors Gamma_t / |k_t|
            //      and q_scale Gamma_t / |q_t|.  Zero outside the sequence's nodes. -
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const int e = ttid + 128 * q2, t = e >> 4, j = e & (kSeg - 1);
                const float rkt = rsqrtf(ka[t * (kSeg + 1)] + kb[t * (kSeg + 1)] + 1e-6f);
                const float rkj = rsqrtf(ka[j * (kSeg + 1)] + kb[j * (kSeg + 1)] + 1e-6f);
                const float rqt = rsqrtf(qqa[t] + qqb[t] + 1e-6f);
                const float g = gm[e];
                const bool in = t < lc;
                const float lk = (in && j < t) ? beta_s[t] * (g * ((ka[e] + kb[e]) * (rkt * rkj))) : 0.f;
                const float c = (in && j <= t) ? a.q_scale * (g * ((qa[e] + qb[e]) * (rqt * rkj))) : 0.f;
                lnt[j * kSeg + t] = -lk;
                cqt[j * kSeg + t] = c;
                if (j == 0) {
                    gsk[t] = gam_s[t] * rkt;
                    gsq[t] = a.q_scale * (gam_s[t] * rqt);
                    rk_s[t] = rkt;
                }
            }
            team_sync(team);  // coefficients of every node are in

            // ---- D: the replay rows' k^, from B's raw rows ----------------------
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int t = tw + 4 * m;
                if (t < lc && staged) {
                    const float4 kh = scale4(*reinterpret_cast<const float4 *>(bt_t + sw_off(t, 4 * lane, kBChunk)),
                                             rk_s[t]);
                    *reinterpret_cast<float4 *>(a.replay + ((n0 + t) * int64_t(a.Hv) + h) * a.rstride + 4 * lane) =
                        kh;
                }
            }
            team_sync(team);  // B is no longer read by the team
            if (ttid == 0) mbar_arrive(bars + B_BFREE + bb);

            // ---- E: per row, r = beta (v - Gamma S0 k^), u = T r, o = Gamma S0 q^ + W r
            // warp-uniform: tcgen05.ld is warp-collective
            const bool ready = __all_sync(0xffffffffu,
                                          wait_or_abort(bars + B_ACCFULL + team, uint32_t(ut & 1), abort_flag) &&
                                              wait_or_abort(bars + B_VFULL + team, uint32_t(ut & 1), abort_flag));
            prefetch(v + 2);
            if (ready) {
                gdn::tc_fence_after_sync();
                const uint32_t trow = tmem + TEAM_COLS * team + (uint32_t(tw * 32) << 16);
                // D = the sum of the partial accumulators, added in fp32, smallest
                // first: A_lo B_lo, A_lo B_hi, A_hi B_lo of both K-halves, then
                // A_hi B_hi of both K-halves
                float dv[32], p1[32];
                gdn::tmem_ld32(trow + LHCOL + 32u, dv);
#pragma unroll 1
                for (int part = 0; part < 5; ++part) {
                    const uint32_t col = part == 0 ? LHCOL : part == 1 ? 32u : part == 2 ? 96u : part == 3 ? 0u : 64u;
                    gdn::tmem_ld32(trow + col, p1);
#pragma unroll
                    for (int i = 0; i < 32; ++i) dv[i] += p1[i];
                }
                gdn::tc_fence_before_sync();
                mbar_arrive(bars + B_ACCEMPTY + team);  // the accumulators may be overwritten

                // r_t = beta_t (v_t - Gamma_t S0 k^_t) and (I + L) u = r by forward
                // substitution in column order: once column j - 1 is in, u_j is
                // final and column j of -L times u_j goes into the later nodes.
                // Nodes travel as packed pairs (u_2p, u_2p+1), so a column costs
                // at most 8 paired FMAs and the chain from u_j to u_j+1 is one.
                // Then o = Gamma S0 q^ + CQ u the same way.
                float vreg[kSeg];
#pragma unroll
                for (int t = 0; t < kSeg; ++t) vreg[t] = t < lc ? stg_v[t * D + row] : 0.f;
                uint64_t up[kSeg / 2], op[kSeg / 2];
#pragma unroll
                for (int p2 = 0; p2 < kSeg / 2; ++p2) {
                    const int t = 2 * p2;
                    const float r0 = beta_s[t] * (vreg[t] - gsk[t] * dv[t]);
                    const float r1 = beta_s[t + 1] * (vreg[t + 1] - gsk[t + 1] * dv[t + 1]);
                    up[p2] = gdn::f2pack(r0, r1);
                    op[p2] = gdn::f2pack(gsq[t] * dv[kSeg + t], gsq[t + 1] * dv[kSeg + t + 1]);
                }
#pragma unroll
                for (int j = 0; j < kSeg - 1; ++j) {
                    const float2 u01 = gdn::f2unpack(up[j / 2]);
                    const float uj = (j & 1) ? u01.y : u01.x;
                    const uint64_t ujj = gdn::f2pack(uj, uj);
                    const ulonglong2 *lcol = reinterpret_cast<const ulonglong2 *>(lnt + j * kSeg);
#pragma unroll
                    for (int q4 = j / 4; q4 < kSeg / 4; ++q4) {  // entries t = 4 q4 .. 4 q4 + 3 (zero for t <= j)
                        const ulonglong2 c = lcol[q4];
                        up[2 * q4] = gdn::fma2(c.x, ujj, up[2 * q4]);
                        up[2 * q4 + 1] = gdn::fma2(c.y, ujj, up[2 * q4 + 1]);
                    }
                }
#pragma unroll
                for (int j = 0; j < kSeg; ++j) {
                    const float2 u01 = gdn::f2unpack(up[j / 2]);
                    const float uj = (j & 1) ? u01.y : u01.x;
                    const uint64_t ujj = gdn::f2pack(uj, uj);
                    const ulonglong2 *ccol = reinterpret_cast<const ulonglong2 *>(cqt + j * kSeg);
#pragma unroll
                    for (int q4 = j / 4; q4 < kSeg / 4; ++q4) {  // entries t = 4 q4 .. 4 q4 + 3 (zero for t < j)
                        const ulonglong2 c = ccol[q4];
                        op[2 * q4] = gdn::fma2(c.x, ujj, op[2 * q4]);
                        op[2 * q4 + 1] = gdn::fma2(c.y, ujj, op[2 * q4 + 1]);
                    }
                }
                float *orow = a.o + (int64_t(n0) * a.Hv + h) * D + row;
                float *urow = a.replay + (int64_t(n0) * a.Hv + h) * a.rstride + D + row;
                const int64_t ostep = int64_t(a.Hv) * D, ustep = int64_t(a.Hv) * a.rstride;
                // a warp's 32 rows are contiguous: each store is one 128-byte line
#pragma unroll
                for (int t = 0; t < kSeg; ++t) {
                    if (t < lc) {
                        const float2 o01 = gdn::f2unpack(op[t / 2]), u01 = gdn::f2unpack(up[t / 2]);
                        orow[t * ostep] = (t & 1) ? o01.y : o01.x;
                        urow[t * ustep] = (t & 1) ? u01.y : u01.x;
                    }
                }
            }
            // after a timeout the team keeps looping (every wait now returns at
            // once) so that all four warps meet at each team barrier
        }
        // after a timeout, a v copy may still be in flight: wait for it (bounded)
        if (*abort_flag && v_issued > 0)
            gdn::mbar_wait_bounded(bars + B_VFULL + team, uint32_t((v_issued - 1) & 1));
    }

    // ---- tear-down -------------------------------------------------------------
    gdn::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort_flag) gdn::record_status(a.status, GDN_DEV_TIMEOUT);
    if (warp == 1) {
        gdn::tc_fence_after_sync();
        gdn::tmem_dealloc(tmem, TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// The state pool viewed as a 2-D tensor [P * H_v * d rows][d floats]; one box
// is [d rows][32 floats] (one 128-byte swizzle row per state row).
int encode_state_map(CUtensorMap *map, const float *ssm, int64_t P, int64_t Hv, int D) {
    auto enc = tensor_map_encoder();
    if (!enc) return GDN_ERR_TMA;
    cuuint64_t gdim[2] = {cuuint64_t(D), cuuint64_t(P * Hv * D)};
    cuuint64_t gstride[1] = {cuuint64_t(D) * 4};
    cuuint32_t box[2] = {cuuint32_t(D >= 32 ? 32 : D), cuuint32_t(D)};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ssm), gdim, gstride, box,
                     estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     D >= 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_TMA;
}

template <int D, int NMAX>
int launch(const CUtensorMap &map, const VerifyArgs &a, cudaStream_t st) {
    using L = Layout<D, NMAX>;
    auto k = tree_verify_kernel<D, NMAX>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L::BYTES)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const dim3 grid{unsigned(a.Hv), unsigned(a.S)};
    return gdn::launch_pdl(k, grid, dim3(kThreads), L::BYTES, st, map, a) == cudaSuccess ? GDN_OK : GDN_ERR_LAUNCH;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

// xc viewed as [N rows][C floats] with boxes of [rows][cols] floats.  The q/k
// map takes boxes of [16 rows][32 floats] (the q or k rows of one sequence's
// 16 nodes, one K-chunk) in the 128-byte swizzle, so a box lands as 16 rows of
// the tensor cores' K-major operand; the v map takes [16 rows][d floats]
// unswizzled (row t of the box = node t's v, contiguous).
int encode_xc_map(CUtensorMap *map, const float *xc, int64_t N, int64_t C, uint32_t rows, uint32_t cols,
                  bool swizzle) {
    auto enc = tensor_map_encoder();
    if (!enc) return GDN_ERR_TMA;
    cuuint64_t gdim[2] = {cuuint64_t(C), cuuint64_t(N)};
    cuuint64_t gstride[1] = {cuuint64_t(C) * 4};
    cuuint32_t box[2] = {cols, rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(xc), gdim, gstride, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GDN_OK : GDN_ERR_TMA;
}

std::atomic<uint64_t> g_stall_ns{0};

int launch_tc(const CUtensorMap &map, const VerifyArgs &a_in, cudaStream_t st) {
    VerifyArgs a = a_in;
    a.stall_ns = gdn::take_test_stall_ns();
    CUtensorMap xmap, vmap;
    if (int rc = encode_xc_map(&xmap, a.xc, a.N, a.C, 16, 32, true)) return rc;
    if (int rc = encode_xc_map(&vmap, a.xc, a.N, a.C, 16, wsv::D, false)) return rc;
    auto k = tree_verify_ws_kernel;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(wsv::BYTES)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int64_t items = int64_t(a.S) * a.Hv;
    const int sms = sm_count();
    if (sms <= 0) return GDN_ERR_LAUNCH;
    // one CTA per SM, each with at most kMaxItems items (more CTAs queue behind)
    int64_t grid = std::max<int64_t>(std::min<int64_t>(items, sms), (items + wsv::kMaxItems - 1) / wsv::kMaxItems);
    return gdn::launch_pdl(k, dim3(unsigned(grid)), dim3(wsv::kThreadsWS), wsv::BYTES, st, map, xmap, vmap, a) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_LAUNCH;
}

// d = 128 with trees of up to 16 nodes: tensor cores; otherwise the FFMA kernel
template <int D>
int launch_d(const CUtensorMap &map, const VerifyArgs &a, cudaStream_t st) {
    if constexpr (D == 128) {
        if (a.max_nodes <= kSeg) return launch_tc(map, a, st);
        return launch<D, gdn::kMaxSeqNodes>(map, a, st);
    } else {
        return a.max_nodes <= kSeg ? launch<D, kSeg>(map, a, st) : launch<D, gdn::kMaxSeqNodes>(map, a, st);
    }
}

}  // namespace

namespace gdn {
int encode_xc_tiles(CUtensorMap *map, const float *xc, int64_t N, int64_t C, uint32_t rows, uint32_t cols,
                    bool swizzle) {
    return encode_xc_map(map, xc, N, C, rows, cols, swizzle);
}
int sm_count_current() { return sm_count(); }
uint64_t take_test_stall_ns() { return g_stall_ns.exchange(0); }
}  // namespace gdn

extern "C" int gdn_tree_verify(const gdn_dims *dims, const float *xc, const float *ba, int64_t ba_stride,
                               const float *dt_bias, const float *A, const float *ssm, float q_scale,
                               const int32_t *parents, const int32_t *node_off, const int32_t *slot_map,
                               float *o, float *replay, int64_t replay_stride, int32_t *status, void *stream) {
    int rc = gdn::check_dims(dims);
    if (rc) return rc;
    const int64_t S = dims->n_seqs, N = dims->n_nodes, P = dims->n_slots;
    const int64_t Hv = dims->h_v, D = dims->d_k, C = gdn::conv_channels(dims);
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

    CUtensorMap map;
    if ((rc = encode_state_map(&map, ssm, P, Hv, int(D)))) return rc;
    VerifyArgs a{xc, ba, ba_stride, dt_bias, A, q_scale, parents, node_off, slot_map, o, replay, replay_stride,
                 status, int(S), int(N), int(P), dims->h_k, int(Hv), int(C), dims->max_seq_nodes, 0};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (D) {
        case 16: return launch_d<16>(map, a, st);
        case 32: return launch_d<32>(map, a, st);
        case 64: return launch_d<64>(map, a, st);
        default: return launch_d<128>(map, a, st);
    }
}

extern "C" void gdn_test_stall_next_verify(uint64_t wait_ns) {
    g_stall_ns.store(std::min<uint64_t>(wait_ns, gdn::kWaitLimitNs));
}
