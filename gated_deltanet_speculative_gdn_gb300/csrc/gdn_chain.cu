// gdn_chain.cu - verify for sequences whose draft tokens form a chain (node i's
// parent is node i - 1), d = 128, in chunked form.
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
// The decay products are plain products along the chain (no ratios).
//
// Mapping (GB300).  A persistent CTA of 256 threads (two per SM) takes one
// (sequence, value head) item at a time and keeps that item's 128 x 128 state
// in registers for the whole chain: thread (rp, cq) holds rows 2rp, 2rp + 1 and
// columns 32 cq .. 32 cq + 31, as packed fp32 pairs.  Per chunk: the raw k, q
// and v rows arrive by bulk copies issued one chunk ahead; each warp
// normalises four of the 32 k/q vectors into a padded shared-memory tile; the
// Gram terms take four lanes per dot product; one warp builds the
// coefficients and T while the rest start the contraction S [k^ | q^]
// (2 rows x 32 columns x 32 vectors per thread with fma.rn.f32x2, the four
// column quarters reduced with three shuffles per two vectors); the solve,
// the output and the state update are local to each warp.  The state never
// leaves the chip between chunks and is never written back: verify leaves
// the pool untouched, and the commit advances it from the replay rows.
#include <algorithm>

#include "gdn_device.cuh"
#include "gdn_internal.h"

namespace {

constexpr int D = 128;
constexpr int kThreads = 256;
constexpr int kChunk = 16;
constexpr int KQS = 8 * 20 + 4;  // padded k^/q^ row: eight groups of 16 floats + 4 each, + 4
constexpr int RS = 36;       // row stride of the a_t | b_t tile [state row][32]
constexpr int US = 20;       // row stride of the u tile [state row][node]
constexpr int CS = 20;       // row stride of the 16 x 16 coefficient matrices
// Column slot of node t in the transposed matrices: even nodes first, then odd
// ones, so that the two threads of a state row (one per parity) each read
// their eight entries of a column as two float4.
__host__ __device__ constexpr int tslot(int t) { return (t & 1) * 8 + (t >> 1); }
// what an item's sequence asks for: run, skip (empty), or a GDN_DEV_* code (> 0)
constexpr int kRun = -1, kSkip = 0;

// float offsets into dynamic shared memory (16-byte aligned)
constexpr int RAWK = 0;                      // [16][128] raw k rows of the chunk
constexpr int RAWQ = RAWK + kChunk * D;      // [16][128] raw q rows
constexpr int VB = RAWQ + kChunk * D;        // [2][16][128] v rows, two chunks
constexpr int KQH = VB + 2 * kChunk * D;     // [32][KQS] k^ (0..15) | q^ (16..31)
constexpr int RES = KQH + 2 * kChunk * KQS;  // [128][RS] a_t (0..15) | b_t (16..31)
constexpr int UB = RES + D * RS;             // [128][US] u_t per state row
constexpr int CKM = UB + D * US;             // [16][CS] gamma_{j->t} k^_j.k^_t (j < t)
constexpr int CQT = CKM + kChunk * CS;       // [16 j][CS] gamma_{j->t} k^_j.q^_t (j <= t), at tslot(t)
constexpr int TT = CQT + kChunk * CS;        // [16 j][CS] T[t][j], at tslot(t)
constexpr int BETA = TT + kChunk * CS;       // [16]
constexpr int DEC = BETA + kChunk;           // [16]
constexpr int GAM = DEC + kChunk;            // [16] Gamma_t
constexpr int WEND = GAM + kChunk;           // [16] gamma_{j->L-1}
constexpr int BARS = WEND + kChunk;          // 3 mbarriers
constexpr int FLOATS = BARS + 8;
constexpr size_t BYTES = size_t(FLOATS) * 4;
static_assert(BARS % 4 == 0, "mbarriers need 8-byte alignment; tiles 16-byte");

struct ChainArgs {
    const float *__restrict__ xc;
    const float *__restrict__ ba;
    int64_t ba_stride;
    const float *__restrict__ dt_bias;
    const float *__restrict__ A;
    const float *__restrict__ ssm;
    float q_scale;
    const int32_t *__restrict__ parents;
    const int32_t *__restrict__ node_off;
    const int32_t *__restrict__ slot_map;
    float *__restrict__ o;
    float *__restrict__ replay;
    int64_t rstride;
    int32_t *status;
    int S, N, P, Hk, Hv, C, max_nodes;
};

// Issues the bulk copies of one chunk's rows (k and q on `bkq`, v on `bv`);
// lanes of one warp each take some rows.  The expected byte counts are set by
// lane 0 before any copy is issued.
__device__ __forceinline__ void issue_chunk(const ChainArgs &a, float *sm, uint64_t *bkq, uint64_t *bv,
                                            float *vdst, int64_t n_first, int L, int koff, int qoff, int voff,
                                            bool kq, bool v, int lane) {
    if (lane == 0) {
        if (kq) gdn::mbar_arrive_expect_tx(bkq, uint32_t(L) * 2 * D * 4);
        if (v) gdn::mbar_arrive_expect_tx(bv, uint32_t(L) * D * 4);
    }
    __syncwarp();
    if (lane < L) {
        const float *row = a.xc + (n_first + lane) * int64_t(a.C);
        if (kq) {
            gdn::bulk_load(sm + RAWK + lane * D, row + koff, D * 4, bkq);
            gdn::bulk_load(sm + RAWQ + lane * D, row + qoff, D * 4, bkq);
        }
        if (v) gdn::bulk_load(vdst + lane * D, row + voff, D * 4, bv);
    }
}

// Warp 0, lanes < 16: the raw gate inputs (b, a) of node `first + lane` if it
// is one of the chunk's L nodes.
__device__ __forceinline__ float2 load_gate_inputs(const ChainArgs &a, int64_t first, int L, int h, int lane) {
    float2 r = make_float2(0.f, 0.f);
    if (lane < L) {
        const float *p = a.ba + (first + lane) * a.ba_stride;
        r = make_float2(__ldg(p + h), __ldg(p + a.Hv + h));
    }
    return r;
}

__global__ void __launch_bounds__(kThreads, 2) chain_verify_kernel(const ChainArgs a) {
    extern __shared__ float4 smem_v4[];
    float *sm = reinterpret_cast<float *>(smem_v4);
    uint64_t *bkq = reinterpret_cast<uint64_t *>(sm + BARS);
    uint64_t *bvv = bkq + 1;  // two: one per v buffer
    __shared__ int hdr[4];    // code (kRun, kSkip or a device error), first node, nodes, slot

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rg = tid >> 3, cg = tid & 7;  // contraction / update: rows 4rg .. 4rg+3, columns 16cg ..
    gdn::grid_dep_launch();
    if (tid == 0) {
        gdn::mbar_init(bkq, 1);
        gdn::mbar_init(bvv, 1);
        gdn::mbar_init(bvv + 1, 1);
        gdn::fence_mbar_init();
    }
    uint32_t ph_kq = 0, ph_v0 = 0, ph_v1 = 0;
    bool pend_kq = false, pend_v0 = false, pend_v1 = false;
    bool waited = false, timed_out = false, aborted = false;
    const int64_t items = int64_t(a.S) * a.Hv;
    const int G = a.Hv / a.Hk;

    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int s = int(it / a.Hv), h = int(it - int64_t(s) * a.Hv);
        // ---- the item's sequence (pure inputs) ----------------------------------
        if (warp == 0) {
            const int n0 = a.node_off[s], n1 = a.node_off[s + 1];
            int code = kRun, slot = 0;
            if (n0 < 0 || n1 < n0 || n1 > a.N || (s == 0 && n0 != 0) || (s == a.S - 1 && n1 != a.N) ||
                n1 - n0 > a.max_nodes)
                code = GDN_DEV_BAD_NODE_OFF;
            else if (n1 == n0)
                code = kSkip;
            else {
                slot = a.slot_map[s];
                if (slot < 0 || slot >= a.P) code = GDN_DEV_BAD_SLOT;
            }
            bool bad = false;
            if (code == kRun)
                for (int i = lane; i < n1 - n0; i += 32) bad |= a.parents[n0 + i] != i - 1;
            if (__any_sync(0xffffffffu, bad)) code = GDN_DEV_BAD_PARENT;
            if (lane == 0) {
                hdr[0] = code;
                hdr[1] = n0;
                hdr[2] = n1 - n0;
                hdr[3] = slot;
            }
        }
        __syncthreads();
        const int code = hdr[0], n0 = hdr[1], n = hdr[2], slot = hdr[3];
        __syncthreads();  // hdr is rewritten by the next item
        if (code == kSkip) continue;
        if (!waited) {
            gdn::grid_dep_wait();  // xc, ba, the state pool, status
            waited = true;
        }
        if (code != kRun) {
            if (tid == 0) gdn::record_status(a.status, code);
            continue;
        }
        const int kh = h / G;
        const int qoff = kh * D, koff = a.Hk * D + kh * D, voff = 2 * a.Hk * D + h * D;
        const float dtb = __ldg(a.dt_bias + h), Ah = __ldg(a.A + h);
        const int nchunks = (n + kChunk - 1) / kChunk;

        // chunk 0's rows and gate inputs, then the state into registers while they travel
        // gate inputs travel one chunk ahead: gate_nxt is loaded a chunk before
        // it is copied into gate_cur, so the copy never waits on the load
        float2 gate_cur = make_float2(0.f, 0.f), gate_nxt = gate_cur;
        if (warp == 0) {
            issue_chunk(a, sm, bkq, bvv, sm + VB, n0, min(kChunk, n), koff, qoff, voff, true, true, lane);
            gate_nxt = load_gate_inputs(a, n0, min(kChunk, n), h, lane);
        }
        pend_kq = true;
        pend_v0 = true;
        if (warp == 1) {
            // the next item's state and first rows toward L2 (a hint; only for
            // offsets that are in range)
            const int64_t it2 = it + gridDim.x;
            if (it2 < items) {
                const int s2 = int(it2 / a.Hv), h2 = int(it2 - int64_t(s2) * a.Hv);
                const int m0 = a.node_off[s2], m1 = a.node_off[s2 + 1], sl2 = a.slot_map[s2];
                if (m0 >= 0 && m1 >= m0 && m1 <= a.N && sl2 >= 0 && sl2 < a.P) {
                    const float *st2 = a.ssm + (int64_t(sl2) * a.Hv + h2) * D * D;
                    if (lane < 4) gdn::bulk_prefetch_l2(st2 + lane * (D * D / 4), D * D);
                    const int kh2 = h2 / G;
                    if (lane < min(kChunk, m1 - m0)) {
                        const float *row = a.xc + (int64_t(m0) + lane) * a.C;
                        gdn::bulk_prefetch_l2(row + kh2 * D, D * 4);
                        gdn::bulk_prefetch_l2(row + a.Hk * D + kh2 * D, D * 4);
                        gdn::bulk_prefetch_l2(row + 2 * a.Hk * D + h2 * D, D * 4);
                    }
                }
            }
        }
        uint64_t st[4][8];  // rows 4rg + r, column pairs 16cg + 2p
        {
            const float *src = a.ssm + (int64_t(slot) * a.Hv + h) * D * D + int64_t(4 * rg) * D + 16 * cg;
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 v = __ldg(reinterpret_cast<const float4 *>(src + r * D) + m);
                    st[r][2 * m] = gdn::f2pack(v.x, v.y);
                    st[r][2 * m + 1] = gdn::f2pack(v.z, v.w);
                }
        }

        for (int c = 0; c < nchunks; ++c) {
            const int L = min(kChunk, n - c * kChunk);
            const int64_t nf = n0 + int64_t(c) * kChunk;  // first node of the chunk
            const int vb = c & 1;
            // the previous chunk is done with every shared tile; a wait that ran out ends the CTA
            if (__syncthreads_or(timed_out)) {
                aborted = true;
                break;
            }
            gate_cur = gate_nxt;
            if (c + 1 < nchunks && warp == 0) {
                const int L1 = min(kChunk, n - (c + 1) * kChunk);
                issue_chunk(a, sm, bkq, bvv + (vb ^ 1), sm + VB + (vb ^ 1) * kChunk * D, nf + kChunk, L1, koff,
                            qoff, voff, false, true, lane);
                gate_nxt = load_gate_inputs(a, nf + kChunk, L1, h, lane);
            }
            if (c + 1 < nchunks) (vb ? pend_v0 : pend_v1) = true;

            // ---- A: the gates, then normalised k^ / q^ ----------------------------
            if (warp == 0 && lane < kChunk) {
                float beta = 0.f, dec = 1.f;
                if (lane < L) {
                    beta = gdn::sigmoid_f(gate_cur.x);
                    dec = expf(gdn::softplus_f(gate_cur.y + dtb) * Ah);
                    a.replay[((nf + lane) * a.Hv + h) * a.rstride + 2 * D] = dec;
                }
                sm[BETA + lane] = beta;
                sm[DEC + lane] = dec;
            }
            if (!gdn::mbar_wait_bounded(bkq, ph_kq)) timed_out = true;
            ph_kq ^= 1;
            pend_kq = false;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int vi = warp + 8 * j;  // 0..15: k^ of node vi; 16..31: q^ of node vi - 16
                const int t = vi & 15;
                float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t < L) val = *reinterpret_cast<const float4 *>(sm + (vi < 16 ? RAWK : RAWQ) + t * D + 4 * lane);
                float ss = val.x * val.x;
                ss = fmaf(val.y, val.y, ss);
                ss = fmaf(val.z, val.z, ss);
                ss = fmaf(val.w, val.w, ss);
                ss = gdn::warp_sum(ss);
                const float inv = rsqrtf(ss + 1e-6f);
                const float4 nv = make_float4(val.x * inv, val.y * inv, val.z * inv, val.w * inv);
                *reinterpret_cast<float4 *>(sm + KQH + vi * KQS + 20 * (lane >> 2) + 4 * (lane & 3)) = nv;
                if (vi < 16 && t < L)
                    *reinterpret_cast<float4 *>(a.replay + ((nf + t) * a.Hv + h) * a.rstride + 4 * lane) = nv;
            }
            __syncthreads();  // k^ / q^ and the gates are in place; the raw k/q tile is free
            if (c + 1 < nchunks) {
                if (warp == 0) {
                    const int L1 = min(kChunk, n - (c + 1) * kChunk);
                    issue_chunk(a, sm, bkq, nullptr, nullptr, nf + kChunk, L1, koff, qoff, voff, true, false, lane);
                }
                pend_kq = true;
            }

            // ---- B: Gram terms scaled into the coefficients; Gamma, end weights --
            // The 16 x 32 products k^_j . [k^_0..15 | q^_0..15] in 4 x 4 tiles, each
            // tile over eight column slices (lanes xor 1, 2, 4), reduced and
            // scattered so that every lane ends with two of the tile's entries.
            {
                const int ks = lane & 7, tile = 4 * warp + (lane >> 3);  // 32 tiles
                const int j0 = 4 * (tile & 3), c0 = 4 * (tile >> 2);     // rows j0.., columns c0..
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    float4 xc[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        xc[q] = *reinterpret_cast<const float4 *>(sm + KQH + (c0 + q) * KQS + 20 * ks + 4 * m);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float4 xj = *reinterpret_cast<const float4 *>(sm + KQH + (j0 + r) * KQS + 20 * ks + 4 * m);
#pragma unroll
                        for (int q = 0; q < 4; ++q) acc[4 * r + q] = gdn::fma4(xj, xc[q], acc[4 * r + q]);
                    }
                }
                // recursive halving: after the three rounds lane ks holds entries 2ks, 2ks + 1
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const bool up = ks & 4;
                    const float keep = up ? acc[8 + e] : acc[e], send = up ? acc[e] : acc[8 + e];
                    acc[e] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool up = ks & 2;
                    const float keep = up ? acc[4 + e] : acc[e], send = up ? acc[e] : acc[4 + e];
                    acc[e] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool up = ks & 1;
                    const float keep = up ? acc[2 + e] : acc[e], send = up ? acc[e] : acc[2 + e];
                    acc[e] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int idx = 2 * ks + e;  // entry (r, q) of the tile
                    const int j = j0 + (idx >> 2), col = c0 + (idx & 3);
                    const bool kk = col < kChunk;  // k^_j . k^_t, else k^_j . q^_t
                    const int t = kk ? col : col - kChunk;
                    float coef = 0.f;
                    if (kk ? j < t : j <= t) {
                        float g = 1.f;  // gamma_{j->t}, as a product
                        for (int s2 = j + 1; s2 <= t; ++s2) g *= sm[DEC + s2];
                        coef = g * acc[e];
                    }
                    if (kk)
                        sm[CKM + t * CS + j] = coef;
                    else
                        sm[CQT + j * CS + tslot(t)] = coef;
                }
                if (tid < kChunk) {
                    float gam = 1.f;
                    for (int s2 = 0; s2 <= tid; ++s2) gam *= sm[DEC + s2];
                    sm[GAM + tid] = gam;
                    float wend = 0.f;
                    if (tid < L) {
                        wend = 1.f;
                        for (int s2 = tid + 1; s2 < L; ++s2) wend *= sm[DEC + s2];
                    }
                    sm[WEND + tid] = wend;
                }
            }
            __syncthreads();

            // ---- T = (I + diag(beta) CK)^-1 diag(beta), one column per lane of warp
            //      0 (forward substitution down the column, kept in registers) -----
            if (warp == 0 && lane < kChunk) {
                const int j = lane;
                float tc[kChunk];
#pragma unroll
                for (int t = 0; t < kChunk; ++t) {
                    const float *ck = sm + CKM + t * CS;
                    float acc = 0.f;
#pragma unroll
                    for (int s2 = 0; s2 < t; ++s2) acc = fmaf(ck[s2], tc[s2], acc);  // tc[s2] = 0 for s2 < j
                    const float b = sm[BETA + t];
                    tc[t] = t == j ? b : (t > j ? -b * acc : 0.f);
                    sm[TT + j * CS + tslot(t)] = tc[t];
                }
            }

            // ---- C: a_t = S k^_t, b_t = S q^_t for the four rows of each thread --
            {
                const float *kq = sm + KQH + 20 * cg;
                float *res = sm + RES;
#pragma unroll 2
                for (int v = 0; v < 2 * kChunk; ++v) {
                    const float *b0 = kq + v * KQS;
                    uint64_t ac[4] = {0, 0, 0, 0};  // per row
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const float4 x = *reinterpret_cast<const float4 *>(b0 + 4 * m);
                        const uint64_t xa = gdn::f2pack(x.x, x.y), xb = gdn::f2pack(x.z, x.w);
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            ac[r] = gdn::fma2(st[r][2 * m], xa, ac[r]);
                            ac[r] = gdn::fma2(st[r][2 * m + 1], xb, ac[r]);
                        }
                    }
                    float p[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float2 f = gdn::f2unpack(ac[r]);
                        p[r] = f.x + f.y;
                    }
                    // reduce over the eight column slices: halving on lane bits 4 and
                    // 2, then both lanes of a pair add; lanes 2i, 2i + 1 end with row
                    // 4rg + i
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const bool up = cg & 4;
                        const float keep = up ? p[2 + e] : p[e], send = up ? p[e] : p[2 + e];
                        p[e] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                    }
                    {
                        const bool up = cg & 2;
                        const float keep = up ? p[1] : p[0], send = up ? p[0] : p[1];
                        p[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                    }
                    p[0] += __shfl_xor_sync(0xffffffffu, p[0], 1);
                    if ((cg & 1) == (v & 1)) res[(4 * rg + (cg >> 1)) * RS + v] = p[0];
                }
            }
            // ---- D: u = T e (e_j = v_j - Gamma_j a_j), then o = Gamma b + CQ u; the
            //      two threads of state row si take the even and the odd nodes ------
            __syncthreads();  // T and every a_t / b_t are in place
            {
                const int si = tid >> 1, sh = tid & 1;
                uint64_t *bv = bvv + vb;
                if (!gdn::mbar_wait_bounded(bv, vb ? ph_v1 : ph_v0)) timed_out = true;
                const float *vrow = sm + VB + vb * kChunk * D + si;
                const float *rrow = sm + RES + si * RS;
                float u[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) u[k] = 0.f;
#pragma unroll 4
                for (int j = 0; j < L; ++j) {
                    const float e = vrow[j * D] - sm[GAM + j] * rrow[j];
                    const float4 t0 = *reinterpret_cast<const float4 *>(sm + TT + j * CS + 8 * sh);
                    const float4 t1 = *reinterpret_cast<const float4 *>(sm + TT + j * CS + 8 * sh + 4);
                    u[0] = fmaf(t0.x, e, u[0]);
                    u[1] = fmaf(t0.y, e, u[1]);
                    u[2] = fmaf(t0.z, e, u[2]);
                    u[3] = fmaf(t0.w, e, u[3]);
                    u[4] = fmaf(t1.x, e, u[4]);
                    u[5] = fmaf(t1.y, e, u[5]);
                    u[6] = fmaf(t1.z, e, u[6]);
                    u[7] = fmaf(t1.w, e, u[7]);
                }
                float *urow = sm + UB + si * US;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int t = 2 * k + sh;
                    urow[t] = u[k];
                    if (t < L) a.replay[((nf + t) * a.Hv + h) * a.rstride + D + si] = u[k];
                }
                __syncwarp();
                float ov[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) ov[k] = sm[GAM + 2 * k + sh] * rrow[kChunk + 2 * k + sh];
#pragma unroll 4
                for (int j = 0; j < L; ++j) {
                    const float uj = urow[j];
                    const float4 c0 = *reinterpret_cast<const float4 *>(sm + CQT + j * CS + 8 * sh);
                    const float4 c1 = *reinterpret_cast<const float4 *>(sm + CQT + j * CS + 8 * sh + 4);
                    ov[0] = fmaf(c0.x, uj, ov[0]);
                    ov[1] = fmaf(c0.y, uj, ov[1]);
                    ov[2] = fmaf(c0.z, uj, ov[2]);
                    ov[3] = fmaf(c0.w, uj, ov[3]);
                    ov[4] = fmaf(c1.x, uj, ov[4]);
                    ov[5] = fmaf(c1.y, uj, ov[5]);
                    ov[6] = fmaf(c1.z, uj, ov[6]);
                    ov[7] = fmaf(c1.w, uj, ov[7]);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int t = 2 * k + sh;
                    if (t < L) a.o[((nf + t) * a.Hv + h) * D + si] = a.q_scale * ov[k];
                }
            }
            (vb ? ph_v1 : ph_v0) ^= 1;
            (vb ? pend_v1 : pend_v0) = false;
            __syncthreads();  // every u_t is in place

            // ---- E: the state at the end of the chunk -----------------------------
            if (c + 1 < nchunks) {
                const float gl = sm[GAM + L - 1];
                const uint64_t g2 = gdn::f2pack(gl, gl);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int m = 0; m < 8; ++m) st[r][m] = gdn::mul2(st[r][m], g2);
                const float *kq = sm + KQH + 20 * cg;
                const float *up = sm + UB + (4 * rg) * US;
#pragma unroll 1
                for (int j4 = 0; j4 < (L + 3) / 4; ++j4) {
                    const float4 w = *reinterpret_cast<const float4 *>(sm + WEND + 4 * j4);
                    float4 ur[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) ur[r] = *reinterpret_cast<const float4 *>(up + r * US + 4 * j4);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const float wj = jj == 0 ? w.x : jj == 1 ? w.y : jj == 2 ? w.z : w.w;
                        uint64_t cc[4];
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float uj = jj == 0 ? ur[r].x : jj == 1 ? ur[r].y : jj == 2 ? ur[r].z : ur[r].w;
                            cc[r] = gdn::f2pack(wj * uj, wj * uj);
                        }
                        const float *krow = kq + (4 * j4 + jj) * KQS;
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const float4 x = *reinterpret_cast<const float4 *>(krow + 4 * m);
                            const uint64_t xa = gdn::f2pack(x.x, x.y), xb = gdn::f2pack(x.z, x.w);
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                st[r][2 * m] = gdn::fma2(cc[r], xa, st[r][2 * m]);
                                st[r][2 * m + 1] = gdn::fma2(cc[r], xb, st[r][2 * m + 1]);
                            }
                        }
                    }
                }
            }
        }
        if (__syncthreads_or(timed_out)) {
            aborted = true;
            break;
        }
    }
    if (aborted && tid == 0) {
        // a copy never landed: give the outstanding ones one more bounded wait
        gdn::record_status(a.status, GDN_DEV_TIMEOUT);
        if (pend_kq) gdn::mbar_wait_bounded(bkq, ph_kq);
        if (pend_v0) gdn::mbar_wait_bounded(bvv, ph_v0);
        if (pend_v1) gdn::mbar_wait_bounded(bvv + 1, ph_v1);
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

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

    const ChainArgs a{xc, ba, ba_stride, dt_bias, A, ssm, q_scale, parents, node_off, slot_map, o, replay,
                      replay_stride, status, int(S), int(N), int(P), dims->h_k, int(Hv), int(C),
                      dims->max_seq_nodes};
    auto k = chain_verify_kernel;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(BYTES)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int sms = sm_count();
    if (sms <= 0) return GDN_ERR_LAUNCH;
    const int64_t items = S * Hv;
    const unsigned grid = unsigned(std::min<int64_t>(items, 2 * int64_t(sms)));
    return gdn::launch_pdl(k, dim3(grid), dim3(kThreads), BYTES, static_cast<cudaStream_t>(stream), a) ==
                   cudaSuccess
               ? GDN_OK
               : GDN_ERR_LAUNCH;
}
