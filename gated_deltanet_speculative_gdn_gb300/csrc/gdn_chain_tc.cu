// gdn_chain_tc.cu - chain verify (d = 128) on the tensor cores, chunked form,
// the state held in tensor memory for the whole chain.
//
// lucebox PR #707 "perf(qwen35): fuse the DFlash2 concurrent verify Gated
// DeltaNet route", Scope and fallback: dense chains keep a path of their own;
// TensorSharp PR #175 "Feature/support dflash2", change 1: the recurrence over
// a run of tokens goes through a chunked GDN kernel.  Same outputs and replay
// rows as the tree verify (a chain is a tree).
//
// Method (per chunk of L <= 16 nodes, S the state at the chunk's start; the
// derivation is in gdn_chain.cu):
//     a_t = S k^_t, b_t = S q^_t                          (the contraction)
//     u   = T (v - Gamma a),  T = (I + diag(beta) CK)^-1 diag(beta)
//     o_t = q_scale (Gamma_t b_t + sum_{j<=t} CQ[t][j] u_j)
//     S  <- Gamma_{L-1} S + sum_j gamma_{j->L-1} u_j k^_j^T (a rank-L update)
//
// Mapping (GB300).  Persistent CTAs, two per SM, one (sequence, head) item at
// a time each.  The item's 128 x 128 fp32 state lives in tensor memory as an
// accumulator (columns 0-127, row i in lane i) from its load to the item's
// last chunk:
//   * the contraction reads it directly as the A operand: D = S [k | q | k_lo
//     | q_lo]^T (tf32, N = 64; the tensor cores read the fp32 state as its
//     tf32 part S_hi) plus S_lo [k | q]^T with S_lo = S - S_hi and the raw
//     rows in fp16 (kind::f16, N = 32).  Every row of S_lo and every raw
//     row is scaled by a power of two chosen from its largest entry before
//     the fp16 rounding, and the epilogue undoes the two scales exactly, so
//     the split does not depend on the scale of the data; S_lo carries
//     2^-10 of S, so fp16's 11-bit mantissa leaves the product at ~2^-21;
//   * the rank-16 update accumulates into it: S += U' [k^ | k^_lo]^T and
//     U'_lo k^^T, with U' = gamma_{j->L-1} u_j in tensor memory (columns
//     224-255, the A operand) and k^ transposed in shared memory;
//   * between the two, the epilogue warps scale it by Gamma_{L-1} (tensor
//     memory load, multiply, store) and rewrite S_lo (fp16, shared memory).
// q/k rows arrive raw by TMA in the 128-byte swizzle (the tensor cores'
// K-major layout); the epilogue applies 1/|k| and 1/|q|.  The contraction
// columns are 128-191 (tf32 part) and 192-223 (fp16 part).
//
// Warp roles (10 warps):
//   0-3  epilogue, thread i = state row i = tensor-memory lane i: the state's
//        load, the per-row solve (u = T e, then o), outputs, U', the scale and
//        the S_lo rewrite;
//   4-7  prep: gates, the lo rows of B and its fp16 copy, the Gram terms (CUDA
//        cores, 4 x 4 tiles over the four K-chunks), coefficients, T (one
//        column per lane, in registers), the replay rows' k^, k^ transposed;
//   8    lane 0: TMA of the next chunk's q/k rows, then the tf32 contraction;
//   9    lane 0: the fp16 contraction, then the update.
// Every mbarrier completes once per chunk, so a chunk counter gives every
// wait's phase.
#include <algorithm>

#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_tma.h"

namespace {
namespace ctc {
constexpr int D = 128, kChunk = 16;
constexpr int kWarps = 10, kThreads = kWarps * 32;
constexpr int kPrep0 = 4, kProdX = 8, kIssueW = 9;
constexpr int kMaxItems = 16;  // items per CTA (two lanes of warp 0 per item at set-up)
constexpr int RS = 20;         // row stride of the 16 x 16 matrices (16-byte rows)

// small area (4-byte words) at the base of shared memory
constexpr int S_CK = 0;                  // [16][RS] CK[t][j], j < t
constexpr int S_GR = S_CK + 16 * RS;     // [16][32] raw k_j . [k | q]_c
constexpr int S_QQ = S_GR + 16 * 32;     // [16] raw q_t . q_t
constexpr int S_BETA = S_QQ + 16, S_DEC = S_BETA + 16;
constexpr int S_CB = S_DEC + 16;         // two buffers (chunk parity) of what the epilogue reads:
constexpr int C_TR = 0;                  //   [16][RS] T transposed: row j holds T[t][j] over t
constexpr int C_CQ = C_TR + 16 * RS;     //   [16][RS] CQ transposed (without q_scale)
constexpr int C_GAM = C_CQ + 16 * RS;    //   [16] Gamma_t
constexpr int C_W = C_GAM + 16;          //   [16] gamma_{j->L-1}
constexpr int C_RK = C_W + 16;           //   [16] 1/|k_t|
constexpr int C_RQ = C_RK + 16;          //   [16] 1/|q_t|
constexpr int C_FS = C_RQ + 16;          //   [32] 2^-f of the fp16 copy of raw row c of [k | q]
constexpr int C_WORDS = C_FS + 32;
constexpr int S_BAR = (S_CB + 2 * C_WORDS + 1) & ~1;
enum { B_LAND, B_BLO, B_PREP, B_KT, B_BFREE, B_DHI, B_DLO, B_DFREE, B_UPRDY, B_UDONE, B_SRDY, B_DRAIN, B_NEVER, N_BARS };
constexpr int S_TMEM = S_BAR + 2 * N_BARS;
constexpr int S_ABORT = S_TMEM + 1;
constexpr int S_NV = S_ABORT + 1;
constexpr int S_ERR = S_NV + 1;
constexpr int S_LIST = (S_ERR + 4) & ~3;  // kMaxItems int4 (item, n0, n, slot)
constexpr int SMALL_WORDS = S_LIST + 4 * kMaxItems;

// tiles (1024-byte aligned, after the small area); 128-byte swizzled rows
constexpr uint32_t kBChunk = 64 * 128;          // B: [64 rows][32 fp32]: raw k | raw q | k lo | q lo
constexpr uint32_t kBBChunk = 32 * 128;         // B in fp16: [32 rows][64 fp16]: raw k | raw q, row-scaled
constexpr uint32_t kSLChunk = 128 * 128;        // S_lo in fp16: [128 rows][64 fp16], row-scaled
constexpr uint32_t T_BT = 0;
constexpr uint32_t T_BB = T_BT + 4 * kBChunk;
constexpr uint32_t T_SL = T_BB + 2 * kBBChunk;
constexpr uint32_t T_KT = T_SL + 2 * kSLChunk;  // k^ transposed: [128 rows (column c)][32 fp32]: hi | lo
constexpr uint32_t TILES = T_KT + 128 * 128;
constexpr size_t BYTES = size_t(SMALL_WORDS) * 4 + 1024 + TILES;
static_assert(BYTES <= 113 * 1024, "two CTAs per SM");

// tensor-memory columns of a CTA
constexpr uint32_t TM_COLS = 256, TM_S = 0, TM_DH = 128, TM_DL = 192, TM_U = 224;
// instruction descriptors: fp32 accumulate, K-major operands, M = 128
constexpr uint32_t IDESC_X = (1u << 4) | (2u << 7) | (2u << 10) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t IDESC_W = (1u << 4) | (0u << 7) | (0u << 10) | ((32u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint32_t IDESC_U = (1u << 4) | (2u << 7) | (2u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// byte offset of 16-byte unit u of row r in a 128-byte swizzled tile
__device__ __forceinline__ uint32_t swz(int r, int u) { return uint32_t(r) * 128u + (uint32_t(u ^ (r & 7)) << 4); }

__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-collective: thread t writes 32 consecutive fp32 columns of lane (taddr lane) + t.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float lo_part(float x) { return x - gdn::tf32_hi(x); }

// Exponent e such that m 2^e lies in [2^14, 2^15) (0 for m = 0): a row scaled by
// 2^e keeps fp16's full 11-bit precision whatever the scale of the data.
__device__ __forceinline__ int fp16_exp(float m) {
    const int be = int((__float_as_uint(m) >> 23) & 0xffu);  // m = 1.f 2^(be - 127) (m >= 0, finite)
    if (be == 0) return 0;                                   // zero (or subnormal): no scaling
    return min(14 - (be - 127), 126);
}
// Exponent e for the lo parts of values whose largest magnitude is m: every
// lo part is below 2^(E - 10) when m = 1.f 2^E, so lo 2^e stays below 2^15.
__device__ __forceinline__ int lo_fp16_exp(float m) {
    const int be = int((__float_as_uint(m) >> 23) & 0xffu);
    if (be == 0) return 0;
    return min(152 - be, 126);
}
// 2^e as a float, for -126 <= e <= 127
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(uint32_t(127 + e) << 23); }

// S_lo of 32 state values, scaled by 2^e, as fp16 into units 4h .. 4h + 3 of row i
__device__ __forceinline__ void store_slo(unsigned char *slr, int i, int h, const float (&sv)[32], float sc) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(slr + swz(i, 4 * h + q)) =
            make_uint4(gdn::pack_f16x2(lo_part(sv[8 * q]) * sc, lo_part(sv[8 * q + 1]) * sc),
                       gdn::pack_f16x2(lo_part(sv[8 * q + 2]) * sc, lo_part(sv[8 * q + 3]) * sc),
                       gdn::pack_f16x2(lo_part(sv[8 * q + 4]) * sc, lo_part(sv[8 * q + 5]) * sc),
                       gdn::pack_f16x2(lo_part(sv[8 * q + 6]) * sc, lo_part(sv[8 * q + 7]) * sc));
}

__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gdn::smem_addr(bar)) : "memory");
}
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (*abort_flag) return false;
    if (gdn::mbar_wait_bounded(bar, parity)) return true;
    *abort_flag = 1;
    return false;
}
__device__ __forceinline__ void prep_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
}  // namespace ctc

struct ChainTcArgs {
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
    uint64_t stall_ns;  // test hook: a wait that nothing ends, for this long (0: none)
};

__global__ void __launch_bounds__(ctc::kThreads, 2)
    chain_verify_tc_kernel(const __grid_constant__ CUtensorMap xmap, const ChainTcArgs a) {
    using namespace ctc;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    int *words = reinterpret_cast<int *>(smem_raw);
    float *fw = reinterpret_cast<float *>(smem_raw);
    unsigned char *tiles = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw + SMALL_WORDS * 4) + 1023) & ~uintptr_t(1023));
    const uint32_t tb = gdn::smem_addr(tiles);
    uint64_t *bars = reinterpret_cast<uint64_t *>(words + S_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(words + S_TMEM);
    volatile int *abort_flag = words + S_ABORT;
    int4 *list = reinterpret_cast<int4 *>(words + S_LIST);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int total = a.S * a.Hv;
    const int G = a.Hv / a.Hk;
    gdn::grid_dep_launch();

    // ---- set-up from the caller's index inputs only, before the wait: this
    //      CTA's chains (two lanes per item check its parents), barriers,
    //      tensor memory ------------------------------------------------------
    if (warp == 0) {
        const int kk = lane >> 1, half = lane & 1;
        const int it = blockIdx.x + kk * gridDim.x;
        const bool in = kk < kMaxItems && it < total;
        int n0 = 0, n = 0, slot = 0, err = 0;
        bool bad = false;
        if (in) {
            const int s = it / a.Hv;
            n0 = a.node_off[s];
            const int n1 = a.node_off[s + 1];
            n = n1 - n0;
            if (n0 < 0 || n1 < n0 || n1 > a.N || (s == 0 && n0 != 0) || (s == a.S - 1 && n1 != a.N) ||
                n > a.max_nodes) {
                err = GDN_DEV_BAD_NODE_OFF;
            } else if (n > 0) {
                slot = a.slot_map[s];
                if (slot < 0 || slot >= a.P) err = GDN_DEV_BAD_SLOT;
            }
            if (!err) {
#pragma unroll 8
                for (int q = 0; q < 32; ++q) {
                    const int i = 32 * half + q;
                    if (i < n) bad |= a.parents[n0 + i] != i - 1;
                }
            }
        }
        bad |= __shfl_xor_sync(0xffffffffu, bad ? 1 : 0, 1) != 0;
        if (!err && bad) err = GDN_DEV_BAD_PARENT;
        if (lane == 0) words[S_ERR] = 0;
        __syncwarp();
        if (err && half == 0) words[S_ERR] = err;  // recorded after the wait
        const bool valid = in && !err && n > 0 && half == 0;
        const unsigned m = __ballot_sync(0xffffffffu, valid);
        if (valid) list[__popc(m & ((1u << lane) - 1u))] = make_int4(it, n0, n, slot);
        if (lane == 0) words[S_NV] = __popc(m);
    }
    if (tid == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            uint32_t count = 1;
            if (i == B_BLO || i == B_PREP || i == B_KT || i == B_DFREE || i == B_UPRDY || i == B_SRDY) count = 4;
            if (i == B_BFREE) count = 6;  // both contraction issuers and the four prep warps
            if (i == B_DRAIN) count = 2;
            gdn::mbar_init(bars + i, count);
        }
        gdn::fence_mbar_init();
        *abort_flag = 0;
    }
    if (warp == 0) {
        gdn::tmem_alloc(tmem_slot, TM_COLS);
        gdn::tmem_relinquish();
    }
    gdn::tc_fence_before_sync();
    __syncthreads();
    gdn::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int nv = words[S_NV];
    gdn::grid_dep_wait();  // xc, ba, the state pool, status
    if (tid == 0 && words[S_ERR]) gdn::record_status(a.status, words[S_ERR]);

    if (warp == kProdX) {
        // ---- q/k rows by TMA, then S_hi [B_hi | B_lo] --------------------------
        if (lane == 0) {
            int g = 0, last_land = -1;
            bool ok = true;
            // test hook: the producer of CTA 0 waits on a barrier that nothing
            // completes, so the wait runs out before any copy is issued, and
            // every other role's wait runs out in turn
            if (a.stall_ns && blockIdx.x == 0 && !gdn::mbar_wait_bounded(bars + B_NEVER, 0, a.stall_ns)) {
                *abort_flag = 1;
                ok = false;
            }
            for (int v = 0; v < nv && ok; ++v) {
                const int4 e = list[v];
                const int h = e.x % a.Hv, kh = h / G;
                const int nch = (e.z + kChunk - 1) / kChunk;
                for (int c = 0; c < nch; ++c, ++g) {
                    if (g > 0 && !wait_or_abort(bars + B_BFREE, uint32_t((g - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint64_t *land = bars + B_LAND;
                    gdn::mbar_arrive_expect_tx(land, 8 * kChunk * 128);
#pragma unroll
                    for (int kc = 0; kc < 4; ++kc) {
                        gdn::tma_load_2d(tiles + T_BT + kc * kBChunk, &xmap, a.Hk * D + kh * D + 32 * kc,
                                         e.y + kChunk * c, land);
                        gdn::tma_load_2d(tiles + T_BT + kc * kBChunk + kChunk * 128, &xmap, kh * D + 32 * kc,
                                         e.y + kChunk * c, land);
                    }
                    last_land = g;
                    if (!wait_or_abort(bars + B_BLO, uint32_t(g & 1), abort_flag) ||
                        !wait_or_abort(bars + B_SRDY, uint32_t(g & 1), abort_flag) ||
                        (g > 0 && !wait_or_abort(bars + B_DFREE, uint32_t((g - 1) & 1), abort_flag))) {
                        ok = false;
                        break;
                    }
                    gdn::tc_fence_after_sync();
#pragma unroll 1
                    for (int ks = 0; ks < 16; ++ks)
                        mma_tf32_ta(tmem + TM_DH, tmem + TM_S + 8 * ks,
                                    gdn::desc_sw128(tb + T_BT + (ks >> 2) * kBChunk) + 2 * (ks & 3), IDESC_X,
                                    ks > 0);
                    gdn::mma_commit(bars + B_DHI);
                    gdn::mma_commit(bars + B_BFREE);
                }
            }
            gdn::mma_commit(bars + B_DRAIN);
            gdn::mbar_wait_bounded(bars + B_DRAIN, 0);
            // after a timeout a q/k copy may still be in flight: wait for it (bounded)
            if (*abort_flag && last_land >= 0) gdn::mbar_wait_bounded(bars + B_LAND, uint32_t(last_land & 1));
        }
    } else if (warp == kIssueW) {
        // ---- S_lo [k | q] in fp16, then the rank-16 update ----------------------
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int v = 0; v < nv && ok; ++v) {
                const int nch = (list[v].z + kChunk - 1) / kChunk;
                for (int c = 0; c < nch; ++c, ++g) {
                    if (!wait_or_abort(bars + B_BLO, uint32_t(g & 1), abort_flag) ||
                        !wait_or_abort(bars + B_SRDY, uint32_t(g & 1), abort_flag) ||
                        (g > 0 && !wait_or_abort(bars + B_DFREE, uint32_t((g - 1) & 1), abort_flag))) {
                        ok = false;
                        break;
                    }
                    gdn::tc_fence_after_sync();
#pragma unroll 1
                    for (int ks = 0; ks < 8; ++ks)
                        gdn::mma_f16(tmem + TM_DL, gdn::desc_sw128(tb + T_SL + (ks >> 2) * kSLChunk) + 2 * (ks & 3),
                                     gdn::desc_sw128(tb + T_BB + (ks >> 2) * kBBChunk) + 2 * (ks & 3), IDESC_W,
                                     ks > 0);
                    gdn::mma_commit(bars + B_DLO);
                    gdn::mma_commit(bars + B_BFREE);
                    if (!wait_or_abort(bars + B_UPRDY, uint32_t(g & 1), abort_flag) ||
                        !wait_or_abort(bars + B_KT, uint32_t(g & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    gdn::tc_fence_after_sync();
                    if (c + 1 < nch) {
                        // S += U'_hi k^_hi + U'_hi k^_lo + U'_lo k^_hi (K = 16: two steps each)
#pragma unroll 1
                        for (int p = 0; p < 3; ++p)
#pragma unroll 1
                            for (int ks = 0; ks < 2; ++ks)
                                mma_tf32_ta(tmem + TM_S, tmem + TM_U + (p == 2 ? 16 : 0) + 8 * ks,
                                            gdn::desc_sw128(tb + T_KT) + (p == 1 ? 4 : 0) + 2 * ks, IDESC_U, 1);
                    }
                    gdn::mma_commit(bars + B_UDONE);
                }
            }
            gdn::mma_commit(bars + B_DRAIN);
            gdn::mbar_wait_bounded(bars + B_DRAIN, 0);
        }
    } else if (warp >= kPrep0) {
        // ---- prep: all four warps walk every chunk (after a timeout too, so
        //      that they keep meeting at their named barrier) ---------------------
        const int pt = tid - kPrep0 * 32;  // 0..127
        float2 gate_nx = make_float2(0.f, 0.f);
        float dtb = 0.f, Ah = 0.f;
        auto load_gates = [&](int v, int c) {
            if (warp != kPrep0 || lane >= kChunk || v >= nv) return;
            const int4 e = list[v];
            const int L = min(kChunk, e.z - kChunk * c);
            if (lane < L) {
                const float *p = a.ba + (int64_t(e.y) + kChunk * c + lane) * a.ba_stride;
                const int h = e.x % a.Hv;
                gate_nx = make_float2(__ldg(p + h), __ldg(p + a.Hv + h));
            }
        };
        load_gates(0, 0);
        int g = 0;
        for (int v = 0; v < nv; ++v) {
            const int4 e = list[v];
            const int h = e.x % a.Hv;
            const int nch = (e.z + kChunk - 1) / kChunk;
            if (warp == kPrep0) {
                dtb = __ldg(a.dt_bias + h);
                Ah = __ldg(a.A + h);
            }
            for (int c = 0; c < nch; ++c, ++g) {
                const int L = min(kChunk, e.z - kChunk * c);
                const int64_t nf = int64_t(e.y) + kChunk * c;
                float *cb = fw + S_CB + (g & 1) * C_WORDS;
                // gates of this chunk (inputs loaded one chunk ahead)
                if (warp == kPrep0 && lane < kChunk) {
                    float beta = 0.f, dec = 1.f;
                    if (lane < L) {
                        beta = gdn::sigmoid_f(gate_nx.x);
                        dec = expf(gdn::softplus_f(gate_nx.y + dtb) * Ah);
                        a.replay[((nf + lane) * a.Hv + h) * a.rstride + 2 * D] = dec;
                    }
                    fw[S_BETA + lane] = beta;
                    fw[S_DEC + lane] = dec;
                }
                if (c + 1 < nch)
                    load_gates(v, c + 1);
                else
                    load_gates(v + 1, 0);
                const bool landed = __all_sync(0xffffffffu, wait_or_abort(bars + B_LAND, uint32_t(g & 1), abort_flag));
                // per raw row r of [k | q]: its lo part into row r + 32, and an fp16
                // copy scaled by a power of two chosen from the row's largest entry.
                // Warp w takes rows 8w .. 8w + 7; lane (kc, ri) the 32 entries of
                // K-chunk kc of row 8w + ri (a quarter-warp: one chunk, eight rows
                // with distinct swizzle phases), the row maximum over four lanes.
                if (landed) {
                    const int r = 8 * (warp - kPrep0) + (lane & 7), kc = lane >> 3;
                    unsigned char *src = tiles + T_BT + kc * kBChunk;
                    float4 x[8];
                    float mx = 0.f;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        x[u] = *reinterpret_cast<const float4 *>(src + swz(r, u));
                        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(x[u].x), fabsf(x[u].y)), fmaxf(fabsf(x[u].z), fabsf(x[u].w))));
                        *reinterpret_cast<float4 *>(src + swz(r + 32, u)) =
                            make_float4(lo_part(x[u].x), lo_part(x[u].y), lo_part(x[u].z), lo_part(x[u].w));
                    }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const int ex = fp16_exp(mx);
                    const float sc = pow2f(ex);
                    if (kc == 0) cb[C_FS + r] = pow2f(-ex);
                    // fp16 K-chunk kc >> 1, units 4 (kc & 1) .. + 3 (8 fp16 each)
                    unsigned char *dst = tiles + T_BB + (kc >> 1) * kBBChunk;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        *reinterpret_cast<uint4 *>(dst + swz(r, 4 * (kc & 1) + q)) =
                            make_uint4(gdn::pack_f16x2(x[2 * q].x * sc, x[2 * q].y * sc),
                                       gdn::pack_f16x2(x[2 * q].z * sc, x[2 * q].w * sc),
                                       gdn::pack_f16x2(x[2 * q + 1].x * sc, x[2 * q + 1].y * sc),
                                       gdn::pack_f16x2(x[2 * q + 1].z * sc, x[2 * q + 1].w * sc));
                }
                gdn::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) arrive(bars + B_BLO);

                // Gram terms of the raw rows: 4 x 4 tiles (rows j0.., columns c0.. of
                // [k | q]) over one K-chunk per lane, reduced over the chunks
                {
                    // quarter-warp = one K-chunk, its eight lanes eight tiles: distinct
                    // rows in one chunk, so the loads avoid bank conflicts
                    // only the 20 tiles the solve reads: row block jb, column block cb
                    // >= jb of the k columns (k . k), then of the q columns (k . q);
                    // five per warp, lanes 5-7 of each quarter idle
                    const int kc = (lane >> 3) & 3, slot = lane & 7;
                    const int tix = 5 * (warp - kPrep0) + min(slot, 4);
                    const int grp = tix >= 10, tk = tix - 10 * grp;
                    const int jb = tk < 4 ? 0 : tk < 7 ? 1 : tk < 9 ? 2 : 3;
                    const int cbl = jb + (tk - (jb == 0 ? 0 : jb == 1 ? 4 : jb == 2 ? 7 : 9));
                    const int j0 = 4 * jb, c0 = 4 * cbl + kChunk * grp;
                    const bool active = slot < 5;
                    const unsigned char *src = tiles + T_BT + kc * kBChunk;
                    float acc[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) acc[q] = 0.f;
#pragma unroll 2
                    for (int u = 0; u < (active ? 8 : 0); ++u) {
                        float4 xc[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) xc[q] = *reinterpret_cast<const float4 *>(src + swz(c0 + q, u));
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            const float4 xj = *reinterpret_cast<const float4 *>(src + swz(j0 + r, u));
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[4 * r + q] = gdn::fma4(xj, xc[q], acc[4 * r + q]);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const bool up = kc & 2;
                        const float keep = up ? acc[8 + q] : acc[q], send = up ? acc[q] : acc[8 + q];
                        acc[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const bool up = kc & 1;
                        const float keep = up ? acc[4 + q] : acc[q], send = up ? acc[q] : acc[4 + q];
                        acc[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
                    }
                    // this lane: row j0 + kc, columns c0 .. c0 + 3
                    if (active)
                        *reinterpret_cast<float4 *>(fw + S_GR + (j0 + kc) * 32 + c0) =
                            make_float4(acc[0], acc[1], acc[2], acc[3]);
                    if (pt < kChunk) {
                        float qq = 0.f;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
#pragma unroll 2
                            for (int u = 0; u < 8; ++u) {
                                const float4 x = *reinterpret_cast<const float4 *>(tiles + T_BT + kk * kBChunk +
                                                                                   swz(kChunk + pt, u));
                                qq = gdn::fma4(x, x, qq);
                            }
                        fw[S_QQ + pt] = qq;
                    }
                }
                prep_sync();
                // norms, Gamma_t and the end weights
                if (pt < kChunk) {
                    cb[C_RK + pt] = rsqrtf(fw[S_GR + pt * 32 + pt] + 1e-6f);
                } else if (pt < 2 * kChunk) {
                    const int t = pt - kChunk;
                    cb[C_RQ + t] = rsqrtf(fw[S_QQ + t] + 1e-6f);
                } else if (pt < 3 * kChunk) {
                    const int t = pt - 2 * kChunk;
                    float gam = 1.f;
                    for (int s2 = 0; s2 <= t; ++s2) gam *= fw[S_DEC + s2];
                    cb[C_GAM + t] = gam;
                } else if (pt < 4 * kChunk) {
                    const int j = pt - 3 * kChunk;
                    float w = 0.f;
                    if (j < L) {
                        w = 1.f;
                        for (int s2 = j + 1; s2 < L; ++s2) w *= fw[S_DEC + s2];
                    }
                    cb[C_W + j] = w;
                }
                prep_sync();
                // CK[t][j] = gamma_{j->t} k^_j . k^_t (j < t), CQ[t][j] = gamma_{j->t} k^_j . q^_t (j <= t)
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int en = pt + 128 * m, t = en >> 4, j = en & 15;
                    float ck = 0.f, cq = 0.f;
                    if (t < L && j <= t) {
                        float gm = 1.f;  // gamma_{j->t}, as a product
                        for (int s2 = j + 1; s2 <= t; ++s2) gm *= fw[S_DEC + s2];
                        const float rkj = cb[C_RK + j];
                        if (j < t) ck = gm * (fw[S_GR + j * 32 + t] * (rkj * cb[C_RK + t]));
                        cq = gm * (fw[S_GR + j * 32 + kChunk + t] * (rkj * cb[C_RQ + t]));
                    }
                    fw[S_CK + t * RS + j] = ck;
                    cb[C_CQ + j * RS + t] = cq;
                }
                prep_sync();
                if (warp == kPrep0) {
                    // T = (I + diag(beta) CK)^-1 diag(beta): lane j forms column j
                    // by forward substitution, in registers
                    if (lane < kChunk) {
                        const int j = lane;
                        float tc[kChunk];
#pragma unroll
                        for (int t = 0; t < kChunk; ++t) {
                            float acc = 0.f;
#pragma unroll
                            for (int s2 = 0; s2 < t; ++s2) acc = fmaf(fw[S_CK + t * RS + s2], tc[s2], acc);
                            const float b = fw[S_BETA + t];
                            tc[t] = t == j ? b : (t > j ? -b * acc : 0.f);
                            cb[C_TR + j * RS + t] = tc[t];
                        }
                    }
                } else if (landed) {
                    // the replay rows' k^ (raw k times 1/|k|)
                    for (int idx = pt - 32; idx < kChunk * 32; idx += 96) {
                        const int t = idx >> 5, u = idx & 31;  // node t, logical 16-byte unit u of 32
                        if (t < L) {
                            const float4 x = *reinterpret_cast<const float4 *>(tiles + T_BT + (u >> 3) * kBChunk +
                                                                               swz(t, u & 7));
                            const float r = cb[C_RK + t];
                            *reinterpret_cast<float4 *>(a.replay + ((nf + t) * a.Hv + h) * a.rstride + 4 * u) =
                                make_float4(x.x * r, x.y * r, x.z * r, x.w * r);
                        }
                    }
                }
                prep_sync();
                __syncwarp();
                if (lane == 0) arrive(bars + B_PREP);
                // k^ transposed for the update, once the previous update has read it:
                // row c = [k^_0..15 [c] | their lo parts]
                const bool upd =
                    __all_sync(0xffffffffu, g == 0 || wait_or_abort(bars + B_UDONE, uint32_t((g - 1) & 1), abort_flag));
                if (upd && landed) {
                    const int c = pt;
                    float hv[kChunk];
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        const float x = *reinterpret_cast<const float *>(
                            tiles + T_BT + (c >> 5) * kBChunk + swz(j, (c & 31) >> 2) + (c & 3) * 4);
                        hv[j] = x * cb[C_RK + j];
                    }
                    unsigned char *row = tiles + T_KT;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        *reinterpret_cast<float4 *>(row + swz(c, u)) =
                            make_float4(hv[4 * u], hv[4 * u + 1], hv[4 * u + 2], hv[4 * u + 3]);
                        *reinterpret_cast<float4 *>(row + swz(c, 4 + u)) =
                            make_float4(lo_part(hv[4 * u]), lo_part(hv[4 * u + 1]), lo_part(hv[4 * u + 2]),
                                        lo_part(hv[4 * u + 3]));
                    }
                }
                gdn::fence_proxy_async_smem();
                prep_sync();  // every prep read of B is done
                if (lane == 0) {
                    arrive(bars + B_KT);
                    arrive(bars + B_BFREE);
                }
            }
        }
    } else {
        // ---- epilogue: thread i = state row i = tensor-memory lane i -----------
        const int i = tid;  // 0..127
        const uint32_t lanes = uint32_t(warp * 32) << 16;
        float row_unscale = 1.f;  // 2^-e of this row's fp16 S_lo
        int g = 0;
        bool ok = true;
        for (int v = 0; v < nv && ok; ++v) {
            const int4 e = list[v];
            const int h = e.x % a.Hv, slot = e.w;
            const int voff = 2 * a.Hk * D + h * D;
            const int nch = (e.z + kChunk - 1) / kChunk;
            // the item's state: row i into tensor memory, then its lo part (fp16,
            // scaled by 2^e from the row's largest lo entry) into S_lo
            {
                const float *src = a.ssm + ((int64_t(slot) * a.Hv + h) * D + i) * D;
                float mx = 0.f;
#pragma unroll 1
                for (int b = 0; b < 4; ++b) {
                    float sv[32];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 x = __ldg(reinterpret_cast<const float4 *>(src + 32 * b) + q);
                        sv[4 * q] = x.x;
                        sv[4 * q + 1] = x.y;
                        sv[4 * q + 2] = x.z;
                        sv[4 * q + 3] = x.w;
                    }
#pragma unroll
                    for (int q = 0; q < 32; ++q) mx = fmaxf(mx, fabsf(sv[q]));
                    tmem_st32(tmem + lanes + TM_S + 32 * b, sv);
                }
                tmem_wait_st();
                const int ex = lo_fp16_exp(mx);
                const float sc = pow2f(ex);
                row_unscale = pow2f(-ex);
#pragma unroll 1
                for (int b = 0; b < 4; ++b) {
                    float sv[32];
                    gdn::tmem_ld32(tmem + lanes + TM_S + 32 * b, sv);
                    store_slo(tiles + T_SL + (b >> 1) * kSLChunk, i, b & 1, sv, sc);
                }
                gdn::fence_proxy_async_smem();
                gdn::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) arrive(bars + B_SRDY);
            }
            for (int c = 0; c < nch; ++c, ++g) {
                const int L = min(kChunk, e.z - kChunk * c);
                const int64_t nf = int64_t(e.y) + kChunk * c;
                const bool last = c + 1 == nch;
                const float *cb = fw + S_CB + (g & 1) * C_WORDS;
                float vr[kChunk];
#pragma unroll
                for (int t = 0; t < kChunk; ++t)
                    vr[t] = t < L ? gdn::ldg_pinned(a.xc + (nf + t) * int64_t(a.C) + voff + i) : 0.f;
                // warp-uniform: the tensor-memory loads below are warp-collective
                if (!__all_sync(0xffffffffu, wait_or_abort(bars + B_DHI, uint32_t(g & 1), abort_flag) &&
                                                 wait_or_abort(bars + B_DLO, uint32_t(g & 1), abort_flag) &&
                                                 wait_or_abort(bars + B_PREP, uint32_t(g & 1), abort_flag))) {
                    ok = false;
                    break;
                }
                gdn::tc_fence_after_sync();
                // a_t (raw k): fp16 part (unscaled) + tf32 lo part + tf32 hi part
                float ar[kChunk], tmp[kChunk];
                gdn::tmem_ld16(tmem + lanes + TM_DL, ar);
                gdn::tmem_ld16(tmem + lanes + TM_DH + 32, tmp);
#pragma unroll
                for (int t = 0; t < kChunk; ++t) ar[t] = fmaf(ar[t], row_unscale * cb[C_FS + t], tmp[t]);
                gdn::tmem_ld16(tmem + lanes + TM_DH, tmp);
                // e_j = v_j - Gamma_j a_j (a_j = S k^_j)
#pragma unroll
                for (int j = 0; j < kChunk; ++j) {
                    const float aj = (ar[j] + tmp[j]) * cb[C_RK + j];
                    vr[j] = j < L ? vr[j] - cb[C_GAM + j] * aj : 0.f;
                }
                // u = T e, column by column (j ascending, as packed node pairs;
                // T[t][j] is zero for t < j)
                float u[kChunk];
                {
                    uint64_t up[kChunk / 2];
#pragma unroll
                    for (int q = 0; q < kChunk / 2; ++q) up[q] = gdn::f2pack(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        const uint64_t ee = gdn::f2pack(vr[j], vr[j]);
                        const ulonglong2 *col = reinterpret_cast<const ulonglong2 *>(cb + C_TR + j * RS);
#pragma unroll
                        for (int q4 = j / 4; q4 < kChunk / 4; ++q4) {
                            const ulonglong2 c = col[q4];
                            up[2 * q4] = gdn::fma2(c.x, ee, up[2 * q4]);
                            up[2 * q4 + 1] = gdn::fma2(c.y, ee, up[2 * q4 + 1]);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kChunk / 2; ++q) {
                        const float2 uv = gdn::f2unpack(up[q]);
                        u[2 * q] = uv.x;
                        u[2 * q + 1] = uv.y;
                    }
                }
#pragma unroll
                for (int t = 0; t < kChunk; ++t)
                    if (t < L) a.replay[((nf + t) * a.Hv + h) * a.rstride + D + i] = u[t];
                // b_t (raw q) the same way, then the accumulators are free
                gdn::tmem_ld16(tmem + lanes + TM_DL + 16, ar);
                gdn::tmem_ld16(tmem + lanes + TM_DH + 48, tmp);
#pragma unroll
                for (int t = 0; t < kChunk; ++t) ar[t] = fmaf(ar[t], row_unscale * cb[C_FS + kChunk + t], tmp[t]);
                gdn::tmem_ld16(tmem + lanes + TM_DH + 16, tmp);
                gdn::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) arrive(bars + B_DFREE);
                // ob_t = Gamma_t b_t (without q_scale)
#pragma unroll
                for (int t = 0; t < kChunk; ++t) ar[t] = cb[C_GAM + t] * ((ar[t] + tmp[t]) * cb[C_RQ + t]);
                // o_t = q_scale (ob_t + sum_{j<=t} CQ[t][j] u_j)
                // (column by column as for u; CQ[t][j] is zero for t < j)
                auto emit_o = [&](const float (&ob)[kChunk], const float (&uu)[kChunk]) {
                    uint64_t op[kChunk / 2];
#pragma unroll
                    for (int q = 0; q < kChunk / 2; ++q) op[q] = gdn::f2pack(ob[2 * q], ob[2 * q + 1]);
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        const uint64_t uj = gdn::f2pack(uu[j], uu[j]);
                        const ulonglong2 *col = reinterpret_cast<const ulonglong2 *>(cb + C_CQ + j * RS);
#pragma unroll
                        for (int q4 = j / 4; q4 < kChunk / 4; ++q4) {
                            const ulonglong2 c = col[q4];
                            op[2 * q4] = gdn::fma2(c.x, uj, op[2 * q4]);
                            op[2 * q4 + 1] = gdn::fma2(c.y, uj, op[2 * q4 + 1]);
                        }
                    }
#pragma unroll
                    for (int t = 0; t < kChunk; ++t) {
                        const float2 ov = gdn::f2unpack(op[t / 2]);
                        if (t < L) a.o[((nf + t) * a.Hv + h) * D + i] = a.q_scale * ((t & 1) ? ov.y : ov.x);
                    }
                };
                if (last) {
                    emit_o(ar, u);
                } else {
                    // U' = gamma_{j->L-1} u_j and its lo part into tensor memory;
                    // the state scaled by Gamma_{L-1}
                    float uw[32];
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        uw[j] = cb[C_W + j] * u[j];
                        uw[kChunk + j] = lo_part(uw[j]);
                    }
                    tmem_st32(tmem + lanes + TM_U, uw);
                    // o waits until the next chunk's products can start: u and ob
                    // rest in the fp16 product's columns, which are free from the
                    // release of the accumulators until this chunk's S_lo is
                    // released (the next products wait for both)
                    {
                        float keep[32];
#pragma unroll
                        for (int t = 0; t < kChunk; ++t) {
                            keep[t] = u[t];
                            keep[kChunk + t] = ar[t];
                        }
                        tmem_st32(tmem + lanes + TM_DL, keep);
                    }
                    const float gl = cb[C_GAM + L - 1];
#pragma unroll 1
                    for (int b = 0; b < 4; b += 2) {
                        float sa[32], sb[32];
                        gdn::tmem_ld32x2(tmem + lanes + TM_S + 32 * b, tmem + lanes + TM_S + 32 * b + 32, sa, sb);
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            sa[q] *= gl;
                            sb[q] *= gl;
                        }
                        tmem_st32(tmem + lanes + TM_S + 32 * b, sa);
                        tmem_st32(tmem + lanes + TM_S + 32 * b + 32, sb);
                    }
                    tmem_wait_st();
                }
                gdn::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) arrive(bars + B_UPRDY);
                if (!__all_sync(0xffffffffu, wait_or_abort(bars + B_UDONE, uint32_t(g & 1), abort_flag))) {
                    ok = false;
                    break;
                }
                gdn::tc_fence_after_sync();
                if (!last) {
                    // S_lo of the updated state (fp16, row-scaled), for the next
                    // chunk's 16-bit product
                    float mx = 0.f;
#pragma unroll 1
                    for (int b = 0; b < 4; b += 2) {
                        float sa[32], sb[32];
                        gdn::tmem_ld32x2(tmem + lanes + TM_S + 32 * b, tmem + lanes + TM_S + 32 * b + 32, sa, sb);
#pragma unroll
                        for (int q = 0; q < 32; ++q) mx = fmaxf(mx, fmaxf(fabsf(sa[q]), fabsf(sb[q])));
                    }
                    const int ex = lo_fp16_exp(mx);
                    const float sc = pow2f(ex);
                    row_unscale = pow2f(-ex);
#pragma unroll 1
                    for (int b = 0; b < 4; ++b) {
                        float sv[32];
                        gdn::tmem_ld32(tmem + lanes + TM_S + 32 * b, sv);
                        store_slo(tiles + T_SL + (b >> 1) * kSLChunk, i, b & 1, sv, sc);
                    }
                    float ku[kChunk], kob[kChunk];
                    gdn::tmem_ld16(tmem + lanes + TM_DL, ku);
                    gdn::tmem_ld16(tmem + lanes + TM_DL + kChunk, kob);
                    gdn::fence_proxy_async_smem();
                    gdn::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) arrive(bars + B_SRDY);
                    emit_o(kob, ku);
                }
            }
        }
    }

    // ---- tear-down ---------------------------------------------------------------
    gdn::tc_fence_before_sync();
    __syncthreads();
    if (tid == 0 && *abort_flag) gdn::record_status(a.status, GDN_DEV_TIMEOUT);
    if (warp == 0) {
        gdn::tc_fence_after_sync();
        gdn::tmem_dealloc(tmem, TM_COLS);
    }
}

}  // namespace

namespace gdn {
// Launches the tensor-core chain kernel; the arguments are validated by the caller.
int launch_chain_tc(const gdn_dims *dims, const float *xc, const float *ba, int64_t ba_stride, const float *dt_bias,
                    const float *A, const float *ssm, float q_scale, const int32_t *parents, const int32_t *node_off,
                    const int32_t *slot_map, float *o, float *replay, int64_t replay_stride, int32_t *status,
                    void *stream) {
    using namespace ctc;
    const int64_t S = dims->n_seqs, N = dims->n_nodes, Hv = dims->h_v;
    const int64_t C = gdn::conv_channels(dims);
    CUtensorMap xmap;
    if (int rc = gdn::encode_xc_tiles(&xmap, xc, N, C, kChunk, 32, true)) return rc;
    const ChainTcArgs a{xc, ba, ba_stride, dt_bias, A, ssm, q_scale, parents, node_off, slot_map, o, replay,
                        replay_stride, status, int(S), int(N), dims->n_slots, dims->h_k, int(Hv), int(C),
                        dims->max_seq_nodes, gdn::take_test_stall_ns()};
    auto k = chain_verify_tc_kernel;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(BYTES)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int sms = gdn::sm_count_current();
    if (sms <= 0) return GDN_ERR_LAUNCH;
    const int64_t items = S * Hv;
    const int64_t grid = std::max<int64_t>(std::min<int64_t>(items, 2 * int64_t(sms)), (items + kMaxItems - 1) / kMaxItems);
    return gdn::launch_pdl(k, dim3(unsigned(grid)), dim3(kThreads), BYTES, static_cast<cudaStream_t>(stream), xmap,
                           a) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_LAUNCH;
}
}  // namespace gdn
