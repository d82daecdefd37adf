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
//  apply      does nothing unless *status is zero.  The path's replay rows are
//             applied in closed form
//                 S = Gamma S0 + sum_j c_j u_j k_j^T,   c_j = prod of decays after j
//             which equals applying S <- decay_j S + u_j k_j^T root first, and
//             the accepted node's window is copied into the slot's conv
//             history.  d = 128: a persistent kernel streaming 64-row units
//             through a ring of bulk copies (commit_stream_kernel, below);
//             d < 128: CTAs of 32 state rows of one (value head, sequence) that
//             hold the rows in registers and stage the path's replay rows in
//             shared memory (commit_apply_kernel).
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_tma.h"

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

// Streaming apply for d = 128: a persistent CTA per SM walks the committing
// units of its share, a unit being 64 state rows (32 KB, half of one head's
// state).  The tile and the path's replay rows (k^_j and the unit's half of
// u_j) arrive by bulk copies into a ring of kStages stages, so each SM keeps
// well over 100 KB of state in flight while it applies earlier units.  A stage
// holds the tile and kEntries path entries; the entries of a longer path past
// those go into the tile's own space once the consumers hold the tile in
// registers (a second phase of the stage's full barrier).
//
// Producer warp p fills stage p for every kStages-th committing unit.  It finds
// its units with a warp-wide scan of `accepted` (one lane per unit, a ballot),
// walks the path (parents two per lane, shuffles), reads the path's decays,
// forms Gamma and the closed-form coefficients with a warp scan, leaves the
// unit, the path and the coefficients in the stage's small area, issues the
// copies, and copies the unit's share of the accepted window into the conv
// history.  Its first unit's walk needs only the caller's index inputs and
// runs before the launch wait.  After the last unit, the producer of the next
// stage in line leaves an end marker there.
//
// Sixteen consumer warps take the stages in ring order and learn everything
// from the stage itself: warp w owns rows 4 w .. 4 w + 3 of the unit (lane l:
// float4 column group l), loads them times Gamma, adds the path's rank-1 terms
// root first (packed pairs of fp32 multiply-adds) and stores them with
// coalesced 128-bit stores.
namespace cst {
constexpr int D = 128;
constexpr int kUnitRows = 64;                   // state rows per unit
constexpr int kEntryFloats = D + kUnitRows;     // k^_j | the unit's 64 entries of u_j
constexpr uint32_t kTileBytes = kUnitRows * D * 4;
constexpr uint32_t kEntryBytes = kEntryFloats * 4;
constexpr int kTileEntries = kTileBytes / kEntryBytes;  // second-phase entries the tile's space holds
constexpr int kConsumerWarps = kUnitRows / 4;
// per-stage small area (4-byte words)
constexpr int SM_M = 0;                         // path length; 0: nothing to apply; -1: no more units
constexpr int SM_GAM = 1;                       // Gamma, the product of the path's decays
constexpr int SM_SLOT = 2;
constexpr int SM_HH = 3;                        // 2 h + half
constexpr int SM_COEF = 4;                      // [64] coefficient of leaf-first entry i
constexpr int SM_NODE = SM_COEF + gdn::kMaxSeqNodes;  // [64] leaf-first entry i's node
constexpr int SM_WORDS = SM_NODE + gdn::kMaxSeqNodes;

// The ring: kStages stages (= producer warps) of one tile and kEntries path
// entries each.  Five stages of 16 entries when no path is longer than 16
// (trees of up to 16 nodes); four of 32 otherwise, so that a path of up to 64
// entries passes in two phases.  Barriers per stage: full (the copies landed;
// one or two phases per unit), tread (every consumer warp holds the tile) and
// empty (every consumer warp is done with the stage), one phase each per unit.
template <int kStages_, int kEntries_>
struct Ring {
    static constexpr int kStages = kStages_, kEntries = kEntries_;
    static constexpr uint32_t kStageBytes = kTileBytes + kEntries * kEntryBytes;
    static constexpr int kThreads = 32 * (kConsumerWarps + kStages);
    static constexpr int kMaxPath = kEntries + kTileEntries;
    static constexpr size_t SMALL_OFF = size_t(kStages) * kStageBytes;
    static constexpr size_t BAR_OFF = SMALL_OFF + size_t(kStages) * SM_WORDS * 4;
    static constexpr size_t BYTES = BAR_OFF + 3 * kStages * 8 + 16;
    static_assert(BYTES <= 227 * 1024, "shared memory");
    static_assert(kStageBytes % 16 == 0 && kEntryBytes % 16 == 0 && BAR_OFF % 8 == 0, "16-byte copies");
    static_assert(kEntries <= 32 && kTileEntries <= 64, "one lane per copied entry");
};
using RingShort = Ring<5, 16>;
using RingLong = Ring<4, 32>;
static_assert(RingLong::kMaxPath >= gdn::kMaxSeqNodes, "any path in two phases");

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (*abort_flag) return false;
    if (gdn::mbar_wait_bounded(bar, parity)) return true;
    *abort_flag = 1;
    return false;
}
__device__ __forceinline__ void arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gdn::smem_addr(bar)) : "memory");
}
__device__ __forceinline__ uint64_t pair_of(float x) { return gdn::f2pack(x, x); }

// A producer's view of its units: the CTA's units u = blockIdx.x + k gridDim.x
// are scanned 32 at a time; committing units are numbered in order, and
// producer p takes those numbered p, p + kStages, ...
struct UnitScan {
    int64_t next_k = 0;   // first CTA-unit index of the next chunk to scan
    unsigned mine = 0;    // this producer's units left in the current chunk (lane bits)
    int64_t chunk_k = 0;  // CTA-unit index of lane 0 of the current chunk
    int live = 0;         // committing units in the chunks scanned so far
};
// Next unit of producer p, or -1; warp-uniform.
template <int kStages>
__device__ __forceinline__ int64_t next_unit(UnitScan &sc, const CommitArgs &a, int64_t units, int p, int lane) {
    while (!sc.mine) {
        const int64_t k0 = sc.next_k;
        if (blockIdx.x + k0 * gridDim.x >= units) return -1;
        const int64_t u = blockIdx.x + (k0 + lane) * gridDim.x;
        const bool live = u < units && a.accepted[u / (2 * a.Hv)] >= 0;
        const unsigned lm = __ballot_sync(0xffffffffu, live);
        const int idx = sc.live + __popc(lm & ((1u << lane) - 1u));  // committing-unit number of this lane
        sc.mine = __ballot_sync(0xffffffffu, live && idx % kStages == p);
        sc.live += __popc(lm);
        sc.chunk_k = k0;
        sc.next_k = k0 + 32;
    }
    const int l = __ffs(sc.mine) - 1;
    sc.mine &= sc.mine - 1;
    return blockIdx.x + (sc.chunk_k + l) * gridDim.x;
}

// The path of unit u (leaf first: entry i's node in lane i % 32 of node_lo /
// node_hi), from the caller's index inputs only.
struct Path {
    int s, h, half, acc, n0, slot, m, node_lo, node_hi;
    bool bad;
};
__device__ __forceinline__ Path walk_path(const CommitArgs &a, int64_t u, int lane, int max_path) {
    Path q;
    q.s = int(u / (2 * a.Hv));
    q.h = int((u >> 1) % a.Hv);
    q.half = int(u & 1);
    q.acc = a.accepted[q.s];
    q.n0 = a.node_off[q.s];
    const int n1 = a.node_off[q.s + 1];
    q.slot = a.slot_map[q.s];
    // the preflight has checked every index (the status is zero); these tests
    // only keep the loads below in bounds
    q.bad = !(q.n0 >= 0 && n1 <= a.N && n1 - q.n0 <= gdn::kMaxSeqNodes && q.acc < n1 - q.n0 && q.slot >= 0 &&
              q.slot < a.P);
    q.node_lo = q.node_hi = -1;
    q.m = 0;
    if (!q.bad) {
        const int p_lo = lane <= q.acc ? a.parents[q.n0 + lane] : -1;
        const int p_hi = lane + 32 <= q.acc ? a.parents[q.n0 + lane + 32] : -1;
        for (int cur = q.acc; cur >= 0 && q.m < gdn::kMaxSeqNodes; ++q.m) {
            if (lane == (q.m & 31)) {
                if (q.m < 32) q.node_lo = cur; else q.node_hi = cur;
            }
            const int nx = __shfl_sync(0xffffffffu, cur < 32 ? p_lo : p_hi, cur & 31);
            q.bad |= nx >= cur;  // parents precede their children
            cur = nx;
        }
    }
    if (q.bad || q.m > max_path) q.m = 0;  // (paths are at most max_seq_nodes long)
    return q;
}
}  // namespace cst

template <class R>
__global__ void __launch_bounds__(R::kThreads, 1) commit_stream_kernel(const CommitArgs a) {
    using namespace cst;
    constexpr int kStages = R::kStages, kEntries = R::kEntries;
    constexpr uint32_t kStageBytes = R::kStageBytes;
    constexpr size_t SMALL_OFF = R::SMALL_OFF, BAR_OFF = R::BAR_OFF;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    int *small = reinterpret_cast<int *>(smem_raw + SMALL_OFF);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw + BAR_OFF);
    uint64_t *tread = full + kStages;
    uint64_t *empty = tread + kStages;
    volatile int *abort_flag = reinterpret_cast<int *>(full + 3 * kStages);  // [1]: the status was not zero
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned all = 0xffffffffu;
    const int64_t units = int64_t(a.S) * a.Hv * 2;
    const int64_t rnode = int64_t(a.Hv) * a.rstride;

    gdn::grid_dep_launch();
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            gdn::mbar_init(full + i, 1);
            gdn::mbar_init(tread + i, kConsumerWarps);
            gdn::mbar_init(empty + i, kConsumerWarps);
        }
        gdn::fence_mbar_init();
        *abort_flag = 0;
    }
    __syncthreads();

    if (warp >= kConsumerWarps) {
        // ---- producer warp p: every kStages-th committing unit, into stage p ----
        const int p = warp - kConsumerWarps;
        uint64_t *fb = full + p;
        int *sa = small + p * SM_WORDS;
        float *sf = reinterpret_cast<float *>(sa);
        unsigned char *stage = smem_raw + size_t(p) * kStageBytes;
        float *ent = reinterpret_cast<float *>(stage + kTileBytes);
        float *ent2 = reinterpret_cast<float *>(stage);  // second phase: the tile's space
        UnitScan sc;
        int nu = 0, fph = 0;  // units issued into stage p, phases of its full barrier
        bool ok = true;
        int64_t u = next_unit<kStages>(sc, a, units, p, lane);
        Path q = walk_path(a, u >= 0 ? u : 0, lane, R::kMaxPath);  // before the wait: index inputs only
        gdn::grid_dep_wait();  // status, the state pool, the replay rows and the windows
        // one reading of the status for the whole CTA: not zero, nothing is committed
        if (p == 0 && lane == 0) abort_flag[1] = *reinterpret_cast<volatile int32_t *>(a.status) != 0;
        asm volatile("bar.sync 1, %0;" ::"r"(32 * kStages) : "memory");
        const bool failed = abort_flag[1] != 0;
        if (failed) u = -1;
        while (u >= 0 && ok) {
            const int m = q.m;
            // the stage's previous unit is done with
            if (!__all_sync(all, nu == 0 || wait_or_abort(empty + p, uint32_t((nu - 1) & 1), abort_flag))) {
                ok = false;
                break;
            }
            ++nu;
            // the tile first (its index inputs are known): it travels while the
            // decays are read; the phase completes only at the arrival below
            if (m && lane == 0) {
                gdn::mbar_expect_tx(fb, kTileBytes);
                gdn::bulk_load(stage, a.ssm + ((int64_t(q.slot) * a.Hv + q.h) * D + kUnitRows * q.half) * D,
                               kTileBytes, fb);
            }
            // coefficient of leaf-first entry i = product of the decays of entries 0 .. i-1
            const float *row0 = a.replay + (int64_t(q.n0) * a.Hv + q.h) * a.rstride;
            const float d_lo = q.m && q.node_lo >= 0 ? __ldg(row0 + q.node_lo * rnode + 2 * D) : 1.0f;
            const float d_hi = q.m && q.node_hi >= 0 ? __ldg(row0 + q.node_hi * rnode + 2 * D) : 1.0f;
            float x_lo = d_lo, x_hi = d_hi;  // inclusive scans
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y_lo = __shfl_up_sync(all, x_lo, o), y_hi = __shfl_up_sync(all, x_hi, o);
                if (lane >= o) {
                    x_lo *= y_lo;
                    x_hi *= y_hi;
                }
            }
            const float tot_lo = __shfl_sync(all, x_lo, 31);
            float c_lo = __shfl_up_sync(all, x_lo, 1), c_hi = __shfl_up_sync(all, x_hi, 1);
            if (lane == 0) {
                c_lo = 1.0f;
                c_hi = 1.0f;
            }
            c_hi *= tot_lo;
            const float gam = tot_lo * __shfl_sync(all, x_hi, 31);
            if (lane < m) {
                sa[SM_COEF + lane] = __float_as_int(c_lo);
                sa[SM_NODE + lane] = q.node_lo;
            }
            if (lane + 32 < m) {
                sa[SM_COEF + lane + 32] = __float_as_int(c_hi);
                sa[SM_NODE + lane + 32] = q.node_hi;
            }
            if (lane == 0) {
                sa[SM_M] = m;
                sf[SM_GAM] = gam;
                sa[SM_SLOT] = q.slot;
                sa[SM_HH] = 2 * q.h + q.half;
            }
            __threadfence_block();
            __syncwarp();
            // phase 1: the tile (above) and the first kEntries entries, root first
            const int cnt = min(m, kEntries), cnt2 = m - cnt;
            if (lane == 0) gdn::mbar_arrive_expect_tx(fb, cnt * kEntryBytes);
            ++fph;
            __syncwarp();
            if (lane < cnt) {
                const float *rr = row0 + sa[SM_NODE + m - 1 - lane] * rnode;
                float *dst = ent + lane * kEntryFloats;
                gdn::bulk_load(dst, rr, D * 4, fb);
                gdn::bulk_load(dst + D, rr + D + kUnitRows * q.half, kUnitRows * 4, fb);
            }
            if (m) {
                // this unit's share of the history copy, conv_hist[slot] <- window of the accepted node
                const int64_t parts = int64_t(a.Hv) * 2;
                float4 *hdst = reinterpret_cast<float4 *>(a.hist + int64_t(q.slot) * 3 * a.C);
                if (!a.wref) {
                    const int64_t total4 = int64_t(3) * a.C / 4, per = (total4 + parts - 1) / parts;
                    const int64_t lo = (2 * int64_t(q.h) + q.half) * per, hi = min(total4, lo + per);
                    const float4 *wsrc =
                        reinterpret_cast<const float4 *>(a.win + (int64_t(q.n0) + q.acc) * 3 * a.C);
                    for (int64_t i = lo + lane; i < hi; i += 32) hdst[i] = __ldg(wsrc + i);
                } else {
                    // compact form: gathered through the accepted node's references from
                    // x rows and the slot's old history; a lane reads all three columns
                    // of its channel group before writing any, so in-place reuse of an
                    // old column is safe (no other thread touches that channel group)
                    const int64_t total4 = a.C / 4, per = (total4 + parts - 1) / parts;
                    const int64_t lo = (2 * int64_t(q.h) + q.half) * per, hi = min(total4, lo + per);
                    const int32_t *ref = a.wref + (int64_t(q.n0) + q.acc) * 3;
                    const int r0 = ref[0], r1 = ref[1], r2 = ref[2];
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
            }
            if (cnt2 > 0) {
                // phase 2: the remaining entries into the tile's space, once every
                // consumer warp holds the tile
                if (!__all_sync(all, wait_or_abort(tread + p, uint32_t((nu - 1) & 1), abort_flag))) {
                    ok = false;
                    break;
                }
                if (lane == 0) gdn::mbar_arrive_expect_tx(fb, cnt2 * kEntryBytes);
                ++fph;
                __syncwarp();
                for (int e = lane; e < cnt2; e += 32) {
                    const float *rr = row0 + sa[SM_NODE + m - 1 - kEntries - e] * rnode;
                    float *dst = ent2 + e * kEntryFloats;
                    gdn::bulk_load(dst, rr, D * 4, fb);
                    gdn::bulk_load(dst + D, rr + D + kUnitRows * q.half, kUnitRows * 4, fb);
                }
            }
            u = next_unit<kStages>(sc, a, units, p, lane);
            if (u >= 0) q = walk_path(a, u, lane, R::kMaxPath);
        }
        // the end marker, in the stage the consumers take after the last unit: the
        // committing units were all scanned, so every producer knows their count
        // (after a status that is not zero, stage 0 ends everything)
        if (ok && (failed ? p == 0 : sc.live % kStages == p)) {
            if (__all_sync(all, nu == 0 || wait_or_abort(empty + p, uint32_t((nu - 1) & 1), abort_flag))) {
                if (lane == 0) {
                    sa[SM_M] = -1;
                    gdn::mbar_arrive_expect_tx(fb, 0);
                }
                ++fph;
            }
        }
        // copies still in flight (after a timeout) land before the CTA exits
        if (fph > 0 && lane == 0) gdn::mbar_wait_bounded(fb, uint32_t((fph - 1) & 1));
    } else {
        // ---- consumers: warp w owns rows 4 w .. 4 w + 3 of each unit ------------
        const int r0 = 4 * warp;
        uint32_t pbits = 0;  // parity of the next phase of each stage's full barrier
        for (int j = 0;; ++j) {
            const int st = j % kStages;
            if (!__all_sync(all, wait_or_abort(full + st, (pbits >> st) & 1u, abort_flag))) break;
            pbits ^= 1u << st;
            const int *sa = small + st * SM_WORDS;
            const float *sf = reinterpret_cast<const float *>(sa);
            const int m = sa[SM_M];
            if (m < 0) break;  // no more units
            const float gam = sf[SM_GAM];
            const int slot = sa[SM_SLOT], hh = sa[SM_HH];
            const unsigned char *stage = smem_raw + size_t(st) * kStageBytes;
            // rows as pairs of fp32: (x, y) and (z, w) of each row
            uint64_t sp[4][2];
            if (m) {
                const uint64_t gg = pair_of(gam);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const ulonglong2 t =
                        *reinterpret_cast<const ulonglong2 *>(stage + ((r0 + r) * D + 4 * lane) * 4);
                    sp[r][0] = gdn::mul2(t.x, gg);
                    sp[r][1] = gdn::mul2(t.y, gg);
                }
            }
            __syncwarp();
            if (lane == 0) arrive(tread + st);  // this warp holds its rows of the tile
            // root first: slot e of phase 1 holds leaf-first entry m - 1 - e, slot e
            // of phase 2 (in the tile's space) entry m - 1 - kEntries - e
            const int cnt = min(m, kEntries), cnt2 = m - cnt;
            auto apply = [&](const float *en, float cj) {
                const ulonglong2 kv = *reinterpret_cast<const ulonglong2 *>(en + 4 * lane);
                const float4 uv = *reinterpret_cast<const float4 *>(en + D + r0);
                const float uu[4] = {uv.x * cj, uv.y * cj, uv.z * cj, uv.w * cj};
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint64_t ur = pair_of(uu[r]);
                    sp[r][0] = gdn::fma2(ur, kv.x, sp[r][0]);
                    sp[r][1] = gdn::fma2(ur, kv.y, sp[r][1]);
                }
            };
            const float *ent = reinterpret_cast<const float *>(stage + kTileBytes);
            for (int e = 0; e < cnt; ++e) apply(ent + e * kEntryFloats, sf[SM_COEF + m - 1 - e]);
            if (cnt2 > 0) {
                if (!__all_sync(all, wait_or_abort(full + st, (pbits >> st) & 1u, abort_flag))) break;
                pbits ^= 1u << st;
                const float *ent2 = reinterpret_cast<const float *>(stage);
                for (int e = 0; e < cnt2; ++e)
                    apply(ent2 + e * kEntryFloats, sf[SM_COEF + m - 1 - kEntries - e]);
            }
            __syncwarp();
            if (lane == 0) arrive(empty + st);  // this warp is done with the stage
            if (!m) continue;
            float *dst = a.ssm + ((int64_t(slot) * a.Hv + (hh >> 1)) * D + kUnitRows * (hh & 1) + r0) * D + 4 * lane;
#pragma unroll
            for (int r = 0; r < 4; ++r)
                *reinterpret_cast<ulonglong2 *>(dst + r * D) = make_ulonglong2(sp[r][0], sp[r][1]);
        }
    }
    __syncthreads();
    if (tid == 0 && *abort_flag) gdn::record_status(a.status, GDN_DEV_TIMEOUT);
}

// One persistent CTA per SM (or per unit, when there are fewer).
template <class R>
int launch_stream(const CommitArgs &a, int64_t units, cudaStream_t st) {
    auto k = commit_stream_kernel<R>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(R::BYTES)) != cudaSuccess)
        return GDN_ERR_LAUNCH;
    const int sms = gdn::sm_count_current();
    if (sms <= 0) return GDN_ERR_LAUNCH;
    const unsigned grid = unsigned(std::min<int64_t>(units, sms));
    return gdn::launch_pdl(k, dim3(grid), dim3(R::kThreads), R::BYTES, st, a) == cudaSuccess ? GDN_OK
                                                                                         : GDN_ERR_LAUNCH;
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
    if (D == cst::D)
        return dims->max_seq_nodes <= cst::RingShort::kEntries ? launch_stream<cst::RingShort>(a, S * Hv * 2, st)
                                                                : launch_stream<cst::RingLong>(a, S * Hv * 2, st);
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
