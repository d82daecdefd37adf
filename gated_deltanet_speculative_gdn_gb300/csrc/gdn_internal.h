// gdn_internal.h - host-side helpers shared by the library's entry points:
// dims checks, alignment and overlap tests.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include "gdn.h"

namespace gdn {

// Largest nodes-per-sequence any kernel variant supports.
constexpr int kMaxSeqNodes = 64;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int64_t conv_channels(const gdn_dims *d) {
    return 2 * static_cast<int64_t>(d->h_k) * d->d_k + static_cast<int64_t>(d->h_v) * d->d_v;
}

inline bool supported_width(int d) { return d == 16 || d == 32 || d == 64 || d == 128; }

// Checks the shape fields every call relies on; GDN_OK or GDN_ERR_DIMS.
inline int check_dims(const gdn_dims *d) {
    if (!d) return GDN_ERR_NULL;
    if (d->n_seqs < 0 || d->n_seqs > 65535 || d->n_nodes < 0 || d->n_slots < 1) return GDN_ERR_DIMS;
    if (d->h_k < 1 || d->h_v < d->h_k || d->h_v % d->h_k != 0 || d->h_v > 65535) return GDN_ERR_DIMS;
    if (d->d_k != d->d_v || !supported_width(d->d_k)) return GDN_ERR_DIMS;
    if (d->d_conv != 4) return GDN_ERR_DIMS;
    if (d->max_seq_nodes < 1 || d->max_seq_nodes > kMaxSeqNodes) return GDN_ERR_DIMS;
    // the state pool is addressed by int32 row coordinates in its TMA descriptor
    if (static_cast<int64_t>(d->n_slots) * d->h_v * d->d_v > INT32_MAX) return GDN_ERR_DIMS;
    if (static_cast<int64_t>(d->n_nodes) * conv_channels(d) * 3 > (int64_t(1) << 40)) return GDN_ERR_DIMS;
    return GDN_OK;
}

// A byte range [p, p + bytes) of one argument, for overlap checks.
struct Span {
    const void *p;
    size_t bytes;
};

inline bool overlaps(const Span &a, const Span &b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const auto a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// GDN_ERR_ALIAS if any output overlaps any input or another output.
inline int check_alias(const Span *outs, int n_out, const Span *ins, int n_in) {
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            if (overlaps(outs[i], ins[j])) return GDN_ERR_ALIAS;
        for (int j = i + 1; j < n_out; ++j)
            if (overlaps(outs[i], outs[j])) return GDN_ERR_ALIAS;
    }
    return GDN_OK;
}

// Launches the tensor-core chain verify (d = 128) for arguments the entry
// point has validated; GDN_OK or a host-side error.
int launch_chain_tc(const gdn_dims *dims, const float *xc, const float *ba, int64_t ba_stride, const float *dt_bias,
                    const float *A, const float *ssm, float q_scale, const int32_t *parents, const int32_t *node_off,
                    const int32_t *slot_map, float *o, float *replay, int64_t replay_stride, int32_t *status,
                    void *stream);

// The pending test stall of gdn_test_stall_next_verify (ns, 0: none); taking
// it clears it, so exactly one tensor-core verify launch receives it.
uint64_t take_test_stall_ns();

// Bytes of a [rows][stride] float tensor of which the last row holds `width`.
inline size_t strided_bytes(int64_t rows, int64_t stride, int64_t width) {
    return rows <= 0 ? 0 : static_cast<size_t>(((rows - 1) * stride + width) * 4);
}

}  // namespace gdn
