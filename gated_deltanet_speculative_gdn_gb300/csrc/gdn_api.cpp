// gdn_api.cpp - status names and the replay-row width helper of the C ABI.
#include "gdn.h"
#include "gdn_internal.h"

extern "C" const char *gdn_status_str(int code) {
    switch (code) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_NULL: return "GDN_ERR_NULL";
        case GDN_ERR_DIMS: return "GDN_ERR_DIMS";
        case GDN_ERR_STRIDE: return "GDN_ERR_STRIDE";
        case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN";
        case GDN_ERR_ALIAS: return "GDN_ERR_ALIAS";
        case GDN_ERR_LAUNCH: return "GDN_ERR_LAUNCH";
        case GDN_ERR_TMA: return "GDN_ERR_TMA";
        case GDN_ERR_ARG: return "GDN_ERR_ARG";
        case GDN_DEV_BAD_NODE_OFF: return "GDN_DEV_BAD_NODE_OFF";
        case GDN_DEV_BAD_PARENT: return "GDN_DEV_BAD_PARENT";
        case GDN_DEV_BAD_SLOT: return "GDN_DEV_BAD_SLOT";
        case GDN_DEV_DUP_SLOT: return "GDN_DEV_DUP_SLOT";
        case GDN_DEV_BAD_ACCEPTED: return "GDN_DEV_BAD_ACCEPTED";
        case GDN_DEV_TIMEOUT: return "GDN_DEV_TIMEOUT";
        case GDN_DEV_BAD_WINDOW: return "GDN_DEV_BAD_WINDOW";
        default: return "unknown";
    }
}

extern "C" size_t gdn_replay_row_floats(int d_k, int d_v) {
    if (!gdn::supported_width(d_k) || !gdn::supported_width(d_v)) return 0;
    const size_t r = static_cast<size_t>(d_k) + static_cast<size_t>(d_v) + 1;
    return (r + 3) & ~static_cast<size_t>(3);
}
