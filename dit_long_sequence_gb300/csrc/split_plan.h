// split_plan.h -- host-only plan of the attention grid's tail split (which
// work items are cut into key-range pieces, and the workspace that holds the
// pieces' partials).  Used by api.cu; no kernel reads anything here, so a
// change to the plan leaves the kernels' source untouched.
#pragma once

#include <cstdint>

#include "internal.h"

namespace dit {

// Tail split of the attention grid: the last partial wave's items (tail =
// items % sms of them) are cut into f = sms / tail key ranges -- one wave of
// pieces -- at most kMaxSplit, each range at least kMinSplitTiles key tiles.
// Behind whole waves f is at least 2 even when tail > sms / 2: the pieces
// then even out the end of the grid.  A grid that is one partial wave and
// fills more than half the SMs is not split (two waves of half items would
// take as long as one of whole items).
struct SplitPlan {
    int64_t first;   // items before the split ones
    int f;           // pieces per split item (1 = no split)
    int64_t n_ctas;  // pieces in total
};
constexpr int kMinSplitTiles = 16;
inline SplitPlan plan_tail_split(int64_t items, int n_kv_tiles, int sms) {
    SplitPlan p{items, 1, 0};
    if (sms <= 0 || n_kv_tiles <= 0 || items <= 0) return p;
    const int64_t tail = items % sms;
    if (tail == 0) return p;
    int64_t f = sms / tail;
    if (items > sms && f < 2) f = 2;
    if (f > kMaxSplit) f = kMaxSplit;
    if (f > n_kv_tiles / kMinSplitTiles) f = n_kv_tiles / kMinSplitTiles;
    if (f < 2) return p;
    p.first = items - tail;
    p.f = static_cast<int>(f);
    p.n_ctas = tail * f;
    return p;
}
// Workspace bytes of a plan: partial O then partial LSE, 256-byte aligned parts.
inline int64_t split_workspace_bytes(const SplitPlan& p, int D) {
    if (p.n_ctas == 0) return 0;
    const int64_t o_bytes = p.n_ctas * 256 * D * 4;
    const int64_t l_bytes = (p.n_ctas * 256 * 4 + 255) / 256 * 256;
    return o_bytes + l_bytes;
}

}  // namespace dit
