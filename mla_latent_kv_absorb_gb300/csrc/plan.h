// plan.h -- layout of the split plan image shared by the host planner and the kernels.
//
// The image is an int32 array.  Header (16 words), then the per-cluster item ranges, then
// the work items (8 words each), then the merge entries (4 words each).  Every section
// starts on a multiple of 8 words (32 bytes) so the kernels can read items as int4 pairs.
#pragma once
#include <stdint.h>

namespace mla {

constexpr int32_t kPlanMagic = 0x504C4D41;  // "AMLP" little-endian
constexpr int32_t kPlanVersion = 2;
constexpr int kPlanHeaderWords = 16;
constexpr int kItemWords = 8;
constexpr int kCombineWords = 4;

enum PlanHeader : int {
    kHdrMagic = 0,
    kHdrVersion = 1,
    kHdrBatch = 2,
    kHdrClusters = 3,
    kHdrItems = 4,
    kHdrPartials = 5,
    kHdrCombine = 6,
    kHdrClusterOff = 7,
    kHdrItemsOff = 8,
    kHdrCombineOff = 9,
    kHdrTotalPages = 10,
    kHdrMaxSplits = 11,
    kHdrTimeoutLo = 12,
    kHdrTimeoutHi = 13,
    kHdrQueriesPerSeq = 14,  // query tokens per sequence (1: ordinary decode)
};

// One work item: pages [page_begin, page_end) of query row `seq` (its visible context length
// is seq_len), whose pages are listed in block-table row `table_row`.  With one query token
// per sequence the two indices are equal; with q tokens per sequence, query row b * q + t is
// token t of sequence b (table row b).  partial_slot < 0: the item covers the whole row and
// writes o_lat / lse directly; otherwise it writes split partial number partial_slot of the
// workspace.
struct PlanItem {
    int32_t seq, page_begin, page_end, seq_len, partial_slot, table_row, pad1, pad2;
};

// A sequence cut into n_parts items whose partials are the consecutive slots
// first_partial .. first_partial + n_parts - 1.
struct PlanCombine {
    int32_t seq, first_partial, n_parts, pad;
};

inline int64_t plan_round8(int64_t w) { return (w + 7) & ~int64_t(7); }

// Workspace: fp32 partial outputs [num_partials][128][512], then fp32 lse [num_partials][128].
constexpr int64_t kPartialOBytes = 128LL * 512 * 4;
constexpr int64_t kPartialLseBytes = 128LL * 4;

}  // namespace mla
