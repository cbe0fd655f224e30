// plan.cpp -- host-side split planning (mla_plan_splits) and status strings.
//
// The decode KV scan is the whole cost at long context and the split reduction that merges
// pieces of one sequence should stay cheap (the Kimi K3 decode time-share page, "Inside the
// blocks": stage 1 scan vs stage 2 KV-split reduction).  So the planner gives every CTA pair
// an equal, contiguous run of pages of the concatenated sequences, and moves a run's edge to
// the nearest sequence edge when it would otherwise leave a sliver of fewer than
// `min_pages_per_split` pages.  A sequence that ends up in one item needs no merge.
//
// By default (and with `item_cost_pages` > 0) the runs are balanced on cost instead of pages: a pair pays that
// many pages' worth for each item after its first (the next item reloads the query into the
// score CTA and the value CTA writes the previous output out).  Greedy packing under a cost cap
// is optimal for contiguous runs (extending a run never lowers its cost), so the planner
// bisects for the smallest cap whose packing fits the pairs and snaps those cuts like equal
// ones.
#include <algorithm>
#include <climits>
#include <cstring>
#include <vector>

#include "../../include/mla.h"
#include "plan.h"

using namespace mla;

// Default charge, in pages, for each item of a CTA pair after its first.  Measured at B=16,
// S=65,536: the decode kernel took 277.8 us with this charge against 284.9 us with equal runs
// (a second item reloads the query and writes an output, about the time of seven pages).
constexpr int32_t kDefaultItemCostPages = 7;

extern "C" const char* mla_status_string(mla_status s)
{
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_ALIGNMENT: return "misaligned pointer (16-byte alignment required)";
        case MLA_ERR_UNSUPPORTED: return "unsupported size";
        case MLA_ERR_WORKSPACE: return "workspace or buffer too small";
        case MLA_ERR_CUDA: return "CUDA runtime or launch failure";
        case MLA_ERR_DEVICE_FAULT: return "device reported an error (see the device error word)";
    }
    return "unknown status";
}

static int64_t plan_words(int64_t batch, int64_t clusters, int64_t items, int64_t combine)
{
    return kPlanHeaderWords + plan_round8(clusters + 1) + items * kItemWords + plan_round8(combine * kCombineWords);
}

// Greedy contiguous packing of the concatenated page list under cost cap T (T >= 1): each run
// takes pages while its cost (pages + item_cost per item after the first) stays within T.
// Returns the number of runs; writes their end points (cuts[0] = 0) when `cuts` is given.
static int64_t pack_runs(const std::vector<int64_t>& start, int batch, int64_t T, int64_t item_cost,
                         std::vector<int64_t>* cuts)
{
    const int64_t total = start[batch];
    if (cuts) cuts->assign(1, 0);
    int64_t g = 0, n = 0;
    int s = 0;
    while (g < total) {
        ++n;
        int64_t cost = 0;
        bool first = true;
        while (g < total) {
            while (start[s + 1] <= g) ++s;
            const int64_t room = T - cost - (first ? 0 : item_cost);
            if (room <= 0) break;
            const int64_t take = std::min(room, start[s + 1] - g);
            cost += (first ? 0 : item_cost) + take;
            g += take;
            first = false;
            if (g < start[s + 1]) break;  // the run ends inside this sequence
        }
        if (cuts) cuts->push_back(g);
    }
    return n;
}

extern "C" size_t mla_plan_bytes_max(int32_t batch, int32_t num_sms)
{
    if (batch <= 0 || num_sms < 2) return 0;
    const int64_t clusters = num_sms / 2;
    // every cluster boundary can cut at most one sequence: items <= batch + clusters
    const int64_t items = (int64_t)batch + clusters;
    return (size_t)(plan_words(batch, clusters, items, batch) * 4);
}

extern "C" mla_status mla_plan_splits(const int32_t* seq_lens, int32_t batch, int32_t num_sms,
                                      const mla_plan_options* opts, void* plan_host, size_t plan_capacity,
                                      mla_plan_info* info)
{
    if (!seq_lens || !plan_host || !info || batch <= 0 || num_sms < 2) return MLA_ERR_INVALID_ARG;
    int32_t min_pages = 8, max_clusters = num_sms / 2, item_cost = kDefaultItemCostPages, qps = 1;
    int64_t timeout_ns = 2000000000LL;
    if (opts) {
        if (opts->min_pages_per_split < 0 || opts->max_clusters < 0 || opts->wait_timeout_ns < 0 ||
            opts->queries_per_seq < 0 || opts->queries_per_seq > MLA_MAX_QUERIES_PER_SEQ)
            return MLA_ERR_INVALID_ARG;
        if (opts->item_cost_pages != 0) item_cost = std::max(0, opts->item_cost_pages);  // < 0: equal page runs
        if (opts->min_pages_per_split > 0) min_pages = opts->min_pages_per_split;
        if (opts->max_clusters > 0) max_clusters = std::min(max_clusters, opts->max_clusters);
        if (opts->wait_timeout_ns > 0) timeout_ns = opts->wait_timeout_ns;
        if (opts->queries_per_seq > 0) qps = opts->queries_per_seq;
    }
    // query rows: token t of sequence b (row b * qps + t) sees the first S_b - qps + 1 + t
    // cached tokens (the cache already holds all of the sequence's query tokens)
    const int64_t rows64 = (int64_t)batch * qps;
    if (rows64 > INT32_MAX / 2) return MLA_ERR_UNSUPPORTED;
    const int32_t rows = (int32_t)rows64;
    if (plan_capacity < mla_plan_bytes_max(rows, num_sms)) return MLA_ERR_WORKSPACE;
    std::vector<int32_t> row_len(rows);
    for (int b = 0; b < batch; ++b) {
        if (seq_lens[b] < qps) return MLA_ERR_INVALID_ARG;  // also rejects S_b < 1
        for (int t = 0; t < qps; ++t) row_len[(int64_t)b * qps + t] = seq_lens[b] - qps + 1 + t;
    }
    batch = rows;
    seq_lens = row_len.data();

    // pages of each query row and where each starts in the concatenated page list
    std::vector<int64_t> pages(batch), start(batch + 1);
    start[0] = 0;
    for (int b = 0; b < batch; ++b) {
        pages[b] = (seq_lens[b] + 63) / 64;
        start[b + 1] = start[b] + pages[b];
    }
    const int64_t total = start[batch];
    if (total > INT32_MAX) return MLA_ERR_UNSUPPORTED;

    // how many CTA pairs: no fewer than min_pages pages each, no more than the GPU holds
    const int64_t want = std::max<int64_t>(1, total / std::max(1, min_pages));
    int64_t C = std::min<int64_t>(max_clusters, want);

    // target cut points: equal page shares, or the cost-balanced packing (which may use fewer pairs)
    std::vector<int64_t> target;
    if (item_cost > 0 && C > 1) {
        int64_t lo = (total + C - 1) / C, hi = total + (int64_t)item_cost * batch;  // one run fits under hi
        while (lo < hi) {
            const int64_t mid = lo + (hi - lo) / 2;
            if (pack_runs(start, batch, mid, item_cost, nullptr) <= C) hi = mid;
            else lo = mid + 1;
        }
        pack_runs(start, batch, lo, item_cost, &target);
        C = (int64_t)target.size() - 1;
    } else {
        target.resize(C + 1);
        for (int64_t k = 0; k <= C; ++k) target[k] = (k * total + C / 2) / C;
    }

    // cut points in the concatenated page list, snapped to sequence edges when a cut would
    // leave fewer than min_pages pages on either side within a sequence
    std::vector<int64_t> cut(C + 1);
    cut[0] = 0;
    cut[C] = total;
    int seq = 0;
    for (int64_t k = 1; k < C; ++k) {
        int64_t g = target[k];
        while (seq < batch && start[seq + 1] <= g) ++seq;   // g lies in sequence `seq`
        if (seq < batch) {
            const int64_t lo = start[seq], hi = start[seq + 1];
            if (g - lo < min_pages) g = lo;
            else if (hi - g < min_pages) g = hi;
        }
        cut[k] = std::max(g, cut[k - 1]);
    }

    // items in global page order; cluster k owns [cut[k], cut[k+1])
    std::vector<PlanItem> items;
    std::vector<int32_t> cluster_begin(C + 1);
    std::vector<int32_t> items_per_seq(batch, 0);
    int s = 0;
    for (int64_t k = 0; k < C; ++k) {
        cluster_begin[k] = (int32_t)items.size();
        int64_t g = cut[k];
        while (s < batch && start[s + 1] <= g) ++s;
        int ss = s;
        while (g < cut[k + 1]) {
            while (start[ss + 1] <= g) ++ss;
            const int64_t e = std::min(cut[k + 1], start[ss + 1]);
            PlanItem it{};
            it.seq = ss;
            it.page_begin = (int32_t)(g - start[ss]);
            it.page_end = (int32_t)(e - start[ss]);
            it.seq_len = seq_lens[ss];
            it.partial_slot = -1;
            it.table_row = ss / qps;
            items.push_back(it);
            ++items_per_seq[ss];
            g = e;
        }
    }
    cluster_begin[C] = (int32_t)items.size();

    // partial slots and merge entries for sequences cut into several items
    std::vector<PlanCombine> combine;
    std::vector<int32_t> first_slot(batch, -1);
    int32_t next_slot = 0, max_splits = 0;
    for (int b = 0; b < batch; ++b) {
        max_splits = std::max(max_splits, items_per_seq[b]);
        if (items_per_seq[b] > 1) {
            first_slot[b] = next_slot;
            combine.push_back(PlanCombine{b, next_slot, items_per_seq[b], 0});
            next_slot += items_per_seq[b];
        }
    }
    std::vector<int32_t> used(batch, 0);
    for (auto& it : items)
        if (items_per_seq[it.seq] > 1) it.partial_slot = first_slot[it.seq] + used[it.seq]++;

    const int64_t n_items = (int64_t)items.size(), n_comb = (int64_t)combine.size();
    const int64_t words = plan_words(batch, C, n_items, n_comb);
    if ((size_t)words * 4 > plan_capacity) return MLA_ERR_WORKSPACE;

    int32_t* w = static_cast<int32_t*>(plan_host);
    std::memset(w, 0, (size_t)words * 4);
    const int64_t cl_off = kPlanHeaderWords;
    const int64_t it_off = cl_off + plan_round8(C + 1);
    const int64_t cb_off = it_off + n_items * kItemWords;
    w[kHdrMagic] = kPlanMagic;
    w[kHdrVersion] = kPlanVersion;
    w[kHdrBatch] = batch;
    w[kHdrClusters] = (int32_t)C;
    w[kHdrItems] = (int32_t)n_items;
    w[kHdrPartials] = next_slot;
    w[kHdrCombine] = (int32_t)n_comb;
    w[kHdrClusterOff] = (int32_t)cl_off;
    w[kHdrItemsOff] = (int32_t)it_off;
    w[kHdrCombineOff] = (int32_t)cb_off;
    w[kHdrTotalPages] = (int32_t)total;
    w[kHdrMaxSplits] = max_splits;
    w[kHdrTimeoutLo] = (int32_t)(uint32_t)(timeout_ns & 0xffffffffu);
    w[kHdrTimeoutHi] = (int32_t)(uint32_t)((uint64_t)timeout_ns >> 32);
    w[kHdrQueriesPerSeq] = qps;
    for (int64_t k = 0; k <= C; ++k) w[cl_off + k] = cluster_begin[k];
    std::memcpy(w + it_off, items.data(), (size_t)n_items * sizeof(PlanItem));
    if (n_comb) std::memcpy(w + cb_off, combine.data(), (size_t)n_comb * sizeof(PlanCombine));

    info->batch = batch;
    info->num_clusters = (int32_t)C;
    info->num_items = (int32_t)n_items;
    info->num_partials = next_slot;
    info->num_combine = (int32_t)n_comb;
    info->max_splits = max_splits;
    info->total_pages = (int32_t)total;
    info->queries_per_seq = qps;
    info->plan_bytes = words * 4;
    info->workspace_bytes = (int64_t)next_slot * (kPartialOBytes + kPartialLseBytes);
    info->wait_timeout_ns = timeout_ns;
    return MLA_OK;
}
