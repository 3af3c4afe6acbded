// expert_parallel.cu -- index arithmetic of expert parallelism: G ranks, each
// owning a contiguous range of the experts, exchange token rows after the
// grouping step and the experts' outputs before the combine.
//
// The pages list expert parallelism as not done ("Phase 19: MoE --
// gpt-oss-20b", section 6); the split builds on the grouping of "Engine"
// (cherenkov), section "Prefill" (tokens grouped by expert, gathered,
// projected, scattered back):
//   - every rank routes its own tokens and groups its (token, slot) pairs by
//     expert (a stable counting sort: the MOE_INTER_PERM order).  Rank g owns
//     experts [first[g], first[g+1]), so that order is already grouped by
//     owning rank: rows [offsets[first[g]], offsets[first[g+1]]) go to rank g.
//   - a receiver gets, from each source rank in rank order, that source's rows
//     of each local expert in expert order.  Its own grouping is expert-major:
//     for each local expert, the rows of source 0, then source 1, ... in each
//     source's order.
//   - the outputs travel back in arrival order, so each source receives them
//     in its own expert order and scatters them to (token, slot) through its
//     permutation; the fixed slot-order combine follows.
// Everything here is integer work on the host, deterministic.
#include "moe_internal.cuh"

namespace {

moe_status ep_fail(const char *msg)
{
    moe::set_last_error(msg);
    return MOE_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

moe_status moe_ep_send_plan(int32_t n_expert, int32_t n_ranks, const int32_t *first_expert, const int32_t *counts,
                            int32_t *send_counts, int32_t *send_displs)
{
    moe::set_last_error("");
    if (n_expert <= 0 || n_ranks <= 0 || !first_expert || !counts || !send_counts || !send_displs)
        return ep_fail("sizes must be positive and pointers non-NULL");
    if (first_expert[0] != 0 || first_expert[n_ranks] != n_expert) return ep_fail("ranges must cover 0 .. n_expert");
    // every bound checked before any count is read: ascending from 0 to n_expert
    for (int g = 0; g < n_ranks; ++g)
        if (first_expert[g + 1] < first_expert[g]) return ep_fail("expert ranges must be ascending");
    int64_t displ = 0;
    for (int g = 0; g < n_ranks; ++g) {
        int64_t c = 0;
        for (int e = first_expert[g]; e < first_expert[g + 1]; ++e) {
            if (counts[e] < 0) return ep_fail("negative count");
            c += counts[e];
        }
        if (displ + c > INT32_MAX) return ep_fail("too many rows");
        send_counts[g] = (int32_t)c;
        send_displs[g] = (int32_t)displ;
        displ += c;
    }
    return MOE_OK;
}

moe_status moe_ep_recv_plan(int32_t n_ranks, int32_t n_local, const int32_t *counts_from, int32_t *recv_counts,
                            int32_t *recv_displs, int32_t *order, int32_t *group_offsets)
{
    moe::set_last_error("");
    if (n_ranks <= 0 || n_local < 0 || !counts_from || !recv_counts || !recv_displs || !group_offsets)
        return ep_fail("sizes must be positive and pointers non-NULL");
    // arrival order: source-major; within a source, its rows expert by expert
    int64_t total = 0;
    for (int g = 0; g < n_ranks; ++g) {
        int64_t c = 0;
        for (int e = 0; e < n_local; ++e) {
            const int32_t v = counts_from[(int64_t)g * n_local + e];
            if (v < 0) return ep_fail("negative count");
            c += v;
        }
        if (total + c > INT32_MAX) return ep_fail("too many rows");
        recv_counts[g] = (int32_t)c;
        recv_displs[g] = (int32_t)total;
        total += c;
    }
    if (total > 0 && !order) return ep_fail("order must be non-NULL when rows arrive");
    // local expert-major order: expert e, then source g, then the source's order
    int64_t pos = 0;
    for (int e = 0; e < n_local; ++e) {
        group_offsets[e] = (int32_t)pos;
        for (int g = 0; g < n_ranks; ++g) {
            int64_t start = recv_displs[g];  // where source g's rows of expert e arrived
            for (int e2 = 0; e2 < e; ++e2) start += counts_from[(int64_t)g * n_local + e2];
            const int32_t c = counts_from[(int64_t)g * n_local + e];
            for (int32_t i = 0; i < c; ++i) order[pos++] = (int32_t)(start + i);
        }
    }
    group_offsets[n_local] = (int32_t)pos;
    return MOE_OK;
}

}  // extern "C"
