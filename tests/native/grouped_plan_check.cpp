// Prints the row-group split softmax's launch plan (grouped_plan.h) for the
// shapes given on standard input, one "M nvec num_sms block per_sm ring_bytes
// min_buffers slots_per_row" line each, as "n slot_vecs nbuf grid".
#include <cstdio>

#include "grouped_plan.h"

int main() {
    long long M, nvec, ring, slots;
    int sms, block, per_sm, minbuf;
    while (std::scanf("%lld %lld %d %d %d %lld %d %lld", &M, &nvec, &sms, &block, &per_sm, &ring, &minbuf, &slots) == 8) {
        const rowops::GroupedLimits lim{block, per_sm, rowops::kGroupedMaxVpt, rowops::kGroupedMaxSlots,
                                        rowops::kGroupedMaxBuffers, ring};
        const rowops::GroupedPlan p = rowops::grouped_plan(M, nvec, sms, minbuf, slots, lim);
        std::printf("%d %lld %d %lld\n", p.n, static_cast<long long>(p.slot_vecs), p.nbuf,
                    static_cast<long long>(p.grid));
    }
    return 0;
}
