// Host-only probe of the launch planner in sdv_plan.h (no GPU, no kernel):
// for each input line "rows nvec resident_warps max_items row_slots K G" it
// prints "chunks chunk_vec row_mode merge_lanes" as the library would plan
// them.  Built and run by tests/test_plan_host.py.
#include <cstdio>
#include <cinttypes>

#include "../draft_verification_sdv_gb300/csrc/sdv_plan.h"

int main() {
    long long rows, nvec, warps, max_items, slots;
    int K, G;
    while (std::scanf("%lld %lld %lld %lld %lld %d %d", &rows, &nvec, &warps, &max_items, &slots, &K,
                      &G) == 7) {
        int chunks = 0;
        int64_t chunk_vec = 0;
        const bool row_mode = sdv::plan_row_mode(rows, slots, nvec);
        if (row_mode) {
            chunks = 1;
            chunk_vec = nvec;
        } else {
            sdv::plan_rowpass_chunks(rows, nvec, warps, max_items, &chunks, &chunk_vec);
        }
        std::printf("%d %" PRId64 " %d %d\n", chunks, chunk_vec, row_mode ? 1 : 0,
                    sdv::select_merge_lanes(K, G, chunks));
    }
    return 0;
}
