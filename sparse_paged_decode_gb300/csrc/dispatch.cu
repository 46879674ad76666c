// dispatch.cu -- picks the kernel for each call.
#include <atomic>

#include "spd_dispatch.h"

namespace spd {

namespace {
std::atomic<uint64_t> g_launches{0};
}

void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }
uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

cudaError_t dispatch_score(const ScoreArgs &a, cudaStream_t stream) {
    count_launches(1);
    return launch_score_generic(a, stream);
}

cudaError_t dispatch_select(const SelectArgs &a, cudaStream_t stream) {
    count_launches(1);
    return launch_select_generic(a, stream);
}

cudaError_t dispatch_attention(const AttnArgs &a, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    count_launches(1);
    return launch_attention_generic(a, stream);
}

size_t workspace_bytes(int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t NB) {
    // split-K partials: one fp32 row of D values plus (max, sum) per q head
    // and split, for up to 2*T*Hq + 16384 rows; plus the work plan.
    const size_t rows = static_cast<size_t>(2 * T * Hq + 16384);
    const size_t partials = rows * static_cast<size_t>(D + 2) * sizeof(float);
    const size_t plan = static_cast<size_t>(T * Hkv + 1) * static_cast<size_t>(NB + 16) * sizeof(int32_t) + 65536;
    return (partials + plan + 255) / 256 * 256;
}

}  // namespace spd
