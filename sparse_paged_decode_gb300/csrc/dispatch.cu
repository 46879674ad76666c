// dispatch.cu -- picks the kernel for each call.
#include <stddef.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "plan.cuh"
#include "sdpa.cuh"
#include "spd_dispatch.h"

namespace spd {

namespace {
std::atomic<uint64_t> g_launches{0};
}

void count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }
uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

namespace {
std::mutex g_dev_mu;
std::map<int, int> g_sms;                              // device -> SM count
std::map<std::pair<int, const void *>, int> g_smem;    // (device, kernel) -> bytes opted in
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) return it->second;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    g_sms[dev] = sms;
    return sms;
}

cudaError_t opt_in_smem(const void *func, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    int &have = g_smem[std::make_pair(dev, func)];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

cudaError_t launch_score_tc(const ScoreArgs &a, cudaStream_t stream, bool *used);
cudaError_t launch_attention_tc(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream, bool *used);
cudaError_t launch_attention_bf16_tc(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream, bool *used);
cudaError_t launch_attention_e4m3_rows(const AttnArgs &a, void *ws, size_t ws_bytes, cudaStream_t stream,
                                       bool *used);
cudaError_t launch_sdpa_tc(const SdpaArgs &a, cudaStream_t stream, bool *used);

namespace {
// per stage (index = spd stage code): 0 fastest kernel the shapes allow,
// 1 the general-layout kernel, 2 (selection only) the rank kernel
thread_local int g_policy[5] = {0, 0, 0, 0, 0};
}

int set_kernel_policy(int stage, int policy) {
    if (stage < 1 || stage > 4) return -1;
    const int old = g_policy[stage];
    g_policy[stage] = policy;
    return old;
}

cudaError_t dispatch_score(const ScoreArgs &a, cudaStream_t stream) {
    count_launches(1);
    bool used = false;
    if (g_policy[1] == 0) {
        cudaError_t e = launch_score_tc(a, stream, &used);
        if (e != cudaSuccess || used) return e;
    }
    return launch_score_generic(a, stream);
}

cudaError_t dispatch_select(const SelectArgs &a, cudaStream_t stream) {
    count_launches(1);
    if (g_policy[2] == 0) return launch_select_fast(a, stream);
    if (g_policy[2] == 2) return launch_select_rank(a, stream);
    return launch_select_generic(a, stream);
}

cudaError_t dispatch_attention(const AttnArgs &a, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    bool used = false;
    cudaError_t e = cudaSuccess;
    // policy 0: the tensor-core kernel of the cache type; 1: the general
    // kernel; for an E4M3 cache, 2: the keys-on-lanes kernel only, 3: the
    // query-rows kernel only.  By default an E4M3 cache takes the query-rows
    // kernel when a request's rows fill wide groups -- on average at least
    // 48 query rows (tokens x q heads of one kv head) per request -- and the
    // keys-on-lanes kernel otherwise: the first one's time per page does not
    // grow with the group's width up to 128 rows, the second one's does, and
    // it is the faster of the two for narrow groups.
    const int pol = g_policy[3];
    if (pol == 0 && a.kv_dt == SPD_BF16) {
        e = launch_attention_bf16_tc(a, workspace, workspace_bytes, stream, &used);
    } else if (a.kv_dt == SPD_E4M3 && (pol == 0 || pol == 2 || pol == 3)) {
        const int64_t G = a.Hkv > 0 ? a.Hq / a.Hkv : 0;
        const bool wide = static_cast<int64_t>(a.T) * G >= 48LL * a.R;
        if (pol == 3 || (pol == 0 && wide)) e = launch_attention_e4m3_rows(a, workspace, workspace_bytes, stream, &used);
        if (e == cudaSuccess && !used && pol != 3) e = launch_attention_tc(a, workspace, workspace_bytes, stream, &used);
    }
    if (e != cudaSuccess) return e;
    if (used) {
        count_launches(3);  // list and unit planner kernels + attention
        return cudaSuccess;
    }
    count_launches(1);
    return launch_attention_generic(a, stream);
}

cudaError_t dispatch_sdpa(const SdpaArgs &a, cudaStream_t stream) {
    count_launches(1);
    if (g_policy[4] == 0) {
        bool used = false;
        cudaError_t e = launch_sdpa_tc(a, stream, &used);
        if (e != cudaSuccess || used) return e;
    }
    return launch_sdpa(a, stream);
}

int workspace_status(const void *workspace, cudaStream_t stream) {
    if (workspace == nullptr) return -1;
    int32_t status = 0;
    if (cudaMemcpyAsync(&status, static_cast<const char *>(workspace) + offsetof(PlanHeader, status), sizeof status,
                        cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return -1;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return -1;
    return status;
}

size_t workspace_bytes(int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t NB) {
    // the work plan (groups, per-pair block lists, units) and the split-K
    // partials of the tensor-core path; see plan.cuh
    return PlanLayout(T, Hq, Hkv, D, NB).total;
}

}  // namespace spd
