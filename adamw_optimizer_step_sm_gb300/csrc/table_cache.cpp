// table_cache.cpp -- adamw_step_table: one optimizer step over a tensor table
// that the caller already holds in device memory.  The table is copied to
// the host, and the plan built for it is kept in a small cache keyed by the
// table's bytes, the mode and the device, so a training loop that passes the
// same device table every step builds its plan once.  Built on the public
// entry points (adamw_plan_create / adamw_step).
#include <cuda_runtime_api.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "adamw_internal.h"

namespace {

struct CachedPlan {
    int device;
    int32_t mode;
    std::vector<adamw_tensor_t> table;
    adamw_plan_t plan;
    uint64_t last_use;
};

constexpr size_t kMaxCachedPlans = 8;

std::mutex g_cache_mu;
std::vector<CachedPlan> g_cache;
uint64_t g_clock = 0;

bool same_table(const std::vector<adamw_tensor_t>& a, const std::vector<adamw_tensor_t>& b) {
    return a.size() == b.size() &&
           (a.empty() || std::memcmp(a.data(), b.data(), a.size() * sizeof(adamw_tensor_t)) == 0);
}

}  // namespace

extern "C" int adamw_step_table(const adamw_tensor_t* d_table, int32_t n_tensors, int32_t mode,
                                const adamw_hparams_t* hp, int64_t step, double* d_grad_norm,
                                int32_t* d_nonfinite, adamw_stream_t stream) {
    if (n_tensors < 0 || (n_tensors > 0 && !d_table) || !hp) return ADAMW_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        adamw::set_cuda_error("cudaGetDevice", cudaGetErrorString(cudaGetLastError()));
        return ADAMW_ERR_CUDA;
    }
    std::vector<adamw_tensor_t> table(static_cast<size_t>(n_tensors));
    if (n_tensors > 0) {
        cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
        if (cudaMemcpyAsync(table.data(), d_table, sizeof(adamw_tensor_t) * table.size(),
                            cudaMemcpyDeviceToHost, st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess) {
            adamw::set_cuda_error("reading the device table", cudaGetErrorString(cudaGetLastError()));
            return ADAMW_ERR_CUDA;
        }
    }
    std::lock_guard<std::mutex> lk(g_cache_mu);
    CachedPlan* hit = nullptr;
    for (CachedPlan& c : g_cache)
        if (c.device == dev && c.mode == mode && same_table(c.table, table)) hit = &c;
    if (!hit) {
        adamw_plan_t plan = nullptr;
        int rc = adamw_plan_create(table.data(), n_tensors, mode, ADAMW_PLAN_NORM, &plan);
        if (rc != ADAMW_OK) return rc;
        if (g_cache.size() >= kMaxCachedPlans) {
            size_t lru = 0;
            for (size_t i = 1; i < g_cache.size(); ++i)
                if (g_cache[i].last_use < g_cache[lru].last_use) lru = i;
            adamw_plan_destroy(g_cache[lru].plan);
            g_cache.erase(g_cache.begin() + long(lru));
        }
        g_cache.push_back({dev, mode, std::move(table), plan, 0});
        hit = &g_cache.back();
    }
    hit->last_use = ++g_clock;
    return adamw_step(hit->plan, hp, step, d_grad_norm, d_nonfinite, stream);
}

extern "C" int adamw_step_table_cache_clear(void) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    int n = int(g_cache.size());
    for (CachedPlan& c : g_cache) adamw_plan_destroy(c.plan);
    g_cache.clear();
    return n;
}
