// adamw_sm.cu -- the C ABI: plans, the step entry points, the norm pass and
// its finalize, the device-resident step's prologue, the on-device learning
// rate schedule, the copy probe and the allocation-free norm entry.  The
// update kernels of each storage mode live in update_m<MODE>.cu and are
// reached through mode_ops<MODE>() (launch.h).
//
// The step is a streaming elementwise update: per element it reads p, g, m, v
// and c (bf16 Kahan mode, 10 B), master, m, v and g (mixed mode, 14 B) or p,
// remainder, m, v and g (remainder mode, 14 B) and writes 8, 14 or 12 B back,
// with about twenty fp32 operations in between.
// That is far below the GPU's ridge point, so HBM bandwidth bounds it and the
// kernels are built to keep DRAM streaming: a persistent grid (SMs x resident
// CTAs) dealt tiles of about 8K elements of the flattened parameter space,
// cut on 2048-element boundaries, round-robin (so the grid sweeps every
// buffer together), chunk descriptors prefetched one ahead, 16-byte vector
// loads issued U vectors ahead of the arithmetic (U per storage mode), fp32
// math, 16-byte stores.  No tensor cores: nothing here is a contraction.
//
// Sources of the method: "[pure bf16 training] w/ AnyPrecisionAdamW and Kahan
// summation" (transformers PR #21312), "Train from scratch" recipe (bf16
// momentum / variance / compensation, Kahan summation, betas 0.9/0.95, weight
// decay 0.1) and "Theoretical memory allocation" (10 vs 16 B/param);
// "Distributed optimizer support for BERT" (NeMo PR #5305), "Usage"
// (distributed_fused_adam: the fp32-state per-shard update).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "adamw_internal.h"
#include "device_common.cuh"
#include "launch.h"

using namespace adamw;

namespace {

// kNormCtas CTAs per SM (four: 64 registers), the occupancy the norm's grid
// is sized by.
__global__ void __launch_bounds__(kBlock, kNormCtas)
norm_partial_kernel(const ChunkPtr* __restrict__ chunks,
                    const int32_t* __restrict__ cta_begin,
                    double* __restrict__ partial, int32_t* __restrict__ flag) {
    const int32_t c0 = cta_begin[blockIdx.x], c1 = cta_begin[blockIdx.x + 1];
    pdl_trigger();
    pdl_wait();
    norm_partial_cta(chunks, c0, c1, partial, flag);
}

// Stage 2: fixed-order fp64 sum of the partials, norm, clip coefficient.
__global__ void __launch_bounds__(kBlock)
norm_finalize_kernel(const double* __restrict__ partial, const int32_t* __restrict__ flag,
                     int32_t n, float max_grad_norm, NormOut* __restrict__ out,
                     double* __restrict__ user_norm, int32_t* __restrict__ user_flag) {
    pdl_trigger();
    pdl_wait();
    double x = 0.0;
    bool bad = false;
    for (int32_t i = threadIdx.x; i < n; i += kBlock) {
        x += __ldcg(partial + i);
        bad |= __ldcg(flag + i) != 0;
    }
    const double tot = block_sum(x);
    const int any = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        const double norm = sqrt(tot);
        double coef = 1.0;
        if (max_grad_norm > 0.0f) {
            coef = double(max_grad_norm) / (norm + 1e-6);
            if (coef > 1.0) coef = 1.0;
        }
        out->norm = norm;
        out->coef = float(coef);
        out->nonfinite = any;
        if (user_norm) *user_norm = norm;
        if (user_flag) *user_flag = any;
    }
}

// One CTA, before the update: finalises the norm when n_partials > 0 (the
// same fixed-order reduction as norm_finalize_kernel), reads the
// hyperparameters and the applied-step counter from device memory, decides
// whether the step is skipped, takes the scalars from the plan's memo or
// computes them (warps 0 and 1, one half each), writes the StepRecord,
// advances the counter for an applied step, and fills the caller's outputs
// (flag -1 for invalid hyperparameters).
__global__ void __launch_bounds__(kBlock)
step_prologue_kernel(const adamw_hparams_t* __restrict__ d_hp, int64_t* __restrict__ d_step,
                     StepRecord* __restrict__ rec, const double* __restrict__ partial,
                     const int32_t* __restrict__ flag, int32_t n_partials, int32_t clip,
                     NormOut* __restrict__ nout, double* __restrict__ user_norm,
                     int32_t* __restrict__ user_flag, const ScalarMemo* __restrict__ memo) {
    __shared__ StepScalars s_sh;
    __shared__ adamw_hparams_t hp_sh;
    __shared__ int skip_sh, hit_sh, any_sh;
    __shared__ int64_t t_sh;
    __shared__ double norm_sh;
    __shared__ float coef_sh;
    pdl_trigger();
    pdl_wait();
    double x = 0.0;
    bool bad = false;
    for (int32_t i = threadIdx.x; i < n_partials; i += kBlock) {
        x += __ldcg(partial + i);
        bad |= __ldcg(flag + i) != 0;
    }
    const double tot = block_sum(x);
    const int any = __syncthreads_or(bad);
    adamw_hparams_t hp;
    int64_t t = 0;
    StepScalars s;
    bool hit = false;
    if (threadIdx.x < 32) hit = memo_fetch_warp(d_hp, d_step, memo, &hp, &t, &s);
    if (threadIdx.x == 0) {
        const bool valid = hparams_valid_dev(hp);
        const double norm = sqrt(tot);
        float coef = 1.0f;
        if (clip && valid && hp.max_grad_norm > 0.0f) {
            double c = double(hp.max_grad_norm) / (norm + 1e-6);
            if (c > 1.0) c = 1.0;
            coef = float(c);
        }
        const int skip = !valid ? 2 : (clip && any) ? 1 : 0;
        hit_sh = skip ? 1 : hit;
        if (!skip && hit) s_sh = s;
        hp_sh = hp;
        skip_sh = skip;
        t_sh = t;
        norm_sh = norm;
        coef_sh = coef;
        any_sh = any;
    }
    __syncthreads();
    if (!hit_sh) make_scalars_cta(hp_sh, t_sh, &s_sh);
    if (threadIdx.x == 0) {
        StepRecord r{};
        r.skip = skip_sh;
        r.coef = coef_sh;
        if (!r.skip) {
            r.s = s_sh;
            r.hp = hp_sh;
            r.t = t_sh;
            *d_step = t_sh;
        }
        *rec = r;
        if (n_partials > 0) {
            nout->norm = norm_sh;
            nout->coef = coef_sh;
            nout->nonfinite = any_sh;
            if (user_norm) *user_norm = norm_sh;
        }
        if (user_flag) *user_flag = skip_sh == 2 ? -1 : (n_partials > 0 ? any_sh : 0);
    }
}

// The linear warm-up / linear decay schedule on the device: d_hp->lr for the
// update t = *d_step + 1, with the host function's fp64 operations.
__global__ void lr_linear_warmup_kernel(adamw_hparams_t* __restrict__ d_hp,
                                        const int64_t* __restrict__ d_step, float base_lr,
                                        int64_t warmup, int64_t total) {
    if (threadIdx.x != 0) return;
    pdl_trigger();
    pdl_wait();
    const int64_t k = __ldcg(d_step);  // applied updates before this one
    double f;
    if (k < warmup) {
        f = __ddiv_rn(double(k), double(warmup > 1 ? warmup : 1));
    } else {
        const double span = double((total - warmup) > 1 ? (total - warmup) : 1);
        f = __ddiv_rn(double(total - k), span);
        if (f < 0.0) f = 0.0;
    }
    d_hp->lr = __double2float_rn(__dmul_rn(double(base_lr), f));
}

// Plain 16-byte streaming copy (HBM ceiling probe).
__global__ void __launch_bounds__(kBlock)
copy_probe_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n) {
    constexpr int U = 4;
    const int64_t stride = int64_t(gridDim.x) * kBlock;
    for (int64_t base = int64_t(blockIdx.x) * kBlock + threadIdx.x; base < n; base += stride * U) {
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * stride < n) r[u] = ld16(src + base + u * stride);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (base + u * stride < n) st16(dst + base + u * stride, r[u]);
    }
}

// ------------------------------------------------------------ host side ----

struct DeviceInfo {
    int sms = 0;
    int occ[kModes][3] = {};
    int occ_norm = 0;
    int occ_copy = 0;
    int occ_fused[kModes] = {};
    int cooperative = 0;
};

std::mutex g_dev_mu;
std::vector<DeviceInfo> g_dev;

bool cuda_ok(cudaError_t e, const char* where) {
    if (e == cudaSuccess) return true;
    set_cuda_error(where, cudaGetErrorString(e));
    return false;
}

// The launchers of a kernel variant (an index into kVariantModes).
const ModeOps& ops(int variant) {
    switch (variant) {
        case 0: return mode_ops<kVariantModes[0]>();
        case 1: return mode_ops<kVariantModes[1]>();
        case 2: return mode_ops<kVariantModes[2]>();
        case 3: return mode_ops<kVariantModes[3]>();
        case 4: return mode_ops<kVariantModes[4]>();
        case 5: return mode_ops<kVariantModes[5]>();
        case 6: return mode_ops<kVariantModes[6]>();
        case 7: return mode_ops<kVariantModes[7]>();
        case 8: return mode_ops<kVariantModes[8]>();
        case 9: return mode_ops<kVariantModes[9]>();
        case 10: return mode_ops<kVariantModes[10]>();
        case 11: return mode_ops<kVariantModes[11]>();
        case 12: return mode_ops<kVariantModes[12]>();
        default: return mode_ops<kVariantModes[13]>();
    }
}
static_assert(kModes == 14, "ops() lists every kernel variant");

int device_info(int dev, DeviceInfo* out) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev >= int(g_dev.size())) g_dev.resize(dev + 1);
    DeviceInfo& d = g_dev[dev];
    if (d.sms == 0) {
        int sms = 0;
        if (!cuda_ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                     "cudaDeviceGetAttribute"))
            return ADAMW_ERR_CUDA;
        for (int m = 0; m < kModes; ++m)
            if (!cuda_ok(ops(m).occupancy(d.occ[m], &d.occ_fused[m]), "occupancy"))
                return ADAMW_ERR_CUDA;
        if (!cuda_ok(cudaDeviceGetAttribute(&d.cooperative, cudaDevAttrCooperativeLaunch, dev),
                     "cudaDeviceGetAttribute"))
            return ADAMW_ERR_CUDA;
        if (!cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                         &d.occ_norm, norm_partial_kernel, kBlock, 0), "occupancy") ||
            !cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                         &d.occ_copy, copy_probe_kernel, kBlock, 0), "occupancy"))
            return ADAMW_ERR_CUDA;
        d.sms = sms;
    }
    *out = d;
    return ADAMW_OK;
}

// Makes the plan's device current for the scope, restoring the caller's.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

cudaError_t launch_norm(const adamw_plan* P, float max_grad_norm, double* user_norm,
                        int32_t* user_flag, cudaStream_t st) {
    cudaError_t e = launch_kernel(norm_partial_kernel, P->nrm.grid, st, P->nrm.chunks,
                                  P->nrm.cta_begin, P->partial, P->flag);
    if (e != cudaSuccess) return e;
    return launch_kernel(norm_finalize_kernel, 1, st, P->partial, P->flag, P->nrm.grid,
                         max_grad_norm, P->norm, user_norm, user_flag);
}

}  // namespace

extern "C" int adamw_plan_create(const adamw_tensor_t* host_table, int32_t n_tensors,
                                 int32_t mode, int32_t flags, adamw_plan_t* out) {
    if (!out) return ADAMW_ERR_INVALID_ARG;
    *out = nullptr;
    if (flags & ~(ADAMW_PLAN_NORM | ADAMW_PLAN_NO_FUSE)) return ADAMW_ERR_INVALID_ARG;
    int rc = validate_table(host_table, n_tensors, mode);
    if (rc != ADAMW_OK) return rc;

    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice")) return ADAMW_ERR_CUDA;
    rc = check_device_access(host_table, n_tensors, mode, dev);
    if (rc != ADAMW_OK) return rc;
    DeviceInfo di;
    rc = device_info(dev, &di);
    if (rc != ADAMW_OK) return rc;

    const int var = mode_variant(mode);
    int occ = di.occ[var][kPlain];
    for (int k = 0; k < 3; ++k) occ = occ < di.occ[var][k] ? occ : di.occ[var][k];
    if (occ < 1) occ = 1;
    int occ_norm = di.occ_norm > 0 ? di.occ_norm : 1;
    if (occ_norm > kNormCtas) occ_norm = kNormCtas;

    int64_t total = 0;
    for (int32_t k = 0; k < n_tensors; ++k) total += host_table[k].numel;
    // Lists whose gradients are at most kFusedMaxGradBytes run clipped steps
    // as one fused cooperative launch (measured faster up to that size).
    const bool fused = (flags & ADAMW_PLAN_NORM) && !(flags & ADAMW_PLAN_NO_FUSE) &&
                       di.cooperative && di.occ_fused[var] > 0 &&
                       total * 2 <= kFusedMaxGradBytes;
    if (fused) occ = occ < di.occ_fused[var] ? occ : di.occ_fused[var];
    const int32_t grid = choose_grid(total, di.sms * occ);
    // the fused kernel's norm pass uses the update grid; plans without it
    // give the norm pass its own, larger grid
    const int32_t grid_norm = !(flags & ADAMW_PLAN_NORM) ? 0
                              : fused ? grid : choose_grid(total, di.sms * occ_norm);

    Partition part, part_norm;
    std::vector<ChunkPtr> cp, cp_norm;
    if (grid > 0) {
        rc = build_partition(host_table, n_tensors, mode, grid, update_tile_elems(total, grid),
                             &part);
        if (rc != ADAMW_OK) return rc;
        chunk_pointers(host_table, mode, part, &cp);
    }
    if (grid_norm > 0) {
        // contiguous ranges (measured faster for the norm pass than the
        // update's round-robin tiles: 56.9 against 62.9 us on OPT-125m)
        rc = build_partition(host_table, n_tensors, mode, grid_norm, 0, &part_norm, 0);
        if (rc != ADAMW_OK) return rc;
        chunk_pointers(host_table, mode, part_norm, &cp_norm);
    }

    adamw_plan* P = new adamw_plan();
    P->device = dev;
    P->mode = mode;
    P->variant = var;
    P->flags = flags;
    P->n_tensors = n_tensors;
    P->total = total;
    P->scalar_elems = part.scalar_elems;
    P->upd.grid = grid;
    P->upd.n_chunks = int64_t(cp.size());
    P->nrm.grid = grid_norm;
    P->nrm.n_chunks = int64_t(cp_norm.size());

    // Layout of the single allocation.
    size_t off = 0;
    const size_t o_t = off; off = align_up(off + sizeof(TensorDev) * size_t(n_tensors), 256);
    const size_t o_c = off; off = align_up(off + sizeof(ChunkPtr) * cp.size(), 256);
    const size_t o_b = off; off = align_up(off + sizeof(int32_t) * (size_t(grid) + 1), 256);
    const size_t o_cn = off; off = align_up(off + sizeof(ChunkPtr) * cp_norm.size(), 256);
    const size_t o_bn = off; off = align_up(off + sizeof(int32_t) * (size_t(grid_norm) + 1), 256);
    const size_t o_p = off; off = align_up(off + sizeof(double) * size_t(grid_norm), 256);
    const size_t o_f = off; off = align_up(off + sizeof(int32_t) * size_t(grid_norm), 256);
    const size_t o_n = off; off = align_up(off + sizeof(NormOut), 256);
    const size_t o_r = off; off = align_up(off + sizeof(StepRecord), 256);
    const size_t o_s = off; off = align_up(off + sizeof(int32_t), 256);
    const size_t o_a = off; off = align_up(off + sizeof(unsigned long long), 256);
    const size_t o_d = off; off = align_up(off + sizeof(unsigned long long), 256);
    const size_t o_m = off; off = align_up(off + 2 * sizeof(ScalarMemo) + sizeof(PowTable), 256);

    if (!cuda_ok(cudaMalloc(&P->block, off), "cudaMalloc")) {
        delete P;
        return ADAMW_ERR_CUDA;
    }
    char* b = static_cast<char*>(P->block);
    P->tensors = reinterpret_cast<TensorDev*>(b + o_t);
    P->upd.chunks = reinterpret_cast<ChunkPtr*>(b + o_c);
    P->upd.cta_begin = reinterpret_cast<int32_t*>(b + o_b);
    P->nrm.chunks = reinterpret_cast<ChunkPtr*>(b + o_cn);
    P->nrm.cta_begin = reinterpret_cast<int32_t*>(b + o_bn);
    P->partial = reinterpret_cast<double*>(b + o_p);
    P->flag = reinterpret_cast<int32_t*>(b + o_f);
    P->norm = reinterpret_cast<NormOut*>(b + o_n);
    P->rec = reinterpret_cast<StepRecord*>(b + o_r);
    P->status = reinterpret_cast<int32_t*>(b + o_s);
    P->arrivals = reinterpret_cast<unsigned long long*>(b + o_a);
    P->sync = reinterpret_cast<unsigned long long*>(b + o_d);
    P->upd.dyn = DynTail{grid > 0 ? part.cta_begin[size_t(grid)] : 0, int32_t(part.n_dyn), P->sync};
    P->memo = reinterpret_cast<ScalarMemo*>(b + o_m);
    P->fused = fused;
#if ADAMW_CHECK_BOUNDS
    for (ChunkPtr& c : cp) c.status = P->status;
    for (ChunkPtr& c : cp_norm) c.status = P->status;
#endif

    auto up = [&](void* dst, const void* src, size_t bytes, const char* what) {
        return bytes == 0 || cuda_ok(cudaMemcpy(dst, src, bytes, cudaMemcpyHostToDevice), what);
    };
    bool ok = cuda_ok(cudaMemset(P->block, 0, off), "cudaMemset");
    ok = ok && up(P->tensors, host_table, sizeof(TensorDev) * size_t(n_tensors), "cudaMemcpy(table)");
    ok = ok && up(P->upd.chunks, cp.data(), sizeof(ChunkPtr) * cp.size(), "cudaMemcpy(chunks)");
    ok = ok && (grid == 0 || up(P->upd.cta_begin, part.cta_begin.data(),
                                sizeof(int32_t) * (size_t(grid) + 1), "cudaMemcpy(cta_begin)"));
    ok = ok && up(P->nrm.chunks, cp_norm.data(), sizeof(ChunkPtr) * cp_norm.size(),
                  "cudaMemcpy(norm chunks)");
    ok = ok && (grid_norm == 0 || up(P->nrm.cta_begin, part_norm.cta_begin.data(),
                                     sizeof(int32_t) * (size_t(grid_norm) + 1),
                                     "cudaMemcpy(norm cta_begin)"));
    if (!ok) {
        cudaFree(P->block);
        delete P;
        return ADAMW_ERR_CUDA;
    }
    *out = P;
    return ADAMW_OK;
}

extern "C" int adamw_step(adamw_plan_t plan, const adamw_hparams_t* hp, int64_t step,
                          double* d_grad_norm, int32_t* d_nonfinite, adamw_stream_t stream) {
    if (!plan) return ADAMW_ERR_INVALID_ARG;
    StepScalars s;
    int rc = make_scalars(hp, step, &s);
    if (rc != ADAMW_OK) return rc;
    const bool clip = hp->max_grad_norm > 0.0f;
    // A clipped step can be skipped; without the flag the caller could not
    // tell, would advance t past a step that wrote nothing, and every later
    // bias correction would be off by one step.
    if (clip && !d_nonfinite) return ADAMW_ERR_INVALID_ARG;
    const bool need_norm = clip || d_grad_norm != nullptr;
    if (need_norm && !(plan->flags & ADAMW_PLAN_NORM)) return ADAMW_ERR_NO_NORM;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    DeviceGuard guard(plan->device);
    if (!guard.ok) {
        set_cuda_error("cudaSetDevice", cudaGetErrorString(cudaGetLastError()));
        return ADAMW_ERR_CUDA;
    }

    if (plan->upd.grid == 0) {  // empty list: nothing to update, norm is 0
        if (d_grad_norm && !cuda_ok(cudaMemsetAsync(d_grad_norm, 0, sizeof(double), st), "memset"))
            return ADAMW_ERR_CUDA;
        if (d_nonfinite && !cuda_ok(cudaMemsetAsync(d_nonfinite, 0, sizeof(int32_t), st), "memset"))
            return ADAMW_ERR_CUDA;
        return ADAMW_OK;
    }

    if (clip && plan->fused) {
        if (!cuda_ok(ops(plan->variant).fused(plan, s, d_grad_norm, d_nonfinite, st), "fused launch"))
            return ADAMW_ERR_CUDA;
        return ADAMW_OK;
    }
    int kind = kPlain;
    int32_t* report = nullptr;
    if (need_norm) {
        if (!cuda_ok(launch_norm(plan, clip ? hp->max_grad_norm : 0.0f, d_grad_norm, d_nonfinite, st),
                     "norm launch"))
            return ADAMW_ERR_CUDA;
        kind = clip ? kClip : kPlain;
    } else if (d_nonfinite) {
        if (!cuda_ok(cudaMemsetAsync(d_nonfinite, 0, sizeof(int32_t), st), "cudaMemsetAsync"))
            return ADAMW_ERR_CUDA;
        kind = kReport;
        report = d_nonfinite;
    }
    if (!cuda_ok(ops(plan->variant).update(plan, kind, false, s, report, st), "update launch"))
        return ADAMW_ERR_CUDA;
    return ADAMW_OK;
}

extern "C" int adamw_grad_norm(adamw_plan_t plan, double* d_grad_norm, int32_t* d_nonfinite,
                               adamw_stream_t stream) {
    if (!plan) return ADAMW_ERR_INVALID_ARG;
    if (!(plan->flags & ADAMW_PLAN_NORM)) return ADAMW_ERR_NO_NORM;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    DeviceGuard guard(plan->device);
    if (!guard.ok) {
        set_cuda_error("cudaSetDevice", cudaGetErrorString(cudaGetLastError()));
        return ADAMW_ERR_CUDA;
    }
    if (plan->nrm.grid == 0) {
        if (d_grad_norm && !cuda_ok(cudaMemsetAsync(d_grad_norm, 0, sizeof(double), st), "memset"))
            return ADAMW_ERR_CUDA;
        if (d_nonfinite && !cuda_ok(cudaMemsetAsync(d_nonfinite, 0, sizeof(int32_t), st), "memset"))
            return ADAMW_ERR_CUDA;
        return ADAMW_OK;
    }
    if (!cuda_ok(launch_norm(plan, 0.0f, d_grad_norm, d_nonfinite, st), "norm launch"))
        return ADAMW_ERR_CUDA;
    return ADAMW_OK;
}

extern "C" int adamw_step_device(adamw_plan_t plan, const adamw_hparams_t* d_hp,
                                 int64_t* d_step, int32_t flags, double* d_grad_norm,
                                 int32_t* d_nonfinite, adamw_stream_t stream) {
    if (!plan || !d_hp || !d_step || (flags & ~(ADAMW_STEP_CLIP | ADAMW_STEP_NORM)))
        return ADAMW_ERR_INVALID_ARG;
    const bool clip = (flags & ADAMW_STEP_CLIP) != 0;
    const bool want_norm = clip || (flags & ADAMW_STEP_NORM) || d_grad_norm != nullptr;
    if (want_norm && !(plan->flags & ADAMW_PLAN_NORM)) return ADAMW_ERR_NO_NORM;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    DeviceGuard guard(plan->device);
    if (!guard.ok) {
        set_cuda_error("cudaSetDevice", cudaGetErrorString(cudaGetLastError()));
        return ADAMW_ERR_CUDA;
    }
    if (!want_norm && plan->upd.grid > 0) {
        // one launch: every CTA computes the scalars, the last one advances
        // the counter
        const cudaError_t e = ops(plan->variant).self(plan, d_nonfinite ? kReport : kPlain, d_hp,
                                                   d_step, d_nonfinite, st);
        return cuda_ok(e, "update launch") ? ADAMW_OK : ADAMW_ERR_CUDA;
    }
    const bool norm_pass = want_norm && plan->nrm.grid > 0;
    if (norm_pass &&
        !cuda_ok(launch_kernel(norm_partial_kernel, plan->nrm.grid, st, plan->nrm.chunks,
                               plan->nrm.cta_begin, plan->partial, plan->flag), "norm launch"))
        return ADAMW_ERR_CUDA;
    if (!cuda_ok(launch_kernel(step_prologue_kernel, 1, st, d_hp, d_step, plan->rec, plan->partial,
                               plan->flag, norm_pass ? plan->nrm.grid : 0, clip ? 1 : 0, plan->norm,
                               d_grad_norm, d_nonfinite, plan->memo),
                 "prologue launch"))
        return ADAMW_ERR_CUDA;
    if (want_norm && !norm_pass && d_grad_norm &&
        !cuda_ok(cudaMemsetAsync(d_grad_norm, 0, sizeof(double), st), "memset"))
        return ADAMW_ERR_CUDA;
    if (plan->upd.grid == 0) return ADAMW_OK;
    const int kind = clip ? kClip : (!want_norm && d_nonfinite) ? kReport : kPlain;
    int32_t* report = (kind == kReport) ? d_nonfinite : nullptr;
    if (!cuda_ok(ops(plan->variant).update(plan, kind, true, StepScalars{}, report, st), "update launch"))
        return ADAMW_ERR_CUDA;
    return ADAMW_OK;
}

extern "C" int adamw_lr_linear_warmup_device(adamw_hparams_t* d_hp, const int64_t* d_step,
                                             float base_lr, int64_t warmup, int64_t total,
                                             adamw_stream_t stream) {
    if (!d_hp || !d_step || warmup < 0 || total < 0 || !std::isfinite(base_lr))
        return ADAMW_ERR_INVALID_ARG;
    // one thread of a kBlock launch does the work
    return cuda_ok(launch_kernel(lr_linear_warmup_kernel, 1, reinterpret_cast<cudaStream_t>(stream),
                                 d_hp, d_step, base_lr, warmup, total),
                   "schedule launch") ? ADAMW_OK : ADAMW_ERR_CUDA;
}

extern "C" int adamw_plan_device_status(adamw_plan_t plan, int32_t* out) {
    if (!plan || !out) return ADAMW_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return ADAMW_ERR_CUDA;
    if (!cuda_ok(cudaDeviceSynchronize(), "cudaDeviceSynchronize") ||
        !cuda_ok(cudaMemcpy(out, plan->status, sizeof(int32_t), cudaMemcpyDeviceToHost),
                 "cudaMemcpy(status)"))
        return ADAMW_ERR_CUDA;
    if (*out != 0) {
        // a wait ran out: clear the word, realign the fused-step barrier
        // counter and zero the claim-and-arrival word, which a launch that
        // gave up may have left part-counted (no kernel of the plan is
        // running after the synchronise)
        const int32_t zero = 0;
        const unsigned long long start = 0;
        if (!cuda_ok(cudaMemcpy(plan->status, &zero, sizeof(int32_t), cudaMemcpyHostToDevice),
                     "cudaMemcpy(status)") ||
            !cuda_ok(cudaMemcpy(plan->arrivals, &start, sizeof(start), cudaMemcpyHostToDevice),
                     "cudaMemcpy(arrivals)") ||
            !cuda_ok(cudaMemcpy(plan->sync, &start, sizeof(start), cudaMemcpyHostToDevice),
                     "cudaMemcpy(sync)"))
            return ADAMW_ERR_CUDA;
    }
    return ADAMW_OK;
}

extern "C" int adamw_plan_test_skew_barrier(adamw_plan_t plan, int64_t delta) {
    if (!plan) return ADAMW_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return ADAMW_ERR_CUDA;
    unsigned long long v = 0;
    if (!cuda_ok(cudaDeviceSynchronize(), "cudaDeviceSynchronize") ||
        !cuda_ok(cudaMemcpy(&v, plan->arrivals, sizeof(v), cudaMemcpyDeviceToHost),
                 "cudaMemcpy(arrivals)"))
        return ADAMW_ERR_CUDA;
    v += static_cast<unsigned long long>(delta);
    return cuda_ok(cudaMemcpy(plan->arrivals, &v, sizeof(v), cudaMemcpyHostToDevice),
                   "cudaMemcpy(arrivals)") ? ADAMW_OK : ADAMW_ERR_CUDA;
}

extern "C" int32_t adamw_build_flags(void) {
    return (ADAMW_CHECK_BOUNDS ? ADAMW_BUILD_CHECK_BOUNDS : 0) |
           (ADAMW_BULK ? ADAMW_BUILD_BULK_STAGING : 0);
}

extern "C" int adamw_plan_test_corrupt_chunk(adamw_plan_t plan, int64_t chunk, int64_t delta) {
    // Only a bounds-checked build may run a chunk that lies: there the
    // kernels refuse it before touching memory.
    if (!ADAMW_CHECK_BOUNDS || !plan || chunk < 0 || chunk >= plan->upd.n_chunks)
        return ADAMW_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return ADAMW_ERR_CUDA;
    int64_t len2 = 0;
    int64_t* at = &plan->upd.chunks[chunk].len2;
    if (!cuda_ok(cudaDeviceSynchronize(), "cudaDeviceSynchronize") ||
        !cuda_ok(cudaMemcpy(&len2, at, sizeof(len2), cudaMemcpyDeviceToHost), "cudaMemcpy(chunk)"))
        return ADAMW_ERR_CUDA;
    len2 += 2 * delta;
    return cuda_ok(cudaMemcpy(at, &len2, sizeof(len2), cudaMemcpyHostToDevice), "cudaMemcpy(chunk)")
               ? ADAMW_OK : ADAMW_ERR_CUDA;
}

extern "C" int adamw_plan_destroy(adamw_plan_t plan) {
    if (!plan) return ADAMW_OK;
    int rc = ADAMW_OK;
    {
        DeviceGuard guard(plan->device);
        if (plan->block) {
            if (!cuda_ok(cudaDeviceSynchronize(), "cudaDeviceSynchronize")) rc = ADAMW_ERR_CUDA;
            if (!cuda_ok(cudaFree(plan->block), "cudaFree")) rc = ADAMW_ERR_CUDA;
        }
    }
    delete plan;
    return rc;
}

extern "C" int adamw_plan_get_info(adamw_plan_t plan, adamw_plan_info_t* out) {
    if (!plan || !out) return ADAMW_ERR_INVALID_ARG;
    out->mode = plan->mode;
    out->n_tensors = plan->n_tensors;
    out->total_elems = plan->total;
    out->grid = plan->upd.grid;
    out->block = kBlock;
    out->n_chunks = plan->upd.n_chunks;
    out->norm_grid = plan->nrm.grid;
    out->fused = plan->fused ? 1 : 0;
    out->scalar_elems = plan->scalar_elems;
    out->device = plan->device;
    out->has_norm = (plan->flags & ADAMW_PLAN_NORM) ? 1 : 0;
    return ADAMW_OK;
}

extern "C" int adamw_copy_probe(void* dst, const void* src, int64_t bytes, adamw_stream_t stream) {
    if (bytes < 0 || (bytes > 0 && (!dst || !src))) return ADAMW_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) % 16 || bytes % 16)
        return ADAMW_ERR_MISALIGNED;
    if (bytes == 0) return ADAMW_OK;
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice")) return ADAMW_ERR_CUDA;
    DeviceInfo di;
    int rc = device_info(dev, &di);
    if (rc != ADAMW_OK) return rc;
    const int64_t n = bytes / 16;
    int64_t grid = int64_t(di.sms) * (di.occ_copy > 0 ? di.occ_copy : 1);
    const int64_t need = (n + kBlock - 1) / kBlock;
    if (grid > need) grid = need;
    copy_probe_kernel<<<int(grid), kBlock, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4*>(dst), static_cast<const uint4*>(src), n);
    return cuda_ok(cudaGetLastError(), "copy launch") ? ADAMW_OK : ADAMW_ERR_CUDA;
}

// ------------------------------------------- global norm without allocation --
//
// adamw_grad_norm_noalloc is adamw_grad_norm for callers that cannot allocate
// device memory.  Instead of a plan's cudaMalloc'd workspace it uses one
// file-scope __device__ array (the tensor list, the per-CTA partials and
// flags, and the finalize record), so a call allocates nothing.  Every GPU
// that loads this library holds the array until the process exits.  The
// list reaches the device as kernel launch parameters, which the runtime
// copies when the launch is made, so the caller's table is not read after
// the call returns.

namespace {

// One tensor of the no-alloc list on the device.
struct NoAllocEntry {
    const uint16_t* grad;
    int64_t numel;
};

constexpr int kNoAllocMaxCtas = 1024;
constexpr size_t kNoAllocTableOff = 0;
constexpr size_t kNoAllocPartialOff =
    (sizeof(NoAllocEntry) * ADAMW_NOALLOC_MAX_TENSORS + 255) / 256 * 256;
constexpr size_t kNoAllocFlagOff = kNoAllocPartialOff + sizeof(double) * kNoAllocMaxCtas;
constexpr size_t kNoAllocOutOff = kNoAllocFlagOff + sizeof(int32_t) * kNoAllocMaxCtas;
constexpr size_t kNoAllocBytes = (kNoAllocOutOff + sizeof(NormOut) + 255) / 256 * 256;

// The scratch (about 76 KiB).  Host code never uses this name as an address:
// on the host it is only a stand-in; noalloc_device() asks the runtime for the
// device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
    bool ready = false;
    unsigned char* base = nullptr;  // device address of g_noalloc_scratch
    int grid = 0;
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Up to CAP entries of the list, passed by value as the parameters of one
// launch (the large form is just under the 32 KiB parameter limit).
template <int CAP>
struct NoAllocPiece {
    int32_t first, count;
    const uint16_t* grad[CAP];
    int64_t numel[CAP];
};
constexpr int kNoAllocSmallPiece = 128;
constexpr int kNoAllocLargePiece = 2000;
static_assert(sizeof(NoAllocPiece<kNoAllocLargePiece>) <= 32764, "launch parameter limit");

// Writes one piece of the list into the scratch's table.
template <int CAP>
__global__ void __launch_bounds__(kBlock)
noalloc_table_kernel(const __grid_constant__ NoAllocPiece<CAP> piece, NoAllocEntry* __restrict__ table) {
    pdl_trigger();
    pdl_wait();
    for (int32_t i = threadIdx.x; i < piece.count; i += kBlock)
        table[piece.first + i] = NoAllocEntry{piece.grad[i], piece.numel[i]};
}

template <int CAP>
cudaError_t upload_noalloc_piece(const adamw_tensor_t* host_table, int32_t first, int32_t count,
                                 NoAllocEntry* table, cudaStream_t st) {
    NoAllocPiece<CAP> piece;
    piece.first = first;
    piece.count = count;
    for (int32_t i = 0; i < count; ++i) {
        piece.grad[i] = static_cast<const uint16_t*>(host_table[first + i].grad);
        piece.numel[i] = host_table[first + i].numel;
    }
    return launch_kernel(noalloc_table_kernel<CAP>, 1, st, piece, table);
}

// Stage 1 without a chunk table: tensor by tensor in list order, every thread
// of the grid takes a fixed share of each tensor (an element of the head that
// 16-byte aligns g, vectors strided by the whole grid, an element of the
// tail).  Sums as in norm_partial_kernel: error-free fp32 groups of exact
// squares, an fp64 recomputation for threads whose groups leave the safe range.
__global__ void __launch_bounds__(kBlock)
norm_partial_noalloc_kernel(const NoAllocEntry* __restrict__ table, int32_t n,
                            double* __restrict__ partial, int32_t* __restrict__ flag) {
    pdl_trigger();
    pdl_wait();
    const int64_t gt = int64_t(blockIdx.x) * kBlock + threadIdx.x;
    const int64_t T = int64_t(gridDim.x) * kBlock;
    constexpr int U = 4;

    auto walk = [&](auto vec, auto elem, auto after_iter) {
        for (int32_t k = 0; k < n; ++k) {
            const uint16_t* g = reinterpret_cast<const uint16_t*>(
                __ldcg(reinterpret_cast<const unsigned long long*>(&table[k].grad)));
            const int64_t len = __ldcg(&table[k].numel);
            if (len <= 0) continue;
            int64_t h = int64_t((16 - (reinterpret_cast<uintptr_t>(g) & 15)) & 15) >> 1;
            if (h > len) h = len;
            if (gt < h) elem(g[gt]);
            const uint16_t* gv = g + h;
            const int64_t nvec = (len - h) / kVec;
            for (int64_t base = gt; base < nvec; base += T * U) {
                uint4 w[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (base + u * T < nvec) w[u] = ld16(gv + (base + u * T) * kVec);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (base + u * T < nvec) vec(w[u]);
                after_iter();
            }
            const int64_t t0 = h + nvec * kVec;
            if (gt < len - t0) elem(g[t0 + gt]);
        }
    };

    Sum2F32x2 grp;
    double acc = 0.0;
    float err = 0.0f;
    bool in_range = true;
    uint32_t nz = 0;
    auto add_word = [&](uint32_t w) {
        const uint64_t x = bf16x2_to_f2(w);
        grp.add(f2_mul(x, x));
    };
    walk(
        [&](const uint4& w) {
            nz |= (w.x | w.y | w.z | w.w) & 0x7fff7fffu;
            add_word(w.x);
            add_word(w.y);
            add_word(w.z);
            add_word(w.w);
        },
        [&](uint16_t hb) {
            nz |= hb & 0x7fffu;
            add_word(hb);   // the high lane adds an exact zero
            in_range &= grp.flush(acc, err);
        },
        [&]() { in_range &= grp.flush(acc, err); });
    in_range &= grp.flush(acc, err);
    double tot = acc + double(err);
    bool bad = false;
    if (!in_range || (nz != 0 && tot < 0x1p-100)) {
        double exact = 0.0;
        walk(
            [&](const uint4& w) {
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const double lo = bf16_lo(ws[j]), hi = bf16_hi(ws[j]);
                    bad |= !isfinite(lo) || !isfinite(hi);
                    exact += lo * lo;
                    exact += hi * hi;
                }
            },
            [&](uint16_t hb) {
                const double x = from_bf16(hb);
                bad |= !isfinite(x);
                exact += x * x;
            },
            [&]() {});
        tot = exact;
    }
    tot = block_sum(tot);
    const int any = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        partial[blockIdx.x] = tot;
        flag[blockIdx.x] = any;
    }
}

// Set-up, once per device, with that device current: the scratch's device
// address and the grid size.
int noalloc_device(int dev, NoAllocDevice* out) {
    if (dev < 0 || dev >= kNoAllocMaxDevices) return ADAMW_ERR_TOO_LARGE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice& d = g_noalloc_dev[dev];
    if (!d.ready) {
        void* ptr = nullptr;
        if (!cuda_ok(cudaGetSymbolAddress(&ptr, g_noalloc_scratch), "cudaGetSymbolAddress"))
            return ADAMW_ERR_CUDA;
        int sms = 0, occ = 0;
        if (!cuda_ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                     "cudaDeviceGetAttribute") ||
            !cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                         &occ, norm_partial_noalloc_kernel, kBlock, 0), "occupancy"))
            return ADAMW_ERR_CUDA;
        const int grid = sms * (occ > 0 ? occ : 1);
        d.base = static_cast<unsigned char*>(ptr);
        d.grid = grid < kNoAllocMaxCtas ? grid : kNoAllocMaxCtas;
        d.ready = true;
    }
    *out = d;
    return ADAMW_OK;
}

}  // namespace

extern "C" int adamw_grad_norm_noalloc(const adamw_tensor_t* host_table, int32_t n_tensors,
                                       double* d_grad_norm, int32_t* d_nonfinite,
                                       adamw_stream_t stream) {
    if (n_tensors < 0 || (n_tensors > 0 && !host_table)) return ADAMW_ERR_INVALID_ARG;
    if (n_tensors > ADAMW_NOALLOC_MAX_TENSORS) return ADAMW_ERR_TOO_LARGE;
    for (int32_t k = 0; k < n_tensors; ++k) {
        const adamw_tensor_t& t = host_table[k];
        if (t.numel < 0 || (t.numel > 0 && !t.grad)) return ADAMW_ERR_INVALID_ARG;
        if (t.numel > 0 && (reinterpret_cast<uintptr_t>(t.grad) & 1)) return ADAMW_ERR_MISALIGNED;
    }
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice")) return ADAMW_ERR_CUDA;
    NoAllocDevice d;
    int rc = noalloc_device(dev, &d);
    if (rc != ADAMW_OK) return rc;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    NoAllocEntry* table = reinterpret_cast<NoAllocEntry*>(d.base + kNoAllocTableOff);
    double* partial = reinterpret_cast<double*>(d.base + kNoAllocPartialOff);
    int32_t* flag = reinterpret_cast<int32_t*>(d.base + kNoAllocFlagOff);
    NormOut* out = reinterpret_cast<NormOut*>(d.base + kNoAllocOutOff);
    // Every CTA writes its partial and flag and the finalize writes the
    // record on every call, so nothing in the scratch has to start at zero.
    // The list goes in the launch parameters of one or more small kernels
    // (copied by the runtime when each launch is made).
    for (int32_t first = 0; first < n_tensors;) {
        const int32_t left = n_tensors - first;
        const cudaError_t e =
            left <= kNoAllocSmallPiece
                ? upload_noalloc_piece<kNoAllocSmallPiece>(host_table, first, left, table, st)
                : upload_noalloc_piece<kNoAllocLargePiece>(
                      host_table, first, left < kNoAllocLargePiece ? left : kNoAllocLargePiece,
                      table, st);
        if (!cuda_ok(e, "table launch")) return ADAMW_ERR_CUDA;
        first += left <= kNoAllocSmallPiece ? left
                 : (left < kNoAllocLargePiece ? left : kNoAllocLargePiece);
    }
    if (!cuda_ok(launch_kernel(norm_partial_noalloc_kernel, d.grid, st,
                               static_cast<const NoAllocEntry*>(table), n_tensors, partial, flag),
                 "norm launch"))
        return ADAMW_ERR_CUDA;
    if (!cuda_ok(launch_kernel(norm_finalize_kernel, 1, st, static_cast<const double*>(partial),
                               static_cast<const int32_t*>(flag), d.grid, 0.0f, out, d_grad_norm,
                               d_nonfinite),
                 "finalize launch"))
        return ADAMW_ERR_CUDA;
    return ADAMW_OK;
}
