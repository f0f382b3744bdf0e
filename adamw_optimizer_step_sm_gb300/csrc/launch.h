// launch.h -- the plan object and the per-storage-mode launchers.
//
// Each storage mode's update kernels are instantiated in a translation unit of
// their own (update_m<MODE>.cu, all from update_mode.inc), so the modes
// compile in parallel; adamw_sm.cu reaches them through the table
// of launchers that mode_ops<MODE>() returns.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "adamw_internal.h"
#include "adamw_sm.h"

// One partition of the plan's list on the device: the chunk descriptors of
// `grid` CTAs and where each CTA's run of chunks begins.
struct DevPartition {
    int32_t grid = 0;
    int64_t n_chunks = 0;
    adamw::ChunkPtr* chunks = nullptr;
    int32_t* cta_begin = nullptr;
    adamw::DynTail dyn = {0, 0, nullptr};   // claimable chunks (update partition only)
};

struct adamw_plan {
    int device = 0;
    int32_t mode = 0;
    int variant = 0;  // index of the mode's kernels in adamw::kVariantModes
    int32_t flags = 0;
    int32_t n_tensors = 0;
    int64_t total = 0;
    int64_t scalar_elems = 0;
    void* block = nullptr;  // one device allocation holding everything below
    adamw::TensorDev* tensors = nullptr;  // the uploaded tensor table
    DevPartition upd;                     // update kernel
    DevPartition nrm;                     // norm partial kernel (its own grid)
    double* partial = nullptr;
    int32_t* flag = nullptr;
    adamw::NormOut* norm = nullptr;
    adamw::StepRecord* rec = nullptr;  // device-resident step path
    int32_t* status = nullptr;         // set by a kernel whose bounded wait ran out
    bool fused = false;                // clipped steps run as one cooperative launch
    unsigned long long* arrivals = nullptr;  // grid-barrier counter of the fused kernel
    // the update partition's claim-and-arrival word (kSyncClaim ...)
    unsigned long long* sync = nullptr;
    adamw::ScalarMemo* memo = nullptr;  // two slots, see ScalarMemo
};

namespace adamw {

// Every kernel of the library is launched with programmatic stream
// serialization (programmatic dependent launch): it may begin while the
// kernel before it in the stream finishes, and waits (griddepcontrol.wait)
// before it touches memory that kernel may write.  This hides the launch gap
// between back-to-back steps.  ADAMW_PDL=0 at build time launches plainly.
#ifndef ADAMW_PDL
#define ADAMW_PDL 1
#endif

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), int grid, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(unsigned(kBlock));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ADAMW_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The launchers of one storage mode.  Every pointer is set.
struct ModeOps {
    // Resident CTAs per SM of the update kernel for each Kind (occ[Kind]) and
    // of the fused clipped kernel.  Also sets any kernel attribute a launch
    // needs, so it runs once per device before the first plan.
    cudaError_t (*occupancy)(int occ[3], int* occ_fused);
    // The update over the plan's partition.  dev: the scalars come from the
    // plan's device-side step record (written by the step prologue) instead
    // of `s`.  `report` receives the non-finite flag when kind == kReport.
    cudaError_t (*update)(const adamw_plan* P, int kind, bool dev, const StepScalars& s,
                          int32_t* report, cudaStream_t st);
    // The one-launch device-resident step (no norm): kind is kPlain or
    // kReport (then user_flag receives the non-finite flag).
    cudaError_t (*self)(const adamw_plan* P, int kind, const adamw_hparams_t* d_hp,
                        int64_t* d_step, int32_t* user_flag, cudaStream_t st);
    // The fused clipped step: norm, grid barrier and update in one
    // cooperative launch over the update grid.
    cudaError_t (*fused)(const adamw_plan* P, const StepScalars& s, double* user_norm,
                         int32_t* user_flag, cudaStream_t st);
};

// mode_ops<MODE>() is defined in update_m<MODE>.cu.
template <int MODE>
const ModeOps& mode_ops();
template <> const ModeOps& mode_ops<0>();
template <> const ModeOps& mode_ops<1>();
template <> const ModeOps& mode_ops<2>();
template <> const ModeOps& mode_ops<3>();
template <> const ModeOps& mode_ops<4>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 1>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 3>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 4>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 5>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 6>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 7>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 9>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 10>();
template <> const ModeOps& mode_ops<ADAMW_MODE_ANYPREC | 11>();

}  // namespace adamw
