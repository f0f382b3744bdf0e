// kernels.cuh -- the update kernels, instantiated once per storage mode by
// update_mode.inc: the update itself (host-computed or prologue-computed
// scalars), the one-launch device-resident step, the fused clipped step, and
// (behind ADAMW_BULK) the cp.async.bulk staged variant of mode A.
#pragma once

#include "device_common.cuh"

namespace {

// DEV: the scalars, clip coefficient and skip decision come from the
// StepRecord the device-resident step path's prologue wrote; CTA 0 also
// computes the next step's scalars into the memo.
template <int MODE, int K, bool DEV>
__global__ void ADAMW_UPDATE_BOUNDS(MODE)
adamw_update_kernel(const ChunkPtr* __restrict__ chunks,
                    const int32_t* __restrict__ cta_begin, StepScalars s,
                    const NormOut* __restrict__ norm, int32_t* __restrict__ report,
                    const StepRecord* __restrict__ rec, ScalarMemo* __restrict__ memo,
                    DynTail dyn) {
    // the chunk table is written once, when the plan is made: read the first
    // descriptor before waiting for the kernel this one may overlap
    const int32_t c0 = cta_begin[blockIdx.x], c1 = cta_begin[blockIdx.x + 1];
    ChunkPtr cur;
    if (c0 < c1) cur = load_chunk(chunks + c0);
    pdl_trigger();
    pdl_wait();
    float coef = 1.0f;
    if constexpr (DEV) {
        if (__ldcg(&rec->skip)) return;   // skipped step: no writes at all
        s = rec->s;
        coef = rec->coef;
        if (blockIdx.x == 0) {
            __shared__ adamw_hparams_t hp_sh;
            __shared__ int64_t t_sh;
            if (threadIdx.x == 0) {
                hp_sh = rec->hp;
                t_sh = rec->t;
            }
            __syncthreads();
            memo_next(memo, hp_sh, t_sh);
        }
    } else if (K == kClip) {
        if (__ldcg(&norm->nonfinite)) return;  // skipped step: no writes at all
        coef = norm->coef;
    }
    bool bad = false;
    update_cta_from<MODE, K>(chunks, c0, c1, cur, s, coef, bad, dyn);
    if (dyn.n > 0 && threadIdx.x == 0) sync_arrive(dyn.sync, false, gridDim.x);
    if (K == kReport) {
        if (__syncthreads_or(bad) && threadIdx.x == 0) *report = 1;
    }
}

// ---- device-resident step without a norm pass: one launch ----
//
// Thread 0 of every CTA reads the hyperparameters and the step counter and
// looks up the scalars of t = *d_step + 1 in the plan's two-slot memo; on a
// miss warps 0 and 1 compute them (the host planner's fp64 operations, two
// independent halves at once).  CTA 0, whose share of the list is short by
// about that much work, first computes the scalars of t + 1 into the memo
// while the others stream (so a run of steps with unchanged
// hyperparameters computes each step's scalars off the critical path); the
// last CTA to finish -- found with an arrival
// counter in the plan's claim-and-arrival word, which also counts the CTAs
// that saw a non-finite gradient, one atomic per CTA -- advances the counter
// and writes the non-finite flag, so no CTA can read a counter that was
// already advanced (each CTA's read of it has returned before its arrival
// is counted).  The kernel's end publishes the last CTA's writes and the
// memo.  Invalid hyperparameters: nothing is updated, the flag is -1.
template <int MODE, int K>
__global__ void ADAMW_SELF_BOUNDS(MODE)
adamw_update_self_kernel(const ChunkPtr* __restrict__ chunks, const int32_t* __restrict__ cta_begin,
                         const adamw_hparams_t* __restrict__ d_hp, int64_t* __restrict__ d_step,
                         int32_t* __restrict__ user_flag, ScalarMemo* __restrict__ memo,
                         DynTail dyn) {
    __shared__ StepScalars s_sh;
    __shared__ adamw_hparams_t hp_sh;
    __shared__ int valid_sh, hit_sh;
    __shared__ int64_t t_sh;
    __shared__ unsigned long long ticket_sh;
    const int32_t c0 = cta_begin[blockIdx.x], c1 = cta_begin[blockIdx.x + 1];
    ChunkPtr cur;
    if (c0 < c1) cur = load_chunk(chunks + c0);
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x < 32) {
        adamw_hparams_t hp;
        int64_t t;
        StepScalars s;
        const bool hit = memo_fetch_warp(d_hp, d_step, memo, &hp, &t, &s);
        if (threadIdx.x == 0) {
            const int valid = hparams_valid_dev(hp);
            hit_sh = valid && hit;
            if (valid && hit) s_sh = s;
            hp_sh = hp;
            valid_sh = valid;
            t_sh = t;
        }
    }
    __syncthreads();
    if (valid_sh && !hit_sh) make_scalars_cta(hp_sh, t_sh, &s_sh);
    if (blockIdx.x == 0 && valid_sh) memo_next(memo, hp_sh, t_sh);
    bool bad = false;
    if (valid_sh) update_cta_from<MODE, K>(chunks, c0, c1, cur, s_sh, 1.0f, bad, dyn);
    const int any = (K == kReport) ? __syncthreads_or(bad) : 0;
    if (threadIdx.x == 0) ticket_sh = sync_arrive(dyn.sync, any != 0, gridDim.x);
    __syncthreads();
    const unsigned long long ticket = ticket_sh;   // the word with this CTA's arrival
    const unsigned int arrived = unsigned((ticket & kSyncArriveMask) / kSyncArrive) - 1u;
    if (threadIdx.x == 0 && arrived == gridDim.x - 1) {  // the last CTA (it zeroed the word)
        if (valid_sh) *d_step = t_sh;
        if (user_flag) *user_flag = valid_sh ? int32_t(ticket >= kSyncFlagged) : -1;
    }
}

template <int MODE>
__global__ void ADAMW_FUSED_BOUNDS(MODE)
adamw_fused_clip_kernel(const ChunkPtr* __restrict__ upd_chunks,
                        const int32_t* __restrict__ upd_begin,
                        const ChunkPtr* __restrict__ nrm_chunks,
                        const int32_t* __restrict__ nrm_begin, StepScalars s,
                        double* __restrict__ partial, int32_t* __restrict__ flag,
                        NormOut* __restrict__ nout, double* __restrict__ user_norm,
                        int32_t* __restrict__ user_flag, unsigned long long* __restrict__ arrivals,
                        int32_t* __restrict__ status, DynTail dyn) {
    __shared__ int passed;
    // the chunk tables are written once, when the plan is made
    const int32_t n0 = nrm_begin[blockIdx.x], n1 = nrm_begin[blockIdx.x + 1];
    ChunkPtr first;
    if (n0 < n1) first = load_chunk(nrm_chunks + n0);
    pdl_trigger();
    pdl_wait();
    norm_partial_cta<kFusedKeepG>(nrm_chunks, n0, n1, partial, flag, n0 < n1 ? &first : nullptr);
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned long long ticket = atomicAdd(arrivals, 1ull);
        const unsigned long long target = (ticket / gridDim.x + 1) * gridDim.x;
        int ok = 0;
        for (uint32_t i = 0; i < kBarrierSpins; ++i) {
            if (load_acquire_u64(arrivals) >= target) {
                ok = 1;
                break;
            }
            __nanosleep(kBarrierSleepNs);
        }
        if (!ok) atomicOr(status, 1);
        passed = ok;
    }
    __syncthreads();
    if (!passed) return;
    // every CTA: the same fixed-order sum as norm_finalize_kernel
    double x = 0.0;
    bool bad = false;
    for (int32_t i = threadIdx.x; i < int32_t(gridDim.x); i += kBlock) {
        x += __ldcg(partial + i);
        bad |= __ldcg(flag + i) != 0;
    }
    const double tot = block_sum(x);
    const int any = __syncthreads_or(bad);
    __shared__ float coef_sh;
    if (threadIdx.x == 0) {
        const double norm = sqrt(tot);
        double coef = double(s.max_grad_norm) / (norm + 1e-6);
        if (coef > 1.0) coef = 1.0;
        coef_sh = float(coef);
        if (blockIdx.x == 0) {
            nout->norm = norm;
            nout->coef = float(coef);
            nout->nonfinite = any;
            if (user_norm) *user_norm = norm;
            if (user_flag) *user_flag = any;
        }
    }
    __syncthreads();
    if (any) return;  // skipped step: no writes
    bool unused = false;
    update_cta<MODE, kClip>(upd_chunks, upd_begin[blockIdx.x], upd_begin[blockIdx.x + 1], s,
                            coef_sh, unused, dyn);
    if (dyn.n > 0 && threadIdx.x == 0) sync_arrive(dyn.sync, false, gridDim.x);
}

// ------------------------------------------- bulk-copy staged update (A) --
//
// Mode A with the five input streams of each stage brought into shared
// memory by cp.async.bulk (one 1-D bulk copy per stream, completion counted
// on an mbarrier) instead of by per-thread 16-byte loads.  Thread 0 issues
// stage j + NS while the CTA computes stage j from shared memory; results
// go straight to global memory with 16-byte stores.  Every mbarrier wait is
// bounded: a wait that does not complete sets *err and the CTA returns.
#if ADAMW_BULK
static_assert(!ADAMW_CHECK_BOUNDS, "the bulk-copy variant has no bounds-checked build");
#ifndef ADAMW_BULK_STAGES
#define ADAMW_BULK_STAGES 2
#endif
#ifndef ADAMW_BULK_ELEMS
#define ADAMW_BULK_ELEMS 4096
#endif
constexpr int kBulkStages = ADAMW_BULK_STAGES;
constexpr int kBulkElems = ADAMW_BULK_ELEMS;  // per stage, multiple of kBlock * kVec
constexpr uint32_t kBulkStreamBytes = kBulkElems * 2;
constexpr size_t kBulkSmem = size_t(kBulkStages) * 5 * kBulkStreamBytes;
static_assert(kBulkElems % (kBlock * kVec) == 0, "a stage is whole vectors of the block");
constexpr uint32_t kWaitLimit = 1u << 20;  // try_wait rounds (about a second) before giving up

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with the given parity; false after kWaitLimit rounds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

struct BulkJob {
    uint16_t* p;
    const uint16_t* g;
    uint16_t* m;
    uint16_t* v;
    uint16_t* c;
    int32_t n;  // elements, a multiple of kVec
};

template <int K>
__global__ void __launch_bounds__(kBlock)
adamw_update_bulk_kernel(const ChunkPtr* __restrict__ chunks, const int32_t* __restrict__ cta_begin,
                         StepScalars s, const NormOut* __restrict__ norm,
                         int32_t* __restrict__ report, int32_t* __restrict__ err) {
    extern __shared__ __align__(128) unsigned char stage_buf[];
    __shared__ __align__(8) uint64_t bar[kBulkStages];
    __shared__ BulkJob job[kBulkStages];
    __shared__ int32_t njobs_sh;

    float coef = 1.0f;
    if (K == kClip) {
        if (norm->nonfinite) return;
        coef = norm->coef;
    }
    const int32_t c0 = cta_begin[blockIdx.x], c1 = cta_begin[blockIdx.x + 1];
    auto buf = [&](int slot, int stream) {
        return reinterpret_cast<uint16_t*>(stage_buf + (size_t(slot) * 5 + stream) * kBulkStreamBytes);
    };

    // producer state (thread 0 only): next chunk and element offset to issue
    int32_t pci = c0;
    int64_t poff = 0;
    auto issue = [&](int slot) {
        while (pci < c1) {
            const ChunkPtr ch = load_chunk(chunks + pci);
            const int64_t len8 = (ch.len2 & 1) ? ((ch.len2 >> 1) / kVec * kVec) : 0;
            if (poff < len8) {
                const int32_t n = int32_t(len8 - poff < kBulkElems ? len8 - poff : kBulkElems);
                BulkJob& jb = job[slot];
                jb.p = static_cast<uint16_t*>(ch.p) + poff;
                jb.g = static_cast<const uint16_t*>(ch.g) + poff;
                jb.m = static_cast<uint16_t*>(ch.m) + poff;
                jb.v = static_cast<uint16_t*>(ch.v) + poff;
                jb.c = static_cast<uint16_t*>(ch.a) + poff;
                jb.n = n;
                const uint32_t bytes = uint32_t(n) * 2;
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                mbar_arrive_expect_tx(&bar[slot], 5 * bytes);
                bulk_load(buf(slot, 0), jb.p, bytes, &bar[slot]);
                bulk_load(buf(slot, 1), jb.g, bytes, &bar[slot]);
                bulk_load(buf(slot, 2), jb.m, bytes, &bar[slot]);
                bulk_load(buf(slot, 3), jb.v, bytes, &bar[slot]);
                bulk_load(buf(slot, 4), jb.c, bytes, &bar[slot]);
                poff += n;
                return;
            }
            ++pci;
            poff = 0;
        }
    };

    if (threadIdx.x == 0) {
        int32_t nj = 0;
        for (int32_t ci = c0; ci < c1; ++ci) {
            const ChunkPtr ch = load_chunk(chunks + ci);
            const int64_t len8 = (ch.len2 & 1) ? ((ch.len2 >> 1) / kVec * kVec) : 0;
            nj += int32_t((len8 + kBulkElems - 1) / kBulkElems);
        }
        njobs_sh = nj;
        for (int i = 0; i < kBulkStages; ++i) mbar_init(&bar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (int i = 0; i < kBulkStages && i < nj; ++i) issue(i);
    }
    __syncthreads();
    const int32_t njobs = njobs_sh;
    bool bad = false;
    int32_t j = 0;
    for (; j < njobs; ++j) {
        const int slot = j % kBulkStages;
        const bool ok = mbar_wait_bounded(&bar[slot], uint32_t(j / kBulkStages) & 1u);
        if (__syncthreads_or(!ok)) break;
        const BulkJob jb = job[slot];
        const int32_t nvec = jb.n / kVec;
#pragma unroll
        for (int u = 0; u < kBulkElems / (kBlock * kVec); ++u) {
            const int32_t i = u * kBlock + threadIdx.x;
            if (i < nvec) {
                uint4 P = *reinterpret_cast<const uint4*>(buf(slot, 0) + i * kVec);
                const uint4 G = *reinterpret_cast<const uint4*>(buf(slot, 1) + i * kVec);
                uint4 M = *reinterpret_cast<const uint4*>(buf(slot, 2) + i * kVec);
                uint4 V = *reinterpret_cast<const uint4*>(buf(slot, 3) + i * kVec);
                uint4 C = *reinterpret_cast<const uint4*>(buf(slot, 4) + i * kVec);
                if (K == kReport)
                    bad |= bf16x2_nonfinite(G.x) | bf16x2_nonfinite(G.y) | bf16x2_nonfinite(G.z) |
                           bf16x2_nonfinite(G.w);
                kahan_x2<K>(s, coef, G.x, P.x, M.x, V.x, C.x);
                kahan_x2<K>(s, coef, G.y, P.y, M.y, V.y, C.y);
                kahan_x2<K>(s, coef, G.z, P.z, M.z, V.z, C.z);
                kahan_x2<K>(s, coef, G.w, P.w, M.w, V.w, C.w);
                st16(jb.p + i * kVec, P);
                st16(jb.m + i * kVec, M);
                st16(jb.v + i * kVec, V);
                st16(jb.c + i * kVec, C);
            }
        }
        __syncthreads();  // every thread is done with the slot
        if (threadIdx.x == 0 && j + kBulkStages < njobs) issue(slot);
    }
    if (j < njobs) {
        // a wait ran out: report it, let the copies already issued land
        // (bounded), and leave without touching anything else
        if (threadIdx.x == 0) {
            atomicOr(err, 1);
            for (int32_t k = j; k < njobs && k < j + kBulkStages; ++k)
                mbar_wait_bounded(&bar[k % kBulkStages], uint32_t(k / kBulkStages) & 1u);
        }
        return;
    }
    // element path: tensors that are not 16-byte aligned, and vector tails
    for (int32_t ci = c0; ci < c1; ++ci) {
        const ChunkPtr ch = load_chunk(chunks + ci);
        const int64_t len = ch.len2 >> 1;
        if (ch.len2 & 1) {
            const int64_t len8 = len / kVec * kVec;
            if (len8 < len) {
                ChunkPtr t = ch;
                t.p = static_cast<uint16_t*>(ch.p) + len8;
                t.g = static_cast<const uint16_t*>(ch.g) + len8;
                t.m = static_cast<uint16_t*>(ch.m) + len8;
                t.v = static_cast<uint16_t*>(ch.v) + len8;
                t.a = static_cast<uint16_t*>(ch.a) + len8;
                kahan_elem_chunk<K>(t, len - len8, s, coef, bad);
            }
        } else {
            kahan_elem_chunk<K>(ch, len, s, coef, bad);
        }
    }
    if (K == kReport) {
        if (__syncthreads_or(bad) && threadIdx.x == 0) *report = 1;
    }
}
#endif  // ADAMW_BULK

}  // namespace
