// device_common.cuh -- device-side building blocks of every kernel: bf16
// helpers, streaming 16-byte loads and stores, the per-element AdamW
// arithmetic of each storage mode, the chunk walkers, the CTA bodies of the
// update and of the norm pass, and the device-side per-step scalars.
//
// Arithmetic order follows the definition in include/adamw_sm.h exactly, with
// the IEEE round-to-nearest intrinsics (__fmul_rn, __fadd_rn, __fdiv_rn,
// __fsqrt_rn) so that no multiply-add is fused and every result is the one a
// strict host implementation of the same formula gives.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <cstring>

#include "adamw_internal.h"

// Everything here has internal linkage: each translation unit that includes
// this header compiles its own copy of what it uses.
namespace {

using namespace adamw;

// ------------------------------------------------------------ helpers ----

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> bf16, round to nearest even, lo in the low half-word.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    uint32_t u;
    memcpy(&u, &r, sizeof u);
    return u;
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float from_bf16(uint16_t h) {
    return __uint_as_float(uint32_t(h) << 16);
}

// Streaming 16-byte accesses.  Every byte is touched once per step.  The
// cache policy of loads and stores is a build-time constant: 0 = default,
// 1 = evict-first (.cs), 2 = L1 no-allocate, 3 = last-use (.lu) for loads.
// Measured on GB300, the default policy is as fast as any hint for lists
// larger than L2 and keeps L2-resident lists resident between steps.
#ifndef ADAMW_LD_POLICY
#define ADAMW_LD_POLICY 0
#endif
#ifndef ADAMW_ST_POLICY
#define ADAMW_ST_POLICY 0
#endif
__device__ __forceinline__ uint4 ld16(const void* p) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#if ADAMW_LD_POLICY == 1
    return __ldcs(q);
#elif ADAMW_LD_POLICY == 2
    uint4 r;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(q));
    return r;
#elif ADAMW_LD_POLICY == 3
    return __ldlu(q);
#else
    return *q;
#endif
}
// A 16-byte load that asks L2 to keep the line (the evict-last policy made
// by keep_policy()): for g in the fused clipped step's norm phase, which the
// update phase reads again.
__device__ __forceinline__ uint64_t keep_policy() {
    uint64_t policy;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}
__device__ __forceinline__ uint4 ld16_keep(const void* p, uint64_t policy) {
    uint4 r;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(policy));
    return r;
}

__device__ __forceinline__ void st16(void* p, uint4 v) {
    uint4* q = reinterpret_cast<uint4*>(p);
#if ADAMW_ST_POLICY == 1
    __stcs(q, v);
#else
    *q = v;
#endif
}

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialization (launch.h), so it may start while
// the kernel before it in the stream is still running: it may read only what
// no earlier kernel writes (the plan's chunk table) before pdl_wait(), which
// returns once every earlier kernel has finished and its writes are visible.
// pdl_trigger() lets the next kernel launch before this one ends (it waits
// in pdl_wait() all the same).  Both are no-ops for a kernel launched
// without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ bool bf16x2_nonfinite(uint32_t w) {
    return ((w & 0x7f80u) == 0x7f80u) || ((w & 0x7f800000u) == 0x7f800000u);
}

// ------------------------------------------------ per-element arithmetic --

// m' and v' of one element (fp32).
__device__ __forceinline__ void moments(const StepScalars& s, float g, float m0,
                                        float v0, float& m1, float& v1) {
    m1 = __fadd_rn(__fmul_rn(s.beta1, m0), __fmul_rn(s.omb1, g));
    v1 = __fadd_rn(__fmul_rn(s.beta2, v0), __fmul_rn(__fmul_rn(s.omb2, g), g));
}

// upd = step_size * (m / (sqrt(v)/sbc2 + eps)) + lrwd * p
__device__ __forceinline__ float update_of(const StepScalars& s, float m, float v,
                                          float p0) {
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.sbc2), s.eps);
    return __fadd_rn(__fmul_rn(s.step_size, __fdiv_rn(m, den)), __fmul_rn(s.lrwd, p0));
}

// bf16 Kahan mode on two elements packed in 32-bit words (lo, hi halves).
template <int K>
__device__ __forceinline__ void kahan_x2(const StepScalars& s, float coef, uint32_t gw,
                                         uint32_t& pw, uint32_t& mw, uint32_t& vw,
                                         uint32_t& cw) {
    float g0 = bf16_lo(gw), g1 = bf16_hi(gw);
    if (K == kClip) {
        g0 = __fmul_rn(g0, coef);
        g1 = __fmul_rn(g1, coef);
    }
    const float p0 = bf16_lo(pw), p1 = bf16_hi(pw);
    float ma, mb, va, vb;
    moments(s, g0, bf16_lo(mw), bf16_lo(vw), ma, va);
    moments(s, g1, bf16_hi(mw), bf16_hi(vw), mb, vb);
    mw = pack_bf16x2(ma, mb);
    vw = pack_bf16x2(va, vb);
    // the stored (bf16) moments feed the update
    const float y0 = __fsub_rn(bf16_lo(cw), update_of(s, bf16_lo(mw), bf16_lo(vw), p0));
    const float y1 = __fsub_rn(bf16_hi(cw), update_of(s, bf16_hi(mw), bf16_hi(vw), p1));
    const uint32_t pn = pack_bf16x2(__fadd_rn(p0, y0), __fadd_rn(p1, y1));
    cw = pack_bf16x2(__fsub_rn(y0, __fsub_rn(bf16_lo(pn), p0)),
                     __fsub_rn(y1, __fsub_rn(bf16_hi(pn), p1)));
    pw = pn;
}

template <int K>
__device__ __forceinline__ void kahan_x1(const StepScalars& s, float coef, uint16_t gh,
                                         uint16_t& ph, uint16_t& mh, uint16_t& vh,
                                         uint16_t& ch) {
    float g = from_bf16(gh);
    if (K == kClip) g = __fmul_rn(g, coef);
    const float p0 = from_bf16(ph);
    float m1, v1;
    moments(s, g, from_bf16(mh), from_bf16(vh), m1, v1);
    mh = to_bf16(m1);
    vh = to_bf16(v1);
    const float y = __fsub_rn(from_bf16(ch), update_of(s, from_bf16(mh), from_bf16(vh), p0));
    const uint16_t pn = to_bf16(__fadd_rn(p0, y));
    ch = to_bf16(__fsub_rn(y, __fsub_rn(from_bf16(pn), p0)));
    ph = pn;
}

// mixed mode on one element; returns the new master.
template <int K>
__device__ __forceinline__ float mixed_x1(const StepScalars& s, float coef, float g,
                                          float p0, float& m, float& v) {
    if (K == kClip) g = __fmul_rn(g, coef);
    float m1, v1;
    moments(s, g, m, v, m1, v1);
    m = m1;
    v = v1;
    return __fsub_rn(p0, update_of(s, m1, v1, p0));
}

// ------------------------------------------------------- chunk walkers ----

// Per storage mode: U, the 16-byte vectors each thread has in flight per
// stream, and B, the resident CTAs per SM the update kernel's register budget
// is fitted to (0: no constraint).  Chosen by measurement on GB300 over the
// OPT-1.3b list (every mode at U = 1..3 and B = none, 2, 3), with the
// interleaved partition cut on 2048-element boundaries: the modes with fp32
// streams favour fewer vectors and more CTAs (or the reverse) according to
// their mix of 2- and 4-byte streams.  ADAMW_UNROLL and ADAMW_MIN_BLOCKS,
// when defined, override the table for every mode.
template <int MODE>
struct UpdateTuning {
    static constexpr int kU =
        MODE == ADAMW_MODE_MIXED_FP32_MASTER ? 1
        : MODE == ADAMW_MODE_BF16_KAHAN_FP32_VAR ? 1
        : MODE == (ADAMW_MODE_ANYPREC | 1) ? 1
        : MODE == (ADAMW_MODE_ANYPREC | 4) ? 1
        : MODE == (ADAMW_MODE_ANYPREC | 7) ? 1
        : MODE == (ADAMW_MODE_ANYPREC | 11) ? 3
        : 2;
    static constexpr int kB =
        MODE == ADAMW_MODE_MIXED_FP32_MASTER ? 2
        : MODE == ADAMW_MODE_BF16_KAHAN_FP32_VAR ? 3
        : MODE == (ADAMW_MODE_ANYPREC | 1) ? 3
        : MODE == (ADAMW_MODE_ANYPREC | 4) ? 3
        : MODE == (ADAMW_MODE_ANYPREC | 7) ? 2
        : MODE == (ADAMW_MODE_ANYPREC | 11) ? 2
        : 0;
#ifdef ADAMW_UNROLL
    static constexpr int kUnroll = ADAMW_UNROLL;
#else
    static constexpr int kUnroll = kU;
#endif
    // Resident CTAs per SM the update kernel reaches with the tuning above
    // (kB where set; otherwise what its registers allowed when the table was
    // fitted).  Where the code around the element loop (the claim loop of the
    // last rounds, the device step's bookkeeping) would cost a CTA per SM,
    // launch bounds hold this occupancy for the modes at 3 or 4 CTAs per SM
    // (at 2 the registers leave room, and the kernels keep the code they
    // were tuned with).
    static constexpr int kOcc =
        kB > 0 ? kB
        : MODE == ADAMW_MODE_BF16_PLAIN ? 4
        : (MODE == ADAMW_MODE_BF16_KAHAN || MODE == (ADAMW_MODE_ANYPREC | 9) ||
           MODE == (ADAMW_MODE_ANYPREC | 10)) ? 3
        : 2;
#ifdef ADAMW_MIN_BLOCKS
    static constexpr int kMinBlocks = ADAMW_MIN_BLOCKS;
#else
    static constexpr int kMinBlocks = kOcc >= 3 ? kOcc : kB;
#endif
    // The one-launch device step runs on the update's grid, so it must reach
    // the same occupancy.
    static constexpr int kSelfMinBlocks = kMinBlocks;
    // The fused clipped step: the update's own tuning.
    static constexpr int kFusedMinBlocks = kB;
};

template <int K, int U>
__device__ __forceinline__ void kahan_vec_chunk(const ChunkPtr& t, int64_t len,
                                                const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    uint16_t* v = static_cast<uint16_t*>(t.v);
    uint16_t* c = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
        uint4 G[U], P[U], M[U], V[U], C[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld16(p + i * kVec);
                M[u] = ld16(m + i * kVec);
                V[u] = ld16(v + i * kVec);
                C[u] = ld16(c + i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                if (K == kReport)
                    bad |= bf16x2_nonfinite(G[u].x) | bf16x2_nonfinite(G[u].y) |
                           bf16x2_nonfinite(G[u].z) | bf16x2_nonfinite(G[u].w);
                kahan_x2<K>(s, coef, G[u].x, P[u].x, M[u].x, V[u].x, C[u].x);
                kahan_x2<K>(s, coef, G[u].y, P[u].y, M[u].y, V[u].y, C[u].y);
                kahan_x2<K>(s, coef, G[u].z, P[u].z, M[u].z, V[u].z, C[u].z);
                kahan_x2<K>(s, coef, G[u].w, P[u].w, M[u].w, V[u].w, C[u].w);
                st16(p + i * kVec, P[u]);
                st16(m + i * kVec, M[u]);
                st16(v + i * kVec, V[u]);
                st16(c + i * kVec, C[u]);
            }
        }
    }
    // ragged end of a vector body (< kVec elements)
    const int64_t tail = len - nvec * kVec;
    if (threadIdx.x < tail) {
        const int64_t i = nvec * kVec + threadIdx.x;
        uint16_t gh = g[i], ph = p[i], mh = m[i], vh = v[i], ch = c[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        kahan_x1<K>(s, coef, gh, ph, mh, vh, ch);
        p[i] = ph; m[i] = mh; v[i] = vh; c[i] = ch;
    }
}

template <int K>
__device__ __forceinline__ void kahan_elem_chunk(const ChunkPtr& t, int64_t len,
                                                 const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    uint16_t* v = static_cast<uint16_t*>(t.v);
    uint16_t* c = static_cast<uint16_t*>(t.a);
    for (int64_t i = threadIdx.x; i < len; i += kBlock) {
        uint16_t gh = g[i], ph = p[i], mh = m[i], vh = v[i], ch = c[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        kahan_x1<K>(s, coef, gh, ph, mh, vh, ch);
        p[i] = ph; m[i] = mh; v[i] = vh; c[i] = ch;
    }
}

// 8 fp32 of a mixed-mode stream = two 16-byte accesses.
struct F8 { float x[8]; };
__device__ __forceinline__ F8 ld32(const float* p) {
    const uint4 a = ld16(p), b = ld16(p + 4);
    return {{__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z), __uint_as_float(a.w),
             __uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z), __uint_as_float(b.w)}};
}
__device__ __forceinline__ void st32(float* p, const F8& v) {
    st16(p, make_uint4(__float_as_uint(v.x[0]), __float_as_uint(v.x[1]),
                       __float_as_uint(v.x[2]), __float_as_uint(v.x[3])));
    st16(p + 4, make_uint4(__float_as_uint(v.x[4]), __float_as_uint(v.x[5]),
                           __float_as_uint(v.x[6]), __float_as_uint(v.x[7])));
}

template <int K, int U>
__device__ __forceinline__ void mixed_vec_chunk(const ChunkPtr& t, int64_t len,
                                                const StepScalars& s, float coef, bool& bad) {
    float* p = static_cast<float*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    float* m = static_cast<float*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* o = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
        uint4 G[U];
        F8 P[U], M[U], V[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld32(p + i * kVec);
                M[u] = ld32(m + i * kVec);
                V[u] = ld32(v + i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                const uint32_t gw[4] = {G[u].x, G[u].y, G[u].z, G[u].w};
                if (K == kReport)
                    bad |= bf16x2_nonfinite(gw[0]) | bf16x2_nonfinite(gw[1]) |
                           bf16x2_nonfinite(gw[2]) | bf16x2_nonfinite(gw[3]);
                uint32_t out[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int a = 2 * j, b = 2 * j + 1;
                    P[u].x[a] = mixed_x1<K>(s, coef, bf16_lo(gw[j]), P[u].x[a], M[u].x[a], V[u].x[a]);
                    P[u].x[b] = mixed_x1<K>(s, coef, bf16_hi(gw[j]), P[u].x[b], M[u].x[b], V[u].x[b]);
                    out[j] = pack_bf16x2(P[u].x[a], P[u].x[b]);
                }
                st32(p + i * kVec, P[u]);
                st32(m + i * kVec, M[u]);
                st32(v + i * kVec, V[u]);
                st16(o + i * kVec, make_uint4(out[0], out[1], out[2], out[3]));
            }
        }
    }
    const int64_t tail = len - nvec * kVec;
    if (threadIdx.x < tail) {
        const int64_t i = nvec * kVec + threadIdx.x;
        const uint16_t gh = g[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        float mi = m[i], vi = v[i];
        const float n = mixed_x1<K>(s, coef, from_bf16(gh), p[i], mi, vi);
        p[i] = n; m[i] = mi; v[i] = vi; o[i] = to_bf16(n);
    }
}

template <int K>
__device__ __forceinline__ void mixed_elem_chunk(const ChunkPtr& t, int64_t len,
                                                 const StepScalars& s, float coef, bool& bad) {
    float* p = static_cast<float*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    float* m = static_cast<float*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* o = static_cast<uint16_t*>(t.a);
    for (int64_t i = threadIdx.x; i < len; i += kBlock) {
        const uint16_t gh = g[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        float mi = m[i], vi = v[i];
        const float n = mixed_x1<K>(s, coef, from_bf16(gh), p[i], mi, vi);
        p[i] = n; m[i] = mi; v[i] = vi; o[i] = to_bf16(n);
    }
}

// bf16 without compensation, two elements per 32-bit word: p' = bf16(p - upd).
template <int K>
__device__ __forceinline__ void plain_x2(const StepScalars& s, float coef, uint32_t gw,
                                         uint32_t& pw, uint32_t& mw, uint32_t& vw) {
    float g0 = bf16_lo(gw), g1 = bf16_hi(gw);
    if (K == kClip) {
        g0 = __fmul_rn(g0, coef);
        g1 = __fmul_rn(g1, coef);
    }
    const float p0 = bf16_lo(pw), p1 = bf16_hi(pw);
    float ma, mb, va, vb;
    moments(s, g0, bf16_lo(mw), bf16_lo(vw), ma, va);
    moments(s, g1, bf16_hi(mw), bf16_hi(vw), mb, vb);
    mw = pack_bf16x2(ma, mb);
    vw = pack_bf16x2(va, vb);
    pw = pack_bf16x2(__fsub_rn(p0, update_of(s, bf16_lo(mw), bf16_lo(vw), p0)),
                     __fsub_rn(p1, update_of(s, bf16_hi(mw), bf16_hi(vw), p1)));
}

template <int K>
__device__ __forceinline__ void plain_x1(const StepScalars& s, float coef, uint16_t gh,
                                         uint16_t& ph, uint16_t& mh, uint16_t& vh) {
    float g = from_bf16(gh);
    if (K == kClip) g = __fmul_rn(g, coef);
    const float p0 = from_bf16(ph);
    float m1, v1;
    moments(s, g, from_bf16(mh), from_bf16(vh), m1, v1);
    mh = to_bf16(m1);
    vh = to_bf16(v1);
    ph = to_bf16(__fsub_rn(p0, update_of(s, from_bf16(mh), from_bf16(vh), p0)));
}

// bf16 Kahan with fp32 variance, one element: v stays fp32.
template <int K>
__device__ __forceinline__ void kahan_v32_x1(const StepScalars& s, float coef, float g,
                                             float p0, float m0, float& v, float c0,
                                             uint16_t& ph, uint16_t& mh, uint16_t& ch) {
    if (K == kClip) g = __fmul_rn(g, coef);
    float m1, v1;
    moments(s, g, m0, v, m1, v1);
    mh = to_bf16(m1);
    v = v1;
    const float y = __fsub_rn(c0, update_of(s, from_bf16(mh), v1, p0));
    ph = to_bf16(__fadd_rn(p0, y));
    ch = to_bf16(__fsub_rn(y, __fsub_rn(from_bf16(ph), p0)));
}

template <int K, int U>
__device__ __forceinline__ void plain_vec_chunk(const ChunkPtr& t, int64_t len,
                                                const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    uint16_t* v = static_cast<uint16_t*>(t.v);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
        uint4 G[U], P[U], M[U], V[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld16(p + i * kVec);
                M[u] = ld16(m + i * kVec);
                V[u] = ld16(v + i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                if (K == kReport)
                    bad |= bf16x2_nonfinite(G[u].x) | bf16x2_nonfinite(G[u].y) |
                           bf16x2_nonfinite(G[u].z) | bf16x2_nonfinite(G[u].w);
                plain_x2<K>(s, coef, G[u].x, P[u].x, M[u].x, V[u].x);
                plain_x2<K>(s, coef, G[u].y, P[u].y, M[u].y, V[u].y);
                plain_x2<K>(s, coef, G[u].z, P[u].z, M[u].z, V[u].z);
                plain_x2<K>(s, coef, G[u].w, P[u].w, M[u].w, V[u].w);
                st16(p + i * kVec, P[u]);
                st16(m + i * kVec, M[u]);
                st16(v + i * kVec, V[u]);
            }
        }
    }
    const int64_t tail = len - nvec * kVec;
    if (threadIdx.x < tail) {
        const int64_t i = nvec * kVec + threadIdx.x;
        uint16_t gh = g[i], ph = p[i], mh = m[i], vh = v[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        plain_x1<K>(s, coef, gh, ph, mh, vh);
        p[i] = ph; m[i] = mh; v[i] = vh;
    }
}

template <int K>
__device__ __forceinline__ void plain_elem_chunk(const ChunkPtr& t, int64_t len,
                                                 const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    uint16_t* v = static_cast<uint16_t*>(t.v);
    for (int64_t i = threadIdx.x; i < len; i += kBlock) {
        uint16_t gh = g[i], ph = p[i], mh = m[i], vh = v[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        plain_x1<K>(s, coef, gh, ph, mh, vh);
        p[i] = ph; m[i] = mh; v[i] = vh;
    }
}

template <int K, int U>
__device__ __forceinline__ void kahan_v32_vec_chunk(const ChunkPtr& t, int64_t len,
                                                    const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* c = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
        uint4 G[U], P[U], M[U], C[U];
        F8 V[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld16(p + i * kVec);
                M[u] = ld16(m + i * kVec);
                V[u] = ld32(v + i * kVec);
                C[u] = ld16(c + i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                const uint32_t gw[4] = {G[u].x, G[u].y, G[u].z, G[u].w};
                const uint32_t pw[4] = {P[u].x, P[u].y, P[u].z, P[u].w};
                const uint32_t mw[4] = {M[u].x, M[u].y, M[u].z, M[u].w};
                const uint32_t cw[4] = {C[u].x, C[u].y, C[u].z, C[u].w};
                if (K == kReport)
                    bad |= bf16x2_nonfinite(gw[0]) | bf16x2_nonfinite(gw[1]) |
                           bf16x2_nonfinite(gw[2]) | bf16x2_nonfinite(gw[3]);
                uint32_t po[4], mo[4], co[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint16_t ph0, mh0, ch0, ph1, mh1, ch1;
                    kahan_v32_x1<K>(s, coef, bf16_lo(gw[j]), bf16_lo(pw[j]), bf16_lo(mw[j]),
                                    V[u].x[2 * j], bf16_lo(cw[j]), ph0, mh0, ch0);
                    kahan_v32_x1<K>(s, coef, bf16_hi(gw[j]), bf16_hi(pw[j]), bf16_hi(mw[j]),
                                    V[u].x[2 * j + 1], bf16_hi(cw[j]), ph1, mh1, ch1);
                    po[j] = uint32_t(ph0) | (uint32_t(ph1) << 16);
                    mo[j] = uint32_t(mh0) | (uint32_t(mh1) << 16);
                    co[j] = uint32_t(ch0) | (uint32_t(ch1) << 16);
                }
                st16(p + i * kVec, make_uint4(po[0], po[1], po[2], po[3]));
                st16(m + i * kVec, make_uint4(mo[0], mo[1], mo[2], mo[3]));
                st32(v + i * kVec, V[u]);
                st16(c + i * kVec, make_uint4(co[0], co[1], co[2], co[3]));
            }
        }
    }
    const int64_t tail = len - nvec * kVec;
    if (threadIdx.x < tail) {
        const int64_t i = nvec * kVec + threadIdx.x;
        const uint16_t gh = g[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        float vi = v[i];
        uint16_t ph, mh, ch;
        kahan_v32_x1<K>(s, coef, from_bf16(gh), from_bf16(p[i]), from_bf16(m[i]), vi,
                        from_bf16(c[i]), ph, mh, ch);
        p[i] = ph; m[i] = mh; v[i] = vi; c[i] = ch;
    }
}

template <int K>
__device__ __forceinline__ void kahan_v32_elem_chunk(const ChunkPtr& t, int64_t len,
                                                     const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* c = static_cast<uint16_t*>(t.a);
    for (int64_t i = threadIdx.x; i < len; i += kBlock) {
        const uint16_t gh = g[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        float vi = v[i];
        uint16_t ph, mh, ch;
        kahan_v32_x1<K>(s, coef, from_bf16(gh), from_bf16(p[i]), from_bf16(m[i]), vi,
                        from_bf16(c[i]), ph, mh, ch);
        p[i] = ph; m[i] = mh; v[i] = vi; c[i] = ch;
    }
}

// ---- any precision: bf16 p and g; exp_avg, exp_avg_sq and the
// compensation each bf16 or fp32, Kahan summation on or off (FLAGS = the
// ADAMW_ANYPREC_* bits of the storage mode).

// The float holding the bf16 nearest to x (round to nearest even).
__device__ __forceinline__ float round_bf16(float x) { return from_bf16(to_bf16(x)); }

// One element.  m, v, c come in as stored and leave as stored (rounded to
// their own type); pn is the new parameter (a bf16 value).
template <int FLAGS, int K>
__device__ __forceinline__ void anyprec_x1(const StepScalars& s, float coef, float g, float p0,
                                           float& m, float& v, float& c, float& pn) {
    constexpr bool kM32 = (FLAGS & ADAMW_ANYPREC_M_FP32) != 0;
    constexpr bool kV32 = (FLAGS & ADAMW_ANYPREC_V_FP32) != 0;
    constexpr bool kC32 = (FLAGS & ADAMW_ANYPREC_C_FP32) != 0;
    constexpr bool kKahan = (FLAGS & ADAMW_ANYPREC_NO_KAHAN) == 0;
    if (K == kClip) g = __fmul_rn(g, coef);
    float m1, v1;
    moments(s, g, m, v, m1, v1);
    m = kM32 ? m1 : round_bf16(m1);
    v = kV32 ? v1 : round_bf16(v1);
    const float upd = update_of(s, m, v, p0);
    if (kKahan) {
        const float y = __fsub_rn(c, upd);
        pn = round_bf16(__fadd_rn(p0, y));
        const float cn = __fsub_rn(y, __fsub_rn(pn, p0));
        c = kC32 ? cn : round_bf16(cn);
    } else {
        pn = round_bf16(__fsub_rn(p0, upd));
    }
}

// Eight consecutive elements of one stream as loaded: bf16 (one 16-byte
// access) or fp32 (two).  set2 takes values that are already of the
// stream's type.
template <bool F32>
struct Raw8;
template <>
struct Raw8<false> {
    uint4 r;
    __device__ __forceinline__ void load(const void* b, int64_t e) {
        r = ld16(static_cast<const uint16_t*>(b) + e);
    }
    __device__ __forceinline__ void store(void* b, int64_t e) const {
        st16(static_cast<uint16_t*>(b) + e, r);
    }
    __device__ __forceinline__ uint32_t word(int w) const {
        return w == 0 ? r.x : w == 1 ? r.y : w == 2 ? r.z : r.w;
    }
    __device__ __forceinline__ float get(int j) const {
        return (j & 1) ? bf16_hi(word(j >> 1)) : bf16_lo(word(j >> 1));
    }
    __device__ __forceinline__ void set2(int w, float lo, float hi) {
        const uint32_t u = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xffff0000u);
        if (w == 0) r.x = u;
        else if (w == 1) r.y = u;
        else if (w == 2) r.z = u;
        else r.w = u;
    }
};
template <>
struct Raw8<true> {
    F8 r;
    __device__ __forceinline__ void load(const void* b, int64_t e) {
        r = ld32(static_cast<const float*>(b) + e);
    }
    __device__ __forceinline__ void store(void* b, int64_t e) const {
        st32(static_cast<float*>(b) + e, r);
    }
    __device__ __forceinline__ float get(int j) const { return r.x[j]; }
    __device__ __forceinline__ void set2(int w, float lo, float hi) {
        r.x[2 * w] = lo;
        r.x[2 * w + 1] = hi;
    }
};

// One element of a bf16 or fp32 stream; the value stored must already be of
// the stream's type.
template <bool F32>
__device__ __forceinline__ float ld1(const void* b, int64_t i) {
    if constexpr (F32) return static_cast<const float*>(b)[i];
    else return from_bf16(static_cast<const uint16_t*>(b)[i]);
}
template <bool F32>
__device__ __forceinline__ void st1(void* b, int64_t i, float x) {
    if constexpr (F32) static_cast<float*>(b)[i] = x;
    else static_cast<uint16_t*>(b)[i] = uint16_t(__float_as_uint(x) >> 16);
}

template <int FLAGS, int K>
__device__ __forceinline__ void anyprec_one(const ChunkPtr& t, int64_t i, const StepScalars& s,
                                            float coef, bool& bad) {
    constexpr bool kM32 = (FLAGS & ADAMW_ANYPREC_M_FP32) != 0;
    constexpr bool kV32 = (FLAGS & ADAMW_ANYPREC_V_FP32) != 0;
    constexpr bool kC32 = (FLAGS & ADAMW_ANYPREC_C_FP32) != 0;
    constexpr bool kKahan = (FLAGS & ADAMW_ANYPREC_NO_KAHAN) == 0;
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t gh = static_cast<const uint16_t*>(t.g)[i];
    if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
    float m = ld1<kM32>(t.m, i), v = ld1<kV32>(t.v, i);
    float c = kKahan ? ld1<kC32>(t.a, i) : 0.0f;
    float pn;
    anyprec_x1<FLAGS, K>(s, coef, from_bf16(gh), from_bf16(p[i]), m, v, c, pn);
    p[i] = uint16_t(__float_as_uint(pn) >> 16);
    st1<kM32>(t.m, i, m);
    st1<kV32>(t.v, i, v);
    if (kKahan) st1<kC32>(t.a, i, c);
}

template <int FLAGS, int K, int U>
__device__ __forceinline__ void anyprec_vec_chunk(const ChunkPtr& t, int64_t len,
                                                  const StepScalars& s, float coef, bool& bad) {
    constexpr bool kM32 = (FLAGS & ADAMW_ANYPREC_M_FP32) != 0;
    constexpr bool kV32 = (FLAGS & ADAMW_ANYPREC_V_FP32) != 0;
    constexpr bool kC32 = (FLAGS & ADAMW_ANYPREC_C_FP32) != 0;
    constexpr bool kKahan = (FLAGS & ADAMW_ANYPREC_NO_KAHAN) == 0;
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
        uint4 G[U], P[U];
        Raw8<kM32> M[U];
        Raw8<kV32> V[U];
        Raw8<kC32> C[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld16(p + i * kVec);
                M[u].load(t.m, i * kVec);
                V[u].load(t.v, i * kVec);
                if (kKahan) C[u].load(t.a, i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                const uint32_t gw[4] = {G[u].x, G[u].y, G[u].z, G[u].w};
                const uint32_t pw[4] = {P[u].x, P[u].y, P[u].z, P[u].w};
                if (K == kReport)
                    bad |= bf16x2_nonfinite(gw[0]) | bf16x2_nonfinite(gw[1]) |
                           bf16x2_nonfinite(gw[2]) | bf16x2_nonfinite(gw[3]);
                uint32_t po[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    float m0 = M[u].get(2 * w), m1 = M[u].get(2 * w + 1);
                    float v0 = V[u].get(2 * w), v1 = V[u].get(2 * w + 1);
                    float c0 = kKahan ? C[u].get(2 * w) : 0.0f;
                    float c1 = kKahan ? C[u].get(2 * w + 1) : 0.0f;
                    float pn0, pn1;
                    anyprec_x1<FLAGS, K>(s, coef, bf16_lo(gw[w]), bf16_lo(pw[w]), m0, v0, c0, pn0);
                    anyprec_x1<FLAGS, K>(s, coef, bf16_hi(gw[w]), bf16_hi(pw[w]), m1, v1, c1, pn1);
                    po[w] = (__float_as_uint(pn0) >> 16) | (__float_as_uint(pn1) & 0xffff0000u);
                    M[u].set2(w, m0, m1);
                    V[u].set2(w, v0, v1);
                    if (kKahan) C[u].set2(w, c0, c1);
                }
                st16(p + i * kVec, make_uint4(po[0], po[1], po[2], po[3]));
                M[u].store(t.m, i * kVec);
                V[u].store(t.v, i * kVec);
                if (kKahan) C[u].store(t.a, i * kVec);
            }
        }
    }
    // ragged end of a vector body (< kVec elements)
    const int64_t tail = len - nvec * kVec;
    if (threadIdx.x < tail) anyprec_one<FLAGS, K>(t, nvec * kVec + threadIdx.x, s, coef, bad);
}

template <int FLAGS, int K>
__device__ __forceinline__ void anyprec_elem_chunk(const ChunkPtr& t, int64_t len,
                                                   const StepScalars& s, float coef, bool& bad) {
    for (int64_t i = threadIdx.x; i < len; i += kBlock) anyprec_one<FLAGS, K>(t, i, s, coef, bad);
}

// Remainder mode: the fp32 master is the bf16 parameter (high half) plus a
// signed 16-bit remainder of the bit pattern.
__device__ __forceinline__ float join_master(uint32_t hi_bits, uint32_t rem16) {
    return __uint_as_float(hi_bits + uint32_t(int32_t(int16_t(uint16_t(rem16)))));
}
// Nearest bf16 high half (ties away from zero) and the remainder restoring it.
__device__ __forceinline__ void split_master(float x, uint32_t& hi16, uint32_t& rem16) {
    const uint32_t u = __float_as_uint(x);
    hi16 = (u + 0x8000u) >> 16;
    rem16 = (u - (hi16 << 16)) & 0xffffu;
}

template <int K, int U>
__device__ __forceinline__ void remainder_vec_chunk(const ChunkPtr& t, int64_t len,
                                                    const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    float* m = static_cast<float*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* r = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
        uint4 G[U], P[U], R[U];
        F8 M[U], V[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld16(p + i * kVec);
                R[u] = ld16(r + i * kVec);
                M[u] = ld32(m + i * kVec);
                V[u] = ld32(v + i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                const uint32_t gw[4] = {G[u].x, G[u].y, G[u].z, G[u].w};
                const uint32_t pw[4] = {P[u].x, P[u].y, P[u].z, P[u].w};
                const uint32_t rw[4] = {R[u].x, R[u].y, R[u].z, R[u].w};
                if (K == kReport)
                    bad |= bf16x2_nonfinite(gw[0]) | bf16x2_nonfinite(gw[1]) |
                           bf16x2_nonfinite(gw[2]) | bf16x2_nonfinite(gw[3]);
                uint32_t po[4], ro[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int a = 2 * j, b = 2 * j + 1;
                    const float n0 = mixed_x1<K>(s, coef, bf16_lo(gw[j]),
                                                 join_master(pw[j] << 16, rw[j]), M[u].x[a], V[u].x[a]);
                    const float n1 = mixed_x1<K>(s, coef, bf16_hi(gw[j]),
                                                 join_master(pw[j] & 0xffff0000u, rw[j] >> 16),
                                                 M[u].x[b], V[u].x[b]);
                    uint32_t h0, r0, h1, r1;
                    split_master(n0, h0, r0);
                    split_master(n1, h1, r1);
                    po[j] = h0 | (h1 << 16);
                    ro[j] = r0 | (r1 << 16);
                }
                st16(p + i * kVec, make_uint4(po[0], po[1], po[2], po[3]));
                st16(r + i * kVec, make_uint4(ro[0], ro[1], ro[2], ro[3]));
                st32(m + i * kVec, M[u]);
                st32(v + i * kVec, V[u]);
            }
        }
    }
    const int64_t tail = len - nvec * kVec;
    if (threadIdx.x < tail) {
        const int64_t i = nvec * kVec + threadIdx.x;
        const uint16_t gh = g[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        float mi = m[i], vi = v[i];
        const float n = mixed_x1<K>(s, coef, from_bf16(gh), join_master(uint32_t(p[i]) << 16, r[i]),
                                    mi, vi);
        uint32_t h, rr;
        split_master(n, h, rr);
        p[i] = uint16_t(h); r[i] = uint16_t(rr); m[i] = mi; v[i] = vi;
    }
}

template <int K>
__device__ __forceinline__ void remainder_elem_chunk(const ChunkPtr& t, int64_t len,
                                                     const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    float* m = static_cast<float*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* r = static_cast<uint16_t*>(t.a);
    for (int64_t i = threadIdx.x; i < len; i += kBlock) {
        const uint16_t gh = g[i];
        if (K == kReport) bad |= (gh & 0x7f80u) == 0x7f80u;
        float mi = m[i], vi = v[i];
        const float n = mixed_x1<K>(s, coef, from_bf16(gh), join_master(uint32_t(p[i]) << 16, r[i]),
                                    mi, vi);
        uint32_t h, rr;
        split_master(n, h, rr);
        p[i] = uint16_t(h); r[i] = uint16_t(rr); m[i] = mi; v[i] = vi;
    }
}

// The update: CTA b walks chunks [cta_begin[b], cta_begin[b+1]).
#define ADAMW_UPDATE_BOUNDS(MODE) __launch_bounds__(kBlock, UpdateTuning<MODE>::kMinBlocks)
#define ADAMW_SELF_BOUNDS(MODE) __launch_bounds__(kBlock, UpdateTuning<MODE>::kSelfMinBlocks)
#define ADAMW_FUSED_BOUNDS(MODE) __launch_bounds__(kBlock, UpdateTuning<MODE>::kFusedMinBlocks)

// One chunk descriptor, read through the read-only path.
__device__ __forceinline__ ChunkPtr load_chunk(const ChunkPtr* c) {
#if ADAMW_CHECK_BOUNDS
    return *c;
#else
    const ulonglong2* q = reinterpret_cast<const ulonglong2*>(c);
    const ulonglong2 a = __ldg(q), b = __ldg(q + 1), d = __ldg(q + 2);
    ChunkPtr r;
    r.p = reinterpret_cast<void*>(a.x);
    r.g = reinterpret_cast<const void*>(a.y);
    r.m = reinterpret_cast<void*>(b.x);
    r.v = reinterpret_cast<void*>(b.y);
    r.a = reinterpret_cast<void*>(d.x);
    r.len2 = static_cast<int64_t>(d.y);
    return r;
#endif
}

// Bytes per element of stream s (param, grad, exp_avg, exp_avg_sq, aux) in
// storage mode MODE, 0 for a stream the mode does not use; written out here
// independently of the host planner's table, so the bounds check
// cross-checks it.
template <int MODE>
__device__ constexpr int stream_bytes(int s) {
    if (MODE >= ADAMW_MODE_ANYPREC) {
        constexpr int f = MODE & 15;
        return s < 2 ? 2 : s == 2 ? ((f & 1) ? 4 : 2) : s == 3 ? ((f & 2) ? 4 : 2)
                                                      : ((f & 8) ? 0 : (f & 4) ? 4 : 2);
    }
    if (MODE == ADAMW_MODE_MIXED_FP32_MASTER) return s == 0 || s == 2 || s == 3 ? 4 : 2;
    if (MODE == ADAMW_MODE_MIXED_BF16_REMAINDER) return s == 2 || s == 3 ? 4 : 2;
    if (MODE == ADAMW_MODE_BF16_PLAIN) return s == 4 ? 0 : 2;
    if (MODE == ADAMW_MODE_BF16_KAHAN_FP32_VAR) return s == 3 ? 4 : 2;
    return 2;
}

#if ADAMW_CHECK_BOUNDS
// Whether the chunk's `len` elements lie inside its tensor's buffers, for
// every stream of MODE selected by `mask` (bit s = stream s).  A chunk that
// does not is reported in the plan's status word; the caller skips it.
template <int MODE>
__device__ __forceinline__ bool chunk_in_bounds(const ChunkPtr& c, int64_t len, int mask = 31) {
    const void* ptr[5] = {c.p, c.g, c.m, c.v, c.a};
    bool ok = len >= 0;
#pragma unroll
    for (int s = 0; s < 5; ++s) {
        const int es = stream_bytes<MODE>(s);
        if (es == 0 || !((mask >> s) & 1)) continue;
        const char* b = static_cast<const char*>(ptr[s]);
        ok = ok && b >= static_cast<const char*>(c.lo[s]) &&
             b + len * es <= static_cast<const char*>(c.hi[s]);
    }
    if (!ok && threadIdx.x == 0) atomicOr(c.status, kStatusBounds);
    return ok;
}
#endif

// ---- one chunk of the update
template <int MODE, int K>
__device__ __forceinline__ void update_chunk(const ChunkPtr& cur, const StepScalars& s, float coef,
                                             bool& bad) {
    constexpr int kU = UpdateTuning<MODE>::kUnroll;
    const int64_t len = cur.len2 >> 1;
    const bool vec = cur.len2 & 1;
#if ADAMW_CHECK_BOUNDS
    if (!chunk_in_bounds<MODE>(cur, len)) return;
#endif
    if constexpr (MODE == ADAMW_MODE_BF16_KAHAN) {
        if (vec) kahan_vec_chunk<K, kU>(cur, len, s, coef, bad);
        else kahan_elem_chunk<K>(cur, len, s, coef, bad);
    } else if constexpr (MODE == ADAMW_MODE_MIXED_FP32_MASTER) {
        if (vec) mixed_vec_chunk<K, kU>(cur, len, s, coef, bad);
        else mixed_elem_chunk<K>(cur, len, s, coef, bad);
    } else if constexpr (MODE == ADAMW_MODE_MIXED_BF16_REMAINDER) {
        if (vec) remainder_vec_chunk<K, kU>(cur, len, s, coef, bad);
        else remainder_elem_chunk<K>(cur, len, s, coef, bad);
    } else if constexpr (MODE == ADAMW_MODE_BF16_PLAIN) {
        if (vec) plain_vec_chunk<K, kU>(cur, len, s, coef, bad);
        else plain_elem_chunk<K>(cur, len, s, coef, bad);
    } else if constexpr (MODE == ADAMW_MODE_BF16_KAHAN_FP32_VAR) {
        if (vec) kahan_v32_vec_chunk<K, kU>(cur, len, s, coef, bad);
        else kahan_v32_elem_chunk<K>(cur, len, s, coef, bad);
    } else {
        constexpr int kFlags = MODE & ~ADAMW_MODE_ANYPREC;
        if (vec) anyprec_vec_chunk<kFlags, K, kU>(cur, len, s, coef, bad);
        else anyprec_elem_chunk<kFlags, K>(cur, len, s, coef, bad);
    }
}

// ---- the CTA's share of the update: its own chunks [c0, c1), each chunk's
// descriptor fetched one ahead (`cur` holds chunk c0 already when c0 < c1),
// then claimable chunks until none is left.
template <int MODE, int K>
__device__ __forceinline__ void update_cta_from(const ChunkPtr* __restrict__ chunks, int32_t c0,
                                                int32_t c1, ChunkPtr cur, const StepScalars& s,
                                                float coef, bool& bad, const DynTail& dyn) {
    for (int32_t ci = c0; ci < c1; ++ci) {
        ChunkPtr nxt = cur;
        if (ci + 1 < c1) nxt = load_chunk(chunks + ci + 1);
        update_chunk<MODE, K>(cur, s, coef, bad);
        cur = nxt;
    }
    if (dyn.n == 0) return;
    // Claims: thread 0 asks for the next piece when a piece starts and
    // hands the answer over when it ends, so the atomic's latency overlaps
    // the piece.  A claim at or past n means the list is done.
    __shared__ int32_t claim_sh;
    if (threadIdx.x == 0) claim_sh = int32_t(atomicAdd(dyn.sync, kSyncClaim) & kSyncClaimMask);
    __syncthreads();
    int32_t i = claim_sh;
    while (i < dyn.n) {
        const ChunkPtr piece = load_chunk(chunks + dyn.begin + i);
        __syncthreads();   // every thread has read claim_sh
        unsigned long long next = 0;
        if (threadIdx.x == 0) next = atomicAdd(dyn.sync, kSyncClaim);
        update_chunk<MODE, K>(piece, s, coef, bad);
        if (threadIdx.x == 0) claim_sh = int32_t(next & kSyncClaimMask);
        __syncthreads();
        i = claim_sh;
    }
}

// The CTA has finished: counts its arrival (and, with `flagged`, that it saw
// a non-finite gradient) in the claim-and-arrival word; returns the word as
// it was before, with this arrival and flag added.  The last CTA to arrive
// zeroes the word.  Thread 0 only.
__device__ __forceinline__ unsigned long long sync_arrive(unsigned long long* sync, bool flagged,
                                                          uint32_t grid) {
    const unsigned long long add = kSyncArrive + (flagged ? kSyncFlagged : 0ull);
    const unsigned long long w = atomicAdd(sync, add) + add;
    if (((w & kSyncArriveMask) / kSyncArrive) == grid) *sync = 0;
    return w;
}

template <int MODE, int K>
__device__ __forceinline__ void update_cta(const ChunkPtr* __restrict__ chunks, int32_t c0,
                                           int32_t c1, const StepScalars& s, float coef,
                                           bool& bad, const DynTail& dyn) {
    ChunkPtr cur;
    if (c0 < c1) cur = load_chunk(chunks + c0);
    update_cta_from<MODE, K>(chunks, c0, c1, cur, s, coef, bad, dyn);
}

// Error-free fp32 accumulation of non-negative terms.  Squares of bf16 values
// are exact in fp32 for |g| in [2^-63, 2^64); a group of terms is summed in
// fp32 with the exact rounding error of every addition collected on the
// side (so no bit of any square is lost), and flushed: its sum into an fp64
// total, its collected error (at most 2^-18 of the sum) into an fp32 sum of
// the errors.  Sum2F32x2 below does this on two lanes at once.
__device__ __forceinline__ float sq(float x) { return __fmul_rn(x, x); }

// Rounds of kNormUnroll vectors between flushes of the norm's error-free
// groups into fp64: 256 elements (128 per lane).
constexpr int kNormFlushRounds = 32 / kNormUnroll > 0 ? 32 / kNormUnroll : 1;

// Packed fp32x2 arithmetic (two IEEE round-to-nearest operations in one
// instruction on sm_100 and later): a 64-bit value holds two floats, lane 0
// in the low word.
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// The two bf16 of a 32-bit word as a packed pair of floats (exact).
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
    return uint64_t(w << 16) | (uint64_t(w & 0xffff0000u) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t x) { return __uint_as_float(uint32_t(x)); }
__device__ __forceinline__ float f2_hi(uint64_t x) { return __uint_as_float(uint32_t(x >> 32)); }

// That accumulation on two interleaved streams of terms at once, one per
// lane of a packed pair, with Knuth's TwoSum (t = s + x; b = t - s; error =
// (s - (t - b)) + (x - b), exact for any two floats without overflow), which
// needs no ordering of its operands (so it packs, and a NaN term stays in
// the sum, where the flush's range check sees it).  Per lane: s + e is the
// exact sum of the lane's terms since the last flush, up to the rounding of
// e itself (relative 2^-24 of an e that is itself at most 2^-17 of s for the
// 128 terms per lane of a group); the group length only bounds that.
struct Sum2F32x2 {
    uint64_t s = 0, e = 0;
    __device__ __forceinline__ void add(uint64_t x) {
        const uint64_t t = f2_add(s, x);
        const uint64_t b = f2_sub(t, s);
        e = f2_add(e, f2_add(f2_sub(s, f2_sub(t, b)), f2_sub(x, b)));
        s = t;
    }
    // Adds both lanes' groups to (acc, err) and restarts them: the two lane
    // sums are joined exactly in fp32 (TwoSum again; its error goes to err
    // with the lanes' own), so the slow fp64 unit sees one conversion and
    // one addition per flush.  False when a group left the range where
    // squares are exact and sums finite.
    __device__ __forceinline__ bool flush(double& acc, float& err) {
        const float s0 = f2_lo(s), s1 = f2_hi(s);
        const bool ok = s0 < 0x1p100f && s1 < 0x1p100f;   // also false for inf and NaN
        const float t = __fadd_rn(s0, s1);
        const float b = __fsub_rn(t, s0);
        const float e01 = __fadd_rn(__fsub_rn(s0, __fsub_rn(t, b)), __fsub_rn(s1, b));
        acc += double(t);
        err = __fadd_rn(err, __fadd_rn(__fadd_rn(f2_lo(e), f2_hi(e)), e01));
        s = 0;
        e = 0;
        return ok;
    }
};

// Walks the g elements of one CTA's chunks that belong to this thread, in a
// fixed order: vec(w) gets 8 packed bf16, elem(h) one bf16, after_iter() runs
// after every group of U vectors.
// `pre`, when set, is chunk c0 already loaded.
template <int U, bool KEEP = false, typename FV, typename FE, typename FI>
__device__ __forceinline__ void for_thread_grads(const ChunkPtr* __restrict__ chunks,
                                                 int32_t c0, int32_t c1, FV vec, FE elem,
                                                 FI after_iter, const ChunkPtr* pre = nullptr) {
    const uint64_t policy = KEEP ? keep_policy() : 0;
    for (int32_t ci = c0; ci < c1; ++ci) {
        const ChunkPtr ch = (pre && ci == c0) ? *pre : load_chunk(chunks + ci);
        const uint16_t* g = static_cast<const uint16_t*>(ch.g);
        const int64_t len = ch.len2 >> 1;
#if ADAMW_CHECK_BOUNDS
        if (!chunk_in_bounds<ADAMW_MODE_BF16_KAHAN>(ch, len, 1 << 1)) continue;  // g only
#endif
        int64_t done = 0;
        if (ch.len2 & 1) {
            const int64_t nvec = len / kVec;
            for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
                uint4 w[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t i = base + int64_t(u) * kBlock;
                    if (i < nvec) w[u] = KEEP ? ld16_keep(g + i * kVec, policy) : ld16(g + i * kVec);
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (base + int64_t(u) * kBlock < nvec) vec(w[u]);
                after_iter();
            }
            done = nvec * kVec;
        }
        for (int64_t i = done + threadIdx.x; i < len; i += kBlock) elem(g[i]);
    }
}

// Deterministic fixed-tree reduction of one fp64 per thread to thread 0.
__device__ __forceinline__ double block_sum(double x) {
    __shared__ double warp_part[kBlock / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
    const int lane_id = threadIdx.x & 31, warp_id = threadIdx.x >> 5;
    if (lane_id == 0) warp_part[warp_id] = x;
    __syncthreads();
    double r = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < kBlock / 32; ++w) r += warp_part[w];
    __syncthreads();
    return r;
}

// Stage 1 of the global norm: one fp64 partial and one flag per CTA, over the
// norm's own partition (so the result depends only on the plan).
// Fast path: error-free fp32 group sums of the exact squares, two lanes
// packed (the low and the high bf16 of each word), flushed every 256
// elements.  A thread whose groups leave [2^-100, 2^100) (huge, tiny, inf or
// NaN gradients) recomputes its elements in fp64, which also decides the
// non-finite flag.
// The CTA's partial sum of squares and non-finite flag, written to
// partial[blockIdx.x] and flag[blockIdx.x].
// KEEP: load g with the evict-last L2 policy (the fused step reads it again).
// `pre`, when set, is chunk c0 already loaded.
template <bool KEEP = false>
__device__ __forceinline__ void norm_partial_cta(const ChunkPtr* __restrict__ chunks, int32_t c0,
                                                 int32_t c1, double* __restrict__ partial,
                                                 int32_t* __restrict__ flag,
                                                 const ChunkPtr* pre = nullptr) {
    Sum2F32x2 grp;
    double acc = 0.0;
    float err = 0.0f;
    bool in_range = true;
    uint32_t nz = 0;
    int rounds = 0;
    auto add_word = [&](uint32_t w) {
        const uint64_t x = bf16x2_to_f2(w);
        grp.add(f2_mul(x, x));
    };
    for_thread_grads<kNormUnroll, KEEP>(
        chunks, c0, c1,
        [&](const uint4& w) {
            nz |= (w.x | w.y | w.z | w.w) & 0x7fff7fffu;
            add_word(w.x);
            add_word(w.y);
            add_word(w.z);
            add_word(w.w);
        },
        [&](uint16_t h) {
            nz |= h & 0x7fffu;
            add_word(h);   // the high lane adds an exact zero
            in_range &= grp.flush(acc, err);
        },
        [&]() {
            if (++rounds == kNormFlushRounds) {   // 256 elements between flushes
                rounds = 0;
                in_range &= grp.flush(acc, err);
            }
        },
        pre);
    in_range &= grp.flush(acc, err);
    double tot = acc + double(err);
    bool bad = false;
    if (!in_range || (nz != 0 && tot < 0x1p-100)) {
        double exact = 0.0;
        for_thread_grads<1>(
            chunks, c0, c1,
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
            [&](uint16_t h) {
                const double x = from_bf16(h);
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

// ---- device-resident step path ----

// beta^t by binary exponentiation, lowest bit of t first, one IEEE fp64
// rounding per multiplication: the same operations as the host planner's.
__device__ double beta_power_dev(double beta, int64_t t) {
    double result = 1.0, square = beta;
    for (; t > 0; t >>= 1) {
        if (t & 1) result = __dmul_rn(result, square);
        square = __dmul_rn(square, square);
    }
    return result;
}

__device__ bool hparams_valid_dev(const adamw_hparams_t& hp) {
    const float f[6] = {hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.max_grad_norm};
    for (float x : f)
        if (!isfinite(x)) return false;
    return hp.lr >= 0.0f && hp.eps > 0.0f && hp.weight_decay >= 0.0f && hp.beta1 >= 0.0f &&
           hp.beta1 < 1.0f && hp.beta2 >= 0.0f && hp.beta2 < 1.0f;
}

// The same power from the squares of beta the exponentiation would compute
// (sq[i] = beta^(2^i)): one multiplication per set bit of t, lowest first,
// so the same roundings in the same order.
__device__ double beta_power_sq(const double* sq, int64_t t) {
    double result = 1.0;
    for (int i = 0; t > 0; ++i, t >>= 1)
        if (t & 1) result = __dmul_rn(result, sq[i]);
    return result;
}

// The host planner's make_scalars, operation for operation, in two halves
// that share nothing, so that two warps can evaluate them at once: part 0
// the beta1 side (step_size, omb1) plus the values copied or derived from lr,
// eps, weight_decay and max_grad_norm; part 1 the beta2 side (sbc2, omb2).
// With `sq` (that part's beta's squares) the power takes them from there.
__device__ __noinline__ void make_scalars_part(const adamw_hparams_t& hp, int64_t t, int part,
                                  StepScalars* out, const double* sq = nullptr) {
    if (part == 0) {
        const double b1 = hp.beta1;
        const double bc1 = __dsub_rn(1.0, sq ? beta_power_sq(sq, t) : beta_power_dev(b1, t));
        out->beta1 = hp.beta1;
        out->omb1 = __double2float_rn(__dsub_rn(1.0, b1));
        out->step_size = __double2float_rn(__ddiv_rn(double(hp.lr), bc1));
        out->eps = hp.eps;
        out->lrwd = __double2float_rn(__dmul_rn(double(hp.lr), double(hp.weight_decay)));
        out->max_grad_norm = hp.max_grad_norm;
    } else {
        const double b2 = hp.beta2;
        const double bc2 = __dsub_rn(1.0, sq ? beta_power_sq(sq, t) : beta_power_dev(b2, t));
        out->beta2 = hp.beta2;
        out->omb2 = __double2float_rn(__dsub_rn(1.0, b2));
        out->sbc2 = __double2float_rn(__dsqrt_rn(bc2));
    }
}

__device__ void make_scalars_dev(const adamw_hparams_t& hp, int64_t t, StepScalars* out) {
    make_scalars_part(hp, t, 0, out);
    make_scalars_part(hp, t, 1, out);
}

// Scalar memo (ScalarMemo): the key of (hp, t), and a lookup.
__device__ __forceinline__ void memo_key(const adamw_hparams_t& hp, int64_t t, uint32_t k[8]) {
    k[0] = __float_as_uint(hp.lr);
    k[1] = __float_as_uint(hp.beta1);
    k[2] = __float_as_uint(hp.beta2);
    k[3] = __float_as_uint(hp.eps);
    k[4] = __float_as_uint(hp.weight_decay);
    k[5] = __float_as_uint(hp.max_grad_norm);
    k[6] = uint32_t(uint64_t(t));
    k[7] = uint32_t(uint64_t(t) >> 32);
}

// Reads the hyperparameters, the applied-step counter and both memo slots
// with one load (or two) per lane of the calling warp -- one round trip to
// L2, few registers per lane; all were written by earlier kernels, so the
// reads go around L1 -- then picks the slot of t = *d_step + 1.  Every lane
// of the warp must call it; every lane gets *hp, *t and the result: whether
// the slot holds the scalars of (*hp, t), which are then in *out.
__device__ __forceinline__ bool memo_fetch_warp(const adamw_hparams_t* __restrict__ d_hp,
                                                const int64_t* __restrict__ d_step,
                                                const ScalarMemo* __restrict__ memo,
                                                adamw_hparams_t* hp, int64_t* t, StepScalars* out) {
    // words: [0, 6) hp, [6, 8) the counter, then kSlot words of each slot
    constexpr int kSlot = int((offsetof(ScalarMemo, valid) + sizeof(int32_t)) / sizeof(uint32_t));
    constexpr int kTotal = 8 + 2 * kSlot;
    static_assert(kTotal <= 64, "two words per lane");
    constexpr int kKey = int(offsetof(ScalarMemo, key) / sizeof(uint32_t));
    constexpr int kS = int(offsetof(ScalarMemo, s) / sizeof(uint32_t));
    constexpr int kValid = int(offsetof(ScalarMemo, valid) / sizeof(uint32_t));
    const int lane = threadIdx.x & 31;
    auto addr = [&](int i) -> const uint32_t* {
        if (i < 6) return reinterpret_cast<const uint32_t*>(d_hp) + i;
        if (i < 8) return reinterpret_cast<const uint32_t*>(d_step) + (i - 6);
        const int j = i - 8;
        return reinterpret_cast<const uint32_t*>(memo + j / kSlot) + j % kSlot;
    };
    const uint32_t w0 = __ldcg(addr(lane));
    const uint32_t w1 = (32 + lane < kTotal) ? __ldcg(addr(32 + lane)) : 0u;
    auto word = [&](int i) {  // word i of the concatenation, i the same in every lane
        return i < 32 ? __shfl_sync(0xffffffffu, w0, i) : __shfl_sync(0xffffffffu, w1, i - 32);
    };
    uint32_t h[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) h[i] = word(i);
    memcpy(hp, h, sizeof(h));
    *t = int64_t(uint64_t(word(6)) | (uint64_t(word(7)) << 32)) + 1;
    const int base = 8 + int(*t & 1) * kSlot;
    uint32_t k[8];
    memo_key(*hp, *t, k);
    bool hit = word(base + kValid) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) hit &= word(base + kKey + i) == k[i];
    uint32_t sw[sizeof(StepScalars) / sizeof(uint32_t)];
#pragma unroll
    for (int i = 0; i < int(sizeof(sw) / sizeof(uint32_t)); ++i) sw[i] = word(base + kS + i);
    if (hit) memcpy(out, sw, sizeof(StepScalars));
    return hit;
}

// Computes the scalars of (hp, t) with warps 0 and 1 of the CTA (one half
// each, see make_scalars_part) into shared *sh; every thread of the CTA
// must call it, and it ends with a barrier.
__device__ __forceinline__ void make_scalars_cta(const adamw_hparams_t& hp, int64_t t,
                                                 StepScalars* sh) {
    if (threadIdx.x == 0) make_scalars_part(hp, t, 0, sh);
    else if (threadIdx.x == 32) make_scalars_part(hp, t, 1, sh);
    __syncthreads();
}

// Writes the scalars of (hp, t), already in *s, into their memo slot (one
// thread; the scalars first, then the key, then the valid word).
__device__ __forceinline__ void memo_store(ScalarMemo* memo, const adamw_hparams_t& hp, int64_t t,
                                           const StepScalars& s) {
    ScalarMemo* m = memo + (t & 1);
    uint32_t k[8];
    memo_key(hp, t, k);
    m->valid = 0;
    m->s = s;
#pragma unroll
    for (int i = 0; i < 8; ++i) m->key[i] = k[i];
    m->valid = 1;
}

// The next step's scalars into the memo, from the squares table (built
// here first when the betas changed): warps 0 and 1 read the table's
// header and both rows in one round trip, then threads 0 and 32 evaluate
// the two halves at once.  Every thread of the CTA calls it; it ends with a
// barrier.  Only CTA 0 of a device-resident update calls it, so the table
// has no other reader or writer while it runs.
__device__ __noinline__ void memo_next(ScalarMemo* memo, const adamw_hparams_t& hp, int64_t t) {
    PowTable* tab = reinterpret_cast<PowTable*>(memo + 2);
    __shared__ double sq_sh[2][64];
    __shared__ int ok_sh;
    __shared__ StepScalars next_sh;
    const uint32_t b1 = __float_as_uint(hp.beta1), b2 = __float_as_uint(hp.beta2);
    if (threadIdx.x < 64) {
        const int row = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const double2 v = __ldcg(reinterpret_cast<const double2*>(tab->sq[row]) + lane);
        sq_sh[row][2 * lane] = v.x;
        sq_sh[row][2 * lane + 1] = v.y;
        if (threadIdx.x == 0)
            ok_sh = __ldcg(&tab->valid) != 0 && __ldcg(&tab->b1) == b1 && __ldcg(&tab->b2) == b2;
    }
    __syncthreads();
    if (!ok_sh) {
        // new betas: the squares, one row per thread, kept for later steps
        if ((threadIdx.x & 31) == 0 && threadIdx.x < 64) {
            double sq = threadIdx.x == 0 ? double(hp.beta1) : double(hp.beta2);
            double* row = sq_sh[threadIdx.x >> 5];
            for (int i = 0; i < 64; ++i) {
                row[i] = sq;
                sq = __dmul_rn(sq, sq);
            }
        }
        __syncthreads();
        if (threadIdx.x < 128) {
            const int row = threadIdx.x >> 6, i = threadIdx.x & 63;
            tab->sq[row][i] = sq_sh[row][i];
        }
        if (threadIdx.x == 0) {
            tab->b1 = b1;
            tab->b2 = b2;
            tab->valid = 1;
        }
    }
    if (threadIdx.x == 0) make_scalars_part(hp, t + 1, 0, &next_sh, sq_sh[0]);
    else if (threadIdx.x == 32) make_scalars_part(hp, t + 1, 1, &next_sh, sq_sh[1]);
    __syncthreads();
    if (threadIdx.x == 0) memo_store(memo, hp, t + 1, next_sh);
}

// ---- fused clipped step (one cooperative launch) ----
//
// For lists whose gradients fit in L2: stage 1 of the norm, a grid barrier,
// then every CTA sums all partials itself in the fixed order (no second
// barrier), decides clip or skip, and updates its share -- the second read
// of g comes from L2.  Needs every CTA resident at once (cooperative launch).
// The barrier is a monotonic 64-bit arrival counter: the CTA whose ticket is
// t waits until the counter reaches the next multiple of the grid.  The wait
// is bounded: a CTA that gives up sets *status and returns without updating.
#ifndef ADAMW_BARRIER_SLEEP_NS
#define ADAMW_BARRIER_SLEEP_NS 64
#endif
constexpr uint32_t kBarrierSleepNs = ADAMW_BARRIER_SLEEP_NS;
// rounds of the bounded wait: about a second, each round a sleep and one
// load from L2 (a few hundred nanoseconds)
constexpr uint32_t kBarrierSpins = uint32_t(1000000000ull / (kBarrierSleepNs + 256));

__device__ __forceinline__ unsigned long long load_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

}  // namespace
