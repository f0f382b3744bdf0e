// adamw_sm.cu -- sm_103a kernels and the device half of the C ABI.
//
// The step is a streaming elementwise update: per element it reads p, g, m, v
// and c (bf16 Kahan mode, 10 B), master, m, v and g (mixed mode, 14 B) or p,
// remainder, m, v and g (remainder mode, 14 B) and writes 8, 14 or 12 B back,
// with about twenty fp32 operations in between.
// That is far below the GPU's ridge point, so HBM bandwidth bounds it and the
// kernels are built to keep DRAM streaming: a persistent grid (SMs x resident
// CTAs) dealt 8K-element tiles of the flattened parameter space round-robin
// (so the grid sweeps every buffer together), chunk descriptors prefetched one
// ahead, 16-byte vector loads issued U vectors ahead of the arithmetic, fp32
// math, 16-byte stores.  No tensor cores: nothing here is a contraction.
//
// Arithmetic order follows the definition in include/adamw_sm.h exactly, with
// the IEEE round-to-nearest intrinsics (__fmul_rn, __fadd_rn, __fdiv_rn,
// __fsqrt_rn) so that no multiply-add is fused and every result is the one a
// strict host implementation of the same formula gives.
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

using namespace adamw;

namespace {

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
__device__ __forceinline__ void st16(void* p, uint4 v) {
    uint4* q = reinterpret_cast<uint4*>(p);
#if ADAMW_ST_POLICY == 1
    __stcs(q, v);
#else
    *q = v;
#endif
}

__device__ __forceinline__ bool bf16x2_nonfinite(uint32_t w) {
    return ((w & 0x7f80u) == 0x7f80u) || ((w & 0x7f800000u) == 0x7f800000u);
}

// Kernel flavours: plain step, clipped step (reads the norm finalize's
// output, skips on non-finite), plain step that also reports non-finite g.
enum Kind { kPlain = 0, kClip = 1, kReport = 2 };

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

// Vectors per thread in flight per stream, and the CTAs per SM the update
// kernel's register budget is fitted to (0: no constraint).
#ifndef ADAMW_UNROLL
#define ADAMW_UNROLL 2
#endif
#ifndef ADAMW_MIN_BLOCKS
#define ADAMW_MIN_BLOCKS 0
#endif
constexpr int kUnroll = ADAMW_UNROLL;

template <int K>
__device__ __forceinline__ void kahan_vec_chunk(const ChunkPtr& t, int64_t len,
                                                const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    uint16_t* v = static_cast<uint16_t*>(t.v);
    uint16_t* c = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * kUnroll) {
        uint4 G[kUnroll], P[kUnroll], M[kUnroll], V[kUnroll], C[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
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
        for (int u = 0; u < kUnroll; ++u) {
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

template <int K>
__device__ __forceinline__ void mixed_vec_chunk(const ChunkPtr& t, int64_t len,
                                                const StepScalars& s, float coef, bool& bad) {
    float* p = static_cast<float*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    float* m = static_cast<float*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* o = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * kUnroll) {
        uint4 G[kUnroll];
        F8 P[kUnroll], M[kUnroll], V[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld32(p + i * kVec);
                M[u] = ld32(m + i * kVec);
                V[u] = ld32(v + i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
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

template <int K>
__device__ __forceinline__ void plain_vec_chunk(const ChunkPtr& t, int64_t len,
                                                const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    uint16_t* v = static_cast<uint16_t*>(t.v);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * kUnroll) {
        uint4 G[kUnroll], P[kUnroll], M[kUnroll], V[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t i = base + int64_t(u) * kBlock;
            if (i < nvec) {
                G[u] = ld16(g + i * kVec);
                P[u] = ld16(p + i * kVec);
                M[u] = ld16(m + i * kVec);
                V[u] = ld16(v + i * kVec);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
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

template <int K>
__device__ __forceinline__ void kahan_v32_vec_chunk(const ChunkPtr& t, int64_t len,
                                                    const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    uint16_t* m = static_cast<uint16_t*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* c = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * kUnroll) {
        uint4 G[kUnroll], P[kUnroll], M[kUnroll], C[kUnroll];
        F8 V[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
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
        for (int u = 0; u < kUnroll; ++u) {
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

template <int K>
__device__ __forceinline__ void remainder_vec_chunk(const ChunkPtr& t, int64_t len,
                                                    const StepScalars& s, float coef, bool& bad) {
    uint16_t* p = static_cast<uint16_t*>(t.p);
    const uint16_t* g = static_cast<const uint16_t*>(t.g);
    float* m = static_cast<float*>(t.m);
    float* v = static_cast<float*>(t.v);
    uint16_t* r = static_cast<uint16_t*>(t.a);
    const int64_t nvec = len / kVec;
    for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * kUnroll) {
        uint4 G[kUnroll], P[kUnroll], R[kUnroll];
        F8 M[kUnroll], V[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
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
        for (int u = 0; u < kUnroll; ++u) {
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

// --------------------------------------------------------------- kernels --

// The update: CTA b walks chunks [cta_begin[b], cta_begin[b+1]).
#if ADAMW_MIN_BLOCKS > 0
#define ADAMW_UPDATE_BOUNDS __launch_bounds__(kBlock, ADAMW_MIN_BLOCKS)
#else
#define ADAMW_UPDATE_BOUNDS __launch_bounds__(kBlock)
#endif

// One chunk descriptor, read through the read-only path.
__device__ __forceinline__ ChunkPtr load_chunk(const ChunkPtr* c) {
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
}

// The update: CTA b walks chunks [cta_begin[b], cta_begin[b+1]), fetching the
// next chunk's descriptor before working on the current one.
template <int MODE, int K>
__device__ __forceinline__ void update_cta(const ChunkPtr* __restrict__ chunks, int32_t c0,
                                           int32_t c1, const StepScalars& s, float coef,
                                           bool& bad);

// DEV: the scalars, clip coefficient and skip decision come from the
// StepRecord the device-resident step path's prologue wrote.
template <int MODE, int K, bool DEV>
__global__ void ADAMW_UPDATE_BOUNDS
adamw_update_kernel(const ChunkPtr* __restrict__ chunks,
                    const int32_t* __restrict__ cta_begin, StepScalars s,
                    const NormOut* __restrict__ norm, int32_t* __restrict__ report,
                    const StepRecord* __restrict__ rec) {
    float coef = 1.0f;
    if (DEV) {
        if (rec->skip) return;        // skipped step: no writes at all
        s = rec->s;
        coef = rec->coef;
    } else if (K == kClip) {
        if (norm->nonfinite) return;  // skipped step: no writes at all
        coef = norm->coef;
    }
    bool bad = false;
    update_cta<MODE, K>(chunks, cta_begin[blockIdx.x], cta_begin[blockIdx.x + 1], s, coef, bad);
    if (K == kReport) {
        if (__syncthreads_or(bad) && threadIdx.x == 0) *report = 1;
    }
}

// ---- the CTA's share of the update: chunks [c0, c1), each chunk's
// descriptor fetched one ahead.
template <int MODE, int K>
__device__ __forceinline__ void update_cta(const ChunkPtr* __restrict__ chunks, int32_t c0,
                                           int32_t c1, const StepScalars& s, float coef,
                                           bool& bad) {
    ChunkPtr cur;
    if (c0 < c1) cur = load_chunk(chunks + c0);
    for (int32_t ci = c0; ci < c1; ++ci) {
        ChunkPtr nxt = cur;
        if (ci + 1 < c1) nxt = load_chunk(chunks + ci + 1);
        const int64_t len = cur.len2 >> 1;
        const bool vec = cur.len2 & 1;
        if (MODE == ADAMW_MODE_BF16_KAHAN) {
            if (vec) kahan_vec_chunk<K>(cur, len, s, coef, bad);
            else kahan_elem_chunk<K>(cur, len, s, coef, bad);
        } else if (MODE == ADAMW_MODE_MIXED_FP32_MASTER) {
            if (vec) mixed_vec_chunk<K>(cur, len, s, coef, bad);
            else mixed_elem_chunk<K>(cur, len, s, coef, bad);
        } else if (MODE == ADAMW_MODE_MIXED_BF16_REMAINDER) {
            if (vec) remainder_vec_chunk<K>(cur, len, s, coef, bad);
            else remainder_elem_chunk<K>(cur, len, s, coef, bad);
        } else if (MODE == ADAMW_MODE_BF16_PLAIN) {
            if (vec) plain_vec_chunk<K>(cur, len, s, coef, bad);
            else plain_elem_chunk<K>(cur, len, s, coef, bad);
        } else {
            if (vec) kahan_v32_vec_chunk<K>(cur, len, s, coef, bad);
            else kahan_v32_elem_chunk<K>(cur, len, s, coef, bad);
        }
        cur = nxt;
    }
}

// ------------------------------------------- bulk-copy staged update (A) --
//
// Mode A with the five input streams of each stage brought into shared
// memory by cp.async.bulk (one 1-D bulk copy per stream, completion counted
// on an mbarrier) instead of by per-thread 16-byte loads.  Thread 0 issues
// stage j + NS while the CTA computes stage j from shared memory; results
// go straight to global memory with 16-byte stores.  Every mbarrier wait is
// bounded: a wait that does not complete sets *err and the CTA returns.
#ifndef ADAMW_BULK
#define ADAMW_BULK 0
#endif
#if ADAMW_BULK
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
            atomicExch(err, 1);
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

// Error-free fp32 accumulation of non-negative terms: s + e is the exact sum
// of everything added since the last flush, up to the rounding of e itself.
// Squares of bf16 values are exact in fp32 for |g| in [2^-63, 2^64); for
// a >= b >= 0 the rounding error of a + b is exactly b - ((a + b) - a)
// (Dekker's Fast2Sum), so no bit of any square is lost; e collects those
// errors.  A group of at most 64 terms is flushed: s into an fp64 sum, e
// (at most 2^-18 of s) into an fp32 sum of the errors.
struct Sum2F32 {
    float s = 0.0f, e = 0.0f;
    __device__ __forceinline__ void add(float x) {
        const float a = fmaxf(s, x), b = fminf(s, x);
        const float t = __fadd_rn(a, b);
        e = __fadd_rn(e, __fsub_rn(b, __fsub_rn(t, a)));
        s = t;
    }
    // Adds the group to (acc, err) and restarts it; false when the group left
    // the range where squares are exact and sums finite.
    __device__ __forceinline__ bool flush(double& acc, float& err) {
        const bool ok = s < 0x1p100f;   // also false for inf and NaN
        acc += double(s);
        err = __fadd_rn(err, e);
        s = 0.0f;
        e = 0.0f;
        return ok;
    }
};

__device__ __forceinline__ float sq(float x) { return __fmul_rn(x, x); }

// Walks the g elements of one CTA's chunks that belong to this thread, in a
// fixed order: vec(w) gets 8 packed bf16, elem(h) one bf16, after_iter() runs
// after every group of U vectors.
template <int U, typename FV, typename FE, typename FI>
__device__ __forceinline__ void for_thread_grads(const ChunkPtr* __restrict__ chunks,
                                                 int32_t c0, int32_t c1, FV vec, FE elem,
                                                 FI after_iter) {
    for (int32_t ci = c0; ci < c1; ++ci) {
        const ChunkPtr ch = load_chunk(chunks + ci);
        const uint16_t* g = static_cast<const uint16_t*>(ch.g);
        const int64_t len = ch.len2 >> 1;
        int64_t done = 0;
        if (ch.len2 & 1) {
            const int64_t nvec = len / kVec;
            for (int64_t base = threadIdx.x; base < nvec; base += int64_t(kBlock) * U) {
                uint4 w[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t i = base + int64_t(u) * kBlock;
                    if (i < nvec) w[u] = ld16(g + i * kVec);
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
// same partition as the update (so the result depends only on the plan).
// Fast path: error-free fp32 group sums of the exact squares, flushed every
// 64 elements.  A thread whose groups leave [2^-100, 2^100) (huge, tiny,
// inf or NaN gradients) recomputes its elements in fp64, which also decides
// the non-finite flag.
__device__ __forceinline__ void norm_partial_cta(const ChunkPtr* __restrict__ chunks, int32_t c0,
                                                 int32_t c1, double* __restrict__ partial,
                                                 int32_t* __restrict__ flag);

__global__ void __launch_bounds__(kBlock)
norm_partial_kernel(const ChunkPtr* __restrict__ chunks,
                    const int32_t* __restrict__ cta_begin,
                    double* __restrict__ partial, int32_t* __restrict__ flag) {
    norm_partial_cta(chunks, cta_begin[blockIdx.x], cta_begin[blockIdx.x + 1], partial, flag);
}

// The CTA's partial sum of squares and non-finite flag, written to
// partial[blockIdx.x] and flag[blockIdx.x].
__device__ __forceinline__ void norm_partial_cta(const ChunkPtr* __restrict__ chunks, int32_t c0,
                                                 int32_t c1, double* __restrict__ partial,
                                                 int32_t* __restrict__ flag) {
    Sum2F32 grp;
    double acc = 0.0;
    float err = 0.0f;
    bool in_range = true;
    uint32_t nz = 0;
    for_thread_grads<8>(
        chunks, c0, c1,
        [&](const uint4& w) {
            nz |= (w.x | w.y | w.z | w.w) & 0x7fff7fffu;
            grp.add(sq(bf16_lo(w.x)));
            grp.add(sq(bf16_hi(w.x)));
            grp.add(sq(bf16_lo(w.y)));
            grp.add(sq(bf16_hi(w.y)));
            grp.add(sq(bf16_lo(w.z)));
            grp.add(sq(bf16_hi(w.z)));
            grp.add(sq(bf16_lo(w.w)));
            grp.add(sq(bf16_hi(w.w)));
        },
        [&](uint16_t h) {
            nz |= h & 0x7fffu;
            grp.add(sq(from_bf16(h)));
            in_range &= grp.flush(acc, err);
        },
        [&]() { in_range &= grp.flush(acc, err); });
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

// Stage 2: fixed-order fp64 sum of the partials, norm, clip coefficient.
__global__ void __launch_bounds__(kBlock)
norm_finalize_kernel(const double* __restrict__ partial, const int32_t* __restrict__ flag,
                     int32_t n, float max_grad_norm, NormOut* __restrict__ out,
                     double* __restrict__ user_norm, int32_t* __restrict__ user_flag) {
    double x = 0.0;
    bool bad = false;
    for (int32_t i = threadIdx.x; i < n; i += kBlock) {
        x += partial[i];
        bad |= flag[i] != 0;
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

// The host planner's make_scalars, operation for operation.
__device__ void make_scalars_dev(const adamw_hparams_t& hp, int64_t t, StepScalars* out) {
    const double b1 = hp.beta1, b2 = hp.beta2;
    const double bc1 = __dsub_rn(1.0, beta_power_dev(b1, t));
    const double bc2 = __dsub_rn(1.0, beta_power_dev(b2, t));
    out->beta1 = hp.beta1;
    out->beta2 = hp.beta2;
    out->omb1 = __double2float_rn(__dsub_rn(1.0, b1));
    out->omb2 = __double2float_rn(__dsub_rn(1.0, b2));
    out->step_size = __double2float_rn(__ddiv_rn(double(hp.lr), bc1));
    out->sbc2 = __double2float_rn(__dsqrt_rn(bc2));
    out->eps = hp.eps;
    out->lrwd = __double2float_rn(__dmul_rn(double(hp.lr), double(hp.weight_decay)));
    out->max_grad_norm = hp.max_grad_norm;
}

// One CTA, before the update: finalises the norm when n_partials > 0 (the
// same fixed-order reduction as norm_finalize_kernel), reads the
// hyperparameters and the applied-step counter from device memory, decides
// whether the step is skipped, writes the StepRecord, advances the counter
// for an applied step, and fills the caller's outputs (flag -1 for invalid
// hyperparameters).
__global__ void __launch_bounds__(kBlock)
step_prologue_kernel(const adamw_hparams_t* __restrict__ d_hp, int64_t* __restrict__ d_step,
                     StepRecord* __restrict__ rec, const double* __restrict__ partial,
                     const int32_t* __restrict__ flag, int32_t n_partials, int32_t clip,
                     NormOut* __restrict__ nout, double* __restrict__ user_norm,
                     int32_t* __restrict__ user_flag) {
    double x = 0.0;
    bool bad = false;
    for (int32_t i = threadIdx.x; i < n_partials; i += kBlock) {
        x += partial[i];
        bad |= flag[i] != 0;
    }
    const double tot = block_sum(x);
    const int any = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        const adamw_hparams_t hp = *d_hp;
        const bool valid = hparams_valid_dev(hp);
        const double norm = sqrt(tot);
        float coef = 1.0f;
        if (clip && valid && hp.max_grad_norm > 0.0f) {
            double c = double(hp.max_grad_norm) / (norm + 1e-6);
            if (c > 1.0) c = 1.0;
            coef = float(c);
        }
        StepRecord r{};
        r.skip = !valid ? 2 : (clip && any) ? 1 : 0;
        r.coef = coef;
        if (!r.skip) {
            const int64_t t = *d_step + 1;
            make_scalars_dev(hp, t, &r.s);
            *d_step = t;
        }
        *rec = r;
        if (n_partials > 0) {
            nout->norm = norm;
            nout->coef = coef;
            nout->nonfinite = any;
            if (user_norm) *user_norm = norm;
        }
        if (user_flag) *user_flag = !valid ? -1 : (n_partials > 0 ? any : 0);
    }
}

// ---- device-resident step without a norm pass: one launch ----
//
// Every CTA reads the hyperparameters and the step counter itself and
// computes the scalars (the host planner's fp64 operations); the last CTA to
// finish -- found with an arrival counter -- advances the counter and writes
// the non-finite flag, so no CTA can read a counter that was already
// advanced.  Invalid hyperparameters: nothing is updated, the flag is -1.
template <int MODE, int K>
__global__ void ADAMW_UPDATE_BOUNDS
adamw_update_self_kernel(const ChunkPtr* __restrict__ chunks, const int32_t* __restrict__ cta_begin,
                         const adamw_hparams_t* __restrict__ d_hp, int64_t* __restrict__ d_step,
                         unsigned int* __restrict__ done, int32_t* __restrict__ flagword,
                         int32_t* __restrict__ user_flag) {
    __shared__ StepScalars s_sh;
    __shared__ int valid_sh;
    __shared__ int64_t t_sh;
    if (threadIdx.x == 0) {
        const adamw_hparams_t hp = *d_hp;
        const int valid = hparams_valid_dev(hp);
        const int64_t t = __ldcg(d_step) + 1;
        if (valid) make_scalars_dev(hp, t, &s_sh);
        valid_sh = valid;
        t_sh = t;
    }
    __syncthreads();
    bool bad = false;
    if (valid_sh)
        update_cta<MODE, K>(chunks, cta_begin[blockIdx.x], cta_begin[blockIdx.x + 1], s_sh, 1.0f,
                            bad);
    const int any = (K == kReport) ? __syncthreads_or(bad) : 0;
    if (threadIdx.x == 0) {
        if (any) atomicOr(flagword, 1);
        __threadfence();
        if (atomicAdd(done, 1u) == gridDim.x - 1) {  // the last CTA
            __threadfence();
            const int32_t f = atomicExch(flagword, 0);
            if (valid_sh) *d_step = t_sh;
            if (user_flag) *user_flag = valid_sh ? f : -1;
            *done = 0;
        }
    }
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
constexpr uint32_t kBarrierSpins = 1u << 21;   // about a second with the sleeps

__device__ __forceinline__ unsigned long long load_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

template <int MODE>
__global__ void ADAMW_UPDATE_BOUNDS
adamw_fused_clip_kernel(const ChunkPtr* __restrict__ upd_chunks,
                        const int32_t* __restrict__ upd_begin,
                        const ChunkPtr* __restrict__ nrm_chunks,
                        const int32_t* __restrict__ nrm_begin, StepScalars s,
                        double* __restrict__ partial, int32_t* __restrict__ flag,
                        NormOut* __restrict__ nout, double* __restrict__ user_norm,
                        int32_t* __restrict__ user_flag, unsigned long long* __restrict__ arrivals,
                        int32_t* __restrict__ status) {
    __shared__ int passed;
    norm_partial_cta(nrm_chunks, nrm_begin[blockIdx.x], nrm_begin[blockIdx.x + 1], partial, flag);
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
            __nanosleep(256);
        }
        if (!ok) atomicExch(status, 1);
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
                            coef_sh, unused);
}

// The linear warm-up / linear decay schedule on the device: d_hp->lr for the
// update t = *d_step + 1, with the host function's fp64 operations.
__global__ void lr_linear_warmup_kernel(adamw_hparams_t* __restrict__ d_hp,
                                        const int64_t* __restrict__ d_step, float base_lr,
                                        int64_t warmup, int64_t total) {
    const int64_t k = *d_step;  // applied updates before this one
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
    int occ_bulk[3] = {0, 0, 0};
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

template <int MODE, int K>
const void* update_fn() { return reinterpret_cast<const void*>(&adamw_update_kernel<MODE, K, false>); }

int device_info(int dev, DeviceInfo* out) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (dev >= int(g_dev.size())) g_dev.resize(dev + 1);
    DeviceInfo& d = g_dev[dev];
    if (d.sms == 0) {
        int sms = 0;
        if (!cuda_ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                     "cudaDeviceGetAttribute"))
            return ADAMW_ERR_CUDA;
        const void* fns[kModes][3] = {
            {update_fn<0, kPlain>(), update_fn<0, kClip>(), update_fn<0, kReport>()},
            {update_fn<1, kPlain>(), update_fn<1, kClip>(), update_fn<1, kReport>()},
            {update_fn<2, kPlain>(), update_fn<2, kClip>(), update_fn<2, kReport>()},
            {update_fn<3, kPlain>(), update_fn<3, kClip>(), update_fn<3, kReport>()},
            {update_fn<4, kPlain>(), update_fn<4, kClip>(), update_fn<4, kReport>()}};
        for (int m = 0; m < kModes; ++m)
            for (int k = 0; k < 3; ++k)
                if (!cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ[m][k], fns[m][k],
                                                                           kBlock, 0),
                             "occupancy"))
                    return ADAMW_ERR_CUDA;
#if ADAMW_BULK
        {
            const void* bulk_fns[3] = {reinterpret_cast<const void*>(&adamw_update_bulk_kernel<kPlain>),
                                       reinterpret_cast<const void*>(&adamw_update_bulk_kernel<kClip>),
                                       reinterpret_cast<const void*>(&adamw_update_bulk_kernel<kReport>)};
            for (int k = 0; k < 3; ++k) {
                if (!cuda_ok(cudaFuncSetAttribute(bulk_fns[k],
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  int(kBulkSmem)), "cudaFuncSetAttribute") ||
                    !cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_bulk[k], bulk_fns[k],
                                                                           kBlock, kBulkSmem),
                             "occupancy"))
                    return ADAMW_ERR_CUDA;
            }
        }
#endif
        {
            const void* fused_fns[kModes] = {
                reinterpret_cast<const void*>(&adamw_fused_clip_kernel<0>),
                reinterpret_cast<const void*>(&adamw_fused_clip_kernel<1>),
                reinterpret_cast<const void*>(&adamw_fused_clip_kernel<2>),
                reinterpret_cast<const void*>(&adamw_fused_clip_kernel<3>),
                reinterpret_cast<const void*>(&adamw_fused_clip_kernel<4>)};
            for (int m = 0; m < kModes; ++m)
                if (!cuda_ok(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ_fused[m],
                                                                           fused_fns[m], kBlock, 0),
                             "occupancy"))
                    return ADAMW_ERR_CUDA;
            if (!cuda_ok(cudaDeviceGetAttribute(&d.cooperative, cudaDevAttrCooperativeLaunch, dev),
                         "cudaDeviceGetAttribute"))
                return ADAMW_ERR_CUDA;
        }
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

// One partition of the plan's list on the device: the chunk descriptors of
// `grid` CTAs and where each CTA's run of chunks begins.
struct DevPartition {
    int32_t grid = 0;
    int64_t n_chunks = 0;
    ChunkPtr* chunks = nullptr;
    int32_t* cta_begin = nullptr;
};

struct adamw_plan {
    int device = 0;
    int32_t mode = 0;
    int32_t flags = 0;
    int32_t n_tensors = 0;
    int64_t total = 0;
    int64_t scalar_elems = 0;
    void* block = nullptr;  // one device allocation holding everything below
    TensorDev* tensors = nullptr;  // the uploaded tensor table
    DevPartition upd;              // update kernel
    DevPartition nrm;              // norm partial kernel (its own grid)
    double* partial = nullptr;
    int32_t* flag = nullptr;
    NormOut* norm = nullptr;
    StepRecord* rec = nullptr;     // device-resident step path
    int32_t* status = nullptr;     // set by a kernel whose bounded wait ran out
    bool fused = false;            // clipped steps run as one cooperative launch
    unsigned long long* arrivals = nullptr;  // grid-barrier counter of the fused kernel
    unsigned int* done = nullptr;  // finished CTAs of a one-launch device step
    int32_t* flagword = nullptr;   // its non-finite flag, collected across CTAs
};

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

template <int MODE, int K, bool DEV>
cudaError_t launch_update(const adamw_plan* P, const StepScalars& s, int32_t* report,
                          cudaStream_t st) {
    adamw_update_kernel<MODE, K, DEV><<<P->upd.grid, kBlock, 0, st>>>(
        P->upd.chunks, P->upd.cta_begin, s, P->norm, report, P->rec);
    return cudaGetLastError();
}

#if ADAMW_BULK
template <int K>
cudaError_t launch_bulk(const adamw_plan* P, const StepScalars& s, int32_t* report,
                        cudaStream_t st) {
    adamw_update_bulk_kernel<K><<<P->upd.grid, kBlock, kBulkSmem, st>>>(
        P->upd.chunks, P->upd.cta_begin, s, P->norm, report, P->status);
    return cudaGetLastError();
}
#endif

template <bool DEV>
cudaError_t launch_update_any(const adamw_plan* P, int kind, const StepScalars& s,
                              int32_t* report, cudaStream_t st) {
#if ADAMW_BULK
    if (!DEV && P->mode == ADAMW_MODE_BF16_KAHAN) {
        if (kind == kPlain) return launch_bulk<kPlain>(P, s, report, st);
        if (kind == kClip) return launch_bulk<kClip>(P, s, report, st);
        return launch_bulk<kReport>(P, s, report, st);
    }
#endif
    if (P->mode == ADAMW_MODE_BF16_KAHAN) {
        if (kind == kPlain) return launch_update<0, kPlain, DEV>(P, s, report, st);
        if (kind == kClip) return launch_update<0, kClip, DEV>(P, s, report, st);
        return launch_update<0, kReport, DEV>(P, s, report, st);
    }
    if (P->mode == ADAMW_MODE_MIXED_FP32_MASTER) {
        if (kind == kPlain) return launch_update<1, kPlain, DEV>(P, s, report, st);
        if (kind == kClip) return launch_update<1, kClip, DEV>(P, s, report, st);
        return launch_update<1, kReport, DEV>(P, s, report, st);
    }
    if (P->mode == ADAMW_MODE_MIXED_BF16_REMAINDER) {
        if (kind == kPlain) return launch_update<2, kPlain, DEV>(P, s, report, st);
        if (kind == kClip) return launch_update<2, kClip, DEV>(P, s, report, st);
        return launch_update<2, kReport, DEV>(P, s, report, st);
    }
    if (P->mode == ADAMW_MODE_BF16_PLAIN) {
        if (kind == kPlain) return launch_update<3, kPlain, DEV>(P, s, report, st);
        if (kind == kClip) return launch_update<3, kClip, DEV>(P, s, report, st);
        return launch_update<3, kReport, DEV>(P, s, report, st);
    }
    if (kind == kPlain) return launch_update<4, kPlain, DEV>(P, s, report, st);
    if (kind == kClip) return launch_update<4, kClip, DEV>(P, s, report, st);
    return launch_update<4, kReport, DEV>(P, s, report, st);
}

template <int MODE, int K>
cudaError_t launch_self_mode(const adamw_plan* P, const adamw_hparams_t* d_hp, int64_t* d_step,
                             int32_t* user_flag, cudaStream_t st) {
    adamw_update_self_kernel<MODE, K><<<P->upd.grid, kBlock, 0, st>>>(
        P->upd.chunks, P->upd.cta_begin, d_hp, d_step, P->done, P->flagword, user_flag);
    return cudaGetLastError();
}

template <int K>
cudaError_t launch_self(const adamw_plan* P, const adamw_hparams_t* d_hp, int64_t* d_step,
                        int32_t* user_flag, cudaStream_t st) {
    switch (P->mode) {
        case 0: return launch_self_mode<0, K>(P, d_hp, d_step, user_flag, st);
        case 1: return launch_self_mode<1, K>(P, d_hp, d_step, user_flag, st);
        case 2: return launch_self_mode<2, K>(P, d_hp, d_step, user_flag, st);
        case 3: return launch_self_mode<3, K>(P, d_hp, d_step, user_flag, st);
        default: return launch_self_mode<4, K>(P, d_hp, d_step, user_flag, st);
    }
}

template <int MODE>
cudaError_t launch_fused_mode(const adamw_plan* P, const StepScalars& s, double* user_norm,
                              int32_t* user_flag, cudaStream_t st) {
    const ChunkPtr* uc = P->upd.chunks;
    const int32_t* ub = P->upd.cta_begin;
    const ChunkPtr* nc = P->nrm.chunks;
    const int32_t* nb = P->nrm.cta_begin;
    StepScalars sc = s;
    double* partial = P->partial;
    int32_t* flag = P->flag;
    NormOut* nout = P->norm;
    unsigned long long* arrivals = P->arrivals;
    int32_t* status = P->status;
    void* args[] = {&uc, &ub, &nc, &nb, &sc, &partial, &flag, &nout, &user_norm, &user_flag,
                    &arrivals, &status};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&adamw_fused_clip_kernel<MODE>),
                                       dim3(P->upd.grid), dim3(kBlock), args, 0, st);
}

cudaError_t launch_fused(const adamw_plan* P, const StepScalars& s, double* user_norm,
                         int32_t* user_flag, cudaStream_t st) {
    switch (P->mode) {
        case 0: return launch_fused_mode<0>(P, s, user_norm, user_flag, st);
        case 1: return launch_fused_mode<1>(P, s, user_norm, user_flag, st);
        case 2: return launch_fused_mode<2>(P, s, user_norm, user_flag, st);
        case 3: return launch_fused_mode<3>(P, s, user_norm, user_flag, st);
        default: return launch_fused_mode<4>(P, s, user_norm, user_flag, st);
    }
}

cudaError_t launch_norm(const adamw_plan* P, float max_grad_norm, double* user_norm,
                        int32_t* user_flag, cudaStream_t st) {
    norm_partial_kernel<<<P->nrm.grid, kBlock, 0, st>>>(P->nrm.chunks, P->nrm.cta_begin,
                                                        P->partial, P->flag);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    norm_finalize_kernel<<<1, kBlock, 0, st>>>(P->partial, P->flag, P->nrm.grid, max_grad_norm,
                                               P->norm, user_norm, user_flag);
    return cudaGetLastError();
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

    int occ = di.occ[mode][kPlain];
    for (int k = 0; k < 3; ++k) occ = occ < di.occ[mode][k] ? occ : di.occ[mode][k];
#if ADAMW_BULK
    if (mode == ADAMW_MODE_BF16_KAHAN)
        for (int k = 0; k < 3; ++k) occ = occ < di.occ_bulk[k] ? occ : di.occ_bulk[k];
#endif
    if (occ < 1) occ = 1;
    const int occ_norm = di.occ_norm > 0 ? di.occ_norm : 1;

    int64_t total = 0;
    for (int32_t k = 0; k < n_tensors; ++k) total += host_table[k].numel;
    // Lists whose gradients fit in half of L2 run clipped steps as one fused
    // cooperative launch (the norm pass leaves g in L2 for the update).
    const bool fused = (flags & ADAMW_PLAN_NORM) && !(flags & ADAMW_PLAN_NO_FUSE) &&
                       di.cooperative && di.occ_fused[mode] > 0 &&
                       total * 2 <= kFusedMaxGradBytes;
    if (fused) occ = occ < di.occ_fused[mode] ? occ : di.occ_fused[mode];
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
        rc = build_partition(host_table, n_tensors, mode, grid_norm, 0, &part_norm);
        if (rc != ADAMW_OK) return rc;
        chunk_pointers(host_table, mode, part_norm, &cp_norm);
    }

    adamw_plan* P = new adamw_plan();
    P->device = dev;
    P->mode = mode;
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
    const size_t o_d = off; off = align_up(off + 2 * sizeof(uint32_t), 256);

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
    P->done = reinterpret_cast<unsigned int*>(b + o_d);
    P->flagword = reinterpret_cast<int32_t*>(b + o_d + sizeof(uint32_t));
    P->fused = fused;

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
        if (!cuda_ok(launch_fused(plan, s, d_grad_norm, d_nonfinite, st), "fused launch"))
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
    if (!cuda_ok(launch_update_any<false>(plan, kind, s, report, st), "update launch"))
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
        const cudaError_t e = d_nonfinite ? launch_self<kReport>(plan, d_hp, d_step, d_nonfinite, st)
                                          : launch_self<kPlain>(plan, d_hp, d_step, nullptr, st);
        return cuda_ok(e, "update launch") ? ADAMW_OK : ADAMW_ERR_CUDA;
    }
    const bool norm_pass = want_norm && plan->nrm.grid > 0;
    if (norm_pass) {
        norm_partial_kernel<<<plan->nrm.grid, kBlock, 0, st>>>(plan->nrm.chunks, plan->nrm.cta_begin,
                                                               plan->partial, plan->flag);
        if (!cuda_ok(cudaGetLastError(), "norm launch")) return ADAMW_ERR_CUDA;
    }
    step_prologue_kernel<<<1, kBlock, 0, st>>>(d_hp, d_step, plan->rec, plan->partial, plan->flag,
                                               norm_pass ? plan->nrm.grid : 0, clip ? 1 : 0,
                                               plan->norm, d_grad_norm, d_nonfinite);
    if (!cuda_ok(cudaGetLastError(), "prologue launch")) return ADAMW_ERR_CUDA;
    if (want_norm && !norm_pass && d_grad_norm &&
        !cuda_ok(cudaMemsetAsync(d_grad_norm, 0, sizeof(double), st), "memset"))
        return ADAMW_ERR_CUDA;
    if (plan->upd.grid == 0) return ADAMW_OK;
    const int kind = clip ? kClip : (!want_norm && d_nonfinite) ? kReport : kPlain;
    int32_t* report = (kind == kReport) ? d_nonfinite : nullptr;
    if (!cuda_ok(launch_update_any<true>(plan, kind, StepScalars{}, report, st), "update launch"))
        return ADAMW_ERR_CUDA;
    return ADAMW_OK;
}

extern "C" int adamw_lr_linear_warmup_device(adamw_hparams_t* d_hp, const int64_t* d_step,
                                             float base_lr, int64_t warmup, int64_t total,
                                             adamw_stream_t stream) {
    if (!d_hp || !d_step || warmup < 0 || total < 0 || !std::isfinite(base_lr))
        return ADAMW_ERR_INVALID_ARG;
    lr_linear_warmup_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        d_hp, d_step, base_lr, warmup, total);
    return cuda_ok(cudaGetLastError(), "schedule launch") ? ADAMW_OK : ADAMW_ERR_CUDA;
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
        // a wait ran out: clear the word and realign the fused-step barrier
        // counter (no kernel of the plan is running after the synchronise)
        const int32_t zero = 0;
        const unsigned long long start = 0;
        if (!cuda_ok(cudaMemcpy(plan->status, &zero, sizeof(int32_t), cudaMemcpyHostToDevice),
                     "cudaMemcpy(status)") ||
            !cuda_ok(cudaMemcpy(plan->arrivals, &start, sizeof(start), cudaMemcpyHostToDevice),
                     "cudaMemcpy(arrivals)"))
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
// file-scope __device__ array (the uploaded tensor list, the per-CTA partials
// and flags, and the finalize record), so a call allocates nothing.  Every GPU
// that loads this library holds the array until the process exits.

namespace {

constexpr int kNoAllocMaxCtas = 1024;
constexpr size_t kNoAllocTableOff = 0;
constexpr size_t kNoAllocPartialOff =
    (sizeof(adamw_tensor_t) * ADAMW_NOALLOC_MAX_TENSORS + 255) / 256 * 256;
constexpr size_t kNoAllocFlagOff = kNoAllocPartialOff + sizeof(double) * kNoAllocMaxCtas;
constexpr size_t kNoAllocOutOff = kNoAllocFlagOff + sizeof(int32_t) * kNoAllocMaxCtas;
constexpr size_t kNoAllocBytes = (kNoAllocOutOff + sizeof(NormOut) + 255) / 256 * 256;

// The scratch (about 208 KiB).  Host code never uses this name as an address:
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

// Stage 1 without a chunk table: tensor by tensor in list order, every thread
// of the grid takes a fixed share of each tensor (an element of the head that
// 16-byte aligns g, vectors strided by the whole grid, an element of the
// tail).  Sums as in norm_partial_kernel: error-free fp32 groups of exact
// squares, an fp64 recomputation for threads whose groups leave the safe range.
__global__ void __launch_bounds__(kBlock)
norm_partial_noalloc_kernel(const adamw_tensor_t* __restrict__ table, int32_t n,
                            double* __restrict__ partial, int32_t* __restrict__ flag) {
    const int64_t gt = int64_t(blockIdx.x) * kBlock + threadIdx.x;
    const int64_t T = int64_t(gridDim.x) * kBlock;
    constexpr int U = 4;

    auto walk = [&](auto vec, auto elem, auto after_iter) {
        for (int32_t k = 0; k < n; ++k) {
            const uint16_t* g = static_cast<const uint16_t*>(table[k].grad);
            const int64_t len = table[k].numel;
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

    Sum2F32 grp;
    double acc = 0.0;
    float err = 0.0f;
    bool in_range = true;
    uint32_t nz = 0;
    walk(
        [&](const uint4& w) {
            nz |= (w.x | w.y | w.z | w.w) & 0x7fff7fffu;
            grp.add(sq(bf16_lo(w.x)));
            grp.add(sq(bf16_hi(w.x)));
            grp.add(sq(bf16_lo(w.y)));
            grp.add(sq(bf16_hi(w.y)));
            grp.add(sq(bf16_lo(w.z)));
            grp.add(sq(bf16_hi(w.z)));
            grp.add(sq(bf16_lo(w.w)));
            grp.add(sq(bf16_hi(w.w)));
        },
        [&](uint16_t hb) {
            nz |= hb & 0x7fffu;
            grp.add(sq(from_bf16(hb)));
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
    adamw_tensor_t* table = reinterpret_cast<adamw_tensor_t*>(d.base + kNoAllocTableOff);
    double* partial = reinterpret_cast<double*>(d.base + kNoAllocPartialOff);
    int32_t* flag = reinterpret_cast<int32_t*>(d.base + kNoAllocFlagOff);
    NormOut* out = reinterpret_cast<NormOut*>(d.base + kNoAllocOutOff);
    // Every CTA writes its partial and flag and the finalize writes the
    // record on every call, so nothing in the scratch has to start at zero.
    if (n_tensors > 0 &&
        !cuda_ok(cudaMemcpyAsync(table, host_table, sizeof(adamw_tensor_t) * size_t(n_tensors),
                                 cudaMemcpyHostToDevice, st), "cudaMemcpyAsync(table)"))
        return ADAMW_ERR_CUDA;
    norm_partial_noalloc_kernel<<<d.grid, kBlock, 0, st>>>(table, n_tensors, partial, flag);
    if (!cuda_ok(cudaGetLastError(), "norm launch")) return ADAMW_ERR_CUDA;
    norm_finalize_kernel<<<1, kBlock, 0, st>>>(partial, flag, d.grid, 0.0f, out, d_grad_norm,
                                               d_nonfinite);
    if (!cuda_ok(cudaGetLastError(), "finalize launch")) return ADAMW_ERR_CUDA;
    return ADAMW_OK;
}
