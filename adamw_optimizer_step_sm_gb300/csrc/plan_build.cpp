// plan_build.cpp -- host-side planning for the multi-tensor AdamW step:
// argument validation, the per-step fp32 scalars, and the partition of a
// tensor list into per-CTA chunks.  Pure host code; needs no GPU.
//
// The pages name the multi-tensor optimizer only ("Distributed optimizer
// support for BERT", NeMo PR #5305, "Usage": fused_adam / distributed_fused_adam
// update a whole model's parameter list in fused launches); this partition is
// this library's own design.  Every CTA of a persistent grid gets the same
// number of elements whatever the tensor sizes: large lists are cut into
// tiles of about 8K elements on 2048-element boundaries of the flattened list
// and dealt round-robin (the grid sweeps the buffers together), small lists
// and the norm pass into one contiguous range per CTA.
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "adamw_internal.h"

namespace adamw {

namespace {

thread_local std::string g_cuda_error;

bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Elements [0, head) take the element path so that every base is 16-byte
// aligned at `head`; -1 when no head < kVec does that.
int vector_head(const adamw_tensor_t& t, int32_t mode) {
    int64_t es[5];
    element_sizes(mode, es);
    const void* ptrs[5] = {t.param, t.grad, t.exp_avg, t.exp_avg_sq, t.aux};
    for (int h = 0; h < kVec; ++h) {
        bool ok = true;
        for (int s = 0; s < 5 && ok; ++s)
            ok = ((reinterpret_cast<uintptr_t>(ptrs[s]) + uintptr_t(h * es[s])) % 16) == 0;
        if (ok) return h;
    }
    return -1;
}

}  // namespace

void element_sizes(int32_t mode, int64_t es[5]) {
    // param, grad, exp_avg, exp_avg_sq, aux (0: aux unused)
    static const int64_t table[5][5] = {
        {2, 2, 2, 2, 2},  // bf16 Kahan
        {4, 2, 4, 4, 2},  // mixed fp32 master
        {2, 2, 4, 4, 2},  // mixed bf16 + remainder
        {2, 2, 2, 2, 0},  // bf16 without compensation
        {2, 2, 2, 4, 2},  // bf16 Kahan, fp32 variance
    };
    if (mode >= ADAMW_MODE_ANYPREC) {
        es[0] = 2;
        es[1] = 2;
        es[2] = (mode & ADAMW_ANYPREC_M_FP32) ? 4 : 2;
        es[3] = (mode & ADAMW_ANYPREC_V_FP32) ? 4 : 2;
        es[4] = (mode & ADAMW_ANYPREC_NO_KAHAN) ? 0 : (mode & ADAMW_ANYPREC_C_FP32) ? 4 : 2;
        return;
    }
    for (int s = 0; s < 5; ++s) es[s] = table[mode][s];
}

int mode_variant(int32_t mode) {
    if (mode >= 0 && mode < 5) return mode;
    if (mode < ADAMW_MODE_ANYPREC || mode >= 2 * ADAMW_MODE_ANYPREC) return -1;
    if ((mode & ADAMW_ANYPREC_NO_KAHAN) && (mode & ADAMW_ANYPREC_C_FP32)) return -1;
    if (mode == ADAMW_MODE_ANYPREC) return ADAMW_MODE_BF16_KAHAN;
    if (mode == (ADAMW_MODE_ANYPREC | ADAMW_ANYPREC_V_FP32)) return ADAMW_MODE_BF16_KAHAN_FP32_VAR;
    if (mode == (ADAMW_MODE_ANYPREC | ADAMW_ANYPREC_NO_KAHAN)) return ADAMW_MODE_BF16_PLAIN;
    for (int k = 5; k < kModes; ++k)
        if (kVariantModes[k] == mode) return k;
    return -1;
}

bool valid_mode(int32_t mode) { return mode_variant(mode) >= 0; }

void set_cuda_error(const char* where, const char* what) {
    g_cuda_error = std::string(where) + ": " + what;
}

const char* last_cuda_error() { return g_cuda_error.c_str(); }

int validate_table(const adamw_tensor_t* table, int32_t n, int32_t mode) {
    if (n < 0) return ADAMW_ERR_INVALID_ARG;
    if (n > 0 && !table) return ADAMW_ERR_INVALID_ARG;
    if (!valid_mode(mode)) return ADAMW_ERR_INVALID_ARG;
    int64_t es[5];
    element_sizes(mode, es);
    for (int32_t k = 0; k < n; ++k) {
        const adamw_tensor_t& t = table[k];
        if (t.numel < 0) return ADAMW_ERR_INVALID_ARG;
        if (t.numel == 0) continue;
        const void* ptrs[5] = {t.param, t.grad, t.exp_avg, t.exp_avg_sq, t.aux};
        for (int s = 0; s < 5; ++s) {
            if (es[s] == 0) continue;  // a buffer the mode does not use
            if (!ptrs[s]) return ADAMW_ERR_INVALID_ARG;
            if (!aligned(ptrs[s], uintptr_t(es[s]))) return ADAMW_ERR_MISALIGNED;
        }
    }
    return ADAMW_OK;
}

int validate_hparams(const adamw_hparams_t* hp, int64_t step) {
    if (!hp || step < 1) return ADAMW_ERR_INVALID_ARG;
    const float f[6] = {hp->lr, hp->beta1, hp->beta2, hp->eps,
                        hp->weight_decay, hp->max_grad_norm};
    for (float x : f)
        if (!std::isfinite(x)) return ADAMW_ERR_INVALID_ARG;
    if (hp->lr < 0.0f || hp->eps <= 0.0f || hp->weight_decay < 0.0f)
        return ADAMW_ERR_INVALID_ARG;
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f)) return ADAMW_ERR_INVALID_ARG;
    if (!(hp->beta2 >= 0.0f && hp->beta2 < 1.0f)) return ADAMW_ERR_INVALID_ARG;
    return ADAMW_OK;
}

// beta^t by binary exponentiation (fp64 multiplications only, lowest bit of
// t first), so the device-resident step path reproduces it exactly.
double beta_power(double beta, int64_t t) {
    double result = 1.0, square = beta;
    for (; t > 0; t >>= 1) {
        if (t & 1) result *= square;
        square *= square;
    }
    return result;
}

// Bias corrections of Kingma & Ba and the decoupled decay factor of
// Loshchilov & Hutter, in fp64 from the fp32 hyperparameters, each rounded
// once to fp32.
int make_scalars(const adamw_hparams_t* hp, int64_t step, StepScalars* out) {
    int rc = validate_hparams(hp, step);
    if (rc != ADAMW_OK) return rc;
    const double b1 = hp->beta1, b2 = hp->beta2;
    const double bc1 = 1.0 - beta_power(b1, step);
    const double bc2 = 1.0 - beta_power(b2, step);
    out->beta1 = hp->beta1;
    out->beta2 = hp->beta2;
    out->omb1 = float(1.0 - b1);
    out->omb2 = float(1.0 - b2);
    out->step_size = float(double(hp->lr) / bc1);
    out->sbc2 = float(std::sqrt(bc2));
    out->eps = hp->eps;
    out->lrwd = float(double(hp->lr) * double(hp->weight_decay));
    out->max_grad_norm = hp->max_grad_norm;
    return ADAMW_OK;
}

int32_t choose_grid(int64_t total, int32_t max_grid) {
    if (total <= 0) return 0;
    if (max_grid < 1) max_grid = 1;
    int64_t want = (total + kMinElemsPerCta - 1) / kMinElemsPerCta;
    return int32_t(want < max_grid ? want : max_grid);
}

int64_t update_tile_elems(int64_t total, int32_t grid) {
    if (kTileElems <= 0 || grid <= 0) return 0;
    const int64_t row = int64_t(grid) * kTileElems;
    if (total < 2 * row) return 0;
    // fewer than kDynMinRounds rounds: the small tile
    if ((total + row / 2) / row < kDynMinRounds) return kSmallTileElems;
    return kTileElems;
}

TileSchedule::TileSchedule(int64_t total, int32_t grid_, int64_t tile_elems, int64_t relief_elems)
    : grid(grid_) {
    // k rounds, the whole number nearest to total / (grid * tile_elems)
    const int64_t per_row = int64_t(grid) * tile_elems;
    k = (total + per_row / 2) / per_row;
    if (k < 1) k = 1;
    // quotas in units of kBalanceAlign elements: CTA 0 short by the relief,
    // the others equal to one unit
    const int64_t units = (total + kBalanceAlign - 1) / kBalanceAlign;
    if (grid == 1) {
        q0 = units;
    } else {
        const int64_t even = units / grid, relief = relief_elems / kBalanceAlign;
        q0 = even > relief ? even - relief : 0;
        base = (units - q0) / (grid - 1);
        extra = (units - q0) % (grid - 1);
    }
    // no round without a cut-aligned unit for every CTA but CTA 0
    const int64_t min_whole = (grid == 1 ? q0 : base) / (kCutAlign / kBalanceAlign);
    if (k > min_whole) k = min_whole > 1 ? min_whole : 1;
}

int64_t TileSchedule::size(int64_t j) const {
    const int64_t r = j / grid, b = j % grid;
    const int64_t q = b == 0 ? q0 : base + (b - 1 < extra ? 1 : 0);   // quota, balance units
    constexpr int64_t per_cut = kCutAlign / kBalanceAlign;
    const int64_t whole = q / per_cut, rest = q % per_cut;  // cut-aligned units + leftover
    int64_t sz = (whole / k + (r < whole % k ? 1 : 0)) * kCutAlign;
    if (r == k - 1) sz += rest * kBalanceAlign;
    return sz;
}

int build_partition(const adamw_tensor_t* table, int32_t n, int32_t mode,
                    int32_t grid, int64_t tile_elems, Partition* out, int64_t relief) {
    int rc = validate_table(table, n, mode);
    if (rc != ADAMW_OK) return rc;
    if (!out || grid < 0 || tile_elems < 0 || tile_elems % kVec || relief < 0 ||
        relief % kBalanceAlign)
        return ADAMW_ERR_INVALID_ARG;
    Partition& P = *out;
    P = Partition();
    for (int32_t k = 0; k < n; ++k) P.total += table[k].numel;
    if (P.total > 0 && grid == 0) return ADAMW_ERR_INVALID_ARG;

    // Segments: per tensor an optional element-path head, then a vector body
    // (or the whole tensor on the element path when no head aligns it).
    struct Seg { int32_t k; int32_t vec; int64_t off, len; };
    std::vector<Seg> segs;
    for (int32_t k = 0; k < n; ++k) {
        const int64_t len = table[k].numel;
        if (len == 0) continue;
        int h = vector_head(table[k], mode);
        if (h < 0 || h >= len) {
            segs.push_back({k, 0, 0, len});
            P.scalar_elems += len;
        } else {
            if (h > 0) {
                segs.push_back({k, 0, 0, h});
                P.scalar_elems += h;
            }
            segs.push_back({k, 1, h, len - h});
        }
    }

    P.cta_begin.assign(size_t(grid) + 1, 0);
    if (P.total == 0) return ADAMW_OK;

#if !ADAMW_TILE_BALANCE
    if (tile_elems > 0) {
        // Interleaved, fixed tiles: cut every segment into tiles of
        // tile_elems and deal the tiles round-robin to the CTAs in list order.
        std::vector<ChunkDev> pieces;
        for (const Seg& s : segs)
            for (int64_t pos = 0; pos < s.len; pos += tile_elems)
                pieces.push_back({s.k, s.vec, s.off + pos,
                                  (s.len - pos < tile_elems) ? s.len - pos : tile_elems});
        std::vector<int64_t> count(size_t(grid) + 1, 0);
        for (size_t j = 0; j < pieces.size(); ++j) ++count[j % grid + 1];
        for (int32_t b = 0; b < grid; ++b) count[b + 1] += count[b];
        P.chunks.resize(pieces.size());
        P.chunk_cta.resize(pieces.size());
        std::vector<int64_t> fill(count.begin(), count.end() - 1);
        for (size_t j = 0; j < pieces.size(); ++j) {
            const int32_t b = int32_t(j % grid);
            P.chunks[fill[b]] = pieces[j];
            P.chunk_cta[fill[b]] = b;
            ++fill[b];
        }
        for (int32_t b = 0; b <= grid; ++b) P.cta_begin[b] = int32_t(count[b]);
        return ADAMW_OK;
    }
#endif
    if (tile_elems > 0) {
        // Interleaved: cut the flattened list (all segments in order) into
        // tiles of about tile_elems and deal them round-robin to the CTAs, so that
        // at any moment the whole grid streams one narrow window of each
        // buffer.  A tile that spans a tensor boundary is several chunks of
        // one CTA.  A cut inside a vector body moves up to the next multiple
        // of kCutAlign elements from the body's start (a whole number of
        // 16-byte vectors; coarser alignment keeps warps' accesses on whole
        // cache lines) and the next tile is shorter by as much.
        // Tile j (round j / grid, CTA j % grid) is sched.size(j) long, so
        // every CTA's tiles add up to its quota (CTA 0's `relief` short, the
        // others' equal) within kBalanceAlign elements.  Cuts that end a
        // tile of the last round move up to
        // kBalanceAlign only (there the quota's leftover is taken), all
        // others to kCutAlign.
        //
        // With kDynTail (and at least kDynMinRounds rounds) the last rounds
        // (kDynSharePct percent of k, at least one, never all) are not
        // dealt: from there on the list is cut into tiles (owner -1) that
        // the CTAs claim at run time, of tile_elems, or with kDynGuided of
        // the work left over twice the grid, rounded up to kCutAlign and
        // capped at tile_elems.
        const TileSchedule sched(P.total, grid, tile_elems, relief);
        const bool dyn = kDynTail && sched.k >= 2 && sched.k >= kDynMinRounds;
        int64_t claim_rounds = (sched.k * kDynSharePct + 99) / 100;
        if (claim_rounds < 1) claim_rounds = 1;
        if (claim_rounds > sched.k - 1) claim_rounds = sched.k - 1;
        const int64_t n_dealt = dyn ? (sched.k - claim_rounds) * int64_t(grid) : INT64_MAX;
        const int64_t two_grids = 2 * int64_t(grid);
        auto size_of = [&](int64_t j, int64_t start) {
            if (j < n_dealt) return sched.size(j);
            if (!kDynGuided) return tile_elems;
            const int64_t left = P.total - start;
            const int64_t want = left > 0 ? (left + two_grids - 1) / two_grids : 0;
            const int64_t sz = (want + kCutAlign - 1) / kCutAlign * kCutAlign;
            return sz < kCutAlign ? kCutAlign : sz > tile_elems ? tile_elems : sz;
        };
        std::vector<ChunkDev> pieces;
        std::vector<int32_t> owner;
        int64_t flat = 0, tile = 0, boundary = size_of(0, 0);
        for (const Seg& s : segs) {
            int64_t pos = 0;
            while (pos < s.len) {
                int64_t take = s.len - pos;
                if (take > boundary - flat) {
                    take = boundary - flat;
                    const int64_t align =
                        (!dyn && sched.last_round(tile)) ? kBalanceAlign : kCutAlign;
                    if (s.vec) take = (pos + take + align - 1) / align * align - pos;
                    if (take > s.len - pos) take = s.len - pos;
                }
                pieces.push_back({s.k, s.vec, s.off + pos, take});
                owner.push_back(tile < n_dealt ? int32_t(tile % grid) : -1);
                pos += take;
                flat += take;
                while (flat >= boundary) {
                    ++tile;
                    boundary += size_of(tile, boundary);
                }
            }
        }
        // every CTA's own chunks in CTA order, then the claimable ones
        std::vector<int64_t> count(size_t(grid) + 2, 0);
        for (int32_t b : owner) ++count[size_t(b < 0 ? grid : b) + 1];
        for (int32_t b = 0; b <= grid; ++b) count[b + 1] += count[b];
        P.chunks.resize(pieces.size());
        P.chunk_cta.resize(pieces.size());
        std::vector<int64_t> fill(count.begin(), count.end() - 1);
        for (size_t j = 0; j < pieces.size(); ++j) {
            const int32_t b = owner[j] < 0 ? grid : owner[j];
            P.chunks[fill[b]] = pieces[j];
            P.chunk_cta[fill[b]] = owner[j];
            ++fill[b];
        }
        for (int32_t b = 0; b <= grid; ++b) P.cta_begin[b] = int32_t(count[b]);
        P.n_dyn = count[size_t(grid) + 1] - count[size_t(grid)];
        // every claim (one per claimable chunk, plus each CTA's last, empty
        // one) is counted in the claim field of the sync word
        if (uint64_t(P.n_dyn) + uint64_t(grid) > kSyncClaimMask) return ADAMW_ERR_TOO_LARGE;
        return ADAMW_OK;
    }

    // Contiguous: an even split of the flattened element space, CTA 0's
    // share `relief` short (never below zero); cuts inside a vector body
    // fall on multiples of kVec from the body's start so every chunk of it
    // starts 16-byte aligned.
    // Shares in whole vectors: CTA 0's the even share less the relief, the
    // others' the rest dealt out so that they differ by one vector at most.
    const int64_t vecs = (P.total + kVec - 1) / kVec;
    const int64_t even = (vecs + grid - 1) / grid, relief_v = relief / kVec;
    const int64_t v0 = grid == 1 ? vecs : even > relief_v ? even - relief_v : 0;
    const int64_t per = grid == 1 ? 0 : (vecs - v0) / (grid - 1);
    const int64_t extra = grid == 1 ? 0 : (vecs - v0) % (grid - 1);
    auto want_of = [&](int32_t b) {
        return (b == 0 ? v0 : per + (b - 1 < extra ? 1 : 0)) * kVec;
    };
    int32_t cta = 0;
    int64_t filled = 0;
    for (const Seg& s : segs) {
        int64_t pos = 0;
        while (pos < s.len) {
            const int64_t want = want_of(cta);
            if (filled >= want && cta < grid - 1) {
                ++cta;
                filled = 0;
                continue;
            }
            int64_t take = s.len - pos;
            if (cta < grid - 1 && take > want - filled) {
                int64_t cap = want - filled;
                take = s.vec ? (cap + kVec - 1) / kVec * kVec : cap;
                if (take > s.len - pos) take = s.len - pos;
            }
            P.chunks.push_back({s.k, s.vec, s.off + pos, take});
            P.chunk_cta.push_back(cta);
            pos += take;
            filled += take;
        }
    }
    // cta_begin[b] = first chunk of CTA b (chunks are emitted in CTA order).
    size_t c = 0;
    for (int32_t b = 0; b <= grid; ++b) {
        while (c < P.chunks.size() && P.chunk_cta[c] < b) ++c;
        P.cta_begin[b] = int32_t(c);
    }
    return ADAMW_OK;
}

void chunk_pointers(const adamw_tensor_t* table, int32_t mode, const Partition& P,
                    std::vector<ChunkPtr>* out) {
    int64_t es[5];
    element_sizes(mode, es);
    out->resize(P.chunks.size());
    for (size_t i = 0; i < P.chunks.size(); ++i) {
        const ChunkDev& c = P.chunks[i];
        const adamw_tensor_t& t = table[c.tensor];
        auto at = [&](const void* base, int64_t es) {
            return static_cast<void*>(static_cast<char*>(const_cast<void*>(base)) + c.off * es);
        };
        ChunkPtr& d = (*out)[i];
        d.p = at(t.param, es[0]);
        d.g = at(t.grad, es[1]);
        d.m = at(t.exp_avg, es[2]);
        d.v = at(t.exp_avg_sq, es[3]);
        d.a = es[4] ? at(t.aux, es[4]) : nullptr;
        d.len2 = 2 * c.len + c.vec;
#if ADAMW_CHECK_BOUNDS
        const void* bases[5] = {t.param, t.grad, t.exp_avg, t.exp_avg_sq, t.aux};
        for (int s = 0; s < 5; ++s) {
            d.lo[s] = es[s] ? bases[s] : nullptr;
            d.hi[s] = es[s] ? static_cast<const char*>(bases[s]) + t.numel * es[s] : nullptr;
        }
        d.status = nullptr;   // set when the plan's device block exists
        d.pad_ = 0;
#endif
    }
}

}  // namespace adamw

// ------------------------------------------------------- host-only ABI ----

extern "C" int adamw_plan_chunks(const adamw_tensor_t* host_table,
                                 int32_t n_tensors, int32_t mode, int32_t grid,
                                 adamw_chunk_t* out, int64_t cap,
                                 int64_t* n_out) {
    if (!n_out || cap < 0 || (cap > 0 && !out) || grid < 1)
        return ADAMW_ERR_INVALID_ARG;
    int rc = adamw::validate_table(host_table, n_tensors, mode);
    if (rc != ADAMW_OK) return rc;
    int64_t total = 0;
    for (int32_t k = 0; k < n_tensors; ++k) total += host_table[k].numel;
    adamw::Partition P;
    rc = adamw::build_partition(host_table, n_tensors, mode, grid,
                                adamw::update_tile_elems(total, grid), &P);
    if (rc != ADAMW_OK) return rc;
    *n_out = int64_t(P.chunks.size());
    if (int64_t(P.chunks.size()) > cap) return ADAMW_ERR_TOO_LARGE;
    for (size_t i = 0; i < P.chunks.size(); ++i) {
        out[i].tensor = P.chunks[i].tensor;
        out[i].vec = P.chunks[i].vec;
        out[i].offset = P.chunks[i].off;
        out[i].len = P.chunks[i].len;
        out[i].cta = P.chunk_cta[i];
        out[i].pad_ = 0;
    }
    return ADAMW_OK;
}

extern "C" int adamw_step_scalars(const adamw_hparams_t* hp, int64_t step,
                                  float out5[5]) {
    if (!out5) return ADAMW_ERR_INVALID_ARG;
    adamw::StepScalars s;
    int rc = adamw::make_scalars(hp, step, &s);
    if (rc != ADAMW_OK) return rc;
    out5[0] = s.step_size;
    out5[1] = s.sbc2;
    out5[2] = s.omb1;
    out5[3] = s.omb2;
    out5[4] = s.lrwd;
    return ADAMW_OK;
}

// The recipe's linear schedule ("--lr_scheduler_type linear --warmup_steps
// W"): the update with k = step - 1 applied updates before it uses
// lr * k / max(1, W) while k < W, then lr * max(0, (T - k) / max(1, T - W)).
extern "C" float adamw_lr_linear_warmup(float base_lr, int64_t step, int64_t warmup,
                                        int64_t total) {
    if (step < 1 || warmup < 0 || total < 0) return 0.0f;
    const int64_t k = step - 1;
    double f;
    if (k < warmup) {
        f = double(k) / double(warmup > 1 ? warmup : 1);
    } else {
        const double span = double((total - warmup) > 1 ? (total - warmup) : 1);
        f = double(total - k) / span;
        if (f < 0.0) f = 0.0;
    }
    return float(double(base_lr) * f);
}

extern "C" const char* adamw_status_string(int status) {
    static thread_local std::string buf;
    switch (status) {
        case ADAMW_OK: return "ok";
        case ADAMW_ERR_INVALID_ARG: return "invalid argument";
        case ADAMW_ERR_MISALIGNED: return "buffer not aligned to its element size";
        case ADAMW_ERR_NO_NORM: return "clipping or norm asked of a plan made without ADAMW_PLAN_NORM";
        case ADAMW_ERR_TOO_LARGE: return "size exceeds a documented limit";
        case ADAMW_ERR_NOT_ACCESSIBLE: return "a buffer is not accessible from the plan's device";
        case ADAMW_ERR_CUDA:
            buf = std::string("CUDA error: ") + adamw::last_cuda_error();
            return buf.c_str();
        default: return "unknown status";
    }
}
