// adamw_internal.h -- types shared by the host planner (plan_build.cpp) and
// the CUDA kernels (adamw_sm.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "adamw_sm.h"

namespace adamw {

// Threads per CTA of the update and norm-partial kernels.
#ifndef ADAMW_BLOCK
#define ADAMW_BLOCK 256
#endif
constexpr int kBlock = ADAMW_BLOCK;
// Elements per vector: 8 bf16 = one 16-byte load; 8 fp32 = two.
constexpr int kVec = 8;
// Largest gradient list (MiB of bf16 gradients) whose clipped steps run as
// one fused launch.  Measured on GB300 with the fp32-master mode, every
// kernel launched with programmatic dependent launch (median us per step,
// fused / three launches): 2M parameters 24.7 / 27.5, 4M 34.1 / 36.0, 8M
// 49.4 / 50.5, 13.85M 70.6 / 71.9, then 24M 117.5 / 116.7, 40M 190.4 /
// 187.9, 80M 373.3 / 371.0: the three launches overlap their ramps, and the
// fused norm phase runs on the update's grid (half the norm kernel's CTAs).
// 32 MiB = 16.7M parameters, between the last win and the first loss.
#ifndef ADAMW_FUSED_MAX_GRAD_MB
#define ADAMW_FUSED_MAX_GRAD_MB 32
#endif
constexpr int64_t kFusedMaxGradBytes = int64_t(ADAMW_FUSED_MAX_GRAD_MB) << 20;
// 1: the fused clipped step's norm phase loads g with the evict-last L2
// policy, so that more of the update phase's second read of g hits L2.
#ifndef ADAMW_FUSED_KEEP_G
#define ADAMW_FUSED_KEEP_G 1
#endif
constexpr bool kFusedKeepG = ADAMW_FUSED_KEEP_G != 0;


// Fewest elements a CTA is given before the grid is shrunk (one vector per
// thread), so tiny lists do not launch idle CTAs.
constexpr int64_t kMinElemsPerCta = int64_t(kBlock) * kVec;

// Device copy of one adamw_tensor_t (same layout).
struct TensorDev {
    void* p;
    const void* g;
    void* m;
    void* v;
    void* a;
    int64_t numel;
};
static_assert(sizeof(TensorDev) == sizeof(adamw_tensor_t), "table layout");

// One piece of one tensor, processed by exactly one CTA (host form).
struct ChunkDev {
    int32_t tensor;
    int32_t vec;     // 1: all five bases 16-byte aligned at `off`
    int64_t off;
    int64_t len;
};

// Bounds-checked build: every chunk also carries the extent of each of its
// tensor's buffers, and the kernels check the chunk against them before any
// access; a chunk that falls outside is skipped and bit 1 (value 2) of the
// plan's device status word is set.  A debugging aid (compute-sanitizer
// stand-in), off by default.
#ifndef ADAMW_CHECK_BOUNDS
#define ADAMW_CHECK_BOUNDS 0
#endif
// 1: the bf16 Kahan update stages its inputs in shared memory with
// cp.async.bulk (a measured alternative, slower on GB300; off by default).
#ifndef ADAMW_BULK
#define ADAMW_BULK 0
#endif
constexpr int32_t kStatusBounds = 2;

// Device form of a chunk: the five stream pointers already offset to the
// chunk's first element, so a CTA can prefetch its next chunk with one
// independent 48-byte load.
struct alignas(16) ChunkPtr {
    void* p;
    const void* g;
    void* m;
    void* v;
    void* a;
    int64_t len2;    // 2 * len + vec
#if ADAMW_CHECK_BOUNDS
    const void* lo[5];   // first byte of each of the tensor's buffers
    const void* hi[5];   // one past its last byte
    int32_t* status;     // the plan's device status word
    int64_t pad_;
#endif
};
static_assert(sizeof(ChunkPtr) == (ADAMW_CHECK_BOUNDS ? 144 : 48), "chunk layout");

// Nominal elements per round-robin tile of the interleaved partition of the
// update kernel (measured on GB300: round-robin tiles beat contiguous per-CTA
// ranges by ~6 % on the 1.3B-parameter list, because the whole grid then
// streams one narrow window of each buffer; 8192 is 1 % faster than 16384 and
// 32768).  The tile actually used is stretched so that every CTA gets the
// same number of tiles.  Lists with fewer than two tiles per CTA, and the
// read-only norm pass, use contiguous ranges.
#ifndef ADAMW_TILE_ELEMS
#define ADAMW_TILE_ELEMS 8192
#endif
// The nominal tile of lists that would get fewer than kDynMinRounds rounds of
// ADAMW_TILE_ELEMS: with smaller tiles they get more rounds, and claimable
// last rounds once those reach kDynMinRounds.  Equal to ADAMW_TILE_ELEMS:
// one tile size for every list.
#ifndef ADAMW_SMALL_TILE_ELEMS
#define ADAMW_SMALL_TILE_ELEMS ADAMW_TILE_ELEMS
#endif
// 1: tiles cut in the flattened list and stretched so every CTA gets the
// same number (cuts inside a tensor at multiples of ADAMW_CUT_ALIGN elements
// from its vector body's start); 0: fixed tiles cut per tensor.
#ifndef ADAMW_TILE_BALANCE
#define ADAMW_TILE_BALANCE 1
#endif
#ifndef ADAMW_CUT_ALIGN
#define ADAMW_CUT_ALIGN 2048
#endif
// Granule of the per-CTA quotas: every CTA of the interleaved partition gets
// the same number of elements to within this many (measured on GB300, the
// 13.85M-element shard on 304 CTAs was 7 % slower when the quotas went by
// whole 8K tiles, five tiles for some CTAs and six for others).
#ifndef ADAMW_BALANCE_ALIGN
#define ADAMW_BALANCE_ALIGN 256
#endif
// The norm pass's resident CTAs per SM (its grid is that times the SMs) and
// 16-byte vectors of g in flight per thread.
#ifndef ADAMW_NORM_CTAS
#define ADAMW_NORM_CTAS 4
#endif
#ifndef ADAMW_NORM_UNROLL
#define ADAMW_NORM_UNROLL 8
#endif
constexpr int kNormCtas = ADAMW_NORM_CTAS;
constexpr int kNormUnroll = ADAMW_NORM_UNROLL;
// 1: the update's last rounds (about kDynSharePct percent of the list) are
// not dealt to CTAs but cut into tiles (at most kTileElems) that the CTAs
// claim with an atomic counter once their own tiles are done, so that CTAs
// on SMs that stream faster take more of them.  Measured on GB300: with
// equal work, the CTAs of one launch ended up to 8 % apart (the 1.3B list:
// 3.29 to 3.58 ms, median 3.41), SM to SM; with the claims within 4 us of
// each other, and the step went from 3.57 to 3.46 ms.
#ifndef ADAMW_DYN_TAIL
#define ADAMW_DYN_TAIL 1
#endif
#ifndef ADAMW_DYN_SHARE_PCT
#define ADAMW_DYN_SHARE_PCT 12
#endif
// Lists of fewer rounds keep every tile dealt: there one tile is a large part
// of a CTA's work and the claims cost more than they even out (measured,
// fp32 master: the 13.85M shard, 6 rounds, 0.5 % slower with claims, 8 %
// with claims of whole tiles; 8M, 3 rounds, 5 % slower; bf16 Kahan lists of
// 40M to 80M, 11 to 21 rounds, 2 to 3 % faster).
#ifndef ADAMW_DYN_MIN_ROUNDS
#define ADAMW_DYN_MIN_ROUNDS 8
#endif
// 1: the claimable tiles shrink towards the end of the list (each about the
// work left over twice the grid, between kCutAlign and kTileElems), so the
// last claims are short and the CTAs end closer together.
#ifndef ADAMW_DYN_GUIDED
#define ADAMW_DYN_GUIDED 1
#endif
constexpr bool kDynTail = ADAMW_DYN_TAIL != 0 && !ADAMW_BULK;
constexpr int kDynSharePct = ADAMW_DYN_SHARE_PCT;
constexpr int64_t kDynMinRounds = ADAMW_DYN_MIN_ROUNDS;
constexpr bool kDynGuided = ADAMW_DYN_GUIDED != 0;
// 1: the fused clipped step is a cooperative launch; 0 (measured 2 us
// faster per step on the 13.85M shard): an ordinary one, with programmatic
// serialization.  Its grid never exceeds what the device holds at once (the
// plan's occupancy), so every CTA becomes resident either way, and the grid
// barrier's wait is bounded.
#ifndef ADAMW_FUSED_COOP
#define ADAMW_FUSED_COOP 0
#endif
// Elements by which CTA 0's share of the update partition is short of the
// others': in the one-launch device step CTA 0 first computes the next
// step's scalars for the memo (fp64, about 1 us on GB300) while the other
// CTAs stream, and this keeps it from ending last (on lists of up to ~4096
// elements per CTA it gets none).  A multiple of kBalanceAlign.
#ifndef ADAMW_MEMO_RELIEF
#define ADAMW_MEMO_RELIEF 4096
#endif
constexpr int64_t kMemoRelief = ADAMW_MEMO_RELIEF;
constexpr int64_t kTileElems = ADAMW_TILE_ELEMS;
constexpr int64_t kSmallTileElems = ADAMW_SMALL_TILE_ELEMS;
constexpr int64_t kCutAlign = ADAMW_CUT_ALIGN;
constexpr int64_t kBalanceAlign = ADAMW_BALANCE_ALIGN;
static_assert(kCutAlign % kVec == 0 && kTileElems % kCutAlign == 0, "tile cut alignment");
static_assert(kSmallTileElems % kCutAlign == 0 && kSmallTileElems <= kTileElems, "small tile");
static_assert(kBalanceAlign % kVec == 0 && kCutAlign % kBalanceAlign == 0, "balance granule");
static_assert(kMemoRelief >= 0 && kMemoRelief % kBalanceAlign == 0, "relief granule");

// Output of the norm finalize kernel, read by the clipped update.
struct NormOut {
    double norm;
    float coef;
    int32_t nonfinite;
};

// The per-step scalars the kernels take by value.
struct StepScalars {
    float beta1, beta2, omb1, omb2;
    float step_size, sbc2, eps, lrwd;
    float max_grad_norm;
};

// What the device-resident step path (adamw_step_device) decides before the
// update runs: the scalars of t = *d_step + 1, the clip coefficient, and
// whether the step is skipped (1: non-finite gradient under clipping,
// 2: invalid hyperparameters); with the hyperparameters and t they came
// from, for the next step's memo.
struct StepRecord {
    StepScalars s;
    float coef;
    int32_t skip;
    adamw_hparams_t hp;
    int32_t pad_;
    int64_t t;
};

// The per-step scalars of one (hyperparameters, t), remembered on the device
// by the device-resident step: CTA 0 of step t's update computes the scalars
// of t + 1 into slot (t + 1) & 1 first, while the others stream (its share
// of the list is kMemoRelief elements short for that), so that the next step
// reads them instead of computing them again.  `key` is
// the bit pattern of the six hyperparameters and of t; `valid` is 0 in a
// slot never written.  A slot that does not match is recomputed, so the
// record only saves time, never changes a result.
struct ScalarMemo {
    uint32_t key[8];
    StepScalars s;
    int32_t valid;
    int32_t pad_[6];
};
static_assert(sizeof(ScalarMemo) == 96, "memo layout");

// The squares beta^(2^i), i = 0..63, of both betas, as the binary
// exponentiation computes them (each the previous one squared, rounded to
// fp64), keyed by the betas' bit patterns; `valid` is 0 until written.  With
// them beta^t is one multiplication per set bit of t, in the same order and
// with the same roundings as the exponentiation itself.  It sits in the plan
// right after the two memo slots; CTA 0 of an update writes and reads it
// (memo_next), nothing else does.
struct PowTable {
    uint32_t b1, b2;
    int32_t valid;
    int32_t pad_;
    double sq[2][64];
};
// memo_next reads the rows 16 bytes at a time from memo + 2 (the memo slots
// start 256-byte aligned in the plan)
static_assert((2 * sizeof(ScalarMemo)) % 16 == 0 && offsetof(PowTable, sq) % 16 == 0,
              "squares table rows 16-byte aligned");

// The plan's claim-and-arrival word of the update partition, one 64-bit
// atomic word: bits 0-23 count the claims of the last rounds' pieces, bits
// 24-43 the CTAs that have finished (the last one to arrive zeroes the word
// for the next launch), bits 44-63 the CTAs that saw a non-finite gradient
// (the one-launch device step's flag).
constexpr unsigned long long kSyncClaim = 1ull;
constexpr unsigned long long kSyncArrive = 1ull << 24;
constexpr unsigned long long kSyncFlagged = 1ull << 44;
constexpr unsigned long long kSyncClaimMask = kSyncArrive - 1;
constexpr unsigned long long kSyncArriveMask = (kSyncFlagged - 1) & ~kSyncClaimMask;

// Where the claimable chunks of the last rounds are, for the kernels.
struct DynTail {
    int32_t begin;                  // index of the first claimable chunk
    int32_t n;                      // how many (0: none; then only the one-launch
                                    // device step counts arrivals)
    unsigned long long* sync;       // the claim-and-arrival word
};

// Kernel flavours: plain step, clipped step (reads the norm finalize's
// output, skips on non-finite), plain step that also reports non-finite g.
enum Kind { kPlain = 0, kClip = 1, kReport = 2 };

// ---- host planner (plan_build.cpp) ----

// Kernel variants: one per storage mode 0..4 and one per any-precision mode
// that is not one of those under another number.
constexpr int kModes = 14;
constexpr int32_t kVariantModes[kModes] = {
    ADAMW_MODE_BF16_KAHAN, ADAMW_MODE_MIXED_FP32_MASTER, ADAMW_MODE_MIXED_BF16_REMAINDER,
    ADAMW_MODE_BF16_PLAIN, ADAMW_MODE_BF16_KAHAN_FP32_VAR,
    ADAMW_MODE_ANYPREC | 1, ADAMW_MODE_ANYPREC | 3, ADAMW_MODE_ANYPREC | 4,
    ADAMW_MODE_ANYPREC | 5, ADAMW_MODE_ANYPREC | 6, ADAMW_MODE_ANYPREC | 7,
    ADAMW_MODE_ANYPREC | 9, ADAMW_MODE_ANYPREC | 10, ADAMW_MODE_ANYPREC | 11};
// The variant (index into kVariantModes) that runs a storage mode; -1 for an
// invalid mode.  The any-precision modes 16, 18 and 24 run variants 0, 4, 3.
int mode_variant(int32_t mode);
bool valid_mode(int32_t mode);
// Bytes per element of param, grad, exp_avg, exp_avg_sq, aux in a mode.
void element_sizes(int32_t mode, int64_t es[5]);

int validate_table(const adamw_tensor_t* table, int32_t n, int32_t mode);
int validate_hparams(const adamw_hparams_t* hp, int64_t step);
int make_scalars(const adamw_hparams_t* hp, int64_t step, StepScalars* out);

// Splits the list over `grid` CTAs.  chunks are ordered by CTA; cta_begin has
// grid + 1 entries (chunks of CTA b are [cta_begin[b], cta_begin[b+1])).
// Chunks of the last rounds of the interleaved partition may be left to
// whichever CTA is free (chunk_cta -1): they follow every CTA's own chunks,
// from index cta_begin[grid], n_dyn of them, and are claimed at run time.
// CTA 0's share is `relief` elements short of the others' (kMemoRelief for
// the update partition, 0 for the norm pass's).
struct Partition {
    std::vector<ChunkDev> chunks;
    std::vector<int32_t> chunk_cta;
    std::vector<int32_t> cta_begin;
    int64_t n_dyn = 0;
    int64_t total = 0;
    int64_t scalar_elems = 0;
};
int build_partition(const adamw_tensor_t* table, int32_t n, int32_t mode,
                    int32_t grid, int64_t tile_elems, Partition* out,
                    int64_t relief = kMemoRelief);

// Device chunks (pointers offset per stream element size) of a partition.
void chunk_pointers(const adamw_tensor_t* table, int32_t mode, const Partition& P,
                    std::vector<ChunkPtr>* out);

// The grid a list of `total` elements gets when at most `max_grid` CTAs fit.
int32_t choose_grid(int64_t total, int32_t max_grid);

// Nominal tile of the update kernel's partition for a list of `total`
// elements on `grid` CTAs: 0 (contiguous ranges) when a CTA would get fewer
// than two tiles of kTileElems, kSmallTileElems when it would get fewer than
// kDynMinRounds, else kTileElems.
int64_t update_tile_elems(int64_t total, int32_t grid);

// Sizes of the interleaved partition's tiles.  With k rounds (the whole
// number nearest to total / (grid * tile_elems)), tile j belongs to CTA
// j % grid in round j / grid.  CTA 0's quota is total / grid less
// `relief` elements (never below zero; with one CTA, everything); the
// other CTAs share the rest, each quota rounded to kBalanceAlign elements
// (theirs differ by one granule at most); a CTA's k tiles are that quota's
// whole kCutAlign units shared out as evenly as the rounds allow (earlier
// rounds take the extra units; a short quota leaves some rounds empty), and
// its last-round tile also takes the quota's leftover granules.  Sizes are
// in the flattened list; the cuts themselves still move to each tensor's
// alignment grid.
struct TileSchedule {
    int32_t grid;
    int64_t k = 1, q0 = 0, base = 0, extra = 0;   // quotas in kBalanceAlign units
    TileSchedule(int64_t total, int32_t grid, int64_t tile_elems, int64_t relief);
    int64_t size(int64_t j) const;
    bool last_round(int64_t j) const { return j / grid >= k - 1; }
};

// Every buffer the mode uses can be dereferenced by `device` (device_access.cpp).
int check_device_access(const adamw_tensor_t* table, int32_t n, int32_t mode, int device);

// Remembers a CUDA error text for adamw_status_string (per host thread).
void set_cuda_error(const char* where, const char* what);
const char* last_cuda_error();

}  // namespace adamw
