/*
 * adamw_ref.c -- plain, slow, CPU oracle for the AdamW optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the definition that the CUDA
 * library is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may build, load or call it.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Build:  gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *         (no FMA contraction: every fp32 operation below rounds once, to
 *         nearest-even, in the order written).
 *
 * What it computes
 * ----------------
 * Decoupled-weight-decay Adam ("AdamW") with bias correction, the optimizer
 * named on both pages:
 *   - "[pure bf16 training] w/ AnyPrecisionAdamW and Kahan summation"
 *     (transformers PR #21312), run recipe "Train from scratch":
 *     adamw_anyprecision with use_kahan_summation=true and bf16 momentum,
 *     variance and compensation buffers; weight_decay 0.1, betas 0.9/0.95,
 *     learning rate 2e-4.  Memory breakdown "bf16 pure: 4+2 optim, 2 grad,
 *     2 weights" = bf16 m, v, c + bf16 g + bf16 p.
 *   - "Distributed optimizer support for BERT" (NeMo PR #5305), "Usage":
 *     distributed_fused_adam, whose per-shard work is the mixed-precision
 *     update with fp32 optimizer state.
 * The pages print no update equation; the reading used here is the textbook
 * one (Loshchilov & Hutter decoupled decay, Kingma & Ba bias correction):
 *
 *   per call, with t = number of applied updates including this one,
 *   scalars computed in fp64 and rounded once to fp32:
 *     bc1 = 1 - b1^t,  bc2 = 1 - b2^t   (b^t by binary exponentiation)
 *     step_size = lr / bc1,  sbc2 = sqrt(bc2)
 *     omb1 = 1 - b1,  omb2 = 1 - b2,  lrwd = lr * wd
 *
 *   per element, fp32, one rounding per operation, in this order:
 *     g   = f32(g_bf16)            [* coef when clipping by global norm]
 *     m'  = (b1 * m) + (omb1 * g)
 *     v'  = (b2 * v) + ((omb2 * g) * g)
 *     den = (sqrt(v') / sbc2) + eps
 *     upd = (step_size * (m' / den)) + (lrwd * p)
 *
 *   bf16 mode (all five buffers bf16; m', v' are rounded to bf16 when stored
 *   and the stored values feed den and upd):
 *     y  = c - upd                    -- the compensation absorbs the update
 *     p' = bf16(p + y)                -- p += c
 *     c' = bf16(y - (p' - p))         -- c keeps what rounding p lost
 *
 *   mixed mode (fp32 master/m/v, bf16 grad in, bf16 param out):
 *     master' = master - upd ;  p_out = bf16(master')
 *
 *   bf16 without compensation (use_kahan_summation=false): p' = bf16(p - upd)
 *   bf16 Kahan with fp32 variance (variance_dtype=float32): v' kept in fp32
 *   any precision (momentum_dtype, variance_dtype, compensation_buffer_dtype
 *   each bfloat16 or float32, Kahan on or off): the same step, each buffer
 *   rounded to its own type when stored and used as stored
 *
 *   remainder mode (the same update; the fp32 master is stored as the bf16
 *   parameter plus a 16-bit remainder, 10 B/param of optimizer state: "2 FP32
 *   optim state + 1 16-bit master param" in the memory estimate of
 *   "Distributed optimizer support for BERT", NeMo PR #5305):
 *     bits(master) = (bits(p16) << 16) + r16     (r16 signed, integer add)
 *     p16 = high half of master rounded to nearest, ties away from zero
 *     (ties cannot round down: the remainder would be +32768)
 *
 *   global-norm clipping (optional): norm = sqrt(sum of g^2) over all
 *   tensors in list order, the sum in compensated fp64; any non-finite g
 *   sets the flag and the step writes nothing; otherwise
 *   coef = (float) min(1, max_norm / (norm + 1e-6)).
 *
 * fp32 -> bf16 is round-to-nearest-even; NaN stays a (quiet) NaN, overflow
 * goes to +-inf, subnormals are kept (no flush to zero).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

typedef struct {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    float max_grad_norm; /* <= 0: no clipping */
} oracle_hparams_t;

/* ---------------------------------------------------------------- bf16 -- */

static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round an fp32 value to the nearest bf16, ties to the even mantissa.
 * Adding 0x7fff plus the lowest kept bit to the 32-bit pattern carries into
 * the kept half exactly when the dropped half is above one half ulp, or equal
 * to it with an odd kept half; a carry out of the mantissa bumps the exponent,
 * which is the correct next bf16 (and the largest finite value rounds to inf
 * when it should). */
static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)             /* NaN: keep sign, quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

void oracle_f32_to_bf16(const float* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

void oracle_bf16_to_f32(const uint16_t* in, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_bits_to_f32(in[i]);
}

/* ------------------------------------------------------ per-call scalars -- */

typedef struct {
    float step_size, sbc2, omb1, omb2, lrwd;
} step_scalars_t;

/* b^t for t >= 1 by binary exponentiation: walk the bits of t from the
 * lowest, multiplying the result by the current square for every set bit;
 * fp64, one rounding per multiplication.  Evaluated this way (IEEE
 * multiplications only, no library pow) the power is the same wherever it is
 * computed.  Relative error below 2*log2(t)+1 fp64 ulps. */
static double power_by_squaring(double b, int64_t t)
{
    double result = 1.0, square = b;
    while (t > 0) {
        if (t & 1) result = result * square;
        square = square * square;
        t >>= 1;
    }
    return result;
}

static step_scalars_t make_scalars(const oracle_hparams_t* hp, int64_t t)
{
    double b1 = (double)hp->beta1, b2 = (double)hp->beta2;
    double bc1 = 1.0 - power_by_squaring(b1, t);
    double bc2 = 1.0 - power_by_squaring(b2, t);
    step_scalars_t s;
    s.step_size = (float)((double)hp->lr / bc1);
    s.sbc2 = (float)sqrt(bc2);
    s.omb1 = (float)(1.0 - b1);
    s.omb2 = (float)(1.0 - b2);
    s.lrwd = (float)((double)hp->lr * (double)hp->weight_decay);
    return s;
}

/* Exposed so that tests can check the scalars themselves. */
void oracle_step_scalars(const oracle_hparams_t* hp, int64_t t, float out5[5])
{
    step_scalars_t s = make_scalars(hp, t);
    out5[0] = s.step_size;
    out5[1] = s.sbc2;
    out5[2] = s.omb1;
    out5[3] = s.omb2;
    out5[4] = s.lrwd;
}

/* ------------------------------------------------------------ bf16 mode -- */

/* One step over one bf16 tensor, Kahan-compensated.  p, m, v, c updated in
 * place; g read only. */
void oracle_adamw_bf16_kahan(uint16_t* p, const uint16_t* g, uint16_t* m,
                             uint16_t* v, uint16_t* c, int64_t n,
                             const oracle_hparams_t* hp, int64_t t, float coef)
{
    step_scalars_t s = make_scalars(hp, t);
    const float b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps;
    const int clip = hp->max_grad_norm > 0.0f;

    for (int64_t i = 0; i < n; ++i) {
        float gi = bf16_bits_to_f32(g[i]);
        if (clip) gi = gi * coef;
        float p0 = bf16_bits_to_f32(p[i]);
        float m0 = bf16_bits_to_f32(m[i]);
        float v0 = bf16_bits_to_f32(v[i]);
        float c0 = bf16_bits_to_f32(c[i]);

        float m1 = (b1 * m0) + (s.omb1 * gi);
        float v1 = (b2 * v0) + ((s.omb2 * gi) * gi);
        uint16_t m1h = f32_to_bf16_rne(m1);
        uint16_t v1h = f32_to_bf16_rne(v1);
        float ms = bf16_bits_to_f32(m1h);
        float vs = bf16_bits_to_f32(v1h);

        float den = (sqrtf(vs) / s.sbc2) + eps;
        float upd = (s.step_size * (ms / den)) + (s.lrwd * p0);

        float y = c0 - upd;
        uint16_t pnh = f32_to_bf16_rne(p0 + y);
        float pn = bf16_bits_to_f32(pnh);
        uint16_t cnh = f32_to_bf16_rne(y - (pn - p0));

        p[i] = pnh;
        m[i] = m1h;
        v[i] = v1h;
        c[i] = cnh;
    }
}

/* The same step without compensation (use_kahan_summation=false): the update
 * is added to the bf16 parameter directly and whatever rounding drops is lost.
 * Used to show the stall that compensation prevents. */
void oracle_adamw_bf16_plain(uint16_t* p, const uint16_t* g, uint16_t* m,
                             uint16_t* v, int64_t n,
                             const oracle_hparams_t* hp, int64_t t, float coef)
{
    step_scalars_t s = make_scalars(hp, t);
    const float b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps;
    const int clip = hp->max_grad_norm > 0.0f;

    for (int64_t i = 0; i < n; ++i) {
        float gi = bf16_bits_to_f32(g[i]);
        if (clip) gi = gi * coef;
        float p0 = bf16_bits_to_f32(p[i]);
        float m1 = (b1 * bf16_bits_to_f32(m[i])) + (s.omb1 * gi);
        float v1 = (b2 * bf16_bits_to_f32(v[i])) + ((s.omb2 * gi) * gi);
        uint16_t m1h = f32_to_bf16_rne(m1);
        uint16_t v1h = f32_to_bf16_rne(v1);
        float den = (sqrtf(bf16_bits_to_f32(v1h)) / s.sbc2) + eps;
        float upd = (s.step_size * (bf16_bits_to_f32(m1h) / den)) + (s.lrwd * p0);
        p[i] = f32_to_bf16_rne(p0 - upd);
        m[i] = m1h;
        v[i] = v1h;
    }
}

/* bf16 parameters, bf16 momentum and compensation, fp32 variance (the
 * run recipe's optim_args with variance_dtype=float32): the same Kahan step
 * as oracle_adamw_bf16_kahan with v kept (and used) in fp32. */
void oracle_adamw_bf16_kahan_v32(uint16_t* p, const uint16_t* g, uint16_t* m,
                                 float* v, uint16_t* c, int64_t n,
                                 const oracle_hparams_t* hp, int64_t t, float coef)
{
    step_scalars_t s = make_scalars(hp, t);
    const float b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps;
    const int clip = hp->max_grad_norm > 0.0f;

    for (int64_t i = 0; i < n; ++i) {
        float gi = bf16_bits_to_f32(g[i]);
        if (clip) gi = gi * coef;
        float p0 = bf16_bits_to_f32(p[i]);
        float c0 = bf16_bits_to_f32(c[i]);
        float m1 = (b1 * bf16_bits_to_f32(m[i])) + (s.omb1 * gi);
        float v1 = (b2 * v[i]) + ((s.omb2 * gi) * gi);
        uint16_t m1h = f32_to_bf16_rne(m1);
        float den = (sqrtf(v1) / s.sbc2) + eps;
        float upd = (s.step_size * (bf16_bits_to_f32(m1h) / den)) + (s.lrwd * p0);
        float y = c0 - upd;
        uint16_t pnh = f32_to_bf16_rne(p0 + y);
        float pn = bf16_bits_to_f32(pnh);
        p[i] = pnh;
        m[i] = m1h;
        v[i] = v1;
        c[i] = f32_to_bf16_rne(y - (pn - p0));
    }
}

/* AnyPrecisionAdamW with a bf16 parameter and gradient and a storage type
 * chosen per optimizer buffer -- the run recipe's optim_args
 * momentum_dtype, variance_dtype, compensation_buffer_dtype (bfloat16 or
 * float32 each) and use_kahan_summation ("[pure bf16 training] w/
 * AnyPrecisionAdamW and Kahan summation", "Train from scratch").
 *
 * flags: 1 = exp_avg is fp32, 2 = exp_avg_sq is fp32, 4 = compensation is
 * fp32, 8 = no Kahan summation (no compensation buffer; flag 4 then invalid).
 * A bf16 buffer holds bf16 bits (uint16_t), an fp32 buffer floats.  Each
 * buffer is rounded to its own type when stored, and the value stored is the
 * value the rest of the step uses.  Flags 0, 2 and 8 are the bf16 Kahan, bf16
 * Kahan with fp32 variance and bf16 without compensation steps above.
 * Returns -1 (and writes nothing) for flag 4 together with flag 8. */
static float load_any(const void* buf, int fp32, int64_t i)
{
    return fp32 ? ((const float*)buf)[i]
                : bf16_bits_to_f32(((const uint16_t*)buf)[i]);
}

/* Stores x in the buffer's type; returns the value stored. */
static float store_any(void* buf, int fp32, int64_t i, float x)
{
    if (fp32) {
        ((float*)buf)[i] = x;
        return x;
    }
    uint16_t h = f32_to_bf16_rne(x);
    ((uint16_t*)buf)[i] = h;
    return bf16_bits_to_f32(h);
}

int32_t oracle_adamw_anyprec(uint16_t* p, const uint16_t* g, void* m, void* v,
                             void* c, int64_t n, int32_t flags,
                             const oracle_hparams_t* hp, int64_t t, float coef)
{
    const int m32 = (flags & 1) != 0, v32 = (flags & 2) != 0;
    const int c32 = (flags & 4) != 0, kahan = (flags & 8) == 0;
    if ((flags & ~15) || (!kahan && c32)) return -1;
    step_scalars_t s = make_scalars(hp, t);
    const float b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps;
    const int clip = hp->max_grad_norm > 0.0f;

    for (int64_t i = 0; i < n; ++i) {
        float gi = bf16_bits_to_f32(g[i]);
        if (clip) gi = gi * coef;
        float p0 = bf16_bits_to_f32(p[i]);

        float m1 = (b1 * load_any(m, m32, i)) + (s.omb1 * gi);
        float v1 = (b2 * load_any(v, v32, i)) + ((s.omb2 * gi) * gi);
        float ms = store_any(m, m32, i, m1);
        float vs = store_any(v, v32, i, v1);

        float den = (sqrtf(vs) / s.sbc2) + eps;
        float upd = (s.step_size * (ms / den)) + (s.lrwd * p0);

        if (kahan) {
            float y = load_any(c, c32, i) - upd;
            uint16_t pnh = f32_to_bf16_rne(p0 + y);
            float pn = bf16_bits_to_f32(pnh);
            store_any(c, c32, i, y - (pn - p0));
            p[i] = pnh;
        } else {
            p[i] = f32_to_bf16_rne(p0 - upd);
        }
    }
    return 0;
}

/* ----------------------------------------------------- learning rate -- */

/* The recipe's --lr_scheduler_type linear --warmup_steps W for T training
 * steps: the update with t applied steps before it (k = t - 1) uses
 * lr * k / max(1, W) while k < W, then lr * max(0, (T - k) / max(1, T - W));
 * fp64, rounded once to fp32.  (The first update of a warm-up therefore uses
 * lr 0, as a scheduler that advances after each optimizer step does.) */
float oracle_lr_linear_warmup(float base_lr, int64_t t, int64_t warmup, int64_t total)
{
    int64_t k = t - 1;
    double f;
    if (k < warmup)
        f = (double)k / (double)(warmup > 1 ? warmup : 1);
    else {
        double span = (double)((total - warmup) > 1 ? (total - warmup) : 1);
        f = (double)(total - k) / span;
        if (f < 0.0) f = 0.0;
    }
    return (float)((double)base_lr * f);
}

/* ----------------------------------------------------------- mixed mode -- */

/* One step over one shard: fp32 master, m, v in place; bf16 grad read;
 * bf16 copy of the new master written to p_out. */
void oracle_adamw_mixed(float* master, const uint16_t* g, float* m, float* v,
                        uint16_t* p_out, int64_t n,
                        const oracle_hparams_t* hp, int64_t t, float coef)
{
    step_scalars_t s = make_scalars(hp, t);
    const float b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps;
    const int clip = hp->max_grad_norm > 0.0f;

    for (int64_t i = 0; i < n; ++i) {
        float gi = bf16_bits_to_f32(g[i]);
        if (clip) gi = gi * coef;
        float p0 = master[i];
        float m1 = (b1 * m[i]) + (s.omb1 * gi);
        float v1 = (b2 * v[i]) + ((s.omb2 * gi) * gi);
        float den = (sqrtf(v1) / s.sbc2) + eps;
        float upd = (s.step_size * (m1 / den)) + (s.lrwd * p0);
        float pn = p0 - upd;
        master[i] = pn;
        m[i] = m1;
        v[i] = v1;
        p_out[i] = f32_to_bf16_rne(pn);
    }
}

/* ------------------------------------------------------ remainder mode -- */

/* The fp32 master held as a bf16 high half and a signed 16-bit remainder of
 * the bit pattern: bits(master) = (bits(p16) << 16) + r16. */
static float master_from_halves(uint16_t p16, int16_t r16)
{
    uint32_t u = ((uint32_t)p16 << 16) + (uint32_t)(int32_t)r16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Splits an fp32 value into its nearest bf16 (ties away from zero in
 * magnitude) and the remainder that restores it exactly. */
static void halves_from_master(float f, uint16_t* p16, int16_t* r16)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t hi = (uint16_t)((u + 0x8000u) >> 16);
    *p16 = hi;
    *r16 = (int16_t)(int32_t)(u - ((uint32_t)hi << 16));
}

void oracle_split_master(const float* in, uint16_t* p16, int16_t* r16, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) halves_from_master(in[i], &p16[i], &r16[i]);
}

void oracle_join_master(const uint16_t* p16, const int16_t* r16, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = master_from_halves(p16[i], r16[i]);
}

/* One step over one shard in remainder mode: p16 (the model's bf16
 * parameter) and r16 in place, fp32 m, v in place, bf16 grad read.  The
 * update is the mixed mode's, on the master the two halves hold. */
void oracle_adamw_remainder(uint16_t* p16, const uint16_t* g, float* m, float* v,
                            int16_t* r16, int64_t n,
                            const oracle_hparams_t* hp, int64_t t, float coef)
{
    step_scalars_t s = make_scalars(hp, t);
    const float b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps;
    const int clip = hp->max_grad_norm > 0.0f;

    for (int64_t i = 0; i < n; ++i) {
        float gi = bf16_bits_to_f32(g[i]);
        if (clip) gi = gi * coef;
        float p0 = master_from_halves(p16[i], r16[i]);
        float m1 = (b1 * m[i]) + (s.omb1 * gi);
        float v1 = (b2 * v[i]) + ((s.omb2 * gi) * gi);
        float den = (sqrtf(v1) / s.sbc2) + eps;
        float upd = (s.step_size * (m1 / den)) + (s.lrwd * p0);
        float pn = p0 - upd;
        m[i] = m1;
        v[i] = v1;
        halves_from_master(pn, &p16[i], &r16[i]);
    }
}

/* ------------------------------------------------- global norm and clip -- */

/* Adds sum of g^2 of one bf16 tensor, in element order, to the running sum
 * acc[0] + acc[1] and ORs a non-finite test into *nonfinite.  Call once per
 * tensor, in list order, starting from acc = {0, 0}.
 *
 * The definition is the exact sum of squares.  A plain fp64 running sum is
 * not close enough to it for long lists: squares below half an ulp of the
 * running sum are dropped every time, which biases the result low (about
 * 1e-10 relative over 125M terms).  The sum is therefore compensated
 * (Kahan-Babuska / Neumaier): acc[1] collects, exactly, what each fp64
 * addition rounds away. */
void oracle_grad_sumsq(const uint16_t* g, int64_t n, double acc[2],
                       int32_t* nonfinite)
{
    double s = acc[0], comp = acc[1];
    int32_t bad = *nonfinite;
    for (int64_t i = 0; i < n; ++i) {
        double x = (double)bf16_bits_to_f32(g[i]);
        if (!isfinite(x)) bad = 1;
        double sq = x * x;
        double t = s + sq;
        if (fabs(s) >= fabs(sq))
            comp += (s - t) + sq;
        else
            comp += (sq - t) + s;
        s = t;
    }
    acc[0] = s;
    acc[1] = comp;
    *nonfinite = bad;
}

/* Global-norm clip factor from the total sum of squares:
 * coef = min(1, max_norm / (norm + 1e-6)), rounded to fp32.  Writes the fp64
 * norm to *norm_out when it is not NULL. */
float oracle_clip_coef(double sumsq, float max_norm, double* norm_out)
{
    double norm = sqrt(sumsq);
    if (norm_out) *norm_out = norm;
    double coef = (double)max_norm / (norm + 1e-6);
    if (coef > 1.0) coef = 1.0;
    return (float)coef;
}

/* ------------------------------------------------ one step over a list -- */

typedef struct {
    void* param;      /* bf16: bf16 p    mixed: fp32 master  remainder: bf16 p */
    const void* grad; /* bf16 */
    void* exp_avg;    /* bf16: bf16      mixed, remainder: fp32 */
    void* exp_avg_sq; /* bf16: bf16      mixed, remainder: fp32 */
    void* aux;        /* bf16: bf16 c    mixed: bf16 p out   remainder: int16 r */
    int64_t numel;
} oracle_tensor_t;

/* The whole optimizer step over a tensor list (host buffers), mode 0 = bf16
 * Kahan, 1 = mixed, 2 = remainder, 3 = bf16 without compensation (aux
 * unused), 4 = bf16 Kahan with fp32 variance, 16 + flags = the
 * any-precision step of oracle_adamw_anyprec (aux = compensation).  With clipping, the norm is taken first over every
 * tensor; a non-finite gradient anywhere makes the call write nothing and
 * return 1 (the caller must not advance t).  Returns 0 after an applied step,
 * -1 for an unknown mode.
 * norm_out (nullable) receives the fp64 norm when clipping. */
int32_t oracle_adamw_list_step(const oracle_tensor_t* list, int32_t n_tensors,
                               int32_t mode, const oracle_hparams_t* hp,
                               int64_t t, double* norm_out)
{
    float coef = 1.0f;
    const int anyprec_ok = mode >= 16 && mode < 32 && (mode & 12) != 12;
    if (!(mode >= 0 && mode <= 4) && !anyprec_ok) return -1;
    if (hp->max_grad_norm > 0.0f) {
        double acc[2] = {0.0, 0.0};
        int32_t bad = 0;
        for (int32_t k = 0; k < n_tensors; ++k)
            oracle_grad_sumsq((const uint16_t*)list[k].grad, list[k].numel,
                              acc, &bad);
        coef = oracle_clip_coef(acc[0] + acc[1], hp->max_grad_norm, norm_out);
        if (bad) return 1;
    }
    for (int32_t k = 0; k < n_tensors; ++k) {
        const oracle_tensor_t* e = &list[k];
        if (mode == 0)
            oracle_adamw_bf16_kahan((uint16_t*)e->param,
                                    (const uint16_t*)e->grad,
                                    (uint16_t*)e->exp_avg,
                                    (uint16_t*)e->exp_avg_sq,
                                    (uint16_t*)e->aux, e->numel, hp, t, coef);
        else if (mode == 2)
            oracle_adamw_remainder((uint16_t*)e->param, (const uint16_t*)e->grad,
                                   (float*)e->exp_avg, (float*)e->exp_avg_sq,
                                   (int16_t*)e->aux, e->numel, hp, t, coef);
        else if (mode == 3)
            oracle_adamw_bf16_plain((uint16_t*)e->param, (const uint16_t*)e->grad,
                                    (uint16_t*)e->exp_avg, (uint16_t*)e->exp_avg_sq,
                                    e->numel, hp, t, coef);
        else if (mode >= 16)
            oracle_adamw_anyprec((uint16_t*)e->param, (const uint16_t*)e->grad,
                                 e->exp_avg, e->exp_avg_sq, e->aux, e->numel,
                                 mode - 16, hp, t, coef);
        else if (mode == 4)
            oracle_adamw_bf16_kahan_v32((uint16_t*)e->param, (const uint16_t*)e->grad,
                                        (uint16_t*)e->exp_avg, (float*)e->exp_avg_sq,
                                        (uint16_t*)e->aux, e->numel, hp, t, coef);
        else
            oracle_adamw_mixed((float*)e->param, (const uint16_t*)e->grad,
                               (float*)e->exp_avg, (float*)e->exp_avg_sq,
                               (uint16_t*)e->aux, e->numel, hp, t, coef);
    }
    return 0;
}
