/*
 * zero_oracle.c -- the oracle for the ZeRO shard optimizer step on a
 * FlatParameter: a plain, slow, single-threaded CPU restatement of what the
 * step computes, written to be checked by eye against the source pages.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "DeepSpeed 与 FSDP" (docs.ifdog.com, foundations/04-training/deepspeed-fsdp)
 *   [P2] "PyTorch FSDP（Fully Sharded Data Parallel）源码级深度解析" (tbr8.org)
 *   [P3] the ZeRO paper reading at 2kiu.com/news/5312103 (its title line,
 *        "企业官网建设流程全解析", does not match its body)
 *
 * Precision.  The pages fix mixed precision: fp16/bf16 parameters and
 * gradients, fp32 master weights and Adam moments ([P1] §逐步推导, [P2] §7.2),
 * with the gradient reduction in fp32 ([P1] §PyTorch FSDP 使用, MixedPrecision
 * reduce_dtype=float32).  So every floating-point operation of the update is
 * one IEEE-754 binary32 operation rounded to nearest-even, in the order the
 * code states; the library is built with -ffp-contract=off so that no
 * multiply-add is fused.  The squared gradient norm is summed exactly and
 * rounded once, so it does not depend on how the flat buffer is sharded.
 *
 * Parity pins (tests/test_oracle_*.py): closed forms of the Adam update,
 * special cases, brute force on tiny buffers, the ZeRO == DDP invariant, the
 * pages' memory figures, a hand-traced loss-scale sequence and an exhaustive
 * cast check against numpy's IEEE conversion.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_EINVAL 1
#define ORA_EOVERFLOW 5

/* ------------------------------------------------------------------------- */
/* Layout: [P2] §3.1 (FlatParameter records {start, end, shape} per parameter,
 * concatenated in order), [P2] §3.3 (`shard_size = full_numel // world_size`),
 * [P1] §FSDP 的分片粒度与 FlatParameter (`flat_param.chunk(world_size)[rank]`).
 * Reading: shard_size = ceil(full_numel / N); the flat buffer is padded with
 * zeros to N * shard_size; rank r owns [r*S, (r+1)*S).                        */
int ora_layout(const int64_t *starts, const int64_t *numels, int32_t n_infos,
               int32_t world_size, int64_t *full_numel, int64_t *shard_size,
               int64_t *padded_numel)
{
    if (!starts || !numels || n_infos < 1 || world_size < 1) return ORA_EINVAL;
    int64_t total = 0;
    for (int32_t k = 0; k < n_infos; ++k) {
        if (numels[k] < 0) return ORA_EINVAL;
        if (starts[k] != total) return ORA_EINVAL;      /* contiguous, in order */
        if (numels[k] > INT64_MAX - total) return ORA_EOVERFLOW;
        total += numels[k];
    }
    int64_t s = total / world_size + (total % world_size != 0);
    if (s != 0 && s > INT64_MAX / world_size) return ORA_EOVERFLOW;
    *full_numel = total;
    *shard_size = s;
    *padded_numel = s * (int64_t)world_size;
    return ORA_OK;
}

/* ------------------------------------------------------------------------- */
/* Memory accounting per GPU, in bytes.
 * [P1] §逐步推导: fp16 params 2Ψ + fp16 grads 2Ψ + fp32 master, m, v 4Ψ each
 *      = 16Ψ for plain data parallelism (stage 0).
 * [P1] §ZeRO-3 的数学总结:
 *      ZeRO-1: 2Ψ + 2Ψ + 12Ψ/N;  ZeRO-2: 2Ψ + 2Ψ/N + 12Ψ/N;
 *      ZeRO-3: 2Ψ/N + 2Ψ/N + 12Ψ/N.
 * Each part is returned rounded up to a whole byte; the total is the exact
 * sum of the three rational parts, rounded up once.                         */
typedef unsigned __int128 u128;

static int ceil_div_u128(u128 num, uint64_t den, uint64_t *out)
{
    u128 q = num / den + (num % den != 0);
    if (q > (u128)UINT64_MAX) return ORA_EOVERFLOW;
    *out = (uint64_t)q;
    return ORA_OK;
}

int ora_memory_breakdown(int32_t stage, uint64_t psi, int32_t world_size,
                         uint64_t *params, uint64_t *grads, uint64_t *optim,
                         uint64_t *total)
{
    if (stage < 0 || stage > 3 || world_size < 1) return ORA_EINVAL;
    const uint64_t n = (uint64_t)world_size;
    /* bytes per parameter of each part, and whether that part is split N ways */
    const uint64_t per[3] = {2, 2, 12};
    const int split[4][3] = {
        {0, 0, 0},   /* pure DP */
        {0, 0, 1},   /* ZeRO-1: optimizer states */
        {0, 1, 1},   /* ZeRO-2: + gradients */
        {1, 1, 1},   /* ZeRO-3: + parameters */
    };
    uint64_t part[3];
    u128 sum_num = 0;                     /* total * n, exactly */
    for (int k = 0; k < 3; ++k) {
        u128 bytes = (u128)per[k] * psi;
        if (split[stage][k]) {
            if (ceil_div_u128(bytes, n, &part[k])) return ORA_EOVERFLOW;
            sum_num += bytes;
        } else {
            if (bytes > (u128)UINT64_MAX) return ORA_EOVERFLOW;
            part[k] = (uint64_t)bytes;
            sum_num += bytes * n;
        }
    }
    uint64_t tot;
    if (ceil_div_u128(sum_num, n, &tot)) return ORA_EOVERFLOW;
    if (params) *params = part[0];
    if (grads) *grads = part[1];
    if (optim) *optim = part[2];
    if (total) *total = tot;
    return ORA_OK;
}

/* ------------------------------------------------------------------------- */
/* Number formats, written from the IEEE-754 definitions.                     */

/* binary16 -> binary32: the value is exactly representable. */
float ora_f16_to_f32(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int man = h & 0x3ff;
    float mag;
    if (e == 0x1f) {
        mag = man ? NAN : INFINITY;
    } else if (e == 0) {
        mag = (float)ldexp((double)man, -24);               /* subnormal */
    } else {
        mag = (float)ldexp((double)(1024 + man), e - 25);   /* (1.man) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* bfloat16 is the top half of a binary32 encoding. */
float ora_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> binary16, round to nearest, ties to even.  Overflow gives inf,
 * tiny values go through the subnormal range, NaN stays a (quiet) NaN.     */
uint16_t ora_f32_to_f16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    const int32_t be = (int32_t)((u >> 23) & 0xffu);
    const uint32_t man = u & 0x7fffffu;
    if (be == 0xff) {
        if (man == 0) return sign | 0x7c00u;
        return (uint16_t)(sign | 0x7e00u | (man >> 13));
    }
    if (be == 0) return sign;          /* fp32 subnormals are below half of the
                                          smallest fp16 subnormal: round to 0 */
    const int32_t e = be - 127;        /* |x| = sig * 2^(e-23), sig in [2^23, 2^24) */
    const uint32_t sig = man | 0x800000u;
    if (e > 15) return sign | 0x7c00u; /* |x| >= 2^16 > largest finite fp16 */
    /* fp16 quantum at this magnitude: 2^(max(e,-14) - 10).  Shift the 24-bit
       significand right so that one unit is that quantum.                   */
    const int32_t qexp = (e >= -14 ? e : -14) - 10;
    const int32_t shift = qexp - (e - 23);           /* >= 13 */
    uint32_t r;
    if (shift >= 25) {
        r = 0;                                       /* below half a quantum */
    } else {
        const uint32_t rem = sig & ((1u << shift) - 1u);
        const uint32_t half = 1u << (shift - 1);
        r = sig >> shift;
        if (rem > half || (rem == half && (r & 1u))) r += 1u;
    }
    if (e >= -14) {
        /* normal: r in [1024, 2048]; a carry into 2048 moves to the next
           binade, and from the top binade to the infinity encoding.         */
        return (uint16_t)(sign | (uint32_t)(((e + 15) << 10) + (int32_t)r - 1024));
    }
    return (uint16_t)(sign | r);                     /* subnormal (or min normal) */
}

/* binary32 -> bfloat16, round to nearest, ties to even.  bfloat16 keeps the
 * binary32 exponent, so rounding the encoding's low 16 bits is exact for
 * normals, subnormals and the overflow to infinity.                        */
uint16_t ora_f32_to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu))
        return (uint16_t)((u >> 16) | 0x40u);        /* quiet NaN */
    uint32_t hi = u >> 16;
    const uint32_t lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
    return (uint16_t)hi;
}

/* ------------------------------------------------------------------------- */
/* Hyper-parameters and loss-scale state.
 * [P3] §5.1 (ds_config): AdamW lr 3e-5, betas [0.9, 0.999], eps 1e-8,
 * weight_decay 0.01; fp16 loss_scale 0 (= dynamic), loss_scale_window 1000,
 * initial_scale_power 16; gradient_clipping 1.0.                            */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;  /* as a JSON config gives them */
    double max_grad_norm;         /* <= 0 disables clipping */
    int32_t dynamic_loss_scale;   /* 1: dynamic (loss_scale 0), 0: static */
    int32_t initial_scale_power;
    int32_t loss_scale_window;
    int32_t pad_;
    double static_loss_scale;
    double min_loss_scale;
} ora_hparams;

typedef struct {
    float scale;
    int32_t good_steps;
    int64_t step_t;               /* number of applied (not skipped) steps */
    int64_t overflow_count;
} ora_scaler;

typedef struct {
    int32_t overflow;
    int32_t skipped;
    double grad_norm;
    float clip_coef;
    float scale_used;
} ora_result;

/* Initial loss-scale state: 2^initial_scale_power when dynamic. */
void ora_scaler_init(const ora_hparams *hp, ora_scaler *st)
{
    st->scale = hp->dynamic_loss_scale ? (float)ldexp(1.0, hp->initial_scale_power)
                                       : (float)hp->static_loss_scale;
    st->good_steps = 0;
    st->step_t = 0;
    st->overflow_count = 0;
}

/* ------------------------------------------------------------------------- */
/* Reduce-scatter, emulated on one host: [P2] §3.3 (`reduce_scatter_tensor`
 * with op AVG or SUM; each rank keeps shard_size elements), [P1] numpy demo
 * (the reduce-scatter is an elementwise sum of the N full gradients followed
 * by the split), [P1] §PyTorch FSDP 使用 (reduce in fp32).  Then the loss
 * scale is divided out ([P3] §5.1 fp16 dynamic loss scale).
 *
 * Contributor c's value for flat element (rank r, i) sits at
 * grads[c*ld + rank_off + i] with rank_off = r*mul.  Elements whose flat
 * index is >= full_numel are padding: their gradient is zero.
 * For each element: acc = 0; acc += f32(grad_c) for c = 0..N-1 in order;
 * AVG divides by N; then g = acc / scale.
 * grad_kind: 0 fp16, 1 bf16, 2 fp32 contributions (fp32 when the reduce runs
 * in reduce_dtype=float32 end to end).                                      */
static float contribution(const void *grads, int32_t grad_kind, int64_t idx)
{
    if (grad_kind == 2) return ((const float *)grads)[idx];
    const uint16_t h = ((const uint16_t *)grads)[idx];
    return grad_kind == 1 ? ora_bf16_to_f32(h) : ora_f16_to_f32(h);
}

void ora_reduce_unscale(int32_t grad_kind, const void *grads, int64_t ld,
                        int64_t rank_off, int32_t n_contrib, int64_t count,
                        int64_t first_flat_index, int64_t full_numel, int32_t avg,
                        float scale, float *g_out)
{
    for (int64_t i = 0; i < count; ++i) {
        if (first_flat_index + i >= full_numel) {
            g_out[i] = 0.0f;
            continue;
        }
        float acc = 0.0f;
        for (int32_t c = 0; c < n_contrib; ++c)
            acc = acc + contribution(grads, grad_kind, (int64_t)c * ld + rank_off + i);
        if (avg) acc = acc / (float)n_contrib;
        g_out[i] = acc / scale;
    }
}

/* Overflow check and the squared L2 norm, computed exactly.
 * [P3] §5.3 (second pitfall): the overflow decision and the clipping must be
 * one global decision, taken on the whole gradient.
 * The norm's plain definition, sqrt(sum g_i^2), is evaluated exactly: the
 * square of a binary32 value is exact in binary64 (24 + 24 significant bits)
 * and its lowest set bit weighs no less than 2^-298 (the square of the
 * smallest subnormal).  A sum of up to 2^40 squares, each below 2^256, stays
 * below 2^297, so a 640-bit fixed-point integer whose unit is 2^-298 holds
 * every partial sum exactly, in any order.  ora_norm_sum rounds it once to
 * the nearest binary64 (ties to even).  Non-finite values only raise the
 * overflow flag (the step is skipped; the norm is then not used).          */
#define ORA_ACC_LIMBS 10
#define ORA_ACC_UNIT_EXP (-298)
typedef struct {
    uint64_t w[ORA_ACC_LIMBS];   /* little-endian 64-bit limbs */
} ora_exact_acc;

static void acc_add_at(ora_exact_acc *a, int limb, uint64_t x)
{
    for (int k = limb; k < ORA_ACC_LIMBS && x; ++k) {
        const uint64_t before = a->w[k];
        a->w[k] = before + x;
        x = a->w[k] < before;               /* carry */
    }
}

static void acc_add_square(ora_exact_acc *a, float gf)
{
    const double x = (double)gf * (double)gf;      /* exact */
    if (x == 0.0) return;
    int q;
    const double f = frexp(x, &q);                 /* x = f * 2^q, f in [0.5, 1) */
    uint64_t m = (uint64_t)ldexp(f, 53);           /* x = m * 2^(q-53), m < 2^53 */
    int off = q - 53 - ORA_ACC_UNIT_EXP;           /* bit position of m's unit */
    if (off < 0) {                                 /* the dropped low bits are 0 */
        m >>= -off;
        off = 0;
    }
    const int limb = off / 64, sh = off % 64;
    acc_add_at(a, limb, m << sh);
    if (sh) acc_add_at(a, limb + 1, m >> (64 - sh));
}

void ora_acc_clear(ora_exact_acc *a)
{
    memset(a, 0, sizeof(*a));
}

/* dst += src, exactly. */
void ora_acc_merge(ora_exact_acc *dst, const ora_exact_acc *src)
{
    uint64_t carry = 0;
    for (int k = 0; k < ORA_ACC_LIMBS; ++k) {
        const uint64_t a = dst->w[k], b = src->w[k];
        const uint64_t s1 = a + b;
        const uint64_t c1 = s1 < a;
        const uint64_t s2 = s1 + carry;
        const uint64_t c2 = s2 < s1;
        dst->w[k] = s2;
        carry = c1 | c2;
    }
}

static int acc_bit(const ora_exact_acc *a, int i)
{
    return (int)((a->w[i / 64] >> (i % 64)) & 1u);
}

/* The accumulated sum rounded to the nearest binary64, ties to even. */
double ora_norm_sum(const ora_exact_acc *a)
{
    int top = -1;
    for (int i = 64 * ORA_ACC_LIMBS - 1; i >= 0; --i)
        if (acc_bit(a, i)) { top = i; break; }
    if (top < 0) return 0.0;
    if (top < 53) {                               /* fits in 53 bits: exact */
        uint64_t v = 0;
        for (int i = top; i >= 0; --i) v = (v << 1) | (uint64_t)acc_bit(a, i);
        return ldexp((double)v, ORA_ACC_UNIT_EXP);
    }
    uint64_t mant = 0;                            /* the top 53 bits */
    for (int i = top; i > top - 53; --i) mant = (mant << 1) | (uint64_t)acc_bit(a, i);
    const int low = top - 53;                     /* highest discarded bit */
    const int round = acc_bit(a, low);
    int sticky = 0;
    for (int i = low - 1; i >= 0 && !sticky; --i) sticky = acc_bit(a, i);
    if (round && (sticky || (mant & 1u))) mant += 1;   /* may carry to 2^53: exact */
    return ldexp((double)mant, low + 1 + ORA_ACC_UNIT_EXP);
}

void ora_norm_accumulate(const float *g, int64_t n, ora_exact_acc *acc, int32_t *overflow)
{
    int32_t of = *overflow;
    for (int64_t i = 0; i < n; ++i) {
        if (!isfinite(g[i])) {
            of = 1;
            continue;
        }
        acc_add_square(acc, g[i]);
    }
    *overflow = of;
}

/* The decision after the norm is known: dynamic loss scale and clipping.
 * [P3] §5.1, §5.3: on overflow the step is skipped and the scale shrinks
 * (halved, not below min_loss_scale); after loss_scale_window consecutive
 * steps without overflow the scale grows (doubled).  The counter restarts on
 * an overflow and on a growth.  A static scale never changes; an overflow
 * still skips the step.  t counts applied steps only.
 * Clipping to gradient_clipping: q = max / (norm + 1e-6) in fp64; the
 * gradient is multiplied by (float)q when q < 1, else left alone.
 * Returns the clip coefficient and whether the step is skipped.             */
void ora_scaler_decide(const ora_hparams *hp, ora_scaler *st, int32_t overflow,
                       double norm, float *coef, int32_t *skip)
{
    if (overflow) {
        *skip = 1;
        *coef = 1.0f;
        st->overflow_count += 1;
        if (hp->dynamic_loss_scale) {
            const float s = st->scale / 2.0f;
            const float lo = (float)hp->min_loss_scale;
            st->scale = s < lo ? lo : s;
            st->good_steps = 0;
        }
        return;
    }
    *skip = 0;
    st->step_t += 1;
    float c = 1.0f;
    if (hp->max_grad_norm > 0.0) {
        const double q = hp->max_grad_norm / (norm + 1e-6);
        if (q < 1.0) c = (float)q;
    }
    *coef = c;
    if (hp->dynamic_loss_scale) {
        st->good_steps += 1;
        if (st->good_steps == hp->loss_scale_window) {
            st->scale = st->scale * 2.0f;
            st->good_steps = 0;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* AdamW on the fp32 master shard, then the cast into the flat buffer.
 * [P1] §ZeRO-Offload (the Adam equations, with bias correction):
 *     m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*g^2;
 *     mh = m / (1 - b1^t);  vh = v / (1 - b2^t);
 *     theta = theta - lr * mh / (sqrt(vh) + eps)
 * [P1] §ZeRO-1 step 2: each rank updates only its own 1/N slice.
 * [P3] §5.1: AdamW with weight_decay, applied decoupled: theta is first
 *     multiplied by (1 - lr*wd), then the Adam step is subtracted.
 * [P1] §ZeRO-1 step 3 / [P2] §3.2: the updated 16-bit shard is what the
 *     all-gather distributes, so it is written into rank r's slot of the
 *     flat, all-gather-shaped buffer.
 * The hyper-parameters arrive in fp64 (as a JSON config or a Python script
 * holds them); every scalar shared by all elements is formed in fp64 and
 * rounded to fp32 once: b1, b2, 1-b1, 1-b2, lr, eps,
 * bc1 = 1 - b1^t, bc2 = 1 - b2^t (pow), decay = 1 - lr*wd.  This is what the
 * numpy demo of [P1] (§用 numpy 模拟 ZeRO 分片过程) computes with float32
 * arrays and Python-float scalars.
 * The per-element order follows the equations left to right; the update
 * term is (lr * mh) / (sqrt(vh) + eps), as the demo evaluates it.          */
void ora_adamw_cast(const ora_hparams *hp, int64_t t, float coef, const float *g,
                    float *theta, float *m, float *v, int64_t n,
                    uint16_t *out, int32_t param_is_bf16)
{
    const float b1 = (float)hp->beta1, b2 = (float)hp->beta2;
    const float omb1 = (float)(1.0 - hp->beta1);
    const float omb2 = (float)(1.0 - hp->beta2);
    const float bc1 = (float)(1.0 - pow(hp->beta1, (double)t));
    const float bc2 = (float)(1.0 - pow(hp->beta2, (double)t));
    const float decay = (float)(1.0 - hp->lr * hp->weight_decay);
    const float lr = (float)hp->lr, eps = (float)hp->eps;
    for (int64_t i = 0; i < n; ++i) {
        const float gc = g[i] * coef;                      /* clipped gradient */
        const float mi = b1 * m[i] + omb1 * gc;             /* momentum */
        const float vi = b2 * v[i] + omb2 * (gc * gc);      /* variance */
        const float mh = mi / bc1;                          /* bias correction */
        const float vh = vi / bc2;
        float th = theta[i] * decay;                        /* decoupled decay */
        th = th - (lr * mh) / (sqrtf(vh) + eps);            /* Adam step */
        m[i] = mi;
        v[i] = vi;
        theta[i] = th;
        out[i] = param_is_bf16 ? ora_f32_to_bf16(th) : ora_f32_to_f16(th);
    }
}

/* ------------------------------------------------------------------------- */
/* The part of a step after the reduce: overflow check and global norm over
 * every stepped shard's reduced gradient g (plus extra_norm_sq, the other
 * ranks' share) -> loss-scale decision and clip coefficient -> AdamW + cast
 * into each rank's slot of the flat buffer.  g holds n_ranks rows of
 * shard_size.  A skipped step leaves master, m, v, t and the flat buffer
 * untouched.                                                               */
static void apply_step(const ora_hparams *hp, ora_scaler *st, int64_t shard_size,
                       int32_t param_is_bf16, const int32_t *ranks, int32_t n_ranks,
                       const float *g, float *const *master, float *const *m,
                       float *const *v, uint16_t *flat_out, double extra_norm_sq,
                       float scale_used, ora_result *res)
{
    ora_exact_acc acc;
    ora_acc_clear(&acc);
    int32_t overflow = 0;
    for (int32_t j = 0; j < n_ranks; ++j)
        ora_norm_accumulate(g + (int64_t)j * shard_size, shard_size, &acc, &overflow);
    const double norm = sqrt(ora_norm_sum(&acc) + extra_norm_sq);
    float coef;
    int32_t skip;
    ora_scaler_decide(hp, st, overflow, norm, &coef, &skip);
    if (!skip) {
        for (int32_t j = 0; j < n_ranks; ++j) {
            const int64_t r = ranks[j];
            ora_adamw_cast(hp, st->step_t, coef, g + (int64_t)j * shard_size,
                           master[j], m[j], v[j], shard_size,
                           flat_out + r * shard_size, param_is_bf16);
        }
    }
    if (res) {
        res->overflow = overflow;
        res->skipped = skip;
        res->grad_norm = norm;
        res->clip_coef = coef;
        res->scale_used = scale_used;
    }
}

static int check_ranks(const int32_t *ranks, int32_t n_ranks, int32_t world_size)
{
    if (!ranks || n_ranks < 1 || world_size < 1) return ORA_EINVAL;
    for (int32_t j = 0; j < n_ranks; ++j)
        if (ranks[j] < 0 || ranks[j] >= world_size) return ORA_EINVAL;
    return ORA_OK;
}

static float *alloc_rows(int64_t shard_size, int32_t n_ranks)
{
    return (float *)malloc(sizeof(float) * (size_t)(shard_size ? shard_size : 1) *
                           (size_t)n_ranks);
}

/* One ZeRO shard step for the stepped ranks ranks[0..n_ranks) (one rank, or
 * all N in an emulation of the whole group): reduce-scatter + unscale of each
 * stepped shard, then apply_step.  master[j], m[j], v[j] point at rank
 * ranks[j]'s shard_size elements.                                           */
int ora_shard_step(const ora_hparams *hp, ora_scaler *st, int32_t world_size,
                   int64_t full_numel, int64_t shard_size, int32_t grad_kind,
                   int32_t param_is_bf16, int32_t avg, const int32_t *ranks,
                   int32_t n_ranks, const void *grads, int64_t ld,
                   int64_t rank_mul, float *const *master, float *const *m,
                   float *const *v, uint16_t *flat_out, double extra_norm_sq,
                   ora_result *res)
{
    if (!hp || !st || shard_size < 0 || check_ranks(ranks, n_ranks, world_size))
        return ORA_EINVAL;
    float *g = alloc_rows(shard_size, n_ranks);
    if (!g) return ORA_EOVERFLOW;
    const float scale_used = st->scale;
    for (int32_t j = 0; j < n_ranks; ++j) {
        const int64_t r = ranks[j];
        ora_reduce_unscale(grad_kind, grads, ld, r * rank_mul, world_size, shard_size,
                           r * shard_size, full_numel, avg, scale_used,
                           g + (int64_t)j * shard_size);
    }
    apply_step(hp, st, shard_size, param_is_bf16, ranks, n_ranks, g, master, m, v,
               flat_out, extra_norm_sq, scale_used, res);
    free(g);
    return ORA_OK;
}

/* Gradient accumulation across micro-steps.  [P1] §实践要点 (gradient
 * accumulation): the loss is divided by the number of micro-steps and the
 * micro-steps' gradients add up before one optimizer step; [P3] §5.1
 * (contiguous_gradients) and §5.3: the reduced gradient partitions live in
 * one contiguous buffer and accumulate there.  Reading: every micro-step's
 * contributions are reduced exactly as in the step (fp32, contributor order,
 * AVG) and added into the rank's fp32 accumulator:
 *     r = reduce(grads);  acc = first ? r : acc + r.
 * The loss scale stays in the accumulator until the optimizer step.         */
int ora_grad_accumulate(int32_t world_size, int64_t full_numel, int64_t shard_size,
                        int32_t grad_kind, int32_t avg, const int32_t *ranks,
                        int32_t n_ranks, const void *grads, int64_t ld, int64_t rank_mul,
                        float *const *acc, int32_t first)
{
    if (shard_size < 0 || check_ranks(ranks, n_ranks, world_size)) return ORA_EINVAL;
    float *r = alloc_rows(shard_size, 1);
    if (!r) return ORA_EOVERFLOW;
    for (int32_t j = 0; j < n_ranks; ++j) {
        const int64_t rk = ranks[j];
        ora_reduce_unscale(grad_kind, grads, ld, rk * rank_mul, world_size, shard_size,
                           rk * shard_size, full_numel, avg, 1.0f, r);
        for (int64_t i = 0; i < shard_size; ++i)
            acc[j][i] = first ? r[i] : acc[j][i] + r[i];
    }
    free(r);
    return ORA_OK;
}

/* The gradient of a step taken from accumulators: the loss scale comes out
 * once, at the optimizer step ([P1] §实践要点, gradient accumulation):
 * g = acc / scale for the `count` elements from flat index first_flat_index;
 * padding elements (flat index >= full_numel) count as zero.               */
void ora_unscale_acc(const float *acc, int64_t count, int64_t first_flat_index,
                     int64_t full_numel, float scale, float *g_out)
{
    for (int64_t i = 0; i < count; ++i)
        g_out[i] = first_flat_index + i >= full_numel ? 0.0f : acc[i] / scale;
}

/* The optimizer step on accumulated shards: ora_unscale_acc, then
 * apply_step.                                                               */
int ora_shard_step_acc(const ora_hparams *hp, ora_scaler *st, int32_t world_size,
                       int64_t full_numel, int64_t shard_size, int32_t param_is_bf16,
                       const int32_t *ranks, int32_t n_ranks, const float *const *acc,
                       float *const *master, float *const *m, float *const *v,
                       uint16_t *flat_out, double extra_norm_sq, ora_result *res)
{
    if (!hp || !st || shard_size < 0 || check_ranks(ranks, n_ranks, world_size))
        return ORA_EINVAL;
    float *g = alloc_rows(shard_size, n_ranks);
    if (!g) return ORA_EOVERFLOW;
    const float scale_used = st->scale;
    for (int32_t j = 0; j < n_ranks; ++j)
        ora_unscale_acc(acc[j], shard_size, (int64_t)ranks[j] * shard_size, full_numel,
                        scale_used, g + (int64_t)j * shard_size);
    apply_step(hp, st, shard_size, param_is_bf16, ranks, n_ranks, g, master, m, v,
               flat_out, extra_norm_sq, scale_used, res);
    free(g);
    return ORA_OK;
}

/* ZeRO++ quantized weight communication ([P1] §ZeRO++: the parameter shard
 * is quantized to int8/int4 before the all-gather and dequantized by the
 * receiver, halving the traffic; [P3] §4.2: the 2-byte fp16 weights go out
 * as INT8 and are restored before local use).  The pages give no scheme.
 * Reading: symmetric absmax int8 over blocks of `block` consecutive elements
 * of each rank's shard (the last block may be short), applied to the 16-bit
 * parameter value that would otherwise be all-gathered (decoded exactly to
 * fp32):
 *     amax = max |p| over the block (NaN ignored);  scale = amax / 127;
 *     q = 0 if scale == 0 or p/scale is NaN, else clamp(rint(p/scale), -127, 127)
 * with rint rounding half to even; the receiver uses q * scale.
 * p: n decoded parameter values; q: n codes; scales: ceil(n/block) floats. */
void ora_quantize_q8(const float *p, int64_t n, int32_t block, int8_t *q, float *scales)
{
    for (int64_t b0 = 0, k = 0; b0 < n; b0 += block, ++k) {
        const int64_t b1 = b0 + block < n ? b0 + block : n;
        float amax = 0.0f;
        for (int64_t i = b0; i < b1; ++i) {
            const float a = fabsf(p[i]);
            if (a > amax) amax = a;                   /* NaN compares false: ignored */
        }
        const float scale = amax / 127.0f;
        scales[k] = scale;
        for (int64_t i = b0; i < b1; ++i) {
            int32_t code = 0;
            if (scale != 0.0f) {
                const float v = p[i] / scale;
                if (!isnan(v)) {
                    const float r = rintf(v);         /* default mode: half to even */
                    code = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int32_t)r);
                }
            }
            q[i] = (int8_t)code;
        }
    }
}

/* Array form of the casts, for exhaustive checks. */
void ora_cast_array(const float *in, int64_t n, uint16_t *out, int32_t to_bf16)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = to_bf16 ? ora_f32_to_bf16(in[i]) : ora_f32_to_f16(in[i]);
}

void ora_decode_array(const uint16_t *in, int64_t n, float *out, int32_t from_bf16)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = from_bf16 ? ora_bf16_to_f32(in[i]) : ora_f16_to_f32(in[i]);
}

/* Plain data parallelism for comparison ([P3] §5.2: ZeRO follows the same
 * optimizer update sequence as DDP): every contributor's full gradient is
 * all-reduced, and the whole flat parameter is updated on one replica.
 * grads: N rows of at least full_numel elements, row stride ld.            */
int ora_ddp_step(const ora_hparams *hp, ora_scaler *st, int32_t n_contrib,
                 int64_t full_numel, int32_t grad_kind, int32_t param_is_bf16,
                 int32_t avg, const void *grads, int64_t ld, float *master,
                 float *m, float *v, uint16_t *out, ora_result *res)
{
    if (!hp || !st || n_contrib < 1 || full_numel < 0) return ORA_EINVAL;
    float *g = alloc_rows(full_numel, 1);
    if (!g) return ORA_EOVERFLOW;
    const float scale_used = st->scale;
    ora_reduce_unscale(grad_kind, grads, ld, 0, n_contrib, full_numel, 0, full_numel, avg,
                       scale_used, g);
    const int32_t rank0 = 0;
    apply_step(hp, st, full_numel, param_is_bf16, &rank0, 1, g, &master, &m, &v, out, 0.0,
               scale_used, res);
    free(g);
    return ORA_OK;
}
