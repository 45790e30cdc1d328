/*
 * zero.h -- C ABI of the GB300 ZeRO shard optimizer step on a FlatParameter.
 *
 * One call of zero_shard_step performs, for the stepped shard(s) of a flat
 * parameter split N ways:
 *   1. the reduce of the N per-rank fp16/bf16 gradient contributions of the
 *      shard (SUM or AVG, accumulated in fp32) -- the reduce half of a
 *      reduce-scatter, with all N contributions already in this GPU's memory;
 *   2. division by the loss scale and an inf/NaN overflow check;
 *   3. the global L2 gradient norm and the clip coefficient;
 *   4. the dynamic-loss-scale decision (overflow: skip the step and halve the
 *      scale; after `loss_scale_window` clean steps: double it);
 *   5. AdamW with bias correction and decoupled weight decay on the fp32
 *      master weights, m and v;
 *   6. the round-to-nearest cast of the updated shard into its slot of the
 *      flat, all-gather-shaped 16-bit parameter buffer.
 *
 * Sources (web pages, by title and section):
 *   "DeepSpeed 与 FSDP" (docs.ifdog.com): §逐步推导 (16 bytes per parameter),
 *     §ZeRO-1/2/3 and §ZeRO-3 的数学总结 (sharded update, reduce-scatter,
 *     all-gather, per-stage memory), §ZeRO-Offload (Adam equations),
 *     §FSDP 的分片粒度与 FlatParameter (flat buffer, chunk per rank).
 *   "PyTorch FSDP（Fully Sharded Data Parallel）源码级深度解析" (tbr8.org):
 *     §3.1 (FlatParameter and its per-parameter {start, end, shape, dtype}
 *     table), §3.3 (reduce_scatter_tensor with op AVG or SUM, shard_size),
 *     §4 (ShardingStrategy), §7.2 (fp32 master weights under bf16 compute).
 *   The ZeRO paper reading at 2kiu.com/news/5312103: §5.1 (DeepSpeed config:
 *     AdamW lr/betas/eps/weight_decay, fp16 loss_scale 0 = dynamic,
 *     loss_scale_window, initial_scale_power, gradient_clipping), §5.3
 *     (overflow detection and clipping are one global decision).
 *
 * Conventions for every function:
 *   - Returns a zero_status; never aborts, never throws, never exits.
 *   - On an error nothing is launched and no state changes.
 *   - Device pointers are plain CUDA device addresses on the device the
 *     handle was created on; the caller owns every buffer it passes and keeps
 *     it alive until the work queued on `stream` has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - The library needs the CUDA driver; it contains no CPU fallback (the
 *     host update of the offload mode is a mode the caller picks, below).
 *   - A handle is not thread-safe: calls on one handle must not overlap.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZERO_OK = 0,
    ZERO_ERR_INVALID_ARG = 1,       /* null pointer, bad size, rank out of range ... */
    ZERO_ERR_UNSUPPORTED_DTYPE = 2, /* dtype not fp16/bf16 */
    ZERO_ERR_ALIGNMENT = 3,         /* pointer not aligned to its element size */
    ZERO_ERR_CUDA = 4,              /* a CUDA runtime call failed (see zero_last_error) */
    ZERO_ERR_OVERFLOW_SIZE = 5,     /* a size or offset does not fit in int64 */
    ZERO_ERR_TIMEOUT = 6,           /* a bounded device wait gave up (in this step, or in an
                                       accumulation since the last step): the step was
                                       skipped.  Fail-stop: every later step is skipped too
                                       until a call that reads a step result reports this
                                       status, which clears the condition */
    ZERO_ERR_NO_MEMORY = 7          /* host or device allocation failed */
} zero_status;

/* ZERO_F32 is a gradient dtype only: fp32 contributions, as a reduce-scatter
 * in reduce_dtype=float32 delivers them ("DeepSpeed 与 FSDP", MixedPrecision
 * example).  Parameters are always 16-bit. */
typedef enum { ZERO_F16 = 0, ZERO_BF16 = 1, ZERO_F32 = 2 } zero_dtype;

/* reduce_scatter_tensor's op ("PyTorch FSDP ... 深度解析" §3.3). */
typedef enum { ZERO_SUM = 0, ZERO_AVG = 1 } zero_reduce_op;

/* One row of the FlatParameter's parameter table ("PyTorch FSDP ... 深度解析"
 * §3.1: start = offset, end = offset + numel, shape, dtype).  Rows must be
 * contiguous and in order: offset[0] == 0, offset[k] == offset[k-1] +
 * numel[k-1]; numel == prod(shape[0..ndim)) (ndim 0 means a scalar,
 * numel 1); 0 <= ndim <= 8; dtype is the parameter's 16-bit dtype. */
typedef struct {
    int64_t offset;
    int64_t numel;
    int32_t ndim;
    int32_t dtype;                  /* zero_dtype */
    int64_t shape[8];
} zero_param_info;

/* Optimizer and loss-scale settings, named after the DeepSpeed config keys
 * (ZeRO reading §5.1).  Reals are fp64 as a config file holds them; every
 * per-element scalar is rounded to fp32 once from fp64: beta1, beta2,
 * 1-beta1, 1-beta2, lr, eps, 1-lr*weight_decay, and the bias corrections
 * 1-beta^t (t = number of applied steps, computed with pow in fp64). */
typedef struct {
    double lr;                      /* 3e-5 in the printed config */
    double beta1, beta2;            /* 0.9, 0.999 */
    double eps;                     /* 1e-8 */
    double weight_decay;            /* 0.01, decoupled: theta *= 1 - lr*wd */
    double max_grad_norm;           /* gradient_clipping, 1.0; <= 0 disables */
    int32_t dynamic_loss_scale;     /* 1: "loss_scale": 0 (dynamic); 0: static */
    int32_t initial_scale_power;    /* 16: initial scale 2^16 */
    int32_t loss_scale_window;      /* 1000 clean steps before doubling (>= 1) */
    int32_t reserved;               /* must be 0 */
    double static_loss_scale;       /* used when dynamic_loss_scale == 0 (> 0) */
    double min_loss_scale;          /* floor of the dynamic scale (> 0), 1.0 */
} zero_hparams;

/* Loss-scale state (lives on the device). */
typedef struct {
    float scale;                    /* scale applied to the next step's gradients */
    int32_t good_steps;             /* consecutive clean steps since the last change */
    int64_t step_t;                 /* applied (not skipped) steps: Adam's t */
    int64_t overflow_count;         /* skipped steps so far */
} zero_scaler_state;

/* What one step did. */
typedef struct {
    int32_t overflow;               /* 1 if any reduced gradient was inf/NaN */
    int32_t skipped;                /* 1 if the update was skipped */
    double grad_norm;               /* global L2 norm of the unscaled gradient */
    float clip_coef;                /* factor applied to the gradient (1 = no clip) */
    float scale_used;               /* loss scale the gradients were divided by */
} zero_step_result;

typedef struct zero_flat zero_flat; /* opaque handle */

/* Create a handle for a FlatParameter sharded `world_size` ways.
 * Layout ("PyTorch FSDP ... 深度解析" §3.1, §3.3; "DeepSpeed 与 FSDP"
 * §FSDP 的分片粒度与 FlatParameter): full_numel = sum of numel;
 * shard_size S = ceil(full_numel / world_size); padded_numel = world_size*S;
 * rank r owns flat elements [r*S, (r+1)*S); elements >= full_numel are
 * padding and carry a zero gradient.
 * grad_dtype: ZERO_F16, ZERO_BF16 or ZERO_F32; param_dtype: ZERO_F16 or
 * ZERO_BF16.  op: ZERO_SUM / ZERO_AVG.
 * The handle binds to the current CUDA device and allocates there the
 * loss-scale state, the per-step scalars and the bias-correction table
 * (a few hundred KB).  The scratch of a step (an fp32 reduced-gradient row of
 * S floats per stepped rank, plus norm partials) is allocated on the first
 * step that needs it and kept: do the first step before any stream capture.
 * *out receives the handle; free it with zero_flat_free.
 * Errors: INVALID_ARG (null, n_infos < 1, world_size < 1, table not
 * contiguous, shape/numel mismatch, bad hparams), UNSUPPORTED_DTYPE,
 * OVERFLOW_SIZE, NO_MEMORY, CUDA. */
zero_status zero_flat_init(const zero_param_info *infos, int32_t n_infos, int32_t world_size,
                           zero_dtype grad_dtype, zero_dtype param_dtype, zero_reduce_op op,
                           const zero_hparams *hp, zero_flat **out);

/* full_numel, shard_size and padded_numel of the handle (any may be NULL):
 * the layout zero_flat_init computed ("PyTorch FSDP ... 深度解析" §3.3,
 * shard_size from the flat parameter's numel and world_size, padded so every
 * rank's chunk is equal; "DeepSpeed 与 FSDP" §FSDP 的分片粒度与 FlatParameter,
 * one flat buffer cut into world_size chunks).  Host only.
 * Errors: INVALID_ARG (NULL handle). */
zero_status zero_flat_layout(const zero_flat *h, int64_t *full_numel, int64_t *shard_size,
                             int64_t *padded_numel);

/* One optimizer step on the stepped ranks ranks[0..n_ranks) (distinct, each
 * in [0, world_size); one rank for a real rank's step, or all N to emulate
 * the whole group on one GPU -- the norm and the overflow flag are then
 * global over every stepped shard).  The step of "DeepSpeed 与 FSDP" §ZeRO-1
 * steps 1-3 (each rank updates its own slice of the optimizer state and
 * writes its slice of the parameters for the all-gather) with the reduce of
 * "PyTorch FSDP ... 深度解析" §3.3 and the mixed-precision, loss-scale and
 * clipping settings of the ZeRO reading §5.1 and §5.3.
 *
 * grads: device, grad_dtype (aligned to its element size); contributor c's
 * gradient for flat element
 *   (rank r, i) is grads[c*grad_ld + r*grad_rank_offset_mul + i],
 *   c in [0, world_size), i in [0, S).  Use grad_ld = padded_numel,
 *   grad_rank_offset_mul = S when each contributor holds the whole padded
 *   flat gradient (the reduce-scatter input), or grad_ld >= S,
 *   grad_rank_offset_mul = 0 when the buffer holds only the stepped rank's
 *   slice of each contribution.  Every addressed element must be readable;
 *   padding elements are not read.  16-byte aligned rows take the vector path.
 * master[j], m[j], v[j]: device fp32, S elements each, rank ranks[j]'s
 *   shard, updated in place (host arrays of n_ranks device pointers).
 * flat_param_out: device, param_dtype, padded_numel elements; rank r's
 *   slot [r*S, (r+1)*S) is overwritten with the cast master shard.  Other
 *   slots are not touched.
 * extra_norm_sq: sum of squared norms of shards not stepped here (other
 *   ranks' share of the global norm); 0 when every shard is stepped or in a
 *   one-rank emulation.
 * res: NULL for a fully asynchronous step; otherwise the step's result is
 *   copied back and `stream` is synchronized before returning.
 * A skipped (overflowed) step leaves master, m, v, step_t and the flat
 * buffer untouched.  Results are deterministic for a given device.
 * Errors: INVALID_ARG, ALIGNMENT (grads not aligned to their element size,
 * out not 2-byte or master/m/v not 4-byte aligned), OVERFLOW_SIZE,
 * NO_MEMORY, CUDA. */
zero_status zero_shard_step(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                            const void *grads, int64_t grad_ld, int64_t grad_rank_offset_mul,
                            float *const *master, float *const *m, float *const *v,
                            void *flat_param_out, double extra_norm_sq, void *stream,
                            zero_step_result *res);

/* Elements per int8 quantization block of the all-gather payload. */
#define ZERO_Q8_BLOCK 256

/* zero_shard_step that also writes the ZeRO++ quantized weight payload
 * ("DeepSpeed 与 FSDP" §ZeRO++: the parameter shard is quantized to int8
 * before the all-gather and dequantized by the receiver, halving the fp16
 * traffic; ZeRO reading §4.2).  Scheme (the pages give none): for every
 * block of ZERO_Q8_BLOCK consecutive elements of a rank's shard (the last
 * block may be short), with p the 16-bit parameter value decoded to fp32,
 *     amax = max |p| (NaN ignored); scale = amax / 127;
 *     q = 0 if scale == 0 or p/scale is NaN, else clamp(rint(p/scale), +-127)
 * (rint: half to even); the receiver uses q * scale.
 * flat_q8_out: device int8, padded_numel elements; rank r's codes go to
 *   [r*S, (r+1)*S).  q8_scales: device fp32, world_size * ceil(S/256)
 *   elements; rank r's scales at [r*nb, (r+1)*nb), nb = ceil(S/256).
 * flat_param_out may be NULL (then only the int8 payload is written).
 * Other arguments, skip semantics and errors as for zero_shard_step. */
zero_status zero_shard_step_q8(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                               const void *grads, int64_t grad_ld, int64_t grad_rank_offset_mul,
                               float *const *master, float *const *m, float *const *v,
                               void *flat_param_out, int8_t *flat_q8_out, float *q8_scales,
                               double extra_norm_sq, void *stream, zero_step_result *res);

/* Gradient accumulation across micro-steps ("DeepSpeed 与 FSDP" §实践要点,
 * gradient accumulation: the loss is divided by the number of micro-steps
 * and their gradients add up before one optimizer step; ZeRO reading §5.1,
 * contiguous_gradients: the reduced gradient partitions live in one
 * contiguous buffer).  For each stepped rank j the micro-step's N
 * contributions are reduced exactly as zero_shard_step reduces them (fp32,
 * contributor order, AVG per the handle's op) and
 *     acc[j][i] = first_micro_step ? r : acc[j][i] + r.
 * The loss scale is not divided out here; zero_shard_step_accumulated does
 * that.  grads: as for zero_shard_step.  acc[j]: device fp32, shard_size
 * elements per stepped rank, caller-owned (one contiguous buffer of
 * n_ranks * shard_size works).  Padding elements accumulate zero.
 * Asynchronous on `stream`; no norm, no state change.
 * Errors: INVALID_ARG, ALIGNMENT, OVERFLOW_SIZE, CUDA. */
zero_status zero_grad_accumulate(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                 const void *grads, int64_t grad_ld, int64_t grad_rank_offset_mul,
                                 float *const *acc, int32_t first_micro_step, void *stream);

/* The optimizer step on accumulated shards ("DeepSpeed 与 FSDP" §实践要点,
 * gradient accumulation: one optimizer step after the micro-steps' gradients
 * have been summed): g = acc[j] / scale (padding elements count as zero),
 * then the overflow check, global norm, loss-scale decision, AdamW and cast
 * exactly as in zero_shard_step.  acc is only read.
 * Other arguments and errors as for zero_shard_step. */
zero_status zero_shard_step_accumulated(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                        const float *const *acc, float *const *master,
                                        float *const *m, float *const *v, void *flat_param_out,
                                        double extra_norm_sq, void *stream, zero_step_result *res);

/* The step split at its global decision ("overflow detection and clipping are
 * one global decision", ZeRO reading §5.3): for a rank that steps several
 * FlatParameters (one handle each, "PyTorch FSDP ... 深度解析" §3.1: one
 * FlatParameter per wrapped module) with one clip norm and one loss-scale
 * decision, and the point where a multi-GPU caller would all-reduce the two
 * scalars across ranks.
 *
 * zero_shard_reduce: K1 exactly as in zero_shard_step -- the reduce, unscale
 * (by the handle's current loss scale), overflow check and norm partials,
 * the unscaled gradient rows kept in the handle's scratch -- and its last
 * block writes this handle's totals to DEVICE memory:
 *     *norm_sq_out = sum of g^2 over the stepped shards (fp64),
 *     *overflow_out = 1 if any g is inf/NaN, else 0.
 * No decision, no state change.  norm_sq_out 8-byte and overflow_out 4-byte
 * aligned device pointers.  Asynchronous on `stream`.
 *
 * zero_shard_apply: the decision from the caller's totals -- *norm_sq (the
 * SUM of the norm_sq_out of every FlatParameter the decision covers, and of
 * every rank's) and *overflow (their MAX), both device memory -- through the
 * handle's loss-scale state machine exactly as zero_shard_step decides, then
 * AdamW and the cast on the gradient rows the preceding zero_shard_reduce
 * left.  Each handle of a group applies the same totals, so all take the
 * same skip / clip / scale decision.  `ranks` must equal those of the
 * preceding zero_shard_reduce on this handle, with no other step on the
 * handle in between, and `stream` must be ordered after that reduce and after
 * the writes of the totals.  res: as for zero_shard_step.
 *
 * zero_shard_reduce followed by zero_shard_apply with its own totals is
 * bit-identical to zero_shard_step.  Errors: as for zero_shard_step;
 * INVALID_ARG for NULL totals or ranks that differ from the reduce's (or no
 * pending reduce); ALIGNMENT for misaligned totals. */
zero_status zero_shard_reduce(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                              const void *grads, int64_t grad_ld, int64_t grad_rank_offset_mul,
                              double *norm_sq_out, int32_t *overflow_out, void *stream);

/* The first half of a split step taken from micro-step accumulators
 * ("DeepSpeed 与 FSDP" §实践要点, gradient accumulation; ZeRO reading §5.1,
 * contiguous_gradients, and §5.3, one decision): for each stepped rank j,
 * g = acc[j] / scale (the handle's current loss scale; padding elements
 * zero) into the handle's gradient rows, the overflow check and this
 * handle's norm^2 and flag written to DEVICE memory as zero_shard_reduce
 * writes them.  zero_shard_apply / zero_shard_apply_partials then decide and
 * update as after zero_shard_reduce; the pair equals
 * zero_shard_step_accumulated on the same accumulators.  acc: device fp32,
 * shard_size elements per stepped rank (4-byte aligned), only read.  Errors:
 * as for zero_shard_reduce. */
zero_status zero_shard_reduce_accumulated(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                          const float *const *acc, double *norm_sq_out,
                                          int32_t *overflow_out, void *stream);
zero_status zero_shard_apply(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                             float *const *master, float *const *m, float *const *v,
                             void *flat_param_out, const double *norm_sq,
                             const int32_t *overflow, void *stream, zero_step_result *res);

/* zero_shard_apply with the cross-rank exchange left as an all-gather: the
 * one global decision of the ZeRO reading §5.3 (overflow and clipping taken
 * over every rank's gradient) from n_parts per-rank partials in device
 * memory -- norm_sq_parts[k] (fp64) and overflow_parts[k] (int32), k <
 * n_parts, e.g. every rank's zero_shard_reduce outputs gathered in rank order
 * -- totalled on the device (the squared norms summed in one fixed order, the
 * flags OR-ed), so every rank that applies the same gathered arrays takes
 * bit for bit the same skip / clip / scale decision, whatever the collective
 * library's reduction order.  Then AdamW and the cast as zero_shard_apply.
 * Other arguments, requirements and errors as for zero_shard_apply;
 * INVALID_ARG for n_parts outside [1, 2^20]. */
zero_status zero_shard_apply_partials(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                      float *const *master, float *const *m, float *const *v,
                                      void *flat_param_out, const double *norm_sq_parts,
                                      const int32_t *overflow_parts, int32_t n_parts,
                                      void *stream, zero_step_result *res);

/* zero_shard_apply_partials that also writes the ZeRO++ int8 weight payload
 * ("DeepSpeed 与 FSDP" §ZeRO++; ZeRO reading §4.2: the parameter shard goes
 * to the all-gather as int8 codes and block scales, half the bytes of fp16),
 * exactly as zero_shard_step_q8 writes it: flat_q8_out (device int8,
 * padded_numel elements, rank r's codes at [r*S, (r+1)*S)) and q8_scales
 * (device fp32, world_size * ceil(S/256), rank r's at [r*nb, (r+1)*nb)).
 * flat_param_out may be NULL (only the payload is written).  The decision
 * from the gathered partials as in zero_shard_apply_partials.  Errors: as for
 * zero_shard_apply_partials; INVALID_ARG for NULL int8 outputs, ALIGNMENT for
 * q8_scales not 4-byte aligned. */
zero_status zero_shard_apply_partials_q8(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                         float *const *master, float *const *m,
                                         float *const *v, void *flat_param_out,
                                         int8_t *flat_q8_out, float *q8_scales,
                                         const double *norm_sq_parts,
                                         const int32_t *overflow_parts, int32_t n_parts,
                                         void *stream, zero_step_result *res);

/* A group: the FlatParameters one rank steps together ("PyTorch FSDP ...
 * 深度解析" §3.1: one FlatParameter per wrapped module) with one clip norm and
 * one loss-scale decision (ZeRO reading §5.3), in one reduce launch and one
 * AdamW launch per 64 (member, stepped rank) rows instead of two launches per
 * FlatParameter.  The members are existing handles that share world_size,
 * grad and param dtypes, op and every zero_hparams field but lr and
 * weight_decay: each member keeps its own two, as a parameter group does
 * ("PyTorch FSDP ... 深度解析" §8, the comparison table: DeepSpeed shards by
 * parameter group), so e.g. biases and norms can step without decay in the
 * same launches.  The rest comes from the first member.  The group owns its
 * own loss-scale state (initialised as a new handle's), bias-correction
 * table and norm partials; the members' own loss-scale states are not used
 * by group steps.
 * A member's handle supplies its layout and its reduced-gradient scratch, so
 * a handle should be stepped either alone or in groups, not both in one
 * step.  The group does not own its members: they must outlive every group
 * call, and zero_group_free leaves them open.  Errors: INVALID_ARG (no
 * members, NULL, members that differ, a member listed twice, members on
 * another device), NO_MEMORY, CUDA. */
typedef struct zero_group zero_group;
zero_status zero_group_init(zero_flat *const *members, int32_t n_members, zero_group **out);

/* The arguments of one member in a group call, those of zero_shard_step /
 * zero_grad_accumulate / zero_shard_step_accumulated / zero_shard_step_q8
 * for that member's handle; each call reads the fields it needs (acc: the
 * member's per-rank fp32 accumulators, used by the accumulation calls only;
 * flat_q8_out and q8_scales: the member's int8 payload, zero_group_step_q8
 * only). */
typedef struct {
    const int32_t *ranks;
    int32_t n_ranks;
    const void *grads;
    int64_t grad_ld;
    int64_t grad_rank_offset_mul;
    float *const *master;
    float *const *m;
    float *const *v;
    void *flat_param_out;
    float *const *acc;
    int8_t *flat_q8_out;
    float *q8_scales;
} zero_group_member;

/* One step of every member (args[k] for the group's member k): the reduce
 * of every member's stepped shards with the group's loss scale, one global
 * norm over all of them plus extra_norm_sq, one overflow decision and loss-
 * scale update (ZeRO reading §5.3: one decision for everything the rank
 * steps), then AdamW and the cast into every member's slot -- the same
 * per-element arithmetic as zero_shard_step.  Asynchronous on `stream` when
 * res is NULL.  Errors: as for zero_shard_step, per member. */
zero_status zero_group_step(zero_group *g, const zero_group_member *args, double extra_norm_sq,
                            void *stream, zero_step_result *res);

/* zero_group_step that also writes every member's int8 all-gather payload
 * ("DeepSpeed 与 FSDP" §ZeRO++; ZeRO reading §4.2) and its block scales, as
 * zero_shard_step_q8 does per member (the same
 * quantization of the same 16-bit values; flat_param_out may be NULL).
 * One reduce launch and one int8-payload AdamW launch per 64 rows.  Errors:
 * as for zero_shard_step_q8, per member. */
zero_status zero_group_step_q8(zero_group *g, const zero_group_member *args, double extra_norm_sq,
                               void *stream, zero_step_result *res);

/* Micro-step accumulation for every member in one launch per 64 rows
 * ("DeepSpeed 与 FSDP" §实践要点, gradient accumulation), as
 * zero_grad_accumulate does per member (acc = r on the first micro-step,
 * acc += r after; the loss scale not divided out).  Reads ranks, grads,
 * grad_ld, grad_rank_offset_mul and acc of each member.  Asynchronous.
 * Errors: as for zero_grad_accumulate, per member. */
zero_status zero_group_accumulate(zero_group *g, const zero_group_member *args,
                                  int32_t first_micro_step, void *stream);

/* The step from every member's accumulators ("DeepSpeed 与 FSDP" §实践要点,
 * gradient accumulation): g = acc / scale (padding zero),
 * one global norm, overflow decision and loss-scale update over all members
 * (ZeRO reading §5.3),
 * then AdamW and the cast -- as zero_shard_step_accumulated does per member,
 * in one norm launch and one AdamW launch per 64 rows.  Reads ranks, acc,
 * master, m, v and flat_param_out of each member.  res: as for
 * zero_shard_step.  Errors: as for zero_shard_step_accumulated, per member. */
zero_status zero_group_step_accumulated(zero_group *g, const zero_group_member *args,
                                        double extra_norm_sq, void *stream,
                                        zero_step_result *res);

/* The ZeRO-Offload form of zero_group_step ("DeepSpeed 与 FSDP"
 * §ZeRO-Offload; ZeRO reading §4.1), as zero_shard_step_offload does
 * per member: one reduce launch per 64 rows with the group's decision, then
 * every member's update split at split_k = gpu_share * shard_size_k (rounded
 * down to 65536 elements, or the whole shard for gpu_share = 1): elements
 * [0, split_k) of every row by one GPU AdamW launch per 64 rows over the
 * host-resident state, the rest by `n_threads` host threads of the group
 * (0: every CPU this process may run on) working through all members' rows
 * at once, the gradient rows coming down in segments and the 16-bit
 * parameters going back segment by segment, as for one handle.  Each member
 * keeps its own lr and weight decay.  Bit-identical to zero_group_step for
 * any split.  master, m, v: HOST fp32 arrays, as for zero_shard_step_offload;
 * flat_param_out: device; the other fields as for zero_group_step.  The
 * group owns the streams and threads; each member's handle owns its pinned
 * buffers (6 bytes per stepped element).  Not capturable in a CUDA graph.
 * Errors: as for zero_shard_step_offload, per member. */
zero_status zero_group_step_offload(zero_group *g, const zero_group_member *args,
                                    double extra_norm_sq, int32_t n_threads, double gpu_share,
                                    void *stream, zero_step_result *res);

/* The group's loss-scale state (synchronizes `stream`) and its restore, as
 * zero_loss_scaler_state / zero_set_loss_scaler_state for a handle (the
 * dynamic loss scale of the ZeRO reading §5.1 and §5.3), and a learning rate
 * set on every member at once (as zero_flat_set_lr on each; zero_flat_set_lr
 * on one member changes that member's rate alone; the `lr` of §5.1's
 * optimizer settings). */
zero_status zero_group_loss_scaler_state(zero_group *g, zero_scaler_state *out, void *stream);
zero_status zero_group_set_loss_scaler_state(zero_group *g, const zero_scaler_state *in,
                                             void *stream);
zero_status zero_group_set_lr(zero_group *g, double lr);
zero_status zero_group_free(zero_group *g);

/* ZeRO-Offload shard step: the optimizer update runs on the host CPU cores
 * ("DeepSpeed 与 FSDP" §ZeRO-Offload: the reduced gradients move to the CPU,
 * the CPU updates the fp32 master weights with Adam, and the 16-bit weights
 * move back to the GPU; ZeRO reading §4.1: optimizer states in CPU memory).
 * On the GPU, exactly as in zero_shard_step: the reduce, unscale, overflow
 * check and norm partials into the handle's fp32 gradient rows, then the
 * loss-scale decision, the clip coefficient and the bias corrections.  The
 * call waits for that decision (one event).  If the step is applied, the
 * update of each stepped rank's state is split at element
 * split = gpu_share * shard_size (rounded down to 65536 elements, or the
 * whole shard for gpu_share = 1):
 *   - elements [0, split): the GPU's AdamW kernel, reading and writing the
 *     host-resident master/m/v over the host link (the host memory must be
 *     pinned, or the device must access pageable memory);
 *   - elements [split, shard_size): `n_threads` host threads (0: every CPU
 *     this process may run on), while the gradient rows come down from HBM in
 *     segments on a stream of the handle; the 16-bit parameters are staged in
 *     pinned memory and each finished segment is copied to
 *     flat_param_out[r * shard_size + ...] on a second stream of the handle.
 * Both halves run at once and do the same sequence of fp32 operations as
 * zero_shard_step, so the results are bit-identical to it for any split.
 * This is the offload mode of the method, never a substitute for the GPU
 * path: the reduce and the decision still need the GPU.
 * master, m, v: HOST fp32 arrays, shard_size elements per stepped rank,
 * 4-byte aligned; fully updated when the call returns.  flat_param_out:
 * device, as for zero_shard_step; when the call returns, `stream` is ordered
 * after every write to it.  grads and the rest: as zero_shard_step.
 * Not capturable in a CUDA graph (host synchronization and host compute).
 * Errors: as for zero_shard_step; INVALID_ARG for n_threads < 0, gpu_share
 * outside [0, 1], or gpu_share > 0 with host memory the GPU cannot access;
 * NO_MEMORY when the pinned buffers (6 bytes per stepped element) cannot be
 * had. */
zero_status zero_shard_step_offload(zero_flat *h, const int32_t *ranks, int32_t n_ranks,
                                    const void *grads, int64_t grad_ld,
                                    int64_t grad_rank_offset_mul, float *const *master,
                                    float *const *m, float *const *v, void *flat_param_out,
                                    double extra_norm_sq, int32_t n_threads, double gpu_share,
                                    void *stream, zero_step_result *res);

/* The host half of zero_shard_step_offload on its own, for a caller that
 * reduces gradients elsewhere: for i < n, with gc = g[i] * clip_coef,
 *     m = b1 m + (1-b1) gc;  v = b2 v + (1-b2) gc^2;
 *     mh = m / (1 - b1^t);  vh = v / (1 - b2^t);
 *     theta = theta (1 - lr wd) - (lr mh) / (sqrt(vh) + eps)
 * ("DeepSpeed 与 FSDP" §ZeRO-Offload, with the decoupled decay of AdamW),
 * each a single fp32 operation, the scalars rounded once to fp32 (1 - beta^t
 * from fp64 pow, t = step_t, the count of applied steps including this one),
 * then param_out[i] = the round-to-nearest-even 16-bit encoding of theta.
 * All pointers are HOST memory: g, master, m, v fp32 (4-byte aligned),
 * param_out 16-bit (2-byte aligned).  n_threads as above.  Needs no GPU.
 * Errors: INVALID_ARG (NULL pointer with n > 0, n < 0, step_t < 1,
 * n_threads < 0, bad hparams), UNSUPPORTED_DTYPE, ALIGNMENT. */
zero_status zero_offload_adamw_host(const zero_hparams *hp, int64_t step_t, float clip_coef,
                                    const float *g, float *master, float *m, float *v,
                                    void *param_out, int64_t n, zero_dtype param_dtype,
                                    int32_t n_threads);

/* Change the learning rate for the steps launched after this call (a
 * schedule's warm-up or decay; the ZeRO reading §5.3 warns that warm-up must
 * be re-tuned when the effective batch changes).  lr is fp64 as in
 * zero_hparams; lr and 1 - lr*weight_decay are rounded to fp32 once, as at
 * init.  Host only: steps already queued keep the rate they were launched
 * with.  Errors: INVALID_ARG (NULL handle, lr negative or not finite). */
zero_status zero_flat_set_lr(zero_flat *h, double lr);

/* Copy the loss-scale state to the host; synchronizes `stream`.  The state
 * is that of the dynamic loss scale of the ZeRO reading §5.1 (fp16
 * "loss_scale": 0 = dynamic, "initial_scale_power", "loss_scale_window",
 * "min_loss_scale") and §5.3 (an overflow skips the step and shrinks the
 * scale; clean steps grow it back): the scale the next step's gradients
 * carry, the clean-step counter, Adam's t (applied steps) and the number of
 * skipped steps.  out: host memory.  Errors: INVALID_ARG (NULL), CUDA. */
zero_status zero_loss_scaler_state(zero_flat *h, zero_scaler_state *out, void *stream);

/* Overwrite the loss-scale state (resume from a checkpoint): the state of
 * the dynamic loss scale of the ZeRO reading §5.1 and §5.3, as
 * zero_loss_scaler_state returns it.  Synchronizes `stream` before and after
 * the copy, so later steps on any stream see it; `in` is host memory.
 * scale > 0, good_steps >= 0, step_t >= 0, overflow_count >= 0, else
 * INVALID_ARG; CUDA if the copy cannot be queued. */
zero_status zero_set_loss_scaler_state(zero_flat *h, const zero_scaler_state *in, void *stream);

/* Model-state bytes per GPU for Psi parameters and N ranks in mixed
 * precision ("DeepSpeed 与 FSDP" §逐步推导 and §ZeRO-3 的数学总结):
 *   stage 0 (plain data parallel): 2Psi + 2Psi + 12Psi = 16Psi
 *   stage 1: 2Psi + 2Psi + 12Psi/N      stage 2: 2Psi + 2Psi/N + 12Psi/N
 *   stage 3: 2Psi/N + 2Psi/N + 12Psi/N
 * (fp16 params, fp16 grads, fp32 master+m+v).  Each part is rounded up to a
 * whole byte; *total is the exact sum rounded up once.  Any output may be
 * NULL.  Host only; needs no GPU.
 * Errors: INVALID_ARG (stage not 0..3, world_size < 1), OVERFLOW_SIZE. */
zero_status zero_memory_bytes(int32_t stage, uint64_t psi, int32_t world_size, uint64_t *total,
                              uint64_t *params, uint64_t *grads, uint64_t *optim);

/* Device bytes the handle holds now (state + scratch). */
zero_status zero_flat_device_bytes(const zero_flat *h, uint64_t *bytes);

/* Per-kernel timing, for measurement tools.  While enabled, every
 * zero_shard_step records CUDA events on its stream around its reduce,
 * finalize and AdamW launches (a few microseconds per step).  The step's
 * decision is normally made inside the reduce launch (by its last block), so
 * ms_finalize is then only the gap between two events.
 * zero_flat_profile_read waits for the recorded events, returns the summed
 * device milliseconds of each kernel class and the number of steps recorded,
 * and clears the record.  Any output may be NULL. */
zero_status zero_flat_profile_enable(zero_flat *h, int32_t enable);
zero_status zero_flat_profile_read(zero_flat *h, double *ms_reduce, double *ms_finalize,
                                   double *ms_adamw, int64_t *steps);

/* Which reduce kernel the handle's last contribution reduce (a step, a split
 * step's first half, or a micro-step accumulation) launched, for measurement
 * tools that name it: *staged = 1 for the bulk-copy (staged) reduce, 0 for
 * the plain one, -1 before the first.  Errors: INVALID_ARG (NULL). */
zero_status zero_flat_profile_reduce_form(const zero_flat *h, int32_t *staged);

/* Size of the device array that zero_shard_step_noalloc uses as scratch. */
#define ZERO_NOALLOC_SCRATCH_BYTES (32u << 20)

/* The shard step for callers that may not allocate device memory.
 * The pages have no counterpart of this entry point: it exists for callers
 * that run where allocating is forbidden or unsafe -- inside a framework
 * whose caching allocator owns all device memory, in runtimes that plan every
 * byte in advance, or in service loops where a cudaMalloc would synchronize
 * the device or fail at a bad moment.  Such callers cannot create a
 * zero_flat handle, because zero_flat_init allocates.
 * Same arithmetic and kernels as zero_shard_step; no handle.  Arguments as
 * for zero_flat_init / zero_shard_step, except:
 *   full_numel: elements of the FlatParameter (shard_size = ceil(full/N));
 *   state: the loss-scale state in HOST memory, read and updated by the call
 *     (start from scale = 2^initial_scale_power, or the static scale, and
 *     zeros); n_ranks <= 64.
 * It calls no cudaMalloc / cudaFree and allocates no host memory.  Its
 * scratch (fp32 reduced-gradient rows, norm partials, step scalars) is one
 * file-scope __device__ array of ZERO_NOALLOC_SCRATCH_BYTES that every GPU
 * which loads this library holds until the process exits; stepped shards
 * needing more than about 8.3M fp32 scratch elements in total
 * (n_ranks * roundup(shard_size, 4)) are rejected with ZERO_ERR_INVALID_ARG
 * and a message in zero_last_error().  Every call shares that array, which
 * keeps the last call's contents: each call begins by overwriting its state
 * block (the caller's loss-scale state, and zeros for the step's scalars and
 * the error word a timed-out bulk-copy wait sets), and its reduce writes
 * every gradient element and partial the later kernels read.  Calls whose
 * GPU work overlaps race on the array: order them.  The call is synchronous: it
 * waits for `stream` before returning the new state (and `res`, if not NULL).
 * The first call on a device looks up the array's address and the launch
 * geometry with that device current; make it before any stream capture. */
zero_status zero_shard_step_noalloc(int64_t full_numel, int32_t world_size, zero_dtype grad_dtype,
                                    zero_dtype param_dtype, zero_reduce_op op,
                                    const zero_hparams *hp, zero_scaler_state *state,
                                    const int32_t *ranks, int32_t n_ranks, const void *grads,
                                    int64_t grad_ld, int64_t grad_rank_offset_mul,
                                    float *const *master, float *const *m, float *const *v,
                                    void *flat_param_out, double extra_norm_sq, void *stream,
                                    zero_step_result *res);

/* Release the handle and its device memory (after the work queued with it
 * has finished; this call synchronizes the handle's device).  NULL is OK. */
zero_status zero_flat_free(zero_flat *h);

/* Static description of a status code. */
const char *zero_status_string(zero_status s);

/* Message of the last error raised on this thread ("" if none). */
const char *zero_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_H */
