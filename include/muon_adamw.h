/*
 * muon_adamw.h -- C ABI of a single-GPU hybrid Muon + AdamW optimizer step
 * for GB300 (sm_103a).
 *
 * The method is the MuonAdamW hybrid optimizer of the OpenDM VLA training
 * stack, as described in the article "VLA训练栈深度揭秘：OpenDM的Muon+AdamW优化器、
 * FSDP分布式训练与混合精度策略" (gsyq.cn/news/451971), section 核心揭秘一:
 *
 *   - routing (参数如何分流): 2-D parameters whose path holds action_expert
 *     and sits under layers, ending in .weight, and that are not embeddings,
 *     lm_head or norms, go to Muon; every other trainable parameter goes to
 *     AdamW; the optim switch "adamw" sends everything to AdamW;
 *   - Muon (Muon 的工作原理, 关键超参默认值): Nesterov momentum 0.95, then
 *     five Newton-Schulz iterations that approximate the orthogonal factor
 *     of the update on its short side, then the step
 *     lr * muon_lr_scale * 0.2 * sqrt(max(rows, cols));
 *   - the training-stack defaults table (训练栈默认参数速查表): gradient
 *     clipping at max_grad_norm 1.0 and the cosine_with_min_lr schedule with
 *     min_lr_rate 0.1.
 *
 * Conventions for every call:
 *   - Return value: MA_OK or an error status. No C++ exception crosses this
 *     boundary. On error a message is kept per thread and read with
 *     muon_adamw_last_error().
 *   - Device pointers are CUDA device addresses in the current device's
 *     primary context (e.g. torch tensors' data_ptr()). Host pointers are
 *     marked "host".
 *   - Tensors are dense and row-major (PyTorch [out, in] for matrices).
 *   - The caller owns parameters, gradients and bf16 shadows; they must stay
 *     allocated at the same address until muon_adamw_destroy(). The library
 *     owns its optimizer state and workspaces (allocated at the first step,
 *     freed by destroy) and never frees caller memory.
 *   - All device work is queued on the stream given to muon_adamw_create();
 *     calls return before the GPU finishes unless stated otherwise.
 *   - A handle is not thread-safe: serialise calls on one handle.
 */
#ifndef MUON_ADAMW_H
#define MUON_ADAMW_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MA_API __attribute__((visibility("default")))
#else
#define MA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct muon_adamw muon_adamw_t; /* opaque handle, owned by the library */

typedef enum {
  MA_OK = 0,
  MA_ERR_ARG = 1,          /* null pointer, bad enum, out-of-range value */
  MA_ERR_SHAPE = 2,        /* ndim/shape not usable for the assigned group */
  MA_ERR_DTYPE = 3,        /* gradient dtype not F32/BF16 */
  MA_ERR_ALIGN = 4,        /* pointer not aligned to its element size */
  MA_ERR_STATE = 5,        /* call not valid now (e.g. register after the first step) */
  MA_ERR_OOM = 6,          /* device allocation failed */
  MA_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed */
  MA_ERR_DEVICE_CHECK = 8, /* a kernel's own check failed (bounded wait ran out) */
  MA_ERR_UNSUPPORTED = 9   /* device is not sm_103 / feature not built */
} ma_status;

typedef enum { MA_MODE_MUON_ADAMW = 0, MA_MODE_ADAMW_ONLY = 1 } ma_mode;      /* optim switch */
typedef enum { MA_BF16_MIXED = 0, MA_FP32_MIXED = 1 } ma_precision;           /* precision_policy */
typedef enum { MA_GROUP_AUTO = 0, MA_GROUP_MUON = 1, MA_GROUP_ADAMW = 2, MA_GROUP_FROZEN = 3 } ma_group;
typedef enum { MA_DT_F32 = 0, MA_DT_BF16 = 1 } ma_dtype;
typedef enum { MA_NS_TCGEN05 = 0, MA_NS_SIMT = 1 } ma_ns_kernel;
/* Form of the Muon momentum. SGD (the step's reading of muon_nesterov):
 * buf <- mu buf + g, update g + mu buf. EMA (a variant): buf <- mu buf +
 * (1 - mu) g, update (1 - mu) g + mu buf. Without Nesterov the update is buf. */
typedef enum { MA_MOMENTUM_SGD = 0, MA_MOMENTUM_EMA = 1 } ma_momentum_form;

/* Longest per-iteration coefficient schedule (ns_schedule_len <= this). */
#define MA_NS_SCHEDULE_MAX 16
/* Distinct (lr_scale, weight_decay_scale) pairs over all parameters,
 * including the default (1, 1) (see muon_adamw_set_param_options). */
#define MA_MAX_OPTION_GROUPS 8

/* Optimizer configuration. Fill with muon_adamw_config_init(), then edit.
 * Defaults (article section in brackets):
 *   mode MA_MODE_MUON_ADAMW; precision MA_BF16_MIXED [核心揭秘三: bf16_mixed is
 *   the default policy; under it the library also writes a bf16 copy of each
 *   updated parameter when a shadow pointer is registered];
 *   muon_momentum 0.95, muon_nesterov 1, ns_steps 5, moonlight_coef 0.2
 *   [关键超参默认值]; muon_lr_scale 1.0 (named there without a value);
 *   ns_a/ns_b/ns_c 3.4445/-4.7750/2.0315 and ns_eps 1e-7 (the standard Muon
 *   quintic; not printed on the page); muon_weight_decay 0.1 (decoupled,
 *   base lr); adam_beta1 0.9, adam_beta2 0.999, adam_eps 1e-8,
 *   adam_weight_decay 0.1; max_grad_norm 1.0 [训练栈默认参数速查表]
 *   (<= 0 disables clipping); clip_eps 1e-6;
 *   ns_kernel MA_NS_TCGEN05: tensor-core kernels, one launch per product for
 *   most shape buckets and one launch per bucket of small matrices (canonical
 *   128 rows or fewer, at most 512 columns) for the whole chain and update
 *   (MA_NS_SIMT selects a slow CUDA-core GEMM used to cross-check them).
 *   With either setting, matrices whose short side is below 64 run
 *   Newton-Schulz in fp32 on the CUDA cores: with bf16 storage, updates of
 *   such matrices whose singular values are all alike (noise-like gradients)
 *   would come out up to 2.7e-2 (relative Frobenius) from the exact
 *   iteration, above the 2e-2 that bf16 Newton-Schulz keeps elsewhere. */
typedef struct {
  int32_t mode;
  int32_t precision;
  int32_t muon_nesterov;
  int32_t ns_steps;
  int32_t ns_kernel;
  /* reserved[0]: cross-check switches for tests, 0 in normal use; each
   * selects another correct path, which the tests check against the oracle
   * (bit 1) or bit for bit against the default (bit 2). Bit 1 runs every
   * Newton-Schulz product without CTA clusters; bit 2 writes the last
   * iteration's parameters from registers instead of through TMA; bit 8 runs
   * small matrices (canonical 128 rows or fewer, at most 512 columns) through
   * the per-product launches instead of the fused one. Other bits and
   * reserved[1..3] must be 0 (MA_ERR_ARG). */
  int32_t reserved[4];
  int32_t muon_momentum_form;          /* ma_momentum_form; default MA_MOMENTUM_SGD */
  /* 1: AdamW parameters whose lower-cased name ends with "bias" or contains
   * "norm" take no weight decay (the HF Trainer convention), unless
   * muon_adamw_set_param_options sets them. Default 0: one weight_decay for
   * all, as the article's defaults table lists it. */
  int32_t adam_decay_exempt_bias_norm;
  /* 0: every Newton-Schulz iteration uses (ns_a, ns_b, ns_c). Otherwise it
   * must equal ns_steps (<= MA_NS_SCHEDULE_MAX) and iteration i uses
   * ns_schedule[i] = {a, b, c}. */
  int32_t ns_schedule_len;
  /* Real-valued settings are doubles (like Python floats); the kernels get
   * fp32 values derived from them on the host, e.g. 1 - adam_beta2 is formed
   * in double before rounding, so 0.999 yields exactly fp32(0.001). */
  double muon_momentum;
  double ns_a, ns_b, ns_c;
  double ns_eps;
  double moonlight_coef;
  double muon_lr_scale;
  double muon_weight_decay;
  double adam_beta1, adam_beta2, adam_eps, adam_weight_decay;
  double max_grad_norm;
  double clip_eps;
  double ns_schedule[MA_NS_SCHEDULE_MAX][3];
} muon_adamw_config;

/* Per-kernel timing collected while profiling is on (see muon_adamw_set_profiling).
 * Index = ma_kernel_kind. ms = summed CUDA-event time of that kernel's launches
 * (events recorded on the stream the kernel runs on); units = algorithmic
 * work of those launches: bytes for HBM-bound kernels, flops for the NS GEMMs
 * (symmetric count: A = XX^T and A*A count the lower triangle only). */
typedef enum {
  MA_K_GRAD_NORM = 0,   /* sum of squares of all gradients */
  MA_K_CLIP = 1,        /* norm finalise + clip coefficient */
  MA_K_MOMENTUM = 2,    /* Muon Nesterov momentum + canonical bf16 pack */
  MA_K_NS_PREP = 3,     /* per-matrix Frobenius scale */
  MA_K_NS_GRAM = 4,     /* A = X X^T (iteration 1 scaled by 1/||G||^2) */
  MA_K_NS_POLY = 5,     /* B = b A + c A A */
  MA_K_NS_UPDATE = 6,   /* X <- B X, iterations 1 .. ns_steps-1 */
  MA_K_ADAMW = 7,       /* fused multi-tensor AdamW */
  MA_K_NS_APPLY = 8,    /* last iteration: B X applied to the parameters (Muon step) */
  MA_K_NS_FUSED = 9,    /* small matrices (s <= 128, l <= 512): every iteration and the step in one launch */
  MA_K_NS_NARROW = 10,  /* narrow matrices (s < 64): fp32 Newton-Schulz and the step on the CUDA cores */
  MA_K_COUNT = 11
} ma_kernel_kind;

typedef struct {
  int64_t launches[MA_K_COUNT];
  double ms[MA_K_COUNT];
  double units[MA_K_COUNT];
  int64_t steps;
} ma_profile;

/* Sizes of the frozen step plan (valid after the first step). */
typedef struct {
  int32_t n_params, n_muon, n_adamw, n_frozen;
  int32_t n_buckets;          /* groups of Muon matrices of equal padded canonical shape */
  int64_t muon_elems, adamw_elems, grad_elems;
  int64_t state_bytes, workspace_bytes;
  double ns_flops_per_step;   /* symmetric algorithmic count */
  double ns_dense_flops_per_step;
  double stream_bytes_per_step; /* algorithmic HBM bytes of the streaming kernels */
} ma_plan_info;

/* Fill *cfg with the defaults listed above. cfg must not be NULL. */
MA_API void muon_adamw_config_init(muon_adamw_config* cfg);

/* Routing predicate of 参数如何分流, as a pure host function: returns 1 when a
 * parameter called `name` (UTF-8, NUL-terminated) with `ndim` dimensions goes
 * to Muon, 0 otherwise (also for name == NULL). The match is: ndim == 2;
 * `name` contains "action_expert"; one dot-separated component equals
 * "layers"; `name` ends with ".weight"; the lower-cased name contains none of
 * "embed", "lm_head", "norm". */
MA_API int muon_adamw_is_muon_param(const char* name, int ndim);

/* Multiplier of the base lr for the cosine_with_min_lr schedule
 * (训练栈默认参数速查表): linear warmup over `warmup` steps, then
 * min_lr_rate + (1 - min_lr_rate) * 0.5 * (1 + cos(pi * progress)),
 * progress = (step - warmup) / (total - warmup). Pure host function. */
MA_API double muon_adamw_cosine_with_min_lr(int64_t step, int64_t total, int64_t warmup, double min_lr_rate);

/* Create an optimizer. cfg: host, copied. cuda_stream: a cudaStream_t (NULL =
 * legacy default stream) on the current device; all work of this handle is
 * ordered on it (a second, library-owned stream runs AdamW concurrently and
 * is joined back before each step returns). *out receives the handle.
 * Errors: MA_ERR_ARG (NULL out/cfg, invalid config values), MA_ERR_UNSUPPORTED
 * (current device is not compute capability 10.3), MA_ERR_CUDA. */
MA_API ma_status muon_adamw_create(const muon_adamw_config* cfg, void* cuda_stream, muon_adamw_t** out);

/* Register one parameter, before the first step.
 *   name        host UTF-8 string (copied), used for routing;
 *   ndim, shape host array of ndim int64 sizes (ndim 0..8, sizes >= 0);
 *   param_fp32  device fp32 master weights, numel elements (updated in place;
 *               may be NULL only for MA_GROUP_FROZEN or numel == 0);
 *   grad        device gradient, numel elements of grad_dtype (MA_DT_BF16 or
 *               MA_DT_F32); read each step, never written; NULL only when
 *               frozen or numel == 0;
 *   param_bf16_shadow  device bf16 copy written after each update when the
 *               precision is MA_BF16_MIXED, or NULL for none;
 *   group_override  MA_GROUP_AUTO applies the routing predicate (and the
 *               mode); MUON/ADAMW/FROZEN force the group (MUON needs ndim 2);
 *   assigned    host out (may be NULL): the group used;
 *   index_out   host out (may be NULL): registration index (0, 1, ...).
 * Errors: MA_ERR_ARG, MA_ERR_SHAPE, MA_ERR_DTYPE, MA_ERR_ALIGN (pointer not
 * aligned to its element size), MA_ERR_STATE (after the first step). */
MA_API ma_status muon_adamw_register_param(muon_adamw_t* h, const char* name, int ndim, const int64_t* shape,
                                    float* param_fp32, const void* grad, int grad_dtype,
                                    void* param_bf16_shadow, int group_override, int* assigned,
                                    int* index_out);

/* Per-parameter multipliers, like a PyTorch parameter group: parameter
 * `index` (registration order) steps with lr * lr_scale, and its decoupled
 * weight decay is weight_decay * weight_decay_scale with that lr. For AdamW:
 * p <- p (1 - lr ls wd ws) - (lr ls / bc1) m / (sqrt(v / bc2) + eps); for a
 * Muon matrix: p <- p (1 - lr ls muon_wd ws) - lr ls muon_lr_scale 0.2
 * sqrt(max(m, n)) O. Default (1, 1); an explicit call overrides
 * adam_decay_exempt_bias_norm for that parameter. Call before the first step.
 * Errors: MA_ERR_ARG (NULL handle, index out of range, a scale negative or
 * not finite), MA_ERR_STATE (after the first step, or a frozen parameter),
 * MA_ERR_UNSUPPORTED (more than MA_MAX_OPTION_GROUPS distinct pairs; the
 * exemption rule's pairs count too and are checked at the first step). */
MA_API ma_status muon_adamw_set_param_options(muon_adamw_t* h, int index, double lr_scale,
                                              double weight_decay_scale);

/* One optimizer step with base learning rate `lr` (the caller applies its
 * schedule, stepped once per optimizer step). The first call freezes the
 * plan and allocates state and workspaces. Queues on the handle's stream:
 * global grad norm and clip coefficient; Muon momentum, Newton-Schulz and
 * update; AdamW. grad_norm_out: host out (NULL = fully asynchronous); when
 * given, the call synchronises the stream and stores the pre-clip global
 * gradient norm, and also reports a failed in-kernel check as
 * MA_ERR_DEVICE_CHECK. Non-finite gradients are not skipped: they propagate
 * into the parameters and the norm. Errors: MA_ERR_ARG (lr not finite),
 * MA_ERR_OOM, MA_ERR_CUDA, MA_ERR_DEVICE_CHECK. */
MA_API ma_status muon_adamw_step(muon_adamw_t* h, double lr, float* grad_norm_out);

/* Wait for the handle's stream and read the kernels' error flag.
 * MA_ERR_DEVICE_CHECK if a bounded in-kernel wait ran out. */
MA_API ma_status muon_adamw_sync(muon_adamw_t* h);

/* Run each step's Newton-Schulz chain (the Frobenius scales and the 3 x
 * ns_steps products, most of a step's launches) as a captured CUDA graph
 * (enable = 1, the default) or as direct launches (0). The graph is captured
 * at the first step that can use it and replayed from then on: the plan never
 * changes after the first step and the lr- and step-dependent scalars are read
 * from HBM (one small host-to-device copy per step). The gradient passes (norm,
 * clip, momentum, AdamW) stay direct launches, so the events of
 * muon_adamw_record_grads_consumed keep their meaning. Direct launches are
 * used while profiling is on, with MA_NS_SIMT, and if a capture ever fails.
 * Results are bitwise the same either way. Errors: MA_ERR_ARG (NULL handle). */
MA_API ma_status muon_adamw_set_graph_mode(muon_adamw_t* h, int enable);

/* Record `cuda_event` (a cudaEvent_t created by the caller) so that it
 * completes once the latest step no longer reads any gradient: after the
 * gradient norm, the Muon momentum pass and the AdamW pass (the Newton-Schulz
 * chain that follows reads none). From then on the caller may overwrite the
 * gradient buffers, e.g. with the next step's gradients, while the step's
 * Newton-Schulz products still run. The event is recorded on a library
 * stream that only waits for those passes, so neither of the step's streams
 * is held back. The article has no counterpart (its optimizer owns no
 * gradient buffers). Errors: MA_ERR_ARG (NULL handle or event), MA_ERR_STATE
 * (no step taken yet), MA_ERR_CUDA. */
MA_API ma_status muon_adamw_record_grads_consumed(muon_adamw_t* h, void* cuda_event);

/* The work order of one tensor-core Newton-Schulz launch (host only; needs no
 * device): `nprob` (1..4) problems in launch order, problem q holding
 * `units[q]` work units of reduction depth `k[q]` (a positive multiple of 64);
 * units are numbered consecutively across the problems. Each unit goes, in
 * that order, to the cluster with the least work so far (a unit costs k / 64
 * plus 6), ties to the lowest cluster; the result is laid out round by round:
 * cluster c runs order[c], order[c + nclusters], ..., and -1 marks a position
 * with no unit. `*npos` receives the table length (a multiple of nclusters).
 * The library builds the same table for every launch at planning time.
 * Errors: MA_ERR_ARG (NULL pointer, nprob outside 1..4, nclusters < 1, a
 * negative unit count or a bad k), MA_ERR_SHAPE (`cap` entries are too few;
 * `*npos` is still set). */
MA_API ma_status muon_adamw_plan_work_order(int nprob, const int64_t* k, const int64_t* units, int nclusters,
                                            int32_t* order, int64_t cap, int64_t* npos);

/* Test hook for the failure path, not for production use. Arms a one-shot
 * stall: in the next step's first Newton-Schulz launch, one CTA issues no
 * operand loads, so its bounded wait (2 s) runs out. The kernel
 * then records the error, drains and releases its resources and returns;
 * that step's result is invalid and the step reports MA_ERR_DEVICE_CHECK
 * when its norm is read (or on muon_adamw_sync). Nothing faults, and the
 * handle and context stay usable for later steps. Errors: MA_ERR_ARG,
 * MA_ERR_UNSUPPORTED (MA_NS_SIMT has no waits). */
MA_API ma_status muon_adamw_test_arm_stall(muon_adamw_t* h);

/* Copy optimizer state of parameter `index` to host memory `dst_host`
 * (numel fp32 values). which = 0: Muon momentum buffer or AdamW first
 * moment; which = 1: AdamW second moment. Synchronises the stream.
 * Errors: MA_ERR_ARG (bad index/which, NULL dst), MA_ERR_STATE (before the
 * first step, or a frozen parameter). */
MA_API ma_status muon_adamw_get_state(muon_adamw_t* h, int index, int which, float* dst_host);

/* Replace the same state from host memory `src_host` (numel fp32 values),
 * for resuming from a checkpoint; also valid before the first step (the
 * plan is then frozen by this call). Synchronises the stream. */
MA_API ma_status muon_adamw_set_state(muon_adamw_t* h, int index, int which, const float* src_host);

/* Step counter t used for bias correction (number of completed steps), and
 * setter for resuming (t >= 0). */
MA_API ma_status muon_adamw_get_step(muon_adamw_t* h, int64_t* t_out);
MA_API ma_status muon_adamw_set_step(muon_adamw_t* h, int64_t t);

/* Last step's global gradient norm and clip coefficient (synchronises). */
MA_API ma_status muon_adamw_last_norm(muon_adamw_t* h, float* total_out, float* coef_out);

/* Plan sizes (after the first step; MA_ERR_STATE before). */
MA_API ma_status muon_adamw_plan_info(muon_adamw_t* h, ma_plan_info* out);

/* Per-kernel CUDA-event timing. enable = 1 records an event pair around every
 * kernel launch of subsequent steps (on the launching stream); 0 stops.
 * get_profile synchronises, folds the recorded events into *out (host) and
 * keeps accumulating; reset clears the totals. */
MA_API ma_status muon_adamw_set_profiling(muon_adamw_t* h, int enable);
MA_API ma_status muon_adamw_get_profile(muon_adamw_t* h, ma_profile* out);
MA_API ma_status muon_adamw_reset_profile(muon_adamw_t* h);

/* Free the library's state and workspaces (after waiting for the stream)
 * and the handle. Caller memory is not touched. h == NULL is MA_ERR_ARG. */
MA_API ma_status muon_adamw_destroy(muon_adamw_t* h);

/* ---- Sharded step: several ranks, one GPU each ----
 * The article runs this optimizer under FSDP on 8 GPUs (核心揭秘一 / 为 FSDP
 * 分片量身定制的细节: MuonShardPlan all-gathers each matrix's shards so that
 * Newton-Schulz sees the whole matrix). Here the step itself is divided over
 * `world` ranks that all hold every parameter and gradient (data parallel,
 * gradients already reduced):
 *   - each Muon matrix is updated whole by one owner rank, chosen
 *     longest-processing-time-first on its dense Newton-Schulz flops
 *     5 (4 s^2 l + 2 s^3), s/l its short/long side;
 *   - AdamW parameters, concatenated in registration order, are split into
 *     `world` contiguous ranges of nearly equal length, each cut moved down
 *     to a multiple of 64 elements of the parameter it falls in;
 *   - every rank computes the sum of squares of the gradients it owns; the
 *     caller all-reduces (sums) these numbers, and every rank clips with the
 *     global norm sqrt(sum) exactly as the single-GPU step does;
 *   - after the step each rank has updated only what it owns: the caller
 *     shares the results (a broadcast of each Muon matrix from its owner, an
 *     all-gather of the AdamW ranges, and the same for bf16 shadows).
 * The library issues no collective and never reads another rank's memory.
 * A rank allocates the state of what it owns only (AdamW m and v for its
 * range). The partition depends only on the registrations and `world`, so
 * every rank computes the same one. */
#define MA_SHARD_MAX_WORLD 4096

/* The partition above as a pure host function (needs no device): n_params
 * parameters with groups[i] (MA_GROUP_MUON / ADAMW / FROZEN), numels[i] and,
 * for Muon matrices, rows[i] x cols[i]. owner_out[i] (n_params entries):
 * the rank that updates Muon matrix i, -1 for the others. begin_out/end_out
 * (n_params * world entries, [i * world + r]): the elements [begin, end) of
 * parameter i that rank r updates (the whole matrix at its owner, a range for
 * AdamW, empty otherwise). Errors: MA_ERR_ARG (NULL pointer, bad group,
 * world outside 1..MA_SHARD_MAX_WORLD), MA_ERR_SHAPE (negative size, a Muon
 * matrix whose rows x cols is not numel). */
MA_API ma_status muon_adamw_plan_shards(int n_params, const int32_t* groups, const int64_t* numels,
                                        const int64_t* rows, const int64_t* cols, int world, int32_t* owner_out,
                                        int64_t* begin_out, int64_t* end_out);

/* Make handle h rank `rank` of `world` (0 <= rank < world), before the first
 * step; world 1 (the default) is the single-GPU step. Errors: MA_ERR_ARG,
 * MA_ERR_STATE (after the first step). */
MA_API ma_status muon_adamw_set_shard(muon_adamw_t* h, int rank, int world);

/* The elements [*begin, *end) of parameter `index` that rank `rank` updates
 * under h's partition (the whole trainable parameter for world 1). Computed
 * from the registrations so far, which are final from the first step on.
 * get_state/set_state of a sharded handle move exactly this rank's range
 * (end - begin values); for a parameter this rank does not update they return
 * MA_ERR_STATE. Errors: MA_ERR_ARG. */
MA_API ma_status muon_adamw_shard_range(muon_adamw_t* h, int index, int rank, int64_t* begin, int64_t* end);

/* First half of a step (any handle; the only way a handle of world > 1
 * steps, muon_adamw_step returns MA_ERR_STATE there): like muon_adamw_step
 * up to the gradient norm, it freezes the plan at the first call, advances
 * the step counter and queues on the handle's stream the sum of squares of
 * the gradients this rank owns, written as one fp64 value to local_sumsq
 * (device pointer, 8-byte aligned). Asynchronous. Errors: MA_ERR_ARG,
 * MA_ERR_ALIGN, MA_ERR_STATE (step_begin twice without step_end), MA_ERR_OOM,
 * MA_ERR_CUDA. */
MA_API ma_status muon_adamw_step_begin(muon_adamw_t* h, double lr, double* local_sumsq);

/* Second half: global_sumsq (device pointer, 8-byte aligned) holds the sum of
 * every rank's local_sumsq, written on or before the handle's stream reaches
 * this point (e.g. an all-reduce queued on that stream); the norm is its
 * square root, the clip coefficient min(1, max_grad_norm / (norm + clip_eps))
 * as in muon_adamw_step, then this rank's Muon matrices and AdamW ranges are
 * updated. grad_norm_out as in muon_adamw_step. Errors: MA_ERR_ARG,
 * MA_ERR_ALIGN, MA_ERR_STATE (no step_begin), MA_ERR_CUDA,
 * MA_ERR_DEVICE_CHECK. */
MA_API ma_status muon_adamw_step_end(muon_adamw_t* h, const double* global_sumsq, float* grad_norm_out);

/* ---- Allocation-free gradient norm ----
 * The article has no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc, such as a host that gives all device memory
 * to its own pool allocator at start-up and forbids later allocations, or a
 * latency-critical loop that cannot accept cudaMalloc's implicit device-wide
 * synchronisation. It computes the same global gradient norm and clip
 * coefficient as muon_adamw_step(), without a handle and without allocating:
 * its scratch is a fixed file-scope device array of MA_NOALLOC_MAX_PARTIALS
 * floats (4 KiB) that every GPU loading this library keeps until the process
 * exits, and the tensor list travels in the kernel's parameters.
 *
 *   grads, numels, dtypes  host arrays of n_tensors entries: device pointer,
 *                          element count, MA_DT_F32 or MA_DT_BF16;
 *   n_tensors              0 .. MA_NOALLOC_MAX_TENSORS; more is MA_ERR_ARG;
 *   max_norm, clip_eps     clip = min(1, max_norm / (norm + clip_eps));
 *                          max_norm <= 0 gives 1; a NaN norm gives NaN;
 *   out_total_coef         device pointer to 2 floats: [0] norm, [1] clip;
 *   cuda_stream            cudaStream_t on the current device (NULL = default).
 * Work is queued on the stream; the call does not wait for it. The first call
 * on a device also looks up the scratch array's device address for that
 * device (cudaGetSymbolAddress), so make that first call before any stream
 * capture. All calls share the one scratch array, which keeps the last call's
 * partial sums; each call rewrites every slot it reads, so nothing needs
 * clearing, but calls whose work overlaps on the GPU (different streams, or
 * host threads racing on one device) corrupt each other's partial sums:
 * order them on one stream. Errors: MA_ERR_ARG, MA_ERR_SHAPE, MA_ERR_DTYPE,
 * MA_ERR_ALIGN, MA_ERR_CUDA; no allocation is attempted on any path. */
#define MA_NOALLOC_MAX_TENSORS 64
#define MA_NOALLOC_MAX_PARTIALS 1024
MA_API ma_status muon_adamw_grad_norm_noalloc(const void* const* grads, const int64_t* numels,
                                              const int32_t* dtypes, int n_tensors, double max_norm,
                                              double clip_eps, float* out_total_coef, void* cuda_stream);

/* Message of the last error on this thread ("" if none). Never NULL. */
MA_API const char* muon_adamw_last_error(void);

/* Library version string, e.g. "0.1.0 sm_103a". */
MA_API const char* muon_adamw_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MUON_ADAMW_H */
