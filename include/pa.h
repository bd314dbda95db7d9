/*
 * pa.h - C ABI of the GB300 PagedAttention step library.
 *
 * One step of a continuous-batching engine's attention layer on one GPU:
 *   1. (optional) rotary embedding of the new Q and K rows,
 *   2. reshape_and_cache: the new K/V rows are written into the shared
 *      paged pool through block_table (in place),
 *   3. causal grouped-query attention of every packed query token over its
 *      sequence's cached context, with optional local window and softcap.
 *
 * The operation is the one specified by "PagedAttention - CUDA Design
 * Document" (onnxruntime 1.29.0 docs, contrib_ops/cuda/paged_attention):
 * section 4 (op contract, input/attribute meaning, in-place cache aliasing),
 * section 4.7 (no host read of device lengths; host values only size
 * launches), section 5.1 (derived write slot), section 8 implementation
 * note P5 (causal bound past + j + 1, window [kv_len - W, kv_len), softcap
 * softcap * tanh(x * scale / softcap), split-KV with log-sum-exp merge),
 * section 9 (-1 block entries are unmapped and masked) and section 15
 * (validation rules); and by "Design: WebGPU PagedAttention" section 3.3
 * (packed tokens delimited by cumulative_sequence_lengths).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers on the handle's device unless
 *     stated otherwise; all tensors are dense row-major.  fp16 tensors are
 *     passed as void* holding IEEE binary16.  int32 tensors as int32_t*.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *   - The caller owns every tensor.  key_cache and value_cache are updated
 *     in place (the op's cache outputs alias its cache inputs).  The library
 *     owns only the workspace allocated by pa_create.
 *   - pa_cache_write and pa_forward never allocate, never synchronise and
 *     never copy device data to the host, so they may be captured into a CUDA
 *     graph (device addresses must then stay fixed across replays).
 *   - Host-checkable errors return PA_INVALID_ARGUMENT / PA_NOT_SUPPORTED
 *     before anything is launched; pa_last_error_message() names the
 *     offending argument.  Device-resident values (lengths, block ids) are
 *     not read by the host: invalid ones are skipped by the kernels without
 *     any out-of-bounds access and recorded in a device error word that
 *     pa_check_device_error() returns.
 *
 * Shapes (T = token_count, B = batch, H = num_heads, Hk = kv_num_heads,
 * D = head_size, bs = block_size, NB = num_blocks, MB = max_blocks_per_seq):
 *   query        [T, H*D]          fp16
 *   key, value   [T, Hk*D]         fp16 (new tokens, not yet rotated)
 *   key_cache    [NB, bs, Hk, D]   fp16, value_cache likewise
 *   block_table  [B, MB]           int32; entry i of row b = block holding
 *                                  positions [i*bs, (i+1)*bs) of sequence b,
 *                                  -1 = not mapped (masked; no write)
 *   cumulative_sequence_lengths [B+1] int32, cum[0] = 0, cum[B] = T
 *   past_sequence_lengths       [B]   int32, cached tokens per sequence
 *   cos_cache, sin_cache [P, rotary_dim/2] fp16 (P = max_rotary_positions)
 *   output       [T, H*D]          fp16
 * Token j of sequence b is packed row cum[b] + j and has position
 * past[b] + j.  Query head h uses kv head h / (H / Hk).
 *
 * Quantized cache (section 8): with cache_dtype PA_CACHE_INT8 or
 * PA_CACHE_FP8_E4M3 the pools hold one signed 8-bit code per element,
 * [NB, bs, Hk, D] bytes, with zero point 0: element value = code * scale.
 * k_scale / v_scale are fp32, [1] (PA_QUANT_PER_TENSOR) or [Hk, D]
 * (PA_QUANT_PER_CHANNEL: kv head k's channel c uses scale[k*D + c]).
 * head_sink (section 6) is an optional fp16 [H]: one extra logit per query
 * head that enters the softmax denominator only.  Both arrive through
 * pa_extra_inputs (pa_cache_write_ex / pa_forward_ex).
 *
 * Packed QKV (section 4): with packed_qkv the query argument holds rows
 * [T, (H + 2*Hk)*D] = [Q heads | K heads | V heads] and key / value are NULL.
 * QK-Norm (section 7): with qk_norm every head of Q and K is replaced, before
 * rotary and before K is cached, by
 *   y[c] = fp16((x[c] * r) * w[c]),  r = 1 / sqrt(sum_j x[j]^2 / D + eps),
 * w = q_norm_weight / k_norm_weight ([D] fp16, shared by all heads); the
 * fp32 sum of squares is one running sum over the channels in ascending
 * order (one rounding per square and per add), then IEEE square root and
 * reciprocal, so the cached K is bit-reproducible.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_handle_s* pa_handle;

typedef enum {
  PA_OK = 0,
  PA_INVALID_ARGUMENT = 1,   /* a host-checkable rule was violated */
  PA_NOT_SUPPORTED = 2,      /* valid op, but not built here (e.g. head_size 80) */
  PA_CUDA_ERROR = 3,         /* a CUDA runtime/driver call failed */
  PA_DEVICE_DATA_ERROR = 4   /* pa_check_device_error found a flagged value */
} pa_status;

/* Bits of the device error word (pa_check_device_error). */
enum {
  PA_DEVERR_CUM = 1,          /* cum[0] != 0, cum not monotone or cum[B] != T */
  PA_DEVERR_BLOCK_ID = 2,     /* block id outside [-1, NB) (access skipped) */
  PA_DEVERR_PAST = 4,         /* past < 0 (sequence skipped) */
  PA_DEVERR_KV_BOUND = 8,     /* past + q_len > kv bound or > MB*bs (sequence skipped) */
  PA_DEVERR_Q_BOUND = 16,     /* q_len > max_query_len_bound (sequence skipped) */
  PA_DEVERR_ROTARY_POS = 32,  /* position >= max_rotary_positions (row left unrotated) */
  PA_DEVERR_TIMEOUT = 64,     /* an internal wait exceeded its limit (kernel gave up; see pa_last_wait_site) */
  PA_DEVERR_SLOT = 128        /* slot_mapping entry outside [-1, NB*bs) (row not written) */
};

/* Cache element types (section 8.2, T_CACHE).  8-bit codes are signed and
 * zero-symmetric; writing a value x stores code = Q(x / scale) with the
 * division in fp32 and Q = round to nearest-even saturated to [-128, 127]
 * (int8) or to +-448 (e4m3fn).
 * PA_CACHE_BF16 selects bfloat16 activations with a bfloat16 cache (section
 * 8.2 registers the kernel for fp16 and bfloat16 activations): query, key,
 * value, both pools, cos_cache / sin_cache, head_sink and the output are
 * then bfloat16 wherever this header says fp16.  Rotary rounds each rotated
 * value to bfloat16 (nearest-even) after the same fp32 arithmetic; the
 * attention contractions take bfloat16 operands (the softmax weights P are
 * rounded to bfloat16 for the P*V contraction) with fp32 accumulation;
 * QK-Norm weights are bfloat16 and its outputs rounded to bfloat16.  The
 * latent layout and pa_forward_no_alloc are fp16 only (PA_NOT_SUPPORTED). */
enum { PA_CACHE_FP16 = 0, PA_CACHE_INT8 = 1, PA_CACHE_FP8_E4M3 = 2, PA_CACHE_BF16 = 3 };

/* Activation types (section 8.2 registers fp16 and bfloat16 activations
 * with every cache type).  PA_ACT_DEFAULT: fp16, or bfloat16 with
 * PA_CACHE_BF16.  PA_ACT_BF16 with an 8-bit cache: query, key, value,
 * cos_cache / sin_cache, head_sink, the QK-Norm weights and the output are
 * bfloat16, transformed (QK-Norm, rotary) with the bfloat16 roundings above;
 * the codes are those of the bfloat16 values (division in fp32).  The
 * attention contractions run on fp16 operands as for fp16 activations (the
 * query is copied as fp16, exact for bfloat16 values in fp16's normal range;
 * |q| beyond 65504 overflows there).  With PA_CACHE_FP16 it is
 * PA_INVALID_ARGUMENT; pa_forward_no_alloc takes PA_ACT_DEFAULT only. */
enum { PA_ACT_DEFAULT = 0, PA_ACT_BF16 = 1 };
/* Cache layout (section 12).  LATENT: one cache key_cache [NB, bs, 1, D] of
 * latent rows (value and value_cache NULL, kv_num_heads 1); every query
 * head attends with its D channels and the output is the weighted sum of
 * the first v_head_size channels of the same rows (absorbed multi-head
 * latent attention); an explicit scale is required.  Built: D = 576,
 * v_head_size = 512, num_heads <= 16 or a multiple of 16, fp16 cache;
 * output [T, H*512].  A sequence with several new tokens (chunked prefill,
 * prefix caching) runs in the same absorbed form, each token attending
 * causally like a one-token decode row (section 12.8). */
enum { PA_LAYOUT_SEPARATE = 0, PA_LAYOUT_LATENT = 1 };
/* Scale granularity (section 8.2, k_quant_type / v_quant_type). */
enum { PA_QUANT_NONE = 0, PA_QUANT_PER_TENSOR = 1, PA_QUANT_PER_CHANNEL = 2 };

/* Static description of a layer, fixed for the handle's lifetime
 * (section 4.5 attributes plus the capacities that size launches, 4.7). */
typedef struct {
  int num_heads;          /* H, > 0, multiple of kv_num_heads */
  int kv_num_heads;       /* Hk, > 0 */
  int head_size;          /* D, multiple of 8; the library runs 64, 128, 256 (576 with the latent layout) */
  int block_size;         /* bs, power of two >= 16 */
  int num_blocks;         /* NB, > 0 */
  int max_blocks_per_seq; /* MB, > 0 (block_table row length) */
  float scale;            /* 0 => 1/sqrt(D) */
  float softcap;          /* 0 => off; > 0 => softcap*tanh(x/softcap) */
  int local_window_size;  /* -1 => off; W >= 1 admits W positions incl. self */
  int do_rotary;          /* 0/1: rotate Q and K before the write */
  int rotary_interleaved; /* 0: pairs (i, i+R/2); 1: pairs (2i, 2i+1) */
  int rotary_dim;         /* R = 2*cos_cache.shape[1]; 0 => D when do_rotary */
  int max_rotary_positions; /* P = cos_cache.shape[0] (rows of the tables) */
  int max_batch;          /* capacity for B across every call on the handle */
  int max_tokens;         /* capacity for T across every call on the handle */
  int max_query_len_bound; /* 0 => max_tokens; upper bound on any q_len */
  int max_kv_len_bound;    /* 0 => MB*bs; upper bound on any past + q_len */
  int cache_dtype;         /* PA_CACHE_*: element type of key_cache / value_cache */
  int k_quant_type;        /* PA_QUANT_*: NONE for 16-bit caches, else PER_TENSOR / PER_CHANNEL */
  int v_quant_type;        /* must equal k_quant_type */
  int packed_qkv;          /* 1: pa_forward's query rows are [Q heads | K heads | V heads], key/value NULL */
  int qk_norm;             /* 1: QK-Norm of Q and K before rotary (q/k_norm_weight required) */
  float qk_norm_epsilon;   /* > 0 (default 1e-6) */
  int kv_cache_layout;     /* PA_LAYOUT_SEPARATE (key_cache + value_cache) or PA_LAYOUT_LATENT */
  int v_head_size;         /* 0 => head_size; != head_size only with PA_LAYOUT_LATENT */
  int rotary_offset;       /* first rotated channel of a head (multiple of 8; latent: v_head_size) */
  int act_dtype;           /* PA_ACT_*: activation type (PA_ACT_BF16 with an 8-bit cache) */
} pa_config;

/* Fills *cfg with the attribute defaults (scale 0, softcap 0, window -1,
 * no rotary, bounds 0, fp16 cache, no packed QKV, no QK-Norm, QK-Norm
 * epsilon 1e-6).  Geometry fields are set to 0 and must be filled. */
PA_API void pa_config_init(pa_config* cfg);

/* Host-only check of a configuration against the validation rules
 * (section 15): H % Hk == 0, D % 8 == 0, bs a power of two >= 16,
 * softcap >= 0, window == -1 or >= 1, rotary_dim even and <= D, positive
 * capacities, quantization NONE exactly for 16-bit caches.  Writes a message
 * naming the field into msg (may be NULL).  Returns PA_INVALID_ARGUMENT or
 * PA_NOT_SUPPORTED on failure.  Not built (PA_NOT_SUPPORTED): 8-bit caches
 * with head_size 64, with k_quant_type != v_quant_type, or with
 * num_heads / kv_num_heads above 16 (8-bit caches run every query row
 * through the decode kernel: a sequence whose q_len * num_heads /
 * kv_num_heads rows exceed one 16-row item runs in chunks of
 * 16 * kv_num_heads / num_heads tokens, section 8.5); a bfloat16 cache
 * with the latent layout.  Touches no GPU. */
PA_API pa_status pa_validate_config(const pa_config* cfg, char* msg, size_t msg_len);

/* Host-only check of one step's arguments (token_count <= max_tokens,
 * batch <= max_batch, required pointers non-NULL (query, key, value and
 * output may be NULL when token_count == 0), rotary tables present iff
 * do_rotary).  query/output may be NULL when checking pa_cache_write
 * (pass for_forward = 0).  Touches no GPU. */
PA_API pa_status pa_check_step(const pa_config* cfg, int for_forward, const void* query,
                        const void* key, const void* value, const void* key_cache,
                        const void* value_cache, const int32_t* block_table,
                        const int32_t* cumulative_sequence_lengths,
                        const int32_t* past_sequence_lengths, int batch,
                        int token_count, const void* cos_cache,
                        const void* sin_cache, const void* output, char* msg,
                        size_t msg_len);

/* Validates cfg, then allocates the device workspace on the current CUDA
 * device (work lists, split-KV partials, rotated-query buffer, error word)
 * sized from the capacities.  May synchronise; never call during capture.
 * On failure *out is NULL and pa_last_error_message(NULL) explains. */
PA_API pa_status pa_create(const pa_config* cfg, pa_handle* out);

/* Steps 1-2 only: rotary on K (if do_rotary) and the paged write of K and V
 * for every new token.  Slot = block_table[b][pos/bs]*bs + pos%bs; a -1
 * entry writes nothing.  Bit-exact: without rotary the rows are copied;
 * with rotary each pair is y1 = x1*c - x2*s, y2 = x2*c + x1*s in fp32 with
 * one rounding per operation, then rounded to fp16. */
PA_API pa_status pa_cache_write(pa_handle h, const void* key, const void* value,
                         void* key_cache, void* value_cache,
                         const int32_t* block_table,
                         const int32_t* cumulative_sequence_lengths,
                         const int32_t* past_sequence_lengths, int batch,
                         int token_count, const void* cos_cache,
                         const void* sin_cache, void* stream);

/* The whole step: rotary on Q and K (if do_rotary), the paged cache write,
 * then attention for every packed query row into output.  Row (t, h) of
 * sequence b attends to positions p in [lo, past_b + j + 1) with
 * lo = max(0, past_b + j + 1 - W) under a window, skipping positions whose
 * block entry is -1; x = scale * <q, k_p>, optionally softcapped; output is
 * the softmax-weighted sum of v_p (0 when no position is admitted).
 * token_count == 0 returns PA_OK and launches nothing. */
PA_API pa_status pa_forward(pa_handle h, const void* query, const void* key,
                     const void* value, void* key_cache, void* value_cache,
                     const int32_t* block_table,
                     const int32_t* cumulative_sequence_lengths,
                     const int32_t* past_sequence_lengths, int batch,
                     int token_count, const void* cos_cache,
                     const void* sin_cache, void* output, void* stream);

/* Optional inputs of the op contract (section 4, inputs 11, 14, 15).  Any
 * pointer may be NULL where its feature is off. */
typedef struct {
  const void* head_sink;  /* [H] fp16, device; NULL = no sink */
  const float* k_scale;   /* device fp32, [1] or [Hk*D]; required iff the cache is 8-bit */
  const float* v_scale;   /* likewise for value_cache */
  const int32_t* slot_mapping; /* [T] int32, device; NULL = derive the write slot from block_table */
  const void* q_norm_weight;   /* [D] fp16, device; required iff qk_norm (with k_norm_weight) */
  const void* k_norm_weight;   /* [D] fp16, device */
} pa_extra_inputs;

/* pa_cache_write with the optional inputs (extra may be NULL).  With an
 * 8-bit cache the written rows are quantized (after rotary) under
 * k_scale / v_scale as stated at PA_CACHE_INT8; bit-exact.
 * slot_mapping (section 5.2) is authoritative for the write: packed row t
 * goes to flat slot slot_mapping[t] of the pool viewed as [NB*bs, Hk, D];
 * -1 writes nothing (the row's query still attends); values outside
 * [-1, NB*bs) write nothing and set PA_DEVERR_SLOT.  block_table still
 * defines what every sequence reads (positions [i*bs, (i+1)*bs) of row b),
 * so a runtime can recycle blocks, e.g. a ring of ceil(W/bs)+1 blocks per
 * sequence under a local window W with -1 entries below the window
 * (section 9.3). */
PA_API pa_status pa_cache_write_ex(pa_handle h, const void* key, const void* value,
                                   void* key_cache, void* value_cache,
                                   const int32_t* block_table,
                                   const int32_t* cumulative_sequence_lengths,
                                   const int32_t* past_sequence_lengths, int batch,
                                   int token_count, const void* cos_cache,
                                   const void* sin_cache, const pa_extra_inputs* extra,
                                   void* stream);

/* pa_forward with the optional inputs (extra may be NULL).  8-bit caches
 * are read at their stored width: a per-tensor K scale multiplies the
 * softmax scale, per-channel K scales are folded into the query
 * (q * k_scale[c], rounded to fp16), and the V scale multiplies the output
 * (section 8.5 phase 3).  head_sink s_h adds exp(s_h - m) to the softmax
 * denominator of every row of head h, m = max(s_h, max logit) (section
 * 6.1); a row with no admitted key still outputs 0. */
PA_API pa_status pa_forward_ex(pa_handle h, const void* query, const void* key,
                               const void* value, void* key_cache, void* value_cache,
                               const int32_t* block_table,
                               const int32_t* cumulative_sequence_lengths,
                               const int32_t* past_sequence_lengths, int batch,
                               int token_count, const void* cos_cache,
                               const void* sin_cache, const pa_extra_inputs* extra,
                               void* output, void* stream);

/* Synchronises the stream of the handle's last call, reads and clears the
 * device error word into *code (0 = clean).  Returns PA_DEVICE_DATA_ERROR
 * when *code != 0.  Not capturable.  With PA_DEVERR_TIMEOUT set, the message
 * (pa_last_error_message) and pa_last_wait_site name the wait that gave up. */
PA_API pa_status pa_check_device_error(pa_handle h, int* code);

/* Wait sites.  Every bounded wait inside the library's kernels has an id
 * (kernel << 8) | index; the first wait of a step that gives up records
 * it beside the error word.  Kernel parts of the id: */
enum {
  PA_SITE_DECODE = 1 << 8,
  PA_SITE_COMBINE = 2 << 8,        /* index 1: the PA_OPT_WAIT_PROBE wait */
  PA_SITE_PREFILL = 3 << 8,        /* one-tile prefill (head_size 256) */
  PA_SITE_PREFILL_PAIR = 4 << 8,   /* two-tile prefill (head_size 64, 128) */
  PA_SITE_LATENT = 5 << 8,         /* latent decode, mma.sync */
  PA_SITE_LATENT_TC = 6 << 8       /* latent decode, tcgen05 */
};
/* The wait-site id read (and cleared) by the last pa_check_device_error on
 * h; 0 when no wait gave up. */
PA_API int pa_last_wait_site(pa_handle h);

/* Message of the last failure on h (or of the last pa_create / validation
 * failure on this thread when h is NULL).  Never NULL. */
PA_API const char* pa_last_error_message(pa_handle h);

/* Frees the workspace.  NULL is accepted. */
PA_API pa_status pa_destroy(pa_handle h);

/* The whole step (as pa_forward) for callers that cannot allocate device
 * memory: code running inside CUDA stream capture, under a memory pool
 * they do not own, in an allocation-free serving loop, or that simply has
 * no handle.  The design pages have no counterpart to this call.
 *
 * It needs no pa_create: cfg is passed on every call, and every scratch
 * buffer (work lists, split-KV partials, the rotated-query buffer, the
 * device error word) lives in one file-scope device array of 64 MiB that
 * each GPU loading this library holds until the process exits.  The call
 * makes no cudaMalloc/cudaFree and no other allocation; the caller still
 * passes every input and the output.  Capacities (max_batch, max_tokens,
 * head counts, head_size, do_rotary) whose scratch would exceed 64 MiB are
 * rejected with PA_INVALID_ARGUMENT and a message giving the size needed.
 *
 * device_error: optional caller-owned device int32 that receives the
 * PA_DEVERR_* bits (OR-ed; the caller clears it).  When NULL the bits go
 * to a word inside the shared scratch, cleared at the start of each call,
 * that the caller cannot read (so is the wait-site id of a timeout).
 *
 * It runs separate fp16 K/V caches without head_sink; an 8-bit or bfloat16
 * cache_dtype, packed_qkv, qk_norm or kv_cache_layout PA_LAYOUT_LATENT
 * returns PA_NOT_SUPPORTED (pa_forward_ex takes all of them and the sink).
 *
 * The first call on a device does a one-time set-up with that device
 * current (looks up the array's device address with cudaGetSymbolAddress,
 * sets the kernels' shared-memory attributes); make that first call before
 * any stream capture.  All calls share the one scratch array, which keeps
 * the last call's contents: calls that can overlap on the GPU (different
 * streams, or concurrent graphs) race on it and must be serialised by the
 * caller. */
PA_API pa_status pa_forward_no_alloc(const pa_config* cfg, const void* query, const void* key,
                                     const void* value, void* key_cache, void* value_cache,
                                     const int32_t* block_table,
                                     const int32_t* cumulative_sequence_lengths,
                                     const int32_t* past_sequence_lengths, int batch,
                                     int token_count, const void* cos_cache,
                                     const void* sin_cache, void* output,
                                     int32_t* device_error, void* stream);

/* ---- tuning and measurement hooks (set outside capture) ---- */
enum {
  PA_OPT_SPLIT_KEYS = 1,      /* > 0: fixed keys per decode split (multiple of 64); 0 = auto */
  PA_OPT_NO_WINDOW_PRUNE = 2, /* 1: walk the whole context and mask instead of pruning */
  PA_OPT_KERNEL_TIMING = 3,   /* 1: record CUDA events around each kernel of pa_forward */
  PA_OPT_DECODE_MAX_ROWS = 4, /* route a sequence to the decode kernel iff q_len*G <= value (0 = never; at most and by
                                 default the rows of a decode item: 8 when G <= 8, else 16) */
  PA_OPT_DECODE_ITEMS_PER_CTA = 5, /* target decode work items per decode CTA when splits are sized automatically:
                                      1..32, or 0 (default) = per step, 1 when the step's sequences x kv heads
                                      (latent: x work units per sequence) fill the decode grid, else 2 */
  PA_OPT_LATENT_TCGEN05 = 6,  /* latent layout: 1 (the default when the query heads are a multiple of 128)
                                 runs the tcgen05 latent kernel (units of 128 heads x half the value
                                 channels), 0 the mma.sync kernel (items of 32 heads, any head count);
                                 1 on other handles is PA_NOT_SUPPORTED */
  PA_OPT_PREFILL_SMS = 7,     /* steps with prompts and decode rows: the prefill kernel runs on P SMs and the
                                 decode kernel beside it on the rest; 0 (default) = P from the step's own work
                                 (cost model), -1 = no split (every prefill CTA works, the decode kernel
                                 fills SMs as they free), > 0 = P fixed (at most SMs - 1) */
  PA_OPT_WAIT_PROBE = 8       /* 1: the combine kernel also runs a bounded wait (2 ms) on a flag nothing sets,
                                 so that the step ends with PA_DEVERR_TIMEOUT at site PA_SITE_COMBINE | 1
                                 (a check of the timeout path; the step's outputs are unaffected) */
};
PA_API pa_status pa_set_option(pa_handle h, int option, int value);

/* Kernel stages of a step, for pa_kernel_time_ms.  In pa_forward the work
 * list and the cache write run as one launch (the prologue), timed as
 * PA_STAGE_WORKLIST; PA_STAGE_CACHE_WRITE times pa_cache_write. */
enum {
  PA_STAGE_WORKLIST = 0,
  PA_STAGE_CACHE_WRITE = 1,
  PA_STAGE_DECODE = 2,
  PA_STAGE_PREFILL = 3,
  PA_STAGE_COMBINE = 4,
  PA_NUM_STAGES = 5
};
/* With PA_OPT_KERNEL_TIMING on: synchronises, then returns in *ms the time
 * between the events recorded on the launch stream around that stage's
 * kernel in the last pa_forward (-1 when it did not launch). */
PA_API pa_status pa_kernel_time_ms(pa_handle h, int stage, float* ms);

/* Number of kernels the last pa_forward / pa_cache_write launched. */
PA_API int pa_last_launch_count(pa_handle h);

/* What the device work list of the last pa_forward on h decided (an
 * inspection hook for tests and tuning; synchronises, not capturable):
 * counts[PA_STEP_COUNTS] receives decode work items (sequence, split),
 * prefill tiles, packed rows merged by the combine kernel, keys per decode
 * split, prefill CTAs kept and decode CTAs kept (with the SM split of a
 * mixed step their sum is at most the SM count times the decode CTAs per
 * SM; without it they are the launched grids). */
enum { PA_STEP_COUNTS = 6 };
PA_API pa_status pa_last_step_counts(pa_handle h, int32_t* counts);

#ifdef __cplusplus
}
#endif
#endif /* PA_H_ */
