// Host side of the C ABI: validation, static planning, workspace, tensor
// maps and the launch sequence of one step.  Nothing here reads a device
// length: every per-step quantity is derived by the work-list kernel on the
// GPU, and the host only sizes launches and workspaces from the handle's
// static capacities ("PagedAttention - CUDA Design Document", section 4.7).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/pa.h"
#include "step.h"

namespace {

// Rates of the SM split's cost model (choose_split in worklist.cuh),
// measured on the mixed 16 x 1024 + 240-decode step: the two-tile prefill
// kernel's rate (772 TFLOP/s on 152 SMs), the decode kernel's bytes per SM
// when it runs on part of the SMs (51-66 GB/s for 56-112 SMs; the per-SM TMA
// inbound ceiling is about 74 GB/s), and the copy bandwidth.  A forced sweep
// of the prefill SMs on that step: 32 -> 894 us, 40 -> 815, 48 -> 829,
// 64 -> 884; without the split 842 us.
constexpr float kPrefillFlopsPerSmUs = 5.0e6f;
constexpr float kDecodeBytesPerSmUs = 55.0e3f;
constexpr float kHbmBytesPerUs = 6.7e6f;

// Largest decode items-per-CTA target (PA_OPT_DECODE_ITEMS_PER_CTA); the
// split-partial workspace is sized for it.
constexpr int kMaxItemsPerCta = 8;

thread_local std::string g_last_msg = "no error";

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

void set_msg(char* msg, size_t len, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_msg = buf;
  if (msg && len) {
    strncpy(msg, buf, len - 1);
    msg[len - 1] = 0;
  }
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Kernel of a wait-site id (site >> 8; the PA_SITE_* values of pa.h).
const char* wait_kernel_name(int k) {
  switch (k) {
    case 1: return "decode";
    case 2: return "combine";
    case 3: return "one-tile prefill";
    case 4: return "two-tile prefill";
    case 5: return "latent mma.sync";
    case 6: return "latent tcgen05";
    default: return "unknown";
  }
}

// 8-bit code caches (quantized); the 16-bit ones are fp16 and bfloat16.
bool quantized(int cache_dtype) { return cache_dtype == PA_CACHE_INT8 || cache_dtype == PA_CACHE_FP8_E4M3; }

// bfloat16 activations: a bfloat16 cache, or act_dtype PA_ACT_BF16 over an 8-bit one.
bool act_bf16(const pa_config& c) { return c.cache_dtype == PA_CACHE_BF16 || c.act_dtype == PA_ACT_BF16; }

int rot_dim_of(const pa_config& c) {
  if (!c.do_rotary) return 0;
  return c.rotary_dim > 0 ? c.rotary_dim : c.head_size;
}

// Whether attention reads a transformed copy of the query (rotated, QK-Norm
// normalized, unpacked from QKV rows, or times per-channel K scales) rather
// than the query itself.  A single per-tensor K scale multiplies the score
// scale instead (exact, CUDA design section 8.5 phase 3).  A bfloat16 query
// over an 8-bit cache is copied as fp16 (the operand type of that kernel).
bool query_copied(const pa_config& c) {
  const bool per_channel_k = quantized(c.cache_dtype) && c.k_quant_type == PA_QUANT_PER_CHANNEL;
  const bool bf16_over_codes = quantized(c.cache_dtype) && c.act_dtype == PA_ACT_BF16;
  return c.do_rotary || per_channel_k || c.packed_qkv || c.qk_norm || bf16_over_codes;
}

}  // namespace

struct pa_handle_s {
  pa_config cfg;
  int device = 0;
  int num_sms = 0;
  int G = 1, R = 0;
  float scale = 0.f;
  int max_q = 0, max_kv = 0;
  int dec_ctas_per_sm = 1, dec_grid = 1;
  bool latent = false;
  int groups = 1, dv = 0;  // decode work-list groups (kv heads, or 16-head groups of a latent step), output width
  int unit_groups = 1;     // decode CTA work units per (sequence, split)
  bool mla_tc_ready = false;  // the tcgen05 latent kernel can serve this handle (query heads a multiple of 128)
  bool mla_tc = false;        // ... and runs (the default; PA_OPT_LATENT_TCGEN05 = 0 selects the mma.sync kernel)
  size_t dec_smem = 0;
  int cap_dec = 1, cap_pre = 1, cap_comb = 1, cap_dseq = 1, cap_part = 1;
  int chunk_tokens = 0;  // > 0: query rows beyond one decode item run as decode entries of this many tokens
  int chunk_rows_max = 0;  // > 0: ... for sequences of at most this many rows (fp16 caches: the others prefill)
  int dec_rows = 16;      // query rows a decode item holds (decode_item_rows of the group)
  int prefill_tile_tokens = 1, prefill_q_tokens = 1, pre_grid = 1, comb_grid = 1;
  size_t pre_smem = 0;
  bool prefill_ready = false;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  pa::SeqInfo* seq = nullptr;   // sequence table
  pa::SeqInfo* dseq = nullptr;  // decode table
  int2* dec_items = nullptr;
  int2* pre_tiles = nullptr;
  int2* comb_rows = nullptr;
  pa::Counters* counters = nullptr;
  int* err = nullptr;
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  __half* q_rot = nullptr;
  int opt_split_keys = 0, opt_no_prune = 0, opt_timing = 0, opt_dec_rows = 0;
  int opt_items_per_cta = 0;  // 0: chosen per step (target_pairs_for)
  int opt_prefill_sms = 0;    // SM split of mixed steps: 0 cost model, -1 none, > 0 prefill CTAs kept
  int opt_wait_probe = 0;     // 1: the combine kernel runs its bounded wait on a flag nothing sets
  int last_site = 0;          // wait site read by the last pa_check_device_error
  cudaEvent_t ev[PA_NUM_STAGES][2] = {};
  bool stage_ran[PA_NUM_STAGES] = {};
  cudaStream_t last_stream = nullptr;
  int last_launches = 0;
  std::string msg = "no error";
};

namespace {

pa_status fail(pa_handle h, pa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_msg = buf;
  if (h) h->msg = buf;
  return st;
}

// Decode (sequence, split) items the work list aims for.  Splits balance
// the decode CTAs' load but cost a merge; measured on GB300: one item per CTA
// is best once the unsplit work units (sequences x kv heads, or latent units)
// fill the grid, two when they do not (few long sequences).
int target_pairs_for(pa_handle h, int batch) {
  const int ug = h->unit_groups;
  int ipc = h->opt_items_per_cta;
  if (ipc <= 0) ipc = (long long)batch * ug >= h->dec_grid ? 1 : pa::kDecodeItemsPerCta;
  return std::max(1, (ipc * h->dec_grid + ug - 1) / ug);
}

pa_status cuda_fail(pa_handle h, cudaError_t e, const char* what) {
  return fail(h, PA_CUDA_ERROR, "%s: %s", what, cudaGetErrorString(e));
}

// 3-D view {D, Hk, NB*bs} of an NHD pool (or {D, H, T} of a packed Q):
// box {64 channels, `heads` heads, `rows` rows}, 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* base, int D, int heads_total, long long rows_total, int heads_box,
                int rows_box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads_total, (cuuint64_t)rows_total};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)heads_total * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)heads_box, (cuuint32_t)rows_box};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 4-D view of an NHD pool {64 channels, NB*bs rows, D/64 chunks, Hk heads}
// (strides: row Hk*D*2 bytes, chunk 128 bytes, head D*2 bytes): a box
// {64, rows, D/64, 1} is one head's page laid out [chunk][row][128 B] with
// the 128-byte swizzle.  Every addressable byte lies inside the pool.
// With 8-bit elements (eb = 1) a chunk holds 128 channels.
bool encode_pool_map(CUtensorMap* m, const void* base, int D, int Hk, long long rows_total, int rows_box,
                     int eb = 2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int per_chunk = 128 / eb;
  cuuint64_t dims[4] = {(cuuint64_t)per_chunk, (cuuint64_t)rows_total, (cuuint64_t)(D / per_chunk), (cuuint64_t)Hk};
  cuuint64_t strides[3] = {(cuuint64_t)Hk * D * eb, 128, (cuuint64_t)D * eb};
  cuuint32_t box[4] = {(cuuint32_t)per_chunk, (cuuint32_t)rows_box, (cuuint32_t)(D / per_chunk), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(m, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                  const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
    else prev = -1;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

void pa_config_init(pa_config* c) {
  if (!c) return;
  memset(c, 0, sizeof(*c));
  c->local_window_size = -1;
  c->qk_norm_epsilon = 1e-6f;
}

pa_status pa_validate_config(const pa_config* c, char* msg, size_t len) {
  if (!c) {
    set_msg(msg, len, "config: NULL");
    return PA_INVALID_ARGUMENT;
  }
  if (c->num_heads <= 0) { set_msg(msg, len, "num_heads must be > 0 (got %d)", c->num_heads); return PA_INVALID_ARGUMENT; }
  if (c->kv_num_heads <= 0) { set_msg(msg, len, "kv_num_heads must be > 0 (got %d)", c->kv_num_heads); return PA_INVALID_ARGUMENT; }
  if (c->num_heads % c->kv_num_heads != 0) {
    set_msg(msg, len, "num_heads %% kv_num_heads must be 0 (got %d %% %d)", c->num_heads, c->kv_num_heads);
    return PA_INVALID_ARGUMENT;
  }
  if (c->head_size <= 0 || c->head_size % 8 != 0) {
    set_msg(msg, len, "head_size must be a positive multiple of 8 (got %d)", c->head_size);
    return PA_INVALID_ARGUMENT;
  }
  if (!is_pow2(c->block_size) || c->block_size < 16) {
    set_msg(msg, len, "block_size must be a power of two >= 16 (got %d)", c->block_size);
    return PA_INVALID_ARGUMENT;
  }
  if (c->num_blocks <= 0) { set_msg(msg, len, "num_blocks must be > 0 (got %d)", c->num_blocks); return PA_INVALID_ARGUMENT; }
  if ((long long)c->num_blocks * c->block_size > (1LL << 31) - 1024) {
    set_msg(msg, len, "num_blocks * block_size must be < 2^31 (got %lld)", (long long)c->num_blocks * c->block_size);
    return PA_INVALID_ARGUMENT;
  }
  if (c->max_blocks_per_seq <= 0) {
    set_msg(msg, len, "max_blocks_per_seq must be > 0 (got %d)", c->max_blocks_per_seq);
    return PA_INVALID_ARGUMENT;
  }
  if ((long long)c->max_blocks_per_seq * c->block_size > (1LL << 30)) {
    set_msg(msg, len, "max_blocks_per_seq * block_size must be <= 2^30");
    return PA_INVALID_ARGUMENT;
  }
  if (!(c->scale >= 0.f) || std::isinf(c->scale)) { set_msg(msg, len, "scale must be finite and >= 0 (got %g)", c->scale); return PA_INVALID_ARGUMENT; }
  if (!(c->softcap >= 0.f) || std::isinf(c->softcap)) { set_msg(msg, len, "softcap must be finite and >= 0 (got %g)", c->softcap); return PA_INVALID_ARGUMENT; }
  if (!(c->local_window_size == -1 || c->local_window_size >= 1)) {
    set_msg(msg, len, "local_window_size must be -1 or >= 1 (got %d)", c->local_window_size);
    return PA_INVALID_ARGUMENT;
  }
  if (c->do_rotary != 0 && c->do_rotary != 1) { set_msg(msg, len, "do_rotary must be 0 or 1 (got %d)", c->do_rotary); return PA_INVALID_ARGUMENT; }
  if (c->rotary_interleaved != 0 && c->rotary_interleaved != 1) {
    set_msg(msg, len, "rotary_interleaved must be 0 or 1 (got %d)", c->rotary_interleaved);
    return PA_INVALID_ARGUMENT;
  }
  if (c->do_rotary) {
    int R = rot_dim_of(*c);
    if (R <= 0 || R % 2 != 0 || R > c->head_size) {
      set_msg(msg, len, "rotary_dim must be even and in [2, head_size] (got %d)", R);
      return PA_INVALID_ARGUMENT;
    }
    if (c->max_rotary_positions <= 0) {
      set_msg(msg, len, "max_rotary_positions (cos_cache.shape[0]) must be > 0 with do_rotary");
      return PA_INVALID_ARGUMENT;
    }
  }
  if (c->max_batch <= 0) { set_msg(msg, len, "max_batch must be > 0 (got %d)", c->max_batch); return PA_INVALID_ARGUMENT; }
  if (c->max_tokens <= 0) { set_msg(msg, len, "max_tokens must be > 0 (got %d)", c->max_tokens); return PA_INVALID_ARGUMENT; }
  if (c->max_query_len_bound < 0 || c->max_kv_len_bound < 0) {
    set_msg(msg, len, "max_query_len_bound and max_kv_len_bound must be >= 0");
    return PA_INVALID_ARGUMENT;
  }
  if (c->cache_dtype < PA_CACHE_FP16 || c->cache_dtype > PA_CACHE_BF16) {
    set_msg(msg, len, "cache_dtype must be PA_CACHE_FP16, PA_CACHE_INT8, PA_CACHE_FP8_E4M3 or PA_CACHE_BF16 (got %d)",
            c->cache_dtype);
    return PA_INVALID_ARGUMENT;
  }
  if (c->act_dtype != PA_ACT_DEFAULT && c->act_dtype != PA_ACT_BF16) {
    set_msg(msg, len, "act_dtype must be PA_ACT_DEFAULT or PA_ACT_BF16 (got %d)", c->act_dtype);
    return PA_INVALID_ARGUMENT;
  }
  if (c->act_dtype == PA_ACT_BF16 && c->cache_dtype == PA_CACHE_FP16) {
    set_msg(msg, len, "act_dtype PA_ACT_BF16 needs an int8, e4m3 or bfloat16 cache (bfloat16 activations "
                      "with 16-bit pools are cache_dtype PA_CACHE_BF16)");
    return PA_INVALID_ARGUMENT;
  }
  for (int qt : {c->k_quant_type, c->v_quant_type})
    if (qt < PA_QUANT_NONE || qt > PA_QUANT_PER_CHANNEL) {
      set_msg(msg, len, "k_quant_type / v_quant_type must be PA_QUANT_NONE, PER_TENSOR or PER_CHANNEL (got %d)", qt);
      return PA_INVALID_ARGUMENT;
    }
  if (!quantized(c->cache_dtype) && (c->k_quant_type != PA_QUANT_NONE || c->v_quant_type != PA_QUANT_NONE)) {
    set_msg(msg, len, "k_quant_type / v_quant_type must be PA_QUANT_NONE with a 16-bit cache");
    return PA_INVALID_ARGUMENT;
  }
  if (quantized(c->cache_dtype) && (c->k_quant_type == PA_QUANT_NONE || c->v_quant_type == PA_QUANT_NONE)) {
    set_msg(msg, len, "an 8-bit cache needs k_quant_type and v_quant_type PER_TENSOR or PER_CHANNEL");
    return PA_INVALID_ARGUMENT;
  }
  if (c->kv_cache_layout != PA_LAYOUT_SEPARATE && c->kv_cache_layout != PA_LAYOUT_LATENT) {
    set_msg(msg, len, "kv_cache_layout must be PA_LAYOUT_SEPARATE or PA_LAYOUT_LATENT (got %d)", c->kv_cache_layout);
    return PA_INVALID_ARGUMENT;
  }
  const bool latent = c->kv_cache_layout == PA_LAYOUT_LATENT;
  if (c->v_head_size < 0 || c->v_head_size > c->head_size) {
    set_msg(msg, len, "v_head_size must be in [0, head_size] (got %d)", c->v_head_size);
    return PA_INVALID_ARGUMENT;
  }
  if (!latent && c->v_head_size != 0 && c->v_head_size != c->head_size) {
    set_msg(msg, len, "v_head_size != head_size requires kv_cache_layout LATENT");
    return PA_INVALID_ARGUMENT;
  }
  if (c->rotary_offset < 0 || c->rotary_offset % 8 != 0 ||
      (c->do_rotary && c->rotary_offset + rot_dim_of(*c) > c->head_size)) {
    set_msg(msg, len, "rotary_offset must be a multiple of 8 with rotary_offset + rotary_dim <= head_size (got %d)",
            c->rotary_offset);
    return PA_INVALID_ARGUMENT;
  }
  if (latent) {
    if (c->kv_num_heads != 1) {
      set_msg(msg, len, "kv_cache_layout LATENT requires kv_num_heads == 1 (got %d)", c->kv_num_heads);
      return PA_INVALID_ARGUMENT;
    }
    if (c->v_head_size != 0 && c->v_head_size != c->head_size && !(c->scale > 0.f)) {
      set_msg(msg, len, "v_head_size != head_size needs an explicit scale (1/sqrt(head_size) is not the model's)");
      return PA_INVALID_ARGUMENT;
    }
    if (c->qk_norm || c->packed_qkv) {
      set_msg(msg, len, "kv_cache_layout LATENT takes neither qk_norm nor packed_qkv");
      return PA_INVALID_ARGUMENT;
    }
    if (c->k_quant_type != PA_QUANT_NONE || c->v_quant_type != PA_QUANT_NONE || c->cache_dtype != PA_CACHE_FP16) {
      set_msg(msg, len, "the latent layout is built for an fp16 cache only");
      return PA_NOT_SUPPORTED;
    }
  }
  if (c->packed_qkv != 0 && c->packed_qkv != 1) {
    set_msg(msg, len, "packed_qkv must be 0 or 1 (got %d)", c->packed_qkv);
    return PA_INVALID_ARGUMENT;
  }
  if (c->qk_norm != 0 && c->qk_norm != 1) {
    set_msg(msg, len, "qk_norm must be 0 or 1 (got %d)", c->qk_norm);
    return PA_INVALID_ARGUMENT;
  }
  if (c->qk_norm && !(c->qk_norm_epsilon > 0.f && std::isfinite(c->qk_norm_epsilon))) {
    set_msg(msg, len, "qk_norm_epsilon must be finite and > 0 (got %g)", c->qk_norm_epsilon);
    return PA_INVALID_ARGUMENT;
  }
  // Valid, but outside what this library runs.
  if (latent) {
    const int dv = c->v_head_size ? c->v_head_size : c->head_size;
    const long long qb =
        c->max_query_len_bound > 0 ? std::min(c->max_query_len_bound, c->max_tokens) : c->max_tokens;
    if (c->head_size != 576 || dv != 512) {
      set_msg(msg, len, "the latent layout is built for head_size 576, v_head_size 512 (got %d, %d)", c->head_size, dv);
      return PA_NOT_SUPPORTED;
    }
    if (c->num_heads > 16 && c->num_heads % 16 != 0) {
      set_msg(msg, len, "the latent layout is built for num_heads <= 16 or a multiple of 16 (got %d)", c->num_heads);
      return PA_NOT_SUPPORTED;
    }
    (void)qb;  // longer query rows run as one-token decode entries
    set_msg(msg, len, "ok");
    return PA_OK;
  }
  if (c->head_size != 64 && c->head_size != 128 && c->head_size != 256) {
    set_msg(msg, len, "head_size %d is valid but this library runs 64, 128 and 256", c->head_size);
    return PA_NOT_SUPPORTED;
  }
  if (c->num_heads / c->kv_num_heads > 128) {
    set_msg(msg, len, "num_heads / kv_num_heads = %d > 128 is not supported", c->num_heads / c->kv_num_heads);
    return PA_NOT_SUPPORTED;
  }
  if (c->do_rotary && rot_dim_of(*c) % 16 != 0) {
    set_msg(msg, len, "rotary_dim %d is valid but this library needs a multiple of 16", rot_dim_of(*c));
    return PA_NOT_SUPPORTED;
  }
  if (c->qk_norm && c->kv_num_heads > 32) {
    set_msg(msg, len, "qk_norm is built for kv_num_heads <= 32 (got %d)", c->kv_num_heads);
    return PA_NOT_SUPPORTED;
  }
  if (quantized(c->cache_dtype)) {
    if (c->k_quant_type != c->v_quant_type) {
      set_msg(msg, len, "k_quant_type and v_quant_type must match in this library");
      return PA_NOT_SUPPORTED;
    }
    if (c->head_size == 64) {
      set_msg(msg, len, "8-bit caches are built for head_size 128 and 256 (got 64)");
      return PA_NOT_SUPPORTED;
    }
    // 8-bit caches run the decode kernel only (longer query rows in chunks of
    // 16 / G tokens), whose items hold one kv head's group of up to 16 rows
    if (c->num_heads / c->kv_num_heads > pa::kDecodeRows) {
      set_msg(msg, len, "8-bit caches are built for num_heads / kv_num_heads <= %d (got %d)", pa::kDecodeRows,
              c->num_heads / c->kv_num_heads);
      return PA_NOT_SUPPORTED;
    }
  }
  set_msg(msg, len, "ok");
  return PA_OK;
}

pa_status pa_check_step(const pa_config* c, int for_forward, const void* query, const void* key, const void* value,
                        const void* key_cache, const void* value_cache, const int32_t* block_table,
                        const int32_t* cum, const int32_t* past, int batch, int token_count, const void* cos_cache,
                        const void* sin_cache, const void* output, char* msg, size_t len) {
  pa_status st = pa_validate_config(c, msg, len);
  if (st != PA_OK) return st;
  if (batch < 1 || batch > c->max_batch) {
    set_msg(msg, len, "batch must be in [1, max_batch=%d] (got %d)", c->max_batch, batch);
    return PA_INVALID_ARGUMENT;
  }
  if (token_count < 0 || token_count > c->max_tokens) {
    set_msg(msg, len, "token_count must be in [0, max_tokens=%d] (got %d)", c->max_tokens, token_count);
    return PA_INVALID_ARGUMENT;
  }
  const bool packed = for_forward != 0 && c->packed_qkv;
  const bool latent = c->kv_cache_layout == PA_LAYOUT_LATENT;
  if (latent && (value || value_cache)) {
    set_msg(msg, len, "value and value_cache must be NULL with kv_cache_layout LATENT");
    return PA_INVALID_ARGUMENT;
  }
  if (packed && (key || value)) {
    set_msg(msg, len, "key and value must be NULL with packed_qkv (the query rows hold Q, K and V)");
    return PA_INVALID_ARGUMENT;
  }
  struct { const void* p; const char* name; int align; bool need; } args[] = {
      {query, "query", 16, for_forward != 0 && token_count > 0},
      {key, "key", 16, !packed && token_count > 0},
      {value, "value", 16, !packed && !latent && token_count > 0},
      {key_cache, "key_cache", 16, true},
      {value_cache, "value_cache", 16, !latent},
      {block_table, "block_table", 4, true},
      {cum, "cumulative_sequence_lengths", 4, true},
      {past, "past_sequence_lengths", 4, true},
      {output, "output", 16, for_forward != 0 && token_count > 0},
  };
  for (auto& a : args) {
    if (a.need && a.p == nullptr) {
      set_msg(msg, len, "%s must not be NULL", a.name);
      return PA_INVALID_ARGUMENT;
    }
    if (a.p && (reinterpret_cast<uintptr_t>(a.p) % a.align) != 0) {
      set_msg(msg, len, "%s must be %d-byte aligned", a.name, a.align);
      return PA_INVALID_ARGUMENT;
    }
  }
  if (!latent && key_cache == value_cache) {
    set_msg(msg, len, "key_cache and value_cache must be distinct buffers");
    return PA_INVALID_ARGUMENT;
  }
  if ((cos_cache == nullptr) != (sin_cache == nullptr)) {
    set_msg(msg, len, "cos_cache and sin_cache must be both present or both absent");
    return PA_INVALID_ARGUMENT;
  }
  if (c->do_rotary && cos_cache == nullptr) {
    set_msg(msg, len, "cos_cache/sin_cache are required when do_rotary == 1");
    return PA_INVALID_ARGUMENT;
  }
  if (!c->do_rotary && cos_cache != nullptr) {
    set_msg(msg, len, "cos_cache/sin_cache given but do_rotary == 0");
    return PA_INVALID_ARGUMENT;
  }
  if (cos_cache && ((reinterpret_cast<uintptr_t>(cos_cache) | reinterpret_cast<uintptr_t>(sin_cache)) % 16)) {
    set_msg(msg, len, "cos_cache and sin_cache must be 16-byte aligned");
    return PA_INVALID_ARGUMENT;
  }
  set_msg(msg, len, "ok");
  return PA_OK;
}

pa_status pa_create(const pa_config* cfg, pa_handle* out) {
  if (!out) return fail(nullptr, PA_INVALID_ARGUMENT, "out must not be NULL");
  *out = nullptr;
  char msg[512];
  pa_status st = pa_validate_config(cfg, msg, sizeof(msg));
  if (st != PA_OK) return fail(nullptr, st, "%s", msg);
  pa_handle h = new pa_handle_s();
  h->cfg = *cfg;
  const pa_config& c = h->cfg;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e != cudaSuccess) { delete h; return cuda_fail(nullptr, e, "cudaGetDevice"); }
  e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) { delete h; return cuda_fail(nullptr, e, "cudaDeviceGetAttribute"); }
  if (!encode_fn()) { delete h; return fail(nullptr, PA_CUDA_ERROR, "cuTensorMapEncodeTiled is unavailable"); }

  h->latent = c.kv_cache_layout == PA_LAYOUT_LATENT;
  // A latent step works on groups of 16 query heads of one token (rows of a
  // decode item); the group plays the part of a kv head in the work list.
  h->G = h->latent ? pa::kDecodeRows : c.num_heads / c.kv_num_heads;
  h->groups = h->latent ? std::max(1, c.num_heads / pa::kDecodeRows) : c.kv_num_heads;
  h->dv = h->latent ? 512 : c.head_size;
  h->dec_rows = pa::decode_item_rows(h->G);  // rows a decode item holds (0: no decode route)
  h->opt_dec_rows = h->dec_rows;
  h->R = rot_dim_of(c);
  h->scale = c.scale > 0.f ? c.scale : 1.f / std::sqrt((float)c.head_size);
  const int kv_cap = c.max_blocks_per_seq * c.block_size;
  h->max_q = c.max_query_len_bound > 0 ? std::min(c.max_query_len_bound, c.max_tokens) : c.max_tokens;
  h->max_kv = c.max_kv_len_bound > 0 ? std::min(c.max_kv_len_bound, kv_cap) : kv_cap;

  if (h->latent) {
    h->mla_tc_ready = c.num_heads % 128 == 0;
    e = pa::mla_configure(&h->dec_smem);
    size_t tc_smem = 0;
    if (e == cudaSuccess && h->mla_tc_ready) e = pa::mla_tc_configure(&tc_smem);
    h->dec_ctas_per_sm = 1;
  } else {
    e = pa::decode_configure(c.head_size, c.cache_dtype, h->G, &h->dec_ctas_per_sm, &h->dec_smem);
  }
  if (e != cudaSuccess) { delete h; return cuda_fail(nullptr, e, "decode kernel attributes"); }
  size_t psmem = 0;
  h->prefill_ready = !h->latent && pa::prefill_configure(c.head_size, &psmem) == cudaSuccess;
  cudaGetLastError();
  h->pre_smem = psmem;

  h->dec_grid = h->num_sms * h->dec_ctas_per_sm;
  // decode CTA work units per (sequence, split): kv heads, or the 32-head
  // groups of a latent step
  // work units per item of the tcgen05 latent kernel: 128-head tiles x value halves
  const int tc_units = h->mla_tc_ready ? 2 * (c.num_heads / 128) : 1;
  h->mla_tc = h->mla_tc_ready;
  h->unit_groups = h->mla_tc ? tc_units : h->latent ? pa::mla_item_groups(h->groups) : h->groups;
  // Query rows beyond one decode item: decode entries of dec_rows / G
  // tokens for 8-bit caches and the latent layout (one token: G is 16
  // there); with fp16 caches only for short multi-token sequences (two
  // chunks at most: each chunk reads the sequence's keys again, and the
  // prefill kernel's fixed cost is not repaid by a few rows), longer ones
  // take the prefill kernel.
  const bool quant = quantized(c.cache_dtype);
  h->chunk_tokens = h->dec_rows > 0 ? std::max(1, h->dec_rows / h->G) : 0;
  h->chunk_rows_max = (h->latent || quant) ? 0 : 2 * h->chunk_tokens * h->G;
  // Decode entries: one per sequence, or one per chunk (with fp16 caches a
  // chunked sequence has more than chunk_tokens tokens and two entries).
  if (h->chunk_rows_max > 0)
    h->cap_dseq = c.max_batch + std::min(c.max_batch, c.max_tokens / (h->chunk_tokens + 1));
  else
    h->cap_dseq = c.max_batch + (h->chunk_tokens ? (c.max_tokens + h->chunk_tokens - 1) / h->chunk_tokens : 0);
  // Decode items: the split targets (room for the items-per-CTA option's
  // maximum, sized for whichever latent kernel makes the most items) plus
  // one last split per entry.  Split partials: with automatic split sizes
  // a step has at most as many full splits as split targets, and at most as
  // many split entries as full splits.
  const int ug_min = h->mla_tc_ready ? std::min(tc_units, pa::mla_item_groups(h->groups)) : h->unit_groups;
  const int target_max = std::max(1, (kMaxItemsPerCta * h->dec_grid + ug_min - 1) / ug_min);
  h->cap_dec = target_max + h->cap_dseq;
  h->cap_part = 2 * target_max;
  // Prefill work units: unit tokens (the work list's tiles) and the tokens
  // of one 128-row query tile (the Q TMA box).
  h->prefill_tile_tokens = pa::prefill_unit_tokens(c.head_size, h->G);
  h->prefill_q_tokens = std::max(1, pa::kPrefillRows / h->G);
  h->cap_pre = (c.max_tokens + h->prefill_tile_tokens - 1) / h->prefill_tile_tokens + c.max_batch;
  h->cap_comb = c.max_tokens;
  h->pre_grid = std::max(1, std::min(h->num_sms, h->cap_pre * c.kv_num_heads));
  h->comb_grid = std::max(1, std::min(h->num_sms * 4, (h->cap_comb * c.num_heads + 7) / 8));

  // Workspace layout (256-byte aligned pieces).
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t D = h->dv, Hk = h->groups;  // split partials: [items, groups or kv heads, 16 rows, output width]
  size_t off = 0;
  size_t o_err = off; off = up(off + 64);
  size_t o_cnt = off; off = up(off + sizeof(pa::Counters));
  size_t o_seq = off; off = up(off + sizeof(pa::SeqInfo) * c.max_batch);
  size_t o_dsq = off; off = up(off + sizeof(pa::SeqInfo) * h->cap_dseq);
  size_t o_dec = off; off = up(off + sizeof(int2) * h->cap_dec);
  size_t o_pre = off; off = up(off + sizeof(int2) * h->cap_pre);
  size_t o_cmb = off; off = up(off + sizeof(int2) * h->cap_comb);
  size_t o_pml = off; off = up(off + sizeof(float2) * h->cap_part * Hk * pa::kDecodeRows);
  size_t o_po = off; off = up(off + sizeof(float) * h->cap_part * Hk * pa::kDecodeRows * D);
  size_t o_qr = off;
  // rotated, normalized, unpacked and/or times k_scale
  const bool q_copy = query_copied(c);
  if (q_copy) off = up(off + 2 * (size_t)c.max_tokens * c.num_heads * c.head_size);
  h->ws_bytes = off;
  e = cudaMalloc(&h->ws, h->ws_bytes);
  if (e != cudaSuccess) { delete h; return cuda_fail(nullptr, e, "cudaMalloc(workspace)"); }
  e = cudaMemset(h->ws, 0, h->ws_bytes);
  if (e != cudaSuccess) { cudaFree(h->ws); delete h; return cuda_fail(nullptr, e, "cudaMemset(workspace)"); }
  uint8_t* w = static_cast<uint8_t*>(h->ws);
  h->err = reinterpret_cast<int*>(w + o_err);
  h->counters = reinterpret_cast<pa::Counters*>(w + o_cnt);
  h->seq = reinterpret_cast<pa::SeqInfo*>(w + o_seq);
  h->dseq = reinterpret_cast<pa::SeqInfo*>(w + o_dsq);
  h->dec_items = reinterpret_cast<int2*>(w + o_dec);
  h->pre_tiles = reinterpret_cast<int2*>(w + o_pre);
  h->comb_rows = reinterpret_cast<int2*>(w + o_cmb);
  h->part_ml = reinterpret_cast<float2*>(w + o_pml);
  h->part_o = reinterpret_cast<float*>(w + o_po);
  h->q_rot = q_copy ? reinterpret_cast<__half*>(w + o_qr) : nullptr;
  for (int i = 0; i < PA_NUM_STAGES; ++i)
    for (int j = 0; j < 2; ++j) cudaEventCreate(&h->ev[i][j]);
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { pa_destroy(h); return cuda_fail(nullptr, e, "pa_create"); }
  *out = h;
  return PA_OK;
}

pa_status pa_destroy(pa_handle h) {
  if (!h) return PA_OK;
  DeviceGuard g(h->device);
  for (int i = 0; i < PA_NUM_STAGES; ++i)
    for (int j = 0; j < 2; ++j)
      if (h->ev[i][j]) cudaEventDestroy(h->ev[i][j]);
  if (h->ws) cudaFree(h->ws);
  delete h;
  return PA_OK;
}

const char* pa_last_error_message(pa_handle h) { return h ? h->msg.c_str() : g_last_msg.c_str(); }

pa_status pa_set_option(pa_handle h, int option, int value) {
  if (!h) return fail(nullptr, PA_INVALID_ARGUMENT, "handle must not be NULL");
  switch (option) {
    case PA_OPT_SPLIT_KEYS: {
      if (value < 0 || value % pa::kStageKeys != 0)
        return fail(h, PA_INVALID_ARGUMENT, "split keys must be 0 or a positive multiple of %d", pa::kStageKeys);
      if (value > 0) {
        // every decode entry split at most max_kv / value + 1 ways
        long long need = (long long)h->cap_dseq * ((h->max_kv + value - 1) / value + 1);
        if (need > h->cap_dec || need > h->cap_part)
          return fail(h, PA_INVALID_ARGUMENT,
                      "split keys %d could need %lld decode items; the workspace holds %d items and %d split "
                      "partials", value, need, h->cap_dec, h->cap_part);
      }
      h->opt_split_keys = value;
      return PA_OK;
    }
    case PA_OPT_NO_WINDOW_PRUNE: h->opt_no_prune = value != 0; return PA_OK;
    case PA_OPT_KERNEL_TIMING: h->opt_timing = value != 0; return PA_OK;
    case PA_OPT_LATENT_TCGEN05:
      if (value != 0 && !h->mla_tc_ready)
        return fail(h, PA_NOT_SUPPORTED, "the tcgen05 latent kernel needs kv_cache_layout LATENT and a multiple of "
                                         "128 query heads");
      h->mla_tc = value != 0;
      h->unit_groups = h->mla_tc ? 2 * (h->cfg.num_heads / 128) : pa::mla_item_groups(h->groups);
      return PA_OK;
    case PA_OPT_DECODE_ITEMS_PER_CTA:
      if (value < 0 || value > kMaxItemsPerCta)
        return fail(h, PA_INVALID_ARGUMENT, "decode items per CTA must be 0 (automatic) or in [1, %d]",
                    kMaxItemsPerCta);
      h->opt_items_per_cta = value;
      return PA_OK;
    case PA_OPT_PREFILL_SMS:
      if (value < -1 || value >= h->num_sms)
        return fail(h, PA_INVALID_ARGUMENT, "prefill SMs must be -1 (no split), 0 (cost model) or in [1, %d]",
                    h->num_sms - 1);
      h->opt_prefill_sms = value;
      return PA_OK;
    case PA_OPT_WAIT_PROBE: h->opt_wait_probe = value != 0; return PA_OK;
    case PA_OPT_DECODE_MAX_ROWS:
      if ((quantized(h->cfg.cache_dtype) || h->latent) && value != h->dec_rows)
        return fail(h, PA_NOT_SUPPORTED, "8-bit caches and the latent layout route every row to decode items");
      if (value < 0 || value > h->dec_rows)
        return fail(h, PA_INVALID_ARGUMENT, "decode max rows must be in [0, %d]", h->dec_rows);
      h->opt_dec_rows = value;
      return PA_OK;
    default: return fail(h, PA_INVALID_ARGUMENT, "unknown option %d", option);
  }
}

int pa_last_launch_count(pa_handle h) { return h ? h->last_launches : 0; }

pa_status pa_kernel_time_ms(pa_handle h, int stage, float* ms) {
  if (!h || !ms || stage < 0 || stage >= PA_NUM_STAGES) return fail(h, PA_INVALID_ARGUMENT, "bad arguments");
  *ms = -1.f;
  if (!h->opt_timing || !h->stage_ran[stage]) return PA_OK;
  DeviceGuard g(h->device);
  cudaError_t e = cudaEventSynchronize(h->ev[stage][1]);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventSynchronize");
  e = cudaEventElapsedTime(ms, h->ev[stage][0], h->ev[stage][1]);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaEventElapsedTime");
  return PA_OK;
}

pa_status pa_check_device_error(pa_handle h, int* code) {
  if (!h || !code) return fail(h, PA_INVALID_ARGUMENT, "bad arguments");
  DeviceGuard g(h->device);
  cudaError_t e = cudaStreamSynchronize(h->last_stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  int v[2] = {0, 0};  // error bits, first wait site that gave up
  e = cudaMemcpy(v, h->err, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemcpy(error word)");
  e = cudaMemset(h->err, 0, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemset(error word)");
  *code = v[0];
  h->last_site = v[1];
  if (v[0] && v[1])
    return fail(h, PA_DEVICE_DATA_ERROR, "device data error bits 0x%x; a wait gave up at site 0x%x (%s kernel, wait %d)",
                v[0], v[1], wait_kernel_name(v[1] >> 8), v[1] & 0xff);
  if (v[0]) return fail(h, PA_DEVICE_DATA_ERROR, "device data error bits 0x%x", v[0]);
  return PA_OK;
}

int pa_last_wait_site(pa_handle h) { return h ? h->last_site : 0; }

pa_status pa_last_step_counts(pa_handle h, int32_t* counts) {
  if (!h || !counts) return fail(h, PA_INVALID_ARGUMENT, "bad arguments");
  DeviceGuard g(h->device);
  cudaError_t e = cudaStreamSynchronize(h->last_stream);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaStreamSynchronize");
  pa::Counters c;
  e = cudaMemcpy(&c, h->counters, sizeof(c), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaMemcpy(counters)");
  const int32_t v[PA_STEP_COUNTS] = {c.n_dec, c.n_pre, c.n_comb, c.split_keys, c.pre_ctas, c.dec_ctas};
  memcpy(counts, v, sizeof(v));
  return PA_OK;
}

}  // extern "C"

namespace {

// Records the stage's start/end events on the launch stream.  Inside a
// stream capture they become external event-record nodes, so the events
// still measure the kernel when the graph is replayed.
void record(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else cudaEventRecord(ev, s);
}

struct StageTimer {
  pa_handle h;
  int stage;
  cudaStream_t s;
  StageTimer(pa_handle h_, int st, cudaStream_t s_) : h(h_), stage(st), s(s_) {
    if (h->opt_timing) record(h->ev[stage][0], s);
  }
  ~StageTimer() {
    if (h->opt_timing) {
      record(h->ev[stage][1], s);
      h->stage_ran[stage] = true;
    }
  }
};

// Parameters of the prologue's rotary / cache-write warps.  Shared by the
// handle's steps and the entry point without a handle, so the two cannot
// drift apart: q_ws is the query-copy workspace (rotated, normalized,
// unpacked and/or times k_scale), used whenever the query is transformed.
pa::CacheWriteParams cache_write_params(const pa_config& c, __half* q_ws, int* err, const void* query,
                                        const void* key, const void* value, void* key_cache, void* value_cache,
                                        const int32_t* block_table, const int32_t* cum, const int32_t* past,
                                        int batch, int token_count, const void* cos_cache, const void* sin_cache,
                                        const pa_extra_inputs* x) {
  const bool quant = quantized(c.cache_dtype);
  const bool latent = c.kv_cache_layout == PA_LAYOUT_LATENT;
  const int R = rot_dim_of(c);
  const bool q_scaled = quant && c.k_quant_type == PA_QUANT_PER_CHANNEL;
  pa::CacheWriteParams p{};
  p.key = static_cast<const __half*>(key);
  p.value = static_cast<const __half*>(value);
  p.query = static_cast<const __half*>(query);
  p.q_rot = (query && query_copied(c)) ? q_ws : nullptr;
  p.key_cache = key_cache;
  p.value_cache = value_cache;
  p.cache_type = c.cache_dtype;
  p.act_bf16 = (quant && c.act_dtype == PA_ACT_BF16) ? 1 : 0;
  p.per_channel = c.k_quant_type == PA_QUANT_PER_CHANNEL;
  p.k_scale = quant ? x->k_scale : nullptr;
  p.v_scale = quant ? x->v_scale : nullptr;
  p.q_scale = (query && q_scaled) ? 1 : 0;
  p.slot_mapping = x->slot_mapping;
  p.packed = (query && c.packed_qkv) ? 1 : 0;
  p.q_stride = (p.packed ? c.num_heads + 2 * c.kv_num_heads : c.num_heads) * c.head_size;
  p.qk_norm = c.qk_norm;
  p.qk_eps = c.qk_norm_epsilon;
  p.q_norm_w = static_cast<const __half*>(x->q_norm_weight);
  p.k_norm_w = static_cast<const __half*>(x->k_norm_weight);
  p.block_table = block_table;
  p.cum = cum;
  p.past = past;
  p.cos_cache = static_cast<const __half*>(cos_cache);
  p.sin_cache = static_cast<const __half*>(sin_cache);
  p.batch = batch;
  p.token_count = token_count;
  p.H = c.num_heads;
  p.Hk = c.kv_num_heads;
  p.D = c.head_size;
  p.bs = c.block_size;
  p.NB = c.num_blocks;
  p.MB = c.max_blocks_per_seq;
  p.rotary = c.do_rotary;
  p.interleaved = c.rotary_interleaved;
  p.rot_dim = R;
  p.rot_positions = c.max_rotary_positions;
  p.rot_offset = c.rotary_offset;
  // A latent query copy keeps only the 64-channel chunks that hold rotated
  // channels; the latent kernels read the others from the query itself.
  p.q_keep_lo = 0;
  p.q_keep_hi = c.head_size;
  if (latent && c.do_rotary) {
    p.q_keep_lo = c.rotary_offset / 64 * 64;
    p.q_keep_hi = (c.rotary_offset + R + 63) / 64 * 64;
  }
  // Spread a token over several warps when Q is rotated too: one for the
  // K/V rows and one per kv_num_heads query heads (same size as a K row).
  p.q_heads_per_part = c.kv_num_heads;
  // 8-bit caches divide every element by its scale: their K and V rows go
  // to separate warps, each for up to half the kv heads
  p.kv_heads_per_part = quant ? std::max(1, (c.kv_num_heads + 1) / 2) : c.kv_num_heads;
  p.kv_parts = quant ? 2 * ((c.kv_num_heads + p.kv_heads_per_part - 1) / p.kv_heads_per_part) : 1;
  p.parts = p.kv_parts + (p.q_rot ? (c.num_heads + p.q_heads_per_part - 1) / p.q_heads_per_part : 0);
  p.err = err;
  return p;
}

const pa_extra_inputs kNoExtra = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};

// The optional inputs against the configuration: scales exactly for 8-bit
// caches, element alignment.
pa_status check_extra(pa_handle h, const pa_extra_inputs* x) {
  const bool quant = quantized(h->cfg.cache_dtype);
  if (quant && (!x->k_scale || !x->v_scale))
    return fail(h, PA_INVALID_ARGUMENT, "k_scale and v_scale are required with an 8-bit cache");
  if (!quant && (x->k_scale || x->v_scale))
    return fail(h, PA_INVALID_ARGUMENT, "k_scale / v_scale given but the cache is 16-bit");
  if ((reinterpret_cast<uintptr_t>(x->k_scale) | reinterpret_cast<uintptr_t>(x->v_scale)) % 4)
    return fail(h, PA_INVALID_ARGUMENT, "k_scale and v_scale must be 4-byte aligned");
  if (reinterpret_cast<uintptr_t>(x->head_sink) % 2)
    return fail(h, PA_INVALID_ARGUMENT, "head_sink must be 2-byte aligned");
  if (reinterpret_cast<uintptr_t>(x->slot_mapping) % 4)
    return fail(h, PA_INVALID_ARGUMENT, "slot_mapping must be 4-byte aligned");
  if (h->cfg.kv_cache_layout == PA_LAYOUT_LATENT && x->head_sink)
    return fail(h, PA_INVALID_ARGUMENT, "head_sink is not taken with kv_cache_layout LATENT");
  if (h->cfg.qk_norm && (!x->q_norm_weight || !x->k_norm_weight))
    return fail(h, PA_INVALID_ARGUMENT, "q_norm_weight and k_norm_weight are both required with qk_norm");
  if (!h->cfg.qk_norm && (x->q_norm_weight || x->k_norm_weight))
    return fail(h, PA_INVALID_ARGUMENT, "q_norm_weight / k_norm_weight given but qk_norm is 0");
  if ((reinterpret_cast<uintptr_t>(x->q_norm_weight) | reinterpret_cast<uintptr_t>(x->k_norm_weight)) % 16)
    return fail(h, PA_INVALID_ARGUMENT, "q_norm_weight and k_norm_weight must be 16-byte aligned");
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_cache_write(pa_handle h, const void* key, const void* value, void* key_cache, void* value_cache,
                         const int32_t* block_table, const int32_t* cum, const int32_t* past, int batch,
                         int token_count, const void* cos_cache, const void* sin_cache, void* stream) {
  return pa_cache_write_ex(h, key, value, key_cache, value_cache, block_table, cum, past, batch, token_count,
                           cos_cache, sin_cache, nullptr, stream);
}

pa_status pa_cache_write_ex(pa_handle h, const void* key, const void* value, void* key_cache, void* value_cache,
                            const int32_t* block_table, const int32_t* cum, const int32_t* past, int batch,
                            int token_count, const void* cos_cache, const void* sin_cache,
                            const pa_extra_inputs* extra, void* stream) {
  if (!h) return fail(nullptr, PA_INVALID_ARGUMENT, "handle must not be NULL");
  char msg[512];
  pa_status st = pa_check_step(&h->cfg, 0, nullptr, key, value, key_cache, value_cache, block_table, cum, past,
                               batch, token_count, cos_cache, sin_cache, nullptr, msg, sizeof(msg));
  if (st != PA_OK) return fail(h, st, "%s", msg);
  const pa_extra_inputs* x = extra ? extra : &kNoExtra;
  st = check_extra(h, x);
  if (st != PA_OK) return st;
  h->last_launches = 0;
  for (bool& r : h->stage_ran) r = false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->last_stream = s;
  if (token_count == 0) return PA_OK;
  DeviceGuard g(h->device);
  pa::CacheWriteParams p = cache_write_params(h->cfg, h->q_rot, h->err, nullptr, key, value, key_cache, value_cache,
                                              block_table, cum, past, batch, token_count, cos_cache, sin_cache, x);
  StageTimer t(h, PA_STAGE_CACHE_WRITE, s);
  cudaError_t e = pa::launch_cache_write(p, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "cache write launch");
  h->last_launches++;
  return PA_OK;
}

pa_status pa_forward(pa_handle h, const void* query, const void* key, const void* value, void* key_cache,
                     void* value_cache, const int32_t* block_table, const int32_t* cum, const int32_t* past,
                     int batch, int token_count, const void* cos_cache, const void* sin_cache, void* output,
                     void* stream) {
  return pa_forward_ex(h, query, key, value, key_cache, value_cache, block_table, cum, past, batch, token_count,
                       cos_cache, sin_cache, nullptr, output, stream);
}

pa_status pa_forward_ex(pa_handle h, const void* query, const void* key, const void* value, void* key_cache,
                        void* value_cache, const int32_t* block_table, const int32_t* cum, const int32_t* past,
                        int batch, int token_count, const void* cos_cache, const void* sin_cache,
                        const pa_extra_inputs* extra, void* output, void* stream) {
  if (!h) return fail(nullptr, PA_INVALID_ARGUMENT, "handle must not be NULL");
  char msg[512];
  pa_status st = pa_check_step(&h->cfg, 1, query, key, value, key_cache, value_cache, block_table, cum, past, batch,
                               token_count, cos_cache, sin_cache, output, msg, sizeof(msg));
  if (st != PA_OK) return fail(h, st, "%s", msg);
  const pa_extra_inputs* x = extra ? extra : &kNoExtra;
  st = check_extra(h, x);
  if (st != PA_OK) return st;
  const bool quant = quantized(h->cfg.cache_dtype);
  const int bf16 = act_bf16(h->cfg) ? 1 : 0;  // head_sink and output are bfloat16
  const __half* sink = static_cast<const __half*>(x->head_sink);
  h->last_launches = 0;
  for (bool& r : h->stage_ran) r = false;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->last_stream = s;
  if (token_count == 0) return PA_OK;  // empty step: nothing to launch
  DeviceGuard g(h->device);
  const pa_config& c = h->cfg;
  const int D = c.head_size;
  const int pool_rows = c.num_blocks * c.block_size;
  const int box_rows = std::min(c.block_size, pa::kStageKeys);

  CUtensorMap tk, tv;
  const int eb = quant ? 1 : 2;
  if (!encode_pool_map(&tk, key_cache, D, c.kv_num_heads, pool_rows, box_rows, eb) ||
      (!h->latent && !encode_pool_map(&tv, value_cache, D, c.kv_num_heads, pool_rows, box_rows, eb)))
    return fail(h, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the K/V pool");

  // The prefill kernel launches unless the query-length bound already routes
  // every sequence to the decode kernel (always so for 8-bit caches; with
  // fp16 caches, up to chunk_rows_max rows while the chunking is on).  When
  // it does, it goes first and the decode kernel runs beside it on the SMs
  // the work list leaves it.
  const bool fp16_chunks = h->chunk_rows_max > 0 && h->opt_dec_rows == h->dec_rows;
  const int decode_rows_max = fp16_chunks ? std::max(h->opt_dec_rows, h->chunk_rows_max) : h->opt_dec_rows;
  const bool needs_prefill = !h->latent && !quant && (long long)h->max_q * h->G > decode_rows_max;
  if (needs_prefill && !h->prefill_ready)
    return fail(h, PA_NOT_SUPPORTED,
                "the query-length bound routes rows to the prefill kernel, which is not available on this device");
  const bool pre_launch = needs_prefill;

  // 1+2. prologue: device work list, rotary and the paged cache write
  {
    pa::WorklistParams p{};
    p.split_sms = (pre_launch && !h->opt_timing && h->opt_prefill_sms >= 0) ? h->num_sms : 0;  // timed kernels run alone
    p.force_pre_ctas = std::max(0, h->opt_prefill_sms);
    p.pre_grid = h->pre_grid;
    p.dec_grid = h->dec_grid;
    p.dec_ctas_per_sm = h->dec_ctas_per_sm;
    p.dec_bytes_per_key = (float)c.kv_num_heads * D * 4;
    p.pre_flops_per_pair = 4.f * D * c.num_heads;
    p.pre_rate_sm = kPrefillFlopsPerSmUs;
    p.dec_rate_sm = kDecodeBytesPerSmUs;
    p.hbm_rate = kHbmBytesPerUs;
    p.cum = cum;
    p.past = past;
    p.batch = batch;
    p.token_count = token_count;
    p.group = h->G;
    p.max_q = h->max_q;
    p.max_kv = h->max_kv;
    p.window = c.local_window_size;
    p.prune = h->opt_no_prune ? 0 : 1;
    p.dec_max_rows = h->opt_dec_rows;
    p.prefill_tile_tokens = h->prefill_tile_tokens;
    p.split_keys_fixed = h->opt_split_keys;
    p.target_pairs = target_pairs_for(h, batch);
    // A split of a tcgen05 latent unit leaves 128 heads x 256 channels of
    // fp32 partials to merge; below 2048 keys the merge costs more than the
    // balance gains (measured on the DeepSeek-V3-shaped step: automatic
    // ~1984 keys 109 us, 2048 97 us, no split 136 us).
    p.min_split_keys = h->mla_tc ? 2048 : pa::kStageKeys;
    // (a lowered decode row limit, an option that sends rows to the prefill
    // kernel, turns the fp16 chunking off)
    p.chunk_tokens = (h->chunk_rows_max == 0 || fp16_chunks) ? h->chunk_tokens : 0;
    p.chunk_rows_max = h->chunk_rows_max;
    p.cap_dec = h->cap_dec;
    p.cap_pre = h->cap_pre;
    p.cap_comb = h->cap_comb;
    p.cap_dseq = h->cap_dseq;
    p.cap_part = h->cap_part;
    p.seq = h->seq;
    p.dseq = h->dseq;
    p.dec_items = h->dec_items;
    p.pre_tiles = h->pre_tiles;
    p.comb_rows = h->comb_rows;
    p.counters = h->counters;
    p.err = h->err;
    pa::CacheWriteParams cp = cache_write_params(h->cfg, h->q_rot, h->err, query, key, value, key_cache,
                                                 value_cache, block_table, cum, past, batch, token_count, cos_cache,
                                                 sin_cache, x);
    StageTimer t(h, PA_STAGE_WORKLIST, s);
    cudaError_t e = pa::launch_prologue(p, cp, h->num_sms, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "prologue launch");
    h->last_launches++;
  }
  const __half* q_att = query_copied(c) ? h->q_rot : static_cast<const __half*>(query);
  if (h->latent) {
    // 3'. latent decode (tensor-core units of 128 heads and half the value
    // channels, or items of 32 heads), then the log-sum-exp combine of its
    // split partials
    const int qt = 1;
    const int tile_rows = std::min(c.block_size, 32);
    const int q_rows = h->mla_tc ? 128 : pa::kDecodeRows;
    // with rotary the query's rotated chunks come from the copy, the rest
    // from the query itself
    const bool q_split = q_att != static_cast<const __half*>(query);
    CUtensorMap tq, tqr, tl;
    if (!encode_map(&tq, query, D, c.num_heads, token_count, q_rows, qt) ||
        (q_split && !encode_map(&tqr, q_att, D, c.num_heads, token_count, q_rows, qt)))
      return fail(h, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the query");
    if (!q_split) tqr = tq;
    // 32-row pages: one 4-D box per tile holds all nine channel chunks
    // ([chunk][key][128 B], the ring slot's layout); smaller pages: one
    // 3-D box per (page, chunk)
    if (h->mla_tc && !(tile_rows == 32 ? encode_pool_map(&tl, key_cache, D, 1, pool_rows, tile_rows)
                                       : encode_map(&tl, key_cache, D, 1, pool_rows, 1, tile_rows)))
      return fail(h, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the latent pool");
    pa::MlaParams p{};
    p.out = static_cast<__half*>(output);
    p.block_table = block_table;
    p.seq = h->dseq;  // the decode table
    p.dec_items = h->dec_items;
    p.counters = h->counters;
    p.part_o = h->part_o;
    p.part_ml = h->part_ml;
    p.err = h->err;
    p.err_site = h->err + 1;
    p.H = c.num_heads;
    p.groups = h->groups;
    p.bs = c.block_size;
    p.MB = c.max_blocks_per_seq;
    p.NB = c.num_blocks;
    p.scale = h->scale;
    p.softcap = c.softcap;
    p.window = c.local_window_size;
    p.oob_row = pool_rows;
    p.log_box_rows = 31 - __builtin_clz((unsigned)box_rows);
    p.log_tile_rows = 31 - __builtin_clz((unsigned)tile_rows);
    p.bt_lines = (int)(((long long)batch * c.max_blocks_per_seq + 31) / 32);
    p.qr_lo = q_split ? c.rotary_offset / 64 : 0;
    p.qr_hi = q_split ? (c.rotary_offset + h->R + 63) / 64 : 0;
    {
      StageTimer t(h, PA_STAGE_DECODE, s);
      cudaError_t e = h->mla_tc ? pa::launch_mla_tc(tq, tqr, tl, p, h->dec_grid, s)
                                : pa::launch_mla_decode(tk, tq, tqr, p, h->dec_grid, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "latent decode launch");
      h->last_launches++;
    }
    pa::CombineParams mp{};
    mp.part_o = h->part_o;
    mp.part_ml = h->part_ml;
    mp.seq = h->dseq;  // the decode table
    mp.comb_rows = h->comb_rows;
    mp.counters = h->counters;
    mp.out = static_cast<__half*>(output);
    mp.H = c.num_heads;
    mp.Hk = h->groups;
    mp.G = pa::kDecodeRows;
    mp.D = h->dv;
    mp.err = h->err;
    mp.err_site = h->err + 1;
    mp.probe_flag = h->opt_wait_probe ? h->err + 2 : nullptr;
    StageTimer t(h, PA_STAGE_COMBINE, s);
    cudaError_t e = pa::launch_combine(mp, h->comb_grid, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "combine launch");
    h->last_launches++;
    return PA_OK;
  }
  // 3. varlen prefill on tensor memory (skipped when the query-length bound
  // already routes every sequence to the decode kernel)
  if (pre_launch) {
    CUtensorMap tq, tkp, tvp;
    const int prow = std::min(c.block_size, pa::prefill_keys_per_tile(D));
    if (!encode_map(&tq, q_att, D, c.num_heads, token_count, h->G, h->prefill_q_tokens) ||
        !encode_map(&tkp, key_cache, D, c.kv_num_heads, pool_rows, 1, prow) ||
        !encode_map(&tvp, value_cache, D, c.kv_num_heads, pool_rows, 1, prow))
      return fail(h, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the prefill maps");
    pa::PrefillParams p{};
    p.out = static_cast<__half*>(output);
    p.head_sink = sink;
    p.bf16 = bf16;
    p.block_table = block_table;
    p.seq = h->seq;
    p.pre_tiles = h->pre_tiles;
    p.counters = h->counters;
    p.err = h->err;
    p.err_site = h->err + 1;
    p.H = c.num_heads;
    p.Hk = c.kv_num_heads;
    p.G = h->G;
    p.bs = c.block_size;
    p.MB = c.max_blocks_per_seq;
    p.NB = c.num_blocks;
    p.tile_tokens = h->prefill_q_tokens;
    p.log_page_rows = 31 - __builtin_clz((unsigned)prow);
    p.scale = h->scale;
    p.softcap = c.softcap;
    p.window = c.local_window_size;
    p.oob_row = pool_rows;
    StageTimer t(h, PA_STAGE_PREFILL, s);
    cudaError_t e = pa::launch_prefill(D, tq, tkp, tvp, p, h->pre_grid, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "prefill launch");
    h->last_launches++;
  }
  // 4. split-KV decode (beside the prefill when both run)
  {
    const int qt = h->G <= pa::kDecodeRows ? pa::kDecodeRows / h->G : 1;
    CUtensorMap tq;
    if (!encode_map(&tq, q_att, D, c.num_heads, token_count, h->G, qt))
      return fail(h, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the query");
    pa::DecodeParams p{};
    p.q_tile_tokens = qt;
    p.log_box_rows = 31 - __builtin_clz((unsigned)box_rows);
    p.out = static_cast<__half*>(output);
    p.head_sink = sink;
    p.cache_type = c.cache_dtype;
    p.act_bf16 = (quant && bf16) ? 1 : 0;
    p.per_channel = c.v_quant_type == PA_QUANT_PER_CHANNEL;
    p.v_scale = x->v_scale;
    p.k_scale_tensor = (quant && c.k_quant_type == PA_QUANT_PER_TENSOR) ? x->k_scale : nullptr;
    p.block_table = block_table;
    p.seq = h->dseq;  // the decode table
    p.dec_items = h->dec_items;
    p.counters = h->counters;
    p.part_o = h->part_o;
    p.part_ml = h->part_ml;
    p.err = h->err;
    p.err_site = h->err + 1;
    p.H = c.num_heads;
    p.Hk = c.kv_num_heads;
    p.G = h->G;
    p.bs = c.block_size;
    p.MB = c.max_blocks_per_seq;
    p.NB = c.num_blocks;
    p.scale = h->scale;
    p.softcap = c.softcap;
    p.window = c.local_window_size;
    p.oob_row = pool_rows;
    p.wait_prologue = pre_launch ? 0 : 1;
    p.bt_lines = p.wait_prologue ? (int)(((long long)batch * c.max_blocks_per_seq + 31) / 32) : 0;
    StageTimer t(h, PA_STAGE_DECODE, s);
    cudaError_t e = pa::launch_decode(D, tk, tv, tq, p, h->dec_grid, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "decode launch");
    h->last_launches++;
  }
  // 5. log-sum-exp combine of split partials
  {
    pa::CombineParams p{};
    p.head_sink = sink;
    p.bf16 = bf16;
    p.part_o = h->part_o;
    p.part_ml = h->part_ml;
    p.seq = h->dseq;  // the decode table
    p.comb_rows = h->comb_rows;
    p.counters = h->counters;
    p.out = static_cast<__half*>(output);
    p.H = c.num_heads;
    p.Hk = c.kv_num_heads;
    p.G = h->G;
    p.D = D;
    p.err = h->err;
    p.err_site = h->err + 1;
    p.probe_flag = h->opt_wait_probe ? h->err + 2 : nullptr;
    StageTimer t(h, PA_STAGE_COMBINE, s);
    cudaError_t e = pa::launch_combine(p, h->comb_grid, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "combine launch");
    h->last_launches++;
  }
  return PA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pa_forward_no_alloc: the whole step without pa_create, for callers that
// cannot allocate device memory.  All scratch (work lists, split-KV partials,
// the rotated-query buffer, the error word) is carved from one file-scope
// device array below, so the call allocates nothing.
namespace {

// Size of the static scratch; every GPU that loads this library holds it.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
__device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
struct NoAllocDevice {
  bool ready = false;                // set-up done (a failed set-up is retried on the next call)
  unsigned char* scratch = nullptr;  // device address of g_no_alloc_scratch
  int num_sms = 0;
  int dec_ctas[3][2] = {{1, 1}, {1, 1}, {1, 1}};  // decode CTAs per SM: head_size 64, 128, 256 x G <= 8, G <= 16
  bool prefill_ok = false;
};
NoAllocDevice g_no_alloc_dev[kMaxDevices];
std::mutex g_no_alloc_mu;

int head_index(int D) { return D == 64 ? 0 : (D == 128 ? 1 : 2); }

// Set-up on the current device, once it succeeds: the scratch array's
// device address (the host-side symbol is not a device pointer), the SM
// count and the kernels' shared-memory attributes.  Returns cudaSuccess or
// the failing call's error (*what names it); a failure leaves the device
// not ready, so a later call tries again.
cudaError_t no_alloc_setup(int dev, NoAllocDevice** out, const char** what) {
  std::lock_guard<std::mutex> lock(g_no_alloc_mu);
  NoAllocDevice* d = &g_no_alloc_dev[dev];
  *out = d;
  if (d->ready) return cudaSuccess;
  NoAllocDevice n;
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
  if (e != cudaSuccess) { *what = "cudaGetSymbolAddress(scratch)"; return e; }
  n.scratch = static_cast<unsigned char*>(ptr);
  e = cudaDeviceGetAttribute(&n.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) { *what = "cudaDeviceGetAttribute"; return e; }
  size_t smem = 0;
  for (int D : {64, 128, 256}) {
    for (int t = 0; t < 2 && e == cudaSuccess; ++t)
      e = pa::decode_configure(D, PA_CACHE_FP16, t ? 16 : 8, &n.dec_ctas[head_index(D)][t], &smem);
    if (e != cudaSuccess) { *what = "decode kernel attributes"; return e; }
  }
  n.prefill_ok = pa::prefill_configure(64, &smem) == cudaSuccess &&
                 pa::prefill_configure(128, &smem) == cudaSuccess &&
                 pa::prefill_configure(256, &smem) == cudaSuccess;
  cudaGetLastError();
  if (!encode_fn()) { *what = "cuTensorMapEncodeTiled lookup"; return cudaErrorNotSupported; }
  n.ready = true;
  *d = n;
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_forward_no_alloc(const pa_config* cfg, const void* query, const void* key, const void* value,
                                         void* key_cache, void* value_cache, const int32_t* block_table,
                                         const int32_t* cum, const int32_t* past, int batch, int token_count,
                                         const void* cos_cache, const void* sin_cache, void* output,
                                         int32_t* device_error, void* stream) {
  char msg[512];
  pa_status st = pa_check_step(cfg, 1, query, key, value, key_cache, value_cache, block_table, cum, past, batch,
                               token_count, cos_cache, sin_cache, output, msg, sizeof(msg));
  if (st != PA_OK) return fail(nullptr, st, "%s", msg);
  if (cfg->cache_dtype != PA_CACHE_FP16 || cfg->act_dtype != PA_ACT_DEFAULT || cfg->packed_qkv || cfg->qk_norm ||
      cfg->kv_cache_layout != PA_LAYOUT_SEPARATE)
    return fail(nullptr, PA_NOT_SUPPORTED,
                "pa_forward_no_alloc runs separate fp16 K/V caches without packed QKV or QK-Norm (no latent "
                "layout, no 8-bit or bfloat16 cache); use pa_forward_ex");
  if (device_error && reinterpret_cast<uintptr_t>(device_error) % 4)
    return fail(nullptr, PA_INVALID_ARGUMENT, "device_error must be 4-byte aligned");
  if (token_count == 0) return PA_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(nullptr, PA_NOT_SUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  NoAllocDevice* nd = nullptr;
  const char* what = "";
  e = no_alloc_setup(dev, &nd, &what);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, what);

  const pa_config& c = *cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int D = c.head_size, H = c.num_heads, Hk = c.kv_num_heads;
  const int G = H / Hk;
  const float scale = c.scale > 0.f ? c.scale : 1.f / std::sqrt((float)D);
  const int kv_cap = c.max_blocks_per_seq * c.block_size;
  const int max_q = c.max_query_len_bound > 0 ? std::min(c.max_query_len_bound, c.max_tokens) : c.max_tokens;
  const int max_kv = c.max_kv_len_bound > 0 ? std::min(c.max_kv_len_bound, kv_cap) : kv_cap;
  // Rows go to the decode kernel iff q_len * G <= 16; the prefill kernel
  // runs only when the query-length bound lets some sequence have more.
  const int dec_max_rows = pa::decode_item_rows(G);
  const bool pre_launch = (long long)max_q * G > dec_max_rows;
  if (pre_launch && !nd->prefill_ok)
    return fail(nullptr, PA_NOT_SUPPORTED,
                "the query-length bound routes rows to the prefill kernel, which is not available on this device");
  const int dec_grid = nd->num_sms * nd->dec_ctas[head_index(D)][G <= 8 ? 0 : 1];
  const int target_pairs = std::max(1, (pa::kDecodeItemsPerCta * dec_grid + Hk - 1) / Hk);
  const int cap_dseq = c.max_batch;  // one decode entry per sequence (no chunks: fp16 caches have the prefill kernel)
  const int cap_dec = target_pairs + cap_dseq;
  const int cap_part = 2 * target_pairs;
  const int tile_tokens = pa::prefill_unit_tokens(D, G);
  const int q_tokens = std::max(1, pa::kPrefillRows / G);
  const int cap_pre = (c.max_tokens + tile_tokens - 1) / tile_tokens + c.max_batch;
  const int cap_comb = c.max_tokens;

  // Scratch layout (256-byte aligned pieces), checked against the maximum.
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off = 0;
  const size_t o_err = off; off = up(off + 64);  // error bits, wait site
  const size_t o_cnt = off; off = up(off + sizeof(pa::Counters));
  const size_t o_seq = off; off = up(off + sizeof(pa::SeqInfo) * c.max_batch);
  const size_t o_dsq = off; off = up(off + sizeof(pa::SeqInfo) * cap_dseq);
  const size_t o_dec = off; off = up(off + sizeof(int2) * cap_dec);
  const size_t o_pre = off; off = up(off + sizeof(int2) * cap_pre);
  const size_t o_cmb = off; off = up(off + sizeof(int2) * cap_comb);
  const size_t o_pml = off; off = up(off + sizeof(float2) * (size_t)cap_part * Hk * pa::kDecodeRows);
  const size_t o_po = off; off = up(off + sizeof(float) * (size_t)cap_part * Hk * pa::kDecodeRows * D);
  const size_t o_qr = off;
  if (c.do_rotary) off = up(off + 2 * (size_t)c.max_tokens * H * D);
  if (off > kNoAllocScratchBytes)
    return fail(nullptr, PA_INVALID_ARGUMENT,
                "these capacities need %zu bytes of scratch; the static scratch holds %zu bytes "
                "(lower max_batch / max_tokens or use pa_create)",
                off, kNoAllocScratchBytes);
  unsigned char* w = nd->scratch;
  int* err_words = reinterpret_cast<int*>(w + o_err);
  int* err = device_error ? device_error : err_words;
  int* err_site = err_words + 1;
  pa::Counters* counters = reinterpret_cast<pa::Counters*>(w + o_cnt);
  pa::SeqInfo* seq = reinterpret_cast<pa::SeqInfo*>(w + o_seq);
  pa::SeqInfo* dseq = reinterpret_cast<pa::SeqInfo*>(w + o_dsq);
  int2* dec_items = reinterpret_cast<int2*>(w + o_dec);
  int2* pre_tiles = reinterpret_cast<int2*>(w + o_pre);
  int2* comb_rows = reinterpret_cast<int2*>(w + o_cmb);
  float2* part_ml = reinterpret_cast<float2*>(w + o_pml);
  float* part_o = reinterpret_cast<float*>(w + o_po);
  __half* q_ws = c.do_rotary ? reinterpret_cast<__half*>(w + o_qr) : nullptr;
  // the shared error bits (when the caller gives no word of its own) and the
  // wait-site word start clean
  e = cudaMemsetAsync(err_words, 0, 2 * sizeof(int), s);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaMemsetAsync(error words)");

  const int pool_rows = c.num_blocks * c.block_size;
  const int box_rows = std::min(c.block_size, pa::kStageKeys);
  CUtensorMap tk, tv;
  if (!encode_pool_map(&tk, key_cache, D, Hk, pool_rows, box_rows) ||
      !encode_pool_map(&tv, value_cache, D, Hk, pool_rows, box_rows))
    return fail(nullptr, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the K/V pool");

  pa::WorklistParams wp{};
  wp.cum = cum;
  wp.past = past;
  wp.batch = batch;
  wp.token_count = token_count;
  wp.group = G;
  wp.max_q = max_q;
  wp.max_kv = max_kv;
  wp.window = c.local_window_size;
  wp.prune = 1;
  wp.dec_max_rows = dec_max_rows;
  wp.prefill_tile_tokens = tile_tokens;
  wp.split_keys_fixed = 0;
  wp.target_pairs = target_pairs;
  wp.min_split_keys = pa::kStageKeys;
  wp.chunk_tokens = 0;
  wp.chunk_rows_max = 0;
  wp.cap_dec = cap_dec;
  wp.cap_pre = cap_pre;
  wp.cap_comb = cap_comb;
  wp.cap_dseq = cap_dseq;
  wp.cap_part = cap_part;
  wp.seq = seq;
  wp.dseq = dseq;
  wp.dec_items = dec_items;
  wp.pre_tiles = pre_tiles;
  wp.comb_rows = comb_rows;
  // no SM split here: the decode kernel follows the prologue, the prefill
  // kernel the decode kernel, each with every CTA working
  const int pre_grid_na = std::max(1, std::min(nd->num_sms, cap_pre * Hk));
  wp.split_sms = 0;
  wp.pre_grid = pre_grid_na;
  wp.dec_grid = dec_grid;
  wp.dec_ctas_per_sm = std::max(1, dec_grid / nd->num_sms);
  wp.counters = counters;
  wp.err = err;
  const pa::CacheWriteParams cp =
      cache_write_params(c, q_ws, err, query, key, value, key_cache, value_cache, block_table, cum, past, batch,
                         token_count, cos_cache, sin_cache, &kNoExtra);
  e = pa::launch_prologue(wp, cp, nd->num_sms, s);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "prologue launch");

  const __half* q_att = c.do_rotary ? q_ws : static_cast<const __half*>(query);
  const int qt = G <= pa::kDecodeRows ? pa::kDecodeRows / G : 1;
  CUtensorMap tq;
  if (!encode_map(&tq, q_att, D, H, token_count, G, qt))
    return fail(nullptr, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the query");
  pa::DecodeParams dp{};
  dp.q_tile_tokens = qt;
  dp.log_box_rows = 31 - __builtin_clz((unsigned)box_rows);
  dp.out = static_cast<__half*>(output);
  dp.block_table = block_table;
  dp.seq = dseq;
  dp.dec_items = dec_items;
  dp.counters = counters;
  dp.part_o = part_o;
  dp.part_ml = part_ml;
  dp.err = err;
  dp.err_site = err_site;
  dp.H = H;
  dp.Hk = Hk;
  dp.G = G;
  dp.bs = c.block_size;
  dp.MB = c.max_blocks_per_seq;
  dp.NB = c.num_blocks;
  dp.scale = scale;
  dp.softcap = c.softcap;
  dp.window = c.local_window_size;
  dp.oob_row = pool_rows;
  dp.wait_prologue = 1;
  e = pa::launch_decode(D, tk, tv, tq, dp, dec_grid, s);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "decode launch");

  if (pre_launch) {
    CUtensorMap tqp, tkp, tvp;
    const int prow = std::min(c.block_size, pa::prefill_keys_per_tile(D));
    if (!encode_map(&tqp, q_att, D, H, token_count, G, q_tokens) ||
        !encode_map(&tkp, key_cache, D, Hk, pool_rows, 1, prow) ||
        !encode_map(&tvp, value_cache, D, Hk, pool_rows, 1, prow))
      return fail(nullptr, PA_CUDA_ERROR, "cuTensorMapEncodeTiled failed for the prefill maps");
    pa::PrefillParams pp{};
    pp.out = static_cast<__half*>(output);
    pp.block_table = block_table;
    pp.seq = seq;
    pp.pre_tiles = pre_tiles;
    pp.counters = counters;
    pp.err = err;
    pp.err_site = err_site;
    pp.H = H;
    pp.Hk = Hk;
    pp.G = G;
    pp.bs = c.block_size;
    pp.MB = c.max_blocks_per_seq;
    pp.NB = c.num_blocks;
    pp.tile_tokens = q_tokens;
    pp.log_page_rows = 31 - __builtin_clz((unsigned)prow);
    pp.scale = scale;
    pp.softcap = c.softcap;
    pp.window = c.local_window_size;
    pp.oob_row = pool_rows;
    e = pa::launch_prefill(D, tqp, tkp, tvp, pp, pre_grid_na, s);
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "prefill launch");
  }

  // The combine kernel waits for its predecessor (the prefill kernel, which
  // waited for the decode kernel, or the decode kernel itself).
  pa::CombineParams mp{};
  mp.part_o = part_o;
  mp.part_ml = part_ml;
  mp.seq = dseq;
  mp.comb_rows = comb_rows;
  mp.counters = counters;
  mp.out = static_cast<__half*>(output);
  mp.H = H;
  mp.Hk = Hk;
  mp.G = G;
  mp.D = D;
  mp.err = err;
  mp.err_site = err_site;
  e = pa::launch_combine(mp, std::max(1, std::min(nd->num_sms * 4, (cap_comb * H + 7) / 8)), s);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "combine launch");
  return PA_OK;
}
