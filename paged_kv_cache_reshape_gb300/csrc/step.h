// Internal structures shared by the host planner and the step kernels.
// Everything per-step that depends on device-resident lengths lives in the
// work list written by the work-list kernel; the host only sizes launches
// from static capacities ("PagedAttention - CUDA Design Document",
// section 4.7, replay-invariance rule).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace pa {

constexpr int kStageKeys = 64;      // keys per decode pipeline stage
constexpr int kDecodeRows = 16;     // most query rows (token x group head) per decode item
// Query rows a decode item serves for a GQA group of G heads: the decode
// kernel's row tiles hold 8 rows, and it runs one tile when G <= 8, two
// otherwise (G <= 16); larger groups have no decode item (0).
__host__ __device__ inline int decode_item_rows(int G) { return G <= 8 ? 8 : (G <= kDecodeRows ? kDecodeRows : 0); }
constexpr int kDecodeWarps = 4;     // consumer warps of the decode kernel
// Decode work items per decode CTA the automatic split size aims for: 2
// measured best on the Llama-3-8B- and Llama-70B-shaped decode steps (fewer
// split sequences to merge, the dynamic queue still balances the tail).
constexpr int kDecodeItemsPerCta = 2;
constexpr int kPrefillRows = 128;   // query rows per prefill tile (UMMA M)
constexpr int kPrefillKeys = 128;   // keys per prefill KV tile (UMMA N of S)

// How a sequence's rows are served: one decode entry, decode entries of
// chunk_tokens tokens each, or the prefill kernel.
enum Route { kRouteNone = 0, kRouteDecode = 1, kRoutePrefill = 2, kRouteChunked = 3 };

// Facts derived on the device each step, in two tables.  The sequence
// table has one entry per sequence (its lengths and prefill tiles).  The
// decode table has one entry per unit of decode work: a sequence whose
// q_len * G query rows fit one decode item, or a chunk of chunk_tokens
// consecutive new tokens of a longer sequence that has no prefill kernel
// (8-bit caches, the latent layout), each chunk attending causally from
// its own first token's position.  Decode items and combine rows refer to
// the decode table.
// Decode items are listed full splits first (every split of every entry
// but its last), then the last, usually shorter, split of each entry,
// longest first, so the dynamic item queue hands out the long items first.
struct SeqInfo {
  int q_len;      // new tokens of the sequence or chunk (0 when the sequence is skipped)
  int kv_len;     // position of its last new token + 1
  int lo;         // first key position walked (64-aligned window start or 0)
  int t0;         // first packed row
  int dec_first;  // item index of split 0 (splits 0..dec_count-2 are consecutive)
  int dec_count;  // decode splits
  int dec_last;   // item index of split dec_count-1
  int pre_first;  // first prefill tile of this sequence (sequence table)
  int pre_count;  // prefill query tiles (sequence table; 0 unless routed to prefill)
  int comb_first; // first combine row of the entry (decode table)
  int b;          // the sequence: its block_table row (decode table)
  int part_first; // split partials of a split entry: slots part_first + split (decode table; -1 unsplit)
};

__host__ __device__ inline int dec_item_of_split(const SeqInfo& s, int split) {
  return split == s.dec_count - 1 ? s.dec_last : s.dec_first + split;
}

struct Counters {
  int n_dec;       // decode items (b, split) pairs
  int n_pre;       // prefill tiles (b, query tile)
  int n_comb;      // packed rows whose splits need the log-sum-exp merge
  int split_keys;  // keys per decode split this step
  int dec_next;    // decode work queue head (reset to 0 by the work-list kernel)
  int pre_next;    // prefill work queue head (reset to 0 by the work-list kernel)
  int pre_ctas;    // prefill CTAs that take work this step; the others exit at once
  int dec_ctas;    // decode CTAs that take work this step
  int pad[4];
};

struct WorklistParams {
  const int* cum;
  const int* past;
  int batch, token_count;
  int group;               // G = H / Hk
  int max_q, max_kv;       // trusted bounds (already clamped to static limits)
  int window;              // -1 or >= 1
  int prune;               // 1: start the walk at the window (block pruning)
  int dec_max_rows;        // decode route iff q_len * G <= this
  int prefill_tile_tokens; // tokens per prefill tile
  int split_keys_fixed;    // > 0 forces keys per split
  int target_pairs;        // desired number of decode (b, split) items
  int min_split_keys;      // smallest automatic split (a multiple of 64)
  int chunk_tokens;        // > 0: a sequence with q_len * G > dec_max_rows goes to the decode kernel
                           // in chunks of this many tokens (chunk_tokens * G <= dec_max_rows);
                           // 0: it goes to the prefill kernel
  int chunk_rows_max;      // > 0: only sequences of at most this many rows (q_len * G) are chunked,
                           // longer ones go to the prefill kernel; 0: every one (no prefill kernel)
  int cap_dec, cap_pre, cap_comb, cap_dseq;
  int cap_part;            // split-partial slots (one per split of a split decode entry)
  // SM split between the prefill and decode kernels.  With split_sms > 0
  // the prefill kernel is launched first, one CTA per SM, and the work list
  // decides how many of its CTAs keep working; the others exit, and the
  // decode kernel, launched next, runs on the SMs they free, concurrently.
  int split_sms;             // SMs to share (0: no split, every CTA works)
  int force_pre_ctas;        // > 0: the prefill CTAs kept, instead of the cost model's choice
  int pre_grid, dec_grid;    // launched CTAs of the two kernels
  int dec_ctas_per_sm;
  float dec_bytes_per_key;   // Hk * D * 4 (K and V, once per kv head)
  float pre_flops_per_pair;  // 4 * D * H per (query token, admitted key)
  float pre_rate_sm;         // prefill FLOP per us per SM
  float dec_rate_sm;         // decode bytes per us per SM
  float hbm_rate;            // bytes per us
  SeqInfo* seq;      // sequence table [batch]
  SeqInfo* dseq;     // decode table [cap_dseq]
  int2* dec_items;   // (decode entry, split)
  int2* pre_tiles;   // (b, tile)
  int2* comb_rows;   // (t, decode entry)
  Counters* counters;
  int* err;
};

// Cache element types (pa.h PA_CACHE_*).  kCacheBF16: bfloat16 activations
// and cache; every 16-bit tensor of the step (declared __half below, bits
// only) then holds bfloat16.
enum CacheType { kCacheF16 = 0, kCacheI8 = 1, kCacheE4M3 = 2, kCacheBF16 = 3 };

struct CacheWriteParams {
  const __half* key;    // [T, Hk*D]
  const __half* value;  // [T, Hk*D]
  const __half* query;  // [T, H*D] or null (cache write only)
  __half* q_rot;        // [T, H*D] query for attention (rotated and/or times k_scale)
  void* key_cache;      // fp16 or 8-bit codes (cache_type)
  void* value_cache;
  int cache_type;       // CacheType
  int act_bf16;         // 8-bit caches: 1 = bfloat16 activations (query, key, value, tables,
                        // norm weights); the query copy is fp16 either way
  int per_channel;      // scales [Hk*D] (1) or [1] (0)
  const float* k_scale; // 8-bit caches: quantization / dequantization scales
  const float* v_scale;
  const int* slot_mapping;  // [T] explicit write slots (-1 = no write) or null
  int packed;               // query rows hold [Q | K | V] (key / value unused)
  int q_stride;             // elements per query input row: H*D, or (H+2Hk)*D when packed
  int qk_norm;              // QK-Norm of Q and K before rotary
  float qk_eps;
  const __half* q_norm_w;   // [D]
  const __half* k_norm_w;   // [D]
  const int* block_table;
  const int* cum;
  const int* past;
  const __half* cos_cache;  // [P, R/2]
  const __half* sin_cache;
  int batch, token_count;
  int H, Hk, D, bs, NB, MB;
  int rotary, interleaved, rot_dim, rot_positions;
  int rot_offset;        // first rotated channel (latent rows rotate their last rot_dim channels)
  int q_keep_lo, q_keep_hi;  // channels of the query copy written besides the rotated ones (latent:
                             // the 64-channel chunks holding them; the kernels read the rest from
                             // the query itself)
  int q_scale;           // 1: the query copy is multiplied by k_scale (8-bit caches)
  int parts;             // warps per token: K/V parts + query parts when Q is transformed
  int kv_parts;          // warps per token for the K and V rows: 1 (both rows), or K and V warps per
                         // kv_heads_per_part heads (8-bit caches)
  int kv_heads_per_part;
  int q_heads_per_part;  // query heads per query part
  int* err;
};

struct DecodeParams {
  __half* out;      // [T, H*D]
  const __half* head_sink;  // [H] or null
  const float* v_scale;     // 8-bit caches: [1] or [Hk*D]
  const float* k_scale_tensor;  // 8-bit caches with one K scale: [1], folded into the score scale
                                // (per-channel K scales are folded into the query copy instead)
  int per_channel;
  int cache_type;
  int act_bf16;             // 8-bit caches: 1 = head_sink and out are bfloat16 (the query
                            // copy the kernel reads is fp16 either way)
  const int* block_table;
  const SeqInfo* seq;       // the decode table
  const int2* dec_items;
  Counters* counters;  // n_dec, split_keys, and the item queue head
  float* part_o;    // [items*Hk*16*D]
  float2* part_ml;  // [items*Hk*16] (max in log2 units, sum)
  int* err;
  int* err_site;    // first wait that gave up (wait site id), or null
  int H, Hk, G, bs, MB, NB;
  float scale;       // softmax scale
  float softcap;     // 0 = off
  int window;        // -1 or >= 1
  int oob_row;       // a TMA row coordinate past the pool (zero fill)
  int q_tile_tokens; // tokens per query TMA box (16 / G)
  int log_box_rows;  // log2(min(block_size, 64)): pool rows per TMA box
  int bt_lines;      // 128-byte lines of the block table (batch rows) to pull into L2 first; 0 = none
  int wait_prologue; // 1: the launch before is the prologue (griddepcontrol.wait
                     // on it); 0: it is the prefill kernel, which has waited for
                     // the prologue before letting this kernel start: this
                     // kernel runs beside it and waits for it (griddepcontrol.wait,
                     // CTA 0) only before exiting, so that this grid completes
                     // after the prefill grid and the combine kernel, which
                     // waits for this grid, ends the step after both
};

struct CombineParams {
  const __half* head_sink;  // [H] or null
  int bf16;                 // 1: head_sink and out are bfloat16
  const float* part_o;
  const float2* part_ml;
  const SeqInfo* seq;       // the decode table
  const int2* comb_rows;
  const Counters* counters;
  __half* out;
  int H, Hk, G, D;
  int* err;
  int* err_site;
  const int* probe_flag;  // non-null: CTA 0 waits (2 ms at most) for *probe_flag != 0, which
                          // nothing sets, and records the timeout (exercises the error path)
};

struct PrefillParams {
  __half* out;
  const __half* head_sink;  // [H] or null
  int bf16;                 // 1: query, pools, head_sink and out are bfloat16
  const int* block_table;
  const SeqInfo* seq;       // the sequence table
  const int2* pre_tiles;
  Counters* counters;  // n_pre and the tile queue head
  int* err;
  int* err_site;
  int H, Hk, G, bs, MB, NB;
  int tile_tokens;  // tokens per 128-row query tile (rows = tile_tokens * G <= 128)
  int log_page_rows;  // log2(min(block_size, keys per KV tile)): pool rows per TMA box
  float scale;
  float softcap;
  int window;
  int oob_row;
};

// Work-list groups of one latent decode item: each item covers 32 query
// heads (two of the 16-head groups its partials are laid out by).
__host__ __device__ inline int mla_item_groups(int groups16) { return (groups16 + 1) / 2; }

struct MlaParams {
  __half* out;           // [T, H, 512]
  const int* block_table;
  const SeqInfo* seq;    // the decode table
  const int2* dec_items;
  Counters* counters;
  float* part_o;         // [items * groups * 16 * 512]
  float2* part_ml;       // [items * groups * 16]
  int* err;
  int* err_site;
  int H, groups;         // query heads, groups of 16 heads (32 heads per work item)
  int bs, MB, NB;
  float scale, softcap;
  int window;
  int oob_row;
  int log_box_rows;      // log2(min(block_size, 64))
  int log_tile_rows;     // log2(min(block_size, 32)): pool rows per box of the tensor-core kernel
  int bt_lines;          // 128-byte lines of the block table (batch rows) to pull into L2 first
  int qr_lo, qr_hi;      // query chunks [qr_lo, qr_hi) read from the rotated copy (map tm_qr),
                         // the others from the query (map tm_q)
};

// Launch with the programmatic stream-serialization attribute, so the
// kernel's CTAs may become resident while the previous kernel on the stream
// finishes; the kernel calls griddepcontrol.wait before touching its
// predecessor's results.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launchers (defined in the .cu files).
cudaError_t launch_cache_write(const CacheWriteParams& p, cudaStream_t s);
// The prologue spreads its (token, part) warps over up to num_sms - 1 blocks
// (a block holds a whole SM: its builder CTA needs every register).
cudaError_t launch_prologue(const WorklistParams& wp, const CacheWriteParams& cp, int num_sms, cudaStream_t s);
// CTAs per SM and shared memory of the decode kernel a GQA group of `group`
// heads runs (its row tiles follow the group).
cudaError_t decode_configure(int head_size, int cache_type, int group, int* ctas_per_sm, size_t* smem);
cudaError_t launch_decode(int head_size, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tq, const DecodeParams& p, int grid, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, int grid, cudaStream_t s);
cudaError_t mla_configure(size_t* smem);
// Latent decode on tcgen05 (query heads a multiple of 128): units of 128 heads
// and half of the value channels; Q map boxes {64, 128 heads, 1 token}, pool
// map boxes {64, 1, min(block_size, 32) rows}.
cudaError_t mla_tc_configure(size_t* smem);
cudaError_t launch_mla_tc(const CUtensorMap& tq, const CUtensorMap& tqr, const CUtensorMap& tl, const MlaParams& p,
                          int grid,
                          cudaStream_t s);
cudaError_t launch_mla_decode(const CUtensorMap& tl, const CUtensorMap& tq, const CUtensorMap& tqr, const MlaParams& p,
                              int grid,
                              cudaStream_t s);
cudaError_t prefill_configure(int head_size, size_t* smem);
int prefill_keys_per_tile(int head_size);
int prefill_unit_tokens(int head_size, int group);  // tokens per prefill work unit
cudaError_t prefill_single_configure(int head_size, size_t* smem);
int prefill_single_keys_per_tile(int head_size);
cudaError_t launch_prefill_single(int head_size, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const PrefillParams& p, int grid, cudaStream_t s);
cudaError_t prefill_pair_configure(int head_size);
cudaError_t launch_prefill_pair(int head_size, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const PrefillParams& p, int grid, cudaStream_t s);
cudaError_t launch_prefill(int head_size, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const PrefillParams& p, int grid, cudaStream_t s);

}  // namespace pa
