// Split-KV paged decode: one work item = (sequence b, split s, kv head k).
//
// The item serves every query row of kv head k's group for all of b's new
// tokens at once (rows r = j*G + g, at most 16), so each K/V element of the
// split is read from HBM exactly once per kv head.  What it computes is the
// paged decode of "PagedAttention - CUDA Design Document", section 8
// implementation note P5: per-row causal bound past + j + 1, sliding window
// [kv_len - W, kv_len), softcap * tanh(x * scale / softcap), -1 block
// entries masked (section 9.3.1), splits merged by log-sum-exp; empty splits
// publish (max = -inf, sum = 0).  The split walk starts at the window
// (section 9.2 block pruning, section 9.3.4 item 2: splits laid over the
// clamped range).
//
// Design for sm_103a (not the pages' CUDA-core kernel):
//  * persistent grid sized from the SM count; a producer warp takes items
//    from a device queue (full splits first) and posts each 64-key stage's
//    description in a shared-memory tag next to the data;
//  * the producer streams K and V through a ring of shared-memory stages
//    straight from the NHD pool with one 4-D TMA box per page and tensor:
//    the pool is viewed as {64 channels, pool rows, D/64 chunks, heads} so
//    a box {64, rows, D/64, 1} lands one head's page as [chunk][row][128 B]
//    with the 128-byte swizzle; the boxes of a stage are issued by several
//    lanes at once; the item's 16 query rows come with one 3-D box
//    {64, G, 16/G} per chunk into a double-buffered Q tile; block ids are
//    fetched 32 rows at a time by the whole warp one window ahead; unmapped
//    pages are fetched from a row past the pool so TMA zero-fills them
//    without reading memory;
//  * four consumer warps each own 16 keys of every stage and run the two
//    contractions on tensor cores (m16n8k16 HMMA, fp16 in, fp32 accumulate):
//    S = Q K^T and O += P V, with an fp32 online softmax whose row max is
//    reduced with warp shuffles;
//  * at the end of an item the four warps' (m, l, O) are merged through the
//    last stage's buffer; a single-split sequence writes fp16 output
//    directly, otherwise fp32 partials go to the combine kernel;
//  * 8-bit caches (int8 / e4m3fn codes, section 8.5 phase 3) are read at
//    their stored width: the pool view has 128 channels per 128-byte chunk;
//    K fragments come from ldmatrix on the code bytes (each lane gets four
//    consecutive channels of one key), which fixes the order in which the
//    16 channels of an m16n8k16 step are contracted, and the Q fragments
//    (with per-channel scales already times k_scale, written by the
//    prologue; one per-tensor K scale multiplies the score scale instead)
//    are loaded in that same order; V fragments come from a transposed ldmatrix (two keys x two
//    channels per lane), split into an even-channel and an odd-channel MMA;
//    codes become fp16 pairs with one byte permute and one conversion; the
//    V scale multiplies the merged output;
//  * head_sink (section 6.1) adds exp(s_h - M) to the final denominator of a
//    single-split row (split rows get it in the combine kernel);
//  * bfloat16 activations with a bfloat16 cache (section 8.2) run the fp16
//    layout and schedule with bfloat16 MMAs: Q and K as stored, P rounded
//    to bfloat16 for O += P V, bfloat16 output and sink.
#include <algorithm>

#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kThreads = (kDecodeWarps + 1) * 32;  // 4 consumer warps + 1 producer warp
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.f;  // log2 of the largest P value tolerated before rescaling

template <int D, int CT, int NT>
struct DecodeCfg {
  static constexpr bool k16 = CT == kCacheF16 || CT == kCacheBF16;  // 16-bit cache elements
  static constexpr int kEb = k16 ? 2 : 1;                   // bytes per cache element
  static constexpr int kChunks = D * kEb / 128;             // 128-byte chunks per K/V row
  static constexpr int kQChunks = D / 64;                   // 128-byte chunks per fp16 query row
  static constexpr int kTileBytes = kStageKeys * D * kEb;   // K (or V) bytes per stage
  static constexpr int kStageBytes = 2 * kTileBytes;        // K + V
  static constexpr int kStages = k16 ? ((D == 256) ? 3 : (D == 128 ? 3 : 6)) : 4;
  static constexpr int kQBytes = kQChunks * 2048;           // 16 rows x 128 B per chunk
  // End-of-item merge: the four warps' 8 * NT x D fp32 partial outputs, in
  // the last stage's buffer when it is large enough, else in a region of
  // their own.
  static constexpr int kMergeBytes = kDecodeWarps * 8 * NT * D * 4;
  // 8-bit pools with one row tile fit three CTAs on an SM (the merge reuses
  // a stage buffer and the registers stay within a third of the file).
  static constexpr int kCtasPerSm = (D == 256) ? 1 : ((!k16 && NT == 1) ? 3 : 2);
  static constexpr int kOwnMerge = kMergeBytes > kStageBytes ? kMergeBytes : 0;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kOwnMerge + 2 * kQBytes + 4 * 16 * 8 +
                                    kStages * 64 + (2 * kStages + 4) * 8;
};

struct StageTag {
  int u;       // item * Hk + k; -1 = no more work
  int key0;    // first key position of the stage
  int end;     // split end (exclusive)
  int flags;   // bits 0..3 zero-filled boxes; bit 8 first stage of the item; bit 9 last stage
  int R;       // valid query rows (q_len * G)
  int past;    // past length of the sequence
  int t0;      // first packed row of the sequence
  int k;       // kv head
  int kv_len;  // past + q_len
  int nsplit;  // splits of the sequence
  int qi;      // Q buffer
  int lo_min;  // smallest admitted position of any row (0 without a window)
  int part;    // split-partial slot of this split (a split entry), -1 for an unsplit one
  int pad[3];
};
constexpr int kFirst = 1 << 8, kLast = 1 << 9;

// Byte offset of 16-byte column `col16` of row `row` inside a 128B-swizzled
// [rows][128 B] tile whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int row, int col16) {
  return (uint32_t)(row * 128 + ((col16 ^ (row & 7)) << 4));
}

// Stage tile layout [box][chunk][row][128 B] (box = 2^log_r pool rows):
// byte offset of (stage key kk, channel chunk, 16-byte column col16).
template <int kChunks>
__device__ __forceinline__ uint32_t tile_off(int kk, int chunk, int col16, int log_r) {
  const int r = kk & ((1 << log_r) - 1), bx = kk >> log_r;
  return ((uint32_t)(bx * kChunks + chunk) << (log_r + 7)) + swz(r, col16);
}

// Two 8-bit codes of w (bytes LO and HI; LO goes to the low half) as an
// fp16 pair.  int8: the code byte plus 128 becomes the low mantissa byte of
// 1024 + code + 128, exact in fp16, and 1152 is subtracted.
template <int CT, int LO, int HI>
__device__ __forceinline__ uint32_t deq2(uint32_t w) {
  if constexpr (CT == kCacheI8) {
    const uint32_t x = __byte_perm(w, 0x64646464u, 0x4040u | LO | (HI << 8)) ^ 0x00800080u;
    const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&x), __half2(__half(1152.f), __half(1152.f)));
    return *reinterpret_cast<const uint32_t*>(&h);
  } else if constexpr (LO == 0 && HI == 1) {  // the low half as it is
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(w));
    return r;
  } else if constexpr (LO == 2 && HI == 3) {  // the high half as it is
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(r) : "r"(w));
    return r;
  } else {
    const uint32_t x = __byte_perm(w, 0u, LO | (HI << 4));
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(x));
    return r;
  }
}

// Value channel of element e of O^T accumulator kk (the consumer's fragment
// coordinates): fp16 pools, 16 channels per accumulator (fg and fg + 8);
// 8-bit pools, the even (kk even) or odd channels of 32 (2fg + parity, and
// 16 more).
template <bool kQ8>
__device__ __forceinline__ int o_channel(int kk, int e, int fg) {
  if constexpr (kQ8) return (kk >> 1) * 32 + 2 * fg + (kk & 1) + 16 * (e >> 1);
  else return kk * 16 + fg + 8 * (e >> 1);
}

template <int D, int CT, int NT>
__device__ __forceinline__ void decode_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const CUtensorMap& tm_q,
                                            const DecodeParams& p) {
  using C = DecodeCfg<D, CT, NT>;
  constexpr bool kQ8 = !C::k16;
  constexpr bool kBF = CT == kCacheBF16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* merge = smem + C::kStages * C::kStageBytes;  // [kOwnMerge] (8-bit caches)
  uint8_t* qbuf = merge + C::kOwnMerge;                  // [2][kQBytes]
  float2* mls = reinterpret_cast<float2*>(qbuf + 2 * C::kQBytes);
  StageTag* tags = reinterpret_cast<StageTag*>(mls + 4 * 16);
  uint64_t* full = reinterpret_cast<uint64_t*>(tags + C::kStages);
  uint64_t* empty = full + C::kStages;
  uint64_t* q_full = empty + C::kStages;
  uint64_t* q_empty = q_full + 2;

  // What does not read the prologue's results is done before waiting for
  // it: barriers, tensor-map prefetch, and this CTA's slice of the block
  // table (a step input) pulled into L2 for the first items' page lookups.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDecodeWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], kDecodeWarps);
    }
    fence_mbar_init();
  }
  if (warp == kDecodeWarps && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_q);
  }
  if (p.bt_lines > 0)
    for (int i = blockIdx.x * kThreads + threadIdx.x; i < p.bt_lines; i += gridDim.x * kThreads)
      prefetch_l2(p.block_table + (size_t)i * 32);

  // Everything below reads the prologue's work list and the pool it wrote.
  // Launched right after the prologue it waits for it; launched after the
  // prefill kernel (which waited for the prologue before letting this kernel
  // start) it runs beside the prefill on the SMs the prefill left free.
  if (p.wait_prologue) griddep_wait();
  const int active = min(p.counters->dec_ctas, p.counters->n_dec * p.Hk);
  if ((int)blockIdx.x >= active) return;  // no item, or an SM kept for the prefill
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kDecodeWarps) {
    // ------------------------------------------------------------ producer
    const int n_work = p.counters->n_dec * p.Hk;
    const int split_keys = p.counters->split_keys;
    const int boxes = kStageKeys >> p.log_box_rows;
    const int qt = p.q_tile_tokens;
    const uint32_t q_bytes = C::kQChunks * p.G * qt * 128;
    int stage = 0;
    uint32_t phase = 0;
    int quse[2] = {0, 0};
    int qi = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      // First item: this CTA's own index; then the shared queue.
      int u = blockIdx.x;
      if (it > 0 && lane == 0) u = active + atomicAdd(&p.counters->dec_next, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u >= n_work) {
        if (lane == 0) {
          if (mbar_wait(&empty[stage], phase ^ 1)) {
            tags[stage].u = -1;
            mbar_arrive(&full[stage]);
          } else {
            note_timeout(p.err, p.err_site, kSiteDecode | 1);
          }
        }
        break;
      }
      const int item = u / p.Hk, k = u - item * p.Hk;
      const int2 bsplit = p.dec_items[item];  // (decode entry, split)
      const SeqInfo si = p.seq[bsplit.x];
      const int b = si.b;                      // the entry's sequence: its block_table row
      const int start = si.lo + bsplit.y * split_keys;
      const int end = min(si.kv_len, start + split_keys);
      const int past = si.kv_len - si.q_len;
      const int lo_min = p.window >= 1 ? max(0, past + 1 - p.window) : 0;

      // Query rows of the item: box {64, G, qt} at (chunk, k*G, t0).
      if (lane == 0) {
        if (!mbar_wait(&q_empty[qi], (quse[qi] & 1) ^ 1)) {
          note_timeout(p.err, p.err_site, kSiteDecode | 2);
          ok = false;
        } else {
          mbar_arrive_expect_tx(&q_full[qi], q_bytes);
          for (int c = 0; c < C::kQChunks; ++c)
            tma_load_3d(qbuf + qi * C::kQBytes + c * 2048, &tm_q, c * 64, k * p.G, si.t0, &q_full[qi]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      quse[qi]++;

      // Block ids, 32 block-table rows per window, one window ahead.
      const int* bt_row = p.block_table + (size_t)b * p.MB;
      auto load_id = [&](int r) -> int {
        return (r < p.MB && r * p.bs < end) ? __ldg(bt_row + r) : -1;
      };
      int win = start / p.bs;
      int id_cur = load_id(win + lane);
      int id_nxt = load_id(win + 32 + lane);

      for (int key0 = start; key0 < end; key0 += kStageKeys) {
        const int rowA = key0 / p.bs;
        if (rowA >= win + 32) {
          win += 32;
          id_cur = id_nxt;
          id_nxt = load_id(win + 32 + lane);
        }
        // Lane 2*bx (K) and 2*bx+1 (V) own box bx of the stage.
        const int bxl = lane >> 1;
        const int pos = key0 + (bxl << p.log_box_rows);
        const int idx = pos / p.bs - win;  // window-relative block row, 0 .. 35
        const int a = __shfl_sync(0xffffffffu, id_cur, idx & 31);
        const int n = __shfl_sync(0xffffffffu, id_nxt, idx & 31);
        const int blk = idx < 32 ? a : n;
        int rc = p.oob_row;
        if (bxl < boxes && pos < end) {
          if (blk >= 0 && blk < p.NB) rc = blk * p.bs + (pos & (p.bs - 1));
          else if (blk != -1 && (lane & 1) == 0) atomicOr(p.err, PA_DEVERR_BLOCK_ID);
        }
        const unsigned zb = __ballot_sync(0xffffffffu, bxl < boxes && (lane & 1) == 0 && rc == p.oob_row);
        int mask = 0;
        for (int bx = 0; bx < boxes; ++bx) mask |= ((zb >> (2 * bx)) & 1) << bx;
        if (lane == 0) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            note_timeout(p.err, p.err_site, kSiteDecode | 3);
            ok = false;
          } else {
            StageTag& t = tags[stage];
            t.u = u;
            t.key0 = key0;
            t.end = end;
            t.flags = mask | (key0 == start ? kFirst : 0) | (key0 + kStageKeys >= end ? kLast : 0);
            t.R = si.q_len * p.G;
            t.past = past;
            t.t0 = si.t0;
            t.k = k;
            t.kv_len = si.kv_len;
            t.nsplit = si.dec_count;
            t.qi = qi;
            t.lo_min = lo_min;
            t.part = si.part_first >= 0 ? si.part_first + bsplit.y : -1;
            mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (bxl < boxes) {
          uint8_t* dst = stages + stage * C::kStageBytes + (lane & 1) * C::kTileBytes +
                         ((uint32_t)bxl * C::kChunks << (p.log_box_rows + 7));
          tma_load_4d(dst, (lane & 1) ? &tm_v : &tm_k, 0, rc, 0, k, &full[stage]);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      qi ^= 1;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Each warp owns 16 keys of every stage.  S^T = K Q^T puts those keys in
  // the MMA's M rows and the item's query rows in its N columns (NT tiles
  // of 8 rows), so a GQA group of up to 8 rows wastes no M rows; the
  // softmax runs per query row over the keys (row maxima by shuffles
  // across the 8 key groups of the warp); O^T += V^T P^T puts the value
  // channels in M.  P^T reaches that MMA's B operand by an in-register
  // transpose (movmatrix) of the S^T accumulators, packed to fp16.
  //
  // Fragment coordinates (m16n8k16): lane = 4 * fg + ft; the S^T
  // accumulator s[n][e] holds key fg + 8 * (e >> 1) and query row
  // 8n + 2 ft + (e & 1); o[kk][n][e] holds value channel ch(kk, e) (see
  // o_channel) and the same query row.
  const int ctid = threadIdx.x;  // 0..127
  const int fg = lane >> 2, ft = lane & 3;
  int stage = 0;
  uint32_t phase = 0;
  int quse[2] = {0, 0};
  // one K scale for the whole cache: exact to fold into the score scale
  // (section 8.5 phase 3); per-channel K scales are in the query copy
  const float scale = p.k_scale_tensor ? p.scale * __ldg(p.k_scale_tensor) : p.scale;
  const bool capped = p.softcap > 0.f;
  const float inv_cap = capped ? 1.f / p.softcap : 0.f;
  const int log_r = p.log_box_rows;
  constexpr int kKS = D / 16;  // 16-channel steps of the contractions

  // Q^T as B fragments, per 16-channel step and row tile (D <= 128; wider
  // heads reload them from shared memory at each use).
  uint32_t qf[(D <= 128) ? kKS : 1][NT][2];
  float m[NT][2], l[NT][2];  // per query row 8n + 2ft + j: running max (log2 units), partial sum
  float o[kKS][NT][4];
  int hi[NT][2], lo[NT][2];
  const uint8_t* qcur = qbuf;

  // B fragment of Q^T for 16-channel step ks and row tile n: fp16 caches
  // take channels 16ks + 2ft, +1 (b0) and 16ks + 8 + 2ft, +1 (b1); 8-bit
  // caches take the contraction order of their K fragments, channels
  // 16ks + 4ft .. +3 (b0: the first two, b1: the last two).
  auto load_qf = [&](int ks, int n, uint32_t* b) {
    const int row = 8 * n + fg;
    if constexpr (kQ8) {
      const int c = ks * 16 + 4 * ft;
      const uint2 x = *reinterpret_cast<const uint2*>(qcur + (c >> 6) * 2048 + ((c & 7) * 2) +
                                                       swz(row, (c & 63) >> 3));
      b[0] = x.x;
      b[1] = x.y;
    } else {
      const uint8_t* q = qcur + ((ks * 16) >> 6) * 2048;
      const __half2 h0 = *reinterpret_cast<const __half2*>(q + swz(row, ((ks * 16) & 63) >> 3) + 4 * ft);
      const __half2 h1 = *reinterpret_cast<const __half2*>(q + swz(row, ((ks * 16 + 8) & 63) >> 3) + 4 * ft);
      b[0] = *reinterpret_cast<const uint32_t*>(&h0);
      b[1] = *reinterpret_cast<const uint32_t*>(&h1);
    }
  };

  while (true) {
    if (!mbar_wait(&full[stage], phase)) {
      if (lane == 0) note_timeout(p.err, p.err_site, kSiteDecode | 4);
      return;
    }
    const StageTag tg = tags[stage];
    if (tg.u < 0) break;

    if (tg.flags & kFirst) {
      // New item: its query fragments, row bounds and a fresh softmax state.
      if (!mbar_wait(&q_full[tg.qi], quse[tg.qi] & 1)) {
        if (lane == 0) note_timeout(p.err, p.err_site, kSiteDecode | 5);
        return;
      }
      quse[tg.qi]++;
      qcur = qbuf + tg.qi * C::kQBytes;
      if constexpr (D <= 128) {
#pragma unroll
        for (int ks = 0; ks < kKS; ++ks)
#pragma unroll
          for (int n = 0; n < NT; ++n) load_qf(ks, n, qf[ks][n]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_empty[tg.qi]);
      }
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int r = 8 * n + 2 * ft + j;
          hi[n][j] = -1;
          lo[n][j] = 0;
          if (r < tg.R) {
            hi[n][j] = tg.past + r / p.G;  // last admitted position of the row
            lo[n][j] = p.window >= 1 ? max(0, hi[n][j] + 1 - p.window) : 0;
          }
          m[n][j] = -INFINITY;
          l[n][j] = 0.f;
        }
#pragma unroll
      for (int kk = 0; kk < kKS; ++kk)
#pragma unroll
        for (int n = 0; n < NT; ++n) o[kk][n][0] = o[kk][n][1] = o[kk][n][2] = o[kk][n][3] = 0.f;
    }

    const int key0 = tg.key0, end = tg.end, mask = tg.flags & 0xff;
    uint8_t* kt = stages + stage * C::kStageBytes;
    uint8_t* vt = kt + C::kTileBytes;
    const int kw = key0 + warp * 16;  // first key position of this warp

    // Keys outside [lo_min, kv_len) are never admitted by any row; their V
    // rows are zeroed in shared memory so stale bytes (e.g. NaN in a partly
    // filled last block) cannot leak through a zero weight.
    const bool edge = (kw + 16 > tg.kv_len) || (kw < tg.lo_min);
    if (edge) {
      for (int i = lane; i < 16 * C::kChunks * 8; i += 32) {
        const int kr = i / (C::kChunks * 8), rem = i % (C::kChunks * 8);
        const int pos = kw + kr;
        if (pos >= tg.kv_len || pos < tg.lo_min) {
          const int c = rem >> 3, col16 = rem & 7;
          *reinterpret_cast<uint4*>(vt + tile_off<C::kChunks>(warp * 16 + kr, c, col16, log_r)) =
              make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
    }

    if (kw < end && kw + 16 > tg.lo_min) {
      // ---- S^T = K Q^T for this warp's 16 keys x the item's query rows
      float s[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
      const int mi = lane >> 3, ri = lane & 7;
      if constexpr (kQ8) {
        // one ldmatrix per 32 channels: matrix mi = keys (mi&1)*8.., channels
        // +16*(mi>>1); lane (fg, ft) gets channels 4ft..4ft+3 of key fg (+8)
#pragma unroll
        for (int ks2 = 0; ks2 < D / 32; ++ks2) {
          const int key = warp * 16 + (mi & 1) * 8 + ri;
          const int c = ks2 * 32 + (mi >> 1) * 16;
          uint32_t kb[4];
          ldsm_x4(smem_u32(kt + tile_off<C::kChunks>(key, c >> 7, (c & 127) >> 4, log_r)), kb[0], kb[1], kb[2],
                  kb[3]);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int ks = 2 * ks2 + hh;
            uint32_t a[4];
            a[0] = deq2<CT, 0, 1>(kb[2 * hh]);
            a[1] = deq2<CT, 0, 1>(kb[2 * hh + 1]);
            a[2] = deq2<CT, 2, 3>(kb[2 * hh]);
            a[3] = deq2<CT, 2, 3>(kb[2 * hh + 1]);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              if constexpr (D <= 128) {
                hmma16816(s[n], a, qf[ks][n][0], qf[ks][n][1]);
              } else {
                uint32_t b[2];
                load_qf(ks, n, b);
                hmma16816(s[n], a, b[0], b[1]);
              }
            }
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < kKS; ++ks) {
          // matrix mi = keys (mi&1)*8.., channels 16ks + (mi>>1)*8: a0..a3
          const int key = warp * 16 + (mi & 1) * 8 + ri;
          const int d16 = ks * 16 + (mi >> 1) * 8;
          uint32_t a[4];
          ldsm_x4(smem_u32(kt + tile_off<C::kChunks>(key, d16 >> 6, (d16 & 63) >> 3, log_r)), a[0], a[1], a[2],
                  a[3]);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            if constexpr (D <= 128) {
              mma16816<kBF>(s[n], a, qf[ks][n][0], qf[ks][n][1]);
            } else {
              uint32_t b[2];
              load_qf(ks, n, b);
              mma16816<kBF>(s[n], a, b[0], b[1]);
            }
          }
        }
      }
      // ---- scale, softcap, mask; per-row max over the warp's keys
      float tmax[NT][2];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        tmax[n][0] = tmax[n][1] = -INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = e & 1;
          const int pos = kw + fg + 8 * (e >> 1);
          const int box = (pos - key0) >> log_r;
          const bool ok = pos < end && pos <= hi[n][j] && pos >= lo[n][j] && !((mask >> box) & 1);
          float x = s[n][e] * scale;
          if (capped) x = p.softcap * tanhf(x * inv_cap);
          x *= kLog2e;
          x = ok ? x : -INFINITY;
          s[n][e] = x;
          tmax[n][j] = fmaxf(tmax[n][j], x);
        }
      }
      // Lazy rescale: the reference max m moves only when a score exceeds
      // it by more than 2^kLazyRescale, so P stays <= 256 and O is rescaled
      // on few stages (the final merge works with any reference).
      float alpha[NT][2], muse[NT][2];
      bool rescale = false;
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float t = tmax[n][j];
          t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 4));
          t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 8));
          t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 16));
          alpha[n][j] = 1.f;
          if (t > m[n][j] + kLazyRescale) {  // also the first finite score (m = -inf)
            alpha[n][j] = (m[n][j] == -INFINITY) ? 0.f : exp2f(m[n][j] - t);
            m[n][j] = t;
            rescale = true;
          }
          muse[n][j] = (m[n][j] == -INFINITY) ? 0.f : m[n][j];
        }
      uint32_t pb[NT][2];  // P^T as B fragments: keys 2ft, +1 (and + 8) of query row 8n + fg
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) pv[e] = exp2f(s[n][e] - muse[n][e & 1]);
        // this lane's keys of rows 8n + 2ft (j = 0) and 8n + 2ft + 1 (j = 1)
        l[n][0] = l[n][0] * alpha[n][0] + (pv[0] + pv[2]);
        l[n][1] = l[n][1] * alpha[n][1] + (pv[1] + pv[3]);
        // the accumulator halves are m8n8 fragments of (key, row); their
        // transposes are (row, key) pairs, the B fragment of O^T += V^T P^T
        pb[n][0] = movmatrix_t(pack2<kBF>(pv[0], pv[1]));
        pb[n][1] = movmatrix_t(pack2<kBF>(pv[2], pv[3]));
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int kk = 0; kk < kKS; ++kk)
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            o[kk][n][0] *= alpha[n][0];
            o[kk][n][1] *= alpha[n][1];
            o[kk][n][2] *= alpha[n][0];
            o[kk][n][3] *= alpha[n][1];
          }
      }
      // ---- O^T += V^T P^T
      if constexpr (kQ8) {
        // matrix mi = keys (mi>>1)*8.., channels +16*(mi&1), transposed: lane
        // (fg, ft) gets keys 2ft, 2ft+1 of channels 2fg, 2fg+1; the even
        // channels feed one MMA (o[2g32]), the odd ones another (o[2g32+1])
#pragma unroll
        for (int g32 = 0; g32 < D / 32; ++g32) {
          const int key = warp * 16 + (mi >> 1) * 8 + ri;
          const int c = g32 * 32 + (mi & 1) * 16;
          uint32_t vb[4];
          ldsm_x4_t(smem_u32(vt + tile_off<C::kChunks>(key, c >> 7, (c & 127) >> 4, log_r)), vb[0], vb[1], vb[2],
                    vb[3]);
          uint32_t ae[4], ao[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            ae[q] = deq2<CT, 0, 2>(vb[q]);
            ao[q] = deq2<CT, 1, 3>(vb[q]);
          }
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            hmma16816(o[2 * g32][n], ae, pb[n][0], pb[n][1]);
            hmma16816(o[2 * g32 + 1][n], ao, pb[n][0], pb[n][1]);
          }
        }
      } else {
#pragma unroll
        for (int nd = 0; nd < kKS; ++nd) {
          // matrix mi = keys (mi>>1)*8.., channels 16nd + (mi&1)*8, transposed:
          // the A fragment of V^T (channels fg, fg + 8; keys 2ft.., 8 + 2ft..)
          const int key = warp * 16 + (mi >> 1) * 8 + ri;
          const int d = nd * 16 + (mi & 1) * 8;
          uint32_t a[4];
          ldsm_x4_t(smem_u32(vt + tile_off<C::kChunks>(key, d >> 6, (d & 63) >> 3, log_r)), a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int n = 0; n < NT; ++n) mma16816<kBF>(o[nd][n], a, pb[n][0], pb[n][1]);
        }
      }
    }

    if (!(tg.flags & kLast)) {
      if (edge) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    } else {
      // ---- end of item: merge the four warps through this stage's buffer
      float lt[NT][2];
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float v = l[n][j];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          lt[n][j] = v;
        }
      named_bar(1, kDecodeWarps * 32);  // every warp is done reading the stage
      float* mrg = reinterpret_cast<float*>(C::kOwnMerge ? merge : kt);
      constexpr int kRows = 8 * NT;  // rows of a warp's partial output in the merge buffer
      float* mw = mrg + warp * kRows * D;
#pragma unroll
      for (int kk = 0; kk < kKS; ++kk)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = 8 * n + 2 * ft + (e & 1);
            mw[row * D + o_channel<kQ8>(kk, e, fg)] = o[kk][n][e];
          }
      if (fg == 0) {
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int j = 0; j < 2; ++j) mls[warp * 16 + 8 * n + 2 * ft + j] = make_float2(m[n][j], lt[n][j]);
      }
      named_bar(1, kDecodeWarps * 32);
      // (the routing keeps R <= kRows; the bound keeps every access inside
      // the merge buffer regardless)
      for (int e = ctid; e < min(tg.R, kRows) * D; e += kDecodeWarps * 32) {
        const int r = e / D, d = e - r * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, mls[w * 16 + r].x);
        float acc = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kDecodeWarps; ++w) {
            const float2 ml = mls[w * 16 + r];
            const float f = exp2f(ml.x - M);
            den += f * ml.y;
            acc += f * mrg[(w * kRows + r) * D + d];
          }
        }
        if constexpr (kQ8) acc *= __ldg(p.v_scale + (p.per_channel ? tg.k * D + d : 0));
        if (tg.nsplit == 1) {
          const int t = tg.t0 + r / p.G, h = tg.k * p.G + r % p.G;
          // bfloat16 sink and output: a bfloat16 cache, or bfloat16 activations over 8-bit codes
          const bool obf = kBF || (kQ8 && p.act_bf16);
          if (p.head_sink && M != -INFINITY) den += exp2f(elem16_to_float(p.head_sink[h], obf) * kLog2e - M);
          p.out[((size_t)t * p.H + h) * D + d] = float_to_elem16(den > 0.f ? acc / den : 0.f, obf);
        } else {
          const size_t row = ((size_t)tg.part * p.Hk + tg.k) * kDecodeRows + r;
          p.part_o[row * D + d] = acc;
          if (d == 0) p.part_ml[row] = make_float2(M, den);
        }
      }
      fence_proxy_async_smem();
      named_bar(1, kDecodeWarps * 32);
      if (lane == 0) {
        mbar_arrive(&empty[stage]);
        if constexpr (D > 128) mbar_arrive(&q_empty[tg.qi]);
      }
    }
    if (++stage == C::kStages) {
      stage = 0;
      phase ^= 1;
    }
  }
}

template <int D, int CT, int NT>
__global__ void __launch_bounds__(kThreads, DecodeCfg<D, CT, NT>::kCtasPerSm)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const DecodeParams p) {
  decode_body<D, CT, NT>(tm_k, tm_v, tm_q, p);
  // Beside the prefill kernel (launched after it): this grid may complete
  // only once the prefill grid has, so the combine kernel, which waits for
  // this grid, ends the step after both.  One thread of CTA 0 suffices.
  if (!p.wait_prologue && blockIdx.x == 0 && threadIdx.x == 0) griddep_wait();
}

template <int D, int CT, int NT>
cudaError_t configure_nt(size_t* smem, int* ctas) {
  using C = DecodeCfg<D, CT, NT>;
  static_assert(C::kOwnMerge >= C::kMergeBytes || C::kStageBytes >= C::kMergeBytes, "merge buffer");
  static_assert(C::kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(C::kCtasPerSm * (C::kSmemBytes + 1024) <= 228 * 1024, "CTAs per SM");
  *smem = C::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, CT, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_kernel<D, CT, NT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, CT, NT>, kThreads, *smem);
  *ctas = n > 0 ? n : 1;
  return e;
}

// The row-tile variant a GQA group of G heads runs (one tile when G <= 8).
template <int D, int CT>
cudaError_t configure_d(int G, size_t* smem, int* ctas) {
  return G <= 8 ? configure_nt<D, CT, 1>(smem, ctas) : configure_nt<D, CT, 2>(smem, ctas);
}

// One row tile (8 query rows per item) when the GQA group has at most 8
// heads, two (16 rows) otherwise.
template <int D, int CT>
cudaError_t launch_dc(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq, const DecodeParams& p,
                      int grid, cudaStream_t s) {
  if (p.G <= 8)
    return launch_pdl(decode_kernel<D, CT, 1>, grid, kThreads, DecodeCfg<D, CT, 1>::kSmemBytes, s, tk, tv, tq, p);
  return launch_pdl(decode_kernel<D, CT, 2>, grid, kThreads, DecodeCfg<D, CT, 2>::kSmemBytes, s, tk, tv, tq, p);
}

}  // namespace

// 8-bit caches are built for head_size 128 and 256.
cudaError_t decode_configure(int head_size, int cache_type, int group, int* ctas_per_sm, size_t* smem) {
  if (cache_type == kCacheF16) {
    switch (head_size) {
      case 64: return configure_d<64, kCacheF16>(group, smem, ctas_per_sm);
      case 128: return configure_d<128, kCacheF16>(group, smem, ctas_per_sm);
      case 256: return configure_d<256, kCacheF16>(group, smem, ctas_per_sm);
      default: return cudaErrorInvalidValue;
    }
  }
  if (cache_type == kCacheBF16) {
    switch (head_size) {
      case 64: return configure_d<64, kCacheBF16>(group, smem, ctas_per_sm);
      case 128: return configure_d<128, kCacheBF16>(group, smem, ctas_per_sm);
      case 256: return configure_d<256, kCacheBF16>(group, smem, ctas_per_sm);
      default: return cudaErrorInvalidValue;
    }
  }
  const bool i8 = cache_type == kCacheI8;
  switch (head_size) {
    case 128: return i8 ? configure_d<128, kCacheI8>(group, smem, ctas_per_sm) : configure_d<128, kCacheE4M3>(group, smem, ctas_per_sm);
    case 256: return i8 ? configure_d<256, kCacheI8>(group, smem, ctas_per_sm) : configure_d<256, kCacheE4M3>(group, smem, ctas_per_sm);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(int head_size, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                          const DecodeParams& p, int grid, cudaStream_t s) {
  if (p.cache_type == kCacheF16) {
    switch (head_size) {
      case 64: return launch_dc<64, kCacheF16>(tk, tv, tq, p, grid, s);
      case 128: return launch_dc<128, kCacheF16>(tk, tv, tq, p, grid, s);
      case 256: return launch_dc<256, kCacheF16>(tk, tv, tq, p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.cache_type == kCacheBF16) {
    switch (head_size) {
      case 64: return launch_dc<64, kCacheBF16>(tk, tv, tq, p, grid, s);
      case 128: return launch_dc<128, kCacheBF16>(tk, tv, tq, p, grid, s);
      case 256: return launch_dc<256, kCacheBF16>(tk, tv, tq, p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  const bool i8 = p.cache_type == kCacheI8;
  switch (head_size) {
    case 128: return i8 ? launch_dc<128, kCacheI8>(tk, tv, tq, p, grid, s) : launch_dc<128, kCacheE4M3>(tk, tv, tq, p, grid, s);
    case 256: return i8 ? launch_dc<256, kCacheI8>(tk, tv, tq, p, grid, s) : launch_dc<256, kCacheE4M3>(tk, tv, tq, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
