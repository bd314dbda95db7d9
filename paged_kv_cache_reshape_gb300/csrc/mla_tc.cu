// Multi-head latent attention decode on tcgen05 tensor cores, for steps
// whose query-head count is a multiple of 128 (the DeepSeek-V3 shape): the
// absorbed form of "PagedAttention - CUDA Design Document", section 12 (one
// latent row of 576 channels per key shared by every query head, V = its
// first 512 channels, explicit scale), with the masks of section 8
// implementation note P5 (causal bound, window, softcap, -1 blocks).
//
// A work unit is (sequence, split of its keys, 128 query heads of its one
// new token, half of the 512 value channels).  The 128 heads are the M rows
// of the MMAs:
//   S = Q K^T      M=128, N=32 keys, K=576: 24 MMAs with Q's first 384
//                  channels read from TMEM, 12 with the last 192 from shared
//                  memory
//   softmax        one thread per head row (TMEM lane), fp32, lazy rescale
//                  (2^8), P written back over S as fp16 pairs
//   O += P V       M=128, N=256 channels, K=32 keys, A = P from TMEM, B =
//                  the same latent tile in shared memory read as V
// The full 128 x 512 fp32 output would fill all 512 TMEM columns, so the two
// halves of the value channels go to two units (two CTAs), each recomputing
// S; they read the same latent tiles, the second read mostly from L2.
//
// TMEM (512 columns): Q channels 0..383 as fp16 pairs [0, 192), S/P of even
// and odd tiles [192, 224) and [224, 256), O [256, 512).  Shared memory: Q
// channels 384..575 (48 KB) and a 4-deep ring of 32-key latent tiles (36 KB
// each, [chunk][key][128 B], 128-byte swizzle; one 4-D TMA box per tile
// with pages of 32 rows or more, else one box per page and chunk).  At a unit's start, once the previous unit's tiles are consumed,
// Q's TMEM part is staged through the first three ring slots and copied
// into TMEM (tcgen05.cp, in issue order before the unit's first S), then
// the ring refills from slot 0.  MMAs issued by one thread complete in
// order, so S(i+1), issued ahead of PV(i), may reuse the columns of
// S/P(i-1) once PV(i-1) is issued.
//
// Warp roles (192 threads, one CTA per SM, persistent over the device
// queue): warps 0-3 softmax and epilogue, warp 4 TMA producer, warp 5 TMEM
// owner and MMA issuer.  Split units write fp32 partials laid out like the
// other decode kernels' (16 rows per item and 16-head group) for the
// combine kernel.
#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kD = 576, kDV = 512, kHalf = kDV / 2;
constexpr int kChunks = kD / 64;                  // 9 chunks of 64 channels
constexpr int kQTChunks = 6;                      // Q chunks held in TMEM (channels 0..383)
constexpr int kQSChunks = kChunks - kQTChunks;    // Q chunks read from shared memory
constexpr int kKeys = 32;                         // keys per latent tile
constexpr int kRows = 128;                        // query heads per unit (MMA M)
constexpr int kThreads = 6 * 32;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kQChunkBytes = kRows * 128;         // one chunk of Q [head][128 B]
constexpr int kQSBytes = kQSChunks * kQChunkBytes;
constexpr int kTileBytes = kChunks * kKeys * 128; // [chunk][key][128 B]
constexpr int kStages = 4;
constexpr int kQCol = 0, kSCol = kQTChunks * 4 * 8, kOCol = 256;  // TMEM columns
constexpr int kTmemCols = 512;
constexpr int kDataBytes = kQSBytes + kStages * kTileBytes;
constexpr int kSmemBytes = 1024 + kDataBytes + 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.f;
static_assert(kQTChunks * kQChunkBytes <= 3 * kTileBytes, "Q staging fits the first ring slots");
static_assert(kSCol + 64 <= kOCol, "TMEM columns");

struct UnitInfo {
  int u;       // work unit; -1 = no more work
  int ht;      // 128-head tile
  int half;    // value channels [half * 256, half * 256 + 256)
  int item;    // (sequence, split) work item
  int t0;      // packed row of the sequence's new token
  int past;    // its position: the last admitted key
  int key0;    // first key of the split (a multiple of 32)
  int end;     // split end (exclusive)
  int n_kv;    // latent tiles of the split
  int lo_min;  // smallest admitted position (window), 0 without one
  int kv_len;  // past + 1
  int nsplit;  // splits of the sequence
  int part;    // split-partial slot of this split, -1 for an unsplit entry
  int pad[3];
};

struct Ctrl {
  UnitInfo info[2];
  uint32_t kv_mask[kStages];  // per stage: bit p = page p zero-filled (unmapped / past the end)
  uint64_t q_full, q_empty, q_staged;  // Q loaded; Q's shared-memory part free; Q's TMEM part copied
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full, o_done;
  uint64_t info_full[2], info_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Ring slot of tile i of a unit: the first tile goes to the slot that does
// not stage Q, so its load overlaps the Q copy into TMEM.
__device__ __forceinline__ int slot_of(int i) { return (i + kStages - 1) % kStages; }

template <bool CAP>
__global__ void __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qr,
                  const __grid_constant__ CUtensorMap tm_l, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs_s = smem;             // Q channels 384..575 [chunk][head][128 B]
  uint8_t* kv_s = qs_s + kQSBytes;  // [kStages][kTileBytes]; slots 0-2 also stage Q channels 0..383
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + kDataBytes);
  volatile int* abort = &ctl->abort;

  // Barriers, tensor-map prefetch and an L2 prefetch of the block table (a
  // step input) before waiting for the prologue; TMEM only once this CTA
  // knows it has work.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    mbar_init(&ctl->q_staged, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctl->kv_full[i], 1);
      mbar_init(&ctl->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->info_full[i], 1);
      mbar_init(&ctl->info_empty[i], 1 + 4);  // MMA thread + 4 softmax warps
    }
    mbar_init(&ctl->p_full, 4);
    mbar_init(&ctl->o_done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_qr);
    prefetch_tmap(&tm_l);
  }
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < p.bt_lines; i += gridDim.x * kThreads)
    prefetch_l2(p.block_table + (size_t)i * 32);

  griddep_wait();  // the work list and the latent rows come from the prologue
  const int n_ht = p.H / kRows;
  const int per_item = 2 * n_ht;  // units per (sequence, split)
  const int n_work = p.counters->n_dec * per_item;
  const int active = min(p.counters->dec_ctas, n_work);
  if ((int)blockIdx.x >= active) return;

  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = ctl->tmem_base;
  const int log_r = p.log_tile_rows;  // log2(min(block_size, 32)): pool rows per TMA box
  const int pages = kKeys >> log_r;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const int split_keys = p.counters->split_keys;
    uint32_t sp = 0, used = 0;  // per ring slot (bit): parity of its loads so far, any load issued
    int q_loads = 0;
    bool ok = true;
    for (uint32_t tt = 0; ok; ++tt) {
      const int slot = tt & 1;
      int u = 0;
      if (lane == 0) {
        if (!wait_or_abort(&ctl->info_empty[slot], ((tt >> 1) & 1) ^ 1, abort, p.err, p.err_site, kSiteMlaTc | 13)) u = -2;
        else u = tt == 0 ? (int)blockIdx.x : active + atomicAdd(&p.counters->dec_next, 1);
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u == -2) break;
      UnitInfo& ti = ctl->info[slot];
      if (u >= n_work) {
        if (lane == 0) {
          ti.u = -1;
          mbar_arrive(&ctl->info_full[slot]);
        }
        break;
      }
      const int item = u / per_item, rest = u - item * per_item;
      const int ht = rest >> 1, half = rest & 1;
      const int2 bsplit = p.dec_items[item];  // (decode entry, split)
      const SeqInfo si = p.seq[bsplit.x];
      const int start = si.lo + bsplit.y * split_keys;
      const int end = min(si.kv_len, start + split_keys);
      const int past = si.kv_len - si.q_len;
      const int n_kv = (end - start + kKeys - 1) / kKeys;
      if (lane == 0) {
        ti.u = u;
        ti.ht = ht;
        ti.half = half;
        ti.item = item;
        ti.t0 = si.t0;
        ti.past = past;
        ti.key0 = start;
        ti.end = end;
        ti.n_kv = n_kv;
        ti.lo_min = p.window >= 1 ? max(0, past + 1 - p.window) : 0;
        ti.kv_len = si.kv_len;
        ti.nsplit = si.dec_count;
        ti.part = si.part_first >= 0 ? si.part_first + bsplit.y : -1;
        mbar_arrive(&ctl->info_full[slot]);
        // Q: the previous unit's tiles are all consumed (the staging slots
        // are free) and its last S has completed (Q's shared-memory part is
        // free); one box {64, 128, 1} per chunk.
        for (int st = 0; st < kStages && ok; ++st)
          ok = wait_or_abort(&ctl->kv_empty[st], ((sp >> st) & 1) ^ 1, abort, p.err, p.err_site, kSiteMlaTc | 14);
        if (ok) ok = wait_or_abort(&ctl->q_empty, (tt & 1) ^ 1, abort, p.err, p.err_site, kSiteMlaTc | 1);
        if (ok) {
          mbar_arrive_expect_tx(&ctl->q_full, kChunks * kQChunkBytes);
          ++q_loads;
          for (int c = 0; c < kChunks; ++c)
            tma_load_3d(c < kQTChunks ? kv_s + c * kQChunkBytes : qs_s + (c - kQTChunks) * kQChunkBytes,
                        c >= p.qr_lo && c < p.qr_hi ? &tm_qr : &tm_q, c * 64, ht * kRows, si.t0, &ctl->q_full);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;

      // Block ids, 32 block-table rows at a time, one per lane.
      const int* bt_row = p.block_table + (size_t)si.b * p.MB;
      auto load_id = [&](int r) -> int { return (r < p.MB && r * p.bs < end) ? __ldg(bt_row + r) : -1; };
      int win = start / p.bs;
      int id = load_id(win + lane);
      for (int i = 0; i < n_kv; ++i) {
        const int st = slot_of(i);
        const int key0 = start + i * kKeys;
        if ((key0 + kKeys - 1) / p.bs >= win + 32) {
          win = key0 / p.bs;
          id = load_id(win + lane);
        }
        // lane pg < pages resolves page pg of this tile
        const int pos = key0 + (lane << log_r);
        const int idx = pos / p.bs - win;
        const int blk = __shfl_sync(0xffffffffu, id, idx & 31);
        int rc = p.oob_row;
        if (lane < pages && pos < end) {
          if (blk >= 0 && blk < p.NB) rc = blk * p.bs + (pos & (p.bs - 1));
          else if (blk != -1) atomicOr(p.err, PA_DEVERR_BLOCK_ID);
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, lane < pages && rc == p.oob_row);
        if (lane == 0) {
          // the slots that staged Q are reused once its copy into TMEM is done
          if (i == 1) ok = wait_or_abort(&ctl->q_staged, tt & 1, abort, p.err, p.err_site, kSiteMlaTc | 2);
          if (ok) ok = wait_or_abort(&ctl->kv_empty[st], ((sp >> st) & 1) ^ 1, abort, p.err, p.err_site, kSiteMlaTc | 15);
          if (ok) {
            ctl->kv_mask[st] = mask;
            mbar_arrive_expect_tx(&ctl->kv_full[st], kTileBytes);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        sp ^= 1u << st;
        used |= 1u << st;
        if (log_r == 5) {
          // one page of 32 keys: one box {64, 32, 9, 1} of the 4-D view
          if (lane == 0) tma_load_4d(kv_s + st * kTileBytes, &tm_l, 0, rc, 0, 0, &ctl->kv_full[st]);
        } else {
          // one box {64, 1, 2^log_r} per (page, chunk); lane -> (page, chunk)
          for (int base = 0; base < pages * kChunks; base += 32) {
            const int bx = base + lane;
            const int lp = min(bx / kChunks, 31), lc = bx % kChunks;
            const int prc = __shfl_sync(0xffffffffu, rc, lp);
            if (bx < pages * kChunks)
              tma_load_3d(kv_s + st * kTileBytes + lc * (kKeys * 128) + ((uint32_t)lp << (log_r + 7)), &tm_l,
                          lc * 64, 0, prc, &ctl->kv_full[st]);
          }
        }
      }
      // The next unit's Q overwrites the staging slots: a one-tile unit has
      // not waited for its copy into TMEM yet.
      if (ok && n_kv < 2) {
        if (lane == 0) ok = wait_or_abort(&ctl->q_staged, tt & 1, abort, p.err, p.err_site, kSiteMlaTc | 3);
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
    }
    if (lane == 0 && *abort) {
      // Gave up: let the copies already issued land before the CTA exits.
      for (uint32_t i = 0; i < kWaitLimit && q_loads > 0 && !mbar_try_wait(&ctl->q_full, (q_loads - 1) & 1); ++i) {
      }
      for (int st = 0; st < kStages; ++st)
        for (uint32_t i = 0;
             i < kWaitLimit && ((used >> st) & 1) && !mbar_try_wait(&ctl->kv_full[st], ((sp >> st) & 1) ^ 1); ++i) {
        }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // (one elect.sync-chosen lane: MMAs issued under it cost far fewer
    // cycles than under a lane-index branch)
    if (elect_one()) {
      constexpr uint32_t idesc_s = umma_idesc_f16(kRows, kKeys, 0, 0);
      constexpr uint32_t idesc_o = umma_idesc_f16(kRows, kHalf, 0, 1);
      const uint64_t desc_k = smem_desc_sw128(0, 16, 1024);          // K-major, + (address >> 4)
      const uint64_t desc_v = smem_desc_sw128(0, kKeys * 128, 1024);  // MN-major V, + (address >> 4)
      const uint32_t qs_addr = smem_u32(qs_s), kv_addr = smem_u32(kv_s);
      uint32_t sp = 0;       // per ring slot (bit): parity of the tiles taken so far
      uint32_t g = 0, v = 0;  // tiles (S buffers) and PVs so far
      bool ok = true;
      for (uint32_t tt = 0; ok; ++tt) {
        const int slot = tt & 1;
        if (!wait_or_abort(&ctl->info_full[slot], (tt >> 1) & 1, abort, p.err, p.err_site, kSiteMlaTc | 4)) break;
        const UnitInfo ti = ctl->info[slot];
        if (ti.u < 0) break;
        if (!wait_or_abort(&ctl->q_full, tt & 1, abort, p.err, p.err_site, kSiteMlaTc | 5)) break;
        tc_fence_after();
        // Q channels 0..383 into TMEM (after the previous unit's last S in
        // issue order); the staging slots are free once the copies complete.
#pragma unroll
        for (int ks = 0; ks < kQTChunks * 4; ++ks)
          tmem_cp_128x256b(tmem + kQCol + 8 * ks, desc_k + ((kv_addr + (ks >> 2) * kQChunkBytes + (ks & 3) * 32) >> 4));
        umma_commit(&ctl->q_staged);
        // S(gi) = Q K^T into S buffer gi & 1: the columns of S/P(gi - 2),
        // whose PV was issued before this.
        auto issue_s = [&](uint32_t gi, int i, bool last) -> bool {
          const int st = slot_of(i);
          if (!wait_or_abort(&ctl->kv_full[st], (sp >> st) & 1, abort, p.err, p.err_site, kSiteMlaTc | 6)) return false;
          sp ^= 1u << st;
          tc_fence_after();
          const uint32_t kb = kv_addr + st * kTileBytes;
          const uint32_t sc = tmem + kSCol + 32 * (gi & 1);
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const uint64_t b = desc_k + ((kb + (ks >> 2) * (kKeys * 128) + (ks & 3) * 32) >> 4);
            if (ks < kQTChunks * 4) {
              umma_f16_ts(sc, tmem + kQCol + 8 * ks, b, idesc_s, ks > 0 ? 1u : 0u);
            } else {
              const int kq = ks - kQTChunks * 4;
              const uint64_t a = desc_k + ((qs_addr + (kq >> 2) * kQChunkBytes + (kq & 3) * 32) >> 4);
              umma_f16(sc, a, b, idesc_s, 1u);
            }
          }
          umma_commit(&ctl->s_full[gi & 1]);
          if (last) umma_commit(&ctl->q_empty);
          return true;
        };
        if (!issue_s(g, 0, ti.n_kv == 1)) break;
        for (int i = 0; i < ti.n_kv; ++i) {
          const uint32_t gi = g + i;
          const int st = slot_of(i);
          // S(gi + 1) goes ahead of PV(gi): it runs while the softmax works
          // on tile gi.
          if (i + 1 < ti.n_kv && !issue_s(gi + 1, i + 1, i + 2 == ti.n_kv)) {
            ok = false;
            break;
          }
          if (!wait_or_abort(&ctl->p_full, v & 1, abort, p.err, p.err_site, kSiteMlaTc | 7)) {
            ok = false;
            break;
          }
          ++v;
          tc_fence_after();
          // O += P(gi) V(gi): P from TMEM (fp16 pairs over S), V = this
          // half's four channel chunks of the same latent tile.
          const uint32_t vb = kv_addr + st * kTileBytes + ti.half * (kHalf / 64) * (kKeys * 128);
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            umma_f16_ts(tmem + kOCol, tmem + kSCol + 32 * (gi & 1) + kk * 8, desc_v + ((vb + kk * 16 * 128) >> 4),
                        idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&ctl->kv_empty[st]);
          umma_commit(&ctl->o_done);
        }
        g += ti.n_kv;
        if (!ok) break;
        mbar_arrive(&ctl->info_empty[slot]);
      }
      // Drain: every MMA and copy issued above has completed before TMEM is freed.
      umma_commit(&ctl->drain);
      for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(&ctl->drain, 0); ++i) {
      }
    }
  } else {
    // ----------------------------------------------------- softmax warps
    const int r = threadIdx.x;  // head row within the unit == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    // Scores become log2-domain logits: x * mul (softcap applies its own).
    const float mul = CAP ? 1.f : p.scale * kLog2e;
    const float cap_in = CAP ? p.scale / p.softcap : 0.f;
    const float cap_out = CAP ? p.softcap * kLog2e : 0.f;
    uint32_t g = 0, v = 0;
    uint32_t sp = 0;  // per ring slot (bit): parity of the tiles taken so far
    float x[kKeys];
    for (uint32_t tt = 0;; ++tt) {
      const int slot = tt & 1;
      if (!wait_or_abort(&ctl->info_full[slot], (tt >> 1) & 1, abort, p.err, p.err_site, kSiteMlaTc | 8)) break;
      const UnitInfo ti = ctl->info[slot];
      if (ti.u < 0) break;
      const int hi = ti.past;                                // last admitted position
      const int lo = p.window >= 1 ? hi + 1 - p.window : 0;  // first admitted position
      float m_ref = -INFINITY;  // reference max (log2 units) of P and O
      float l = 0.f;
      bool ok = true;
      for (int i = 0; i < ti.n_kv; ++i) {
        const uint32_t gi = g + i;
        const int sb = gi & 1;        // S buffer
        const int st = slot_of(i);    // ring slot of the tile
        const int key0 = ti.key0 + i * kKeys;
        if (!wait_or_abort(&ctl->s_full[sb], (gi >> 1) & 1, abort, p.err, p.err_site, kSiteMlaTc | 9) ||
            !wait_or_abort(&ctl->kv_full[st], (sp >> st) & 1, abort, p.err, p.err_site, kSiteMlaTc | 10)) {
          ok = false;
          break;
        }
        sp ^= 1u << st;
        tc_fence_after();
        tmem_ld32(lane_addr + kSCol + 32 * sb, x);
        tmem_ld_wait();
        if constexpr (CAP) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) x[c] = cap_out * tanhf(x[c] * cap_in);
        }
        // Admitted columns of this tile: [c_lo, c_hi] minus zero-filled pages.
        const uint32_t mask = ctl->kv_mask[st];
        const int c_lo = max(lo - key0, 0);
        const int c_hi = min(min(hi, ti.end - 1) - key0, kKeys - 1);
        if (c_lo > 0 || c_hi < kKeys - 1) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) x[c] = (c >= c_lo && c <= c_hi) ? x[c] : -INFINITY;
        }
        if (mask != 0) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) x[c] = ((mask >> (c >> log_r)) & 1) ? -INFINITY : x[c];
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) tmax = fmaxf(tmax, x[c]);
        const float cand = tmax * mul;
        float alpha = 1.f;
        if (cand > m_ref + kLazyRescale || (m_ref == -INFINITY && cand != -INFINITY)) {
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - cand);
          m_ref = cand;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        float rs = 0.f;
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int c = 0; c < kKeys; c += 2) {
          const float e0 = ex2(fmaf(x[c], mul, -m_use)), e1 = ex2(fmaf(x[c + 1], mul, -m_use));
          rs += e0 + e1;
          pk[c / 2] = pack_half2(e0, e1);
        }
        l = l * alpha + rs;
        // Before P(gi) is published, PV(gi - 1) has completed (needed anyway
        // before O is rescaled).  Waiting on every tile, not only on a
        // rescale, keeps the barrier phases sound: S(gi + 1) is issued ahead
        // of PV(gi), so without this wait a warp could finish tile gi + 1
        // before a slower warp finished tile gi and arrive twice in one phase
        // of the four-warp p_full barrier (PV(gi) would read a partial P, and
        // the phases seen by the slower warp would then run two ahead, so its
        // parity waits stall until they time out); and the epilogue's parity
        // wait on o_done could see that barrier two phases behind and pass
        // before the unit's last PVs.  PV(gi - 1) needs P(gi - 1), published a
        // tile ago, so this wait rarely waits.
        if (i > 0) {
          if (!wait_or_abort(&ctl->o_done, (v + i - 1) & 1, abort, p.err, p.err_site, kSiteMlaTc | 11)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            float o[32];
#pragma unroll 1
            for (int c = 0; c < kHalf / 32; ++c) {
              tmem_ld32(lane_addr + kOCol + 32 * c, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(lane_addr + kOCol + 32 * c, o);
            }
          }
        }
        // Never-admitted keys of an edge tile: zero their rows of this
        // half's value channels so stale bytes (a partly filled last block)
        // cannot leak through P = 0.
        if (key0 + kKeys > ti.kv_len || key0 < ti.lo_min) {
          uint8_t* vs = kv_s + st * kTileBytes + ti.half * (kHalf / 64) * (kKeys * 128);
          for (int idx = r; idx < kKeys * (kHalf / 64) * 8; idx += 128) {
            const int kr = idx / ((kHalf / 64) * 8), rem = idx % ((kHalf / 64) * 8);
            const int pos = key0 + kr;
            if (pos >= ti.kv_len || pos < ti.lo_min) {
              const int c = rem >> 3, col16 = rem & 7;
              *reinterpret_cast<uint4*>(vs + c * (kKeys * 128) + kr * 128 + ((col16 ^ (kr & 7)) << 4)) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        // P -> TMEM over S: keys 0..31 as 16 columns of fp16 pairs
        tmem_st16(lane_addr + kSCol + 32 * sb, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full);
      }
      if (!ok) break;
      // epilogue: O / l -> fp16 output rows, or fp32 partials of a split
      if (!wait_or_abort(&ctl->o_done, (v + ti.n_kv - 1) & 1, abort, p.err, p.err_site, kSiteMlaTc | 12)) break;
      tc_fence_after();
      const int h = ti.ht * kRows + r;
      const int c0 = ti.half * kHalf;
      if (ti.nsplit == 1) {
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        __half* dst = p.out + ((size_t)ti.t0 * p.H + h) * kDV + c0;
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          float o[32];
          tmem_ld32(lane_addr + kOCol + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_half2(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l);
            w.y = pack_half2(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l);
            w.z = pack_half2(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l);
            w.w = pack_half2(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l);
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * q) = w;
          }
        }
      } else {
        // rows of 16-head group h / 16 of the item, as the combine kernel reads them
        const size_t prow = ((size_t)ti.part * p.groups + h / kDecodeRows) * kDecodeRows + h % kDecodeRows;
        float* dst = p.part_o + prow * kDV + c0;
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          float o[32];
          tmem_ld32(lane_addr + kOCol + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(dst + 32 * c + 4 * q) = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2],
                                                                           o[4 * q + 3]);
        }
        if (ti.half == 0) p.part_ml[prow] = make_float2(m_ref, l);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->info_empty[slot]);
      g += ti.n_kv;
      v += ti.n_kv;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool CAP>
cudaError_t configure_cap() {
  static_assert(sizeof(Ctrl) <= 1024, "control block");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  return cudaFuncSetAttribute(mla_tc_kernel<CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

}  // namespace

cudaError_t mla_tc_configure(size_t* smem) {
  *smem = kSmemBytes;
  cudaError_t e = configure_cap<false>();
  return e != cudaSuccess ? e : configure_cap<true>();
}

cudaError_t launch_mla_tc(const CUtensorMap& tq, const CUtensorMap& tqr, const CUtensorMap& tl, const MlaParams& p,
                          int grid, cudaStream_t s) {
  if (p.softcap > 0.f) return launch_pdl(mla_tc_kernel<true>, grid, kThreads, kSmemBytes, s, tq, tqr, tl, p);
  return launch_pdl(mla_tc_kernel<false>, grid, kThreads, kSmemBytes, s, tq, tqr, tl, p);
}

}  // namespace pa
