// Varlen causal prefill over the paged pool on tcgen05 tensor cores.
//
// A tile is (sequence b, kv head k, 128 query rows) where the rows are
// 128/G consecutive new tokens of b times the G query heads that share kv
// head k (row r = token j * G + head g), so every K/V tile fetched serves
// the whole GQA group.  For each 128-key (64 for head_size 256) KV tile:
//   S = Q K^T        tcgen05.mma, M=128, N=keys, K=head_size -> TMEM
//   softmax          one thread per row reads its S row from TMEM, applies
//                    scale, softcap, the causal bound past + j + 1, the
//                    window [kv_len - W, kv_len) and -1 blocks, keeps the
//                    running max / sum in fp32 and writes P (fp16) to shared
//                    memory
//   O += P V         tcgen05.mma, M=128, N=head_size, K=keys -> TMEM
// then O / l is written as fp16.  This is the online-softmax flash
// iteration of the CPU GQA notes (onnxruntime 1.27.0 docs,
// contrib_ops/cpu/gqa, "Flash Attention Path", steps 1-5) with the masks of
// "PagedAttention - CUDA Design Document" section 8 implementation note P5
// and section 9.3.1.  Unlike the vendored Flash kernel of that document
// (section 18.1), a KV tile may span several pages: each page is its own
// TMA box, so any power-of-two block_size >= 16 works.
//
// The running max is kept lazily: a row rescales its O accumulator (a TMEM
// read-modify-write) only when its max grows by more than 2^8, so P stays
// below 256 and the final O / l is unchanged (both carry the same factor).
//
// Warp roles (192 threads, one CTA per SM, persistent over a device queue):
//   warps 0-3  softmax + epilogue (thread = query row = TMEM lane)
//   warp 4     TMA producer: tile descriptions, Q tile (double-buffered for
//              head_size <= 128), K/V tiles (2 stages; one lane per box)
//   warp 5     TMEM owner and MMA issuer (one elected thread)
// S for KV tile i+1 is computed while the softmax warps work on tile i, and
// the softmax computes P for tile i while P V of tile i-1 is still running.
// BF: bfloat16 activations (section 8.2): bfloat16 A/B in the MMA
// instruction descriptors, P stored as bfloat16, bfloat16 sink and output.
#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kThreads = 6 * 32;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.f;  // log2 of the largest P value tolerated before rescaling

template <int D>
struct PrefillCfg {
  static constexpr int kKeys = (D == 256) ? 64 : 128;   // keys per KV tile
  static constexpr int kChunks = D / 64;                // 128-byte channel chunks
  static constexpr int kQBufs = (D == 256) ? 1 : 2;     // Q tiles in flight
  static constexpr int kQBytes = kPrefillRows * D * 2;  // [chunk][128 rows][128 B]
  static constexpr int kPBytes = kPrefillRows * kKeys * 2;
  static constexpr int kTileBytes = kKeys * D * 2;      // K or V tile [chunk][keys][128 B]
  static constexpr int kStages = 2;
  static constexpr int kSCol = 0, kOCol = kKeys;        // TMEM columns of S and O
  static constexpr int kTmemCols = (kKeys + D <= 256) ? 256 : 512;
  static constexpr int kDataBytes = kQBufs * kQBytes + kPBytes + kStages * 2 * kTileBytes;
  static constexpr int kSmemBytes = 1024 + kDataBytes + 1024;
};

struct TileInfo {
  int u;       // work unit (tile * Hk + k); -1 = no more work
  int k;       // kv head
  int t0;      // packed row of the tile's first token
  int ntok;    // valid tokens in the tile
  int pos0;    // position of the tile's first token (past + q0)
  int key_lo;  // first key of the first KV tile
  int n_kv;    // KV tiles
  int kv_len;  // past + q_len of the sequence
  int lo_min;  // smallest position any row admits
  int pad[7];
};

struct Ctrl {
  TileInfo info[2];
  uint32_t kv_mask[2];  // per stage: bit p = page p zero-filled (unmapped / past the end)
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[2], kv_empty[2];
  uint64_t s_full, s_free, p_full, o_done;
  uint64_t info_full[2], info_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D, bool CAP, bool BF>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int KEYS = C::kKeys;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;                          // [kQBufs][kQBytes]
  uint8_t* p_s = q_s + C::kQBufs * C::kQBytes;  // [kPBytes]
  uint8_t* kv_s = p_s + C::kPBytes;             // stage st: K at st*2*tile, V right after
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + C::kDataBytes);
  volatile int* abort = &ctl->abort;

  // The work list and the pool come from the prologue.  Steps without
  // prefill work (and CTAs beyond the work) leave before touching TMEM.
  griddep_wait();
  griddep_launch_dependents();  // the decode kernel may start on the SMs this grid leaves free
  const int n_work = p.counters->n_pre * p.Hk;
  // CTAs beyond the work or beyond the work list's SM split leave at once.
  const int active = min(n_work, p.counters->pre_ctas);
  if ((int)blockIdx.x >= active) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
      mbar_init(&ctl->kv_full[i], 1);
      mbar_init(&ctl->kv_empty[i], 1);
      mbar_init(&ctl->info_full[i], 1);
      mbar_init(&ctl->info_empty[i], 1 + 4);  // MMA thread + 4 softmax warps
    }
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->s_free, 4);
    mbar_init(&ctl->p_full, 4);
    mbar_init(&ctl->o_done, 1);
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int log_r = p.log_page_rows;  // log2(min(block_size, KEYS))
  const int pages = KEYS >> log_r;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const uint32_t q_bytes = C::kChunks * p.G * p.tile_tokens * 128;
    uint32_t g = 0;
    int last_q = -1;  // last tile whose Q load was issued
    bool ok = true;
    for (uint32_t tt = 0; ok; ++tt) {
      const int slot = tt & 1;
      int u = 0;
      if (lane == 0) {
        // First tile: this CTA's own index; then the shared queue.
        if (!wait_or_abort(&ctl->info_empty[slot], ((tt >> 1) & 1) ^ 1, abort, p.err, p.err_site, kSitePrefill | 11)) u = -2;
        else u = tt == 0 ? (int)blockIdx.x : active + atomicAdd(&p.counters->pre_next, 1);
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u == -2) break;
      TileInfo& ti = ctl->info[slot];
      if (u >= n_work) {
        if (lane == 0) {
          ti.u = -1;
          mbar_arrive(&ctl->info_full[slot]);
        }
        break;
      }
      const int tile = u / p.Hk, k = u - tile * p.Hk;
      const int2 bq = p.pre_tiles[tile];
      const SeqInfo si = p.seq[bq.x];
      const int q0 = bq.y * p.tile_tokens;
      const int ntok = min(p.tile_tokens, si.q_len - q0);
      const int pos0 = si.kv_len - si.q_len + q0;
      const int hi_end = pos0 + ntok;  // one past the last row's last admitted key
      const int lo_min = p.window >= 1 ? max(0, pos0 + 1 - p.window) : 0;
      const int key_lo = lo_min & ~(KEYS - 1);
      const int n_kv = (hi_end - key_lo + KEYS - 1) / KEYS;
      const int t0 = si.t0 + q0;
      if (lane == 0) {
        ti.u = u;
        ti.k = k;
        ti.t0 = t0;
        ti.ntok = ntok;
        ti.pos0 = pos0;
        ti.key_lo = key_lo;
        ti.n_kv = n_kv;
        ti.kv_len = si.kv_len;
        ti.lo_min = lo_min;
        mbar_arrive(&ctl->info_full[slot]);
        // Q tile: box {64, G, tile_tokens} per channel chunk.
        const int qb = tt % C::kQBufs;
        if (!wait_or_abort(&ctl->q_empty[qb], ((tt / C::kQBufs) & 1) ^ 1, abort, p.err, p.err_site, kSitePrefill | 13)) {
          ok = false;
        } else {
          mbar_arrive_expect_tx(&ctl->q_full[qb], q_bytes);
          last_q = (int)tt;
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(q_s + qb * C::kQBytes + c * (kPrefillRows * 128), &tm_q, c * 64, k * p.G, t0,
                        &ctl->q_full[qb]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;

      // Block ids, 32 block-table rows at a time, one per lane.
      const int* bt_row = p.block_table + (size_t)bq.x * p.MB;
      auto load_id = [&](int r) -> int {
        return (r < p.MB && r * p.bs < hi_end) ? __ldg(bt_row + r) : -1;
      };
      int win = key_lo / p.bs;
      int id = load_id(win + lane);
      for (int i = 0; i < n_kv; ++i, ++g) {
        const int st = g & 1;
        const int key0 = key_lo + i * KEYS;
        if ((key0 + KEYS - 1) / p.bs >= win + 32) {
          win = key0 / p.bs;
          id = load_id(win + lane);
        }
        // lane pg < pages resolves page pg of this tile
        const int pos = key0 + (lane << log_r);
        const int idx = pos / p.bs - win;
        const int blk = __shfl_sync(0xffffffffu, id, idx & 31);
        int rc = p.oob_row;
        if (lane < pages && pos < hi_end) {
          if (blk >= 0 && blk < p.NB) rc = blk * p.bs + (pos & (p.bs - 1));
          else if (blk != -1) atomicOr(p.err, PA_DEVERR_BLOCK_ID);
        }
        const uint32_t mask = __ballot_sync(0xffffffffu, lane < pages && rc == p.oob_row);
        if (lane == 0) {
          if (!wait_or_abort(&ctl->kv_empty[st], ((g >> 1) & 1) ^ 1, abort, p.err, p.err_site, kSitePrefill | 12)) {
            ok = false;
          } else {
            ctl->kv_mask[st] = mask;
            mbar_arrive_expect_tx(&ctl->kv_full[st], 2 * C::kTileBytes);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // one box {64, 1, R} per (page, chunk, K|V); lane -> (page, chunk, tensor)
        const int lp = lane / (2 * C::kChunks), lc = (lane >> 1) % C::kChunks;
        const int prc = __shfl_sync(0xffffffffu, rc, lp & 31);
        if (lp < pages) {
          uint8_t* dst = kv_s + st * 2 * C::kTileBytes + (lane & 1) * C::kTileBytes + lc * (KEYS * 128) +
                         ((uint32_t)lp << (log_r + 7));
          tma_load_3d(dst, (lane & 1) ? &tm_v : &tm_k, lc * 64, k, prc, &ctl->kv_full[st]);
        }
      }
    }
    if (lane == 0 && *abort) {
      // Gave up: let the copies already issued land before the CTA exits.
      for (uint32_t i = 0; i < kWaitLimit && last_q >= 0 &&
                           !mbar_try_wait(&ctl->q_full[last_q % C::kQBufs], (last_q / C::kQBufs) & 1);
           ++i) {
      }
      for (int d = 1; d <= 2 && (int)g - d >= 0; ++d) {
        const uint32_t gl = g - d;
        for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(&ctl->kv_full[gl & 1], (gl >> 1) & 1); ++i) {
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // (one elect.sync-chosen lane: MMAs issued under it cost far fewer
    // cycles than under a lane-index branch)
    if (elect_one()) {
      constexpr uint32_t idesc_s = umma_idesc_f16(kPrefillRows, KEYS, 0, 0, BF ? 1 : 0);
      constexpr uint32_t idesc_o = umma_idesc_f16(kPrefillRows, D, 0, 1, BF ? 1 : 0);
      const uint32_t p_addr = smem_u32(p_s), kv_addr = smem_u32(kv_s);
      uint32_t g = 0, s_issued = 0, v = 0;
      bool ok = true;
      for (uint32_t tt = 0; ok; ++tt) {
        const int slot = tt & 1;
        if (!wait_or_abort(&ctl->info_full[slot], (tt >> 1) & 1, abort, p.err, p.err_site, kSitePrefill | 1)) break;
        const TileInfo ti = ctl->info[slot];
        if (ti.u < 0) break;
        const int qb = tt % C::kQBufs;
        if (!wait_or_abort(&ctl->q_full[qb], (tt / C::kQBufs) & 1, abort, p.err, p.err_site, kSitePrefill | 2)) break;
        tc_fence_after();
        const uint32_t q_addr = smem_u32(q_s + qb * C::kQBytes);
        // S(i) = Q K_i^T into TMEM columns [kSCol, kSCol + KEYS)
        auto issue_s = [&](uint32_t gi, bool last) -> bool {
          const int st = gi & 1;
          if (!wait_or_abort(&ctl->kv_full[st], (gi >> 1) & 1, abort, p.err, p.err_site, kSitePrefill | 3)) return false;
          if (s_issued > 0 && !wait_or_abort(&ctl->s_free, (s_issued - 1) & 1, abort, p.err, p.err_site, kSitePrefill | 4)) return false;
          tc_fence_after();
          const uint32_t kb = kv_addr + st * 2 * C::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t a = smem_desc_sw128(q_addr + (ks >> 2) * (kPrefillRows * 128) + (ks & 3) * 32, 16, 1024);
            const uint64_t b = smem_desc_sw128(kb + (ks >> 2) * (KEYS * 128) + (ks & 3) * 32, 16, 1024);
            umma_f16(tmem + C::kSCol, a, b, idesc_s, ks > 0);
          }
          umma_commit(&ctl->s_full);
          if (last) umma_commit(&ctl->q_empty[qb]);
          ++s_issued;
          return true;
        };
        if (!issue_s(g, ti.n_kv == 1)) break;
        for (int i = 0; i < ti.n_kv; ++i) {
          const uint32_t gi = g + i;
          if (i + 1 < ti.n_kv && !issue_s(gi + 1, i + 2 == ti.n_kv)) {
            ok = false;
            break;
          }
          if (!wait_or_abort(&ctl->p_full, v & 1, abort, p.err, p.err_site, kSitePrefill | 5)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int st = gi & 1;
          const uint32_t vb = kv_addr + st * 2 * C::kTileBytes + C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < KEYS / 16; ++kk) {
            const uint64_t a = smem_desc_sw128(p_addr + (kk >> 2) * (kPrefillRows * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t b = smem_desc_sw128(vb + kk * 16 * 128, KEYS * 128, 1024);
            umma_f16(tmem + C::kOCol, a, b, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&ctl->kv_empty[st]);
          umma_commit(&ctl->o_done);
          ++v;
        }
        g += ti.n_kv;
        if (!ok) break;
        mbar_arrive(&ctl->info_empty[slot]);
      }
      // Drain: every MMA issued above has completed before TMEM is freed.
      umma_commit(&ctl->drain);
      for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(&ctl->drain, 0); ++i) {
      }
    }
  } else {
    // ----------------------------------------------------- softmax warps
    const int r = threadIdx.x;  // query row == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    // Scores become log2-domain logits: x * mul (softcap applies its own).
    const float mul = CAP ? 1.f : p.scale * kLog2e;
    const float cap_in = CAP ? p.scale / p.softcap : 0.f;
    const float cap_out = CAP ? p.softcap * kLog2e : 0.f;
    uint32_t g = 0, s_cnt = 0, v = 0;
    float x[KEYS];
    for (uint32_t tt = 0;; ++tt) {
      const int slot = tt & 1;
      if (!wait_or_abort(&ctl->info_full[slot], (tt >> 1) & 1, abort, p.err, p.err_site, kSitePrefill | 6)) break;
      const TileInfo ti = ctl->info[slot];
      if (ti.u < 0) break;
      const int j = r / p.G;
      const bool row_ok = j < ti.ntok;
      const int hi = ti.pos0 + j;                            // last admitted position
      const int lo = p.window >= 1 ? hi + 1 - p.window : 0;  // first admitted position
      float m_ref = -INFINITY;  // reference max (log2 units) of P and O
      float l = 0.f;
      bool ok = true;
      for (int i = 0; i < ti.n_kv; ++i) {
        const uint32_t gi = g + i;
        const int st = gi & 1;
        const int key0 = ti.key_lo + i * KEYS;
        if (!wait_or_abort(&ctl->s_full, s_cnt & 1, abort, p.err, p.err_site, kSitePrefill | 7) ||
            !wait_or_abort(&ctl->kv_full[st], (gi >> 1) & 1, abort, p.err, p.err_site, kSitePrefill | 8)) {
          ok = false;
          break;
        }
        ++s_cnt;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < KEYS / 32; ++c) tmem_ld32(lane_addr + C::kSCol + 32 * c, x + 32 * c);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->s_free);

        if constexpr (CAP) {
#pragma unroll
          for (int c = 0; c < KEYS; ++c) x[c] = cap_out * tanhf(x[c] * cap_in);
        }
        // Admitted columns of this tile for this row: [c_lo, c_hi] minus
        // zero-filled pages.
        const uint32_t mask = ctl->kv_mask[st];
        const int c_lo = row_ok ? max(lo - key0, 0) : KEYS;
        const int c_hi = row_ok ? min(hi - key0, KEYS - 1) : -1;
        if (c_lo > 0 || c_hi < KEYS - 1) {
#pragma unroll
          for (int c = 0; c < KEYS; ++c) x[c] = (c >= c_lo && c <= c_hi) ? x[c] : -INFINITY;
        }
        if (mask != 0) {
#pragma unroll
          for (int c = 0; c < KEYS; ++c) x[c] = ((mask >> (c >> log_r)) & 1) ? -INFINITY : x[c];
        }
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < KEYS; ++c) tmax = fmaxf(tmax, x[c]);
        const float cand = tmax * mul;
        float alpha = 1.f;
        if (cand > m_ref + kLazyRescale || (m_ref == -INFINITY && cand != -INFINITY)) {
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - cand);
          m_ref = cand;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        float rs = 0.f;
#pragma unroll
        for (int c = 0; c < KEYS; ++c) {
          const float e = ex2(fmaf(x[c], mul, -m_use));
          x[c] = e;
          rs += e;
        }
        l = l * alpha + rs;
        // PV(i-1) must be done before O is rescaled and P is overwritten.
        if (i > 0) {
          if (!wait_or_abort(&ctl->o_done, (v + i - 1) & 1, abort, p.err, p.err_site, kSitePrefill | 9)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            float o[32];
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              tmem_ld32(lane_addr + C::kOCol + 32 * c, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(lane_addr + C::kOCol + 32 * c, o);
            }
            tmem_st_wait();
          }
        }
        // Never-admitted keys of an edge tile: zero their V rows so stale
        // bytes (a partly filled last block) cannot leak through P = 0.
        if (key0 + KEYS > ti.kv_len || key0 < ti.lo_min) {
          uint8_t* vs = kv_s + st * 2 * C::kTileBytes + C::kTileBytes;
          for (int idx = r; idx < KEYS * C::kChunks * 8; idx += 128) {
            const int kr = idx / (C::kChunks * 8), rem = idx % (C::kChunks * 8);
            const int pos = key0 + kr;
            if (pos >= ti.kv_len || pos < ti.lo_min) {
              const int c = rem >> 3, col16 = rem & 7;
              *reinterpret_cast<uint4*>(vs + c * (KEYS * 128) + kr * 128 + ((col16 ^ (kr & 7)) << 4)) =
                  make_uint4(0, 0, 0, 0);
            }
          }
        }
        // P row r -> shared memory, K-major 128-byte swizzled [key chunk][row][128 B]
#pragma unroll
        for (int c8 = 0; c8 < KEYS / 8; ++c8) {
          uint4 w;
          w.x = pack2<BF>(x[8 * c8 + 0], x[8 * c8 + 1]);
          w.y = pack2<BF>(x[8 * c8 + 2], x[8 * c8 + 3]);
          w.z = pack2<BF>(x[8 * c8 + 4], x[8 * c8 + 5]);
          w.w = pack2<BF>(x[8 * c8 + 6], x[8 * c8 + 7]);
          const int kc = c8 >> 3, col16 = c8 & 7;
          *reinterpret_cast<uint4*>(p_s + kc * (kPrefillRows * 128) + r * 128 + ((col16 ^ (r & 7)) << 4)) = w;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full);
      }
      if (!ok) break;
      // epilogue: O / l -> fp16 output rows
      if (!wait_or_abort(&ctl->o_done, (v + ti.n_kv - 1) & 1, abort, p.err, p.err_site, kSitePrefill | 10)) break;
      tc_fence_after();
      const int t = ti.t0 + j, h = ti.k * p.G + (r - j * p.G);
      // head_sink (section 6.1): exp(s_h - m) joins the denominator
      if (p.head_sink && m_ref != -INFINITY) l += ex2(elem16_to_float(p.head_sink[h], BF) * kLog2e - m_ref);
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      __half* dst = p.out + ((size_t)t * p.H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(lane_addr + C::kOCol + 32 * c, o);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2<BF>(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l);
            w.y = pack2<BF>(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l);
            w.z = pack2<BF>(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l);
            w.w = pack2<BF>(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l);
            *reinterpret_cast<uint4*>(dst + 32 * c + 8 * q) = w;
          }
        }
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
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool CAP>
cudaError_t configure_dc() {
  static_assert(sizeof(Ctrl) <= 1024, "control block");
  static_assert(PrefillCfg<D>::kSmemBytes <= 227 * 1024, "shared memory");
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, CAP, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)PrefillCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_kernel<D, CAP, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)PrefillCfg<D>::kSmemBytes);
}

template <int D>
cudaError_t configure_d(size_t* smem) {
  *smem = PrefillCfg<D>::kSmemBytes;
  cudaError_t e = configure_dc<D, false>();
  return e != cudaSuccess ? e : configure_dc<D, true>();
}

template <int D, bool BF>
cudaError_t launch_db(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                      int grid, cudaStream_t s) {
  if (p.softcap > 0.f)
    return launch_pdl(prefill_kernel<D, true, BF>, grid, kThreads, PrefillCfg<D>::kSmemBytes, s, tq, tk, tv, p);
  return launch_pdl(prefill_kernel<D, false, BF>, grid, kThreads, PrefillCfg<D>::kSmemBytes, s, tq, tk, tv, p);
}

template <int D>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     int grid, cudaStream_t s) {
  return p.bf16 ? launch_db<D, true>(tq, tk, tv, p, grid, s) : launch_db<D, false>(tq, tk, tv, p, grid, s);
}

}  // namespace

cudaError_t prefill_single_configure(int head_size, size_t* smem) {
  switch (head_size) {
    case 64: return configure_d<64>(smem);
    case 128: return configure_d<128>(smem);
    case 256: return configure_d<256>(smem);
    default: return cudaErrorInvalidValue;
  }
}

int prefill_single_keys_per_tile(int head_size) { return head_size == 256 ? 64 : 128; }

cudaError_t launch_prefill_single(int head_size, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int grid, cudaStream_t s) {
  switch (head_size) {
    case 64: return launch_d<64>(tq, tk, tv, p, grid, s);
    case 128: return launch_d<128>(tq, tk, tv, p, grid, s);
    case 256: return launch_d<256>(tq, tk, tv, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
