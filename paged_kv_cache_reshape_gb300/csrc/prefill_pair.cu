// Varlen causal prefill, two 128-row query tiles per CTA (head_size 64/128).
//
// Same operation as prefill.cu (S = Q K^T, masked online softmax, O += P V
// on tcgen05 tensor cores; the masks of "PagedAttention - CUDA Design
// Document" section 8 implementation note P5 and section 9.3.1; the flash
// iteration of the CPU GQA notes, onnxruntime 1.27.0 docs,
// contrib_ops/cpu/gqa, "Flash Attention Path"), organised so that the tensor
// core is kept busy:
//   * a unit is 256 query rows of one sequence and kv head: tile A (the
//     first 128/G tokens) and tile B (the next 128/G), G heads per token;
//     every 64-key K/V tile fetched is used by both tiles;
//   * two softmax warpgroups, one per tile, alternate: while one computes
//     P for its tile the tensor core runs the other tile's S and PV;
//   * P goes back into tensor memory (fp16 pairs over the tile's S columns)
//     and feeds the PV MMA as its A operand, so it never touches shared
//     memory; MMAs issued by one thread complete in order, so S(i+1) may
//     reuse the columns once PV(i) is issued, and a wait on S(i+1) also
//     covers PV(i);
//   * TMEM: S_A, S_B (64 columns each), O_A, O_B (head_size each);
//   * shared memory: Q double-buffered (both tiles), 3 K/V stages of 64 keys.
//
// Roles (320 threads, one CTA per SM, persistent over a device queue):
//   warps 0-3 softmax of tile A, warps 4-7 softmax of tile B (thread = row =
//   TMEM lane), warp 8 TMA producer, warp 9 TMEM owner + MMA issuer.
#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kThreads = 10 * 32;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kKeys = 64;     // keys per K/V tile
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.f;  // log2 of the largest P value tolerated before rescaling

template <int D>
struct PairCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kQTileBytes = kPrefillRows * D * 2;  // one 128-row tile [chunk][row][128 B]
  static constexpr int kQBufBytes = 2 * kQTileBytes;         // tiles A and B
  static constexpr int kKVBytes = kKeys * D * 2;             // K or V tile [chunk][key][128 B]
  static constexpr int kStageBytes = 2 * kKVBytes;
  // TMEM columns of S (and P) and of O for tile X (0 = A, 1 = B)
  static __host__ __device__ constexpr int s_col(int X) { return X * kKeys; }
  static __host__ __device__ constexpr int o_col(int X) { return 2 * kKeys + X * D; }
  static constexpr int kTmemCols = (2 * kKeys + 2 * D <= 256) ? 256 : 512;
  static constexpr int kDataBytes = 2 * kQBufBytes + kStages * kStageBytes;
  static constexpr int kSmemBytes = 1024 + kDataBytes + 1024;
};

struct UnitInfo {
  int u;        // work unit (tile * Hk + k); -1 = no more work
  int k;        // kv head
  int t0;       // packed row of the unit's first token
  int ntok[2];  // valid tokens of tiles A and B (B may have 0)
  int pos0;     // position of the unit's first token
  int key_lo;   // first key of the first K/V tile
  int n_kv[2];  // K/V tiles needed by A and by B (n_kv[1] >= n_kv[0])
  int kv_len;   // past + q_len of the sequence
  int lo_min;   // smallest position any row admits
  int pad[5];
};

struct Ctrl {
  UnitInfo info[2];
  uint32_t kv_mask[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t info_full[2], info_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023) == 1023 && *abort) return false;
  }
  *abort = 1;
  atomicOr(err, PA_DEVERR_TIMEOUT);
  return false;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, bool CAP>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using C = PairCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;                       // [2 buffers][tiles A, B]
  uint8_t* kv_s = q_s + 2 * C::kQBufBytes;   // [stage][K, V]
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + C::kDataBytes);
  volatile int* abort = &ctl->abort;

  griddep_wait();  // the work list and the pool come from the prologue
  const int n_work = p.counters->n_pre * p.Hk;
  if ((int)blockIdx.x >= n_work) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], 4);
      mbar_init(&ctl->o_done[i], 1);
      mbar_init(&ctl->info_full[i], 1);
      mbar_init(&ctl->info_empty[i], 1 + 8);  // MMA thread + 8 softmax warps
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctl->kv_full[i], 1);
      mbar_init(&ctl->kv_empty[i], 1);
    }
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
  const int log_r = p.log_page_rows;  // log2(min(block_size, 64))
  const int pages = kKeys >> log_r;
  const int tq = p.tile_tokens;       // tokens per 128-row tile

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    const uint32_t q_bytes = C::kChunks * p.G * tq * 128;
    uint32_t g = 0;
    int last_q = -1;
    bool ok = true;
    for (uint32_t tt = 0; ok; ++tt) {
      const int slot = tt & 1;
      int u = 0;
      if (lane == 0) {
        // First unit: this CTA's own index; then the shared queue.
        if (!wait_or_abort(&ctl->info_empty[slot], ((tt >> 1) & 1) ^ 1, abort, p.err)) u = -2;
        else u = tt == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(&p.counters->pre_next, 1);
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u == -2) break;
      UnitInfo& ui = ctl->info[slot];
      if (u >= n_work) {
        if (lane == 0) {
          ui.u = -1;
          mbar_arrive(&ctl->info_full[slot]);
        }
        break;
      }
      const int tile = u / p.Hk, k = u - tile * p.Hk;
      const int2 bq = p.pre_tiles[tile];
      const SeqInfo si = p.seq[bq.x];
      const int q0 = bq.y * 2 * tq;
      const int nt = min(2 * tq, si.q_len - q0);
      const int ntA = min(tq, nt), ntB = nt - ntA;
      const int pos0 = si.kv_len - si.q_len + q0;
      const int lo_min = p.window >= 1 ? max(0, pos0 + 1 - p.window) : 0;
      const int key_lo = lo_min & ~(kKeys - 1);
      const int nA = (pos0 + ntA - key_lo + kKeys - 1) / kKeys;
      const int nB = ntB > 0 ? (pos0 + nt - key_lo + kKeys - 1) / kKeys : nA;
      const int hi_end = pos0 + nt;
      const int t0 = si.t0 + q0;
      if (lane == 0) {
        ui.u = u;
        ui.k = k;
        ui.t0 = t0;
        ui.ntok[0] = ntA;
        ui.ntok[1] = ntB;
        ui.pos0 = pos0;
        ui.key_lo = key_lo;
        ui.n_kv[0] = nA;
        ui.n_kv[1] = nB;
        ui.kv_len = si.kv_len;
        ui.lo_min = lo_min;
        mbar_arrive(&ctl->info_full[slot]);
        const int qb = tt & 1;
        if (!wait_or_abort(&ctl->q_empty[qb], ((tt >> 1) & 1) ^ 1, abort, p.err)) {
          ok = false;
        } else {
          mbar_arrive_expect_tx(&ctl->q_full[qb], 2 * q_bytes);
          last_q = (int)tt;
          uint8_t* qd = q_s + qb * C::kQBufBytes;
          for (int half = 0; half < 2; ++half)
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(qd + half * C::kQTileBytes + c * (kPrefillRows * 128), &tm_q, c * 64, k * p.G,
                          t0 + half * tq, &ctl->q_full[qb]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;

      const int* bt_row = p.block_table + (size_t)bq.x * p.MB;
      auto load_id = [&](int r) -> int {
        return (r < p.MB && r * p.bs < hi_end) ? __ldg(bt_row + r) : -1;
      };
      int win = key_lo / p.bs;
      int id = load_id(win + lane);
      for (int i = 0; i < nB; ++i, ++g) {
        const int st = g % kStages;
        const int key0 = key_lo + i * kKeys;
        if ((key0 + kKeys - 1) / p.bs >= win + 32) {
          win = key0 / p.bs;
          id = load_id(win + lane);
        }
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
          if (!wait_or_abort(&ctl->kv_empty[st], ((g / kStages) & 1) ^ 1, abort, p.err)) {
            ok = false;
          } else {
            ctl->kv_mask[st] = mask;
            mbar_arrive_expect_tx(&ctl->kv_full[st], C::kStageBytes);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // one box {64, 1, R} per (page, chunk, K|V)
        const int lp = lane / (2 * C::kChunks), lc = (lane >> 1) % C::kChunks;
        const int prc = __shfl_sync(0xffffffffu, rc, lp & 31);
        if (lp < pages) {
          uint8_t* dst = kv_s + st * C::kStageBytes + (lane & 1) * C::kKVBytes + lc * (kKeys * 128) +
                         ((uint32_t)lp << (log_r + 7));
          tma_load_3d(dst, (lane & 1) ? &tm_v : &tm_k, lc * 64, k, prc, &ctl->kv_full[st]);
        }
      }
    }
    if (lane == 0 && *abort) {
      // Gave up: let the copies already issued land before the CTA exits.
      for (uint32_t i = 0; i < kWaitLimit && last_q >= 0 &&
                           !mbar_try_wait(&ctl->q_full[last_q & 1], (last_q >> 1) & 1);
           ++i) {
      }
      for (int d = 1; d <= kStages && (int)g - d >= 0; ++d) {
        const uint32_t gl = g - d;
        for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(&ctl->kv_full[gl % kStages], (gl / kStages) & 1);
             ++i) {
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_f16(kPrefillRows, kKeys, 0, 0);
      constexpr uint32_t idesc_o = umma_idesc_f16(kPrefillRows, D, 0, 1);
      const uint32_t kv_addr = smem_u32(kv_s);
      uint32_t g = 0, pcnt[2] = {0, 0};
      bool ok = true;
      for (uint32_t tt = 0; ok; ++tt) {
        const int slot = tt & 1;
        if (!wait_or_abort(&ctl->info_full[slot], (tt >> 1) & 1, abort, p.err)) break;
        const UnitInfo ui = ctl->info[slot];
        if (ui.u < 0) break;
        const int qb = tt & 1;
        if (!wait_or_abort(&ctl->q_full[qb], (tt >> 1) & 1, abort, p.err)) break;
        tc_fence_after();
        const uint32_t q_addr = smem_u32(q_s + qb * C::kQBufBytes);
        const int n_last = ui.n_kv[1];
        // S_X(i) = Q_X K_i^T; the unit's last S releases the Q buffer.
        auto issue_s = [&](int X, int i) -> bool {
          const uint32_t gi = g + i;
          const int st = gi % kStages;
          if (!wait_or_abort(&ctl->kv_full[st], (gi / kStages) & 1, abort, p.err)) return false;
          tc_fence_after();
          const uint32_t kb = kv_addr + st * C::kStageBytes;
          const uint32_t qa = q_addr + X * C::kQTileBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t a = smem_desc_sw128(qa + (ks >> 2) * (kPrefillRows * 128) + (ks & 3) * 32, 16, 1024);
            const uint64_t b = smem_desc_sw128(kb + (ks >> 2) * (kKeys * 128) + (ks & 3) * 32, 16, 1024);
            umma_f16(tmem + C::s_col(X), a, b, idesc_s, ks > 0);
          }
          umma_commit(&ctl->s_full[X]);
          if (X == 1 && i == n_last - 1) umma_commit(&ctl->q_empty[qb]);
          return true;
        };
        // O_X += P_X(i) V_i with P_X read from TMEM (fp16 pairs over S_X).
        auto issue_pv = [&](int X, int i) -> bool {
          if (!wait_or_abort(&ctl->p_full[X], pcnt[X] & 1, abort, p.err)) return false;
          ++pcnt[X];
          tc_fence_after();
          const int st = (g + i) % kStages;
          const uint32_t vb = kv_addr + st * C::kStageBytes + C::kKVBytes;
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            const uint64_t b = smem_desc_sw128(vb + kk * 16 * 128, kKeys * 128, 1024);
            umma_f16_ts(tmem + C::o_col(X), tmem + C::s_col(X) + kk * 8, b, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
          }
          return true;
        };
        if (!issue_s(0, 0) || !issue_s(1, 0)) break;
        for (int i = 0; i < n_last && ok; ++i) {
          if (i < ui.n_kv[0]) {
            if (!issue_pv(0, i)) { ok = false; break; }
            if (i == ui.n_kv[0] - 1) umma_commit(&ctl->o_done[0]);
            else if (!issue_s(0, i + 1)) { ok = false; break; }
          }
          if (!issue_pv(1, i)) { ok = false; break; }
          umma_commit(&ctl->kv_empty[(g + i) % kStages]);
          if (i == n_last - 1) umma_commit(&ctl->o_done[1]);
          else if (!issue_s(1, i + 1)) { ok = false; break; }
        }
        g += n_last;
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
    const int X = warp >> 2;                  // 0: tile A, 1: tile B
    const int r = threadIdx.x & 127;          // query row == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float mul = CAP ? 1.f : p.scale * kLog2e;
    const float cap_in = CAP ? p.scale / p.softcap : 0.f;
    const float cap_out = CAP ? p.softcap * kLog2e : 0.f;
    uint32_t g = 0, scnt = 0, ocnt = 0;
    float x[kKeys];
    for (uint32_t tt = 0;; ++tt) {
      const int slot = tt & 1;
      if (!wait_or_abort(&ctl->info_full[slot], (tt >> 1) & 1, abort, p.err)) break;
      const UnitInfo ui = ctl->info[slot];
      if (ui.u < 0) break;
      const int j = r / p.G;
      const bool row_ok = j < ui.ntok[X];
      const int hi = ui.pos0 + X * tq + j;                   // last admitted position
      const int lo = p.window >= 1 ? hi + 1 - p.window : 0;  // first admitted position
      const int n_x = ui.n_kv[X];
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int i = 0; i < n_x; ++i) {
        const uint32_t gi = g + i;
        const int st = gi % kStages;
        const int key0 = ui.key_lo + i * kKeys;
        // s_full(i) also covers PV(i-1): MMAs complete in issue order.
        if (!wait_or_abort(&ctl->s_full[X], scnt & 1, abort, p.err) ||
            !wait_or_abort(&ctl->kv_full[st], (gi / kStages) & 1, abort, p.err)) {
          ok = false;
          break;
        }
        ++scnt;
        tc_fence_after();
        tmem_ld32(lane_addr + C::s_col(X), x);
        tmem_ld32(lane_addr + C::s_col(X) + 32, x + 32);
        tmem_ld_wait();
        if constexpr (CAP) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) x[c] = cap_out * tanhf(x[c] * cap_in);
        }
        const uint32_t mask = ctl->kv_mask[st];
        const int c_lo = row_ok ? max(lo - key0, 0) : kKeys;
        const int c_hi = row_ok ? min(hi - key0, kKeys - 1) : -1;
        if (c_lo > 0 || c_hi < kKeys - 1) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) x[c] = (c >= c_lo && c <= c_hi) ? x[c] : -INFINITY;
        }
        if (mask != 0) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) x[c] = ((mask >> (c >> log_r)) & 1) ? -INFINITY : x[c];
        }
        // Row max as a tree (a 64-long dependent chain would dominate).
        float mx[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) mx[c] = fmaxf(fmaxf(x[c], x[c + 16]), fmaxf(x[c + 32], x[c + 48]));
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) mx[c] = fmaxf(mx[c], mx[c + w]);
        const float tmax = mx[0];
        const float cand = tmax * mul;
        float alpha = 1.f;
        if (cand > m_ref + kLazyRescale || (m_ref == -INFINITY && cand != -INFINITY)) {
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - cand);
          m_ref = cand;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        float sums[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int c = 0; c < kKeys; c += 2) {
          const float e0 = ex2(fmaf(x[c], mul, -m_use));
          const float e1 = ex2(fmaf(x[c + 1], mul, -m_use));
          sums[(c >> 1) & 7] += e0 + e1;
          pk[c / 2] = pack_half2(e0, e1);
        }
        const float rs = ((sums[0] + sums[1]) + (sums[2] + sums[3])) + ((sums[4] + sums[5]) + (sums[6] + sums[7]));
        l = l * alpha + rs;
        if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          float o[32];
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            tmem_ld32(lane_addr + C::o_col(X) + 32 * c, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(lane_addr + C::o_col(X) + 32 * c, o);
          }
        }
        // Never-admitted keys of an edge tile: zero their V rows (tile A does
        // it while it uses the tile, tile B for the tiles A skips).
        if ((X == 0 || i >= ui.n_kv[0]) && (key0 + kKeys > ui.kv_len || key0 < ui.lo_min)) {
          uint8_t* vs = kv_s + st * C::kStageBytes + C::kKVBytes;
          for (int idx = r; idx < kKeys * C::kChunks * 8; idx += 128) {
            const int kr = idx / (C::kChunks * 8), rem = idx % (C::kChunks * 8);
            const int pos = key0 + kr;
            if (pos >= ui.kv_len || pos < ui.lo_min) {
              const int c = rem >> 3, col16 = rem & 7;
              *reinterpret_cast<uint4*>(vs + c * (kKeys * 128) + kr * 128 + ((col16 ^ (kr & 7)) << 4)) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        // P_X -> TMEM over S_X (32 columns of fp16 pairs)
        tmem_st32(lane_addr + C::s_col(X), reinterpret_cast<const float*>(pk));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[X]);
      }
      if (!ok) break;
      // epilogue: O_X / l -> fp16 output rows
      if (!wait_or_abort(&ctl->o_done[X], ocnt & 1, abort, p.err)) break;
      ++ocnt;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const int t = ui.t0 + X * tq + j, h = ui.k * p.G + (r - j * p.G);
      __half* dst = p.out + ((size_t)t * p.H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(lane_addr + C::o_col(X) + 32 * c, o);
        tmem_ld_wait();
        if (row_ok) {
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
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->info_empty[slot]);
      g += ui.n_kv[1];
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
  static_assert(PairCfg<D>::kSmemBytes <= 227 * 1024, "shared memory");
  return cudaFuncSetAttribute(prefill_pair_kernel<D, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)PairCfg<D>::kSmemBytes);
}

template <int D>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     int grid, cudaStream_t s) {
  if (p.softcap > 0.f)
    return launch_pdl(prefill_pair_kernel<D, true>, grid, kThreads, PairCfg<D>::kSmemBytes, s, tq, tk, tv, p);
  return launch_pdl(prefill_pair_kernel<D, false>, grid, kThreads, PairCfg<D>::kSmemBytes, s, tq, tk, tv, p);
}

}  // namespace

cudaError_t prefill_pair_configure(int head_size) {
  cudaError_t e;
  switch (head_size) {
    case 64:
      e = configure_dc<64, false>();
      return e != cudaSuccess ? e : configure_dc<64, true>();
    case 128:
      e = configure_dc<128, false>();
      return e != cudaSuccess ? e : configure_dc<128, true>();
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_prefill_pair(int head_size, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const PrefillParams& p, int grid, cudaStream_t s) {
  switch (head_size) {
    case 64: return launch_d<64>(tq, tk, tv, p, grid, s);
    case 128: return launch_d<128>(tq, tk, tv, p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

// Dispatch: head_size 64 and 128 use the two-tile kernel above, 256 (whose
// two tiles would not fit in tensor memory) the one-tile kernel.
bool prefill_uses_pairs(int head_size) { return head_size <= 128; }

cudaError_t prefill_configure(int head_size, size_t* smem) {
  if (prefill_uses_pairs(head_size)) {
    *smem = head_size == 64 ? PairCfg<64>::kSmemBytes : PairCfg<128>::kSmemBytes;
    return prefill_pair_configure(head_size);
  }
  return prefill_single_configure(head_size, smem);
}

int prefill_keys_per_tile(int head_size) {
  return prefill_uses_pairs(head_size) ? kKeys : prefill_single_keys_per_tile(head_size);
}

int prefill_unit_tokens(int head_size, int group) {
  const int tile = group <= kPrefillRows ? kPrefillRows / group : 1;
  return prefill_uses_pairs(head_size) ? 2 * tile : tile;
}

cudaError_t launch_prefill(int head_size, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int grid, cudaStream_t s) {
  if (prefill_uses_pairs(head_size)) return launch_prefill_pair(head_size, tq, tk, tv, p, grid, s);
  return launch_prefill_single(head_size, tq, tk, tv, p, grid, s);
}

}  // namespace pa
