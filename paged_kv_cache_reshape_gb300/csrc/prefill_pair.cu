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
//     every 128-key K/V tile fetched is used by both tiles;
//   * S = Q K^T runs as M=128, N=128 MMAs: at N=128 the tensor core reads
//     8 KB of shared memory per 64-cycle MMA, within the 128 B/clk port
//     (at N=64 it would read 6 KB per 32 cycles and wait on shared memory);
//   * two softmax warpgroups, one per tile, alternate: while one computes
//     P for its tile the tensor core runs the other tile's PV and next S;
//   * P goes back into tensor memory (fp16 pairs over the tile's S columns)
//     and feeds the PV MMA as its A operand, so it never touches shared
//     memory; MMAs issued by one thread complete in order, so S(i+1) may
//     reuse the columns once PV(i) is issued, and a wait on S(i+1) also
//     covers PV(i);
//   * the softmax does two fp32 lanes per instruction (f32x2 FMA/ADD) and a
//     three-input max;
//   * TMEM: S_A, S_B (128 columns each), O_A, O_B (head_size each);
//   * bfloat16 activations (section 8.2; BF): the same kernel with bfloat16
//     A/B in the MMA instruction descriptors, P packed as bfloat16 pairs,
//     bfloat16 sink and output;
//   * shared memory: one Q buffer per tile, a ring of K and V tile slots
//     loaded in the order they are used: K0 V0 K1 V1 ...
//
// Roles (512 threads = 4 warpgroups, one CTA per SM, persistent over a
// device queue; registers moved between warpgroups with setmaxnreg):
//   warpgroup 0 / 1: softmax of tile A / B (thread = row = TMEM lane);
//   warpgroup 2: epilogue of both tiles: reads O from TMEM (releasing it to
//     the next unit at once), divides by the row sums, stores the output;
//   warpgroup 3: warp 12 K/V producer (TMA), warp 13 TMEM owner + MMA
//     issuer, warp 14 work fetcher (device queue -> unit ring, Q loads).
#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kThreads = 16 * 32;
constexpr int kEpiWarp0 = 8, kProducerWarp = 12, kMmaWarp = 13, kFetchWarp = 14;
// Registers per thread after the split (launch: 65536 / 512 = 128 each).
constexpr int kRegSoftmax = 184, kRegEpilogue = 64, kRegControl = 80;
static_assert(2 * kRegSoftmax + kRegEpilogue + kRegControl == 4 * 128, "register split");
constexpr int kKeys = 128;  // keys per K/V tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.f;  // log2 of the largest P value tolerated before rescaling
constexpr int kSmemLimit = 227 * 1024;
constexpr int kCtrlBytes = 2048;

template <int D>
struct PairCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kQTileBytes = kPrefillRows * D * 2;  // one 128-row tile [chunk][row][128 B]
  static constexpr int kSlotBytes = kKeys * D * 2;           // one K or V tile [chunk][key][128 B]
  static constexpr int kSlotsFit = (kSmemLimit - 1024 - kCtrlBytes - 2 * kQTileBytes) / kSlotBytes;
  static constexpr int kSlots = kSlotsFit > 8 ? 8 : kSlotsFit;
  // TMEM columns of S (and P) and of O for tile X (0 = A, 1 = B)
  static __host__ __device__ constexpr int s_col(int X) { return X * kKeys; }
  static __host__ __device__ constexpr int o_col(int X) { return 2 * kKeys + X * D; }
  static constexpr int kTmemCols = 512;
  static constexpr int kDataBytes = 2 * kQTileBytes + kSlots * kSlotBytes;
  static constexpr int kSmemBytes = 1024 + kDataBytes + kCtrlBytes;
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
  int b;        // sequence (row of the block table)
  int pad[4];
};

constexpr int kInfoRing = 4;  // units published ahead of their use
// Page masks of the K/V tiles in flight, each published with an mbarrier
// arrive before the tile's K load is issued.  The producer runs at most
// kSlots / 2 + 1 tiles ahead of the softmax warpgroups (it reuses a slot only
// after the MMAs that read it, which follow the softmax of older tiles), so
// an entry is rewritten only after both warpgroups have read it and a
// barrier never runs a full phase ahead of its reader.
constexpr int kMaskRing = 8;

struct Ctrl {
  UnitInfo info[kInfoRing];
  uint32_t kv_mask[kMaskRing];   // per K/V tile (tile number mod ring): its pages that are unmapped
  uint64_t mask_full[kMaskRing];  // one arrive per publication
  uint64_t q_full[2], q_empty[2];  // per tile (A, B): its Q buffer
  uint64_t full[8], empty[8];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t l_full[2], l_empty[2];
  uint64_t info_full[kInfoRing], info_empty[kInfoRing];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float l_row[2][kPrefillRows];  // per tile: the softmax row sums of the unit, for the epilogue
};

__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// Maximum of N values as a tree of three-input max.
template <int N>
__device__ __forceinline__ float max_tree(const float* v) {
  if constexpr (N == 1) {
    return v[0];
  } else {
    constexpr int M = (N + 2) / 3;
    float w[M];
#pragma unroll
    for (int k = 0; k < M; ++k) {
      if (3 * k + 2 < N) w[k] = max3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
      else if (3 * k + 1 < N) w[k] = fmaxf(v[3 * k], v[3 * k + 1]);
      else w[k] = v[3 * k];
    }
    return max_tree<M>(w);
  }
}

// Two fp32 lanes in one 64-bit register (Blackwell f32x2 arithmetic).
__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
template <int D, bool CAP, bool BF>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const PrefillParams p) {
  using C = PairCfg<D>;
  constexpr int S = C::kSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;                       // [tile A, tile B]
  uint8_t* kv_s = q_s + 2 * C::kQTileBytes;  // [slot]: K_i is load 2i, V_i load 2i+1
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + C::kDataBytes);
  volatile int* abort = &ctl->abort;

  griddep_wait();  // the work list and the pool come from the prologue
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
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], 4);
      mbar_init(&ctl->o_done[i], 1);
      mbar_init(&ctl->o_free[i], 4);
      mbar_init(&ctl->l_full[i], 4);
      mbar_init(&ctl->l_empty[i], 4);
    }
    for (int i = 0; i < kInfoRing; ++i) {
      mbar_init(&ctl->info_full[i], 1);
      mbar_init(&ctl->info_empty[i], 1 + 8 + 4 + 1);  // MMA, softmax, epilogue and K/V producer warps
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], 1);
    }
    for (int i = 0; i < kMaskRing; ++i) mbar_init(&ctl->mask_full[i], 1);
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
  const int log_r = p.log_page_rows;  // log2(min(block_size, 128))
  const int pages = kKeys >> log_r;
  const int tq = p.tile_tokens;       // tokens per 128-row tile

  // Register split: each warpgroup resizes at the top of its own branch
  // (the allocator budgets a branch from the setmaxnreg that dominates it).
  if (warp >= kProducerWarp) {
   regs_dec<kRegControl>();
   if (warp == kFetchWarp) {
    // ------------------------------------------------------------ fetcher
    // Takes units from the device queue, publishes them in the unit ring
    // (up to kInfoRing - 1 ahead of their use) and loads their Q tiles as
    // soon as the previous unit's last S MMAs on it have completed.  Kept apart
    // from the K/V producer: the queue atomic and the two dependent global
    // loads per unit would otherwise stall the K/V stream.
    if (lane == 0) prefetch_tmap(&tm_q);
    const uint32_t q_bytes = C::kChunks * p.G * tq * 128;
    uint32_t q_loads = 0;  // Q tile loads issued so far (A, B, A, B, ...)
    bool ok = true;
    for (uint32_t tt = 0; ok; ++tt) {
      int u = 0;
      if (lane == 0) u = tt == 0 ? (int)blockIdx.x : active + atomicAdd(&p.counters->pre_next, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      UnitInfo f;
      f.u = -1;
      if (u < n_work) {
        const int tile = u / p.Hk, k = u - tile * p.Hk;
        const int2 bq = p.pre_tiles[tile];
        const SeqInfo si = p.seq[bq.x];
        const int q0 = bq.y * 2 * tq;
        const int nt = min(2 * tq, si.q_len - q0);
        const int ntA = min(tq, nt), ntB = nt - ntA;
        const int pos0 = si.kv_len - si.q_len + q0;
        const int lo_min = p.window >= 1 ? max(0, pos0 + 1 - p.window) : 0;
        const int key_lo = lo_min & ~(kKeys - 1);
        f.u = u;
        f.k = k;
        f.b = bq.x;
        f.t0 = si.t0 + q0;
        f.ntok[0] = ntA;
        f.ntok[1] = ntB;
        f.pos0 = pos0;
        f.key_lo = key_lo;
        f.n_kv[0] = (pos0 + ntA - key_lo + kKeys - 1) / kKeys;
        f.n_kv[1] = ntB > 0 ? (pos0 + nt - key_lo + kKeys - 1) / kKeys : f.n_kv[0];
        f.kv_len = si.kv_len;
        f.lo_min = lo_min;
      }
      const int slot = tt % kInfoRing;
      if (lane == 0) {
        if (!wait_or_abort(&ctl->info_empty[slot], ((tt / kInfoRing) & 1) ^ 1, abort, p.err, p.err_site, kSitePrefillPair | 12)) {
          ok = false;
        } else {
          ctl->info[slot] = f;
          mbar_arrive(&ctl->info_full[slot]);
        }
        // Q tile X of unit tt into its buffer once unit tt-1's S_X MMAs are done
        for (int X = 0; X < 2 && ok && f.u >= 0; ++X) {
          if (!wait_or_abort(&ctl->q_empty[X], (tt & 1) ^ 1, abort, p.err, p.err_site, kSitePrefillPair | 1)) {
            ok = false;
          } else {
            mbar_arrive_expect_tx(&ctl->q_full[X], q_bytes);
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_3d(q_s + X * C::kQTileBytes + c * (kPrefillRows * 128), &tm_q, c * 64, f.k * p.G,
                          f.t0 + X * tq, &ctl->q_full[X]);
            ++q_loads;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (f.u < 0) break;
    }
    if (lane == 0 && *abort) {
      // Gave up: let the copies already issued land before the CTA exits.
      for (int d = 1; d <= 2 && (int)q_loads - d >= 0; ++d) {
        const uint32_t n = q_loads - d;
        for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(&ctl->q_full[n & 1], (n >> 1) & 1); ++i) {
        }
      }
    }
   } else if (warp == kProducerWarp) {
    // ------------------------------------------------------- K/V producer
    // Streams the K and V tiles of every published unit through the ring.
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    uint32_t n_loads = 0;  // K/V slot loads issued so far
    bool ok = true;
    // One K or V tile into the next ring slot: lane l copies page
    // l / chunks, 64-column chunk l % chunks (a box of {64, 1, page rows}).
    auto load_tile = [&](const CUtensorMap* tm, int k, int rc, bool is_v, uint32_t mask) -> bool {
      const int slot = n_loads % S;
      if (lane == 0) {
        if (!wait_or_abort(&ctl->empty[slot], ((n_loads / S) & 1) ^ 1, abort, p.err, p.err_site, kSitePrefillPair | 13)) {
          ok = false;
        } else {
          if (!is_v) {
            ctl->kv_mask[(n_loads >> 1) % kMaskRing] = mask;
            mbar_arrive(&ctl->mask_full[(n_loads >> 1) % kMaskRing]);
          }
          mbar_arrive_expect_tx(&ctl->full[slot], C::kSlotBytes);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return false;
      const int lp = lane / C::kChunks, lc = lane % C::kChunks;
      const int prc = __shfl_sync(0xffffffffu, rc, lp & 31);
      if (lp < pages) {
        uint8_t* dst = kv_s + slot * C::kSlotBytes + lc * (kKeys * 128) + ((uint32_t)lp << (log_r + 7));
        tma_load_3d(dst, tm, lc * 64, k, prc, &ctl->full[slot]);
      }
      ++n_loads;
      return true;
    };
    for (uint32_t tt = 0; ok; ++tt) {
      const int slot = tt % kInfoRing;
      int got = 1;
      if (lane == 0) got = wait_or_abort(&ctl->info_full[slot], (tt / kInfoRing) & 1, abort, p.err, p.err_site, kSitePrefillPair | 2) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      const UnitInfo cur = ctl->info[slot];
      if (cur.u < 0) break;
      const int hi_end = cur.pos0 + cur.ntok[0] + cur.ntok[1];
      const int* bt_row = p.block_table + (size_t)cur.b * p.MB;
      auto load_id = [&](int r) -> int {
        return (r < p.MB && r * p.bs < hi_end) ? __ldg(bt_row + r) : -1;
      };
      int win = cur.key_lo / p.bs;
      int id = load_id(win + lane);
      for (int i = 0; i < cur.n_kv[1]; ++i) {
        const int key0 = cur.key_lo + i * kKeys;
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
        if (!load_tile(&tm_k, cur.k, rc, false, mask) || !load_tile(&tm_v, cur.k, rc, true, 0)) break;
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(&ctl->info_empty[slot]);
    }
    if (lane == 0 && *abort) {
      // Gave up: let the copies already issued land before the CTA exits.
      for (int d = 1; d <= S && (int)n_loads - d >= 0; ++d) {
        const uint32_t n = n_loads - d;
        for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(&ctl->full[n % S], (n / S) & 1); ++i) {
        }
      }
    }
   } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // One lane, elected with elect.sync, runs the whole loop: it waits on
    // the barriers alone (a warp-wide wait and vote per barrier costs several
    // times more) and issues the tcgen05 instructions.
    constexpr uint32_t idesc_s = umma_idesc_f16(kPrefillRows, kKeys, 0, 0, BF ? 1 : 0);
    constexpr uint32_t idesc_o = umma_idesc_f16(kPrefillRows, D, 0, 1, BF ? 1 : 0);
    const uint64_t desc_k = smem_desc_sw128(0, 16, 1024);           // K-major Q and K, + (address >> 4)
    const uint64_t desc_v = smem_desc_sw128(0, kKeys * 128, 1024);  // MN-major V, + (address >> 4)
    const uint32_t kv_addr = smem_u32(kv_s);
    const bool leader = elect_one();
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) -> bool {
      return wait_or_abort(bar, parity, abort, p.err, p.err_site, kSitePrefillPair | 3);
    };
    uint32_t g = 0, pcnt[2] = {0, 0};
    bool ok = leader;
    for (uint32_t tt = 0; ok; ++tt) {
      const int slot = tt % kInfoRing;
      if (!wait_bar(&ctl->info_full[slot], (tt / kInfoRing) & 1)) break;
      const UnitInfo& ui = ctl->info[slot];
      if (ui.u < 0) break;
      const int nA = ui.n_kv[0], n_last = ui.n_kv[1];
      const uint32_t q_addr = smem_u32(q_s);
      // S_X(i) = Q_X K_i^T.  K_i is released after tile B's S, Q_X after
      // the unit's last S_X.
      auto issue_s = [&](int X, int i) -> bool {
        const uint32_t n = 2 * (g + i);
        const int st = n % S;
        if (i == 0 && !wait_bar(&ctl->q_full[X], tt & 1)) return false;
        // tile A's S(i) already waited for K_i (this thread, same phase)
        if ((X == 0 || i >= nA) && !wait_bar(&ctl->full[st], (n / S) & 1)) return false;
        tc_fence_after();
        const uint64_t a0 = desc_k + ((q_addr + X * C::kQTileBytes) >> 4);
        const uint64_t b0 = desc_k + ((kv_addr + st * C::kSlotBytes) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          umma_f16(tmem + C::s_col(X), a0 + (((ks >> 2) * (kPrefillRows * 128) + (ks & 3) * 32) >> 4),
                   b0 + (((ks >> 2) * (kKeys * 128) + (ks & 3) * 32) >> 4), idesc_s, ks > 0);
        umma_commit(&ctl->s_full[X]);
        if (X == 1) umma_commit(&ctl->empty[st]);
        if (i == (X ? n_last : nA) - 1) umma_commit(&ctl->q_empty[X]);
        return true;
      };
      // O_X += P_X(i) V_i with P_X read from TMEM (fp16 pairs over S_X).
      // V_i is released after tile B's PV.
      auto issue_pv = [&](int X, int i) -> bool {
        if (!wait_bar(&ctl->p_full[X], pcnt[X] & 1)) return false;
        ++pcnt[X];
        // the unit's first PV overwrites O_X: the epilogue has read the last unit's
        if (i == 0 && tt > 0 && !wait_bar(&ctl->o_free[X], (tt - 1) & 1)) return false;
        const uint32_t n = 2 * (g + i) + 1;
        const int st = n % S;
        if ((X == 0 || i >= nA) && !wait_bar(&ctl->full[st], (n / S) & 1)) return false;
        tc_fence_after();
        const uint64_t b0 = desc_v + ((kv_addr + st * C::kSlotBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          umma_f16_ts(tmem + C::o_col(X), tmem + C::s_col(X) + kk * 8, b0 + ((kk * 16 * 128) >> 4), idesc_o,
                      (i > 0 || kk > 0) ? 1u : 0u);
        if (X == 1) umma_commit(&ctl->empty[st]);
        return true;
      };
      if (!issue_s(0, 0) || !issue_s(1, 0)) break;
      for (int i = 0; i < n_last && ok; ++i) {
        if (i < nA) {
          if (!issue_pv(0, i)) { ok = false; break; }
          if (i == nA - 1) {
            umma_commit(&ctl->o_done[0]);
          } else if (!issue_s(0, i + 1)) {
            ok = false;
            break;
          }
        }
        if (!issue_pv(1, i)) { ok = false; break; }
        if (i == n_last - 1) {
          umma_commit(&ctl->o_done[1]);
        } else if (!issue_s(1, i + 1)) {
          ok = false;
          break;
        }
      }
      g += n_last;
      if (!ok) break;
      mbar_arrive(&ctl->info_empty[slot]);
    }
    // Drain: every MMA issued above has completed before TMEM is freed.
    if (leader) {
      umma_commit(&ctl->drain);
      for (uint32_t i = 0; i < kWaitLimit && !mbar_try_wait(&ctl->drain, 0); ++i) {
      }
    }
    __syncwarp();
   }
  } else if (warp < kEpiWarp0) {
    regs_inc<kRegSoftmax>();
    // ----------------------------------------------------- softmax warps
    const int X = warp >> 2;                  // 0: tile A, 1: tile B
    const int r = threadIdx.x & 127;          // query row == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float mul = CAP ? 1.f : p.scale * kLog2e;
    const float cap_in = CAP ? p.scale / p.softcap : 0.f;
    const float cap_out = CAP ? p.softcap * kLog2e : 0.f;
    uint32_t g = 0, scnt = 0;
    float x[kKeys];
    for (uint32_t tt = 0;; ++tt) {
      const int slot = tt % kInfoRing;
      if (!wait_or_abort(&ctl->info_full[slot], (tt / kInfoRing) & 1, abort, p.err, p.err_site, kSitePrefillPair | 4)) break;
      const UnitInfo& ui = ctl->info[slot];
      if (ui.u < 0) break;
      // The unit's fields, read once (shared-memory loads are slow while
      // the tensor core streams operands)
      const int j = r / p.G;
      const bool row_ok = j < ui.ntok[X];
      const int hi = ui.pos0 + X * tq + j;                   // last admitted position
      const int lo = p.window >= 1 ? hi + 1 - p.window : 0;  // first admitted position
      const int n_x = ui.n_kv[X];
      const int key_lo = ui.key_lo;
      // Tiles whose never-admitted keys need zero V rows: tile A does it
      // while it uses the tile, tile B for the tiles A skips.
      const int vz_from = X == 0 ? 0 : ui.n_kv[0];
      const int vz_kv_len = ui.kv_len, vz_lo_min = ui.lo_min;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int i = 0; i < n_x; ++i) {
        const uint32_t nv = 2 * (g + i) + 1, tile = g + i;
        const int sv = nv % S;
        const int key0 = key_lo + i * kKeys;
        // The page mask was published before the tile's K load: it is read
        // before the wait for S, which hides the shared-memory load (read
        // after it, the load stalled the diagonal tile's rows for ~1800
        // cycles while the next unit's Q tile streamed in).  s_full(i) also
        // covers PV(i-1): MMAs complete in issue order.
        if (!wait_or_abort(&ctl->mask_full[tile % kMaskRing], (tile / kMaskRing) & 1, abort, p.err, p.err_site,
                           kSitePrefillPair | 6)) {
          ok = false;
          break;
        }
        const uint32_t mask = ctl->kv_mask[tile % kMaskRing];
        if (!wait_or_abort(&ctl->s_full[X], scnt & 1, abort, p.err, p.err_site, kSitePrefillPair | 5)) {
          ok = false;
          break;
        }
        ++scnt;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kKeys; c += 32) tmem_ld32(lane_addr + C::s_col(X) + c, x + c);
        tmem_ld_wait();
        if constexpr (CAP) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) x[c] = cap_out * tanhf(x[c] * cap_in);
        }
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
        const float cand = max_tree<kKeys>(x) * mul;
        float alpha = 1.f;
        if (cand > m_ref + kLazyRescale || (m_ref == -INFINITY && cand != -INFINITY)) {
          alpha = m_ref == -INFINITY ? 0.f : ex2(m_ref - cand);
          m_ref = cand;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        const uint64_t mul2 = f2(mul, mul), neg_m2 = f2(-m_use, -m_use);
        uint64_t sum2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int h = 0; h < kKeys; h += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const uint64_t arg = fma2(f2(x[h + 2 * q], x[h + 2 * q + 1]), mul2, neg_m2);
            float a0, a1;
            unf2(arg, a0, a1);
            const float e0 = ex2(a0), e1 = ex2(a1);
            sum2[q & 3] = add2(sum2[q & 3], f2(e0, e1));
            pk[q] = pack2<BF>(e0, e1);
          }
          // P_X -> TMEM over S_X: keys h..h+31 as 16 columns of fp16 pairs
          tmem_st16(lane_addr + C::s_col(X) + h / 2, pk);
        }
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
        if (i >= vz_from && (key0 + kKeys > vz_kv_len || key0 < vz_lo_min)) {
          uint8_t* vs = kv_s + sv * C::kSlotBytes;
          if (!wait_or_abort(&ctl->full[sv], (nv / S) & 1, abort, p.err, p.err_site, kSitePrefillPair | 7)) {
            ok = false;
            break;
          }
          for (int idx = r; idx < kKeys * C::kChunks * 8; idx += 128) {
            const int kr = idx / (C::kChunks * 8), rem = idx % (C::kChunks * 8);
            const int pos = key0 + kr;
            if (pos >= vz_kv_len || pos < vz_lo_min) {
              const int c = rem >> 3, col16 = rem & 7;
              *reinterpret_cast<uint4*>(vs + c * (kKeys * 128) + kr * 128 + ((col16 ^ (kr & 7)) << 4)) =
                  make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[X]);
        // the row sum is off the path to the PV MMA
        float s0, s1, s2, s3;
        unf2(add2(sum2[0], sum2[1]), s0, s1);
        unf2(add2(sum2[2], sum2[3]), s2, s3);
        l = l * alpha + ((s0 + s1) + (s2 + s3));
      }
      if (!ok) break;
      // head_sink (section 6.1): one more denominator term, exp(s_h - m), in
      // log2 units relative to the row's reference maximum
      if (p.head_sink && m_ref != -INFINITY)
        l += ex2(elem16_to_float(p.head_sink[ui.k * p.G + (r - j * p.G)], BF) * kLog2e - m_ref);
      // The row sum goes to the epilogue warpgroup (its previous value has
      // been read once l_empty completes).
      if (!wait_or_abort(&ctl->l_empty[X], (tt & 1) ^ 1, abort, p.err, p.err_site, kSitePrefillPair | 8)) break;
      ctl->l_row[X][r] = l;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->l_full[X]);
      if (lane == 0) mbar_arrive(&ctl->info_empty[slot]);
      g += ui.n_kv[1];
    }
  } else {
    regs_dec<kRegEpilogue>();
    // ---------------------------------------------------------- epilogue
    // For each tile of the unit: O_X / l -> fp16 output rows.  O is read
    // from TMEM 32 columns at a time; after the last read it is released to
    // the next unit's first PV.
    const int r = threadIdx.x - kEpiWarp0 * 32;  // row == TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    uint32_t ocnt[2] = {0, 0};
    for (uint32_t tt = 0;; ++tt) {
      const int slot = tt % kInfoRing;
      if (!wait_or_abort(&ctl->info_full[slot], (tt / kInfoRing) & 1, abort, p.err, p.err_site, kSitePrefillPair | 9)) break;
      const UnitInfo& ui = ctl->info[slot];
      if (ui.u < 0) break;
      const int j = r / p.G;
      bool ok = true;
      for (int X = 0; X < 2 && ok; ++X) {
        if (!wait_or_abort(&ctl->o_done[X], ocnt[X] & 1, abort, p.err, p.err_site, kSitePrefillPair | 10) ||
            !wait_or_abort(&ctl->l_full[X], tt & 1, abort, p.err, p.err_site, kSitePrefillPair | 11)) {
          ok = false;
          break;
        }
        ++ocnt[X];
        tc_fence_after();
        const float l = ctl->l_row[X][r];
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->l_empty[X]);
        const bool row_ok = j < ui.ntok[X];
        const int t = ui.t0 + X * tq + j, h = ui.k * p.G + (r - j * p.G);
        __half* dst = p.out + ((size_t)t * p.H + h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(lane_addr + C::o_col(X) + 32 * c, o);
          tmem_ld_wait();
          if (c == D / 32 - 1) {
            // O_X is read: the next unit's first PV may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->o_free[X]);
          }
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
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->info_empty[slot]);
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
  static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");
  static_assert(PairCfg<D>::kSmemBytes <= kSmemLimit, "shared memory");
  static_assert(PairCfg<D>::kSlots >= 3, "K/V ring");
  static_assert(PairCfg<D>::kSlots / 2 + 2 <= kMaskRing, "page mask ring");
  static_assert(2 * kKeys + 2 * D <= PairCfg<D>::kTmemCols, "tensor memory");
  cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel<D, CAP, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)PairCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_pair_kernel<D, CAP, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)PairCfg<D>::kSmemBytes);
}

template <int D, bool BF>
cudaError_t launch_db(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                      int grid, cudaStream_t s) {
  if (p.softcap > 0.f)
    return launch_pdl(prefill_pair_kernel<D, true, BF>, grid, kThreads, PairCfg<D>::kSmemBytes, s, tq, tk, tv, p);
  return launch_pdl(prefill_pair_kernel<D, false, BF>, grid, kThreads, PairCfg<D>::kSmemBytes, s, tq, tk, tv, p);
}

template <int D>
cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                     int grid, cudaStream_t s) {
  return p.bf16 ? launch_db<D, true>(tq, tk, tv, p, grid, s) : launch_db<D, false>(tq, tk, tv, p, grid, s);
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
