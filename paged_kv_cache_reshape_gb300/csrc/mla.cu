// Multi-head latent attention decode over one latent cache: the absorbed
// form of "PagedAttention - CUDA Design Document", section 12 (one kv head
// shared by every query head, key rows of D = 576 latent channels, V = the
// first DV = 512 channels of the same rows, an explicit softmax scale), with
// the masks of section 8 implementation note P5 (causal bound, window,
// softcap, -1 block entries masked).
//
// One work item = (sequence, split of its keys, group of 32 query heads of
// its one new token).  Design for sm_103a:
//  * a producer warp takes items from the device queue, loads the group's
//    32 query rows (two 16-row TMA boxes per 64-channel chunk) and streams
//    64-key stages of latent rows through a 2-deep ring (4-D pool view, one
//    box per page); each stage is read once and serves as both K and V for
//    all 32 heads;
//  * two consumer warpgroups, one per 16 heads, each of four warps: S = Q K^T
//    is split by keys (16 keys per warp, 36 m16n8k16 steps over 576
//    channels, spread over independent accumulators); the row maximum of the
//    stage is combined through shared memory, so the group's warps share one
//    running maximum (lazy rescale by 2^8); P goes to shared memory as fp16;
//    O += P V is split by channels (128 of the 512 per warp, all 64 keys),
//    which keeps each warp's accumulator at 64 registers; the two
//    warpgroups synchronise only through the stage ring;
//  * a single-split item writes fp16 output rows; otherwise fp32 partials
//    and (max, sum) go to the combine kernel, laid out like the decode
//    kernel's (16 rows per item and 16-head group).
#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kD = 576, kDV = 512;
constexpr int kChunks = kD / 64;                 // 9 chunks of 64 channels (128 B)
constexpr int kKeys = 64;                        // keys per stage
constexpr int kStages = 2;
constexpr int kTileBytes = kKeys * kD * 2;       // 72 KB
constexpr int kQBytes = kChunks * 4096;          // per chunk: two 16-row boxes of 128 B rows
constexpr int kPBytes = 16 * kKeys * 2;          // P [16 rows][64 keys] fp16, 128-byte rows, per warpgroup
constexpr int kGroupWarps = 4;                   // consumer warps of one 16-head warpgroup
constexpr int kWarps = 2 * kGroupWarps;          // consumer warps
// 12 warps: the two consumer warpgroups and a control warpgroup whose first
// warp is the producer (registers are allocated per warpgroup, so a ninth
// warp costs a fourth of the file anyway; the split gives it back).
constexpr int kThreads = 3 * 128;
#ifndef MLA_REG_CONTROL
#define MLA_REG_CONTROL 40
#endif
constexpr int kRegControl = MLA_REG_CONTROL;
constexpr int kRegConsumer = (65536 / kThreads / 8 * 8 * 3 - kRegControl) / 2 / 8 * 8;
static_assert(2 * kRegConsumer + kRegControl <= 3 * (65536 / kThreads / 8 * 8), "register split");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazyRescale = 8.f;
constexpr int kFirst = 1 << 8, kLast = 1 << 9;
#ifndef MLA_S_CHAINS
#define MLA_S_CHAINS 4  // independent accumulator pairs of S = Q K^T (divides 36)
#endif
static_assert((kD / 16) % MLA_S_CHAINS == 0, "chains divide the k-steps");

struct Tag {
  int u;       // item * (32-head groups) + group; -1 = no more work
  int key0, end, flags;
  int past, t0, hg, kv_len;
  int nsplit, qi, lo_min;
  int part;    // split-partial slot of this split, -1 for an unsplit entry
};

constexpr int kSmemBytes = 1024 + kStages * kTileBytes + 2 * kQBytes + 2 * kPBytes + 2 * kWarps * 16 * 4 +
                           kStages * (int)sizeof(Tag) + (2 * kStages + 4) * 8;

__device__ __forceinline__ uint32_t swz(int row, int col16) {
  return (uint32_t)(row * 128 + ((col16 ^ (row & 7)) << 4));
}

// Stage layout [box][chunk][row][128 B] (box = 2^log_r pool rows).
__device__ __forceinline__ uint32_t tile_off(int kk, int chunk, int col16, int log_r) {
  const int r = kk & ((1 << log_r) - 1), bx = kk >> log_r;
  return ((uint32_t)(bx * kChunks + chunk) << (log_r + 7)) + swz(r, col16);
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_l, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_qr,
                      const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* qbuf = stages + kStages * kTileBytes;  // [2][kQBytes]
  uint8_t* pbuf = qbuf + 2 * kQBytes;             // [warpgroup][16][128 B], swizzled
  float* red_m = reinterpret_cast<float*>(pbuf + 2 * kPBytes);  // [warp][16]
  float* red_l = red_m + kWarps * 16;                       // [warp][16]
  Tag* tags = reinterpret_cast<Tag*>(red_l + kWarps * 16);
  uint64_t* full = reinterpret_cast<uint64_t*>(tags + kStages);
  uint64_t* empty = full + kStages;
  uint64_t* q_full = empty + kStages;
  uint64_t* q_empty = q_full + 2;

  griddep_wait();  // the work list and the pool come from the prologue
  const int groups32 = mla_item_groups(p.groups);  // 32-head groups of a work item
  const int n_work = p.counters->n_dec * groups32;
  const int active = min(p.counters->dec_ctas, n_work);
  if ((int)blockIdx.x >= active) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], kWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp >= kWarps) {
    regs_dec<kRegControl>();
    if (warp > kWarps) return;
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_l);
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_qr);
    }
    const int split_keys = p.counters->split_keys;
    const int boxes = kKeys >> p.log_box_rows;
    int stage = 0;
    uint32_t phase = 0;
    int quse[2] = {0, 0};
    int qi = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
      int u = blockIdx.x;
      if (it > 0 && lane == 0) u = active + atomicAdd(&p.counters->dec_next, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u >= n_work) {
        if (lane == 0) {
          if (mbar_wait(&empty[stage], phase ^ 1)) {
            tags[stage].u = -1;
            mbar_arrive(&full[stage]);
          } else {
            note_timeout(p.err, p.err_site, kSiteMla | 1);
          }
        }
        break;
      }
      const int item = u / groups32, hg = u - item * groups32;
      const int2 bsplit = p.dec_items[item];  // (decode entry, split)
      const SeqInfo si = p.seq[bsplit.x];
      const int b = si.b;                      // the entry's sequence: its block_table row
      const int start = si.lo + bsplit.y * split_keys;
      const int end = min(si.kv_len, start + split_keys);
      const int past = si.kv_len - si.q_len;
      const int lo_min = p.window >= 1 ? max(0, past + 1 - p.window) : 0;
      if (lane == 0) {
        if (!mbar_wait(&q_empty[qi], (quse[qi] & 1) ^ 1)) {
          note_timeout(p.err, p.err_site, kSiteMla | 2);
          ok = false;
        } else {
          mbar_arrive_expect_tx(&q_full[qi], kQBytes);
          for (int c = 0; c < kChunks; ++c)
            for (int w = 0; w < 2; ++w)  // rows past H (a group beyond the heads) read as zeros
              tma_load_3d(qbuf + qi * kQBytes + c * 4096 + w * 2048, c >= p.qr_lo && c < p.qr_hi ? &tm_qr : &tm_q,
                          c * 64, hg * 32 + w * 16, si.t0,
                          &q_full[qi]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      quse[qi]++;
      const int* bt_row = p.block_table + (size_t)b * p.MB;
      auto load_id = [&](int r) -> int { return (r < p.MB && r * p.bs < end) ? __ldg(bt_row + r) : -1; };
      int win = start / p.bs;
      int id_cur = load_id(win + lane);
      int id_nxt = load_id(win + 32 + lane);
      for (int key0 = start; key0 < end; key0 += kKeys) {
        const int rowA = key0 / p.bs;
        if (rowA >= win + 32) {
          win += 32;
          id_cur = id_nxt;
          id_nxt = load_id(win + 32 + lane);
        }
        const int pos = key0 + (lane << p.log_box_rows);  // lane = box of the stage
        const int idx = pos / p.bs - win;
        const int a = __shfl_sync(0xffffffffu, id_cur, idx & 31);
        const int n = __shfl_sync(0xffffffffu, id_nxt, idx & 31);
        const int blk = idx < 32 ? a : n;
        int rc = p.oob_row;
        if (lane < boxes && pos < end) {
          if (blk >= 0 && blk < p.NB) rc = blk * p.bs + (pos & (p.bs - 1));
          else if (blk != -1) atomicOr(p.err, PA_DEVERR_BLOCK_ID);
        }
        const unsigned mask = __ballot_sync(0xffffffffu, lane < boxes && rc == p.oob_row);
        if (lane == 0) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            note_timeout(p.err, p.err_site, kSiteMla | 3);
            ok = false;
          } else {
            Tag& t = tags[stage];
            t.u = u;
            t.key0 = key0;
            t.end = end;
            t.flags = (int)(mask & 0xff) | (key0 == start ? kFirst : 0) | (key0 + kKeys >= end ? kLast : 0);
            t.past = past;
            t.t0 = si.t0;
            t.hg = hg;
            t.kv_len = si.kv_len;
            t.nsplit = si.dec_count;
            t.qi = qi;
            t.lo_min = lo_min;
            t.part = si.part_first >= 0 ? si.part_first + bsplit.y : -1;
            mbar_arrive_expect_tx(&full[stage], kTileBytes);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane < boxes)
          tma_load_4d(stages + stage * kTileBytes + ((uint32_t)lane * kChunks << (p.log_box_rows + 7)), &tm_l, 0,
                      rc, 0, 0, &full[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      qi ^= 1;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  regs_inc<kRegConsumer>();
  const int wg = warp / kGroupWarps, wi = warp % kGroupWarps;  // warpgroup (16 heads), warp in it
  const int bar_id = 1 + wg;
  uint8_t* pg = pbuf + wg * kPBytes;
  const int r0 = lane >> 2, r1 = r0 + 8;
  const int cq = 2 * (lane & 3);
  const int mi = lane >> 3, ri = lane & 7;
  const int log_r = p.log_box_rows;
  const bool capped = p.softcap > 0.f;
  const float inv_cap = capped ? 1.f / p.softcap : 0.f;
  int stage = 0;
  uint32_t phase = 0;
  int quse[2] = {0, 0};
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[16][4];
  const uint8_t* qcur = qbuf;
  while (true) {
    if (!mbar_wait(&full[stage], phase)) {
      if (lane == 0) note_timeout(p.err, p.err_site, kSiteMla | 4);
      return;
    }
    const Tag tg = tags[stage];
    if (tg.u < 0) break;
    if (tg.flags & kFirst) {
      if (!mbar_wait(&q_full[tg.qi], quse[tg.qi] & 1)) {
        if (lane == 0) note_timeout(p.err, p.err_site, kSiteMla | 5);
        return;
      }
      quse[tg.qi]++;
      qcur = qbuf + tg.qi * kQBytes + wg * 2048;
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    }
    const uint8_t* kt = stages + stage * kTileBytes;
    const int key0 = tg.key0, mask = tg.flags & 0xff;
    const int kw = key0 + wi * 16;
    // Keys outside [lo_min, kv_len): zero their rows (V is read by every warp;
    // warp wi of both warpgroups zeroes the same rows, with the same zeros).
    if (kw + 16 > tg.kv_len || kw < tg.lo_min) {
      for (int i = lane; i < 16 * kChunks * 8; i += 32) {
        const int kr = i / (kChunks * 8), rem = i % (kChunks * 8);
        const int pos = kw + kr;
        if (pos >= tg.kv_len || pos < tg.lo_min)
          *reinterpret_cast<uint4*>(const_cast<uint8_t*>(kt) + tile_off(wi * 16 + kr, rem >> 3, rem & 7, log_r)) =
              make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    // ---- S = Q K^T for 16 rows x this warp's 16 keys, the 36 k-steps spread
    // over kChains independent accumulator pairs (summed at the end) so that
    // consecutive MMAs do not wait on each other's results
    constexpr int kChains = MLA_S_CHAINS;
    float sc[kChains][2][4];
#pragma unroll
    for (int c = 0; c < kChains; ++c)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[c][0][e] = sc[c][1][e] = 0.f;
#pragma unroll 2
    for (int ks0 = 0; ks0 < kD / 16; ks0 += kChains) {
#pragma unroll
      for (int c = 0; c < kChains; ++c) {
        const int ks = ks0 + c;
        uint32_t a[4], b0, b1, b2, b3;
        const int row = (mi & 1) * 8 + ri, col = ks * 16 + (mi >> 1) * 8;
        ldsm_x4(smem_u32(qcur + (col >> 6) * 4096 + swz(row, (col & 63) >> 3)), a[0], a[1], a[2], a[3]);
        const int key = wi * 16 + (mi >> 1) * 8 + ri;
        const int d16 = ks * 16 + (mi & 1) * 8;
        ldsm_x4(smem_u32(kt + tile_off(key, d16 >> 6, (d16 & 63) >> 3, log_r)), b0, b1, b2, b3);
        hmma16816(sc[c][0], a, b0, b1);
        hmma16816(sc[c][1], a, b2, b3);
      }
    }
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float t = sc[0][nt][e];
#pragma unroll
        for (int c = 1; c < kChains; ++c) t += sc[c][nt][e];
        s[nt][e] = t;
      }
    // ---- mask (causal / window / unmapped page), scale, softcap; stage row max
    const int hi = tg.past;  // the token's position: the last admitted key
    const int lo = p.window >= 1 ? max(0, hi + 1 - p.window) : 0;
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int pos = kw + nt * 8 + cq + (e & 1);
        const int box = (pos - key0) >> log_r;
        const bool ok = pos < tg.end && pos <= hi && pos >= lo && !((mask >> box) & 1);
        float x = s[nt][e] * p.scale;
        if (capped) x = p.softcap * tanhf(x * inv_cap);
        x = ok ? x * kLog2e : -INFINITY;
        s[nt][e] = x;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
      tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
    }
    if ((lane & 3) == 0) {
      red_m[warp * 16 + r0] = tmax[0];
      red_m[warp * 16 + r1] = tmax[1];
    }
    named_bar(bar_id, kGroupWarps * 32);  // the group's maxima are in; its warps are past the last PV
    float alpha[2], muse[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = i ? r1 : r0;
      float t = red_m[wg * kGroupWarps * 16 + r];
#pragma unroll
      for (int w = 1; w < kGroupWarps; ++w) t = fmaxf(t, red_m[(wg * kGroupWarps + w) * 16 + r]);
      alpha[i] = 1.f;
      if (t > m[i] + kLazyRescale) {
        alpha[i] = (m[i] == -INFINITY) ? 0.f : exp2f(m[i] - t);
        m[i] = t;
      }
      muse[i] = (m[i] == -INFINITY) ? 0.f : m[i];
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = exp2f(s[nt][e] - muse[e >> 1]);
        s[nt][e] = pv;
        rs[e >> 1] += pv;
      }
      // P rows r0 / r1, keys wi*16 + nt*8 + cq, +1
      const int key = wi * 16 + nt * 8 + cq;
      *reinterpret_cast<uint32_t*>(pg + swz(r0, key >> 3) + (key & 7) * 2) = pack_half2(s[nt][0], s[nt][1]);
      *reinterpret_cast<uint32_t*>(pg + swz(r1, key >> 3) + (key & 7) * 2) = pack_half2(s[nt][2], s[nt][3]);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 1);
      rs[i] += __shfl_xor_sync(0xffffffffu, rs[i], 2);
      l[i] = l[i] * alpha[i] + rs[i];
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= alpha[0];
        o[i][1] *= alpha[0];
        o[i][2] *= alpha[1];
        o[i][3] *= alpha[1];
      }
    }
    named_bar(bar_id, kGroupWarps * 32);  // P and the zeroed V rows are visible to the group's warps
    // ---- O[:, 128*wi .. +128) += P V over the stage's 64 keys
#pragma unroll
    for (int ks = 0; ks < kKeys / 16; ++ks) {
      uint32_t a[4];
      const int row = (mi & 1) * 8 + ri, col = ks * 16 + (mi >> 1) * 8;
      ldsm_x4(smem_u32(pg + swz(row, col >> 3)), a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int nd = 0; nd < 8; ++nd) {
        const int key = ks * 16 + (mi & 1) * 8 + ri;
        const int d = wi * 128 + nd * 16 + (mi >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(kt + tile_off(key, d >> 6, (d & 63) >> 3, log_r)), b0, b1, b2, b3);
        hmma16816(o[2 * nd], a, b0, b1);
        hmma16816(o[2 * nd + 1], a, b2, b3);
      }
    }
    fence_proxy_async_smem();  // zeroed rows were written through the generic proxy
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);

    if (tg.flags & kLast) {
      // ---- end of item: row sums over the warps, output or partials
      if ((lane & 3) == 0) {
        red_l[warp * 16 + r0] = l[0];
        red_l[warp * 16 + r1] = l[1];
      }
      named_bar(bar_id, kGroupWarps * 32);
      float lt[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int r = i ? r1 : r0;
        lt[i] = 0.f;
#pragma unroll
        for (int w = 0; w < kGroupWarps; ++w) lt[i] += red_l[(wg * kGroupWarps + w) * 16 + r];
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = i ? r1 : r0;
        const int h = tg.hg * 32 + wg * 16 + row;
        if (h >= p.H) continue;
        if (tg.nsplit == 1) {
          const float inv = lt[i] > 0.f ? 1.f / lt[i] : 0.f;
          __half* dst = p.out + ((size_t)tg.t0 * p.H + h) * kDV + wi * 128 + cq;
#pragma unroll
          for (int nd = 0; nd < 16; ++nd)
            *reinterpret_cast<uint32_t*>(dst + nd * 8) = pack_half2(o[nd][2 * i] * inv, o[nd][2 * i + 1] * inv);
        } else {
          // partial rows of 16-head group 2 * hg + wg (h < H keeps it < groups)
          const size_t prow = ((size_t)tg.part * p.groups + tg.hg * 2 + wg) * kDecodeRows + row;
          float* dst = p.part_o + prow * kDV + wi * 128 + cq;
#pragma unroll
          for (int nd = 0; nd < 16; ++nd)
            *reinterpret_cast<float2*>(dst + nd * 8) = make_float2(o[nd][2 * i], o[nd][2 * i + 1]);
          if (wi == 0 && (lane & 3) == 0) p.part_ml[prow] = make_float2(m[i], lt[i]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_empty[tg.qi]);
    }
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1;
    }
  }
}

}  // namespace

cudaError_t mla_configure(size_t* smem) {
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  *smem = kSmemBytes;
  return cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_mla_decode(const CUtensorMap& tl, const CUtensorMap& tq, const CUtensorMap& tqr, const MlaParams& p,
                              int grid, cudaStream_t s) {
  return launch_pdl(mla_decode_kernel, grid, kThreads, kSmemBytes, s, tl, tq, tqr, p);
}

}  // namespace pa
