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
//  * persistent grid (a multiple of the SM count); CTAs stride over items;
//  * one producer warp streams 64-key stages of K and V through a ring of
//    shared-memory buffers with 3-D TMA boxes {64 ch, 1 head, rows} straight
//    from the NHD pool (one box per page and 64-channel chunk, 128-byte
//    swizzle), completion on mbarriers; unmapped pages are fetched from a
//    row past the pool so TMA zero-fills them without a memory read;
//  * four consumer warps each own 16 keys of every stage and run the two
//    contractions on tensor cores (m16n8k16 HMMA, fp16 in, fp32 accumulate):
//    S = Q K^T and O += P V, with an fp32 online softmax whose row max is
//    reduced with warp shuffles;
//  * at the end of an item the four warps' (m, l, O) are merged through the
//    last stage's buffer; a single-split sequence writes fp16 output
//    directly, otherwise fp32 partials go to the combine kernel.
#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kThreads = (kDecodeWarps + 1) * 32;  // 4 consumer warps + 1 producer warp
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecodeCfg {
  static constexpr int kChunks = D / 64;                       // 64-channel (128 B) chunks per row
  static constexpr int kTileBytes = kStageKeys * D * 2;        // K (or V) bytes per stage
  static constexpr int kStageBytes = 2 * kTileBytes;           // K + V
  static constexpr int kStages = (D == 256) ? 3 : (D == 128 ? 3 : 6);
  static constexpr int kQStride = D + 8;                       // padded Q row (halves)
  static constexpr int kQBytes = kDecodeRows * kQStride * 2;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kQBytes + 4 * 16 * 8 + kStages * 16 +
                                    2 * kStages * 8 + 64;
};

struct StageTag {
  int mask;  // bit i: box i of the stage was zero-filled (unmapped or past the end)
  int pad[3];
};

// Byte offset of 16-byte column `col16` of row `row` inside a 128B-swizzled
// [rows][128 B] tile whose base is 1024-byte aligned.
__device__ __forceinline__ uint32_t swz(int row, int col16) {
  return (uint32_t)(row * 128 + ((col16 ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeParams p) {
  using C = DecodeCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  __half* qs = reinterpret_cast<__half*>(smem + C::kStages * C::kStageBytes);
  float2* mls = reinterpret_cast<float2*>(smem + C::kStages * C::kStageBytes + C::kQBytes);
  StageTag* tags = reinterpret_cast<StageTag*>(mls + 4 * 16);
  uint64_t* full = reinterpret_cast<uint64_t*>(tags + C::kStages);
  uint64_t* empty = full + C::kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDecodeWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int n_work = p.counters->n_dec * p.Hk;
  const int split_keys = p.counters->split_keys;
  const int rows_per_box = p.bs < kStageKeys ? p.bs : kStageKeys;
  const int boxes = kStageKeys / rows_per_box;

  if (warp == kDecodeWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      int stage = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < n_work; u += gridDim.x) {
        const int item = u / p.Hk, k = u - item * p.Hk;
        const int2 bsplit = p.dec_items[item];
        const int b = bsplit.x;
        const SeqInfo si = p.seq[b];
        const int start = si.lo + bsplit.y * split_keys;
        const int end = min(si.kv_len, start + split_keys);
        for (int key0 = start; key0 < end; key0 += kStageKeys) {
          if (!mbar_wait(&empty[stage], phase ^ 1)) {
            atomicOr(p.err, PA_DEVERR_TIMEOUT);
            return;
          }
          int mask = 0;
          int rowc[kStageKeys / 16];
          for (int bx = 0; bx < boxes; ++bx) {
            const int pos = key0 + bx * rows_per_box;
            int rc = p.oob_row;
            if (pos < end) {
              const int blk = __ldg(p.block_table + (size_t)b * p.MB + pos / p.bs);
              if (blk >= 0 && blk < p.NB) {
                rc = blk * p.bs + (pos & (p.bs - 1));
              } else if (blk != -1) {
                atomicOr(p.err, PA_DEVERR_BLOCK_ID);
              }
            }
            if (rc == p.oob_row) mask |= 1 << bx;
            rowc[bx] = rc;
          }
          tags[stage].mask = mask;
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          uint8_t* kdst = stages + stage * C::kStageBytes;
          uint8_t* vdst = kdst + C::kTileBytes;
          for (int bx = 0; bx < boxes; ++bx) {
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              const uint32_t off = c * (kStageKeys * 128) + bx * rows_per_box * 128;
              tma_load_3d(kdst + off, &tm_k, c * 64, k, rowc[bx], &full[stage]);
              tma_load_3d(vdst + off, &tm_v, c * 64, k, rowc[bx], &full[stage]);
            }
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = threadIdx.x;  // 0..127
  const int r0 = lane >> 2, r1 = r0 + 8;
  const int cq = 2 * (lane & 3);
  int stage = 0;
  uint32_t phase = 0;
  const float scale = p.scale;
  const bool capped = p.softcap > 0.f;
  const float inv_cap = capped ? 1.f / p.softcap : 0.f;

  for (int u = blockIdx.x; u < n_work; u += gridDim.x) {
    const int item = u / p.Hk, k = u - item * p.Hk;
    const int2 bsplit = p.dec_items[item];
    const int b = bsplit.x;
    const SeqInfo si = p.seq[b];
    const int start = si.lo + bsplit.y * split_keys;
    const int end = min(si.kv_len, start + split_keys);
    const int R = si.q_len * p.G;
    const int past = si.kv_len - si.q_len;

    // Stage this item's query rows (16 x D, zero past R) into padded smem.
    for (int i = ctid; i < kDecodeRows * (D / 8); i += kDecodeWarps * 32) {
      const int r = i / (D / 8), c8 = i % (D / 8);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int t = si.t0 + r / p.G, h = k * p.G + r % p.G;
        v = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)t * p.H + h) * D + c8 * 8));
      }
      *reinterpret_cast<uint4*>(qs + r * C::kQStride + c8 * 8) = v;
    }
    named_bar(1, kDecodeWarps * 32);

    uint32_t qf[(D <= 128) ? D / 16 : 1][4];
    if constexpr (D <= 128) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int mi = lane >> 3, ri = lane & 7;
        const int row = (mi & 1) * 8 + ri, col = ks * 16 + (mi >> 1) * 8;
        ldsm_x4(smem_u32(qs + row * C::kQStride + col), qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3]);
      }
    }

    // Per-row causal and window bounds (rows beyond R admit nothing).
    int hi0 = -1, hi1 = -1, lo0 = 0, lo1 = 0;
    if (r0 < R) {
      hi0 = past + r0 / p.G;  // last admitted position
      lo0 = p.window >= 1 ? max(0, hi0 + 1 - p.window) : 0;
    }
    if (r1 < R) {
      hi1 = past + r1 / p.G;
      lo1 = p.window >= 1 ? max(0, hi1 + 1 - p.window) : 0;
    }
    // Keys outside [lo_min, kv_len) are never admitted by any row; their V
    // rows are zeroed in shared memory before use so stale bytes (e.g. NaN
    // in a partly filled last block) cannot leak through a zero weight.
    const int lo_min = p.window >= 1 ? max(0, past + 1 - p.window) : 0;

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    int last_stage = stage;
    for (int key0 = start; key0 < end; key0 += kStageKeys) {
      if (!mbar_wait(&full[stage], phase)) {
        if (lane == 0) atomicOr(p.err, PA_DEVERR_TIMEOUT);
        return;
      }
      const int mask = tags[stage].mask;
      uint8_t* kt = stages + stage * C::kStageBytes;
      uint8_t* vt = kt + C::kTileBytes;
      const int kw = key0 + warp * 16;  // first key position of this warp

      // Zero V rows of never-admitted keys among this warp's 16.
      const bool edge = (kw + 16 > si.kv_len) || (kw < lo_min);
      if (edge) {
        for (int i = lane; i < 16 * C::kChunks * 8; i += 32) {
          const int kr = i / (C::kChunks * 8), rem = i % (C::kChunks * 8);
          const int pos = kw + kr;
          if (pos >= si.kv_len || pos < lo_min) {
            const int c = rem >> 3, col16 = rem & 7;
            *reinterpret_cast<uint4*>(vt + c * (kStageKeys * 128) + (warp * 16 + kr) * 128 + col16 * 16) =
                make_uint4(0, 0, 0, 0);
          }
        }
        __syncwarp();
      }

      if (kw < end && kw + 16 > lo_min) {
        // ---- S = Q K^T for 16 rows x 16 keys
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          uint32_t a[4];
          if constexpr (D <= 128) {
            a[0] = qf[ks][0]; a[1] = qf[ks][1]; a[2] = qf[ks][2]; a[3] = qf[ks][3];
          } else {
            const int mi = lane >> 3, ri = lane & 7;
            const int row = (mi & 1) * 8 + ri, col = ks * 16 + (mi >> 1) * 8;
            ldsm_x4(smem_u32(qs + row * C::kQStride + col), a[0], a[1], a[2], a[3]);
          }
          const int mi = lane >> 3, ri = lane & 7;
          const int key = warp * 16 + (mi >> 1) * 8 + ri;
          const int d16 = ks * 16 + (mi & 1) * 8;
          const uint32_t addr = smem_u32(kt + (d16 >> 6) * (kStageKeys * 128) + swz(key, (d16 & 63) >> 3));
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          hmma16816(s[0], a, b0, b1);
          hmma16816(s[1], a, b2, b3);
        }
        // ---- scale, softcap, mask; row max
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int pos = kw + nt * 8 + cq + (e & 1);
            const int hi = (e < 2) ? hi0 : hi1;
            const int lo = (e < 2) ? lo0 : lo1;
            const int box = (pos - key0) / rows_per_box;
            const bool ok = pos < end && pos <= hi && pos >= lo && !((mask >> box) & 1);
            float x = s[nt][e] * scale;
            if (capped) x = p.softcap * tanhf(x * inv_cap);
            x *= kLog2e;
            x = ok ? x : -INFINITY;
            s[nt][e] = x;
            tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
          }
        }
        float alpha[2], muse[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
          tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
          const float mn = fmaxf(m[i], tmax[i]);
          muse[i] = (mn == -INFINITY) ? 0.f : mn;
          alpha[i] = exp2f(m[i] - muse[i]);
          m[i] = mn;
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
        }
        l[0] = l[0] * alpha[0] + rs[0];
        l[1] = l[1] * alpha[1] + rs[1];
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
          o[i][0] *= alpha[0];
          o[i][1] *= alpha[0];
          o[i][2] *= alpha[1];
          o[i][3] *= alpha[1];
        }
        uint32_t pa[4];
        pa[0] = pack_half2(s[0][0], s[0][1]);
        pa[1] = pack_half2(s[0][2], s[0][3]);
        pa[2] = pack_half2(s[1][0], s[1][1]);
        pa[3] = pack_half2(s[1][2], s[1][3]);
        // ---- O += P V
#pragma unroll
        for (int nd = 0; nd < D / 16; ++nd) {
          const int mi = lane >> 3, ri = lane & 7;
          const int key = warp * 16 + (mi & 1) * 8 + ri;
          const int d = nd * 16 + (mi >> 1) * 8;
          const uint32_t addr = smem_u32(vt + (d >> 6) * (kStageKeys * 128) + swz(key, (d & 63) >> 3));
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          hmma16816(o[2 * nd], pa, b0, b1);
          hmma16816(o[2 * nd + 1], pa, b2, b3);
        }
      }
      last_stage = stage;
      const bool last = key0 + kStageKeys >= end;
      if (!last) {
        if (edge) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
      }
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1;
      }
    }

    // ---- merge the four warps through the last stage's buffer
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
      l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
    }
    named_bar(1, kDecodeWarps * 32);  // every warp is done reading the stage
    float* mrg = reinterpret_cast<float*>(stages + last_stage * C::kStageBytes);
    float* mw = mrg + warp * 16 * D;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      const int d = i * 8 + cq;
      *reinterpret_cast<float2*>(mw + r0 * D + d) = make_float2(o[i][0], o[i][1]);
      *reinterpret_cast<float2*>(mw + r1 * D + d) = make_float2(o[i][2], o[i][3]);
    }
    if ((lane & 3) == 0) {
      mls[warp * 16 + r0] = make_float2(m[0], l[0]);
      mls[warp * 16 + r1] = make_float2(m[1], l[1]);
    }
    named_bar(1, kDecodeWarps * 32);
    const int nsplit = si.dec_count;
    for (int e = ctid; e < R * D; e += kDecodeWarps * 32) {
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
          acc += f * mrg[(w * 16 + r) * D + d];
        }
      }
      if (nsplit == 1) {
        const int t = si.t0 + r / p.G, h = k * p.G + r % p.G;
        p.out[((size_t)t * p.H + h) * D + d] = __float2half_rn(den > 0.f ? acc / den : 0.f);
      } else {
        const size_t row = (size_t)u * kDecodeRows + r;
        p.part_o[row * D + d] = acc;
        if (d == 0) p.part_ml[row] = make_float2(M, den);
      }
    }
    fence_proxy_async_smem();
    named_bar(1, kDecodeWarps * 32);
    if (lane == 0) mbar_arrive(&empty[last_stage]);
  }
}

template <int D>
cudaError_t configure_d(size_t* smem) {
  *smem = DecodeCfg<D>::kSmemBytes;
  return cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)DecodeCfg<D>::kSmemBytes);
}

}  // namespace

cudaError_t decode_configure(int head_size, int* ctas_per_sm, size_t* smem) {
  cudaError_t e;
  switch (head_size) {
    case 64: e = configure_d<64>(smem); break;
    case 128: e = configure_d<128>(smem); break;
    case 256: e = configure_d<256>(smem); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  int n = 0;
  switch (head_size) {
    case 64: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<64>, kThreads, *smem); break;
    case 128: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<128>, kThreads, *smem); break;
    default: e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<256>, kThreads, *smem); break;
  }
  *ctas_per_sm = n > 0 ? n : 1;
  return e;
}

cudaError_t launch_decode(int head_size, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                          int grid, cudaStream_t s) {
  switch (head_size) {
    case 64: decode_kernel<64><<<grid, kThreads, DecodeCfg<64>::kSmemBytes, s>>>(tk, tv, p); break;
    case 128: decode_kernel<128><<<grid, kThreads, DecodeCfg<128>::kSmemBytes, s>>>(tk, tv, p); break;
    case 256: decode_kernel<256><<<grid, kThreads, DecodeCfg<256>::kSmemBytes, s>>>(tk, tv, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace pa
