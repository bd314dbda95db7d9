// Rotary + reshape_and_cache: one warp per packed token.
//
// Slot derivation is the derived-slot rule of "PagedAttention - CUDA Design
// Document", section 5.1 (owner sequence by binary search over
// cumulative_sequence_lengths, guarded against rows past cum[B] as section
// 18.2 asks; position past_b + j; block_table row position / block_size).
// A -1 block entry means "not mapped" (section 9.3.1): nothing is written.
// An explicit slot_mapping (section 5.2) replaces the derivation for the
// write (-1 = no write); the block table still defines what is read.
// K is rotated before it is stored (section 7.2 / 12.5: the cache holds the
// already-rotated K); Q is rotated into a workspace for the attention kernels.
//
// Rotary arithmetic is fixed so the pool is bit-reproducible: per pair,
//   y1 = rn(rn(x1*c) - rn(x2*s)),  y2 = rn(rn(x2*c) + rn(x1*s))
// in fp32 (no fused multiply-add), then fp16 round-to-nearest-even.  With
// bfloat16 activations (section 8.2) the inputs and tables are bfloat16,
// the same fp32 steps run and each y is rounded to bfloat16 (nearest-even);
// a 16-bit row that is not rotated is copied bit for bit either way.
//
// Every row moves as 16-byte vectors: the NHD pool stores a token's
// [Hk, D] slice contiguously, so a warp writes one contiguous run of
// Hk*D*2 bytes per tensor (fully coalesced).
//
// 8-bit caches (section 8.4, quantize as the rows are scattered): each fp16
// (or bfloat16) value x (after rotary) is stored as the code of y = x / scale, the
// division in fp32 (IEEE), rounded to nearest-even and saturated to
// [-128, 127] (int8) or to +-448 (e4m3fn); scale is k_scale / v_scale[0] or
// [k*D + c] per channel.  The query copy for attention is then multiplied by
// the K scale (fp32 product rounded to fp16), which folds the K
// dequantization into Q (section 8.5 phase 3).  With bfloat16 activations
// the rows are transformed in bfloat16 as for a bfloat16 cache and the
// query copy is written as fp16 (the score contraction over 8-bit codes
// takes fp16 operands).
//
// QK-Norm (section 7, before rotary; the normalized K is what is cached):
// each head's factor r = 1 / sqrt(sum x^2 / D + eps) takes its fp32 sum of
// squares as one running sum over the channels in ascending order (one
// lane per head, one rounding per square and per add, no fused
// multiply-add; IEEE square root and reciprocal), and every loaded channel
// becomes fp16((x * r) * w) (bfloat16 with bfloat16 activations).
// Packed QKV rows (section 4) are read in place: Q, K and V heads of token
// t start at t*(H+2Hk)*D, + H*D and + (H+Hk)*D.
#include <algorithm>
#include <type_traits>

#include "ptx.cuh"
#include "step.h"
#include "worklist.cuh"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kWarpsPerBlock = 4;

__device__ __forceinline__ void rotate_pair(__half x1, __half x2, __half c, __half s, __half& y1, __half& y2,
                                            bool bf16) {
  float fx1 = elem16_to_float(x1, bf16), fx2 = elem16_to_float(x2, bf16);
  float fc = elem16_to_float(c, bf16), fs = elem16_to_float(s, bf16);
  float a = __fsub_rn(__fmul_rn(fx1, fc), __fmul_rn(fx2, fs));
  float b = __fadd_rn(__fmul_rn(fx2, fc), __fmul_rn(fx1, fs));
  y1 = float_to_elem16(a, bf16);
  y2 = float_to_elem16(b, bf16);
}

union Vec8 {
  uint4 u;
  __half h[8];
};

// An ordinary (generic) load: this file reads no input through the
// read-only data cache (see the note at EmitCode).
template <typename T>
__device__ __forceinline__ T ld_plain(const T* ptr) {
  return *ptr;
}

// Emitters: where the eight fp16 values of channels [ch, ch + 8) of head h
// of a transformed row go.
struct EmitHalf {  // fp16 row
  __half* dst;
  int D;
  __device__ __forceinline__ void operator()(int h, int ch, const Vec8& v) const {
    *reinterpret_cast<uint4*>(dst + (size_t)h * D + ch) = v.u;
  }
};

// Code of the 16-bit value x (fp16, or bfloat16 bits when bf16).
__device__ __forceinline__ uint32_t code8(__half x, float s, int type, bool bf16) {
  const float y = __fdiv_rn(elem16_to_float(x, bf16), s);
  if (type == kCacheI8) {
    const int r = min(max(__float2int_rn(y), -128), 127);
    return (uint32_t)r & 0xffu;
  }
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(0.f), "f"(y));  // low byte <- y
  return c & 0xffu;
}

// (Every load of this file is an ordinary load (ld_plain) and every function
// and emitter is inlined into the kernels, the emitters passed by value, so
// that no address of a kernel parameter or of a local object reaches a
// load: two builds of the prologue whose rotated 8-bit K rows went through
// row_transform with read-only-cache loads and an emitter passed by
// reference stopped with cudaErrorInvalidAddressSpace, each reproducibly,
// while every input address was a device tensor in range.)
struct EmitCode {  // 8-bit codes; scale[0] or scale[(head0 + h) * D + c]
  uint8_t* dst;
  int D, type, per_channel, head0;
  const float* scale;
  bool bf16;  // the row holds bfloat16 activations
  __device__ __forceinline__ void operator()(int h, int ch, const Vec8& v) const {
    const float* sc = scale + (per_channel ? (size_t)(head0 + h) * D + ch : 0);
    uint32_t w[2] = {0, 0};
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e >> 2] |= code8(v.h[e], sc[per_channel ? e : 0], type, bf16) << (8 * (e & 3));
    *reinterpret_cast<uint2*>(dst + (size_t)h * D + ch) = make_uint2(w[0], w[1]);
  }
};

struct EmitScaledHalf {  // fp16 row times the K scale of its kv head (query heads head0 + h)
  __half* dst;
  int D, G, per_channel, head0;
  const float* scale;
  bool bf16;  // the row holds bfloat16 activations (the copy is fp16 all the same)
  __device__ __forceinline__ void operator()(int h, int ch, const Vec8& v) const {
    const float* sc = scale + (per_channel ? (size_t)((head0 + h) / G) * D + ch : 0);
    Vec8 y;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      y.h[e] = __float2half_rn(__fmul_rn(elem16_to_float(v.h[e], bf16), sc[per_channel ? e : 0]));
    *reinterpret_cast<uint4*>(dst + (size_t)h * D + ch) = y.u;
  }
};

// bfloat16 row stored as fp16 (the query copy of a bfloat16 step over an
// 8-bit cache, whose score contraction runs on fp16 operands): the
// conversion is exact for every bfloat16 value inside fp16's normal range.
struct EmitHalfOfBf16 {
  __half* dst;
  int D;
  __device__ __forceinline__ void operator()(int h, int ch, const Vec8& v) const {
    Vec8 y;
#pragma unroll
    for (int e = 0; e < 8; ++e) y.h[e] = __float2half_rn(elem16_to_float(v.h[e], true));
    *reinterpret_cast<uint4*>(dst + (size_t)h * D + ch) = y.u;
  }
};

// QK-Norm factors of the nheads (<= 32) heads of one row: lane h sums the
// squares of head h as one running fp32 sum in channel order (the order
// stated at the top of the file), then stores rn[h].  bf16: the row holds
// bfloat16.
__device__ __forceinline__ void norm_factors(const __half* src, int nheads, int D, float eps, float* rn, int lane,
                             bool bf16) {
  if (lane < nheads) {
    const __half* x = src + (size_t)lane * D;
    float acc = 0.f;
    for (int c = 0; c < D; c += 8) {
      Vec8 v;
      v.u = ld_plain(reinterpret_cast<const uint4*>(x + c));
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float f = elem16_to_float(v.h[e], bf16);
        acc = __fadd_rn(acc, __fmul_rn(f, f));
      }
    }
    const float mean = __fmul_rn(acc, 1.f / (float)D);
    rn[lane] = __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps)));
  }
  __syncwarp();
}

// Copies (rotate = false) or rotates one [nheads, D] row of src and hands
// every 8-channel group to `emit`.  With rn (QK-Norm factors per head) and
// nw (the [D] weight), every loaded value is first normalized.  R % 16 == 0
// is checked on the host.  Channels outside [keep_lo, keep_hi) that are not
// rotated are not emitted at all (a latent query's copy keeps only the
// 64-channel chunks that hold its rotated channels).  bf16: the row, the
// weight and the tables hold bfloat16.
template <typename Emit>
__device__ __forceinline__ void row_transform(const __half* src, const Emit emit, int nheads, int D, bool rotate,
                              int R, int interleaved, const __half* cos_row, const __half* sin_row, int lane,
                              const float* rn = nullptr, const __half* nw = nullptr, int off = 0, int keep_lo = 0,
                              int keep_hi = 1 << 30, bool bf16 = false) {
  const bool keep_all = keep_lo <= 0 && keep_hi >= D;
  const int chunks_per_head = D / 8;
  auto ld8 = [&](int h, int ch) -> Vec8 {
    Vec8 v;
    v.u = ld_plain(reinterpret_cast<const uint4*>(src + (size_t)h * D + ch));
    if (rn) {
      const float r = rn[h];
      Vec8 w;
      w.u = ld_plain(reinterpret_cast<const uint4*>(nw + ch));
#pragma unroll
      for (int e = 0; e < 8; ++e)
        v.h[e] = float_to_elem16(__fmul_rn(__fmul_rn(elem16_to_float(v.h[e], bf16), r), elem16_to_float(w.h[e], bf16)),
                                 bf16);
    }
    return v;
  };
  if (!rotate) {
    if constexpr (std::is_same<Emit, EmitHalf>::value) {
      if (!rn && keep_all) {  // plain copy of a contiguous [nheads, D] row
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(emit.dst);
        const int n = nheads * chunks_per_head;
        // Four loads per lane in flight before their stores: the source and
        // the pool are separate tensors, which the compiler cannot assume
        // for ordinary loads, so a load-store loop would wait on each load.
        for (int i0 = lane; i0 < n; i0 += 4 * 32) {
          uint4 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (i0 + 32 * k < n) v[k] = ld_plain(s4 + i0 + 32 * k);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (i0 + 32 * k < n) d4[i0 + 32 * k] = v[k];
        }
        return;
      }
    }
    for (int i = lane; i < nheads * chunks_per_head; i += 32) {
      const int h = i / chunks_per_head, ch = 8 * (i % chunks_per_head);
      if (ch >= keep_lo && ch < keep_hi) emit(h, ch, ld8(h, ch));
    }
    return;
  }
  const int half = R / 2;
  if (!interleaved) {
    // Pair chunks: channels off + [8c, 8c+8) with off + [half + 8c, half + 8c + 8);
    // the chunks outside [off, off + R) are copied.
    const int pairs = half / 8;
    const int copies = (D - R) / 8;
    const int per_head = pairs + copies;
    for (int i = lane; i < nheads * per_head; i += 32) {
      int h = i / per_head, c = i % per_head;
      if (c < pairs) {
        Vec8 a = ld8(h, off + 8 * c), b = ld8(h, off + half + 8 * c), cs, sn, ya, yb;
        cs.u = ld_plain(reinterpret_cast<const uint4*>(cos_row + 8 * c));
        sn.u = ld_plain(reinterpret_cast<const uint4*>(sin_row + 8 * c));
#pragma unroll
        for (int e = 0; e < 8; ++e) rotate_pair(a.h[e], b.h[e], cs.h[e], sn.h[e], ya.h[e], yb.h[e], bf16);
        emit(h, off + 8 * c, ya);
        emit(h, off + half + 8 * c, yb);
      } else {
        const int cc = 8 * (c - pairs);
        const int ch = cc < off ? cc : cc + R;
        if (ch >= keep_lo && ch < keep_hi) emit(h, ch, ld8(h, ch));
      }
    }
  } else {
    // Each 8-channel chunk of [off, off + R) holds four (2i, 2i+1) pairs.
    const int rchunks = R / 8, c0 = off / 8;
    for (int i = lane; i < nheads * chunks_per_head; i += 32) {
      int h = i / chunks_per_head, c = i % chunks_per_head;
      const bool rot = c >= c0 && c < c0 + rchunks;
      if (!rot && (8 * c < keep_lo || 8 * c >= keep_hi)) continue;
      Vec8 a = ld8(h, 8 * c), y;
      if (rot) {
        uint2 cu = ld_plain(reinterpret_cast<const uint2*>(cos_row + 4 * (c - c0)));
        uint2 su = ld_plain(reinterpret_cast<const uint2*>(sin_row + 4 * (c - c0)));
        const __half* cv = reinterpret_cast<const __half*>(&cu);
        const __half* sv = reinterpret_cast<const __half*>(&su);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          rotate_pair(a.h[2 * e], a.h[2 * e + 1], cv[e], sv[e], y.h[2 * e], y.h[2 * e + 1], bf16);
      } else {
        y.u = a.u;
      }
      emit(h, 8 * c, y);
    }
  }
}

// One warp's share of packed row t.  Part 0 writes the K (rotated) and V
// rows into the pool; parts 1.. rotate query heads [(part-1)*qh, part*qh)
// into the rotated-query workspace (only with rotary in pa_forward).  `cum`
// is the cumulative length array, either the caller's (global) or a
// shared-memory copy.
__device__ __forceinline__ void write_token(const CacheWriteParams& p, const int* cum, int t, int part, int lane, float* rn) {
  // Owner sequence: largest b with cum[b] <= t.
  int lo = 0, hi = p.batch;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (cum[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int b = lo;
  const int c0 = cum[b], c1 = cum[b + 1];
  const int past = ld_plain(p.past + b);
  if (t < c0 || t >= c1 || c0 < 0) {
    if (lane == 0 && part == 0) atomicOr(p.err, PA_DEVERR_CUM);
    return;
  }
  if (past < 0) {
    if (lane == 0 && part == 0) atomicOr(p.err, PA_DEVERR_PAST);
    return;
  }
  const int pos = past + (t - c0);
  bool rotate = p.rotary != 0;
  if (rotate && pos >= p.rot_positions) {
    if (lane == 0 && part == 0) atomicOr(p.err, PA_DEVERR_ROTARY_POS);
    rotate = false;  // never read past the tables
  }
  const int half = p.rot_dim / 2;
  const __half* cos_row = rotate ? p.cos_cache + (size_t)pos * half : nullptr;
  const __half* sin_row = rotate ? p.sin_cache + (size_t)pos * half : nullptr;

  // bfloat16 activations: a bfloat16 cache, or act_bf16 over an 8-bit one
  const bool abf = p.cache_type == kCacheBF16 || p.act_bf16;
  if (part >= p.kv_parts) {
    const int h0 = (part - p.kv_parts) * p.q_heads_per_part;
    const int nh = min(p.q_heads_per_part, p.H - h0);
    const __half* qsrc = p.query + (size_t)t * p.q_stride + (size_t)h0 * p.D;
    const size_t qoff = ((size_t)t * p.H + h0) * p.D;
    const float* qrn = nullptr;
    if (p.qk_norm) {
      norm_factors(qsrc, nh, p.D, p.qk_eps, rn, lane, abf);
      qrn = rn;
    }
    if (p.q_scale)
      row_transform(qsrc, EmitScaledHalf{p.q_rot + qoff, p.D, p.H / p.Hk, p.per_channel, h0, p.k_scale, abf},
                    nh, p.D, rotate, p.rot_dim, p.interleaved, cos_row, sin_row, lane, qrn, p.q_norm_w,
                    p.rot_offset, 0, 1 << 30, abf);
    else if (p.act_bf16)
      row_transform(qsrc, EmitHalfOfBf16{p.q_rot + qoff, p.D}, nh, p.D, rotate, p.rot_dim, p.interleaved,
                    cos_row, sin_row, lane, qrn, p.q_norm_w, p.rot_offset, 0, 1 << 30, true);
    else
      row_transform(qsrc, EmitHalf{p.q_rot + qoff, p.D}, nh, p.D, rotate, p.rot_dim, p.interleaved,
                    cos_row, sin_row, lane, qrn, p.q_norm_w, p.rot_offset, p.q_keep_lo, p.q_keep_hi,
                    p.cache_type == kCacheBF16);
    return;
  }

  size_t slot;
  if (p.slot_mapping) {
    // explicit slot (section 5.2): authoritative, -1 = no write
    const int s = ld_plain(p.slot_mapping + t);
    if (s == -1) return;
    if (s < -1 || (long long)s >= (long long)p.NB * p.bs) {
      if (lane == 0) atomicOr(p.err, PA_DEVERR_SLOT);
      return;
    }
    slot = (size_t)s;
  } else {
    const int row = pos / p.bs;
    if (row >= p.MB) {
      if (lane == 0) atomicOr(p.err, PA_DEVERR_KV_BOUND);
      return;
    }
    const int blk = ld_plain(p.block_table + (size_t)b * p.MB + row);
    if (blk == -1) return;  // not mapped: no write
    if (blk < -1 || blk >= p.NB) {
      if (lane == 0) atomicOr(p.err, PA_DEVERR_BLOCK_ID);
      return;
    }
    slot = (size_t)blk * p.bs + (pos & (p.bs - 1));
  }
  const size_t kv_row = (size_t)p.Hk * p.D;
  const __half* ksrc = p.packed ? p.query + (size_t)t * p.q_stride + (size_t)p.H * p.D : p.key + (size_t)t * kv_row;
  const __half* vsrc =
      p.packed ? p.query + (size_t)t * p.q_stride + (size_t)(p.H + p.Hk) * p.D : p.value + (size_t)t * kv_row;
  if (p.kv_parts > 1) {
    // 8-bit caches: part 2i quantizes K heads [i*hp, (i+1)*hp), part 2i+1
    // the same V heads (the per-element division spread over more warps)
    const int hp = p.kv_heads_per_part, h0 = (part >> 1) * hp, nh = min(hp, p.Hk - h0);
    if (nh <= 0) return;
    const size_t doff = slot * kv_row + (size_t)h0 * p.D;
    if ((part & 1) == 0) {
      const float* krn = nullptr;
      if (p.qk_norm) {
        norm_factors(ksrc + (size_t)h0 * p.D, nh, p.D, p.qk_eps, rn, lane, abf);
        krn = rn;
      }
      row_transform(ksrc + (size_t)h0 * p.D,
                    EmitCode{static_cast<uint8_t*>(p.key_cache) + doff, p.D, p.cache_type, p.per_channel, h0,
                             p.k_scale, abf},
                    nh, p.D, rotate, p.rot_dim, p.interleaved, cos_row, sin_row, lane, krn, p.k_norm_w,
                    p.rot_offset, 0, 1 << 30, abf);
    } else {
      row_transform(vsrc + (size_t)h0 * p.D,
                    EmitCode{static_cast<uint8_t*>(p.value_cache) + doff, p.D, p.cache_type, p.per_channel, h0,
                             p.v_scale, abf},
                    nh, p.D, false, 0, 0, nullptr, nullptr, lane);
    }
    return;
  }
  const float* krn = nullptr;
  if (p.qk_norm) {
    norm_factors(ksrc, p.Hk, p.D, p.qk_eps, rn, lane, abf);
    krn = rn;
  }
  if (p.cache_type == kCacheF16 || p.cache_type == kCacheBF16) {
    row_transform(ksrc, EmitHalf{static_cast<__half*>(p.key_cache) + slot * kv_row, p.D},
                  p.Hk, p.D, rotate, p.rot_dim, p.interleaved, cos_row, sin_row, lane, krn, p.k_norm_w,
                  p.rot_offset, 0, 1 << 30, p.cache_type == kCacheBF16);
    if (p.value_cache)  // none for a latent cache (V is part of the latent rows)
      row_transform(vsrc, EmitHalf{static_cast<__half*>(p.value_cache) + slot * kv_row, p.D}, p.Hk, p.D, false,
                    0, 0, nullptr, nullptr, lane);
  } else {
    row_transform(ksrc,
                  EmitCode{static_cast<uint8_t*>(p.key_cache) + slot * kv_row, p.D, p.cache_type, p.per_channel, 0,
                           p.k_scale, abf},
                  p.Hk, p.D, rotate, p.rot_dim, p.interleaved, cos_row, sin_row, lane, krn, p.k_norm_w,
                  p.rot_offset, 0, 1 << 30, abf);
    row_transform(vsrc,
                  EmitCode{static_cast<uint8_t*>(p.value_cache) + slot * kv_row, p.D, p.cache_type, p.per_channel, 0,
                           p.v_scale, abf},
                  p.Hk, p.D, false, 0, 0, nullptr, nullptr, lane);
  }
}

// Sequences whose cumulative lengths are staged in shared memory (one
// coalesced read instead of a chain of dependent global reads per token).
constexpr int kCumCache = 4096;

__device__ const int* stage_cum(const CacheWriteParams& p, int* cum_s) {
  if (p.batch + 1 > kCumCache) return p.cum;
  for (int i = threadIdx.x; i <= p.batch; i += blockDim.x) cum_s[i] = ld_plain(p.cum + i);
  __syncthreads();
  return cum_s;
}

// QK-Norm factors: one slot per head of a warp's row (kv_num_heads <= 32
// is checked on the host when QK-Norm is on).
constexpr int kMaxNormHeads = 32;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) cache_write_kernel(CacheWriteParams p) {
  __shared__ int cum_s[kCumCache];
  __shared__ float rn_s[kWarpsPerBlock][kMaxNormHeads];
  const int* cum = stage_cum(p, cum_s);
  const int w = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (w < p.token_count * p.parts)
    write_token(p, cum, w / p.parts, w % p.parts, threadIdx.x & 31, rn_s[threadIdx.x >> 5]);
}

// The step's prologue in one launch: CTA 0 builds the work list while the
// other CTAs (wpb writing warps each, one warp per (token, part)) rotate
// and write the new rows.  The two jobs read only the step's inputs, so
// they overlap.
constexpr int kPrologueWarps = worklist::kThreads / 32;  // at most this many writing warps per block

__global__ void __launch_bounds__(worklist::kThreads, 1) prologue_kernel(WorklistParams wp, CacheWriteParams cp,
                                                                         int wpb) {
  // Let the attention kernels' CTAs get resident early; they wait for this
  // grid's completion before reading anything it writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0) {
    worklist::build(wp);
    return;
  }
  __shared__ int cum_s[kCumCache];
  __shared__ float rn_s[kPrologueWarps][kMaxNormHeads];
  const int* cum = stage_cum(cp, cum_s);
  if ((threadIdx.x >> 5) >= wpb) return;  // wpb writing warps per block
  const int w = (blockIdx.x - 1) * wpb + (threadIdx.x >> 5);
  if (w < cp.token_count * cp.parts)
    write_token(cp, cum, w / cp.parts, w % cp.parts, threadIdx.x & 31, rn_s[threadIdx.x >> 5]);
}

}  // namespace

cudaError_t launch_cache_write(const CacheWriteParams& p, cudaStream_t s) {
  int blocks = (p.token_count * p.parts + kWarpsPerBlock - 1) / kWarpsPerBlock;
  cache_write_kernel<<<blocks, kWarpsPerBlock * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prologue(const WorklistParams& wp, const CacheWriteParams& cp, int num_sms, cudaStream_t s) {
  // Few warps per block while the warps fit the free SMs (their conversions
  // then run on separate SMs), up to 32 per block for large steps.
  const long long warps = (long long)cp.token_count * cp.parts;
  const int spread = std::max(1, num_sms - 1);
  const int wpb = (int)std::min<long long>(kPrologueWarps, std::max<long long>(1, (warps + spread - 1) / spread));
  const int blocks = 1 + (int)((warps + wpb - 1) / wpb);
  prologue_kernel<<<blocks, worklist::kThreads, 0, s>>>(wp, cp, wpb);
  return cudaGetLastError();
}

}  // namespace pa
