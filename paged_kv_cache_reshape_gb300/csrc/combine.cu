// Log-sum-exp merge of split-KV partials (flash decoding phase 2):
//   M = max_s m_s,  out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
// with O_s the unnormalised partial output and l_s its softmax sum, skipping
// empty splits (l_s = 0, m_s = -inf).  This is the merge of the CPU GQA notes
// (onnxruntime 1.27.0 docs, contrib_ops/cpu/gqa, "Flash Decoding" phase 2)
// and of PagedDecodeReduce ("PagedAttention - CUDA Design Document", section
// 8 implementation note P5).  Maxima are kept in log2 units by the decode
// kernel, hence base-2 exponentials.  A row whose splits are all empty
// outputs 0.  With head_sink (same CUDA design, section 6.1) the row's
// denominator also gets exp(s_h - M), the sink in log2 units.  BF: the
// sink and the output are bfloat16 (bfloat16 activations, section 8.2).
//
// One warp per (packed row, query head); the work list holds only the rows
// of sequences that were split, so the grid is a small persistent one.
#include "ptx.cuh"
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2eC = 1.4426950408889634f;

// Adds f * (the kPer floats at po) into acc, in 16-byte loads when kPer
// is a multiple of 4.
template <int kPer>
__device__ __forceinline__ void axpy(float* acc, float f, const float* po) {
  if constexpr (kPer % 4 == 0) {
#pragma unroll
    for (int i = 0; i < kPer; i += 4) {
      const float4 a = *reinterpret_cast<const float4*>(po + i);
      acc[i] += f * a.x;
      acc[i + 1] += f * a.y;
      acc[i + 2] += f * a.z;
      acc[i + 3] += f * a.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] += f * po[i];
  }
}

template <int D, bool BF>
__global__ void __launch_bounds__(kWarps * 32) combine_kernel(CombineParams p) {
  constexpr int kPer = D / 32;  // channels per lane
  const int lane = threadIdx.x & 31;
  // The work list (row count, rows, sequence info) is the prologue's, which
  // had completed before the decode kernel let this grid start: this warp's
  // first row is read before waiting for the decode kernel's partials.
  const int n = p.counters->n_comb * p.H;
  const int first = blockIdx.x * kWarps + (threadIdx.x >> 5);
  int2 tb0 = make_int2(0, 0);
  SeqInfo si0{};
  if (first < n) {
    tb0 = p.comb_rows[first / p.H];
    si0 = p.seq[tb0.y];
  }
  // The partials come from the decode kernel.  In a step with prompts the
  // decode kernel's grid completes only after the prefill grid beside it
  // (its CTA 0 waits for it before exiting), so once this returns every
  // kernel of the step before this one has completed.
  griddep_wait();
  if (p.probe_flag && blockIdx.x == 0 && threadIdx.x == 0) {
    // A bounded wait for a flag nothing sets: it runs out after 2 ms and
    // records the timeout and this site in the error words.
    const volatile int* f = p.probe_flag;
    const uint64_t t0 = global_ns();
    while (*f == 0 && global_ns() - t0 < 2000000ull) __nanosleep(1000);
    if (*f == 0) note_timeout(p.err, p.err_site, kSiteCombine | 1);
  }
  for (int idx = first; idx < n; idx += gridDim.x * kWarps) {
    const int ci = idx / p.H, h = idx - ci * p.H;
    const int2 tb = idx == first ? tb0 : p.comb_rows[ci];
    const SeqInfo si = idx == first ? si0 : p.seq[tb.y];
    const int j = tb.x - si.t0;
    const int k = h / p.G, g = h - k * p.G;
    const int r = j * p.G + g;
    const int ns = si.dec_count;
    auto row_of = [&](int s) -> size_t { return ((size_t)(si.part_first + s) * p.Hk + k) * kDecodeRows + r; };
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    float den = 0.f;
    if (ns <= 32) {
      // Lane s holds split s's (m, l); the weights reach every lane by
      // shuffle and the partial rows are loaded four splits at a time.
      const float2 ml = lane < ns ? p.part_ml[row_of(lane)] : make_float2(-INFINITY, 0.f);
      float M = ml.x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float f_own = (M != -INFINITY && ml.y != 0.f) ? exp2f(ml.x - M) : 0.f;  // 0 for empty splits
      float dl = f_own * ml.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
      den = dl;
      if (p.head_sink && M != -INFINITY) den += exp2f(elem16_to_float(p.head_sink[h], BF) * kLog2eC - M);
      for (int s0 = 0; s0 < ns; s0 += 4) {
        float f[4];
        const float* po[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int s = min(s0 + q, ns - 1);
          f[q] = __shfl_sync(0xffffffffu, f_own, s);
          if (s0 + q >= ns) f[q] = 0.f;
          po[q] = p.part_o + row_of(s) * D + lane * kPer;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (f[q] != 0.f) axpy<kPer>(acc, f[q], po[q]);
      }
    } else {
      float M = -INFINITY;
      for (int s = lane; s < ns; s += 32) M = fmaxf(M, p.part_ml[row_of(s)].x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      if (M != -INFINITY) {
        for (int s = 0; s < ns; ++s) {
          const float2 ml = p.part_ml[row_of(s)];
          if (ml.y == 0.f) continue;  // empty split
          const float f = exp2f(ml.x - M);
          den += f * ml.y;
          axpy<kPer>(acc, f, p.part_o + row_of(s) * D + lane * kPer);
        }
        if (p.head_sink) den += exp2f(elem16_to_float(p.head_sink[h], BF) * kLog2eC - M);
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __half* out = p.out + ((size_t)tb.x * p.H + h) * D + lane * kPer;
    if constexpr (kPer % 8 == 0) {
#pragma unroll
      for (int i = 0; i < kPer; i += 8)
        *reinterpret_cast<uint4*>(out + i) =
            make_uint4(pack2<BF>(acc[i] * inv, acc[i + 1] * inv), pack2<BF>(acc[i + 2] * inv, acc[i + 3] * inv),
                       pack2<BF>(acc[i + 4] * inv, acc[i + 5] * inv), pack2<BF>(acc[i + 6] * inv, acc[i + 7] * inv));
    } else {
#pragma unroll
      for (int i = 0; i < kPer; i += 2) *reinterpret_cast<uint32_t*>(out + i) = pack2<BF>(acc[i] * inv, acc[i + 1] * inv);
    }
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int grid, cudaStream_t s) {
  if (p.bf16) {
    switch (p.D) {  // (the latent layout's 512-channel rows are fp16 only)
      case 64: return launch_pdl(combine_kernel<64, true>, grid, kWarps * 32, 0, s, p);
      case 128: return launch_pdl(combine_kernel<128, true>, grid, kWarps * 32, 0, s, p);
      case 256: return launch_pdl(combine_kernel<256, true>, grid, kWarps * 32, 0, s, p);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (p.D) {
    case 64: return launch_pdl(combine_kernel<64, false>, grid, kWarps * 32, 0, s, p);
    case 128: return launch_pdl(combine_kernel<128, false>, grid, kWarps * 32, 0, s, p);
    case 256: return launch_pdl(combine_kernel<256, false>, grid, kWarps * 32, 0, s, p);
    case 512: return launch_pdl(combine_kernel<512, false>, grid, kWarps * 32, 0, s, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
