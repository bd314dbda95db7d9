// Device-side work-list builder: everything a step needs to know about the
// per-sequence lengths is derived here, on the GPU, from
// cumulative_sequence_lengths and past_sequence_lengths, so no length ever
// travels to the host and the step stays capturable ("PagedAttention - CUDA
// Design Document", section 4.7; "Design: WebGPU PagedAttention", section 5
// Phase 2 "Move seqlen_k construction to the GPU").
//
// One CTA of 1024 threads walks the batch in chunks of 1024 sequences with a
// carried block scan, so there is no cap on the batch size (the design's
// section 18.3 names the 256-sequence BlockScan cap as a defect).
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace {

constexpr int kThreads = 1024;

struct Int3 {
  int a, b, c;
};

// Exclusive scan of three counters across the block; returns the prefix and
// writes the block totals to *tot.  All threads must call it.
__device__ Int3 block_exclusive_scan3(Int3 v, Int3* tot) {
  __shared__ Int3 warp_sums[32];
  __shared__ Int3 total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Int3 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int a = __shfl_up_sync(0xffffffffu, inc.a, o);
    int b = __shfl_up_sync(0xffffffffu, inc.b, o);
    int c = __shfl_up_sync(0xffffffffu, inc.c, o);
    if (lane >= o) {
      inc.a += a;
      inc.b += b;
      inc.c += c;
    }
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    Int3 w = warp_sums[lane];
    Int3 wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int a = __shfl_up_sync(0xffffffffu, wi.a, o);
      int b = __shfl_up_sync(0xffffffffu, wi.b, o);
      int c = __shfl_up_sync(0xffffffffu, wi.c, o);
      if (lane >= o) {
        wi.a += a;
        wi.b += b;
        wi.c += c;
      }
    }
    warp_sums[lane] = Int3{wi.a - w.a, wi.b - w.b, wi.c - w.c};
    if (lane == 31) total = wi;
  }
  __syncthreads();
  *tot = total;
  Int3 base = warp_sums[warp];
  Int3 out{base.a + inc.a - v.a, base.b + inc.b - v.b, base.c + inc.c - v.c};
  __syncthreads();
  return out;
}

__device__ long long block_sum_ll(long long v) {
  __shared__ long long sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sums[warp] = v;
  __syncthreads();
  long long r = 0;
  if (warp == 0) {
    r = sums[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    if (lane == 0) sums[0] = r;
  }
  __syncthreads();
  r = sums[0];
  __syncthreads();
  return r;
}

// Validated lengths of sequence b; q_len = 0 marks a skipped sequence.
struct Lens {
  int q, past, t0, lo, route;
};

__device__ Lens read_lens(const WorklistParams& p, int b, int* err_bits) {
  Lens L{0, 0, 0, 0, kRouteNone};
  int c0 = p.cum[b], c1 = p.cum[b + 1], past = p.past[b];
  int bad = 0;
  if (b == 0 && c0 != 0) bad |= PA_DEVERR_CUM;
  if (b == p.batch - 1 && c1 != p.token_count) bad |= PA_DEVERR_CUM;
  if (c1 < c0 || c0 < 0 || c1 > p.token_count) bad |= PA_DEVERR_CUM;
  if (past < 0) bad |= PA_DEVERR_PAST;
  int q = bad ? 0 : c1 - c0;
  if (!bad && q > p.max_q) bad |= PA_DEVERR_Q_BOUND;
  if (!bad && (long long)past + q > (long long)p.max_kv) bad |= PA_DEVERR_KV_BOUND;
  *err_bits |= bad;
  if (bad || q == 0) return L;
  L.q = q;
  L.past = past;
  L.t0 = c0;
  // First key any row of this sequence may attend to, aligned down to a
  // 64-key stage.  With a window W the earliest admitted position of the
  // first new token is past + 1 - W (section 9.2 block-table pruning).
  int lo = 0;
  if (p.prune && p.window >= 1) lo = max(0, past + 1 - p.window);
  L.lo = lo & ~(kStageKeys - 1);
  L.route = (q * p.group <= p.dec_max_rows) ? kRouteDecode : kRoutePrefill;
  return L;
}

__global__ void __launch_bounds__(kThreads, 1) worklist_kernel(WorklistParams p) {
  int err_bits = 0;
  // Pass 1: total decode span, which sets the keys per split.
  long long span = 0;
  for (int base = 0; base < p.batch; base += kThreads) {
    int b = base + threadIdx.x;
    if (b < p.batch) {
      int dummy = 0;
      Lens L = read_lens(p, b, &dummy);
      if (L.route == kRouteDecode) span += (long long)(L.past + L.q - L.lo);
    }
  }
  long long total = block_sum_ll(span);
  int split_keys = p.split_keys_fixed;
  if (split_keys <= 0) {
    long long per = (total + p.target_pairs - 1) / max(p.target_pairs, 1);
    per = (per + kStageKeys - 1) / kStageKeys * kStageKeys;
    split_keys = (int)min(max(per, (long long)kStageKeys), (long long)(1 << 30));
  }

  // Pass 2: counts, scans, work items.
  Int3 carry{0, 0, 0};
  for (int base = 0; base < p.batch; base += kThreads) {
    int b = base + threadIdx.x;
    Lens L{0, 0, 0, 0, kRouteNone};
    Int3 cnt{0, 0, 0};
    if (b < p.batch) {
      L = read_lens(p, b, &err_bits);
      if (L.route == kRouteDecode) {
        int kv = L.past + L.q;
        cnt.a = (kv - L.lo + split_keys - 1) / split_keys;
        if (cnt.a > 1) cnt.c = L.q;
      } else if (L.route == kRoutePrefill) {
        cnt.b = (L.q + p.prefill_tile_tokens - 1) / p.prefill_tile_tokens;
      }
    }
    Int3 tot;
    Int3 pre = block_exclusive_scan3(cnt, &tot);
    if (b < p.batch) {
      SeqInfo si;
      si.q_len = L.q;
      si.kv_len = L.past + L.q;
      si.lo = L.lo;
      si.t0 = L.t0;
      si.dec_first = carry.a + pre.a;
      si.dec_count = cnt.a;
      si.pre_first = carry.b + pre.b;
      si.pre_count = cnt.b;
      p.seq[b] = si;
      // Capacity guards: the host sized every list from static bounds that
      // these counts cannot exceed for validated lengths; if one ever would,
      // nothing is written past the list and the whole step is dropped below.
      for (int s = 0; s < cnt.a; ++s)
        if (si.dec_first + s < p.cap_dec) p.dec_items[si.dec_first + s] = make_int2(b, s);
      for (int s = 0; s < cnt.b; ++s)
        if (si.pre_first + s < p.cap_pre) p.pre_tiles[si.pre_first + s] = make_int2(b, s);
      int c0 = carry.c + pre.c;
      for (int j = 0; j < cnt.c; ++j)
        if (c0 + j < p.cap_comb) p.comb_rows[c0 + j] = make_int2(L.t0 + j, b);
    }
    carry.a += tot.a;
    carry.b += tot.b;
    carry.c += tot.c;
  }
  if (threadIdx.x == 0) {
    Counters c;
    bool overflow = carry.a > p.cap_dec || carry.b > p.cap_pre || carry.c > p.cap_comb;
    if (overflow) err_bits |= PA_DEVERR_KV_BOUND;
    c.n_dec = overflow ? 0 : carry.a;
    c.n_pre = overflow ? 0 : carry.b;
    c.n_comb = overflow ? 0 : carry.c;
    c.split_keys = split_keys;
    *p.counters = c;
  }
  if (err_bits) atomicOr(p.err, err_bits);
}

}  // namespace

cudaError_t launch_worklist(const WorklistParams& p, cudaStream_t s) {
  worklist_kernel<<<1, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
